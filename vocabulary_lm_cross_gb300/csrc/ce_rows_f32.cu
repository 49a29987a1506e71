// ce_rows_f32.cu -- instantiations of the row kernel for f32 logits.
#include "ce_rows.cuh"

namespace vlmce {
namespace ce {
RowKernel rows_kernel_f32(bool softcap) {
    return softcap ? rows_kernel<false, true> : rows_kernel<false, false>;
}
}  // namespace ce
}  // namespace vlmce
