// ce_rows_bf16.cu -- instantiations of the row kernel for bf16 logits.
#include "ce_rows.cuh"

namespace vlmce {
namespace ce {
RowKernel rows_kernel_bf16(bool softcap) {
    return softcap ? rows_kernel<true, true> : rows_kernel<true, false>;
}
}  // namespace ce
}  // namespace vlmce
