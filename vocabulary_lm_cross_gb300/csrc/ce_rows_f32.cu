// ce_rows_f32.cu -- instantiations of the row kernel for f32 logits.
#include "ce_rows.cuh"

namespace vlmce {
namespace ce {
namespace rows {
Kernel kernel_f32(bool softcap) { return softcap ? ce_rows_kernel<false, true> : ce_rows_kernel<false, false>; }
}  // namespace rows
}  // namespace ce
}  // namespace vlmce
