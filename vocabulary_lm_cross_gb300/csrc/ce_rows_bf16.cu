// ce_rows_bf16.cu -- instantiations of the row kernel for bf16 logits.
#include "ce_rows.cuh"

namespace vlmce {
namespace ce {
namespace rows {
Kernel kernel_bf16(bool softcap) { return softcap ? ce_rows_kernel<true, true> : ce_rows_kernel<true, false>; }
}  // namespace rows
}  // namespace ce
}  // namespace vlmce
