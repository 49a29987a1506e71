// ce_split_bf16.cu -- instantiations of the V-split kernel for bf16 logits.
#include "ce_split.cuh"

namespace vlmce {
namespace ce {
namespace split {
SplitKernel split_kernel_bf16(bool softcap) {
    return softcap ? ce_split_kernel<true, true> : ce_split_kernel<true, false>;
}
}  // namespace split
}  // namespace ce
}  // namespace vlmce
