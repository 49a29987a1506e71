// ce_split_f32.cu -- instantiations of the V-split kernel for f32 logits.
#include "ce_split.cuh"

namespace vlmce {
namespace ce {
namespace split {
SplitKernel split_kernel_f32(bool softcap) {
    return softcap ? ce_split_kernel<false, true> : ce_split_kernel<false, false>;
}
}  // namespace split
}  // namespace ce
}  // namespace vlmce
