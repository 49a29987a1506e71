// ce_rows_f32.cu -- instantiations of the row kernel for f32 logits.
#include "ce_rows.cuh"

namespace vlmce {
namespace ce {
namespace rows {
Kernel kernel_f32(bool softcap, int threads) {
    if (threads == kTinyThreads) return ce_rows_kernel<false, false, kTinyThreads>;  // no softcap
    if (threads == kShortThreads)
        return softcap ? ce_rows_kernel<false, true, kShortThreads> : ce_rows_kernel<false, false, kShortThreads>;
    return softcap ? ce_rows_kernel<false, true, kThreads> : ce_rows_kernel<false, false, kThreads>;
}
}  // namespace rows
}  // namespace ce
}  // namespace vlmce
