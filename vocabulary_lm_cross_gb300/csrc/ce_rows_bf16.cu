// ce_rows_bf16.cu -- instantiations of the row kernel for bf16 logits.
#include "ce_rows.cuh"

namespace vlmce {
namespace ce {
namespace rows {
Kernel kernel_bf16(bool softcap, int threads) {
    if (threads == kTinyThreads) return ce_rows_kernel<true, false, kTinyThreads>;  // no softcap
    if (threads == kShortThreads)
        return softcap ? ce_rows_kernel<true, true, kShortThreads> : ce_rows_kernel<true, false, kShortThreads>;
    return softcap ? ce_rows_kernel<true, true, kThreads> : ce_rows_kernel<true, false, kThreads>;
}
}  // namespace rows
}  // namespace ce
}  // namespace vlmce
