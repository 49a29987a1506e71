// ce_rows_bf16.cu -- instantiations of the row kernel for bf16 logits.
#include "ce_rows.cuh"

namespace vlmce {
namespace ce {
namespace rows {
Kernel kernel_bf16(bool softcap, int threads, bool fwd_only) {
    if (softcap) {
        if (threads == kShortThreads) return ce_rows_kernel<true, true, kShortThreads>;
        return ce_rows_kernel<true, true, kThreads>;
    }
    if (fwd_only) {  // the argmax column deferred (no pass 2)
        if (threads == kTinyThreads) return ce_rows_kernel<true, false, kTinyThreads, true>;
        if (threads == kShortThreads) return ce_rows_kernel<true, false, kShortThreads, true>;
        return ce_rows_kernel<true, false, kThreads, true>;
    }
    if (threads == kTinyThreads) return ce_rows_kernel<true, false, kTinyThreads>;
    if (threads == kShortThreads) return ce_rows_kernel<true, false, kShortThreads>;
    return ce_rows_kernel<true, false, kThreads>;
}
}  // namespace rows
}  // namespace ce
}  // namespace vlmce
