// ce_rows_f32.cu -- instantiations of the row kernel for f32 logits.
#include "ce_rows.cuh"

namespace vlmce {
namespace ce {
namespace rows {
Kernel kernel_f32(bool softcap, int threads, bool fwd_only) {
    if (softcap) {
        if (threads == kShortThreads) return ce_rows_kernel<false, true, kShortThreads>;
        return ce_rows_kernel<false, true, kThreads>;
    }
    if (fwd_only) {  // the argmax column deferred (no pass 2)
        if (threads == kTinyThreads) return ce_rows_kernel<false, false, kTinyThreads, true>;
        if (threads == kShortThreads) return ce_rows_kernel<false, false, kShortThreads, true>;
        return ce_rows_kernel<false, false, kThreads, true>;
    }
    if (threads == kTinyThreads) return ce_rows_kernel<false, false, kTinyThreads>;
    if (threads == kShortThreads) return ce_rows_kernel<false, false, kShortThreads>;
    return ce_rows_kernel<false, false, kThreads>;
}
}  // namespace rows
}  // namespace ce
}  // namespace vlmce
