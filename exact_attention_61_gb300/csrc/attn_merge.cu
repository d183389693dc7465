// Merge kernel of the split-key forward (instances and launcher).
#include "attn_fwd_kernel.cuh"
#include "attn_internal.h"

namespace attn_sm103 {

// One CTA per (head, query row), launched as a programmatic dependent of the kernel ahead
// of it on the stream (the one that wrote the partials): its launch overlaps that kernel's
// tail, and the kernel waits for it to complete before reading anything.
cudaError_t launch_merge(bool bf16, const MergeParams& p, cudaStream_t s) {
    const long long rows = static_cast<long long>(p.BH) * p.Nq;
    if (rows < 1 || rows > INT32_MAX) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(static_cast<unsigned>(rows));
    cfg.blockDim = dim3(kMergeWarps * 32);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (bf16) return cudaLaunchKernelEx(&cfg, attn_merge_kernel<true>, p);
    return cudaLaunchKernelEx(&cfg, attn_merge_kernel<false>, p);
}

}  // namespace attn_sm103
