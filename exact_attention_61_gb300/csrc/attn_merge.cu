// Merge kernel of the split-key forward (instances and launcher).
#include "attn_fwd_kernel.cuh"
#include "attn_internal.h"

namespace attn_sm103 {

cudaError_t launch_merge(bool bf16, const MergeParams& p, cudaStream_t s) {
    const long long rows = static_cast<long long>(p.BH) * p.Nq;
    const unsigned blocks = static_cast<unsigned>((rows * 32 + 127) / 128);
    if (bf16)
        attn_merge_kernel<true><<<blocks, 128, 0, s>>>(p);
    else
        attn_merge_kernel<false><<<blocks, 128, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace attn_sm103
