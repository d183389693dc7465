// The two small kernels around the backward: D / lse2 / zeroed dQ accumulator before
// it, and the scaled dQ cast after it.
#include "attn_bwd_internal.h"
#include "attn_bwd_kernel.cuh"

namespace attn_sm103 {

cudaError_t launch_bwd_prep(bool bf16, const BwdPrepParams& p, cudaStream_t s) {
    const long long rows = static_cast<long long>(p.BH) * p.Npad;
    const unsigned blocks = static_cast<unsigned>((rows * (p.d / 8) + 255) / 256);
    if (bf16)
        attn_bwd_prep_kernel<true><<<blocks, 256, 0, s>>>(p);
    else
        attn_bwd_prep_kernel<false><<<blocks, 256, 0, s>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_bwd_convert(bool bf16, const BwdConvertParams& p, cudaStream_t s) {
    const unsigned blocks = static_cast<unsigned>((p.n / 4 + 255) / 256);
    if (bf16)
        attn_bwd_convert_kernel<true><<<blocks, 256, 0, s>>>(p);
    else
        attn_bwd_convert_kernel<false><<<blocks, 256, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace attn_sm103
