// Internal interface between the C-ABI host code and the kernel instances.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

namespace attn_sm103 {

// Scalar arguments of the forward kernel (the four tensor maps are passed beside it).
struct FwdParams {
    float* lse;      // [BH, N] fp32, natural-log logsumexp of the scaled scores
    uint32_t* err;   // device status record {code, block, where, iteration}
    int N;           // sequence length (queries = keys)
    int BH;          // batch * heads
    int n_ctiles;    // ceil(N / 256): CTA tiles per head
    float qk_scale;  // scale * log2(e), > 0
};

// Query rows one CTA of the forward kernel owns.
constexpr int kFwdRowsPerCta = 256;

// Enqueue one forward launch. maps = {Q, K, V, O} tensor maps (3-D: d, N, B*H;
// 64 x 128 boxes, 128-byte swizzle). Implemented once per (d, dtype) in
// attn_fwd_inst.cu; `causal` picks the template instance.
cudaError_t launch_fwd_d64_f16(bool causal, const CUtensorMap* maps, const FwdParams& p, cudaStream_t s);
cudaError_t launch_fwd_d64_bf16(bool causal, const CUtensorMap* maps, const FwdParams& p, cudaStream_t s);
cudaError_t launch_fwd_d128_f16(bool causal, const CUtensorMap* maps, const FwdParams& p, cudaStream_t s);
cudaError_t launch_fwd_d128_bf16(bool causal, const CUtensorMap* maps, const FwdParams& p, cudaStream_t s);

// Host helpers shared by the C-ABI entry points (defined in attn_host.cu).
int cuda_fail(cudaError_t e);  // records e for attn_last_cuda_error(); returns ATTN_ERR_CUDA
PFN_cuTensorMapEncodeTiled_v12000 encode_fn(cudaError_t* err);
uint32_t* status_ptr(int dev, cudaError_t* err);
CUresult make_map(PFN_cuTensorMapEncodeTiled_v12000 enc, CUtensorMap* map, const void* ptr,
                  int64_t BH, int64_t N, int64_t d, int dtype);
cudaError_t select_device_of(const void* ptr, int* dev_out);
extern thread_local int g_last_cuda_error;

}  // namespace attn_sm103
