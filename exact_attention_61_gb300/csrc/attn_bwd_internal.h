// Internal interface between the C ABI (attn_host.cu) and the backward kernels
// (attn_bwd_inst.cu, attn_bwd_aux.cu). Not part of the public API.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace attn_sm103 {

// Rows of the per-head vectors in the workspace are padded to whole 128-row tiles.
constexpr int kBwdTile = 128;

struct BwdParams {
    const float* lse2;  // [BH][Npad] -LSE * log2(e); -inf on padded rows (P = 0 there)
    const float* dvec;  // [BH][Npad] -D = -rowsum(dO * O); 0 on padded rows
    float* dq_acc;      // [BH][N][d] fp32 sum of dS K over the key tiles (unscaled)
    int* item_counter;  // persistent kernel: next work item to claim (zeroed by the prologue)
    void* dk;           // [BH][N][d] dtype
    void* dv;           // [BH][N][d] dtype
    uint32_t* err;      // device status record {code, block, where, iteration}
    int Nq;             // query rows per head
    int Nk;             // keys per head
    int Npad;           // Nq rounded up to a multiple of 128
    int BH;             // batch * heads
    int H;              // heads (batch element of head bh is bh / H)
    int n_ktiles;       // ceil(Nk / 128): CTAs per head
    // Masks beyond the plain causal one (EXT kernels only; the same readings as the
    // forward's): valid keys per batch element, diagonal alignment, window bounds.
    const int32_t* kv_lens;  // [B] or null
    int align_br;            // diagonal of row i: key i (0) or i + n_b - Nq (1)
    int win_right;           // causal kernels: key j visible to row i iff j <= diag + win_right
    int win_left;            // >= 0: j >= diag - win_left; < 0: unbounded
    float qk_scale;     // scale * log2(e)
    float scale;
};

struct BwdPrepParams {
    const void* o;      // [BH][N][d] dtype
    const void* dout;   // [BH][N][d] dtype
    const float* lse;   // [BH][N] natural log
    float* lse2;        // [BH][Npad]
    float* dvec;        // [BH][Npad]
    float* dq_acc;      // [BH][N][d], zeroed here
    int* item_counter;  // zeroed here
    int N, Npad, BH, d;  // N: query rows
};

struct BwdConvertParams {
    const float* dq_acc;  // [BH][N][d]
    void* dq;             // [BH][N][d] dtype
    float scale;
    long long n;          // BH * N * d
};

// maps: Q, K, V, dO (3-D [BH][N][d] 16-bit, 64 x 128 boxes, 128-byte swizzle), then the
// fp32 dQ accumulator (3-D [BH][N][d], 32 x 128 boxes, 128-byte swizzle).
cudaError_t launch_bwd_d64_f16(bool causal, bool ext, const CUtensorMap* maps, const BwdParams& p,
                               cudaStream_t s);
cudaError_t launch_bwd_d64_bf16(bool causal, bool ext, const CUtensorMap* maps, const BwdParams& p,
                               cudaStream_t s);
cudaError_t launch_bwd_d128_f16(bool causal, bool ext, const CUtensorMap* maps, const BwdParams& p,
                               cudaStream_t s);
cudaError_t launch_bwd_d128_bf16(bool causal, bool ext, const CUtensorMap* maps, const BwdParams& p,
                               cudaStream_t s);
cudaError_t launch_bwd_prep(bool bf16, const BwdPrepParams& p, cudaStream_t s);
cudaError_t launch_bwd_convert(bool bf16, const BwdConvertParams& p, cudaStream_t s);

}  // namespace attn_sm103
