// Internal interface between the C-ABI host code and the kernel instances.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

namespace attn_sm103 {

// Scalar arguments of the forward kernel (the four tensor maps are passed beside it).
struct FwdParams {
    float* lse;       // [BH, Nq] fp32, natural-log logsumexp of the scaled scores
    uint32_t* err;    // device status record {code, block, where, iteration}
    int Nq;           // query rows per head
    int Nk;           // keys per head
    int BH;           // batch * heads
    int n_ctiles;     // ceil(Nq / 256): CTA tiles per head
    float qk_scale;   // scale * log2(e), > 0
    int H;            // heads (batch element of head bh is bh / H)
    const int32_t* kv_lens;  // [B] valid keys per batch element (clamped to [0, Nk]), or null
    int align_br;     // diagonal of row i: key i (0) or i + n_b - Nq (1, bottom-right)
    int win_right;    // causal kernels: row i sees keys j <= diagonal + win_right
    int win_left;     // >= 0: row i sees keys j >= diagonal - win_left; < 0: unbounded
    int tiles_per_split;  // key tiles per split (split s covers tiles [s*tps, (s+1)*tps))
    int n_splits;         // gridDim.y
    float* o_part;    // split mode: [BH][n_splits][Nq][d] fp32 partial outputs (O_s = O/l)
    float* lse_part;  // split mode: [BH][n_splits][Nq] fp32 partial log2-sum-exp (-inf if empty)
};

// Merge of split partials into O (dtype) and LSE (natural log).
struct MergeParams {
    const float* o_part;
    const float* lse_part;
    void* o;
    float* lse;
    int BH, Nq, d, n_splits;
};

// Query rows one CTA of the forward kernel owns.
constexpr int kFwdRowsPerCta = 256;

// Enqueue one forward launch. maps = {Q, K, V, O} tensor maps (3-D: d, N, B*H;
// 64 x 128 boxes, 128-byte swizzle). Implemented once per (d, dtype) in
// attn_fwd_inst.cu; `causal` picks the template instance.
// `split` selects the instance that writes fp32 partials (p.n_splits > 1); the
// grid is (n_ctiles * BH, n_splits).
cudaError_t launch_fwd_d64_f16(bool causal, bool split, bool ext, const CUtensorMap* maps, const FwdParams& p,
                               cudaStream_t s);
cudaError_t launch_fwd_d64_bf16(bool causal, bool split, bool ext, const CUtensorMap* maps, const FwdParams& p,
                               cudaStream_t s);
cudaError_t launch_fwd_d128_f16(bool causal, bool split, bool ext, const CUtensorMap* maps, const FwdParams& p,
                               cudaStream_t s);
cudaError_t launch_fwd_d128_bf16(bool causal, bool split, bool ext, const CUtensorMap* maps, const FwdParams& p,
                               cudaStream_t s);
cudaError_t launch_merge(bool bf16, const MergeParams& p, cudaStream_t s);

// Streaming decode (attn_decode.cu): up to kDecodeMaxRows query rows against a long key
// sequence, masks none / causal in either alignment (no padding or window), on the CUDA
// cores: each warp streams K and V tiles of decode_tile_keys keys through its own ring of
// 1-D bulk copies and keeps the online softmax in fp32. The keys of a head are cut into
// n_ranges ranges of range_keys keys (a multiple of the tile); with n_ranges > 1 each
// range writes fp32 O/l and its log2-sum-exp to the split partials of MergeParams' layout
// ([BH][S][Nq][d], then [BH][S][Nq]) for launch_merge, with n_ranges = 1 the final O and
// LSE directly.
constexpr int kDecodeMaxRows = 4;
inline bool fwd_uses_decode(int64_t Nq, bool ext) { return Nq <= kDecodeMaxRows && !ext; }

struct DecodeParams {
    const void* q;
    const void* k;
    const void* v;
    void* o;           // [BH][Nq][d] dtype, when n_ranges == 1
    float* lse;        // [BH][Nq], natural log, when n_ranges == 1
    float* o_part;     // split partials, when n_ranges > 1
    float* lse_part;
    uint32_t* err;     // device status record
    int BH, Nq, Nk;
    int n_ranges, range_keys;
    int causal, align_br;  // align_br: diagonal of row i is i + Nk - Nq (else i)
    float qk_scale;        // scale * log2(e)
};

struct DecodePlan {
    int64_t n_ranges, range_keys, grid;
    uint64_t o_part_bytes, bytes;  // workspace as in SplitPlan (0 when n_ranges == 1)
};
// Keys per K/V tile and warps per CTA of the decode kernel (one CTA per SM, 192 KB of
// shared memory at most) for head dimension d and Nq query rows: 32-key tiles (copies of
// 8 or 16 KB); as many warps as the registers allow, three stages per warp (two for
// several rows at d = 64, whose twelve warps would not fit three).
constexpr int decode_tile_keys(int64_t, int64_t) { return 32; }
constexpr int decode_warps(int64_t d, int64_t nq) { return d == 128 ? 4 : (nq == 1 ? 8 : 12); }
constexpr int decode_stages(int64_t d, int64_t nq) { return d == 64 && nq > 1 ? 2 : 3; }
DecodePlan plan_decode(int64_t BH, int64_t Nq, int64_t Nk, int64_t d, size_t ws_bytes, int64_t sms);
cudaError_t launch_decode(int64_t d, bool bf16, const DecodeParams& p, int64_t grid, cudaStream_t s);

// How the keys are split over CTAs (n_splits = 1: no split, no workspace).
struct SplitPlan {
    int64_t n_splits, tiles_per_split;
    uint64_t o_part_bytes, bytes;  // workspace: fp32 O partials, then fp32 LSE partials
};
SplitPlan plan_split(int64_t BH, int64_t Nq, int64_t Nk, int64_t d, size_t ws_bytes, int64_t sms);

// SMs of a device (cached per device; 0 if the query fails), and of the current device
// for the workspace and plan queries (kDefaultSmCount, a GB300's, without a device).
constexpr int64_t kDefaultSmCount = 152;
int device_sm_count(int dev);
int64_t current_sm_count();

// Static scratch of attn_fwd_kv_static (attn_static_scratch.cu): its size, and its device
// address on device `dev` (current), or null with *err set.
constexpr size_t kStaticScratchBytes = size_t(16) << 20;
void* static_scratch_ptr(int dev, cudaError_t* err);

// Host helpers shared by the C-ABI entry points (defined in attn_host.cu).
int cuda_fail(cudaError_t e);  // records e for attn_last_cuda_error(); returns ATTN_ERR_CUDA
PFN_cuTensorMapEncodeTiled_v12000 encode_fn(cudaError_t* err);
uint32_t* status_ptr(int dev, cudaError_t* err);
CUresult make_map(PFN_cuTensorMapEncodeTiled_v12000 enc, CUtensorMap* map, const void* ptr,
                  int64_t BH, int64_t N, int64_t d, int dtype);
cudaError_t select_device_of(const void* ptr, int* dev_out);
extern thread_local int g_last_cuda_error;

}  // namespace attn_sm103
