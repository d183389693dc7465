// C ABI of the attention forward (see include/attn.h): argument validation,
// tensor-map encoding, device status record and dispatch to the kernel instances.
#include <algorithm>
#include <atomic>
#include <climits>
#include <cmath>
#include <cstdint>
#include <cstring>

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include "attn.h"
#include "attn_bwd_internal.h"
#include "attn_internal.h"

namespace attn_sm103 {

thread_local int g_last_cuda_error = 0;

// Device status record written by the kernels when a bounded wait gives up:
// {status bits, linear block index, role*1000 + barrier id, loop iteration}.
__device__ uint32_t g_status[4];

int cuda_fail(cudaError_t e) {
    g_last_cuda_error = static_cast<int>(e);
    return ATTN_ERR_CUDA;
}

// cuTensorMapEncodeTiled, resolved once through the runtime (no link-time libcuda).
PFN_cuTensorMapEncodeTiled_v12000 encode_fn(cudaError_t* err) {
    static std::atomic<PFN_cuTensorMapEncodeTiled_v12000> fn{nullptr};
    PFN_cuTensorMapEncodeTiled_v12000 f = fn.load(std::memory_order_acquire);
    if (f) return f;
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                                     cudaEnableDefault, &q);
    if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !p) {
        *err = e != cudaSuccess ? e : cudaErrorSymbolNotFound;
        return nullptr;
    }
    f = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    fn.store(f, std::memory_order_release);
    return f;
}

// Device address of g_status on the current device (cached per device).
uint32_t* status_ptr(int dev, cudaError_t* err) {
    static std::atomic<uintptr_t> cache[64];
    if (dev >= 0 && dev < 64) {
        uintptr_t v = cache[dev].load(std::memory_order_acquire);
        if (v) return reinterpret_cast<uint32_t*>(v);
    }
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_status);
    if (e != cudaSuccess) {
        *err = e;
        return nullptr;
    }
    if (dev >= 0 && dev < 64) cache[dev].store(reinterpret_cast<uintptr_t>(p), std::memory_order_release);
    return static_cast<uint32_t*>(p);
}

// Scratch of attn_fwd_kv_static: split partials live in this file-scope array instead
// of caller memory. A plan needs B*H * splits * Nq * (d+1) * 4 bytes; keys are split only
// while B*H * ceil(Nq/256) < 304, into at most ceil(8*152 / (B*H)) ranges, so
// B*H * splits < 1216 + 304 and 16 MiB holds every plan with Nq <= 16 (at most
// 1520 * 16 * 129 * 4 bytes, about 12.5 MB).
constexpr size_t kStaticScratchBytes = size_t(16) << 20;
static __device__ __align__(256) unsigned char g_kv_scratch[kStaticScratchBytes];

// Device address of g_kv_scratch on the current device (looked up once per device).
void* static_scratch_ptr(int dev, cudaError_t* err) {
    static std::atomic<uintptr_t> cache[64];
    if (dev >= 0 && dev < 64) {
        uintptr_t v = cache[dev].load(std::memory_order_acquire);
        if (v) return reinterpret_cast<void*>(v);
    }
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_kv_scratch);
    if (e != cudaSuccess) {
        *err = e;
        return nullptr;
    }
    if (dev >= 0 && dev < 64) cache[dev].store(reinterpret_cast<uintptr_t>(p), std::memory_order_release);
    return p;
}

namespace {

bool ranges_overlap(const void* a, uint64_t na, const void* b, uint64_t nb) {
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    return a0 < b0 + nb && b0 < a0 + na;
}

int validate(const void* q, const void* k, const void* v, const void* o, const float* lse, int64_t B,
             int64_t H, int64_t Nq, int64_t Nk, int64_t d, int mask, float scale, int dtype, const void* ws,
             size_t ws_bytes) {
    if (!q || !k || !v || !o || !lse) return ATTN_ERR_INVALID_ARG;
    if (B < 1 || H < 1 || Nq < 1 || Nk < 1 || d < 1) return ATTN_ERR_INVALID_ARG;
    if (dtype != ATTN_FP16 && dtype != ATTN_BF16) return ATTN_ERR_INVALID_ARG;
    if (mask < ATTN_MASK_NONE || mask > ATTN_MASK_CAUSAL_BOTTOM_RIGHT) return ATTN_ERR_INVALID_ARG;
    if (!std::isfinite(scale) || !(scale > 0.f)) return ATTN_ERR_INVALID_ARG;
    if (d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED;
    const uintptr_t ptrs[6] = {reinterpret_cast<uintptr_t>(q), reinterpret_cast<uintptr_t>(k),
                               reinterpret_cast<uintptr_t>(v), reinterpret_cast<uintptr_t>(o),
                               reinterpret_cast<uintptr_t>(lse), reinterpret_cast<uintptr_t>(ws)};
    for (uintptr_t p : ptrs)
        if (p % 16u) return ATTN_ERR_MISALIGNED;
    const int64_t lim31 = (int64_t(1) << 31) - 1;
    if (B > lim31 || H > lim31 || Nq > lim31 || Nk > lim31) return ATTN_ERR_UNSUPPORTED;
    if (B * H > lim31) return ATTN_ERR_UNSUPPORTED;
    const int64_t BH = B * H;
    if (BH > (int64_t(1) << 62) / (Nq * d) || BH > (int64_t(1) << 62) / (Nk * d)) return ATTN_ERR_UNSUPPORTED;
    const int64_t n_ctiles = (Nq + kFwdRowsPerCta - 1) / kFwdRowsPerCta;
    if (n_ctiles * BH > lim31) return ATTN_ERR_UNSUPPORTED;
    const uint64_t q_bytes = static_cast<uint64_t>(BH * Nq * d) * 2u;
    const uint64_t kv_bytes = static_cast<uint64_t>(BH * Nk * d) * 2u;
    const uint64_t lse_bytes = static_cast<uint64_t>(BH * Nq) * 4u;
    if (ranges_overlap(o, q_bytes, q, q_bytes) || ranges_overlap(o, q_bytes, k, kv_bytes) ||
        ranges_overlap(o, q_bytes, v, kv_bytes) || ranges_overlap(o, q_bytes, lse, lse_bytes) ||
        ranges_overlap(lse, lse_bytes, q, q_bytes) || ranges_overlap(lse, lse_bytes, k, kv_bytes) ||
        ranges_overlap(lse, lse_bytes, v, kv_bytes))
        return ATTN_ERR_INVALID_ARG;
    if (ws && ws_bytes) {
        const void* all[5] = {q, k, v, o, lse};
        const uint64_t sz[5] = {q_bytes, kv_bytes, kv_bytes, q_bytes, lse_bytes};
        for (int i = 0; i < 5; ++i)
            if (ranges_overlap(ws, ws_bytes, all[i], sz[i])) return ATTN_ERR_INVALID_ARG;
    }
    return ATTN_OK;
}

}  // namespace

// 3-D tensor map over a contiguous [BH][N][d] 16-bit array: box 64 x 128 x 1,
// 128-byte swizzle, out-of-range rows read as zero and are not written.
CUresult make_map(PFN_cuTensorMapEncodeTiled_v12000 enc, CUtensorMap* map, const void* ptr,
                  int64_t BH, int64_t N, int64_t d, int dtype) {
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N),
                                static_cast<cuuint64_t>(BH)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(d * 2), static_cast<cuuint64_t>(N * d * 2)};
    const cuuint32_t box[3] = {64, 128, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    return enc(map, dtype == ATTN_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
               3, const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

// Make the device that owns `ptr` current for this runtime instance.
cudaError_t select_device_of(const void* ptr, int* dev_out) {
    cudaPointerAttributes attr;
    cudaError_t e = cudaPointerGetAttributes(&attr, ptr);
    if (e != cudaSuccess) return e;
    if (attr.type != cudaMemoryTypeDevice && attr.type != cudaMemoryTypeManaged)
        return cudaErrorInvalidDevicePointer;
    int cur = -1;
    e = cudaGetDevice(&cur);
    if (e != cudaSuccess) return e;
    if (cur != attr.device) {
        e = cudaSetDevice(attr.device);
        if (e != cudaSuccess) return e;
    }
    *dev_out = attr.device;
    return cudaSuccess;
}

// Split of the keys over CTAs for few query rows (decoding). Only while the query rows
// alone give fewer than two CTAs per SM of a 152-SM GB300. The number of ranges S
// minimises a wave model of the launch: one CTA fits per SM, so the time is about
// ceil(CTAs * S / 152) waves of (tiles per range + 2) tile times, the 2 standing for a
// CTA's set-up and epilogue. At most eight waves of CTAs (beyond that a longer launch
// gains little and the workspace grows); limited by the workspace; S = 1: no split.
constexpr int64_t kSplitTargetCtas = 2 * 152;
constexpr int64_t kSmCount = 152;
constexpr int64_t kCtaCostTiles = 2;

SplitPlan plan_split(int64_t BH, int64_t Nq, int64_t Nk, int64_t d, size_t ws_bytes) {
    SplitPlan pl{1, 0, 0, 0};
    const int64_t n_kv_all = (Nk + 127) / 128;
    pl.tiles_per_split = n_kv_all;
    const int64_t ctas = ((Nq + kFwdRowsPerCta - 1) / kFwdRowsPerCta) * BH;
    if (ctas >= kSplitTargetCtas) return pl;  // enough CTAs already
    const uint64_t per_split = static_cast<uint64_t>(BH) * Nq * (d + 1) * 4u;
    const int64_t fit = static_cast<int64_t>(ws_bytes / per_split);
    const int64_t cap = (8 * kSmCount + ctas - 1) / ctas;
    const int64_t lim = std::min<int64_t>(std::min<int64_t>(std::min<int64_t>(n_kv_all, 65535), fit), cap);
    auto waves = [&](int64_t c) { return (c + kSmCount - 1) / kSmCount; };
    int64_t n = 1;
    int64_t best = waves(ctas) * (n_kv_all + kCtaCostTiles);
    for (int64_t c = 2; c <= lim; ++c) {
        const int64_t t = (n_kv_all + c - 1) / c;  // tiles per range
        const int64_t cost = waves(ctas * ((n_kv_all + t - 1) / t)) * (t + kCtaCostTiles);
        if (cost < best) {
            best = cost;
            n = c;
        }
    }
    if (n <= 1) return pl;
    const int64_t tps = (n_kv_all + n - 1) / n;
    pl.tiles_per_split = tps;
    pl.n_splits = (n_kv_all + tps - 1) / tps;
    if (pl.n_splits <= 1) {
        pl.n_splits = 1;
        pl.tiles_per_split = n_kv_all;
        return pl;
    }
    pl.o_part_bytes = static_cast<uint64_t>(BH) * pl.n_splits * Nq * d * 4u;
    pl.bytes = pl.o_part_bytes + static_cast<uint64_t>(BH) * pl.n_splits * Nq * 4u;
    return pl;
}

namespace {

// Which keys a row sees, beyond j < (valid keys of its batch element).
struct MaskSpec {
    bool causal;              // upper bound j <= diagonal + win_right
    int align_br;             // diagonal of row i: i (0) or i + n_b - Nq (1)
    int win_right;            // >= 0 when causal
    int win_left;             // lower bound j >= diagonal - win_left, or < 0: none
    const int32_t* kv_lens;   // device [B] valid keys, or null
};

MaskSpec mask_of(int mask) {
    MaskSpec m{mask != ATTN_MASK_NONE, mask == ATTN_MASK_CAUSAL_BOTTOM_RIGHT ? 1 : 0, 0, -1, nullptr};
    return m;
}

int fwd_core(const void* q, const void* k, const void* v, void* o, float* lse, int64_t B, int64_t H,
             int64_t Nq, int64_t Nk, int64_t d, const MaskSpec& ms, float scale, int dtype, void* ws,
             size_t ws_bytes, void* stream) {
    int dev = 0;
    cudaError_t e = select_device_of(q, &dev);
    if (e != cudaSuccess) return cuda_fail(e);
    e = cudaSuccess;
    PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn(&e);
    if (!enc) return cuda_fail(e);
    uint32_t* status = status_ptr(dev, &e);
    if (!status) return cuda_fail(e);

    const int64_t BH = B * H;
    const SplitPlan plan = plan_split(BH, Nq, Nk, d, ws ? ws_bytes : 0);
    alignas(64) CUtensorMap maps[4];
    const void* ptrs[4] = {q, k, v, o};
    const int64_t rows[4] = {Nq, Nk, Nk, Nq};
    for (int i = 0; i < 4; ++i) {
        const CUresult r = make_map(enc, &maps[i], ptrs[i], BH, rows[i], d, dtype);
        if (r != CUDA_SUCCESS) {
            g_last_cuda_error = 100000 + static_cast<int>(r);
            return ATTN_ERR_CUDA;
        }
    }
    FwdParams p;
    p.lse = lse;
    p.err = status;
    p.Nq = static_cast<int>(Nq);
    p.Nk = static_cast<int>(Nk);
    p.BH = static_cast<int>(BH);
    p.n_ctiles = static_cast<int>((Nq + kFwdRowsPerCta - 1) / kFwdRowsPerCta);
    p.qk_scale = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
    p.H = static_cast<int>(H);
    p.kv_lens = ms.kv_lens;
    p.align_br = ms.align_br;
    p.win_right = ms.win_right;
    p.win_left = ms.win_left;
    p.n_splits = static_cast<int>(plan.n_splits);
    p.tiles_per_split = static_cast<int>(plan.tiles_per_split);
    const bool split = plan.n_splits > 1;
    p.o_part = split ? static_cast<float*>(ws) : nullptr;
    p.lse_part = split ? reinterpret_cast<float*>(static_cast<char*>(ws) + plan.o_part_bytes) : nullptr;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const bool c = ms.causal;
    // Padding or a window other than the plain causal mask needs the extended instances.
    const bool x = ms.kv_lens != nullptr || ms.win_left >= 0 || ms.win_right != 0;
    if (d == 64)
        e = dtype == ATTN_BF16 ? launch_fwd_d64_bf16(c, split, x, maps, p, s)
                               : launch_fwd_d64_f16(c, split, x, maps, p, s);
    else
        e = dtype == ATTN_BF16 ? launch_fwd_d128_bf16(c, split, x, maps, p, s)
                               : launch_fwd_d128_f16(c, split, x, maps, p, s);
    if (e != cudaSuccess) return cuda_fail(e);
    if (split) {
        MergeParams mp{p.o_part, p.lse_part, o, lse, p.BH, p.Nq, static_cast<int>(d), p.n_splits};
        e = launch_merge(dtype == ATTN_BF16, mp, s);
        if (e != cudaSuccess) return cuda_fail(e);
    }
    return ATTN_OK;
}

int fwd_kv_impl(const void* q, const void* k, const void* v, void* o, float* lse, int64_t B, int64_t H,
                int64_t Nq, int64_t Nk, int64_t d, int mask, float scale, int dtype, void* ws,
                size_t ws_bytes, void* stream) {
    const int st = validate(q, k, v, o, lse, B, H, Nq, Nk, d, mask, scale, dtype, ws, ws_bytes);
    if (st != ATTN_OK) return st;
    return fwd_core(q, k, v, o, lse, B, H, Nq, Nk, d, mask_of(mask), scale, dtype, ws, ws_bytes, stream);
}

// Window bounds beyond Nq + Nk keys bind nothing: they become "unbounded" (-1).
int window_spec(int64_t Nq, int64_t Nk, int64_t left, int64_t right, const int32_t* kv_lens, int align,
                MaskSpec* out) {
    if (align != ATTN_ALIGN_TOP_LEFT && align != ATTN_ALIGN_BOTTOM_RIGHT) return ATTN_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(kv_lens) % 4u) return ATTN_ERR_MISALIGNED;
    if (Nq + Nk > (int64_t(1) << 30)) return ATTN_ERR_UNSUPPORTED;  // keeps i + offsets in int
    const int64_t span = Nq + Nk;
    out->align_br = align == ATTN_ALIGN_BOTTOM_RIGHT ? 1 : 0;
    out->causal = right >= 0 && right < span;
    out->win_right = out->causal ? static_cast<int>(right) : 0;
    out->win_left = (left >= 0 && left < span) ? static_cast<int>(left) : -1;
    out->kv_lens = kv_lens;
    return ATTN_OK;
}

struct WinArgs {
    const void *q, *k, *v;
    void* o;
    float* lse;
    int64_t B, H, Nq, Nk, d, left, right;
    const int32_t* kv_lens;
    int align;
    float scale;
    int dtype;
    void* ws;
    size_t ws_bytes;
    void* stream;
};

int win_validate(const WinArgs& a, MaskSpec* ms) {
    const int st = validate(a.q, a.k, a.v, a.o, a.lse, a.B, a.H, a.Nq, a.Nk, a.d, ATTN_MASK_NONE, a.scale,
                            a.dtype, a.ws, a.ws_bytes);
    if (st != ATTN_OK) return st;
    return window_spec(a.Nq, a.Nk, a.left, a.right, a.kv_lens, a.align, ms);
}

int win_impl(const WinArgs& a) {
    MaskSpec ms;
    const int st = win_validate(a, &ms);
    if (st != ATTN_OK) return st;
    return fwd_core(a.q, a.k, a.v, a.o, a.lse, a.B, a.H, a.Nq, a.Nk, a.d, ms, a.scale, a.dtype, a.ws, a.ws_bytes,
                    a.stream);
}

int run_win(void* ctx) { return win_impl(*static_cast<const WinArgs*>(ctx)); }

int checked(int (*run)(void*), void* ctx, const void* q, void* stream) {
    int dev = 0;
    cudaError_t e = select_device_of(q, &dev);
    if (e != cudaSuccess) return cuda_fail(e);
    uint32_t* status = status_ptr(dev, &e);
    if (!status) return cuda_fail(e);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    e = cudaMemsetAsync(status, 0, 4 * sizeof(uint32_t), s);
    if (e != cudaSuccess) return cuda_fail(e);
    const int st = run(ctx);
    if (st != ATTN_OK) return st;
    e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e);
    uint32_t host[4] = {0, 0, 0, 0};
    e = cudaMemcpy(host, status, sizeof(host), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e);
    return host[0] ? ATTN_ERR_TIMEOUT : ATTN_OK;
}

struct KvArgs {
    const void *q, *k, *v;
    void* o;
    float* lse;
    int64_t B, H, Nq, Nk, d;
    int mask;
    float scale;
    int dtype;
    void* ws;
    size_t ws_bytes;
    void* stream;
};

int run_kv(void* ctx) {
    const KvArgs* a = static_cast<const KvArgs*>(ctx);
    return fwd_kv_impl(a->q, a->k, a->v, a->o, a->lse, a->B, a->H, a->Nq, a->Nk, a->d, a->mask, a->scale,
                       a->dtype, a->ws, a->ws_bytes, a->stream);
}

// ---- backward ------------------------------------------------------------------------------

struct BwdLayout {
    int64_t Npad;
    uint64_t lse2_off, dvec_off, dq_off, bytes;
};

BwdLayout bwd_layout(int64_t BH, int64_t N, int64_t d) {
    BwdLayout L;
    L.Npad = (N + kBwdTile - 1) / kBwdTile * kBwdTile;
    L.lse2_off = 0;
    L.dvec_off = static_cast<uint64_t>(BH) * L.Npad * 4u;
    L.dq_off = 2 * L.dvec_off;
    L.bytes = L.dq_off + static_cast<uint64_t>(BH) * N * d * 4u;
    return L;
}

struct BwdArgs {
    const void *q, *k, *v, *o;
    const float* lse;
    const void* dout;
    void *dq, *dk, *dv;
    int64_t B, H, Nq, Nk, d;
    MaskSpec ms;
    float scale;
    int dtype;
    void* ws;
    size_t ws_bytes;
    void* stream;
};

int bwd_validate(const BwdArgs& a) {
    if (!a.q || !a.k || !a.v || !a.o || !a.lse || !a.dout || !a.dq || !a.dk || !a.dv || !a.ws)
        return ATTN_ERR_INVALID_ARG;
    if (a.B < 1 || a.H < 1 || a.Nq < 1 || a.Nk < 1 || a.d < 1) return ATTN_ERR_INVALID_ARG;
    if (a.dtype != ATTN_FP16 && a.dtype != ATTN_BF16) return ATTN_ERR_INVALID_ARG;
    if (!std::isfinite(a.scale) || !(a.scale > 0.f)) return ATTN_ERR_INVALID_ARG;
    if (a.d != 64 && a.d != 128) return ATTN_ERR_UNSUPPORTED;
    const void* ptrs[10] = {a.q, a.k, a.v, a.o, a.lse, a.dout, a.dq, a.dk, a.dv, a.ws};
    for (const void* p : ptrs)
        if (reinterpret_cast<uintptr_t>(p) % 16u) return ATTN_ERR_MISALIGNED;
    const int64_t lim31 = (int64_t(1) << 31) - 1;
    if (a.B > lim31 || a.H > lim31 || a.Nq > lim31 || a.Nk > lim31 || a.B * a.H > lim31)
        return ATTN_ERR_UNSUPPORTED;
    const int64_t BH = a.B * a.H;
    const int64_t Nmax = a.Nq > a.Nk ? a.Nq : a.Nk;
    if (BH > (int64_t(1) << 60) / (Nmax * a.d)) return ATTN_ERR_UNSUPPORTED;
    const BwdLayout L = bwd_layout(BH, a.Nq, a.d);
    if (((a.Nk + kBwdTile - 1) / kBwdTile) * BH > lim31) return ATTN_ERR_UNSUPPORTED;
    if (a.ws_bytes < L.bytes) return ATTN_ERR_INVALID_ARG;
    const uint64_t tq = static_cast<uint64_t>(BH * a.Nq * a.d) * 2u;  // q, o, dout, dq
    const uint64_t tk = static_cast<uint64_t>(BH * a.Nk * a.d) * 2u;  // k, v, dk, dv
    const uint64_t lb = static_cast<uint64_t>(BH * a.Nq) * 4u;
    // outputs (dq, dk, dv, workspace) overlap nothing
    const void* outs[4] = {a.dq, a.dk, a.dv, a.ws};
    const uint64_t osz[4] = {tq, tk, tk, L.bytes};
    const void* all[10] = {a.q, a.k, a.v, a.o, a.lse, a.dout, a.dq, a.dk, a.dv, a.ws};
    const uint64_t asz[10] = {tq, tk, tk, tq, lb, tq, tq, tk, tk, L.bytes};
    for (int i = 0; i < 4; ++i)
        for (int j = 0; j < 10; ++j)
            if (all[j] != outs[i] && ranges_overlap(outs[i], osz[i], all[j], asz[j])) return ATTN_ERR_INVALID_ARG;
    // an output given twice (dq == dk, say) is an overlap as well
    for (int i = 0; i < 4; ++i)
        for (int j = i + 1; j < 4; ++j)
            if (outs[i] == outs[j]) return ATTN_ERR_INVALID_ARG;
    for (int i = 0; i < 4; ++i)
        for (int j = 0; j < 6; ++j)
            if (outs[i] == all[j]) return ATTN_ERR_INVALID_ARG;
    return ATTN_OK;
}

int bwd_impl(const BwdArgs& a) {
    const int st = bwd_validate(a);
    if (st != ATTN_OK) return st;
    int dev = 0;
    cudaError_t e = select_device_of(a.q, &dev);
    if (e != cudaSuccess) return cuda_fail(e);
    e = cudaSuccess;
    PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn(&e);
    if (!enc) return cuda_fail(e);
    uint32_t* status = status_ptr(dev, &e);
    if (!status) return cuda_fail(e);
    const int64_t BH = a.B * a.H;
    const BwdLayout L = bwd_layout(BH, a.Nq, a.d);
    char* ws = static_cast<char*>(a.ws);
    float* lse2 = reinterpret_cast<float*>(ws + L.lse2_off);
    float* dvec = reinterpret_cast<float*>(ws + L.dvec_off);
    float* dq_acc = reinterpret_cast<float*>(ws + L.dq_off);
    alignas(64) CUtensorMap maps[5];
    const void* ptrs[4] = {a.q, a.k, a.v, a.dout};
    const int64_t rows[4] = {a.Nq, a.Nk, a.Nk, a.Nq};
    for (int i = 0; i < 5; ++i) {
        CUresult r;
        if (i < 4) {
            r = make_map(enc, &maps[i], ptrs[i], BH, rows[i], a.d, a.dtype);
        } else {  // fp32 dQ accumulator, 32-column boxes (128 bytes: the swizzle span)
            const cuuint64_t dims[3] = {static_cast<cuuint64_t>(a.d), static_cast<cuuint64_t>(a.Nq),
                                        static_cast<cuuint64_t>(BH)};
            const cuuint64_t strides[2] = {static_cast<cuuint64_t>(a.d * 4), static_cast<cuuint64_t>(a.Nq * a.d * 4)};
            const cuuint32_t box[3] = {32, 128, 1};
            const cuuint32_t estr[3] = {1, 1, 1};
            r = enc(&maps[4], CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, dq_acc, dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        }
        if (r != CUDA_SUCCESS) {
            g_last_cuda_error = 100000 + static_cast<int>(r);
            return ATTN_ERR_CUDA;
        }
    }
    const bool bf16 = a.dtype == ATTN_BF16;
    cudaStream_t s = static_cast<cudaStream_t>(a.stream);

    BwdPrepParams pp{a.o, a.dout, a.lse, lse2, dvec, dq_acc, static_cast<int>(a.Nq), static_cast<int>(L.Npad),
                     static_cast<int>(BH), static_cast<int>(a.d)};
    e = launch_bwd_prep(bf16, pp, s);
    if (e != cudaSuccess) return cuda_fail(e);

    BwdParams p;
    p.lse2 = lse2;
    p.dvec = dvec;
    p.dq_acc = dq_acc;
    p.dk = a.dk;
    p.dv = a.dv;
    p.err = status;
    p.Nq = static_cast<int>(a.Nq);
    p.Nk = static_cast<int>(a.Nk);
    p.Npad = static_cast<int>(L.Npad);
    p.BH = static_cast<int>(BH);
    p.H = static_cast<int>(a.H);
    p.n_ktiles = static_cast<int>((a.Nk + kBwdTile - 1) / kBwdTile);
    p.kv_lens = a.ms.kv_lens;
    p.align_br = a.ms.align_br;
    p.win_right = a.ms.win_right;
    p.win_left = a.ms.win_left;
    p.qk_scale = static_cast<float>(static_cast<double>(a.scale) * 1.4426950408889634);
    p.scale = a.scale;
    const bool c = a.ms.causal;
    // Padding, a window or Nq != Nk need the extended instances.
    const bool x = a.ms.kv_lens != nullptr || a.ms.win_left >= 0 || a.ms.win_right != 0 || a.Nq != a.Nk;
    if (a.d == 64)
        e = bf16 ? launch_bwd_d64_bf16(c, x, maps, p, s) : launch_bwd_d64_f16(c, x, maps, p, s);
    else
        e = bf16 ? launch_bwd_d128_bf16(c, x, maps, p, s) : launch_bwd_d128_f16(c, x, maps, p, s);
    if (e != cudaSuccess) return cuda_fail(e);

    BwdConvertParams cp{dq_acc, a.dq, a.scale, static_cast<long long>(BH * a.Nq * a.d)};
    e = launch_bwd_convert(bf16, cp, s);
    if (e != cudaSuccess) return cuda_fail(e);
    return ATTN_OK;
}

int run_bwd(void* ctx) { return bwd_impl(*static_cast<const BwdArgs*>(ctx)); }

}  // namespace
}  // namespace attn_sm103

using namespace attn_sm103;

extern "C" {

int attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int64_t B, int64_t H,
             int64_t N, int64_t d, int causal, float scale, int dtype, void* stream) {
    const int mask = causal ? ATTN_MASK_CAUSAL : ATTN_MASK_NONE;
    return fwd_kv_impl(q, k, v, o, lse, B, H, N, N, d, mask, scale, dtype, nullptr, 0, stream);
}

int attn_fwd_checked(const void* q, const void* k, const void* v, void* o, float* lse, int64_t B,
                     int64_t H, int64_t N, int64_t d, int causal, float scale, int dtype, void* stream) {
    const int mask = causal ? ATTN_MASK_CAUSAL : ATTN_MASK_NONE;
    const int st = validate(q, k, v, o, lse, B, H, N, N, d, mask, scale, dtype, nullptr, 0);
    if (st != ATTN_OK) return st;
    KvArgs a{q, k, v, o, lse, B, H, N, N, d, mask, scale, dtype, nullptr, 0, stream};
    return checked(run_kv, &a, q, stream);
}

size_t attn_fwd_kv_workspace_bytes(int64_t B, int64_t H, int64_t Nq, int64_t Nk, int64_t d) {
    if (B < 1 || H < 1 || Nq < 1 || Nk < 1 || (d != 64 && d != 128)) return 0;
    if (B > INT32_MAX || H > INT32_MAX || Nq > INT32_MAX || Nk > INT32_MAX || B * H > INT32_MAX) return 0;
    return static_cast<size_t>(plan_split(B * H, Nq, Nk, d, SIZE_MAX).bytes);
}

int attn_fwd_kv(const void* q, const void* k, const void* v, void* o, float* lse, int64_t B, int64_t H,
                int64_t Nq, int64_t Nk, int64_t d, int mask, float scale, int dtype, void* workspace,
                size_t workspace_bytes, void* stream) {
    return fwd_kv_impl(q, k, v, o, lse, B, H, Nq, Nk, d, mask, scale, dtype, workspace, workspace_bytes,
                       stream);
}

int attn_fwd_kv_checked(const void* q, const void* k, const void* v, void* o, float* lse, int64_t B,
                        int64_t H, int64_t Nq, int64_t Nk, int64_t d, int mask, float scale, int dtype,
                        void* workspace, size_t workspace_bytes, void* stream) {
    const int st = validate(q, k, v, o, lse, B, H, Nq, Nk, d, mask, scale, dtype, workspace, workspace_bytes);
    if (st != ATTN_OK) return st;
    KvArgs a{q, k, v, o, lse, B, H, Nq, Nk, d, mask, scale, dtype, workspace, workspace_bytes, stream};
    return checked(run_kv, &a, q, stream);
}

int attn_fwd_kv_static(const void* q, const void* k, const void* v, void* o, float* lse, int64_t B,
                       int64_t H, int64_t Nq, int64_t Nk, int64_t d, int mask, float scale, int dtype,
                       void* stream) {
    const int st = validate(q, k, v, o, lse, B, H, Nq, Nk, d, mask, scale, dtype, nullptr, 0);
    if (st != ATTN_OK) return st;
    if (plan_split(B * H, Nq, Nk, d, SIZE_MAX).bytes > kStaticScratchBytes) return ATTN_ERR_SCRATCH_TOO_SMALL;
    int dev = 0;
    cudaError_t e = select_device_of(q, &dev);
    if (e != cudaSuccess) return cuda_fail(e);
    void* scratch = static_scratch_ptr(dev, &e);
    if (!scratch) return cuda_fail(e);
    return fwd_kv_impl(q, k, v, o, lse, B, H, Nq, Nk, d, mask, scale, dtype, scratch, kStaticScratchBytes,
                       stream);
}

int attn_fwd_window(const void* q, const void* k, const void* v, void* o, float* lse, int64_t B, int64_t H,
                    int64_t Nq, int64_t Nk, int64_t d, int64_t window_left, int64_t window_right,
                    const int32_t* kv_lens, int align, float scale, int dtype, void* workspace,
                    size_t workspace_bytes, void* stream) {
    const WinArgs a{q, k, v, o, lse, B, H, Nq, Nk, d, window_left, window_right, kv_lens, align, scale, dtype,
                    workspace, workspace_bytes, stream};
    return win_impl(a);
}

int attn_fwd_window_checked(const void* q, const void* k, const void* v, void* o, float* lse, int64_t B,
                            int64_t H, int64_t Nq, int64_t Nk, int64_t d, int64_t window_left,
                            int64_t window_right, const int32_t* kv_lens, int align, float scale, int dtype,
                            void* workspace, size_t workspace_bytes, void* stream) {
    WinArgs a{q, k, v, o, lse, B, H, Nq, Nk, d, window_left, window_right, kv_lens, align, scale, dtype,
              workspace, workspace_bytes, stream};
    MaskSpec ms;
    const int st = win_validate(a, &ms);
    if (st != ATTN_OK) return st;
    return checked(run_win, &a, q, stream);
}

size_t attn_bwd_workspace_bytes(int64_t B, int64_t H, int64_t N, int64_t d) {
    if (B < 1 || H < 1 || N < 1 || (d != 64 && d != 128)) return 0;
    if (B > INT32_MAX || H > INT32_MAX || N > INT32_MAX || B * H > INT32_MAX) return 0;
    if (B * H > (int64_t(1) << 60) / (N * d)) return 0;
    return static_cast<size_t>(bwd_layout(B * H, N, d).bytes);
}

int attn_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dout,
             void* dq, void* dk, void* dv, int64_t B, int64_t H, int64_t N, int64_t d, int causal, float scale,
             int dtype, void* workspace, size_t workspace_bytes, void* stream) {
    const BwdArgs a{q, k, v, o, lse, dout, dq, dk, dv, B, H, N, N, d, mask_of(causal ? ATTN_MASK_CAUSAL : ATTN_MASK_NONE),
                    scale, dtype, workspace, workspace_bytes, stream};
    return bwd_impl(a);
}

int attn_bwd_window(const void* q, const void* k, const void* v, const void* o, const float* lse,
                    const void* dout, void* dq, void* dk, void* dv, int64_t B, int64_t H, int64_t Nq, int64_t Nk,
                    int64_t d, int64_t window_left, int64_t window_right, const int32_t* kv_lens, int align,
                    float scale, int dtype, void* workspace, size_t workspace_bytes, void* stream) {
    BwdArgs a{q, k, v, o, lse, dout, dq, dk, dv, B, H, Nq, Nk, d, MaskSpec{}, scale, dtype, workspace,
              workspace_bytes, stream};
    const int st = window_spec(Nq, Nk, window_left, window_right, kv_lens, align, &a.ms);
    if (st != ATTN_OK) return st;
    return bwd_impl(a);
}

int attn_bwd_window_checked(const void* q, const void* k, const void* v, const void* o, const float* lse,
                            const void* dout, void* dq, void* dk, void* dv, int64_t B, int64_t H, int64_t Nq,
                            int64_t Nk, int64_t d, int64_t window_left, int64_t window_right,
                            const int32_t* kv_lens, int align, float scale, int dtype, void* workspace,
                            size_t workspace_bytes, void* stream) {
    BwdArgs a{q, k, v, o, lse, dout, dq, dk, dv, B, H, Nq, Nk, d, MaskSpec{}, scale, dtype, workspace,
              workspace_bytes, stream};
    int st = window_spec(Nq, Nk, window_left, window_right, kv_lens, align, &a.ms);
    if (st != ATTN_OK) return st;
    st = bwd_validate(a);
    if (st != ATTN_OK) return st;
    return checked(run_bwd, &a, q, stream);
}

int attn_bwd_checked(const void* q, const void* k, const void* v, const void* o, const float* lse,
                     const void* dout, void* dq, void* dk, void* dv, int64_t B, int64_t H, int64_t N,
                     int64_t d, int causal, float scale, int dtype, void* workspace, size_t workspace_bytes,
                     void* stream) {
    BwdArgs a{q, k, v, o, lse, dout, dq, dk, dv, B, H, N, N, d, mask_of(causal ? ATTN_MASK_CAUSAL : ATTN_MASK_NONE),
              scale, dtype, workspace, workspace_bytes, stream};
    const int st = bwd_validate(a);
    if (st != ATTN_OK) return st;
    return checked(run_bwd, &a, q, stream);
}

const char* attn_strerror(int status) {
    switch (status) {
        case ATTN_OK: return "ok";
        case ATTN_ERR_INVALID_ARG: return "invalid argument (null pointer, size < 1, bad scale or dtype, or overlapping outputs)";
        case ATTN_ERR_UNSUPPORTED: return "unsupported (head dimension must be 64 or 128; sizes within the documented limits)";
        case ATTN_ERR_MISALIGNED: return "misaligned pointer (all tensors must be 16-byte aligned)";
        case ATTN_ERR_CUDA: return "CUDA error (see attn_last_cuda_error)";
        case ATTN_ERR_TIMEOUT: return "device-side wait timed out (outputs undefined)";
        case ATTN_ERR_SCRATCH_TOO_SMALL:
            return "the split of the keys needs more than the 16 MiB static scratch of attn_fwd_kv_static "
                   "(use attn_fwd_kv with a workspace)";
        default: return "unknown status";
    }
}

int attn_last_cuda_error(void) { return g_last_cuda_error; }

int attn_device_error_info(int32_t info[4]) {
    if (!info) return ATTN_ERR_INVALID_ARG;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    uint32_t* status = status_ptr(dev, &e);
    if (!status) return cuda_fail(e);
    uint32_t host[4];
    e = cudaMemcpy(host, status, sizeof(host), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e);
    for (int i = 0; i < 4; ++i) info[i] = static_cast<int32_t>(host[i]);
    return ATTN_OK;
}

}  // extern "C"
