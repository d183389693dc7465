// C ABI of the attention forward (see include/attn.h): argument validation,
// tensor-map encoding, device status record and dispatch to the kernel instances.
#include <algorithm>
#include <atomic>
#include <climits>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include "attn.h"
#include "attn_probe.h"
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

// SMs of a device (looked up once per device), or 0 if the query fails.
int device_sm_count(int dev) {
    static std::atomic<int> cache[64];
    if (dev >= 0 && dev < 64) {
        const int v = cache[dev].load(std::memory_order_acquire);
        if (v > 0) return v;
    }
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1) return 0;
    if (dev >= 0 && dev < 64) cache[dev].store(n, std::memory_order_release);
    return n;
}

// SMs of the current device for the size queries; a GB300's 152 when there is none.
int64_t current_sm_count() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return kDefaultSmCount;
    }
    const int n = device_sm_count(dev);
    if (n < 1) {
        cudaGetLastError();
        return kDefaultSmCount;
    }
    return n;
}

// Split of the keys over CTAs for few query rows (decoding). Only while the query rows
// alone give fewer than two CTAs per SM. The number of ranges S minimises a wave model
// of the launch: one CTA fits per SM, so the time is about ceil(CTAs * S / sms) waves of
// (tiles per range + 2) tile times, the 2 standing for a CTA's set-up and epilogue. At
// most eight waves of CTAs (beyond that a longer launch gains little and the workspace
// grows); limited by the workspace; S = 1: no split.
constexpr int64_t kCtaCostTiles = 2;

SplitPlan plan_split(int64_t BH, int64_t Nq, int64_t Nk, int64_t d, size_t ws_bytes, int64_t sms) {
    SplitPlan pl{1, 0, 0, 0};
    const int64_t n_kv_all = (Nk + 127) / 128;
    pl.tiles_per_split = n_kv_all;
    sms = std::max<int64_t>(sms, 1);
    const int64_t ctas = ((Nq + kFwdRowsPerCta - 1) / kFwdRowsPerCta) * BH;
    if (ctas >= 2 * sms) return pl;  // enough CTAs already
    const uint64_t per_split = static_cast<uint64_t>(BH) * Nq * (d + 1) * 4u;
    const int64_t fit = static_cast<int64_t>(ws_bytes / per_split);
    const int64_t cap = (8 * sms + ctas - 1) / ctas;
    const int64_t lim = std::min<int64_t>(std::min<int64_t>(std::min<int64_t>(n_kv_all, 65535), fit), cap);
    auto waves = [&](int64_t c) { return (c + sms - 1) / sms; };
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

// Ranges of the keys for the streaming decode kernel: each (head, range) unit is one warp's
// work, units go round-robin over every warp of a one-CTA-per-SM grid. The number of
// ranges per head S minimises the slowest warp's work, ceil(BH * S / warps) units of
// (tiles per range + 1) tile times, the 1 standing for a unit's start and its partial
// output. Limited by the workspace (S = 1: no workspace, the kernel writes O directly).
DecodePlan plan_decode(int64_t BH, int64_t Nq, int64_t Nk, int64_t d, size_t ws_bytes, int64_t sms) {
    sms = std::max<int64_t>(sms, 1);
    const int64_t warps = sms * decode_warps(d, Nq);
    const int64_t tile = decode_tile_keys(d, Nq);
    const int64_t n_t = (Nk + tile - 1) / tile;  // tiles per head
    const uint64_t per_range = static_cast<uint64_t>(BH) * Nq * (d + 1) * 4u;
    const int64_t fit = static_cast<int64_t>(ws_bytes / per_range);
    // at most 4096 ranges, and fewer than 2^30 units (the kernel indexes them in int)
    const int64_t lim = std::min<int64_t>(std::min<int64_t>(std::min<int64_t>(n_t, fit), 4096),
                                          (int64_t(1) << 30) / std::max<int64_t>(BH, 1));
    auto cost = [&](int64_t tpr) {
        const int64_t ranges = (n_t + tpr - 1) / tpr;
        return ((BH * ranges + warps - 1) / warps) * (tpr + 1);
    };
    int64_t best_tpr = n_t;
    int64_t best = cost(n_t);
    // every c <= lim gives tpr = ceil(n_t / c); visit each distinct tpr once, largest first
    // (the next c with a smaller tpr is ceil(n_t / (tpr - 1)))
    for (int64_t c = 2; c <= lim;) {
        const int64_t tpr = (n_t + c - 1) / c;
        const int64_t k = cost(tpr);
        if (k < best) {
            best = k;
            best_tpr = tpr;
        }
        if (tpr <= 1) break;
        c = (n_t + tpr - 2) / (tpr - 1);
    }
    DecodePlan pl{};
    pl.range_keys = best_tpr * tile;
    pl.n_ranges = (Nk + pl.range_keys - 1) / pl.range_keys;
    const int64_t units = BH * pl.n_ranges;
    pl.grid = std::min<int64_t>(sms, (units + decode_warps(d, Nq) - 1) / decode_warps(d, Nq));
    if (pl.n_ranges > 1) {
        pl.o_part_bytes = static_cast<uint64_t>(BH) * pl.n_ranges * Nq * d * 4u;
        pl.bytes = pl.o_part_bytes + static_cast<uint64_t>(BH) * pl.n_ranges * Nq * 4u;
    }
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
    const int64_t sms = device_sm_count(dev);
    if (sms < 1) return cuda_fail(cudaErrorInvalidDevice);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // Padding or a window other than the plain causal mask needs the extended instances.
    const bool x = ms.kv_lens != nullptr || ms.win_left >= 0 || ms.win_right != 0;
    if (fwd_uses_decode(Nq, x)) {
        const DecodePlan dp = plan_decode(BH, Nq, Nk, d, ws ? ws_bytes : 0, sms);
        DecodeParams p{};
        p.q = q;
        p.k = k;
        p.v = v;
        p.o = o;
        p.lse = lse;
        p.err = status;
        p.BH = static_cast<int>(BH);
        p.Nq = static_cast<int>(Nq);
        p.Nk = static_cast<int>(Nk);
        p.n_ranges = static_cast<int>(dp.n_ranges);
        p.range_keys = static_cast<int>(dp.range_keys);
        p.causal = ms.causal ? 1 : 0;
        p.align_br = ms.align_br;
        p.qk_scale = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
        const bool dsplit = dp.n_ranges > 1;
        p.o_part = dsplit ? static_cast<float*>(ws) : nullptr;
        p.lse_part = dsplit ? reinterpret_cast<float*>(static_cast<char*>(ws) + dp.o_part_bytes) : nullptr;
        e = launch_decode(d, dtype == ATTN_BF16, p, dp.grid, s);
        if (e != cudaSuccess) return cuda_fail(e);
        if (dsplit) {
            MergeParams mp{p.o_part, p.lse_part, o, lse, p.BH, p.Nq, static_cast<int>(d), p.n_ranges};
            e = launch_merge(dtype == ATTN_BF16, mp, s);
            if (e != cudaSuccess) return cuda_fail(e);
        }
        return ATTN_OK;
    }
    const SplitPlan plan = plan_split(BH, Nq, Nk, d, ws ? ws_bytes : 0, sms);
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
    const bool c = ms.causal;
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
    uint64_t lse2_off, dvec_off, dq_off, counter_off, bytes;
};

BwdLayout bwd_layout(int64_t BH, int64_t N, int64_t d) {
    BwdLayout L;
    L.Npad = (N + kBwdTile - 1) / kBwdTile * kBwdTile;
    L.lse2_off = 0;
    L.dvec_off = static_cast<uint64_t>(BH) * L.Npad * 4u;
    L.dq_off = 2 * L.dvec_off;
    // the persistent kernel's work-item counter (zeroed by the prologue)
    L.counter_off = L.dq_off + static_cast<uint64_t>(BH) * N * d * 4u;
    L.bytes = L.counter_off + 16u;
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
    int* item_counter = reinterpret_cast<int*>(ws + L.counter_off);
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

    BwdPrepParams pp{a.o, a.dout, a.lse, lse2, dvec, dq_acc, item_counter, static_cast<int>(a.Nq),
                     static_cast<int>(L.Npad), static_cast<int>(BH), static_cast<int>(a.d)};
    e = launch_bwd_prep(bf16, pp, s);
    if (e != cudaSuccess) return cuda_fail(e);

    BwdParams p;
    p.lse2 = lse2;
    p.dvec = dvec;
    p.dq_acc = dq_acc;
    p.item_counter = item_counter;
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

// ---- forward from host buffers -------------------------------------------------------------
// The heads are processed in chunks: the copy of chunk c+1's q, k, v to the device overlaps
// the kernel of chunk c, and the copy of chunk c's o and lse back to the host overlaps the
// kernels after it. Copies run on two library-owned streams (one per direction), the
// kernels on the caller's stream; events order the three.

constexpr int kHostMaxChunks = 16;
constexpr int kHostMaxDevices = 64;

struct HostPlan {
    int64_t heads_per_chunk, n_chunks;
};

// Chunks of about two full waves of 256-row work items (one CTA per SM): a chunk is
// large enough to fill the GPU, and two waves per chunk keep the waves of the whole
// problem (which the chunks add up to) near those of one launch. At most 16 chunks.
HostPlan plan_host(int64_t BH, int64_t N, int64_t sms) {
    const int64_t ctiles = (N + kFwdRowsPerCta - 1) / kFwdRowsPerCta;
    int64_t h = std::max<int64_t>(1, (2 * std::max<int64_t>(sms, 1) + ctiles - 1) / ctiles);
    h = std::max<int64_t>(h, (BH + kHostMaxChunks - 1) / kHostMaxChunks);
    h = std::min<int64_t>(h, BH);
    return HostPlan{h, (BH + h - 1) / h};
}

// Device staging of one call inside the caller's workspace: q, k, v, o ([BH][N][d] 16-bit)
// and lse ([BH][N] fp32), each starting on a 256-byte boundary.
struct HostLayout {
    uint64_t q, k, v, o, lse, bytes;
};

HostLayout host_layout(int64_t BH, int64_t N, int64_t d) {
    auto up = [](uint64_t x) { return (x + 255u) & ~uint64_t(255); };
    const uint64_t x = up(static_cast<uint64_t>(BH) * N * d * 2u);
    HostLayout L;
    L.q = 0;
    L.k = x;
    L.v = 2 * x;
    L.o = 3 * x;
    L.lse = 4 * x;
    L.bytes = 4 * x + up(static_cast<uint64_t>(BH) * N * 4u);
    return L;
}

// Sizes for which host_layout cannot overflow (the remaining rules are validate()'s).
bool host_sizes_ok(int64_t B, int64_t H, int64_t N, int64_t d) {
    if (B < 1 || H < 1 || N < 1 || (d != 64 && d != 128)) return false;
    if (B > INT32_MAX || H > INT32_MAX || N > INT32_MAX || B * H > INT32_MAX) return false;
    return B * H <= (int64_t(1) << 58) / (N * d);
}

// Library-owned streams and events of one device, made on the first call there and kept
// for the life of the process. Calls on one device enqueue under `mu`, so an event is
// never recorded by one call between another call's record of it and its wait on it.
struct HostCtx {
    std::mutex mu;
    bool ready = false;
    cudaStream_t h2d = nullptr, d2h = nullptr;
    cudaEvent_t start = nullptr, h2d_done = nullptr, d2h_done = nullptr;
    cudaEvent_t in_ready[kHostMaxChunks] = {}, out_ready[kHostMaxChunks] = {};

    cudaError_t init() {
        if (ready) return cudaSuccess;
        cudaError_t e = cudaStreamCreateWithFlags(&h2d, cudaStreamNonBlocking);
        if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&d2h, cudaStreamNonBlocking);
        cudaEvent_t* evs[3 + 2 * kHostMaxChunks];
        int n = 0;
        evs[n++] = &start;
        evs[n++] = &h2d_done;
        evs[n++] = &d2h_done;
        for (int c = 0; c < kHostMaxChunks; ++c) {
            evs[n++] = &in_ready[c];
            evs[n++] = &out_ready[c];
        }
        for (int i = 0; i < n && e == cudaSuccess; ++i) e = cudaEventCreateWithFlags(evs[i], cudaEventDisableTiming);
        if (e != cudaSuccess) {
            for (int i = 0; i < n; ++i)
                if (*evs[i]) {
                    cudaEventDestroy(*evs[i]);
                    *evs[i] = nullptr;
                }
            if (h2d) cudaStreamDestroy(h2d);
            if (d2h) cudaStreamDestroy(d2h);
            h2d = d2h = nullptr;
            return e;
        }
        ready = true;
        return cudaSuccess;
    }
};

HostCtx g_host_ctx[kHostMaxDevices];

struct HostArgs {
    const void *q, *k, *v;  // host (or any) memory, [B, H, N, d] of dtype
    void* o;                // host (or any) memory, [B, H, N, d] of dtype
    float* lse;             // host (or any) memory, [B, H, N] fp32
    void* ws;               // device workspace
    size_t ws_bytes;
    int64_t B, H, N, d;
    int causal;
    float scale;
    int dtype;
    void* stream;
};

// q = k = v = NULL: the inputs are already in the workspace (staged by an earlier call).
bool host_inputs_staged(const HostArgs& a) { return !a.q && !a.k && !a.v; }

int host_validate(const HostArgs& a, HostLayout* L) {
    const bool staged = host_inputs_staged(a);
    if ((!staged && (!a.q || !a.k || !a.v)) || !a.o || !a.lse || !a.ws) return ATTN_ERR_INVALID_ARG;
    if (a.B < 1 || a.H < 1 || a.N < 1 || a.d < 1) return ATTN_ERR_INVALID_ARG;
    if (a.d != 64 && a.d != 128) return ATTN_ERR_UNSUPPORTED;
    if (!host_sizes_ok(a.B, a.H, a.N, a.d)) return ATTN_ERR_UNSUPPORTED;
    if (reinterpret_cast<uintptr_t>(a.ws) % 256u) return ATTN_ERR_MISALIGNED;
    const int64_t BH = a.B * a.H;
    *L = host_layout(BH, a.N, a.d);
    if (a.ws_bytes < L->bytes) return ATTN_ERR_INVALID_ARG;
    // The device staging buffers must pass every rule of attn_fwd.
    char* w = static_cast<char*>(a.ws);
    const int st = validate(w + L->q, w + L->k, w + L->v, w + L->o, reinterpret_cast<float*>(w + L->lse), a.B,
                            a.H, a.N, a.N, a.d, a.causal ? ATTN_MASK_CAUSAL : ATTN_MASK_NONE, a.scale, a.dtype,
                            nullptr, 0);
    if (st != ATTN_OK) return st;
    // Host outputs overlap neither each other, nor the inputs, nor the workspace.
    const uint64_t qb = static_cast<uint64_t>(BH) * a.N * a.d * 2u, lb = static_cast<uint64_t>(BH) * a.N * 4u;
    const void* ins[3] = {a.q, a.k, a.v};
    for (int i = 0; i < 3 && !staged; ++i)
        if (ranges_overlap(a.o, qb, ins[i], qb) || ranges_overlap(a.lse, lb, ins[i], qb)) return ATTN_ERR_INVALID_ARG;
    if (ranges_overlap(a.o, qb, a.lse, lb)) return ATTN_ERR_INVALID_ARG;
    const void* all[5] = {a.o, a.lse, a.q, a.k, a.v};
    const uint64_t sz[5] = {qb, lb, qb, qb, qb};
    for (int i = 0; i < (staged ? 2 : 5); ++i)
        if (ranges_overlap(a.ws, L->bytes, all[i], sz[i])) return ATTN_ERR_INVALID_ARG;
    return ATTN_OK;
}

int host_impl(const HostArgs& a) {
    HostLayout L;
    const int st0 = host_validate(a, &L);
    if (st0 != ATTN_OK) return st0;
    int dev = 0;
    cudaError_t e = select_device_of(a.ws, &dev);  // the workspace must be device memory
    if (e != cudaSuccess) return cuda_fail(e);
    if (dev < 0 || dev >= kHostMaxDevices) return ATTN_ERR_UNSUPPORTED;
    HostCtx& ctx = g_host_ctx[dev];
    std::lock_guard<std::mutex> lock(ctx.mu);
    e = ctx.init();
    if (e != cudaSuccess) return cuda_fail(e);

    const int64_t BH = a.B * a.H;
    const int64_t sms = device_sm_count(dev);
    if (sms < 1) return cuda_fail(cudaErrorInvalidDevice);
    const HostPlan pl = plan_host(BH, a.N, sms);
    const uint64_t head = static_cast<uint64_t>(a.N) * a.d * 2u, lhead = static_cast<uint64_t>(a.N) * 4u;
    char* w = static_cast<char*>(a.ws);
    const char* hq = static_cast<const char*>(a.q);
    const char* hk = static_cast<const char*>(a.k);
    const char* hv = static_cast<const char*>(a.v);
    char* ho = static_cast<char*>(a.o);
    char* hl = reinterpret_cast<char*>(a.lse);
    cudaStream_t s = static_cast<cudaStream_t>(a.stream);
    const MaskSpec ms = mask_of(a.causal ? ATTN_MASK_CAUSAL : ATTN_MASK_NONE);

    // Everything before this call on `stream` precedes the copies (they may read or
    // write host buffers that earlier work produces or consumes).
    e = cudaEventRecord(ctx.start, s);
    if (e != cudaSuccess) return cuda_fail(e);
    e = cudaStreamWaitEvent(ctx.h2d, ctx.start, 0);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(ctx.d2h, ctx.start, 0);
    // From here on, whatever happens, `stream` is made to wait for both copy streams
    // before returning, so that later work on it sees this call's copies finished.
    int status = ATTN_OK;
    auto fail = [&](cudaError_t err) {
        if (status == ATTN_OK) status = cuda_fail(err);
    };
    if (e != cudaSuccess) fail(e);
    const bool staged = host_inputs_staged(a);
    for (int64_t c = 0; c < pl.n_chunks && status == ATTN_OK && !staged; ++c) {
        const int64_t h0 = c * pl.heads_per_chunk;
        const uint64_t off = static_cast<uint64_t>(h0) * head;
        const uint64_t n = static_cast<uint64_t>(std::min(pl.heads_per_chunk, BH - h0)) * head;
        e = cudaMemcpyAsync(w + L.q + off, hq + off, n, cudaMemcpyDefault, ctx.h2d);
        if (e == cudaSuccess) e = cudaMemcpyAsync(w + L.k + off, hk + off, n, cudaMemcpyDefault, ctx.h2d);
        if (e == cudaSuccess) e = cudaMemcpyAsync(w + L.v + off, hv + off, n, cudaMemcpyDefault, ctx.h2d);
        if (e == cudaSuccess) e = cudaEventRecord(ctx.in_ready[c], ctx.h2d);
        if (e != cudaSuccess) fail(e);
    }
    int64_t launched = 0;
    for (int64_t c = 0; c < pl.n_chunks && status == ATTN_OK; ++c) {
        const int64_t h0 = c * pl.heads_per_chunk;
        const int64_t hc = std::min(pl.heads_per_chunk, BH - h0);
        const uint64_t off = static_cast<uint64_t>(h0) * head, loff = static_cast<uint64_t>(h0) * lhead;
        e = staged ? cudaSuccess : cudaStreamWaitEvent(s, ctx.in_ready[c], 0);
        if (e != cudaSuccess) {
            fail(e);
            break;
        }
        // one chunk = hc consecutive (b, h) pairs: a [1, hc, N, d] problem
        const int st = fwd_core(w + L.q + off, w + L.k + off, w + L.v + off, w + L.o + off,
                                reinterpret_cast<float*>(w + L.lse + loff), 1, hc, a.N, a.N, a.d, ms, a.scale,
                                a.dtype, nullptr, 0, s);
        if (st != ATTN_OK) {
            status = st;
            break;
        }
        e = cudaEventRecord(ctx.out_ready[c], s);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(ctx.d2h, ctx.out_ready[c], 0);
        if (e != cudaSuccess) {
            fail(e);
            break;
        }
        launched = c + 1;
    }
    for (int64_t c = 0; c < launched && status == ATTN_OK; ++c) {
        const int64_t h0 = c * pl.heads_per_chunk;
        const int64_t hc = std::min(pl.heads_per_chunk, BH - h0);
        const uint64_t off = static_cast<uint64_t>(h0) * head, loff = static_cast<uint64_t>(h0) * lhead;
        // The copy stream has waited for out_ready[c], recorded after chunk c's kernel.
        e = cudaMemcpyAsync(ho + off, w + L.o + off, static_cast<uint64_t>(hc) * head, cudaMemcpyDefault, ctx.d2h);
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(hl + loff, w + L.lse + loff, static_cast<uint64_t>(hc) * lhead, cudaMemcpyDefault,
                                ctx.d2h);
        if (e != cudaSuccess) fail(e);
    }
    e = cudaEventRecord(ctx.h2d_done, ctx.h2d);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(s, ctx.h2d_done, 0);
    if (e != cudaSuccess) fail(e);
    e = cudaEventRecord(ctx.d2h_done, ctx.d2h);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(s, ctx.d2h_done, 0);
    if (e != cudaSuccess) fail(e);
    return status;
}

int run_host(void* ctx) { return host_impl(*static_cast<const HostArgs*>(ctx)); }

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
    const int64_t sms = current_sm_count();
    // A call with at most kDecodeMaxRows rows runs the decode kernel unless it has padding
    // or a window (attn_fwd_window shares this query): room for either plan.
    uint64_t bytes = plan_split(B * H, Nq, Nk, d, SIZE_MAX, sms).bytes;
    if (Nq <= kDecodeMaxRows) bytes = std::max(bytes, plan_decode(B * H, Nq, Nk, d, SIZE_MAX, sms).bytes);
    return static_cast<size_t>(bytes);
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
    // Sizes the scratch cannot hold are refused on the host first (with the current
    // device's SM count), then again for the device that owns q.
    if (plan_split(B * H, Nq, Nk, d, SIZE_MAX, current_sm_count()).bytes > kStaticScratchBytes)
        return ATTN_ERR_SCRATCH_TOO_SMALL;
    int dev = 0;
    cudaError_t e = select_device_of(q, &dev);
    if (e != cudaSuccess) return cuda_fail(e);
    const int64_t sms = device_sm_count(dev);
    if (sms < 1) return cuda_fail(cudaErrorInvalidDevice);
    if (plan_split(B * H, Nq, Nk, d, SIZE_MAX, sms).bytes > kStaticScratchBytes) return ATTN_ERR_SCRATCH_TOO_SMALL;
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

int64_t attn_fwd_host_plan(int64_t B, int64_t H, int64_t N, int64_t d, int64_t* heads_per_chunk) {
    if (!host_sizes_ok(B, H, N, d)) return 0;
    const HostPlan pl = plan_host(B * H, N, current_sm_count());
    if (heads_per_chunk) *heads_per_chunk = pl.heads_per_chunk;
    return pl.n_chunks;
}

size_t attn_fwd_host_workspace_bytes(int64_t B, int64_t H, int64_t N, int64_t d) {
    if (!host_sizes_ok(B, H, N, d)) return 0;
    return static_cast<size_t>(host_layout(B * H, N, d).bytes);
}

int attn_fwd_host(const void* q, const void* k, const void* v, void* o, float* lse, int64_t B, int64_t H,
                  int64_t N, int64_t d, int causal, float scale, int dtype, void* workspace,
                  size_t workspace_bytes, void* stream) {
    const HostArgs a{q, k, v, o, lse, workspace, workspace_bytes, B, H, N, d, causal, scale, dtype, stream};
    return host_impl(a);
}

int attn_fwd_host_checked(const void* q, const void* k, const void* v, void* o, float* lse, int64_t B,
                          int64_t H, int64_t N, int64_t d, int causal, float scale, int dtype, void* workspace,
                          size_t workspace_bytes, void* stream) {
    HostArgs a{q, k, v, o, lse, workspace, workspace_bytes, B, H, N, d, causal, scale, dtype, stream};
    HostLayout L;
    const int st = host_validate(a, &L);
    if (st != ATTN_OK) return st;
    return checked(run_host, &a, workspace, stream);
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

int attn_probe_plan_split(int64_t BH, int64_t Nq, int64_t Nk, int64_t d, size_t ws_bytes, int64_t sms,
                          int64_t out[3]) {
    if (!out || BH < 1 || Nq < 1 || Nk < 1 || (d != 64 && d != 128) || sms < 1) return ATTN_ERR_INVALID_ARG;
    const SplitPlan pl = plan_split(BH, Nq, Nk, d, ws_bytes, sms);
    out[0] = pl.n_splits;
    out[1] = pl.tiles_per_split;
    out[2] = static_cast<int64_t>(pl.bytes);
    return ATTN_OK;
}

int attn_probe_plan_decode(int64_t BH, int64_t Nq, int64_t Nk, int64_t d, size_t ws_bytes, int64_t sms,
                           int64_t out[4]) {
    if (!out || BH < 1 || BH > INT32_MAX || Nq < 1 || Nq > kDecodeMaxRows || Nk < 1 || Nk > INT32_MAX ||
        (d != 64 && d != 128) || sms < 1)
        return ATTN_ERR_INVALID_ARG;
    const DecodePlan pl = plan_decode(BH, Nq, Nk, d, ws_bytes, sms);
    out[0] = pl.n_ranges;
    out[1] = pl.range_keys;
    out[2] = pl.grid;
    out[3] = static_cast<int64_t>(pl.bytes);
    return ATTN_OK;
}

int64_t attn_probe_plan_host(int64_t BH, int64_t N, int64_t sms, int64_t* heads_per_chunk) {
    if (BH < 1 || N < 1 || sms < 1) return 0;
    const HostPlan pl = plan_host(BH, N, sms);
    if (heads_per_chunk) *heads_per_chunk = pl.heads_per_chunk;
    return pl.n_chunks;
}

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
