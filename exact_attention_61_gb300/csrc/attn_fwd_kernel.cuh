// Fused exact attention forward for sm_103a: TMA-fed K/V ring, tcgen05 MMAs
// accumulating in tensor memory, warp-specialised load / MMA / softmax roles.
//
// What it computes, per head and query row i (natural-log LSE):
//   O[i] = sum_{j visible} softmax_j(scale * q_i.k_j) v_j,  LSE[i] = ln sum_j exp(scale*q_i.k_j)
// following the tiled online-softmax forward of "如何用 profiler 逐步优化 Triton
// FlashAttention-2 kernel" (profile-driven FlashAttention-2 page):
//  - "Where the last article left off": tiles of query rows, a loop over key
//    tiles, running max m, running sum l and unnormalised O kept in fp32;
//  - "Round 4 / exp2": raw scores S = Q K^T, m kept in log2 units of the scaled
//    scores, P = 2^(S*qk_scale - m), alpha = 2^(m_old - m_new), and at the end
//    O / l and L = (m + log2 l) ln 2 with qk_scale = scale * log2(e) > 0;
//  - "Round 4 / Causal tile-skipping": key tiles past the diagonal are never
//    visited; only the diagonal tile and a ragged last tile are masked
//    (k_pos < N and, when causal, k_pos <= q_pos);
//  - "Round 4 / The P cast": P is rounded to the input dtype for the second product
//    and l sums the fp32 P (it gives the LSE). The page finds the order makes no
//    difference for its kernel, which rescales on every tile, so each tile's largest
//    P is exactly 1. With the lazy rescale below that P can be any value up to 2^8,
//    and its rounding would stay in the numerator only: an error proportional to |O|
//    (up to 0.4 % of |O| on the x2-scaled long problem). So O is normalised by l plus
//    lc, the sum over tiles of (rounded - fp32) of each tile's largest P: one ex2 per
//    row and tile instead of a second sum over every rounded P.
//
// GB300 design (differs from the pages' Triton/Ada kernels):
//  - one CTA owns 2 x 128 query rows of one (b, h). Each 128-row Q tile has one
//    softmax warpgroup; one thread owns one query row, i.e. one TMEM lane, so the
//    row max and row sum need no cross-thread reduction at all;
//  - one TMA warp streams 128-key K and V tiles into a multi-stage shared-memory
//    ring (128-byte swizzle); one thread issues every tcgen05.mma:
//      S_t = Q_t K_j^T   (SMEM x SMEM -> TMEM fp32, 128 x 128)
//      O_t += P_t V_j    (P from TMEM, 16-bit, aliasing S_t; V MN-major in SMEM)
//    interleaved as S_0(j), PV_1(j-1), S_1(j), PV_0(j) so that the tensor core
//    works on one Q tile while the other tile's softmax runs;
//  - rescaling of O is lazy: a row keeps a stale maximum until the new maximum
//    exceeds it by more than kRescaleTau (log2 units). P then stays <= 2^tau,
//    and the result is unchanged because O and l share the stale maximum;
//  - every mbarrier wait is bounded by a timer; on expiry the kernel records an
//    error, stops issuing work, drains its copies and MMAs, frees TMEM and exits.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <climits>

#include "attn_internal.h"
#include "sm103_ptx.cuh"

namespace attn_sm103 {

constexpr uint64_t kWaitTimeoutNs = 1500ull * 1000ull * 1000ull;  // 1.5 s
constexpr float kRescaleTau = 8.0f;                                // log2 units
constexpr uint32_t kErrTimeout = 1u;

// Roles, for the error record.
enum : uint32_t { kRoleLoad = 1, kRoleMma = 2, kRoleSoftmax0 = 3, kRoleSoftmax1 = 4 };

template <int D>
struct FwdCfg {
    static_assert(D == 64 || D == 128, "head dimension must be 64 or 128");
    static constexpr int BM = 128;  // query rows per Q tile = TMEM lanes
    static constexpr int BN = 128;  // keys per K/V tile
    static constexpr int kQTiles = 2;
    static constexpr int kRowsPerCta = BM * kQTiles;
    static_assert(kRowsPerCta == kFwdRowsPerCta, "host and kernel disagree on rows per CTA");
    static constexpr int kStages = D == 64 ? 4 : 2;
    // S/P buffers in TMEM, rotated over the jobs of both Q tiles: with 3 buffers a
    // tile's next S is computed while its softmax still runs.
    static constexpr int kSBufs = D == 64 ? 3 : 2;
    static constexpr int kBoxBytes = 128 * 128;  // one TMA box: 128 rows x 64 elements x 2 B
    static constexpr int kChunks = D / 64;       // boxes per 128-row tile
    static constexpr int kTileBytes = 128 * D * 2;
    static constexpr int kOffQ = 0;
    static constexpr int kOffK = kOffQ + kQTiles * kTileBytes;
    static constexpr int kOffV = kOffK + kStages * kTileBytes;
    static constexpr int kOffBar = kOffV + kStages * kTileBytes;
    // barriers: q_full[2] k_full[St] v_full[St] kv_empty[St] s_full[Sb] p_full[Sb] o_done[2]
    //           o_final[2] drain
    static constexpr int kBarQFull = 0;
    static constexpr int kBarKFull = 2;
    static constexpr int kBarVFull = kBarKFull + kStages;
    static constexpr int kBarKvEmpty = kBarVFull + kStages;
    static constexpr int kBarSFull = kBarKvEmpty + kStages;
    static constexpr int kBarPFull = kBarSFull + kSBufs;
    static constexpr int kBarODone = kBarPFull + kSBufs;
    static constexpr int kBarOFinal = kBarODone + 2;
    static constexpr int kBarDrain = kBarOFinal + 2;
    static constexpr int kNumBars = kBarDrain + 1;
    static constexpr int kOffMisc = kOffBar + kNumBars * 8;
    static constexpr int kSmemBytes = kOffMisc + 16 + 1024;  // + slack to align the base
    // TMEM columns: S/P buffers [0, 128*kSBufs), then O_0 and O_1 (D columns each)
    __device__ static constexpr uint32_t colS(int b) { return 128u * b; }
    __device__ static constexpr uint32_t colO(int t) { return 128u * kSBufs + D * t; }
    static_assert(128 * kSBufs + 2 * D <= 512, "TMEM budget");
    static constexpr uint32_t kTmemCols = 512;
    static constexpr int kThreads = 320;  // warps 0-3 softmax 0, 4-7 softmax 1, 8 MMA, 9 TMA
    static constexpr int kWarpMma = 8;
    static constexpr int kWarpLoad = 9;
};

// The CTA's MMA jobs, in issue order: for each K/V tile j, tile 0 then tile 1 (each
// only while that Q tile still needs keys). Q tile 1 never needs fewer K/V tiles
// than Q tile 0 (n1 is 0, n0 or n0 + 1), so the order is dense:
//   jobs 2j, 2j+1 for j < n0, then job 2*n0 for tile 1's extra diagonal tile.
struct JobOrder {
    int n0, n1;
    __device__ int total() const { return n0 + n1; }
    __device__ int job(int t, int j) const {
        if (n1 == 0) return j;
        return j < n0 ? 2 * j + t : 2 * n0 + (j - n0);
    }
    __device__ void tile_of(int g, int& t, int& j) const {
        if (n1 == 0) { t = 0; j = g; }
        else if (g < 2 * n0) { t = g & 1; j = g >> 1; }
        else { t = 1; j = n0 + (g - 2 * n0); }
    }
    // The last job that reads K/V tile j (after it, the ring stage can be refilled).
    __device__ int last_job(int j) const { return n1 == 0 ? j : job(1, j); }
    // The first job that reads K/V tile j (the one that waits for its copy to land).
    __device__ int first_job(int j) const { return (n1 == 0 || j < n0) ? job(0, j) : job(1, j); }
};

// Bounded wait state shared by all roles of one CTA.
struct WaitCtx {
    uint32_t* err;
    volatile uint32_t* abort;  // shared memory: set once any role of this CTA gave up
    uint32_t block;
};

static __device__ __noinline__ void record_timeout(const WaitCtx& w, uint32_t where, uint32_t iter) {
    if (atomicCAS(w.err, 0u, kErrTimeout) == 0u) {
        w.err[1] = w.block;
        w.err[2] = where;
        w.err[3] = iter;
        __threadfence();
    }
    *w.abort = 1u;
}

// Single-thread bounded wait. With honor_abort, gives up as soon as another role of
// the CTA has given up; without it (draining), waits for the phase up to the timeout.
static __device__ __forceinline__ bool wait_slow(uint32_t bar, uint32_t parity, const WaitCtx& w,
                                       uint32_t where, uint32_t iter, bool honor_abort) {
    const uint64_t t0 = global_timer_ns();
    for (uint32_t n = 0;; ++n) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((n & 63u) == 63u) {
            if (honor_abort && *w.abort) return false;
            if (global_timer_ns() - t0 > kWaitTimeoutNs) {
                record_timeout(w, where, iter);
                return false;
            }
        }
    }
}

static __device__ __forceinline__ bool wait_one(uint32_t bar, uint32_t parity, const WaitCtx& w,
                                         uint32_t where, uint32_t iter, bool honor_abort = true) {
    if (mbar_try_wait(bar, parity)) return true;
    return wait_slow(bar, parity, w, where, iter, honor_abort);
}

// Whole-warp bounded wait: every lane observes the phase; lane 0 decides when to
// give up so that the outcome is warp-uniform.
static __device__ __forceinline__ bool wait_warp_slow(uint32_t bar, uint32_t parity, const WaitCtx& w,
                                            uint32_t where, uint32_t iter, bool honor_abort) {
    const uint32_t lane = threadIdx.x & 31u;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t n = 0;; ++n) {
        const bool done = mbar_try_wait(bar, parity);
        if (__all_sync(0xffffffffu, done)) return true;
        if ((n & 63u) == 63u) {
            uint32_t give_up = 0;
            if (lane == 0) {
                if (honor_abort && *w.abort) give_up = 1;
                else if (global_timer_ns() - t0 > kWaitTimeoutNs) give_up = 2;
            }
            give_up = __shfl_sync(0xffffffffu, give_up, 0);
            if (give_up) {
                if (lane == 0 && give_up == 2) record_timeout(w, where, iter);
                return false;
            }
        }
    }
}

static __device__ __forceinline__ bool wait_warp(uint32_t bar, uint32_t parity, const WaitCtx& w,
                                          uint32_t where, uint32_t iter, bool honor_abort = true) {
    const bool done = mbar_try_wait(bar, parity);
    if (__all_sync(0xffffffffu, done)) return true;
    return wait_warp_slow(bar, parity, w, where, iter, honor_abort);
}

// Whole-warp bounded wait for the single-warp MMA issuers: while the phase is pending the
// warp sleeps in try_wait (up to 20 us per try, resuming when the phase completes) rather
// than polling, so it takes no issue slots from the softmax warps of its SMSP. The
// abort flag and the time limit are checked after every try.
static __device__ __forceinline__ bool wait_warp_sleep(uint32_t bar, uint32_t parity, const WaitCtx& w,
                                                uint32_t where, uint32_t iter, bool honor_abort = true) {
    if (__all_sync(0xffffffffu, mbar_try_wait(bar, parity))) return true;
    const uint32_t lane = threadIdx.x & 31u;
    const uint64_t t0 = global_timer_ns();
    for (;;) {
        if (__all_sync(0xffffffffu, mbar_try_wait_sleep<20000u>(bar, parity))) return true;
        uint32_t give_up = 0;
        if (lane == 0) {
            if (honor_abort && *w.abort) give_up = 1;
            else if (global_timer_ns() - t0 > kWaitTimeoutNs) give_up = 2;
        }
        give_up = __shfl_sync(0xffffffffu, give_up, 0);
        if (give_up) {
            if (lane == 0 && give_up == 2) record_timeout(w, where, iter);
            return false;
        }
    }
}

template <bool BF16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    if constexpr (BF16) {
        __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<uint32_t*>(&h);
    } else {
        __half2 h = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<uint32_t*>(&h);
    }
}

// The two 16-bit values of a packed pair, widened exactly to fp32 (bf16: the high 16
// bits of an fp32; fp16: a conversion).
template <bool BF16>
__device__ __forceinline__ float2 unpack2(uint32_t w) {
    if constexpr (BF16) {
        return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
    } else {
        __half2 h = *reinterpret_cast<__half2*>(&w);
        return __half22float2(h);
    }
}

// Rounding of a tile's largest P (the P of its row maximum, computed exactly as the
// exp loop computes it) to the input dtype: rounded - fp32. Zero for a row with no
// visible key in the tile (its maximum is -inf).
template <bool BF16>
__device__ __forceinline__ float max_p_rounding(float row_max, float qk, float m_use) {
    const float pm = ex2_ftz(fmaf(row_max, qk, -m_use));
    return unpack2<BF16>(pack2<BF16>(pm, 0.f)).x - pm;
}

__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// Row maximum of 128 values held as 4 x 32 raw fp32 words (8 independent chains).
__device__ __forceinline__ float row_max128(const uint32_t (&sr)[4][32]) {
    float acc[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        const uint32_t* x = &sr[c >> 1][(c & 1) * 16];
        float a = fmax3(__uint_as_float(x[0]), __uint_as_float(x[1]), __uint_as_float(x[2]));
#pragma unroll
        for (int k = 3; k < 15; k += 2) a = fmax3(a, __uint_as_float(x[k]), __uint_as_float(x[k + 1]));
        acc[c] = fmaxf(a, __uint_as_float(x[15]));
    }
    return fmaxf(fmax3(acc[0], acc[1], acc[2]), fmax3(fmax3(acc[3], acc[4], acc[5]), acc[6], acc[7]));
}

// SPLIT: this CTA covers key tiles [blockIdx.y * tiles_per_split, ...) only and writes
// fp32 partials (O_s = O/l and log2-sum-exp) instead of O and LSE.
// EXT: per-batch valid key counts, a left window bound and a right bound other than the
// diagonal; without it those parameters are ignored and the code is not compiled in.
template <int D, bool CAUSAL, bool BF16, bool SPLIT, bool EXT>
__global__ void __launch_bounds__(FwdCfg<D>::kThreads, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                    const FwdParams p) {
    using C = FwdCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* smem = smem_raw + (base - raw);

    const uint32_t warp = threadIdx.x >> 5;
    const uint32_t lane = threadIdx.x & 31u;

    auto bar = [&](int i) -> uint32_t { return base + C::kOffBar + 8u * i; };
    auto sQ = [&](int t) -> uint32_t { return base + C::kOffQ + t * C::kTileBytes; };
    auto sK = [&](int s) -> uint32_t { return base + C::kOffK + s * C::kTileBytes; };
    auto sV = [&](int s) -> uint32_t { return base + C::kOffV + s * C::kTileBytes; };
    uint32_t* misc = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);  // [0] tmem base, [1] abort

    // ---- which rows this CTA owns (heaviest causal tiles are launched first) --------
    const int bh = static_cast<int>(blockIdx.x % static_cast<uint32_t>(p.BH));
    const int ct = p.n_ctiles - 1 - static_cast<int>(blockIdx.x / static_cast<uint32_t>(p.BH));
    const int Nq = p.Nq;
    // Valid keys of this batch element (key padding): the first Nk of its keys.
    const int Nk = (EXT && p.kv_lens) ? min(max(p.kv_lens[bh / p.H], 0), p.Nk) : p.Nk;
    // The diagonal of row i is key i (top-left) or i + Nk - Nq (bottom-right: the query
    // rows are the last Nq positions, as in decoding). Under the causal mask row i sees
    // keys j <= i + off; with a left window only keys j >= i + lo_off.
    const int diag = p.align_br ? Nk - Nq : 0;
    const int off = diag + (EXT ? p.win_right : 0);
    const bool has_lo = EXT && p.win_left >= 0;
    const int lo_off = diag - p.win_left;
    const int n_kv_all = (Nk + C::BN - 1) / C::BN;
    int kv_begin = SPLIT ? static_cast<int>(blockIdx.y) * p.tiles_per_split : 0;
    const int kv_end = SPLIT ? min(n_kv_all, kv_begin + p.tiles_per_split) : n_kv_all;
    // Key tiles wholly left of the first row's window are never visited. The second Q
    // tile starts with the first (at most one extra, fully masked tile for it).
    if (has_lo) {
        const int first_key = ct * C::kRowsPerCta + lo_off;
        if (first_key > 0) kv_begin = max(kv_begin, first_key / C::BN);
    }
    // First query row and number of key tiles of each Q tile (kept in scalars: an
    // array indexed by the tile would live in local memory).
    // Key tiles a Q tile needs: all of [kv_begin, kv_end), or, under the causal mask,
    // those up to the one holding the last visible key of its last row.
    auto tiles_for = [&](int r0) -> int {
        if (r0 >= Nq) return 0;
        int end = n_kv_all;
        if (CAUSAL) {
            const int last_key = min(r0 + C::BM - 1, Nq - 1) + off;
            end = last_key < 0 ? 0 : min(n_kv_all, last_key / C::BN + 1);
        }
        return max(0, min(end, kv_end) - kv_begin);
    };
    const int row0_0 = ct * C::kRowsPerCta, row0_1 = row0_0 + C::BM;
    const int nkv_0 = tiles_for(row0_0);
    const int nkv_1 = tiles_for(row0_1);
    auto row0 = [&](int t) { return t ? row0_1 : row0_0; };
    auto n_kv = [&](int t) { return t ? nkv_1 : nkv_0; };
    const int n_max = max(nkv_0, nkv_1);
    const JobOrder jobs{nkv_0, nkv_1};

    WaitCtx wc{p.err, misc + 1, blockIdx.x};

    if (threadIdx.x == 0) {
        for (int i = 0; i < C::kNumBars; ++i) {
            const bool p_full = i >= C::kBarPFull && i < C::kBarPFull + C::kSBufs;
            mbar_init(bar(i), p_full ? 4u : 1u);  // P ready: one arrive per softmax warp
        }
        misc[1] = 0u;
        fence_mbar_init();
    }
    if (warp == C::kWarpMma) {
        tmem_alloc(smem_addr(misc), C::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = misc[0];

    if (warp == C::kWarpLoad) {
        // ================================ TMA producer ================================
        if (lane == 0) {
            tma_prefetch_desc(&tmQ);
            tma_prefetch_desc(&tmK);
            tma_prefetch_desc(&tmV);
            const uint64_t pol_q = l2_policy_evict_first();
            const uint64_t pol_kv = l2_policy_evict_last();
            for (int t = 0; t < 2; ++t) {
                if (n_kv(t) == 0) continue;
                mbar_arrive_expect_tx(bar(C::kBarQFull + t), C::kTileBytes);
                for (int c = 0; c < C::kChunks; ++c)
                    tma_load_3d_hint(sQ(t) + c * C::kBoxBytes, &tmQ, bar(C::kBarQFull + t), c * 64,
                                     row0(t), bh, pol_q);
            }
            int issued = 0;
            for (int j = 0; j < n_max; ++j) {
                const int s = j % C::kStages;
                if (j >= C::kStages &&
                    !wait_one(bar(C::kBarKvEmpty + s), ((j / C::kStages) - 1) & 1, wc,
                              kRoleLoad * 1000 + C::kBarKvEmpty + s, j))
                    break;
                mbar_arrive_expect_tx(bar(C::kBarKFull + s), C::kTileBytes);
                for (int c = 0; c < C::kChunks; ++c)
                    tma_load_3d_hint(sK(s) + c * C::kBoxBytes, &tmK, bar(C::kBarKFull + s), c * 64,
                                     (kv_begin + j) * C::BN, bh, pol_kv);
                mbar_arrive_expect_tx(bar(C::kBarVFull + s), C::kTileBytes);
                for (int c = 0; c < C::kChunks; ++c)
                    tma_load_3d_hint(sV(s) + c * C::kBoxBytes, &tmV, bar(C::kBarVFull + s), c * 64,
                                     (kv_begin + j) * C::BN, bh, pol_kv);
                issued = j + 1;
            }
            // Drain: every copy issued into this CTA's shared memory has landed before
            // the CTA can exit (on the normal path these phases completed long ago).
            for (int t = 0; t < 2; ++t)
                if (n_kv(t) > 0) wait_one(bar(C::kBarQFull + t), 0, wc, kRoleLoad * 1000 + 90 + t, 0, false);
            for (int jj = max(0, issued - C::kStages); jj < issued; ++jj) {
                const int s = jj % C::kStages;
                const uint32_t ph = (jj / C::kStages) & 1;
                wait_one(bar(C::kBarKFull + s), ph, wc, kRoleLoad * 1000 + 80, jj, false);
                wait_one(bar(C::kBarVFull + s), ph, wc, kRoleLoad * 1000 + 81, jj, false);
            }
        }
        __syncwarp();
    } else if (warp == C::kWarpMma) {
        // ================================ MMA issuer ==================================
        // The whole warp walks the job list with warp-uniform values; elect.sync picks
        // the lane that issues each tcgen05 instruction.
        {
            constexpr uint32_t idesc_s = idesc_f16_f32acc(BF16, 128, 128, false);
            constexpr uint32_t idesc_o = idesc_f16_f32acc(BF16, 128, D, true);
            // Descriptors of every operand buffer, built once; an MMA adds its byte
            // offset (>> 4) to the start-address field.
            const uint64_t dq0 = sdesc_sw128(sQ(0), 16, 1024), dq1 = sdesc_sw128(sQ(1), 16, 1024);
            const uint64_t dk0 = sdesc_sw128(sK(0), 16, 1024);
            const uint64_t dv0 = sdesc_sw128(sV(0), C::kBoxBytes, 1024);
            constexpr uint64_t kStageStep = C::kTileBytes >> 4;

            bool ok = true;
            for (int t = 0; t < 2 && ok; ++t)
                if (n_kv(t) > 0)
                    ok = wait_warp(bar(C::kBarQFull + t), 0, wc, kRoleMma * 1000 + C::kBarQFull + t, 0);
            tc_fence_after_sync();

            const int G = jobs.total();
            // S = Q_t K_j^T into S/P buffer g % kSBufs.
            auto issue_s = [&](int g) -> bool {
                int t, j;
                jobs.tile_of(g, t, j);
                const int s = j % C::kStages;
                if (!wait_warp(bar(C::kBarKFull + s), (j / C::kStages) & 1, wc,
                               kRoleMma * 1000 + C::kBarKFull + s, g))
                    return false;
                tc_fence_after_sync();
                const uint64_t a0 = t ? dq1 : dq0;
                const uint64_t b0 = dk0 + s * kStageStep;
                const uint32_t d = tmem + C::colS(g % C::kSBufs);
#pragma unroll
                for (int c = 0; c < C::kChunks; ++c) {
                    const uint64_t off = (c * C::kBoxBytes) >> 4;
                    mma_qk64_warp(d, a0 + off, b0 + off, idesc_s, c > 0 ? 1u : 0u);
                }
                mma_commit_warp(bar(C::kBarSFull + g % C::kSBufs));
                return true;
            };
            for (int g = 0; g < min(C::kSBufs, G) && ok; ++g) ok = issue_s(g);
            for (int g = 0; g < G && ok; ++g) {
                int t, j;
                jobs.tile_of(g, t, j);
                const int b = g % C::kSBufs;
                const int s = j % C::kStages;
                if (!wait_warp(bar(C::kBarPFull + b), (g / C::kSBufs) & 1, wc, kRoleMma * 1000 + C::kBarPFull + b, g) ||
                    !wait_warp(bar(C::kBarVFull + s), (j / C::kStages) & 1, wc, kRoleMma * 1000 + C::kBarVFull + s, g)) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                // O_t += P V_j, P (16-bit) read from the S/P buffer.
                const uint64_t b0 = dv0 + s * kStageStep;
                mma_pv128_warp(tmem + C::colO(t), tmem + C::colS(b), b0, idesc_o, j > 0 ? 1u : 0u);
                mma_commit_warp(bar(C::kBarODone + t));
                if (j == n_kv(t) - 1) mma_commit_warp(bar(C::kBarOFinal + t));
                if (g == jobs.last_job(j)) mma_commit_warp(bar(C::kBarKvEmpty + s));
                if (g + C::kSBufs < G) ok = issue_s(g + C::kSBufs);
            }
            // Drain: all MMAs issued by this warp are complete before TMEM is freed.
            mma_commit_warp(bar(C::kBarDrain));
            wait_warp(bar(C::kBarDrain), 0, wc, kRoleMma * 1000 + C::kBarDrain, 0, false);
        }
        __syncwarp();
    } else {
        // ================================ softmax warpgroups ==========================
        const int t = static_cast<int>(warp >> 2);
        const uint32_t wq = warp & 3u;            // TMEM lane quarter of this warp
        const uint32_t r = wq * 32u + lane;       // row inside the Q tile = TMEM lane
        const int q_row = row0(t) + static_cast<int>(r);
        const uint32_t role = t == 0 ? kRoleSoftmax0 : kRoleSoftmax1;
        const uint32_t lane_base = tmem_addr(tmem, wq * 32u, 0);
        const uint32_t tO = lane_base + C::colO(t);
        const float qk = p.qk_scale;
        const float2 qk2 = make_float2(qk, qk);

        bool ok = n_kv(t) > 0;
        // Only one Q tile has key tiles (the second is past the last row, or, with the
        // bottom-right mask, the first sees no key): its jobs are consecutive.
        const bool single_tile = nkv_0 == 0 || nkv_1 == 0;
        // Warps whose 32 rows are all past the last query row (few query rows, as in
        // decoding) skip the softmax arithmetic; their rows of O are never stored.
        const bool warp_has_rows = row0(t) + static_cast<int>(wq * 32u) < Nq;
        float m = -INFINITY;  // running max, log2 units of the scaled scores (possibly stale)
        float l = 0.f;        // running sum of P (fp32), relative to m: the LSE
        float lc = 0.f;       // rounding of each tile's largest P, relative to m: O / (l + lc)
        for (int j = 0; j < n_kv(t) && ok; ++j) {
            const int g = jobs.job(t, j);
            const int b = g % C::kSBufs;
            const uint32_t tS = lane_base + C::colS(b);
            if (!wait_warp(bar(C::kBarSFull + b), (g / C::kSBufs) & 1, wc, role * 1000 + C::kBarSFull + b, j)) {
                ok = false;
                break;
            }
            tc_fence_after_sync();
            if (!warp_has_rows) {
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(C::kBarPFull + b));
                continue;
            }
            uint32_t sr[4][32];
#pragma unroll
            for (int c = 0; c < 4; ++c) tmem_ld32(tS + c * 32, sr[c]);
            tmem_ld_wait();
#pragma unroll
            for (int c = 0; c < 4; ++c) reg_fence(sr[c]);

            const int k0 = (kv_begin + j) * C::BN;
            const bool need_mask = (k0 + C::BN > Nk) || (CAUSAL && k0 + C::BN - 1 > row0(t) + off) ||
                                   (has_lo && k0 < row0(t) + C::BM - 1 + lo_off);
            if (need_mask) {
                // keys in [lim_lo, lim) are visible
                const int lim = CAUSAL ? min(Nk, q_row + off + 1) : Nk;
                const int lim_lo = has_lo ? q_row + lo_off : INT_MIN;
#pragma unroll
                for (int c = 0; c < 4; ++c)
#pragma unroll
                    for (int e = 0; e < 32; ++e) {
                        const int key = k0 + c * 32 + e;
                        if (key >= lim || key < lim_lo) sr[c][e] = __float_as_uint(-INFINITY);
                    }
            }
            const float row_max = row_max128(sr);
            float m_new = fmaxf(m, row_max * qk);
            if (m_new - m <= kRescaleTau) m_new = m;  // keep the stale max (false when m = -inf)
            const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
            // rescale factor of the old state; exactly 1 when the maximum is kept
            const float alpha = (m == m_use) ? 1.f : ex2_ftz(m - m_use);
            const float2 neg_m2 = make_float2(-m_use, -m_use);

            uint32_t pk[2][32];
            float2 sum2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
            for (int i = 0; i < 64; ++i) {
                const float2 x = make_float2(__uint_as_float(sr[(2 * i) >> 5][(2 * i) & 31]),
                                             __uint_as_float(sr[(2 * i + 1) >> 5][(2 * i + 1) & 31]));
                const float2 y = __ffma2_rn(x, qk2, neg_m2);
                const float2 pr = make_float2(ex2_ftz(y.x), ex2_ftz(y.y));
                sum2[i & 1] = __fadd2_rn(sum2[i & 1], pr);
                pk[i >> 5][i & 31] = pack2<BF16>(pr.x, pr.y);
            }
            const float2 s2 = __fadd2_rn(sum2[0], sum2[1]);
            l = l * alpha + (s2.x + s2.y);
            lc = lc * alpha + max_p_rounding<BF16>(row_max, qk, m_use);
            tmem_st32(tS, pk[0]);
            tmem_st32(tS + 32, pk[1]);
            tmem_st_wait();

            // Before O is rescaled, the last O += P V into it must be complete. With
            // both Q tiles active the jobs interleave, so S of this job was issued
            // after O += P(j-2) V and waiting for that S leaves o_done with j-1 or j
            // completed phases: one parity wait is unambiguous. With one Q tile the
            // jobs are consecutive and this warpgroup may run two jobs ahead of its
            // O += P V; it then waits at every job so that it never falls behind.
            const bool rescale = j > 0 && __any_sync(0xffffffffu, alpha != 1.f);
            if ((rescale || (single_tile && j > 0)) &&
                !wait_warp(bar(C::kBarODone + t), (j - 1) & 1, wc, role * 1000 + C::kBarODone + t, j)) {
                ok = false;
                break;
            }
            if (rescale) {
                tc_fence_after_sync();
                const float2 a2 = make_float2(alpha, alpha);
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t o[32];
                    tmem_ld32(tO + c * 32, o);
                    tmem_ld_wait();
                    reg_fence(o);
#pragma unroll
                    for (int e = 0; e < 32; e += 2) {
                        const float2 v = __fmul2_rn(make_float2(__uint_as_float(o[e]), __uint_as_float(o[e + 1])), a2);
                        o[e] = __float_as_uint(v.x);
                        o[e + 1] = __float_as_uint(v.y);
                    }
                    tmem_st32(tO + c * 32, o);
                }
                tmem_st_wait();
            }
            m = m_new;
            // Every lane's TMEM stores are complete (wait::st) and fenced; the warp
            // barrier orders them before lane 0's release-arrive.
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(C::kBarPFull + b));
        }

        // ---- epilogue -----------------------------------------------------------------
        // A row with no visible key (possible only with causal Nq > Nk, or in a split of
        // the keys) has l = 0: its output is O = 0 and LSE = -inf.
        if (ok) {
            // o_final completes once, after the last O += P V of this tile.
            ok = wait_warp(bar(C::kBarOFinal + t), 0, wc, role * 1000 + C::kBarOFinal + t, n_kv(t));
        }
        const float m_fin = (m == -INFINITY) ? 0.f : m;
        const float inv_l = l > 0.f ? 1.f / (l + lc) : 0.f;
        const float lse2 = l > 0.f ? m_fin + log2f(l) : -INFINITY;  // log2 units
        if constexpr (SPLIT) {
            // fp32 partials for the merge: O_s = O / l and log2-sum-exp of this key range.
            const bool valid_tile = row0(t) < Nq;
            if (valid_tile && warp_has_rows && (n_kv(t) == 0 || ok)) {
                const size_t prow = (static_cast<size_t>(bh) * p.n_splits + blockIdx.y) * Nq + q_row;
                float* dst = p.o_part + prow * D;
                if (n_kv(t) > 0) tc_fence_after_sync();
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t o[32];
                    if (n_kv(t) > 0) {
                        tmem_ld32(tO + c * 32, o);
                        tmem_ld_wait();
                        reg_fence(o);
                    }
                    if (q_row < Nq) {
#pragma unroll
                        for (int e = 0; e < 32; e += 4) {
                            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
                            if (n_kv(t) > 0)
                                v = make_float4(__uint_as_float(o[e]) * inv_l, __uint_as_float(o[e + 1]) * inv_l,
                                                __uint_as_float(o[e + 2]) * inv_l, __uint_as_float(o[e + 3]) * inv_l);
                            *reinterpret_cast<float4*>(dst + c * 32 + e) = v;
                        }
                    }
                }
                if (q_row < Nq) p.lse_part[prow] = n_kv(t) > 0 ? lse2 : -INFINITY;
            }
        } else {
            // O / l -> dtype -> swizzled SMEM (reusing this Q tile) -> TMA store. A tile
            // that sees no key at all stores zeros (its Q was never loaded).
            const bool valid_tile = row0(t) < Nq;
            const bool has_kv = n_kv(t) > 0;
            if ((ok || !has_kv) && valid_tile && warp_has_rows) {
                if (has_kv) tc_fence_after_sync();
                uint8_t* stage = smem + C::kOffQ + t * C::kTileBytes;
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t o[32];
                    if (has_kv) {
                        tmem_ld32(tO + c * 32, o);
                        tmem_ld_wait();
                        reg_fence(o);
                    } else {
#pragma unroll
                        for (int e = 0; e < 32; ++e) o[e] = 0u;
                    }
                    uint32_t h[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        h[e] = pack2<BF16>(__uint_as_float(o[2 * e]) * inv_l, __uint_as_float(o[2 * e + 1]) * inv_l);
                    const int box = c >> 1;
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const uint32_t chunk = (c & 1) * 4 + i;
                        uint4 v = make_uint4(h[4 * i], h[4 * i + 1], h[4 * i + 2], h[4 * i + 3]);
                        *reinterpret_cast<uint4*>(stage + box * C::kBoxBytes + sw128_offset(r, chunk)) = v;
                    }
                }
                if (q_row < Nq)
                    p.lse[static_cast<size_t>(bh) * Nq + q_row] = lse2 * 0.69314718055994530942f;
            }
            fence_proxy_async_smem();
            if (valid_tile) named_bar_sync(1 + t, 128);
            if (valid_tile && wq == 0 && lane == 0 && *wc.abort == 0u) {
                tma_prefetch_desc(&tmO);
                for (int c = 0; c < C::kChunks; ++c)
                    tma_store_3d(&tmO, sQ(t) + c * C::kBoxBytes, c * 64, row0(t), bh);
                tma_store_commit();
                tma_store_wait_all();
            }
        }
    }

    tc_fence_before_sync();
    __syncthreads();
    if (warp == C::kWarpMma) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, C::kTmemCols);
    }
}

// Merge of split partials: per (b, h, query row), with log2-sum-exp values x_s of the
// splits, X = max_s x_s, w_s = 2^(x_s - X), O = sum_s w_s O_s / sum_s w_s and
// LSE = (X + log2 sum_s w_s) ln 2. One CTA of kMergeWarps warps per row: the threads share
// out the splits for X; each warp sums the weighted O_s of every kMergeWarps-th split with
// its lanes over the head dimension; the warps' sums are added in shared memory. Splits
// without keys (x_s = -inf) are skipped, so their partial outputs are never read. Launched
// as a dependent of the kernel that wrote the partials, it waits for that kernel first.
constexpr int kMergeWarps = 8;

template <bool BF16>
__global__ void __launch_bounds__(kMergeWarps * 32) attn_merge_kernel(const MergeParams p) {
    griddep_wait();
    __shared__ float red[kMergeWarps][129];
    const int warp = static_cast<int>(threadIdx.x >> 5);
    const int lane = static_cast<int>(threadIdx.x & 31u);
    const int row = static_cast<int>(blockIdx.x);
    const int bh = row / p.Nq, i = row % p.Nq;
    const int S = p.n_splits;
    const float* lp = p.lse_part + static_cast<size_t>(bh) * S * p.Nq + i;
    // X = max_s x_s over all threads
    float X = -INFINITY;
    for (int s = static_cast<int>(threadIdx.x); s < S; s += kMergeWarps * 32)
        X = fmaxf(X, lp[static_cast<size_t>(s) * p.Nq]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) X = fmaxf(X, __shfl_xor_sync(0xffffffffu, X, off));
    if (lane == 0) red[warp][128] = X;
    __syncthreads();
    X = red[0][128];
#pragma unroll
    for (int w = 1; w < kMergeWarps; ++w) X = fmaxf(X, red[w][128]);
    __syncthreads();
    const int per_lane = p.d / 32;  // 2 or 4
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    float wsum = 0.f;  // this warp's splits (the same value in every lane)
    if (X != -INFINITY) {
#pragma unroll 2
        for (int s = warp; s < S; s += kMergeWarps) {
            const float x = lp[static_cast<size_t>(s) * p.Nq];
            if (x == -INFINITY) continue;
            const float w = ex2_ftz(x - X);
            wsum += w;
            const float* op = p.o_part + ((static_cast<size_t>(bh) * S + s) * p.Nq + i) * p.d + lane * per_lane;
            if (per_lane == 4) {
                const float4 v = *reinterpret_cast<const float4*>(op);
                acc[0] += w * v.x;
                acc[1] += w * v.y;
                acc[2] += w * v.z;
                acc[3] += w * v.w;
            } else {
                const float2 v = *reinterpret_cast<const float2*>(op);
                acc[0] += w * v.x;
                acc[1] += w * v.y;
            }
        }
    }
    for (int e = 0; e < per_lane; ++e) red[warp][lane * per_lane + e] = acc[e];
    if (lane == 0) red[warp][128] = wsum;
    __syncthreads();
    if (warp != 0) return;
    wsum = 0.f;
#pragma unroll
    for (int w = 0; w < kMergeWarps; ++w) wsum += red[w][128];
    for (int e = 0; e < per_lane; ++e) {
        float a = 0.f;
#pragma unroll
        for (int w = 0; w < kMergeWarps; ++w) a += red[w][lane * per_lane + e];
        acc[e] = a;
    }
    const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
    const size_t orow = (static_cast<size_t>(bh) * p.Nq + i) * p.d + lane * per_lane;
    if constexpr (BF16) {
        __nv_bfloat16* o = static_cast<__nv_bfloat16*>(p.o);
        for (int e = 0; e < per_lane; ++e) o[orow + e] = __float2bfloat16_rn(acc[e] * inv);
    } else {
        __half* o = static_cast<__half*>(p.o);
        for (int e = 0; e < per_lane; ++e) o[orow + e] = __float2half_rn(acc[e] * inv);
    }
    if (lane == 0)
        p.lse[static_cast<size_t>(bh) * p.Nq + i] =
            wsum > 0.f ? (X + log2f(wsum)) * 0.69314718055994530942f : -INFINITY;
}

}  // namespace attn_sm103
