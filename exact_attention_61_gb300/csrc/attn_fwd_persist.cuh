// Persistent fused attention forward for head dimension 64 on sm_103a: one CTA per
// SM walks a static list of work items (256 query rows of one head), so that the next
// item's Q load and first S = Q K^T overlap the current item's last O += P V and its
// output store.
//
// It computes what the one-item kernel in attn_fwd_kernel.cuh computes, with the same
// arithmetic in the same order, following the tiled online-softmax forward of
// "如何用 profiler 逐步优化 Triton FlashAttention-2 kernel" ("Where the last article
// left off", "Round 4 / exp2", "Round 4 / Causal tile-skipping", "Round 4 / The P
// cast"); the outputs are equal bit for bit. What differs is who issues what:
//  - warp 8 issues every S = Q K^T (SMEM x SMEM -> TMEM, 128 x 128) into three S/P
//    buffers that rotate over the CTA's job stream (job = one Q tile against one K/V
//    tile). S of job g reuses the buffer of job g-3 once O += P V of job g-3 has
//    completed (pv_done); having seen that, warp 8 also hands the K/V ring stage back
//    to the loader when job g-3 was the last reader of its tile;
//  - the softmax warpgroup of Q tile t writes P (16-bit) over S in TMEM and hands it to
//    warp 11, which issues every O_t += P V (P from TMEM, V MN-major in SMEM). With
//    the S and P V issues in two warps, neither issuer's waits and commits hold up the
//    other's MMAs (one warp issuing both paced the earlier one-item kernel);
//  - warp 9 loads Q (two buffers, so item a+1's Q lands while item a runs) and the K/V
//    ring; warp 10 stores O by TMA from the staging tile the softmax warpgroup wrote
//    and returns the Q buffer to the loader.
// Registers: the two softmax warpgroups raise their budget (setmaxnreg) to 208 per
// thread, the warpgroup of single-warp roles lowers its own to 88.
//
// Every mbarrier wait is bounded (as in the one-item kernel): on expiry a role records
// the error, stops issuing work, drains its copies and MMAs, and the CTA exits. Every
// parity wait is exact (the barrier is at most one phase short of the awaited one when
// the wait starts); the reason is given at each barrier that needs one.
#pragma once

#include "attn_fwd_kernel.cuh"

namespace attn_sm103 {

struct PersistCfg {
    static constexpr int D = 64;
    static constexpr int BM = 128;
    static constexpr int BN = 128;
    static constexpr int kStages = 4;
    static constexpr int kSBufs = 3;
    static constexpr int kTileBytes = 128 * D * 2;  // 16 KB: one 128 x 64 16-bit box
    static constexpr int kOffQ = 0;                 // Q[buffer][tile]
    static constexpr int kOffK = kOffQ + 4 * kTileBytes;
    static constexpr int kOffV = kOffK + kStages * kTileBytes;
    static constexpr int kOffBar = kOffV + kStages * kTileBytes;
    // barriers
    static constexpr int kBarQFull = 0;                   // [buf][tile]: 4
    static constexpr int kBarQEmpty = kBarQFull + 4;      // [buf][tile]: 4
    static constexpr int kBarKFull = kBarQEmpty + 4;      // [stage]
    static constexpr int kBarVFull = kBarKFull + kStages;
    static constexpr int kBarKvEmpty = kBarVFull + kStages;
    static constexpr int kBarSFull = kBarKvEmpty + kStages;  // [tile][buf]
    static constexpr int kBarPvDone = kBarSFull + 2 * kSBufs;  // [buf]
    static constexpr int kBarPFull = kBarPvDone + kSBufs;      // [buf] (PV warp mode)
    static constexpr int kBarODone = kBarPFull + kSBufs;       // [tile][2]
    static constexpr int kBarOStaged = kBarODone + 4;          // [buf][tile]: O staged for the store warp
    static constexpr int kBarDrain = kBarOStaged + 4;          // [issuer]: S, P V
    static constexpr int kNumBars = kBarDrain + 4;
    static constexpr int kOffMisc = kOffBar + kNumBars * 8;
    static constexpr int kSmemBytes = kOffMisc + 16 + 1024;
    static constexpr int kThreads = 384;
    static constexpr int kWarpS = 8;
    static constexpr int kWarpLoad = 9;
    static constexpr int kWarpStore = 10;
    static constexpr int kWarpPv = 11;
    static constexpr int kRegsSoftmax = 208;
    static constexpr int kRegsOther = 88;
    __device__ static constexpr uint32_t colS(int b) { return 128u * b; }
    __device__ static constexpr uint32_t colO(int t) { return 128u * kSBufs + D * t; }
    static_assert(128 * kSBufs + 2 * D <= 512, "TMEM budget");
};

// Registers per thread the kernel must be launched with for the setmaxnreg split above
// (2 x 128 x 208 + 128 x 88 = 384 x 168); the host checks it before the first launch.
constexpr int kPersistLaunchRegs = 168;

// One work item: query rows [row0, row0 + 256) of head bh.
struct PItem {
    int bh, row0, n0, n1;
};

template <bool CAUSAL>
__device__ __forceinline__ PItem persist_item(int it, const FwdParams& p) {
    PItem w;
    int ct;
    if (CAUSAL) {  // heaviest rows first
        ct = p.n_ctiles - 1 - it / p.BH;
        w.bh = it % p.BH;
    } else {  // a head's items together (its K and V stay in L2)
        w.bh = it / p.n_ctiles;
        ct = it % p.n_ctiles;
    }
    w.row0 = ct * 256;
    const int n_kv_all = (p.Nk + 127) / 128;
    auto tiles_for = [&](int r0) -> int {
        if (r0 >= p.Nq) return 0;
        if (!CAUSAL) return n_kv_all;
        const int last_key = min(r0 + 127, p.Nq - 1);
        return min(n_kv_all, last_key / 128 + 1);
    };
    w.n0 = tiles_for(w.row0);
    w.n1 = tiles_for(w.row0 + 128);
    return w;
}

// The k-th item of this CTA (snake order over rounds of gridDim.x items), or -1.
__device__ __forceinline__ int persist_item_index(int k, int n_items) {
    const int G = static_cast<int>(gridDim.x), c = static_cast<int>(blockIdx.x);
    const int it = k * G + ((k & 1) ? G - 1 - c : c);
    return it < n_items ? it : -1;
}

template <bool CAUSAL, bool BF16>
__global__ void __launch_bounds__(PersistCfg::kThreads, 1)
    attn_fwd_persist_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                            const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                            const FwdParams p) {
    using C = PersistCfg;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* smem = smem_raw + (base - raw);

    const uint32_t warp = threadIdx.x >> 5;
    const uint32_t lane = threadIdx.x & 31u;

    auto bar = [&](int i) -> uint32_t { return base + C::kOffBar + 8u * i; };
    auto sQ = [&](int buf, int t) -> uint32_t { return base + C::kOffQ + (buf * 2 + t) * C::kTileBytes; };
    auto sK = [&](int s) -> uint32_t { return base + C::kOffK + s * C::kTileBytes; };
    auto sV = [&](int s) -> uint32_t { return base + C::kOffV + s * C::kTileBytes; };
    uint32_t* misc = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);  // [0] tmem base, [1] abort

    const int n_items = p.n_ctiles * p.BH;
    WaitCtx wc{p.err, misc + 1, blockIdx.x};

    if (threadIdx.x == 0) {
        for (int i = 0; i < C::kNumBars; ++i) {
            uint32_t cnt = 1u;
            if (i >= C::kBarPFull && i < C::kBarPFull + C::kSBufs) cnt = 4u;  // one arrive per softmax warp
            if (i >= C::kBarOStaged && i < C::kBarOStaged + 4) cnt = 4u;  // o_staged
            mbar_init(bar(i), cnt);
        }
        misc[1] = 0u;
        fence_mbar_init();
    }
    if (warp == C::kWarpS) {
        tmem_alloc(smem_addr(misc), 512);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = misc[0];

    // Each warpgroup's branch starts with its register budget, so that the budget holds
    // for all of the code the branch runs.
    if (warp >= 8) {
        regs_decrease<C::kRegsOther>();
        if (warp == C::kWarpLoad) {
            // ================================ TMA loader ==================================
            if (lane == 0) {
                tma_prefetch_desc(&tmQ);
                tma_prefetch_desc(&tmK);
                tma_prefetch_desc(&tmV);
                const uint64_t pol_q = l2_policy_evict_first();
                const uint64_t pol_kv = l2_policy_evict_last();
                int G = 0;   // key tiles loaded so far (ring position)
                int aq = 0;  // items whose Q loads were issued
                bool ok = true;
                for (int it; ok && (it = persist_item_index(aq, n_items)) >= 0;) {
                    const PItem w = persist_item<CAUSAL>(it, p);
                    const int a = aq;
                    const int qb = a & 1;
                    for (int t = 0; t < 2 && ok && a >= 2; ++t)
                        ok = wait_one(bar(C::kBarQEmpty + qb * 2 + t), ((a >> 1) - 1) & 1, wc,
                                      kRoleLoad * 1000 + C::kBarQEmpty + qb * 2 + t, a);
                    if (!ok) break;
                    // Both Q tiles of the item (a tile past the last row loads nothing and
                    // completes its phase at once), so every buffer sees one phase per item.
                    for (int t = 0; t < 2; ++t) {
                        const int nt = t ? w.n1 : w.n0;
                        mbar_arrive_expect_tx(bar(C::kBarQFull + qb * 2 + t), nt > 0 ? C::kTileBytes : 0u);
                        if (nt > 0)
                            tma_load_3d_hint(sQ(qb, t), &tmQ, bar(C::kBarQFull + qb * 2 + t), 0, w.row0 + t * 128,
                                             w.bh, pol_q);
                    }
                    aq = a + 1;
                    const int nmax = max(w.n0, w.n1);
                    for (int j = 0; j < nmax && ok; ++j, ++G) {
                        const int s = G % C::kStages;
                        if (G >= C::kStages &&
                            !wait_one(bar(C::kBarKvEmpty + s), ((G / C::kStages) - 1) & 1, wc,
                                      kRoleLoad * 1000 + C::kBarKvEmpty + s, G)) {
                            ok = false;
                            break;
                        }
                        mbar_arrive_expect_tx(bar(C::kBarKFull + s), C::kTileBytes);
                        tma_load_3d_hint(sK(s), &tmK, bar(C::kBarKFull + s), 0, j * C::BN, w.bh, pol_kv);
                        mbar_arrive_expect_tx(bar(C::kBarVFull + s), C::kTileBytes);
                        tma_load_3d_hint(sV(s), &tmV, bar(C::kBarVFull + s), 0, j * C::BN, w.bh, pol_kv);
                    }
                }
                // Drain: every copy issued into shared memory has landed before exit.
                for (int aa = max(0, aq - 2); aa < aq; ++aa)
                    for (int t = 0; t < 2; ++t)
                        wait_one(bar(C::kBarQFull + (aa & 1) * 2 + t), (aa >> 1) & 1, wc, kRoleLoad * 1000 + 90 + t, aa,
                                 false);
                for (int gg = max(0, G - C::kStages); gg < G; ++gg) {
                    const int s = gg % C::kStages;
                    const uint32_t ph = (gg / C::kStages) & 1;
                    wait_one(bar(C::kBarKFull + s), ph, wc, kRoleLoad * 1000 + 80, gg, false);
                    wait_one(bar(C::kBarVFull + s), ph, wc, kRoleLoad * 1000 + 81, gg, false);
                }
            }
            __syncwarp();
        } else if (warp == C::kWarpS) {
            // ================================ S issuer ====================================
            constexpr uint32_t idesc_s = idesc_f16_f32acc(BF16, 128, 128, false);
            const uint64_t dk0 = sdesc_sw128(sK(0), 16, 1024);
            constexpr uint64_t kStageStep = C::kTileBytes >> 4;
            int g = 0;      // jobs issued so far
            int Gb = 0;     // ring position of the current item's first key tile
            uint32_t pend = 0;  // per S/P buffer: ring stage of the job in it | 0x80 if it was its tile's last reader
            bool ok = true;
            int a = 0;
            for (int it; ok && (it = persist_item_index(a, n_items)) >= 0; ++a) {
                const PItem w = persist_item<CAUSAL>(it, p);
                const int qb = a & 1;
                for (int t = 0; t < 2 && ok; ++t)
                    ok = wait_warp_sleep(bar(C::kBarQFull + qb * 2 + t), (a >> 1) & 1, wc,
                                   kRoleMma * 1000 + C::kBarQFull + qb * 2 + t, a);
                const JobOrder jobs{w.n0, w.n1};
                const int njobs = jobs.total();
                for (int jj = 0; jj < njobs && ok; ++jj, ++g) {
                    int t, j;
                    jobs.tile_of(jj, t, j);
                    const int Gt = Gb + j;
                    const int s = Gt % C::kStages;
                    const int b = g % C::kSBufs;
                    if (!wait_warp_sleep(bar(C::kBarKFull + s), (Gt / C::kStages) & 1, wc, kRoleMma * 1000 + C::kBarKFull + s,
                                   g)) {
                        ok = false;
                        break;
                    }
                    if (g >= C::kSBufs) {
                        // O += P V of job g-3 (same buffer) is complete: the buffer is free, and
                        // if that job was the last reader of its K/V tile, the stage is too.
                        if (!wait_warp_sleep(bar(C::kBarPvDone + b), ((g / C::kSBufs) - 1) & 1, wc,
                                       kRoleMma * 1000 + C::kBarPvDone + b, g)) {
                            ok = false;
                            break;
                        }
                        const uint32_t info = (pend >> (8 * b)) & 0xffu;
                        if ((info & 0x80u) && lane == 0) mbar_arrive(bar(C::kBarKvEmpty + (info & 7u)));
                    }
                    tc_fence_after_sync();
                    const uint64_t a0 = sdesc_sw128(sQ(qb, t), 16, 1024);
                    mma_qk64_warp(tmem + C::colS(b), a0, dk0 + s * kStageStep, idesc_s, 0u);
                    mma_commit_warp(bar(C::kBarSFull + t * C::kSBufs + b));
                    const uint32_t info = static_cast<uint32_t>(s) | (jj == jobs.last_job(j) ? 0x80u : 0u);
                    pend = (pend & ~(0xffu << (8 * b))) | (info << (8 * b));
                }
                Gb += max(w.n0, w.n1);
            }
            // Drain: the last O += P V groups have completed (every S before them has too).
            for (int r = max(0, g - C::kSBufs); r < g && ok; ++r)
                ok = wait_warp_sleep(bar(C::kBarPvDone + r % C::kSBufs), (r / C::kSBufs) & 1, wc,
                               kRoleMma * 1000 + C::kBarPvDone + r % C::kSBufs, r);
            mma_commit_warp(bar(C::kBarDrain + 0));
            wait_warp_sleep(bar(C::kBarDrain + 0), 0, wc, kRoleMma * 1000 + C::kBarDrain, 0, false);
            __syncwarp();
        } else if (warp == C::kWarpStore) {
            // ================================ O store =====================================
            // Per item and Q tile: wait for the softmax warpgroup's staging tile, store it,
            // and once the store has read it, hand the Q buffer back to the loader.
            // o_staged is per Q buffer and tile: a warpgroup stages into a buffer again
            // only after the loader reloaded it, i.e. after this warp stored the previous
            // output from it, so no o_staged barrier completes a phase ahead of its wait.
            int a = 0;
            uint32_t staged = 0;  // parity per (buffer, tile) of the o_staged phases seen
            bool ok = true;
            for (int it; (it = persist_item_index(a, n_items)) >= 0; ++a) {
                const PItem w = persist_item<CAUSAL>(it, p);
                const int qb = a & 1;
#pragma unroll
                for (int t = 0; t < 2; ++t) {
                    const int nt = t ? w.n1 : w.n0;
                    if (nt > 0) {
                        const int sb = qb * 2 + t;
                        if (ok)
                            ok = wait_warp(bar(C::kBarOStaged + sb), (staged >> sb) & 1u, wc,
                                           kRoleLoad * 1000 + C::kBarOStaged + sb, a);
                        staged ^= 1u << sb;
                        if (ok && lane == 0) {
                            tma_store_3d(&tmO, sQ(qb, t), 0, w.row0 + t * 128, w.bh);
                            tma_store_commit();
                            tma_store_wait_read_all();
                        }
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar(C::kBarQEmpty + qb * 2 + t));
                }
            }
            if (lane == 0) tma_store_wait_all();
            __syncwarp();
        } else if (warp == C::kWarpPv) {
            // ================================ P V issuer ==================================
            {
                constexpr uint32_t idesc_o = idesc_f16_f32acc(BF16, 128, C::D, true);
                const uint64_t dv0 = sdesc_sw128(sV(0), C::kTileBytes, 1024);
                constexpr uint64_t kStageStep = C::kTileBytes >> 4;
                int g = 0, Gb = 0;
                int kk0 = 0, kk1 = 0;  // O += P V issued per Q tile
                bool ok = true;
                int a = 0;
                for (int it; ok && (it = persist_item_index(a, n_items)) >= 0; ++a) {
                    const PItem w = persist_item<CAUSAL>(it, p);
                    const JobOrder jobs{w.n0, w.n1};
                    const int njobs = jobs.total();
                    for (int jj = 0; jj < njobs && ok; ++jj, ++g) {
                        int t, j;
                        jobs.tile_of(jj, t, j);
                        const int b = g % C::kSBufs;
                        const int Gt = Gb + j;
                        const int s = Gt % C::kStages;
                        // p_full: one phase per job in this buffer, awaited in job order; the
                        // next one needs S(g+3) in the buffer, which waits for this O += P V.
                        // The first O += P V of an item (it overwrites O) also needs the
                        // previous item's O read out: the softmax warpgroup reads it (and
                        // waits for the loads) before it writes the item's first P, so
                        // p_full implies it.
                        if (!wait_warp_sleep(bar(C::kBarPFull + b), (g / C::kSBufs) & 1, wc, kRoleMma * 1000 + C::kBarPFull + b,
                                       g) ||
                            !wait_warp_sleep(bar(C::kBarVFull + s), (Gt / C::kStages) & 1, wc,
                                       kRoleMma * 1000 + C::kBarVFull + s, g)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after_sync();
                        int& kk = t ? kk1 : kk0;
                        mma_pv128_warp(tmem + C::colO(t), tmem + C::colS(b), dv0 + s * kStageStep, idesc_o,
                                       j > 0 ? 1u : 0u);
                        mma_commit_warp(bar(C::kBarODone + t * 2 + (kk & 1)));  // before pv_done
                        mma_commit_warp(bar(C::kBarPvDone + b));
                        ++kk;
                    }
                    Gb += max(w.n0, w.n1);
                }
                mma_commit_warp(bar(C::kBarDrain + 1));
                wait_warp_sleep(bar(C::kBarDrain + 1), 0, wc, kRoleMma * 1000 + C::kBarDrain + 1, 0, false);
            }
            __syncwarp();
        }
    } else {
        regs_increase<C::kRegsSoftmax>();
        // ================================ softmax warpgroups ==========================
        const int t = static_cast<int>(warp >> 2);
        const uint32_t wq = warp & 3u;       // TMEM lane quarter of this warp
        const uint32_t r = wq * 32u + lane;  // row inside the Q tile = TMEM lane
        const uint32_t role = t == 0 ? kRoleSoftmax0 : kRoleSoftmax1;
        const uint32_t lane_base = tmem_addr(tmem, wq * 32u, 0);
        const uint32_t tO = lane_base + C::colO(t);
        const float qk = p.qk_scale;
        const float2 qk2 = make_float2(qk, qk);

        bool ok = true;
        int kk = 0;          // O_t += P V issued so far (all items)
        uint32_t sp = 0;     // parity per S/P buffer of this tile's s_full barriers
        int g0 = 0, Gb = 0;  // first job / first ring position of the current item
        int a = 0;
        for (int it; (it = persist_item_index(a, n_items)) >= 0; ++a) {
            const PItem w = persist_item<CAUSAL>(it, p);
            const JobOrder jobs{w.n0, w.n1};
            const int nt = t ? w.n1 : w.n0;
            const int row0 = w.row0 + t * 128;
            const int q_row = row0 + static_cast<int>(r);
            const bool warp_has_rows = row0 + static_cast<int>(wq * 32u) < p.Nq;
            const int qb = a & 1;
            float m = -INFINITY;  // running max, log2 units (possibly stale)
            float l = 0.f;        // running sum of P (fp32), relative to m: the LSE
            float lc = 0.f;       // rounding of each tile's largest P, relative to m: O / (l + lc)
            for (int j = 0; j < nt; ++j) {
                const int g = g0 + jobs.job(t, j);
                const int b = g % C::kSBufs;
                const uint32_t tS = lane_base + C::colS(b);
                const uint32_t par = (sp >> b) & 1u;
                sp ^= 1u << b;
                if (ok)
                    ok = wait_warp(bar(C::kBarSFull + t * C::kSBufs + b), par, wc,
                                   role * 1000 + C::kBarSFull + t * C::kSBufs + b, g);
                bool rescale = false;
                float alpha = 1.f;
                if (ok && warp_has_rows) {
                    tc_fence_after_sync();
                    uint32_t sr[4][32];
#pragma unroll
                    for (int c = 0; c < 4; ++c) tmem_ld32(tS + c * 32, sr[c]);
                    tmem_ld_wait();
#pragma unroll
                    for (int c = 0; c < 4; ++c) reg_fence(sr[c]);
                    const int k0 = j * C::BN;
                    const bool need_mask = (k0 + C::BN > p.Nk) || (CAUSAL && k0 + C::BN - 1 > row0);
                    if (need_mask) {
                        const int lim = CAUSAL ? min(p.Nk, q_row + 1) : p.Nk;
#pragma unroll
                        for (int c = 0; c < 4; ++c)
#pragma unroll
                            for (int e = 0; e < 32; ++e)
                                if (k0 + c * 32 + e >= lim) sr[c][e] = __float_as_uint(-INFINITY);
                    }
                    const float row_max = row_max128(sr);
                    float m_new = fmaxf(m, row_max * qk);
                    if (m_new - m <= kRescaleTau) m_new = m;
                    const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
                    alpha = (m == m_use) ? 1.f : ex2_ftz(m - m_use);
                    // whether any row of the warp rescales O: decided here, off the P hand-off
                    rescale = j > 0 && __any_sync(0xffffffffu, alpha != 1.f);
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
                    m = m_new;
                }
                // Rescale O_t once O_t += P V of this tile's previous job has completed
                // (every earlier one has: see the parity argument at the o_done waits).
                if (rescale && ok)
                    ok = wait_warp(bar(C::kBarODone + t * 2 + ((kk - 1) & 1)), ((kk - 1) >> 1) & 1, wc,
                                   role * 1000 + C::kBarODone + t * 2, j);
                if (rescale && ok) {
                    tc_fence_after_sync();
                    const float2 a2 = make_float2(alpha, alpha);
#pragma unroll
                    for (int c = 0; c < C::D / 32; ++c) {
                        uint32_t o[32];
                        tmem_ld32(tO + c * 32, o);
                        tmem_ld_wait();
                        reg_fence(o);
#pragma unroll
                        for (int e = 0; e < 32; e += 2) {
                            const float2 v =
                                __fmul2_rn(make_float2(__uint_as_float(o[e]), __uint_as_float(o[e + 1])), a2);
                            o[e] = __float_as_uint(v.x);
                            o[e + 1] = __float_as_uint(v.y);
                        }
                        tmem_st32(tO + c * 32, o);
                    }
                    tmem_st_wait();
                }
                // P of this warp's rows is in TMEM (wait::st above) and ordered before
                // the arrive; the P V issuer waits for all four warps.
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0 && ok) mbar_arrive(bar(C::kBarPFull + b));
                ++kk;
            }

            // ---- epilogue of this item's Q tile ------------------------------------------
            if (nt > 0) {
                // Wait for the last two O_t += P V in order: when the previous one has
                // completed, so has every earlier one (one issuing thread), and the last
                // one's parity wait is exact.
                if (ok && kk >= 2)
                    ok = wait_warp(bar(C::kBarODone + t * 2 + ((kk - 2) & 1)), ((kk - 2) >> 1) & 1, wc,
                                   role * 1000 + C::kBarODone + t * 2, kk);
                if (ok)
                    ok = wait_warp(bar(C::kBarODone + t * 2 + ((kk - 1) & 1)), ((kk - 1) >> 1) & 1, wc,
                                   role * 1000 + C::kBarODone + t * 2 + 1, kk);
                const float m_fin = (m == -INFINITY) ? 0.f : m;
                const float inv_l = l > 0.f ? 1.f / (l + lc) : 0.f;
                const float lse2 = l > 0.f ? m_fin + log2f(l) : -INFINITY;
                if (ok && warp_has_rows) {
                    tc_fence_after_sync();
                    uint8_t* stage = smem + C::kOffQ + (qb * 2 + t) * C::kTileBytes;
#pragma unroll
                    for (int c = 0; c < C::D / 32; ++c) {
                        uint32_t o[32];
                        tmem_ld32(tO + c * 32, o);
                        tmem_ld_wait();
                        reg_fence(o);
                        uint32_t h[16];
#pragma unroll
                        for (int e = 0; e < 16; ++e)
                            h[e] = pack2<BF16>(__uint_as_float(o[2 * e]) * inv_l,
                                               __uint_as_float(o[2 * e + 1]) * inv_l);
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const uint32_t chunk = (c & 1) * 4 + i;
                            *reinterpret_cast<uint4*>(stage + sw128_offset(r, chunk)) =
                                make_uint4(h[4 * i], h[4 * i + 1], h[4 * i + 2], h[4 * i + 3]);
                        }
                    }
                    if (q_row < p.Nq) p.lse[static_cast<size_t>(w.bh) * p.Nq + q_row] = lse2 * 0.69314718055994530942f;
                }
                fence_proxy_async_smem();
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0 && ok) mbar_arrive(bar(C::kBarOStaged + qb * 2 + t));  // ready to store
            }
            g0 += jobs.total();
            Gb += max(w.n0, w.n1);
        }
        __syncwarp();
    }

    tc_fence_before_sync();
    __syncthreads();
    if (warp == C::kWarpS) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, 512);
    }
}

}  // namespace attn_sm103
