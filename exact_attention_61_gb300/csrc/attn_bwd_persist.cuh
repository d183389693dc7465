// Persistent attention backward for head dimension 64 (no padding or window masks): one
// CTA per SM claims work items, each one 128-key tile of one head, from a list in the
// one-item kernel's CTA order, so that an item's dK/dV epilogue and the last dQ reduce
// overlap the next item's K/V load, its copy into tensor memory and its first S^T/dP^T.
// Causal items are claimed from a counter in global memory (zeroed by the prologue
// kernel), in list order, each by whichever CTA asks first: they differ in length (a key
// tile sees from 1 to all Q tiles), and a static assignment left some SMs 15 % more work
// than the average. Non-causal items are all alike and go round-robin (item k of CTA c is
// c + k * gridDim.x). The loader picks the next item once the current one's copies are
// issued, and passes each item to the other roles through a ring of four slots in shared
// memory, written before the loader's arrive on the K/V barrier of that item; an item
// past the list is passed on as -1 and ends every role.
//
// Per item it computes what attn_bwd_kernel computes at d = 64, with the same arithmetic
// in the same order (the dQ accumulator receives the same tiles; only the order in which
// the CTAs add them differs, as between any two launches): the FlashAttention-2 backward
// that "如何用 profiler 逐步优化 Triton FlashAttention-2 kernel" ("Future articles") names,
// from the L the forward writes ("Round 4 / exp2"). The roles:
//  - warps 0-7: two compute warpgroups, one per 64-query half of each Q tile;
//  - warps 8-11: read each dQ tile out and add it to the fp32 accumulator by TMA
//    reduce-add;
//  - warp 12 issues the MMAs and, at the start of each item, the copies of K and V into
//    TMEM (tcgen05.cp); warp 13 drives TMA.
// Every barrier that paces Q tiles counts the CTA's Q tiles over all its items; the ones
// that pace items (K/V landed, item read by the dQ warps, dK/dV final, dK/dV read out)
// count items.
// Across an item boundary:
//  - the loader reloads K and V (shared memory) once every MMA of the previous item is
//    done (kBarAcc), since the last dQ products read K there and V shares the second dS
//    buffer;
//  - once they land, the MMA warp copies them into TMEM (the previous item's S^T/dP^T,
//    which read the old copies, are done too) and issues the new item's first S^T/dP^T
//    behind the copies; the compute warpgroups write dS over V's shared memory only after
//    those S^T/dP^T completed, and so after the copy of V;
//  - the MMA warp issues the item's first dV/dK (which overwrite the accumulators) only
//    after the compute warpgroups have read the previous item's dV and dK out
//    (kBarAccFree).
// Every wait is bounded as in the other kernels.
#pragma once

#include "attn_bwd_kernel.cuh"

namespace attn_sm103 {

// Work item x of the list (the one-item kernel's CTA order): key tile kt of head bh.
template <bool CAUSAL>
__device__ __forceinline__ void bwd_persist_item(int x, const BwdParams& p, int& bh, int& kt) {
    const int n_kt = p.n_ktiles;
    if (CAUSAL) {
        const int grp = x / (kBwdHeadGroup * n_kt);
        const int gh = min(kBwdHeadGroup, p.BH - grp * kBwdHeadGroup);
        const int idx = x - grp * kBwdHeadGroup * n_kt;
        kt = idx / gh;
        bh = grp * kBwdHeadGroup + idx % gh;
    } else {
        bh = x / n_kt;
        kt = x % n_kt;
    }
}

template <bool CAUSAL, bool BF16>
__global__ void __launch_bounds__(BwdCfg<64>::kThreads, 1)
    attn_bwd_persist_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                            const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
                            const __grid_constant__ CUtensorMap tmDQ, const BwdParams p) {
    using C = BwdCfg<64>;
    constexpr int D = 64;
    static_assert(C::kEarlyNext && C::kKvTmem, "the persistent kernel is the d = 64 form");
    extern __shared__ __align__(1024) uint8_t smem_bwd[];
    const uint32_t base = smem_addr(smem_bwd);
    if (base & 1023u) {  // uniform over the CTA: nothing has been set up yet
        if (threadIdx.x == 0) {
            if (atomicCAS(p.err, 0u, kErrSmemAlign) == 0u) p.err[1] = blockIdx.x;
        }
        return;
    }
    const uint32_t warp = threadIdx.x >> 5;
    const uint32_t lane = threadIdx.x & 31u;
    auto bar = [&](int i) -> uint32_t { return base + C::kOffBar + 8u * i; };
    auto sQ = [&](int s) -> uint32_t { return base + C::kOffStage + s * C::kStageBytes; };
    auto sDO = [&](int s) -> uint32_t { return sQ(s) + C::kTileBytes; };
    uint32_t* misc = reinterpret_cast<uint32_t*>(smem_bwd + C::kOffMisc);  // [0] tmem, [1] abort

    volatile int* items = reinterpret_cast<volatile int*>(misc + 4);  // claimed items, ring of 4
    const int n_items = p.BH * p.n_ktiles;
    const int n_qt = p.Npad / 128;
    // Q tiles of key tile kt: all of them, or from the diagonal on under the causal mask.
    auto q_begin = [&](int kt) { return CAUSAL ? min(n_qt, kt) : 0; };
    WaitCtx wc{p.err, misc + 1, blockIdx.x};

    if (threadIdx.x == 0) {
        for (int i = 0; i < C::kNumBars; ++i) {
            uint32_t count = 1;
            if (i >= C::kBarQdEmpty && i < C::kBarQdEmpty + C::kStages) count = 1 + 8 + 1;  // MMA, compute, dQ store
            if (i == C::kBarPds || i == C::kBarPds + 1) count = 4;                         // a compute warpgroup
            if (i == C::kBarDqRead || i == C::kBarDqItem) count = 4;                          // dQ warps
            if (i == C::kBarAccFree) count = 8;                                            // compute warps
            mbar_init(bar(i), count);
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
            tma_prefetch_desc(&tmDO);
            const uint64_t pol_kv = l2_policy_evict_first();  // read by this item only
            const uint64_t pol_q = l2_policy_evict_last();    // read by every key tile of the head
            bool ok = true;
            int gi = 0;        // Q tiles loaded so far (all items)
            int k = 0;         // items started
            int last_kv = -1;  // item whose K/V copy may still be in flight
            // Non-causal items are all alike: item k of the CTA is blockIdx.x + k * gridDim.x.
            // Causal items are claimed from the counter.
            int n_claims = 0;
            auto claim = [&]() -> int {
                const int x = CAUSAL ? atomicAdd(p.item_counter, 1)
                                     : static_cast<int>(blockIdx.x) + n_claims * static_cast<int>(gridDim.x);
                ++n_claims;
                return x < n_items ? x : -1;
            };
            int x_next = claim();
            for (;; ++k) {
                const int x = x_next;
                items[k & 3] = x;
                // Before the K/V barrier's next phase, every role has passed its wait on the
                // previous one: the MMA and compute warps, since every MMA of the previous item
                // is done (kBarAcc); the dQ warps by their own arrive (with one-tile items the
                // MMAs can finish while the dQ warps are still on the item before). Then no
                // role's parity wait can fall two phases behind.
                if (k > 0 && !wait_one(bar(C::kBarDqItem), (k - 1) & 1, wc, kRoleBwdLoad * 1000 + 93, k)) break;
                if (x < 0) {
                    // No more items: complete the K/V barrier's next phase with no bytes so that
                    // the other roles read the -1. As for an item, only once every MMA of the
                    // previous item is done (its copy has landed).
                    if (k > 0 && !wait_one(bar(C::kBarAcc), (k - 1) & 1, wc, kRoleBwdLoad * 1000 + 92, k)) break;
                    last_kv = -1;
                    mbar_arrive(bar(C::kBarKV));
                    break;
                }
                int bh, kt;
                bwd_persist_item<CAUSAL>(x, p, bh, kt);
                const int qt0 = q_begin(kt);
                const int n_it = n_qt - qt0;
                // K and V of the item, once every MMA of the previous one is done (which also
                // means the previous item's K/V copy landed).
                if (k > 0 && !wait_one(bar(C::kBarAcc), (k - 1) & 1, wc, kRoleBwdLoad * 1000 + C::kBarAcc, k)) break;
                mbar_arrive_expect_tx(bar(C::kBarKV), 2 * C::kTileBytes);
                tma_load_3d_hint(base + C::kOffK, &tmK, bar(C::kBarKV), 0, kt * 128, bh, pol_kv);
                tma_load_3d_hint(base + C::kOffV, &tmV, bar(C::kBarKV), 0, kt * 128, bh, pol_kv);
                last_kv = k;
                for (int it = 0; it < n_it; ++it, ++gi) {
                    const int s = gi % C::kStages;
                    if (gi >= C::kStages &&
                        !wait_one(bar(C::kBarQdEmpty + s), ((gi / C::kStages) - 1) & 1, wc,
                                  kRoleBwdLoad * 1000 + C::kBarQdEmpty + s, gi)) {
                        ok = false;
                        break;
                    }
                    const int q0 = (qt0 + it) * 128;
                    const uint32_t fb = bar(C::kBarQdFull + s);
                    mbar_arrive_expect_tx(fb, 2 * C::kTileBytes + C::kVecBytes);
                    tma_load_3d_hint(sQ(s), &tmQ, fb, 0, q0, bh, pol_q);
                    tma_load_3d_hint(sDO(s), &tmDO, fb, 0, q0, bh, pol_q);
                    const size_t vrow = static_cast<size_t>(bh) * p.Npad + q0;
                    const uint32_t vdst = base + C::kOffVec + s * C::kVecBytes;
                    bulk_load(vdst, p.lse2 + vrow, 512, fb);
                    bulk_load(vdst + 512, p.dvec + vrow, 512, fb);
                }
                if (!ok) break;
                // The next item, claimed once this one's copies are issued (the claim's latency
                // then overlaps them). Prefetching its K and V into L2 here was measured slower.
                x_next = claim();
            }
            // Drain: every copy into this CTA's shared memory has landed before it exits.
            if (last_kv >= 0) wait_one(bar(C::kBarKV), last_kv & 1, wc, kRoleBwdLoad * 1000 + 90, last_kv, false);
            for (int jj = max(0, gi - C::kStages); jj < gi; ++jj)
                wait_one(bar(C::kBarQdFull + jj % C::kStages), (jj / C::kStages) & 1, wc, kRoleBwdLoad * 1000 + 91, jj,
                         false);
        }
        __syncwarp();
    } else if (warp == C::kWarpMma) {
        // ================================ MMA issuer ==================================
        constexpr uint32_t idesc_h = idesc_f16_f32acc(BF16, 128, 64, false);         // S^T/dP^T half: N = 64
        constexpr uint32_t idesc_o = idesc_f16_f32acc(BF16, 128, D, true);           // TMEM x MN-major
        constexpr uint32_t idesc_q = idesc_f16_f32acc_ab(BF16, 128, D, true, true);  // MN x MN
        const uint64_t dK_mn = sdesc_sw128(base + C::kOffK, C::kBoxBytes, 1024);      // K as B, MN-major
        const uint64_t dDS = sdesc_sw128(base + C::kOffDS, C::kBoxBytes, 1024);       // dS as A, MN-major
        constexpr uint64_t kStageStep = C::kStageBytes >> 4;
        constexpr uint64_t kTileStep = C::kTileBytes >> 4;
        constexpr uint64_t kHalfRows = (64 * 128) >> 4;  // 64 rows of a 128-byte-swizzled box
        const uint64_t dQ_k0 = sdesc_sw128(sQ(0), 16, 1024);
        const uint64_t dQ_mn0 = sdesc_sw128(sQ(0), C::kBoxBytes, 1024);

        // S^T/dP^T of half h of Q tile gi (global count): K and V from TMEM, Q and dO
        // K-major from the tile's stage; commit to the half's barrier.
        auto issue_sdp_half = [&](int gi, int h) -> bool {
            const int si = gi % C::kStages;
            if (h == 0 && !wait_warp_sleep(bar(C::kBarQdFull + si), (gi / C::kStages) & 1, wc,
                                           kRoleBwdMma * 1000 + C::kBarQdFull + si, gi))
                return false;
            tc_fence_after_sync();
            const uint64_t q_k = dQ_k0 + si * kStageStep + h * kHalfRows;
            mma_ts_k64_warp(tmem + C::colS + 64u * h, tmem + C::colK, q_k, idesc_h);
            mma_ts_k64_warp(tmem + C::colDP + 64u * h, tmem + C::colV, q_k + kTileStep, idesc_h);
            mma_commit_warp(bar(C::kBarSdp + h));
            return true;
        };

        const uint64_t dK_cp = sdesc_sw128(base + C::kOffK, 16, 1024);  // K, V as K-major copy sources
        const uint64_t dV_cp = sdesc_sw128(base + C::kOffV, 16, 1024);
        bool ok = true;
        int gi = 0;  // Q tiles issued so far (all items)
        for (int k = 0; ok; ++k) {
            ok = wait_warp_sleep(bar(C::kBarKV), k & 1, wc, kRoleBwdMma * 1000 + C::kBarKV, k);
            if (!ok) break;
            const int x = items[k & 3];
            if (x < 0) break;
            int bh, kt;
            bwd_persist_item<CAUSAL>(x, p, bh, kt);
            const int n_it = n_qt - q_begin(kt);
            tc_fence_after_sync();
            // K and V into TMEM, the A operands of S^T and dP^T. The previous item's MMAs,
            // which read the old copies, are complete: the loader reloaded K and V only
            // after its kBarAcc.
            tmem_cp_tile64_warp(tmem + C::colK, dK_cp);
            tmem_cp_tile64_warp(tmem + C::colV, dV_cp);
            ok = issue_sdp_half(gi, 0) && issue_sdp_half(gi, 1);
            for (int it = 0; it < n_it && ok; ++it, ++gi) {
                const int s = gi % C::kStages;
                const uint64_t q_mn = dQ_mn0 + s * kStageStep;
                const uint64_t do_mn = q_mn + kTileStep;
                for (int h = 0; h < 2 && ok; ++h) {
                    ok = wait_warp_sleep(bar(C::kBarPds + h), gi & 1, wc, kRoleBwdMma * 1000 + C::kBarPds + h, gi);
                    // The item's first dV/dK overwrite the accumulators: the previous item's
                    // must have been read out.
                    if (ok && it == 0 && h == 0 && k > 0)
                        ok = wait_warp_sleep(bar(C::kBarAccFree), (k - 1) & 1, wc, kRoleBwdMma * 1000 + C::kBarAccFree,
                                             k);
                    if (!ok) break;
                    tc_fence_after_sync();
                    const uint32_t acc = (it > 0 || h > 0) ? 1u : 0u;
                    mma_pv64_tmem_warp(tmem + C::colDV, tmem + C::colS + 64u * h, do_mn + h * kHalfRows, idesc_o, acc);
                    mma_pv64_tmem_warp(tmem + C::colDK, tmem + C::colDP + 64u * h, q_mn + h * kHalfRows, idesc_o, acc);
                    if (it + 1 < n_it) ok = issue_sdp_half(gi + 1, h);
                }
                // The dQ columns of the previous Q tile must have been read out.
                if (ok && gi > 0)
                    ok = wait_warp_sleep(bar(C::kBarDqRead), (gi - 1) & 1, wc, kRoleBwdMma * 1000 + C::kBarDqRead, gi);
                if (!ok) break;
                tc_fence_after_sync();
                mma_mn128_warp(tmem + C::colDQ, dDS + (((gi & 1) * (128 * 128 * 2)) >> 4), dK_mn, idesc_q, 0u);
                mma_commit_warp(bar(C::kBarDqFull));
                mma_commit_warp(bar(C::kBarQdEmpty + s));
            }
            if (ok) mma_commit_warp(bar(C::kBarAcc));  // dK, dV final; K, V free
        }
        // Drain: all MMAs issued by this warp are complete before TMEM is freed.
        mma_commit_warp(bar(C::kBarDrain));
        wait_warp(bar(C::kBarDrain), 0, wc, kRoleBwdMma * 1000 + C::kBarDrain, 0, false);
        __syncwarp();
    } else if (warp >= C::kWarpDq) {
        // ================================ dQ read-out and reduce ======================
        const uint32_t wq = warp - C::kWarpDq;
        const uint32_t r = wq * 32u + lane;
        const uint32_t lane_base = tmem_addr(tmem, wq * 32u, 0);
        const bool leader = warp == C::kWarpDq && lane == 0;
        if (leader) tma_prefetch_desc(&tmDQ);
        bool ok = true;
        int gi = 0;
        for (int k = 0; ok; ++k) {
            ok = wait_warp_sleep(bar(C::kBarKV), k & 1, wc, kRoleBwdDq * 1000 + C::kBarKV, k);
            if (!ok) break;
            const int x = items[k & 3];
            if (x < 0) break;  // no more items
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(C::kBarDqItem));
            int bh, kt;
            bwd_persist_item<CAUSAL>(x, p, bh, kt);
            const int qt0 = q_begin(kt);
            const int n_it = n_qt - qt0;
            for (int it = 0; it < n_it; ++it, ++gi) {
                if (!wait_warp_sleep(bar(C::kBarDqFull), gi & 1, wc, kRoleBwdDq * 1000 + C::kBarDqFull, gi)) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                const int q0 = (qt0 + it) * 128;
                const int s = gi % C::kStages;
                const uint32_t stage = sQ(s);
#pragma unroll 1
                for (int b = 0; b < D / 32; ++b) {
                    uint32_t o[32];
                    tmem_ld32(lane_base + C::colDQ + 32 * b, o);
                    tmem_ld_wait();
                    reg_fence(o);
                    const uint32_t row = stage + b * C::kDqBoxBytes + r * 128u;
#pragma unroll
                    for (int ch = 0; ch < 8; ++ch)
                        st_shared_v4(row + ((ch ^ (r & 7u)) << 4), o[4 * ch], o[4 * ch + 1], o[4 * ch + 2], o[4 * ch + 3]);
                }
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(C::kBarDqRead));  // the dQ columns are free
                fence_proxy_async_smem();
                named_bar_sync(1, 128);
                if (leader) {
                    if (*wc.abort == 0u) {
#pragma unroll 1
                        for (int b = 0; b < D / 32; ++b)
                            tma_reduce_add_3d(&tmDQ, stage + b * C::kDqBoxBytes, 32 * b, q0, bh);
                        tma_store_commit();
                    }
                    // The stage goes back to the loader once the reduce has read it.
                    tma_store_wait_read_all();
                    mbar_arrive(bar(C::kBarQdEmpty + s));
                }
            }
        }
        // Every reduce is complete in global memory before the CTA exits.
        if (leader) tma_store_wait_all();
    } else {
        // ================================ compute warpgroups ==========================
        // Warpgroup h handles query columns [64h, 64h + 64) of S^T and dP^T.
        const uint32_t h = warp >> 2;
        const uint32_t wq = warp & 3u;       // TMEM lane quarter
        const uint32_t r = wq * 32u + lane;  // key row in the tile = TMEM lane
        const uint32_t lane_base = tmem_addr(tmem, wq * 32u, 0);
        const float qk = p.qk_scale;
        const float2 qk2 = make_float2(qk, qk);
        const uint32_t sDS0 = base + C::kOffDS + h * C::kBoxBytes + r * 128u;
        bool ok = true;
        int gi = 0;
        for (int k = 0; ok; ++k) {
            // the item (or the -1 that ends the list), written before the K/V barrier's arrive
            ok = wait_warp_sleep(bar(C::kBarKV), k & 1, wc, kRoleBwdCompute * 1000 + C::kBarKV, k);
            if (!ok) break;
            const int x = items[k & 3];
            if (x < 0) break;
            int bh, kt;
            bwd_persist_item<CAUSAL>(x, p, bh, kt);
            const int qt0 = q_begin(kt);
            const int n_it = n_qt - qt0;
            const int j = kt * 128 + static_cast<int>(r);  // this thread's key
            const bool key_out = j >= p.Nk;                // past Nk: P = 0
            for (int it = 0; it < n_it && ok; ++it, ++gi) {
                const int s = gi % C::kStages;
                const int q0 = (qt0 + it) * 128;
                if (!wait_warp_sleep(bar(C::kBarQdFull + s), (gi / C::kStages) & 1, wc,
                                     kRoleBwdCompute * 1000 + C::kBarQdFull + s, gi) ||
                    !wait_warp_sleep(bar(C::kBarSdp + h), gi & 1, wc, kRoleBwdCompute * 1000 + C::kBarSdp + h, gi)) {
                    ok = false;
                    break;
                }
                // S^T/dP^T of this half complete also means the dQ product that last read
                // this Q tile's dS buffer (two tiles back; issued before them) is done.
                tc_fence_after_sync();
                const uint32_t sDS = sDS0 + (gi & 1) * (128 * 128 * 2);
                const float* vec = reinterpret_cast<const float*>(smem_bwd + C::kOffVec + s * C::kVecBytes);
                const float* nlse2 = vec + 64 * h;        // -LSE log2(e) of this half's query rows
                const float* ndvec = vec + 128 + 64 * h;  // -D
                // Whether some query row of this tile may not see this thread's key.
                const bool mask_tile = key_out || (CAUSAL && j > q0);
#pragma unroll 1
                for (int c = 0; c < 2; ++c) {
                    const uint32_t col32 = 64u * h + 32u * c;  // first fp32 column of this chunk
                    uint32_t sr[32], dr[32];
                    tmem_ld32(lane_base + C::colS + col32, sr);
                    tmem_ld32(lane_base + C::colDP + col32, dr);
                    tmem_ld_wait();
                    reg_fence(sr);
                    reg_fence(dr);
                    uint32_t pk[16], dk[16];
#pragma unroll
                    for (int e = 0; e < 32; e += 4) {
                        const int col = 32 * c + e;  // within this half
                        // -LSE log2(e) and -D of four query rows (the prologue stores them negated)
                        const float4 nl = *reinterpret_cast<const float4*>(nlse2 + col);
                        const float4 nd = *reinterpret_cast<const float4*>(ndvec + col);
                        const float2 y0 = __ffma2_rn(make_float2(__uint_as_float(sr[e]), __uint_as_float(sr[e + 1])),
                                                     qk2, make_float2(nl.x, nl.y));
                        const float2 y1 = __ffma2_rn(
                            make_float2(__uint_as_float(sr[e + 2]), __uint_as_float(sr[e + 3])), qk2,
                            make_float2(nl.z, nl.w));
                        float pe[4] = {ex2_ftz(y0.x), ex2_ftz(y0.y), ex2_ftz(y1.x), ex2_ftz(y1.y)};
                        if (mask_tile) {
                            const int q = q0 + 64 * static_cast<int>(h) + col;  // query row of pe[0]
#pragma unroll
                            for (int kk = 0; kk < 4; ++kk)
                                if (key_out || (CAUSAL && j > q + kk)) pe[kk] = 0.f;
                        }
                        const float2 p0 = make_float2(pe[0], pe[1]), p1 = make_float2(pe[2], pe[3]);
                        const float2 ds0 = __fmul2_rn(
                            p0, __fadd2_rn(make_float2(__uint_as_float(dr[e]), __uint_as_float(dr[e + 1])),
                                           make_float2(nd.x, nd.y)));
                        const float2 ds1 = __fmul2_rn(
                            p1, __fadd2_rn(make_float2(__uint_as_float(dr[e + 2]), __uint_as_float(dr[e + 3])),
                                           make_float2(nd.z, nd.w)));
                        pk[e >> 1] = pack2<BF16>(p0.x, p0.y);
                        pk[(e >> 1) + 1] = pack2<BF16>(p1.x, p1.y);
                        dk[e >> 1] = pack2<BF16>(ds0.x, ds0.y);
                        dk[(e >> 1) + 1] = pack2<BF16>(ds1.x, ds1.y);
                    }
                    // 16-bit P^T / dS^T packed in place: half h lives in columns
                    // [64h, 64h + 32), chunk c in its 16 columns (already read above).
                    tmem_st16(lane_base + C::colS + 64u * h + 16u * c, pk);
                    tmem_st16(lane_base + C::colDP + 64u * h + 16u * c, dk);
                    // dS for the dQ product: element (query m, key r) of an MN-major operand,
                    // 128-byte swizzle; half h is box h, chunk c its 16-byte chunks 4c..4c+3.
#pragma unroll
                    for (int t = 0; t < 4; ++t) {
                        const uint32_t chunk = 4u * c + t;
                        st_shared_v4(sDS + ((chunk ^ (r & 7u)) << 4), dk[4 * t], dk[4 * t + 1], dk[4 * t + 2],
                                     dk[4 * t + 3]);
                    }
                }
                tmem_st_wait();
                fence_proxy_async_smem();
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(bar(C::kBarPds + h));
                    mbar_arrive(bar(C::kBarQdEmpty + s));
                }
            }
            // ---- epilogue: dV and dK of this thread's key, columns [d/2 h, d/2 (h+1)) ---
            if (ok) ok = wait_warp_sleep(bar(C::kBarAcc), k & 1, wc, kRoleBwdCompute * 1000 + C::kBarAcc, k);
            if (!ok) break;
            tc_fence_after_sync();
#pragma unroll 1
            for (int which = 0; which < 2; ++which) {
                const uint32_t col = which == 0 ? C::colDV : C::colDK;
                const float mul = which == 0 ? 1.f : p.scale;
                uint8_t* out = static_cast<uint8_t*>(which == 0 ? p.dv : p.dk);
                uint32_t o[32];
                tmem_ld32(lane_base + col + 32 * h, o);
                tmem_ld_wait();
                reg_fence(o);
                if (j < p.Nk) {
                    uint4* row = reinterpret_cast<uint4*>(out + ((static_cast<size_t>(bh) * p.Nk + j) * D + 32 * h) * 2);
#pragma unroll
                    for (int e = 0; e < 32; e += 8)
                        row[e >> 3] = make_uint4(
                            pack2<BF16>(__uint_as_float(o[e]) * mul, __uint_as_float(o[e + 1]) * mul),
                            pack2<BF16>(__uint_as_float(o[e + 2]) * mul, __uint_as_float(o[e + 3]) * mul),
                            pack2<BF16>(__uint_as_float(o[e + 4]) * mul, __uint_as_float(o[e + 5]) * mul),
                            pack2<BF16>(__uint_as_float(o[e + 6]) * mul, __uint_as_float(o[e + 7]) * mul));
                }
            }
            // dV and dK are read out: the next item's first dV/dK may overwrite them.
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(C::kBarAccFree));
        }
    }

    tc_fence_before_sync();
    __syncthreads();
    if (warp == C::kWarpMma) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, C::kTmemCols);
    }
}

}  // namespace attn_sm103
