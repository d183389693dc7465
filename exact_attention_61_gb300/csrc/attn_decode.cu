// Streaming decode attention on sm_103a: up to four query rows per head against a long
// key sequence (a KV-cache decode step), the regime that "Getting the kernel correct,
// then benchmarking it honestly" ("Next") names as the extension after the forward.
// Per row it computes what the forward computes (scores q k^T scaled, masked keys left
// out, online softmax, O = sum_j p_j v_j / l, LSE = ln of the sum of exponentials), with P
// and every sum kept in fp32.
//
// The work is bound by HBM (each K and V byte is used for one to four rows), so it stays
// on the CUDA cores and is laid out for streaming:
//  - every warp works alone on units (head, range of keys), units assigned round-robin
//    over all warps of the grid (one CTA per SM; the host's plan picks the ranges);
//  - lane 0 of a warp streams the unit's K and V tiles (32 keys; a head's keys are
//    contiguous, so one 1-D bulk copy per tile and tensor) through the warp's own
//    two- or three-stage ring, with an evict-first L2 policy; the ring runs across units;
//  - each key row is read as 16-byte chunks by CH = d/8 consecutive lanes (one chunk per
//    lane), so a warp reads G = 32/CH whole rows per shared-memory load, conflict-free;
//    a lane keeps its chunk of each query row (times scale * log2 e) in registers, and the
//    partial dot products are summed over the CH lanes by shuffles;
//  - the softmax state (running max m, sum l) is per row and shared by the warp; each
//    lane accumulates O for its 8 head dimensions over the keys its lane group read.
//    The groups' l and O are summed at the end of the unit. Rescaling is lazy, as in the
//    forward: a row keeps its maximum until a tile's exceeds it by more than kRescaleTau
//    (log2 units), so O and l are rescaled only then (P stays below 2^8 in fp32);
//  - with several rows, the dot products of the CH lanes of a key row are summed by a
//    transposed reduction that leaves one row's score per lane, so the softmax runs once
//    per lane and key; P of every row is then fetched from its lane for O += P V.
// A unit writes O / l and its log2-sum-exp to the split partials (merged by
// attn_merge_kernel), or, with one range per head, the final O and LSE.
#include <atomic>

#include "attn_fwd_kernel.cuh"
#include "attn_internal.h"

namespace attn_sm103 {
namespace {

constexpr uint32_t kRoleDecode = 5;

template <int D, int NQ>
struct DecCfg {
    static constexpr int kWarps = decode_warps(D, NQ);
    static constexpr int kThreads = 32 * kWarps;
    static constexpr int T = decode_tile_keys(D, NQ);
    static constexpr int kStages = decode_stages(D, NQ);
    static constexpr int kTileBytes = T * D * 2;        // one K or V tile
    static constexpr int kStageBytes = 2 * kTileBytes;  // K, then V
    static constexpr int kWarpBytes = kStages * kStageBytes;
    static constexpr int kOffBar = kWarps * kWarpBytes;
    static constexpr int kOffMisc = kOffBar + kWarps * kStages * 8;
    static constexpr int kSmemBytes = kOffMisc + 16 + 128;  // + alignment slack
    static constexpr int CH = D / 8;                       // lanes per key row
    static constexpr int G = 32 / CH;                      // key rows per load
    static constexpr int kSteps = T / G;
    static_assert(kSmemBytes <= 227 * 1024, "shared memory");
};

// 8 values of a 16-byte chunk as fp32.
template <bool BF16>
__device__ __forceinline__ void unpack8(const uint4& c, float2 (&f)[4]) {
    f[0] = unpack2<BF16>(c.x);
    f[1] = unpack2<BF16>(c.y);
    f[2] = unpack2<BF16>(c.z);
    f[3] = unpack2<BF16>(c.w);
}

template <int D, int NQ, bool BF16>
__global__ void __launch_bounds__(DecCfg<D, NQ>::kThreads, 1) attn_decode_kernel(const DecodeParams p) {
    using C = DecCfg<D, NQ>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 127u) & ~127u;
    uint8_t* smem = smem_raw + (base - raw);
    const int warp = static_cast<int>(threadIdx.x >> 5);
    const int lane = static_cast<int>(threadIdx.x & 31u);
    uint32_t* misc = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);  // [0] abort flag
    WaitCtx wc{p.err, misc, blockIdx.x};
    const uint32_t wbase = base + static_cast<uint32_t>(warp * C::kWarpBytes);
    const uint8_t* wsm = smem + warp * C::kWarpBytes;
    auto bar = [&](int s) -> uint32_t { return base + C::kOffBar + 8u * (warp * C::kStages + s); };

    if (threadIdx.x == 0) misc[0] = 0u;
    if (lane == 0) {
        for (int s = 0; s < C::kStages; ++s) mbar_init(bar(s), 1u);
        fence_mbar_init();
    }
    __syncthreads();

    const int grp = lane / C::CH;
    const int ch = lane % C::CH;
    // Keys row r sees: [0, lim[r]) (rows past Nq see none and are not written).
    int lim[NQ];
#pragma unroll
    for (int r = 0; r < NQ; ++r) {
        int e = p.Nk;
        if (p.causal) e = p.align_br ? r + p.Nk - p.Nq + 1 : r + 1;
        lim[r] = r < p.Nq ? max(0, min(p.Nk, e)) : 0;
    }
    int vis = 0;  // keys any row sees
#pragma unroll
    for (int r = 0; r < NQ; ++r) vis = max(vis, lim[r]);
    int lim_min = vis;  // keys every real row sees
#pragma unroll
    for (int r = 0; r < NQ; ++r)
        if (r < p.Nq) lim_min = min(lim_min, lim[r]);
    // With NQ = 4 the score of one query row ends in each lane after the reduction over
    // the CH lanes of a key row: row rho = 2 * bit2 + bit1 of the lane (bit 0, and bit 3
    // for CH = 16, hold copies); src(r) is the first lane of the group holding row r.
    const int rho = ((lane >> 2) & 1) * 2 + ((lane >> 1) & 1);
    const int lim_rho = lim[rho < NQ ? rho : 0];
    const int gbase = lane & ~(C::CH - 1);
    auto src = [&](int r) { return gbase + ((r >> 1) << 2) + ((r & 1) << 1); };

    const int W = static_cast<int>(gridDim.x) * C::kWarps;
    const int gw = static_cast<int>(blockIdx.x) * C::kWarps + warp;
    const int U = p.BH * p.n_ranges;
    // Tiles of unit u that hold visible keys: [kb, ke) of head bh.
    auto unit_tiles = [&](int u, int& bh, int& kb, int& ke) -> int {
        bh = u / p.n_ranges;
        kb = (u - bh * p.n_ranges) * p.range_keys;
        ke = min(min(p.Nk, kb + p.range_keys), vis);
        return ke > kb ? (ke - kb + C::T - 1) / C::T : 0;
    };

    // ---- producer (lane 0 issues; every lane walks the cursor) ---------------------------
    const uint64_t pol = l2_policy_evict_first();
    const char* kg = static_cast<const char*>(p.k);
    const char* vg = static_cast<const char*>(p.v);
    int pu = gw, pt = 0, pnt = 0, pbh = 0, pkb = 0, pke = 0;
    // first unit with tiles at or after pu (pt = 0)
    auto p_seek = [&]() -> bool {
        for (; pu < U; pu += W) {
            pnt = unit_tiles(pu, pbh, pkb, pke);
            if (pnt > 0) return true;
        }
        return false;
    };
    bool pvalid = p_seek();
    uint32_t n_issued = 0, n_done = 0;
    auto p_issue_next = [&]() {
        if (!pvalid) return;
        const int key0 = pkb + pt * C::T;
        const uint32_t bytes = static_cast<uint32_t>(min(C::T, pke - key0) * D * 2);
        const int s = static_cast<int>(n_issued % C::kStages);
        if (lane == 0) {
            const size_t off = (static_cast<size_t>(pbh) * p.Nk + key0) * (D * 2);
            fence_proxy_async_smem();  // the warp's reads of this stage precede the copy
            mbar_arrive_expect_tx(bar(s), 2u * bytes);
            bulk_load_hint(wbase + s * C::kStageBytes, kg + off, bytes, bar(s), pol);
            bulk_load_hint(wbase + s * C::kStageBytes + C::kTileBytes, vg + off, bytes, bar(s), pol);
        }
        ++n_issued;
        if (++pt == pnt) {
            pt = 0;
            pu += W;
            pvalid = p_seek();
        }
    };
    for (int i = 0; i < C::kStages; ++i) p_issue_next();
    griddep_launch_dependents();  // the merge may start launching (it waits for this grid)

    // ---- consumer ------------------------------------------------------------------------
    const char* qg = static_cast<const char*>(p.q);
    bool ok = true;
    for (int u = gw; u < U && ok; u += W) {
        int bh, kb, ke;
        const int nt = unit_tiles(u, bh, kb, ke);
        // this lane's chunk of each query row, times scale * log2(e)
        float2 qf[NQ][4];
#pragma unroll
        for (int r = 0; r < NQ; ++r) {
            uint4 c = make_uint4(0u, 0u, 0u, 0u);
            if (r < p.Nq)
                c = *reinterpret_cast<const uint4*>(qg + ((static_cast<size_t>(bh) * p.Nq + r) * D + ch * 8) * 2);
            unpack8<BF16>(c, qf[r]);
#pragma unroll
            for (int e = 0; e < 4; ++e) qf[r][e] = make_float2(qf[r][e].x * p.qk_scale, qf[r][e].y * p.qk_scale);
        }
        float m[NQ], l[NQ];
        float2 o[NQ][4];
#pragma unroll
        for (int r = 0; r < NQ; ++r) {
            m[r] = -INFINITY;
            l[r] = 0.f;
#pragma unroll
            for (int e = 0; e < 4; ++e) o[r][e] = make_float2(0.f, 0.f);
        }
        for (int t = 0; t < nt; ++t) {
            const int s = static_cast<int>(n_done % C::kStages);
            if (!wait_warp(bar(s), (n_done / C::kStages) & 1u, wc, kRoleDecode * 1000 + s, n_done)) {
                ok = false;
                break;
            }
            const uint8_t* sk = wsm + s * C::kStageBytes;
            const uint8_t* sv = sk + C::kTileBytes;
            const int key0 = kb + t * C::T;
            const int rows = min(C::T, ke - key0);  // rows this tile's copies wrote
            // no key of the tile is masked for any real row (the common case)
            const bool full = rows == C::T && key0 + C::T <= lim_min;
            if constexpr (NQ == 1) {
                // scores (log2 units): partial dot products over this lane's 8 dimensions,
                // summed over the CH lanes of the key row
                float sc[C::kSteps];
#pragma unroll
                for (int st = 0; st < C::kSteps; ++st) {
                    const int key = st * C::G + grp;
                    float2 kf[4];
                    unpack8<BF16>(*reinterpret_cast<const uint4*>(sk + key * (D * 2) + ch * 16), kf);
                    float2 a = __fmul2_rn(qf[0][0], kf[0]);
                    a = __ffma2_rn(qf[0][1], kf[1], a);
                    a = __ffma2_rn(qf[0][2], kf[2], a);
                    a = __ffma2_rn(qf[0][3], kf[3], a);
                    float x = a.x + a.y;
#pragma unroll
                    for (int off = 1; off < C::CH; off <<= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
                    sc[st] = (full || (key < rows && key0 + key < lim[0])) ? x : -INFINITY;
                }
                // online softmax over the tile
                float mx = -INFINITY;
#pragma unroll
                for (int st = 0; st < C::kSteps; ++st) mx = fmaxf(mx, sc[st]);
#pragma unroll
                for (int off = C::CH; off < 32; off <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
                float m_new = fmaxf(m[0], mx);
                if (m_new - m[0] <= kRescaleTau) m_new = m[0];  // keep the maximum (false from -inf)
                const float m_use = m_new == -INFINITY ? 0.f : m_new;
                const float alpha = m[0] == m_use ? 1.f : ex2_ftz(m[0] - m_use);  // 0 from an empty state
                m[0] = m_new;
                if (alpha != 1.f) {  // warp-uniform: m is the warp's
                    l[0] *= alpha;
                    const float2 a2 = make_float2(alpha, alpha);
#pragma unroll
                    for (int e = 0; e < 4; ++e) o[0][e] = __fmul2_rn(o[0][e], a2);
                }
#pragma unroll
                for (int st = 0; st < C::kSteps; ++st) {
                    sc[st] = ex2_ftz(sc[st] - m_use);
                    l[0] += sc[st];
                }
                // O += P V over this lane group's keys and this lane's 8 dimensions
#pragma unroll
                for (int st = 0; st < C::kSteps; ++st) {
                    const int key = st * C::G + grp;
                    if (full || key < rows) {
                        float2 vf[4];
                        unpack8<BF16>(*reinterpret_cast<const uint4*>(sv + key * (D * 2) + ch * 16), vf);
                        const float2 p2 = make_float2(sc[st], sc[st]);
#pragma unroll
                        for (int e = 0; e < 4; ++e) o[0][e] = __ffma2_rn(p2, vf[e], o[0][e]);
                    }
                }
            } else {
                // scores: four partial dot products per lane, then a transposed reduction
                // over the CH lanes of the key row that leaves row rho's score in the lane
                // (two partials exchanged across bit 2, one across bit 1, then plain sums)
                float sc[C::kSteps];
                const bool b2 = (lane >> 2) & 1, b1 = (lane >> 1) & 1;
#pragma unroll
                for (int st = 0; st < C::kSteps; ++st) {
                    const int key = st * C::G + grp;
                    float2 kf[4];
                    unpack8<BF16>(*reinterpret_cast<const uint4*>(sk + key * (D * 2) + ch * 16), kf);
                    float x[4];
#pragma unroll
                    for (int r = 0; r < 4; ++r) {
                        float2 a = __fmul2_rn(qf[r][0], kf[0]);
                        a = __ffma2_rn(qf[r][1], kf[1], a);
                        a = __ffma2_rn(qf[r][2], kf[2], a);
                        a = __ffma2_rn(qf[r][3], kf[3], a);
                        x[r] = a.x + a.y;
                    }
                    // across bit 2: keep rows {0,1} (bit2 = 0) or {2,3}
                    const float ka = b2 ? x[2] : x[0], kb2 = b2 ? x[3] : x[1];
                    const float ga = b2 ? x[0] : x[2], gb = b2 ? x[1] : x[3];
                    const float ya = ka + __shfl_xor_sync(0xffffffffu, ga, 4);
                    const float yb = kb2 + __shfl_xor_sync(0xffffffffu, gb, 4);
                    // across bit 1: keep row 2 * bit2 + bit1
                    float z = (b1 ? yb : ya) + __shfl_xor_sync(0xffffffffu, b1 ? ya : yb, 2);
                    z += __shfl_xor_sync(0xffffffffu, z, 1);
                    if constexpr (C::CH == 16) z += __shfl_xor_sync(0xffffffffu, z, 8);
                    sc[st] = (full || (key < rows && key0 + key < lim_rho)) ? z : -INFINITY;
                }
                // online softmax of row rho over the tile (state m[0], l[0] of that row)
                float mx = -INFINITY;
#pragma unroll
                for (int st = 0; st < C::kSteps; ++st) mx = fmaxf(mx, sc[st]);
#pragma unroll
                for (int off = C::CH; off < 32; off <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
                float m_new = fmaxf(m[0], mx);
                if (m_new - m[0] <= kRescaleTau) m_new = m[0];  // keep the maximum (false from -inf)
                const float m_use = m_new == -INFINITY ? 0.f : m_new;
                const float alpha = m[0] == m_use ? 1.f : ex2_ftz(m[0] - m_use);  // 0 from an empty state
                m[0] = m_new;
                l[0] *= alpha;
#pragma unroll
                for (int st = 0; st < C::kSteps; ++st) {
                    sc[st] = ex2_ftz(sc[st] - m_use);
                    l[0] += sc[st];
                }
                if (__any_sync(0xffffffffu, alpha != 1.f)) {  // some row's maximum moved
#pragma unroll
                    for (int r = 0; r < 4; ++r) {
                        const float ar = __shfl_sync(0xffffffffu, alpha, src(r));
                        const float2 a2 = make_float2(ar, ar);
#pragma unroll
                        for (int e = 0; e < 4; ++e) o[r][e] = __fmul2_rn(o[r][e], a2);
                    }
                }
                // O += P V: every row's P of the key fetched from its lane, then this lane's
                // 8 dimensions of each row
#pragma unroll
                for (int st = 0; st < C::kSteps; ++st) {
                    const int key = st * C::G + grp;
                    float pr[4];
#pragma unroll
                    for (int r = 0; r < 4; ++r) pr[r] = __shfl_sync(0xffffffffu, sc[st], src(r));
                    if (full || key < rows) {
                        float2 vf[4];
                        unpack8<BF16>(*reinterpret_cast<const uint4*>(sv + key * (D * 2) + ch * 16), vf);
#pragma unroll
                        for (int r = 0; r < 4; ++r) {
                            const float2 p2 = make_float2(pr[r], pr[r]);
#pragma unroll
                            for (int e = 0; e < 4; ++e) o[r][e] = __ffma2_rn(p2, vf[e], o[r][e]);
                        }
                    }
                }
            }
            __syncwarp();  // every lane is done with the stage before it is refilled
            ++n_done;
            p_issue_next();
        }
        if (!ok) break;
        // sum the lane groups' l and O (all relative to the same m)
#pragma unroll
        for (int off = C::CH; off < 32; off <<= 1) l[0] += __shfl_xor_sync(0xffffffffu, l[0], off);
#pragma unroll
        for (int r = 0; r < NQ; ++r)
#pragma unroll
            for (int off = C::CH; off < 32; off <<= 1) {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    o[r][e].x += __shfl_xor_sync(0xffffffffu, o[r][e].x, off);
                    o[r][e].y += __shfl_xor_sync(0xffffffffu, o[r][e].y, off);
                }
            }
        if constexpr (NQ > 1) {  // row r's l and m from the lanes that hold row r
            const float l_own = l[0], m_own = m[0];
#pragma unroll
            for (int r = 0; r < NQ; ++r) {
                l[r] = __shfl_sync(0xffffffffu, l_own, src(r));
                m[r] = __shfl_sync(0xffffffffu, m_own, src(r));
            }
        }
        const int rg = u - bh * p.n_ranges;
#pragma unroll
        for (int r = 0; r < NQ; ++r) {
            if (r >= p.Nq || grp != 0) continue;
            const float inv = l[r] > 0.f ? 1.f / l[r] : 0.f;
            const float lse2 = l[r] > 0.f ? m[r] + log2f(l[r]) : -INFINITY;
            if (p.n_ranges == 1) {
                uint4 w;
                w.x = pack2<BF16>(o[r][0].x * inv, o[r][0].y * inv);
                w.y = pack2<BF16>(o[r][1].x * inv, o[r][1].y * inv);
                w.z = pack2<BF16>(o[r][2].x * inv, o[r][2].y * inv);
                w.w = pack2<BF16>(o[r][3].x * inv, o[r][3].y * inv);
                *reinterpret_cast<uint4*>(static_cast<char*>(p.o) + ((static_cast<size_t>(bh) * p.Nq + r) * D + ch * 8) * 2) = w;
                if (ch == 0) p.lse[static_cast<size_t>(bh) * p.Nq + r] = lse2 * 0.69314718055994530942f;
            } else {
                const size_t row = (static_cast<size_t>(bh) * p.n_ranges + rg) * p.Nq + r;
                float4* dst = reinterpret_cast<float4*>(p.o_part + row * D + ch * 8);
                dst[0] = make_float4(o[r][0].x * inv, o[r][0].y * inv, o[r][1].x * inv, o[r][1].y * inv);
                dst[1] = make_float4(o[r][2].x * inv, o[r][2].y * inv, o[r][3].x * inv, o[r][3].y * inv);
                if (ch == 0) p.lse_part[row] = lse2;
            }
        }
    }
    // Every copy issued into this warp's stages has landed before the CTA exits.
    while (n_done < n_issued) {
        wait_warp(bar(static_cast<int>(n_done % C::kStages)), (n_done / C::kStages) & 1u, wc,
                  kRoleDecode * 1000 + 90, n_done, false);
        ++n_done;
    }
}

template <int D, int NQ, bool BF16>
cudaError_t launch_one_decode(const DecodeParams& p, int64_t grid, cudaStream_t s) {
    using C = DecCfg<D, NQ>;
    auto* kern = attn_decode_kernel<D, NQ, BF16>;
    static std::atomic<uint64_t> configured{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = dev < 64 ? (1ull << dev) : 0ull;
    if (!bit || !(configured.load(std::memory_order_acquire) & bit)) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
        if (e != cudaSuccess) return e;
        configured.fetch_or(bit, std::memory_order_acq_rel);
    }
    kern<<<static_cast<unsigned>(grid), C::kThreads, C::kSmemBytes, s>>>(p);
    return cudaGetLastError();
}

template <int D, bool BF16>
cudaError_t launch_rows(const DecodeParams& p, int64_t grid, cudaStream_t s) {
    return p.Nq == 1 ? launch_one_decode<D, 1, BF16>(p, grid, s) : launch_one_decode<D, kDecodeMaxRows, BF16>(p, grid, s);
}

}  // namespace

cudaError_t launch_decode(int64_t d, bool bf16, const DecodeParams& p, int64_t grid, cudaStream_t s) {
    if (p.Nq < 1 || p.Nq > kDecodeMaxRows || grid < 1) return cudaErrorInvalidValue;
    if (d == 64) return bf16 ? launch_rows<64, true>(p, grid, s) : launch_rows<64, false>(p, grid, s);
    if (d == 128) return bf16 ? launch_rows<128, true>(p, grid, s) : launch_rows<128, false>(p, grid, s);
    return cudaErrorInvalidValue;
}

}  // namespace attn_sm103
