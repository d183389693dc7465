// Exact attention backward for sm_103a: dQ, dK, dV of sum(dO * O) from the saved LSE.
//
// What it computes, per head, for keys j and query rows i that see them
// (natural-log LSE from the forward, D_i = dO_i . O_i):
//   P_ij  = exp(scale q_i.k_j - LSE_i)
//   dV_j  = sum_i P_ij dO_i
//   dP_ij = dO_i . v_j,   dS_ij = P_ij (dP_ij - D_i)
//   dK_j  = scale sum_i dS_ij q_i,   dQ_i = scale sum_j dS_ij k_j
// This is the FlashAttention-2 backward that "如何用 profiler 逐步优化 Triton
// FlashAttention-2 kernel" ("Future articles") names as the next kernel: it
// consumes the L the forward writes ("Round 4 / exp2": natural-log units), and
// it has two accumulations in different directions (dK, dV over query rows; dQ
// over key tiles).
//
// GB300 design:
//  - one CTA owns one 128-key tile of one head and loops over the 128-row Q tiles
//    that see it (all of them, or those from the diagonal on under the causal
//    mask). K and V stay in shared memory; Q, dO and the per-row LSE/D vectors
//    stream through a TMA ring;
//  - one warp issues the tcgen05 MMAs, all into tensor memory (at d = 64 after copying
//    K and V into TMEM with tcgen05.cp, which the tensor core runs ahead of them):
//      S^T  = K Q^T     (128 keys x 128 queries, fp32; d = 64: K from TMEM)
//      dP^T = V dO^T    (128 x 128, fp32; d = 64: V from TMEM)
//      dV  += P^T dO    (P^T 16-bit in TMEM over S^T; dO MN-major in SMEM)
//      dK  += dS^T Q    (dS^T 16-bit in TMEM over dP^T; Q MN-major in SMEM)
//      dQ   = dS K      (dS 16-bit in SMEM, MN-major; K MN-major in SMEM)
//  - two warpgroups, one thread per key row (= TMEM lane) and half of the 128
//    query columns each, turn S^T and dP^T into P^T and dS^T with exp2 and the
//    LSE folded in log2 units, and write dS for the dQ product to shared memory.
//    At d = 64 each half has its own S^T/dP^T and P^T/dS^T hand-off, so one
//    warpgroup's math overlaps the other half's products;
//  - a third warpgroup adds each dQ tile into an fp32 workspace (dQ gathers over key
//    tiles owned by other CTAs) by staging it in shared memory and a TMA bulk
//    reduce-add, off the critical path of the other two;
//  - dK and dV stay in TMEM for the whole loop and are stored once at the end;
//  - every mbarrier wait is bounded, as in the forward kernel.
#pragma once

#include "attn_bwd_internal.h"
#include "attn_fwd_kernel.cuh"

namespace attn_sm103 {

enum : uint32_t { kRoleBwdLoad = 5, kRoleBwdMma = 6, kRoleBwdCompute = 7, kRoleBwdDq = 8 };
constexpr int kBwdHeadGroup = 8;  // heads whose causal key tiles are ordered together
constexpr uint32_t kErrSmemAlign = 2u;

// ---- tcgen05 / bulk-copy forms only the backward uses ------------------------------------

// D = A B over 128 rows of K with both operands MN-major in shared memory: 8 MMAs of
// K = 16, each advancing 16 rows = 2048 bytes = 128 descriptor units on A and on B.
__device__ __forceinline__ void mma_mn128_warp(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                               uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred e, p, one;\n\t.reg .b64 ad, bd;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "setp.eq.b32 one, 0, 0;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t"
        "add.u64 ad, %1, 128;\n\tadd.u64 bd, %2, 128;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], ad, bd, %3, one;\n\t"
        "add.u64 ad, %1, 256;\n\tadd.u64 bd, %2, 256;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], ad, bd, %3, one;\n\t"
        "add.u64 ad, %1, 384;\n\tadd.u64 bd, %2, 384;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], ad, bd, %3, one;\n\t"
        "add.u64 ad, %1, 512;\n\tadd.u64 bd, %2, 512;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], ad, bd, %3, one;\n\t"
        "add.u64 ad, %1, 640;\n\tadd.u64 bd, %2, 640;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], ad, bd, %3, one;\n\t"
        "add.u64 ad, %1, 768;\n\tadd.u64 bd, %2, 768;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], ad, bd, %3, one;\n\t"
        "add.u64 ad, %1, 896;\n\tadd.u64 bd, %2, 896;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], ad, bd, %3, one;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// D (+)= A B over 128 rows of K with A (16-bit) in TMEM stored as two halves: K rows
// 0-63 in columns [a, a+32) and K rows 64-127 in [a+64, a+96) (each compute warpgroup
// packs its half of the 128 fp32 columns in place). B MN-major in SMEM, advancing 16
// rows = 128 descriptor units per MMA. `accumulate` applies to the first MMA.
__device__ __forceinline__ void mma_pv128_halves_warp(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                                      uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred e, p, one;\n\t.reg .b32 ta;\n\t.reg .b64 bd;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "setp.eq.b32 one, 0, 0;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t"
        "add.u32 ta, %1, 8;\n\tadd.u64 bd, %2, 128;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], bd, %3, one;\n\t"
        "add.u32 ta, %1, 16;\n\tadd.u64 bd, %2, 256;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], bd, %3, one;\n\t"
        "add.u32 ta, %1, 24;\n\tadd.u64 bd, %2, 384;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], bd, %3, one;\n\t"
        "add.u32 ta, %1, 64;\n\tadd.u64 bd, %2, 512;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], bd, %3, one;\n\t"
        "add.u32 ta, %1, 72;\n\tadd.u64 bd, %2, 640;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], bd, %3, one;\n\t"
        "add.u32 ta, %1, 80;\n\tadd.u64 bd, %2, 768;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], bd, %3, one;\n\t"
        "add.u32 ta, %1, 88;\n\tadd.u64 bd, %2, 896;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], bd, %3, one;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// D (+)= A B over 64 rows of K with A (16-bit) in TMEM columns [a, a+32) and B MN-major
// in SMEM: 4 MMAs of K = 16, A advancing 8 columns and B 16 rows = 128 descriptor units.
// `accumulate` applies to the first MMA.
__device__ __forceinline__ void mma_pv64_tmem_warp(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                                   uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred e, p, one;\n\t.reg .b32 ta;\n\t.reg .b64 bd;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "setp.eq.b32 one, 0, 0;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t"
        "add.u32 ta, %1, 8;\n\tadd.u64 bd, %2, 128;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], bd, %3, one;\n\t"
        "add.u32 ta, %1, 16;\n\tadd.u64 bd, %2, 256;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], bd, %3, one;\n\t"
        "add.u32 ta, %1, 24;\n\tadd.u64 bd, %2, 384;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], bd, %3, one;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// D = A B^T over K = 64 with A (16-bit, M x 64) in TMEM columns [a, a+32) and B K-major
// in SMEM (128-byte swizzle): 4 MMAs of K = 16, A advancing 8 columns and B 32 bytes.
__device__ __forceinline__ void mma_ts_k64_warp(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                                uint32_t idesc) {
    asm volatile(
        "{\n\t.reg .pred e, zero, one;\n\t.reg .b32 ta;\n\t.reg .b64 bd;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "setp.ne.b32 zero, 0, 0;\n\t"
        "setp.eq.b32 one, 0, 0;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, zero;\n\t"
        "add.u32 ta, %1, 8;\n\tadd.u64 bd, %2, 2;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], bd, %3, one;\n\t"
        "add.u32 ta, %1, 16;\n\tadd.u64 bd, %2, 4;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], bd, %3, one;\n\t"
        "add.u32 ta, %1, 24;\n\tadd.u64 bd, %2, 6;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], bd, %3, one;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc)
        : "memory");
}

// Instruction descriptor with the major-ness of A chosen too (bit 15; A from SMEM).
__host__ __device__ constexpr uint32_t idesc_f16_f32acc_ab(bool bf16, int M, int N, bool a_mn_major,
                                                           bool b_mn_major) {
    return idesc_f16_f32acc(bf16, M, N, b_mn_major) | ((a_mn_major ? 1u : 0u) << 15);
}

// Warp-wide: thread t writes 16 consecutive 32-bit columns of TMEM lane (lane_base + t).
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, "
        "%12, %13, %14, %15, %16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}

// Global -> shared plain bulk copy of `bytes` (multiple of 16; both addresses 16-byte
// aligned); completion is signalled on `bar` as transaction bytes.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

// Shared -> global element-wise fp32 add of a 3-D box (bulk async-group completion).
// Rows outside the tensor are skipped.
__device__ __forceinline__ void tma_reduce_add_3d(const CUtensorMap* map, uint32_t src, int32_t c0, int32_t c1,
                                                  int32_t c2) {
    asm volatile(
        "cp.reduce.async.bulk.tensor.3d.global.shared::cta.add.tile.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
            map),
        "r"(src), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d)
                 : "memory");
}

// ---- configuration -----------------------------------------------------------------------

template <int D>
struct BwdCfg {
    static_assert(D == 64 || D == 128, "head dimension must be 64 or 128");
    // Q/dO ring depth. Each stage is held until the dQ reduce-add of its tile has read
    // it, so the ring also absorbs the latency of those L2 reductions.
    static constexpr int kStages = D == 64 ? 4 : 2;
    static constexpr int kBoxBytes = 128 * 128;         // one TMA box: 128 rows x 64 elements x 2 B
    static constexpr int kChunks = D / 64;              // boxes per 128-row tile
    static constexpr int kTileBytes = 128 * D * 2;
    static constexpr int kOffK = 0;
    // dS: 128 keys x 128 queries, MN-major. At d = 64, V is read from shared memory only
    // once, to copy it into TMEM before any dS is written, so it lands in the second dS
    // buffer (which frees the room for a fourth ring stage).
    static constexpr int kOffDS = kOffK + kTileBytes + (D == 64 ? 0 : kTileBytes);
    static constexpr int kOffV = D == 64 ? kOffDS + 128 * 128 * 2 : kOffK + kTileBytes;
    // d = 64: a Q tile is two halves of 64 query columns, one per compute warpgroup, each
    // with its own S^T/dP^T commit and P^T/dS^T hand-off. S^T and dP^T of half h of the next
    // tile are issued right after dV and dK of half h of this one, before dQ, so one
    // warpgroup's math overlaps the other half's products and dQ; dS then alternates
    // between two buffers (d = 128 keeps its dQ tile over S^T and the plain order).
    static constexpr bool kEarlyNext = D == 64;
    static constexpr int kDsBufs = kEarlyNext ? 2 : 1;
    static constexpr int kOffStage = kOffDS + kDsBufs * 128 * 128 * 2;
    static constexpr int kStageBytes = 2 * kTileBytes;  // Q, then dO
    // The fp32 dQ tile (128 rows x d, exactly one Q/dO ring stage) is staged in the ring
    // stage of its own iteration, in boxes of 32 columns x 128 rows with the 128-byte
    // swizzle, and added to the accumulator by TMA. Every MMA of the iteration has
    // finished reading the stage once dQ is done; the stage returns to the loader only
    // after the reduce has read it.
    static constexpr int kDqBoxBytes = 128 * 32 * 4;
    static_assert((D / 32) * kDqBoxBytes == kStageBytes, "dQ tile = one ring stage");
    static constexpr int kOffVec = kOffStage + kStages * kStageBytes;
    static constexpr int kVecBytes = 2 * 128 * 4;       // lse2[128], D[128] per stage
    static constexpr int kOffBar = kOffVec + kStages * kVecBytes;
    static constexpr int kBarKV = 0;
    static constexpr int kBarQdFull = 1;
    static constexpr int kBarQdEmpty = kBarQdFull + kStages;
    static constexpr int kBarSdp = kBarQdEmpty + kStages;  // [half]: S^T and dP^T in TMEM
    static constexpr int kBarPds = kBarSdp + 2;            // [half]: P^T, dS^T in TMEM, dS in SMEM
    static constexpr int kBarDqFull = kBarPds + 2;         // dQ tile in TMEM
    static constexpr int kBarDqRead = kBarDqFull + 1;      // dQ tile read out
    static constexpr int kBarAcc = kBarDqRead + 1;         // dK, dV final
    static constexpr int kBarDqItem = kBarAcc + 1;         // persistent form: the dQ warps read the item
    static constexpr int kBarAccFree = kBarDqItem + 1;     // persistent form: dK, dV read out
    static constexpr int kBarDrain = kBarAccFree + 1;
    static constexpr int kNumBars = kBarDrain + 1;
    static constexpr int kOffMisc = kOffBar + kNumBars * 8;
    // The dynamic shared-memory base is 1024-byte aligned (declared so and checked at
    // run time): d = 128 leaves no room for alignment slack. misc: [0] TMEM base, [1] abort
    // flag, [4..8) the persistent kernel's ring of claimed work items.
    static constexpr int kSmemBytes = kOffMisc + 32;
    static_assert(kSmemBytes <= 232448, "shared memory budget");
    // TMEM columns: S^T/P^T, dP^T/dS^T, dV, dK, and the dQ tile (d = 128: over S^T).
    static constexpr uint32_t colS = 0, colDP = 128, colDV = 256, colDK = 256 + D;
    static constexpr uint32_t colDQ = D == 64 ? 384u : 0u;
    // d = 64: K and V (16-bit, two elements per column) are the A operands of S^T and dP^T
    // from TMEM, so the tensor core reads only Q and dO from shared memory for them.
    static constexpr bool kKvTmem = kEarlyNext;
    static constexpr uint32_t colK = 448, colV = 480;
    static constexpr uint32_t kTmemCols = 512;
    static_assert(!kKvTmem || (colDQ + D <= colK && colV + D / 2 <= kTmemCols), "TMEM budget");
    // warps 0-3: compute, query columns 0-63; 4-7: compute, columns 64-127;
    // 8-11: dQ read-out; 12: MMA; 13: TMA
    static constexpr int kThreads = 448;
    static constexpr int kWarpDq = 8;
    static constexpr int kWarpMma = 12;
    static constexpr int kWarpLoad = 13;
};

// EXT: key padding, a window and Nq != Nk (the forward's EXT readings); without it the
// code for them is compiled out and Nq = Nk, top-left.
template <int D, bool CAUSAL, bool BF16, bool EXT>
__global__ void __launch_bounds__(BwdCfg<D>::kThreads, 1)
    attn_bwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
                    const __grid_constant__ CUtensorMap tmDQ, const BwdParams p) {
    using C = BwdCfg<D>;
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

    // CTA order. Non-causal: a head's key tiles run together, so its Q, dO and dQ
    // accumulator stay in L2. Causal: heads in groups of kBwdHeadGroup, whose key tiles run
    // heaviest first (key tile 0 sees every Q tile), so the group's working set stays in L2
    // and the grid still ends on light tiles.
    const int n_kt_grid = static_cast<int>(gridDim.x) / p.BH;
    int bh, kt;
    if (CAUSAL) {
        const int x = static_cast<int>(blockIdx.x);
        const int grp = x / (kBwdHeadGroup * n_kt_grid);
        const int gh = min(kBwdHeadGroup, p.BH - grp * kBwdHeadGroup);  // heads in this group
        const int idx = x - grp * kBwdHeadGroup * n_kt_grid;
        kt = idx / gh;
        bh = grp * kBwdHeadGroup + idx % gh;
    } else {
        bh = static_cast<int>(blockIdx.x) / n_kt_grid;
        kt = static_cast<int>(blockIdx.x) % n_kt_grid;
    }
    const int Nq = p.Nq, Nk = p.Nk;
    const int j0 = kt * 128;
    // Valid keys of this batch element; key j is visible to query row i iff j < n_b and,
    // with the causal mask, j <= i + up and, with a left window, j >= i + lo.
    const int n_b = (EXT && p.kv_lens) ? min(max(p.kv_lens[bh / p.H], 0), Nk) : Nk;
    const int diag_off = (EXT && p.align_br) ? n_b - Nq : 0;
    const int up = diag_off + (EXT ? p.win_right : 0);
    const bool has_lo = EXT && p.win_left >= 0;
    const int lo = diag_off - (EXT ? p.win_left : 0);
    // The Q tiles that see at least one key of this tile.
    const int n_qt = p.Npad / 128;
    int qt_begin = 0, qt_end = n_qt;
    if (CAUSAL) {
        const int i_min = j0 - up;  // first row that sees key j0
        qt_begin = i_min <= 0 ? 0 : min(n_qt, i_min / 128);
    }
    if (has_lo) {
        const int i_max = min(j0 + 127, n_b - 1) - lo;  // last row that sees the last valid key
        qt_end = i_max < 0 ? 0 : min(n_qt, i_max / 128 + 1);
    }
    if (j0 >= n_b) qt_end = qt_begin;  // no valid key here: dK = dV = 0
    const int qt0 = qt_begin;
    const int n_it = max(0, qt_end - qt_begin);
    WaitCtx wc{p.err, misc + 1, blockIdx.x};

    if (threadIdx.x == 0) {
        for (int i = 0; i < C::kNumBars; ++i) {
            uint32_t count = 1;
            if (i >= C::kBarQdEmpty && i < C::kBarQdEmpty + C::kStages)
                count = 1 + 8 + 1;  // MMA, compute warps, dQ store
            if (i == C::kBarPds || i == C::kBarPds + 1) count = C::kEarlyNext ? 4 : 8;  // compute warps
            if (i == C::kBarDqRead) count = 4;                                           // dQ warps
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
            const uint64_t pol_kv = l2_policy_evict_first();  // read by this CTA only
            const uint64_t pol_q = l2_policy_evict_last();    // read by every key tile of the head
            mbar_arrive_expect_tx(bar(C::kBarKV), 2 * C::kTileBytes);
            for (int c = 0; c < C::kChunks; ++c) {
                tma_load_3d_hint(base + C::kOffK + c * C::kBoxBytes, &tmK, bar(C::kBarKV), c * 64, j0, bh, pol_kv);
                tma_load_3d_hint(base + C::kOffV + c * C::kBoxBytes, &tmV, bar(C::kBarKV), c * 64, j0, bh, pol_kv);
            }
            int issued = 0;
            for (int it = 0; it < n_it; ++it) {
                const int s = it % C::kStages;
                if (it >= C::kStages &&
                    !wait_one(bar(C::kBarQdEmpty + s), ((it / C::kStages) - 1) & 1, wc,
                              kRoleBwdLoad * 1000 + C::kBarQdEmpty + s, it))
                    break;
                const int q0 = (qt0 + it) * 128;
                const uint32_t fb = bar(C::kBarQdFull + s);
                mbar_arrive_expect_tx(fb, 2 * C::kTileBytes + C::kVecBytes);
                for (int c = 0; c < C::kChunks; ++c) {
                    tma_load_3d_hint(sQ(s) + c * C::kBoxBytes, &tmQ, fb, c * 64, q0, bh, pol_q);
                    tma_load_3d_hint(sDO(s) + c * C::kBoxBytes, &tmDO, fb, c * 64, q0, bh, pol_q);
                }
                const size_t vrow = static_cast<size_t>(bh) * p.Npad + q0;
                const uint32_t vdst = base + C::kOffVec + s * C::kVecBytes;
                bulk_load(vdst, p.lse2 + vrow, 512, fb);
                bulk_load(vdst + 512, p.dvec + vrow, 512, fb);
                issued = it + 1;
            }
            // Drain: every copy into this CTA's shared memory has landed before it exits.
            wait_one(bar(C::kBarKV), 0, wc, kRoleBwdLoad * 1000 + 90, 0, false);
            for (int jj = max(0, issued - C::kStages); jj < issued; ++jj)
                wait_one(bar(C::kBarQdFull + jj % C::kStages), (jj / C::kStages) & 1, wc,
                         kRoleBwdLoad * 1000 + 91, jj, false);
        }
        __syncwarp();
    } else if (warp == C::kWarpMma) {
        // ================================ MMA issuer ==================================
        constexpr uint32_t idesc_s = idesc_f16_f32acc(BF16, 128, 128, false);        // K-major x K-major
        constexpr uint32_t idesc_o = idesc_f16_f32acc(BF16, 128, D, true);           // TMEM x MN-major
        constexpr uint32_t idesc_q = idesc_f16_f32acc_ab(BF16, 128, D, true, true);  // MN x MN
        const uint64_t dK_k = sdesc_sw128(base + C::kOffK, 16, 1024);            // K as A, K-major
        const uint64_t dV_k = sdesc_sw128(base + C::kOffV, 16, 1024);            // V as A, K-major
        const uint64_t dK_mn = sdesc_sw128(base + C::kOffK, C::kBoxBytes, 1024); // K as B, MN-major
        const uint64_t dDS = sdesc_sw128(base + C::kOffDS, C::kBoxBytes, 1024);  // dS as A, MN-major
        constexpr uint64_t kStageStep = C::kStageBytes >> 4;
        constexpr uint64_t kTileStep = C::kTileBytes >> 4;
        const uint64_t dQ_k0 = sdesc_sw128(sQ(0), 16, 1024);
        const uint64_t dQ_mn0 = sdesc_sw128(sQ(0), C::kBoxBytes, 1024);

        bool ok = wait_warp(bar(C::kBarKV), 0, wc, kRoleBwdMma * 1000 + C::kBarKV, 0);
        if (ok) tc_fence_after_sync();
        // d = 64: K and V into TMEM, the A operands of S^T and dP^T (K stays in shared memory
        // for dQ). The tensor core runs the MMAs issued after the copies behind them.
        if constexpr (C::kKvTmem) {
            if (ok && n_it > 0) {
                tmem_cp_tile64_warp(tmem + C::colK, dK_k);
                tmem_cp_tile64_warp(tmem + C::colV, dV_k);
            }
        }
        if constexpr (C::kEarlyNext) {
            // d = 64, per Q tile: for each half h (query columns [64h, 64h + 64), warpgroup
            // h), once its P^T/dS^T are ready: dV += P_h^T dO_h and dK += dS_h^T Q_h (K = 64
            // queries), then S^T/dP^T of half h of the next tile, which overwrite P_h^T/dS_h^T
            // only after dV and dK have read them (issue order). dQ of the tile comes last.
            constexpr uint32_t idesc_h = idesc_f16_f32acc(BF16, 128, 64, false);  // N = 64 queries
            constexpr uint64_t kHalfRows = (64 * 128) >> 4;  // 64 rows of a 128-byte-swizzled box
            auto issue_sdp_half = [&](int i, int h) -> bool {
                const int si = i % C::kStages;
                if (h == 0 && !wait_warp_sleep(bar(C::kBarQdFull + si), (i / C::kStages) & 1, wc,
                                         kRoleBwdMma * 1000 + C::kBarQdFull + si, i))
                    return false;
                tc_fence_after_sync();
                const uint64_t q_k = dQ_k0 + si * kStageStep + h * kHalfRows;
                mma_ts_k64_warp(tmem + C::colS + 64u * h, tmem + C::colK, q_k, idesc_h);
                mma_ts_k64_warp(tmem + C::colDP + 64u * h, tmem + C::colV, q_k + kTileStep, idesc_h);
                mma_commit_warp(bar(C::kBarSdp + h));
                return true;
            };
            if (ok && n_it > 0) ok = issue_sdp_half(0, 0) && issue_sdp_half(0, 1);
            for (int it = 0; it < n_it && ok; ++it) {
                const int s = it % C::kStages;
                const uint64_t q_mn = dQ_mn0 + s * kStageStep;
                const uint64_t do_mn = q_mn + kTileStep;
                for (int h = 0; h < 2 && ok; ++h) {
                    ok = wait_warp_sleep(bar(C::kBarPds + h), it & 1, wc, kRoleBwdMma * 1000 + C::kBarPds + h, it);
                    if (!ok) break;
                    tc_fence_after_sync();
                    const uint32_t acc = (it > 0 || h > 0) ? 1u : 0u;
                    mma_pv64_tmem_warp(tmem + C::colDV, tmem + C::colS + 64u * h, do_mn + h * kHalfRows, idesc_o, acc);
                    mma_pv64_tmem_warp(tmem + C::colDK, tmem + C::colDP + 64u * h, q_mn + h * kHalfRows, idesc_o, acc);
                    if (it + 1 < n_it) ok = issue_sdp_half(it + 1, h);
                }
                // The dQ columns of the previous tile must have been read out.
                if (ok && it > 0)
                    ok = wait_warp_sleep(bar(C::kBarDqRead), (it - 1) & 1, wc, kRoleBwdMma * 1000 + C::kBarDqRead, it);
                if (!ok) break;
                tc_fence_after_sync();
                mma_mn128_warp(tmem + C::colDQ, dDS + (((it & 1) * (128 * 128 * 2)) >> 4), dK_mn, idesc_q, 0u);
                mma_commit_warp(bar(C::kBarDqFull));
                mma_commit_warp(bar(C::kBarQdEmpty + s));
            }
        } else {
            // d = 128, per Q tile: S^T and dP^T (the dQ tile of the previous one lives in the
            // S^T columns, so it must have been read out), then dV, dK and dQ.
            for (int it = 0; it < n_it && ok; ++it) {
                const int s = it % C::kStages;
                if (it > 0 &&
                    !wait_warp(bar(C::kBarDqRead), (it - 1) & 1, wc, kRoleBwdMma * 1000 + C::kBarDqRead, it)) {
                    ok = false;
                    break;
                }
                if (!wait_warp(bar(C::kBarQdFull + s), (it / C::kStages) & 1, wc,
                               kRoleBwdMma * 1000 + C::kBarQdFull + s, it)) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                const uint64_t q_k = dQ_k0 + s * kStageStep;
                const uint64_t do_k = q_k + kTileStep;
#pragma unroll
                for (int c = 0; c < C::kChunks; ++c) {
                    const uint64_t off = (c * C::kBoxBytes) >> 4;
                    mma_qk64_warp(tmem + C::colS, dK_k + off, q_k + off, idesc_s, c > 0 ? 1u : 0u);
                }
#pragma unroll
                for (int c = 0; c < C::kChunks; ++c) {
                    const uint64_t off = (c * C::kBoxBytes) >> 4;
                    mma_qk64_warp(tmem + C::colDP, dV_k + off, do_k + off, idesc_s, c > 0 ? 1u : 0u);
                }
                mma_commit_warp(bar(C::kBarSdp));
                if (!wait_warp(bar(C::kBarPds), it & 1, wc, kRoleBwdMma * 1000 + C::kBarPds, it)) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                const uint64_t q_mn = dQ_mn0 + s * kStageStep;
                const uint64_t do_mn = q_mn + kTileStep;
                mma_pv128_halves_warp(tmem + C::colDV, tmem + C::colS, do_mn, idesc_o, it > 0 ? 1u : 0u);
                mma_pv128_halves_warp(tmem + C::colDK, tmem + C::colDP, q_mn, idesc_o, it > 0 ? 1u : 0u);
                mma_mn128_warp(tmem + C::colDQ, dDS, dK_mn, idesc_q, 0u);
                mma_commit_warp(bar(C::kBarDqFull));
                mma_commit_warp(bar(C::kBarQdEmpty + s));
            }
        }
        if (ok) mma_commit_warp(bar(C::kBarAcc));
        // Drain: all MMAs issued by this warp are complete before TMEM is freed.
        mma_commit_warp(bar(C::kBarDrain));
        wait_warp(bar(C::kBarDrain), 0, wc, kRoleBwdMma * 1000 + C::kBarDrain, 0, false);
        __syncwarp();
    } else if (warp >= C::kWarpDq) {
        // ================================ dQ read-out ==================================
        // TMEM lane r of the dQ tile is query q0 + r; the tile is added to the fp32
        // accumulator (other CTAs add the other key tiles' parts) through the swizzled
        // ring stage of its iteration and a TMA bulk reduce-add.
        const uint32_t wq = warp - C::kWarpDq;
        const uint32_t r = wq * 32u + lane;
        const uint32_t lane_base = tmem_addr(tmem, wq * 32u, 0);
        const bool leader = warp == C::kWarpDq && lane == 0;
        if (leader) tma_prefetch_desc(&tmDQ);
        for (int it = 0; it < n_it; ++it) {
            if (!wait_warp_sleep(bar(C::kBarDqFull), it & 1, wc, kRoleBwdDq * 1000 + C::kBarDqFull, it)) break;
            tc_fence_after_sync();
            const int q0 = (qt0 + it) * 128;
            const int s = it % C::kStages;
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
        // Every reduce is complete in global memory before the CTA exits.
        if (leader) tma_store_wait_all();
    } else {
        // ================================ compute warpgroups ==========================
        // Warpgroup h handles query columns [64h, 64h + 64) of S^T and dP^T.
        const uint32_t h = warp >> 2;
        const uint32_t wq = warp & 3u;               // TMEM lane quarter
        const uint32_t r = wq * 32u + lane;          // key row in the tile = TMEM lane
        const int j = j0 + static_cast<int>(r);      // this thread's key
        const uint32_t lane_base = tmem_addr(tmem, wq * 32u, 0);
        const float qk = p.qk_scale;
        const float2 qk2 = make_float2(qk, qk);
        const uint32_t sDS0 = base + C::kOffDS + h * C::kBoxBytes + r * 128u;
        const int hb = C::kEarlyNext ? static_cast<int>(h) : 0;  // this half's S/dP and P/dS barriers
        bool ok = true;
        for (int it = 0; it < n_it && ok; ++it) {
            const int s = it % C::kStages;
            const int q0 = (qt0 + it) * 128;
            if (!wait_warp_sleep(bar(C::kBarQdFull + s), (it / C::kStages) & 1, wc,
                           kRoleBwdCompute * 1000 + C::kBarQdFull + s, it) ||
                !wait_warp_sleep(bar(C::kBarSdp + hb), it & 1, wc, kRoleBwdCompute * 1000 + C::kBarSdp + hb, it)) {
                ok = false;
                break;
            }
            // S^T(it) and dP^T(it) complete also means the dQ product that last read this
            // iteration's dS buffer (iteration it-1, or it-2 with two buffers; issued before
            // them) has finished reading it.
            tc_fence_after_sync();
            const uint32_t sDS = sDS0 + (C::kEarlyNext ? (it & 1) * (128 * 128 * 2) : 0);
            const float* vec = reinterpret_cast<const float*>(smem_bwd + C::kOffVec + s * C::kVecBytes);
            const float* nlse2 = vec + 64 * h;        // -LSE log2(e) of this half's query rows
            const float* ndvec = vec + 128 + 64 * h;  // -D
            const bool key_out = j >= n_b;  // padded (or past Nk) key row: P = 0
            // Whether some query row of this tile may not see this thread's key.
            const bool mask_tile = key_out || (CAUSAL && j > q0 + up) || (has_lo && j < q0 + 127 + lo);
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
                    const float2 y0 = __ffma2_rn(make_float2(__uint_as_float(sr[e]), __uint_as_float(sr[e + 1])), qk2,
                                                 make_float2(nl.x, nl.y));
                    const float2 y1 = __ffma2_rn(make_float2(__uint_as_float(sr[e + 2]), __uint_as_float(sr[e + 3])),
                                                 qk2, make_float2(nl.z, nl.w));
                    float pe[4] = {ex2_ftz(y0.x), ex2_ftz(y0.y), ex2_ftz(y1.x), ex2_ftz(y1.y)};
                    if (mask_tile) {
                        const int q = q0 + 64 * static_cast<int>(h) + col;  // query row of pe[0]
#pragma unroll
                        for (int k = 0; k < 4; ++k)
                            if (key_out || (CAUSAL && j > q + k + up) || (has_lo && j < q + k + lo)) pe[k] = 0.f;
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
                mbar_arrive(bar(C::kBarPds + hb));
                mbar_arrive(bar(C::kBarQdEmpty + s));
            }
        }
        // ---- epilogue: dV and dK of this thread's key, columns [d/2 h, d/2 (h+1)) -----
        // A key tile no query row sees (EXT only) stores zeros: its TMEM was never written.
        if (ok) ok = wait_warp(bar(C::kBarAcc), 0, wc, kRoleBwdCompute * 1000 + C::kBarAcc, n_it);
        if (ok) {
            const bool any = n_it > 0;
            if (any) tc_fence_after_sync();
#pragma unroll 1
            for (int which = 0; which < 2; ++which) {
                const uint32_t col = which == 0 ? C::colDV : C::colDK;
                const float mul = which == 0 ? 1.f : p.scale;
                uint8_t* out = static_cast<uint8_t*>(which == 0 ? p.dv : p.dk);
#pragma unroll 1
                for (int c = h * (D / 64); c < (h + 1) * (D / 64); ++c) {
                    uint32_t o[32];
                    if (any) {
                        tmem_ld32(lane_base + col + 32 * c, o);
                        tmem_ld_wait();
                        reg_fence(o);
                    } else {
#pragma unroll
                        for (int e = 0; e < 32; ++e) o[e] = 0u;
                    }
                    if (j < Nk) {
                        uint4* row = reinterpret_cast<uint4*>(out + ((static_cast<size_t>(bh) * Nk + j) * D + 32 * c) * 2);
#pragma unroll
                        for (int e = 0; e < 32; e += 8)
                            row[e >> 3] = make_uint4(
                                pack2<BF16>(__uint_as_float(o[e]) * mul, __uint_as_float(o[e + 1]) * mul),
                                pack2<BF16>(__uint_as_float(o[e + 2]) * mul, __uint_as_float(o[e + 3]) * mul),
                                pack2<BF16>(__uint_as_float(o[e + 4]) * mul, __uint_as_float(o[e + 5]) * mul),
                                pack2<BF16>(__uint_as_float(o[e + 6]) * mul, __uint_as_float(o[e + 7]) * mul));
                    }
                }
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

// -D_i = -rowsum(dO * O), -lse2_i = -LSE_i log2(e) (-inf where LSE = -inf or i >= N, so
// that P = 0 there), the zeroed dQ accumulator and the persistent kernel's zeroed work
// counter. Each thread takes 8 consecutive elements (16 bytes of O and of dO, 32 bytes of
// the accumulator) of one row of [BH][Npad], d/8 threads per row summed by shuffles. The
// main kernel adds the vectors, so they are stored negated.
template <bool BF16>
__global__ void __launch_bounds__(256) attn_bwd_prep_kernel(const BwdPrepParams p) {
    const int tpr = p.d / 8;  // threads per row: 8 or 16, a divisor of the warp
    const long long t = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    const long long row = t / tpr;
    const int sub = static_cast<int>(t % tpr);
    if (blockIdx.x == 0 && threadIdx.x == 0) *p.item_counter = 0;
    const bool valid = row < static_cast<long long>(p.BH) * p.Npad;
    const int bh = valid ? static_cast<int>(row / p.Npad) : 0, i = valid ? static_cast<int>(row % p.Npad) : 0;
    float acc = 0.f;
    if (valid && i < p.N) {
        const size_t off = (static_cast<size_t>(bh) * p.N + i) * p.d + sub * 8;
        const uint4 o = *reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.o) + off);
        const uint4 g = *reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.dout) + off);
        const uint32_t ow[4] = {o.x, o.y, o.z, o.w}, gw[4] = {g.x, g.y, g.z, g.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 a = unpack2<BF16>(ow[e]), b = unpack2<BF16>(gw[e]);
            acc = fmaf(a.x, b.x, acc);
            acc = fmaf(a.y, b.y, acc);
        }
        float4* z = reinterpret_cast<float4*>(p.dq_acc + off);
        z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
        z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    for (int w = tpr / 2; w > 0; w >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, w);
    if (valid && sub == 0) {
        const size_t vrow = static_cast<size_t>(bh) * p.Npad + i;
        if (i >= p.N) {
            p.lse2[vrow] = -INFINITY;
            p.dvec[vrow] = -0.f;
        } else {
            const float l = p.lse[static_cast<size_t>(bh) * p.N + i];
            p.lse2[vrow] = l == -INFINITY ? -INFINITY : -(l * 1.4426950408889634f);
            p.dvec[vrow] = -acc;
        }
    }
}

// dQ = scale * dq_acc, rounded once to the dtype. Four elements per thread.
template <bool BF16>
__global__ void __launch_bounds__(256) attn_bwd_convert_kernel(const BwdConvertParams p) {
    const long long i4 = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) * 4;
    if (i4 >= p.n) return;
    const float4 a = *reinterpret_cast<const float4*>(p.dq_acc + i4);
    uint2 out = make_uint2(pack2<BF16>(a.x * p.scale, a.y * p.scale), pack2<BF16>(a.z * p.scale, a.w * p.scale));
    *reinterpret_cast<uint2*>(static_cast<uint8_t*>(p.dq) + i4 * 2) = out;
}

}  // namespace attn_sm103
