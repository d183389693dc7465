// Tile probe: the two tensor-core products of the forward kernel on one 128-row
// tile, through the same TMA maps, shared-memory descriptors, instruction
// descriptors and TMEM layouts (see include/attn_probe.h).
#include <cuda_runtime.h>

#include "attn.h"
#include "attn_probe.h"
#include "attn_fwd_kernel.cuh"
#include "attn_internal.h"

namespace attn_sm103 {
namespace {

template <int D, bool BF16>
__global__ void __launch_bounds__(128, 1)
    probe_tile_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                      const __grid_constant__ CUtensorMap tmV, const uint32_t* __restrict__ p_in,
                      float* __restrict__ s_out, float* __restrict__ o_out, uint32_t* err) {
    constexpr int kTile = 128 * D * 2;
    constexpr int kBox = 128 * 128;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* smem = smem_raw + (base - raw);
    const uint32_t sQ = base, sK = base + kTile, sV = base + 2 * kTile;
    const uint32_t bars = base + 3 * kTile;  // [0] loads, [1] S done, [2] O done
    uint32_t* misc = reinterpret_cast<uint32_t*>(smem + 3 * kTile + 64);
    const uint32_t warp = threadIdx.x >> 5, lane = threadIdx.x & 31u;
    const uint32_t r = threadIdx.x;  // row = TMEM lane

    if (threadIdx.x == 0) {
        for (int i = 0; i < 3; ++i) mbar_init(bars + 8 * i, 1);
        misc[1] = 0u;
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(smem_addr(misc), 256);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = misc[0];
    WaitCtx wc{err, misc + 1, 0};

    if (threadIdx.x == 0) {
        mbar_arrive_expect_tx(bars, 3 * kTile);
        for (int c = 0; c < D / 64; ++c) {
            tma_load_3d(sQ + c * kBox, &tmQ, bars, c * 64, 0, 0);
            tma_load_3d(sK + c * kBox, &tmK, bars, c * 64, 0, 0);
            tma_load_3d(sV + c * kBox, &tmV, bars, c * 64, 0, 0);
        }
    }
    bool ok = wait_warp(bars, 0, wc, 1, 0);
    if (ok && warp == 0) {
        tc_fence_after_sync();
        constexpr uint32_t idesc_s = idesc_f16_f32acc(BF16, 128, 128, false);
#pragma unroll
        for (int c = 0; c < D / 64; ++c)
            mma_qk64_warp(tmem, sdesc_sw128(sQ + c * kBox, 16, 1024), sdesc_sw128(sK + c * kBox, 16, 1024),
                          idesc_s, c > 0 ? 1u : 0u);
        mma_commit_warp(bars + 8);
    }
    if (ok) ok = wait_warp(bars + 8, 0, wc, 2, 0);
    const uint32_t tS = tmem_addr(tmem, warp * 32u, 0);
    const uint32_t tO = tmem_addr(tmem, warp * 32u, 128);
    if (ok) {
        tc_fence_after_sync();
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            uint32_t v[32];
            tmem_ld32(tS + c * 32, v);
            tmem_ld_wait();
            reg_fence(v);
            for (int e = 0; e < 32; ++e) s_out[r * 128 + c * 32 + e] = __uint_as_float(v[e]);
        }
        // P (row r, 128 16-bit values = 64 packed words) into the S columns.
        uint32_t pk[2][32];
        for (int i = 0; i < 64; ++i) pk[i >> 5][i & 31] = p_in[r * 64 + i];
        tmem_st32(tS, pk[0]);
        tmem_st32(tS + 32, pk[1]);
        tmem_st_wait();
    }
    tc_fence_before_sync();
    __syncthreads();
    ok = ok && misc[1] == 0u;
    if (ok && warp == 0) {
        tc_fence_after_sync();
        constexpr uint32_t idesc_o = idesc_f16_f32acc(BF16, 128, D, true);
        mma_pv128_warp(tmem + 128, tmem, sdesc_sw128(sV, kBox, 1024), idesc_o, 0u);
        mma_commit_warp(bars + 16);
    }
    if (ok) ok = wait_warp(bars + 16, 0, wc, 3, 0);
    if (ok) {
        tc_fence_after_sync();
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
            uint32_t v[32];
            tmem_ld32(tO + c * 32, v);
            tmem_ld_wait();
            reg_fence(v);
            for (int e = 0; e < 32; ++e) o_out[r * D + c * 32 + e] = __uint_as_float(v[e]);
        }
    }
    // Drain the tensor core before freeing TMEM (covers an aborted run too).
    if (warp == 0) {
        mma_commit_warp(bars + 16);
        wait_warp(bars + 16, ok ? 1 : 0, wc, 4, 0, false);
    }
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, 256);
    }
}

template <int D, bool BF16>
cudaError_t launch_probe(const CUtensorMap* m, const void* p, float* s, float* o, uint32_t* err,
                         cudaStream_t st) {
    constexpr int kSmem = 3 * 128 * D * 2 + 128 + 1024;
    auto* kern = probe_tile_kernel<D, BF16>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e != cudaSuccess) return e;
    kern<<<1, 128, kSmem, st>>>(m[0], m[1], m[2], static_cast<const uint32_t*>(p), s, o, err);
    return cudaGetLastError();
}

}  // namespace
}  // namespace attn_sm103

using namespace attn_sm103;

namespace attn_sm103 {
namespace {

// Two warps wait, through the kernels' own bounded wait, on mbarriers that nothing ever
// completes: warp 0 gives up when its time limit runs out and records the timeout; warp 1
// sees the CTA's abort flag and gives up without recording. Shared memory only.
__global__ void __launch_bounds__(64, 1) probe_wait_timeout_kernel(uint32_t* err) {
    __shared__ __align__(8) uint64_t bars[2];
    __shared__ uint32_t abort_flag;
    const uint32_t warp = threadIdx.x >> 5;
    if (threadIdx.x == 0) {
        mbar_init(smem_addr(&bars[0]), 1);
        mbar_init(smem_addr(&bars[1]), 1);
        abort_flag = 0u;
        fence_mbar_init();
    }
    __syncthreads();
    WaitCtx wc{err, &abort_flag, blockIdx.x};
    const uint32_t where = 9000u + warp;  // role 9 (this probe), barrier = warp
    if (warp == 1) {  // start half a second later, so that warp 0's limit runs out first
        const uint64_t t0 = global_timer_ns();
        while (global_timer_ns() - t0 < 500ull * 1000ull * 1000ull) {
        }
    }
    wait_warp(smem_addr(&bars[warp]), 0, wc, where, 7u + warp, true);
    __syncthreads();
}

}  // namespace
}  // namespace attn_sm103

extern "C" int attn_probe_wait_timeout(void* stream) {
    using namespace attn_sm103;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    uint32_t* status = status_ptr(dev, &e);
    if (!status) return cuda_fail(e);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    e = cudaMemsetAsync(status, 0, 16, st);
    if (e != cudaSuccess) return cuda_fail(e);
    probe_wait_timeout_kernel<<<1, 64, 0, st>>>(status);
    e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e);
    e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_fail(e);
    uint32_t host[4] = {0, 0, 0, 0};
    e = cudaMemcpy(host, status, sizeof(host), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e);
    return host[0] ? ATTN_ERR_TIMEOUT : ATTN_OK;
}

extern "C" int attn_probe_tile(const void* q, const void* k, const void* v, const void* p, float* s_out,
                               float* o_out, int64_t d, int dtype, void* stream) {
    if (!q || !k || !v || !p || !s_out || !o_out) return ATTN_ERR_INVALID_ARG;
    if (dtype != ATTN_FP16 && dtype != ATTN_BF16) return ATTN_ERR_INVALID_ARG;
    if (d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED;
    const uintptr_t ptrs[6] = {reinterpret_cast<uintptr_t>(q), reinterpret_cast<uintptr_t>(k),
                               reinterpret_cast<uintptr_t>(v), reinterpret_cast<uintptr_t>(p),
                               reinterpret_cast<uintptr_t>(s_out), reinterpret_cast<uintptr_t>(o_out)};
    for (uintptr_t a : ptrs)
        if (a % 16u) return ATTN_ERR_MISALIGNED;
    int dev = 0;
    cudaError_t e = select_device_of(q, &dev);
    if (e != cudaSuccess) return cuda_fail(e);
    PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn(&e);
    if (!enc) return cuda_fail(e);
    uint32_t* status = status_ptr(dev, &e);
    if (!status) return cuda_fail(e);
    alignas(64) CUtensorMap maps[3];
    const void* src[3] = {q, k, v};
    for (int i = 0; i < 3; ++i) {
        const CUresult r = make_map(enc, &maps[i], src[i], 1, 128, d, dtype);
        if (r != CUDA_SUCCESS) {
            g_last_cuda_error = 100000 + static_cast<int>(r);
            return ATTN_ERR_CUDA;
        }
    }
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    e = cudaMemsetAsync(status, 0, 16, st);
    if (e != cudaSuccess) return cuda_fail(e);
    if (d == 64)
        e = dtype == ATTN_BF16 ? launch_probe<64, true>(maps, p, s_out, o_out, status, st)
                               : launch_probe<64, false>(maps, p, s_out, o_out, status, st);
    else
        e = dtype == ATTN_BF16 ? launch_probe<128, true>(maps, p, s_out, o_out, status, st)
                               : launch_probe<128, false>(maps, p, s_out, o_out, status, st);
    if (e != cudaSuccess) return cuda_fail(e);
    e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_fail(e);
    uint32_t host[4];
    e = cudaMemcpy(host, status, sizeof(host), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e);
    return host[0] ? ATTN_ERR_TIMEOUT : ATTN_OK;
}
