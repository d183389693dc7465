// One (head dimension, dtype) pair of forward-kernel instances: causal or not, whole
// key range or split of the keys.
// Compiled once per pair with -DATTN_INST_D=<64|128> -DATTN_INST_BF16=<0|1>.
#include <atomic>

#include "attn_fwd_kernel.cuh"
#include "attn_fwd_persist.cuh"
#include "attn_internal.h"

#if !defined(ATTN_INST_D) || !defined(ATTN_INST_BF16)
#error "compile with -DATTN_INST_D=<64|128> -DATTN_INST_BF16=<0|1>"
#endif

#ifndef ATTN_PERSIST
#define ATTN_PERSIST 1
#endif

namespace attn_sm103 {
namespace {

constexpr bool kPersistEnabled = ATTN_PERSIST != 0;

template <int D, bool CAUSAL, bool BF16, bool SPLIT, bool EXT>
cudaError_t launch_one(const CUtensorMap* m, const FwdParams& p, cudaStream_t s) {
    using C = FwdCfg<D>;
    auto* kern = attn_fwd_kernel<D, CAUSAL, BF16, SPLIT, EXT>;
    // The dynamic shared-memory opt-in is per device; remember which devices have it.
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
    const dim3 grid(static_cast<unsigned>(p.n_ctiles) * static_cast<unsigned>(p.BH),
                    SPLIT ? static_cast<unsigned>(p.n_splits) : 1u);
    kern<<<grid, C::kThreads, C::kSmemBytes, s>>>(m[0], m[1], m[2], m[3], p);
    return cudaGetLastError();
}

// The persistent head-dimension-64 forward: one CTA per SM (fewer if there are fewer
// work items). Its warpgroups rebalance registers with setmaxnreg, which needs the
// kernel to be launched with exactly kPersistLaunchRegs registers per thread; any
// other count is refused here rather than risking an increase that cannot be met.
template <bool CAUSAL, bool BF16>
cudaError_t launch_persist(const CUtensorMap* m, const FwdParams& p, cudaStream_t s) {
    using C = PersistCfg;
    auto* kern = attn_fwd_persist_kernel<CAUSAL, BF16>;
    static std::atomic<uint64_t> configured{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = dev < 64 ? (1ull << dev) : 0ull;
    if (!bit || !(configured.load(std::memory_order_acquire) & bit)) {
        cudaFuncAttributes fa;
        e = cudaFuncGetAttributes(&fa, kern);
        if (e != cudaSuccess) return e;
        if (fa.numRegs != kPersistLaunchRegs) return cudaErrorInvalidConfiguration;
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
        if (e != cudaSuccess) return e;
        configured.fetch_or(bit, std::memory_order_acq_rel);
    }
    const int sms = device_sm_count(dev);
    if (sms < 1) return cudaErrorInvalidDevice;
    const long long items = static_cast<long long>(p.n_ctiles) * p.BH;
    const unsigned grid = static_cast<unsigned>(items < sms ? items : sms);
    kern<<<grid, C::kThreads, C::kSmemBytes, s>>>(m[0], m[1], m[2], m[3], p);
    return cudaGetLastError();
}

}  // namespace

#define ATTN_CAT2(a, b) a##b
#define ATTN_CAT(a, b) ATTN_CAT2(a, b)
#if ATTN_INST_BF16
#define ATTN_DT_SUFFIX bf16
#else
#define ATTN_DT_SUFFIX f16
#endif
#define ATTN_LAUNCH_NAME ATTN_CAT(ATTN_CAT(ATTN_CAT(launch_fwd_d, ATTN_INST_D), _), ATTN_DT_SUFFIX)

cudaError_t ATTN_LAUNCH_NAME(bool causal, bool split, bool ext, const CUtensorMap* maps, const FwdParams& p,
                             cudaStream_t s) {
    constexpr bool kBf16 = ATTN_INST_BF16 != 0;
    constexpr int kD = ATTN_INST_D;
    if (ext) {
        if (split)
            return causal ? launch_one<kD, true, kBf16, true, true>(maps, p, s)
                          : launch_one<kD, false, kBf16, true, true>(maps, p, s);
        return causal ? launch_one<kD, true, kBf16, false, true>(maps, p, s)
                      : launch_one<kD, false, kBf16, false, true>(maps, p, s);
    }
    if (split)
        return causal ? launch_one<kD, true, kBf16, true, false>(maps, p, s)
                      : launch_one<kD, false, kBf16, true, false>(maps, p, s);
    // The square problem (Nq = Nk, top-left causal mask) at head dimension 64 runs on the
    // persistent kernel; every other form on the one-item kernel.
    if constexpr (kD == 64 && kPersistEnabled) {
        if (p.Nq == p.Nk && p.align_br == 0)
            return causal ? launch_persist<true, kBf16>(maps, p, s) : launch_persist<false, kBf16>(maps, p, s);
    }
    return causal ? launch_one<kD, true, kBf16, false, false>(maps, p, s)
                  : launch_one<kD, false, kBf16, false, false>(maps, p, s);
}

}  // namespace attn_sm103
