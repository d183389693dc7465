// One (head dimension, dtype) pair of backward-kernel instances: causal or not, plain or
// with padding / windows / Nq != Nk.
// Compiled once per pair with -DATTN_INST_D=<64|128> -DATTN_INST_BF16=<0|1>.
#include <atomic>

#include "attn_bwd_internal.h"
#include "attn_bwd_kernel.cuh"
#include "attn_bwd_persist.cuh"

#if !defined(ATTN_INST_D) || !defined(ATTN_INST_BF16)
#error "compile with -DATTN_INST_D=<64|128> -DATTN_INST_BF16=<0|1>"
#endif

namespace attn_sm103 {
namespace {

template <int D, bool CAUSAL, bool BF16, bool EXT>
cudaError_t launch_bwd_one(const CUtensorMap* m, const BwdParams& p, cudaStream_t s) {
    using C = BwdCfg<D>;
    auto* kern = attn_bwd_kernel<D, CAUSAL, BF16, EXT>;
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
    const unsigned grid = static_cast<unsigned>(p.n_ktiles) * static_cast<unsigned>(p.BH);
    kern<<<grid, C::kThreads, C::kSmemBytes, s>>>(m[0], m[1], m[2], m[3], m[4], p);
    return cudaGetLastError();
}

// The persistent d = 64 backward (no padding or window masks): one CTA per SM, fewer if
// there are fewer key tiles in all.
template <bool CAUSAL, bool BF16>
cudaError_t launch_bwd_persist(const CUtensorMap* m, const BwdParams& p, cudaStream_t s) {
    using C = BwdCfg<64>;
    auto* kern = attn_bwd_persist_kernel<CAUSAL, BF16>;
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
    const int sms = device_sm_count(dev);
    if (sms < 1) return cudaErrorInvalidDevice;
    const long long items = static_cast<long long>(p.n_ktiles) * p.BH;
    const unsigned grid = static_cast<unsigned>(items < sms ? items : sms);
    kern<<<grid, C::kThreads, C::kSmemBytes, s>>>(m[0], m[1], m[2], m[3], m[4], p);
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
#define ATTN_BWD_NAME ATTN_CAT(ATTN_CAT(ATTN_CAT(launch_bwd_d, ATTN_INST_D), _), ATTN_DT_SUFFIX)

cudaError_t ATTN_BWD_NAME(bool causal, bool ext, const CUtensorMap* maps, const BwdParams& p, cudaStream_t s) {
    constexpr bool kBf16 = ATTN_INST_BF16 != 0;
    constexpr int kD = ATTN_INST_D;
    if (ext)
        return causal ? launch_bwd_one<kD, true, kBf16, true>(maps, p, s)
                      : launch_bwd_one<kD, false, kBf16, true>(maps, p, s);
#if ATTN_INST_D == 64
    return causal ? launch_bwd_persist<true, kBf16>(maps, p, s) : launch_bwd_persist<false, kBf16>(maps, p, s);
#else
    return causal ? launch_bwd_one<kD, true, kBf16, false>(maps, p, s)
                  : launch_bwd_one<kD, false, kBf16, false>(maps, p, s);
#endif
}

}  // namespace attn_sm103
