// The device scratch of attn_fwd_kv_static, in a translation unit of its own: CUDA loads
// a module's device memory when the module is first used, so only a process that calls
// attn_fwd_kv_static holds these 16 MiB per device; attn_fwd and the other entry points
// never touch this module.
#include <atomic>
#include <cstdint>

#include <cuda_runtime.h>

#include "attn_internal.h"

namespace attn_sm103 {

// Split partials of attn_fwd_kv_static live in this file-scope array instead of caller
// memory. A plan needs B*H * splits * Nq * (d+1) * 4 bytes; keys are split only while
// B*H * ceil(Nq/256) < 2 * SMs, into at most ceil(8 * SMs / (B*H)) ranges, so
// B*H * splits < 10 * SMs and 16 MiB holds every plan with Nq <= 16 on GPUs of up to 200
// SMs (at most 2000 * 16 * 129 * 4 bytes, about 16.5e6; a GB300's 152 SMs need 12.5e6).
static __device__ __align__(256) unsigned char g_kv_scratch[kStaticScratchBytes];

// Device address of g_kv_scratch on device `dev`, which must be current (looked up
// with cudaGetSymbolAddress once per device and cached).
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

}  // namespace attn_sm103
