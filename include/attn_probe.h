/*
 * attn_probe.h -- test hook that runs the two tensor-core products of the
 * attention forward on one 128-row tile, through exactly the TMA, shared-memory
 * descriptor, tcgen05 and TMEM forms the forward kernel uses.
 *
 * The products are the two contractions of the FlashAttention-2 inner loop
 * ("如何用 profiler 逐步优化 Triton FlashAttention-2 kernel", Round 4 / exp2:
 * S_ij = Q_i K_j^T on raw scores; Round 4 / The P cast: P rounded to the input
 * dtype, then P V_j on the 16-bit tensor-core path).
 *
 * It exists so that descriptor or layout mistakes show up as a wrong number on
 * one tile rather than as a wrong attention output. Not part of the product API.
 */
#ifndef ATTN_GB300_ATTN_PROBE_H
#define ATTN_GB300_ATTN_PROBE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/*
 * attn_probe_tile -- one CTA, synchronous on `stream` (it synchronises before
 * returning).
 *  q, k, v : DEVICE, contiguous row-major [128][d] of `dtype` (attn_dtype_t).
 *  p       : DEVICE, contiguous row-major [128][128] of `dtype`.
 *  s_out   : DEVICE, [128][128] fp32, receives S = q k^T   (tcgen05, SMEM x SMEM).
 *  o_out   : DEVICE, [128][d]   fp32, receives O = p v     (tcgen05, P from TMEM,
 *            V as an MN-major shared-memory operand).
 *  d in {64, 128}. All pointers 16-byte aligned.
 * Returns an attn_status_t (ATTN_ERR_TIMEOUT if a device wait gave up).
 */
int attn_probe_tile(const void* q, const void* k, const void* v, const void* p, float* s_out,
                    float* o_out, int64_t d, int dtype, void* stream);

/*
 * attn_probe_wait_timeout -- failure-detection test hook. Launches one CTA whose two
 * warps wait, through the same bounded mbarrier wait the attention kernels use, on
 * barriers that nothing ever completes: the first gives up after the kernels' wait
 * limit (1.5 s) and records {code 1, block 0, 9000, 7} in the device status record;
 * the second starts half a second later, sees the CTA's abort flag and gives up
 * without recording. No fault, trap
 * or hang is involved and the context stays usable. Synchronous on `stream` (current
 * device). Returns ATTN_ERR_TIMEOUT when the timeout was recorded (the expected
 * outcome), ATTN_OK if not, ATTN_ERR_CUDA on a CUDA error. The pages have no
 * counterpart; it exists to test the timeout path on a GPU.
 */
int attn_probe_wait_timeout(void* stream);

/*
 * attn_probe_plan_split / attn_probe_plan_host -- the host planners of attn_fwd_kv
 * (split of the keys over CTAs) and attn_fwd_host (chunks of heads) for a GPU with
 * `sms` SMs, so that tests can check them for other SM counts without such a GPU.
 * The entry points themselves plan with the SM count of the device they run on.
 * Pure host arithmetic.
 *  plan_split: out[0] = key ranges (1: no split), out[1] = key tiles per range,
 *              out[2] = workspace bytes the plan uses; `ws_bytes` caps the ranges
 *              as it does for attn_fwd_kv. Returns ATTN_OK or ATTN_ERR_INVALID_ARG.
 *  plan_host:  returns the number of chunks and stores the heads per chunk.
 */
int attn_probe_plan_split(int64_t BH, int64_t Nq, int64_t Nk, int64_t d, size_t ws_bytes, int64_t sms,
                          int64_t out[3]);
int64_t attn_probe_plan_host(int64_t BH, int64_t N, int64_t sms, int64_t* heads_per_chunk);

/*
 * attn_probe_plan_decode -- the plan of the streaming decode kernel that attn_fwd_kv
 * runs for Nq <= 4 without padding or window, for a GPU with `sms` SMs and a
 * workspace of `ws_bytes`: out[0] = key ranges per head (1: no workspace used, the
 * kernel writes O and LSE itself), out[1] = keys per range (a multiple of 32),
 * out[2] = CTAs launched, out[3] = workspace bytes the plan uses. Host arithmetic
 * only. Returns ATTN_ERR_INVALID_ARG for sizes outside the decode kernel's range.
 */
int attn_probe_plan_decode(int64_t BH, int64_t Nq, int64_t Nk, int64_t d, size_t ws_bytes, int64_t sms,
                           int64_t out[4]);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_GB300_ATTN_PROBE_H */
