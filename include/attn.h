/*
 * attn.h -- C ABI of the fused exact scaled-dot-product attention forward for
 * NVIDIA GB300 (sm_103a).
 *
 * The operation (plain definition, per head and query row i):
 *
 *     O[i,:]  = sum_{j in V_i} softmax_j(scale * q_i . k_j) * v_j
 *     LSE[i]  = ln sum_{j in V_i} exp(scale * q_i . k_j)
 *     V_i     = { 0 <= j < N }, or { 0 <= j <= i } under the causal mask
 *
 * Sources for the operation and its argument list:
 *  - "Programming an attention kernel in Triton", Kernel 4 (a self-attention
 *    kernel): scores = scale * Q K^T, masked keys set to -inf, row softmax,
 *    weights times V.
 *  - "如何用 profiler 逐步优化 Triton FlashAttention-2 kernel" (profile-driven
 *    FlashAttention-2 page), "What the compiler did": the kernel takes
 *    Q, K, V, O, L, the sequence lengths, the scale, the head dimension D and
 *    is_causal; "Round 4 / Causal tile-skipping" fixes the mask as
 *    k_pos <= q_pos (top-left aligned); "Round 4 / exp2" fixes L as the
 *    natural-log logsumexp of the scaled scores.
 *  - "如何用 profiler ...", "A small program to profile": Q, K, V, O are stored
 *    as contiguous (B*H, N, D) blocks and viewed as (B, H, N, D).
 *
 * Conventions shared by every call below:
 *  - q, k, v, o: DEVICE pointers to contiguous row-major [B, H, N, d] arrays of
 *    `dtype` (fp16 or bf16). lse: DEVICE pointer to a contiguous [B, H, N] fp32
 *    array. All five must be 16-byte aligned. o and lse must not overlap each
 *    other or the inputs. The inputs are only read.
 *  - The caller owns and allocates all device memory. The library allocates no
 *    device memory; it keeps a few host-side caches (function attributes and
 *    the driver entry point) that are set up on first use.
 *  - `stream` is a cudaStream_t (NULL = the legacy default stream). The call is
 *    asynchronous on that stream; argument errors are reported synchronously,
 *    before anything is enqueued.
 *  - Supported: d in {64, 128}; B, H, N >= 1; B*H < 2^31; N < 2^31;
 *    B*H*N*d < 2^62; scale finite and > 0 (the kernel folds scale*log2(e)
 *    into one positive factor applied after the row maximum, which needs a
 *    positive scale). Anything else is rejected; there is no fallback path.
 *  - Thread-safe: concurrent calls on different streams are allowed.
 *  - Accumulation is fp32; O is rounded once to `dtype` (round to nearest even).
 */
#ifndef ATTN_GB300_ATTN_H
#define ATTN_GB300_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    ATTN_FP16 = 0,
    ATTN_BF16 = 1
} attn_dtype_t;

/* Mask of attn_fwd_kv (attn_fwd's `causal` != 0 is ATTN_MASK_CAUSAL). */
typedef enum {
    ATTN_MASK_NONE = 0,                /* every key                                     */
    ATTN_MASK_CAUSAL = 1,              /* row i sees keys j <= i (top-left)             */
    ATTN_MASK_CAUSAL_BOTTOM_RIGHT = 2  /* row i sees keys j <= i + Nk - Nq: the query
                                          rows are the last Nq positions (decoding)    */
} attn_mask_t;

/* Diagonal alignment of attn_fwd_window. */
typedef enum {
    ATTN_ALIGN_TOP_LEFT = 0,     /* row i's diagonal is key i                      */
    ATTN_ALIGN_BOTTOM_RIGHT = 1  /* row i's diagonal is key i + n_b - Nq, n_b the
                                    valid keys of its batch element                */
} attn_align_t;

typedef enum {
    ATTN_OK = 0,
    ATTN_ERR_INVALID_ARG = 1,  /* null pointer, size < 1, bad scale or dtype, overlap   */
    ATTN_ERR_UNSUPPORTED = 2,  /* valid but not built: d not in {64,128}, sizes too big */
    ATTN_ERR_MISALIGNED = 3,   /* a pointer is not 16-byte aligned                        */
    ATTN_ERR_CUDA = 4,         /* a CUDA runtime/driver call failed; see
                                  attn_last_cuda_error()                                  */
    ATTN_ERR_TIMEOUT = 5,      /* a device-side wait ran out (attn_fwd_checked only); the
                                  outputs are undefined and the context stays usable      */
    ATTN_ERR_SCRATCH_TOO_SMALL = 6 /* attn_fwd_kv_static: the split of the keys for these
                                  sizes needs more than its static scratch               */
} attn_status_t;

/*
 * attn_fwd -- enqueue the forward pass on `stream`.
 *
 * Computes o = softmax(scale * q k^T [+ causal mask]) v and lse (natural log)
 * for every (b, h) and query row, as defined at the top of this header.
 * causal != 0 selects the top-left mask j <= i. dtype is an attn_dtype_t.
 * Returns ATTN_OK once the kernel is enqueued, or an error status with nothing
 * enqueued. Device-side faults surface at the caller's next synchronisation.
 */
int attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
             int64_t B, int64_t H, int64_t N, int64_t d, int causal, float scale,
             int dtype, void* stream);

/*
 * attn_fwd_checked -- attn_fwd, then synchronise `stream` and read the device
 * status word. Returns ATTN_ERR_TIMEOUT if any device-side wait gave up (the
 * kernel bounds every wait instead of spinning forever), ATTN_ERR_CUDA if the
 * launch or the synchronisation failed, else ATTN_OK. Meant for tests and
 * debugging: it blocks the calling host thread. It clears the device status
 * word before the launch, so concurrent checked calls on different streams
 * may see each other's status.
 */
int attn_fwd_checked(const void* q, const void* k, const void* v, void* o, float* lse,
                     int64_t B, int64_t H, int64_t N, int64_t d, int causal, float scale,
                     int dtype, void* stream);

/*
 * attn_fwd_kv -- forward pass of Nq query rows against Nk keys, enqueued on
 * `stream`: a KV-cache decode step (Nq small, Nk the cache length) or any other
 * pair of lengths.
 *
 * Sources: "Programming an attention kernel in Triton", Kernel 4, runs queries
 * against a longer key/value sequence (a single query against ten keys among its
 * tests); the kernel of the profile-driven FlashAttention-2 page takes N_QUERIES
 * and N_KEYS separately and masks k_pos <= q_pos ("Round 4 / Causal
 * tile-skipping"), which is ATTN_MASK_CAUSAL; "Getting the kernel correct, then
 * benchmarking it honestly" names KV-cache decode as the next extension, whose
 * new query rows are the last positions of the sequence:
 * ATTN_MASK_CAUSAL_BOTTOM_RIGHT.
 *
 *  - q, o: DEVICE [B, H, Nq, d] of `dtype`; k, v: DEVICE [B, H, Nk, d] of
 *    `dtype`; lse: DEVICE [B, H, Nq] fp32. Alignment, overlap and size rules
 *    as above, with Nq and Nk in place of N.
 *  - mask: an attn_mask_t; anything else is ATTN_ERR_INVALID_ARG. A row that
 *    sees no key (bottom-right with Nq > Nk) gets O = 0 and LSE = -inf.
 *  - Nq <= 4: a streaming kernel on the CUDA cores runs instead of the tensor-core
 *    kernel (a decode step reads each K and V byte for at most four rows, so the
 *    call is bound by HBM). Each warp streams K and V tiles of 32 keys with bulk
 *    copies and keeps P and every sum in fp32. Its keys are cut into ranges as a
 *    balance model of the grid's warps favours; with a workspace, the ranges'
 *    fp32 partial outputs go there and a second kernel merges them, and with
 *    none (or too little for two ranges) each head is one range, written
 *    directly.
 *  - workspace: optional DEVICE scratch owned by the caller (16-byte aligned,
 *    not overlapping the other arrays; NULL or 0 bytes allowed). When the
 *    query rows alone give too few CTAs for the GPU (fewer than two per SM),
 *    the keys may be split into ranges (as many as a wave model of the launch
 *    favours, at most eight waves of CTAs) processed by separate CTAs whose fp32 partial outputs and
 *    log-sum-exps go to the workspace and are merged by a second kernel on the
 *    same stream; how many ranges is bounded by workspace_bytes, and with too
 *    little workspace the call runs unsplit (same results up to fp32
 *    rounding order, fewer CTAs). Nothing in it needs to be initialised; it
 *    is read and written only by the kernels of this call, so calls that may
 *    run at the same time need workspaces of their own. The split of the
 *    keys has no counterpart in the pages: it is this library's way of
 *    filling the GPU when Nq is small.
 *  - Returns as attn_fwd.
 */
int attn_fwd_kv(const void* q, const void* k, const void* v, void* o, float* lse,
                int64_t B, int64_t H, int64_t Nq, int64_t Nk, int64_t d, int mask,
                float scale, int dtype, void* workspace, size_t workspace_bytes,
                void* stream);

/* attn_fwd_kv_checked -- attn_fwd_kv, then synchronise and read the device
 * status word, as attn_fwd_checked. */
int attn_fwd_kv_checked(const void* q, const void* k, const void* v, void* o, float* lse,
                        int64_t B, int64_t H, int64_t Nq, int64_t Nk, int64_t d, int mask,
                        float scale, int dtype, void* workspace, size_t workspace_bytes,
                        void* stream);

/* attn_fwd_kv_workspace_bytes -- the workspace size with which attn_fwd_kv uses
 * its full split of the keys for these sizes on the current device (0: it never
 * splits them); for Nq <= 4 the larger of the decode kernel's plan and the
 * tensor-core split's (attn_fwd_window shares this query and runs the latter). The split depends on the GPU's SM count, which this looks up once
 * per device (a GB300's 152 without a device); otherwise host arithmetic. A
 * smaller workspace is never wrong: the call then splits the keys less. 0 for
 * sizes attn_fwd_kv rejects. */
size_t attn_fwd_kv_workspace_bytes(int64_t B, int64_t H, int64_t Nq, int64_t Nk, int64_t d);

/*
 * attn_fwd_window -- attn_fwd_kv with a sliding window and key padding.
 *
 * Source: "如何用 profiler 逐步优化 Triton FlashAttention-2 kernel", "Future
 * articles", names padding masks and sliding windows as the kernels in which a
 * row can be fully masked (so a -inf sentinel must be handled); the page defines
 * neither, and this call takes the plain readings:
 *  - kv_lens: optional DEVICE int32 [B] (4-byte aligned; NULL = all Nk): batch
 *    element b has n_b = kv_lens[b] valid keys, its first n_b (right padding).
 *    Values are clamped to [0, Nk] on the device.
 *  - align: an attn_align_t giving the diagonal of row i (i, or i + n_b - Nq).
 *  - row i sees the valid keys j with diag - window_left <= j <= diag +
 *    window_right; a negative bound (or one beyond Nq + Nk) is unbounded on that
 *    side. window_right = 0 is the causal mask; (-1, -1) is no window.
 *  - A row that sees no key gets O = 0 and LSE = -inf.
 *  - Everything else (layouts, workspace and its split of the keys, errors) as
 *    attn_fwd_kv. Nq + Nk must not exceed 2^30 (ATTN_ERR_UNSUPPORTED).
 */
int attn_fwd_window(const void* q, const void* k, const void* v, void* o, float* lse,
                    int64_t B, int64_t H, int64_t Nq, int64_t Nk, int64_t d,
                    int64_t window_left, int64_t window_right, const int32_t* kv_lens,
                    int align, float scale, int dtype, void* workspace,
                    size_t workspace_bytes, void* stream);

/* attn_fwd_window_checked -- attn_fwd_window, then synchronise and read the device
 * status word, as attn_fwd_checked. */
int attn_fwd_window_checked(const void* q, const void* k, const void* v, void* o,
                            float* lse, int64_t B, int64_t H, int64_t Nq, int64_t Nk,
                            int64_t d, int64_t window_left, int64_t window_right,
                            const int32_t* kv_lens, int align, float scale, int dtype,
                            void* workspace, size_t workspace_bytes, void* stream);

/*
 * attn_bwd -- enqueue the backward pass on `stream`: the gradients of sum(dO * O)
 * with respect to q, k and v for the forward defined at the top of this header
 * (same mask and scale), from the forward's o and lse.
 *
 *   P_ij = exp(scale q_i.k_j - LSE_i) over the visible keys, D_i = dO_i . O_i,
 *   dV_j = sum_i P_ij dO_i,   dS_ij = P_ij (dO_i . v_j - D_i),
 *   dQ_i = scale sum_j dS_ij k_j,   dK_j = scale sum_i dS_ij q_i.
 *
 * Sources: "如何用 profiler 逐步优化 Triton FlashAttention-2 kernel", "Future
 * articles", names the FA2 backward as the next kernel, one that consumes the L
 * the forward saves ("Round 4 / exp2": natural-log units) and accumulates in two
 * directions; the forward there is a torch.autograd.Function, so the backward is
 * the chain rule through the definition.
 *
 *  - q, k, v, o, dout: DEVICE [B, H, N, d] of `dtype`, read only; lse: DEVICE
 *    [B, H, N] fp32 from attn_fwd with the same q, k, v, causal and scale.
 *  - dq, dk, dv: DEVICE [B, H, N, d] of `dtype`, written (rounded once from fp32).
 *  - workspace: DEVICE scratch owned by the caller, at least
 *    attn_bwd_workspace_bytes(B, H, N, d) bytes (fp32 D and LSE vectors, the dQ
 *    accumulator and the counter of the d = 64 kernel's work items); nothing in it
 *    needs to be initialised. Calls that may run at the same time need workspaces of
 *    their own.
 *  - All ten pointers 16-byte aligned; the outputs and the workspace must not
 *    overlap each other or any input. Sizes and scale as for attn_fwd.
 *  - dQ is summed over key tiles with fp32 atomic additions, so its last bits
 *    may differ from run to run; dK and dV are deterministic (at d = 64 the key
 *    tiles are handed to the CTAs in the order they ask, which changes only the
 *    order of those dQ additions).
 *  - Returns ATTN_OK once the three kernels are enqueued, or an error status
 *    with nothing enqueued (ATTN_ERR_INVALID_ARG also for a short workspace).
 */
int attn_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
             const void* dout, void* dq, void* dk, void* dv, int64_t B, int64_t H,
             int64_t N, int64_t d, int causal, float scale, int dtype, void* workspace,
             size_t workspace_bytes, void* stream);

/* attn_bwd_checked -- attn_bwd, then synchronise and read the device status
 * word, as attn_fwd_checked. */
int attn_bwd_checked(const void* q, const void* k, const void* v, const void* o,
                     const float* lse, const void* dout, void* dq, void* dk, void* dv,
                     int64_t B, int64_t H, int64_t N, int64_t d, int causal, float scale,
                     int dtype, void* workspace, size_t workspace_bytes, void* stream);

/*
 * attn_bwd_window -- the backward of attn_fwd_window: Nq query rows against Nk keys
 * with key padding, a sliding window and the diagonal alignment, each row over
 * exactly the keys the forward lets it see (same arguments and readings as
 * attn_fwd_window). q, o, dout, dq: [B, H, Nq, d]; k, v, dk, dv: [B, H, Nk, d];
 * lse [B, H, Nq] from attn_fwd_window with the same arguments.
 *  - Rows that see no key get dQ = 0; padded keys get dK = dV = 0.
 *  - The workspace is attn_bwd_workspace_bytes(B, H, Nq, d) bytes.
 *  - Everything else as attn_bwd.
 */
int attn_bwd_window(const void* q, const void* k, const void* v, const void* o,
                    const float* lse, const void* dout, void* dq, void* dk, void* dv,
                    int64_t B, int64_t H, int64_t Nq, int64_t Nk, int64_t d,
                    int64_t window_left, int64_t window_right, const int32_t* kv_lens,
                    int align, float scale, int dtype, void* workspace,
                    size_t workspace_bytes, void* stream);

/* attn_bwd_window_checked -- attn_bwd_window, then synchronise and read the device
 * status word, as attn_fwd_checked. */
int attn_bwd_window_checked(const void* q, const void* k, const void* v, const void* o,
                            const float* lse, const void* dout, void* dq, void* dk,
                            void* dv, int64_t B, int64_t H, int64_t Nq, int64_t Nk,
                            int64_t d, int64_t window_left, int64_t window_right,
                            const int32_t* kv_lens, int align, float scale, int dtype,
                            void* workspace, size_t workspace_bytes, void* stream);

/* attn_bwd_workspace_bytes -- workspace attn_bwd needs for these sizes (N = the query
 * rows; for attn_bwd_window pass Nq): 8 bytes per row padded to 128 rows, plus 4*d
 * bytes per row, plus 16 bytes (a work-item counter) (0 for sizes attn_bwd rejects).
 * Pure host arithmetic, no CUDA call. */
size_t attn_bwd_workspace_bytes(int64_t B, int64_t H, int64_t N, int64_t d);

/*
 * attn_fwd_kv_static -- attn_fwd_kv that allocates nothing and takes no
 * workspace: the split partials go to a static device array of 16 MiB
 * (16777216 bytes) inside this library. The
 * pages have no counterpart; it exists for callers that must not allocate or
 * pass device scratch on the call path.
 *  - Arguments, masks and results as attn_fwd_kv. Sizes whose full tensor-core
 *    split of the keys needs more than the scratch are rejected with
 *    ATTN_ERR_SCRATCH_TOO_SMALL before anything is enqueued. On GPUs of up to
 *    200 SMs (a GB300 has 152) every size with Nq <= 16 fits. With Nq <= 4 the
 *    decode kernel runs with as many key ranges as the scratch holds.
 *  - Nothing in the scratch needs to start at zero: each call writes every
 *    partial it reads before reading it.
 *  - No device or host memory is allocated (no cudaMalloc/cudaFree, no
 *    allocating library). The first call on a device looks up the scratch
 *    address with cudaGetSymbolAddress (that device current) and caches it;
 *    make that first call before any stream capture.
 *  - There is one scratch per device: calls that may overlap in time (other
 *    streams, other host threads) race on it and give wrong results.
 *    Serialise them, or use attn_fwd_kv with a workspace of their own.
 */
int attn_fwd_kv_static(const void* q, const void* k, const void* v, void* o, float* lse,
                       int64_t B, int64_t H, int64_t Nq, int64_t Nk, int64_t d, int mask,
                       float scale, int dtype, void* stream);

/*
 * attn_fwd_host -- attn_fwd for inputs and outputs in HOST memory: copies q, k, v
 * to the device, runs the forward and copies o and lse back, all enqueued on
 * `stream`. The pages have no counterpart (their kernels take device tensors);
 * it is the call for a caller whose arrays live on the host, and it computes
 * exactly what attn_fwd computes (bit for bit: the same kernel on the same
 * heads).
 *  - q, k, v, o: [B, H, N, d] of `dtype`, lse: [B, H, N] fp32, contiguous, in
 *    host memory (page-locked memory lets the copies overlap the kernels;
 *    pageable memory works but the copies then block the calling thread). Any
 *    alignment. o and lse must not overlap each other, the inputs or the
 *    workspace.
 *  - q, k and v may all three be NULL: the inputs are then the ones already in
 *    the workspace, staged there by an earlier attn_fwd_host call with the same
 *    B, H, N, d and dtype (e.g. to run the other mask on the same inputs without
 *    copying them again). That call must be ordered before this one, for
 *    instance by enqueuing both on `stream`. Only o and lse are copied then.
 *  - workspace: DEVICE memory owned by the caller, 256-byte aligned, of at
 *    least attn_fwd_host_workspace_bytes(B, H, N, d) bytes; the call runs on
 *    the device that owns it. It stages the five arrays on the device: nothing
 *    in it needs initialising, and calls that may run at the same time need
 *    workspaces of their own. After the call it holds q, k, v, o and lse at
 *    the offsets of the layout below.
 *  - Pipelining: the B*H heads are processed in attn_fwd_host_plan() chunks
 *    of consecutive heads. The copy of chunk c+1's inputs overlaps chunk c's
 *    kernel and the copy of chunk c's outputs overlaps the kernels after it.
 *    The copies run on two streams the library creates on the first call on a
 *    device (with 35 events) and keeps; the kernels run on `stream`. Every
 *    copy follows the work enqueued on `stream` before the call, and work
 *    enqueued on `stream` after it follows every copy. o and lse are complete
 *    once `stream` has reached that point (e.g. after cudaStreamSynchronize).
 *  - Workspace layout (bytes, each part rounded up to 256): q at 0, k at X,
 *    v at 2X, o at 3X, lse at 4X, with X = B*H*N*d*2; total 4X + B*H*N*4.
 *  - Errors: as attn_fwd (with one or two of q, k, v NULL an invalid argument),
 *    plus ATTN_ERR_INVALID_ARG for a null or too small workspace and ATTN_ERR_MISALIGNED for a workspace not 256-byte aligned,
 *    all before anything is enqueued. Host threads enqueuing on one device
 *    are serialised by a lock of the library.
 */
int attn_fwd_host(const void* q, const void* k, const void* v, void* o, float* lse,
                  int64_t B, int64_t H, int64_t N, int64_t d, int causal, float scale,
                  int dtype, void* workspace, size_t workspace_bytes, void* stream);

/* attn_fwd_host_checked -- attn_fwd_host, then synchronise `stream` and read the
 * device status word, as attn_fwd_checked. */
int attn_fwd_host_checked(const void* q, const void* k, const void* v, void* o, float* lse,
                          int64_t B, int64_t H, int64_t N, int64_t d, int causal, float scale,
                          int dtype, void* workspace, size_t workspace_bytes, void* stream);

/* attn_fwd_host_workspace_bytes -- workspace attn_fwd_host needs (layout above);
 * 0 for sizes it rejects. Pure host arithmetic, no CUDA call. */
size_t attn_fwd_host_workspace_bytes(int64_t B, int64_t H, int64_t N, int64_t d);

/* attn_fwd_host_plan -- the chunks of attn_fwd_host on the current device: returns
 * their number (0 for sizes it rejects) and stores the heads per chunk (the last
 * chunk holds the rest) in *heads_per_chunk when it is not NULL. A chunk is about
 * two full waves of 256-row work items of the GPU (ceil(2 * SMs / ceil(N/256))
 * heads, i.e. ceil(304 / ceil(N/256)) on a 152-SM GB300), with at most 16 chunks.
 * The SM count is looked up once per device (152 without a device). */
int64_t attn_fwd_host_plan(int64_t B, int64_t H, int64_t N, int64_t d, int64_t* heads_per_chunk);

/* attn_strerror -- static, human-readable text for an attn_status_t. Never NULL. */
const char* attn_strerror(int status);

/* attn_last_cuda_error -- the cudaError_t behind the last ATTN_ERR_CUDA returned
 * on the calling host thread (0 if none). */
int attn_last_cuda_error(void);

/*
 * attn_device_error_info -- copy the device status record into info[0..3]:
 * {status bits, linear block index, role*1000 + barrier id, loop iteration}
 * of the first wait that gave up since the record was last cleared (all zero if
 * none). Synchronous (reads device memory of the current device). Returns
 * ATTN_OK or ATTN_ERR_CUDA; ATTN_ERR_INVALID_ARG if info is NULL. Diagnostics
 * only; the pages have no counterpart.
 */
int attn_device_error_info(int32_t info[4]);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_GB300_ATTN_H */
