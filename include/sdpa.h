/*
 * sdpa.h -- C ABI of the GB300 (sm_103a) fused scaled-dot-product attention
 * library (libsdpa_gb300.so).
 *
 * The operation (forward), as "Inside NVIDIA's cuDNN Graph API" (tradepoint.io),
 * section 5 "SDPA (Flash Attention) with causal masking" builds it:
 *
 *     O = softmax(attn_scale * Q K^T + mask) V
 *
 * with the causal mask aligned top-left (diagonal_alignment TOP_LEFT,
 * right_bound 0): query row i attends to key j iff j <= i.  The same page
 * counts its cost as 4*b*h*s*s*d*0.5 FLOPs when causal.  Besides O the
 * forward writes the per-row statistic
 *
 *     LSE_i = ln sum_{j allowed} exp(attn_scale * Q_i . K_j)
 *
 * (natural log of the scaled scores), fp32, in aten's logsumexp layout for
 * dense tensors and token-major for packed tensors (cudnn-frontend PR #554,
 * dense-backward and THD-statistics notes).  A row with no allowed key (only
 * possible when its sequence has zero keys) gets O = 0 and LSE = -inf
 * (cudnn-frontend PR #554, FP8 d512 notes on fully-masked rows).
 *
 * The backward recomputes P from the stored LSE and returns dQ, dK, dV in
 * the layouts of Q, K, V (cudnn-frontend PR #554, "dense backward" notes).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - All tensor pointers are DEVICE pointers owned by the caller.  The
 *    library allocates no device memory and never synchronises the host; it
 *    enqueues work on `stream` (0 = legacy default stream) and returns.
 *  - Element types: `dtype` is SDPA_BF16 or SDPA_FP16 for q, k, v, o, dout,
 *    dq, dk, dv.  lse is always fp32.  Arithmetic is fp32 throughout
 *    (tensor-core fp32 accumulation, fp32 softmax statistics).
 *  - Head dimension d must be 64 or 128.
 *  - Every tensor pointer must be 16-byte aligned and tensors are dense
 *    (contiguous innermost dimension, no gaps), as the pages' descriptor
 *    contract requires (cudnn-frontend PR #554, "normalize dense operands").
 *  - Arguments are validated before anything is enqueued; on an error the
 *    function returns a non-zero sdpa_status, writes nothing, and
 *    sdpa_last_error() describes the problem.
 *  - Empty problems (any of b, h, s_q, total_q equal to 0) return SDPA_OK
 *    without launching.  s_kv == 0 (or a sequence with no keys) is valid and
 *    yields dead rows.
 *  - Host scalars (total_q, total_kv, max_seqlen_*) describe the packed
 *    problem so that nothing is read back from the device (cudnn-frontend
 *    PR #554, "no D2H sync in varlen backward" and "max_s_kv grid hint").
 *    The device-side cu_seqlens must be non-decreasing, start at 0 and end
 *    at total_q / total_kv; this is the caller's contract and is not checked.
 *  - Calls are thread-safe; sdpa_last_error() is per host thread.
 */
#ifndef SDPA_GB300_H
#define SDPA_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Opaque CUDA stream handle (a cudaStream_t); NULL is the legacy stream. */
typedef void *sdpa_stream_t;

typedef enum {
    SDPA_OK = 0,
    SDPA_ERR_INVALID_ARG = 1, /* negative size, NULL pointer, aliasing, bad flag */
    SDPA_ERR_UNSUPPORTED = 2, /* d not in {64,128}, unknown dtype, wrong GPU */
    SDPA_ERR_MISALIGNED = 3,  /* a tensor pointer is not 16-byte aligned */
    SDPA_ERR_WORKSPACE = 4,   /* workspace NULL or smaller than required */
    SDPA_ERR_CUDA = 5,        /* a CUDA runtime/driver call failed */
    SDPA_ERR_TIMEOUT = 6      /* a kernel gave up on a bounded wait */
} sdpa_status;

typedef enum {
    SDPA_BF16 = 0,
    SDPA_FP16 = 1,
    SDPA_FP8_E4M3 = 2 /* sdpa_fwd_fp8 / sdpa_varlen_fwd_fp8 only: OCP E4M3 ("FN") */
} sdpa_dtype;

/*
 * Masks of the extended entry points (cudnn-frontend PR #554, the `sdpa`
 * op's is_causal, causal_bottom_right and window_left arguments).  Within one
 * sequence of Lq queries and Lkv keys, query i sees key j iff lo_i <= j <
 * hi_i, with delta = Lkv - Lq for SDPA_MASK_CAUSAL_BOTTOM_RIGHT and 0
 * otherwise:
 *   hi_i = Lkv                          for SDPA_MASK_NONE,
 *   hi_i = min(Lkv, i + delta + 1)      for the two causal masks;
 *   lo_i = max(0, i + delta - window_left) when window_left >= 0 (that many
 *          keys left of the diagonal stay visible), 0 when window_left = -1.
 * A query row that sees no key gets O = 0 and LSE = -inf and adds nothing to
 * any gradient (bottom-right alignment with Lq > Lkv leaves the first
 * Lq - Lkv rows so).
 */
typedef enum {
    SDPA_MASK_NONE = 0,
    SDPA_MASK_CAUSAL = 1,              /* top-left: j <= i */
    SDPA_MASK_CAUSAL_BOTTOM_RIGHT = 2  /* j <= i + Lkv - Lq */
} sdpa_mask;

/*
 * Dense forward (BHSD).
 *   q, o : [b, h, s_q, d]   (dtype)      k, v : [b, h, s_kv, d] (dtype)
 *   lse  : [b, h, s_q] fp32, or NULL to skip writing it.
 *   attn_scale: multiplier of Q K^T (the pages' default is 1/sqrt(d); the
 *   ABI takes it explicitly).  causal: 0 or 1 (top-left alignment).
 * o and lse must not overlap q, k or v.
 */
int sdpa_fwd(const void *q, const void *k, const void *v, void *o, float *lse,
             int b, int h, int s_q, int s_kv, int d, float attn_scale,
             int causal, int dtype, sdpa_stream_t stream);

/*
 * Packed (THD / varlen) forward.
 *   q, o : [total_q, h, d]   k, v : [total_kv, h, d]   lse : [total_q, h] fp32
 *   (token-major) or NULL.
 *   cu_seqlens_q, cu_seqlens_kv : int32 device arrays [num_seqs + 1], prefix
 *   sums of the per-sequence lengths (cudnn-frontend PR #554, THD notes).
 *   Sequence n owns query tokens [cu_q[n], cu_q[n+1]) and key tokens
 *   [cu_kv[n], cu_kv[n+1]); the causal mask is top-left within it.
 *   max_seqlen_q / max_seqlen_kv: upper bounds of the per-sequence lengths
 *   (host values; used to size the launch).
 * Rows of q/k/v past total_q/total_kv are never read, so a buffer allocated
 * with spare capacity may hold anything (even NaN) there (cudnn-frontend PR
 * #554, "clamp the f16 THD K/V descriptors to the packed total").
 */
int sdpa_varlen_fwd(const void *q, const void *k, const void *v, void *o,
                    float *lse, const int32_t *cu_seqlens_q,
                    const int32_t *cu_seqlens_kv, int num_seqs, int total_q,
                    int total_kv, int max_seqlen_q, int max_seqlen_kv, int h,
                    int d, float attn_scale, int causal, int dtype,
                    sdpa_stream_t stream);

/*
 * Extended dense forward: grouped key/value heads and the masks above.
 *   q, o : [b, h, s_q, d]   k, v : [b, h_kv, s_kv, d]   lse : [b, h, s_q] or NULL
 *   h must be a multiple of h_kv (h_kv = h: one key/value head per query
 *   head; h_kv = 1: multi-query); query head hq reads key/value head
 *   hq / (h / h_kv) (cudnn-frontend PR #554 GQA cases).
 *   mask: an sdpa_mask value.  window_left: -1 (none) or >= 0.
 * sdpa_fwd(..., causal, ...) is this call with h_kv = h, mask = causal ?
 * SDPA_MASK_CAUSAL : SDPA_MASK_NONE and window_left = -1.
 */
int sdpa_fwd_ex(const void *q, const void *k, const void *v, void *o, float *lse,
                int b, int h, int h_kv, int s_q, int s_kv, int d,
                float attn_scale, int mask, int window_left, int dtype,
                sdpa_stream_t stream);

/*
 * Extended packed forward: as sdpa_varlen_fwd with k, v : [total_kv, h_kv, d]
 * and the mask / window of sdpa_fwd_ex, applied per sequence with that
 * sequence's own lengths (the bottom-right offset is Lkv(n) - Lq(n)).
 */
int sdpa_varlen_fwd_ex(const void *q, const void *k, const void *v, void *o,
                       float *lse, const int32_t *cu_seqlens_q,
                       const int32_t *cu_seqlens_kv, int num_seqs, int total_q,
                       int total_kv, int max_seqlen_q, int max_seqlen_kv, int h,
                       int h_kv, int d, float attn_scale, int mask,
                       int window_left, int dtype, sdpa_stream_t stream);

/*
 * FP8 forward (cudnn-frontend PR #554, per-tensor FP8 forward): q, k, v hold
 * E4M3 codes (one byte per element, layouts and masks as sdpa_fwd_ex, d =
 * 128) standing for the real values code * descale_x.
 *   descale_q, descale_k, descale_v : fp32 scalars in DEVICE memory, read by
 *     the kernel (no host read-back); descale_q * descale_k joins the
 *     softmax multiplier, descale_v the output factor.
 *   out_dtype : SDPA_BF16, SDPA_FP16 or SDPA_FP8_E4M3 for o; an E4M3 output
 *     holds round-to-nearest, saturated codes of O * (*scale_o) (scale_o, a
 *     device fp32 scalar, is required then and ignored otherwise).
 *   amax_o : NULL, or a device fp32 scalar that receives max |O| over the
 *     whole output, taken on the real-valued O before any output scaling or
 *     rounding (the call sets it to 0 first, on `stream`).
 *   lse : as sdpa_fwd_ex, of the real-valued scores.
 * P enters the P V product as E4M3 (relative rounding error <= 2^-4 per
 * element); the row sums and the LSE use the unrounded fp32 P.
 */
int sdpa_fwd_fp8(const void *q, const void *k, const void *v, void *o,
                 float *lse, const float *descale_q, const float *descale_k,
                 const float *descale_v, const float *scale_o, float *amax_o,
                 int b, int h, int h_kv, int s_q, int s_kv, int d,
                 float attn_scale, int mask, int window_left, int out_dtype,
                 sdpa_stream_t stream);

/* Packed FP8 forward: sdpa_varlen_fwd_ex's layout and masks with the FP8
 * arguments of sdpa_fwd_fp8. */
int sdpa_varlen_fwd_fp8(const void *q, const void *k, const void *v, void *o,
                        float *lse, const float *descale_q,
                        const float *descale_k, const float *descale_v,
                        const float *scale_o, float *amax_o,
                        const int32_t *cu_seqlens_q,
                        const int32_t *cu_seqlens_kv, int num_seqs,
                        int total_q, int total_kv, int max_seqlen_q,
                        int max_seqlen_kv, int h, int h_kv, int d,
                        float attn_scale, int mask, int window_left,
                        int out_dtype, sdpa_stream_t stream);

/*
 * Workspace bytes sdpa_bwd needs: an fp32 dQ accumulator [b,h,s_q,d] and
 * 16 bytes of fp32 row terms per query row [b,h,s_q]: -LSE/scale and
 * -D_i, D_i = sum_k dO_ik O_ik, each as a pair of tf32-exact parts
 * (cudnn-frontend PR #554: the backward chain's "do_dot" step and its fp32
 * dQ accumulator), each part rounded up to 256 bytes.  Returns 0 for an
 * empty problem, (size_t)-1 for invalid sizes.
 */
size_t sdpa_bwd_workspace_size(int b, int h, int s_q, int d);

/*
 * Dense backward (BHSD).  Same shapes and flags as the sdpa_fwd call that
 * produced o and lse (lse must not be NULL).  dout : [b,h,s_q,d].
 * Writes dq [b,h,s_q,d], dk, dv [b,h,s_kv,d] in dtype.  `workspace` is a
 * device buffer of at least sdpa_bwd_workspace_size(b,h,s_q,d) bytes, owned
 * by the caller; its contents on entry do not matter and it must not be used
 * by another call until this one completes on `stream`.
 * dQ is accumulated with fp32 atomics, so its low bits may differ from run
 * to run; dK and dV are deterministic.
 */
int sdpa_bwd(const void *q, const void *k, const void *v, const void *o,
             const void *dout, const float *lse, void *dq, void *dk, void *dv,
             int b, int h, int s_q, int s_kv, int d, float attn_scale,
             int causal, int dtype, void *workspace, size_t workspace_bytes,
             sdpa_stream_t stream);

/* Workspace bytes sdpa_varlen_bwd needs (same content as the dense one, sized
 * by the packed token count). */
size_t sdpa_varlen_bwd_workspace_size(int total_q, int h, int d);

/*
 * Packed (THD) backward.  Arguments as sdpa_varlen_fwd, plus o, dout
 * [total_q,h,d], lse [total_q,h] fp32 from that forward, outputs dq
 * [total_q,h,d], dk, dv [total_kv,h,d] and the workspace.
 * It is the backward of the packed path of cudnn-frontend PR #554 ("THD /
 * varlen" notes): the gradients keep the packed layouts of q, k and v, the
 * token-major statistics of the forward are read as they are (no repadding
 * into a dense layout), and nothing is read back to the host -- the PR's fix
 * "drop the 2*B D2H syncs from the varlen backward" is why the totals and
 * maximum lengths are host arguments here too.  Sequences are independent:
 * dK, dV of sequence n take contributions of its own queries only.
 */
int sdpa_varlen_bwd(const void *q, const void *k, const void *v, const void *o,
                    const void *dout, const float *lse, void *dq, void *dk,
                    void *dv, const int32_t *cu_seqlens_q,
                    const int32_t *cu_seqlens_kv, int num_seqs, int total_q,
                    int total_kv, int max_seqlen_q, int max_seqlen_kv, int h,
                    int d, float attn_scale, int causal, int dtype,
                    void *workspace, size_t workspace_bytes,
                    sdpa_stream_t stream);

/* Workspace bytes of the extended backward calls; the query-side sizes
 * decide it, h_kv does not.  deterministic = 0: the same content as
 * sdpa_bwd's (fp32 dQ accumulator and row terms); 1: the row terms alone,
 * 16 bytes per query row.  (size_t)-1 for invalid arguments. */
size_t sdpa_bwd_ex_workspace_size(int b, int h, int s_q, int d, int deterministic);
size_t sdpa_varlen_bwd_ex_workspace_size(int total_q, int h, int d, int deterministic);

/*
 * Extended dense backward: the gradients of sdpa_fwd_ex with the same
 * arguments.  dq : [b, h, s_q, d]; dk, dv : [b, h_kv, s_kv, d], each the sum
 * over the h / h_kv query heads that share the key/value head
 * (cudnn-frontend PR #554: "GQA reduces" in the backward chain).
 * deterministic: 0 accumulates dQ with fp32 reductions whose order may vary
 * between runs (dK and dV are reproducible either way); 1 gives bitwise
 * reproducible gradients: dQ is then computed by a separate query-stationary
 * pass that recomputes S and dP per key tile and writes dQ once (cudnn-
 * frontend PR #554: a separate dQ pass instead of atomics), at about 1.4x
 * the tensor-core work of the default.
 */
int sdpa_bwd_ex(const void *q, const void *k, const void *v, const void *o,
                const void *dout, const float *lse, void *dq, void *dk,
                void *dv, int b, int h, int h_kv, int s_q, int s_kv, int d,
                float attn_scale, int mask, int window_left, int deterministic,
                int dtype, void *workspace, size_t workspace_bytes,
                sdpa_stream_t stream);

/* Extended packed backward: sdpa_varlen_bwd with the arguments of
 * sdpa_varlen_fwd_ex and sdpa_bwd_ex. */
int sdpa_varlen_bwd_ex(const void *q, const void *k, const void *v,
                       const void *o, const void *dout, const float *lse,
                       void *dq, void *dk, void *dv,
                       const int32_t *cu_seqlens_q,
                       const int32_t *cu_seqlens_kv, int num_seqs,
                       int total_q, int total_kv, int max_seqlen_q,
                       int max_seqlen_kv, int h, int h_kv, int d,
                       float attn_scale, int mask, int window_left,
                       int deterministic, int dtype, void *workspace,
                       size_t workspace_bytes, sdpa_stream_t stream);

/*
 * Dense backward that allocates nothing and takes no workspace (the pages
 * have no counterpart of this entry point).
 *
 * For callers that cannot allocate device memory themselves: plug-in or
 * callback code running inside another runtime that owns every device
 * allocation and hands out no workspace, or a latency-critical loop where a
 * cudaMalloc, which may synchronise the device, is not allowed.  Arguments
 * and results are those of sdpa_bwd without workspace/workspace_bytes; the
 * caller still passes every input and output buffer.
 *
 * The scratch that sdpa_bwd keeps in its workspace comes instead from a
 * 32 MiB array inside the library's device image, which every GPU that
 * loads the library holds until the process exits.  Problems whose
 * sdpa_bwd_workspace_size exceeds 32 MiB (about b*h*s_q*(d+4)*4 bytes: up
 * to 63,550 rows of b*h*s_q at d = 128) are rejected with
 * SDPA_ERR_WORKSPACE before anything is launched.
 *  - The first call on each device looks up the array's device address
 *    (cudaGetSymbolAddress, with that device current) and keeps it; make
 *    that first call before any stream capture.  The kept address belongs
 *    to the device's context, so after a cudaDeviceReset of a device (which
 *    ends that context) do not call this entry point on it again in the
 *    same process.
 *  - All calls share the one array, so calls whose work can overlap on the
 *    GPU (other streams, other host threads) race on it and give wrong
 *    gradients; serialise them.  Each call rewrites the part of the array it
 *    uses before reading it, so leftovers of an earlier call do no harm.
 *  - Calls no cudaMalloc, cudaFree or allocating library routine.
 */
int sdpa_bwd_noalloc(const void *q, const void *k, const void *v,
                     const void *o, const void *dout, const float *lse,
                     void *dq, void *dk, void *dv, int b, int h, int s_q,
                     int s_kv, int d, float attn_scale, int causal, int dtype,
                     sdpa_stream_t stream);

/*
 * Message describing the last non-OK status returned on this host thread
 * ("" if none).  The pointer stays valid until the next call on the thread.
 * TransformerEngine PR #2964 moves its C API from a bare "no backend" code
 * to a status plus the real error text (its probe functions return an empty
 * string or the message, and the backend query returns the pair); every
 * entry point here follows that convention: a non-zero sdpa_status, and this
 * call for the text naming the argument or CUDA call that failed.
 */
const char *sdpa_last_error(void);

/*
 * Reads and clears the library's device error word on the current device:
 * kernels that give up on a bounded wait (about two seconds) record the
 * failure there instead of hanging.  Synchronises `stream` first.  Returns
 * SDPA_OK, SDPA_ERR_TIMEOUT (message says which kernel and which wait) or
 * SDPA_ERR_CUDA.  It reports device-side failures in the same status-plus-
 * message form as sdpa_last_error (TransformerEngine PR #2964's C-API error
 * message); it is the one call that synchronises, so the launching calls
 * keep cudnn-frontend PR #554's "no host sync" rule and a caller checks
 * when it chooses (the debug-build device check of the pages' descriptor
 * contract).
 */
int sdpa_check_device_error(sdpa_stream_t stream);

/*
 * Failure-detection self-test (no counterpart on the pages).  Enqueues on
 * `stream` one small kernel whose bounded wait -- the same code every kernel
 * waits with, here with a limit of `limit_us` microseconds (1 .. 2,000,000)
 * instead of two seconds -- polls a barrier phase that nothing completes.
 * The wait expires, records its kernel ("selftest") and site in the error
 * word, and the kernel exits: the next sdpa_check_device_error returns
 * SDPA_ERR_TIMEOUT and clears the word.  Nothing faults or hangs.
 */
int sdpa_selftest_wait_timeout(int limit_us, sdpa_stream_t stream);

/*
 * Measurement hook (no counterpart on the pages).  While both events are
 * non-NULL, every later call on this host thread records `start_event` on
 * its stream immediately before launching its main kernel (the forward
 * kernel, or the backward's main kernel, followed in deterministic mode by
 * its dQ pass) and `stop_event` immediately after,
 * so a caller can time that kernel alone with cudaEventElapsedTime.  The
 * events are cudaEvent_t handles owned by the caller; pass NULL, NULL to
 * stop.  Recording adds no synchronisation.
 */
void sdpa_set_kernel_timer(void *start_event, void *stop_event);

/*
 * Forward kernel choice for later calls on this host thread (a tuning and
 * testing hook; no counterpart on the pages).  0 (default): automatic -- the
 * two-tile kernel (256 query rows per work unit, two softmax warpgroups
 * ping-ponging on the tensor core) for dense problems whose query and key
 * lengths reach 1024, for packed lists without a left window of up to 95
 * sequences (d = 128, 16-bit inputs) or 1023 (d = 64 or FP8 inputs), and for
 * longer packed lists whose mean sequence lengths total_q / num_seqs and
 * total_kv / num_seqs reach 2048; the one-tile kernel (128 rows per unit)
 * otherwise.  FP8 inputs with a left window, and 16-bit inputs with a left
 * window at d = 64, always take the one-tile kernel.  1: always one-tile.
 * 2: the two-tile kernel wherever it applies.  Both compute the same result to
 * rounding.
 * Returns SDPA_ERR_INVALID_ARG for other values.
 */
int sdpa_set_forward_variant(int variant);

/*
 * Backward main-kernel choice for later calls on this host thread (a tuning
 * and testing hook; no counterpart on the pages).  0 (default): automatic --
 * the persistent kernel (one CTA per SM, each taking (key/value slice, key
 * tile) units from a counter) where units are short: dense problems whose
 * units average at most 8 (query head, query tile) pairs, and packed lists of
 * up to 128 sequences whose estimated mean (from total_kv / num_seqs, the
 * mask and the window) is at most 3; one CTA per unit otherwise.  1: always
 * one CTA per unit.  2: the persistent kernel wherever it applies (not for
 * packed lists of more than 128 sequences).  Both give the same dK and dV bit
 * for bit, and dQ to rounding (its fp32 additions may come in another order).
 * Returns SDPA_ERR_INVALID_ARG for other values.
 */
int sdpa_set_backward_variant(int variant);

/* Main kernel that this host thread's last backward call launched (or would
 * have launched, had it had a unit of work): 1 one CTA per unit, 2 persistent;
 * 0 before the first call that reached the choice. */
int sdpa_last_backward_variant(void);

/* Testing hook: at most max_ctas CTAs for the persistent backward kernel on
 * this host thread (0, the default: one per SM), so that small problems
 * exercise CTAs that take many units each.  The result is the same.
 * Returns SDPA_ERR_INVALID_ARG for a negative count. */
int sdpa_set_backward_grid_limit(int max_ctas);

/* Library version string, e.g. "sdpa_gb300 0.10 sm_103a"; the
 * minor number changes whenever a kernel changes. */
const char *sdpa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SDPA_GB300_H */
