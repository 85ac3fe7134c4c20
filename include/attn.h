/*
 * attn.h -- C ABI of the GB300 (sm_103a) exact tiled attention library.
 *
 * The library computes exact scaled-dot-product attention over packed ragged
 * batches,
 *
 *     O = softmax(scale * Q K^T + mask) V,
 *
 * tile by tile with the online-softmax recurrence (running max, rescaled
 * denominator and accumulator, final divide: "formal-correctness", section
 * "The FlashAttention Proof"), saves the natural-log logsumexp of the scaled
 * logits per query row, and provides the recompute-based backward (dQ, dK,
 * dV; GQA gradients summed over each shared KV head:
 * "attention-algorithm-error-and-complexity-tests", third and fourth
 * paragraphs).
 *
 * Layout ("THD", row-major, contiguous, no padding between tokens):
 *   q, o, dout, dq : [total_q, n_heads_q,  head_dim]
 *   k, v, dk, dv   : [total_k, n_heads_kv, head_dim]
 *   lse            : [n_heads_q, total_q] fp32
 *   cu_seqlens_q/k : int32 [batch + 1], device memory, cu[0] = 0,
 *                    non-decreasing, cu[batch] = total.  Sequence s owns
 *                    tokens cu[s] .. cu[s+1]-1 and its positions restart at
 *                    0 ("causal-mask-and-ragged-sequence-layouts", first
 *                    paragraph).  A zero-length sequence and batch = 0 are
 *                    legal and do nothing.
 *
 * Mask rules (same page, third and fourth paragraphs), for zero-based
 * in-sequence query position i and key position j of one sequence with Nq
 * queries and Nk keys:
 *   ATTN_MASK_NONE           every key of the sequence;
 *   ATTN_CAUSAL_TOP_LEFT     j <= i;
 *   ATTN_CAUSAL_BOTTOM_RIGHT j <= i + Nk - Nq.
 * window (every call that takes a mask): 0 leaves the rule as it is; W > 0
 * bounds it to the W key positions that end at the causal bound, i.e. it
 * also requires j > i - W (top-left) or j > i + Nk - Nq - W (bottom-right),
 * so every row sees at most W keys and the pair count grows linearly with
 * the sequence length ("attention-algorithm-error-and-complexity-tests",
 * fifth paragraph).  W > 0 needs a causal kind; a negative W, or W > 0 with
 * ATTN_MASK_NONE, is ATTN_ERR_INVALID_ARG.
 * bias_slopes (every call that takes a mask): NULL for none, or a device
 * array of n_heads_q finite fp32 slopes m_h that add the linear positional
 * bias  -m_h * |i + off - j|  to every allowed logit of query head h, where
 * off = Nk - Nq for ATTN_CAUSAL_BOTTOM_RIGHT and 0 otherwise: the distance of
 * key j from the row's causal bound.  It follows the in-sequence positions
 * (so it is the same for a sequence packed anywhere) and the backward
 * rebuilds it from the same positions ("causal-mask-and-ragged-sequence-
 * layouts", sixth paragraph).
 * Pairs from different sequences are never allowed; tile lanes past a
 * sequence's end never enter the max, the denominator or a gradient sum
 * (same page, second paragraph).  A row with no allowed key gets O = 0 and
 * lse = -inf, and contributes nothing to the backward.
 *
 * GQA: n_heads_q must be a multiple of n_heads_kv; query head h reads KV head
 * h / (n_heads_q / n_heads_kv) (contiguous grouping).
 *
 * Ownership: the caller owns and allocates every buffer (device memory);
 * the library allocates nothing on any call path.  Every call is
 * asynchronous on `stream` (a cudaStream_t passed as void*; NULL is the
 * legacy default stream).  max_seqlen_* and total_* come from the host so no
 * call synchronises.  Argument errors are returned before anything is
 * launched.  Errors the device detects (cu_seqlens inconsistent with the
 * sizes passed, a bounded wait that expired) are recorded in a per-device
 * flag that attn_get_device_error() reads.
 */
#ifndef ATTN_GB300_H
#define ATTN_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  ATTN_OK = 0,
  ATTN_ERR_INVALID_ARG = 1,    /* null pointer, negative size, bad enum, ... */
  ATTN_ERR_UNSUPPORTED = 2,    /* head_dim, dtype or feature not built       */
  ATTN_ERR_WORKSPACE = 3,      /* workspace missing or smaller than needed   */
  ATTN_ERR_CUDA = 4,           /* a CUDA runtime call failed                 */
  ATTN_ERR_DEVICE_TIMEOUT = 5, /* a bounded device wait expired              */
  ATTN_ERR_DEVICE_BOUNDS = 6,  /* cu_seqlens disagree with the sizes passed  */
  ATTN_ERR_SCRATCH_LIMIT = 7,  /* needs more than the static scratch holds   */
  ATTN_ERR_DEVICE_RANGE = 8    /* a bf16 backward input is infinite or NaN */
} attn_status;

typedef enum {
  ATTN_MASK_NONE = 0,
  ATTN_CAUSAL_TOP_LEFT = 1,
  ATTN_CAUSAL_BOTTOM_RIGHT = 2
} attn_mask_kind;

typedef enum {
  ATTN_DTYPE_BF16 = 0, /* bf16 inputs/outputs, fp32 accumulation */
  ATTN_DTYPE_FP32 = 1  /* fp32 inputs/outputs, fp32 arithmetic   */
} attn_dtype;

/*
 * Layouts other than contiguous THD ("causal-mask-and-ragged-sequence-
 * layouts", fifth paragraph: noncontiguous layouts where supported).  For
 * each [tokens, heads, head_dim] tensor, {token stride, head stride} in
 * elements: element c of (token t, head h) is at t * s[0] + h * s[1] + c, the
 * head_dim features contiguous.  Contiguous THD is {n_heads * head_dim,
 * head_dim}.  Every stride must be positive and, times the element size, a
 * multiple of 16 bytes (so 8 elements for bf16, 4 for fp32); tensors must be
 * 16-byte aligned; outputs must not overlap each other or any input.  A
 * typical use: q, k and v as views of one fused projection output
 * [T, Hq + 2 Hkv, d] (token stride (Hq + 2 Hkv) d), and dq, dk, dv written
 * into the matching fused gradient buffer.  lse, o_f32 and the workspace
 * keep the layouts given below.
 */
typedef struct {
  int64_t q[2], k[2], v[2], o[2];        /* read by both calls (o by attn_bwd)  */
  int64_t dout[2], dq[2], dk[2], dv[2];  /* attn_bwd only                        */
} attn_strides;

/*
 * Workspace bytes attn_fwd needs for these sizes on the current device (0 when
 * the chosen plan needs none).  The split-KV decode plan keeps one partial
 * output row (fp32) and one partial logsumexp per key split in it.  Returns
 * (size_t)-1 for arguments attn_fwd would reject.
 */
size_t attn_fwd_workspace_size(int batch, int max_seqlen_q, int max_seqlen_k,
                               int total_q, int n_heads_q, int n_heads_kv,
                               int head_dim, int window, attn_dtype dtype);

/*
 * Forward ("formal-correctness", "The FlashAttention Proof": the online
 * softmax recurrence; "causal-mask-and-ragged-sequence-layouts": mask rules).
 *   q, k, v      inputs, layouts above, element type `dtype`.
 *   o            output [total_q, n_heads_q, head_dim], type `dtype`.
 *   lse          output [n_heads_q, total_q] fp32, natural log of the sum of
 *                exp(scale * q.k) over the allowed keys; -inf for empty rows.
 *                May be NULL when not wanted.
 *   o_f32        optional output [total_q, n_heads_q, head_dim] fp32: the
 *                normalised output before its rounding to `dtype`.  Pass it
 *                on to attn_bwd, which then forms D_i = dO_i . O_i from it
 *                instead of recomputing that output.  NULL skips it.
 *   scale        finite softmax scale (usually 1/sqrt(head_dim)).
 *   workspace    device scratch of at least attn_fwd_workspace_size() bytes,
 *                256-byte aligned (may be NULL when that size is 0).
 * head_dim must be 64 or 128.  bf16 q, k, v and o must be 16-byte aligned
 * (tensor-memory-accelerator loads).  Returns ATTN_OK once the kernels are
 * queued.
 */
attn_status attn_fwd(const void *q, const void *k, const void *v, void *o,
                     float *lse, float *o_f32, const int32_t *cu_seqlens_q,
                     const int32_t *cu_seqlens_k, int batch, int max_seqlen_q,
                     int max_seqlen_k, int total_q, int total_k, int n_heads_q,
                     int n_heads_kv, int head_dim, float scale,
                     attn_mask_kind mask, int window, const float *bias_slopes,
                     attn_dtype dtype, void *workspace, size_t workspace_bytes,
                     void *stream);

/*
 * An explicit bias tensor added to the logits ("attention-algorithm-error-
 * and-complexity-tests", third paragraph: bias and mask terms enter the
 * logits before the softmax).  Entry (sequence s, query head h, in-sequence
 * row i, in-sequence key j) is
 *   data[s * seq_stride + h * head_stride + i * row_stride + j]
 * (fp32, element strides, >= 0; a stride of 0 broadcasts, so a
 * [B, Hq, max_seqlen_q, max_seqlen_k] tensor or any of its broadcasts over
 * sequences or heads fits), in the units of the scaled logits: the logit of
 * an allowed pair is scale * q.k + positional bias + entry.  An entry of
 * -inf removes the pair (an explicit mask); a row without any finite logit
 * is an empty row (O = 0, lse = -inf).  +inf and NaN entries are not
 * allowed.  The caller owns the device memory, which must cover every entry
 * of the [batch, n_heads_q, max_seqlen_q, max_seqlen_k] box the strides
 * describe (the tensor-core forward may read entries outside the allowed
 * pairs, and then ignores them) and stay valid until the call's kernels
 * finish.
 */
typedef struct {
  const float *data;
  int64_t seq_stride, head_stride, row_stride;
} attn_bias_tensor;

/*
 * attn_fwd with the layouts of q, k, v and o given by `strides` (NULL: the
 * contiguous layouts) and an optional explicit bias tensor `bias` (NULL:
 * none; both NULL is exactly attn_fwd).  Same results; ATTN_ERR_INVALID_ARG
 * for a stride that breaks the rules above, a negative bias stride or a bias
 * without data.  bf16 calls with a bias tensor, a positive scale and no
 * bias_slopes run on the tensor-core prefill kernel: with head_dim 128, an
 * even GQA group, head_stride 0 and a 16-byte aligned base, row and
 * sequence stride, the entries stream through shared memory by TMA and the
 * softmax adds them; otherwise they are stored into the score buffer before
 * Q K^T accumulates onto them; other calls
 * with a bias tensor (fp32, a non-positive scale, or slopes as well) run on
 * the CUDA-core kernels (one warp per query row and head).
 */
attn_status attn_fwd_ex(const attn_strides *strides, const attn_bias_tensor *bias, const void *q,
                        const void *k, const void *v, void *o, float *lse,
                        float *o_f32, const int32_t *cu_seqlens_q,
                        const int32_t *cu_seqlens_k, int batch,
                        int max_seqlen_q, int max_seqlen_k, int total_q,
                        int total_k, int n_heads_q, int n_heads_kv,
                        int head_dim, float scale, attn_mask_kind mask,
                        int window, const float *bias_slopes, attn_dtype dtype,
                        void *workspace, size_t workspace_bytes, void *stream);

/*
 * Workspace bytes attn_bwd needs: the per-row terms D_i = dO_i . O_i and the
 * base-2 logsumexp ([n_heads_q, total_q] fp32 each) and, for bf16, fp16
 * copies of q, dout, k and v (plus 256 bytes for their largest magnitudes):
 * the tensor-core backward multiplies in fp16 so that the probabilities P
 * and the score gradients dS it feeds to the tensor cores keep 11
 * significant bits (bf16 keeps 8, which is not enough for a key seen by
 * thousands of rows).  Each copy is scaled by a power of two that brings the
 * tensor's largest magnitude into [4, 8), so every element within 2^19 of
 * it is copied exactly, at any overall magnitude of the inputs; the kernels
 * undo the factors exactly.  For bf16 with head_dim 128 it also holds the
 * fused backward's fp32 dQ accumulator ([total_q, n_heads_q, 128]).
 * (size_t)-1 for bad arguments.
 */
size_t attn_bwd_workspace_size(int batch, int max_seqlen_q, int max_seqlen_k,
                               int total_q, int total_k, int n_heads_q,
                               int n_heads_kv, int head_dim, attn_dtype dtype);

/*
 * Backward at upstream gradient dout, recomputing the probabilities from q, k
 * and the saved lse with the same mask rule, window and bias as the forward
 * ("causal-mask-and-ragged-sequence-layouts", sixth paragraph):
 *   dV_j = sum_i P_ij dO_i,  dS_ij = P_ij (dO_i . v_j - dO_i . O_i),
 *   dQ_i = scale sum_j dS_ij k_j,  dK_j = scale sum_i dS_ij q_i,
 * with dK and dV summed over the query heads that share each KV head
 * ("attention-algorithm-error-and-complexity-tests", third paragraph).
 *   o, lse   the forward's outputs for the same inputs.
 *   o_f32    the forward's optional fp32 output, or NULL.  D_i must not
 *            carry the rounding of O (with value rows that share a large
 *            offset it would exceed the gradient tolerance), so for bf16
 *            without o_f32 the backward first recomputes the fp32 output
 *            with the prefill forward kernel, whose epilogue writes D_i
 *            instead of O (one extra forward pass of work; pass o_f32 to
 *            skip it).  fp32 calls form D_i from o itself.
 *   dq       [total_q, n_heads_q, head_dim]; dk, dv [total_k, n_heads_kv,
 *            head_dim]; type `dtype`.  Fully overwritten (rows no query
 *            reaches get zeros).
 * For bf16, an infinity or NaN in q, k, v or dout sets ATTN_ERR_DEVICE_RANGE
 * on the device flag.  dq, dk and dv must be 16-byte aligned.  For bf16 with
 * head_dim 128, dq is summed over key tiles with fp32 reductions (its last
 * bits can vary from call to call) unless attn_set_deterministic(1) selects
 * the two-kernel form; dk and dv are reproducible in both forms.
 */
attn_status attn_bwd(const void *q, const void *k, const void *v,
                     const void *o, const float *lse, const float *o_f32,
                     const void *dout,
                     void *dq, void *dk, void *dv,
                     const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k,
                     int batch, int max_seqlen_q, int max_seqlen_k,
                     int total_q, int total_k, int n_heads_q, int n_heads_kv,
                     int head_dim, float scale, attn_mask_kind mask,
                     int window, const float *bias_slopes, attn_dtype dtype,
                     void *workspace, size_t workspace_bytes, void *stream);

/*
 * attn_bwd with the layouts of q, k, v, o, dout, dq, dk and dv given by
 * `strides` (NULL: contiguous) and the forward's explicit bias tensor `bias`
 * (NULL: none; both NULL is exactly attn_bwd), rebuilt in the recomputed
 * logits.  The workspace size does not depend on either.  With a bias tensor
 * the tensor-core backward runs under the same conditions as the forward's
 * (bf16, positive scale, no bias_slopes); otherwise the CUDA-core backward.
 */
attn_status attn_bwd_ex(const attn_strides *strides, const attn_bias_tensor *bias, const void *q,
                        const void *k, const void *v, const void *o,
                        const float *lse, const float *o_f32, const void *dout,
                        void *dq, void *dk, void *dv,
                        const int32_t *cu_seqlens_q,
                        const int32_t *cu_seqlens_k, int batch,
                        int max_seqlen_q, int max_seqlen_k, int total_q,
                        int total_k, int n_heads_q, int n_heads_kv,
                        int head_dim, float scale, attn_mask_kind mask,
                        int window, const float *bias_slopes, attn_dtype dtype,
                        void *workspace, size_t workspace_bytes, void *stream);

/*
 * Mask probe (diagnostic): writes, for one query head, the packed allowed-pair
 * matrix that the kernels' tile planner and mask predicate produce, as bytes
 * out[total_q * total_k] (1 = allowed).  It runs the same device code the
 * attention kernels use to bound and mask their tiles, so tests can compare
 * it bit for bit with an independent definition.  tile_rows (16, 32, 64 or
 * 128) is the number of query tokens per tile the planner assumes: 128 for
 * one head per tile, 128 / group when the query heads of a KV head share a
 * tile.  `out` is caller-owned device memory; total_q * total_k must be
 * below 2^31.
 */
attn_status attn_mask_probe(const int32_t *cu_seqlens_q,
                            const int32_t *cu_seqlens_k, int batch,
                            int max_seqlen_q, int max_seqlen_k, int total_q,
                            int total_k, attn_mask_kind mask, int window,
                            int tile_rows, uint8_t *out, void *stream);

/*
 * Synchronises `stream`, then reads and clears the current device's error
 * flag.  Returns ATTN_OK, ATTN_ERR_DEVICE_BOUNDS, ATTN_ERR_DEVICE_TIMEOUT, or
 * ATTN_ERR_CUDA when the synchronisation itself failed.
 */
attn_status attn_get_device_error(void *stream);

/*
 * Forward that allocates nothing, not even through the caller: for callers
 * that cannot hand the library a workspace.  Typical ones are plug-ins and
 * embedded runtimes whose host owns a fixed, pre-planned device memory pool
 * and exposes no allocator to them, and latency-critical serving loops where
 * a cudaMalloc (which can synchronise the device, or fail under memory
 * pressure) is not allowed once the loop runs.  The pages have no
 * counterpart: this is a packaging variant of attn_fwd, not a different
 * computation.
 *
 * Same arguments, layouts and results as attn_fwd, minus the workspace.  The
 * split-KV decode plan keeps its per-split partial outputs in one array of
 * ATTN_STATIC_SCRATCH_BYTES (64 MiB) that the library holds in device memory
 * of every GPU it is loaded on, until the process exits.  A problem whose
 * split scratch would exceed that array is rejected with
 * ATTN_ERR_SCRATCH_LIMIT before anything is launched; plans that need no
 * scratch run exactly as in attn_fwd.
 *
 * The array's device address is looked up on the first call on each device
 * (make that first call outside any stream capture).  All calls share the
 * array: calls whose kernels overlap on the GPU (different streams, or
 * different host threads, without ordering between them) race on it and
 * must be serialised by the caller.  Every scratch entry a call reads is
 * written earlier in the same call, so nothing needs clearing between calls.
 */
#define ATTN_STATIC_SCRATCH_BYTES (64u << 20)
attn_status attn_fwd_static_scratch(const void *q, const void *k, const void *v,
                                    void *o, float *lse, float *o_f32,
                                    const int32_t *cu_seqlens_q,
                                    const int32_t *cu_seqlens_k, int batch,
                                    int max_seqlen_q, int max_seqlen_k,
                                    int total_q, int total_k, int n_heads_q,
                                    int n_heads_kv, int head_dim, float scale,
                                    attn_mask_kind mask, int window,
                                    const float *bias_slopes, attn_dtype dtype,
                                    void *stream);

/*
 * Bound, in nanoseconds, of every wait inside the library's kernels (one
 * thread waiting for another role of its block: a copy, a product, a
 * softmax step), for the calls made after it; 0 restores the default of
 * 2 s.  A wait that reaches the bound gives up: the block stops issuing
 * work, waits (bounded, 2 s) for its copies and products already in
 * flight, frees its tensor memory and exits, and the call's outputs are
 * undefined; attn_get_device_error() then returns ATTN_ERR_DEVICE_TIMEOUT.
 * A bound below 1000 ns gives up at the first wait whose condition is not
 * already met, which makes a timeout reproducible for tests of that path.
 * The setting is process-wide (all host threads, all devices).  The pages
 * have no counterpart: this is failure handling of the library itself.
 */
void attn_set_wait_limit_ns(uint64_t ns);

/*
 * Backward form for the bf16 calls that follow (process-wide, all host
 * threads and devices).  0, the default: with head_dim 128 the tensor-core
 * backward runs as one kernel per 128-key tile that computes S and dP once
 * per (row, key) pair and produces dK, dV and the tile's dQ contributions;
 * dQ is summed over key tiles in an fp32 accumulator with global reductions,
 * so its rounding depends on the order in which CTAs finish and can differ
 * in the last bits from run to run.  Nonzero: two kernels, one owning dK and
 * dV and one owning dQ (S and dP computed in both), no reductions, every
 * gradient reproducible bit for bit.  head_dim 64 and fp32 calls always take
 * the reproducible form.  attn_get_deterministic returns the setting.
 */
void attn_set_deterministic(int on);
int attn_get_deterministic(void);

/* Static description of a status code. */
const char *attn_status_string(attn_status status);

/*
 * The kernel plan the calling thread's last attn_fwd / attn_bwd chose (kernel
 * names, grid sizes, splits), so timings can be tied to the kernel that ran
 * ("attention-algorithm-error-and-complexity-tests", sixth paragraph).
 * Thread-local, valid until the thread's next call.
 */
const char *attn_last_plan(void);

/* Library ABI version (major * 100 + minor). */
int attn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_GB300_H */
