/*
 * gqaw.h -- C ABI of the windowed-KV-cache GroupQueryAttention step for GB300 (sm_103a).
 *
 * One call computes one com.microsoft::GroupQueryAttention step over a sliding-window
 * ("windowed") KV cache, as specified by these pages:
 *
 *  [P1] onnxruntime PR #32419 "Specify GroupQueryAttention windowed KV cache layout
 *       contract", Description: capacity C (dimension 2 of past_key), window
 *       W = local_window_size, G = C - W + 1, resident count
 *           L(T) = T                          if T <= C
 *           L(T) = T - G * ceil((T - C) / G)  otherwise,
 *       row i of present_key/present_value holds absolute position T - L + i for
 *       i in [0, L) and rows [L, C) are unspecified; any S >= 1 is accepted, including
 *       S > C; rejecting k draft tokens needs no cache edit and is exact iff
 *       L(T - k) == L(T) - k; the attention_bias last dimension stays
 *       total_sequence_length, indexed by absolute key position.  Review thread:
 *       T is per batch item, T_b = seqlens_k[b] + 1.
 *  [P2] onnxruntime PR #31142 "[CPU] Add windowed kv cache for GQA", Key design
 *       decisions: drifting layout (a whole G-row block is reclaimed at once),
 *       compaction skipped on drifting steps, staging for hazardous multi-token
 *       steps; review thread: planner arithmetic in 64-bit, P = seqlens_k[b] + 1 - S.
 *  [P3] onnxruntime/mobius issue #111 "GQA In-Place KV Cache: Investigation Report",
 *       Part 1.1 (inputs and outputs, BNSH caches), 1.2 (past and present may be one
 *       buffer), 1.3 (num_heads, kv_num_heads, scale = 1/sqrt(head_dim) by default,
 *       local_window_size, softcap with 0 = disabled, smooth_softmax), and the
 *       optional head_sink input of Part 1.1.
 *  [P4] onnxruntime PR #34226 "Fix CPU Attention causal mask for q_len=1 with past_key
 *       and kv_len > 1", Description: key j is visible to query i iff
 *       j <= i + past_sequence_length.
 *
 * What a step computes, per batch item b (T = seqlens_k[b] + 1, P = T - S,
 * Lp = L(P), Lt = L(T)):
 *   - the query of new token s sits at absolute position i = P + s and attends the
 *     keys j with i - W < j <= i (causal rule of [P4] plus the local window of W keys
 *     including itself); query head h reads kv head h / (num_heads / kv_num_heads);
 *     logit z_j = scale * q.k_j, then softcap * tanh(z_j / softcap) if softcap > 0,
 *     then + attention_bias[b, h, s, j]; softmax over the visible keys, its
 *     denominator joined by exp(head_sink[h]) (or exp(0) with smooth_softmax) when a
 *     sink is given; output is the weighted sum of the values, rounded to the cache
 *     dtype;
 *   - present rows [0, Lt) receive the Lt most recent positions of the past rows
 *     [0, Lp) followed by the S new rows (bit copies);
 *   - with a quantized cache (cache_dtype), the S new key and value rows become codes
 *     round_to_nearest_even(x / scale) computed in float and saturated to the code type
 *     (int8 [-128, 127]; e4m3 finite up to 448); attention reads every key and value,
 *     the new ones included, as code * scale;
 *   - with do_rotary, the S new query and key rows are first turned by the rotary
 *     embedding of their positions (pairs of dimensions (x1, x2) -> (x1 cos - x2 sin,
 *     x2 cos + x1 sin) with cos/sin from row pos of the caches; RoFormer's rotation),
 *     rounded once to dtype; the turned keys are the ones attended and stored.
 *
 * Memory.  The caller owns every buffer.  The library allocates nothing; all work is
 * enqueued on the caller's stream and the call returns without synchronising.
 *
 * Errors.  Every function returning gqaw_status checks its arguments on the host first
 * and, if they are wrong, returns an error code before enqueuing anything and leaves
 * every output untouched; gqaw_last_error() then describes the problem.  Per-item
 * problems only visible on the device (seqlens_k[b] + 1 - S < 0, or
 * seqlens_k[b] + 1 > total_sequence_length) set a bit of the device status word kept in
 * the workspace; that item's output and present rows are then unspecified and the
 * other items are computed normally.  gqaw_device_status() reads the word.  No kernel
 * traps; every wait inside a kernel is bounded and sets a status bit if it expires.
 */
#ifndef GQAW_H
#define GQAW_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum gqaw_status {
  GQAW_OK = 0,
  GQAW_EINVAL = 1,      /* an argument is malformed (null, misaligned, out of range) */
  GQAW_EUNSUPPORTED = 2, /* well formed but not implemented (e.g. head_size 96) */
  GQAW_ECUDA = 3,       /* a CUDA runtime call failed; gqaw_last_error() has its message */
  GQAW_EWORKSPACE = 4,  /* workspace missing, misaligned or smaller than gqaw_workspace_bytes() */
  GQAW_EDEVICE = 5      /* gqaw_device_status(): the device status word is non-zero */
} gqaw_status;

typedef enum gqaw_dtype {
  GQAW_F32 = 0,  /* float32 query/key/value/cache/output */
  GQAW_BF16 = 1, /* bfloat16 query/key/value/cache/output */
  GQAW_I8 = 2,   /* cache_dtype only: int8 codes of a quantized cache */
  GQAW_E4M3 = 3  /* cache_dtype only: fp8 e4m3 codes (OCP 8-bit floating point) */
} gqaw_dtype;

/* Bits of the device status word. */
#define GQAW_DEV_BAD_SEQLEN 1u /* some seqlens_k[b] + 1 - S < 0 or > total_sequence_length */
#define GQAW_DEV_TIMEOUT 2u    /* a bounded in-kernel wait expired (an internal fault) */
#define GQAW_DEV_BAD_POSITION 4u /* a rotary position outside [0, rotary_cache_len) */
#define GQAW_DEV_QUERY_RANGE 8u  /* quantized cache on the tensor-core small-step path
                                    (head_size 128, S x group <= 32): a finite query
                                    element of magnitude >= 65520, which has no finite
                                    fp16 value; the output is then unspecified */
#define GQAW_DEV_INTERNAL 16u    /* an internal consistency check failed (a library
                                    fault): the step's results are unspecified */

/* Arguments of one step.  All tensor pointers are DEVICE pointers.  Layouts are
 * row-major with the shapes given; "BNSH" is (batch, kv head, row, head_size).
 * Alignment: every tensor pointer except seqlens_k, attention_bias and head_sink must be
 * 16-byte aligned; those three 4-byte aligned; workspace 256-byte aligned. */
typedef struct gqaw_step_args {
  int32_t batch_size;            /* B >= 0; B == 0 is a valid empty step */
  int32_t sequence_length;       /* S >= 1 new tokens per item (same S for every item) */
  int32_t num_heads;             /* Nq >= 1 */
  int32_t kv_num_heads;          /* Nkv >= 1, Nq % Nkv == 0 */
  int32_t head_size;             /* D: one of 8, 16, 32, 64, 128, 256 */
  int32_t capacity;              /* C >= 1: rows per (b, kv head) slice of the caches */
  int32_t local_window_size;     /* W, 1 <= W <= C */
  int32_t dtype;                 /* gqaw_dtype of query/key/value/caches/output */
  float scale;                   /* > 0, or 0 for the default 1/sqrt(D) */
  float softcap;                 /* >= 0; 0 disables soft-capping */
  int32_t total_sequence_length; /* host scalar >= S: max_b T_b, the bias column count */
  int32_t split_keys;            /* 0: automatic; > 0 overrides the keys per split-K chunk */
  const void *query;             /* (B, S, Nq*D) */
  const void *key;               /* (B, S, Nkv*D): the S new keys */
  const void *value;             /* (B, S, Nkv*D): the S new values */
  const void *past_key;          /* (B, Nkv, C, D) BNSH; rows [0, L(P_b)) are read */
  const void *past_value;        /* (B, Nkv, C, D) BNSH */
  void *present_key;             /* (B, Nkv, C, D): == past_key (in place) or disjoint */
  void *present_value;           /* (B, Nkv, C, D): == past_value (in place) or disjoint */
  const int32_t *seqlens_k;      /* (B,) int32: T_b - 1 */
  const float *attention_bias;   /* NULL, or fp32 element [b*sb + h*sh + s*ss + j] with
                                    j in [0, total_sequence_length) the absolute key
                                    position; the last dimension is contiguous */
  int64_t bias_stride_b;         /* sb >= 0 (elements; 0 broadcasts over the batch) */
  int64_t bias_stride_h;         /* sh >= 0 (0 broadcasts over heads) */
  int64_t bias_stride_s;         /* ss >= 0 */
  void *output;                  /* (B, S, Nq*D) */
  void *workspace;               /* device scratch of gqaw_workspace_bytes() bytes, zeroed
                                    once with gqaw_workspace_init() before first use (and
                                    again after a device error); it holds the device
                                    status word, the list of items whose rows move, the
                                    split-K tickets and partial results.  Every completed
                                    step leaves its counters and tickets at zero.  Where
                                    the tickets sit depends on the step's shape (B, S,
                                    kernel, split count): the library remembers, per
                                    workspace address, the ticket region of the last
                                    step enqueued on it, and a step whose region differs
                                    first clears its own (one cudaMemsetAsync on its
                                    stream), so one workspace serves steps of any shape
                                    in stream order.  A CUDA graph replays only the
                                    clears recorded while it was captured: between replays
                                    and direct calls of another shape on one workspace,
                                    call gqaw_workspace_init().  Steps that share a
                                    workspace must not overlap on the GPU. */
  size_t workspace_bytes;
  int32_t *resident_len_out;     /* NULL, or (B,) int32 receiving L(T_b) */
  const float *head_sink;        /* NULL, or (Nq,) fp32: one sink logit per query head
                                    ([P3] Part 1.1, input 11); 4-byte aligned */
  int32_t smooth_softmax;        /* non-zero: a sink logit of 0 for every head ([P3]
                                    Part 1.3); ignored when head_sink is given */
  int32_t do_rotary;             /* non-zero: turn the new query and key rows by the
                                    rotary embedding before use ([P3] Part 1.3).  The
                                    turn is computed in fp32 and rounded once to the
                                    cache dtype (or its code), so the stored key rows
                                    may differ by one rounding step from a turn in
                                    higher precision: present keys are bit-exact copies
                                    of the step's inputs only without do_rotary (values
                                    always are) */
  int32_t rotary_interleaved;    /* non-zero: pairs (2i, 2i+1); 0: pairs (i, i + rd/2) */
  int32_t rotary_dim;            /* rd: even, 2 <= rd <= D; 0 means D.  Dimensions from
                                    rd on are not turned */
  int32_t rotary_cache_len;      /* >= 1: rows of cos_cache and sin_cache */
  const void *cos_cache;         /* (rotary_cache_len, rd/2) in dtype, element-aligned */
  const void *sin_cache;         /* (rotary_cache_len, rd/2) in dtype, element-aligned */
  const int64_t *position_ids;   /* NULL (token s of item b at position
                                    seqlens_k[b] + 1 - S + s), or (B, S) int64, 8-byte
                                    aligned ([P3] Part 1.1) */
  int32_t cache_dtype;           /* 0: the caches hold `dtype`; GQAW_I8 or GQAW_E4M3: they
                                    hold 1-byte codes of a quantized cache ([P3] Part 1.1,
                                    k_scale and v_scale); needs dtype GQAW_BF16 and
                                    head_size 64, 128 or 256.  With head_size 128 and
                                    S x group <= 32 the tensor cores take the query as
                                    fp16: elements must stay below 65520 in magnitude
                                    (else GQAW_DEV_QUERY_RANGE), and those below fp16's
                                    normal range (6.1e-5) keep its subnormal spacing
                                    (6e-8) */
  const float *k_scale;          /* quantized cache: device fp32 scalar, > 0; a key code c
                                    stands for c * k_scale.  Otherwise ignored */
  const float *v_scale;          /* quantized cache: the same for values */
} gqaw_step_args;

/* L(T) of [P1] in 64-bit arithmetic.  Pure host function.  Returns -1 if T < 0,
 * C < 1, W < 1 or W > C. */
int64_t gqaw_resident_len(int64_t T, int64_t C, int64_t W);

/* Rollback rule of [P1]: 1 if rejecting the last k tokens of a cache of length T is
 * exact (L(T - k) == L(T) - k), 0 if not, -1 on invalid arguments (k < 0, k > T, or
 * invalid T, C, W as for gqaw_resident_len).  Pure host function. */
int gqaw_rollback_exact(int64_t T, int64_t k, int64_t C, int64_t W);

/* Workspace bytes the step needs for these arguments (only the size fields, dtype and
 * split_keys are read; pointers may be NULL).  Returns 0 if the sizes are invalid
 * (gqaw_last_error() says why).  Always at least 256. */
size_t gqaw_workspace_bytes(const gqaw_step_args *args);

/* Zero all `workspace_bytes` bytes of `workspace` on `stream` (cudaMemsetAsync), and
 * note that the workspace is clean (the next step needs no ticket clear). */
gqaw_status gqaw_workspace_init(void *workspace, size_t workspace_bytes, void *stream);

/* One whole step, enqueued on `stream` (a cudaStream_t; NULL = the legacy default
 * stream): attention over the pre-step cache rows and the new rows, then the cache
 * update (block compaction on eviction steps, append of the new rows).  Equivalent to
 * gqaw_attend() followed by gqaw_update_cache() on the same stream. */
gqaw_status gqa_windowed_step(const gqaw_step_args *args, void *stream);

/* First phase only (one kernel): the attention over the pre-step rows and the new rows,
 * including the merge of split key chunks, so the output is complete when it ends;
 * resident_len_out; the append of the new rows of every item that reclaims no block
 * with past == present (rows [L(P), L(P) + S), which no query reads).  Items that
 * reclaim a block ([P2] block compaction), and all items when present is a separate
 * buffer, are recorded in the workspace for gqaw_update_cache(), except what the
 * small-step tensor-core kernel (bf16 cache, head_size 128, S * group <= 32) writes
 * itself from the key and value tiles it reads: the whole update of an item whose
 * surviving rows lie in its window, and with a separate present buffer the window's
 * rows (only the rows below the window are then recorded). */
gqaw_status gqaw_attend(const gqaw_step_args *args, void *stream);

/* Second phase only (one kernel): for the items gqaw_attend() recorded, moves the
 * surviving rows and appends the new rows; then clears the record.  Must follow
 * gqaw_attend() with the same arguments on the same stream (the in-place update
 * overwrites rows the attention reads). */
gqaw_status gqaw_update_cache(const gqaw_step_args *args, void *stream);

/* Copy the device status word of `workspace` to *flags (synchronises `stream`); zero it
 * afterwards if `reset` is non-zero.  Returns GQAW_EDEVICE if the word was non-zero. */
gqaw_status gqaw_device_status(void *workspace, uint32_t *flags, int reset, void *stream);

/* Message of the last error returned on the calling thread ("" if none). */
const char *gqaw_last_error(void);

/* Number of kernels this library has launched in this process. */
uint64_t gqaw_launch_count(void);

/* sizeof(gqaw_step_args) as compiled into the library, so that a binding written in
 * another language can check its copy of the struct layout. */
size_t gqaw_step_args_size(void);

/* Size of the static scratch used by gqa_windowed_step_noalloc (8 MiB). */
#define GQAW_NOALLOC_SCRATCH_BYTES (8u * 1024u * 1024u)

/* The same step as gqa_windowed_step, for callers that cannot allocate device memory
 * (for example a plugin inside an inference runtime that owns all device memory and
 * gives the plugin no allocator, or a serving loop that allows no allocation after
 * start-up).  The pages have no counterpart: this is a deployment variant only.
 *
 * The split-K scratch normally taken from args->workspace comes instead from a
 * fixed-size array compiled into the library (GQAW_NOALLOC_SCRATCH_BYTES; every GPU
 * that loads the library holds it until the process exits).  args->workspace and
 * args->workspace_bytes are ignored; all other fields mean what they mean for
 * gqa_windowed_step.  Nothing is allocated: no cudaMalloc, no cudaFree, no allocating
 * library call.
 *
 * The first call on a device looks up the array's device address (cudaGetSymbolAddress,
 * with that device current) and zeroes the whole array with cudaMemsetAsync on
 * `stream`; make that first call before any stream capture.  Later calls reuse the
 * address.  Every call on a device shares the one array, which keeps the previous
 * call's contents.  So every call first clears, with one cudaMemsetAsync of a few KB on
 * `stream`, the part of the array that its step needs at zero: the device status word,
 * the cache-update counters and list, and the split-K tickets, whose place depends on
 * the step's shape.  A call therefore never depends on what an earlier call left there,
 * whatever its shape, even one that stopped on a device error.  The split-K partials
 * that follow are always written before they are read.  Calls that overlap on the GPU
 * (several streams at once) race on the array and must be ordered by the caller.  The
 * device status word lives in the array and is not reported by this entry point.
 *
 * Returns GQAW_EWORKSPACE, before enqueuing anything, when the step needs more scratch
 * than the array holds (gqaw_workspace_bytes(args) > GQAW_NOALLOC_SCRATCH_BYTES); the
 * other errors are those of gqa_windowed_step. */
gqaw_status gqa_windowed_step_noalloc(const gqaw_step_args *args, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* GQAW_H */
