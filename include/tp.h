/*
 * tp.h -- C ABI of the tensor-parallel transformer block on one GPU.
 *
 * The block is the Megatron-style decomposition described on
 * undercodenews.com/?p=110319, section "the Original": Q/K/V and the first
 * FFN linear are column-parallel (every shard multiplies the full input by
 * its slice of the output features, so shard s owns heads
 * [s*H/tp, (s+1)*H/tp)), attention runs per shard over its own heads, and
 * the output projection and the second FFN linear are row-parallel, their
 * per-shard partial products being summed by an all-reduce.  Here all tp
 * shards are logical partitions of one GPU's memory and the all-reduce is a
 * sum of the partials inside the row-parallel GEMM's accumulator.
 *
 * Block computed by tp_block_forward (residuals, activation, mask and scale
 * are readings where the pages are silent; the design notes list them):
 *     Q, K, V = X Wq^T, X Wk^T, X Wv^T                 (column-parallel, by head)
 *     A       = concat_j softmax(Q_j K_j^T / sqrt(d_head) + mask) V_j
 *     H       = X + sum_s A_s Wo_s^T                    (row-parallel + reduce)
 *     U       = silu(H Wg^T) * (H Wu^T)   or  gelu(H W1^T)   (column-parallel)
 *     Y       = H + sum_s U_s Wd_s^T                    (row-parallel + reduce)
 *
 * Conventions shared by every call:
 *  - Pointers named "device" point to device memory owned by the caller; the
 *    library never allocates device memory and never frees caller memory.
 *    A plan owns only host metadata (and cached TMA descriptors).
 *  - Matrices are row-major.  Weights use the [out_features, in_features]
 *    layout.  M = batch * seq tokens; token t of sequence b is row b*seq + t.
 *  - "act" tensors have the plan's storage dtype (bf16 or fp32); fp32 tensors
 *    are always fp32.  bf16 is IEEE bfloat16 (round to nearest even).
 *  - `stream` is a cudaStream_t passed as void*; NULL is the legacy default
 *    stream.  Every call only enqueues work and returns; results are ready
 *    when the stream reaches them.
 *  - Arguments are validated on the host before anything is enqueued; a call
 *    that returns a validation error (any code but TP_ERR_CUDA) has enqueued
 *    nothing -- the whole-block calls check every step's arguments before
 *    their first launch.  Device pointers must be
 *    16-byte aligned (TP_ERR_ALIGNMENT otherwise).  Launch failures return
 *    TP_ERR_CUDA.  Device-side bounded waits that give up record a code that
 *    tp_sync_status() reports as TP_ERR_DEVICE_TIMEOUT.
 *  - A plan is immutable after creation and may be used from several host
 *    threads and streams at once, provided calls in flight at the same time
 *    do not share output or workspace buffers.
 *  - Tracing: every call that enqueues work opens an NVTX range named after
 *    the call for its host duration; the whole-block calls add one range per
 *    step ("S1 column QKV" ... "S5 row FFN-down + reduce", "RMSNorm(...)")
 *    and per stacked layer, so profilers attribute each launch to its step.
 */
#ifndef TP_H_
#define TP_H_

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct tp_plan_s* tp_plan_t;

typedef enum {
    TP_OK = 0,
    TP_ERR_NULL_ARG = 1,              /* a required pointer is NULL            */
    TP_ERR_INVALID_DIM = 2,           /* a dimension or size is <= 0 / out of range */
    TP_ERR_DEGREE_RANGE = 3,          /* tp_degree < 1 or tp_degree > n_heads  */
    TP_ERR_HEADS_NOT_DIVISIBLE = 4,   /* n_heads % tp_degree != 0              */
    TP_ERR_FFN_NOT_DIVISIBLE = 5,     /* d_ffn % tp_degree != 0                */
    TP_ERR_DMODEL_NOT_DIVISIBLE = 6,  /* d_model % n_heads != 0                */
    TP_ERR_ALIGNMENT = 7,             /* pointer not 16-byte aligned, or a width
                                         not a multiple of 8 elements          */
    TP_ERR_WORKSPACE_TOO_SMALL = 8,
    TP_ERR_UNSUPPORTED = 9,           /* valid plan, shape the library has no kernel for */
    TP_ERR_CUDA = 10,                 /* a CUDA runtime/launch error           */
    TP_ERR_DEVICE_TIMEOUT = 11        /* a device-side bounded wait gave up    */
} tp_status;

typedef enum { TP_ACT_GELU = 0, TP_ACT_SWIGLU = 1 } tp_act;
typedef enum { TP_BF16 = 0, TP_FP32 = 1 } tp_dtype;
typedef enum { TP_QKV = 0, TP_FFN_UP = 1 } tp_column_which;
typedef enum { TP_ATTN_OUT = 0, TP_FFN_DOWN = 1 } tp_row_which;

/* Human-readable name of a status code (static string, never NULL). */
const char* tp_status_string(tp_status s);

/* Text of the last CUDA error that made a call on this host thread return
 * TP_ERR_CUDA ("" if none).  Thread-local storage owned by the library. */
const char* tp_last_cuda_error(void);

/*
 * Create a plan.  Degree rule from undercodenews.com/?p=110319, "the
 * Original" (degree <= head count, head count and FFN width divisible by
 * the degree) and "What Is Tensor Parallelism?" (netray.co), "Tensor
 * Parallelism Explained".  Checks, first failure returned:
 *   d_model, n_heads, d_ffn > 0            else TP_ERR_INVALID_DIM
 *   tp_degree >= 1                         else TP_ERR_DEGREE_RANGE
 *   d_model % n_heads == 0                 else TP_ERR_DMODEL_NOT_DIVISIBLE
 *   tp_degree <= n_heads                   else TP_ERR_DEGREE_RANGE
 *   n_heads % tp_degree == 0               else TP_ERR_HEADS_NOT_DIVISIBLE
 *   d_ffn % tp_degree == 0                 else TP_ERR_FFN_NOT_DIVISIBLE
 * then the library's storage constraint: d_model, d_head and d_ffn/tp
 * multiples of 8 (TP_ERR_ALIGNMENT), so that every row starts 16-byte
 * aligned.  An unknown act/dtype gives TP_ERR_UNSUPPORTED.
 * tp_plan_create uses SwiGLU and bf16.  On error *out is set to NULL.
 * Host only: touches no GPU.
 */
tp_status tp_plan_create(int d_model, int n_heads, int d_ffn, int tp_degree, tp_plan_t* out);
tp_status tp_plan_create_ex(int d_model, int n_heads, int d_ffn, int tp_degree,
                            tp_act act, tp_dtype dtype, tp_plan_t* out);
void tp_plan_destroy(tp_plan_t plan);

/*
 * Bytes the caller must provide: the packed shard-major weights (written by
 * tp_shard_weights) and the workspace tp_block_forward needs for `batch`
 * sequences of `seq` new tokens.  Either output pointer may be NULL.
 */
tp_status tp_plan_sizes(tp_plan_t plan, int batch, int seq,
                        size_t* packed_weight_bytes, size_t* workspace_bytes);

/* Bytes of scratch tp_attention_heads needs for this call shape (0 for
 * prefill-shaped calls; split-KV partials for single-token decode). */
tp_status tp_attention_scratch_bytes(tp_plan_t plan, int batch, int seq_q, int cache_cap,
                                     size_t* bytes);

/* Bytes of the optional scratch that tp_column_linear / tp_row_linear_reduce
 * take for M token rows (0 when no kernel for that shape uses it). */
tp_status tp_linear_scratch_bytes(tp_plan_t plan, int M, size_t* bytes);

/*
 * Pack full weights (device, plan dtype, [out, in] row-major) into the
 * shard-major layout the kernels read (device, `packed`, at least
 * packed_weight_bytes).  Shard s receives: the Q, K and V rows of its heads
 * (column-parallel by head); the columns of Wo that meet its heads
 * (row-parallel); its d_ffn/tp rows of Wg and Wu interleaved in blocks of g
 * rows (g gate rows, the g matching up rows, ...; g = 32 when d_ffn/tp is a
 * multiple of 32, else 16, else 8) or its rows of W1; its d_ffn/tp columns
 * of Wd.  Wup must be NULL for GELU plans and non-NULL for SwiGLU plans.
 */
tp_status tp_shard_weights(tp_plan_t plan, const void* Wq, const void* Wk, const void* Wv,
                           const void* Wo, const void* W1_or_Wgate, const void* Wup,
                           const void* Wdown, void* packed, void* stream);

/*
 * Column-parallel linear over all shards in one launch
 * (undercodenews.com/?p=110319, "the Original": each shard multiplies the
 * full input by its slice of the output features).
 *   x          device act [M, d_model]
 *   out_shards device act [tp][M][n_s], where
 *      TP_QKV:    n_s = 3*h_l*d_head, row = [Q of its h_l heads | K | V],
 *                 each head's d_head columns contiguous, heads in order;
 *      TP_FFN_UP: n_s = d_ffn/tp, the activated U_s = silu(x Wg_s^T) *
 *                 (x Wu_s^T) (SwiGLU) or gelu(x W1_s^T) (GELU, erf form).
 *   scratch    device, nullable, scratch_bytes >= tp_linear_scratch_bytes(M)
 *              to be used; contents on entry are ignored (a call that
 *              splits tiles first clears the 16 KB counter block at the
 *              start of the scratch, on the same stream; the whole-block
 *              calls clear it once for their four linears).  With it, a
 *              tensor-core GEMM whose output tiles would leave SMs idle in
 *              the last wave cuts each tile of that wave into equal
 *              k-parts on different SMs (run before the whole tiles): every
 *              part writes its fp32 partial sums to the scratch and counts
 *              itself in; at the end of its SM's work (bounded wait for the
 *              tile's other parts) each part adds the partials of its own
 *              rows of the tile in part order 0, 1, ... and applies the
 *              epilogue -- inside the same launch, with no second pass.
 *              Calls in flight at the same time need separate
 *              scratch.
 * M >= 1.
 */
tp_status tp_column_linear(tp_plan_t plan, int which, const void* x, int M,
                           const void* packed, void* out_shards, void* scratch,
                           size_t scratch_bytes, void* stream);

/*
 * Row-parallel linear with the all-reduce fused in (same page and section:
 * the input's column blocks meet the weight's matching row blocks and the
 * partials are summed).  Computes
 *   out_f32[M, d] = residual + sum_{s=0}^{tp-1} in_shards[s] W_s^T
 * with the shard partials accumulated in fp32, in shard order, in the
 * GEMM's accumulator -- no partial ever goes to memory.
 *   in_shards  device act [tp][M][k_s]; k_s = h_l*d_head (TP_ATTN_OUT) or
 *              d_ffn/tp (TP_FFN_DOWN)
 *   residual   device, nullable, [M, d]: plan dtype for TP_ATTN_OUT (the
 *              block input), fp32 for TP_FFN_DOWN (H)
 *   out_f32    device fp32 [M, d]
 *   out_act    device act [M, d], nullable: a copy of out_f32 in the plan
 *              dtype (the operand of the next column-parallel linear)
 *   scratch    as in tp_column_linear.  When a tile is cut into parts, a
 *              part spans consecutive k-blocks of the shard-major reduction
 *              (so it may cover several shards' partials), and the parts'
 *              fp32 sums are added in part order.
 */
tp_status tp_row_linear_reduce(tp_plan_t plan, int which, const void* in_shards, int M,
                               const void* packed, const void* residual, void* out_f32,
                               void* out_act, void* scratch, size_t scratch_bytes,
                               void* stream);

/*
 * Per-shard multi-head attention over each shard's own heads
 * (undercodenews.com/?p=110319, "the Original": every head attends
 * independently, no communication).  For each sequence b, shard s and local
 * head j (global head h = s*h_l + j):
 *   O = softmax(Q K^T / sqrt(d_head) + mask) V
 * The seq_q query tokens sit at positions cache_pos .. cache_pos+seq_q-1.
 * With causal != 0 a query at position p sees keys at positions <= p.
 *   qkv_shards  device act [tp][batch*seq_q][3*h_l*d_head] (tp_column_linear
 *               TP_QKV layout)
 *   k_cache, v_cache  device act [batch][n_heads][cache_cap][d_head], or both
 *               NULL.  When given, the new tokens' K and V are written at
 *               positions cache_pos.. and attention runs over positions
 *               0 .. cache_pos+seq_q-1 of the cache ("Tensor Parallelism:
 *               Splitting One Layer Across GPUs" (byteledger), "Interaction
 *               with the rest of serving": the KV cache is split with the
 *               heads -- head h's cache rows belong to its shard).  When
 *               NULL, cache_pos must be 0 and the seq_q tokens attend among
 *               themselves.
 *   out_shards  device act [tp][batch*seq_q][h_l*d_head]
 *   scratch     device, scratch_bytes >= tp_attention_scratch_bytes(); may be
 *               NULL when that is 0.  Contents on entry are ignored.
 */
tp_status tp_attention_heads(tp_plan_t plan, const void* qkv_shards, int batch, int seq_q,
                             int causal, void* k_cache, void* v_cache, int cache_cap,
                             int cache_pos, void* out_shards, void* scratch,
                             size_t scratch_bytes, void* stream);

/*
 * Single-token decode attention that allocates nothing and takes no scratch
 * buffer.  (The pages have no counterpart: this serves callers that cannot
 * allocate device memory on their decode path -- code running inside a
 * memory pool it does not own, a host framework that forbids cudaMalloc
 * there, or a process whose allocator is exhausted.)
 * Same result as tp_attention_heads(plan, qkv_shards, batch, 1, causal=1,
 * k_cache, v_cache, cache_cap, cache_pos, out_shards, scratch, ...): the new
 * token's K/V are written at cache_pos and each head attends over positions
 * 0..cache_pos.  The split-KV partials go to a fixed 8 MiB device array
 * inside the library (held by every GPU that loads it until process exit)
 * instead of `scratch`; batch * n_heads * 64 * (d_head + 2) * 4 bytes must
 * fit in it, else TP_ERR_WORKSPACE_TOO_SMALL and nothing is enqueued.
 *  - The first call on each device looks up that array's device address
 *    (cudaGetSymbolAddress, with the device current); make that first call
 *    before any stream capture.  The address is kept for the life of the
 *    process and does not survive cudaDeviceReset().
 *  - All calls on a device share the one array, so calls that can overlap
 *    on the GPU (different streams, no ordering between them) race and give
 *    wrong results; order them on one stream or with events.
 *  - The array keeps the last call's partials; every call rewrites what it
 *    reads, so no clearing is needed.
 */
tp_status tp_attention_decode_noalloc(tp_plan_t plan, const void* qkv_shards, int batch,
                                      void* k_cache, void* v_cache, int cache_cap, int cache_pos,
                                      void* out_shards, void* stream);

/*
 * The whole block: column QKV, attention, row O + reduce (+x), column
 * FFN-up + activation, row FFN-down + reduce (+H).
 *   x         device act [batch*seq][d_model]
 *   k_cache/v_cache/cache_cap/cache_pos   as in tp_attention_heads
 *   packed    device, from tp_shard_weights
 *   workspace device, ws_bytes >= tp_plan_sizes(batch, seq) workspace bytes
 *             (contents on entry are ignored; it holds the linears'
 *             scratch, see tp_column_linear)
 *   out_f32   device fp32 [batch*seq][d_model] = Y
 */
tp_status tp_block_forward(tp_plan_t plan, const void* x, int batch, int seq, int causal,
                           void* k_cache, void* v_cache, int cache_cap, int cache_pos,
                           const void* packed, void* workspace, size_t ws_bytes,
                           void* out_f32, void* stream);

/*
 * A stack of n_layers blocks of the plan's shape (each with its own packed
 * weights and, optionally, its own KV cache), the output of layer l feeding
 * layer l + 1 -- the layers a device_map or pipeline split would place on
 * different GPUs (undercodenews "device-map-vs-tensor-parallelism-exposed",
 * "the Original"; undercodenews.com/?p=110319), here all tensor-parallel on
 * one GPU.  Between layers the activation is stored in the plan dtype (the
 * next layer's input is the plan-dtype copy of the previous layer's Y);
 * out_f32 receives the last layer's Y.
 *   packed_layers  host array of n_layers device pointers (tp_shard_weights)
 *   k_caches, v_caches  host arrays of n_layers device caches (as in
 *                  tp_attention_heads) or both NULL
 *   workspace      device, ws_bytes >= tp_stack_workspace_bytes(batch, seq)
 */
tp_status tp_stack_workspace_bytes(tp_plan_t plan, int batch, int seq, size_t* bytes);
tp_status tp_stack_forward(tp_plan_t plan, int n_layers, const void* const* packed_layers, const void* x,
                           int batch, int seq, int causal, void* const* k_caches, void* const* v_caches,
                           int cache_cap, int cache_pos, void* workspace, size_t ws_bytes, void* out_f32,
                           void* stream);

/*
 * Sequence parallelism around the tensor-parallel regions (undercodenews.com/
 * ?p=110319, "What Undercode Say": tensor parallelism is combined with
 * sequence parallelism, which spreads the sequence's tokens across the
 * devices; the mechanics below are the usual reading, not on the page).
 * Outside the tensor-parallel linears and attention the M = batch*seq token
 * rows (row b*seq + t) are held as tp slices: slice s = rows
 * [s*M/tp, (s+1)*M/tp), stored from base + s * slice_stride elements of the
 * buffer's own type, rows of d_model elements (so slices may live in
 * separate, padded regions).  The all-reduce after a row-parallel linear
 * becomes a reduce-scatter -- every row's shard-order sum (plus its
 * residual) is written into its slice -- and a column-parallel linear reads
 * the all-gather of the slices (its tensor-core GEMM reads the rows straight
 * from the slices through its tensor map).  Results equal those of the
 * plain calls on the concatenated rows.
 * Requirements (else nothing is enqueued): bf16 plan (TP_ERR_UNSUPPORTED);
 * M divisible by tp (TP_ERR_INVALID_DIM); M / tp and slice_stride multiples
 * of 8 (TP_ERR_ALIGNMENT); slice_stride >= (M / tp) * d_model
 * (TP_ERR_INVALID_DIM).  All three run on the tensor-core GEMMs.
 *
 * tp_column_linear_gather: as tp_column_linear, x given as slices
 *   (device act); TP_ERR_UNSUPPORTED for a pre-norm plan, as there.
 * tp_row_linear_reduce_scatter: as tp_row_linear_reduce, with residual
 *   (nullable), out_f32 and out_act (nullable) given as slices, all with
 *   slice_stride.
 * tp_block_forward_seq: as tp_block_forward (same workspace; caches as
 *   there; pre-norm plans too: the norms run
 *   on the slices' rows), x as slices x_stride apart, Y (fp32) written as
 *   slices y_stride apart; H stays in the workspace.
 */
tp_status tp_column_linear_gather(tp_plan_t plan, int which, const void* x_slices, long long slice_stride, int M,
                                  const void* packed, void* out_shards, void* scratch, size_t scratch_bytes,
                                  void* stream);
tp_status tp_row_linear_reduce_scatter(tp_plan_t plan, int which, const void* in_shards, int M, const void* packed,
                                       const void* residual_slices, void* out_f32_slices, void* out_act_slices,
                                       long long slice_stride, void* scratch, size_t scratch_bytes, void* stream);
tp_status tp_block_forward_seq(tp_plan_t plan, const void* x_slices, long long x_stride, int batch, int seq,
                               int causal, void* k_cache, void* v_cache, int cache_cap, int cache_pos,
                               const void* packed, void* workspace, size_t ws_bytes, void* out_f32_slices,
                               long long y_stride, void* stream);

/*
 * Pre-norm (LLaMA-style) variant of the block.  Norms and rotary embedding
 * are not on the pages ("What Is Tensor Parallelism?", netray.co, and
 * undercodenews.com/?p=110319 shard only the linears and attention); this
 * is the usual reading of a LLaMA-shaped block, with the same
 * tensor-parallel split:
 *   H = X + Attn(RMSNorm(X; g_attn)),  Y = H + SwiGLU-FFN(RMSNorm(H; g_ffn)),
 *   RMSNorm(x; g) = x / sqrt(mean(x^2) + rms_eps) * g,
 * and Q, K rotated per head: the pair (2i, 2i+1) of the token at absolute
 * position p (cache_pos + t) by the angle p * rope_theta^(-2i/d_head)
 * (rope_theta 0: no rotation).  The KV cache holds rotated keys.
 *
 * tp_plan_create_llama: bf16, SwiGLU; rms_eps > 0 and finite, rope_theta
 *   >= 0 and finite (else TP_ERR_INVALID_DIM); the tp_plan_create_ex rules;
 *   d_ffn/tp a multiple of 32 (else TP_ERR_UNSUPPORTED).
 * tp_shard_weights_llama: as tp_shard_weights, then the gains g_attn,
 *   g_ffn (device, bf16 [d_model], 16-byte aligned) are multiplied into the
 *   packed QKV and gate/up columns (W diag(g), rounded to bf16), so the
 *   norm costs one fp32 row scale in the linears' epilogues.
 *   TP_ERR_UNSUPPORTED on a plan not made by tp_plan_create_llama.
 * tp_block_forward / tp_stack_forward take such a plan unchanged (the
 *   workspace sizes include the per-row scales); tp_column_linear returns
 *   TP_ERR_UNSUPPORTED for it (its inputs lack the norm scales and
 *   positions); tp_row_linear_reduce and tp_attention_heads are unchanged.
 */
tp_status tp_plan_create_llama(int d_model, int n_heads, int d_ffn, int tp_degree, float rms_eps,
                               float rope_theta, tp_plan_t* out);
tp_status tp_shard_weights_llama(tp_plan_t plan, const void* Wq, const void* Wk, const void* Wv,
                                 const void* Wo, const void* Wgate, const void* Wup, const void* Wdown,
                                 const void* g_attn, const void* g_ffn, void* packed, void* stream);

/*
 * Wait for `stream`, then report (and clear) the first device-side error
 * recorded by a bounded wait in this library's kernels on the current
 * device: TP_ERR_DEVICE_TIMEOUT, TP_ERR_CUDA on a CUDA error, else TP_OK.
 * After TP_ERR_DEVICE_TIMEOUT the outputs of the calls since the last
 * check are undefined.  The device address of the error word (like that of
 * tp_attention_decode_noalloc's array) is looked up once per device and
 * kept for the life of the process: it does not survive cudaDeviceReset().
 */
tp_status tp_sync_status(void* stream);

/*
 * Limit of every bounded device-side wait (mbarrier waits of the
 * tensor-core kernels, the split-tile counters of the linears), in
 * nanoseconds of %globaltimer, for launches enqueued after the call; 0
 * restores the default of 2 s.  A wait that runs out records the error
 * tp_sync_status() reports, and its kernel leaves early with its tensor
 * memory freed.  Meant for tests of that failure path (a short limit makes
 * waits run out); process-wide, not tied to a plan.
 */
void tp_set_wait_timeout_ns(unsigned long long ns);

/*
 * Host-only description (no GPU needed) of how tp_column_linear (which =
 * TP_QKV / TP_FFN_UP, row = 0) or tp_row_linear_reduce (which =
 * TP_ATTN_OUT / TP_FFN_DOWN, row = 1) would run M token rows with a linear
 * scratch of scratch_bytes, on a GPU with `sms` SMs of which `pair_slots`
 * SM pairs fit at once (148 and 74 on a B300).  kernel: 0 tensor-core
 * GEMM, 1 weight streaming on the tensor cores (2..32 rows), 2 weight
 * streaming on the CUDA cores, 3 fp32 CUDA-core GEMM.  For kernel 0: tiles
 * (256 x 256 on SM pairs when paired, else 128 x 256), k-blocks of 64 per
 * tile, the tiles run whole, the parts each remaining tile is cut into
 * (the parts run first), the work items, the units launched and the bytes
 * of scratch the launch touches (<= scratch_bytes).
 */
typedef struct {
    int kernel, paired, tiles, k_blocks_per_tile, whole_tiles, parts, items, units;
    size_t scratch_bytes_touched;
} tp_linear_schedule_t;
tp_status tp_linear_schedule(tp_plan_t plan, int row, int which, int M, size_t scratch_bytes, int sms,
                             int pair_slots, tp_linear_schedule_t* out);

#ifdef __cplusplus
}
#endif

#endif /* TP_H_ */
