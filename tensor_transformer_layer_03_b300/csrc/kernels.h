// Internal launch interface between the C ABI (tp_api.cu) and the kernels.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace tpk {

// ---- weight packing (pack.cu) ----------------------------------------------
// dst[s][r][c], r < 3*hl*dh: rows of Wq/Wk/Wv belonging to shard s's heads.
cudaError_t pack_qkv(int esize, const void* Wq, const void* Wk, const void* Wv, void* dst, int tp, int hl,
                     int dh, int d, cudaStream_t st);
// dst[s][n][k] = src[n][s*ks + k]   (src is [N][tp*ks])
cudaError_t pack_cols(int esize, const void* src, void* dst, int tp, int N, int ks, cudaStream_t st);
// SwiGLU: dst[s][r][c] with `granule`-row blocks alternating gate/up of shard s.
// GELU (Wu == nullptr): dst[s][r][c] = W1[s*fl + r][c].
cudaError_t pack_up(int esize, const void* Wg, const void* Wu, void* dst, int tp, int fl, int d, int granule,
                    cudaStream_t st);

// ---- SIMT path (simt.cu): fp32 plans, and shapes the tensor-core path does not take
enum SimtEpi { EPI_STORE = 0, EPI_GELU = 1, EPI_SWIGLU = 2, EPI_ROW_REDUCE = 3 };

struct SimtGemm {
    int epi;
    int is_bf16;
    const void* A;        // [.., M, lda]
    long long a_shard;    // elements between shards of A (0: shared input)
    int lda;
    const void* W;        // [.., N, ldw]
    long long w_shard;
    int ldw;
    int M, N, K;          // N = W rows per shard, K = reduction length per shard
    int col_shards;       // grid.z: shards computed side by side (column)
    int red_shards;       // shards summed into one output (row reduce)
    void* out;            // column: act [cs][M][ldo]; row: fp32 [M][ldo]
    long long out_shard;
    int ldo;
    void* out2;           // row: optional act copy
    const void* residual; // row: optional
    int residual_f32;
    int granule;          // SwiGLU: gate/up interleave block (rows)
};
cudaError_t simt_gemm(const SimtGemm& g, cudaStream_t st);

struct AttnArgs {
    int is_bf16;
    const void* qkv;      // [tp][B*Tq][3*hl*dh]
    const void* kc;       // cache [B][H][cap][dh] or nullptr
    const void* vc;
    void* out;            // [tp][B*Tq][hl*dh]
    int B, Tq, H, hl, dh, cap, pos, causal;
    float scale;
};
// K/V of the new tokens -> cache positions pos..pos+Tq-1
cudaError_t kv_append(const AttnArgs& a, void* kc, void* vc, cudaStream_t st);
cudaError_t simt_attention(const AttnArgs& a, cudaStream_t st);

// ---- tensor-core GEMM (gemm_tc.cu): bf16 in, fp32 accumulate in TMEM -------
struct TcGemm {
    int epi;              // EPI_STORE / EPI_GELU / EPI_SWIGLU / EPI_ROW_REDUCE
    const void* A;        // bf16 [shards?][M][lda]
    long long a_shard;    // elements between A shards (0 for column-parallel)
    int lda;
    const void* W;        // bf16 [shards][N][K]
    long long w_shard;
    int M, N, K;          // per shard: N = W rows, K = reduction length
    int shards;
    int reduce;           // 1: sum all shards into one output (row-parallel)
    void* out;
    long long out_shard;
    int ldo;
    int granule;
    void* out2;
    const void* residual;
    int residual_f32;
    // pre-norm variant (column-parallel launches only): the accumulator row
    // m is scaled by row_scale[m] (1/rms of input row m; the norm's gain is
    // folded into W), and for rope_cols > 0 the first rope_cols columns of
    // every shard (its Q and K heads) get rotary position embedding: pair
    // (2i, 2i+1) of a head of width rope_dh in row m rotated by the angle
    // whose (cos, sin) is rope_cs[(m % rope_seq) * rope_dh / 2 + i]
    const float* row_scale;
    int rope_cols, rope_dh, rope_seq;
    const float2* rope_cs;
    // sequence-parallel layouts (slice_rows > 0, a multiple of 8): row m of
    // the token rows lives in slice m / slice_rows at row m % slice_rows;
    // the slices of a column-parallel input A are a_slice elements apart,
    // those of a row-parallel launch's out / out2 out_slice and of its
    // residual res_slice apart (all multiples of 8)
    int slice_rows;
    long long a_slice, out_slice, res_slice;
};
bool tc_gemm_supported(int M, int N, int K);
// scratch (nullable): the split tiles' counters and fp32 partial sums; at
// most tc_gemm_scratch_bytes() is touched.  Without scratch every launch
// runs whole tiles only.  A launch that splits tiles clears the counters
// first (a few KB, on `st`) unless *counters_zero says they are known to
// be zero; it then sets *counters_zero, because a launch that completes
// leaves them zero (a chain of launches on one scratch clears once).
size_t tc_gemm_scratch_bytes();
cudaError_t tc_gemm(const TcGemm& g, int* dev_err, void* scratch, size_t scratch_bytes, cudaStream_t st,
                    bool* counters_zero = nullptr);
// Host-only description of a tc_gemm launch on a GPU with `sms` SMs of which
// `pair_slots` SM pairs can be co-resident (0: no paired launches).
struct TcSchedule {
    int paired;            // 2-SM tiles (256 rows) or single-SM tiles (128 rows)
    int tiles, kbt;        // output tiles, k-blocks per tile
    int whole, parts;      // tiles run whole; parts per remaining (split) tile
    int items, units;      // work items (split parts first, then whole tiles), units (SM pairs or SMs)
    size_t scratch_touched;  // bytes of scratch the launch reads or writes
};
TcSchedule tc_gemm_schedule(const TcGemm& g, size_t scratch_bytes, int sms, int pair_slots);
// Limit of every bounded wait in the tensor-core kernels (ns).
unsigned long long wait_timeout_ns();

// ---- small-M weight streaming (gemv.cu): same arguments as the GEMM ---------
typedef TcGemm GemvArgs;
constexpr int GEMV_MAX_M = 8;
// Token rows the tensor-core weight stream (gemv_mma) takes at most; the
// dispatch prefers it to the tensor-core GEMM over the whole range (7B
// decode step, tp 2, one B300: 142 vs 175 us at 9 rows, 163 vs 197 at 16,
// 242 vs 265 at 32 -- the weight bytes are read once either way, and the
// 128-row GEMM tiles are mostly empty).
constexpr int GEMV_MMA_MAX_ROWS = 32;
constexpr int GEMV_MMA_DISPATCH_ROWS = GEMV_MMA_MAX_ROWS;
// Dispatch for 2..GEMV_MMA_DISPATCH_ROWS rows: gemv_mma where it applies;
// else this CUDA-core loop up to this many rows and the tensor-core GEMM
// (split tiles) above it -- at 8 rows the loop is bound by its conversions
// and FMAs (7B decode step, one B300: 285 us at 8 rows vs 150 us on the
// tensor-core GEMM).
constexpr int GEMV_PREFERRED_MAX_M = 4;
bool gemv_supported(const GemvArgs& g);
cudaError_t gemv(const GemvArgs& g, int* dev_err, cudaStream_t st);
// 2..GEMV_MMA_MAX_ROWS rows with the products on the tensor cores
// (gemv_mma.cu): K a multiple of 32, N a multiple of 16, SwiGLU granule a
// multiple of 16, row-parallel launches with at most 8 shards.
bool gemv_mma_supported(const GemvArgs& g);
cudaError_t gemv_mma(const GemvArgs& g, cudaStream_t st);

// ---- pre-norm helpers (norm.cu) ----------------------------------------------
// W[r][c] *= gamma[c] for rows x d (plan dtype, rounded back to it).
cudaError_t scale_cols(int esize, void* W, long long rows, int d, const void* gamma, cudaStream_t st);
// Rotary table: cs[t * half + i] = (cos, sin) of (pos0 + t) * 2^(-(2i / (2 half)) * log2_theta)
// for t < seq, i < half (half = d_head / 2).
struct RopeTable {
    float2* cs;
    int seq, pos0, half;
    float log2_theta;
};
// r[m] = 1 / sqrt(mean_c x[m][c]^2 + eps), x bf16 (x_f32 = 0) or fp32,
// d a multiple of 8 and rows 16-byte aligned; the same launch fills
// rope->cs when rope is non-null.  slice_rows > 0: row m of x lives in
// slice m / slice_rows, slices slice_stride elements apart.
cudaError_t rms_rows(const void* x, int x_f32, int M, int d, float eps, float* r, const RopeTable* rope,
                     cudaStream_t st, int slice_rows = 0, long long slice_stride = 0);

// ---- tensor-core attention (attn_tc.cu) --------------------------------------
bool tc_attention_supported(const AttnArgs& a);
// dev_err: device word where bounded waits record a timeout
cudaError_t tc_attention(const AttnArgs& a, int* dev_err, cudaStream_t st);

// ---- single-token decode (decode.cu) ------------------------------------------
// Split-KV attention: partial (max, sum, output) per key chunk in `scratch`
// ([B][H][DECODE_MAX_SPLITS][dh + 2] floats), then a combine pass.  Also
// writes the new token's K/V (from the QKV buffer) into the cache at pos.
constexpr int DECODE_MAX_SPLITS = 64;
cudaError_t decode_attention(const AttnArgs& a, float* scratch, cudaStream_t st);

}  // namespace tpk
