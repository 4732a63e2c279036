// Tensor-core GEMM for the column- and row-parallel linears (bf16 in, fp32
// accumulate), written for sm_103a with tcgen05 + TMEM + TMA.
//
//   column-parallel (undercodenews.com/?p=110319, "the Original": each shard
//   multiplies the full input by its slice of the output features):
//       out[s][m][n] = epi( sum_k A[m][k] * W[s][n][k] ),  all shards in one
//       launch (a grouped GEMM whose groups share A);
//   row-parallel with the all-reduce fused in (same section: matching column
//   blocks of the input and row blocks of the weight, partials summed):
//       out[m][n] = residual[m][n] + sum_s sum_k A[s][m][k] * W[s][n][k]
//       -- every shard's partial product is accumulated, in shard order, into
//       the same TMEM accumulator.
//
// Two variants of one persistent kernel (one CTA per SM, 320 threads):
//  * PAIR (M > 128): clusters of two CTAs on neighbouring SMs compute a
//    256 x 256 output tile with 2-SM MMAs (tcgen05 .cta_group::2, M = 256):
//    each CTA stages its own 128 rows of A and 128 of the 256 rows of W, the
//    even CTA issues the MMAs, and each CTA's TMEM holds its 128 output rows.
//    32 KB per k-block per SM, 6-stage ring.
//  * single (M <= 128): 128 x 256 tiles on one SM, 48 KB stages, 4 deep.
// Roles in each CTA:
//   warp 0   TMA producer (128-byte swizzle, ring of k-blocks of 64);
//   warp 1   TMEM allocator; in the issuing CTA also the MMA thread:
//            tcgen05.mma kind::f16, K = 16 steps, into one of two 256-column
//            fp32 TMEM accumulators;
//   warps 2-9 epilogue: tcgen05.ld of the finished accumulator (warp w its
//            32-lane quarter w % 4 and one 128-column half), through a
//            per-warp XOR-swizzled shared staging block so that global
//            stores are row-contiguous, activation / residual.
// The epilogue of item i overlaps the main loop of item i+1 (two TMEM
// accumulators = all 512 columns).
//
// Work decomposition: when the output tiles do not fill every unit (SM pair
// or SM) in the last round, the tiles that fill whole rounds run whole and
// each remaining tile is cut into `parts` equal k-ranges on different
// units; the parts run first, the whole tiles after them.  A part writes its raw fp32 sums to the caller's scratch, counts
// itself in (per tile, CTA and warp quarter), waits (bounded) for the
// tile's other parts, and then reduces its own share of the tile's rows
// over all parts, in part order, and runs the epilogue on them -- the
// split reduction happens inside this launch, spread over the parts.  The
// counters go back to zero when the last part leaves.
//
// Every wait is bounded: after `timeout_ns` the waiting role records
// TP_ERR_DEVICE_TIMEOUT's device code, raises a CTA-wide abort flag and
// leaves its loop; in-flight tensor-core work is drained and TMEM freed
// before the CTA exits, and the two CTAs of a pair leave together.
#include <atomic>
#include <cuda.h>

#include "common.cuh"
#include "kernels.h"
#include "tc_ptx.cuh"

namespace tpk {

namespace {

#ifndef TP_GEMM_PAIR_STAGES
#define TP_GEMM_PAIR_STAGES 6  // shared-memory ring depth of the paired kernel
#endif

constexpr int BN = 256, BK = 64;          // output columns per tile, K per stage
constexpr int A_ROWS = 128;                // A rows staged per CTA
constexpr int TMEM_COLS = 512;
constexpr int EPI_WARPS = 8;               // two per TMEM lane quarter, one per 128-column half
constexpr int NUM_THREADS = 64 + 32 * EPI_WARPS;
constexpr int HALF_N = BN / 2;             // columns per epilogue warp
constexpr int STG_FLOATS = 32 * 32;        // one epilogue warp's 32 x 32 staging block
constexpr int STG_BYTES = EPI_WARPS * STG_FLOATS * 4;
constexpr int PART_FLOATS = 32 * HALF_N;   // one warp's 32 rows x 128 columns of a split partial
constexpr int SPLIT_ROUNDS_MAX = 4;        // split parts per unit at most
constexpr int FIX_BYTES = 24 * 1024;       // each epilogue warp's share of the idle ring at the end of the work

template <bool PAIR>
struct GCfg;
template <bool PAIR>
struct GCfg {
    static constexpr int TILE_M = PAIR ? 256 : 128;   // output rows per tile
    static constexpr int W_ROWS = PAIR ? BN / 2 : BN;  // W rows staged per CTA
    static constexpr int A_BYTES = A_ROWS * BK * 2;
    static constexpr int STAGE_BYTES = A_BYTES + W_ROWS * BK * 2;
    static constexpr int STAGES = PAIR ? TP_GEMM_PAIR_STAGES : 4;
    static constexpr int GROUP_M = PAIR ? 8 : 16;       // row blocks per raster band (2048 rows)
    static constexpr int RANKS = PAIR ? 2 : 1;
    static constexpr int SMEM = STAGES * STAGE_BYTES + STG_BYTES + 1024 + 256;
    // instruction descriptor: D fp32, A/B bf16, both K-major
    static constexpr uint32_t IDESC = ptx::idesc_bf16(TILE_M, BN, false);
    static_assert(STAGES * STAGE_BYTES >= EPI_WARPS * FIX_BYTES, "the epilogue warps' end-of-work buffers live in the ring");
};

struct Params {
    int epi, M, N, K, shards, reduce;
    int m_blocks, n_blocks, n_tiles, k_blocks;  // n_blocks per shard (column) or total (row)
    void* out;
    long long out_shard;
    int ldo;
    void* out2;
    const void* residual;
    int residual_f32;
    int granule;
    int* err;
    unsigned long long timeout_ns;
    // Work items: with S = n_items - dp_items split items, item i < S is
    // part i % parts (k-blocks [kbt*j/parts, kbt*(j+1)/parts)) of tile
    // dp_items + i / parts, and item S + t is the whole tile t < dp_items;
    // unit u takes items u, u + units, ...  The parts come first, so the
    // whole tiles' main loops follow them without a break.  Every part
    // writes its fp32 sums to `partials` ([item][rank][warp][32][128]) and
    // counts itself in (`flags`: [split tile][rank][warp] x {arrived,
    // left}: zero at the start of the launch, and the last part out of a
    // block returns them to zero); at the end of the unit's work -- when this SM no longer
    // streams operands, so its loads are fast -- each part reduces its own
    // rows of the tile over all parts, in part order, and applies the
    // epilogue.
    int dp_items, n_items, parts;
    float* partials;
    int* flags;
    // pre-norm variant: see TcGemm
    const float* row_scale;
    int rope_cols, rope_dh, rope_seq;
    const float2* rope_cs;
    // sequence-parallel layouts (see TcGemm): rows per slice (0: none), the
    // row-parallel outputs' and residual's distance between slices, and the
    // A rows staged per TMA box of a gathered column-parallel input
    int slice_rows;
    long long out_slice, res_slice;
    int a_box;
};

// Layout instantiations of the kernel (SL): 0 plain; 1 sequence-parallel
// slices of any multiple of 8 rows; 2 slices of a multiple of 128 rows (an
// A box and an epilogue warp's 32-row block never cross a slice).
//
// Element offset of row `row` (column 0) of a row-parallel output / of the
// residual: plain [M][ldo] (SL 0), or slice row / slice_rows at `slice`
// elements per slice.
template <int SL>
__device__ __forceinline__ long long out_row(const Params& p, int row) {
    if (!SL) return (long long)row * p.ldo;
    return (long long)(row / p.slice_rows) * p.out_slice + (long long)(row % p.slice_rows) * p.ldo;
}
template <int SL>
__device__ __forceinline__ long long res_row(const Params& p, int row) {
    if (!SL) return (long long)row * p.ldo;
    return (long long)(row / p.slice_rows) * p.res_slice + (long long)(row % p.slice_rows) * p.ldo;
}

// Row offsets of an epilogue warp's 32-row block (rows row_base .. +31,
// row_base a multiple of 32): when no slice boundary can fall inside the
// block (plain layout, or slices of a multiple of 32 rows) the offsets are
// the block's first row's plus r * ldo; otherwise each row is mapped.
template <int SL>
struct RowMap {
    long long out0, res0;
    int row_base;
    bool fast;
    __device__ __forceinline__ RowMap(const Params& p, int rb) {
        row_base = rb;
        fast = p.slice_rows % 32 == 0;
        out0 = out_row<SL>(p, rb);
        res0 = res_row<SL>(p, rb);
    }
    __device__ __forceinline__ long long out(const Params& p, int r) const {
        return fast ? out0 + (long long)r * p.ldo : out_row<SL>(p, row_base + r);
    }
    __device__ __forceinline__ long long res(const Params& p, int r) const {
        return fast ? res0 + (long long)r * p.ldo : res_row<SL>(p, row_base + r);
    }
};
// plain layout: row r of the block is row row_base + r of [M][ldo]
template <>
struct RowMap<0> {
    int row_base;
    __device__ __forceinline__ RowMap(const Params&, int rb) : row_base(rb) {}
    __device__ __forceinline__ long long out(const Params& p, int r) const { return (long long)(row_base + r) * p.ldo; }
    __device__ __forceinline__ long long res(const Params& p, int r) const { return (long long)(row_base + r) * p.ldo; }
};
// slices of a multiple of 128 rows: the block lies in one slice
template <>
struct RowMap<2> {
    int slice, srow;  // the block's slice and its first row in it
    __device__ __forceinline__ RowMap(const Params& p, int rb) : slice(rb / p.slice_rows), srow(rb % p.slice_rows) {}
    __device__ __forceinline__ long long out(const Params& p, int r) const {
        return (long long)slice * p.out_slice + (long long)(srow + r) * p.ldo;
    }
    __device__ __forceinline__ long long res(const Params& p, int r) const {
        return (long long)slice * p.res_slice + (long long)(srow + r) * p.ldo;
    }
};

// Four consecutive finished row-parallel outputs at element offset o of
// the output rows (residual already added): fp32 out + optional plan-dtype
// copy.
__device__ __forceinline__ void store_row4(const Params& p, long long o, float4 t);

// Rotary position embedding of N consecutive values of one row starting at
// column `col` of a shard (col a multiple of N, N a multiple of 4): pairs
// (2i, 2i+1) of each head of width p.rope_dh rotated by the table's angle
// for the row's position; only columns below p.rope_cols (the shard's Q and
// K heads; a multiple of 8) are rotated.  d_head is a multiple of 8, so 4
// columns never straddle two heads or the Q/K-V boundary, and each float4
// of the table holds their two pairs.
template <int N>
__device__ __forceinline__ void apply_rope(const Params& p, int row, int col, float (&v)[N]) {
    if (col >= p.rope_cols) return;
    const int half = p.rope_dh / 2;
    const float2* tr = p.rope_cs + (long long)(row % p.rope_seq) * half;
    int hc = col % p.rope_dh;  // column within the head, advanced 4 at a time
#pragma unroll
    for (int q = 0; q < N / 4; ++q) {
        if (col + 4 * q >= p.rope_cols) break;
        const float4 c = *reinterpret_cast<const float4*>(tr + hc / 2);
        const float a0 = v[4 * q], b0 = v[4 * q + 1], a1 = v[4 * q + 2], b1 = v[4 * q + 3];
        v[4 * q] = a0 * c.x - b0 * c.y;
        v[4 * q + 1] = a0 * c.y + b0 * c.x;
        v[4 * q + 2] = a1 * c.z - b1 * c.w;
        v[4 * q + 3] = a1 * c.w + b1 * c.z;
        hc += 4;
        if (hc >= p.rope_dh) hc -= p.rope_dh;
    }
}

using namespace ptx;

// Output tile t -> (row block, shard, column block).  Tiles run in bands of
// `group_m` row blocks: inside a band the row block varies fastest, then the
// column block (shard-major for column-parallel launches), so the tiles in
// flight at once cover a compact rectangle and both the activation rows and
// the weight rows they share stay in L2 even when M is large.
__device__ __forceinline__ void tile_coords(const Params& p, int t, int group_m, int& m_blk, int& shard, int& n_blk) {
    const int nb = p.reduce ? p.n_blocks : p.n_blocks * p.shards;  // column tiles across shards
    const int per_group = group_m * nb;
    const int first_m = (t / per_group) * group_m;
    const int gm = min(p.m_blocks - first_m, group_m);
    const int r = t % per_group;
    m_blk = first_m + r % gm;
    const int nn = r / gm;
    shard = p.reduce ? 0 : nn / p.n_blocks;
    n_blk = p.reduce ? nn : nn % p.n_blocks;
}

// One piece of a unit's work: a tile and its k-block range; for a part of
// a split tile (sk >= 0) its part index and split-item index.
struct Item {
    int tile, k0, k1, part, sk;
};

// The work of one unit, in order (the producer, the MMA issuer and the
// epilogue warps each walk it with their own copy).
struct Work {
    int w, n_units, kbt;
    __device__ void init(int unit, int n_units_, int kbt_) {
        w = unit;
        n_units = n_units_;
        kbt = kbt_;
    }
    __device__ bool next(const Params& p, Item& it) {
        if (w >= p.n_items) return false;
        const int n_split = p.n_items - p.dp_items;
        if (w >= n_split) {
            it.tile = w - n_split;
            it.k0 = 0;
            it.k1 = kbt;
            it.part = 0;
            it.sk = -1;
        } else {
            it.sk = w;
            it.part = w % p.parts;
            it.tile = p.dp_items + w / p.parts;
            it.k0 = (int)((long long)kbt * it.part / p.parts);
            it.k1 = (int)((long long)kbt * (it.part + 1) / p.parts);
        }
        w += n_units;
        return true;
    }
};

__device__ __forceinline__ uint64_t sw128_kmajor(uint32_t saddr) { return sw128_desc(saddr, 16, 1024); }

// ---- epilogue helpers ------------------------------------------------------
// The accumulator comes out of TMEM one row per lane (32 consecutive columns
// per lane); a 32 x 32 block goes through this warp's shared staging block
// so that every global access of the warp covers 4 rows x 128 contiguous
// bytes instead of 32 scattered rows.

// The block is 32 rows of 128 bytes with the 16-byte chunk j of row r
// stored at position j ^ (r % 8), so that both the row-per-lane writes and
// the 4-rows-per-instruction reads hit 8 distinct chunk positions per phase.
__device__ __forceinline__ void stage_put(float* stg, int lane, const float (&v)[32]) {
    float* row = stg + lane * 32;
#pragma unroll
    for (int q = 0; q < 8; ++q)
        *reinterpret_cast<float4*>(row + 4 * (q ^ (lane & 7))) =
            make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
}
// Row 4i + lane / 8, columns 4 (lane % 8) .. + 3 of the staged block.
__device__ __forceinline__ float4 stage_get(const float* stg, int lane, int i) {
    const int r = 4 * i + (lane >> 3);
    return *reinterpret_cast<const float4*>(stg + r * 32 + 4 * ((lane & 7) ^ (r & 7)));
}

// 16-byte asynchronous copy global -> shared (cached in L2 only); many can
// be in flight per thread without holding registers.
__device__ __forceinline__ void cp_async16(uint32_t saddr, const void* g) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(saddr), "l"(g) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}

// Pull `bytes` (a multiple of 16, 16-byte aligned) into L2 ahead of use.
__device__ __forceinline__ void prefetch_l2(const void* ptr, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(ptr), "r"(bytes) : "memory");
}

__device__ __forceinline__ uint2 pack_bf16x4(float4 t) { return make_uint2(pack_bf16x2(t.x, t.y), pack_bf16x2(t.z, t.w)); }

__device__ __forceinline__ float4 add4(float4 a, float4 b) { return make_float4(a.x + b.x, a.y + b.y, a.z + b.z, a.w + b.w); }

__device__ __forceinline__ void store_row4(const Params& p, long long o, float4 t) {
    *reinterpret_cast<float4*>((float*)p.out + o) = t;
    if (p.out2) *reinterpret_cast<uint2*>((bf16*)p.out2 + o) = pack_bf16x4(t);
}

// Four consecutive finished column-parallel outputs (row, col .. col+3) of
// a shard, activation already applied: a bf16 store.
__device__ __forceinline__ void store4(const Params& p, int shard, int row, int col, float4 t) {
    *reinterpret_cast<uint2*>((bf16*)p.out + shard * p.out_shard + (long long)row * p.ldo + col) = pack_bf16x4(t);
}

// Column-parallel per-element epilogue of N consecutive columns of one row
// (col a multiple of N): row scale, rotary embedding, GELU.
template <int N>
__device__ __forceinline__ void col_epilogue(const Params& p, int row, int col, float (&v)[N]) {
    if (p.row_scale) {
        const float rs = row < p.M ? p.row_scale[row] : 0.f;
#pragma unroll
        for (int j = 0; j < N; ++j) v[j] *= rs;
    }
    if (p.rope_cols > 0) apply_rope<N>(p, row, col, v);
    if (p.epi == EPI_GELU) {
#pragma unroll
        for (int j = 0; j < N; ++j) v[j] = gelu_erf(v[j]);
    }
}

// The residual rows [r0, r1) of this warp's 32, columns col0 .. col0+127,
// pulled into L2 ahead of the epilogue that adds them (one row per lane).
template <int SL>
__device__ __forceinline__ void prefetch_residual(const Params& p, int lane, int row_base, int r0, int r1, int col0) {
    if (p.epi != EPI_ROW_REDUCE || p.residual == nullptr || col0 >= p.N) return;
    const int r = r0 + lane, grow = row_base + r;
    if (r >= r1 || grow >= p.M) return;
    const int es = p.residual_f32 ? 4 : 2;
    const int ncols = min(HALF_N, p.N - col0);  // a multiple of 8
    prefetch_l2((const char*)p.residual + (res_row<SL>(p, grow) + col0) * es, (uint32_t)(ncols * es));
}

// Whole tile of a column-parallel launch: this warp's 32 rows x 128
// columns (col0 = first column of the warp's half) from TMEM (tbase = the
// half's first column) through the staging block; the per-element epilogue
// runs after the transpose, 4 columns of one row per lane.
__device__ __forceinline__ void epilogue_col(const Params& p, uint32_t tbase, float* stg, int lane, int row_base,
                                             int shard, int col0) {
    if (p.epi == EPI_SWIGLU) {
#pragma unroll 1
        for (int g = 0; g < HALF_N / 64; ++g) {
            float gate[32], up[32];
            __syncwarp();
            tmem_ld32(tbase + 64 * g, gate);
            tmem_ld32(tbase + 64 * g + 32, up);
            const int pc = col0 + 64 * g;  // packed column of this gate block
            if (pc >= p.N) break;
            float4 gv[8];
            stage_put(stg, lane, gate);
            __syncwarp();
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                gv[i] = stage_get(stg, lane, i);
            }
            __syncwarp();
            stage_put(stg, lane, up);
            __syncwarp();
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int grow = row_base + 4 * i + (lane >> 3);
                const float4 u = stage_get(stg, lane, i);
                const float rs = p.row_scale ? (grow < p.M ? p.row_scale[grow] : 0.f) : 1.f;
                const float4 o = make_float4(silu(gv[i].x * rs) * (u.x * rs), silu(gv[i].y * rs) * (u.y * rs),
                                             silu(gv[i].z * rs) * (u.z * rs), silu(gv[i].w * rs) * (u.w * rs));
                if (grow < p.M)
                    *reinterpret_cast<uint2*>((bf16*)p.out + shard * p.out_shard + (long long)grow * p.ldo + pc / 2 +
                                              4 * (lane & 7)) = pack_bf16x4(o);
            }
            __syncwarp();
        }
        return;
    }
#pragma unroll 1
    for (int c = 0; c < HALF_N / 32; ++c) {
        float v[32];
        __syncwarp();
        tmem_ld32(tbase + 32 * c, v);
        const int cc = col0 + 32 * c;
        if (cc >= p.N) break;  // (warp-uniform; later chunks are further right)
        stage_put(stg, lane, v);
        __syncwarp();
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int grow = row_base + 4 * i + (lane >> 3), gcol = cc + 4 * (lane & 7);
            const float4 t = stage_get(stg, lane, i);
            float e[4] = {t.x, t.y, t.z, t.w};
            col_epilogue<4>(p, grow, gcol, e);
            if (grow < p.M && gcol < p.N) store4(p, shard, grow, gcol, make_float4(e[0], e[1], e[2], e[3]));
        }
    }
}

__device__ __forceinline__ float4 bf16x4_to_float4(uint2 r) {
    const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&r.x));
    const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&r.y));
    return make_float4(a.x, a.y, b.x, b.y);
}

// Whole tile of a row-parallel launch: this warp's 32 rows x 128 columns
// plus the residual (RES 0: none, 1: bf16, 2: fp32).  Global loads take
// about a microsecond while the tensor cores stream operands, so the
// residual of chunk c + 1 is loaded while chunk c is stored (and the rows
// were pulled into L2 while the MMAs ran).
template <int RES, int SL>
__device__ __forceinline__ void epilogue_row(const Params& p, uint32_t tbase, float* stg, int lane, int row_base,
                                             int col0, float* rbuf) {
    constexpr int NC = HALF_N / 32;
    constexpr int L = 1;
    const RowMap<SL> rm(p, row_base);
    if (RES != 0 && rbuf != nullptr) {
        // the unit's last tile: the ring is idle, so the whole residual
        // block (32 rows x 128 columns, 512-byte rows) is copied into this
        // warp's share of it at once
        constexpr int ES = RES == 2 ? 4 : 2;
        const uint32_t sb = smem_u32(rbuf);
        const int gcol = col0 + lane * 16 / ES;
        if (lane < HALF_N * ES / 16 && gcol < p.N) {
#pragma unroll 4
            for (int r = 0; r < 32; ++r) {
                const int grow = row_base + r;
                if (grow < p.M) cp_async16(sb + r * 512 + lane * 16, (const char*)p.residual + (rm.res(p, r) + gcol) * ES);
            }
        }
        cp_async_wait_all();
        __syncwarp();
#pragma unroll 1
        for (int c = 0; c < NC; ++c) {
            float v[32];
            __syncwarp();
            tmem_ld32(tbase + 32 * c, v);
            const int cc = col0 + 32 * c;
            if (cc >= p.N) break;
            stage_put(stg, lane, v);
            __syncwarp();
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int rr = 4 * i + (lane >> 3), lc = 32 * c + 4 * (lane & 7);
                const int grow = row_base + rr, gcol = cc + 4 * (lane & 7);
                float4 t = stage_get(stg, lane, i);
                if (RES == 2) t = add4(t, *reinterpret_cast<const float4*>(rbuf + rr * HALF_N + lc));
                if (RES == 1) t = add4(t, bf16x4_to_float4(*reinterpret_cast<const uint2*>(
                                              reinterpret_cast<const char*>(rbuf) + rr * 512 + lc * 2)));
                if (grow < p.M && gcol < p.N) store_row4(p, rm.out(p, rr) + gcol, t);
            }
        }
        return;
    }
    // one residual slot: 4 values of row 4i + lane / 8, columns c0 + 4 (lane % 8) .. + 3, as raw words
    auto fetch = [=](int c0, int i) -> float4 {
        const int grow = row_base + 4 * i + (lane >> 3), gcol = c0 + 4 * (lane & 7);
        const bool ok = grow < p.M && gcol < p.N;
        const long long o = rm.res(p, 4 * i + (lane >> 3)) + gcol;
        if (RES == 1) {
            const uint2 r = ok ? *reinterpret_cast<const uint2*>((const bf16*)p.residual + o) : make_uint2(0u, 0u);
            return make_float4(__uint_as_float(r.x), __uint_as_float(r.y), 0.f, 0.f);
        }
        return ok ? *reinterpret_cast<const float4*>((const float*)p.residual + o) : make_float4(0.f, 0.f, 0.f, 0.f);
    };
    float4 rs[L][8];
    if (RES != 0) {
#pragma unroll
        for (int c = 0; c < L; ++c)
#pragma unroll
            for (int i = 0; i < 8; ++i) rs[c][i] = fetch(col0 + 32 * c, i);
    }
#pragma unroll
    for (int c = 0; c < NC; ++c) {
        float v[32];
        __syncwarp();
        tmem_ld32(tbase + 32 * c, v);
        const int cc = col0 + 32 * c;
        if (cc >= p.N) break;  // (warp-uniform; later chunks are further right)
        stage_put(stg, lane, v);
        __syncwarp();
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int grow = row_base + 4 * i + (lane >> 3), gcol = cc + 4 * (lane & 7);
            float4 t = stage_get(stg, lane, i);
            if (RES == 1)
                t = add4(t, bf16x4_to_float4(make_uint2(__float_as_uint(rs[c % L][i].x), __float_as_uint(rs[c % L][i].y))));
            if (RES == 2) t = add4(t, rs[c % L][i]);
            if (RES != 0 && c + L < NC) rs[c % L][i] = fetch(cc + 32 * L, i);  // this slot's next use
            if (grow < p.M && gcol < p.N) store_row4(p, rm.out(p, 4 * i + (lane >> 3)) + gcol, t);
        }
    }
}

// Part of a split tile: this warp's 32 rows x 128 columns of raw fp32 sums
// to its partial block (row-major, 512-byte rows, coalesced).
__device__ __forceinline__ void write_partial(uint32_t tbase, float* stg, int lane, float* part, int nrows) {
    if (nrows <= 0) return;  // every row of this warp's block is past M
#pragma unroll 1
    for (int c = 0; c < HALF_N / 32; ++c) {
        float v[32];
        __syncwarp();
        tmem_ld32(tbase + 32 * c, v);
        stage_put(stg, lane, v);
        __syncwarp();
#pragma unroll
        for (int i = 0; i < 8; ++i)
            if (4 * i + (lane >> 3) < nrows)  // rows past M are never read back
                __stcg(reinterpret_cast<float4*>(part + (4 * i + (lane >> 3)) * HALF_N + 32 * c + 4 * (lane & 7)),
                       stage_get(stg, lane, i));
    }
}

// Bounded wait (one thread) until *cnt reaches `target`.
__device__ __noinline__ bool wait_count(const int* cnt, int target, volatile int* abort_flag, int* err,
                                        unsigned long long timeout_ns) {
    const unsigned long long t0 = globaltimer();
    for (;;) {
        int v;
        asm volatile("ld.acquire.gpu.s32 %0, [%1];" : "=r"(v) : "l"(cnt) : "memory");
        if (v >= target) return true;
        if (*abort_flag) return false;
        if (globaltimer() - t0 > timeout_ns) {
            *abort_flag = 1;
            record_error(err, DEV_ERR_TIMEOUT);
            return false;
        }
        __nanosleep(64);
    }
}

// The rows [r0, r1) of this warp's 32 that this part owns, columns col0 ..
// col0+127: the sum of all parts' partials (part order 0..parts-1), then the
// epilogue.  `base` is part 0's block for this warp, `pstride` the distance
// between parts, `buf` this warp's share of the idle ring: every part's
// rows and the residual rows are copied into it at once (one memory
// latency for the whole reduction), then summed from shared memory.
template <int SL>
__device__ __forceinline__ void reduce_rows(const Params& p, const float* base, long long pstride, int lane,
                                            int row_base, int r0, int r1, int shard, int col0, float* buf) {
    const int nr = r1 - r0;  // (parts + 1) * nr <= 48 rows of 512 bytes fit FIX_BYTES
    const RowMap<SL> rm(p, row_base);
    const bool has_res = p.epi == EPI_ROW_REDUCE && p.residual != nullptr;
    const int es = p.residual_f32 ? 4 : 2;
    const uint32_t sb = smem_u32(buf);
    const int res_off = p.parts * nr * HALF_N;  // floats: residual rows after the parts' rows
    for (int i = 0; i < p.parts; ++i)
        for (int j = 0; j < nr; ++j)
            cp_async16(sb + ((i * nr + j) * HALF_N + 4 * lane) * 4, base + i * pstride + (long long)(r0 + j) * HALF_N + 4 * lane);
    if (has_res) {
        const int gcol = col0 + lane * 16 / es;
        if (lane < HALF_N * es / 16 && gcol < p.N)
            for (int j = 0; j < nr; ++j) {
                const int grow = row_base + r0 + j;
                if (grow < p.M)
                    cp_async16(sb + res_off * 4 + j * 512 + lane * 16,
                               (const char*)p.residual + (rm.res(p, r0 + j) + gcol) * es);
            }
    }
    cp_async_wait_all();
    __syncwarp();
    if (p.epi == EPI_SWIGLU) {
        // lane -> row j + lane / 16, gate columns 64 b + 4 (lane % 8) .. + 3 of the half (b = lane / 8 % 2)
        // and the matching up columns 32 further
        const int b = (lane >> 3) & 1;
        const int gl = 64 * b + 4 * (lane & 7);
        if (col0 + 64 * b >= p.N) return;
        for (int j = lane >> 4; j < nr; j += 2) {
            const int grow = row_base + r0 + j;
            if (grow >= p.M) break;
            float4 g = make_float4(0.f, 0.f, 0.f, 0.f), u = g;
            for (int i = 0; i < p.parts; ++i) {
                const float* q = buf + (i * nr + j) * HALF_N + gl;
                g = add4(g, *reinterpret_cast<const float4*>(q));
                u = add4(u, *reinterpret_cast<const float4*>(q + 32));
            }
            const float rs = p.row_scale ? p.row_scale[grow] : 1.f;
            const float4 o = make_float4(silu(g.x * rs) * (u.x * rs), silu(g.y * rs) * (u.y * rs),
                                         silu(g.z * rs) * (u.z * rs), silu(g.w * rs) * (u.w * rs));
            *reinterpret_cast<uint2*>((bf16*)p.out + shard * p.out_shard + (long long)grow * p.ldo +
                                      (col0 + 64 * b) / 2 + 4 * (lane & 7)) = pack_bf16x4(o);
        }
        return;
    }
    // lane -> columns 4 lane .. 4 lane + 3 of every row
    const int gcol = col0 + 4 * lane;
    if (gcol >= p.N) return;
    for (int j = 0; j < nr; ++j) {
        const int grow = row_base + r0 + j;
        if (grow >= p.M) break;
        float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int i = 0; i < p.parts; ++i) a = add4(a, *reinterpret_cast<const float4*>(buf + (i * nr + j) * HALF_N + 4 * lane));
        if (p.epi == EPI_ROW_REDUCE) {
            if (has_res) {
                const char* rrow = reinterpret_cast<const char*>(buf + res_off) + j * 512;
                a = add4(a, es == 4 ? *reinterpret_cast<const float4*>(rrow + 16 * lane)
                                    : bf16x4_to_float4(*reinterpret_cast<const uint2*>(rrow + 8 * lane)));
            }
            store_row4(p, rm.out(p, r0 + j) + gcol, a);
        } else {
            float v[4] = {a.x, a.y, a.z, a.w};
            col_epilogue<4>(p, grow, gcol, v);
            store4(p, shard, grow, gcol, make_float4(v[0], v[1], v[2], v[3]));
        }
    }
}

// The reductions of a warp's pending split parts: items w0, w0 + n_units,
// ... (n of them).  For each, wait (bounded) until all parts of its tile
// have counted in, reduce this part's rows of the warp's block (those
// below M) over all parts, and count out.  False when a wait gave up.
template <class C, int SL>
__device__ __noinline__ bool split_fixups(const Params& p, int w0, int n, int n_units, int kbt, uint32_t rank,
                                          int quarter, int half, int lane, volatile int* abort_flag, float* buf) {
    const int qh = quarter * 2 + half;
    const long long pstride = (long long)C::RANKS * EPI_WARPS * PART_FLOATS;
    for (int k = 0; k < n; ++k) {
        // item w0 + k * n_units is part w % parts of tile dp_items + w / parts
        Item it;
        it.sk = w0 + k * n_units;
        it.part = it.sk % p.parts;
        it.tile = p.dp_items + it.sk / p.parts;
        int m_blk, shard, n_blk;
        tile_coords(p, it.tile, C::GROUP_M, m_blk, shard, n_blk);
        const int row_base = m_blk * C::TILE_M + (int)rank * A_ROWS + quarter * 32;
        if (row_base >= p.M) continue;  // the whole block is past M: its parts never counted in
        int* fl = p.flags + (((long long)(it.tile - p.dp_items) * C::RANKS + rank) * EPI_WARPS + qh) * 2;
        // this part's rows of the warp's 32, those past M dropped
        const int r0 = 32 * it.part / p.parts;
        const int r1 = min(32 * (it.part + 1) / p.parts, p.M - row_base);
        if (r1 > r0) {
            int got = 1;
            if (lane == 0) got = wait_count(fl, p.parts, abort_flag, p.err, p.timeout_ns) ? 1 : 0;
            got = __shfl_sync(0xffffffffu, got, 0);
            if (!got) return false;
            __threadfence();
            const float* base0 = p.partials +
                                 ((long long)(it.sk - it.part) * C::RANKS + rank) * EPI_WARPS * PART_FLOATS +
                                 (long long)qh * PART_FLOATS;
            reduce_rows<SL>(p, base0, pstride, lane, row_base, r0, r1, shard, n_blk * BN + half * HALF_N, buf);
            __syncwarp();
        }
        // count out; every part counted in before it counts out, so the
        // last one out finds the block's parts all in and all done, and
        // returns both counters to zero for the next launch on this scratch
        if (lane == 0) {
            if (atomicAdd(fl + 1, 1) == p.parts - 1) {
                atomicExch(fl, 0);
                atomicExch(fl + 1, 0);
            }
        }
    }
    return true;
}

// PAIR: 256-row tiles on an SM pair (cta_group::2), else 128-row tiles on
// one SM.  SL: the layout (out_row): a sequence-parallel layout (gathered
// input rows or sliced row-parallel outputs) has its own instantiation, so
// the plain one carries none of its code.
template <bool PAIR, int SL>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmW, Params p) {
    using C = GCfg<PAIR>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    float* stage_area = reinterpret_cast<float*>(smem + C::STAGES * C::STAGE_BYTES);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::STAGES * C::STAGE_BYTES + STG_BYTES);
    uint64_t* empty = full + C::STAGES;
    uint64_t* tmem_full = empty + C::STAGES;
    uint64_t* tmem_empty = tmem_full + 2;
    uint64_t* drain = tmem_empty + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    griddep_launch_dependents();  // the next kernel may set up while this one runs
    // PAIR: rank in the cluster (0 issues the MMAs) and the item stream of the pair
    const uint32_t rank = PAIR ? cluster_ctarank() : 0u;
    const int unit = PAIR ? (int)(blockIdx.x / 2) : (int)blockIdx.x;
    const int n_units = PAIR ? (int)(gridDim.x / 2) : (int)gridDim.x;

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&tmem_full[b], 1);
            mbar_init(&tmem_empty[b], (PAIR ? 2 : 1) * EPI_WARPS);  // epilogue warps of both CTAs
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        fence_async_smem();
    }
    if (warp == 1) {
        if constexpr (PAIR)
            tmem_alloc_pair(tmem_slot, TMEM_COLS);
        else
            tmem_alloc(tmem_slot, TMEM_COLS);
    }
    tc_fence_before();
    __syncthreads();
    if constexpr (PAIR) cluster_sync();  // the peer's barriers are initialised before any remote arrive
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    // everything below may read what the previous kernel of the stream wrote
    // (operands, residual, row scales) or reuse its scratch
    griddep_wait();
    const int kbt = p.reduce ? p.shards * p.k_blocks : p.k_blocks;  // k-blocks per tile

    if (warp == 0) {
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            Work wk;
            wk.init(unit, n_units, kbt);
            Item it;
            while (ok && wk.next(p, it)) {
                int m_blk, shard, n_blk;
                tile_coords(p, it.tile, C::GROUP_M, m_blk, shard, n_blk);
                const int a_row = m_blk * C::TILE_M + (int)rank * A_ROWS;
                const int w_row = n_blk * BN + (int)rank * C::W_ROWS;
                // gathered rows in 128-row-aligned slices: one box, its
                // coordinates fixed for the tile
                const int a_x = SL == 2 && p.a_box ? a_row % p.slice_rows : a_row;
                const int a_s = SL == 2 && p.a_box ? a_row / p.slice_rows : 0;
                for (int kb = it.k0; kb < it.k1; ++kb) {
                    if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, p.err, p.timeout_ns)) {
                        ok = false;
                        break;
                    }
                    const int s = p.reduce ? kb / p.k_blocks : shard;
                    const int kk = (p.reduce ? kb % p.k_blocks : kb) * BK;
                    const uint32_t sa = smem_u32(smem + stage * C::STAGE_BYTES);
                    if constexpr (PAIR) {
                        // both CTAs' copies complete on the issuing CTA's barrier
                        const uint32_t bar0 = mapa_shared(smem_u32(&full[stage]), 0);
                        if (rank == 0) mbar_expect_tx(&full[stage], 2 * C::STAGE_BYTES);
                        if (SL == 1 && p.a_box)
                            for (int j = 0; j < A_ROWS; j += p.a_box)  // gathered rows: one box per slice piece
                                tma_load_3d_pair(sa + j * BK * 2, &tmA, bar0, kk, (a_row + j) % p.slice_rows,
                                                 (a_row + j) / p.slice_rows);
                        else if (SL == 2 && p.a_box)
                            tma_load_3d_pair(sa, &tmA, bar0, kk, a_x, a_s);
                        else
                            tma_load_3d_pair(sa, &tmA, bar0, kk, a_row, p.reduce ? s : 0);
                        tma_load_3d_pair(sa + C::A_BYTES, &tmW, bar0, kk, w_row, s);
                    } else {
                        mbar_expect_tx(&full[stage], C::STAGE_BYTES);
                        if (SL == 1 && p.a_box)
                            for (int j = 0; j < A_ROWS; j += p.a_box)
                                tma_load_3d(sa + j * BK * 2, &tmA, smem_u32(&full[stage]), kk, (a_row + j) % p.slice_rows,
                                            (a_row + j) / p.slice_rows);
                        else if (SL == 2 && p.a_box)
                            tma_load_3d(sa, &tmA, smem_u32(&full[stage]), kk, a_x, a_s);
                        else
                            tma_load_3d(sa, &tmA, smem_u32(&full[stage]), kk, a_row, p.reduce ? s : 0);
                        tma_load_3d(sa + C::A_BYTES, &tmW, smem_u32(&full[stage]), kk, w_row, s);
                    }
                    if (++stage == C::STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (!ok) {
                // let copies already issued land before the CTA goes away
                const unsigned long long t0 = globaltimer();
                while (globaltimer() - t0 < 1000000ull) __nanosleep(1000);
            }
        }
    } else if (warp == 1) {
        if (lane == 0 && rank == 0) {
            int stage = 0;
            uint32_t phase = 0;
            int i = 0;
            bool ok = true;
            Work wk;
            wk.init(unit, n_units, kbt);
            Item it;
            for (; ok && wk.next(p, it); ++i) {
                const int buf = i & 1;
                const uint32_t acc_phase = (uint32_t)(i >> 1) & 1u;
                if (!mbar_wait(&tmem_empty[buf], acc_phase ^ 1u, abort_flag, p.err, p.timeout_ns)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + (uint32_t)(buf * BN);
                for (int kb = it.k0; kb < it.k1; ++kb) {
                    if (!mbar_wait(&full[stage], phase, abort_flag, p.err, p.timeout_ns)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sa = smem_u32(smem + stage * C::STAGE_BYTES);
                    const uint64_t adesc = sw128_kmajor(sa);
                    const uint64_t bdesc = sw128_kmajor(sa + C::A_BYTES);
#pragma unroll
                    for (int k = 0; k < BK / 16; ++k) {  // +32 bytes per K step inside the swizzle row
                        const uint32_t acc = (kb > it.k0 || k > 0) ? 1u : 0u;
                        if constexpr (PAIR)
                            umma_f16_pair(d_tmem, adesc + (uint64_t)(2 * k), bdesc + (uint64_t)(2 * k), C::IDESC, acc);
                        else
                            umma_f16(d_tmem, adesc + (uint64_t)(2 * k), bdesc + (uint64_t)(2 * k), C::IDESC, acc);
                    }
                    if constexpr (PAIR)
                        umma_commit_pair(&empty[stage], 3);  // frees the stage in both CTAs
                    else
                        umma_commit(&empty[stage]);
                    if (++stage == C::STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (ok) {
                    if constexpr (PAIR)
                        umma_commit_pair(&tmem_full[buf], 3);
                    else
                        umma_commit(&tmem_full[buf]);
                }
            }
            // drain: wait for every MMA issued by this thread before TMEM is freed
            if constexpr (PAIR)
                umma_commit_pair(drain, 1);
            else
                umma_commit(drain);
            const uint32_t a = smem_u32(drain);
            const unsigned long long t0 = globaltimer();
            while (!mbar_try_wait(a, 0)) {
                if (globaltimer() - t0 > drain_limit_ns(p.timeout_ns)) {
                    record_error(p.err, DEV_ERR_TIMEOUT);
                    break;
                }
            }
        }
    } else {
        // epilogue warps 2..9 -> TMEM lane quarter warp % 4 (2,3,0,1,2,3,0,1)
        // and column half (warp - 2) / 4; each warp works on its own 32 rows
        // x 128 columns and never waits for the other epilogue warps
        const int quarter = warp & 3, half = (warp - 2) >> 2, qh = quarter * 2 + half;
        float* stg = stage_area + (warp - 2) * STG_FLOATS;
        // L2 prefetch of the residual rows this warp will add for an item
        auto prefetch_item = [&](const Item& it) {
            int m_blk, shard, n_blk;
            tile_coords(p, it.tile, C::GROUP_M, m_blk, shard, n_blk);
            const int rb = m_blk * C::TILE_M + (int)rank * A_ROWS + quarter * 32;
            const int r0 = it.sk >= 0 ? 32 * it.part / p.parts : 0;
            const int r1 = it.sk >= 0 ? 32 * (it.part + 1) / p.parts : 32;
            prefetch_residual<SL>(p, lane, rb, r0, r1, n_blk * BN + half * HALF_N);
        };
        // A part's partial is written (and TMEM handed back) as soon as its
        // MMAs are done; its reduction waits for the end of the unit's work,
        // so it neither stalls the main loops nor competes with their
        // operand stream for this SM's loads, and no partial write ever
        // waits for another unit.
        int pend_w = 0, n_pend = 0;  // parts to reduce: items pend_w, pend_w + n_units, ...
        bool ok = true;
        // this warp's share of the ring, used only once the unit's last
        // MMAs have completed (no copy or MMA touches the ring then)
        float* fixbuf = reinterpret_cast<float*>(smem + (warp - 2) * FIX_BYTES);
        Work wk;
        wk.init(unit, n_units, kbt);
        Item it;
        int i = 0;
        for (; wk.next(p, it); ++i) {
            prefetch_item(it);  // (its MMAs are usually still running)
            const int buf = i & 1;
            const uint32_t acc_phase = (uint32_t)(i >> 1) & 1u;
            if (!mbar_wait_warp(&tmem_full[buf], acc_phase, abort_flag, p.err, p.timeout_ns)) {
                ok = false;
                break;
            }
            tc_fence_after();
            int m_blk, shard, n_blk;
            tile_coords(p, it.tile, C::GROUP_M, m_blk, shard, n_blk);
            const int row_base = m_blk * C::TILE_M + (int)rank * A_ROWS + quarter * 32;
            const uint32_t tbase =
                tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(buf * BN + half * HALF_N);
            const int col0 = n_blk * BN + half * HALF_N;
            if (it.sk < 0) {
                if (p.epi != EPI_ROW_REDUCE)
                    epilogue_col(p, tbase, stg, lane, row_base, shard, col0);
                else {
                    Work peek = wk;
                    Item nx;
                    float* rbuf = peek.next(p, nx) ? nullptr : fixbuf;  // last item: the ring is idle
                    if (p.residual == nullptr)
                        epilogue_row<0, SL>(p, tbase, stg, lane, row_base, col0, nullptr);
                    else if (p.residual_f32)
                        epilogue_row<2, SL>(p, tbase, stg, lane, row_base, col0, rbuf);
                    else
                        epilogue_row<1, SL>(p, tbase, stg, lane, row_base, col0, rbuf);
                }
            } else {
                float* part = p.partials + ((long long)it.sk * C::RANKS + rank) * EPI_WARPS * PART_FLOATS +
                              (long long)qh * PART_FLOATS;
                write_partial(tbase, stg, lane, part, p.M - row_base);
            }
            // the accumulator is in registers / memory now: hand TMEM back
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if constexpr (PAIR)
                    mbar_arrive_cluster(mapa_shared(smem_u32(&tmem_empty[buf]), 0));  // the issuing CTA's
                else
                    mbar_arrive(&tmem_empty[buf]);
            }
            if (it.sk >= 0) {
                // count this part in (its partial is complete and visible)
                int* fl = p.flags + (((long long)(it.tile - p.dp_items) * C::RANKS + rank) * EPI_WARPS + qh) * 2;
                __threadfence();
                __syncwarp();
                if (lane == 0 && row_base < p.M) atomicAdd(fl, 1);
                if (n_pend++ == 0) pend_w = it.sk;
            }
        }
        if (ok && n_pend > 0)
            split_fixups<C, SL>(p, pend_w, n_pend, n_units, kbt, rank, quarter, half, lane, abort_flag, fixbuf);
    }

    tc_fence_before();
    __syncthreads();
    if constexpr (PAIR) cluster_sync();  // no remote arrive or MMA write lands after the peer leaves
    tc_fence_after();
    if (warp == 1) {
        if constexpr (PAIR)
            tmem_dealloc_pair(tmem_base, TMEM_COLS);
        else
            tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static std::atomic<EncodeTiledFn> fn{nullptr};  // racing first calls store the same address
    EncodeTiledFn f = fn.load();
    if (!f) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess) {
            f = reinterpret_cast<EncodeTiledFn>(p);
            fn.store(f);
        }
    }
    return f;
}

// 3-D bf16 tensor [d2][d1][d0] (d0 contiguous), box {64, box1, 1}, 128B swizzle.
bool make_map(CUtensorMap* m, const void* base, uint64_t d0, uint64_t d1, uint64_t d2, uint64_t stride1_bytes,
              uint64_t stride2_bytes, uint32_t box1) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {d0, d1, d2};
    cuuint64_t strides[2] = {stride1_bytes, stride2_bytes};
    cuuint32_t box[3] = {(cuuint32_t)BK, box1, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

int sm_count() {
    static std::atomic<int> n[64];  // per device; racing first calls store the same value
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) return 148;
    int v = n[dev].load();
    if (!v) {
        cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
        n[dev].store(v);
    }
    return v > 0 ? v : 148;
}

}  // namespace

bool tc_gemm_supported(int M, int N, int K) { return M >= 1 && N >= 1 && K >= 8 && K % 8 == 0; }

namespace {

// Co-resident clusters of two for the paired kernel (an SM pair must come
// from one GPC, so this can be below SMs / 2).
int pair_slots() {
    static std::atomic<int> n[64];  // per device; racing first calls store the same value
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) return 0;
    if (!n[dev].load()) {
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.gridDim = dim3(2 * 74, 1, 1);
        cfg.blockDim = dim3(NUM_THREADS, 1, 1);
        cfg.dynamicSmemBytes = GCfg<true>::SMEM;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int c = 0;
        if (cudaOccupancyMaxActiveClusters(&c, tc_gemm_kernel<true, 0>, &cfg) != cudaSuccess || c <= 0) {
            cudaGetLastError();
            c = -1;
        }
        n[dev].store(c);
    }
    const int v = n[dev].load();
    return v > 0 ? v : 0;
}

template <bool PAIR>
cudaError_t set_smem_attr() {
    static std::atomic<bool> done[64];  // per device; racing first calls set the same attribute
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && !done[dev].load()) {
        cudaError_t e =
            cudaFuncSetAttribute(tc_gemm_kernel<PAIR, 0>, cudaFuncAttributeMaxDynamicSharedMemorySize, GCfg<PAIR>::SMEM);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(tc_gemm_kernel<PAIR, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     GCfg<PAIR>::SMEM);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(tc_gemm_kernel<PAIR, 2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     GCfg<PAIR>::SMEM);
        if (e != cudaSuccess) return e;
        done[dev].store(true);
    }
    return cudaSuccess;
}

// Split tiles: at most this many parts per tile, at least this many
// k-blocks per part, at most this many split items per unit (the partials'
// scratch); writing a part's 128 KB partial per SM takes about as long as
// SPLIT_EPI_KB k-blocks of MMAs, so shorter parts leave the epilogue
// behind; the reductions at the end of the launch are left exposed
// (SPLIT_COST_KB) and move every partial twice (written, read back):
// about SPLIT_MB_PER_KB MB of that traffic over the whole GPU costs one
// k-block of time (a k-block of a tile takes ~0.4 us).  The two constants
// were fitted to split / whole-tile timings of the 7B-shaped linears on a
// B300 (M = 128 .. 4096): a split paid off only where it saved more than
// ~10 us plus the traffic.  Partial rows past M are neither written nor
// read, so with fewer rows than a tile holds (few-token decode) the
// traffic shrinks with the row fill, and so does the exposed reduction
// (down to a quarter: its latency stays).
constexpr int SPLIT_MAX_PARTS = 16, SPLIT_MIN_KB = 4, SPLIT_MAX_ROUNDS = SPLIT_ROUNDS_MAX, SPLIT_EPI_KB = 6,
              SPLIT_COST_KB = 24;
constexpr double SPLIT_MB_PER_KB = 1.2;
constexpr size_t FLAG_BYTES = 16384;  // [split tile][rank][epilogue warp][2] ints; split tiles < units <= SMs

struct Decomp {
    int dp, parts, n_items, units;
    size_t scratch;  // bytes of scratch touched
};

// Work decomposition over `units` co-resident units (SM pairs or SMs) for
// T tiles of kbt k-blocks: the tiles that fill whole rounds run whole; the
// remaining tiles are cut into equal k-parts (run first) so that the units
// end evenly loaded.  The makespan (in k-blocks per unit) decides.  fill:
// the share of the tiles' rows that lie below M.
Decomp choose_decomp(int T, int kbt, int units, int ranks, double fill, size_t scratch_bytes) {
    Decomp d{T, 1, T, T < units ? T : units, 0};
    long long best = (long long)((T + units - 1) / units) * kbt;
    if (scratch_bytes <= FLAG_BYTES) return d;
    const int full = T / units, rem = T - full * units;
    if (rem == 0 || (size_t)rem * ranks * EPI_WARPS * 2 * sizeof(int) > FLAG_BYTES) return d;
    for (int parts = 2; parts <= SPLIT_MAX_PARTS && kbt / parts >= SPLIT_MIN_KB; ++parts) {
        const long long items = (long long)rem * parts;
        if (items > (long long)SPLIT_MAX_ROUNDS * units) break;
        const size_t need = FLAG_BYTES + (size_t)items * ranks * A_ROWS * BN * sizeof(float);
        if (need > scratch_bytes) break;
        const long long rounds = (items + units - 1) / units;
        const long long per_item = (kbt + parts - 1) / parts;
        const double traffic_mb = 2.0 * fill * (double)items * ranks * A_ROWS * BN * sizeof(float) / 1e6;
        const long long span = (long long)full * kbt + rounds * (per_item > SPLIT_EPI_KB ? per_item : SPLIT_EPI_KB) +
                               (long long)(SPLIT_COST_KB * (fill > 0.25 ? fill : 0.25)) +
                               (long long)(traffic_mb / SPLIT_MB_PER_KB);
        if (span < best) {
            best = span;
            d.dp = full * units;
            d.parts = parts;
            d.n_items = (int)(d.dp + items);
            d.units = units;
            d.scratch = need;
        }
    }
    return d;
}

template <bool PAIR>
cudaError_t gemm_launch(const TcGemm& g, int* dev_err, int slots, void* scratch, size_t scratch_bytes,
                        cudaStream_t st, bool* counters_zero) {
    using C = GCfg<PAIR>;
    CUtensorMap tmA, tmW;
    const uint64_t a_shards = g.reduce ? (uint64_t)g.shards : 1;
    int a_box = 0;
    if (!g.reduce && g.slice_rows > 0) {
        // gathered input [slices][slice_rows][K]: boxes of the largest power
        // of two <= 128 rows dividing slice_rows, so that no box crosses a
        // slice (slice_rows is a multiple of 8; each box lands on a 1 KB
        // boundary of the stage, as the 128-byte swizzle needs)
        a_box = A_ROWS;
        while (g.slice_rows % a_box) a_box /= 2;
        const uint64_t n_slices = (uint64_t)((g.M + g.slice_rows - 1) / g.slice_rows);
        if (!make_map(&tmA, g.A, (uint64_t)g.K, (uint64_t)g.slice_rows, n_slices, (uint64_t)g.lda * 2,
                      (uint64_t)g.a_slice * 2, (uint32_t)a_box))
            return cudaErrorInvalidValue;
    } else if (!make_map(&tmA, g.A, (uint64_t)g.K, (uint64_t)g.M, a_shards, (uint64_t)g.lda * 2,
                         (uint64_t)g.M * g.lda * 2, A_ROWS)) {
        return cudaErrorInvalidValue;
    }
    if (!make_map(&tmW, g.W, (uint64_t)g.K, (uint64_t)g.N, (uint64_t)g.shards, (uint64_t)g.K * 2,
                  (uint64_t)g.w_shard * 2, C::W_ROWS))
        return cudaErrorInvalidValue;
    Params p{};
    p.epi = g.epi;
    p.M = g.M;
    p.N = g.N;
    p.K = g.K;
    p.shards = g.shards;
    p.reduce = g.reduce;
    p.m_blocks = (g.M + C::TILE_M - 1) / C::TILE_M;
    p.n_blocks = (g.N + BN - 1) / BN;
    p.k_blocks = (g.K + BK - 1) / BK;
    p.n_tiles = p.m_blocks * p.n_blocks * (g.reduce ? 1 : g.shards);
    p.out = g.out;
    p.out_shard = g.out_shard;
    p.ldo = g.ldo;
    p.out2 = g.out2;
    p.residual = g.residual;
    p.residual_f32 = g.residual_f32;
    p.granule = g.granule;
    p.err = dev_err;
    p.timeout_ns = wait_timeout_ns();
    p.row_scale = g.row_scale;
    p.rope_cols = g.rope_cols;
    p.rope_dh = g.rope_dh;
    p.rope_seq = g.rope_seq > 0 ? g.rope_seq : 1;
    p.rope_cs = g.rope_cs;
    p.slice_rows = g.slice_rows > 0 ? g.slice_rows : 0;
    p.out_slice = g.out_slice;
    p.res_slice = g.res_slice;
    p.a_box = a_box;
    const int kbt = (g.reduce ? g.shards : 1) * p.k_blocks;
    const double fill = (double)g.M / ((double)p.m_blocks * C::TILE_M);
    const Decomp d = choose_decomp(p.n_tiles, kbt, slots, C::RANKS, fill, scratch ? scratch_bytes : 0);
    p.dp_items = d.dp;
    p.parts = d.parts;
    p.n_items = d.n_items;
    if (d.parts > 1) {
        p.flags = static_cast<int*>(scratch);
        p.partials = reinterpret_cast<float*>(static_cast<char*>(scratch) + FLAG_BYTES);
        // the split tiles' counters start at zero whatever the scratch held
        // (a few KB; only launches that split, and not already known to
        // find them zero, pay for it)
        if (!counters_zero || !*counters_zero) {
            const cudaError_t e = cudaMemsetAsync(scratch, 0, FLAG_BYTES, st);
            if (e != cudaSuccess) return e;
        }
        if (counters_zero) *counters_zero = true;
    }
    const int units = d.units;
    // programmatic dependent launch: this grid may start while the previous
    // kernel of the stream finishes (the kernel waits before its first read)
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = PAIR ? 2 : 1;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.gridDim = dim3((PAIR ? 2 : 1) * units, 1, 1);
    cfg.blockDim = dim3(NUM_THREADS, 1, 1);
    cfg.dynamicSmemBytes = C::SMEM;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = PAIR ? 2 : 1;
    // sliced layouts (a gathered input, or row-parallel outputs / residual in
    // slices) take their own instantiation, so that the plain one carries
    // neither the per-row slice mapping nor the gathered loads (in the
    // producer's loop they cost the plain 7B prefill linears 5-12 us)
    if (p.slice_rows > 0 && p.slice_rows % A_ROWS == 0) return cudaLaunchKernelEx(&cfg, tc_gemm_kernel<PAIR, 2>, tmA, tmW, p);
    if (p.slice_rows > 0) return cudaLaunchKernelEx(&cfg, tc_gemm_kernel<PAIR, 1>, tmA, tmW, p);
    return cudaLaunchKernelEx(&cfg, tc_gemm_kernel<PAIR, 0>, tmA, tmW, p);
}

}  // namespace

size_t tc_gemm_scratch_bytes() {
    // split items <= SPLIT_MAX_ROUNDS per unit, and ranks x units <= SMs, so
    // the partials never exceed SPLIT_MAX_ROUNDS 128 x 256 fp32 blocks per SM
    return FLAG_BYTES + (size_t)SPLIT_MAX_ROUNDS * sm_count() * A_ROWS * BN * sizeof(float);
}

TcSchedule tc_gemm_schedule(const TcGemm& g, size_t scratch_bytes, int sms, int slots) {
    TcSchedule r{};
    r.paired = g.M > A_ROWS && slots > 0;
    const int tile_m = r.paired ? 256 : 128;
    const int m_blocks = (g.M + tile_m - 1) / tile_m, n_blocks = (g.N + BN - 1) / BN;
    r.tiles = m_blocks * n_blocks * (g.reduce ? 1 : g.shards);
    r.kbt = (g.reduce ? g.shards : 1) * ((g.K + BK - 1) / BK);
    const int ranks = r.paired ? 2 : 1;
    const double fill = (double)g.M / ((double)m_blocks * tile_m);
    const Decomp d = choose_decomp(r.tiles, r.kbt, r.paired ? slots : sms, ranks, fill, scratch_bytes);
    r.units = d.units;
    r.scratch_touched = d.scratch;
    r.whole = d.dp;
    r.parts = d.parts;
    r.items = d.n_items;
    return r;
}

cudaError_t tc_gemm(const TcGemm& g, int* dev_err, void* scratch, size_t scratch_bytes, cudaStream_t st,
                    bool* counters_zero) {
    if (g.epi == EPI_SWIGLU && (g.granule != 32 || g.N % 64 != 0)) return cudaErrorNotSupported;
    if (g.N % 8 != 0 || g.ldo % 8 != 0) return cudaErrorNotSupported;  // 4- and 8-wide vector stores
    if (g.slice_rows < 0 || (g.slice_rows > 0 && (g.slice_rows % 8 != 0 || g.a_slice % 8 != 0 || g.out_slice % 8 != 0 ||
                                                 g.res_slice % 8 != 0)))
        return cudaErrorNotSupported;
    cudaError_t e = set_smem_attr<false>();
    if (e == cudaSuccess) e = set_smem_attr<true>();
    if (e != cudaSuccess) return e;
    // 2-SM tiles once there is more than one 128-row block of tokens
    if (g.M > A_ROWS) {
        const int slots = pair_slots();
        if (slots > 0) return gemm_launch<true>(g, dev_err, slots, scratch, scratch_bytes, st, counters_zero);
    }
    return gemm_launch<false>(g, dev_err, sm_count(), scratch, scratch_bytes, st, counters_zero);
}

}  // namespace tpk
