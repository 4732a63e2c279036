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
//       the same TMEM accumulator, so no partial is ever written to memory.
//
// Two variants of one persistent kernel (one CTA per SM, 192 threads):
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
//   warps 2-5 epilogue: tcgen05.ld of the finished accumulator (each warp its
//            32-lane quarter), activation / residual, stores to global.
// The epilogue of tile i overlaps the main loop of tile i+1 (two TMEM
// accumulators = all 512 columns).  Every mbarrier wait is bounded: after
// `timeout_ns` the waiting role records TP_ERR_DEVICE_TIMEOUT's device code,
// raises a CTA-wide abort flag and leaves its loop; in-flight tensor-core
// work is drained and TMEM freed before the CTA exits, and the two CTAs of a
// pair leave together.
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
constexpr int NUM_THREADS = 192;
constexpr unsigned long long DEFAULT_TIMEOUT_NS = 2000000000ull;  // 2 s

template <bool PAIR>
struct GCfg {
    static constexpr int TILE_M = PAIR ? 256 : 128;   // output rows per tile
    static constexpr int W_ROWS = PAIR ? BN / 2 : BN;  // W rows staged per CTA
    static constexpr int A_BYTES = A_ROWS * BK * 2;
    static constexpr int STAGE_BYTES = A_BYTES + W_ROWS * BK * 2;
    static constexpr int STAGES = PAIR ? TP_GEMM_PAIR_STAGES : 4;
    static constexpr int GROUP_M = PAIR ? 8 : 16;       // row blocks per raster band (2048 rows)
    static constexpr int SMEM = STAGES * STAGE_BYTES + 1024 + 256;
    // instruction descriptor: D fp32, A/B bf16, both K-major
    static constexpr uint32_t IDESC = ptx::idesc_bf16(TILE_M, BN, false);
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
    // split-K: the k-blocks of every tile are cut into `splits` equal ranges
    // computed by different units; each writes its fp32 partial sums to
    // partials[split][shard][row][col] (row < M, col < N) and
    // splitk_reduce_k sums them in split order and applies the epilogue
    int splits;
    float* partials;
    // pre-norm variant: see TcGemm
    const float* row_scale;
    int rope_cols, rope_dh, rope_seq;
    const float2* rope_cs;
};

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

// One unit's work: items w = unit, unit + n_units, ... of the sequence
// (split-major, tile-minor, so units in flight together share k ranges and
// operand tiles); item w is tile w % n_tiles over the k-blocks of split
// w / n_tiles.
struct Seg {
    int tile, split, k0, k1;
};
struct Sched {
    int w, n_items, n_tiles, kbt, splits, n_units;
    __device__ void init(const Params& p, int unit, int n_units_, int kbt_) {
        w = unit;
        n_units = n_units_;
        n_tiles = p.n_tiles;
        kbt = kbt_;
        splits = p.splits;
        n_items = n_tiles * splits;
    }
    __device__ bool next(Seg& g) {
        if (w >= n_items) return false;
        g.tile = w % n_tiles;
        g.split = w / n_tiles;
        g.k0 = (int)((long long)kbt * g.split / splits);
        g.k1 = (int)((long long)kbt * (g.split + 1) / splits);
        w += n_units;
        return true;
    }
};

__device__ __forceinline__ uint64_t sw128_kmajor(uint32_t saddr) { return sw128_desc(saddr, 16, 1024); }

// 32 consecutive bf16 of one row; `n_valid` of them inside the matrix.
__device__ __forceinline__ void store_row_bf16(bf16* dst, const float (&v)[32], int n_valid) {
    if (n_valid >= 32) {
        uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
        for (int q = 0; q < 4; ++q)
            d4[q] = make_uint4(pack_bf16x2(v[8 * q + 0], v[8 * q + 1]), pack_bf16x2(v[8 * q + 2], v[8 * q + 3]),
                               pack_bf16x2(v[8 * q + 4], v[8 * q + 5]), pack_bf16x2(v[8 * q + 6], v[8 * q + 7]));
    } else {
#pragma unroll
        for (int i = 0; i < 32; ++i)
            if (i < n_valid) dst[i] = __float2bfloat16_rn(v[i]);
    }
}

template <bool PAIR>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmW, Params p) {
    using C = GCfg<PAIR>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::STAGES * C::STAGE_BYTES);
    uint64_t* empty = full + C::STAGES;
    uint64_t* tmem_full = empty + C::STAGES;
    uint64_t* tmem_empty = tmem_full + 2;
    uint64_t* drain = tmem_empty + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    // PAIR: rank in the cluster (0 issues the MMAs) and the tile stream of the pair
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
            mbar_init(&tmem_empty[b], PAIR ? 8 : 4);  // epilogue warps of both CTAs
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
    const int kb_per_tile = p.reduce ? p.shards * p.k_blocks : p.k_blocks;

    if (warp == 0) {
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            Sched sc;
            sc.init(p, unit, n_units, kb_per_tile);
            Seg g;
            while (ok && sc.next(g)) {
                const int t = g.tile;
                int m_blk, shard, n_blk;
                tile_coords(p, t, C::GROUP_M, m_blk, shard, n_blk);
                const int a_row = m_blk * C::TILE_M + (int)rank * A_ROWS;
                const int w_row = n_blk * BN + (int)rank * C::W_ROWS;
                for (int kb = g.k0; kb < g.k1; ++kb) {
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
                        tma_load_3d_pair(sa, &tmA, bar0, kk, a_row, p.reduce ? s : 0);
                        tma_load_3d_pair(sa + C::A_BYTES, &tmW, bar0, kk, w_row, s);
                    } else {
                        mbar_expect_tx(&full[stage], C::STAGE_BYTES);
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
            Sched sc;
            sc.init(p, unit, n_units, kb_per_tile);
            Seg g;
            for (; ok && sc.next(g); ++i) {
                const int buf = i & 1;
                const uint32_t acc_phase = (uint32_t)(i >> 1) & 1u;
                if (!mbar_wait(&tmem_empty[buf], acc_phase ^ 1u, abort_flag, p.err, p.timeout_ns)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + (uint32_t)(buf * BN);
                for (int kb = g.k0; kb < g.k1; ++kb) {
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
                        const uint32_t acc = (kb > g.k0 || k > 0) ? 1u : 0u;
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
                if (globaltimer() - t0 > p.timeout_ns) {
                    record_error(p.err, DEV_ERR_TIMEOUT);
                    break;
                }
            }
        }
    } else {
        // epilogue warps 2..5 -> TMEM lane quarters 2,3,0,1
        const int quarter = warp & 3;
        int i = 0;
        Sched sc;
        sc.init(p, unit, n_units, kb_per_tile);
        Seg sg;
        for (; sc.next(sg); ++i) {
            const int t = sg.tile;
            const int buf = i & 1;
            const uint32_t acc_phase = (uint32_t)(i >> 1) & 1u;
            if (!mbar_wait_warp(&tmem_full[buf], acc_phase, abort_flag, p.err, p.timeout_ns)) break;
            tc_fence_after();
            int m_blk, shard, n_blk;
            tile_coords(p, t, C::GROUP_M, m_blk, shard, n_blk);
            const int row = m_blk * C::TILE_M + (int)rank * A_ROWS + quarter * 32 + lane;
            const uint32_t tbase = tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(buf * BN);
            const int col_base = n_blk * BN;
            const bool row_ok = row < p.M;
            if (p.splits > 1) {
                // split-K: raw fp32 partial sums of this split
                // [split][shard][row][col]; a row-parallel launch has one output "shard"
                const int n_sh = p.reduce ? 1 : p.shards;
                float* dst = p.partials + (((long long)sg.split * n_sh + shard) * p.M + row) * p.N;
#pragma unroll 1
                for (int c = 0; c < BN / 32; ++c) {
                    float v[32];
                    __syncwarp();
                    tmem_ld32(tbase + 32 * c, v);
                    const int col = col_base + 32 * c;
                    if (!row_ok || col >= p.N) continue;
                    if (col + 32 <= p.N) {
                        float4* d4 = reinterpret_cast<float4*>(dst + col);
#pragma unroll
                        for (int q = 0; q < 8; ++q)
                            __stcg(d4 + q, make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]));
                    } else {
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            if (col + j < p.N) dst[col + j] = v[j];
                    }
                }
            } else if (p.epi == EPI_SWIGLU) {
                bf16* out = (bf16*)p.out + shard * p.out_shard + (long long)row * p.ldo;
#pragma unroll 1
                for (int g = 0; g < BN / 64; ++g) {
                    float gate[32], up[32];
                    __syncwarp();
                    tmem_ld32(tbase + 64 * g, gate);
                    tmem_ld32(tbase + 64 * g + 32, up);
                    const int pc = col_base + 64 * g;  // packed column of this gate block
                    if (row_ok && pc < p.N) {
                        const float rs = p.row_scale ? p.row_scale[row] : 1.f;
#pragma unroll
                        for (int j = 0; j < 32; ++j) gate[j] = silu(gate[j] * rs) * (up[j] * rs);
                        store_row_bf16(out + pc / 2, gate, 32);
                    }
                }
            } else if (p.epi == EPI_ROW_REDUCE) {
                const long long roff = (long long)row * p.ldo;
#pragma unroll 1
                for (int c = 0; c < BN / 32; ++c) {
                    float v[32];
                    __syncwarp();
                    tmem_ld32(tbase + 32 * c, v);
                    const int col = col_base + 32 * c;
                    if (!row_ok || col >= p.N) continue;
                    const int nv = min(32, p.N - col);
                    if (p.residual) {
                        if (p.residual_f32) {
                            const float* r = (const float*)p.residual + roff + col;
                            if (nv == 32) {
#pragma unroll
                                for (int q = 0; q < 8; ++q) {
                                    const float4 x = reinterpret_cast<const float4*>(r)[q];
                                    v[4 * q] += x.x;
                                    v[4 * q + 1] += x.y;
                                    v[4 * q + 2] += x.z;
                                    v[4 * q + 3] += x.w;
                                }
                            } else {
#pragma unroll
                                for (int j = 0; j < 32; ++j)
                                    if (j < nv) v[j] += r[j];
                            }
                        } else {
                            const bf16* r = (const bf16*)p.residual + roff + col;
                            if (nv == 32) {
#pragma unroll
                                for (int q = 0; q < 4; ++q) {
                                    const uint4 x = reinterpret_cast<const uint4*>(r)[q];
                                    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&x);
#pragma unroll
                                    for (int e = 0; e < 4; ++e) {
                                        const float2 f = __bfloat1622float2(h[e]);
                                        v[8 * q + 2 * e] += f.x;
                                        v[8 * q + 2 * e + 1] += f.y;
                                    }
                                }
                            } else {
#pragma unroll
                                for (int j = 0; j < 32; ++j)
                                    if (j < nv) v[j] += __bfloat162float(r[j]);
                            }
                        }
                    }
                    float* o = (float*)p.out + roff + col;
                    if (nv == 32) {
#pragma unroll
                        for (int q = 0; q < 8; ++q)
                            reinterpret_cast<float4*>(o)[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
                    } else {
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            if (j < nv) o[j] = v[j];
                    }
                    if (p.out2) store_row_bf16((bf16*)p.out2 + roff + col, v, nv);
                }
            } else {
                bf16* out = (bf16*)p.out + shard * p.out_shard + (long long)row * p.ldo;
#pragma unroll 1
                for (int c = 0; c < BN / 32; ++c) {
                    float v[32];
                    __syncwarp();
                    tmem_ld32(tbase + 32 * c, v);
                    const int col = col_base + 32 * c;
                    if (!row_ok || col >= p.N) continue;
                    if (p.row_scale) {
                        const float rs = p.row_scale[row];
#pragma unroll
                        for (int j = 0; j < 32; ++j) v[j] *= rs;
                    }
                    if (p.rope_cols > 0) apply_rope<32>(p, row, col, v);
                    if (p.epi == EPI_GELU) {
#pragma unroll
                        for (int j = 0; j < 32; ++j) v[j] = gelu_erf(v[j]);
                    }
                    store_row_bf16(out + col, v, min(32, p.N - col));
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if constexpr (PAIR)
                    mbar_arrive_cluster(mapa_shared(smem_u32(&tmem_empty[buf]), 0));  // the issuing CTA's
                else
                    mbar_arrive(&tmem_empty[buf]);
            }
        }
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

// Split-K second pass: out = epilogue(sum over splits of the partial sums),
// the splits added in order 0..S-1 (the result does not depend on which SM
// computed which split).  Four consecutive output columns per thread.
__global__ void __launch_bounds__(256) splitk_reduce_k(Params p) {
    const int n_out = p.epi == EPI_SWIGLU ? p.N / 2 : p.N;  // output columns per shard
    const int n_sh = p.reduce ? 1 : p.shards;
    const long long quads = (long long)n_sh * p.M * n_out / 4;
    const long long split_stride = (long long)n_sh * p.M * p.N;
    for (long long q = blockIdx.x * (long long)blockDim.x + threadIdx.x; q < quads;
         q += (long long)gridDim.x * blockDim.x) {
        const long long e = q * 4;
        const int col = (int)(e % n_out);
        const long long rs = e / n_out;  // shard * M + row
        const int row = (int)(rs % p.M), shard = (int)(rs / p.M);
        const float* base = p.partials + rs * p.N;
        float v[4];
        if (p.epi == EPI_SWIGLU) {
            // packed columns: gate block of 32, then the matching up block
            const int g = (col / 32) * 64 + col % 32;
            float4 ga = __ldcg(reinterpret_cast<const float4*>(base + g));
            float4 ua = __ldcg(reinterpret_cast<const float4*>(base + g + 32));
            for (int sp = 1; sp < p.splits; ++sp) {
                const float4 gb = __ldcg(reinterpret_cast<const float4*>(base + sp * split_stride + g));
                const float4 ub = __ldcg(reinterpret_cast<const float4*>(base + sp * split_stride + g + 32));
                ga.x += gb.x; ga.y += gb.y; ga.z += gb.z; ga.w += gb.w;
                ua.x += ub.x; ua.y += ub.y; ua.z += ub.z; ua.w += ub.w;
            }
            const float sc = p.row_scale ? p.row_scale[row] : 1.f;
            v[0] = silu(ga.x * sc) * (ua.x * sc);
            v[1] = silu(ga.y * sc) * (ua.y * sc);
            v[2] = silu(ga.z * sc) * (ua.z * sc);
            v[3] = silu(ga.w * sc) * (ua.w * sc);
        } else {
            float4 a = __ldcg(reinterpret_cast<const float4*>(base + col));
            for (int sp = 1; sp < p.splits; ++sp) {
                const float4 b = __ldcg(reinterpret_cast<const float4*>(base + sp * split_stride + col));
                a.x += b.x; a.y += b.y; a.z += b.z; a.w += b.w;
            }
            v[0] = a.x;
            v[1] = a.y;
            v[2] = a.z;
            v[3] = a.w;
            if (p.row_scale) {
                const float sc = p.row_scale[row];
#pragma unroll
                for (int j = 0; j < 4; ++j) v[j] *= sc;
            }
            if (p.rope_cols > 0) apply_rope<4>(p, row, col, v);
            if (p.epi == EPI_GELU) {
#pragma unroll
                for (int j = 0; j < 4; ++j) v[j] = gelu_erf(v[j]);
            }
        }
        if (p.epi == EPI_ROW_REDUCE) {
            const long long o = (long long)row * p.ldo + col;
            if (p.residual) {
                if (p.residual_f32) {
                    const float4 r = *reinterpret_cast<const float4*>((const float*)p.residual + o);
                    v[0] += r.x; v[1] += r.y; v[2] += r.z; v[3] += r.w;
                } else {
                    const uint2 r = *reinterpret_cast<const uint2*>((const bf16*)p.residual + o);
                    const float2 r0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&r.x));
                    const float2 r1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&r.y));
                    v[0] += r0.x; v[1] += r0.y; v[2] += r1.x; v[3] += r1.y;
                }
            }
            *reinterpret_cast<float4*>((float*)p.out + o) = make_float4(v[0], v[1], v[2], v[3]);
            if (p.out2)
                *reinterpret_cast<uint2*>((bf16*)p.out2 + o) = make_uint2(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]));
        } else {
            bf16* o = (bf16*)p.out + shard * p.out_shard + (long long)row * p.ldo + col;
            *reinterpret_cast<uint2*>(o) = make_uint2(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]));
        }
    }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    }
    return fn;
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
        if (cudaOccupancyMaxActiveClusters(&c, tc_gemm_kernel<true>, &cfg) != cudaSuccess || c <= 0) {
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
            cudaFuncSetAttribute(tc_gemm_kernel<PAIR>, cudaFuncAttributeMaxDynamicSharedMemorySize, GCfg<PAIR>::SMEM);
        if (e != cudaSuccess) return e;
        done[dev].store(true);
    }
    return cudaSuccess;
}

// Largest split factor; a split keeps at least this many k-blocks.
constexpr int SPLITK_MAX = 16, SPLITK_MIN_KB = 4;

template <bool PAIR>
cudaError_t gemm_launch(const TcGemm& g, int* dev_err, int slots, void* scratch, size_t scratch_bytes,
                        cudaStream_t st) {
    using C = GCfg<PAIR>;
    CUtensorMap tmA, tmW;
    const uint64_t a_shards = g.reduce ? (uint64_t)g.shards : 1;
    if (!make_map(&tmA, g.A, (uint64_t)g.K, (uint64_t)g.M, a_shards, (uint64_t)g.lda * 2,
                  (uint64_t)g.M * g.lda * 2, A_ROWS))
        return cudaErrorInvalidValue;
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
    p.timeout_ns = DEFAULT_TIMEOUT_NS;
    p.row_scale = g.row_scale;
    p.rope_cols = g.rope_cols;
    p.rope_dh = g.rope_dh;
    p.rope_seq = g.rope_seq > 0 ? g.rope_seq : 1;
    p.rope_cs = g.rope_cs;
    p.splits = 1;
    // split-K when whole tiles would leave at least half of the units idle
    if (scratch && 2 * p.n_tiles <= slots) {
        const int kbt = (g.reduce ? g.shards : 1) * p.k_blocks;
        int S = slots / p.n_tiles;
        if (S > SPLITK_MAX) S = SPLITK_MAX;
        if (S > kbt / SPLITK_MIN_KB) S = kbt / SPLITK_MIN_KB;
        const size_t need = (size_t)S * (g.reduce ? 1 : g.shards) * g.M * g.N * sizeof(float);
        if (S >= 2 && need <= scratch_bytes) {
            p.splits = S;
            p.partials = static_cast<float*>(scratch);
        }
    }
    const int items = p.n_tiles * p.splits;
    const int units = items < slots ? items : slots;
    cudaError_t e = cudaSuccess;
    if constexpr (PAIR) {
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.gridDim = dim3(2 * units, 1, 1);
        cfg.blockDim = dim3(NUM_THREADS, 1, 1);
        cfg.dynamicSmemBytes = C::SMEM;
        cfg.stream = st;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        e = cudaLaunchKernelEx(&cfg, tc_gemm_kernel<true>, tmA, tmW, p);
    } else {
        tc_gemm_kernel<false><<<units, NUM_THREADS, C::SMEM, st>>>(tmA, tmW, p);
        e = cudaGetLastError();
    }
    if (e != cudaSuccess || p.splits == 1) return e;
    const long long quads = (long long)(g.reduce ? 1 : g.shards) * g.M * (g.epi == EPI_SWIGLU ? g.N / 2 : g.N) / 4;
    long long blocks = (quads + 255) / 256;
    if (blocks > 8LL * sm_count()) blocks = 8LL * sm_count();
    splitk_reduce_k<<<(unsigned)blocks, 256, 0, st>>>(p);
    return cudaGetLastError();
}

}  // namespace

size_t tc_gemm_scratch_bytes() {
    // S * tiles <= units, so the partials never exceed one 128 x 256 fp32 tile per SM
    return (size_t)sm_count() * A_ROWS * BN * sizeof(float);
}

cudaError_t tc_gemm(const TcGemm& g, int* dev_err, void* scratch, size_t scratch_bytes, cudaStream_t st) {
    if (g.epi == EPI_SWIGLU && (g.granule != 32 || g.N % 64 != 0)) return cudaErrorNotSupported;
    cudaError_t e = set_smem_attr<false>();
    if (e == cudaSuccess) e = set_smem_attr<true>();
    if (e != cudaSuccess) return e;
    // 2-SM tiles once there is more than one 128-row block of tokens
    if (g.M > A_ROWS) {
        const int slots = pair_slots();
        if (slots > 0) return gemm_launch<true>(g, dev_err, slots, scratch, scratch_bytes, st);
    }
    return gemm_launch<false>(g, dev_err, sm_count(), scratch, scratch_bytes, st);
}

}  // namespace tpk
