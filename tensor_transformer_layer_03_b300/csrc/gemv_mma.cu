// Weight streaming for 2..32 token rows with the products on the tensor
// cores (the batched one-token decode step).
//
// At a handful of rows the linears still read every weight byte once and
// are bound by HBM, but a CUDA-core loop pays a bf16 -> fp32 conversion and
// 8 FMAs per row for every 16 bytes of weights, which at 4..8 rows costs
// more issue slots than the bandwidth leaves.  Here one warp-wide
// mma.m16n8k16 (bf16 in, fp32 accumulate) takes 16 weight rows x 16 k
// against up to 8 token rows, so a 32-wide k-block of 16 rows (1 KB of
// weights) costs two 16-byte loads and two MMAs per lane whatever the row
// count.  The operands go from the load registers straight into the MMA:
// the dot product is a sum over k, so A and B only have to agree on which
// memory element sits in which k slot; lane (g, c) loads elements
// [8c, 8c + 8) of weight rows g and g + 8 and of token row g, and the first
// four of them fill its slots {2c, 2c+1, 2c+8, 2c+9} of one MMA, the last
// four those of the second.  Above 8 token rows the same weight registers
// meet NT = 2 or 4 groups of 8 token rows (lane (g, c) also loads token
// rows g + 8, g + 16, ...): the weight stream, which is what costs, is read
// once whatever the row count.
//
// Layout of the work (as in the other linears: undercodenews.com/?p=110319,
// "the Original"): a block owns 16 output rows of one shard (column-
// parallel; for SwiGLU 16 gate rows and the 16 matching up rows) or 16
// output features (row-parallel, summed over all shards: the fused
// all-reduce); its S warps split the k range (row-parallel: shard-major),
// and warp 0 adds their partial tiles in warp order through shared memory
// and runs the epilogue.  Launched with programmatic dependent launch.
#include <atomic>
#include "common.cuh"
#include "kernels.h"

namespace tpk {

namespace {

constexpr int MU = 4;         // 32-wide k-blocks in flight per lane
constexpr int MMA_MAX_WARPS = 8;

__device__ __forceinline__ uint4 ld_stream16(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// One 32-wide k-block: lo / hi = elements [8c, 8c+8) of weight rows g and
// g + 8, x = the same elements of token row g (A fragment: a0 row g, a1 row
// g+8 at slots 2c..2c+1, a2 / a3 at slots 2c+8..2c+9; B fragment: b0 slots
// 2c..2c+1, b1 slots 2c+8..2c+9 of column g).
__device__ __forceinline__ void kblock(float (&d)[4], const uint4& lo, const uint4& hi, const uint4& x) {
    mma_bf16_16816(d, lo.x, hi.x, lo.y, hi.y, x.x, x.y);
    mma_bf16_16816(d, lo.z, hi.z, lo.w, hi.w, x.z, x.w);
}

// d[r][t] += rows [0, 16) of group r (w0: group 0, w1: group 1; row stride
// ldw) times token rows [8t, 8t + 8) of x (stride ldx; rows >= M count as
// zero) over the k-blocks [kb0, kb1).  Accumulator element j of lane
// (g, c) in d[r][t]: row g + 8 * (j / 2), token 8t + 2c + j % 2.
template <int NR, int NT>
__device__ __forceinline__ void mma_dot(float (&d)[NR][NT][4], const bf16* __restrict__ w0,
                                        const bf16* __restrict__ w1, long long ldw, const bf16* __restrict__ x,
                                        long long ldx, int M, int kb0, int kb1) {
    // k-blocks per batch: the loads of batch j + 1 are issued before batch
    // j's MMAs, so two batches are in flight per lane (software pipeline;
    // the weight stream is latency-bound with only ~20 warps per SM); fewer
    // per batch with more token groups (registers)
    constexpr int U = NT == 1 ? (NR == 2 ? 2 : MU) : (NT == 2 ? 2 : 1);
    const int lane = threadIdx.x & 31, g = lane >> 2, c = lane & 3;
    bool xv[NT];
    const bf16* xr[NT];
#pragma unroll
    for (int t = 0; t < NT; ++t) {
        xv[t] = g + 8 * t < M;
        xr[t] = x + (xv[t] ? (long long)(g + 8 * t) * ldx : 0) + 8 * c;
    }
    const bf16* wl[NR];
    wl[0] = w0 + (long long)g * ldw + 8 * c;
    if (NR > 1) wl[NR - 1] = w1 + (long long)g * ldw + 8 * c;
    const long long hi_off = 8 * ldw;
    struct Batch {
        uint4 lo[NR][U], hi[NR][U], xx[NT][U];
    };
    auto load = [&](Batch& b, int kb) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
#pragma unroll
            for (int r = 0; r < NR; ++r) {
                b.lo[r][u] = ld_stream16(wl[r] + (kb + u) * 32);
                b.hi[r][u] = ld_stream16(wl[r] + hi_off + (kb + u) * 32);
            }
        }
#pragma unroll
        for (int t = 0; t < NT; ++t)
#pragma unroll
            for (int u = 0; u < U; ++u)
                b.xx[t][u] = xv[t] ? __ldg(reinterpret_cast<const uint4*>(xr[t] + (kb + u) * 32)) : make_uint4(0, 0, 0, 0);
    };
    auto mma = [&](const Batch& b) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
#pragma unroll
            for (int r = 0; r < NR; ++r)
#pragma unroll
                for (int t = 0; t < NT; ++t) kblock(d[r][t], b.lo[r][u], b.hi[r][u], b.xx[t][u]);
        }
    };
    int kb = kb0;
    if (kb + U <= kb1) {
        Batch cur, nxt;
        load(cur, kb);
        kb += U;
        for (; kb + U <= kb1; kb += U) {
            load(nxt, kb);
            mma(cur);
            cur = nxt;
        }
        mma(cur);
    }
    for (; kb < kb1; ++kb) {
        uint4 xx[NT];
#pragma unroll
        for (int t = 0; t < NT; ++t)
            xx[t] = xv[t] ? __ldg(reinterpret_cast<const uint4*>(xr[t] + kb * 32)) : make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int r = 0; r < NR; ++r) {
            const uint4 lo = ld_stream16(wl[r] + kb * 32), hi = ld_stream16(wl[r] + hi_off + kb * 32);
#pragma unroll
            for (int t = 0; t < NT; ++t) kblock(d[r][t], lo, hi, xx[t]);
        }
    }
}

// Warp 0 receives the sum of the S warps' tiles, added in warp order.
// Returns false in the other warps (which then leave).
template <int NR, int NT>
__device__ __forceinline__ bool reduce_warps(float (&d)[NR][NT][4], int S) {
    __shared__ float red[MMA_MAX_WARPS][NR * NT][4][32];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (S == 1) return true;
#pragma unroll
    for (int r = 0; r < NR; ++r)
#pragma unroll
        for (int t = 0; t < NT; ++t)
#pragma unroll
            for (int j = 0; j < 4; ++j) red[warp][r * NT + t][j][lane] = d[r][t][j];
    __syncthreads();
    if (warp != 0) return false;
#pragma unroll
    for (int r = 0; r < NR; ++r)
#pragma unroll
        for (int t = 0; t < NT; ++t)
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                float v = red[0][r * NT + t][j][lane];
                for (int w = 1; w < S; ++w) v += red[w][r * NT + t][j][lane];
                d[r][t][j] = v;
            }
    return true;
}

__device__ __forceinline__ void pdl_entry() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// STORE / GELU epilogue of gemv_mma_col_k (warp 0): row scale, rotary
// embedding of the Q and K columns, activation, bf16 store.
template <int EPI>
__device__ __forceinline__ void store_rows(const GemvArgs& g, const float (&d)[4], bf16* out, int n0, int mbase,
                                           float rs0, float rs1) {
    const int lane = threadIdx.x & 31, gq = lane >> 2, m0 = mbase + 2 * (lane & 3);
    float v[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) v[j] = d[j] * ((j & 1) ? rs1 : rs0);
    if (g.rope_cols > 0) {
        // rows 2i and 2i+1 sit in lanes gq and gq ^ 1 (lane ^ 4), same tokens
        float p[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) p[j] = __shfl_xor_sync(0xffffffffu, v[j], 4);
        const bool odd = gq & 1;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int n = n0 + gq + 8 * (j >> 1), m = m0 + (j & 1);
            if (n < g.rope_cols && m < g.M) {
                const float2 cs =
                    g.rope_cs[(long long)(m % (g.rope_seq > 0 ? g.rope_seq : 1)) * (g.rope_dh / 2) + (n % g.rope_dh) / 2];
                v[j] = odd ? p[j] * cs.y + v[j] * cs.x : v[j] * cs.x - p[j] * cs.y;
            }
        }
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int n = n0 + gq + 8 * (j >> 1), m = m0 + (j & 1);
        float o = v[j];
        if (EPI == EPI_GELU) o = gelu_erf(o);
        if (m < g.M) out[(long long)m * g.ldo + n] = __float2bfloat16_rn(o);
    }
}

// Column-parallel: block b = 16 rows of one shard (STORE / GELU, with the
// optional row scale and rotary embedding) or 16 gate rows + their 16 up
// rows (SwiGLU).
template <int EPI, int NT>
__global__ void __launch_bounds__(MMA_MAX_WARPS * 32) gemv_mma_col_k(GemvArgs g, int S) {
    constexpr int NR = EPI == EPI_SWIGLU ? 2 : 1;
    pdl_entry();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, gq = lane >> 2, c = lane & 3;
    int s, n0;
    if (EPI == EPI_SWIGLU) {
        const int per_shard = g.N / 32, gpb = g.granule / 16;
        s = blockIdx.x / per_shard;
        const int q = blockIdx.x % per_shard;
        n0 = (q / gpb) * 2 * g.granule + (q % gpb) * 16;  // first gate row; its up rows start granule later
    } else {
        const int per_shard = g.N / 16;
        s = blockIdx.x / per_shard;
        n0 = (blockIdx.x % per_shard) * 16;
    }
    const bf16* W = (const bf16*)g.W + s * g.w_shard + (long long)n0 * g.K;
    const int nkb = g.K / 32;
    float d[NR][NT][4];
#pragma unroll
    for (int r = 0; r < NR; ++r)
#pragma unroll
        for (int t = 0; t < NT; ++t)
#pragma unroll
            for (int j = 0; j < 4; ++j) d[r][t][j] = 0.f;
    mma_dot<NR, NT>(d, W, W + (long long)g.granule * g.K, g.K, (const bf16*)g.A, g.lda, g.M, warp * nkb / S,
                    (warp + 1) * nkb / S);
    if (!reduce_warps<NR, NT>(d, S)) return;
    bf16* out = (bf16*)g.out + s * g.out_shard;
#pragma unroll
    for (int t = 0; t < NT; ++t) {
        const int m0 = 8 * t + 2 * c;
        const float rs0 = g.row_scale && m0 < g.M ? g.row_scale[m0] : 1.f;
        const float rs1 = g.row_scale && m0 + 1 < g.M ? g.row_scale[m0 + 1] : 1.f;
        if constexpr (EPI == EPI_SWIGLU) {
            const int col0 = (n0 / (2 * g.granule)) * g.granule + n0 % (2 * g.granule) + gq;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int m = m0 + (j & 1), col = col0 + 8 * (j >> 1);
                const float rs = (j & 1) ? rs1 : rs0;
                if (m < g.M)
                    out[(long long)m * g.ldo + col] =
                        __float2bfloat16_rn(silu(d[0][t][j] * rs) * (d[NR - 1][t][j] * rs));
            }
        } else {
            store_rows<EPI>(g, d[0][t], out, n0, 8 * t, rs0, rs1);
        }
    }
}

// Row-parallel with the fused all-reduce: block b = output features
// [16b, 16b + 16); warp w takes shard w / Sk and the (w % Sk)-th part of
// its k range, so the warp-order sum is shard-major.
template <int NT>
__global__ void __launch_bounds__(MMA_MAX_WARPS * 32) gemv_mma_row_k(GemvArgs g, int Sk) {
    pdl_entry();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, gq = lane >> 2, c = lane & 3;
    const int S = g.shards * Sk;
    const int s = warp / Sk, part = warp % Sk;
    const int n0 = blockIdx.x * 16;
    const int nkb = g.K / 32;
    float d[1][NT][4];
#pragma unroll
    for (int t = 0; t < NT; ++t)
#pragma unroll
        for (int j = 0; j < 4; ++j) d[0][t][j] = 0.f;
    const bf16* W = (const bf16*)g.W + s * g.w_shard + (long long)n0 * g.K;
    mma_dot<1, NT>(d, W, W, g.K, (const bf16*)g.A + s * g.a_shard, g.lda, g.M, part * nkb / Sk,
                   (part + 1) * nkb / Sk);
    if (!reduce_warps<1, NT>(d, S)) return;
#pragma unroll
    for (int t = 0; t < NT; ++t)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int n = n0 + gq + 8 * (j >> 1), m = 8 * t + 2 * c + (j & 1);
            if (m >= g.M) continue;
            const long long o = (long long)m * g.ldo + n;
            float v = d[0][t][j];
            if (g.residual)
                v += g.residual_f32 ? ((const float*)g.residual)[o] : __bfloat162float(((const bf16*)g.residual)[o]);
            ((float*)g.out)[o] = v;
            if (g.out2) ((bf16*)g.out2)[o] = __float2bfloat16_rn(v);
        }
}

int sm_count_mma() {
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

cudaError_t launch(void (*kern)(GemvArgs, int), int blocks, int warps, cudaStream_t st, const GemvArgs& g, int arg) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3(blocks);
    cfg.blockDim = dim3(warps * 32);
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, g, arg);
}

}  // namespace

bool gemv_mma_supported(const GemvArgs& g) {
    if (g.M < 2 || g.M > GEMV_MMA_MAX_ROWS || g.K % 32 != 0 || g.lda % 8 != 0 || g.N % 16 != 0 || g.shards < 1) return false;
    if (g.reduce) return g.epi == EPI_ROW_REDUCE && g.shards <= MMA_MAX_WARPS;
    if (g.epi == EPI_SWIGLU) return g.granule % 16 == 0 && g.N % (2 * g.granule) == 0;
    return g.epi == EPI_STORE || g.epi == EPI_GELU;
}

namespace {

template <int NT>
cudaError_t gemv_mma_nt(const GemvArgs& g, cudaStream_t st) {
    const int nkb = g.K / 32;
    const int target_warps = sm_count_mma() * 16;  // enough 16-byte loads in flight to cover HBM latency
    if (g.reduce) {
        int Sk = MMA_MAX_WARPS / g.shards;
        if (Sk < 1) Sk = 1;
        if (Sk > nkb) Sk = nkb;
        return launch(gemv_mma_row_k<NT>, g.N / 16, g.shards * Sk, st, g, Sk);
    }
    const int blocks = g.shards * (g.epi == EPI_SWIGLU ? g.N / 32 : g.N / 16);
    int S = (target_warps + blocks - 1) / blocks;
    if (S > MMA_MAX_WARPS) S = MMA_MAX_WARPS;
    if (S > nkb) S = nkb;
    if (S < 1) S = 1;
    void (*kern)(GemvArgs, int) = g.epi == EPI_SWIGLU ? gemv_mma_col_k<EPI_SWIGLU, NT>
                                  : g.epi == EPI_GELU ? gemv_mma_col_k<EPI_GELU, NT>
                                                      : gemv_mma_col_k<EPI_STORE, NT>;
    return launch(kern, blocks, S, st, g, S);
}

}  // namespace

cudaError_t gemv_mma(const GemvArgs& g, cudaStream_t st) {
    if (g.M <= 8) return gemv_mma_nt<1>(g, st);
    if (g.M <= 16) return gemv_mma_nt<2>(g, st);
    return gemv_mma_nt<4>(g, st);
}

}  // namespace tpk
