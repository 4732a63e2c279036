// Weight-streaming kernels for the small-M (decode) regime, bf16.
//
// With one to a few tokens per step every weight element is used M times, so
// the linears are bound by reading the packed weights once from HBM.  Each
// warp owns whole weight rows and streams them with 16-byte non-allocating
// loads (four in flight per lane); the M input rows sit in shared memory.
//
//  * column-parallel (undercodenews.com/?p=110319, "the Original": every
//    shard multiplies the full input by its slice of the output features):
//    all shards' rows form one list; SwiGLU rows come in gate/up blocks of 32
//    (the packing's interleave), so a warp takes a gate row and its up row
//    and writes silu(gate) * up.
//  * row-parallel with the all-reduce fused in (same section): the warp that
//    owns output feature n walks row n of every shard's weight block in
//    shard order and sums the partial dot products in registers.
#include "common.cuh"
#include "kernels.h"

namespace tpk {

namespace {

constexpr int GV_THREADS = 256;
constexpr int GV_WARPS = GV_THREADS / 32;

__device__ __forceinline__ uint4 ld_stream(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ void bf16x8_to_f32(const uint4& v, float (&f)[8]) {
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 t = __bfloat1622float2(h[i]);
        f[2 * i] = t.x;
        f[2 * i + 1] = t.y;
    }
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    return v;
}

// dot products of one weight row (K bf16, 16-byte aligned) with M input rows
// held in shared memory as fp32 [M][K]; partial sums per lane.
template <int MAXM>
__device__ __forceinline__ void row_dots(const bf16* w, const float* xs, int K, int M, float (&acc)[MAXM]) {
    const int lane = threadIdx.x % 32;
    const int nch = K / 8;
    int c = lane;
    for (; c + 96 < nch; c += 128) {
        uint4 v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) v[u] = ld_stream(w + (c + 32 * u) * 8);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            float f[8];
            bf16x8_to_f32(v[u], f);
            const int k = (c + 32 * u) * 8;
#pragma unroll
            for (int m = 0; m < MAXM; ++m) {
                if (m < M) {
                    const float4 x0 = *reinterpret_cast<const float4*>(xs + m * K + k);
                    const float4 x1 = *reinterpret_cast<const float4*>(xs + m * K + k + 4);
                    acc[m] += f[0] * x0.x + f[1] * x0.y + f[2] * x0.z + f[3] * x0.w + f[4] * x1.x + f[5] * x1.y +
                              f[6] * x1.z + f[7] * x1.w;
                }
            }
        }
    }
    for (; c < nch; c += 32) {
        const uint4 v = ld_stream(w + c * 8);
        float f[8];
        bf16x8_to_f32(v, f);
        const int k = c * 8;
#pragma unroll
        for (int m = 0; m < MAXM; ++m) {
            if (m < M) {
                const float4 x0 = *reinterpret_cast<const float4*>(xs + m * K + k);
                const float4 x1 = *reinterpret_cast<const float4*>(xs + m * K + k + 4);
                acc[m] += f[0] * x0.x + f[1] * x0.y + f[2] * x0.z + f[3] * x0.w + f[4] * x1.x + f[5] * x1.y +
                          f[6] * x1.z + f[7] * x1.w;
            }
        }
    }
}

// x [M][K] bf16 (row stride lda) -> shared fp32 [M][K]
__device__ __forceinline__ void stage_input(float* xs, const bf16* x, int M, int K, long long lda) {
    for (int i = threadIdx.x; i < M * (K / 8); i += GV_THREADS) {
        const int m = i / (K / 8), c = i % (K / 8);
        const uint4 v = *reinterpret_cast<const uint4*>(x + m * lda + c * 8);
        float f[8];
        bf16x8_to_f32(v, f);
        float4* d = reinterpret_cast<float4*>(xs + m * K + c * 8);
        d[0] = make_float4(f[0], f[1], f[2], f[3]);
        d[1] = make_float4(f[4], f[5], f[6], f[7]);
    }
    __syncthreads();
}

template <int MAXM, int EPI>
__global__ void __launch_bounds__(GV_THREADS) gemv_col_k(GemvArgs g) {
    extern __shared__ __align__(16) float gv_xs[];
    stage_input(gv_xs, (const bf16*)g.A, g.M, g.K, g.lda);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int gw = blockIdx.x * GV_WARPS + warp, nw = gridDim.x * GV_WARPS;
    const bf16* W = (const bf16*)g.W;
    if (EPI == EPI_SWIGLU) {
        // work item = one output column of U: gate row and up row of its group
        const int n_out = g.N / 2;  // per shard
        const int items = g.shards * n_out;
        for (int it = gw; it < items; it += nw) {
            const int s = it / n_out, j = it % n_out;
            const int grp = j / g.granule, w = j % g.granule;
            const long long gate_row = (long long)s * g.N + grp * 2 * g.granule + w;
            float ag[MAXM], au[MAXM];
#pragma unroll
            for (int m = 0; m < MAXM; ++m) ag[m] = au[m] = 0.f;
            row_dots<MAXM>(W + gate_row * g.K, gv_xs, g.K, g.M, ag);
            row_dots<MAXM>(W + (gate_row + g.granule) * g.K, gv_xs, g.K, g.M, au);
#pragma unroll
            for (int m = 0; m < MAXM; ++m) {
                if (m < g.M) {
                    const float gs = warp_sum(ag[m]), us = warp_sum(au[m]);
                    if (lane == 0)
                        ((bf16*)g.out)[s * g.out_shard + (long long)m * g.ldo + j] = __float2bfloat16_rn(silu(gs) * us);
                }
            }
        }
    } else {
        const int items = g.shards * g.N;
        for (int it = gw; it < items; it += nw) {
            const int s = it / g.N, n = it % g.N;
            float acc[MAXM];
#pragma unroll
            for (int m = 0; m < MAXM; ++m) acc[m] = 0.f;
            row_dots<MAXM>(W + (long long)it * g.K, gv_xs, g.K, g.M, acc);
#pragma unroll
            for (int m = 0; m < MAXM; ++m) {
                if (m < g.M) {
                    float v = warp_sum(acc[m]);
                    if (EPI == EPI_GELU) v = gelu_erf(v);
                    if (lane == 0) ((bf16*)g.out)[s * g.out_shard + (long long)m * g.ldo + n] = __float2bfloat16_rn(v);
                }
            }
        }
    }
}

// row-parallel: out[m][n] = residual + sum_s <A_s[m][:], W_s[n][:]>
template <int MAXM>
__global__ void __launch_bounds__(GV_THREADS) gemv_row_k(GemvArgs g) {
    extern __shared__ __align__(16) float gv_xs[];
    // stage all shards' inputs: [shard][M][K]
    for (int s = 0; s < g.shards; ++s) {
        const bf16* a = (const bf16*)g.A + s * g.a_shard;
        for (int i = threadIdx.x; i < g.M * (g.K / 8); i += GV_THREADS) {
            const int m = i / (g.K / 8), c = i % (g.K / 8);
            const uint4 v = *reinterpret_cast<const uint4*>(a + m * (long long)g.lda + c * 8);
            float f[8];
            bf16x8_to_f32(v, f);
            float4* d = reinterpret_cast<float4*>(gv_xs + ((long long)s * g.M + m) * g.K + c * 8);
            d[0] = make_float4(f[0], f[1], f[2], f[3]);
            d[1] = make_float4(f[4], f[5], f[6], f[7]);
        }
    }
    __syncthreads();
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int gw = blockIdx.x * GV_WARPS + warp, nw = gridDim.x * GV_WARPS;
    const bf16* W = (const bf16*)g.W;
    for (int n = gw; n < g.N; n += nw) {
        float acc[MAXM];
#pragma unroll
        for (int m = 0; m < MAXM; ++m) acc[m] = 0.f;
        for (int s = 0; s < g.shards; ++s)  // shard order: the fused all-reduce
            row_dots<MAXM>(W + s * g.w_shard + (long long)n * g.K, gv_xs + (long long)s * g.M * g.K, g.K, g.M, acc);
#pragma unroll
        for (int m = 0; m < MAXM; ++m) {
            if (m < g.M) {
                float v = warp_sum(acc[m]);
                if (lane == 0) {
                    const long long o = (long long)m * g.ldo + n;
                    if (g.residual)
                        v += g.residual_f32 ? ((const float*)g.residual)[o] : __bfloat162float(((const bf16*)g.residual)[o]);
                    ((float*)g.out)[o] = v;
                    if (g.out2) ((bf16*)g.out2)[o] = __float2bfloat16_rn(v);
                }
            }
        }
    }
}

int sm_count_dev() {
    static int n[64] = {0};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) return 148;
    if (!n[dev]) cudaDeviceGetAttribute(&n[dev], cudaDevAttrMultiProcessorCount, dev);
    return n[dev] > 0 ? n[dev] : 148;
}

template <typename K>
cudaError_t set_smem(K kernel, size_t bytes, bool& done) {
    if (done) return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (e == cudaSuccess) done = true;
    return e;
}

}  // namespace

size_t gemv_smem_bytes(const GemvArgs& g) {
    return (size_t)(g.reduce ? g.shards : 1) * g.M * g.K * sizeof(float);
}

bool gemv_supported(const GemvArgs& g) {
    return g.M >= 1 && g.M <= GEMV_MAX_M && g.K % 8 == 0 && g.lda % 8 == 0 && gemv_smem_bytes(g) <= 200 * 1024 &&
           (g.epi != EPI_SWIGLU || (g.N % (2 * g.granule) == 0));
}

cudaError_t gemv(const GemvArgs& g, cudaStream_t st) {
    const size_t smem = gemv_smem_bytes(g);
    const int items = g.reduce ? g.N : g.shards * (g.epi == EPI_SWIGLU ? g.N / 2 : g.N);
    int blocks = (items + GV_WARPS - 1) / GV_WARPS;
    const int cap = sm_count_dev() * 8;
    if (blocks > cap) blocks = cap;
    static bool a0 = false, a1 = false, a2 = false, a3 = false;
    cudaError_t e;
    if (g.reduce) {
        if ((e = set_smem(gemv_row_k<GEMV_MAX_M>, 200 * 1024, a0)) != cudaSuccess) return e;
        gemv_row_k<GEMV_MAX_M><<<blocks, GV_THREADS, smem, st>>>(g);
    } else if (g.epi == EPI_SWIGLU) {
        if ((e = set_smem(gemv_col_k<GEMV_MAX_M, EPI_SWIGLU>, 200 * 1024, a1)) != cudaSuccess) return e;
        gemv_col_k<GEMV_MAX_M, EPI_SWIGLU><<<blocks, GV_THREADS, smem, st>>>(g);
    } else if (g.epi == EPI_GELU) {
        if ((e = set_smem(gemv_col_k<GEMV_MAX_M, EPI_GELU>, 200 * 1024, a2)) != cudaSuccess) return e;
        gemv_col_k<GEMV_MAX_M, EPI_GELU><<<blocks, GV_THREADS, smem, st>>>(g);
    } else {
        if ((e = set_smem(gemv_col_k<GEMV_MAX_M, EPI_STORE>, 200 * 1024, a3)) != cudaSuccess) return e;
        gemv_col_k<GEMV_MAX_M, EPI_STORE><<<blocks, GV_THREADS, smem, st>>>(g);
    }
    return cudaGetLastError();
}

}  // namespace tpk
