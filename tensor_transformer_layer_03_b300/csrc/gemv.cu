// Weight-streaming kernels for the small-M (decode) regime, bf16, with the
// products on the CUDA cores: the one-token-row step, and 2..8 rows where
// the tensor-core streaming kernels (gemv_mma.cu) do not apply.
//
// With one to a few tokens per step every weight element is used M times, so
// the linears are bound by reading the packed weights once from HBM.  Each
// warp owns whole work items and streams two weight rows at a time with
// 16-byte non-allocating loads (16 in flight per lane); the M input rows are
// read through the read-only cache (every warp of the GPU reads the same few
// KB, so they stay in L1/L2).  Kernels are specialised on the number of token
// rows so the registers go to loads in flight, not to unused accumulators.
// The grid gives every warp the same number of items with all blocks
// resident at once.  Launches allow programmatic dependent launch: a kernel
// lets the next one start at entry and waits (griddepcontrol.wait) for the
// previous one before reading its input rows, so launch latency and block
// start-up overlap the previous kernel's tail.
//
//  * column-parallel (undercodenews.com/?p=110319, "the Original": every
//    shard multiplies the full input by its slice of the output features):
//    all shards' rows form one list; SwiGLU rows come in gate/up blocks (the
//    packing's interleave), so a warp takes a gate row and its up row and
//    writes silu(gate) * up.
//  * row-parallel with the all-reduce fused in (same section): the warp that
//    owns output feature n walks row n of every shard's weight block in
//    shard order and sums the partial dot products in registers.
#include <atomic>
#include "common.cuh"
#include "kernels.h"

namespace tpk {

namespace {

constexpr int GV_THREADS = 256;
constexpr int GV_WARPS = GV_THREADS / 32;
constexpr int GV_UNROLL = 8;  // 16-byte weight loads in flight per lane and row

__device__ __forceinline__ uint4 ld_stream(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ float dot8(const uint4& w, const uint4& x) {
    const __nv_bfloat162* a = reinterpret_cast<const __nv_bfloat162*>(&w);
    const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&x);
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 fa = __bfloat1622float2(a[i]);
        const float2 fb = __bfloat1622float2(b[i]);
        s = fmaf(fa.x, fb.x, s);
        s = fmaf(fa.y, fb.y, s);
    }
    return s;
}

// Programmatic dependent launch: let the next kernel in the stream start
// (it waits for this one before reading its outputs) / wait for the
// previous kernel's results.  No-ops when the launch did not allow it.
__device__ __forceinline__ void pdl_launch_next() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait_prev() { asm volatile("griddepcontrol.wait;" ::: "memory"); }


__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    return v;
}

// Per-lane partial dot products of one weight row (K bf16) with MT input
// rows x[m][0..K) (row stride ldx), accumulated into acc.
template <int MT>
__device__ __forceinline__ void row_dots(const bf16* __restrict__ w, const bf16* __restrict__ x, long long ldx,
                                         int K, float (&acc)[MT]) {
    const int lane = threadIdx.x % 32;
    const int nch = K / 8;
    int c = lane;
    for (; c + 32 * (GV_UNROLL - 1) < nch; c += 32 * GV_UNROLL) {
        uint4 v[GV_UNROLL];
#pragma unroll
        for (int u = 0; u < GV_UNROLL; ++u) v[u] = ld_stream(w + (c + 32 * u) * 8);
#pragma unroll
        for (int u = 0; u < GV_UNROLL; ++u) {
#pragma unroll
            for (int m = 0; m < MT; ++m)
                acc[m] += dot8(v[u], __ldg(reinterpret_cast<const uint4*>(x + m * ldx + (c + 32 * u) * 8)));
        }
    }
    for (; c < nch; c += 32) {
        const uint4 v = ld_stream(w + c * 8);
#pragma unroll
        for (int m = 0; m < MT; ++m) acc[m] += dot8(v, __ldg(reinterpret_cast<const uint4*>(x + m * ldx + c * 8)));
    }
}

// 8 bf16 (one 16-byte chunk) to fp32: element 2i is the low half of word i.
__device__ __forceinline__ void cvt8(const uint4& v, float (&f)[8]) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}

// Both rows' partial dot products with one 16-byte chunk of each: every
// weight chunk is converted once for all MT input rows, and with SAME_X
// (x0 == x1) every input chunk once for both weight rows.
template <int MT, bool SAME_X>
__device__ __forceinline__ void chunk_dots2(const uint4& a, const uint4& b, const bf16* __restrict__ x0,
                                            const bf16* __restrict__ x1, long long ldx, int off, float (&acc0)[MT],
                                            float (&acc1)[MT]) {
    float fa[8], fb[8];
    cvt8(a, fa);
    cvt8(b, fb);
#pragma unroll
    for (int m = 0; m < MT; ++m) {
        float xa[8], xb[8];
        cvt8(__ldg(reinterpret_cast<const uint4*>(x0 + m * ldx + off)), xa);
        if (SAME_X) {
#pragma unroll
            for (int j = 0; j < 8; ++j) xb[j] = xa[j];
        } else {
            cvt8(__ldg(reinterpret_cast<const uint4*>(x1 + m * ldx + off)), xb);
        }
        float s0 = 0.f, s1 = 0.f;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            s0 = fmaf(fa[j], xa[j], s0);
            s1 = fmaf(fb[j], xb[j], s1);
        }
        acc0[m] += s0;
        acc1[m] += s1;
    }
}

// The same for two weight rows at once (w0 with inputs x0, w1 with x1;
// SAME_X when x0 == x1): their loads are issued together, 2 * GV_UNROLL in
// flight per lane.
template <int MT, bool SAME_X>
__device__ __forceinline__ void row_dots2(const bf16* __restrict__ w0, const bf16* __restrict__ x0,
                                          const bf16* __restrict__ w1, const bf16* __restrict__ x1, long long ldx,
                                          int K, float (&acc0)[MT], float (&acc1)[MT]) {
    const int lane = threadIdx.x % 32;
    const int nch = K / 8;
    int c = lane;
    for (; c + 32 * (GV_UNROLL - 1) < nch; c += 32 * GV_UNROLL) {
        uint4 v0[GV_UNROLL], v1[GV_UNROLL];
#pragma unroll
        for (int u = 0; u < GV_UNROLL; ++u) {
            v0[u] = ld_stream(w0 + (c + 32 * u) * 8);
            v1[u] = ld_stream(w1 + (c + 32 * u) * 8);
        }
#pragma unroll
        for (int u = 0; u < GV_UNROLL; ++u)
            chunk_dots2<MT, SAME_X>(v0[u], v1[u], x0, x1, ldx, (c + 32 * u) * 8, acc0, acc1);
    }
    for (; c < nch; c += 32)
        chunk_dots2<MT, SAME_X>(ld_stream(w0 + c * 8), ld_stream(w1 + c * 8), x0, x1, ldx, c * 8, acc0, acc1);
}

template <int MT, int EPI>
__global__ void __launch_bounds__(GV_THREADS) gemv_col_k(GemvArgs g) {
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int gw = blockIdx.x * GV_WARPS + warp, nw = gridDim.x * GV_WARPS;
    const bf16* W = (const bf16*)g.W;
    const bf16* X = (const bf16*)g.A;
    pdl_launch_next();
    pdl_wait_prev();
    if (EPI == EPI_SWIGLU) {
        const int n_out = g.N / 2;  // U columns per shard
        const int items = g.shards * n_out;
        for (int it = gw; it < items; it += nw) {
            const int s = it / n_out, j = it % n_out;
            const int grp = j / g.granule, w = j % g.granule;
            const long long gate_row = (long long)s * g.N + grp * 2 * g.granule + w;
            float ag[MT], au[MT];
#pragma unroll
            for (int m = 0; m < MT; ++m) ag[m] = au[m] = 0.f;
            row_dots2<MT, true>(W + gate_row * g.K, X, W + (gate_row + g.granule) * g.K, X, g.lda, g.K, ag, au);
#pragma unroll
            for (int m = 0; m < MT; ++m) {
                const float rs = g.row_scale ? g.row_scale[m] : 1.f;  // pre-norm: 1/rms of input row m
                const float gs = warp_sum(ag[m]) * rs, us = warp_sum(au[m]) * rs;
                if (lane == 0)
                    ((bf16*)g.out)[s * g.out_shard + (long long)m * g.ldo + j] = __float2bfloat16_rn(silu(gs) * us);
            }
        }
    } else if (g.rope_cols > 0) {
        // rotary embedding rotates output pairs (2i, 2i+1): a warp takes the
        // adjacent items 2k, 2k+1 (N is even, so a pair never straddles shards)
        const int pairs = g.shards * g.N / 2;
        for (int k = gw; k < pairs; k += nw) {
            const int it = 2 * k;
            float acc[2][MT];
#pragma unroll
            for (int m = 0; m < MT; ++m) acc[0][m] = acc[1][m] = 0.f;
            row_dots2<MT, true>(W + (long long)it * g.K, X, W + (long long)(it + 1) * g.K, X, g.lda, g.K, acc[0], acc[1]);
            const int s = it / g.N, n = it % g.N;
#pragma unroll
            for (int m = 0; m < MT; ++m) {
                const float rs = g.row_scale ? g.row_scale[m] : 1.f;
                float a = warp_sum(acc[0][m]) * rs, b = warp_sum(acc[1][m]) * rs;
                if (n < g.rope_cols) {
                    const float2 c =
                        g.rope_cs[(long long)(m % (g.rope_seq > 0 ? g.rope_seq : 1)) * (g.rope_dh / 2) +
                                  (n % g.rope_dh) / 2];
                    const float a2 = a * c.x - b * c.y;
                    b = a * c.y + b * c.x;
                    a = a2;
                }
                if (lane == 0) {
                    bf16* o = (bf16*)g.out + s * g.out_shard + (long long)m * g.ldo + n;
                    o[0] = __float2bfloat16_rn(a);
                    o[1] = __float2bfloat16_rn(b);
                }
            }
        }
    } else {
        // items it and it + nw together (two rows' loads in flight)
        const int items = g.shards * g.N;
        for (int it = gw; it < items; it += 2 * nw) {
            const int it2 = it + nw;
            float acc[2][MT];
#pragma unroll
            for (int m = 0; m < MT; ++m) acc[0][m] = acc[1][m] = 0.f;
            if (it2 < items)
                row_dots2<MT, true>(W + (long long)it * g.K, X, W + (long long)it2 * g.K, X, g.lda, g.K, acc[0], acc[1]);
            else
                row_dots<MT>(W + (long long)it * g.K, X, g.lda, g.K, acc[0]);
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                const int itr = r ? it2 : it;
                if (itr >= items) break;
                const int s = itr / g.N, n = itr % g.N;
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                    float v = warp_sum(acc[r][m]);
                    if (g.row_scale) v *= g.row_scale[m];
                    if (EPI == EPI_GELU) v = gelu_erf(v);
                    if (lane == 0) ((bf16*)g.out)[s * g.out_shard + (long long)m * g.ldo + n] = __float2bfloat16_rn(v);
                }
            }
        }
    }
}

// row-parallel: out[m][n] = residual + sum_s <A_s[m][:], W_s[n][:]>
template <int MT>
__device__ __forceinline__ void row_store(const GemvArgs& g, int n, float (&acc)[MT]) {
    const int lane = threadIdx.x % 32;
#pragma unroll
    for (int m = 0; m < MT; ++m) {
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

// Row-parallel: a warp owns output features n and n + nw and walks row n
// and row n + nw of every shard's weight block in shard order (the fused
// all-reduce), both rows reading the same shard input.
template <int MT>
__global__ void __launch_bounds__(GV_THREADS) gemv_row_k(GemvArgs g) {
    const int warp = threadIdx.x / 32;
    const int gw = blockIdx.x * GV_WARPS + warp, nw = gridDim.x * GV_WARPS;
    const bf16* W = (const bf16*)g.W;
    const bf16* A = (const bf16*)g.A;
    pdl_launch_next();
    pdl_wait_prev();
    for (int n = gw; n < g.N; n += 2 * nw) {
        const int n2 = n + nw;
        float acc[MT], acc2[MT];
#pragma unroll
        for (int m = 0; m < MT; ++m) acc[m] = acc2[m] = 0.f;
        for (int s = 0; s < g.shards; ++s) {
            const bf16* Ws = W + s * g.w_shard;
            const bf16* As = A + s * g.a_shard;
            float p[MT], p2[MT];
#pragma unroll
            for (int m = 0; m < MT; ++m) p[m] = p2[m] = 0.f;
            if (n2 < g.N)
                row_dots2<MT, true>(Ws + (long long)n * g.K, As, Ws + (long long)n2 * g.K, As, g.lda, g.K, p, p2);
            else
                row_dots<MT>(Ws + (long long)n * g.K, As, g.lda, g.K, p);
#pragma unroll
            for (int m = 0; m < MT; ++m) {
                acc[m] += p[m];
                acc2[m] += p2[m];
            }
        }
        row_store<MT>(g, n, acc);
        if (n2 < g.N) row_store<MT>(g, n2, acc2);
    }
}

int sm_count_dev() {
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

// Grid: every warp gets the same number of items (ceil(items / warps)),
// with all blocks resident at once, so no partial second wave trails.
// Launched with programmatic dependent launch allowed.
template <int MT>
cudaError_t gemv_launch(const GemvArgs& g, cudaStream_t st) {
    const int items = g.reduce ? g.N : g.shards * (g.epi == EPI_SWIGLU ? g.N / 2 : g.N);
    void (*kern)(GemvArgs) = g.reduce ? gemv_row_k<MT>
                             : g.epi == EPI_SWIGLU ? gemv_col_k<MT, EPI_SWIGLU>
                             : g.epi == EPI_GELU   ? gemv_col_k<MT, EPI_GELU>
                                                   : gemv_col_k<MT, EPI_STORE>;
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, GV_THREADS, 0) != cudaSuccess || per_sm < 1) {
        cudaGetLastError();
        per_sm = 1;
    }
    const int resident_warps = sm_count_dev() * per_sm * GV_WARPS;
    const int per_warp = (items + resident_warps - 1) / resident_warps;
    const int warps = (items + per_warp - 1) / per_warp;
    const int blocks = (warps + GV_WARPS - 1) / GV_WARPS;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3(blocks > 0 ? blocks : 1);
    cfg.blockDim = dim3(GV_THREADS);
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, g);
}

}  // namespace

bool gemv_supported(const GemvArgs& g) {
    return g.M >= 1 && g.M <= GEMV_MAX_M && g.K % 8 == 0 && g.lda % 8 == 0 &&
           (g.epi != EPI_SWIGLU || (g.N % (2 * g.granule) == 0));
}

cudaError_t gemv(const GemvArgs& g, int* /*dev_err: no bounded waits here*/, cudaStream_t st) {
    switch (g.M) {
        case 1: return gemv_launch<1>(g, st);
        case 2: return gemv_launch<2>(g, st);
        case 3: return gemv_launch<3>(g, st);
        case 4: return gemv_launch<4>(g, st);
        case 5: return gemv_launch<5>(g, st);
        case 6: return gemv_launch<6>(g, st);
        case 7: return gemv_launch<7>(g, st);
        default: return gemv_launch<8>(g, st);
    }
}

}  // namespace tpk
