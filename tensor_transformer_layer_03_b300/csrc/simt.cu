// CUDA-core (SIMT) kernels: the fp32 path of every step, and the path for
// shapes the tensor-core kernels do not take.
//
//  * simt_gemm: shared-memory tiled GEMM, 64x64 output tile per 256-thread
//    block, fp32 accumulate.  Column-parallel launches put one shard per
//    grid.z slice; row-parallel launches loop over the shards inside the
//    block and keep one accumulator, so the all-reduce of the partials
//    happens in registers (undercodenews.com/?p=110319, "the Original").
//  * simt_attention: one block per (16 queries, head, sequence); K/V tiles of
//    32 keys staged in shared memory; one warp per query row with an online
//    softmax (warp-shuffle row max and row sum).
#include <math.h>

#include "common.cuh"
#include "kernels.h"

namespace tpk {

namespace {

constexpr int BM = 64, BN = 64, BK = 16;

template <typename T, int EPI>
__global__ void __launch_bounds__(256) simt_gemm_k(SimtGemm g, int granule) {
    __shared__ float As[BK][BM + 4];
    __shared__ float Ws[BK][BN + 4];
    __shared__ float Cs[BM][BN + 1];
    const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
    const int m0 = blockIdx.y * BM, n0 = blockIdx.x * BN, cs = blockIdx.z;
    const T* A = (const T*)g.A + cs * g.a_shard;
    const T* W = (const T*)g.W + cs * g.w_shard;
    float acc[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;

    for (int rs = 0; rs < g.red_shards; ++rs) {
        const T* Ar = A + rs * g.a_shard;
        const T* Wr = W + rs * g.w_shard;
        for (int k0 = 0; k0 < g.K; k0 += BK) {
            for (int i = threadIdx.x; i < BM * BK; i += 256) {
                const int r = i / BK, kk = i % BK, k = k0 + kk;
                const int m = m0 + r, n = n0 + r;
                As[kk][r] = (m < g.M && k < g.K) ? to_f(Ar[(long long)m * g.lda + k]) : 0.f;
                Ws[kk][r] = (n < g.N && k < g.K) ? to_f(Wr[(long long)n * g.ldw + k]) : 0.f;
            }
            __syncthreads();
#pragma unroll
            for (int kk = 0; kk < BK; ++kk) {
                float a[4], b[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) a[i] = As[kk][ty + 16 * i];
#pragma unroll
                for (int j = 0; j < 4; ++j) b[j] = Ws[kk][tx + 16 * j];
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
            }
            __syncthreads();
        }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) Cs[ty + 16 * i][tx + 16 * j] = acc[i][j];
    __syncthreads();

    if (EPI == EPI_SWIGLU) {
        // packed columns come in groups of 2*granule: gate block, then up block
        T* out = (T*)g.out + cs * g.out_shard;
        for (int i = threadIdx.x; i < BM * (BN / 2); i += 256) {
            const int r = i / (BN / 2), jj = i % (BN / 2);
            const int grp = jj / granule, w = jj % granule;
            const int c = grp * 2 * granule + w;  // gate column within the tile
            const int m = m0 + r, n = n0 + c;
            if (m < g.M && n < g.N) {
                const long long ncol = (long long)(n / (2 * granule)) * granule + w;
                out[(long long)m * g.ldo + ncol] = from_f<T>(silu(Cs[r][c]) * Cs[r][c + granule]);
            }
        }
    } else if (EPI == EPI_ROW_REDUCE) {
        float* out = (float*)g.out;
        for (int i = threadIdx.x; i < BM * BN; i += 256) {
            const int r = i / BN, c = i % BN, m = m0 + r, n = n0 + c;
            if (m < g.M && n < g.N) {
                const long long o = (long long)m * g.ldo + n;
                float v = Cs[r][c];
                if (g.residual)
                    v += g.residual_f32 ? ((const float*)g.residual)[o] : to_f(((const T*)g.residual)[o]);
                out[o] = v;
                if (g.out2) ((T*)g.out2)[o] = from_f<T>(v);
            }
        }
    } else {
        T* out = (T*)g.out + cs * g.out_shard;
        for (int i = threadIdx.x; i < BM * BN; i += 256) {
            const int r = i / BN, c = i % BN, m = m0 + r, n = n0 + c;
            if (m < g.M && n < g.N) {
                float v = Cs[r][c];
                if (EPI == EPI_GELU) v = gelu_erf(v);
                out[(long long)m * g.ldo + n] = from_f<T>(v);
            }
        }
    }
}

template <typename T>
cudaError_t simt_gemm_t(const SimtGemm& g, int granule, cudaStream_t st) {
    dim3 grid((g.N + BN - 1) / BN, (g.M + BM - 1) / BM, g.col_shards);
    switch (g.epi) {
        case EPI_STORE: simt_gemm_k<T, EPI_STORE><<<grid, 256, 0, st>>>(g, granule); break;
        case EPI_GELU: simt_gemm_k<T, EPI_GELU><<<grid, 256, 0, st>>>(g, granule); break;
        case EPI_SWIGLU: simt_gemm_k<T, EPI_SWIGLU><<<grid, 256, 0, st>>>(g, granule); break;
        default: simt_gemm_k<T, EPI_ROW_REDUCE><<<grid, 256, 0, st>>>(g, granule); break;
    }
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// attention
// ---------------------------------------------------------------------------

constexpr int QT = 16, KT = 32;

template <typename T, int DH>
__global__ void __launch_bounds__(256) simt_attn_k(AttnArgs a) {
    constexpr int NPL = DH / 32;
    __shared__ float Qs[QT][DH];
    __shared__ float Ks[KT][DH + 1];
    __shared__ float Vs[KT][DH];
    const int b = blockIdx.z, h = blockIdx.y, q0 = blockIdx.x * QT;
    const int s = h / a.hl, jl = h % a.hl;
    const int lane = threadIdx.x % 32, w = threadIdx.x / 32;
    const long long M = (long long)a.B * a.Tq;
    const int rowlen = 3 * a.hl * DH;
    const T* qkv = (const T*)a.qkv + s * M * rowlen;
    const bool from_cache = a.kc != nullptr;

    for (int i = threadIdx.x; i < QT * DH; i += 256) {
        const int r = i / DH, c = i % DH, t = q0 + r;
        Qs[r][c] = t < a.Tq ? to_f(qkv[((long long)b * a.Tq + t) * rowlen + jl * DH + c]) * a.scale : 0.f;
    }
    const int nkeys = a.pos + a.Tq;
    const int kmax = a.causal ? min(nkeys, a.pos + q0 + QT) : nkeys;

    float mrow[2], lrow[2], o[2][NPL];
#pragma unroll
    for (int qi = 0; qi < 2; ++qi) {
        mrow[qi] = -INFINITY;
        lrow[qi] = 0.f;
#pragma unroll
        for (int e = 0; e < NPL; ++e) o[qi][e] = 0.f;
    }

    for (int k0 = 0; k0 < kmax; k0 += KT) {
        __syncthreads();
        for (int i = threadIdx.x; i < KT * DH; i += 256) {
            const int r = i / DH, c = i % DH, key = k0 + r;
            float kv = 0.f, vv = 0.f;
            if (key < kmax) {
                if (from_cache) {
                    const long long off = (((long long)b * a.H + h) * a.cap + key) * DH + c;
                    kv = to_f(((const T*)a.kc)[off]);
                    vv = to_f(((const T*)a.vc)[off]);
                } else {
                    const long long off = ((long long)b * a.Tq + key) * rowlen + jl * DH + c;
                    kv = to_f(qkv[off + a.hl * DH]);
                    vv = to_f(qkv[off + 2 * a.hl * DH]);
                }
            }
            Ks[r][c] = kv;
            Vs[r][c] = vv;
        }
        __syncthreads();
#pragma unroll
        for (int qi = 0; qi < 2; ++qi) {
            const int ql = w * 2 + qi, t = q0 + ql;
            if (t >= a.Tq) continue;
            const int qpos = a.pos + t, key = k0 + lane;
            float sc = -INFINITY;
            if (key < kmax && (!a.causal || key <= qpos)) {
                float dot = 0.f;
#pragma unroll 8
                for (int c = 0; c < DH; ++c) dot = fmaf(Qs[ql][c], Ks[lane][c], dot);
                sc = dot;
            }
            float mt = sc;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, off));
            const float mnew = fmaxf(mrow[qi], mt);
            if (mnew == -INFINITY) continue;
            const float p = sc == -INFINITY ? 0.f : expf(sc - mnew);
            const float corr = mrow[qi] == -INFINITY ? 0.f : expf(mrow[qi] - mnew);
            float ps = p;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, off);
            lrow[qi] = lrow[qi] * corr + ps;
#pragma unroll
            for (int e = 0; e < NPL; ++e) o[qi][e] *= corr;
            for (int j = 0; j < KT; ++j) {
                const float pj = __shfl_sync(0xffffffffu, p, j);
#pragma unroll
                for (int e = 0; e < NPL; ++e) o[qi][e] = fmaf(pj, Vs[j][lane + 32 * e], o[qi][e]);
            }
            mrow[qi] = mnew;
        }
    }
    T* out = (T*)a.out + s * M * (a.hl * DH);
#pragma unroll
    for (int qi = 0; qi < 2; ++qi) {
        const int t = q0 + w * 2 + qi;
        if (t >= a.Tq) continue;
        const float inv = 1.f / lrow[qi];
#pragma unroll
        for (int e = 0; e < NPL; ++e)
            out[((long long)b * a.Tq + t) * (a.hl * DH) + jl * DH + lane + 32 * e] = from_f<T>(o[qi][e] * inv);
    }
}

template <typename T>
__global__ void kv_append_k(AttnArgs a, T* __restrict__ kc, T* __restrict__ vc) {
    const long long total = (long long)a.B * a.Tq * a.H * a.dh;
    const long long M = (long long)a.B * a.Tq;
    const int rowlen = 3 * a.hl * a.dh;
    const T* qkv = (const T*)a.qkv;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
         i += (long long)gridDim.x * blockDim.x) {
        const int c = (int)(i % a.dh);
        const int h = (int)((i / a.dh) % a.H);
        const long long bt = i / ((long long)a.dh * a.H);  // b*Tq + t
        const int t = (int)(bt % a.Tq);
        const long long b = bt / a.Tq;
        const int s = h / a.hl, jl = h % a.hl;
        const long long src = (long long)s * M * rowlen + bt * rowlen + jl * a.dh + c;
        const long long dst = ((b * a.H + h) * a.cap + a.pos + t) * a.dh + c;
        kc[dst] = qkv[src + a.hl * a.dh];
        vc[dst] = qkv[src + 2 * a.hl * a.dh];
    }
}

template <typename T, int DH>
cudaError_t simt_attn_launch(const AttnArgs& a, cudaStream_t st) {
    dim3 grid((a.Tq + QT - 1) / QT, a.H, a.B);
    simt_attn_k<T, DH><<<grid, 256, 0, st>>>(a);
    return cudaGetLastError();
}

template <typename T>
cudaError_t simt_attn_t(const AttnArgs& a, cudaStream_t st) {
    switch (a.dh) {
        case 32: return simt_attn_launch<T, 32>(a, st);
        case 64: return simt_attn_launch<T, 64>(a, st);
        case 128: return simt_attn_launch<T, 128>(a, st);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t simt_gemm(const SimtGemm& g, cudaStream_t st) {
    return g.is_bf16 ? simt_gemm_t<bf16>(g, g.granule, st) : simt_gemm_t<float>(g, g.granule, st);
}

cudaError_t simt_attention(const AttnArgs& a, cudaStream_t st) {
    return a.is_bf16 ? simt_attn_t<bf16>(a, st) : simt_attn_t<float>(a, st);
}

cudaError_t kv_append(const AttnArgs& a, void* kc, void* vc, cudaStream_t st) {
    const long long total = (long long)a.B * a.Tq * a.H * a.dh;
    long long blocks = (total + 255) / 256;
    if (blocks > 148 * 16) blocks = 148 * 16;
    if (blocks < 1) blocks = 1;
    if (a.is_bf16)
        kv_append_k<bf16><<<(int)blocks, 256, 0, st>>>(a, (bf16*)kc, (bf16*)vc);
    else
        kv_append_k<float><<<(int)blocks, 256, 0, st>>>(a, (float*)kc, (float*)vc);
    return cudaGetLastError();
}

}  // namespace tpk
