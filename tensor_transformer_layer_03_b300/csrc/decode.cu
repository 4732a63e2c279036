// Single-token decode attention over the per-head KV cache.
//
// Each head's cache rows belong to the shard that owns the head ("Tensor
// Parallelism: Splitting One Layer Across GPUs" (byteledger), "Interaction
// with the rest of serving"), so a (sequence, head) pair is independent work.
// One query row per head leaves too little parallelism for one block per
// head, so the keys are split into chunks: pass 1 computes, per chunk, the
// running max m, the sum l of exp(s - m) and the unnormalised output
// sum_j exp(s_j - m) v_j; pass 2 merges the chunks with the usual
// log-sum-exp rescaling and writes softmax(q K^T / sqrt(d_head)) V.
#include <math.h>

#include "common.cuh"
#include "kernels.h"

namespace tpk {

namespace {

constexpr int DEC_THREADS = 128;  // keys scored per sub-chunk (one per thread)

__device__ __forceinline__ float block_reduce(float v, float* red, bool is_max) {
    const int lane = threadIdx.x % 32, w = threadIdx.x / 32;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const float o = __shfl_xor_sync(0xffffffffu, v, off);
        v = is_max ? fmaxf(v, o) : v + o;
    }
    __syncthreads();
    if (lane == 0) red[w] = v;
    __syncthreads();
    float r = red[0];
#pragma unroll
    for (int i = 1; i < DEC_THREADS / 32; ++i) r = is_max ? fmaxf(r, red[i]) : r + red[i];
    return r;
}

template <typename T, int DH>
__global__ void __launch_bounds__(DEC_THREADS) decode_split_k(AttnArgs a, float* __restrict__ part, int chunk,
                                                              int nsplit) {
    constexpr int G = DEC_THREADS / DH;  // key groups in the P.V pass
    __shared__ float qs[DH];
    __shared__ float ps[DEC_THREADS];
    __shared__ float red[DEC_THREADS / 32];
    __shared__ float ored[G][DH];
    const int c = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int s = h / a.hl, jl = h % a.hl;
    const long long M = (long long)a.B;  // one query token per sequence
    const T* q = (const T*)a.qkv + ((long long)s * M + b) * (3 * a.hl * DH) + jl * DH;
    for (int i = threadIdx.x; i < DH; i += DEC_THREADS) qs[i] = to_f(q[i]) * a.scale;
    const int L = a.pos + 1;
    const int k0 = c * chunk, k1 = min(L, k0 + chunk);
    const T* kbase = (const T*)a.kc + ((long long)b * a.H + h) * a.cap * DH;
    const T* vbase = (const T*)a.vc + ((long long)b * a.H + h) * a.cap * DH;
    const int dim = threadIdx.x % DH, grp = threadIdx.x / DH;
    float m_run = -INFINITY, l_run = 0.f, o_acc = 0.f;
    __syncthreads();
    for (int sub = k0; sub < k1; sub += DEC_THREADS) {
        const int key = sub + threadIdx.x;
        float sc = -INFINITY;
        if (key < k1) {
            const T* kr = kbase + (long long)key * DH;
            float dot = 0.f;
#pragma unroll 16
            for (int i = 0; i < DH; ++i) dot = fmaf(qs[i], to_f(kr[i]), dot);
            sc = dot;
        }
        const float mt = block_reduce(sc, red, true);
        const float mnew = fmaxf(m_run, mt);
        const float p = key < k1 ? expf(sc - mnew) : 0.f;
        ps[threadIdx.x] = p;
        const float lt = block_reduce(p, red, false);  // also orders the ps writes
        const float corr = m_run == -INFINITY ? 0.f : expf(m_run - mnew);
        l_run = l_run * corr + lt;
        o_acc *= corr;
        const int nk = min(DEC_THREADS, k1 - sub);
        for (int j = grp; j < nk; j += G) o_acc = fmaf(ps[j], to_f(vbase[(long long)(sub + j) * DH + dim]), o_acc);
        m_run = mnew;
        __syncthreads();
    }
    ored[grp][dim] = o_acc;
    __syncthreads();
    float* dst = part + (((long long)b * a.H + h) * DECODE_MAX_SPLITS + c) * (DH + 2);
    if (threadIdx.x < DH) {
        float o = 0.f;
#pragma unroll
        for (int g2 = 0; g2 < G; ++g2) o += ored[g2][threadIdx.x];
        dst[2 + threadIdx.x] = o;
    }
    if (threadIdx.x == 0) {
        dst[0] = m_run;
        dst[1] = l_run;
    }
}

template <typename T, int DH>
__global__ void __launch_bounds__(DH) decode_combine_k(AttnArgs a, const float* __restrict__ part, int nsplit) {
    const int h = blockIdx.x, b = blockIdx.y;
    const int s = h / a.hl, jl = h % a.hl;
    const float* src = part + ((long long)b * a.H + h) * DECODE_MAX_SPLITS * (DH + 2);
    float mx = -INFINITY;
    for (int c = 0; c < nsplit; ++c) mx = fmaxf(mx, src[c * (DH + 2)]);
    float l = 0.f, o = 0.f;
    for (int c = 0; c < nsplit; ++c) {
        const float* pc = src + c * (DH + 2);
        const float w = expf(pc[0] - mx);
        l = fmaf(pc[1], w, l);
        o = fmaf(pc[2 + threadIdx.x], w, o);
    }
    T* out = (T*)a.out + ((long long)s * a.B + b) * (a.hl * DH) + jl * DH;
    out[threadIdx.x] = from_f<T>(o / l);
}

// bf16 variant of pass 1 with 16-byte loads: DH/8 lanes share a key row
// (each lane one 16-byte slice), so a warp scores 32/(DH/8) keys per step
// with fully coalesced loads; the chunk is walked in sub-chunks of SUB keys
// with the online max/sum; in the P.V pass each lane owns DH/32 dimensions
// and the four warps take interleaved keys.
constexpr int SUB = 256;

// DPL consecutive bf16 (DPL = 1, 2 or 4; 2*DPL-byte aligned) as floats
template <int DPL>
__device__ __forceinline__ void load_dims(const bf16* p, float (&f)[DPL]) {
    if constexpr (DPL == 4) {
        const uint2 v = *reinterpret_cast<const uint2*>(p);
        const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
        const float2 a = __bfloat1622float2(h[0]), b = __bfloat1622float2(h[1]);
        f[0] = a.x;
        f[1] = a.y;
        f[2] = b.x;
        f[3] = b.y;
    } else if constexpr (DPL == 2) {
        const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(p));
        f[0] = a.x;
        f[1] = a.y;
    } else {
        f[0] = __bfloat162float(p[0]);
    }
}

template <int DH>
__global__ void __launch_bounds__(DEC_THREADS) decode_split_bf16_k(AttnArgs a, float* __restrict__ part, int chunk) {
    constexpr int LPK = DH / 8;    // lanes per key row
    constexpr int KPW = 32 / LPK;  // keys per warp step
    constexpr int DPL = DH / 32;   // output dims per lane
    constexpr int NW = DEC_THREADS / 32;
    __shared__ float sc[SUB];
    __shared__ float red[NW];
    __shared__ float ored[NW][DH];
    const int c = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int s = h / a.hl, jl = h % a.hl;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int sub_l = lane % LPK, kq = lane / LPK;
    const bf16* q = (const bf16*)a.qkv + ((long long)s * a.B + b) * (3 * a.hl * DH) + jl * DH;
    float qv[8];
    {
        const uint4 v = *reinterpret_cast<const uint4*>(q + sub_l * 8);
        const __nv_bfloat162* hq = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 f = __bfloat1622float2(hq[i]);
            qv[2 * i] = f.x * a.scale;
            qv[2 * i + 1] = f.y * a.scale;
        }
    }
    const int L = a.pos + 1;
    const int k0 = c * chunk, k1 = min(L, k0 + chunk);
    const bf16* kbase = (const bf16*)a.kc + ((long long)b * a.H + h) * a.cap * DH;
    const bf16* vbase = (const bf16*)a.vc + ((long long)b * a.H + h) * a.cap * DH;
    float m_run = -INFINITY, l_run = 0.f;
    float o[DPL];
#pragma unroll
    for (int e = 0; e < DPL; ++e) o[e] = 0.f;

    for (int sub = k0; sub < k1; sub += SUB) {
        const int n = min(SUB, k1 - sub);
        for (int j0 = warp * KPW; j0 < n; j0 += NW * KPW) {
            const int j = j0 + kq;
            float d = 0.f;
            if (j < n) {
                const uint4 v = *reinterpret_cast<const uint4*>(kbase + (long long)(sub + j) * DH + sub_l * 8);
                const __nv_bfloat162* hk = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float2 f = __bfloat1622float2(hk[i]);
                    d = fmaf(qv[2 * i], f.x, d);
                    d = fmaf(qv[2 * i + 1], f.y, d);
                }
            }
#pragma unroll
            for (int off = LPK / 2; off > 0; off >>= 1) d += __shfl_xor_sync(0xffffffffu, d, off);
            if (sub_l == 0 && j < n) sc[j] = d;
        }
        __syncthreads();
        float mt = -INFINITY;
        for (int j = threadIdx.x; j < n; j += DEC_THREADS) mt = fmaxf(mt, sc[j]);
        mt = block_reduce(mt, red, true);
        const float mnew = fmaxf(m_run, mt);
        float lt = 0.f;
        for (int j = threadIdx.x; j < n; j += DEC_THREADS) {
            const float p = expf(sc[j] - mnew);
            sc[j] = p;
            lt += p;
        }
        lt = block_reduce(lt, red, false);  // its barriers also publish sc[]
        const float corr = m_run == -INFINITY ? 0.f : expf(m_run - mnew);
        l_run = l_run * corr + lt;
#pragma unroll
        for (int e = 0; e < DPL; ++e) o[e] *= corr;
        for (int j = warp; j < n; j += NW) {
            const float p = sc[j];
            float v[DPL];
            load_dims<DPL>(vbase + (long long)(sub + j) * DH + lane * DPL, v);
#pragma unroll
            for (int e = 0; e < DPL; ++e) o[e] = fmaf(p, v[e], o[e]);
        }
        m_run = mnew;
        __syncthreads();  // sc[] is rewritten by the next sub-chunk
    }
#pragma unroll
    for (int e = 0; e < DPL; ++e) ored[warp][lane * DPL + e] = o[e];
    __syncthreads();
    float* dst = part + (((long long)b * a.H + h) * DECODE_MAX_SPLITS + c) * (DH + 2);
    for (int i = threadIdx.x; i < DH; i += DEC_THREADS) {
        float acc = 0.f;
#pragma unroll
        for (int w2 = 0; w2 < NW; ++w2) acc += ored[w2][i];
        dst[2 + i] = acc;
    }
    if (threadIdx.x == 0) {
        dst[0] = m_run;
        dst[1] = l_run;
    }
}

// bf16 single-token pass 1: one block (4 warps) per (sequence, head, chunk
// of 64 keys), 16 keys per warp.  Loads are coalesced: in each load
// instruction a warp reads 512 contiguous bytes of the K (then V) cache,
// i.e. KPI whole key rows, one 16-byte chunk (8 dimensions) per lane; every
// K and V load of the chunk is issued before any is used, so a chunk costs
// one memory round trip.  A lane keeps q for its 8 dimensions; a key's score
// is reduced over the CH lanes that hold its row (shuffles), P V is summed in
// registers over the warp's keys and across the 4 warps in shared memory.
// The new token's K/V row (position pos) comes from the QKV buffer and is
// written into the cache here, so no separate append pass runs.  Scores in
// log2 units; partial (m, l, o) as in the kernels above.
constexpr int DC_KEYS = 64;

template <int DH>
__global__ void __launch_bounds__(DEC_THREADS) decode_chunk_bf16_k(AttnArgs a, float* __restrict__ part) {
    constexpr int CH = DH / 8;           // 16-byte chunks per key row (16 or 8)
    constexpr int KPI = 32 / CH;         // key rows per warp load instruction
    constexpr int NW = DEC_THREADS / 32;
    constexpr int KPW = DC_KEYS / NW;    // keys per warp
    constexpr int NI = KPW / KPI;        // load instructions per warp and matrix
    __shared__ float red[2][NW];
    __shared__ float ored[NW][DH];
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int c = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int s = h / a.hl, jl = h % a.hl;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int ch = lane % CH, r = lane / CH;  // this lane's 8 dimensions, and which row of the instruction
    const int L = a.pos + 1;
    const int kw = c * DC_KEYS + warp * KPW;  // first key of this warp
    const bf16* qkv_row = (const bf16*)a.qkv + ((long long)s * a.B + b) * (3 * a.hl * DH);
    bf16* kcache = (bf16*)a.kc + ((long long)b * a.H + h) * a.cap * DH;
    bf16* vcache = (bf16*)a.vc + ((long long)b * a.H + h) * a.cap * DH;
    // everything read below (Q, the new K/V, and cache rows appended by
    // earlier steps' kernels) may come from kernels still finishing
    asm volatile("griddepcontrol.wait;" ::: "memory");
    uint4 kv[NI], vv[NI];
#pragma unroll
    for (int i = 0; i < NI; ++i) {
        const int key = kw + i * KPI + r;
        kv[i] = vv[i] = make_uint4(0u, 0u, 0u, 0u);
        if (key < L && key != a.pos) {
            kv[i] = reinterpret_cast<const uint4*>(kcache + (long long)key * DH)[ch];
            vv[i] = reinterpret_cast<const uint4*>(vcache + (long long)key * DH)[ch];
        }
    }
    float q[8];
    {
        const uint4 qv = reinterpret_cast<const uint4*>(qkv_row + jl * DH)[ch];
        const __nv_bfloat162* hq = reinterpret_cast<const __nv_bfloat162*>(&qv);
        const float sl2 = a.scale * 1.4426950408889634f;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 f = __bfloat1622float2(hq[e]);
            q[2 * e] = f.x * sl2;
            q[2 * e + 1] = f.y * sl2;
        }
    }
    // the new token's row: from the QKV buffer, and into the cache
#pragma unroll
    for (int i = 0; i < NI; ++i) {
        const int key = kw + i * KPI + r;
        if (key == a.pos) {
            kv[i] = reinterpret_cast<const uint4*>(qkv_row + (a.hl + jl) * DH)[ch];
            vv[i] = reinterpret_cast<const uint4*>(qkv_row + (2 * a.hl + jl) * DH)[ch];
            reinterpret_cast<uint4*>(kcache + (long long)key * DH)[ch] = kv[i];
            reinterpret_cast<uint4*>(vcache + (long long)key * DH)[ch] = vv[i];
        }
    }
    // scores of this lane's NI keys (equal across the CH lanes of a row)
    float sc[NI];
    float mx = -INFINITY;
#pragma unroll
    for (int i = 0; i < NI; ++i) {
        const __nv_bfloat162* hk = reinterpret_cast<const __nv_bfloat162*>(&kv[i]);
        float d = 0.f;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 f = __bfloat1622float2(hk[e]);
            d = fmaf(q[2 * e], f.x, d);
            d = fmaf(q[2 * e + 1], f.y, d);
        }
#pragma unroll
        for (int off = CH / 2; off > 0; off >>= 1) d += __shfl_xor_sync(0xffffffffu, d, off);
        sc[i] = (kw + i * KPI + r < L) ? d : -INFINITY;
        mx = fmaxf(mx, sc[i]);
    }
#pragma unroll
    for (int off = CH; off < 32; off <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    if (lane == 0) red[0][warp] = mx;
    __syncthreads();
    float m = red[0][0];
#pragma unroll
    for (int w2 = 1; w2 < NW; ++w2) m = fmaxf(m, red[0][w2]);
    // p and the running sums; o over this lane's keys and 8 dimensions
    float l = 0.f, o[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) o[e] = 0.f;
#pragma unroll
    for (int i = 0; i < NI; ++i) {
        const float pr = exp2f(sc[i] - m);  // 0 for keys past the end (-inf)
        l += pr;
        const __nv_bfloat162* hv = reinterpret_cast<const __nv_bfloat162*>(&vv[i]);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 f = __bfloat1622float2(hv[e]);
            o[2 * e] = fmaf(pr, f.x, o[2 * e]);
            o[2 * e + 1] = fmaf(pr, f.y, o[2 * e + 1]);
        }
    }
    // sum over the rows of the warp (lanes with the same chunk), then warps
#pragma unroll
    for (int off = CH; off < 32; off <<= 1) {
        l += __shfl_xor_sync(0xffffffffu, l, off);
#pragma unroll
        for (int e = 0; e < 8; ++e) o[e] += __shfl_xor_sync(0xffffffffu, o[e], off);
    }
    if (r == 0) {
#pragma unroll
        for (int e = 0; e < 8; ++e) ored[warp][ch * 8 + e] = o[e];
    }
    if (lane == 0) red[1][warp] = l;
    __syncthreads();
    float* dst = part + (((long long)b * a.H + h) * DECODE_MAX_SPLITS + c) * (DH + 2);
    for (int i = threadIdx.x; i < DH; i += DEC_THREADS) {
        float acc = 0.f;
#pragma unroll
        for (int w2 = 0; w2 < NW; ++w2) acc += ored[w2][i];
        dst[2 + i] = acc;
    }
    if (threadIdx.x == 0) {
        float lt = 0.f;
#pragma unroll
        for (int w2 = 0; w2 < NW; ++w2) lt += red[1][w2];
        dst[0] = m;
        dst[1] = lt;
    }
}

// bf16 pass 2: merge the chunks of one (sequence, head).  The chunk maxima
// and sums are read in parallel (one chunk per thread), then each thread
// sums one output dimension over the chunks.
template <int DH>
__global__ void __launch_bounds__(DH) decode_merge_bf16_k(AttnArgs a, const float* __restrict__ part, int nsplit) {
    __shared__ float w[DECODE_MAX_SPLITS];
    __shared__ float red[DH / 32 > 0 ? DH / 32 : 1];
    __shared__ float tot;
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int h = blockIdx.x, b = blockIdx.y;
    const int s = h / a.hl, jl = h % a.hl;
    const int t = threadIdx.x;
    const float* src = part + ((long long)b * a.H + h) * DECODE_MAX_SPLITS * (DH + 2);
    float mc = -INFINITY, lc = 0.f;
    for (int c = t; c < nsplit; c += DH) {
        mc = fmaxf(mc, src[c * (DH + 2)]);
    }
    // block max of the chunk maxima
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mc = fmaxf(mc, __shfl_xor_sync(0xffffffffu, mc, off));
    if (t % 32 == 0) red[t / 32] = mc;
    __syncthreads();
    float mx = red[0];
#pragma unroll
    for (int i = 1; i < DH / 32; ++i) mx = fmaxf(mx, red[i]);
    for (int c = t; c < nsplit; c += DH) {
        const float wc = exp2f(src[c * (DH + 2)] - mx);
        w[c] = wc;
        lc = fmaf(src[c * (DH + 2) + 1], wc, lc);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) lc += __shfl_xor_sync(0xffffffffu, lc, off);
    __syncthreads();
    if (t % 32 == 0) red[t / 32] = lc;
    __syncthreads();
    if (t == 0) {
        float l = 0.f;
        for (int i = 0; i < DH / 32; ++i) l += red[i];
        tot = l;
    }
    __syncthreads();
    float o = 0.f;
#pragma unroll 8
    for (int c = 0; c < nsplit; ++c) o = fmaf(src[c * (DH + 2) + 2 + t], w[c], o);
    bf16* out = (bf16*)a.out + ((long long)s * a.B + b) * (a.hl * DH) + jl * DH;
    out[t] = __float2bfloat16_rn(o / tot);
}

// Launch with programmatic dependent launch allowed: the kernel may start
// while the previous kernel in the stream finishes; it waits
// (griddepcontrol.wait) before reading what that kernel wrote.
template <typename K, typename... Args>
cudaError_t launch_pdl(K kernel, dim3 grid, dim3 block, cudaStream_t st, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

template <typename T, int DH>
cudaError_t decode_launch(const AttnArgs& a, float* scratch, cudaStream_t st) {
    const int L = a.pos + 1;
    int nsplit, chunk;
    if (a.is_bf16) {
        if (DH == 64 || DH == 128) {
            nsplit = (L + DC_KEYS - 1) / DC_KEYS;
            if (nsplit <= DECODE_MAX_SPLITS) {
                cudaError_t e = launch_pdl(decode_chunk_bf16_k<DH>, dim3(nsplit, a.H, a.B), dim3(DEC_THREADS), st, a,
                                           scratch);
                if (e != cudaSuccess) return e;
                return launch_pdl(decode_merge_bf16_k<DH>, dim3(a.H, a.B), dim3(DH), st, a,
                                  static_cast<const float*>(scratch), nsplit);
            }
        }
        // long caches (or other head widths): chunks of about 64 keys, at most
        // DECODE_MAX_SPLITS of them, after a separate append of the new K/V
        cudaError_t e = kv_append(a, const_cast<void*>(a.kc), const_cast<void*>(a.vc), st);
        if (e != cudaSuccess) return e;
        nsplit = (L + 63) / 64;
        if (nsplit > DECODE_MAX_SPLITS) nsplit = DECODE_MAX_SPLITS;
        chunk = (L + nsplit - 1) / nsplit;
        nsplit = (L + chunk - 1) / chunk;
        decode_split_bf16_k<DH><<<dim3(nsplit, a.H, a.B), DEC_THREADS, 0, st>>>(a, scratch, chunk);
    } else {
        cudaError_t e = kv_append(a, const_cast<void*>(a.kc), const_cast<void*>(a.vc), st);
        if (e != cudaSuccess) return e;
        nsplit = (L + DEC_THREADS - 1) / DEC_THREADS;
        chunk = DEC_THREADS;
        if (nsplit > DECODE_MAX_SPLITS) {
            chunk = ((L + DECODE_MAX_SPLITS - 1) / DECODE_MAX_SPLITS + DEC_THREADS - 1) / DEC_THREADS * DEC_THREADS;
            nsplit = (L + chunk - 1) / chunk;
        }
        decode_split_k<T, DH><<<dim3(nsplit, a.H, a.B), DEC_THREADS, 0, st>>>(a, scratch, chunk, nsplit);
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    decode_combine_k<T, DH><<<dim3(a.H, a.B), DH, 0, st>>>(a, scratch, nsplit);
    return cudaGetLastError();
}

template <typename T>
cudaError_t decode_t(const AttnArgs& a, float* scratch, cudaStream_t st) {
    switch (a.dh) {
        case 32: return decode_launch<T, 32>(a, scratch, st);
        case 64: return decode_launch<T, 64>(a, scratch, st);
        case 128: return decode_launch<T, 128>(a, scratch, st);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t decode_attention(const AttnArgs& a, float* scratch, cudaStream_t st) {
    return a.is_bf16 ? decode_t<bf16>(a, scratch, st) : decode_t<float>(a, scratch, st);
}

}  // namespace tpk
