// Pieces of the pre-norm (RMSNorm) variant of the block that are not inside
// the linears.  RMSNorm(x; g) W^T = diag(1/rms(x)) x (W diag(g))^T, so the
// gain g is folded into the packed weight columns once (scale_cols) and the
// per-row factor 1/rms is computed here (rms_rows) and applied to the
// accumulator rows in the GEMM epilogue -- the tensor-core main loop is the
// same as for the plain block.  (Norms are not on the source pages; this is
// the LLaMA-style reading of the block.)
#include "common.cuh"
#include "kernels.h"

namespace tpk {

namespace {

template <typename E>
__global__ void scale_cols_k(E* __restrict__ W, long long rows, int d, const E* __restrict__ g) {
    const long long total = rows * d;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
         i += (long long)gridDim.x * blockDim.x)
        W[i] = from_f<E>(to_f(W[i]) * to_f(g[i % d]));
}

// one warp per row; fp32 sum of squares, each lane reading 8-element
// (16- or 32-byte) chunks; d is a multiple of 8
__device__ __forceinline__ float sumsq8(const bf16* p) {
    const uint4 u = *reinterpret_cast<const uint4*>(p);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
    float s = 0.f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const float lo = __uint_as_float(w[j] << 16), hi = __uint_as_float(w[j] & 0xffff0000u);
        s = fmaf(lo, lo, fmaf(hi, hi, s));
    }
    return s;
}

__device__ __forceinline__ float sumsq8(const float* p) {
    const float4 a = reinterpret_cast<const float4*>(p)[0], b = reinterpret_cast<const float4*>(p)[1];
    return a.x * a.x + a.y * a.y + a.z * a.z + a.w * a.w + b.x * b.x + b.y * b.y + b.z * b.z + b.w * b.w;
}

// Launched with programmatic dependent launch: lets the next kernel start
// at entry and waits for the previous one before reading x or writing.
// Four chunks per lane are loaded before they are summed (memory-level
// parallelism).  Blocks past the first rms_blocks fill the rotary table.
template <typename E>
__global__ void rms_rows_k(const E* __restrict__ x, int M, int d, float eps, float* __restrict__ r, RopeTable rt,
                           int rms_blocks, int slice_rows, long long slice_stride) {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if ((int)blockIdx.x >= rms_blocks) {
        const int idx = ((int)blockIdx.x - rms_blocks) * blockDim.x + threadIdx.x;
        if (idx < rt.seq * rt.half) {
            const int t = idx / rt.half, i = idx % rt.half;
            const float ang = (float)(rt.pos0 + t) * exp2f(-(float)(2 * i) / (float)(2 * rt.half) * rt.log2_theta);
            float sn, cs;
            sincosf(ang, &sn, &cs);
            rt.cs[idx] = make_float2(cs, sn);
        }
        return;
    }
    const int lane = threadIdx.x % 32;
    const int row = blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
    if (row >= M) return;
    // (sequence-parallel input: row m in slice m / slice_rows)
    const E* xr = x + (slice_rows ? (long long)(row / slice_rows) * slice_stride + (long long)(row % slice_rows) * d
                                  : (long long)row * d);
    float s = 0.f;
    int c = lane * 8;
    for (; c + 3 * 256 < d; c += 4 * 256) {
        const float a = sumsq8(xr + c), b = sumsq8(xr + c + 256), e = sumsq8(xr + c + 512),
                    f = sumsq8(xr + c + 768);
        s += (a + b) + (e + f);
    }
    for (; c < d; c += 256) s += sumsq8(xr + c);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    if (lane == 0) r[row] = rsqrtf(s / (float)d + eps);
}

}  // namespace

cudaError_t scale_cols(int esize, void* W, long long rows, int d, const void* gamma, cudaStream_t st) {
    long long total = rows * d;
    long long b = (total + 255) / 256;
    const int blocks = (int)(b < 148 * 32 ? (b < 1 ? 1 : b) : 148 * 32);
    if (esize == 2)
        scale_cols_k<bf16><<<blocks, 256, 0, st>>>((bf16*)W, rows, d, (const bf16*)gamma);
    else
        scale_cols_k<float><<<blocks, 256, 0, st>>>((float*)W, rows, d, (const float*)gamma);
    return cudaGetLastError();
}

cudaError_t rms_rows(const void* x, int x_f32, int M, int d, float eps, float* r, const RopeTable* rope,
                     cudaStream_t st, int slice_rows, long long slice_stride) {
    const int rms_blocks = (M + 7) / 8;
    RopeTable rt = {};
    if (rope) rt = *rope;
    const long long entries = rope ? (long long)rt.seq * rt.half : 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(rms_blocks + (unsigned)((entries + 255) / 256));
    cfg.blockDim = dim3(256);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (x_f32)
        return cudaLaunchKernelEx(&cfg, rms_rows_k<float>, (const float*)x, M, d, eps, r, rt, rms_blocks, slice_rows,
                                  slice_stride);
    return cudaLaunchKernelEx(&cfg, rms_rows_k<bf16>, (const bf16*)x, M, d, eps, r, rt, rms_blocks, slice_rows,
                              slice_stride);
}

}  // namespace tpk
