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

template <typename E>
__global__ void rms_rows_k(const E* __restrict__ x, int M, int d, float eps, float* __restrict__ r) {
    const int lane = threadIdx.x % 32;
    const int row = blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
    if (row >= M) return;
    const E* xr = x + (long long)row * d;
    float s = 0.f;
    for (int c = lane * 8; c < d; c += 256) s += sumsq8(xr + c);
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

cudaError_t rms_rows(const void* x, int x_f32, int M, int d, float eps, float* r, cudaStream_t st) {
    const int blocks = (M + 7) / 8;
    if (x_f32)
        rms_rows_k<float><<<blocks, 256, 0, st>>>((const float*)x, M, d, eps, r);
    else
        rms_rows_k<bf16><<<blocks, 256, 0, st>>>((const bf16*)x, M, d, eps, r);
    return cudaGetLastError();
}

}  // namespace tpk
