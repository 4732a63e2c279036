// Packing of full [out, in] weights into the shard-major layout the GEMMs read.
//
// Column-parallel weights (Q/K/V by head, FFN-up) keep whole rows, so shard s
// is a contiguous block of rows; row-parallel weights (Wo, Wd) are split by
// input feature, so shard s's columns are gathered into a contiguous
// [N][k_s] block (undercodenews.com/?p=110319, "the Original").
#include "kernels.h"

namespace tpk {

namespace {

template <typename E>
__global__ void pack_qkv_k(const E* __restrict__ Wq, const E* __restrict__ Wk, const E* __restrict__ Wv,
                           E* __restrict__ dst, int tp, int hl, int dh, int d) {
    const long long rows_s = 3LL * hl * dh;
    const long long total = (long long)tp * rows_s * d;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
         i += (long long)gridDim.x * blockDim.x) {
        long long c = i % d;
        long long r = (i / d) % rows_s;
        long long s = i / (d * rows_s);
        int which = (int)(r / ((long long)hl * dh));
        long long within = r % ((long long)hl * dh);
        long long grow = s * hl * dh + within;
        const E* src = which == 0 ? Wq : (which == 1 ? Wk : Wv);
        dst[i] = src[grow * d + c];
    }
}

template <typename E>
__global__ void pack_cols_k(const E* __restrict__ src, E* __restrict__ dst, int tp, int N, int ks) {
    const long long total = (long long)tp * N * ks;
    const long long ld = (long long)tp * ks;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
         i += (long long)gridDim.x * blockDim.x) {
        long long k = i % ks;
        long long n = (i / ks) % N;
        long long s = i / ((long long)ks * N);
        dst[i] = src[n * ld + s * ks + k];
    }
}

template <typename E>
__global__ void pack_up_k(const E* __restrict__ Wg, const E* __restrict__ Wu, E* __restrict__ dst, int tp, int fl,
                          int d, int g) {
    const int rows_s = Wu ? 2 * fl : fl;
    const long long total = (long long)tp * rows_s * d;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
         i += (long long)gridDim.x * blockDim.x) {
        long long c = i % d;
        long long r = (i / d) % rows_s;
        long long s = i / ((long long)d * rows_s);
        if (Wu) {
            // groups of 2g rows: g gate rows, then the g matching up rows
            long long grp = r / (2 * g), q = r % (2 * g);
            long long frow = s * fl + grp * g + (q % g);
            dst[i] = (q < g ? Wg : Wu)[frow * d + c];
        } else {
            dst[i] = Wg[(s * fl + r) * d + c];
        }
    }
}

int grid_for(long long total) {
    long long b = (total + 255) / 256;
    return (int)(b < 148 * 32 ? (b < 1 ? 1 : b) : 148 * 32);
}

}  // namespace

cudaError_t pack_qkv(int esize, const void* Wq, const void* Wk, const void* Wv, void* dst, int tp, int hl, int dh,
                     int d, cudaStream_t st) {
    long long total = (long long)tp * 3 * hl * dh * d;
    if (esize == 2)
        pack_qkv_k<uint16_t><<<grid_for(total), 256, 0, st>>>((const uint16_t*)Wq, (const uint16_t*)Wk,
                                                              (const uint16_t*)Wv, (uint16_t*)dst, tp, hl, dh, d);
    else
        pack_qkv_k<uint32_t><<<grid_for(total), 256, 0, st>>>((const uint32_t*)Wq, (const uint32_t*)Wk,
                                                              (const uint32_t*)Wv, (uint32_t*)dst, tp, hl, dh, d);
    return cudaGetLastError();
}

cudaError_t pack_cols(int esize, const void* src, void* dst, int tp, int N, int ks, cudaStream_t st) {
    long long total = (long long)tp * N * ks;
    if (esize == 2)
        pack_cols_k<uint16_t><<<grid_for(total), 256, 0, st>>>((const uint16_t*)src, (uint16_t*)dst, tp, N, ks);
    else
        pack_cols_k<uint32_t><<<grid_for(total), 256, 0, st>>>((const uint32_t*)src, (uint32_t*)dst, tp, N, ks);
    return cudaGetLastError();
}

cudaError_t pack_up(int esize, const void* Wg, const void* Wu, void* dst, int tp, int fl, int d, int granule,
                    cudaStream_t st) {
    long long total = (long long)tp * (Wu ? 2 : 1) * fl * d;
    if (esize == 2)
        pack_up_k<uint16_t><<<grid_for(total), 256, 0, st>>>((const uint16_t*)Wg, (const uint16_t*)Wu,
                                                             (uint16_t*)dst, tp, fl, d, granule);
    else
        pack_up_k<uint32_t><<<grid_for(total), 256, 0, st>>>((const uint32_t*)Wg, (const uint32_t*)Wu,
                                                             (uint32_t*)dst, tp, fl, d, granule);
    return cudaGetLastError();
}

}  // namespace tpk
