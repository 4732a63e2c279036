// Prefill attention on the tensor cores (bf16 in, fp32 softmax/accumulate).
//
// Per shard, head and 64-query tile: O = softmax(Q K^T / sqrt(d_head) + mask) V
// with the online (running max / running sum) softmax, so the T x T score
// matrix never leaves registers.  Heads are independent, so every (sequence,
// head) pair is separate work and no shard talks to another
// (undercodenews.com/?p=110319, "the Original": each GPU computes attention
// locally for its heads).
//
// CTA = 4 warps, 16 query rows per warp, 64 keys per step.  Q stays in
// registers; K and V tiles are double-buffered in shared memory with
// cp.async (16-byte chunks, XOR-swizzled rows so ldmatrix is conflict-free).
// S = Q K^T and O += P V use mma.sync m16n8k16 (bf16 x bf16 -> fp32); the
// row max and row sum are reduced across each quad of lanes with warp
// shuffles; P is re-packed from the S accumulators into the A operand of the
// P V product without touching shared memory.
#include <math.h>

#include "common.cuh"
#include "kernels.h"

namespace tpk {

namespace {

constexpr int FA_BM = 64, FA_BN = 64, FA_THREADS = 128;

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// 16-byte async copy global -> shared; src_bytes == 0 fills zeros.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, int src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}

// byte offset of 16-byte chunk c of row r in a [rows][D] bf16 tile
template <int D>
__device__ __forceinline__ uint32_t swz(int r, int c) {
    return (uint32_t)(r * (D * 2) + ((c ^ (r & 7)) << 4));
}

// rows [r0, r0+ROWS) of a [rows][D] matrix with row stride `ld` (elements)
// into a swizzled tile; rows >= nrows are zero-filled.
template <int D, int ROWS>
__device__ __forceinline__ void load_tile(uint32_t s_base, const bf16* g, long long ld, int r0, int nrows) {
    constexpr int CH = D / 8;  // 16-byte chunks per row
    for (int i = threadIdx.x; i < ROWS * CH; i += FA_THREADS) {
        const int r = i / CH, c = i % CH;
        const int row = r0 + r;
        const bool ok = row < nrows;
        const bf16* src = g + (ok ? (long long)row * ld : 0) + c * 8;
        cp_async16(s_base + swz<D>(r, c), src, ok ? 16 : 0);
    }
}

template <int D, bool CAUSAL>
__global__ void __launch_bounds__(FA_THREADS) flash_fwd_k(AttnArgs a) {
    extern __shared__ __align__(128) uint8_t fa_smem[];
    constexpr int TILE_BYTES = FA_BN * D * 2;
    const uint32_t sQ = smem_addr(fa_smem);
    const uint32_t sK = sQ + FA_BM * D * 2;        // 2 buffers
    const uint32_t sV = sK + 2 * TILE_BYTES;        // 2 buffers

    const int qtile = gridDim.x - 1 - blockIdx.x;  // longest (causal) tiles first
    const int h = blockIdx.y, b = blockIdx.z;
    const int s = h / a.hl, jl = h % a.hl;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int g = lane / 4, t4 = lane % 4;
    const long long M = (long long)a.B * a.Tq;
    const int rowlen = 3 * a.hl * D;
    const bf16* base = (const bf16*)a.qkv + s * M * rowlen + (long long)b * a.Tq * rowlen;
    const bf16* Qg = base + jl * D;
    const bf16 *Kg, *Vg;
    long long kv_ld;
    if (a.kc) {
        Kg = (const bf16*)a.kc + ((long long)b * a.H + h) * a.cap * D;
        Vg = (const bf16*)a.vc + ((long long)b * a.H + h) * a.cap * D;
        kv_ld = D;
    } else {
        Kg = base + a.hl * D + jl * D;
        Vg = base + 2 * a.hl * D + jl * D;
        kv_ld = rowlen;
    }
    const int q0 = qtile * FA_BM;
    const int nkeys = a.pos + a.Tq;
    const int kmax = CAUSAL ? min(nkeys, a.pos + q0 + FA_BM) : nkeys;
    const int n_kt = (kmax + FA_BN - 1) / FA_BN;

    load_tile<D, FA_BM>(sQ, Qg, rowlen, q0, a.Tq);
    load_tile<D, FA_BN>(sK, Kg, kv_ld, 0, kmax);
    load_tile<D, FA_BN>(sV, Vg, kv_ld, 0, kmax);
    cp_async_commit();

    // scores are kept in log2 units: x = s * scale * log2(e)
    const float sl2 = a.scale * 1.4426950408889634f;
    float o[D / 8][4];
#pragma unroll
    for (int i = 0; i < D / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    float mrow[2] = {-INFINITY, -INFINITY}, lrow[2] = {0.f, 0.f};
    uint32_t qf[D / 16][4];
    const int qrow_base = a.pos + q0 + warp * 16;  // absolute position of the warp's first row

    for (int kt = 0; kt < n_kt; ++kt) {
        const int buf = kt & 1;
        if (kt + 1 < n_kt) {
            load_tile<D, FA_BN>(sK + (buf ^ 1) * TILE_BYTES, Kg, kv_ld, (kt + 1) * FA_BN, kmax);
            load_tile<D, FA_BN>(sV + (buf ^ 1) * TILE_BYTES, Vg, kv_ld, (kt + 1) * FA_BN, kmax);
            cp_async_commit();
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncthreads();
        if (kt == 0) {
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const int r = warp * 16 + (lane % 8) + ((lane / 8) % 2) * 8;
                const int c = kk * 2 + lane / 16;
                ldsm_x4(sQ + swz<D>(r, c), qf[kk][0], qf[kk][1], qf[kk][2], qf[kk][3]);
            }
        }
        const uint32_t kb = sK + buf * TILE_BYTES, vb = sV + buf * TILE_BYTES;
        // S = Q K^T for 16 rows x 64 keys
        float sc[FA_BN / 8][4];
#pragma unroll
        for (int i = 0; i < FA_BN / 8; ++i) sc[i][0] = sc[i][1] = sc[i][2] = sc[i][3] = 0.f;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
#pragma unroll
            for (int np = 0; np < FA_BN / 16; ++np) {
                uint32_t b0, b1, b2, b3;
                const int r = np * 16 + (lane % 8) + (lane / 16) * 8;
                const int c = kk * 2 + (lane / 8) % 2;
                ldsm_x4(kb + swz<D>(r, c), b0, b1, b2, b3);
                mma_bf16(sc[2 * np], qf[kk][0], qf[kk][1], qf[kk][2], qf[kk][3], b0, b1);
                mma_bf16(sc[2 * np + 1], qf[kk][0], qf[kk][1], qf[kk][2], qf[kk][3], b2, b3);
            }
        }
        // mask (causal diagonal tiles and the ragged key tail), running max
        const int k0 = kt * FA_BN;
        const bool need_mask = (k0 + FA_BN > kmax) || (CAUSAL && k0 + FA_BN - 1 > qrow_base);
        float mx[2] = {mrow[0], mrow[1]};
#pragma unroll
        for (int i = 0; i < FA_BN / 8; ++i) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                float x = sc[i][e] * sl2;
                if (need_mask) {
                    const int key = k0 + i * 8 + 2 * t4 + (e & 1);
                    const int qpos = qrow_base + g + (e >> 1) * 8;
                    if (key >= kmax || (CAUSAL && key > qpos)) x = -INFINITY;
                }
                sc[i][e] = x;
                mx[e >> 1] = fmaxf(mx[e >> 1], x);
            }
        }
        float corr[2];
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 1));
            mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 2));
            corr[r] = mrow[r] == -INFINITY ? 0.f : exp2f(mrow[r] - mx[r]);
            mrow[r] = mx[r];
        }
        const float mb[2] = {mx[0] == -INFINITY ? 0.f : mx[0], mx[1] == -INFINITY ? 0.f : mx[1]};
        float rs[2] = {0.f, 0.f};
#pragma unroll
        for (int i = 0; i < FA_BN / 8; ++i) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float p = exp2f(sc[i][e] - mb[e >> 1]);
                sc[i][e] = p;
                rs[e >> 1] += p;
            }
        }
#pragma unroll
        for (int r = 0; r < 2; ++r) lrow[r] = lrow[r] * corr[r] + rs[r];
#pragma unroll
        for (int i = 0; i < D / 8; ++i) {
            o[i][0] *= corr[0];
            o[i][1] *= corr[0];
            o[i][2] *= corr[1];
            o[i][3] *= corr[1];
        }
        // O += P V: P's accumulator layout is the A-operand layout of the next mma
#pragma unroll
        for (int kk = 0; kk < FA_BN / 16; ++kk) {
            const uint32_t a0 = pack2(sc[2 * kk][0], sc[2 * kk][1]);
            const uint32_t a1 = pack2(sc[2 * kk][2], sc[2 * kk][3]);
            const uint32_t a2 = pack2(sc[2 * kk + 1][0], sc[2 * kk + 1][1]);
            const uint32_t a3 = pack2(sc[2 * kk + 1][2], sc[2 * kk + 1][3]);
#pragma unroll
            for (int np = 0; np < D / 16; ++np) {
                uint32_t b0, b1, b2, b3;
                const int r = kk * 16 + (lane % 8) + ((lane / 8) % 2) * 8;
                const int c = np * 2 + lane / 16;
                ldsm_x4_t(vb + swz<D>(r, c), b0, b1, b2, b3);
                mma_bf16(o[2 * np], a0, a1, a2, a3, b0, b1);
                mma_bf16(o[2 * np + 1], a0, a1, a2, a3, b2, b3);
            }
        }
        __syncthreads();  // the buffer is refilled by the next iteration's loads
    }
    // finish: row sums across the quad, normalise, store bf16
    float inv[2];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        float l = lrow[r];
        l += __shfl_xor_sync(0xffffffffu, l, 1);
        l += __shfl_xor_sync(0xffffffffu, l, 2);
        inv[r] = 1.f / l;
    }
    bf16* out = (bf16*)a.out + s * M * (a.hl * D) + (long long)b * a.Tq * (a.hl * D) + jl * D;
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        const int t = q0 + warp * 16 + g + r * 8;
        if (t < a.Tq) {
            uint32_t* dst = reinterpret_cast<uint32_t*>(out + (long long)t * (a.hl * D));
#pragma unroll
            for (int i = 0; i < D / 8; ++i) dst[i * 4 + t4] = pack2(o[i][2 * r] * inv[r], o[i][2 * r + 1] * inv[r]);
        }
    }
}

template <int D, bool CAUSAL>
cudaError_t flash_launch(const AttnArgs& a, cudaStream_t st) {
    constexpr int SMEM = FA_BM * D * 2 + 4 * FA_BN * D * 2;
    static bool attr[64] = {false};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && !attr[dev]) {
        cudaError_t e = cudaFuncSetAttribute(flash_fwd_k<D, CAUSAL>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
        if (e != cudaSuccess) return e;
        attr[dev] = true;
    }
    dim3 grid((a.Tq + FA_BM - 1) / FA_BM, a.H, a.B);
    flash_fwd_k<D, CAUSAL><<<grid, FA_THREADS, SMEM, st>>>(a);
    return cudaGetLastError();
}

}  // namespace

bool tc_attention_supported(const AttnArgs& a) { return a.is_bf16 && (a.dh == 64 || a.dh == 128); }

cudaError_t tc_attention(const AttnArgs& a, cudaStream_t st) {
    if (a.dh == 128) return a.causal ? flash_launch<128, true>(a, st) : flash_launch<128, false>(a, st);
    if (a.dh == 64) return a.causal ? flash_launch<64, true>(a, st) : flash_launch<64, false>(a, st);
    return cudaErrorNotSupported;
}

}  // namespace tpk
