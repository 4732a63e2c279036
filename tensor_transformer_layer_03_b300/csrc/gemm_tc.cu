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
// Kernel structure (one persistent CTA per SM, 192 threads):
//   warp 0   TMA producer: 128x64 tile of A and 256x64 tile of W per stage,
//            128-byte swizzle, 4-stage shared-memory ring (48 KB per stage);
//   warp 1   TMEM allocator and MMA issuer: tcgen05.mma kind::f16, M=128,
//            N=256, K=16, into one of two 128x256 fp32 TMEM accumulators;
//   warps 2-5 epilogue: tcgen05.ld of the finished accumulator (each warp its
//            32-lane quarter), activation / residual, stores to global.
// The epilogue of tile i overlaps the main loop of tile i+1 (two TMEM
// accumulators = all 512 columns).  Every mbarrier wait is bounded: after
// `timeout_ns` the waiting role records TP_ERR_DEVICE_TIMEOUT's device code,
// raises a CTA-wide abort flag and leaves its loop; in-flight tensor-core
// work is drained and TMEM freed before the CTA exits.
#include <cuda.h>

#include "common.cuh"
#include "kernels.h"
#include "tc_ptx.cuh"

namespace tpk {

namespace {

constexpr int BM = 128, BN = 256, BK = 64, STAGES = 4;
constexpr int A_STAGE_BYTES = BM * BK * 2;  // 16 KB
constexpr int B_STAGE_BYTES = BN * BK * 2;  // 32 KB
constexpr int STAGE_BYTES = A_STAGE_BYTES + B_STAGE_BYTES;
constexpr int TMEM_COLS = 512;
constexpr int NUM_THREADS = 192;
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 + 256;
constexpr unsigned long long DEFAULT_TIMEOUT_NS = 2000000000ull;  // 2 s

// instruction descriptor: D fp32, A/B bf16, both K-major, M=128, N=256
constexpr uint32_t IDESC = ptx::idesc_bf16(BM, BN, false);

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
};

using namespace ptx;

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
        for (int i = 0; i < n_valid; ++i) dst[i] = __float2bfloat16_rn(v[i]);
    }
}

__global__ void __launch_bounds__(NUM_THREADS, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmW, Params p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + STAGES * STAGE_BYTES);
    uint64_t* empty = full + STAGES;
    uint64_t* tmem_full = empty + STAGES;
    uint64_t* tmem_empty = tmem_full + 2;
    uint64_t* drain = tmem_empty + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&tmem_full[b], 1);
            mbar_init(&tmem_empty[b], 4);
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                     "r"(TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const int kb_per_tile = p.reduce ? p.shards * p.k_blocks : p.k_blocks;

    if (warp == 0) {
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < p.n_tiles && ok; t += gridDim.x) {
                const int m_blk = t % p.m_blocks;
                const int rest = t / p.m_blocks;
                const int shard = p.reduce ? 0 : rest / p.n_blocks;
                const int n_blk = p.reduce ? rest : rest % p.n_blocks;
                for (int kb = 0; kb < kb_per_tile; ++kb) {
                    if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, p.err, p.timeout_ns)) {
                        ok = false;
                        break;
                    }
                    const int s = p.reduce ? kb / p.k_blocks : shard;
                    const int kk = (p.reduce ? kb % p.k_blocks : kb) * BK;
                    uint8_t* sa = smem + stage * STAGE_BYTES;
                    mbar_expect_tx(&full[stage], STAGE_BYTES);
                    tma_load_3d(smem_u32(sa), &tmA, smem_u32(&full[stage]), kk, m_blk * BM, p.reduce ? s : 0);
                    tma_load_3d(smem_u32(sa + A_STAGE_BYTES), &tmW, smem_u32(&full[stage]), kk, n_blk * BN, s);
                    if (++stage == STAGES) {
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
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            int i = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < p.n_tiles && ok; t += gridDim.x, ++i) {
                const int buf = i & 1;
                const uint32_t acc_phase = (uint32_t)(i >> 1) & 1u;
                if (!mbar_wait(&tmem_empty[buf], acc_phase ^ 1u, abort_flag, p.err, p.timeout_ns)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + (uint32_t)(buf * BN);
                for (int kb = 0; kb < kb_per_tile; ++kb) {
                    if (!mbar_wait(&full[stage], phase, abort_flag, p.err, p.timeout_ns)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sa = smem_u32(smem + stage * STAGE_BYTES);
                    const uint64_t adesc = sw128_kmajor(sa);
                    const uint64_t bdesc = sw128_kmajor(sa + A_STAGE_BYTES);
#pragma unroll
                    for (int k = 0; k < BK / 16; ++k)  // +32 bytes per K step inside the swizzle row
                        umma_f16(d_tmem, adesc + (uint64_t)(2 * k), bdesc + (uint64_t)(2 * k), IDESC,
                                  (kb > 0 || k > 0) ? 1u : 0u);
                    umma_commit(&empty[stage]);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (ok) umma_commit(&tmem_full[buf]);
            }
            // drain: wait for every MMA issued by this thread before TMEM is freed
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
        for (int t = blockIdx.x; t < p.n_tiles; t += gridDim.x, ++i) {
            const int buf = i & 1;
            const uint32_t acc_phase = (uint32_t)(i >> 1) & 1u;
            if (!mbar_wait_warp(&tmem_full[buf], acc_phase, abort_flag, p.err, p.timeout_ns)) break;
            tc_fence_after();
            const int m_blk = t % p.m_blocks;
            const int rest = t / p.m_blocks;
            const int shard = p.reduce ? 0 : rest / p.n_blocks;
            const int n_blk = p.reduce ? rest : rest % p.n_blocks;
            const int row = m_blk * BM + quarter * 32 + lane;
            const uint32_t tbase = tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(buf * BN);
            const int col_base = n_blk * BN;
            const bool row_ok = row < p.M;
            if (p.epi == EPI_SWIGLU) {
                bf16* out = (bf16*)p.out + shard * p.out_shard + (long long)row * p.ldo;
#pragma unroll 1
                for (int g = 0; g < BN / 64; ++g) {
                    float gate[32], up[32];
                    __syncwarp();
                    tmem_ld32(tbase + 64 * g, gate);
                    tmem_ld32(tbase + 64 * g + 32, up);
                    const int pc = col_base + 64 * g;  // packed column of this gate block
                    if (row_ok && pc < p.N) {
#pragma unroll
                        for (int j = 0; j < 32; ++j) gate[j] = silu(gate[j]) * up[j];
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
                                for (int j = 0; j < nv; ++j) v[j] += r[j];
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
                                for (int j = 0; j < nv; ++j) v[j] += __bfloat162float(r[j]);
                            }
                        }
                    }
                    float* o = (float*)p.out + roff + col;
                    if (nv == 32) {
#pragma unroll
                        for (int q = 0; q < 8; ++q)
                            reinterpret_cast<float4*>(o)[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
                    } else {
                        for (int j = 0; j < nv; ++j) o[j] = v[j];
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
                    if (p.epi == EPI_GELU) {
#pragma unroll
                        for (int j = 0; j < 32; ++j) v[j] = gelu_erf(v[j]);
                    }
                    store_row_bf16(out + col, v, min(32, p.N - col));
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tmem_empty[buf]);
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) {
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(TMEM_COLS)
                     : "memory");
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
    static int n[64] = {0};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) return 148;
    if (!n[dev]) cudaDeviceGetAttribute(&n[dev], cudaDevAttrMultiProcessorCount, dev);
    return n[dev] > 0 ? n[dev] : 148;
}

}  // namespace

bool tc_gemm_supported(int M, int N, int K) { return M >= 1 && N >= 1 && K >= 8 && K % 8 == 0; }

cudaError_t tc_gemm(const TcGemm& g, int* dev_err, cudaStream_t st) {
    static bool attr_set[64] = {false};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && !attr_set[dev]) {
        cudaError_t e = cudaFuncSetAttribute(tc_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
        if (e != cudaSuccess) return e;
        attr_set[dev] = true;
    }
    if (g.epi == EPI_SWIGLU && (g.granule != 32 || g.N % 64 != 0)) return cudaErrorNotSupported;
    CUtensorMap tmA, tmW;
    const uint64_t a_shards = g.reduce ? (uint64_t)g.shards : 1;
    if (!make_map(&tmA, g.A, (uint64_t)g.K, (uint64_t)g.M, a_shards, (uint64_t)g.lda * 2,
                  (uint64_t)g.M * g.lda * 2, BM))
        return cudaErrorInvalidValue;
    if (!make_map(&tmW, g.W, (uint64_t)g.K, (uint64_t)g.N, (uint64_t)g.shards, (uint64_t)g.K * 2,
                  (uint64_t)g.w_shard * 2, BN))
        return cudaErrorInvalidValue;
    Params p{};
    p.epi = g.epi;
    p.M = g.M;
    p.N = g.N;
    p.K = g.K;
    p.shards = g.shards;
    p.reduce = g.reduce;
    p.m_blocks = (g.M + BM - 1) / BM;
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
    const int grid = p.n_tiles < sm_count() ? p.n_tiles : sm_count();
    tc_gemm_kernel<<<grid, NUM_THREADS, SMEM_BYTES, st>>>(tmA, tmW, p);
    return cudaGetLastError();
}

}  // namespace tpk
