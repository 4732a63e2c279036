// Prefill attention on the 5th-generation tensor cores (bf16 in, fp32
// softmax and accumulation), for sm_103a.
//
// Per shard, head and query tile: O = softmax(Q K^T / sqrt(d_head) + mask) V
// with the online (running max / running sum) softmax, so the T x T score
// matrix never reaches memory.  Heads are independent: no shard talks to
// another (undercodenews.com/?p=110319, "the Original": each GPU computes
// attention locally for its heads).
//
// One CTA = one (sequence, head) and two 128-row query tiles that take turns
// on the tensor core, 320 threads:
//   warp 0     TMA producer: both Q tiles once, then K_j, V_j (128 keys x
//              d_head, 128-byte swizzle) into a 5-slot shared-memory ring;
//   warp 1     TMEM allocator and MMA issuer (one thread):
//                S_t  = Q_t K_j^T          (M 128, N 128 keys, K = d_head)
//                O_t += P_t V_j            (M 128, N = d_head, K = 128 keys;
//                                           P read from TMEM as the A
//                                           operand, V read MN-major straight
//                                           from the TMA tile, no transpose)
//              issued in the order PV_0(j), S_0(j+1), PV_1(j), S_1(j+1), so
//              the tensor core works on one tile while the other's softmax
//              runs;
//   warps 2-5  softmax of tile 0, warps 6-9 softmax of tile 1: one thread per
//              query row (its TMEM lane) loads the row of S, applies scale and
//              mask, updates the running max, rescales its O row in TMEM when
//              the max grew by more than 2^8 (otherwise the stale max is kept;
//              the factor cancels in O / l), writes P = 2^(s - m) as bf16
//              pairs back over the first 64 columns of its row of S (the A
//              operand of the next P V) and adds P to its running sum; at the
//              end it normalises O by the sum and stores the bf16 row.
// TMEM: S_0 at column 0, S_1 at 128 (P_t over the first 64 columns of S_t),
// O_0 at 256, O_1 at 256 + d_head.
// Every mbarrier wait is bounded (tp_set_wait_timeout_ns of %globaltimer, 2 s
// by default): on expiry the kernel records a device error, raises a CTA
// abort flag, drains its MMAs and frees TMEM before returning.
#include <atomic>
#include <math.h>

#include "common.cuh"
#include "kernels.h"
#include "tc_ptx.cuh"

namespace tpk {

namespace {

using namespace ptx;

constexpr int AT_ROWS = 128;   // query rows per tile (MMA M)
constexpr int AT_KEYS = 128;   // keys per step (MMA N of S, K of P V)
constexpr int AT_SLOTS = 5;    // K/V ring slots
constexpr int AT_THREADS = 320;
constexpr int HALF_BYTES = 128 * 64 * 2;  // one 128-row x 64-column swizzled half tile
constexpr float RESCALE_LOG2 = 8.0f;      // rescale O only when the max grows by > 2^8

template <int D>
struct Cfg {
    static constexpr int TILE = 128 * D * 2;  // a Q, K or V tile: D/64 halves
    static constexpr int Q_OFF = 0;
    static constexpr int RING_OFF = Q_OFF + 2 * TILE;
    static constexpr int BAR_OFF = RING_OFF + AT_SLOTS * TILE;
    static constexpr int SMEM = BAR_OFF + 256 + 1024;  // + barriers + alignment slack
    static constexpr uint32_t TMEM_COLS = 512;
};

struct Params {
    int n_pairs;          // pairs of query tiles per (sequence, head)
    int H, B, hl, Tq, pos, causal, nkeys;
    int cached;           // K/V from the cache maps (else from the QKV buffer)
    float scale_log2;     // softmax scale * log2(e)
    bf16* out;            // [tp][B*Tq][hl*D]
    long long out_shard;
    int out_ld;
    int* err;
    unsigned long long timeout_ns;
};

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Three-input maximum and paired fp32 arithmetic (one instruction for two
// lanes of work): the softmax thread issues about a third fewer
// instructions per score.  Pairs are (first, second) = (low, high) word.
__device__ __forceinline__ float max3f(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}
__device__ __forceinline__ unsigned long long f2(float a, float b) {
    unsigned long long r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
    return r;
}
__device__ __forceinline__ void f2split(unsigned long long r, float& a, float& b) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(r));
}
__device__ __forceinline__ unsigned long long fma2(unsigned long long a, unsigned long long b, unsigned long long c) {
    unsigned long long d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ unsigned long long add2(unsigned long long a, unsigned long long b) {
    unsigned long long d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

// K-major operand: `bytes` into the tile along K (a multiple of 32 below 128
// selects the 16-element K step inside the swizzle row; 64-column halves
// follow each other HALF_BYTES apart).
__device__ __forceinline__ uint64_t kmajor_desc(uint32_t tile, int k_elem) {
    return sw128_desc(tile + (uint32_t)(k_elem / 64) * HALF_BYTES + (uint32_t)(k_elem % 64) * 2, 16, 1024);
}

template <int D>
__global__ void __launch_bounds__(AT_THREADS, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, Params p) {
    using C = Cfg<D>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::BAR_OFF);
    uint64_t* q_full = bars;                 // 1
    uint64_t* kv_full = bars + 1;            // AT_SLOTS
    uint64_t* kv_empty = kv_full + AT_SLOTS; // AT_SLOTS
    uint64_t* s_full = kv_empty + AT_SLOTS;  // 2
    uint64_t* p_full = s_full + 2;           // 2
    uint64_t* o_full = p_full + 2;           // 2
    uint64_t* drain = o_full + 2;            // 1
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    griddep_launch_dependents();  // the next kernel may set up while this one runs
    const int hb = p.H * p.B;
    const int pair = p.n_pairs - 1 - (int)(blockIdx.x / hb);  // longest (causal) work first
    const int head = (int)(blockIdx.x % hb) % p.H;
    const int b = (int)(blockIdx.x % hb) / p.H;
    const int s = head / p.hl, jl = head % p.hl;

    // query tile t covers rows q0(t) .. q0(t)+127 of the sequence and needs
    // key tiles 0 .. nkt(t)-1
    auto q0 = [&](int t) { return pair * 2 * AT_ROWS + t * AT_ROWS; };
    auto nkt = [&](int t) {
        if (q0(t) >= p.Tq) return 0;
        const int kmax = p.causal ? min(p.nkeys, p.pos + q0(t) + AT_ROWS) : p.nkeys;
        return (kmax + AT_KEYS - 1) / AT_KEYS;
    };
    const bool valid1 = q0(1) < p.Tq;
    const int n_kt = nkt(valid1 ? 1 : 0);  // key tiles loaded (tile 1 needs every one of them)
    const int last_t = valid1 ? 1 : 0;     // the last tile to use each K_j / V_j

    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        for (int i = 0; i < AT_SLOTS; ++i) {
            mbar_init(&kv_full[i], 1);
            mbar_init(&kv_empty[i], 1);
        }
        for (int t = 0; t < 2; ++t) {
            mbar_init(&s_full[t], 1);
            mbar_init(&p_full[t], 4);
            mbar_init(&o_full[t], 1);
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        fence_async_smem();
    }
    if (warp == 1) tmem_alloc(tmem_slot, C::TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    griddep_wait();  // Q/K/V and the cache were written by the previous kernels
    const uint32_t tmem_base = *tmem_slot;
    const uint32_t sQ = smem_u32(smem + C::Q_OFF);
    const uint32_t sRing = smem_u32(smem + C::RING_OFF);

    // column of head jl's Q / K / V in a QKV row, and the map coordinates
    const int rowq = jl * D;
    const int c2 = p.cached ? head : b;
    const int c3 = p.cached ? b : s;
    const int kcol = p.cached ? 0 : (p.hl + jl) * D;
    const int vcol = p.cached ? 0 : (2 * p.hl + jl) * D;

    if (warp == 0) {
        if (lane == 0) {
            bool ok = true;
            mbar_expect_tx(q_full, (valid1 ? 2 : 1) * C::TILE);
            for (int t = 0; t < (valid1 ? 2 : 1); ++t) {
                for (int h = 0; h < D / 64; ++h)
                    tma_load_4d(sQ + t * C::TILE + h * HALF_BYTES, &tmQ, smem_u32(q_full), rowq + h * 64, q0(t), b,
                                s);
            }
            for (int i = 0; i < 2 * n_kt && ok; ++i) {
                const int slot = i % AT_SLOTS;
                const uint32_t ph = (uint32_t)(i / AT_SLOTS) & 1u;
                if (!mbar_wait(&kv_empty[slot], ph ^ 1u, abort_flag, p.err, p.timeout_ns)) {
                    ok = false;
                    break;
                }
                const int j = i >> 1;
                const bool is_v = i & 1;
                const CUtensorMap* map = is_v ? &tmV : &tmK;
                const int col = is_v ? vcol : kcol;
                mbar_expect_tx(&kv_full[slot], C::TILE);
                for (int h = 0; h < D / 64; ++h)
                    tma_load_4d(sRing + slot * C::TILE + h * HALF_BYTES, map, smem_u32(&kv_full[slot]), col + h * 64,
                                j * AT_KEYS, c2, c3);
            }
            if (!ok) {
                const unsigned long long t0 = globaltimer();
                while (globaltimer() - t0 < 1000000ull) __nanosleep(1000);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t IDESC_S = idesc_bf16(AT_ROWS, AT_KEYS, false);
            constexpr uint32_t IDESC_O = idesc_bf16(AT_ROWS, D, true);
            const int nkt0 = nkt(0), nkt1 = nkt(1);
            // descriptor bases; the start-address field counts 16-byte units,
            // so a byte offset o inside the tile is + (o >> 4)
            const uint64_t dq0 = sw128_desc(sQ, 16, 1024), dq1 = sw128_desc(sQ + C::TILE, 16, 1024);
            const uint64_t dk = sw128_desc(sRing, 16, 1024);              // K tiles: K-major over d_head
            const uint64_t dv = sw128_desc(sRing, HALF_BYTES, 1024);      // V tiles: MN-major (d_head)
            bool ok = mbar_wait(q_full, 0, abort_flag, p.err, p.timeout_ns);
            tc_fence_after();
            int kv_seen = -1;  // ring items known to have landed
            // step -1 issues S_t(0); step j >= 0 issues P V_t(j) then S_t(j+1), t = 0, 1
            for (int j = -1; j < n_kt && ok; ++j) {
#pragma unroll 1
                for (int t = 0; t < 2 && ok; ++t) {
                    const int nk = t ? nkt1 : nkt0;
                    if (j >= 0 && j < nk) {
                        // P V_t(j): P from TMEM (bf16 pairs over the first half of S_t)
                        const int item = 2 * j + 1;
                        while (ok && kv_seen < item) {
                            const int n = kv_seen + 1;
                            ok = mbar_wait(&kv_full[n % AT_SLOTS], (uint32_t)(n / AT_SLOTS) & 1u, abort_flag, p.err,
                                           p.timeout_ns);
                            kv_seen = n;
                        }
                        ok = ok && mbar_wait(&p_full[t], (uint32_t)j & 1u, abort_flag, p.err, p.timeout_ns);
                        if (!ok) break;
                        tc_fence_after();
                        const int slot = item % AT_SLOTS;
                        const uint64_t vd = dv + (uint64_t)((slot * C::TILE) >> 4);
                        const uint32_t p_t = tmem_base + t * AT_KEYS;
                        const uint32_t o_t = tmem_base + 2 * AT_KEYS + t * D;
#pragma unroll
                        for (int kk = 0; kk < AT_KEYS / 16; ++kk)
                            umma_f16_ta(o_t, p_t + kk * 8, vd + (uint64_t)(kk * 128), IDESC_O,
                                        (j > 0 || kk > 0) ? 1u : 0u);
                        if (t == last_t) umma_commit(&kv_empty[slot]);
                        if (j == nk - 1) umma_commit(&o_full[t]);
                    }
                    if (j + 1 < nk) {
                        // S_t(j+1) = Q_t K_{j+1}^T
                        const int item = 2 * (j + 1);
                        while (ok && kv_seen < item) {
                            const int n = kv_seen + 1;
                            ok = mbar_wait(&kv_full[n % AT_SLOTS], (uint32_t)(n / AT_SLOTS) & 1u, abort_flag, p.err,
                                           p.timeout_ns);
                            kv_seen = n;
                        }
                        if (!ok) break;
                        tc_fence_after();
                        const int slot = item % AT_SLOTS;
                        const uint64_t kd = dk + (uint64_t)((slot * C::TILE) >> 4);
                        const uint64_t qd = t ? dq1 : dq0;
#pragma unroll
                        for (int kk = 0; kk < D / 16; ++kk) {
                            const uint64_t off = (uint64_t)((kk / 4) * (HALF_BYTES >> 4) + (kk % 4) * 2);
                            umma_f16(tmem_base + t * AT_KEYS, qd + off, kd + off, IDESC_S, kk > 0 ? 1u : 0u);
                        }
                        umma_commit(&s_full[t]);
                        if (t == last_t) umma_commit(&kv_empty[slot]);
                    }
                }
            }
            // drain: every MMA issued here completes before TMEM is freed
            umma_commit(drain);
            const uint32_t a = smem_u32(drain);
            const unsigned long long t0 = globaltimer();
            while (!mbar_try_wait(a, 0)) {
                if (globaltimer() - t0 > drain_limit_ns(p.timeout_ns)) {
                    record_error(p.err, DEV_ERR_TIMEOUT);
                    break;
                }
            }
        }
    } else {
        // softmax warps: tile t, TMEM lane quarter q (a warp may only touch
        // lanes 32*(warp % 4) .. +31)
        const int t = (warp - 2) / 4;
        const int quarter = warp & 3;
        const int row = quarter * 32 + lane;  // row of the tile = TMEM lane
        const int q0t = q0(t), nkt_t = nkt(t);
        if (nkt_t > 0) {
            const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
            const uint32_t tS = tmem_base + lane_off + t * AT_KEYS;
            const uint32_t tO = tmem_base + lane_off + 2 * AT_KEYS + t * D;
            const int qpos = p.pos + q0t + row;          // absolute position of this query
            const int warp_qmin = p.pos + q0t + quarter * 32;
            float m_used = -INFINITY, l = 0.f;
            bool ok = true;
            for (int j = 0; j < nkt_t; ++j) {
                if (!mbar_wait_warp(&s_full[t], (uint32_t)j & 1u, abort_flag, p.err, p.timeout_ns)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                // this row of S, all 128 columns in one TMEM round trip; scores
                // stay raw, the scale is folded into the exponent below
                float sv[AT_KEYS];
                {
                    uint32_t r[4][32];
#pragma unroll
                    for (int c = 0; c < 4; ++c) tmem_ld32_nowait(tS + 32 * c, r[c]);
                    tmem_ld_wait();
#pragma unroll
                    for (int c = 0; c < 4; ++c)
#pragma unroll
                        for (int i = 0; i < 32; ++i) sv[32 * c + i] = __uint_as_float(r[c][i]);
                }
                const int k0 = j * AT_KEYS;
                const bool masked = (k0 + AT_KEYS > p.nkeys) || (p.causal && k0 + AT_KEYS - 1 > warp_qmin);
                if (masked) {
                    const int lim = (p.causal ? min(p.nkeys - 1, qpos) : p.nkeys - 1) - k0;  // last visible column
#pragma unroll
                    for (int i = 0; i < AT_KEYS; ++i)
                        if (i > lim) sv[i] = -INFINITY;
                }
                // row max over 8 independent chains, two new scores per step
                float m8[8];
#pragma unroll
                for (int c = 0; c < 8; ++c) m8[c] = fmaxf(sv[2 * c], sv[2 * c + 1]);
#pragma unroll
                for (int k = 1; k < AT_KEYS / 16; ++k)
#pragma unroll
                    for (int c = 0; c < 8; ++c) m8[c] = max3f(m8[c], sv[16 * k + 2 * c], sv[16 * k + 2 * c + 1]);
                const float mx = fmaxf(max3f(m8[0], m8[1], m8[2]), max3f(m8[3], m8[4], max3f(m8[5], m8[6], m8[7]))) *
                                 p.scale_log2;
                // keep the stale max unless the row max grew by more than 2^8
                const bool grow = j == 0 || mx > m_used + RESCALE_LOG2;
                const float m_new = grow ? fmaxf(m_used, mx) : m_used;
                const float corr = (j > 0 && grow) ? ex2(m_used - m_new) : 1.f;
                m_used = m_new;
                const float neg_m = m_used == -INFINITY ? 0.f : -m_used;
                const unsigned long long scale2 = f2(p.scale_log2, p.scale_log2), negm2 = f2(neg_m, neg_m);
                // row sum in 4 paired accumulators: pair k holds the partial
                // sums of the columns 2i, 2i + 1 with i % 4 = k
                unsigned long long rs2[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) rs2[k] = 0ull;
                // P = 2^(s - m) as bf16 pairs written back over the first 64
                // columns of this row of S (in registers already), where the
                // P V product reads its A operand
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    uint32_t pk[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        float a0, a1;
                        f2split(fma2(f2(sv[32 * q + 2 * i], sv[32 * q + 2 * i + 1]), scale2, negm2), a0, a1);
                        const float e0 = ex2(a0), e1 = ex2(a1);
                        rs2[i & 3] = add2(rs2[i & 3], f2(e0, e1));
                        pk[i] = pack_bf16x2(e0, e1);
                    }
                    tmem_st16u(tS + 16 * q, pk);
                }
                float rs8[8];
#pragma unroll
                for (int k = 0; k < 4; ++k) f2split(rs2[k], rs8[2 * k], rs8[2 * k + 1]);
                const float rs = ((rs8[0] + rs8[1]) + (rs8[2] + rs8[3])) + ((rs8[4] + rs8[5]) + (rs8[6] + rs8[7]));
                // the scores are dead here: rescale this row of O (rare) before
                // the next P V accumulates into it
                if (__any_sync(0xffffffffu, corr != 1.f)) {
#pragma unroll 1
                    for (int c = 0; c < D / 32; ++c) {
                        float ov[32];
                        tmem_ld32(tO + 32 * c, ov);
#pragma unroll
                        for (int i = 0; i < 32; ++i) ov[i] *= corr;
                        tmem_st32(tO + 32 * c, ov);
                    }
                    tmem_st_wait();
                }
                l = l * corr;
                l += rs;
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&p_full[t]);
            }
            if (ok && mbar_wait_warp(&o_full[t], 0, abort_flag, p.err, p.timeout_ns)) {
                tc_fence_after();
                const float inv = 1.f / l;
                const bool row_ok = q0t + row < p.Tq;
                bf16* dst = p.out + s * p.out_shard + ((long long)b * p.Tq + q0t + row) * p.out_ld + jl * D;
#pragma unroll 1
                for (int c = 0; c < D / 32; ++c) {
                    float ov[32];
                    tmem_ld32(tO + 32 * c, ov);
                    if (row_ok) {
                        uint4* d4 = reinterpret_cast<uint4*>(dst + 32 * c);
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            d4[q] = make_uint4(pack_bf16x2(ov[8 * q] * inv, ov[8 * q + 1] * inv),
                                               pack_bf16x2(ov[8 * q + 2] * inv, ov[8 * q + 3] * inv),
                                               pack_bf16x2(ov[8 * q + 4] * inv, ov[8 * q + 5] * inv),
                                               pack_bf16x2(ov[8 * q + 6] * inv, ov[8 * q + 7] * inv));
                    }
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem_base, C::TMEM_COLS);
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static std::atomic<EncodeTiledFn> fn{nullptr};  // racing first calls store the same address
    EncodeTiledFn f = fn.load();
    if (!f) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess) {
            f = reinterpret_cast<EncodeTiledFn>(p);
            fn.store(f);
        }
    }
    return f;
}

// 4-D bf16 tensor [d3][d2][d1][d0] (d0 contiguous), box {64, 128, 1, 1},
// 128-byte swizzle; reads outside the tensor fill zeros.
bool make_map4(CUtensorMap* m, const void* base, const uint64_t (&dims)[4], const uint64_t (&strides_bytes)[3]) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t d[4] = {dims[0], dims[1], dims[2], dims[3]};
    cuuint64_t st[3] = {strides_bytes[0], strides_bytes[1], strides_bytes[2]};
    cuuint32_t box[4] = {64, 128, 1, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), d, st, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D>
cudaError_t attn_launch(const AttnArgs& a, int* dev_err, cudaStream_t st) {
    using C = Cfg<D>;
    static std::atomic<bool> smem_set[64];  // per device; racing first calls set the same attribute
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && !smem_set[dev].load()) {
        cudaError_t e = cudaFuncSetAttribute(attn_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
        if (e != cudaSuccess) return e;
        smem_set[dev].store(true);
    }
    const uint64_t rowlen = 3ull * a.hl * D;
    const uint64_t M = (uint64_t)a.B * a.Tq;
    CUtensorMap mq, mk, mv;
    // QKV buffer viewed as [tp][B][Tq][3*hl*D]
    const uint64_t qdims[4] = {rowlen, (uint64_t)a.Tq, (uint64_t)a.B, (uint64_t)(a.H / a.hl)};
    const uint64_t qstr[3] = {rowlen * 2, (uint64_t)a.Tq * rowlen * 2, M * rowlen * 2};
    if (!make_map4(&mq, a.qkv, qdims, qstr)) return cudaErrorInvalidValue;
    const int nkeys = a.pos + a.Tq;
    if (a.kc) {
        // cache [B][H][cap][D], cut at the last valid key so the rows past it
        // read as zeros
        const uint64_t kdims[4] = {(uint64_t)D, (uint64_t)nkeys, (uint64_t)a.H, (uint64_t)a.B};
        const uint64_t kstr[3] = {(uint64_t)D * 2, (uint64_t)a.cap * D * 2, (uint64_t)a.H * a.cap * D * 2};
        if (!make_map4(&mk, a.kc, kdims, kstr) || !make_map4(&mv, a.vc, kdims, kstr)) return cudaErrorInvalidValue;
    } else {
        mk = mq;
        mv = mq;
    }
    Params p{};
    p.n_pairs = (a.Tq + 2 * AT_ROWS - 1) / (2 * AT_ROWS);
    p.H = a.H;
    p.B = a.B;
    p.hl = a.hl;
    p.Tq = a.Tq;
    p.pos = a.pos;
    p.causal = a.causal;
    p.nkeys = nkeys;
    p.cached = a.kc != nullptr;
    p.scale_log2 = a.scale * 1.4426950408889634f;
    p.out = (bf16*)a.out;
    p.out_shard = (long long)M * a.hl * D;
    p.out_ld = a.hl * D;
    p.err = dev_err;
    p.timeout_ns = wait_timeout_ns();
    const long long grid = (long long)p.n_pairs * a.H * a.B;
    if (grid <= 0 || grid > 0x7fffffffLL) return cudaErrorInvalidValue;
    // programmatic dependent launch: CTAs may start while the previous kernel
    // of the stream finishes (the kernel waits before its first read)
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    cfg.blockDim = dim3(AT_THREADS, 1, 1);
    cfg.dynamicSmemBytes = C::SMEM;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, attn_tc_kernel<D>, mq, mk, mv, p);
}

}  // namespace

bool tc_attention_supported(const AttnArgs& a) {
    // TMA needs 16-byte aligned row strides: 3*hl*dh and dh bf16 elements are
    // multiples of 8 for dh in {64, 128}
    return a.is_bf16 && (a.dh == 64 || a.dh == 128);
}

cudaError_t tc_attention(const AttnArgs& a, int* dev_err, cudaStream_t st) {
    if (a.dh == 128) return attn_launch<128>(a, dev_err, st);
    if (a.dh == 64) return attn_launch<64>(a, dev_err, st);
    return cudaErrorNotSupported;
}

}  // namespace tpk
