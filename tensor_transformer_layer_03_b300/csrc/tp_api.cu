// C ABI of the tensor-parallel block: plan, validation, layout and dispatch.
//
// Everything here runs on the host.  Calls validate their arguments before
// enqueuing anything, then launch the kernels of pack.cu, simt.cu,
// gemm_tc.cu, attn_tc.cu and decode.cu on the caller's stream.
#include <atomic>
#include <limits.h>
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include <new>

#include <nvtx3/nvToolsExt.h>

#include "kernels.h"
#include "plan.h"
#include "tp.h"

// First device-side error recorded by a bounded wait (0 = none).  Kernels
// receive its address; tp_sync_status reads and clears it.
__device__ int g_tp_device_error;

namespace {

thread_local char g_last_cuda_error[256] = "";

constexpr unsigned long long DEFAULT_WAIT_TIMEOUT_NS = 2000000000ull;  // 2 s
std::atomic<unsigned long long> g_wait_timeout_ns{DEFAULT_WAIT_TIMEOUT_NS};

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

bool misaligned(const void* p) { return tpk::misaligned16(p); }

tp_status cuda_status(cudaError_t e) { return tpk::status_from_cuda(e); }

int* device_error_word() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return nullptr;
    static std::atomic<int*> addr[64];  // per device; racing first calls store the same address
    if (dev < 0 || dev >= 64) return nullptr;
    int* a = addr[dev].load();
    if (!a) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_tp_device_error) != cudaSuccess) return nullptr;
        a = static_cast<int*>(p);
        addr[dev].store(a);
    }
    return a;
}

// NVTX range for the lifetime of a scope: every ABI call and every block
// step shows up by name in nsys / ncu (--nvtx) timelines.  Without an
// attached tool the push and pop are no-ops.
struct Range {
    explicit Range(const char* name) { nvtxRangePushA(name); }
    ~Range() { nvtxRangePop(); }
    Range(const Range&) = delete;
    Range& operator=(const Range&) = delete;
};

struct Workspace {
    size_t qkv, attn, hf32, hact, u, scratch, gemm, rs, rope, total;
};

// Split-tile scratch of the tensor-core GEMMs (fp32 partials and their
// counters; bf16 plans, M past the weight-streaming range); 0 when no GEMM
// of this shape would use it.
size_t linear_scratch_bytes(const tp_plan_s* p, long long M) {
    if (p->dtype != TP_BF16 || M <= tpk::GEMV_PREFERRED_MAX_M) return 0;
    return tpk::tc_gemm_scratch_bytes();
}

size_t attn_scratch_bytes(const tp_plan_s* p, int batch, int seq_q) {
    if (seq_q != 1) return 0;
    return align_up((size_t)batch * p->H * tpk::DECODE_MAX_SPLITS * (p->dh + 2) * sizeof(float), 256);
}

Workspace workspace_layout(const tp_plan_s* p, int batch, int seq) {
    const size_t M = (size_t)batch * seq, es = p->esize;
    Workspace w;
    size_t o = 0;
    w.qkv = o;   o = align_up(o + (size_t)p->tp * M * 3 * p->hl * p->dh * es, 1024);
    w.attn = o;  o = align_up(o + (size_t)p->tp * M * p->hl * p->dh * es, 1024);
    w.hf32 = o;  o = align_up(o + M * p->d * sizeof(float), 1024);
    w.hact = o;  o = align_up(o + M * p->d * es, 1024);
    w.u = o;     o = align_up(o + (size_t)p->tp * M * p->fl * es, 1024);
    w.scratch = o; o = align_up(o + attn_scratch_bytes(p, batch, seq), 1024);
    w.gemm = o;    o = align_up(o + linear_scratch_bytes(p, (long long)batch * seq), 1024);
    w.rs = o;      o = align_up(o + (p->llama ? 2 * M * sizeof(float) : 0), 1024);  // 1/rms of x and of H
    w.rope = o;    o = align_up(o + (p->llama ? (size_t)seq * (p->dh / 2) * sizeof(float2) : 0), 1024);
    w.total = o;
    return w;
}

const char* ptr_at(const void* base, size_t off) { return static_cast<const char*>(base) + off; }
char* ptr_at(void* base, size_t off) { return static_cast<char*>(base) + off; }

// Block workspace plus the two plan-dtype activation buffers of a stack.
size_t stack_workspace_bytes(const tp_plan_s* p, int batch, int seq) {
    return workspace_layout(p, batch, seq).total + 2 * align_up((size_t)batch * seq * p->d * p->esize, 1024);
}

// Argument checks of tp_attention_heads that need no buffer contents; the
// whole-block calls run them before enqueuing anything.
tp_status attention_check(const tp_plan_s* p, int batch, int seq_q, const void* k_cache, const void* v_cache,
                          int cache_cap, int cache_pos) {
    if ((k_cache == nullptr) != (v_cache == nullptr)) return TP_ERR_NULL_ARG;
    if (batch <= 0 || seq_q <= 0 || cache_pos < 0) return TP_ERR_INVALID_DIM;
    if ((long long)batch * seq_q > INT_MAX) return TP_ERR_INVALID_DIM;  // token rows are int in the kernels
    const bool cached = k_cache != nullptr;
    if (!cached && cache_pos != 0) return TP_ERR_INVALID_DIM;
    if (cached && (cache_cap <= 0 || (long long)cache_pos + seq_q > cache_cap)) return TP_ERR_INVALID_DIM;
    if (misaligned(k_cache) || misaligned(v_cache)) return TP_ERR_ALIGNMENT;
    if (p->dh != 32 && p->dh != 64 && p->dh != 128) return TP_ERR_UNSUPPORTED;
    return TP_OK;
}

}  // namespace

// The block S1..S5 on a validated workspace layout; out_act (nullable)
// receives a plan-dtype copy of Y (the next layer's input in a stack).
// Sequence-parallel layout of the block's input x and output Y: token row
// m in slice m / slice_rows, slices x_stride / y_stride elements apart
// (slice_rows 0: the plain [M][d] layout).
struct SeqLayout {
    int slice_rows = 0;
    long long x_stride = 0, y_stride = 0;
};

static tp_status block_forward_impl(tp_plan_t p, const void* x, int batch, int seq, int causal, void* k_cache,
                                    void* v_cache, int cache_cap, int cache_pos, const void* packed, void* workspace,
                                    const Workspace& w, void* out_f32, void* out_act, void* stream,
                                    const SeqLayout& sp = SeqLayout());

// Pre-norm extras of a column-parallel launch: row scales (1/rms of the
// input rows) and the rotary embedding of the QKV output.
struct ColumnExtras {
    const float* row_scale = nullptr;
    const float2* rope_cs = nullptr;  // rotary (cos, sin) table, NULL: no rotation
    int rope_seq = 1;
    int slice_rows = 0;               // sequence-parallel input: rows gathered from slices
    long long a_slice = 0;            // elements between the input's slices
    bool* counters_zero = nullptr;    // chain of launches on one scratch (see tpk::tc_gemm)
};

static tp_status row_linear_impl(tp_plan_t p, int which, const void* in_shards, int M, const void* packed,
                                 const void* residual, void* out_f32, void* out_act, void* scratch,
                                 size_t scratch_bytes, cudaStream_t st, int slice_rows = 0, long long res_slice = 0,
                                 long long out_slice = 0, bool* counters_zero = nullptr);

static tp_status column_linear_impl(tp_plan_t p, int which, const void* x, int M, const void* packed,
                                    void* out_shards, void* scratch, size_t scratch_bytes, const ColumnExtras& ex,
                                    cudaStream_t st);

unsigned long long tpk::wait_timeout_ns() { return g_wait_timeout_ns.load(); }

// The linear launches: argument records of the tensor-core / weight-streaming
// kernels, and which kernel a call runs (shared by the calls and by
// tp_linear_schedule, so the schedule query reports what the calls do).
enum LinearKernel { LK_TC = 0, LK_GEMV_MMA = 1, LK_GEMV = 2, LK_SIMT = 3 };

static tpk::TcGemm column_gemm(const tp_plan_s* p, int which, const void* x, int M, const void* packed,
                               void* out_shards, const ColumnExtras& ex) {
    const bool qkv = which == TP_QKV;
    const int N = qkv ? 3 * p->hl * p->dh : p->up_rows;  // W rows per shard
    const int n_out = qkv ? N : p->fl;                     // output columns per shard
    tpk::TcGemm g{};
    g.epi = qkv ? tpk::EPI_STORE : (p->act == TP_ACT_SWIGLU ? tpk::EPI_SWIGLU : tpk::EPI_GELU);
    g.A = x;
    g.a_shard = 0;
    g.lda = p->d;
    g.W = ptr_at(packed, qkv ? p->off_qkv : p->off_up);
    g.w_shard = (long long)N * p->d;
    g.M = M;
    g.N = N;
    g.K = p->d;
    g.shards = p->tp;
    g.reduce = 0;
    g.out = out_shards;
    g.out_shard = (long long)M * n_out;
    g.ldo = n_out;
    g.granule = p->granule;
    g.row_scale = ex.row_scale;
    if (ex.rope_cs) {
        g.rope_cols = 2 * p->hl * p->dh;  // the Q and K heads of each shard's [Q | K | V] row
        g.rope_dh = p->dh;
        g.rope_seq = ex.rope_seq;
        g.rope_cs = ex.rope_cs;
    }
    g.slice_rows = ex.slice_rows;
    g.a_slice = ex.a_slice;
    return g;
}

static tpk::TcGemm row_gemm(const tp_plan_s* p, int which, const void* in_shards, int M, const void* packed,
                            const void* residual, void* out_f32, void* out_act) {
    const bool attn = which == TP_ATTN_OUT;
    const int ks = attn ? p->hl * p->dh : p->fl;
    tpk::TcGemm g{};
    g.epi = tpk::EPI_ROW_REDUCE;
    g.A = in_shards;
    g.a_shard = (long long)M * ks;
    g.lda = ks;
    g.W = ptr_at(packed, attn ? p->off_o : p->off_down);
    g.w_shard = (long long)p->d * ks;
    g.M = M;
    g.N = p->d;
    g.K = ks;
    g.shards = p->tp;
    g.reduce = 1;
    g.out = out_f32;
    g.ldo = p->d;
    g.out2 = out_act;
    g.residual = residual;
    g.residual_f32 = attn ? (p->dtype == TP_FP32) : 1;
    return g;
}

static LinearKernel pick_linear(const tp_plan_s* p, const tpk::TcGemm& g) {
    if (p->dtype != TP_BF16) return LK_SIMT;
    const int M = g.M;
    if (M >= 2 && M <= tpk::GEMV_MMA_DISPATCH_ROWS && tpk::gemv_mma_supported(g)) return LK_GEMV_MMA;
    const bool tc_ok = tpk::tc_gemm_supported(M, g.N, g.K) && (g.epi != tpk::EPI_SWIGLU || g.granule == 32);
    if (tpk::gemv_supported(g) && (M <= tpk::GEMV_PREFERRED_MAX_M || !tc_ok)) return LK_GEMV;
    return tc_ok ? LK_TC : LK_SIMT;
}

// Launch the bf16 linear `g` on the kernel pick_linear chose.
static tp_status run_linear(LinearKernel k, const tpk::TcGemm& g, void* scratch, size_t scratch_bytes,
                            cudaStream_t st, bool* counters_zero = nullptr) {
    switch (k) {
        case LK_GEMV_MMA: return cuda_status(tpk::gemv_mma(g, st));
        case LK_GEMV: return cuda_status(tpk::gemv(g, device_error_word(), st));
        case LK_TC:
            return cuda_status(
                tpk::tc_gemm(g, device_error_word(), scratch, scratch ? scratch_bytes : 0, st, counters_zero));
        default: return TP_ERR_UNSUPPORTED;
    }
}

tp_status tpk::status_from_cuda(cudaError_t e) {
    if (e == cudaSuccess) return TP_OK;
    strncpy(g_last_cuda_error, cudaGetErrorString(e), sizeof(g_last_cuda_error) - 1);
    return TP_ERR_CUDA;
}

static tp_status block_forward_impl(tp_plan_t p, const void* x, int batch, int seq, int causal, void* k_cache,
                                    void* v_cache, int cache_cap, int cache_pos, const void* packed, void* workspace,
                                    const Workspace& w, void* out_f32, void* out_act, void* stream,
                                    const SeqLayout& sp) {
    const int M = batch * seq;
    // sequence-parallel: x and Y in slices; H stays in the workspace as
    // contiguous slices (slice s = rows s * slice_rows.., the plain layout)
    const long long h_slice = (long long)sp.slice_rows * p->d;
    void* qkv = ptr_at(workspace, w.qkv);
    void* attn = ptr_at(workspace, w.attn);
    void* hf32 = ptr_at(workspace, w.hf32);
    void* hact = ptr_at(workspace, w.hact);
    void* u = ptr_at(workspace, w.u);
    void* gs = w.rs > w.gemm ? ptr_at(workspace, w.gemm) : nullptr;
    const size_t gsb = w.rs - w.gemm;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    float* r1 = reinterpret_cast<float*>(ptr_at(workspace, w.rs));
    float* r2 = r1 + M;
    // the four linears share the split-tile scratch: the first that splits
    // clears its counters, and each completed launch leaves them zero
    bool cz = false;
    ColumnExtras ex1, ex2;
    ex1.counters_zero = ex2.counters_zero = &cz;
    if (p->llama) {
        const Range r("RMSNorm(X) + rotary table");
        // RMSNorm of x (its gain is in the packed QKV rows) and, in the same
        // launch, the rotary table of positions cache_pos + t, applied in
        // the QKV epilogue
        tpk::RopeTable rt = {};
        rt.cs = reinterpret_cast<float2*>(ptr_at(workspace, w.rope));
        rt.seq = seq;
        rt.pos0 = cache_pos;
        rt.half = p->dh / 2;
        rt.log2_theta = p->rope_theta > 0.f ? log2f(p->rope_theta) : 0.f;
        const bool rope = p->rope_theta > 0.f;
        cudaError_t e = tpk::rms_rows(x, p->dtype == TP_FP32, M, p->d, p->eps, r1, rope ? &rt : nullptr, st,
                                      sp.slice_rows, sp.x_stride);
        if (e != cudaSuccess) return cuda_status(e);
        ex1.row_scale = r1;
        ex1.rope_cs = rope ? rt.cs : nullptr;
        ex1.rope_seq = seq;
        ex2.row_scale = r2;
    }
    ex1.slice_rows = sp.slice_rows;  // S1 gathers x from its slices
    ex1.a_slice = sp.x_stride;
    tp_status s;
    {
        const Range r("S1 column QKV");
        s = column_linear_impl(p, TP_QKV, x, M, packed, qkv, gs, gsb, ex1, st);
    }
    if (s != TP_OK) return s;
    {
        const Range r("S2 attention");
        s = tp_attention_heads(p, qkv, batch, seq, causal, k_cache, v_cache, cache_cap, cache_pos, attn,
                               ptr_at(workspace, w.scratch), w.gemm - w.scratch, stream);
    }
    if (s != TP_OK) return s;
    {
        const Range r("S3 row O + reduce");
        s = row_linear_impl(p, TP_ATTN_OUT, attn, M, packed, x, hf32, hact, gs, gsb, st, sp.slice_rows, sp.x_stride,
                            h_slice, &cz);
    }
    if (s != TP_OK) return s;
    if (p->llama) {  // RMSNorm of H: scale from the fp32 H, the GEMM reads its plan-dtype copy
        const Range r("RMSNorm(H)");
        cudaError_t e = tpk::rms_rows(hf32, 1, M, p->d, p->eps, r2, nullptr, st);
        if (e != cudaSuccess) return cuda_status(e);
    }
    {
        const Range r("S4 column FFN-up");
        s = column_linear_impl(p, TP_FFN_UP, hact, M, packed, u, gs, gsb, ex2, st);
    }
    if (s != TP_OK) return s;
    const Range r("S5 row FFN-down + reduce");
    return row_linear_impl(p, TP_FFN_DOWN, u, M, packed, hf32, out_f32, out_act, gs, gsb, st, sp.slice_rows, h_slice,
                           sp.y_stride, &cz);
}

extern "C" {

const char* tp_status_string(tp_status s) {
    switch (s) {
        case TP_OK: return "TP_OK";
        case TP_ERR_NULL_ARG: return "TP_ERR_NULL_ARG";
        case TP_ERR_INVALID_DIM: return "TP_ERR_INVALID_DIM";
        case TP_ERR_DEGREE_RANGE: return "TP_ERR_DEGREE_RANGE";
        case TP_ERR_HEADS_NOT_DIVISIBLE: return "TP_ERR_HEADS_NOT_DIVISIBLE";
        case TP_ERR_FFN_NOT_DIVISIBLE: return "TP_ERR_FFN_NOT_DIVISIBLE";
        case TP_ERR_DMODEL_NOT_DIVISIBLE: return "TP_ERR_DMODEL_NOT_DIVISIBLE";
        case TP_ERR_ALIGNMENT: return "TP_ERR_ALIGNMENT";
        case TP_ERR_WORKSPACE_TOO_SMALL: return "TP_ERR_WORKSPACE_TOO_SMALL";
        case TP_ERR_UNSUPPORTED: return "TP_ERR_UNSUPPORTED";
        case TP_ERR_CUDA: return "TP_ERR_CUDA";
        case TP_ERR_DEVICE_TIMEOUT: return "TP_ERR_DEVICE_TIMEOUT";
    }
    return "TP_ERR_UNKNOWN";
}

const char* tp_last_cuda_error(void) { return g_last_cuda_error; }

tp_status tp_plan_create_ex(int d_model, int n_heads, int d_ffn, int tp_degree, tp_act act, tp_dtype dtype,
                            tp_plan_t* out) {
    if (!out) return TP_ERR_NULL_ARG;
    *out = nullptr;
    if (d_model <= 0 || n_heads <= 0 || d_ffn <= 0) return TP_ERR_INVALID_DIM;
    if (tp_degree < 1) return TP_ERR_DEGREE_RANGE;
    if (d_model % n_heads != 0) return TP_ERR_DMODEL_NOT_DIVISIBLE;
    if (tp_degree > n_heads) return TP_ERR_DEGREE_RANGE;
    if (n_heads % tp_degree != 0) return TP_ERR_HEADS_NOT_DIVISIBLE;
    if (d_ffn % tp_degree != 0) return TP_ERR_FFN_NOT_DIVISIBLE;
    if ((act != TP_ACT_GELU && act != TP_ACT_SWIGLU) || (dtype != TP_BF16 && dtype != TP_FP32))
        return TP_ERR_UNSUPPORTED;
    const int dh = d_model / n_heads, fl = d_ffn / tp_degree;
    if (d_model % 8 || dh % 8 || fl % 8) return TP_ERR_ALIGNMENT;

    tp_plan_s* p = new (std::nothrow) tp_plan_s;
    if (!p) return TP_ERR_UNSUPPORTED;
    p->d = d_model;
    p->H = n_heads;
    p->dh = dh;
    p->f = d_ffn;
    p->tp = tp_degree;
    p->hl = n_heads / tp_degree;
    p->fl = fl;
    p->granule = fl % 32 == 0 ? 32 : (fl % 16 == 0 ? 16 : 8);
    p->act = act;
    p->dtype = dtype;
    p->esize = dtype == TP_BF16 ? 2 : 4;
    p->up_rows = act == TP_ACT_SWIGLU ? 2 * fl : fl;
    p->llama = 0;
    p->eps = 0.f;
    p->rope_theta = 0.f;
    const size_t es = p->esize, d = d_model, T = tp_degree;
    size_t o = 0;
    p->off_qkv = o;  o = align_up(o + T * 3 * p->hl * dh * d * es, 1024);
    p->off_o = o;    o = align_up(o + T * d * p->hl * dh * es, 1024);
    p->off_up = o;   o = align_up(o + T * p->up_rows * d * es, 1024);
    p->off_down = o; o = align_up(o + T * d * fl * es, 1024);
    p->packed_bytes = o;
    *out = p;
    return TP_OK;
}

tp_status tp_plan_create(int d_model, int n_heads, int d_ffn, int tp_degree, tp_plan_t* out) {
    return tp_plan_create_ex(d_model, n_heads, d_ffn, tp_degree, TP_ACT_SWIGLU, TP_BF16, out);
}

tp_status tp_plan_create_llama(int d_model, int n_heads, int d_ffn, int tp_degree, float rms_eps, float rope_theta,
                               tp_plan_t* out) {
    if (!out) return TP_ERR_NULL_ARG;
    *out = nullptr;
    if (!(rms_eps > 0.f) || !isfinite(rms_eps) || !(rope_theta >= 0.f) || !isfinite(rope_theta))
        return TP_ERR_INVALID_DIM;
    const tp_status s = tp_plan_create_ex(d_model, n_heads, d_ffn, tp_degree, TP_ACT_SWIGLU, TP_BF16, out);
    if (s != TP_OK) return s;
    tp_plan_s* p = *out;
    if (p->granule != 32) {  // the tensor-core SwiGLU epilogue pairs 32-row gate/up blocks
        delete p;
        *out = nullptr;
        return TP_ERR_UNSUPPORTED;
    }
    p->llama = 1;
    p->eps = rms_eps;
    p->rope_theta = rope_theta;
    return TP_OK;
}

void tp_plan_destroy(tp_plan_t plan) { delete plan; }

tp_status tp_plan_sizes(tp_plan_t p, int batch, int seq, size_t* packed_weight_bytes, size_t* workspace_bytes) {
    if (!p) return TP_ERR_NULL_ARG;
    if (batch <= 0 || seq <= 0) return TP_ERR_INVALID_DIM;
    if (packed_weight_bytes) *packed_weight_bytes = p->packed_bytes;
    if (workspace_bytes) *workspace_bytes = workspace_layout(p, batch, seq).total;
    return TP_OK;
}

tp_status tp_attention_scratch_bytes(tp_plan_t p, int batch, int seq_q, int cache_cap, size_t* bytes) {
    if (!p || !bytes) return TP_ERR_NULL_ARG;
    if (batch <= 0 || seq_q <= 0 || cache_cap < 0) return TP_ERR_INVALID_DIM;
    *bytes = attn_scratch_bytes(p, batch, seq_q);
    return TP_OK;
}

tp_status tp_linear_scratch_bytes(tp_plan_t p, int M, size_t* bytes) {
    if (!p || !bytes) return TP_ERR_NULL_ARG;
    if (M <= 0) return TP_ERR_INVALID_DIM;
    *bytes = linear_scratch_bytes(p, M);
    return TP_OK;
}

tp_status tp_shard_weights(tp_plan_t p, const void* Wq, const void* Wk, const void* Wv, const void* Wo,
                           const void* W1_or_Wgate, const void* Wup, const void* Wdown, void* packed,
                           void* stream) {
    const Range trace_("tp_shard_weights");
    if (!p || !Wq || !Wk || !Wv || !Wo || !W1_or_Wgate || !Wdown || !packed) return TP_ERR_NULL_ARG;
    if ((p->act == TP_ACT_SWIGLU) != (Wup != nullptr)) return TP_ERR_NULL_ARG;
    const void* all[] = {Wq, Wk, Wv, Wo, W1_or_Wgate, Wup, Wdown, packed};
    for (const void* q : all)
        if (misaligned(q)) return TP_ERR_ALIGNMENT;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int es = p->esize;
    cudaError_t e = tpk::pack_qkv(es, Wq, Wk, Wv, ptr_at(packed, p->off_qkv), p->tp, p->hl, p->dh, p->d, st);
    if (e == cudaSuccess) e = tpk::pack_cols(es, Wo, ptr_at(packed, p->off_o), p->tp, p->d, p->hl * p->dh, st);
    if (e == cudaSuccess)
        e = tpk::pack_up(es, W1_or_Wgate, Wup, ptr_at(packed, p->off_up), p->tp, p->fl, p->d, p->granule, st);
    if (e == cudaSuccess) e = tpk::pack_cols(es, Wdown, ptr_at(packed, p->off_down), p->tp, p->d, p->fl, st);
    return cuda_status(e);
}

tp_status tp_shard_weights_llama(tp_plan_t p, const void* Wq, const void* Wk, const void* Wv, const void* Wo,
                                 const void* Wgate, const void* Wup, const void* Wdown, const void* g_attn,
                                 const void* g_ffn, void* packed, void* stream) {
    const Range trace_("tp_shard_weights_llama");
    if (!p || !g_attn || !g_ffn) return TP_ERR_NULL_ARG;
    if (!p->llama) return TP_ERR_UNSUPPORTED;
    if (misaligned(g_attn) || misaligned(g_ffn)) return TP_ERR_ALIGNMENT;
    const tp_status s = tp_shard_weights(p, Wq, Wk, Wv, Wo, Wgate, Wup, Wdown, packed, stream);
    if (s != TP_OK) return s;
    // fold the norms' gains into the columns of the rows that read the
    // normed activations: all QKV rows and all gate/up rows
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e = tpk::scale_cols(p->esize, ptr_at(packed, p->off_qkv), (long long)p->tp * 3 * p->hl * p->dh,
                                    p->d, g_attn, st);
    if (e == cudaSuccess)
        e = tpk::scale_cols(p->esize, ptr_at(packed, p->off_up), (long long)p->tp * p->up_rows, p->d, g_ffn, st);
    return cuda_status(e);
}

tp_status tp_column_linear(tp_plan_t p, int which, const void* x, int M, const void* packed, void* out_shards,
                           void* scratch, size_t scratch_bytes, void* stream) {
    const Range trace_("tp_column_linear");
    if (!p || !x || !packed || !out_shards) return TP_ERR_NULL_ARG;
    if (M <= 0 || (which != TP_QKV && which != TP_FFN_UP)) return TP_ERR_INVALID_DIM;
    if (misaligned(x) || misaligned(packed) || misaligned(out_shards) || misaligned(scratch))
        return TP_ERR_ALIGNMENT;
    // a pre-norm plan's column linears need the norm scales and positions
    // that only the whole-block calls compute
    if (p->llama) return TP_ERR_UNSUPPORTED;
    return column_linear_impl(p, which, x, M, packed, out_shards, scratch, scratch_bytes, ColumnExtras(),
                              static_cast<cudaStream_t>(stream));
}

}  // extern "C"

static tp_status column_linear_impl(tp_plan_t p, int which, const void* x, int M, const void* packed,
                                    void* out_shards, void* scratch, size_t scratch_bytes, const ColumnExtras& ex,
                                    cudaStream_t st) {
    const bool qkv = which == TP_QKV;
    const int N = qkv ? 3 * p->hl * p->dh : p->up_rows;  // W rows per shard
    const int n_out = qkv ? N : p->fl;                     // output columns per shard
    const void* W = ptr_at(packed, qkv ? p->off_qkv : p->off_up);
    const int epi = qkv ? tpk::EPI_STORE : (p->act == TP_ACT_SWIGLU ? tpk::EPI_SWIGLU : tpk::EPI_GELU);
    if (p->dtype == TP_BF16) {
        const tpk::TcGemm g = column_gemm(p, which, x, M, packed, out_shards, ex);
        if (ex.slice_rows > 0)  // gathered rows: the tensor-core GEMM reads them through its tensor map
            return tpk::tc_gemm_supported(M, g.N, g.K)
                       ? run_linear(LK_TC, g, scratch, scratch_bytes, st, ex.counters_zero)
                       : TP_ERR_UNSUPPORTED;
        const LinearKernel k = pick_linear(p, g);
        if (k != LK_SIMT) return run_linear(k, g, scratch, scratch_bytes, st, ex.counters_zero);
    }
    if (ex.slice_rows > 0) return TP_ERR_UNSUPPORTED;
    if (ex.row_scale) return TP_ERR_UNSUPPORTED;  // (plan creation rules this out for pre-norm plans)
    tpk::SimtGemm g{};
    g.epi = epi;
    g.is_bf16 = p->dtype == TP_BF16;
    g.A = x;
    g.a_shard = 0;
    g.lda = p->d;
    g.W = W;
    g.w_shard = (long long)N * p->d;
    g.ldw = p->d;
    g.M = M;
    g.N = N;
    g.K = p->d;
    g.col_shards = p->tp;
    g.red_shards = 1;
    g.out = out_shards;
    g.out_shard = (long long)M * n_out;
    g.ldo = n_out;
    g.granule = p->granule;
    return cuda_status(tpk::simt_gemm(g, st));
}

extern "C" {

tp_status tp_row_linear_reduce(tp_plan_t p, int which, const void* in_shards, int M, const void* packed,
                               const void* residual, void* out_f32, void* out_act, void* scratch,
                               size_t scratch_bytes, void* stream) {
    const Range trace_("tp_row_linear_reduce");
    if (!p || !in_shards || !packed || !out_f32) return TP_ERR_NULL_ARG;
    if (M <= 0 || (which != TP_ATTN_OUT && which != TP_FFN_DOWN)) return TP_ERR_INVALID_DIM;
    if (misaligned(in_shards) || misaligned(packed) || misaligned(residual) || misaligned(out_f32) ||
        misaligned(out_act) || misaligned(scratch))
        return TP_ERR_ALIGNMENT;
    return row_linear_impl(p, which, in_shards, M, packed, residual, out_f32, out_act, scratch, scratch_bytes,
                           static_cast<cudaStream_t>(stream));
}

}  // extern "C"

static tp_status row_linear_impl(tp_plan_t p, int which, const void* in_shards, int M, const void* packed,
                                 const void* residual, void* out_f32, void* out_act, void* scratch,
                                 size_t scratch_bytes, cudaStream_t st, int slice_rows, long long res_slice,
                                 long long out_slice, bool* counters_zero) {
    const bool attn = which == TP_ATTN_OUT;
    const int ks = attn ? p->hl * p->dh : p->fl;
    const void* W = ptr_at(packed, attn ? p->off_o : p->off_down);
    const int res_f32 = attn ? (p->dtype == TP_FP32) : 1;
    if (p->dtype == TP_BF16) {
        tpk::TcGemm g = row_gemm(p, which, in_shards, M, packed, residual, out_f32, out_act);
        if (slice_rows > 0) {  // reduce-scatter: the tensor-core GEMM writes each row into its slice
            g.slice_rows = slice_rows;
            g.res_slice = res_slice;
            g.out_slice = out_slice;
            return tpk::tc_gemm_supported(M, g.N, g.K)
                       ? run_linear(LK_TC, g, scratch, scratch_bytes, st, counters_zero)
                       : TP_ERR_UNSUPPORTED;
        }
        const LinearKernel k = pick_linear(p, g);
        if (k != LK_SIMT) return run_linear(k, g, scratch, scratch_bytes, st, counters_zero);
    }
    if (slice_rows > 0) return TP_ERR_UNSUPPORTED;
    tpk::SimtGemm g{};
    g.epi = tpk::EPI_ROW_REDUCE;
    g.is_bf16 = p->dtype == TP_BF16;
    g.A = in_shards;
    g.a_shard = (long long)M * ks;
    g.lda = ks;
    g.W = W;
    g.w_shard = (long long)p->d * ks;
    g.ldw = ks;
    g.M = M;
    g.N = p->d;
    g.K = ks;
    g.col_shards = 1;
    g.red_shards = p->tp;
    g.out = out_f32;
    g.ldo = p->d;
    g.out2 = out_act;
    g.residual = residual;
    g.residual_f32 = res_f32;
    return cuda_status(tpk::simt_gemm(g, st));
}

// Checks of a sequence-parallel call: bf16 plan, M token rows in tp slices
// of M / tp rows (a multiple of 8), slices `stride` elements apart (at
// least a slice, a multiple of 8).
static tp_status seq_check(const tp_plan_s* p, long long M, long long stride) {
    if (p->dtype != TP_BF16) return TP_ERR_UNSUPPORTED;
    if (M <= 0 || M % p->tp != 0) return TP_ERR_INVALID_DIM;
    const long long ms = M / p->tp;
    if (ms % 8 != 0 || stride % 8 != 0) return TP_ERR_ALIGNMENT;
    if (stride < ms * p->d) return TP_ERR_INVALID_DIM;
    return TP_OK;
}

extern "C" {

tp_status tp_column_linear_gather(tp_plan_t p, int which, const void* x_slices, long long slice_stride, int M,
                                  const void* packed, void* out_shards, void* scratch, size_t scratch_bytes,
                                  void* stream) {
    const Range trace_("tp_column_linear_gather");
    if (!p || !x_slices || !packed || !out_shards) return TP_ERR_NULL_ARG;
    if (M <= 0 || (which != TP_QKV && which != TP_FFN_UP)) return TP_ERR_INVALID_DIM;
    if (misaligned(x_slices) || misaligned(packed) || misaligned(out_shards) || misaligned(scratch))
        return TP_ERR_ALIGNMENT;
    if (p->llama) return TP_ERR_UNSUPPORTED;
    const tp_status c = seq_check(p, M, slice_stride);
    if (c != TP_OK) return c;
    ColumnExtras ex;
    ex.slice_rows = M / p->tp;
    ex.a_slice = slice_stride;
    return column_linear_impl(p, which, x_slices, M, packed, out_shards, scratch, scratch_bytes, ex,
                              static_cast<cudaStream_t>(stream));
}

tp_status tp_row_linear_reduce_scatter(tp_plan_t p, int which, const void* in_shards, int M, const void* packed,
                                       const void* residual_slices, void* out_f32_slices, void* out_act_slices,
                                       long long slice_stride, void* scratch, size_t scratch_bytes, void* stream) {
    const Range trace_("tp_row_linear_reduce_scatter");
    if (!p || !in_shards || !packed || !out_f32_slices) return TP_ERR_NULL_ARG;
    if (M <= 0 || (which != TP_ATTN_OUT && which != TP_FFN_DOWN)) return TP_ERR_INVALID_DIM;
    if (misaligned(in_shards) || misaligned(packed) || misaligned(residual_slices) || misaligned(out_f32_slices) ||
        misaligned(out_act_slices) || misaligned(scratch))
        return TP_ERR_ALIGNMENT;
    const tp_status c = seq_check(p, M, slice_stride);
    if (c != TP_OK) return c;
    return row_linear_impl(p, which, in_shards, M, packed, residual_slices, out_f32_slices, out_act_slices, scratch,
                           scratch_bytes, static_cast<cudaStream_t>(stream), M / p->tp, slice_stride, slice_stride);
}

tp_status tp_block_forward_seq(tp_plan_t p, const void* x_slices, long long x_stride, int batch, int seq,
                               int causal, void* k_cache, void* v_cache, int cache_cap, int cache_pos,
                               const void* packed, void* workspace, size_t ws_bytes, void* out_f32_slices,
                               long long y_stride, void* stream) {
    const Range trace_("tp_block_forward_seq");
    if (!p || !x_slices || !packed || !workspace || !out_f32_slices) return TP_ERR_NULL_ARG;
    if (batch <= 0 || seq <= 0) return TP_ERR_INVALID_DIM;
    if (misaligned(workspace) || misaligned(x_slices) || misaligned(packed) || misaligned(out_f32_slices))
        return TP_ERR_ALIGNMENT;
    const long long M = (long long)batch * seq;
    tp_status c = seq_check(p, M, x_stride);
    if (c == TP_OK) c = seq_check(p, M, y_stride);
    if (c != TP_OK) return c;
    const tp_status chk = attention_check(p, batch, seq, k_cache, v_cache, cache_cap, cache_pos);
    if (chk != TP_OK) return chk;
    const Workspace w = workspace_layout(p, batch, seq);
    if (ws_bytes < w.total) return TP_ERR_WORKSPACE_TOO_SMALL;
    SeqLayout sp;
    sp.slice_rows = (int)(M / p->tp);
    sp.x_stride = x_stride;
    sp.y_stride = y_stride;
    return block_forward_impl(p, x_slices, batch, seq, causal, k_cache, v_cache, cache_cap, cache_pos, packed,
                              workspace, w, out_f32_slices, nullptr, stream, sp);
}

tp_status tp_attention_heads(tp_plan_t p, const void* qkv_shards, int batch, int seq_q, int causal, void* k_cache,
                             void* v_cache, int cache_cap, int cache_pos, void* out_shards, void* scratch,
                             size_t scratch_bytes, void* stream) {
    const Range trace_("tp_attention_heads");
    if (!p || !qkv_shards || !out_shards) return TP_ERR_NULL_ARG;
    if (misaligned(qkv_shards) || misaligned(out_shards) || misaligned(scratch)) return TP_ERR_ALIGNMENT;
    const tp_status chk = attention_check(p, batch, seq_q, k_cache, v_cache, cache_cap, cache_pos);
    if (chk != TP_OK) return chk;
    const bool cached = k_cache != nullptr;
    const size_t need = cached ? attn_scratch_bytes(p, batch, seq_q) : 0;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    tpk::AttnArgs a{};
    a.is_bf16 = p->dtype == TP_BF16;
    a.qkv = qkv_shards;
    a.kc = k_cache;
    a.vc = v_cache;
    a.out = out_shards;
    a.B = batch;
    a.Tq = seq_q;
    a.H = p->H;
    a.hl = p->hl;
    a.dh = p->dh;
    a.cap = cached ? cache_cap : 0;
    a.pos = cache_pos;
    a.causal = causal ? 1 : 0;
    a.scale = 1.0f / sqrtf((float)p->dh);
    const bool split_kv = cached && seq_q == 1 && need > 0;
    if (split_kv && !scratch) return TP_ERR_NULL_ARG;
    if (split_kv && scratch_bytes < need) return TP_ERR_WORKSPACE_TOO_SMALL;
    cudaError_t e = cudaSuccess;
    if (cached && !split_kv) {  // (the single-token path appends inside its kernels)
        e = tpk::kv_append(a, k_cache, v_cache, st);
        if (e != cudaSuccess) return cuda_status(e);
    }
    if (split_kv) {
        e = tpk::decode_attention(a, static_cast<float*>(scratch), st);
    } else if (a.is_bf16 && tpk::tc_attention_supported(a)) {
        e = tpk::tc_attention(a, device_error_word(), st);
    } else {
        e = tpk::simt_attention(a, st);
    }
    return cuda_status(e);
}

tp_status tp_block_forward(tp_plan_t p, const void* x, int batch, int seq, int causal, void* k_cache,
                           void* v_cache, int cache_cap, int cache_pos, const void* packed, void* workspace,
                           size_t ws_bytes, void* out_f32, void* stream) {
    const Range trace_("tp_block_forward");
    if (!p || !x || !packed || !workspace || !out_f32) return TP_ERR_NULL_ARG;
    if (batch <= 0 || seq <= 0) return TP_ERR_INVALID_DIM;
    if (misaligned(workspace) || misaligned(x) || misaligned(packed) || misaligned(out_f32)) return TP_ERR_ALIGNMENT;
    const tp_status chk = attention_check(p, batch, seq, k_cache, v_cache, cache_cap, cache_pos);
    if (chk != TP_OK) return chk;
    const Workspace w = workspace_layout(p, batch, seq);
    if (ws_bytes < w.total) return TP_ERR_WORKSPACE_TOO_SMALL;
    return block_forward_impl(p, x, batch, seq, causal, k_cache, v_cache, cache_cap, cache_pos, packed, workspace,
                              w, out_f32, nullptr, stream);
}

tp_status tp_stack_workspace_bytes(tp_plan_t p, int batch, int seq, size_t* bytes) {
    if (!p || !bytes) return TP_ERR_NULL_ARG;
    if (batch <= 0 || seq <= 0) return TP_ERR_INVALID_DIM;
    *bytes = stack_workspace_bytes(p, batch, seq);
    return TP_OK;
}

tp_status tp_stack_forward(tp_plan_t p, int n_layers, const void* const* packed_layers, const void* x, int batch,
                           int seq, int causal, void* const* k_caches, void* const* v_caches, int cache_cap,
                           int cache_pos, void* workspace, size_t ws_bytes, void* out_f32, void* stream) {
    const Range trace_("tp_stack_forward");
    if (!p || !packed_layers || !x || !workspace || !out_f32) return TP_ERR_NULL_ARG;
    if (n_layers <= 0 || batch <= 0 || seq <= 0) return TP_ERR_INVALID_DIM;
    if ((k_caches == nullptr) != (v_caches == nullptr)) return TP_ERR_NULL_ARG;
    for (int l = 0; l < n_layers; ++l) {
        if (!packed_layers[l]) return TP_ERR_NULL_ARG;
        if (misaligned(packed_layers[l])) return TP_ERR_ALIGNMENT;
        if (k_caches && (!k_caches[l] || !v_caches[l])) return TP_ERR_NULL_ARG;
    }
    if (misaligned(workspace) || misaligned(x) || misaligned(out_f32)) return TP_ERR_ALIGNMENT;
    for (int l = 0; l < n_layers; ++l) {
        const tp_status chk = attention_check(p, batch, seq, k_caches ? k_caches[l] : nullptr,
                                              v_caches ? v_caches[l] : nullptr, cache_cap, cache_pos);
        if (chk != TP_OK) return chk;
    }
    if (ws_bytes < stack_workspace_bytes(p, batch, seq)) return TP_ERR_WORKSPACE_TOO_SMALL;
    const Workspace w = workspace_layout(p, batch, seq);
    // two plan-dtype activation buffers after the block workspace: layer l
    // writes its output's copy into act[l % 2], layer l + 1 reads it
    const size_t act_bytes = align_up((size_t)batch * seq * p->d * p->esize, 1024);
    void* act[2] = {ptr_at(workspace, w.total), ptr_at(workspace, w.total + act_bytes)};
    for (int l = 0; l < n_layers; ++l) {
        char name[32];
        snprintf(name, sizeof name, "layer %d", l);
        const Range r(name);
        const void* in = l == 0 ? x : act[(l - 1) % 2];
        void* copy = l + 1 < n_layers ? act[l % 2] : nullptr;
        const tp_status s =
            block_forward_impl(p, in, batch, seq, causal, k_caches ? k_caches[l] : nullptr,
                               v_caches ? v_caches[l] : nullptr, cache_cap, cache_pos, packed_layers[l], workspace, w,
                               out_f32, copy, stream);
        if (s != TP_OK) return s;
    }
    return TP_OK;
}

void tp_set_wait_timeout_ns(unsigned long long ns) {
    g_wait_timeout_ns.store(ns ? ns : DEFAULT_WAIT_TIMEOUT_NS);
}

tp_status tp_linear_schedule(tp_plan_t p, int row, int which, int M, size_t scratch_bytes, int sms, int pair_slots,
                             tp_linear_schedule_t* out) {
    if (!p || !out) return TP_ERR_NULL_ARG;
    if (M <= 0 || sms <= 0 || pair_slots < 0 || (row != 0 && row != 1) || (which != 0 && which != 1))
        return TP_ERR_INVALID_DIM;
    static const int zero_rows[1] = {0};
    const void* fake = zero_rows;  // never dereferenced: only the shapes matter here
    const tpk::TcGemm g = row ? row_gemm(p, which, fake, M, fake, nullptr, nullptr, nullptr)
                              : column_gemm(p, which, fake, M, fake, nullptr, ColumnExtras());
    *out = tp_linear_schedule_t{};
    const LinearKernel k = pick_linear(p, g);
    out->kernel = (int)k;
    if (k == LK_TC) {
        const tpk::TcSchedule r = tpk::tc_gemm_schedule(g, scratch_bytes, sms, pair_slots);
        out->paired = r.paired;
        out->tiles = r.tiles;
        out->k_blocks_per_tile = r.kbt;
        out->whole_tiles = r.whole;
        out->parts = r.parts;
        out->items = r.items;
        out->units = r.units;
        out->scratch_bytes_touched = r.scratch_touched;
    }
    return TP_OK;
}

tp_status tp_sync_status(void* stream) {
    cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_status(e);
    int* word = device_error_word();
    if (!word) return cuda_status(cudaGetLastError());
    int h = 0;
    e = cudaMemcpy(&h, word, sizeof(int), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_status(e);
    if (h != 0) {
        const int zero = 0;
        e = cudaMemcpy(word, &zero, sizeof(int), cudaMemcpyHostToDevice);
        if (e != cudaSuccess) return cuda_status(e);
        return TP_ERR_DEVICE_TIMEOUT;
    }
    return TP_OK;
}

}  // extern "C"
