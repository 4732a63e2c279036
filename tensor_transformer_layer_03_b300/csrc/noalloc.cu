// Single-token decode attention whose split-KV scratch lives in a fixed,
// file-scope device array instead of caller-provided memory.
//
// Some callers cannot allocate device memory at the point where they run a
// decode step: code that runs inside a memory pool it does not own, a plugin
// or host framework that forbids cudaMalloc on its hot path, or a process
// whose allocator is already exhausted.  For them this entry point takes only
// the inputs and outputs; the per-chunk partials that tp_attention_heads
// keeps in the caller's `scratch` buffer go to NOALLOC_SCRATCH_BYTES of
// device memory reserved here, which every GPU that loads the library holds
// until the process exits.  The call allocates nothing (no cudaMalloc, no
// cudaFree, no allocating library routine).
#include <nvtx3/nvToolsExt.h>
#include <mutex>

#include "kernels.h"
#include "plan.h"
#include "tp.h"

namespace {

constexpr size_t NOALLOC_SCRATCH_BYTES = 8u << 20;  // 8 MiB per device

// Split-KV partials of the last call on this device.  Every call rewrites
// every slot it later reads, so nothing needs clearing between calls.
static __device__ __align__(256) float g_noalloc_scratch[NOALLOC_SCRATCH_BYTES / sizeof(float)];

constexpr int MAX_DEVICES = 64;
std::mutex g_setup_mutex;
float* g_scratch_addr[MAX_DEVICES] = {nullptr};

// Device address of g_noalloc_scratch on the current device.  In host code
// the array's name is only a host-side stand-in, so the address comes from
// cudaGetSymbolAddress, once per device, with that device current.
cudaError_t scratch_address(float** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= MAX_DEVICES) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (!g_scratch_addr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_addr[dev] = static_cast<float*>(p);
    }
    *out = g_scratch_addr[dev];
    return cudaSuccess;
}

}  // namespace

extern "C" tp_status tp_attention_decode_noalloc(tp_plan_t p, const void* qkv_shards, int batch, void* k_cache,
                                                 void* v_cache, int cache_cap, int cache_pos, void* out_shards,
                                                 void* stream) {
    // named in profiler timelines like the other calls (a no-op without a tool)
    struct Range {
        Range() { nvtxRangePushA("tp_attention_decode_noalloc"); }
        ~Range() { nvtxRangePop(); }
    } trace_;
    if (!p || !qkv_shards || !k_cache || !v_cache || !out_shards) return TP_ERR_NULL_ARG;
    if (batch <= 0 || cache_pos < 0 || cache_cap <= 0 || (long long)cache_pos + 1 > cache_cap)
        return TP_ERR_INVALID_DIM;
    if (tpk::misaligned16(qkv_shards) || tpk::misaligned16(k_cache) || tpk::misaligned16(v_cache) ||
        tpk::misaligned16(out_shards))
        return TP_ERR_ALIGNMENT;
    if (p->dh != 32 && p->dh != 64 && p->dh != 128) return TP_ERR_UNSUPPORTED;
    const size_t need = (size_t)batch * p->H * tpk::DECODE_MAX_SPLITS * (p->dh + 2) * sizeof(float);
    if (need > NOALLOC_SCRATCH_BYTES) return TP_ERR_WORKSPACE_TOO_SMALL;
    float* scratch = nullptr;
    cudaError_t e = scratch_address(&scratch);
    if (e != cudaSuccess) return tpk::status_from_cuda(e);
    tpk::AttnArgs a{};
    a.is_bf16 = p->dtype == TP_BF16;
    a.qkv = qkv_shards;
    a.kc = k_cache;
    a.vc = v_cache;
    a.out = out_shards;
    a.B = batch;
    a.Tq = 1;
    a.H = p->H;
    a.hl = p->hl;
    a.dh = p->dh;
    a.cap = cache_cap;
    a.pos = cache_pos;
    a.causal = 1;
    a.scale = 1.0f / sqrtf((float)p->dh);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    e = tpk::decode_attention(a, scratch, st);  // also appends the new token's K/V
    return tpk::status_from_cuda(e);
}
