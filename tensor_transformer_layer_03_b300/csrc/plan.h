// Host-side plan record shared by the C-ABI translation units.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "tp.h"

struct tp_plan_s {
    int d, H, dh, f, tp, hl, fl, granule, up_rows;
    tp_act act;
    tp_dtype dtype;
    int esize;
    // pre-norm variant (tp_plan_create_llama): RMSNorm before attention and
    // FFN, rotary embedding of Q and K (rope_theta 0: none)
    int llama;
    float eps, rope_theta;
    size_t off_qkv, off_o, off_up, off_down, packed_bytes;
};

namespace tpk {

inline bool misaligned16(const void* p) { return p && (reinterpret_cast<uintptr_t>(p) & 15u) != 0; }

// TP_OK for cudaSuccess; otherwise records the CUDA error text for
// tp_last_cuda_error() and returns TP_ERR_CUDA.
tp_status status_from_cuda(cudaError_t e);

}  // namespace tpk
