// Tensor-core GEMM (tcgen05 + TMEM + TMA) -- not wired yet.
#include "kernels.h"

namespace tpk {
bool tc_gemm_supported(int, int, int) { return false; }
cudaError_t tc_gemm(const TcGemm&, int*, cudaStream_t) { return cudaErrorNotSupported; }
bool tc_attention_supported(const AttnArgs&) { return false; }
cudaError_t tc_attention(const AttnArgs&, cudaStream_t) { return cudaErrorNotSupported; }
}  // namespace tpk
