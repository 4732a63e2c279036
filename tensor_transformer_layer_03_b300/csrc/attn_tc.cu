// Tensor-core attention for prefill -- not wired yet.
#include "kernels.h"

namespace tpk {
bool tc_attention_supported(const AttnArgs&) { return false; }
cudaError_t tc_attention(const AttnArgs&, cudaStream_t) { return cudaErrorNotSupported; }
}  // namespace tpk
