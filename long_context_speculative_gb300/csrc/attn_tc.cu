// Tensor-core (tcgen05 + TMA) history kernel of verify attention.
#include "attn.cuh"

namespace rapid {

bool attn_prefix_tc_supported(const AttnParams&, int) { return false; }

cudaError_t launch_attn_prefix_tc(const AttnParams&, cudaStream_t) { return cudaErrorNotSupported; }

}  // namespace rapid
