// attn_tc.cu -- union attention on tcgen05 tensor cores (placeholder until the
// kernel lands): the variant reports an unsupported launch.
#include "qsa_common.cuh"

namespace qsa {
cudaError_t launch_attn_tc(const AttnArgs&, cudaStream_t) { return cudaErrorNotSupported; }
}  // namespace qsa
