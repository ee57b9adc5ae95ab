// Split kernel, tensor-core variant for a shared latent KV (D_qk 576, D_v 512).
// Not built yet: every MLA-shaped problem reports DA_ERR_UNSUPPORTED.
#include "common.cuh"

namespace da {

bool mla_supported(int) { return false; }
int mla_ctas_per_sm() { return 1; }
cudaError_t launch_split_mla(const Launch&, int, cudaStream_t) { return cudaErrorNotSupported; }

}  // namespace da
