// Tensor-core sparse MQA attention over the shared index rows (tcgen05 / TMEM).
#include "kernels_tc.cuh"

namespace tsi {

bool tc_attn_supported(int, int, int, int, bool) { return false; }
size_t tc_attn_workspace_bytes(int, int, int, int, int) { return 0; }
cudaError_t launch_attn_tc(const AttnArgs&, void*, cudaStream_t) { return cudaErrorNotSupported; }

}  // namespace tsi
