// Tensor-core lightning indexer + streaming top-k (tcgen05 / TMEM / TMA).
#include "kernels_tc.cuh"

namespace tsi {

bool tc_indexer_supported(int, int, int) { return false; }
size_t tc_indexer_workspace_bytes(int, int, int, int) { return 0; }
cudaError_t launch_indexer_tc(const IndexerArgs&, void*, cudaStream_t) {
    return cudaErrorNotSupported;
}

}  // namespace tsi
