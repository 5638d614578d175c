// Host-side interface of the cross-layer top-k overlap kernel.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace tsi {

// inter[r] = |S_a(r) ∩ S_b(r)|, card_a[r] = |S_a(r)| for rows r of two [rows][topk]
// index buffers (entries < 0 are padding).
cudaError_t launch_topk_overlap(const int32_t* idx_a, const int32_t* idx_b, int rows, int topk,
                                int32_t* inter, int32_t* card_a, unsigned* err,
                                cudaStream_t st);

}  // namespace tsi
