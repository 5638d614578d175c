// Host-side interface of the indexer + top-k kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace tsi {

struct IndexerArgs {
    const void* qI;
    const void* kI;
    const void* w;
    int qk_dtype, w_dtype;
    int B, T, S, H_I, d_I, topk;
    const int32_t* kv_len;
    int32_t* idx;
    float* score;
    unsigned* err;  // device error word
};

// CUDA-core path (any supported shape).
bool generic_supported(int H_I, int d_I);
void generic_split_plan(int rows, int S, int* n_splits, int* chunk);
size_t generic_workspace_bytes(int B, int T, int S, int topk);
cudaError_t launch_indexer_generic(const IndexerArgs& a, void* workspace, cudaStream_t st);

// Merge per-split candidate lists ([rows][n_splits][topk] keys + counts) into the
// final rank-ordered rows (CUDA-core selector).
cudaError_t launch_topk_merge(int rows, int topk, int n_splits, const uint64_t* cand,
                              const int* cand_cnt, int32_t* idx, float* score, unsigned* err,
                              cudaStream_t st);

// Rank one unordered list of at most topk distinct keys per row ([rows][topk] keys +
// counts) into rank-ordered idx / score rows.
cudaError_t launch_topk_rank(int rows, int topk, const uint64_t* cand, const int* cand_cnt,
                             int32_t* idx, float* score, unsigned* err, cudaStream_t st);

}  // namespace tsi
