// Host-side interface of the tensor-core (tcgen05 / TMEM / TMA) kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "attn_generic.cuh"
#include "indexer_generic.cuh"

namespace tsi {

// Indexer + top-k with tcgen05 MMAs (BF16 or E4M3 inputs, H_I = 64, d_I = 128).
bool tc_indexer_supported(int qk_dtype, int H_I, int d_I);
size_t tc_indexer_workspace_bytes(int qk_dtype, int B, int T, int S, int topk,
                                  bool two_pass = false);
// Only the split (decode) candidate lists, for callers that take unordered candidates.
size_t tc_indexer_split_workspace_bytes(int qk_dtype, int B, int T, int S, int topk);
cudaError_t launch_indexer_tc(const IndexerArgs& a, void* workspace, cudaStream_t st);

// Sparse MQA attention over a 576-d latent (value = first 512 dims), H = 64.
bool tc_attn_supported(int H, int Hkv, int Dqk, int Dv, bool v_from_k);
size_t tc_attn_workspace_bytes(int B, int T, int H, int Dv, int topk);
cudaError_t launch_attn_tc(const AttnArgs& a, void* workspace, cudaStream_t st);

// Group-centroid KL target of a Full layer's indexer over the group's layers (H = 64,
// Dqk = 576 latent keys), from the layers' queries, keys and attention log-partitions.
constexpr int kMaxIndexKlLayers = 8;
struct IndexKlArgs {
    int n_layers;
    const void* const* q;  // [n_layers] of [B,T,64,576] bf16
    const void* const* k;  // [n_layers] of [B,S,576] bf16
    const float* const* lse;  // [n_layers] of [B,T,64] fp32
    int B, T, S;
    float scale;
    const int32_t* idx;  // [B,T,topk]
    const float* score;  // [B,T,topk]
    int topk;
    const int32_t* kv_len;
    float* loss;  // [B,T]
    float* grad;  // [B,T,topk] or nullptr
    float* pbar;  // [B,T,topk] or nullptr
    unsigned* err;
};
bool tc_index_kl_supported(int H, int Dqk);

// One thread waits on an mbarrier that nothing completes; the bounded wait runs out and
// sets kErrTimeout in `err` (self-test of the failure path).
cudaError_t launch_wait_timeout_probe(unsigned* err, cudaStream_t st);
cudaError_t launch_index_kl_tc(const IndexKlArgs& a, cudaStream_t st);

}  // namespace tsi
