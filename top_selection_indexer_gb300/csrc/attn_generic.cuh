// Host-side interface of the sparse-attention kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace tsi {

struct AttnArgs {
    const void* q;  // [B,T,H,Dqk] bf16
    const void* k;  // [B,S,Hkv,Dqk] bf16
    const void* v;  // [B,S,Hkv,Dv] bf16 or nullptr (value = first Dv dims of k)
    int B, T, S, H, Hkv, Dqk, Dv;
    float scale;
    const int32_t* idx;  // [B,T,topk]
    int topk;
    const int32_t* kv_len;
    void* out;  // [B,T,H,Dv] bf16
    unsigned* err;
    float* lse = nullptr;  // [B,T,H] fp32 or nullptr: ln sum_s exp(scale * Q.K) (-inf: no key)
};

bool attn_generic_supported(int H, int Hkv, int Dqk, int Dv, bool v_from_k);
void attn_generic_split_plan(int rows, int topk, int* n_splits, int* per_split);
size_t attn_generic_workspace_bytes(int B, int T, int H, int Dv, int topk);
cudaError_t launch_attn_generic(const AttnArgs& a, void* workspace, cudaStream_t st);

// Merge split partials (slot = (row*n_splits + split)*H + h: unnormalized O [Dv], then
// (max, sum) in base-2 units) into bf16 rows of a.out.
cudaError_t launch_attn_combine(const AttnArgs& a, int n_splits, const float* part_o,
                                const float* part_ml, cudaStream_t st);

}  // namespace tsi
