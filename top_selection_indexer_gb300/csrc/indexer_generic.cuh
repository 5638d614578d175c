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
    // Key shards (context parallelism): the keys kI[b, 0 .. S) sit at positions
    // key_offset .. key_offset + S - 1 of a cache of S_total keys (0 = S); query positions
    // and the positions in the results are those of the whole cache.
    int64_t key_offset = 0;
    int S_total = 0;
    // Non-null: each row's top-k leaves as unordered 64-bit rank keys [B*T][topk] with
    // counts [B*T] instead of rank-ordered idx / score.
    uint64_t* out_cand = nullptr;
    int* out_cnt = nullptr;
    // Tensor-core path with several query rows per sequence: store every score for a
    // second, selecting pass instead of selecting inside the scoring kernel (the default,
    // where no score reaches HBM).
    bool two_pass = false;
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

// General merge: list l of row r holds cand_cnt[r * cnt_row + l * cnt_list] keys at
// cand + r * row_stride + l * list_stride.  Writes rank-ordered idx / score, or (out_keys
// non-null) each row's top-k as unordered keys [rows][topk] with counts [rows].
cudaError_t launch_topk_merge_strided(int rows, int topk, int n_lists, const uint64_t* cand,
                                      int64_t row_stride, int64_t list_stride,
                                      const int* cand_cnt, int64_t cnt_row, int64_t cnt_list,
                                      int32_t* idx, float* score, uint64_t* out_keys,
                                      int* out_cnt, unsigned* err, cudaStream_t st);

// The same with each row's lists split into groups of lists_per_group, one block per
// (row, group): output row r * groups + g holds group g's top-k of row r as unordered keys
// (out_keys required when there is more than one group).  append_cap > 0: each group's
// top-k is appended instead to row r's list out_keys[r * append_cap ...] at the cursor
// out_cnt[r], which the caller zeroes first.
cudaError_t launch_topk_merge_grouped(int rows, int topk, int n_lists, int lists_per_group,
                                      const uint64_t* cand, int64_t row_stride,
                                      int64_t list_stride, const int* cand_cnt, int64_t cnt_row,
                                      int64_t cnt_list, int32_t* idx, float* score,
                                      uint64_t* out_keys, int* out_cnt, unsigned* err,
                                      cudaStream_t st, int append_cap = 0);

// Merge in two stages when rows are few and lists many (decode): groups of lists are merged
// by separate blocks into `stage` (topk_merge_stage_bytes), then each row's group results;
// the top k of a union is the top k of the union of its parts' top k, so the result equals
// the one-stage merge.  For rank-ordered output the groups (at most three, when each fits
// one block's staging) append to one list per row and the select-and-rank kernel finishes;
// otherwise about sqrt(n_lists) groups of about sqrt(n_lists) lists, then one merge block
// per row.  Falls back to one stage when grouping does not pay or stage is null.
int topk_merge_group_size(int rows, int n_lists);
size_t topk_merge_stage_bytes(int rows, int topk, int n_lists);
cudaError_t launch_topk_merge_two_stage(int rows, int topk, int n_lists, const uint64_t* cand,
                                        int64_t row_stride, int64_t list_stride,
                                        const int* cand_cnt, int64_t cnt_row, int64_t cnt_list,
                                        void* stage, int32_t* idx, float* score,
                                        uint64_t* out_keys, int* out_cnt, unsigned* err,
                                        cudaStream_t st);

// Stored score rows of one chunk of query rows (the two-pass tensor-core indexer): row
// rr = b * rows + (t - t0) of `scores` (stride ld floats, a multiple of 4, 16-byte aligned
// base) holds I[b, t, s] for the call's keys s = 0 .. n_t - 1, n_t = min(S, p_t + 1 -
// key_offset) (p_t the row's position in the whole cache).  Each row's top-k (positions
// in the whole cache) goes rank-ordered to idx / score [(b * T + t) * topk ..] (score may
// be null), or, when idx is null, as unordered 64-bit rank keys to cand[(b * T + t) *
// topk ..] with its count at cand_cnt[b * T + t].
struct ScoreRows {
    const float* scores;
    int64_t ld;
    int B, T, S, S_total, topk;
    int t0, rows;
    int64_t key_offset;
    const int32_t* kv_len;
    int32_t* idx;
    float* score;
    uint64_t* cand;
    int* cand_cnt;
    unsigned* err;
};
size_t topk_rows_smem_bytes();
cudaError_t launch_topk_rows(const ScoreRows& r, cudaStream_t st);

// One unordered list of distinct keys per row ([rows][stride] keys + counts [rows], at most
// stride keys a list) into each row's min(count, topk) best as rank-ordered idx / score
// rows.  topk <= stride <= topk_rank_max_stride().
int topk_rank_max_stride();
cudaError_t launch_topk_rank(int rows, int topk, int stride, const uint64_t* cand,
                             const int* cand_cnt, int32_t* idx, float* score, unsigned* err,
                             cudaStream_t st);

}  // namespace tsi
