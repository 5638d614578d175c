/*
 * tsi.h -- C ABI of the GB300 (sm_103a) DSA lightning-indexer + top-k + IndexShare
 * sparse-attention library (libtsi.so).
 *
 * The library computes, on the GPU:
 *   1. the lightning-indexer score I[t,s] = sum_j w[t,j] * ReLU(qI[t,j] . kI[s]) for
 *      every causal pair s <= p_t ("GLM-5.2 技术报告速览", §IndexShare, the score
 *      equation; one index key per position shared by all H_I heads);
 *   2. the top-k keys of every query row, ties going to the lower key index
 *      (same section: k = 2048 << L; "GLM-5: from Vibe Coding to Agentic Engineering"
 *      (Chinese translation) §3.2 "DSA RL 要点" asks for a deterministic top-k);
 *   3. sparse attention over those keys for every layer of an IndexShare group: the
 *      Full layer's index rows are reused by the Shared layers, each layer with its
 *      own Q/K/V ("GLM-5.2 技术报告速览" §IndexShare; "GLM 5.2: Built for Long Horizon
 *      Tasks" §5.2 and discussion §3).
 *
 * Conventions shared by every entry point
 *   - All tensor arguments are DEVICE pointers to dense row-major arrays owned by the
 *     caller; the library never allocates, frees or retains them.  Arrays of pointers
 *     (the per-layer q/k/v/out lists) are HOST arrays of device pointers.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  Every call only
 *     enqueues work on `stream` and returns; results are ready when the stream is.
 *   - Arguments are checked on the host before anything is launched.  A non-OK status
 *     means nothing was launched (except TSI_ERR_CUDA, which reports a failed launch);
 *     tsi_last_error() then describes the problem.
 *   - Query row t of sequence b sits at position p = kv_len[b] - T + t (kv_len NULL:
 *     kv_len[b] = S).  Prefill (T == S) gives p = t; decode (T == 1) gives
 *     p = kv_len[b] - 1.  Device-side kv_len values are clamped to [0, S].
 *   - Device-side waits are bounded; a wait that runs out, or a failed device check,
 *     sets a device error word instead of trapping.  tsi_device_status() reads it.
 */
#ifndef TSI_H
#define TSI_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    TSI_OK = 0,
    TSI_ERR_INVALID_ARG = 1,   /* bad shape, NULL pointer, misaligned pointer */
    TSI_ERR_UNSUPPORTED = 2,   /* valid request this build does not implement */
    TSI_ERR_WORKSPACE = 3,     /* workspace NULL or smaller than the query says */
    TSI_ERR_CUDA = 4,          /* a CUDA runtime call or kernel launch failed */
    TSI_ERR_TIMEOUT = 5,       /* a bounded device-side wait ran out */
    TSI_ERR_DEVICE_ASSERT = 6  /* a device-side consistency check failed */
} tsi_status;

/* Element types.  E4M3 is the FP8 "fn" format (bias 7, no infinities); stored bytes
 * are the values (no scale factors). */
typedef enum { TSI_F32 = 0, TSI_BF16 = 1, TSI_E4M3 = 2 } tsi_dtype;

#define TSI_MAX_TOPK 2048

/*
 * Workspace bytes needed by tsi_indexer_topk for these sizes (0 when none is needed).
 *   - Tensor-core path: candidate lists of 8-byte keys plus a count per list.  With
 *     several query rows per sequence and one key range per row: one list per row of the
 *     row selector's capacity (4352 keys for e4m3, 5888 for bf16: the keys at or above the
 *     row's threshold, which the ranking kernel selects from), the per-row admission
 *     thresholds, a list of unit indices (4 B per 4 rows of e4m3, per 2 rows of bf16) and
 *     every 32nd key row of the cache (B x ceil(S / 32) rows); at B = 1, T = S = 131072:
 *     ~4.6 GB.  Otherwise topk keys per row and key split.
 *   - Decode-sized requests (few rows, long caches) on either path: the per-split lists and
 *     merge staging space.
 */
size_t tsi_indexer_topk_workspace(int B, int T, int S, int H_I, int d_I, int topk,
                                  int qk_dtype);

/*
 * Lightning-indexer score + causal top-k ("GLM-5.2 技术报告速览", §IndexShare).
 * On the tensor-core path no score leaves the scoring kernel: each row's top k is
 * selected in the kernel's epilogue (the pages' Ascend operator likewise fuses score,
 * ReLU and top-k: "GLM-5: from Vibe Coding to Agentic Engineering" (Chinese translation),
 * §5).  With several query rows per sequence the kernel first scores every 32nd key to
 * set each row's admission threshold, then scores all keys admitting only those at or
 * above it; rows the sample misjudged are redone from no threshold, so the result is exact
 * for any input.
 *
 *   qI     [B, T, H_I, d_I]  qk_dtype (F32, BF16 or E4M3)   index queries
 *   kI     [B, S, d_I]       qk_dtype                        index-key cache
 *   w      [B, T, H_I]       w_dtype (F32 or BF16)            per-head gate weights
 *   kv_len [B] int32 or NULL                                  cached length per sequence
 *   idx    [B, T, topk] int32 (out)  key positions in rank order: higher score first,
 *          equal scores by lower position; rows with fewer than topk causal keys are
 *          padded with -1 after their p+1 keys.
 *   score  [B, T, topk] float (out, may be NULL)  the fp32 score of each idx entry,
 *          -inf for padding.
 *
 * Scores are accumulated in fp32 (tensor cores for BF16/E4M3 with H_I = 64, d_I = 128,
 * except BF16 with one query per sequence, T = 1; CUDA cores otherwise).
 * 1 <= topk <= TSI_MAX_TOPK, d_I <= 256, H_I <= 128.  Pointers must be 16-byte aligned.
 * Requires workspace_bytes >= tsi_indexer_topk_workspace(...).
 */
tsi_status tsi_indexer_topk(const void* qI, const void* kI, const void* w, int qk_dtype,
                            int w_dtype, int B, int T, int S, int H_I, int d_I, int topk,
                            const int32_t* kv_len, int32_t* idx, float* score, void* workspace,
                            size_t workspace_bytes, void* stream);

/*
 * tsi_indexer_topk under the name that states its property: every score stays on chip
 * (same source, same passages as tsi_indexer_topk).  Arguments, layouts, rules and the
 * workspace query are those of tsi_indexer_topk.
 */
size_t tsi_indexer_topk_onchip_workspace(int B, int T, int S, int H_I, int d_I, int topk,
                                         int qk_dtype);
tsi_status tsi_indexer_topk_onchip(const void* qI, const void* kI, const void* w, int qk_dtype,
                                   int w_dtype, int B, int T, int S, int H_I, int d_I, int topk,
                                   const int32_t* kv_len, int32_t* idx, float* score,
                                   void* workspace, size_t workspace_bytes, void* stream);

/*
 * The same results as tsi_indexer_topk (same source: "GLM-5.2 技术报告速览", §IndexShare)
 * from two passes on the tensor-core path with several query rows per sequence: the fp32
 * scores of a chunk of query rows are written to the workspace (rows of S, rounded up to
 * 4, floats for every sequence; the chunk as many rows as fit in about 8 GiB, all T rows
 * when they fit), then one block per row selects and ranks its top k from them.  It costs
 * 4 B of HBM writes and reads per causal pair.  Shapes the tensor-core path does not take,
 * and one query row per sequence, run exactly as in tsi_indexer_topk.  Arguments, layouts
 * and rules as tsi_indexer_topk, with workspace_bytes >=
 * tsi_indexer_topk_two_pass_workspace(...).
 */
size_t tsi_indexer_topk_two_pass_workspace(int B, int T, int S, int H_I, int d_I, int topk,
                                           int qk_dtype);
tsi_status tsi_indexer_topk_two_pass(const void* qI, const void* kI, const void* w,
                                     int qk_dtype, int w_dtype, int B, int T, int S, int H_I,
                                     int d_I, int topk, const int32_t* kv_len, int32_t* idx,
                                     float* score, void* workspace, size_t workspace_bytes,
                                     void* stream);

/*
 * tsi_indexer_topk without a workspace argument and without allocating anything.
 * The paper has no counterpart: this is a convenience of this library.
 *
 * Meant for callers that cannot allocate device memory while they run, such as a
 * serving loop whose device memory is fixed at start-up, or code called from inside a
 * custom device allocator, where a nested cudaMalloc would recurse into the allocator
 * or synchronize the device.  The scratch that tsi_indexer_topk takes from the caller's
 * workspace (per-split candidate lists when few rows scan long caches, as in decode)
 * lives here in one fixed array compiled into the library: 8 MiB of device memory,
 * held by every GPU that loads the library until the process exits
 * (tsi_indexer_topk_noalloc_limit() returns the size).
 *
 * Arguments, layouts and results are those of tsi_indexer_topk; the scores always come
 * from the CUDA-core path (identical indices on integer-valued inputs, the same
 * near-tie behaviour otherwise).  A request whose scratch would exceed the array
 * (tsi_indexer_topk_workspace for the same sizes, with CUDA-core shapes) returns
 * TSI_ERR_UNSUPPORTED and launches nothing.  The call performs no cudaMalloc, cudaFree
 * or other allocating call.
 *
 * The first call on each device looks up the array's device address
 * (cudaGetSymbolAddress) while that device is current; make that first call before any
 * stream capture.  All calls on a device share the one array, which keeps whatever the
 * last call left in it (each call writes every scratch slot before reading it, so
 * nothing needs clearing).  Calls whose kernels overlap on the GPU -- different streams,
 * or different host threads -- race on the array and give undefined results: serialize
 * them on one stream.
 */
tsi_status tsi_indexer_topk_noalloc(const void* qI, const void* kI, const void* w, int qk_dtype,
                                    int w_dtype, int B, int T, int S, int H_I, int d_I,
                                    int topk, const int32_t* kv_len, int32_t* idx, float* score,
                                    void* stream);

/* Bytes of the built-in scratch array used by tsi_indexer_topk_noalloc. */
size_t tsi_indexer_topk_noalloc_limit(void);

/* Workspace bytes needed by tsi_sparse_attn_group for these sizes (0 when none). */
size_t tsi_sparse_attn_workspace(int B, int T, int S, int H, int Hkv, int Dqk, int Dv,
                                 int topk);

/*
 * Sparse attention for the n_layers layers of one IndexShare group over ONE shared
 * index buffer ("GLM-5.2 技术报告速览" §IndexShare; "GLM 5.2: Built for Long Horizon
 * Tasks" §5.2): for every layer l, query row (b,t) and head h,
 *
 *   O_l[b,t,h,:] = sum_{s in S} softmax_s(scale * Q_l[b,t,h,:] . K_l[b,s,g,:]) V_l[b,s,g,:]
 *
 * with g = h / (H / Hkv) and S the entries of idx[b,t,:] inside [0, kv_len[b]) (the -1
 * padding is not a key).  A row with no key gets O = 0.
 *
 *   q[l]   [B, T, H, Dqk]   bf16
 *   k[l]   [B, S, Hkv, Dqk] bf16
 *   v[l]   [B, S, Hkv, Dv]  bf16, or v == NULL / v[l] == NULL: the value is the first
 *          Dv dims of the key row (MLA latent: 576 = 512 + 64, value = first 512)
 *   idx    [B, T, topk] int32, shared by all layers (the Full layer's selection)
 *   out[l] [B, T, H, Dv]    bf16 (out)
 *
 * Softmax and accumulation run in fp32.  H % Hkv == 0, Dqk <= 576, Dv <= 512,
 * 1 <= topk <= TSI_MAX_TOPK.  Pointers must be 16-byte aligned.  Layers run one after
 * another on `stream`.
 */
tsi_status tsi_sparse_attn_group(int n_layers, const void* const* q, const void* const* k,
                                 const void* const* v, int B, int T, int S, int H, int Hkv,
                                 int Dqk, int Dv, float scale, const int32_t* idx, int topk,
                                 const int32_t* kv_len, void* const* out, void* workspace,
                                 size_t workspace_bytes, void* stream);

/*
 * tsi_sparse_attn_group that also returns each layer's per-head log-partition
 *
 *   lse[l]  [B, T, H] fp32 (out) or lse == NULL: ln sum_{s in S} exp(scale * Q_l[b,t,h,:] .
 *           K_l[b,s,g,:]) over the same keys S as the output; -inf for a row with no key.
 *
 * The sum is the one that normalises the output (the tensor-core path sums the bf16
 * probabilities that multiply V).  It is what tsi_index_kl needs to turn recomputed logits
 * back into the layer's attention probabilities.  Other arguments and rules as
 * tsi_sparse_attn_group; lse[l] must be 16-byte aligned.
 */
tsi_status tsi_sparse_attn_group_lse(int n_layers, const void* const* q, const void* const* k,
                                     const void* const* v, int B, int T, int S, int H, int Hkv,
                                     int Dqk, int Dv, float scale, const int32_t* idx, int topk,
                                     const int32_t* kv_len, void* const* out, float* const* lse,
                                     void* workspace, size_t workspace_bytes, void* stream);

/*
 * Group-centroid KL target of the Full layer's indexer ("GLM-5.2 技术报告速览"
 * §IndexShare, "少数层挑，其余层复用": the indexer that serves a group of m + 1 layers is
 * fitted, by KL, to pbar_t = 1/(m+1) sum_j p^(l+j)_t, the mean of the group's
 * head-averaged attention distributions).  For every query row t of the group (one Full
 * layer then its Shared layers, n_layers = m + 1) and its selected keys S_t (the entries
 * of idx[b,t,:] inside [0, kv_len[b])):
 *
 *   p_l[t,s]  = 1/H sum_h exp(scale * Q_l[b,t,h,:] . K_l[b,s,:] - lse_l[b,t,h])
 *   pbar[t,s] = 1/n_layers sum_l p_l[t,s]
 *   q[t,s]    = exp(I[t,s]) / sum_{s' in S_t} exp(I[t,s'])      (I = score)
 *   loss[t]   = sum_{s in S_t, pbar > 0} pbar[t,s] (ln pbar[t,s] - ln q[t,s])
 *   grad[t,s] = q[t,s] - pbar[t,s]          (d loss[t] / d I[t,s]; pbar sums to one)
 *
 *   q[l]      [B, T, 64, 576] bf16: layer l's attention queries (H = 64)
 *   k[l]      [B, S, 576] bf16: layer l's latent key cache (one KV head)
 *   lse[l]    [B, T, 64] fp32: layer l's log-partition, from tsi_sparse_attn_group_lse with
 *             the same idx, kv_len and scale
 *   idx       [B, T, topk] int32: the group's shared index rows
 *   score     [B, T, topk] fp32: the indexer scores of those entries, I[t, idx[t,i]] (the
 *             score output of tsi_indexer_topk); read only where the entry is a key
 *   loss      [B, T] fp32 (out): 0 for a row with no key
 *   grad      [B, T, topk] fp32 (out) or NULL: in idx order, 0 where the entry is no key
 *   pbar      [B, T, topk] fp32 (out) or NULL: the centroid in idx order, 0 where no key
 *
 * Logits come from bf16 products summed in fp32 on the tensor core, probabilities in fp32;
 * the loss uses fp32 exp / log.  1 <= n_layers <= 8, 1 <= topk <= TSI_MAX_TOPK; H = 64 and
 * Dqk = 576 only (TSI_ERR_UNSUPPORTED otherwise).  Pointers must be 16-byte aligned.
 */
tsi_status tsi_index_kl(int n_layers, const void* const* q, const void* const* k,
                        const float* const* lse, int B, int T, int S, int H, int Dqk, float scale,
                        const int32_t* idx, const float* score, int topk, const int32_t* kv_len,
                        float* loss, float* grad, float* pbar, void* stream);

/*
 * One key shard of a context-parallel indexer ("GLM 5.2: Built for Long Horizon Tasks",
 * discussion §4: context parallelism (CP / DCP) for single very long requests, the context
 * split over ranks; the score and top-k are those of tsi_indexer_topk).  A rank holding keys key_offset ..
 * key_offset + S_shard - 1 of a cache of S_total keys finds, for every query row, the top k
 * of its shard; merging the shards' lists (tsi_topk_merge) gives exactly the rows that
 * tsi_indexer_topk computes over the whole cache.
 *
 *   qI, w     as tsi_indexer_topk (all B x T query rows)
 *   kI        [B, S_shard, d_I] qk_dtype: the shard's keys
 *   kv_len    [B] int32 or NULL: cached length per sequence in the WHOLE cache (NULL:
 *             S_total); query row t sits at position kv_len[b] - T + t, as always
 *   cand      [B*T, topk] uint64 (out): per row the shard's best keys as rank keys
 *             (order(score) << 32 | (0xFFFFFFFF - position), positions of the whole cache),
 *             unordered; entries past the count are left as they were
 *   cand_cnt  [B*T] int32 (out): how many keys of the row the shard holds, at most topk
 *
 * Requires 0 <= key_offset, key_offset + S_shard <= S_total, and
 * workspace_bytes >= tsi_indexer_topk_shard_workspace(...): what tsi_indexer_topk_workspace
 * describes for S_shard keys except the candidate lists, which are the caller's cand
 * (0 when nothing else is needed).  Other rules as tsi_indexer_topk.
 */
size_t tsi_indexer_topk_shard_workspace(int B, int T, int S_shard, int H_I, int d_I, int topk,
                                        int qk_dtype);
tsi_status tsi_indexer_topk_shard(const void* qI, const void* kI, const void* w, int qk_dtype,
                                  int w_dtype, int B, int T, int S_total, int64_t key_offset,
                                  int S_shard, int H_I, int d_I, int topk, const int32_t* kv_len,
                                  uint64_t* cand, int32_t* cand_cnt, void* workspace,
                                  size_t workspace_bytes, void* stream);

/*
 * Merge of candidate lists (the exchange step of the context-parallel indexer: every
 * rank's tsi_indexer_topk_shard output, gathered): for each row, the top k of the union
 * of its n_lists lists, written as tsi_indexer_topk writes them (rank order, -1 / -inf
 * padding).  Rank keys are distinct within a row, so the result does not depend on the
 * order of the lists.
 *
 *   cand      [n_lists, rows, topk] uint64 device, list-major (the layout of an
 *             all-gather of the ranks' cand buffers)
 *   cand_cnt  [n_lists, rows] int32 device: valid entries of each list, each <= topk
 *   idx       [rows, topk] int32 device (out); score [rows, topk] float (out, may be NULL)
 *
 * 1 <= n_lists <= 1024, 1 <= topk <= TSI_MAX_TOPK; pointers 16-byte aligned.
 */
tsi_status tsi_topk_merge(const uint64_t* cand, const int32_t* cand_cnt, int n_lists, int rows,
                          int topk, int32_t* idx, float* score, void* stream);

/*
 * Layer schedule of an IndexShare stack ("GLM 5.2: Built for Long Horizon Tasks" §5.2:
 * the model config's index_topk_freq, index_skip_topk_offset and index_topk_pattern, with
 * periodic full, shared, shared, shared layer types after the offset; "GLM-5.2
 * 技术报告速览" §IndexShare: a Full layer runs its indexer, a Shared layer reuses the index
 * rows of the nearest Full layer before it).
 *
 *   pattern  NULL, or a string of exactly n_layers characters 'F' (Full) / 'S' (Shared)
 *            that overrides freq and skip_offset.  When NULL, layers l < skip_offset are
 *            Full, and from skip_offset on the types repeat with period freq, the first of
 *            each period Full (freq = 4, skip_offset = 3: F F F F S S S F S S S ...).
 *   anchor   [n_layers] int32, HOST (out): the layer whose indexer gives layer l its index
 *            rows; anchor[l] == l exactly for the Full layers.
 *
 * Layer 0 must be Full.  TSI_ERR_INVALID_ARG for n_layers < 0, freq < 1, skip_offset < 0,
 * a pattern of the wrong length or with other characters, a Shared layer 0, or a NULL
 * anchor with n_layers > 0.  Host only: launches nothing.
 */
tsi_status tsi_index_share_layers(int n_layers, int freq, int skip_offset, const char* pattern,
                                  int32_t* anchor);

/*
 * Cross-layer top-k overlap ("GLM-5.2 技术报告速览" §IndexShare: the pairwise overlap of
 * the per-layer top-k index sets that makes reuse across layers possible, 0.7-1.0 between
 * adjacent layers).  For every row r of two index buffers:
 *
 *   idx_a, idx_b  [rows, topk] int32 device: index rows (entries < 0 are padding, the rest
 *                 distinct positions within a row, as tsi_indexer_topk writes them)
 *   inter         [rows] int32 device (out): |S_a(r) ∩ S_b(r)|
 *   card_a        [rows] int32 device (out): |S_a(r)|, the entries >= 0 of row r of idx_a
 *
 * The overlap rate of a row is inter / card_a (rows with card_a = 0 have none).  A repeated
 * position within a row of idx_a sets the device error word (tsi_device_status then returns
 * TSI_ERR_DEVICE_ASSERT).  1 <= topk <= TSI_MAX_TOPK; pointers 16-byte aligned.
 */
tsi_status tsi_topk_overlap(const int32_t* idx_a, const int32_t* idx_b, int rows, int topk,
                            int32_t* inter, int32_t* card_a, void* stream);

/*
 * Self-test of the failure path, for tests of error handling without a GPU fault.  Launches
 * one block in which a single thread waits, through the same bounded-wait helper the
 * tensor-core kernels use, on an mbarrier that nothing completes.  After the wait's clock
 * budget (about a second) the helper sets the device error word and the kernel returns:
 * nothing faults, traps or spins without bound.  tsi_device_status(stream) then returns
 * TSI_ERR_TIMEOUT (and clears the word), and the context stays usable.  Returns TSI_OK once
 * launched.
 */
tsi_status tsi_selftest_wait_timeout(void* stream);

/*
 * Waits for `stream`, then reads and clears the device error word of the current
 * device.  Returns TSI_OK, TSI_ERR_TIMEOUT (a bounded wait ran out),
 * TSI_ERR_DEVICE_ASSERT (a device check failed) or TSI_ERR_CUDA.
 */
tsi_status tsi_device_status(void* stream);

/* Message for the last non-OK status returned on this host thread ("" if none). */
const char* tsi_last_error(void);

/* Which kernels serve a shape: 1 = tensor-core (tcgen05) path, 0 = CUDA-core path,
 * -1 = unsupported.  For the indexer this is the path of requests with several queries
 * per sequence (T > 1); BF16 requests with T = 1 take the CUDA-core path.  v_from_k != 0
 * means the value is the first Dv dims of the key. */
int tsi_indexer_topk_path(int qk_dtype, int H_I, int d_I);
int tsi_sparse_attn_path(int H, int Hkv, int Dqk, int Dv, int v_from_k);

/* Number of kernels this library has launched in this process (all threads). */
uint64_t tsi_launch_count(void);

/* Library version, major*10000 + minor*100 + patch. */
int tsi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* TSI_H */
