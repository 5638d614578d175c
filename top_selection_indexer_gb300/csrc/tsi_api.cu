// C ABI of libtsi.so: argument checks, path selection, error reporting.
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <mutex>

#include "attn_generic.cuh"
#include "indexer_generic.cuh"
#include "kernels_tc.cuh"
#include "overlap.cuh"
#include "tsi_common.cuh"

namespace tsi {
static std::atomic<uint64_t> g_launches{0};
void note_launches(int n) { g_launches.fetch_add(static_cast<uint64_t>(n)); }
}  // namespace tsi

namespace {

thread_local char g_msg[512] = "";

tsi_status fail(tsi_status st, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_msg, sizeof g_msg, fmt, ap);
    va_end(ap);
    return st;
}

tsi_status ok() {
    g_msg[0] = '\0';
    return TSI_OK;
}

// Device error word, one per device (context); kernels atomicOr flags into it.
__device__ unsigned g_dev_err;

constexpr int kMaxDevices = 64;
unsigned* g_err_ptr[kMaxDevices] = {};
std::mutex g_err_mu;

tsi_status device_error_word(unsigned** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(TSI_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    if (dev < 0 || dev >= kMaxDevices) return fail(TSI_ERR_CUDA, "device id %d out of range", dev);
    std::lock_guard<std::mutex> lk(g_err_mu);
    if (!g_err_ptr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_dev_err);
        if (e != cudaSuccess)
            return fail(TSI_ERR_CUDA, "cudaGetSymbolAddress: %s", cudaGetErrorString(e));
        g_err_ptr[dev] = static_cast<unsigned*>(p);
    }
    *out = g_err_ptr[dev];
    return TSI_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool qk_dtype_ok(int dt) { return dt == TSI_F32 || dt == TSI_BF16 || dt == TSI_E4M3; }
bool w_dtype_ok(int dt) { return dt == TSI_F32 || dt == TSI_BF16; }

bool use_tc_indexer(int qk_dtype, int H_I, int d_I) {
    return tsi::tc_indexer_supported(qk_dtype, H_I, d_I);
}

// The tensor-core path for a request.  bf16 requests of one query per sequence go to the
// CUDA-core path: the tensor-core pass with one bf16 query row per unit faulted on key
// caches of repeated rows, cause not found, so it does not run.
bool use_tc_indexer(int qk_dtype, int H_I, int d_I, int T) {
    return use_tc_indexer(qk_dtype, H_I, d_I) && !(qk_dtype == TSI_BF16 && T == 1);
}

bool use_tc_attn(int H, int Hkv, int Dqk, int Dv, bool v_from_k) {
    return tsi::tc_attn_supported(H, Hkv, Dqk, Dv, v_from_k);
}

}  // namespace

namespace {

size_t indexer_workspace(int B, int T, int S, int H_I, int d_I, int topk, int qk_dtype,
                         bool two_pass) {
    if (B <= 0 || T <= 0 || S < 0 || topk < 1) return 0;
    if (use_tc_indexer(qk_dtype, H_I, d_I, T))
        return tsi::tc_indexer_workspace_bytes(qk_dtype, B, T, S, topk, two_pass);
    return tsi::generic_workspace_bytes(B, T, S, topk);
}

// tsi_indexer_topk and its two-pass form: two_pass stores the tensor-core path's scores for
// a second, selecting kernel instead of selecting in the scoring kernel's epilogue.
tsi_status indexer_topk(const void* qI, const void* kI, const void* w, int qk_dtype, int w_dtype,
                        int B, int T, int S, int H_I, int d_I, int topk, const int32_t* kv_len,
                        int32_t* idx, float* score, void* workspace, size_t workspace_bytes,
                        void* stream, bool two_pass) {
    if (!qk_dtype_ok(qk_dtype)) return fail(TSI_ERR_INVALID_ARG, "qk_dtype %d unknown", qk_dtype);
    if (!w_dtype_ok(w_dtype)) return fail(TSI_ERR_INVALID_ARG, "w_dtype %d unknown", w_dtype);
    if (B < 0 || T < 0 || S < 0)
        return fail(TSI_ERR_INVALID_ARG, "negative size (B=%d T=%d S=%d)", B, T, S);
    if (topk < 1 || topk > TSI_MAX_TOPK)
        return fail(TSI_ERR_UNSUPPORTED, "topk=%d outside [1, %d]", topk, TSI_MAX_TOPK);
    if (H_I < 1 || d_I < 1) return fail(TSI_ERR_INVALID_ARG, "H_I=%d d_I=%d", H_I, d_I);
    const bool tc = use_tc_indexer(qk_dtype, H_I, d_I, T);
    if (!tc && !tsi::generic_supported(H_I, d_I))
        return fail(TSI_ERR_UNSUPPORTED, "H_I=%d d_I=%d unsupported (d_I<=256, H_I<=128, "
                    "H_I*d_I<=8192)", H_I, d_I);
    if (static_cast<int64_t>(B) * T > (1ll << 31) - 1 || static_cast<int64_t>(B) * S > (1ll << 31) - 1)
        return fail(TSI_ERR_UNSUPPORTED, "B*T or B*S exceeds 2^31-1");
    if (B == 0 || T == 0) return ok();
    if (!qI || !w || !idx || (S > 0 && !kI))
        return fail(TSI_ERR_INVALID_ARG, "NULL tensor pointer");
    if (!aligned16(qI) || !aligned16(kI) || !aligned16(w) || !aligned16(idx) ||
        !aligned16(score) || !aligned16(kv_len))
        return fail(TSI_ERR_INVALID_ARG, "tensor pointers must be 16-byte aligned");
    const size_t need = indexer_workspace(B, T, S, H_I, d_I, topk, qk_dtype, two_pass);
    if (workspace_bytes < need || (need > 0 && !workspace))
        return fail(TSI_ERR_WORKSPACE, "workspace %zu bytes, need %zu", workspace_bytes, need);
    if (need > 0 && !aligned16(workspace))
        return fail(TSI_ERR_INVALID_ARG, "workspace must be 16-byte aligned");
    unsigned* err = nullptr;
    tsi_status st = device_error_word(&err);
    if (st != TSI_OK) return st;
    tsi::IndexerArgs a{qI, kI, w, qk_dtype, w_dtype, B, T, S, H_I, d_I, topk, kv_len,
                       idx, score, err};
    a.two_pass = two_pass;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = tc ? tsi::launch_indexer_tc(a, workspace, s)
                       : tsi::launch_indexer_generic(a, workspace, s);
    if (e != cudaSuccess) return fail(TSI_ERR_CUDA, "indexer launch: %s", cudaGetErrorString(e));
    return ok();
}

}  // namespace

extern "C" {

int tsi_version(void) { return 100; }

uint64_t tsi_launch_count(void) { return tsi::g_launches.load(); }

int tsi_indexer_topk_path(int qk_dtype, int H_I, int d_I) {
    if (!qk_dtype_ok(qk_dtype)) return -1;
    if (use_tc_indexer(qk_dtype, H_I, d_I)) return 1;
    return tsi::generic_supported(H_I, d_I) ? 0 : -1;
}

int tsi_sparse_attn_path(int H, int Hkv, int Dqk, int Dv, int v_from_k) {
    if (use_tc_attn(H, Hkv, Dqk, Dv, v_from_k != 0)) return 1;
    return tsi::attn_generic_supported(H, Hkv, Dqk, Dv, v_from_k != 0) ? 0 : -1;
}

const char* tsi_last_error(void) { return g_msg; }

size_t tsi_indexer_topk_workspace(int B, int T, int S, int H_I, int d_I, int topk,
                                  int qk_dtype) {
    return indexer_workspace(B, T, S, H_I, d_I, topk, qk_dtype, false);
}

size_t tsi_indexer_topk_onchip_workspace(int B, int T, int S, int H_I, int d_I, int topk,
                                         int qk_dtype) {
    return indexer_workspace(B, T, S, H_I, d_I, topk, qk_dtype, false);
}

size_t tsi_indexer_topk_two_pass_workspace(int B, int T, int S, int H_I, int d_I, int topk,
                                           int qk_dtype) {
    return indexer_workspace(B, T, S, H_I, d_I, topk, qk_dtype, true);
}

tsi_status tsi_indexer_topk(const void* qI, const void* kI, const void* w, int qk_dtype,
                            int w_dtype, int B, int T, int S, int H_I, int d_I, int topk,
                            const int32_t* kv_len, int32_t* idx, float* score, void* workspace,
                            size_t workspace_bytes, void* stream) {
    return indexer_topk(qI, kI, w, qk_dtype, w_dtype, B, T, S, H_I, d_I, topk, kv_len, idx, score,
                        workspace, workspace_bytes, stream, false);
}

tsi_status tsi_indexer_topk_onchip(const void* qI, const void* kI, const void* w, int qk_dtype,
                                   int w_dtype, int B, int T, int S, int H_I, int d_I, int topk,
                                   const int32_t* kv_len, int32_t* idx, float* score,
                                   void* workspace, size_t workspace_bytes, void* stream) {
    return indexer_topk(qI, kI, w, qk_dtype, w_dtype, B, T, S, H_I, d_I, topk, kv_len, idx, score,
                        workspace, workspace_bytes, stream, false);
}

tsi_status tsi_indexer_topk_two_pass(const void* qI, const void* kI, const void* w, int qk_dtype,
                                     int w_dtype, int B, int T, int S, int H_I, int d_I, int topk,
                                     const int32_t* kv_len, int32_t* idx, float* score,
                                     void* workspace, size_t workspace_bytes, void* stream) {
    return indexer_topk(qI, kI, w, qk_dtype, w_dtype, B, T, S, H_I, d_I, topk, kv_len, idx, score,
                        workspace, workspace_bytes, stream, true);
}

size_t tsi_indexer_topk_shard_workspace(int B, int T, int S_shard, int H_I, int d_I, int topk,
                                        int qk_dtype) {
    if (B <= 0 || T <= 0 || S_shard < 0 || topk < 1) return 0;
    if (use_tc_indexer(qk_dtype, H_I, d_I, T))
        return tsi::tc_indexer_split_workspace_bytes(qk_dtype, B, T, S_shard, topk);
    return tsi::generic_workspace_bytes(B, T, S_shard, topk);
}

tsi_status tsi_indexer_topk_shard(const void* qI, const void* kI, const void* w, int qk_dtype,
                                  int w_dtype, int B, int T, int S_total, int64_t key_offset,
                                  int S_shard, int H_I, int d_I, int topk, const int32_t* kv_len,
                                  uint64_t* cand, int32_t* cand_cnt, void* workspace,
                                  size_t workspace_bytes, void* stream) {
    if (!qk_dtype_ok(qk_dtype)) return fail(TSI_ERR_INVALID_ARG, "qk_dtype %d unknown", qk_dtype);
    if (!w_dtype_ok(w_dtype)) return fail(TSI_ERR_INVALID_ARG, "w_dtype %d unknown", w_dtype);
    if (B < 0 || T < 0 || S_shard < 0 || S_total < 0)
        return fail(TSI_ERR_INVALID_ARG, "negative size (B=%d T=%d S_total=%d S_shard=%d)", B, T,
                    S_total, S_shard);
    if (key_offset < 0 || key_offset + S_shard > S_total)
        return fail(TSI_ERR_INVALID_ARG, "shard [%lld, %lld) outside the cache of %d keys",
                    static_cast<long long>(key_offset),
                    static_cast<long long>(key_offset + S_shard), S_total);
    if (topk < 1 || topk > TSI_MAX_TOPK)
        return fail(TSI_ERR_UNSUPPORTED, "topk=%d outside [1, %d]", topk, TSI_MAX_TOPK);
    if (H_I < 1 || d_I < 1) return fail(TSI_ERR_INVALID_ARG, "H_I=%d d_I=%d", H_I, d_I);
    const bool tc = use_tc_indexer(qk_dtype, H_I, d_I, T);
    if (!tc && !tsi::generic_supported(H_I, d_I))
        return fail(TSI_ERR_UNSUPPORTED, "H_I=%d d_I=%d unsupported (d_I<=256, H_I<=128, "
                    "H_I*d_I<=8192)", H_I, d_I);
    if (static_cast<int64_t>(B) * T > (1ll << 31) - 1 ||
        static_cast<int64_t>(B) * S_total > (1ll << 31) - 1)
        return fail(TSI_ERR_UNSUPPORTED, "B*T or B*S_total exceeds 2^31-1");
    if (B == 0 || T == 0) return ok();
    if (!qI || !w || !cand || !cand_cnt || (S_shard > 0 && !kI))
        return fail(TSI_ERR_INVALID_ARG, "NULL tensor pointer");
    if (!aligned16(qI) || !aligned16(kI) || !aligned16(w) || !aligned16(cand) ||
        !aligned16(cand_cnt) || !aligned16(kv_len))
        return fail(TSI_ERR_INVALID_ARG, "tensor pointers must be 16-byte aligned");
    const size_t need = tsi_indexer_topk_shard_workspace(B, T, S_shard, H_I, d_I, topk, qk_dtype);
    if (workspace_bytes < need || (need > 0 && !workspace))
        return fail(TSI_ERR_WORKSPACE, "workspace %zu bytes, need %zu", workspace_bytes, need);
    if (need > 0 && !aligned16(workspace))
        return fail(TSI_ERR_INVALID_ARG, "workspace must be 16-byte aligned");
    unsigned* err = nullptr;
    tsi_status st = device_error_word(&err);
    if (st != TSI_OK) return st;
    tsi::IndexerArgs a{qI, kI, w, qk_dtype, w_dtype, B, T, S_shard, H_I, d_I, topk, kv_len,
                       nullptr, nullptr, err};
    a.key_offset = key_offset;
    a.S_total = S_total;
    a.out_cand = cand;
    a.out_cnt = cand_cnt;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = tc ? tsi::launch_indexer_tc(a, workspace, s)
                       : tsi::launch_indexer_generic(a, workspace, s);
    if (e != cudaSuccess) return fail(TSI_ERR_CUDA, "indexer launch: %s", cudaGetErrorString(e));
    return ok();
}

tsi_status tsi_topk_merge(const uint64_t* cand, const int32_t* cand_cnt, int n_lists, int rows,
                          int topk, int32_t* idx, float* score, void* stream) {
    if (rows < 0 || n_lists < 0) return fail(TSI_ERR_INVALID_ARG, "rows=%d n_lists=%d", rows, n_lists);
    if (topk < 1 || topk > TSI_MAX_TOPK)
        return fail(TSI_ERR_UNSUPPORTED, "topk=%d outside [1, %d]", topk, TSI_MAX_TOPK);
    if (n_lists > 1024) return fail(TSI_ERR_UNSUPPORTED, "n_lists=%d above 1024", n_lists);
    if (rows == 0) return ok();
    if (n_lists == 0) return fail(TSI_ERR_INVALID_ARG, "no candidate lists");
    if (!cand || !cand_cnt || !idx) return fail(TSI_ERR_INVALID_ARG, "NULL pointer");
    if (!aligned16(cand) || !aligned16(cand_cnt) || !aligned16(idx) || !aligned16(score))
        return fail(TSI_ERR_INVALID_ARG, "pointers must be 16-byte aligned");
    unsigned* err = nullptr;
    tsi_status st = device_error_word(&err);
    if (st != TSI_OK) return st;
    cudaError_t e = tsi::launch_topk_merge_strided(
        rows, topk, n_lists, cand, topk, static_cast<int64_t>(rows) * topk, cand_cnt, 1, rows,
        idx, score, nullptr, nullptr, err, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return fail(TSI_ERR_CUDA, "merge launch: %s", cudaGetErrorString(e));
    return ok();
}

size_t tsi_sparse_attn_workspace(int B, int T, int S, int H, int Hkv, int Dqk, int Dv,
                                 int topk) {
    if (B <= 0 || T <= 0 || topk < 1 || H < 1) return 0;
    // the value layout does not change the workspace: ask for the larger of the two paths
    size_t a = tsi::attn_generic_workspace_bytes(B, T, H, Dv, topk);
    size_t b = use_tc_attn(H, Hkv, Dqk, Dv, true) ? tsi::tc_attn_workspace_bytes(B, T, H, Dv, topk)
                                                  : 0;
    return a > b ? a : b;
}

tsi_status tsi_sparse_attn_group(int n_layers, const void* const* q, const void* const* k,
                                 const void* const* v, int B, int T, int S, int H, int Hkv,
                                 int Dqk, int Dv, float scale, const int32_t* idx, int topk,
                                 const int32_t* kv_len, void* const* out, void* workspace,
                                 size_t workspace_bytes, void* stream) {
    return tsi_sparse_attn_group_lse(n_layers, q, k, v, B, T, S, H, Hkv, Dqk, Dv, scale, idx,
                                     topk, kv_len, out, nullptr, workspace, workspace_bytes,
                                     stream);
}

tsi_status tsi_sparse_attn_group_lse(int n_layers, const void* const* q, const void* const* k,
                                     const void* const* v, int B, int T, int S, int H, int Hkv,
                                     int Dqk, int Dv, float scale, const int32_t* idx, int topk,
                                     const int32_t* kv_len, void* const* out, float* const* lse,
                                     void* workspace, size_t workspace_bytes, void* stream) {
    if (n_layers < 0) return fail(TSI_ERR_INVALID_ARG, "n_layers=%d", n_layers);
    if (B < 0 || T < 0 || S < 0)
        return fail(TSI_ERR_INVALID_ARG, "negative size (B=%d T=%d S=%d)", B, T, S);
    if (topk < 1 || topk > TSI_MAX_TOPK)
        return fail(TSI_ERR_UNSUPPORTED, "topk=%d outside [1, %d]", topk, TSI_MAX_TOPK);
    if (H < 1 || Hkv < 1 || H % Hkv != 0)
        return fail(TSI_ERR_INVALID_ARG, "H=%d must be a positive multiple of Hkv=%d", H, Hkv);
    if (Dqk < 1 || Dv < 1) return fail(TSI_ERR_INVALID_ARG, "Dqk=%d Dv=%d", Dqk, Dv);
    if (!std::isfinite(scale)) return fail(TSI_ERR_INVALID_ARG, "scale is not finite");
    if (static_cast<int64_t>(B) * T > (1ll << 31) - 1 || static_cast<int64_t>(B) * S > (1ll << 31) - 1)
        return fail(TSI_ERR_UNSUPPORTED, "B*T or B*S exceeds 2^31-1");
    if (n_layers == 0 || B == 0 || T == 0) return ok();
    if (!q || !k || !out || !idx) return fail(TSI_ERR_INVALID_ARG, "NULL pointer list");
    if (!aligned16(idx) || !aligned16(kv_len))
        return fail(TSI_ERR_INVALID_ARG, "idx / kv_len must be 16-byte aligned");
    for (int l = 0; l < n_layers; ++l) {
        const void* vl = v ? v[l] : nullptr;
        const bool vk = vl == nullptr;
        if (!q[l] || !out[l] || (S > 0 && !k[l]))
            return fail(TSI_ERR_INVALID_ARG, "layer %d: NULL tensor pointer", l);
        if (!aligned16(q[l]) || !aligned16(k[l]) || !aligned16(vl) || !aligned16(out[l]))
            return fail(TSI_ERR_INVALID_ARG, "layer %d: pointers must be 16-byte aligned", l);
        if (lse && !aligned16(lse[l]))
            return fail(TSI_ERR_INVALID_ARG, "layer %d: lse must be 16-byte aligned", l);
        if (!use_tc_attn(H, Hkv, Dqk, Dv, vk) && !tsi::attn_generic_supported(H, Hkv, Dqk, Dv, vk))
            return fail(TSI_ERR_UNSUPPORTED, "H=%d Hkv=%d Dqk=%d Dv=%d%s unsupported (Dqk<=576, "
                        "Dv<=512)", H, Hkv, Dqk, Dv, vk ? " (value from key)" : "");
    }
    const size_t need = tsi_sparse_attn_workspace(B, T, S, H, Hkv, Dqk, Dv, topk);
    if (workspace_bytes < need || (need > 0 && !workspace))
        return fail(TSI_ERR_WORKSPACE, "workspace %zu bytes, need %zu", workspace_bytes, need);
    if (need > 0 && !aligned16(workspace))
        return fail(TSI_ERR_INVALID_ARG, "workspace must be 16-byte aligned");
    unsigned* err = nullptr;
    tsi_status st = device_error_word(&err);
    if (st != TSI_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    for (int l = 0; l < n_layers; ++l) {
        const void* vl = v ? v[l] : nullptr;
        tsi::AttnArgs a{q[l], k[l], vl, B, T, S, H, Hkv, Dqk, Dv, scale, idx, topk, kv_len,
                        out[l], err, lse ? lse[l] : nullptr};
        cudaError_t e = use_tc_attn(H, Hkv, Dqk, Dv, vl == nullptr)
                            ? tsi::launch_attn_tc(a, workspace, s)
                            : tsi::launch_attn_generic(a, workspace, s);
        if (e != cudaSuccess)
            return fail(TSI_ERR_CUDA, "attention launch (layer %d): %s", l, cudaGetErrorString(e));
    }
    return ok();
}

tsi_status tsi_index_kl(int n_layers, const void* const* q, const void* const* k,
                        const float* const* lse, int B, int T, int S, int H, int Dqk, float scale,
                        const int32_t* idx, const float* score, int topk, const int32_t* kv_len,
                        float* loss, float* grad, float* pbar, void* stream) {
    if (n_layers < 1 || n_layers > tsi::kMaxIndexKlLayers)
        return fail(TSI_ERR_INVALID_ARG, "n_layers=%d outside [1, %d]", n_layers,
                    tsi::kMaxIndexKlLayers);
    if (B < 0 || T < 0 || S < 0)
        return fail(TSI_ERR_INVALID_ARG, "negative size (B=%d T=%d S=%d)", B, T, S);
    if (topk < 1 || topk > TSI_MAX_TOPK)
        return fail(TSI_ERR_UNSUPPORTED, "topk=%d outside [1, %d]", topk, TSI_MAX_TOPK);
    if (!tsi::tc_index_kl_supported(H, Dqk))
        return fail(TSI_ERR_UNSUPPORTED, "H=%d Dqk=%d unsupported (64 heads over the 576-d latent)",
                    H, Dqk);
    if (!std::isfinite(scale)) return fail(TSI_ERR_INVALID_ARG, "scale is not finite");
    if (static_cast<int64_t>(B) * T * H > (1ll << 31) - 1 || static_cast<int64_t>(B) * S > (1ll << 31) - 1)
        return fail(TSI_ERR_UNSUPPORTED, "B*T*H or B*S exceeds 2^31-1");
    if (B == 0 || T == 0) return ok();
    if (!q || !k || !lse || !idx || !score || !loss)
        return fail(TSI_ERR_INVALID_ARG, "NULL pointer (q, k, lse, idx, score and loss are required)");
    if (!aligned16(idx) || !aligned16(score) || !aligned16(kv_len) || !aligned16(loss) ||
        !aligned16(grad) || !aligned16(pbar))
        return fail(TSI_ERR_INVALID_ARG, "idx / score / kv_len / loss / grad / pbar must be 16-byte aligned");
    for (int l = 0; l < n_layers; ++l) {
        if (!q[l] || !lse[l] || (S > 0 && !k[l]))
            return fail(TSI_ERR_INVALID_ARG, "layer %d: NULL tensor pointer", l);
        if (!aligned16(q[l]) || !aligned16(k[l]) || !aligned16(lse[l]))
            return fail(TSI_ERR_INVALID_ARG, "layer %d: pointers must be 16-byte aligned", l);
    }
    unsigned* err = nullptr;
    tsi_status st = device_error_word(&err);
    if (st != TSI_OK) return st;
    tsi::IndexKlArgs a{n_layers, q, k, lse, B, T, S, scale, idx, score, topk, kv_len,
                       loss, grad, pbar, err};
    cudaError_t e = tsi::launch_index_kl_tc(a, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return fail(TSI_ERR_CUDA, "index KL launch: %s", cudaGetErrorString(e));
    return ok();
}

tsi_status tsi_selftest_wait_timeout(void* stream) {
    unsigned* err = nullptr;
    tsi_status st = device_error_word(&err);
    if (st != TSI_OK) return st;
    cudaError_t e = tsi::launch_wait_timeout_probe(err, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return fail(TSI_ERR_CUDA, "self-test launch: %s", cudaGetErrorString(e));
    return ok();
}

tsi_status tsi_index_share_layers(int n_layers, int freq, int skip_offset, const char* pattern,
                                  int32_t* anchor) {
    if (n_layers < 0) return fail(TSI_ERR_INVALID_ARG, "n_layers=%d", n_layers);
    if (n_layers == 0) return ok();
    if (!anchor) return fail(TSI_ERR_INVALID_ARG, "NULL anchor array");
    if (pattern) {
        for (int l = 0; l < n_layers; ++l) {
            const char c = pattern[l];
            if (c != 'F' && c != 'S')
                return fail(TSI_ERR_INVALID_ARG, "pattern[%d] is not 'F' or 'S' (or the pattern "
                            "is shorter than %d layers)", l, n_layers);
        }
        if (pattern[n_layers] != '\0')
            return fail(TSI_ERR_INVALID_ARG, "pattern is longer than %d layers", n_layers);
    } else if (freq < 1 || skip_offset < 0) {
        return fail(TSI_ERR_INVALID_ARG, "freq=%d skip_offset=%d", freq, skip_offset);
    }
    int last_full = -1;
    for (int l = 0; l < n_layers; ++l) {
        const bool full = pattern ? pattern[l] == 'F'
                                  : (l < skip_offset || (l - skip_offset) % freq == 0);
        if (full) last_full = l;
        if (last_full < 0) return fail(TSI_ERR_INVALID_ARG, "layer 0 must be a Full layer");
        anchor[l] = last_full;
    }
    return ok();
}

tsi_status tsi_topk_overlap(const int32_t* idx_a, const int32_t* idx_b, int rows, int topk,
                            int32_t* inter, int32_t* card_a, void* stream) {
    if (rows < 0) return fail(TSI_ERR_INVALID_ARG, "rows=%d", rows);
    if (topk < 1 || topk > TSI_MAX_TOPK)
        return fail(TSI_ERR_UNSUPPORTED, "topk=%d outside [1, %d]", topk, TSI_MAX_TOPK);
    if (rows == 0) return ok();
    if (!idx_a || !idx_b || !inter || !card_a) return fail(TSI_ERR_INVALID_ARG, "NULL pointer");
    if (!aligned16(idx_a) || !aligned16(idx_b) || !aligned16(inter) || !aligned16(card_a))
        return fail(TSI_ERR_INVALID_ARG, "pointers must be 16-byte aligned");
    unsigned* err = nullptr;
    tsi_status st = device_error_word(&err);
    if (st != TSI_OK) return st;
    cudaError_t e = tsi::launch_topk_overlap(idx_a, idx_b, rows, topk, inter, card_a, err,
                                             static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return fail(TSI_ERR_CUDA, "overlap launch: %s", cudaGetErrorString(e));
    return ok();
}

tsi_status tsi_device_status(void* stream) {
    cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return fail(TSI_ERR_CUDA, "stream: %s", cudaGetErrorString(e));
    unsigned* err = nullptr;
    tsi_status st = device_error_word(&err);
    if (st != TSI_OK) return st;
    unsigned word = 0;
    e = cudaMemcpy(&word, err, sizeof word, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return fail(TSI_ERR_CUDA, "read error word: %s", cudaGetErrorString(e));
    if (word) {
        const unsigned zero = 0;
        e = cudaMemcpy(err, &zero, sizeof zero, cudaMemcpyHostToDevice);
        if (e != cudaSuccess) return fail(TSI_ERR_CUDA, "clear error word: %s", cudaGetErrorString(e));
    }
    if (word & tsi::kErrTimeout)
        return fail(TSI_ERR_TIMEOUT, "a bounded device-side wait ran out (word 0x%x)", word);
    if (word & tsi::kErrAssert)
        return fail(TSI_ERR_DEVICE_ASSERT, "a device-side check failed (word 0x%x)", word);
    return ok();
}

}  // extern "C"

// ---------------------------------------------------------------------------------------
// Allocation-free indexer + top-k.
//
// For callers that cannot allocate device memory while they run: a serving loop whose
// device memory budget is fixed at start-up, or code called from inside a custom device
// allocator, where a nested cudaMalloc would recurse into the allocator or synchronize the
// device.  tsi_indexer_topk needs a caller-provided workspace when rows are few and key
// ranges are split across thread blocks (decode); this variant keeps that scratch in one
// fixed array compiled into the library instead.
//
// The array below is in device memory of every GPU that loads the library and stays
// there until the process exits.  Its host-side name is only a stand-in for the device
// symbol, so the device address is looked up with cudaGetSymbolAddress, once per device,
// on the first call made while that device is current.
// ---------------------------------------------------------------------------------------

static constexpr size_t kNoAllocScratchBytes = size_t(8) << 20;  // 8 MiB per device
static __device__ __align__(256) unsigned char tsi_noalloc_scratch[kNoAllocScratchBytes];

namespace {

void* g_noalloc_ptr[kMaxDevices] = {};
std::mutex g_noalloc_mu;

// Device address of tsi_noalloc_scratch on the current device (looked up once).
tsi_status noalloc_scratch_address(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(TSI_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    if (dev < 0 || dev >= kMaxDevices) return fail(TSI_ERR_CUDA, "device id %d out of range", dev);
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, tsi_noalloc_scratch);
        if (e != cudaSuccess)
            return fail(TSI_ERR_CUDA, "cudaGetSymbolAddress(scratch): %s", cudaGetErrorString(e));
        g_noalloc_ptr[dev] = p;
    }
    *out = g_noalloc_ptr[dev];
    return TSI_OK;
}

}  // namespace

extern "C" {

size_t tsi_indexer_topk_noalloc_limit(void) { return kNoAllocScratchBytes; }

tsi_status tsi_indexer_topk_noalloc(const void* qI, const void* kI, const void* w, int qk_dtype,
                                    int w_dtype, int B, int T, int S, int H_I, int d_I,
                                    int topk, const int32_t* kv_len, int32_t* idx, float* score,
                                    void* stream) {
    if (!qk_dtype_ok(qk_dtype)) return fail(TSI_ERR_INVALID_ARG, "qk_dtype %d unknown", qk_dtype);
    if (!w_dtype_ok(w_dtype)) return fail(TSI_ERR_INVALID_ARG, "w_dtype %d unknown", w_dtype);
    if (B < 0 || T < 0 || S < 0)
        return fail(TSI_ERR_INVALID_ARG, "negative size (B=%d T=%d S=%d)", B, T, S);
    if (topk < 1 || topk > TSI_MAX_TOPK)
        return fail(TSI_ERR_UNSUPPORTED, "topk=%d outside [1, %d]", topk, TSI_MAX_TOPK);
    if (H_I < 1 || d_I < 1) return fail(TSI_ERR_INVALID_ARG, "H_I=%d d_I=%d", H_I, d_I);
    if (!tsi::generic_supported(H_I, d_I))
        return fail(TSI_ERR_UNSUPPORTED, "H_I=%d d_I=%d unsupported (d_I<=256, H_I<=128, "
                    "H_I*d_I<=8192)", H_I, d_I);
    if (static_cast<int64_t>(B) * T > (1ll << 31) - 1 || static_cast<int64_t>(B) * S > (1ll << 31) - 1)
        return fail(TSI_ERR_UNSUPPORTED, "B*T or B*S exceeds 2^31-1");
    const size_t need = tsi::generic_workspace_bytes(B, T, S, topk);
    if (need > kNoAllocScratchBytes)
        return fail(TSI_ERR_UNSUPPORTED,
                    "request needs %zu bytes of scratch, more than the %zu-byte built-in array; "
                    "use tsi_indexer_topk with a workspace", need, kNoAllocScratchBytes);
    if (B == 0 || T == 0) return ok();
    if (!qI || !w || !idx || (S > 0 && !kI))
        return fail(TSI_ERR_INVALID_ARG, "NULL tensor pointer");
    if (!aligned16(qI) || !aligned16(kI) || !aligned16(w) || !aligned16(idx) ||
        !aligned16(score) || !aligned16(kv_len))
        return fail(TSI_ERR_INVALID_ARG, "tensor pointers must be 16-byte aligned");
    void* scratch = nullptr;
    tsi_status st = TSI_OK;
    if (need > 0) {
        st = noalloc_scratch_address(&scratch);
        if (st != TSI_OK) return st;
    }
    unsigned* err = nullptr;
    st = device_error_word(&err);
    if (st != TSI_OK) return st;
    // Every split writes its candidate count and list before the merge reads them, so
    // nothing in the scratch array has to start at zero.
    tsi::IndexerArgs a{qI, kI, w, qk_dtype, w_dtype, B, T, S, H_I, d_I, topk, kv_len,
                       idx, score, err};
    cudaError_t e = tsi::launch_indexer_generic(a, scratch, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return fail(TSI_ERR_CUDA, "indexer launch: %s", cudaGetErrorString(e));
    return ok();
}

}  // extern "C"
