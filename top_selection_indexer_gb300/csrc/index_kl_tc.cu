// Group-centroid KL target of a Full layer's indexer, fused over the group's layers
// (tcgen05 / TMEM).
//
// "GLM-5.2 技术报告速览" §IndexShare, "少数层挑，其余层复用": the indexer that serves a
// group of m + 1 layers is fitted, by KL, to the centroid of their head-averaged attention
// distributions,  pbar_t = 1/(m+1) sum_j p^(l+j)_t.  On the row's selected keys S_t (the
// only keys the group's sparse attention sees):
//
//   p^(l)_t[s] = 1/H sum_h exp(scale * Q_l[t,h] . K_l[s] - lse_l[t,h])
//   q_t[s]     = softmax_{s in S_t} I[t,s]
//   loss[t]    = sum_s pbar_t[s] (ln pbar_t[s] - ln q_t[s]),   grad = q_t - pbar_t
//
// with lse_l the per-head log-partition the layer's attention kernel already computed.
// The attention probabilities are never stored: each layer's logits are recomputed on the
// tensor core as S^T[key, h] = K_tile . Q^T (128 gathered keys x 64 heads, the product of
// the attention kernel), and one epilogue thread per key folds its 64 heads into one
// probability, accumulated over the layers in registers.  The key gather dominates:
// 1152 bytes per selected key per layer.
//
// Roles of one persistent CTA (512 threads), one query row at a time:
//   warps 0..3   epilogue: TMEM lane quadrant = warp; thread = key slot of the tile; the
//                row's loss, gradient and centroid at the end of its last layer.  Thread 0
//                also loads each layer's Q by TMA once the MMAs of the layer before are done.
//   warp 4       TMEM allocator + single-thread MMA issuer (S^T double-buffered in TMEM)
//   warps 5..15  gather of the selected latent rows (16-byte cp.async, swizzled chunks)
#include <mutex>

#include <cudaTypedefs.h>

#include "kernels_tc.cuh"
#include "latent_gather.cuh"
#include "tc_common.cuh"

namespace tsi {
namespace {

using latent::kChunkBytes;
using latent::kChunks;
using latent::kDqk;
using latent::kKeys;
constexpr int kHeads = 64;
constexpr int kMaxTiles = TSI_MAX_TOPK / kKeys;  // 16: a row's keys, 128 per tile
constexpr int kQChunkBytes = kHeads * 128;
constexpr int kThreads = 512;
constexpr int kEpiThreads = 128;
constexpr int kMmaWarp = 4;
constexpr int kGatherBase = 160;  // first gather thread (warp 5)
constexpr int kGather = kThreads - kGatherBase;  // 352
constexpr int kEpiBar = 1;
constexpr int kTmemCols = 128;  // two S^T buffers of 64 columns
constexpr uint32_t kIdescS = tc::instr_desc(1, 128, 64, 0, 0);
constexpr float kLog2e = 1.4426950408889634f;

struct Smem {
    uint64_t kv_full[kChunks];
    uint64_t kv_empty[kChunks];
    uint64_t q_full;
    uint64_t s_full[2];
    uint64_t s_empty[2];
    uint64_t done;
    alignas(16) float nl[kMaxIndexKlLayers][kHeads];  // -lse * log2(e) of the row, per layer and head
    float red[3][4];  // per-warp partials of the row reductions
    uint32_t tmem_slot;
    int abort;
};
constexpr int kSmemBytes = 1024 + kChunks * kQChunkBytes + kChunks * kChunkBytes + sizeof(Smem);

struct QMaps {
    CUtensorMap q[kMaxIndexKlLayers];  // [rows * 64, 576] bf16 per layer, 64 x 64 boxes
};

struct KlParams {
    const uint16_t* k[kMaxIndexKlLayers];  // [B, S, 576] per layer
    const float* lse[kMaxIndexKlLayers];  // [rows, 64] per layer
    const int32_t* idx;  // [rows, topk]
    const float* score;  // [rows, topk]
    const int32_t* kv_len;
    float* loss;  // [rows]
    float* grad;  // [rows, topk] or nullptr
    float* pbar;  // [rows, topk] or nullptr
    int n_layers, B, T, S, topk, n_tiles, rows;
    float scale_log2;
    float inv_norm;  // 1 / (n_layers * 64)
    unsigned* err;
};

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Sum (op 0) or maximum (op 1) over the 128 epilogue threads, in a fixed order.
__device__ __forceinline__ float epi_reduce(float v, int op, float* red, int warp, int lane) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float u = __shfl_xor_sync(kFull, v, o);
        v = op ? fmaxf(v, u) : v + u;
    }
    if (lane == 0) red[warp] = v;
    named_bar(kEpiBar, kEpiThreads);
    return op ? fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]))
              : (red[0] + red[1]) + (red[2] + red[3]);
}

// TMA loads of the 64 query rows of `row` in `layer` (nine 64-dim chunks).
__device__ __forceinline__ void load_q(const QMaps& maps, uint8_t* qs, int layer, int row,
                                       uint64_t* q_full) {
    tc::mbar_expect_tx(q_full, kChunks * kQChunkBytes);
    for (int c = 0; c < kChunks; ++c)
        tc::tma_load_2d(qs + c * kQChunkBytes, &maps.q[layer], c * 64, row * kHeads, q_full);
}

__global__ void __launch_bounds__(kThreads, 1)
    tsi_index_kl_tc_kernel(const __grid_constant__ QMaps maps, const __grid_constant__ KlParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* qs = base;
    uint8_t* kv = qs + kChunks * kQChunkBytes;
    Smem& sm = *reinterpret_cast<Smem*>(kv + kChunks * kChunkBytes);
    volatile int* abort = &sm.abort;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int c = 0; c < kChunks; ++c) {
            tc::mbar_init(&sm.kv_full[c], kGather);
            tc::mbar_init(&sm.kv_empty[c], 1);
        }
        tc::mbar_init(&sm.q_full, 1);
        for (int b = 0; b < 2; ++b) {
            tc::mbar_init(&sm.s_full[b], 1);
            tc::mbar_init(&sm.s_empty[b], kEpiThreads);
        }
        tc::mbar_init(&sm.done, 1);
        sm.abort = 0;
        tc::fence_barrier_init();
    }
    if (warp == kMmaWarp) tc::tmem_alloc(&sm.tmem_slot, kTmemCols);
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = sm.tmem_slot;
    const uint32_t q_addr = tc::smem_addr(qs);
    const uint32_t kv_addr = tc::smem_addr(kv);

    if (warp == kMmaWarp) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            int it = 0, qn = 0;
            for (int row = blockIdx.x; row < p.rows; row += gridDim.x) {
                for (int l = 0; l < p.n_layers; ++l, ++qn) {
                    tc::mbar_wait(&sm.q_full, qn & 1, abort, p.err);
                    for (int t = 0; t < p.n_tiles; ++t, ++it) {
                        const int b = it & 1;
                        tc::mbar_wait(&sm.s_empty[b], ((it >> 1) & 1) ^ 1, abort, p.err);
                        tc::tc_fence_after();
                        for (int c = 0; c < kChunks; ++c) {
                            tc::mbar_wait(&sm.kv_full[c], it & 1, abort, p.err);
                            tc::fence_proxy_async();  // cp.async landed via the generic proxy
                            tc::tc_fence_after();
                            if (!*abort) {
#pragma unroll
                                for (int kk = 0; kk < 4; ++kk) {
                                    const uint64_t da = tc::smem_desc(
                                        kv_addr + c * kChunkBytes + kk * 32, 16, 1024);
                                    const uint64_t db = tc::smem_desc(
                                        q_addr + c * kQChunkBytes + kk * 32, 16, 1024);
                                    tc::mma_bf16(tmem + 64 * b, da, db, kIdescS, (c | kk) ? 1u : 0u);
                                }
                            }
                            tc::mma_commit(&sm.kv_empty[c]);
                        }
                        tc::mma_commit(&sm.s_full[b]);
                    }
                }
            }
            tc::mma_commit(&sm.done);
            if (!tc::mbar_wait(&sm.done, 0, abort, p.err))
                tc::mbar_drain(&sm.done, 0);  // issued MMAs finish before TMEM is freed
        }
    } else if (warp > kMmaWarp) {
        // ------------------------------------------------------------ gather
        const int g = threadIdx.x - kGatherBase;
        int it = 0;
        for (int row = blockIdx.x; row < p.rows; row += gridDim.x) {
            const int bs = row / p.T;
            const int64_t len = seq_len(p.kv_len, bs, p.S);
            const int32_t* irow = p.idx + static_cast<int64_t>(row) * p.topk;
            for (int l = 0; l < p.n_layers; ++l) {
                const uint16_t* kseq = p.k[l] + static_cast<int64_t>(bs) * p.S * kDqk;
                for (int t = 0; t < p.n_tiles; ++t, ++it)
                    latent::gather_tile<kGather>(kseq, len, irow, p.topk, t, it, g, kv_addr,
                                                 sm.kv_empty, sm.kv_full, abort, p.err);
            }
        }
        asm volatile("cp.async.wait_all;" ::: "memory");
    } else {
        // ------------------------------------------------------------ epilogue
        const int k = warp * 32 + lane;  // key slot of a tile == TMEM lane
        const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
        const float neg_inf = -__int_as_float(0x7f800000);
        int it = 0, q_issued = 0;
        if (threadIdx.x == 0 && blockIdx.x < p.rows) {
            load_q(maps, qs, 0, blockIdx.x, &sm.q_full);
            ++q_issued;
        }
        for (int row = blockIdx.x; row < p.rows; row += gridDim.x) {
            const int bs = row / p.T;
            const int64_t len = seq_len(p.kv_len, bs, p.S);
            const int32_t* irow = p.idx + static_cast<int64_t>(row) * p.topk;
            for (int i = threadIdx.x; i < p.n_layers * kHeads; i += kEpiThreads)
                sm.nl[i / kHeads][i % kHeads] =
                    -p.lse[i / kHeads][static_cast<int64_t>(row) * kHeads + i % kHeads] * kLog2e;
            named_bar(kEpiBar, kEpiThreads);
            float pacc[kMaxTiles];  // head sums of this thread's keys, over the layers
#pragma unroll
            for (int t = 0; t < kMaxTiles; ++t) pacc[t] = 0.f;
            for (int l = 0; l < p.n_layers; ++l) {
                const float* nl = sm.nl[l];
#pragma unroll
                for (int t = 0; t < kMaxTiles; ++t) {
                    if (t < p.n_tiles) {
                        const int b = it & 1;
                        tc::mbar_wait(&sm.s_full[b], (it >> 1) & 1, abort, p.err);
                        tc::tc_fence_after();
                        if (threadIdx.x == 0 && t == p.n_tiles - 1 && !*abort) {
                            // every MMA of this layer is done: the Q buffer is free
                            const int nl_ = l + 1 < p.n_layers ? l + 1 : 0;
                            const int nr = l + 1 < p.n_layers ? row : row + gridDim.x;
                            if (nr < p.rows) {
                                load_q(maps, qs, nl_, nr, &sm.q_full);
                                ++q_issued;
                            }
                        }
                        uint32_t z[64];  // logits of this key, heads 0..63
                        TSI_TMEM_LD32(tmem + lane_base + 64 * b, z);
                        TSI_TMEM_LD32(tmem + lane_base + 64 * b + 32, (z + 32));
                        tc::tmem_wait_ld();
                        tc::tc_fence_before();
                        tc::mbar_arrive(&sm.s_empty[b]);
                        float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
                        for (int h = 0; h < kHeads; h += 4) {
                            const float4 n4 = *reinterpret_cast<const float4*>(nl + h);
                            acc0 += ex2(fmaf(__uint_as_float(z[h]), p.scale_log2, n4.x));
                            acc1 += ex2(fmaf(__uint_as_float(z[h + 1]), p.scale_log2, n4.y));
                            acc0 += ex2(fmaf(__uint_as_float(z[h + 2]), p.scale_log2, n4.z));
                            acc1 += ex2(fmaf(__uint_as_float(z[h + 3]), p.scale_log2, n4.w));
                        }
                        pacc[t] += acc0 + acc1;
                        ++it;
                    }
                }
            }
            // ------------------------------------------ the row's KL and gradient
            float sc[kMaxTiles], pb[kMaxTiles];
            float m = neg_inf;
#pragma unroll
            for (int t = 0; t < kMaxTiles; ++t) {
                const int e = t * kKeys + k;
                const int s = (t < p.n_tiles && e < p.topk) ? irow[e] : -1;
                const bool valid = s >= 0 && s < len;
                sc[t] = valid ? p.score[static_cast<int64_t>(row) * p.topk + e] : neg_inf;
                pb[t] = valid ? pacc[t] * p.inv_norm : -1.f;  // -1 marks a non-key
                m = fmaxf(m, sc[t]);
            }
            m = epi_reduce(m, 1, sm.red[0], warp, lane);
            float z = 0.f;
#pragma unroll
            for (int t = 0; t < kMaxTiles; ++t)
                if (pb[t] >= 0.f) z += expf(sc[t] - m);
            z = epi_reduce(z, 0, sm.red[1], warp, lane);
            const float log_z = m + logf(z);
            float kl = 0.f;
#pragma unroll
            for (int t = 0; t < kMaxTiles; ++t)
                if (pb[t] > 0.f) kl += pb[t] * (logf(pb[t]) - (sc[t] - log_z));
            kl = epi_reduce(kl, 0, sm.red[2], warp, lane);
            if (threadIdx.x == 0) p.loss[row] = z > 0.f ? kl : 0.f;
#pragma unroll
            for (int t = 0; t < kMaxTiles; ++t) {
                const int e = t * kKeys + k;
                if (t < p.n_tiles && e < p.topk) {
                    const int64_t o = static_cast<int64_t>(row) * p.topk + e;
                    const bool valid = pb[t] >= 0.f;
                    if (p.grad) p.grad[o] = valid ? expf(sc[t] - log_z) - pb[t] : 0.f;
                    if (p.pbar) p.pbar[o] = valid ? pb[t] : 0.f;
                }
            }
        }
        // a Q load still in flight after an abort must land before the CTA exits
        if (threadIdx.x == 0 && *abort && q_issued > 0) {
            const long long t0 = clock64();
            while (!tc::mbar_try_wait(&sm.q_full, (q_issued - 1) & 1) &&
                   clock64() - t0 < tc::kWaitCycles) {
            }
        }
    }
    tc::tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc::tc_fence_after();
        tc::tmem_dealloc(tmem, kTmemCols);
    }
}

// ------------------------------------------------------------------------------ host

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        cudaDriverEntryPointQueryResult q;
        void* f = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    });
    return fn;
}

int sm_count() {
    static int n = 0;
    static std::once_flag once;
    std::call_once(once, [] {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        if (n <= 0) n = 152;
    });
    return n;
}

}  // namespace

bool tc_index_kl_supported(int H, int Dqk) { return H == kHeads && Dqk == kDqk; }

cudaError_t launch_index_kl_tc(const IndexKlArgs& a, cudaStream_t st) {
    const int rows = a.B * a.T;
    if (rows == 0) return cudaSuccess;
    if (a.n_layers < 1 || a.n_layers > kMaxIndexKlLayers) return cudaErrorInvalidValue;
    auto fn = encode_fn();
    if (!fn) return cudaErrorNotSupported;
    QMaps maps;
    KlParams p{};
    for (int l = 0; l < a.n_layers; ++l) {
        cuuint64_t dims[2] = {static_cast<cuuint64_t>(kDqk), static_cast<cuuint64_t>(rows) * kHeads};
        cuuint64_t strides[1] = {static_cast<cuuint64_t>(kDqk) * 2};
        cuuint32_t box[2] = {64, kHeads};
        cuuint32_t estr[2] = {1, 1};
        if (fn(&maps.q[l], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(a.q[l]), dims,
               strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
        p.k[l] = static_cast<const uint16_t*>(a.k[l]);
        p.lse[l] = a.lse[l];
    }
    for (int l = a.n_layers; l < kMaxIndexKlLayers; ++l) maps.q[l] = maps.q[0];
    p.idx = a.idx;
    p.score = a.score;
    p.kv_len = a.kv_len;
    p.loss = a.loss;
    p.grad = a.grad;
    p.pbar = a.pbar;
    p.n_layers = a.n_layers;
    p.B = a.B;
    p.T = a.T;
    p.S = a.S;
    p.topk = a.topk;
    p.n_tiles = (a.topk + kKeys - 1) / kKeys;
    p.rows = rows;
    p.scale_log2 = a.scale * kLog2e;
    p.inv_norm = 1.f / static_cast<float>(a.n_layers * kHeads);
    p.err = a.err;
    cudaError_t e = cudaFuncSetAttribute(tsi_index_kl_tc_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    const int grid = rows < sm_count() ? rows : sm_count();
    tsi_index_kl_tc_kernel<<<grid, kThreads, kSmemBytes, st>>>(maps, p);
    note_launches(1);
    return cudaGetLastError();
}

}  // namespace tsi
