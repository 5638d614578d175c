// Tensor-core sparse MQA attention over the shared index rows (tcgen05 / TMEM).
//
// For every query row t (64 heads) of a layer and its selected keys S_t:
//   O[t,h] = sum_{s in S_t} softmax_s(scale * Q[t,h] . K[s]) V[s]
// with K = the 576-d latent row of key s and V = its first 512 dims ("GLM-5.2
// 技术报告速览" §IndexShare: each layer runs its own sparse attention over the Full
// layer's index set; "GLM 5.2: Built for Long Horizon Tasks" discussion §3: 576-d MLA
// latent, 512 compressed + 64 RoPE dims, sparse attention over the indices).
//
// Both products are computed transposed so that the 128 gathered keys of a tile are the
// MMA's M dimension and the 64 heads its N dimension:
//   S^T[key, h] = K_tile . Q^T         (A = key rows, K-major; B = Q rows, K-major)
//   O^T[d, h]  += V_tile^T . P^T       (A = the same key rows read MN-major as V^T,
//                                       B = P^T written by the softmax threads)
// O^T (512 x 64 fp32) lives in TMEM for the whole row; S^T takes 64 more columns.  One
// softmax thread owns one key (one TMEM lane of S^T) and all 64 heads of it, so the
// exponentials, the bf16 rounding of P and the running row sums need no cross-thread
// traffic; the running max per head is refreshed only when a logit exceeds it by 2^16
// (always on the first tile of a row), and then O^T is rescaled in place.
//
// Roles of one persistent CTA (512 threads):
//   warp 4        TMEM allocator + single-thread MMA issuer
//   other warps   gather: 16-byte cp.async of the selected latent rows into nine 128-byte-
//                 swizzled 64-dim chunk tiles (per-chunk mbarriers); warp 5 also loads Q
//                 by TMA.  The gather rate of cp.async grows with the number of issuing
//                 warps, so all 15 take part.
//   warps 0..3,   softmax (writes P^T over the RoPE chunk once S^T is done) and the row
//   8..11         epilogue (1/l normalisation, bf16 stores), heads 0..31 on warps 0..3 and
//                 32..63 on warps 8..11: two warps per TMEM lane quadrant.  They gather
//                 the next tile after writing P, when its chunks start to free up.
// Row sums l[h] = sum_s P[h,s] come from the tensor core too: a fifth M=128 block
// multiplies a 128-byte tile of ones (no-swizzle descriptor, zero strides: every core
// matrix reads the same bytes) by P^T, so l sums exactly the bf16 P that multiplies V.
// Few rows (decode): a row's key tiles are split over CTAs and the unnormalised partials
// are merged by the combine kernel.
#include <mutex>

#include <cudaTypedefs.h>

#include "kernels_tc.cuh"
#include "latent_gather.cuh"
#include "tc_common.cuh"
#include "topk_select.cuh"

namespace tsi {
namespace {

constexpr int kKeys = 128;  // keys per tile: MMA M of S^T, MMA K of O^T
constexpr int kHeads = 64;  // MMA N
constexpr int kDqk = 576;
constexpr int kDv = 512;
constexpr int kChunks = kDqk / 64;  // 9 chunks of 64 dims (128 bytes) per latent row
constexpr int kKVChunkBytes = kKeys * 128;
static_assert(kKeys == latent::kKeys && kChunks == latent::kChunks &&
                  kKVChunkBytes == latent::kChunkBytes && kDqk == latent::kDqk,
              "the gather helper fills the tiles this kernel multiplies");
constexpr int kQChunkBytes = kHeads * 128;
constexpr int kPSlot = 8;  // the RoPE chunk's slot holds P^T once S^T is done
// 16 warps: warp 4 issues the MMAs; the other 15 gather.  Warps 0..3 and 8..11 also run
// the softmax and the row epilogue, warps 0..3 for heads 0..31 and 8..11 for heads
// 32..63 of the keys in their TMEM lane quadrant (warp % 4).
constexpr int kThreads = 512;
constexpr int kMmaWarp = 4;
constexpr int kGather = kThreads - 32;  // gathering threads (all but the MMA warp)
constexpr int kGatherQ = 128;  // gather index of the thread that loads Q (warp 5, lane 0)
constexpr int kSoftThreads = 256;
constexpr int kSoftBar = 1;
__device__ __forceinline__ bool is_softmax_warp(int w) { return (w & 4) == 0; }
constexpr int kTmemCols = 512;
constexpr int kColS = 0;
constexpr int kColO = 64;  // O^T block m (d rows 128m..128m+127) at columns 64 + 64m
constexpr int kColL = kColO + 256;  // row sums (every lane holds the same 64 values)
constexpr float kRescaleLog2 = 16.f;
constexpr uint32_t kIdescS = tc::instr_desc(1, 128, 64, 0, 0);
constexpr uint32_t kIdescO = tc::instr_desc(1, 128, 64, 1, 1);
constexpr uint32_t kIdescL = tc::instr_desc(1, 128, 64, 0, 1);

constexpr int kMiscBytes = 64 * 4 * 4 + 4 * 64 * 4 + 32 * 8 + 16;
constexpr int kSmemBytes = 1024 + kChunks * kQChunkBytes + kChunks * kKVChunkBytes + kMiscBytes;

struct AttnTcParams {
    const uint16_t* k;  // latent [B, S, 576] bf16
    const int32_t* idx;  // [B*T, topk]
    const int32_t* kv_len;
    __nv_bfloat16* out;  // [B*T, 64, 512]
    float* part_o;  // split partials or nullptr
    float* part_ml;
    int B, T, S, topk;
    int tiles_per_row, n_splits, tiles_per_split, n_units;
    float scale_log2;
    unsigned* err;
    float* lse;  // [B*T, 64] or nullptr (unsplit rows; split rows get it from the combine)
};

struct Work {
    int row, b, split, tile0, tile1;
};

__device__ __forceinline__ Work work_of(const AttnTcParams& p, int u) {
    Work w;
    w.split = u % p.n_splits;
    w.row = u / p.n_splits;
    w.b = w.row / p.T;
    w.tile0 = w.split * p.tiles_per_split;
    w.tile1 = w.tile0 + p.tiles_per_split < p.tiles_per_row ? w.tile0 + p.tiles_per_split
                                                             : p.tiles_per_row;
    return w;
}

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
    const uint32_t lo = __bfloat16_as_ushort(__float2bfloat16_rn(a));
    const uint32_t hi = __bfloat16_as_ushort(__float2bfloat16_rn(b));
    return lo | (hi << 16);
}

// This thread's share of the gather of key tile t of work item W (the latent rows of the
// row's selected keys, zero-filled past kv_len and past topk).
__device__ __forceinline__ void gather_tile(const AttnTcParams& p, const Work& W, int t, int it,
                                            int g, uint32_t kv_addr, uint64_t* kv_empty,
                                            uint64_t* kv_full, volatile int* abort) {
    latent::gather_tile<kGather>(p.k + static_cast<int64_t>(W.b) * p.S * kDqk,
                                 seq_len(p.kv_len, W.b, p.S),
                                 p.idx + static_cast<int64_t>(W.row) * p.topk, p.topk, t, it, g,
                                 kv_addr, kv_empty, kv_full, abort, p.err);
}

__global__ void __launch_bounds__(kThreads, 1)
    tsi_attn_tc_kernel(const __grid_constant__ CUtensorMap tmap_q, const AttnTcParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* qs = base;
    uint8_t* kv = qs + kChunks * kQChunkBytes;
    float* m_s = reinterpret_cast<float*>(kv + kChunks * kKVChunkBytes);  // running max [64]
    uint32_t* tmax_s = reinterpret_cast<uint32_t*>(m_s + 64);  // tile max (order bits) [64]
    float* alpha_s = reinterpret_cast<float*>(tmax_s + 64);  // rescale factors [64]
    float* l_s = alpha_s + 64;  // row sums of the unit [64]
    uint16_t* ones = reinterpret_cast<uint16_t*>(l_s + 64);  // 64 x bf16 1.0 (128 bytes)
    uint64_t* bars = reinterpret_cast<uint64_t*>(l_s + 64 + 4 * 64);
    uint64_t* kv_full = bars;
    uint64_t* kv_empty = bars + kChunks;
    uint64_t* q_full = bars + 2 * kChunks;
    uint64_t* q_empty = q_full + 1;
    uint64_t* s_full = q_full + 2;
    uint64_t* p_full = q_full + 3;
    uint64_t* o_full = q_full + 4;
    uint64_t* o_empty = q_full + 5;
    uint64_t* done = q_full + 6;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(q_full + 7);
    volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x < 64) ones[threadIdx.x] = 0x3F80;  // bf16 1.0
    tc::fence_proxy_async();  // read by the tensor core
    if (threadIdx.x == 0) {
        for (int c = 0; c < kChunks; ++c) {
            tc::mbar_init(&kv_full[c], kGather);
            tc::mbar_init(&kv_empty[c], 1);
        }
        tc::mbar_init(q_full, 1);
        tc::mbar_init(q_empty, 1);
        tc::mbar_init(s_full, 1);
        tc::mbar_init(p_full, kSoftThreads);
        tc::mbar_init(o_full, 1);
        tc::mbar_init(o_empty, kSoftThreads);
        tc::mbar_init(done, 1);
        *abort = 0;
        tc::fence_barrier_init();
    }
    if (warp == kMmaWarp) {
        tc::tmem_alloc(tmem_slot, kTmemCols);
        if (lane == 0) tc::prefetch_tmap(&tmap_q);
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t q_addr = tc::smem_addr(qs);
    const uint32_t kv_addr = tc::smem_addr(kv);

    if (warp == kMmaWarp) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            int it = 0, r_it = 0;
            for (int u = blockIdx.x; u < p.n_units; u += gridDim.x, ++r_it) {
                const Work W = work_of(p, u);
                tc::mbar_wait(q_full, r_it & 1, abort, p.err);
                for (int t = W.tile0; t < W.tile1; ++t, ++it) {
                    const bool first = t == W.tile0;
                    for (int c = 0; c < kChunks; ++c) {
                        tc::mbar_wait(&kv_full[c], it & 1, abort, p.err);
                        tc::fence_proxy_async();  // cp.async landed via the generic proxy
                        tc::tc_fence_after();
                        if (!*abort) {
#pragma unroll
                            for (int kk = 0; kk < 4; ++kk) {
                                const uint64_t da = tc::smem_desc(
                                    kv_addr + c * kKVChunkBytes + kk * 32, 16, 1024);
                                const uint64_t db = tc::smem_desc(
                                    q_addr + c * kQChunkBytes + kk * 32, 16, 1024);
                                tc::mma_bf16(tmem + kColS, da, db, kIdescS, (c | kk) ? 1u : 0u);
                            }
                        }
                    }
                    tc::mma_commit(s_full);
                    if (t == W.tile1 - 1) tc::mma_commit(q_empty);
                    tc::mbar_wait(p_full, it & 1, abort, p.err);
                    if (first) tc::mbar_wait(o_empty, (r_it & 1) ^ 1, abort, p.err);
                    tc::fence_proxy_async();  // P^T written with generic stores
                    tc::tc_fence_after();
                    for (int m = 0; m < 4; ++m) {
                        if (!*abort) {
#pragma unroll
                            for (int kk = 0; kk < 8; ++kk) {
                                const uint64_t da = tc::smem_desc(
                                    kv_addr + 2 * m * kKVChunkBytes + kk * 2048, kKVChunkBytes, 1024);
                                const uint64_t db = tc::smem_desc(
                                    kv_addr + kPSlot * kKVChunkBytes + kk * 2048, kKVChunkBytes, 1024);
                                tc::mma_bf16(tmem + kColO + 64 * m, da, db, kIdescO,
                                             (first && kk == 0) ? 0u : 1u);
                            }
                        }
                        tc::mma_commit(&kv_empty[2 * m]);
                        tc::mma_commit(&kv_empty[2 * m + 1]);
                    }
                    if (!*abort) {  // row sums: ones[128 x 16] . P^T per 16-key step
                        const uint64_t da = tc::smem_desc(tc::smem_addr(ones), 0, 0, 0);
#pragma unroll
                        for (int kk = 0; kk < 8; ++kk) {
                            const uint64_t db = tc::smem_desc(
                                kv_addr + kPSlot * kKVChunkBytes + kk * 2048, kKVChunkBytes, 1024);
                            tc::mma_bf16(tmem + kColL, da, db, kIdescL, (first && kk == 0) ? 0u : 1u);
                        }
                    }
                    tc::mma_commit(&kv_empty[kPSlot]);
                }
                tc::mma_commit(o_full);
            }
            tc::mma_commit(done);
            tc::mbar_wait(done, 0, abort, p.err);
        }
    } else {
        // gather index: threads 0..127 and 160..511 (warp 4 issues the MMAs)
        const int g = threadIdx.x < 128 ? static_cast<int>(threadIdx.x) : threadIdx.x - 32;
        int it = 0, r_it = 0;
        if (!is_softmax_warp(warp)) {
            // -------------------------------------------------------- gather only
            for (int u = blockIdx.x; u < p.n_units; u += gridDim.x, ++r_it) {
                const Work W = work_of(p, u);
                if (g == kGatherQ) {
                    tc::mbar_wait(q_empty, (r_it & 1) ^ 1, abort, p.err);
                    if (!*abort) {
                        tc::mbar_expect_tx(q_full, kChunks * kQChunkBytes);
                        for (int c = 0; c < kChunks; ++c)
                            tc::tma_load_2d(qs + c * kQChunkBytes, &tmap_q, c * 64,
                                            W.row * kHeads, q_full);
                    }
                }
                for (int t = W.tile0; t < W.tile1; ++t, ++it)
                    gather_tile(p, W, t, it, g, kv_addr, kv_empty, kv_full, abort);
            }
        } else {
            // -------------------------------------------- gather, softmax + row epilogue
            const int sw = warp < 4 ? warp : warp - 4;  // softmax warp 0..7
            const int st = sw * 32 + lane;
            const int quad = warp & 3;  // TMEM lanes 32*quad .. 32*quad+31
            const int h0 = 32 * (warp >> 3);  // this warp's heads h0 .. h0+31
            const int k = quad * 32 + lane;  // key slot of the tile owned by this thread
            const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
            const float neg_inf = -__int_as_float(0x7f800000);
            uint8_t* prow = kv + kPSlot * kKVChunkBytes + (k >> 3) * 1024 + (k & 7) * 128;
            for (int u = blockIdx.x; u < p.n_units; u += gridDim.x, ++r_it) {
                const Work W = work_of(p, u);
                const int64_t len = seq_len(p.kv_len, W.b, p.S);
                const int32_t* irow = p.idx + static_cast<int64_t>(W.row) * p.topk;
                if (st < 64) {
                    m_s[st] = neg_inf;
                    tmax_s[st] = 0u;
                }
                named_bar(kSoftBar, kSoftThreads);
                for (int t = W.tile0; t < W.tile1; ++t, ++it) {
                    // the chunks of tile t free up as the MMA finishes tile t-1 with them,
                    // and this warp has already written that tile's P
                    gather_tile(p, W, t, it, g, kv_addr, kv_empty, kv_full, abort);
                    const int e = t * kKeys + k;
                    const int s = e < p.topk ? irow[e] : -1;
                    const bool valid = s >= 0 && s < len;
                    tc::mbar_wait(s_full, it & 1, abort, p.err);
                    tc::tc_fence_after();
                    const uint32_t s_addr = tmem + lane_base + kColS + h0;
                    uint32_t z[32];  // logits of this key for heads h0 .. h0+31
                    TSI_TMEM_LD32(s_addr, z);
                    tc::tmem_wait_ld();
                    // does any logit of the tile exceed the running max of its head by 2^16?
                    bool over = false;
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        over |= valid && (__uint_as_float(z[j]) * p.scale_log2 > m_s[h0 + j] + kRescaleLog2);
                    if (tc::bar_red_or(kSoftBar, kSoftThreads, over)) {
                        // exact tile max per head, new running max, rescale what O^T holds
#pragma unroll
                        for (int j = 0; j < 32; ++j) {
                            const float zh = valid ? __uint_as_float(z[j]) * p.scale_log2 : neg_inf;
                            const uint32_t v = __reduce_max_sync(kFull, score_order_bits(zh));
                            if (lane == 0) atomicMax(&tmax_s[h0 + j], v);
                        }
                        named_bar(kSoftBar, kSoftThreads);
                        if (st < 64) {
                            const float mo = m_s[st];
                            const float mn = fmaxf(mo, order_bits_score(tmax_s[st]));
                            alpha_s[st] = mo == neg_inf ? 0.f : ex2(mo - mn);
                            m_s[st] = mn;
                            tmax_s[st] = 0u;
                        }
                        named_bar(kSoftBar, kSoftThreads);
                        if (t != W.tile0) {
                            for (int m = 0; m < 5; ++m) {  // the 4 O^T blocks and the row sums
                                uint32_t o[32];
                                const uint32_t ta = tmem + lane_base + kColO + 64 * m + h0;
                                TSI_TMEM_LD32(ta, o);
                                tc::tmem_wait_ld();
#pragma unroll
                                for (int j = 0; j < 32; ++j)
                                    o[j] = __float_as_uint(__uint_as_float(o[j]) * alpha_s[h0 + j]);
                                TSI_TMEM_ST32(ta, o);
                            }
                            tc::tmem_wait_st();
                        }
                    }
                    // P^T row of this key: heads h0 .. h0+31 as bf16, four 16-byte pieces of
                    // the 128-byte-swizzled row (MN-major B operand)
#pragma unroll
                    for (int jj = 0; jj < 4; ++jj) {
                        const int j = (h0 >> 3) + jj;
                        float pv[8];
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            const int h = 8 * j + i;
                            const float zh = __uint_as_float(z[8 * jj + i]) * p.scale_log2;
                            pv[i] = valid ? ex2(zh - m_s[h]) : 0.f;
                        }
                        uint4 v;
                        v.x = pack_bf16(pv[0], pv[1]);
                        v.y = pack_bf16(pv[2], pv[3]);
                        v.z = pack_bf16(pv[4], pv[5]);
                        v.w = pack_bf16(pv[6], pv[7]);
                        *reinterpret_cast<uint4*>(prow + ((j ^ (k & 7)) << 4)) = v;
                    }
                    tc::fence_proxy_async();
                    tc::tc_fence_before();
                    tc::mbar_arrive(p_full);
                }
                // ------------------------------------------------------ row epilogue
                tc::mbar_wait(o_full, r_it & 1, abort, p.err);
                tc::tc_fence_after();
                uint32_t lv[32];  // row sums of heads h0 .. h0+31 (same in every lane)
                TSI_TMEM_LD32(tmem + lane_base + kColL + h0, lv);
                tc::tmem_wait_ld();
                if (quad == 0 && lane == 0) {
#pragma unroll
                    for (int j = 0; j < 32; ++j) l_s[h0 + j] = __uint_as_float(lv[j]);
                }
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const float L = __uint_as_float(lv[j]);
                    lv[j] = __float_as_uint(L > 0.f ? 1.f / L : 0.f);
                }
                for (int m = 0; m < 4; ++m) {
                    const int d = 128 * m + 32 * quad + lane;
                    uint32_t o[32];
                    TSI_TMEM_LD32(tmem + lane_base + kColO + 64 * m + h0, o);
                    tc::tmem_wait_ld();
                    if (p.part_o) {
                        float* po = p.part_o +
                                    ((static_cast<int64_t>(W.row) * p.n_splits + W.split) * kHeads + h0) * kDv + d;
#pragma unroll
                        for (int j = 0; j < 32; ++j) po[static_cast<int64_t>(j) * kDv] = __uint_as_float(o[j]);
                    } else {
                        __nv_bfloat16* out = p.out + (static_cast<int64_t>(W.row) * kHeads + h0) * kDv + d;
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            out[static_cast<int64_t>(j) * kDv] =
                                __float2bfloat16_rn(__uint_as_float(o[j]) * __uint_as_float(lv[j]));
                    }
                }
                if (p.part_o) {
                    named_bar(kSoftBar, kSoftThreads);
                    if (st < 64) {
                        const int64_t slot = (static_cast<int64_t>(W.row) * p.n_splits + W.split) * kHeads + st;
                        p.part_ml[2 * slot] = m_s[st];
                        p.part_ml[2 * slot + 1] = l_s[st];
                    }
                } else if (p.lse) {
                    named_bar(kSoftBar, kSoftThreads);
                    if (st < 64) p.lse[static_cast<int64_t>(W.row) * kHeads + st] = lse_of(m_s[st], l_s[st]);
                }
                tc::tc_fence_before();
                tc::mbar_arrive(o_empty);
            }
        }
        asm volatile("cp.async.wait_all;" ::: "memory");
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

constexpr int kPlanSMs = 152;

void attn_tc_plan(int rows, int topk, int* n_splits, int* tiles_per_split, int* tiles) {
    const int nt = (topk + kKeys - 1) / kKeys;
    int ns = 1;
    if (rows > 0 && rows < kPlanSMs) {
        ns = (2 * kPlanSMs + rows - 1) / rows;
        if (ns > nt) ns = nt;
        if (ns < 1) ns = 1;
    }
    const int tps = (nt + ns - 1) / ns;
    *tiles = nt;
    *tiles_per_split = tps;
    *n_splits = (nt + tps - 1) / tps;
}

int sm_count() {
    static int n = 0;
    static std::once_flag once;
    std::call_once(once, [] {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        if (n <= 0) n = kPlanSMs;
    });
    return n;
}

}  // namespace

bool tc_attn_supported(int H, int Hkv, int Dqk, int Dv, bool v_from_k) {
    return H == kHeads && Hkv == 1 && Dqk == kDqk && Dv == kDv && v_from_k;
}

size_t tc_attn_workspace_bytes(int B, int T, int H, int Dv, int topk) {
    int ns, tps, nt;
    attn_tc_plan(B * T, topk, &ns, &tps, &nt);
    if (ns <= 1) return 0;
    const size_t slots = static_cast<size_t>(B) * T * ns * H;
    return slots * Dv * sizeof(float) + slots * 2 * sizeof(float);
}

cudaError_t launch_attn_tc(const AttnArgs& a, void* workspace, cudaStream_t st) {
    const int rows = a.B * a.T;
    if (rows == 0) return cudaSuccess;
    auto fn = encode_fn();
    if (!fn) return cudaErrorNotSupported;
    CUtensorMap tq;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(kDqk), static_cast<cuuint64_t>(rows) * kHeads};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(kDqk) * 2};
    cuuint32_t box[2] = {64, kHeads};
    cuuint32_t estr[2] = {1, 1};
    if (fn(&tq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(a.q), dims, strides, box,
           estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    AttnTcParams p{};
    p.k = static_cast<const uint16_t*>(a.k);
    p.idx = a.idx;
    p.kv_len = a.kv_len;
    p.out = static_cast<__nv_bfloat16*>(a.out);
    p.B = a.B;
    p.T = a.T;
    p.S = a.S;
    p.topk = a.topk;
    attn_tc_plan(rows, a.topk, &p.n_splits, &p.tiles_per_split, &p.tiles_per_row);
    p.n_units = rows * p.n_splits;
    p.scale_log2 = a.scale * 1.4426950408889634f;
    p.err = a.err;
    p.lse = a.lse;
    if (p.n_splits > 1) {
        p.part_o = static_cast<float*>(workspace);
        p.part_ml = p.part_o + static_cast<size_t>(rows) * p.n_splits * kHeads * kDv;
    }
    cudaError_t e = cudaFuncSetAttribute(tsi_attn_tc_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    const int grid = p.n_units < sm_count() ? p.n_units : sm_count();
    tsi_attn_tc_kernel<<<grid, kThreads, kSmemBytes, st>>>(tq, p);
    note_launches(1);
    e = cudaGetLastError();
    if (e != cudaSuccess || p.n_splits == 1) return e;
    return launch_attn_combine(a, p.n_splits, p.part_o, p.part_ml, st);
}

}  // namespace tsi
