// Tensor-core sparse MQA attention over the shared index rows (tcgen05 / TMEM).
//
// For every query row t (64 heads) of a layer and its selected keys S_t:
//   O[t,h] = sum_{s in S_t} softmax_s(scale * Q[t,h] . K[s]) V[s]
// with K = the 576-d latent row of key s and V = its first 512 dims ("GLM-5.2
// 技术报告速览" §IndexShare: each layer runs its own sparse attention over the Full
// layer's index set; "GLM 5.2: Built for Long Horizon Tasks" discussion §3: 576-d MLA
// latent, 512 compressed + 64 RoPE dims, sparse attention over the indices).
//
// A row's keys are taken 64 at a time (a half-tile) through two 72 KB shared-memory
// buffers, so the gather of the next half-tile runs while the current one is multiplied:
//   S[h, key]   = Q . K_half^T          (M = 64 heads, N = 64 keys, K = 576; A = Q rows,
//                                        B = the gathered key rows, both K-major)
//   O^T[d, h]  += V_half^T . P^T        (M = 128 value dims x 4 blocks, N = 64 heads,
//                                        K = 64 keys; A = the same key rows read MN-major
//                                        as V^T, B = P^T written by the softmax threads)
// O^T (512 x 64 fp32) lives in TMEM for the whole row; S takes 2 x 64 more columns (the
// M = 64 accumulator puts head h on TMEM lane 32 (h / 16) + h % 16).  Four softmax threads
// share a head (16 keys each), so the running max, the row sum of the bf16 probabilities
// that multiply V and P^T's row need two shuffles and no shared memory.  The
// running max is refreshed only when a logit exceeds it by 2^16 (always on a row's first
// keys), and then O^T is rescaled in place.
//
// Roles of one persistent CTA (512 threads):
//   warps 0..3    softmax (heads 16 w .. 16 w + 15, four threads per head, 16 keys each)
//                 and the row epilogue (O^T's value dims); thread 0 also loads Q by TMA
//   warp 4        TMEM allocator + issuer of the S products (lane 0 issues)
//   warp 5        issuer of the P.V products (lane 0 issues): the two streams of tcgen05
//                 work wait on different inputs, so neither holds up the other
//   warps 6..15   gather: 16-byte cp.async of the selected latent rows into the 128-byte-
//                 swizzled chunks of a half-tile buffer, one mbarrier per buffer
// Few rows (decode): a row's half-tiles are split over CTAs and the unnormalised partials
// are merged by the combine kernel.
#include <mutex>

#include <cudaTypedefs.h>

#include "kernels_tc.cuh"
#include "tc_common.cuh"
#include "topk_select.cuh"

namespace tsi {
namespace {

constexpr int kHalf = 64;  // keys per half-tile: MMA N of S, MMA K of O^T
constexpr int kHeads = 64;  // MMA M of S
constexpr int kDqk = 576;
constexpr int kDv = 512;
constexpr int kChunks = kDqk / 64;  // 9 chunks of 64 dims (128 bytes) per latent row
constexpr int kChunkBytes = kHalf * 128;  // one chunk of a half-tile: 8 KB
constexpr int kBufBytes = kChunks * kChunkBytes;  // one half-tile buffer: 72 KB
constexpr int kQChunkBytes = kHeads * 128;
constexpr int kPSlot = 8;  // the RoPE chunk's slot holds P^T once S is done
constexpr int kThreads = 512;
constexpr int kSoftThreads = 128;  // warps 0..3
constexpr int kMmaWarp = 4;  // issues S; also allocates TMEM
constexpr int kPvWarp = 5;  // issues P.V
constexpr int kGatherBase = 192;  // warp 6
constexpr int kGather = kThreads - kGatherBase;  // 320
constexpr int kPieces = kHalf * 8;  // 16-byte pieces per chunk of a half-tile
constexpr int kGatherPer = (kPieces + kGather - 1) / kGather;  // 2
constexpr int kSoftBar = 1;
constexpr int kTmemCols = 512;
constexpr int kColO = 0;  // O^T block m (value dims 128m .. 128m+127) at columns 64m
constexpr int kColS = 256;  // S buffer b at columns 256 + 64b
constexpr float kRescaleLog2 = 16.f;
constexpr uint32_t kIdescS = tc::instr_desc(1, 64, 64, 0, 0);
constexpr uint32_t kIdescO = tc::instr_desc(1, 128, 64, 1, 0);

struct Smem {
    uint64_t full[2];  // half-tile buffer b gathered
    uint64_t empty[2];  // half-tile buffer b released by its P.V
    uint64_t q_full;
    uint64_t s_full[2];
    uint64_t s_empty[2];
    uint64_t p_full[2];  // P^T of half-tile x written (x & 1: the softmax of x + 1 may
                         // finish before the MMA issuer has seen x's phase)
    uint64_t pv_done;
    uint64_t o_full;
    uint64_t o_empty;
    uint64_t done[2];  // each MMA issuer's work complete
    float alpha[kHeads];  // rescale factors of a running-max refresh
    alignas(16) float linv[kHeads];  // 1 / row sum, for the epilogue (read as float4)
    uint32_t tmem_slot;
    int abort;
};
constexpr int kSmemBytes =
    1024 + kChunks * kQChunkBytes + 2 * kBufBytes + static_cast<int>(sizeof(Smem));

struct AttnTcParams {
    const uint16_t* k;  // latent [B, S, 576] bf16
    const int32_t* idx;  // [B*T, topk]
    const int32_t* kv_len;
    __nv_bfloat16* out;  // [B*T, 64, 512]
    float* part_o;  // split partials or nullptr
    float* part_ml;
    int B, T, S, topk;
    int halves_per_row, n_splits, halves_per_split, n_units;
    float scale_log2;
    unsigned* err;
    float* lse;  // [B*T, 64] or nullptr (unsplit rows; split rows get it from the combine)
};

struct Work {
    int row, b, split, h0, h1;  // half-tiles h0 .. h1-1 of the row
};

__device__ __forceinline__ Work work_of(const AttnTcParams& p, int u) {
    Work w;
    w.split = u % p.n_splits;
    w.row = u / p.n_splits;
    w.b = w.row / p.T;
    w.h0 = w.split * p.halves_per_split;
    w.h1 = w.h0 + p.halves_per_split < p.halves_per_row ? w.h0 + p.halves_per_split
                                                         : p.halves_per_row;
    return w;
}

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b, float& sum) {
    const __nv_bfloat16 x = __float2bfloat16_rn(a);
    const __nv_bfloat16 y = __float2bfloat16_rn(b);
    sum += __bfloat162float(x) + __bfloat162float(y);
    return static_cast<uint32_t>(__bfloat16_as_ushort(x)) |
           (static_cast<uint32_t>(__bfloat16_as_ushort(y)) << 16);
}

__device__ __forceinline__ void load_q(const CUtensorMap* map, uint8_t* qs, int row,
                                       uint64_t* q_full) {
    tc::mbar_expect_tx(q_full, kChunks * kQChunkBytes);
    for (int c = 0; c < kChunks; ++c)
        tc::tma_load_2d(qs + c * kQChunkBytes, map, c * 64, row * kHeads, q_full);
}

__global__ void __launch_bounds__(kThreads, 1)
    tsi_attn_tc_kernel(const __grid_constant__ CUtensorMap tmap_q,
                       const __grid_constant__ AttnTcParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* qs = base;
    uint8_t* kv = qs + kChunks * kQChunkBytes;
    Smem& sm = *reinterpret_cast<Smem*>(kv + 2 * kBufBytes);
    volatile int* abort = &sm.abort;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int b = 0; b < 2; ++b) {
            tc::mbar_init(&sm.full[b], kGather);
            tc::mbar_init(&sm.empty[b], 1);
            tc::mbar_init(&sm.s_full[b], 1);
            tc::mbar_init(&sm.s_empty[b], kSoftThreads);
            tc::mbar_init(&sm.p_full[b], kSoftThreads);
        }
        tc::mbar_init(&sm.q_full, 1);
        tc::mbar_init(&sm.pv_done, 1);
        tc::mbar_init(&sm.o_full, 1);
        tc::mbar_init(&sm.o_empty, kSoftThreads);
        tc::mbar_init(&sm.done[0], 1);
        tc::mbar_init(&sm.done[1], 1);
        sm.abort = 0;
        tc::fence_barrier_init();
    }
    if (warp == kMmaWarp) {
        tc::tmem_alloc(&sm.tmem_slot, kTmemCols);
        if (lane == 0) tc::prefetch_tmap(&tmap_q);
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = sm.tmem_slot;
    const uint32_t q_addr = tc::smem_addr(qs);
    const uint32_t kv_addr = tc::smem_addr(kv);

    if (warp == kMmaWarp || warp == kPvWarp) {
        // ------------------------------------------------------------ MMA issuers
        // Two warps issue tcgen05 work: warp 4 the S products as key half-tiles land, warp 5
        // the P.V products as the softmax finishes them, so neither waits on the other's
        // inputs (each commits only its own barriers).  The whole warp runs the loop (its
        // descriptors stay warp-uniform); lane 0 issues every MMA and commit.
        const bool leader = lane == 0;
        if (warp == kMmaWarp) {
            int it = 0, un = 0;
            for (int u = blockIdx.x; u < p.n_units; u += gridDim.x, ++un) {
                const Work W = work_of(p, u);
                tc::mbar_wait(&sm.q_full, un & 1, abort, p.err);
                for (int hh = W.h0; hh < W.h1; ++hh, ++it) {
                    const int b = it & 1;
                    tc::mbar_wait(&sm.full[b], (it >> 1) & 1, abort, p.err);
                    tc::mbar_wait(&sm.s_empty[b], ((it >> 1) & 1) ^ 1, abort, p.err);
                    tc::fence_proxy_async();  // cp.async landed via the generic proxy
                    tc::tc_fence_after();
                    if (!*abort) {
                        // descriptors as base + byte offset / 16 (the start-address field
                        // holds addr / 16; shared addresses stay below 2^18, no carry)
                        const uint64_t da0 = tc::smem_desc(q_addr, 16, 1024);
                        const uint64_t db0 = tc::smem_desc(kv_addr + b * kBufBytes, 16, 1024);
#pragma unroll
                        for (int c = 0; c < kChunks; ++c) {
#pragma unroll
                            for (int kk = 0; kk < 4; ++kk)
                                if (leader)
                                    tc::mma_bf16(tmem + kColS + 64 * b,
                                                 da0 + ((c * kQChunkBytes + kk * 32) >> 4),
                                                 db0 + ((c * kChunkBytes + kk * 32) >> 4),
                                                 kIdescS, (c | kk) ? 1u : 0u);
                        }
                    }
                    if (leader) tc::mma_commit(&sm.s_full[b]);
                }
            }
            if (leader) tc::mma_commit(&sm.done[0]);
            if (!tc::mbar_wait(&sm.done[0], 0, abort, p.err))
                tc::mbar_drain(&sm.done[0], 0);  // issued MMAs finish before TMEM is freed
        } else {
            int it = 0, un = 0;
            for (int u = blockIdx.x; u < p.n_units; u += gridDim.x, ++un) {
                const Work W = work_of(p, u);
                for (int hh = W.h0; hh < W.h1; ++hh, ++it) {
                    const int b = it & 1;
                    tc::mbar_wait(&sm.p_full[b], (it >> 1) & 1, abort, p.err);
                    if (hh == W.h0) tc::mbar_wait(&sm.o_empty, (un & 1) ^ 1, abort, p.err);
                    tc::fence_proxy_async();  // P^T written with generic stores
                    tc::tc_fence_after();
                    if (!*abort) {
                        const uint32_t kb = kv_addr + b * kBufBytes;
                        const uint64_t da0 = tc::smem_desc(kb, kChunkBytes, 1024);
                        const uint64_t db0 = tc::smem_desc(kb + kPSlot * kChunkBytes, 16, 1024);
                        const uint32_t first = hh == W.h0 ? 0u : 1u;
#pragma unroll
                        for (int m = 0; m < 4; ++m) {
#pragma unroll
                            for (int kk = 0; kk < 4; ++kk)
                                if (leader)
                                    tc::mma_bf16(tmem + kColO + 64 * m,
                                                 da0 + ((2 * m * kChunkBytes + kk * 2048) >> 4),
                                                 db0 + ((kk * 32) >> 4), kIdescO,
                                                 kk == 0 ? first : 1u);
                        }
                    }
                    if (leader) tc::mma_commit(&sm.empty[b]);
                    if (leader) tc::mma_commit(&sm.pv_done);
                }
                if (leader) tc::mma_commit(&sm.o_full);
            }
            if (leader) tc::mma_commit(&sm.done[1]);
            if (!tc::mbar_wait(&sm.done[1], 0, abort, p.err))
                tc::mbar_drain(&sm.done[1], 0);  // issued MMAs finish before TMEM is freed
        }
    } else if (warp > kPvWarp) {
        // ------------------------------------------------------------ gather
        const int g = threadIdx.x - kGatherBase;
        int it = 0;
        for (int u = blockIdx.x; u < p.n_units; u += gridDim.x) {
            const Work W = work_of(p, u);
            const int64_t len = seq_len(p.kv_len, W.b, p.S);
            const int32_t* irow = p.idx + static_cast<int64_t>(W.row) * p.topk;
            const uint16_t* kseq = p.k + static_cast<int64_t>(W.b) * p.S * kDqk;
            for (int hh = W.h0; hh < W.h1; ++hh, ++it) {
                const int b = it & 1;
                const uint16_t* src[kGatherPer];
                uint32_t nbytes[kGatherPer];
                uint32_t dst[kGatherPer];
#pragma unroll
                for (int j = 0; j < kGatherPer; ++j) {
                    const int piece = g + kGather * j;
                    const int k = (piece >> 3) & (kHalf - 1);
                    const int sub = piece & 7;
                    const int e = hh * kHalf + k;
                    const int s = (piece < kPieces && e < p.topk) ? irow[e] : -1;
                    const bool ok = s >= 0 && s < len;
                    src[j] = ok ? kseq + static_cast<int64_t>(s) * kDqk + sub * 8 : kseq;
                    nbytes[j] = ok ? 16u : 0u;
                    dst[j] = kv_addr + b * kBufBytes + (k >> 3) * 1024 + (k & 7) * 128 +
                             ((sub ^ (k & 7)) << 4);
                }
                tc::mbar_wait(&sm.empty[b], ((it >> 1) & 1) ^ 1, abort, p.err);
                for (int c = 0; c < kChunks; ++c) {
#pragma unroll
                    for (int j = 0; j < kGatherPer; ++j) {
                        if (g + kGather * j < kPieces)
                            tc::cp_async16(dst[j] + c * kChunkBytes,
                                           src[j] + (nbytes[j] ? c * 64 : 0), nbytes[j]);
                    }
                }
                tc::cp_async_arrive_noinc(&sm.full[b]);
            }
        }
        asm volatile("cp.async.wait_all;" ::: "memory");
    } else {
        // ------------------------------------------------- softmax + row epilogue
        // The S buffer's 16 used lanes of this warp's quadrant are read in the 16x256b
        // shape: thread T holds heads hA = 16 q + T / 4 and hB = hA + 8, keys
        // 8 m + 2 (T % 4) + {0, 1} for m = 0..7 (registers 4m, 4m+1 for hA, 4m+2, 4m+3 for
        // hB); the four threads of a head combine maxima and sums with two shuffles.
        const int q = warp;  // TMEM lane quadrant
        const int t4 = lane & 3;
        const int hA = 16 * q + (lane >> 2);
        const int hB = hA + 8;
        const uint32_t lane_base = static_cast<uint32_t>(32 * q) << 16;
        const float neg_inf = -__int_as_float(0x7f800000);
        int it = 0, un = 0, q_issued = 0;
        if (threadIdx.x == 0 && blockIdx.x < p.n_units) {
            load_q(&tmap_q, qs, work_of(p, blockIdx.x).row, &sm.q_full);
            ++q_issued;
        }
        for (int u = blockIdx.x; u < p.n_units; u += gridDim.x, ++un) {
            const Work W = work_of(p, u);
            const int nh = W.h1 - W.h0;
            const int64_t len = seq_len(p.kv_len, W.b, p.S);
            const int32_t* irow = p.idx + static_cast<int64_t>(W.row) * p.topk;
            float mA = neg_inf, mB = neg_inf;  // running maxima (base 2, scaled)
            float lA = 0.f, lB = 0.f;  // this thread's share of the row sums
            for (int j = 0; j < nh; ++j, ++it) {
                const int b = it & 1;
                // which of the half-tile's 64 entries are keys: bit k of va / vb = entry k / 32+k
                const int e0 = (W.h0 + j) * kHalf;
                const int sa = e0 + lane < p.topk ? irow[e0 + lane] : -1;
                const int sb = e0 + 32 + lane < p.topk ? irow[e0 + 32 + lane] : -1;
                const uint32_t va = __ballot_sync(kFull, sa >= 0 && sa < len);
                const uint32_t vb = __ballot_sync(kFull, sb >= 0 && sb < len);
                uint32_t vbits = 0;  // bit 2m+e: key 8m + 2 t4 + e is a key
#pragma unroll
                for (int m = 0; m < 8; ++m) {
                    const uint32_t w = m < 4 ? va : vb;
                    vbits |= ((w >> ((8 * m + 2 * t4) & 31)) & 3u) << (2 * m);
                }
                tc::mbar_wait(&sm.s_full[b], (it >> 1) & 1, abort, p.err);
                tc::tc_fence_after();
                if (threadIdx.x == 0 && j == nh - 1 && !*abort) {
                    // every S of this unit is done: the Q buffer is free for the next unit
                    const int nu = u + gridDim.x;
                    if (nu < p.n_units) {
                        load_q(&tmap_q, qs, work_of(p, nu).row, &sm.q_full);
                        ++q_issued;
                    }
                }
                uint32_t r[32];
                TSI_TMEM_LD16x256_X8(tmem + lane_base + kColS + 64 * b, r);
                tc::tmem_wait_ld();
                tc::tc_fence_before();
                tc::mbar_arrive(&sm.s_empty[b]);
                float xa = neg_inf, xb = neg_inf;
#pragma unroll
                for (int m = 0; m < 8; ++m) {
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const float za = __uint_as_float(r[4 * m + e]) * p.scale_log2;
                        const float zb = __uint_as_float(r[4 * m + 2 + e]) * p.scale_log2;
                        r[4 * m + e] = __float_as_uint(za);
                        r[4 * m + 2 + e] = __float_as_uint(zb);
                        if ((vbits >> (2 * m + e)) & 1u) {
                            xa = fmaxf(xa, za);
                            xb = fmaxf(xb, zb);
                        }
                    }
                }
#pragma unroll
                for (int o = 1; o < 4; o <<= 1) {
                    xa = fmaxf(xa, __shfl_xor_sync(kFull, xa, o));
                    xb = fmaxf(xb, __shfl_xor_sync(kFull, xb, o));
                }
                const bool needA = xa > mA + kRescaleLog2;
                const bool needB = xb > mB + kRescaleLog2;
                const bool rescale = tc::bar_red_or(kSoftBar, kSoftThreads, needA || needB);
                float alphaA = 1.f, alphaB = 1.f;
                if (needA) {
                    alphaA = mA == neg_inf ? 0.f : ex2(mA - xa);
                    mA = xa;
                }
                if (needB) {
                    alphaB = mB == neg_inf ? 0.f : ex2(mB - xb);
                    mB = xb;
                }
                // P^T rows of heads hA, hB (K-major B operand over the RoPE chunk's slot): the
                // two keys of piece m go to bytes 4 t4 .. 4 t4 + 3 of the swizzled piece
                uint8_t* pslot = kv + b * kBufBytes + kPSlot * kChunkBytes;
                uint8_t* prowA = pslot + (hA >> 3) * 1024 + (hA & 7) * 128 + 4 * t4;
                uint8_t* prowB = pslot + (hB >> 3) * 1024 + (hB & 7) * 128 + 4 * t4;
                float sA = 0.f, sB = 0.f;
#pragma unroll
                for (int m = 0; m < 8; ++m) {
                    const bool v0 = (vbits >> (2 * m)) & 1u;
                    const bool v1 = (vbits >> (2 * m + 1)) & 1u;
                    const float a0 = v0 ? ex2(__uint_as_float(r[4 * m]) - mA) : 0.f;
                    const float a1 = v1 ? ex2(__uint_as_float(r[4 * m + 1]) - mA) : 0.f;
                    const float b0 = v0 ? ex2(__uint_as_float(r[4 * m + 2]) - mB) : 0.f;
                    const float b1 = v1 ? ex2(__uint_as_float(r[4 * m + 3]) - mB) : 0.f;
                    *reinterpret_cast<uint32_t*>(prowA + ((m ^ (hA & 7)) << 4)) =
                        pack_bf16(a0, a1, sA);
                    *reinterpret_cast<uint32_t*>(prowB + ((m ^ (hB & 7)) << 4)) =
                        pack_bf16(b0, b1, sB);
                }
                lA = lA * alphaA + sA;
                lB = lB * alphaB + sB;
                if (rescale && j > 0) {  // O^T holds this unit's earlier half-tiles: rescale it
                    if (t4 == 0) {
                        sm.alpha[hA] = alphaA;
                        sm.alpha[hB] = alphaB;
                    }
                    tc::mbar_wait(&sm.pv_done, (it - 1) & 1, abort, p.err);
                    named_bar(kSoftBar, kSoftThreads);
                    tc::tc_fence_after();
#pragma unroll 1
                    for (int m = 0; m < 4; ++m) {  // rare: one 32-column block at a time
#pragma unroll 1
                        for (int half = 0; half < 2; ++half) {
                            uint32_t o[32];
                            const uint32_t ta = tmem + lane_base + kColO + 64 * m + 32 * half;
                            TSI_TMEM_LD32(ta, o);
                            tc::tmem_wait_ld();
#pragma unroll
                            for (int i = 0; i < 32; ++i)
                                o[i] = __float_as_uint(__uint_as_float(o[i]) *
                                                       sm.alpha[32 * half + i]);
                            TSI_TMEM_ST32(ta, o);
                        }
                    }
                    tc::tmem_wait_st();
                }
                tc::fence_proxy_async();
                tc::tc_fence_before();
                tc::mbar_arrive(&sm.p_full[b]);
            }
            // ------------------------------------------------------ row epilogue
#pragma unroll
            for (int o = 1; o < 4; o <<= 1) {
                lA += __shfl_xor_sync(kFull, lA, o);
                lB += __shfl_xor_sync(kFull, lB, o);
            }
            tc::mbar_wait(&sm.o_full, un & 1, abort, p.err);
            tc::tc_fence_after();
            if (t4 == 0) {
                sm.linv[hA] = lA > 0.f ? 1.f / lA : 0.f;
                sm.linv[hB] = lB > 0.f ? 1.f / lB : 0.f;
                if (p.part_o) {
                    const int64_t slot0 =
                        (static_cast<int64_t>(W.row) * p.n_splits + W.split) * kHeads;
                    p.part_ml[2 * (slot0 + hA)] = mA;
                    p.part_ml[2 * (slot0 + hA) + 1] = lA;
                    p.part_ml[2 * (slot0 + hB)] = mB;
                    p.part_ml[2 * (slot0 + hB) + 1] = lB;
                } else if (p.lse) {
                    p.lse[static_cast<int64_t>(W.row) * kHeads + hA] = lse_of(mA, lA);
                    p.lse[static_cast<int64_t>(W.row) * kHeads + hB] = lse_of(mB, lB);
                }
            }
            named_bar(kSoftBar, kSoftThreads);
            for (int m = 0; m < 4; ++m) {
                const int d = 128 * m + 32 * q + lane;  // this thread's value dim (TMEM lane)
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    uint32_t o[32];  // O^T[d, heads 32 half .. 32 half + 31]
                    TSI_TMEM_LD32(tmem + lane_base + kColO + 64 * m + 32 * half, o);
                    tc::tmem_wait_ld();
                    if (p.part_o) {
                        float* po = p.part_o +
                                    ((static_cast<int64_t>(W.row) * p.n_splits + W.split) * kHeads +
                                     32 * half) * kDv + d;
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            po[static_cast<int64_t>(i) * kDv] = __uint_as_float(o[i]);
                    } else {
                        // the 32 factors first: read between the stores, each would wait for
                        // its shared-memory load (the stores may alias it for the compiler)
                        float li[32];
#pragma unroll
                        for (int i = 0; i < 32; i += 4) {
                            const float4 v = *reinterpret_cast<const float4*>(&sm.linv[32 * half + i]);
                            li[i] = v.x;
                            li[i + 1] = v.y;
                            li[i + 2] = v.z;
                            li[i + 3] = v.w;
                        }
                        __nv_bfloat16* out =
                            p.out + (static_cast<int64_t>(W.row) * kHeads + 32 * half) * kDv + d;
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            out[static_cast<int64_t>(i) * kDv] =
                                __float2bfloat16_rn(__uint_as_float(o[i]) * li[i]);
                    }
                }
            }
            tc::tc_fence_before();
            tc::mbar_arrive(&sm.o_empty);
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

constexpr int kPlanSMs = 152;

// Half-tiles per row, and for few rows (decode) the split of a row's half-tiles over CTAs.
void attn_tc_plan(int rows, int topk, int* n_splits, int* halves_per_split, int* halves) {
    const int nh = (topk + kHalf - 1) / kHalf;
    int ns = 1;
    if (rows > 0 && rows < kPlanSMs) {
        ns = (kPlanSMs + rows - 1) / rows;
        if (ns > nh) ns = nh;
        if (ns < 1) ns = 1;
    }
    const int hps = (nh + ns - 1) / ns;
    *halves = nh;
    *halves_per_split = hps;
    *n_splits = (nh + hps - 1) / hps;
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
    int ns, hps, nh;
    attn_tc_plan(B * T, topk, &ns, &hps, &nh);
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
    attn_tc_plan(rows, a.topk, &p.n_splits, &p.halves_per_split, &p.halves_per_row);
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
