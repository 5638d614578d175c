// Exact top-k of stored score rows: the second pass of the two-pass tensor-core indexer.
//
// The tensor-core pass writes each query row's scores I[t, s] ("GLM-5.2 技术报告速览",
// §IndexShare: the indexer score over the keys s <= p_t, then the k = 2048 best) to a
// row-major fp32 scratch buffer.  Here one block takes one row:
//   1. A row longer than the selector's buffer first reads a block sample (one group of
//      four scores in every G >= 32) and sets the admission threshold at or below the
//      sample's m-th key, m chosen so that the whole row holds, with a margin of 1.5,
//      more than k keys at or above it.
//   2. One barrier-free pass appends every key of the row at or above the threshold to
//      the shared-memory buffer (topk_select.cuh), loads four deep in flight.
//   3. If the buffer overflowed, or fewer than k keys reached a sampled threshold (the
//      sample misled), the row is streamed once more through the selector with room
//      checks, from that threshold or from 0: the result is exact in every case.
//   4. The row's k best keys are ranked in shared memory and written as idx / score (or,
//      for key shards, left unordered as 64-bit rank keys for the merge).
// Out of the tensor-core kernel, the selection no longer stalls the MMA pipeline.
#include "indexer_generic.cuh"
#include "rank_sort.cuh"
#include "topk_select.cuh"

namespace tsi {
namespace {

constexpr int kRowThreads = 256;
constexpr int kRowCap = 5120;      // keys held per row (a sampled row needs about 1.5 k)
constexpr int kPerThread = 4;      // keys a thread offers per round of the checked stream
constexpr int kRound = kPerThread * kRowThreads;
constexpr int kSampleEvery = 32;   // at least one float4 of every 32 in the sample
constexpr int kDepth = 4;          // float4 loads of the filter pass in flight per thread

static_assert(kRowCap - 2 * kRound > TSI_MAX_TOPK, "the room trigger lies above k keys");
static_assert(kRowThreads == kRankThreads && kRowCap >= 2 * kRankN,
              "the block ranks in its buffer, the second half as scratch");

using Sel = TopKSelector<kRowThreads, kRowCap>;

// The checked stream: the row's float4 pieces j = 0 .. (n + 3) / 4 - 1 (piece j at row +
// 4 j, its keys at positions pos0 + 4 j + {0..3}, keys past n excluded) are offered in
// rounds of one piece per thread, with a room check before each round; the next round's
// piece loads while the current one is offered.
__device__ __forceinline__ void stream_row(Sel& sel, const float* row, int64_t n, uint32_t pos0,
                                           int topk) {
    // The OR over the block of "held > trigger" is the same in every thread.  A thread's
    // count may miss the last round's offers of other threads, and this round adds one
    // more, so the trigger leaves two rounds of room.
    constexpr int kTrigger = kRowCap - 2 * kRound;
    const int64_t n4 = (n + 3) / 4;
    auto load = [&](int64_t j) {
        return j < n4 ? __ldcs(reinterpret_cast<const float4*>(row + 4 * j))
                      : make_float4(0.f, 0.f, 0.f, 0.f);
    };
    int64_t j = threadIdx.x;
    float4 v = load(j);
    for (int64_t base = 0; base < n4; base += kRowThreads) {
        const float4 w = load(j + kRowThreads);  // next round, in flight meanwhile
        if (__syncthreads_or(sel.count() > kTrigger)) {
            const int held = sel.settled_count();
            if (held > (topk + kTrigger) / 2) sel.compact(topk, held, false, (kTrigger - topk) / 4);
        }
        const uint64_t thr = *reinterpret_cast<volatile uint64_t*>(sel.thr);
        const float floor = score_floor(thr);
        const int64_t left = j < n4 ? n - 4 * j : 0;  // keys of the piece in the row
        const uint32_t p = pos0 + static_cast<uint32_t>(4 * j);
        sel.offer2_scored(left > 0, v.x, p, left > 1, v.y, p + 1, thr, floor);
        sel.offer2_scored(left > 2, v.z, p + 2, left > 3, v.w, p + 3, thr, floor);
        j += kRowThreads;
        v = w;
    }
}

// Appends every key of float4 pieces j = 0 .. (n + 3) / 4 - 1 (piece j read from row + 4 j
// stride4, its keys at positions pos0 + 4 j stride4 + {0..3}, keys past n excluded) that
// lies at or above `threshold`, with no room check and no barrier: the count may run past
// the buffer (the caller checks; keys whose slot lies beyond it are not stored).  Per
// iteration a thread holds kDepth pieces (the next kDepth load meanwhile), marks the keys
// that pass in a bit mask, and its warp reserves the slots of all of them with one atomic
// (offsets from a warp scan of the per-thread counts).  A key passes when its score lies
// above the threshold's score; a score equal to it (rare) is decided by the 64-bit key, in
// a branch that only warps holding such a score take.  Indices fit 32 bits: n < 2^31.
__device__ __forceinline__ void filter_row(Sel& sel, const float* row, int n, int stride4,
                                           uint32_t pos0, uint64_t threshold) {
    const float floor = score_floor(threshold);
    const int n4 = (n + 3) / 4;
    const int lane = threadIdx.x & 31;
    auto load = [&](int j) {
        return j < n4 ? __ldcs(reinterpret_cast<const float4*>(row + 4 * j * stride4))
                      : make_float4(0.f, 0.f, 0.f, 0.f);
    };
    float4 v[kDepth];
    int j = threadIdx.x;
#pragma unroll
    for (int d = 0; d < kDepth; ++d) v[d] = load(j + d * kRowThreads);
    for (int base = 0; base < n4; base += kDepth * kRowThreads) {
        float4 w[kDepth];
#pragma unroll
        for (int d = 0; d < kDepth; ++d) w[d] = load(j + (kDepth + d) * kRowThreads);
        unsigned mask = 0u, tie = 0u;  // bit 4 d + e: key e of piece d passes / ties
#pragma unroll
        for (int d = 0; d < kDepth; ++d) {
            const int jj = j + d * kRowThreads;
            const int keys = jj < n4 ? min(4, n - 4 * jj) : 0;  // keys of the piece in the row
            const float x[4] = {v[d].x, v[d].y, v[d].z, v[d].w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                mask |= static_cast<unsigned>(e < keys && x[e] > floor) << (4 * d + e);
                tie |= static_cast<unsigned>(e < keys && x[e] == floor) << (4 * d + e);
            }
        }
        if (__any_sync(kFull, tie != 0u)) {
#pragma unroll
            for (int d = 0; d < kDepth; ++d) {
                const uint32_t p = pos0 + 4u * static_cast<uint32_t>(j + d * kRowThreads) *
                                                static_cast<uint32_t>(stride4);
                const float x[4] = {v[d].x, v[d].y, v[d].z, v[d].w};
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    if (((tie >> (4 * d + e)) & 1u) && make_key(x[e], p + e) >= threshold)
                        mask |= 1u << (4 * d + e);
            }
        }
        const int c = __popc(mask);
        int incl = c;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int t = __shfl_up_sync(kFull, incl, o);
            if (lane >= o) incl += t;
        }
        const int total = __shfl_sync(kFull, incl, 31);
        if (total) {
            int at = 0;
            if (lane == 31) at = atomicAdd(&sel.ctl[0], total);
            at = __shfl_sync(kFull, at, 31) + incl - c;
#pragma unroll
            for (int d = 0; d < kDepth; ++d) {
                const uint32_t p = pos0 + 4u * static_cast<uint32_t>(j + d * kRowThreads) *
                                                static_cast<uint32_t>(stride4);
                const float x[4] = {v[d].x, v[d].y, v[d].z, v[d].w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    if ((mask >> (4 * d + e)) & 1u) {
                        if (at < kRowCap) sel.buf[at] = make_key(x[e], p + e);
                        ++at;
                    }
                }
            }
        }
        j += kDepth * kRowThreads;
#pragma unroll
        for (int d = 0; d < kDepth; ++d) v[d] = w[d];
    }
}

__global__ void __launch_bounds__(kRowThreads) topk_rows_kernel(const ScoreRows r) {
    extern __shared__ __align__(16) uint8_t smem[];
    Sel sel;
    sel.bind(smem, threadIdx.x, 1, r.err);
    const int rr = blockIdx.x;  // row of the chunk: sequence rr / rows, row t0 + rr % rows
    const int b = rr / r.rows;
    const int t = r.t0 + rr % r.rows;
    int64_t limit = query_position(r.kv_len, b, r.T, r.S_total, t) + 1 - r.key_offset;
    limit = limit < 0 ? 0 : (limit > r.S ? r.S : limit);
    const float* row = r.scores + static_cast<int64_t>(rr) * r.ld;
    const uint32_t pos0 = static_cast<uint32_t>(r.key_offset);
    sel.reset();
    uint64_t start = 0ull;  // admission threshold of the full pass
    if (limit > kRowCap) {
        // sample: the first float4 of every G (G >= 32, at most kRowCap sampled keys)
        int64_t G = (limit + kRowCap - 1) / kRowCap;
        G = G < kSampleEvery ? kSampleEvery : G;
        const int64_t whole = limit / (4 * G);  // blocks of G pieces wholly inside the row
        filter_row(sel, row, static_cast<int>(4 * whole), static_cast<int>(G), pos0, 0ull);
        // The row holds limit / (4 whole) keys per sampled key, so m sampled keys at or
        // above the threshold promise about m limit / (4 whole) row keys: m = 1.5 k 4 whole
        // / limit leaves a margin of 1.5.  A loose compaction stops at a bin edge at or
        // below the m-th sampled key.
        const int64_t m = (3 * static_cast<int64_t>(r.topk) * 4 * whole + 2 * limit - 1) /
                          (2 * limit);
        const int held = sel.settled_count();
        if (held > m) {
            // only the threshold is needed: the buffer is emptied right after
            sel.compact(static_cast<int>(m), held, false, static_cast<int>(m / 4), false);
            start = *reinterpret_cast<volatile uint64_t*>(sel.thr);
        }
        sel.restart(start);
    }
    filter_row(sel, row, static_cast<int>(limit), 1, pos0, start);
    const int held = sel.settled_count();
    if (held > kRowCap || (start != 0ull && held < r.topk)) {
        // the buffer overflowed, or the sample misled: stream the row with room checks
        sel.restart(held > kRowCap ? start : 0ull);
        stream_row(sel, row, limit, pos0, r.topk);
    }
    const int64_t slot = static_cast<int64_t>(b) * r.T + t;
    if (!r.idx) {
        sel.dump(r.topk, r.cand + slot * r.topk, r.cand_cnt + slot);
        return;
    }
    // the exact top k, then ranked by rank_merge_write (rank_sort.cuh) over the first kRankN
    // slots (empty slots hold key 0, below every real key), the next kRankN as scratch
    sel.compact(r.topk, sel.settled_count());
    const int n = sel.settled_count();
    for (int i = n + threadIdx.x; i < kRankN; i += kRowThreads) sel.buf[i] = 0ull;
    sel.sync();
    rank_merge_write(sel.buf, sel.buf + kRankN, n, r.topk, r.idx + slot * r.topk,
                     r.score ? r.score + slot * r.topk : nullptr, threadIdx.x, 1);
}

}  // namespace

size_t topk_rows_smem_bytes() {
    return (selector_smem_bytes<kRowCap>() + 15) & ~static_cast<size_t>(15);
}

cudaError_t launch_topk_rows(const ScoreRows& r, cudaStream_t st) {
    const int blocks = r.B * r.rows;
    if (blocks == 0) return cudaSuccess;
    const int smem = static_cast<int>(topk_rows_smem_bytes());
    cudaError_t e = cudaFuncSetAttribute(topk_rows_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    topk_rows_kernel<<<blocks, kRowThreads, smem, st>>>(r);
    note_launches(1);
    return cudaGetLastError();
}

}  // namespace tsi
