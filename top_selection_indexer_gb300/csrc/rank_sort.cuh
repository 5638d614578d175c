// Rank-ordering of one row's top-k keys held in shared memory: per-warp bitonic sorts in
// registers, then merges along the merge path (used by the ranking and merge kernels of
// indexer_generic.cu and by the row selection of topk_rows.cu).
#pragma once

#include "topk_select.cuh"

namespace tsi {

constexpr int kRankThreads = 256;
constexpr int kRankPer = 8;  // keys per thread, consecutive ranks
constexpr int kRankN = kRankThreads * kRankPer;
static_assert(kRankN >= TSI_MAX_TOPK, "one block ranks a whole row");

// Compare-exchange of a bitonic network: afterwards a >= b when `desc`, else a <= b.
__device__ __forceinline__ void rank_cas(uint64_t& a, uint64_t& b, bool desc) {
    const bool swap = desc ? (a < b) : (a > b);
    const uint64_t lo = swap ? b : a;
    const uint64_t hi = swap ? a : b;
    a = lo;
    b = hi;
}

// Bitonic stage at distance D < kRankPer inside one thread's slots 8t .. 8t+7.
template <int D>
__device__ __forceinline__ void in_thread_stage(uint64_t (&x)[kRankPer], int t, int size) {
#pragma unroll
    for (int j = 0; j < kRankPer; ++j)
        if ((j & D) == 0) rank_cas(x[j], x[j | D], ((kRankPer * t + j) & size) == 0);
}

// Rank n <= topk distinct keys held in xs[0 .. kRankN) (empty slots hold key 0, below
// every real key) and write idx / score rows in rank order, -1 / -inf after the n-th.
// Each warp sorts its 256 slots (thread t holds slots 8t .. 8t+7) in registers with a
// bitonic network (exchanges inside the thread or by warp shuffles, no block barrier),
// then three merge levels in shared memory join the eight sorted runs (256 -> 512 ->
// 1024 -> 2048).  At a merge level thread t produces outputs 8t .. 8t+7 of the merged
// array: a binary search along the merge path finds how many of the first 8t outputs come
// from the first run, then it merges 8 keys.  Keys are distinct
// (or 0, the empty slots, which sort last), so the path is unique.  xs2 is scratch of
// kRankN keys; threads t = 0 .. 255 take part (barrier `bar`).
static __device__ void rank_merge_write(uint64_t* xs, uint64_t* xs2, int n, int topk, int32_t* io,
                                        float* so, int t, int bar) {
    const int lane = t & 31;
    uint64_t x[kRankPer];
#pragma unroll
    for (int j = 0; j < kRankPer; ++j) x[j] = xs[kRankPer * t + j];
    // 1. one sorted (descending) run of 256 keys per warp: slot 8 lane + j of the warp
    for (int size = 2; size <= 32 * kRankPer; size <<= 1) {
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            if (stride < kRankPer) {
                if (stride == 4)
                    in_thread_stage<4>(x, lane, size);
                else if (stride == 2)
                    in_thread_stage<2>(x, lane, size);
                else
                    in_thread_stage<1>(x, lane, size);
            } else {
                const int lm = stride / kRankPer;  // partner lane distance
                const bool upper = (lane & lm) != 0;
                const bool desc = ((kRankPer * lane) & size) == 0;
                const bool keep_max = desc != upper;
#pragma unroll
                for (int j = 0; j < kRankPer; ++j) {
                    const uint64_t y = __shfl_xor_sync(0xFFFFFFFFu, x[j], lm);
                    x[j] = keep_max ? (x[j] > y ? x[j] : y) : (x[j] < y ? x[j] : y);
                }
            }
        }
    }
    named_bar(bar, kRankThreads);  // every thread has read its slots
#pragma unroll
    for (int j = 0; j < kRankPer; ++j) xs[kRankPer * t + j] = x[j];
    named_bar(bar, kRankThreads);
    // 2. merge pairs of runs of length L into runs of 2 L
    uint64_t* src = xs;
    uint64_t* dst = xs2;
    for (int L = 32 * kRankPer; L < kRankN; L <<= 1) {
        const int d0 = kRankPer * t;
        const int d = d0 % (2 * L);  // output index inside this merge
        const uint64_t* A = src + (d0 - d);
        const uint64_t* B = A + L;
        int lo = d > L ? d - L : 0;
        int hi = d < L ? d : L;
        while (lo < hi) {  // how many of the first d outputs come from A
            const int mid = (lo + hi) >> 1;
            if (A[mid] > B[d - 1 - mid])
                lo = mid + 1;
            else
                hi = mid;
        }
        int i = lo, k = d - lo;
        const bool last = 2 * L == kRankN;
#pragma unroll
        for (int j = 0; j < kRankPer; ++j) {
            const bool from_a = k >= L || (i < L && A[i] > B[k]);
            const uint64_t v = from_a ? A[i] : B[k];
            i += from_a ? 1 : 0;
            k += from_a ? 0 : 1;
            if (last) {
                const int r = d0 + j;
                if (r < topk) {
                    const bool real = r < n;
                    io[r] = real ? key_position(v) : -1;
                    if (so) so[r] = real ? key_score(v) : -__int_as_float(0x7f800000);
                }
            } else {
                dst[d0 + j] = v;
            }
        }
        named_bar(bar, kRankThreads);
        uint64_t* tmp = src;
        src = dst;
        dst = tmp;
    }
}

}  // namespace tsi
