// Rank-ordering of one row's top-k keys held in shared memory: a bitonic sorting network
// with the keys in registers (used by the ranking kernels of indexer_generic.cu and by the
// row selection of topk_rows.cu).
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
// every real key) and write idx / score rows in rank order, -1 / -inf after the n-th.  A
// bitonic sorting network over the 2048 slots sorts descending; threads t = 0 .. 255 of
// the block take part (their only barrier is named barrier `bar`).  Thread t holds slots
// 8t .. 8t+7 in registers: exchanges at distance < 8 stay in the thread, distances 8..255
// go through warp shuffles, and only the six stages at distance >= 256 go through shared
// memory.
static __device__ void rank_sort_write(uint64_t* xs, int n, int topk, int32_t* io, float* so,
                                       int t, int bar) {
    uint64_t x[kRankPer];
#pragma unroll
    for (int j = 0; j < kRankPer; ++j) x[j] = xs[kRankPer * t + j];

    for (int size = 2; size <= kRankN; size <<= 1) {
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            if (stride < kRankPer) {
                // compile-time distances keep x[] in registers
                if (stride == 4)
                    in_thread_stage<4>(x, t, size);
                else if (stride == 2)
                    in_thread_stage<2>(x, t, size);
                else
                    in_thread_stage<1>(x, t, size);
            } else if (stride < 32 * kRankPer) {
                const int lm = stride / kRankPer;  // partner lane distance
                const bool upper = (t & lm) != 0;
                const bool desc = ((kRankPer * t) & size) == 0;
                const bool keep_max = desc != upper;
#pragma unroll
                for (int j = 0; j < kRankPer; ++j) {
                    const uint64_t y = __shfl_xor_sync(0xFFFFFFFFu, x[j], lm);
                    x[j] = keep_max ? (x[j] > y ? x[j] : y) : (x[j] < y ? x[j] : y);
                }
            } else {
                const int tm = stride / kRankPer;  // partner thread distance
                const bool upper = (t & tm) != 0;
                const bool desc = ((kRankPer * t) & size) == 0;
                const bool keep_max = desc != upper;
                named_bar(bar, kRankThreads);  // the previous exchange has been read
#pragma unroll
                for (int j = 0; j < kRankPer; ++j) xs[kRankPer * t + j] = x[j];
                named_bar(bar, kRankThreads);
#pragma unroll
                for (int j = 0; j < kRankPer; ++j) {
                    const uint64_t y = xs[kRankPer * (t ^ tm) + j];
                    x[j] = keep_max ? (x[j] > y ? x[j] : y) : (x[j] < y ? x[j] : y);
                }
            }
        }
    }
#pragma unroll
    for (int j = 0; j < kRankPer; ++j) {
        const int r = kRankPer * t + j;
        if (r < topk) {
            const bool real = r < n;
            io[r] = real ? key_position(x[j]) : -1;
            if (so) so[r] = real ? key_score(x[j]) : -__int_as_float(0x7f800000);
        }
    }
}

}  // namespace tsi
