// Cross-layer top-k overlap: |S_a ∩ S_b| per query row for two index buffers.
//
// The observation behind IndexShare is that the top-k sets chosen by neighbouring
// layers' indexers largely coincide ("GLM-5.2 技术报告速览", §IndexShare: pairwise overlap
// of the per-layer top-k indices, 0.7-1.0 between adjacent layers).  This kernel measures
// it: for every row, the number of positions the two rows have in common and the number
// of positions of row a (entries < 0 are padding, not positions).
//
// One block per row.  Row b's positions go into an open-addressing hash table of
// 2 * TSI_MAX_TOPK slots in shared memory (load factor <= 1/2, linear probing, inserts by
// atomicCAS); row a's positions are then looked up.  The positions of one row are
// distinct, as top-k rows are.
#include "overlap.cuh"
#include "tsi_common.cuh"

namespace tsi {
namespace {

constexpr int kOvThreads = 256;
constexpr int kSlots = 2 * TSI_MAX_TOPK;  // power of two
constexpr int kEmpty = -1;

__device__ __forceinline__ uint32_t slot_of(int32_t pos) {
    return (static_cast<uint32_t>(pos) * 2654435761u) >> (32 - 12);  // 12 bits: kSlots = 4096
}
static_assert(kSlots == 4096, "slot_of takes the top 12 bits of the product");

constexpr int kPer = TSI_MAX_TOPK / kOvThreads;  // positions per thread and row

__global__ void __launch_bounds__(kOvThreads) topk_overlap_kernel(const int32_t* idx_a,
                                                                   const int32_t* idx_b,
                                                                   int topk, int32_t* inter,
                                                                   int32_t* card_a,
                                                                   unsigned* err) {
    __shared__ int32_t table[kSlots];
    __shared__ int counts[2];
    const int row = blockIdx.x;
    const int32_t* a = idx_a + static_cast<int64_t>(row) * topk;
    const int32_t* b = idx_b + static_cast<int64_t>(row) * topk;
    // both rows' entries of this thread first, so that their load latencies overlap
    int32_t pa[kPer], pb[kPer];
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
        const int i = threadIdx.x + j * kOvThreads;
        pa[j] = i < topk ? a[i] : kEmpty;
        pb[j] = i < topk ? b[i] : kEmpty;
    }
    for (int i = threadIdx.x; i < kSlots; i += kOvThreads) table[i] = kEmpty;
    if (threadIdx.x < 2) counts[threadIdx.x] = 0;
    __syncthreads();
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
        const int32_t pos = pb[j];
        if (pos < 0) continue;
        uint32_t h = slot_of(pos);
        for (int probe = 0; probe < kSlots; ++probe, h = (h + 1) & (kSlots - 1)) {
            const int32_t old = atomicCAS(&table[h], kEmpty, pos);
            if (old == kEmpty || old == pos) break;  // inserted (or already there)
        }
    }
    __syncthreads();
    int hit = 0, mine = 0;
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
        const int32_t pos = pa[j];
        if (pos < 0) continue;
        ++mine;
        uint32_t h = slot_of(pos);
        for (int probe = 0; probe < kSlots; ++probe, h = (h + 1) & (kSlots - 1)) {
            const int32_t v = table[h];
            if (v == pos) {
                ++hit;
                break;
            }
            if (v == kEmpty) break;
        }
    }
    // block sums: warp shuffles, then one shared atomic per warp
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        hit += __shfl_xor_sync(0xFFFFFFFFu, hit, o);
        mine += __shfl_xor_sync(0xFFFFFFFFu, mine, o);
    }
    if ((threadIdx.x & 31) == 0) {
        atomicAdd(&counts[0], hit);
        atomicAdd(&counts[1], mine);
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        if (counts[0] > counts[1]) atomicOr(err, kErrAssert);  // a repeated position in a row
        inter[row] = counts[0];
        card_a[row] = counts[1];
    }
}

}  // namespace

cudaError_t launch_topk_overlap(const int32_t* idx_a, const int32_t* idx_b, int rows, int topk,
                                int32_t* inter, int32_t* card_a, unsigned* err,
                                cudaStream_t st) {
    if (rows == 0) return cudaSuccess;
    topk_overlap_kernel<<<rows, kOvThreads, 0, st>>>(idx_a, idx_b, topk, inter, card_a, err);
    note_launches(1);
    return cudaGetLastError();
}

}  // namespace tsi
