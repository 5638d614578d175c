// Lightning-indexer score + streaming top-k on CUDA cores (any dtype / head shape).
//
// I[t,s] = sum_j w[t,j] * ReLU(qI[t,j] . kI[s]) for s <= p_t ("GLM-5.2 技术报告速览",
// §IndexShare), accumulated in fp32, selected by the shared-memory TopKSelector.
// This path serves the shapes the tensor-core kernel does not (fp32 inputs, H_I != 64,
// d_I != 128).  One thread block scores one query row over one key range; when rows are
// few (decode) the keys are split across blocks and a merge kernel selects the final
// top-k from the per-split candidate lists.
#include "indexer_generic.cuh"
#include "topk_select.cuh"

namespace tsi {
namespace {

constexpr int kNT = 256;
constexpr int kCAP = 4096;
constexpr int kTK = 64;  // keys per tile
constexpr int kParts = kNT / kTK;  // threads per key

__global__ void __launch_bounds__(kNT) indexer_generic_kernel(IndexerArgs a, int n_splits,
                                                              int chunk, uint64_t* cand,
                                                              int* cand_cnt) {
    extern __shared__ __align__(16) uint8_t smem[];
    TopKSelector<kNT, kCAP> sel;
    int off = sel.bind(smem, threadIdx.x, 0, a.err);
    off = (off + 15) & ~15;
    const int dq = a.d_I + 1;  // padded row stride (bank spread)
    float* q_s = reinterpret_cast<float*>(smem + off);
    float* w_s = q_s + a.H_I * dq;
    float* k_s = w_s + ((a.H_I + 3) & ~3);

    const int row = blockIdx.x;
    const int split = blockIdx.y;
    const int b = row / a.T;
    const int t = row % a.T;
    const int64_t p = query_position(a.kv_len, b, a.T, a.S, t);
    const int64_t n_keys = p + 1 > 0 ? p + 1 : 0;
    const int64_t key_lo = static_cast<int64_t>(split) * chunk;
    const int64_t key_hi = key_lo + chunk < n_keys ? key_lo + chunk : n_keys;

    const int64_t qbase = static_cast<int64_t>(row) * a.H_I * a.d_I;
    for (int i = threadIdx.x; i < a.H_I * a.d_I; i += kNT)
        q_s[(i / a.d_I) * dq + (i % a.d_I)] = load_elem(a.qI, qbase + i, a.qk_dtype);
    for (int i = threadIdx.x; i < a.H_I; i += kNT)
        w_s[i] = load_elem(a.w, static_cast<int64_t>(row) * a.H_I + i, a.w_dtype);
    sel.reset();

    const int kk = threadIdx.x / kParts;  // key within tile
    const int part = threadIdx.x % kParts;  // head subset
    const int64_t kseq = static_cast<int64_t>(b) * a.S * a.d_I;
    for (int64_t tile = key_lo; tile < key_hi; tile += kTK) {
        const int nt = static_cast<int>(key_hi - tile < kTK ? key_hi - tile : kTK);
        for (int i = threadIdx.x; i < nt * a.d_I; i += kNT)
            k_s[(i / a.d_I) * dq + (i % a.d_I)] =
                load_elem(a.kI, kseq + (tile + i / a.d_I) * a.d_I + (i % a.d_I), a.qk_dtype);
        __syncthreads();
        float acc = 0.f;
        if (kk < nt) {
            const float* kr = k_s + kk * dq;
            for (int j = part; j < a.H_I; j += kParts) {
                const float* qr = q_s + j * dq;
                float dot = 0.f;
                for (int d = 0; d < a.d_I; ++d) dot = fmaf(qr[d], kr[d], dot);
                acc = fmaf(w_s[j], fmaxf(dot, 0.f), acc);
            }
        }
        acc += __shfl_xor_sync(kFull, acc, 1);
        acc += __shfl_xor_sync(kFull, acc, 2);
        sel.make_room(a.topk);
        sel.offer(kk < nt && part == 0, make_key(acc, static_cast<uint32_t>(tile + kk)));
        __syncthreads();
    }
    if (n_splits == 1) {
        sel.finalize(a.topk, a.idx + static_cast<int64_t>(row) * a.topk,
                     a.score ? a.score + static_cast<int64_t>(row) * a.topk : nullptr);
    } else {
        const int64_t slot = static_cast<int64_t>(row) * n_splits + split;
        sel.dump(a.topk, cand + slot * a.topk, cand_cnt + slot);
    }
}

__global__ void __launch_bounds__(kNT) topk_merge_kernel(int topk, int n_splits,
                                                         const uint64_t* cand,
                                                         const int* cand_cnt, int32_t* idx,
                                                         float* score, unsigned* err) {
    extern __shared__ __align__(16) uint8_t smem[];
    TopKSelector<kNT, kCAP> sel;
    sel.bind(smem, threadIdx.x, 0, err);
    sel.reset();
    const int row = blockIdx.x;
    for (int sp = 0; sp < n_splits; ++sp) {
        const int64_t slot = static_cast<int64_t>(row) * n_splits + sp;
        const int cnt = cand_cnt[slot];
        const uint64_t* c = cand + slot * topk;
        for (int base = 0; base < cnt; base += kNT) {
            sel.make_room(topk);
            const int i = base + threadIdx.x;
            sel.offer(i < cnt, i < cnt ? c[i] : 0ull);
        }
    }
    sel.finalize(topk, idx + static_cast<int64_t>(row) * topk,
                 score ? score + static_cast<int64_t>(row) * topk : nullptr);
}

int generic_smem_bytes(int H_I, int d_I) {
    int off = (selector_smem_bytes<kCAP>() + 15) & ~15;
    return off + (H_I * (d_I + 1) + ((H_I + 3) & ~3) + kTK * (d_I + 1)) * 4;
}

}  // namespace

void generic_split_plan(int rows, int S, int* n_splits, int* chunk) {
    int ns = 1;
    if (rows > 0 && rows < 2 * 152 && S > 8192) {
        const int by_keys = (S + 4095) / 4096;
        const int by_occupancy = (4 * 152 + rows - 1) / rows;
        ns = by_keys < by_occupancy ? by_keys : by_occupancy;
        if (ns < 1) ns = 1;
    }
    int ch = (S + ns - 1) / ns;
    ch = (ch + kTK - 1) / kTK * kTK;
    if (ch < kTK) ch = kTK;
    *n_splits = ns;
    *chunk = ch;
}

size_t generic_workspace_bytes(int B, int T, int S, int topk) {
    int ns, ch;
    const int rows = B * T;
    generic_split_plan(rows, S, &ns, &ch);
    if (ns <= 1) return 0;
    const size_t slots = static_cast<size_t>(rows) * ns;
    return slots * topk * sizeof(uint64_t) + ((slots * sizeof(int) + 255) & ~size_t(255));
}

bool generic_supported(int H_I, int d_I) {
    return H_I >= 1 && d_I >= 1 && d_I <= 256 && H_I <= 128 && H_I * d_I <= 8192;
}

cudaError_t launch_indexer_generic(const IndexerArgs& a, void* workspace, cudaStream_t st) {
    const int rows = a.B * a.T;
    int ns, ch;
    generic_split_plan(rows, a.S, &ns, &ch);
    const int smem = generic_smem_bytes(a.H_I, a.d_I);
    cudaError_t e = cudaFuncSetAttribute(indexer_generic_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    uint64_t* cand = nullptr;
    int* cnt = nullptr;
    if (ns > 1) {
        cand = static_cast<uint64_t*>(workspace);
        cnt = reinterpret_cast<int*>(cand + static_cast<size_t>(rows) * ns * a.topk);
    }
    indexer_generic_kernel<<<dim3(rows, ns), kNT, smem, st>>>(a, ns, ch, cand, cnt);
    note_launches(1);
    e = cudaGetLastError();
    if (e != cudaSuccess || ns == 1) return e;
    const int msmem = selector_smem_bytes<kCAP>();
    e = cudaFuncSetAttribute(topk_merge_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             msmem);
    if (e != cudaSuccess) return e;
    topk_merge_kernel<<<rows, kNT, msmem, st>>>(a.topk, ns, cand, cnt, a.idx, a.score, a.err);
    note_launches(1);
    return cudaGetLastError();
}

}  // namespace tsi

namespace tsi {
namespace {

// ------------------------------------------------------------------------- ranking

constexpr int kRankThreads = 256;
constexpr int kRankPer = 8;  // keys per thread, consecutive ranks
constexpr int kRankN = kRankThreads * kRankPer;
static_assert(kRankN >= TSI_MAX_TOPK, "one block ranks a whole row");

// Compare-exchange of a bitonic network: afterwards a >= b when `desc`, else a <= b.
__device__ __forceinline__ void cas(uint64_t& a, uint64_t& b, bool desc) {
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
        if ((j & D) == 0) cas(x[j], x[j | D], ((kRankPer * t + j) & size) == 0);
}

// One block per row: the row's n <= topk distinct keys (unordered) become idx / score in
// rank order, -1 / -inf after the n-th.  A bitonic sorting network over 2048 slots
// (empty slots hold key 0, below every real key) sorts descending.  Thread t holds slots
// 8t .. 8t+7 in registers: exchanges at distance < 8 stay in the thread, distances 8..255
// go through warp shuffles, and only the six stages at distance >= 256 go through shared
// memory.
__global__ void __launch_bounds__(kRankThreads) topk_rank_kernel(int topk, const uint64_t* cand,
                                                                  const int* cand_cnt,
                                                                  int32_t* idx, float* score,
                                                                  unsigned* err) {
    __shared__ __align__(16) uint64_t xs[kRankN];
    const int row = blockIdx.x;
    const int t = threadIdx.x;
    int n = cand_cnt[row];
    if (n < 0 || n > topk) {
        if (t == 0) atomicOr(err, kErrAssert);
        n = n < 0 ? 0 : topk;
    }
    const uint64_t* c = cand + static_cast<int64_t>(row) * topk;
    for (int i = t; i < kRankN; i += kRankThreads) xs[i] = i < n ? c[i] : 0ull;
    __syncthreads();
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
                __syncthreads();  // the previous exchange has been read
#pragma unroll
                for (int j = 0; j < kRankPer; ++j) xs[kRankPer * t + j] = x[j];
                __syncthreads();
#pragma unroll
                for (int j = 0; j < kRankPer; ++j) {
                    const uint64_t y = xs[kRankPer * (t ^ tm) + j];
                    x[j] = keep_max ? (x[j] > y ? x[j] : y) : (x[j] < y ? x[j] : y);
                }
            }
        }
    }
    int32_t* io = idx + static_cast<int64_t>(row) * topk;
    float* so = score ? score + static_cast<int64_t>(row) * topk : nullptr;
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

}  // namespace

cudaError_t launch_topk_rank(int rows, int topk, const uint64_t* cand, const int* cand_cnt,
                             int32_t* idx, float* score, unsigned* err, cudaStream_t st) {
    if (rows == 0) return cudaSuccess;
    topk_rank_kernel<<<rows, kRankThreads, 0, st>>>(topk, cand, cand_cnt, idx, score, err);
    note_launches(1);
    return cudaGetLastError();
}

cudaError_t launch_topk_merge(int rows, int topk, int n_splits, const uint64_t* cand,
                              const int* cand_cnt, int32_t* idx, float* score, unsigned* err,
                              cudaStream_t st) {
    const int msmem = selector_smem_bytes<kCAP>();
    cudaError_t e = cudaFuncSetAttribute(topk_merge_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, msmem);
    if (e != cudaSuccess) return e;
    topk_merge_kernel<<<rows, kNT, msmem, st>>>(topk, n_splits, cand, cand_cnt, idx, score, err);
    note_launches(1);
    return cudaGetLastError();
}

}  // namespace tsi
