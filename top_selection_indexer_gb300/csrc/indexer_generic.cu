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
