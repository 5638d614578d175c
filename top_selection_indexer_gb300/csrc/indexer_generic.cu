// Lightning-indexer score + streaming top-k on CUDA cores (any dtype / head shape).
//
// I[t,s] = sum_j w[t,j] * ReLU(qI[t,j] . kI[s]) for s <= p_t ("GLM-5.2 技术报告速览",
// §IndexShare), accumulated in fp32, selected by the shared-memory TopKSelector.
// This path serves the shapes the tensor-core kernel does not (fp32 inputs, H_I != 64,
// d_I != 128).  One thread block scores one query row over one key range; when rows are
// few (decode) the keys are split across blocks and a merge kernel selects the final
// top-k from the per-split candidate lists.
#include "indexer_generic.cuh"
#include "rank_sort.cuh"
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
    // position relative to the first key of this call: keys 0 .. p of kI are causal
    const int64_t p = query_position(a.kv_len, b, a.T, a.S_total, t) - a.key_offset;
    int64_t n_keys = p + 1 > 0 ? p + 1 : 0;
    if (n_keys > a.S) n_keys = a.S;
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
        sel.offer(kk < nt && part == 0,
                  make_key(acc, static_cast<uint32_t>(tile + kk + a.key_offset)));
        __syncthreads();
    }
    if (n_splits == 1 && !cand) {
        sel.finalize(a.topk, a.idx + static_cast<int64_t>(row) * a.topk,
                     a.score ? a.score + static_cast<int64_t>(row) * a.topk : nullptr);
    } else {
        const int64_t slot = static_cast<int64_t>(row) * n_splits + split;
        sel.dump(a.topk, cand + slot * a.topk, cand_cnt + slot);
    }
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

cudaError_t launch_indexer_generic(const IndexerArgs& args, void* workspace, cudaStream_t st) {
    IndexerArgs a = args;
    if (a.S_total == 0) a.S_total = a.S;
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
    } else if (a.out_cand) {  // one list per row: the candidates are the output
        cand = a.out_cand;
        cnt = a.out_cnt;
    }
    indexer_generic_kernel<<<dim3(rows, ns), kNT, smem, st>>>(a, ns, ch, cand, cnt);
    note_launches(1);
    e = cudaGetLastError();
    if (e != cudaSuccess || ns == 1) return e;
    return launch_topk_merge_strided(rows, a.topk, ns, cand, static_cast<int64_t>(ns) * a.topk,
                                     a.topk, cnt, ns, 1, a.idx, a.score, a.out_cand, a.out_cnt,
                                     a.err, st);
}

}  // namespace tsi

namespace tsi {
namespace {

// ------------------------------------------------------------------------- ranking

// One block per row: the row's n distinct keys (unordered, n <= the list's stride) become
// its min(n, topk) best as idx / score in rank order.
//
// Bucket rank.  The keys of a row lie in [kmin, kmax]; (key - kmin) >> shift, with the
// shift that maps kmax - kmin below 2^kRankBucketBits, splits them into 2048 buckets of
// equal width whose order is the key order (buckets aligned to the key range, not to bit
// boundaries: a range that crosses a power of two in score is not coarsened).  A histogram
// and an exclusive scan (largest bucket first) give each bucket its first rank.  A bucket whose
// first rank is k or more holds no key of the result and is skipped; the keys of the
// others are scattered into their buckets, and each key's rank is its bucket's first rank
// plus the number of larger keys in its bucket.  The ranking walks the scattered keys in
// bucket order, so the threads of a warp mostly count within one bucket: equal loop lengths,
// broadcast reads.  Rank keys are distinct, so the ranks are a permutation.  A row with more than kRankBucketMax keys in one of the buckets it keeps
// (many equal scores, or keys crowded below an outlier) takes the general path instead: an
// exact MSD radix select of its k best (when it holds more than k), then the bitonic sorts
// and merges of rank_merge_write, so the work per key stays bounded.
constexpr int kRankBucketBits = 11;
constexpr int kRankBuckets = 1 << kRankBucketBits;
constexpr int kRankBucketMax = 32;
constexpr int kRankListIn = 24;  // list slots per thread of the wide form: 6144 keys a row

// NT threads a block (256, or 1024 for few rows: shorter latency per row); IN list slots per
// thread: a list holds at most IN * NT keys.
template <int NT, int IN>
__global__ void __launch_bounds__(NT, NT > NT ? 1 : IN <= 17 ? 4 : 3)
    topk_rank_kernel(int topk, int stride, const uint64_t* cand, const int* cand_cnt,
                     int32_t* idx, float* score, unsigned* err) {
    // xs: the kept buckets' keys (at most k - 1 + kRankBucketMax), then the ranked keys; the
    // general path uses the first 2 kRankN as keys and ranking scratch.  cnt: keys per
    // bucket, then the bucket's first rank.  fill: scatter cursors; the radix select's
    // histogram.  (kRankSmemBytes of dynamic shared memory.)
    extern __shared__ __align__(16) uint64_t rank_smem[];
    uint64_t* xs = rank_smem;
    unsigned* cnt = reinterpret_cast<unsigned*>(rank_smem + 2 * kRankN + kRankBucketMax);
    unsigned* fill = cnt + kRankBuckets;
    __shared__ unsigned long long rng[2];
    constexpr int kScanPer = kRankBuckets / NT;  // buckets per thread in the scan
    static_assert(kScanPer * NT == kRankBuckets, "scan layout");
    __shared__ unsigned wsum[NT / 32];
    // big bucket, keys in the kept buckets; radix select: bin, keys above it, keys in it
    __shared__ int ctl[4];
    const int row = blockIdx.x;
    const int t = threadIdx.x;
    const int lane = t & 31, wid = t >> 5;
    int n = cand_cnt[row];
    if (n < 0 || n > stride || n > IN * NT) {
        if (t == 0) atomicOr(err, kErrAssert);
        n = n < 0 ? 0 : (stride < IN * NT ? stride : IN * NT);
    }
    const int n_out = n < topk ? n : topk;
    const uint64_t* c = cand + static_cast<int64_t>(row) * stride;
    int32_t* io = idx + static_cast<int64_t>(row) * topk;
    float* so = score ? score + static_cast<int64_t>(row) * topk : nullptr;
    // this thread's keys: slots t + 256 j (0 past the n-th: below every real key)
    uint64_t x[IN];
    uint64_t hi = 0ull, lo = ~0ull;
#pragma unroll
    for (int j = 0; j < IN; ++j) {
        const int i = t + NT * j;
        x[j] = i < n ? c[i] : 0ull;
        if (i < n) {
            hi = x[j] > hi ? x[j] : hi;
            lo = x[j] < lo ? x[j] : lo;
        }
    }
    for (int i = t; i < kRankBuckets; i += NT) {
        cnt[i] = 0u;
        fill[i] = 0u;
    }
    if (t == 0) {
        rng[0] = 0ull;
        rng[1] = ~0ull;
        ctl[0] = 0;
        ctl[1] = n;  // every bucket is kept when the row holds at most k keys
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const uint64_t h2 = __shfl_xor_sync(kFull, hi, o);
        const uint64_t l2 = __shfl_xor_sync(kFull, lo, o);
        hi = h2 > hi ? h2 : hi;
        lo = l2 < lo ? l2 : lo;
    }
    __syncthreads();
    if (lane == 0 && n > 0) {
        atomicMax(&rng[0], static_cast<unsigned long long>(hi));
        atomicMin(&rng[1], static_cast<unsigned long long>(lo));
    }
    __syncthreads();
    hi = rng[0];
    lo = n > 0 ? rng[1] : hi;
    // bucket b of key v: (v - kmin) >> shift, largest first
    const uint64_t width = hi - lo;
    const int wbits = width ? 64 - __clzll(static_cast<long long>(width)) : 0;
    const int shift = wbits > kRankBucketBits ? wbits - kRankBucketBits : 0;
    auto bucket = [&](uint64_t v) {
        return static_cast<unsigned>(kRankBuckets - 1) - static_cast<unsigned>((v - lo) >> shift);
    };
#pragma unroll
    for (int j = 0; j < IN; ++j)
        if (t + NT * j < n) atomicAdd(&cnt[bucket(x[j])], 1u);
    __syncthreads();
    // exclusive scan of the counts: thread t owns buckets kScanPer t .. + kScanPer - 1
    unsigned v[kScanPer];
    unsigned own = 0u;
#pragma unroll
    for (int j = 0; j < kScanPer; ++j) {
        v[j] = cnt[kScanPer * t + j];
        own += v[j];
    }
    unsigned incl = own;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const unsigned y = __shfl_up_sync(kFull, incl, o);
        if (lane >= o) incl += y;
    }
    if (lane == 31) wsum[wid] = incl;
    __syncthreads();
    unsigned base = 0u;
    for (int w = 0; w < wid; ++w) base += wsum[w];
    {
        unsigned run = base + incl - own;
        bool big = false;
#pragma unroll
        for (int j = 0; j < kScanPer; ++j) {
            cnt[kScanPer * t + j] = run;  // first rank of the bucket
            // a kept bucket (first rank below k) must be small enough to count in
            big |= run < static_cast<unsigned>(topk) && v[j] > static_cast<unsigned>(kRankBucketMax);
            // the bucket holding rank k - 1 ends the kept buckets' keys
            if (run < static_cast<unsigned>(topk) && run + v[j] >= static_cast<unsigned>(topk))
                ctl[1] = static_cast<int>(run + v[j]);
            run += v[j];
        }
        if (big) ctl[0] = 1;
    }
    __syncthreads();
    if (ctl[0] == 0) {
        // scatter the kept buckets' keys into bucket order
#pragma unroll
        for (int j = 0; j < IN; ++j) {
            if (t + NT * j < n) {
                const unsigned b = bucket(x[j]);
                const unsigned first = cnt[b];
                if (first < static_cast<unsigned>(topk)) xs[first + atomicAdd(&fill[b], 1u)] = x[j];
            }
        }
        __syncthreads();
        // rank = first rank of the bucket + larger keys in the bucket, for the kept buckets'
        // keys xs[0, kept) in bucket order; the result goes to the second part of xs, then
        // out in rank order (consecutive threads, consecutive ranks)
        uint64_t* ranked = xs + kRankN + kRankBucketMax;
        const int kept = ctl[1];
        for (int i = t; i < kept; i += NT) {
            const uint64_t y = xs[i];
            const unsigned b = bucket(y);
            const unsigned first = cnt[b];
            const unsigned m = fill[b];
            unsigned r = first;
            for (unsigned q = first; q < first + m; ++q) r += xs[q] > y ? 1u : 0u;
            if (r < static_cast<unsigned>(topk)) ranked[r] = y;
        }
        __syncthreads();
        constexpr int kW = 4;  // ranks read ahead of the stores
        for (int r0 = t; r0 < topk; r0 += kW * NT) {
            uint64_t y[kW];
#pragma unroll
            for (int j = 0; j < kW; ++j) {
                const int r = r0 + j * NT;
                y[j] = r < n_out ? ranked[r] : 0ull;
            }
#pragma unroll
            for (int j = 0; j < kW; ++j) {
                const int r = r0 + j * NT;
                if (r < topk) {
                    const bool real = r < n_out;
                    io[r] = real ? key_position(y[j]) : -1;
                    if (so) so[r] = real ? key_score(y[j]) : -__int_as_float(0x7f800000);
                }
            }
        }
        return;
    }
    // General path.  More than k keys: an exact MSD radix select finds the k-th largest
    // key (the bits above the highest bit in which the smallest and largest keys differ are
    // common to all; then one digit of up to 8 bits per pass narrows down the bin of the
    // k-th key until that bin holds exactly the keys still needed); keys at or above the
    // resulting prefix are exactly the k best.
    uint64_t prefix = 0ull;
    if (n > topk) {
        unsigned* hist = fill;  // 256 bins, zero from the start of the kernel
        const int top = 63 - __clzll(static_cast<long long>(hi ^ lo));  // n > 1: keys differ
        prefix = top == 63 ? 0ull : (hi & ~((2ull << top) - 1ull));
        int width = top + 1 < 8 ? top + 1 : 8;
        int sh = top + 1 - width;
        int need = topk;
        while (true) {
            const int end = sh + width;
            const uint64_t hmask = end >= 64 ? 0ull : ~((1ull << end) - 1ull);
            const unsigned dmask = (1u << width) - 1u;
#pragma unroll
            for (int j = 0; j < IN; ++j)
                if (t + NT * j < n && (x[j] & hmask) == prefix)
                    atomicAdd(&hist[static_cast<unsigned>(x[j] >> sh) & dmask], 1u);
            __syncthreads();
            if (t < 32) {
                // lane l scans bins 255-8l .. 248-8l (descending key order), then clears them
                unsigned cb[8];
                unsigned sum = 0;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    cb[j] = hist[255 - (t * 8 + j)];
                    sum += cb[j];
                }
#pragma unroll
                for (int j = 0; j < 8; ++j) hist[255 - (t * 8 + j)] = 0u;
                if (t == 0) ctl[1] = -1;
                __syncwarp();
                unsigned inc = sum;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const unsigned y = __shfl_up_sync(kFull, inc, o);
                    if (t >= o) inc += y;
                }
                const unsigned exc = inc - sum;
                if (exc < static_cast<unsigned>(need) && static_cast<unsigned>(need) <= inc) {
                    unsigned above = exc;
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        if (above + cb[j] >= static_cast<unsigned>(need)) {
                            ctl[1] = 255 - (t * 8 + j);
                            ctl[2] = static_cast<int>(above);
                            ctl[3] = static_cast<int>(cb[j]);
                            break;
                        }
                        above += cb[j];
                    }
                }
            }
            __syncthreads();
            const int d = ctl[1];
            if (d < 0) {  // no bin holds the k-th key: counts are inconsistent
                if (t == 0) atomicOr(err, kErrAssert);
                break;
            }
            prefix |= static_cast<uint64_t>(d) << sh;
            need -= ctl[2];
            const bool done = ctl[3] == need || sh == 0;
            __syncthreads();  // every thread has read ctl before the next scan writes it
            if (done) break;
            width = sh < 8 ? sh : 8;
            sh -= width;
        }
    }
    // the (at most k) kept keys into xs[0 .. n_out), the rest of the first kRankN slots 0
    for (int i = t; i < kRankN; i += NT) xs[i] = 0ull;
    if (t == 0) ctl[2] = 0;
    __syncthreads();
#pragma unroll
    for (int j = 0; j < IN; ++j) {
        const bool keep = t + NT * j < n && x[j] >= prefix;
        const unsigned m = __ballot_sync(kFull, keep);
        if (m) {
            int at = 0;
            if (lane == 0) at = atomicAdd(&ctl[2], __popc(m));
            at = __shfl_sync(kFull, at, 0);
            const int pos = at + __popc(m & ((1u << lane) - 1u));
            if (keep && pos < kRankN) xs[pos] = x[j];
        }
    }
    __syncthreads();
    if (t == 0 && ctl[2] != n_out) atomicOr(err, kErrAssert);
    if (t < kRankThreads) rank_merge_write(xs, xs + kRankN, n_out, topk, io, so, t, 1);
}

// ------------------------------------------------------------------- split merge

constexpr int kMaxSplits = 1024;  // candidate lists per row the merge accepts
constexpr size_t kMaxStageBytes = 160 * 1024;  // candidates a merge block stages in smem

// One block per row: the row's n_splits candidate lists (each the exact top-k of one key
// range, unordered) -> the row's top k in rank order (or, with out_keys, as unordered keys
// and a count).  List l of row r: cand_cnt[r * cnt_row + l * cnt_list] keys at
// cand + r * row_stride + l * list_stride.  An MSD radix select runs directly
// over the lists in global memory: the bits above the highest bit in which the smallest
// and the largest candidate differ are skipped, then 8-bit digits narrow down the bin of
// the k-th key until exactly k keys are at or above the prefix (keys are distinct).  The
// k survivors are gathered into shared memory and ranked by rank_merge_write.
template <int kMergeThreads>
__global__ void __launch_bounds__(kMergeThreads) topk_split_merge_kernel(
    int topk, int n_splits, int lists_per_group, const uint64_t* cand, int64_t row_stride,
    int64_t list_stride, const int* cand_cnt, int64_t cnt_row, int64_t cnt_list, int32_t* idx,
    float* score, uint64_t* out_keys, int* out_cnt, int staged, int append_cap, unsigned* err) {
    // staged: the block's candidate slots are copied once into dynamic shared memory and
    // every pass reads them there (empty slots hold 0, which no rank key equals: its low
    // word is 0xFFFFFFFF - position).  append_cap > 0 (with out_keys): the block appends its
    // survivors to input row `row`'s list, out_keys[row * append_cap ...], at a cursor
    // out_cnt[row] (zero before the launch), instead of writing list v of its own.
    extern __shared__ uint64_t stg[];
    __shared__ __align__(16) uint64_t xs[2 * kRankN];  // keys, then ranking scratch
    __shared__ unsigned hist[256];
    __shared__ unsigned long long range[2];
    __shared__ int ctl[4];  // 0 digit, 1 above, 2 in-bin, 3 write cursor
    __shared__ int cnt_s[kMaxSplits];
    __shared__ int total_s;
    // output row v: lists first .. first + lists_per_group - 1 of input row `row` (a row's
    // lists fall into ceil(n_splits / lists_per_group) groups, merged by separate blocks)
    const int v = blockIdx.x;
    const int n_groups = (n_splits + lists_per_group - 1) / lists_per_group;
    const int row = v / n_groups;
    const int first = (v - row * n_groups) * lists_per_group;
    n_splits = n_splits - first < lists_per_group ? n_splits - first : lists_per_group;
    const int tid = threadIdx.x;
    const uint64_t* rc = cand + static_cast<int64_t>(row) * row_stride +
                         static_cast<int64_t>(first) * list_stride;
    const int* cc = cand_cnt + static_cast<int64_t>(row) * cnt_row +
                    static_cast<int64_t>(first) * cnt_list;
    if (tid == 0) total_s = 0;
    __syncthreads();
    for (int sp = tid; sp < n_splits; sp += kMergeThreads) {
        int c = cc[static_cast<int64_t>(sp) * cnt_list];
        if (c < 0 || c > topk) {
            atomicOr(err, kErrAssert);
            c = 0;
        }
        cnt_s[sp] = c;
        atomicAdd(&total_s, c);
    }
    __syncthreads();
    const int total = total_s;
    // every candidate slot of the row: `f(key, valid)` in every lane (warp-uniform calls,
    // so f may use warp collectives).  Slot s is entry s % topk of list s / topk; a pass
    // walks the slots four per thread at a time so that a thread's loads are independent.
    const int n_slots = n_splits * topk;
    if (staged) {
        for (int slot = tid; slot < n_slots; slot += kMergeThreads) {
            const int sp = slot / topk;
            const int j = slot - sp * topk;
            stg[slot] = j < cnt_s[sp] ? rc[static_cast<int64_t>(sp) * list_stride + j] : 0ull;
        }
        __syncthreads();
    }
    auto for_each = [&](auto f) {
        constexpr int U = 4;
        for (int base = 0; base < n_slots; base += U * kMergeThreads) {
            uint64_t x[U];
            bool ok[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int slot = base + u * kMergeThreads + tid;
                if (staged) {
                    x[u] = slot < n_slots ? stg[slot] : 0ull;
                    ok[u] = x[u] != 0ull;
                } else {
                    const int sp = slot / topk;
                    const int j = slot - sp * topk;
                    ok[u] = slot < n_slots && j < cnt_s[sp < n_splits ? sp : 0];
                    x[u] = ok[u] ? rc[static_cast<int64_t>(sp) * list_stride + j] : 0ull;
                }
            }
#pragma unroll
            for (int u = 0; u < U; ++u) f(x[u], ok[u]);
        }
    };
    const int lane = tid & 31;
    for (int i = tid; i < 256; i += kMergeThreads) hist[i] = 0u;
    if (tid == 0) {
        range[0] = ~0ull;
        range[1] = 0ull;
        ctl[3] = 0;
    }
    __syncthreads();
    uint64_t prefix = 0ull;  // keys >= prefix are kept
    const int n = total < topk ? total : topk;
    if (total > topk) {
        uint64_t lo = ~0ull, hi = 0ull;
        for_each([&](uint64_t x, bool ok) {
            if (ok) {
                lo = x < lo ? x : lo;
                hi = x > hi ? x : hi;
            }
        });
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const uint64_t l2 = __shfl_xor_sync(0xFFFFFFFFu, lo, o);
            const uint64_t h2 = __shfl_xor_sync(0xFFFFFFFFu, hi, o);
            lo = l2 < lo ? l2 : lo;
            hi = h2 > hi ? h2 : hi;
        }
        if ((tid & 31) == 0) {
            atomicMin(&range[0], static_cast<unsigned long long>(lo));
            atomicMax(&range[1], static_cast<unsigned long long>(hi));
        }
        __syncthreads();
        lo = range[0];
        hi = range[1];
        const int top = lo == hi ? 0 : 63 - __clzll(static_cast<long long>(lo ^ hi));
        prefix = top == 63 ? 0ull : (hi & ~((2ull << top) - 1ull));
        int width = top + 1 < 8 ? top + 1 : 8;
        int shift = top + 1 - width;
        int need = topk;
        while (true) {
            const int end = shift + width;
            const uint64_t hmask = end >= 64 ? 0ull : ~((1ull << end) - 1ull);
            const unsigned dmask = (1u << width) - 1u;
            for_each([&](uint64_t x, bool ok) {
                if (ok && (x & hmask) == prefix)
                    atomicAdd(&hist[static_cast<unsigned>(x >> shift) & dmask], 1u);
            });
            __syncthreads();
            if (tid < 32) {
                // lane l scans bins 255-8l .. 248-8l (descending key order), then clears them
                unsigned c[8];
                unsigned sum = 0;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    c[j] = hist[255 - (tid * 8 + j)];
                    sum += c[j];
                }
#pragma unroll
                for (int j = 0; j < 8; ++j) hist[255 - (tid * 8 + j)] = 0u;
                if (tid == 0) ctl[0] = -1;
                __syncwarp();
                unsigned incl = sum;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const unsigned v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
                    if (tid >= o) incl += v;
                }
                const unsigned excl = incl - sum;
                if (excl < static_cast<unsigned>(need) && static_cast<unsigned>(need) <= incl) {
                    unsigned above = excl;
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        if (above + c[j] >= static_cast<unsigned>(need)) {
                            ctl[0] = 255 - (tid * 8 + j);
                            ctl[1] = static_cast<int>(above);
                            ctl[2] = static_cast<int>(c[j]);
                            break;
                        }
                        above += c[j];
                    }
                }
            }
            __syncthreads();
            const int d = ctl[0];
            if (d < 0) {  // no bin holds the k-th key: counts are inconsistent
                if (tid == 0) atomicOr(err, kErrAssert);
                break;
            }
            prefix |= static_cast<uint64_t>(d) << shift;
            need -= ctl[1];
            const bool done = ctl[2] == need || shift == 0;
            __syncthreads();  // every thread has read ctl before the next scan writes it
            if (done) break;
            width = shift < 8 ? shift : 8;
            shift -= width;
        }
    }
    // the survivors (all candidates when there are at most k of them) into shared memory
    for (int i = tid; i < kRankN; i += kMergeThreads) xs[i] = 0ull;
    __syncthreads();
    for_each([&](uint64_t x, bool ok) {
        const bool keep = ok && x >= prefix;
        const unsigned m = __ballot_sync(0xFFFFFFFFu, keep);
        if (m) {
            int at = 0;
            if (lane == 0) at = atomicAdd(&ctl[3], __popc(m));
            at = __shfl_sync(0xFFFFFFFFu, at, 0);
            const int pos = at + __popc(m & ((1u << lane) - 1u));
            if (keep && pos < kRankN) xs[pos] = x;
        }
    });
    __syncthreads();
    if (tid == 0 && ctl[3] != n) atomicOr(err, kErrAssert);
    if (out_keys && append_cap > 0) {  // the survivors appended to the row's list
        if (tid == 0) ctl[0] = atomicAdd(&out_cnt[row], n);
        __syncthreads();
        const int at = ctl[0];
        if (at + n > append_cap) {
            if (tid == 0) atomicOr(err, kErrAssert);
            return;
        }
        for (int i = tid; i < n; i += kMergeThreads)
            out_keys[static_cast<int64_t>(row) * append_cap + at + i] = xs[i];
        return;
    }
    if (out_keys) {  // the survivors themselves, unordered
        for (int i = tid; i < n; i += kMergeThreads)
            out_keys[static_cast<int64_t>(v) * topk + i] = xs[i];
        if (tid == 0) out_cnt[v] = n;
        return;
    }
    if (tid < kRankThreads)
        rank_merge_write(xs, xs + kRankN, n, topk, idx + static_cast<int64_t>(v) * topk,
                         score ? score + static_cast<int64_t>(v) * topk : nullptr, tid, 1);
}

}  // namespace

int topk_rank_max_stride() { return kRankListIn * kRankThreads; }

constexpr int kRankSmemBytes = (2 * kRankN + kRankBucketMax) * 8 + 2 * kRankBuckets * 4;

template <int NT, int IN>
cudaError_t rank_launch(int rows, int topk, int stride, const uint64_t* cand, const int* cand_cnt,
                        int32_t* idx, float* score, unsigned* err, cudaStream_t st) {
    static cudaError_t attr = cudaFuncSetAttribute(
        topk_rank_kernel<NT, IN>, cudaFuncAttributeMaxDynamicSharedMemorySize, kRankSmemBytes);
    if (attr != cudaSuccess) return attr;
    topk_rank_kernel<NT, IN><<<rows, NT, kRankSmemBytes, st>>>(topk, stride, cand, cand_cnt, idx,
                                                              score, err);
    return cudaSuccess;
}

cudaError_t launch_topk_rank(int rows, int topk, int stride, const uint64_t* cand,
                             const int* cand_cnt, int32_t* idx, float* score, unsigned* err,
                             cudaStream_t st) {
    if (rows == 0) return cudaSuccess;
    if (stride < topk || stride > topk_rank_max_stride()) return cudaErrorInvalidValue;
    // Few rows (decode): one wide block per row, the row's latency is the call's.  Else
    // 256 threads and the fewest list slots per thread that hold the stride (registers:
    // blocks per SM).
    constexpr int kWide = 1024;
    const cudaError_t e =
        rows < 152 ? (stride <= 2 * kWide
                          ? rank_launch<kWide, 2>(rows, topk, stride, cand, cand_cnt, idx, score,
                                                  err, st)
                          : rank_launch<kWide, kRankListIn * kRankThreads / kWide>(
                                rows, topk, stride, cand, cand_cnt, idx, score, err, st))
        : stride <= kRankN ? rank_launch<kRankThreads, kRankPer>(rows, topk, stride, cand,
                                                                 cand_cnt, idx, score, err, st)
        : stride <= 17 * kRankThreads
            ? rank_launch<kRankThreads, 17>(rows, topk, stride, cand, cand_cnt, idx, score, err,
                                            st)
            : rank_launch<kRankThreads, kRankListIn>(rows, topk, stride, cand, cand_cnt, idx,
                                                     score, err, st);
    if (e != cudaSuccess) return e;
    note_launches(1);
    return cudaGetLastError();
}

cudaError_t launch_topk_merge(int rows, int topk, int n_splits, const uint64_t* cand,
                              const int* cand_cnt, int32_t* idx, float* score, unsigned* err,
                              cudaStream_t st) {
    return launch_topk_merge_strided(rows, topk, n_splits, cand,
                                     static_cast<int64_t>(n_splits) * topk, topk, cand_cnt,
                                     n_splits, 1, idx, score, nullptr, nullptr, err, st);
}

cudaError_t launch_topk_merge_strided(int rows, int topk, int n_lists, const uint64_t* cand,
                                      int64_t row_stride, int64_t list_stride,
                                      const int* cand_cnt, int64_t cnt_row, int64_t cnt_list,
                                      int32_t* idx, float* score, uint64_t* out_keys,
                                      int* out_cnt, unsigned* err, cudaStream_t st) {
    return launch_topk_merge_grouped(rows, topk, n_lists, n_lists, cand, row_stride, list_stride,
                                     cand_cnt, cnt_row, cnt_list, idx, score, out_keys, out_cnt,
                                     err, st, 0);
}

cudaError_t launch_topk_merge_grouped(int rows, int topk, int n_lists, int lists_per_group,
                                      const uint64_t* cand, int64_t row_stride,
                                      int64_t list_stride, const int* cand_cnt, int64_t cnt_row,
                                      int64_t cnt_list, int32_t* idx, float* score,
                                      uint64_t* out_keys, int* out_cnt, unsigned* err,
                                      cudaStream_t st, int append_cap) {
    if (rows == 0) return cudaSuccess;
    if (n_lists < 1 || n_lists > kMaxSplits || lists_per_group < 1) return cudaErrorInvalidValue;
    const int groups = (n_lists + lists_per_group - 1) / lists_per_group;
    if (groups > 1 && !out_keys) return cudaErrorInvalidValue;  // partial merges stay unordered
    const int64_t blocks = static_cast<int64_t>(rows) * groups;
    if (blocks > 0x7FFFFFFF) return cudaErrorInvalidValue;
    // few blocks (decode): wide blocks, candidates staged in shared memory when they fit;
    // many: several narrower blocks per SM reading the lists where they are
    if (blocks < 4 * 152) {
        const int per_block = (lists_per_group < n_lists ? lists_per_group : n_lists);
        const size_t stage = static_cast<size_t>(per_block) * topk * sizeof(uint64_t);
        const int staged = stage <= kMaxStageBytes ? 1 : 0;
        if (staged) {
            cudaError_t e = cudaFuncSetAttribute(topk_split_merge_kernel<1024>,
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 static_cast<int>(kMaxStageBytes));
            if (e != cudaSuccess) return e;
        }
        topk_split_merge_kernel<1024><<<static_cast<int>(blocks), 1024, staged ? stage : 0, st>>>(
            topk, n_lists, lists_per_group, cand, row_stride, list_stride, cand_cnt, cnt_row,
            cnt_list, idx, score, out_keys, out_cnt, staged, append_cap, err);
    } else {
        topk_split_merge_kernel<kRankThreads><<<static_cast<int>(blocks), kRankThreads, 0, st>>>(
            topk, n_lists, lists_per_group, cand, row_stride, list_stride, cand_cnt, cnt_row,
            cnt_list, idx, score, out_keys, out_cnt, 0, append_cap, err);
    }
    note_launches(1);
    return cudaGetLastError();
}

int topk_merge_group_size(int rows, int n_lists) {
    if (n_lists < 8 || rows >= 152) return n_lists;  // one pass is parallel enough
    int g = 1;
    while (g * g < n_lists) ++g;  // about sqrt(n) lists per group, then about sqrt(n) groups
    return g;
}

size_t topk_merge_stage_bytes(int rows, int topk, int n_lists) {
    const int g = topk_merge_group_size(rows, n_lists);
    if (g >= n_lists) return 0;
    const size_t lists = static_cast<size_t>(rows) * ((n_lists + g - 1) / g);
    return lists * topk * sizeof(uint64_t) + ((lists * sizeof(int) + 255) & ~size_t(255));
}

cudaError_t launch_topk_merge_two_stage(int rows, int topk, int n_lists, const uint64_t* cand,
                                        int64_t row_stride, int64_t list_stride,
                                        const int* cand_cnt, int64_t cnt_row, int64_t cnt_list,
                                        void* stage, int32_t* idx, float* score,
                                        uint64_t* out_keys, int* out_cnt, unsigned* err,
                                        cudaStream_t st) {
    const int g = topk_merge_group_size(rows, n_lists);
    if (g >= n_lists || !stage)
        return launch_topk_merge_strided(rows, topk, n_lists, cand, row_stride, list_stride,
                                         cand_cnt, cnt_row, cnt_list, idx, score, out_keys,
                                         out_cnt, err, st);
    // Rank-ordered output: groups of lists merged by separate blocks, each appending its
    // top k to one list per row, which the select-and-rank kernel finishes (it takes up to
    // topk_rank_max_stride() keys a row) -- when at most that many group results per row
    // fit, and each group's lists fit one block's staging.
    const int groups_r = topk_rank_max_stride() / topk < 3 ? topk_rank_max_stride() / topk : 3;
    const int g_r = groups_r > 0 ? (n_lists + groups_r - 1) / groups_r : n_lists + 1;
    const size_t row_keys = static_cast<size_t>(groups_r) * topk;
    const size_t need = rows * row_keys * sizeof(uint64_t) + rows * sizeof(int);
    if (!out_keys && groups_r > 1 && g_r < n_lists &&
        static_cast<size_t>(g_r) * topk * sizeof(uint64_t) <= kMaxStageBytes &&
        need <= topk_merge_stage_bytes(rows, topk, n_lists)) {
        uint64_t* rkeys = static_cast<uint64_t*>(stage);
        int* rcnt = reinterpret_cast<int*>(rkeys + rows * row_keys);
        cudaError_t e = cudaMemsetAsync(rcnt, 0, rows * sizeof(int), st);
        if (e != cudaSuccess) return e;
        e = launch_topk_merge_grouped(rows, topk, n_lists, g_r, cand, row_stride, list_stride,
                                      cand_cnt, cnt_row, cnt_list, nullptr, nullptr, rkeys, rcnt,
                                      err, st, static_cast<int>(row_keys));
        if (e != cudaSuccess) return e;
        return launch_topk_rank(rows, topk, static_cast<int>(row_keys), rkeys, rcnt, idx, score,
                                err, st);
    }
    const int groups = (n_lists + g - 1) / g;
    uint64_t* skeys = static_cast<uint64_t*>(stage);
    int* scnt = reinterpret_cast<int*>(skeys + static_cast<size_t>(rows) * groups * topk);
    cudaError_t e = launch_topk_merge_grouped(rows, topk, n_lists, g, cand, row_stride,
                                              list_stride, cand_cnt, cnt_row, cnt_list, nullptr,
                                              nullptr, skeys, scnt, err, st);
    if (e != cudaSuccess) return e;
    return launch_topk_merge_strided(rows, topk, groups, skeys,
                                     static_cast<int64_t>(groups) * topk, topk, scnt, groups, 1,
                                     idx, score, out_keys, out_cnt, err, st);
}

}  // namespace tsi
