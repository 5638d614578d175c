// Tensor-core lightning indexer for sm_103a (tcgen05 / TMEM / TMA).
//
// I[t,s] = sum_j w[t,j] * ReLU(qI[t,j] . kI[s]) for s <= p_t, then the top-k keys of
// each row ("GLM-5.2 技术报告速览", §IndexShare: the score equation, k = 2048; the
// ReLU form is chosen there for speed and FP8 friendliness).  One kernel, three modes:
//   - capped and select (the default): each 128-key tile is scored in TMEM and streamed
//     into a shared-memory top-k selector per query row, so no score reaches HBM.  With
//     several query rows per sequence the call runs the kernel three times:
//       1. (capped) on a strided sample of the keys (every 32nd, gathered into the
//          workspace) with a small k' per row: the k'-th largest sampled score becomes the
//          row's admission threshold, about c k keys of the row lie above it;
//       2. (capped) on all keys, admitting only scores at or above that threshold: about
//          c k appends per row instead of the ~k ln(L / k) of a selector that starts from
//          nothing; the buffer is sized so that it never needs a room check, an append is
//          the raw (score bits, position) pair (the rank key is built once, when the unit
//          ends), the rounds over tiles wholly inside the row skip the bounds tests, and
//          each row leaves every key it holds, unordered, for the ranking kernel (which
//          keeps the k best);
//       3. (select: room checks, compactions) on the units where some row ended with
//          fewer than k keys admitted or overflowed its buffer (the sample misjudged it),
//          from no threshold at all: the result is exact for any input.
//     With one query per sequence (decode) the select mode runs once over key chunks, each
//     chunk leaving its exact k best for the merge kernels.
//   - store (the two-pass alternative): every causal score goes to a row-major fp32 buffer,
//     a chunk of query rows at a time; topk_rows.cu then selects and ranks each row's k
//     best keys from it, at 4 B of HBM writes and reads per causal pair.
//
// MMA shape: keys on M (128 rows of kI per tile, the A operand), the 64 heads of R
// consecutive query rows on N = 64 R (the B operand), d_I = 128 on K, fp32 accumulators
// in TMEM.  R = 4 for e4m3 (N = 256), 2 for bf16 (N = 128), 1 for decode.  The larger R,
// the more query rows share each key tile: fewer tiles, MMA issues and barrier round
// trips, less L2 traffic.  An epilogue warp reads its 32 TMEM lanes (keys) of its row's 64
// columns as two 16-lane slices in the 16x256b shape (see tile_score): each thread holds
// two keys x 16 heads per slice, so its 16 gate weights stay in registers for the unit.
//
// Roles of one persistent CTA (608 threads):
//   warp 0       TMA producer: Q tile of the unit, key tiles into a ring of stages, the
//                next unit's query rows and gate weights prefetched into L2
//   warps 1, 18  MMA issuers (lane 0 issues): warp 1 the even tiles, warp 18 the odd ones
//                (512 TMEM columns: 512 / N accumulators, so the MMA runs that many tiles
//                ahead; two issuers overlap each other's barrier waits).  Warp 1 also
//                allocates TMEM.
//   warps 2..17  R epilogue groups of 16 / R warps, one per query row of the unit; group
//                r reads columns [64r, 64r+64) of an accumulator (and, selecting, owns a
//                selector).  With 16 / R > 4 warps per row, the row's warp sets share out
//                the tiles.
// Units (R consecutive query rows x one key range) are visited longest first and spread
// round-robin over the CTAs (or taken from a list of units, for the third launch).
#include <mutex>

#include <cudaTypedefs.h>

#include "kernels_tc.cuh"
#include "tc_common.cuh"
#include "topk_select.cuh"

namespace tsi {
namespace {

constexpr int kTileKeys = 128;  // MMA M
constexpr int kEpiWarps = 16;
constexpr int kMmaWarp2 = 2 + kEpiWarps;  // the second MMA issuer (odd tiles)
constexpr int kThreads = 96 + 32 * kEpiWarps;
constexpr int kTmemCols = 512;
constexpr int kChunkBytes = 128 * 128;  // one 128-row x 128-byte swizzled tile
constexpr int kAllBar = 8;  // named barrier of all epilogue warps (selectors use 1..4)

template <int QK>
struct TileCfg;
template <>
struct TileCfg<TSI_E4M3> {
    static constexpr int kRows = 4;    // query rows per unit
    static constexpr int kCap = 4352;  // selector capacity per row (several rows per unit)
    static constexpr int kChunks = 1;  // 128-byte pieces of a d_I = 128 row
    static constexpr int kStages = 4;
    static constexpr int kSelStages = 3;  // key stages beside R selectors
    static constexpr uint32_t kFmt = 0;
    static constexpr int kKSteps = 4;  // K = 32 per MMA
};
template <>
struct TileCfg<TSI_BF16> {
    static constexpr int kRows = 2;
    static constexpr int kCap = 5888;
    static constexpr int kChunks = 2;
    static constexpr int kStages = 3;
    static constexpr int kSelStages = 3;
    static constexpr uint32_t kFmt = 1;
    static constexpr int kKSteps = 4;  // per chunk, K = 16 per MMA
};

// store: scores to HBM.  select: each row's selector checks its room once per round and
// compacts when it runs low (exact from any start).  capped: no room check at all, for
// launches where a row's admitted keys are expected to fit (the sampled-threshold launches);
// a row whose keys overflow the buffer is reported like a row that came short.
enum : int { kModeStore = 0, kModeSelect = 1, kModeCapped = 2 };

// R = query rows per unit: the format's default, or 1 for one query per sequence (decode),
// where the four warp sets of the single row share out the key tiles instead of idling.
// kMode: the epilogue stores the scores, or selects each row's top k itself.
template <int QK, int R = TileCfg<QK>::kRows, int kMode = kModeSelect>
struct Lay {
    using C = TileCfg<QK>;
    static constexpr bool kStore = kMode == kModeStore;
    static constexpr int kR = R;
    // selector capacity: the row's warp sets offer up to 4 kGroupThreads keys between two
    // room checks (see the trigger in the epilogue), beyond the k that are kept
    static constexpr int kCap = R == 1 ? 5120 : C::kCap;
    static constexpr int kStages = (R > 1 && !kStore) ? C::kSelStages : C::kStages;
    static constexpr int kN = 64 * kR;             // MMA N
    static constexpr int kAccBufs = kTmemCols / kN;
    static constexpr int kSubs = 4 / kR;           // warp sets per row sharing out the tiles
    static constexpr int kGroupThreads = 128 * kSubs;
    static constexpr int kReaders = 4 * kR;        // warps reading each accumulator
    static constexpr int kStageBytes = C::kChunks * kChunkBytes;
    static constexpr int kQChunkBytes = kN * 128;  // kN rows of 128 bytes per K chunk
    static constexpr int kQBytes = C::kChunks * kQChunkBytes;
    // the store variant keeps no selector: scores go to global memory
    static constexpr int kSelBytes = kStore ? 0 : (selector_smem_bytes<kCap>() + 15) & ~15;
    static constexpr uint32_t kIdesc = tc::instr_desc(C::kFmt, kTileKeys, kN);
    static constexpr int kBars = 2 * kStages + 2 * kAccBufs + 3;
    static constexpr int kSmem = 1024 /* alignment slack */ + kStages * kStageBytes +
                                 kQBytes + kR * kSelBytes + kBars * 8 + 16;
    // a room check happens once per round (two tiles of each warp set); between two checks
    // a thread's view of the count may miss the other warps' last round, and the next round
    // adds at most 2 kGroupThreads keys
    static constexpr int kTrigger = kCap - 4 * kGroupThreads;
    static_assert(kSmem <= 227 * 1024, "shared memory");
    static_assert(kEpiWarps == 4 * kR * kSubs, "every epilogue warp has a row");
};

// Key sample of the threshold launch: every 32nd key.
constexpr int kSampleShift = 5;

struct TcParams {
    const void* w;
    int w_dtype;
    int B, T, S, topk;
    int S_total;  // length of the whole cache (the keys here are a shard of it)
    int64_t key_offset;  // position of key 0 of kI in the whole cache
    const int32_t* kv_len;
    int32_t* idx;
    float* score;
    uint64_t* cand;
    int* cand_cnt;
    // Keys per candidate list: 0, lists of topk keys, each row's (chunk's) exact k best; or
    // the selector's capacity, every key the row held (the ranking kernel keeps the k best,
    // so no exact selection stalls this kernel at the end of a unit).
    int cand_stride;
    int n_chunks, chunk_keys, n_units;
    int t_begin, t_end;  // query rows [t_begin, t_end) of every sequence in this launch
    float* scores;       // store variant: row (b, t) at (b * (t_end - t_begin) + t - t_begin) * ld
    int64_t ld;
    unsigned* err;
    // Key i of this launch sits at position i << key_shift (0: every key; kSampleShift: the
    // threshold launch's sample, key rows gathered into a buffer of their own).
    int key_shift;
    // Select mode, optional: per-row admission thresholds to start from ([B * T] scores);
    // per-row thresholds to produce instead of candidate lists (the threshold launch: the
    // topk-th largest sampled score, -inf where every key fits the selector anyway);
    // units whose rows came short of k keys (appended to fail_list, counted in fail_count);
    // the units to visit (unit_list[0 .. *unit_count), instead of all n_units).
    const float* tau_in;
    float* tau_out;
    int* fail_list;
    int* fail_count;
    const int* unit_list;
    const int* unit_count;
    // raw query rows and their size (the next unit's rows and gate weights are prefetched
    // into L2 while the current unit runs)
    const uint8_t* q_raw;
    int q_row_bytes, w_bytes;
};

struct Unit {
    int b, t_hi, chunk;
    int64_t key_lo, key_hi;
    int ntiles;
};

// Unit u: row group j = u / (B * n_chunks) counted from the end of the launch's rows
// (longest rows first), sequence b, key chunk.  Rows t_hi - R + 1 .. t_hi (the first may be
// below t_begin: those belong to another launch and are skipped).
template <int R>
__device__ __forceinline__ Unit unit_of(const TcParams& p, int u) {
    Unit U;
    U.chunk = u % p.n_chunks;
    const int pu = u / p.n_chunks;
    const int j = pu / p.B;
    U.b = pu % p.B;
    U.t_hi = p.t_end - 1 - R * j;
    // positions relative to key 0 of this call; keys beyond the shard are not here
    const int64_t p_hi = query_position(p.kv_len, U.b, p.T, p.S_total, U.t_hi) - p.key_offset;
    int64_t end = p_hi >= 0 ? (p_hi >> p.key_shift) + 1 : 0;
    if (end > p.S) end = p.S;
    U.key_lo = static_cast<int64_t>(U.chunk) * p.chunk_keys;
    U.key_hi = U.key_lo + p.chunk_keys < end ? U.key_lo + p.chunk_keys : end;
    if (U.key_hi < U.key_lo) U.key_hi = U.key_lo;
    U.ntiles = static_cast<int>((U.key_hi - U.key_lo + kTileKeys - 1) / kTileKeys);
    return U;
}

// Wait for a phase that is usually complete already: one probe, then the bounded wait.
__device__ __forceinline__ bool wait_fast(uint64_t* bar, uint32_t parity, bool probed,
                                          volatile int* abort, unsigned* err) {
    return probed || tc::mbar_wait(bar, parity, abort, err);
}

// Head-pair slots (of the eight in each 32-column load) whose ReLU runs on the ALU pipe as
// a max with 0; the others run on the FMA pipe as x + |x| = 2 ReLU(x) (exact) against
// halved gate weights.  Either way w * ReLU(x) is the same product, so the split only
// balances the two pipes and never changes a score.  Two of eight for the four-row e4m3
// units, one for the two-row bf16 units (N = 128), whose MMAs leave the epilogue more time.
template <int N>
constexpr int alu_slots() {
    return N == 128 ? 1 : 2;
}

// Key lane (within the warp's 32 TMEM lanes) whose score tile_score returns to this
// thread: lane 8 (T % 4) + T / 4 of thread T.
__device__ __forceinline__ int scored_lane(int lane) { return 8 * (lane & 3) + (lane >> 2); }

// The 16 gate weights this thread needs (see tile_score), each duplicated into both halves
// of a pair and halved where its ReLU is formed as x + |x|: slot j = 8 ch + 2 m + e holds
// head 32 ch + 8 m + 2 (T % 4) + e.  (Halving a gate weight below 2^-125, a subnormal,
// would drop its last bit; no gate weight is that small.)
template <int N>
__device__ __forceinline__ void load_gates(float2 (&wd)[16], const void* w, int64_t row_h0,
                                           int w_dtype, int lane) {
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        const int ch = j >> 3, m = (j >> 1) & 3, e = j & 1;
        const float f = (j & 7) < alu_slots<N>() ? 1.f : 0.5f;
        const float g = f * load_elem(w, row_h0 + 32 * ch + 8 * m + 2 * (lane & 3) + e, w_dtype);
        wd[j] = make_float2(g, g);
    }
}

// Scores of query row r of the unit from accumulator buffer a: the sum over the 64 heads of
// w[h] * max(0, q[h].k).
//
// The warp reads its 32 TMEM lanes (keys) as two 16-lane slices, each in two loads of 32
// columns (16x256b shape).  Thread T then holds, per slice, two keys (lanes L = T / 4 and
// L + 8 of the slice) x 16 heads (8 m + 2 c + {0, 1} of each load, c = T % 4), so it needs
// only those 16 gate weights, kept in registers for the whole unit.  Each packed FMA adds
// one head of both keys, so a slice leaves one (key L, key L + 8) pair of partial sums.
// The four threads with equal L then reduce-scatter their two pairs in two shuffle steps:
// thread c ends with the whole sum of key lane 8 c + L (scored_lane), added in a fixed
// order.  The buffer is released to the MMA once the last columns are in registers.
template <int N>
__device__ __forceinline__ float tile_score(uint32_t tmem, int quad, int r, int a, uint64_t* tempty,
                                            const float2 (&wd)[16]) {
    tc::tc_fence_after();
    const uint32_t taddr = tmem + (static_cast<uint32_t>(quad * 32) << 16) + a * N + r * 64;
    float2 part[2];  // per slice: (key L, key L + 8) partial sums over this thread's heads
#pragma unroll
    for (int slice = 0; slice < 2; ++slice) {
        float2 acc0 = make_float2(0.f, 0.f), acc1 = acc0;
#pragma unroll
        for (int ch = 0; ch < 2; ++ch) {
            uint32_t v[16];
            TSI_TMEM_LD16x256_X4(taddr + (static_cast<uint32_t>(16 * slice) << 16) + 32 * ch, v);
            tc::tmem_wait_ld();
            if (slice == 1 && ch == 1) {
                tc::tc_fence_before();
                __syncwarp();
                if ((threadIdx.x & 31) == 0) tc::mbar_arrive(&tempty[a]);
            }
#pragma unroll
            for (int m = 0; m < 4; ++m) {
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int j = 8 * ch + 2 * m + e;
                    const float x = __uint_as_float(v[4 * m + e]);
                    const float y = __uint_as_float(v[4 * m + 2 + e]);
                    const float2 rx = (j & 7) < alu_slots<N>()
                                          ? make_float2(fmaxf(x, 0.f), fmaxf(y, 0.f))
                                          : make_float2(__fadd_rn(x, fabsf(x)),
                                                        __fadd_rn(y, fabsf(y)));
                    if (e == 0)
                        acc0 = __ffma2_rn(wd[j], rx, acc0);
                    else
                        acc1 = __ffma2_rn(wd[j], rx, acc1);
                }
            }
        }
        part[slice] = __fadd2_rn(acc0, acc1);
    }
    // reduce-scatter over the quad: first the slices (xor 2), then the two keys (xor 1)
    const int c = threadIdx.x & 3;
    const bool hi = (c >> 1) & 1;
    const float2 send = hi ? part[0] : part[1];
    const float2 keep = hi ? part[1] : part[0];
    const float2 got = make_float2(__shfl_xor_sync(0xFFFFFFFFu, send.x, 2),
                                   __shfl_xor_sync(0xFFFFFFFFu, send.y, 2));
    const float2 t = __fadd2_rn(keep, got);
    const bool odd = c & 1;
    const float other = __shfl_xor_sync(0xFFFFFFFFu, odd ? t.x : t.y, 1);
    return __fadd_rn(odd ? t.y : t.x, other);
}

template <int QK, int R, int kMode>
__global__ void __launch_bounds__(kThreads, 1)
    tsi_indexer_tc_kernel(const __grid_constant__ CUtensorMap tmap_k,
                          const __grid_constant__ CUtensorMap tmap_q, const TcParams p) {
    using C = TileCfg<QK>;
    using L = Lay<QK, R, kMode>;
    constexpr bool kStore = L::kStore;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* stages = base;
    uint8_t* qbuf = stages + L::kStages * L::kStageBytes;
    uint8_t* sel_mem = qbuf + L::kQBytes;
    uint64_t* bars = reinterpret_cast<uint64_t*>(sel_mem + R * L::kSelBytes);
    uint64_t* full = bars;
    uint64_t* empty = full + L::kStages;
    uint64_t* tfull = empty + L::kStages;
    uint64_t* tempty = tfull + L::kAccBufs;
    uint64_t* qfull = tempty + L::kAccBufs;
    uint64_t* qempty = qfull + 1;
    uint64_t* done = qempty + 1;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);
    volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < L::kStages; ++s) {
            tc::mbar_init(&full[s], 1);
            tc::mbar_init(&empty[s], 1);
        }
        for (int a = 0; a < L::kAccBufs; ++a) {
            tc::mbar_init(&tfull[a], 1);
            tc::mbar_init(&tempty[a], L::kReaders);
        }
        tc::mbar_init(qfull, 1);
        tc::mbar_init(qempty, 2);  // both MMA issuers
        tc::mbar_init(done, 2);
        *abort = 0;
        tc::fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        tc::prefetch_tmap(&tmap_k);
        tc::prefetch_tmap(&tmap_q);
    }
    if (warp == 1) tc::tmem_alloc(tmem_slot, kTmemCols);
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // units of this launch: all of them, or those listed by an earlier launch
    const int n_units = p.unit_list ? *reinterpret_cast<const volatile int*>(p.unit_count)
                                    : p.n_units;

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            int s = 0;
            uint32_t ph = 0;  // phase of the ring slot s
            int unit_it = 0;
            int q_last = -1;  // unit of the last query load issued
            uint32_t loaded = 0, last_ph = 0;  // per slot (bit s): loaded once, last phase
            for (int j = blockIdx.x; j < n_units; j += gridDim.x, ++unit_it) {
                const Unit U = unit_of<R>(p, p.unit_list ? p.unit_list[j] : j);
                tc::mbar_wait(qempty, (unit_it & 1) ^ 1, abort, p.err);
                if (!*abort) {
                    q_last = unit_it;
                    tc::mbar_expect_tx(qfull, L::kQBytes);
                    const int qrow = (U.b * p.T + U.t_hi - (R - 1)) * 64;
                    for (int c = 0; c < C::kChunks; ++c)
                        for (int h = 0; h < L::kN; h += 128)
                            tc::tma_load_2d(qbuf + c * L::kQChunkBytes + h * 128, &tmap_q, c * 64,
                                            qrow + h, qfull);
                    // the next unit's query rows and gate weights into L2, so that its Q load
                    // and the epilogue's gate loads do not wait on HBM
                    const int jn = j + gridDim.x;
                    if (jn < n_units) {
                        const Unit Un = unit_of<R>(p, p.unit_list ? p.unit_list[jn] : jn);
                        int64_t r0 = static_cast<int64_t>(Un.b) * p.T + Un.t_hi - (R - 1);
                        const int64_t r1 = static_cast<int64_t>(Un.b) * p.T + Un.t_hi + 1;
                        if (r0 < static_cast<int64_t>(Un.b) * p.T) r0 = static_cast<int64_t>(Un.b) * p.T;
                        if (r1 > r0) {
                            tc::prefetch_l2(p.q_raw + r0 * 64 * p.q_row_bytes,
                                            static_cast<uint32_t>((r1 - r0) * 64 * p.q_row_bytes));
                            tc::prefetch_l2(static_cast<const uint8_t*>(p.w) + r0 * 64 * p.w_bytes,
                                            static_cast<uint32_t>((r1 - r0) * 64 * p.w_bytes));
                        }
                    }
                }
                for (int i = 0; i < U.ntiles; ++i) {
                    const bool ready = tc::mbar_try_wait(&empty[s], ph ^ 1);
                    if (wait_fast(&empty[s], ph ^ 1, ready, abort, p.err) && !*abort) {
                        loaded |= 1u << s;
                        last_ph = (last_ph & ~(1u << s)) | (ph << s);
                        tc::mbar_expect_tx(&full[s], L::kStageBytes);
                        const int krow = static_cast<int>(static_cast<int64_t>(U.b) * p.S + U.key_lo +
                                                          static_cast<int64_t>(i) * kTileKeys);
                        for (int c = 0; c < C::kChunks; ++c)
                            tc::tma_load_2d(stages + s * L::kStageBytes + c * kChunkBytes, &tmap_k,
                                            c * 64, krow, &full[s]);
                    }
                    if (++s == L::kStages) {
                        s = 0;
                        ph ^= 1;
                    }
                }
            }
            if (*abort) {  // loads still in flight must land before the CTA exits (at most
                           // one per slot: a slot is reloaded only after its data was used)
                if (q_last >= 0) tc::mbar_drain(qfull, q_last & 1);
                for (int i = 0; i < L::kStages; ++i)
                    if ((loaded >> i) & 1u) tc::mbar_drain(&full[i], (last_ph >> i) & 1u);
            }
        }
    } else if (warp == 1 || warp == kMmaWarp2) {
        // ------------------------------------------------------------ MMA issuers
        // The whole warp runs the loop (its descriptors stay warp-uniform); lane 0 issues
        // every MMA and commit.
        const bool leader = lane == 0;
        {
            const int mine = warp == 1 ? 0 : 1;  // tiles t of the CTA with t % 2 == mine
            int s = 0, a = 0, t = 0;
            uint32_t ph = 0, aph = 0;  // phases of ring slot s and accumulator a
            int unit_it = 0;
            const uint64_t adesc = tc::smem_desc(tc::smem_addr(stages), 16, 1024);
            const uint64_t bdesc = tc::smem_desc(tc::smem_addr(qbuf), 16, 1024);
            for (int j = blockIdx.x; j < n_units; j += gridDim.x, ++unit_it) {
                const Unit U = unit_of<R>(p, p.unit_list ? p.unit_list[j] : j);
                tc::mbar_wait(qfull, unit_it & 1, abort, p.err);
                for (int i = 0; i < U.ntiles; ++i, ++t) {
                    if ((t & 1) != mine) {  // the other issuer's tile: keep the ring counters
                        if (++s == L::kStages) {
                            s = 0;
                            ph ^= 1;
                        }
                        if (++a == L::kAccBufs) {
                            a = 0;
                            aph ^= 1;
                        }
                        continue;
                    }
                    // probe both barriers back to back so their latencies overlap
                    const bool f_ok = tc::mbar_try_wait(&full[s], ph);
                    const bool e_ok = tc::mbar_try_wait(&tempty[a], aph ^ 1);
                    const bool go = wait_fast(&full[s], ph, f_ok, abort, p.err) &&
                                    wait_fast(&tempty[a], aph ^ 1, e_ok, abort, p.err);
                    tc::tc_fence_after();
                    if (go) {
                        const uint32_t d = tmem + a * L::kN;
                        const uint64_t a0 = adesc + ((s * L::kStageBytes) >> 4);
#pragma unroll
                        for (int c = 0; c < C::kChunks; ++c) {
#pragma unroll
                            for (int k = 0; k < C::kKSteps; ++k) {
                                // descriptors address 16-byte units: offsets add directly
                                const uint64_t da = a0 + ((c * kChunkBytes + k * 32) >> 4);
                                const uint64_t db = bdesc + ((c * L::kQChunkBytes + k * 32) >> 4);
                                const uint32_t accum = (c | k) ? 1u : 0u;
                                if (leader) {
                                    if (QK == TSI_E4M3)
                                        tc::mma_f8(d, da, db, L::kIdesc, accum);
                                    else
                                        tc::mma_bf16(d, da, db, L::kIdesc, accum);
                                }
                            }
                        }
                    }
                    if (leader) tc::mma_commit(&empty[s]);
                    if (leader) tc::mma_commit(&tfull[a]);
                    if (++s == L::kStages) {
                        s = 0;
                        ph ^= 1;
                    }
                    if (++a == L::kAccBufs) {
                        a = 0;
                        aph ^= 1;
                    }
                }
                if (leader) tc::mma_commit(qempty);
            }
            // every MMA issued by both threads has finished before TMEM is released
            if (leader) tc::mma_commit(done);
            if (!tc::mbar_wait(done, 0, abort, p.err)) tc::mbar_drain(done, 0);
        }
    } else {
        // ------------------------------------------------------------ epilogue groups
        const int ew = warp - 2;
        const int r = ew / (4 * L::kSubs);  // query row of the unit handled by this group
        const int sub = (ew >> 2) % L::kSubs;  // this warp scores tiles i with i % kSubs == sub
        const int quad = warp & 3;  // TMEM lanes [32*quad, 32*quad+32) this warp may read
        const int gtid = (ew % (4 * L::kSubs)) * 32 + lane;
        TopKSelector<L::kGroupThreads, L::kCap> sel;
        if (!kStore) sel.bind(sel_mem + r * L::kSelBytes, gtid, 1 + r, p.err);
        int acc_base = 0;  // accumulator counter of the unit's first tile
        for (int j = blockIdx.x; j < n_units; j += gridDim.x) {
            const int u = p.unit_list ? p.unit_list[j] : j;
            const Unit U = unit_of<R>(p, u);
            const int t = U.t_hi - (R - 1) + r;
            const bool row_ok = t >= p.t_begin;
            const int64_t row = static_cast<int64_t>(U.b) * p.T + t;
            int64_t limit = 0;  // keys s < limit belong to this row
            int64_t n_row = 0;  // keys of the row in the whole call (before key chunks)
            float2 wd[16];  // this thread's 16 gate weights of the row (see load_gates)
#pragma unroll
            for (int m = 0; m < 16; ++m) wd[m] = make_float2(0.f, 0.f);
            if (row_ok) {
                const int64_t pr = query_position(p.kv_len, U.b, p.T, p.S_total, t) - p.key_offset;
                n_row = pr >= 0 ? (pr >> p.key_shift) + 1 : 0;
                if (n_row > p.S) n_row = p.S;
                limit = n_row < U.key_hi ? n_row : U.key_hi;
                load_gates<L::kN>(wd, p.w, row * 64, p.w_dtype, lane);
            }
            // key of this thread's score in a tile
            const int off = quad * 32 + scored_lane(lane);
            if constexpr (kStore) {
                // every tile of the row: its scores to the row's stored scores (a warp writes
                // 32 consecutive keys, one 128-byte line); the selection runs afterwards
                float* srow_t = p.scores + (static_cast<int64_t>(U.b) * (p.t_end - p.t_begin) +
                                            (t - p.t_begin)) * p.ld + U.key_lo + off;
                const int64_t rest64 = limit - U.key_lo - off;
                const int rest = rest64 < 0 ? 0 : rest64 > (1 << 30) ? (1 << 30)
                                                                     : static_cast<int>(rest64);
                for (int i = sub; i < U.ntiles; i += L::kSubs) {
                    const int acc = acc_base + i;
                    const int a = acc % L::kAccBufs;
                    tc::mbar_wait_ready(&tfull[a], (acc / L::kAccBufs) & 1, abort, p.err);
                    const float sc = tile_score<L::kN>(tmem, quad, r, a, tempty, wd);
                    if (i * kTileKeys < rest) srow_t[i * kTileKeys] = sc;
                }
                acc_base += U.ntiles;
                continue;
            }
            // Start from the row's admission threshold (its keys with a score at or above
            // tau), or from nothing: always for a row whose keys all fit the buffer (the
            // threshold launch may skip such rows).
            float tau = -__int_as_float(0x7f800000);
            if (p.tau_in && row_ok && n_row > L::kCap) tau = p.tau_in[row];
            const bool has_tau = tau > -__int_as_float(0x7f800000);
            sel.reset(has_tau ? static_cast<uint64_t>(score_order_bits(tau)) << 32 : 0ull);
            const uint32_t pos0 = static_cast<uint32_t>(U.key_lo + p.key_offset) + off;
            // keys of the row at or after this thread's key of tile 0 (tile i holds it at
            // 128 i): tile i's key belongs to the row when 128 i < rest
            int64_t rest64 = limit - U.key_lo - off;
            const int rest = rest64 < 0 ? 0 : rest64 > (1 << 30) ? (1 << 30) : static_cast<int>(rest64);
            int i0 = 0;
            if constexpr (kMode == kModeCapped && L::kSubs == 1) {
                // Rounds whose two tiles hold only keys of the row, for every thread: no bounds
                // checks (tile i is whole when (i + 1) * 128 <= limit - key_lo).
                int64_t nf64 = (limit - U.key_lo) / kTileKeys;
                const int n_full = nf64 < 0 ? 0 : nf64 > U.ntiles ? U.ntiles : static_cast<int>(nf64);
                for (; i0 + 2 <= n_full; i0 += 2) {
                    const unsigned acc_a = static_cast<unsigned>(acc_base + i0);
                    const unsigned acc_b = acc_a + 1u;
                    const int a_a = static_cast<int>(acc_a % L::kAccBufs);
                    const int a_b = static_cast<int>(acc_b % L::kAccBufs);
                    tc::mbar_wait_ready(&tfull[a_a], (acc_a / L::kAccBufs) & 1u, abort, p.err);
                    const float s_a = tile_score<L::kN>(tmem, quad, r, a_a, tempty, wd);
                    tc::mbar_wait_ready(&tfull[a_b], (acc_b / L::kAccBufs) & 1u, abort, p.err);
                    const float s_b = tile_score<L::kN>(tmem, quad, r, a_b, tempty, wd);
                    sel.offer2_capped(true, s_a, pos0 + static_cast<uint32_t>(i0 * kTileKeys),
                                      true, s_b, pos0 + static_cast<uint32_t>((i0 + 1) * kTileKeys),
                                      tau);
                }
            }
            // per round each warp scores two of its tiles and offers both keys at once (the
            // rest of the unit's tiles: bounds checked)
            for (; i0 < U.ntiles; i0 += 2 * L::kSubs) {
                const int ia = i0 + sub, ib = i0 + L::kSubs + sub;
                float sc[2] = {0.f, 0.f};
#pragma unroll
                for (int jj = 0; jj < 2; ++jj) {
                    const int i = jj ? ib : ia;
                    if (i < U.ntiles) {
                        const int acc = acc_base + i;
                        const int a = acc % L::kAccBufs;
                        tc::mbar_wait_ready(&tfull[a], (acc / L::kAccBufs) & 1, abort, p.err);
                        sc[jj] = tile_score<L::kN>(tmem, quad, r, a, tempty, wd);
                    }
                }
                const bool ok_a = ia * kTileKeys < rest, ok_b = ib * kTileKeys < rest;
                const uint32_t pa = pos0 + static_cast<uint32_t>(ia * kTileKeys);
                const uint32_t pb = pos0 + static_cast<uint32_t>(ib * kTileKeys);
                if constexpr (kMode == kModeCapped) {
                    sel.offer2_capped(ok_a, sc[0], pa, ok_b, sc[1], pb, tau);
                } else {
                    // Room for the round's offers: the row's warps meet once per round.  Each
                    // thread's count may miss the other warps' offers of the last round (at
                    // most 2 NT keys), and this round adds at most 2 NT more, so the trigger
                    // leaves 4 NT of room.  The row then settles its exact count and compacts.
                    if (tc::bar_red_or(1 + r, L::kGroupThreads, sel.count() > L::kTrigger)) {
                        const int held = sel.settled_count();
                        if (held > L::kTrigger)
                            sel.compact(p.topk, held, false, (L::kTrigger - p.topk) / 4);
                    }
                    const uint64_t thr = *reinterpret_cast<volatile uint64_t*>(sel.thr);
                    sel.offer2_scored(ok_a, sc[0], pa, ok_b, sc[1], pb, thr, score_floor(thr));
                }
            }
            acc_base += U.ntiles;
            bool short_row = false;
            if (row_ok) {
                const int held = sel.settled_count();
                const bool lost = held > L::kCap;  // capped: keys past the buffer were dropped
                if (p.tau_out) {
                    // Threshold launch: the topk-th largest sampled score bounds the row's
                    // admission in the full launch (at least topk of its keys reach it).  A row
                    // whose keys all fit the selector starts from nothing instead, and so does
                    // one whose sample did not fit (its full launch then overflows and the
                    // unit is redone from no threshold).
                    float out = -__int_as_float(0x7f800000);
                    const int64_t n_full = n_row << p.key_shift;  // upper bound of the row's keys
                    if (!lost && held > p.topk && n_full > L::kCap) {
                        if constexpr (kMode == kModeCapped) sel.keys_from_raw(held);
                        sel.compact(p.topk, held, true, 0, false);
                        out = score_floor(*reinterpret_cast<volatile uint64_t*>(sel.thr));
                    }
                    if (gtid == 0) p.tau_out[row] = out;
                    sel.sync();
                } else {
                    // Admission from a threshold may leave a row with fewer than k keys (fewer
                    // than min(k, its keys) at or above the threshold), or, capped, with more
                    // than the buffer holds: such a unit is done again from nothing by a later
                    // launch; its lists are not written here.
                    int64_t n_here = limit - U.key_lo;
                    if (n_here < 0) n_here = 0;
                    const int need = n_here < p.topk ? static_cast<int>(n_here) : p.topk;
                    short_row = lost || (has_tau && held < need);
                    if (!short_row) {
                        // the row's (chunk's) held keys, or its k best, unordered; the
                        // ranking or merge kernel takes them from there
                        const int64_t slot = row * p.n_chunks + U.chunk;
                        if constexpr (kMode == kModeCapped) {  // the buffer holds raw pairs
                            if (p.cand_stride) {
                                sel.dump_all_raw(p.cand + slot * p.cand_stride, p.cand_cnt + slot);
                            } else {
                                sel.keys_from_raw(held);
                                sel.dump(p.topk, p.cand + slot * p.topk, p.cand_cnt + slot);
                            }
                        } else if (p.cand_stride) {
                            sel.dump_all(p.cand + slot * p.cand_stride, p.cand_cnt + slot);
                        } else {
                            sel.dump(p.topk, p.cand + slot * p.topk, p.cand_cnt + slot);
                        }
                    }
                }
            }
            if (p.fail_list) {  // one barrier per unit: record it if any row came short
                if (tc::bar_red_or(kAllBar, 32 * kEpiWarps, short_row) && ew == 0 && lane == 0)
                    p.fail_list[atomicAdd(p.fail_count, 1)] = u;
            }
        }
    }
    tc::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
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

// Row-major [rows, 128 elements] tensor, boxes of box_rows rows x 128 bytes, 128-byte swizzle.
bool encode_rows128(CUtensorMap* map, const void* ptr, int64_t rows, int qk_dtype,
                    uint32_t box_rows = 128) {
    auto fn = encode_fn();
    if (!fn) return false;
    const bool bf16 = qk_dtype == TSI_BF16;
    cuuint64_t dims[2] = {128, static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(bf16 ? 256 : 128)};
    cuuint32_t box[2] = {bf16 ? 64u : 128u, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8, 2,
                    const_cast<void*>(ptr), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

constexpr int kPlanSMs = 152;

int rows_per_unit(int qk_dtype, int T) {
    return T == 1 ? 1 : qk_dtype == TSI_E4M3 ? TileCfg<TSI_E4M3>::kRows : TileCfg<TSI_BF16>::kRows;
}

// Key chunks per row for decode-sized requests (too few units to fill the GPU).
void tc_plan(int qk_dtype, int B, int T, int S, int* n_chunks, int* chunk_keys) {
    const int R = rows_per_unit(qk_dtype, T);
    const int64_t groups = static_cast<int64_t>(B) * ((T + R - 1) / R);
    int nc = 1;
    if (groups < kPlanSMs && S > 4096) {
        const int by_keys = (S + 2047) / 2048;
        const int by_sm = static_cast<int>((kPlanSMs + groups - 1) / groups);
        nc = by_keys < by_sm ? by_keys : by_sm;
        if (nc < 1) nc = 1;
    }
    int ck = (S + nc - 1) / nc;
    ck = (ck + kTileKeys - 1) / kTileKeys * kTileKeys;
    if (ck < kTileKeys) ck = kTileKeys;
    *n_chunks = nc;
    *chunk_keys = ck;
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

// Stored-score layout of the two-pass path: rows of ld floats (a multiple of 4, so that a
// row starts on 16 bytes), at most about kScoreScratch bytes per launch pair.
constexpr size_t kScoreScratch = size_t(8) << 30;

int64_t score_ld(int S) { return (static_cast<int64_t>(S) + 3) & ~int64_t(3); }

// Query rows per launch pair of the two-pass path: a multiple of R, all T when they fit.
int score_chunk_rows(int qk_dtype, int B, int T, int S) {
    const int R = rows_per_unit(qk_dtype, T);
    const int64_t per_row = static_cast<int64_t>(B) * score_ld(S) * 4;
    int64_t rows = per_row > 0 ? static_cast<int64_t>(kScoreScratch) / per_row : T;
    rows = rows / R * R;
    if (rows < R) rows = R;
    return rows >= T ? T : static_cast<int>(rows);
}

size_t score_scratch_bytes(int qk_dtype, int B, int T, int S) {
    if (rows_per_unit(qk_dtype, T) == 1) return 0;  // decode selects inside the kernel
    return static_cast<size_t>(B) * score_chunk_rows(qk_dtype, B, T, S) * score_ld(S) * 4;
}

// Candidate lists [slots][topk] (8 bytes a key) and their counts [slots] right after them;
// the size keeps whatever follows on a 16-byte boundary.
size_t cand_bytes(int B, int T, int topk, int n_chunks) {
    const size_t slots = static_cast<size_t>(B) * T * n_chunks;
    return ((slots * topk * sizeof(uint64_t) + 15) & ~size_t(15)) +
           ((slots * sizeof(int) + 255) & ~size_t(255));
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Selection from a sampled threshold: with several query rows per unit and one key range
// per row (no key chunks), the three select launches (see the top of the file) apply.
bool sampled_plan(int qk_dtype, int B, int T, int S) {
    if (rows_per_unit(qk_dtype, T) == 1) return false;
    int nc, ck;
    tc_plan(qk_dtype, B, T, S, &nc, &ck);
    return nc == 1;
}

int sample_keys(int S) { return (S + (1 << kSampleShift) - 1) >> kSampleShift; }

// Keys per candidate list of the sampled-threshold launches: the row selector's capacity.
int sampled_list_stride(int qk_dtype) {
    return qk_dtype == TSI_BF16 ? Lay<TSI_BF16, TileCfg<TSI_BF16>::kRows, kModeSelect>::kCap
                                : Lay<TSI_E4M3, TileCfg<TSI_E4M3>::kRows, kModeSelect>::kCap;
}

int64_t n_units_of(int qk_dtype, int B, int T) {
    const int R = rows_per_unit(qk_dtype, T);
    return static_cast<int64_t>(B) * ((T + R - 1) / R);
}

// Workspace of the sampled-threshold selection after the candidate lists: per-row
// thresholds, the short-unit count and list, the gathered key sample.
struct SampledWs {
    float* tau;
    int* fail_count;
    int* fail_list;
    uint8_t* keys;
    size_t bytes;
};

SampledWs sampled_ws(uint8_t* base, int qk_dtype, int B, int T, int S) {
    SampledWs w{};
    const size_t rows = static_cast<size_t>(B) * T;
    size_t off = 0;
    w.tau = reinterpret_cast<float*>(base + off);
    off = align_up(off + rows * 4, 256);
    w.fail_count = reinterpret_cast<int*>(base + off);
    off += 256;
    w.fail_list = reinterpret_cast<int*>(base + off);
    off = align_up(off + static_cast<size_t>(n_units_of(qk_dtype, B, T)) * 4, 1024);
    w.keys = base + off;
    off += align_up(static_cast<size_t>(B) * sample_keys(S) * (qk_dtype == TSI_BF16 ? 256 : 128),
                    1024);
    w.bytes = off;
    return w;
}

// Every 32nd key row (row bytes = 128 or 256) of each sequence into a buffer of its own,
// [B][ceil(S / 32)] rows; thread 0 also clears the short-unit count of the call.
__global__ void sample_keys_kernel(const uint4* __restrict__ kI, uint4* __restrict__ out, int B,
                                   int S, int S_s, int row_vec, int* fail_count) {
    const int64_t n = static_cast<int64_t>(B) * S_s * row_vec;
    const int64_t i0 = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (i0 == 0) *fail_count = 0;
    for (int64_t i = i0; i < n; i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t v = i % row_vec;
        const int64_t rs = i / row_vec;  // sampled row of the whole buffer
        const int64_t b = rs / S_s;
        const int64_t key = (rs - b * S_s) << kSampleShift;
        out[i] = kI[(b * S + key) * row_vec + v];
    }
}

// Target of the threshold launch: the row's ceil(c k / 32)-th largest sampled score, so that
// about c k keys of the row reach it.  c = 1.55: with 100 sampled keys above it for k = 2048
// the count of admitted keys varies by ~10% (the fraction of keys above the m-th of n
// sampled is Beta(m, n - m + 1)), so fewer than k (-3.5 sigma) or more than the 4352-key
// buffer (+3.7 sigma) happens to a few rows in 10^4; their units are redone exactly.
int sample_topk(int topk) {
    const int m = (155 * topk + 100 * (1 << kSampleShift) - 1) / (100 * (1 << kSampleShift));
    return m < 1 ? 1 : m;
}

template <int QK, int R, int kMode>
cudaError_t launch_qk(const IndexerArgs& a, void* workspace, cudaStream_t st) {
    using L = Lay<QK, R, kMode>;
    constexpr bool kStore = L::kStore;
    CUtensorMap tk, tq;
    // the query box is one unit's rows (64 per query row), at most 128 per copy
    if (!encode_rows128(&tk, a.kI, static_cast<int64_t>(a.B) * a.S, QK) ||
        !encode_rows128(&tq, a.qI, static_cast<int64_t>(a.B) * a.T * 64, QK,
                        L::kN < 128 ? L::kN : 128))
        return cudaErrorInvalidValue;
    TcParams p{};
    p.w = a.w;
    p.w_dtype = a.w_dtype;
    p.B = a.B;
    p.T = a.T;
    p.S = a.S;
    p.topk = a.topk;
    p.S_total = a.S_total ? a.S_total : a.S;
    p.key_offset = a.key_offset;
    p.kv_len = a.kv_len;
    p.idx = a.idx;
    p.score = a.score;
    p.err = a.err;
    p.q_raw = static_cast<const uint8_t*>(a.qI);
    p.q_row_bytes = QK == TSI_BF16 ? 256 : 128;
    p.w_bytes = a.w_dtype == TSI_BF16 ? 2 : 4;
    tc_plan(QK, a.B, a.T, a.S, &p.n_chunks, &p.chunk_keys);
    const int rows = a.B * a.T;
    // Candidate lists: the caller's (one list per row), else the workspace's (the fused
    // variant: one per key chunk).  The store variant ranks each row itself, or leaves it
    // unordered in the caller's lists, so its workspace holds the stored scores only.  The
    // sampled-threshold launches write each row's held keys to lists of the selector's
    // capacity, and the ranking kernel selects from them.
    const int lists = p.n_chunks;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    const bool wide = !kStore && R > 1 && lists == 1 && !a.out_cand;
    const int stride = wide ? L::kCap : a.topk;
    if ((kStore || lists == 1) && a.out_cand) {
        p.cand = a.out_cand;
        p.cand_cnt = a.out_cnt;
    } else if (!kStore) {
        p.cand = reinterpret_cast<uint64_t*>(ws);
        p.cand_cnt = reinterpret_cast<int*>(p.cand + static_cast<size_t>(rows) * lists * stride);
        p.cand_stride = wide ? stride : 0;
        ws += cand_bytes(a.B, a.T, stride, lists);
    }
    constexpr int smem = L::kSmem;
    cudaError_t e = cudaFuncSetAttribute(tsi_indexer_tc_kernel<QK, R, kMode>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    // the sampled-threshold launches run the capped form of the select kernel
    constexpr int kCapMode = kMode == kModeSelect ? kModeCapped : kMode;
    static_assert(Lay<QK, R, kCapMode>::kSmem == smem, "one layout for both select forms");
    if constexpr (kMode == kModeSelect && R > 1) {
        e = cudaFuncSetAttribute(tsi_indexer_tc_kernel<QK, R, kCapMode>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
    }
    const int chunk_rows = kStore ? score_chunk_rows(QK, a.B, a.T, a.S) : a.T;
    p.scores = kStore ? reinterpret_cast<float*>(ws) : nullptr;
    p.ld = score_ld(a.S);
    if constexpr (!kStore && R > 1) if (lists == 1) {
        // ---- selection from a sampled threshold: sample, threshold, full, short units
        const SampledWs sw = sampled_ws(ws, QK, a.B, a.T, a.S);
        const int S_s = sample_keys(a.S);
        const int row_vec = QK == TSI_BF16 ? 16 : 8;
        const int64_t n_vec = static_cast<int64_t>(a.B) * S_s * row_vec;
        int blocks = static_cast<int>((n_vec + 255) / 256);
        if (blocks > 4 * sm_count()) blocks = 4 * sm_count();
        if (blocks < 1) blocks = 1;
        sample_keys_kernel<<<blocks, 256, 0, st>>>(static_cast<const uint4*>(a.kI),
                                                     reinterpret_cast<uint4*>(sw.keys), a.B, a.S,
                                                     S_s, row_vec, sw.fail_count);
        note_launches(1);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        CUtensorMap ts;
        if (!encode_rows128(&ts, sw.keys, static_cast<int64_t>(a.B) * S_s, QK))
            return cudaErrorInvalidValue;
        p.t_begin = 0;
        p.t_end = a.T;
        p.n_units = static_cast<int>(n_units_of(QK, a.B, a.T));
        const int grid = p.n_units < sm_count() ? p.n_units : sm_count();
        // 1. thresholds from the sample, for the units (longest first) that hold a row with
        // more keys than the buffer: without per-sequence lengths they are the first B J
        // units, row group j having t_hi = T - 1 - R j; the full launch gives rows that fit
        // the buffer no threshold
        int64_t thr_units = p.n_units;
        if (!a.kv_len) {
            int64_t J = 0;
            for (;; ++J) {
                const int64_t t_hi = static_cast<int64_t>(a.T) - 1 - static_cast<int64_t>(R) * J;
                if (t_hi < 0) break;
                const int64_t pos = static_cast<int64_t>(p.S_total) - a.T + t_hi - a.key_offset;
                int64_t n = pos >= 0 ? (pos >> kSampleShift) + 1 : 0;
                if (n > S_s) n = S_s;
                if ((n << kSampleShift) <= L::kCap) break;
            }
            thr_units = static_cast<int64_t>(a.B) * J;
        }
        TcParams ps = p;
        ps.S = S_s;
        ps.key_shift = kSampleShift;
        ps.topk = sample_topk(a.topk);
        ps.tau_out = sw.tau;
        ps.n_units = static_cast<int>(thr_units);
        if (thr_units > 0) {
            const int grid_thr = thr_units < sm_count() ? static_cast<int>(thr_units) : sm_count();
            tsi_indexer_tc_kernel<QK, R, kCapMode><<<grid_thr, kThreads, smem, st>>>(ts, tq, ps);
            note_launches(1);
            if ((e = cudaGetLastError()) != cudaSuccess) return e;
        }
        // 2. every key, admitted from the thresholds; short units listed
        TcParams pf = p;
        pf.tau_in = sw.tau;
        pf.fail_list = sw.fail_list;
        pf.fail_count = sw.fail_count;
        tsi_indexer_tc_kernel<QK, R, kCapMode><<<grid, kThreads, smem, st>>>(tk, tq, pf);
        note_launches(1);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        // 3. the listed units again, from no threshold, with room checks (a launch whose
        // CTAs find no unit return at once)
        TcParams pr = p;
        pr.unit_list = sw.fail_list;
        pr.unit_count = sw.fail_count;
        tsi_indexer_tc_kernel<QK, R, kMode><<<grid, kThreads, smem, st>>>(tk, tq, pr);
        note_launches(1);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        return a.out_cand ? e
                          : launch_topk_rank(rows, a.topk, stride, p.cand, p.cand_cnt, a.idx,
                                             a.score, a.err, st);
    }
    // Launch pairs over chunks of query rows, the last rows first (each chunk's rows are
    // a multiple of R except the first rows of the sequences).
    for (int t_end = a.T; t_end > 0; t_end -= chunk_rows) {
        p.t_end = t_end;
        p.t_begin = t_end > chunk_rows ? t_end - chunk_rows : 0;
        const int n = p.t_end - p.t_begin;
        p.n_units = static_cast<int>(static_cast<int64_t>(a.B) * ((n + R - 1) / R) * p.n_chunks);
        const int grid = p.n_units < sm_count() ? p.n_units : sm_count();
        tsi_indexer_tc_kernel<QK, R, kMode><<<grid, kThreads, smem, st>>>(tk, tq, p);
        note_launches(1);
        e = cudaGetLastError();
        if (e != cudaSuccess || !kStore) break;
        ScoreRows sr{};
        sr.scores = p.scores;
        sr.ld = p.ld;
        sr.B = a.B;
        sr.T = a.T;
        sr.S = a.S;
        sr.S_total = p.S_total;
        sr.topk = a.topk;
        sr.t0 = p.t_begin;
        sr.rows = n;
        sr.key_offset = a.key_offset;
        sr.kv_len = a.kv_len;
        sr.idx = a.out_cand ? nullptr : a.idx;
        sr.score = a.out_cand ? nullptr : a.score;
        sr.cand = p.cand;
        sr.cand_cnt = p.cand_cnt;
        sr.err = a.err;
        e = launch_topk_rows(sr, st);
        if (e != cudaSuccess) break;
    }
    if (e != cudaSuccess || kStore) return e;
    if (lists == 1)
        return a.out_cand ? e
                          : launch_topk_rank(rows, a.topk, stride, p.cand, p.cand_cnt, a.idx,
                                             a.score, a.err, st);
    // decode: the chunk lists of few rows are merged in two stages (stage space after them)
    void* stage = reinterpret_cast<uint8_t*>(p.cand_cnt) +
                  ((static_cast<size_t>(rows) * p.n_chunks * sizeof(int) + 255) & ~size_t(255));
    return launch_topk_merge_two_stage(rows, a.topk, p.n_chunks, p.cand,
                                       static_cast<int64_t>(p.n_chunks) * a.topk, a.topk,
                                       p.cand_cnt, p.n_chunks, 1, stage, a.idx, a.score,
                                       a.out_cand, a.out_cnt, a.err, st);
}

}  // namespace

bool tc_indexer_supported(int qk_dtype, int H_I, int d_I) {
    return (qk_dtype == TSI_BF16 || qk_dtype == TSI_E4M3) && H_I == 64 && d_I == 128;
}

size_t tc_indexer_workspace_bytes(int qk_dtype, int B, int T, int S, int topk, bool two_pass) {
    if (rows_per_unit(qk_dtype, T) > 1 && two_pass)  // two passes: the stored scores
        return score_scratch_bytes(qk_dtype, B, T, S);
    int nc, ck;
    tc_plan(qk_dtype, B, T, S, &nc, &ck);
    // the sampled-threshold launches keep each row's held keys (lists of the selector's
    // capacity); the others each row's or chunk's k best
    const bool sampled = sampled_plan(qk_dtype, B, T, S);
    const int stride = sampled ? sampled_list_stride(qk_dtype) : topk;
    size_t n = cand_bytes(B, T, stride, nc) +
               (nc > 1 ? topk_merge_stage_bytes(B * T, topk, nc) : 0);
    if (sampled) n += sampled_ws(nullptr, qk_dtype, B, T, S).bytes;
    return n;
}

size_t tc_indexer_split_workspace_bytes(int qk_dtype, int B, int T, int S, int topk) {
    // the caller's lists take the candidates of a one-list-per-row launch; what remains is
    // the sampled selection's scratch, or the chunk lists and their merge stage
    int nc, ck;
    tc_plan(qk_dtype, B, T, S, &nc, &ck);
    if (sampled_plan(qk_dtype, B, T, S)) return sampled_ws(nullptr, qk_dtype, B, T, S).bytes;
    return nc <= 1 ? 0 : tc_indexer_workspace_bytes(qk_dtype, B, T, S, topk, false);
}

cudaError_t launch_indexer_tc(const IndexerArgs& a, void* workspace, cudaStream_t st) {
    if (a.B * a.T == 0) return cudaSuccess;
    if (rows_per_unit(a.qk_dtype, a.T) == 1)
        return a.qk_dtype == TSI_E4M3 ? launch_qk<TSI_E4M3, 1, kModeSelect>(a, workspace, st)
                                      : launch_qk<TSI_BF16, 1, kModeSelect>(a, workspace, st);
    if (a.two_pass)
        return a.qk_dtype == TSI_E4M3
                   ? launch_qk<TSI_E4M3, TileCfg<TSI_E4M3>::kRows, kModeStore>(a, workspace, st)
                   : launch_qk<TSI_BF16, TileCfg<TSI_BF16>::kRows, kModeStore>(a, workspace, st);
    return a.qk_dtype == TSI_E4M3
               ? launch_qk<TSI_E4M3, TileCfg<TSI_E4M3>::kRows, kModeSelect>(a, workspace, st)
               : launch_qk<TSI_BF16, TileCfg<TSI_BF16>::kRows, kModeSelect>(a, workspace, st);
}

}  // namespace tsi
