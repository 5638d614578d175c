// Tensor-core lightning indexer for sm_103a (tcgen05 / TMEM / TMA).
//
// I[t,s] = sum_j w[t,j] * ReLU(qI[t,j] . kI[s]) for s <= p_t, then the top-k keys of
// each row ("GLM-5.2 技术报告速览", §IndexShare: the score equation, k = 2048; the
// ReLU form is chosen there for speed and FP8 friendliness).  Two variants of one kernel:
//   - store (the default for several query rows per sequence): every causal score goes
//     to a row-major fp32 buffer, a chunk of query rows at a time; topk_rows.cu then
//     selects and ranks each row's k best keys from it.  The selection thus never stalls
//     the MMA pipeline, at 4 B of HBM writes per causal pair.
//   - select (one query row per sequence, and any launch asked to keep its scores on
//     chip): each 128-key tile is scored in TMEM and streamed into a shared-memory top-k
//     selector per query row, so no score reaches HBM; each row (or key chunk) leaves its
//     k best keys unordered, for the ranking or merge kernels.
//
// MMA shape: keys on M (128 rows of kI per tile, the A operand), the 64 heads of R
// consecutive query rows on N = 64 R (the B operand), d_I = 128 on K, fp32 accumulators
// in TMEM.  R = 4 for e4m3 (N = 256), 2 for bf16 (N = 128), 1 for decode.  The larger R,
// the more query rows share each key tile: fewer tiles, MMA issues and barrier round
// trips, less L2 traffic.  An epilogue warp reads its 32 TMEM lanes (keys) in the
// 16x256b shape (see tile_score): each thread sums 16 heads of two keys, four threads
// combine their sums with two shuffles.
//
// Roles of one persistent CTA (576 threads):
//   warp 0       TMA producer: Q tile of the unit, key tiles into a ring of stages
//   warp 1       TMEM allocator + single-thread MMA issuer (512 TMEM columns: 512 / N
//                accumulators, so the MMA runs that many tiles ahead)
//   warps 2..17  R epilogue groups of 16 / R warps, one per query row of the unit; group
//                r reads columns [64r, 64r+64) of an accumulator (and, selecting, owns a
//                selector).  With 16 / R > 4 warps per row, the row's warp sets share out
//                the tiles.
// Units (R consecutive query rows x one key range) are visited longest first and spread
// round-robin over the CTAs.
#include <mutex>

#include <cudaTypedefs.h>

#include "kernels_tc.cuh"
#include "tc_common.cuh"
#include "topk_select.cuh"

namespace tsi {
namespace {

constexpr int kTileKeys = 128;  // MMA M
constexpr int kEpiWarps = 16;
constexpr int kThreads = 64 + 32 * kEpiWarps;
constexpr int kTmemCols = 512;
constexpr int kChunkBytes = 128 * 128;  // one 128-row x 128-byte swizzled tile
constexpr int kAllBar = 8;  // named barrier of all epilogue warps (selectors use 1..4)

template <int QK>
struct TileCfg;
template <>
struct TileCfg<TSI_E4M3> {
    static constexpr int kRows = 4;    // query rows per unit
    static constexpr int kCap = 3584;  // selector capacity per row (on-chip selection)
    static constexpr int kChunks = 1;  // 128-byte pieces of a d_I = 128 row
    static constexpr int kStages = 4;
    static constexpr uint32_t kFmt = 0;
    static constexpr int kKSteps = 4;  // K = 32 per MMA
};
template <>
struct TileCfg<TSI_BF16> {
    static constexpr int kRows = 2;
    static constexpr int kCap = 4096;
    static constexpr int kChunks = 2;
    static constexpr int kStages = 3;
    static constexpr uint32_t kFmt = 1;
    static constexpr int kKSteps = 4;  // per chunk, K = 16 per MMA
};

// R = query rows per unit: the format's default, or 1 for one query per sequence (decode),
// where the four warp sets of the single row share out the key tiles instead of idling.
// kStore: the epilogue stores the scores; otherwise it selects each row's top k itself.
template <int QK, int R = TileCfg<QK>::kRows, bool kStore = false>
struct Lay {
    using C = TileCfg<QK>;
    static constexpr int kR = R;
    // selector capacity: the row's warp sets offer up to 4 kGroupThreads keys between two
    // room checks (see the trigger in the epilogue), beyond the k that are kept
    static constexpr int kCap = R == 1 ? 5120 : C::kCap;
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
    static constexpr int kBars = 2 * C::kStages + 2 * kAccBufs + 3;
    static constexpr int kSmem = 1024 /* alignment slack */ + C::kStages * kStageBytes +
                                 kQBytes + kR * kSelBytes + kBars * 8 + 16;
    static_assert(kSmem <= 227 * 1024, "shared memory");
    static_assert(kEpiWarps == 4 * kR * kSubs, "every epilogue warp has a row");
};

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
    int n_chunks, chunk_keys, n_units;
    int t_begin, t_end;  // query rows [t_begin, t_end) of every sequence in this launch
    float* scores;       // store variant: row (b, t) at (b * (t_end - t_begin) + t - t_begin) * ld
    int64_t ld;
    unsigned* err;
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
    int64_t end = p_hi + 1 > 0 ? p_hi + 1 : 0;
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

// 2 ReLU(x) of two accumulator words as x + |x|: exact (2x for x > 0, +0 otherwise), and an
// add on the FMA pipe instead of a max on the half-rate ALU pipe.  The gate weights are
// halved to match, so w/2 * (x + |x|) is exactly the product w * ReLU(x).
__device__ __forceinline__ float2 relu2_twice(uint32_t a, uint32_t b) {
    const float x = __uint_as_float(a), y = __uint_as_float(b);
    return make_float2(__fadd_rn(x, fabsf(x)), __fadd_rn(y, fabsf(y)));
}

// Key lane (within the warp's 32 TMEM lanes) whose score tile_score returns to this
// thread: lane 8 (T % 4) + T / 4 of thread T.
__device__ __forceinline__ int scored_lane(int lane) { return 8 * (lane & 3) + (lane >> 2); }

// Scores of query row r of the unit from accumulator buffer a: sum over the 64 heads of
// w[h] * max(0, q[h].k), in packed fp32 pairs (w2 holds w / 2, see relu2_twice).
//
// The warp reads its 32 TMEM lanes (keys) as two 16-lane slices of the row's 64 columns
// (16x256b shape).  Thread T then holds, for two keys, the head pairs 8m + 2c + {0, 1}
// (c = T % 4, m = 0..7), so it needs only those 16 gate weights -- w2[m], kept in
// registers for the whole unit instead of being re-read from shared memory for every
// tile.  The four threads with equal T / 4 add their partial sums with two butterfly
// shuffles (every one of them ends with the same value).  Thread T returns the score of
// key lane scored_lane(T).  The buffer is released to the MMA once the second slice is in
// registers.
template <int N>
__device__ __forceinline__ float tile_score(uint32_t tmem, int quad, int r, int a, uint64_t* tempty,
                                            const float2 (&w2)[8]) {
    tc::tc_fence_after();
    const int c = threadIdx.x & 3;
    const uint32_t taddr = tmem + (static_cast<uint32_t>(quad * 32) << 16) + a * N + r * 64;
    float mine = 0.f;
#pragma unroll
    for (int slice = 0; slice < 2; ++slice) {
        uint32_t v[32];
        TSI_TMEM_LD16x256_X8(taddr + (static_cast<uint32_t>(16 * slice) << 16), v);
        tc::tmem_wait_ld();
        if (slice == 1) {
            tc::tc_fence_before();
            __syncwarp();
            if ((threadIdx.x & 31) == 0) tc::mbar_arrive(&tempty[a]);
        }
        // two accumulators per key for a shorter dependency chain
        float2 a0 = make_float2(0.f, 0.f), a1 = a0, b0 = a0, b1 = a0;
#pragma unroll
        for (int m = 0; m < 8; m += 2) {
            a0 = __ffma2_rn(w2[m], relu2_twice(v[4 * m + 0], v[4 * m + 1]), a0);
            b0 = __ffma2_rn(w2[m], relu2_twice(v[4 * m + 2], v[4 * m + 3]), b0);
            a1 = __ffma2_rn(w2[m + 1], relu2_twice(v[4 * m + 4], v[4 * m + 5]), a1);
            b1 = __ffma2_rn(w2[m + 1], relu2_twice(v[4 * m + 6], v[4 * m + 7]), b1);
        }
        float sa = (a0.x + a0.y) + (a1.x + a1.y);  // key lane 16 slice + T / 4
        float sb = (b0.x + b0.y) + (b1.x + b1.y);  // key lane 16 slice + 8 + T / 4
        sa += __shfl_xor_sync(0xFFFFFFFFu, sa, 1);
        sb += __shfl_xor_sync(0xFFFFFFFFu, sb, 1);
        sa += __shfl_xor_sync(0xFFFFFFFFu, sa, 2);
        sb += __shfl_xor_sync(0xFFFFFFFFu, sb, 2);
        if (c == 2 * slice) mine = sa;
        if (c == 2 * slice + 1) mine = sb;
    }
    return mine;
}

template <int QK, int R, bool kStore>
__global__ void __launch_bounds__(kThreads, 1)
    tsi_indexer_tc_kernel(const __grid_constant__ CUtensorMap tmap_k,
                          const __grid_constant__ CUtensorMap tmap_q, const TcParams p) {
    using C = TileCfg<QK>;
    using L = Lay<QK, R, kStore>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* stages = base;
    uint8_t* qbuf = stages + C::kStages * L::kStageBytes;
    uint8_t* sel_mem = qbuf + L::kQBytes;
    uint64_t* bars = reinterpret_cast<uint64_t*>(sel_mem + R * L::kSelBytes);
    uint64_t* full = bars;
    uint64_t* empty = full + C::kStages;
    uint64_t* tfull = empty + C::kStages;
    uint64_t* tempty = tfull + L::kAccBufs;
    uint64_t* qfull = tempty + L::kAccBufs;
    uint64_t* qempty = qfull + 1;
    uint64_t* done = qempty + 1;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);
    volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::kStages; ++s) {
            tc::mbar_init(&full[s], 1);
            tc::mbar_init(&empty[s], 1);
        }
        for (int a = 0; a < L::kAccBufs; ++a) {
            tc::mbar_init(&tfull[a], 1);
            tc::mbar_init(&tempty[a], L::kReaders);
        }
        tc::mbar_init(qfull, 1);
        tc::mbar_init(qempty, 1);
        tc::mbar_init(done, 1);
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

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            int s = 0;
            uint32_t ph = 0;  // phase of the ring slot s
            int unit_it = 0;
            int q_last = -1;  // unit of the last query load issued
            uint32_t loaded = 0, last_ph = 0;  // per slot (bit s): loaded once, last phase
            for (int u = blockIdx.x; u < p.n_units; u += gridDim.x, ++unit_it) {
                const Unit U = unit_of<R>(p, u);
                tc::mbar_wait(qempty, (unit_it & 1) ^ 1, abort, p.err);
                if (!*abort) {
                    q_last = unit_it;
                    tc::mbar_expect_tx(qfull, L::kQBytes);
                    const int qrow = (U.b * p.T + U.t_hi - (R - 1)) * 64;
                    for (int c = 0; c < C::kChunks; ++c)
                        for (int h = 0; h < L::kN; h += 128)
                            tc::tma_load_2d(qbuf + c * L::kQChunkBytes + h * 128, &tmap_q, c * 64,
                                            qrow + h, qfull);
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
                    if (++s == C::kStages) {
                        s = 0;
                        ph ^= 1;
                    }
                }
            }
            if (*abort) {  // loads still in flight must land before the CTA exits (at most
                           // one per slot: a slot is reloaded only after its data was used)
                if (q_last >= 0) tc::mbar_drain(qfull, q_last & 1);
                for (int i = 0; i < C::kStages; ++i)
                    if ((loaded >> i) & 1u) tc::mbar_drain(&full[i], (last_ph >> i) & 1u);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            int s = 0, a = 0;
            uint32_t ph = 0, aph = 0;  // phases of ring slot s and accumulator a
            int unit_it = 0;
            const uint64_t adesc = tc::smem_desc(tc::smem_addr(stages), 16, 1024);
            const uint64_t bdesc = tc::smem_desc(tc::smem_addr(qbuf), 16, 1024);
            for (int u = blockIdx.x; u < p.n_units; u += gridDim.x, ++unit_it) {
                const Unit U = unit_of<R>(p, u);
                tc::mbar_wait(qfull, unit_it & 1, abort, p.err);
                for (int i = 0; i < U.ntiles; ++i) {
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
                                if (QK == TSI_E4M3)
                                    tc::mma_f8(d, da, db, L::kIdesc, accum);
                                else
                                    tc::mma_bf16(d, da, db, L::kIdesc, accum);
                            }
                        }
                    }
                    tc::mma_commit(&empty[s]);
                    tc::mma_commit(&tfull[a]);
                    if (++s == C::kStages) {
                        s = 0;
                        ph ^= 1;
                    }
                    if (++a == L::kAccBufs) {
                        a = 0;
                        aph ^= 1;
                    }
                }
                tc::mma_commit(qempty);
            }
            // every MMA issued by this thread has finished before TMEM is released
            tc::mma_commit(done);
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
        for (int u = blockIdx.x; u < p.n_units; u += gridDim.x) {
            const Unit U = unit_of<R>(p, u);
            const int t = U.t_hi - (R - 1) + r;
            const bool row_ok = t >= p.t_begin;
            int64_t limit = 0;  // keys s < limit belong to this row
            float2 w2[8];
#pragma unroll
            for (int m = 0; m < 8; ++m) w2[m] = make_float2(0.f, 0.f);
            if (row_ok) {
                const int64_t pr = query_position(p.kv_len, U.b, p.T, p.S_total, t) - p.key_offset;
                limit = pr + 1 < U.key_hi ? pr + 1 : U.key_hi;
                const int64_t wrow = (static_cast<int64_t>(U.b) * p.T + t) * 64;
                // this thread's 16 gate weights, halved (see tile_score, relu2_twice)
#pragma unroll
                for (int m = 0; m < 8; ++m) {
                    const int64_t h = wrow + 8 * m + 2 * (lane & 3);
                    w2[m] = make_float2(0.5f * load_elem(p.w, h, p.w_dtype),
                                        0.5f * load_elem(p.w, h + 1, p.w_dtype));
                }
            }
            // key of this thread's score in a tile: off; whole-cache position of key 0
            const int off = quad * 32 + scored_lane(lane);
            if constexpr (kStore) {
                // every tile of the row: its scores to the row's stored scores (a warp writes
                // 32 consecutive keys, one 128-byte line); the selection runs afterwards
                float* srow = p.scores + (static_cast<int64_t>(U.b) * (p.t_end - p.t_begin) +
                                          (t - p.t_begin)) * p.ld;
                for (int i = sub; i < U.ntiles; i += L::kSubs) {
                    const int acc = acc_base + i;
                    const int a = acc % L::kAccBufs;
                    tc::mbar_wait(&tfull[a], (acc / L::kAccBufs) & 1, abort, p.err);
                    const float sc = tile_score<L::kN>(tmem, quad, r, a, tempty, w2);
                    const int64_t key = U.key_lo + static_cast<int64_t>(i) * kTileKeys + off;
                    if (key < limit) srow[key] = sc;
                }
                acc_base += U.ntiles;
                continue;
            }
            // per round each warp scores two of its tiles, then one room check covers the
            // group's offers of both
            sel.reset();
            const uint32_t pos0 = static_cast<uint32_t>(U.key_lo + p.key_offset);
            for (int i0 = 0; i0 < U.ntiles; i0 += 2 * L::kSubs) {
                float sc[2];
                int rem[2];  // keys of tile i that belong to this row (0..128)
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    const int i = i0 + j * L::kSubs + sub;
                    const int64_t left = limit - (U.key_lo + static_cast<int64_t>(i) * kTileKeys);
                    rem[j] = left <= 0 ? 0 : left >= kTileKeys ? kTileKeys : static_cast<int>(left);
                    sc[j] = 0.f;
                    if (i < U.ntiles) {
                        const int acc = acc_base + i;
                        const int a = acc % L::kAccBufs;
                        tc::mbar_wait(&tfull[a], (acc / L::kAccBufs) & 1, abort, p.err);
                        sc[j] = tile_score<L::kN>(tmem, quad, r, a, tempty, w2);
                    }
                }
                // Room for the round's offers.  All epilogue warps meet here (they wait for
                // the same accumulators anyway): when some row is about to fill, every row
                // past half full compacts in the same stall of the MMA pipeline instead of
                // each stalling it on its own.
                // One barrier: each thread's count may miss the other warps' offers of the
                // last round (at most 2 NT keys), and this round adds at most 2 NT more, so
                // the trigger leaves 4 NT of room.  The rows then settle their exact counts.
                constexpr int kTrigger = L::kCap - 4 * L::kGroupThreads;
                if (tc::bar_red_or(kAllBar, 32 * kEpiWarps, sel.count() > kTrigger)) {
                    const int held = sel.settled_count();
                    if (held > (p.topk + kTrigger) / 2)
                        sel.compact(p.topk, held, false, (kTrigger - p.topk) / 4);
                }
                const uint64_t thr = *reinterpret_cast<volatile uint64_t*>(sel.thr);
                const uint32_t i_a = static_cast<uint32_t>((i0 + sub) * kTileKeys + off);
                const uint32_t i_b = static_cast<uint32_t>((i0 + L::kSubs + sub) * kTileKeys + off);
                sel.offer2_scored(off < rem[0], sc[0], pos0 + i_a, off < rem[1], sc[1], pos0 + i_b,
                                  thr, score_floor(thr));
            }
            acc_base += U.ntiles;
            if (row_ok) {
                // the row's (chunk's) k best keys, unordered; the merge kernel ranks them
                const int64_t row = static_cast<int64_t>(U.b) * p.T + t;
                const int64_t slot = row * p.n_chunks + U.chunk;
                sel.dump(p.topk, p.cand + slot * p.topk, p.cand_cnt + slot);
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

template <int QK, int R, bool kStore>
cudaError_t launch_qk(const IndexerArgs& a, void* workspace, cudaStream_t st) {
    using L = Lay<QK, R, kStore>;
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
    tc_plan(QK, a.B, a.T, a.S, &p.n_chunks, &p.chunk_keys);
    const int rows = a.B * a.T;
    // Candidate lists: the caller's (one list per row), else the workspace's (the fused
    // variant: one per key chunk).  The store variant ranks each row itself, or leaves it
    // unordered in the caller's lists, so its workspace holds the stored scores only.
    const int lists = p.n_chunks;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    if ((kStore || lists == 1) && a.out_cand) {
        p.cand = a.out_cand;
        p.cand_cnt = a.out_cnt;
    } else if (!kStore) {
        p.cand = reinterpret_cast<uint64_t*>(ws);
        p.cand_cnt = reinterpret_cast<int*>(p.cand + static_cast<size_t>(rows) * lists * a.topk);
        ws += cand_bytes(a.B, a.T, a.topk, lists);
    }
    constexpr int smem = L::kSmem;
    cudaError_t e = cudaFuncSetAttribute(tsi_indexer_tc_kernel<QK, R, kStore>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    const int chunk_rows = kStore ? score_chunk_rows(QK, a.B, a.T, a.S) : a.T;
    p.scores = kStore ? reinterpret_cast<float*>(ws) : nullptr;
    p.ld = score_ld(a.S);
    // Launch pairs over chunks of query rows, the last rows first (each chunk's rows are
    // a multiple of R except the first rows of the sequences).
    for (int t_end = a.T; t_end > 0; t_end -= chunk_rows) {
        p.t_end = t_end;
        p.t_begin = t_end > chunk_rows ? t_end - chunk_rows : 0;
        const int n = p.t_end - p.t_begin;
        p.n_units = static_cast<int>(static_cast<int64_t>(a.B) * ((n + R - 1) / R) * p.n_chunks);
        const int grid = p.n_units < sm_count() ? p.n_units : sm_count();
        tsi_indexer_tc_kernel<QK, R, kStore><<<grid, kThreads, smem, st>>>(tk, tq, p);
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
                          : launch_topk_rank(rows, a.topk, p.cand, p.cand_cnt, a.idx, a.score,
                                             a.err, st);
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

size_t tc_indexer_workspace_bytes(int qk_dtype, int B, int T, int S, int topk, bool onchip) {
    if (rows_per_unit(qk_dtype, T) > 1 && !onchip)  // two passes: the stored scores
        return score_scratch_bytes(qk_dtype, B, T, S);
    int nc, ck;
    tc_plan(qk_dtype, B, T, S, &nc, &ck);
    return cand_bytes(B, T, topk, nc) +
           (nc > 1 ? topk_merge_stage_bytes(B * T, topk, nc) : 0);
}

size_t tc_indexer_split_workspace_bytes(int qk_dtype, int B, int T, int S, int topk) {
    // the caller's lists take the candidates of a one-list-per-row launch
    if (rows_per_unit(qk_dtype, T) > 1) return score_scratch_bytes(qk_dtype, B, T, S);
    int nc, ck;
    tc_plan(qk_dtype, B, T, S, &nc, &ck);
    return nc <= 1 ? 0 : tc_indexer_workspace_bytes(qk_dtype, B, T, S, topk, false);
}

cudaError_t launch_indexer_tc(const IndexerArgs& a, void* workspace, cudaStream_t st) {
    if (a.B * a.T == 0) return cudaSuccess;
    if (rows_per_unit(a.qk_dtype, a.T) == 1)
        return a.qk_dtype == TSI_E4M3 ? launch_qk<TSI_E4M3, 1, false>(a, workspace, st)
                                      : launch_qk<TSI_BF16, 1, false>(a, workspace, st);
    if (a.onchip)
        return a.qk_dtype == TSI_E4M3
                   ? launch_qk<TSI_E4M3, TileCfg<TSI_E4M3>::kRows, false>(a, workspace, st)
                   : launch_qk<TSI_BF16, TileCfg<TSI_BF16>::kRows, false>(a, workspace, st);
    return a.qk_dtype == TSI_E4M3
               ? launch_qk<TSI_E4M3, TileCfg<TSI_E4M3>::kRows, true>(a, workspace, st)
               : launch_qk<TSI_BF16, TileCfg<TSI_BF16>::kRows, true>(a, workspace, st);
}

}  // namespace tsi
