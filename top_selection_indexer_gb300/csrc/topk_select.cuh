// Streaming exact top-k selection in shared memory.
//
// Every candidate is a 64-bit key  (order(score) << 32) | (0xFFFFFFFF - s):  the upper
// word orders fp32 scores as unsigned integers (-0.0 folded onto +0.0), the lower word
// makes a lower key position compare higher.  Keys are therefore unique and their
// unsigned order is exactly the rank order "higher score first, equal scores by lower
// position" (the deterministic top-k that "GLM-5: from Vibe Coding to Agentic
// Engineering" (Chinese translation) §3.2 asks for, with the lower-index tie rule).
//
// A group of NT threads owns one selector: a buffer of CAP keys, an admission
// threshold `thr` and a 256-bin histogram.  (The capped offers append raw (score bits,
// position) pairs instead, turned into keys in one pass before anything compares them.)  Keys >= thr are appended; when the buffer
// is nearly full a radix select over the key bits finds the bound T with exactly k
// keys >= T, drops the rest and raises thr to T.  Invariant: every dropped key is
// smaller than k kept keys, so the buffer always holds the top k of all offered keys.
#pragma once

#include "tsi_common.cuh"

namespace tsi {

__device__ __forceinline__ uint32_t score_order_bits(float x) {
    uint32_t u = __float_as_uint(x);
    if (u == 0x80000000u) u = 0u;  // -0.0 ranks as +0.0
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float order_bits_score(uint32_t o) {
    uint32_t u = (o & 0x80000000u) ? (o & 0x7FFFFFFFu) : ~o;
    return __uint_as_float(u);
}

__device__ __forceinline__ uint64_t make_key(float score, uint32_t s) {
    return (static_cast<uint64_t>(score_order_bits(score)) << 32) |
           static_cast<uint64_t>(0xFFFFFFFFu - s);
}

// A candidate before it becomes a key: the score's bits above the position.  The capped
// offers store these (one move, no arithmetic on the scoring path) and the buffer is turned
// into keys once, when the unit ends.
__device__ __forceinline__ uint64_t raw_pair(float score, uint32_t s) {
    return (static_cast<uint64_t>(__float_as_uint(score)) << 32) | static_cast<uint64_t>(s);
}

__device__ __forceinline__ uint64_t key_of_raw(uint64_t r) {
    return make_key(__uint_as_float(static_cast<uint32_t>(r >> 32)), static_cast<uint32_t>(r));
}

// The smallest fp32 score whose keys can reach `threshold`: a finite score x has
// make_key(x, s) >= threshold for some s exactly when x >= score_floor(threshold) (the
// order is monotone in the score, -0.0 and +0.0 alike).  Thresholds whose score word lies
// below every real score give -inf.
__device__ __forceinline__ float score_floor(uint64_t threshold) {
    const uint32_t o = static_cast<uint32_t>(threshold >> 32);
    return o < 0x00800000u ? -__int_as_float(0x7f800000) : order_bits_score(o);
}

__device__ __forceinline__ int32_t key_position(uint64_t key) {
    return static_cast<int32_t>(0xFFFFFFFFu - static_cast<uint32_t>(key));
}

__device__ __forceinline__ float key_score(uint64_t key) {
    return order_bits_score(static_cast<uint32_t>(key >> 32));
}

// Shared-memory footprint of one selector (bytes), excluding alignment slack.
template <int CAP>
constexpr int selector_smem_bytes() {
    return CAP * 8 + 256 * 4 + 8 * 4 + 8 + 16;
}

template <int NT, int CAP>
struct TopKSelector {
    static_assert(NT % 32 == 0, "whole warps");
    static_assert(CAP % NT == 0, "CAP must be a multiple of NT");
    static_assert(CAP >= TSI_MAX_TOPK + 2 * NT, "room for k keys plus two rounds");

    uint64_t* buf;   // [CAP]
    unsigned* hist;  // [256]
    int* ctl;        // [8]: 0 count, 1 digit, 2 above, 3 in-bin, 4 write cursor
    uint64_t* thr;   // admission threshold
    uint64_t* rng;   // [2]: largest and smallest held key, during a compaction
    int tid;         // 0..NT-1 within the group
    int bar_id;      // named barrier of the group
    unsigned* err;   // device error word: consistency checks record kErrAssert here

    // Carve the selector out of `smem` (8-byte aligned); returns the bytes used.
    __device__ int bind(uint8_t* smem, int tid_, int bar_id_, unsigned* err_) {
        err = err_;
        buf = reinterpret_cast<uint64_t*>(smem);
        hist = reinterpret_cast<unsigned*>(smem + CAP * 8);
        ctl = reinterpret_cast<int*>(smem + CAP * 8 + 256 * 4);
        thr = reinterpret_cast<uint64_t*>(smem + CAP * 8 + 256 * 4 + 8 * 4);
        rng = thr + 1;
        tid = tid_;
        bar_id = bar_id_;
        return selector_smem_bytes<CAP>();
    }

    __device__ __forceinline__ void sync() const { named_bar(bar_id, NT); }

    __device__ __forceinline__ int count() const {
        return *reinterpret_cast<volatile int*>(&ctl[0]);
    }

    // Collective: empty the selector; keys below `threshold` are never admitted.
    __device__ void reset(uint64_t threshold = 0ull) {
        sync();
        if (tid == 0) {
            ctl[0] = 0;
            ctl[4] = 0;
            *thr = threshold;
            rng[0] = 0ull;
            rng[1] = ~0ull;
        }
        for (int i = tid; i < 256; i += NT) hist[i] = 0u;
        sync();
    }

    // Collective over the NT threads: each thread may carry one key.  The caller has
    // made room (count() + NT <= CAP) with make_room().
    __device__ __forceinline__ void offer(bool has, uint64_t key) {
        const int lane = threadIdx.x & 31;
        const bool take = has && key >= *thr;
        const unsigned m = __ballot_sync(kFull, take);
        if (m) {
            const int leader = __ffs(m) - 1;
            int base = 0;
            if (lane == leader) base = atomicAdd(&ctl[0], __popc(m));
            base = __shfl_sync(kFull, base, leader);
            const int pos = base + __popc(m & ((1u << lane) - 1u));
            if (take) {
                if (pos < CAP)
                    buf[pos] = key;
                else
                    atomicOr(err, kErrAssert);
            }
        }
    }

    // Collective: the held count, read by every thread of the group.  The second barrier
    // keeps any thread from offering (and bumping the count) before all have read it, so
    // every thread takes the same branch on the value.
    __device__ __forceinline__ int settled_count() {
        sync();
        const int n = count();
        sync();
        return n;
    }

    // Collective: ensure room for `rounds` more rounds of NT offers.  Returns the admission
    // threshold to offer against until the next make_room (the same in every thread).
    __device__ __forceinline__ uint64_t make_room(int k, int rounds = 1) {
        const int n = settled_count();
        if (n > CAP - rounds * NT) compact(k, n, false, (CAP - rounds * NT - k) / 4);
        return *reinterpret_cast<volatile uint64_t*>(thr);
    }

    // Collective: empty the buffer; from now on only keys >= threshold are admitted.
    __device__ void restart(uint64_t threshold) {
        sync();
        if (tid == 0) {
            ctl[0] = 0;
            ctl[4] = 0;
            *thr = threshold;
            rng[0] = 0ull;
            rng[1] = ~0ull;
        }
        sync();
    }

    // Collective: offer against a threshold returned by make_room.
    __device__ __forceinline__ void offer_thr(bool has, uint64_t key, uint64_t threshold) {
        const int lane = threadIdx.x & 31;
        const bool take = has && key >= threshold;
        const unsigned m = __ballot_sync(kFull, take);
        if (m) {
            const int leader = __ffs(m) - 1;
            int base = 0;
            if (lane == leader) base = atomicAdd(&ctl[0], __popc(m));
            base = __shfl_sync(kFull, base, leader);
            const int pos = base + __popc(m & ((1u << lane) - 1u));
            if (take) {
                if (pos < CAP)
                    buf[pos] = key;
                else
                    atomicOr(err, kErrAssert);
            }
        }
    }

    // Warp-collective: offer_thr of two keys per thread with one shared-memory reservation
    // for the warp (one atomic round trip instead of two).
    __device__ __forceinline__ void offer2_thr(bool has0, uint64_t key0, bool has1, uint64_t key1,
                                               uint64_t threshold) {
        const int lane = threadIdx.x & 31;
        const bool t0 = has0 && key0 >= threshold;
        const bool t1 = has1 && key1 >= threshold;
        const unsigned m0 = __ballot_sync(kFull, t0);
        const unsigned m1 = __ballot_sync(kFull, t1);
        const int n0 = __popc(m0);
        const int n = n0 + __popc(m1);
        if (n) {
            int base = 0;
            if (lane == 0) base = atomicAdd(&ctl[0], n);
            base = __shfl_sync(kFull, base, 0);
            const unsigned below = (1u << lane) - 1u;
            const int p0 = base + __popc(m0 & below);
            const int p1 = base + n0 + __popc(m1 & below);
            if (t0) {
                if (p0 < CAP)
                    buf[p0] = key0;
                else
                    atomicOr(err, kErrAssert);
            }
            if (t1) {
                if (p1 < CAP)
                    buf[p1] = key1;
                else
                    atomicOr(err, kErrAssert);
            }
        }
    }

    // Warp-collective: offer2_thr of two scored positions per thread, (s0, pos0) and
    // (s1, pos1), each taken part only when ok0 / ok1.  Most offers fall below the
    // threshold once the row has seen a few thousand keys, so the fp32 scores are first
    // compared with the threshold's score (score_floor of `threshold`): a key below it is
    // below the threshold whatever its position, and a warp with no lane at or above it
    // builds no 64-bit key at all.
    __device__ __forceinline__ void offer2_scored(bool ok0, float s0, uint32_t pos0, bool ok1,
                                                  float s1, uint32_t pos1, uint64_t threshold,
                                                  float floor) {
        const bool c0 = ok0 && s0 >= floor;
        const bool c1 = ok1 && s1 >= floor;
        if (!__any_sync(kFull, c0 || c1)) return;
        offer2_thr(c0, make_key(s0, pos0), c1, make_key(s1, pos1), threshold);
    }

    // Warp-collective: append two scored positions per thread whose score reaches `floor`
    // (every key of such a score is at least the threshold the selector was reset to), with
    // no room check: slots past CAP are not written and the count runs on beyond CAP, so a
    // caller that finds settled_count() > CAP knows keys were lost.  One shared-memory
    // reservation per warp.  The buffer receives raw_pair()s, not keys: keys_from_raw() or
    // dump_all_raw() converts them before anything compares them.
    __device__ __forceinline__ void offer2_capped(bool ok0, float s0, uint32_t pos0, bool ok1,
                                                  float s1, uint32_t pos1, float floor) {
        const bool t0 = ok0 && s0 >= floor;
        const bool t1 = ok1 && s1 >= floor;
        const unsigned m0 = __ballot_sync(kFull, t0);
        const unsigned m1 = __ballot_sync(kFull, t1);
        if ((m0 | m1) == 0u) return;
        const int lane = threadIdx.x & 31;
        const int n0 = __popc(m0);
        int base = 0;
        if (lane == 0) base = atomicAdd(&ctl[0], n0 + __popc(m1));
        base = __shfl_sync(kFull, base, 0);
        const unsigned below = (1u << lane) - 1u;
        const int p0 = base + __popc(m0 & below);
        const int p1 = base + n0 + __popc(m1 & below);
        if (t0 && p0 < CAP) buf[p0] = raw_pair(s0, pos0);
        if (t1 && p1 < CAP) buf[p1] = raw_pair(s1, pos1);
    }

    // Collective: turn the first n (at most CAP) held raw_pair()s into keys in place.
    __device__ void keys_from_raw(int n) {
        if (n > CAP) n = CAP;
        for (int i = tid; i < n; i += NT) buf[i] = key_of_raw(buf[i]);
        sync();
    }

    // Collective: drop held keys that cannot be among the k largest (no-op when n <= k).
    // `n` must be a settled_count() result (the same value in every thread).
    //
    // An MSD radix select over the 64-bit keys.  Every held key lies between the admission
    // threshold and the largest held key, so the bits above the highest bit in which
    // those two differ are common to all keys and skipped; then one digit of up to 8 bits
    // per pass narrows down the bin holding the k-th largest key.  exact: refine until
    // exactly k keys are kept.  Otherwise stop at the first digit whose bin keeps at most
    // k + slack keys: every key dropped is below the k-th largest, so nothing of the
    // final top k is lost.  The admission threshold rises to the kept bin's lower edge.
    // move = false only sets that threshold and leaves the buffer as it is (for a caller
    // that empties it next).  Between compactions hist[] is all zero, rng[0] is 0 and
    // rng[1] all ones.
    __device__ void compact(int k, int n, bool exact = true, int slack = 0, bool move = true) {
        if (n <= k) return;
        constexpr int U = 4;  // keys in flight per thread
        // the range of the held keys: bits above the highest bit in which the smallest and
        // the largest differ are common to all of them
        uint64_t hi = 0ull, mn = ~0ull;
        for (int b = 0; b < n; b += U * NT) {
            uint64_t x[U];
#pragma unroll
            for (int j = 0; j < U; ++j) {
                const int i = b + j * NT + tid;
                x[j] = i < n ? buf[i] : 0ull;
            }
#pragma unroll
            for (int j = 0; j < U; ++j) {
                hi = x[j] > hi ? x[j] : hi;
                if (b + j * NT + tid < n) mn = x[j] < mn ? x[j] : mn;
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const uint64_t h2 = __shfl_xor_sync(kFull, hi, o);
            const uint64_t m2 = __shfl_xor_sync(kFull, mn, o);
            hi = h2 > hi ? h2 : hi;
            mn = m2 < mn ? m2 : mn;
        }
        if ((threadIdx.x & 31) == 0) {
            atomicMax(reinterpret_cast<unsigned long long*>(rng), static_cast<unsigned long long>(hi));
            atomicMin(reinterpret_cast<unsigned long long*>(rng + 1),
                      static_cast<unsigned long long>(mn));
        }
        sync();
        hi = rng[0];
        const uint64_t lo = rng[1];
        if (hi <= lo || lo < *thr) {  // n >= 2 distinct keys, all >= the threshold
            if (tid == 0) atomicOr(err, kErrAssert);
            return;
        }
        const int top = 63 - __clzll(static_cast<long long>(lo ^ hi));
        uint64_t prefix = top == 63 ? 0ull : (hi & ~((2ull << top) - 1ull));
        int width = top + 1 < 8 ? top + 1 : 8;
        int shift = top + 1 - width;
        int need = k;
        int inbin = 0;
        while (true) {
            const int end = shift + width;
            const uint64_t hmask = end >= 64 ? 0ull : ~((1ull << end) - 1ull);
            const unsigned dmask = (1u << width) - 1u;
            for (int b = 0; b < n; b += U * NT) {
                uint64_t x[U];
#pragma unroll
                for (int j = 0; j < U; ++j) {
                    const int i = b + j * NT + tid;
                    x[j] = i < n ? buf[i] : 0ull;
                }
#pragma unroll
                for (int j = 0; j < U; ++j) {
                    if (b + j * NT + tid < n && (x[j] & hmask) == prefix)
                        atomicAdd(&hist[static_cast<unsigned>(x[j] >> shift) & dmask], 1u);
                }
            }
            sync();
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
                if (tid == 0) {
                    ctl[1] = -1;
                    rng[0] = 0ull;  // every thread read them before the barrier above
                    rng[1] = ~0ull;
                }
                __syncwarp();
                unsigned incl = sum;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const unsigned v = __shfl_up_sync(kFull, incl, o);
                    if (tid >= o) incl += v;
                }
                const unsigned excl = incl - sum;
                if (excl < static_cast<unsigned>(need) && static_cast<unsigned>(need) <= incl) {
                    unsigned above = excl;
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        if (above + c[j] >= static_cast<unsigned>(need)) {
                            ctl[1] = 255 - (tid * 8 + j);
                            ctl[2] = static_cast<int>(above);
                            ctl[3] = static_cast<int>(c[j]);
                            break;
                        }
                        above += c[j];
                    }
                }
            }
            sync();
            const int d = ctl[1];
            if (d < 0) {  // no bin holds the k-th key: counts are inconsistent
                if (tid == 0) atomicOr(err, kErrAssert);
                return;
            }
            prefix |= static_cast<uint64_t>(d) << shift;
            need -= ctl[2];
            inbin = ctl[3];
            // keys >= prefix: the k - need above the bin plus the whole bin
            if (inbin == need || shift == 0 || (!exact && k - need + inbin <= k + slack)) break;
            width = shift < 8 ? shift : 8;
            shift -= width;
        }
        const int kept = k - need + inbin;
        if (!move) {  // every thread has read ctl[] before the loop's last barrier
            if (tid == 0) *thr = prefix;
            sync();
            return;
        }
        // keep keys >= prefix, compacted to the front in place.  Each round reads the next
        // kRound * NT slots into registers before any thread writes; a write lands below
        // the count kept so far, which is below every later read.  A warp reserves the
        // slots for all its keys of the round with one atomic (offsets from a warp scan
        // of the per-thread counts).  ctl[4] is 0 here: the last user set it back (or
        // reset() did).
        constexpr int kRound = 8;
        const int lane = threadIdx.x & 31;
        for (int base = 0; base < n; base += kRound * NT) {
            uint64_t v[kRound];
            unsigned keep = 0u;  // bit j: v[j] is kept
#pragma unroll
            for (int j = 0; j < kRound; ++j) {
                const int i = base + j * NT + tid;
                v[j] = i < n ? buf[i] : 0ull;
                if (i < n && v[j] >= prefix) keep |= 1u << j;
            }
            const int c = __popc(keep);
            int incl = c;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int t = __shfl_up_sync(kFull, incl, o);
                if (lane >= o) incl += t;
            }
            int at = 0;
            if (lane == 31 && incl) at = atomicAdd(&ctl[4], incl);
            at = __shfl_sync(kFull, at, 31) + incl - c;
            sync();
#pragma unroll
            for (int j = 0; j < kRound; ++j) {
                if ((keep >> j) & 1u) {
                    if (at < CAP) buf[at] = v[j];
                    ++at;
                }
            }
        }
        sync();
        if (tid == 0) {
            const int got = ctl[4];
            if (got != kept || (exact && kept != k)) atomicOr(err, kErrAssert);
            ctl[0] = got < CAP ? got : CAP;
            ctl[4] = 0;
            *thr = prefix;
        }
        sync();
    }

    // Collective: sort buf[0..P) descending (P a power of two).
    __device__ void sort_desc(int P) {
        for (int size = 2; size <= P; size <<= 1) {
            for (int stride = size >> 1; stride > 0; stride >>= 1) {
                for (int i = tid; i < (P >> 1); i += NT) {
                    const int lo = 2 * i - (i & (stride - 1));
                    const int hi = lo + stride;
                    const uint64_t a = buf[lo];
                    const uint64_t b = buf[hi];
                    const bool desc = (lo & size) == 0;
                    if ((a < b) == desc) {
                        buf[lo] = b;
                        buf[hi] = a;
                    }
                }
                sync();
            }
        }
    }

    // Collective: write the top k in rank order; positions past the held count get
    // -1 (and -inf scores).
    __device__ void finalize(int k, int32_t* idx_out, float* score_out) {
        compact(k, settled_count());
        const int n = settled_count();
        int P = 1;
        while (P < n) P <<= 1;
        for (int i = n + tid; i < P; i += NT) buf[i] = 0ull;
        sync();
        sort_desc(P);
        for (int i = tid; i < k; i += NT) {
            if (i < n) {
                const uint64_t key = buf[i];
                idx_out[i] = key_position(key);
                if (score_out) score_out[i] = key_score(key);
            } else {
                idx_out[i] = -1;
                if (score_out) score_out[i] = -__int_as_float(0x7f800000);
            }
        }
        sync();
    }

    // Collective: every held key (no selection), unordered, and the count; the caller's list
    // has room for CAP keys.
    __device__ void dump_all(uint64_t* out, int* out_count) {
        const int n = settled_count();
        for (int i = tid; i < n; i += NT) out[i] = buf[i];
        if (tid == 0) *out_count = n;
        sync();
    }

    // Collective: dump_all of a buffer of raw_pair()s, each turned into its key on the way.
    // Four reads ahead of the stores: a read between them would wait on its own latency.
    __device__ void dump_all_raw(uint64_t* out, int* out_count) {
        const int n = settled_count();
        constexpr int U = 4;
        for (int b = tid; b < n; b += U * NT) {
            uint64_t v[U];
#pragma unroll
            for (int j = 0; j < U; ++j) v[j] = b + j * NT < n ? buf[b + j * NT] : 0ull;
#pragma unroll
            for (int j = 0; j < U; ++j)
                if (b + j * NT < n) out[b + j * NT] = key_of_raw(v[j]);
        }
        if (tid == 0) *out_count = n;
        sync();
    }

    // Collective: the k largest held keys (an exact compaction first), unordered, and their
    // count.
    __device__ void dump(int k, uint64_t* out, int* out_count) {
        compact(k, settled_count());
        const int n = settled_count();
        for (int i = tid; i < n; i += NT) out[i] = buf[i];
        if (tid == 0) *out_count = n;
        sync();
    }
};

}  // namespace tsi
