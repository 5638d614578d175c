// Gather of selected 576-d latent rows (bf16) into 128-byte-swizzled shared-memory tiles,
// the A operand of S^T = K_tile . Q^T for 128 keys at a time.  Shared by the sparse
// attention kernel and the group-centroid KL kernel, which both read the keys of a row's
// shared index set ("GLM-5.2 技术报告速览" §IndexShare: each layer of the group reads the
// keys the Full layer selected).
#pragma once

#include "tc_common.cuh"
#include "tsi_common.cuh"

namespace tsi {
namespace latent {

constexpr int kKeys = 128;  // keys per tile (MMA M)
constexpr int kDqk = 576;  // latent row: 512 compressed + 64 RoPE dims
constexpr int kChunks = kDqk / 64;  // nine 64-dim (128-byte) chunks per row
constexpr int kChunkBytes = kKeys * 128;  // one chunk of a tile: 16 KB

// This thread's share of the gather of key tile t (entries t*128 .. t*128+127 of the row's
// index list irow).  A chunk is 128 keys x 8 pieces of 16 bytes laid out as the K-major
// SW128 operand: 8-key groups of 1024 bytes, piece j of key k at 16 * (j ^ (k & 7)).
// Gather thread g of NG copies pieces g, g + NG, ... of every chunk, chunk c into ring slot
// c once the MMA has released it (kv_empty[c], phase it ^ 1), then arrives on kv_full[c]
// when its copies land.  Keys outside [0, len) and entries past topk are zero-filled.
//   kseq  the sequence's latent rows [S, 576] bf16
template <int NG>
__device__ __forceinline__ void gather_tile(const uint16_t* kseq, int64_t len, const int32_t* irow,
                                            int topk, int t, int it, int g, uint32_t kv_addr,
                                            uint64_t* kv_empty, uint64_t* kv_full,
                                            volatile int* abort, unsigned* err) {
    constexpr int kPer = (kKeys * 8 + NG - 1) / NG;
    const uint16_t* src[kPer];
    uint32_t nbytes[kPer];
    uint32_t dst0[kPer];
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
        const int piece = g + NG * j;
        const int k = (piece >> 3) & (kKeys - 1);
        const int sub = piece & 7;
        const int e = t * kKeys + k;
        const int s = (piece < kKeys * 8 && e < topk) ? irow[e] : -1;
        const bool ok = s >= 0 && s < len;
        src[j] = ok ? kseq + static_cast<int64_t>(s) * kDqk + sub * 8 : kseq;
        nbytes[j] = ok ? 16u : 0u;
        dst0[j] = kv_addr + (k >> 3) * 1024 + (k & 7) * 128 + ((sub ^ (k & 7)) << 4);
    }
    for (int c = 0; c < kChunks; ++c) {
        tc::mbar_wait(&kv_empty[c], (it & 1) ^ 1, abort, err);
#pragma unroll
        for (int j = 0; j < kPer; ++j) {
            if (g + NG * j < kKeys * 8)
                tc::cp_async16(dst0[j] + c * kChunkBytes, src[j] + (nbytes[j] ? c * 64 : 0),
                               nbytes[j]);
        }
        tc::cp_async_arrive_noinc(&kv_full[c]);
    }
}

}  // namespace latent
}  // namespace tsi
