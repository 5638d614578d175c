// Shared device helpers of the CUDA library (not used by the CPU oracle).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/tsi.h"

namespace tsi {

// Device error word bits (set with atomicOr, read by tsi_device_status).
enum : unsigned { kErrTimeout = 1u, kErrAssert = 2u };

constexpr unsigned kFull = 0xFFFFFFFFu;

__device__ __forceinline__ float bf16_bits_to_float(uint16_t b) {
    return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

__device__ __forceinline__ float e4m3_to_float(uint8_t b) {
    __half_raw h = __nv_cvt_fp8_to_halfraw(static_cast<__nv_fp8_storage_t>(b), __NV_E4M3);
    return __half2float(__half(h));
}

// Element i of a tensor stored as dtype `dt` (TSI_F32 / TSI_BF16 / TSI_E4M3).
__device__ __forceinline__ float load_elem(const void* base, int64_t i, int dt) {
    if (dt == TSI_F32) return static_cast<const float*>(base)[i];
    if (dt == TSI_BF16) return bf16_bits_to_float(static_cast<const uint16_t*>(base)[i]);
    return e4m3_to_float(static_cast<const uint8_t*>(base)[i]);
}

// Position of query row t of sequence b (kv_len clamped to [0, S]).
__device__ __forceinline__ int64_t query_position(const int32_t* kv_len, int b, int T, int S,
                                                  int t) {
    int64_t len = kv_len ? static_cast<int64_t>(kv_len[b]) : static_cast<int64_t>(S);
    len = len < 0 ? 0 : (len > S ? S : len);
    return len - T + t;
}

__device__ __forceinline__ int64_t seq_len(const int32_t* kv_len, int b, int S) {
    int64_t len = kv_len ? static_cast<int64_t>(kv_len[b]) : static_cast<int64_t>(S);
    return len < 0 ? 0 : (len > S ? S : len);
}

// ln sum_s exp(x_s) from the base-2 running maximum m (of x_s * log2(e)) and the sum
// l = sum_s 2^(x_s log2(e) - m) of an online softmax; -inf when nothing was summed.
__device__ __forceinline__ float lse_of(float m, float l) {
    return l > 0.f ? (m + log2f(l)) * 0.69314718055994531f : -__int_as_float(0x7f800000);
}

// Counts kernel launches made by the library (reported by tsi_launch_count).
void note_launches(int n);

// Named barrier over `n` threads (a multiple of 32); id 0 with the whole block is
// __syncthreads().
__device__ __forceinline__ void named_bar(int id, int n) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

}  // namespace tsi
