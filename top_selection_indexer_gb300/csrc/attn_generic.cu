// Sparse attention over the shared index rows on CUDA cores (any head shape).
//
// O[t,h] = sum_{s in S_t} softmax_s(scale * Q[t,h] . K[s,g]) V[s,g], g = h / (H/Hkv),
// S_t = the row's index entries inside [0, kv_len[b])  ("GLM-5.2 技术报告速览"
// §IndexShare; "GLM 5.2: Built for Long Horizon Tasks" discussion §3).  One warp owns
// one (row, head) and streams the row's selected keys with an online softmax in fp32
// (base-2 exponentials, the scale folded with log2(e) into the query).  Rows can be
// split over several blocks along the index list (decode); a combine kernel merges the
// partial (max, sum, accumulator) triples.
#include "attn_generic.cuh"
#include "tsi_common.cuh"

namespace tsi {
namespace {

constexpr int kWarps = 4;
constexpr int kMaxDq = 576 / 32;  // query/key registers per lane
constexpr int kMaxDv = 512 / 32;  // value registers per lane

__global__ void __launch_bounds__(kWarps * 32) attn_generic_kernel(AttnArgs a, int n_splits,
                                                                   int per_split,
                                                                   float* part_o,
                                                                   float* part_ml) {
    const int lane = threadIdx.x & 31;
    const int h = blockIdx.y * kWarps + (threadIdx.x >> 5);
    if (h >= a.H) return;
    const int row = blockIdx.x;
    const int split = blockIdx.z;
    const int b = row / a.T;
    const int g = h / (a.H / a.Hkv);
    const int64_t len = seq_len(a.kv_len, b, a.S);
    const uint16_t* q = static_cast<const uint16_t*>(a.q) +
                        (static_cast<int64_t>(row) * a.H + h) * a.Dqk;
    const uint16_t* kbase = static_cast<const uint16_t*>(a.k);
    const uint16_t* vbase = static_cast<const uint16_t*>(a.v);
    const float qscale = a.scale * 1.4426950408889634f;  // log2(e)

    float qr[kMaxDq];
#pragma unroll
    for (int i = 0; i < kMaxDq; ++i) {
        const int d = lane + 32 * i;
        qr[i] = d < a.Dqk ? bf16_bits_to_float(q[d]) * qscale : 0.f;
    }
    float acc[kMaxDv];
#pragma unroll
    for (int i = 0; i < kMaxDv; ++i) acc[i] = 0.f;
    float m = -__int_as_float(0x7f800000);
    float l = 0.f;

    const int32_t* sel = a.idx + static_cast<int64_t>(row) * a.topk;
    const int e_lo = split * per_split;
    const int e_hi = e_lo + per_split < a.topk ? e_lo + per_split : a.topk;
    for (int e = e_lo; e < e_hi; ++e) {
        const int s = sel[e];
        if (s < 0 || s >= len) continue;
        const int64_t kv_row = (static_cast<int64_t>(b) * a.S + s) * a.Hkv + g;
        const uint16_t* kr = kbase + kv_row * a.Dqk;
        float dot = 0.f;
#pragma unroll
        for (int i = 0; i < kMaxDq; ++i) {
            const int d = lane + 32 * i;
            if (d < a.Dqk) dot = fmaf(qr[i], bf16_bits_to_float(kr[d]), dot);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) dot += __shfl_xor_sync(kFull, dot, o);
        const float m_new = fmaxf(m, dot);
        const float corr = exp2f(m - m_new);
        const float pr = exp2f(dot - m_new);
        l = l * corr + pr;
        const uint16_t* vr = vbase ? vbase + kv_row * a.Dv : kr;
#pragma unroll
        for (int i = 0; i < kMaxDv; ++i) {
            const int d = lane + 32 * i;
            const float vv = d < a.Dv ? bf16_bits_to_float(vr[d]) : 0.f;
            acc[i] = fmaf(pr, vv, acc[i] * corr);
        }
        m = m_new;
    }
    if (n_splits == 1) {
        __nv_bfloat16* o = static_cast<__nv_bfloat16*>(a.out) +
                           (static_cast<int64_t>(row) * a.H + h) * a.Dv;
        const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
        for (int i = 0; i < kMaxDv; ++i) {
            const int d = lane + 32 * i;
            if (d < a.Dv) o[d] = __float2bfloat16_rn(acc[i] * inv);
        }
        if (a.lse && lane == 0)
            a.lse[static_cast<int64_t>(row) * a.H + h] = lse_of(m, l);
    } else {
        const int64_t slot = (static_cast<int64_t>(row) * n_splits + split) * a.H + h;
        float* po = part_o + slot * a.Dv;
#pragma unroll
        for (int i = 0; i < kMaxDv; ++i) {
            const int d = lane + 32 * i;
            if (d < a.Dv) po[d] = acc[i];
        }
        if (lane == 0) {
            part_ml[2 * slot] = m;
            part_ml[2 * slot + 1] = l;
        }
    }
}

// One block per (row, head): merge the split partials.  The splits' maxima and sums go
// through shared memory once; each thread then owns four value dims (float4 loads when Dv
// is a multiple of 4) and accumulates them over the splits.
constexpr int kCombineThreads = 128;
constexpr int kMaxCombineSplits = 256;

__global__ void __launch_bounds__(kCombineThreads) attn_combine_kernel(
    AttnArgs a, int n_splits, const float* part_o, const float* part_ml) {
    __shared__ float wsp[kMaxCombineSplits];  // weight of split sp: 2^(m_sp - M)
    const int row = blockIdx.x;
    const int h = blockIdx.y;
    const int tid = threadIdx.x;
    const float neg_inf = -__int_as_float(0x7f800000);
    const int64_t slot0 = static_cast<int64_t>(row) * n_splits * a.H + h;
    float m = neg_inf;
    for (int sp = tid; sp < n_splits; sp += kCombineThreads) {
        const float l = part_ml[2 * (slot0 + static_cast<int64_t>(sp) * a.H) + 1];
        if (l > 0.f) m = fmaxf(m, part_ml[2 * (slot0 + static_cast<int64_t>(sp) * a.H)]);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, o));
    if ((tid & 31) == 0) wsp[tid >> 5] = m;  // per-warp maxima (reused below)
    __syncthreads();
    float M = neg_inf;
    for (int w = 0; w < kCombineThreads / 32; ++w) M = fmaxf(M, wsp[w]);
    __syncthreads();
    float L = 0.f;
    for (int sp = tid; sp < n_splits; sp += kCombineThreads) {
        const int64_t sl = slot0 + static_cast<int64_t>(sp) * a.H;
        const float l = part_ml[2 * sl + 1];
        const float w = l > 0.f ? exp2f(part_ml[2 * sl] - M) : 0.f;
        wsp[sp] = w;
        L += l * w;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) L += __shfl_xor_sync(kFull, L, o);
    __shared__ float lsum[kCombineThreads / 32];
    __syncthreads();  // every split weight written
    if ((tid & 31) == 0) lsum[tid >> 5] = L;
    __syncthreads();
    float Lt = 0.f;
    for (int w = 0; w < kCombineThreads / 32; ++w) Lt += lsum[w];
    const float inv = Lt > 0.f ? 1.f / Lt : 0.f;
    if (a.lse && tid == 0) a.lse[static_cast<int64_t>(row) * a.H + h] = lse_of(M, Lt);
    __nv_bfloat16* o = static_cast<__nv_bfloat16*>(a.out) + (static_cast<int64_t>(row) * a.H + h) * a.Dv;
    if ((a.Dv & 3) == 0) {
        // eight splits' partials load at once, then accumulate in split order.  Every
        // split has its slot in the workspace, so the loads stay in bounds; a split
        // without keys has weight 0 and its slot (possibly never written) is not used.
        constexpr int kBatch = 8;
        for (int d = 4 * tid; d < a.Dv; d += 4 * kCombineThreads) {
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
            int sp = 0;
            for (; sp + kBatch <= n_splits; sp += kBatch) {
                float w[kBatch];
                float4 v[kBatch];
#pragma unroll
                for (int u = 0; u < kBatch; ++u) {
                    w[u] = wsp[sp + u];
                    v[u] = *reinterpret_cast<const float4*>(
                        part_o + (slot0 + static_cast<int64_t>(sp + u) * a.H) * a.Dv + d);
                }
#pragma unroll
                for (int u = 0; u < kBatch; ++u) {
                    if (w[u] == 0.f) continue;
                    acc.x = fmaf(w[u], v[u].x, acc.x);
                    acc.y = fmaf(w[u], v[u].y, acc.y);
                    acc.z = fmaf(w[u], v[u].z, acc.z);
                    acc.w = fmaf(w[u], v[u].w, acc.w);
                }
            }
            for (; sp < n_splits; ++sp) {
                const float w = wsp[sp];
                if (w == 0.f) continue;
                const float4 v = *reinterpret_cast<const float4*>(
                    part_o + (slot0 + static_cast<int64_t>(sp) * a.H) * a.Dv + d);
                acc.x = fmaf(w, v.x, acc.x);
                acc.y = fmaf(w, v.y, acc.y);
                acc.z = fmaf(w, v.z, acc.z);
                acc.w = fmaf(w, v.w, acc.w);
            }
            o[d] = __float2bfloat16_rn(acc.x * inv);
            o[d + 1] = __float2bfloat16_rn(acc.y * inv);
            o[d + 2] = __float2bfloat16_rn(acc.z * inv);
            o[d + 3] = __float2bfloat16_rn(acc.w * inv);
        }
    } else {
        for (int d = tid; d < a.Dv; d += kCombineThreads) {
            float acc = 0.f;
            for (int sp = 0; sp < n_splits; ++sp) {
                const float w = wsp[sp];
                if (w != 0.f)
                    acc = fmaf(w, part_o[(slot0 + static_cast<int64_t>(sp) * a.H) * a.Dv + d], acc);
            }
            o[d] = __float2bfloat16_rn(acc * inv);
        }
    }
}

}  // namespace

void attn_generic_split_plan(int rows, int topk, int* n_splits, int* per_split) {
    int ns = 1;
    if (rows > 0 && rows < 152) {
        ns = (topk + 127) / 128;
        const int cap = (2 * 152 + rows - 1) / rows;
        if (ns > cap) ns = cap;
        if (ns < 1) ns = 1;
    }
    *n_splits = ns;
    *per_split = (topk + ns - 1) / ns;
}

size_t attn_generic_workspace_bytes(int B, int T, int H, int Dv, int topk) {
    int ns, ps;
    const int rows = B * T;
    attn_generic_split_plan(rows, topk, &ns, &ps);
    if (ns <= 1) return 0;
    const size_t slots = static_cast<size_t>(rows) * ns * H;
    return slots * Dv * sizeof(float) + slots * 2 * sizeof(float);
}

bool attn_generic_supported(int H, int Hkv, int Dqk, int Dv, bool v_from_k) {
    return H >= 1 && Hkv >= 1 && H % Hkv == 0 && Dqk >= 1 && Dqk <= 576 && Dv >= 1 &&
           Dv <= 512 && (!v_from_k || Dv <= Dqk);
}

cudaError_t launch_attn_generic(const AttnArgs& a, void* workspace, cudaStream_t st) {
    const int rows = a.B * a.T;
    int ns, ps;
    attn_generic_split_plan(rows, a.topk, &ns, &ps);
    float* part_o = nullptr;
    float* part_ml = nullptr;
    if (ns > 1) {
        part_o = static_cast<float*>(workspace);
        part_ml = part_o + static_cast<size_t>(rows) * ns * a.H * a.Dv;
    }
    const dim3 grid(rows, (a.H + kWarps - 1) / kWarps, ns);
    attn_generic_kernel<<<grid, kWarps * 32, 0, st>>>(a, ns, ps, part_o, part_ml);
    note_launches(1);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess || ns == 1) return e;
    attn_combine_kernel<<<dim3(rows, a.H), kCombineThreads, 0, st>>>(a, ns, part_o, part_ml);
    note_launches(1);
    return cudaGetLastError();
}

}  // namespace tsi

namespace tsi {

cudaError_t launch_attn_combine(const AttnArgs& a, int n_splits, const float* part_o,
                                const float* part_ml, cudaStream_t st) {
    if (n_splits > kMaxCombineSplits) return cudaErrorInvalidValue;
    attn_combine_kernel<<<dim3(a.B * a.T, a.H), kCombineThreads, 0, st>>>(a, n_splits, part_o,
                                                                           part_ml);
    note_launches(1);
    return cudaGetLastError();
}

}  // namespace tsi
