// fa_decode.cu -- split-K forward for a few query rows against a long key
// sequence ("Lab 06 - Attention kernels", "Check yourself" item 2 and
// "Stretch": with one query row per head the only parallelism of a plain
// FlashAttention forward is batch x heads; split-K partitions the keys across
// programs, each computing a partial (m, l, acc), and a small reduction merges
// them with the same rescaling rule as the online softmax).
//
// The work is HBM-bound (about Tq FLOP per byte of K/V), so it runs on the
// CUDA cores: each warp streams groups of consecutive key/value rows with
// coalesced loads (lane = slice of the head dimension), reduces the scores
// across the warp, and keeps per-query running (m, l, acc); the warps of a
// CTA merge in shared memory and write one partial per key chunk.  A second
// kernel merges the chunks: m = max_s m_s, l = sum_s 2^(m_s - m) l_s,
// O = sum_s 2^(m_s - m) acc_s / l, LSE = (m + log2 l) ln 2.
#include <cuda_runtime.h>

#include "fa_internal.h"
#include "fa_ptx.cuh"

namespace fa {
namespace {

constexpr int kDecThreads = 128;
constexpr int kDecWarps = kDecThreads / 32;
constexpr float kLn2 = 0.69314718055994530942f;
constexpr float kLog2e = 1.44269504088896340736f;

struct DecParams {
    const __nv_bfloat16* q;
    const __nv_bfloat16* k;
    const __nv_bfloat16* v;
    float* part_m;    // [BH][n_split][Tq]        running max (log2 units)
    float* part_l;    // [BH][n_split][Tq]        running sum
    float* part_acc;  // [BH][n_split][Tq][D]     unnormalised output
    int Tq, Tk, n_split, chunk;
    float sl2;  // scale * log2(e)
};

template <int E>
__device__ __forceinline__ void load_slice(const __nv_bfloat16* row, int lane, float (&out)[E]) {
    if constexpr (E == 4) {
        const uint2 u = *reinterpret_cast<const uint2*>(row + lane * 4);
        const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.x));
        const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.y));
        out[0] = a.x; out[1] = a.y; out[2] = b.x; out[3] = b.y;
    } else {
        const uint32_t u = *reinterpret_cast<const uint32_t*>(row + lane * 2);
        const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u));
        out[0] = a.x; out[1] = a.y;
    }
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}
__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
    return x;
}

// One CTA = one key chunk of one (batch, head); TQ = compile-time bound on Tq.
template <int D, int TQ>
__global__ void __launch_bounds__(kDecThreads) fa_decode_partial_kernel(DecParams p) {
    constexpr int E = D / 32;               // head-dimension elements per lane
    // keys per warp step: 4 keeps registers low enough for ~8 resident CTAs
    // per SM; the many warps, not deep per-warp batches, carry the bytes in
    // flight (measured at B=8 H=32 Tk=32768 D=128: 8 keys 5.70 TB/s, 4 keys
    // 6.47 TB/s, 2 keys 6.12 TB/s)
    constexpr int G = 4;
    const int split = blockIdx.x, bh = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int k0 = split * p.chunk;
    const int k1 = min(k0 + p.chunk, p.Tk);
    const int Tq = p.Tq;

    float qr[TQ][E];
#pragma unroll
    for (int t = 0; t < TQ; ++t) {
        if (t < Tq) {
            load_slice<E>(p.q + (static_cast<size_t>(bh) * Tq + t) * D, lane, qr[t]);
#pragma unroll
            for (int e = 0; e < E; ++e) qr[t][e] *= p.sl2;  // scores come out in log2 units
        } else {
#pragma unroll
            for (int e = 0; e < E; ++e) qr[t][e] = 0.f;
        }
    }
    float m[TQ], l[TQ], acc[TQ][E];
#pragma unroll
    for (int t = 0; t < TQ; ++t) {
        m[t] = -INFINITY;
        l[t] = 0.f;
#pragma unroll
        for (int e = 0; e < E; ++e) acc[t][e] = 0.f;
    }
    const __nv_bfloat16* kb = p.k + static_cast<size_t>(bh) * p.Tk * D;
    const __nv_bfloat16* vb = p.v + static_cast<size_t>(bh) * p.Tk * D;
    for (int g0 = k0 + warp * G; g0 < k1; g0 += kDecWarps * G) {
        float kf[G][E], vf[G][E];
#pragma unroll
        for (int g = 0; g < G; ++g) {
            if (g0 + g < k1) {
                load_slice<E>(kb + static_cast<size_t>(g0 + g) * D, lane, kf[g]);
                load_slice<E>(vb + static_cast<size_t>(g0 + g) * D, lane, vf[g]);
            } else {
#pragma unroll
                for (int e = 0; e < E; ++e) kf[g][e] = vf[g][e] = 0.f;
            }
        }
#pragma unroll
        for (int t = 0; t < TQ; ++t) {
            float s[G];
#pragma unroll
            for (int g = 0; g < G; ++g) {
                float part = 0.f;
#pragma unroll
                for (int e = 0; e < E; ++e) part = fmaf(qr[t][e], kf[g][e], part);
                s[g] = (g0 + g < k1) ? warp_sum(part) : -INFINITY;
            }
            float mg = s[0];
#pragma unroll
            for (int g = 1; g < G; ++g) mg = fmaxf(mg, s[g]);
            const float m_new = fmaxf(m[t], mg);  // finite: key g0 < k1 exists
            const float alpha = (m[t] == -INFINITY) ? 0.f : ex2_approx(m[t] - m_new);
            l[t] *= alpha;
#pragma unroll
            for (int e = 0; e < E; ++e) acc[t][e] *= alpha;
#pragma unroll
            for (int g = 0; g < G; ++g) {
                const float pg = ex2_approx(s[g] - m_new);
                l[t] += pg;
#pragma unroll
                for (int e = 0; e < E; ++e) acc[t][e] = fmaf(pg, vf[g][e], acc[t][e]);
            }
            m[t] = m_new;
        }
    }
    // merge the warps of this CTA
    __shared__ float sm_m[kDecWarps][TQ], sm_l[kDecWarps][TQ];
    __shared__ float sm_acc[kDecWarps][TQ][D];
#pragma unroll
    for (int t = 0; t < TQ; ++t) {
        if (lane == 0) {
            sm_m[warp][t] = m[t];
            sm_l[warp][t] = l[t];
        }
#pragma unroll
        for (int e = 0; e < E; ++e) sm_acc[warp][t][lane * E + e] = acc[t][e];
    }
    __syncthreads();
    for (int t = warp; t < Tq; t += kDecWarps) {
        float mm = -INFINITY;
#pragma unroll
        for (int w = 0; w < kDecWarps; ++w) mm = fmaxf(mm, sm_m[w][t]);
        float wts[kDecWarps], ll = 0.f;
#pragma unroll
        for (int w = 0; w < kDecWarps; ++w) {
            wts[w] = (sm_m[w][t] == -INFINITY) ? 0.f : ex2_approx(sm_m[w][t] - mm);  // warps with no keys add 0
            ll = fmaf(wts[w], sm_l[w][t], ll);
        }
        const size_t base = (static_cast<size_t>(bh) * p.n_split + split) * Tq + t;
        for (int d = lane; d < D; d += 32) {
            float a = 0.f;
#pragma unroll
            for (int w = 0; w < kDecWarps; ++w) a = fmaf(wts[w], sm_acc[w][t][d], a);
            p.part_acc[base * D + d] = a;
        }
        if (lane == 0) {
            p.part_m[base] = mm;
            p.part_l[base] = ll;
        }
    }
}

// One warp per (batch*head, query row): merge the key chunks.
template <int D>
__global__ void __launch_bounds__(128) fa_decode_merge_kernel(const float* __restrict__ part_m,
                                                              const float* __restrict__ part_l,
                                                              const float* __restrict__ part_acc,
                                                              __nv_bfloat16* __restrict__ o, float* __restrict__ lse,
                                                              int BH, int Tq, int n_split) {
    const int r = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
    if (r >= BH * Tq) return;  // whole warp leaves together
    const int bh = r / Tq, t = r % Tq;
    auto idx = [&](int s) { return (static_cast<size_t>(bh) * n_split + s) * Tq + t; };
    float mm = -INFINITY;
    for (int s = lane; s < n_split; s += 32) mm = fmaxf(mm, part_m[idx(s)]);
    mm = warp_max(mm);
    float ll = 0.f;
    for (int s = lane; s < n_split; s += 32) ll = fmaf(ex2_approx(part_m[idx(s)] - mm), part_l[idx(s)], ll);
    ll = warp_sum(ll);
    const float inv = 1.f / ll;
    for (int d = lane; d < D; d += 32) {
        float a = 0.f;
        for (int s = 0; s < n_split; ++s) a = fmaf(ex2_approx(part_m[idx(s)] - mm), part_acc[idx(s) * D + d], a);
        o[(static_cast<size_t>(bh) * Tq + t) * D + d] = __float2bfloat16_rn(a * inv);
    }
    if (lane == 0) lse[static_cast<size_t>(bh) * Tq + t] = (mm + __log2f(ll)) * kLn2;
}

template <int D, int TQ>
void launch_partial(const DecParams& p, int BH, cudaStream_t st) {
    fa_decode_partial_kernel<D, TQ><<<dim3(p.n_split, BH), kDecThreads, 0, st>>>(p);
}

}  // namespace

int launch_decode(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Tq, int Tk,
                  int D, float scale, cudaStream_t stream, int num_sms) {
    const int BH = B * H;
    // about two waves of resident CTAs (chunks of at least 256 keys): 16 CTAs
    // per SM measured 6.56 TB/s against 6.47 at 32 and 6.40 at 64
    const long long want = 16LL * num_sms;
    int n_split = static_cast<int>((want + BH - 1) / BH);
    const int max_split = (Tk + 255) / 256;
    n_split = n_split < 1 ? 1 : (n_split > max_split ? max_split : n_split);
    int chunk = (Tk + n_split - 1) / n_split;
    chunk = (chunk + 31) / 32 * 32;
    n_split = (Tk + chunk - 1) / chunk;
    const size_t n_part = static_cast<size_t>(BH) * n_split * Tq;
    const size_t bytes = n_part * 4 * 2 + n_part * D * 4 + 512;
    void* ws = nullptr;
    if (cudaMallocAsync(&ws, bytes, stream) != cudaSuccess) {
        cudaGetLastError();
        return -6;
    }
    DecParams p;
    p.q = static_cast<const __nv_bfloat16*>(q);
    p.k = static_cast<const __nv_bfloat16*>(k);
    p.v = static_cast<const __nv_bfloat16*>(v);
    p.part_m = static_cast<float*>(ws);
    p.part_l = p.part_m + n_part;
    p.part_acc = reinterpret_cast<float*>((reinterpret_cast<uintptr_t>(p.part_l + n_part) + 255) & ~uintptr_t(255));
    p.Tq = Tq;
    p.Tk = Tk;
    p.n_split = n_split;
    p.chunk = chunk;
    p.sl2 = scale * kLog2e;
    const int tq = Tq <= 1 ? 1 : Tq <= 2 ? 2 : Tq <= 4 ? 4 : 8;
    if (D == 64) {
        if (tq == 1) launch_partial<64, 1>(p, BH, stream);
        else if (tq == 2) launch_partial<64, 2>(p, BH, stream);
        else if (tq == 4) launch_partial<64, 4>(p, BH, stream);
        else launch_partial<64, 8>(p, BH, stream);
    } else {
        if (tq == 1) launch_partial<128, 1>(p, BH, stream);
        else if (tq == 2) launch_partial<128, 2>(p, BH, stream);
        else if (tq == 4) launch_partial<128, 4>(p, BH, stream);
        else launch_partial<128, 8>(p, BH, stream);
    }
    int rc = cudaGetLastError() == cudaSuccess ? 0 : -5;
    if (rc == 0) {
        const int warps = BH * Tq;
        const int blocks = (warps * 32 + 127) / 128;
        if (D == 64)
            fa_decode_merge_kernel<64><<<blocks, 128, 0, stream>>>(p.part_m, p.part_l, p.part_acc,
                                                                   static_cast<__nv_bfloat16*>(o), lse, BH, Tq,
                                                                   n_split);
        else
            fa_decode_merge_kernel<128><<<blocks, 128, 0, stream>>>(p.part_m, p.part_l, p.part_acc,
                                                                    static_cast<__nv_bfloat16*>(o), lse, BH, Tq,
                                                                    n_split);
        if (cudaGetLastError() != cudaSuccess) rc = -5;
    }
    if (cudaFreeAsync(ws, stream) != cudaSuccess && rc == 0) rc = -5;
    return rc;
}

}  // namespace fa
