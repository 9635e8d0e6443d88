// fa_bwd.cu -- exact attention backward on sm_103a ("Lab 06 - Attention
// kernels", section 4: D = rowsum(dO o O); P = exp(S - LSE) recomputed per
// tile; dV = P^T dO; dP = dO V^T; dS = P o (dP - D); dQ = dS K scale;
// dK = dS^T Q scale).
//
// The backward is split as "Lab 06", "Stretch" describes: one kernel with key
// tiles outer for dK and dV, one with query tiles outer for dQ, each
// recomputing S and dP, so that no tile's contribution needs a reduction in
// global memory.  Three kernels on the caller's stream:
//   fa_bwd_pre   D_i = sum_d dO_id O_id (fp32) and LSE in log2 units, both
//                stored negated and padded to a multiple of 128 rows.
//   fa_bwd_dkdv  key tiles outer, query tiles inner ("Lab 06", section 4:
//                dK and dV accumulate in one place).  One CTA per (key tile
//                of 128, batch * key/value head).  Warp roles:
//                  warps 0-7   compute: P^T = exp2(S^T c - LSE2) and
//                              dS^T = P^T o (dP^T - D), half of the query
//                              columns each (TMEM lane = key row)
//                  warp 8      TMA producer (K, V once; per query tile Q with
//                              -LSE2, -D and dO, each into a ring)
//                  warp 9      tcgen05 issuer: dP^T = V dO^T, dV += P^T dO
//                              (P^T from TMEM), S^T = K Q^T, dK += dS^T Q
//                and the compute warps store dK*scale and dV at the end.
//   fa_bwd_dq    query tiles outer, key tiles inner: dQ receives a
//                contribution from every key tile, so it is summed here in
//                TMEM instead of by reductions into global memory.  One CTA
//                per (query tile of 128, batch * query head); S and dP are
//                recomputed (S = Q K^T, dP = dO V^T), dS goes to TMEM as bf16
//                and dQ += dS K; dQ*scale leaves once, in bf16.
// The two main kernels read the same inputs and write disjoint outputs.
// At D = 64, on grids of at least one dK/dV CTA per SM, the backward keeps
// section 4's own loop order instead: fa_bwd_dkdv (FUSE) also computes each
// query tile's dS K and adds it into an fp32 dQ accumulator with TMA
// reduce-adds (zeroed by fa_bwd_pre), and fa_bwd_dq_convert writes dQ*scale
// in bf16.  The sum order of those adds varies from run to run;
// fa_set_deterministic(1) selects the two-kernel form.
#include <cuda_runtime.h>

#include <mutex>

#include "fa.h"
#include "fa_check.cuh"
#include "fa_internal.h"
#include "fa_ptx.cuh"
#include "fa_sched.h"
#include "fa_tmap.h"

namespace fa {

static __device__ int g_status_bwd;

namespace {

constexpr int kBwdThreads = 320;  // both main kernels: 8 compute warps, producer, MMA issuer
constexpr float kLog2e = 1.44269504088896340736f;
constexpr int kSmemLimit = 232448;  // opt-in shared memory per CTA

// The dynamic shared-memory window, 1024-byte aligned by hand when the
// layout leaves room for it.  Without that room the window must already be
// aligned (the kernels check it and report an error otherwise): 128-byte
// swizzle atoms need 1024-byte alignment.
template <int kSlack>
__device__ __forceinline__ uint8_t* smem_window(uint8_t* raw) {
    if constexpr (kSlack != 0)
        return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
    return raw;
}

// ---------------------------------------------------------------- dK / dV kernel layout
// FUSE (D = 64 only): the same kernel also computes each query tile's dQ
// contribution dS K (dS staged in shared memory) and adds it into an fp32
// dQ accumulator in global memory with TMA reduce-adds, so the backward needs
// no second pass over the key tiles.
template <int D, bool FUSE = false>
struct DkvCfg {
    static_assert(!FUSE || D == 64, "the fused dQ path fits in tensor memory at D = 64 only");
    static constexpr int BM = bwd_bm(D);             // query rows per inner iteration
    static constexpr int kAtomsD = D / 64;
    static constexpr int kKVBytes = 128 * D * 2;     // one K or V tile
    static constexpr int kQBytes = BM * D * 2;       // one Q or dO tile
    // Q (with its -LSE2 and -D vectors) and dO travel in separate rings.
    // (FUSE: one stage less in each ring, to make room for two dS buffers)
    static constexpr int kQStages = FUSE ? 3 : ((D == 128) ? 2 : 4);
    static constexpr int kDOStages = FUSE ? 2 : ((D == 128) ? 2 : 3);
    static constexpr int kQStageBytes = kQBytes + 1024;  // + -LSE2[BM], -D[BM] (<= 1 KB)
    static constexpr int kKOff = 0;
    static constexpr int kVOff = kKVBytes;
    static constexpr int kQRingOff = 2 * kKVBytes;
    static constexpr int kDORingOff = kQRingOff + kQStages * kQStageBytes;
    // FUSE: dS of two query tiles (bf16, 128 keys x BM queries each, queries
    // contiguous: the MN-major A operand of dQ = dS K), then the fp32 staging of
    // one dQ tile (BM rows x D: per compute warp 32 rows x 32 columns, 4 KB in the
    // 128-byte swizzled layout)
    static constexpr int kDSOff = kDORingOff + kDOStages * kQBytes;
    static constexpr int kDSBufBytes = 128 * BM * 2;
    static constexpr int kDSBytes = FUSE ? 2 * kDSBufBytes : 0;
    static constexpr int kStgOff = kDSOff + kDSBytes;
    static constexpr int kStgBytes = FUSE ? BM * D * 4 : 0;
    static constexpr int kBarOff = kStgOff + kStgBytes;
    // kv_full, q_full[], q_empty[], do_full[], do_empty[], s_full, dp_full, p_full, ds_full, dkv_full, mma_done,
    // epi[2]; FUSE: dq_full[2], dq_empty[2]
    static constexpr int kNumBars = 1 + 2 * kQStages + 2 * kDOStages + 8 + (FUSE ? 4 : 0);
    static constexpr int kMiscOff = kBarOff + kNumBars * 8;
    static constexpr int kPayload = kMiscOff + 16;   // + TMEM address slot, abort flag
    static constexpr int kSlack = (kPayload + 1024 <= kSmemLimit) ? 1024 : 0;
    static constexpr int kSmemBytes = kPayload + kSlack;
    static_assert(kSmemBytes <= kSmemLimit, "shared memory budget");
    static_assert(kDSOff % 1024 == 0 && kStgOff % 1024 == 0, "swizzle atoms need 1024-byte alignment");
    // TMEM columns: S^T, with P^T (bf16 pairs) written over the S^T columns its
    // warpgroup has already read; dP^T, with dS^T written over it the same way;
    // dV; dK; FUSE: two dQ buffers (a query tile's dS K, 128 query lanes x D),
    // so one is read out while the next is computed.  Both MMA operands that
    // come from the compute warps for dV and dK (P^T, dS^T) are read from
    // TMEM, which keeps them off shared memory: the K-major products already
    // use its full bandwidth.
    static constexpr uint32_t kS = 0;                // S^T [128 keys][BM] fp32
    static constexpr uint32_t kP = BM / 4;           // P^T: warpgroup h at kP + 32 h
    static constexpr uint32_t kDP = BM;              // dP^T [128 keys][BM] fp32
    static constexpr uint32_t kDS = kDP + BM / 4;    // dS^T: warpgroup h at kDS + 32 h
    static constexpr uint32_t kDV = 2 * BM;          // dV [128 keys][D] fp32
    static constexpr uint32_t kDK = kDV + D;         // dK [128 keys][D] fp32
    __host__ __device__ static constexpr uint32_t kDQ(int b) { return kDK + D + D * b; }
    static_assert((FUSE ? kDK + 3 * D : kDK + D) <= 512, "TMEM budget");
    static constexpr uint32_t kIdescS = idesc_bf16_f32(128, BM, false, false);
    static constexpr uint32_t kIdescDKV = idesc_bf16_f32(128, D, false, true);
    // dQ = dS K: M = BM queries, N = D, K = 128 keys; dS and K both MN-major
    static constexpr uint32_t kIdescDQ = idesc_bf16_f32(BM, D, true, true);
};

// ---------------------------------------------------------------- dQ kernel layout
template <int D>
struct DqCfg {
    static constexpr int kAtomsD = D / 64;
    static constexpr int kTileBytes = 128 * D * 2;   // one 128-row Q, dO, K or V tile
    static constexpr int kKStages = 3, kVStages = 2; // K_j feeds S(j) two tiles ahead and dQ(j); V_j feeds dP(j)
    static constexpr int kQOff = 0;
    static constexpr int kDOOff = kTileBytes;
    static constexpr int kKOff = 2 * kTileBytes;
    static constexpr int kVOff = kKOff + kKStages * kTileBytes;
    static constexpr int kBarOff = kVOff + kVStages * kTileBytes;
    // qdo_full, qdo_empty, k_full[], k_empty[], v_full[], v_empty[], s_full[2], dp_full, ds_full, dq_full,
    // dq_empty, mma_done, item_full[4], item_empty[4]
    static constexpr int kNumBars = 2 + 2 * kKStages + 2 * kVStages + 2 + 5 + 8;
    static constexpr int kMiscOff = kBarOff + kNumBars * 8;
    static constexpr int kPayload = kMiscOff + 32;   // + TMEM address slot, abort flag, item ring (4 ints)
    static constexpr int kSlack = (kPayload + 1024 <= kSmemLimit) ? 1024 : 0;
    static constexpr int kSmemBytes = kPayload + kSlack;
    static_assert(kSmemBytes <= kSmemLimit, "shared memory budget");
    // TMEM columns: S[2] (dS, bf16 pairs, written over the S columns its
    // warpgroup has read: warpgroup h at kS(b) + 32 + 32 h), dP, dQ.
    __device__ static constexpr uint32_t kS(int b) { return 128u * b; }
    static constexpr uint32_t kDSCol = 32;
    static constexpr uint32_t kDP = 256;
    static constexpr uint32_t kDQ = 384;
    static_assert(kDQ + D <= 512, "TMEM budget");
    static constexpr uint32_t kIdescS = idesc_bf16_f32(128, 128, false, false);
    static constexpr uint32_t kIdescDQ = idesc_bf16_f32(128, D, false, true);
};

struct BwdParams {
    const float* lse2;   // [B*Hq][T_pad] -LSE * log2(e)
    const float* dvec;   // [B*Hq][T_pad] -D
    __nv_bfloat16* dq;    // dQ kernel: output, stored row by row
    int n_items;          // dQ kernel: (query tile, query head) work items
    __nv_bfloat16* dk;
    __nv_bfloat16* dv;
    int T, T_pad, n_kt;   // n_kt = 128-row tiles (key tiles = query tiles)
    int kt_major;         // dK/dV kernel: CTA order key tile major (else head major)
    int* dq_next;         // dQ kernel: next item to hand out (zeroed by the preprocess kernel)
    int BH;               // rows of the grid: B*Hkv (dK/dV kernel) or B*Hq (dQ kernel)
    int Hq, Hkv, group;   // query heads, key/value heads, Hq / Hkv
    float scale;
    float sl2, sl2_eff;
    int prescale;
    unsigned long long timeout_ns;
    int inject;           // test hook: 2 = the dK/dV grid's first CTA drops its third Q fill (its first
                          // when it has fewer), 3 = the dQ grid's first CTA drops its first K fill (its
                          // waits then run out)
    // Packed variable-length batch (VARLEN kernels): sequence s occupies rows
    // cu_seqlens[s] .. cu_seqlens[s+1]-1 of the (total, H, D) tensors; T above
    // is then the longest length the caller promises, and a "head" index bh
    // of the grids is h * n_seq + s (per-row vectors: bh * T_pad + t).
    const int* cu_seqlens;
    int n_seq, total;
};

// Sequence of grid row bh: its length and first packed row (VARLEN), or the
// dense T and row 0.  A sequence longer than T, or outside the packed rows,
// is reported (FA_ERR_SEQLEN) and treated as empty by every role alike.
struct SeqSpan {
    int T, row0, head;
};
template <bool VARLEN>
__device__ __forceinline__ SeqSpan seq_span(const BwdParams& p, int bh) {
    if constexpr (!VARLEN) {
        return SeqSpan{p.T, 0, bh};
    } else {
        const int sq = bh % p.n_seq;
        SeqSpan r{0, p.cu_seqlens[sq], bh / p.n_seq};
        r.T = p.cu_seqlens[sq + 1] - r.row0;
        if (r.T < 0 || r.T > p.T || r.row0 < 0 || r.row0 + r.T > p.total) {
            atomicCAS(&g_status_bwd, 0, kStatusBadSeqlen);
            r.T = 0;
            r.row0 = 0;
        }
        return r;
    }
}

struct Ctl {
    volatile int* abort;
    unsigned long long timeout_ns;
};

// Slow path of a bounded wait.  kSleep: the hardware suspends the polling
// thread between checks (for waits off the critical path, so that polling
// does not take issue slots from busy warps on the same sub-partition);
// otherwise the thread polls back to back (lowest wake-up latency).
template <bool kSleep>
__device__ __noinline__ bool wait_slow(uint32_t bar, uint32_t parity, Ctl c) {
    uint64_t t0 = globaltimer_ns();
    while (true) {
        if (kSleep ? mbar_try_wait_sleep(bar, parity, 20000u) : mbar_try_wait(bar, parity)) return true;
        if (*c.abort) return false;
        if (globaltimer_ns() - t0 > c.timeout_ns) {
            *c.abort = 1;
            atomicCAS(&g_status_bwd, 0, kStatusTimeout);
            return false;
        }
    }
}
// Bounded wait: true when the phase completed, false when the CTA aborted
// (this wait ran out of time, or another role already gave up).
template <bool kSleep = true>
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, Ctl c) {
    if (mbar_try_wait(bar, parity)) return true;
    return wait_slow<kSleep>(bar, parity, c);
}
template <bool kSleep = true>
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, Ctl c) {
    int ok = 0;
    if ((threadIdx.x & 31) == 0) ok = wait_bar<kSleep>(bar, parity, c);
    return __shfl_sync(0xffffffffu, ok, 0) != 0;
}
// Bounded wait taken by every lane of a converged warp; the result is the same
// in all lanes.  The MMA warps wait this way: the issue loop then stays
// warp-uniform and elect.sync picks the lane that issues, which keeps the
// tensor pipe fed across waits and fences (a loop run by lane 0 alone leaves
// a gap of about 60 cycles at each wait).
template <bool kSleep = false>
__device__ __forceinline__ bool wait_all(uint32_t bar, uint32_t parity, Ctl c) {
    const bool ok = mbar_try_wait(bar, parity) || wait_slow<kSleep>(bar, parity, c);
    return __all_sync(0xffffffffu, ok);
}


// ---------------------------------------------------------------- preprocess
// D_i = rowsum(dO o O) ("Lab 06", section 4) and LSE2 = LSE * log2(e), both
// stored NEGATED (the main kernels add them with FMAs); rows t >= T of the
// padded vectors are 0.  8 elements per thread.
template <int D, bool VARLEN>
__global__ void __launch_bounds__(256) fa_bwd_pre_kernel(const __nv_bfloat16* __restrict__ o,
                                                         const __nv_bfloat16* __restrict__ dO,
                                                         const float* __restrict__ lse, float* __restrict__ dvec,
                                                         float* __restrict__ lse2, int BH, int T, int T_pad,
                                                         int* __restrict__ dq_next, const int* __restrict__ cu_seqlens,
                                                         int n_seq, int H, int total, float* __restrict__ dqacc) {
    constexpr int TPR = D / 8;            // threads per row
    constexpr int RPW = 32 / TPR;         // rows per warp
    if (blockIdx.x == 0 && threadIdx.x == 0) *dq_next = 0;  // the dQ kernel's item counter
    const long long rows = static_cast<long long>(BH) * T_pad;
    const int lane = threadIdx.x & 31, sub = lane % TPR;
    const long long n_warps = static_cast<long long>(gridDim.x) * (blockDim.x / 32);
    // warp-uniform loop: every lane reaches the shuffles below
    for (long long wr = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) / 32; wr * RPW < rows;
         wr += n_warps) {
        const long long r = wr * RPW + lane / TPR;
        const bool in = r < rows;
        const int bh = in ? static_cast<int>(r / T_pad) : 0, t = in ? static_cast<int>(r % T_pad) : T_pad;
        // this row's place in O / dO and in LSE; rows t >= len are padding
        int len = T;
        size_t orow = static_cast<size_t>(bh) * T + t, lrow = orow;
        if constexpr (VARLEN) {
            const int sq = bh % n_seq, h = bh / n_seq, row0 = cu_seqlens[sq];
            len = cu_seqlens[sq + 1] - row0;
            if (len < 0 || len > T || row0 < 0 || row0 + len > total) len = 0;  // reported by the main kernels
            orow = static_cast<size_t>(row0 + t) * H + h;
            lrow = static_cast<size_t>(h) * total + row0 + t;
        }
        float acc = 0.f;
        if (in && t < len) {
            const size_t off = orow * D + sub * 8;
            const uint4 a = *reinterpret_cast<const uint4*>(o + off);
            const uint4 b = *reinterpret_cast<const uint4*>(dO + off);
            const __nv_bfloat162* pa = reinterpret_cast<const __nv_bfloat162*>(&a);
            const __nv_bfloat162* pb = reinterpret_cast<const __nv_bfloat162*>(&b);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float2 fa2 = __bfloat1622float2(pa[e]);
                const float2 fb2 = __bfloat1622float2(pb[e]);
                acc = fmaf(fa2.x, fb2.x, acc);
                acc = fmaf(fa2.y, fb2.y, acc);
            }
        }
#pragma unroll
        for (int m = TPR / 2; m > 0; m >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, m, TPR);
        if (in && sub == 0) {
            dvec[r] = -acc;
            lse2[r] = (t < len) ? -lse[lrow] * kLog2e : 0.f;
        }
        if (dqacc != nullptr && in) {  // the fused backward's fp32 dQ accumulator starts at 0
            float4* z = reinterpret_cast<float4*>(dqacc + static_cast<size_t>(r) * D + sub * 8);
            z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
            z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
    }
}

// dQ = bf16(dQacc * scale) for the rows t < T of the fused backward's fp32
// accumulator (B*H, T_pad, D); 8 elements per thread.
template <int D>
__global__ void __launch_bounds__(256) fa_bwd_dq_convert_kernel(const float* __restrict__ acc,
                                                                __nv_bfloat16* __restrict__ dq, int BH, int T,
                                                                int T_pad, float scale) {
    constexpr int G = D / 8;
    const long long n = static_cast<long long>(BH) * T * G;
    for (long long g = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; g < n;
         g += static_cast<long long>(gridDim.x) * blockDim.x) {
        const long long row = g / G;
        const int c8 = static_cast<int>(g % G);
        const long long bh = row / T, t = row % T;
        const float4* src = reinterpret_cast<const float4*>(acc + (bh * T_pad + t) * D + c8 * 8);
        const float4 a = src[0], b = src[1];
        uint4 o;
        o.x = pack_bf16x2(a.x * scale, a.y * scale);
        o.y = pack_bf16x2(a.z * scale, a.w * scale);
        o.z = pack_bf16x2(b.x * scale, b.y * scale);
        o.w = pack_bf16x2(b.z * scale, b.w * scale);
        reinterpret_cast<uint4*>(dq + row * D + c8 * 8)[0] = o;
    }
}

// ---------------------------------------------------------------- dK / dV kernel
template <int D, bool CAUSAL, bool VARLEN, bool FUSE = false>
__global__ void __launch_bounds__(kBwdThreads, 1)
    fa_bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                       const __grid_constant__ CUtensorMap tm_dk, const __grid_constant__ CUtensorMap tm_dv,
                       const __grid_constant__ CUtensorMap tm_dqacc, BwdParams p) {
    using C = DkvCfg<D, FUSE>;
    constexpr int BM = C::BM;
    constexpr int NQS = C::kQStages, NDS = C::kDOStages;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = smem_window<C::kSlack>(smem_raw);
    const uint32_t sbase = smem_u32(smem);
    if constexpr (C::kSlack == 0) {
        if (sbase & 1023u) {
            if (threadIdx.x == 0) atomicCAS(&g_status_bwd, 0, kStatusSmemAlign);
            return;
        }
    }
    const uint32_t sK = sbase + C::kKOff, sV = sbase + C::kVOff;
    auto sQ = [&](int st) { return sbase + C::kQRingOff + st * C::kQStageBytes; };
    auto sLse = [&](int st) { return sQ(st) + C::kQBytes; };
    auto sDv = [&](int st) { return sLse(st) + BM * 4; };
    auto sdO = [&](int st) { return sbase + C::kDORingOff + st * C::kQBytes; };
    const uint32_t bars = sbase + C::kBarOff;
    const uint32_t kv_full = bars;
    auto q_full = [&](int st) { return bars + 8u * (1 + st); };
    auto q_empty = [&](int st) { return bars + 8u * (1 + NQS + st); };
    auto do_full = [&](int st) { return bars + 8u * (1 + 2 * NQS + st); };
    auto do_empty = [&](int st) { return bars + 8u * (1 + 2 * NQS + NDS + st); };
    const uint32_t b0 = bars + 8u * (1 + 2 * NQS + 2 * NDS);
    const uint32_t s_full = b0;         // S^T(i) in TMEM
    const uint32_t dp_full = b0 + 8;    // dP^T(i) in TMEM
    const uint32_t p_full = b0 + 16;    // P^T(i) written over S^T(i)        (8 compute warps)
    const uint32_t ds_full = b0 + 24;   // dS^T(i) written over dP^T(i)      (8 compute warps)
    const uint32_t dkv_full = b0 + 32;  // every dK / dV MMA done
    const uint32_t mma_done = b0 + 40;
    auto epi_bar = [&](int hh) { return b0 + 48 + 8u * hh; };  // warpgroup hh staged its output (4 warps)
    // FUSE: dQ buffer b holds a finished dS K (MMA) / was read out (8 compute warps)
    auto dq_full = [&](int b) { return b0 + 64 + 8u * b; };
    auto dq_empty = [&](int b) { return b0 + 80 + 8u * b; };
    const uint32_t sDS = sbase + C::kDSOff, sStg = sbase + C::kStgOff;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kMiscOff);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kMiscOff + 4);
    const Ctl ctl{abort_flag, p.timeout_ns};

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // The dQ grid needs nothing from this one: it may launch as soon as every
    // CTA of this grid has started (its CTAs then fill SMs freed in the tail).
    griddep_launch_dependents();
    // CTA order.  Head major: the key tiles of one head run together (their Q
    // and dO stay in L2), heavy key tiles first within a head.  Key tile
    // major: every head's heavy key tiles first, which shortens the causal
    // tail when there are few waves of CTAs (grouped heads make fewer,
    // heavier CTAs).  With grouped heads the CTA walks the query tiles of
    // every query head that shares this K/V head, so dK and dV sum over the
    // group in TMEM.
    const int bh = p.kt_major ? static_cast<int>(blockIdx.x % p.BH) : static_cast<int>(blockIdx.x / p.n_kt);
    const int kt = p.kt_major ? static_cast<int>(blockIdx.x / p.BH) : static_cast<int>(blockIdx.x % p.n_kt);
    // the sequence of this row of the grid (packed batches: its own length and rows)
    const SeqSpan span = seq_span<VARLEN>(p, bh);
    const int T = span.T;
    if (kt * kBN >= T) return;  // a shorter sequence has fewer key tiles: the whole CTA leaves
    // TMA coordinates (y, z) of the 128-row tile starting at row r0 of grid row bhx
    auto tile_yz = [&](int r0, int bhx, int& y, int& z) {
        if constexpr (VARLEN) {
            y = span.head;  // packed (total, H, D): (D, H, rows)
            z = span.row0 + r0;
        } else {
            y = r0;
            z = bhx;
        }
    };
    const int q_begin = bwd_q_begin(T, CAUSAL, kt, BM), q_end = bwd_q_end(T, BM);
    const int n_q = q_end - q_begin;
    const int n_it = n_q * p.group;
    const int bhq0 = (bh / p.Hkv) * p.Hq + (bh % p.Hkv) * p.group;  // first query head of the group
    auto q_tile_of = [&](int it) { return q_begin + it % n_q; };
    auto q_head_of = [&](int it) { return bhq0 + it / n_q; };

    if (tid == 0) {
        mbar_init(kv_full, 1);
        for (int st = 0; st < NQS; ++st) {
            mbar_init(q_full(st), 1);
            mbar_init(q_empty(st), 1);
        }
        for (int st = 0; st < NDS; ++st) {
            mbar_init(do_full(st), 1);
            mbar_init(do_empty(st), 1);
        }
        mbar_init(s_full, 1);
        mbar_init(dp_full, 1);
        mbar_init(p_full, 8);
        mbar_init(ds_full, 8);
        mbar_init(dkv_full, 1);
        mbar_init(mma_done, 1);
        mbar_init(epi_bar(0), 4);
        mbar_init(epi_bar(1), 4);
        if constexpr (FUSE) {
            for (int b = 0; b < 2; ++b) {
                mbar_init(dq_full(b), 1);
                mbar_init(dq_empty(b), 8);
            }
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 9) {
        tmem_alloc(smem_u32(tmem_slot), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(tmem_slot);

    if (warp == 8) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            uint32_t q_armed = 0, do_armed = 0;  // fills issued per ring
            int q_skipped = -1;                  // Q fill the test hook dropped
            const uint64_t pol_kv = l2_policy_evict_first();
            const uint64_t pol_q = l2_policy_evict_last();
            int ky, kz;
            tile_yz(kt * kBN, bh, ky, kz);
            // the key tile starts inside its sequence and its head exists
            const bool kv_ok = FA_CHECK(kt * kBN < T && bh >= 0 && bh < p.BH, &g_status_bwd, abort_flag);
            if (kv_ok) mbar_arrive_expect_tx(kv_full, 2 * C::kKVBytes);
            for (int a = 0; kv_ok && a < C::kAtomsD; ++a) {
                tma_load_3d_hint(sK + a * 128 * 128, &tm_k, kv_full, 64 * a, ky, kz, pol_kv);
                tma_load_3d_hint(sV + a * 128 * 128, &tm_v, kv_full, 64 * a, ky, kz, pol_kv);
            }
            for (int it = 0; it < n_it; ++it) {
                const int qt = q_tile_of(it), bhq = q_head_of(it);
                {   // Q tile with its -LSE2 and -D vectors
                    const int st = it % NQS;
                    if (!wait_bar(q_empty(st), ((it / NQS) & 1) ^ 1, ctl)) break;
                    const uint32_t fb = q_full(st);
                    const size_t voff = static_cast<size_t>(bhq) * p.T_pad + static_cast<size_t>(qt) * BM;
                    // the query tile and head exist, the stage lies inside the window and the
                    // -LSE2 / -D slices inside their (B*Hq, T_pad) vectors
                    if (!FA_CHECK(qt >= 0 && qt * BM < T && bhq >= 0 && bhq < p.BH * p.group && st < NQS &&
                                      C::kQRingOff + (st + 1) * C::kQStageBytes <= C::kDORingOff &&
                                      voff + BM <= static_cast<size_t>(p.BH) * p.group * p.T_pad,
                                  &g_status_bwd, abort_flag))
                        break;
                    // test hook: never deliver the third Q tile (the first when there are fewer)
                    if (it == (n_it > 2 ? 2 : 0) && p.inject == 2 && blockIdx.x == 0) {
                        q_skipped = static_cast<int>(q_armed++);
                    } else {
                        mbar_arrive_expect_tx(fb, C::kQBytes + 2 * BM * 4);
                        ++q_armed;
                        int qy, qz;
                        tile_yz(qt * BM, bhq, qy, qz);
                        for (int a = 0; a < C::kAtomsD; ++a)
                            tma_load_3d_hint(sQ(st) + a * BM * 128, &tm_q, fb, 64 * a, qy, qz, pol_q);
                        bulk_load_1d(sLse(st), p.lse2 + voff, BM * 4, fb);
                        bulk_load_1d(sDv(st), p.dvec + voff, BM * 4, fb);
                    }
                }
                {   // dO tile
                    const int st = it % NDS;
                    if (!wait_bar(do_empty(st), ((it / NDS) & 1) ^ 1, ctl)) break;
                    if (!FA_CHECK(st < NDS && C::kDORingOff + (st + 1) * C::kQBytes <= C::kBarOff, &g_status_bwd,
                                  abort_flag))
                        break;
                    const uint32_t fb = do_full(st);
                    mbar_arrive_expect_tx(fb, C::kQBytes);
                    ++do_armed;
                    int qy, qz;
                    tile_yz(qt * BM, bhq, qy, qz);
                    for (int a = 0; a < C::kAtomsD; ++a)
                        tma_load_3d_hint(sdO(st) + a * BM * 128, &tm_do, fb, 64 * a, qy, qz, pol_q);
                }
            }
            // drain: copies still in flight must land before the CTA exits
            volatile int never = 0;
            Ctl drain{&never, 100000000ull};
            if (kv_ok) wait_bar(kv_full, 0, drain);
            for (uint32_t f = q_armed > NQS ? q_armed - NQS : 0; f < q_armed; ++f)
                if (static_cast<int>(f) != q_skipped) wait_bar(q_full(f % NQS), (f / NQS) & 1, drain);
            for (uint32_t f = do_armed > NDS ? do_armed - NDS : 0; f < do_armed; ++f)
                wait_bar(do_full(f % NDS), (f / NDS) & 1, drain);
        }
    } else if (warp == 9) {
        // ------------------------------------------------------------ MMA issuer
        // The whole warp runs the loop; the elected lane issues and commits.
        {
            const bool leader = elect_one_sync();
            // Descriptors are built once; a stage / k-step is an offset in 16-byte units.
            const SDesc dK_km = sdesc_make(sK, 16, 1024), dV_km = sdesc_make(sV, 16, 1024);
            const SDesc dQ_km = sdesc_make(sQ(0), 16, 1024), dO_km = sdesc_make(sdO(0), 16, 1024);
            const SDesc dQ_mn = sdesc_make(sQ(0), BM * 128, 1024), dO_mn = sdesc_make(sdO(0), BM * 128, 1024);
            // FUSE: dS (queries contiguous, 64-query column blocks 128 x 128 B apart) and K
            // (D contiguous) as the MN-major operands of dQ = dS K
            const SDesc dDS_mn = sdesc_make(sDS, 128 * 128, 1024), dK_mn = sdesc_make(sK, 128 * 128, 1024);
            constexpr uint32_t kQStage16 = C::kQStageBytes >> 4, kDOStage16 = C::kQBytes >> 4;
            constexpr int NKV = BM / 16;  // k-steps of dV and dK
            // S^T = K Q^T: M = 128 keys, N = BM, K = D (both K-major)
            auto issue_s = [&](int st) {
                const uint32_t so = st * kQStage16;
#pragma unroll
                for (int s = 0; s < D / 16; ++s)
                    if (leader) mma_ss_d(tmem + C::kS, dK_km, ((s >> 2) * (128 * 128) + (s & 3) * 32) >> 4, dQ_km,
                             so + (((s >> 2) * (BM * 128) + (s & 3) * 32) >> 4), C::kIdescS, s > 0);
                if (leader) mma_commit(s_full);
            };
            // dP^T = V dO^T
            auto issue_dp = [&](int st) {
                const uint32_t so = st * kDOStage16;
#pragma unroll
                for (int s = 0; s < D / 16; ++s)
                    if (leader) mma_ss_d(tmem + C::kDP, dV_km, ((s >> 2) * (128 * 128) + (s & 3) * 32) >> 4, dO_km,
                             so + (((s >> 2) * (BM * 128) + (s & 3) * 32) >> 4), C::kIdescS, s > 0);
                if (leader) mma_commit(dp_full);
            };
            // Per query tile i, in issue order:
            //   dV += P^T(i) dO(i)         P^T from TMEM (over S^T(i)), dO MN-major
            //   S^T(i+1)                   into the S^T columns (dV(i) was the last reader)
            //   dK += dS^T(i) Q(i)         dS^T from TMEM (over dP^T(i)), Q MN-major
            //   dP^T(i+1)                  into the dP^T columns (dK(i) was the last reader)
            // The compute warps turn dP^T(i) into dS^T(i) while dV(i) and S^T(i+1)
            // run, and S^T(i+1) into P^T(i+1) while dK(i) and dP^T(i+1) run.
            if (!wait_all(kv_full, 0, ctl)) goto mma_teardown;
            if (!wait_all(q_full(0), 0, ctl)) goto mma_teardown;
            tc_fence_after();
            issue_s(0);
            if (!wait_all(do_full(0), 0, ctl)) goto mma_teardown;
            tc_fence_after();
            issue_dp(0);
            for (int it = 0; it < n_it; ++it) {
                const int qs = it % NQS, ds = it % NDS;
                if (!wait_all(p_full, it & 1, ctl)) goto mma_teardown;
                tc_fence_after();
#pragma unroll
                for (int s = 0; s < NKV; ++s)
                    if (leader) mma_ts_d(tmem + C::kDV, tmem + C::kP + s * 8, dO_mn, ds * kDOStage16 + s * (2048 >> 4),
                             C::kIdescDKV, (it > 0 || s > 0) ? 1u : 0u);
                if (leader) mma_commit(do_empty(ds));
                if (it + 1 < n_it) {
                    if (!wait_all(q_full((it + 1) % NQS), ((it + 1) / NQS) & 1, ctl))
                        goto mma_teardown;
                    tc_fence_after();
                    issue_s((it + 1) % NQS);
                }
                if (!wait_all(ds_full, it & 1, ctl)) goto mma_teardown;
                tc_fence_after();
#pragma unroll
                for (int s = 0; s < NKV; ++s)
                    if (leader) mma_ts_d(tmem + C::kDK, tmem + C::kDS + s * 8, dQ_mn, qs * kQStage16 + s * (2048 >> 4),
                             C::kIdescDKV, (it > 0 || s > 0) ? 1u : 0u);
                if (leader) mma_commit(q_empty(qs));
                if (it + 1 < n_it) {
                    const int ds1 = (it + 1) % NDS;
                    if (!wait_all(do_full(ds1), ((it + 1) / NDS) & 1, ctl)) goto mma_teardown;
                    tc_fence_after();
                    issue_dp(ds1);
                }
                if constexpr (FUSE) {
                    // dQ(it) = dS(it) K into TMEM buffer it & 1, once the compute warps have
                    // read out dQ(it - 2) from it.  dS(it) has been in shared-memory buffer
                    // it & 1 since ds_full; issued after dP^T(it+1), so the compute warps
                    // get dP^T(it+1) without waiting for it.
                    const int b = it & 1;
                    if (it >= 2 && !wait_all(dq_empty(b), ((it >> 1) - 1) & 1, ctl)) goto mma_teardown;
                    tc_fence_after();
                    const uint32_t dso = static_cast<uint32_t>(b * C::kDSBufBytes) >> 4;
#pragma unroll
                    for (int s = 0; s < 128 / 16; ++s)
                        if (leader) mma_ss_d(tmem + C::kDQ(b), dDS_mn, dso + s * (2048 >> 4), dK_mn, s * (2048 >> 4),
                                             C::kIdescDQ, s > 0 ? 1u : 0u);
                    if (leader) mma_commit(dq_full(b));
                }
            }
            if (leader) mma_commit(dkv_full);
        mma_teardown:
            if (leader) {
                mma_commit(mma_done);
                volatile int never = 0;
                Ctl drain{&never, 100000000ull};
                wait_bar(mma_done, 0, drain);
            }
            __syncwarp();
        }
    } else {
        // ------------------------------------------------------------ compute (warps 0-7) + dK/dV epilogue
        // Warpgroup h takes query columns 64h .. 64h+63.  TMEM is read and written
        // in the 16-lane shapes: for half hf of the warp's 32 lanes, register
        // 4k + i of a 16x256b load holds key row 16 hf + t/4 (+8 for i >= 2) and
        // query column 64h + 8k + 2 (t % 4) + (i % 2); register 2k + i of a
        // 16x128b store goes to key row 16 hf + t/4 (+8 for i = 1), pair column
        // 4k + t % 4.  So each thread needs the -LSE2 and -D values of only 16
        // query columns, 4 distinct addresses per warp and load.
        const int h = warp >> 2, wq = warp & 3, t4 = lane & 3;
        const int key_base = kt * kBN + 32 * wq + (lane >> 2);  // + 16 hf + 8 i2
        const uint32_t lane_base = tmem + ((32u * wq) << 16);
        const float eff = p.sl2_eff, sl2 = p.sl2;
        const bool prescale = p.prescale != 0;
        const uint64_t eff2 = f2(eff, eff);
        bool ok = true;
        // FUSE: read dQ(j) = dS(j) K out of TMEM buffer j & 1 (this warpgroup's 32 of
        // the D columns, one query row per thread), stage the warp's 32 rows in its
        // own 4 KB of shared memory in the 128-byte swizzled layout of the
        // accumulator's tensor map, and add them into the fp32 accumulator with
        // one TMA reduce from lane 0.  Each warp reuses its staging only after its
        // own previous reduce has read it, so the warps never wait for each other.
        // Every wait is bounded; false when the CTA gave up.
        const uint32_t stg_w = sStg + (h * 4 + wq) * 4096;
        auto drain_dq = [&](int j) -> bool {
            const int b = j & 1;
            if (!warp_wait(dq_full(b), (j >> 1) & 1, ctl)) return false;
            tc_fence_after();
            uint32_t v[32];
            tmem_ld32(lane_base + C::kDQ(b) + 32 * h, v);
            tmem_ld_wait();
            reg_fence32(v);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(dq_empty(b));
                bulk_wait_read0();  // this warp's previous reduce has read its staging
            }
            __syncwarp();
            const uint32_t rowa = stg_w + lane * 128;
#pragma unroll
            for (int c = 0; c < 8; ++c)
                st_shared_v4(rowa + ((c ^ (lane & 7)) << 4), v[4 * c], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3]);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                const int qtj = q_tile_of(j), bhqj = q_head_of(j);
                if (FA_CHECK(qtj * BM < T && bhqj >= 0 && bhqj < p.BH * p.group, &g_status_bwd, abort_flag)) {
                    tma_reduce_add_3d(&tm_dqacc, stg_w, 32 * h, qtj * BM + 32 * wq, bhqj);
                    bulk_commit();
                }
            }
            return true;
        };
        for (int it = 0; it < n_it; ++it) {
            const int st = it % NQS;
            const int qt = q_tile_of(it), q0 = qt * BM;
            const bool masked = bwd_tile_class(T, CAUSAL, BM, qt, kt) == kMasked;
            if (!warp_wait(q_full(st), (it / NQS) & 1, ctl) || !warp_wait<false>(s_full, it & 1, ctl)) {
                ok = false;
                break;
            }
            tc_fence_after();
            // this thread's 16 query columns: 64h + 8k + 2 t4 + {0, 1}
            const float2* lse2v = reinterpret_cast<const float2*>(smem + (sLse(st) - sbase)) + 32 * h + t4;
            const float2* dv2v = reinterpret_cast<const float2*>(smem + (sDv(st) - sbase)) + 32 * h + t4;
            uint32_t sr[64];
            tmem_ld_16x256b_x8(lane_base + C::kS + 64 * h, sr);
            tmem_ld_16x256b_x8(lane_base + (16u << 16) + C::kS + 64 * h, sr + 32);
            tmem_ld_wait();
            reg_fence32(sr);
            reg_fence32(sr + 32);
            float* pf = reinterpret_cast<float*>(sr);
            if (prescale) {
#pragma unroll
                for (int e = 0; e < 64; ++e) pf[e] *= sl2;
            }
            // P^T = exp2(S^T c - LSE2): one packed FMA per pair of columns
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const float2 l2 = lse2v[4 * k];
                const uint64_t nl = f2(l2.x, l2.y);
#pragma unroll
                for (int r = 0; r < 4; ++r) {  // r = 2 hf + i2
                    const int e = 32 * (r >> 1) + 4 * k + 2 * (r & 1);
                    float x0, x1;
                    f2_split(fma2(f2(pf[e], pf[e + 1]), eff2, nl), x0, x1);
                    pf[e] = ex2_approx(x0);
                    pf[e + 1] = ex2_approx(x1);
                }
            }
            if (masked) {
#pragma unroll
                for (int k = 0; k < 8; ++k)
#pragma unroll
                    for (int r = 0; r < 4; ++r) {
                        const int e = 32 * (r >> 1) + 4 * k + 2 * (r & 1);
                        const int key = key_base + 16 * (r >> 1) + 8 * (r & 1);
                        const int q = q0 + 64 * h + 8 * k + 2 * t4;
                        if (!bwd_elem_visible(T, CAUSAL, q, key)) pf[e] = 0.f;
                        if (!bwd_elem_visible(T, CAUSAL, q + 1, key)) pf[e + 1] = 0.f;
                    }
            }
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                uint32_t pk[16];
#pragma unroll
                for (int k = 0; k < 8; ++k)
#pragma unroll
                    for (int i2 = 0; i2 < 2; ++i2) {
                        const int e = 32 * hf + 4 * k + 2 * i2;
                        pk[2 * k + i2] = pack_bf16x2(pf[e], pf[e + 1]);
                    }
                tmem_st_16x128b_x8(lane_base + ((16u * hf) << 16) + C::kP + 32 * h, pk);
            }
            // dV(it) needs only P^T: release it before dP^T is even ready
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(p_full);
            if (!warp_wait<false>(dp_full, it & 1, ctl)) {
                ok = false;
                break;
            }
            tc_fence_after();
            uint32_t dr[64];
            tmem_ld_16x256b_x8(lane_base + C::kDP + 64 * h, dr);
            tmem_ld_16x256b_x8(lane_base + (16u << 16) + C::kDP + 64 * h, dr + 32);
            tmem_ld_wait();
            reg_fence32(dr);
            reg_fence32(dr + 32);
            // dS^T = P^T o (dP^T - D), bf16 pairs written over the dP^T columns this
            // warpgroup has just read (dP^T(it) completing implies dK(it-1), the
            // previous reader of those columns, completed: it was issued before)
            uint32_t dsw[32];
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const float2 d2 = dv2v[4 * k];
                const uint64_t nd = f2(d2.x, d2.y);
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    const int e = 32 * (r >> 1) + 4 * k + 2 * (r & 1);
                    const uint64_t t2 = add2(f2(__uint_as_float(dr[e]), __uint_as_float(dr[e + 1])), nd);
                    float d0, d1;
                    f2_split(mul2(f2(pf[e], pf[e + 1]), t2), d0, d1);
                    dsw[16 * (r >> 1) + 2 * k + (r & 1)] = pack_bf16x2(d0, d1);
                }
            }
            tmem_st_16x128b_x8(lane_base + C::kDS + 32 * h, dsw);
            tmem_st_16x128b_x8(lane_base + (16u << 16) + C::kDS + 32 * h, dsw + 16);
            if constexpr (FUSE) {
                // dS into shared-memory buffer it & 1 for dQ = dS K, queries contiguous:
                // key row k of this warpgroup's 64-query block at k * 128 bytes,
                // 16-byte chunk c (queries 8c .. 8c+7) at position c ^ (k % 8).  The
                // registers are already in the 8 x 8 fragment layout (row = key,
                // column pair = two queries), so each stmatrix writes four such
                // blocks.  dQ(it - 2), the last reader of this buffer, was issued
                // before dP^T(it), so it completed before dP^T(it) did.
                const int rr = lane & 7, mi = lane >> 3;
                const uint32_t sDSb = sDS + (it & 1) * C::kDSBufBytes;
#pragma unroll
                for (int hf = 0; hf < 2; ++hf)
#pragma unroll
                    for (int i2 = 0; i2 < 2; ++i2) {
                        const int key = 32 * wq + 16 * hf + 8 * i2 + rr;
                        const uint32_t rowa = sDSb + h * (128 * 128) + key * 128;
                        const int b = 16 * hf + i2;
#pragma unroll
                        for (int g = 0; g < 2; ++g)
                            stmatrix_x4(rowa + (((4 * g + mi) ^ rr) << 4), dsw[b + 8 * g], dsw[b + 8 * g + 2],
                                        dsw[b + 8 * g + 4], dsw[b + 8 * g + 6]);
                    }
                fence_proxy_async_smem();
            }
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(ds_full);
            // FUSE: the previous query tile's dQ (issued after dP^T(it)) is read out
            // while the tensor pipe runs dK(it), dP^T(it+1) and dQ(it)
            if constexpr (FUSE) {
                if (it > 0 && !drain_dq(it - 1)) {
                    ok = false;
                    break;
                }
            }
        }
        if constexpr (FUSE) {
            if (ok && n_it > 0 && !drain_dq(n_it - 1)) ok = false;
        }
        // epilogue: warpgroup 0 stores dK * scale, warpgroup 1 stores dV.  Each
        // stages its 128 x D bf16 tile in shared memory in the 128-byte swizzled
        // layout of the tensor maps (dK in Q ring stage 0, dV in dO ring stage 0:
        // every MMA has completed, so nothing reads them any more) and one
        // thread writes it out with TMA stores, which clip rows past T.
        if (VARLEN && ok && warp_wait(dkv_full, 0, ctl)) {
            // packed rows past this sequence's end belong to the next one: row by row
            tc_fence_after();
            const int key = kt * kBN + 32 * wq + lane;  // 32x32b shape: this thread's own lane
            const uint32_t col = h ? C::kDV : C::kDK;
            const float mul = h ? 1.f : p.scale;
            __nv_bfloat16* out = (h ? p.dv : p.dk) + (static_cast<size_t>(span.row0 + key) * p.Hq + span.head) * D;
#pragma unroll
            for (int ch = 0; ch < D / 32; ++ch) {
                uint32_t v[32];
                tmem_ld32(lane_base + col + 32 * ch, v);
                tmem_ld_wait();
                reg_fence32(v);
                if (key < T) {
                    uint4* dst = reinterpret_cast<uint4*>(out + 32 * ch);
#pragma unroll
                    for (int g = 0; g < 4; ++g) {
                        uint4 w;
                        w.x = pack_bf16x2(__uint_as_float(v[8 * g + 0]) * mul, __uint_as_float(v[8 * g + 1]) * mul);
                        w.y = pack_bf16x2(__uint_as_float(v[8 * g + 2]) * mul, __uint_as_float(v[8 * g + 3]) * mul);
                        w.z = pack_bf16x2(__uint_as_float(v[8 * g + 4]) * mul, __uint_as_float(v[8 * g + 5]) * mul);
                        w.w = pack_bf16x2(__uint_as_float(v[8 * g + 6]) * mul, __uint_as_float(v[8 * g + 7]) * mul);
                        dst[g] = w;
                    }
                }
            }
        } else if (!VARLEN && ok && warp_wait(dkv_full, 0, ctl)) {
            tc_fence_after();
            const uint32_t row = 32u * wq + lane;  // 32x32b shape: this thread's own lane (key row)
            const uint32_t col = h ? C::kDV : C::kDK;
            const float mul = h ? 1.f : p.scale;
            const uint32_t stage = h ? sdO(0) : sQ(0);
#pragma unroll
            for (int ch = 0; ch < D / 32; ++ch) {
                uint32_t v[32];
                tmem_ld32(lane_base + col + 32 * ch, v);
                tmem_ld_wait();
                reg_fence32(v);
                const uint32_t atom = stage + (ch >> 1) * (BM * 128);
#pragma unroll
                for (int g = 0; g < 4; ++g) {
                    uint32_t w4[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        w4[e] = pack_bf16x2(__uint_as_float(v[8 * g + 2 * e]) * mul,
                                            __uint_as_float(v[8 * g + 2 * e + 1]) * mul);
                    st_shared_v4(atom + sw128_off(row, (ch & 1) * 4 + g), w4[0], w4[1], w4[2], w4[3]);
                }
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(epi_bar(h));
            if (wq == 0 && lane == 0 && wait_bar(epi_bar(h), 0, ctl) &&
                FA_CHECK(kt * kBN < T && bh >= 0 && bh < p.BH, &g_status_bwd, abort_flag)) {
                for (int a = 0; a < C::kAtomsD; ++a)
                    tma_store_3d(h ? &tm_dv : &tm_dk, stage + a * (BM * 128), 64 * a, kt * kBN, bh);
                bulk_commit();
                bulk_wait0();
            }
        }
        // FUSE: the dQ reduce-adds read shared memory and must land before the CTA exits
        if (FUSE && lane == 0) bulk_wait0();
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 9) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// ---------------------------------------------------------------- dQ kernel
// Work items are (query tile, query head) pairs, handed out one at a time from
// a counter in global memory: a persistent CTA (one per SM) takes the next
// item whenever it is ready for one, so the CTAs that start early (the grid
// may launch during the dK/dV grid's tail) or draw light items do more of
// them.  Item w in order:
//   causal masking  heaviest query tiles first across all heads (a tile sees
//                   more key tiles the later it is), which keeps the end of
//                   the grid balanced;
//   no masking      head by head (every item weighs the same), so the items in
//                   flight cover a few heads and their K and V stay in L2.
template <bool CAUSAL>
__device__ __forceinline__ void dq_item_at(int w, const BwdParams& p, int& bh, int& qt) {
    if constexpr (CAUSAL) {
        bh = w % p.BH;
        qt = p.n_kt - 1 - w / p.BH;
    } else {
        bh = w / p.n_kt;
        qt = w % p.n_kt;
    }
}
constexpr int kDqItemRing = 4;  // item numbers passed from the producer to the other roles

template <int D, bool CAUSAL, bool VARLEN>
__global__ void __launch_bounds__(kBwdThreads, 1)
    fa_bwd_dq_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                     BwdParams p) {
    using C = DqCfg<D>;
    constexpr int NKS = C::kKStages, NVS = C::kVStages;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = smem_window<C::kSlack>(smem_raw);
    const uint32_t sbase = smem_u32(smem);
    if constexpr (C::kSlack == 0) {
        if (sbase & 1023u) {
            if (threadIdx.x == 0) atomicCAS(&g_status_bwd, 0, kStatusSmemAlign);
            return;
        }
    }
    const uint32_t sQ = sbase + C::kQOff, sdO = sbase + C::kDOOff;
    auto sK = [&](int st) { return sbase + C::kKOff + st * C::kTileBytes; };
    auto sV = [&](int st) { return sbase + C::kVOff + st * C::kTileBytes; };
    const uint32_t bars = sbase + C::kBarOff;
    const uint32_t qdo_full = bars, qdo_empty = bars + 8;
    auto k_full = [&](int st) { return bars + 8u * (2 + st); };
    auto k_empty = [&](int st) { return bars + 8u * (2 + NKS + st); };
    auto v_full = [&](int st) { return bars + 8u * (2 + 2 * NKS + st); };
    auto v_empty = [&](int st) { return bars + 8u * (2 + 2 * NKS + NVS + st); };
    const uint32_t b0 = bars + 8u * (2 + 2 * NKS + 2 * NVS);
    auto s_full = [&](int b) { return b0 + 8u * b; };  // S number g lands in buffer g & 1
    const uint32_t dp_full = b0 + 16;                   // dP in TMEM
    const uint32_t ds_full = b0 + 24;                   // dS written over S, dP read (8 warps)
    const uint32_t dq_full = b0 + 32;                   // every dQ MMA of the item done
    const uint32_t dq_empty = b0 + 40;                  // dQ read out of TMEM (8 warps)
    const uint32_t mma_done = b0 + 48;
    // item ring: the producer writes item numbers, the MMA warp and the 8 compute warps read them
    auto item_full = [&](int i) { return b0 + 56 + 8u * i; };
    auto item_empty = [&](int i) { return b0 + 56 + 8u * (kDqItemRing + i); };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kMiscOff);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kMiscOff + 4);
    volatile int* item_ring = reinterpret_cast<volatile int*>(smem + C::kMiscOff + 16);
    const Ctl ctl{abort_flag, p.timeout_ns};

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int T = p.T;
    struct Item {
        int bh, qt, bh_kv, n;
        int T, row0, head;  // its sequence: length, first packed row, head (VARLEN)
    };
    auto item = [&](int bh, int qt) {
        Item it;
        it.bh = bh;
        it.qt = qt;
        it.bh_kv = (it.bh / p.Hq) * p.Hkv + (it.bh % p.Hq) / p.group;
        const SeqSpan span = seq_span<VARLEN>(p, bh);
        it.T = span.T;
        it.row0 = span.row0;
        it.head = span.head;
        it.n = it.qt * 128 < it.T ? fwd_num_kv_tiles(it.T, CAUSAL, it.qt) : 0;  // key tiles this query tile sees
        return it;
    };
    // TMA coordinates (y, z) of the 128-row tile starting at row r0 of grid row bhx of item it
    auto tile_yz = [&](const Item& it, int r0, int bhx, int& y, int& z) {
        if constexpr (VARLEN) {
            y = it.head;  // packed (total, H, D): (D, H, rows)
            z = it.row0 + r0;
        } else {
            y = r0;
            z = bhx;
        }
    };

    if (tid == 0) {
        mbar_init(qdo_full, 1);
        mbar_init(qdo_empty, 1);
        for (int st = 0; st < NKS; ++st) {
            mbar_init(k_full(st), 1);
            mbar_init(k_empty(st), 1);
        }
        for (int st = 0; st < NVS; ++st) {
            mbar_init(v_full(st), 1);
            mbar_init(v_empty(st), 1);
        }
        mbar_init(s_full(0), 1);
        mbar_init(s_full(1), 1);
        mbar_init(dp_full, 1);
        mbar_init(ds_full, 8);
        mbar_init(dq_full, 1);
        mbar_init(dq_empty, 8);
        mbar_init(mma_done, 1);
        for (int i = 0; i < kDqItemRing; ++i) {
            mbar_init(item_full(i), 1);
            mbar_init(item_empty(i), 9);  // the MMA warp and the 8 compute warps
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 9) {
        tmem_alloc(smem_u32(tmem_slot), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(tmem_slot);

    if (warp == 8) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            uint32_t kf = 0, vf = 0, qf = 0;  // fills issued (K ring, V ring, Q/dO pair)
            int k_skipped = -1;               // K fill the test hook dropped
            const uint64_t pol_kv = l2_policy_evict_last();   // K, V of a head serve all its query tiles
            const uint64_t pol_q = l2_policy_evict_first();
            for (int k = 0;; ++k) {
                // take the next item and pass its number on (a number past the
                // last item tells the other roles to stop)
                const int slot = k % kDqItemRing;
                if (!wait_bar(item_empty(slot), ((k / kDqItemRing) & 1) ^ 1, ctl)) break;
                // (query tiles past a shorter sequence's end are skipped here, so
                // the other roles only see items with work)
                int w;
                Item it;
                while (true) {
                    w = atomicAdd(p.dq_next, 1);
                    if (w >= p.n_items) break;
                    int w_bh, w_qt;
                    dq_item_at<CAUSAL>(w, p, w_bh, w_qt);
                    it = item(w_bh, w_qt);
                    if (it.n > 0) break;
                }
                item_ring[slot] = w;
                mbar_arrive(item_full(slot));
                if (w >= p.n_items) break;
                if (!wait_bar(qdo_empty, (qf & 1) ^ 1, ctl)) break;
                // the item's query tile starts inside its sequence and its heads exist
                if (!FA_CHECK(it.qt >= 0 && it.qt * 128 < it.T && it.bh >= 0 && it.bh < p.BH && it.bh_kv >= 0 &&
                                  it.bh_kv < p.BH / p.group,
                              &g_status_bwd, abort_flag))
                    break;
                mbar_arrive_expect_tx(qdo_full, 2 * C::kTileBytes);
                ++qf;
                int qy, qz;
                tile_yz(it, it.qt * 128, it.bh, qy, qz);
                for (int a = 0; a < C::kAtomsD; ++a) {
                    tma_load_3d_hint(sQ + a * 128 * 128, &tm_q, qdo_full, 64 * a, qy, qz, pol_q);
                    tma_load_3d_hint(sdO + a * 128 * 128, &tm_do, qdo_full, 64 * a, qy, qz, pol_q);
                }
                bool fail = false;
                for (int j = 0; j < it.n; ++j) {
                    {
                        const int st = kf % NKS;
                        if (!wait_bar(k_empty(st), ((kf / NKS) & 1) ^ 1, ctl) ||
                            !FA_CHECK(j * kBN < it.T && st < NKS && C::kKOff + (st + 1) * C::kTileBytes <= C::kVOff,
                                      &g_status_bwd, abort_flag)) {
                            fail = true;
                            break;
                        }
                        if (kf == 0 && p.inject == 3 && blockIdx.x == 0) {  // test hook: never deliver this tile
                            k_skipped = static_cast<int>(kf++);
                        } else {
                            mbar_arrive_expect_tx(k_full(st), C::kTileBytes);
                            ++kf;
                            int ky, kz;
                            tile_yz(it, j * kBN, it.bh_kv, ky, kz);
                            for (int a = 0; a < C::kAtomsD; ++a)
                                tma_load_3d_hint(sK(st) + a * 128 * 128, &tm_k, k_full(st), 64 * a, ky, kz, pol_kv);
                        }
                    }
                    {
                        const int st = vf % NVS;
                        if (!wait_bar(v_empty(st), ((vf / NVS) & 1) ^ 1, ctl) ||
                            !FA_CHECK(st < NVS && C::kVOff + (st + 1) * C::kTileBytes <= C::kBarOff, &g_status_bwd,
                                      abort_flag)) {
                            fail = true;
                            break;
                        }
                        mbar_arrive_expect_tx(v_full(st), C::kTileBytes);
                        ++vf;
                        int vy, vz;
                        tile_yz(it, j * kBN, it.bh_kv, vy, vz);
                        for (int a = 0; a < C::kAtomsD; ++a)
                            tma_load_3d_hint(sV(st) + a * 128 * 128, &tm_v, v_full(st), 64 * a, vy, vz, pol_kv);
                    }
                }
                if (fail) break;
            }
            // drain: copies still in flight must land before the CTA exits
            volatile int never = 0;
            Ctl drain{&never, 100000000ull};
            if (qf) wait_bar(qdo_full, (qf - 1) & 1, drain);
            for (uint32_t f = kf > NKS ? kf - NKS : 0; f < kf; ++f)
                if (static_cast<int>(f) != k_skipped) wait_bar(k_full(f % NKS), (f / NKS) & 1, drain);
            for (uint32_t f = vf > NVS ? vf - NVS : 0; f < vf; ++f) wait_bar(v_full(f % NVS), (f / NVS) & 1, drain);
        }
    } else if (warp == 9) {
        // ------------------------------------------------------------ MMA issuer
        // The whole warp runs the loop; the elected lane issues and commits.
        {
            const bool leader = elect_one_sync();
            const SDesc dQ_km = sdesc_make(sQ, 16, 1024), dO_km = sdesc_make(sdO, 16, 1024);
            const SDesc dK_km = sdesc_make(sK(0), 16, 1024), dV_km = sdesc_make(sV(0), 16, 1024);
            const SDesc dK_mn = sdesc_make(sK(0), 128 * 128, 1024);
            constexpr uint32_t kTile16 = C::kTileBytes >> 4;
            uint32_t kc = 0, vc = 0, sc = 0, dsc = 0, qc = 0, item_no = 0;  // K, V, S, dS, Q/dO consumed so far
            // S number g = Q K_j^T into buffer g & 1: M = 128 queries, N = 128 keys, K = D (both K-major)
            auto issue_s = [&](uint32_t kidx, uint32_t g) -> bool {
                const int ks = kidx % NKS;
                if (!wait_all(k_full(ks), (kidx / NKS) & 1, ctl)) return false;
                tc_fence_after();
#pragma unroll
                for (int s = 0; s < D / 16; ++s) {
                    const uint32_t off = ((s >> 2) * (128 * 128) + (s & 3) * 32) >> 4;
                    if (leader) mma_ss_d(tmem + C::kS(g & 1), dQ_km, off, dK_km, ks * kTile16 + off, C::kIdescS, s > 0);
                }
                if (leader) mma_commit(s_full(g & 1));
                return true;
            };
            // dP = dO V^T
            auto issue_dp = [&](uint32_t vidx) -> bool {
                const int vs = vidx % NVS;
                if (!wait_all(v_full(vs), (vidx / NVS) & 1, ctl)) return false;
                tc_fence_after();
#pragma unroll
                for (int s = 0; s < D / 16; ++s) {
                    const uint32_t off = ((s >> 2) * (128 * 128) + (s & 3) * 32) >> 4;
                    if (leader) mma_ss_d(tmem + C::kDP, dO_km, off, dV_km, vs * kTile16 + off, C::kIdescS, s > 0);
                }
                if (leader) {
                    mma_commit(dp_full);
                    mma_commit(v_empty(vs));
                }
                return true;
            };
            // Per item: S(0), dP(0), S(1); then per key tile j, in issue order:
            //   dP(j+1)                    the compute warps have read dP(j)
            //   dQ += dS(j) K_j            dS from TMEM (over S(j)), K MN-major
            //   S(j+2)                     into the buffer of S(j) (dQ(j) was its last reader)
            // The compute warps turn S(j+1) and dP(j+1) into dS(j+1) while these run.
            for (int k = 0;; ++k) {
                const int slot = k % kDqItemRing;
                if (!wait_all(item_full(slot), (k / kDqItemRing) & 1, ctl)) goto mma_teardown;
                const int w = item_ring[slot];
                __syncwarp();
                if (lane == 0) mbar_arrive(item_empty(slot));
                if (w >= p.n_items) break;
                int w_bh, w_qt;
                dq_item_at<CAUSAL>(w, p, w_bh, w_qt);
                const Item it = item(w_bh, w_qt);
                if (!wait_all(qdo_full, qc & 1, ctl)) goto mma_teardown;
                ++qc;
                tc_fence_after();
                if (!issue_s(kc, sc)) goto mma_teardown;
                if (!issue_dp(vc)) goto mma_teardown;
                if (it.n > 1 && !issue_s(kc + 1, sc + 1)) goto mma_teardown;
                for (int j = 0; j < it.n; ++j) {
                    if (!wait_all(ds_full, dsc & 1, ctl)) goto mma_teardown;
                    ++dsc;
                    tc_fence_after();
                    if (j + 1 < it.n && !issue_dp(vc + j + 1)) goto mma_teardown;
                    if (j == it.n - 1 && leader) mma_commit(qdo_empty);  // every S and dP of the item is issued
                    if (j == 0) {
                        // the previous item's dQ must have left TMEM
                        if (!wait_all(dq_empty, (item_no & 1) ^ 1, ctl)) goto mma_teardown;
                        tc_fence_after();
                    }
                    const int ks = (kc + j) % NKS, b = (sc + j) & 1;
#pragma unroll
                    for (int s = 0; s < kBN / 16; ++s)
                        if (leader) mma_ts_d(tmem + C::kDQ, tmem + C::kS(b) + C::kDSCol + s * 8, dK_mn,
                                 ks * kTile16 + s * (2048 >> 4), C::kIdescDQ, (j > 0 || s > 0) ? 1u : 0u);
                    if (leader) mma_commit(k_empty(ks));
                    if (j + 2 < it.n && !issue_s(kc + j + 2, sc + j + 2)) goto mma_teardown;
                }
                if (leader) mma_commit(dq_full);
                kc += it.n;
                vc += it.n;
                sc += it.n;
                ++item_no;
            }
        mma_teardown:
            if (leader) {
                mma_commit(mma_done);
                volatile int never = 0;
                Ctl drain{&never, 100000000ull};
                wait_bar(mma_done, 0, drain);
            }
            __syncwarp();
        }
    } else {
        // ------------------------------------------------------------ compute (warps 0-7) + dQ epilogue
        // thread = query row (TMEM lane); warpgroup h takes key columns 64h .. 64h+63
        const int h = warp >> 2, wq = warp & 3;
        const int r = 32 * wq + lane;
        const uint32_t lane_base = tmem + ((32u * wq) << 16);
        const float eff = p.sl2_eff, sl2 = p.sl2;
        const bool prescale = p.prescale != 0;
        const uint64_t eff2 = f2(eff, eff);
        uint32_t sc = 0, vc = 0, item_no = 0;  // S and dP numbers, items done: as in the MMA warp
        for (int k = 0;; ++k) {
            const int slot = k % kDqItemRing;
            if (!wait_all(item_full(slot), (k / kDqItemRing) & 1, ctl)) goto compute_done;
            const int w = item_ring[slot];
            __syncwarp();
            if (lane == 0) mbar_arrive(item_empty(slot));
            if (w >= p.n_items) break;
            int w_bh, w_qt;
            dq_item_at<CAUSAL>(w, p, w_bh, w_qt);
            const Item it = item(w_bh, w_qt);
            const int q = it.qt * 128 + r;
            if (!FA_CHECK(it.bh >= 0 && it.bh < p.BH && q < p.T_pad, &g_status_bwd, abort_flag)) goto compute_done;
            // -LSE2 and -D of this row (0 on padded rows q >= T, which the mask zeroes anyway)
            const float nlse = p.lse2[static_cast<size_t>(it.bh) * p.T_pad + q];
            const float nd = p.dvec[static_cast<size_t>(it.bh) * p.T_pad + q];
            const uint64_t nlse2 = f2(nlse, nlse), nd2 = f2(nd, nd);
            for (int j = 0; j < it.n; ++j) {
                const uint32_t g = sc + j, b = g & 1;
                const bool masked = bwd_tile_class(it.T, CAUSAL, 128, it.qt, j) == kMasked;
                if (!warp_wait<false>(s_full(b), (g >> 1) & 1, ctl)) goto compute_done;
                tc_fence_after();
                uint32_t sr[64];
                tmem_ld32(lane_base + C::kS(b) + 64 * h, sr);
                tmem_ld32(lane_base + C::kS(b) + 64 * h + 32, sr + 32);
                tmem_ld_wait();
                reg_fence32(sr);
                reg_fence32(sr + 32);
                float* pf = reinterpret_cast<float*>(sr);
                if (prescale) {
#pragma unroll
                    for (int e = 0; e < 64; ++e) pf[e] *= sl2;
                }
                // P = exp2(S c - LSE2)
#pragma unroll
                for (int e = 0; e < 64; e += 2) {
                    float x0, x1;
                    f2_split(fma2(f2(pf[e], pf[e + 1]), eff2, nlse2), x0, x1);
                    pf[e] = ex2_approx(x0);
                    pf[e + 1] = ex2_approx(x1);
                }
                if (masked) {
                    const int key0 = j * kBN + 64 * h;
#pragma unroll
                    for (int e = 0; e < 64; ++e)
                        if (!bwd_elem_visible(it.T, CAUSAL, q, key0 + e)) pf[e] = 0.f;
                }
                if (!warp_wait<false>(dp_full, (vc + j) & 1, ctl)) goto compute_done;
                tc_fence_after();
#pragma unroll
                for (int ch = 0; ch < 2; ++ch) {
                    uint32_t dr[32];
                    tmem_ld32(lane_base + C::kDP + 64 * h + 32 * ch, dr);
                    tmem_ld_wait();
                    reg_fence32(dr);
                    // dS = P o (dP - D), bf16 pairs over this warpgroup's S columns
                    uint32_t pk[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        const uint64_t t2 = add2(f2(__uint_as_float(dr[2 * e]), __uint_as_float(dr[2 * e + 1])), nd2);
                        float d0, d1;
                        f2_split(mul2(f2(pf[32 * ch + 2 * e], pf[32 * ch + 2 * e + 1]), t2), d0, d1);
                        pk[e] = pack_bf16x2(d0, d1);
                    }
                    tmem_st16(lane_base + C::kS(b) + C::kDSCol + 32 * h + 16 * ch, pk);
                }
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(ds_full);
            }
            sc += it.n;
            vc += it.n;
            // epilogue: dQ * scale -> bf16, stored row by row (d columns of this warpgroup);
            // TMEM is handed back as soon as the values are in registers
            {
                if (!warp_wait(dq_full, item_no & 1, ctl)) goto compute_done;
                ++item_no;
                tc_fence_after();
                constexpr int kCols = D / 2;  // d columns per warpgroup
                uint32_t v[kCols];
#pragma unroll
                for (int c = 0; c < kCols / 32; ++c) tmem_ld32(lane_base + C::kDQ + h * kCols + 32 * c, v + 32 * c);
                tmem_ld_wait();
#pragma unroll
                for (int c = 0; c < kCols / 32; ++c) reg_fence32(v + 32 * c);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(dq_empty);
                if (q < it.T) {
                    const size_t drow = VARLEN ? static_cast<size_t>(it.row0 + q) * p.Hq + it.head
                                               : static_cast<size_t>(it.bh) * T + q;
                    uint4* dst = reinterpret_cast<uint4*>(p.dq + drow * D + h * kCols);
#pragma unroll
                    for (int g = 0; g < kCols / 8; ++g) {
                        uint4 o;
                        o.x = pack_bf16x2(__uint_as_float(v[8 * g + 0]) * p.scale, __uint_as_float(v[8 * g + 1]) * p.scale);
                        o.y = pack_bf16x2(__uint_as_float(v[8 * g + 2]) * p.scale, __uint_as_float(v[8 * g + 3]) * p.scale);
                        o.z = pack_bf16x2(__uint_as_float(v[8 * g + 4]) * p.scale, __uint_as_float(v[8 * g + 5]) * p.scale);
                        o.w = pack_bf16x2(__uint_as_float(v[8 * g + 6]) * p.scale, __uint_as_float(v[8 * g + 7]) * p.scale);
                        dst[g] = o;
                    }
                }
            }
        }
    compute_done:;
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 9) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
    // This grid may have started while the dK/dV grid was still running (the
    // two read the same inputs and write disjoint outputs).  It ends only after
    // that grid has, so work after this launch sees dK and dV complete.
    griddep_wait();
}

template <typename K>
bool set_smem_once(K kern, int bytes, bool& done) {
    if (!done) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess)
            return false;
        done = true;
    }
    return true;
}

// The fused backward (D = 64): one dK/dV grid that also adds every query
// tile's dQ contribution into the fp32 accumulator (zeroed by the
// preprocess kernel), then the conversion of the accumulator to bf16 dQ.
template <bool CAUSAL>
int launch_fused_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& tdo,
                   const CUtensorMap& tdk, const CUtensorMap& tdv, const CUtensorMap& tacc, BwdParams p, int BHq,
                   int BHkv, const float* acc, cudaStream_t st, const DebugKnobs& dbg, int num_sms) {
    constexpr int D = 64;
    static bool attr = false;
    auto ka = fa_bwd_dkdv_kernel<D, CAUSAL, false, true>;
    if (!set_smem_once(ka, DkvCfg<D, true>::kSmemBytes, attr)) return -5;
    if (dbg.ev[2]) cudaEventRecord(dbg.ev[2], st);
    p.BH = BHkv;
    p.kt_major = (p.n_kt * BHkv < 8 * num_sms) ? 1 : 0;
    ka<<<p.n_kt * BHkv, kBwdThreads, DkvCfg<D, true>::kSmemBytes, st>>>(tq, tk, tv, tdo, tdk, tdv, tacc, p);
    if (cudaGetLastError() != cudaSuccess) return -5;
    if (dbg.ev[3]) cudaEventRecord(dbg.ev[3], st);
    const long long groups = static_cast<long long>(BHq) * p.T * (D / 8);
    const long long blocks = (groups + 255) / 256;
    const int grid = static_cast<int>(blocks < 8LL * num_sms ? blocks : 8LL * num_sms);
    fa_bwd_dq_convert_kernel<D><<<grid, 256, 0, st>>>(acc, p.dq, BHq, p.T, p.T_pad, p.scale);
    if (cudaGetLastError() != cudaSuccess) return -5;
    if (dbg.ev[4]) cudaEventRecord(dbg.ev[4], st);
    return 0;
}

template <int D, bool CAUSAL, bool VARLEN>
int launch_main_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& tdo,
                  const CUtensorMap& tdk, const CUtensorMap& tdv, BwdParams p, int BHq, int BHkv, cudaStream_t st,
                  const DebugKnobs& dbg, int num_sms) {
    static bool attr_a = false, attr_b = false;
    auto ka = fa_bwd_dkdv_kernel<D, CAUSAL, VARLEN>;
    auto kb = fa_bwd_dq_kernel<D, CAUSAL, VARLEN>;
    if (!set_smem_once(ka, DkvCfg<D>::kSmemBytes, attr_a) || !set_smem_once(kb, DqCfg<D>::kSmemBytes, attr_b))
        return -5;
    if (dbg.ev[2]) cudaEventRecord(dbg.ev[2], st);
    p.BH = BHkv;
    // key-tile-major order below 8 waves of CTAs (measured: GQA with 4 K/V heads
    // 0.86 -> 0.71 ms, D = 64 T = 2048 0.129 -> 0.114 ms); head major above
    // (T = 8192, 32 heads: 0.771 vs 0.792 ms key-tile major)
    p.kt_major = (p.n_kt * BHkv < 8 * num_sms) ? 1 : 0;
    ka<<<p.n_kt * BHkv, kBwdThreads, DkvCfg<D>::kSmemBytes, st>>>(tq, tk, tv, tdo, tdk, tdv, tq, p);
    if (cudaGetLastError() != cudaSuccess) return -5;
    if (dbg.ev[3]) cudaEventRecord(dbg.ev[3], st);
    p.BH = BHq;
    p.n_items = p.n_kt * BHq;
    const int grid_b = p.n_items < num_sms ? p.n_items : num_sms;  // persistent: one CTA per SM
    {
        // programmatic dependent launch: the dQ grid may start during the dK/dV
        // grid's tail (it waits for that grid only before it exits)
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(grid_b);
        cfg.blockDim = dim3(kBwdThreads);
        cfg.dynamicSmemBytes = DqCfg<D>::kSmemBytes;
        cfg.stream = st;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if (cudaLaunchKernelEx(&cfg, kb, tq, tk, tv, tdo, p) != cudaSuccess) return -5;
    }
    if (cudaGetLastError() != cudaSuccess) return -5;
    if (dbg.ev[4]) cudaEventRecord(dbg.ev[4], st);
    return 0;
}

// Preprocess + both main kernels, with the workspace (two vectors of
// B*Hq*T_pad floats at ws, each 256-byte aligned, then the dQ kernel's item
// counter) already in place.
int run_bwd(const void* q, const void* k, const void* v, const void* o, const void* dO, const float* lse, void* dq,
            void* dk, void* dv, int B, int Hq, int Hkv, int T, int D, float scale, bool causal, void* ws,
            bool fuse, cudaStream_t stream, const DebugKnobs& dbg, int num_sms) {
    const int BH = B * Hq, BHkv = B * Hkv;
    const int T_pad = cdiv(T, 128) * 128;
    const size_t bytes_vec = (static_cast<size_t>(BH) * T_pad * 4 + 255) / 256 * 256;
    float* dvec = static_cast<float*>(ws);
    float* lse2 = reinterpret_cast<float*>(static_cast<char*>(ws) + bytes_vec);
    int* dq_next = reinterpret_cast<int*>(static_cast<char*>(ws) + 2 * bytes_vec);
    // fused backward: the fp32 dQ accumulator follows the item counter (256-byte aligned)
    float* dqacc = fuse ? reinterpret_cast<float*>(static_cast<char*>(ws) + 2 * bytes_vec + 256) : nullptr;
    CUtensorMap tq, tk, tv, tdo, tdk, tdv, tacc;
    if (!make_tmap_bhtd(&tq, q, BH, T, D, 128) || !make_tmap_bhtd(&tk, k, BHkv, T, D, 128) ||
        !make_tmap_bhtd(&tv, v, BHkv, T, D, 128) || !make_tmap_bhtd(&tdo, dO, BH, T, D, 128) ||
        !make_tmap_bhtd(&tdk, dk, BHkv, T, D, 128) || !make_tmap_bhtd(&tdv, dv, BHkv, T, D, 128))
        return -5;
    if (fuse && (D != 64 || !make_tmap_f32_acc(&tacc, dqacc, BH, T_pad, D, 32))) return -5;
    const long long rows = static_cast<long long>(BH) * T_pad;
    const long long blocks = (rows * (D / 8) + 255) / 256;
    const int pre_grid = static_cast<int>(blocks < 8LL * num_sms ? blocks : 8LL * num_sms);
    if (D == 64)
        fa_bwd_pre_kernel<64, false><<<pre_grid, 256, 0, stream>>>(
            static_cast<const __nv_bfloat16*>(o), static_cast<const __nv_bfloat16*>(dO), lse, dvec, lse2, BH, T, T_pad,
            dq_next, nullptr, 1, Hq, 0, dqacc);
    else
        fa_bwd_pre_kernel<128, false><<<pre_grid, 256, 0, stream>>>(
            static_cast<const __nv_bfloat16*>(o), static_cast<const __nv_bfloat16*>(dO), lse, dvec, lse2, BH, T, T_pad,
            dq_next, nullptr, 1, Hq, 0, nullptr);
    if (cudaGetLastError() != cudaSuccess) return -5;
    BwdParams p;
    p.lse2 = lse2;
    p.dvec = dvec;
    p.dq_next = dq_next;
    p.dq = static_cast<__nv_bfloat16*>(dq);
    p.n_items = 0;
    p.dk = static_cast<__nv_bfloat16*>(dk);
    p.dv = static_cast<__nv_bfloat16*>(dv);
    p.T = T;
    p.T_pad = T_pad;
    p.n_kt = cdiv(T, kBN);
    p.kt_major = 0;
    p.BH = BHkv;
    p.Hq = Hq;
    p.Hkv = Hkv;
    p.group = Hq / Hkv;
    p.scale = scale;
    p.sl2 = scale * kLog2e;
    p.prescale = p.sl2 > 0.f ? 0 : 1;
    p.sl2_eff = p.prescale ? 1.f : p.sl2;
    p.timeout_ns = dbg.timeout_ns;
    p.inject = dbg.inject;
    p.cu_seqlens = nullptr;
    p.n_seq = 1;
    p.total = 0;
    if (fuse)
        return causal ? launch_fused_t<true>(tq, tk, tv, tdo, tdk, tdv, tacc, p, BH, BHkv, dqacc, stream, dbg, num_sms)
                      : launch_fused_t<false>(tq, tk, tv, tdo, tdk, tdv, tacc, p, BH, BHkv, dqacc, stream, dbg,
                                              num_sms);
    if (D == 64)
        return causal ? launch_main_t<64, true, false>(tq, tk, tv, tdo, tdk, tdv, p, BH, BHkv, stream, dbg, num_sms)
                      : launch_main_t<64, false, false>(tq, tk, tv, tdo, tdk, tdv, p, BH, BHkv, stream, dbg, num_sms);
    return causal ? launch_main_t<128, true, false>(tq, tk, tv, tdo, tdk, tdv, p, BH, BHkv, stream, dbg, num_sms)
                  : launch_main_t<128, false, false>(tq, tk, tv, tdo, tdk, tdv, p, BH, BHkv, stream, dbg, num_sms);
}

// Packed variable-length backward: (total, H, D) tensors, sequences given by
// cu_seqlens; the per-row vectors are laid out per (head, sequence) with
// max_seqlen rounded up to 128 rows each.  ws as for run_bwd, sized by
// bwd_varlen_scratch_bytes.
int run_bwd_varlen(const void* q, const void* k, const void* v, const void* o, const void* dO, const float* lse,
                   void* dq, void* dk, void* dv, const int* cu_seqlens, int n_seq, int max_seqlen, int total, int H,
                   int D, float scale, bool causal, void* ws, cudaStream_t stream, const DebugKnobs& dbg,
                   int num_sms) {
    const int BH = H * n_seq;
    const int T_pad = cdiv(max_seqlen, 128) * 128;
    const size_t bytes_vec = (static_cast<size_t>(BH) * T_pad * 4 + 255) / 256 * 256;
    float* dvec = static_cast<float*>(ws);
    float* lse2 = reinterpret_cast<float*>(static_cast<char*>(ws) + bytes_vec);
    int* dq_next = reinterpret_cast<int*>(static_cast<char*>(ws) + 2 * bytes_vec);
    CUtensorMap tq, tk, tv, tdo;
    if (!make_tmap_packed(&tq, q, total, H, D, 128) || !make_tmap_packed(&tk, k, total, H, D, 128) ||
        !make_tmap_packed(&tv, v, total, H, D, 128) || !make_tmap_packed(&tdo, dO, total, H, D, 128))
        return -5;
    const long long rows = static_cast<long long>(BH) * T_pad;
    const long long blocks = (rows * (D / 8) + 255) / 256;
    const int pre_grid = static_cast<int>(blocks < 8LL * num_sms ? blocks : 8LL * num_sms);
    if (D == 64)
        fa_bwd_pre_kernel<64, true><<<pre_grid, 256, 0, stream>>>(
            static_cast<const __nv_bfloat16*>(o), static_cast<const __nv_bfloat16*>(dO), lse, dvec, lse2, BH,
            max_seqlen, T_pad, dq_next, cu_seqlens, n_seq, H, total, nullptr);
    else
        fa_bwd_pre_kernel<128, true><<<pre_grid, 256, 0, stream>>>(
            static_cast<const __nv_bfloat16*>(o), static_cast<const __nv_bfloat16*>(dO), lse, dvec, lse2, BH,
            max_seqlen, T_pad, dq_next, cu_seqlens, n_seq, H, total, nullptr);
    if (cudaGetLastError() != cudaSuccess) return -5;
    BwdParams p;
    p.lse2 = lse2;
    p.dvec = dvec;
    p.dq_next = dq_next;
    p.dq = static_cast<__nv_bfloat16*>(dq);
    p.n_items = 0;
    p.dk = static_cast<__nv_bfloat16*>(dk);
    p.dv = static_cast<__nv_bfloat16*>(dv);
    p.T = max_seqlen;
    p.T_pad = T_pad;
    p.n_kt = cdiv(max_seqlen, kBN);
    p.kt_major = 0;
    p.BH = BH;
    p.Hq = H;
    p.Hkv = H;
    p.group = 1;
    p.scale = scale;
    p.sl2 = scale * kLog2e;
    p.prescale = p.sl2 > 0.f ? 0 : 1;
    p.sl2_eff = p.prescale ? 1.f : p.sl2;
    p.timeout_ns = dbg.timeout_ns;
    p.inject = dbg.inject;
    p.cu_seqlens = cu_seqlens;
    p.n_seq = n_seq;
    p.total = total;
    // dK and dV leave row by row (no TMA store), so their map arguments are placeholders
    if (D == 64)
        return causal ? launch_main_t<64, true, true>(tq, tk, tv, tdo, tq, tq, p, BH, BH, stream, dbg, num_sms)
                      : launch_main_t<64, false, true>(tq, tk, tv, tdo, tq, tq, p, BH, BH, stream, dbg, num_sms);
    return causal ? launch_main_t<128, true, true>(tq, tk, tv, tdo, tq, tq, p, BH, BH, stream, dbg, num_sms)
                  : launch_main_t<128, false, true>(tq, tk, tv, tdo, tq, tq, p, BH, BH, stream, dbg, num_sms);
}

}  // namespace

size_t bwd_scratch_bytes(int B, int H, int T, int D) {
    (void)D;
    const size_t BH = static_cast<size_t>(B) * H;
    const size_t T_pad = static_cast<size_t>(cdiv(T, 128)) * 128;
    const size_t bytes_vec = (BH * T_pad * 4 + 255) / 256 * 256;
    return 2 * bytes_vec + 256;  // + the dQ kernel's item counter
}
// The fused backward (D = 64) when it fills the GPU: with fewer dK/dV CTAs
// than SMs the two-kernel form is faster, its dQ grid running on the SMs the
// dK/dV grid leaves idle (B=1 H=8 T=1024: 24 us two-kernel, 32 us fused).
bool bwd_fuses(int D, int n_kt, int BHkv, int num_sms, const DebugKnobs& dbg) {
    return D == 64 && !dbg.deterministic && static_cast<long long>(n_kt) * BHkv >= num_sms;
}
bool bwd_fuses_host(int B, int Hkv, int T, int D, int num_sms, bool deterministic) {
    DebugKnobs k{};
    k.deterministic = deterministic ? 1 : 0;
    return bwd_fuses(D, cdiv(T, kBN), B * Hkv, num_sms, k);
}
size_t bwd_workspace_bytes(int B, int H, int T, int D, bool fuse) {
    const size_t T_pad = static_cast<size_t>(cdiv(T, 128)) * 128;
    // fused: + the fp32 dQ accumulator (B*H, T_pad, D)
    return bwd_scratch_bytes(B, H, T, D) + (fuse ? static_cast<size_t>(B) * H * T_pad * D * 4 : 0);
}

size_t bwd_varlen_scratch_bytes(int n_seq, int H, int max_seqlen) {
    const size_t BH = static_cast<size_t>(n_seq) * H;
    const size_t T_pad = static_cast<size_t>(cdiv(max_seqlen, 128)) * 128;
    const size_t bytes_vec = (BH * T_pad * 4 + 255) / 256 * 256;
    return 2 * bytes_vec + 256;
}

int launch_bwd_varlen(const void* q, const void* k, const void* v, const void* o, const void* dO, const float* lse,
                      void* dq, void* dk, void* dv, const int* cu_seqlens, int n_seq, int max_seqlen, int total,
                      int H, int D, float scale, bool causal, cudaStream_t stream, const DebugKnobs& dbg,
                      int num_sms) {
    void* ws = nullptr;
    if (cudaMallocAsync(&ws, bwd_varlen_scratch_bytes(n_seq, H, max_seqlen), stream) != cudaSuccess) {
        cudaGetLastError();
        return -6;
    }
    int rc = run_bwd_varlen(q, k, v, o, dO, lse, dq, dk, dv, cu_seqlens, n_seq, max_seqlen, total, H, D, scale,
                            causal, ws, stream, dbg, num_sms);
    if (cudaFreeAsync(ws, stream) != cudaSuccess && rc == 0) rc = -5;
    return rc;
}

int launch_bwd(const void* q, const void* k, const void* v, const void* o, const void* dO, const float* lse,
               void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int T, int D, float scale, bool causal,
               cudaStream_t stream, const DebugKnobs& dbg, int num_sms) {
    const bool fuse = bwd_fuses(D, cdiv(T, kBN), B * Hkv, num_sms, dbg);
    void* ws = nullptr;
    if (cudaMallocAsync(&ws, bwd_workspace_bytes(B, Hq, T, D, fuse), stream) != cudaSuccess) {
        cudaGetLastError();
        return -6;
    }
    int rc = run_bwd(q, k, v, o, dO, lse, dq, dk, dv, B, Hq, Hkv, T, D, scale, causal, ws, fuse, stream, dbg,
                     num_sms);
    if (cudaFreeAsync(ws, stream) != cudaSuccess && rc == 0) rc = -5;
    return rc;
}

// ---------------------------------------------------------------- fixed scratch
// Workspace for fa_bwd_noalloc, for callers that cannot allocate device
// memory at call time.  It lives in the module's global memory, so every GPU
// that loads this module holds it until the process exits.  Kernels receive
// its device address from the host; the host-side symbol itself is only a
// stand-in and must never be passed to a kernel.
static __device__ __align__(256) unsigned char g_bwd_scratch[FA_BWD_NOALLOC_SCRATCH_BYTES];

namespace {
constexpr int kScratchMaxDevices = 64;
std::once_flag g_scratch_once[kScratchMaxDevices];
void* g_scratch_ptr[kScratchMaxDevices];
cudaError_t g_scratch_err[kScratchMaxDevices];

// Device address of g_bwd_scratch on the current device, looked up once per
// device (the first fa_bwd_noalloc call on that device does it) and kept for
// the process lifetime: it belongs to the context current at that first
// call, and is stale after cudaDeviceReset or in another context.
void* scratch_address(int dev) {
    std::call_once(g_scratch_once[dev], [dev] {
        void* p = nullptr;
        g_scratch_err[dev] = cudaGetSymbolAddress(&p, g_bwd_scratch);
        g_scratch_ptr[dev] = p;
    });
    return g_scratch_err[dev] == cudaSuccess ? g_scratch_ptr[dev] : nullptr;
}
}  // namespace

int launch_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const void* dO, const float* lse,
                       void* dq, void* dk, void* dv, int B, int H, int T, int D, float scale, bool causal,
                       cudaStream_t stream, const DebugKnobs& dbg, int num_sms) {
    if (bwd_scratch_bytes(B, H, T, D) > FA_BWD_NOALLOC_SCRATCH_BYTES) return -10;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kScratchMaxDevices) return -5;
    void* ws = scratch_address(dev);
    if (!ws) return -5;
    // the preprocess kernel rewrites both vectors, so the previous call's contents do not matter
    return run_bwd(q, k, v, o, dO, lse, dq, dk, dv, B, H, H, T, D, scale, causal, ws, false, stream, dbg, num_sms);
}

int bwd_take_status() {
    int h = 0, z = 0;
    if (cudaMemcpyFromSymbol(&h, g_status_bwd, sizeof(int)) != cudaSuccess) return -5;
    if (cudaMemcpyToSymbol(g_status_bwd, &z, sizeof(int)) != cudaSuccess) return -5;
    return h;
}

}  // namespace fa
