// fa_bwd.cu -- exact attention backward on sm_103a ("Lab 06 - Attention
// kernels", section 4: D = rowsum(dO o O); P = exp(S - LSE) recomputed per
// tile; dV = P^T dO; dP = dO V^T; dS = P o (dP - D); dQ = dS K scale;
// dK = dS^T Q scale; key tiles outer, query tiles inner, so dK and dV
// accumulate in one place while dQ receives a contribution from every key
// tile).
//
// Three kernels on the caller's stream:
//   fa_bwd_pre   D_i = sum_d dO_id O_id (fp32), LSE in log2 units, both
//                padded to a multiple of 128 rows; zero the fp32 dQ
//                accumulator.
//   fa_bwd_main  one CTA per (key tile of 128, batch*head).  Warp roles:
//                  warps 0-7   compute: P^T = exp2(S^T c - LSE2) and
//                              dS^T = P^T o (dP^T - D) for half of the query
//                              columns each (TMEM lane = key row)
//                  warps 8-11  dQ drain (fp32 reductions into the
//                              accumulator) and the dK/dV epilogue
//                  warp 12     TMA producer (K, V once; per query tile Q with
//                              -LSE2, -D into a 4-stage ring, dO into a 3-stage ring)
//                  warp 13     tcgen05 issuer
//                Per query tile: S^T = K Q^T and dP^T = V dO^T into TMEM;
//                dV += P^T dO with P^T read from TMEM; dK += dS^T Q and the
//                dQ tile (dS K, or its transpose at D = 128) from dS^T in
//                shared memory.
//   fa_bwd_dq    dQ = bf16(dQacc * scale).
#include <cuda_runtime.h>

#include <mutex>

#include "fa.h"
#include "fa_internal.h"
#include "fa_ptx.cuh"
#include "fa_sched.h"
#include "fa_tmap.h"

namespace fa {

static __device__ int g_status_bwd;

// Optional cycle tracing of one CTA's pipeline (build with -DFA_TRACE; off in
// the library): slot = event kind, index = query-tile iteration.
#ifdef FA_TRACE
constexpr int kTraceSlots = 28, kTraceLen = 512;
static __device__ unsigned long long g_trace[kTraceSlots][kTraceLen];
#define FA_TRACE_EVENT(slot, idx)                                                  \
    do {                                                                           \
        if (blockIdx.x == 0 && (idx) < kTraceLen) g_trace[slot][idx] = clock64(); \
    } while (0)
#else
#define FA_TRACE_EVENT(slot, idx) \
    do {                          \
    } while (0)
#endif

namespace {

#ifndef FA_CRIT_SLEEP
#define FA_CRIT_SLEEP 0
#endif
// Waits on the MMA <-> compute critical path poll back to back unless built
// with FA_CRIT_SLEEP=1; every other wait lets the hardware park the thread.
constexpr bool kCritSleep = FA_CRIT_SLEEP != 0;

constexpr int kBwdThreads = 448;
constexpr float kLog2e = 1.44269504088896340736f;

template <int D>
struct BwdCfg {
    static constexpr int BM = bwd_bm(D);             // query rows per inner iteration
    static constexpr int kHalf = BM / 2;             // query columns per compute warpgroup
    static constexpr int kAtomsD = D / 64;
    static constexpr bool kDqT = (D == 128);         // dQ^T = K^T dS^T (M = D) instead of dQ = dS K (M = BM)
    // D = 128: two S^T buffers, P^T aliased into the S buffer it came from at
    // column offset BM/4 (each compute warpgroup then overwrites only columns
    // it has itself already read).  D = 64: one S^T buffer, P^T in its own region.
    static constexpr bool kSDouble = (D == 128);
    static constexpr int kKVBytes = 128 * D * 2;     // one K or V tile
    static constexpr int kQBytes = BM * D * 2;       // one Q or dO tile
    // Q (with its -LSE2 and -D vectors) and dO travel in separate rings: S(i+2)
    // needs Q two tiles ahead while dO is needed one tile ahead.
    static constexpr int kQStages = 4, kDOStages = 3;
    static constexpr int kQStageBytes = kQBytes + 1024;  // + -LSE2[BM], -D[BM] (<= 1 KB)
    static constexpr int kDSBytes = 128 * BM * 2;    // dS^T tile [128 keys][BM queries] bf16
    static constexpr int kKOff = 0;
    static constexpr int kVOff = kKVBytes;
    static constexpr int kQRingOff = 2 * kKVBytes;
    static constexpr int kDORingOff = kQRingOff + kQStages * kQStageBytes;
    static constexpr int kDSOff = kDORingOff + kDOStages * kQBytes;
    static constexpr int kBarOff = kDSOff + 2 * kDSBytes;
    // kv_full, q_full[4], q_empty[4], do_full[3], do_empty[3], s_full[2], dp_full, p_full,
    // ds_empty[2], dq_full, dq_empty, dkv_full, mma_done, p_free
    static constexpr int kNumBars = 1 + 2 * kQStages + 2 * kDOStages + 2 + 2 + 2 + 5;
    static constexpr int kMiscOff = kBarOff + kNumBars * 8;
    static constexpr int kSmemBytes = kMiscOff + 16 + 1024;
    static_assert(kSmemBytes <= 232448, "shared memory budget");
    // TMEM columns
    static constexpr uint32_t kS = 0;                                  // S^T [128 keys][BM] fp32 (x2 at D = 128)
    static constexpr uint32_t kDP = kSDouble ? 2 * BM : BM;            // dP^T [128 keys][BM] fp32
    static constexpr uint32_t kP = kDP + BM;                           // P^T bf16 pairs (single-S layout only)
    static constexpr uint32_t kDQ = kSDouble ? kDP + BM : kP + BM / 2; // dQ^T [D][BM] or dQ [BM][D]: 64 columns
    static constexpr uint32_t kDV = kDQ + 64;                          // dV [128 keys][D] fp32
    static constexpr uint32_t kDK = kDV + D;                           // dK [128 keys][D] fp32
    static_assert(kDK + D <= 512, "TMEM budget");
    static constexpr uint32_t kIdescS = idesc_bf16_f32(128, BM, false, false);
    static constexpr uint32_t kIdescDKV = idesc_bf16_f32(128, D, false, true);
    static constexpr uint32_t kIdescDQ = idesc_bf16_f32(128, 64, true, true);
};

struct BwdParams {
    const float* lse2;   // [BH][T_pad] -LSE * log2(e)
    const float* dvec;   // [BH][T_pad] -D
    float* dqacc;        // [BH][T][D]
    __nv_bfloat16* dk;
    __nv_bfloat16* dv;
    int T, T_pad, BH, n_kt;  // BH = batch * key/value heads (one CTA row per K/V head)
    int Hq, Hkv, group;       // query heads, key/value heads, Hq / Hkv
    float scale;
    float sl2, sl2_eff;
    int prescale;
    unsigned long long timeout_ns;
};

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

// ---------------------------------------------------------------- preprocess
// D_i = rowsum(dO o O) ("Lab 06", section 4) and LSE2 = LSE * log2(e), both
// stored NEGATED (the main kernel adds them with packed FMAs); rows t >= T
// of the padded vectors are 0; dQacc = 0.  8 elements per thread.
template <int D>
__global__ void __launch_bounds__(256) fa_bwd_pre_kernel(const __nv_bfloat16* __restrict__ o,
                                                         const __nv_bfloat16* __restrict__ dO,
                                                         const float* __restrict__ lse, float* __restrict__ dvec,
                                                         float* __restrict__ lse2, float* __restrict__ dqacc, int BH,
                                                         int T, int T_pad) {
    constexpr int TPR = D / 8;            // threads per row
    constexpr int RPW = 32 / TPR;         // rows per warp
    const long long total = static_cast<long long>(BH) * T_pad;
    const int lane = threadIdx.x & 31, sub = lane % TPR;
    const long long n_warps = static_cast<long long>(gridDim.x) * (blockDim.x / 32);
    // warp-uniform loop: every lane reaches the shuffles below
    for (long long wr = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) / 32; wr * RPW < total;
         wr += n_warps) {
        const long long r = wr * RPW + lane / TPR;
        const bool in = r < total;
        const int bh = in ? static_cast<int>(r / T_pad) : 0, t = in ? static_cast<int>(r % T_pad) : T_pad;
        float acc = 0.f;
        if (in && t < T) {
            const size_t off = (static_cast<size_t>(bh) * T + t) * D + sub * 8;
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
            float4* z = reinterpret_cast<float4*>(dqacc + off);
            z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
            z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int m = TPR / 2; m > 0; m >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, m, TPR);
        if (in && sub == 0) {
            dvec[r] = -acc;
            lse2[r] = (t < T) ? -lse[static_cast<size_t>(bh) * T + t] * kLog2e : 0.f;
        }
    }
}

// ---------------------------------------------------------------- dQ convert
__global__ void __launch_bounds__(256) fa_bwd_dq_kernel(const float* __restrict__ dqacc,
                                                        __nv_bfloat16* __restrict__ dq, long long n8, float scale) {
    for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n8;
         i += static_cast<long long>(gridDim.x) * blockDim.x) {
        const float4 a = reinterpret_cast<const float4*>(dqacc)[2 * i];
        const float4 b = reinterpret_cast<const float4*>(dqacc)[2 * i + 1];
        uint4 w;
        w.x = pack_bf16x2(a.x * scale, a.y * scale);
        w.y = pack_bf16x2(a.z * scale, a.w * scale);
        w.z = pack_bf16x2(b.x * scale, b.y * scale);
        w.w = pack_bf16x2(b.z * scale, b.w * scale);
        reinterpret_cast<uint4*>(dq)[i] = w;
    }
}

// ---------------------------------------------------------------- main kernel
template <int D, bool CAUSAL>
__global__ void __launch_bounds__(kBwdThreads, 1)
    fa_bwd_main_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                       BwdParams p) {
    using C = BwdCfg<D>;
    constexpr int BM = C::BM;
    constexpr int NQS = C::kQStages, NDS = C::kDOStages;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const uint32_t sK = sbase + C::kKOff, sV = sbase + C::kVOff;
    auto sQ = [&](int st) { return sbase + C::kQRingOff + st * C::kQStageBytes; };
    auto sLse = [&](int st) { return sQ(st) + C::kQBytes; };
    auto sDv = [&](int st) { return sLse(st) + BM * 4; };
    auto sdO = [&](int st) { return sbase + C::kDORingOff + st * C::kQBytes; };
    auto sDS = [&](int b) { return sbase + C::kDSOff + b * C::kDSBytes; };
    const uint32_t bars = sbase + C::kBarOff;
    const uint32_t kv_full = bars;
    auto q_full = [&](int st) { return bars + 8u * (1 + st); };
    auto q_empty = [&](int st) { return bars + 8u * (1 + NQS + st); };
    auto do_full = [&](int st) { return bars + 8u * (1 + 2 * NQS + st); };
    auto do_empty = [&](int st) { return bars + 8u * (1 + 2 * NQS + NDS + st); };
    const uint32_t b0 = bars + 8u * (1 + 2 * NQS + 2 * NDS);
    auto s_full = [&](int b) { return b0 + 8u * b; };  // one per S buffer
    const uint32_t dp_full = b0 + 16;
    const uint32_t p_full = b0 + 24;
    auto ds_empty = [&](int b) { return b0 + 32 + 8u * b; };
    const uint32_t dq_full = b0 + 48;
    const uint32_t dq_empty = b0 + 56;
    const uint32_t dkv_full = b0 + 64;
    const uint32_t mma_done = b0 + 72;
    const uint32_t p_free = b0 + 80;  // single-S layout: P region free again (dV done)
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kMiscOff);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kMiscOff + 4);
    const Ctl ctl{abort_flag, p.timeout_ns};

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int T = p.T;
    // head-major order: the key tiles of one head run together (their Q, dO
    // and dQ accumulator stay in L2); within a head, heavy key tiles first.
    // With grouped heads the CTA walks the query tiles of every query head that
    // shares this K/V head, so dK and dV sum over the group in TMEM.
    const int bh = blockIdx.x / p.n_kt, kt = blockIdx.x % p.n_kt;  // bh: batch * Hkv + K/V head
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
        mbar_init(s_full(0), 1);
        mbar_init(s_full(1), 1);
        mbar_init(dp_full, 1);
        mbar_init(p_full, 8);
        mbar_init(ds_empty(0), 1);
        mbar_init(ds_empty(1), 1);
        mbar_init(dq_full, 1);
        mbar_init(dq_empty, 4);
        mbar_init(dkv_full, 1);
        mbar_init(mma_done, 1);
        mbar_init(p_free, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 13) {
        tmem_alloc(smem_u32(tmem_slot), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(tmem_slot);

    if (warp == 12) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            uint32_t q_armed = 0, do_armed = 0;  // fills issued per ring
            const uint64_t pol_kv = l2_policy_evict_first();
            const uint64_t pol_q = l2_policy_evict_last();
            mbar_arrive_expect_tx(kv_full, 2 * C::kKVBytes);
            for (int a = 0; a < C::kAtomsD; ++a) {
                tma_load_3d_hint(sK + a * 128 * 128, &tm_k, kv_full, 64 * a, kt * kBN, bh, pol_kv);
                tma_load_3d_hint(sV + a * 128 * 128, &tm_v, kv_full, 64 * a, kt * kBN, bh, pol_kv);
            }
            for (int it = 0; it < n_it; ++it) {
                const int qt = q_tile_of(it), bhq = q_head_of(it);
                {   // Q tile with its -LSE2 and -D vectors
                    const int st = it % NQS;
                    if (!wait_bar(q_empty(st), ((it / NQS) & 1) ^ 1, ctl)) break;
                    const uint32_t fb = q_full(st);
                    mbar_arrive_expect_tx(fb, C::kQBytes + 2 * BM * 4);
                    ++q_armed;
                    for (int a = 0; a < C::kAtomsD; ++a)
                        tma_load_3d_hint(sQ(st) + a * BM * 128, &tm_q, fb, 64 * a, qt * BM, bhq, pol_q);
                    const size_t voff = static_cast<size_t>(bhq) * p.T_pad + static_cast<size_t>(qt) * BM;
                    bulk_load_1d(sLse(st), p.lse2 + voff, BM * 4, fb);
                    bulk_load_1d(sDv(st), p.dvec + voff, BM * 4, fb);
                }
                {   // dO tile
                    const int st = it % NDS;
                    if (!wait_bar(do_empty(st), ((it / NDS) & 1) ^ 1, ctl)) break;
                    const uint32_t fb = do_full(st);
                    mbar_arrive_expect_tx(fb, C::kQBytes);
                    ++do_armed;
                    for (int a = 0; a < C::kAtomsD; ++a)
                        tma_load_3d_hint(sdO(st) + a * BM * 128, &tm_do, fb, 64 * a, qt * BM, bhq, pol_q);
                }
            }
            // drain: copies still in flight must land before the CTA exits
            volatile int never = 0;
            Ctl drain{&never, 100000000ull};
            wait_bar(kv_full, 0, drain);
            for (uint32_t f = q_armed > NQS ? q_armed - NQS : 0; f < q_armed; ++f)
                wait_bar(q_full(f % NQS), (f / NQS) & 1, drain);
            for (uint32_t f = do_armed > NDS ? do_armed - NDS : 0; f < do_armed; ++f)
                wait_bar(do_full(f % NDS), (f / NDS) & 1, drain);
        }
    } else if (warp == 13) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            // Descriptors are built once; a stage / buffer / k-step is an offset in 16-byte units.
            const SDesc dK_km = sdesc_make(sK, 16, 1024), dV_km = sdesc_make(sV, 16, 1024);
            const SDesc dK_mn = sdesc_make(sK, 128 * 128, 1024);
            const SDesc dQ_km = sdesc_make(sQ(0), 16, 1024), dO_km = sdesc_make(sdO(0), 16, 1024);
            const SDesc dQ_mn = sdesc_make(sQ(0), BM * 128, 1024), dO_mn = sdesc_make(sdO(0), BM * 128, 1024);
            const SDesc dS_km = sdesc_make(sDS(0), 16, 1024), dS_mn = sdesc_make(sDS(0), 128 * 128, 1024);
            constexpr uint32_t kQStage16 = C::kQStageBytes >> 4, kDOStage16 = C::kQBytes >> 4;
            constexpr uint32_t kDS16 = C::kDSBytes >> 4;
            // S^T = K Q^T into S buffer b: M = 128 keys, N = BM, K = D (both K-major)
            auto issue_s = [&](int st, int b) {
                const uint32_t so = st * kQStage16;
#pragma unroll
                for (int s = 0; s < D / 16; ++s)
                    mma_ss_d(tmem + C::kS + b * BM, dK_km, ((s >> 2) * (128 * 128) + (s & 3) * 32) >> 4, dQ_km,
                             so + (((s >> 2) * (BM * 128) + (s & 3) * 32) >> 4), C::kIdescS, s > 0);
                mma_commit(s_full(b));
            };
            // dP^T = V dO^T
            auto issue_dp = [&](int st) {
                const uint32_t so = st * kDOStage16;
#pragma unroll
                for (int s = 0; s < D / 16; ++s)
                    mma_ss_d(tmem + C::kDP, dV_km, ((s >> 2) * (128 * 128) + (s & 3) * 32) >> 4, dO_km,
                             so + (((s >> 2) * (BM * 128) + (s & 3) * 32) >> 4), C::kIdescS, s > 0);
                mma_commit(dp_full);
            };
            // One k-step of dV, dK or the dQ tile.  These are transposed-operand (or
            // TMEM-operand) MMAs: back to back on one accumulator they run slower than
            // when consecutive instructions alternate between independent accumulators,
            // so the issue order below interleaves their k-steps.
            auto step_dv = [&](int st, int b, int it, int s) {
                const uint32_t pcol = C::kSDouble ? (C::kS + b * BM + BM / 4) : C::kP;
                mma_ts_d(tmem + C::kDV, tmem + pcol + s * 8, dO_mn, st * kDOStage16 + s * (2048 >> 4), C::kIdescDKV,
                         (it > 0 || s > 0) ? 1u : 0u);
            };
            auto step_dk = [&](int st, int b, int it, int s) {
                mma_ss_d(tmem + C::kDK, dS_km, b * kDS16 + (((s >> 2) * (128 * 128) + (s & 3) * 32) >> 4), dQ_mn,
                         st * kQStage16 + s * (2048 >> 4), C::kIdescDKV, (it > 0 || s > 0) ? 1u : 0u);
            };
            auto step_dq = [&](int b, int s) {
                if constexpr (C::kDqT)  // dQ^T [D][BM] = K^T dS^T
                    mma_ss_d(tmem + C::kDQ, dK_mn, s * (2048 >> 4), dS_mn, b * kDS16 + s * (2048 >> 4), C::kIdescDQ,
                             s > 0);
                else  // dQ [BM][D] = dS K
                    mma_ss_d(tmem + C::kDQ, dS_mn, b * kDS16 + s * (2048 >> 4), dK_mn, s * (2048 >> 4), C::kIdescDQ,
                             s > 0);
            };
            constexpr int NKV = BM / 16, NQ = 128 / 16;  // k-steps of dV / dK and of the dQ tile
            if (!wait_bar(kv_full, 0, ctl)) goto mma_teardown;
            if (!wait_bar(q_full(0), 0, ctl)) goto mma_teardown;
            tc_fence_after();
            issue_s(0, 0);
            if (!wait_bar(do_full(0), 0, ctl)) goto mma_teardown;
            tc_fence_after();
            issue_dp(0);
            if constexpr (C::kSDouble) {
                if (n_it > 1) {
                    if (!wait_bar(q_full(1), 0, ctl)) goto mma_teardown;
                    tc_fence_after();
                    issue_s(1, 1);
                }
            }
            for (int it = 0; it < n_it; ++it) {
                const int qs = it % NQS, ds = it % NDS, b = it & 1;
                if (!wait_bar<kCritSleep>(p_full, it & 1, ctl)) goto mma_teardown;
                FA_TRACE_EVENT(0, it);
                tc_fence_after();
                if constexpr (C::kSDouble) {
                    // S(it+1) already sits in the other buffer.  dP(it+1) first (the compute
                    // warps need it soonest), then dV(it) -- the only reader of P(it), aliased
                    // in buffer b -- so that S(it+2) can refill buffer b right away.
                    if (it + 1 < n_it) {
                        if (!wait_bar<kCritSleep>(do_full((it + 1) % NDS), ((it + 1) / NDS) & 1, ctl))
                            goto mma_teardown;
                        tc_fence_after();
                        issue_dp((it + 1) % NDS);
                    }
#pragma unroll
                    for (int s2 = 0; s2 < NKV; ++s2) step_dv(ds, b, it, s2);
                    mma_commit(do_empty(ds));
                    if (it + 2 < n_it) {
                        if (!wait_bar<kCritSleep>(q_full((it + 2) % NQS), ((it + 2) / NQS) & 1, ctl))
                            goto mma_teardown;
                        FA_TRACE_EVENT(11, it);
                        tc_fence_after();
                        issue_s((it + 2) % NQS, b);
                    }
                    FA_TRACE_EVENT(1, it);
                    if (it > 0) {
                        if (!wait_bar<kCritSleep>(dq_empty, (it - 1) & 1, ctl)) goto mma_teardown;
                        tc_fence_after();
                    }
                    // dQ0 dK0 dQ1 dK1 ... dQ3 dK3 dQ4 .. dQ7: alternate accumulators where possible
#pragma unroll
                    for (int s2 = 0; s2 < NQ; ++s2) {
                        step_dq(b, s2);
                        if (s2 < NKV) step_dk(qs, b, it, s2);
                    }
                    mma_commit(dq_full);
                    mma_commit(q_empty(qs));
                    mma_commit(ds_empty(b));
                    FA_TRACE_EVENT(2, it);
                } else {
                    // single S buffer (compute(it) has read it): S and dP of it+1 first
                    if (it + 1 < n_it) {
                        if (!wait_bar<kCritSleep>(q_full((it + 1) % NQS), ((it + 1) / NQS) & 1, ctl))
                            goto mma_teardown;
                        tc_fence_after();
                        issue_s((it + 1) % NQS, 0);
                        if (!wait_bar<kCritSleep>(do_full((it + 1) % NDS), ((it + 1) / NDS) & 1, ctl))
                            goto mma_teardown;
                        tc_fence_after();
                        issue_dp((it + 1) % NDS);
                    }
#pragma unroll
                    for (int s2 = 0; s2 < NKV; ++s2) step_dv(ds, b, it, s2);
                    mma_commit(p_free);
                    mma_commit(do_empty(ds));
                    if (it > 0) {
                        if (!wait_bar<kCritSleep>(dq_empty, (it - 1) & 1, ctl)) goto mma_teardown;
                        tc_fence_after();
                    }
                    // dQ0 dK0 dQ1 dK1 ...
#pragma unroll
                    for (int s2 = 0; s2 < NQ; ++s2) {
                        step_dq(b, s2);
                        if (s2 < NKV) step_dk(qs, b, it, s2);
                    }
                    mma_commit(dq_full);
                    mma_commit(q_empty(qs));
                    mma_commit(ds_empty(b));
                }
            }
            mma_commit(dkv_full);
        mma_teardown:
            mma_commit(mma_done);
            volatile int never = 0;
            Ctl drain{&never, 100000000ull};
            wait_bar(mma_done, 0, drain);
        }
    } else if (warp < 8) {
        // ------------------------------------------------------------ compute
        const int h = warp >> 2, wq = warp & 3;
        const int key = kt * kBN + 32 * wq + lane;
        const uint32_t lane_base = tmem + ((32u * wq) << 16);
        const float eff = p.sl2_eff, sl2 = p.sl2;
        const bool prescale = p.prescale != 0;
        constexpr int NCH = C::kHalf / 32;  // 32-column chunks per thread
        for (int it = 0; it < n_it; ++it) {
            const int st = it % NQS, b = it & 1;
            const int sb = C::kSDouble ? b : 0;
            const int qt = q_tile_of(it), q0 = qt * BM;
            const bool masked = bwd_tile_class(T, CAUSAL, BM, qt, kt) == kMasked;
            if (!warp_wait(q_full(st), (it / NQS) & 1, ctl)) break;
            if (!warp_wait<kCritSleep>(s_full(sb), C::kSDouble ? ((it >> 1) & 1) : (it & 1), ctl)) break;
            if (warp == 0 && lane == 0) FA_TRACE_EVENT(3, it);
            if (lane == 0) FA_TRACE_EVENT(18 + warp, it);
            tc_fence_after();
            const float4* lse4 = reinterpret_cast<const float4*>(smem + (sLse(st) - sbase));
            const float4* dv4 = reinterpret_cast<const float4*>(smem + (sDv(st) - sbase));
            // P^T for all of this thread's columns (S fully read before P is written over it)
            uint32_t sr[C::kHalf];
#pragma unroll
            for (int ch = 0; ch < NCH; ++ch)
                tmem_ld32(lane_base + C::kS + sb * BM + h * C::kHalf + 32 * ch, sr + 32 * ch);
            tmem_ld_wait();
#pragma unroll
            for (int ch = 0; ch < NCH; ++ch) reg_fence32(sr + 32 * ch);
            float* pf = reinterpret_cast<float*>(sr);
            if (prescale) {
#pragma unroll
                for (int e = 0; e < C::kHalf; ++e) pf[e] *= sl2;
            }
            // P^T = exp2(S^T c - LSE2): one packed FMA per pair (the smem vector holds -LSE2)
            const uint64_t eff2 = f2(eff, eff);
#pragma unroll
            for (int e4 = 0; e4 < C::kHalf / 4; ++e4) {
                const float4 l4 = lse4[(h * C::kHalf) / 4 + e4];
                float x0, x1, x2, x3;
                f2_split(fma2(f2(pf[4 * e4 + 0], pf[4 * e4 + 1]), eff2, f2(l4.x, l4.y)), x0, x1);
                f2_split(fma2(f2(pf[4 * e4 + 2], pf[4 * e4 + 3]), eff2, f2(l4.z, l4.w)), x2, x3);
                pf[4 * e4 + 0] = ex2_approx(x0);
                pf[4 * e4 + 1] = ex2_approx(x1);
                pf[4 * e4 + 2] = ex2_approx(x2);
                pf[4 * e4 + 3] = ex2_approx(x3);
            }
            if (masked) {
#pragma unroll
                for (int e = 0; e < C::kHalf; ++e)
                    if (!bwd_elem_visible(T, CAUSAL, q0 + h * C::kHalf + e, key)) pf[e] = 0.f;
            }
            {
                uint32_t pk[C::kHalf / 2];
#pragma unroll
                for (int e = 0; e < C::kHalf / 2; ++e) pk[e] = pack_bf16x2(pf[2 * e], pf[2 * e + 1]);
                if constexpr (!C::kSDouble) {
                    // P has its own region; dV(it-1) must have read the previous P
                    if (it > 0 && !warp_wait(p_free, (it - 1) & 1, ctl)) break;
                }
                const uint32_t pcol =
                    C::kSDouble ? (C::kS + sb * BM + BM / 4 + h * C::kHalf / 2) : (C::kP + h * C::kHalf / 2);
#pragma unroll
                for (int c = 0; c < C::kHalf / 32; ++c) tmem_st16(lane_base + pcol + 16 * c, pk + 16 * c);
            }
            if (warp == 0 && lane == 0) FA_TRACE_EVENT(4, it);
            if (!warp_wait<kCritSleep>(dp_full, it & 1, ctl)) break;
            if (warp == 0 && lane == 0) FA_TRACE_EVENT(5, it);
            if (lane == 0 && warp == 1) FA_TRACE_EVENT(26, it);
            if (lane == 0 && warp == 5) FA_TRACE_EVENT(27, it);
            if (!warp_wait(ds_empty(b), ((it >> 1) & 1) ^ 1, ctl)) break;
            tc_fence_after();
            const uint32_t ds_base = sDS(b);
#pragma unroll
            for (int ch = 0; ch < NCH; ++ch) {
                const int c0 = h * C::kHalf + 32 * ch;
                uint32_t dr[32];
                tmem_ld32(lane_base + C::kDP + c0, dr);
                tmem_ld_wait();
                reg_fence32(dr);
                // dS^T row `key`, query columns c0 .. c0+31 -> 4 chunks of 8 in the swizzled tile
#pragma unroll
                for (int g = 0; g < 4; ++g) {
                    // dS^T = P^T o (dP^T - D): packed add of -D, packed multiply
                    const float4 da = dv4[(c0 + 8 * g) / 4], db = dv4[(c0 + 8 * g) / 4 + 1];
                    const uint64_t nd[4] = {f2(da.x, da.y), f2(da.z, da.w), f2(db.x, db.y), f2(db.z, db.w)};
                    uint32_t w4[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int c = 8 * g + 2 * e;
                        const uint64_t t2 = add2(f2(__uint_as_float(dr[c]), __uint_as_float(dr[c + 1])), nd[e]);
                        float d0, d1;
                        f2_split(mul2(f2(pf[32 * ch + c], pf[32 * ch + c + 1]), t2), d0, d1);
                        w4[e] = pack_bf16x2(d0, d1);
                    }
                    const int col = c0 + 8 * g;
                    st_shared_v4(ds_base + (col >> 6) * (128 * 128) + sw128_off(32 * wq + lane, (col & 63) >> 3),
                                 w4[0], w4[1], w4[2], w4[3]);
                }
            }
            tmem_st_wait();
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) FA_TRACE_EVENT(6 + (warp == 0 ? 0 : 0), it);
            if (lane == 0 && warp > 0) FA_TRACE_EVENT(12 + warp - 1, it);
            if (warp == 7 && lane == 0) FA_TRACE_EVENT(9, it);
            if (lane == 0) mbar_arrive(p_full);
        }
    } else {
        // ------------------------------------------------------------ dQ drain + dK/dV epilogue (warps 8-11)
        const int wq = warp - 8;
        const uint32_t lane_base = tmem + ((32u * wq) << 16);
        const int r = 32 * wq + lane;  // TMEM lane of this thread
        bool ok = true;
        for (int it = 0; it < n_it; ++it) {
            const int q0 = q_tile_of(it) * BM, bhq = q_head_of(it);
            if (!warp_wait(dq_full, it & 1, ctl)) {
                ok = false;
                break;
            }
            if (warp == 8 && lane == 0) FA_TRACE_EVENT(7, it);
            tc_fence_after();
            uint32_t v[64];
            tmem_ld32(lane_base + C::kDQ, v);
            tmem_ld32(lane_base + C::kDQ + 32, v + 32);
            tmem_ld_wait();
            reg_fence32(v);
            reg_fence32(v + 32);
            // the tile is in registers: hand the TMEM columns back before the reductions
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(dq_empty);
            if constexpr (C::kDqT) {
                // lane = d; columns = queries q0 .. q0+63
                float* base = p.dqacc + (static_cast<size_t>(bhq) * T + q0) * D + r;
                if (q0 + 64 <= T) {
#pragma unroll
                    for (int e = 0; e < 64; ++e) atomicAdd(base + static_cast<size_t>(e) * D, __uint_as_float(v[e]));
                } else {
#pragma unroll
                    for (int e = 0; e < 64; ++e)
                        if (q0 + e < T) atomicAdd(base + static_cast<size_t>(e) * D, __uint_as_float(v[e]));
                }
            } else {
                // lane = query row q0 + r; columns = d
                if (q0 + r < T) {
                    float* base = p.dqacc + (static_cast<size_t>(bhq) * T + q0 + r) * D;
#pragma unroll
                    for (int e = 0; e < 64; e += 4)
                        red_add_v4_f32(base + e, __uint_as_float(v[e]), __uint_as_float(v[e + 1]),
                                       __uint_as_float(v[e + 2]), __uint_as_float(v[e + 3]));
                }
            }
            if (warp == 8 && lane == 0) FA_TRACE_EVENT(8, it);
        }
        if (ok && warp_wait(dkv_full, 0, ctl)) {
            tc_fence_after();
            const int key = kt * kBN + r;
#pragma unroll
            for (int which = 0; which < 2; ++which) {
                const uint32_t col = which ? C::kDV : C::kDK;
                const float mul = which ? 1.f : p.scale;
                __nv_bfloat16* out = which ? p.dv : p.dk;
#pragma unroll
                for (int ch = 0; ch < D / 32; ++ch) {
                    uint32_t v[32];
                    tmem_ld32(lane_base + col + 32 * ch, v);
                    tmem_ld_wait();
                    reg_fence32(v);
                    if (key < T) {
                        uint4* dst = reinterpret_cast<uint4*>(out + (static_cast<size_t>(bh) * T + key) * D + 32 * ch);
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
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 13) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

template <int D, bool CAUSAL>
int launch_main_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& tdo,
                  const BwdParams& p, cudaStream_t st) {
    static bool attr_set = false;
    auto kern = fa_bwd_main_kernel<D, CAUSAL>;
    if (!attr_set) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, BwdCfg<D>::kSmemBytes) !=
            cudaSuccess)
            return -5;
        attr_set = true;
    }
    kern<<<p.n_kt * p.BH, kBwdThreads, BwdCfg<D>::kSmemBytes, st>>>(tq, tk, tv, tdo, p);
    return cudaGetLastError() == cudaSuccess ? 0 : -5;
}

}  // namespace

int launch_bwd(const void* q, const void* k, const void* v, const void* o, const void* dO, const float* lse,
               void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int T, int D, float scale, bool causal,
               cudaStream_t stream, const DebugKnobs& dbg, int num_sms) {
    const int BH = B * Hq;        // query heads: D, LSE2, dQ accumulator, Q/dO tensor maps
    const int BHkv = B * Hkv;     // key/value heads: K/V tensor maps, grid rows
    const int T_pad = cdiv(T, 128) * 128;
    const size_t n_vec = static_cast<size_t>(BH) * T_pad;
    const size_t n_acc = static_cast<size_t>(BH) * T * D;
    const size_t bytes_vec = (n_vec * 4 + 255) / 256 * 256;
    const size_t bytes = 2 * bytes_vec + n_acc * 4;
    void* ws = nullptr;
    if (cudaMallocAsync(&ws, bytes, stream) != cudaSuccess) {
        cudaGetLastError();
        return -6;
    }
    float* dvec = static_cast<float*>(ws);
    float* lse2 = reinterpret_cast<float*>(static_cast<char*>(ws) + bytes_vec);
    float* dqacc = reinterpret_cast<float*>(static_cast<char*>(ws) + 2 * bytes_vec);
    int rc = 0;
    CUtensorMap tq, tk, tv, tdo;
    const int bm = bwd_bm(D);
    if (!make_tmap_bhtd(&tq, q, BH, T, D, bm) || !make_tmap_bhtd(&tk, k, BHkv, T, D, 128) ||
        !make_tmap_bhtd(&tv, v, BHkv, T, D, 128) || !make_tmap_bhtd(&tdo, dO, BH, T, D, bm)) {
        rc = -5;
    } else {
        const long long rows = static_cast<long long>(BH) * T_pad;
        const int tpr = D / 8;
        long long blocks = (rows * tpr + 255) / 256;
        const int pre_grid = static_cast<int>(blocks < 8LL * num_sms ? blocks : 8LL * num_sms);
        if (D == 64)
            fa_bwd_pre_kernel<64><<<pre_grid, 256, 0, stream>>>(static_cast<const __nv_bfloat16*>(o),
                                                                static_cast<const __nv_bfloat16*>(dO), lse, dvec,
                                                                lse2, dqacc, BH, T, T_pad);
        else
            fa_bwd_pre_kernel<128><<<pre_grid, 256, 0, stream>>>(static_cast<const __nv_bfloat16*>(o),
                                                                 static_cast<const __nv_bfloat16*>(dO), lse, dvec,
                                                                 lse2, dqacc, BH, T, T_pad);
        if (cudaGetLastError() != cudaSuccess) rc = -5;
        if (rc == 0) {
            BwdParams p;
            p.lse2 = lse2;
            p.dvec = dvec;
            p.dqacc = dqacc;
            p.dk = static_cast<__nv_bfloat16*>(dk);
            p.dv = static_cast<__nv_bfloat16*>(dv);
            p.T = T;
            p.T_pad = T_pad;
            p.BH = BHkv;
            p.Hq = Hq;
            p.Hkv = Hkv;
            p.group = Hq / Hkv;
            p.n_kt = cdiv(T, kBN);
            p.scale = scale;
            p.sl2 = scale * kLog2e;
            p.prescale = p.sl2 > 0.f ? 0 : 1;
            p.sl2_eff = p.prescale ? 1.f : p.sl2;
            p.timeout_ns = dbg.timeout_ns;
            if (dbg.ev[2]) cudaEventRecord(dbg.ev[2], stream);
            if (D == 64)
                rc = causal ? launch_main_t<64, true>(tq, tk, tv, tdo, p, stream)
                            : launch_main_t<64, false>(tq, tk, tv, tdo, p, stream);
            else
                rc = causal ? launch_main_t<128, true>(tq, tk, tv, tdo, p, stream)
                            : launch_main_t<128, false>(tq, tk, tv, tdo, p, stream);
            if (dbg.ev[3]) cudaEventRecord(dbg.ev[3], stream);
        }
        if (rc == 0) {
            const long long n8 = static_cast<long long>(n_acc / 8);
            long long blocks8 = (n8 + 255) / 256;
            const int g = static_cast<int>(blocks8 < 8LL * num_sms ? blocks8 : 8LL * num_sms);
            fa_bwd_dq_kernel<<<g, 256, 0, stream>>>(dqacc, static_cast<__nv_bfloat16*>(dq), n8, scale);
            if (cudaGetLastError() != cudaSuccess) rc = -5;
        }
    }
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
// device (the first fa_bwd_noalloc call on that device does it).
void* scratch_address(int dev) {
    std::call_once(g_scratch_once[dev], [dev] {
        void* p = nullptr;
        g_scratch_err[dev] = cudaGetSymbolAddress(&p, g_bwd_scratch);
        g_scratch_ptr[dev] = p;
    });
    return g_scratch_err[dev] == cudaSuccess ? g_scratch_ptr[dev] : nullptr;
}
}  // namespace

size_t bwd_scratch_bytes(int B, int H, int T, int D) {
    const size_t BH = static_cast<size_t>(B) * H;
    const size_t T_pad = static_cast<size_t>(cdiv(T, 128)) * 128;
    const size_t bytes_vec = (BH * T_pad * 4 + 255) / 256 * 256;
    return 2 * bytes_vec + BH * static_cast<size_t>(T) * D * 4;
}

int launch_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const void* dO, const float* lse,
                       void* dq, void* dk, void* dv, int B, int H, int T, int D, float scale, bool causal,
                       cudaStream_t stream, const DebugKnobs& dbg, int num_sms) {
    if (bwd_scratch_bytes(B, H, T, D) > FA_BWD_NOALLOC_SCRATCH_BYTES) return -10;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kScratchMaxDevices) return -5;
    void* ws = scratch_address(dev);
    if (!ws) return -5;
    const int BH = B * H;
    const int T_pad = cdiv(T, 128) * 128;
    const size_t bytes_vec = (static_cast<size_t>(BH) * T_pad * 4 + 255) / 256 * 256;
    const size_t n_acc = static_cast<size_t>(BH) * T * D;
    float* dvec = static_cast<float*>(ws);
    float* lse2 = reinterpret_cast<float*>(static_cast<char*>(ws) + bytes_vec);
    float* dqacc = reinterpret_cast<float*>(static_cast<char*>(ws) + 2 * bytes_vec);
    CUtensorMap tq, tk, tv, tdo;
    const int bm = bwd_bm(D);
    if (!make_tmap_bhtd(&tq, q, BH, T, D, bm) || !make_tmap_bhtd(&tk, k, BH, T, D, 128) ||
        !make_tmap_bhtd(&tv, v, BH, T, D, 128) || !make_tmap_bhtd(&tdo, dO, BH, T, D, bm))
        return -5;
    // preprocess clears the accumulator, so the previous call's contents do not matter
    const long long rows = static_cast<long long>(BH) * T_pad;
    const long long blocks = (rows * (D / 8) + 255) / 256;
    const int pre_grid = static_cast<int>(blocks < 8LL * num_sms ? blocks : 8LL * num_sms);
    if (D == 64)
        fa_bwd_pre_kernel<64><<<pre_grid, 256, 0, stream>>>(static_cast<const __nv_bfloat16*>(o),
                                                            static_cast<const __nv_bfloat16*>(dO), lse, dvec, lse2,
                                                            dqacc, BH, T, T_pad);
    else
        fa_bwd_pre_kernel<128><<<pre_grid, 256, 0, stream>>>(static_cast<const __nv_bfloat16*>(o),
                                                             static_cast<const __nv_bfloat16*>(dO), lse, dvec, lse2,
                                                             dqacc, BH, T, T_pad);
    if (cudaGetLastError() != cudaSuccess) return -5;
    BwdParams p;
    p.lse2 = lse2;
    p.dvec = dvec;
    p.dqacc = dqacc;
    p.dk = static_cast<__nv_bfloat16*>(dk);
    p.dv = static_cast<__nv_bfloat16*>(dv);
    p.T = T;
    p.T_pad = T_pad;
    p.BH = BH;
    p.Hq = p.Hkv = H;
    p.group = 1;
    p.n_kt = cdiv(T, kBN);
    p.scale = scale;
    p.sl2 = scale * kLog2e;
    p.prescale = p.sl2 > 0.f ? 0 : 1;
    p.sl2_eff = p.prescale ? 1.f : p.sl2;
    p.timeout_ns = dbg.timeout_ns;
    int rc;
    if (D == 64)
        rc = causal ? launch_main_t<64, true>(tq, tk, tv, tdo, p, stream)
                    : launch_main_t<64, false>(tq, tk, tv, tdo, p, stream);
    else
        rc = causal ? launch_main_t<128, true>(tq, tk, tv, tdo, p, stream)
                    : launch_main_t<128, false>(tq, tk, tv, tdo, p, stream);
    if (rc != 0) return rc;
    const long long n8 = static_cast<long long>(n_acc / 8);
    const long long blocks8 = (n8 + 255) / 256;
    const int g = static_cast<int>(blocks8 < 8LL * num_sms ? blocks8 : 8LL * num_sms);
    fa_bwd_dq_kernel<<<g, 256, 0, stream>>>(dqacc, static_cast<__nv_bfloat16*>(dq), n8, scale);
    return cudaGetLastError() == cudaSuccess ? 0 : -5;
}

#ifdef FA_TRACE
// Copies the trace of the last traced launch (kTraceSlots x kTraceLen cycle stamps).
extern "C" int fa_trace_read(unsigned long long* host) {
    return cudaMemcpyFromSymbol(host, g_trace, sizeof(g_trace)) == cudaSuccess ? 0 : -5;
}
#endif

int bwd_take_status() {
    int h = 0, z = 0;
    if (cudaMemcpyFromSymbol(&h, g_status_bwd, sizeof(int)) != cudaSuccess) return -5;
    if (cudaMemcpyToSymbol(g_status_bwd, &z, sizeof(int)) != cudaSuccess) return -5;
    return h;
}

}  // namespace fa
