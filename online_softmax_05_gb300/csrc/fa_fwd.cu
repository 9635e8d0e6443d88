// fa_fwd.cu -- exact attention forward on sm_103a with the online-softmax
// recurrence ("Lab 06 - Attention kernels", section 3; "Triton
// FlashAttention-2 forward", section "The kernel"; "Flash Attention and
// Kernel Optimization", sections "Running softmax state", "Causal masking",
// "Output and saved state").
//
// One persistent CTA per SM walks work items (pair of 128-row query tiles,
// batch*head; when there are too few pairs to fill half the SMs, a single
// query tile whose key tiles the two softmax warpgroups split, their running
// states merged at the end).  Warp roles:
//   warps 0-3  softmax for query tile 0 (one TMEM lane = one query row each)
//   warps 4-7  softmax for query tile 1
//   warp 8     TMA producer: Q tiles once per item, K/V tiles into a ring
//   warp 9     tcgen05 issuer: S = Q K^T into TMEM, O += P V with P in TMEM
// Per key tile j the softmax warps read S_t(j) from TMEM, update the running
// max m (log2 domain, scale*log2(e) folded in), rescale O when m grows
// (see the rescale policy below), write P = exp2(S*c - m) as bf16 back
// into the same TMEM columns and hand it to the MMA warp.  The two query
// tiles ping-pong: the softmax of one overlaps the tensor-core work of the
// other.  Finally O = acc / l goes out through shared memory with a TMA store
// and LSE = (m + log2 l) * ln 2 is written per row.
//
// Rescale policy: O = acc / l and LSE = m_used + log l hold for ANY
// reference m_used ("Lab 06", section 2, "Why the rescale is exact"), so the
// rescale could be deferred while the max grows by less than a threshold.
// It is not: P is rounded to bf16 before P V, and a dominant weight
// 2^delta (0 < delta) is not a bf16 number, so a near-one-hot row would
// carry up to 2^-9 relative error in O.  With the reference equal to the
// running max the dominant weight is exp2(0) = 1, exact in bf16.
#include <cuda_runtime.h>

#include "fa_check.cuh"
#include "fa_internal.h"
#include "fa_ptx.cuh"
#include "fa_sched.h"
#include "fa_tmap.h"

namespace fa {

static __device__ int g_status_fwd;

namespace {

constexpr int kFwdThreads = 320;
constexpr float kRescaleThreshold = 0.0f;  // log2 units; see the rescale policy above
constexpr float kLn2 = 0.69314718055994530942f;
constexpr float kLog2e = 1.44269504088896340736f;

template <int D>
struct FwdCfg {
    static constexpr int kAtoms = D / 64;             // 128-byte swizzle atoms per row
    static constexpr int kAtomBytes = 128 * 128;      // one atom column of a 128-row tile
    static constexpr int kTileBytes = 128 * D * 2;    // one 128 x D bf16 tile
    static constexpr int kStages = (D == 128) ? 4 : 8;
    static constexpr int kQOff = 0;
    static constexpr int kKVOff = 2 * kTileBytes;
    static constexpr int kBarOff = kKVOff + kStages * kTileBytes;
    // barriers: q_full[2] q_empty[2] kv_full[S] kv_empty[S] s_full[2] p_full[2] o_full[2] epi[2] mma_done
    // ph_full[2] mrg_full mrg_done
    static constexpr int kNumBars = 4 + 2 * kStages + 8 + 1 + 2 + 2;
    // split items: the second warpgroup's row max and row sum, 2 x 128 floats
    static constexpr int kMrgOff = kBarOff + kNumBars * 8;
    static constexpr int kMiscOff = kMrgOff + 2 * 128 * 4;
    static constexpr int kSmemBytes = kMiscOff + 16 + 1024;  // + tmem slot, abort flag, alignment slack
    // TMEM columns (512 allocated): S0, S1 (P aliases their first 64 columns), O0, O1
    __device__ static constexpr uint32_t kS(int t) { return 128u * t; }
    __device__ static constexpr uint32_t kO(int t) { return 256u + 128u * t; }
    static constexpr uint32_t kIdescS = idesc_bf16_f32(128, 128, false, false);
    static constexpr uint32_t kIdescPV = idesc_bf16_f32(128, D, false, true);
};

struct FwdParams {
    float* lse;
    int T, BH, n_pairs, n_items;
    int Hq, Hkv, group;   // query heads, key/value heads, Hq / Hkv
    // Packed variable-length batch: sequence s occupies rows cu_seqlens[s] ..
    // cu_seqlens[s+1]-1 of (total, H, D) tensors (T above is then the longest
    // length the caller promises; items past a sequence's end are skipped).
    const int* cu_seqlens;
    int n_seq, total;
    __nv_bfloat16* o_packed;  // O of the packed layout (stored row by row, not by TMA)
    int head_pairs;       // 1: the two query tiles of an item are two heads of one group at the same rows
    int n_tiles;          // query tiles per head
    int single_tiles;     // 1: an item is one query tile whose key tiles the two softmax warpgroups split
                          // (few items: each gets an SM of its own)
    int head_major;       // 1: items of one head are consecutive (no causal masking: every item weighs the
                          // same, so the CTAs in flight share few heads' K/V tiles in L2)
    float sl2_eff;  // multiplier applied inside exp2: scale*log2e, or 1 when prescaled
    float sl2;      // scale * log2(e)
    int prescale;   // 1 when scale <= 0: scores are multiplied by sl2 before the max
    unsigned long long timeout_ns;
    int inject;
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
            atomicCAS(&g_status_fwd, 0, kStatusTimeout);
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
// Warp-uniform wait: lane 0 polls, the result is broadcast.
template <bool kSleep = true>
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, Ctl c) {
    int ok = 0;
    if ((threadIdx.x & 31) == 0) ok = wait_bar<kSleep>(bar, parity, c);
    return __shfl_sync(0xffffffffu, ok, 0) != 0;
}
// Bounded wait taken by every lane of a converged warp; the result is the same
// in all lanes.  The MMA warp waits this way: the issue loop then stays
// warp-uniform and elect.sync picks the lane that issues, which keeps the
// tensor pipe fed across waits and fences (a loop run by lane 0 alone leaves
// a gap of about 60 cycles at each wait).
template <bool kSleep = false>
__device__ __forceinline__ bool wait_all(uint32_t bar, uint32_t parity, Ctl c) {
    const bool ok = mbar_try_wait(bar, parity) || wait_slow<kSleep>(bar, parity, c);
    return __all_sync(0xffffffffu, ok);
}

// A work item: two 128-row query tiles that share every K/V tile they read.
// Without grouped heads (or with an odd group) they are consecutive tiles of
// one head; with an even group of query heads per K/V head they are the same
// rows of two heads of one group ("Lab 06", "Check yourself" item 7: a K/V
// tile loaded once serves several query heads).
struct FwdItem {
    int tile[2];  // query tile index of each half (within its sequence)
    int bh[2];    // head coordinate of each half's Q / O rows in the tensor maps
    int bh_kv;    // head coordinate of the K/V rows
    int T;        // length of this item's sequence
    int row0;     // row coordinate of the sequence's first token (0 unless packed)
    bool valid0;  // the first half has rows < T (false: skip the item)
    bool valid1;  // the second half has rows < T
};
template <bool VARLEN>
__device__ __forceinline__ FwdItem fwd_item(int w, const FwdParams& p) {
    FwdItem it;
    it.T = p.T;
    it.row0 = 0;
    it.valid0 = true;
    if constexpr (VARLEN) {
        // items: (pair of query tiles, sequence, head), heaviest pairs first
        const int per_pair = p.n_seq * p.Hq;
        const int pair = p.n_pairs - 1 - w / per_pair, rem = w % per_pair;
        const int sq = rem / p.Hq, h = rem % p.Hq;
        it.row0 = p.cu_seqlens[sq];
        it.T = p.cu_seqlens[sq + 1] - it.row0;
        it.tile[0] = 2 * pair;
        it.tile[1] = 2 * pair + 1;
        it.bh[0] = it.bh[1] = h;
        it.bh_kv = h / p.group;
        // a sequence that is longer than max_seqlen, negative, or outside the
        // packed rows is skipped by every role alike and reported
        const bool bad = it.T < 0 || it.T > p.T || it.row0 < 0 || it.row0 + it.T > p.total;
        if (bad) {
            atomicCAS(&g_status_fwd, 0, kStatusBadSeqlen);
            it.T = 0;
        }
        it.valid0 = it.tile[0] * kFwdBM < it.T;
        it.valid1 = it.tile[1] * kFwdBM < it.T;
        return it;
    }
    if (p.single_tiles) {
        // (query tile, head), heaviest tiles first; the second half is empty
        const int t = p.head_major ? w % p.n_tiles : p.n_tiles - 1 - w / p.BH;
        const int bh = p.head_major ? w / p.n_tiles : w % p.BH;
        it.tile[0] = it.tile[1] = t;  // the second warpgroup takes the second half of the key tiles
        it.bh[0] = it.bh[1] = bh;
        it.bh_kv = (bh / p.Hq) * p.Hkv + (bh % p.Hq) / p.group;
        it.valid1 = false;  // no second Q tile
    } else if (p.head_pairs) {
        const int per_t = p.BH / 2;  // head pairs over all batches
        const int t = p.head_major ? w % p.n_tiles : p.n_tiles - 1 - w / per_t;
        const int rem = p.head_major ? w / p.n_tiles : w % per_t;
        const int hp = rem % (p.Hq / 2), b = rem / (p.Hq / 2);
        it.tile[0] = it.tile[1] = t;
        it.bh[0] = b * p.Hq + 2 * hp;
        it.bh[1] = it.bh[0] + 1;
        it.bh_kv = b * p.Hkv + (2 * hp) / p.group;
        it.valid1 = true;
    } else {
        const int pair = p.head_major ? w % p.n_pairs : p.n_pairs - 1 - w / p.BH;
        const int bh = p.head_major ? w / p.n_pairs : w % p.BH;
        it.tile[0] = 2 * pair;
        it.tile[1] = 2 * pair + 1;
        it.bh[0] = it.bh[1] = bh;
        it.bh_kv = (bh / p.Hq) * p.Hkv + (bh % p.Hq) / p.group;
        it.valid1 = it.tile[1] * kFwdBM < p.T;
    }
    return it;
}

// Item k of this CTA in snake order over items sorted heaviest first
// (causal: later query tiles see more key tiles).
__device__ __forceinline__ int item_of(int k, int n_items) {
    int G = gridDim.x;
    int w = k * G + ((k & 1) ? (G - 1 - static_cast<int>(blockIdx.x)) : static_cast<int>(blockIdx.x));
    return w < n_items ? w : -1;
}

// SPLIT: every item is one query tile whose key tiles the two softmax
// warpgroups split (launched when the items are too few to fill the SMs);
// compiled apart so the paired kernel carries none of it.
template <int D, bool CAUSAL, bool VARLEN, bool SPLIT>
__global__ void __launch_bounds__(kFwdThreads, 1)
    fa_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o, FwdParams p) {
    using C = FwdCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const uint32_t sQ[2] = {sbase + C::kQOff, sbase + C::kQOff + C::kTileBytes};
    const uint32_t sKV = sbase + C::kKVOff;
    const uint32_t bars = sbase + C::kBarOff;
    auto q_full = [&](int t) { return bars + 8u * t; };
    auto q_empty = [&](int t) { return bars + 8u * (2 + t); };
    auto kv_full = [&](int s) { return bars + 8u * (4 + s); };
    auto kv_empty = [&](int s) { return bars + 8u * (4 + C::kStages + s); };
    auto s_full = [&](int t) { return bars + 8u * (4 + 2 * C::kStages + t); };
    auto p_full = [&](int t) { return bars + 8u * (6 + 2 * C::kStages + t); };
    auto o_full = [&](int t) { return bars + 8u * (8 + 2 * C::kStages + t); };
    auto epi_bar = [&](int t) { return bars + 8u * (10 + 2 * C::kStages + t); };
    const uint32_t mma_done = bars + 8u * (12 + 2 * C::kStages);
    // ph_full(t): the first half of P (keys 0..63) and the O rescale are done
    auto ph_full = [&](int t) { return bars + 8u * (13 + 2 * C::kStages + t); };
    // split items: the second warpgroup published its row max and sum, its O is complete
    // (4 warps) / the first warpgroup has read them and that O (4 warps)
    const uint32_t mrg_full = bars + 8u * (15 + 2 * C::kStages), mrg_done = bars + 8u * (16 + 2 * C::kStages);
    float* mrg = reinterpret_cast<float*>(smem + C::kMrgOff);  // [0][row] max (log2 units), [1][row] sum
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kMiscOff);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kMiscOff + 4);
    const Ctl ctl{abort_flag, p.timeout_ns};

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    if (tid == 0) {
        for (int t = 0; t < 2; ++t) {
            mbar_init(q_full(t), 1);
            mbar_init(q_empty(t), 1);
            mbar_init(s_full(t), 1);
            mbar_init(p_full(t), 4);
            mbar_init(ph_full(t), 4);
            mbar_init(o_full(t), 1);
            mbar_init(epi_bar(t), 4);
        }
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(kv_full(s), 1);
            mbar_init(kv_empty(s), 1);
        }
        mbar_init(mma_done, 1);
        mbar_init(mrg_full, 4);
        mbar_init(mrg_done, 4);
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
            uint32_t kv_cnt = 0, q_cnt[2] = {0, 0};
            uint32_t q_armed[2] = {0, 0};
            int skipped_fill = -1;  // fill index the test hook dropped
            const uint64_t pol_kv = l2_policy_evict_last();
            const uint64_t pol_q = l2_policy_evict_first();
            bool skip_first = (p.inject == 1);
            for (int k = 0;; ++k) {
                int w = item_of(k, p.n_items);
                if (w < 0) break;
                const FwdItem item = fwd_item<VARLEN>(w, p);
                if (!item.valid0) continue;
                const bool valid1 = item.valid1;
                const int n0 = fwd_num_kv_tiles(item.T, CAUSAL, item.tile[0]);
                const int n1 = valid1 ? fwd_num_kv_tiles(item.T, CAUSAL, item.tile[1]) : 0;
                const int nmax = n0 > n1 ? n0 : n1;
                const int bh = item.bh_kv;
                for (int t = 0; t < 2; ++t) {
                    if (t == 1 && !valid1) continue;
                    if (!wait_bar(q_empty(t), (q_cnt[t] & 1) ^ 1, ctl)) goto producer_done;
                    ++q_cnt[t];
                    const int qrow = item.row0 + item.tile[t] * kFwdBM;
                    // the tile starts inside its sequence and its head exists
                    if (!FA_CHECK(item.tile[t] * kFwdBM < item.T && qrow < (VARLEN ? p.total : p.T) &&
                                      item.bh[t] >= 0 && item.bh[t] < p.BH,
                                  &g_status_fwd, abort_flag))
                        goto producer_done;
                    mbar_arrive_expect_tx(q_full(t), C::kTileBytes);
                    ++q_armed[t];
                    for (int a = 0; a < C::kAtoms; ++a)
                        tma_load_3d_hint(sQ[t] + a * C::kAtomBytes, &tm_q, q_full(t), 64 * a,
                                         VARLEN ? item.bh[t] : qrow, VARLEN ? qrow : item.bh[t], pol_q);
                }
                // one K (kind 0) or V (kind 1) tile into the next ring stage
                auto fill = [&](int kind, int jt) -> bool {
                    const uint32_t slot = kv_cnt % C::kStages;
                    if (!wait_bar(kv_empty(slot), ((kv_cnt / C::kStages) & 1) ^ 1, ctl)) return false;
                    ++kv_cnt;
                    if (skip_first) {  // test hook: never deliver this tile
                        skip_first = false;
                        skipped_fill = static_cast<int>(kv_cnt - 1);
                        return true;
                    }
                    const int krow = item.row0 + jt * kBN;
                    // the key tile is one this query tile needs, inside the tensor, and its ring
                    // stage lies inside the shared-memory window
                    if (!FA_CHECK(jt * kBN < item.T && bh >= 0 && bh < p.BH / p.group &&
                                      C::kKVOff + (slot + 1) * C::kTileBytes <= C::kBarOff,
                                  &g_status_fwd, abort_flag)) {
                        --kv_cnt;  // nothing was armed: the drain must not wait for this fill
                        return false;
                    }
                    mbar_arrive_expect_tx(kv_full(slot), C::kTileBytes);
                    const CUtensorMap* tm = kind ? &tm_v : &tm_k;
                    for (int a = 0; a < C::kAtoms; ++a)
                        tma_load_3d_hint(sKV + slot * C::kTileBytes + a * C::kAtomBytes, tm, kv_full(slot), 64 * a,
                                         VARLEN ? bh : krow, VARLEN ? krow : bh, pol_kv);
                    return true;
                };
                if constexpr (SPLIT) {
                    // split item: warpgroup 0 takes key tiles 0 .. h-1, warpgroup 1 h .. n0-1,
                    // filled in the order the MMA warp consumes them
                    const int h = (n0 + 1) / 2, m1 = n0 - h;
                    if (!fill(0, 0)) goto producer_done;
                    if (m1 > 0 && !fill(0, h)) goto producer_done;
                    for (int j = 0; j < h; ++j) {
                        if (!fill(1, j)) goto producer_done;
                        if (j + 1 < h && !fill(0, j + 1)) goto producer_done;
                        if (j < m1) {
                            if (!fill(1, h + j)) goto producer_done;
                            if (j + 1 < m1 && !fill(0, h + j + 1)) goto producer_done;
                        }
                    }
                } else {
                    for (int j = 0; j < nmax; ++j)
                        for (int kind = 0; kind < 2; ++kind)
                            if (!fill(kind, j)) goto producer_done;
                }
            }
        producer_done:
            // make sure no copy is still landing in shared memory before exit
            Ctl drain{abort_flag, 100000000ull};
            volatile int never = 0;
            drain.abort = &never;
            // the last kStages fills are the only ones that can still be in flight
            for (uint32_t f = kv_cnt > C::kStages ? kv_cnt - C::kStages : 0; f < kv_cnt; ++f)
                if (static_cast<int>(f) != skipped_fill)
                    wait_bar(kv_full(f % C::kStages), (f / C::kStages) & 1, drain);
            for (int t = 0; t < 2; ++t)
                if (q_armed[t]) wait_bar(q_full(t), (q_armed[t] - 1) & 1, drain);
        }
    } else if (warp == 9) {
        // ------------------------------------------------------------ MMA issuer
        // The whole warp runs the loop; the elected lane issues and commits.
        {
            const bool leader = elect_one_sync();
            uint32_t kv_cnt = 0, q_cnt[2] = {0, 0}, p_cnt[2] = {0, 0};
            // Descriptors are built once; a tile / slot / k-step is an offset in 16-byte units.
            const SDesc dQ_km = sdesc_make(sQ[0], 16, 1024);
            const SDesc dKV_km = sdesc_make(sKV, 16, 1024);
            const SDesc dKV_mn = sdesc_make(sKV, C::kAtomBytes, 1024);
            constexpr uint32_t kTile16 = C::kTileBytes >> 4;
            // S_t = Q K^T into S buffer t, Q from Q buffer qb (split items: both use buffer 0)
            auto issue_s = [&](int t, uint32_t slot, int qb) {
                if (!FA_CHECK(t >= 0 && t < 2 && qb >= 0 && qb < 2 && slot < C::kStages && C::kS(t) + 128 <= 512u,
                              &g_status_fwd, abort_flag))
                    return;
                const uint32_t qo = qb * kTile16, ko = slot * kTile16;
#pragma unroll
                for (int s = 0; s < D / 16; ++s) {
                    const uint32_t off = ((s >> 2) * C::kAtomBytes + (s & 3) * 32) >> 4;
                    if (leader) mma_ss_d(tmem + C::kS(t), dQ_km, qo + off, dKV_km, ko + off, C::kIdescS, s > 0);
                }
            };
            // half h of O += P V: keys 64h .. 64h+63 (k-steps 4h .. 4h+3)
            auto issue_pv_half = [&](int t, uint32_t slot, bool acc, int h) {
                if (!FA_CHECK(t >= 0 && t < 2 && slot < C::kStages && C::kO(t) + D <= 512u, &g_status_fwd, abort_flag))
                    return;
                const uint32_t vo = slot * kTile16;
#pragma unroll
                for (int s = 4 * h; s < 4 * h + 4; ++s)
                    if (leader) mma_ts_d(tmem + C::kO(t), tmem + C::kS(t) + s * 8, dKV_mn, vo + s * (2048 >> 4), C::kIdescPV,
                             (acc || s > 0) ? 1u : 0u);
            };
            for (int k = 0;; ++k) {
                int w = item_of(k, p.n_items);
                if (w < 0) break;
                const FwdItem item = fwd_item<VARLEN>(w, p);
                if (!item.valid0) continue;
                const bool valid1 = item.valid1;
                const int n0 = fwd_num_kv_tiles(item.T, CAUSAL, item.tile[0]);
                const int n1 = valid1 ? fwd_num_kv_tiles(item.T, CAUSAL, item.tile[1]) : 0;
                const int nmax = n0 > n1 ? n0 : n1;
                if (!wait_all(q_full(0), q_cnt[0] & 1, ctl)) goto mma_done_label;
                ++q_cnt[0];
                if (valid1) {
                    if (!wait_all(q_full(1), q_cnt[1] & 1, ctl)) goto mma_done_label;
                    ++q_cnt[1];
                }
                if constexpr (SPLIT) {
                    // Split item: one query tile (Q buffer 0); S buffer / warpgroup 0 takes key
                    // tiles 0 .. h-1, S buffer / warpgroup 1 takes h .. n0-1, each with its own K
                    // and V tiles, in the order the producer fills them.
                    const int h = (n0 + 1) / 2, cnt[2] = {h, n0 - h};
                    auto next_slot = [&](uint32_t& slot) -> bool {
                        slot = kv_cnt % C::kStages;
                        if (!wait_all(kv_full(slot), (kv_cnt / C::kStages) & 1, ctl)) return false;
                        ++kv_cnt;
                        tc_fence_after();
                        return true;
                    };
                    for (int t = 0; t < 2; ++t) {
                        if (cnt[t] == 0) continue;
                        uint32_t ks;
                        if (!next_slot(ks)) goto mma_done_label;
                        issue_s(t, ks, 0);
                        if (leader) {
                            mma_commit(s_full(t));
                            mma_commit(kv_empty(ks));
                        }
                    }
                    for (int j = 0; j < h; ++j) {
                        for (int t = 0; t < 2; ++t) {
                            if (j >= cnt[t]) continue;
                            uint32_t vs;
                            if (!next_slot(vs)) goto mma_done_label;
                            if (!wait_all(ph_full(t), p_cnt[t] & 1, ctl)) goto mma_done_label;
                            tc_fence_after();
                            issue_pv_half(t, vs, j > 0, 0);
                            if (!wait_all(p_full(t), p_cnt[t] & 1, ctl)) goto mma_done_label;
                            ++p_cnt[t];
                            tc_fence_after();
                            issue_pv_half(t, vs, true, 1);
                            if (leader) mma_commit(kv_empty(vs));
                            if (j + 1 < cnt[t]) {
                                uint32_t ks;
                                if (!next_slot(ks)) goto mma_done_label;
                                issue_s(t, ks, 0);
                                if (leader) {
                                    mma_commit(s_full(t));
                                    mma_commit(kv_empty(ks));
                                }
                            } else {
                                if (leader) mma_commit(o_full(t));
                            }
                        }
                    }
                    continue;
                }
                {
                    const uint32_t ks = kv_cnt % C::kStages;
                    if (!wait_all(kv_full(ks), (kv_cnt / C::kStages) & 1, ctl)) goto mma_done_label;
                    ++kv_cnt;
                    tc_fence_after();
                    issue_s(0, ks, 0);
                    if (leader) mma_commit(s_full(0));
                    if (n1 > 0) {
                        issue_s(1, ks, 1);
                        if (leader) mma_commit(s_full(1));
                    }
                    if (leader) mma_commit(kv_empty(ks));
                }
                for (int j = 0; j < nmax; ++j) {
                    const uint32_t vs = kv_cnt % C::kStages;
                    if (!wait_all(kv_full(vs), (kv_cnt / C::kStages) & 1, ctl)) goto mma_done_label;
                    ++kv_cnt;
                    tc_fence_after();
                    const bool has_next = j + 1 < nmax;
                    const uint32_t ks = kv_cnt % C::kStages;
                    bool k_ready = false;
                    for (int t = 0; t < 2; ++t) {
                        const int n = t ? n1 : n0;
                        if (j >= n) continue;
                        // the first half of P·V as soon as its half of P is in TMEM
                        if (!wait_all(ph_full(t), p_cnt[t] & 1, ctl)) goto mma_done_label;
                        tc_fence_after();
                        issue_pv_half(t, vs, j > 0, 0);
                        if (!wait_all(p_full(t), p_cnt[t] & 1, ctl)) goto mma_done_label;
                        ++p_cnt[t];
                        tc_fence_after();
                        issue_pv_half(t, vs, true, 1);
                        if (j + 1 < n) {
                            if (!k_ready) {
                                if (!wait_all(kv_full(ks), (kv_cnt / C::kStages) & 1, ctl)) goto mma_done_label;
                                tc_fence_after();
                                k_ready = true;
                            }
                            issue_s(t, ks, t);
                            if (leader) mma_commit(s_full(t));
                        } else {
                            if (leader) mma_commit(o_full(t));
                        }
                    }
                    if (leader) mma_commit(kv_empty(vs));
                    if (has_next) {
                        if (!k_ready) {
                            if (!wait_all(kv_full(ks), (kv_cnt / C::kStages) & 1, ctl)) goto mma_done_label;
                        }
                        if (leader) mma_commit(kv_empty(ks));
                        ++kv_cnt;
                    }
                }
            }
        mma_done_label:
            // every MMA issued so far must finish before TMEM is released
            if (leader) {
                mma_commit(mma_done);
                Ctl drain{abort_flag, 100000000ull};
                volatile int never = 0;
                drain.abort = &never;
                wait_bar(mma_done, 0, drain);
            }
            __syncwarp();
        }
    } else {
        // ------------------------------------------------------------ softmax (tile t)
        const int t = warp >> 2, wq = warp & 3;
        const int r_local = 32 * wq + lane;
        const uint32_t lane_base = tmem + ((32u * wq) << 16);
        const uint32_t tS = lane_base + C::kS(t), tO = lane_base + C::kO(t);
        uint32_t s_cnt = 0, o_cnt = 0, epi_cnt = 0, mrg_cnt = 0;
        const float eff = p.sl2_eff;
        constexpr bool split = SPLIT;
        if (!FA_CHECK(t < 2 && C::kS(t) + 128 <= 512u && C::kO(t) + D <= 512u, &g_status_fwd, abort_flag))
            goto softmax_done;
        for (int k = 0;; ++k) {
            int w = item_of(k, p.n_items);
            if (w < 0) break;
            const FwdItem item = fwd_item<VARLEN>(w, p);
            const int tile = item.tile[t], bh = item.bh[t], T = item.T;
            if (tile * kFwdBM >= T) continue;  // the second tile of an item may be empty (or the whole item)
            const int row = tile * kFwdBM + r_local;  // row within the sequence
            const int n_all = fwd_num_kv_tiles(T, CAUSAL, tile);
            // split item: this warpgroup's share of the key tiles (the first half, rounded up,
            // for warpgroup 0); otherwise all of them
            const int h_split = (n_all + 1) / 2;
            const int j_off = (split && t == 1) ? h_split : 0;
            const int n = split ? (t == 0 ? h_split : n_all - h_split) : n_all;
            float m_used = -INFINITY, l = 0.f;
            for (int jj = 0; jj < n; ++jj) {
                const int j = jj + j_off;  // key tile
                if (!warp_wait<false>(s_full(t), s_cnt & 1, ctl)) goto softmax_done;
                ++s_cnt;
                tc_fence_after();
                uint32_t sr[128];
#pragma unroll
                for (int c = 0; c < 4; ++c) tmem_ld32(tS + 32 * c, sr + 32 * c);
                tmem_ld_wait();
#pragma unroll
                for (int c = 0; c < 4; ++c) reg_fence32(sr + 32 * c);
                float* s = reinterpret_cast<float*>(sr);
                if (p.prescale) {
                    const uint64_t sl2x2 = f2(p.sl2, p.sl2);
#pragma unroll
                    for (int c = 0; c < 64; ++c) {
                        const uint64_t v = mul2(f2(s[2 * c], s[2 * c + 1]), sl2x2);
                        f2_split(v, s[2 * c], s[2 * c + 1]);
                    }
                }
                if (fwd_tile_class(T, CAUSAL, tile, j) == kMasked) {
                    const int key0 = j * kBN;
#pragma unroll
                    for (int c = 0; c < 128; ++c)
                        if (!elem_visible(T, CAUSAL, row, key0 + c)) s[c] = -INFINITY;
                }
                // row max: 8 independent chains of 3-input max, then a small tree
                float mx8[8];
#pragma unroll
                for (int c = 0; c < 8; ++c) mx8[c] = fmaxf(s[c], s[c + 8]);
#pragma unroll
                for (int c = 16; c < 128; c += 16)
#pragma unroll
                    for (int a = 0; a < 8; ++a) mx8[a] = fmax3(mx8[a], s[c + a], s[c + 8 + a]);
                const float mx = fmax3(fmax3(mx8[0], mx8[1], mx8[2]), fmax3(mx8[3], mx8[4], mx8[5]),
                                       fmaxf(mx8[6], mx8[7]));
                const float m_tile = mx * eff;
                const float m_new = fmaxf(m_used, m_tile);
                float alpha = 1.f;
                bool need = false;
                if (jj == 0) {
                    m_used = m_new;
                } else if (m_new > m_used + kRescaleThreshold) {
                    need = true;
                    alpha = ex2_approx(m_used - m_new);
                    m_used = m_new;
                    l *= alpha;
                }
                // P = exp2(S * c - m) in two halves of 64 keys: packed FMA for the
                // argument, packed add for the row sum.  The first half, together
                // with the O rescale, is released to the MMA warp before the second
                // half is computed, so the first half of P·V runs beside it.
                const uint64_t eff2 = f2(eff, eff), neg2 = f2(-m_used, -m_used);
                uint64_t lp2[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
                for (int c = 0; c < 32; ++c) {
                    float x0, x1;
                    f2_split(fma2(f2(s[2 * c], s[2 * c + 1]), eff2, neg2), x0, x1);
                    const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
                    lp2[c & 3] = add2(lp2[c & 3], f2(p0, p1));
                    sr[c] = pack_bf16x2(p0, p1);
                }
                tmem_st32(tS, sr);
                // O already holds PV(j-1) (S(j) was committed after it); rescale it
                // before PV(j) starts, only when some row's reference max moved.  The
                // first 64 S registers are free again: two 32-column chunks in flight.
                if (__any_sync(0xffffffffu, need)) {
                    uint32_t* orr = sr;
                    const uint64_t a2 = f2(alpha, alpha);
#pragma unroll
                    for (int c2 = 0; c2 < D / 64; ++c2) {
                        tmem_ld32(tO + 64 * c2, orr);
                        tmem_ld32(tO + 64 * c2 + 32, orr + 32);
                        tmem_ld_wait();
                        reg_fence32(orr);
                        reg_fence32(orr + 32);
#pragma unroll
                        for (int e = 0; e < 64; e += 2) {
                            float o0, o1;
                            f2_split(mul2(f2(__uint_as_float(orr[e]), __uint_as_float(orr[e + 1])), a2), o0, o1);
                            orr[e] = __float_as_uint(o0);
                            orr[e + 1] = __float_as_uint(o1);
                        }
                        tmem_st32(tO + 64 * c2, orr);
                        tmem_st32(tO + 64 * c2 + 32, orr + 32);
                    }
                }
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(ph_full(t));
#pragma unroll
                for (int c = 32; c < 64; ++c) {
                    float x0, x1;
                    f2_split(fma2(f2(s[2 * c], s[2 * c + 1]), eff2, neg2), x0, x1);
                    const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
                    lp2[c & 3] = add2(lp2[c & 3], f2(p0, p1));
                    sr[c] = pack_bf16x2(p0, p1);
                }
                {
                    float a0, a1;
                    f2_split(add2(add2(lp2[0], lp2[1]), add2(lp2[2], lp2[3])), a0, a1);
                    l += a0 + a1;
                }
                tmem_st32(tS + 32, sr + 32);
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(p_full(t));
            }
            // ---- split item: warpgroup 1 hands its row state to warpgroup 0 and waits until its O
            // has been read; warpgroup 0 merges the two halves with the online-softmax rule
            // ("Lab 06", section 2: state from disjoint key ranges combines by rescaling)
            float a0 = 1.f, a1 = 0.f;
            const bool has1 = split && (n_all - h_split) > 0;
            if (split && t == 1) {
                if (n > 0) {
                    if (!warp_wait(o_full(1), o_cnt & 1, ctl)) goto softmax_done;
                    ++o_cnt;
                }
                mrg[r_local] = n > 0 ? m_used : -INFINITY;
                mrg[128 + r_local] = n > 0 ? l : 0.f;
                __syncwarp();
                if (lane == 0) mbar_arrive(mrg_full);
                if (!warp_wait(mrg_done, mrg_cnt & 1, ctl)) goto softmax_done;
                ++mrg_cnt;
                continue;
            }
            if (!warp_wait(o_full(t), o_cnt & 1, ctl)) goto softmax_done;
            ++o_cnt;
            if (split) {
                if (!warp_wait(mrg_full, mrg_cnt & 1, ctl)) goto softmax_done;
                ++mrg_cnt;
                const float m1 = reinterpret_cast<volatile float*>(mrg)[r_local];
                const float l1 = reinterpret_cast<volatile float*>(mrg)[128 + r_local];
                if (has1) {
                    const float mm = fmaxf(m_used, m1);
                    a0 = ex2_approx(m_used - mm);
                    a1 = ex2_approx(m1 - mm);
                    l = l * a0 + l1 * a1;
                    m_used = mm;
                }
            }
            tc_fence_after();
            if constexpr (VARLEN) {
                // packed rows past this sequence's end belong to the next one: store row by row
                const float inv = 1.f / l;
                __nv_bfloat16* dst = p.o_packed + (static_cast<size_t>(item.row0 + row) * p.Hq + bh) * D;
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t orr[32];
                    tmem_ld32(tO + 32 * c, orr);
                    tmem_ld_wait();
                    reg_fence32(orr);
                    if (row < T) {
#pragma unroll
                        for (int q4 = 0; q4 < 4; ++q4) {
                            uint4 w4;
                            w4.x = pack_bf16x2(__uint_as_float(orr[8 * q4 + 0]) * inv, __uint_as_float(orr[8 * q4 + 1]) * inv);
                            w4.y = pack_bf16x2(__uint_as_float(orr[8 * q4 + 2]) * inv, __uint_as_float(orr[8 * q4 + 3]) * inv);
                            w4.z = pack_bf16x2(__uint_as_float(orr[8 * q4 + 4]) * inv, __uint_as_float(orr[8 * q4 + 5]) * inv);
                            w4.w = pack_bf16x2(__uint_as_float(orr[8 * q4 + 6]) * inv, __uint_as_float(orr[8 * q4 + 7]) * inv);
                            reinterpret_cast<uint4*>(dst + 32 * c)[q4] = w4;
                        }
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(epi_bar(t));
                if (wq == 0 && lane == 0) {
                    wait_bar(epi_bar(t), epi_cnt & 1, ctl);
                    mbar_arrive(q_empty(t));  // every S MMA reading this Q tile completed before o_full
                }
                ++epi_cnt;
                if (row < T)
                    p.lse[static_cast<size_t>(bh) * p.total + item.row0 + row] = (m_used + __log2f(l)) * kLn2;
            } else {
                const float inv = 1.f / l;
                const uint32_t tO1 = lane_base + C::kO(1);
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t orr[32];
                    tmem_ld32(tO + 32 * c, orr);
                    if (has1) {
                        uint32_t o1[32];
                        tmem_ld32(tO1 + 32 * c, o1);
                        tmem_ld_wait();
                        reg_fence32(orr);
                        reg_fence32(o1);
#pragma unroll
                        for (int e = 0; e < 32; ++e)
                            orr[e] = __float_as_uint(fmaf(__uint_as_float(orr[e]), a0, __uint_as_float(o1[e]) * a1));
                    } else {
                        tmem_ld_wait();
                        reg_fence32(orr);
                    }
                    const int col0 = 32 * c;
                    const uint32_t atom = sQ[t] + (col0 >> 6) * C::kAtomBytes;
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4) {
                        const uint32_t chunk = ((col0 & 63) >> 3) + q4;
                        uint32_t w4[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            w4[e] = pack_bf16x2(__uint_as_float(orr[8 * q4 + 2 * e]) * inv,
                                                __uint_as_float(orr[8 * q4 + 2 * e + 1]) * inv);
                        st_shared_v4(atom + sw128_off(r_local, chunk), w4[0], w4[1], w4[2], w4[3]);
                    }
                }
                fence_proxy_async_smem();
                tc_fence_before();
                __syncwarp();
                if (split && lane == 0) mbar_arrive(mrg_done);  // warpgroup 1's O has been read
                if (lane == 0) mbar_arrive(epi_bar(t));
                if (wq == 0 && lane == 0) {
                    if (wait_bar(epi_bar(t), epi_cnt & 1, ctl) &&
                        FA_CHECK(tile * kFwdBM < T && bh >= 0 && bh < p.BH, &g_status_fwd, abort_flag)) {
                        for (int a = 0; a < C::kAtoms; ++a)
                            tma_store_3d(&tm_o, sQ[t] + a * C::kAtomBytes, 64 * a, tile * kFwdBM, bh);
                        bulk_commit();
                        bulk_wait_read0();
                    }
                    mbar_arrive(q_empty(t));
                }
                ++epi_cnt;
                if (row < T && FA_CHECK(bh < p.BH, &g_status_fwd, abort_flag))
                    p.lse[static_cast<size_t>(bh) * T + row] = (m_used + __log2f(l)) * kLn2;
            }
        }
    softmax_done:;
        if (wq == 0 && lane == 0) bulk_wait0();
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 9) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

template <int D, bool CAUSAL, bool VARLEN = false, bool SPLIT = false>
int launch_fwd_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& to,
                 const FwdParams& p, int grid, cudaStream_t st) {
    static bool attr_set = false;
    auto kern = fa_fwd_kernel<D, CAUSAL, VARLEN, SPLIT>;
    if (!attr_set) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, FwdCfg<D>::kSmemBytes) !=
            cudaSuccess)
            return -5;
        attr_set = true;
    }
    kern<<<grid, kFwdThreads, FwdCfg<D>::kSmemBytes, st>>>(tq, tk, tv, to, p);
    return cudaGetLastError() == cudaSuccess ? 0 : -5;
}

}  // namespace

int launch_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv, int T,
               int D, float scale, bool causal, cudaStream_t stream, const DebugKnobs& dbg, int num_sms) {
    const int BH = B * Hq, BHkv = B * Hkv;
    CUtensorMap tq, tk, tv, to;
    if (!make_tmap_bhtd(&tq, q, BH, T, D, 128) || !make_tmap_bhtd(&tk, k, BHkv, T, D, 128) ||
        !make_tmap_bhtd(&tv, v, BHkv, T, D, 128) || !make_tmap_bhtd(&to, o, BH, T, D, 128))
        return -5;
    FwdParams p;
    p.lse = lse;
    p.T = T;
    p.BH = BH;
    p.Hq = Hq;
    p.Hkv = Hkv;
    p.group = Hq / Hkv;
    p.n_tiles = cdiv(T, kFwdBM);
    p.n_pairs = cdiv(T, 2 * kFwdBM);
    p.head_pairs = (p.group % 2 == 0) ? 1 : 0;
    p.n_items = p.head_pairs ? p.n_tiles * (BH / 2) : p.n_pairs * BH;
    // Few items: give every query tile an SM of its own.  One tile's step
    // (S, softmax, P V in sequence) is shorter than a pair's ping-pong step, and
    // the SMs that pairs would leave idle do the other halves.
    p.single_tiles = (2LL * p.n_items <= num_sms) ? 1 : 0;
    if (p.single_tiles) p.n_items = p.n_tiles * BH;
    // Without causal masking every item costs the same, so heaviest-first order
    // buys nothing; head-major order keeps the K/V tiles of the few heads in
    // flight in L2 (B=8 H=32 T=3000: 4.9 GB of DRAM reads per launch with the
    // items of all 152 CTAs in different heads, for 0.6 GB of inputs).
    p.head_major = causal ? 0 : 1;
    p.cu_seqlens = nullptr;
    p.n_seq = B;
    p.total = B * T;
    p.o_packed = nullptr;
    p.sl2 = scale * kLog2e;
    p.prescale = (p.sl2 > 0.f) ? 0 : 1;
    p.sl2_eff = p.prescale ? 1.f : p.sl2;
    p.timeout_ns = dbg.timeout_ns;
    p.inject = dbg.inject;
    const int grid = p.n_items < num_sms ? p.n_items : num_sms;
    if (dbg.ev[0]) cudaEventRecord(dbg.ev[0], stream);
    int rc;
    if (p.single_tiles) {
        if (D == 64)
            rc = causal ? launch_fwd_t<64, true, false, true>(tq, tk, tv, to, p, grid, stream)
                        : launch_fwd_t<64, false, false, true>(tq, tk, tv, to, p, grid, stream);
        else
            rc = causal ? launch_fwd_t<128, true, false, true>(tq, tk, tv, to, p, grid, stream)
                        : launch_fwd_t<128, false, false, true>(tq, tk, tv, to, p, grid, stream);
    } else if (D == 64) {
        rc = causal ? launch_fwd_t<64, true>(tq, tk, tv, to, p, grid, stream)
                    : launch_fwd_t<64, false>(tq, tk, tv, to, p, grid, stream);
    } else {
        rc = causal ? launch_fwd_t<128, true>(tq, tk, tv, to, p, grid, stream)
                    : launch_fwd_t<128, false>(tq, tk, tv, to, p, grid, stream);
    }
    if (dbg.ev[1]) cudaEventRecord(dbg.ev[1], stream);
    return rc;
}

int launch_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse, const int* cu_seqlens,
                      int n_seq, int max_seqlen, int total, int H, int D, float scale, bool causal,
                      cudaStream_t stream, const DebugKnobs& dbg, int num_sms) {
    CUtensorMap tq, tk, tv;
    if (!make_tmap_packed(&tq, q, total, H, D, 128) || !make_tmap_packed(&tk, k, total, H, D, 128) ||
        !make_tmap_packed(&tv, v, total, H, D, 128))
        return -5;
    FwdParams p;
    p.lse = lse;
    p.T = max_seqlen;
    p.BH = H;
    p.Hq = p.Hkv = H;
    p.group = 1;
    p.head_pairs = 0;
    p.single_tiles = 0;
    p.head_major = 0;
    p.n_tiles = cdiv(max_seqlen, kFwdBM);
    p.n_pairs = cdiv(max_seqlen, 2 * kFwdBM);
    p.n_items = p.n_pairs * n_seq * H;
    p.cu_seqlens = cu_seqlens;
    p.n_seq = n_seq;
    p.total = total;
    p.o_packed = static_cast<__nv_bfloat16*>(o);
    p.sl2 = scale * kLog2e;
    p.prescale = (p.sl2 > 0.f) ? 0 : 1;
    p.sl2_eff = p.prescale ? 1.f : p.sl2;
    p.timeout_ns = dbg.timeout_ns;
    p.inject = dbg.inject;
    const int grid = p.n_items < num_sms ? p.n_items : num_sms;
    if (D == 64)
        return causal ? launch_fwd_t<64, true, true>(tq, tk, tv, tq, p, grid, stream)
                      : launch_fwd_t<64, false, true>(tq, tk, tv, tq, p, grid, stream);
    return causal ? launch_fwd_t<128, true, true>(tq, tk, tv, tq, p, grid, stream)
                  : launch_fwd_t<128, false, true>(tq, tk, tv, tq, p, grid, stream);
}

int fwd_take_status() {
    int h = 0, z = 0;
    if (cudaMemcpyFromSymbol(&h, g_status_fwd, sizeof(int)) != cudaSuccess) return -5;
    if (cudaMemcpyToSymbol(g_status_fwd, &z, sizeof(int)) != cudaSuccess) return -5;
    return h;
}

}  // namespace fa
