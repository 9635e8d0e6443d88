// fa_probe.cu -- test-only bring-up kernels (built into libfa_probe.so, not
// part of libfa.so).  They check, one at a time, the encodings the attention
// kernels rely on: the 128-byte swizzle TMA writes, the shared-memory and
// instruction descriptors of tcgen05.mma for K-major and MN-major operands,
// an A operand read from tensor memory, and tcgen05.ld of the accumulator.
// Every wait is bounded; a run that times out returns an error code.
#include <cuda_runtime.h>

#include "fa_ptx.cuh"
#include "fa_tmap.h"

namespace fa {
namespace {

constexpr uint64_t kProbeTimeoutNs = 2000000000ull;

__device__ bool probe_wait(uint32_t bar, uint32_t parity, int* err) {
    if (mbar_try_wait(bar, parity)) return true;
    uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer_ns() - t0 > kProbeTimeoutNs) {
            atomicExch(err, 1);
            return false;
        }
    }
    return true;
}

// Byte address of element (r, c) of a tile stored with 128-byte swizzle in
// 64-element-wide column blocks; block b starts at b * rows * 128.
__device__ __forceinline__ uint32_t sw_elem(uint32_t base, int rows, int r, int c) {
    int blk = c >> 6, cc = c & 63;
    return base + blk * rows * 128 + sw128_off(r, cc >> 3) + (cc & 7) * 2;
}

// a_mode: 0 = A in smem K-major ([M][K] in global), 1 = A in smem MN-major
//         ([K][M] in global), 2 = A in TMEM (from [M][K] in global).
// b_mode: 0 = B in smem K-major ([N][K] in global), 1 = B in smem MN-major
//         ([K][N] in global).
// out[m][n] = sum_k A(m,k) B(k,n), fp32, M = 128.
__global__ void __launch_bounds__(128, 1)
    probe_mma_kernel(int a_mode, int b_mode, int N, int K, const __nv_bfloat16* A, const __nv_bfloat16* B,
                     float* out, int* err) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int M = 128;
    uint32_t sA = smem_u32(smem);
    uint32_t sB = sA + M * K * 2;
    uint32_t bar = sB + N * K * 2;
    uint32_t tslot = bar + 8;
    int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    if (warp == 0) {
        tmem_alloc(tslot, 512);
        tmem_relinquish();
    }
    if (tid == 0) {
        mbar_init(bar, 1);
        fence_mbar_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + (tslot - sA));

    // stage A
    if (a_mode == 0) {
        for (int e = tid; e < M * K; e += 128) {
            int m = e / K, k = e % K;
            uint32_t a = sw_elem(sA, M, m, k);
            __nv_bfloat16 x = A[m * K + k];
            asm volatile("st.shared.b16 [%0], %1;" ::"r"(a), "h"(*reinterpret_cast<uint16_t*>(&x)));
        }
    } else if (a_mode == 1) {
        for (int e = tid; e < M * K; e += 128) {
            int k = e / M, m = e % M;
            uint32_t a = sw_elem(sA, K, k, m);
            __nv_bfloat16 x = A[k * M + m];
            asm volatile("st.shared.b16 [%0], %1;" ::"r"(a), "h"(*reinterpret_cast<uint16_t*>(&x)));
        }
    } else {
        // thread = row m; columns 256.. hold A packed two bf16 per 32-bit column
        int m = tid;
        for (int c0 = 0; c0 < K / 2; c0 += 16) {
            uint32_t r[16];
            for (int c = 0; c < 16; ++c) {
                __nv_bfloat162 h;
                h.x = A[m * K + 2 * (c0 + c)];
                h.y = A[m * K + 2 * (c0 + c) + 1];
                r[c] = *reinterpret_cast<uint32_t*>(&h);
            }
            tmem_st16(tmem + ((32u * warp) << 16) + 256u + c0, r);
        }
        tmem_st_wait();
    }
    // stage B
    if (b_mode == 0) {
        for (int e = tid; e < N * K; e += 128) {
            int n = e / K, k = e % K;
            uint32_t a = sw_elem(sB, N, n, k);
            __nv_bfloat16 x = B[n * K + k];
            asm volatile("st.shared.b16 [%0], %1;" ::"r"(a), "h"(*reinterpret_cast<uint16_t*>(&x)));
        }
    } else {
        for (int e = tid; e < N * K; e += 128) {
            int k = e / N, n = e % N;
            uint32_t a = sw_elem(sB, K, k, n);
            __nv_bfloat16 x = B[k * N + n];
            asm volatile("st.shared.b16 [%0], %1;" ::"r"(a), "h"(*reinterpret_cast<uint16_t*>(&x)));
        }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    if (tid == 0) {
        uint32_t idesc = idesc_bf16_f32(M, N, a_mode == 1, b_mode == 1);
        for (int s = 0; s < K / 16; ++s) {
            uint64_t bdesc = (b_mode == 0) ? sdesc_sw128(sB + (s >> 2) * N * 128 + (s & 3) * 32, 16, 1024)
                                           : sdesc_sw128(sB + s * 2048, K * 128, 1024);
            if (a_mode == 2) {
                mma_ts(tmem, tmem + 256u + s * 8, bdesc, idesc, s > 0);
            } else {
                uint64_t adesc = (a_mode == 0) ? sdesc_sw128(sA + (s >> 2) * M * 128 + (s & 3) * 32, 16, 1024)
                                               : sdesc_sw128(sA + s * 2048, K * 128, 1024);
                mma_ss(tmem, adesc, bdesc, idesc, s > 0);
            }
        }
        mma_commit(bar);
    }
    __syncwarp();
    bool ok = probe_wait(bar, 0, err);
    tc_fence_after();
    if (ok) {
        int m = 32 * warp + lane;
        for (int c0 = 0; c0 < N; c0 += 32) {
            uint32_t r[32];
            tmem_ld32(tmem + ((32u * warp) << 16) + c0, r);
            tmem_ld_wait();
            reg_fence32(r);
            for (int c = 0; c < 32; ++c) out[m * N + c0 + c] = __uint_as_float(r[c]);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 512);
}

// TMA 128-byte-swizzle load of one (box_rows x D) tile of a (BH, T, D) bf16
// tensor at (row0, bh); the raw shared-memory bytes are copied to `dst`.
__global__ void __launch_bounds__(128, 1)
    probe_tma_kernel(const __grid_constant__ CUtensorMap map, int D, int box_rows, int row0, int bh, uint8_t* dst,
                     int* err) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint32_t s = smem_u32(smem);
    int bytes = box_rows * D * 2;
    uint32_t bar = s + bytes;
    if (threadIdx.x == 0) {
        mbar_init(bar, 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        mbar_arrive_expect_tx(bar, bytes);
        for (int a = 0; a < D / 64; ++a) tma_load_3d(s + a * box_rows * 128, &map, bar, 64 * a, row0, bh);
    }
    bool ok = probe_wait(bar, 0, err);
    if (ok)
        for (int i = threadIdx.x; i < bytes; i += blockDim.x) dst[i] = smem[i];
}

// Issues n_chains chains of CHAIN back-to-back MMAs (unrolled: the issuing
// thread must spend far less than an MMA per instruction).
template <int CHAIN>
__device__ __forceinline__ void chain_issue(int kind, int n_chains, uint32_t tmem, uint64_t da, uint64_t db, bool bmn,
                                            uint32_t idesc) {
    const uint64_t bstep = bmn ? 128u : 2u;
    for (int c = 0; c < n_chains; ++c) {
        const uint32_t acc = tmem + ((c & 1) ? 128u : 0u);
        if (kind == 2) {
#pragma unroll
            for (int s = 0; s < CHAIN; ++s) mma_ts(acc, tmem + 384u + (s & 3) * 8, db + (s & 3) * bstep, idesc, s > 0);
        } else {
#pragma unroll
            for (int s = 0; s < CHAIN; ++s) mma_ss(acc, da + (s & 3) * 2, db + (s & 3) * bstep, idesc, s > 0);
        }
    }
}

// Cost of tcgen05.mma chains: n instructions of 128 x N x 16 split into
// chains of `chain` instructions, each chain accumulating into one of two
// TMEM accumulators (they alternate chain by chain).  kind 0: A and B
// K-major in smem; 1: A K-major, B MN-major; 2: A from TMEM, B MN-major.
// Cycles from the first issue to the completion of the last are written to out[0].
__global__ void __launch_bounds__(128, 1) probe_mma_chain_kernel(int N, int n, int chain, int kind, long long* out,
                                                                 int* err) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sA = smem_u32(smem);
    const uint32_t sB = sA + 128 * 64 * 2;           // 16 KB of A (K-major, 4 k-steps per 128-byte row)
    const uint32_t bar = sB + 2 * 128 * 128;         // 32 KB of B (two 64-wide atoms of 128 rows)
    const uint32_t tslot = bar + 8;
    const int tid = threadIdx.x, warp = tid >> 5;
    for (int i = tid; i < (128 * 64 * 2 + 2 * 128 * 128) / 4; i += 128) reinterpret_cast<uint32_t*>(smem)[i] = 0x3f803f80u;
    if (warp == 0) {
        tmem_alloc(tslot, 512);
        tmem_relinquish();
    }
    if (tid == 0) {
        mbar_init(bar, 1);
        fence_mbar_init();
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + (tslot - sA));
    if (tid == 0) {
        const bool bmn = kind != 0;
        const uint32_t idesc = idesc_bf16_f32(128, N, false, bmn);
        const uint64_t da = sdesc_sw128(sA, 16, 1024);
        const uint64_t db = bmn ? sdesc_sw128(sB, 128 * 128, 1024) : sdesc_sw128(sB, 16, 1024);
        const long long t0 = clock64();
        switch (chain) {
            case 1: chain_issue<1>(kind, n / 1, tmem, da, db, bmn, idesc); break;
            case 2: chain_issue<2>(kind, n / 2, tmem, da, db, bmn, idesc); break;
            case 4: chain_issue<4>(kind, n / 4, tmem, da, db, bmn, idesc); break;
            case 8: chain_issue<8>(kind, n / 8, tmem, da, db, bmn, idesc); break;
            case 16: chain_issue<16>(kind, n / 16, tmem, da, db, bmn, idesc); break;
            default: chain_issue<32>(kind, n / 32, tmem, da, db, bmn, idesc); break;
        }
        mma_commit(bar);
        probe_wait(bar, 0, err);
        out[0] = clock64() - t0;
    }
    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 512);
}

// Sequences of 8-instruction chains shaped like the attention kernels' loops
// (128 x 128 x 16 bf16 MMAs; n_iter iterations of three chains each):
//   mode 0  SS, SS, SS chains into three accumulators (columns 0, 128, 256)
//   mode 1  mode 0 plus a tcgen05.commit to an mbarrier after every chain
//   mode 2  mode 1 plus, before every chain, a try_wait on an mbarrier phase
//           that has already completed and a tcgen05 fence (what the kernels
//           do when an operand is already there)
//   mode 3  the dQ kernel's loop: SS (dP, columns 256), TS with A from
//           columns 32.. of the S buffer (dQ, columns 384), SS (S, columns
//           0 / 128 alternating), commits and waits as in mode 2
// mode | 4: the same with the operands in shared memory filled with
// pseudo-random bf16 values instead of 1.0.
// SYNC (modes 2 and 3): 0 = wait, then fence; 1 = the wait alone; 2 = the
// fence alone; 3 = the wait issued before the last two MMAs of the previous
// chain, the fence after that chain.
// WIDE: the whole warp runs the loop and elect.sync picks the issuing lane
// (else lane 0 runs it alone).  RTOFF: the smem descriptors get an offset
// known only at run time (always 0), like the kernels' ring stages.
// Cycles from the first issue to the completion of the last MMA go to out[0].
template <int SYNC, bool WIDE, bool RTOFF>
__global__ void __launch_bounds__(128, 1) probe_mma_seq_kernel(int mode, int n_iter, long long* out, int* err) {
    out += blockIdx.x;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sA = smem_u32(smem);
    const uint32_t sB = sA + 128 * 128 * 2;          // A: 128 rows x 128 K (two 64-wide atoms), 32 KB
    const uint32_t bar = sB + 128 * 128 * 2;         // B: 128 rows x 128 (two atoms), 32 KB
    const uint32_t bar2 = bar + 8, bar3 = bar + 16;
    const uint32_t tslot = bar + 24;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const bool noisy = (mode & 4) != 0;
    const int bg = (mode >> 3) & 3;  // 1: warps 1-3 stream TMEM loads; 2: shared-memory loads
    mode &= 3;
    volatile int* done = reinterpret_cast<volatile int*>(smem + (tslot - sA) + 8);
    for (int i = tid; i < (2 * 128 * 128 * 2) / 4; i += 128) {
        uint32_t w = 0x3f803f80u;  // 1.0 in both halves
        if (noisy) {
            // two bf16 of random sign, exponent 2^-8 .. 2^-1 and mantissa
            // (an integer hash of the index: the values only have to toggle)
            uint32_t h = uint32_t(i) * 0x9E3779B1u;
            h ^= h >> 15;
            h *= 0x85EBCA77u;
            h ^= h >> 13;
            w = (h & 0x807f807fu) | 0x3c003c00u | ((h >> 3) & 0x03800380u);
        }
        reinterpret_cast<uint32_t*>(smem)[i] = w;
    }
    if (warp == 0) {
        tmem_alloc(tslot, 512);
        tmem_relinquish();
    }
    if (tid == 0) {
        mbar_init(bar, 1);
        mbar_init(bar2, 1);
        mbar_init(bar3, 1);
        *done = 0;
        fence_mbar_init();
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + (tslot - sA));
    if (tid == 0) mbar_arrive(bar3);  // a phase that has completed: waits on it return at once
    __syncwarp();
    if (warp != 0 && bg != 0) {
        // background traffic until warp 0 is done (at most 2^20 rounds)
        uint32_t acc = 0;
        for (int it = 0; it < (1 << 20) && !*done; ++it) {
            if (bg == 1) {
                uint32_t r[32];
                tmem_ld32(tmem + ((32u * warp) << 16) + 256u, r);
                tmem_ld_wait();
                reg_fence32(r);
                acc ^= r[it & 31];
            } else {
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const uint32_t off = ((static_cast<uint32_t>(it) * 8u + u) * 512u + lane * 16u) & (65536u - 1u);
                    uint32_t a, b, c, d;
                    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                                 : "=r"(a), "=r"(b), "=r"(c), "=r"(d)
                                 : "r"(sA + off));
                    acc ^= a ^ b ^ c ^ d;
                }
            }
        }
        if (acc == 0x12345678u) *done = 2;  // keeps the loads
    }
    if (warp == 0 && (WIDE || lane == 0)) {
        const bool leader = WIDE ? elect_one_sync() : true;
        const uint32_t id_kk = idesc_bf16_f32(128, 128, false, false);
        const uint32_t id_mn = idesc_bf16_f32(128, 128, false, true);
        const SDesc dA = sdesc_make(sA, 16, 1024), dB = sdesc_make(sB, 16, 1024);
        const SDesc dBmn = sdesc_make(sB, 128 * 128, 1024);
        bool early_ok = true;
        auto chain_ss = [&](uint32_t acc, uint32_t so) {
#pragma unroll
            for (int s = 0; s < 8; ++s) {
                const uint32_t off = ((s >> 2) * (128 * 128) + (s & 3) * 32) >> 4;
                if (leader) mma_ss_d(acc, dA, off, dB, off + so, id_kk, s > 0);
                if constexpr (SYNC == 3)
                    if (s == 5 && mode >= 2) early_ok = mbar_try_wait(bar3, 0);
            }
        };
        auto chain_ts = [&](uint32_t acc, uint32_t a_col, uint32_t so) {
#pragma unroll
            for (int s = 0; s < 8; ++s) {
                if (leader) mma_ts_d(acc, a_col + s * 8, dBmn, s * (2048 >> 4) + so, id_mn, 1u);
                if constexpr (SYNC == 3)
                    if (s == 5) early_ok = mbar_try_wait(bar3, 0);
            }
        };
        auto between = [&]() {
            if (mode >= 1 && leader) mma_commit(bar2);
            if (mode >= 2) {
                if constexpr (SYNC == 0 || SYNC == 1)
                    if (!mbar_try_wait(bar3, 0)) atomicExch(err, 3);
                if constexpr (SYNC == 3)
                    if (!early_ok) atomicExch(err, 3);
                if constexpr (SYNC != 1) tc_fence_after();
            }
        };
        const long long t0 = clock64();
        for (int it = 0; it < n_iter; ++it) {
            const uint32_t so = RTOFF ? (static_cast<uint32_t>(it) >> 20) << 10 : 0u;
            if (mode <= 2) {
                chain_ss(tmem + 0, so);
                between();
                chain_ss(tmem + 128, so);
                between();
                chain_ss(tmem + 256, so);
                between();
            } else {
                chain_ss(tmem + 256, so);
                between();
                chain_ts(tmem + 384, tmem + (it & 1) * 128 + 32, so);
                between();
                chain_ss(tmem + (it & 1) * 128, so);
                between();
            }
        }
        if (leader) mma_commit(bar);
        probe_wait(bar, 0, err);
        if (lane == 0) out[0] = clock64() - t0;
        *done = 1;
    }
    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 512);
}

template <int SYNC, bool WIDE, bool RTOFF>
void launch_seq(int mode, int n_iter, long long* out, int* err, int ctas, int smem) {
    cudaFuncSetAttribute(probe_mma_seq_kernel<SYNC, WIDE, RTOFF>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    probe_mma_seq_kernel<SYNC, WIDE, RTOFF><<<ctas, 128, smem>>>(mode, n_iter, out, err);
}

// Lane/column layout of tcgen05.ld.16x256b.x8 and tcgen05.st.16x128b.x8.
// Every TMEM cell (lane l, column c) of columns 0..63 is first written with
// (l << 16) | c through 32x32b stores; each warp then loads its lanes
// 32w .. 32w+15 and 32w+16 .. 32w+31 with the 16x256b shape and records the
// 2 x 32 registers of each thread in ld_out[w][t][64].  Then each thread
// stores 16 registers (w << 24) | (t << 16) | j with the 16x128b shape at
// lanes 32w .. 32w+15, columns 128 .. 159, and the cells are read back with
// 32x32b loads into st_out[lane][32].
__global__ void __launch_bounds__(128, 1) probe_tmem_layout_kernel(uint32_t* ld_out, uint32_t* st_out) {
    __shared__ uint32_t tslot;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (warp == 0) {
        tmem_alloc(smem_u32(&tslot), 256);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tslot;
    const uint32_t lane_base = tmem + ((32u * warp) << 16);
    const uint32_t l = 32u * warp + lane;
    uint32_t v[32];
    for (int half = 0; half < 2; ++half) {
        for (int c = 0; c < 32; ++c) v[c] = (l << 16) | (32u * half + c);
        tmem_st32(lane_base + 32 * half, v);
    }
    tmem_st_wait();
    for (int half = 0; half < 2; ++half) {
        uint32_t r[32];
        tmem_ld_16x256b_x8(lane_base + ((16u * half) << 16), r);
        tmem_ld_wait();
        reg_fence32(r);
        for (int j = 0; j < 32; ++j) ld_out[(warp * 32 + lane) * 64 + 32 * half + j] = r[j];
    }
    uint32_t w16[16];
    for (int j = 0; j < 16; ++j) w16[j] = (uint32_t(warp) << 24) | (uint32_t(lane) << 16) | uint32_t(j);
    for (int c = 0; c < 32; ++c) v[c] = 0xffffffffu;
    tmem_st32(lane_base + 128, v);
    tmem_st_wait();
    tmem_st_16x128b_x8(lane_base + 128, w16);
    tmem_st_wait();
    {
        uint32_t r[32];
        tmem_ld32(lane_base + 128, r);
        tmem_ld_wait();
        reg_fence32(r);
        for (int c = 0; c < 32; ++c) st_out[l * 32 + c] = r[c];
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 256);
}

// Throughput of the softmax's special-function work, 8 independent chains
// per thread; cycles for `iters` rounds are written to out[warp]:
//   mode 0  8 ex2.approx (MUFU) per round
//   mode 1  8 exp2 as a polynomial on the FMA/ALU pipes (round-to-nearest by
//           the 1.5*2^23 add, degree-3 least-squares fit of 2^f on
//           [-1/2, 1/2], integer add into the exponent)
//   mode 2  4 cvt.rn.bf16x2.f32 packs per round (each pair unpacked again
//           by a mask, a shift and two adds, so the chains continue)
//   mode 3  modes 0 and 2 interleaved: 8 ex2 and 4 packs per round, the
//           softmax's mix (every P pair is exponentiated, then packed)
__device__ __forceinline__ float exp2_poly3(float x) {
    x = fmaxf(x, -126.f);
    const float t = x + 12582912.f;  // 1.5 * 2^23: rounds x to an integer in the low mantissa bits
    const float r = t - 12582912.f;
    const float f = x - r;             // in [-0.5, 0.5]
    float p = fmaf(fmaf(fmaf(0.0555041f, f, 0.2402265f), f, 0.6931472f), f, 1.0f);
    return __int_as_float(__float_as_int(p) + (__float_as_int(t) << 23));
}
__global__ void probe_exp2_rate_kernel(int mode, int iters, float* sink, long long* out) {
    float v[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) v[c] = -0.001f * (threadIdx.x + c);
    __syncthreads();
    long long t0 = clock64();
    for (int i = 0; i < iters; ++i) {
        if (mode <= 1) {
#pragma unroll
            for (int c = 0; c < 8; ++c) v[c] = (mode == 0 ? ex2_approx(v[c]) : exp2_poly3(v[c])) - 1.0f;
        } else {
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const float a = mode == 3 ? ex2_approx(v[2 * c]) : v[2 * c];
                const float b = mode == 3 ? ex2_approx(v[2 * c + 1]) : v[2 * c + 1];
                const uint32_t w = pack_bf16x2(a, b);
                v[2 * c] = __uint_as_float(w & 0xffff0000u) - 1.0f;
                v[2 * c + 1] = __uint_as_float(w << 16) - 1.0f;
            }
        }
    }
    long long t1 = clock64();
    float acc = 0.f;
#pragma unroll
    for (int c = 0; c < 8; ++c) acc += v[c];
    sink[threadIdx.x] = acc;
    if ((threadIdx.x & 31) == 0) out[threadIdx.x >> 5] = t1 - t0;
}

}  // namespace
}  // namespace fa

extern "C" {

int probe_exp2_rate(int mode, int iters, int warps, long long* out_host, float* max_rel_err) {
    float* sink = nullptr;
    long long* out = nullptr;
    if (warps < 1 || warps > 32 || mode < 0 || mode > 3 || iters < 1 || iters > (1 << 20)) return -1;
    cudaMalloc(&sink, 1024 * sizeof(float));
    cudaMalloc(&out, 32 * sizeof(long long));
    fa::probe_exp2_rate_kernel<<<1, 32 * warps>>>(mode, iters, sink, out);
    cudaError_t e = cudaDeviceSynchronize();
    cudaMemcpy(out_host, out, warps * sizeof(long long), cudaMemcpyDeviceToHost);
    cudaFree(sink);
    cudaFree(out);
    (void)max_rel_err;
    return e == cudaSuccess ? 0 : -5;
}


int probe_mma_chain(int N, int n, int chain, int kind, long long* out_host) {
    if (!(N == 64 || N == 128) || n < 1 || n > 4096 || !(chain == 1 || chain == 2 || chain == 4 || chain == 8 ||
                                                        chain == 16 || chain == 32) ||
        n % chain || kind < 0 || kind > 2)
        return -1;
    int* err = nullptr;
    long long* out = nullptr;
    if (cudaMalloc(&err, sizeof(int)) != cudaSuccess) return -5;
    if (cudaMalloc(&out, sizeof(long long)) != cudaSuccess) return -5;
    cudaMemset(err, 0, sizeof(int));
    const int smem = 1024 + 128 * 64 * 2 + 2 * 128 * 128 + 64;
    cudaFuncSetAttribute(fa::probe_mma_chain_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    fa::probe_mma_chain_kernel<<<1, 128, smem>>>(N, n, chain, kind, out, err);
    cudaError_t e = cudaDeviceSynchronize();
    int h = 0;
    cudaMemcpy(&h, err, sizeof(int), cudaMemcpyDeviceToHost);
    cudaMemcpy(out_host, out, sizeof(long long), cudaMemcpyDeviceToHost);
    cudaFree(err);
    cudaFree(out);
    if (e != cudaSuccess) return -5;
    return h ? -7 : 0;
}


// ctas: number of CTAs (one per SM at this shared-memory size) running the
// same sequence at once; out_host receives one count per CTA.
// mode bits: 0-1 loop, 2 random operands, 3-4 SYNC, 5 WIDE, 6 RTOFF, 7-8 background traffic
// (1 TMEM loads, 2 shared-memory loads by warps 1-3; see probe_mma_seq_kernel)
int probe_mma_seq(int mode, int n_iter, int ctas, long long* out_host) {
    if (mode < 0 || mode > 511 || ((mode >> 7) & 3) == 3 || n_iter < 1 || n_iter > 4096 || ctas < 1 || ctas > 1024) return -1;
    int* err = nullptr;
    long long* out = nullptr;
    if (cudaMalloc(&err, sizeof(int)) != cudaSuccess) return -5;
    if (cudaMalloc(&out, ctas * sizeof(long long)) != cudaSuccess) return -5;
    cudaMemset(err, 0, sizeof(int));
    // more than half of the SM's shared memory: at most one CTA per SM
    const int smem = 120 * 1024;
    using Seq = void (*)(int, int, long long*, int*, int, int);
    static const Seq kSeq[16] = {
        fa::launch_seq<0, false, false>, fa::launch_seq<0, false, true>, fa::launch_seq<0, true, false>,
        fa::launch_seq<0, true, true>,   fa::launch_seq<1, false, false>, fa::launch_seq<1, false, true>,
        fa::launch_seq<1, true, false>,  fa::launch_seq<1, true, true>,   fa::launch_seq<2, false, false>,
        fa::launch_seq<2, false, true>,  fa::launch_seq<2, true, false>,  fa::launch_seq<2, true, true>,
        fa::launch_seq<3, false, false>, fa::launch_seq<3, false, true>,  fa::launch_seq<3, true, false>,
        fa::launch_seq<3, true, true>};
    kSeq[((mode >> 3) & 3) * 4 + ((mode >> 5) & 1) * 2 + ((mode >> 6) & 1)]((mode & 7) | (((mode >> 7) & 3) << 3), n_iter, out, err, ctas, smem);
    cudaError_t e = cudaDeviceSynchronize();
    int h = 0;
    cudaMemcpy(&h, err, sizeof(int), cudaMemcpyDeviceToHost);
    cudaMemcpy(out_host, out, ctas * sizeof(long long), cudaMemcpyDeviceToHost);
    cudaFree(err);
    cudaFree(out);
    if (e != cudaSuccess) return -5;
    return h ? -7 : 0;
}

int probe_tmem_layout(uint32_t* ld_host, uint32_t* st_host) {
    uint32_t *ld = nullptr, *st = nullptr;
    if (cudaMalloc(&ld, 128 * 64 * 4) != cudaSuccess) return -5;
    if (cudaMalloc(&st, 128 * 32 * 4) != cudaSuccess) return -5;
    fa::probe_tmem_layout_kernel<<<1, 128>>>(ld, st);
    cudaError_t e = cudaDeviceSynchronize();
    cudaMemcpy(ld_host, ld, 128 * 64 * 4, cudaMemcpyDeviceToHost);
    cudaMemcpy(st_host, st, 128 * 32 * 4, cudaMemcpyDeviceToHost);
    cudaFree(ld);
    cudaFree(st);
    return e == cudaSuccess ? 0 : -5;
}

int probe_mma(int a_mode, int b_mode, int N, int K, const void* A, const void* B, float* out) {
    if (a_mode < 0 || a_mode > 2 || b_mode < 0 || b_mode > 1) return -1;
    if (!(N == 64 || N == 128) || !(K == 64 || K == 128)) return -1;
    int* err = nullptr;
    if (cudaMalloc(&err, sizeof(int)) != cudaSuccess) return -5;
    cudaMemset(err, 0, sizeof(int));
    int smem = 1024 + 128 * K * 2 + N * K * 2 + 64;
    cudaFuncSetAttribute(fa::probe_mma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    fa::probe_mma_kernel<<<1, 128, smem>>>(a_mode, b_mode, N, K, static_cast<const __nv_bfloat16*>(A),
                                           static_cast<const __nv_bfloat16*>(B), out, err);
    cudaError_t e = cudaDeviceSynchronize();
    int h = 0;
    cudaMemcpy(&h, err, sizeof(int), cudaMemcpyDeviceToHost);
    cudaFree(err);
    if (e != cudaSuccess) return -5;
    return h ? -7 : 0;
}

int probe_tma(const void* src, int BH, int T, int D, int box_rows, int row0, int bh, void* dst) {
    CUtensorMap map;
    if (!fa::make_tmap_bhtd(&map, src, BH, T, D, box_rows)) return -5;
    int* err = nullptr;
    if (cudaMalloc(&err, sizeof(int)) != cudaSuccess) return -5;
    cudaMemset(err, 0, sizeof(int));
    int smem = 1024 + box_rows * D * 2 + 64;
    cudaFuncSetAttribute(fa::probe_tma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    fa::probe_tma_kernel<<<1, 128, smem>>>(map, D, box_rows, row0, bh, static_cast<uint8_t*>(dst), err);
    cudaError_t e = cudaDeviceSynchronize();
    int h = 0;
    cudaMemcpy(&h, err, sizeof(int), cudaMemcpyDeviceToHost);
    cudaFree(err);
    if (e != cudaSuccess) return -5;
    return h ? -7 : 0;
}

}  // extern "C"
