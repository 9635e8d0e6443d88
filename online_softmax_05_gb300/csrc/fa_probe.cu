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

}  // namespace
}  // namespace fa

extern "C" {

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
