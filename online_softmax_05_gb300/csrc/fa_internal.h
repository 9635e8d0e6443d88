// fa_internal.h -- declarations shared by the library's translation units.
#pragma once

#include <cuda_runtime.h>

namespace fa {

struct DebugKnobs {
    unsigned long long timeout_ns;  // bound of every in-kernel wait
    int inject;                     // fault-injection mode (0 = off)
    cudaEvent_t ev[5];              // measurement hook: fwd begin/end; bwd: before dK/dV, between, after dQ (may be null)
    int deterministic;              // 1: the backward never sums into global memory (two-kernel form at every D)
};

// Status word values written by kernels (mirror of fa_status).
constexpr int kStatusTimeout = -7;
constexpr int kStatusBadSeqlen = -11;
constexpr int kStatusSmemAlign = -4;  // a kernel's dynamic shared-memory window was not 1024-byte aligned
constexpr int kStatusDebugCheck = -12;  // debug build: a run-time index failed its bounds check

// Launchers: arguments already validated by the C-ABI layer.
// Hq query heads share Hkv key/value heads (Hq % Hkv == 0; Hkv == Hq is plain attention).
int launch_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv, int T,
               int D, float scale, bool causal, cudaStream_t stream, const DebugKnobs& dbg, int num_sms);
int launch_bwd(const void* q, const void* k, const void* v, const void* o, const void* dO, const float* lse,
               void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int T, int D, float scale, bool causal,
               cudaStream_t stream, const DebugKnobs& dbg, int num_sms);

// Forward over a packed variable-length batch: (total, H, D) tensors, LSE (H, total).
int launch_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse, const int* cu_seqlens,
                      int n_seq, int max_seqlen, int total, int H, int D, float scale, bool causal,
                      cudaStream_t stream, const DebugKnobs& dbg, int num_sms);

// Backward over a packed variable-length batch (the same layout; dq, dk, dv (total, H, D)).
int launch_bwd_varlen(const void* q, const void* k, const void* v, const void* o, const void* dO, const float* lse,
                      void* dq, void* dk, void* dv, const int* cu_seqlens, int n_seq, int max_seqlen, int total,
                      int H, int D, float scale, bool causal, cudaStream_t stream, const DebugKnobs& dbg,
                      int num_sms);

// Split-K decoding forward (fa_decode.cu).
int launch_decode(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Tq, int Tk,
                  int D, float scale, cudaStream_t stream, int num_sms);

// Backward with the library's fixed device scratch buffer instead of an
// allocation; returns -10 if the problem does not fit, without launching.
size_t bwd_scratch_bytes(int B, int H, int T, int D);
// Whether fa_bwd sums dQ inside the dK/dV kernel for this shape on a GPU with num_sms SMs.
bool bwd_fuses_host(int B, int Hkv, int T, int D, int num_sms, bool deterministic);
int launch_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const void* dO, const float* lse,
                       void* dq, void* dk, void* dv, int B, int H, int T, int D, float scale, bool causal,
                       cudaStream_t stream, const DebugKnobs& dbg, int num_sms);

// Read and clear the device status word of each translation unit on the
// current device (caller synchronises first).  Return 0 or a negative code.
int fwd_take_status();
int bwd_take_status();

}  // namespace fa
