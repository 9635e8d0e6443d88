// fa_api.cu -- the C ABI of libfa.so (declared in include/fa.h): argument
// validation, device checks and dispatch to the kernel launchers.  Every
// argument check runs before the first CUDA call, so a rejected call enqueues
// nothing and needs no GPU.
#include <cuda_runtime.h>

#include <atomic>
#include <climits>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "fa.h"
#include "fa_internal.h"
#include "fa_sched.h"

namespace {

std::atomic<unsigned long long> g_timeout_ns{2000000000ull};
std::atomic<int> g_inject{0};
std::atomic<int> g_deterministic{0};
std::atomic<void*> g_events[5] = {nullptr, nullptr, nullptr, nullptr, nullptr};

constexpr int kMaxDevices = 64;
std::once_flag g_dev_once[kMaxDevices];
int g_dev_sms[kMaxDevices];
int g_dev_arch_ok[kMaxDevices];

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_shape(int B, int H, int T, int D, float scale, int causal) {
    if (B < 1 || H < 1 || T < 1) return FA_ERR_SHAPE;
    const long long rows = static_cast<long long>(B) * H * T;
    if (rows > INT_MAX || static_cast<long long>(B) * H > (1 << 30)) return FA_ERR_SHAPE;
    if (D != 64 && D != 128) return FA_ERR_UNSUPPORTED;
    if (causal != 0 && causal != 1) return FA_ERR_ARG;
    if (!std::isfinite(scale)) return FA_ERR_ARG;
    return FA_OK;
}

struct Range {
    uintptr_t lo, hi;
};
Range range_of(const void* p, size_t bytes) {
    uintptr_t a = reinterpret_cast<uintptr_t>(p);
    return {a, a + bytes};
}
bool overlap(Range a, Range b) { return a.lo < b.hi && b.lo < a.hi; }

// Resolve the current device, its SM count and whether it is sm_103.
int current_device(int* dev_out, int* sms_out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return FA_ERR_CUDA;
    std::call_once(g_dev_once[dev], [dev] {
        int major = 0, minor = 0, sms = 0;
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        g_dev_sms[dev] = sms;
        g_dev_arch_ok[dev] = (major == 10 && minor == 3) ? 1 : 0;
    });
    if (!g_dev_arch_ok[dev]) return FA_ERR_ARCH;
    *dev_out = dev;
    *sms_out = g_dev_sms[dev] > 0 ? g_dev_sms[dev] : 1;
    return FA_OK;
}

fa::DebugKnobs knobs() {
    fa::DebugKnobs k{g_timeout_ns.load(), g_inject.load(), {}, g_deterministic.load()};
    for (int i = 0; i < 5; ++i) k.ev[i] = static_cast<cudaEvent_t>(g_events[i].load());
    return k;
}

}  // namespace

extern "C" {

int fa_version(void) { return 100; }

const char* fa_strerror(int status) {
    switch (status) {
        case FA_OK: return "ok";
        case FA_ERR_NULL: return "a required pointer is NULL";
        case FA_ERR_SHAPE: return "B, H and T (Tq, Tk) must be >= 1 and B*H*T must fit in a 32-bit index";
        case FA_ERR_UNSUPPORTED: return "head dimension D must be 64 or 128 (and fa_decode takes at most 8 query rows)";
        case FA_ERR_ALIGN: return "tensor base pointers must be 16-byte aligned";
        case FA_ERR_CUDA: return "a CUDA runtime or driver call failed";
        case FA_ERR_NOMEM: return "stream-ordered workspace allocation failed";
        case FA_ERR_DEVICE_TIMEOUT: return "a kernel's bounded wait ran out (pipeline stall); outputs are invalid";
        case FA_ERR_ARG: return "causal must be 0 or 1, scale finite, and outputs must not overlap other buffers";
        case FA_ERR_ARCH: return "the current device is not compute capability 10.3 (sm_103a)";
        case FA_ERR_SEQLEN: return "a cu_seqlens length is negative or above max_seqlen (recorded by the kernel)";
        case FA_ERR_SCRATCH: return "fa_bwd_noalloc: the problem needs more than the fixed 64 MiB scratch buffer";
        case FA_ERR_DEBUG_CHECK: return "debug library: a kernel's run-time index failed its bounds check (access skipped)";
        default: return "unknown fa_status";
    }
}

}  // extern "C"

namespace {

// Shared checks and dispatch of the forward; Hq query heads over Hkv K/V heads.
int fwd_impl(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv, int T, int D,
             float scale, int causal, void* stream) {
    if (!q || !k || !v || !o || !lse) return FA_ERR_NULL;
    if (Hkv < 1 || Hq < 1 || Hq % Hkv != 0) return FA_ERR_SHAPE;
    int rc = check_shape(B, Hq, T, D, scale, causal);
    if (rc != FA_OK) return rc;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse)) return FA_ERR_ALIGN;
    const size_t nq = static_cast<size_t>(B) * Hq * T * D * 2, nk = static_cast<size_t>(B) * Hkv * T * D * 2;
    const size_t nl = static_cast<size_t>(B) * Hq * T * 4;
    const Range rq = range_of(q, nq), rk = range_of(k, nk), rv = range_of(v, nk), ro = range_of(o, nq),
                rl = range_of(lse, nl);
    if (overlap(ro, rq) || overlap(ro, rk) || overlap(ro, rv) || overlap(ro, rl) || overlap(rl, rq) ||
        overlap(rl, rk) || overlap(rl, rv))
        return FA_ERR_ARG;
    int dev = 0, sms = 0;
    rc = current_device(&dev, &sms);
    if (rc != FA_OK) return rc;
    return fa::launch_fwd(q, k, v, o, lse, B, Hq, Hkv, T, D, scale, causal != 0, static_cast<cudaStream_t>(stream),
                          knobs(), sms);
}

// Shared checks and dispatch of the backward.
int bwd_impl(const void* q, const void* k, const void* v, const void* o, const void* dO, const float* lse, void* dq,
             void* dk, void* dv, int B, int Hq, int Hkv, int T, int D, float scale, int causal, void* stream) {
    if (!q || !k || !v || !o || !dO || !lse || !dq || !dk || !dv) return FA_ERR_NULL;
    if (Hkv < 1 || Hq < 1 || Hq % Hkv != 0) return FA_ERR_SHAPE;
    int rc = check_shape(B, Hq, T, D, scale, causal);
    if (rc != FA_OK) return rc;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(dO) || !aligned16(lse) ||
        !aligned16(dq) || !aligned16(dk) || !aligned16(dv))
        return FA_ERR_ALIGN;
    const size_t nq = static_cast<size_t>(B) * Hq * T * D * 2, nk = static_cast<size_t>(B) * Hkv * T * D * 2;
    const size_t nl = static_cast<size_t>(B) * Hq * T * 4;
    const Range ins[6] = {range_of(q, nq), range_of(k, nk), range_of(v, nk), range_of(o, nq), range_of(dO, nq),
                          range_of(lse, nl)};
    const Range outs[3] = {range_of(dq, nq), range_of(dk, nk), range_of(dv, nk)};
    for (int a = 0; a < 3; ++a) {
        for (int b = 0; b < 6; ++b)
            if (overlap(outs[a], ins[b])) return FA_ERR_ARG;
        for (int b = a + 1; b < 3; ++b)
            if (overlap(outs[a], outs[b])) return FA_ERR_ARG;
    }
    int dev = 0, sms = 0;
    rc = current_device(&dev, &sms);
    if (rc != FA_OK) return rc;
    return fa::launch_bwd(q, k, v, o, dO, lse, dq, dk, dv, B, Hq, Hkv, T, D, scale, causal != 0,
                          static_cast<cudaStream_t>(stream), knobs(), sms);
}

}  // namespace

extern "C" {

int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int T, int D, float scale,
           int causal, void* stream) {
    return fwd_impl(q, k, v, o, lse, B, H, H, T, D, scale, causal, stream);
}

int fa_bwd(const void* q, const void* k, const void* v, const void* o, const void* dO, const float* lse, void* dq,
           void* dk, void* dv, int B, int H, int T, int D, float scale, int causal, void* stream) {
    return bwd_impl(q, k, v, o, dO, lse, dq, dk, dv, B, H, H, T, D, scale, causal, stream);
}

int fa_fwd_gqa(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv, int T,
               int D, float scale, int causal, void* stream) {
    return fwd_impl(q, k, v, o, lse, B, Hq, Hkv, T, D, scale, causal, stream);
}

int fa_bwd_gqa(const void* q, const void* k, const void* v, const void* o, const void* dO, const float* lse, void* dq,
               void* dk, void* dv, int B, int Hq, int Hkv, int T, int D, float scale, int causal, void* stream) {
    return bwd_impl(q, k, v, o, dO, lse, dq, dk, dv, B, Hq, Hkv, T, D, scale, causal, stream);
}

int fa_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse, const int* cu_seqlens, int n_seq,
                  int max_seqlen, int total, int H, int D, float scale, int causal, void* stream) {
    if (!q || !k || !v || !o || !lse || !cu_seqlens) return FA_ERR_NULL;
    if (n_seq < 1 || max_seqlen < 1 || total < 1 || H < 1) return FA_ERR_SHAPE;
    if (static_cast<long long>(total) * H > INT_MAX || static_cast<long long>(n_seq) * H > (1 << 30))
        return FA_ERR_SHAPE;
    if (D != 64 && D != 128) return FA_ERR_UNSUPPORTED;
    if (causal != 0 && causal != 1) return FA_ERR_ARG;
    if (!std::isfinite(scale)) return FA_ERR_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse) ||
        (reinterpret_cast<uintptr_t>(cu_seqlens) & 3u))
        return FA_ERR_ALIGN;
    const size_t n = static_cast<size_t>(total) * H * D * 2, nl = static_cast<size_t>(total) * H * 4;
    const Range rq = range_of(q, n), rk = range_of(k, n), rv = range_of(v, n), ro = range_of(o, n),
                rl = range_of(lse, nl), rc_ = range_of(cu_seqlens, static_cast<size_t>(n_seq + 1) * 4);
    if (overlap(ro, rq) || overlap(ro, rk) || overlap(ro, rv) || overlap(ro, rl) || overlap(rl, rq) ||
        overlap(rl, rk) || overlap(rl, rv) || overlap(ro, rc_) || overlap(rl, rc_))
        return FA_ERR_ARG;
    int dev = 0, sms = 0;
    int rc = current_device(&dev, &sms);
    if (rc != FA_OK) return rc;
    return fa::launch_fwd_varlen(q, k, v, o, lse, cu_seqlens, n_seq, max_seqlen, total, H, D, scale, causal != 0,
                                 static_cast<cudaStream_t>(stream), knobs(), sms);
}

int fa_bwd_varlen(const void* q, const void* k, const void* v, const void* o, const void* dO, const float* lse,
                  void* dq, void* dk, void* dv, const int* cu_seqlens, int n_seq, int max_seqlen, int total, int H,
                  int D, float scale, int causal, void* stream) {
    if (!q || !k || !v || !o || !dO || !lse || !dq || !dk || !dv || !cu_seqlens) return FA_ERR_NULL;
    if (n_seq < 1 || max_seqlen < 1 || total < 1 || H < 1) return FA_ERR_SHAPE;
    if (static_cast<long long>(total) * H > INT_MAX || static_cast<long long>(n_seq) * H > (1 << 30) ||
        static_cast<long long>(n_seq) * H * ((max_seqlen + 127) / 128) > INT_MAX)
        return FA_ERR_SHAPE;
    if (D != 64 && D != 128) return FA_ERR_UNSUPPORTED;
    if (causal != 0 && causal != 1) return FA_ERR_ARG;
    if (!std::isfinite(scale)) return FA_ERR_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(dO) || !aligned16(lse) ||
        !aligned16(dq) || !aligned16(dk) || !aligned16(dv) || (reinterpret_cast<uintptr_t>(cu_seqlens) & 3u))
        return FA_ERR_ALIGN;
    const size_t n = static_cast<size_t>(total) * H * D * 2, nl = static_cast<size_t>(total) * H * 4;
    const Range ins[7] = {range_of(q, n),   range_of(k, n),   range_of(v, n),
                          range_of(o, n),   range_of(dO, n),  range_of(lse, nl),
                          range_of(cu_seqlens, static_cast<size_t>(n_seq + 1) * 4)};
    const Range outs[3] = {range_of(dq, n), range_of(dk, n), range_of(dv, n)};
    for (int a = 0; a < 3; ++a) {
        for (int b = 0; b < 7; ++b)
            if (overlap(outs[a], ins[b])) return FA_ERR_ARG;
        for (int b = a + 1; b < 3; ++b)
            if (overlap(outs[a], outs[b])) return FA_ERR_ARG;
    }
    int dev = 0, sms = 0;
    int rc = current_device(&dev, &sms);
    if (rc != FA_OK) return rc;
    return fa::launch_bwd_varlen(q, k, v, o, dO, lse, dq, dk, dv, cu_seqlens, n_seq, max_seqlen, total, H, D, scale,
                                 causal != 0, static_cast<cudaStream_t>(stream), knobs(), sms);
}

int fa_decode(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Tq, int Tk, int D,
              float scale, void* stream) {
    if (!q || !k || !v || !o || !lse) return FA_ERR_NULL;
    if (B < 1 || H < 1 || Tq < 1 || Tk < 1) return FA_ERR_SHAPE;
    if (static_cast<long long>(B) * H > (1 << 30) || static_cast<long long>(B) * H * Tk > INT_MAX) return FA_ERR_SHAPE;
    if (Tq > 8) return FA_ERR_UNSUPPORTED;
    if (D != 64 && D != 128) return FA_ERR_UNSUPPORTED;
    if (!std::isfinite(scale)) return FA_ERR_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse)) return FA_ERR_ALIGN;
    const size_t nq = static_cast<size_t>(B) * H * Tq * D * 2, nk = static_cast<size_t>(B) * H * Tk * D * 2;
    const size_t nl = static_cast<size_t>(B) * H * Tq * 4;
    const Range rq = range_of(q, nq), rk = range_of(k, nk), rv = range_of(v, nk), ro = range_of(o, nq),
                rl = range_of(lse, nl);
    if (overlap(ro, rq) || overlap(ro, rk) || overlap(ro, rv) || overlap(ro, rl) || overlap(rl, rq) ||
        overlap(rl, rk) || overlap(rl, rv))
        return FA_ERR_ARG;
    int dev = 0, sms = 0;
    int rc = current_device(&dev, &sms);
    if (rc != FA_OK) return rc;
    return fa::launch_decode(q, k, v, o, lse, B, H, Tq, Tk, D, scale, static_cast<cudaStream_t>(stream), sms);
}

// Same checks as fa_bwd, then the fixed-scratch backward (see include/fa.h:
// for callers that cannot allocate device memory at call time).
int fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const void* dO, const float* lse,
                   void* dq, void* dk, void* dv, int B, int H, int T, int D, float scale, int causal, void* stream) {
    if (!q || !k || !v || !o || !dO || !lse || !dq || !dk || !dv) return FA_ERR_NULL;
    int rc = check_shape(B, H, T, D, scale, causal);
    if (rc != FA_OK) return rc;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(dO) || !aligned16(lse) ||
        !aligned16(dq) || !aligned16(dk) || !aligned16(dv))
        return FA_ERR_ALIGN;
    const size_t n = static_cast<size_t>(B) * H * T * D * 2, nl = static_cast<size_t>(B) * H * T * 4;
    const Range ins[6] = {range_of(q, n), range_of(k, n), range_of(v, n), range_of(o, n), range_of(dO, n),
                          range_of(lse, nl)};
    const Range outs[3] = {range_of(dq, n), range_of(dk, n), range_of(dv, n)};
    for (int a = 0; a < 3; ++a) {
        for (int b = 0; b < 6; ++b)
            if (overlap(outs[a], ins[b])) return FA_ERR_ARG;
        for (int b = a + 1; b < 3; ++b)
            if (overlap(outs[a], outs[b])) return FA_ERR_ARG;
    }
    if (fa::bwd_scratch_bytes(B, H, T, D) > FA_BWD_NOALLOC_SCRATCH_BYTES) return FA_ERR_SCRATCH;
    int dev = 0, sms = 0;
    rc = current_device(&dev, &sms);
    if (rc != FA_OK) return rc;
    return fa::launch_bwd_noalloc(q, k, v, o, dO, lse, dq, dk, dv, B, H, T, D, scale, causal != 0,
                                  static_cast<cudaStream_t>(stream), knobs(), sms);
}

int fa_get_device_status(void* stream) {
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return FA_ERR_CUDA;
    int a = fa::fwd_take_status();
    int b = fa::bwd_take_status();
    if (a == -5 || b == -5) return FA_ERR_CUDA;
    return a != 0 ? a : b;
}

int fa_sched_tile_rows(int D, int* bm_fwd, int* bn, int* bm_bwd) {
    if (!bm_fwd || !bn || !bm_bwd) return FA_ERR_NULL;
    if (D != 64 && D != 128) return FA_ERR_UNSUPPORTED;
    *bm_fwd = fa::kFwdBM;
    *bn = fa::kBN;
    *bm_bwd = fa::bwd_bm(D);
    return FA_OK;
}

int fa_sched_fwd_tile_class(int T, int causal, int qt, int kt) {
    if (T < 1 || qt < 0 || kt < 0) return FA_ERR_SHAPE;
    return fa::fwd_tile_class(T, causal != 0, qt, kt);
}

int fa_sched_bwd_tile_class(int T, int D, int causal, int qt, int kt) {
    if (T < 1 || qt < 0 || kt < 0) return FA_ERR_SHAPE;
    if (D != 64 && D != 128) return FA_ERR_UNSUPPORTED;
    return fa::bwd_tile_class(T, causal != 0, fa::bwd_bm(D), qt, kt);
}

int fa_sched_fwd_keep(int T, int causal, int i, int j) {
    if (T < 1 || i < 0 || j < 0) return FA_ERR_SHAPE;
    return fa::fwd_keep(T, causal != 0, i, j) ? 1 : 0;
}

int fa_sched_bwd_keep(int T, int D, int causal, int i, int j) {
    if (T < 1 || i < 0 || j < 0) return FA_ERR_SHAPE;
    if (D != 64 && D != 128) return FA_ERR_UNSUPPORTED;
    return fa::bwd_keep(T, causal != 0, fa::bwd_bm(D), i, j) ? 1 : 0;
}

int fa_debug_set_wait_timeout_ns(unsigned long long ns) {
    if (ns == 0) return FA_ERR_ARG;
    g_timeout_ns.store(ns);
    return FA_OK;
}

int fa_set_timing_events(void* fwd_begin, void* fwd_end, void* bwd_begin, void* bwd_mid, void* bwd_end) {
    g_events[0].store(fwd_begin);
    g_events[1].store(fwd_end);
    g_events[2].store(bwd_begin);
    g_events[3].store(bwd_mid);
    g_events[4].store(bwd_end);
    return FA_OK;
}

int fa_bwd_sums_dq_in_place(int B, int Hkv, int T, int D) {
    if (B < 1 || Hkv < 1 || T < 1) return FA_ERR_SHAPE;
    if (D != 64 && D != 128) return FA_ERR_UNSUPPORTED;
    int dev = 0, sms = 0;
    const int rc = current_device(&dev, &sms);
    if (rc != FA_OK) return rc;
    return fa::bwd_fuses_host(B, Hkv, T, D, sms, g_deterministic.load() != 0) ? 1 : 0;
}

int fa_set_deterministic(int on) {
    if (on != 0 && on != 1) return FA_ERR_ARG;
    g_deterministic.store(on);
    return FA_OK;
}

int fa_debug_checks_enabled(void) {
#ifdef FA_DEBUG
    return 1;
#else
    return 0;
#endif
}

int fa_debug_inject(int mode) {
    if (mode < 0 || mode > 3) return FA_ERR_ARG;
    g_inject.store(mode);
    return FA_OK;
}

}  // extern "C"
