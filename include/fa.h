/*
 * fa.h -- C ABI of the GB300 (sm_103a) exact-attention library (libfa.so).
 *
 * What it computes (pages: "Lab 06 - Attention kernels: online softmax ->
 * FlashAttention -> Triton", sections 3 and 4; "Triton FlashAttention-2
 * forward", section "The kernel"; "Flash Attention and Kernel Optimization",
 * sections "Running softmax state", "Causal masking", "Output and saved
 * state"):
 *
 *   forward   S = Q K^T * scale, key j visible to query i iff j <= i when
 *             causal; O = softmax(S) V; LSE_i = log sum_j exp(S_ij)
 *             (natural log of the scaled scores), computed tile by tile
 *             with the online-softmax recurrence, never forming S in memory.
 *   backward  D_i = rowsum(dO o O); P = exp(S - LSE) recomputed per tile;
 *             dV = P^T dO; dP = dO V^T; dS = P o (dP - D);
 *             dQ = dS K * scale; dK = dS^T Q * scale.
 *
 * Layout.  Every tensor is contiguous (B, H, T, D) in bf16
 * (__nv_bfloat16, passed as void*), row stride D elements, head stride T*D.
 * LSE is contiguous (B, H, T) float32.  D must be 64 or 128.  T_q = T_k = T.
 *
 * Memory and ownership.  All tensor pointers are DEVICE pointers on the
 * current CUDA device, allocated and owned by the caller; the library keeps
 * no pointer after a call returns.  Base pointers must be 16-byte aligned
 * (the kernels move tiles with TMA).  Outputs must not overlap inputs.
 *
 * Streams.  `stream` is a cudaStream_t passed as void* (NULL = legacy default
 * stream).  Calls are asynchronous: they enqueue kernels on `stream` and
 * return without synchronising.  fa_bwd takes its workspace (two vectors of
 * B*H*T_pad floats, T_pad = T rounded up to 128: D and log2-scaled LSE, plus
 * 256 bytes for a work counter)
 * stream-ordered with cudaMallocAsync on `stream` and releases it with
 * cudaFreeAsync on the same stream before returning.  Nothing on these paths
 * synchronises, so every compute entry point may be called while `stream` is
 * being captured into a CUDA graph (the workspace becomes allocation nodes,
 * the backward's overlapped second kernel a programmatic dependency); a
 * replay reads the input buffers as they are at replay time.
 * fa_get_device_status synchronises and must not be captured.
 *
 * Errors.  Every entry point validates its arguments before launching
 * anything; on a validation error nothing is enqueued.  Return value 0
 * (FA_OK) or a negative fa_status.  A kernel that detects a stalled pipeline
 * (a bounded wait that ran out) records FA_ERR_DEVICE_TIMEOUT in a device
 * status word and exits cleanly; read it with fa_get_device_status.
 */
#ifndef FA_H_
#define FA_H_

#ifdef __cplusplus
extern "C" {
#endif

typedef enum fa_status {
    FA_OK = 0,
    FA_ERR_NULL = -1,            /* a required pointer is NULL */
    FA_ERR_SHAPE = -2,           /* B, H, T (Tq, Tk) out of range, or a size overflows the index types */
    FA_ERR_UNSUPPORTED = -3,     /* D is not 64 or 128 */
    FA_ERR_ALIGN = -4,           /* a base pointer is not 16-byte aligned */
    FA_ERR_CUDA = -5,            /* a CUDA runtime / driver call failed (launch, attribute, tensor map) */
    FA_ERR_NOMEM = -6,           /* stream-ordered workspace allocation failed */
    FA_ERR_DEVICE_TIMEOUT = -7,  /* a kernel's bounded wait ran out (pipeline stall); outputs invalid */
    FA_ERR_ARG = -8,             /* causal not 0/1, or scale not finite */
    FA_ERR_ARCH = -9,            /* current device is not compute capability 10.3 (sm_103a) */
    FA_ERR_SCRATCH = -10,        /* fa_bwd_noalloc: problem needs more than its fixed scratch buffer */
    FA_ERR_SEQLEN = -11,         /* recorded by a kernel: a cu_seqlens length is negative or above max_seqlen */
    FA_ERR_DEBUG_CHECK = -12     /* debug library only: a kernel's run-time index failed its bounds check */
} fa_status;

/*
 * Forward pass.
 *   q, k, v  in : (B, H, T, D) bf16
 *   o        out: (B, H, T, D) bf16, O = softmax(Q K^T scale [+ causal mask]) V
 *   lse      out: (B, H, T) float32, natural-log log-sum-exp of the scaled,
 *                 masked scores of each row (the only statistic the backward
 *                 needs: "Lab 06", section 4 and "Check yourself" item 3)
 *   scale       : finite float multiplying Q K^T (usually 1/sqrt(D))
 *   causal      : 0 = full attention, 1 = key j visible to query i iff j <= i
 */
int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
           int B, int H, int T, int D, float scale, int causal, void* stream);

/*
 * Backward pass.
 *   q, k, v, o, dO in : (B, H, T, D) bf16 (o from fa_fwd on the same inputs)
 *   lse            in : (B, H, T) float32 from fa_fwd
 *   dq, dk, dv     out: (B, H, T, D) bf16 gradients of sum(dO o O) with
 *                       respect to q, k, v (overwritten, not accumulated)
 *   B, H, T, D, scale, causal: as in fa_fwd.
 * dq is accumulated in float32 across key tiles and rounded to bf16 once:
 *   D = 128: in a second kernel that walks the key tiles of each query tile;
 *     no global-memory reductions, so the result is deterministic.
 *   D = 64, when the dk/dv grid (one CTA per 128-key tile and key/value
 *     head) has at least one CTA per SM: by the same kernel that computes
 *     dk and dv (key tiles outer, as "Lab 06", section 4 orders the loops),
 *     which adds each key tile's contribution into a float32 accumulator in
 *     the workspace with reduce-adds; the order of those additions varies
 *     from run to run, so dq may differ in its last bits between runs (dk
 *     and dv do not).  Smaller grids use the two-kernel form.
 *     fa_set_deterministic(1) selects the two-kernel form at D = 64 always.
 * Workspace: stream-ordered with cudaMallocAsync on `stream`, released before
 * returning: two vectors of B*H*T_pad floats plus 256 bytes (T_pad = T
 * rounded up to 128), and when dq is summed by reduce-adds (above) the
 * float32 dq accumulator, B*H*T_pad*D floats.  FA_ERR_NOMEM if it cannot be
 * had.
 */
int fa_bwd(const void* q, const void* k, const void* v, const void* o, const void* dO,
           const float* lse, void* dq, void* dk, void* dv,
           int B, int H, int T, int D, float scale, int causal, void* stream);

/*
 * Backward pass that allocates nothing.  The pages have no counterpart to
 * this entry point: it exists for callers that cannot allocate device memory
 * at call time, for example code running inside a memory pool that must not
 * grow, or a runtime whose allocator is not reachable from the calling
 * thread.  fa_bwd takes its workspace with cudaMallocAsync; this variant
 * instead uses a fixed scratch buffer compiled into the library
 * (FA_BWD_NOALLOC_SCRATCH_BYTES = 64 MiB of device memory, reserved on every
 * GPU that loads the library's backward module, held until the process
 * exits).  It calls no cudaMalloc, cudaFree or other allocating routine.
 *
 * Same arguments, layout, results and asynchrony as fa_bwd.  The caller
 * still owns every input and output.
 * Limit: 8 * B*H*T_pad + 256 bytes (each of the two vectors rounded up to
 *   256 bytes) must not exceed the scratch size, where T_pad is T rounded up
 *   to a multiple of 128 (B*H*T_pad just under 8 M rows); larger problems
 *   return FA_ERR_SCRATCH and nothing is enqueued.
 * Set-up: the first call on each device looks up the buffer's device
 *   address (cudaGetSymbolAddress) in the context current at that moment and
 *   keeps it for the rest of the process; make that first call before any
 *   stream capture.  The kept address belongs to that context: after
 *   cudaDeviceReset, or from another (non-primary) context on the same
 *   device, it is stale, so do not call fa_bwd_noalloc there.
 * Sharing: every call uses the same buffer, which keeps the previous call's
 *   contents (the backward rewrites all of it before reading it).  Calls whose
 *   work overlaps on the GPU (different streams, or different host threads
 *   without ordering) race on the buffer and corrupt each other's results;
 *   serialise them.
 */
#define FA_BWD_NOALLOC_SCRATCH_BYTES (64ull << 20)
int fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const void* dO,
                   const float* lse, void* dq, void* dk, void* dv,
                   int B, int H, int T, int D, float scale, int causal, void* stream);

/*
 * Grouped-query attention ("Lab 06 - Attention kernels", "Check yourself"
 * item 7): Hq query heads share Hkv key/value heads, Hq % Hkv == 0, query
 * head h using key/value head h / (Hq / Hkv).  Same computation, layout,
 * asynchrony and errors as fa_fwd / fa_bwd with
 *   q, o, dO, dq : (B, Hq, T, D) bf16;  lse : (B, Hq, T) float32
 *   k, v, dk, dv : (B, Hkv, T, D) bf16
 * dk and dv sum the contributions of every query head of the group.  The
 * forward pairs two query heads of one group on the same rows in a CTA, so
 * each K/V tile loaded into shared memory serves both; the backward walks the
 * query tiles of the whole group per key tile.  Hkv == Hq is plain attention.
 * FA_ERR_SHAPE if Hq or Hkv < 1 or Hq % Hkv != 0.
 */
int fa_fwd_gqa(const void* q, const void* k, const void* v, void* o, float* lse,
               int B, int Hq, int Hkv, int T, int D, float scale, int causal, void* stream);
int fa_bwd_gqa(const void* q, const void* k, const void* v, const void* o, const void* dO,
               const float* lse, void* dq, void* dk, void* dv,
               int B, int Hq, int Hkv, int T, int D, float scale, int causal, void* stream);

/*
 * Forward over a packed batch of variable-length sequences ("Triton
 * FlashAttention-2 forward", "Exercises": a cu_seqlens index packs requests of
 * different lengths into one launch).  Sequence s occupies rows
 * cu_seqlens[s] .. cu_seqlens[s+1]-1 of the packed tensors and attends only
 * to itself (causal alignment relative to its own first token).
 *   q, k, v    in : (total, H, D) bf16, packed
 *   o          out: (total, H, D) bf16
 *   lse        out: (H, total) float32
 *   cu_seqlens in : DEVICE int32[n_seq + 1], cu_seqlens[0] = 0, non-decreasing,
 *                   cu_seqlens[n_seq] = total (lengths may be 0)
 *   max_seqlen    : an upper bound on every length (the caller knows it; the
 *                   library does not read cu_seqlens on the host)
 * A length above max_seqlen (or negative) is detected by the kernel and
 * reported as FA_ERR_SEQLEN by fa_get_device_status; those outputs are invalid.
 * Other arguments and errors as in fa_fwd.  No workspace.
 */
int fa_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse,
                  const int* cu_seqlens, int n_seq, int max_seqlen, int total, int H, int D,
                  float scale, int causal, void* stream);

/*
 * Backward of fa_fwd_varlen over the same packed batch ("Triton
 * FlashAttention-2 forward", "Exercises": the cu_seqlens packing; the
 * gradients as in fa_bwd, "Lab 06 - Attention kernels", section 4).  Each
 * sequence's gradients involve only its own rows.
 *   q, k, v, o, dO in : (total, H, D) bf16, packed; o and lse from fa_fwd_varlen
 *   lse            in : (H, total) float32
 *   dq, dk, dv     out: (total, H, D) bf16
 *   cu_seqlens, n_seq, max_seqlen, total: as in fa_fwd_varlen
 * Workspace: like fa_bwd's, stream-ordered with cudaMallocAsync on `stream`:
 * two vectors of H * n_seq * T_pad floats (T_pad = max_seqlen rounded up to
 * 128) plus 256 bytes, released before returning.
 * A length above max_seqlen (or negative) is reported as FA_ERR_SEQLEN by
 * fa_get_device_status; that sequence's gradients are left unwritten.
 * FA_ERR_ARG if an output overlaps an input or another output; other
 * arguments and errors as in fa_fwd_varlen and fa_bwd.
 */
int fa_bwd_varlen(const void* q, const void* k, const void* v, const void* o, const void* dO,
                  const float* lse, void* dq, void* dk, void* dv, const int* cu_seqlens,
                  int n_seq, int max_seqlen, int total, int H, int D, float scale, int causal,
                  void* stream);

/*
 * Decoding forward, split over the keys ("Lab 06 - Attention kernels",
 * "Check yourself" item 2 and "Stretch": a few new query rows against a long
 * key/value cache).  Each of the Tq query rows of a head attends to ALL Tk
 * keys of the same head (no mask).  The keys are split into chunks processed
 * in parallel, each producing a partial (m, l, acc); a second kernel merges
 * them with the online-softmax rescaling rule.
 *   q       in : (B, H, Tq, D) bf16, 1 <= Tq <= 8
 *   k, v    in : (B, H, Tk, D) bf16, Tk >= 1
 *   o       out: (B, H, Tq, D) bf16
 *   lse     out: (B, H, Tq) float32, natural-log log-sum-exp of the scaled scores
 *   scale, stream: as in fa_fwd.  D must be 64 or 128.
 * Workspace: the partials (B*H*n_chunks*Tq*(D + 2) floats) are taken with
 * cudaMallocAsync on `stream` and released before returning.
 */
int fa_decode(const void* q, const void* k, const void* v, void* o, float* lse,
              int B, int H, int Tq, int Tk, int D, float scale, void* stream);

/* Static, NUL-terminated description of a status code (never NULL). */
const char* fa_strerror(int status);

/*
 * Synchronises `stream`, returns the device status word recorded by the
 * library's kernels on the current device since the last call (FA_OK,
 * FA_ERR_DEVICE_TIMEOUT or FA_ERR_SEQLEN), and clears it.  Returns FA_ERR_CUDA if the
 * synchronisation itself fails.
 */
int fa_get_device_status(void* stream);

/* Library ABI version (major * 100 + minor). */
int fa_version(void);

/*
 * Host-only schedule queries (no GPU needed).  They evaluate the exact index
 * logic the kernels use, so tests can compare it with a brute-force mask.
 *
 * fa_sched_fwd_tile_class / fa_sched_bwd_tile_class: class of the tile pair
 *   (query tile qt, key tile kt) as the forward / backward kernel sees it:
 *   0 = skipped (never loaded), 1 = full (no element mask), 2 = masked
 *   element by element.  The backward's query tile height depends on D.
 * fa_sched_fwd_keep / fa_sched_bwd_keep: 1 iff the kernel's composition of
 *   tile loop bounds, tile class and element mask keeps score (i, j).
 *   i and j may range over the padded extent (multiples of the tile sizes).
 * fa_sched_tile_rows: query tile height (fwd) or key tile height (bwd keys)
 *   and backward query tile height for head size D: writes bm_fwd, bn, bm_bwd.
 * Return negative fa_status on bad arguments.
 */
int fa_sched_fwd_tile_class(int T, int causal, int qt, int kt);
int fa_sched_bwd_tile_class(int T, int D, int causal, int qt, int kt);
int fa_sched_fwd_keep(int T, int causal, int i, int j);
int fa_sched_bwd_keep(int T, int D, int causal, int i, int j);
int fa_sched_tile_rows(int D, int* bm_fwd, int* bn, int* bm_bwd);

/*
 * Test hooks (host state, read at the next launch; default off).
 * fa_debug_set_wait_timeout_ns: bound of every in-kernel wait (default 2 s).
 * fa_debug_inject: 0 = off; 1 = the forward's load warp skips its first
 *   K/V tile copy; 2 = the load warp of the backward's first dK/dV CTA skips
 *   its third Q tile copy (its first when it has fewer); 3 = the load warp of
 *   the backward's first dQ CTA skips its first K tile copy.  The waits that depend on the missing copy
 *   run out, the CTA gives up (it waits, bounded, for its copies and MMAs in
 *   flight, frees its tensor memory and exits) and FA_ERR_DEVICE_TIMEOUT is
 *   reported instead of a hang; the outputs of that call are not valid.
 *   Used to test failure detection without faulting the GPU.  Other values
 *   return FA_ERR_ARG.
 */
int fa_debug_set_wait_timeout_ns(unsigned long long ns);
int fa_debug_inject(int mode);

/*
 * Backward determinism (host state, read by each fa_bwd / fa_bwd_gqa call;
 * default 0).  1: the backward never sums into global memory, so dq, dk and
 * dv are bitwise reproducible at every D (the two-kernel form; slower at
 * D = 64).  0: at D = 64 the backward computes dq in its dk/dv kernel and
 * sums the key tiles' contributions with float32 reduce-adds (see fa_bwd).
 * Returns FA_ERR_ARG unless on is 0 or 1.  fa_bwd_varlen and fa_bwd_noalloc
 * are always deterministic.
 */
int fa_set_deterministic(int on);

/*
 * Host query (no launch): 1 if fa_bwd / fa_bwd_gqa on this shape, on the
 * current device and in the current determinism mode, computes dq inside its
 * dk/dv kernel and sums it with reduce-adds (then its second kernel is the
 * conversion of the float32 accumulator to bf16 dq), 0 if it runs the
 * two-kernel form.  FA_ERR_SHAPE / FA_ERR_UNSUPPORTED for bad sizes,
 * FA_ERR_ARCH or FA_ERR_CUDA without a suitable current device.
 */
int fa_bwd_sums_dq_in_place(int B, int Hkv, int T, int D);

/*
 * 1 in the debug build of the library (compiled with FA_DEBUG), 0 in the
 * product build.  In the debug build every kernel checks the tile
 * coordinates, ring stages, per-row vector offsets and tensor-memory columns
 * it computes at run time before it uses them; a failed check skips the
 * access, makes the CTA give up through its bounded-wait exit path, and is
 * reported by fa_get_device_status as FA_ERR_DEBUG_CHECK.  Nothing traps.
 */
int fa_debug_checks_enabled(void);

/*
 * Measurement hook (default off; host state read by each call).  When the
 * pointers are non-NULL, later calls record these CUDA events (cudaEvent_t
 * passed as void*, created and owned by the caller) on the call's stream:
 * fwd_begin / fwd_end immediately around the forward kernel; bwd_begin
 * before the backward's dK/dV kernel, bwd_mid between it and the dQ kernel,
 * bwd_end after the dQ kernel (the preprocess is outside).  Pass NULLs to
 * turn it off.  Used to time the dominant kernels inside a timed region
 * without a profiler.
 */
int fa_set_timing_events(void* fwd_begin, void* fwd_end, void* bwd_begin, void* bwd_mid, void* bwd_end);

#ifdef __cplusplus
}
#endif

#endif /* FA_H_ */
