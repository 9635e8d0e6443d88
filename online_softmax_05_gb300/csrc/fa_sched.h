// fa_sched.h -- tile schedule and mask logic shared by the kernels and the
// host-side schedule queries (plain C++; compiled for host and device).
//
// "Lab 06 - Attention kernels", section 3: under causal masking a query tile
// needs the key tiles up to the one holding its last row (skip the rest),
// key tiles wholly at or below the diagonal need no mask ("full"), the tile
// crossing the diagonal is masked element by element ("diag").  "Common
// bugs": the last key tile needed is the one containing row i1 - 1; keys past
// T are masked.  Rows past T (padding of the last query tile) are never
// stored; in the backward they are masked so they contribute nothing.
#pragma once

#if defined(__CUDACC__)
#define FA_HD __host__ __device__ __forceinline__
#else
#define FA_HD inline
#endif

namespace fa {

constexpr int kFwdBM = 128;  // forward query tile rows (one TMEM lane per row)
constexpr int kBN = 128;     // key tile rows, forward and backward

// Backward query tile rows: 128 at both head sizes.  The transposed-operand
// MMAs of the backward cost a fixed ~118 cycles per instruction up to N = 128,
// so 128-row query tiles halve their count per unit of work.
FA_HD constexpr int bwd_bm(int /*D*/) { return 128; }

FA_HD int cdiv(int a, int b) { return (a + b - 1) / b; }
FA_HD int imin(int a, int b) { return a < b ? a : b; }

enum TileClass : int { kSkip = 0, kFull = 1, kMasked = 2 };

// Score (i, j) is visible iff key j exists and, under causal masking, j <= i.
FA_HD bool elem_visible(int T, bool causal, int i, int j) { return j < T && (!causal || j <= i); }

// Class of the (rows [r0, r0+nr), keys [c0, c0+nc)) tile over its rows < T.
// `mask_pad_rows` also masks rows >= T (backward: padded queries must add 0).
FA_HD int tile_class(int T, bool causal, int r0, int nr, int c0, int nc, bool mask_pad_rows) {
    int last_row = imin(r0 + nr, T) - 1;  // last real row of the tile
    if (last_row < r0) return kSkip;      // no real rows at all
    if (c0 >= T) return kSkip;
    if (causal && c0 > last_row) return kSkip;
    bool full = (c0 + nc <= T) && (!causal || c0 + nc - 1 <= r0) && (!mask_pad_rows || r0 + nr <= T);
    return full ? kFull : kMasked;
}

// ---- forward: query tile qt (rows qt*kFwdBM ...), key tiles 0 .. n-1
FA_HD int fwd_num_kv_tiles(int T, bool causal, int qt) {
    if (!causal) return cdiv(T, kBN);
    int last_row = imin((qt + 1) * kFwdBM, T) - 1;
    return last_row / kBN + 1;
}
FA_HD int fwd_tile_class(int T, bool causal, int qt, int kt) {
    if (qt * kFwdBM >= T || kt >= fwd_num_kv_tiles(T, causal, qt)) return kSkip;
    return tile_class(T, causal, qt * kFwdBM, kFwdBM, kt * kBN, kBN, false);
}
// Forward kernel's composition: loop bound, then tile class, then element mask.
FA_HD bool fwd_keep(int T, bool causal, int i, int j) {
    int qt = i / kFwdBM, kt = j / kBN;
    int c = fwd_tile_class(T, causal, qt, kt);
    if (c == kSkip) return false;
    if (c == kFull) return true;
    return elem_visible(T, causal, i, j);
}

// ---- backward: key tile kt, query tiles q_begin .. q_end-1 of height bm
FA_HD int bwd_q_begin(int T, bool causal, int kt, int bm) { return causal ? (kt * kBN) / bm : 0; }
FA_HD int bwd_q_end(int T, int bm) { return cdiv(T, bm); }
FA_HD int bwd_tile_class(int T, bool causal, int bm, int qt, int kt) {
    if (kt * kBN >= T || qt < bwd_q_begin(T, causal, kt, bm) || qt >= bwd_q_end(T, bm)) return kSkip;
    return tile_class(T, causal, qt * bm, bm, kt * kBN, kBN, true);
}
FA_HD bool bwd_elem_visible(int T, bool causal, int i, int j) { return i < T && elem_visible(T, causal, i, j); }
FA_HD bool bwd_keep(int T, bool causal, int bm, int i, int j) {
    int qt = i / bm, kt = j / kBN;
    int c = bwd_tile_class(T, causal, bm, qt, kt);
    if (c == kSkip) return false;
    if (c == kFull) return true;
    return bwd_elem_visible(T, causal, i, j);
}

}  // namespace fa
