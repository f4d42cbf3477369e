// Workspace layout shared by the calls of libtb.
#pragma once

#include <stddef.h>
#include <stdint.h>

#include "tb.h"

namespace tb {

constexpr int kRadixBits = 11;
constexpr int kRadixBins = 1 << kRadixBits;  // 2048 bins per radix digit
constexpr int kCandCap = 4096;                // largest threshold bin resolved by candidates
constexpr int kMaxChunks = 512;               // CTAs that may share one row
constexpr int kAttnSplitTok = 64;             // fewest selected tokens per attention split
constexpr int kAttnMaxSplits = 128;           // most splits per row
constexpr int kFastEntMax = 1024;             // window entries one CTA of the fast decode step may publish
constexpr int kFastRecBytes = 32 + 8 * kFastEntMax;   // header + (key, token) entries

// Per-row control block of the distributed radix select. Zero between calls.
struct RowCtl {
    uint32_t bar;                    // group-barrier arrivals
    uint32_t done;                   // CTAs finished with this row
    uint32_t ncand;                  // candidates appended
    uint32_t general_steps;          // fast decode steps of this row that needed the general select (statistic)
    uint32_t hist[3][kRadixBins];    // one global histogram per radix pass
    uint32_t above[kMaxChunks];      // per chunk: elements above the threshold bin
    uint32_t eq[kMaxChunks];         // per chunk: elements inside it
    uint2 cand[kCandCap];            // (key, token) of the threshold bin's elements
};

struct WsLayout {
    size_t rowctl_off = 0;   // rows x RowCtl
    size_t attn_ctl_off = 0; // rows x uint32 (split-merge counters)
    size_t part_off = 0;     // rows x max_splits x G x (D + 2) fp32 partials
    size_t scores_off = 0;   // rows x n_max fp32 (decode-step scores; keys of the fast step's re-split)
    size_t rec_off = 0;      // rows x fused chunks x kFastRecBytes (fast decode step records)
    size_t blk_off = 0;      // rows x blk_stride bytes (fast decode step per-block counts)
    int64_t blk_stride = 0;
    size_t total = 0;
    int64_t max_splits = 0;
};

inline size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Tokens per split: at least kAttnSplitTok, more when the row would need
// over kAttnMaxSplits splits.
inline int64_t attn_split_tokens(int64_t sel_stride) {
    int64_t t = (sel_stride + kAttnMaxSplits - 1) / kAttnMaxSplits;
    return t < kAttnSplitTok ? kAttnSplitTok : t;
}

inline int64_t attn_splits(int64_t sel_stride) {
    const int64_t t = attn_split_tokens(sel_stride);
    return (sel_stride + t - 1) / t;
}

inline WsLayout ws_layout(const tb_shape &s, int64_t n_max, int64_t sel_stride_max, int64_t fused_chunks_max) {
    WsLayout L;
    const int64_t rows = (int64_t)s.B * s.Hkv;
    const int64_t G = s.Hkv > 0 ? s.Hq / s.Hkv : 1;
    int64_t splits = attn_splits(sel_stride_max > 0 ? sel_stride_max : 1);
    if (fused_chunks_max > splits) splits = fused_chunks_max;
    L.max_splits = splits;
    size_t off = 0;
    L.rowctl_off = off;
    off = round_up(off + (size_t)rows * sizeof(RowCtl), 256);
    L.attn_ctl_off = off;
    off = round_up(off + (size_t)rows * sizeof(uint32_t), 256);
    L.part_off = off;
    off = round_up(off + (size_t)rows * splits * G * (s.D + 2) * sizeof(float), 256);
    L.scores_off = off;
    off = round_up(off + (size_t)rows * (n_max > 0 ? n_max : 1) * sizeof(float), 256);
    if (fused_chunks_max > 0) {
        L.rec_off = off;
        off = round_up(off + (size_t)rows * fused_chunks_max * kFastRecBytes, 256);
        L.blk_stride = (int64_t)round_up((size_t)((n_max + 31) / 32), 16);
        L.blk_off = off;
        off = round_up(off + (size_t)rows * L.blk_stride, 256);
    }
    L.total = off;
    return L;
}

}  // namespace tb
