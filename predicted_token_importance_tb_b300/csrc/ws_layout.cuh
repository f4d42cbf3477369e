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

// The three-kernel decode step (pipe_step.cu): per-row control and result
// block. Zero between calls (the row's last CTAs put back what they used);
// hist is the row's 12-bit histogram of score keys.
constexpr int kPipeHBits = 12;
constexpr int kPipeHBins = 1 << kPipeHBits;
constexpr int kPipeMaxChunks = 64;            // CTAs that may share one row in the pipeline
constexpr int kPipeCandCap = 4096;            // threshold-bin entries per row resolved in shared memory
struct PipeRow {
    uint32_t done2;                  // bracket CTAs finished with this row
    uint32_t done3;                  // attention CTAs finished with this row
    uint32_t ncand;                  // threshold-bin entries appended to the row's candidate list
    uint32_t overflow;               // more of them than the list holds (the resolver then rescans the keys)
    uint32_t b1;                     // result: the k-th token's 12-bit bin
    uint32_t cut_key;                // result: key of the k-th ranked token among [0, n)
    int32_t cut_idx;                 // result: its index
    int32_t k1;                      // result: tokens kept among [0, n)
    uint32_t cab[kPipeMaxChunks];    // per chunk: tokens above the threshold bin
    int32_t offs[kPipeMaxChunks + 4];// result: output offset of each chunk's kept tokens (offs[C] = k1)
    uint32_t hist[kPipeHBins];       // 12-bit histogram of the row's score keys
};

// Test hook of the single-launch step, at a fixed offset after the row
// control blocks; zero in normal use (tb_workspace_init clears it). A
// non-zero wait_limit_ns replaces the limit of the kernel's bounded waits;
// skip_arrive_cta = c + 1 makes chunk c of row 0 leave out its arrival at the
// row's exchange, so that row's waits run out and report TB_ERR_TIMEOUT (a
// barrier that nothing completes, without any fault).
struct WsDebug {
    uint64_t wait_limit_ns;
    int32_t skip_arrive_cta;
    int32_t pad[61];
};

struct WsLayout {
    size_t rowctl_off = 0;   // rows x RowCtl
    size_t debug_off = 0;    // one WsDebug
    size_t attn_ctl_off = 0; // rows x uint32 (split-merge counters)
    size_t part_off = 0;     // rows x max_splits x G x (D + 2) fp32 partials
    size_t scores_off = 0;   // rows x n_max fp32 (decode-step scores; keys of the fast step's re-split)
    size_t rec_off = 0;      // rows x fused chunks x kFastRecBytes (fast decode step records)
    size_t blk_off = 0;      // rows x blk_stride bytes (fast decode step per-block counts)
    int64_t blk_stride = 0;
    size_t pipe_off = 0;     // rows x PipeRow (three-kernel step)
    size_t pipe_keys_off = 0;// rows x pipe_keys_stride uint32 score keys
    int64_t pipe_keys_stride = 0;
    size_t pipe_part_off = 0;// rows x kPipeMaxChunks x G x (D + 2) fp32 partials
    size_t pipe_cand_off = 0;// rows x kPipeCandCap (key, token) threshold-bin entries
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

// Partial slots per row: ceil(sel_stride / kAttnSplitTok), at most kAttnMaxSplits. It never decreases with
// sel_stride (a workspace sized for a larger stride holds every smaller call's partials) and covers the
// splits of attn_split_tokens.
inline int64_t attn_splits(int64_t sel_stride) {
    const int64_t s = (sel_stride + kAttnSplitTok - 1) / kAttnSplitTok;
    return s < kAttnMaxSplits ? s : kAttnMaxSplits;
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
    L.debug_off = off;
    off = round_up(off + sizeof(WsDebug), 256);
    L.attn_ctl_off = off;
    off = round_up(off + (size_t)rows * sizeof(uint32_t), 256);
    // the three-kernel step's control blocks sit at an offset that depends on the shape only, so a later
    // call with another token count finds the zeroed counters the previous call left
    L.pipe_off = off;
    off = round_up(off + (size_t)rows * sizeof(PipeRow), 256);
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
    // the three-kernel step's score keys and partials
    L.pipe_keys_stride = (int64_t)round_up((size_t)(n_max > 0 ? n_max : 1), 4);
    L.pipe_keys_off = off;
    off = round_up(off + (size_t)rows * L.pipe_keys_stride * sizeof(uint32_t), 256);
    L.pipe_part_off = off;
    off = round_up(off + (size_t)rows * kPipeMaxChunks * G * (s.D + 2) * sizeof(float), 256);
    L.pipe_cand_off = off;
    off = round_up(off + (size_t)rows * kPipeCandCap * 8, 256);
    L.total = off;
    return L;
}

}  // namespace tb
