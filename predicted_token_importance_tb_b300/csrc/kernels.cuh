// Launchers of the libtb kernels (host side, internal).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "tb.h"
#include "ws_layout.cuh"

namespace tb {

// n_seq (device, [B], may be null): sequence b holds n_seq[b] + 1 tokens; the
// scores of its later positions are -inf. after_append: the append kernel was
// launched just before on the same stream and triggers its dependents at its
// start; the score kernel runs as its programmatic dependent (only the CTA
// that reads the appended row, the row's or sequence's last, waits for it).
cudaError_t launch_score(const tb_shape &sh, const uint16_t *q_imp, const uint16_t *Kp, int64_t n, int agg,
                         float *s, int64_t lds, cudaStream_t st, const int64_t *n_seq = nullptr,
                         bool after_append = false);

// rows x n scores (row stride lds) -> rows x k ascending indices; when sel
// is given the indices also go to sel (row stride sel_stride) and k to counts.
cudaError_t launch_topk(int rows, const float *s, int64_t lds, int64_t n, int32_t k, int32_t *idx, RowCtl *ctl,
                        int32_t *dev_status, cudaStream_t st, int32_t *sel = nullptr, int32_t sel_stride = 0,
                        int32_t *counts = nullptr);

cudaError_t launch_expand(int rows, const int32_t *idx, int32_t k, int32_t r, int64_t n_pred, int64_t n_t,
                          int32_t *sel, int32_t sel_stride, int32_t *counts, int32_t *dev_status, cudaStream_t st);
// A ragged batch at a prediction: row (b, h) widens within [0, n_seq[b] + 1).
cudaError_t launch_expand_ragged(int rows, int Hkv, const int64_t *n_seq, const int32_t *idx, int32_t k, int32_t r,
                                 int32_t *sel, int32_t sel_stride, int32_t *counts, int32_t *dev_status,
                                 cudaStream_t st);
// sel row = [0, prefix_end) ++ windows of (idx + idx_off) clipped to
// [body_lo, body_hi) ++ [tail_start, n_t) (ranges disjoint and ascending).
cudaError_t launch_expand_ranges(int rows, const int32_t *idx, int32_t k, int32_t r, int64_t idx_off,
                                 int64_t prefix_end, int64_t body_lo, int64_t body_hi, int64_t tail_start,
                                 int64_t n_t, int32_t *sel, int32_t sel_stride, int32_t *counts, int32_t *dev_status,
                                 cudaStream_t st);

cudaError_t launch_attn(const tb_shape &sh, const uint16_t *q, const uint16_t *K, const uint16_t *V,
                        const int32_t *sel, const int32_t *counts, int32_t sel_stride, float scale, uint16_t *out,
                        uint32_t *attn_ctl, float *partials, int32_t *dev_status, cudaStream_t st);

// The same with up to three rounds of bulk copies in flight per CTA and two
// CTAs per SM (attn_stream.cu; D = 64 or 128, G <= 16, K/V in device memory).
bool attn_stream_supported(const tb_shape &sh);
// A step inside a prediction interval whose append kernel (K/V rows and projected key of the new token, no
// selection entry) was launched just before on the same stream: the streamed attention runs as that kernel's
// programmatic dependent, reads the new token's K/V rows from K_new / V_new, and adds the tail entry
// (sel[row][count] = pos, count + 1) once the append has finished. pos < 0: none of this.
struct AttnAppend {
    const uint16_t *K_new = nullptr, *V_new = nullptr;
    int32_t *sel = nullptr, *counts = nullptr;
    int64_t pos = -1;
};
cudaError_t launch_attn_stream(const tb_shape &sh, const uint16_t *q, const uint16_t *K, const uint16_t *V,
                               const int32_t *sel, const int32_t *counts, int32_t sel_stride, float scale,
                               uint16_t *out, uint32_t *attn_ctl, float *partials, int32_t *dev_status,
                               cudaStream_t st, const AttnAppend *app = nullptr);
// True when launch_attn (and so launch_attn_stream) serves this shape and K/V placement.
bool attn_stream_serves(const tb_shape &sh, const uint16_t *K, const uint16_t *V);
// True when K and V are device memory (answer kept per thread for the last pair asked).
bool kv_on_device(const void *K, const void *V);

// The same on the tensor cores (D = 64 or 128, G <= 16).
bool attn_mma_supported(const tb_shape &sh);
cudaError_t launch_attn_mma(const tb_shape &sh, const uint16_t *q, const uint16_t *K, const uint16_t *V,
                            const int32_t *sel, const int32_t *counts, int32_t sel_stride, float scale, uint16_t *out,
                            uint32_t *attn_ctl, float *partials, int32_t *dev_status, cudaStream_t st);

// One new row per (b, h): cache writes, its projection and (optionally) the
// tail entry of the selection.
// pos_seq (device, [B], may be null): per-sequence positions instead of pos.
cudaError_t launch_append(const tb_shape &sh, const uint16_t *K_new, const uint16_t *V_new, const uint16_t *Wk,
                          uint16_t *K, uint16_t *V, uint16_t *Kp, int64_t pos, int32_t *sel, int32_t sel_stride,
                          int32_t *counts, int32_t *dev_status, cudaStream_t st, const int64_t *pos_seq = nullptr);

// Kp rows [pos0, pos0 + n_new) from K_src (row stride src_stride per head).
// path: 0 automatic, 1 CUDA cores, 2 tensor cores (tcgen05).
cudaError_t launch_project(const tb_shape &sh, const uint16_t *K_src, int64_t src_stride, const uint16_t *Wk,
                           uint16_t *Kp, int64_t pos0, int64_t n_new, int32_t *dev_status, cudaStream_t st,
                           int path = 0);

// The whole decode step (T == 1, r == 0) as one cooperative kernel.
bool fused_step_supported(const tb_shape &sh, int64_t n_tokens, int32_t k);
int64_t fused_chunks(const tb_shape &sh, int64_t n_tokens);
cudaError_t launch_fused_step(const tb_shape &sh, const tb_step_params &p, int64_t n, const uint16_t *q,
                              const uint16_t *q_imp, const uint16_t *K_new, const uint16_t *V_new,
                              const uint16_t *Wk, uint16_t *K, uint16_t *V, uint16_t *Kp, int32_t *idx_state,
                              int32_t *sel, int32_t *counts, uint16_t *out, RowCtl *ctl, uint32_t *attn_ctl,
                              float *partials, int32_t sel_stride, int32_t *dev_status, cudaStream_t st);

// The decode step (T == 1, r == 0) as one cooperative kernel with a single
// exchange between the CTAs of a row (fused_fast.cu).
struct FastWs {
    RowCtl *ctl;
    float *part;
    uint8_t *rec;
    uint8_t *blk_above;
    int64_t blk_stride;
    uint32_t *keys_g;
    int64_t keys_stride;
    const WsDebug *dbg;
};
bool fused_fast_supported(const tb_shape &sh, int64_t n_tokens, int32_t k);
cudaError_t launch_fused_fast(const tb_shape &sh, const tb_step_params &p, int64_t n, const uint16_t *q,
                              const uint16_t *q_imp, const uint16_t *K_new, const uint16_t *V_new,
                              const uint16_t *Wk, uint16_t *K, uint16_t *V, uint16_t *Kp, int32_t *idx_state,
                              int32_t *sel, int32_t *counts, uint16_t *out, const FastWs &w, int32_t sel_stride,
                              int32_t *dev_status, cudaStream_t st, int32_t k_keep = 0, int64_t keep_lo = 0,
                              int64_t keep_hi = INT64_MAX, int32_t *centres = nullptr, int64_t cpre = 0,
                              int32_t ck = 0);
// k_keep > 0: keep that many tokens instead of p.k, with the tokens outside
// [keep_lo, keep_hi) forced in (maximal key); centres (ck per row, may be
// null) then receive the kept tokens of [keep_lo, keep_hi) minus keep_lo,
// which sit at sel slots cpre .. cpre + ck.

// The decode step (T == 1, r == 0) as three kernels with no grid-wide waits
// (pipe_step.cu): selection over the n cached tokens (scores, keys, the row's
// histogram), the bracket (the exact cut and each chunk's output offset),
// then the attention kernel that appends token n, lets it displace the row's
// k-th token when it scores above it, and attends. The bracket and the
// attention kernel are programmatic dependent launches. chain: the attention
// kernel follows the previous layer's attention kernel on its stream and its
// own layer's bracket kernel on another (the multi-layer step); otherwise it
// follows its own bracket kernel.
struct PipeGeom {
    int C;    // chunks (CTAs) per row
    int cs;   // tokens per chunk, a multiple of 16
};
bool pipe_supported(const tb_shape &sh, int64_t n, int32_t k);
PipeGeom pipe_geom(const tb_shape &sh, int64_t n);
cudaError_t launch_pipe_select(const tb_shape &sh, const PipeGeom &g, int agg, int64_t n, const uint16_t *q_imp,
                               const uint16_t *Kp, PipeRow *ctl, uint32_t *keys, int64_t keys_stride, bool chain,
                               int32_t *dev_status, cudaStream_t st);
cudaError_t launch_pipe_bracket(const tb_shape &sh, const PipeGeom &g, int32_t k, int64_t n, PipeRow *ctl,
                                const uint32_t *keys, int64_t keys_stride, uint2 *cand, int32_t *dev_status,
                                cudaStream_t st);
cudaError_t launch_pipe_attend(const tb_shape &sh, const PipeGeom &g, const tb_step_params &p, int64_t n, bool chain,
                               const uint16_t *q, const uint16_t *q_imp, const uint16_t *K_new, const uint16_t *V_new,
                               const uint16_t *Wk, uint16_t *K, uint16_t *V, uint16_t *Kp, int32_t *idx, int32_t *sel,
                               int32_t sel_stride, int32_t *counts, uint16_t *out, PipeRow *ctl, const uint32_t *keys,
                               int64_t keys_stride, float *part, int32_t *dev_status, cudaStream_t st);

// The predictor MLP for B tokens: h [B, F] = SiLU(x W1^T) (fp32), q_imp [B, O] =
// RNE(h W2^T). E and F multiples of 8, B <= 16.
cudaError_t launch_predict(const uint16_t *x, const uint16_t *W1, const uint16_t *W2, int B, int E, int F, int O,
                           float *h, uint16_t *q_imp, cudaStream_t st);

}  // namespace tb
