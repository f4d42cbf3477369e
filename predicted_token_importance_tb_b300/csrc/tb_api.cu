// C ABI of libtb: argument checks, workspace carving and launches. Every
// entry point opens an NVTX range of its own name (header-only NVTX 3: it
// costs a pointer test unless a profiling tool is attached).
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>

#include "kernels.cuh"
#include "tb_internal.cuh"
#include "ws_layout.cuh"

namespace tb {

struct NvtxRange {
    explicit NvtxRange(const char *name) { nvtxRangePushA(name); }
    ~NvtxRange() { nvtxRangePop(); }
};

const DevInfo &dev_info() {
    static thread_local DevInfo info;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return info;
    if (info.device != dev) {
        info.device = dev;
        cudaDeviceGetAttribute(&info.sms, cudaDevAttrMultiProcessorCount, dev);
        cudaDeviceGetAttribute(&info.l2_bytes, cudaDevAttrL2CacheSize, dev);
        cudaDeviceGetAttribute(&info.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    }
    return info;
}

static tb_status check_shape(const tb_shape *s) {
    if (!s) return TB_ERR_INVALID_ARG;
    if (s->B <= 0 || s->Hq <= 0 || s->Hkv <= 0 || s->D <= 0 || s->dp <= 0 || s->cap <= 0) return TB_ERR_INVALID_ARG;
    if (s->Hq % s->Hkv != 0) return TB_ERR_INVALID_ARG;
    if (s->Hq / s->Hkv > 16) return TB_ERR_UNSUPPORTED;
    if (s->D % 8 != 0 || s->dp % 8 != 0 || s->D > 256 || s->dp > 256) return TB_ERR_UNSUPPORTED;
    // attention groups of D/8 lanes must tile a warp
    const int tpg = s->D / 8;
    if (32 % tpg != 0) return TB_ERR_UNSUPPORTED;
    if (s->cap >= (int64_t)1 << 31) return TB_ERR_UNSUPPORTED;
    if ((int64_t)s->B * s->Hkv > (1 << 16)) return TB_ERR_UNSUPPORTED;
    return TB_OK;
}

static tb_status from_cuda(cudaError_t e) {
    if (e == cudaSuccess) return TB_OK;
    if (e == cudaErrorInvalidValue) return TB_ERR_UNSUPPORTED;
    return TB_ERR_CUDA;
}

#define TB_CHECK(x)                      \
    do {                                 \
        tb_status _st = (x);             \
        if (_st != TB_OK) return _st;    \
    } while (0)

#define TB_PTR(p)                                                   \
    do {                                                            \
        if (!(p)) return TB_ERR_INVALID_ARG;                        \
        if (!aligned16(p)) return TB_ERR_UNSUPPORTED;               \
    } while (0)

static WsLayout layout_for(const tb_shape &s, int64_t n_scores, int64_t sel_stride, int64_t fused_chunks_max) {
    return ws_layout(s, n_scores, sel_stride, fused_chunks_max);
}

// True when K and V are device memory (the bulk copies of the three-kernel
// step read them; pinned host K/V take the other paths). The answer for the
// last pair asked is kept per thread.
bool kv_on_device(const void *K, const void *V) {
    static thread_local const void *last_k = nullptr, *last_v = nullptr;
    static thread_local bool last = false;
    if (K == last_k && V == last_v) return last;
    bool ok = true;
    for (const void *p : {K, V}) {
        cudaPointerAttributes at;
        if (cudaPointerGetAttributes(&at, p) != cudaSuccess || at.type != cudaMemoryTypeDevice) {
            cudaGetLastError();
            ok = false;
        }
    }
    last_k = K;
    last_v = V;
    last = ok;
    return ok;
}

// Events that order the multi-layer step's two streams, created once per
// host thread and device.
struct StackEvents {
    int device = -1;
    cudaEvent_t fork = nullptr, sel = nullptr, join = nullptr;
};
static cudaError_t stack_events(StackEvents **out) {
    static thread_local StackEvents ev[16];
    const int dev = dev_info().device;
    if (dev < 0 || dev >= 16) return cudaErrorInvalidDevice;
    StackEvents &e = ev[dev];
    if (e.device != dev) {
        for (cudaEvent_t *x : {&e.fork, &e.sel, &e.join}) {
            cudaError_t r = cudaEventCreateWithFlags(x, cudaEventDisableTiming);
            if (r != cudaSuccess) return r;
        }
        e.device = dev;
    }
    *out = &e;
    return cudaSuccess;
}

}  // namespace tb

using namespace tb;

extern "C" {

const char *tb_status_string(tb_status st) {
    switch (st) {
        case TB_OK: return "ok";
        case TB_ERR_INVALID_ARG: return "invalid argument";
        case TB_ERR_UNSUPPORTED: return "unsupported shape or alignment";
        case TB_ERR_WORKSPACE: return "workspace missing or too small";
        case TB_ERR_CUDA: return "CUDA runtime error";
        case TB_ERR_TIMEOUT: return "device-side wait timed out";
        case TB_ERR_NONFINITE: return "non-finite (NaN) importance score";
    }
    return "unknown status";
}

int32_t tb_version(void) { return 1; }

tb_status tb_workspace_size(const tb_shape *shape, int64_t n_max, int32_t k_max, int32_t sel_stride_max,
                            size_t *bytes) {
    TB_CHECK(check_shape(shape));
    if (!bytes || n_max < 0 || k_max < 0 || sel_stride_max < 0) return TB_ERR_INVALID_ARG;
    int64_t ss = sel_stride_max > k_max ? sel_stride_max : k_max;
    const int64_t n_tok = n_max + 1;   // a decode step scores the appended token too
    *bytes = layout_for(*shape, n_tok, ss, fused_chunks(*shape, n_tok)).total;
    return TB_OK;
}

tb_status tb_workspace_init(void *ws, size_t ws_bytes, cudaStream_t stream) {
    NvtxRange nvtx_range("tb_workspace_init");
    if (!ws || ws_bytes == 0) return TB_ERR_INVALID_ARG;
    return from_cuda(cudaMemsetAsync(ws, 0, ws_bytes, stream));
}

tb_status tb_project_append(const tb_shape *shape, const tb_bf16 *K_src, int64_t src_stride, const tb_bf16 *Wk,
                            tb_bf16 *Kp, int64_t pos0, int64_t n_new, void *ws, size_t ws_bytes,
                            int32_t *dev_status, cudaStream_t stream) {
    NvtxRange nvtx_range("tb_project_append");
    (void)ws;
    (void)ws_bytes;
    TB_CHECK(check_shape(shape));
    if (n_new < 0 || pos0 < 0 || pos0 + n_new > shape->cap || n_new > src_stride) return TB_ERR_INVALID_ARG;
    if (n_new == 0) return TB_OK;
    TB_PTR(K_src);
    TB_PTR(Wk);
    TB_PTR(Kp);
    const size_t smem = ((size_t)shape->D * shape->dp + 64 * (size_t)(shape->D + 1)) * sizeof(float);
    if (smem > 227 * 1024) return TB_ERR_UNSUPPORTED;
    return from_cuda(launch_project(*shape, K_src, src_stride, Wk, Kp, pos0, n_new, dev_status, stream));
}

tb_status tb_score(const tb_shape *shape, const tb_bf16 *q_imp, const tb_bf16 *Kp, int64_t n, int32_t agg,
                   float *s, int32_t *dev_status, cudaStream_t stream) {
    NvtxRange nvtx_range("tb_score");
    (void)dev_status;
    TB_CHECK(check_shape(shape));
    if (n < 0 || n > shape->cap) return TB_ERR_INVALID_ARG;
    if (agg != TB_AGG_MEAN && agg != TB_AGG_MAX) return TB_ERR_INVALID_ARG;
    if (n == 0) return TB_OK;
    TB_PTR(q_imp);
    TB_PTR(Kp);
    if (!s) return TB_ERR_INVALID_ARG;
    return from_cuda(launch_score(*shape, q_imp, Kp, n, agg, s, n, stream));
}

tb_status tb_topk(const tb_shape *shape, const float *s, int64_t n, int32_t k, int32_t *idx, void *ws,
                  size_t ws_bytes, int32_t *dev_status, cudaStream_t stream) {
    NvtxRange nvtx_range("tb_topk");
    TB_CHECK(check_shape(shape));
    if (n < 0 || k < 0 || k > n) return TB_ERR_INVALID_ARG;
    if (k == 0) return TB_OK;
    if (!s || !idx) return TB_ERR_INVALID_ARG;
    if (n >= ((int64_t)1 << 31) - 1) return TB_ERR_UNSUPPORTED;
    const WsLayout L = layout_for(*shape, 0, 1, 0);
    if (!ws || ws_bytes < L.total) return TB_ERR_WORKSPACE;
    RowCtl *ctl = reinterpret_cast<RowCtl *>(static_cast<uint8_t *>(ws) + L.rowctl_off);
    return from_cuda(launch_topk(shape->B * shape->Hkv, s, n, n, k, idx, ctl, dev_status, stream));
}

tb_status tb_expand(const tb_shape *shape, const int32_t *idx, int32_t k, int32_t r, int64_t n_pred, int64_t n_t,
                    int32_t *sel, int32_t sel_stride, int32_t *counts, int32_t *dev_status, cudaStream_t stream) {
    NvtxRange nvtx_range("tb_expand");
    TB_CHECK(check_shape(shape));
    if (k < 0 || r < 0 || n_pred < 0 || n_t < n_pred || sel_stride <= 0 || n_t > shape->cap) return TB_ERR_INVALID_ARG;
    if ((k > 0 && !idx) || !sel || !counts) return TB_ERR_INVALID_ARG;
    return from_cuda(launch_expand(shape->B * shape->Hkv, idx, k, r, n_pred, n_t, sel, sel_stride, counts,
                                   dev_status, stream));
}

tb_status tb_sparse_decode_attn(const tb_shape *shape, const tb_bf16 *q, const tb_bf16 *K, const tb_bf16 *V,
                                const int32_t *sel, const int32_t *counts, int32_t sel_stride, float scale,
                                tb_bf16 *out, void *ws, size_t ws_bytes, int32_t *dev_status,
                                cudaStream_t stream) {
    NvtxRange nvtx_range("tb_sparse_decode_attn");
    TB_CHECK(check_shape(shape));
    if (sel_stride <= 0 || !sel) return TB_ERR_INVALID_ARG;
    TB_PTR(q);
    TB_PTR(K);
    TB_PTR(V);
    TB_PTR(out);
    const WsLayout L = layout_for(*shape, 0, sel_stride, 0);
    if (!ws || ws_bytes < L.total) return TB_ERR_WORKSPACE;
    uint8_t *w = static_cast<uint8_t *>(ws);
    return from_cuda(launch_attn(*shape, q, K, V, sel, counts, sel_stride, scale, out,
                                 reinterpret_cast<uint32_t *>(w + L.attn_ctl_off),
                                 reinterpret_cast<float *>(w + L.part_off), dev_status, stream));
}

tb_status tb_decode_step(const tb_shape *shape, const tb_step_params *p, int64_t t, int64_t n, const tb_bf16 *q,
                         const tb_bf16 *q_imp, const tb_bf16 *K_new, const tb_bf16 *V_new, const tb_bf16 *Wk,
                         tb_bf16 *K, tb_bf16 *V, tb_bf16 *Kp, int32_t *idx_state, int64_t *n_pred, int32_t *sel,
                         int32_t sel_stride, int32_t *counts, tb_bf16 *out, void *ws, size_t ws_bytes,
                         int32_t *dev_status, cudaStream_t stream) {
    NvtxRange nvtx_range("tb_decode_step");
    TB_CHECK(check_shape(shape));
    if (!p || !n_pred || !idx_state || !sel || !counts) return TB_ERR_INVALID_ARG;
    if (p->T < 1 || p->r < 0 || p->k < 1 || (p->agg != TB_AGG_MEAN && p->agg != TB_AGG_MAX)) return TB_ERR_INVALID_ARG;
    if (t < 0 || n < 0 || n + 1 > shape->cap) return TB_ERR_INVALID_ARG;
    TB_PTR(q);
    TB_PTR(q_imp);
    TB_PTR(K_new);
    TB_PTR(V_new);
    TB_PTR(Wk);
    TB_PTR(K);
    TB_PTR(V);
    TB_PTR(Kp);
    TB_PTR(out);
    if (p->flags & ~(TB_STEP_UNFUSED | TB_STEP_BUDGET_NEIGHBOURS | TB_STEP_PIPELINE)) return TB_ERR_INVALID_ARG;
    const int64_t n_t = n + 1;
    const bool predict = (t % p->T) == 0;
    // centres per prediction: k, or k / (2r + 1) (at least one) when the
    // widened selection must stay within the budget
    const int32_t kc = (p->flags & TB_STEP_BUDGET_NEIGHBOURS) ? (p->k / (2 * p->r + 1) > 0 ? p->k / (2 * p->r + 1) : 1)
                                                              : p->k;
    if (predict && kc > n_t) return TB_ERR_INVALID_ARG;
    if (!predict && (*n_pred <= 0 || *n_pred > n)) return TB_ERR_INVALID_ARG;   // a step of this interval is missing
    const int64_t np = predict ? n_t : *n_pred;
    int64_t body = (int64_t)kc * (2 * (int64_t)p->r + 1);
    if (body > np) body = np;
    if ((int64_t)sel_stride < body + (n_t - np)) return TB_ERR_INVALID_ARG;
    const int rows = shape->B * shape->Hkv;
    const bool one_launch = predict && p->T == 1 && p->r == 0 && !(p->flags & TB_STEP_UNFUSED);
    const bool pipe = one_launch && (p->flags & TB_STEP_PIPELINE) && pipe_supported(*shape, n, p->k) &&
                      kv_on_device(K, V);
    const bool fast = one_launch && !pipe && fused_fast_supported(*shape, n_t, p->k);
    const bool fused = one_launch && !pipe && !fast && fused_step_supported(*shape, n_t, p->k);
    const WsLayout L = layout_for(*shape, n_t, sel_stride, (fused || fast) ? fused_chunks(*shape, n_t) : 0);
    if (!ws || ws_bytes < L.total) return TB_ERR_WORKSPACE;
    uint8_t *w = static_cast<uint8_t *>(ws);
    RowCtl *ctl = reinterpret_cast<RowCtl *>(w + L.rowctl_off);
    uint32_t *actl = reinterpret_cast<uint32_t *>(w + L.attn_ctl_off);
    float *part = reinterpret_cast<float *>(w + L.part_off);
    float *scores = reinterpret_cast<float *>(w + L.scores_off);
    cudaError_t e;
    if (pipe) {
        // selection over the n cached tokens, the bracket (the exact cut), then the attention kernel (append,
        // the new token against the cut, gather, attention); the last two are programmatic dependents
        const PipeGeom g = pipe_geom(*shape, n);
        PipeRow *prow = reinterpret_cast<PipeRow *>(w + L.pipe_off);
        uint32_t *keys = reinterpret_cast<uint32_t *>(w + L.pipe_keys_off);
        e = launch_pipe_select(*shape, g, p->agg, n, q_imp, Kp, prow, keys, L.pipe_keys_stride, false, dev_status,
                               stream);
        if (e != cudaSuccess) return from_cuda(e);
        e = launch_pipe_bracket(*shape, g, p->k, n, prow, keys, L.pipe_keys_stride,
                                reinterpret_cast<uint2 *>(w + L.pipe_cand_off), dev_status, stream);
        if (e != cudaSuccess) return from_cuda(e);
        e = launch_pipe_attend(*shape, g, *p, n, false, q, q_imp, K_new, V_new, Wk, K, V, Kp, idx_state, sel,
                               sel_stride, counts, out, prow, keys, L.pipe_keys_stride,
                               reinterpret_cast<float *>(w + L.pipe_part_off), dev_status, stream);
        if (e != cudaSuccess) return from_cuda(e);
        *n_pred = n_t;
        return TB_OK;
    }
    if (fast) {
        FastWs fw;
        fw.ctl = ctl;
        fw.part = part;
        fw.rec = w + L.rec_off;
        fw.blk_above = w + L.blk_off;
        fw.blk_stride = L.blk_stride;
        fw.keys_g = reinterpret_cast<uint32_t *>(scores);
        fw.keys_stride = n_t;
        fw.dbg = reinterpret_cast<const WsDebug *>(w + L.debug_off);
        e = launch_fused_fast(*shape, *p, n, q, q_imp, K_new, V_new, Wk, K, V, Kp, idx_state, sel, counts, out, fw,
                              sel_stride, dev_status, stream);
        if (e != cudaSuccess) return from_cuda(e);
        *n_pred = n_t;
        return TB_OK;
    }
    if (fused) {
        e = launch_fused_step(*shape, *p, n, q, q_imp, K_new, V_new, Wk, K, V, Kp, idx_state, sel, counts, out, ctl,
                              actl, part, sel_stride, dev_status, stream);
        if (e != cudaSuccess) return from_cuda(e);
        *n_pred = n_t;
        return TB_OK;
    }
    // 1. append (and, inside an interval, the tail entry of the selection; the streamed attention adds that
    // entry itself when it serves the call, and starts while the append runs)
    const bool fold = !predict && attn_stream_serves(*shape, K, V);
    e = launch_append(*shape, K_new, V_new, Wk, K, V, Kp, n, predict || fold ? nullptr : sel, sel_stride, counts,
                      dev_status, stream);
    if (e != cudaSuccess) return from_cuda(e);
    if (predict) {
        // 2. score the n+1 tokens, select, widen
        e = launch_score(*shape, q_imp, Kp, n_t, p->agg, scores, n_t, stream, nullptr, true);
        if (e != cudaSuccess) return from_cuda(e);
        if (p->r == 0 && p->T == 1) {
            // no neighbours and no tail: the selection is the prediction itself
            e = launch_topk(rows, scores, n_t, n_t, p->k, idx_state, ctl, dev_status, stream, sel, sel_stride, counts);
            if (e != cudaSuccess) return from_cuda(e);
        } else {
            e = launch_topk(rows, scores, n_t, n_t, kc, idx_state, ctl, dev_status, stream);
            if (e != cudaSuccess) return from_cuda(e);
            e = launch_expand(rows, idx_state, kc, p->r, n_t, n_t, sel, sel_stride, counts, dev_status, stream);
            if (e != cudaSuccess) return from_cuda(e);
        }
        *n_pred = n_t;
    }
    // 3. attention over the selection
    if (fold) {
        AttnAppend app;
        app.K_new = K_new;
        app.V_new = V_new;
        app.sel = sel;
        app.counts = counts;
        app.pos = n;
        e = launch_attn_stream(*shape, q, K, V, sel, counts, sel_stride, p->scale, out, actl, part, dev_status,
                               stream, &app);
    } else {
        e = launch_attn(*shape, q, K, V, sel, counts, sel_stride, p->scale, out, actl, part, dev_status, stream);
    }
    return from_cuda(e);
}

tb_status tb_decode_layers(const tb_shape *shape, const tb_step_params *p, int64_t n, int32_t L,
                           const tb_layer_buffers *layers, int32_t sel_stride, int32_t *dev_status, cudaStream_t stream,
                           cudaStream_t select_stream) {
    NvtxRange nvtx_range("tb_decode_layers");
    TB_CHECK(check_shape(shape));
    if (!p || !layers || L < 1) return TB_ERR_INVALID_ARG;
    if (p->T != 1 || p->r != 0 || p->k < 1 || (p->agg != TB_AGG_MEAN && p->agg != TB_AGG_MAX)) return TB_ERR_INVALID_ARG;
    if (p->flags != 0) return TB_ERR_INVALID_ARG;
    if (n < 0 || n + 1 > shape->cap || p->k > n + 1) return TB_ERR_INVALID_ARG;
    if (sel_stride < p->k) return TB_ERR_INVALID_ARG;
    if (!pipe_supported(*shape, n, p->k)) return TB_ERR_UNSUPPORTED;
    if (select_stream == stream) return TB_ERR_INVALID_ARG;
    const WsLayout Lw = layout_for(*shape, n + 1, sel_stride, 0);
    for (int32_t l = 0; l < L; ++l) {
        const tb_layer_buffers &y = layers[l];
        TB_PTR(y.q);
        TB_PTR(y.q_imp);
        TB_PTR(y.K_new);
        TB_PTR(y.V_new);
        TB_PTR(y.Wk);
        TB_PTR(y.K);
        TB_PTR(y.V);
        TB_PTR(y.Kp);
        TB_PTR(y.out);
        if (!y.idx_state || !y.sel || !y.counts) return TB_ERR_INVALID_ARG;
        if (!y.ws || y.ws_bytes < Lw.total) return TB_ERR_WORKSPACE;
        for (int32_t m = 0; m < l; ++m)
            if (layers[m].ws == y.ws) return TB_ERR_INVALID_ARG;   // layers overlap on the GPU: one workspace each
    }
    for (int32_t l = 0; l < L; ++l)
        if (!kv_on_device(layers[l].K, layers[l].V)) return TB_ERR_UNSUPPORTED;
    StackEvents *ev = nullptr;
    cudaError_t e = stack_events(&ev);
    if (e != cudaSuccess) return from_cuda(e);
    const PipeGeom g = pipe_geom(*shape, n);
    // the selection stream starts after everything already on the caller's stream (the previous step's appends)
    if ((e = cudaEventRecord(ev->fork, stream)) != cudaSuccess) return from_cuda(e);
    if ((e = cudaStreamWaitEvent(select_stream, ev->fork, 0)) != cudaSuccess) return from_cuda(e);
    for (int32_t l = 0; l < L; ++l) {
        const tb_layer_buffers &y = layers[l];
        uint8_t *w = static_cast<uint8_t *>(y.ws);
        PipeRow *prow = reinterpret_cast<PipeRow *>(w + Lw.pipe_off);
        uint32_t *keys = reinterpret_cast<uint32_t *>(w + Lw.pipe_keys_off);
        e = launch_pipe_select(*shape, g, p->agg, n, y.q_imp, y.Kp, prow, keys, Lw.pipe_keys_stride, true,
                               dev_status, select_stream);
        if (e != cudaSuccess) return from_cuda(e);
        e = launch_pipe_bracket(*shape, g, p->k, n, prow, keys, Lw.pipe_keys_stride,
                                reinterpret_cast<uint2 *>(w + Lw.pipe_cand_off), dev_status, select_stream);
        if (e != cudaSuccess) return from_cuda(e);
        if ((e = cudaEventRecord(ev->sel, select_stream)) != cudaSuccess) return from_cuda(e);
        if ((e = cudaStreamWaitEvent(stream, ev->sel, 0)) != cudaSuccess) return from_cuda(e);
        e = launch_pipe_attend(*shape, g, *p, n, true, y.q, y.q_imp, y.K_new, y.V_new, y.Wk, y.K, y.V, y.Kp,
                               y.idx_state, y.sel, sel_stride, y.counts, y.out, prow, keys, Lw.pipe_keys_stride,
                               reinterpret_cast<float *>(w + Lw.pipe_part_off), dev_status, stream);
        if (e != cudaSuccess) return from_cuda(e);
    }
    if ((e = cudaEventRecord(ev->join, select_stream)) != cudaSuccess) return from_cuda(e);
    if ((e = cudaStreamWaitEvent(stream, ev->join, 0)) != cudaSuccess) return from_cuda(e);
    return TB_OK;
}

tb_status tb_decode_step_ragged(const tb_shape *shape, const tb_step_params *p, int64_t t, const int64_t *n_host,
                                const int64_t *n_dev, const tb_bf16 *q, const tb_bf16 *q_imp, const tb_bf16 *K_new,
                                const tb_bf16 *V_new, const tb_bf16 *Wk, tb_bf16 *K, tb_bf16 *V, tb_bf16 *Kp,
                                int32_t *idx_state, int64_t *n_pred, int32_t *sel, int32_t sel_stride, int32_t *counts,
                                tb_bf16 *out, void *ws, size_t ws_bytes, int32_t *dev_status, cudaStream_t stream) {
    NvtxRange nvtx_range("tb_decode_step_ragged");
    TB_CHECK(check_shape(shape));
    if (!p || !n_host || !n_dev || !n_pred || !idx_state || !sel || !counts) return TB_ERR_INVALID_ARG;
    if (p->T < 1 || p->r < 0 || p->k < 1 || (p->agg != TB_AGG_MEAN && p->agg != TB_AGG_MAX)) return TB_ERR_INVALID_ARG;
    if (p->flags & ~(TB_STEP_UNFUSED | TB_STEP_BUDGET_NEIGHBOURS)) return TB_ERR_INVALID_ARG;
    if (t < 0) return TB_ERR_INVALID_ARG;
    TB_PTR(q);
    TB_PTR(q_imp);
    TB_PTR(K_new);
    TB_PTR(V_new);
    TB_PTR(Wk);
    TB_PTR(K);
    TB_PTR(V);
    TB_PTR(Kp);
    TB_PTR(out);
    const bool predict = (t % p->T) == 0;
    const int32_t kc = (p->flags & TB_STEP_BUDGET_NEIGHBOURS) ? (p->k / (2 * p->r + 1) > 0 ? p->k / (2 * p->r + 1) : 1)
                                                              : p->k;
    int64_t n_lo = INT64_MAX, n_hi = -1;
    for (int b = 0; b < shape->B; ++b) {
        const int64_t nb = n_host[b];
        if (nb < 0 || nb + 1 > shape->cap) return TB_ERR_INVALID_ARG;
        if (!predict && (n_pred[b] <= 0 || n_pred[b] > nb)) return TB_ERR_INVALID_ARG;
        n_lo = nb < n_lo ? nb : n_lo;
        n_hi = nb > n_hi ? nb : n_hi;
    }
    const int64_t nt_hi = n_hi + 1;
    if (predict && kc > n_lo + 1) return TB_ERR_INVALID_ARG;
    int64_t body = (int64_t)kc * (2 * (int64_t)p->r + 1);
    if (body > nt_hi) body = nt_hi;
    int64_t tail = 0;   // the longest tail of the interval so far
    if (!predict)
        for (int b = 0; b < shape->B; ++b) tail = (n_host[b] + 1 - n_pred[b]) > tail ? n_host[b] + 1 - n_pred[b] : tail;
    if ((int64_t)sel_stride < body + (predict ? 0 : tail)) return TB_ERR_INVALID_ARG;
    const int rows = shape->B * shape->Hkv;
    const WsLayout L = layout_for(*shape, nt_hi, sel_stride, 0);
    if (!ws || ws_bytes < L.total) return TB_ERR_WORKSPACE;
    uint8_t *w = static_cast<uint8_t *>(ws);
    RowCtl *ctl = reinterpret_cast<RowCtl *>(w + L.rowctl_off);
    uint32_t *actl = reinterpret_cast<uint32_t *>(w + L.attn_ctl_off);
    float *part = reinterpret_cast<float *>(w + L.part_off);
    float *scores = reinterpret_cast<float *>(w + L.scores_off);
    // 1. append at each sequence's own position (and the tail entry inside an interval)
    cudaError_t e = launch_append(*shape, K_new, V_new, Wk, K, V, Kp, 0, predict ? nullptr : sel, sel_stride, counts,
                                  dev_status, stream, n_dev);
    if (e != cudaSuccess) return from_cuda(e);
    if (predict) {
        // 2. score up to the longest sequence (later positions of the shorter ones score -inf), select, widen
        e = launch_score(*shape, q_imp, Kp, nt_hi, p->agg, scores, nt_hi, stream, n_dev, true);
        if (e != cudaSuccess) return from_cuda(e);
        if (p->r == 0 && p->T == 1) {
            e = launch_topk(rows, scores, nt_hi, nt_hi, kc, idx_state, ctl, dev_status, stream, sel, sel_stride, counts);
            if (e != cudaSuccess) return from_cuda(e);
        } else {
            e = launch_topk(rows, scores, nt_hi, nt_hi, kc, idx_state, ctl, dev_status, stream);
            if (e != cudaSuccess) return from_cuda(e);
            e = launch_expand_ragged(rows, shape->Hkv, n_dev, idx_state, kc, p->r, sel, sel_stride, counts, dev_status,
                                     stream);
            if (e != cudaSuccess) return from_cuda(e);
        }
        for (int b = 0; b < shape->B; ++b) n_pred[b] = n_host[b] + 1;
    }
    // 3. attention over the selection
    e = launch_attn(*shape, q, K, V, sel, counts, sel_stride, p->scale, out, actl, part, dev_status, stream);
    return from_cuda(e);
}

tb_status tb_predict_queries(const tb_bf16 *x, const tb_bf16 *W1, const tb_bf16 *W2, int32_t B, int32_t E,
                             int32_t F, int32_t O, tb_bf16 *q_imp, void *ws, size_t ws_bytes, int32_t *dev_status,
                             cudaStream_t stream) {
    NvtxRange nvtx_range("tb_predict_queries");
    (void)dev_status;   // nothing on this path is detected on the device
    if (B < 1 || E < 1 || F < 1 || O < 1) return TB_ERR_INVALID_ARG;
    if (B > 16 || E % 8 != 0 || F % 8 != 0) return TB_ERR_UNSUPPORTED;
    if ((int64_t)B * E * 2 > 200 * 1024 || (int64_t)B * F * 4 > 200 * 1024) return TB_ERR_UNSUPPORTED;
    TB_PTR(x);
    TB_PTR(W1);
    TB_PTR(W2);
    TB_PTR(q_imp);
    TB_PTR(ws);
    if (ws_bytes < (size_t)B * F * 4) return TB_ERR_WORKSPACE;
    return from_cuda(launch_predict(x, W1, W2, B, E, F, O, static_cast<float *>(ws), q_imp, stream));
}

tb_status tb_decode_step_buffered(const tb_shape *shape, const tb_step_params *p, const tb_buffer_params *bp,
                                  int64_t t, int64_t n, const tb_bf16 *q, const tb_bf16 *q_imp,
                                  const tb_bf16 *K_new, const tb_bf16 *V_new, const tb_bf16 *Wk, tb_bf16 *K,
                                  tb_bf16 *V, tb_bf16 *Kp, int32_t *idx_state, int64_t *n_pred, int64_t *proj_end,
                                  int32_t *sel, int32_t sel_stride, int32_t *counts, tb_bf16 *out, void *ws,
                                  size_t ws_bytes, int32_t *dev_status, cudaStream_t stream) {
    NvtxRange nvtx_range("tb_decode_step_buffered");
    TB_CHECK(check_shape(shape));
    if (!p || !bp || !n_pred || !proj_end || !idx_state || !sel || !counts) return TB_ERR_INVALID_ARG;
    if (p->T < 1 || p->r < 0 || p->k < 1 || (p->agg != TB_AGG_MEAN && p->agg != TB_AGG_MAX)) return TB_ERR_INVALID_ARG;
    if (p->flags & ~(TB_STEP_UNFUSED | TB_STEP_BUDGET_NEIGHBOURS)) return TB_ERR_INVALID_ARG;
    if (bp->sink < 0 || bp->window < 1) return TB_ERR_INVALID_ARG;
    if (t < 0 || n < 0 || n + 1 > shape->cap) return TB_ERR_INVALID_ARG;
    if (*proj_end < 0 || *proj_end > n) return TB_ERR_INVALID_ARG;
    TB_PTR(q);
    TB_PTR(q_imp);
    TB_PTR(K_new);
    TB_PTR(V_new);
    TB_PTR(Wk);
    TB_PTR(K);
    TB_PTR(V);
    TB_PTR(Kp);
    TB_PTR(out);
    const int64_t n_t = n + 1, S = bp->sink, W = bp->window;
    const bool predict = (t % p->T) == 0;
    if (!predict && (*n_pred <= 0 || *n_pred > n)) return TB_ERR_INVALID_ARG;   // a step of this interval is missing
    const int32_t kc0 = (p->flags & TB_STEP_BUDGET_NEIGHBOURS) ? (p->k / (2 * p->r + 1) > 0 ? p->k / (2 * p->r + 1) : 1)
                                                               : p->k;
    // batches that have left the window, and the ranges of the selection
    int64_t P = *proj_end;
    if (predict && n_t - W - P >= W) P += W * ((n_t - W - P) / W);
    const int64_t nc = P > S ? P - S : 0;                       // candidates [S, P)
    const int32_t kc = predict ? (int32_t)(nc < kc0 ? nc : kc0) : 0;
    const int64_t pre = S < n_t ? S : n_t;                      // sink prefix [0, pre)
    const int64_t tail0 = P > pre ? P : pre;                     // window [tail0, n_t)
    if (predict) {
        int64_t body = (int64_t)kc * (2 * (int64_t)p->r + 1);
        if (body > nc) body = nc;
        if ((int64_t)sel_stride < pre + body + (n_t - tail0)) return TB_ERR_INVALID_ARG;   // (the interval's
        // later steps add one entry each; the append kernel checks those on the device)
    }
    const int rows = shape->B * shape->Hkv;
    // a prediction at every step without neighbours runs as the single-launch
    // step: the sink and window tokens take the maximal key, so keeping
    // k_keep = sink + kc + window tokens keeps exactly them and the top kc
    // candidates, in ascending order
    const int32_t k_keep = (int32_t)(pre + kc + (n_t - tail0));
    const bool one_launch = predict && p->T == 1 && p->r == 0 && !(p->flags & TB_STEP_UNFUSED) &&
                            (int64_t)sel_stride >= k_keep && fused_fast_supported(*shape, n_t, k_keep);
    const WsLayout L = layout_for(*shape, n_t, sel_stride, one_launch ? fused_chunks(*shape, n_t) : 0);
    if (!ws || ws_bytes < L.total) return TB_ERR_WORKSPACE;
    uint8_t *w = static_cast<uint8_t *>(ws);
    RowCtl *ctl = reinterpret_cast<RowCtl *>(w + L.rowctl_off);
    uint32_t *actl = reinterpret_cast<uint32_t *>(w + L.attn_ctl_off);
    float *part = reinterpret_cast<float *>(w + L.part_off);
    float *scores = reinterpret_cast<float *>(w + L.scores_off);
    cudaError_t e;
    if (one_launch) {
        if (P > *proj_end) {   // the batches that left the window first
            e = launch_project(*shape, K + *proj_end * shape->D, shape->cap, Wk, Kp, *proj_end, P - *proj_end,
                               dev_status, stream);
            if (e != cudaSuccess) return from_cuda(e);
            *proj_end = P;
        }
        FastWs fw;
        fw.ctl = ctl;
        fw.part = part;
        fw.rec = w + L.rec_off;
        fw.blk_above = w + L.blk_off;
        fw.blk_stride = L.blk_stride;
        fw.keys_g = reinterpret_cast<uint32_t *>(scores);
        fw.keys_stride = n_t;
        fw.dbg = reinterpret_cast<const WsDebug *>(w + L.debug_off);
        // candidates [S, P): everything outside is forced (with P <= S, everything)
        e = launch_fused_fast(*shape, *p, n, q, q_imp, K_new, V_new, Wk, K, V, Kp, nullptr, sel, counts, out, fw,
                              sel_stride, dev_status, stream, k_keep, S, P > S ? P : S, idx_state, pre, kc);
        if (e != cudaSuccess) return from_cuda(e);
        *n_pred = n_t;
        return TB_OK;
    }
    // 1. append K/V (and, inside an interval, the tail entry of the selection)
    e = launch_append(*shape, K_new, V_new, nullptr, K, V, nullptr, n, predict ? nullptr : sel, sel_stride,
                      counts, dev_status, stream);
    if (e != cudaSuccess) return from_cuda(e);
    if (predict) {
        // 2. the batches that left the window -> Kp; score the candidates, select, widen, add sink and window
        if (P > *proj_end) {
            e = launch_project(*shape, K + *proj_end * shape->D, shape->cap, Wk, Kp, *proj_end, P - *proj_end,
                               dev_status, stream);
            if (e != cudaSuccess) return from_cuda(e);
            *proj_end = P;
        }
        if (kc > 0) {
            e = launch_score(*shape, q_imp, Kp + S * shape->dp, nc, p->agg, scores, nc, stream);
            if (e != cudaSuccess) return from_cuda(e);
            e = launch_topk(rows, scores, nc, nc, kc, idx_state, ctl, dev_status, stream);
            if (e != cudaSuccess) return from_cuda(e);
        }
        e = launch_expand_ranges(rows, idx_state, kc, p->r, S, pre, S, P, tail0, n_t, sel, sel_stride, counts,
                                 dev_status, stream);
        if (e != cudaSuccess) return from_cuda(e);
        *n_pred = n_t;
    }
    // 3. attention over the selection
    e = launch_attn(*shape, q, K, V, sel, counts, sel_stride, p->scale, out, actl, part, dev_status, stream);
    return from_cuda(e);
}

}  // extern "C"
