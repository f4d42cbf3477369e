/*
 * tb.h -- C ABI of the TokenButler decode-time hot path on one B300 (sm_103a).
 *
 * The method ("TokenButler: Token Importance is Predictable"; arXiv abstract
 * and the gist.science technical summary): every KV head keeps a
 * low-dimensional copy of its keys, Kp = K . Wk. At a decode step an
 * importance query scores all cached tokens against Kp, a fixed budget of k
 * individual tokens per KV head is kept, optionally reused for T steps and
 * widened by +-r neighbours, and exact softmax attention runs over only those
 * full-precision K/V rows while the whole cache stays in device memory.
 *
 * Conventions shared by every call
 * --------------------------------
 *  - bf16 tensors travel as raw 16-bit patterns (tb_bf16). All tensor
 *    pointers are DEVICE pointers, 16-byte aligned, dense row-major, with
 *    one exception: K and V of tb_sparse_decode_attn and tb_decode_step may
 *    be pinned host memory that the device reaches through unified
 *    addressing (cudaMallocHost / cudaHostAlloc). That is the offloaded
 *    cache of the TokenButler abstract and the gist.science summary
 *    ("Significance"): only the selected rows (and the appended row) cross
 *    the host link, while Kp, which every step streams whole, stays in
 *    device memory. Same results, host-link speed.
 *  - Shapes: B batch, Hq query heads, Hkv KV heads (G = Hq/Hkv query heads
 *    share one KV head), D head dim, dp projected dim, cap cache rows.
 *      K, V  : [B, Hkv, cap, D]        Kp : [B, Hkv, cap, dp]
 *      Wk    : [Hkv, D, dp]            q  : [B, Hq, D]
 *      q_imp : [B, Hq, dp]             s  : [B, Hkv, n] (fp32)
 *      idx   : [B, Hkv, k] (int32)     sel: [B, Hkv, sel_stride] (int32)
 *      out   : [B, Hq, D]
 *  - Limits: D in {8, 16, 32, 64, 128, 256} (D/8 lanes tile a warp), dp a
 *    multiple of 8 and <= 256, Hq % Hkv == 0, G <= 16, cap < 2^31.
 *    Violations return TB_ERR_UNSUPPORTED or TB_ERR_INVALID_ARG before
 *    anything is enqueued.
 *  - The caller owns all memory; the library allocates none. Scratch comes
 *    from a caller-provided workspace of tb_workspace_size() bytes that must
 *    be zero-filled before its first use (tb_workspace_init); every call that
 *    completes puts the control words it used back to zero, so later calls
 *    need no re-initialisation. One workspace may serve every call, but calls
 *    sharing a workspace must not overlap on the GPU.
 *  - Every call is asynchronous on the caller's stream. The returned status
 *    covers argument checks and the launch. Errors found on the device
 *    (a bad index, a NaN score, a wait that timed out) are written to
 *    *dev_status (a device int32, may be NULL) as a tb_status code; the first
 *    one written sticks until the caller resets the word to 0. After
 *    TB_ERR_TIMEOUT the workspace must be zero-filled again.
 *  - No call aborts, traps or throws across this boundary.
 */
#ifndef TB_H_
#define TB_H_

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define TB_API __attribute__((visibility("default")))
#else
#define TB_API
#endif

typedef uint16_t tb_bf16;

typedef enum {
    TB_OK = 0,
    TB_ERR_INVALID_ARG = 1,   /* bad pointer, size, index or combination */
    TB_ERR_UNSUPPORTED = 2,   /* shape or alignment outside the limits above */
    TB_ERR_WORKSPACE = 3,     /* workspace missing or smaller than required */
    TB_ERR_CUDA = 4,          /* a CUDA runtime call failed (launch, attribute) */
    TB_ERR_TIMEOUT = 5,       /* a bounded device-side wait gave up */
    TB_ERR_NONFINITE = 6      /* a NaN importance score */
} tb_status;

#define TB_AGG_MEAN 0  /* group score = mean of the G query heads' dot products */
#define TB_AGG_MAX 1   /* group score = max of them */

typedef struct {
    int32_t B, Hq, Hkv, D, dp;
    int64_t cap;
} tb_shape;

/* Per-layer decode settings. */
typedef struct {
    int32_t k;      /* budget per (batch, KV head), 1 <= k */
    int32_t T;      /* prediction interval in steps, >= 1 */
    int32_t r;      /* neighbour radius, >= 0 */
    int32_t agg;    /* TB_AGG_MEAN or TB_AGG_MAX */
    float scale;    /* softmax scale, normally 1/sqrt(D) */
    int32_t flags;  /* 0, or TB_STEP_UNFUSED */
} tb_step_params;

/* tb_step_params.flags: run the step as separate kernels even where the
   single fused launch applies (same results; for comparison and debugging). */
#define TB_STEP_UNFUSED 1
/* tb_step_params.flags: budget-preserving neighbour fetching (a variant of
   the gist.science summary's Neighbor Fetching, Optimizations): a prediction
   keeps kc = max(1, k / (2r + 1)) centres instead of k, so the widened
   selection holds at most k tokens (plus the tail). idx_state then holds kc
   entries per row, packed ([B, Hkv, kc]). With r == 0 it changes nothing. */
#define TB_STEP_BUDGET_NEIGHBOURS 2
/* tb_step_params.flags: run a step with a prediction, T == 1 and r == 0 as
   three kernels with no grid-wide waits instead of the single cooperative
   kernel: the top k of the n cached tokens is selected first (their scores,
   then the exact cut), then token n is appended and displaces the k-th of
   them when it scores above it, which is the top k of all n + 1 tokens. Needs
   D in {64, 128}, dp in {16, 32, 64}, G <= 16, n >= 1024 and K/V in device
   memory (otherwise the flag is ignored). Same results up to the fp32
   rounding of the scores. These kernels also carry tb_decode_layers. */
#define TB_STEP_PIPELINE 4

/* Text for a status code (static storage). */
TB_API const char *tb_status_string(tb_status st);

/* ABI version, currently 1. */
TB_API int32_t tb_version(void);

/*
 * Bytes of workspace that any call below needs for shapes up to `shape`,
 * token counts up to n_max, budgets up to k_max and selections of up to
 * sel_stride_max rows. Written to *bytes.
 */
TB_API tb_status tb_workspace_size(const tb_shape *shape, int64_t n_max, int32_t k_max,
                            int32_t sel_stride_max, size_t *bytes);

/* Zero-fill a workspace on `stream` (needed once, and after TB_ERR_TIMEOUT). */
TB_API tb_status tb_workspace_init(void *ws, size_t ws_bytes, cudaStream_t stream);

/*
 * Key projection into the low-dimensional cache ("Core Architecture",
 * Key-Cache Projection: the consumer layer's full keys are multiplied by a
 * trained matrix into the importance space; "Optimizations", Batching: many
 * tokens are projected in one call rather than one per step).
 *
 *   Kp[b,h,pos0+i,:] = RNE_bf16( K_src[b,h,i,:] . Wk[h] )   0 <= i < n_new
 *
 * fp32 accumulation. K_src row i of head (b,h) is at
 * K_src + ((b*Hkv + h)*src_stride + i)*D, so passing the cache itself with
 * src_stride = cap and K_src = K + pos0*D projects rows already stored there.
 * Requires pos0 + n_new <= cap and n_new <= src_stride.
 * Large n_new runs on the tensor cores (tcgen05, TMA-fed).
 */
TB_API tb_status tb_project_append(const tb_shape *shape, const tb_bf16 *K_src, int64_t src_stride,
                            const tb_bf16 *Wk, tb_bf16 *Kp, int64_t pos0, int64_t n_new,
                            void *ws, size_t ws_bytes, int32_t *dev_status, cudaStream_t stream);

/*
 * Importance scores ("Core Architecture", Scoring: a token's importance is
 * the inner product of the predicted query with its projected key).
 *
 *   s[b,h,t] = agg_{g<G} sum_i q_imp[b,h*G+g,i] * Kp[b,h,t,i]    0 <= t < n
 *
 * fp32; agg is TB_AGG_MEAN or TB_AGG_MAX. s is dense [B, Hkv, n].
 */
TB_API tb_status tb_score(const tb_shape *shape, const tb_bf16 *q_imp, const tb_bf16 *Kp, int64_t n,
                   int32_t agg, float *s, int32_t *dev_status, cudaStream_t stream);

/*
 * Per-token selection with a fixed budget (arXiv abstract: individual tokens,
 * k of them, are kept at each step). For each (b,h) row of s [B,Hkv,n], idx
 * receives the k tokens with the largest scores, ties to the lower index,
 * in ascending index order. 0 <= k <= n. -0.0 ties with +0.0; a NaN score
 * writes TB_ERR_NONFINITE to *dev_status (the NaN then ranks lowest).
 * Exact: the result is bit-identical to a full sort of the fp32 scores.
 */
TB_API tb_status tb_topk(const tb_shape *shape, const float *s, int64_t n, int32_t k, int32_t *idx,
                  void *ws, size_t ws_bytes, int32_t *dev_status, cudaStream_t stream);

/*
 * Neighbour fetching and the prediction-interval tail ("Optimizations",
 * Prediction Interval & Neighbor Fetching). For each row, from idx [.,k]
 * (strictly ascending, within [0, n_pred)):
 *   sel = sorted unique union of [i-r, i+r] clipped to [0, n_pred), followed
 *         by n_pred, n_pred+1, ..., n_t-1 (tokens appended since prediction)
 *   counts = its length (<= sel_stride, else TB_ERR_INVALID_ARG on device).
 */
TB_API tb_status tb_expand(const tb_shape *shape, const int32_t *idx, int32_t k, int32_t r,
                    int64_t n_pred, int64_t n_t, int32_t *sel, int32_t sel_stride,
                    int32_t *counts, int32_t *dev_status, cudaStream_t stream);

/*
 * Exact attention over the selected rows (arXiv abstract; "Significance":
 * the full cache is kept and only the relevant tokens are read).
 *
 *   out[b,hq,:] = sum_{j in sel[b,h]} softmax_j(scale * q[b,hq].K[b,h,j]) V[b,h,j]
 *
 * with h = hq / G; the first counts[b,h] entries of each sel row are used
 * (counts == NULL: all sel_stride). fp32 online softmax split over the
 * selection, merged in-kernel. An entry outside [0, cap) or an empty row is
 * skipped and writes TB_ERR_INVALID_ARG to *dev_status.
 */
TB_API tb_status tb_sparse_decode_attn(const tb_shape *shape, const tb_bf16 *q, const tb_bf16 *K,
                                const tb_bf16 *V, const int32_t *sel, const int32_t *counts,
                                int32_t sel_stride, float scale, tb_bf16 *out,
                                void *ws, size_t ws_bytes, int32_t *dev_status,
                                cudaStream_t stream);

/*
 * One decode step of one layer, all of the above in order ("Optimizations":
 * the predictor runs once every T steps, its selection is reused in between
 * and widened by neighbours).
 *   1. append: K[.,.,n] = K_new, V[.,.,n] = V_new, Kp[.,.,n] = RNE(K_new . Wk)
 *   2. if t % T == 0: score the n+1 tokens, keep the top k in idx_state,
 *      *n_pred = n+1 (host scalar), then sel = expand(idx_state, r, n_pred, n+1)
 *      else sel += [n] (the tail since the prediction)
 *   3. out = attention of q over sel.
 * K_new, V_new: [B, Hkv, D]. idx_state [B,Hkv,k], sel [B,Hkv,sel_stride] and
 * counts [B,Hkv] persist across the steps of an interval; sel_stride must be
 * >= min(n+1, kc(2r+1)) + T - 1, kc = k (or k / (2r+1), at least 1, with
 * TB_STEP_BUDGET_NEIGHBOURS). The steps of an interval must be issued in
 * order with consecutive t and n. With T == 1 and r == 0 the step runs as one
 * cooperative kernel where the shape allows (see TB_STEP_PIPELINE for the
 * three-kernel form).
 */
TB_API tb_status tb_decode_step(const tb_shape *shape, const tb_step_params *params, int64_t t, int64_t n,
                         const tb_bf16 *q, const tb_bf16 *q_imp, const tb_bf16 *K_new,
                         const tb_bf16 *V_new, const tb_bf16 *Wk, tb_bf16 *K, tb_bf16 *V,
                         tb_bf16 *Kp, int32_t *idx_state, int64_t *n_pred, int32_t *sel,
                         int32_t sel_stride, int32_t *counts, tb_bf16 *out,
                         void *ws, size_t ws_bytes, int32_t *dev_status, cudaStream_t stream);

/* One layer's buffers for tb_decode_layers; each as for tb_decode_step. The
   workspace (tb_workspace_size bytes, zero-filled once) is the layer's own:
   the layers' kernels overlap on the GPU. */
typedef struct {
    const tb_bf16 *q, *q_imp, *K_new, *V_new, *Wk;
    tb_bf16 *K, *V, *Kp;
    int32_t *idx_state, *sel, *counts;
    tb_bf16 *out;
    void *ws;
    size_t ws_bytes;
} tb_layer_buffers;

/*
 * One decode step of L consumer layers that share one producer layer
 * ("TokenButler: Token Importance is Predictable", gist.science summary,
 * Core Architecture: the importance queries are predicted at a producer
 * layer and scored against the projected keys of the layers after it).
 * Layer l's result is exactly tb_decode_step's with a prediction, T == 1 and
 * r == 0, on layers[l]; n is every layer's token count before the append.
 *
 * Because every layer's q_imp is known before the first of them runs, the
 * selection of layer l (its n cached tokens scored against q_imp, the top k
 * kept) needs nothing from layer l - 1 and runs on select_stream while
 * earlier layers attend on `stream`. Layer l's attention kernel (the append
 * of its new token, that token scored against the layer's k-th, the gather
 * and the attention) runs on `stream` in layer order after its own
 * selection; it gathers the kept rows first and reads q, K_new and V_new,
 * which in a model come from layer l - 1's output, only once layer l - 1's
 * attention kernel has finished. select_stream first waits for the work
 * already on `stream`; on return `stream` waits for select_stream. Two
 * events per host thread and device are created on first use (no device
 * memory). Needs the shapes of TB_STEP_PIPELINE, k <=
 * n + 1, sel_stride >= k, device-resident K/V and one workspace per layer;
 * otherwise TB_ERR_UNSUPPORTED or TB_ERR_INVALID_ARG before anything is
 * enqueued.
 */
TB_API tb_status tb_decode_layers(const tb_shape *shape, const tb_step_params *params, int64_t n, int32_t L,
                                  const tb_layer_buffers *layers, int32_t sel_stride, int32_t *dev_status,
                                  cudaStream_t stream, cudaStream_t select_stream);

/*
 * tb_decode_step for a ragged batch: sequence b holds n[b] tokens before
 * this step's append (the method's descriptions batch sequences without
 * saying how their lengths may differ). Per sequence the step is exactly
 * tb_decode_step's: the new K/V/Kp rows go to position n[b], a prediction
 * scores that sequence's n[b] + 1 tokens and keeps the top k, the widening
 * stays inside them, and between predictions the sequence's new token joins
 * its selection.
 * n_host [B] (host) and n_dev [B] (device) hold the same values;
 * n_pred [B] is the host state of the interval, one entry per sequence.
 * Needs k <= n[b] + 1 for every b at a prediction and sel_stride >=
 * min(max_b n[b] + 1, k (2r+1)) + T - 1. Always separate kernels.
 */
TB_API tb_status tb_decode_step_ragged(const tb_shape *shape, const tb_step_params *params, int64_t t,
                                       const int64_t *n_host, const int64_t *n_dev, const tb_bf16 *q,
                                       const tb_bf16 *q_imp, const tb_bf16 *K_new, const tb_bf16 *V_new,
                                       const tb_bf16 *Wk, tb_bf16 *K, tb_bf16 *V, tb_bf16 *Kp,
                                       int32_t *idx_state, int64_t *n_pred, int32_t *sel, int32_t sel_stride,
                                       int32_t *counts, tb_bf16 *out, void *ws, size_t ws_bytes,
                                       int32_t *dev_status, cudaStream_t stream);

/*
 * The importance-query predictor ("TokenButler: Token Importance is
 * Predictable", gist.science summary, Core Architecture, Query Prediction: a
 * small multi-layer perceptron from a producer layer's hidden state to G
 * low-dimensional importance queries for each KV head), for B tokens:
 *   h     = SiLU(x . W1^T)          x [B, E] bf16, W1 [F, E] bf16, h fp32
 *   q_imp = RNE_bf16(h . W2^T)      W2 [O, F] bf16, q_imp [B, O] = [B, Hq, dp]
 * The method's descriptions give no depth, width, activation or bias: two layers, no bias,
 * SiLU (the activation of the base models' MLPs), fp32 accumulation and one
 * rounding at the end are this library's reading. Limits: 1 <= B <= 16,
 * E and F multiples of 8, B E 2 and B F 4 bytes <= 200 KB. ws: at least
 * B F 4 bytes of device memory for h (no zero-fill needed).
 */
TB_API tb_status tb_predict_queries(const tb_bf16 *x, const tb_bf16 *W1, const tb_bf16 *W2, int32_t B,
                                    int32_t E, int32_t F, int32_t O, tb_bf16 *q_imp, void *ws,
                                    size_t ws_bytes, int32_t *dev_status, cudaStream_t stream);

/*
 * Sink and local-window buffers ("TokenButler: Token Importance is
 * Predictable", gist.science summary, Inference Strategy: the first S tokens
 * and a window of the newest tokens are always kept, the important tokens
 * come from the predictor; Optimizations, Batching: keys are projected in
 * batches of W tokens instead of at every step).
 */
typedef struct {
    int32_t sink;     /* S >= 0: tokens [0, S) are always attended */
    int32_t window;   /* W >= 1: at least the newest W tokens are always attended; Kp grows in batches of W */
} tb_buffer_params;

/*
 * One decode step of one layer with the three buffers. With n_t = n + 1:
 *   1. append: K[.,.,n] = K_new, V[.,.,n] = V_new (no projection here)
 *   2. if t % T == 0:
 *        P = *proj_end + W * floor((n_t - W - *proj_end) / W) if that adds a
 *        batch: Kp[., ., *proj_end : P) = RNE(K rows . Wk) in one launch,
 *        *proj_end = P; then the candidates [S, P) are scored, the top kc
 *        kept in idx_state (kc = k, or the TB_STEP_BUDGET_NEIGHBOURS count,
 *        at most P - S; indices relative to S) and
 *          sel = [0, min(S, n_t)) ++ widen(idx + S, r) within [S, P)
 *                ++ [max(P, min(S, n_t)), n_t),
 *        *n_pred = n_t
 *      else sel += [n]
 *   3. out = attention of q over sel.
 * So the window holds the tokens since the last batch, W to 2W - 1 of them
 * at a prediction (plus the steps of the interval). *proj_end (host scalar)
 * is the number of rows Kp holds; start it at the rows projected before
 * (for instance by tb_project_append at prefill). sel_stride must be at least
 * min(S, n_t) + min(P - S, kc (2r+1)) + (n_t - max(P, min(S, n_t))) at every
 * prediction (else TB_ERR_INVALID_ARG), and each later step of the interval
 * adds one entry (TB_ERR_INVALID_ARG on the device when it does not fit). params->flags may hold
 * TB_STEP_BUDGET_NEIGHBOURS; the step always runs as separate kernels.
 * Pointers and layouts as for tb_decode_step.
 */
TB_API tb_status tb_decode_step_buffered(const tb_shape *shape, const tb_step_params *params,
                                         const tb_buffer_params *buffers, int64_t t, int64_t n, const tb_bf16 *q,
                                         const tb_bf16 *q_imp, const tb_bf16 *K_new, const tb_bf16 *V_new,
                                         const tb_bf16 *Wk, tb_bf16 *K, tb_bf16 *V, tb_bf16 *Kp,
                                         int32_t *idx_state, int64_t *n_pred, int64_t *proj_end, int32_t *sel,
                                         int32_t sel_stride, int32_t *counts, tb_bf16 *out, void *ws,
                                         size_t ws_bytes, int32_t *dev_status, cudaStream_t stream);

/*
 * tb_topk without a workspace. The paper has no counterpart to this call; it
 * exists for callers that cannot allocate device memory at all, so cannot
 * hand tb_topk its scratch: code embedded in a host runtime that owns every
 * device allocation and gives its plug-ins none, or a serving process whose
 * memory is fixed once at start-up.
 *
 * Same arguments and results as tb_topk (bit-identical idx), minus ws and
 * ws_bytes. The selection's scratch is a static device array compiled into
 * the library, sized for TB_TOPK_NOALLOC_MAX_ROWS rows of B*Hkv; every GPU
 * that loads the library holds it (about 3.9 MB) until the process exits.
 * The call allocates nothing: no cudaMalloc, no cudaFree, no allocating
 * library routine. It clears the part of the array it uses (an asynchronous
 * memset on `stream`) before its kernel runs.
 *
 * Errors: B*Hkv > TB_TOPK_NOALLOC_MAX_ROWS returns TB_ERR_UNSUPPORTED; the
 * other checks and device-side errors are those of tb_topk.
 * The first call on each device looks up the array's device address
 * (cudaGetSymbolAddress, with that device current) and keeps it for the life
 * of the process; make that first call before any stream capture, and do not
 * use the library across a cudaDeviceReset (the kept address would then
 * point into the torn-down context). All calls on a device share the one array, so
 * calls that overlap on the GPU (concurrent streams, or several host threads)
 * race and give wrong results: serialise them.
 */
#define TB_TOPK_NOALLOC_MAX_ROWS 64

TB_API tb_status tb_topk_noalloc(const tb_shape *shape, const float *s, int64_t n, int32_t k, int32_t *idx,
                                 int32_t *dev_status, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* TB_H_ */
