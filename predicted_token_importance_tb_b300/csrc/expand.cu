// Neighbour fetching and the prediction-interval tail ("TokenButler: Token
// Importance is Predictable", gist.science summary, Optimizations:
// Prediction Interval & Neighbor Fetching), and the buffered step's selection
// (Inference Strategy): sink prefix, widened important tokens, local window.
//
// idx is strictly ascending, so the union of the windows [i-r, i+r] is a
// running merge: window j adds exactly the tokens in
// [max(i_j - r, i_{j-1} + r + 1, 0), min(i_j + r, n_pred - 1)]. One CTA per
// row counts those spans, scans the counts for output offsets and writes
// them, then appends the tail [n_pred, n_t). In general (launch_expand_ranges)
// the row is [0, prefix_end), then the windows of idx + idx_off clipped to
// [body_lo, body_hi), then [tail_start, n_t); the three ranges must be
// disjoint and ascending.
#include "tb_internal.cuh"
#include "kernels.cuh"

namespace tb {

constexpr int kExpandThreads = 1024;

__global__ void __launch_bounds__(kExpandThreads)
expand_kernel(const int32_t *__restrict__ idx, int32_t k, int32_t r, int64_t idx_off, int64_t prefix_end,
              int64_t body_lo, int64_t body_hi, int64_t tail_start, int64_t n_t, int32_t *__restrict__ sel,
              int32_t sel_stride, int32_t *__restrict__ counts, int32_t *dev_status, const int64_t *__restrict__ n_seq,
              int Hkv) {
    __shared__ uint32_t scan[33];
    const int row = blockIdx.x;
    if (n_seq) body_hi = tail_start = n_t = n_seq[row / Hkv] + 1;   // ragged batch at a prediction
    const int32_t *irow = idx + (int64_t)row * k;
    int32_t *srow = sel + (int64_t)row * sel_stride;
    // the prefix [0, prefix_end) first
    for (int64_t x = threadIdx.x; x < prefix_end; x += blockDim.x)
        if (x < (int64_t)sel_stride) srow[x] = (int32_t)x;
    uint32_t base = (uint32_t)prefix_end;
    bool bad = false;
    for (int j0 = 0; j0 < k; j0 += blockDim.x) {
        const int j = j0 + threadIdx.x;
        int64_t lo = 0, hi = -1;
        if (j < k) {
            const int64_t i = (int64_t)irow[j] + idx_off;
            const int64_t prev = j > 0 ? (int64_t)irow[j - 1] + idx_off : INT64_MIN / 4;
            if (i < body_lo || i >= body_hi || (j > 0 && i <= prev)) {
                bad = true;
            } else {
                lo = i - r;
                if (j > 0 && prev + r + 1 > lo) lo = prev + r + 1;
                if (lo < body_lo) lo = body_lo;
                hi = i + r;
                if (hi > body_hi - 1) hi = body_hi - 1;
            }
        }
        const uint32_t c = hi >= lo ? (uint32_t)(hi - lo + 1) : 0u;
        uint32_t tot;
        const uint32_t off = base + block_exclusive_scan(c, scan, tot);
        for (int64_t t = lo; t <= hi; ++t) {
            const uint64_t pos = off + (uint64_t)(t - lo);
            if (pos < (uint64_t)sel_stride) srow[pos] = (int32_t)t;
        }
        base += tot;
    }
    const int64_t tail = n_t > tail_start ? n_t - tail_start : 0;
    for (int64_t x = threadIdx.x; x < tail; x += blockDim.x) {
        const uint64_t pos = base + (uint64_t)x;
        if (pos < (uint64_t)sel_stride) srow[pos] = (int32_t)(tail_start + x);
    }
    const uint64_t total = base + (uint64_t)tail;
    if (bad) set_status(dev_status, TB_ERR_INVALID_ARG);
    if (threadIdx.x == 0) {
        if (total > (uint64_t)sel_stride) set_status(dev_status, TB_ERR_INVALID_ARG);
        counts[row] = (int32_t)(total > (uint64_t)sel_stride ? sel_stride : total);
    }
}

cudaError_t launch_expand(int rows, const int32_t *idx, int32_t k, int32_t r, int64_t n_pred, int64_t n_t,
                          int32_t *sel, int32_t sel_stride, int32_t *counts, int32_t *dev_status, cudaStream_t st) {
    return launch_expand_ranges(rows, idx, k, r, 0, 0, 0, n_pred, n_pred, n_t, sel, sel_stride, counts, dev_status,
                                st);
}

cudaError_t launch_expand_ragged(int rows, int Hkv, const int64_t *n_seq, const int32_t *idx, int32_t k, int32_t r,
                                 int32_t *sel, int32_t sel_stride, int32_t *counts, int32_t *dev_status,
                                 cudaStream_t st) {
    if (rows <= 0) return cudaSuccess;
    expand_kernel<<<rows, kExpandThreads, 0, st>>>(idx, k, r, 0, 0, 0, 0, 0, 0, sel, sel_stride, counts, dev_status,
                                                   n_seq, Hkv);
    return cudaGetLastError();
}

cudaError_t launch_expand_ranges(int rows, const int32_t *idx, int32_t k, int32_t r, int64_t idx_off,
                                 int64_t prefix_end, int64_t body_lo, int64_t body_hi, int64_t tail_start,
                                 int64_t n_t, int32_t *sel, int32_t sel_stride, int32_t *counts, int32_t *dev_status,
                                 cudaStream_t st) {
    if (rows <= 0) return cudaSuccess;
    expand_kernel<<<rows, kExpandThreads, 0, st>>>(idx, k, r, idx_off, prefix_end, body_lo, body_hi, tail_start, n_t,
                                                   sel, sel_stride, counts, dev_status, nullptr, 1);
    return cudaGetLastError();
}

}  // namespace tb
