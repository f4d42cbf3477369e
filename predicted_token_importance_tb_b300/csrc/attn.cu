// Exact attention over the selected K/V rows ("TokenButler: Token Importance
// is Predictable": the full cache stays resident and only the selected tokens
// are read).
//
// Split-N decode attention with an online softmax. Grid = (splits, rows);
// a CTA takes kAttnSplitTok consecutive entries of its row's selection. A
// group of D/8 lanes owns one token at a time: each lane loads 16 bytes of
// the K row and 16 bytes of the V row (a group reads the 2*2*D bytes of a
// token as two contiguous segments), and kUnroll tokens per group are in
// flight before any of them is used. The G query heads of the KV head are
// served from the same gathered rows. Partial (max, sum, acc[D]) per split go
// to the workspace; the last CTA of a row to finish merges them.
#include "attn_core.cuh"
#include "kernels.cuh"

namespace tb {

constexpr int kAttnThreads = 128;

template <int GM>
__global__ void __launch_bounds__(kAttnThreads)
attn_split_kernel(const uint16_t *__restrict__ q, const uint16_t *__restrict__ K, const uint16_t *__restrict__ V,
                  const int32_t *__restrict__ sel, const int32_t *__restrict__ counts, int32_t sel_stride,
                  int64_t cap, int Hq, int Hkv, int D, float scale, uint16_t *__restrict__ out,
                  uint32_t *__restrict__ attn_ctl, float *__restrict__ part, int split_tok, int32_t *dev_status) {
    extern __shared__ float comb[];   // [warps][G][2 + D], later the merge scratch
    __shared__ uint32_t last;
    const int G = Hq / Hkv;
    const int row = blockIdx.y;
    const int split = blockIdx.x;
    const int nsplit = gridDim.x;
    const int b = row / Hkv, h = row % Hkv;
    const int gl = (threadIdx.x & 31) % (D / 8);

    const int cnt = counts ? counts[row] : sel_stride;
    const int cnt_c = cnt < 0 ? 0 : (cnt > sel_stride ? sel_stride : cnt);
    if (threadIdx.x == 0 && split == 0 && (cnt <= 0 || cnt > sel_stride)) set_status(dev_status, TB_ERR_INVALID_ARG);
    const int j0 = split * split_tok;
    const int j1 = min(j0 + split_tok, cnt_c);
    const int32_t *srow = sel + (int64_t)row * sel_stride + j0;

    AttnLane<GM> A;
    attn_init(A, q + ((int64_t)b * Hq + (int64_t)h * G) * D, G, D, gl, scale);
    attn_tokens(A, G, D, j1 > j0 ? j1 - j0 : 0, [&](int j) -> int64_t {
        const int32_t t = __ldg(srow + j);
        return t < 0 ? (int64_t)-2 : (int64_t)t;   // a negative entry is invalid, not a skip
    }, K + (int64_t)row * cap * D, V + (int64_t)row * cap * D, cap, dev_status);

    const int sg = 2 + D;
    float *prow = part + (int64_t)row * nsplit * G * sg;
    attn_block_combine(A, G, D, comb, prow + (int64_t)split * G * sg);

    // the last CTA of the row merges the splits
    if (threadIdx.x == 0) {
        __threadfence();
        const uint32_t prev = atomicAdd(attn_ctl + row, 1u);
        last = (prev == (uint32_t)(nsplit - 1)) ? 1u : 0u;
    }
    __syncthreads();
    if (!last) return;
    __threadfence();
    attn_merge(prow, nsplit, G, D, out + ((int64_t)b * Hq + (int64_t)h * G) * D, dev_status, comb);
    if (threadIdx.x == 0) attn_ctl[row] = 0;   // ready for the next call
}

cudaError_t launch_attn(const tb_shape &sh, const uint16_t *q, const uint16_t *K, const uint16_t *V,
                        const int32_t *sel, const int32_t *counts, int32_t sel_stride, float scale, uint16_t *out,
                        uint32_t *attn_ctl, float *partials, int32_t *dev_status, cudaStream_t st) {
    const int rows = sh.B * sh.Hkv;
    const int G = sh.Hq / sh.Hkv;
    if (rows <= 0) return cudaSuccess;
    if (attn_stream_supported(sh) && kv_on_device(K, V))
        return launch_attn_stream(sh, q, K, V, sel, counts, sel_stride, scale, out, attn_ctl, partials, dev_status,
                                  st);
    if (attn_mma_supported(sh))
        return launch_attn_mma(sh, q, K, V, sel, counts, sel_stride, scale, out, attn_ctl, partials, dev_status, st);
    const int64_t nsplit = attn_splits(sel_stride);
    const int split_tok = (int)attn_split_tokens(sel_stride);
    dim3 grid((unsigned)nsplit, (unsigned)rows);
    size_t smem = (size_t)(kAttnThreads / 32) * G * (2 + sh.D) * sizeof(float);
    const size_t merge_smem = (size_t)(2 * nsplit * G + G) * sizeof(float);
    if (merge_smem > smem) smem = merge_smem;
    if (smem > 48 * 1024) {
        // G * D large: allow the larger carve-out once per instantiation
        cudaFuncSetAttribute(attn_split_kernel<16>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        cudaFuncSetAttribute(attn_split_kernel<8>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    }
#define TB_ATTN_CASE(GMC)                                                                                      \
    attn_split_kernel<GMC><<<grid, kAttnThreads, smem, st>>>(q, K, V, sel, counts, sel_stride, sh.cap, sh.Hq, \
                                                            sh.Hkv, sh.D, scale, out, attn_ctl, partials,     \
                                                            split_tok, dev_status)
    if (G <= 1) TB_ATTN_CASE(1);
    else if (G <= 2) TB_ATTN_CASE(2);
    else if (G <= 4) TB_ATTN_CASE(4);
    else if (G <= 8) TB_ATTN_CASE(8);
    else TB_ATTN_CASE(16);
#undef TB_ATTN_CASE
    return cudaGetLastError();
}

}  // namespace tb
