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
#include "tb_internal.cuh"
#include "kernels.cuh"

namespace tb {

constexpr int kAttnThreads = 128;
constexpr int kUnroll = 4;
constexpr float kLog2e = 1.4426950408889634f;

template <int GM>
__global__ void __launch_bounds__(kAttnThreads)
attn_split_kernel(const uint16_t *__restrict__ q, const uint16_t *__restrict__ K, const uint16_t *__restrict__ V,
                  const int32_t *__restrict__ sel, const int32_t *__restrict__ counts, int32_t sel_stride,
                  int64_t cap, int Hq, int Hkv, int D, float scale, uint16_t *__restrict__ out,
                  uint32_t *__restrict__ attn_ctl, float *__restrict__ part, int32_t *dev_status) {
    const int G = Hq / Hkv;
    const int row = blockIdx.y;
    const int split = blockIdx.x;
    const int nsplit = gridDim.x;
    const int b = row / Hkv, h = row % Hkv;
    const int TPG = D / 8;                 // lanes per token
    const int groups_per_warp = 32 / TPG;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int gl = lane % TPG;             // lane within the group: dims [8*gl, 8*gl+8)
    const int grp = warp * groups_per_warp + lane / TPG;
    const int ngroups = (blockDim.x / 32) * groups_per_warp;

    extern __shared__ float sm[];
    // [ngroups][GM][2 + D] per-group partials, then merge scratch
    float *gpart = sm;

    // query (pre-scaled into the exp2 domain), this lane's 8 dims per head
    float qv[GM][8];
    const uint16_t *qrow = q + ((int64_t)b * Hq + (int64_t)h * G) * D;
#pragma unroll
    for (int g = 0; g < GM; ++g) {
        if (g < G) {
            uint4 w = *reinterpret_cast<const uint4 *>(qrow + (int64_t)g * D + 8 * gl);
            const float sc = scale * kLog2e;
            qv[g][0] = bf16_lo(w.x) * sc; qv[g][1] = bf16_hi(w.x) * sc;
            qv[g][2] = bf16_lo(w.y) * sc; qv[g][3] = bf16_hi(w.y) * sc;
            qv[g][4] = bf16_lo(w.z) * sc; qv[g][5] = bf16_hi(w.z) * sc;
            qv[g][6] = bf16_lo(w.w) * sc; qv[g][7] = bf16_hi(w.w) * sc;
        } else {
#pragma unroll
            for (int j = 0; j < 8; ++j) qv[g][j] = 0.f;
        }
    }
    float m[GM], l[GM], acc[GM][8];
#pragma unroll
    for (int g = 0; g < GM; ++g) {
        m[g] = -INFINITY;
        l[g] = 0.f;
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[g][j] = 0.f;
    }

    const int cnt = counts ? counts[row] : sel_stride;
    const int cnt_c = cnt < 0 ? 0 : (cnt > sel_stride ? sel_stride : cnt);
    if (threadIdx.x == 0 && split == 0 && (cnt <= 0 || cnt > sel_stride)) set_status(dev_status, TB_ERR_INVALID_ARG);
    const int j0 = split * kAttnSplitTok;
    const int j1 = min(j0 + kAttnSplitTok, cnt_c);
    const int32_t *srow = sel + (int64_t)row * sel_stride;
    const uint16_t *Kh = K + (int64_t)row * cap * D;
    const uint16_t *Vh = V + (int64_t)row * cap * D;

    // The loop bound depends on the warp only (all lanes of a warp iterate
    // together: the group reductions below are warp shuffles).
    const int gi = lane / TPG;
    for (int jw = j0 + warp * groups_per_warp; jw < j1; jw += ngroups * kUnroll) {
        uint4 kv[kUnroll], vv[kUnroll];
        bool valid[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int j = jw + gi + u * ngroups;
            valid[u] = false;
            if (j < j1) {
                const int32_t t = __ldg(srow + j);
                if (t >= 0 && (int64_t)t < cap) {
                    valid[u] = true;
                    kv[u] = __ldcs(reinterpret_cast<const uint4 *>(Kh + (int64_t)t * D + 8 * gl));
                    vv[u] = __ldcs(reinterpret_cast<const uint4 *>(Vh + (int64_t)t * D + 8 * gl));
                } else {
                    set_status(dev_status, TB_ERR_INVALID_ARG);
                }
            }
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            float kf[8];
            if (valid[u]) {
                kf[0] = bf16_lo(kv[u].x); kf[1] = bf16_hi(kv[u].x);
                kf[2] = bf16_lo(kv[u].y); kf[3] = bf16_hi(kv[u].y);
                kf[4] = bf16_lo(kv[u].z); kf[5] = bf16_hi(kv[u].z);
                kf[6] = bf16_lo(kv[u].w); kf[7] = bf16_hi(kv[u].w);
            } else {
#pragma unroll
                for (int j = 0; j < 8; ++j) kf[j] = 0.f;
            }
            float z[GM];
#pragma unroll
            for (int g = 0; g < GM; ++g) {
                float a = 0.f;
#pragma unroll
                for (int j = 0; j < 8; ++j) a = fmaf(qv[g][j], kf[j], a);
                z[g] = a;
            }
            // reduce the partial dot products across the TPG lanes of the group
            for (int o = TPG / 2; o > 0; o >>= 1) {
#pragma unroll
                for (int g = 0; g < GM; ++g) z[g] += __shfl_xor_sync(0xFFFFFFFFu, z[g], o);
            }
            if (valid[u]) {
                float vf[8];
                vf[0] = bf16_lo(vv[u].x); vf[1] = bf16_hi(vv[u].x);
                vf[2] = bf16_lo(vv[u].y); vf[3] = bf16_hi(vv[u].y);
                vf[4] = bf16_lo(vv[u].z); vf[5] = bf16_hi(vv[u].z);
                vf[6] = bf16_lo(vv[u].w); vf[7] = bf16_hi(vv[u].w);
#pragma unroll
                for (int g = 0; g < GM; ++g) {
                    if (g < G) {
                        const float mn = fmaxf(m[g], z[g]);
                        const float corr = exp2f(m[g] - mn);   // 0 when m was -inf
                        const float p = exp2f(z[g] - mn);
                        l[g] = l[g] * corr + p;
#pragma unroll
                        for (int j = 0; j < 8; ++j) acc[g][j] = fmaf(acc[g][j], corr, p * vf[j]);
                        m[g] = mn;
                    }
                }
            }
        }
    }

    // ---- combine the groups of this CTA
    const int stride_g = 2 + D;
#pragma unroll
    for (int g = 0; g < GM; ++g) {
        if (g < G) {
            float *dst = gpart + ((int64_t)grp * G + g) * stride_g;
            if (gl == 0) {
                dst[0] = m[g];
                dst[1] = l[g];
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) dst[2 + 8 * gl + j] = acc[g][j];
        }
    }
    __syncthreads();
    float *prow = part + (((int64_t)row * nsplit + split) * G) * stride_g;
    for (int x = threadIdx.x; x < G * D; x += blockDim.x) {
        const int g = x / D, d = x % D;
        float M = -INFINITY;
        for (int p = 0; p < ngroups; ++p) M = fmaxf(M, gpart[((int64_t)p * G + g) * stride_g]);
        float L = 0.f, A = 0.f;
        if (M != -INFINITY) {
            for (int p = 0; p < ngroups; ++p) {
                const float *src = gpart + ((int64_t)p * G + g) * stride_g;
                const float w = exp2f(src[0] - M);
                L += w * src[1];
                A += w * src[2 + d];
            }
        }
        float *dst = prow + (int64_t)g * stride_g;
        if (d == 0) {
            dst[0] = M;
            dst[1] = L;
        }
        dst[2 + d] = A;
    }

    // ---- last CTA of the row merges the splits
    __shared__ uint32_t last;
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        const uint32_t prev = atomicAdd(attn_ctl + row, 1u);
        last = (prev == (uint32_t)(nsplit - 1)) ? 1u : 0u;
    }
    __syncthreads();
    if (!last) return;
    __threadfence();
    const float *pr = part + ((int64_t)row * nsplit * G) * stride_g;
    for (int x = threadIdx.x; x < G * D; x += blockDim.x) {
        const int g = x / D, d = x % D;
        float M = -INFINITY;
        for (int sp = 0; sp < nsplit; ++sp) M = fmaxf(M, __ldcg(pr + ((int64_t)sp * G + g) * stride_g));
        float L = 0.f, A = 0.f;
        if (M != -INFINITY) {
            for (int sp = 0; sp < nsplit; ++sp) {
                const float *src = pr + ((int64_t)sp * G + g) * stride_g;
                const float w = exp2f(__ldcg(src) - M);
                L += w * __ldcg(src + 1);
                A += w * __ldcg(src + 2 + d);
            }
        }
        const float o = L > 0.f ? A / L : 0.f;
        out[((int64_t)b * Hq + (int64_t)h * G + g) * D + d] = f_to_bf16(o);
    }
    if (threadIdx.x == 0) attn_ctl[row] = 0;   // ready for the next call
}

cudaError_t launch_attn(const tb_shape &sh, const uint16_t *q, const uint16_t *K, const uint16_t *V,
                        const int32_t *sel, const int32_t *counts, int32_t sel_stride, float scale, uint16_t *out,
                        uint32_t *attn_ctl, float *partials, int32_t *dev_status, cudaStream_t st) {
    const int rows = sh.B * sh.Hkv;
    const int G = sh.Hq / sh.Hkv;
    if (rows <= 0) return cudaSuccess;
    const int64_t nsplit = attn_splits(sel_stride);
    dim3 grid((unsigned)nsplit, (unsigned)rows);
    const int TPG = sh.D / 8;
    const int ngroups = (kAttnThreads / 32) * (32 / TPG);
    const size_t smem = (size_t)ngroups * G * (2 + sh.D) * sizeof(float);
    if (smem > 48 * 1024) {
        // G * D large: allow the larger carve-out once per instantiation
        cudaFuncSetAttribute(attn_split_kernel<16>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        cudaFuncSetAttribute(attn_split_kernel<8>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    }
#define TB_ATTN_CASE(GMC)                                                                                      \
    attn_split_kernel<GMC><<<grid, kAttnThreads, smem, st>>>(q, K, V, sel, counts, sel_stride, sh.cap, sh.Hq, \
                                                            sh.Hkv, sh.D, scale, out, attn_ctl, partials,     \
                                                            dev_status)
    if (G <= 1) TB_ATTN_CASE(1);
    else if (G <= 2) TB_ATTN_CASE(2);
    else if (G <= 4) TB_ATTN_CASE(4);
    else if (G <= 8) TB_ATTN_CASE(8);
    else TB_ATTN_CASE(16);
#undef TB_ATTN_CASE
    return cudaGetLastError();
}

}  // namespace tb
