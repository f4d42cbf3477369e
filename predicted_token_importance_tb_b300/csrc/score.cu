// Importance scores: s[b,h,t] = agg_g q_imp[b,h*G+g,:] . Kp[b,h,t,:]
// ("TokenButler: Token Importance is Predictable", gist.science summary,
// Core Architecture, Scoring).
//
// HBM-bound stream of Kp (2*dp bytes per token). One thread per token; each
// thread reads its dp/8 16-byte vectors (consecutive threads read
// consecutive rows, so a warp's loads cover one contiguous span). The G
// importance queries of the KV head sit in shared memory as fp32; with the
// mean aggregation they are folded into their group mean first (the mean of
// dot products equals the dot product with the mean query).
#include "tb_internal.cuh"
#include "kernels.cuh"

namespace tb {

constexpr int kScoreThreads = 256;

template <int NV>
__device__ __forceinline__ void load_row(const uint4 *p, uint4 (&v)[NV]) {
#pragma unroll
    for (int i = 0; i < NV; ++i) v[i] = __ldcs(p + i);
}

__device__ __forceinline__ float dot8(const float *q, uint4 v, float acc) {
    acc = fmaf(q[0], bf16_lo(v.x), acc);
    acc = fmaf(q[1], bf16_hi(v.x), acc);
    acc = fmaf(q[2], bf16_lo(v.y), acc);
    acc = fmaf(q[3], bf16_hi(v.y), acc);
    acc = fmaf(q[4], bf16_lo(v.z), acc);
    acc = fmaf(q[5], bf16_hi(v.z), acc);
    acc = fmaf(q[6], bf16_lo(v.w), acc);
    acc = fmaf(q[7], bf16_hi(v.w), acc);
    return acc;
}

// NV = dp/8 known at compile time (0: runtime nv).
template <int NV>
__global__ void __launch_bounds__(kScoreThreads)
score_kernel(const uint16_t *__restrict__ q_imp, const uint16_t *__restrict__ Kp, int64_t cap, int64_t n,
             int Hq, int Hkv, int dp, int agg, float *__restrict__ s, int64_t lds, const int64_t *__restrict__ n_seq) {
    extern __shared__ float qs[];   // [G][dp] (MAX) or [dp] (MEAN)
    const int row = blockIdx.y;
    const int b = row / Hkv, h = row % Hkv;
    const int G = Hq / Hkv;
    const uint16_t *qrow = q_imp + ((int64_t)b * Hq + (int64_t)h * G) * dp;
    if (agg == TB_AGG_MEAN) {
        const float inv = 1.0f / (float)G;
        for (int i = threadIdx.x; i < dp; i += blockDim.x) {
            float a = 0.f;
            for (int g = 0; g < G; ++g) a += bf16_to_f(qrow[g * dp + i]);
            qs[i] = a * inv;
        }
    } else {
        for (int i = threadIdx.x; i < G * dp; i += blockDim.x) qs[i] = bf16_to_f(qrow[i]);
    }
    __syncthreads();
    const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= n) return;
    if (n_seq && t > n_seq[b]) {   // beyond this sequence's tokens (n_seq[b] + 1 of them): never selected
        s[(int64_t)row * lds + t] = -INFINITY;
        return;
    }
    const int nv = NV > 0 ? NV : dp / 8;
    const uint4 *p = reinterpret_cast<const uint4 *>(Kp + ((int64_t)row * cap + t) * dp);
    float out;
    constexpr int NVX = NV > 0 ? NV : 1;
    if (NV > 0) {
        uint4 v[NVX];
        load_row<NVX>(p, v);
        if (agg == TB_AGG_MEAN) {
            float acc = 0.f;
#pragma unroll
            for (int i = 0; i < NVX; ++i) acc = dot8(qs + 8 * i, v[i], acc);
            out = acc;
        } else {
            out = -INFINITY;
            for (int g = 0; g < G; ++g) {
                float acc = 0.f;
#pragma unroll
                for (int i = 0; i < NVX; ++i) acc = dot8(qs + g * dp + 8 * i, v[i], acc);
                out = fmaxf(out, acc);
            }
        }
    } else {
        if (agg == TB_AGG_MEAN) {
            float acc = 0.f;
            for (int i = 0; i < nv; ++i) acc = dot8(qs + 8 * i, __ldcs(p + i), acc);
            out = acc;
        } else {
            out = -INFINITY;
            for (int g = 0; g < G; ++g) {
                float acc = 0.f;
                for (int i = 0; i < nv; ++i) acc = dot8(qs + g * dp + 8 * i, __ldcs(p + i), acc);
                out = fmaxf(out, acc);
            }
        }
    }
    s[(int64_t)row * lds + t] = out;
}

cudaError_t launch_score(const tb_shape &sh, const uint16_t *q_imp, const uint16_t *Kp, int64_t n, int agg,
                         float *s, int64_t lds, cudaStream_t st, const int64_t *n_seq) {
    const int rows = sh.B * sh.Hkv;
    if (n <= 0 || rows <= 0) return cudaSuccess;
    const int G = sh.Hq / sh.Hkv;
    dim3 grid((unsigned)((n + kScoreThreads - 1) / kScoreThreads), (unsigned)rows);
    size_t smem = (size_t)(agg == TB_AGG_MEAN ? 1 : G) * sh.dp * sizeof(float);
    const int nv = sh.dp / 8;
#define TB_SCORE_CASE(NVC)                                                                                 \
    case NVC:                                                                                              \
        score_kernel<NVC><<<grid, kScoreThreads, smem, st>>>(q_imp, Kp, sh.cap, n, sh.Hq, sh.Hkv, sh.dp, agg, \
                                                             s, lds, n_seq);                                      \
        break;
    switch (nv) {
        TB_SCORE_CASE(1)
        TB_SCORE_CASE(2)
        TB_SCORE_CASE(4)
        TB_SCORE_CASE(8)
        default:
            score_kernel<0><<<grid, kScoreThreads, smem, st>>>(q_imp, Kp, sh.cap, n, sh.Hq, sh.Hkv, sh.dp, agg, s,
                                                               lds, n_seq);
    }
#undef TB_SCORE_CASE
    return cudaGetLastError();
}

}  // namespace tb
