// Gather-attention building blocks shared by the split attention kernel and
// the fused decode step ("TokenButler: Token Importance is Predictable":
// exact attention over only the selected full-precision K/V rows).
//
// A group of TPG = D/8 lanes owns one token at a time; lane gl of the group
// holds dims [8*gl, 8*gl+8) of the query heads, of the K row it scores and
// of the V row it accumulates. Each group keeps an online-softmax state
// (running max m, sum l, acc[8]) per query head in the exp2 domain (the
// query is pre-scaled by scale*log2(e)). States of groups, CTAs and splits
// merge with the usual rescaling by exp2(m_i - max).
#pragma once

#include "tb_internal.cuh"

namespace tb {

constexpr int kAttnUnroll = 4;             // tokens per group in flight
constexpr float kLog2e = 1.4426950408889634f;

template <int GM>
struct AttnLane {
    float qv[GM][8];
    float m[GM], l[GM], acc[GM][8];
};

__device__ __forceinline__ float rescale_w(float m, float M) { return m == -INFINITY ? 0.f : exp2f(m - M); }

__device__ __forceinline__ void unpack8(uint4 v, float (&f)[8]) {
    f[0] = bf16_lo(v.x); f[1] = bf16_hi(v.x);
    f[2] = bf16_lo(v.y); f[3] = bf16_hi(v.y);
    f[4] = bf16_lo(v.z); f[5] = bf16_hi(v.z);
    f[6] = bf16_lo(v.w); f[7] = bf16_hi(v.w);
}

// qrow: the G query rows of this KV head ([G][D] bf16).
template <int GM>
__device__ __forceinline__ void attn_init(AttnLane<GM> &A, const uint16_t *qrow, int G, int D, int gl, float scale) {
    const float sc = scale * kLog2e;
#pragma unroll
    for (int g = 0; g < GM; ++g) {
        if (g < G) {
            float f[8];
            unpack8(*reinterpret_cast<const uint4 *>(qrow + (int64_t)g * D + 8 * gl), f);
#pragma unroll
            for (int j = 0; j < 8; ++j) A.qv[g][j] = f[j] * sc;
        } else {
#pragma unroll
            for (int j = 0; j < 8; ++j) A.qv[g][j] = 0.f;
        }
        A.m[g] = -INFINITY;
        A.l[g] = 0.f;
#pragma unroll
        for (int j = 0; j < 8; ++j) A.acc[g][j] = 0.f;
    }
}

// Attend entries j in [0, cnt) of a token list; tok(j) gives the cache row
// (or a negative value to skip it). All lanes of a warp run the same number of
// iterations (the dot products are reduced with warp shuffles).
template <int GM, class TokFn>
__device__ __forceinline__ void attn_tokens(AttnLane<GM> &A, int G, int D, int cnt, TokFn tok, const uint16_t *Kh,
                                            const uint16_t *Vh, int64_t cap, int32_t *dev_status) {
    const int TPG = D / 8;
    const int gpw = 32 / TPG;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int gi = lane / TPG, gl = lane % TPG;
    const int ngroups = (blockDim.x >> 5) * gpw;
    for (int jw = warp * gpw; jw < cnt; jw += ngroups * kAttnUnroll) {
        uint4 kv[kAttnUnroll], vv[kAttnUnroll];
        bool valid[kAttnUnroll];
#pragma unroll
        for (int u = 0; u < kAttnUnroll; ++u) {
            const int j = jw + gi + u * ngroups;
            valid[u] = false;
            if (j < cnt) {
                const int64_t t = tok(j);
                if (t >= 0 && t < cap) {
                    valid[u] = true;
                    kv[u] = __ldcs(reinterpret_cast<const uint4 *>(Kh + t * D + 8 * gl));
                    vv[u] = __ldcs(reinterpret_cast<const uint4 *>(Vh + t * D + 8 * gl));
                } else if (t != -1) {
                    set_status(dev_status, TB_ERR_INVALID_ARG);
                }
            }
        }
#pragma unroll
        for (int u = 0; u < kAttnUnroll; ++u) {
            float kf[8];
            if (valid[u]) {
                unpack8(kv[u], kf);
            } else {
#pragma unroll
                for (int j = 0; j < 8; ++j) kf[j] = 0.f;
            }
            float z[GM];
#pragma unroll
            for (int g = 0; g < GM; ++g) {
                float a = 0.f;
#pragma unroll
                for (int j = 0; j < 8; ++j) a = fmaf(A.qv[g][j], kf[j], a);
                z[g] = a;
            }
            for (int o = TPG / 2; o > 0; o >>= 1) {
#pragma unroll
                for (int g = 0; g < GM; ++g) z[g] += __shfl_xor_sync(0xFFFFFFFFu, z[g], o);
            }
            if (valid[u]) {
                float vf[8];
                unpack8(vv[u], vf);
#pragma unroll
                for (int g = 0; g < GM; ++g) {
                    if (g < G) {
                        const float mn = fmaxf(A.m[g], z[g]);
                        const float corr = exp2f(A.m[g] - mn);   // 0 while m is -inf
                        const float p = exp2f(z[g] - mn);
                        A.l[g] = fmaf(A.l[g], corr, p);
#pragma unroll
                        for (int j = 0; j < 8; ++j) A.acc[g][j] = fmaf(A.acc[g][j], corr, p * vf[j]);
                        A.m[g] = mn;
                    }
                }
            }
        }
    }
}

// Attend rows already staged in shared memory: row(j) points at the K row of
// entry j (D bf16), its V row follows at +D. Same lane layout and warp rule
// as attn_tokens.
template <int GM, class RowFn>
__device__ __forceinline__ void attn_stage_rows(AttnLane<GM> &A, int G, int D, int cnt, RowFn row) {
    const int TPG = D / 8;
    const int gpw = 32 / TPG;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int gi = lane / TPG, gl = lane % TPG;
    const int ngroups = (blockDim.x >> 5) * gpw;
    for (int jw = warp * gpw; jw < cnt; jw += ngroups) {
        const int j = jw + gi;
        const bool valid = j < cnt;
        float kf[8];
        uint4 vv = make_uint4(0, 0, 0, 0);
        if (valid) {
            const uint16_t *r = row(j);
            unpack8(*reinterpret_cast<const uint4 *>(r + 8 * gl), kf);
            vv = *reinterpret_cast<const uint4 *>(r + D + 8 * gl);
        } else {
#pragma unroll
            for (int x = 0; x < 8; ++x) kf[x] = 0.f;
        }
        float z[GM];
#pragma unroll
        for (int g = 0; g < GM; ++g) {
            float acc = 0.f;
#pragma unroll
            for (int x = 0; x < 8; ++x) acc = fmaf(A.qv[g][x], kf[x], acc);
            z[g] = acc;
        }
        for (int o = TPG / 2; o > 0; o >>= 1) {
#pragma unroll
            for (int g = 0; g < GM; ++g) z[g] += __shfl_xor_sync(0xFFFFFFFFu, z[g], o);
        }
        if (valid) {
            float vf[8];
            unpack8(vv, vf);
#pragma unroll
            for (int g = 0; g < GM; ++g) {
                if (g < G) {
                    const float mn = fmaxf(A.m[g], z[g]);
                    const float corr = exp2f(A.m[g] - mn);
                    const float p = exp2f(z[g] - mn);
                    A.l[g] = fmaf(A.l[g], corr, p);
#pragma unroll
                    for (int x = 0; x < 8; ++x) A.acc[g][x] = fmaf(A.acc[g][x], corr, p * vf[x]);
                    A.m[g] = mn;
                }
            }
        }
    }
}

// Merge the lane groups of the CTA into one partial state per query head and
// store it at dst[g * (2 + D)] = (m, l, acc[D]). comb: shared scratch of
// (blockDim/32) * G * (2 + D) floats. All threads must call it.
template <int GM>
__device__ __forceinline__ void attn_block_combine(AttnLane<GM> &A, int G, int D, float *comb, float *dst) {
    const int TPG = D / 8;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    const int gl = lane % TPG;
    // groups of one warp: butterfly over the group index
    for (int o = TPG; o < 32; o <<= 1) {
#pragma unroll
        for (int g = 0; g < GM; ++g) {
            const float mo = __shfl_xor_sync(0xFFFFFFFFu, A.m[g], o);
            const float lo = __shfl_xor_sync(0xFFFFFFFFu, A.l[g], o);
            const float M = fmaxf(A.m[g], mo);
            const float w1 = rescale_w(A.m[g], M), w2 = rescale_w(mo, M);
            A.l[g] = A.l[g] * w1 + lo * w2;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const float ao = __shfl_xor_sync(0xFFFFFFFFu, A.acc[g][j], o);
                A.acc[g][j] = A.acc[g][j] * w1 + ao * w2;
            }
            A.m[g] = M;
        }
    }
    const int sg = 2 + D;
    if (lane < TPG) {
#pragma unroll
        for (int g = 0; g < GM; ++g) {
            if (g < G) {
                float *c = comb + ((int64_t)warp * G + g) * sg;
                if (gl == 0) {
                    c[0] = A.m[g];
                    c[1] = A.l[g];
                }
#pragma unroll
                for (int j = 0; j < 8; ++j) c[2 + 8 * gl + j] = A.acc[g][j];
            }
        }
    }
    __syncthreads();
    for (int x = threadIdx.x; x < G * D; x += blockDim.x) {
        const int g = x / D, d = x % D;
        float M = -INFINITY;
        for (int w = 0; w < nw; ++w) M = fmaxf(M, comb[((int64_t)w * G + g) * sg]);
        float L = 0.f, Acc = 0.f;
        for (int w = 0; w < nw; ++w) {
            const float *c = comb + ((int64_t)w * G + g) * sg;
            const float wt = rescale_w(c[0], M);
            L += wt * c[1];
            Acc += wt * c[2 + d];
        }
        float *o = dst + (int64_t)g * sg;
        if (d == 0) {
            o[0] = M;
            o[1] = L;
        }
        o[2 + d] = Acc;
    }
    __syncthreads();
}

// Merge nsplit partial states (each G x (2 + D) floats, consecutive) into the
// G output rows (bf16). sm: shared scratch of 2 * nsplit * G + G floats.
// Each thread first issues the loads of its outputs' accumulators for a batch
// of up to 32 splits, then the (max, sum) pairs go to shared memory with one
// load per thread, so a batch costs one L2 round trip. Records
// TB_ERR_INVALID_ARG when a row saw no token. All threads must call it.
__device__ __forceinline__ void attn_merge(const float *part, int nsplit, int G, int D, uint16_t *out_rows,
                                           int32_t *dev_status, float *sm) {
    constexpr int kBatch = 32;
    const int sg = 2 + D;
    float *ms = sm;                      // [nsplit * G] max
    float *ls = sm + nsplit * G;         // [nsplit * G] sums
    for (int x0 = 0; x0 < G * D; x0 += blockDim.x) {
        const int x = x0 + threadIdx.x;
        const bool active = x < G * D;
        const int g = active ? x / D : 0, d = active ? x % D : 0;
        float M = -INFINITY, L = 0.f, Acc = 0.f;
        for (int sp0 = 0; sp0 < nsplit; sp0 += kBatch) {
            float av[kBatch];
#pragma unroll
            for (int u = 0; u < kBatch; ++u)
                av[u] = (active && sp0 + u < nsplit) ? __ldcg(part + ((int64_t)(sp0 + u) * G + g) * sg + 2 + d) : 0.f;
            __syncthreads();
            const int nb = nsplit - sp0 < kBatch ? nsplit - sp0 : kBatch;
            for (int i = threadIdx.x; i < nb * G; i += blockDim.x) {
                ms[i] = __ldcg(part + ((int64_t)sp0 * G + i) * sg);
                ls[i] = __ldcg(part + ((int64_t)sp0 * G + i) * sg + 1);
            }
            __syncthreads();
            float Mb = M;
            for (int u = 0; u < nb; ++u) Mb = fmaxf(Mb, ms[u * G + g]);
            const float r = rescale_w(M, Mb);
            L *= r;
            Acc *= r;
#pragma unroll
            for (int u = 0; u < kBatch; ++u) {
                if (u < nb) {
                    const float w = rescale_w(ms[u * G + g], Mb);
                    L = fmaf(w, ls[u * G + g], L);
                    Acc = fmaf(w, av[u], Acc);
                }
            }
            M = Mb;
        }
        if (active) {
            if (!(L > 0.f)) set_status(dev_status, TB_ERR_INVALID_ARG);
            out_rows[(int64_t)g * D + d] = f_to_bf16(L > 0.f ? Acc / L : 0.f);
        }
    }
}

}  // namespace tb
