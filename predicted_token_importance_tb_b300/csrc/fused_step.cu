// One decode step with a fresh prediction (interval T = 1, no neighbours) as a
// single cooperative launch ("TokenButler: Token Importance is Predictable":
// project the new key, score every cached token with the importance query,
// keep a fixed per-token budget, attend over only the kept full-precision
// rows).
//
// Grid = rows x C CTAs; CTA (row, c) owns tokens [c*L, c*L + L) of its
// (batch, KV head) row for the whole step:
//   1. the owner of token n appends K_new / V_new and projects K_new into Kp;
//   2. it streams its slice of Kp (16-byte loads, HBM-bound) into scores
//      held in shared memory as order-preserving keys;
//   3. the row's CTAs run the distributed radix select (topk_core.cuh);
//      after the threshold bin is known every CTA already gathers and
//      attends the tokens above it, hiding the last selection barrier;
//   4. each CTA writes its kept tokens (ascending) and attends the kept
//      tokens of the threshold bin, then stores one partial softmax state;
//   5. the last CTA of the row to finish merges the C partials into the
//      output rows and puts the row's control words back to zero.
// Scores never leave shared memory; the only global traffic besides the
// algorithmic bytes is the histogram/candidate exchange and the partials.
#include <string.h>

#include "fused_common.cuh"
#include "kernels.cuh"

namespace tb {

constexpr int kFusedThreads = 512;
constexpr int kFusedLMax = 8192;
constexpr int kFusedMaxSms = 160;        // workspace sizing headroom over the SM count
constexpr int kScoreUnroll = 4;

struct FusedArgs {
    const uint16_t *q, *q_imp, *K_new, *V_new, *Wk;
    uint16_t *K, *V, *Kp;
    int32_t *idx, *sel, *counts;
    uint16_t *out;
    RowCtl *ctl;
    float *part;
    int32_t *dev_status;
    int64_t cap, n;
    int Hq, Hkv, D, dp, k, agg, sel_stride;
    float scale;
    int C, L;
};

__host__ __device__ inline int comb_floats(int G, int D) { return comb_floats_for(kFusedThreads, G, D); }

__host__ __device__ inline size_t fused_smem_bytes(int L, int G, int D, int dp) {
    size_t b = (size_t)L * 4                       // keys
               + (size_t)kRadixBins * 4            // hist
               + (size_t)kCandCap * 8              // candidates
               + (size_t)kMaxChunks * 4            // per-chunk counts
               + 33 * 4 + 8 * 4 + 16               // scan, misc, abort flag
               + (size_t)L * 4                     // token list
               + (size_t)comb_floats(G, D) * 4     // group-combine scratch
               + (size_t)G * dp * 4                // importance query(s)
               + (size_t)dp * 4 + (size_t)D * 4;   // new key row (projected, raw)
    return (b + 15) / 16 * 16;
}

template <int NV, int GM>
__global__ void __launch_bounds__(kFusedThreads, 1)
fused_step_kernel(const FusedArgs a) {
    extern __shared__ __align__(16) uint8_t smem[];
    const int G = a.Hq / a.Hkv;
    const int L = a.L, C = a.C;
    const int row = blockIdx.x / C;
    const int c = blockIdx.x % C;
    const int b = row / a.Hkv, h = row % a.Hkv;
    const int64_t n_t = a.n + 1;
    const int64_t t0 = (int64_t)c * L;
    const int Lc = (int)((n_t - t0) < L ? (n_t - t0) : L);
    const int dp = NV > 0 ? NV * 8 : a.dp;
    const int D = a.D;

    // ---- shared memory
    SelectSmem S;
    uint32_t *p = reinterpret_cast<uint32_t *>(smem);
    S.keys = p; p += L;
    S.hist = p; p += kRadixBins;
    S.ckey = p; p += kCandCap;
    S.cidx = p; p += kCandCap;
    S.ccount = p; p += kMaxChunks;
    S.scan = p; p += 33;
    S.misc = p; p += 8;
    S.abort_flag = reinterpret_cast<int *>(p); p += 4;
    int32_t *list = reinterpret_cast<int32_t *>(p); p += L;
    float *comb = reinterpret_cast<float *>(p); p += comb_floats(G, D);
    float *qs = reinterpret_cast<float *>(p); p += G * dp;
    float *kpn = reinterpret_cast<float *>(p); p += dp;
    float *knew = reinterpret_cast<float *>(p);

    if (threadIdx.x == 0) *S.abort_flag = 0;

    // ---- importance query of this KV head
    const uint16_t *qi = a.q_imp + ((int64_t)b * a.Hq + (int64_t)h * G) * dp;
    if (a.agg == TB_AGG_MEAN) {
        const float inv = 1.0f / (float)G;
        for (int i = threadIdx.x; i < dp; i += blockDim.x) {
            float s = 0.f;
            for (int g = 0; g < G; ++g) s += bf16_to_f(qi[g * dp + i]);
            qs[i] = s * inv;
        }
    } else {
        for (int i = threadIdx.x; i < G * dp; i += blockDim.x) qs[i] = bf16_to_f(qi[i]);
    }

    // ---- 1. append (the CTA owning token n)
    const bool owner = a.n >= t0 && a.n < t0 + Lc;
    const uint16_t *Kh = a.K + (int64_t)row * a.cap * D;
    const uint16_t *Vh = a.V + (int64_t)row * a.cap * D;
    if (owner) step_append_project(a.K_new, a.V_new, a.Wk, a.K, a.V, a.Kp, a.cap, a.n, row, h, D, dp, knew, kpn, comb);
    __syncthreads();

    // ---- 2. scores of this chunk -> keys in shared memory
    // Each thread issues the loads of up to kScoreUnroll tokens before using
    // any of them, so a CTA keeps its whole slice of Kp in flight.
    bool nan_seen = false;
    {
        const uint16_t *Kpr = a.Kp + ((int64_t)row * a.cap + t0) * dp;
        if (NV > 0 && a.agg == TB_AGG_MEAN) {
            constexpr int NVX = NV > 0 ? NV : 1;
            constexpr int U = kScoreUnroll;
            for (int e0 = threadIdx.x; e0 < Lc; e0 += U * blockDim.x) {
                uint4 v[U][NVX];
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int e = e0 + u * blockDim.x;
                    if (e < Lc && t0 + e != a.n) {
                        const uint4 *src = reinterpret_cast<const uint4 *>(Kpr + (int64_t)e * dp);
#pragma unroll
                        for (int i = 0; i < NVX; ++i) v[u][i] = __ldcs(src + i);
                    }
                }
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int e = e0 + u * blockDim.x;
                    if (e < Lc) {
                        float sc = 0.f;
                        if (t0 + e == a.n) {
                            for (int i = 0; i < dp; ++i) sc = fmaf(qs[i], kpn[i], sc);
                        } else {
#pragma unroll
                            for (int i = 0; i < NVX; ++i) {
                                float f[8];
                                unpack8(v[u][i], f);
#pragma unroll
                                for (int x = 0; x < 8; ++x) sc = fmaf(qs[8 * i + x], f[x], sc);
                            }
                        }
                        S.keys[e] = score_key(sc, nan_seen);
                    }
                }
            }
        } else {
            // general dp / max aggregation: one token per thread at a time
            const int nv = dp / 8;
            for (int e = threadIdx.x; e < Lc; e += blockDim.x) {
                const int64_t t = t0 + e;
                const uint4 *src = reinterpret_cast<const uint4 *>(Kpr + (int64_t)e * dp);
                float sc = -INFINITY;
                const int ng = a.agg == TB_AGG_MEAN ? 1 : G;
                for (int g = 0; g < ng; ++g) {
                    float s2 = 0.f;
                    for (int i = 0; i < nv; ++i) {
                        float f[8];
                        if (t == a.n) {
#pragma unroll
                            for (int x = 0; x < 8; ++x) f[x] = kpn[8 * i + x];
                        } else {
                            unpack8(__ldcs(src + i), f);
                        }
#pragma unroll
                        for (int x = 0; x < 8; ++x) s2 = fmaf(qs[g * dp + 8 * i + x], f[x], s2);
                    }
                    sc = fmaxf(sc, s2);
                }
                S.keys[e] = score_key(sc, nan_seen);
            }
        }
    }
    if (nan_seen) set_status(a.dev_status, TB_ERR_NONFINITE);
    __syncthreads();

    // ---- 3-4. exact selection; attention over this chunk's kept tokens
    RowCtl *rc = a.ctl + row;
    const int TPG = D / 8;
    const int gl = (threadIdx.x & 31) % TPG;
    AttnLane<GM> A;
    attn_init(A, a.q + ((int64_t)b * a.Hq + (int64_t)h * G) * D, G, D, gl, a.scale);
    if (!chunk_select_attend(A, rc, S, list, Lc, L, c, C, 0, (uint32_t)a.k, t0, Kh, Vh, a.cap, G, D,
                             a.idx + (int64_t)row * a.k, a.sel + (int64_t)row * a.sel_stride, a.dev_status))
        return;
    if (c == 0 && threadIdx.x == 0) a.counts[row] = a.k;

    // ---- 5. partial state; the row's last CTA merges and resets the row
    row_finish(A, rc, a.part + (int64_t)row * C * G * (2 + D), c, C, G, D,
               a.out + ((int64_t)b * a.Hq + (int64_t)h * G) * D, comb, reinterpret_cast<float *>(S.ckey), &S.misc[6],
               true, a.dev_status);
}

// ------------------------------------------------------------------ host side

struct FusedPlan {
    int C = 0, L = 0;
    size_t smem = 0;
};

template <int NV, int GM>
static int fused_blocks_per_sm(size_t smem) {
    cudaFuncSetAttribute(fused_step_kernel<NV, GM>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    int per = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, fused_step_kernel<NV, GM>, kFusedThreads, smem) !=
        cudaSuccess)
        return 0;
    return per;
}

static int group_max(int G) { return G <= 1 ? 1 : G <= 2 ? 2 : G <= 4 ? 4 : G <= 8 ? 8 : 16; }

// Largest number of CTAs per row the GPU can keep resident for this shape.
static FusedPlan plan_fused(const tb_shape &sh, int64_t n_tokens, int sms, int blocks_per_sm) {
    FusedPlan P;
    const int rows = sh.B * sh.Hkv;
    const int G = sh.Hq / sh.Hkv;
    int64_t C = (int64_t)blocks_per_sm * sms / rows;
    const int64_t maxC = (n_tokens + 31) / 32;
    // the merge keeps 2 * C * G + G floats in the candidate area (2 * kCandCap words)
    const int64_t maxC_merge = (2 * kCandCap - G) / (2 * G);
    if (C > maxC_merge) C = maxC_merge;
    if (C > maxC) C = maxC;
    if (C > kMaxChunks) C = kMaxChunks;
    if (C < 1) return P;
    int64_t L = (n_tokens + C - 1) / C;
    L = (L + 31) / 32 * 32;
    if (L > kFusedLMax) return P;
    C = (n_tokens + L - 1) / L;
    P.C = (int)C;
    P.L = (int)L;
    P.smem = fused_smem_bytes(P.L, G, sh.D, sh.dp);
    return P;
}

int64_t fused_chunks(const tb_shape &sh, int64_t n_tokens) {
    // upper bound used to size the workspace: two CTAs per SM on a large part
    const int rows = sh.B * sh.Hkv;
    int64_t C = 2LL * kFusedMaxSms / (rows > 0 ? rows : 1);
    const int64_t maxC = (n_tokens + 31) / 32;
    if (C > maxC) C = maxC;
    if (C > kMaxChunks) C = kMaxChunks;
    return C < 1 ? 1 : C;
}

static bool resolve_plan_uncached(const tb_shape &sh, int64_t n_tokens, FusedPlan &P, int &nvsel, int &gm);

// Resolve the launch plan for this device; the last answer is cached (a
// decode loop asks the same question every step).
static bool resolve_plan(const tb_shape &sh, int64_t n_tokens, FusedPlan &P, int &nvsel, int &gm) {
    struct Key {
        int dev, B, Hq, Hkv, D, dp;
        int64_t n;
    };
    static thread_local Key last = {-2, 0, 0, 0, 0, 0, 0};
    static thread_local bool last_ok = false;
    static thread_local FusedPlan last_plan;
    static thread_local int last_nv = 0, last_gm = 0;
    const int dev = dev_info().device;
    Key k = {dev, sh.B, sh.Hq, sh.Hkv, sh.D, sh.dp, n_tokens};
    if (memcmp(&k, &last, sizeof k) != 0) {
        last_ok = resolve_plan_uncached(sh, n_tokens, last_plan, last_nv, last_gm);
        last = k;
    }
    P = last_plan;
    nvsel = last_nv;
    gm = last_gm;
    return last_ok;
}

static bool resolve_plan_uncached(const tb_shape &sh, int64_t n_tokens, FusedPlan &P, int &nvsel, int &gm) {
    const DevInfo &di = dev_info();
    if (di.sms <= 0) return false;
    const int G = sh.Hq / sh.Hkv;
    gm = group_max(G);
    const int nv = sh.dp / 8;
    nvsel = (nv == 4) ? nv : 0;   // dp = 32 has the unrolled stream; other widths the general loop
    for (int per = 2; per >= 1; --per) {
        FusedPlan Q = plan_fused(sh, n_tokens, di.sms, per);
        if (Q.C == 0) continue;
        if (Q.smem > (size_t)di.max_smem_optin) continue;
        int occ = 0;
#define TB_OCC(NVC, GMC) \
    if (nvsel == NVC && gm == GMC) occ = fused_blocks_per_sm<NVC, GMC>(Q.smem);
        TB_OCC(0, 1) TB_OCC(0, 2) TB_OCC(0, 4) TB_OCC(0, 8) TB_OCC(0, 16)
        TB_OCC(4, 1) TB_OCC(4, 2) TB_OCC(4, 4) TB_OCC(4, 8) TB_OCC(4, 16)
#undef TB_OCC
        if (occ >= per && (int64_t)Q.C * sh.B * sh.Hkv <= (int64_t)occ * di.sms) {
            P = Q;
            return true;
        }
    }
    return false;
}

bool fused_step_supported(const tb_shape &sh, int64_t n_tokens, int32_t k) {
    if (k < 1 || k > n_tokens) return false;
    FusedPlan P;
    int nv, gm;
    if (!resolve_plan(sh, n_tokens, P, nv, gm)) return false;
    return P.C <= fused_chunks(sh, n_tokens);
}

cudaError_t launch_fused_step(const tb_shape &sh, const tb_step_params &p, int64_t n, const uint16_t *q,
                              const uint16_t *q_imp, const uint16_t *K_new, const uint16_t *V_new,
                              const uint16_t *Wk, uint16_t *K, uint16_t *V, uint16_t *Kp, int32_t *idx_state,
                              int32_t *sel, int32_t *counts, uint16_t *out, RowCtl *ctl, uint32_t *attn_ctl,
                              float *partials, int32_t sel_stride, int32_t *dev_status, cudaStream_t st) {
    (void)attn_ctl;
    FusedPlan P;
    int nv, gm;
    if (!resolve_plan(sh, n + 1, P, nv, gm)) return cudaErrorNotSupported;
    FusedArgs a;
    a.q = q; a.q_imp = q_imp; a.K_new = K_new; a.V_new = V_new; a.Wk = Wk;
    a.K = K; a.V = V; a.Kp = Kp;
    a.idx = idx_state; a.sel = sel; a.counts = counts; a.out = out;
    a.ctl = ctl; a.part = partials; a.dev_status = dev_status;
    a.cap = sh.cap; a.n = n;
    a.Hq = sh.Hq; a.Hkv = sh.Hkv; a.D = sh.D; a.dp = sh.dp; a.k = p.k; a.agg = p.agg; a.sel_stride = sel_stride;
    a.scale = p.scale;
    a.C = P.C; a.L = P.L;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(P.C * sh.B * sh.Hkv));
    cfg.blockDim = dim3(kFusedThreads);
    cfg.dynamicSmemBytes = P.smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
#define TB_LAUNCH(NVC, GMC) \
    if (nv == NVC && gm == GMC) return cudaLaunchKernelEx(&cfg, fused_step_kernel<NVC, GMC>, a);
    TB_LAUNCH(0, 1) TB_LAUNCH(0, 2) TB_LAUNCH(0, 4) TB_LAUNCH(0, 8) TB_LAUNCH(0, 16)
    TB_LAUNCH(4, 1) TB_LAUNCH(4, 2) TB_LAUNCH(4, 4) TB_LAUNCH(4, 8) TB_LAUNCH(4, 16)
#undef TB_LAUNCH
    return cudaErrorNotSupported;
}

}  // namespace tb
