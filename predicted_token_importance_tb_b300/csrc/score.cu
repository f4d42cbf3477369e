// Importance scores: s[b,h,t] = agg_g q_imp[b,h*G+g,:] . Kp[b,h,t,:]
// ("TokenButler: Token Importance is Predictable", gist.science summary,
// Core Architecture, Scoring).
//
// HBM-bound stream of Kp (2*dp bytes per token). A warp scores 32
// consecutive tokens; each of its dp/8 load instructions reads 512 contiguous
// bytes and the lanes of a row add their partial dot products by shuffles.
// Long rows go through a shared-memory ring of cp.async tiles per warp
// (score_ring_kernel), shorter ones one tile per CTA in registers
// (score_kernel). The G importance queries of the KV head sit in shared memory
// as fp32; with the mean aggregation they are folded into their group mean
// first (the mean of dot products equals the dot product with the mean query).
// Any other dp (a multiple of 8): one thread per token (score_kernel_any).
#include "tb_internal.cuh"
#include "kernels.cuh"

namespace tb {

constexpr int kScoreThreads = 256;
constexpr int kScoreMultiMin = 8;   // tiles per CTA below which one tile per CTA is used

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

// Scores of one token from its Kp row v (NV 16-byte vectors) against the staged query (MEAN: the group-mean
// query; MAX: the G queries).
template <int NV>
__device__ __forceinline__ float score_of(const float *qs, const uint4 (&v)[NV], int agg, int G, int dp) {
    if (agg == TB_AGG_MEAN) {
        float acc = 0.f;
#pragma unroll
        for (int i = 0; i < NV; ++i) acc = dot8(qs + 8 * i, v[i], acc);
        return acc;
    }
    float out = -INFINITY;
    for (int g = 0; g < G; ++g) {
        float acc = 0.f;
#pragma unroll
        for (int i = 0; i < NV; ++i) acc = dot8(qs + g * dp + 8 * i, v[i], acc);
        out = fmaxf(out, acc);
    }
    return out;
}

// Stage the KV head's importance queries in shared memory as fp32 (MEAN: their group mean).
__device__ __forceinline__ void stage_queries(const uint16_t *qrow, int agg, int G, int dp, float *qs) {
    if (agg == TB_AGG_MEAN) {
        const float inv = 1.0f / (float)G;
        for (int i = threadIdx.x; i < dp; i += blockDim.x) {
            float a = 0.f;
#pragma unroll 8
            for (int g = 0; g < G; ++g) a += bf16_to_f(__ldg(qrow + g * dp + i));
            qs[i] = a * inv;
        }
    } else {
        for (int i = threadIdx.x; i < G * dp; i += blockDim.x) qs[i] = bf16_to_f(__ldg(qrow + i));
    }
}

// NV = dp/8 known at compile time. A CTA scores one tile of kScoreThreads consecutive tokens of one row; warp w
// takes tokens [32w, 32w + 32), and each of its NV load instructions reads 512 contiguous bytes: the NV 16-byte
// pieces of 32/NV consecutive rows, lane l holding piece l % NV of one of them. Every lane dots its piece with
// the matching 8 query dims and the NV lanes of a row add their sums by shuffles. The tile's rows are requested
// before the queries are staged.
template <int NV>
__global__ void __launch_bounds__(kScoreThreads, NV <= 4 ? 6 : 4)
score_kernel(const uint16_t *__restrict__ q_imp, const uint16_t *__restrict__ Kp, int64_t cap, int64_t n,
             int Hq, int Hkv, int dp, int agg, float *__restrict__ s, int64_t lds, const int64_t *__restrict__ n_seq,
             int U, int after_append) {
    extern __shared__ float qs[];   // [G][dp] (MAX) or [dp] (MEAN)
    constexpr int TPI = 32 / NV;    // rows per load instruction of a warp
    const int row = blockIdx.y;
    const int b = row / Hkv, h = row % Hkv;
    const int G = Hq / Hkv;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, pc = lane % NV;
    // tokens past this sequence's n_seq[b] + 1 are scored -inf (never selected)
    const int64_t n_lim = n_seq ? (n_seq[b] + 1 < n ? n_seq[b] + 1 : n) : n;
    // launched as the append kernel's programmatic dependent: only the CTA holding the appended token (the
    // sequence's last, n_lim - 1) reads what that kernel writes, so only it waits for it to finish
    if (after_append && blockIdx.x == (n_lim - 1) / ((int64_t)U * kScoreThreads))
        asm volatile("griddepcontrol.wait;" ::: "memory");
    const int64_t w0 = (int64_t)blockIdx.x * U * kScoreThreads + warp * 32;
    const uint4 *krow = reinterpret_cast<const uint4 *>(Kp + (int64_t)row * cap * dp);
    float *srow = s + (int64_t)row * lds;
    uint4 v0[NV];
    auto load = [&](int u, uint4 (&v)[NV]) {
#pragma unroll
        for (int j = 0; j < NV; ++j) {
            const int64_t t = w0 + (int64_t)u * kScoreThreads + j * TPI + lane / NV;
            if (t < n_lim) v[j] = __ldcs(krow + t * NV + pc);
        }
    };
    load(0, v0);
    stage_queries(q_imp + ((int64_t)b * Hq + (int64_t)h * G) * dp, agg, G, dp, qs);
    __syncthreads();
    float qv[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) qv[i] = qs[8 * pc + i];   // MEAN: this lane's 8 query dims
    auto emit = [&](int u, const uint4 (&v)[NV]) {
        // row j * TPI + lane / NV of the warp's 32: its score, in every lane of its group
        float mine = 0.f;
#pragma unroll
        for (int j = 0; j < NV; ++j) {
            float sc;
            if (agg == TB_AGG_MEAN) {
                sc = dot8(qv, v[j], 0.f);
#pragma unroll
                for (int o = 1; o < NV; o <<= 1) sc += __shfl_xor_sync(0xFFFFFFFFu, sc, o);
            } else {
                sc = -INFINITY;
                for (int g = 0; g < G; ++g) {
                    float d = dot8(qs + g * dp + 8 * pc, v[j], 0.f);
#pragma unroll
                    for (int o = 1; o < NV; o <<= 1) d += __shfl_xor_sync(0xFFFFFFFFu, d, o);
                    sc = fmaxf(sc, d);
                }
            }
            if (pc == j) mine = sc;
        }
        // lane l writes row (l % NV) * TPI + l / NV: the warp's 32 scores in one store
        const int64_t t = w0 + (int64_t)u * kScoreThreads + pc * TPI + lane / NV;
        if (t < n) srow[t] = t < n_lim ? mine : -INFINITY;
    };
    emit(0, v0);
}

constexpr int kScoreDepth = 4;   // tiles in a warp's ring: three in flight while one is scored

// Long rows: a CTA scores U tiles of kScoreThreads tokens of one row. Each warp keeps a ring of kScoreDepth
// copies of its 32-token slice of a tile in shared memory, filled by 16-byte cp.async pieces in the same
// 512-byte-per-instruction order as score_kernel, so three tiles are in flight per warp without holding
// registers; the scoring is score_kernel's.
template <int NV>
__global__ void __launch_bounds__(kScoreThreads, NV <= 2 ? 4 : (NV <= 4 ? 3 : 1))
score_ring_kernel(const uint16_t *__restrict__ q_imp, const uint16_t *__restrict__ Kp, int64_t cap, int64_t n,
                  int Hq, int Hkv, int dp, int agg, float *__restrict__ s, int64_t lds,
                  const int64_t *__restrict__ n_seq, int U, int after_append) {
    extern __shared__ __align__(16) uint8_t smb[];
    constexpr int TPI = 32 / NV, WT = 512 * NV;   // rows per load instruction; bytes of a warp's slice
    const int row = blockIdx.y;
    const int b = row / Hkv, h = row % Hkv;
    const int G = Hq / Hkv;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, pc = lane % NV;
    float *qs = reinterpret_cast<float *>(smb + (kScoreThreads / 32) * kScoreDepth * WT);
    const uint32_t rb = (uint32_t)__cvta_generic_to_shared(smb + warp * kScoreDepth * WT) + lane * 16;
    const int64_t n_lim = n_seq ? (n_seq[b] + 1 < n ? n_seq[b] + 1 : n) : n;
    if (after_append && blockIdx.x == (n_lim - 1) / ((int64_t)U * kScoreThreads))   // see score_kernel
        asm volatile("griddepcontrol.wait;" ::: "memory");
    const int64_t w0 = (int64_t)blockIdx.x * U * kScoreThreads + warp * 32;
    const uint4 *krow = reinterpret_cast<const uint4 *>(Kp + (int64_t)row * cap * dp);
    float *srow = s + (int64_t)row * lds;
    auto issue = [&](int u) {   // this warp's slice of tile u into ring slot u % kScoreDepth
        const uint32_t dst = rb + (uint32_t)((u % kScoreDepth) * WT);
#pragma unroll
        for (int j = 0; j < NV; ++j) {
            const int64_t t = w0 + (int64_t)u * kScoreThreads + j * TPI + lane / NV;
            if (t < n_lim)
                asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst + j * 512), "l"(krow + t * NV + pc)
                             : "memory");
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
    };
    int issued = 0;
    for (; issued < kScoreDepth - 1 && issued < U; ++issued) issue(issued);
    stage_queries(q_imp + ((int64_t)b * Hq + (int64_t)h * G) * dp, agg, G, dp, qs);
    __syncthreads();
    float qv[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) qv[i] = qs[8 * pc + i];   // MEAN: this lane's 8 query dims
    for (int u = 0; u < U; ++u) {
        // this lane's pieces of tile u have landed once at most issued - u - 1 groups are pending
        const int pend = issued - u - 1;
        if (pend >= 2) asm volatile("cp.async.wait_group 2;" ::: "memory");
        else if (pend == 1) asm volatile("cp.async.wait_group 1;" ::: "memory");
        else asm volatile("cp.async.wait_group 0;" ::: "memory");
        __syncwarp();   // every lane's pieces of the slice are visible to the warp
        uint4 v[NV];
        const uint32_t src = rb + (uint32_t)((u % kScoreDepth) * WT);
#pragma unroll
        for (int j = 0; j < NV; ++j)
            asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(v[j].x), "=r"(v[j].y), "=r"(v[j].z), "=r"(v[j].w)
                         : "r"(src + j * 512));
        __syncwarp();   // the slot of tile u - 1, refilled next, was read by every lane
        if (issued < U) issue(issued++);
        float mine = 0.f;
#pragma unroll
        for (int j = 0; j < NV; ++j) {
            float sc;
            if (agg == TB_AGG_MEAN) {
                sc = dot8(qv, v[j], 0.f);
#pragma unroll
                for (int o = 1; o < NV; o <<= 1) sc += __shfl_xor_sync(0xFFFFFFFFu, sc, o);
            } else {
                sc = -INFINITY;
                for (int g = 0; g < G; ++g) {
                    float d = dot8(qs + g * dp + 8 * pc, v[j], 0.f);
#pragma unroll
                    for (int o = 1; o < NV; o <<= 1) d += __shfl_xor_sync(0xFFFFFFFFu, d, o);
                    sc = fmaxf(sc, d);
                }
            }
            if (pc == j) mine = sc;
        }
        const int64_t t = w0 + (int64_t)u * kScoreThreads + pc * TPI + lane / NV;
        if (t < n) srow[t] = t < n_lim ? mine : -INFINITY;
    }
}

// Any dp that is a multiple of 8: one token per thread.
__global__ void __launch_bounds__(kScoreThreads)
score_kernel_any(const uint16_t *__restrict__ q_imp, const uint16_t *__restrict__ Kp, int64_t cap, int64_t n,
                 int Hq, int Hkv, int dp, int agg, float *__restrict__ s, int64_t lds,
                 const int64_t *__restrict__ n_seq) {
    extern __shared__ float qs[];
    const int row = blockIdx.y;
    const int b = row / Hkv, h = row % Hkv;
    const int G = Hq / Hkv;
    stage_queries(q_imp + ((int64_t)b * Hq + (int64_t)h * G) * dp, agg, G, dp, qs);
    __syncthreads();
    const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= n) return;
    if (n_seq && t > n_seq[b]) {
        s[(int64_t)row * lds + t] = -INFINITY;
        return;
    }
    const int nv = dp / 8;
    const uint4 *p = reinterpret_cast<const uint4 *>(Kp + ((int64_t)row * cap + t) * dp);
    float out = -INFINITY;
    if (agg == TB_AGG_MEAN) {
        out = 0.f;
        for (int i = 0; i < nv; ++i) out = dot8(qs + 8 * i, __ldcs(p + i), out);
    } else {
        for (int g = 0; g < G; ++g) {
            float acc = 0.f;
            for (int i = 0; i < nv; ++i) acc = dot8(qs + g * dp + 8 * i, __ldcs(p + i), acc);
            out = fmaxf(out, acc);
        }
    }
    s[(int64_t)row * lds + t] = out;
}

cudaError_t launch_score(const tb_shape &sh, const uint16_t *q_imp, const uint16_t *Kp, int64_t n, int agg,
                         float *s, int64_t lds, cudaStream_t st, const int64_t *n_seq, bool after_append) {
    const int rows = sh.B * sh.Hkv;
    if (n <= 0 || rows <= 0) return cudaSuccess;
    const int G = sh.Hq / sh.Hkv;
    const size_t smem = (size_t)(agg == TB_AGG_MEAN ? 1 : G) * sh.dp * sizeof(float);
    const int nv = sh.dp / 8;
    // tiles per CTA: one (many light CTAs) unless the stream is long enough to leave several tiles per CTA
    // at four CTAs per SM; then up to 8
    const int sms = dev_info().sms > 0 ? dev_info().sms : 148;
    const int64_t tiles = (n + kScoreThreads - 1) / kScoreThreads;
    int64_t U = tiles * rows / (4LL * sms);
    if (U > 8) U = 8;
    if (U < kScoreMultiMin) U = 1;
    const dim3 grid((unsigned)((tiles + U - 1) / U), (unsigned)rows);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kScoreThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = after_append ? 1 : 0;
    const int aa = after_append ? 1 : 0;
    const size_t ring_smem = (size_t)(kScoreThreads / 32) * kScoreDepth * 512 * nv + smem;
#define TB_SCORE_CASE(NVC)                                                                                        \
    case NVC:                                                                                                     \
        if (U > 1) {                                                                                              \
            cfg.dynamicSmemBytes = ring_smem;                                                                     \
            static thread_local int attr_dev_##NVC = -1;                                                          \
            if (attr_dev_##NVC != dev_info().device) {                                                            \
                cudaError_t e = cudaFuncSetAttribute(score_ring_kernel<NVC>,                                      \
                                                     cudaFuncAttributeMaxDynamicSharedMemorySize, (int)ring_smem); \
                if (e != cudaSuccess) return e;                                                                   \
                attr_dev_##NVC = dev_info().device;                                                               \
            }                                                                                                     \
            return cudaLaunchKernelEx(&cfg, score_ring_kernel<NVC>, q_imp, Kp, sh.cap, n, sh.Hq, sh.Hkv, sh.dp,   \
                                      agg, s, lds, n_seq, (int)U, aa);                                            \
        }                                                                                                         \
        return cudaLaunchKernelEx(&cfg, score_kernel<NVC>, q_imp, Kp, sh.cap, n, sh.Hq, sh.Hkv, sh.dp, agg, s,    \
                                  lds, n_seq, 1, aa);
    switch (nv) {
        TB_SCORE_CASE(1)
        TB_SCORE_CASE(2)
        TB_SCORE_CASE(4)
        TB_SCORE_CASE(8)
        default:
            score_kernel_any<<<dim3((unsigned)tiles, (unsigned)rows), kScoreThreads, smem, st>>>(
                q_imp, Kp, sh.cap, n, sh.Hq, sh.Hkv, sh.dp, agg, s, lds, n_seq);
    }
#undef TB_SCORE_CASE
    return cudaGetLastError();
}

}  // namespace tb
