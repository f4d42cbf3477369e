// Standalone fixed-budget top-k over rows of fp32 scores (one cooperative
// launch; the selection machinery is in topk_core.cuh).
#include "kernels.cuh"
#include "topk_core.cuh"

namespace tb {

constexpr int kTopkThreads = 512;
constexpr int kTopkLMax = 16384;   // keys per CTA held in shared memory

__host__ __device__ inline size_t topk_smem_bytes(int L) {
    return (size_t)L * 4 + (size_t)kRadixBins * 4 + (size_t)kCandCap * 8 + (size_t)kMaxChunks * 4 + 33 * 4 +
           8 * 4 + 16;
}

__device__ __forceinline__ SelectSmem carve_select_smem(uint8_t *base, int L) {
    SelectSmem S;
    uint32_t *p = reinterpret_cast<uint32_t *>(base);
    S.keys = p;
    p += L;
    S.hist = p;
    p += kRadixBins;
    S.ckey = p;
    p += kCandCap;
    S.cidx = p;
    p += kCandCap;
    S.ccount = p;
    p += kMaxChunks;
    S.scan = p;
    p += 33;
    S.misc = p;
    p += 8;
    S.abort_flag = reinterpret_cast<int *>(p);
    return S;
}

__global__ void __launch_bounds__(kTopkThreads)
topk_kernel(const float *__restrict__ s, int64_t lds, int64_t n, uint32_t k, int32_t *__restrict__ idx,
            RowCtl *__restrict__ ctl, int row0, int C, int L, int32_t *dev_status, int32_t *sel, int32_t sel_stride,
            int32_t *counts) {
    extern __shared__ __align__(16) uint8_t smem[];
    SelectSmem S = carve_select_smem(smem, L);
    const int row = row0 + blockIdx.x / C;
    const int c = blockIdx.x % C;
    const int64_t t0 = (int64_t)c * L;
    const int Lc = (int)((n - t0) < L ? (n - t0) : L);
    if (threadIdx.x == 0) *S.abort_flag = 0;
    bool nan_seen = false;
    const float *srow = s + (int64_t)row * lds + t0;
    if ((reinterpret_cast<uintptr_t>(srow) & 15) == 0) {   // four scores per load, four loads in flight
        const int L4 = Lc >> 2;
        const float4 *s4 = reinterpret_cast<const float4 *>(srow);
#pragma unroll 4
        for (int e = threadIdx.x; e < L4; e += blockDim.x) {
            const float4 v = __ldg(s4 + e);
            uint4 kv;
            kv.x = score_key(v.x, nan_seen);
            kv.y = score_key(v.y, nan_seen);
            kv.z = score_key(v.z, nan_seen);
            kv.w = score_key(v.w, nan_seen);
            reinterpret_cast<uint4 *>(S.keys)[e] = kv;
        }
        for (int e = 4 * L4 + threadIdx.x; e < Lc; e += blockDim.x) S.keys[e] = score_key(__ldg(srow + e), nan_seen);
    } else {
        for (int e = threadIdx.x; e < Lc; e += blockDim.x) S.keys[e] = score_key(__ldg(srow + e), nan_seen);
    }
    if (nan_seen) set_status(dev_status, TB_ERR_NONFINITE);
    __syncthreads();
    RowCtl *rc = ctl + row;
    SelectResult R = group_select(rc, S, Lc, L, c, C, k, dev_status);
    if (!R.ok) return;
    write_kept(R, S, Lc, (uint32_t)t0, idx + (int64_t)row * k, sel ? sel + (int64_t)row * sel_stride : nullptr);
    if (sel && c == 0 && threadIdx.x == 0) counts[row] = (int32_t)k;
    group_release(rc, C, S);
}

struct TopkPlan {
    int L = 0, C = 0, rows_per_launch = 0;
    size_t smem = 0;
};

static int topk_capacity(size_t smem) {
    static thread_local int cached_dev = -1;   // per thread: no shared mutable state between callers
    static thread_local size_t cached_smem = 0;
    static thread_local int cached_cap = 0;
    const DevInfo &di = dev_info();
    if (cached_dev == di.device && cached_smem == smem) return cached_cap;
    cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, topk_kernel, kTopkThreads, smem) != cudaSuccess)
        per_sm = 0;
    cached_dev = di.device;
    cached_smem = smem;
    cached_cap = per_sm * di.sms;
    return cached_cap;
}

static TopkPlan plan_topk(int rows, int64_t n) {
    TopkPlan P;
    // Enough chunks to spread the rows over the GPU, none longer than kTopkLMax.
    const int sms = dev_info().sms > 0 ? dev_info().sms : 148;
    int64_t want_ctas = 2LL * sms;
    int64_t C = (want_ctas + rows - 1) / rows;
    int64_t minC = (n + kTopkLMax - 1) / kTopkLMax;
    int64_t maxC = (n + 1023) / 1024;   // chunks of at least 1024 tokens
    if (C > maxC) C = maxC;
    if (C < minC) C = minC;
    if (C < 1) C = 1;
    if (C > kMaxChunks) C = kMaxChunks;
    // fewer, longer chunks while that lets every row into one cooperative launch (a second launch costs a
    // whole extra pass over the scores)
    for (;;) {
        int64_t L = (n + C - 1) / C;
        L = (L + 31) / 32 * 32;
        const int64_t Cq = (n + L - 1) / L;
        P.L = (int)L;
        P.C = (int)Cq;
        P.smem = topk_smem_bytes(P.L);
        const int cap = topk_capacity(P.smem);
        P.rows_per_launch = cap >= P.C ? cap / P.C : 0;
        if (P.rows_per_launch >= rows || Cq <= minC || C <= 1) break;
        C = Cq - 1;
    }
    if (P.rows_per_launch > rows) P.rows_per_launch = rows;
    return P;
}

cudaError_t launch_topk(int rows, const float *s, int64_t lds, int64_t n, int32_t k, int32_t *idx, RowCtl *ctl,
                        int32_t *dev_status, cudaStream_t st, int32_t *sel, int32_t sel_stride, int32_t *counts) {
    if (rows <= 0 || k <= 0 || n <= 0) return cudaSuccess;
    if (n > (int64_t)kTopkLMax * kMaxChunks) return cudaErrorInvalidValue;
    TopkPlan P = plan_topk(rows, n);
    if (P.rows_per_launch <= 0) return cudaErrorCooperativeLaunchTooLarge;
    for (int r0 = 0; r0 < rows; r0 += P.rows_per_launch) {
        const int nr = (rows - r0) < P.rows_per_launch ? (rows - r0) : P.rows_per_launch;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)(nr * P.C));
        cfg.blockDim = dim3(kTopkThreads);
        cfg.dynamicSmemBytes = P.smem;
        cfg.stream = st;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeCooperative;
        attr[0].val.cooperative = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        cudaError_t e = cudaLaunchKernelEx(&cfg, topk_kernel, s, lds, n, (uint32_t)k, idx, ctl, r0, P.C, P.L,
                                           dev_status, sel, sel_stride, counts);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace tb
