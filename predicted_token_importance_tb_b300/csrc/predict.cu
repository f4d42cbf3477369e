// The importance-query predictor's forward pass ("TokenButler: Token
// Importance is Predictable", gist.science summary, Core Architecture, Query
// Prediction: a small multi-layer perceptron turns a producer layer's hidden
// state into G low-dimensional importance queries for each KV head).
//
//   h = SiLU(x W1^T)      x [B, E] bf16, W1 [F, E] bf16, h [B, F] fp32
//   q_imp = RNE_bf16(h W2^T)            W2 [O, F] bf16, O = Hq dp
//
// Decode runs it for a handful of tokens, so both layers are GEMVs bound by
// the weight stream: a warp per output row reads the row once with 16-byte
// loads and keeps one fp32 accumulator per token; the tokens' inputs sit in
// shared memory. Two launches (the second needs all of h); the second runs as
// the first's programmatic dependent and streams its weights while the first
// still runs.
#include "tb_internal.cuh"
#include "kernels.cuh"

namespace tb {

constexpr int kPredThreads = 256;
constexpr int kPredWarps = kPredThreads / 32;

__device__ __forceinline__ float silu(float v) { return v / (1.0f + expf(-v)); }

__device__ __forceinline__ void load8(const uint16_t *p, float (&f)[8]) {
    const uint4 u = *reinterpret_cast<const uint4 *>(p);
    f[0] = bf16_lo(u.x); f[1] = bf16_hi(u.x);
    f[2] = bf16_lo(u.y); f[3] = bf16_hi(u.y);
    f[4] = bf16_lo(u.z); f[5] = bf16_hi(u.z);
    f[6] = bf16_lo(u.w); f[7] = bf16_hi(u.w);
}
__device__ __forceinline__ void load8(const float *p, float (&f)[8]) {
    const float4 a = *reinterpret_cast<const float4 *>(p), b = *reinterpret_cast<const float4 *>(p + 4);
    f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
    f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
}

// out[b, o] = act(sum_e in[b, e] W[o, e]) for o < O, b < B <= BT <= 16;
// IN = uint16_t (bf16) or float; OUT_BF16 rounds once to bf16, else fp32.
// A lane holds kPredGroup 16-byte pieces of its row in flight at a time; the
// first group of the warp's first row is requested before the inputs are
// staged, so the weight stream starts at once.
constexpr int kPredGroup = 8;

__device__ __forceinline__ void unpack_w(const uint4 u, float (&f)[8]) {
    f[0] = bf16_lo(u.x); f[1] = bf16_hi(u.x);
    f[2] = bf16_lo(u.y); f[3] = bf16_hi(u.y);
    f[4] = bf16_lo(u.z); f[5] = bf16_hi(u.z);
    f[6] = bf16_lo(u.w); f[7] = bf16_hi(u.w);
}

// PDL: 1 = the first layer (its dependent may launch at once), 2 = the second layer, launched as that
// dependent: it requests its first weight pieces, then waits for the first layer before reading h.
template <typename IN, int BT, bool SILU, bool OUT_BF16, int PDL>
__global__ void __launch_bounds__(kPredThreads)
gemv_rows_kernel(const IN *__restrict__ in, const uint16_t *__restrict__ W, int B, int E, int O,
                 void *__restrict__ out) {
    if (PDL == 1) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    extern __shared__ __align__(16) uint8_t smem[];
    IN *xs = reinterpret_cast<IN *>(smem);
    constexpr int PER16 = 16 / sizeof(IN);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int o = blockIdx.x * kPredWarps + warp;
    uint4 wg[kPredGroup];
    auto fetch = [&](int row, int e0) {   // pieces e0 + 256 g + 8 lane of the row
#pragma unroll
        for (int g = 0; g < kPredGroup; ++g) {
            const int e = e0 + 256 * g + 8 * lane;
            wg[g] = (row < O && e < E) ? __ldg(reinterpret_cast<const uint4 *>(W + (int64_t)row * E + e))
                                       : make_uint4(0, 0, 0, 0);
        }
    };
    fetch(o, 0);
    if (PDL == 2) asm volatile("griddepcontrol.wait;" ::: "memory");   // h is complete
    for (int x = threadIdx.x; x < B * E / PER16; x += blockDim.x)
        reinterpret_cast<uint4 *>(xs)[x] = reinterpret_cast<const uint4 *>(in)[x];
    __syncthreads();
    for (; o < O; o += gridDim.x * kPredWarps) {
        float acc[BT];
#pragma unroll
        for (int b = 0; b < BT; ++b) acc[b] = 0.f;
        for (int e0 = 0; e0 < E; e0 += 256 * kPredGroup) {
            if (e0 > 0) fetch(o, e0);
#pragma unroll
            for (int g = 0; g < kPredGroup; ++g) {
                const int e = e0 + 256 * g + 8 * lane;
                if (e < E) {
                    float w[8];
                    unpack_w(wg[g], w);
#pragma unroll
                    for (int b = 0; b < BT; ++b) {
                        if (b < B) {
                            float xv[8];
                            load8(xs + (int64_t)b * E + e, xv);
#pragma unroll
                            for (int j = 0; j < 8; ++j) acc[b] = fmaf(w[j], xv[j], acc[b]);
                        }
                    }
                }
            }
        }
        if (o + gridDim.x * kPredWarps < O) fetch(o + gridDim.x * kPredWarps, 0);   // the next row's first group
#pragma unroll
        for (int b = 0; b < BT; ++b) {
#pragma unroll
            for (int s = 16; s > 0; s >>= 1) acc[b] += __shfl_xor_sync(0xFFFFFFFFu, acc[b], s);
        }
        if (lane < B) {
            float v = 0.f;
#pragma unroll
            for (int b = 0; b < BT; ++b)
                if (b == lane) v = acc[b];
            if (SILU) v = silu(v);
            if (OUT_BF16)
                reinterpret_cast<uint16_t *>(out)[(int64_t)lane * O + o] = f_to_bf16(v);
            else
                reinterpret_cast<float *>(out)[(int64_t)lane * O + o] = v;
        }
    }
}

template <typename IN, bool SILU, bool OUT_BF16, int PDL>
static cudaError_t launch_gemv(const IN *in, const uint16_t *W, int B, int E, int O, void *out, cudaStream_t st) {
    const size_t smem = (size_t)B * E * sizeof(IN);
    const int sms = dev_info().sms > 0 ? dev_info().sms : 148;
    int grid = (O + kPredWarps - 1) / kPredWarps;
    if (grid > 8 * sms) grid = 8 * sms;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kPredThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = PDL == 2 ? 1 : 0;
#define TB_GEMV_CASE(BTV)                                                                                     \
    do {                                                                                                      \
        cudaError_t e = cudaFuncSetAttribute(gemv_rows_kernel<IN, BTV, SILU, OUT_BF16, PDL>,                  \
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);         \
        if (e != cudaSuccess) return e;                                                                       \
        return cudaLaunchKernelEx(&cfg, gemv_rows_kernel<IN, BTV, SILU, OUT_BF16, PDL>, in, W, B, E, O, out); \
    } while (0)
    if (B <= 1) TB_GEMV_CASE(1);
    else if (B <= 4) TB_GEMV_CASE(4);
    else if (B <= 8) TB_GEMV_CASE(8);
    else TB_GEMV_CASE(16);
#undef TB_GEMV_CASE
    return cudaGetLastError();
}

cudaError_t launch_predict(const uint16_t *x, const uint16_t *W1, const uint16_t *W2, int B, int E, int F, int O,
                           float *h, uint16_t *q_imp, cudaStream_t st) {
    if (B <= 0) return cudaSuccess;
    cudaError_t e = launch_gemv<uint16_t, true, false, 1>(x, W1, B, E, F, h, st);
    if (e != cudaSuccess) return e;
    return launch_gemv<float, false, true, 2>(h, W2, B, F, O, q_imp, st);
}

}  // namespace tb
