// Batched key projection Kp = RNE_bf16(K . Wk) for prefill / batched append
// ("TokenButler: Token Importance is Predictable", gist.science summary,
// Core Architecture: Key-Cache Projection; Optimizations: Batching).
//
// CUDA-core path: one CTA projects 64 rows of one (b, h). Used for batches
// that the tensor-core kernel (project_tc.cu) does not take.
#include "tb_internal.cuh"
#include "kernels.cuh"

namespace tb {

constexpr int kProjRows = 64;
constexpr int kProjThreads = 256;

__global__ void __launch_bounds__(kProjThreads)
project_simple_kernel(const uint16_t *__restrict__ K_src, int64_t src_stride, const uint16_t *__restrict__ Wk,
                      uint16_t *__restrict__ Kp, int64_t cap, int Hkv, int D, int dp, int64_t pos0, int64_t n_new) {
    extern __shared__ float sm[];
    float *w = sm;                    // [D][dp]
    float *kt = sm + (int64_t)D * dp; // [kProjRows][D + 1]
    const int row = blockIdx.y;
    const int h = row % Hkv;
    const int64_t r0 = (int64_t)blockIdx.x * kProjRows;
    const uint16_t *W = Wk + (int64_t)h * D * dp;
    for (int x = threadIdx.x; x < D * dp; x += blockDim.x) w[x] = bf16_to_f(W[x]);
    const uint16_t *src = K_src + (int64_t)row * src_stride * D;
    for (int x = threadIdx.x; x < kProjRows * D; x += blockDim.x) {
        const int rr = x / D, d = x % D;
        const int64_t t = r0 + rr;
        kt[rr * (D + 1) + d] = t < n_new ? bf16_to_f(src[t * D + d]) : 0.f;
    }
    __syncthreads();
    const int rr = threadIdx.x % kProjRows;
    const int js = threadIdx.x / kProjRows;
    const int nslice = blockDim.x / kProjRows;
    const int64_t t = r0 + rr;
    if (t >= n_new) return;
    uint16_t *dst = Kp + ((int64_t)row * cap + pos0 + t) * dp;
    for (int j = js; j < dp; j += nslice) {
        float a = 0.f;
        for (int d = 0; d < D; ++d) a = fmaf(kt[rr * (D + 1) + d], w[d * dp + j], a);
        dst[j] = f_to_bf16(a);
    }
}

cudaError_t launch_project_simple(const tb_shape &sh, const uint16_t *K_src, int64_t src_stride,
                                  const uint16_t *Wk, uint16_t *Kp, int64_t pos0, int64_t n_new, cudaStream_t st) {
    const int rows = sh.B * sh.Hkv;
    if (rows <= 0 || n_new <= 0) return cudaSuccess;
    const size_t smem = ((size_t)sh.D * sh.dp + (size_t)kProjRows * (sh.D + 1)) * sizeof(float);
    static thread_local int attr_dev = -1;   // the attribute belongs to each device's context
    if (attr_dev != dev_info().device) {
        cudaFuncSetAttribute(project_simple_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
        attr_dev = dev_info().device;
    }
    dim3 grid((unsigned)((n_new + kProjRows - 1) / kProjRows), (unsigned)rows);
    project_simple_kernel<<<grid, kProjThreads, smem, st>>>(K_src, src_stride, Wk, Kp, sh.cap, sh.Hkv, sh.D, sh.dp,
                                                            pos0, n_new);
    return cudaGetLastError();
}

bool project_tc_supported(const tb_shape &sh, int64_t n_new);
cudaError_t launch_project_tc(const tb_shape &sh, const uint16_t *K_src, int64_t src_stride, const uint16_t *Wk,
                              uint16_t *Kp, int64_t pos0, int64_t n_new, int32_t *dev_status, cudaStream_t st);

cudaError_t launch_project(const tb_shape &sh, const uint16_t *K_src, int64_t src_stride, const uint16_t *Wk,
                           uint16_t *Kp, int64_t pos0, int64_t n_new, int32_t *dev_status, cudaStream_t st,
                           int path) {
    // path: 0 automatic (tensor cores for batches of >= 128 rows), 1 CUDA cores, 2 tensor cores
    const bool tc = path == 2 || (path == 0 && project_tc_supported(sh, n_new));
    if (tc) {
        if (!project_tc_supported(sh, n_new)) return cudaErrorInvalidValue;
        return launch_project_tc(sh, K_src, src_stride, Wk, Kp, pos0, n_new, dev_status, st);
    }
    return launch_project_simple(sh, K_src, src_stride, Wk, Kp, pos0, n_new, st);
}

}  // namespace tb
