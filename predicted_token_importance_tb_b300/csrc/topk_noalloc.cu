// tb_topk_noalloc: the fixed-budget top-k of tb_topk for callers that cannot
// allocate device memory and so cannot provide a workspace.
//
// The selection's per-row control blocks (histograms, barrier counters,
// candidate list) live in one file-scope device array instead of a
// caller-provided workspace. The array is part of the library image: every
// GPU that loads libtb holds it (kNoAllocRows * sizeof(RowCtl) bytes, about
// 3.9 MB) until the process exits. Host code reaches it only through the
// address cudaGetSymbolAddress returns for the current device.
#include <mutex>

#include "kernels.cuh"
#include "tb_internal.cuh"
#include "ws_layout.cuh"

namespace tb {

constexpr int kNoAllocRows = TB_TOPK_NOALLOC_MAX_ROWS;
constexpr int kNoAllocMaxDevices = 64;

static __device__ __align__(256) RowCtl g_topk_noalloc_ctl[kNoAllocRows];

// Device address of g_topk_noalloc_ctl on the current device, looked up once
// per device (the symbol's host-side name is not a device address).
static cudaError_t noalloc_scratch(RowCtl **out) {
    static std::mutex mu;
    static RowCtl *ptr[kNoAllocMaxDevices] = {};
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kNoAllocMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (!ptr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_topk_noalloc_ctl);
        if (e != cudaSuccess) return e;
        ptr[dev] = static_cast<RowCtl *>(p);
    }
    *out = ptr[dev];
    return cudaSuccess;
}

}  // namespace tb

using namespace tb;

extern "C" TB_API tb_status tb_topk_noalloc(const tb_shape *shape, const float *s, int64_t n, int32_t k,
                                            int32_t *idx, int32_t *dev_status, cudaStream_t stream) {
    if (!shape) return TB_ERR_INVALID_ARG;
    if (shape->B <= 0 || shape->Hkv <= 0) return TB_ERR_INVALID_ARG;
    const int64_t rows = (int64_t)shape->B * shape->Hkv;
    if (rows > kNoAllocRows) return TB_ERR_UNSUPPORTED;
    if (n < 0 || k < 0 || k > n) return TB_ERR_INVALID_ARG;
    if (k == 0) return TB_OK;
    if (!s || !idx) return TB_ERR_INVALID_ARG;
    if (n >= ((int64_t)1 << 31) - 1) return TB_ERR_UNSUPPORTED;
    RowCtl *ctl = nullptr;
    cudaError_t e = noalloc_scratch(&ctl);
    if (e != cudaSuccess) return TB_ERR_CUDA;
    // The array keeps whatever the previous call (or a timed-out one) left:
    // clear the control blocks this call uses before the kernel runs.
    e = cudaMemsetAsync(ctl, 0, (size_t)rows * sizeof(RowCtl), stream);
    if (e != cudaSuccess) return TB_ERR_CUDA;
    e = launch_topk((int)rows, s, n, n, k, idx, ctl, dev_status, stream);
    if (e == cudaSuccess) return TB_OK;
    return e == cudaErrorInvalidValue ? TB_ERR_UNSUPPORTED : TB_ERR_CUDA;
}
