// Decode-step append: the step's new key/value rows go into the cache and the
// key is projected into the low-dimensional cache ("TokenButler: Token
// Importance is Predictable", gist.science summary, Core Architecture,
// Key-Cache Projection). One CTA per (b, h); thread j < dp accumulates output
// j over a slice of D, the slices are summed in shared memory (fp32), then
// rounded once to bf16. With Kp == nullptr only the K/V rows are written (the
// buffered step projects in batches instead).
#include "tb_internal.cuh"
#include "kernels.cuh"

namespace tb {

constexpr int kAppendThreads = 256;

__global__ void __launch_bounds__(kAppendThreads)
append_kernel(const uint16_t *__restrict__ K_new, const uint16_t *__restrict__ V_new,
              const uint16_t *__restrict__ Wk, uint16_t *__restrict__ K, uint16_t *__restrict__ V,
              uint16_t *__restrict__ Kp, int64_t cap, int Hkv, int D, int dp, int64_t pos, int32_t *sel,
              int32_t sel_stride, int32_t *counts, int32_t *dev_status, const int64_t *__restrict__ pos_seq) {
    extern __shared__ float sh[];   // knew[D] then partial[kAppendThreads]
    // a programmatic dependent (the streamed attention of a step inside an interval) may start now: it does
    // not read what this kernel writes before it has waited for this grid
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    float *knew = sh;
    float *part = sh + D;
    const int row = blockIdx.x;
    const int h = row % Hkv;
    if (pos_seq) pos = pos_seq[row / Hkv];   // ragged batch: this sequence's position
    const uint16_t *kn = K_new + (int64_t)row * D;
    const uint16_t *vn = V_new + (int64_t)row * D;
    uint16_t *Krow = K + ((int64_t)row * cap + pos) * D;
    uint16_t *Vrow = V + ((int64_t)row * cap + pos) * D;
    for (int d = threadIdx.x; d < D; d += blockDim.x) {
        const uint16_t kb = kn[d];
        knew[d] = bf16_to_f(kb);
        Krow[d] = kb;
        Vrow[d] = vn[d];
    }
    __syncthreads();
    if (Kp != nullptr) {   // (uniform)
        const uint16_t *W = Wk + (int64_t)h * D * dp;
        uint16_t *kp = Kp + ((int64_t)row * cap + pos) * dp;
        // outputs j in [j0, j0 + jn) at a time; the threads split D among them
        const int slices = blockDim.x / (dp < (int)blockDim.x ? dp : (int)blockDim.x);
        for (int j0 = 0; j0 < dp; j0 += blockDim.x / slices) {
            const int jn = blockDim.x / slices;
            const int j = j0 + (int)threadIdx.x % jn;
            const int sl = (int)threadIdx.x / jn;
            const int dlen = (D + slices - 1) / slices;
            float a = 0.f;
            if (j < dp) {
                const int d0 = sl * dlen, d1 = min(D, d0 + dlen);
                for (int d = d0; d < d1; ++d) a = fmaf(knew[d], bf16_to_f(W[(int64_t)d * dp + j]), a);
            }
            part[threadIdx.x] = a;
            __syncthreads();
            if (sl == 0 && j < dp) {
                float tot = 0.f;
                for (int x = 0; x < slices; ++x) tot += part[x * jn + (int)threadIdx.x % jn];
                kp[j] = f_to_bf16(tot);
            }
            __syncthreads();
        }
    }
    if (sel && threadIdx.x == 0) {
        const int32_t c = counts[row];
        if (c >= 0 && c < sel_stride) {
            sel[(int64_t)row * sel_stride + c] = (int32_t)pos;
            counts[row] = c + 1;
        } else {
            set_status(dev_status, TB_ERR_INVALID_ARG);
        }
    }
}

cudaError_t launch_append(const tb_shape &sh, const uint16_t *K_new, const uint16_t *V_new, const uint16_t *Wk,
                          uint16_t *K, uint16_t *V, uint16_t *Kp, int64_t pos, int32_t *sel, int32_t sel_stride,
                          int32_t *counts, int32_t *dev_status, cudaStream_t st, const int64_t *pos_seq) {
    const int rows = sh.B * sh.Hkv;
    if (rows <= 0) return cudaSuccess;
    const size_t smem = (size_t)(sh.D + kAppendThreads) * sizeof(float);
    append_kernel<<<rows, kAppendThreads, smem, st>>>(K_new, V_new, Wk, K, V, Kp, sh.cap, sh.Hkv, sh.D, sh.dp, pos,
                                                      sel, sel_stride, counts, dev_status, pos_seq);
    return cudaGetLastError();
}

}  // namespace tb
