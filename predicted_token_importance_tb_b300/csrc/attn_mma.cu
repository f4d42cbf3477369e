// Exact attention over the selected K/V rows on the tensor cores
// ("TokenButler: Token Importance is Predictable": the full cache stays
// resident and only the selected tokens are read).
//
// Grid = (splits, rows); a CTA of four warps takes split_tok consecutive
// entries of its row's selection, in rounds of kAMTok rows. Every lane copies
// one 16-byte chunk of a K or V row into shared memory (cp.async), so a
// round's rows are all in flight at once; invalid entries (outside [0, cap))
// are reported and their slots zeroed. The warps then attend chunks of 16
// staged rows with m16n8k16 MMAs (attn_mma.cuh), their states are combined
// into one partial (max, sum, acc[D]) per query head, and the row's last CTA
// merges the splits.
#include "attn_mma.cuh"
#include "kernels.cuh"

namespace tb {

constexpr int kAMThreads = 128;
constexpr int kAMWarps = kAMThreads / 32;
constexpr int kAMTok = 128;   // rows staged per round

__host__ __device__ inline size_t attn_mma_smem_bytes(int D) {
    return (size_t)kAMTok * mma_slot_bytes(D) + 16 * (2 * D + 16) + kAMTok + kAMTok * 4;
}

template <int DT>
__global__ void __launch_bounds__(kAMThreads)
attn_mma_kernel(const uint16_t *__restrict__ q, const uint16_t *__restrict__ K, const uint16_t *__restrict__ V,
                const int32_t *__restrict__ sel, const int32_t *__restrict__ counts, int32_t sel_stride, int64_t cap,
                int Hq, int Hkv, float scale, uint16_t *__restrict__ out, uint32_t *__restrict__ attn_ctl,
                float *__restrict__ part, int split_tok, int32_t *dev_status) {
    extern __shared__ __align__(128) uint8_t smb[];
    __shared__ uint32_t last;
    constexpr int SB = 4 * DT + 16, CPR = DT / 8, RPW = 32 / (2 * CPR), NT = DT / 8;
    uint8_t *X = smb;
    uint8_t *qsm = X + (size_t)kAMTok * SB;
    uint8_t *kept = qsm + 16 * (2 * DT + 16);
    int32_t *toks = reinterpret_cast<int32_t *>(kept + kAMTok);   // this round's selection entries
    const int G = Hq / Hkv;
    const int row = blockIdx.y, split = blockIdx.x, nsplit = gridDim.x;
    const int b = row / Hkv, h = row % Hkv;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;

    const int cnt = counts ? counts[row] : sel_stride;
    const int cnt_c = cnt < 0 ? 0 : (cnt > sel_stride ? sel_stride : cnt);
    if (threadIdx.x == 0 && split == 0 && (cnt <= 0 || cnt > sel_stride)) set_status(dev_status, TB_ERR_INVALID_ARG);
    const int j0 = split * split_tok;
    const int j1 = min(j0 + split_tok, cnt_c);
    const int32_t *srow = sel + (int64_t)row * sel_stride;
    const uint16_t *Kh = K + (int64_t)row * cap * DT;
    const uint16_t *Vh = V + (int64_t)row * cap * DT;

    // query tile: the G heads as rows of a 16-row bf16 tile (zero-padded)
    const uint16_t *qrow = q + ((int64_t)b * Hq + (int64_t)h * G) * DT;
    for (int x = threadIdx.x; x < 16 * CPR; x += blockDim.x) {
        const int g = x / CPR, cc = x % CPR;
        uint4 v = make_uint4(0, 0, 0, 0);
        if (g < G) v = *reinterpret_cast<const uint4 *>(qrow + g * DT + cc * 8);
        *reinterpret_cast<uint4 *>(qsm + g * (2 * DT + 16) + cc * 16) = v;
    }

    MmaAttn<NT> A;
    A.m0 = A.m1 = -INFINITY;
    A.l0 = A.l1 = 0.f;
#pragma unroll
    for (int t = 0; t < NT; ++t) A.o[t][0] = A.o[t][1] = A.o[t][2] = A.o[t][3] = 0.f;
    const float qscale = scale * kLog2e;
    const int rl = lane % (2 * CPR);
    const bool rl_v = rl >= CPR;
    const int rl_c = rl_v ? rl - CPR : rl;
    for (int r0 = j0; r0 < j1; r0 += kAMTok) {
        const int nr = min(kAMTok, j1 - r0);
        const int npad = (nr + 15) & ~15;
        __syncthreads();   // the previous round's rows are consumed
        for (int s = threadIdx.x; s < npad; s += blockDim.x) toks[s] = s < nr ? __ldg(srow + r0 + s) : -1;
        __syncthreads();
        for (int s = warp * RPW + lane / (2 * CPR); s < npad; s += kAMWarps * RPW) {
            const int32_t t = toks[s];
            const bool valid = t >= 0 && (int64_t)t < cap;
            if (s < nr && !valid && rl == 0) set_status(dev_status, TB_ERR_INVALID_ARG);
            uint8_t *dst = X + (size_t)s * SB + (rl_v ? 2 * DT : 0) + rl_c * 16;
            if (valid) cp_async16(dst, (rl_v ? Vh : Kh) + (int64_t)t * DT + rl_c * 8);
            st_shared_zero16_if(dst, !valid);
            if (rl == 0) kept[s] = valid ? 1 : 0;
        }
        cp_async_commit();
        cp_async_wait_all();
        __syncthreads();
        mma_attend<DT, kAMWarps>(A, X, SB, nr, kept, 0, qsm, qscale);
    }

    // the warps' states -> this split's partial (m, l, acc[D]) per head
    A.l0 += __shfl_xor_sync(0xFFFFFFFFu, A.l0, 1);
    A.l0 += __shfl_xor_sync(0xFFFFFFFFu, A.l0, 2);
    A.l1 += __shfl_xor_sync(0xFFFFFFFFu, A.l1, 1);
    A.l1 += __shfl_xor_sync(0xFFFFFFFFu, A.l1, 2);
    __syncthreads();   // X is free: warp states go there
    float *ws = reinterpret_cast<float *>(X);
    const int sg = 2 + DT;
    {
        const int g0 = lane >> 2, d0 = 2 * (lane & 3);
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            const int g = g0 + 8 * half;
            if (g < G) {
                float *w = ws + ((int64_t)warp * G + g) * sg;
                if ((lane & 3) == 0) {
                    w[0] = half ? A.m1 : A.m0;
                    w[1] = half ? A.l1 : A.l0;
                }
#pragma unroll
                for (int t = 0; t < NT; ++t)
                    *reinterpret_cast<float2 *>(w + 2 + 8 * t + d0) = make_float2(A.o[t][2 * half], A.o[t][2 * half + 1]);
            }
        }
    }
    __syncthreads();
    float *prow = part + (int64_t)row * nsplit * G * sg;
    for (int x = threadIdx.x; x < G * DT; x += blockDim.x) {
        const int g = x / DT, d = x % DT;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kAMWarps; ++w) M = fmaxf(M, ws[((int64_t)w * G + g) * sg]);
        float L = 0.f, Acc = 0.f;
#pragma unroll
        for (int w = 0; w < kAMWarps; ++w) {
            const float *sw = ws + ((int64_t)w * G + g) * sg;
            const float wt = rescale_w(sw[0], M);
            L = fmaf(wt, sw[1], L);
            Acc = fmaf(wt, sw[2 + d], Acc);
        }
        float *o = prow + ((int64_t)split * G + g) * sg;
        if (d == 0) {
            o[0] = M;
            o[1] = L;
        }
        o[2 + d] = Acc;
    }

    // the last CTA of the row merges the splits
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        const uint32_t prev = atomicAdd(attn_ctl + row, 1u);
        last = (prev == (uint32_t)(nsplit - 1)) ? 1u : 0u;
    }
    __syncthreads();
    if (!last) return;
    __threadfence();
    attn_merge(prow, nsplit, G, DT, out + ((int64_t)b * Hq + (int64_t)h * G) * DT, dev_status,
               reinterpret_cast<float *>(X));
    if (threadIdx.x == 0) attn_ctl[row] = 0;   // ready for the next call
}

bool attn_mma_supported(const tb_shape &sh) {
    const int G = sh.Hq / sh.Hkv;
    return (sh.D == 64 || sh.D == 128) && G <= 16;
}

cudaError_t launch_attn_mma(const tb_shape &sh, const uint16_t *q, const uint16_t *K, const uint16_t *V,
                            const int32_t *sel, const int32_t *counts, int32_t sel_stride, float scale, uint16_t *out,
                            uint32_t *attn_ctl, float *partials, int32_t *dev_status, cudaStream_t st) {
    const int rows = sh.B * sh.Hkv;
    if (rows <= 0) return cudaSuccess;
    if (!attn_mma_supported(sh)) return cudaErrorNotSupported;
    // splits of at least kAMTok entries, at most as many as the workspace holds
    int64_t split_tok = (sel_stride + kAttnMaxSplits - 1) / kAttnMaxSplits;
    if (split_tok < kAMTok) split_tok = kAMTok;
    const int64_t nsplit = (sel_stride + split_tok - 1) / split_tok;
    dim3 grid((unsigned)nsplit, (unsigned)rows);
    const size_t smem = attn_mma_smem_bytes(sh.D);
#define TB_AM_CASE(DTT)                                                                                      \
    do {                                                                                                     \
        cudaError_t e = cudaFuncSetAttribute(attn_mma_kernel<DTT>, cudaFuncAttributeMaxDynamicSharedMemorySize, \
                                             (int)smem);                                                     \
        if (e != cudaSuccess) return e;                                                                      \
        attn_mma_kernel<DTT><<<grid, kAMThreads, smem, st>>>(q, K, V, sel, counts, sel_stride, sh.cap, sh.Hq, \
                                                              sh.Hkv, scale, out, attn_ctl, partials,        \
                                                              (int)split_tok, dev_status);                   \
    } while (0)
    if (sh.D == 64) TB_AM_CASE(64);
    else TB_AM_CASE(128);
#undef TB_AM_CASE
    return cudaGetLastError();
}

}  // namespace tb
