// Exact attention over given selections, streamed ("TokenButler: Token
// Importance is Predictable": the full cache stays resident and only the
// selected tokens' K/V rows are read; gist.science summary, Optimizations:
// between predictions the same selection, plus the newest tokens, is reused).
//
// Grid (chunks, rows), two CTAs of four warps per SM: a CTA takes a
// contiguous slice of its row's selection, cut into chunks of 16 entries that
// its warps take in turn. Each warp streams its own chunks: its lanes issue
// the bulk copies of the chunk's K and V rows (one row per lane) onto the
// warp's own barrier, up to three chunks are in flight, and the oldest is
// attended on the tensor cores (attn_mma.cuh) by that warp alone, so the
// steady state has no CTA-wide barrier. The warps' softmax states are
// combined into the CTA's partial and the row's last CTA merges them. Entries
// outside [0, cap) are reported and masked (their slots read row 0 of the
// head).
#include "attn_mma.cuh"
#include "kernels.cuh"

namespace tb {

constexpr int kAsThreads = 128;
constexpr int kAsWarps = kAsThreads / 32;
constexpr int kAsChunk = 16;   // entries per warp chunk (one tensor-core tile of slots)
constexpr int kAsSets = 3;     // chunks in flight per warp

__host__ __device__ constexpr int attn_stream_smem_bytes(int DT) {
    return kAsSets * kAsWarps * kAsChunk * (4 * DT + 16)   // chunk buffers: set s holds warp w's chunk at w
           + 16 * (2 * DT + 16)                            // query tile
           + kAsSets * kAsWarps * kAsChunk;                // per-slot flags (valid entry)
}

template <int DT>
__global__ void __launch_bounds__(kAsThreads, 2) attn_stream_kernel(
    const uint16_t *__restrict__ q, const uint16_t *__restrict__ K, const uint16_t *__restrict__ V,
    const int32_t *__restrict__ sel, const int32_t *__restrict__ counts, int32_t sel_stride, int64_t cap, int Hq,
    int Hkv, float scale, uint16_t *__restrict__ out, uint32_t *__restrict__ attn_ctl, float *__restrict__ part,
    int per_cta, int32_t *dev_status) {
    extern __shared__ __align__(128) uint8_t smb[];
    __shared__ __align__(8) uint64_t bars[kAsSets][kAsWarps];
    __shared__ int s_abort;
    __shared__ uint32_t s_last;
    constexpr int SB = 4 * DT + 16, CPR = DT / 8, NT = DT / 8, QS = 2 * DT + 16;
    constexpr int SET = kAsWarps * kAsChunk;   // slots per set
    uint8_t *X = smb;
    uint8_t *qsm = X + kAsSets * SET * SB;
    uint8_t *flag = qsm + 16 * QS;
    const int G = Hq / Hkv;
    const int row = blockIdx.y, chunk = blockIdx.x, nchunk = gridDim.x;
    const int b = row / Hkv, h = row % Hkv;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint16_t *Kh = K + (int64_t)row * cap * DT;
    const uint16_t *Vh = V + (int64_t)row * cap * DT;
    const int32_t *srow = sel + (int64_t)row * sel_stride;

    const int cnt = counts ? counts[row] : sel_stride;
    const int cnt_c = cnt < 0 ? 0 : (cnt > sel_stride ? sel_stride : cnt);
    if (tid == 0 && chunk == 0 && (cnt <= 0 || cnt > sel_stride)) set_status(dev_status, TB_ERR_INVALID_ARG);
    const int j0 = chunk * per_cta;
    const int j1 = j0 + per_cta < cnt_c ? j0 + per_cta : cnt_c;
    const int nch = j1 > j0 ? (j1 - j0 + kAsChunk - 1) / kAsChunk : 0;   // chunks of the CTA's slice

    if (tid == 0) {
        s_abort = 0;
        for (int i = 0; i < kAsSets; ++i)
            for (int w = 0; w < kAsWarps; ++w) mbarrier_init(&bars[i][w], 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    // query tile: the G heads as rows of a 16-row bf16 tile (zero-padded); chunk buffers start zeroed, so a
    // padding slot always holds finite values (zeros or an earlier valid row)
    for (int x = tid; x < 16 * CPR; x += kAsThreads) {
        const int gq = x / CPR, cq = x % CPR;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (gq < G) v = *reinterpret_cast<const uint4 *>(q + ((int64_t)b * Hq + (int64_t)h * G + gq) * DT + cq * 8);
        *reinterpret_cast<uint4 *>(qsm + gq * QS + cq * 16) = v;
    }
    for (int x = tid; x < kAsSets * SET * SB / 16; x += kAsThreads)
        reinterpret_cast<uint4 *>(X)[x] = make_uint4(0u, 0u, 0u, 0u);
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncthreads();

    // every warp streams its own chunks (w, w + kAsWarps, ...) through its own slots of the kAsSets sets,
    // waiting only on its own barriers: lane l copies the K (even l) or V (odd l) row of entry l / 2
    uint32_t phase[kAsSets] = {};
    int c_issue = 0, c_done = 0;   // this warp's chunks issued / consumed
    const int my_chunks = nch > warp ? (nch - warp + kAsWarps - 1) / kAsWarps : 0;
    auto issue = [&]() {
        const int set = c_issue % kAsSets;
        const int e0 = j0 + (warp + c_issue * kAsWarps) * kAsChunk;
        const int c = j1 - e0 < kAsChunk ? j1 - e0 : kAsChunk;
        const int slot0 = set * SET + warp * kAsChunk;
        if (lane == 0) mbarrier_arrive_expect_tx(&bars[set][warp], (uint32_t)(c * 4 * DT));
        const int ent = lane >> 1;
        if (ent < c) {
            int64_t t = __ldg(srow + e0 + ent);
            const bool valid = t >= 0 && t < cap;
            if (!valid) t = 0;
            if ((lane & 1) == 0) {
                if (!valid) set_status(dev_status, TB_ERR_INVALID_ARG);
                flag[slot0 + ent] = valid ? 1 : 0;
            }
            uint8_t *dst = X + (size_t)(slot0 + ent) * SB + ((lane & 1) ? 2 * DT : 0);
            bulk_g2s(dst, ((lane & 1) ? Vh : Kh) + t * DT, 2 * DT, &bars[set][warp]);
        } else if ((lane & 1) == 0 && ent < kAsChunk) {
            flag[slot0 + ent] = 0;
        }
        ++c_issue;
    };

    MmaAttn<NT> A;
    A.m0 = A.m1 = -INFINITY;
    A.l0 = A.l1 = 0.f;
#pragma unroll
    for (int t = 0; t < NT; ++t) A.o[t][0] = A.o[t][1] = A.o[t][2] = A.o[t][3] = 0.f;
    const float qscale = scale * kLog2e;
    bool ok = true;
    while (c_issue < my_chunks && c_issue - c_done < kAsSets) issue();
    while (c_done < c_issue) {
        const int set = c_done % kAsSets;
        if (!mbarrier_wait_bounded(&bars[set][warp], phase[set], kWaitLimitNs)) {
            ok = false;
            set_status(dev_status, TB_ERR_TIMEOUT);
            break;
        }
        __syncwarp();
        phase[set] ^= 1u;
        const int e0 = j0 + (warp + c_done * kAsWarps) * kAsChunk;
        const int c = j1 - e0 < kAsChunk ? j1 - e0 : kAsChunk;
        // the set's tile of warp w is chunk w of the set: this warp attends it alone
        mma_attend<DT, kAsWarps, true>(A, X + (size_t)set * SET * SB, SB, warp * kAsChunk + c, flag, set * SET, qsm,
                                       qscale);
        __syncwarp();   // the chunk's slots are free again
        ++c_done;
        if (c_issue < my_chunks) issue();
    }
    if (!ok) {
        s_abort = 1;
        for (int r = c_done; r < c_issue; ++r)
            mbarrier_wait_bounded(&bars[r % kAsSets][warp], phase[r % kAsSets], kWaitLimitNs);
    }
    __syncthreads();
    if (s_abort) return;

    // the warps' states -> this chunk's partial (m, l, acc[D]) per head
    A.l0 += __shfl_xor_sync(0xFFFFFFFFu, A.l0, 1);
    A.l0 += __shfl_xor_sync(0xFFFFFFFFu, A.l0, 2);
    A.l1 += __shfl_xor_sync(0xFFFFFFFFu, A.l1, 1);
    A.l1 += __shfl_xor_sync(0xFFFFFFFFu, A.l1, 2);
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
    float *prow = part + (int64_t)row * nchunk * G * sg;
    for (int x = tid; x < G * DT; x += kAsThreads) {
        const int g = x / DT, d = x % DT;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kAsWarps; ++w) M = fmaxf(M, ws[((int64_t)w * G + g) * sg]);
        float L = 0.f, Acc = 0.f;
#pragma unroll
        for (int w = 0; w < kAsWarps; ++w) {
            const float *sw = ws + ((int64_t)w * G + g) * sg;
            const float wt = rescale_w(sw[0], M);
            L = fmaf(wt, sw[1], L);
            Acc = fmaf(wt, sw[2 + d], Acc);
        }
        float *o = prow + ((int64_t)chunk * G + g) * sg;
        if (d == 0) {
            o[0] = M;
            o[1] = L;
        }
        o[2 + d] = Acc;
    }
    // the last CTA of the row merges the chunks
    __syncthreads();
    if (tid == 0) {
        __threadfence();
        const uint32_t prev = atomicAdd(attn_ctl + row, 1u);
        s_last = prev == (uint32_t)(nchunk - 1) ? 1u : 0u;
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    attn_merge(prow, nchunk, G, DT, out + ((int64_t)b * Hq + (int64_t)h * G) * DT, dev_status,
               reinterpret_cast<float *>(X));
    if (tid == 0) attn_ctl[row] = 0;   // ready for the next call
}

bool attn_stream_supported(const tb_shape &sh) {
    const int G = sh.Hq / sh.Hkv;
    return (sh.D == 64 || sh.D == 128) && G <= 16;
}

cudaError_t launch_attn_stream(const tb_shape &sh, const uint16_t *q, const uint16_t *K, const uint16_t *V,
                               const int32_t *sel, const int32_t *counts, int32_t sel_stride, float scale,
                               uint16_t *out, uint32_t *attn_ctl, float *partials, int32_t *dev_status,
                               cudaStream_t st) {
    const int rows = sh.B * sh.Hkv;
    if (rows <= 0) return cudaSuccess;
    if (!attn_stream_supported(sh)) return cudaErrorNotSupported;
    // chunks: about two CTAs per SM over all rows, each at least one round, no more than the workspace's
    // partial slots (attn_splits(sel_stride) per row)
    const int sms = dev_info().sms > 0 ? dev_info().sms : 148;
    int64_t C = (2 * (int64_t)sms) / rows;
    const int64_t cmax = attn_splits(sel_stride);
    const int64_t cround = (sel_stride + kAsChunk * kAsWarps - 1) / (kAsChunk * kAsWarps);
    if (C > cmax) C = cmax;
    if (C > cround) C = cround;
    if (C < 1) C = 1;
    const int per = (int)((sel_stride + C - 1) / C);
    C = (sel_stride + per - 1) / per;
    dim3 grid((unsigned)C, (unsigned)rows);
    const size_t smem = (size_t)attn_stream_smem_bytes(sh.D);
    static thread_local int attr_dev[2] = {-1, -1};
    const int slot = sh.D == 64 ? 0 : 1;
    if (attr_dev[slot] != dev_info().device) {
        cudaError_t e = sh.D == 64 ? cudaFuncSetAttribute(attn_stream_kernel<64>,
                                                          cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)
                                   : cudaFuncSetAttribute(attn_stream_kernel<128>,
                                                          cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        attr_dev[slot] = dev_info().device;
    }
    if (sh.D == 64)
        attn_stream_kernel<64><<<grid, kAsThreads, smem, st>>>(q, K, V, sel, counts, sel_stride, sh.cap, sh.Hq, sh.Hkv,
                                                               scale, out, attn_ctl, partials, per, dev_status);
    else
        attn_stream_kernel<128><<<grid, kAsThreads, smem, st>>>(q, K, V, sel, counts, sel_stride, sh.cap, sh.Hq,
                                                                sh.Hkv, scale, out, attn_ctl, partials, per, dev_status);
    return cudaGetLastError();
}

}  // namespace tb
