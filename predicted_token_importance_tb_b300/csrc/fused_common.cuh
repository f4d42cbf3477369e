// Pieces shared by the single-launch decode-step kernels ("TokenButler: Token
// Importance is Predictable": project the new key, score every cached token,
// keep a fixed per-token budget, attend over only the kept rows).
//
//  - step_append_project: the CTA owning the new token writes K_new / V_new
//    into the cache and projects K_new into its Kp row (fp32 sum, one RNE).
//  - chunk_select_attend: exact top-k of a row split into contiguous chunks
//    (topk_core.cuh), attending the kept tokens of this CTA's chunk and
//    writing them, ascending, to idx and sel.
//  - row_finish: this CTA's partial softmax state goes to the workspace; the
//    row's last CTA merges the partials into the output rows and puts the
//    row's control words back to zero.
#pragma once

#include "attn_core.cuh"
#include "topk_core.cuh"

namespace tb {

// Scratch floats attn_block_combine needs for nthreads threads.
__host__ __device__ inline int comb_floats_for(int nthreads, int G, int D) {
    const int f = (nthreads / 32) * G * (2 + D);
    return f > nthreads ? f : nthreads;
}

// The step's append, split in two so the loads can fly while other work runs:
// append_issue loads this thread's slice of Wk and its element of K_new and
// V_new into registers; append_finish writes the K/V row into the cache and
// projects the key into its Kp row: thread (j, slice) accumulates output j
// over a slice of D in fp32, the slices are summed in comb and the sum is
// rounded once to bf16. knew [D] and kpn [dp] (shared fp32) receive the new
// key and its projected row; comb is shared scratch of blockDim.x floats.
constexpr int kAppendW = 8;   // Wk values a thread keeps in registers

struct AppendRegs {
    uint16_t wv[kAppendW];
    uint16_t kb, vb;
};

__device__ __forceinline__ AppendRegs append_issue(const uint16_t *K_new, const uint16_t *V_new, const uint16_t *Wk,
                                                   int row, int h, int D, int dp) {
    AppendRegs r;
    const uint16_t *W = Wk + (int64_t)h * D * dp;
    const int jn = dp < (int)blockDim.x ? dp : (int)blockDim.x;
    const int slices = blockDim.x / jn;
    const int dlen = (D + slices - 1) / slices;
    const int j = threadIdx.x % jn, sl = threadIdx.x / jn;
    const int d0 = sl * dlen, d1 = min(D, d0 + dlen);
#pragma unroll
    for (int u = 0; u < kAppendW; ++u) r.wv[u] = (sl < slices && d0 + u < d1) ? W[(int64_t)(d0 + u) * dp + j] : (uint16_t)0;
    r.kb = (int)threadIdx.x < D ? K_new[(int64_t)row * D + threadIdx.x] : (uint16_t)0;
    r.vb = (int)threadIdx.x < D ? V_new[(int64_t)row * D + threadIdx.x] : (uint16_t)0;
    return r;
}

// All threads of the CTA must call it.
__device__ __forceinline__ void append_finish(const AppendRegs &r, const uint16_t *K_new, const uint16_t *V_new,
                                              const uint16_t *Wk, uint16_t *K, uint16_t *V, uint16_t *Kp,
                                              int64_t cap, int64_t n, int row, int h, int D, int dp, float *knew,
                                              float *kpn, float *comb) {
    uint16_t *Kr = K + ((int64_t)row * cap + n) * D;
    uint16_t *Vr = V + ((int64_t)row * cap + n) * D;
    for (int d = threadIdx.x; d < D; d += blockDim.x) {
        const uint16_t k2 = d == (int)threadIdx.x ? r.kb : K_new[(int64_t)row * D + d];
        const uint16_t v2 = d == (int)threadIdx.x ? r.vb : V_new[(int64_t)row * D + d];
        knew[d] = bf16_to_f(k2);
        Kr[d] = k2;
        Vr[d] = v2;
    }
    __syncthreads();
    const uint16_t *W = Wk + (int64_t)h * D * dp;
    const int jn = dp < (int)blockDim.x ? dp : (int)blockDim.x;
    const int slices = blockDim.x / jn;
    const int dlen = (D + slices - 1) / slices;
    const int j = threadIdx.x % jn, sl = threadIdx.x / jn;
    const int d0 = sl * dlen, d1 = min(D, d0 + dlen);
    if (sl < slices) {
        float acc = 0.f;
#pragma unroll
        for (int u = 0; u < kAppendW; ++u)
            if (d0 + u < d1) acc = fmaf(knew[d0 + u], bf16_to_f(r.wv[u]), acc);
        for (int d = d0 + kAppendW; d < d1; ++d) acc = fmaf(knew[d], bf16_to_f(W[(int64_t)d * dp + j]), acc);
        comb[sl * jn + j] = acc;
    }
    __syncthreads();
    if (threadIdx.x < dp) {
        float s = 0.f;
        for (int x = 0; x < slices; ++x) s += comb[x * jn + threadIdx.x];
        const uint16_t pb = f_to_bf16(s);
        Kp[((int64_t)row * cap + n) * dp + threadIdx.x] = pb;
        kpn[threadIdx.x] = bf16_to_f(pb);
    }
    __syncthreads();
}

// Both halves back to back. All threads of the CTA must call it.
__device__ __forceinline__ void step_append_project(const uint16_t *K_new, const uint16_t *V_new, const uint16_t *Wk,
                                                    uint16_t *K, uint16_t *V, uint16_t *Kp, int64_t cap, int64_t n,
                                                    int row, int h, int D, int dp, float *knew, float *kpn,
                                                    float *comb) {
    const AppendRegs r = append_issue(K_new, V_new, Wk, row, h, D, dp);
    append_finish(r, K_new, V_new, Wk, K, V, Kp, cap, n, row, h, D, dp, knew, kpn, comb);
}

// Exact selection over contiguous chunks plus attention over this CTA's kept
// tokens. S.keys[0..Lc) hold the keys of tokens t0 .. t0+Lc-1 (chunk c of C,
// chunk length L); list is shared scratch of L ints. irow / srow receive the
// row's kept tokens in ascending order. bar_base: phases of rc->bar already
// completed in this launch. Returns false when a group wait timed out.
template <int GM>
__device__ bool chunk_select_attend(AttnLane<GM> &A, RowCtl *rc, SelectSmem &S, int32_t *list, int Lc, int L, int c,
                                    int C, int bar_base, uint32_t k, int64_t t0, const uint16_t *Kh,
                                    const uint16_t *Vh, int64_t cap, int G, int D, int32_t *irow, int32_t *srow,
                                    int32_t *dev_status) {
    SelectBegin B = group_select_begin(rc, S, Lc, L, c, C, k, dev_status, bar_base);
    if (!B.ok) return false;
    // tokens above the threshold bin are kept whatever the exact threshold:
    // attend them while the last selection barrier completes
    uint32_t n_above = 0;
    for (int e0 = 0; e0 < Lc; e0 += blockDim.x) {
        const int e = e0 + threadIdx.x;
        const uint32_t f = (e < Lc && above_bin(B, S.keys[e])) ? 1u : 0u;
        uint32_t tot;
        const uint32_t pos = block_exclusive_scan(f, S.scan, tot);
        if (f) list[n_above + pos] = e;
        n_above += tot;
    }
    __syncthreads();
    attn_tokens(A, G, D, (int)n_above, [&](int j) -> int64_t { return t0 + list[j]; }, Kh, Vh, cap, dev_status);
    __syncthreads();
    // exact threshold; kept tokens out (ascending); attend the kept bin tokens
    SelectResult R = group_select_end(rc, S, B, L, c, C, dev_status);
    if (!R.ok) return false;
    uint32_t base_kept = 0, base_tied = 0, n_bin = 0;
    for (int e0 = 0; e0 < Lc; e0 += blockDim.x) {
        const int e = e0 + threadIdx.x;
        uint32_t key = 0, tied = 0;
        if (e < Lc) {
            key = S.keys[e];
            tied = (R.mode == 1 && key == R.tkey) ? 1u : 0u;
        }
        uint32_t ttot;
        const uint32_t tied_before = base_tied + block_exclusive_scan(tied, S.scan, ttot);
        const bool kept = e < Lc && is_kept(R, key, (uint32_t)(t0 + e), tied_before);
        const uint32_t kf = kept ? 1u : 0u;
        const uint32_t bf = (kept && !above_bin(B, key)) ? 1u : 0u;
        uint32_t ktot, btot;
        const uint32_t pos = block_exclusive_scan(kf, S.scan, ktot);
        const uint32_t bpos = block_exclusive_scan(bf, S.scan, btot);
        if (kept) {
            const uint32_t slot = R.offset + base_kept + pos;
            if (irow) irow[slot] = (int32_t)(t0 + e);
            srow[slot] = (int32_t)(t0 + e);
        }
        if (bf) list[n_bin + bpos] = e;
        base_kept += ktot;
        base_tied += ttot;
        n_bin += btot;
    }
    __syncthreads();
    attn_tokens(A, G, D, (int)n_bin, [&](int j) -> int64_t { return t0 + list[j]; }, Kh, Vh, cap, dev_status);
    return true;
}

// The row's last CTA to finish merges the C partial states (this CTA's is
// already stored at prow + c * G * (2 + D)) into the G output rows and
// resets the row's control block (the radix histograms and candidate count
// only when reset_hist). msm: shared scratch of 2*C*G + G floats; flag: one
// shared word. All threads of the CTA must call it.
__device__ __forceinline__ void row_merge_tail(RowCtl *rc, const float *prow, int C, int G, int D,
                                               uint16_t *out_rows, float *msm, uint32_t *flag, bool reset_hist,
                                               int32_t *dev_status) {
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        const uint32_t prev = atomicAdd(&rc->done, 1u);
        *flag = (prev == (uint32_t)(C - 1)) ? 1u : 0u;
    }
    __syncthreads();
    if (!*flag) return;
    __threadfence();
    attn_merge(prow, C, G, D, out_rows, dev_status, msm);
    if (reset_hist)
        for (int x = threadIdx.x; x < 3 * kRadixBins; x += blockDim.x) (&rc->hist[0][0])[x] = 0;
    if (threadIdx.x == 0) {
        rc->bar = 0;
        rc->ncand = 0;
        rc->done = 0;
    }
}

// The row's last-arriving CTA merges the C partial states (m, l, acc[D]) per
// head into out_rows ([G][D] bf16) and resets the row's control words; the
// others return false at once. Arrival is one acq_rel atomic by thread 0
// (release of the CTA's partial, acquire of the others' for the merger),
// ordered with the CTA's other threads by the barriers around it. The merger
// requests its first accumulators before the weights are known (one round
// trip for up to 32 chunks), then weights exp2(m_c - M) and w l per (chunk,
// head) go to
// `scratch` (4 C G floats of shared memory). Returns true in the CTA that
// merged; that CTA also resets the row's control words (and the radix
// histograms when reset_hist). flag: one shared word. All threads call it.
__device__ __forceinline__ bool row_merge_last(RowCtl *rc, const float *prow, int C, int G, int D,
                                               uint16_t *out_rows, uint32_t *flag, bool reset_hist,
                                               int32_t *dev_status, float *scratch) {
    constexpr int kBatch = 32;   // chunks per round trip
    __syncthreads();
    if (threadIdx.x == 0) {
        uint32_t prev;
        asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(prev) : "l"(&rc->done) : "memory");
        *flag = (prev == (uint32_t)(C - 1)) ? 1u : 0u;
    }
    __syncthreads();
    if (!*flag) return false;
    const int sg = 2 + D, CG = C * G;
    float *ms = scratch, *ls = scratch + CG, *wt = scratch + 2 * CG, *wl = scratch + 3 * CG;
    // a thread per output (g, d); its first batch of accumulators is
    // requested before the weights are known
    const int x0 = threadIdx.x;
    const bool act0 = x0 < G * D;
    const int g0 = act0 ? x0 / D : 0, d0 = act0 ? x0 % D : 0;
    float av[kBatch];
#pragma unroll
    for (int u = 0; u < kBatch; ++u) av[u] = (act0 && u < C) ? __ldcg(prow + (u * G + g0) * sg + 2 + d0) : 0.f;
    for (int y = threadIdx.x; y < CG; y += blockDim.x) {
        ms[y] = __ldcg(prow + (int64_t)y * sg);
        ls[y] = __ldcg(prow + (int64_t)y * sg + 1);
    }
    __syncthreads();
    for (int y = threadIdx.x; y < CG; y += blockDim.x) {
        const int g = y % G;
        float M = -INFINITY;
        for (int u0 = 0; u0 < C; u0 += kBatch) {
#pragma unroll
            for (int u = 0; u < kBatch; ++u)
                if (u0 + u < C) M = fmaxf(M, ms[(u0 + u) * G + g]);
        }
        const float w = rescale_w(ms[y], M);
        wt[y] = w;
        wl[y] = w * ls[y];
    }
    __syncthreads();
    for (int x = x0; x < G * D; x += blockDim.x) {
        const int g = x / D, d = x % D;
        float L = 0.f, Acc = 0.f;
        for (int u0 = 0; u0 < C; u0 += kBatch) {
            if (x != x0 || u0 != 0) {
#pragma unroll
                for (int u = 0; u < kBatch; ++u)
                    av[u] = u0 + u < C ? __ldcg(prow + ((int64_t)(u0 + u) * G + g) * sg + 2 + d) : 0.f;
            }
#pragma unroll
            for (int u = 0; u < kBatch; ++u) {
                if (u0 + u < C) {
                    L += wl[(u0 + u) * G + g];
                    Acc = fmaf(wt[(u0 + u) * G + g], av[u], Acc);
                }
            }
        }
        if (!(L > 0.f)) set_status(dev_status, TB_ERR_INVALID_ARG);
        out_rows[(int64_t)g * D + d] = f_to_bf16(L > 0.f ? Acc / L : 0.f);
    }
    if (reset_hist)
        for (int x = threadIdx.x; x < 3 * kRadixBins; x += blockDim.x) (&rc->hist[0][0])[x] = 0;
    if (threadIdx.x == 0) {
        rc->bar = 0;
        rc->ncand = 0;
        rc->done = 0;
    }
    return true;
}

// Partial state of this CTA -> workspace, then row_merge_tail.
// comb: shared scratch of comb_floats_for(blockDim.x, G, D) floats.
template <int GM>
__device__ void row_finish(AttnLane<GM> &A, RowCtl *rc, float *prow, int c, int C, int G, int D, uint16_t *out_rows,
                           float *comb, float *msm, uint32_t *flag, bool reset_hist, int32_t *dev_status) {
    attn_block_combine(A, G, D, comb, prow + (int64_t)c * G * (2 + D));
    row_merge_tail(rc, prow, C, G, D, out_rows, msm, flag, reset_hist, dev_status);
}

}  // namespace tb
