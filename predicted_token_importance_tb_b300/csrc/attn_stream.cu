// Exact attention over given selections, streamed ("TokenButler: Token
// Importance is Predictable": the full cache stays resident and only the
// selected tokens' K/V rows are read; gist.science summary, Optimizations:
// between predictions the same selection, plus the newest tokens, is reused).
//
// Grid (C, rows) of four-warp CTAs: the C CTAs of a row split its realised
// count into equal slices of whole 16-entry chunks that their warps take in
// turn. Each warp streams its own chunks: its lanes copy the chunk's K and V
// rows in 16-byte pieces (cp.async, one commit group per chunk) and the oldest
// landed chunk is attended on the tensor cores by that warp alone, so the
// steady state has no CTA-wide barrier. (One bulk copy per 256-byte row was
// tried first: the per-copy cost of the bulk-copy unit held each SM to about
// 20 GB/s.) With at most eight heads per KV head the keys are the MMA rows
// (kt_attend); otherwise the heads are (attn_mma.cuh). Three CTAs per SM with
// two chunks in flight per warp, or two CTAs with three. The warps' softmax
// states are combined into the CTA's partial; a row of up to eight CTAs is one
// thread-block cluster that merges the partials through distributed shared
// memory, a larger row's last CTA merges them from the workspace. Entries
// outside [0, cap) are reported and masked (their slots read row 0 of the
// head).
#include "attn_mma.cuh"
#include "kernels.cuh"

namespace tb {

constexpr int kAsThreads = 128;
constexpr int kAsWarps = kAsThreads / 32;
constexpr int kAsChunk = 16;   // entries per warp chunk (one tensor-core tile of slots)
constexpr int kAsClusterMax = 8;   // most CTAs per row that merge as one cluster (the portable cluster size; 9-CTA
                                   // clusters measured slower: they pack poorly onto the GPCs)

// SETS: chunks in flight per warp.
__host__ __device__ constexpr int attn_stream_smem_bytes(int DT, int SETS) {
    return SETS * kAsWarps * kAsChunk * (4 * DT + 16)   // chunk buffers: set s holds warp w's chunk at w
           + 16 * (2 * DT + 16)                         // query tile
           + SETS * kAsWarps * kAsChunk;                // per-slot flags (valid entry)
}

// Barrier over the CTAs of a thread-block cluster (release / acquire of their shared memory).
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// fp32 load from the shared memory of CTA `rank` of this cluster, at the address `a` has in this CTA.
__device__ __forceinline__ float ld_cluster_f32(uint32_t a, int rank) {
    uint32_t r;
    float v;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(rank));
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(r) : "memory");
    return v;
}

// 16-byte asynchronous copy global -> shared, destination given as a shared-window address.
__device__ __forceinline__ void cp_async16_sa(uint32_t dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}

// Transpose of an 8x8 b16 matrix held in the mma fragment layout (row lane/4, columns 2(lane%4) and +1).
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t a) {
    uint32_t d;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(a));
    return d;
}

// Attention state of one warp with the keys as the MMA rows: S^T = K Q^T (16 keys x 8 heads per chunk) and
// O^T += V^T P^T (DT/16 tiles of 16 dims x 8 heads). Lane l holds heads 2(l%4) and 2(l%4)+1 (at most 8
// heads, zero-padded), the running maxima of those heads (exp2 domain, equal across the lanes that share
// l%4) and partial sums over its own keys (summed across lanes at the end).
template <int DT>
struct KtAttn {
    float m0, m1, l0, l1;
    float o[DT / 16][4];
    uint32_t qb[DT / 16][2];   // Q^T as the B operand, one pair per 16-dim step
};

// One chunk of 16 staged slots (K row at xs + s*SB, V row at +2*DT) on the tensor cores; slots whose flag
// is zero are masked (their V rows must hold finite values).
template <int DT>
__device__ __forceinline__ void kt_attend(KtAttn<DT> &A, uint32_t xs, int SB, const uint8_t *flag, float qscale) {
    constexpr int KS = DT / 16;
    const int lane = threadIdx.x & 31;
    float s[4] = {0.f, 0.f, 0.f, 0.f}, t[4] = {0.f, 0.f, 0.f, 0.f};   // even / odd k-steps
    const uint32_t ka = xs + (uint32_t)((lane & 7) + 8 * ((lane >> 3) & 1)) * SB + 16 * (lane >> 4);
#pragma unroll
    for (int kk = 0; kk < KS; kk += 2) {
        uint32_t a0, a1, a2, a3, e0, e1, e2, e3;
        ldsm_x4(ka + kk * 32, a0, a1, a2, a3);
        ldsm_x4(ka + kk * 32 + 32, e0, e1, e2, e3);
        mma_bf16_16816(s, a0, a1, a2, a3, A.qb[kk][0], A.qb[kk][1]);
        mma_bf16_16816(t, e0, e1, e2, e3, A.qb[kk + 1][0], A.qb[kk + 1][1]);
    }
    // keys k = lane/4 and k + 8; heads h0 = 2(lane%4), h1 = h0 + 1
    const int k0 = lane >> 2;
    const bool f0 = flag[k0] != 0, f8 = flag[k0 + 8] != 0;
    const float z00 = f0 ? (s[0] + t[0]) * qscale : -INFINITY, z01 = f0 ? (s[1] + t[1]) * qscale : -INFINITY;
    const float z80 = f8 ? (s[2] + t[2]) * qscale : -INFINITY, z81 = f8 ? (s[3] + t[3]) * qscale : -INFINITY;
    float mx0 = fmaxf(z00, z80), mx1 = fmaxf(z01, z81);
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xFFFFFFFFu, mx0, off));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xFFFFFFFFu, mx1, off));
    }
    const float n0 = fmaxf(A.m0, mx0), n1 = fmaxf(A.m1, mx1);
    const float c0 = n0 == -INFINITY ? 1.f : exp2f(A.m0 - n0);
    const float c1 = n1 == -INFINITY ? 1.f : exp2f(A.m1 - n1);
    const float p00 = n0 == -INFINITY ? 0.f : exp2f(z00 - n0), p80 = n0 == -INFINITY ? 0.f : exp2f(z80 - n0);
    const float p01 = n1 == -INFINITY ? 0.f : exp2f(z01 - n1), p81 = n1 == -INFINITY ? 0.f : exp2f(z81 - n1);
    A.l0 = A.l0 * c0 + (p00 + p80);
    A.l1 = A.l1 * c1 + (p01 + p81);
    A.m0 = n0;
    A.m1 = n1;
    if (__any_sync(0xFFFFFFFFu, c0 != 1.f || c1 != 1.f)) {
#pragma unroll
        for (int mt = 0; mt < KS; ++mt) {
            A.o[mt][0] *= c0;
            A.o[mt][1] *= c1;
            A.o[mt][2] *= c0;
            A.o[mt][3] *= c1;
        }
    }
    // P^T as the B operand: the transposes of the two 8x8 blocks (keys 0-7, 8-15) of P[key][head]
    const uint32_t b0 = movmatrix_trans(pack_bf16x2(p00, p01));
    const uint32_t b1 = movmatrix_trans(pack_bf16x2(p80, p81));
    // V^T tiles from the V rows by transposed loads: lanes address keys (lane&7) + 8(lane>>4), dims +8((lane>>3)&1)
    const uint32_t va = xs + (uint32_t)((lane & 7) + 8 * (lane >> 4)) * SB + 2 * DT + 16 * ((lane >> 3) & 1);
#pragma unroll
    for (int mt = 0; mt < KS; ++mt) {
        uint32_t a0, a1, a2, a3;
        ldsm_x4_trans(va + mt * 32, a0, a1, a2, a3);
        mma_bf16_16816(A.o[mt], a0, a1, a2, a3, b0, b1);
    }
}


// Merge of nsplit partials (m, l, acc[DT] per head, fp32) into one row's G output heads (bf16). Every thread
// takes up to four outputs and issues their values of eight partials at once, and the maxima and sums go to
// shared memory while the first values are in flight, so a merge of up to eight partials is one round trip
// to L2. sm holds 2 * nsplit * G floats.
template <int DT>
__device__ __forceinline__ void stream_merge(const float *__restrict__ part, int nsplit, int G,
                                             uint16_t *__restrict__ out_rows, int32_t *dev_status, float *sm) {
    constexpr int kU = 4, kB = 8;
    const int sg = 2 + DT, tid = threadIdx.x, no = G * DT;
    float *ms = sm, *ls = sm + nsplit * G;
    for (int x0 = 0; x0 < no; x0 += kAsThreads * kU) {
        float M[kU], L[kU], Acc[kU];
        int g[kU], d[kU];
        bool act[kU];
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            const int x = x0 + tid + u * kAsThreads;
            act[u] = x < no;
            g[u] = act[u] ? x / DT : 0;
            d[u] = act[u] ? x % DT : 0;
            M[u] = -INFINITY;
            L[u] = Acc[u] = 0.f;
        }
        for (int s0 = 0; s0 < nsplit; s0 += kB) {
            float av[kU][kB];
#pragma unroll
            for (int u = 0; u < kU; ++u)
#pragma unroll
                for (int b = 0; b < kB; ++b)
                    av[u][b] = (act[u] && s0 + b < nsplit)
                                   ? __ldcg(part + ((int64_t)(s0 + b) * G + g[u]) * sg + 2 + d[u])
                                   : 0.f;
            if (x0 == 0 && s0 == 0) {   // the maxima and sums, while the first values are in flight
                for (int i = tid; i < nsplit * G; i += kAsThreads) {
                    ms[i] = __ldcg(part + (int64_t)i * sg);
                    ls[i] = __ldcg(part + (int64_t)i * sg + 1);
                }
                __syncthreads();
            }
#pragma unroll
            for (int u = 0; u < kU; ++u) {
                float Mb = M[u];
#pragma unroll
                for (int b = 0; b < kB; ++b)
                    if (s0 + b < nsplit) Mb = fmaxf(Mb, ms[(s0 + b) * G + g[u]]);
                const float r = rescale_w(M[u], Mb);
                L[u] *= r;
                Acc[u] *= r;
#pragma unroll
                for (int b = 0; b < kB; ++b) {
                    if (s0 + b < nsplit) {
                        const float w = rescale_w(ms[(s0 + b) * G + g[u]], Mb);
                        L[u] = fmaf(w, ls[(s0 + b) * G + g[u]], L[u]);
                        Acc[u] = fmaf(w, av[u][b], Acc[u]);
                    }
                }
                M[u] = Mb;
            }
        }
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            if (act[u]) {
                if (!(L[u] > 0.f)) set_status(dev_status, TB_ERR_INVALID_ARG);
                out_rows[(int64_t)g[u] * DT + d[u]] = f_to_bf16(L[u] > 0.f ? Acc[u] / L[u] : 0.f);
            }
        }
    }
}

// Grid (C, rows): CTA c of a row takes the c-th of C equal slices (whole chunks of 16) of the row's realised
// count, whose chunks its warps take in turn. The warps' states are combined into the CTA's partial
// (m, l, acc[D] per head). SETS chunks in flight per warp, MINB CTAs per SM. app.pos >= 0: a step inside a
// prediction interval (see AttnAppend). CL: the row's C CTAs are one cluster, keep their partials in shared memory
// and each merges a slice of the outputs through distributed shared memory; otherwise the partials go to the
// workspace and the row's last arriving CTA merges them. KT: keys as the MMA rows (G <= 8); otherwise the G
// heads are the rows (G <= 16).
template <int DT, bool KT, int SETS, int MINB, bool CL>
__global__ void __launch_bounds__(kAsThreads, MINB) attn_stream_kernel(
    const uint16_t *__restrict__ q, const uint16_t *__restrict__ K, const uint16_t *__restrict__ V,
    const int32_t *__restrict__ sel, const int32_t *__restrict__ counts, int32_t sel_stride, int64_t cap, int Hq,
    int Hkv, float scale, uint16_t *__restrict__ out, uint32_t *__restrict__ attn_ctl,
    float *__restrict__ part, int32_t *dev_status, AttnAppend app) {
    extern __shared__ __align__(128) uint8_t smb[];
    __shared__ uint32_t s_last;
    constexpr int SB = 4 * DT + 16, CPR = DT / 8, NT = DT / 8, QS = 2 * DT + 16;
    constexpr int SET = kAsWarps * kAsChunk;   // slots per set
    uint8_t *X = smb;
    uint8_t *qsm = X + SETS * SET * SB;
    uint8_t *flag = qsm + 16 * QS;
    const int G = Hq / Hkv;
    const int sg = 2 + DT;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int row = blockIdx.y, chunk = blockIdx.x, nchunk = gridDim.x;
    const int b = row / Hkv, h = row % Hkv;

    const int cnt0 = counts ? counts[row] : sel_stride;
    // with an append, the new token is entry cnt0 (its K/V rows read from K_new / V_new) when there is room
    const bool room = app.pos >= 0 && cnt0 >= 0 && cnt0 < sel_stride;
    const int cnt = room ? cnt0 + 1 : cnt0;
    const int new_e = room ? cnt0 : -1;
    const int cnt_c = cnt < 0 ? 0 : (cnt > sel_stride ? sel_stride : cnt);
    if (tid == 0 && chunk == 0 && ((app.pos >= 0 && !room) || cnt <= 0 || cnt > sel_stride))
        set_status(dev_status, TB_ERR_INVALID_ARG);
    // equal slices of the row's realised count, in whole chunks
    const int per = ((cnt_c + nchunk - 1) / nchunk + kAsChunk - 1) / kAsChunk * kAsChunk;
    const int j0 = chunk * per;
    const int j1 = j0 + per < cnt_c ? j0 + per : cnt_c;
    const int nch = j1 > j0 ? (j1 - j0 + kAsChunk - 1) / kAsChunk : 0;   // chunks of the CTA's slice

    constexpr int P = DT / 8;          // 16-byte pieces of a K or V row
    constexpr int LPE = 2 * P;         // lanes per entry (its K and V pieces)
    constexpr int EPI = 32 / LPE;      // entries per copy instruction of the warp
    const int pr = lane % LPE;
    const bool pv = pr >= P;
    const uint32_t xs = smem_addr(X);
    const uint32_t dst_lane = (uint32_t)((lane / LPE) * SB + (pv ? 2 * DT : 0) + (pv ? pr - P : pr) * 16);
    const uint16_t *src = (pv ? V : K) + (int64_t)row * cap * DT + (pv ? pr - P : pr) * 8;
    const uint16_t *src_new = app.pos >= 0 ? (pv ? app.V_new : app.K_new) + (int64_t)row * DT + (pv ? pr - P : pr) * 8
                                           : src;
    const int32_t *srow = sel + (int64_t)row * sel_stride;
    const float qscale = scale * kLog2e;

    // every warp streams its own chunks (w, w + kAsWarps, ...) through its own slots of the SETS sets: the
    // lanes copy the chunk's K and V rows in 16-byte pieces (cp.async, one commit group per chunk) and wait for
    // their own groups only. Lane l holds the selection entry l % 16 of the next two chunks to issue, loaded
    // ahead so that their latency overlaps the copies and the attention before them.
    int c_issue = 0, c_done = 0;   // this warp's chunks issued / consumed
    const int my_chunks = nch > warp ? (nch - warp + kAsWarps - 1) / kAsWarps : 0;
    auto load_idx = [&](int kk) -> int32_t {   // entry lane % 16 of this warp's chunk kk, -1 past the slice
        const int e = j0 + (warp + kk * kAsWarps) * kAsChunk + (lane & (kAsChunk - 1));
        return (kk < my_chunks && e < j1) ? (e == new_e ? (int32_t)app.pos : __ldg(srow + e)) : -1;
    };
    int32_t pidx = load_idx(0), pnext = load_idx(1);
    auto issue = [&]() {
        const int e0 = j0 + (warp + c_issue * kAsWarps) * kAsChunk;
        const int cc = j1 - e0 < kAsChunk ? j1 - e0 : kAsChunk;
        const int slot0 = (c_issue % SETS) * SET + warp * kAsChunk;
        const bool valid_l = pidx >= 0 && (int64_t)pidx < cap;
        if (lane < kAsChunk) {
            if (lane < cc && !valid_l) set_status(dev_status, TB_ERR_INVALID_ARG);
            flag[slot0 + lane] = (lane < cc && valid_l) ? 1 : 0;
        }
        const int32_t tl = valid_l ? pidx : 0;
        const uint32_t dst0 = xs + (uint32_t)slot0 * SB + dst_lane;
#pragma unroll
        for (int it = 0; it < kAsChunk / EPI; ++it) {
            const int ent = it * EPI + lane / LPE;
            const int32_t t = __shfl_sync(0xFFFFFFFFu, tl, ent);
            if (ent < cc)
                cp_async16_sa(dst0 + (uint32_t)(it * EPI * SB), e0 + ent == new_e ? src_new : src + (int64_t)t * DT);
            else if (pv)   // a padding slot's V row must hold finite values (its weight is zero)
                asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(dst0 + (uint32_t)(it * EPI * SB)),
                             "r"(0u)
                             : "memory");
        }
        cp_async_commit();
        ++c_issue;
        pidx = pnext;
        pnext = load_idx(c_issue + 1);
    };

    // the first chunks are in flight before the query tile is loaded
    while (c_issue < my_chunks && c_issue - c_done < SETS) issue();
    // query tile: the G heads as rows of a 16-row bf16 tile (zero-padded)
    for (int x = tid; x < 16 * CPR; x += kAsThreads) {
        const int gq = x / CPR, cq = x % CPR;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (gq < G) v = *reinterpret_cast<const uint4 *>(q + ((int64_t)b * Hq + (int64_t)h * G + gq) * DT + cq * 8);
        *reinterpret_cast<uint4 *>(qsm + gq * QS + cq * 16) = v;
    }
    __syncthreads();

    MmaAttn<NT> A{};   // heads-as-rows state (KT = false)
    KtAttn<DT> B{};    // keys-as-rows state (KT = true)
    if constexpr (KT) {
        B.m0 = B.m1 = -INFINITY;
#pragma unroll
        for (int mt = 0; mt < DT / 16; ++mt) {
            const uint8_t *qr = qsm + (lane >> 2) * QS + (mt * 16 + 2 * (lane & 3)) * 2;
            B.qb[mt][0] = *reinterpret_cast<const uint32_t *>(qr);
            B.qb[mt][1] = *reinterpret_cast<const uint32_t *>(qr + 16);
        }
    } else {
        A.m0 = A.m1 = -INFINITY;
    }
    while (c_done < c_issue) {
        const int set = c_done % SETS;
        // this lane's pieces of chunk c_done have landed once at most c_issue - c_done - 1 groups are pending
        const int pend = c_issue - c_done - 1;
        if (pend >= 2) asm volatile("cp.async.wait_group 2;" ::: "memory");
        else if (pend == 1) asm volatile("cp.async.wait_group 1;" ::: "memory");
        else asm volatile("cp.async.wait_group 0;" ::: "memory");
        __syncwarp();   // every lane's pieces of the chunk are visible to the warp
        // the set's tile of warp w is chunk w of the set: this warp attends it alone
        if constexpr (KT) {
            kt_attend<DT>(B, xs + (uint32_t)(set * SET + warp * kAsChunk) * SB, SB, flag + set * SET + warp * kAsChunk,
                          qscale);
        } else {
            const int e0 = j0 + (warp + c_done * kAsWarps) * kAsChunk;
            const int cc = j1 - e0 < kAsChunk ? j1 - e0 : kAsChunk;
            mma_attend<DT, kAsWarps, true>(A, X + (size_t)set * SET * SB, SB, warp * kAsChunk + cc, flag, set * SET,
                                           qsm, qscale);
        }
        __syncwarp();   // the chunk's slots are free again
        ++c_done;
        if (c_issue < my_chunks) issue();
    }
    __syncthreads();   // every warp is done with the chunk buffers

    // the warps' states -> shared memory -> this CTA's partial (m, l, acc[D]) per head
    float *ws = reinterpret_cast<float *>(X);
    if constexpr (KT) {
        float l0 = B.l0, l1 = B.l1;
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
            l0 += __shfl_xor_sync(0xFFFFFFFFu, l0, off);
            l1 += __shfl_xor_sync(0xFFFFFFFFu, l1, off);
        }
        const int dr = lane >> 2;
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int g = 2 * (lane & 3) + j;
            if (g < G) {
                float *w = ws + ((int64_t)warp * G + g) * sg;
                if (lane < 4) {
                    w[0] = j ? B.m1 : B.m0;
                    w[1] = j ? l1 : l0;
                }
#pragma unroll
                for (int mt = 0; mt < DT / 16; ++mt) {
                    w[2 + mt * 16 + dr] = B.o[mt][j];
                    w[2 + mt * 16 + dr + 8] = B.o[mt][2 + j];
                }
            }
        }
    } else {
        float l0 = A.l0, l1 = A.l1;
        l0 += __shfl_xor_sync(0xFFFFFFFFu, l0, 1);
        l0 += __shfl_xor_sync(0xFFFFFFFFu, l0, 2);
        l1 += __shfl_xor_sync(0xFFFFFFFFu, l1, 1);
        l1 += __shfl_xor_sync(0xFFFFFFFFu, l1, 2);
        const int g0 = lane >> 2, d0 = 2 * (lane & 3);
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            const int g = g0 + 8 * half;
            if (g < G) {
                float *w = ws + ((int64_t)warp * G + g) * sg;
                if ((lane & 3) == 0) {
                    w[0] = half ? A.m1 : A.m0;
                    w[1] = half ? l1 : l0;
                }
#pragma unroll
                for (int t = 0; t < NT; ++t)
                    *reinterpret_cast<float2 *>(w + 2 + 8 * t + d0) = make_float2(A.o[t][2 * half], A.o[t][2 * half + 1]);
            }
        }
    }
    __syncthreads();
    if constexpr (CL) {
        float *cp = ws + (int64_t)kAsWarps * G * sg;   // this CTA's partial: (m, l, acc[D]) per head
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
            if (d == 0) {
                cp[g * sg] = M;
                cp[g * sg + 1] = L;
            }
            cp[g * sg + 2 + d] = Acc;
        }
        cluster_sync();   // every partial of the row is complete and visible to the cluster
        if (app.pos >= 0 && chunk == 0) {
            // the append kernel this launch depends on has finished; every CTA of the row has read the old
            // count (they passed the barrier), so the tail entry joins the selection now
            asm volatile("griddepcontrol.wait;" ::: "memory");
            if (tid == 0 && room) {
                app.sel[(int64_t)row * sel_stride + cnt0] = (int32_t)app.pos;
                app.counts[row] = cnt0 + 1;
            }
        }
        // this CTA's slice of the G x D outputs, merged over the cluster's partials
        const uint32_t cpa = smem_addr(cp);
        const int span = (G * DT + nchunk - 1) / nchunk;
        const int x1 = (chunk + 1) * span < G * DT ? (chunk + 1) * span : G * DT;
        uint16_t *orow = out + ((int64_t)b * Hq + (int64_t)h * G) * DT;
        for (int x = chunk * span + tid; x < x1; x += kAsThreads) {
            const int g = x / DT, d = x % DT;
            float mj[kAsClusterMax];
            float M = -INFINITY;
#pragma unroll
            for (int j = 0; j < kAsClusterMax; ++j) {
                mj[j] = j < nchunk ? ld_cluster_f32(cpa + (uint32_t)(g * sg) * 4u, j) : -INFINITY;
                M = fmaxf(M, mj[j]);
            }
            float L = 0.f, Acc = 0.f;
#pragma unroll
            for (int j = 0; j < kAsClusterMax; ++j) {
                if (j < nchunk) {
                    const float w = rescale_w(mj[j], M);
                    L = fmaf(w, ld_cluster_f32(cpa + (uint32_t)(g * sg + 1) * 4u, j), L);
                    Acc = fmaf(w, ld_cluster_f32(cpa + (uint32_t)(g * sg + 2 + d) * 4u, j), Acc);
                }
            }
            if (!(L > 0.f)) set_status(dev_status, TB_ERR_INVALID_ARG);
            orow[x] = f_to_bf16(L > 0.f ? Acc / L : 0.f);
        }
        cluster_sync();   // no CTA leaves while the others still read its partial
        return;
    }
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
    // the last CTA of the row merges the row's partials
    __syncthreads();
    if (tid == 0) {
        __threadfence();
        const uint32_t prev = atomicAdd(attn_ctl + row, 1u);
        s_last = prev == (uint32_t)(nchunk - 1) ? 1u : 0u;
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    stream_merge<DT>(prow, nchunk, G, out + ((int64_t)b * Hq + (int64_t)h * G) * DT, dev_status,
                     reinterpret_cast<float *>(X));
    if (tid == 0) attn_ctl[row] = 0;   // ready for the next call
    if (app.pos >= 0) {
        // the append kernel this launch depends on has finished (the grid ends after it); every CTA of the
        // row has read the old count, so the tail entry joins the selection now
        asm volatile("griddepcontrol.wait;" ::: "memory");
        if (tid == 0 && room) {
            app.sel[(int64_t)row * sel_stride + cnt0] = (int32_t)app.pos;
            app.counts[row] = cnt0 + 1;
        }
    }
}

bool attn_stream_supported(const tb_shape &sh) {
    const int G = sh.Hq / sh.Hkv;
    return (sh.D == 64 || sh.D == 128) && G <= 16;
}

template <int DT, bool KT, int SETS, int MINB>
static cudaError_t launch_as(const tb_shape &sh, const uint16_t *q, const uint16_t *K, const uint16_t *V,
                             const int32_t *sel, const int32_t *counts, int32_t sel_stride, float scale,
                             uint16_t *out, uint32_t *attn_ctl, float *partials, int32_t *dev_status,
                             cudaStream_t st, int slot, const AttnAppend &app) {
    const int rows = sh.B * sh.Hkv;
    // CTAs per row: about MINB CTAs per SM over all rows, each at least one round of its warps' chunks, no
    // more than the workspace's partial slots per row, and few enough that the merge's scratch (2 floats per
    // head and partial) fits the chunk buffers
    const int sms = dev_info().sms > 0 ? dev_info().sms : 148;
    int64_t C = ((int64_t)MINB * sms) / rows;
    const int64_t cmax = attn_splits(sel_stride);
    const int64_t cround = (sel_stride + kAsChunk * kAsWarps - 1) / (kAsChunk * kAsWarps);
    const int64_t cfit = (int64_t)SETS * kAsWarps * kAsChunk * (4 * DT + 16) / (8 * (sh.Hq / sh.Hkv));
    if (C > cmax) C = cmax;
    if (C > cround) C = cround;
    if (C > cfit) C = cfit;
    if (C < 1) C = 1;
    // above the cluster limit by a little (or in the three-CTA form, by up to 2x): fewer CTAs per row, but the
    // cluster merge
    if (C > kAsClusterMax && (MINB == 3 || C <= kAsClusterMax + kAsClusterMax / 2)) C = kAsClusterMax;
    const int per = (int)((sel_stride + C - 1) / C);
    C = (sel_stride + per - 1) / per;
    const size_t smem = (size_t)attn_stream_smem_bytes(DT, SETS);
    // up to kAsClusterMax CTAs per row: the row is one cluster and merges in distributed shared memory
    const bool cl = C <= kAsClusterMax;
    static thread_local int attr_dev[12] = {-1, -1, -1, -1, -1, -1, -1, -1, -1, -1, -1, -1};
    auto fn = cl ? attn_stream_kernel<DT, KT, SETS, MINB, true> : attn_stream_kernel<DT, KT, SETS, MINB, false>;
    const int s2 = 2 * slot + (cl ? 1 : 0);
    if (attr_dev[s2] != dev_info().device) {
        cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        attr_dev[s2] = dev_info().device;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)C, (unsigned)rows);
    cfg.blockDim = dim3(kAsThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    int na = 0;
    if (cl) {
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = (unsigned)C;
        attr[na].val.clusterDim.y = 1;
        attr[na].val.clusterDim.z = 1;
        ++na;
    }
    if (app.pos >= 0) {   // after the append kernel, as its programmatic dependent: it streams while the append runs
        attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    return cudaLaunchKernelEx(&cfg, fn, q, K, V, sel, counts, sel_stride, sh.cap, sh.Hq, sh.Hkv, scale, out,
                              attn_ctl, partials, dev_status, app);
}

cudaError_t launch_attn_stream(const tb_shape &sh, const uint16_t *q, const uint16_t *K, const uint16_t *V,
                               const int32_t *sel, const int32_t *counts, int32_t sel_stride, float scale,
                               uint16_t *out, uint32_t *attn_ctl, float *partials, int32_t *dev_status,
                               cudaStream_t st, const AttnAppend *app) {
    const int rows = sh.B * sh.Hkv;
    if (rows <= 0 || sel_stride <= 0) return cudaSuccess;
    if (!attn_stream_supported(sh)) return cudaErrorNotSupported;
    const AttnAppend none;
    const AttnAppend &ap = app ? *app : none;
    if (ap.pos >= 0 && (!ap.K_new || !ap.V_new || !ap.sel || !ap.counts || !counts)) return cudaErrorInvalidValue;
    // keys-as-rows form: three CTAs per SM with two chunks in flight per warp when a row needs at most twice
    // the cluster limit of CTAs (it then takes one cluster; twelve warps per SM stream faster than eight),
    // else two CTAs per SM with three chunks in flight
    const bool kt = sh.Hq / sh.Hkv <= 8;
    const int sms = dev_info().sms > 0 ? dev_info().sms : 148;
    const bool three = kt && (3 * sms) / rows <= 2 * kAsClusterMax;
    if (sh.D == 64) {
        if (three)
            return launch_as<64, true, 2, 3>(sh, q, K, V, sel, counts, sel_stride, scale, out, attn_ctl, partials,
                                             dev_status, st, 4, ap);
        return kt ? launch_as<64, true, 3, 2>(sh, q, K, V, sel, counts, sel_stride, scale, out, attn_ctl, partials,
                                              dev_status, st, 0, ap)
                  : launch_as<64, false, 3, 2>(sh, q, K, V, sel, counts, sel_stride, scale, out, attn_ctl,
                                               partials, dev_status, st, 1, ap);
    }
    if (three)
        return launch_as<128, true, 2, 3>(sh, q, K, V, sel, counts, sel_stride, scale, out, attn_ctl, partials,
                                          dev_status, st, 5, ap);
    return kt ? launch_as<128, true, 3, 2>(sh, q, K, V, sel, counts, sel_stride, scale, out, attn_ctl, partials,
                                           dev_status, st, 2, ap)
              : launch_as<128, false, 3, 2>(sh, q, K, V, sel, counts, sel_stride, scale, out, attn_ctl, partials,
                                            dev_status, st, 3, ap);
}

bool attn_stream_serves(const tb_shape &sh, const uint16_t *K, const uint16_t *V) {
    return attn_stream_supported(sh) && kv_on_device(K, V);
}

}  // namespace tb
