// One decode step with a fresh prediction (interval T = 1, no neighbours) as a
// single cooperative launch with one exchange between the CTAs of a row
// ("TokenButler: Token Importance is Predictable": score every cached token
// with the importance query, keep a fixed per-token budget, attend over only
// the kept full-precision rows).
//
// Grid = rows x C CTAs, one per SM. The tokens of a row are dealt to its C
// CTAs in blocks of 32 (CTA c owns blocks c, c + C, c + 2C, ...), so every CTA
// holds a sample of the whole row and its local score distribution follows
// the row's.
//
//   1. Copies bring the CTA's blocks of Kp into shared memory; the CTA owning
//      token n also stages Wk, K_new and V_new, projects K_new and puts the
//      fresh Kp row in place before it is scored. Scores become
//      order-preserving keys.
//   2. Locally about t_c = k L_c / n of the CTA's L_c tokens are kept, with a
//      binomial spread sigma = sqrt(t_c (1 - k/n)). From its histogram the
//      CTA picks a window of 16-bit score prefixes [lo, hi] holding its local
//      ranks t_c -+ (5 sigma + 4) and publishes: the count above the window,
//      per-block counts above it, and every (key, token) inside it.
//   3. It starts gathering the K/V rows of its tokens above the window (all
//      of them are kept) into shared memory, then waits for the row's single
//      exchange.
//   4. All records of the row are read. If the windows intersect in [L, H]
//      and the row's k-th largest element lies there, the exact threshold T
//      (the composite of score key and token, lower token first) follows from
//      the entries inside [L, H]: a fine histogram finds the 16-bit bin of
//      the k-th element and a rank count inside that bin finds T. The
//      window's kept tokens join the gather. Per-block kept counts of the
//      whole row give every CTA the slots of its kept tokens in the
//      ascending idx / sel rows.
//      Otherwise (a window missed: rare unless the score layout is blocky)
//      the CTAs re-split the row into contiguous chunks through the workspace
//      and run the general distributed radix select (topk_core.cuh).
//   5. Attention over the gathered rows runs on the tensor cores: per warp,
//      chunks of 16 rows, S = Q K^T and O += P V as m16n8k16 bf16 MMAs with
//      fp32 accumulation and an online softmax (exp2 domain, fp32). The
//      warps' states are combined into one partial per CTA; after a second
//      row barrier (idx / sel are written while it fills) every CTA merges a
//      slice of the row's outputs from the C partials.
#include <string.h>

#include "async_copy.cuh"
#include "attn_mma.cuh"
#include "fused_common.cuh"
#include "kernels.cuh"

namespace tb {

constexpr int kFFThreads = 512;
constexpr int kFFWarps = kFFThreads / 32;
constexpr int kFFEntMax = kFastEntMax;
constexpr int kFFEntPerThread = 8;  // entries of one record a thread reads
constexpr int kFFStageMax = 512;    // K/V rows gathered into shared memory per round
constexpr int kFFFine = 128;        // fine bins: 4 coarse bins x 32
constexpr int kFFKpGroups = 4;      // Kp blocks arrive in commit groups, scored as each lands
constexpr uint32_t kNone = 0xFFFFFFFFu;

struct FFHdr {
    uint32_t above, lo, hi, n_ent, valid, pad0, pad1, pad2;
};
constexpr int kFFRecBytes = kFastRecBytes;
static_assert(sizeof(FFHdr) == 32, "record header is 32 bytes");
static_assert(kFFKpGroups == 4, "four commit groups (40, 30, 20, 10 % of the blocks)");

struct FFArgs {
    const uint16_t *q, *q_imp, *K_new, *V_new, *Wk;
    uint16_t *K, *V, *Kp;
    int32_t *idx, *sel, *counts;
    uint16_t *out;
    RowCtl *ctl;
    float *part;
    uint8_t *rec;        // rows x C records of kFFRecBytes
    uint8_t *blk_above;  // rows x blk_stride: per 32-token block, tokens above the owner's window
    uint32_t *keys_g;    // rows x keys_stride: keys in token order (general path)
    const WsDebug *dbg;  // test hook (zero in normal use)
    int32_t *dev_status;
    int64_t cap, n, keys_stride;
    int64_t keep_lo, keep_hi;   // tokens t < keep_lo or t >= keep_hi are always kept (maximal key)
    int32_t *centres;           // if set: the kept tokens of [keep_lo, keep_hi) minus keep_lo, ck per row,
    int64_t cpre;               // taken from slots cpre .. cpre + ck of each sel row
    int ck;
    int Hq, Hkv, D, k, agg, sel_stride;
    float scale;
    int C, NB, blk_stride, stage_cap;
};

// Shared-memory layout (byte offsets, each 16-byte aligned).
struct FFLayout {
    int X, qsm, keys, hist, fine, ckey, cidx, ccount, scan, misc, abort_, cnt, bcnt, stok, skey, kpn, knew, total;
};

__host__ __device__ inline int ff_a16(int x) { return (x + 15) & ~15; }
__host__ __device__ inline int ff_slot_bytes(int D) { return mma_slot_bytes(D); }

__host__ __device__ inline FFLayout ff_layout(int NB, int C, int stage_cap, int G, int D, int dp) {
    FFLayout L;
    int x = 0;
    int xb = NB * 32 * dp * 2;                                   // Kp blocks
    const int sb = stage_cap * ff_slot_bytes(D);                 // gathered K/V rows
    const int wb = kFFWarps * G * (2 + D) * 4;                         // per-warp attention states
    const int mb = 4 * C * G * 4 > 3 * (G * D + C) * 4 ? 4 * C * G * 4 : 3 * (G * D + C) * 4;   // merge scratch
    const int cb = comb_floats_for(kFFThreads, G, D) * 4;        // general path's combine scratch
    if (sb > xb) xb = sb;
    if (wb > xb) xb = wb;
    if (mb > xb) xb = mb;
    if (cb > xb) xb = cb;
    L.X = x; x += ff_a16(xb);
    L.qsm = x; x += 16 * (2 * D + 16);
    L.keys = x; x += ff_a16(NB * 32 * 4);
    L.hist = x; x += kRadixBins * 4;
    L.fine = x; x += kFFFine * 4;
    L.ckey = x; x += kCandCap * 4;
    L.cidx = x; x += kCandCap * 4;
    L.ccount = x; x += kMaxChunks * 4;
    L.scan = x; x += 36 * 4;
    L.misc = x; x += 16 * 4;
    L.abort_ = x; x += 16;
    L.cnt = x; x += 32 * 4;
    L.bcnt = x; x += ff_a16(NB * C * 4);
    L.stok = x; x += ff_a16(NB * 32 * 4);
    L.skey = x; x += ff_a16(NB * 32 * 4);
    L.kpn = x; x += ff_a16(dp * 2);
    L.knew = x; x += ff_a16(D * 4);   // K_new and V_new rows (bf16)
    L.total = x;
    return L;
}

// counters in the cnt region
enum {
    CN_ABOVE = 0, CN_WIN, CN_CAND, CN_AE, CN_L, CN_H, CN_VALID, CN_ASUM, CN_RANGE, CN_BM, CN_FLAG, CN_WK
};

// Wait until at most n (0..7) of this thread's cp.async groups are pending.
__device__ __forceinline__ void cp_async_wait_pending(int n) {
    switch (n) {
        case 0: asm volatile("cp.async.wait_group 0;" ::: "memory"); break;
        case 1: asm volatile("cp.async.wait_group 1;" ::: "memory"); break;
        case 2: asm volatile("cp.async.wait_group 2;" ::: "memory"); break;
        case 3: asm volatile("cp.async.wait_group 3;" ::: "memory"); break;
        case 4: asm volatile("cp.async.wait_group 4;" ::: "memory"); break;
        case 5: asm volatile("cp.async.wait_group 5;" ::: "memory"); break;
        case 6: asm volatile("cp.async.wait_group 6;" ::: "memory"); break;
        default: asm volatile("cp.async.wait_group 7;" ::: "memory"); break;
    }
}

// Order-preserving fp32 <-> uint32 for maxima by integer atomics (NaN-free
// inputs; -inf maps above 0, so a zero word is below every value).
__device__ __forceinline__ uint32_t order_key(float f) {
    const uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float order_key_inv(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// Warp-aggregated slot allocation on a shared counter: lanes with `want`
// get consecutive slots. All lanes of the warp must call it.
__device__ __forceinline__ uint32_t warp_alloc(uint32_t *ctr, bool want) {
    const uint32_t m = __ballot_sync(0xFFFFFFFFu, want);
    const int lane = threadIdx.x & 31;
    uint32_t base = 0;
    if (m) {
        const int leader = __ffs(m) - 1;
        if (lane == leader) base = atomicAdd(ctr, (uint32_t)__popc(m));
        base = __shfl_sync(0xFFFFFFFFu, base, leader);
    }
    return base + (uint32_t)__popc(m & ((1u << lane) - 1u));
}

// Four counters hist[hi - 3 .. hi] (hi + 1 a multiple of 4, 16-byte aligned)
// in one 16-byte load, highest first.
__device__ __forceinline__ void load_top4(const uint32_t *hist, int hi, uint32_t (&v)[4]) {
    const uint4 u = *reinterpret_cast<const uint4 *>(hist + hi - 3);
    v[0] = u.w;
    v[1] = u.z;
    v[2] = u.y;
    v[3] = u.x;
}

// Bins of two targets (ranks from the top, 1-based; 0 = none) in the
// kRadixBins-bin histogram, four bins per thread of the CTA's kFFThreads.
// out = {bin1, above1, bin2, above2}, kNone where a target is 0 or beyond
// the total. All threads call.
__device__ __forceinline__ void find_two_bins(const uint32_t *hist, uint32_t need1, uint32_t need2, uint32_t *scan,
                                              uint32_t *out) {
    static_assert(kRadixBins == 4 * kFFThreads, "four bins per thread");
    if (threadIdx.x == 0) out[0] = out[1] = out[2] = out[3] = kNone;
    const int hi = kRadixBins - 1 - threadIdx.x * 4;
    uint32_t hv[4];
    load_top4(hist, hi, hv);
    const uint32_t local = hv[0] + hv[1] + hv[2] + hv[3];
    uint32_t total;
    const uint32_t above = block_exclusive_scan(local, scan, total);
    for (int t = 0; t < 2; ++t) {
        const uint32_t need = t == 0 ? need1 : need2;
        if (need >= 1 && above < need && need <= above + local) {
            uint32_t a = above;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                if (need <= a + hv[j]) {
                    out[2 * t] = (uint32_t)(hi - j);
                    out[2 * t + 1] = a;
                    break;
                }
                a += hv[j];
            }
        }
    }
    __syncthreads();
}

// One warp: bins of up to two targets among kFFFine fine bins with `base`
// elements above them. out[t] = bin (kNone if not inside), out[2 + t] =
// elements above that bin, out[4 + t] = elements in it.
__device__ __forceinline__ void warp_find_fine(const uint32_t *fine, uint32_t base, uint32_t need1, uint32_t need2,
                                            uint32_t *out) {
    const int lane = threadIdx.x & 31;
    const int hi = kFFFine - 1 - lane * 4;
    uint32_t fv[4];
    load_top4(fine, hi, fv);
    const uint32_t local = fv[0] + fv[1] + fv[2] + fv[3];
    uint32_t x = local;
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, x, o);
        if (lane >= o) x += y;
    }
    const uint32_t above = base + x - local;
    if (lane == 0) out[0] = out[1] = kNone;
    __syncwarp();
    for (int t = 0; t < 2; ++t) {
        const uint32_t need = t == 0 ? need1 : need2;
        if (need >= 1 && above < need && need <= above + local) {
            uint32_t a = above;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const uint32_t c = fv[j];
                if (need <= a + c) {
                    out[t] = (uint32_t)(hi - j);
                    out[2 + t] = a;
                    out[4 + t] = c;
                    break;
                }
                a += c;
            }
        }
    }
    __syncwarp();
}

// Exclusive prefix over n <= 8 blockDim.x shared counters in place (v 16-byte
// aligned; all threads call): eight consecutive counters per thread in two
// 16-byte loads, a warp scan, the warps' totals through scratch (>= 32
// words), one barrier between.
__device__ __forceinline__ void scan8_inplace(uint32_t *v, int n, uint32_t *scratch) {
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    const int x0 = 8 * t;
    uint32_t a[8];
    if (x0 + 8 <= n) {
        const uint4 p = *reinterpret_cast<const uint4 *>(v + x0), q = *reinterpret_cast<const uint4 *>(v + x0 + 4);
        a[0] = p.x; a[1] = p.y; a[2] = p.z; a[3] = p.w;
        a[4] = q.x; a[5] = q.y; a[6] = q.z; a[7] = q.w;
    } else {
#pragma unroll
        for (int j = 0; j < 8; ++j) a[j] = x0 + j < n ? v[x0 + j] : 0u;
    }
    uint32_t loc = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) loc += a[j];
    uint32_t inc = loc;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, inc, o);
        if (lane >= o) inc += y;
    }
    if (lane == 31) scratch[warp] = inc;
    __syncthreads();
    uint32_t run = inc - loc;
    for (int w = 0; w < warp; ++w) run += scratch[w];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const uint32_t c = a[j];
        a[j] = run;
        run += c;
    }
    if (x0 + 8 <= n) {
        *reinterpret_cast<uint4 *>(v + x0) = make_uint4(a[0], a[1], a[2], a[3]);
        *reinterpret_cast<uint4 *>(v + x0 + 4) = make_uint4(a[4], a[5], a[6], a[7]);
    } else {
#pragma unroll
        for (int j = 0; j < 8; ++j)
            if (x0 + j < n) v[x0 + j] = a[j];
    }
    __syncthreads();
}

// Exclusive prefix over n shared counters in place (all threads call).
__device__ __forceinline__ void block_scan_inplace(uint32_t *v, int n, uint32_t *scan) {
    const int per = (n + blockDim.x - 1) / blockDim.x;
    const int x0 = threadIdx.x * per;
    uint32_t loc = 0;
    for (int x = x0; x < x0 + per && x < n; ++x) loc += v[x];
    uint32_t tot;
    uint32_t run = block_exclusive_scan(loc, scan, tot);
    for (int x = x0; x < x0 + per && x < n; ++x) {
        const uint32_t t = v[x];
        v[x] = run;
        run += t;
    }
    __syncthreads();
}

// The owner CTA's append. Wk of head h ([DT][DP] bf16), K_new and V_new
// rows come into shared memory by cp.async with the first Kp group, so that
// the owner issues no register loads and no global stores while the Kp
// stream is in flight. Projection: one warp per pair of outputs (16 warps x
// 2 = 32 outputs at most), lane l takes dims l, l + 32, ...; the fp32 dot
// products are summed across the warp and rounded once to bf16. The K / V /
// Kp rows of token n go to global memory once the stream has landed.
template <int DT, int DP>
__device__ __forceinline__ void append_issue(const uint16_t *K_new, const uint16_t *V_new, const uint16_t *Wk, int row,
                                             int h, uint8_t *wsm, uint8_t *kvn) {
    const uint8_t *W = reinterpret_cast<const uint8_t *>(Wk + (int64_t)h * DT * DP);
    for (int x = threadIdx.x; x < DT * DP * 2 / 16; x += blockDim.x) cp_async16(wsm + 16 * x, W + 16 * x);
    constexpr int CR = DT * 2 / 16;   // 16-byte chunks of a K / V row
    if ((int)threadIdx.x < 2 * CR) {
        const int v = (int)threadIdx.x / CR, ch = (int)threadIdx.x % CR;
        cp_async16(kvn + v * DT * 2 + 16 * ch,
                   reinterpret_cast<const uint8_t *>((v ? V_new : K_new) + (int64_t)row * DT) + 16 * ch);
    }
}

// kpn [DP] (shared bf16) <- the projected row; wsm and kvn landed and
// visible. Warp w takes dims [w DT/16, (w+1) DT/16) and lane l output l % DP
// (lanes of one warp read consecutive Wk entries: no bank conflicts); the 16
// warps' fp32 partial sums meet in red [16 x 32] and are rounded once to bf16.
// Needs 16 warps; the caller synchronises before reading kpn.
template <int DT, int DP>
__device__ __forceinline__ void append_project(const uint16_t *wsm, const uint16_t *kn, float *red, uint16_t *kpn) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    constexpr int DPW = DT / 16;      // dims per warp
    constexpr int LPJ = 32 / DP;      // lanes per output
    constexpr int DPL = DPW / LPJ;    // dims per lane
    static_assert(DPL * LPJ == DPW && DPL >= 1, "dims split evenly over the lanes of an output");
    static_assert(kFFThreads == 512, "16 warps");
    const int j = lane % DP, d0 = warp * DPW + (lane / DP) * DPL;
    float acc = 0.f;
#pragma unroll
    for (int i = 0; i < DPL; ++i) acc = fmaf(bf16_to_f(kn[d0 + i]), bf16_to_f(wsm[(d0 + i) * DP + j]), acc);
    red[threadIdx.x] = acc;
    __syncthreads();
    if ((int)threadIdx.x < DP) {
        float sum = 0.f;
#pragma unroll
        for (int w = 0; w < 16; ++w)
#pragma unroll
            for (int hh = 0; hh < LPJ; ++hh) sum += red[w * 32 + hh * DP + threadIdx.x];
        kpn[threadIdx.x] = f_to_bf16(sum);
    }
}

// K / V / Kp rows of token n from shared memory to the caches (16-byte stores).
template <int DT, int DP>
__device__ __forceinline__ void append_store(const uint8_t *kvn, const uint16_t *kpn, uint16_t *K, uint16_t *V,
                                             uint16_t *Kp, int64_t cap, int64_t n, int row) {
    constexpr int CR = DT * 2 / 16, CP = DP * 2 / 16;
    const int x = threadIdx.x;
    if (x < 2 * CR) {
        const int v = x / CR, ch = x % CR;
        reinterpret_cast<uint4 *>((v ? V : K) + ((int64_t)row * cap + n) * DT)[ch] =
            reinterpret_cast<const uint4 *>(kvn + v * DT * 2)[ch];
    } else if (x < 2 * CR + CP) {
        reinterpret_cast<uint4 *>(Kp + ((int64_t)row * cap + n) * DP)[x - 2 * CR] =
            reinterpret_cast<const uint4 *>(kpn)[x - 2 * CR];
    }
}

// The row's merge, spread over its C CTAs (after the row's second barrier):
// CTA c takes outputs x in [c NX, (c + 1) NX) of the G x D, NX = ceil(G D /
// C). A thread per (chunk u, output x) loads m, l and acc of that chunk (all
// loads in flight together), finds M_x = max_u m over shared memory and
// leaves w l and w acc, w = exp2(m - M_x); a thread per output sums them over
// the chunks and rounds once to bf16. scratch: 3 C NX floats of shared
// memory. C NX <= G D + C <= 2048 + 148 fits kMergePer pairs per thread.
constexpr int kMergePer = 5;
__device__ __forceinline__ void row_merge_slice(const float *prow, int C, int c, int G, int D, uint16_t *out_rows,
                                                float *scratch, int32_t *dev_status) {
    const int sg = 2 + D, GD = G * D;
    const int NX = (GD + C - 1) / C;
    const int x_lo = c * NX;
    const int nx = GD - x_lo < NX ? GD - x_lo : NX;   // (<= 0 for trailing CTAs)
    const int CN = C * NX;
    if (CN > kMergePer * (int)blockDim.x) {   // (not reached for G <= 16, D <= 128)
        if (threadIdx.x == 0) set_status(dev_status, TB_ERR_UNSUPPORTED);
        return;
    }
    float *mm = scratch, *pl = scratch + CN, *pa = scratch + 2 * CN;
    float m[kMergePer], l[kMergePer], av[kMergePer];
#pragma unroll
    for (int k = 0; k < kMergePer; ++k) {
        const int t = threadIdx.x + k * blockDim.x;
        const int u = t / NX, xl = t % NX;
        m[k] = -INFINITY;
        l[k] = av[k] = 0.f;
        if (t < CN && xl < nx) {
            const int x = x_lo + xl, g = x / D, d = x % D;
            const float *p = prow + ((int64_t)u * G + g) * sg;
            m[k] = __ldcg(p);
            l[k] = __ldcg(p + 1);
            av[k] = __ldcg(p + 2 + d);
        }
    }
#pragma unroll
    for (int k = 0; k < kMergePer; ++k) {
        const int t = threadIdx.x + k * blockDim.x;
        if (t < CN) mm[t] = m[k];
    }
    __syncthreads();
#pragma unroll
    for (int k = 0; k < kMergePer; ++k) {
        const int t = threadIdx.x + k * blockDim.x;
        if (t < CN) {
            const int xl = t % NX;
            float M = -INFINITY;
#pragma unroll 6
            for (int u = 0; u < C; ++u) M = fmaxf(M, mm[u * NX + xl]);
            const float w = rescale_w(m[k], M);
            pl[t] = w * l[k];
            pa[t] = w * av[k];
        }
    }
    __syncthreads();
    for (int xl = threadIdx.x; xl < nx; xl += blockDim.x) {
        float L = 0.f, A = 0.f;
#pragma unroll 6
        for (int u = 0; u < C; ++u) {
            L += pl[u * NX + xl];
            A += pa[u * NX + xl];
        }
        if (!(L > 0.f)) set_status(dev_status, TB_ERR_INVALID_ARG);
        out_rows[x_lo + xl] = f_to_bf16(L > 0.f ? A / L : 0.f);
    }
}

// Arguments of the general path, passed by value (the kernel parameters stay
// in the parameter space).
struct FFGeneral {
    RowCtl *rc;
    uint32_t *kg;            // this row's keys in token order
    int32_t *irow, *srow;    // this row's idx / sel
    int32_t *dev_status;
    const uint16_t *Kh, *Vh, *qrow;
    float *prow;
    int64_t cap, n_t;
    int C, c, nb, G, D, k;
    float scale;
};

// The general path (rare): keys to the workspace in token order, re-split
// into contiguous chunks, general distributed select with CUDA-core
// attention, this CTA's partial state to the workspace.
template <int GM>
__device__ __noinline__ bool ff_general_path(const FFGeneral g, SelectSmem S, int32_t *list, float *comb) {
    for (int e = threadIdx.x; e < g.nb * 32; e += blockDim.x) {
        const int64_t t = ((int64_t)(g.c + (e >> 5) * g.C) << 5) + (e & 31);
        if (t < g.n_t) g.kg[t] = S.keys[e];
    }
    if (threadIdx.x == 0 && g.c == 0) atomicAdd(&g.rc->general_steps, 1u);
    if (!group_barrier(&g.rc->bar, (uint32_t)(2 * g.C), S.abort_flag, g.dev_status)) return false;
    const int Ls = (int)((((g.n_t + g.C - 1) / g.C) + 31) / 32 * 32);
    const int64_t t0 = (int64_t)g.c * Ls;
    const int Lcs = (int)(g.n_t - t0 < Ls ? (g.n_t - t0 > 0 ? g.n_t - t0 : 0) : Ls);
    for (int e = threadIdx.x; e < Lcs; e += blockDim.x) S.keys[e] = __ldcg(g.kg + t0 + e);
    __syncthreads();
    AttnLane<GM> A;
    attn_init(A, g.qrow, g.G, g.D, (threadIdx.x & 31) % (g.D / 8), g.scale);
    if (!chunk_select_attend(A, g.rc, S, list, Lcs, Ls, g.c, g.C, 2, (uint32_t)g.k, t0, g.Kh, g.Vh, g.cap, g.G, g.D,
                             g.irow, g.srow, g.dev_status))
        return false;
    attn_block_combine(A, g.G, g.D, comb, g.prow + (int64_t)g.c * g.G * (2 + g.D));
    return true;
}

// FK: the forced-keep variant (sink / window tokens at the maximal key,
// centres written); the plain step compiles without that code.
template <int CPT, int DT, int GM, bool FK>
__global__ void __launch_bounds__(kFFThreads, 1) fused_fast_kernel(const FFArgs a) {
    extern __shared__ __align__(128) uint8_t smb[];
    constexpr int DP = CPT * 8;
    constexpr int NT = DT / 8;
    const int G = a.Hq / a.Hkv;
    const int C = a.C, NB = a.NB;
    const int row = blockIdx.x / C, c = blockIdx.x % C;
    const int b = row / a.Hkv, h = row % a.Hkv;
    const int64_t n_t = a.n + 1;
    // the workspace's test hook: a shorter limit for the exchange waits, one CTA of row 0 that leaves out its
    // arrival (both zero in normal use)
    const uint64_t wlim = a.dbg->wait_limit_ns ? a.dbg->wait_limit_ns : kWaitLimitNs;
    const bool skip_arrive = row == 0 && a.dbg->skip_arrive_cta == c + 1;
    const int nblk = (int)((n_t + 31) >> 5);
    const int nb = c < nblk ? (nblk - 1 - c) / C + 1 : 0;   // blocks this CTA owns
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int SB = ff_slot_bytes(DT);

    const FFLayout Y = ff_layout(NB, C, a.stage_cap, G, DT, DP);
    uint8_t *X = smb + Y.X;
    uint8_t *qsm = smb + Y.qsm;
    SelectSmem S;
    S.keys = reinterpret_cast<uint32_t *>(smb + Y.keys);
    S.hist = reinterpret_cast<uint32_t *>(smb + Y.hist);
    S.ckey = reinterpret_cast<uint32_t *>(smb + Y.ckey);
    S.cidx = reinterpret_cast<uint32_t *>(smb + Y.cidx);
    S.ccount = reinterpret_cast<uint32_t *>(smb + Y.ccount);
    S.scan = reinterpret_cast<uint32_t *>(smb + Y.scan);
    S.misc = reinterpret_cast<uint32_t *>(smb + Y.misc);
    S.abort_flag = reinterpret_cast<int *>(smb + Y.abort_);
    uint32_t *fine = reinterpret_cast<uint32_t *>(smb + Y.fine);
    uint32_t *cnt = reinterpret_cast<uint32_t *>(smb + Y.cnt);
    uint32_t *bcnt = reinterpret_cast<uint32_t *>(smb + Y.bcnt);
    int32_t *stok = reinterpret_cast<int32_t *>(smb + Y.stok);
    uint32_t *skey = reinterpret_cast<uint32_t *>(smb + Y.skey);
    uint16_t *kpn = reinterpret_cast<uint16_t *>(smb + Y.kpn);
    const int LIST = NB * 32;   // capacity of stok / skey

    auto tok_of = [&](int e) -> int64_t { return ((int64_t)(c + (e >> 5) * C) << 5) + (e & 31); };

    // ---- 0. counters and the copy barrier
    if (threadIdx.x < 32) cnt[threadIdx.x] = threadIdx.x == CN_H ? 0xFFFFu : threadIdx.x == CN_VALID ? 1u : 0u;
    if (threadIdx.x == 0) *S.abort_flag = 0;
    __syncthreads();

    // ---- 1. the step's small inputs first, so that their loads do not queue
    // behind the Kp stream: importance rows (as MMA B fragments and as fp32
    // rows), the attention query tile, and the owner's append operands
    const int blk_n = (int)(a.n >> 5);
    const bool owner = (blk_n % C) == c;
    int Lv = nb * 32;   // owned tokens (only the row's last block may be partial): local e < Lv
    if (nb > 0 && ((nblk - 1) % C) == c) Lv -= (int)((int64_t)nblk * 32 - n_t);
    const uint16_t *qi = a.q_imp + ((int64_t)b * a.Hq + (int64_t)h * G) * DP;
    const uint16_t *qrow = a.q + ((int64_t)b * a.Hq + (int64_t)h * G) * DT;
    // importance rows as MMA B fragments: lane (g, q) holds head g (+8) at the
    // dims q*DP/4 .. (q+1)*DP/4 (the token rows use the same dim order)
    constexpr int KSP = DP / 16;         // k-steps of 16 dims
    constexpr int WPL = DP / 8;          // 32-bit words of a row per lane
    constexpr int NHG = GM > 8 ? 2 : 1;  // groups of 8 heads
    uint32_t qb[NHG][WPL];
    {
        const int g = lane >> 2, q = lane & 3;
#pragma unroll
        for (int hg = 0; hg < NHG; ++hg) {
            const int head = hg * 8 + g;
            const uint32_t *src = reinterpret_cast<const uint32_t *>(qi + head * DP + q * (DP / 4));
#pragma unroll
            for (int w = 0; w < WPL; ++w) qb[hg][w] = head < G ? src[w] : 0u;
        }
    }
    const int qg = threadIdx.x / (DT / 8), qc = threadIdx.x % (DT / 8);   // Q tile chunk of this thread
    uint4 qv = make_uint4(0, 0, 0, 0);
    if (qg < G) qv = *reinterpret_cast<const uint4 *>(qrow + qg * DT + qc * 8);
    // the owner's Wk rows (and the projection's partial sums) are staged
    // where the candidate lists go later
    static_assert(DT * DP * 2 <= kCandCap * 4 && kFFThreads * 4 <= kCandCap * 4, "append staging fits");
    uint8_t *wsm = smb + Y.ckey;
    uint8_t *kvn = smb + Y.knew;
    if (owner) append_issue<DT, DP>(a.K_new, a.V_new, a.Wk, row, h, wsm, kvn);   // (in commit group 0)

    // ---- 1a. Kp blocks -> shared memory: 16-byte cp.async by every thread,
    // consecutive threads on consecutive chunks, in commit groups of 40, 30,
    // 20 and 10 % of the CTA's blocks: scoring starts on the first groups,
    // and little of it is left once the last one lands
    const int gb1 = (4 * nb) / 10, gb2 = (7 * nb) / 10, gb3 = (9 * nb) / 10;   // first blocks of groups 1..3
    auto group_of = [&](int j) -> int { return (j >= gb1) + (j >= gb2) + (j >= gb3); };
    {
        constexpr int CPB = 32 * DP * 2 / 16;   // 16-byte chunks per block
        const uint16_t *Kpr = a.Kp + (int64_t)row * a.cap * DP;
        for (int g = 0; g < kFFKpGroups; ++g) {
            const int j0 = g == 0 ? 0 : g == 1 ? gb1 : g == 2 ? gb2 : gb3;
            const int j1 = g == 0 ? gb1 : g == 1 ? gb2 : g == 2 ? gb3 : nb;
            for (int x = threadIdx.x; x < (j1 - j0) * CPB; x += blockDim.x) {
                const int j = j0 + x / CPB, ch = x % CPB;
                const int64_t blk = (int64_t)c + (int64_t)j * C;
                if (blk * 32 + (ch * 16) / (DP * 2) < n_t)
                    cp_async16(X + (size_t)j * 32 * DP * 2 + ch * 16,
                               reinterpret_cast<const uint8_t *>(Kpr + blk * 32 * DP) + ch * 16);
            }
            cp_async_commit();
        }
    }
    // ---- 1b. the small inputs to shared memory; histograms cleared
    if (qg < 16) *reinterpret_cast<uint4 *>(qsm + qg * (2 * DT + 16) + qc * 16) = qv;
    for (int x = threadIdx.x; x < kRadixBins; x += blockDim.x) S.hist[x] = 0;
    for (int x = threadIdx.x; x < kFFFine; x += blockDim.x) fine[x] = 0;
    const uint16_t *Kh = a.K + (int64_t)row * a.cap * DT;
    const uint16_t *Vh = a.V + (int64_t)row * a.cap * DT;
    __syncthreads();

    // ---- 2. scores on the tensor cores: tiles of 16 tokens (A) x 8 heads (B),
    // m16n8k16; per token the G dot products are averaged (or maxed), then the
    // order-preserving key and its coarse bin
    bool nan_seen = false;
    const bool forcing = FK && (a.keep_lo > 0 || a.keep_hi < n_t);   // (uniform)
    {
        const int g = lane >> 2, q = lane & 3;
        const float invG = 1.0f / (float)G;
        const int ntile = (nb * 32) >> 4;
        int grp = -1;
        // the owner's appended token: local row and the group of its block
        const int en = (blk_n / C) * 32 + (int)(a.n & 31);
        const int g_n = owner ? group_of(blk_n / C) : -1;
        for (int tt = 0; tt < ntile; tt += kFFWarps) {
            // every thread waits for its own copies of the group, then the CTA
            // barrier makes all threads' copies of it visible
            const int gt = group_of(min((tt + kFFWarps - 1) >> 1, nb - 1));   // last group any warp needs now
            while (grp < gt) {
                ++grp;
                cp_async_wait_pending(kFFKpGroups - 1 - grp);
                __syncthreads();
                if (owner && grp == 0) {   // Wk, K_new and V_new arrived with group 0
                    append_project<DT, DP>(reinterpret_cast<const uint16_t *>(wsm),
                                           reinterpret_cast<const uint16_t *>(kvn),
                                           reinterpret_cast<float *>(S.cidx), kpn);
                    __syncthreads();
                }
                if (grp == g_n) {   // the fresh Kp row replaces the copied one before it is scored
                    if ((int)threadIdx.x < DP / 8)
                        *reinterpret_cast<uint4 *>(X + (size_t)en * DP * 2 + 16 * threadIdx.x) =
                            reinterpret_cast<const uint4 *>(kpn)[threadIdx.x];
                    __syncthreads();
                }
            }
            if (tt + warp >= ntile) continue;
            const int tw = tt + warp;
            const uint8_t *tb = X + (size_t)tw * 16 * DP * 2 + q * (DP / 2);
            uint32_t w0[WPL], w1[WPL];
            if (WPL == 4) {
                const uint4 u0 = *reinterpret_cast<const uint4 *>(tb + g * DP * 2);
                const uint4 u1 = *reinterpret_cast<const uint4 *>(tb + (g + 8) * DP * 2);
                w0[0] = u0.x; w0[1] = u0.y; w0[WPL > 2 ? 2 : 0] = u0.z; w0[WPL > 3 ? 3 : 0] = u0.w;
                w1[0] = u1.x; w1[1] = u1.y; w1[WPL > 2 ? 2 : 0] = u1.z; w1[WPL > 3 ? 3 : 0] = u1.w;
            } else {
                const uint2 u0 = *reinterpret_cast<const uint2 *>(tb + g * DP * 2);
                const uint2 u1 = *reinterpret_cast<const uint2 *>(tb + (g + 8) * DP * 2);
                w0[0] = u0.x; w0[1] = u0.y;
                w1[0] = u1.x; w1[1] = u1.y;
            }
            float ca[NHG][4];
#pragma unroll
            for (int hg = 0; hg < NHG; ++hg) {
                ca[hg][0] = ca[hg][1] = ca[hg][2] = ca[hg][3] = 0.f;
#pragma unroll
                for (int ks = 0; ks < KSP; ++ks)
                    mma_bf16_16816(ca[hg], w0[2 * ks], w1[2 * ks], w0[2 * ks + 1], w1[2 * ks + 1], qb[hg][2 * ks],
                                   qb[hg][2 * ks + 1]);
            }
            float v0, v1;
            if (a.agg == TB_AGG_MEAN) {
                v0 = 0.f;
                v1 = 0.f;
#pragma unroll
                for (int hg = 0; hg < NHG; ++hg) {
                    v0 += ca[hg][0] + ca[hg][1];
                    v1 += ca[hg][2] + ca[hg][3];
                }
                v0 += __shfl_xor_sync(0xFFFFFFFFu, v0, 1);
                v1 += __shfl_xor_sync(0xFFFFFFFFu, v1, 1);
                v0 += __shfl_xor_sync(0xFFFFFFFFu, v0, 2);
                v1 += __shfl_xor_sync(0xFFFFFFFFu, v1, 2);
                v0 *= invG;
                v1 *= invG;
            } else {
                v0 = -INFINITY;
                v1 = -INFINITY;
#pragma unroll
                for (int hg = 0; hg < NHG; ++hg) {
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        if (hg * 8 + 2 * q + u < G) {
                            v0 = fmaxf(v0, ca[hg][u]);
                            v1 = fmaxf(v1, ca[hg][2 + u]);
                        }
                    }
                }
                v0 = fmaxf(v0, __shfl_xor_sync(0xFFFFFFFFu, v0, 1));
                v1 = fmaxf(v1, __shfl_xor_sync(0xFFFFFFFFu, v1, 1));
                v0 = fmaxf(v0, __shfl_xor_sync(0xFFFFFFFFu, v0, 2));
                v1 = fmaxf(v1, __shfl_xor_sync(0xFFFFFFFFu, v1, 2));
            }
            if (q < 2) {
                const int e = tw * 16 + g + 8 * q;
                uint32_t key = 0;
                if (e < Lv) {
                    // forced tokens (their Kp rows need not exist) rank above every score
                    bool forced = false;
                    if (forcing) {
                        const int64_t t = tok_of(e);
                        forced = t < a.keep_lo || t >= a.keep_hi;
                    }
                    key = forced ? 0xFFFFFFFFu : score_key(q ? v1 : v0, nan_seen);
                    atomicAdd(&S.hist[key >> 21], 1u);
                }
                S.keys[e] = key;
            }
        }
    }
    cp_async_wait_all();   // (the groups are complete; nothing may reuse X while a copy could land)
    if (owner) append_store<DT, DP>(kvn, kpn, a.K, a.V, a.Kp, a.cap, a.n, row);
    if (nan_seen) set_status(a.dev_status, TB_ERR_NONFINITE);
    __syncthreads();

    // ---- 3. local window around the row's threshold
    uint32_t need_hi = 0, need_lo = 0;   // ranks from the top; 0 = no bound on that side
    {
        const int t_c = (int)(((int64_t)a.k * Lv + n_t / 2) / n_t);
        const float p = (float)a.k / (float)n_t;
        const int R = (int)ceilf(5.0f * sqrtf((float)t_c * (1.0f - p))) + 4;
        if (t_c - R >= 0 && Lv > 0) need_hi = (uint32_t)(t_c - R + 1);
        if (t_c + R <= Lv) need_lo = (uint32_t)(t_c + R);
    }
    uint32_t *bins = S.misc;   // {Bhi, Ahi, Blo, Alo}
    find_two_bins(S.hist, need_hi, need_lo, S.scan, bins);
    const uint32_t Bhi = bins[0], Blo = bins[2];
    uint32_t F0 = 0;
    if (Bhi != kNone) F0 = Bhi >= 3 ? Bhi - 3 : 0;
    else if (Blo != kNone) F0 = Blo >= 3 ? Blo - 3 : 0;
    {
        uint32_t n_up = 0;   // keys above the fine range
        for (int e = threadIdx.x; e < Lv; e += blockDim.x) {
            const uint32_t key = S.keys[e];
            const uint32_t cb = key >> 21;
            if (cb >= F0 && cb <= F0 + 3) atomicAdd(&fine[(key >> 16) - (F0 << 5)], 1u);
            n_up += cb > F0 + 3 ? 1u : 0u;
        }
        n_up = __reduce_add_sync(0xFFFFFFFFu, n_up);
        if (lane == 0 && n_up) atomicAdd(&cnt[CN_RANGE], n_up);
    }
    __syncthreads();
    if (warp == 0) warp_find_fine(fine, cnt[CN_RANGE], need_hi, need_lo, S.misc + 4);
    __syncthreads();
    uint32_t hi16 = 0xFFFFu, lo16 = 0u;
    if (Bhi != kNone) hi16 = S.misc[4] != kNone ? (F0 << 5) + S.misc[4] : ((Bhi << 5) | 31u);
    if (Blo != kNone) lo16 = S.misc[5] != kNone ? (F0 << 5) + S.misc[5] : (Blo << 5);
    if (need_hi == 0) hi16 = 0xFFFFu;
    if (need_lo == 0) lo16 = 0u;

    // ---- 4. publish the record; tokens above the window at the front of
    // stok, tokens inside it at the back
    RowCtl *rc = a.ctl + row;
    uint8_t *myrec = a.rec + ((int64_t)row * C + c) * kFFRecBytes;
    uint2 *myent = reinterpret_cast<uint2 *>(myrec + sizeof(FFHdr));
    uint8_t *blkab = a.blk_above + (int64_t)row * a.blk_stride;
    // a warp takes whole blocks; its slots are reserved with one atomic per
    // list (first pass: counts), then filled in order (second pass)
    {
        const uint32_t lt = (1u << lane) - 1u;
        uint32_t na = 0, nw = 0;
        for (int e = threadIdx.x; e < nb * 32; e += blockDim.x) {
            const uint32_t pf = S.keys[e] >> 16;
            const bool valid = e < Lv;
            const bool above = valid && pf > hi16;
            const uint32_t ab = __ballot_sync(0xFFFFFFFFu, above);
            const uint32_t wb = __ballot_sync(0xFFFFFFFFu, valid && !above && pf >= lo16);
            if (lane == 0) blkab[c + (e >> 5) * C] = (uint8_t)__popc(ab);
            na += (uint32_t)__popc(ab);
            nw += (uint32_t)__popc(wb);
        }
        uint32_t as = 0, ws = 0;
        if (lane == 0) {
            if (na) as = atomicAdd(&cnt[CN_ABOVE], na);
            if (nw) ws = atomicAdd(&cnt[CN_WIN], nw);
        }
        as = __shfl_sync(0xFFFFFFFFu, as, 0);
        ws = __shfl_sync(0xFFFFFFFFu, ws, 0);
        for (int e = threadIdx.x; e < nb * 32 && (na | nw); e += blockDim.x) {
            const int64_t t = tok_of(e);
            const uint32_t key = S.keys[e];
            const uint32_t pf = key >> 16;
            const bool valid = e < Lv;
            const bool above = valid && pf > hi16;
            const bool inwin = valid && !above && pf >= lo16;
            const uint32_t ab = __ballot_sync(0xFFFFFFFFu, above);
            const uint32_t wb = __ballot_sync(0xFFFFFFFFu, inwin);
            if (above) {
                const uint32_t sl = as + (uint32_t)__popc(ab & lt);
                stok[sl] = (int32_t)t;
                skey[sl] = key;
            }
            if (inwin) {
                const uint32_t sl = ws + (uint32_t)__popc(wb & lt);
                stok[LIST - 1 - sl] = (int32_t)t;
                skey[LIST - 1 - sl] = key;
                if (sl < (uint32_t)kFFEntMax) myent[sl] = make_uint2(key, (uint32_t)t);
            }
            as += (uint32_t)__popc(ab);
            ws += (uint32_t)__popc(wb);
        }
    }
    __syncthreads();
    const int n_above = (int)cnt[CN_ABOVE], n_win = (int)cnt[CN_WIN];
    if (threadIdx.x == 0) {
        FFHdr hd;
        hd.above = (uint32_t)n_above;
        hd.lo = lo16;
        hd.hi = hi16;
        hd.n_ent = (uint32_t)n_win;
        hd.valid = n_win <= kFFEntMax ? 1u : 0u;
        hd.pad0 = hd.pad1 = hd.pad2 = 0;
        *reinterpret_cast<FFHdr *>(myrec) = hd;
    }
    if (!skip_arrive) group_arrive(&rc->bar);
    else __syncthreads();

    // ---- 4b. the attention list: the tokens above the window (every one of
    // them is kept), then the window's kept tokens (wk, known after the
    // exchange); its K/V rows are gathered into X, the first ones now.
    int32_t *wk = reinterpret_cast<int32_t *>(S.hist);
    auto att_tok = [&](int i) -> int64_t { return i < n_above ? stok[i] : wk[i - n_above]; };
    constexpr int CPR = DT / 8;   // 16-byte chunks per row
    // a group of 2*CPR lanes copies one row's K and V (one 16-byte chunk each)
    constexpr int RPW = 32 / (2 * CPR);   // rows per warp per pass
    const int rl = lane % (2 * CPR);
    const bool rl_v = rl >= CPR;
    const int rl_c = rl_v ? rl - CPR : rl;
    // list entries r0 + s -> slots s, for s in [s0, s1)
    auto gather_rows = [&](int r0, int s0, int s1) {
        for (int s = s0 + warp * RPW + lane / (2 * CPR); s < s1; s += kFFWarps * RPW) {
            const int64_t t = att_tok(r0 + s);
            cp_async16(X + (size_t)s * SB + (rl_v ? 2 * DT : 0) + rl_c * 16, (rl_v ? Vh : Kh) + t * DT + rl_c * 8);
        }
        cp_async_commit();
    };
    const int n_r1 = n_above < a.stage_cap ? n_above : a.stage_cap;
    gather_rows(0, 0, n_r1);

    // ---- 5. the row's exchange; read every record of the row
    if (!group_wait(&rc->bar, (uint32_t)C, S.abort_flag, a.dev_status, wlim)) {
        cp_async_wait_all();
        return;
    }
    const int P = blockDim.x / C;   // threads per record
    const int rr = threadIdx.x / P, rsub = threadIdx.x % P;
    uint4 hd4 = make_uint4(0, 0, 0, 0);
    uint32_t hvalid = 1;
    uint2 ent[kFFEntPerThread];
    const uint8_t *rrec = a.rec + ((int64_t)row * C + (rr < C ? rr : 0)) * kFFRecBytes;
    if (rr < C) {
        hd4 = __ldcg(reinterpret_cast<const uint4 *>(rrec));
        hvalid = __ldcg(reinterpret_cast<const uint32_t *>(rrec) + 4);
    }
    // entries 2 q and 2 q + 1 per 16-byte load, q = rsub + P j: thread entry
    // i is record entry ent_index(i)
    auto ent_index = [&](int i) -> int { return 2 * (rsub + P * (i >> 1)) + (i & 1); };
#pragma unroll
    for (int j = 0; j < kFFEntPerThread / 2; ++j) {
        const int q = rsub + P * j;
        uint4 v = make_uint4(0, 0, 0, 0);
        if (rr < C && 2 * q + 1 < kFFEntMax) v = __ldcg(reinterpret_cast<const uint4 *>(rrec + sizeof(FFHdr)) + q);
        ent[2 * j] = make_uint2(v.x, v.y);
        ent[2 * j + 1] = make_uint2(v.z, v.w);
    }
    // per-block counts above the owners' windows, four blocks per load
    for (int x4 = threadIdx.x; 4 * x4 < nblk; x4 += blockDim.x) {
        const uint32_t v = __ldcg(reinterpret_cast<const uint32_t *>(blkab) + x4);
#pragma unroll
        for (int j = 0; j < 4; ++j)
            if (4 * x4 + j < nblk) bcnt[4 * x4 + j] = (v >> (8 * j)) & 0xFFu;
    }
    if (rr < C && rsub == 0) {
        atomicMax(&cnt[CN_L], hd4.y);
        atomicMin(&cnt[CN_H], hd4.z);
        atomicAdd(&cnt[CN_ASUM], hd4.x);
        if (!hvalid || hd4.w > (uint32_t)(P * kFFEntPerThread)) cnt[CN_VALID] = 0;
    }
    __syncthreads();
    const uint32_t Lw = cnt[CN_L], Hw = cnt[CN_H];
    bool fast = cnt[CN_VALID] != 0 && Lw <= Hw;
    uint32_t is_cand = 0;
    if (fast) {
        // per thread: entries above the intersection (counted per block) and
        // candidates inside it; one atomic per warp and counter
        uint32_t n_hi = 0, n_c = 0;
#pragma unroll
        for (int i = 0; i < kFFEntPerThread; ++i) {
            const bool have = rr < C && (uint32_t)ent_index(i) < hd4.w;
            const uint32_t pf = ent[i].x >> 16;
            const bool hi_side = have && pf > Hw;
            const bool cand = have && !hi_side && pf >= Lw;
            if (hi_side) atomicAdd(&bcnt[ent[i].y >> 5], 1u);
            n_hi += hi_side ? 1u : 0u;
            n_c += cand ? 1u : 0u;
            if (cand) is_cand |= 1u << i;
        }
        uint32_t x = n_c;   // inclusive scan of the candidate counts over the warp
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, x, o);
            if (lane >= o) x += y;
        }
        const uint32_t hw_tot = __reduce_add_sync(0xFFFFFFFFu, n_hi);
        uint32_t base = 0;
        if (lane == 31) {
            if (hw_tot) atomicAdd(&cnt[CN_AE], hw_tot);
            if (x) base = atomicAdd(&cnt[CN_CAND], x);
        }
        uint32_t cs = __shfl_sync(0xFFFFFFFFu, base, 31) + x - n_c;
#pragma unroll
        for (int i = 0; i < kFFEntPerThread; ++i) {
            if ((is_cand >> i) & 1u) {
                if (cs < (uint32_t)kCandCap) {
                    S.ckey[cs] = ent[i].x;
                    S.cidx[cs] = ent[i].y;
                }
                ++cs;
            }
        }
    }
    __syncthreads();
    const uint32_t m = cnt[CN_CAND];
    const int64_t need = (int64_t)a.k - (int64_t)cnt[CN_ASUM] - (int64_t)cnt[CN_AE];
    fast = fast && m <= (uint32_t)kCandCap && need >= 1 && need <= (int64_t)m;

    // ---- 5b. the exact threshold T among the candidates
    uint64_t T = 0;
    uint64_t *Tsm = reinterpret_cast<uint64_t *>(S.misc + 8);
    if (fast) {
        bool done = false;
        if (Hw - Lw < (uint32_t)kFFFine) {
            for (int x = threadIdx.x; x < kFFFine; x += blockDim.x) fine[x] = 0;
            __syncthreads();
            for (uint32_t e = threadIdx.x; e < m; e += blockDim.x) atomicAdd(&fine[(S.ckey[e] >> 16) - Lw], 1u);
            __syncthreads();
            if (warp == 0) warp_find_fine(fine, 0, (uint32_t)need, 0, S.misc);
            __syncthreads();
            const uint32_t bstar = S.misc[0], babove = S.misc[2], bc = S.misc[4];
            if (bstar != kNone && bc <= (uint32_t)kFFThreads) {
                // rank count inside the bin (composites are distinct)
                uint64_t *comp = reinterpret_cast<uint64_t *>(S.hist);
                for (uint32_t e0 = 0; e0 < m; e0 += blockDim.x) {
                    const uint32_t e = e0 + threadIdx.x;
                    const bool in = e < m && ((S.ckey[e] >> 16) - Lw) == bstar;
                    const uint32_t sl = warp_alloc(&cnt[CN_BM], in);
                    if (in) comp[sl] = composite(S.ckey[e], S.cidx[e]);
                }
                __syncthreads();
                const uint32_t need2 = (uint32_t)need - babove;
                if (threadIdx.x < bc) {
                    const uint64_t v = comp[threadIdx.x];
                    uint32_t rank = 0;
                    for (uint32_t j = 0; j < bc; ++j) rank += comp[j] > v ? 1u : 0u;
                    if (rank == need2 - 1) *Tsm = v;
                }
                __syncthreads();
                T = *Tsm;
                done = true;
            }
        }
        if (!done) T = local_select(S.ckey, S.cidx, m, (uint32_t)need, 32, S);
    }

    float *prow = a.part + (int64_t)row * C * G * (2 + DT);
    if (fast) {
        // ---- 5c. per-block kept counts of the row; the window's kept tokens
        // -> wk
#pragma unroll
        for (int i = 0; i < kFFEntPerThread; ++i)
            if (((is_cand >> i) & 1u) && composite(ent[i].x, ent[i].y) >= T) atomicAdd(&bcnt[ent[i].y >> 5], 1u);
        __syncthreads();   // (the selection's scratch in S.hist is dead)
        for (int i0 = 0; i0 < n_win; i0 += blockDim.x) {
            const int i = i0 + (int)threadIdx.x;
            const bool kp = i < n_win && composite(skey[LIST - 1 - i], (uint32_t)stok[LIST - 1 - i]) >= T;
            const uint32_t sl = warp_alloc(&cnt[CN_WK], kp);
            if (kp) wk[sl] = stok[LIST - 1 - i];
        }
        __syncthreads();
        const int n_att = n_above + (int)cnt[CN_WK];
        // the first round's window rows are requested now; while they arrive,
        // the per-block kept counts become the blocks' first slots in idx / sel
        const int nr0 = n_att < a.stage_cap ? n_att : a.stage_cap;
        gather_rows(0, n_r1, nr0);
        if (nblk <= 8 * kFFThreads) scan8_inplace(bcnt, nblk, S.scan);
        else block_scan_inplace(bcnt, nblk, S.scan);
        // ---- 6. attention over the gathered rows, round by round
        MmaAttn<NT> A;
        A.m0 = A.m1 = -INFINITY;
        A.l0 = A.l1 = 0.f;
#pragma unroll
        for (int t = 0; t < NT; ++t) A.o[t][0] = A.o[t][1] = A.o[t][2] = A.o[t][3] = 0.f;
        const float qscale = a.scale * kLog2e;
        for (int r0 = 0; r0 < n_att; r0 += a.stage_cap) {
            const int nr = n_att - r0 < a.stage_cap ? n_att - r0 : a.stage_cap;
            if (r0 > 0) {
                __syncthreads();   // the previous round's rows are consumed
                gather_rows(r0, 0, nr);
            }
            // the padding rows up to a multiple of 16 hold zeros in V
            const int npad = (nr + 15) & ~15;
            for (int s = nr + warp * RPW + lane / (2 * CPR); s < npad; s += kFFWarps * RPW)
                if (rl_v) st_shared_zero16_if(X + (size_t)s * SB + 2 * DT + rl_c * 16, true);
            cp_async_wait_all();
            __syncthreads();
            mma_attend<DT, kFFWarps, false>(A, X, SB, nr, nullptr, 0, qsm, qscale);
        }
        // ---- 6b. combine the warps' states into this CTA's partial
        A.l0 += __shfl_xor_sync(0xFFFFFFFFu, A.l0, 1);
        A.l0 += __shfl_xor_sync(0xFFFFFFFFu, A.l0, 2);
        A.l1 += __shfl_xor_sync(0xFFFFFFFFu, A.l1, 1);
        A.l1 += __shfl_xor_sync(0xFFFFFFFFu, A.l1, 2);
        // the CTA's max per head: one shared atomicMax per warp and head on
        // order-preserving keys (cnt[16 + g], zero = below every key)
        uint32_t *mkey = cnt + 16;
        {
            const int g0 = lane >> 2;
            if ((lane & 3) == 0) {
                if (g0 < G) atomicMax(&mkey[g0], order_key(A.m0));
                if (g0 + 8 < G) atomicMax(&mkey[g0 + 8], order_key(A.m1));
            }
        }
        __syncthreads();   // (X is free: the warps' scaled states go there)
        float *ws = reinterpret_cast<float *>(X);
        const int sg = 2 + DT;
        {
            const int g0 = lane >> 2, d0 = 2 * (lane & 3);
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                const int g = g0 + 8 * half;
                if (g < G) {
                    const float wt = rescale_w(half ? A.m1 : A.m0, order_key_inv(mkey[g]));
                    float *w = ws + ((int64_t)warp * G + g) * sg;
                    if ((lane & 3) == 0) w[1] = wt * (half ? A.l1 : A.l0);
#pragma unroll
                    for (int t = 0; t < NT; ++t)
                        *reinterpret_cast<float2 *>(w + 2 + 8 * t + d0) =
                            make_float2(wt * A.o[t][2 * half], wt * A.o[t][2 * half + 1]);
                }
            }
        }
        __syncthreads();
        for (int x = threadIdx.x; x < G * DT; x += blockDim.x) {
            const int g = x / DT, d = x % DT;
            float L = 0.f, Acc = 0.f;
#pragma unroll
            for (int w = 0; w < kFFWarps; ++w) {
                const float *sw = ws + (w * G + g) * sg;
                L += sw[1];
                Acc += sw[2 + d];
            }
            float *o = prow + ((int64_t)c * G + g) * sg;
            if (d == 0) {
                o[0] = order_key_inv(mkey[g]);
                o[1] = L;
            }
            o[2 + d] = Acc;
        }
        // ---- 6c. the row's second barrier; every CTA merges a slice of the
        // outputs. The last CTA to count itself done resets the row's control
        // words (all have passed the barrier by then).
        group_arrive(&rc->bar);
        // ---- 6d. idx / sel while the other CTAs finish: slots from the row's
        // per-block kept counts (scanned above)
        {
            int32_t *irow = a.idx ? a.idx + (int64_t)row * a.k : nullptr;
            int32_t *srow = a.sel + (int64_t)row * a.sel_stride;
            for (int e = threadIdx.x; e < nb * 32; e += blockDim.x) {
                const int64_t t = tok_of(e);
                const bool kp = e < Lv && composite(S.keys[e], (uint32_t)t) >= T;
                const uint32_t km = __ballot_sync(0xFFFFFFFFu, kp);
                const uint32_t slot = bcnt[t >> 5] + (uint32_t)__popc(km & ((1u << lane) - 1u));
                if (kp && slot < (uint32_t)a.k) {
                    if (!FK || irow) irow[slot] = (int32_t)t;
                    srow[slot] = (int32_t)t;
                    if (FK && a.centres && t >= a.keep_lo && t < a.keep_hi)
                        a.centres[(int64_t)row * a.ck + ((int64_t)slot - a.cpre)] = (int32_t)(t - a.keep_lo);
                }
                if (kp && slot >= (uint32_t)a.k) set_status(a.dev_status, TB_ERR_INVALID_ARG);
            }
            if (c == 0 && threadIdx.x == 0) a.counts[row] = a.k;
        }
        if (!group_wait(&rc->bar, 2u * (uint32_t)C, S.abort_flag, a.dev_status, wlim)) return;
        uint32_t done_prev = 0;
        if (threadIdx.x == 0) done_prev = atomicAdd(&rc->done, 1u);
        row_merge_slice(prow, C, c, G, DT, a.out + ((int64_t)b * a.Hq + (int64_t)h * G) * DT,
                        reinterpret_cast<float *>(X), a.dev_status);
        if (threadIdx.x == 0 && done_prev == (uint32_t)(C - 1)) {
            rc->bar = 0;
            rc->ncand = 0;
            rc->done = 0;
        }
    } else {
        cp_async_wait_all();
        FFGeneral gp;
        gp.rc = rc;
        gp.kg = a.keys_g + (int64_t)row * a.keys_stride;
        gp.irow = a.idx ? a.idx + (int64_t)row * a.k : nullptr;
        gp.srow = a.sel + (int64_t)row * a.sel_stride;
        gp.dev_status = a.dev_status;
        gp.Kh = Kh;
        gp.Vh = Vh;
        gp.qrow = qrow;
        gp.prow = prow;
        gp.cap = a.cap;
        gp.n_t = n_t;
        gp.C = C;
        gp.c = c;
        gp.nb = nb;
        gp.G = G;
        gp.D = DT;
        gp.k = a.k;
        gp.scale = a.scale;
        if (!ff_general_path<GM>(gp, S, stok, reinterpret_cast<float *>(X))) return;
        if (c == 0 && threadIdx.x == 0) a.counts[row] = a.k;
        // ---- 7. the row's last CTA merges (and copies the centres, when asked, from the finished sel row)
        if (row_merge_last(rc, prow, C, G, DT, a.out + ((int64_t)b * a.Hq + (int64_t)h * G) * DT, &cnt[CN_FLAG],
                           true, a.dev_status, reinterpret_cast<float *>(X)) &&
            FK && a.centres) {
            const int32_t *srow = a.sel + (int64_t)row * a.sel_stride;
            for (int j = threadIdx.x; j < a.ck; j += blockDim.x)
                a.centres[(int64_t)row * a.ck + j] = __ldcg(srow + a.cpre + j) - (int32_t)a.keep_lo;
        }
    }
}

// ------------------------------------------------------------------ host side

struct FFPlan {
    int C = 0, NB = 0, stage_cap = 0, cpt = 0, gm = 0;
    size_t smem = 0;
};

static int ff_gm(int G) { return G <= 1 ? 1 : G <= 4 ? 4 : 16; }

template <int CPT, int DT, int GM>
static int ff_occupancy(size_t smem) {
    if (cudaFuncSetAttribute(fused_fast_kernel<CPT, DT, GM, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem) != cudaSuccess ||
        cudaFuncSetAttribute(fused_fast_kernel<CPT, DT, GM, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem) != cudaSuccess)
        return 0;
    int per = 0, per_fk = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, fused_fast_kernel<CPT, DT, GM, false>, kFFThreads, smem) !=
            cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_fk, fused_fast_kernel<CPT, DT, GM, true>, kFFThreads,
                                                      smem) != cudaSuccess)
        return 0;
    return per < per_fk ? per : per_fk;
}

#define TB_FF_CASES(X) X(2, 64, 1) X(2, 64, 4) X(2, 64, 16) X(2, 128, 1) X(2, 128, 4) X(2, 128, 16) \
    X(4, 64, 1) X(4, 64, 4) X(4, 64, 16) X(4, 128, 1) X(4, 128, 4) X(4, 128, 16)

static bool ff_plan_uncached(const tb_shape &sh, int64_t n_t, FFPlan &P) {
    const DevInfo &di = dev_info();
    if (di.sms <= 0) return false;
    const int cpt = sh.dp / 8;
    if (sh.dp % 8 != 0 || (cpt != 2 && cpt != 4)) return false;
    if (sh.D != 64 && sh.D != 128) return false;
    const int G = sh.Hq / sh.Hkv;
    if (G > 16) return false;
    const int rows = sh.B * sh.Hkv;
    const int64_t nblk = (n_t + 31) / 32;
    int64_t C = di.sms / rows;
    if (C > nblk) C = nblk;
    if (C > kMaxChunks) C = kMaxChunks;
    if (C < 1) return false;
    const int64_t NB = (nblk + C - 1) / C;
    if (NB * 32 > 16384) return false;                 // keys and lists must fit shared memory
    if (2 * C * G + G > 2 * kCandCap) return false;     // merge scratch
    int lo = 16, hi = kFFStageMax;                       // largest round of gathered rows that fits
    if (ff_layout((int)NB, (int)C, lo, G, sh.D, sh.dp).total > di.max_smem_optin) return false;
    while (lo < hi) {
        const int mid = (lo + hi + 1) / 2;
        if (ff_layout((int)NB, (int)C, mid, G, sh.D, sh.dp).total <= di.max_smem_optin) lo = mid;
        else hi = mid - 1;
    }
    P.C = (int)C;
    P.NB = (int)NB;
    P.stage_cap = lo & ~15;
    P.cpt = cpt;
    P.gm = ff_gm(G);
    P.smem = (size_t)ff_layout(P.NB, P.C, P.stage_cap, G, sh.D, sh.dp).total;
    int occ = 0;
#define TB_FF_OCC(CP, DTT, GMC) \
    if (P.cpt == CP && sh.D == DTT && P.gm == GMC) occ = ff_occupancy<CP, DTT, GMC>(P.smem);
    TB_FF_CASES(TB_FF_OCC)
#undef TB_FF_OCC
    return occ >= 1 && (int64_t)rows * C <= (int64_t)occ * di.sms;
}

static bool ff_plan(const tb_shape &sh, int64_t n_t, FFPlan &P) {
    struct Key {
        int dev, B, Hq, Hkv, D, dp;
        int64_t n;
    };
    static thread_local Key last = {-2, 0, 0, 0, 0, 0, 0};
    static thread_local bool last_ok = false;
    static thread_local FFPlan last_plan;
    Key k = {dev_info().device, sh.B, sh.Hq, sh.Hkv, sh.D, sh.dp, n_t};
    if (memcmp(&k, &last, sizeof k) != 0) {
        last_plan = FFPlan();
        last_ok = ff_plan_uncached(sh, n_t, last_plan);
        last = k;
    }
    P = last_plan;
    return last_ok;
}

bool fused_fast_supported(const tb_shape &sh, int64_t n_tokens, int32_t k) {
    if (k < 1 || k > n_tokens) return false;
    FFPlan P;
    if (!ff_plan(sh, n_tokens, P)) return false;
    return P.C <= fused_chunks(sh, n_tokens);
}

cudaError_t launch_fused_fast(const tb_shape &sh, const tb_step_params &p, int64_t n, const uint16_t *q,
                              const uint16_t *q_imp, const uint16_t *K_new, const uint16_t *V_new,
                              const uint16_t *Wk, uint16_t *K, uint16_t *V, uint16_t *Kp, int32_t *idx_state,
                              int32_t *sel, int32_t *counts, uint16_t *out, const FastWs &w, int32_t sel_stride,
                              int32_t *dev_status, cudaStream_t st, int32_t k_keep, int64_t keep_lo,
                              int64_t keep_hi, int32_t *centres, int64_t cpre, int32_t ck) {
    FFPlan P;
    if (!ff_plan(sh, n + 1, P)) return cudaErrorNotSupported;
    FFArgs a;
    a.q = q; a.q_imp = q_imp; a.K_new = K_new; a.V_new = V_new; a.Wk = Wk;
    a.K = K; a.V = V; a.Kp = Kp;
    a.idx = idx_state; a.sel = sel; a.counts = counts; a.out = out;
    a.ctl = w.ctl; a.part = w.part; a.rec = w.rec; a.blk_above = w.blk_above; a.keys_g = w.keys_g; a.dbg = w.dbg;
    a.dev_status = dev_status;
    a.cap = sh.cap; a.n = n; a.keys_stride = w.keys_stride;
    a.Hq = sh.Hq; a.Hkv = sh.Hkv; a.D = sh.D; a.k = k_keep > 0 ? k_keep : p.k; a.agg = p.agg;
    a.sel_stride = sel_stride;
    a.keep_lo = keep_lo;
    a.keep_hi = keep_hi;
    a.centres = ck > 0 ? centres : nullptr;
    a.cpre = cpre;
    a.ck = ck;
    a.scale = p.scale;
    a.C = P.C; a.NB = P.NB; a.blk_stride = (int)w.blk_stride; a.stage_cap = P.stage_cap;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(P.C * sh.B * sh.Hkv));
    cfg.blockDim = dim3(kFFThreads);
    cfg.dynamicSmemBytes = P.smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
#define TB_FF_LAUNCH(CP, DTT, GMC)                                                          \
    if (P.cpt == CP && sh.D == DTT && P.gm == GMC)                                          \
        return k_keep > 0 ? cudaLaunchKernelEx(&cfg, fused_fast_kernel<CP, DTT, GMC, true>, a) \
                          : cudaLaunchKernelEx(&cfg, fused_fast_kernel<CP, DTT, GMC, false>, a);
    TB_FF_CASES(TB_FF_LAUNCH)
#undef TB_FF_LAUNCH
    return cudaErrorNotSupported;
}

}  // namespace tb
