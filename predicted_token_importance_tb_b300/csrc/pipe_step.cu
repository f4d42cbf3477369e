// The decode step (T = 1, r = 0) as three kernels with no grid-wide waits
// ("TokenButler: Token Importance is Predictable", gist.science summary,
// Core Architecture: the importance query scores every cached token against
// its projected key and a fixed budget of individual tokens is kept; arXiv
// abstract and Significance: exact attention over only those rows, the full
// cache kept in device memory).
//
// pipe_select_kernel, grid (chunks, rows): each CTA streams its chunk of the
//   row's projected keys [0, n) through a ring of bulk copies, scores every
//   token, stores its order-preserving key and adds it to the row's 12-bit
//   histogram.
// pipe_bracket_kernel, grid (chunks, rows), a programmatic dependent of the
//   selection: every CTA finds the bin b1 that holds the row's k-th ranked
//   token, counts its chunk's tokens above b1 and lists the ones inside; the
//   row's last CTA resolves the k-th ranked token exactly among those (radix
//   passes over the 64-bit value key:~index) and writes the cut and every
//   chunk's output offset.
// pipe_attend_kernel, grid (chunks, rows), a programmatic dependent of the
//   bracket: appends the new token n (its K and V rows and its projected
//   key), scores it with the same arithmetic, and decides whether it
//   displaces the row's k-th token (the top k of n + 1 tokens is the top k of
//   {top k of [0, n)} plus token n). It writes its chunk's kept tokens to idx
//   and sel at the chunk's offset, gathers their K/V rows with bulk copies
//   (up to three rounds in flight), attends on the tensor cores, and the
//   row's last CTA merges the chunks' partial softmax states.
//
// Two orders of the attention kernel's work: STEP (the kernel follows the
// bracket of the same step: this step's inputs are read and the tokens above
// b1, which are kept whatever the cut, are gathered before the programmatic
// wait; the cut's results are read after it) and CHAIN (the kernel follows
// the previous layer's attention kernel on its stream and its own layer's
// bracket on the other: everything waits for both, and the early launch only
// hides the launch itself).
#include "attn_mma.cuh"
#include "kernels.cuh"

namespace tb {

constexpr int kPipeThreads = 256;
constexpr int kPipeWarps = kPipeThreads / 32;
constexpr int kPipeStageTok = 256;   // tokens per stage of the projected-key ring
constexpr int kPipeMaxStages = 8;    // stages in flight per CTA (at most)
constexpr int kPipeRound = 64;       // K/V rows per gather round
constexpr int kPipeSeg = 2048;       // keys compacted per segment (8 per thread)

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ------------------------------------------------------------------ scores

__device__ __forceinline__ float pdot8(const float *q, uint4 v, float acc) {
    acc = fmaf(q[0], bf16_lo(v.x), acc);
    acc = fmaf(q[1], bf16_hi(v.x), acc);
    acc = fmaf(q[2], bf16_lo(v.y), acc);
    acc = fmaf(q[3], bf16_hi(v.y), acc);
    acc = fmaf(q[4], bf16_lo(v.z), acc);
    acc = fmaf(q[5], bf16_hi(v.z), acc);
    acc = fmaf(q[6], bf16_lo(v.w), acc);
    acc = fmaf(q[7], bf16_hi(v.w), acc);
    return acc;
}

// Order in which token t reads its NV 16-byte pieces: consecutive tokens start
// at different pieces, so eight lanes reading eight rows touch eight distinct
// bank groups of shared memory.
template <int NV>
__device__ __forceinline__ int piece_rot(int64_t t) {
    constexpr int SH = NV >= 8 ? 0 : NV == 4 ? 1 : NV == 2 ? 2 : 3;
    return (int)((t >> SH) & (NV - 1));
}

// fp32 importance score of token t from its projected key (NV pieces in
// shared memory): the dot product with the group-mean query (mean) or the
// largest of the G heads' dot products (max). qv holds the mean query [dp]
// or the G queries [G][dp]. The pieces are summed in piece_rot order; the
// selection and the attention kernel both score through this function, so a
// token's score is the same number in both.
template <int NV>
__device__ __forceinline__ float pipe_score(const float *qv, const uint4 *kp, int64_t t, int G, int agg) {
    const int rot = piece_rot<NV>(t);
    uint4 v[NV];
#pragma unroll
    for (int j = 0; j < NV; ++j) v[j] = kp[(j + rot) & (NV - 1)];
    if (agg == TB_AGG_MEAN) {
        float acc = 0.f;
#pragma unroll
        for (int j = 0; j < NV; ++j) acc = pdot8(qv + 8 * ((j + rot) & (NV - 1)), v[j], acc);
        return acc;
    }
    float out = -INFINITY;
    for (int g = 0; g < G; ++g) {
        float acc = 0.f;
#pragma unroll
        for (int j = 0; j < NV; ++j) acc = pdot8(qv + g * NV * 8 + 8 * ((j + rot) & (NV - 1)), v[j], acc);
        out = fmaxf(out, acc);
    }
    return out;
}

// The KV head's importance queries as fp32 in shared memory: their mean over
// the G heads (mean, summed in head order) or all G of them (max). Every
// value is loaded by its own thread, so the loads are in flight together.
// qv holds G * dp floats. All threads must call it.
__device__ __forceinline__ void pipe_load_qimp(const uint16_t *q_imp, int b, int h, int Hq, int G, int dp, int agg,
                                               float *qv) {
    const uint16_t *qrow = q_imp + ((int64_t)b * Hq + (int64_t)h * G) * dp;
    for (int i = threadIdx.x; i < G * dp; i += blockDim.x) qv[i] = bf16_to_f(qrow[i]);
    __syncthreads();
    if (agg == TB_AGG_MEAN) {
        const float inv = 1.0f / (float)G;
        if ((int)threadIdx.x < dp) {
            float a = 0.f;
            for (int g = 0; g < G; ++g) a += qv[g * dp + threadIdx.x];
            qv[threadIdx.x] = a * inv;   // (only this thread reads or writes column threadIdx.x)
        }
    }
}

// Total order of the selection: a token ranks above another when its key is
// larger, or the keys are equal and its index smaller.
__device__ __forceinline__ uint64_t rank_value(uint32_t key, int64_t t) {
    return ((uint64_t)key << 32) | (uint64_t)(~(uint32_t)t);
}

// The row's histogram (kPipeHBins words in global memory) into registers:
// every thread's four 16-byte loads are in flight together.
struct HistRegs {
    uint4 v[kPipeHBins / (4 * kPipeThreads)];
};
__device__ __forceinline__ HistRegs hist_load(const uint32_t *g) {
    HistRegs r;
    const uint4 *g4 = reinterpret_cast<const uint4 *>(g);
#pragma unroll
    for (int i = 0; i < kPipeHBins / (4 * kPipeThreads); ++i) r.v[i] = __ldcg(g4 + i * kPipeThreads + threadIdx.x);
    return r;
}
__device__ __forceinline__ void hist_store(const HistRegs &r, uint32_t *s) {
    uint4 *s4 = reinterpret_cast<uint4 *>(s);
#pragma unroll
    for (int i = 0; i < kPipeHBins / (4 * kPipeThreads); ++i) s4[i * kPipeThreads + threadIdx.x] = r.v[i];
}

// All threads wait for phase `parity` of `bar`, bounded; false (and
// TB_ERR_TIMEOUT recorded) if any thread gave up.
__device__ __forceinline__ bool pipe_wait(uint64_t *bar, uint32_t parity, int *abort_flag, int32_t *dev_status) {
    if (!mbarrier_wait_bounded(bar, parity, kWaitLimitNs)) {
        *abort_flag = 1;
        set_status(dev_status, TB_ERR_TIMEOUT);
    }
    __syncthreads();
    return *abort_flag == 0;
}

// ------------------------------------------------------------------ selection

struct PipeSel {
    const uint16_t *q_imp, *Kp;
    PipeRow *ctl;
    uint32_t *keys;
    int64_t keys_stride, cap, n;
    int Hq, Hkv, agg, C, cs;
    int stages;   // stages of the ring in flight (<= kPipeMaxStages)
    int32_t *dev_status;
};

// Digit d of a histogram h[0, nb) (counted from the top) holding the need-th
// largest entry: above = entries in the digits above d. nb is a multiple of
// the block size. All threads must call it; the result is in *sd, *sabove.
__device__ __forceinline__ void pick_digit(const uint32_t *h, int nb, uint32_t need, uint32_t *scan,
                                           uint32_t *sd, uint32_t *sabove) {
    const int per = nb / kPipeThreads;
    const int hi = nb - per * (int)threadIdx.x;   // this thread's bins [hi - per, hi), top first
    uint32_t local = 0;
    for (int j = hi - 1; j >= hi - per; --j) local += h[j];
    uint32_t total;
    const uint32_t excl = block_exclusive_scan(local, scan, total);
    if (excl < need && excl + local >= need) {
        uint32_t acc = excl;
        for (int j = hi - 1; j >= hi - per; --j) {
            if (acc + h[j] >= need) {
                *sd = (uint32_t)j;
                *sabove = acc;
                break;
            }
            acc += h[j];
        }
    }
    __syncthreads();
}

// Stream the chunk's projected keys, score every token, store its key, and
// add the chunk's histogram to the row's.
template <int NV>
__global__ void __launch_bounds__(kPipeThreads) pipe_select_kernel(const PipeSel a) {
    extern __shared__ __align__(128) uint8_t smb[];
    __shared__ __align__(8) uint64_t bars[kPipeMaxStages];
    __shared__ int s_abort;
    constexpr int DP = NV * 8;
    constexpr int STB = kPipeStageTok * DP * 2;   // bytes per stage
    const int S = a.stages;
    uint8_t *ring = smb;
    uint32_t *hist = reinterpret_cast<uint32_t *>(ring + S * STB);
    float *qv = reinterpret_cast<float *>(hist + kPipeHBins);
    const int row = blockIdx.y, chunk = blockIdx.x;
    const int b = row / a.Hkv, h = row % a.Hkv, G = a.Hq / a.Hkv;
    const int64_t t0 = (int64_t)chunk * a.cs;
    const int64_t t1 = t0 + a.cs < a.n ? t0 + a.cs : a.n;
    const int ntok = t1 > t0 ? (int)(t1 - t0) : 0;
    const int nst = (ntok + kPipeStageTok - 1) / kPipeStageTok;
    const uint8_t *src = reinterpret_cast<const uint8_t *>(a.Kp + ((int64_t)row * a.cap + t0) * DP);
    PipeRow *ctl = a.ctl + row;

    pdl_trigger();   // the bracket kernel may be scheduled now; it waits for this grid to finish
    if (threadIdx.x == 0) {
        s_abort = 0;
        for (int s = 0; s < S; ++s) mbarrier_init(&bars[s], 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        for (int s = 0; s < S && s < nst; ++s) {
            const int nt = min(kPipeStageTok, ntok - s * kPipeStageTok);
            mbarrier_arrive_expect_tx(&bars[s], (uint32_t)(nt * DP * 2));
            bulk_g2s(ring + s * STB, src + (int64_t)s * STB, (uint32_t)(nt * DP * 2), &bars[s]);
        }
    }
    pipe_load_qimp(a.q_imp, b, h, a.Hq, G, DP, a.agg, qv);
    for (int i = threadIdx.x; i < kPipeHBins; i += kPipeThreads) hist[i] = 0u;
    __syncthreads();

    bool nan_seen = false;
    uint32_t *krow = a.keys + (int64_t)row * a.keys_stride;
    int st_stop = nst;   // the stage whose wait gave up, if one did
    for (int st = 0; st < nst; ++st) {
        const int slot = st % S;
        if (!pipe_wait(&bars[slot], (uint32_t)(st / S) & 1u, &s_abort, a.dev_status)) {
            st_stop = st;
            break;
        }
        const int nt = min(kPipeStageTok, ntok - st * kPipeStageTok);
        if ((int)threadIdx.x < nt) {
            const int64_t t = t0 + (int64_t)st * kPipeStageTok + threadIdx.x;
            const uint4 *kp = reinterpret_cast<const uint4 *>(ring + slot * STB) + threadIdx.x * NV;
            const uint32_t key = score_key(pipe_score<NV>(qv, kp, t, G, a.agg), nan_seen);
            krow[t] = key;
            atomicAdd(&hist[key >> (32 - kPipeHBits)], 1u);
        }
        __syncthreads();   // the stage's buffer is consumed
        if (threadIdx.x == 0 && st + S < nst) {
            const int s2 = st + S;
            const int nt2 = min(kPipeStageTok, ntok - s2 * kPipeStageTok);
            mbarrier_arrive_expect_tx(&bars[slot], (uint32_t)(nt2 * DP * 2));
            bulk_g2s(ring + slot * STB, src + (int64_t)s2 * STB, (uint32_t)(nt2 * DP * 2), &bars[slot]);
        }
    }
    if (nan_seen) set_status(a.dev_status, TB_ERR_NONFINITE);
    if (s_abort) {
        // a timed-out wait (recorded in the status word): wait, bounded, for the copies this CTA still has
        // in flight (stages [st_stop, st_stop + S) were issued and not consumed) before it exits
        for (int st = st_stop; st < nst && st < st_stop + S; ++st)
            mbarrier_wait_bounded(&bars[st % S], (uint32_t)(st / S) & 1u, kWaitLimitNs);
        return;
    }
    for (int i = threadIdx.x; i < kPipeHBins; i += kPipeThreads) {
        const uint32_t c = hist[i];
        if (c) atomicAdd(ctl->hist + i, c);
    }
}

// ------------------------------------------------------------------ bracket

struct PipeBr {
    PipeRow *ctl;
    const uint32_t *keys;
    uint2 *cand;
    int64_t keys_stride, n;
    int k, C, cs;
    int32_t *dev_status;
};

// One radix pass of the cut: the histogram of the w bits below the top pbits
// of every entry whose top pbits equal prefix, then the digit holding the
// need-th largest. Entries come from the shared list (LIST) or from the
// row's keys in global memory. h holds 1 << w words. All threads call it.
template <bool LIST>
__device__ void radix_pass(const uint2 *list, uint32_t c, const uint32_t *krow, int64_t n, uint64_t &prefix,
                           int &pbits, uint32_t &need, int w, uint32_t *h, uint32_t *scan, uint32_t *sd,
                           uint32_t *sabove) {
    const int nb = 1 << w;
    const int tid = threadIdx.x;
    __syncthreads();
    for (int i = tid; i < nb; i += kPipeThreads) h[i] = 0u;
    __syncthreads();
    const int sh_hi = 64 - pbits, sh_lo = 64 - pbits - w;
    const uint32_t mask = (uint32_t)(nb - 1);
    if (LIST) {
        for (uint32_t i = tid; i < c; i += kPipeThreads) {
            const uint64_t v = rank_value(list[i].x, list[i].y);
            if ((v >> sh_hi) == prefix) atomicAdd(&h[(uint32_t)(v >> sh_lo) & mask], 1u);
        }
    } else {
        const uint4 *k4 = reinterpret_cast<const uint4 *>(krow);
        const int64_t n4 = (n + 3) / 4;
        for (int64_t i = tid; i < n4; i += kPipeThreads) {
            const uint4 v4 = __ldcg(k4 + i);
            const uint32_t kk[4] = {v4.x, v4.y, v4.z, v4.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int64_t t = 4 * i + j;
                if (t < n) {
                    const uint64_t v = rank_value(kk[j], t);
                    if ((v >> sh_hi) == prefix) atomicAdd(&h[(uint32_t)(v >> sh_lo) & mask], 1u);
                }
            }
        }
    }
    __syncthreads();
    pick_digit(h, nb, need, scan, sd, sabove);
    prefix = (prefix << w) | *sd;
    pbits += w;
    need -= *sabove;
}

// Each CTA: the row's threshold bin b1 (the 12-bit bin of the k1-th ranked
// token, k1 = min(k, n)) from the finished histogram; its chunk's tokens
// above b1 are counted and those inside b1 appended to the row's candidate
// list. The row's last CTA resolves the k1-th ranked token exactly among the
// candidates (radix passes over key:~index) and writes the cut and every
// chunk's output offset.
__global__ void __launch_bounds__(kPipeThreads) pipe_bracket_kernel(const PipeBr a) {
    extern __shared__ __align__(128) uint8_t smb[];
    __shared__ uint32_t scan[40];
    __shared__ uint32_t s_d, s_above, s_last, s_red[kPipeWarps];
    __shared__ uint32_t s_cin[kPipeMaxChunks];
    __shared__ uint64_t s_tail[32], s_vcut;
    __shared__ uint32_t s_nloc, s_gbase;
    uint32_t *h = reinterpret_cast<uint32_t *>(smb);                 // kPipeHBins words
    uint2 *L = reinterpret_cast<uint2 *>(smb + kPipeHBins * 4);        // kPipeCandCap entries
    const int row = blockIdx.y, chunk = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    PipeRow *ctl = a.ctl + row;
    const int64_t n = a.n;
    const uint32_t k1 = (uint32_t)(a.k < n ? a.k : n);
    const uint32_t *krow = a.keys + (int64_t)row * a.keys_stride;
    uint2 *crow = a.cand + (int64_t)row * kPipeCandCap;

    pdl_wait();      // the selection kernel has finished: keys and histogram are complete
    pdl_trigger();   // the attention kernel may start; its early phase reads only those
    hist_store(hist_load(ctl->hist), h);
    __syncthreads();
    pick_digit(h, kPipeHBins, k1, scan, &s_d, &s_above);
    const uint32_t b1 = s_d, A1 = s_above;

    // this chunk: tokens above b1, and the entries of b1 gathered in a local list (L; the last CTA reuses
    // the space), then copied to the row's list at a place reserved with one atomic
    if (tid == 0) s_nloc = 0u;
    __syncthreads();
    const int64_t t0 = (int64_t)chunk * a.cs;
    const int64_t t1 = t0 + a.cs < n ? t0 + a.cs : n;
    const uint4 *k4 = reinterpret_cast<const uint4 *>(krow + t0);
    const int n4 = (int)((t1 - t0 + 3) / 4);
    constexpr int UB = 8;   // 16-byte loads in flight per thread
    uint32_t above = 0;
    for (int base = 0; base < n4; base += kPipeThreads * UB) {
        uint4 v[UB];
#pragma unroll
        for (int u = 0; u < UB; ++u) {
            const int i = base + u * kPipeThreads + tid;
            v[u] = i < n4 ? __ldcg(k4 + i) : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int u = 0; u < UB; ++u) {
            const int i = base + u * kPipeThreads + tid;
            const uint32_t kk[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int64_t t = t0 + 4 * (int64_t)i + j;
                if (i < n4 && t < t1) {
                    const uint32_t top = kk[j] >> (32 - kPipeHBits);
                    if (top > b1) {
                        ++above;
                    } else if (top == b1) {
                        const uint32_t p = atomicAdd(&s_nloc, 1u);
                        if (p < (uint32_t)kPipeCandCap) L[p] = make_uint2(kk[j], (uint32_t)t);
                    }
                }
            }
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) above += __shfl_xor_sync(0xFFFFFFFFu, above, o);
    if (lane == 0) s_red[warp] = above;
    __syncthreads();
    const uint32_t nloc = s_nloc < (uint32_t)kPipeCandCap ? s_nloc : (uint32_t)kPipeCandCap;
    if (tid == 0) {
        uint32_t sum = 0;
        for (int w = 0; w < kPipeWarps; ++w) sum += s_red[w];
        ctl->cab[chunk] = sum;
        s_gbase = nloc ? atomicAdd(&ctl->ncand, nloc) : 0u;
        if (s_nloc > (uint32_t)kPipeCandCap || s_gbase + nloc > (uint32_t)kPipeCandCap) atomicOr(&ctl->overflow, 1u);
    }
    __syncthreads();
    for (uint32_t i = tid; i < nloc; i += kPipeThreads)
        if (s_gbase + i < (uint32_t)kPipeCandCap) crow[s_gbase + i] = L[i];
    __syncthreads();
    if (tid == 0) {
        __threadfence();
        const uint32_t prev = atomicAdd(&ctl->done2, 1u);
        s_last = prev == (uint32_t)(a.C - 1) ? 1u : 0u;
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();

    // the row's last CTA: the exact cut inside b1
    uint64_t prefix = b1;
    int pbits = kPipeHBits;
    uint32_t need = k1 - A1;
    const uint32_t nc = __ldcg(&ctl->ncand);
    const bool listed = __ldcg(&ctl->overflow) == 0u;
    for (int i = tid; i < kPipeMaxChunks; i += kPipeThreads) s_cin[i] = 0u;
    const int widths[5] = {10, 10, 11, 11, 10};
    uint64_t v_cut;
    if (listed) {
        for (uint32_t i = tid; i < nc; i += kPipeThreads) L[i] = __ldcg(crow + i);
        radix_pass<true>(L, nc, nullptr, 0, prefix, pbits, need, widths[0], h, scan, &s_d, &s_above);
        const uint32_t c2 = h[s_d];   // entries sharing the top 22 bits of the cut
        if (c2 <= 32) {
            // few left: one warp gathers them and ranks each against the others
            if (warp == 0) {
                uint32_t got = 0;
                for (uint32_t base = 0; base < nc; base += 32) {
                    const uint32_t i = base + lane;
                    uint64_t v = 0;
                    bool m = false;
                    if (i < nc) {
                        v = rank_value(L[i].x, L[i].y);
                        m = (v >> (64 - pbits)) == prefix;
                    }
                    const uint32_t ball = __ballot_sync(0xFFFFFFFFu, m);
                    if (m) s_tail[got + __popc(ball & ((1u << lane) - 1u))] = v;
                    got += __popc(ball);
                }
                __syncwarp();
                const uint64_t v = lane < (int)c2 ? s_tail[lane] : 0;
                uint32_t above = 0;
                for (uint32_t j = 0; j < c2; ++j) above += s_tail[j] > v ? 1u : 0u;
                if (lane < (int)c2 && above == need - 1) s_vcut = v;
            }
            __syncthreads();
            v_cut = s_vcut;
        } else {
            for (int wi = 1; wi < 5; ++wi)
                radix_pass<true>(L, nc, nullptr, 0, prefix, pbits, need, widths[wi], h, scan, &s_d, &s_above);
            v_cut = prefix;
        }
    } else {
        for (int wi = 0; wi < 5; ++wi)
            radix_pass<false>(nullptr, 0, krow, n, prefix, pbits, need, widths[wi], h, scan, &s_d, &s_above);
        v_cut = prefix;   // all 64 bits: the k1-th ranked token
    }
    // kept tokens inside b1 per chunk
    if (listed) {
        for (uint32_t i = tid; i < nc; i += kPipeThreads) {
            const uint2 e = L[i];
            if (rank_value(e.x, e.y) >= v_cut) atomicAdd(&s_cin[e.y / (uint32_t)a.cs], 1u);
        }
    } else {
        const uint4 *r4 = reinterpret_cast<const uint4 *>(krow);
        const int64_t m4 = (n + 3) / 4;
        for (int64_t i = tid; i < m4; i += kPipeThreads) {
            const uint4 v4 = __ldcg(r4 + i);
            const uint32_t kk[4] = {v4.x, v4.y, v4.z, v4.w};
            uint32_t in = 0;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int64_t t = 4 * i + j;
                if (t < n && (kk[j] >> (32 - kPipeHBits)) == b1 && rank_value(kk[j], t) >= v_cut) ++in;
            }
            if (in) atomicAdd(&s_cin[(4 * i) / a.cs], in);
        }
    }
    __syncthreads();
    for (int c = tid; c < a.C; c += kPipeThreads) s_cin[c] += __ldcg(&ctl->cab[c]);
    __syncthreads();
    if (tid == 0) {
        int acc = 0;
        for (int c = 0; c < a.C; ++c) {
            ctl->offs[c] = acc;
            acc += (int)s_cin[c];
        }
        ctl->offs[a.C] = acc;
        if (acc != (int)k1) set_status(a.dev_status, TB_ERR_INVALID_ARG);   // cannot happen: counts disagree
        ctl->b1 = b1;
        ctl->cut_key = (uint32_t)(v_cut >> 32);
        ctl->cut_idx = (int32_t)(~(uint32_t)v_cut);
        ctl->k1 = (int32_t)k1;
        ctl->done2 = 0u;   // ready for the next call
        ctl->ncand = 0u;
        ctl->overflow = 0u;
    }
}

// ------------------------------------------------------------------ attention

struct PipeAttn {
    const uint16_t *q, *q_imp, *K_new, *V_new, *Wk;
    uint16_t *K, *V, *Kp;
    int32_t *idx, *sel, *counts;
    uint16_t *out;
    PipeRow *ctl;
    const uint32_t *keys;
    int64_t keys_stride;
    float *part;
    int64_t cap, n;
    int Hq, Hkv, agg, k, C, cs, sel_stride;
    float scale;
    int32_t *dev_status;
};

constexpr int kPipeBufs = 3;   // gather rounds in flight

__host__ __device__ constexpr int pipe_attn_smem_bytes(int DT, int DP) {
    return kPipeBufs * kPipeRound * (4 * DT + 16)   // gather rounds
           + 16 * (4 * DT + 16)                     // the new token's slot (+15 zero slots)
           + 16 * (2 * DT + 16)                     // query tile
           + kPipeSeg * 4                           // keys of the current segment
           + kPipeSeg * 4                           // tokens queued for gathering
           + 16 * DP * 4                            // importance queries
           + DT * 4                                 // the new key (fp32)
           + kPipeThreads * 4;                      // projection partial sums
}

template <int DT, int NV, bool CHAIN>
__global__ void __maxnreg__(168) pipe_attend_kernel(const PipeAttn a) {
    extern __shared__ __align__(128) uint8_t smb[];
    __shared__ uint32_t scan[40];
    __shared__ __align__(16) uint16_t kpn[64];   // the new token's projected key (bf16 bits), read as uint4
    __shared__ int s_abort, s_cnt[kPipeBufs];
    __shared__ uint32_t s_d, s_above, s_b1, s_ck, s_last;
    __shared__ int32_t s_ci, s_k1, s_off;
    constexpr int SB = 4 * DT + 16, CPR = DT / 8, NT = DT / 8, QS = 2 * DT + 16, DP = NV * 8;
    uint8_t *X = smb;
    uint8_t *xn = X + kPipeBufs * kPipeRound * SB;
    uint8_t *qsm = xn + 16 * SB;
    uint32_t *segk = reinterpret_cast<uint32_t *>(qsm + 16 * QS);
    int32_t *queue = reinterpret_cast<int32_t *>(segk + kPipeSeg);
    float *qv = reinterpret_cast<float *>(queue + kPipeSeg);
    float *kn = qv + 16 * DP;
    float *comb = kn + DT;
    const int row = blockIdx.y, chunk = blockIdx.x;
    const int b = row / a.Hkv, h = row % a.Hkv, G = a.Hq / a.Hkv;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t n = a.n;
    const int64_t t0 = (int64_t)chunk * a.cs;
    const int64_t t1 = t0 + a.cs < n ? t0 + a.cs : n;
    const bool owner = chunk == a.C - 1;   // appends the new token, attends it and writes its entry
    const uint16_t *Kh = a.K + (int64_t)row * a.cap * DT;
    const uint16_t *Vh = a.V + (int64_t)row * a.cap * DT;
    const uint32_t *krow = a.keys + (int64_t)row * a.keys_stride;
    PipeRow *ctl = a.ctl + row;

    pdl_trigger();
    if (tid == 0) s_abort = 0;
    __syncthreads();
    int r_issue = 0, r_done = 0;   // gather rounds issued and consumed (uniform); one cp.async group each

    // this step's own inputs: query tile, the new K/V row (slot 0 of xn), its projected key and score
    uint32_t key_n = 0;
    auto part_inputs = [&]() {
        constexpr int SL = kPipeThreads / DP, DL = DT / SL;
        const int j = tid % DP, sl = tid / DP;
        // every global load of this phase is issued before any of them is used
        uint16_t wreg[DL];   // this thread's slice of Wk[h][:, j]
        {
            const uint16_t *W = a.Wk + ((int64_t)h * DT + sl * DL) * DP + j;
#pragma unroll
            for (int d = 0; d < DL; ++d) wreg[d] = W[(int64_t)d * DP];
        }
        const int gq = tid / CPR, cq = tid % CPR;   // one 16-byte piece of the 16 x D query tile per thread
        uint4 q4 = make_uint4(0u, 0u, 0u, 0u);
        if (gq < G) q4 = *reinterpret_cast<const uint4 *>(a.q + ((int64_t)b * a.Hq + (int64_t)h * G + gq) * DT + cq * 8);
        const uint16_t *kn_src = a.K_new + (int64_t)row * DT, *vn_src = a.V_new + (int64_t)row * DT;
        uint4 nv4 = make_uint4(0u, 0u, 0u, 0u);    // piece tid of the new K row (tid < CPR) or V row
        if (tid < CPR) nv4 = *reinterpret_cast<const uint4 *>(kn_src + tid * 8);
        else if (tid < 2 * CPR) nv4 = *reinterpret_cast<const uint4 *>(vn_src + (tid - CPR) * 8);
        pipe_load_qimp(a.q_imp, b, h, a.Hq, G, DP, a.agg, qv);
        if (tid < 16 * CPR) *reinterpret_cast<uint4 *>(qsm + gq * QS + cq * 16) = q4;
        for (int x = tid; x < SB; x += kPipeThreads)   // the 16 slots of xn: slot 0 = (K_new, V_new), rest zero
            *reinterpret_cast<uint4 *>(xn + x * 16) = (x == tid && tid < 2 * CPR) ? nv4 : make_uint4(0u, 0u, 0u, 0u);
        if (tid < CPR) {
            kn[tid * 8 + 0] = bf16_lo(nv4.x);
            kn[tid * 8 + 1] = bf16_hi(nv4.x);
            kn[tid * 8 + 2] = bf16_lo(nv4.y);
            kn[tid * 8 + 3] = bf16_hi(nv4.y);
            kn[tid * 8 + 4] = bf16_lo(nv4.z);
            kn[tid * 8 + 5] = bf16_hi(nv4.z);
            kn[tid * 8 + 6] = bf16_lo(nv4.w);
            kn[tid * 8 + 7] = bf16_hi(nv4.w);
        }
        __syncthreads();
        // Kp row of the new token: fp32 sums over slices of D, added in slice order, one rounding
        {
            float acc = 0.f;
#pragma unroll
            for (int d = 0; d < DL; ++d) acc = fmaf(kn[sl * DL + d], bf16_to_f(wreg[d]), acc);
            comb[tid] = acc;
        }
        __syncthreads();
        if (tid < DP) {
            float sum = 0.f;
            for (int s2 = 0; s2 < SL; ++s2) sum += comb[s2 * DP + tid];
            kpn[tid] = f_to_bf16(sum);
        }
        __syncthreads();
        bool nan_seen = false;
        key_n = score_key(pipe_score<NV>(qv, reinterpret_cast<const uint4 *>(kpn), n, G, a.agg), nan_seen);
        if (nan_seen && tid == 0) set_status(a.dev_status, TB_ERR_NONFINITE);
        if (owner) {
            if (tid < 2 * CPR) {
                uint16_t *dst = (tid < CPR ? a.K : a.V) + ((int64_t)row * a.cap + n) * DT + (tid % CPR) * 8;
                *reinterpret_cast<uint4 *>(dst) = nv4;
            }
            if (tid < DP) a.Kp[((int64_t)row * a.cap + n) * DP + tid] = kpn[tid];
        }
    };

    // the bracket kernel's result for this row and chunk
    auto part_cut = [&]() {
        if (tid == 0) {
            s_b1 = __ldcg(&ctl->b1);
            s_ck = __ldcg(&ctl->cut_key);
            s_ci = __ldcg(&ctl->cut_idx);
            s_k1 = __ldcg(&ctl->k1);
            s_off = __ldcg(&ctl->offs[chunk]);
        }
        __syncthreads();
    };

    // keys [lo, hi) of the chunk (hi - lo <= kPipeSeg) into segk, 8 per thread
    auto load_seg = [&](int64_t lo, int64_t hi) {
        const int64_t tb = lo + 8 * tid;
        const uint4 *p = reinterpret_cast<const uint4 *>(krow + tb);
        const uint4 x0 = tb < hi ? __ldcg(p) : make_uint4(0u, 0u, 0u, 0u);
        const uint4 x1 = tb + 4 < hi ? __ldcg(p + 1) : make_uint4(0u, 0u, 0u, 0u);
        *reinterpret_cast<uint4 *>(segk + 8 * tid) = x0;
        *reinterpret_cast<uint4 *>(segk + 8 * tid + 4) = x1;
        __syncthreads();
    };

    // one round: up to kPipeRound queued tokens' K/V rows into buffer r_issue % kPipeBufs in 16-byte cp.async
    // pieces from every thread (one bulk copy per 256-byte row, as before, is held back by the bulk-copy unit's
    // per-copy cost); padding slots up to a multiple of 16 get zeros (their V rows must be finite)
    auto issue = [&](int q0, int cnt) {
        const int buf = r_issue % kPipeBufs;
        uint8_t *Xb = X + (size_t)buf * kPipeRound * SB;
        const int pad_hi = (cnt + 15) & ~15;
        for (int x = tid; x < (pad_hi - cnt) * (SB / 16); x += kPipeThreads)
            *reinterpret_cast<uint4 *>(Xb + (size_t)(cnt + x / (SB / 16)) * SB + (x % (SB / 16)) * 16) =
                make_uint4(0u, 0u, 0u, 0u);
        if (tid == 0) s_cnt[buf] = cnt;
        __syncthreads();
        for (int x = tid; x < cnt * 2 * CPR; x += kPipeThreads) {
            const int ent = x / (2 * CPR), r = x % (2 * CPR);
            const bool isv = r >= CPR;
            const int pc = isv ? r - CPR : r;
            const int64_t t = queue[q0 + ent];
            cp_async16(Xb + (size_t)ent * SB + (isv ? 2 * DT : 0) + pc * 16, (isv ? Vh : Kh) + t * DT + pc * 8);
        }
        cp_async_commit();
        ++r_issue;
    };

    MmaAttn<NT> A;
    A.m0 = A.m1 = -INFINITY;
    A.l0 = A.l1 = 0.f;
#pragma unroll
    for (int t = 0; t < NT; ++t) A.o[t][0] = A.o[t][1] = A.o[t][2] = A.o[t][3] = 0.f;
    const float qscale = a.scale * kLog2e;

    // the oldest round in flight: wait, attend
    auto consume = [&]() -> bool {
        const int buf = r_done % kPipeBufs;
        // this thread's pieces of round r_done have landed once at most r_issue - r_done - 1 groups are pending
        const int pend = r_issue - r_done - 1;
        if (pend >= 2) asm volatile("cp.async.wait_group 2;" ::: "memory");
        else if (pend == 1) asm volatile("cp.async.wait_group 1;" ::: "memory");
        else asm volatile("cp.async.wait_group 0;" ::: "memory");
        __syncthreads();   // every thread's pieces of the round are visible to the CTA
        mma_attend<DT, kPipeWarps, false>(A, X + (size_t)buf * kPipeRound * SB, SB, s_cnt[buf], nullptr, 0, qsm,
                                          qscale);
        __syncthreads();   // the buffer is free again
        ++r_done;
        return true;
    };

    // issue the queue [q0, qlen) round by round, keeping up to kPipeBufs rounds in flight
    auto drain = [&](int q0, int qlen, bool finish) -> bool {
        while (true) {
            while (r_issue - r_done < kPipeBufs && q0 < qlen) {
                const int cnt = qlen - q0 < kPipeRound ? qlen - q0 : kPipeRound;
                issue(q0, cnt);
                q0 += cnt;
            }
            if (q0 >= qlen && (!finish || r_done == r_issue)) return true;
            if (!consume()) return false;
        }
    };

    // tokens above the threshold bin in segk[0, len) (positions lo..): those are kept whatever the cut
    // -> queue, ascending; returns how many
    auto queue_certain = [&](int64_t lo, int len, uint32_t b1) -> int {
        uint32_t mask = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int i = 8 * tid + j;
            if (i < len && (segk[i] >> (32 - kPipeHBits)) > b1) mask |= 1u << j;
        }
        uint32_t total;
        uint32_t pos = block_exclusive_scan(__popc(mask), scan, total);
#pragma unroll
        for (int j = 0; j < 8; ++j)
            if (mask & (1u << j)) queue[pos++] = (int32_t)(lo + 8 * tid + j);
        __syncthreads();
        return (int)total;
    };

    uint32_t b1;
    const int64_t seg0_hi = t0 + kPipeSeg < t1 ? t0 + kPipeSeg : t1;
    int pre = 0;   // certainly kept tokens of segment 0 whose gather is issued before the wait
    if (!CHAIN) {
        // the threshold bin, from the row's finished histogram (this kernel started after the bracket
        // kernel's wait, so after the selection kernel finished); its loads fly while this step's inputs
        // are read; X is free until the first gather
        const HistRegs hr = hist_load(ctl->hist);
        part_inputs();
        uint32_t *hh = reinterpret_cast<uint32_t *>(X);
        hist_store(hr, hh);
        __syncthreads();
        pick_digit(hh, kPipeHBins, (uint32_t)(a.k < n ? a.k : n), scan, &s_d, &s_above);
        b1 = s_d;
        load_seg(t0, seg0_hi);
        const int nq = queue_certain(t0, (int)(seg0_hi - t0), b1);
        pre = nq < kPipeBufs * kPipeRound ? nq : kPipeBufs * kPipeRound;
        drain(0, pre, false);
        pdl_wait();   // the bracket kernel has finished: the cut and the offsets are final
        part_cut();
    } else {
        // the previous layer's attention kernel and this layer's bracket kernel have both finished once the
        // wait returns (a captured graph may make either dependency the programmatic one)
        pdl_wait();
        part_cut();
        b1 = s_b1;
        load_seg(t0, seg0_hi);
        const int nq = queue_certain(t0, (int)(seg0_hi - t0), b1);
        pre = nq < kPipeBufs * kPipeRound ? nq : kPipeBufs * kPipeRound;
        drain(0, pre, false);   // the gathers fly while this layer's inputs are read
        part_inputs();
    }
    if (b1 != s_b1) set_status(a.dev_status, TB_ERR_INVALID_ARG);   // cannot happen: same histogram

    // does the new token displace the k-th ranked one?
    const bool room = s_k1 < a.k;                       // k = n + 1: every token is kept
    const bool include_n = room || key_n > s_ck;        // (n ranks below the cut on equal keys)
    const bool drop = !room && include_n;
    const int32_t e = s_ci;
    const uint64_t v_cut = rank_value(s_ck, s_ci);
    int32_t *irow = a.idx + (int64_t)row * a.k;
    int32_t *srow = a.sel + (int64_t)row * a.sel_stride;
    const int kmax = a.k - (include_n ? 1 : 0);
    // the chunk offsets count the dropped token in its own chunk: later chunks move down one place (inside
    // that chunk the kept mask below already leaves it out)
    const int shift = (drop && (int64_t)e < t0) ? 1 : 0;

    // every segment: the kept tokens' entries of idx and sel, and their gather (segment 0's first `pre`
    // certainly kept tokens are in flight already); the next segment's keys are requested while this one is
    // worked on, and gather rounds stay in flight from one segment to the next
    int rank_base = 0;
    bool ok = true;
    const int nseg = (int)((t1 - t0 + kPipeSeg - 1) / kPipeSeg);
    for (int sidx = 0; sidx < nseg && ok; ++sidx) {
        const int64_t lo = t0 + (int64_t)sidx * kPipeSeg;
        const int64_t hi = lo + kPipeSeg < t1 ? lo + kPipeSeg : t1;
        const int len = (int)(hi - lo);
        uint4 nx0 = make_uint4(0u, 0u, 0u, 0u), nx1 = make_uint4(0u, 0u, 0u, 0u);
        if (sidx + 1 < nseg) {
            const int64_t nlo = hi, nhi = hi + kPipeSeg < t1 ? hi + kPipeSeg : t1;
            const int64_t tb = nlo + 8 * tid;
            const uint4 *p = reinterpret_cast<const uint4 *>(krow + tb);
            if (tb < nhi) nx0 = __ldcg(p);
            if (tb + 4 < nhi) nx1 = __ldcg(p + 1);
        }
        uint32_t kept = 0, cert = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int i = 8 * tid + j;
            const int64_t t = lo + i;
            if (i < len) {
                const uint32_t key = segk[i], top = key >> (32 - kPipeHBits);
                const bool c = top > b1;
                const bool in = top == b1 && rank_value(key, t) >= v_cut && !(drop && t == e);
                if (c) cert |= 1u << j;
                if (c || in) kept |= 1u << j;
            }
        }
        // positions in idx / sel
        uint32_t total;
        uint32_t pos = block_exclusive_scan(__popc(kept), scan, total);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            if (kept & (1u << j)) {
                const int64_t t = lo + 8 * tid + j;
                const int p = s_off + rank_base + (int)pos - shift;
                if (p >= 0 && p < kmax) {
                    irow[p] = (int32_t)t;
                    srow[p] = (int32_t)t;
                } else {
                    set_status(a.dev_status, TB_ERR_INVALID_ARG);   // a selection result out of range
                }
                ++pos;
            }
        }
        rank_base += (int)total;
        // the gather queue: the kept tokens not issued before the wait (all of them past segment 0)
        uint32_t cpos = 0, ctot = 0;
        if (sidx == 0) cpos = block_exclusive_scan(__popc(cert), scan, ctot);
        uint32_t mq = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            if (kept & (1u << j)) {
                const bool issued = sidx == 0 && (cert & (1u << j)) && cpos < (uint32_t)pre;
                if (!issued) mq |= 1u << j;
            }
            if (cert & (1u << j)) ++cpos;
        }
        uint32_t qt;
        uint32_t qp = block_exclusive_scan(__popc(mq), scan, qt);
        // (the scans' barriers order this segment's reads of segk and the previous queue's issue before
        // these writes)
#pragma unroll
        for (int j = 0; j < 8; ++j)
            if (mq & (1u << j)) queue[qp++] = (int32_t)(lo + 8 * tid + j);
        *reinterpret_cast<uint4 *>(segk + 8 * tid) = nx0;
        *reinterpret_cast<uint4 *>(segk + 8 * tid + 4) = nx1;
        __syncthreads();
        ok = drain(0, (int)qt, sidx + 1 == nseg);
    }
    if (s_abort || !ok) {
        // the gather rounds still in flight land before the CTA exits
        asm volatile("cp.async.wait_all;" ::: "memory");
        return;
    }
    if (owner) {
        if (include_n) mma_attend<DT, kPipeWarps, false>(A, xn, SB, 1, nullptr, 0, qsm, qscale);
        if (tid == 0) {
            if (include_n) {
                irow[a.k - 1] = (int32_t)n;
                srow[a.k - 1] = (int32_t)n;
            }
            a.counts[row] = a.k;
        }
    }

    // the warps' states -> this chunk's partial (m, l, acc[D]) per head
    A.l0 += __shfl_xor_sync(0xFFFFFFFFu, A.l0, 1);
    A.l0 += __shfl_xor_sync(0xFFFFFFFFu, A.l0, 2);
    A.l1 += __shfl_xor_sync(0xFFFFFFFFu, A.l1, 1);
    A.l1 += __shfl_xor_sync(0xFFFFFFFFu, A.l1, 2);
    __syncthreads();   // X is free: the warps' states go there
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
    float *prow = a.part + (int64_t)row * kPipeMaxChunks * G * sg;
    for (int x = tid; x < G * DT; x += kPipeThreads) {
        const int g = x / DT, d = x % DT;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kPipeWarps; ++w) M = fmaxf(M, ws[((int64_t)w * G + g) * sg]);
        float Lsum = 0.f, Acc = 0.f;
#pragma unroll
        for (int w = 0; w < kPipeWarps; ++w) {
            const float *sw = ws + ((int64_t)w * G + g) * sg;
            const float wt = rescale_w(sw[0], M);
            Lsum = fmaf(wt, sw[1], Lsum);
            Acc = fmaf(wt, sw[2 + d], Acc);
        }
        float *o = prow + ((int64_t)chunk * G + g) * sg;
        if (d == 0) {
            o[0] = M;
            o[1] = Lsum;
        }
        o[2 + d] = Acc;
    }
    // the last CTA of the row merges the chunks, then clears the row's histogram for the next call
    __syncthreads();
    if (tid == 0) {
        __threadfence();
        const uint32_t prev = atomicAdd(&ctl->done3, 1u);
        s_last = prev == (uint32_t)(a.C - 1) ? 1u : 0u;
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    attn_merge(prow, a.C, G, DT, a.out + ((int64_t)b * a.Hq + (int64_t)h * G) * DT, a.dev_status,
               reinterpret_cast<float *>(X));
    for (int i = tid; i < kPipeHBins; i += kPipeThreads) ctl->hist[i] = 0u;
    if (tid == 0) ctl->done3 = 0u;   // ready for the next call
}

// ------------------------------------------------------------------ host

bool pipe_supported(const tb_shape &sh, int64_t n, int32_t k) {
    const int G = sh.Hq / sh.Hkv;
    if (!(sh.D == 64 || sh.D == 128)) return false;
    if (!(sh.dp == 16 || sh.dp == 32 || sh.dp == 64)) return false;
    if (G > 16) return false;
    if (n < 1024 || k < 1 || (int64_t)k > n + 1) return false;
    if (n + 1 > ((int64_t)1 << 31) - 1) return false;
    return true;
}

PipeGeom pipe_geom(const tb_shape &sh, int64_t n) {
    const int rows = sh.B * sh.Hkv;
    const int sms = dev_info().sms > 0 ? dev_info().sms : 148;
    int C = sms / rows;
    if (C < 1) C = 1;
    if (C > kPipeMaxChunks) C = kPipeMaxChunks;
    int64_t cs = (n + C - 1) / C;
    cs = (cs + 15) / 16 * 16;
    PipeGeom g;
    g.cs = (int)cs;
    g.C = (int)((n + cs - 1) / cs);
    return g;
}

static size_t pipe_select_smem(int dp, int stages) {
    return (size_t)stages * kPipeStageTok * dp * 2 + kPipeHBins * 4 + 16 * dp * 4;
}

// Most ring stages the selection kernel's shared memory holds (227 KB per CTA).
static int pipe_select_max_stages(int dp) {
    int s = kPipeMaxStages;
    while (s > 2 && pipe_select_smem(dp, s) > (size_t)227 * 1024) --s;
    return s;
}

// Kernel attributes set once per thread and device (slot: one per kernel instance).
template <typename F>
static cudaError_t ensure_smem_attr(F *fn, size_t smem, int slot) {
    static thread_local int done_dev[32];
    static thread_local bool init = false;
    if (!init) {
        for (int &d : done_dev) d = -1;
        init = true;
    }
    const int dev = dev_info().device;
    if (done_dev[slot] == dev) return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e == cudaSuccess) done_dev[slot] = dev;
    return e;
}

static cudaLaunchConfig_t pdl_config(dim3 grid, size_t smem, cudaStream_t st, cudaLaunchAttribute *attr) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kPipeThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cfg;
}

cudaError_t launch_pipe_select(const tb_shape &sh, const PipeGeom &g, int agg, int64_t n, const uint16_t *q_imp,
                               const uint16_t *Kp, PipeRow *ctl, uint32_t *keys, int64_t keys_stride, bool chain,
                               int32_t *dev_status, cudaStream_t st) {
    PipeSel a;
    a.q_imp = q_imp;
    a.Kp = Kp;
    a.ctl = ctl;
    a.keys = keys;
    a.keys_stride = keys_stride;
    a.cap = sh.cap;
    a.n = n;
    a.Hq = sh.Hq;
    a.Hkv = sh.Hkv;
    a.agg = agg;
    a.C = g.C;
    a.cs = g.cs;
    // in the multi-layer step the selection shares its SMs with the previous layer's attention kernel: a
    // shorter ring leaves room for both
    const int smax = pipe_select_max_stages(sh.dp);
    a.stages = chain ? (smax < 4 ? smax : 4) : smax;
    a.dev_status = dev_status;
    const size_t smem = pipe_select_smem(sh.dp, a.stages);
    dim3 grid((unsigned)g.C, (unsigned)(sh.B * sh.Hkv));
    cudaError_t e;
#define TB_PS_CASE(NVC, SLOT)                                                        \
    do {                                                                             \
        e = ensure_smem_attr(pipe_select_kernel<NVC>, pipe_select_smem(sh.dp, smax), SLOT); \
        if (e != cudaSuccess) return e;                                              \
        pipe_select_kernel<NVC><<<grid, kPipeThreads, smem, st>>>(a);                \
    } while (0)
    if (sh.dp == 16) TB_PS_CASE(2, 0);
    else if (sh.dp == 32) TB_PS_CASE(4, 1);
    else TB_PS_CASE(8, 2);
#undef TB_PS_CASE
    return cudaGetLastError();
}

cudaError_t launch_pipe_bracket(const tb_shape &sh, const PipeGeom &g, int32_t k, int64_t n, PipeRow *ctl,
                                const uint32_t *keys, int64_t keys_stride, uint2 *cand, int32_t *dev_status,
                                cudaStream_t st) {
    PipeBr a;
    a.ctl = ctl;
    a.keys = keys;
    a.cand = cand;
    a.keys_stride = keys_stride;
    a.n = n;
    a.k = k;
    a.C = g.C;
    a.cs = g.cs;
    a.dev_status = dev_status;
    const size_t smem = (size_t)kPipeHBins * 4 + (size_t)kPipeCandCap * 8;
    cudaError_t e = ensure_smem_attr(pipe_bracket_kernel, smem, 3);
    if (e != cudaSuccess) return e;
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t cfg = pdl_config(dim3((unsigned)g.C, (unsigned)(sh.B * sh.Hkv)), smem, st, attr);
    return cudaLaunchKernelEx(&cfg, pipe_bracket_kernel, a);
}

cudaError_t launch_pipe_attend(const tb_shape &sh, const PipeGeom &g, const tb_step_params &p, int64_t n, bool chain,
                               const uint16_t *q, const uint16_t *q_imp, const uint16_t *K_new, const uint16_t *V_new,
                               const uint16_t *Wk, uint16_t *K, uint16_t *V, uint16_t *Kp, int32_t *idx, int32_t *sel,
                               int32_t sel_stride, int32_t *counts, uint16_t *out, PipeRow *ctl, const uint32_t *keys,
                               int64_t keys_stride, float *part, int32_t *dev_status, cudaStream_t st) {
    PipeAttn a;
    a.q = q;
    a.q_imp = q_imp;
    a.K_new = K_new;
    a.V_new = V_new;
    a.Wk = Wk;
    a.K = K;
    a.V = V;
    a.Kp = Kp;
    a.idx = idx;
    a.sel = sel;
    a.counts = counts;
    a.out = out;
    a.ctl = ctl;
    a.keys = keys;
    a.keys_stride = keys_stride;
    a.part = part;
    a.cap = sh.cap;
    a.n = n;
    a.Hq = sh.Hq;
    a.Hkv = sh.Hkv;
    a.agg = p.agg;
    a.k = p.k;
    a.C = g.C;
    a.cs = g.cs;
    a.sel_stride = sel_stride;
    a.scale = p.scale;
    a.dev_status = dev_status;
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t cfg = pdl_config(dim3((unsigned)g.C, (unsigned)(sh.B * sh.Hkv)), 0, st, attr);
    cudaError_t e;
#define TB_PA_CASE(DTT, NVC, CH, SLOT)                                                            \
    do {                                                                                          \
        const size_t smem = (size_t)pipe_attn_smem_bytes(DTT, NVC * 8);                           \
        e = ensure_smem_attr(pipe_attend_kernel<DTT, NVC, CH>, smem, SLOT);                       \
        if (e != cudaSuccess) return e;                                                           \
        cfg.dynamicSmemBytes = smem;                                                              \
        return cudaLaunchKernelEx(&cfg, pipe_attend_kernel<DTT, NVC, CH>, a);                     \
    } while (0)
#define TB_PA_DP(DTT, CH, BASE)                            \
    do {                                                   \
        if (sh.dp == 16) TB_PA_CASE(DTT, 2, CH, BASE);     \
        if (sh.dp == 32) TB_PA_CASE(DTT, 4, CH, BASE + 1); \
        TB_PA_CASE(DTT, 8, CH, BASE + 2);                  \
    } while (0)
    if (sh.D == 64) {
        if (chain) TB_PA_DP(64, true, 4);
        TB_PA_DP(64, false, 7);
    }
    if (chain) TB_PA_DP(128, true, 10);
    TB_PA_DP(128, false, 13);
#undef TB_PA_DP
#undef TB_PA_CASE
}

}  // namespace tb
