// Distributed exact top-k (radix select) over one row held by a group of CTAs.
//
// Selection rule ("TokenButler: Token Importance is Predictable", arXiv
// abstract: individual tokens are kept, k of them per row): keep the k tokens of
// the row with the largest scores; ties go to the lower token index. Ordering
// is by the 64-bit composite (key << 32) | (~token), key the order-preserving
// image of the fp32 score, so every element has a distinct rank and the
// selection is exactly that of a full sort.
//
// A row of n scores is split into C consecutive chunks of L tokens, one per
// CTA. Each CTA holds its chunk's keys in shared memory. Radix passes over
// 11-bit digits build a global histogram per pass (one group barrier each)
// until the bin holding the k-th element is small enough to be resolved from
// a candidate list (one more barrier), which every CTA of the group then
// resolves redundantly in shared memory. No CTA waits for a second launch.
#pragma once

#include "tb_internal.cuh"
#include "ws_layout.cuh"

namespace tb {

// Shared-memory working set of one CTA of the group.
struct SelectSmem {
    uint32_t *keys;     // [L]   keys of this chunk
    uint32_t *hist;     // [kRadixBins]
    uint32_t *ckey;     // [kCandCap] candidate keys
    uint32_t *cidx;     // [kCandCap] candidate tokens
    uint32_t *ccount;   // [kMaxChunks] per-chunk count of selected candidates / prefix
    uint32_t *scan;     // [33]
    uint32_t *misc;     // [8]
    int *abort_flag;    // [1]
};

// Result of the threshold search, identical in every CTA of the group.
struct SelectResult {
    int mode;           // 0: take composite >= compT; 1: ties by index (TIE)
    uint64_t compT;     // mode 0 threshold
    uint32_t tkey;      // mode 1: the tied key
    uint32_t take;      // mode 1: tied elements this CTA keeps (lowest tokens first)
    uint32_t offset;    // first output slot of this CTA
    uint32_t count;     // outputs of this CTA
    bool ok;            // false when a wait timed out
};

__device__ __forceinline__ uint64_t composite(uint32_t key, uint32_t tok) {
    return ((uint64_t)key << 32) | (uint64_t)(0xFFFFFFFFu - tok);
}

// Find the bin b of `hist` (nbins <= kRadixBins, counts in smem) such that
// the elements in bins above b number fewer than `need` and those in bins >= b
// number at least `need`. Writes misc[0] = b, misc[1] = count above b,
// misc[2] = count in b. All threads must call it (barriers inside).
__device__ __forceinline__ void find_threshold_bin(const uint32_t *hist, uint32_t need, uint32_t *scan,
                                                   uint32_t *misc) {
    const int per = kRadixBins / blockDim.x;  // bins per thread, from the top
    const int hi = kRadixBins - 1 - threadIdx.x * per;
    uint32_t local = 0;
    for (int j = 0; j < per; ++j) local += hist[hi - j];
    uint32_t total;
    uint32_t above = block_exclusive_scan(local, scan, total);
    if (above < need && need <= above + local) {
        uint32_t a = above;
        for (int j = 0; j < per; ++j) {
            uint32_t c = hist[hi - j];
            if (need <= a + c) {
                misc[0] = (uint32_t)(hi - j);
                misc[1] = a;
                misc[2] = c;
                break;
            }
            a += c;
        }
    }
    __syncthreads();
}

// Radix select among `m` candidates in smem over the low `rbits` (<= 64)
// bits of their composites (the bits above are equal for all of them).
// Returns the composite threshold's low part: exactly `need` candidates have
// low part >= the result. All threads must call it.
__device__ __forceinline__ uint64_t local_select(const uint32_t *ckey, const uint32_t *cidx, uint32_t m,
                                                 uint32_t need, int shift, SelectSmem &S) {
    // low part of a candidate: ((key & (2^shift - 1)) << 32) | ~token  (shift + 32 bits)
    const uint32_t kmask = shift >= 32 ? 0xFFFFFFFFu : ((1u << shift) - 1u);
    int rem = shift + 32;
    uint64_t pre = 0;
    uint32_t need_l = need;
    while (rem > 0) {
        const int bits = rem >= kRadixBits ? kRadixBits : rem;
        rem -= bits;
        for (int b = threadIdx.x; b < kRadixBins; b += blockDim.x) S.hist[b] = 0;
        __syncthreads();
        const int upper = rem + bits;
        for (uint32_t e = threadIdx.x; e < m; e += blockDim.x) {
            uint64_t v = ((uint64_t)(ckey[e] & kmask) << 32) | (uint64_t)(0xFFFFFFFFu - cidx[e]);
            uint64_t top = upper >= 64 ? 0 : (v >> upper);
            if (top == pre) atomicAdd(&S.hist[(uint32_t)(v >> rem) & ((1u << bits) - 1u)], 1u);
        }
        __syncthreads();
        find_threshold_bin(S.hist, need_l, S.scan, S.misc);
        const uint32_t b = S.misc[0], above = S.misc[1], cnt = S.misc[2];
        need_l -= above;
        pre = (pre << bits) | b;
        __syncthreads();
        if (cnt == need_l) return pre << rem;   // the whole bin is kept
    }
    return pre;
}

// State carried from group_select_begin to group_select_end.
struct SelectBegin {
    uint32_t prefix;    // resolved top bits of the threshold bin
    int shift;          // bits below them
    uint32_t need;      // elements still needed from the bin
    uint32_t bincount;  // elements in the bin (whole row)
    int mode_all, mode_cand;
    int nbar;           // group barriers used so far (the last one only arrived)
    bool ok;
};

// First half of the group's threshold search: the global radix passes, then
// this chunk's counts and candidates are published and the CTA ARRIVES on
// the final barrier without waiting, so it can work on tokens that are kept
// whatever the exact threshold (those above the bin) in the meantime.
// Keys of this CTA's chunk are in S.keys[0..Lc). Chunk c of C covers tokens
// c*L .. c*L+Lc-1; budget k with 1 <= k <= n. bar_base: phases of ctl->bar
// the group has already completed in this launch.
__device__ __forceinline__ SelectBegin group_select_begin(RowCtl *ctl, SelectSmem &S, int Lc, int L, int c, int C,
                                                          uint32_t k, int32_t *dev_status, int bar_base = 0) {
    SelectBegin B;
    B.ok = true;
    uint32_t prefix = 0, need = k, bincount = 0;
    int shift = 32;
    int nbar = bar_base;
    for (int pass = 0; pass < 3; ++pass) {
        const int bits = pass < 2 ? kRadixBits : 32 - 2 * kRadixBits;
        const int upper = shift;   // bits above this pass's digit are fixed to `prefix`
        shift -= bits;
        for (int b = threadIdx.x; b < kRadixBins; b += blockDim.x) S.hist[b] = 0;
        __syncthreads();
        for (int e = threadIdx.x; e < Lc; e += blockDim.x) {
            uint32_t key = S.keys[e];
            bool match = (upper >= 32) || ((key >> upper) == prefix);
            if (match) atomicAdd(&S.hist[(key >> shift) & ((1u << bits) - 1u)], 1u);
        }
        __syncthreads();
        for (int b = threadIdx.x; b < kRadixBins; b += blockDim.x) {
            uint32_t v = S.hist[b];
            if (v) atomicAdd(&ctl->hist[pass][b], v);
        }
        ++nbar;
        if (!group_barrier(&ctl->bar, (uint32_t)(nbar * C), S.abort_flag, dev_status)) { B.ok = false; return B; }
        for (int b = threadIdx.x; b < kRadixBins; b += blockDim.x) S.hist[b] = __ldcg(&ctl->hist[pass][b]);
        __syncthreads();
        find_threshold_bin(S.hist, need, S.scan, S.misc);
        const uint32_t b = S.misc[0], above = S.misc[1];
        bincount = S.misc[2];
        need -= above;
        prefix = (prefix << bits) | b;
        __syncthreads();
        if (bincount <= (uint32_t)kCandCap || bincount == need) break;
    }
    // classify this chunk against the threshold bin, publish counts
    const int mode_all = (bincount == need);
    const int mode_cand = !mode_all && bincount <= (uint32_t)kCandCap;
    uint32_t my_above = 0, my_eq = 0;
    for (int e = threadIdx.x; e < Lc; e += blockDim.x) {
        uint32_t top = S.keys[e] >> shift;   // shift < 32 here
        if (top > prefix) ++my_above;
        else if (top == prefix) ++my_eq;
    }
    // one scan of both counts: above in the high half, equal in the low half (a chunk holds < 2^16 keys)
    uint32_t tot;
    const uint32_t before = block_exclusive_scan((my_above << 16) | my_eq, S.scan, tot);
    const uint32_t chunk_above = tot >> 16, chunk_eq = tot & 0xFFFFu;
    const uint32_t eq_before = before & 0xFFFFu;
    if (mode_cand) {   // the chunk's candidates, at slots reserved with one atomic per CTA
        if (threadIdx.x == 0) S.misc[7] = atomicAdd(&ctl->ncand, chunk_eq);
        __syncthreads();
        uint32_t slot = S.misc[7] + eq_before;
        for (int e = threadIdx.x; e < Lc; e += blockDim.x) {
            if ((S.keys[e] >> shift) == prefix) {
                if (slot < (uint32_t)kCandCap) ctl->cand[slot] = make_uint2(S.keys[e], (uint32_t)(c * L + e));
                ++slot;
            }
        }
    }
    if (threadIdx.x == 0) {
        ctl->above[c] = chunk_above;
        ctl->eq[c] = chunk_eq;
    }
    ++nbar;
    group_arrive(&ctl->bar);
    B.prefix = prefix;
    B.shift = shift;
    B.need = need;
    B.bincount = bincount;
    B.mode_all = mode_all;
    B.mode_cand = mode_cand;
    B.nbar = nbar;
    return B;
}

// Is this key above the threshold bin (kept whatever the exact threshold)?
__device__ __forceinline__ bool above_bin(const SelectBegin &B, uint32_t key) { return (key >> B.shift) > B.prefix; }

// Second half: wait for every chunk's counts, resolve the exact threshold
// and this CTA's output slots (identically in every CTA of the group).
__device__ __forceinline__ SelectResult group_select_end(RowCtl *ctl, SelectSmem &S, const SelectBegin &B, int L,
                                                         int c, int C, int32_t *dev_status) {
    SelectResult R;
    R.ok = true;
    if (!group_wait(&ctl->bar, (uint32_t)(B.nbar * C), S.abort_flag, dev_status)) { R.ok = false; return R; }
    const uint32_t prefix = B.prefix, need = B.need;
    const int shift = B.shift;
    if (B.mode_cand) {
        const uint32_t m = B.bincount;
        for (uint32_t e = threadIdx.x; e < m; e += blockDim.x) {
            uint2 v = __ldcg(&ctl->cand[e]);
            S.ckey[e] = v.x;
            S.cidx[e] = v.y;
        }
        for (int j = threadIdx.x; j < C; j += blockDim.x) S.ccount[j] = 0;
        __syncthreads();
        const uint64_t low = local_select(S.ckey, S.cidx, m, need, shift, S);
        const uint64_t hi_part = (uint64_t)(prefix << shift) << 32;   // shift <= 21 here
        R.compT = hi_part + low;
        for (uint32_t e = threadIdx.x; e < m; e += blockDim.x)
            if (composite(S.ckey[e], S.cidx[e]) >= R.compT) atomicAdd(&S.ccount[S.cidx[e] / (uint32_t)L], 1u);
        __syncthreads();
        for (int j = threadIdx.x; j < C; j += blockDim.x) S.ccount[j] += __ldcg(&ctl->above[j]);
        R.mode = 0;
    } else if (B.mode_all) {
        R.compT = (uint64_t)(prefix << shift) << 32;
        for (int j = threadIdx.x; j < C; j += blockDim.x) S.ccount[j] = __ldcg(&ctl->above[j]) + __ldcg(&ctl->eq[j]);
        R.mode = 0;
    } else {
        // all 32 key bits resolved (shift == 0) and more tied elements than
        // the budget has room for: keep the lowest tokens, chunk by chunk
        R.mode = 1;
        R.tkey = prefix;
        if (threadIdx.x == 0) {
            uint32_t left = need;
            for (int j = 0; j < C; ++j) {
                uint32_t e = __ldcg(&ctl->eq[j]);
                uint32_t t = e < left ? e : left;
                left -= t;
                S.ccount[j] = __ldcg(&ctl->above[j]) + t;
                if (j == c) S.misc[3] = t;
            }
        }
    }
    __syncthreads();
    if (R.mode == 1) R.take = S.misc[3];
    // exclusive prefix over chunks -> this CTA's output offset
    if (threadIdx.x == 0) {
        uint32_t off = 0;
        for (int j = 0; j < c; ++j) off += S.ccount[j];
        S.misc[4] = off;
        S.misc[5] = S.ccount[c];
    }
    __syncthreads();
    R.offset = S.misc[4];
    R.count = S.misc[5];
    __syncthreads();
    return R;
}

// The whole threshold search (both halves back to back).
__device__ __forceinline__ SelectResult group_select(RowCtl *ctl, SelectSmem &S, int Lc, int L, int c, int C,
                                                     uint32_t k, int32_t *dev_status, int bar_base = 0) {
    SelectBegin B = group_select_begin(ctl, S, Lc, L, c, C, k, dev_status, bar_base);
    if (!B.ok) {
        SelectResult R;
        R.ok = false;
        return R;
    }
    return group_select_end(ctl, S, B, L, c, C, dev_status);
}

// Is element e (key, token) of this chunk kept? For mode 1 the caller passes
// the number of tied elements before it in the chunk.
__device__ __forceinline__ bool is_kept(const SelectResult &R, uint32_t key, uint32_t tok, uint32_t tied_before) {
    if (R.mode == 0) return composite(key, tok) >= R.compT;
    if (key > R.tkey) return true;
    return key == R.tkey && tied_before < R.take;
}

// Write the kept tokens of this chunk, ascending, to out[R.offset ...] (and
// to out2 when given). The chunk's keys are in S.keys; token of element e is
// tok0 + e; S.keys is overwritten. Warp w takes a contiguous run of the
// chunk in stripes of 32 and finds its kept elements with ballots (in mode 1
// the tied elements are counted first, since ties go to the lowest tokens);
// one block scan over the warps' counts gives each warp its first output slot.
__device__ __forceinline__ void write_kept(const SelectResult &R, SelectSmem &S, int Lc, uint32_t tok0,
                                          int32_t *out, int32_t *out2 = nullptr) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    const int per = ((Lc + nw - 1) / nw + 31) & ~31;
    const int e0 = warp * per, e1 = e0 + per < Lc ? e0 + per : Lc;
    const uint32_t lt = (1u << lane) - 1u;
    uint32_t tot;
    uint32_t tied_base = 0;
    if (R.mode == 1) {   // tied elements in the warps before this one
        uint32_t nt = 0;
        for (int b = e0; b < e1; b += 32) {
            const int e = b + lane;
            nt += __popc(__ballot_sync(0xFFFFFFFFu, e < e1 && S.keys[e] == R.tkey));
        }
        tied_base = block_exclusive_scan(lane == 0 ? nt : 0u, S.scan, tot);
        tied_base = __shfl_sync(0xFFFFFFFFu, tied_base, 0);
    }
    // kept(e): the element's ballot of the stripe, advancing the tie rank in mode 1
    auto stripe = [&](int b, uint32_t &run) -> uint32_t {
        const int e = b + lane;
        const bool in = e < e1;
        const uint32_t key = in ? S.keys[e] : 0u;
        bool kp;
        if (R.mode == 0) {
            kp = in && composite(key, tok0 + (uint32_t)e) >= R.compT;
        } else {
            const uint32_t tb = __ballot_sync(0xFFFFFFFFu, in && key == R.tkey);
            kp = in && (key > R.tkey || (key == R.tkey && run + __popc(tb & lt) < R.take));
            run += __popc(tb);
        }
        return __ballot_sync(0xFFFFFFFFu, kp);
    };
    if (R.mode == 0) {
        // one pass: each warp compacts its kept tokens in place over its own run of S.keys (a kept token is
        // written at or before the position it was read from); one block scan places the runs
        uint32_t nk = 0;
        for (int b = e0; b < e1; b += 32) {
            const int e = b + lane;
            const bool kp = e < e1 && composite(S.keys[e], tok0 + (uint32_t)e) >= R.compT;
            const uint32_t kb = __ballot_sync(0xFFFFFFFFu, kp);
            __syncwarp();   // the whole stripe is read before any lane writes into it
            if (kp) S.keys[e0 + nk + __popc(kb & lt)] = tok0 + (uint32_t)e;
            nk += __popc(kb);
        }
        uint32_t wpos = block_exclusive_scan(lane == 0 ? nk : 0u, S.scan, tot);
        wpos = R.offset + __shfl_sync(0xFFFFFFFFu, wpos, 0);
        for (uint32_t i = lane; i < nk; i += 32) {
            out[wpos + i] = (int32_t)S.keys[e0 + i];
            if (out2) out2[wpos + i] = (int32_t)S.keys[e0 + i];
        }
        return;
    }
    uint32_t nk = 0, run = tied_base;
    for (int b = e0; b < e1; b += 32) nk += __popc(stripe(b, run));
    uint32_t pos = block_exclusive_scan(lane == 0 ? nk : 0u, S.scan, tot);
    pos = R.offset + __shfl_sync(0xFFFFFFFFu, pos, 0);
    run = tied_base;
    for (int b = e0; b < e1; b += 32) {
        const uint32_t kb = stripe(b, run);
        if ((kb >> lane) & 1u) {
            const uint32_t at = pos + __popc(kb & lt);
            out[at] = (int32_t)(tok0 + (uint32_t)(b + lane));
            if (out2) out2[at] = (int32_t)(tok0 + (uint32_t)(b + lane));
        }
        pos += __popc(kb);
    }
}

// Last CTA of the group to arrive puts the row's control block back to zero.
__device__ __forceinline__ void group_release(RowCtl *ctl, int C, SelectSmem &S) {
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        uint32_t prev = atomicAdd(&ctl->done, 1u);
        S.misc[6] = (prev == (uint32_t)(C - 1)) ? 1u : 0u;
    }
    __syncthreads();
    if (S.misc[6]) {
        __threadfence();
        for (int b = threadIdx.x; b < 3 * kRadixBins; b += blockDim.x) (&ctl->hist[0][0])[b] = 0;
        if (threadIdx.x == 0) {
            ctl->bar = 0;
            ctl->ncand = 0;
            ctl->done = 0;
        }
    }
}

}  // namespace tb
