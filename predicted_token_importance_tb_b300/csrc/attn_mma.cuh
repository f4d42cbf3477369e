// Attention over K/V rows staged in shared memory, on the tensor cores
// ("TokenButler: Token Importance is Predictable": exact attention over only
// the selected full-precision rows).
//
// Slot s of the staging area holds a K row at X + s*SB and its V row at
// X + s*SB + 2*D (bf16), SB = 4*D + 16 (the 16-byte skew spreads eight
// consecutive rows over all banks for ldmatrix). A warp takes chunks of 16
// slots: S = Q K^T with m16n8k16 bf16 MMAs (the G query heads are the rows
// of a 16-row tile, zero-padded; fp32 accumulation), an online softmax in the
// exp2 domain (fp32), and O += P V with P rounded to bf16. Slots whose flag
// is zero (or, with FLAGS = false, slots >= n) are masked; their V rows must
// hold finite values (zeros).
#pragma once

#include "async_copy.cuh"
#include "attn_core.cuh"

namespace tb {

// Shared bytes of one staged K/V row pair.
__host__ __device__ inline int mma_slot_bytes(int D) { return 4 * D + 16; }

// 16 zero bytes to shared memory where cond holds (a predicated store, no branch).
__device__ __forceinline__ void st_shared_zero16_if(void *p, bool cond) {
    asm volatile("{\n\t.reg .pred q;\n\tsetp.ne.u32 q, %1, 0;\n\t@q st.shared.v4.u32 [%0], {%2, %2, %2, %2};\n\t}" ::"r"(
                     smem_addr(p)),
                 "r"((uint32_t)cond), "r"(0u)
                 : "memory");
}

// Per-warp attention state on the tensor cores: rows g = lane/4 and g + 8 of
// the 16-row tiles (query heads; rows >= G are zero padding), O over NT
// n-tiles of 8 dims.
template <int NT>
struct MmaAttn {
    float m0, m1, l0, l1;
    float o[NT][4];
};

// Attend slots [0, n) of the gathered rows (K row at X + s*SB, V row at
// +2D) for the slots whose kept flag (kept[kept_off + s]) is set, or for all
// of them with FLAGS = false (kept unused); chunks of 16 slots per warp.
template <int DT, int NW, bool FLAGS = true>
__device__ __forceinline__ void mma_attend(MmaAttn<DT / 8> &A, const uint8_t *X, int SB, int n, const uint8_t *kept,
                                           int kept_off, const uint8_t *qsm, float qscale) {
    constexpr int NT = DT / 8, KS = DT / 16, QS = 2 * DT + 16;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint32_t xs = smem_addr(X), qa = smem_addr(qsm);
    const int nch = (n + 15) >> 4;
    for (int ch = warp; ch < nch; ch += NW) {
        const int s0 = ch * 16;
        // S = Q K^T for slots s0 .. s0+15 (two n-tiles of 8)
        // kept flags of this lane's columns s0 + 8j + 2(lane%4) + {0,1}
        // (the flags are zero past the gathered rows)
        uint32_t f0, f1;
        if (FLAGS) {
            f0 = *reinterpret_cast<const uint16_t *>(kept + kept_off + s0 + 2 * (lane & 3));
            f1 = *reinterpret_cast<const uint16_t *>(kept + kept_off + s0 + 8 + 2 * (lane & 3));
        } else {   // the same byte pattern from the count
            const int c0 = s0 + 2 * (lane & 3);
            f0 = (c0 < n ? 0x01u : 0u) | (c0 + 1 < n ? 0x100u : 0u);
            f1 = (c0 + 8 < n ? 0x01u : 0u) | (c0 + 9 < n ? 0x100u : 0u);
        }
        // S = Q K^T, two independent accumulator chains per n-tile (even / odd k-steps)
        float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
        float sd[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
        const int kt = s0 + 8 * (lane >> 4) + (lane & 7);        // K row this lane addresses
        const uint32_t krow = xs + (uint32_t)kt * SB + 16 * ((lane >> 3) & 1);
        const uint32_t qrow = qa + (uint32_t)((lane & 7) + 8 * ((lane >> 3) & 1)) * QS + 16 * (lane >> 4);
#pragma unroll
        for (int kk = 0; kk < KS; kk += 2) {
            uint32_t a0, a1, a2, a3, b0, b1, b2, b3;
            uint32_t e0, e1, e2, e3, g0, g1, g2, g3;
            ldsm_x4(qrow + kk * 32, a0, a1, a2, a3);
            ldsm_x4(krow + kk * 32, b0, b1, b2, b3);
            ldsm_x4(qrow + kk * 32 + 32, e0, e1, e2, e3);
            ldsm_x4(krow + kk * 32 + 32, g0, g1, g2, g3);
            mma_bf16_16816(sc[0], a0, a1, a2, a3, b0, b1);
            mma_bf16_16816(sc[1], a0, a1, a2, a3, b2, b3);
            mma_bf16_16816(sd[0], e0, e1, e2, e3, g0, g1);
            mma_bf16_16816(sd[1], e0, e1, e2, e3, g2, g3);
        }
        // online softmax (exp2 domain); columns of this lane: s0 + 8j + 2(lane%4) + {0,1}
        float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
        for (int j = 0; j < 2; ++j) {
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const bool on = (((j ? f1 : f0) >> (8 * u)) & 0xFFu) != 0u;
                const float z0 = (sc[j][u] + sd[j][u]) * qscale, z1 = (sc[j][2 + u] + sd[j][2 + u]) * qscale;
                sc[j][u] = on ? z0 : -INFINITY;
                sc[j][2 + u] = on ? z1 : -INFINITY;
                mx0 = fmaxf(mx0, sc[j][u]);
                mx1 = fmaxf(mx1, sc[j][2 + u]);
            }
        }
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xFFFFFFFFu, mx0, 1));
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xFFFFFFFFu, mx0, 2));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xFFFFFFFFu, mx1, 1));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xFFFFFFFFu, mx1, 2));
        const float n0 = fmaxf(A.m0, mx0), n1 = fmaxf(A.m1, mx1);
        const float c0 = n0 == -INFINITY ? 1.f : exp2f(A.m0 - n0);
        const float c1 = n1 == -INFINITY ? 1.f : exp2f(A.m1 - n1);
        float p[2][4];
#pragma unroll
        for (int j = 0; j < 2; ++j) {
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                p[j][u] = n0 == -INFINITY ? 0.f : exp2f(sc[j][u] - n0);
                p[j][2 + u] = n1 == -INFINITY ? 0.f : exp2f(sc[j][2 + u] - n1);
            }
        }
        A.l0 = A.l0 * c0 + (p[0][0] + p[0][1] + p[1][0] + p[1][1]);
        A.l1 = A.l1 * c1 + (p[0][2] + p[0][3] + p[1][2] + p[1][3]);
        A.m0 = n0;
        A.m1 = n1;
#pragma unroll
        for (int t = 0; t < NT; ++t) {
            A.o[t][0] *= c0;
            A.o[t][1] *= c0;
            A.o[t][2] *= c1;
            A.o[t][3] *= c1;
        }
        // O += P V: A operand from p (row, 16 slots), B from V rows (transposed loads)
        const uint32_t pa0 = pack_bf16x2(p[0][0], p[0][1]), pa1 = pack_bf16x2(p[0][2], p[0][3]);
        const uint32_t pa2 = pack_bf16x2(p[1][0], p[1][1]), pa3 = pack_bf16x2(p[1][2], p[1][3]);
        const int vt = s0 + 8 * ((lane >> 3) & 1) + (lane & 7);   // V row this lane addresses
        const uint32_t vrow = xs + (uint32_t)vt * SB + 2 * DT + 16 * (lane >> 4);
#pragma unroll
        for (int jp = 0; jp < NT / 2; ++jp) {
            uint32_t b0, b1, b2, b3;
            ldsm_x4_trans(vrow + jp * 32, b0, b1, b2, b3);
            mma_bf16_16816(A.o[2 * jp], pa0, pa1, pa2, pa3, b0, b1);
            mma_bf16_16816(A.o[2 * jp + 1], pa0, pa1, pa2, pa3, b2, b3);
        }
    }
}

}  // namespace tb
