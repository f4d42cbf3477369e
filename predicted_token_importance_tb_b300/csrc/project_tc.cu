// Batched key projection on the 5th-generation tensor cores ("TokenButler:
// Token Importance is Predictable", gist.science summary, Core Architecture:
// Key-Cache Projection; Optimizations: Batching).
//
//   Kp[b,h,pos0+r,:] = RNE_bf16( K_src[b,h,r,:] . Wk[h] )   (fp32 accumulation)
//
// Per (b, h) this is a [n_new x D] . [D x dp] GEMM: 2*D flops per 2*D bytes
// read, i.e. HBM-bound; the tensor cores are used so the arithmetic never
// becomes the limit. A persistent CTA per SM walks 128-row tiles:
//   warp 0  (one lane) TMA-loads the tile's K rows into a 4-stage ring
//           (128B-swizzled boxes of 64 columns x 128 rows);
//   warp 1  (one lane) issues tcgen05.mma (M=128, N=dp, K=16 per
//           instruction) from shared memory into one of two TMEM
//           accumulators and commits to mbarriers;
//   warps 2-5 read the accumulator back with tcgen05.ld (one output row per
//           thread), round to bf16 and store the row.
// Each CTA takes a contiguous range of tiles. Wk[h]^T of the KV heads that
// range uses sits in shared memory in the same swizzled K-major layout for
// the whole launch; warps 1-5 stage it while warp 0's first loads are in
// flight.
// Every wait is bounded; on a timeout the CTA records TB_ERR_TIMEOUT, waits
// (bounded) for its copies in flight, frees its TMEM and returns.
#include <cuda.h>
#include <string.h>

#include "kernels.cuh"
#include "tb_internal.cuh"

namespace tb {

constexpr int kTcM = 128;
constexpr int kTcStages = 4;
constexpr int kTcThreads = 192;
constexpr int kBoxCols = 64;                 // bf16 columns per 128-byte swizzle row
constexpr int kBoxBytes = kBoxCols * 2 * kTcM;   // 16 KB

// ------------------------------------------------------------------ PTX helpers

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait on an mbarrier phase; false (and *abort set) on timeout.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, volatile int *abort_flag,
                                          int32_t *dev_status) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (*abort_flag) return false;
        if (global_ns() - t0 > kWaitLimitNs) {
            *abort_flag = 1;
            set_status(dev_status, TB_ERR_TIMEOUT);
            return false;
        }
    }
    return true;
}

__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, int x, int y, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
        "[%4];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

// Shared-memory matrix descriptor: K-major operand, 128-byte swizzle, 8-row
// groups 1024 bytes apart.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFF);        // start address
    d |= (uint64_t)1 << 16;                        // leading byte offset (unused for this layout)
    d |= (uint64_t)(1024 >> 4) << 32;              // stride byte offset
    d |= (uint64_t)1 << 46;                        // descriptor version
    d |= (uint64_t)2 << 61;                        // 128-byte swizzle
    return d;
}

// Instruction descriptor of kind::f16: bf16 A and B (both K-major), fp32 D.
__host__ __device__ constexpr uint32_t mma_idesc(int M, int N) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void mma_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
        "%14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// ------------------------------------------------------------------ kernel

struct TcArgs {
    const uint16_t *Wk;
    uint16_t *Kp;
    int32_t *dev_status;
    int64_t cap, pos0, n_new, src_stride;
    int Hkv, D, dp, tiles_per_head, ntiles, tmem_cols;
};

__host__ __device__ inline size_t tc_smem_bytes(int Hkv, int D, int dp) {
    const int kh = D / kBoxCols;
    return 1024                                          // alignment slack
           + (size_t)kTcStages * kh * kBoxBytes          // A ring
           + (size_t)Hkv * kh * dp * 128                 // Wk^T of every KV head, swizzled
           + 256;                                        // barriers, TMEM address, flags
}

__global__ void __launch_bounds__(kTcThreads, 1)
project_tc_kernel(const __grid_constant__ CUtensorMap tmap, const TcArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int KH = a.D / kBoxCols;
    const size_t b_head_bytes = (size_t)KH * a.dp * 128;
    uint8_t *ringA = base;
    uint8_t *smB = ringA + (size_t)kTcStages * KH * kBoxBytes;
    uint8_t *ctl = smB + (size_t)a.Hkv * b_head_bytes;
    uint64_t *full = reinterpret_cast<uint64_t *>(ctl);
    uint64_t *empty = full + kTcStages;
    uint64_t *tfull = empty + kTcStages;
    uint64_t *tempty = tfull + 2;
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(tempty + 2);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_holder + 1);
    volatile int *consumed = abort_flag + 1;             // stages the MMA lane has consumed

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // this CTA's contiguous range of tiles
    const int tile_lo = (int)((int64_t)blockIdx.x * a.ntiles / gridDim.x);
    const int tile_hi = (int)((int64_t)(blockIdx.x + 1) * a.ntiles / gridDim.x);

    // Barriers and the TMEM accumulators first, so that the producer can
    // start streaming K before Wk is staged.
    if (threadIdx.x == 0) {
        for (int s = 0; s < kTcStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(&tfull[s], 1);
            mbar_init(&tempty[s], 128);
        }
        *abort_flag = 0;
        *consumed = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_holder)),
                     "r"(a.tmem_cols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    const uint32_t idesc = mma_idesc(kTcM, a.dp);

    if (warp != 0) {
        // Warps 1-5 stage Wk[h]^T of the KV heads this CTA's tiles use (a
        // contiguous tile range touches one or two heads, all Hkv only when it
        // spans that many), K-major with the 128-byte swizzle: element (j, d)
        // of head h lives in half kh = d / 64 at row j, byte 2*(d % 64) of
        // the row, whose 16-byte chunk index is XORed with (j % 8). 16-byte
        // loads of eight consecutive j, four in flight per thread.
        const int hd_lo = tile_lo / a.tiles_per_head;
        const int hd_hi = (tile_hi - 1) / a.tiles_per_head;
        const int nh = min(hd_hi - hd_lo + 1, a.Hkv);
        const int n8h = a.D * a.dp / 8;   // dp is a multiple of 8
        const int t = threadIdx.x - 32, nt = kTcThreads - 32;
#pragma unroll 4
        for (int x8 = t; x8 < nh * n8h; x8 += nt) {
            const int h = (hd_lo + x8 / n8h) % a.Hkv;
            const int x = 8 * (x8 % n8h);
            const uint4 u = __ldg(reinterpret_cast<const uint4 *>(a.Wk + (size_t)h * a.D * a.dp + x));
            const int d = x / a.dp, j0 = x % a.dp;
            const int kh = d / kBoxCols, byte = (d % kBoxCols) * 2;
            const uint32_t wv[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int j = j0 + i;
                const int chunk = (byte >> 4) ^ (j & 7);
                uint8_t *dst = smB + (size_t)h * b_head_bytes + (size_t)kh * a.dp * 128 + (size_t)j * 128 +
                               chunk * 16 + (byte & 15);
                *reinterpret_cast<uint16_t *>(dst) = (uint16_t)(i & 1 ? wv[i >> 1] >> 16 : wv[i >> 1] & 0xFFFFu);
            }
        }
        // the writes become visible to the tensor cores' (async) proxy, then
        // warps 1-5 meet before the first MMA reads them
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        asm volatile("bar.sync 1, %0;" ::"r"(kTcThreads - 32) : "memory");
    }

    if (warp == 0) {
        // ---------------- producer: TMA loads of the K tiles
        if (lane == 0) {
            int it = 0;
            for (int tile = tile_lo; tile < tile_hi && !*abort_flag; ++tile, ++it) {
                const int s = it % kTcStages;
                const uint32_t ph = (uint32_t)(it / kTcStages) & 1u;
                if (!mbar_wait(&empty[s], ph ^ 1u, abort_flag, a.dev_status)) break;
                const int head = tile / a.tiles_per_head;
                const int rt = tile % a.tiles_per_head;
                const int y = (int)((int64_t)head * a.src_stride + (int64_t)rt * kTcM);
                mbar_expect_tx(&full[s], (uint32_t)(KH * kBoxBytes));
                for (int kh = 0; kh < KH; ++kh)
                    tma_load_2d(ringA + ((size_t)s * KH + kh) * kBoxBytes, &tmap, kh * kBoxCols, y, &full[s]);
            }
            if (*abort_flag) {
                // let every load this lane issued land before the CTA leaves
                for (int j = *consumed; j < it; ++j) {
                    const int s = j % kTcStages;
                    const uint32_t ph = (uint32_t)(j / kTcStages) & 1u;
                    const uint64_t t0 = global_ns();
                    while (!mbar_try_wait(&full[s], ph) && global_ns() - t0 < kWaitLimitNs) {
                    }
                }
            }
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer
        if (lane == 0) {
            int it = 0;
            for (int tile = tile_lo; tile < tile_hi && !*abort_flag; ++tile, ++it) {
                const int s = it % kTcStages;
                const uint32_t ph = (uint32_t)(it / kTcStages) & 1u;
                const int acc = it & 1;
                const uint32_t aph = (uint32_t)(it >> 1) & 1u;
                const int h = (tile / a.tiles_per_head) % a.Hkv;
                if (!mbar_wait(&tempty[acc], aph ^ 1u, abort_flag, a.dev_status)) break;
                if (!mbar_wait(&full[s], ph, abort_flag, a.dev_status)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem + (uint32_t)(acc * a.dp);
                for (int kh = 0; kh < KH; ++kh) {
                    const uint32_t a0 = smem_u32(ringA + ((size_t)s * KH + kh) * kBoxBytes);
                    const uint32_t b0 = smem_u32(smB + (size_t)h * b_head_bytes + (size_t)kh * a.dp * 128);
#pragma unroll
                    for (int kk = 0; kk < kBoxCols / 16; ++kk)
                        mma_bf16(d_tmem, sw128_desc(a0 + kk * 32), sw128_desc(b0 + kk * 32), idesc,
                                 (kh | kk) != 0 ? 1u : 0u);
                }
                mma_commit(&empty[s]);
                mma_commit(&tfull[acc]);
                *consumed = it + 1;
            }
        }
    } else {
        // ---------------- epilogue: TMEM -> registers -> bf16 rows
        const int q = warp & 3;                 // TMEM lane quarter this warp may read
        const int r = q * 32 + lane;            // row of the tile
        int it = 0;
        for (int tile = tile_lo; tile < tile_hi; ++tile, ++it) {
            const int acc = it & 1;
            const uint32_t aph = (uint32_t)(it >> 1) & 1u;
            const int head = tile / a.tiles_per_head;
            const int rt = tile % a.tiles_per_head;
            if (!mbar_wait(&tfull[acc], aph, abort_flag, a.dev_status)) break;
            tc_fence_after();
            const int64_t row = (int64_t)rt * kTcM + r;
            uint16_t *dst = a.Kp + ((int64_t)head * a.cap + a.pos0 + row) * a.dp;
            const uint32_t taddr = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * a.dp);
            for (int c0 = 0; c0 < a.dp; c0 += 16) {
                float v[16];
                tmem_ld16(taddr + (uint32_t)c0, v);
                if (row < a.n_new) {
                    uint32_t w[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        w[i] = (uint32_t)f_to_bf16(v[2 * i]) | ((uint32_t)f_to_bf16(v[2 * i + 1]) << 16);
                    uint4 *o = reinterpret_cast<uint4 *>(dst + c0);
                    o[0] = make_uint4(w[0], w[1], w[2], w[3]);
                    o[1] = make_uint4(w[4], w[5], w[6], w[7]);
                }
            }
            tc_fence_before();
            mbar_arrive(&tempty[acc]);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(a.tmem_cols)
                     : "memory");
    }
}

// ------------------------------------------------------------------ host side

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
    // looked up once per process; the initialisation of a function-local
    // static is thread-safe
    static const EncodeTiledFn fn = [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            return reinterpret_cast<EncodeTiledFn>(p);
        return static_cast<EncodeTiledFn>(nullptr);
    }();
    return fn;
}

bool project_tc_supported(const tb_shape &sh, int64_t n_new) {
    if (n_new < kTcM) return false;                    // small batches: CUDA cores
    if (sh.D % kBoxCols != 0 || sh.D > 256) return false;
    if (sh.dp % 16 != 0 || sh.dp < 16 || sh.dp > 256) return false;
    if (!encode_fn()) return false;
    return tc_smem_bytes(sh.Hkv, sh.D, sh.dp) <= (size_t)dev_info().max_smem_optin;
}

cudaError_t launch_project_tc(const tb_shape &sh, const uint16_t *K_src, int64_t src_stride, const uint16_t *Wk,
                              uint16_t *Kp, int64_t pos0, int64_t n_new, int32_t *dev_status, cudaStream_t st) {
    const int heads = sh.B * sh.Hkv;
    CUtensorMap map;
    memset(&map, 0, sizeof map);
    const cuuint64_t rows = (cuuint64_t)(heads - 1) * (cuuint64_t)src_stride + (cuuint64_t)n_new;
    cuuint64_t gdim[2] = {(cuuint64_t)sh.D, rows};
    cuuint64_t gstride[1] = {(cuuint64_t)sh.D * 2};
    cuuint32_t box[2] = {(cuuint32_t)kBoxCols, (cuuint32_t)kTcM};
    cuuint32_t estride[2] = {1, 1};
    CUresult r = encode_fn()(&map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t *>(K_src), gdim, gstride,
                             box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    TcArgs a;
    a.Wk = Wk;
    a.Kp = Kp;
    a.dev_status = dev_status;
    a.cap = sh.cap;
    a.pos0 = pos0;
    a.n_new = n_new;
    a.src_stride = src_stride;
    a.Hkv = sh.Hkv;
    a.D = sh.D;
    a.dp = sh.dp;
    a.tiles_per_head = (int)((n_new + kTcM - 1) / kTcM);
    a.ntiles = a.tiles_per_head * heads;
    int cols = 32;
    while (cols < 2 * sh.dp) cols <<= 1;
    a.tmem_cols = cols;
    const size_t smem = tc_smem_bytes(sh.Hkv, sh.D, sh.dp);
    static thread_local int attr_dev = -1;   // per thread and device: the attribute lives in each context
    static thread_local size_t attr = 0;
    if (attr_dev != dev_info().device || attr < smem) {
        cudaError_t e = cudaFuncSetAttribute(project_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        attr_dev = dev_info().device;
        attr = smem;
    }
    int grid = dev_info().sms > 0 ? dev_info().sms : 148;
    if (grid > a.ntiles) grid = a.ntiles;
    project_tc_kernel<<<grid, kTcThreads, smem, st>>>(map, a);
    return cudaGetLastError();
}

}  // namespace tb
