// Internal helpers shared by the kernels of libtb (sm_103a only).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "tb.h"

namespace tb {

// ------------------------------------------------------------------ status

__device__ __forceinline__ void set_status(int32_t *dev_status, int32_t code) {
    if (dev_status) atomicCAS(dev_status, 0, code);
}

// ------------------------------------------------------------------ bf16

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
__device__ __forceinline__ float bf16_to_f(uint16_t h) { return __uint_as_float(((uint32_t)h) << 16); }

// fp32 -> bf16 bits, round to nearest even (the hardware conversion).
__device__ __forceinline__ uint16_t f_to_bf16(float f) {
    return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}

// ------------------------------------------------------------------ keys

// Order-preserving map fp32 -> uint32: a > b  <=>  key(a) > key(b).
// -0.0 is folded onto +0.0 first so the two tie; a NaN maps to 0 (lowest)
// and raises the flag.
__device__ __forceinline__ uint32_t score_key(float f, bool &nan_seen) {
    uint32_t u = __float_as_uint(f);
    if ((u & 0x7FFFFFFFu) > 0x7F800000u) { nan_seen = true; return 0u; }
    if (u == 0x80000000u) u = 0u;
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// ------------------------------------------------------------------ sync

__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ uint32_t ld_acquire(const uint32_t *p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Longest a device-side wait may spin before it gives up (nanoseconds).
constexpr uint64_t kWaitLimitNs = 2000000000ull;

// Split-phase group barrier on a counter shared by a group of CTAs: every CTA
// arrives once per phase; a CTA waits until the counter reaches `target`
// (phase count x group size). The wait is bounded: after kWaitLimitNs it
// gives up, sets *abort_flag (shared) and records TB_ERR_TIMEOUT.
// Arrival: the CTA's barrier orders its threads' writes before thread 0's
// release add, which makes them visible at GPU scope before the count moves.
__device__ __forceinline__ void group_arrive(uint32_t *ctr) {
    __syncthreads();
    if (threadIdx.x == 0) asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(ctr) : "memory");
}

// Wait: thread 0 polls with acquire loads, then the CTA barrier passes the
// acquired view on to every thread of the CTA.
__device__ __forceinline__ bool group_wait(uint32_t *ctr, uint32_t target, int *abort_flag, int32_t *dev_status,
                                           uint64_t limit_ns = kWaitLimitNs) {
    if (threadIdx.x == 0) {
        if (ld_acquire(ctr) < target) {
            const uint64_t t0 = global_ns();
            while (ld_acquire(ctr) < target) {
                if (global_ns() - t0 > limit_ns) {
                    *abort_flag = 1;
                    set_status(dev_status, TB_ERR_TIMEOUT);
                    break;
                }
            }
        }
    }
    __syncthreads();   // (thread 0's acquire orders the CTA's later reads)
    return *abort_flag == 0;
}

__device__ __forceinline__ bool group_barrier(uint32_t *ctr, uint32_t target, int *abort_flag,
                                              int32_t *dev_status, uint64_t limit_ns = kWaitLimitNs) {
    group_arrive(ctr);
    return group_wait(ctr, target, abort_flag, dev_status, limit_ns);
}

// ------------------------------------------------------------------ scans

// Exclusive prefix sum of one uint32 per thread over the block, plus the total.
// `scratch` needs (blockDim.x/32 + 1) words of shared memory. Contains
// __syncthreads(); every thread of the block must call it.
__device__ __forceinline__ uint32_t block_exclusive_scan(uint32_t v, uint32_t *scratch, uint32_t &total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    uint32_t x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        uint32_t y = __shfl_up_sync(0xFFFFFFFFu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) scratch[warp] = x;
    __syncthreads();
    if (warp == 0) {
        uint32_t w = lane < nw ? scratch[lane] : 0u;
        uint32_t wx = w;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            uint32_t y = __shfl_up_sync(0xFFFFFFFFu, wx, o);
            if (lane >= o) wx += y;
        }
        if (lane < nw) scratch[lane] = wx - w;
        if (lane == 31) scratch[32] = wx;
    }
    __syncthreads();
    uint32_t r = scratch[warp] + x - v;
    total = scratch[32];
    __syncthreads();
    return r;
}

// ------------------------------------------------------------------ host side

struct DevInfo {
    int device = -1;
    int sms = 0;
    int l2_bytes = 0;
    int max_smem_optin = 0;
};
const DevInfo &dev_info();

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace tb
