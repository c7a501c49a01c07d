// Decoupled look-back over per-partition descriptors, used by the scans and
// radix sorts (gm_sort.cu).
//
// A descriptor is a 32-bit word: its top two bits say whether it holds the
// partition's own aggregate (F_AGG) or its inclusive prefix (F_PRE), the low
// 30 bits the value; 0 means not yet published.
#pragma once

#include <cuda/atomic>

#include "gm_internal.cuh"

namespace gm {

constexpr uint32_t F_AGG = 1u << 30;
constexpr uint32_t F_PRE = 2u << 30;
constexpr uint32_t V_MASK = (1u << 30) - 1;

__device__ __forceinline__ uint32_t ld_relaxed(uint32_t* p)
{
    cuda::atomic_ref<uint32_t, cuda::thread_scope_device> r(*p);
    return r.load(cuda::memory_order_relaxed);
}

__device__ __forceinline__ void st_relaxed(uint32_t* p, uint32_t v)
{
    cuda::atomic_ref<uint32_t, cuda::thread_scope_device> r(*p);
    r.store(v, cuda::memory_order_relaxed);
}

// Exclusive scan of one value per thread over a block of NT threads.
template <int NT>
__device__ __forceinline__ uint32_t block_excl_scan(uint32_t v, uint32_t* s_warp, uint32_t& total)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint32_t x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) s_warp[warp] = x;
    __syncthreads();
    if (warp == 0) {
        uint32_t y = lane < NT / 32 ? s_warp[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            uint32_t z = __shfl_up_sync(0xffffffffu, y, o);
            if (lane >= o) y += z;
        }
        if (lane < NT / 32) s_warp[lane] = y;
    }
    __syncthreads();
    uint32_t before = warp > 0 ? s_warp[warp - 1] : 0;
    total = s_warp[NT / 32 - 1];
    __syncthreads();
    return before + x - v;
}

// Walks back from partition p - 1 summing aggregates until an inclusive
// prefix is found.  Bounded: gives up after `limit` polls of one slot (and
// sets GM_FLAG_TIMEOUT in counters).  A block that gives up returns the sum
// of the aggregates it has seen, which is at most the true prefix, so every
// offset built from it stays below the true one (the callers' writes stay
// inside their buffers).
__device__ __forceinline__ uint32_t look_back(uint32_t* desc, int p, int stride, int32_t* counters, uint32_t limit)
{
    uint32_t excl = 0;
    int q = p - 1;
    uint32_t spins = 0;
    while (q >= 0) {
        uint32_t d = ld_relaxed(desc + (int64_t)q * stride);
        uint32_t flag = d & ~V_MASK;
        if (flag == 0) {
            if (++spins > limit) {
                atomicOr(counters + GM_CNT_FLAGS, GM_FLAG_TIMEOUT);
                break;
            }
            continue;
        }
        excl += d & V_MASK;
        if (flag == F_PRE) break;
        --q;
        spins = 0;
    }
    return excl;
}

}  // namespace gm
