// common.cuh -- small device and launch helpers shared by the kernel files.
#pragma once

#include <cstdint>

#include <cuda_runtime.h>

#include "internal.h"

namespace osr {
namespace detail {

// ---------------------------------------------------------------------------
// Block-wide double sum with a fixed shuffle pattern: the same inputs in the
// same threads always give the same bits.  Result valid in thread 0.
// ---------------------------------------------------------------------------
template <int kThreads>
__device__ __forceinline__ double block_sum(double x)
{
    __shared__ double warp_sums[kThreads / 32];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
        x += __shfl_down_sync(0xffffffffu, x, off);
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    __syncthreads();  // warp_sums may still be read by a previous call
    if (lane == 0)
        warp_sums[warp] = x;
    __syncthreads();
    if (warp == 0) {
        x = lane < kThreads / 32 ? warp_sums[lane] : 0.0;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1)
            x += __shfl_down_sync(0xffffffffu, x, off);
    }
    return x;
}

inline bool aligned16(const void* p)
{
    return (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
}

inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Resident blocks of `kernel` on the whole device; *err receives the
// occupancy query's own status (not the runtime's last error).
inline int resident_blocks(const void* kernel, int threads, int sm_count, cudaError_t* err)
{
    int per_sm = 0;
    const cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads, 0);
    if (e != cudaSuccess && *err == cudaSuccess)
        *err = e;
    if (e != cudaSuccess || per_sm < 1)
        per_sm = 1;
    return per_sm * sm_count;
}

}  // namespace detail
}  // namespace osr
