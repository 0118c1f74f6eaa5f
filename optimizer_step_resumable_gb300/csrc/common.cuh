// common.cuh -- small device and launch helpers shared by the kernel files.
#pragma once

#include <cstdint>

#include <cuda_bf16.h>
#include <cuda_fp16.h>
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

// ---------------------------------------------------------------------------
// Gradient and weight-copy element types: float, bfloat16 (the top half of
// a binary32) and IEEE binary16.  Widening to float is exact; narrowing
// rounds to nearest, ties to even (CUDA's _rn conversions).
// ---------------------------------------------------------------------------
template <typename G>
__device__ __forceinline__ float4 load4_cs(const G* p);  // 4 elements, streaming

template <>
__device__ __forceinline__ float4 load4_cs<float>(const float* p)
{
    return __ldcs(reinterpret_cast<const float4*>(p));
}

template <>
__device__ __forceinline__ float4 load4_cs<__nv_bfloat16>(const __nv_bfloat16* p)
{
    const uint2 r = __ldcs(reinterpret_cast<const uint2*>(p));
    return make_float4(__uint_as_float(r.x << 16), __uint_as_float(r.x & 0xffff0000u),
                       __uint_as_float(r.y << 16), __uint_as_float(r.y & 0xffff0000u));
}

template <>
__device__ __forceinline__ float4 load4_cs<__half>(const __half* p)
{
    const uint2 r = __ldcs(reinterpret_cast<const uint2*>(p));
    return make_float4(__half2float(__ushort_as_half(static_cast<unsigned short>(r.x & 0xffffu))),
                       __half2float(__ushort_as_half(static_cast<unsigned short>(r.x >> 16))),
                       __half2float(__ushort_as_half(static_cast<unsigned short>(r.y & 0xffffu))),
                       __half2float(__ushort_as_half(static_cast<unsigned short>(r.y >> 16))));
}

// 4 elements with the default L2 caching (ld.global.cg): for data that a
// following kernel reads again (the norm's read of g, which the fused kernel
// reads next), so that it may still find it in L2
template <typename G>
__device__ __forceinline__ float4 load4_cg(const G* p);

template <>
__device__ __forceinline__ float4 load4_cg<float>(const float* p)
{
    return __ldcg(reinterpret_cast<const float4*>(p));
}

template <>
__device__ __forceinline__ float4 load4_cg<__nv_bfloat16>(const __nv_bfloat16* p)
{
    const uint2 r = __ldcg(reinterpret_cast<const uint2*>(p));
    return make_float4(__uint_as_float(r.x << 16), __uint_as_float(r.x & 0xffff0000u),
                       __uint_as_float(r.y << 16), __uint_as_float(r.y & 0xffff0000u));
}

template <>
__device__ __forceinline__ float4 load4_cg<__half>(const __half* p)
{
    const uint2 r = __ldcg(reinterpret_cast<const uint2*>(p));
    return make_float4(__half2float(__ushort_as_half(static_cast<unsigned short>(r.x & 0xffffu))),
                       __half2float(__ushort_as_half(static_cast<unsigned short>(r.x >> 16))),
                       __half2float(__ushort_as_half(static_cast<unsigned short>(r.y & 0xffffu))),
                       __half2float(__ushort_as_half(static_cast<unsigned short>(r.y >> 16))));
}

__device__ __forceinline__ float load1(const float* p) { return *p; }
__device__ __forceinline__ float load1(const __nv_bfloat16* p) { return __bfloat162float(*p); }
__device__ __forceinline__ float load1(const __half* p) { return __half2float(*p); }

// four zeros over 4 elements of g (the fused zero_grads)
__device__ __forceinline__ void store4_zero_cs(float* p)
{
    __stcs(reinterpret_cast<float4*>(p), make_float4(0.f, 0.f, 0.f, 0.f));
}
__device__ __forceinline__ void store4_zero_cs(__nv_bfloat16* p)
{
    __stcs(reinterpret_cast<uint2*>(p), make_uint2(0u, 0u));
}
__device__ __forceinline__ void store4_zero_cs(__half* p)
{
    __stcs(reinterpret_cast<uint2*>(p), make_uint2(0u, 0u));
}
__device__ __forceinline__ void store1_zero(float* p) { *p = 0.0f; }
__device__ __forceinline__ void store1_zero(__nv_bfloat16* p) { *p = __float2bfloat16_rn(0.0f); }
__device__ __forceinline__ void store1_zero(__half* p) { *p = __float2half_rn(0.0f); }

// 16-bit copy of 4 new weights (round to nearest even)
__device__ __forceinline__ unsigned bits16(__nv_bfloat16 h) { return __bfloat16_as_ushort(h); }
__device__ __forceinline__ unsigned bits16(__half h) { return __half_as_ushort(h); }
__device__ __forceinline__ __nv_bfloat16 narrow(float x, __nv_bfloat16*) { return __float2bfloat16_rn(x); }
__device__ __forceinline__ __half narrow(float x, __half*) { return __float2half_rn(x); }

template <typename WL>
__device__ __forceinline__ void store4_lp_cs(WL* p, float4 w)
{
    const unsigned a = bits16(narrow(w.x, p)), b = bits16(narrow(w.y, p));
    const unsigned c = bits16(narrow(w.z, p)), d = bits16(narrow(w.w, p));
    __stcs(reinterpret_cast<uint2*>(p), make_uint2(a | (b << 16), c | (d << 16)));
}
template <typename WL>
__device__ __forceinline__ void store1_lp(WL* p, float w)
{
    *p = narrow(w, p);
}

inline bool aligned16(const void* p)
{
    return (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
}

inline bool aligned8(const void* p)
{
    return (reinterpret_cast<uintptr_t>(p) & 7u) == 0;
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
