// pack.cu -- the checkpoint pack (row a5): the step_NNNNNN.bin image
// [int32 step][int32 n][n f32 w][n f32 m][n f32 v] written into a device
// staging buffer, for sm_103a.
//
// "Grow a Language Model: Checkpoints" (unhomeschool.com), sections "Format"
// and "Total size": five contiguous regions, 8 + 12 n bytes, no other
// metadata.  HBM-bound: 24 bytes per parameter (read w, m, v; write image).
#include <cstdint>

#include <cuda_runtime.h>

#include "common.cuh"
#include "internal.h"

namespace osr {
namespace {

// ---------------------------------------------------------------------------
// Checkpoint pack: [int32 step][int32 n][w][m][v] into the staging image.
// image is 8-byte aligned and image + 8 is 16-byte aligned; with n % 4 == 0
// the three regions are 16-byte aligned and copied as float4.
// ---------------------------------------------------------------------------
constexpr int kPackThreads = 256;
constexpr int kPackVec = 4;

__device__ __forceinline__ void copy_f4(float4* __restrict__ dst,
                                        const float4* __restrict__ src, int64_t n4)
{
    constexpr int64_t chunk = int64_t(kPackThreads) * kPackVec;
    const int64_t nchunks = n4 / chunk;
    for (int64_t c = blockIdx.x; c < nchunks; c += gridDim.x) {
        const int64_t i0 = c * chunk + threadIdx.x;
        float4 r[kPackVec];
#pragma unroll
        for (int j = 0; j < kPackVec; ++j)
            r[j] = __ldcs(src + i0 + j * kPackThreads);
#pragma unroll
        for (int j = 0; j < kPackVec; ++j)
            __stcs(dst + i0 + j * kPackThreads, r[j]);
    }
    const int64_t gtid = int64_t(blockIdx.x) * kPackThreads + threadIdx.x;
    for (int64_t i = nchunks * chunk + gtid; i < n4; i += int64_t(gridDim.x) * kPackThreads)
        __stcs(dst + i, __ldcs(src + i));
}

__device__ __forceinline__ void copy_f1(float* __restrict__ dst,
                                        const float* __restrict__ src, int64_t n)
{
    const int64_t gtid = int64_t(blockIdx.x) * kPackThreads + threadIdx.x;
    for (int64_t i = gtid; i < n; i += int64_t(gridDim.x) * kPackThreads)
        dst[i] = src[i];
}

template <bool kVec>
__global__ void __launch_bounds__(kPackThreads)
    k_ckpt_pack(const float* __restrict__ w, const float* __restrict__ m,
                const float* __restrict__ v, int64_t n, int32_t step,
                unsigned char* __restrict__ image)
{
    if (blockIdx.x == 0 && threadIdx.x == 0)
        *reinterpret_cast<int2*>(image) = make_int2(step, int32_t(n));
    float* dst = reinterpret_cast<float*>(image + 8);
    if (kVec) {
        const int64_t n4 = n >> 2;
        copy_f4(reinterpret_cast<float4*>(dst), reinterpret_cast<const float4*>(w), n4);
        copy_f4(reinterpret_cast<float4*>(dst + n), reinterpret_cast<const float4*>(m), n4);
        copy_f4(reinterpret_cast<float4*>(dst + 2 * n), reinterpret_cast<const float4*>(v), n4);
    } else {
        copy_f1(dst, w, n);
        copy_f1(dst + n, m, n);
        copy_f1(dst + 2 * n, v, n);
    }
}

}  // namespace

int query_pack_caps(int sm_count, KernelCaps* caps)
{
    cudaError_t err = cudaSuccess;
    caps->pack_vec = detail::resident_blocks(reinterpret_cast<const void*>(&k_ckpt_pack<true>),
                                             kPackThreads, sm_count, &err);
    caps->pack_scalar = detail::resident_blocks(
        reinterpret_cast<const void*>(&k_ckpt_pack<false>), kPackThreads, sm_count, &err);
    return int(err);
}

int launch_pack(const float* w, const float* m, const float* v, int64_t n,
                int32_t step, unsigned char* image, const KernelCaps& caps,
                void* stream)
{
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const bool vec = (n % 4 == 0) && detail::aligned16(w) && detail::aligned16(m) && detail::aligned16(v) &&
                     detail::aligned16(image + 8);
    if (vec) {
        const int cap = caps.pack_vec;
        const int64_t want = detail::ceil_div(n >> 2, int64_t(kPackThreads) * kPackVec);
        const int blocks = int(want < 1 ? 1 : (want > cap ? cap : want));
        k_ckpt_pack<true><<<blocks, kPackThreads, 0, s>>>(w, m, v, n, step, image);
    } else {
        const int cap = caps.pack_scalar;
        const int64_t want = detail::ceil_div(n, kPackThreads);
        const int blocks = int(want < 1 ? 1 : (want > cap ? cap : want));
        k_ckpt_pack<false><<<blocks, kPackThreads, 0, s>>>(w, m, v, n, step, image);
    }
    return int(cudaGetLastError());
}

}  // namespace osr
