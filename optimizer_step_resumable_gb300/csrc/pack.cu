// pack.cu -- the checkpoint pack (row a5): the parts of the step_NNNNNN.bin
// image [int32 step][int32 n][n f32 w][n f32 m][n f32 v] written into a
// device staging buffer, for sm_103a.
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
// Checkpoint pack: the header [int32 step][int32 n] and the w, m, v regions
// into the device staging slots (each 256-byte aligned; the copy to the host
// places them at their file offsets).  A pure copy of 12 n bytes: the three
// arrays are read and written in the same pass (six float4 streams, like the
// fused step), and the stores start on cache-line boundaries -- with the
// regions 16 bytes past a boundary, as in a contiguous device image, the same
// copy ran at 0.79-0.86 of the copy bandwidth at 2^30 parameters instead of
// about 1.0.
// ---------------------------------------------------------------------------
constexpr int kPackThreads = 256;
constexpr int kPackVec = 2;           // float4 of each array per thread per chunk
constexpr int kPackBlocksPerSm = 8;   // measured best: two rounds of resident blocks

// ctr (may be NULL): chunk counters as in the fused kernel (handed out by an
// atomic counter, reset by the last block out); NULL: chunks dealt out
// cyclically by block.
template <bool kVec>
__global__ void __launch_bounds__(kPackThreads, 4)
    k_ckpt_pack(const float* __restrict__ w, const float* __restrict__ m,
                const float* __restrict__ v, int64_t n, int32_t step, int2* __restrict__ header,
                float* __restrict__ dw, float* __restrict__ dm, float* __restrict__ dv,
                uint32_t* __restrict__ ctr)
{
    if (blockIdx.x == 0 && threadIdx.x == 0)
        *header = make_int2(step, int32_t(n));
    const int64_t gtid = int64_t(blockIdx.x) * kPackThreads + threadIdx.x;
    const int64_t stride = int64_t(gridDim.x) * kPackThreads;
    int64_t done = 0;  // elements covered by the vector part
    if (kVec) {
        const float4* w4 = reinterpret_cast<const float4*>(w);
        const float4* m4 = reinterpret_cast<const float4*>(m);
        const float4* v4 = reinterpret_cast<const float4*>(v);
        float4* dw4 = reinterpret_cast<float4*>(dw);
        float4* dm4 = reinterpret_cast<float4*>(dm);
        float4* dv4 = reinterpret_cast<float4*>(dv);
        const int64_t n4 = n >> 2;
        constexpr int64_t chunk = int64_t(kPackThreads) * kPackVec;
        const int64_t nchunks = n4 / chunk;
        __shared__ uint32_t s_next[2];
        int buf = 0;
        int64_t c = blockIdx.x;
        if (ctr) {
            if (threadIdx.x == 0)
                s_next[0] = atomicAdd(ctr, 1u);
            __syncthreads();
            c = s_next[0];
        }
        while (c < nchunks) {
            if (ctr && threadIdx.x == 0)
                s_next[buf ^ 1] = atomicAdd(ctr, 1u);
            const int64_t i0 = c * chunk + threadIdx.x;
            float4 a[kPackVec], b[kPackVec], e[kPackVec];
#pragma unroll
            for (int j = 0; j < kPackVec; ++j) {
                a[j] = __ldcs(w4 + i0 + j * kPackThreads);
                b[j] = __ldcs(m4 + i0 + j * kPackThreads);
                e[j] = __ldcs(v4 + i0 + j * kPackThreads);
            }
#pragma unroll
            for (int j = 0; j < kPackVec; ++j) {
                __stcs(dw4 + i0 + j * kPackThreads, a[j]);
                __stcs(dm4 + i0 + j * kPackThreads, b[j]);
                __stcs(dv4 + i0 + j * kPackThreads, e[j]);
            }
            if (ctr) {
                __syncthreads();
                buf ^= 1;
                c = s_next[buf];
            } else {
                c += gridDim.x;
            }
        }
        if (ctr && threadIdx.x == 0) {
            __threadfence();
            if (atomicAdd(ctr + 1, 1u) == gridDim.x - 1) {
                atomicExch(ctr, 0u);
                atomicExch(ctr + 1, 0u);
            }
        }
        for (int64_t i = nchunks * chunk + gtid; i < n4; i += stride) {
            __stcs(dw4 + i, __ldcs(w4 + i));
            __stcs(dm4 + i, __ldcs(m4 + i));
            __stcs(dv4 + i, __ldcs(v4 + i));
        }
        done = n4 << 2;
    }
    for (int64_t i = done + gtid; i < n; i += stride) {
        dw[i] = w[i];
        dm[i] = m[i];
        dv[i] = v[i];
    }
}

// ---------------------------------------------------------------------------
// Staging -> pinned host image, by the SMs (the side stream's alternative to
// the copy engine).  Region r of the image starts at byte 8 + 4 n (r - 1) of
// the page-aligned host image: 16-byte aligned when that offset is, else 8-
// or 4-byte aligned, so each float4 read from the (256-byte aligned) slot is
// stored as one 16-byte, two 8-byte or four 4-byte stores.  One block per SM
// on the side stream: measured on GB300, the copy engine's copy into pinned
// memory just written to a file took 80-116 ms for 1.33 GB where this took
// 7-14 ms (both 6.9 ms into a fresh buffer); the concurrent steps lose about
// 4 ms in all.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void copy_region_to_host(const float4* __restrict__ src,
                                                    unsigned char* dst, int64_t n)
{
    const int64_t n4 = n >> 2;
    const int64_t gtid = int64_t(blockIdx.x) * kPackThreads + threadIdx.x;
    const int64_t stride = int64_t(gridDim.x) * kPackThreads;
    const unsigned mis = unsigned(reinterpret_cast<uintptr_t>(dst) & 15u);
    if (mis == 0) {
        float4* d = reinterpret_cast<float4*>(dst);
        for (int64_t i = gtid; i < n4; i += stride)
            __stcs(d + i, __ldcs(src + i));
    } else if (mis == 8) {
        uint2* d = reinterpret_cast<uint2*>(dst);
        for (int64_t i = gtid; i < n4; i += stride) {
            const float4 x = __ldcs(src + i);
            __stcs(d + 2 * i, make_uint2(__float_as_uint(x.x), __float_as_uint(x.y)));
            __stcs(d + 2 * i + 1, make_uint2(__float_as_uint(x.z), __float_as_uint(x.w)));
        }
    } else {
        float* d = reinterpret_cast<float*>(dst);
        for (int64_t i = gtid; i < n4; i += stride) {
            const float4 x = __ldcs(src + i);
            __stcs(d + 4 * i, x.x);
            __stcs(d + 4 * i + 1, x.y);
            __stcs(d + 4 * i + 2, x.z);
            __stcs(d + 4 * i + 3, x.w);
        }
    }
    const float* s1 = reinterpret_cast<const float*>(src);
    float* d1 = reinterpret_cast<float*>(dst);
    for (int64_t e = (n4 << 2) + gtid; e < n; e += stride)
        d1[e] = s1[e];
}

__global__ void __launch_bounds__(kPackThreads)
    k_stage_to_host(const int2* __restrict__ header, const float* __restrict__ sw,
                    const float* __restrict__ sm, const float* __restrict__ sv, int64_t n,
                    unsigned char* image)
{
    if (blockIdx.x == 0 && threadIdx.x == 0)
        *reinterpret_cast<int2*>(image) = *header;
    const int64_t rb = 4 * n;
    copy_region_to_host(reinterpret_cast<const float4*>(sw), image + 8, n);
    copy_region_to_host(reinterpret_cast<const float4*>(sm), image + 8 + rb, n);
    copy_region_to_host(reinterpret_cast<const float4*>(sv), image + 8 + 2 * rb, n);
}

}  // namespace

int launch_stage_to_host(const unsigned char* header, const float* sw, const float* sm,
                         const float* sv, int64_t n, unsigned char* image_dev, int blocks,
                         void* stream)
{
    k_stage_to_host<<<blocks, kPackThreads, 0, static_cast<cudaStream_t>(stream)>>>(
        reinterpret_cast<const int2*>(header), sw, sm, sv, n, image_dev);
    return int(cudaGetLastError());
}

int query_pack_caps(int sm_count, KernelCaps* caps)
{
    caps->pack_vec = kPackBlocksPerSm * sm_count;
    caps->pack_scalar = kPackBlocksPerSm * sm_count;
    return int(cudaSuccess);
}

int launch_pack(const float* w, const float* m, const float* v, int64_t n, int32_t step,
                unsigned char* header, float* dw, float* dm, float* dv, const KernelCaps& caps,
                void* stream, uint32_t* chunk_ctr)
{
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int2* h = reinterpret_cast<int2*>(header);
    if (detail::aligned16(w) && detail::aligned16(m) && detail::aligned16(v)) {
        const int cap = caps.pack_vec;
        const int64_t want = detail::ceil_div(n >> 2, int64_t(kPackThreads) * kPackVec);
        const int blocks = int(want < 1 ? 1 : (want > cap ? cap : want));
        k_ckpt_pack<true><<<blocks, kPackThreads, 0, s>>>(w, m, v, n, step, h, dw, dm, dv,
                                                          chunk_ctr);
    } else {
        const int cap = caps.pack_scalar;
        const int64_t want = detail::ceil_div(n, kPackThreads);
        const int blocks = int(want < 1 ? 1 : (want > cap ? cap : want));
        k_ckpt_pack<false><<<blocks, kPackThreads, 0, s>>>(w, m, v, n, step, h, dw, dm, dv,
                                                           nullptr);
    }
    return int(cudaGetLastError());
}

}  // namespace osr
