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
// the page-aligned host image, which is 16-byte aligned or 4, 8 or 12 bytes
// short of it; the kH floats up to the boundary are copied one by one, and
// each thread then writes whole aligned 16-byte units, assembling each from
// two neighbouring float4 of the (256-byte aligned) staging slot.
//
// Measured on GB300 with the 110M list (1.33 GB image): host stores stall
// the memory pipeline of the SM that issues them, so the steps running
// beside the copy lose time on every SM that holds a copy block.  One block
// per SM (256 threads, 8- and 16-byte stores as the alignment allowed) cost
// the concurrent steps 4.7 ms per checkpoint (each overlapped step 1.22 ms
// instead of 0.436) for a 9.3 ms copy; a quarter of the SMs with 1024
// threads each and aligned 16-byte stores copy in 7.9 ms and cost 0.39 ms.
// The copy engine was no way out: its first copy into pages that the CPU or
// the disk path had just touched took 50-150 ms (6.9 ms otherwise).
// ---------------------------------------------------------------------------
constexpr int kStageThreads = 1024;
constexpr int kStageSmsPerBlock = 4;

// The 16 bytes that start kH floats into a, continuing into b.
template <int kH>
__device__ __forceinline__ float4 shift_floats(const float4& a, const float4& b)
{
    if constexpr (kH == 1)
        return make_float4(a.y, a.z, a.w, b.x);
    else if constexpr (kH == 2)
        return make_float4(a.z, a.w, b.x, b.y);
    else
        return make_float4(a.w, b.x, b.y, b.z);
}

// One region: n floats from the slot src (16-byte aligned, readable up to
// its float4 count ceil(n / 4)) to dst, whose first 16-byte boundary is kH
// floats in.
template <int kH>
__device__ __forceinline__ void copy_region_to_host(const float* __restrict__ src, float* dst,
                                                    int64_t n)
{
    const int64_t gtid = int64_t(blockIdx.x) * kStageThreads + threadIdx.x;
    const int64_t stride = int64_t(gridDim.x) * kStageThreads;
    if (kH > 0 && gtid < kH && gtid < n)
        __stcs(dst + gtid, src[gtid]);
    // body: dst floats [kH, kH + 4 nb) as aligned float4; the b operand of
    // unit i is slot float4 i + 1 <= nb <= ceil(n / 4) - 1 (kH >= 1)
    const int64_t nb = n > kH ? (n - kH) >> 2 : 0;
    const float4* __restrict__ s4 = reinterpret_cast<const float4*>(src);
    float4* d4 = reinterpret_cast<float4*>(dst + kH);
    for (int64_t i = gtid; i < nb; i += stride) {
        const float4 a = __ldcs(s4 + i);
        if constexpr (kH == 0) {
            __stcs(d4 + i, a);
        } else {
            const float4 b = __ldcs(s4 + i + 1);
            __stcs(d4 + i, shift_floats<kH>(a, b));
        }
    }
    for (int64_t e = kH + 4 * nb + gtid; e < n; e += stride)
        __stcs(dst + e, src[e]);
}

// Floats from the start of region r (1..3) to its first 16-byte boundary,
// for an image that starts on one: region r starts at byte 8 + 4 n (r - 1).
template <int kNmod4, int kRegion>
__host__ __device__ constexpr int head_floats()
{
    return ((16 - ((8 + 4 * kNmod4 * (kRegion - 1)) & 15)) & 15) / 4;
}

// kNmod4 = n % 4 fixes the three regions' alignment (image 16-byte aligned).
template <int kNmod4>
__global__ void __launch_bounds__(kStageThreads, 1)
    k_stage_to_host(const int2* __restrict__ header, const float* __restrict__ sw,
                    const float* __restrict__ sm, const float* __restrict__ sv, int64_t n,
                    unsigned char* image)
{
    if (blockIdx.x == 0 && threadIdx.x == 0)
        *reinterpret_cast<int2*>(image) = *header;
    float* body = reinterpret_cast<float*>(image + 8);
    copy_region_to_host<head_floats<kNmod4, 1>()>(sw, body, n);
    copy_region_to_host<head_floats<kNmod4, 2>()>(sm, body + n, n);
    copy_region_to_host<head_floats<kNmod4, 3>()>(sv, body + 2 * n, n);
}

}  // namespace

int launch_stage_to_host(const unsigned char* header, const float* sw, const float* sm,
                         const float* sv, int64_t n, unsigned char* image_dev, int sm_count,
                         void* stream)
{
    if (reinterpret_cast<uintptr_t>(image_dev) & 15u)
        return int(cudaErrorInvalidValue);
    const int blocks = sm_count / kStageSmsPerBlock > 0 ? sm_count / kStageSmsPerBlock : 1;
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int2* h = reinterpret_cast<const int2*>(header);
    switch (n & 3) {
    case 0: k_stage_to_host<0><<<blocks, kStageThreads, 0, s>>>(h, sw, sm, sv, n, image_dev); break;
    case 1: k_stage_to_host<1><<<blocks, kStageThreads, 0, s>>>(h, sw, sm, sv, n, image_dev); break;
    case 2: k_stage_to_host<2><<<blocks, kStageThreads, 0, s>>>(h, sw, sm, sv, n, image_dev); break;
    default: k_stage_to_host<3><<<blocks, kStageThreads, 0, s>>>(h, sw, sm, sv, n, image_dev); break;
    }
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
