// kernels.cu -- the streaming kernels of the clipped-AdamW step and of the
// checkpoint pack, for sm_103a.
//
// All three are HBM-bound (about 0.5 flop per byte), so the design is about
// bytes: each array is touched once per kernel with 128-bit accesses and
// streaming (evict-first) cache hints, enough independent loads in flight
// per thread to cover HBM latency, and grids sized to the resident blocks of
// all 152 SMs.  No tensor cores: nothing here is a contraction.
//
// Method sources: "Training as a Recoverable State Transition" (aihero.club),
// section "The Exact Targets of Clipping and AdamW" (global L2 clip; AdamW
// with bias correction and decoupled decay); "Grow a Language Model:
// Checkpoints" (unhomeschool.com), section "Format" (the file image);
// "Grow a Language Model: Backprop", section "Every forward op gets a
// backward twin" (the clip kernels k_grad_norm_partial / k_grad_norm_final /
// k_grad_scale, which this file replaces by one reduction kernel and one
// fused scale+update kernel).
#include <cfloat>
#include <cstdint>

#include <cuda_runtime.h>

#include "internal.h"

namespace osr {
namespace {

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

// (a^2 + b^2) + (c^2 + d^2): two fused multiply-adds and one add, each
// correctly rounded in float32.
__device__ __forceinline__ float sumsq4(float4 a)
{
    return __fadd_rn(__fmaf_rn(a.x, a.x, __fmul_rn(a.y, a.y)),
                     __fmaf_rn(a.z, a.z, __fmul_rn(a.w, a.w)));
}

// Sum of squares of one run of 4*U values.  Fast path: float32 squares,
// pairwise tree (depth 2 + log2 U), so the relative error is at most about
// (3 + log2 U) units of 2^-24 -- 3.6e-7 for U = 8 -- and the run is flushed
// into the caller's double accumulator.  Runs whose float32 sum leaves
// [2^-100, FLT_MAX] (overflow, inf, nan, or values so small that squares
// underflow) are recomputed exactly in double; all-zero runs (common for
// embedding rows no token touched) skip that and contribute 0.
template <int U>
__device__ __forceinline__ double run_sumsq(const float4 (&x)[U])
{
    float q[U];
#pragma unroll
    for (int j = 0; j < U; ++j)
        q[j] = sumsq4(x[j]);
#pragma unroll
    for (int s = 1; s < U; s <<= 1)
#pragma unroll
        for (int j = 0; j + s < U; j += 2 * s)
            q[j] = __fadd_rn(q[j], q[j + s]);
    const float r = q[0];
    if (r >= 0x1p-100f && r <= FLT_MAX)
        return double(r);
    unsigned bits = 0;
#pragma unroll
    for (int j = 0; j < U; ++j)
        bits |= (__float_as_uint(x[j].x) | __float_as_uint(x[j].y) |
                 __float_as_uint(x[j].z) | __float_as_uint(x[j].w)) & 0x7fffffffu;
    if (bits == 0)
        return 0.0;
    double d = 0.0;
#pragma unroll
    for (int j = 0; j < U; ++j) {
        d += double(x[j].x) * double(x[j].x);
        d += double(x[j].y) * double(x[j].y);
        d += double(x[j].z) * double(x[j].z);
        d += double(x[j].w) * double(x[j].w);
    }
    return d;
}

// ---------------------------------------------------------------------------
// Global L2 norm, two levels in one launch.
//
// Level 1: the flat vector is cut into tiles of kNormTileElems elements;
// block b takes tiles b, b + P, b + 2P, ... (P = norm_blocks(n), a function
// of n alone).  Thread t of a tile holds U = kNormVecPerThread float4s at
// float4 index j*256 + t (coalesced), sums their squares as one run, and
// adds the run into a double.  The block's doubles are summed with a fixed
// shuffle tree into partials[b].
// Level 2: the block that finishes last (atomic ticket) sums partials[0..P)
// in a fixed order -- independent of which block that is -- takes the square
// root and the clip factor, and publishes the result.  No block waits on
// another; the ticket counter is reset for the next launch.
// ---------------------------------------------------------------------------
template <bool kVec>
__global__ void __launch_bounds__(kNormThreads)
    k_grad_norm(const float* __restrict__ g, int64_t n, double clip,
                double* __restrict__ partials, unsigned int* __restrict__ counter,
                NormResult* __restrict__ d_res, NormResult* h_res)
{
    constexpr int U = kNormVecPerThread;
    const int tid = threadIdx.x;
    const int64_t ntiles = (n + kNormTileElems - 1) / kNormTileElems;
    const int64_t nfull = n / kNormTileElems;
    double acc = 0.0;
    for (int64_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
        const int64_t base = tile * kNormTileElems;
        float4 x[U];
        if (tile < nfull) {
            if (kVec) {
                const float4* p = reinterpret_cast<const float4*>(g + base) + tid;
#pragma unroll
                for (int j = 0; j < U; ++j)
                    x[j] = __ldcs(p + j * kNormThreads);
            } else {
#pragma unroll
                for (int j = 0; j < U; ++j) {
                    const float* p = g + base + (int64_t(j * kNormThreads + tid) << 2);
                    x[j] = make_float4(__ldcs(p), __ldcs(p + 1), __ldcs(p + 2), __ldcs(p + 3));
                }
            }
        } else {
#pragma unroll
            for (int j = 0; j < U; ++j) {
                const int64_t e = base + (int64_t(j * kNormThreads + tid) << 2);
                x[j].x = e < n ? g[e] : 0.0f;
                x[j].y = e + 1 < n ? g[e + 1] : 0.0f;
                x[j].z = e + 2 < n ? g[e + 2] : 0.0f;
                x[j].w = e + 3 < n ? g[e + 3] : 0.0f;
            }
        }
        acc += run_sumsq<U>(x);
    }

    acc = block_sum<kNormThreads>(acc);
    __shared__ bool is_last;
    if (tid == 0) {
        partials[blockIdx.x] = acc;
        __threadfence();
        const unsigned ticket = atomicAdd(counter, 1u);
        is_last = (ticket == gridDim.x - 1);
    }
    __syncthreads();
    if (!is_last)
        return;
    __threadfence();
    double s = 0.0;
    for (int i = tid; i < int(gridDim.x); i += kNormThreads)
        s += __ldcg(partials + i);
    s = block_sum<kNormThreads>(s);
    if (tid == 0) {
        NormResult r;
        r.sumsq = s;
        r.norm = sqrt(s);
        const bool finite = isfinite(r.norm);
        r.nonfinite = finite ? 0 : 1;
        r.scale = (finite && r.norm > clip) ? float(clip / r.norm) : 1.0f;
        r.seq = d_res->seq + 1u;
        r.pad = 0;
        *d_res = r;
        if (h_res) {
            volatile NormResult* h = h_res;
            h->sumsq = r.sumsq;
            h->norm = r.norm;
            h->scale = r.scale;
            h->nonfinite = r.nonfinite;
            h->seq = r.seq;
            __threadfence_system();
        }
        *counter = 0u;
    }
}

// ---------------------------------------------------------------------------
// Fused clip + AdamW: one element.  Every operation is an explicitly
// rounded float32 intrinsic (IEEE square root and division; no fast-math),
// in this order:
//   g_hat = g s
//   m     = beta1 m + (1 - beta1) g_hat             (one fma)
//   v     = beta2 v + ((1 - beta2) g_hat) g_hat      (one fma; the factor
//                                                     first, so g_hat^2 never
//                                                     overflows on its own)
//   denom = sqrt(v) / sqrt(1 - beta2^t) + eps        (one fma) = sqrt(v_hat)+eps
//   w     = w (1 - lr wd) - (lr / (1 - beta1^t)) (m / denom)      (one fma)
// ---------------------------------------------------------------------------
__device__ __forceinline__ void adamw_elem(float& w, float g, float& m, float& v,
                                           float s, const StepScalars& k)
{
    const float gh = __fmul_rn(g, s);
    m = __fmaf_rn(k.beta1, m, __fmul_rn(k.omb1, gh));
    v = __fmaf_rn(k.beta2, v, __fmul_rn(__fmul_rn(k.omb2, gh), gh));
    const float denom = __fmaf_rn(__fsqrt_rn(v), k.inv_sqrt_bc2, k.eps);
    const float upd = __fmul_rn(k.step_size, __fdiv_rn(m, denom));
    w = __fmaf_rn(w, k.decay, -upd);
}

__device__ __forceinline__ void adamw4(float4& w, float4 g, float4& m, float4& v,
                                       float s, const StepScalars& k)
{
    adamw_elem(w.x, g.x, m.x, v.x, s, k);
    adamw_elem(w.y, g.y, m.y, v.y, s, k);
    adamw_elem(w.z, g.z, m.z, v.z, s, k);
    adamw_elem(w.w, g.w, m.w, v.w, s, k);
}

constexpr int kStepThreads = 256;
constexpr int kStepVec = 2;  // float4 of each array per thread per chunk

// Reads w, g, m, v once and writes w, m, v once (28 bytes per parameter).
// The clip factor and the non-finite flag come from the norm kernel's
// result in device memory, so nothing returns to the host between kernels.
template <bool kVec>
__global__ void __launch_bounds__(kStepThreads)
    k_clip_adamw(float* __restrict__ w, const float* __restrict__ g,
                 float* __restrict__ m, float* __restrict__ v, int64_t n,
                 StepScalars k, const NormResult* __restrict__ res)
{
    if (res->nonfinite)
        return;
    const float s = res->scale;
    const int64_t gtid = int64_t(blockIdx.x) * kStepThreads + threadIdx.x;
    const int64_t stride = int64_t(gridDim.x) * kStepThreads;
    if (kVec) {
        float4* w4 = reinterpret_cast<float4*>(w);
        const float4* g4 = reinterpret_cast<const float4*>(g);
        float4* m4 = reinterpret_cast<float4*>(m);
        float4* v4 = reinterpret_cast<float4*>(v);
        const int64_t n4 = n >> 2;
        constexpr int64_t chunk = int64_t(kStepThreads) * kStepVec;
        const int64_t nchunks = n4 / chunk;
        for (int64_t c = blockIdx.x; c < nchunks; c += gridDim.x) {
            const int64_t i0 = c * chunk + threadIdx.x;
            float4 W[kStepVec], G[kStepVec], M[kStepVec], V[kStepVec];
#pragma unroll
            for (int j = 0; j < kStepVec; ++j) {
                const int64_t i = i0 + j * kStepThreads;
                W[j] = __ldcs(w4 + i);
                G[j] = __ldcs(g4 + i);
                M[j] = __ldcs(m4 + i);
                V[j] = __ldcs(v4 + i);
            }
#pragma unroll
            for (int j = 0; j < kStepVec; ++j)
                adamw4(W[j], G[j], M[j], V[j], s, k);
#pragma unroll
            for (int j = 0; j < kStepVec; ++j) {
                const int64_t i = i0 + j * kStepThreads;
                __stcs(w4 + i, W[j]);
                __stcs(m4 + i, M[j]);
                __stcs(v4 + i, V[j]);
            }
        }
        for (int64_t i = nchunks * chunk + gtid; i < n4; i += stride) {
            float4 W = __ldcs(w4 + i), G = __ldcs(g4 + i), M = __ldcs(m4 + i),
                   V = __ldcs(v4 + i);
            adamw4(W, G, M, V, s, k);
            __stcs(w4 + i, W);
            __stcs(m4 + i, M);
            __stcs(v4 + i, V);
        }
        if (gtid < (n & 3)) {
            const int64_t e = (n4 << 2) + gtid;
            float W = w[e], M = m[e], V = v[e];
            adamw_elem(W, g[e], M, V, s, k);
            w[e] = W;
            m[e] = M;
            v[e] = V;
        }
    } else {
        for (int64_t e = gtid; e < n; e += stride) {
            float W = __ldcs(w + e), M = __ldcs(m + e), V = __ldcs(v + e);
            adamw_elem(W, __ldcs(g + e), M, V, s, k);
            __stcs(w + e, W);
            __stcs(m + e, M);
            __stcs(v + e, V);
        }
    }
}

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

inline bool aligned16(const void* p)
{
    return (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
}

inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

int resident_blocks(const void* kernel, int threads, int sm_count)
{
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads, 0) != cudaSuccess ||
        per_sm < 1)
        per_sm = 1;
    return per_sm * sm_count;
}

}  // namespace

int launch_norm(const float* g, int64_t n, double clip, double* partials,
                unsigned int* counter, NormResult* d_res, NormResult* h_res_dev,
                void* stream)
{
    const int blocks = norm_blocks(n);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (aligned16(g))
        k_grad_norm<true><<<blocks, kNormThreads, 0, s>>>(g, n, clip, partials, counter,
                                                           d_res, h_res_dev);
    else
        k_grad_norm<false><<<blocks, kNormThreads, 0, s>>>(g, n, clip, partials, counter,
                                                            d_res, h_res_dev);
    return int(cudaGetLastError());
}

int query_kernel_caps(int sm_count, KernelCaps* caps)
{
    caps->step_vec = resident_blocks(reinterpret_cast<const void*>(&k_clip_adamw<true>),
                                     kStepThreads, sm_count);
    caps->step_scalar = resident_blocks(reinterpret_cast<const void*>(&k_clip_adamw<false>),
                                        kStepThreads, sm_count);
    caps->pack_vec = resident_blocks(reinterpret_cast<const void*>(&k_ckpt_pack<true>),
                                     kPackThreads, sm_count);
    caps->pack_scalar = resident_blocks(reinterpret_cast<const void*>(&k_ckpt_pack<false>),
                                        kPackThreads, sm_count);
    return int(cudaGetLastError());
}

int launch_adamw(float* w, const float* g, float* m, float* v, int64_t n,
                 const StepScalars& k, const NormResult* d_res, const KernelCaps& caps,
                 void* stream)
{
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const bool vec = aligned16(w) && aligned16(g) && aligned16(m) && aligned16(v);
    if (vec) {
        const int cap = caps.step_vec;
        const int64_t want = ceil_div(n >> 2, int64_t(kStepThreads) * kStepVec);
        const int blocks = int(want < 1 ? 1 : (want > cap ? cap : want));
        k_clip_adamw<true><<<blocks, kStepThreads, 0, s>>>(w, g, m, v, n, k, d_res);
    } else {
        const int cap = caps.step_scalar;
        const int64_t want = ceil_div(n, kStepThreads);
        const int blocks = int(want < 1 ? 1 : (want > cap ? cap : want));
        k_clip_adamw<false><<<blocks, kStepThreads, 0, s>>>(w, g, m, v, n, k, d_res);
    }
    return int(cudaGetLastError());
}

int launch_pack(const float* w, const float* m, const float* v, int64_t n,
                int32_t step, unsigned char* image, const KernelCaps& caps,
                void* stream)
{
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const bool vec = (n % 4 == 0) && aligned16(w) && aligned16(m) && aligned16(v) &&
                     aligned16(image + 8);
    if (vec) {
        const int cap = caps.pack_vec;
        const int64_t want = ceil_div(n >> 2, int64_t(kPackThreads) * kPackVec);
        const int blocks = int(want < 1 ? 1 : (want > cap ? cap : want));
        k_ckpt_pack<true><<<blocks, kPackThreads, 0, s>>>(w, m, v, n, step, image);
    } else {
        const int cap = caps.pack_scalar;
        const int64_t want = ceil_div(n, kPackThreads);
        const int blocks = int(want < 1 ? 1 : (want > cap ? cap : want));
        k_ckpt_pack<false><<<blocks, kPackThreads, 0, s>>>(w, m, v, n, step, image);
    }
    return int(cudaGetLastError());
}

}  // namespace osr
