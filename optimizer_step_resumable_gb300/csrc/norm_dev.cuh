// norm_dev.cuh -- device pieces of the global-norm reduction shared by the
// norm kernel (norm.cu) and the one-launch step (onepass.cu): the tile
// loads, the per-run sum of squares, the fixed-order sum of the block
// partials and the result record.  Both kernels build their partial sums
// from these, over the same tile partition, so they agree bit for bit.
//
// "Training as a Recoverable State Transition" (aihero.club), section "The
// Exact Targets of Clipping and AdamW": the global L2 norm of the joined
// gradient vector and the clip factor c / ||g|| when ||g|| exceeds c.
#pragma once

#include <cfloat>
#include <cstdint>

#include <cuda_runtime.h>

#include "common.cuh"
#include "internal.h"

namespace osr {
namespace normdev {

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

// This thread's share of one tile restricted to elements [lo, hi): exact
// double squares (used only on tiles where a tensor of the offset table
// starts, to split the tile between tensors).
template <int U>
__device__ __forceinline__ double thread_sumsq_in(const float4 (&x)[U], int64_t base, int tid,
                                                  int64_t lo, int64_t hi)
{
    double d = 0.0;
#pragma unroll
    for (int j = 0; j < U; ++j) {
        const int64_t e = base + (int64_t(j * kNormThreads + tid) << 2);
        const float c[4] = {x[j].x, x[j].y, x[j].z, x[j].w};
#pragma unroll
        for (int q = 0; q < 4; ++q)
            if (e + q >= lo && e + q < hi)
                d += double(c[q]) * double(c[q]);
    }
    return d;
}

// Loads this thread's U float4s of tile `tile` (element base tile *
// kNormTileElems; float4 index j * 256 + tid, coalesced).  Full tiles use
// vector loads (kVec: 16-byte aligned float32, or 8-byte aligned 16-bit
// types) or four scalar loads; the ragged last tile reads zeros past n.  The
// loads keep L2's default priority rather than evict-first: the fused kernel
// reads g again right after, and at up to a few tens of millions of
// parameters it then finds much of g in L2 (measured on GB300: the step 5-12%
// faster at 2^21-2^24 and 12.8M, the same from 2^25 up).
template <int U, bool kVec, typename G>
__device__ __forceinline__ void load_tile(const G* __restrict__ g, int64_t n, int64_t nfull,
                                          int64_t tile, int tid, float4 (&x)[U])
{
    const int64_t base = tile * kNormTileElems;
    if (tile < nfull) {
        if constexpr (kVec) {
#pragma unroll
            for (int j = 0; j < U; ++j)
                x[j] = detail::load4_cg<G>(g + base + (int64_t(j * kNormThreads + tid) << 2));
        } else {  // float32 at a 4-byte (not 16-byte) boundary
#pragma unroll
            for (int j = 0; j < U; ++j) {
                const G* p = g + base + (int64_t(j * kNormThreads + tid) << 2);
                x[j] = make_float4(__ldcg(p), __ldcg(p + 1), __ldcg(p + 2), __ldcg(p + 3));
            }
        }
    } else {
#pragma unroll
        for (int j = 0; j < U; ++j) {
            const int64_t e = base + (int64_t(j * kNormThreads + tid) << 2);
            x[j].x = e < n ? detail::load1(g + e) : 0.0f;
            x[j].y = e + 1 < n ? detail::load1(g + e + 1) : 0.0f;
            x[j].z = e + 2 < n ? detail::load1(g + e + 2) : 0.0f;
            x[j].w = e + 3 < n ? detail::load1(g + e + 3) : 0.0f;
        }
    }
}

// Level 2: the sum of partials[0..P) in a fixed order (a strided sum per
// thread, then the fixed shuffle tree); valid in thread 0.  All threads of
// the block must call it.
__device__ __forceinline__ double sum_partials(const double* partials, int P)
{
    double s = 0.0;
    for (int i = threadIdx.x; i < P; i += kNormThreads)
        s += __ldcg(partials + i);
    return detail::block_sum<kNormThreads>(s);
}

// The result of a reduction with sum of squares s: the norm of the scaled
// gradient grad_scale * g, and the factor applied to raw g (grad_scale times
// the clip factor), rounded once.
__device__ __forceinline__ NormResult make_result(double s, double clip, double grad_scale,
                                                  uint32_t seq)
{
    NormResult r;
    r.sumsq = s;
    r.norm = grad_scale * sqrt(s);
    const bool finite = isfinite(r.norm);
    r.nonfinite = finite ? 0 : 1;
    r.scale = float(grad_scale * ((finite && r.norm > clip) ? clip / r.norm : 1.0));
    r.seq = seq;
    r.fault = 0;
    return r;
}

// Writes r to the device record and, if given, its host-mapped mirror, field
// by field; the fault word is left alone (only a timed-out wait sets it and
// only the host clears it).  No system-scope fence: the host reads the
// mirror only after synchronizing with an event recorded behind this grid,
// and a grid's writes to mapped memory are visible once it has completed (a
// fence here cost about 2 us at the end of every reduction).
__device__ __forceinline__ void publish(const NormResult& r, NormResult* d_res,
                                        NormResult* h_res)
{
    d_res->sumsq = r.sumsq;
    d_res->norm = r.norm;
    d_res->scale = r.scale;
    d_res->nonfinite = r.nonfinite;
    d_res->seq = r.seq;
    if (h_res) {
        volatile NormResult* h = h_res;
        h->sumsq = r.sumsq;
        h->norm = r.norm;
        h->scale = r.scale;
        h->nonfinite = r.nonfinite;
        h->seq = r.seq;
    }
}

}  // namespace normdev
}  // namespace osr
