// adamw_dev.cuh -- the per-element clip + AdamW update and the vector pass
// over a flat state, shared by the fused kernel (step.cu) and the one-launch
// step (onepass.cu), so that both produce the same bits for every element.
//
// "Training as a Recoverable State Transition" (aihero.club), section "The
// Exact Targets of Clipping and AdamW".
#pragma once

#include <cstdint>
#include <type_traits>

#include <cuda_runtime.h>

#include "common.cuh"
#include "internal.h"

namespace osr {
namespace adamwdev {

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
//   w     = w d - (lr / (1 - beta1^t)) (m / denom)   (one fma)
// where d = 1 - lr wd, or exactly 1 for an element exempt from decay.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void adamw_elem(float& w, float g, float& m, float& v,
                                           float s, const StepScalars& k, float d)
{
    const float gh = __fmul_rn(g, s);
    m = __fmaf_rn(k.beta1, m, __fmul_rn(k.omb1, gh));
    v = __fmaf_rn(k.beta2, v, __fmul_rn(__fmul_rn(k.omb2, gh), gh));
    const float denom = __fmaf_rn(__fsqrt_rn(v), k.inv_sqrt_bc2, k.eps);
    const float upd = __fmul_rn(k.step_size, __fdiv_rn(m, denom));
    w = __fmaf_rn(w, d, -upd);
}

// bits: the decay flags of the four elements (bit j set: element j decays).
__device__ __forceinline__ void adamw4(float4& w, float4 g, float4& m, float4& v,
                                       float s, const StepScalars& k, uint32_t bits)
{
    adamw_elem(w.x, g.x, m.x, v.x, s, k, (bits & 1u) ? k.decay : 1.0f);
    adamw_elem(w.y, g.y, m.y, v.y, s, k, (bits & 2u) ? k.decay : 1.0f);
    adamw_elem(w.z, g.z, m.z, v.z, s, k, (bits & 4u) ? k.decay : 1.0f);
    adamw_elem(w.w, g.w, m.w, v.w, s, k, (bits & 8u) ? k.decay : 1.0f);
}

// Per-group weight decay: element e decays when bit e % 32 of word e / 32 of
// the mask is set.  The flags of the float4 at float4 index i are the nibble
// (i % 8) of word i / 8.  Without kMask every element decays, and the
// selects fold away at compile time.
template <bool kMask>
__device__ __forceinline__ uint32_t decay_nibble(const uint32_t* __restrict__ mask, int64_t i)
{
    if constexpr (kMask)
        return (__ldg(mask + (i >> 3)) >> ((int(i) & 7) << 2)) & 0xFu;
    else
        return 0xFu;
}

template <bool kMask>
__device__ __forceinline__ float decay_one(const uint32_t* __restrict__ mask, int64_t e,
                                           const StepScalars& k)
{
    if constexpr (kMask)
        return ((__ldg(mask + (e >> 5)) >> (int(e) & 31)) & 1u) ? k.decay : 1.0f;
    else
        return k.decay;
}

constexpr int kStepThreads = 256;
constexpr int kStepVec = 2;  // float4 of each array per thread per chunk

// The vector pass over all of [0, n) by one grid: chunks of kStepVec float4
// per thread dealt out cyclically over the blocks, then the float4 tail,
// then the last n % 4 elements.  w, g, m, v (and w_lp) at 16-byte (16-bit
// types: 8-byte) boundaries.  s is the factor applied to each gradient
// element; kZero writes 0 into g after reading it; WL, if not void, is the
// type of a 16-bit copy of the new weights; kMask reads k.decay_mask.
template <bool kZero, typename G, typename WL, bool kMask>
__device__ __forceinline__ void vector_pass(float* __restrict__ w, const G* __restrict__ g,
                                            float* __restrict__ m, float* __restrict__ v,
                                            int64_t n, float s, const StepScalars& k,
                                            WL* __restrict__ w_lp)
{
    constexpr bool kCopy = !std::is_void<WL>::value;
    const uint32_t* __restrict__ decay_mask = k.decay_mask;
    G* const gw = const_cast<G*>(g);  // written through the pointer it is read from
    const int64_t gtid = int64_t(blockIdx.x) * kStepThreads + threadIdx.x;
    const int64_t stride = int64_t(gridDim.x) * kStepThreads;
    {
        float4* w4 = reinterpret_cast<float4*>(w);
        float4* m4 = reinterpret_cast<float4*>(m);
        float4* v4 = reinterpret_cast<float4*>(v);
        const int64_t n4 = n >> 2;
        constexpr int64_t chunk = int64_t(kStepThreads) * kStepVec;
        const int64_t nchunks = n4 / chunk;
        // Chunks: handed out by an atomic counter when k.chunk_ctr is set --
        // a block that starts late (its SM busy with another kernel) simply
        // takes fewer -- else dealt out cyclically by block.  Thread 0 asks
        // for the block's next chunk while the current one is processed.
        __shared__ uint32_t s_next[2];
        uint32_t* const ctr = k.chunk_ctr;
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
            float4 W[kStepVec], G4[kStepVec], M[kStepVec], V[kStepVec];
            uint32_t D[kStepVec];
#pragma unroll
            for (int j = 0; j < kStepVec; ++j) {
                const int64_t i = i0 + j * kStepThreads;
                W[j] = __ldcs(w4 + i);
                G4[j] = detail::load4_cs<G>(g + (i << 2));
                M[j] = __ldcs(m4 + i);
                V[j] = __ldcs(v4 + i);
                D[j] = decay_nibble<kMask>(decay_mask, i);
            }
#pragma unroll
            for (int j = 0; j < kStepVec; ++j)
                adamw4(W[j], G4[j], M[j], V[j], s, k, D[j]);
#pragma unroll
            for (int j = 0; j < kStepVec; ++j) {
                const int64_t i = i0 + j * kStepThreads;
                __stcs(w4 + i, W[j]);
                __stcs(m4 + i, M[j]);
                __stcs(v4 + i, V[j]);
                if constexpr (kZero)
                    detail::store4_zero_cs(gw + (i << 2));
                if constexpr (kCopy)
                    detail::store4_lp_cs(w_lp + (i << 2), W[j]);
            }
            if (ctr) {
                __syncthreads();  // the prefetched index is visible; s_next[buf] is free
                buf ^= 1;
                c = s_next[buf];
            } else {
                c += gridDim.x;
            }
        }
        if (ctr && threadIdx.x == 0) {
            // every block has drawn its last index before it counts itself
            // out; the last one out resets the counters for the next launch
            __threadfence();
            if (atomicAdd(ctr + 1, 1u) == gridDim.x - 1) {
                atomicExch(ctr, 0u);
                atomicExch(ctr + 1, 0u);
            }
        }
        for (int64_t i = nchunks * chunk + gtid; i < n4; i += stride) {
            float4 W = __ldcs(w4 + i), G4 = detail::load4_cs<G>(g + (i << 2)),
                   M = __ldcs(m4 + i), V = __ldcs(v4 + i);
            adamw4(W, G4, M, V, s, k, decay_nibble<kMask>(decay_mask, i));
            __stcs(w4 + i, W);
            __stcs(m4 + i, M);
            __stcs(v4 + i, V);
            if constexpr (kZero)
                detail::store4_zero_cs(gw + (i << 2));
            if constexpr (kCopy)
                detail::store4_lp_cs(w_lp + (i << 2), W);
        }
        if (gtid < (n & 3)) {
            const int64_t e = (n4 << 2) + gtid;
            float W = w[e], M = m[e], V = v[e];
            adamw_elem(W, detail::load1(g + e), M, V, s, k, decay_one<kMask>(decay_mask, e, k));
            w[e] = W;
            m[e] = M;
            v[e] = V;
            if constexpr (kZero)
                detail::store1_zero(gw + e);
            if constexpr (kCopy)
                detail::store1_lp(w_lp + e, W);
        }
    }
}

}  // namespace adamwdev
}  // namespace osr
