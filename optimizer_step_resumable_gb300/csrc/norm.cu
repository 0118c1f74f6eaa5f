// norm.cu -- global L2 norm of the flattened gradient and the clip factor
// (rows a1 and a2 of the step), for sm_103a.
//
// "Training as a Recoverable State Transition" (aihero.club), section "The
// Exact Targets of Clipping and AdamW": all gradients are joined into one
// vector g; if ||g||_2 exceeds the threshold c every element is scaled by
// c / ||g||_2.  "Grow a Language Model: Backprop" (unhomeschool.com), section
// "Every forward op gets a backward twin", names the engine's two kernels
// k_grad_norm_partial and k_grad_norm_final; here both levels are one
// launch.  HBM-bound: 4 bytes per parameter.
#include <cfloat>
#include <cstdint>

#include <cuda_runtime.h>

#include "common.cuh"
#include "internal.h"
#include "norm_dev.cuh"

namespace osr {
namespace {

using detail::block_sum;

using normdev::run_sumsq;
using normdev::thread_sumsq_in;

// ---------------------------------------------------------------------------
// Global L2 norm, two levels in one launch.
//
// Level 1: the flat vector is cut into tiles of kNormTileElems elements;
// block b takes the contiguous tiles [T b / P, T (b + 1) / P) (T tiles,
// P = norm_blocks(n): a function of n alone).  Thread t of a tile holds
// U = kNormVecPerThread float4s at float4 index j*256 + t (coalesced), sums
// their squares as one run, and adds the run into a double.  The block's
// doubles are summed with a fixed shuffle tree into partials[b].
// Level 2: the block that finishes last (atomic ticket) sums partials[0..P)
// in a fixed order -- independent of which block that is -- takes the square
// root and the clip factor, and publishes the result.  No block waits on
// another; the ticket counter is reset for the next launch.
//
// kTail = false: no ticket and no last block -- each block writes its
// partial and leaves.  The fused kernel launched right after (a programmatic
// dependent, or plain stream order) then sums the partials itself, in the
// same order, once per block (NormFinish): the step's result is the same
// bits, and the serial tail -- fence, ticket atomic, fence, reads of the
// partials, result stores, about 3 us on GB300 at every size -- is no longer
// between the two kernels.
//
// kSegs: also the sum of squares of each tensor of the offset table, at no
// extra traffic.  Because a block's tiles are contiguous, its threads keep
// one running sum for the tensor they are in; on a tile where a tensor
// starts, each thread splits its elements between the tensors (exact
// doubles) and the block writes the finished tensor's share to its next
// segment slot (slots laid out by the host: block b's tensors are
// kfirst[b] .. kfirst[b+1], their slots start at segbase[b]).  The host adds
// each tensor's slots in block order.
// ---------------------------------------------------------------------------
// (at least 4 resident blocks per SM, so that the fixed 608-block grid is one
// wave on 152 SMs whichever variant runs)
template <bool kVec, bool kSegs, typename G, bool kTail>
__global__ void __launch_bounds__(kNormThreads, 4)
    k_grad_norm(const G* __restrict__ g, int64_t n, double clip, double grad_scale,
                double* __restrict__ partials, unsigned int* __restrict__ counter,
                NormResult* __restrict__ d_res, NormResult* h_res, TensorSegs segs)
{
    constexpr int U = kNormVecPerThread;
    const int tid = threadIdx.x;
    // Let a kernel launched after this one with programmatic serialization
    // start now: it waits (griddepcontrol.wait) for this grid's completion
    // before it reads anything this kernel writes.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int64_t ntiles = (n + kNormTileElems - 1) / kNormTileElems;
    const int64_t nfull = n / kNormTileElems;
    const int64_t t_lo = ntiles * int64_t(blockIdx.x) / int64_t(gridDim.x);
    const int64_t t_hi = ntiles * int64_t(blockIdx.x + 1) / int64_t(gridDim.x);
    double acc = 0.0;
    double seg = 0.0;
    int32_t k = 0, slot = 0;
    int64_t next_start = 0;  // where tensor k + 1 starts
    if (kSegs) {
        k = segs.kfirst[blockIdx.x];
        slot = segs.segbase[blockIdx.x];
        next_start = segs.offsets[k + 1];
    }
    for (int64_t tile = t_lo; tile < t_hi; ++tile) {
        const int64_t base = tile * kNormTileElems;
        float4 x[U];
        normdev::load_tile<U, kVec, G>(g, n, nfull, tile, tid, x);
        const double r = run_sumsq<U>(x);
        acc += r;
        if (kSegs) {
            const int64_t tile_end = base + kNormTileElems < n ? base + kNormTileElems : n;
            if (tile_end <= next_start) {
                seg += r;  // the whole tile lies in tensor k
            } else {
                // block-uniform branch: every thread sees the same tile
                int64_t lo = base;
                for (;;) {
                    const int64_t hi = next_start < tile_end ? next_start : tile_end;
                    seg += thread_sumsq_in<U>(x, base, tid, lo, hi);
                    if (next_start >= tile_end)
                        break;
                    const double done = block_sum<kNormThreads>(seg);
                    if (tid == 0)
                        segs.seg_sums[slot] = done;
                    seg = 0.0;
                    ++slot;
                    ++k;
                    lo = next_start;
                    next_start = segs.offsets[k + 1];
                }
            }
        }
    }
    if (kSegs) {
        const double done = block_sum<kNormThreads>(seg);
        if (tid == 0)
            segs.seg_sums[slot] = done;
    }

    acc = block_sum<kNormThreads>(acc);
    if constexpr (!kTail) {
        if (tid == 0)
            partials[blockIdx.x] = acc;
        return;
    }
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
    const double s = normdev::sum_partials(partials, int(gridDim.x));
    if (tid == 0) {
        normdev::publish(normdev::make_result(s, clip, grad_scale, d_res->seq + 1u), d_res,
                         h_res);
        *counter = 0u;
    }
}

}  // namespace

namespace {

template <typename G, bool kVec, bool kTail>
void launch_norm_tail(const void* g, int64_t n, double clip, double* partials,
                      unsigned int* counter, NormResult* d_res, NormResult* h_res_dev,
                      cudaStream_t s, double grad_scale, const TensorSegs* segs)
{
    const int blocks = norm_blocks(n);
    const TensorSegs none{nullptr, nullptr, nullptr, nullptr};
    const G* gt = static_cast<const G*>(g);
    if (segs)
        k_grad_norm<kVec, true, G, kTail><<<blocks, kNormThreads, 0, s>>>(
            gt, n, clip, grad_scale, partials, counter, d_res, h_res_dev, *segs);
    else
        k_grad_norm<kVec, false, G, kTail><<<blocks, kNormThreads, 0, s>>>(
            gt, n, clip, grad_scale, partials, counter, d_res, h_res_dev, none);
}

template <typename G, bool kVec>
void launch_norm_typed(const void* g, int64_t n, double clip, double* partials,
                       unsigned int* counter, NormResult* d_res, NormResult* h_res_dev,
                       cudaStream_t s, double grad_scale, const TensorSegs* segs, bool tail)
{
    if (tail)
        launch_norm_tail<G, kVec, true>(g, n, clip, partials, counter, d_res, h_res_dev, s,
                                        grad_scale, segs);
    else
        launch_norm_tail<G, kVec, false>(g, n, clip, partials, counter, d_res, h_res_dev, s,
                                         grad_scale, segs);
}

}  // namespace

int launch_norm(const void* g, int64_t n, double clip, double* partials,
                unsigned int* counter, NormResult* d_res, NormResult* h_res_dev,
                void* stream, double grad_scale, const TensorSegs* segs, int32_t g_dtype,
                bool tail)
{
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    switch (g_dtype) {
    case kDtypeBF16:  // 8-byte alignment checked by the caller
        launch_norm_typed<__nv_bfloat16, true>(g, n, clip, partials, counter, d_res, h_res_dev,
                                               s, grad_scale, segs, tail);
        break;
    case kDtypeF16:
        launch_norm_typed<__half, true>(g, n, clip, partials, counter, d_res, h_res_dev, s,
                                        grad_scale, segs, tail);
        break;
    default:
        if (detail::aligned16(g))
            launch_norm_typed<float, true>(g, n, clip, partials, counter, d_res, h_res_dev, s,
                                           grad_scale, segs, tail);
        else
            launch_norm_typed<float, false>(g, n, clip, partials, counter, d_res, h_res_dev, s,
                                            grad_scale, segs, tail);
    }
    return int(cudaGetLastError());
}

int norm_node_params(NormNodeArgs* a, cudaKernelNodeParams* p)
{
    a->ptrs[0] = &a->g;
    a->ptrs[1] = &a->n;
    a->ptrs[2] = &a->clip;
    a->ptrs[3] = &a->grad_scale;
    a->ptrs[4] = &a->partials;
    a->ptrs[5] = &a->counter;
    a->ptrs[6] = &a->d_res;
    a->ptrs[7] = &a->h_res;
    a->segs = TensorSegs{nullptr, nullptr, nullptr, nullptr};
    a->ptrs[8] = &a->segs;
    // without the last block: the fused node finishes the reduction
    p->func = detail::aligned16(a->g)
                  ? reinterpret_cast<void*>(&k_grad_norm<true, false, float, false>)
                  : reinterpret_cast<void*>(&k_grad_norm<false, false, float, false>);
    p->gridDim = dim3(unsigned(norm_blocks(a->n)));
    p->blockDim = dim3(kNormThreads);
    p->sharedMemBytes = 0;
    p->kernelParams = a->ptrs;
    p->extra = nullptr;
    return 0;
}

}  // namespace osr
