// ranks.cu -- the global clip factor of a sharded state from the ranks'
// gathered sums of squares, on the device.
//
// "Training as a Recoverable State Transition" (aihero.club), section "The
// Exact Targets of Clipping and AdamW": the clip uses the norm of all
// gradients joined into one vector.  With the state sharded over ranks
// ("Checkpoint and Sharded Resume", AI Engineering from Scratch, lesson 80:
// each rank holds a contiguous shard of the parameters), each rank reduces
// its shard, the ranks exchange one double each (an all-gather, issued by the
// caller on the device), and every rank adds them here in rank order -- the
// same order and the same formula as the host-side exchange, so the same
// bits, with no host round trip in the step.
#include <cstdint>

#include <cuda_runtime.h>

#include "common.cuh"
#include "internal.h"
#include "norm_dev.cuh"

namespace osr {
namespace {

// One thread: S = sum of rank_sumsq[0..world) in rank order; publishes the
// norm grad_scale sqrt(S), the factor and the non-finite flag as the norm
// kernel does, for the fused kernel that follows (a programmatic dependent).
__global__ void __launch_bounds__(32)
    k_rank_total(const double* __restrict__ rank_sumsq, int32_t world, double clip,
                 double grad_scale, NormResult* __restrict__ d_res, NormResult* h_res)
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (threadIdx.x != 0)
        return;
    double s = 0.0;
    for (int32_t r = 0; r < world; ++r)
        s += rank_sumsq[r];
    normdev::publish(normdev::make_result(s, clip, grad_scale, d_res->seq + 1u), d_res, h_res);
}

}  // namespace

int launch_rank_total(const double* rank_sumsq, int32_t world, double clip, double grad_scale,
                      NormResult* d_res, NormResult* h_res, void* stream)
{
    k_rank_total<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(rank_sumsq, world, clip,
                                                                  grad_scale, d_res, h_res);
    return int(cudaGetLastError());
}

}  // namespace osr
