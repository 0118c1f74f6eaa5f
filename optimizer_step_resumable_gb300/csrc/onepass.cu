// onepass.cu -- the whole optimizer step (global norm, clip factor, fused
// clip + AdamW) in one cooperative launch, for states small enough that the
// fixed cost of two launches dominates the step.
//
// "Training as a Recoverable State Transition" (aihero.club), section "The
// Exact Targets of Clipping and AdamW": the norm of the joined gradient, the
// clip factor, then the AdamW update of every parameter.  "Grow a Language
// Model: Backprop" (unhomeschool.com) counts about a hundred launches per
// training step as the engine's overhead; for a small state the optimizer's
// share shrinks from two launches to one here.
//
// Blocks 0 .. P-1 (P = norm_blocks(n)) compute exactly the partial sums of
// the norm kernel (same tiles, same loads, same run sums, same block tree),
// every block then waits at a grid barrier, sums the P partials in the norm
// kernel's fixed order (so every block holds the same bits of the norm and
// the clip factor as the two-launch step), and the grid runs the same vector
// pass as the fused kernel.  The results are bit-identical to the two-launch
// step.  The grid is launched cooperatively, so all its blocks are resident
// at once and the barrier is always reached; each wait is still bounded
// (about a second) and a block that gives up sets the result record's fault
// word, skips the update and leaves; the host reports the fault.
//
// States whose norm partition has at most 8 blocks (n <= 65,536) run the
// same two phases in thread-block clusters of 8 CTAs instead: every cluster
// computes all P partials itself (CTA r of the cluster the norm kernel's
// block r, into the cluster's own slots) and meets at its hardware barrier
// (release / acquire at cluster scope), so no block waits for another
// cluster: no cooperative launch, no counter, no wait to bound.  The
// clusters then share the update.  Same partials, same order, same bits.
#include <cstdint>

#include <cuda_runtime.h>

#include "adamw_dev.cuh"
#include "common.cuh"
#include "internal.h"
#include "norm_dev.cuh"

namespace osr {
namespace {

constexpr uint64_t kBarrierWaitNs = 1000000000ull;  // one second
constexpr uint32_t kBarrierMaxPolls = 1u << 26;       // backstop on the poll count

__device__ __forceinline__ uint64_t global_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ uint32_t load_acquire(const uint32_t* p)
{
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Polls *count until it reaches target; false if the wait ran out.
__device__ bool wait_for_count(const uint32_t* count, uint32_t target)
{
    const uint64_t t0 = global_ns();
    for (uint32_t poll = 0; poll < kBarrierMaxPolls; ++poll) {
        if (load_acquire(count) >= target)
            return true;
        if (global_ns() - t0 > kBarrierWaitNs)
            return false;
        __nanosleep(poll < 32 ? 20 : 200);
    }
    return false;
}

// bar[0]: arrivals, bar[1]: departures (both 0 between launches: the last
// block to leave resets them).  expect: the arrivals to wait for -- gridDim.x,
// or more to exercise the timeout.
template <bool kZero, bool kMask>
__global__ void __launch_bounds__(kNormThreads, 4)
    k_clip_adamw_onepass(float* __restrict__ w, float* __restrict__ g, float* __restrict__ m,
                         float* __restrict__ v, int64_t n, StepScalars k, double clip,
                         double grad_scale, double* __restrict__ partials, int32_t P,
                         uint32_t* __restrict__ bar,
                         uint32_t expect, NormResult* __restrict__ d_res, NormResult* h_res)
{
    static_assert(adamwdev::kStepThreads == kNormThreads, "one block shape for both phases");
    constexpr int U = kNormVecPerThread;
    const int tid = threadIdx.x;
    __shared__ int s_ok, s_skip;
    __shared__ float s_scale;

    // Level 1 (blocks < P): this block's partial sum, as the norm kernel
    // computes it.
    if (int(blockIdx.x) < P) {
        const int64_t ntiles = (n + kNormTileElems - 1) / kNormTileElems;
        const int64_t nfull = n / kNormTileElems;
        const int64_t t_lo = ntiles * int64_t(blockIdx.x) / int64_t(P);
        const int64_t t_hi = ntiles * int64_t(blockIdx.x + 1) / int64_t(P);
        double acc = 0.0;
        for (int64_t tile = t_lo; tile < t_hi; ++tile) {
            float4 x[U];
            normdev::load_tile<U, true, float>(g, n, nfull, tile, tid, x);
            acc += normdev::run_sumsq<U>(x);
        }
        acc = detail::block_sum<kNormThreads>(acc);
        if (tid == 0)
            partials[blockIdx.x] = acc;
    }

    // Grid barrier: every block's partial is written before any block reads.
    if (tid == 0) {
        __threadfence();
        atomicAdd(&bar[0], 1u);
        s_ok = wait_for_count(&bar[0], expect) ? 1 : 0;
        __threadfence();
    }
    __syncthreads();
    const bool ok = s_ok != 0;

    // Level 2: every block sums the partials in the norm kernel's order.
    if (ok) {
        const double s = normdev::sum_partials(partials, P);
        if (tid == 0) {
            // only block 0 publishes, so only it reads the record's sequence number
            const NormResult r = normdev::make_result(
                s, clip, grad_scale, blockIdx.x == 0 ? d_res->seq + 1u : 0u);
            s_scale = r.scale;
            s_skip = r.nonfinite;
            if (blockIdx.x == 0)
                normdev::publish(r, d_res, h_res);
        }
    } else if (tid == 0 && h_res) {  // the host reads the fault from its mirror
        volatile NormResult* h = h_res;  // (after the grid completes: no fence)
        h->fault = 1u;
    }
    __syncthreads();
    // Leave the barrier; the last block out resets it for the next launch.
    // (Every block has finished polling bar[0] before it counts itself out.)
    if (tid == 0) {
        const uint32_t out = atomicAdd(&bar[1], 1u);
        if (out == gridDim.x - 1) {
            atomicExch(&bar[0], 0u);
            atomicExch(&bar[1], 0u);
        }
    }
    if (!ok || s_skip)
        return;
    adamwdev::vector_pass<kZero, float, void, kMask>(w, g, m, v, n, s_scale, k, nullptr);
}

// Clusters enough for one chunk of the update per CTA (whole clusters; at
// most 4 for n <= kClusterMaxN, so the slots fit the partials scratch).
int cluster_grid(int64_t n)
{
    const int64_t chunk = int64_t(adamwdev::kStepThreads) * adamwdev::kStepVec;
    const int64_t want = detail::ceil_div(n >> 2, chunk);
    const int64_t clusters = detail::ceil_div(want < 1 ? 1 : want, int64_t(kClusterCtas));
    return int(clusters) * kClusterCtas;
}
static_assert(((kClusterMaxN >> 2) + int64_t(adamwdev::kStepThreads) * adamwdev::kStepVec - 1) /
                      (int64_t(adamwdev::kStepThreads) * adamwdev::kStepVec) +
                  kClusterCtas <=
                  kNormBlocksMax,
              "every cluster's partial slots fit the partials scratch");

// The step of a state of at most kClusterMaxN parameters in clusters of
// kClusterCtas CTAs.  Arguments as k_clip_adamw_onepass (bar and expect are
// not used), so the graph node takes either kernel with one argument list;
// cluster c keeps its partials in partials[c * kClusterCtas ...].  Every
// cluster reads all of g for its norm, so the gradient is never zeroed here
// (a cluster could still be reading what another has updated): zero_grad
// steps take the grid form.  The grid has at least n / 8 threads, so each
// thread owns at most kStepVec float4 of the state (float4 index gtid + j *
// stride) and one of the last n % 4 elements; it loads them before the
// barrier, which hides their latency behind the norm.
template <bool kMask>
__global__ void __cluster_dims__(kClusterCtas, 1, 1) __launch_bounds__(kNormThreads)
    k_clip_adamw_cluster(float* __restrict__ w, float* __restrict__ g, float* __restrict__ m,
                         float* __restrict__ v, int64_t n, StepScalars k, double clip,
                         double grad_scale, double* __restrict__ partials, int32_t P,
                         uint32_t* __restrict__ bar, uint32_t expect,
                         NormResult* __restrict__ d_res, NormResult* h_res)
{
    constexpr int U = kNormVecPerThread;
    constexpr int J = adamwdev::kStepVec;
    const int tid = threadIdx.x;
    __shared__ int s_skip;
    __shared__ float s_scale;
    // this thread's part of the update, loaded first
    const int64_t n4 = n >> 2;
    const int64_t gtid = int64_t(blockIdx.x) * kNormThreads + tid;
    const int64_t stride = int64_t(gridDim.x) * kNormThreads;
    float4* w4 = reinterpret_cast<float4*>(w);
    float4* m4 = reinterpret_cast<float4*>(m);
    float4* v4 = reinterpret_cast<float4*>(v);
    const float4* g4 = reinterpret_cast<const float4*>(g);
    float4 W[J], G[J], M[J], V[J];
    uint32_t D[J];
#pragma unroll
    for (int j = 0; j < J; ++j) {
        const int64_t i = gtid + j * stride;
        if (i < n4) {
            W[j] = __ldcs(w4 + i);
            G[j] = __ldcs(g4 + i);
            M[j] = __ldcs(m4 + i);
            V[j] = __ldcs(v4 + i);
            D[j] = adamwdev::decay_nibble<kMask>(k.decay_mask, i);
        }
    }
    const int64_t e_tail = (n4 << 2) + gtid;  // one of the last n % 4 elements
    const bool has_tail = e_tail < n;
    float tw = 0.f, tg = 0.f, tm = 0.f, tv = 0.f;
    if (has_tail) {
        tw = w[e_tail];
        tg = g[e_tail];
        tm = m[e_tail];
        tv = v[e_tail];
    }

    const int rank = int(blockIdx.x) % kClusterCtas;  // clusters: consecutive blocks
    double* const mine = partials + (int(blockIdx.x) - rank);
    if (rank < P) {  // this CTA's partial, as the norm kernel's block `rank`
        const int64_t ntiles = (n + kNormTileElems - 1) / kNormTileElems;
        const int64_t nfull = n / kNormTileElems;
        const int64_t t_lo = ntiles * int64_t(rank) / int64_t(P);
        const int64_t t_hi = ntiles * int64_t(rank + 1) / int64_t(P);
        double acc = 0.0;
        for (int64_t tile = t_lo; tile < t_hi; ++tile) {
            float4 x[U];
            normdev::load_tile<U, true, float>(g, n, nfull, tile, tid, x);
            acc += normdev::run_sumsq<U>(x);
        }
        acc = detail::block_sum<kNormThreads>(acc);
        if (tid == 0)
            mine[rank] = acc;
    }
    // Every thread of the cluster arrives (release: the partials written
    // before) and waits (acquire: all of them visible after).
    asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
    const double s = normdev::sum_partials(mine, P);
    if (tid == 0) {
        // only block 0 publishes, so only it reads the record's sequence number
        const NormResult r =
            normdev::make_result(s, clip, grad_scale, blockIdx.x == 0 ? d_res->seq + 1u : 0u);
        s_scale = r.scale;
        s_skip = r.nonfinite;
        if (blockIdx.x == 0)
            normdev::publish(r, d_res, h_res);
    }
    __syncthreads();
    if (s_skip)
        return;
    const float sc = s_scale;
#pragma unroll
    for (int j = 0; j < J; ++j) {
        const int64_t i = gtid + j * stride;
        if (i < n4) {
            adamwdev::adamw4(W[j], G[j], M[j], V[j], sc, k, D[j]);
            __stcs(w4 + i, W[j]);
            __stcs(m4 + i, M[j]);
            __stcs(v4 + i, V[j]);
        }
    }
    if (has_tail) {
        adamwdev::adamw_elem(tw, tg, tm, tv, sc, k,
                             adamwdev::decay_one<kMask>(k.decay_mask, e_tail, k));
        w[e_tail] = tw;
        m[e_tail] = tm;
        v[e_tail] = tv;
    }
}

template <bool kMask>
int launch_cluster_typed(cudaStream_t s, float* w, float* g, float* m, float* v, int64_t n,
                         const StepScalars& k, double clip, double grad_scale, double* partials,
                         NormResult* d_res, NormResult* h_res)
{
    const int32_t P = norm_blocks(n);
    k_clip_adamw_cluster<kMask><<<cluster_grid(n), kNormThreads, 0, s>>>(
        w, g, m, v, n, k, clip, grad_scale, partials, P, nullptr, 0u, d_res, h_res);
    return int(cudaGetLastError());
}

template <bool kZero, bool kMask>
int launch_typed(int blocks, cudaStream_t s, float* w, float* g, float* m, float* v, int64_t n,
                 const StepScalars& k, double clip, double grad_scale, double* partials,
                 uint32_t* bar, uint32_t expect, NormResult* d_res, NormResult* h_res)
{
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(unsigned(blocks));
    cfg.blockDim = dim3(kNormThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const int32_t P = norm_blocks(n);
    return int(cudaLaunchKernelEx(&cfg, &k_clip_adamw_onepass<kZero, kMask>, w, g, m, v, n, k,
                                  clip, grad_scale, partials, P, bar, expect, d_res, h_res));
}

}  // namespace

bool onepass_is_cluster(int64_t n) { return n <= kClusterMaxN; }

int query_onepass_blocks(int sm_count, int* blocks_out)
{
    cudaError_t err = cudaSuccess;
    int least = 1 << 30;
    const void* fns[4] = {reinterpret_cast<const void*>(&k_clip_adamw_onepass<false, false>),
                          reinterpret_cast<const void*>(&k_clip_adamw_onepass<true, false>),
                          reinterpret_cast<const void*>(&k_clip_adamw_onepass<false, true>),
                          reinterpret_cast<const void*>(&k_clip_adamw_onepass<true, true>)};
    for (const void* f : fns) {
        const int r = detail::resident_blocks(f, kNormThreads, sm_count, &err);
        least = r < least ? r : least;
    }
    *blocks_out = least;
    return int(err);
}

int onepass_grid(int64_t n, int capacity)
{
    // enough blocks for the norm's partition and for one chunk of the vector
    // pass each, no more than can be resident at once
    const int P = norm_blocks(n);
    const int64_t chunk = int64_t(adamwdev::kStepThreads) * adamwdev::kStepVec;
    const int64_t want = detail::ceil_div(n >> 2, chunk);
    int blocks = int(want > P ? (want < capacity ? want : capacity) : P);
    return blocks > P ? blocks : P;
}

int onepass_node_params(OnepassNodeArgs* a, int capacity, bool fault_test,
                        cudaKernelNodeParams* p)
{
    const int blocks = onepass_grid(a->n, capacity);
    a->P = norm_blocks(a->n);
    a->expect = uint32_t(blocks) + (fault_test ? 1u : 0u);
    void** q = a->ptrs;
    q[0] = &a->w;
    q[1] = &a->g;
    q[2] = &a->m;
    q[3] = &a->v;
    q[4] = &a->n;
    q[5] = &a->k;
    q[6] = &a->clip;
    q[7] = &a->grad_scale;
    q[8] = &a->partials;
    q[9] = &a->P;
    q[10] = &a->bar;
    q[11] = &a->expect;
    q[12] = &a->d_res;
    q[13] = &a->h_res;
    if (onepass_is_cluster(a->n)) {  // no barrier to time out: fault_test does not apply
        a->expect = 0u;
        p->func = a->k.decay_mask ? reinterpret_cast<void*>(&k_clip_adamw_cluster<true>)
                                  : reinterpret_cast<void*>(&k_clip_adamw_cluster<false>);
        p->gridDim = dim3(unsigned(cluster_grid(a->n)));
        p->blockDim = dim3(kNormThreads);
        p->sharedMemBytes = 0;
        p->kernelParams = a->ptrs;
        p->extra = nullptr;
        return 0;
    }
    p->func = a->k.decay_mask ? reinterpret_cast<void*>(&k_clip_adamw_onepass<false, true>)
                              : reinterpret_cast<void*>(&k_clip_adamw_onepass<false, false>);
    p->gridDim = dim3(unsigned(blocks));
    p->blockDim = dim3(kNormThreads);
    p->sharedMemBytes = 0;
    p->kernelParams = a->ptrs;
    p->extra = nullptr;
    return blocks <= capacity ? 0 : int(cudaErrorCooperativeLaunchTooLarge);
}

int launch_onepass(float* w, float* g, float* m, float* v, int64_t n, const StepScalars& k,
                   double clip, double grad_scale, double* partials, uint32_t* bar,
                   bool fault_test, NormResult* d_res, NormResult* h_res, int capacity,
                   bool zero_grad, void* stream)
{
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const bool mask = k.decay_mask != nullptr;
    // the cluster form unless the gradient is zeroed or the timeout is tested
    if (onepass_is_cluster(n) && !zero_grad && !fault_test)
        return mask ? launch_cluster_typed<true>(s, w, g, m, v, n, k, clip, grad_scale, partials,
                                                 d_res, h_res)
                    : launch_cluster_typed<false>(s, w, g, m, v, n, k, clip, grad_scale,
                                                  partials, d_res, h_res);
    const int blocks = onepass_grid(n, capacity);
    if (blocks > capacity)
        return int(cudaErrorCooperativeLaunchTooLarge);  // callers check first
    const uint32_t expect = uint32_t(blocks) + (fault_test ? 1u : 0u);
    if (zero_grad)
        return mask ? launch_typed<true, true>(blocks, s, w, g, m, v, n, k, clip, grad_scale,
                                               partials, bar, expect, d_res, h_res)
                    : launch_typed<true, false>(blocks, s, w, g, m, v, n, k, clip, grad_scale,
                                                partials, bar, expect, d_res, h_res);
    return mask ? launch_typed<false, true>(blocks, s, w, g, m, v, n, k, clip, grad_scale,
                                            partials, bar, expect, d_res, h_res)
                : launch_typed<false, false>(blocks, s, w, g, m, v, n, k, clip, grad_scale,
                                             partials, bar, expect, d_res, h_res);
}

}  // namespace osr
