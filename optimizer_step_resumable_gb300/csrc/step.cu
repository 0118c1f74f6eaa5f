// step.cu -- the fused clip-scale + AdamW pass (rows a3 and a4 of the step),
// for sm_103a.
//
// "Training as a Recoverable State Transition" (aihero.club), section "The
// Exact Targets of Clipping and AdamW": m = beta1 m + (1 - beta1) g,
// v = beta2 v + (1 - beta2) g^2, bias corrections 1 - beta^t, and the
// decoupled decay w (1 - lr wd) applied before subtracting
// lr m_hat / (sqrt(v_hat) + eps), for every parameter.  The clip factor is
// applied here to each gradient element as it is read, so the gradient is
// never rescaled in memory (the engine's k_grad_scale pass of "Grow a
// Language Model: Backprop" is folded in).  HBM-bound: 28 bytes per
// parameter (read w, g, m, v; write w, m, v).
#include <cstdint>
#include <type_traits>

#include <cuda_runtime.h>

#include "adamw_dev.cuh"
#include "common.cuh"
#include "internal.h"
#include "norm_dev.cuh"

namespace osr {
namespace {

using adamwdev::adamw_elem;
using adamwdev::decay_one;
using adamwdev::kStepThreads;
using adamwdev::kStepVec;

// Reads w, g, m, v once and writes w, m, v once (28 bytes per parameter
// with a float32 gradient).  The clip factor and the non-finite flag come
// from the norm kernel's result in device memory, so nothing returns to the
// host between kernels; with res == nullptr the factor is k.scale (the host
// computed it from a global sum of squares).  G is the gradient's element
// type (float, bfloat16, binary16; widened exactly).  kZero also writes 0
// into g after reading it ("zero_grads" for the next accumulation).  WL, if
// not void, is the type of a 16-bit copy of the new weights written to w_lp
// (rounded to nearest even) for the next forward pass.  kMask: k.decay_mask
// holds one decay flag per element, as decay_nibble reads it.
// With k.fin.partials set, the norm kernel before this one left only its
// per-block partial sums: every block adds them up here in the norm kernel's
// fixed order (normdev::sum_partials, the same bits in every block), takes
// the factor from the total, and block 0 publishes the result record.
// (at least 4 resident blocks per SM, the occupancy the launch is sized for,
// whichever variant runs)
template <bool kVec, bool kZero, typename G, typename WL, bool kMask>
__global__ void __launch_bounds__(kStepThreads, 4)
    k_clip_adamw(float* __restrict__ w, const G* __restrict__ g,
                 float* __restrict__ m, float* __restrict__ v, int64_t n,
                 StepScalars k, const NormResult* __restrict__ res, WL* __restrict__ w_lp)
{
    const uint32_t* __restrict__ decay_mask = k.decay_mask;
    // When launched right behind the norm kernel with programmatic
    // serialization, this grid may start while that kernel still runs: warm
    // L2 with this block's first chunk (inputs the norm kernel does not
    // write), then wait for the norm grid to finish before reading its
    // result.  Launched normally, the wait returns at once.
    static_assert(kStepThreads == kNormThreads, "the block sums the norm partials");
    if (kVec && (res || k.fin.partials)) {
        const int64_t i0 = int64_t(blockIdx.x) * kStepThreads * kStepVec + threadIdx.x;
        if ((i0 + (kStepVec - 1) * kStepThreads) < (n >> 2)) {
#pragma unroll
            for (int j = 0; j < kStepVec; ++j) {
                const int64_t e = (i0 + j * kStepThreads) << 2;
                asm volatile("prefetch.global.L2 [%0];" ::"l"(w + e));
                asm volatile("prefetch.global.L2 [%0];" ::"l"(g + e));
                asm volatile("prefetch.global.L2 [%0];" ::"l"(m + e));
                asm volatile("prefetch.global.L2 [%0];" ::"l"(v + e));
            }
        }
    }
    asm volatile("griddepcontrol.wait;" ::: "memory");
    float s = k.scale;
    if (k.fin.partials) {
        __shared__ float s_scale;
        __shared__ int s_skip;
        const double total = normdev::sum_partials(k.fin.partials, k.fin.nparts);
        if (threadIdx.x == 0) {
            // only block 0 publishes, so only it reads the record's sequence number
            const NormResult r = normdev::make_result(
                total, k.fin.clip, k.fin.grad_scale, blockIdx.x == 0 ? k.fin.d_res->seq + 1u : 0u);
            s_scale = r.scale;
            s_skip = r.nonfinite;
            if (blockIdx.x == 0)
                normdev::publish(r, k.fin.d_res, k.fin.h_res);
        }
        __syncthreads();
        if (s_skip)
            return;
        s = s_scale;
    } else if (res) {
        if (res->nonfinite)
            return;
        s = res->scale;
    }
    // written through the same restrict pointer it is read from
    G* const gw = const_cast<G*>(g);
    const int64_t gtid = int64_t(blockIdx.x) * kStepThreads + threadIdx.x;
    const int64_t stride = int64_t(gridDim.x) * kStepThreads;
    if constexpr (kVec) {
        adamwdev::vector_pass<kZero, G, WL, kMask>(w, g, m, v, n, s, k, w_lp);
    } else {  // float32 state at 4-byte boundaries, float32 gradient, no copy
        for (int64_t e = gtid; e < n; e += stride) {
            float W = __ldcs(w + e), M = __ldcs(m + e), V = __ldcs(v + e);
            adamw_elem(W, __ldcs(g + e), M, V, s, k, decay_one<kMask>(decay_mask, e, k));
            __stcs(w + e, W);
            __stcs(m + e, M);
            __stcs(v + e, V);
            if constexpr (kZero)
                __stcs(gw + e, 0.0f);
        }
    }
}

// Launches the fused kernel; with `programmatic`, as a programmatic
// dependent of the kernel before it in the stream (that kernel must be the
// norm reduction, whose blocks release it early).
template <bool kVec, bool kZero, typename G, typename WL, bool kMask>
void launch_step(int blocks, cudaStream_t s, bool programmatic, float* w, const void* g,
                 float* m, float* v, int64_t n, const StepScalars& k, const NormResult* d_res,
                 void* w_lp)
{
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(unsigned(blocks));
    cfg.blockDim = dim3(kStepThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = programmatic ? 1 : 0;
    // status: cudaGetLastError in the caller
    cudaLaunchKernelEx(&cfg, &k_clip_adamw<kVec, kZero, G, WL, kMask>, w,
                       static_cast<const G*>(g), m, v, n, k, d_res, static_cast<WL*>(w_lp));
}

template <bool kZero, typename G, bool kMask>
void launch_vec(int blocks, cudaStream_t s, bool pdl, float* w, const void* g, float* m,
                float* v, int64_t n, const StepScalars& k, const NormResult* d_res, void* w_lp,
                int32_t w_lp_dtype)
{
    if (!w_lp)
        launch_step<true, kZero, G, void, kMask>(blocks, s, pdl, w, g, m, v, n, k, d_res, w_lp);
    else if (w_lp_dtype == kDtypeF16)
        launch_step<true, kZero, G, __half, kMask>(blocks, s, pdl, w, g, m, v, n, k, d_res,
                                                   w_lp);
    else
        launch_step<true, kZero, G, __nv_bfloat16, kMask>(blocks, s, pdl, w, g, m, v, n, k,
                                                          d_res, w_lp);
}

template <bool kZero, bool kMask>
void launch_vec_any(int32_t g_dtype, int blocks, cudaStream_t s, bool pdl, float* w,
                    const void* g, float* m, float* v, int64_t n, const StepScalars& k,
                    const NormResult* d_res, void* w_lp, int32_t w_lp_dtype)
{
    if (g_dtype == kDtypeBF16)
        launch_vec<kZero, __nv_bfloat16, kMask>(blocks, s, pdl, w, g, m, v, n, k, d_res, w_lp,
                                                w_lp_dtype);
    else if (g_dtype == kDtypeF16)
        launch_vec<kZero, __half, kMask>(blocks, s, pdl, w, g, m, v, n, k, d_res, w_lp,
                                         w_lp_dtype);
    else
        launch_vec<kZero, float, kMask>(blocks, s, pdl, w, g, m, v, n, k, d_res, w_lp,
                                        w_lp_dtype);
}

template <bool kMask>
void launch_any(bool vec, bool zero_grad, int32_t g_dtype, int blocks, cudaStream_t s,
                bool pdl, float* w, const void* g, float* m, float* v, int64_t n,
                const StepScalars& k, const NormResult* d_res, void* w_lp, int32_t w_lp_dtype)
{
    if (vec) {
        if (zero_grad)
            launch_vec_any<true, kMask>(g_dtype, blocks, s, pdl, w, g, m, v, n, k, d_res, w_lp,
                                        w_lp_dtype);
        else
            launch_vec_any<false, kMask>(g_dtype, blocks, s, pdl, w, g, m, v, n, k, d_res,
                                         w_lp, w_lp_dtype);
    } else if (zero_grad) {
        launch_step<false, true, float, void, kMask>(blocks, s, pdl, w, g, m, v, n, k, d_res,
                                                     nullptr);
    } else {
        launch_step<false, false, float, void, kMask>(blocks, s, pdl, w, g, m, v, n, k, d_res,
                                                      nullptr);
    }
}

}  // namespace

int query_step_caps(int sm_count, KernelCaps* caps)
{
    // the other variants have the same shape and the same register budget
    cudaError_t err = cudaSuccess;
    caps->step_vec = detail::resident_blocks(
        reinterpret_cast<const void*>(&k_clip_adamw<true, false, float, void, false>),
        kStepThreads, sm_count, &err);
    caps->step_scalar = detail::resident_blocks(
        reinterpret_cast<const void*>(&k_clip_adamw<false, false, float, void, false>),
        kStepThreads, sm_count, &err);
    return int(err);
}

int launch_adamw(float* w, const void* g, float* m, float* v, int64_t n,
                 const StepScalars& k, const NormResult* d_res, const KernelCaps& caps,
                 void* stream, bool zero_grad, bool programmatic, int32_t g_dtype, void* w_lp,
                 int32_t w_lp_dtype)
{
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const bool plain = g_dtype == kDtypeF32 && !w_lp;
    const bool vec = detail::aligned16(w) && detail::aligned16(m) && detail::aligned16(v) &&
                     (g_dtype == kDtypeF32 ? detail::aligned16(g) : detail::aligned8(g)) &&
                     (!w_lp || detail::aligned8(w_lp));
    if (!vec && !plain)
        return int(cudaErrorMisalignedAddress);  // callers refuse this before launching
    const int cap = vec ? caps.step_vec : caps.step_scalar;
    const int64_t want = vec ? detail::ceil_div(n >> 2, int64_t(kStepThreads) * kStepVec)
                             : detail::ceil_div(n, kStepThreads);
    const int blocks = int(want < 1 ? 1 : (want > cap ? cap : want));
    if (k.decay_mask)
        launch_any<true>(vec, zero_grad, g_dtype, blocks, s, programmatic, w, g, m, v, n, k,
                         d_res, w_lp, w_lp_dtype);
    else
        launch_any<false>(vec, zero_grad, g_dtype, blocks, s, programmatic, w, g, m, v, n, k,
                          d_res, w_lp, w_lp_dtype);
    return int(cudaGetLastError());
}

int adamw_node_params(AdamwNodeArgs* a, const KernelCaps& caps, cudaKernelNodeParams* p)
{
    a->ptrs[0] = &a->w;
    a->ptrs[1] = &a->g;
    a->ptrs[2] = &a->m;
    a->ptrs[3] = &a->v;
    a->ptrs[4] = &a->n;
    a->ptrs[5] = &a->k;
    a->ptrs[6] = &a->d_res;
    a->w_lp = nullptr;
    a->ptrs[7] = &a->w_lp;
    const bool vec = detail::aligned16(a->w) && detail::aligned16(a->g) &&
                     detail::aligned16(a->m) && detail::aligned16(a->v);
    int64_t want;
    int cap;
    const bool mask = a->k.decay_mask != nullptr;
    if (vec) {
        p->func = mask ? reinterpret_cast<void*>(&k_clip_adamw<true, false, float, void, true>)
                       : reinterpret_cast<void*>(&k_clip_adamw<true, false, float, void, false>);
        want = detail::ceil_div(a->n >> 2, int64_t(kStepThreads) * kStepVec);
        cap = caps.step_vec;
    } else {
        p->func = mask ? reinterpret_cast<void*>(&k_clip_adamw<false, false, float, void, true>)
                       : reinterpret_cast<void*>(&k_clip_adamw<false, false, float, void, false>);
        want = detail::ceil_div(a->n, kStepThreads);
        cap = caps.step_scalar;
    }
    p->gridDim = dim3(unsigned(want < 1 ? 1 : (want > cap ? cap : want)));
    p->blockDim = dim3(kStepThreads);
    p->sharedMemBytes = 0;
    p->kernelParams = a->ptrs;
    p->extra = nullptr;
    return 0;
}

}  // namespace osr
