// graph.cu -- one optimizer step as a CUDA graph (norm kernel node, then the
// fused clip+AdamW node; for states the one-launch step serves, that step as
// one node: a cluster, or a cooperative grid) for states small enough that launch latency
// dominates.  The per-step scalars (bias corrections depend on t) are kernel
// arguments, so each step rewrites the two nodes' parameters in the
// instantiated graph (cudaGraphExecKernelNodeSetParams, which leaves launches
// already in flight untouched) and launches it once.
#include <cmath>
#include <cstdint>

#include <cuda_runtime.h>

#include "context.h"
#include "internal.h"

namespace osr {

void graph_release(adamw_ctx* c)
{
    if (c->graph_exec)
        cudaGraphExecDestroy(c->graph_exec);
    if (c->graph)
        cudaGraphDestroy(c->graph);
    c->graph_exec = nullptr;
    c->graph = nullptr;
    c->graph_norm = c->graph_step = nullptr;
    c->graph_w = c->graph_m = c->graph_v = nullptr;
    c->graph_g = nullptr;
}

namespace {

void fill_args(const adamw_ctx* c, double clip, const StepScalars& k, NormNodeArgs* na,
               AdamwNodeArgs* aa, cudaKernelNodeParams* np, cudaKernelNodeParams* ap)
{
    na->g = c->graph_g;
    na->n = c->n;
    na->clip = clip;
    na->grad_scale = 1.0;
    na->partials = c->d_partials;
    na->counter = c->d_counter;
    na->d_res = c->d_res;
    na->h_res = c->h_res_dev;
    norm_node_params(na, np);
    aa->w = c->graph_w;
    aa->g = c->graph_g;
    aa->m = c->graph_m;
    aa->v = c->graph_v;
    aa->n = c->n;
    aa->k = k;
    // the norm node leaves its partials: the fused node sums them
    aa->k.fin = NormFinish{c->d_partials, norm_blocks(c->n), clip, 1.0, c->d_res, c->h_res_dev};
    aa->d_res = nullptr;
    adamw_node_params(aa, c->caps, ap);
}

int cuda_fail(cudaError_t e, const char* what)
{
    return fail(ADAMW_ECUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Whether the graph takes the one-launch step -- the rule adamw_clip_step
// follows when its stream is being captured: the one-launch node only in its
// cluster form (up to 65,536 parameters), since in a graph, with no launch
// overhead to save, the two-node step costs less GPU time than the
// cooperative grid above that size.  The barrier-timeout test flag asks for
// the grid (its next graph step rebuilds the graph).
bool want_onepass(const adamw_ctx* c)
{
    return c->onepass && c->n <= c->onepass_max_n &&
           (onepass_is_cluster(c->n) || c->onepass_fault_test) &&
           onepass_grid(c->n, c->onepass_capacity) <= c->onepass_capacity &&
           aligned16(c->graph_w) && aligned16(c->graph_g) && aligned16(c->graph_m) &&
           aligned16(c->graph_v);
}

void fill_onepass(const adamw_ctx* c, double clip, const StepScalars& k, bool fault_test,
                  OnepassNodeArgs* a, cudaKernelNodeParams* p)
{
    a->w = c->graph_w;
    a->g = const_cast<float*>(c->graph_g);
    a->m = c->graph_m;
    a->v = c->graph_v;
    a->n = c->n;
    a->k = k;
    a->clip = clip;
    a->grad_scale = 1.0;
    a->partials = c->d_partials;
    a->bar = c->d_bar;
    a->d_res = c->d_res;
    a->h_res = c->h_res_dev;
    onepass_node_params(a, c->onepass_capacity, fault_test, p);
}

// Builds and instantiates the two-node graph over the context's graph_*
// pointers.  The fused node's kernel variant depends on whether decay flags
// are set (an instantiated node cannot change its function), so the graph
// remembers that and is rebuilt when it changes.
int graph_build(adamw_ctx* ctx)
{
    if (want_onepass(ctx)) {
        OnepassNodeArgs oa;
        cudaKernelNodeParams op{};
        fill_onepass(ctx, INFINITY, make_step_scalars(ctx, 1, 0.0, 0.0), false, &oa, &op);
        cudaLaunchAttributeValue coop{};
        coop.cooperative = 1;
        cudaError_t e;
        int rc = ADAMW_OK;
        if ((e = cudaGraphCreate(&ctx->graph, 0)) != cudaSuccess)
            rc = cuda_fail(e, "cudaGraphCreate");
        else if ((e = cudaGraphAddKernelNode(&ctx->graph_norm, ctx->graph, nullptr, 0, &op)) !=
                 cudaSuccess)
            rc = cuda_fail(e, "cudaGraphAddKernelNode(one-launch step)");
        else if (!onepass_is_cluster(ctx->n) &&  // a cluster node needs no attribute
                 (e = cudaGraphKernelNodeSetAttribute(ctx->graph_norm,
                                                      cudaLaunchAttributeCooperative, &coop)) !=
                     cudaSuccess)
            rc = cuda_fail(e, "cudaGraphKernelNodeSetAttribute(cooperative)");
        else if ((e = cudaGraphInstantiate(&ctx->graph_exec, ctx->graph, 0)) != cudaSuccess)
            rc = cuda_fail(e, "cudaGraphInstantiate");
        if (rc != ADAMW_OK) {
            graph_release(ctx);
        } else {
            ctx->graph_mask = ctx->decay_mask_on;
            ctx->graph_onepass = true;
        }
        return rc;
    }
    ctx->graph_onepass = false;
    NormNodeArgs na;
    AdamwNodeArgs aa;
    cudaKernelNodeParams np{}, ap{};
    fill_args(ctx, INFINITY, make_step_scalars(ctx, 1, 0.0, 0.0), &na, &aa, &np, &ap);
    cudaError_t e;
    int rc = ADAMW_OK;
    if ((e = cudaGraphCreate(&ctx->graph, 0)) != cudaSuccess)
        rc = cuda_fail(e, "cudaGraphCreate");
    else if ((e = cudaGraphAddKernelNode(&ctx->graph_norm, ctx->graph, nullptr, 0, &np)) !=
             cudaSuccess)
        rc = cuda_fail(e, "cudaGraphAddKernelNode(norm)");
    else if ((e = cudaGraphAddKernelNode(&ctx->graph_step, ctx->graph, &ctx->graph_norm, 1,
                                         &ap)) != cudaSuccess)
        rc = cuda_fail(e, "cudaGraphAddKernelNode(step)");
    else if ((e = cudaGraphInstantiate(&ctx->graph_exec, ctx->graph, 0)) != cudaSuccess)
        rc = cuda_fail(e, "cudaGraphInstantiate");
    if (rc != ADAMW_OK)
        graph_release(ctx);
    else
        ctx->graph_mask = ctx->decay_mask_on;
    return rc;
}

}  // namespace
}  // namespace osr

extern "C" {

int adamw_graph_create(adamw_ctx* ctx, float* d_w, const float* d_g, float* d_m, float* d_v)
{
    using osr::fail;
    osr::clear_error();
    if (!ctx)
        return fail(ADAMW_EINVAL, "ctx is NULL");
    const void* ptrs[4] = {d_w, d_g, d_m, d_v};
    for (const void* p : ptrs)
        if (!p || (reinterpret_cast<uintptr_t>(p) & 3u))
            return fail(ADAMW_EINVAL, "adamw_graph_create: null or unaligned state pointer");
    int prev = -1;
    cudaGetDevice(&prev);
    if (prev != ctx->device)
        cudaSetDevice(ctx->device);
    osr::graph_release(ctx);
    ctx->graph_w = d_w;
    ctx->graph_g = d_g;
    ctx->graph_m = d_m;
    ctx->graph_v = d_v;
    const int rc = osr::graph_build(ctx);
    if (prev >= 0 && prev != ctx->device)
        cudaSetDevice(prev);
    return rc;
}

int adamw_graph_step(adamw_ctx* ctx, int32_t t, double lr, double wd, double clip, void* stream)
{
    using osr::fail;
    osr::clear_error();
    if (!ctx)
        return fail(ADAMW_EINVAL, "ctx is NULL");
    if (!ctx->graph_exec)
        return fail(ADAMW_ESTATE, "no step graph: call adamw_graph_create first");
    if (t < 1)
        return fail(ADAMW_EINVAL, "t=%d: the first update has t = 1", t);
    if (!(lr >= 0.0 && std::isfinite(lr)) || !(wd >= 0.0 && std::isfinite(wd)) || !(clip > 0.0))
        return fail(ADAMW_EINVAL, "need finite lr, wd >= 0 and clip > 0");
    int prev = -1;
    cudaGetDevice(&prev);
    if (prev != ctx->device)
        cudaSetDevice(ctx->device);
    int rc = ADAMW_OK;
    if (ctx->graph_mask != ctx->decay_mask_on || ctx->graph_onepass != osr::want_onepass(ctx)) {
        // decay flags set or cleared, or the one-launch option changed, since
        // the graph was built
        float* w = ctx->graph_w;
        const float* g = ctx->graph_g;
        float* m = ctx->graph_m;
        float* v = ctx->graph_v;
        osr::graph_release(ctx);
        ctx->graph_w = w;
        ctx->graph_g = g;
        ctx->graph_m = m;
        ctx->graph_v = v;
        rc = osr::graph_build(ctx);
        if (rc != ADAMW_OK) {
            if (prev >= 0 && prev != ctx->device)
                cudaSetDevice(prev);
            return rc;
        }
    }
    osr::NormNodeArgs na;
    osr::AdamwNodeArgs aa;
    osr::OnepassNodeArgs oa;
    cudaKernelNodeParams np{}, ap{};
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (ctx->graph_onepass) {
        const bool fault_test = ctx->onepass_fault_test;
        ctx->onepass_fault_test = false;
        osr::fill_onepass(ctx, clip, osr::make_step_scalars(ctx, t, lr, wd), fault_test, &oa,
                          &np);
        if ((e = cudaGraphExecKernelNodeSetParams(ctx->graph_exec, ctx->graph_norm, &np)) !=
            cudaSuccess)
            rc = osr::cuda_fail(e, "cudaGraphExecKernelNodeSetParams(one-launch step)");
    } else {
        osr::fill_args(ctx, clip, osr::make_step_scalars(ctx, t, lr, wd), &na, &aa, &np, &ap);
        if ((e = cudaGraphExecKernelNodeSetParams(ctx->graph_exec, ctx->graph_norm, &np)) !=
            cudaSuccess)
            rc = osr::cuda_fail(e, "cudaGraphExecKernelNodeSetParams(norm)");
        else if ((e = cudaGraphExecKernelNodeSetParams(ctx->graph_exec, ctx->graph_step, &ap)) !=
                 cudaSuccess)
            rc = osr::cuda_fail(e, "cudaGraphExecKernelNodeSetParams(step)");
    }
    if (rc == ADAMW_OK && (e = cudaGraphLaunch(ctx->graph_exec, s)) != cudaSuccess)
        rc = osr::cuda_fail(e, "cudaGraphLaunch");
    if (rc == ADAMW_OK)
        ctx->segs_launched = false;  // the graph's reduction writes no per-tensor sums
    if (rc == ADAMW_OK) {
        cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
        cudaStreamIsCapturing(s, &cap);
        if (cap == cudaStreamCaptureStatusNone) {
            if ((e = cudaEventRecord(ctx->ev_norm, s)) != cudaSuccess)
                rc = osr::cuda_fail(e, "cudaEventRecord");
            else
                ctx->norm_launched = true;
        }
    }
    if (prev >= 0 && prev != ctx->device)
        cudaSetDevice(prev);
    return rc;
}

int adamw_graph_destroy(adamw_ctx* ctx)
{
    osr::clear_error();
    if (!ctx)
        return osr::fail(ADAMW_EINVAL, "ctx is NULL");
    osr::graph_release(ctx);
    return ADAMW_OK;
}

}  // extern "C"
