// api.cu -- the C ABI entry points of include/adamw_ckpt.h: the context that
// owns all scratch, the host-side scalars, the launch sequence of one step,
// and the checkpoint pack / write / read around the staging images.
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <new>
#include <vector>

#include <cuda_runtime.h>
#include <unistd.h>

#include "context.h"
#include "internal.h"

namespace {

using osr::fail;

constexpr size_t kScratchHead = 256;  // NormResult + counter, padded

int cuda_fail(cudaError_t e, const char* what)
{
    return fail(ADAMW_ECUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

#define CUDA_TRY(expr)                                       \
    do {                                                     \
        cudaError_t e_ = (expr);                             \
        if (e_ != cudaSuccess) return cuda_fail(e_, #expr);  \
    } while (0)

// Makes ctx->device current for the scope of one call and restores the
// caller's device afterwards.
class DeviceScope {
public:
    explicit DeviceScope(int device)
    {
        if (cudaGetDevice(&prev_) != cudaSuccess)
            prev_ = -1;
        if (prev_ != device && cudaSetDevice(device) == cudaSuccess)
            switched_ = true;
    }
    ~DeviceScope()
    {
        if (switched_ && prev_ >= 0)
            cudaSetDevice(prev_);
    }

private:
    int prev_ = -1;
    bool switched_ = false;
};

bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_state_ptr(const void* p, const char* name)
{
    if (!p)
        return fail(ADAMW_EINVAL, "%s is NULL", name);
    if (!aligned4(p))
        return fail(ADAMW_EINVAL, "%s is not 4-byte aligned", name);
    return ADAMW_OK;
}

void free_ctx(adamw_ctx* c)
{
    if (!c)
        return;
    osr::writer_stop(c);
    osr::graph_release(c);
    if (c->device >= 0) {
        DeviceScope scope(c->device);
        if (c->ev_d2h && c->d2h_pending)
            cudaEventSynchronize(c->ev_d2h);
        if (c->ev_norm && c->norm_launched)
            cudaEventSynchronize(c->ev_norm);
        if (c->ev_norm) cudaEventDestroy(c->ev_norm);
        if (c->ev_pack) cudaEventDestroy(c->ev_pack);
        if (c->ev_d2h) cudaEventDestroy(c->ev_d2h);
        if (c->d_scratch) cudaFree(c->d_scratch);
        if (c->d_tab_offsets) cudaFree(c->d_tab_offsets);
        if (c->d_kfirst) cudaFree(c->d_kfirst);
        if (c->d_segbase) cudaFree(c->d_segbase);
        if (c->d_seg_sums) cudaFree(c->d_seg_sums);
        if (c->h_seg_sums) cudaFreeHost(c->h_seg_sums);
        if (c->h_res) cudaFreeHost(c->h_res);
        if (c->d_image_alloc) cudaFree(c->d_image_alloc);
        if (c->h_image_alloc) cudaFreeHost(c->h_image_alloc);
        if (c->d_decay_mask) cudaFree(c->d_decay_mask);
    }
    delete c;
}

int validate_table(int64_t n, const int64_t* offsets, const int64_t* numels, int32_t nt)
{
    if (n < 1 || n > INT32_MAX)
        return fail(ADAMW_EINVAL, "n_params=%lld outside [1, 2^31-1]", (long long)n);
    if (nt < 0)
        return fail(ADAMW_EINVAL, "n_tensors=%d is negative", nt);
    if (nt == 0) {
        if (offsets || numels)
            return fail(ADAMW_EINVAL, "n_tensors=0 needs NULL offsets and numels");
        return ADAMW_OK;
    }
    if (!offsets || !numels)
        return fail(ADAMW_EINVAL, "offset table is NULL");
    int64_t expect = 0;
    for (int32_t k = 0; k < nt; ++k) {
        if (numels[k] <= 0)
            return fail(ADAMW_EINVAL, "tensor %d has numel %lld", k, (long long)numels[k]);
        if (offsets[k] != expect)
            return fail(ADAMW_EINVAL,
                        "tensor %d starts at %lld, expected %lld (table must be sorted, "
                        "contiguous, without gaps or overlap)",
                        k, (long long)offsets[k], (long long)expect);
        if (numels[k] > n - expect)
            return fail(ADAMW_EINVAL, "tensor %d ends past n_params", k);
        expect += numels[k];
    }
    if (expect != n)
        return fail(ADAMW_EINVAL, "tensors cover %lld of %lld parameters", (long long)expect,
                    (long long)n);
    return ADAMW_OK;
}

// tail = false: the norm kernel leaves only its partials, and the fused
// kernel launched next finishes the reduction (osr::NormFinish).
int launch_norm_on(adamw_ctx* c, const void* g, double clip, void* stream,
                   double grad_scale = 1.0, bool tensor_sums = false,
                   int32_t g_dtype = ADAMW_DTYPE_F32, bool tail = true)
{
    const osr::TensorSegs segs{c->d_tab_offsets, c->d_kfirst, c->d_segbase, c->d_seg_sums};
    const int e = osr::launch_norm(g, c->n, clip, c->d_partials, c->d_counter, c->d_res,
                                   c->h_res_dev, stream, grad_scale,
                                   tensor_sums ? &segs : nullptr, g_dtype, tail);
    if (e != cudaSuccess)
        return cuda_fail(cudaError_t(e), "norm kernel launch");
    c->segs_launched = tensor_sums;
    return ADAMW_OK;
}

// Per-tensor sums from the segment slots of the last reduction, added in
// block order (deterministic).  Waits for that reduction.
int read_tensor_sums(adamw_ctx* c, double* out)
{
    if (!c->norm_launched || !c->segs_launched)
        return fail(ADAMW_ESTATE, "the last reduction did not compute per-tensor sums");
    CUDA_TRY(cudaEventSynchronize(c->ev_norm));
    CUDA_TRY(cudaMemcpy(c->h_seg_sums, c->d_seg_sums, sizeof(double) * size_t(c->nseg),
                        cudaMemcpyDeviceToHost));
    const size_t nt = c->offsets.size();
    for (size_t k = 0; k < nt; ++k)
        out[k] = 0.0;
    const int blocks = int(c->kfirst.size());
    for (int b = 0; b < blocks; ++b)
        for (int32_t s = c->segbase[size_t(b)]; s < c->segbase[size_t(b) + 1]; ++s)
            out[size_t(c->kfirst[size_t(b)] + (s - c->segbase[size_t(b)]))] += c->h_seg_sums[s];
    return ADAMW_OK;
}

// Marks the end of a reduction for adamw_last_norm.  Inside a stream
// capture the record would belong to the graph, not to a launch the host
// can wait for, so captured steps are not tracked.
int mark_norm(adamw_ctx* c, cudaStream_t st)
{
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    CUDA_TRY(cudaStreamIsCapturing(st, &cap));
    if (cap != cudaStreamCaptureStatusNone)
        return ADAMW_OK;
    CUDA_TRY(cudaEventRecord(c->ev_norm, st));
    c->norm_launched = true;
    return ADAMW_OK;
}

int read_norm(adamw_ctx* c, double* norm_out, float* scale_out)
{
    if (!c->norm_launched)
        return fail(ADAMW_ESTATE, "no norm reduction has run on this context");
    CUDA_TRY(cudaEventSynchronize(c->ev_norm));
    volatile osr::NormResult* r = c->h_res;
    if (r->fault) {
        r->fault = 0u;
        return fail(ADAMW_ECUDA,
                    "the one-launch step's grid barrier wait ran out: that step skipped its "
                    "update (w, m, v as before it)");
    }
    const double norm = r->norm;
    const float scale = r->scale;
    const int nonfinite = r->nonfinite;
    if (norm_out)
        *norm_out = norm;
    if (scale_out)
        *scale_out = scale;
    if (nonfinite)
        return fail(ADAMW_ENONFINITE, "gradient norm is %g: the update was skipped", norm);
    return ADAMW_OK;
}

}  // namespace

namespace osr {

StepScalars make_step_scalars(const adamw_ctx* c, int32_t t, double lr, double wd)
{
    // Bias-correction and decay scalars, in double on the host, rounded to
    // float once.
    const double bc1 = 1.0 - std::pow(c->beta1, double(t));
    const double bc2 = 1.0 - std::pow(c->beta2, double(t));
    StepScalars k;
    k.beta1 = float(c->beta1);
    k.omb1 = float(1.0 - c->beta1);
    k.beta2 = float(c->beta2);
    k.omb2 = float(1.0 - c->beta2);
    k.eps = float(c->eps);
    k.step_size = float(lr / bc1);
    k.inv_sqrt_bc2 = float(1.0 / std::sqrt(bc2));
    k.decay = float(1.0 - lr * wd);
    k.scale = 1.0f;
    k.decay_mask = c->decay_mask_on ? c->d_decay_mask : nullptr;
    k.chunk_ctr = (c->dynamic_chunks && c->n >= kDynamicChunksMinN) ? c->d_chunk_ctr : nullptr;
    k.fin = NormFinish{nullptr, 0, 0.0, 1.0, nullptr, nullptr};
    return k;
}

// Sets bits [lo, hi) of a bit array (bit e % 32 of word e / 32).
void set_bit_range(uint32_t* words, int64_t lo, int64_t hi)
{
    while (lo < hi && (lo & 31)) {
        words[lo >> 5] |= 1u << (lo & 31);
        ++lo;
    }
    for (; lo + 32 <= hi; lo += 32)
        words[lo >> 5] = 0xffffffffu;
    for (; lo < hi; ++lo)
        words[lo >> 5] |= 1u << (lo & 31);
}

}  // namespace osr

extern "C" {

int adamw_create(int64_t n_params, const int64_t* offsets, const int64_t* numels,
                 int32_t n_tensors, int32_t flags, adamw_ctx** out)
{
    osr::clear_error();
    if (!out)
        return fail(ADAMW_EINVAL, "out is NULL");
    *out = nullptr;
    int rc = validate_table(n_params, offsets, numels, n_tensors);
    if (rc != ADAMW_OK)
        return rc;
    if (flags & ~ADAMW_CREATE_NO_CKPT)
        return fail(ADAMW_EINVAL, "unknown flags 0x%x", flags);

    adamw_ctx* c = new (std::nothrow) adamw_ctx;
    if (!c)
        return fail(ADAMW_EINVAL, "out of host memory");
    c->n = n_params;
    if (n_tensors > 0) {
        c->offsets.assign(offsets, offsets + n_tensors);
        c->numels.assign(numels, numels + n_tensors);
    } else {
        c->offsets.assign(1, 0);
        c->numels.assign(1, n_params);
    }
    auto bail = [&](int status) {
        free_ctx(c);
        return status;
    };
    cudaError_t e = cudaGetDevice(&c->device);
    if (e != cudaSuccess) {
        c->device = -1;
        return bail(cuda_fail(e, "cudaGetDevice"));
    }
    if ((e = cudaDeviceGetAttribute(&c->sm_count, cudaDevAttrMultiProcessorCount, c->device)) !=
        cudaSuccess)
        return bail(cuda_fail(e, "cudaDeviceGetAttribute"));
    if (int qe = osr::query_step_caps(c->sm_count, &c->caps))
        return bail(cuda_fail(cudaError_t(qe), "occupancy query"));
    if (int qe = osr::query_pack_caps(c->sm_count, &c->caps))
        return bail(cuda_fail(cudaError_t(qe), "occupancy query"));
    {
        int coop = 0;
        cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, c->device);
        if (int qe = osr::query_onepass_blocks(c->sm_count, &c->onepass_capacity))
            return bail(cuda_fail(cudaError_t(qe), "occupancy query"));
        c->onepass_max_n = coop ? osr::kOnePassMaxN : 0;
    }

    const size_t scratch = kScratchHead + sizeof(double) * osr::kNormBlocksMax;
    if ((e = cudaMalloc(&c->d_scratch, scratch)) != cudaSuccess)
        return bail(cuda_fail(e, "cudaMalloc(norm scratch)"));
    if ((e = cudaMemset(c->d_scratch, 0, scratch)) != cudaSuccess)
        return bail(cuda_fail(e, "cudaMemset(norm scratch)"));
    c->d_res = reinterpret_cast<osr::NormResult*>(c->d_scratch);
    c->d_counter = reinterpret_cast<unsigned int*>(c->d_scratch + sizeof(osr::NormResult));
    c->d_bar = reinterpret_cast<uint32_t*>(c->d_scratch + 64);
    c->d_chunk_ctr = reinterpret_cast<uint32_t*>(c->d_scratch + 72);
    c->d_pack_ctr = reinterpret_cast<uint32_t*>(c->d_scratch + 80);
    static_assert(sizeof(osr::NormResult) + sizeof(unsigned int) <= 64 && 80 + 8 <= kScratchHead,
                  "scratch head layout");
    c->d_partials = reinterpret_cast<double*>(c->d_scratch + kScratchHead);
    if ((e = cudaHostAlloc(reinterpret_cast<void**>(&c->h_res), sizeof(osr::NormResult),
                           cudaHostAllocMapped)) != cudaSuccess) {
        c->h_res = nullptr;
        return bail(cuda_fail(e, "cudaHostAlloc(norm mirror)"));
    }
    std::memset(c->h_res, 0, sizeof(osr::NormResult));
    if ((e = cudaHostGetDevicePointer(reinterpret_cast<void**>(&c->h_res_dev), c->h_res, 0)) !=
        cudaSuccess)
        return bail(cuda_fail(e, "cudaHostGetDevicePointer"));
    if ((e = cudaEventCreateWithFlags(&c->ev_norm, cudaEventDisableTiming)) != cudaSuccess)
        return bail(cuda_fail(e, "cudaEventCreate"));

    // per-tensor sums: each norm block's range [lo, hi) touches the tensors
    // kfirst .. klast; their slots follow the previous block's
    {
        const int blocks = osr::norm_blocks(n_params);
        std::vector<int64_t> tab(c->offsets);
        tab.push_back(n_params);
        c->kfirst.assign(size_t(blocks), 0);
        c->segbase.assign(size_t(blocks) + 1, 0);
        auto tensor_of = [&](int64_t e) {  // last k with offsets[k] <= e
            return int32_t(std::upper_bound(tab.begin(), tab.end() - 1, e) - tab.begin() - 1);
        };
        for (int b = 0; b < blocks; ++b) {
            const int64_t lo = osr::norm_block_tile(n_params, b) * osr::kNormTileElems;
            int64_t hi = osr::norm_block_tile(n_params, b + 1) * osr::kNormTileElems;
            if (hi > n_params)
                hi = n_params;
            c->kfirst[size_t(b)] = tensor_of(lo);
            c->segbase[size_t(b) + 1] =
                c->segbase[size_t(b)] + (tensor_of(hi - 1) - c->kfirst[size_t(b)] + 1);
        }
        c->nseg = c->segbase[size_t(blocks)];
        if ((e = cudaMalloc(&c->d_tab_offsets, sizeof(int64_t) * tab.size())) != cudaSuccess ||
            (e = cudaMalloc(&c->d_kfirst, sizeof(int32_t) * size_t(blocks))) != cudaSuccess ||
            (e = cudaMalloc(&c->d_segbase, sizeof(int32_t) * (size_t(blocks) + 1))) !=
                cudaSuccess ||
            (e = cudaMalloc(&c->d_seg_sums, sizeof(double) * size_t(c->nseg))) != cudaSuccess ||
            (e = cudaHostAlloc(reinterpret_cast<void**>(&c->h_seg_sums),
                               sizeof(double) * size_t(c->nseg), cudaHostAllocDefault)) !=
                cudaSuccess)
            return bail(cuda_fail(e, "allocating the per-tensor scratch"));
        if ((e = cudaMemcpy(c->d_tab_offsets, tab.data(), sizeof(int64_t) * tab.size(),
                            cudaMemcpyHostToDevice)) != cudaSuccess ||
            (e = cudaMemcpy(c->d_kfirst, c->kfirst.data(), sizeof(int32_t) * size_t(blocks),
                            cudaMemcpyHostToDevice)) != cudaSuccess ||
            (e = cudaMemcpy(c->d_segbase, c->segbase.data(),
                            sizeof(int32_t) * (size_t(blocks) + 1), cudaMemcpyHostToDevice)) !=
                cudaSuccess)
            return bail(cuda_fail(e, "uploading the offset table"));
    }

    if (!(flags & ADAMW_CREATE_NO_CKPT)) {
        const size_t bytes = c->stage_bytes();
        if ((e = cudaMalloc(&c->d_image_alloc, bytes)) != cudaSuccess) {
            c->d_image_alloc = nullptr;
            return bail(cuda_fail(e, "cudaMalloc(checkpoint staging)"));
        }
        if ((e = cudaHostAlloc(reinterpret_cast<void**>(&c->h_image_alloc),
                               c->h_image_capacity(), cudaHostAllocMapped)) != cudaSuccess) {
            c->h_image_alloc = nullptr;
            return bail(cuda_fail(e, "cudaHostAlloc(checkpoint image)"));
        }
        if ((e = cudaHostGetDevicePointer(reinterpret_cast<void**>(&c->h_image_dev),
                                          c->h_image_alloc, 0)) != cudaSuccess)
            return bail(cuda_fail(e, "cudaHostGetDevicePointer(checkpoint image)"));
        if ((e = cudaEventCreateWithFlags(&c->ev_pack, cudaEventDisableTiming)) != cudaSuccess ||
            (e = cudaEventCreateWithFlags(&c->ev_d2h, cudaEventDisableTiming)) != cudaSuccess)
            return bail(cuda_fail(e, "cudaEventCreate"));
        c->has_ckpt = true;
    }
    if ((e = cudaDeviceSynchronize()) != cudaSuccess)
        return bail(cuda_fail(e, "cudaDeviceSynchronize"));
    *out = c;
    return ADAMW_OK;
}

int adamw_destroy(adamw_ctx* ctx)
{
    osr::clear_error();
    free_ctx(ctx);
    return ADAMW_OK;
}

int adamw_set_hparams(adamw_ctx* ctx, double beta1, double beta2, double eps)
{
    osr::clear_error();
    if (!ctx)
        return fail(ADAMW_EINVAL, "ctx is NULL");
    if (!(beta1 >= 0.0 && beta1 < 1.0) || !(beta2 >= 0.0 && beta2 < 1.0) ||
        !(eps >= 0.0 && std::isfinite(eps)))
        return fail(ADAMW_EINVAL, "need 0 <= beta1, beta2 < 1 and finite eps >= 0");
    ctx->beta1 = beta1;
    ctx->beta2 = beta2;
    ctx->eps = eps;
    return ADAMW_OK;
}

int adamw_set_decay_mask(adamw_ctx* ctx, const uint8_t* decay, int32_t n_tensors)
{
    osr::clear_error();
    if (!ctx)
        return fail(ADAMW_EINVAL, "ctx is NULL");
    bool all = true;
    if (decay) {
        if (n_tensors != int32_t(ctx->offsets.size()))
            return fail(ADAMW_EINVAL, "n_tensors=%d, the context's table has %d tensors",
                        n_tensors, int32_t(ctx->offsets.size()));
        for (int32_t k = 0; k < n_tensors; ++k)
            all = all && decay[k] != 0;
    }
    DeviceScope scope(ctx->device);
    // no step of this context may still be reading the flags being replaced
    CUDA_TRY(cudaDeviceSynchronize());
    if (all) {  // decay everywhere: the kernels need no flags
        ctx->decay_mask_on = false;
        return ADAMW_OK;
    }
    const size_t words = size_t((ctx->n + 31) / 32);
    std::vector<uint32_t> h(words, 0u);
    for (int32_t k = 0; k < n_tensors; ++k)
        if (decay[k])
            osr::set_bit_range(h.data(), ctx->offsets[k], ctx->offsets[k] + ctx->numels[k]);
    if (!ctx->d_decay_mask) {
        cudaError_t e = cudaMalloc(&ctx->d_decay_mask, (words * 4 + 15) & ~size_t(15));
        if (e != cudaSuccess) {
            ctx->d_decay_mask = nullptr;
            return cuda_fail(e, "cudaMalloc(decay flags)");
        }
    }
    CUDA_TRY(cudaMemcpy(ctx->d_decay_mask, h.data(), words * 4, cudaMemcpyHostToDevice));
    ctx->decay_mask_on = true;
    return ADAMW_OK;
}

int64_t adamw_num_params(const adamw_ctx* ctx) { return ctx ? ctx->n : -1; }

int32_t adamw_num_tensors(const adamw_ctx* ctx)
{
    return ctx ? int32_t(ctx->offsets.size()) : -1;
}

int grad_global_norm(adamw_ctx* ctx, const float* d_g, double* h_norm, void* stream)
{
    osr::clear_error();
    if (!ctx)
        return fail(ADAMW_EINVAL, "ctx is NULL");
    int rc = check_state_ptr(d_g, "d_g");
    if (rc != ADAMW_OK)
        return rc;
    DeviceScope scope(ctx->device);
    rc = launch_norm_on(ctx, d_g, INFINITY, stream);
    if (rc == ADAMW_OK)
        rc = mark_norm(ctx, static_cast<cudaStream_t>(stream));
    if (rc != ADAMW_OK || !h_norm)
        return rc;
    return read_norm(ctx, h_norm, nullptr);
}

int adamw_clip_step(adamw_ctx* ctx, float* d_w, const float* d_g, float* d_m, float* d_v,
                    int32_t t, double lr, double wd, double clip, void* stream)
{
    return adamw_clip_step_ex(ctx, d_w, const_cast<float*>(d_g), d_m, d_v, t, lr, wd, clip, 1.0,
                              -1.0, 0, stream);
}

int adamw_clip_step_ex(adamw_ctx* ctx, float* d_w, float* d_g, float* d_m, float* d_v,
                       int32_t t, double lr, double wd, double clip, double grad_scale,
                       double global_sumsq, int32_t flags, void* stream)
{
    return adamw_clip_step_mixed(ctx, d_w, d_g, ADAMW_DTYPE_F32, d_m, d_v, nullptr,
                                 ADAMW_DTYPE_BF16, t, lr, wd, clip, grad_scale, global_sumsq,
                                 flags, stream);
}

// The step behind adamw_clip_step_mixed (and _ex, plain) and
// adamw_clip_step_gathered (d_rank_sumsq != NULL: the global sum of squares
// is added up on the device from the ranks' gathered values).
static int step_impl(adamw_ctx* ctx, float* d_w, void* d_g, int32_t g_dtype, float* d_m, float* d_v,
              void* d_w_lp, int32_t w_lp_dtype, int32_t t, double lr, double wd, double clip,
              double grad_scale, double global_sumsq, const double* d_rank_sumsq,
              int32_t world, int32_t flags, void* stream)
{
    osr::clear_error();
    if (!ctx)
        return fail(ADAMW_EINVAL, "ctx is NULL");
    int rc;
    if ((rc = check_state_ptr(d_w, "d_w")) || (rc = check_state_ptr(d_m, "d_m")) ||
        (rc = check_state_ptr(d_v, "d_v")))
        return rc;
    if (g_dtype != ADAMW_DTYPE_F32 && g_dtype != ADAMW_DTYPE_BF16 && g_dtype != ADAMW_DTYPE_F16)
        return fail(ADAMW_EINVAL, "g_dtype=%d is not F32, BF16 or F16", g_dtype);
    if (d_w_lp && w_lp_dtype != ADAMW_DTYPE_BF16 && w_lp_dtype != ADAMW_DTYPE_F16)
        return fail(ADAMW_EINVAL, "w_lp_dtype=%d is not BF16 or F16", w_lp_dtype);
    if (!d_g)
        return fail(ADAMW_EINVAL, "d_g is NULL");
    if (g_dtype == ADAMW_DTYPE_F32 && !d_w_lp) {
        if ((rc = check_state_ptr(d_g, "d_g")))
            return rc;
    } else {
        const uintptr_t ga = reinterpret_cast<uintptr_t>(d_g);
        if ((reinterpret_cast<uintptr_t>(d_w) | reinterpret_cast<uintptr_t>(d_m) |
             reinterpret_cast<uintptr_t>(d_v)) & 15u ||
            (g_dtype == ADAMW_DTYPE_F32 ? (ga & 15u) : (ga & 7u)) ||
            (reinterpret_cast<uintptr_t>(d_w_lp) & 7u))
            return fail(ADAMW_EINVAL,
                        "16-bit gradients or a weight copy need w, m, v (and a float32 g) on "
                        "16-byte boundaries, a 16-bit g and the copy on 8-byte boundaries");
    }
    if (t < 1)
        return fail(ADAMW_EINVAL, "t=%d: the first update has t = 1", t);
    if (!(lr >= 0.0 && std::isfinite(lr)) || !(wd >= 0.0 && std::isfinite(wd)))
        return fail(ADAMW_EINVAL, "lr=%g wd=%g must be finite and >= 0", lr, wd);
    if (!(clip > 0.0))
        return fail(ADAMW_EINVAL, "clip=%g must be > 0 (INFINITY disables clipping)", clip);
    if (!(grad_scale > 0.0 && std::isfinite(grad_scale)))
        return fail(ADAMW_EINVAL, "grad_scale=%g must be finite and > 0", grad_scale);
    if (flags & ~(ADAMW_ZERO_GRAD | ADAMW_TENSOR_NORMS))
        return fail(ADAMW_EINVAL, "unknown flags 0x%x", flags);
    const bool gathered = d_rank_sumsq != nullptr;
    if (gathered && (world < 1 || (reinterpret_cast<uintptr_t>(d_rank_sumsq) & 7u)))
        return fail(ADAMW_EINVAL, "world=%d must be >= 1, d_rank_sumsq 8-byte aligned", world);
    if (gathered && (flags & ADAMW_TENSOR_NORMS))
        return fail(ADAMW_EINVAL, "per-tensor norms need the shard's own reduction");
    const bool external = !gathered && !(global_sumsq < 0.0);  // NaN counts as given

    osr::StepScalars k = osr::make_step_scalars(ctx, t, lr, wd);
    if (external) {
        // the global norm of the sharded gradient, from the ranks' sums
        const double norm = grad_scale * std::sqrt(global_sumsq);
        if (!std::isfinite(norm))
            return fail(ADAMW_ENONFINITE, "global gradient norm is %g: the update was skipped",
                        norm);
        k.scale = float(grad_scale * (norm > clip ? clip / norm : 1.0));
    }

    DeviceScope scope(ctx->device);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaEvent_t prof[3] = {ctx->prof[0], ctx->prof[1], ctx->prof[2]};
    ctx->prof[0] = ctx->prof[1] = ctx->prof[2] = nullptr;
    if (prof[0])
        CUDA_TRY(cudaEventRecord(prof[0], st));
    // Small states: the whole step as one launch (same bits as the two
    // launches below); not when an event was asked for between the two
    // kernels.  Launched from the host, one launch saves about 2 us of launch
    // overhead per step up to 2^19 parameters.  Captured into a graph, where
    // launch overhead is gone, only the cluster form (up to 65,536
    // parameters, without zero-grad) is kept: above it the cooperative
    // grid's barrier costs more GPU time than the two overlapping launches
    // (measured on GB300: 7.7 vs 6.3 us at 2^17, 8.9 vs 7.2 us at 2^19).
    // The barrier-timeout test flag still takes the grid.
    cudaStreamCaptureStatus capturing = cudaStreamCaptureStatusNone;
    CUDA_TRY(cudaStreamIsCapturing(st, &capturing));
    const bool cluster_form = osr::onepass_is_cluster(ctx->n) && !(flags & ADAMW_ZERO_GRAD);
    if (!external && !gathered && g_dtype == ADAMW_DTYPE_F32 && !d_w_lp &&
        !(flags & ADAMW_TENSOR_NORMS) &&
        (capturing == cudaStreamCaptureStatusNone || cluster_form || ctx->onepass_fault_test) &&
        !prof[1] && ctx->onepass && ctx->n <= ctx->onepass_max_n &&
        osr::onepass_grid(ctx->n, ctx->onepass_capacity) <= ctx->onepass_capacity &&
        aligned16(d_w) && aligned16(d_g) && aligned16(d_m) && aligned16(d_v)) {
        const bool fault_test = ctx->onepass_fault_test;
        ctx->onepass_fault_test = false;
        const int e = osr::launch_onepass(
            d_w, static_cast<float*>(d_g), d_m, d_v, ctx->n, k, clip, grad_scale,
            ctx->d_partials, ctx->d_bar, fault_test, ctx->d_res, ctx->h_res_dev,
            ctx->onepass_capacity, (flags & ADAMW_ZERO_GRAD) != 0, stream);
        if (e != cudaSuccess)
            return cuda_fail(cudaError_t(e), "one-launch step");
        ctx->segs_launched = false;  // this reduction wrote no per-tensor sums
        if (prof[2])
            CUDA_TRY(cudaEventRecord(prof[2], st));
        return mark_norm(ctx, st);
    }
    if (gathered) {
        const int e = osr::launch_rank_total(d_rank_sumsq, world, clip, grad_scale, ctx->d_res,
                                             ctx->h_res_dev, stream);
        if (e != cudaSuccess)
            return cuda_fail(cudaError_t(e), "global-sum kernel launch");
        ctx->segs_launched = false;
    } else if (!external) {
        // the norm kernel writes its partials; the fused kernel sums them
        rc = launch_norm_on(ctx, d_g, clip, stream, grad_scale,
                            (flags & ADAMW_TENSOR_NORMS) != 0, g_dtype, false);
        if (rc != ADAMW_OK)
            return rc;
        k.fin = osr::NormFinish{ctx->d_partials, osr::norm_blocks(ctx->n), clip, grad_scale,
                                ctx->d_res, ctx->h_res_dev};
    }
    if (prof[1])
        CUDA_TRY(cudaEventRecord(prof[1], st));
    // programmatic launch only straight behind the norm kernel (no event
    // recorded in between)
    const bool programmatic = !external && !prof[1] && ctx->pdl;
    const int e = osr::launch_adamw(d_w, d_g, d_m, d_v, ctx->n, k, external ? nullptr : ctx->d_res,
                                    ctx->caps, stream, (flags & ADAMW_ZERO_GRAD) != 0,
                                    programmatic, g_dtype, d_w_lp, w_lp_dtype);
    if (e != cudaSuccess)
        return cuda_fail(cudaError_t(e), "clip+AdamW kernel launch");
    if (prof[2])
        CUDA_TRY(cudaEventRecord(prof[2], st));
    if (!external)  // the norm result is complete once the step is
        return mark_norm(ctx, st);
    return ADAMW_OK;
}

int adamw_clip_step_mixed(adamw_ctx* ctx, float* d_w, void* d_g, int32_t g_dtype, float* d_m,
                          float* d_v, void* d_w_lp, int32_t w_lp_dtype, int32_t t, double lr,
                          double wd, double clip, double grad_scale, double global_sumsq,
                          int32_t flags, void* stream)
{
    return step_impl(ctx, d_w, d_g, g_dtype, d_m, d_v, d_w_lp, w_lp_dtype, t, lr, wd, clip,
                     grad_scale, global_sumsq, nullptr, 0, flags, stream);
}

int adamw_clip_step_gathered(adamw_ctx* ctx, float* d_w, void* d_g, int32_t g_dtype, float* d_m,
                             float* d_v, int32_t t, double lr, double wd, double clip,
                             double grad_scale, const double* d_rank_sumsq, int32_t world,
                             int32_t flags, void* stream)
{
    osr::clear_error();
    if (!d_rank_sumsq)
        return fail(ADAMW_EINVAL, "d_rank_sumsq is NULL");
    return step_impl(ctx, d_w, d_g, g_dtype, d_m, d_v, nullptr, ADAMW_DTYPE_BF16, t, lr, wd,
                     clip, grad_scale, -1.0, d_rank_sumsq, world, flags, stream);
}

int adamw_rank_total(const double* h_rank_sumsq, int32_t world, double clip, double grad_scale,
                     double* sumsq_out, double* norm_out, float* scale_out)
{
    osr::clear_error();
    if (!h_rank_sumsq || world < 1)
        return fail(ADAMW_EINVAL, "h_rank_sumsq is NULL or world=%d < 1", world);
    if (!(clip > 0.0))
        return fail(ADAMW_EINVAL, "clip=%g must be > 0 (INFINITY disables clipping)", clip);
    if (!(grad_scale > 0.0 && std::isfinite(grad_scale)))
        return fail(ADAMW_EINVAL, "grad_scale=%g must be finite and > 0", grad_scale);
    // rank order, one double addition per rank (the device form, the
    // k_rank_total kernel, adds in the same order)
    double s = 0.0;
    for (int32_t r = 0; r < world; ++r) {
        const double x = h_rank_sumsq[r];
        if (x < 0.0)
            return fail(ADAMW_EINVAL, "rank %d's sum of squares is negative (%g)", r, x);
        s += x;
    }
    const double norm = grad_scale * std::sqrt(s);
    const bool finite = std::isfinite(norm);
    if (sumsq_out)
        *sumsq_out = s;
    if (norm_out)
        *norm_out = norm;
    if (scale_out)
        *scale_out = float(grad_scale * ((finite && norm > clip) ? clip / norm : 1.0));
    if (!finite)
        return fail(ADAMW_ENONFINITE, "global gradient norm is %g", norm);
    return ADAMW_OK;
}

int adamw_clip_step_ranks(adamw_ctx* ctx, float* d_w, void* d_g, int32_t g_dtype, float* d_m,
                          float* d_v, int32_t t, double lr, double wd, double clip,
                          double grad_scale, const double* h_rank_sumsq, int32_t world,
                          int32_t flags, void* stream)
{
    if (flags & ADAMW_TENSOR_NORMS) {
        osr::clear_error();
        return fail(ADAMW_EINVAL, "per-tensor norms need the shard's own reduction");
    }
    double total = 0.0;
    const int rc = adamw_rank_total(h_rank_sumsq, world, clip, grad_scale, &total, nullptr,
                                    nullptr);
    if (rc != ADAMW_OK)  // a non-finite global norm: nothing is launched
        return rc;
    return step_impl(ctx, d_w, d_g, g_dtype, d_m, d_v, nullptr, ADAMW_DTYPE_BF16, t, lr, wd,
                     clip, grad_scale, total, nullptr, 0, flags, stream);
}

int grad_sumsq_to(adamw_ctx* ctx, const void* d_g, int32_t g_dtype, double* d_out, void* stream)
{
    osr::clear_error();
    if (!ctx || !d_out || (reinterpret_cast<uintptr_t>(d_out) & 7u))
        return fail(ADAMW_EINVAL, "ctx is NULL or d_out NULL / not 8-byte aligned");
    int rc = ADAMW_OK;
    if (g_dtype == ADAMW_DTYPE_F32)
        rc = check_state_ptr(d_g, "d_g");
    else if (g_dtype != ADAMW_DTYPE_BF16 && g_dtype != ADAMW_DTYPE_F16)
        rc = fail(ADAMW_EINVAL, "g_dtype=%d is not F32, BF16 or F16", g_dtype);
    else if (!d_g || (reinterpret_cast<uintptr_t>(d_g) & 7u))
        rc = fail(ADAMW_EINVAL, "a 16-bit d_g must be on an 8-byte boundary");
    if (rc != ADAMW_OK)
        return rc;
    DeviceScope scope(ctx->device);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    rc = launch_norm_on(ctx, d_g, INFINITY, stream, 1.0, false, g_dtype);
    if (rc != ADAMW_OK)
        return rc;
    CUDA_TRY(cudaMemcpyAsync(d_out, &ctx->d_res->sumsq, sizeof(double), cudaMemcpyDeviceToDevice,
                             st));
    return mark_norm(ctx, st);
}

int grad_tensor_sumsq(adamw_ctx* ctx, const float* d_g, double* h_out, void* stream)
{
    osr::clear_error();
    if (!ctx || !h_out)
        return fail(ADAMW_EINVAL, "ctx or h_out is NULL");
    int rc = check_state_ptr(d_g, "d_g");
    if (rc != ADAMW_OK)
        return rc;
    DeviceScope scope(ctx->device);
    rc = launch_norm_on(ctx, d_g, INFINITY, stream, 1.0, true);
    if (rc == ADAMW_OK)
        rc = mark_norm(ctx, static_cast<cudaStream_t>(stream));
    if (rc != ADAMW_OK)
        return rc;
    rc = read_tensor_sums(ctx, h_out);
    if (rc != ADAMW_OK)
        return rc;
    return read_norm(ctx, nullptr, nullptr);
}

int adamw_last_tensor_sumsq(adamw_ctx* ctx, double* h_out)
{
    osr::clear_error();
    if (!ctx || !h_out)
        return fail(ADAMW_EINVAL, "ctx or h_out is NULL");
    DeviceScope scope(ctx->device);
    return read_tensor_sums(ctx, h_out);
}

int adamw_set_launch_options(adamw_ctx* ctx, int32_t flags)
{
    osr::clear_error();
    if (!ctx)
        return fail(ADAMW_EINVAL, "ctx is NULL");
    if (flags & ~(ADAMW_LAUNCH_NO_PDL | ADAMW_LAUNCH_NO_ONEPASS |
                  ADAMW_LAUNCH_TEST_BARRIER_TIMEOUT | ADAMW_LAUNCH_STATIC_CHUNKS))
        return fail(ADAMW_EINVAL, "unknown launch flags 0x%x", flags);
    ctx->dynamic_chunks = !(flags & ADAMW_LAUNCH_STATIC_CHUNKS);
    ctx->pdl = !(flags & ADAMW_LAUNCH_NO_PDL);
    ctx->onepass = !(flags & ADAMW_LAUNCH_NO_ONEPASS);
    ctx->onepass_fault_test = (flags & ADAMW_LAUNCH_TEST_BARRIER_TIMEOUT) != 0;
    return ADAMW_OK;
}

int grad_sumsq(adamw_ctx* ctx, const float* d_g, double* h_sumsq, void* stream)
{
    return grad_sumsq_typed(ctx, d_g, ADAMW_DTYPE_F32, h_sumsq, stream);
}

int grad_sumsq_typed(adamw_ctx* ctx, const void* d_g, int32_t g_dtype, double* h_sumsq,
                     void* stream)
{
    osr::clear_error();
    if (!ctx || !h_sumsq)
        return fail(ADAMW_EINVAL, "ctx or h_sumsq is NULL");
    int rc = ADAMW_OK;
    if (g_dtype == ADAMW_DTYPE_F32)
        rc = check_state_ptr(d_g, "d_g");
    else if (g_dtype != ADAMW_DTYPE_BF16 && g_dtype != ADAMW_DTYPE_F16)
        rc = fail(ADAMW_EINVAL, "g_dtype=%d is not F32, BF16 or F16", g_dtype);
    else if (!d_g || (reinterpret_cast<uintptr_t>(d_g) & 7u))
        rc = fail(ADAMW_EINVAL, "a 16-bit d_g must be on an 8-byte boundary");
    if (rc != ADAMW_OK)
        return rc;
    DeviceScope scope(ctx->device);
    rc = launch_norm_on(ctx, d_g, INFINITY, stream, 1.0, false, g_dtype);
    if (rc == ADAMW_OK)
        rc = mark_norm(ctx, static_cast<cudaStream_t>(stream));
    if (rc != ADAMW_OK)
        return rc;
    rc = read_norm(ctx, nullptr, nullptr);
    *h_sumsq = static_cast<const volatile osr::NormResult*>(ctx->h_res)->sumsq;
    return rc;
}

int adamw_record_events(adamw_ctx* ctx, void* ev_begin, void* ev_mid, void* ev_end)
{
    osr::clear_error();
    if (!ctx)
        return fail(ADAMW_EINVAL, "ctx is NULL");
    ctx->prof[0] = static_cast<cudaEvent_t>(ev_begin);
    ctx->prof[1] = static_cast<cudaEvent_t>(ev_mid);
    ctx->prof[2] = static_cast<cudaEvent_t>(ev_end);
    return ADAMW_OK;
}

int adamw_last_norm(adamw_ctx* ctx, double* norm_out, float* scale_out)
{
    osr::clear_error();
    if (!ctx)
        return fail(ADAMW_EINVAL, "ctx is NULL");
    DeviceScope scope(ctx->device);
    return read_norm(ctx, norm_out, scale_out);
}

int ckpt_pack(adamw_ctx* ctx, int32_t step, const float* d_w, const float* d_m,
              const float* d_v, void* main_stream, void* side_stream)
{
    osr::clear_error();
    if (!ctx)
        return fail(ADAMW_EINVAL, "ctx is NULL");
    if (!ctx->has_ckpt)
        return fail(ADAMW_ESTATE, "context was created without checkpoint staging");
    int rc;
    if ((rc = check_state_ptr(d_w, "d_w")) || (rc = check_state_ptr(d_m, "d_m")) ||
        (rc = check_state_ptr(d_v, "d_v")))
        return rc;
    if (step < 0)
        return fail(ADAMW_EINVAL, "step=%d is negative", step);
    // The pinned image may still be read by a write in flight.
    osr::writer_drain(ctx);
    DeviceScope scope(ctx->device);
    cudaStream_t mainst = static_cast<cudaStream_t>(main_stream);
    cudaStream_t side = static_cast<cudaStream_t>(side_stream);
    // The staging image may still be read by the previous copy.
    if (ctx->d2h_pending)
        CUDA_TRY(cudaStreamWaitEvent(mainst, ctx->ev_d2h, 0));
    const int e = osr::launch_pack(d_w, d_m, d_v, ctx->n, step, ctx->d_stage(0),
                                   reinterpret_cast<float*>(ctx->d_stage(1)),
                                   reinterpret_cast<float*>(ctx->d_stage(2)),
                                   reinterpret_cast<float*>(ctx->d_stage(3)), ctx->caps,
                                   main_stream,
                                   (ctx->dynamic_chunks && ctx->n >= osr::kDynamicChunksMinN)
                                       ? ctx->d_pack_ctr
                                       : nullptr);
    if (e != cudaSuccess)
        return cuda_fail(cudaError_t(e), "pack kernel launch");
    CUDA_TRY(cudaEventRecord(ctx->ev_pack, mainst));
    if (side != mainst)
        CUDA_TRY(cudaStreamWaitEvent(side, ctx->ev_pack, 0));
    // the header and the three regions to their file offsets in the image
    // (the kernel writes whole 16-byte units from a 16-byte aligned image;
    // a mapped pinned allocation starts on a page)
    if (ctx->copy_engine || (reinterpret_cast<uintptr_t>(ctx->h_image_dev) & 15u)) {
        const size_t rb = size_t(4) * size_t(ctx->n);
        CUDA_TRY(cudaMemcpyAsync(ctx->h_image(), ctx->d_stage(0), 8, cudaMemcpyDeviceToHost,
                                 side));
        for (int r = 1; r <= 3; ++r)
            CUDA_TRY(cudaMemcpyAsync(ctx->h_image() + 8 + size_t(r - 1) * rb, ctx->d_stage(r),
                                     rb, cudaMemcpyDeviceToHost, side));
    } else {
        const int ce = osr::launch_stage_to_host(
            ctx->d_stage(0), reinterpret_cast<const float*>(ctx->d_stage(1)),
            reinterpret_cast<const float*>(ctx->d_stage(2)),
            reinterpret_cast<const float*>(ctx->d_stage(3)), ctx->n, ctx->h_image_dev,
            ctx->sm_count, side);
        if (ce != cudaSuccess)
            return cuda_fail(cudaError_t(ce), "staging copy kernel launch");
    }
    CUDA_TRY(cudaEventRecord(ctx->ev_d2h, side));
    ctx->packed = true;
    ctx->d2h_pending = true;
    ctx->packed_step = step;
    return ADAMW_OK;
}

int ckpt_read(adamw_ctx* ctx, const char* path, int32_t* step_out, float* d_w, float* d_m,
              float* d_v, void* stream)
{
    osr::clear_error();
    if (!ctx || !path)
        return fail(ADAMW_EINVAL, "ctx or path is NULL");
    if (!ctx->has_ckpt)
        return fail(ADAMW_ESTATE, "context was created without checkpoint staging");
    int rc;
    if ((rc = check_state_ptr(d_w, "d_w")) || (rc = check_state_ptr(d_m, "d_m")) ||
        (rc = check_state_ptr(d_v, "d_v")))
        return rc;
    osr::writer_drain(ctx);
    DeviceScope scope(ctx->device);
    if (ctx->d2h_pending) {
        CUDA_TRY(cudaEventSynchronize(ctx->ev_d2h));
        ctx->d2h_pending = false;
    }
    int32_t step = -1;
    int fd = -1;
    rc = osr::open_validated(path, int32_t(ctx->n), &step, nullptr, &fd);
    if (rc != ADAMW_OK)
        return rc;
    ctx->packed = false;  // the pinned image is about to hold the file instead
    const size_t bytes = size_t(ctx->n) * 4u;
    unsigned char* body = ctx->h_image() + 8;
    rc = osr::read_exact(fd, body, 3 * bytes, path);
    ::close(fd);
    if (rc != ADAMW_OK)
        return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    CUDA_TRY(cudaMemcpyAsync(d_w, body, bytes, cudaMemcpyHostToDevice, s));
    CUDA_TRY(cudaMemcpyAsync(d_m, body + bytes, bytes, cudaMemcpyHostToDevice, s));
    CUDA_TRY(cudaMemcpyAsync(d_v, body + 2 * bytes, bytes, cudaMemcpyHostToDevice, s));
    CUDA_TRY(cudaStreamSynchronize(s));
    if (step_out)
        *step_out = step;
    return ADAMW_OK;
}

int ckpt_read_range(adamw_ctx* ctx, const char* path, int64_t offset, int32_t* step_out,
                    float* d_w, float* d_m, float* d_v, void* stream)
{
    osr::clear_error();
    if (!ctx || !path)
        return fail(ADAMW_EINVAL, "ctx or path is NULL");
    if (!ctx->has_ckpt)
        return fail(ADAMW_ESTATE, "context was created without checkpoint staging");
    int rc;
    if ((rc = check_state_ptr(d_w, "d_w")) || (rc = check_state_ptr(d_m, "d_m")) ||
        (rc = check_state_ptr(d_v, "d_v")))
        return rc;
    if (offset < 0)
        return fail(ADAMW_EINVAL, "offset=%lld is negative", (long long)offset);
    osr::writer_drain(ctx);
    DeviceScope scope(ctx->device);
    if (ctx->d2h_pending) {
        CUDA_TRY(cudaEventSynchronize(ctx->ev_d2h));
        ctx->d2h_pending = false;
    }
    int32_t step = -1, nf = -1;
    int fd = -1;
    rc = osr::open_validated(path, -1, &step, &nf, &fd);
    if (rc != ADAMW_OK)
        return rc;
    if (offset + ctx->n > int64_t(nf)) {
        ::close(fd);
        return fail(ADAMW_EMISMATCH, "%s holds %d parameters; [%lld, %lld) is out of range", path,
                    nf, (long long)offset, (long long)(offset + ctx->n));
    }
    ctx->packed = false;  // the pinned image is about to hold the file's range
    const size_t bytes = size_t(ctx->n) * 4u;
    unsigned char* body = ctx->h_image() + 8;
    for (int r = 0; r < 3 && rc == ADAMW_OK; ++r)
        rc = osr::pread_exact(fd, body + size_t(r) * bytes, bytes,
                              8 + 4 * (int64_t(nf) * r + offset), path);
    ::close(fd);
    if (rc != ADAMW_OK)
        return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    CUDA_TRY(cudaMemcpyAsync(d_w, body, bytes, cudaMemcpyHostToDevice, s));
    CUDA_TRY(cudaMemcpyAsync(d_m, body + bytes, bytes, cudaMemcpyHostToDevice, s));
    CUDA_TRY(cudaMemcpyAsync(d_v, body + 2 * bytes, bytes, cudaMemcpyHostToDevice, s));
    CUDA_TRY(cudaStreamSynchronize(s));
    if (step_out)
        *step_out = step;
    return ADAMW_OK;
}

}  // extern "C"
