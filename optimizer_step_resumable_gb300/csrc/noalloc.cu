// noalloc.cu -- the clipped-AdamW step for callers that must not allocate.
//
// adamw_create allocates the reduction scratch (and checkpoint staging)
// with cudaMalloc / cudaHostAlloc.  Some callers cannot do that: code that
// runs under a framework or serving process which owns every byte of device
// memory through its own pool and treats any other allocation as a budget
// violation; plug-ins that are handed only their input and output buffers
// through a narrow C interface and have no object whose lifetime could own
// scratch; and latency-critical paths where cudaMalloc / cudaFree would
// synchronise the device and stall every other stream.  This file serves them
// with one entry point whose only scratch is a small file-scope device array.
//
// The array holds the norm reduction's result record, its block ticket
// counter and one double partial per block.  Because the reduction grid is
// capped at kNormBlocksMax blocks whatever n is, the array has a fixed size
// (256 + 8 x 608 = 5,120 bytes) and serves every n up to 2^31 - 1.  Every
// GPU that loads this library holds it until the process exits.
#include <cmath>
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "internal.h"

namespace osr {
namespace {

constexpr size_t kHeadBytes = 256;  // NormResult + ticket counter, padded
constexpr size_t kNoAllocScratchBytes = kHeadBytes + sizeof(double) * kNormBlocksMax;

// The scratch.  In host code this name is only a stand-in for the device
// symbol; its device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;

struct DeviceSetup {
    bool ready = false;
    unsigned char* scratch = nullptr;  // device address of g_noalloc_scratch
    KernelCaps caps{};
};

std::mutex g_setup_mutex;
DeviceSetup g_setup[kMaxDevices];

// Once per device, with that device current: resolve the scratch's device
// address and the kernels' resident-block counts.  Allocates nothing.
int setup_device(int device, DeviceSetup** out)
{
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    DeviceSetup& s = g_setup[device];
    if (!s.ready) {
        void* ptr = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
        if (e != cudaSuccess)
            return fail(ADAMW_ECUDA, "cudaGetSymbolAddress(no-alloc scratch): %s",
                        cudaGetErrorString(e));
        int sms = 0;
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device);
        if (e != cudaSuccess)
            return fail(ADAMW_ECUDA, "cudaDeviceGetAttribute: %s", cudaGetErrorString(e));
        if (int qe = query_step_caps(sms, &s.caps))
            return fail(ADAMW_ECUDA, "occupancy query: %s", cudaGetErrorString(cudaError_t(qe)));
        s.scratch = static_cast<unsigned char*>(ptr);
        s.ready = true;
    }
    *out = &s;
    return ADAMW_OK;
}

bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

}  // namespace
}  // namespace osr

extern "C" int adamw_clip_step_noalloc(float* d_w, const float* d_g, float* d_m, float* d_v,
                                       int64_t n, int32_t t, double lr, double wd,
                                       double clip, double beta1, double beta2, double eps,
                                       double* d_norm_out, void* stream)
{
    using osr::fail;
    osr::clear_error();
    if (n < 1 || n > INT32_MAX)
        return fail(ADAMW_EINVAL,
                    "adamw_clip_step_noalloc: n=%lld outside [1, 2^31-1], the largest state "
                    "its fixed %zu-byte scratch serves",
                    (long long)n, osr::kNoAllocScratchBytes);
    const size_t need = osr::kHeadBytes + sizeof(double) * size_t(osr::norm_blocks(n));
    if (need > osr::kNoAllocScratchBytes)
        return fail(ADAMW_EINVAL, "adamw_clip_step_noalloc: n=%lld needs %zu scratch bytes > %zu",
                    (long long)n, need, osr::kNoAllocScratchBytes);
    const void* ptrs[4] = {d_w, d_g, d_m, d_v};
    for (const void* p : ptrs)
        if (!p || !osr::aligned4(p))
            return fail(ADAMW_EINVAL, "adamw_clip_step_noalloc: null or unaligned state pointer");
    if (t < 1)
        return fail(ADAMW_EINVAL, "adamw_clip_step_noalloc: t=%d, the first update has t = 1", t);
    if (!(lr >= 0.0 && std::isfinite(lr)) || !(wd >= 0.0 && std::isfinite(wd)) || !(clip > 0.0))
        return fail(ADAMW_EINVAL, "adamw_clip_step_noalloc: need finite lr, wd >= 0 and clip > 0");
    if (!(beta1 >= 0.0 && beta1 < 1.0) || !(beta2 >= 0.0 && beta2 < 1.0) ||
        !(eps >= 0.0 && std::isfinite(eps)))
        return fail(ADAMW_EINVAL, "adamw_clip_step_noalloc: need 0 <= beta < 1, finite eps >= 0");

    int device = -1;
    cudaError_t e = cudaGetDevice(&device);
    if (e != cudaSuccess)
        return fail(ADAMW_ECUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    if (device < 0 || device >= osr::kMaxDevices)
        return fail(ADAMW_EINVAL, "adamw_clip_step_noalloc: device %d >= %d", device,
                    osr::kMaxDevices);
    osr::DeviceSetup* s = nullptr;
    int rc = osr::setup_device(device, &s);
    if (rc != ADAMW_OK)
        return rc;

    osr::NormResult* res = reinterpret_cast<osr::NormResult*>(s->scratch);
    unsigned int* counter =
        reinterpret_cast<unsigned int*>(s->scratch + sizeof(osr::NormResult));
    double* partials = reinterpret_cast<double*>(s->scratch + osr::kHeadBytes);
    cudaStream_t st = static_cast<cudaStream_t>(stream);

    // The array keeps whatever the last call left; the block ticket counter
    // must start at zero.
    if ((e = cudaMemsetAsync(counter, 0, sizeof(unsigned int), st)) != cudaSuccess)
        return fail(ADAMW_ECUDA, "cudaMemsetAsync: %s", cudaGetErrorString(e));

    const double bc1 = 1.0 - std::pow(beta1, double(t));
    const double bc2 = 1.0 - std::pow(beta2, double(t));
    osr::StepScalars k{};  // (k.fin unused: the norm kernel publishes its result)
    k.beta1 = float(beta1);
    k.omb1 = float(1.0 - beta1);
    k.beta2 = float(beta2);
    k.omb2 = float(1.0 - beta2);
    k.eps = float(eps);
    k.step_size = float(lr / bc1);
    k.inv_sqrt_bc2 = float(1.0 / std::sqrt(bc2));
    k.decay = float(1.0 - lr * wd);
    k.scale = 1.0f;  // unused: the factor comes from the norm result
    k.decay_mask = nullptr;  // decay on every parameter
    k.chunk_ctr = nullptr;   // chunks dealt out cyclically (no counter scratch)

    int le = osr::launch_norm(d_g, n, clip, partials, counter, res, nullptr, stream);
    if (le != cudaSuccess)
        return fail(ADAMW_ECUDA, "norm kernel launch: %s", cudaGetErrorString(cudaError_t(le)));
    le = osr::launch_adamw(d_w, d_g, d_m, d_v, n, k, res, s->caps, stream);
    if (le != cudaSuccess)
        return fail(ADAMW_ECUDA, "clip+AdamW kernel launch: %s",
                    cudaGetErrorString(cudaError_t(le)));
    if (d_norm_out) {
        e = cudaMemcpyAsync(d_norm_out, &res->norm, sizeof(double), cudaMemcpyDeviceToDevice, st);
        if (e != cudaSuccess)
            return fail(ADAMW_ECUDA, "cudaMemcpyAsync(norm): %s", cudaGetErrorString(e));
    }
    return ADAMW_OK;
}
