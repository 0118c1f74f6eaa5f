// gen.cu -- device twin of synthetic/__init__.py: fills a float32 buffer with
// the same counter-based draws the numpy code makes, bit for bit.  Test and
// benchmark input generation only; it holds no optimizer arithmetic.
//
// hash(key, i) = SplitMix64 output function (Steele, Lea & Flood, OOPSLA
// 2014) of key + (i + 1) * 0x9E3779B97F4A7C15; value = (sum of the four
// 16-bit lanes - 131070) * scale, one float32 multiply; an outlier (top 32
// bits of hash(okey, i) below othr) is multiplied by omul.
#include <cstdint>

#include <cuda_runtime.h>

namespace {

__device__ __forceinline__ uint64_t mix64(uint64_t z)
{
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

__global__ void k_synth_fill(float* __restrict__ out, int64_t n, uint64_t key, float scale,
                             uint64_t okey, uint32_t othr, float omul)
{
    const int64_t stride = int64_t(gridDim.x) * blockDim.x;
    for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride) {
        const uint64_t c = uint64_t(i) + 1ull;
        const uint64_t h = mix64(key + c * 0x9E3779B97F4A7C15ull);
        const int32_t s = int32_t(h & 0xFFFFu) + int32_t((h >> 16) & 0xFFFFu) +
                          int32_t((h >> 32) & 0xFFFFu) + int32_t(h >> 48) - 131070;
        float x = __fmul_rn(float(s), scale);
        if (othr != 0u) {
            const uint64_t ho = mix64(okey + c * 0x9E3779B97F4A7C15ull);
            if (uint32_t(ho >> 32) < othr)
                x = __fmul_rn(x, omul);
        }
        out[i] = x;
    }
}

}  // namespace

extern "C" int synth_fill(float* out, int64_t n, uint64_t key, float scale, uint64_t okey,
                          uint32_t othr, float omul, void* stream)
{
    if (n <= 0)
        return 0;
    if (!out)
        return int(cudaErrorInvalidValue);
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    int64_t blocks = (n + 255) / 256;
    const int64_t cap = int64_t(sms > 0 ? sms : 1) * 8;
    if (blocks > cap)
        blocks = cap;
    k_synth_fill<<<int(blocks), 256, 0, static_cast<cudaStream_t>(stream)>>>(
        out, n, key, scale, okey, othr, omul);
    return int(cudaGetLastError());
}
