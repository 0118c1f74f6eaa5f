// internal.h -- declarations shared by the library's translation units.
// Not part of the public ABI (that is include/adamw_ckpt.h).
#pragma once

#include <cstddef>
#include <cstdint>

#include "adamw_ckpt.h"

namespace osr {

// ---------------------------------------------------------------------------
// Error reporting: every failing entry point stores one line per thread.
// ---------------------------------------------------------------------------
int fail(int status, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
void clear_error();
const char* last_error_text();

// ---------------------------------------------------------------------------
// Norm reduction result, written by the last block of the norm kernel into
// device scratch (read by the fused step kernel) and into a pinned, mapped
// host mirror (read by adamw_last_norm without a copy).
// ---------------------------------------------------------------------------
struct NormResult {
    double sumsq;       // sum of g_i^2 of the raw gradient (fixed-order, double)
    double norm;        // grad_scale * sqrt(sumsq): the norm of the scaled gradient
    float scale;        // factor applied to raw g: grad_scale * clip factor
    int32_t nonfinite;  // 1 if norm is inf or nan (the step is skipped)
    uint32_t seq;       // incremented by every reduction (host staleness check)
    uint32_t fault;     // host mirror only: set by a one-launch step whose grid
                        // barrier wait ran out; cleared by the host
};

// The second level of a norm reduction whose kernel ran without its last
// block (partials only): every block of the fused kernel that follows sums
// partials[0..nparts) in the norm kernel's fixed order itself -- the same
// bits in every block -- and block 0 publishes the result record.
struct NormFinish {
    const double* partials;  // NULL: not used (the factor comes from elsewhere)
    int32_t nparts;
    double clip, grad_scale;
    NormResult* d_res;  // result record (device)
    NormResult* h_res;  // its host-mapped mirror (device address), may be NULL
};

// Per-step scalars, computed on the host in double and rounded to float once.
struct StepScalars {
    float beta1, omb1;      // beta1 and 1 - beta1
    float beta2, omb2;      // beta2 and 1 - beta2
    float eps;
    float step_size;        // lr / (1 - beta1^t)
    float inv_sqrt_bc2;     // 1 / sqrt(1 - beta2^t)
    float decay;            // 1 - lr * wd
    float scale;            // gradient factor when no norm result is read
    // Per-element decay flags (bit e % 32 of word e / 32 set: element e
    // decays); NULL: every element decays.
    const uint32_t* decay_mask;
    // Dynamic chunk scheduling of the fused kernel: [0] the next chunk to
    // hand out, [1] blocks done (both 0 between launches: the last block
    // out resets them).  NULL: chunks are dealt out cyclically by block.
    uint32_t* chunk_ctr;
    // Finish of the norm reduction in the fused kernel (see NormFinish).
    NormFinish fin;
};

// Tunables of the kernels (fixed at compile time; used in norm.cu, step.cu).
constexpr int kNormThreads = 256;
constexpr int kNormVecPerThread = 8;                 // float4 per thread per tile
constexpr int64_t kNormTileElems = int64_t(kNormThreads) * kNormVecPerThread * 4;
// At most 608 = 4 x 152 blocks: four 256-thread blocks of the norm kernel are
// resident per SM at its register count, so the grid is one wave on GB300.
// A constant, not derived from the device, so that results depend on n only.
constexpr int kNormBlocksMax = 608;

// Number of blocks of the norm reduction for n elements: a function of n
// only, so the reduction order (and hence every bit of the result) is too.
inline int norm_blocks(int64_t n)
{
    int64_t tiles = (n + kNormTileElems - 1) / kNormTileElems;
    if (tiles < 1) tiles = 1;
    return tiles > kNormBlocksMax ? kNormBlocksMax : int(tiles);
}

// Resident-block counts of the grid-stride kernels on this device (their
// grids are capped there: one wave of persistent blocks).
struct KernelCaps {
    int step_vec, step_scalar, pack_vec, pack_scalar;
};

// Kernel launchers (norm.cu, step.cu, pack.cu).  All return cudaError_t as int.
int query_step_caps(int sm_count, KernelCaps* caps);
int query_pack_caps(int sm_count, KernelCaps* caps);
// Per-tensor outputs of the norm kernel (see norm.cu).  offsets: n_tensors
// + 1 entries (the last is n); kfirst / segbase: per block, the first tensor
// its range touches and the index of its first segment slot; seg_sums: one
// double per (block, tensor) pair.
struct TensorSegs {
    const int64_t* offsets;
    const int32_t* kfirst;
    const int32_t* segbase;
    double* seg_sums;
};
// Block b of the norm kernel reduces the contiguous tiles
// [ntiles b / P, ntiles (b + 1) / P) (P = norm_blocks(n)).
inline int64_t norm_block_tile(int64_t n, int b)
{
    const int64_t ntiles = (n + kNormTileElems - 1) / kNormTileElems;
    return ntiles * int64_t(b) / int64_t(norm_blocks(n));
}

// The norm kernel publishes norm = grad_scale sqrt(sum g^2) and the factor
// applied to g: grad_scale * (norm > clip ? clip / norm : 1); with segs, also
// the per-tensor segment sums.
// Element types of the gradient and of the optional 16-bit weight copy.
constexpr int32_t kDtypeF32 = 0, kDtypeBF16 = 1, kDtypeF16 = 2;

// tail = false: the kernel only writes its P partials (no ticket, no last
// block); the fused kernel launched next finishes the reduction (NormFinish).
int launch_norm(const void* g, int64_t n, double clip, double* partials,
                unsigned int* counter, NormResult* d_res, NormResult* h_res_dev,
                void* stream, double grad_scale = 1.0, const TensorSegs* segs = nullptr,
                int32_t g_dtype = kDtypeF32, bool tail = true);
// g of type g_dtype (16-byte aligned for float32 on the vector path, 8-byte
// for 16-bit types); w_lp (may be NULL) receives the new weights rounded to
// w_lp_dtype (bfloat16 or binary16; 8-byte aligned).  16-bit types and the
// copy need 16-byte aligned w, m, v.
int launch_adamw(float* w, const void* g, float* m, float* v, int64_t n,
                 const StepScalars& k, const NormResult* d_res,
                 const KernelCaps& caps, void* stream, bool zero_grad = false,
                 bool programmatic = false, int32_t g_dtype = kDtypeF32,
                 void* w_lp = nullptr, int32_t w_lp_dtype = kDtypeBF16);
// The one-launch step (onepass.cu): norm, clip factor and update in one
// cooperative grid of onepass_grid(n, capacity) blocks; bar: two zeroed
// uint32 barrier counters; fault_test: wait for one block more than the grid
// has (the barrier times out).  w, g, m, v 16-byte aligned, float32 g.
int query_onepass_blocks(int sm_count, int* blocks_out);
// States of at most kClusterMaxN parameters (a norm partition of at most
// kClusterCtas blocks) take the one-launch step as one thread-block cluster
// with a hardware barrier instead of a cooperative grid (onepass.cu).
constexpr int kClusterCtas = 8;
constexpr int64_t kClusterMaxN = int64_t(kClusterCtas) * kNormTileElems;
bool onepass_is_cluster(int64_t n);
int onepass_grid(int64_t n, int capacity);
int launch_onepass(float* w, float* g, float* m, float* v, int64_t n, const StepScalars& k,
                   double clip, double grad_scale, double* partials, uint32_t* bar,
                   bool fault_test, NormResult* d_res, NormResult* h_res, int capacity,
                   bool zero_grad, void* stream);
// Staging slots -> the pinned host image (its device address), by a quarter
// of the SMs: header (8 bytes) then w, m, v at their file offsets.
int launch_stage_to_host(const unsigned char* header, const float* sw, const float* sm,
                         const float* sv, int64_t n, unsigned char* image_dev, int sm_count,
                         void* stream);
// The global result of a sharded state from the ranks' gathered sums of
// squares (ranks.cu): published to d_res / h_res like a norm reduction.
int launch_rank_total(const double* rank_sumsq, int32_t world, double clip, double grad_scale,
                      NormResult* d_res, NormResult* h_res, void* stream);
// Chunks are handed out by a counter (fused and pack kernels) from this many
// parameters up (measured on GB300: +3-8% from 2^24, where a block gets 13
// chunks or more; below, the counter's atomics and block barriers cost more
// than the balance saves, e.g. 0.86 vs 0.96 of peak at 2^22).
constexpr int64_t kDynamicChunksMinN = int64_t(1) << 24;
// States up to this many parameters take the one-launch step by default
// (measured on GB300: below about 2^20 it saves 2 us per step; from 2^20 up
// the two launches, which overlap, are faster).
constexpr int64_t kOnePassMaxN = int64_t(1) << 19;
// The pack: header (8 bytes, 8-byte aligned) and the w, m, v regions
// (16-byte aligned; 256-byte aligned for full speed) of the staging buffer.
int launch_pack(const float* w, const float* m, const float* v, int64_t n, int32_t step,
                unsigned char* header, float* dw, float* dm, float* dv, const KernelCaps& caps,
                void* stream, uint32_t* chunk_ctr = nullptr);

// Kernel-node parameters for a CUDA graph of one step (graph.cu).  The
// argument structs own the values that kernelParams point into.
// (The step graph's norm node runs without its last block: the fused node
// finishes the reduction.)
struct NormNodeArgs {
    const float* g;
    int64_t n;
    double clip, grad_scale;
    double* partials;
    unsigned int* counter;
    NormResult* d_res;
    NormResult* h_res;
    TensorSegs segs;
    void* ptrs[9];
};
struct AdamwNodeArgs {
    float* w;
    const float* g;
    float* m;
    float* v;
    int64_t n;
    StepScalars k;
    const NormResult* d_res;
    void* w_lp;  // always NULL in the step graph
    void* ptrs[8];
};
// The one-launch step as a single (cooperative) graph node.
struct OnepassNodeArgs {
    float* w;
    float* g;
    float* m;
    float* v;
    int64_t n;
    StepScalars k;
    double clip, grad_scale;
    double* partials;
    int32_t P;
    uint32_t* bar;
    uint32_t expect;
    NormResult* d_res;
    NormResult* h_res;
    void* ptrs[14];
};
}  // namespace osr
struct cudaKernelNodeParams;
namespace osr {
int norm_node_params(NormNodeArgs* a, cudaKernelNodeParams* p);
int adamw_node_params(AdamwNodeArgs* a, const KernelCaps& caps, cudaKernelNodeParams* p);
// fault_test: the node's barrier waits for one block more than its grid.
int onepass_node_params(OnepassNodeArgs* a, int capacity, bool fault_test,
                        cudaKernelNodeParams* p);

}  // namespace osr
