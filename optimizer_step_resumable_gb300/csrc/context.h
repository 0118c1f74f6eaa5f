// context.h -- the adamw_ctx object behind the C ABI (internal).
#pragma once

#include <condition_variable>
#include <cstdint>
#include <mutex>
#include <string>
#include <thread>
#include <vector>

#include <cuda_runtime.h>

#include "ckpt_io.h"
#include "internal.h"

namespace osr {

// The context's checkpoint writer thread and its one-slot job queue: at most
// one write is queued or running at a time.
struct WriterState {
    std::thread thread;
    std::mutex mu;
    std::condition_variable cv;
    bool started = false, stop = false;
    bool pending = false, running = false;  // a job queued / being written
    // the job
    std::string dir;
    int32_t step = -1;
    // result of the last finished job
    bool have_result = false, collected = true;
    int status = ADAMW_OK;
    std::string error, path;
};

}  // namespace osr

struct adamw_ctx {
    int64_t n = 0;
    std::vector<int64_t> offsets, numels;
    int device = -1;
    int sm_count = 0;
    osr::KernelCaps caps{};
    double beta1 = 0.9, beta2 = 0.999, eps = 1e-8;

    // norm scratch: [NormResult | counter | barrier x 2 | chunk counters x 2 |
    //                pack counters x 2 | pad]
    //               [partials x kNormBlocksMax]
    unsigned char* d_scratch = nullptr;
    osr::NormResult* d_res = nullptr;
    unsigned int* d_counter = nullptr;
    double* d_partials = nullptr;
    osr::NormResult* h_res = nullptr;      // pinned, mapped: host view
    osr::NormResult* h_res_dev = nullptr;  // device view of the same memory
    cudaEvent_t ev_norm = nullptr;
    bool norm_launched = false;

    // Per-tensor sums of squares: the table on the device, the norm grid's
    // per-block segment layout (host and device), the segment sums.
    int64_t* d_tab_offsets = nullptr;  // n_tensors + 1 (last = n)
    int32_t* d_kfirst = nullptr;       // per norm block
    int32_t* d_segbase = nullptr;      // per norm block + 1
    double* d_seg_sums = nullptr;
    double* h_seg_sums = nullptr;      // pinned
    std::vector<int32_t> kfirst, segbase;
    int32_t nseg = 0;
    bool segs_launched = false;        // the last reduction also wrote segments
    cudaEvent_t prof[3] = {nullptr, nullptr, nullptr};  // one-shot instrumentation
    bool pdl = true;  // launch the fused kernel as a programmatic dependent
    // One-launch step for small states: cooperative grid capacity, barrier
    // counters (in the scratch head), enabled, size limit, one-shot test of
    // the barrier timeout.
    int onepass_capacity = 0;
    uint32_t* d_bar = nullptr;
    uint32_t* d_chunk_ctr = nullptr;  // the fused kernel's chunk counters
    uint32_t* d_pack_ctr = nullptr;   // the pack kernel's (its own: it may run on another stream)
    bool dynamic_chunks = true;
    bool onepass = true;
    int64_t onepass_max_n = 0;
    bool onepass_fault_test = false;
    // Per-tensor decay flags expanded to one bit per element (allocated by
    // the first adamw_set_decay_mask that exempts a tensor).
    uint32_t* d_decay_mask = nullptr;
    bool decay_mask_on = false;

    // Checkpoint staging.  On the device: the 8-byte header and the w, m, v
    // regions each in its own 256-byte aligned slot (d_stage(r), r = 0 for the
    // header, 1..3 for w, m, v), so that the pack kernel's stores start on
    // cache-line boundaries; the copy to the host puts them at their file
    // offsets.  On the host: the file image, contiguous, at the (page-aligned)
    // start of its allocation, padded to a whole number of 4 KiB blocks, so
    // that the writer can hand it to the disk with O_DIRECT.
    bool has_ckpt = false;
    unsigned char* d_image_alloc = nullptr;
    unsigned char* h_image_alloc = nullptr;
    cudaEvent_t ev_pack = nullptr, ev_d2h = nullptr;
    bool packed = false, d2h_pending = false;
    int32_t packed_step = -1;

    // A CUDA graph of one step (graph.cu): norm node -> fused-kernel node.
    cudaGraph_t graph = nullptr;
    cudaGraphExec_t graph_exec = nullptr;
    cudaGraphNode_t graph_norm = nullptr, graph_step = nullptr;
    float* graph_w = nullptr;
    const float* graph_g = nullptr;
    float* graph_m = nullptr;
    float* graph_v = nullptr;
    bool graph_mask = false;  // the graph's fused node reads decay flags
    bool graph_onepass = false;  // one node, the one-launch step (graph_norm), not two

    // Checkpoint writing: options and the writer thread.
    int32_t keep = 0;                   // rotation: newest files kept (0 = all)
    int32_t write_flags = osr::kWriteDirect;
    bool copy_engine = false;  // staging -> host by cudaMemcpyAsync, not the SM kernel
    unsigned char* h_image_dev = nullptr;  // device address of the pinned host image
    osr::WriterState writer;

    static constexpr size_t kStageAlign = 256;
    size_t stage_region_bytes() const
    {
        return (size_t(4) * size_t(n) + kStageAlign - 1) / kStageAlign * kStageAlign;
    }
    size_t stage_bytes() const { return kStageAlign + 3 * stage_region_bytes(); }
    unsigned char* d_stage(int r) const
    {
        return d_image_alloc + (r == 0 ? 0 : kStageAlign + size_t(r - 1) * stage_region_bytes());
    }
    unsigned char* h_image() const { return h_image_alloc; }
    size_t image_bytes() const { return size_t(8 + 12 * n); }
    size_t h_image_capacity() const { return osr::round_up_block(image_bytes()); }
};


namespace osr {
// Waits (host side) until the context's writer holds no job; afterwards the
// pinned image may be overwritten.  No-op when no writer thread was started.
void writer_drain(adamw_ctx* c);
// Lets the writer finish its queued job, then joins the thread.
void writer_stop(adamw_ctx* c);
// Per-step scalars (bias corrections, step size, decay) from the context's
// betas and eps, computed in double and rounded to float once (api.cu).
StepScalars make_step_scalars(const adamw_ctx* c, int32_t t, double lr, double wd);
// Frees the context's step graph, if any (graph.cu).
void graph_release(adamw_ctx* c);
}  // namespace osr
