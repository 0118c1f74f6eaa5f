// writer.cu -- the context's checkpoint writer thread, asynchronous writes,
// rotation options, and the step-boundary checkpoint policy.
//
// "Grow a Language Model: Checkpoints" (unhomeschool.com): a checkpoint
// every 100 steps (section "Five decisions", cadence), SIGTERM = write and
// exit, SIGUSR1 = write and continue, both after the step in flight (section
// "SIGTERM & SIGUSR1").  "Checkpoint and Sharded Resume" (AI Engineering from
// Scratch, lesson 80), sections "Production patterns in the wild" and
// "Exercises": write asynchronously on a separate thread so training
// continues, block the next save until the previous one finished, keep only
// the newest K checkpoints.
//
// One write is in flight at most: the pinned host image is single-buffered,
// so the next pack (which copies into it) waits on the host for the writer.
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <string>
#include <vector>

#include <cuda_runtime.h>
#include <unistd.h>

#include "context.h"
#include "internal.h"

namespace osr {
namespace {

void writer_main(adamw_ctx* c)
{
    cudaSetDevice(c->device);
    WriterState& w = c->writer;
    std::unique_lock<std::mutex> lk(w.mu);
    for (;;) {
        w.cv.wait(lk, [&] { return w.stop || w.pending; });
        if (!w.pending)
            break;  // asked to stop, nothing queued
        w.pending = false;
        w.running = true;
        const std::string dir = w.dir;
        const int32_t step = w.step;
        const int32_t keep = c->keep;
        const int32_t flags = c->write_flags;
        lk.unlock();

        clear_error();
        int rc = ADAMW_OK;
        char path[4200] = {0};
        const cudaError_t e = cudaEventSynchronize(c->ev_d2h);
        if (e != cudaSuccess) {
            rc = fail(ADAMW_ECUDA, "waiting for the checkpoint copy: %s", cudaGetErrorString(e));
        } else {
            const IoPiece piece{c->h_image(), c->image_bytes(), c->h_image_capacity()};
            rc = write_file_atomic(dir.c_str(), step, &piece, 1, path, sizeof path, flags);
            if (rc == ADAMW_OK && keep > 0)
                rc = rotate_files(dir.c_str(), keep, nullptr);
        }
        const std::string err = rc == ADAMW_OK ? std::string() : std::string(last_error_text());

        lk.lock();
        w.running = false;
        w.have_result = true;
        w.collected = false;
        w.status = rc;
        w.error = err;
        w.path = path;
        w.cv.notify_all();
    }
}

}  // namespace

void writer_drain(adamw_ctx* c)
{
    WriterState& w = c->writer;
    if (!w.started)
        return;
    std::unique_lock<std::mutex> lk(w.mu);
    w.cv.wait(lk, [&] { return !w.pending && !w.running; });
}

void writer_stop(adamw_ctx* c)
{
    WriterState& w = c->writer;
    if (!w.started)
        return;
    {
        std::lock_guard<std::mutex> lk(w.mu);
        w.stop = true;
    }
    w.cv.notify_all();
    w.thread.join();
    w.started = false;
}

}  // namespace osr

extern "C" {

int ckpt_write_async(adamw_ctx* ctx, const char* dir)
{
    osr::clear_error();
    if (!ctx || !dir)
        return osr::fail(ADAMW_EINVAL, "ctx or dir is NULL");
    if (!ctx->packed)
        return osr::fail(ADAMW_ESTATE, "no packed checkpoint: call ckpt_pack first");
    osr::writer_drain(ctx);
    osr::WriterState& w = ctx->writer;
    {
        std::lock_guard<std::mutex> lk(w.mu);
        if (w.have_result && !w.collected && w.status != ADAMW_OK) {
            w.collected = true;
            return osr::fail(w.status, "the previous asynchronous checkpoint write failed: %s",
                             w.error.c_str());
        }
        if (!w.started) {
            w.stop = false;
            w.thread = std::thread(osr::writer_main, ctx);
            w.started = true;
        }
        w.dir = dir;
        w.step = ctx->packed_step;
        w.pending = true;
    }
    w.cv.notify_all();
    return ADAMW_OK;
}

int ckpt_wait(adamw_ctx* ctx, char* path_out, size_t path_cap)
{
    osr::clear_error();
    if (!ctx)
        return osr::fail(ADAMW_EINVAL, "ctx is NULL");
    osr::writer_drain(ctx);
    osr::WriterState& w = ctx->writer;
    std::lock_guard<std::mutex> lk(w.mu);
    if (path_out && path_cap > 0)
        path_out[0] = '\0';
    if (!w.have_result)
        return ADAMW_OK;
    w.collected = true;
    if (w.status != ADAMW_OK)
        return osr::fail(w.status, "%s", w.error.c_str());
    if (path_out && path_cap > 0) {
        if (w.path.size() + 1 > path_cap)
            return osr::fail(ADAMW_EINVAL, "path buffer too small (file written)");
        std::memcpy(path_out, w.path.c_str(), w.path.size() + 1);
    }
    return ADAMW_OK;
}

int ckpt_write(adamw_ctx* ctx, const char* dir, char* path_out, size_t path_cap)
{
    const int rc = ckpt_write_async(ctx, dir);
    if (rc != ADAMW_OK)
        return rc;
    return ckpt_wait(ctx, path_out, path_cap);
}

int ckpt_set_options(adamw_ctx* ctx, int32_t keep, int32_t flags)
{
    osr::clear_error();
    if (!ctx)
        return osr::fail(ADAMW_EINVAL, "ctx is NULL");
    if (keep < 0 || (flags & ~(CKPT_DIRECT | CKPT_COPY_ENGINE)))
        return osr::fail(ADAMW_EINVAL, "keep=%d must be >= 0; unknown flags 0x%x", keep, flags);
    osr::writer_drain(ctx);
    ctx->keep = keep;
    ctx->write_flags = (flags & CKPT_DIRECT) ? osr::kWriteDirect : 0;
    ctx->copy_engine = (flags & CKPT_COPY_ENGINE) != 0;
    return ADAMW_OK;
}

int ckpt_step_end(adamw_ctx* ctx, int32_t step, const float* d_w, const float* d_m,
                  const float* d_v, void* main_stream, void* side_stream, const char* dir,
                  int32_t every, int32_t* action_out)
{
    osr::clear_error();
    if (action_out)
        *action_out = CKPT_ACTION_NONE;
    if (!ctx || !dir || every < 0)
        return osr::fail(ADAMW_EINVAL, "ckpt_step_end: null ctx/dir or negative cadence");
    const int32_t req = ckpt_signals_take();
    const bool due = every > 0 && step > 0 && step % every == 0;
    if (!due && !req)
        return ADAMW_OK;
    int rc = ckpt_pack(ctx, step, d_w, d_m, d_v, main_stream, side_stream);
    if (rc != ADAMW_OK)
        return rc;
    if (req & CKPT_REQ_EXIT) {
        rc = ckpt_write(ctx, dir, nullptr, 0);
        if (rc == ADAMW_OK && action_out)
            *action_out = CKPT_ACTION_EXIT;
        return rc;
    }
    rc = ckpt_write_async(ctx, dir);
    if (rc == ADAMW_OK && action_out)
        *action_out = CKPT_ACTION_WRITING;
    return rc;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Sharded checkpoint, GPU side ("Checkpoint and Sharded Resume", lesson 80):
// this context holds one rank's shard of the flat state.
// ---------------------------------------------------------------------------
extern "C" {

int ckpt_shard_write(adamw_ctx* ctx, const char* dir, int32_t rank, char* sha256_hex_out)
{
    osr::clear_error();
    if (!ctx || !dir || rank < 0 || !sha256_hex_out)
        return osr::fail(ADAMW_EINVAL, "ckpt_shard_write: bad arguments");
    if (!ctx->packed)
        return osr::fail(ADAMW_ESTATE, "no packed checkpoint: call ckpt_pack first");
    osr::writer_drain(ctx);
    {
        const cudaError_t e = cudaEventSynchronize(ctx->ev_d2h);
        if (e != cudaSuccess)
            return osr::fail(ADAMW_ECUDA, "waiting for the checkpoint copy: %s",
                             cudaGetErrorString(e));
    }
    ctx->d2h_pending = false;
    std::string staging;
    int rc = osr::shard_staging_dir(dir, ctx->packed_step, &staging);
    if (rc != ADAMW_OK)
        return rc;
    char name[64];
    std::snprintf(name, sizeof name, "rank%d.bin", int(rank));
    const osr::IoPiece piece{ctx->h_image(), ctx->image_bytes(), ctx->h_image_capacity()};
    rc = osr::write_named_file(staging.c_str(), name, &piece, 1, ctx->write_flags);
    if (rc != ADAMW_OK)
        return rc;
    osr::Sha256 h;
    h.update(ctx->h_image(), ctx->image_bytes());
    if (!h.final_hex(sha256_hex_out))
        return osr::fail(ADAMW_EIO, "%s: the digest could not be computed", name);
    return ADAMW_OK;
}

int ckpt_shard_read(adamw_ctx* ctx, const char* step_dir, int32_t rank, int32_t expected_world,
                    int32_t* step_out, float* d_w, float* d_m, float* d_v, void* stream)
{
    osr::clear_error();
    if (!ctx || !step_dir || rank < 0 || !d_w || !d_m || !d_v)
        return osr::fail(ADAMW_EINVAL, "ckpt_shard_read: bad arguments");
    if (!ctx->has_ckpt)
        return osr::fail(ADAMW_ESTATE, "context was created without checkpoint staging");
    std::vector<int64_t> off, num;
    std::vector<std::string> paths, digests;
    int32_t step = -1;
    // manifest and every shard's size and header; this rank's digest below
    int rc = osr::load_manifest(step_dir, expected_world, false, &step, &off, &num, &paths,
                                &digests);
    if (rc != ADAMW_OK)
        return rc;
    if (rank >= int32_t(off.size()))
        return osr::fail(ADAMW_EMISMATCH, "rank %d of a %zu-shard checkpoint", rank, off.size());
    if (num[size_t(rank)] != ctx->n)
        return osr::fail(ADAMW_EMISMATCH, "shard %d holds %lld parameters, context has %lld",
                         rank, (long long)num[size_t(rank)], (long long)ctx->n);
    osr::writer_drain(ctx);
    if (ctx->d2h_pending) {
        const cudaError_t e = cudaEventSynchronize(ctx->ev_d2h);
        if (e != cudaSuccess)
            return osr::fail(ADAMW_ECUDA, "cudaEventSynchronize: %s", cudaGetErrorString(e));
        ctx->d2h_pending = false;
    }
    const std::string path = std::string(step_dir) + "/" + paths[size_t(rank)];
    int fd = -1;
    int32_t fstep = -1, fn = -1;
    rc = osr::open_validated(path.c_str(), int32_t(ctx->n), &fstep, &fn, &fd);
    if (rc != ADAMW_OK)
        return rc;
    ctx->packed = false;  // the pinned image now holds the file
    unsigned char* img = ctx->h_image();
    for (int i = 0; i < 4; ++i) {
        img[i] = static_cast<unsigned char>((uint32_t(fstep) >> (8 * i)) & 0xffu);
        img[4 + i] = static_cast<unsigned char>((uint32_t(fn) >> (8 * i)) & 0xffu);
    }
    const size_t bytes = size_t(ctx->n) * 4u;
    rc = osr::read_exact(fd, img + 8, 3 * bytes, path.c_str());
    ::close(fd);
    if (rc != ADAMW_OK)
        return rc;
    char hex[65];
    osr::Sha256 h;
    h.update(img, ctx->image_bytes());
    if (!h.final_hex(hex))
        return osr::fail(ADAMW_EIO, "%s: the digest could not be computed", path.c_str());
    if (digests[size_t(rank)] != hex)
        return osr::fail(ADAMW_EFORMAT, "%s: sha256 %s, manifest says %s (partial or corrupted "
                         "write)", path.c_str(), hex, digests[size_t(rank)].c_str());
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    if ((e = cudaMemcpyAsync(d_w, img + 8, bytes, cudaMemcpyHostToDevice, s)) != cudaSuccess ||
        (e = cudaMemcpyAsync(d_m, img + 8 + bytes, bytes, cudaMemcpyHostToDevice, s)) !=
            cudaSuccess ||
        (e = cudaMemcpyAsync(d_v, img + 8 + 2 * bytes, bytes, cudaMemcpyHostToDevice, s)) !=
            cudaSuccess ||
        (e = cudaStreamSynchronize(s)) != cudaSuccess)
        return osr::fail(ADAMW_ECUDA, "shard upload: %s", cudaGetErrorString(e));
    if (step_out)
        *step_out = step;
    return ADAMW_OK;
}

}  // extern "C"
