// ckpt_io.cpp -- host side of the step_NNNNNN.bin checkpoint: the atomic
// writer and the validating reader.  Plain POSIX, no CUDA.
//
// Format ("Grow a Language Model: Checkpoints", unhomeschool.com, sections
// "Format" and "Total size"): [int32 step][int32 n][n f32 w][n f32 m]
// [n f32 v], 8 + 12 n bytes, no other metadata; little-endian.
// Atomicity ("Checkpoint and Sharded Resume", AI Engineering from Scratch
// lesson 80, section "Atomic write"): write <name>.tmp, fsync, rename over
// <name>, fsync the directory.  Refusal of bad files (same page, "Three
// failure modes"): header, sign, parameter count and exact size are checked
// before any byte of the arrays is used.
#include <cerrno>
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <cstring>

#include <algorithm>
#include <atomic>
#include <csignal>
#include <string>
#include <utility>
#include <vector>

#include <dirent.h>
#include <fcntl.h>
#include <sys/stat.h>
#include <unistd.h>

#include "ckpt_io.h"
#include "internal.h"

namespace osr {

namespace {
thread_local char g_last_error[512];

bool little_endian_host()
{
    const uint32_t one = 1;
    unsigned char b;
    std::memcpy(&b, &one, 1);
    return b == 1;
}

void put_le32(unsigned char* p, uint32_t x)
{
    for (int i = 0; i < 4; ++i)
        p[i] = static_cast<unsigned char>((x >> (8 * i)) & 0xffu);
}

}  // namespace

uint32_t get_le32(const unsigned char* p)
{
    return uint32_t(p[0]) | (uint32_t(p[1]) << 8) | (uint32_t(p[2]) << 16) |
           (uint32_t(p[3]) << 24);
}

namespace {

int write_exact(int fd, const void* src, size_t bytes, const char* path, int* err_out = nullptr)
{
    const unsigned char* p = static_cast<const unsigned char*>(src);
    while (bytes > 0) {
        // Linux moves at most ~2 GiB per write(); loop on short writes.
        const size_t want = bytes > (size_t(1) << 30) ? (size_t(1) << 30) : bytes;
        const ssize_t got = ::write(fd, p, want);
        if (got < 0) {
            const int e = errno;
            if (e == EINTR)
                continue;
            if (err_out)
                *err_out = e;
            return fail(ADAMW_EIO, "write %s: %s", path, std::strerror(e));
        }
        p += got;
        bytes -= size_t(got);
    }
    return ADAMW_OK;
}
// fsync of the directory that holds a file just renamed, so that the rename
// itself is on disk.  A directory that cannot be opened read-only, or a file
// system that does not sync directories (fsync: EINVAL, ENOTSUP, EROFS), is
// tolerated; any other failure (EIO, ENOSPC, ...) means the rename may not be
// durable and is reported as ADAMW_EIO.
int sync_dir(const char* dir)
{
    const int dfd = ::open(dir, O_RDONLY | O_DIRECTORY | O_CLOEXEC);
    if (dfd < 0)
        return ADAMW_OK;
    int rc = ADAMW_OK;
    if (::fsync(dfd) != 0 && errno != EINVAL && errno != ENOTSUP && errno != EROFS)
        rc = fail(ADAMW_EIO, "fsync of directory %s: %s (the rename may not be durable)", dir,
                  std::strerror(errno));
    ::close(dfd);
    return rc;
}

}  // namespace

int fail(int status, const char* fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    std::vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
    va_end(ap);
    return status;
}

void clear_error() { g_last_error[0] = '\0'; }

const char* last_error_text() { return g_last_error; }

int read_exact(int fd, void* dst, size_t bytes, const char* path)
{
    unsigned char* p = static_cast<unsigned char*>(dst);
    while (bytes > 0) {
        const size_t want = bytes > (size_t(1) << 30) ? (size_t(1) << 30) : bytes;
        const ssize_t got = ::read(fd, p, want);
        if (got < 0) {
            if (errno == EINTR)
                continue;
            return fail(ADAMW_EIO, "read %s: %s", path, std::strerror(errno));
        }
        if (got == 0)
            return fail(ADAMW_ESIZE, "%s: file ended early", path);
        p += got;
        bytes -= size_t(got);
    }
    return ADAMW_OK;
}

int write_file_atomic(const char* dir, int32_t step, const IoPiece* pieces,
                      int npieces, char* path_out, size_t path_cap, int32_t flags)
{
    if (!dir || step < 0)
        return fail(ADAMW_EINVAL, "ckpt write: null directory or negative step");
    char name[32];
    std::snprintf(name, sizeof name, "step_%06d.bin", int(step));
    return write_named_file(dir, name, pieces, npieces, flags, path_out, path_cap);
}

int write_named_file(const char* dir, const char* name, const IoPiece* pieces, int npieces,
                     int32_t flags, char* path_out, size_t path_cap)
{
    if (!dir || !name)
        return fail(ADAMW_EINVAL, "ckpt write: null directory or name");
    if (!little_endian_host())
        return fail(ADAMW_EINVAL, "ckpt write: big-endian host not supported");
    char final_path[4096], tmp_path[4112];
    const int len = std::snprintf(final_path, sizeof final_path, "%s/%s", dir, name);
    if (len < 0 || size_t(len) >= sizeof final_path)
        return fail(ADAMW_EINVAL, "ckpt write: directory name too long");
    std::snprintf(tmp_path, sizeof tmp_path, "%s.tmp", final_path);

    // O_DIRECT moves the pinned image straight to the device (no page-cache
    // copy); it needs a block-aligned buffer, length and offset, so the last
    // partial block is written whole from the buffer's padding and the file
    // is then truncated to its exact size.
    const bool want_direct = (flags & kWriteDirect) && npieces == 1 &&
                             (reinterpret_cast<uintptr_t>(pieces[0].data) % kIoBlock) == 0 &&
                             pieces[0].capacity >= round_up_block(pieces[0].bytes);
    int fd = -1;
    bool direct = false;
    if (want_direct) {
        fd = ::open(tmp_path, O_WRONLY | O_CREAT | O_TRUNC | O_CLOEXEC | O_DIRECT, 0644);
        direct = fd >= 0;
    }
    if (fd < 0)  // not requested, or refused by the file system (e.g. EINVAL)
        fd = ::open(tmp_path, O_WRONLY | O_CREAT | O_TRUNC | O_CLOEXEC, 0644);
    if (fd < 0)
        return fail(ADAMW_EIO, "open %s: %s", tmp_path, std::strerror(errno));
    int rc = ADAMW_OK;
    if (direct) {
        const size_t whole = round_up_block(pieces[0].bytes);
        int werr = 0;
        rc = write_exact(fd, pieces[0].data, whole, tmp_path, &werr);
        if (rc != ADAMW_OK && werr == EINVAL) {
            // the device refused this alignment after all: rewrite buffered
            ::close(fd);
            fd = ::open(tmp_path, O_WRONLY | O_CREAT | O_TRUNC | O_CLOEXEC, 0644);
            if (fd < 0)
                return fail(ADAMW_EIO, "open %s: %s", tmp_path, std::strerror(errno));
            direct = false;
            rc = write_exact(fd, pieces[0].data, pieces[0].bytes, tmp_path);
        } else if (rc == ADAMW_OK && ::ftruncate(fd, off_t(pieces[0].bytes)) != 0) {
            rc = fail(ADAMW_EIO, "ftruncate %s: %s", tmp_path, std::strerror(errno));
        }
    } else {
        for (int i = 0; i < npieces && rc == ADAMW_OK; ++i)
            rc = write_exact(fd, pieces[i].data, pieces[i].bytes, tmp_path);
    }
    if (rc == ADAMW_OK && ::fsync(fd) != 0)
        rc = fail(ADAMW_EIO, "fsync %s: %s", tmp_path, std::strerror(errno));
    if (::close(fd) != 0 && rc == ADAMW_OK)
        rc = fail(ADAMW_EIO, "close %s: %s", tmp_path, std::strerror(errno));
    if (rc != ADAMW_OK) {
        ::unlink(tmp_path);
        return rc;
    }
    if (::rename(tmp_path, final_path) != 0) {
        rc = fail(ADAMW_EIO, "rename %s: %s", tmp_path, std::strerror(errno));
        ::unlink(tmp_path);
        return rc;
    }
    if ((rc = sync_dir(dir)) != ADAMW_OK)
        return rc;
    if (path_out && path_cap > 0) {
        if (size_t(len) + 1 > path_cap)
            return fail(ADAMW_EINVAL, "ckpt write: path buffer too small (file written)");
        std::memcpy(path_out, final_path, size_t(len) + 1);
    }
    return ADAMW_OK;
}

// Checkpoint rotation ("Checkpoint and Sharded Resume", lesson 80, section
// "Production patterns in the wild": keep the last K checkpoints and delete
// the oldest, or the disk fills up mid-run and the next write fails).
int rotate_files(const char* dir, int32_t keep, int32_t* removed)
{
    if (removed)
        *removed = 0;
    if (!dir || keep < 0)
        return fail(ADAMW_EINVAL, "ckpt rotate: null directory or negative keep");
    if (keep == 0)
        return ADAMW_OK;
    DIR* d = ::opendir(dir);
    if (!d)
        return fail(ADAMW_EIO, "opendir %s: %s", dir, std::strerror(errno));
    std::vector<std::pair<long long, std::string>> files;
    while (struct dirent* e = ::readdir(d)) {
        const char* nm = e->d_name;
        const size_t L = std::strlen(nm);
        if (L < 10 || std::strncmp(nm, "step_", 5) != 0 || std::strcmp(nm + L - 4, ".bin") != 0)
            continue;
        bool digits = L - 9 <= 12;
        for (size_t i = 5; i < L - 4 && digits; ++i)
            digits = nm[i] >= '0' && nm[i] <= '9';
        if (!digits)
            continue;
        files.emplace_back(std::atoll(std::string(nm + 5, L - 9).c_str()), std::string(nm));
    }
    ::closedir(d);
    std::sort(files.begin(), files.end(),
              [](const auto& a, const auto& b) { return a.first > b.first; });
    int rc = ADAMW_OK;
    for (size_t i = size_t(keep); i < files.size(); ++i) {
        const std::string p = std::string(dir) + "/" + files[i].second;
        if (::unlink(p.c_str()) != 0)
            rc = fail(ADAMW_EIO, "unlink %s: %s", p.c_str(), std::strerror(errno));
        else if (removed)
            ++*removed;
    }
    return rc;
}

int pread_exact(int fd, void* dst, size_t bytes, int64_t offset, const char* path)
{
    unsigned char* p = static_cast<unsigned char*>(dst);
    while (bytes > 0) {
        const size_t want = bytes > (size_t(1) << 30) ? (size_t(1) << 30) : bytes;
        const ssize_t got = ::pread(fd, p, want, off_t(offset));
        if (got < 0) {
            if (errno == EINTR)
                continue;
            return fail(ADAMW_EIO, "read %s: %s", path, std::strerror(errno));
        }
        if (got == 0)
            return fail(ADAMW_ESIZE, "%s: file ended early", path);
        p += got;
        offset += got;
        bytes -= size_t(got);
    }
    return ADAMW_OK;
}

AtomicFile::~AtomicFile()
{
    if (fd_ >= 0) {
        ::close(fd_);
        ::unlink(tmp_.c_str());
    }
}

int AtomicFile::open(const char* dir, const char* name)
{
    if (!dir || !name)
        return fail(ADAMW_EINVAL, "ckpt write: null directory or name");
    if (fd_ >= 0)
        return fail(ADAMW_ESTATE, "ckpt write: file already open");
    dir_ = dir;
    final_ = dir_ + "/" + name;
    tmp_ = final_ + ".tmp";
    if (final_.size() >= 4096)
        return fail(ADAMW_EINVAL, "ckpt write: directory name too long");
    fd_ = ::open(tmp_.c_str(), O_WRONLY | O_CREAT | O_TRUNC | O_CLOEXEC, 0644);
    if (fd_ < 0)
        return fail(ADAMW_EIO, "open %s: %s", tmp_.c_str(), std::strerror(errno));
    return ADAMW_OK;
}

int AtomicFile::write(const void* data, size_t bytes)
{
    if (fd_ < 0)
        return fail(ADAMW_ESTATE, "ckpt write: no open file");
    return write_exact(fd_, data, bytes, tmp_.c_str());
}

int AtomicFile::commit(char* path_out, size_t path_cap)
{
    if (fd_ < 0)
        return fail(ADAMW_ESTATE, "ckpt write: no open file");
    int rc = ADAMW_OK;
    if (::fsync(fd_) != 0)
        rc = fail(ADAMW_EIO, "fsync %s: %s", tmp_.c_str(), std::strerror(errno));
    if (::close(fd_) != 0 && rc == ADAMW_OK)
        rc = fail(ADAMW_EIO, "close %s: %s", tmp_.c_str(), std::strerror(errno));
    fd_ = -1;
    if (rc == ADAMW_OK && ::rename(tmp_.c_str(), final_.c_str()) != 0)
        rc = fail(ADAMW_EIO, "rename %s: %s", tmp_.c_str(), std::strerror(errno));
    if (rc != ADAMW_OK) {
        ::unlink(tmp_.c_str());
        return rc;
    }
    if ((rc = sync_dir(dir_.c_str())) != ADAMW_OK)
        return rc;
    if (path_out && path_cap > 0) {
        if (final_.size() + 1 > path_cap)
            return fail(ADAMW_EINVAL, "ckpt write: path buffer too small (file written)");
        std::memcpy(path_out, final_.c_str(), final_.size() + 1);
    }
    return ADAMW_OK;
}

int open_validated(const char* path, int32_t n_expected, int32_t* step_out,
                   int32_t* n_out, int* fd_out)
{
    *fd_out = -1;
    if (!path)
        return fail(ADAMW_EINVAL, "ckpt read: null path");
    if (!little_endian_host())
        return fail(ADAMW_EINVAL, "ckpt read: big-endian host not supported");
    const int fd = ::open(path, O_RDONLY | O_CLOEXEC);
    if (fd < 0)
        return fail(ADAMW_EIO, "open %s: %s", path, std::strerror(errno));
    struct stat st;
    if (::fstat(fd, &st) != 0) {
        const int e = errno;
        ::close(fd);
        return fail(ADAMW_EIO, "stat %s: %s", path, std::strerror(e));
    }
    unsigned char header[8];
    if (st.st_size < 8) {
        ::close(fd);
        return fail(ADAMW_ESIZE, "%s: %lld bytes, shorter than the 8-byte header", path,
                    (long long)st.st_size);
    }
    int rc = read_exact(fd, header, 8, path);
    if (rc != ADAMW_OK) {
        ::close(fd);
        return rc;
    }
    const int32_t step = int32_t(get_le32(header));
    const int32_t n = int32_t(get_le32(header + 4));
    if (step < 0 || n < 0) {
        ::close(fd);
        return fail(ADAMW_EFORMAT, "%s: header step=%d n=%d (negative)", path, step, n);
    }
    if (n_expected >= 0 && n != n_expected) {
        ::close(fd);
        return fail(ADAMW_EMISMATCH, "%s: holds %d parameters, expected %d", path, n,
                    n_expected);
    }
    const int64_t want = 8 + 12 * int64_t(n);
    if (int64_t(st.st_size) != want) {
        ::close(fd);
        return fail(ADAMW_ESIZE, "%s: %lld bytes, expected 8 + 12 x %d = %lld", path,
                    (long long)st.st_size, n, (long long)want);
    }
    if (step_out)
        *step_out = step;
    if (n_out)
        *n_out = n;
    *fd_out = fd;
    return ADAMW_OK;
}

}  // namespace osr

extern "C" {

int64_t ckpt_file_size(int64_t n)
{
    if (n < 0 || n > INT32_MAX)
        return -1;
    return 8 + 12 * n;
}

int ckpt_write_host(const char* dir, int32_t step, int32_t n, const float* h_w,
                    const float* h_m, const float* h_v, char* path_out,
                    size_t path_cap)
{
    osr::clear_error();
    if (n < 0 || (n > 0 && (!h_w || !h_m || !h_v)))
        return osr::fail(ADAMW_EINVAL, "ckpt_write_host: bad n or null array");
    unsigned char header[8];
    osr::put_le32(header, uint32_t(step));
    osr::put_le32(header + 4, uint32_t(n));
    const size_t bytes = size_t(n) * 4u;
    const osr::IoPiece pieces[4] = {
        {header, 8, 8}, {h_w, bytes, bytes}, {h_m, bytes, bytes}, {h_v, bytes, bytes}};
    return osr::write_file_atomic(dir, step, pieces, 4, path_out, path_cap);
}

int ckpt_write_image(const char* dir, const void* image, int64_t bytes, int64_t capacity,
                     int32_t flags, char* path_out, size_t path_cap)
{
    osr::clear_error();
    if (!image || bytes < 8 || capacity < bytes)
        return osr::fail(ADAMW_EINVAL, "ckpt_write_image: null image or bad sizes");
    const unsigned char* h = static_cast<const unsigned char*>(image);
    const int32_t step = int32_t(osr::get_le32(h));
    const int32_t n = int32_t(osr::get_le32(h + 4));
    if (step < 0 || n < 0 || bytes != 8 + 12 * int64_t(n))
        return osr::fail(ADAMW_EINVAL,
                         "ckpt_write_image: header step=%d n=%d does not describe %lld bytes", step,
                         n, (long long)bytes);
    const osr::IoPiece piece{image, size_t(bytes), size_t(capacity)};
    return osr::write_file_atomic(dir, step, &piece, 1, path_out, path_cap,
                                  flags & osr::kWriteDirect);
}

int ckpt_rotate(const char* dir, int32_t keep, int32_t* removed)
{
    osr::clear_error();
    return osr::rotate_files(dir, keep, removed);
}

// ---------------------------------------------------------------------------
// Signals ("Grow a Language Model: Checkpoints", section "SIGTERM & SIGUSR1"):
// SIGTERM = finish the step, write a checkpoint, exit; SIGUSR1 = finish the
// step, write a checkpoint, continue.  The handler only records the request;
// the training loop acts on it at the next step boundary.
// ---------------------------------------------------------------------------
namespace {
std::atomic<int> g_signal_requests{0};
static_assert(std::atomic<int>::is_always_lock_free, "signal flag must be lock-free");

extern "C" void on_ckpt_signal(int sig)
{
    g_signal_requests.fetch_or(sig == SIGTERM ? CKPT_REQ_EXIT : CKPT_REQ_WRITE);
}
}  // namespace

int ckpt_signals_install(int32_t mask)
{
    osr::clear_error();
    if (mask & ~(CKPT_REQ_WRITE | CKPT_REQ_EXIT))
        return osr::fail(ADAMW_EINVAL, "ckpt_signals_install: unknown mask bits 0x%x", mask);
    struct sigaction sa;
    std::memset(&sa, 0, sizeof sa);
    sa.sa_handler = on_ckpt_signal;
    sigemptyset(&sa.sa_mask);
    sa.sa_flags = SA_RESTART;
    if ((mask & CKPT_REQ_WRITE) && ::sigaction(SIGUSR1, &sa, nullptr) != 0)
        return osr::fail(ADAMW_EINVAL, "sigaction(SIGUSR1): %s", std::strerror(errno));
    if ((mask & CKPT_REQ_EXIT) && ::sigaction(SIGTERM, &sa, nullptr) != 0)
        return osr::fail(ADAMW_EINVAL, "sigaction(SIGTERM): %s", std::strerror(errno));
    return ADAMW_OK;
}

int32_t ckpt_signals_take(void) { return g_signal_requests.exchange(0); }

int ckpt_probe(const char* path, int32_t n_expected, int32_t* step_out, int32_t* n_out)
{
    osr::clear_error();
    int fd = -1;
    const int rc = osr::open_validated(path, n_expected, step_out, n_out, &fd);
    if (fd >= 0)
        ::close(fd);
    return rc;
}

const char* adamw_strerror(int status)
{
    switch (status) {
    case ADAMW_OK: return "ADAMW_OK";
    case ADAMW_EINVAL: return "ADAMW_EINVAL: invalid argument";
    case ADAMW_ECUDA: return "ADAMW_ECUDA: CUDA runtime error";
    case ADAMW_EIO: return "ADAMW_EIO: file I/O error";
    case ADAMW_EFORMAT: return "ADAMW_EFORMAT: bad checkpoint header";
    case ADAMW_ESIZE: return "ADAMW_ESIZE: checkpoint size is not 8 + 12 n";
    case ADAMW_EMISMATCH: return "ADAMW_EMISMATCH: checkpoint parameter count differs";
    case ADAMW_ENONFINITE: return "ADAMW_ENONFINITE: gradient norm is not finite";
    case ADAMW_ESTATE: return "ADAMW_ESTATE: call out of order";
    default: return "unknown status";
    }
}

const char* adamw_last_error(void) { return osr::last_error_text(); }

}  // extern "C"
