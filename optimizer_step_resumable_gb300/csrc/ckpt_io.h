// ckpt_io.h -- host-side checkpoint file I/O shared by the library's
// translation units: the atomic writers, the validating readers, SHA-256 and
// the sharded manifest (internal; plain POSIX, no CUDA).
#pragma once

#include <cstddef>
#include <cstdint>
#include <string>
#include <vector>

namespace osr {

// Host file I/O (ckpt_io.cpp).
constexpr size_t kIoBlock = 4096;  // O_DIRECT alignment of address, length and offset
inline size_t round_up_block(size_t b) { return (b + kIoBlock - 1) / kIoBlock * kIoBlock; }
constexpr int32_t kWriteDirect = 1;  // try O_DIRECT (falls back when refused)

struct IoPiece {
    const void* data;
    size_t bytes;
    size_t capacity;  // readable bytes at data (>= bytes); O_DIRECT needs
                      // round_up_block(bytes)
};
// Writes the pieces, in order, to <dir>/step_%06d.bin atomically.  With
// kWriteDirect and a single 4 KiB-aligned piece of enough capacity, the data
// goes to the disk with O_DIRECT (whole blocks, then ftruncate to size).
int write_file_atomic(const char* dir, int32_t step, const IoPiece* pieces,
                      int npieces, char* path_out, size_t path_cap, int32_t flags = 0);
// The same for any file name in dir (used for the shard files).
int write_named_file(const char* dir, const char* name, const IoPiece* pieces, int npieces,
                     int32_t flags, char* path_out = nullptr, size_t path_cap = 0);
// Deletes all but the `keep` newest step_<digits>.bin files of dir.
int rotate_files(const char* dir, int32_t keep, int32_t* removed);

// SHA-256 (FIPS 180-4), incremental (sha256.cpp).  The digest is computed
// by the system's libcrypto (OpenSSL 3, which uses the CPU's SHA
// instructions) when it can be loaded, else by the library's own code from
// the standard; both give the same digest.  OSR_SHA256=builtin in the
// environment (read once, at the first digest) selects the library's own.
class Sha256 {
public:
    Sha256() { reset(); }
    ~Sha256();
    Sha256(const Sha256&) = delete;
    Sha256& operator=(const Sha256&) = delete;
    void reset();
    void update(const void* data, size_t bytes);
    // 64 lowercase hex digits + NUL; false if libcrypto reported an error
    // (out is then not a digest).
    bool final_hex(char out[65]);
    static bool uses_libcrypto();

private:
    void* evp_ = nullptr;  // libcrypto's digest context, or NULL: own code
    bool evp_failed_ = false;
    uint32_t h_[8];
    uint64_t len_;
    unsigned char buf_[64];
    size_t fill_;
};

// Sharded checkpoint (manifest.cpp).
// Creates (if needed) <dir>/step_NNNNNN.tmp, where the ranks write their files.
int shard_staging_dir(const char* dir, int32_t step, std::string* out);
// Parses and checks <step_dir>/manifest.json against expected_world (< 0:
// any) and every listed shard file (size, header, sha256 if verify).
int load_manifest(const char* step_dir, int32_t expected_world, bool verify, int32_t* step_out,
                  std::vector<int64_t>* offsets, std::vector<int64_t>* numels,
                  std::vector<std::string>* paths, std::vector<std::string>* digests);
// Validates header and size; on success *fd_out is an open descriptor
// positioned after the header (caller closes it).
int open_validated(const char* path, int32_t n_expected, int32_t* step_out,
                   int32_t* n_out, int* fd_out);
int read_exact(int fd, void* dst, size_t bytes, const char* path);
// Reads exactly bytes at offset; ADAMW_ESIZE if the file ends first.
int pread_exact(int fd, void* dst, size_t bytes, int64_t offset, const char* path);
// A file written in pieces and made visible atomically: <dir>/<name>.tmp,
// then commit() fsyncs it, renames it over <dir>/<name> and fsyncs dir.
// Destroyed without a commit, it removes the .tmp.
class AtomicFile {
public:
    AtomicFile() = default;
    AtomicFile(const AtomicFile&) = delete;
    AtomicFile& operator=(const AtomicFile&) = delete;
    ~AtomicFile();
    int open(const char* dir, const char* name);
    int write(const void* data, size_t bytes);
    int commit(char* path_out, size_t path_cap);

private:
    int fd_ = -1;
    std::string dir_, tmp_, final_;
};

}  // namespace osr
