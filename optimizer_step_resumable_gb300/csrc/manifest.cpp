// manifest.cpp -- the sharded checkpoint: per-rank shard files and the
// manifest that records which rank owns which range ("Checkpoint and Sharded
// Resume", AI Engineering from Scratch, phase 19 lesson 80).  Host-only.
//
// Layout (one directory per checkpoint):
//     <dir>/step_NNNNNN/rank<R>.bin     shard of rank R: the step_NNNNNN.bin
//                                       format over that rank's range
//     <dir>/step_NNNNNN/manifest.json   {"world_size", "step",
//         "wall_clock_seconds", "shards": [{"rank", "path", "sha256",
//         "param_shard_offset", "param_shard_numel"}], "schema_version": 1}
// Atomicity (section "Atomic write"): every rank writes and fsyncs its file in
// <dir>/step_NNNNNN.tmp/; rank 0 then writes the manifest there (tmp, fsync,
// rename) and renames the whole directory to step_NNNNNN, so a crash at any
// point leaves either the complete new checkpoint or none of it, and the
// previous checkpoints untouched.  The loader refuses the three failure modes
// of section "Three failure modes the schema must guard against": a changed
// world size, a shard count that does not match it, and a partial or
// corrupted shard (size, header or sha256 mismatch).
#include <cerrno>
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <string>
#include <vector>

#include <dirent.h>
#include <fcntl.h>
#include <sys/stat.h>
#include <unistd.h>

#include "ckpt_io.h"
#include "internal.h"

namespace osr {
namespace {

// ---------------------------------------------------------------------------
// A minimal JSON reader for the manifest (objects, arrays, strings with the
// standard escapes, numbers, true/false/null).
// ---------------------------------------------------------------------------
struct JValue {
    enum Kind { Null, Bool, Num, Str, Arr, Obj } kind = Null;
    bool b = false;
    double num = 0.0;
    bool is_int = false;
    long long i = 0;
    std::string s;
    std::vector<JValue> items;
    std::vector<std::pair<std::string, JValue>> fields;
    const JValue* get(const char* key) const
    {
        for (const auto& f : fields)
            if (f.first == key)
                return &f.second;
        return nullptr;
    }
};

struct JParser {
    const char* p;
    const char* end;
    bool ok = true;

    void ws()
    {
        while (p < end && (*p == ' ' || *p == '\t' || *p == '\n' || *p == '\r'))
            ++p;
    }
    bool lit(const char* w)
    {
        const size_t L = std::strlen(w);
        if (size_t(end - p) < L || std::strncmp(p, w, L) != 0)
            return ok = false;
        p += L;
        return true;
    }
    bool string(std::string& out)
    {
        if (p >= end || *p != '"')
            return ok = false;
        ++p;
        while (p < end && *p != '"') {
            if (*p == '\\') {
                if (++p >= end)
                    return ok = false;
                switch (*p) {
                case '"': out += '"'; break;
                case '\\': out += '\\'; break;
                case '/': out += '/'; break;
                case 'n': out += '\n'; break;
                case 't': out += '\t'; break;
                case 'r': out += '\r'; break;
                case 'b': out += '\b'; break;
                case 'f': out += '\f'; break;
                case 'u': {
                    if (end - p < 5)
                        return ok = false;
                    unsigned code = 0;
                    for (int k = 1; k <= 4; ++k) {
                        const char c = p[k];
                        code <<= 4;
                        if (c >= '0' && c <= '9') code |= unsigned(c - '0');
                        else if (c >= 'a' && c <= 'f') code |= unsigned(c - 'a' + 10);
                        else if (c >= 'A' && c <= 'F') code |= unsigned(c - 'A' + 10);
                        else return ok = false;
                    }
                    if (code >= 0x80)
                        return ok = false;  // the manifest is ASCII
                    out += char(code);
                    p += 4;
                    break;
                }
                default: return ok = false;
                }
                ++p;
            } else {
                out += *p++;
            }
        }
        if (p >= end)
            return ok = false;
        ++p;
        return true;
    }
    bool value(JValue& v, int depth)
    {
        if (depth > 16)
            return ok = false;
        ws();
        if (p >= end)
            return ok = false;
        const char c = *p;
        if (c == '{') {
            v.kind = JValue::Obj;
            ++p;
            ws();
            if (p < end && *p == '}') {
                ++p;
                return true;
            }
            for (;;) {
                ws();
                std::string key;
                if (!string(key))
                    return false;
                ws();
                if (p >= end || *p != ':')
                    return ok = false;
                ++p;
                JValue item;
                if (!value(item, depth + 1))
                    return false;
                v.fields.emplace_back(std::move(key), std::move(item));
                ws();
                if (p < end && *p == ',') { ++p; continue; }
                if (p < end && *p == '}') { ++p; return true; }
                return ok = false;
            }
        }
        if (c == '[') {
            v.kind = JValue::Arr;
            ++p;
            ws();
            if (p < end && *p == ']') {
                ++p;
                return true;
            }
            for (;;) {
                JValue item;
                if (!value(item, depth + 1))
                    return false;
                v.items.push_back(std::move(item));
                ws();
                if (p < end && *p == ',') { ++p; continue; }
                if (p < end && *p == ']') { ++p; return true; }
                return ok = false;
            }
        }
        if (c == '"') {
            v.kind = JValue::Str;
            return string(v.s);
        }
        if (c == 't') { v.kind = JValue::Bool; v.b = true; return lit("true"); }
        if (c == 'f') { v.kind = JValue::Bool; return lit("false"); }
        if (c == 'n') { v.kind = JValue::Null; return lit("null"); }
        // number
        const char* q = p;
        if (q < end && (*q == '-' || *q == '+')) ++q;
        bool frac = false;
        while (q < end && ((*q >= '0' && *q <= '9') || *q == '.' || *q == 'e' || *q == 'E' ||
                           *q == '-' || *q == '+')) {
            if (*q == '.' || *q == 'e' || *q == 'E') frac = true;
            ++q;
        }
        if (q == p)
            return ok = false;
        const std::string tok(p, q);
        char* stop = nullptr;
        v.kind = JValue::Num;
        v.num = std::strtod(tok.c_str(), &stop);
        if (!stop || *stop)
            return ok = false;
        if (!frac) {
            v.is_int = true;
            v.i = std::strtoll(tok.c_str(), &stop, 10);
        }
        p = q;
        return true;
    }
};

bool parse_json(const std::string& text, JValue& out)
{
    JParser jp{text.data(), text.data() + text.size()};
    if (!jp.value(out, 0) || !jp.ok)
        return false;
    jp.ws();
    return jp.p == jp.end;
}

std::string step_dir_name(const char* dir, int32_t step, bool staging)
{
    char buf[4200];
    std::snprintf(buf, sizeof buf, "%s/step_%06d%s", dir, int(step), staging ? ".tmp" : "");
    return buf;
}

int fsync_path(const std::string& path, int flags)
{
    const int fd = ::open(path.c_str(), flags | O_CLOEXEC);
    if (fd < 0)
        return fail(ADAMW_EIO, "open %s: %s", path.c_str(), std::strerror(errno));
    const int r = ::fsync(fd);
    ::close(fd);
    if (r != 0)
        return fail(ADAMW_EIO, "fsync %s: %s", path.c_str(), std::strerror(errno));
    return ADAMW_OK;
}

int write_small_file(const std::string& path, const std::string& data)
{
    const int fd = ::open(path.c_str(), O_WRONLY | O_CREAT | O_TRUNC | O_CLOEXEC, 0644);
    if (fd < 0)
        return fail(ADAMW_EIO, "open %s: %s", path.c_str(), std::strerror(errno));
    const char* p = data.data();
    size_t left = data.size();
    while (left > 0) {
        const ssize_t got = ::write(fd, p, left);
        if (got < 0) {
            if (errno == EINTR)
                continue;
            const int e = errno;
            ::close(fd);
            return fail(ADAMW_EIO, "write %s: %s", path.c_str(), std::strerror(e));
        }
        p += got;
        left -= size_t(got);
    }
    if (::fsync(fd) != 0) {
        const int e = errno;
        ::close(fd);
        return fail(ADAMW_EIO, "fsync %s: %s", path.c_str(), std::strerror(e));
    }
    ::close(fd);
    return ADAMW_OK;
}

int remove_tree(const std::string& path)
{
    DIR* d = ::opendir(path.c_str());
    if (!d)
        return ::unlink(path.c_str()) == 0 ? ADAMW_OK : ADAMW_EIO;
    while (struct dirent* e = ::readdir(d)) {
        if (!std::strcmp(e->d_name, ".") || !std::strcmp(e->d_name, ".."))
            continue;
        ::unlink((path + "/" + e->d_name).c_str());
    }
    ::closedir(d);
    return ::rmdir(path.c_str()) == 0 ? ADAMW_OK : ADAMW_EIO;
}

bool valid_hex64(const char* h)
{
    for (int i = 0; i < 64; ++i) {
        const char c = h[i];
        if (!((c >= '0' && c <= '9') || (c >= 'a' && c <= 'f')))
            return false;
    }
    return true;
}

}  // namespace

int shard_staging_dir(const char* dir, int32_t step, std::string* out)
{
    if (!dir || step < 0)
        return fail(ADAMW_EINVAL, "shard write: null directory or negative step");
    *out = step_dir_name(dir, step, true);
    if (::mkdir(out->c_str(), 0755) != 0 && errno != EEXIST)
        return fail(ADAMW_EIO, "mkdir %s: %s", out->c_str(), std::strerror(errno));
    return ADAMW_OK;
}

// Reads and validates <step_dir>/manifest.json and each listed shard (size,
// header, and, if verify, sha256).  Fills the layout.
int load_manifest(const char* step_dir, int32_t expected_world, bool verify, int32_t* step_out,
                  std::vector<int64_t>* offsets, std::vector<int64_t>* numels,
                  std::vector<std::string>* paths, std::vector<std::string>* digests)
{
    if (!step_dir)
        return fail(ADAMW_EINVAL, "manifest: null directory");
    const std::string mpath = std::string(step_dir) + "/manifest.json";
    const int fd = ::open(mpath.c_str(), O_RDONLY | O_CLOEXEC);
    if (fd < 0)
        return fail(ADAMW_EIO, "open %s: %s", mpath.c_str(), std::strerror(errno));
    std::string text;
    char buf[65536];
    for (;;) {
        const ssize_t got = ::read(fd, buf, sizeof buf);
        if (got < 0 && errno == EINTR)
            continue;
        if (got <= 0)
            break;
        text.append(buf, size_t(got));
        if (text.size() > (size_t(64) << 20))
            break;
    }
    ::close(fd);
    JValue root;
    if (!parse_json(text, root) || root.kind != JValue::Obj)
        return fail(ADAMW_EFORMAT, "%s: not a JSON object", mpath.c_str());
    auto int_field = [&](const JValue& o, const char* k, long long* v) {
        const JValue* f = o.get(k);
        if (!f || f->kind != JValue::Num || !f->is_int)
            return false;
        *v = f->i;
        return true;
    };
    long long schema = 0, world = 0, step = 0;
    if (!int_field(root, "schema_version", &schema) || schema != 1)
        return fail(ADAMW_EFORMAT, "%s: schema_version is not 1", mpath.c_str());
    if (!int_field(root, "world_size", &world) || world < 1 || world > (1 << 20))
        return fail(ADAMW_EFORMAT, "%s: bad world_size", mpath.c_str());
    if (!int_field(root, "step", &step) || step < 0 || step > INT32_MAX)
        return fail(ADAMW_EFORMAT, "%s: bad step", mpath.c_str());
    const JValue* wall = root.get("wall_clock_seconds");
    if (!wall || wall->kind != JValue::Num)
        return fail(ADAMW_EFORMAT, "%s: bad wall_clock_seconds", mpath.c_str());
    if (expected_world >= 0 && world != expected_world)
        return fail(ADAMW_EMISMATCH,
                    "%s: saved with world_size %lld, loading with %d (world size changed)",
                    mpath.c_str(), world, expected_world);
    const JValue* shards = root.get("shards");
    if (!shards || shards->kind != JValue::Arr)
        return fail(ADAMW_EFORMAT, "%s: no shards array", mpath.c_str());
    if ((long long)shards->items.size() != world)
        return fail(ADAMW_EMISMATCH, "%s: %zu shards listed for world_size %lld", mpath.c_str(),
                    shards->items.size(), world);
    offsets->assign(size_t(world), -1);
    numels->assign(size_t(world), -1);
    paths->assign(size_t(world), std::string());
    digests->assign(size_t(world), std::string());
    for (const JValue& sh : shards->items) {
        long long rank = -1, off = -1, num = -1;
        if (sh.kind != JValue::Obj || !int_field(sh, "rank", &rank) ||
            !int_field(sh, "param_shard_offset", &off) ||
            !int_field(sh, "param_shard_numel", &num))
            return fail(ADAMW_EFORMAT, "%s: malformed shard entry", mpath.c_str());
        const JValue* path = sh.get("path");
        const JValue* sha = sh.get("sha256");
        if (!path || path->kind != JValue::Str || !sha || sha->kind != JValue::Str)
            return fail(ADAMW_EFORMAT, "%s: shard without path or sha256", mpath.c_str());
        if (rank < 0 || rank >= world || (*offsets)[size_t(rank)] != -1)
            return fail(ADAMW_EMISMATCH, "%s: rank %lld missing, repeated or out of range",
                        mpath.c_str(), rank);
        if (off < 0 || num < 1 || num > INT32_MAX)
            return fail(ADAMW_EFORMAT, "%s: bad range of rank %lld", mpath.c_str(), rank);
        if (path->s.empty() || path->s.find('/') != std::string::npos || path->s == "." ||
            path->s == "..")
            return fail(ADAMW_EFORMAT, "%s: shard path must be a file name", mpath.c_str());
        if (sha->s.size() != 64 || !valid_hex64(sha->s.c_str()))
            return fail(ADAMW_EFORMAT, "%s: bad sha256 of rank %lld", mpath.c_str(), rank);
        (*offsets)[size_t(rank)] = off;
        (*numels)[size_t(rank)] = num;
        (*paths)[size_t(rank)] = path->s;
        (*digests)[size_t(rank)] = sha->s;
    }
    int64_t expect = 0;
    for (long long r = 0; r < world; ++r) {
        if ((*offsets)[size_t(r)] != expect)
            return fail(ADAMW_EFORMAT, "%s: shard ranges are not contiguous in rank order",
                        mpath.c_str());
        expect += (*numels)[size_t(r)];
    }
    // every shard file: exact size and header, and (if asked) its digest
    for (long long r = 0; r < world; ++r) {
        const std::string sp = std::string(step_dir) + "/" + (*paths)[size_t(r)];
        int32_t fstep = -1, fn = -1;
        int sfd = -1;
        int rc = open_validated(sp.c_str(), int32_t((*numels)[size_t(r)]), &fstep, &fn, &sfd);
        if (rc != ADAMW_OK)
            return fail(rc, "shard of rank %lld: %s", r, last_error_text());
        if (fstep != step) {
            ::close(sfd);
            return fail(ADAMW_EMISMATCH, "%s: step %d, manifest says %lld", sp.c_str(), fstep,
                        step);
        }
        if (verify) {
            Sha256 h;
            unsigned char header[8];
            for (int i = 0; i < 4; ++i) {
                header[i] = static_cast<unsigned char>((uint32_t(fstep) >> (8 * i)) & 0xffu);
                header[4 + i] = static_cast<unsigned char>((uint32_t(fn) >> (8 * i)) & 0xffu);
            }
            h.update(header, 8);
            std::vector<unsigned char> chunk(size_t(4) << 20);
            for (;;) {
                const ssize_t got = ::read(sfd, chunk.data(), chunk.size());
                if (got < 0 && errno == EINTR)
                    continue;
                if (got < 0) {
                    const int e = errno;
                    ::close(sfd);
                    return fail(ADAMW_EIO, "read %s: %s", sp.c_str(), std::strerror(e));
                }
                if (got == 0)
                    break;
                h.update(chunk.data(), size_t(got));
            }
            char hex[65];
            if (!h.final_hex(hex)) {
                ::close(sfd);
                return fail(ADAMW_EIO, "%s: the digest could not be computed", sp.c_str());
            }
            if ((*digests)[size_t(r)] != hex) {
                ::close(sfd);
                return fail(ADAMW_EFORMAT, "%s: sha256 %s, manifest says %s (partial or corrupted "
                            "write)", sp.c_str(), hex, (*digests)[size_t(r)].c_str());
            }
        }
        ::close(sfd);
    }
    if (step_out)
        *step_out = int32_t(step);
    return ADAMW_OK;
}

}  // namespace osr

extern "C" {

int ckpt_shard_write_host(const char* dir, int32_t step, int32_t rank, int32_t n,
                          const float* h_w, const float* h_m, const float* h_v,
                          char* sha256_hex_out)
{
    osr::clear_error();
    if (rank < 0 || n < 1 || !h_w || !h_m || !h_v || !sha256_hex_out)
        return osr::fail(ADAMW_EINVAL, "ckpt_shard_write_host: bad arguments");
    std::string staging;
    int rc = osr::shard_staging_dir(dir, step, &staging);
    if (rc != ADAMW_OK)
        return rc;
    unsigned char header[8];
    for (int i = 0; i < 4; ++i) {
        header[i] = static_cast<unsigned char>((uint32_t(step) >> (8 * i)) & 0xffu);
        header[4 + i] = static_cast<unsigned char>((uint32_t(n) >> (8 * i)) & 0xffu);
    }
    const size_t bytes = size_t(n) * 4u;
    const osr::IoPiece pieces[4] = {
        {header, 8, 8}, {h_w, bytes, bytes}, {h_m, bytes, bytes}, {h_v, bytes, bytes}};
    char name[64];
    std::snprintf(name, sizeof name, "rank%d.bin", int(rank));
    rc = osr::write_named_file(staging.c_str(), name, pieces, 4, 0);
    if (rc != ADAMW_OK)
        return rc;
    osr::Sha256 h;
    for (const auto& p : pieces)
        h.update(p.data, p.bytes);
    if (!h.final_hex(sha256_hex_out))
        return osr::fail(ADAMW_EIO, "rank%d.bin: the digest could not be computed", int(rank));
    return ADAMW_OK;
}

int ckpt_manifest_commit(const char* dir, int32_t step, int32_t world, double wall_clock_seconds,
                         const int64_t* offsets, const int64_t* numels, const char* sha256_hex,
                         char* path_out, size_t path_cap)
{
    osr::clear_error();
    if (!dir || step < 0 || world < 1 || !offsets || !numels || !sha256_hex ||
        !std::isfinite(wall_clock_seconds))
        return osr::fail(ADAMW_EINVAL, "ckpt_manifest_commit: bad arguments");
    if (std::strlen(sha256_hex) != size_t(64) * size_t(world))
        return osr::fail(ADAMW_EINVAL, "ckpt_manifest_commit: need %d x 64 hex digits", world);
    int64_t expect = 0;
    for (int32_t r = 0; r < world; ++r) {
        if (offsets[r] != expect || numels[r] < 1 || numels[r] > INT32_MAX ||
            !osr::valid_hex64(sha256_hex + 64 * size_t(r)))
            return osr::fail(ADAMW_EINVAL,
                             "ckpt_manifest_commit: shard %d range or digest is invalid", r);
        expect += numels[r];
    }
    const std::string staging = osr::step_dir_name(dir, step, true);
    const std::string final_dir = osr::step_dir_name(dir, step, false);
    // every listed shard must be in the staging directory, complete
    for (int32_t r = 0; r < world; ++r) {
        char sp[4300];
        std::snprintf(sp, sizeof sp, "%s/rank%d.bin", staging.c_str(), int(r));
        if (ckpt_probe(sp, int32_t(numels[r]), nullptr, nullptr) != ADAMW_OK)
            return osr::fail(ADAMW_ESTATE, "ckpt_manifest_commit: shard %d not ready: %s", r,
                             osr::last_error_text());
    }
    std::string js = "{\n  \"world_size\": " + std::to_string(world) + ",\n  \"step\": " +
                     std::to_string(step) + ",\n  \"wall_clock_seconds\": ";
    char num[64];
    std::snprintf(num, sizeof num, "%.17g", wall_clock_seconds);
    std::string wall = num;
    if (wall.find_first_of(".eEn") == std::string::npos)
        wall += ".0";
    js += wall + ",\n  \"shards\": [";
    for (int32_t r = 0; r < world; ++r) {
        js += r ? ",\n" : "\n";
        js += "    {\"rank\": " + std::to_string(r) + ", \"path\": \"rank" + std::to_string(r) +
              ".bin\", \"sha256\": \"" + std::string(sha256_hex + 64 * size_t(r), 64) +
              "\", \"param_shard_offset\": " + std::to_string(offsets[r]) +
              ", \"param_shard_numel\": " + std::to_string(numels[r]) + "}";
    }
    js += "\n  ],\n  \"schema_version\": 1\n}\n";
    const std::string mtmp = staging + "/manifest.json.tmp";
    int rc = osr::write_small_file(mtmp, js);
    if (rc != ADAMW_OK)
        return rc;
    if (::rename(mtmp.c_str(), (staging + "/manifest.json").c_str()) != 0)
        return osr::fail(ADAMW_EIO, "rename %s: %s", mtmp.c_str(), std::strerror(errno));
    // drop anything a crashed earlier attempt left behind (e.g. more ranks)
    if (DIR* d = ::opendir(staging.c_str())) {
        while (struct dirent* e = ::readdir(d)) {
            const std::string nm = e->d_name;
            if (nm == "." || nm == ".." || nm == "manifest.json")
                continue;
            int r = -1;
            char tail = 0;
            if (std::sscanf(nm.c_str(), "rank%d.bi%c", &r, &tail) == 2 && tail == 'n' &&
                r >= 0 && r < world && nm == "rank" + std::to_string(r) + ".bin")
                continue;
            ::unlink((staging + "/" + nm).c_str());
        }
        ::closedir(d);
    }
    if ((rc = osr::fsync_path(staging, O_RDONLY)) != ADAMW_OK)
        return rc;
    // the directory rename is the commit point
    struct stat st;
    std::string old;
    if (::stat(final_dir.c_str(), &st) == 0) {
        old = final_dir + ".old." + std::to_string(::getpid());
        if (::rename(final_dir.c_str(), old.c_str()) != 0)
            return osr::fail(ADAMW_EIO, "rename %s: %s", final_dir.c_str(), std::strerror(errno));
    }
    if (::rename(staging.c_str(), final_dir.c_str()) != 0)
        return osr::fail(ADAMW_EIO, "rename %s: %s", staging.c_str(), std::strerror(errno));
    if ((rc = osr::fsync_path(dir, O_RDONLY)) != ADAMW_OK)
        return rc;
    if (!old.empty())
        osr::remove_tree(old);
    if (path_out && path_cap > 0) {
        if (final_dir.size() + 1 > path_cap)
            return osr::fail(ADAMW_EINVAL, "path buffer too small (checkpoint committed)");
        std::memcpy(path_out, final_dir.c_str(), final_dir.size() + 1);
    }
    return ADAMW_OK;
}

int ckpt_manifest_load(const char* step_dir, int32_t expected_world, int32_t verify_sha256,
                       int32_t* step_out, int32_t* world_out, int64_t* offsets_out,
                       int64_t* numels_out, int32_t cap)
{
    osr::clear_error();
    std::vector<int64_t> off, num;
    std::vector<std::string> paths, digests;
    int32_t step = -1;
    const int rc = osr::load_manifest(step_dir, expected_world, verify_sha256 != 0, &step, &off,
                                      &num, &paths, &digests);
    if (rc != ADAMW_OK)
        return rc;
    if (world_out)
        *world_out = int32_t(off.size());
    if (step_out)
        *step_out = step;
    if (offsets_out || numels_out) {
        if (cap < int32_t(off.size()))
            return osr::fail(ADAMW_EINVAL, "ckpt_manifest_load: %zu shards, room for %d",
                             off.size(), cap);
        for (size_t r = 0; r < off.size(); ++r) {
            if (offsets_out)
                offsets_out[r] = off[r];
            if (numels_out)
                numels_out[r] = num[r];
        }
    }
    return ADAMW_OK;
}

// The flat state from the shards (section "Three failure modes the schema
// must guard against": each shard's param_shard_offset and param_shard_numel
// put its range back at its place in the flat parameter vector).  Streams
// the w regions of all shards in rank order, then the m regions, then the v
// regions, into <out_dir>/step_NNNNNN.bin (atomic: .tmp, fsync, rename).  A
// shard's bytes reach its SHA-256 in file order (header, w, m, v), so every
// digest is checked without a second read; on a mismatch no file appears.
int ckpt_consolidate(const char* step_dir, int32_t expected_world, const char* out_dir,
                     char* path_out, size_t path_cap)
{
    osr::clear_error();
    if (!step_dir || !out_dir)
        return osr::fail(ADAMW_EINVAL, "ckpt_consolidate: null directory");
    std::vector<int64_t> off, num;
    std::vector<std::string> paths, digests;
    int32_t step = -1;
    int rc = osr::load_manifest(step_dir, expected_world, false, &step, &off, &num, &paths,
                                &digests);
    if (rc != ADAMW_OK)
        return rc;
    const size_t world = off.size();
    const int64_t n = off.back() + num.back();
    if (n > INT32_MAX)
        return osr::fail(ADAMW_ESIZE, "%s: %lld parameters in all do not fit the header",
                         step_dir, (long long)n);
    auto le_header = [](int32_t a, int32_t b, unsigned char* h) {
        for (int i = 0; i < 4; ++i) {
            h[i] = static_cast<unsigned char>((uint32_t(a) >> (8 * i)) & 0xffu);
            h[4 + i] = static_cast<unsigned char>((uint32_t(b) >> (8 * i)) & 0xffu);
        }
    };
    std::vector<int> fds(world, -1);
    std::vector<osr::Sha256> hashes(world);
    std::vector<std::string> spaths(world);
    auto close_all = [&] {
        for (int& fd : fds)
            if (fd >= 0) {
                ::close(fd);
                fd = -1;
            }
    };
    for (size_t r = 0; r < world && rc == ADAMW_OK; ++r) {
        spaths[r] = std::string(step_dir) + "/" + paths[r];
        int32_t fstep = -1, fn = -1;
        rc = osr::open_validated(spaths[r].c_str(), int32_t(num[r]), &fstep, &fn, &fds[r]);
        if (rc == ADAMW_OK && fstep != step)
            rc = osr::fail(ADAMW_EMISMATCH, "%s: step %d, manifest says %d", spaths[r].c_str(),
                           fstep, step);
        if (rc == ADAMW_OK) {
            unsigned char h[8];
            le_header(fstep, fn, h);
            hashes[r].update(h, 8);
        }
    }
    if (rc != ADAMW_OK) {
        close_all();
        return rc;
    }
    char name[32];
    std::snprintf(name, sizeof name, "step_%06d.bin", int(step));
    osr::AtomicFile out;
    rc = out.open(out_dir, name);
    if (rc == ADAMW_OK) {
        unsigned char h[8];
        le_header(step, int32_t(n), h);
        rc = out.write(h, 8);
    }
    std::vector<unsigned char> buf(size_t(8) << 20);
    for (int region = 0; region < 3 && rc == ADAMW_OK; ++region)
        for (size_t r = 0; r < world && rc == ADAMW_OK; ++r) {
            int64_t pos = 8 + 4 * num[r] * region;
            int64_t left = 4 * num[r];
            while (left > 0 && rc == ADAMW_OK) {
                const size_t k = left < int64_t(buf.size()) ? size_t(left) : buf.size();
                rc = osr::pread_exact(fds[r], buf.data(), k, pos, spaths[r].c_str());
                if (rc == ADAMW_OK) {
                    hashes[r].update(buf.data(), k);
                    rc = out.write(buf.data(), k);
                }
                pos += int64_t(k);
                left -= int64_t(k);
            }
        }
    close_all();
    for (size_t r = 0; r < world && rc == ADAMW_OK; ++r) {
        char hex[65];
        if (!hashes[r].final_hex(hex))
            rc = osr::fail(ADAMW_EIO, "%s: the digest could not be computed", spaths[r].c_str());
        else if (digests[r] != hex)
            rc = osr::fail(ADAMW_EFORMAT, "%s: sha256 %s, manifest says %s (partial or corrupted "
                           "write)", spaths[r].c_str(), hex, digests[r].c_str());
    }
    if (rc != ADAMW_OK)
        return rc;  // the unfinished .tmp goes with `out`
    return out.commit(path_out, path_cap);
}

}  // extern "C"
