// sha256.cpp -- SHA-256 (FIPS PUB 180-4, "Secure Hash Standard", section
// 6.2) for the shard digests of the sharded checkpoint's manifest.
//
// Two backends with one result.  The system's libcrypto (OpenSSL 3), loaded
// at run time through its public EVP digest interface, hashes with the CPU's
// SHA instructions: 2.0 GB/s on one Grace core (1.1 GB/s on an x86 core)
// against 160 MB/s for portable code, which for a 1.33 GB shard is 0.65 s
// instead of 8.  When it
// cannot be loaded (or OSR_SHA256=builtin), the library's own portable code
// runs, written from the standard's description: 512-bit blocks, a 64-word
// message schedule, 64 rounds with the functions Ch, Maj, Sigma0/1 and
// sigma0/1, the big-endian length padding of section 5.1.1.
#include <cstdint>
#include <cstdlib>
#include <cstring>

#include <dlfcn.h>

#include "ckpt_io.h"
#include "internal.h"

namespace osr {
namespace {

// First 32 bits of the fractional parts of the cube roots of the first 64
// primes (FIPS 180-4, section 4.2.2).
constexpr uint32_t kRound[64] = {
    0x428a2f98, 0x71374491, 0xb5c0fbcf, 0xe9b5dba5, 0x3956c25b, 0x59f111f1, 0x923f82a4,
    0xab1c5ed5, 0xd807aa98, 0x12835b01, 0x243185be, 0x550c7dc3, 0x72be5d74, 0x80deb1fe,
    0x9bdc06a7, 0xc19bf174, 0xe49b69c1, 0xefbe4786, 0x0fc19dc6, 0x240ca1cc, 0x2de92c6f,
    0x4a7484aa, 0x5cb0a9dc, 0x76f988da, 0x983e5152, 0xa831c66d, 0xb00327c8, 0xbf597fc7,
    0xc6e00bf3, 0xd5a79147, 0x06ca6351, 0x14292967, 0x27b70a85, 0x2e1b2138, 0x4d2c6dfc,
    0x53380d13, 0x650a7354, 0x766a0abb, 0x81c2c92e, 0x92722c85, 0xa2bfe8a1, 0xa81a664b,
    0xc24b8b70, 0xc76c51a3, 0xd192e819, 0xd6990624, 0xf40e3585, 0x106aa070, 0x19a4c116,
    0x1e376c08, 0x2748774c, 0x34b0bcb5, 0x391c0cb3, 0x4ed8aa4a, 0x5b9cca4f, 0x682e6ff3,
    0x748f82ee, 0x78a5636f, 0x84c87814, 0x8cc70208, 0x90befffa, 0xa4506ceb, 0xbef9a3f7,
    0xc67178f2};

// First 32 bits of the fractional parts of the square roots of the first 8
// primes (section 5.3.3).
constexpr uint32_t kInit[8] = {0x6a09e667, 0xbb67ae85, 0x3c6ef372, 0xa54ff53a,
                               0x510e527f, 0x9b05688c, 0x1f83d9ab, 0x5be0cd19};

inline uint32_t rotr(uint32_t x, int r) { return (x >> r) | (x << (32 - r)); }

void compress(uint32_t h[8], const unsigned char* block)
{
    uint32_t w[64];
    for (int t = 0; t < 16; ++t)
        w[t] = (uint32_t(block[4 * t]) << 24) | (uint32_t(block[4 * t + 1]) << 16) |
               (uint32_t(block[4 * t + 2]) << 8) | uint32_t(block[4 * t + 3]);
    for (int t = 16; t < 64; ++t) {
        const uint32_t s0 = rotr(w[t - 15], 7) ^ rotr(w[t - 15], 18) ^ (w[t - 15] >> 3);
        const uint32_t s1 = rotr(w[t - 2], 17) ^ rotr(w[t - 2], 19) ^ (w[t - 2] >> 10);
        w[t] = w[t - 16] + s0 + w[t - 7] + s1;
    }
    uint32_t a = h[0], b = h[1], c = h[2], d = h[3], e = h[4], f = h[5], g = h[6], k = h[7];
    for (int t = 0; t < 64; ++t) {
        const uint32_t S1 = rotr(e, 6) ^ rotr(e, 11) ^ rotr(e, 25);
        const uint32_t ch = (e & f) ^ (~e & g);
        const uint32_t t1 = k + S1 + ch + kRound[t] + w[t];
        const uint32_t S0 = rotr(a, 2) ^ rotr(a, 13) ^ rotr(a, 22);
        const uint32_t maj = (a & b) ^ (a & c) ^ (b & c);
        const uint32_t t2 = S0 + maj;
        k = g;
        g = f;
        f = e;
        e = d + t1;
        d = c;
        c = b;
        b = a;
        a = t1 + t2;
    }
    h[0] += a;
    h[1] += b;
    h[2] += c;
    h[3] += d;
    h[4] += e;
    h[5] += f;
    h[6] += g;
    h[7] += k;
}

// libcrypto's EVP digest interface (public OpenSSL 3 API), resolved once.
struct Evp {
    void* (*ctx_new)() = nullptr;
    void (*ctx_free)(void*) = nullptr;
    const void* (*sha256)() = nullptr;
    int (*init)(void*, const void*, void*) = nullptr;
    int (*update)(void*, const void*, size_t) = nullptr;
    int (*final)(void*, unsigned char*, unsigned int*) = nullptr;
    bool ok = false;
};

template <typename F>
bool resolve(void* lib, const char* name, F* out)
{
    *out = reinterpret_cast<F>(::dlsym(lib, name));
    return *out != nullptr;
}

const Evp& evp()
{
    static const Evp e = [] {
        Evp r;
        const char* choice = std::getenv("OSR_SHA256");
        if (choice && std::strcmp(choice, "builtin") == 0)
            return r;
        void* lib = ::dlopen("libcrypto.so.3", RTLD_NOW | RTLD_LOCAL);
        if (!lib)
            return r;  // kept open for the life of the process once found
        r.ok = resolve(lib, "EVP_MD_CTX_new", &r.ctx_new) &&
               resolve(lib, "EVP_MD_CTX_free", &r.ctx_free) &&
               resolve(lib, "EVP_sha256", &r.sha256) &&
               resolve(lib, "EVP_DigestInit_ex", &r.init) &&
               resolve(lib, "EVP_DigestUpdate", &r.update) &&
               resolve(lib, "EVP_DigestFinal_ex", &r.final) && r.sha256() != nullptr;
        return r;
    }();
    return e;
}

}  // namespace

bool Sha256::uses_libcrypto() { return evp().ok; }

Sha256::~Sha256()
{
    if (evp_)
        evp().ctx_free(evp_);
}

void Sha256::reset()
{
    std::memcpy(h_, kInit, sizeof h_);
    len_ = 0;
    fill_ = 0;
    evp_failed_ = false;
    const Evp& e = evp();
    if (!e.ok)
        return;
    if (!evp_)
        evp_ = e.ctx_new();
    if (evp_ && e.init(evp_, e.sha256(), nullptr) != 1) {  // own code instead
        e.ctx_free(evp_);
        evp_ = nullptr;
    }
}

void Sha256::update(const void* data, size_t bytes)
{
    if (evp_) {
        if (bytes > 0 && evp().update(evp_, data, bytes) != 1)
            evp_failed_ = true;
        return;
    }
    const unsigned char* p = static_cast<const unsigned char*>(data);
    len_ += bytes;
    if (fill_) {
        const size_t take = bytes < 64 - fill_ ? bytes : 64 - fill_;
        std::memcpy(buf_ + fill_, p, take);
        fill_ += take;
        p += take;
        bytes -= take;
        if (fill_ < 64)
            return;
        compress(h_, buf_);
        fill_ = 0;
    }
    for (; bytes >= 64; p += 64, bytes -= 64)
        compress(h_, p);
    std::memcpy(buf_, p, bytes);
    fill_ = bytes;
}

bool Sha256::final_hex(char out[65])
{
    unsigned char digest[32];
    bool ok = true;
    if (evp_) {
        unsigned int len = 0;
        ok = !evp_failed_ && evp().final(evp_, digest, &len) == 1 && len == 32;
    } else {
        // padding: a 1 bit, zeros, then the message length in bits, big-endian
        const uint64_t bits = len_ * 8u;
        const unsigned char one = 0x80, zero = 0x00;
        update(&one, 1);
        while (fill_ != 56)
            update(&zero, 1);
        unsigned char lenbe[8];
        for (int i = 0; i < 8; ++i)
            lenbe[i] = static_cast<unsigned char>(bits >> (56 - 8 * i));
        update(lenbe, 8);
        for (int i = 0; i < 8; ++i)
            for (int j = 0; j < 4; ++j)
                digest[4 * i + j] = static_cast<unsigned char>((h_[i] >> (24 - 8 * j)) & 0xffu);
    }
    static const char hex[] = "0123456789abcdef";
    for (int i = 0; i < 32; ++i) {
        out[2 * i] = ok ? hex[digest[i] >> 4] : '0';
        out[2 * i + 1] = ok ? hex[digest[i] & 15] : '0';
    }
    out[64] = '\0';
    return ok;
}

}  // namespace osr

extern "C" int ckpt_sha256_hex(const void* data, int64_t bytes, char* hex_out)
{
    osr::clear_error();
    if ((!data && bytes > 0) || bytes < 0 || !hex_out)
        return osr::fail(ADAMW_EINVAL, "ckpt_sha256_hex: bad arguments");
    osr::Sha256 s;
    s.update(data, size_t(bytes));
    if (!s.final_hex(hex_out))
        return osr::fail(ADAMW_EIO, "ckpt_sha256_hex: libcrypto reported an error");
    return ADAMW_OK;
}

extern "C" int ckpt_sha256_backend(void) { return osr::Sha256::uses_libcrypto() ? 1 : 0; }
