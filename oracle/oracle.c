/*
 * oracle.c -- plain CPU oracle for the clipped-AdamW optimizer step and the
 * step_NNNNNN.bin checkpoint.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library calls, links or
 * loads this file; only the tests, the smoke check and the benchmark's CPU
 * baseline do.  It shares no source, header, constant or helper with the
 * CUDA library: it restates the method from the pages it was written from,
 * one definition at a time, in double precision over float32 state, with no
 * blocking, fusion or reordering beyond what those definitions state.
 *
 * Sources (cited by page title and section):
 *  [T]  "Training as a Recoverable State Transition" (aihero.club, Language
 *       Models from Scratch): sections "The Exact Targets of Clipping and
 *       AdamW", "Example 1: The First One-Dimensional Step and Moment State",
 *       and "The Checkpoint Contract and a Real Recovery Test".
 *  [C]  "Grow a Language Model: Checkpoints" (unhomeschool.com, Georgian and
 *       Spanish editions): sections "Format", "Region by region",
 *       "Total size", "Why save m & v".
 *  [S]  "Checkpoint and Sharded Resume" (AI Engineering from Scratch, phase 19
 *       lesson 80): sections "Atomic write" and "Three failure modes".
 *
 * Build: any C99 compiler, -O2 -ffp-contract=off (no fused multiply-add, so
 * that every operation below is one IEEE double rounding on x86 and Arm
 * alike), no -ffast-math.
 */
#define _POSIX_C_SOURCE 200809L
#include <errno.h>
#include <fcntl.h>
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>
#include <sys/stat.h>
#include <unistd.h>

/* Status codes of this file (its own; the CUDA library has its own set). */
#define OR_OK 0
#define OR_EINVAL 1     /* bad argument                                    */
#define OR_EIO 2        /* open/read/write/fsync/rename failed             */
#define OR_EFORMAT 3    /* header fields impossible (negative step or n)   */
#define OR_ESIZE 4      /* file size disagrees with 8 + 12 n, or truncated */
#define OR_EMISMATCH 5  /* n in the file differs from the expected n       */
#define OR_ENONFINITE 6 /* gradient norm is inf or nan: state left as is   */

int oracle_version(void) { return 1; }

/* ------------------------------------------------------------------------
 * Global L2 norm of the concatenated gradient.  [T] "The Exact Targets of
 * Clipping and AdamW": all parameter gradients are joined into one vector g
 * and its Euclidean norm ||g||_2 is taken.  Each float32 value is widened to
 * double; its square is exact in double (24-bit significand squared fits in
 * 53 bits); the squares are summed in index order.
 * ---------------------------------------------------------------------- */
double oracle_sumsq(const float* g, int64_t n)
{
    double s = 0.0;
    for (int64_t i = 0; i < n; ++i) {
        double x = (double)g[i];
        s = s + x * x;
    }
    return s;
}

double oracle_global_norm(const float* g, int64_t n)
{
    return sqrt(oracle_sumsq(g, n));
}

/* ------------------------------------------------------------------------
 * Per-tensor sums of squares.  "Training as a Recoverable State Transition"
 * (aihero.club), section "The Exact Targets of Clipping and AdamW": the norms
 * of all parameters are recorded to detect numerical faults.  Tensor k is
 * g[offsets[k] .. offsets[k] + numels[k]); each sum is taken in index order
 * in double, like the global one.
 * ---------------------------------------------------------------------- */
void oracle_tensor_sumsq(const float* g, const int64_t* offsets,
                         const int64_t* numels, int32_t n_tensors, double* out)
{
    for (int32_t k = 0; k < n_tensors; ++k)
        out[k] = oracle_sumsq(g + offsets[k], numels[k]);
}

/* ------------------------------------------------------------------------
 * Clip factor.  [T] "The Exact Targets of Clipping and AdamW": when the norm
 * exceeds the threshold c the whole vector is multiplied by c/||g||,
 * otherwise it is left unchanged; one c for all layers.  The worked code on
 * that page uses min(1, c/|g|), i.e. a strict ">" and no epsilon; a zero
 * norm therefore never divides.
 * ---------------------------------------------------------------------- */
double oracle_clip_scale(double norm, double c)
{
    if (norm > c)
        return c / norm;
    return 1.0;
}

/* ------------------------------------------------------------------------
 * One AdamW update of one parameter, every intermediate in double.
 * [T] "The Exact Targets of Clipping and AdamW":
 *   m_t = beta1 m + (1-beta1) g          (first moment, EMA of gradients)
 *   v_t = beta2 v + (1-beta2) g^2        (second moment, EMA of squares)
 *   m_hat = m_t / (1 - beta1^t)          (bias correction, t counts updates
 *   v_hat = v_t / (1 - beta2^t)           and the first update has t = 1)
 *   w <- w (1 - lr wd) - lr m_hat / (sqrt(v_hat) + eps)
 * The decay multiplies the old weight first and is applied to every
 * parameter; eps is added to sqrt(v_hat), not to v.  Here g is the already
 * clipped gradient g_hat = s * g.
 * ---------------------------------------------------------------------- */
typedef struct {
    double g_hat;     /* clipped gradient s*g                    */
    double m;         /* new first moment m_t                    */
    double v;         /* new second moment v_t                   */
    double m_hat;     /* bias-corrected first moment             */
    double v_hat;     /* bias-corrected second moment            */
    double w_decayed; /* w (1 - lr wd)                           */
    double update;    /* lr m_hat / (sqrt(v_hat) + eps)          */
    double w;         /* new weight w_decayed - update           */
} oracle_terms;

void oracle_adamw_element(double w, double g, double m, double v, double s,
                          int32_t t, double lr, double wd, double beta1,
                          double beta2, double eps, oracle_terms* out)
{
    double g_hat = g * s;
    double m_t = beta1 * m + (1.0 - beta1) * g_hat;
    double v_t = beta2 * v + (1.0 - beta2) * (g_hat * g_hat);
    double m_hat = m_t / (1.0 - pow(beta1, (double)t));
    double v_hat = v_t / (1.0 - pow(beta2, (double)t));
    double w_decayed = w * (1.0 - lr * wd);
    double update = lr * m_hat / (sqrt(v_hat) + eps);
    out->g_hat = g_hat;
    out->m = m_t;
    out->v = v_t;
    out->m_hat = m_hat;
    out->v_hat = v_hat;
    out->w_decayed = w_decayed;
    out->update = update;
    out->w = w_decayed - update;
}

/* ------------------------------------------------------------------------
 * One full optimizer step over the flat float32 state: global norm, clip
 * factor, AdamW per element, each new value rounded to float32 once.
 * [T] "The Exact Targets of Clipping and AdamW" (the step order: record the
 * norm, clip globally, then step).  A non-finite norm leaves w, m, v as they
 * are and returns OR_ENONFINITE (the page asks only that norms be recorded
 * to detect numerical faults; skipping the update is this oracle's reading).
 * ---------------------------------------------------------------------- */
int oracle_adamw_clip_step(float* w, const float* g, float* m, float* v,
                           int64_t n, int32_t t, double lr, double wd,
                           double clip, double beta1, double beta2, double eps,
                           double* norm_out)
{
    if (n < 0 || t < 1)
        return OR_EINVAL;
    double norm = oracle_global_norm(g, n);
    if (norm_out)
        *norm_out = norm;
    if (!isfinite(norm))
        return OR_ENONFINITE;
    double s = oracle_clip_scale(norm, clip);
    for (int64_t i = 0; i < n; ++i) {
        oracle_terms r;
        oracle_adamw_element((double)w[i], (double)g[i], (double)m[i],
                             (double)v[i], s, t, lr, wd, beta1, beta2, eps, &r);
        w[i] = (float)r.w;
        m[i] = (float)r.m;
        v[i] = (float)r.v;
    }
    return OR_OK;
}

/* ------------------------------------------------------------------------
 * The step after gradient accumulation.  "Grow a Language Model: Backprop"
 * (unhomeschool.com), section "Accumulation across micro-batches": backward
 * adds each micro-batch's gradient into the buffer, scale_grads(1/n_micro)
 * averages it, then the optimizer step runs (and zero_grads clears the
 * buffer).  Here every gradient value is first multiplied by grad_scale in
 * double; the norm, the clip and the update then see the scaled vector.
 * ---------------------------------------------------------------------- */
int oracle_adamw_clip_step_scaled(float* w, const float* g, float* m, float* v,
                                  int64_t n, int32_t t, double lr, double wd,
                                  double clip, double grad_scale, double beta1,
                                  double beta2, double eps, double* norm_out)
{
    if (n < 0 || t < 1)
        return OR_EINVAL;
    double sumsq = 0.0;
    for (int64_t i = 0; i < n; ++i) {
        double x = (double)g[i] * grad_scale;
        sumsq = sumsq + x * x;
    }
    double norm = sqrt(sumsq);
    if (norm_out)
        *norm_out = norm;
    if (!isfinite(norm))
        return OR_ENONFINITE;
    double s = oracle_clip_scale(norm, clip);
    for (int64_t i = 0; i < n; ++i) {
        oracle_terms r;
        oracle_adamw_element((double)w[i], (double)g[i] * grad_scale,
                             (double)m[i], (double)v[i], s, t, lr, wd, beta1,
                             beta2, eps, &r);
        w[i] = (float)r.w;
        m[i] = (float)r.m;
        v[i] = (float)r.v;
    }
    return OR_OK;
}

/* ------------------------------------------------------------------------
 * 16-bit formats of the mixed-precision step.  "Grow a Language Model:
 * Backprop" (unhomeschool.com): FP16 gradient buffers (section "Where the
 * gradients live": ~240 MB at FP16 for 120M parameters) and an FP16 cuBLAS
 * path (section "Framework overhead").  The optimizer keeps float32 master
 * weights and moments; gradients arrive in bfloat16 or IEEE binary16, and a
 * 16-bit copy of the new weights is produced for the next forward pass.
 * Decoding is exact; encoding rounds to nearest, ties to even.
 *
 * bfloat16: the top 16 bits of a binary32 value.
 * binary16 (IEEE 754-2008): 1 sign bit, 5 exponent bits (bias 15), 10
 * fraction bits; exponent 0 = zero or subnormal (fraction x 2^-24),
 * exponent 31 = inf or nan.
 * ---------------------------------------------------------------------- */
#define DT_F32 0
#define DT_BF16 1
#define DT_F16 2

double oracle_decode16(uint16_t h, int32_t dtype)
{
    if (dtype == DT_BF16) {
        uint32_t bits = (uint32_t)h << 16;
        float f;
        memcpy(&f, &bits, 4);
        return (double)f;
    }
    int sign = (h >> 15) & 1;
    int ex = (h >> 10) & 31;
    int frac = h & 1023;
    double mag;
    if (ex == 0)
        mag = ldexp((double)frac, -24);
    else if (ex == 31)
        mag = frac ? NAN : INFINITY;
    else
        mag = ldexp((double)(1024 + frac), ex - 25);
    return sign ? -mag : mag;
}

uint16_t oracle_encode16(float x, int32_t dtype)
{
    uint32_t bits;
    memcpy(&bits, &x, 4);
    if (dtype == DT_BF16) {
        if ((bits & 0x7fffffffu) > 0x7f800000u)          /* nan: keep it a nan */
            return (uint16_t)((bits >> 16) | 0x0040u);
        uint32_t lsb = (bits >> 16) & 1u;
        return (uint16_t)((bits + 0x7fffu + lsb) >> 16);  /* nearest, ties even */
    }
    /* binary16: nearest representable value, ties to the even fraction */
    uint16_t sign = (uint16_t)((bits >> 16) & 0x8000u);
    double a = fabs((double)x);
    if (x != x)
        return (uint16_t)(sign | 0x7e00u);
    if (a >= 65520.0)                                    /* rounds past 65504 */
        return (uint16_t)(sign | 0x7c00u);
    /* step between neighbours at a: 2^-24 below 2^-14, else 2^(e-10) */
    int e;
    frexp(a, &e);                                        /* a = f 2^e, f in [0.5,1) */
    int q = (e - 1 < -14) ? -24 : (e - 1) - 10;          /* exponent of one step */
    double steps = ldexp(a, -q);                         /* exact: a is a float */
    double fl = floor(steps);
    double rem = steps - fl;
    uint32_t k = (uint32_t)fl;
    if (rem > 0.5 || (rem == 0.5 && (k & 1u)))
        k += 1;
    /* k steps of 2^q: rebuild the encoding */
    double val = ldexp((double)k, q);
    if (val == 0.0)
        return sign;
    int ve;
    frexp(val, &ve);
    if (ve - 1 < -14)                                    /* subnormal */
        return (uint16_t)(sign | (uint16_t)k);
    uint32_t exp_field = (uint32_t)(ve - 1 + 15);
    uint32_t frac_field = (uint32_t)(ldexp(val, -(ve - 1)) * 1024.0 - 1024.0);
    return (uint16_t)(sign | (exp_field << 10) | frac_field);
}

/* The step with a 16-bit (or float32) gradient and an optional 16-bit copy
 * of the new weights: each gradient value decoded exactly, times
 * grad_scale, then norm, clip and update as oracle_adamw_clip_step_scaled;
 * w_lp (if not NULL) receives the new float32 weights rounded to w_lp_dtype. */
int oracle_adamw_clip_step_mixed(float* w, const void* g, int32_t g_dtype, float* m,
                                 float* v, uint16_t* w_lp, int32_t w_lp_dtype,
                                 int64_t n, int32_t t, double lr, double wd,
                                 double clip, double grad_scale, double beta1,
                                 double beta2, double eps, double* norm_out)
{
    if (n < 0 || t < 1)
        return OR_EINVAL;
    double sumsq = 0.0;
    for (int64_t i = 0; i < n; ++i) {
        double gi = g_dtype == DT_F32 ? (double)((const float*)g)[i]
                                      : oracle_decode16(((const uint16_t*)g)[i], g_dtype);
        double x = gi * grad_scale;
        sumsq = sumsq + x * x;
    }
    double norm = sqrt(sumsq);
    if (norm_out)
        *norm_out = norm;
    if (!isfinite(norm))
        return OR_ENONFINITE;
    double s = oracle_clip_scale(norm, clip);
    for (int64_t i = 0; i < n; ++i) {
        double gi = g_dtype == DT_F32 ? (double)((const float*)g)[i]
                                      : oracle_decode16(((const uint16_t*)g)[i], g_dtype);
        oracle_terms r;
        oracle_adamw_element((double)w[i], gi * grad_scale, (double)m[i],
                             (double)v[i], s, t, lr, wd, beta1, beta2, eps, &r);
        w[i] = (float)r.w;
        m[i] = (float)r.m;
        v[i] = (float)r.v;
        if (w_lp)
            w_lp[i] = oracle_encode16(w[i], w_lp_dtype);
    }
    return OR_OK;
}

/* The update half of the step over the index range [lo, hi) only, in place,
 * given the clip factor s of the whole gradient: the same per-element
 * definition as oracle_adamw_clip_step's loop.  Used to run the oracle on
 * several host threads (each a disjoint range) for the CPU baseline. */
int oracle_adamw_update_range(float* w, const float* g, float* m, float* v,
                              int64_t lo, int64_t hi, double s, int32_t t,
                              double lr, double wd, double beta1, double beta2,
                              double eps)
{
    if (lo < 0 || hi < lo || t < 1)
        return OR_EINVAL;
    for (int64_t j = lo; j < hi; ++j) {
        oracle_terms r;
        oracle_adamw_element((double)w[j], (double)g[j], (double)m[j],
                             (double)v[j], s, t, lr, wd, beta1, beta2, eps, &r);
        w[j] = (float)r.w;
        m[j] = (float)r.m;
        v[j] = (float)r.v;
    }
    return OR_OK;
}

/* ------------------------------------------------------------------------
 * Per-group weight decay.  [T] "The Exact Targets of Clipping and AdamW":
 * the lesson applies the decoupled decay to every parameter, normalisation
 * gains and biases included, as a simple convention that it does not claim
 * to be the best grouping.  The other grouping kept here: a flag per tensor
 * of the offset table; a tensor whose flag is 0 is updated with wd = 0 (its
 * old weight is multiplied by exactly 1), every other tensor with wd.  The
 * norm and the clip factor stay global over all of g.  The tensors must
 * tile [0, n) in order (offsets[k] + numels[k] == offsets[k + 1]).
 * ---------------------------------------------------------------------- */
int oracle_adamw_clip_step_masked(float* w, const float* g, float* m, float* v,
                                  int64_t n, const int64_t* offsets,
                                  const int64_t* numels, int32_t n_tensors,
                                  const uint8_t* decay, int32_t t, double lr,
                                  double wd, double clip, double beta1,
                                  double beta2, double eps, double* norm_out)
{
    if (n < 0 || t < 1 || n_tensors < 0)
        return OR_EINVAL;
    int64_t next = 0;
    for (int32_t k = 0; k < n_tensors; ++k) {
        if (offsets[k] != next || numels[k] < 0)
            return OR_EINVAL;
        next = offsets[k] + numels[k];
    }
    if (next != n)
        return OR_EINVAL;
    double norm = oracle_global_norm(g, n);
    if (norm_out)
        *norm_out = norm;
    if (!isfinite(norm))
        return OR_ENONFINITE;
    double s = oracle_clip_scale(norm, clip);
    for (int32_t k = 0; k < n_tensors; ++k) {
        double wd_k = decay[k] ? wd : 0.0;
        for (int64_t i = offsets[k]; i < offsets[k] + numels[k]; ++i) {
            oracle_terms r;
            oracle_adamw_element((double)w[i], (double)g[i], (double)m[i],
                                 (double)v[i], s, t, lr, wd_k, beta1, beta2,
                                 eps, &r);
            w[i] = (float)r.w;
            m[i] = (float)r.m;
            v[i] = (float)r.v;
        }
    }
    return OR_OK;
}

/* The same update at chosen indices only, given the clip factor s (from a
 * full-vector norm computed separately).  Used to check outputs of a large
 * state one element at a time.  Results go to the *_out arrays. */
void oracle_adamw_at(const int64_t* idx, int64_t k, const float* w,
                     const float* g, const float* m, const float* v, double s,
                     int32_t t, double lr, double wd, double beta1,
                     double beta2, double eps, float* w_out, float* m_out,
                     float* v_out)
{
    for (int64_t j = 0; j < k; ++j) {
        int64_t i = idx[j];
        oracle_terms r;
        oracle_adamw_element((double)w[i], (double)g[i], (double)m[i],
                             (double)v[i], s, t, lr, wd, beta1, beta2, eps, &r);
        w_out[j] = (float)r.w;
        m_out[j] = (float)r.m;
        v_out[j] = (float)r.v;
    }
}

/* All eight double terms of the update at chosen indices (row j of out holds
 * g_hat, m, v, m_hat, v_hat, w_decayed, update, w for idx[j]).  The tests
 * use them as the magnitudes that a float32 result may differ by, relative
 * to: the new weight is a difference of two terms that can cancel. */
void oracle_adamw_terms_at(const int64_t* idx, int64_t k, const float* w,
                           const float* g, const float* m, const float* v,
                           double s, int32_t t, double lr, double wd,
                           double beta1, double beta2, double eps, double* out)
{
    for (int64_t j = 0; j < k; ++j) {
        int64_t i = idx[j];
        oracle_terms r;
        oracle_adamw_element((double)w[i], (double)g[i], (double)m[i],
                             (double)v[i], s, t, lr, wd, beta1, beta2, eps, &r);
        double* o = out + 8 * j;
        o[0] = r.g_hat;
        o[1] = r.m;
        o[2] = r.v;
        o[3] = r.m_hat;
        o[4] = r.v_hat;
        o[5] = r.w_decayed;
        o[6] = r.update;
        o[7] = r.w;
    }
}

/* ------------------------------------------------------------------------
 * The step_NNNNNN.bin image.  [C] "Format" / "Region by region" /
 * "Total size": five contiguous regions
 *     [int32 step][int32 n_params][n x f32 weights][n x f32 m][n x f32 v],
 * 8 + 12 n bytes in total, no other metadata.  The pages do not state the
 * byte order; this oracle writes little-endian two's-complement integers and
 * little-endian IEEE binary32 floats, one byte at a time for the header so
 * that the order is explicit.
 * ---------------------------------------------------------------------- */
static void put_le32(unsigned char* p, uint32_t x)
{
    p[0] = (unsigned char)(x & 0xffu);
    p[1] = (unsigned char)((x >> 8) & 0xffu);
    p[2] = (unsigned char)((x >> 16) & 0xffu);
    p[3] = (unsigned char)((x >> 24) & 0xffu);
}

static uint32_t get_le32(const unsigned char* p)
{
    return (uint32_t)p[0] | ((uint32_t)p[1] << 8) | ((uint32_t)p[2] << 16) |
           ((uint32_t)p[3] << 24);
}

static int host_is_little_endian(void)
{
    uint32_t one = 1;
    unsigned char b;
    memcpy(&b, &one, 1);
    return b == 1;
}

int64_t oracle_ckpt_size(int64_t n) { return 8 + 12 * n; }

/* Writes the 8 + 12 n byte image into out. */
int oracle_pack(int32_t step, int32_t n, const float* w, const float* m,
                const float* v, unsigned char* out)
{
    if (n < 0 || step < 0 || !host_is_little_endian())
        return OR_EINVAL;
    put_le32(out, (uint32_t)step);
    put_le32(out + 4, (uint32_t)n);
    size_t bytes = (size_t)n * 4u;
    memcpy(out + 8, w, bytes);
    memcpy(out + 8 + bytes, m, bytes);
    memcpy(out + 8 + 2 * bytes, v, bytes);
    return OR_OK;
}

static int write_all(FILE* f, const void* p, size_t bytes)
{
    return fwrite(p, 1, bytes, f) == bytes ? OR_OK : OR_EIO;
}

/* ------------------------------------------------------------------------
 * Atomic checkpoint write.  [S] "Atomic write": write the data to
 * <name>.tmp, fsync it, then rename over the final name; POSIX rename on one
 * file system is atomic, so a crash before the rename leaves the previous
 * checkpoint live.  The directory is fsynced after the rename so that the
 * new name itself is durable.  File name: step_%06d.bin ([C] uses
 * step_NNNNNN.bin and step_112700.bin).
 * ---------------------------------------------------------------------- */
int oracle_ckpt_write(const char* dir, int32_t step, int32_t n, const float* w,
                      const float* m, const float* v, char* path_out,
                      size_t path_cap)
{
    if (!dir || n < 0 || step < 0 || !host_is_little_endian())
        return OR_EINVAL;
    char final_path[4096], tmp_path[4112];
    int len = snprintf(final_path, sizeof final_path, "%s/step_%06d.bin", dir,
                       (int)step);
    if (len < 0 || (size_t)len >= sizeof final_path)
        return OR_EINVAL;
    snprintf(tmp_path, sizeof tmp_path, "%s.tmp", final_path);

    FILE* f = fopen(tmp_path, "wb");
    if (!f)
        return OR_EIO;
    unsigned char header[8];
    put_le32(header, (uint32_t)step);
    put_le32(header + 4, (uint32_t)n);
    size_t bytes = (size_t)n * 4u;
    int rc = write_all(f, header, 8);
    if (rc == OR_OK)
        rc = write_all(f, w, bytes);
    if (rc == OR_OK)
        rc = write_all(f, m, bytes);
    if (rc == OR_OK)
        rc = write_all(f, v, bytes);
    if (rc == OR_OK && fflush(f) != 0)
        rc = OR_EIO;
    if (rc == OR_OK && fsync(fileno(f)) != 0)
        rc = OR_EIO;
    if (fclose(f) != 0 && rc == OR_OK)
        rc = OR_EIO;
    if (rc != OR_OK) {
        unlink(tmp_path);
        return rc;
    }
    if (rename(tmp_path, final_path) != 0) {
        unlink(tmp_path);
        return OR_EIO;
    }
    int dfd = open(dir, O_RDONLY);
    if (dfd >= 0) {
        fsync(dfd);
        close(dfd);
    }
    if (path_out && path_cap > 0)
        snprintf(path_out, path_cap, "%s", final_path);
    return OR_OK;
}

/* ------------------------------------------------------------------------
 * Validating read.  [S] "Three failure modes" asks that a bad checkpoint be
 * refused loudly instead of loaded silently; for the single-file format of
 * [C] the checks available are: the header is readable, step and n are not
 * negative, n equals the caller's parameter count, and the file holds
 * exactly 8 + 12 n bytes (a partial write is shorter).  Only after all
 * checks pass are w, m, v filled.
 * ---------------------------------------------------------------------- */
int oracle_ckpt_read(const char* path, int32_t n_expected, int32_t* step_out,
                     float* w, float* m, float* v)
{
    if (!path || n_expected < 0 || !host_is_little_endian())
        return OR_EINVAL;
    FILE* f = fopen(path, "rb");
    if (!f)
        return OR_EIO;
    struct stat st;
    if (fstat(fileno(f), &st) != 0) {
        fclose(f);
        return OR_EIO;
    }
    unsigned char header[8];
    if (st.st_size < 8 || fread(header, 1, 8, f) != 8) {
        fclose(f);
        return OR_ESIZE;
    }
    int32_t step = (int32_t)get_le32(header);
    int32_t n = (int32_t)get_le32(header + 4);
    if (step < 0 || n < 0) {
        fclose(f);
        return OR_EFORMAT;
    }
    if (n != n_expected) {
        fclose(f);
        return OR_EMISMATCH;
    }
    if ((int64_t)st.st_size != oracle_ckpt_size(n)) {
        fclose(f);
        return OR_ESIZE;
    }
    size_t bytes = (size_t)n * 4u;
    if (fread(w, 1, bytes, f) != bytes || fread(m, 1, bytes, f) != bytes ||
        fread(v, 1, bytes, f) != bytes) {
        fclose(f);
        return OR_ESIZE;
    }
    fclose(f);
    if (step_out)
        *step_out = step;
    return OR_OK;
}
