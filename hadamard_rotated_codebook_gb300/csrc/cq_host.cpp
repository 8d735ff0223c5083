// cq_host.cpp -- host side of libcq: error reporting, codebooks, byte
// accounting, argument validation for the device entry points, and the
// .cact-shaped container.
#include <cerrno>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <string>
#include <vector>

#include "cq_internal.h"

namespace cq {

static thread_local char g_err[512] = "";

int set_error(int code, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof(g_err), fmt, ap);
    va_end(ap);
    return code;
}

void clear_error() { g_err[0] = '\0'; }

// Prefixes the current message with "descriptor i: " and returns `code`.
static int prefix_error(int code, int i) {
    char tmp[sizeof(g_err)];
    std::snprintf(tmp, sizeof(tmp), "descriptor %d: %.480s", i, g_err);
    std::memcpy(g_err, tmp, sizeof(g_err));
    return code;
}

int check_codebook(const float *cb, int bits) {
    const int L = levels_of(bits);
    if (L < 0) return set_error(CQ_ERR_ARG, "bits must be 2, 3, 4 or 5 (ternary), got %d", bits);
    if (!cb) return set_error(CQ_ERR_ARG, "codebook is NULL");
    for (int j = 0; j < L; ++j)
        if (!std::isfinite(cb[j])) return set_error(CQ_ERR_ARG, "codebook[%d] is not finite", j);
    for (int j = 0; j + 1 < L; ++j)
        if (!(cb[j] < cb[j + 1]))
            return set_error(CQ_ERR_ARG, "codebook must be strictly increasing (entry %d)", j);
    return CQ_OK;
}

static bool is_pow2(uint64_t v) { return v && !(v & (v - 1)); }

// Upper tail of the standard normal and its density.
static double upper_tail(double x) { return 0.5 * std::erfc(x / std::sqrt(2.0)); }
static double density(double x) {
    return std::isinf(x) ? 0.0 : std::exp(-0.5 * x * x) / std::sqrt(2.0 * M_PI);
}

// Positive half of the L-level Lloyd-Max quantiser of N(0,1), L even. The
// density is symmetric, so the optimal quantiser is too and only the
// positive cells [t_i, t_{i+1}) with t_0 = 0 need iterating.
static void lloyd_max_half(int L, double *c) {
    const int h = L / 2;
    for (int i = 0; i < h; ++i) c[i] = (i + 0.5) * 3.0 / h;
    std::vector<double> t(h + 1);
    for (int it = 0; it < 1000000; ++it) {
        t[0] = 0.0;
        for (int i = 1; i < h; ++i) t[i] = 0.5 * (c[i - 1] + c[i]);
        t[h] = INFINITY;
        double change = 0.0;
        for (int i = 0; i < h; ++i) {
            double mass = upper_tail(t[i]) - upper_tail(t[i + 1]);
            double ci = (density(t[i]) - density(t[i + 1])) / mass;
            change = std::fmax(change, std::fabs(ci - c[i]));
            c[i] = ci;
        }
        if (change < 1e-15) break;
    }
}

// Level by code (16 entries): the codebook, or for the ternary marker the
// 2-bit crumbs read as signed (01 -> +c, 11 -> -c, 10 -> -2c, never written).
void level_table(int bits, const float *codebook, float lv[16]) {
    for (int j = 0; j < 16; ++j) lv[j] = 0.0f;
    if (bits == 5) {
        const float c = codebook[2];
        lv[1] = c;
        lv[2] = -2.0f * c;
        lv[3] = -c;
    } else {
        for (int j = 0; j < levels_of(bits); ++j) lv[j] = codebook[j];
    }
}

}  // namespace cq

using namespace cq;

extern "C" {

const char *cq_last_error(void) { return g_err; }

int cq_version(void) { return 10000; }

int cq_levels(int bits) { return levels_of(bits); }

int cq_code_width(int bits) { return width_of(bits); }

int cq_codebook_init(int bits, int group, float *levels, size_t cap, size_t *n_levels) {
    clear_error();
    const int L = levels_of(bits);
    if (L < 0) return set_error(CQ_ERR_ARG, "bits must be 1, 2, 3, 4 or 5, got %d", bits);
    if (group < 8 || !is_pow2((uint64_t)group))
        return set_error(CQ_ERR_ARG, "group must be a power of two >= 8, got %d", group);
    if (n_levels) *n_levels = (size_t)L;
    if (!levels) return CQ_OK;
    if (cap < (size_t)L) return set_error(CQ_ERR_ARG, "levels buffer holds %zu, need %d", cap, L);
    const double scale = 1.0 / std::sqrt((double)group);
    if (bits == 5) {
        // [NJ] "Shared codebooks": ternary levels {-1.2240064, 0, +1.2240064}/sqrt(group).
        float c = (float)(1.2240064 * scale);
        levels[0] = -c;
        levels[1] = 0.0f;
        levels[2] = c;
        return CQ_OK;
    }
    double half[8];
    lloyd_max_half(L, half);
    for (int i = 0; i < L / 2; ++i) {
        float v = (float)(half[i] * scale);
        levels[L / 2 + i] = v;
        levels[L / 2 - 1 - i] = -v;
    }
    return CQ_OK;
}

uint64_t cq_packed_bytes(int out, int in, int group, int bits) {
    if (out < 0 || in < 0 || group < 8 || !is_pow2((uint64_t)group) || levels_of(bits) < 0) return 0;
    const uint64_t ip = ((uint64_t)in + group - 1) / group * group;
    return (uint64_t)out * ip * (uint64_t)width_of(bits) / 8 + (uint64_t)out * (ip / group) * 2;
}

// ------------------------------------------------------------ device calls --

// wide: the entry point also takes group 64 and binary codes (encode, GEMV,
// row gather); the GEMM and the KV cache take group 128 and 2..5 bits.
static int check_matrix(int out, int in, int group, int bits, bool wide = true) {
    if (levels_of(bits) < 0) return set_error(CQ_ERR_ARG, "bits must be 1, 2, 3, 4 or 5, got %d", bits);
    if (wide && group != kGroup && group != kGroup64)
        return set_error(CQ_ERR_SHAPE, "this entry point supports group = 64 or 128, got %d", group);
    if (!wide && group != kGroup)
        return set_error(CQ_ERR_SHAPE, "this entry point supports group = 128 only, got %d", group);
    if (!wide && bits == 1) return set_error(CQ_ERR_SHAPE, "this entry point does not take binary codes");
    if (out < 0 || in < 0) return set_error(CQ_ERR_SHAPE, "negative size out=%d in=%d", out, in);
    if ((int64_t)out * in_padded(in, group) > ((int64_t)1 << 40))
        return set_error(CQ_ERR_SHAPE, "matrix too large");
    return CQ_OK;
}

int cq_encode(const float *W, int out, int in, int group, int bits, const float *codebook,
              uint8_t *blob, void *stream) {
    clear_error();
    int st = check_matrix(out, in, group, bits);
    if (st) return st;
    if ((st = check_codebook(codebook, bits))) return st;
    if (out == 0 || in == 0) return CQ_OK;  // empty matrix: nothing to write
    if (!W || !blob) return set_error(CQ_ERR_ARG, "W and blob must be non-null");
    return launch_encode(W, out, in, group, bits, codebook, blob, stream);
}

int cq_act_quant_int8(const float *X, int M, int in, int8_t *Xq, float *s, void *stream) {
    clear_error();
    if (M < 0 || in < 0) return set_error(CQ_ERR_SHAPE, "negative size");
    if (M == 0) return CQ_OK;
    if (!X || !Xq || !s) return set_error(CQ_ERR_ARG, "null pointer");
    return launch_act_quant(X, M, in, Xq, s, stream);
}

static int check_gemv_desc(const cq_gemv_desc &d, int i) {
    int st = check_matrix(d.out, d.in, d.group, d.bits);
    if (st) return prefix_error(st, i);
    if ((st = check_codebook(d.codebook, d.bits))) return prefix_error(st, i);
    if (d.B < 1 || d.B > CQ_GEMV_MAX_BATCH)
        return set_error(CQ_ERR_SHAPE, "descriptor %d: batch must be 1..%d, got %d", i, CQ_GEMV_MAX_BATCH, d.B);
    if (d.x_dtype != CQ_X_F32 && d.x_dtype != CQ_X_I8 && d.x_dtype != CQ_X_F32Q)
        return set_error(CQ_ERR_ARG, "descriptor %d: unknown x_dtype %d", i, d.x_dtype);
    if (d.out > 0 && !d.y) return set_error(CQ_ERR_ARG, "descriptor %d: null y", i);
    if (d.out > 0 && d.in > 0 && !d.blob) return set_error(CQ_ERR_ARG, "descriptor %d: null blob", i);
    if (d.out > 0 && d.in > 0 && !d.x) return set_error(CQ_ERR_ARG, "descriptor %d: null x", i);
    if (reinterpret_cast<uintptr_t>(d.blob) & 15)
        return set_error(CQ_ERR_ARG, "descriptor %d: blob must be 16-byte aligned", i);
    if (d.x_dtype == CQ_X_I8 && d.out > 0 && !d.x_scale)
        return set_error(CQ_ERR_ARG, "descriptor %d: int8 activations need x_scale", i);
    return CQ_OK;
}

int cq_gemv(const uint8_t *blob, int out, int in, int group, int bits, const float *codebook,
            const void *x, int x_dtype, const float *x_scale, int B, float *y, void *stream) {
    cq_gemv_desc d;
    d.blob = blob;
    d.x = x;
    d.x_scale = x_scale;
    d.y = y;
    d.codebook = codebook;
    d.out = out;
    d.in = in;
    d.group = group;
    d.bits = bits;
    d.x_dtype = x_dtype;
    d.B = B;
    return cq_gemv_grouped(&d, 1, stream);
}

int cq_gemv_grouped(const cq_gemv_desc *descs, int n, void *stream) {
    clear_error();
    if (!descs || n < 1 || n > CQ_MAX_GROUPED)
        return set_error(CQ_ERR_ARG, "need 1..%d descriptors, got %d", CQ_MAX_GROUPED, n);
    for (int i = 0; i < n; ++i) {
        int st = check_gemv_desc(descs[i], i);
        if (st) return st;
    }
    return launch_gemv_grouped(descs, n, stream);
}

int cq_gemv_shared(const uint8_t *const *blobs, const int *outs, int n_mats, int in, int group, int bits,
                   const float *codebook, const void *x, int x_dtype, const float *x_scale, int B, float *const *ys,
                   void *stream) {
    clear_error();
    if (!blobs || !outs || !ys) return set_error(CQ_ERR_ARG, "null blobs, outs or ys array");
    if (n_mats < 1 || n_mats > CQ_MAX_GROUPED)
        return set_error(CQ_ERR_ARG, "need 1..%d matrices, got %d", CQ_MAX_GROUPED, n_mats);
    cq_gemv_desc d[CQ_MAX_GROUPED];
    for (int j = 0; j < n_mats; ++j) {
        d[j].blob = blobs[j];
        d[j].x = x;
        d[j].x_scale = x_scale;
        d[j].y = ys[j];
        d[j].codebook = codebook;
        d[j].out = outs[j];
        d[j].in = in;
        d[j].group = group;
        d[j].bits = bits;
        d[j].x_dtype = x_dtype;
        d[j].B = B;
    }
    return cq_gemv_grouped(d, n_mats, stream);
}

int cq_gather_rows(const uint8_t *blob, int out, int in, int group, int bits, const float *codebook,
                   const int32_t *idx, int n, float *dst, void *stream) {
    clear_error();
    int st = check_matrix(out, in, group, bits);
    if (st) return st;
    if ((st = check_codebook(codebook, bits))) return st;
    if (n < 0) return set_error(CQ_ERR_SHAPE, "negative row count %d", n);
    if (n == 0 || in == 0) return CQ_OK;
    if (!idx || !dst) return set_error(CQ_ERR_ARG, "null idx or dst");
    if (out > 0 && !blob) return set_error(CQ_ERR_ARG, "null blob");
    if (reinterpret_cast<uintptr_t>(blob) & 15) return set_error(CQ_ERR_ARG, "blob must be 16-byte aligned");
    float lv[16];
    level_table(bits, codebook, lv);
    return launch_gather_rows(blob, out, in, group, bits, lv, idx, n, dst, stream);
}

int cq_kv_write(uint8_t *cache, int cap, int in, int bits, const float *codebook, const float *rows, int t0, int n,
                void *stream) {
    clear_error();
    int st = check_matrix(cap, in, kGroup, bits, false);
    if (st) return st;
    if ((st = check_codebook(codebook, bits))) return st;
    if (n < 0 || t0 < 0 || (long long)t0 + n > cap)
        return set_error(CQ_ERR_SHAPE, "rows %d..%lld outside a cache of %d rows", t0, (long long)t0 + n - 1, cap);
    if (n == 0 || in == 0) return CQ_OK;
    if (!cache || !rows) return set_error(CQ_ERR_ARG, "null cache or rows");
    if (reinterpret_cast<uintptr_t>(cache) & 15) return set_error(CQ_ERR_ARG, "cache must be 16-byte aligned");
    const size_t rb = (size_t)in_padded(in) * width_of(bits) / 8, ng = in_padded(in) / kGroup;
    uint8_t *codes = cache + (size_t)t0 * rb;
    uint8_t *norms = cache + (size_t)cap * rb + 2 * ng * (size_t)t0;
    return launch_encode_rows(rows, n, in, kGroup, bits, codebook, codes, norms, stream);
}

int cq_kv_attend(const cq_kv_geom *g, const cq_kv_seq *seqs, int n_seqs, void *stream) {
    clear_error();
    if (!g || !seqs) return set_error(CQ_ERR_ARG, "null geometry or sequence array");
    if (n_seqs < 1) return set_error(CQ_ERR_ARG, "need at least one sequence, got %d", n_seqs);
    if (g->n_q_heads < 1 || g->n_q_heads > 16 || g->n_kv_heads < 1 || g->n_q_heads % g->n_kv_heads)
        return set_error(CQ_ERR_SHAPE, "need 1..16 query heads, a multiple of the %d key/value heads; got %d",
                         g->n_kv_heads, g->n_q_heads);
    if (g->head_dim_k < 1 || g->head_dim_v < 1 || (long long)g->n_kv_heads * g->head_dim_k > 512 ||
        (long long)g->n_kv_heads * g->head_dim_v > 512)
        return set_error(CQ_ERR_SHAPE, "cache rows of %d x %d (keys) and %d x %d (values) exceed 512 or are empty",
                         g->n_kv_heads, g->head_dim_k, g->n_kv_heads, g->head_dim_v);
    if (width_of(g->k_bits) < 2 || width_of(g->v_bits) < 2)
        return set_error(CQ_ERR_ARG, "bits must be 2, 3, 4 or 5 (got %d, %d)", g->k_bits, g->v_bits);
    int st = check_codebook(g->k_codebook, g->k_bits);
    if (st) return st;
    if ((st = check_codebook(g->v_codebook, g->v_bits))) return st;
    if (!std::isfinite(g->scale)) return set_error(CQ_ERR_ARG, "scale must be finite");
    for (int i = 0; i < n_seqs; ++i) {
        const cq_kv_seq &s = seqs[i];
        if (s.cap < 0 || s.n_tokens < 0 || s.n_tokens > s.cap)
            return set_error(CQ_ERR_SHAPE, "sequence %d: n_tokens %d outside 0..cap (%d)", i, s.n_tokens, s.cap);
        if (!s.o || (s.n_tokens > 0 && (!s.q || !s.k_cache || !s.v_cache)))
            return set_error(CQ_ERR_ARG, "sequence %d: null cache, q or o", i);
        if ((reinterpret_cast<uintptr_t>(s.k_cache) | reinterpret_cast<uintptr_t>(s.v_cache)) & 15)
            return set_error(CQ_ERR_ARG, "sequence %d: caches must be 16-byte aligned", i);
    }
    float lk[16], lv[16];
    level_table(g->k_bits, g->k_codebook, lk);
    level_table(g->v_bits, g->v_codebook, lv);
    return launch_kv_attend(*g, seqs, n_seqs, lk, lv, stream);
}

static int check_gemm_desc(const cq_gemm_desc &d, int i) {
    // binary codes at any width; groups of 64 on inputs of whole 128-wide
    // spans up to 512 (the product that rotates the weight rows)
    int st = check_matrix(d.out, d.in, d.group, d.bits, true);
    if (st) return prefix_error(st, i);
    if (d.group == kGroup64 && (d.in % kGroup != 0 || d.in > 4 * kGroup))
        return prefix_error(set_error(CQ_ERR_SHAPE, "groups of 64 need in a multiple of 128 and at most 512, got %d", d.in), i);
    if ((st = check_codebook(d.codebook, d.bits))) return prefix_error(st, i);
    if (d.M < 0) return set_error(CQ_ERR_SHAPE, "descriptor %d: negative M", i);
    if (d.M > 0 && d.out > 0 && !d.Y) return set_error(CQ_ERR_ARG, "descriptor %d: null Y", i);
    if (d.M > 0 && d.out > 0 && d.in > 0 && (!d.blob || !d.Xq || !d.x_scale))
        return set_error(CQ_ERR_ARG, "descriptor %d: null blob, Xq or x_scale", i);
    if (reinterpret_cast<uintptr_t>(d.blob) & 15)
        return set_error(CQ_ERR_ARG, "descriptor %d: blob must be 16-byte aligned", i);
    return CQ_OK;
}

}  // extern "C"

namespace cq {
int check_gemm_args(const cq_gemm_desc &d) { return check_gemm_desc(d, 0); }
}  // namespace cq

extern "C" {

int cq_gemm(const uint8_t *blob, int out, int in, int group, int bits, const float *codebook,
            const int8_t *Xq, const float *x_scale, int M, float *Y, void *stream) {
    cq_gemm_desc d;
    d.blob = blob;
    d.Xq = Xq;
    d.x_scale = x_scale;
    d.Y = Y;
    d.codebook = codebook;
    d.out = out;
    d.in = in;
    d.group = group;
    d.bits = bits;
    d.M = M;
    return cq_gemm_grouped(&d, 1, stream);
}

int cq_gemm_grouped(const cq_gemm_desc *descs, int n, void *stream) {
    clear_error();
    if (!descs || n < 1 || n > CQ_MAX_GROUPED)
        return set_error(CQ_ERR_ARG, "need 1..%d descriptors, got %d", CQ_MAX_GROUPED, n);
    for (int i = 0; i < n; ++i) {
        int st = check_gemm_desc(descs[i], i);
        if (st) return st;
    }
    return launch_gemm_grouped(descs, n, stream);
}

int cq_device_status(void *stream) {
    clear_error();
    return read_and_clear_device_status(stream);
}


// --------------------------------------------------------------- container --

struct cq_cact {
    std::vector<uint8_t> bytes;
    uint32_t n = 0;
    uint32_t group = 0;
    float codebook[28];
    std::vector<cq_tensor_desc> t;
};

static void put_u16(std::vector<uint8_t> &b, size_t o, uint16_t v) {
    b[o] = (uint8_t)v;
    b[o + 1] = (uint8_t)(v >> 8);
}
static void put_u32(std::vector<uint8_t> &b, size_t o, uint32_t v) {
    for (int i = 0; i < 4; ++i) b[o + i] = (uint8_t)(v >> (8 * i));
}
static void put_u64(std::vector<uint8_t> &b, size_t o, uint64_t v) {
    for (int i = 0; i < 8; ++i) b[o + i] = (uint8_t)(v >> (8 * i));
}
static uint32_t get_u32(const uint8_t *p) {
    return (uint32_t)p[0] | ((uint32_t)p[1] << 8) | ((uint32_t)p[2] << 16) | ((uint32_t)p[3] << 24);
}
static uint64_t get_u64(const uint8_t *p) { return (uint64_t)get_u32(p) | ((uint64_t)get_u32(p + 4) << 32); }

static uint64_t align_up(uint64_t v, uint64_t a) { return (v + a - 1) / a * a; }

// Element count of a descriptor; false on overflow.
static bool element_count(const cq_tensor_desc &d, uint64_t *count) {
    uint64_t n = 1;
    for (int i = 0; i < d.ndim; ++i) {
        if (d.shape[i] && n > UINT64_MAX / d.shape[i]) return false;
        n *= d.shape[i];
    }
    *count = n;
    return true;
}

// Shared record validation for the writer and the reader. Returns a static
// message or nullptr.
static const char *record_problem(const cq_tensor_desc &d) {
    if (d.dtype < CQ_DTYPE_FP16 || d.dtype > CQ_DTYPE_RAW) return "unknown dtype";
    if (d.ndim > 4) return "ndim > 4";
    for (int i = d.ndim; i < 4; ++i)
        if (d.shape[i] != 0) return "unused shape entries must be 0";
    if (d.dtype == CQ_DTYPE_FP16 || d.dtype == CQ_DTYPE_FP32) {
        uint64_t n = 0;
        if (!element_count(d, &n)) return "shape overflows";
        const uint64_t es = d.dtype == CQ_DTYPE_FP16 ? 2 : 4;
        if (n > UINT64_MAX / es || n * es != d.nbytes) return "nbytes does not match shape";
        if (d.group != 0 || d.bits != 0) return "group/bits must be 0 for FP16/FP32";
    } else if (d.dtype == CQ_DTYPE_CQ) {
        if (d.ndim != 2) return "a CQ tensor must be 2-D [out, in]";
        if (d.group < 8 || !is_pow2(d.group)) return "CQ group must be a power of two >= 8";
        if (levels_of((int)d.bits) < 0) return "CQ bits must be 2, 3, 4 or 5";
        if (d.shape[0] > INT32_MAX || d.shape[1] > INT32_MAX) return "CQ shape too large";
        uint64_t want = cq_packed_bytes((int)d.shape[0], (int)d.shape[1], (int)d.group, (int)d.bits);
        if (want != d.nbytes) return "CQ nbytes inconsistent with shape, group and bits";
    } else {  // RAW
        if (d.group != 0 || d.bits != 0) return "group/bits must be 0 for RAW";
    }
    return nullptr;
}

int cq_cact_write(const char *path, const cq_tensor_desc *t, int n, const float codebook[28],
                  uint32_t default_group) {
    clear_error();
    if (!path || n < 0 || (n > 0 && !t) || !codebook) return set_error(CQ_ERR_ARG, "null argument");
    for (int i = 0; i < n; ++i) {
        const char *p = record_problem(t[i]);
        if (p) return set_error(CQ_ERR_ARG, "tensor %d: %s", i, p);
        if (t[i].nbytes && !t[i].data) return set_error(CQ_ERR_ARG, "tensor %d: null data", i);
    }
    const uint64_t dir_off = CQ_CACT_HEADER_BYTES + 4ull * CQ_CACT_CODEBOOK_LEN;
    uint64_t off = align_up(dir_off + (uint64_t)n * CQ_CACT_RECORD_BYTES, CQ_CACT_ALIGN);
    std::vector<uint64_t> offs(n);
    for (int i = 0; i < n; ++i) {
        offs[i] = off;
        off = align_up(off + t[i].nbytes, CQ_CACT_ALIGN);
    }
    std::vector<uint8_t> b(off, 0);
    put_u32(b, 0, CQ_CACT_TAG);
    put_u32(b, 4, CQ_CACT_VERSION);
    put_u32(b, 8, CQ_CACT_HEADER_BYTES);
    put_u32(b, 12, (uint32_t)n);
    put_u32(b, 16, CQ_CACT_CODEBOOK_LEN);
    put_u32(b, 20, default_group);
    std::memcpy(b.data() + CQ_CACT_HEADER_BYTES, codebook, 4 * CQ_CACT_CODEBOOK_LEN);
    for (int i = 0; i < n; ++i) {
        size_t r = dir_off + (size_t)i * CQ_CACT_RECORD_BYTES;
        b[r] = t[i].dtype;
        b[r + 1] = t[i].ndim;
        put_u16(b, r + 2, 0);
        for (int k = 0; k < 4; ++k) put_u32(b, r + 4 + 4 * k, t[i].shape[k]);
        put_u64(b, r + 20, offs[i]);
        put_u64(b, r + 28, t[i].nbytes);
        put_u32(b, r + 36, t[i].group);
        put_u32(b, r + 40, t[i].bits);
        if (t[i].nbytes) std::memcpy(b.data() + offs[i], t[i].data, t[i].nbytes);
    }
    std::string tmp = std::string(path) + ".tmp";
    FILE *f = std::fopen(tmp.c_str(), "wb");
    if (!f) return set_error(CQ_ERR_IO, "cannot open %s: %s", tmp.c_str(), std::strerror(errno));
    size_t wr = std::fwrite(b.data(), 1, b.size(), f);
    int cl = std::fclose(f);
    if (wr != b.size() || cl != 0) {
        std::remove(tmp.c_str());
        return set_error(CQ_ERR_IO, "short write to %s", tmp.c_str());
    }
    if (std::rename(tmp.c_str(), path) != 0) {
        std::remove(tmp.c_str());
        return set_error(CQ_ERR_IO, "cannot rename to %s: %s", path, std::strerror(errno));
    }
    return CQ_OK;
}

static int parse(cq_cact *h) {
    const uint8_t *b = h->bytes.data();
    const uint64_t size = h->bytes.size();
    if (size < 4) return set_error(CQ_ERR_FORMAT, "file shorter than its tag");
    const uint32_t tag = get_u32(b);
    if (tag == 0x05E12A83u || tag == 0x05E12A84u)
        return set_error(CQ_ERR_FORMAT,
                         "this is a Needle %s .cact archive (tag 0x%08X); this reader takes the "
                         "CQGB layout (tag 0x%08X) only",
                         tag == 0x05E12A83u ? "2" : "3", tag, CQ_CACT_TAG);
    if (tag != CQ_CACT_TAG) return set_error(CQ_ERR_FORMAT, "unknown tag 0x%08X", tag);
    if (size < CQ_CACT_HEADER_BYTES) return set_error(CQ_ERR_FORMAT, "truncated header");
    if (get_u32(b + 4) != CQ_CACT_VERSION)
        return set_error(CQ_ERR_FORMAT, "unsupported version %u", get_u32(b + 4));
    if (get_u32(b + 8) != CQ_CACT_HEADER_BYTES) return set_error(CQ_ERR_FORMAT, "bad header size");
    const uint32_t n = get_u32(b + 12);
    if (get_u32(b + 16) != CQ_CACT_CODEBOOK_LEN) return set_error(CQ_ERR_FORMAT, "bad codebook length");
    h->group = get_u32(b + 20);
    for (int i = 6; i < 16; ++i)
        if (get_u32(b + 4 * i) != 0) return set_error(CQ_ERR_FORMAT, "reserved header field %d is not 0", i);
    const uint64_t dir_off = CQ_CACT_HEADER_BYTES + 4ull * CQ_CACT_CODEBOOK_LEN;
    if ((uint64_t)n > (size - std::min<uint64_t>(size, dir_off)) / CQ_CACT_RECORD_BYTES)
        return set_error(CQ_ERR_FORMAT, "directory of %u records does not fit in %llu bytes", n,
                         (unsigned long long)size);
    std::memcpy(h->codebook, b + CQ_CACT_HEADER_BYTES, sizeof(h->codebook));
    for (int j = 0; j < 28; ++j)
        if (!std::isfinite(h->codebook[j])) return set_error(CQ_ERR_FORMAT, "codebook entry %d not finite", j);
    const uint64_t data_start = dir_off + (uint64_t)n * CQ_CACT_RECORD_BYTES;
    h->t.resize(n);
    for (uint32_t i = 0; i < n; ++i) {
        const uint8_t *r = b + dir_off + (uint64_t)i * CQ_CACT_RECORD_BYTES;
        cq_tensor_desc d;
        d.dtype = r[0];
        d.ndim = r[1];
        if (r[2] || r[3]) return set_error(CQ_ERR_FORMAT, "record %u: padding not zero", i);
        for (int k = 0; k < 4; ++k) d.shape[k] = get_u32(r + 4 + 4 * k);
        const uint64_t offset = get_u64(r + 20);
        d.nbytes = get_u64(r + 28);
        d.group = get_u32(r + 36);
        d.bits = get_u32(r + 40);
        if (offset % CQ_CACT_ALIGN) return set_error(CQ_ERR_FORMAT, "record %u: offset not 64-byte aligned", i);
        if (offset < data_start) return set_error(CQ_ERR_FORMAT, "record %u: blob overlaps the directory", i);
        if (offset > size || d.nbytes > size - offset)
            return set_error(CQ_ERR_FORMAT, "record %u: blob [%llu, +%llu) outside the %llu-byte file", i,
                             (unsigned long long)offset, (unsigned long long)d.nbytes,
                             (unsigned long long)size);
        const char *p = record_problem(d);
        if (p) return set_error(CQ_ERR_FORMAT, "record %u: %s", i, p);
        d.data = b + offset;
        h->t[i] = d;
    }
    h->n = n;
    return CQ_OK;
}

int cq_cact_open_memory(const void *bytes, uint64_t size, cq_cact **out) {
    clear_error();
    if (!out || (!bytes && size)) return set_error(CQ_ERR_ARG, "null argument");
    *out = nullptr;
    cq_cact *h = new (std::nothrow) cq_cact;
    if (!h) return set_error(CQ_ERR_NOMEM, "out of host memory");
    try {
        h->bytes.assign((const uint8_t *)bytes, (const uint8_t *)bytes + size);
    } catch (...) {
        delete h;
        return set_error(CQ_ERR_NOMEM, "out of host memory");
    }
    int st = parse(h);
    if (st) {
        delete h;
        return st;
    }
    *out = h;
    return CQ_OK;
}

int cq_cact_open(const char *path, cq_cact **out) {
    clear_error();
    if (!path || !out) return set_error(CQ_ERR_ARG, "null argument");
    *out = nullptr;
    FILE *f = std::fopen(path, "rb");
    if (!f) return set_error(CQ_ERR_IO, "cannot open %s: %s", path, std::strerror(errno));
    std::vector<uint8_t> buf;
    uint8_t chunk[1 << 16];
    size_t r;
    while ((r = std::fread(chunk, 1, sizeof(chunk), f)) > 0) buf.insert(buf.end(), chunk, chunk + r);
    bool err = std::ferror(f);
    std::fclose(f);
    if (err) return set_error(CQ_ERR_IO, "read error on %s", path);
    cq_cact *h = new (std::nothrow) cq_cact;
    if (!h) return set_error(CQ_ERR_NOMEM, "out of host memory");
    h->bytes.swap(buf);
    int st = parse(h);
    if (st) {
        delete h;
        return st;
    }
    *out = h;
    return CQ_OK;
}

int cq_cact_count(const cq_cact *h) { return h ? (int)h->n : -1; }

int cq_cact_codebook(const cq_cact *h, float out[28]) {
    clear_error();
    if (!h || !out) return set_error(CQ_ERR_ARG, "null argument");
    std::memcpy(out, h->codebook, sizeof(h->codebook));
    return CQ_OK;
}

uint32_t cq_cact_default_group(const cq_cact *h) { return h ? h->group : 0; }

int cq_cact_tensor(const cq_cact *h, int i, cq_tensor_desc *d) {
    clear_error();
    if (!h || !d) return set_error(CQ_ERR_ARG, "null argument");
    if (i < 0 || (uint32_t)i >= h->n) return set_error(CQ_ERR_ARG, "tensor index %d out of range", i);
    *d = h->t[i];
    return CQ_OK;
}

void cq_cact_close(cq_cact *h) { delete h; }

}  // extern "C"
