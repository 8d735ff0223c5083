/*
 * cq_oracle.c -- TEST INFRASTRUCTURE ONLY (see cq_oracle.h).
 *
 * Plain C99, double precision, explicit matrices, no blocking or fusion.
 * Compiled with -O2 -ffp-contract=off and without -ffast-math so that
 * every float expression below is evaluated exactly as written.
 */
#include "cq_oracle.h"

#include <float.h>
#include <math.h>
#include <stdlib.h>
#include <string.h>

#ifndef M_PI
#define M_PI 3.14159265358979323846
#endif
#ifndef M_SQRT2
#define M_SQRT2 1.41421356237309504880
#endif

static int is_pow2(int n) { return n > 0 && (n & (n - 1)) == 0; }

static int parity(unsigned v)
{
    int p = 0;
    while (v) {
        p ^= 1;
        v &= v - 1;
    }
    return p;
}

/* ---------------------------------------------------------------- H -- */

int cqo_hadamard(int n, double *H)
{
    if (!is_pow2(n) || !H)
        return -1;
    const double s = 1.0 / sqrt((double)n);
    for (int i = 0; i < n; ++i)
        for (int k = 0; k < n; ++k)
            H[(size_t)i * n + k] = parity((unsigned)(i & k)) ? -s : s;
    return 0;
}

/* ------------------------------------------------------- Lloyd-Max -- */

static double normal_pdf(double x)
{
    if (isinf(x))
        return 0.0;
    return exp(-0.5 * x * x) / sqrt(2.0 * M_PI);
}

/* Probability mass of N(0,1) on [a, b], using the tail that keeps the
 * subtraction well conditioned. */
static double normal_mass(double a, double b)
{
    if (a >= 0.0) /* both in the upper half: Q(a) - Q(b), Q = upper tail */
        return 0.5 * erfc(a / M_SQRT2) - 0.5 * erfc(b / M_SQRT2);
    if (b <= 0.0) /* both in the lower half: Q(-b) - Q(-a) */
        return 0.5 * erfc(-b / M_SQRT2) - 0.5 * erfc(-a / M_SQRT2);
    return 1.0 - 0.5 * erfc(-a / M_SQRT2) - 0.5 * erfc(b / M_SQRT2);
}

int cqo_lloyd_max_normal(int L, int max_iter, double tol, double *c)
{
    if (L < 2 || !c || max_iter < 1)
        return -1;
    /* Any increasing start converges for a log-concave density. */
    for (int j = 0; j < L; ++j)
        c[j] = -2.0 + 4.0 * (j + 0.5) / L;
    double *t = (double *)malloc(sizeof(double) * (L + 1));
    if (!t)
        return -1;
    int it;
    for (it = 1; it <= max_iter; ++it) {
        t[0] = -INFINITY;
        t[L] = INFINITY;
        for (int j = 1; j < L; ++j)
            t[j] = 0.5 * (c[j - 1] + c[j]); /* nearest-neighbour condition */
        double change = 0.0;
        for (int j = 0; j < L; ++j) {
            /* centroid condition: E[X | t_j < X < t_{j+1}] */
            double cj = (normal_pdf(t[j]) - normal_pdf(t[j + 1])) /
                        normal_mass(t[j], t[j + 1]);
            double d = fabs(cj - c[j]);
            if (d > change)
                change = d;
            c[j] = cj;
        }
        if (change < tol)
            break;
    }
    free(t);
    return it;
}

static int cmp_double(const void *a, const void *b)
{
    double x = *(const double *)a, y = *(const double *)b;
    return (x > y) - (x < y);
}

int cqo_lloyd_max_samples(const double *x, long n, int L, int iters,
                          double *c)
{
    if (!x || n < 2 || L < 2 || !c || iters < 0)
        return -1;
    double *s = (double *)malloc(sizeof(double) * (size_t)n);
    double *sum = (double *)malloc(sizeof(double) * L);
    long *cnt = (long *)malloc(sizeof(long) * L);
    double *t = (double *)malloc(sizeof(double) * (L + 1));
    if (!s || !sum || !cnt || !t) {
        free(s); free(sum); free(cnt); free(t);
        return -1;
    }
    memcpy(s, x, sizeof(double) * (size_t)n);
    qsort(s, (size_t)n, sizeof(double), cmp_double);
    /* Quantile start: probability (j+1/2)/L, linear interpolation between
     * the order statistics at position p*(n-1). */
    for (int j = 0; j < L; ++j) {
        double p = (j + 0.5) / L;
        double pos = p * (double)(n - 1);
        long lo = (long)floor(pos);
        double fr = pos - (double)lo;
        long hi = lo + 1 < n ? lo + 1 : lo;
        c[j] = s[lo] + fr * (s[hi] - s[lo]);
    }
    for (int it = 0; it < iters; ++it) {
        for (int j = 1; j < L; ++j)
            t[j] = 0.5 * (c[j - 1] + c[j]);
        for (int j = 0; j < L; ++j) {
            sum[j] = 0.0;
            cnt[j] = 0;
        }
        /* Nearest centre for each sample; with sorted centres the cell of
         * a sample is the number of midpoints it exceeds. */
        for (long i = 0; i < n; ++i) {
            int j = 0;
            while (j < L - 1 && x[i] > t[j + 1])
                ++j;
            sum[j] += x[i];
            cnt[j] += 1;
        }
        for (int j = 0; j < L; ++j)
            if (cnt[j] > 0)
                c[j] = sum[j] / (double)cnt[j];
    }
    free(s); free(sum); free(cnt); free(t);
    return 0;
}

/* ------------------------------------------------------------ fp16 -- */

uint16_t cqo_f32_to_f16(float f)
{
    uint32_t xb;
    memcpy(&xb, &f, 4);
    uint16_t sign = (uint16_t)((xb >> 16) & 0x8000u);
    uint32_t ax = xb & 0x7fffffffu;
    if (ax > 0x7f800000u) /* NaN: keep it quiet */
        return (uint16_t)(sign | 0x7e00u);
    if (ax == 0x7f800000u)
        return (uint16_t)(sign | 0x7c00u);
    double a = fabs((double)f);
    /* 65520 is halfway between 65504 (largest finite) and 2^16: ties go to
     * the even significand, which is the overflow to infinity. */
    if (a >= 65520.0)
        return (uint16_t)(sign | 0x7c00u);
    if (a < ldexp(1.0, -14)) {
        /* Subnormal: value = m * 2^-24 with integer m in [0, 1024]. */
        double m = rint(ldexp(a, 24)); /* exact scaling, round half even */
        return (uint16_t)(sign | (uint16_t)m); /* m = 1024 is 2^-14 */
    }
    int e;
    frexp(a, &e);                  /* a = f * 2^e, f in [0.5, 1) */
    double m = rint(ldexp(a, 11 - e)); /* significand in [1024, 2048] */
    int E = e - 1 + 15;
    if (m >= 2048.0) {
        m *= 0.5;
        E += 1;
    }
    if (E >= 31)
        return (uint16_t)(sign | 0x7c00u);
    return (uint16_t)(sign | (uint16_t)(E << 10) | (uint16_t)(m - 1024.0));
}

float cqo_f16_to_f32(uint16_t h)
{
    int s = (h >> 15) & 1;
    int E = (h >> 10) & 31;
    int m = h & 1023;
    double v;
    if (E == 0)
        v = ldexp((double)m, -24);
    else if (E == 31)
        v = m ? NAN : INFINITY;
    else
        v = ldexp(1024.0 + m, E - 25);
    return (float)(s ? -v : v);
}

/* ----------------------------------------------------------- format -- */

int cqo_levels(int bits)
{
    switch (bits) {
    case 1: return 2; /* binary: eight codes per byte ([CF] "Cactus Quants") */
    case 2: return 4;
    case 3: return 8;
    case 4: return 16;
    case 5: return 3;
    default: return -1;
    }
}

int cqo_width(int bits)
{
    switch (bits) {
    case 1: return 1;
    case 2: return 2;
    case 3: return 3;
    case 4: return 4;
    case 5: return 2;
    default: return -1;
    }
}

static int check_shape(int out, int in, int group, int bits)
{
    if (out < 0 || in < 0 || !is_pow2(group) || group < 8)
        return -1;
    if (cqo_levels(bits) < 0)
        return -1;
    return 0;
}

static int in_padded(int in, int group) { return (in + group - 1) / group * group; }

uint64_t cqo_packed_bytes(int out, int in, int group, int bits)
{
    if (check_shape(out, in, group, bits))
        return 0;
    uint64_t ip = (uint64_t)in_padded(in, group);
    uint64_t w = (uint64_t)cqo_width(bits);
    return (uint64_t)out * ip * w / 8 + (uint64_t)out * (ip / group) * 2;
}

static int check_codebook(const float *cb, int L)
{
    for (int j = 0; j + 1 < L; ++j)
        if (!(cb[j] < cb[j + 1]))
            return -1;
    return 0;
}

/* Bit k of the row bitstream. */
static void put_bits(uint8_t *row, long bitpos, int width, unsigned v)
{
    for (int b = 0; b < width; ++b)
        if ((v >> b) & 1u)
            row[(bitpos + b) >> 3] |= (uint8_t)(1u << ((bitpos + b) & 7));
}

static unsigned get_bits(const uint8_t *row, long bitpos, int width)
{
    unsigned v = 0;
    for (int b = 0; b < width; ++b)
        v |= (unsigned)((row[(bitpos + b) >> 3] >> ((bitpos + b) & 7)) & 1u) << b;
    return v;
}

long cqo_encode(const float *W, int out, int in, int group, int bits,
                const float *cb, uint8_t *blob, uint8_t *flags, double eps)
{
    if (check_shape(out, in, group, bits) || !cb || !blob || (out && in && !W))
        return -1;
    const int L = cqo_levels(bits), width = cqo_width(bits);
    if (check_codebook(cb, L))
        return -1;
    const int ip = in_padded(in, group), ng = ip / group;
    const size_t rowBytes = (size_t)ip * width / 8;
    uint8_t *codes = blob;
    uint8_t *normb = blob + (size_t)out * rowBytes;
    memset(codes, 0, (size_t)out * rowBytes);

    double *H = (double *)malloc(sizeof(double) * group * group);
    double *w = (double *)malloc(sizeof(double) * group);
    double *r = (double *)malloc(sizeof(double) * group);
    if (!H || !w || !r) {
        free(H); free(w); free(r);
        return -1;
    }
    cqo_hadamard(group, H);
    long nflag = 0;
    for (int o = 0; o < out; ++o) {
        uint8_t *row = codes + (size_t)o * rowBytes;
        for (int g = 0; g < ng; ++g) {
            /* zero-pad the input axis to a multiple of the group */
            for (int i = 0; i < group; ++i) {
                int col = g * group + i;
                w[i] = col < in ? (double)W[(size_t)o * in + col] : 0.0;
            }
            /* rotate: r = w . H (row vector times the explicit matrix) */
            for (int k = 0; k < group; ++k) {
                double acc = 0.0;
                for (int i = 0; i < group; ++i)
                    acc += w[i] * H[(size_t)i * group + k];
                r[k] = acc;
            }
            /* group length, held in fp32 */
            double ss = 0.0;
            for (int k = 0; k < group; ++k)
                ss += r[k] * r[k];
            float n32 = (float)sqrt(ss);
            double den = (double)n32 > 1e-12 ? (double)n32 : 1e-12;
            for (int k = 0; k < group; ++k) {
                double u = r[k] / den; /* direction, normalised by the unrounded norm */
                float u32 = (float)u;
                int best = 0;
                float bd = fabsf(u32 - cb[0]);
                for (int j = 1; j < L; ++j) {
                    float d = fabsf(u32 - cb[j]);
                    if (d < bd) { /* strict: ties keep the smaller index */
                        bd = d;
                        best = j;
                    }
                }
                int flag = 0;
                for (int j = 0; j + 1 < L; ++j) {
                    double mid = 0.5 * ((double)cb[j] + (double)cb[j + 1]);
                    if (fabs(u - mid) < eps)
                        flag = 1;
                }
                if (flags)
                    flags[(size_t)o * ip + (size_t)g * group + k] = (uint8_t)flag;
                nflag += flag;
                /* ternary: index 0,1,2 = -c,0,+c -> crumb (idx-1) mod 4 */
                unsigned code = bits == 5 ? (unsigned)((best - 1) & 3) : (unsigned)best;
                put_bits(row, (long)(g * group + k) * width, width, code);
            }
            uint16_t h = cqo_f32_to_f16(n32);
            size_t ni = (size_t)o * ng + g;
            normb[2 * ni] = (uint8_t)(h & 0xff);
            normb[2 * ni + 1] = (uint8_t)(h >> 8);
        }
    }
    free(H); free(w); free(r);
    return nflag;
}

int cqo_unpack(const uint8_t *blob, int out, int in, int group, int bits,
               int *codes, uint16_t *norms)
{
    if (check_shape(out, in, group, bits) || !blob)
        return -1;
    const int width = cqo_width(bits);
    const int ip = in_padded(in, group), ng = ip / group;
    const size_t rowBytes = (size_t)ip * width / 8;
    const uint8_t *normb = blob + (size_t)out * rowBytes;
    for (int o = 0; o < out; ++o) {
        if (codes)
            for (int k = 0; k < ip; ++k)
                codes[(size_t)o * ip + k] =
                    (int)get_bits(blob + (size_t)o * rowBytes, (long)k * width, width);
        if (norms)
            for (int g = 0; g < ng; ++g) {
                size_t ni = (size_t)o * ng + g;
                norms[ni] = (uint16_t)(normb[2 * ni] | (normb[2 * ni + 1] << 8));
            }
    }
    return 0;
}

/* Level value of one stored code. */
static double level_of(unsigned code, int bits, const float *cb)
{
    if (bits == 5) {
        int s = (code & 2u) ? (int)code - 4 : (int)code; /* 2-bit sign extension */
        return (double)s * (double)cb[2];
    }
    return (double)cb[code];
}

int cqo_dequant(const uint8_t *blob, int out, int in, int group, int bits,
                const float *cb, double *What)
{
    if (check_shape(out, in, group, bits) || !blob || !cb || !What)
        return -1;
    const int width = cqo_width(bits);
    const int ip = in_padded(in, group), ng = ip / group;
    const size_t rowBytes = (size_t)ip * width / 8;
    const uint8_t *normb = blob + (size_t)out * rowBytes;
    double *H = (double *)malloc(sizeof(double) * group * group);
    double *v = (double *)malloc(sizeof(double) * group);
    if (!H || !v) {
        free(H); free(v);
        return -1;
    }
    cqo_hadamard(group, H);
    for (int o = 0; o < out; ++o) {
        const uint8_t *row = blob + (size_t)o * rowBytes;
        for (int g = 0; g < ng; ++g) {
            size_t ni = (size_t)o * ng + g;
            uint16_t hb = (uint16_t)(normb[2 * ni] | (normb[2 * ni + 1] << 8));
            double n = (double)cqo_f16_to_f32(hb);
            for (int k = 0; k < group; ++k)
                v[k] = level_of(get_bits(row, (long)(g * group + k) * width, width),
                                bits, cb) * n;
            /* w_hat = v . H, keep only the unpadded columns */
            for (int i = 0; i < group; ++i) {
                int col = g * group + i;
                if (col >= in)
                    break;
                double acc = 0.0;
                for (int k = 0; k < group; ++k)
                    acc += v[k] * H[(size_t)k * group + i];
                What[(size_t)o * in + col] = acc;
            }
        }
    }
    free(H); free(v);
    return 0;
}

void cqo_matmul(const double *What, int out, int in, const double *X, int B,
                double *Y, double *Bound)
{
    for (int t = 0; t < B; ++t)
        for (int o = 0; o < out; ++o) {
            double acc = 0.0, bnd = 0.0;
            for (int k = 0; k < in; ++k) {
                double a = What[(size_t)o * in + k], b = X[(size_t)t * in + k];
                acc += a * b;
                bnd += fabs(a) * fabs(b);
            }
            if (Y)
                Y[(size_t)t * out + o] = acc;
            if (Bound)
                Bound[(size_t)t * out + o] = bnd;
        }
}

int cqo_matmul_rotated(const uint8_t *blob, int out, int in, int group,
                       int bits, const float *cb, const double *X, int B,
                       double *Y)
{
    if (check_shape(out, in, group, bits) || !blob || !cb || !X || !Y)
        return -1;
    const int width = cqo_width(bits);
    const int ip = in_padded(in, group), ng = ip / group;
    const size_t rowBytes = (size_t)ip * width / 8;
    const uint8_t *normb = blob + (size_t)out * rowBytes;
    double *H = (double *)malloc(sizeof(double) * group * group);
    double *z = (double *)malloc(sizeof(double) * (size_t)B * ip);
    if (!H || !z) {
        free(H); free(z);
        return -1;
    }
    cqo_hadamard(group, H);
    /* z_g = H . x_g for every token and group (x zero-padded) */
    for (int t = 0; t < B; ++t)
        for (int g = 0; g < ng; ++g)
            for (int k = 0; k < group; ++k) {
                double acc = 0.0;
                for (int i = 0; i < group; ++i) {
                    int col = g * group + i;
                    double xv = col < in ? X[(size_t)t * in + col] : 0.0;
                    acc += H[(size_t)k * group + i] * xv;
                }
                z[(size_t)t * ip + (size_t)g * group + k] = acc;
            }
    for (int t = 0; t < B; ++t)
        for (int o = 0; o < out; ++o) {
            const uint8_t *row = blob + (size_t)o * rowBytes;
            double y = 0.0;
            for (int g = 0; g < ng; ++g) {
                size_t ni = (size_t)o * ng + g;
                uint16_t hb = (uint16_t)(normb[2 * ni] | (normb[2 * ni + 1] << 8));
                double d = 0.0;
                for (int k = 0; k < group; ++k)
                    d += level_of(get_bits(row, (long)(g * group + k) * width, width),
                                  bits, cb) *
                         z[(size_t)t * ip + (size_t)g * group + k];
                y += (double)cqo_f16_to_f32(hb) * d;
            }
            Y[(size_t)t * out + o] = y;
        }
    free(H); free(z);
    return 0;
}

void cqo_act_quant_int8(const float *X, int B, int in, int8_t *Q, float *S)
{
    for (int t = 0; t < B; ++t) {
        const float *x = X + (size_t)t * in;
        float amax = 0.0f;
        for (int k = 0; k < in; ++k) {
            float a = fabsf(x[k]);
            if (a > amax)
                amax = a;
        }
        float s = amax > 0.0f ? amax / 127.0f : 1.0f;
        S[t] = s;
        for (int k = 0; k < in; ++k) {
            float v = rintf(x[k] / s);
            if (v > 127.0f)
                v = 127.0f;
            if (v < -128.0f)
                v = -128.0f;
            Q[(size_t)t * in + k] = (int8_t)v;
        }
    }
}
