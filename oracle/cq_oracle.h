/*
 * cq_oracle.h -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, obviously correct CPU restatement of Cactus Quants (CQ):
 * the Hadamard-rotated codebook encoding of a weight matrix and the matrix
 * product over it. Every routine works in double precision with an explicit
 * Hadamard matrix, except where the pages fix a narrower precision (the fp32
 * group norm, its fp16 storage, and the fp32 nearest-level search).
 *
 * Only the tests, the package smoke check and the benchmark's CPU baseline
 * may load this library. The product path never links, imports or calls it.
 *
 * Sources (page title, section):
 *   [CF]  "The .cact format" (cactuscompute.com blog), "Cactus Quants",
 *         "How the kernel reads it".
 *   [NJ]  "The .cact archive and Cactus Quants" (needle.js tutorial),
 *         "Shared codebooks", "Anatomy of a CQ matrix", "2-bit", "4-bit",
 *         "3-bit", "Reconstructing one group".
 *   [ON]  OpenNeedle docs/reference.md, CQ quantisation and file-format
 *         sections (the rotate / norm / argmin / fp16 recipe, the tie rule,
 *         the codebook recipe, the rotated-domain identity, fake_quant_act).
 *
 * Parity status of each function is stated beside it; a function that has
 * no independent pin says "parity unpinned".
 */
#ifndef CQ_ORACLE_H
#define CQ_ORACLE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Normalised Sylvester Hadamard matrix, natural order:
 * H[i*n+k] = (-1)^popcount(i&k) / sqrt(n). n must be a power of two.
 * [CF] "Cactus Quants"; [ON] "Sylvester/Walsh-Hadamard". Pinned by
 * H0*H0^T = n*I in integers and by norm preservation. */
int cqo_hadamard(int n, double *H);

/* Lloyd-Max scalar quantiser for the standard normal density, iterated
 * on the exact density to a fixed point (centroid and midpoint conditions).
 * L levels, returned sorted ascending, NOT divided by sqrt(group).
 * Pinned by the closed form for L=2 (+-sqrt(2/pi)), by the ternary constant
 * printed in [NJ] "Shared codebooks" for L=3, and by direct minimisation of
 * the distortion integral. Returns iterations used, or -1 on bad input. */
int cqo_lloyd_max_normal(int L, int max_iter, double tol, double *levels);

/* Lloyd-Max on a finite sample (the official codebook recipe in [ON]):
 * centres start at the sample quantiles (j+1/2)/L (linear interpolation
 * between order statistics), then `iters` rounds of nearest-centre
 * assignment and cell means. Levels returned sorted, not scaled.
 * Pinned by the CQ2 header codebook printed in [ON]. */
int cqo_lloyd_max_samples(const double *x, long n, int L, int iters,
                          double *levels);

/* IEEE binary16 conversions, round to nearest even. Pinned against numpy. */
uint16_t cqo_f32_to_f16(float f);
float cqo_f16_to_f32(uint16_t h);

/* Number of levels and packed code width for a record `bits` value
 * (1 = binary, two levels, one bit per code; 2, 3, 4; 5 = ternary marker
 * with 3 levels in 2-bit crumbs). */
int cqo_levels(int bits);
int cqo_width(int bits);

/* Blob size per [NJ] "Anatomy of a CQ matrix":
 * out*in_pad*width/8 + out*(in_pad/group)*2. 0 on bad arguments.
 * Pinned by the Needle-2 size table in [ON]. */
uint64_t cqo_packed_bytes(int out, int in, int group, int bits);

/* Encode W[out][in] (fp32, row-major) into a CQ blob: per row and group,
 * r = w.H (explicit matrix, double), n = fp32(sqrt(sum r^2)),
 * u = r / max(n, 1e-12), q_k = argmin_j |fp32(u_k) - c_j| in fp32 with ties
 * to the smaller index, fp16 norm, LSB-first bitstream per row.
 * Ternary (bits=5): codebook = {-c, 0, +c}, crumbs 0->00, +c->01, -c->11.
 * `codebook` holds cqo_levels(bits) floats, strictly increasing, already
 * divided by sqrt(group). If `flags` is non-NULL it receives, per padded
 * coordinate [out][in_pad], 1 when the double-precision u lies within
 * `eps` of a midpoint between adjacent levels (a decision boundary).
 * Returns the number of flagged coordinates, or -1 on bad input.
 * Pinned by worked examples with closed forms and by brute force on tiny
 * groups. */
long cqo_encode(const float *W, int out, int in, int group, int bits,
                const float *codebook, uint8_t *blob, uint8_t *flags,
                double eps);

/* Read back codes [out][in_pad] (level indices; for ternary the raw 2-bit
 * crumb) and fp16 norm bits [out][in_pad/group] from a blob. */
int cqo_unpack(const uint8_t *blob, int out, int in, int group, int bits,
               int *codes, uint16_t *norms);

/* Dequantise: w_hat_g = (c[q] * fp32(n_store)) . H, cropped to `in`.
 * Ternary crumbs are sign-extended (00 -> 0, 01 -> +1, 11 -> -1, and the
 * never-written 10 -> -2) and multiplied by the positive level.
 * [NJ] "Reconstructing one group"; [ON]. Output double What[out][in]. */
int cqo_dequant(const uint8_t *blob, int out, int in, int group, int bits,
                const float *codebook, double *What);

/* Plain definition of the product: Y[t][o] = sum_k What[o][k] X[t][k] in
 * double, and Bound[t][o] = sum_k |What[o][k]| |X[t][k]| (the tolerance
 * scale). Either output may be NULL. */
void cqo_matmul(const double *What, int out, int in, const double *X, int B,
                double *Y, double *Bound);

/* Second route through the rotated-domain identity of [ON] and [NJ]:
 * Y[t][o] = sum_g n_store[o][g] * <c[q[o,g,:]], H x_g> in double, with the
 * explicit matrix. Must agree with cqo_dequant + cqo_matmul to rounding. */
int cqo_matmul_rotated(const uint8_t *blob, int out, int in, int group,
                       int bits, const float *codebook, const double *X,
                       int B, double *Y);

/* Per-token int8 activation quantisation ([ON] fake_quant_act):
 * s = absmax/127 (fp32), q = clamp(rint(x/s), -128, 127) in fp32;
 * an all-zero row gets s = 1 and q = 0. Q[B][in], S[B]. */
void cqo_act_quant_int8(const float *X, int B, int in, int8_t *Q, float *S);

#ifdef __cplusplus
}
#endif
#endif
