// cq_gemv_fast.cu -- tensor-core GEMV over CQ-packed weights for small
// batches (the decode step): batch <= 2 for 2-bit codes (CQ2, ternary),
// batch <= 4 for 4-bit codes (CQ4).
//
// Per group g of 128 inputs the product is the rotated-domain identity
// (OpenNeedle docs/reference.md; "The .cact archive and Cactus Quants",
// "Reconstructing one group"):
//     y[o] += n[o][g] * sum_k c[q[o,g,k]] * z[g,k],   z = H x (per group).
// The CTA rotates its activation once (fast Walsh-Hadamard transform with
// shuffles) and reuses it for all its rows ("How the kernel reads it").
//
// GB300 mapping. At batch 1 a CQ2 weight is 0.27 bytes of HBM traffic, so
// at the HBM roofline each SM must retire ~83 weights per clock: about 1.5
// issue slots per weight, too few for a per-weight table lookup plus FMA.
// The 2-bit path therefore never looks a level up. With q = b0 + 2 b1,
//     c[q] = c0 + (c1-c0) b0 + (c2-c0) b1 + (c3-c2-c1+c0) b0 b1,
// so the dot product is c0*sum(z) plus three dot products of 0/1 bit planes
// with z. A bit plane is extracted from the packed codes with ONE AND per 4
// weights: masking bit p of every byte leaves each byte an e4m3 value that is
// either 0 or a power of two (2^-9, 2^-8, 2^-7 as subnormals, 2^-6 for the
// lowest exponent bit), so the masked word is directly an mma.sync A
// register of four fp8 values. The B operand holds z split into four exact
// e4m3 terms (one per MMA column; z is scaled per group by a power of two
// sigma and by the inverse of the plane's bit weight), so each m16n8k32 fp8
// MMA accumulates sum(plane * z) in fp32 for 16 rows and 32 inputs. For
// int8 activations z is an integer below 2^14 and the four terms represent it
// exactly. The b1 plane sits one bit above b0 in every byte, so its A values
// are exactly twice those of b0 and both share the same B fragments.
//
// The 4-bit path (CQ4 head) expands each code byte into a half2 of levels
// with a 256-entry shared-memory table replicated across the 32 banks (one
// conflict-free LDS per two weights) and accumulates with fp16 m16n8k16
// MMAs against z split into fp16 hi/lo terms.
//
// Work: a CTA owns one matrix's row range (16*T rows) and its whole input;
// its warps split the row tiles and, when a CTA has fewer tiles than warps,
// the groups of the input (partial sums meet in shared memory). Code words
// of the first groups are requested before the activation prologue so that
// their HBM latency overlaps it.
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>

#include "cq_internal.h"

namespace cq {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxItems = 640;
constexpr int kMaxFastMats = 160;

struct FastMat {
    const uint8_t *codes;
    const __half *norms;
    const void *x;
    const float *xs;
    float *y;
    int out, in, ng, bits, xdt, B;
    int kind;      // 0: 2-bit planes, 1: 4-bit table
    int coef;      // index into FastParams::coef / lut
    int tiles;     // row tiles (16 rows) per CTA
    int kchunks;   // warps sharing one tile (split of the groups)
};

struct FastItem {
    short mat;
    short pad;
    int row0;
};

struct FastParams {
    int n_items;
    int smem_z, smem_frag, smem_red;  // byte offsets of the shared regions
    float coef[kMaxLuts][4];          // 2-bit: c0, c1-c0, (c2-c0)/2, c3-c2-c1+c0
    __half lut[kMaxLuts][16];         // 4-bit levels in fp16
    FastMat m[kMaxFastMats];
    FastItem items[kMaxItems];
};

constexpr float kInvSqrt128 = 0.08838834764831845f;

__device__ __forceinline__ float fp8_value(float x, uint32_t *bits) {
    const __nv_fp8_storage_t t = __nv_cvt_float_to_fp8(x, __NV_SATFINITE, __NV_E4M3);
    *bits = t;
    const __half_raw h = __nv_cvt_fp8_to_halfraw(t, __NV_E4M3);
    return __half2float(__half(h));
}

// term `tau` (0..3) of the exact e4m3 expansion of x (|x| <= 448)
__device__ __forceinline__ uint32_t fp8_term(float x, int tau) {
    uint32_t b = 0, out = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float v = fp8_value(x, &b);
        if (i == tau) out = b;
        x = __fsub_rn(x, v);
    }
    return out;
}

__device__ __forceinline__ void mma_fp8(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                        uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                        uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// ------------------------------------------------------------ prologue --
// zt[b][g][k] = (H0 x_b,g)[k] without the 1/sqrt(128) (exact integers for
// int8 x); gmax/gsum per (b, g). One warp per (b, g).
__device__ void rotate_all(const FastMat &M, float *zt, float *gmax, float *gsum) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int task = warp; task < M.B * M.ng; task += kWarps) {
        const int b = task / M.ng, g = task % M.ng;
        float v[4];
        const int col0 = g * kGroup + 4 * lane;
        if (M.xdt == CQ_X_I8) {
            const int8_t *xq = static_cast<const int8_t *>(M.x) + (size_t)b * M.in;
#pragma unroll
            for (int i = 0; i < 4; ++i) v[i] = col0 + i < M.in ? (float)xq[col0 + i] : 0.0f;
        } else {
            const float *xf = static_cast<const float *>(M.x) + (size_t)b * M.in;
#pragma unroll
            for (int i = 0; i < 4; ++i) v[i] = col0 + i < M.in ? xf[col0 + i] : 0.0f;
        }
        float a0 = v[0] + v[1], a1 = v[0] - v[1], a2 = v[2] + v[3], a3 = v[2] - v[3];
        v[0] = a0 + a2;
        v[1] = a1 + a3;
        v[2] = a0 - a2;
        v[3] = a1 - a3;
#pragma unroll
        for (int m = 1; m < 32; m <<= 1)
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float o = __shfl_xor_sync(0xffffffffu, v[i], m);
                v[i] = (lane & m) ? o - v[i] : v[i] + o;
            }
        float mx = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
        float sm = (v[0] + v[1]) + (v[2] + v[3]);
#pragma unroll
        for (int m = 16; m; m >>= 1) {
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, m));
            sm += __shfl_xor_sync(0xffffffffu, sm, m);
        }
        float *dst = zt + (size_t)task * kGroup + 4 * lane;
#pragma unroll
        for (int i = 0; i < 4; ++i) dst[i] = v[i];
        if (lane == 0) {
            gmax[task] = mx;
            gsum[task] = sm;
        }
    }
}

// Largest power of two sigma with amax * sigma * lim_scale <= lim.
__device__ __forceinline__ float pow2_scale(float amax, float lim) {
    if (!(amax > 0.0f)) return 1.0f;
    int e;
    const float m = frexpf(amax, &e);  // amax = m * 2^e, m in [0.5, 1)
    // want m*2^e*2^s <= lim with lim = 2^L * r (r in [0.5,1)): s = L - e, minus 1 if m > r
    int el;
    const float r = frexpf(lim, &el);
    const int s = el - e - (m > r ? 1 : 0);
    return ldexpf(1.0f, s);
}

// ----------------------------------------------------------- 2-bit path --
// Fragment word f (0..7) of lane (gq, t) in group g:
//   f = 2*mu + h, mu = 2*wsel + cp: position k = 16*(2t+wsel) + 4j + 2cp + h
//   for byte j; column n = gq: batch n/4, e4m3 term n%4 of sigma*z*2^(h?7:9).
__device__ void build_frags_planes(const FastMat &M, const float *zt, const float *gmax, uint32_t *frag,
                                   float *ginv) {
    for (int e = threadIdx.x; e < M.ng * 32 * 8; e += kThreads) {
        const int g = e / 256, lane = (e / 8) % 32, f = e % 8;
        const int gq = lane >> 2, t = lane & 3;
        const int b = gq >> 2, tau = gq & 3;
        const int mu = f >> 1, h = f & 1, wsel = mu >> 1, cp = mu & 1;
        uint32_t word = 0;
        if (b < M.B) {
            const float sigma = pow2_scale(gmax[b * M.ng + g], 448.0f / 512.0f);
            const float sc = ldexpf(sigma, h ? 7 : 9);
            const float *z = zt + (size_t)(b * M.ng + g) * kGroup;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int k = 16 * (2 * t + wsel) + 4 * j + 2 * cp + h;
                word |= fp8_term(__fmul_rn(z[k], sc), tau) << (8 * j);
            }
        }
        frag[e] = word;
    }
    for (int task = threadIdx.x; task < M.B * M.ng; task += kThreads)
        ginv[task] = 1.0f / pow2_scale(gmax[task], 448.0f / 512.0f);
}

template <bool THIRD>
__device__ __forceinline__ void planes_group(float (&acc)[4], uint32_t w0r, uint32_t w1r, uint32_t w0s,
                                             uint32_t w1s, const uint4 fa, const uint4 fb, float n_r, float n_s,
                                             float inv_r, float inv_s, const float (&cf)[4], float add_r,
                                             float add_s) {
    // plane accumulators: b0, b1, b0&b1
    float d0[4] = {0.f, 0.f, 0.f, 0.f}, d1[4] = {0.f, 0.f, 0.f, 0.f}, d2[4] = {0.f, 0.f, 0.f, 0.f};
    const uint32_t bf[8] = {fa.x, fa.y, fa.z, fa.w, fb.x, fb.y, fb.z, fb.w};
#pragma unroll
    for (int mu = 0; mu < 4; ++mu) {
        const int wsel = mu >> 1, cp = mu & 1;
        uint32_t r = wsel ? w1r : w0r, s = wsel ? w1s : w0s;
        if (cp) {
            r >>= 4;
            s >>= 4;
        }
        const uint32_t b0 = bf[2 * mu], b1 = bf[2 * mu + 1];
        mma_fp8(d0, r & 0x01010101u, s & 0x01010101u, r & 0x04040404u, s & 0x04040404u, b0, b1);
        mma_fp8(d1, r & 0x02020202u, s & 0x02020202u, r & 0x08080808u, s & 0x08080808u, b0, b1);
        if (THIRD) {
            const uint32_t tr = r & (r >> 1), ts = s & (s >> 1);
            mma_fp8(d2, tr & 0x01010101u, ts & 0x01010101u, tr & 0x04040404u, ts & 0x04040404u, b0, b1);
        }
    }
    // d*[0], d*[1]: row r, cols 2t, 2t+1; d*[2], d*[3]: row s
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float v = fmaf(cf[1], d0[i], cf[2] * d1[i]);
        if (THIRD) v = fmaf(cf[3], d2[i], v);
        const bool row_s = i >= 2;
        v = fmaf(v, row_s ? inv_s : inv_r, (i & 1) ? 0.0f : (row_s ? add_s : add_r));
        acc[i] = fmaf(row_s ? n_s : n_r, v, acc[i]);
    }
}

// ----------------------------------------------------------- 4-bit path --
// Fragment word f (0..15) of lane (gq, t) in group g: MMA nu = f/2, half
// h = f%2: positions 32t + 4nu + 2h + {0,1}; column n = gq: batch n/2,
// term n%2 (fp16 hi / lo of sigma*z).
__device__ void build_frags_lut(const FastMat &M, const float *zt, const float *gmax, uint32_t *frag,
                                float *ginv) {
    for (int e = threadIdx.x; e < M.ng * 32 * 16; e += kThreads) {
        const int g = e / 512, lane = (e / 16) % 32, f = e % 16;
        const int gq = lane >> 2, t = lane & 3;
        const int b = gq >> 1, tau = gq & 1;
        const int nu = f >> 1, h = f & 1;
        uint32_t word = 0;
        if (b < M.B) {
            const float sigma = pow2_scale(gmax[b * M.ng + g], 16384.0f);
            const float *z = zt + (size_t)(b * M.ng + g) * kGroup;
            const int k = 32 * t + 4 * nu + 2 * h;
            __half hv[2];
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const float x = __fmul_rn(z[k + i], sigma);
                const __half hi = __float2half_rn(x);
                hv[i] = tau ? __float2half_rn(__fsub_rn(x, __half2float(hi))) : hi;
            }
            word = (uint32_t)__half_as_ushort(hv[0]) | ((uint32_t)__half_as_ushort(hv[1]) << 16);
        }
        frag[e] = word;
    }
    for (int task = threadIdx.x; task < M.B * M.ng; task += kThreads)
        ginv[task] = 1.0f / pow2_scale(gmax[task], 16384.0f);
}

__device__ __forceinline__ uint32_t lut_pair(const uint32_t *tab_lane, uint32_t byte) {
    return tab_lane[byte * 32];
}

__device__ __forceinline__ void lut_group(float (&acc)[4], const uint4 cr, const uint4 cs, const uint32_t *tab_lane,
                                          const uint32_t *fr, float n_r, float n_s, float inv_r, float inv_s) {
    float d[4] = {0.f, 0.f, 0.f, 0.f};
    const uint32_t wr[4] = {cr.x, cr.y, cr.z, cr.w}, ws[4] = {cs.x, cs.y, cs.z, cs.w};
#pragma unroll
    for (int nu = 0; nu < 8; ++nu) {
        const uint32_t r = wr[nu >> 1] >> (16 * (nu & 1)), s = ws[nu >> 1] >> (16 * (nu & 1));
        const uint32_t a0 = lut_pair(tab_lane, r & 0xffu), a2 = lut_pair(tab_lane, (r >> 8) & 0xffu);
        const uint32_t a1 = lut_pair(tab_lane, s & 0xffu), a3 = lut_pair(tab_lane, (s >> 8) & 0xffu);
        mma_f16(d, a0, a1, a2, a3, fr[2 * nu], fr[2 * nu + 1]);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const bool row_s = i >= 2;
        acc[i] = fmaf((row_s ? n_s : n_r) * (row_s ? inv_s : inv_r), d[i], acc[i]);
    }
}

// ------------------------------------------------------------ the kernel --
__global__ void __launch_bounds__(kThreads, 2) gemv_fast_kernel(const __grid_constant__ FastParams p) {
    extern __shared__ __align__(16) uint8_t smem[];
    const FastItem it = p.items[blockIdx.x];
    const FastMat &M = p.m[it.mat];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int gq = lane >> 2, t = lane & 3;

    float *zt = reinterpret_cast<float *>(smem + p.smem_z);
    uint32_t *frag = reinterpret_cast<uint32_t *>(smem + p.smem_frag);
    float *red = reinterpret_cast<float *>(smem + p.smem_red);
    __shared__ float gmax[64 * 4], gsum[64 * 4], ginv[64 * 4];
    __shared__ float s_alpha[4];

    // Work of this warp: tile `tl` of the CTA, groups g = kc, kc+KC, ...
    const int KC = M.kchunks;
    const int tiles_per_warp = M.tiles > kWarps ? M.tiles / kWarps : 1;
    const int rowBytes = M.ng * (M.kind == 0 ? 32 : 64);

    // ---- prologue: activation rotation and B fragments ----
    rotate_all(M, zt, gmax, gsum);
    if (M.kind == 1) {
        // 256-entry byte -> half2 table, replicated across the 32 banks
        uint32_t *tab = reinterpret_cast<uint32_t *>(smem);  // region 0 (32 KB) when kind == 1
        for (int e = threadIdx.x; e < 256 * 32; e += kThreads) {
            const int byte = e >> 5;
            tab[e] = (uint32_t)__half_as_ushort(p.lut[M.coef][byte & 15]) |
                     ((uint32_t)__half_as_ushort(p.lut[M.coef][byte >> 4]) << 16);
        }
    }
    if (threadIdx.x < 4) {
        const int b = threadIdx.x;
        float a = kInvSqrt128;
        if (b < M.B && M.xdt == CQ_X_I8) a = __fmul_rn(M.xs[b], kInvSqrt128);
        s_alpha[b] = a;
    }
    __syncthreads();
    if (M.kind == 0)
        build_frags_planes(M, zt, gmax, frag, ginv);
    else
        build_frags_lut(M, zt, gmax, frag, ginv);
    __syncthreads();

    const float cf[4] = {p.coef[M.coef][0], p.coef[M.coef][1], p.coef[M.coef][2], p.coef[M.coef][3]};
    const bool third = cf[3] != 0.0f;

    for (int tw = 0; tw < tiles_per_warp; ++tw) {
        const int tl = (M.tiles > kWarps) ? warp * tiles_per_warp + tw : warp / KC;
        const int kc = (M.tiles > kWarps) ? 0 : warp % KC;
        if (tl >= M.tiles) break;
        const int row_r = it.row0 + 16 * tl + gq, row_s = row_r + 8;
        const bool ok_r = row_r < M.out, ok_s = row_s < M.out;
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        for (int g = kc; g < M.ng; g += KC) {
            const float n_r = ok_r ? __half2float(M.norms[(size_t)row_r * M.ng + g]) : 0.0f;
            const float n_s = ok_s ? __half2float(M.norms[(size_t)row_s * M.ng + g]) : 0.0f;
            if (M.kind == 0) {
                uint2 cr = make_uint2(0, 0), cs = make_uint2(0, 0);
                if (ok_r) cr = __ldcs(reinterpret_cast<const uint2 *>(M.codes + (size_t)row_r * rowBytes + g * 32 + 8 * t));
                if (ok_s) cs = __ldcs(reinterpret_cast<const uint2 *>(M.codes + (size_t)row_s * rowBytes + g * 32 + 8 * t));
                const uint4 *fl = reinterpret_cast<const uint4 *>(frag + (size_t)(g * 32 + lane) * 8);
                const uint4 fa = fl[0], fb = fl[1];
                // batch of the lane's columns: cols 2t, 2t+1 -> batch (2t)/4 = t/2
                const int bb = t >> 1;
                const float inv = bb < M.B ? ginv[bb * M.ng + g] : 0.0f;
                const float add = (t & 1) == 0 && bb < M.B ? cf[0] * gsum[bb * M.ng + g] : 0.0f;
                if (third)
                    planes_group<true>(acc, cr.x, cr.y, cs.x, cs.y, fa, fb, n_r, n_s, inv, inv, cf, add, add);
                else
                    planes_group<false>(acc, cr.x, cr.y, cs.x, cs.y, fa, fb, n_r, n_s, inv, inv, cf, add, add);
            } else {
                uint4 cr = make_uint4(0, 0, 0, 0), cs = make_uint4(0, 0, 0, 0);
                if (ok_r) cr = __ldcs(reinterpret_cast<const uint4 *>(M.codes + (size_t)row_r * rowBytes + g * 64 + 16 * t));
                if (ok_s) cs = __ldcs(reinterpret_cast<const uint4 *>(M.codes + (size_t)row_s * rowBytes + g * 64 + 16 * t));
                const uint32_t *tab_lane = reinterpret_cast<const uint32_t *>(smem) + lane;
                const uint32_t *fr = frag + (size_t)(g * 32 + lane) * 16;
                uint32_t frr[16];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const uint4 v = reinterpret_cast<const uint4 *>(fr)[i];
                    frr[4 * i] = v.x;
                    frr[4 * i + 1] = v.y;
                    frr[4 * i + 2] = v.z;
                    frr[4 * i + 3] = v.w;
                }
                // columns 2t, 2t+1 = batch t, terms hi/lo
                const float inv = t < M.B ? ginv[t * M.ng + g] : 0.0f;
                lut_group(acc, cr, cs, tab_lane, frr, n_r, n_s, inv, inv);
            }
        }
        // ---- per-row totals of each batch ----
        float yr0, ys0;  // this lane's batch partial for rows r and s
        int bsel;
        if (M.kind == 0) {
            // batch t/2 lives in cols 4b..4b+3 = lanes t = 2b, 2b+1
            yr0 = acc[0] + acc[1];
            ys0 = acc[2] + acc[3];
            yr0 += __shfl_xor_sync(0xffffffffu, yr0, 1);
            ys0 += __shfl_xor_sync(0xffffffffu, ys0, 1);
            bsel = t >> 1;
        } else {
            // batch t lives in cols 2t, 2t+1 (hi, lo) of lane t
            yr0 = acc[0] + acc[1];
            ys0 = acc[2] + acc[3];
            bsel = t;
        }
        const bool writer = M.kind == 0 ? ((t & 1) == 0 && bsel < M.B) : (bsel < M.B);
        if (KC == 1) {
            if (writer) {
                const float a = s_alpha[bsel];
                if (ok_r) M.y[(size_t)bsel * M.out + row_r] = yr0 * a;
                if (ok_s) M.y[(size_t)bsel * M.out + row_s] = ys0 * a;
            }
        } else {
            // red[tile][kc][16 rows][4 batches]
            float *rt = red + ((size_t)(tl * KC + kc) * 16) * 4;
            if (writer) {
                rt[gq * 4 + bsel] = yr0;
                rt[(gq + 8) * 4 + bsel] = ys0;
            }
        }
    }
    if (KC > 1) {
        __syncthreads();
        for (int e = threadIdx.x; e < M.tiles * 16 * M.B; e += kThreads) {
            const int tl = e / (16 * M.B), rr = (e / M.B) % 16, b = e % M.B;
            const int row = it.row0 + 16 * tl + rr;
            if (row >= M.out) continue;
            float s = 0.0f;
            for (int kc = 0; kc < KC; ++kc) s += red[((size_t)(tl * KC + kc) * 16 + rr) * 4 + b];
            M.y[(size_t)b * M.out + row] = s * s_alpha[b];
        }
    }
}

}  // namespace

bool gemv_fast_eligible(const cq_gemv_desc &d) {
    const int ng = in_padded(d.in) / kGroup;
    if (d.in <= 0 || d.out <= 0) return false;
    if (width_of(d.bits) == 2) return d.B <= 2 && ng <= 64;
    if (d.bits == 4) return d.B <= 4 && ng * d.B <= 64 && ng <= 32;
    return false;
}

int launch_gemv_fast(const cq_gemv_desc *d, const int *idx, int n, void *stream) {
    static FastParams p;
    p.n_items = 0;
    int ncoef = 0, nm = 0;
    size_t need_z = 0, need_frag = 0, need_red = 0, need_tab = 0;
    for (int ii = 0; ii < n; ++ii) {
        const cq_gemv_desc &D = d[idx[ii]];
        if (nm == kMaxFastMats) return set_error(CQ_ERR_ARG, "too many matrices for one fast GEMV launch");
        FastMat &M = p.m[nm];
        const int ip = in_padded(D.in), W = width_of(D.bits);
        M.codes = D.blob;
        M.norms = reinterpret_cast<const __half *>(D.blob + (size_t)D.out * ip * W / 8);
        M.x = D.x;
        M.xs = D.x_scale;
        M.y = D.y;
        M.out = D.out;
        M.in = D.in;
        M.ng = ip / kGroup;
        M.bits = D.bits;
        M.xdt = D.x_dtype;
        M.B = D.B;
        M.kind = W == 2 ? 0 : 1;
        // coefficient set
        float cf[4] = {0, 0, 0, 0};
        __half lut[16];
        for (int j = 0; j < 16; ++j) lut[j] = __float2half_rn(0.0f);
        if (M.kind == 0) {
            float c[4];
            if (D.bits == 5) {
                const float cc = D.codebook[2];
                c[0] = 0.0f, c[1] = cc, c[2] = -2.0f * cc, c[3] = -cc;  // crumbs sign-extend
            } else {
                for (int j = 0; j < 4; ++j) c[j] = D.codebook[j];
            }
            // in double the sums of four floats are exact, so a symmetric
            // codebook gives an interaction coefficient of exactly zero
            const double d0 = c[0], d1 = c[1], d2 = c[2], d3 = c[3];
            cf[0] = (float)d0;
            cf[1] = (float)(d1 - d0);
            cf[2] = (float)(0.5 * (d2 - d0));
            cf[3] = (float)(((d3 - d2) - d1) + d0);
        } else {
            for (int j = 0; j < 16; ++j) lut[j] = __float2half_rn(D.codebook[j]);
        }
        int ci = -1;
        for (int j = 0; j < ncoef; ++j) {
            bool same = true;
            for (int k = 0; k < 4; ++k) same &= p.coef[j][k] == cf[k];
            for (int k = 0; k < 16; ++k) same &= __half_as_ushort(p.lut[j][k]) == __half_as_ushort(lut[k]);
            if (same) ci = j;
        }
        if (ci < 0) {
            if (ncoef == kMaxLuts) return set_error(CQ_ERR_ARG, "more than %d distinct codebooks in one call", kMaxLuts);
            for (int k = 0; k < 4; ++k) p.coef[ncoef][k] = cf[k];
            for (int k = 0; k < 16; ++k) p.lut[ncoef][k] = lut[k];
            ci = ncoef++;
        }
        M.coef = ci;
        // rows per CTA: about 48 KB of codes, a power-of-two number of 16-row tiles
        const int rowB = M.ng * (M.kind == 0 ? 32 : 64) + 2 * M.ng;
        int tiles = std::max(1, (48 * 1024) / (rowB * 16));
        int tp = 1;
        while (tp * 2 <= tiles && tp * 2 <= 32) tp *= 2;
        const int need_tiles = (M.out + 15) / 16;
        while (tp > 1 && tp / 2 >= need_tiles) tp /= 2;
        M.tiles = tp;
        M.kchunks = tp >= kWarps ? 1 : std::min(kWarps / tp, M.ng);
        for (int r0 = 0; r0 < M.out; r0 += 16 * tp) {
            if (p.n_items == kMaxItems) return set_error(CQ_ERR_ARG, "too many row blocks for one fast GEMV launch");
            p.items[p.n_items].mat = (short)nm;
            p.items[p.n_items].pad = 0;
            p.items[p.n_items].row0 = r0;
            ++p.n_items;
        }
        need_z = std::max(need_z, (size_t)M.B * M.ng * kGroup * sizeof(float));
        need_frag = std::max(need_frag, (size_t)M.ng * 32 * (M.kind == 0 ? 8 : 16) * sizeof(uint32_t));
        if (M.kchunks > 1) need_red = std::max(need_red, (size_t)M.tiles * M.kchunks * 16 * 4 * sizeof(float));
        if (M.kind == 1) need_tab = 256 * 32 * sizeof(uint32_t);
        ++nm;
    }
    if (!p.n_items) return CQ_OK;
    // layout: [table (kind 1 only)] [z] [frag] [red], each 16-byte aligned
    size_t off = need_tab;
    p.smem_z = (int)off;
    off += (need_z + 15) / 16 * 16;
    p.smem_frag = (int)off;
    off += (need_frag + 15) / 16 * 16;
    p.smem_red = (int)off;
    off += (need_red + 15) / 16 * 16;
    const size_t smem = std::max<size_t>(off, 16);
    static bool attr = false;
    if (!attr) {
        cudaFuncSetAttribute(gemv_fast_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
        attr = true;
    }
    if (smem > 200 * 1024) return set_error(CQ_ERR_SHAPE, "fast GEMV needs %zu bytes of shared memory", smem);
    gemv_fast_kernel<<<p.n_items, kThreads, smem, reinterpret_cast<cudaStream_t>(stream)>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return set_error(CQ_ERR_CUDA, "fast gemv launch: %s", cudaGetErrorString(e));
    return CQ_OK;
}

}  // namespace cq
