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
// Work: a CTA owns one matrix's row range (16*T rows) and its whole input.
// At entry it issues 16-byte cp.async copies of its contiguous code rows and
// norms into shared memory (rows padded so the MMA operand reads are free of
// bank conflicts; rows past the matrix are zero-filled), computes the
// activation prologue while they land, then its warps split the row tiles
// and, when a CTA has fewer tiles than warps, the groups of the input
// (partial sums meet in shared memory).
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
constexpr int kMaxFastMats = 200;
constexpr int kMaxFastItems = 2048;

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
    int item0;     // first CTA of this matrix
    int row_stride;  // shared-memory bytes per code row (padded against bank conflicts)
};

static_assert(sizeof(FastMat) % 4 == 0 && sizeof(FastMat) / 4 <= 256, "descriptor copy");

struct FastParams {
    int n_items;
    // byte offsets of the shared regions: code rows, norms, operand terms,
    // B fragments, partial sums, 4-bit level table
    int smem_codes, smem_norms, smem_z, smem_frag, smem_red, smem_tab;
    float coef[kMaxLuts][4];          // 2-bit: c0, c1-c0, (c2-c0)/2, c3-c2-c1+c0
    __half lut[kMaxLuts][16];         // 4-bit levels in fp16
    FastMat m[kMaxFastMats];
    int n_mats;
    uint8_t item_mat[kMaxFastItems];  // CTA -> matrix
};

constexpr float kInvSqrt128 = 0.08838834764831845f;

__device__ __forceinline__ float fp8_value(float x, uint32_t *bits) {
    const __nv_fp8_storage_t t = __nv_cvt_float_to_fp8(x, __NV_SATFINITE, __NV_E4M3);
    *bits = t;
    const __half_raw h = __nv_cvt_fp8_to_halfraw(t, __NV_E4M3);
    return __half2float(__half(h));
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
// Largest power of two sigma with amax * sigma <= lim (1 for amax == 0).
__device__ __forceinline__ float pow2_scale(float amax, float lim) {
    if (!(amax > 0.0f)) return 1.0f;
    const float q = __fdiv_rn(lim, amax);
    const int E = min(max((__float_as_int(q) >> 23) & 0xff, 1), 254);
    float s = __int_as_float(E << 23);             // 2^(E-127) <= q
    if (__fmul_rn(amax, s) > lim) s *= 0.5f;       // guard the rounding of q
    return s;
}

// Activation values of rotation task `task` (b, g = task / ng, task % ng):
// lane holds x[b][g*128 + 4 lane + i], zero past `in`.
__device__ __forceinline__ void load_x_task(const FastMat &M, int task, int lane, float (&v)[4]) {
    const int b = task / M.ng, g = task % M.ng;
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
}

__device__ __forceinline__ void load_x(const FastMat &M, int warp, int lane, float (&v)[4]) {
    if (warp < M.B * M.ng)
        load_x_task(M, warp, lane, v);
    else
        v[0] = v[1] = v[2] = v[3] = 0.0f;
}

// Rotation of every (batch row b, group g) by one warp: z = H0 x_{b,g}
// (without the 1/sqrt(128); exact integers for int8 x). Each position k is
// stored as the operand terms the MMAs consume:
//   2-bit path: four e4m3 terms of sigma * z[k] * 2^(k odd ? 7 : 9), byte tau
//   4-bit path: fp16 hi | lo of sigma * z[k]
// with sigma a power of two per (b, g); also sum(z) and 1/sigma per (b, g).
// `xv` holds the values of the warp's first task (loaded early).
__device__ void rotate_all(const FastMat &M, int warp, int lane, const float (&xv)[4], uint32_t *termw, float *gsum,
                           float *ginv) {
    for (int task = warp; task < M.B * M.ng; task += kWarps) {
        float v[4];
        if (task == warp) {
#pragma unroll
            for (int i = 0; i < 4; ++i) v[i] = xv[i];
        } else {
            load_x_task(M, task, lane, v);
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
        const float sigma = M.kind == 0 ? pow2_scale(mx, 448.0f / 512.0f) : pow2_scale(mx, 16384.0f);
        uint32_t *dst = termw + (size_t)task * kGroup + 4 * lane;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            uint32_t w = 0;
            if (M.kind == 0) {
                float x = __fmul_rn(v[i], sigma * ((i & 1) ? 128.0f : 512.0f));  // k = 4 lane + i
#pragma unroll
                for (int tau = 0; tau < 4; ++tau) {
                    uint32_t bits;
                    const float tv = fp8_value(x, &bits);
                    w |= bits << (8 * tau);
                    x = __fsub_rn(x, tv);
                }
            } else {
                const float x = __fmul_rn(v[i], sigma);
                const __half hi = __float2half_rn(x);
                const __half lo = __float2half_rn(__fsub_rn(x, __half2float(hi)));
                w = (uint32_t)__half_as_ushort(hi) | ((uint32_t)__half_as_ushort(lo) << 16);
            }
            dst[i] = w;
        }
        if (lane == 0) {
            gsum[task] = sm;
            ginv[task] = 1.0f / sigma;
        }
    }
}

// ----------------------------------------------------------- 2-bit path --
// Fragment word f (0..7) of lane (gq, t) in group g:
//   f = 2*mu + h, mu = 2*wsel + cp: byte j holds position
//   k = 16*(2t+wsel) + 4j + 2cp + h; column n = gq: batch n/4, term n%4.
__device__ void build_frags_planes(const FastMat &M, const uint32_t *termw, uint32_t *frag) {
    for (int e = threadIdx.x; e < M.ng * 32 * 8; e += kThreads) {
        const int g = e / 256, lane = (e / 8) % 32, f = e % 8;
        const int gq = lane >> 2, t = lane & 3;
        const int b = gq >> 2, tau = gq & 3;
        const int mu = f >> 1, h = f & 1, wsel = mu >> 1, cp = mu & 1;
        uint32_t word = 0;
        if (b < M.B) {
            const uint32_t *tw = termw + (size_t)(b * M.ng + g) * kGroup + 16 * (2 * t + wsel) + 2 * cp + h;
#pragma unroll
            for (int j = 0; j < 4; ++j) word |= ((tw[4 * j] >> (8 * tau)) & 0xffu) << (8 * j);
        }
        frag[e] = word;
    }
}

template <bool THIRD>
__device__ __forceinline__ void planes_group(float (&acc)[4], uint2 cr, uint2 cs, const uint4 fa, const uint4 fb,
                                             float n_r, float n_s, float inv, const float (&cf)[4], float add) {
    // plane accumulators (b0, b1, b0&b1), two independent chains each
    float d[3][2][4];
#pragma unroll
    for (int a = 0; a < 3; ++a)
#pragma unroll
        for (int c = 0; c < 2; ++c)
#pragma unroll
            for (int i = 0; i < 4; ++i) d[a][c][i] = 0.0f;
    const uint32_t bf[8] = {fa.x, fa.y, fa.z, fa.w, fb.x, fb.y, fb.z, fb.w};
#pragma unroll
    for (int mu = 0; mu < 4; ++mu) {
        const int wsel = mu >> 1, cp = mu & 1;
        uint32_t r = wsel ? cr.y : cr.x, s = wsel ? cs.y : cs.x;
        if (cp) {
            r >>= 4;
            s >>= 4;
        }
        const uint32_t b0 = bf[2 * mu], b1 = bf[2 * mu + 1];
        mma_fp8(d[0][cp], r & 0x01010101u, s & 0x01010101u, r & 0x04040404u, s & 0x04040404u, b0, b1);
        mma_fp8(d[1][cp], r & 0x02020202u, s & 0x02020202u, r & 0x08080808u, s & 0x08080808u, b0, b1);
        if (THIRD) {
            const uint32_t tr = r & (r >> 1), ts = s & (s >> 1);
            mma_fp8(d[2][cp], tr & 0x01010101u, ts & 0x01010101u, tr & 0x04040404u, ts & 0x04040404u, b0, b1);
        }
    }
    // d[.][.][0], [1]: row r, cols 2t, 2t+1; [2], [3]: row s
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float v = fmaf(cf[1], d[0][0][i] + d[0][1][i], cf[2] * (d[1][0][i] + d[1][1][i]));
        if (THIRD) v = fmaf(cf[3], d[2][0][i] + d[2][1][i], v);
        v = fmaf(v, inv, (i & 1) ? 0.0f : add);
        acc[i] = fmaf(i >= 2 ? n_s : n_r, v, acc[i]);
    }
}

// ----------------------------------------------------------- 4-bit path --
// Fragment word f (0..15) of lane (gq, t) in group g: MMA nu = f/2, half
// h = f%2: positions 32t + 4nu + 2h + {0,1}; column n = gq: batch n/2,
// term n%2 (fp16 hi / lo).
__device__ void build_frags_lut(const FastMat &M, const uint32_t *termw, uint32_t *frag) {
    for (int e = threadIdx.x; e < M.ng * 32 * 16; e += kThreads) {
        const int g = e / 512, lane = (e / 16) % 32, f = e % 16;
        const int gq = lane >> 2, t = lane & 3;
        const int b = gq >> 1, tau = gq & 1;
        const int nu = f >> 1, h = f & 1;
        uint32_t word = 0;
        if (b < M.B) {
            const uint32_t *tw = termw + (size_t)(b * M.ng + g) * kGroup + 32 * t + 4 * nu + 2 * h;
            word = ((tw[0] >> (16 * tau)) & 0xffffu) | (((tw[1] >> (16 * tau)) & 0xffffu) << 16);
        }
        frag[e] = word;
    }
}

__device__ __forceinline__ void lut_group(float (&acc)[4], const uint4 cr, const uint4 cs, const uint32_t *tab_lane,
                                          const uint32_t *fr, float n_r, float n_s, float inv) {
    float d[4] = {0.f, 0.f, 0.f, 0.f};
    const uint32_t wr[4] = {cr.x, cr.y, cr.z, cr.w}, ws[4] = {cs.x, cs.y, cs.z, cs.w};
    uint32_t frr[16];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint4 v = reinterpret_cast<const uint4 *>(fr)[i];
        frr[4 * i] = v.x;
        frr[4 * i + 1] = v.y;
        frr[4 * i + 2] = v.z;
        frr[4 * i + 3] = v.w;
    }
#pragma unroll
    for (int nu = 0; nu < 8; ++nu) {
        const uint32_t r = wr[nu >> 1] >> (16 * (nu & 1)), s = ws[nu >> 1] >> (16 * (nu & 1));
        const uint32_t a0 = tab_lane[(r & 0xffu) * 32], a2 = tab_lane[((r >> 8) & 0xffu) * 32];
        const uint32_t a1 = tab_lane[(s & 0xffu) * 32], a3 = tab_lane[((s >> 8) & 0xffu) * 32];
        mma_f16(d, a0, a1, a2, a3, frr[2 * nu], frr[2 * nu + 1]);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[i] = fmaf((i >= 2 ? n_s : n_r) * inv, d[i], acc[i]);
}

// ------------------------------------------------------------ the kernel --
__device__ __forceinline__ void cp_async16(void *dst, const void *src, int src_bytes) {
    const uint32_t d = (uint32_t)__cvta_generic_to_shared(dst);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(d), "l"(src), "r"(src_bytes) : "memory");
}

__global__ void __launch_bounds__(kThreads, 2) gemv_fast_kernel(const __grid_constant__ FastParams p) {
    extern __shared__ __align__(16) uint8_t smem[];
    // one copy of this CTA's matrix descriptor in shared memory (parameter
    // reads with a runtime index would otherwise repeat inside the loops)
    __shared__ FastMat sM;
    const int mi = p.item_mat[blockIdx.x];
    if (threadIdx.x < (int)(sizeof(FastMat) / 4))
        reinterpret_cast<uint32_t *>(&sM)[threadIdx.x] = reinterpret_cast<const uint32_t *>(&p.m[mi])[threadIdx.x];
    __syncthreads();
    const FastMat &M = sM;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int gq = lane >> 2, t = lane & 3;
    const int ng = M.ng, B = M.B, kind = M.kind, tiles = M.tiles;
    const int row0 = ((int)blockIdx.x - M.item0) * 16 * tiles;
    const int nrows = 16 * tiles;
    const int rowBytes = ng * (kind == 0 ? 32 : 64);
    const int rs = M.row_stride;  // padded shared-memory row stride (bytes)

    uint8_t *sc = smem + p.smem_codes;                             // [nrows][rs]
    __half *sn = reinterpret_cast<__half *>(smem + p.smem_norms);  // [nrows][ng]
    uint32_t *termw = reinterpret_cast<uint32_t *>(smem + p.smem_z);
    uint32_t *frag = reinterpret_cast<uint32_t *>(smem + p.smem_frag);
    float *red = reinterpret_cast<float *>(smem + p.smem_red);
    __shared__ float gsum[64 * 4], ginv[64 * 4];
    __shared__ float s_alpha[4];

    // ---- 1. the activation values of this warp's first rotation task ----
    float xv[4];
    load_x(M, warp, lane, xv);

    // ---- 2. code rows and norms -> shared memory (16-byte cp.async; rows
    // past the matrix zero-filled); they land while the prologue runs ----
    {
        const int cpr = rowBytes / 16;  // 16-byte chunks per code row
        const int rows_valid = min(nrows, M.out - row0);
        if (cpr <= 32) {
            // a warp copies rpi rows per step, lane -> (row lr, chunk lc)
            const int rpi = 32 / cpr, lr = lane / cpr, lc = lane - lr * cpr;
            if (lr < rpi)
                for (int r = warp * rpi + lr; r < nrows; r += kWarps * rpi) {
                    const bool ok = r < rows_valid;
                    cp_async16(sc + (size_t)r * rs + 16 * lc,
                               M.codes + (size_t)(ok ? row0 + r : 0) * rowBytes + 16 * lc, ok ? 16 : 0);
                }
        } else {
            for (int r = warp; r < nrows; r += kWarps) {
                const bool ok = r < rows_valid;
                for (int c = lane; c < cpr; c += 32)
                    cp_async16(sc + (size_t)r * rs + 16 * c, M.codes + (size_t)(ok ? row0 + r : 0) * rowBytes + 16 * c,
                               ok ? 16 : 0);
            }
        }
        const int nbytes = nrows * ng * 2, avail = rows_valid * ng * 2;
        const uint8_t *src = reinterpret_cast<const uint8_t *>(M.norms + (size_t)row0 * ng);
        for (int c = threadIdx.x; 16 * c < nbytes; c += kThreads) {
            const int left = avail - 16 * c;
            const int n = left >= 16 ? 16 : (left > 0 ? left : 0);
            cp_async16(reinterpret_cast<uint8_t *>(sn) + 16 * c, n ? src + 16 * c : src, n);
        }
        asm volatile("cp.async.commit_group;\n" ::);
    }

    // ---- 3. prologue: rotation, operand terms, B fragments ----
    rotate_all(M, warp, lane, xv, termw, gsum, ginv);
    if (kind == 1) {
        // 256-entry byte -> half2 table, replicated across the 32 banks
        uint32_t *tab = reinterpret_cast<uint32_t *>(smem + p.smem_tab);
        for (int e = threadIdx.x; e < 256 * 32; e += kThreads) {
            const int byte = e >> 5;  // uniform per warp
            tab[e] = (uint32_t)__half_as_ushort(p.lut[M.coef][byte & 15]) |
                     ((uint32_t)__half_as_ushort(p.lut[M.coef][byte >> 4]) << 16);
        }
    }
    if (threadIdx.x < 4) {
        const int b = threadIdx.x;
        float a = kInvSqrt128;
        if (b < B && M.xdt == CQ_X_I8) a = __fmul_rn(M.xs[b], kInvSqrt128);
        s_alpha[b] = a;
    }
    __syncthreads();
    if (kind == 0)
        build_frags_planes(M, termw, frag);
    else
        build_frags_lut(M, termw, frag);
    asm volatile("cp.async.wait_all;\n" ::: "memory");
    __syncthreads();

    // ---- 4. products. Warp w takes tiles w, w+8, ... with every group
    // (two tiles at a time share each group's B fragments), or, with fewer
    // tiles than warps, one tile and every KC-th group ----
    const int KC = M.kchunks;
    const bool wide = tiles >= kWarps;
    const int step = wide ? kWarps : tiles + 1;
    const int kc = wide ? 0 : warp % KC;
    const float cf[4] = {p.coef[M.coef][0], p.coef[M.coef][1], p.coef[M.coef][2], p.coef[M.coef][3]};
    const bool third = cf[3] != 0.0f;

#pragma unroll 1
    for (int ta = wide ? warp : warp / KC; ta < tiles; ta += 2 * step) {
        const int tb = ta + step;
        const bool has_b = tb < tiles;
        float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
        const int ra = 16 * ta + gq, rb = 16 * (has_b ? tb : ta) + gq;  // local rows (and +8)
        if (kind == 0) {
            const int bb = t >> 1;  // batch of this lane's columns 2t, 2t+1
#pragma unroll 1
            for (int g = kc; g < ng; g += KC) {
                const uint4 *fl = reinterpret_cast<const uint4 *>(frag + (size_t)(g * 32 + lane) * 8);
                const uint4 fa = fl[0], fb = fl[1];
                const float inv = bb < B ? ginv[bb * ng + g] : 0.0f;
                const float add = (t & 1) == 0 && bb < B ? cf[0] * gsum[bb * ng + g] : 0.0f;
                const uint2 c0 = *reinterpret_cast<const uint2 *>(sc + (size_t)ra * rs + g * 32 + 8 * t);
                const uint2 c1 = *reinterpret_cast<const uint2 *>(sc + (size_t)(ra + 8) * rs + g * 32 + 8 * t);
                const uint2 c2 = *reinterpret_cast<const uint2 *>(sc + (size_t)rb * rs + g * 32 + 8 * t);
                const uint2 c3 = *reinterpret_cast<const uint2 *>(sc + (size_t)(rb + 8) * rs + g * 32 + 8 * t);
                const float n0 = __half2float(sn[ra * ng + g]), n1 = __half2float(sn[(ra + 8) * ng + g]);
                const float n2 = __half2float(sn[rb * ng + g]), n3 = __half2float(sn[(rb + 8) * ng + g]);
                if (third) {
                    planes_group<true>(acc[0], c0, c1, fa, fb, n0, n1, inv, cf, add);
                    if (has_b) planes_group<true>(acc[1], c2, c3, fa, fb, n2, n3, inv, cf, add);
                } else {
                    planes_group<false>(acc[0], c0, c1, fa, fb, n0, n1, inv, cf, add);
                    if (has_b) planes_group<false>(acc[1], c2, c3, fa, fb, n2, n3, inv, cf, add);
                }
            }
        } else {
            const uint32_t *tab_lane = reinterpret_cast<const uint32_t *>(smem + p.smem_tab) + lane;
#pragma unroll 1
            for (int g = kc; g < ng; g += KC) {
                const uint32_t *fr = frag + (size_t)(g * 32 + lane) * 16;
                uint32_t frr[16];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const uint4 v = reinterpret_cast<const uint4 *>(fr)[i];
                    frr[4 * i] = v.x, frr[4 * i + 1] = v.y, frr[4 * i + 2] = v.z, frr[4 * i + 3] = v.w;
                }
                const float inv = t < B ? ginv[t * ng + g] : 0.0f;
                const uint4 c0 = *reinterpret_cast<const uint4 *>(sc + (size_t)ra * rs + g * 64 + 16 * t);
                const uint4 c1 = *reinterpret_cast<const uint4 *>(sc + (size_t)(ra + 8) * rs + g * 64 + 16 * t);
                lut_group(acc[0], c0, c1, tab_lane, frr, __half2float(sn[ra * ng + g]),
                          __half2float(sn[(ra + 8) * ng + g]), inv);
                if (has_b) {
                    const uint4 c2 = *reinterpret_cast<const uint4 *>(sc + (size_t)rb * rs + g * 64 + 16 * t);
                    const uint4 c3 = *reinterpret_cast<const uint4 *>(sc + (size_t)(rb + 8) * rs + g * 64 + 16 * t);
                    lut_group(acc[1], c2, c3, tab_lane, frr, __half2float(sn[rb * ng + g]),
                              __half2float(sn[(rb + 8) * ng + g]), inv);
                }
            }
        }
        // per-row totals of each batch, for both tiles
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            if (h == 1 && !has_b) break;
            const int tl = h ? tb : ta;
            const int row_r = row0 + 16 * tl + gq, row_s = row_r + 8;
            float yr = acc[h][0] + acc[h][1], ys = acc[h][2] + acc[h][3];
            int bsel;
            bool writer;
            if (kind == 0) {  // batch b in cols 4b..4b+3 = lanes t = 2b, 2b+1
                yr += __shfl_xor_sync(0xffffffffu, yr, 1);
                ys += __shfl_xor_sync(0xffffffffu, ys, 1);
                bsel = t >> 1;
                writer = (t & 1) == 0 && bsel < B;
            } else {  // batch t in cols 2t, 2t+1 (hi, lo terms) of lane t
                bsel = t;
                writer = bsel < B;
            }
            if (KC == 1) {
                if (writer) {
                    const float a = s_alpha[bsel];
                    if (row_r < M.out) M.y[(size_t)bsel * M.out + row_r] = yr * a;
                    if (row_s < M.out) M.y[(size_t)bsel * M.out + row_s] = ys * a;
                }
            } else if (writer) {
                float *rt = red + ((size_t)(tl * KC + kc) * 16) * 4;
                rt[gq * 4 + bsel] = yr;
                rt[(gq + 8) * 4 + bsel] = ys;
            }
        }
    }
    if (KC > 1) {
        __syncthreads();
        for (int e = threadIdx.x; e < tiles * 16 * B; e += kThreads) {
            const int tl = e / (16 * B), rr = (e / B) % 16, b = e % B;
            const int row = row0 + 16 * tl + rr;
            if (row >= M.out) continue;
            float sum = 0.0f;
            for (int c = 0; c < KC; ++c) sum += red[((size_t)(tl * KC + c) * 16 + rr) * 4 + b];
            M.y[(size_t)b * M.out + row] = sum * s_alpha[b];
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

// Shared-memory needs of one launch (maxima over its matrices).
struct Need {
    size_t codes = 0, norms = 0, z = 0, frag = 0, red = 0, tab = 0;
};

// Launches the kernel over the CTAs gathered in p; resets p.
static int flush(FastParams &p, int &nm, int &ncoef, Need &need, cudaStream_t st) {
    if (!p.n_items) return CQ_OK;
    size_t off = 0;
    auto place = [&](int &field, size_t bytes) {
        field = (int)off;
        off += (bytes + 15) / 16 * 16;
    };
    place(p.smem_codes, need.codes);
    place(p.smem_norms, need.norms);
    place(p.smem_z, need.z);
    place(p.smem_frag, need.frag);
    place(p.smem_red, need.red);
    place(p.smem_tab, need.tab);
    const size_t smem = std::max<size_t>(off, 16);
    p.n_mats = nm;
    static bool attr = false;
    if (!attr) {
        cudaFuncSetAttribute(gemv_fast_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
        attr = true;
    }
    if (smem > 200 * 1024) return set_error(CQ_ERR_SHAPE, "fast GEMV needs %zu bytes of shared memory", smem);
    gemv_fast_kernel<<<p.n_items, kThreads, smem, st>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return set_error(CQ_ERR_CUDA, "fast gemv launch: %s", cudaGetErrorString(e));
    p.n_items = 0;
    nm = 0;
    ncoef = 0;
    need = Need();
    return CQ_OK;
}

int launch_gemv_fast(const cq_gemv_desc *d, const int *idx, int n, void *stream) {
    static FastParams p;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    p.n_items = 0;
    int ncoef = 0, nm = 0;
    Need need;
    for (int ii = 0; ii < n; ++ii) {
        const cq_gemv_desc &D = d[idx[ii]];
        const int ip = in_padded(D.in), W = width_of(D.bits), ng = ip / kGroup;
        const int kind = W == 2 ? 0 : 1;
        // rows per CTA: about 48 KB of codes, a power-of-two number of 16-row tiles
        const int rowB = ng * (kind == 0 ? 32 : 64) + 2 * ng;
        const int tiles = std::max(1, (48 * 1024) / (rowB * 16));
        int tp = 1;
        while (tp * 2 <= tiles && tp * 2 <= 32) tp *= 2;
        const int need_tiles = (D.out + 15) / 16;
        while (tp > 1 && tp / 2 >= need_tiles) tp /= 2;
        const int items = (D.out + 16 * tp - 1) / (16 * tp);
        if (nm == kMaxFastMats || p.n_items + items > kMaxFastItems) {
            const int e = flush(p, nm, ncoef, need, st);
            if (e) return e;
        }
        FastMat &M = p.m[nm];
        M.codes = D.blob;
        M.norms = reinterpret_cast<const __half *>(D.blob + (size_t)D.out * ip * W / 8);
        M.x = D.x;
        M.xs = D.x_scale;
        M.y = D.y;
        M.out = D.out;
        M.in = D.in;
        M.ng = ng;
        M.bits = D.bits;
        M.xdt = D.x_dtype;
        M.B = D.B;
        M.kind = kind;
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
            if (ncoef == kMaxLuts) {
                const int e = flush(p, nm, ncoef, need, st);
                if (e) return e;
                --ii;  // redo this descriptor in a fresh launch
                continue;
            }
            for (int k = 0; k < 4; ++k) p.coef[ncoef][k] = cf[k];
            for (int k = 0; k < 16; ++k) p.lut[ncoef][k] = lut[k];
            ci = ncoef++;
        }
        M.coef = ci;
        M.tiles = tp;
        M.kchunks = tp >= kWarps ? 1 : std::min(kWarps / tp, M.ng);
        // row stride in shared memory: the 2-bit path reads 8 bytes per lane
        // (rows of a half-warp must start 8 banks apart), the 4-bit path 16
        // bytes (rows of a quarter-warp 16 banks apart)
        const int rowBytes = M.ng * (M.kind == 0 ? 32 : 64);
        const int want = M.kind == 0 ? 32 : 64;
        M.row_stride = rowBytes + (((want - rowBytes) % 128) + 128) % 128;

        if (items > kMaxFastItems) return set_error(CQ_ERR_SHAPE, "matrix too tall for one fast GEMV launch");
        M.item0 = p.n_items;
        for (int k = 0; k < items; ++k) p.item_mat[p.n_items + k] = (uint8_t)nm;
        p.n_items += items;
        const size_t nrows = 16 * (size_t)tp;
        need.codes = std::max(need.codes, nrows * M.row_stride);
        need.norms = std::max(need.norms, nrows * M.ng * 2);
        need.z = std::max(need.z, (size_t)M.B * M.ng * kGroup * sizeof(uint32_t));
        need.frag = std::max(need.frag, (size_t)M.ng * 32 * (M.kind == 0 ? 8 : 16) * sizeof(uint32_t));
        if (M.kchunks > 1) need.red = std::max(need.red, (size_t)M.tiles * M.kchunks * 16 * 4 * sizeof(float));
        if (M.kind == 1) need.tab = 256 * 32 * sizeof(uint32_t);
        ++nm;
    }
    return flush(p, nm, ncoef, need, st);
}

}  // namespace cq
