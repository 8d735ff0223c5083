// cq_gemv_fast.cu -- tensor-core GEMV over CQ-packed weights at small
// batches: the tile kernel (inputs of up to 12 groups: the decode step) and
// the streamed kernel (inputs of 16 to 32 groups).
//
// Per group g of 128 inputs the product is the rotated-domain identity
// (OpenNeedle docs/reference.md; "The .cact archive and Cactus Quants",
// "Reconstructing one group"):
//     y[o] += n[o][g] * sum_k c[q[o,g,k]] * z[g,k],   z = H x (per group).
// The activation is rotated once per thread block and laid out as MMA
// operand fragments in shared memory; the weights are never expanded
// beyond the registers that feed one MMA ("How the kernel reads it").
//
// GB300 mapping. The weights stay packed in HBM and in shared memory. Code
// bytes become fp16 levels in registers -- through byte -> levels tables
// replicated across the shared-memory banks (conflict-free lookups), or,
// for 2-bit codes, partly by byte permutes over the levels' bytes held in
// registers -- and feed mma.sync m16n8k16 (fp16 in, fp32 accumulate) as the
// A operand. z enters as the B operand split into fp16 hi + lo terms (two
// MMA columns per batch row), so the products are exact up to the fp16
// rounding of the levels. Each norm and the activation's power-of-two scale
// are applied in fp32 per row and group.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>

#include "cq_internal.h"

namespace cq {

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxFastB = 4;
constexpr int kMaxFastNg = 32;
constexpr int kFragWords = 16;  // B-fragment words per lane and group

struct FastMat {
    const uint8_t *codes;
    const __half *norms;
    const void *x;
    const float *xs;
    float *y;
    int out, in, ng, bits, xdt, B;
    int kind;      // 0: 2-bit codes, 1: 4-bit codes, 2: 1-bit codes, 3: 3-bit codes
    int lut;       // index into the launch's level tables
    int tiles;     // row tiles (16 rows) per CTA
    int kchunks;   // warps sharing one tile (split of the groups)
    int item0;     // first CTA of this matrix
    int row_stride;  // shared-memory bytes per code row (padded against bank conflicts)
};

static_assert(sizeof(FastMat) % 4 == 0 && sizeof(FastMat) / 4 <= 256, "descriptor copy");

constexpr float kInvSqrt128 = 0.08838834764831845f;

__device__ __forceinline__ void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                        uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void cp_async16(void *dst, const void *src, int src_bytes) {
    const uint32_t d = (uint32_t)__cvta_generic_to_shared(dst);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(d), "l"(src), "r"(src_bytes) : "memory");
}

// ------------------------------------------------------------ rotation --
// Largest power of two sigma with amax * sigma <= lim (1 for amax == 0).
__device__ __forceinline__ float pow2_scale(float amax, float lim) {
    if (!(amax > 0.0f)) return 1.0f;
    const float q = __fdiv_rn(lim, amax);
    const int E = min(max((__float_as_int(q) >> 23) & 0xff, 1), 254);
    float s = __int_as_float(E << 23);             // 2^(E-127) <= q
    if (__fmul_rn(amax, s) > lim) s *= 0.5f;       // guard the rounding of q
    return s;
}

// Activation values of (batch row b, group g): lane holds
// x[b][g*128 + 4 lane + i], zero past `in`.
__device__ __forceinline__ void load_x_bg(const FastMat &A, int b, int g, int lane, float (&v)[4]) {
    const int col0 = g * kGroup + 4 * lane;
    if (A.xdt == CQ_X_I8 && (A.in & 3) == 0 && (reinterpret_cast<uintptr_t>(A.x) & 3) == 0) {
        // one 4-byte load, kept in program order (issued before the copies
        // and the table that follow it)
        uint32_t w = 0;
        if (col0 < A.in)
            asm volatile("ld.global.b32 %0, [%1];\n"
                         : "=r"(w)
                         : "l"(static_cast<const int8_t *>(A.x) + (size_t)b * A.in + col0));
#pragma unroll
        for (int i = 0; i < 4; ++i) v[i] = (float)(int8_t)(w >> (8 * i));
    } else if (A.xdt == CQ_X_I8) {
        const int8_t *xq = static_cast<const int8_t *>(A.x) + (size_t)b * A.in;
#pragma unroll
        for (int i = 0; i < 4; ++i) v[i] = col0 + i < A.in ? (float)xq[col0 + i] : 0.0f;
    } else {
        const float *xf = static_cast<const float *>(A.x) + (size_t)b * A.in;
#pragma unroll
        for (int i = 0; i < 4; ++i) v[i] = col0 + i < A.in ? xf[col0 + i] : 0.0f;
    }
}

// Rotation of (b, g) by one warp, from the values load_x_bg gave this lane:
// z = H0 x_{b,g} (without the 1/sqrt(128); exact integers for int8 x). Position k is written to terms[k] as fp16
// hi | lo of sigma * z[k], sigma a power of two per (b, g) (|sigma z| <=
// 2^14, so hi + lo carries z to ~2^-22 relative); returns 1/sigma.
template <bool G64 = false>
__device__ float rotate_bg(float (&v)[4], int lane, uint32_t *terms) {
    float a0 = v[0] + v[1], a1 = v[0] - v[1], a2 = v[2] + v[3], a3 = v[2] - v[3];
    v[0] = a0 + a2;
    v[1] = a1 + a3;
    v[2] = a0 - a2;
    v[3] = a1 - a3;
#pragma unroll
    for (int m = 1; m < (G64 ? 16 : 32); m <<= 1)  // groups of 64: positions 0-63 and 64-127 apart
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float o = __shfl_xor_sync(0xffffffffu, v[i], m);
            v[i] = (lane & m) ? o - v[i] : v[i] + o;
        }
    float mx = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
#pragma unroll
    for (int m = 16; m; m >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, m));
    const float sigma = pow2_scale(mx, 16384.0f);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float x = __fmul_rn(v[i], sigma);
        const __half hi = __float2half_rn(x);
        const __half lo = __float2half_rn(__fsub_rn(x, __half2float(hi)));
        terms[4 * lane + i] = (uint32_t)__half_as_ushort(hi) | ((uint32_t)__half_as_ushort(lo) << 16);
    }
    return 1.0f / sigma;
}

// B-fragment words of one group from the terms of every batch row
// (terms[b][k]). Word f (0..15) of lane (gq, t): MMA nu = f/2, half h = f%2,
// positions 32t + 4nu + 2h + {0,1}; column n = gq: batch n/2, term n%2
// (fp16 hi / lo). dst receives the group's words as [f/4][lane][f%4], so
// that a warp's 16-byte load of words 4i..4i+3 is contiguous across lanes
// (free of bank conflicts).
__device__ void frag_words(const FastMat &A, const uint32_t (*terms)[kGroup], int lane, uint32_t *dst) {
    const int gq = lane >> 2, t = lane & 3;
    const int b = gq >> 1, tau = gq & 1;
    uint32_t w[kFragWords];
#pragma unroll
    for (int f = 0; f < kFragWords; ++f) {
        const int nu = f >> 1, h = f & 1;
        uint32_t word = 0;
        if (b < A.B) {
            const uint32_t *tw = terms[b] + 32 * t + 4 * nu + 2 * h;
            word = ((tw[0] >> (16 * tau)) & 0xffffu) | (((tw[1] >> (16 * tau)) & 0xffffu) << 16);
        }
        w[f] = word;
    }
    uint4 *d4 = reinterpret_cast<uint4 *>(dst);
#pragma unroll
    for (int i = 0; i < 4; ++i) d4[i * 32 + lane] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
}

// -------------------------------------------------------------- products --
// One 16-row tile and one group: rows r (gq) and s (gq + 8), lane t. The
// lane's code bytes of each row (8 for 2-bit codes, 16 for 4-bit codes)
// cover positions 32t .. 32t+31 of the group; MMA nu takes positions
// 32t + 4nu .. +3, i.e. byte nu (2-bit) or bytes 2nu, 2nu+1 (4-bit).
// d[0], d[1]: row r, columns 2t, 2t+1 (hi, lo terms of batch t); d[2], d[3]:
// row s.
__device__ __forceinline__ void lut2_group(float (&acc)[4], uint2 cr, uint2 cs, const uint2 *tab_lane,
                                           const uint32_t (&fr)[kFragWords], float nr, float ns) {
    float d[4] = {0.f, 0.f, 0.f, 0.f};
    const uint32_t wr[2] = {cr.x, cr.y}, ws[2] = {cs.x, cs.y};
#pragma unroll
    for (int nu = 0; nu < 8; ++nu) {
        const uint32_t br = __byte_perm(wr[nu >> 2], 0, 0x4440 + (nu & 3));
        const uint32_t bs = __byte_perm(ws[nu >> 2], 0, 0x4440 + (nu & 3));
        const uint2 er = tab_lane[br * 16], es = tab_lane[bs * 16];
        mma_f16(d, er.x, es.x, er.y, es.y, fr[2 * nu], fr[2 * nu + 1]);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[i] = fmaf(i >= 2 ? ns : nr, d[i], acc[i]);
}

// 1-bit codes: the lane's 4 code bytes of each row cover positions 32t ..
// 32t+31; MMA nu takes positions 32t + 4nu .. +3, nibble nu of the word.
__device__ __forceinline__ void lut1_group(float (&acc)[4], uint32_t cr, uint32_t cs, const uint2 *tab_lane,
                                           const uint32_t (&fr)[kFragWords], float nr, float ns) {
    float d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int nu = 0; nu < 8; ++nu) {
        const uint2 er = tab_lane[((cr >> (4 * nu)) & 15u) * 16], es = tab_lane[((cs >> (4 * nu)) & 15u) * 16];
        mma_f16(d, er.x, es.x, er.y, es.y, fr[2 * nu], fr[2 * nu + 1]);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[i] = fmaf(i >= 2 ? ns : nr, d[i], acc[i]);
}

// The lane's three code words of a 3-bit row at `p` (12 bytes from 4-byte
// aligned shared memory), with a zero word after them.
__device__ __forceinline__ void load3(const uint8_t *p, uint32_t (&w)[4]) {
    const uint32_t *q = reinterpret_cast<const uint32_t *>(p);
    w[0] = q[0];
    w[1] = q[1];
    w[2] = q[2];
    w[3] = 0u;
}

// 3-bit codes: the lane's 12 code bytes of each row (three words) cover
// positions 32t .. 32t+31; MMA nu takes the 6-bit code pairs at bits 12 nu
// and 12 nu + 6 of them (a pair may straddle two words), each a lookup of
// two fp16 levels.
__device__ __forceinline__ void lut3_group(float (&acc)[4], const uint32_t (&wr)[4], const uint32_t (&ws)[4],
                                           const uint32_t *tab_lane, const uint32_t (&fr)[kFragWords], float nr,
                                           float ns) {
    float d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int nu = 0; nu < 8; ++nu) {
        const int b0 = 12 * nu, b1 = b0 + 6;
        const uint32_t p0 = __funnelshift_r(wr[b0 >> 5], wr[(b0 >> 5) + 1], b0 & 31) & 63u;
        const uint32_t p1 = __funnelshift_r(wr[b1 >> 5], wr[(b1 >> 5) + 1], b1 & 31) & 63u;
        const uint32_t q0 = __funnelshift_r(ws[b0 >> 5], ws[(b0 >> 5) + 1], b0 & 31) & 63u;
        const uint32_t q1 = __funnelshift_r(ws[b1 >> 5], ws[(b1 >> 5) + 1], b1 & 31) & 63u;
        mma_f16(d, tab_lane[p0 * 32], tab_lane[q0 * 32], tab_lane[p1 * 32], tab_lane[q1 * 32], fr[2 * nu],
                fr[2 * nu + 1]);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[i] = fmaf(i >= 2 ? ns : nr, d[i], acc[i]);
}

__device__ __forceinline__ void lut4_group(float (&acc)[4], uint4 cr, uint4 cs, const uint32_t *tab_lane,
                                           const uint32_t (&fr)[kFragWords], float nr, float ns) {
    float d[4] = {0.f, 0.f, 0.f, 0.f};
    const uint32_t wr[4] = {cr.x, cr.y, cr.z, cr.w}, ws[4] = {cs.x, cs.y, cs.z, cs.w};
#pragma unroll
    for (int nu = 0; nu < 8; ++nu) {
        const uint32_t r = wr[nu >> 1] >> (16 * (nu & 1)), s = ws[nu >> 1] >> (16 * (nu & 1));
        const uint32_t a0 = tab_lane[(r & 0xffu) * 32], a2 = tab_lane[((r >> 8) & 0xffu) * 32];
        const uint32_t a1 = tab_lane[(s & 0xffu) * 32], a3 = tab_lane[((s >> 8) & 0xffu) * 32];
        mma_f16(d, a0, a1, a2, a3, fr[2 * nu], fr[2 * nu + 1]);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[i] = fmaf(i >= 2 ? ns : nr, d[i], acc[i]);
}

// Level table of this matrix's codes in shared memory at `tab`: 2-bit codes
// a byte -> four fp16 levels (16 copies, so that a half-warp's 8-byte lookups
// hit distinct banks); 4-bit codes a byte -> two levels (32 copies); 1-bit
// codes a nibble -> four levels (16 copies).
template <bool WITH3 = false>  // 3-bit tables only where the kernel takes 3-bit codes
__device__ __forceinline__ void build_level_table(int kind, const __half *lv, uint8_t *tab) {
    if (WITH3 && kind == 3) {  // a 6-bit code pair -> two fp16 levels, 32 copies
        uint32_t *t = reinterpret_cast<uint32_t *>(tab);
        for (int e = threadIdx.x; e < 64 * 32; e += kThreads) {
            const int v = e >> 5;
            t[e] = (uint32_t)__half_as_ushort(lv[v & 7]) | ((uint32_t)__half_as_ushort(lv[v >> 3]) << 16);
        }
    } else if (kind == 2) {
        uint2 *t = reinterpret_cast<uint2 *>(tab);
        for (int e = threadIdx.x; e < 16 * 16; e += kThreads) {
            const int v = e >> 4;
            t[e] = make_uint2(
                (uint32_t)__half_as_ushort(lv[v & 1]) | ((uint32_t)__half_as_ushort(lv[(v >> 1) & 1]) << 16),
                (uint32_t)__half_as_ushort(lv[(v >> 2) & 1]) | ((uint32_t)__half_as_ushort(lv[v >> 3]) << 16));
        }
    } else if (kind == 0) {
        uint2 *t = reinterpret_cast<uint2 *>(tab);
        for (int e = threadIdx.x; e < 256 * 16; e += kThreads) {
            const int v = e >> 4;
            t[e] = make_uint2(
                (uint32_t)__half_as_ushort(lv[v & 3]) | ((uint32_t)__half_as_ushort(lv[(v >> 2) & 3]) << 16),
                (uint32_t)__half_as_ushort(lv[(v >> 4) & 3]) | ((uint32_t)__half_as_ushort(lv[v >> 6]) << 16));
        }
    } else {
        uint32_t *t = reinterpret_cast<uint32_t *>(tab);
        for (int e = threadIdx.x; e < 256 * 32; e += kThreads) {
            const int v = e >> 5;
            t[e] = (uint32_t)__half_as_ushort(lv[v & 15]) | ((uint32_t)__half_as_ushort(lv[v >> 4]) << 16);
        }
    }
}

// The activation of M as B fragments: warp w rotates groups w, w+8, ... of
// every batch row (scratch `terms`: kWarps x kMaxFastB x 128 words) into
// frag[g] and 1/sigma into ginv[b][g]. No block barrier: the caller syncs.
template <bool G64 = false>
__device__ __forceinline__ void rotate_activation(const FastMat &M, uint8_t *terms_base, uint32_t *frag, float *ginv) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, ng = M.ng, B = M.B;
    float xv[kMaxFastB][4];
    if (warp < ng)  // the first group's values, requested before anything else
#pragma unroll
        for (int b = 0; b < kMaxFastB; ++b)
            if (b < B) load_x_bg(M, b, warp, lane, xv[b]);
    uint32_t(*terms)[kGroup] = reinterpret_cast<uint32_t(*)[kGroup]>(terms_base) + warp * kMaxFastB;
    for (int g = warp; g < ng; g += kWarps) {
#pragma unroll
        for (int b = 0; b < kMaxFastB; ++b) {
            if (b >= B) break;
            if (g != warp) load_x_bg(M, b, g, lane, xv[b]);
            const float inv = rotate_bg<G64>(xv[b], lane, terms[b]);
            if (lane == 0) ginv[b * ng + g] = inv;
        }
        __syncwarp();
        frag_words(M, terms, lane, frag + (size_t)g * 32 * kFragWords);
        __syncwarp();
    }
}

// Groups of 64 (streamed kernel): a lane quarter owns 32 consecutive
// positions of a 128-span and one MMA sums all four quarters, so the two
// halves run as separate chains d (quarters 0-1) and e (2-3), each MMA
// reading the B words of the other half as zero, and take their own norms.
template <int KIND>
__device__ __forceinline__ void lut_group64(float (&acc)[4], const uint8_t *rowr, const uint8_t *rows,
                                            const void *tab, const uint32_t (&fr)[kFragWords], float nr, float ns,
                                            float hr, float hs) {
    const int lane = threadIdx.x & 31, t = lane & 3;
    const bool lo = t < 2;
    float d[4] = {0.f, 0.f, 0.f, 0.f}, e[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int nu = 0; nu < 8; ++nu) {
        uint32_t a0, a1, a2, a3;
        if (KIND == 0) {  // 2-bit: byte nu of the lane's 8 bytes
            const uint2 *tb = static_cast<const uint2 *>(tab) + (lane & 15);
            const uint2 er = tb[(uint32_t)rowr[8 * t + nu] * 16], es = tb[(uint32_t)rows[8 * t + nu] * 16];
            a0 = er.x, a1 = es.x, a2 = er.y, a3 = es.y;
        } else if (KIND == 2) {  // 1-bit: nibble nu of the lane's 4 bytes
            const uint2 *tb = static_cast<const uint2 *>(tab) + (lane & 15);
            const uint32_t wr = rowr[4 * t + (nu >> 1)] >> (4 * (nu & 1)), ws = rows[4 * t + (nu >> 1)] >> (4 * (nu & 1));
            const uint2 er = tb[(wr & 15u) * 16], es = tb[(ws & 15u) * 16];
            a0 = er.x, a1 = es.x, a2 = er.y, a3 = es.y;
        } else {  // 4-bit: bytes 2nu, 2nu+1 of the lane's 16 bytes
            const uint32_t *tb = static_cast<const uint32_t *>(tab) + lane;
            a0 = tb[(uint32_t)rowr[16 * t + 2 * nu] * 32], a2 = tb[(uint32_t)rowr[16 * t + 2 * nu + 1] * 32];
            a1 = tb[(uint32_t)rows[16 * t + 2 * nu] * 32], a3 = tb[(uint32_t)rows[16 * t + 2 * nu + 1] * 32];
        }
        mma_f16(d, a0, a1, a2, a3, lo ? fr[2 * nu] : 0u, lo ? fr[2 * nu + 1] : 0u);
        mma_f16(e, a0, a1, a2, a3, lo ? 0u : fr[2 * nu], lo ? 0u : fr[2 * nu + 1]);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        acc[i] = fmaf(i >= 2 ? ns : nr, d[i], acc[i]);
        acc[i] = fmaf(i >= 2 ? hs : hr, e[i], acc[i]);
    }
}

// --------------------------------------------------------- the tile kernel --
// GEMV over inputs of at most 12 groups at batch <= 4 (the decode step). The
// 16-row tiles of a launch, in the order of its matrices, are cut into runs
// of about equal bytes, one run per CTA and two CTAs per SM. A CTA copies its
// run's code rows and norms into shared memory and builds its level table
// before it waits for the grid ahead of it on the stream (programmatic
// dependent launch), so that those copies overlap the previous launch; then
// it rotates each distinct activation its run reads once (an activation
// "slot": the FWHT of a group in one warp, its fp16 hi + lo terms moved into
// MMA B fragments by warp shuffles), and its warps take the run's tiles
// round-robin, each tile with all of its groups, and write the outputs.
//
// 2-bit codes (CQ2, ternary crumbs) are expanded to fp16 levels two ways,
// half of each lane's code bytes each way, so that neither the shared-memory
// pipe nor the integer pipe carries all of the expansion: bytes 0-3 of a
// lane's 8 code bytes per row and group go through the byte -> four levels
// table (one 8-byte lookup per byte); bytes 4-7 are expanded in registers:
// the four 2-bit fields at bit 2i of the word's bytes become byte selectors
// (c -> c | (c | 4) << 4) of a byte permute over the four levels' low and
// high bytes, which yields the fp16 pairs (field i of bytes 4,5) and (field i
// of bytes 6,7). The MMA k order of those pairs differs from the table's;
// the activation fragments are laid out to match ("hybrid" layout). 4-bit
// and 1-bit codes use their tables only ("natural" layout).
constexpr int kTileMaxMats = 144;
constexpr int kTileMaxSegs = 448;
constexpr int kTileMaxCtas = 320;
constexpr int kTileRunSegs = 8;            // matrices per run
constexpr int kTileSlots = 6;              // distinct activations per run (at most 12 / ng)
constexpr int kTileFragGroups = 12;        // activation fragments per CTA: slots x groups
constexpr int kTileMaxNg = 12;
constexpr int kTileCodeBudget = 48 * 1024;  // shared-memory bytes of code rows per run (padded rows)

struct TileSeg {
    int mat;     // matrix (index into TileParams::m)
    int tile0;   // first 16-row tile of the matrix in this run
    int ntiles;  // tiles of the matrix in this run
    int slot;    // activation slot of the run
};

struct TileParams {
    int smem_tab, smem_codes, smem_norms, smem_frag;  // byte offsets of the shared regions
    int cta_seg[kTileMaxCtas + 1];                    // segments of CTA c: cta_seg[c] .. cta_seg[c+1]-1
    TileSeg seg[kTileMaxSegs];
    __half lut[kMaxLuts][16];
    FastMat m[kTileMaxMats];
};

static_assert(sizeof(TileParams) <= 32000, "kernel parameter block");

// z of one batch row and group after rotate_bg, as this lane's four
// positions 4 lane + i (fp16 hi | lo << 16); returns the B-fragment words
// of batch row b into w (lanes whose MMA column is another batch row keep
// their words). Word f of lane (gq, t): MMA j = f / 2, half h = f % 2.
// Natural layout: positions 32t + 4j + 2h + {0, 1}; hybrid layout, MMAs
// j >= 4: positions 32t + 16 + 8h + (j - 4) + {0, 4}. Column gq holds batch
// row gq / 2, term gq % 2 (hi / lo).
template <bool HYB>
__device__ __forceinline__ void frag_from_lanes(const uint32_t (&e)[4], int b, int lane, uint32_t (&w)[kFragWords]) {
    const int gq = lane >> 2, t = lane & 3, tau = 16 * (gq & 1);
    const bool mine = (gq >> 1) == b;
#pragma unroll
    for (int f = 0; f < kFragWords; ++f) {
        const int j = f >> 1, h = f & 1;
        uint32_t a, c;
        if (!HYB || j < 4) {
            a = __shfl_sync(0xffffffffu, e[2 * h], 8 * t + j);
            c = __shfl_sync(0xffffffffu, e[2 * h + 1], 8 * t + j);
        } else {
            a = __shfl_sync(0xffffffffu, e[j - 4], 8 * t + 4 + 2 * h);
            c = __shfl_sync(0xffffffffu, e[j - 4], 8 * t + 5 + 2 * h);
        }
        if (mine) w[f] = ((a >> tau) & 0xffffu) | (((c >> tau) & 0xffffu) << 16);
    }
}

// Rotation of (batch row b, group g) by one warp from this lane's values v
// (load_x_bg): z = H0 x (exact integers for int8 x), scaled by a power of
// two sigma (|sigma z| <= 2^14) and split into fp16 hi + lo terms, returned
// per position 4 lane + i in e; returns 1/sigma.
__device__ __forceinline__ float rotate_regs(float (&v)[4], int lane, uint32_t (&e)[4]) {
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
#pragma unroll
    for (int m = 16; m; m >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, m));
    const float sigma = pow2_scale(mx, 16384.0f);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float x = __fmul_rn(v[i], sigma);
        const __half hi = __float2half_rn(x);
        const __half lo = __float2half_rn(__fsub_rn(x, __half2float(hi)));
        e[i] = (uint32_t)__half_as_ushort(hi) | ((uint32_t)__half_as_ushort(lo) << 16);
    }
    return 1.0f / sigma;
}

// Register expansion of 2-bit codes: the fields at bit 2i of the four bytes
// of w, as fp16 level pairs (bytes 0, 1) in lo[i] and (bytes 2, 3) in hi[i].
// llo / lhi hold the low / high bytes of the four levels.
__device__ __forceinline__ void expand2_regs(uint32_t w, uint32_t llo, uint32_t lhi, uint32_t (&lo)[4],
                                             uint32_t (&hi)[4]) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t x = (w >> (2 * i)) & 0x03030303u;
        const uint32_t s = x * 0x11u + 0x40404040u;  // c -> selector nibbles c, c | 4
        lo[i] = __byte_perm(llo, lhi, s);
        hi[i] = __byte_perm(llo, lhi, s >> 16);
    }
}

// One 16-row tile and one group: rows gq (codes cr) and gq + 8 (cs) of this
// lane, products of the group's 8 MMAs into d.
template <int KIND>
__device__ __forceinline__ void tile_group(float (&d)[4], const uint8_t *r0, const uint8_t *r1, const uint8_t *tab,
                                           uint32_t llo, uint32_t lhi, const uint32_t (&fr)[kFragWords], int lane) {
    const int t = lane & 3;
    if (KIND == 0) {  // 2-bit: bytes 8t .. 8t+7 of the group
        const uint2 cr = *reinterpret_cast<const uint2 *>(r0 + 8 * t);
        const uint2 cs = *reinterpret_cast<const uint2 *>(r1 + 8 * t);
        const uint8_t *tb = tab + 8 * (lane & 15);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint2 er = *reinterpret_cast<const uint2 *>(tb + 128 * __byte_perm(cr.x, 0, 0x4440 + i));
            const uint2 es = *reinterpret_cast<const uint2 *>(tb + 128 * __byte_perm(cs.x, 0, 0x4440 + i));
            mma_f16(d, er.x, es.x, er.y, es.y, fr[2 * i], fr[2 * i + 1]);
        }
        uint32_t rl[4], rh[4], sl[4], sh[4];
        expand2_regs(cr.y, llo, lhi, rl, rh);
        expand2_regs(cs.y, llo, lhi, sl, sh);
#pragma unroll
        for (int i = 0; i < 4; ++i) mma_f16(d, rl[i], sl[i], rh[i], sh[i], fr[8 + 2 * i], fr[9 + 2 * i]);
    } else if (KIND == 1) {  // 4-bit: bytes 16t .. 16t+15, MMA j takes bytes 2j, 2j+1
        const uint4 cr = *reinterpret_cast<const uint4 *>(r0 + 16 * t);
        const uint4 cs = *reinterpret_cast<const uint4 *>(r1 + 16 * t);
        const uint32_t wr[4] = {cr.x, cr.y, cr.z, cr.w}, ws[4] = {cs.x, cs.y, cs.z, cs.w};
        const uint8_t *tb = tab + 4 * lane;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const uint32_t r = wr[j >> 1] >> (16 * (j & 1)), s = ws[j >> 1] >> (16 * (j & 1));
            const uint32_t a0 = *reinterpret_cast<const uint32_t *>(tb + 128 * (r & 0xffu));
            const uint32_t a2 = *reinterpret_cast<const uint32_t *>(tb + 128 * ((r >> 8) & 0xffu));
            const uint32_t a1 = *reinterpret_cast<const uint32_t *>(tb + 128 * (s & 0xffu));
            const uint32_t a3 = *reinterpret_cast<const uint32_t *>(tb + 128 * ((s >> 8) & 0xffu));
            mma_f16(d, a0, a1, a2, a3, fr[2 * j], fr[2 * j + 1]);
        }
    } else {  // 1-bit: bytes 4t .. 4t+3, MMA j takes nibble j
        const uint32_t cr = *reinterpret_cast<const uint32_t *>(r0 + 4 * t);
        const uint32_t cs = *reinterpret_cast<const uint32_t *>(r1 + 4 * t);
        const uint8_t *tb = tab + 8 * (lane & 15);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const uint2 er = *reinterpret_cast<const uint2 *>(tb + 128 * ((cr >> (4 * j)) & 15u));
            const uint2 es = *reinterpret_cast<const uint2 *>(tb + 128 * ((cs >> (4 * j)) & 15u));
            mma_f16(d, er.x, es.x, er.y, es.y, fr[2 * j], fr[2 * j + 1]);
        }
    }
}

template <int KIND>
__device__ __forceinline__ void tile_run(const TileParams &p, const FastMat *sM, const TileSeg *sS, const int *s_tp,
                                         const int *s_cb, const int *s_nb, const int *s_slot_g0,
                                         const float (*s_ginv)[kMaxFastB][kTileMaxNg],
                                         const float (*s_alpha)[kMaxFastB], uint8_t *smem, uint32_t llo, uint32_t lhi,
                                         int nseg) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, gq = lane >> 2, t = lane & 3;
    const uint8_t *sc = smem + p.smem_codes, *sn = smem + p.smem_norms, *tab = smem + p.smem_tab;
    const uint32_t *frag = reinterpret_cast<const uint32_t *>(smem + p.smem_frag);
    const int total = s_tp[nseg];
    int s = 0;
#pragma unroll 1
    for (int tt = warp; tt < total; tt += kWarps) {
        while (tt >= s_tp[s + 1]) ++s;
        const FastMat &M = sM[s];
        const int ng = M.ng, B = M.B, rs = M.row_stride, sl = sS[s].slot;
        const int lt = tt - s_tp[s];  // tile of this segment
        const uint8_t *rowr = sc + s_cb[s] + (size_t)(16 * lt + gq) * rs;
        const __half *nr = reinterpret_cast<const __half *>(sn + s_nb[s]) + (16 * lt + gq) * ng;
        const bool live = gq < 2 * B;  // this lane's B column belongs to a batch row
        const int gbytes = KIND == 0 ? 32 : KIND == 1 ? 64 : 16;
        const uint32_t *fs = frag + (size_t)s_slot_g0[sl] * 32 * kFragWords;  // the slot's fragments
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 1
        for (int g = 0; g < ng; ++g) {
            uint32_t fr[kFragWords];
            const uint4 *fl = reinterpret_cast<const uint4 *>(fs + (size_t)g * 32 * kFragWords) + lane;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const uint4 v = live ? fl[32 * k] : make_uint4(0, 0, 0, 0);
                fr[4 * k] = v.x, fr[4 * k + 1] = v.y, fr[4 * k + 2] = v.z, fr[4 * k + 3] = v.w;
            }
            float d[4] = {0.f, 0.f, 0.f, 0.f};
            tile_group<KIND>(d, rowr + g * gbytes, rowr + 8 * rs + g * gbytes, tab, llo, lhi, fr, lane);
            const float inv = t < B ? s_ginv[sl][t][g] : 0.0f;
            const float n0 = __half2float(nr[g]) * inv, n1 = __half2float(nr[8 * ng + g]) * inv;
            acc[0] = fmaf(n0, d[0], acc[0]);
            acc[1] = fmaf(n0, d[1], acc[1]);
            acc[2] = fmaf(n1, d[2], acc[2]);
            acc[3] = fmaf(n1, d[3], acc[3]);
        }
        // columns 2t, 2t+1: hi and lo terms of batch row t
        if (t < B) {
            const int row = 16 * (sS[s].tile0 + lt) + gq;
            const float a = s_alpha[sl][t];
            if (row < M.out) M.y[(size_t)t * M.out + row] = (acc[0] + acc[1]) * a;
            if (row + 8 < M.out) M.y[(size_t)t * M.out + row + 8] = (acc[2] + acc[3]) * a;
        }
    }
}

__global__ void __launch_bounds__(kThreads, 2) gemv_tile_kernel(const __grid_constant__ TileParams p) {
    extern __shared__ __align__(16) uint8_t smem[];
    __shared__ FastMat sM[kTileRunSegs];
    __shared__ TileSeg sS[kTileRunSegs];
    __shared__ int s_tp[kTileRunSegs + 1];  // first run tile of each segment
    __shared__ int s_cb[kTileRunSegs];      // byte offset of each segment's code rows
    __shared__ int s_nb[kTileRunSegs];      // byte offset of each segment's norms
    __shared__ int s_slot_seg[kTileSlots];  // a segment of each slot
    __shared__ int s_slot_g0[kTileSlots];   // first fragment group of each slot
    __shared__ __half s_lv[16];
    __shared__ float s_ginv[kTileSlots][kMaxFastB][kTileMaxNg];  // 1/sigma per slot, batch row, group
    __shared__ float s_alpha[kTileSlots][kMaxFastB];             // output scale per slot and batch row
    // The next launch on the stream may start its blocks as soon as this
    // grid's blocks are resident: its copies and table do not depend on this
    // grid, and it waits for this grid before it reads activations or writes
    // outputs.
    asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int s0 = p.cta_seg[blockIdx.x], nseg = p.cta_seg[blockIdx.x + 1] - s0;
    constexpr int kMatWords = sizeof(FastMat) / 4;
    for (int e = threadIdx.x; e < nseg * kMatWords; e += kThreads) {
        const int s = e / kMatWords, w = e - s * kMatWords;
        reinterpret_cast<uint32_t *>(&sM[s])[w] = reinterpret_cast<const uint32_t *>(&p.m[p.seg[s0 + s].mat])[w];
    }
    if (threadIdx.x < nseg) sS[threadIdx.x] = p.seg[s0 + threadIdx.x];
    __syncthreads();
    if (threadIdx.x == 0) {
        int tp = 0, cb = 0, nb = 0;
        for (int s = 0; s < nseg; ++s) {
            s_tp[s] = tp;
            s_cb[s] = cb;
            s_nb[s] = nb;
            tp += sS[s].ntiles;
            cb += 16 * sS[s].ntiles * sM[s].row_stride;
            nb += (32 * sS[s].ntiles * sM[s].ng + 15) / 16 * 16;
            s_slot_seg[sS[s].slot] = s;
        }
        s_tp[nseg] = tp;
        // slots are numbered in run order: slot k+1 starts after slot k's groups
        int g0 = 0;
        for (int sl = 0; sl < kTileSlots; ++sl) {
            s_slot_g0[sl] = g0;
            for (int s = 0; s < nseg; ++s)
                if (sS[s].slot == sl) {
                    g0 += sM[s].ng;
                    break;
                }
        }
    }
    if (threadIdx.x >= 32 && threadIdx.x < 48) s_lv[threadIdx.x - 32] = p.lut[p.m[p.seg[s0].mat].lut][threadIdx.x - 32];
    __syncthreads();
    const int kind = sM[0].kind;

    // ---- 1. code rows and norms of the run -> shared memory (16-byte
    // cp.async; rows past a matrix zero-filled), then the level table ----
    for (int s = 0; s < nseg; ++s) {
        const FastMat &M = sM[s];
        const int rowBytes = M.ng * (kind == 0 ? 32 : kind == 1 ? 64 : 16), cpr = rowBytes / 16, rs = M.row_stride;
        const int row0 = 16 * sS[s].tile0, nrows = 16 * sS[s].ntiles, valid = min(nrows, M.out - row0);
        uint8_t *dst = smem + p.smem_codes + s_cb[s];
        for (int c = threadIdx.x; c < nrows * cpr; c += kThreads) {
            const int r = c / cpr, k = c - r * cpr;
            const bool ok = r < valid;
            cp_async16(dst + (size_t)r * rs + 16 * k, M.codes + (size_t)(ok ? row0 + r : 0) * rowBytes + 16 * k,
                       ok ? 16 : 0);
        }
        const int nbytes = nrows * M.ng * 2, avail = valid * M.ng * 2;
        const uint8_t *src = reinterpret_cast<const uint8_t *>(M.norms + (size_t)row0 * M.ng);
        uint8_t *nd = smem + p.smem_norms + s_nb[s];
        for (int c = threadIdx.x; 16 * c < nbytes; c += kThreads) {
            const int left = avail - 16 * c, n = left >= 16 ? 16 : (left > 0 ? left : 0);
            cp_async16(nd + 16 * c, n ? src + 16 * c : src, n);
        }
    }
    asm volatile("cp.async.commit_group;\n" ::);
    build_level_table(kind, s_lv, smem + p.smem_tab);
    // the four 2-bit levels' low and high bytes, for the register expansion
    uint32_t llo = 0, lhi = 0;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        const uint32_t h = __half_as_ushort(s_lv[c]);
        llo |= (h & 0xffu) << (8 * c);
        lhi |= (h >> 8) << (8 * c);
    }

    // ---- 2. the activations, once the grid ahead of this one on the stream
    // (which may have written them) is complete: warp w rotates the
    // (slot, group) tasks w, w+8, ... for every batch row of the slot ----
    asm volatile("griddepcontrol.wait;\n" ::: "memory");
    int nslot = 0;
    for (int s = 0; s < nseg; ++s) nslot = max(nslot, sS[s].slot + 1);
    if (threadIdx.x < nslot * kMaxFastB) {
        const int sl = threadIdx.x / kMaxFastB, b = threadIdx.x % kMaxFastB;
        const FastMat &A = sM[s_slot_seg[sl]];
        s_alpha[sl][b] = b < A.B && A.xdt == CQ_X_I8 ? __fmul_rn(A.xs[b], kInvSqrt128) : kInvSqrt128;
    }
    {
        int task = 0;
        uint32_t *frag = reinterpret_cast<uint32_t *>(smem + p.smem_frag);
        for (int sl = 0; sl < nslot; ++sl) {
            const FastMat &A = sM[s_slot_seg[sl]];
            for (int g = 0; g < A.ng; ++g, ++task) {
                if (task % kWarps != warp) continue;
                uint32_t w[kFragWords];
#pragma unroll
                for (int f = 0; f < kFragWords; ++f) w[f] = 0u;
                for (int b = 0; b < A.B; ++b) {
                    float v[4];
                    uint32_t e[4];
                    load_x_bg(A, b, g, lane, v);
                    const float inv = rotate_regs(v, lane, e);
                    if (lane == 0) s_ginv[sl][b][g] = inv;
                    if (kind == 0) frag_from_lanes<true>(e, b, lane, w);
                    else frag_from_lanes<false>(e, b, lane, w);
                }
                uint4 *d4 = reinterpret_cast<uint4 *>(frag + (size_t)(s_slot_g0[sl] + g) * 32 * kFragWords);
#pragma unroll
                for (int i = 0; i < 4; ++i) d4[i * 32 + lane] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
            }
        }
    }
    asm volatile("cp.async.wait_all;\n" ::: "memory");
    __syncthreads();

    // ---- 3. products: warp w takes the run's tiles w, w+8, ... ----
    if (kind == 0) tile_run<0>(p, sM, sS, s_tp, s_cb, s_nb, s_slot_g0, s_ginv, s_alpha, smem, llo, lhi, nseg);
    else if (kind == 1) tile_run<1>(p, sM, sS, s_tp, s_cb, s_nb, s_slot_g0, s_ginv, s_alpha, smem, llo, lhi, nseg);
    else tile_run<2>(p, sM, sS, s_tp, s_cb, s_nb, s_slot_g0, s_ginv, s_alpha, smem, llo, lhi, nseg);
}

// ------------------------------------------------- wide inputs, streamed --
// For inputs of 16 to 32 groups: one block per SM walks an equal run of the
// call's 16-row tiles (runs cross matrix boundaries). Per matrix it meets, it
// builds the level table (when the codebook changes) and rotates the
// activation once; then the code rows of each tile stream through three
// shared-memory stages (16-byte cp.async, two tiles ahead), every warp takes
// every eighth group of the tile, and the partial sums meet in shared memory.
constexpr int kStreamMats = 200;
constexpr int kStreamStages = 3;

struct StreamParams {
    int n_mats, total_tiles;
    int tiles_before[kStreamMats + 1];  // first tile of each matrix in the flat order
    int smem_tab, smem_terms, smem_frag, smem_red, smem_stage, stage_bytes, n_stages;
    __half lut[kStreamMats][16];
    FastMat m[kStreamMats];
};

// G64: groups of 64 (two norms per 128-span and two MMA chains).
template <bool G64>
__global__ void __launch_bounds__(kThreads, 1) gemv_stream_kernel(const __grid_constant__ StreamParams p) {
    extern __shared__ __align__(16) uint8_t smem[];
    __shared__ FastMat sM;
    __shared__ __half s_lv[16];
    __shared__ float ginv[kMaxFastB * kMaxFastNg];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, gq = lane >> 2, t = lane & 3;
    uint32_t *frag = reinterpret_cast<uint32_t *>(smem + p.smem_frag);
    float *red = reinterpret_cast<float *>(smem + p.smem_red);  // [kWarps][16 rows][kMaxFastB]
    const uint2 *tab2 = reinterpret_cast<const uint2 *>(smem + p.smem_tab) + (lane & 15);
    const uint32_t *tab4 = reinterpret_cast<const uint32_t *>(smem + p.smem_tab) + lane;

    const int T = p.total_tiles, G = gridDim.x, bid = blockIdx.x;
    const int x_end = (int)(((long long)(bid + 1) * T) / G);
    int cur_lut = -1;
    for (int x = (int)(((long long)bid * T) / G); x < x_end;) {
        int lo = 0, hi = p.n_mats - 1;  // the matrix holding tile x
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (p.tiles_before[mid] <= x) lo = mid;
            else hi = mid - 1;
        }
        const int mi = lo, seg_end = min(x_end, p.tiles_before[mi + 1]);
        __syncthreads();  // the previous segment is done with sM, the table, the fragments and the stages
        if (threadIdx.x < (int)(sizeof(FastMat) / 4))
            reinterpret_cast<uint32_t *>(&sM)[threadIdx.x] = reinterpret_cast<const uint32_t *>(&p.m[mi])[threadIdx.x];
        else if (threadIdx.x >= 128 && threadIdx.x < 144)
            s_lv[threadIdx.x - 128] = p.lut[mi][threadIdx.x - 128];
        __syncthreads();
        const FastMat &M = sM;
        const int ng = M.ng, B = M.B, kind = M.kind, rs = M.row_stride;
        const int nn = G64 ? 2 * ng : ng;  // norms per row
        const float gscale = G64 ? 0.125f : kInvSqrt128;  // 1/sqrt(group)
        const int rowBytes = ng * (kind == 0 ? 32 : kind == 1 ? 64 : kind == 3 ? 48 : 16), cpr = rowBytes / 16;
        const int t0 = x - p.tiles_before[mi], ntile = seg_end - x;  // first tile of the matrix, tiles here
        if (M.lut != cur_lut) {
            build_level_table<true>(kind, s_lv, smem + p.smem_tab);
            cur_lut = M.lut;
        }
        rotate_activation<G64>(M, smem + p.smem_terms, frag, ginv);

        // copies of the segment's i-th tile into stage i % NS: its code rows
        // (rows past the matrix zero-filled), then its norms
        const int NS = p.n_stages;
        auto issue = [&](int i) {
            if (i < ntile) {
                uint8_t *st = smem + p.smem_stage + (i % NS) * p.stage_bytes;
                const int row0 = 16 * (t0 + i), valid = min(16, M.out - row0);
                for (int c = threadIdx.x; c < 16 * cpr; c += kThreads) {
                    const int r = c / cpr, k = c - r * cpr;
                    const bool ok = r < valid;
                    cp_async16(st + r * rs + 16 * k, M.codes + (size_t)(ok ? row0 + r : 0) * rowBytes + 16 * k,
                               ok ? 16 : 0);
                }
                const int nbytes = 16 * nn * 2, avail = valid * nn * 2;
                const uint8_t *src = reinterpret_cast<const uint8_t *>(M.norms + (size_t)row0 * nn);
                for (int c = threadIdx.x; 16 * c < nbytes; c += kThreads) {
                    const int left = avail - 16 * c, n = left >= 16 ? 16 : (left > 0 ? left : 0);
                    cp_async16(st + 16 * rs + 16 * c, n ? src + 16 * c : src, n);
                }
            }
            asm volatile("cp.async.commit_group;\n" ::);
        };
        for (int k = 0; k + 1 < NS; ++k) issue(k);
        const bool live = gq < 2 * B;  // this lane's B column belongs to a batch row
        for (int i = 0; i < ntile; ++i) {
            issue(i + NS - 1);
            // tile i landed (NS - 1 younger groups may still fly); the fragments are complete
            if (NS == 4) asm volatile("cp.async.wait_group 3;\n" ::: "memory");
            else asm volatile("cp.async.wait_group 2;\n" ::: "memory");
            __syncthreads();
            const uint8_t *sc = smem + p.smem_stage + (i % NS) * p.stage_bytes;
            const __half *sn = reinterpret_cast<const __half *>(sc + 16 * rs);
            float acc[4] = {0.f, 0.f, 0.f, 0.f};
            for (int g = warp; g < ng; g += kWarps) {
                uint32_t fr[kFragWords];
                const uint4 *fl = reinterpret_cast<const uint4 *>(frag + (size_t)g * 32 * kFragWords) + lane;
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const uint4 v = live ? fl[32 * k] : make_uint4(0, 0, 0, 0);
                    fr[4 * k] = v.x, fr[4 * k + 1] = v.y, fr[4 * k + 2] = v.z, fr[4 * k + 3] = v.w;
                }
                const float inv = t < B ? ginv[t * ng + g] : 0.0f;
                if (G64) {
                    const float n0 = __half2float(sn[gq * nn + 2 * g]) * inv;
                    const float n1 = __half2float(sn[(gq + 8) * nn + 2 * g]) * inv;
                    const float h0 = __half2float(sn[gq * nn + 2 * g + 1]) * inv;
                    const float h1 = __half2float(sn[(gq + 8) * nn + 2 * g + 1]) * inv;
                    const int gb = g * (kind == 0 ? 32 : kind == 1 ? 64 : kind == 3 ? 48 : 16);
                    const uint8_t *r0 = sc + gq * rs + gb, *r1 = sc + (gq + 8) * rs + gb;
                    const void *tab = smem + p.smem_tab;
                    if (kind == 2) lut_group64<2>(acc, r0, r1, tab, fr, n0, n1, h0, h1);
                    else if (kind == 0) lut_group64<0>(acc, r0, r1, tab, fr, n0, n1, h0, h1);
                    else lut_group64<1>(acc, r0, r1, tab, fr, n0, n1, h0, h1);
                    continue;
                }
                const float n0 = __half2float(sn[gq * ng + g]) * inv, n1 = __half2float(sn[(gq + 8) * ng + g]) * inv;
                if (kind == 3) {
                    uint32_t w0[4], w1[4];
                    load3(sc + gq * rs + g * 48 + 12 * t, w0);
                    load3(sc + (gq + 8) * rs + g * 48 + 12 * t, w1);
                    lut3_group(acc, w0, w1, tab4, fr, n0, n1);
                } else if (kind == 2) {
                    const uint32_t c0 = *reinterpret_cast<const uint32_t *>(sc + gq * rs + g * 16 + 4 * t);
                    const uint32_t c1 = *reinterpret_cast<const uint32_t *>(sc + (gq + 8) * rs + g * 16 + 4 * t);
                    lut1_group(acc, c0, c1, tab2, fr, n0, n1);
                } else if (kind == 0) {
                    const uint2 c0 = *reinterpret_cast<const uint2 *>(sc + gq * rs + g * 32 + 8 * t);
                    const uint2 c1 = *reinterpret_cast<const uint2 *>(sc + (gq + 8) * rs + g * 32 + 8 * t);
                    lut2_group(acc, c0, c1, tab2, fr, n0, n1);
                } else {
                    const uint4 c0 = *reinterpret_cast<const uint4 *>(sc + gq * rs + g * 64 + 16 * t);
                    const uint4 c1 = *reinterpret_cast<const uint4 *>(sc + (gq + 8) * rs + g * 64 + 16 * t);
                    lut4_group(acc, c0, c1, tab4, fr, n0, n1);
                }
            }
            if (t < B) {  // columns 2t, 2t+1: hi and lo terms of batch row t
                red[(warp * 16 + gq) * kMaxFastB + t] = acc[0] + acc[1];
                red[(warp * 16 + gq + 8) * kMaxFastB + t] = acc[2] + acc[3];
            }
            __syncthreads();  // partial sums complete; the stage may be refilled
            if (threadIdx.x < 16 * B) {
                const int r = threadIdx.x / B, b = threadIdx.x - r * B, row = 16 * (t0 + i) + r;
                float sum = 0.0f;
#pragma unroll
                for (int w = 0; w < kWarps; ++w) sum += red[(w * 16 + r) * kMaxFastB + b];
                if (row < M.out) {
                    const float ab = M.xdt == CQ_X_I8 ? __fmul_rn(M.xs[b], gscale) : gscale;
                    M.y[(size_t)b * M.out + row] = sum * ab;
                }
            }
        }
        asm volatile("cp.async.wait_all;\n" ::: "memory");
        x = seg_end;
    }
}

}  // namespace

bool gemv_stream_eligible(const cq_gemv_desc &d) {
    const int ng = in_padded(d.in) / kGroup, W = width_of(d.bits);
    // groups of 64 in whole 128-spans only
    const bool grp = d.group == kGroup || (d.group == kGroup64 && d.in % kGroup == 0 && W != 3);
    return grp && d.out > 0 && (W >= 1 && W <= 4) && d.B <= kMaxFastB && ng >= 16 && ng <= kMaxFastNg;
}

int launch_gemv_stream_g(const cq_gemv_desc *d, const int *idx, int n, bool g64, void *stream);

int launch_gemv_stream(const cq_gemv_desc *d, const int *idx_all, int n_all, void *stream) {
    // groups of 128 and of 64 go to separate instances
    int i128[CQ_MAX_GROUPED], i64[CQ_MAX_GROUPED], n128 = 0, n64 = 0;
    for (int i = 0; i < n_all; ++i) {
        if (d[idx_all[i]].group == kGroup64) i64[n64++] = idx_all[i];
        else i128[n128++] = idx_all[i];
    }
    for (int pass = 0; pass < 2; ++pass) {
        const int rc = launch_gemv_stream_g(d, pass ? i64 : i128, pass ? n64 : n128, pass == 1, stream);
        if (rc) return rc;
    }
    return CQ_OK;
}

int launch_gemv_stream_g(const cq_gemv_desc *d, const int *idx, int n, bool g64, void *stream) {
    static thread_local StreamParams p;  // large: off the stack, one per host thread
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    for (int base = 0; base < n; base += kStreamMats) {
        const int cnt = std::min(kStreamMats, n - base);
        int tiles = 0, ng_max = 0, row_max = 0;
        for (int j = 0; j < cnt; ++j) {
            const cq_gemv_desc &D = d[idx[base + j]];
            const int ip = in_padded(D.in), W = width_of(D.bits), ng = ip / kGroup;
            FastMat &M = p.m[j];
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
            M.kind = W == 2 ? 0 : W == 4 ? 1 : W == 3 ? 3 : 2;
            M.lut = j;  // one table per matrix; rebuilt only when it changes along a block's run
            M.tiles = M.kchunks = M.item0 = 0;
            const int rowBytes = ng * (M.kind == 0 ? 32 : M.kind == 1 ? 64 : M.kind == 3 ? 48 : 16);
            const int want = M.kind == 0 ? 32 : M.kind == 1 ? 64 : M.kind == 3 ? 48 : 16;  // see launch_gemv_fast
            M.row_stride = rowBytes + (((want - rowBytes) % 128) + 128) % 128;
            float lv[16];
            level_table(D.bits, D.codebook, lv);
            for (int k = 0; k < 16; ++k) p.lut[j][k] = __float2half_rn(lv[k]);
            // the same levels as the previous matrix: keep its table
            if (j > 0) {
                bool same = p.m[j - 1].kind == M.kind;
                for (int k = 0; k < 16; ++k) same &= __half_as_ushort(p.lut[j][k]) == __half_as_ushort(p.lut[j - 1][k]);
                if (same) M.lut = p.m[j - 1].lut;
            }
            p.tiles_before[j] = tiles;
            tiles += (D.out + 15) / 16;
            ng_max = std::max(ng_max, ng);
            row_max = std::max(row_max, M.row_stride);
        }
        p.tiles_before[cnt] = tiles;
        p.n_mats = cnt;
        p.total_tiles = tiles;
        size_t off = 0;
        auto place = [&](int &field, size_t bytes) {
            field = (int)off;
            off += (bytes + 15) / 16 * 16;
        };
        place(p.smem_tab, 256 * 32 * sizeof(uint32_t));
        place(p.smem_terms, (size_t)kWarps * kMaxFastB * kGroup * sizeof(uint32_t));
        place(p.smem_frag, (size_t)ng_max * 32 * kFragWords * sizeof(uint32_t));
        place(p.smem_red, (size_t)kWarps * 16 * kMaxFastB * sizeof(float));
        p.stage_bytes = (16 * row_max + 32 * ng_max * (g64 ? 2 : 1) + 15) / 16 * 16;
        p.n_stages = kStreamStages;
        place(p.smem_stage, (size_t)p.n_stages * p.stage_bytes);
        const size_t smem = off;
        {
            const int rc = ensure_smem(g64 ? reinterpret_cast<const void *>(gemv_stream_kernel<true>)
                                           : reinterpret_cast<const void *>(gemv_stream_kernel<false>),
                                       smem);
            if (rc) return rc;
        }
        const int grid = std::min(tiles, sm_count());
        if (g64) gemv_stream_kernel<true><<<grid, kThreads, smem, st>>>(p);
        else gemv_stream_kernel<false><<<grid, kThreads, smem, st>>>(p);
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return set_error(CQ_ERR_CUDA, "streamed gemv launch: %s", cudaGetErrorString(e));
    }
    return CQ_OK;
}

bool gemv_fast_eligible(const cq_gemv_desc &d) {
    const int ng = in_padded(d.in) / kGroup;
    if (d.in <= 0 || d.out <= 0 || d.group != kGroup) return false;
    const int W = width_of(d.bits);
    return (W == 1 || W == 2 || W == 4) && d.B <= kMaxFastB && ng <= kTileMaxNg && !gemv_stream_eligible(d);
}

namespace {

int tile_kind(int W) { return W == 2 ? 0 : W == 4 ? 1 : 2; }
int tile_gbytes(int kind) { return kind == 0 ? 32 : kind == 1 ? 64 : 16; }

// Shared-memory row stride of a code row: the 2-bit path reads 8 bytes per
// lane (the rows of a half-warp start 8 banks apart), the 4-bit path 16
// bytes (the rows of a quarter-warp 16 banks apart), the 1-bit path 4 bytes
// (the warp's eight rows 4 banks apart).
int tile_row_stride(int kind, int ng) {
    const int rowBytes = ng * tile_gbytes(kind), want = tile_gbytes(kind);
    return rowBytes + (((want - rowBytes) % 128) + 128) % 128;
}

// The level table by code of a descriptor (ternary crumbs sign-extend).
void tile_levels(const cq_gemv_desc &D, __half lut[16]) {
    for (int j = 0; j < 16; ++j) lut[j] = __float2half_rn(0.0f);
    if (D.bits == 5) {
        const float c = D.codebook[2];
        lut[1] = __float2half_rn(c);
        lut[2] = __float2half_rn(-2.0f * c);
        lut[3] = __float2half_rn(-c);
    } else {
        for (int j = 0; j < levels_of(D.bits); ++j) lut[j] = __float2half_rn(D.codebook[j]);
    }
}

// One launch being assembled: matrices, runs (one per CTA) and their
// segments, and the shared-memory maxima over its runs.
struct TileBuild {
    TileParams *p;
    int nm = 0, nseg = 0, ncta = 0, nlut = 0;
    size_t codes_max = 0, norms_max = 0;
    bool table = false;  // some run needs a 32 KB level table
    // the open run
    int run_seg0 = 0, run_tiles = 0, run_kind = -1, run_lut = -1, run_nslot = 0, run_groups = 0;
    size_t run_bytes = 0, run_codes = 0, run_norms = 0;
    const cq_gemv_desc *run_key = nullptr;  // descriptor of the open slot's activation
};

bool same_activation(const cq_gemv_desc *a, const cq_gemv_desc *b) {
    return a && b && a->x == b->x && a->x_scale == b->x_scale && a->B == b->B && a->x_dtype == b->x_dtype &&
           a->in == b->in;
}

void close_run(TileBuild &L) {
    if (L.nseg == L.run_seg0) return;
    L.p->cta_seg[++L.ncta] = L.nseg;
    L.codes_max = std::max(L.codes_max, L.run_codes);
    L.norms_max = std::max(L.norms_max, L.run_norms);
    if (L.run_kind != 2) L.table = true;
    L.run_seg0 = L.nseg;
    L.run_tiles = 0;
    L.run_kind = L.run_lut = -1;
    L.run_nslot = L.run_groups = 0;
    L.run_bytes = L.run_codes = L.run_norms = 0;
    L.run_key = nullptr;
}

int tile_flush(TileBuild &L, cudaStream_t st) {
    close_run(L);
    if (L.ncta) {
        TileParams &p = *L.p;
        size_t off = 0;
        auto place = [&](int &field, size_t bytes) {
            field = (int)off;
            off += (bytes + 15) / 16 * 16;
        };
        place(p.smem_tab, L.table ? 256 * 32 * sizeof(uint32_t) : 16 * 16 * sizeof(uint2));
        place(p.smem_codes, L.codes_max);
        place(p.smem_norms, L.norms_max);
        place(p.smem_frag, (size_t)kTileFragGroups * 32 * kFragWords * sizeof(uint32_t));
        const size_t smem = off;
        const int rc = ensure_smem(reinterpret_cast<const void *>(gemv_tile_kernel), smem);
        if (rc) return rc;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)L.ncta);
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = smem;
        cfg.stream = st;
        cudaLaunchAttribute at[1];
        at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        at[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = at;
        cfg.numAttrs = 1;
        cudaLaunchKernelEx(&cfg, gemv_tile_kernel, p);
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return set_error(CQ_ERR_CUDA, "tile gemv launch: %s", cudaGetErrorString(e));
    }
    L.nm = L.nseg = L.ncta = L.nlut = 0;
    L.run_seg0 = 0;
    L.codes_max = L.norms_max = 0;
    L.table = false;
    L.p->cta_seg[0] = 0;
    return CQ_OK;
}

}  // namespace

int launch_gemv_fast(const cq_gemv_desc *d, const int *idx, int n, void *stream) {
    static thread_local TileParams p;  // large: off the stack, one per host thread
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    TileBuild L;
    L.p = &p;
    p.cta_seg[0] = 0;
    // the byte target of a run: the launch's bytes (padded code rows and
    // norms) spread over two CTAs per SM, at least kMinTiles tiles
    constexpr int kMinTiles = 4;
    size_t total = 0;
    for (int ii = 0; ii < n; ++ii) {
        const cq_gemv_desc &D = d[idx[ii]];
        const int ng = in_padded(D.in) / kGroup, kind = tile_kind(width_of(D.bits));
        total += (size_t)((D.out + 15) / 16) * (16 * tile_row_stride(kind, ng) + 32 * ng);
    }
    const size_t target = std::max<size_t>(1, total / (2 * (size_t)sm_count()) * 100 / 94);
    for (int ii = 0; ii < n; ++ii) {
        const cq_gemv_desc &D = d[idx[ii]];
        const int ng = in_padded(D.in) / kGroup, W = width_of(D.bits), kind = tile_kind(W);
        const int rs = tile_row_stride(kind, ng), tiles = (D.out + 15) / 16;
        const size_t tile_codes = 16 * (size_t)rs, tile_norms = 32 * (size_t)ng;
        __half lut[16];
        tile_levels(D, lut);
        int mi = -1, li = -1;
        for (int tl = 0; tl < tiles; ++tl) {
            // the matrix and its level table in the current launch (again
            // after a flush)
            if (mi < 0) {
                if (L.nm == kTileMaxMats) {
                    const int rc = tile_flush(L, st);
                    if (rc) return rc;
                }
                li = -1;
                for (int j = 0; j < L.nlut; ++j) {
                    bool same = true;
                    for (int k = 0; k < 16; ++k) same &= __half_as_ushort(p.lut[j][k]) == __half_as_ushort(lut[k]);
                    if (same) li = j;
                }
                if (li < 0) {
                    if (L.nlut == kMaxLuts) {
                        const int rc = tile_flush(L, st);
                        if (rc) return rc;
                    }
                    for (int k = 0; k < 16; ++k) p.lut[L.nlut][k] = lut[k];
                    li = L.nlut++;
                }
                FastMat &M = p.m[L.nm];
                M.codes = D.blob;
                M.norms = reinterpret_cast<const __half *>(D.blob + (size_t)D.out * in_padded(D.in) * W / 8);
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
                M.lut = li;
                M.tiles = M.kchunks = M.item0 = 0;
                M.row_stride = rs;
                mi = L.nm++;
            }
            // does this tile start a new run?
            const bool new_slot = !same_activation(L.run_key, &D);
            bool cut = L.run_tiles > 0 &&
                       (kind != L.run_kind || li != L.run_lut || L.run_codes + tile_codes > (size_t)kTileCodeBudget ||
                        (L.run_bytes + tile_codes + tile_norms > target && L.run_tiles >= kMinTiles) ||
                        (new_slot && (L.run_nslot == kTileSlots || L.run_groups + ng > kTileFragGroups)));
            const bool new_seg = cut || L.nseg == L.run_seg0 || p.seg[L.nseg - 1].mat != mi;
            if (!cut && new_seg && L.nseg - L.run_seg0 == kTileRunSegs) cut = true;
            if (cut) {
                close_run(L);
                if (L.ncta == kTileMaxCtas || L.nseg + kTileRunSegs > kTileMaxSegs) {
                    const int rc = tile_flush(L, st);
                    if (rc) return rc;
                    mi = -1;
                    --tl;  // add this tile again, to the new launch
                    continue;
                }
            }
            if (L.run_tiles == 0) {
                L.run_kind = kind;
                L.run_lut = li;
            }
            if (!same_activation(L.run_key, &D)) {
                L.run_key = &D;
                ++L.run_nslot;
                L.run_groups += ng;
            }
            if (cut || new_seg) {
                TileSeg &S = p.seg[L.nseg++];
                S.mat = mi;
                S.tile0 = tl;
                S.ntiles = 0;
                S.slot = L.run_nslot - 1;
                L.run_norms = (L.run_norms + 15) / 16 * 16;  // each segment's norms start 16-byte aligned
            }
            ++p.seg[L.nseg - 1].ntiles;
            ++L.run_tiles;
            L.run_bytes += tile_codes + tile_norms;
            L.run_codes += tile_codes;
            L.run_norms += tile_norms;
        }
    }
    return tile_flush(L, st);
}

}  // namespace cq
