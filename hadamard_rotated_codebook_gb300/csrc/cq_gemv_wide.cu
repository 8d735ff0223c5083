// cq_gemv_wide.cu -- tensor-core GEMV over CQ-packed weights for wide
// inputs (16 groups and more at group 128, groups of 64 in whole 128-spans)
// and for batches of 5 to 16.
//
// Per group g of 128 inputs the product is the rotated-domain identity
// (OpenNeedle docs/reference.md; "The .cact archive and Cactus Quants",
// "Reconstructing one group"):
//     y[b][o] = sum_g n[o][g] * sum_k c[q[o,g,k]] * z[b,g,k],   z = H x (per group).
//
// Two kinds of products:
//  - gemv_split_kernel (further below), batches of 1 to 4 with 1- to 4-bit
//    codes at group 128 and 1-, 2- and 4-bit codes at group 64: one launch
//    per call. Each block
//    rotates the activation groups of its (matrix, k-slice) pairs itself
//    (one warp per group and batch row, the FWHT in registers, fp16 terms
//    written straight into the MMA B-fragment layout in shared memory) and
//    its warps stream (matrix, k-slice, 16-row tile) units through private
//    TMA pipelines.
//  - gemv_wide_kernel, the rest (batches of 5 to 16): behind a
//    rotation launch, act_frag_kernel, which rotates every distinct
//    activation of the call once into a workspace in the same fragment
//    layout, with 1/sigma per (batch row, group). One block per SM walks an
//    equal run of the call's 16-row tiles. Before it waits for the rotation
//    it builds its level table and starts its code copies; then it copies
//    the fragments of its matrix's activation into shared memory once, and
//    streams the tiles through shared-memory stages in slices of about 512
//    code bytes per row. The warps split a slice's groups: each expands its
//    groups' code bytes to fp16 levels through the replicated byte -> levels
//    table (the A operand of mma.sync m16n8k16, fp32 accumulation) and
//    multiplies them with the fragments of every batch row; a tile's partial
//    sums meet in shared memory.
//
// Precision. Batches of 1 to 4 carry z as fp16 hi + lo terms (two MMA
// columns per batch row, z to ~2^-22 relative). Batches of 5 to 16 carry z as
// one fp16 term (one column per batch row, relative error <= 2^-11, the same
// order as the fp16 rounding of the levels), which halves the MMAs; both are
// far inside the product tolerance |y - y_ref| <= 2e-3 sum |w||x|.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <vector>

#include "cq_internal.h"

namespace cq {

namespace {

constexpr int kWThreads = 256;  // the rotation kernel
constexpr int kWWarps = kWThreads / 32;
constexpr int kWGThreads = 512;  // the product kernel: 16 warps per SM
constexpr int kWGWarps = kWGThreads / 32;
constexpr int kWMaxMats = 128;   // matrices per main launch
constexpr int kWMaxActs = 128;   // activations per rotation launch
constexpr int kWMaxB = 16;
constexpr int kWMaxStages = 16;  // shared-memory stages of code slices (as many as fit)
constexpr int kWFragBudget = 136 * 1024;  // shared-memory bytes of one activation's fragments and 1/sigma
constexpr float kWInvSqrt128 = 0.08838834764831845f;

// ------------------------------------------------------------- rotation --
struct WAct {
    const void *x;     // [B][in], fp32 or int8
    const float *xs;   // [B] for int8
    int xdt, in, ng, B;
    int g64;           // groups of 64 (told apart from the same x read at group 128)
    int cols;          // fragment columns: 2B (hi, lo) for B <= 4, else 8 * ceil(B / 8) (hi)
    long long frag;    // word offset of the fragments in the workspace: [g][4 k][cols][4 t][4 words]
    long long ginv;    // float offset of 1/sigma [B][ng] in the workspace
};

struct WActParams {
    int n;
    int task0[kWMaxActs + 1];  // first warp task of each activation
    uint32_t *frag;
    float *ginv;
    WAct a[kWMaxActs];
};

__device__ __forceinline__ float w_pow2_scale(float amax, float lim) {
    if (!(amax > 0.0f)) return 1.0f;
    const float q = __fdiv_rn(lim, amax);
    const int E = min(max((__float_as_int(q) >> 23) & 0xff, 1), 254);
    float s = __int_as_float(E << 23);        // 2^(E-127) <= q
    if (__fmul_rn(amax, s) > lim) s *= 0.5f;  // guard the rounding of q
    return s;
}

// One warp per (activation, group, batch row): the FWHT of the row's group
// (lane l holds positions 4l .. 4l+3), then the fragment words of its
// column(s). Word f = 2j + h of MMA lane (gq, t) holds positions
// 32t + 4j + 2h + {0, 1}: lane l = 8t + j owns exactly the positions of words
// 2j and 2j + 1 of lane t. Words are stored 4 to a 16-byte unit, the units of
// one k = f / 4 consecutive over (column, t), so that a warp's 16-byte loads
// of them are free of bank conflicts. (This launch serves the sliced
// kernel; the split products rotate their activations themselves.)
__global__ void __launch_bounds__(kWThreads) act_frag_kernel(const __grid_constant__ WActParams p) {
    // the GEMV launched after this one may start its prologue at once
    asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
    const int lane = threadIdx.x & 31;
    const int task = blockIdx.x * kWWarps + (threadIdx.x >> 5);
    if (task >= p.task0[p.n]) return;
    int lo = 0, hi = p.n - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (p.task0[mid] <= task) lo = mid;
        else hi = mid - 1;
    }
    const WAct &A = p.a[lo];
    const int local = task - p.task0[lo], g = local / A.B, b = local - g * A.B;
    float v[4];
    const int col0 = g * kGroup + 4 * lane;
    if (A.xdt == CQ_X_I8) {
        const int8_t *xq = static_cast<const int8_t *>(A.x) + (size_t)b * A.in;
#pragma unroll
        for (int i = 0; i < 4; ++i) v[i] = col0 + i < A.in ? (float)xq[col0 + i] : 0.0f;
    } else {
        const float *xf = static_cast<const float *>(A.x) + (size_t)b * A.in;
#pragma unroll
        for (int i = 0; i < 4; ++i) v[i] = col0 + i < A.in ? xf[col0 + i] : 0.0f;
    }
    {
        const float a0 = v[0] + v[1], a1 = v[0] - v[1], a2 = v[2] + v[3], a3 = v[2] - v[3];
        v[0] = a0 + a2;
        v[1] = a1 + a3;
        v[2] = a0 - a2;
        v[3] = a1 - a3;
    }
#pragma unroll
    for (int m = 1; m < 32; m <<= 1)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float o = __shfl_xor_sync(0xffffffffu, v[i], m);
            v[i] = (lane & m) ? o - v[i] : v[i] + o;
        }
    // int8 activations give integers |z| <= 128 * 128, which hi + lo carry
    // exactly unscaled; otherwise scale by a power of two to |sigma z| <= 2^14
    float sigma = 1.0f;
    if (A.xdt != CQ_X_I8) {
        float mx = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
#pragma unroll
        for (int m = 16; m; m >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, m));
        sigma = w_pow2_scale(mx, 16384.0f);
    }
    uint32_t hi16[4], lo16[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float x = __fmul_rn(v[i], sigma);
        const __half h = __float2half_rn(x);
        const __half l = __float2half_rn(__fsub_rn(x, __half2float(h)));
        hi16[i] = __half_as_ushort(h);
        lo16[i] = __half_as_ushort(l);
    }
    const int t = lane >> 3, j = lane & 7;
    const bool hilo = A.B <= 4;
    uint32_t *base = p.frag + A.frag;
    const int k = j >> 1, w2 = 2 * (j & 1);  // words 2j, 2j+1: unit k, offset w2
    {
        const int c = hilo ? 2 * b : b;  // the column of the hi terms
        uint2 *dst = reinterpret_cast<uint2 *>(base + ((((size_t)g * 4 + k) * A.cols + c) * 4 + t) * 4 + w2);
        *dst = make_uint2(hi16[0] | (hi16[1] << 16), hi16[2] | (hi16[3] << 16));
    }
    if (hilo) {
        uint2 *dst = reinterpret_cast<uint2 *>(base + ((((size_t)g * 4 + k) * A.cols + 2 * b + 1) * 4 + t) * 4 + w2);
        *dst = make_uint2(lo16[0] | (lo16[1] << 16), lo16[2] | (lo16[3] << 16));
    }
    if (lane == 0) p.ginv[A.ginv + (size_t)b * A.ng + g] = 1.0f / sigma;
}

// ------------------------------------------------------------------ GEMV --
struct WMat {
    const uint8_t *codes;
    const __half *norms;
    float *y;
    const float *xs;
    int out, ng, B, xdt, kind, lut;
    int act;   // index of its activation (fragments, 1/sigma)
    int gs;    // groups per slice
    int rs;    // shared-memory row stride of a slice (bytes)
};

struct WParams {
    int n_mats, total_tiles;
    int tiles_before[kWMaxMats + 1];           // first flat tile of each matrix
    int smem_frag, smem_stage, smem_red, stage_bytes;  // byte offsets (the table is at offset 0)
    int n_stages;
    unsigned int *status;                      // device status word (bounded waits)
    const uint32_t *frag;                      // the rotation's workspace
    const float *ginv;
    long long act_frag[kWMaxMats];             // word offset of each matrix's fragments
    long long act_ginv[kWMaxMats];             // float offset of each matrix's 1/sigma
    int act_cols[kWMaxMats];
    __half lut[kMaxLuts][16];
    WMat m[kWMaxMats];
};

static_assert(sizeof(WParams) <= 32000, "kernel parameter block");

__device__ __forceinline__ void w_mma(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void w_cp16(void *dst, const void *src, int src_bytes) {
    const uint32_t d = (uint32_t)__cvta_generic_to_shared(dst);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(d), "l"(src), "r"(src_bytes) : "memory");
}

// Level tables in shared memory at `tab`, replicated so that each lane reads
// its own copy (conflict-free whatever the codes): 2-bit codes a byte -> the
// fp16 levels of its four 2-bit fields (16 copies of 8 bytes), 4-bit codes a
// byte -> two levels (32 copies of 4 bytes), 1-bit codes a nibble -> four
// levels (16 copies), 3-bit codes a 6-bit pair -> two levels (32 copies).
__device__ void w_build_table(int kind, const __half *lv, uint8_t *tab) {
    auto h = [&](int c) { return (uint32_t)__half_as_ushort(lv[c]); };
    if (kind == 0) {
        uint2 *t = reinterpret_cast<uint2 *>(tab);
        for (int e = threadIdx.x; e < 256 * 16; e += kWGThreads) {
            const int v = e >> 4;
            t[e] = make_uint2(h(v & 3) | (h((v >> 2) & 3) << 16), h((v >> 4) & 3) | (h(v >> 6) << 16));
        }
    } else if (kind == 1) {
        uint32_t *t = reinterpret_cast<uint32_t *>(tab);
        for (int e = threadIdx.x; e < 256 * 32; e += kWGThreads) {
            const int v = e >> 5;
            t[e] = h(v & 15) | (h(v >> 4) << 16);
        }
    } else if (kind == 2) {
        uint2 *t = reinterpret_cast<uint2 *>(tab);
        for (int e = threadIdx.x; e < 16 * 16; e += kWGThreads) {
            const int v = e >> 4;
            t[e] = make_uint2(h(v & 1) | (h((v >> 1) & 1) << 16), h((v >> 2) & 1) | (h(v >> 3) << 16));
        }
    } else {
        uint32_t *t = reinterpret_cast<uint32_t *>(tab);
        for (int e = threadIdx.x; e < 64 * 32; e += kWGThreads) {
            const int v = e >> 5;
            t[e] = h(v & 7) | (h(v >> 3) << 16);
        }
    }
}

// The code words of one group for this lane: rows gq (r0) and gq + 8 (r1) of
// a tile, the lane's share of the group's bytes (2-bit: 8 bytes, 4-bit: 16,
// 1-bit: 4, 3-bit: 12).
struct WCodes {
    uint32_t r[4], s[4];
};

template <int KIND>
__device__ __forceinline__ void w_load(const uint8_t *r0, const uint8_t *r1, int t, WCodes &c) {
    if (KIND == 0) {
        const uint2 a = *reinterpret_cast<const uint2 *>(r0 + 8 * t), b = *reinterpret_cast<const uint2 *>(r1 + 8 * t);
        c.r[0] = a.x, c.r[1] = a.y, c.s[0] = b.x, c.s[1] = b.y;
    } else if (KIND == 1) {
        const uint4 a = *reinterpret_cast<const uint4 *>(r0 + 16 * t), b = *reinterpret_cast<const uint4 *>(r1 + 16 * t);
        c.r[0] = a.x, c.r[1] = a.y, c.r[2] = a.z, c.r[3] = a.w, c.s[0] = b.x, c.s[1] = b.y, c.s[2] = b.z, c.s[3] = b.w;
    } else if (KIND == 2) {
        c.r[0] = *reinterpret_cast<const uint32_t *>(r0 + 4 * t), c.s[0] = *reinterpret_cast<const uint32_t *>(r1 + 4 * t);
    } else {
        const uint32_t *q0 = reinterpret_cast<const uint32_t *>(r0 + 12 * t), *q1 = reinterpret_cast<const uint32_t *>(r1 + 12 * t);
        c.r[0] = q0[0], c.r[1] = q0[1], c.r[2] = q0[2], c.r[3] = 0u;
        c.s[0] = q1[0], c.s[1] = q1[1], c.s[2] = q1[2], c.s[3] = 0u;
    }
}

// The A fragment of MMA nu (positions 32t + 4nu .. +3 of the group):
// {row gq positions 0-1, row gq+8 positions 0-1, row gq positions 2-3,
// row gq+8 positions 2-3}, through the replicated level tables. For 2-bit
// and 1-bit codes one lookup serves both rows: the index is made of row gq's
// codes of a position pair (low bits) and row gq+8's codes of the same pair
// (high bits), and the entry's two words are then fragment registers a0, a1
// (or a2, a3) as they stand.
template <int KIND>
__device__ __forceinline__ void w_decode(const WCodes &c, int nu, const uint8_t *tab, int lane, uint32_t (&a)[4]) {
    if (KIND == 0) {  // byte nu of the lane's 8: low nibbles (positions 0-1), high nibbles (2-3)
        const uint2 *tb = reinterpret_cast<const uint2 *>(tab) + (lane & 15);
        const uint32_t wr = c.r[nu >> 2], ws = c.s[nu >> 2];
        const uint32_t lo = (wr & 0x0f0f0f0fu) | ((ws << 4) & 0xf0f0f0f0u);
        const uint32_t hi = ((wr >> 4) & 0x0f0f0f0fu) | (ws & 0xf0f0f0f0u);
        const uint2 e0 = tb[__byte_perm(lo, 0, 0x4440 + (nu & 3)) * 16];
        const uint2 e1 = tb[__byte_perm(hi, 0, 0x4440 + (nu & 3)) * 16];
        a[0] = e0.x, a[1] = e0.y, a[2] = e1.x, a[3] = e1.y;
    } else if (KIND == 1) {  // bytes 2nu, 2nu+1 of the lane's 16 -> two levels each
        const uint32_t *tb = reinterpret_cast<const uint32_t *>(tab) + lane;
        const uint32_t r = c.r[nu >> 1] >> (16 * (nu & 1)), s = c.s[nu >> 1] >> (16 * (nu & 1));
        a[0] = tb[(r & 0xffu) * 32], a[2] = tb[((r >> 8) & 0xffu) * 32];
        a[1] = tb[(s & 0xffu) * 32], a[3] = tb[((s >> 8) & 0xffu) * 32];
    } else if (KIND == 2) {  // nibble nu of the lane's 4 bytes: bit pairs 0-1 (positions 0-1) and 2-3 (2-3)
        const uint2 *tb = reinterpret_cast<const uint2 *>(tab) + (lane & 15);
        const uint32_t lo = (c.r[0] & 0x33333333u) | ((c.s[0] << 2) & 0xccccccccu);
        const uint32_t hi = ((c.r[0] >> 2) & 0x33333333u) | (c.s[0] & 0xccccccccu);
        const uint2 e0 = tb[((lo >> (4 * nu)) & 15u) * 16], e1 = tb[((hi >> (4 * nu)) & 15u) * 16];
        a[0] = e0.x, a[1] = e0.y, a[2] = e1.x, a[3] = e1.y;
    } else {  // the 6-bit code pairs at bits 12 nu and 12 nu + 6 of the lane's 12 bytes
        const uint32_t *tb = reinterpret_cast<const uint32_t *>(tab) + lane;
        const int b0 = 12 * nu, b1 = b0 + 6;
        const uint32_t p0 = __funnelshift_r(c.r[b0 >> 5], c.r[(b0 >> 5) + 1], b0 & 31) & 63u;
        const uint32_t p1 = __funnelshift_r(c.r[b1 >> 5], c.r[(b1 >> 5) + 1], b1 & 31) & 63u;
        const uint32_t s0 = __funnelshift_r(c.s[b0 >> 5], c.s[(b0 >> 5) + 1], b0 & 31) & 63u;
        const uint32_t s1 = __funnelshift_r(c.s[b1 >> 5], c.s[(b1 >> 5) + 1], b1 & 31) & 63u;
        a[0] = tb[p0 * 32], a[1] = tb[s0 * 32], a[2] = tb[p1 * 32], a[3] = tb[s1 * 32];
    }
}

// One group of a slice for this warp: the MMAs of every column block, the
// norms and 1/sigma into acc.
template <int KIND, int NB, bool HILO>
__device__ __forceinline__ void w_group(const uint8_t *r0, int rs, const uint8_t *tab, const uint32_t *frag, int g,
                                        int cols, int B, int ng, float n0, float n1, const float *ginv,
                                        float (&acc)[NB][4]) {
    const int lane = threadIdx.x & 31, gq = lane >> 2, t = lane & 3;
    WCodes c;
    w_load<KIND>(r0, r0 + 8 * rs, t, c);
    uint32_t fr[NB][16];
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) {
        const int col = HILO ? gq : 8 * nb + gq;  // this lane's fragment column
        const bool live = HILO ? col < 2 * B : col < B;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const uint4 v = live ? reinterpret_cast<const uint4 *>(frag)[(((size_t)g * 4 + k) * cols + col) * 4 + t]
                                 : make_uint4(0, 0, 0, 0);
            fr[nb][4 * k] = v.x, fr[nb][4 * k + 1] = v.y, fr[nb][4 * k + 2] = v.z, fr[nb][4 * k + 3] = v.w;
        }
    }
    float d[NB][4];
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) d[nb][0] = d[nb][1] = d[nb][2] = d[nb][3] = 0.0f;
#pragma unroll
    for (int nu = 0; nu < 8; ++nu) {
        uint32_t a[4];
        w_decode<KIND>(c, nu, tab, lane, a);
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) w_mma(d[nb], a, fr[nb][2 * nu], fr[nb][2 * nu + 1]);
    }
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) {
        if (HILO) {  // columns 2t, 2t+1: hi and lo terms of batch row t
            const float iv = t < B ? ginv[t * ng + g] : 0.0f;
            acc[nb][0] = fmaf(n0 * iv, d[nb][0], acc[nb][0]);
            acc[nb][1] = fmaf(n0 * iv, d[nb][1], acc[nb][1]);
            acc[nb][2] = fmaf(n1 * iv, d[nb][2], acc[nb][2]);
            acc[nb][3] = fmaf(n1 * iv, d[nb][3], acc[nb][3]);
        } else {  // columns 8nb + 2t, 8nb + 2t + 1: the batch rows of those indices
            const int b0 = 8 * nb + 2 * t;
            const float i0 = b0 < B ? ginv[b0 * ng + g] : 0.0f, i1 = b0 + 1 < B ? ginv[(b0 + 1) * ng + g] : 0.0f;
            acc[nb][0] = fmaf(n0 * i0, d[nb][0], acc[nb][0]);
            acc[nb][1] = fmaf(n0 * i1, d[nb][1], acc[nb][1]);
            acc[nb][2] = fmaf(n1 * i0, d[nb][2], acc[nb][2]);
            acc[nb][3] = fmaf(n1 * i1, d[nb][3], acc[nb][3]);
        }
    }
}

// Code bytes per group of each kind (2-bit, 4-bit, 1-bit, 3-bit codes).
__host__ __device__ __forceinline__ int w_gbytes(int kind) {
    return kind == 0 ? 32 : kind == 1 ? 64 : kind == 2 ? 16 : 48;
}

template <int NB, bool HILO>
__global__ void __launch_bounds__(kWGThreads, 1) gemv_wide_kernel(const __grid_constant__ WParams p) {
    extern __shared__ __align__(16) uint8_t smem[];
    __shared__ WMat sM;
    __shared__ __half s_lv[16];
    __shared__ float s_alpha[kWMaxB];
    __shared__ __align__(8) uint64_t s_bar[kWMaxStages];  // one per stage: every thread's copies of the slice landed
    asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
    const int NS = p.n_stages;
    const uint32_t bars = (uint32_t)__cvta_generic_to_shared(&s_bar[0]);
    if (threadIdx.x == 0) {
        for (int q = 0; q < NS; ++q) asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(bars + 8 * q), "r"(kWGThreads));
        asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    }
    __syncthreads();
    int fills = 0;  // slices issued so far by this block: stage fills % NS, phase (fills / NS) & 1
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, gq = lane >> 2, t = lane & 3;
    const uint8_t *tab = smem;
    uint32_t *frag = reinterpret_cast<uint32_t *>(smem + p.smem_frag);
    float *ginv = reinterpret_cast<float *>(smem + p.smem_frag) + 0;  // placed after the fragments (below)
    float *red = reinterpret_cast<float *>(smem + p.smem_red);       // [8 warps][16 rows][B]
    const int T = p.total_tiles, G = gridDim.x, bid = blockIdx.x;
    const int x_end = (int)(((long long)(bid + 1) * T) / G);
    int cur_lut = -1, cur_act = -1;
    bool waited = false;
    for (int x = (int)(((long long)bid * T) / G); x < x_end;) {
        int lo = 0, hi = p.n_mats - 1;  // the matrix holding tile x
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (p.tiles_before[mid] <= x) lo = mid;
            else hi = mid - 1;
        }
        const int mi = lo, seg_end = min(x_end, p.tiles_before[mi + 1]);
        __syncthreads();  // the previous segment is done with sM, the table, the fragments and the stages
        if (threadIdx.x < (int)(sizeof(WMat) / 4))
            reinterpret_cast<uint32_t *>(&sM)[threadIdx.x] = reinterpret_cast<const uint32_t *>(&p.m[mi])[threadIdx.x];
        else if (threadIdx.x >= 64 && threadIdx.x < 80)
            s_lv[threadIdx.x - 64] = p.lut[p.m[mi].lut][threadIdx.x - 64];
        __syncthreads();
        const WMat &M = sM;
        const int ng = M.ng, B = M.B, kind = M.kind, gb = w_gbytes(kind), rs = M.rs, gs = M.gs;
        const int nslice = (ng + gs - 1) / gs, rowBytes = ng * gb;
        const int t0 = x - p.tiles_before[mi], ntile = seg_end - x, nsl = ntile * nslice;
        ginv = reinterpret_cast<float *>(smem + p.smem_frag + (size_t)ng * p.act_cols[mi] * 256);
        if (M.lut != cur_lut) {
            w_build_table(kind, s_lv, smem);
            cur_lut = M.lut;
        }
        // copies of slice i of the segment into the next stage of the ring: the code
        // bytes of its groups for the tile's 16 rows (rows past the matrix
        // zero-filled), then all of the tile's norms
        auto issue = [&](int i) {
            const int q = (fills + i) % NS;
            if (i < nsl) {
                uint8_t *st = smem + p.smem_stage + q * p.stage_bytes;
                const int tile = t0 + i / nslice, g0 = (i % nslice) * gs, gcnt = min(gs, ng - g0);
                const int cpr = gcnt * gb / 16, row0 = 16 * tile, valid = min(16, M.out - row0);
                for (int c = threadIdx.x; c < 16 * cpr; c += kWGThreads) {
                    const int r = c / cpr, k = c - r * cpr;
                    const bool ok = r < valid;
                    w_cp16(st + r * rs + 16 * k, M.codes + (size_t)(ok ? row0 + r : 0) * rowBytes + g0 * gb + 16 * k,
                           ok ? 16 : 0);
                }
                const int nbytes = 32 * ng, avail = valid * ng * 2;
                const uint8_t *src = reinterpret_cast<const uint8_t *>(M.norms + (size_t)row0 * ng);
                for (int c = threadIdx.x; 16 * c < nbytes; c += kWGThreads) {
                    const int left = avail - 16 * c, n = left >= 16 ? 16 : (left > 0 ? left : 0);
                    w_cp16(st + 16 * rs + 16 * c, n ? src + 16 * c : src, n);
                }
                // the stage's barrier completes once every thread's copies so far have landed
                asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];\n" ::"r"(bars + 8 * q) : "memory");
            }
        };
        for (int k = 0; k + 1 < NS; ++k) issue(k);
        if (!waited) {  // the rotation of the activations is complete and visible
            asm volatile("griddepcontrol.wait;\n" ::: "memory");
            waited = true;
        }
        const int cols = p.act_cols[mi];
        if (M.act != cur_act) {  // the activation's fragments and 1/sigma -> shared memory
            const uint4 *fs = reinterpret_cast<const uint4 *>(p.frag + p.act_frag[mi]);
            uint4 *fd = reinterpret_cast<uint4 *>(frag);
            const int n4 = ng * cols * 16;  // 16-byte words
            for (int e = threadIdx.x; e < n4; e += kWGThreads) w_cp16(fd + e, fs + e, 16);
            for (int e = threadIdx.x; e < B * ng; e += kWGThreads) ginv[e] = p.ginv[p.act_ginv[mi] + e];
            asm volatile("cp.async.wait_all;\n" ::: "memory");  // (the stage copies issued above too)
            cur_act = M.act;
        }
        if (threadIdx.x < B)
            s_alpha[threadIdx.x] = M.xdt == CQ_X_I8 ? __fmul_rn(M.xs[threadIdx.x], kWInvSqrt128) : kWInvSqrt128;
        __syncthreads();  // the table, the fragments, 1/sigma and the output scales are in place
        float acc[NB][4];
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) acc[nb][0] = acc[nb][1] = acc[nb][2] = acc[nb][3] = 0.0f;
        for (int i = 0; i < nsl; ++i) {
            issue(i + NS - 1);
            {  // bounded wait for slice i (every thread's share of its copies)
                const int q = (fills + i) % NS;
                const uint32_t par = ((fills + i) / NS) & 1;
                bool ok = false;
                for (unsigned it = 0; it < (1u << 20) && !ok; ++it) {
                    uint32_t r;
                    asm volatile(
                        "{\n .reg .pred pp;\n mbarrier.try_wait.parity.shared::cta.b64 pp, [%1], %2, %3;\n selp.u32 %0, 1, 0, pp;\n}\n"
                        : "=r"(r)
                        : "r"(bars + 8 * q), "r"(par), "r"(1000u)
                        : "memory");
                    ok = r != 0;
                }
                if (!ok && threadIdx.x == 0 && p.status) atomicOr(p.status, 0x47570001u);
            }
            const uint8_t *st = smem + p.smem_stage + ((fills + i) % NS) * p.stage_bytes;
            const __half *sn = reinterpret_cast<const __half *>(st + 16 * rs);
            const int tile = t0 + i / nslice, sidx = i % nslice, g0 = sidx * gs, gcnt = min(gs, ng - g0);
            for (int gl = warp; gl < gcnt; gl += kWGWarps) {
                const int g = g0 + gl;
                const uint8_t *r0 = st + gq * rs + gl * gb;
                const float n0 = __half2float(sn[gq * ng + g]), n1 = __half2float(sn[(gq + 8) * ng + g]);
                if (kind == 0) w_group<0, NB, HILO>(r0, rs, tab, frag, g, cols, B, ng, n0, n1, ginv, acc);
                else if (kind == 1) w_group<1, NB, HILO>(r0, rs, tab, frag, g, cols, B, ng, n0, n1, ginv, acc);
                else if (kind == 2) w_group<2, NB, HILO>(r0, rs, tab, frag, g, cols, B, ng, n0, n1, ginv, acc);
                else w_group<3, NB, HILO>(r0, rs, tab, frag, g, cols, B, ng, n0, n1, ginv, acc);
            }
            if (sidx == nslice - 1) {  // the tile is complete: its warps' partial sums meet
#pragma unroll
                for (int nb = 0; nb < NB; ++nb) {
                    if (HILO) {
                        if (t < B) {
                            red[(warp * 16 + gq) * B + t] = acc[nb][0] + acc[nb][1];
                            red[(warp * 16 + gq + 8) * B + t] = acc[nb][2] + acc[nb][3];
                        }
                    } else {
                        const int b0 = 8 * nb + 2 * t;
                        if (b0 < B) {
                            red[(warp * 16 + gq) * B + b0] = acc[nb][0];
                            red[(warp * 16 + gq + 8) * B + b0] = acc[nb][2];
                        }
                        if (b0 + 1 < B) {
                            red[(warp * 16 + gq) * B + b0 + 1] = acc[nb][1];
                            red[(warp * 16 + gq + 8) * B + b0 + 1] = acc[nb][3];
                        }
                    }
                    acc[nb][0] = acc[nb][1] = acc[nb][2] = acc[nb][3] = 0.0f;
                }
                __syncthreads();
                if (threadIdx.x < 16 * B) {
                    const int r = threadIdx.x / B, b = threadIdx.x - r * B, row = 16 * tile + r;
                    float sum = 0.0f;
#pragma unroll
                    for (int w = 0; w < kWGWarps; ++w) sum += red[(w * 16 + r) * B + b];
                    if (row < M.out) M.y[(size_t)b * M.out + row] = sum * s_alpha[b];
                }
            }
            __syncthreads();  // the stage (and the partial sums) may be reused
        }
        asm volatile("cp.async.wait_all;\n" ::: "memory");
        fills += nsl;
        x = seg_end;
    }
    if (!waited) asm volatile("griddepcontrol.wait;\n" ::: "memory");
}


// ----------------------------------------------------- split products --
// gemv_split_kernel: the products with the work cut finer than a block's
// run of tiles and every warp on its own pipeline. It takes batches of 1 to
// 4 with 1-, 2-, 3- and 4-bit codes at group 128, and 1-, 2- and 4-bit codes
// at group 64 (larger batches run faster on the sliced kernel above). A
// unit is (matrix, k-slice of its groups, 16-row tile); units are numbered
// matrix by matrix, k-slice by k-slice, tile fastest, and each block takes an
// equal contiguous range of them, split evenly over its 16 warps. A matrix
// is cut into k-slices only when its tiles alone would leave more than three
// quarters of the warps idle (one 4096-row matrix has 256 tiles for 2432
// warps); the k-slices of a tile then
// leave their partial sums in a workspace and the last one to finish (a
// counter per tile) adds them in k-slice order, so the result does not
// depend on the order in which they finish.
//
// Every warp streams its own units through shared-memory stages of one
// chunk each: two stages of 16 rows x 256 code bytes (eight CQ2 128-spans,
// four CQ4 spans, sixteen binary spans) or x 192 (four CQ3 spans). One lane per row issues a 1-D TMA bulk copy of the row's chunk (completion
// on the stage's mbarrier) and a cp.async of its norms. No block barrier runs inside the loop. A block
// rotates the activation groups of the (matrix, k-slice) pairs of its range
// into shared memory once, after the launch before it is complete (one
// launch per call: no rotation launch on the critical path).
constexpr int kSWarps = 16;
constexpr int kSThreads = 32 * kSWarps;
constexpr int kSStages = 2;
constexpr int kSMaxMats = 128;
constexpr int kSMaxPairs = 24;  // (matrix, k-slice) pairs of one block's range

struct SMat {
    const uint8_t *codes;
    const __half *norms;
    float *y;
    const float *xs;
    long long unit0;  // first unit of the matrix
    const void *x;    // the activation [B][in], fp32 or int8
    int act;          // which distinct activation of the launch x is
    int in;
    int out, ng, B, xdt, cols;
    int tiles, nks, gk;  // 16-row tiles, k-slices, groups per k-slice
    int cnt0;            // first tile counter (k-sliced matrices)
    long long part0;     // first partial-sum slot [unit][16][B] (k-sliced matrices)
};

struct SParams {
    int n_mats;
    long long total_units;
    long long units_before[kSMaxMats + 1];
    float *part;
    unsigned int *cnt;
    unsigned int *status;
    int smem_frag, frag_budget, smem_stage;
    __half lut[16];
    SMat m[kSMaxMats];
};

static_assert(sizeof(SParams) <= 32000, "kernel parameter block");

// Code bytes per group and groups per chunk of each kind.
__host__ __device__ constexpr int s_gbytes(int kind) { return kind == 0 ? 32 : kind == 1 ? 64 : kind == 2 ? 16 : 48; }
__host__ __device__ constexpr int s_gc(int kind) { return kind == 0 ? 8 : kind == 1 ? 4 : kind == 2 ? 16 : 4; }
// Row stride of a stage: the chunk plus padding that spreads a warp's reads
// of its rows over the banks (as for the sliced kernel's stages). 3-bit
// codes: each lane reads three words at 12t, rows 240 bytes (28 banks) apart,
// so a warp's 32 reads of one word index fall in 32 distinct banks. Groups
// of 64 read 4-byte words (2-bit codes) or 8-byte words (4-bit) of each half,
// rows 4 and 8 banks apart; 1-bit codes 2-byte halves, rows 4 banks apart.
__host__ __device__ constexpr int s_rs(int kind, bool g64 = false) {
    return g64 ? (kind == 1 ? 288 : 272) : kind == 0 ? 288 : kind == 1 ? 320 : kind == 2 ? 272 : 240;
}
// Bytes of norms per row of a stage (a multiple of 16): one fp16 norm per
// group, two per 128-span for groups of 64.
__host__ __device__ constexpr int s_nr(int kind, bool g64 = false) {
    return (2 * s_gc(kind) * (g64 ? 2 : 1) + 15) / 16 * 16;
}
__host__ __device__ constexpr int s_stage_bytes(int kind, bool g64 = false) {
    return 16 * s_rs(kind, g64) + 16 * s_nr(kind, g64);
}

// One (matrix, k-slice) pair of a block's range and where its fragments and
// 1/sigma sit in shared memory.
struct SPair {
    long long u_end;  // units of the pair in the range end here
    int m, s, g_lo, g_n, frag_off, ginv_off;  // frag_off in 16-byte units, ginv_off in floats
};

__device__ __forceinline__ uint32_t s_smem(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

// Bounded wait on an mbarrier phase: false after about a second.
__device__ __forceinline__ bool s_wait(uint32_t bar, uint32_t parity) {
    for (unsigned it = 0; it < (1u << 20); ++it) {
        uint32_t r;
        asm volatile(
            "{\n .reg .pred pp;\n mbarrier.try_wait.parity.shared::cta.b64 pp, [%1], %2, %3;\n selp.u32 %0, 1, 0, pp;\n}\n"
            : "=r"(r)
            : "r"(bar), "r"(parity), "r"(1000u)
            : "memory");
        if (r) return true;
    }
    return false;
}

// The code words of one 128-span of groups of 64 for this lane, in the
// half-major order of the fragments: MMA nu reads positions
// 64 (nu / 4) + 16t + 4 (nu % 4) .. +3, so the words of each half are loaded
// apart and w_decode then indexes them as it does for groups of 128.
template <int KIND>
__device__ __forceinline__ void s_load64(const uint8_t *r0, const uint8_t *r1, int t, WCodes &c) {
    if (KIND == 0) {  // bytes 4t .. 4t+3 of each 16-byte half
        c.r[0] = *reinterpret_cast<const uint32_t *>(r0 + 4 * t), c.r[1] = *reinterpret_cast<const uint32_t *>(r0 + 16 + 4 * t);
        c.s[0] = *reinterpret_cast<const uint32_t *>(r1 + 4 * t), c.s[1] = *reinterpret_cast<const uint32_t *>(r1 + 16 + 4 * t);
    } else if (KIND == 1) {  // bytes 8t .. 8t+7 of each 32-byte half
        const uint2 a = *reinterpret_cast<const uint2 *>(r0 + 8 * t), b = *reinterpret_cast<const uint2 *>(r0 + 32 + 8 * t);
        const uint2 e = *reinterpret_cast<const uint2 *>(r1 + 8 * t), f = *reinterpret_cast<const uint2 *>(r1 + 32 + 8 * t);
        c.r[0] = a.x, c.r[1] = a.y, c.r[2] = b.x, c.r[3] = b.y, c.s[0] = e.x, c.s[1] = e.y, c.s[2] = f.x, c.s[3] = f.y;
    } else {  // 1-bit codes: bytes 2t, 2t+1 of each 8-byte half, as one word
        const uint16_t *q0 = reinterpret_cast<const uint16_t *>(r0), *q1 = reinterpret_cast<const uint16_t *>(r1);
        c.r[0] = (uint32_t)q0[t] | ((uint32_t)q0[4 + t] << 16);
        c.s[0] = (uint32_t)q1[t] | ((uint32_t)q1[4 + t] << 16);
    }
}

// Two groups of a chunk (g, g + 1) as two independent MMA chains (fragment
// columns 2b and 2b + 1: the hi and lo terms of batch row b); the second
// group's codes, fragments and norms are zero when `two` is false (its chain
// then adds nothing). G64: g and g + 1 are
// 128-spans of two groups of 64 each; MMAs 0-3 and 4-7 of a span then run as
// separate chains, scaled by the norms of the first half (n..) and of the
// second (m..).
template <int KIND, bool G64>
__device__ __forceinline__ void s_group2(const uint8_t *r0, int rs, const uint8_t *tab, const uint32_t *frag, int g,
                                         int cols, int B, int ngs, float n0a, float n1a, float n0b, float n1b,
                                         float m0a, float m1a, float m0b, float m1b, bool two, const float *ginv,
                                         const uint4 *zero, float (&acc)[4]) {
    static_assert(!G64 || KIND != 3, "groups of 64: 1-, 2- and 4-bit codes");
    const int lane = threadIdx.x & 31, gq = lane >> 2, t = lane & 3;
    constexpr int GB = s_gbytes(KIND);
    WCodes ca, cb;
    if (G64) s_load64<KIND>(r0, r0 + 8 * rs, t, ca);
    else w_load<KIND>(r0, r0 + 8 * rs, t, ca);
    if (two) {
        if (G64) s_load64<KIND>(r0 + GB, r0 + GB + 8 * rs, t, cb);
        else w_load<KIND>(r0 + GB, r0 + GB + 8 * rs, t, cb);
    } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) cb.r[i] = cb.s[i] = 0u;
    }
    // this lane's fragment column gq; lanes of columns past the batch read
    // the zero block (one address, no selects on the loaded words)
    const bool live = gq < 2 * B;
    const uint4 *f4 = reinterpret_cast<const uint4 *>(frag);
    const uint4 *pa = live ? f4 + (((size_t)g * 4) * cols + gq) * 4 + t : zero;
    const uint4 *pb = live && two ? f4 + (((size_t)(g + 1) * 4) * cols + gq) * 4 + t : zero;
    const int sa = live ? cols * 4 : 0, sb = live && two ? cols * 4 : 0;
    uint32_t fa[16], fb[16];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const uint4 va = pa[k * sa], vb = pb[k * sb];
        fa[4 * k] = va.x, fa[4 * k + 1] = va.y, fa[4 * k + 2] = va.z, fa[4 * k + 3] = va.w;
        fb[4 * k] = vb.x, fb[4 * k + 1] = vb.y, fb[4 * k + 2] = vb.z, fb[4 * k + 3] = vb.w;
    }
    float da[4] = {0.f, 0.f, 0.f, 0.f}, db[4] = {0.f, 0.f, 0.f, 0.f};
    float ea[4] = {0.f, 0.f, 0.f, 0.f}, eb[4] = {0.f, 0.f, 0.f, 0.f};  // second halves (G64)
#pragma unroll
    for (int nu = 0; nu < 8; ++nu) {
        uint32_t a[4], b[4];
        w_decode<KIND>(ca, nu, tab, lane, a);
        w_decode<KIND>(cb, nu, tab, lane, b);
        if (G64 && nu >= 4) {
            w_mma(ea, a, fa[2 * nu], fa[2 * nu + 1]);
            w_mma(eb, b, fb[2 * nu], fb[2 * nu + 1]);
        } else {
            w_mma(da, a, fa[2 * nu], fa[2 * nu + 1]);
            w_mma(db, b, fb[2 * nu], fb[2 * nu + 1]);
        }
    }
    // this lane's outputs: columns 2t, 2t+1 (hi and lo terms of batch row t)
    const float ia = t < B ? ginv[t * ngs + g] : 0.0f, ib = t < B && two ? ginv[t * ngs + g + 1] : 0.0f;
    acc[0] = fmaf(n0b * ib, db[0], fmaf(n0a * ia, da[0], acc[0]));
    acc[1] = fmaf(n0b * ib, db[1], fmaf(n0a * ia, da[1], acc[1]));
    acc[2] = fmaf(n1b * ib, db[2], fmaf(n1a * ia, da[2], acc[2]));
    acc[3] = fmaf(n1b * ib, db[3], fmaf(n1a * ia, da[3], acc[3]));
    if (G64) {
        acc[0] = fmaf(m0b * ib, eb[0], fmaf(m0a * ia, ea[0], acc[0]));
        acc[1] = fmaf(m0b * ib, eb[1], fmaf(m0a * ia, ea[1], acc[1]));
        acc[2] = fmaf(m1b * ib, eb[2], fmaf(m1a * ia, ea[2], acc[2]));
        acc[3] = fmaf(m1b * ib, eb[3], fmaf(m1a * ia, ea[3], acc[3]));
    }
}

template <int KIND, bool G64>
__global__ void __launch_bounds__(kSThreads, 1) gemv_split_kernel(const __grid_constant__ SParams p) {
    constexpr int GC = s_gc(KIND), GB = s_gbytes(KIND), RS = s_rs(KIND, G64), SB = s_stage_bytes(KIND, G64);
    constexpr int NS = kSStages;
    constexpr int NR = s_nr(KIND, G64) / 2;  // norms per row of a stage
    constexpr int NPS = G64 ? 2 : 1;         // norms per 128-span
    constexpr float kScale = G64 ? 0.125f : kWInvSqrt128;  // 1 / sqrt(group)
    extern __shared__ __align__(16) uint8_t smem[];
    __shared__ __align__(8) uint64_t s_bar[kSWarps * kSStages];
    __shared__ SPair s_pair[kSMaxPairs + 1];
    __shared__ SMat s_mat[kSMaxPairs];
    __shared__ __half s_lv[16];
    __shared__ int s_npair, s_bad;
    __shared__ uint4 s_zero;  // what fragment loads of columns past the batch read
    asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, gq = lane >> 2, t = lane & 3;
    const long long U = p.total_units;
    const long long cu0 = U * blockIdx.x / gridDim.x, cu1 = U * (blockIdx.x + 1) / gridDim.x;
    const long long wu0 = cu0 + (cu1 - cu0) * warp / kSWarps, wu1 = cu0 + (cu1 - cu0) * (warp + 1) / kSWarps;

    if (warp == 1) {  // the stage barriers
        for (int i = lane; i < kSWarps * NS; i += 32)
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;\n" ::"r"(s_smem(&s_bar[i])));
        __syncwarp();
        if (lane == 0) {
            asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
            s_zero = make_uint4(0, 0, 0, 0);
        }
    } else if (warp == 0) {
        // the matrix of the range's first unit: the last m with units_before[m] <= cu0
        // (the lanes compare 32 entries at a time; the table is ascending)
        int m0 = -1;
        for (int base = 0; base <= p.n_mats; base += 32) {
            const int i = base + lane;
            m0 += __popc(__ballot_sync(0xffffffffu, i <= p.n_mats && p.units_before[i] <= cu0));
        }
        if (lane == 0) {
            // the (matrix, k-slice) pairs of the range, and where their fragments go
            int n = 0, foff = 0, goff = 0, pm = -1;
            long long u = cu0;
            int m = max(m0, 0);
            while (u < cu1 && n < kSMaxPairs) {
                while (p.units_before[m + 1] <= u) ++m;
                const SMat &M = p.m[m];
                const long long unit0 = M.unit0;
                const int tiles = M.tiles, gk = M.gk, ng = M.ng, cols = M.cols, B = M.B;
                const int act = M.act;
                const int s = (int)((u - unit0) / tiles);
                const long long end = min(cu1, unit0 + (long long)(s + 1) * tiles);
                SPair &P = s_pair[n];
                P.u_end = end;
                P.m = m;
                P.s = s;
                P.g_lo = s * gk;
                P.g_n = min(gk, ng - P.g_lo);
                // a pair that reads the same fragments as the one before shares them
                const bool same = n > 0 && p.m[pm].act == act && p.m[pm].cols == cols && s_pair[n - 1].g_lo == P.g_lo &&
                                  s_pair[n - 1].g_n == P.g_n && p.m[pm].B == B;
                if (same) {
                    P.frag_off = s_pair[n - 1].frag_off;
                    P.ginv_off = s_pair[n - 1].ginv_off;
                } else {
                    P.frag_off = foff;
                    P.ginv_off = goff;
                    foff += P.g_n * cols * 16;
                    goff += B * P.g_n;
                }
                pm = m;
                ++n;
                u = end;
            }
            s_pair[n].u_end = 0x7fffffffffffffffLL;  // sentinel
            s_npair = n;
            // the host planned every range to fit; a block whose range does not
            // is reported and does nothing
            s_bad = u < cu1 || (size_t)foff * 16 + (size_t)goff * 4 > (size_t)p.frag_budget;
            if (s_bad && p.status) atomicOr(p.status, 0x47570010u);
        }
        __syncwarp();
        // the pairs' matrix descriptors, word by word across the lanes
        for (int n = 0; n < s_npair; ++n) {
            const uint32_t *src = reinterpret_cast<const uint32_t *>(&p.m[s_pair[n].m]);
            for (int w = lane; w < (int)(sizeof(SMat) / 4); w += 32) reinterpret_cast<uint32_t *>(&s_mat[n])[w] = src[w];
        }
    }
    if (threadIdx.x < 16) s_lv[threadIdx.x] = p.lut[threadIdx.x];
    __syncthreads();
    w_build_table(KIND, s_lv, smem);
    const bool ok_range = !s_bad && s_npair > 0;

    uint8_t *stage0 = smem + p.smem_stage + (size_t)warp * NS * SB;
    const uint32_t bar0 = s_smem(&s_bar[warp * NS]);
    bool abort = !ok_range;

    // ---- the warp's chunk stream: the issue side runs NS - 1 chunks ahead
    // of the products. Each side keeps its unit's numbers in registers
    // (read from shared memory once per unit). ----
    long long iu = wu0;                   // issue side: unit, pair, chunk, chunks
    int ipair = 0, ic = 0, inch = 0, iga0 = 0, igend = 0, ivalid = 0;
    const uint8_t *irow = nullptr;        // this lane's code row (lanes < 16)
    const __half *inrow = nullptr;        // and its norms
    auto iload = [&]() {
        while (iu >= s_pair[ipair].u_end) ++ipair;
        const SPair &P = s_pair[ipair];
        const SMat &M = s_mat[ipair];
        const int row0 = 16 * (int)(iu - M.unit0 - (long long)P.s * M.tiles);
        iga0 = P.g_lo;
        igend = P.g_lo + P.g_n;
        inch = (P.g_n + GC - 1) / GC;
        ic = 0;
        ivalid = min(16, M.out - row0);
        const int r = row0 + min(lane & 15, ivalid - 1);  // rows past the matrix repeat the last one
        irow = M.codes + (size_t)r * M.ng * GB;
        inrow = M.norms + (size_t)r * M.ng * NPS;
    };
    int iq = 0, copied = 0;  // next stage to fill; chunks with copies so far
    auto issue = [&]() {
        if (iu < wu1 && !abort) {
            uint8_t *st = stage0 + iq * SB;
            const int ga = iga0 + ic * GC, gcnt = min(GC, igend - ga), bytes = gcnt * GB;
            const uint32_t bar = bar0 + 8 * iq;
            // earlier generic reads of the stage come before the copy rewrites it
            asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
            __syncwarp();
            if (lane == 0)
                asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(bar), "r"(ivalid * bytes)
                             : "memory");
            __syncwarp();
            if (lane < ivalid)
                asm volatile(
                    "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(
                        s_smem(st + lane * RS)),
                    "l"(irow + (size_t)ga * GB), "r"(bytes), "r"(bar)
                    : "memory");
            if (lane < 16) {  // this row's norms of the chunk
                const __half *src = inrow + ga * NPS;
                const int nn = gcnt * NPS;
                __half *dst = reinterpret_cast<__half *>(st + 16 * RS + lane * 2 * NR);
                if ((nn & 7) == 0 && (reinterpret_cast<uintptr_t>(src) & 15) == 0) {
#pragma unroll
                    for (int i = 0; i < GC * NPS; i += 8)
                        if (i < nn)
                            asm volatile("cp.async.ca.shared.global [%0], [%1], 16;\n" ::"r"(s_smem(dst + i)),
                                         "l"(src + i)
                                         : "memory");
                } else if (((reinterpret_cast<uintptr_t>(src) & 3) == 0) && (nn & 1) == 0) {
#pragma unroll
                    for (int i = 0; i < GC * NPS; i += 2)
                        if (i < nn)
                            asm volatile("cp.async.ca.shared.global [%0], [%1], 4;\n" ::"r"(s_smem(dst + i)), "l"(src + i)
                                         : "memory");
                } else {
                    for (int i = 0; i < nn; ++i) dst[i] = src[i];
                }
            }
            if (++ic == inch && ++iu < wu1) iload();
            ++copied;
        }
        asm volatile("cp.async.commit_group;\n" ::: "memory");
        iq = iq + 1 == NS ? 0 : iq + 1;
    };
    if (wu0 < wu1 && !abort) iload();
    // the code copies do not depend on the launch before this one
    for (int i = 0; i + 1 < NS; ++i) issue();

    // ---- fragments and 1/sigma of the range's pairs: this block rotates the
    // k-slice groups of each distinct (activation, k-slice) it meets, once
    // the launch before this one (which may write the activation) is
    // complete. A task is (pair, group of the slice, batch row): one warp
    // runs the FWHT of the group in registers (lane l holds positions
    // 4l .. 4l+3) and writes the fp16 hi and lo terms of sigma z straight
    // into the MMA B-fragment layout, as the rotation launch does for the
    // sliced kernel. Groups of 64 stop before the butterfly stage that mixes
    // a span's halves (lane bit 4 is position bit 6) and take a half-major
    // word order: word 2j + h of MMA lane t holds positions
    // 64 (j / 4) + 16t + 4 (j % 4) + 2h + {0, 1}, so MMAs 0-3 of a span read
    // only its first half and MMAs 4-7 only its second (lane
    // l = 16 (j / 4) + 4t + j % 4 owns them). ----
    asm volatile("griddepcontrol.wait;\n" ::: "memory");
    uint4 *sfrag = reinterpret_cast<uint4 *>(smem + p.smem_frag);
    float *sginv = reinterpret_cast<float *>(smem + p.smem_frag);
    int ginv_base = 0, ntask = 0;  // after every pair's fragments; rotation tasks of the range
    for (int i = 0; i < (ok_range ? s_npair : 0); ++i) {
        ginv_base = max(ginv_base, s_pair[i].frag_off + s_pair[i].g_n * s_mat[i].cols * 16);
        if (i == 0 || s_pair[i].frag_off != s_pair[i - 1].frag_off) ntask += s_pair[i].g_n * s_mat[i].B;
    }
    sginv += 4 * ginv_base;
    for (int task = warp; task < ntask; task += kSWarps) {
        int i = 0, base = 0;  // the pair of the task
        for (;; ++i) {
            if (i > 0 && s_pair[i].frag_off == s_pair[i - 1].frag_off) continue;
            const int nt = s_pair[i].g_n * s_mat[i].B;
            if (task < base + nt) break;
            base += nt;
        }
        const SPair &P = s_pair[i];
        const SMat &M = s_mat[i];
        const int local = task - base, gl = local / M.B, b = local - gl * M.B;
        const int col0 = (P.g_lo + gl) * kGroup + 4 * lane;
        float v[4];
        if (M.xdt == CQ_X_I8) {
            const int8_t *xq = static_cast<const int8_t *>(M.x) + (size_t)b * M.in;
#pragma unroll
            for (int k = 0; k < 4; ++k) v[k] = col0 + k < M.in ? (float)xq[col0 + k] : 0.0f;
        } else {
            const float *xf = static_cast<const float *>(M.x) + (size_t)b * M.in;
#pragma unroll
            for (int k = 0; k < 4; ++k) v[k] = col0 + k < M.in ? xf[col0 + k] : 0.0f;
        }
        {
            const float a0 = v[0] + v[1], a1 = v[0] - v[1], a2 = v[2] + v[3], a3 = v[2] - v[3];
            v[0] = a0 + a2;
            v[1] = a1 + a3;
            v[2] = a0 - a2;
            v[3] = a1 - a3;
        }
#pragma unroll
        for (int m = 1; m < (G64 ? 16 : 32); m <<= 1)  // lane bit 4 is position bit 6: the halves of a span
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float o = __shfl_xor_sync(0xffffffffu, v[k], m);
                v[k] = (lane & m) ? o - v[k] : v[k] + o;
            }
        // int8 activations give integers |z| <= 128 * 128, which hi + lo carry
        // exactly unscaled; otherwise scale by a power of two to |sigma z| <= 2^14
        float sigma = 1.0f;
        if (M.xdt != CQ_X_I8) {
            float mx = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
#pragma unroll
            for (int m = 16; m; m >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, m));
            sigma = w_pow2_scale(mx, 16384.0f);
        }
        uint32_t hi16[4], lo16[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float xs = __fmul_rn(v[k], sigma);
            const __half h = __float2half_rn(xs);
            const __half l = __float2half_rn(__fsub_rn(xs, __half2float(h)));
            hi16[k] = __half_as_ushort(h);
            lo16[k] = __half_as_ushort(l);
        }
        // this lane's positions are words 2j, 2j+1 of MMA lane t (unit k = j / 2, offset 2 (j % 2))
        const int tt = G64 ? (lane >> 2) & 3 : lane >> 3, j = G64 ? ((lane >> 4) << 2) | (lane & 3) : lane & 7;
        uint32_t *fw = reinterpret_cast<uint32_t *>(sfrag + P.frag_off);
        const int k = j >> 1, w2 = 2 * (j & 1);
        *reinterpret_cast<uint2 *>(fw + ((((size_t)gl * 4 + k) * M.cols + 2 * b) * 4 + tt) * 4 + w2) =
            make_uint2(hi16[0] | (hi16[1] << 16), hi16[2] | (hi16[3] << 16));
        *reinterpret_cast<uint2 *>(fw + ((((size_t)gl * 4 + k) * M.cols + 2 * b + 1) * 4 + tt) * 4 + w2) =
            make_uint2(lo16[0] | (lo16[1] << 16), lo16[2] | (lo16[3] << 16));
        if (lane == 0) sginv[P.ginv_off + b * P.g_n + gl] = 1.0f / sigma;
    }
    __syncthreads();

    // ---- the products ----
    long long cu = wu0;  // product side: unit, pair, chunk, chunks
    int cpair = 0, cc = 0, cnch = 0, cglo = 0, cgend = 0, ccols = 0, cB = 0, cgn = 0, ct = 0;
    const uint32_t *cfrag = nullptr;
    const float *cginv = nullptr;
    auto cload = [&]() {
        while (cu >= s_pair[cpair].u_end) ++cpair;
        const SPair &P = s_pair[cpair];
        const SMat &M = s_mat[cpair];
        ct = (int)(cu - M.unit0 - (long long)P.s * M.tiles);
        cglo = P.g_lo;
        cgn = P.g_n;
        cgend = P.g_lo + P.g_n;
        cnch = (P.g_n + GC - 1) / GC;
        cc = 0;
        ccols = M.cols;
        cB = M.B;
        cfrag = reinterpret_cast<const uint32_t *>(sfrag + P.frag_off);
        cginv = sginv + P.ginv_off;
    };
    if (wu0 < wu1 && !abort) cload();
    int cq = 0, done = 0;
    uint32_t phase = 0;  // bit q: parity of stage q's next completion
    float acc[4] = {0.f, 0.f, 0.f, 0.f};  // rows gq, gq + 8 x columns 2t, 2t + 1 (hi, lo of batch row t)
    const uint8_t *tab = smem;
    while (cu < wu1 && !abort) {
        issue();
        if (!s_wait(bar0 + 8 * cq, (phase >> cq) & 1u)) {
            if (lane == 0 && p.status) atomicOr(p.status, 0x47570011u);
            abort = true;
            break;
        }
        phase ^= 1u << cq;
        asm volatile("cp.async.wait_group %0;\n" ::"n"(NS - 1) : "memory");
        __syncwarp();
        const uint8_t *st = stage0 + cq * SB;
        const __half *sn = reinterpret_cast<const __half *>(st + 16 * RS);
        const int gl0 = cc * GC, gcnt = min(GC, cgn - gl0);  // the chunk's groups, local to the k-slice
#pragma unroll
        for (int gl = 0; gl < GC; gl += 2) {
            if (gl < gcnt) {
                const bool two = gl + 1 < gcnt;
                // norms of rows gq and gq + 8: span gl (a) and gl + 1 (b);
                // for groups of 64 the first halves' (n) and second halves' (m)
                const __half *s0 = sn + gq * NR + gl * NPS, *s1 = sn + (gq + 8) * NR + gl * NPS;
                const float n0a = __half2float(s0[0]), n1a = __half2float(s1[0]);
                const float n0b = two ? __half2float(s0[NPS]) : 0.0f, n1b = two ? __half2float(s1[NPS]) : 0.0f;
                float m0a = n0a, m1a = n1a, m0b = n0b, m1b = n1b;
                if (G64) {
                    m0a = __half2float(s0[1]);
                    m1a = __half2float(s1[1]);
                    m0b = two ? __half2float(s0[3]) : 0.0f;
                    m1b = two ? __half2float(s1[3]) : 0.0f;
                }
                s_group2<KIND, G64>(st + gq * RS + gl * GB, RS, tab, cfrag, gl0 + gl, ccols, cB, cgn, n0a, n1a, n0b,
                                    n1b, m0a, m1a, m0b, m1b, two, cginv, &s_zero, acc);
            }
        }
        cq = cq + 1 == NS ? 0 : cq + 1;
        ++done;
        if (++cc == cnch) {  // the unit is complete
            const SMat &M = s_mat[cpair];
            const int B = cB;
            const int row_r = 16 * ct + gq, row_s = row_r + 8;
            // this lane's values: batch row t, rows gq and gq + 8 (hi + lo terms)
            const float vr = acc[0] + acc[1], vs = acc[2] + acc[3];
            acc[0] = acc[1] = acc[2] = acc[3] = 0.0f;
            if (M.nks == 1) {
                if (t < B) {
                    const float a = M.xdt == CQ_X_I8 ? __fmul_rn(M.xs[t], kScale) : kScale;
                    if (row_r < M.out) M.y[(size_t)t * M.out + row_r] = vr * a;
                    if (row_s < M.out) M.y[(size_t)t * M.out + row_s] = vs * a;
                }
            } else {
                // partial sums of this k-slice, then the tile's counter
                const int s = cglo / M.gk;
                float *part = p.part + (M.part0 + (long long)s * M.tiles + ct) * 16 * B;
                if (t < B) {
                    part[gq * B + t] = vr;
                    part[(gq + 8) * B + t] = vs;
                }
                __threadfence();
                __syncwarp();
                unsigned old = 0;
                if (lane == 0) old = atomicAdd(p.cnt + M.cnt0 + ct, 1u);
                old = __shfl_sync(0xffffffffu, old, 0);
                if (old == (unsigned)M.nks - 1) {  // the last k-slice of the tile: add them in order
                    __threadfence();
                    const float *base = p.part + (M.part0 + ct) * 16 * B;
                    // lane l adds elements l, l + 32, ...; its loads (element i,
                    // k-slice s2 in the order q = i * nks + s2) go out 16 at a
                    // time (the host keeps them to one batch), then the sums run
                    // in k-slice order
                    const int E = 16 * B, ne = (E + 31) / 32, tot = ne * M.nks;
                    const size_t sstride = (size_t)M.tiles * 16 * B;
                    float sum = 0.0f;
                    int cur = -1;
                    auto put = [&](int i, float v2) {
                        const int e2 = lane + 32 * i;
                        if (e2 >= E) return;
                        const int r = e2 / B, b = e2 - r * B, row = 16 * ct + r;
                        if (row < M.out) {
                            const float a = M.xdt == CQ_X_I8 ? __fmul_rn(M.xs[b], kScale) : kScale;
                            M.y[(size_t)b * M.out + row] = v2 * a;
                        }
                    };
                    for (int q0 = 0; q0 < tot; q0 += 16) {
                        float vv[16];
#pragma unroll
                        for (int j = 0; j < 16; ++j) {
                            const int q = q0 + j, i = q / M.nks, s2 = q - i * M.nks, e2 = lane + 32 * i;
                            vv[j] = (q < tot && e2 < E) ? __ldcg(base + (size_t)s2 * sstride + e2) : 0.0f;
                        }
#pragma unroll
                        for (int j = 0; j < 16; ++j) {
                            const int q = q0 + j;
                            if (q >= tot) break;
                            const int i = q / M.nks;
                            if (i != cur) {
                                if (cur >= 0) put(cur, sum);
                                sum = 0.0f;
                                cur = i;
                            }
                            sum += vv[j];
                        }
                    }
                    if (cur >= 0) put(cur, sum);
                    if (lane == 0) p.cnt[M.cnt0 + ct] = 0u;  // ready for the next launch
                }
            }
            if (++cu < wu1) cload();
        }
    }
    // copies still in flight land before the block exits (bounded)
    asm volatile("cp.async.wait_all;\n" ::: "memory");
    for (int i = done; i < copied; ++i) {
        s_wait(bar0 + 8 * cq, (phase >> cq) & 1u);
        phase ^= 1u << cq;
        cq = cq + 1 == NS ? 0 : cq + 1;
    }
}

}  // namespace

namespace {

int w_kind(int bits) {
    const int W = width_of(bits);
    return W == 2 ? 0 : W == 4 ? 1 : W == 1 ? 2 : 3;
}
int w_cols(int B) { return B <= 4 ? 2 * B : 8 * ((B + 7) / 8); }
// groups per slice: about 1 KB of codes per row, 16 warps sharing a slice's groups
int w_gs(int kind) { return kind == 0 ? 32 : kind == 1 ? 16 : kind == 2 ? 64 : 16; }

// Shared-memory row stride of a slice: the 2-bit path reads 8 bytes per lane
// (the rows of a half-warp start 8 banks apart), the 4-bit path 16 bytes (a
// quarter-warp's rows 16 banks apart), the 1-bit path 4 bytes (the warp's
// eight rows 4 banks apart), the 3-bit path three words (rows 48 mod 128
// bytes apart put a warp's reads on 32 banks).
int w_row_stride(int kind, int ng) {
    const int gb = w_gbytes(kind), bytes = std::min(ng, w_gs(kind)) * gb;
    const int want = kind == 0 ? 32 : kind == 1 ? 64 : kind == 2 ? 16 : 48;
    return bytes + (((want - bytes) % 128) + 128) % 128;
}

size_t w_frag_bytes(int ng, int B) { return (size_t)ng * w_cols(B) * 256 + (size_t)B * ng * 4; }

// ---- split products: host planning ----
// Groups per k-slice and k-slice count of a matrix of ng groups for split
// factor S (k-slices of whole chunks, except a matrix narrower than one).
void s_slices(int ng, int S, int kind, int &gk, int &nks) {
    const int gc = s_gc(kind);
    gk = (ng + S - 1) / S;
    gk = (gk + gc - 1) / gc * gc;
    if (gk > ng) gk = ng;
    nks = (ng + gk - 1) / gk;
}

size_t s_table_bytes(int kind) { return kind == 0 || kind == 1 ? 32768 : kind == 2 ? 2048 : 8192; }

// Fills p for the matrices sel[0..cnt) (one code width, one codebook, one
// batch class): picks the smallest split factor that gives a quarter of the
// grid's warps a unit (or splits as far as chunks allow) and whose every
// block range fits its fragments in shared memory. Returns the dynamic
// shared memory, or 0 if no split fits (the caller uses the sliced kernel).
size_t plan_split(SParams &p, const cq_gemv_desc *d, const int *idx, const int *sel, int cnt, const int *act_of,
                  const WAct *acts, int kind, bool g64, int grid, long long &part_floats, int &counters) {
    if (cnt > kSMaxMats) return 0;
    const size_t stages = (size_t)kSWarps * kSStages * s_stage_bytes(kind, g64);
    const size_t limit = 227 * 1024 - 6 * 1024;  // dynamic shared memory next to the static arrays
    if (s_table_bytes(kind) + stages >= limit) return 0;
    const size_t budget = limit - s_table_bytes(kind) - stages;
    const long long W = (long long)grid * kSWarps;
    static thread_local std::vector<int> gk, nks, tiles;
    static thread_local std::vector<long long> unit0;
    gk.resize(cnt);
    nks.resize(cnt);
    tiles.resize(cnt);
    unit0.resize(cnt + 1);
    for (int S = 1; S <= 1024; S *= 2) {
        long long U = 0;
        bool more = false;  // a larger S would split some matrix further
        for (int j = 0; j < cnt; ++j) {
            const cq_gemv_desc &D = d[idx[sel[j]]];
            const int ng = in_padded(D.in) / kGroup;
            // at most 16 partial sums per lane for the tile's last k-slice to add
            const int cap = std::max(1, 16 / ((16 * D.B + 31) / 32));
            const int Sj = std::min(S, cap);
            s_slices(ng, Sj, kind, gk[j], nks[j]);
            int g2, n2;
            s_slices(ng, std::min(2 * S, cap), kind, g2, n2);
            more |= n2 > nks[j];
            tiles[j] = (D.out + 15) / 16;
            unit0[j] = U;
            U += (long long)tiles[j] * nks[j];
        }
        unit0[cnt] = U;
        // a unit ends in a fence and an atomic when its matrix is k-sliced,
        // so slices stop once a quarter of the warps have a unit
        if (4 * U < W && more) continue;
        // every block's range: its (matrix, k-slice) pairs and their fragments
        bool fits = true;
        for (int b = 0; b < grid && fits; ++b) {
            const long long c0 = U * b / grid, c1 = U * (b + 1) / grid;
            long long u = c0;
            int m = 0, pairs = 0, pm = -1, ps = -1;
            size_t bytes = 0;
            while (u < c1) {
                while (unit0[m + 1] <= u) ++m;
                const int s = (int)((u - unit0[m]) / tiles[m]);
                const cq_gemv_desc &D = d[idx[sel[m]]];
                const int ng = in_padded(D.in) / kGroup, gn = std::min(gk[m], ng - s * gk[m]);
                const WAct &A = acts[act_of[sel[m]]];
                const bool same = pm >= 0 && act_of[sel[pm]] == act_of[sel[m]] && ps == s && gk[pm] == gk[m];
                if (!same) bytes += (size_t)gn * A.cols * 256 + (size_t)A.B * gn * 4;
                pm = m;
                ps = s;
                ++pairs;
                u = std::min(c1, unit0[m] + (long long)(s + 1) * tiles[m]);
            }
            fits = pairs <= kSMaxPairs && bytes <= budget;
        }
        if (!fits) {
            if (!more) return 0;
            continue;
        }
        // accepted: the parameter block
        p.n_mats = cnt;
        p.total_units = U;
        for (int j = 0; j < cnt; ++j) {
            const int ii = sel[j];
            const cq_gemv_desc &D = d[idx[ii]];
            const WAct &A = acts[act_of[ii]];
            const int W_ = width_of(D.bits), ng = in_padded(D.in) / kGroup;
            SMat &M = p.m[j];
            M.codes = D.blob;
            M.norms = reinterpret_cast<const __half *>(D.blob + (size_t)D.out * in_padded(D.in) * W_ / 8);
            M.y = D.y;
            M.xs = D.x_scale;
            M.unit0 = unit0[j];
            M.x = D.x;
            M.act = act_of[ii];
            M.in = D.in;
            M.out = D.out;
            M.ng = ng;
            M.B = D.B;
            M.xdt = D.x_dtype;
            M.cols = A.cols;
            M.tiles = tiles[j];
            M.nks = nks[j];
            M.gk = gk[j];
            M.cnt0 = 0;
            M.part0 = 0;
            if (nks[j] > 1) {
                M.cnt0 = counters;
                counters += tiles[j];
                M.part0 = part_floats / (16 * D.B);  // slots of 16 * B floats
                if (part_floats % (16 * D.B)) {      // align the matrix's first slot
                    M.part0 += 1;
                    part_floats = M.part0 * 16 * D.B;
                }
                part_floats += (long long)tiles[j] * nks[j] * 16 * D.B;
            }
            p.units_before[j] = unit0[j];
        }
        p.units_before[cnt] = U;
        p.smem_frag = (int)s_table_bytes(kind);
        p.frag_budget = (int)budget;
        p.smem_stage = (int)(s_table_bytes(kind) + budget);
        return (size_t)p.smem_stage + stages;
    }
    return 0;
}

template <int KIND, bool G64>
int s_launch(const SParams &p, int grid, size_t smem, cudaStream_t st) {
    auto k = gemv_split_kernel<KIND, G64>;
    const int rc = ensure_smem(reinterpret_cast<const void *>(k), smem);
    if (rc) return rc;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kSThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    cudaLaunchKernelEx(&cfg, k, p);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return set_error(CQ_ERR_CUDA, "split gemv launch: %s", cudaGetErrorString(e));
    return CQ_OK;
}

template <int NB, bool HILO>
int w_launch(WParams &p, int grid, size_t smem, cudaStream_t st) {
    auto k = gemv_wide_kernel<NB, HILO>;
    const int rc = ensure_smem(reinterpret_cast<const void *>(k), smem);
    if (rc) return rc;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kWGThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    cudaLaunchKernelEx(&cfg, k, p);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return set_error(CQ_ERR_CUDA, "wide gemv launch: %s", cudaGetErrorString(e));
    return CQ_OK;
}

}  // namespace

bool gemv_wide_eligible(const cq_gemv_desc &d) {
    if (d.in <= 0 || d.out <= 0 || d.B < 1 || d.B > kWMaxB) return false;
    const int W = width_of(d.bits), ng = in_padded(d.in) / kGroup;
    if (W < 1 || W > 4 || ng > 128) return false;
    // groups of 64 in whole 128-spans: the split products only (batches up
    // to 4, 1-, 2- and 4-bit codes)
    if (d.group == kGroup64) return d.in % kGroup == 0 && d.B <= 4 && W != 3;
    return d.group == kGroup && w_frag_bytes(ng, d.B) <= (size_t)kWFragBudget;
}

int launch_gemv_wide(const cq_gemv_desc *d, const int *idx, int n, void *stream, int *rejected, int *n_rejected) {
    *n_rejected = 0;
    if (n <= 0) return CQ_OK;
    static thread_local WActParams ap;  // large: off the stack, one per host thread
    static thread_local WParams wp;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    // ---- the distinct activations of the call (descriptors reading the
    // same activation share one rotation) ----
    int act_of[CQ_MAX_GROUPED];
    int n_act = 0;
    static thread_local WAct acts[CQ_MAX_GROUPED];
    for (int ii = 0; ii < n; ++ii) {
        const cq_gemv_desc &D = d[idx[ii]];
        int a = -1;
        for (int j = 0; j < n_act; ++j)
            if (acts[j].x == D.x && acts[j].xs == D.x_scale && acts[j].xdt == D.x_dtype && acts[j].in == D.in &&
                acts[j].B == D.B && acts[j].g64 == (D.group == kGroup64))
                a = j;
        if (a < 0) {
            WAct &A = acts[n_act];
            A.x = D.x;
            A.xs = D.x_scale;
            A.xdt = D.x_dtype;
            A.in = D.in;
            A.ng = in_padded(D.in) / kGroup;
            A.B = D.B;
            A.g64 = D.group == kGroup64;
            A.cols = w_cols(D.B);
            A.frag = A.ginv = 0;
            a = n_act++;
        }
        act_of[ii] = a;
    }
    // ---- the split launches: one per (batch class, code width, group,
    // codebook); what does not fit them goes to the sliced kernel (groups of
    // 128) or back to the caller (groups of 64) ----
    struct Plan {
        int kind;
        bool g64;
        size_t smem;
    };
    static thread_local std::vector<SParams> plans;
    std::vector<Plan> meta;
    bool sliced[CQ_MAX_GROUPED] = {};
    const int grid = sm_count();
    long long part_floats = 0;
    int counters = 0;
    {
        bool taken[CQ_MAX_GROUPED] = {};
        for (int ii = 0; ii < n; ++ii) {
            if (taken[ii]) continue;
            const cq_gemv_desc &D0 = d[idx[ii]];
            const int cls = D0.B <= 4 ? 0 : D0.B <= 8 ? 1 : 2, kind = w_kind(D0.bits);
            const bool g64 = D0.group == kGroup64;
            float lv0[16];
            level_table(D0.bits, D0.codebook, lv0);
            int sel[CQ_MAX_GROUPED], cnt = 0;
            for (int jj = ii; jj < n; ++jj) {
                if (taken[jj]) continue;
                const cq_gemv_desc &D = d[idx[jj]];
                const int c2 = D.B <= 4 ? 0 : D.B <= 8 ? 1 : 2;
                if (c2 != cls || w_kind(D.bits) != kind || (D.group == kGroup64) != g64) continue;
                float lv[16];
                level_table(D.bits, D.codebook, lv);
                bool same = true;
                for (int k = 0; k < 16; ++k)
                    same &= __half_as_ushort(__float2half_rn(lv[k])) == __half_as_ushort(__float2half_rn(lv0[k]));
                if (!same) continue;
                taken[jj] = true;
                sel[cnt++] = jj;
            }
            // the split products serve batches of up to 4; larger batches run
            // faster on the sliced kernel
            if (cls != 0) {  // never groups of 64 (see gemv_wide_eligible)
                for (int j = 0; j < cnt; ++j) sliced[sel[j]] = true;
                continue;
            }
            for (int b0 = 0; b0 < cnt; b0 += kSMaxMats) {
                const int c = std::min(kSMaxMats, cnt - b0);
                if (plans.size() <= meta.size()) plans.resize(meta.size() + 1);
                SParams &P = plans[meta.size()];
                const size_t smem =
                    plan_split(P, d, idx, sel + b0, c, act_of, acts, kind, g64, grid, part_floats, counters);
                if (!smem) {
                    for (int j = 0; j < c; ++j) {
                        if (g64) rejected[(*n_rejected)++] = idx[sel[b0 + j]];
                        else sliced[sel[b0 + j]] = true;
                    }
                    continue;
                }
                for (int k = 0; k < 16; ++k) P.lut[k] = __float2half_rn(lv0[k]);
                meta.push_back({kind, g64, smem});
            }
        }
    }
    // ---- workspace: the fragments of the activations that the sliced
    // kernel reads (the split products rotate their own), then 1/sigma and
    // the split products' partial sums; the tile counters live apart,
    // zeroed when allocated and left zero by every launch ----
    bool need[CQ_MAX_GROUPED] = {};
    for (int ii = 0; ii < n; ++ii)
        if (sliced[ii]) need[act_of[ii]] = true;
    long long words = 0, floats = 0;
    for (int a = 0; a < n_act; ++a) {
        if (!need[a]) continue;
        acts[a].frag = words;
        acts[a].ginv = floats;
        words += (long long)acts[a].ng * acts[a].cols * 64;
        floats += (long long)acts[a].B * acts[a].ng;
    }
    int err = 0;
    const size_t ws_bytes = (size_t)words * 4 + (size_t)floats * 4 + (size_t)part_floats * 4 + 64;
    uint8_t *ws = static_cast<uint8_t *>(stream_workspace(stream, 2, ws_bytes, &err));
    if (!ws) return err;
    uint32_t *frag = reinterpret_cast<uint32_t *>(ws);
    float *ginv = reinterpret_cast<float *>(ws + (size_t)words * 4);
    float *part = ginv + floats;
    unsigned int *cnt = nullptr;
    if (counters) {
        cnt = stream_counters(stream, (size_t)counters, &err);
        if (!cnt) return err;
    }
    // ---- 1. one rotation launch per kWMaxActs activations of the sliced kernel ----
    {
        int sel_act[CQ_MAX_GROUPED], na = 0;
        for (int a = 0; a < n_act; ++a)
            if (need[a]) sel_act[na++] = a;
        for (int a0 = 0; a0 < na; a0 += kWMaxActs) {
            const int c = std::min(kWMaxActs, na - a0);
            ap.n = c;
            ap.frag = frag;
            ap.ginv = ginv;
            int tasks = 0;
            for (int j = 0; j < c; ++j) {
                ap.a[j] = acts[sel_act[a0 + j]];
                ap.task0[j] = tasks;
                tasks += ap.a[j].ng * ap.a[j].B;
            }
            ap.task0[c] = tasks;
            act_frag_kernel<<<(tasks + kWWarps - 1) / kWWarps, kWThreads, 0, st>>>(ap);
            const cudaError_t e = cudaGetLastError();
            if (e != cudaSuccess) return set_error(CQ_ERR_CUDA, "activation rotation launch: %s", cudaGetErrorString(e));
        }
    }
    // ---- 2. the split products ----
    for (size_t k = 0; k < meta.size(); ++k) {
        SParams &P = plans[k];
        P.part = part;
        P.cnt = cnt;
        P.status = device_status_ptr();
        const bool g64 = meta[k].g64;
        const size_t smem = meta[k].smem;
        int rc = CQ_OK;
        switch (meta[k].kind) {
        case 0: rc = g64 ? s_launch<0, true>(P, grid, smem, st) : s_launch<0, false>(P, grid, smem, st); break;
        case 1: rc = g64 ? s_launch<1, true>(P, grid, smem, st) : s_launch<1, false>(P, grid, smem, st); break;
        case 2: rc = g64 ? s_launch<2, true>(P, grid, smem, st) : s_launch<2, false>(P, grid, smem, st); break;
        default: rc = s_launch<3, false>(P, grid, smem, st); break;  // 3-bit codes: group 128 only
        }
        if (rc) return rc;
    }
    // ---- 3. the rest: the sliced products, one launch per batch class ----
    for (int cls = 0; cls < 3; ++cls) {
        int sel[CQ_MAX_GROUPED], ns = 0;
        for (int ii = 0; ii < n; ++ii) {
            const int B = d[idx[ii]].B, c = B <= 4 ? 0 : B <= 8 ? 1 : 2;
            if (c == cls && sliced[ii]) sel[ns++] = ii;
        }
        for (int base = 0; base < ns; base += kWMaxMats) {
            const int cnt = std::min(kWMaxMats, ns - base);
            WParams &p = wp;
            int tiles = 0, nlut = 0;
            size_t frag_max = 0, stage_max = 0, red_max = 0;
            for (int j = 0; j < cnt; ++j) {
                const int ii = sel[base + j];
                const cq_gemv_desc &D = d[idx[ii]];
                const int kind = w_kind(D.bits), ng = in_padded(D.in) / kGroup, W = width_of(D.bits);
                WMat &M = p.m[j];
                M.codes = D.blob;
                M.norms = reinterpret_cast<const __half *>(D.blob + (size_t)D.out * in_padded(D.in) * W / 8);
                M.y = D.y;
                M.xs = D.x_scale;
                M.out = D.out;
                M.ng = ng;
                M.B = D.B;
                M.xdt = D.x_dtype;
                M.kind = kind;
                M.act = act_of[ii];
                M.gs = std::min(ng, w_gs(kind));
                M.rs = w_row_stride(kind, ng);
                float lv[16];
                level_table(D.bits, D.codebook, lv);
                __half lut[16];
                for (int k = 0; k < 16; ++k) lut[k] = __float2half_rn(lv[k]);
                int li = -1;
                for (int q = 0; q < nlut; ++q) {
                    bool same = true;
                    for (int k = 0; k < 16; ++k) same &= __half_as_ushort(p.lut[q][k]) == __half_as_ushort(lut[k]);
                    if (same) li = q;
                }
                if (li < 0) {
                    if (nlut == kMaxLuts) return set_error(CQ_ERR_ARG, "more than %d distinct codebooks in one call", kMaxLuts);
                    for (int k = 0; k < 16; ++k) p.lut[nlut][k] = lut[k];
                    li = nlut++;
                }
                M.lut = li;
                const WAct &A = acts[M.act];
                p.act_frag[j] = A.frag;
                p.act_ginv[j] = A.ginv;
                p.act_cols[j] = A.cols;
                p.tiles_before[j] = tiles;
                tiles += (D.out + 15) / 16;
                frag_max = std::max(frag_max, w_frag_bytes(ng, D.B));
                stage_max = std::max(stage_max, (size_t)16 * M.rs + 32 * (size_t)ng);
                red_max = std::max(red_max, (size_t)kWGWarps * 16 * D.B * sizeof(float));
            }
            p.n_mats = cnt;
            p.total_tiles = tiles;
            p.tiles_before[cnt] = tiles;
            p.frag = frag;
            p.ginv = ginv;
            size_t off = 32 * 1024;  // the level table at offset 0 (the largest: 32 KB)
            auto place = [&](int &field, size_t bytes) {
                field = (int)off;
                off += (bytes + 127) / 128 * 128;
            };
            place(p.smem_frag, frag_max);
            place(p.smem_red, red_max);
            p.stage_bytes = (int)((stage_max + 127) / 128 * 128);
            // as many stages as fit (the copies in flight hide the memory latency)
            const size_t budget = 225 * 1024;
            p.n_stages = (int)std::min<size_t>(kWMaxStages, off < budget ? (budget - off) / p.stage_bytes : 0);
            if (p.n_stages < 2) return set_error(CQ_ERR_SHAPE, "wide GEMV: shared memory for fewer than two stages");
            place(p.smem_stage, (size_t)p.n_stages * p.stage_bytes);
            p.status = device_status_ptr();
            const size_t smem = off;
            const int grid = std::min(tiles, sm_count());
            int rc = CQ_OK;
            if (cls == 0) rc = w_launch<1, true>(p, grid, smem, st);
            else if (cls == 1) rc = w_launch<1, false>(p, grid, smem, st);
            else rc = w_launch<2, false>(p, grid, smem, st);
            if (rc) return rc;
        }
    }
    return CQ_OK;
}

}  // namespace cq
