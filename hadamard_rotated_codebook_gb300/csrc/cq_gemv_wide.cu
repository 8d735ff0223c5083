// cq_gemv_wide.cu -- tensor-core GEMV over CQ-packed weights for wide inputs
// (16 groups and more) and for batches of 5 to 16: every code width at
// group 128.
//
// Per group g of 128 inputs the product is the rotated-domain identity
// (OpenNeedle docs/reference.md; "The .cact archive and Cactus Quants",
// "Reconstructing one group"):
//     y[b][o] = sum_g n[o][g] * sum_k c[q[o,g,k]] * z[b,g,k],   z = H x (per group).
//
// Two launches per call.
//  1. act_frag_kernel rotates every distinct activation of the call once:
//     one warp per (activation, group, batch row) computes z = H0 x with the
//     FWHT in registers and writes its fp16 terms straight into the MMA B
//     fragment layout in a workspace (a lane's four positions are exactly
//     two fragment words, so no shuffles are needed), with 1/sigma per
//     (batch row, group).
//  2. gemv_wide_kernel, launched as a programmatic dependent of the first:
//     one block per SM walks an equal run of the call's 16-row tiles.
//     Before it waits for the rotation it builds its level table and starts
//     its code copies; then it copies the fragments of its matrix's
//     activation into shared memory once, and streams the tiles through four
//     shared-memory stages in slices of about 512 code bytes per row. The
//     eight warps split a slice's groups: each expands its groups' code bytes
//     to fp16 levels through the replicated byte -> levels table (the A
//     operand of mma.sync m16n8k16, fp32 accumulation) and multiplies them
//     with the fragments of every batch row; a tile's partial sums meet in
//     shared memory.
//
// Precision. Batches of 1 to 4 carry z as fp16 hi + lo terms (two MMA
// columns per batch row, z to ~2^-22 relative). Batches of 5 to 16 carry z as
// one fp16 term (one column per batch row, relative error <= 2^-11, the same
// order as the fp16 rounding of the levels), which halves the MMAs; both are
// far inside the product tolerance |y - y_ref| <= 2e-3 sum |w||x|.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>

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
// of them are free of bank conflicts.
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
// its own copy (conflict-free whatever the codes): 2-bit codes a byte -> four
// fp16 levels (16 copies of 8 bytes), 4-bit codes a byte -> two levels (32
// copies of 4 bytes), 1-bit codes a nibble -> four levels (16 copies), 3-bit
// codes a 6-bit pair -> two levels (32 copies).
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
// row gq+8 positions 2-3}, through the replicated level tables.
template <int KIND>
__device__ __forceinline__ void w_decode(const WCodes &c, int nu, const uint8_t *tab, int lane, uint32_t (&a)[4]) {
    if (KIND == 0) {  // byte nu of the lane's 8 -> four levels
        const uint2 *tb = reinterpret_cast<const uint2 *>(tab) + (lane & 15);
        const uint2 er = tb[__byte_perm(c.r[nu >> 2], 0, 0x4440 + (nu & 3)) * 16];
        const uint2 es = tb[__byte_perm(c.s[nu >> 2], 0, 0x4440 + (nu & 3)) * 16];
        a[0] = er.x, a[1] = es.x, a[2] = er.y, a[3] = es.y;
    } else if (KIND == 1) {  // bytes 2nu, 2nu+1 of the lane's 16 -> two levels each
        const uint32_t *tb = reinterpret_cast<const uint32_t *>(tab) + lane;
        const uint32_t r = c.r[nu >> 1] >> (16 * (nu & 1)), s = c.s[nu >> 1] >> (16 * (nu & 1));
        a[0] = tb[(r & 0xffu) * 32], a[2] = tb[((r >> 8) & 0xffu) * 32];
        a[1] = tb[(s & 0xffu) * 32], a[3] = tb[((s >> 8) & 0xffu) * 32];
    } else if (KIND == 2) {  // nibble nu of the lane's 4 bytes -> four levels
        const uint2 *tb = reinterpret_cast<const uint2 *>(tab) + (lane & 15);
        const uint2 er = tb[((c.r[0] >> (4 * nu)) & 15u) * 16], es = tb[((c.s[0] >> (4 * nu)) & 15u) * 16];
        a[0] = er.x, a[1] = es.x, a[2] = er.y, a[3] = es.y;
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
    if (d.group != kGroup || d.in <= 0 || d.out <= 0 || d.B < 1 || d.B > kWMaxB) return false;
    const int W = width_of(d.bits), ng = in_padded(d.in) / kGroup;
    if (W < 1 || W > 4 || ng > 128) return false;
    return w_frag_bytes(ng, d.B) <= (size_t)kWFragBudget;
}

int launch_gemv_wide(const cq_gemv_desc *d, const int *idx, int n, void *stream) {
    if (n <= 0) return CQ_OK;
    static thread_local WActParams ap;  // large: off the stack, one per host thread
    static thread_local WParams wp;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    // ---- the distinct activations of the call (consecutive descriptors
    // reading the same activation share one rotation) ----
    int act_of[CQ_MAX_GROUPED];
    int n_act = 0;
    long long words = 0, floats = 0;
    static thread_local WAct acts[CQ_MAX_GROUPED];
    for (int ii = 0; ii < n; ++ii) {
        const cq_gemv_desc &D = d[idx[ii]];
        int a = -1;
        for (int j = 0; j < n_act; ++j)
            if (acts[j].x == D.x && acts[j].xs == D.x_scale && acts[j].xdt == D.x_dtype && acts[j].in == D.in &&
                acts[j].B == D.B)
                a = j;
        if (a < 0) {
            WAct &A = acts[n_act];
            A.x = D.x;
            A.xs = D.x_scale;
            A.xdt = D.x_dtype;
            A.in = D.in;
            A.ng = in_padded(D.in) / kGroup;
            A.B = D.B;
            A.cols = w_cols(D.B);
            A.frag = words;
            A.ginv = floats;
            words += (long long)A.ng * A.cols * 64;
            floats += (long long)A.B * A.ng;
            a = n_act++;
        }
        act_of[ii] = a;
    }
    int err = 0;
    const size_t ws_bytes = (size_t)words * 4 + (size_t)floats * 4 + 16;
    uint8_t *ws = static_cast<uint8_t *>(stream_workspace(stream, 2, ws_bytes, &err));
    if (!ws) return err;
    uint32_t *frag = reinterpret_cast<uint32_t *>(ws);
    float *ginv = reinterpret_cast<float *>(ws + (size_t)words * 4);
    // ---- 1. one rotation launch per kWMaxActs activations ----
    for (int a0 = 0; a0 < n_act; a0 += kWMaxActs) {
        const int cnt = std::min(kWMaxActs, n_act - a0);
        ap.n = cnt;
        ap.frag = frag;
        ap.ginv = ginv;
        int tasks = 0;
        for (int j = 0; j < cnt; ++j) {
            ap.a[j] = acts[a0 + j];
            ap.task0[j] = tasks;
            tasks += acts[a0 + j].ng * acts[a0 + j].B;
        }
        ap.task0[cnt] = tasks;
        act_frag_kernel<<<(tasks + kWWarps - 1) / kWWarps, kWThreads, 0, st>>>(ap);
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return set_error(CQ_ERR_CUDA, "activation rotation launch: %s", cudaGetErrorString(e));
    }
    // ---- 2. the products: one launch per batch class, kWMaxMats matrices each ----
    for (int cls = 0; cls < 3; ++cls) {
        int sel[CQ_MAX_GROUPED], ns = 0;
        for (int ii = 0; ii < n; ++ii) {
            const int B = d[idx[ii]].B, c = B <= 4 ? 0 : B <= 8 ? 1 : 2;
            if (c == cls) sel[ns++] = ii;
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
