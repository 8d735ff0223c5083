// cq_encode.cu -- CQ encoder and per-token int8 activation quantiser.
//
// Encoder ("The .cact format", "Cactus Quants"; OpenNeedle docs/reference.md,
// CQ quantisation): per group of 128 weights along the input axis,
//   r = w . H (normalised Sylvester Hadamard), n = fp32 |r|,
//   u = r / max(n, 1e-12), q_k = nearest level (ties -> smaller index),
//   store fp16(n) and the codes as an LSB-first bitstream per row.
//
// GB300 mapping. The encoder streams 4 bytes in per weight and writes
// ~0.27 bytes out, so it is bound by HBM; the arithmetic per weight (7
// butterfly adds, a scale, the level search, packing) must stay inside the
// issue budget that leaves. A CTA of 256 threads stages 128 groups (64 KB)
// in shared memory with coalesced 16-byte loads; two threads own one group,
// 64 values each, split on bit 2 of the coordinate. Each thread reads its
// 16 chunks of 16 bytes with an XOR swizzle (chunk 2*(j^f)+h, f = pair&3)
// that keeps every quarter-warp on 8 distinct bank groups. The swizzle
// permutes the inputs of the transform by XOR, which only flips the signs
// of outputs (H(x o xor_f) = diag((-1)^<f,m>) H x); the sign is folded into
// the per-coordinate scale. Six butterfly stages run in registers and one
// across the thread pair with a shuffle.
//
// Exactness. Codes: the nearest-level search in fp32 with ties to the
// smaller index is a step function of u whose steps sit at fixed fp32
// thresholds T_j (the first u with fl(c_{j+1}-u) < fl(u-c_j)); each CTA finds
// them once by bisection over the ordered fp32 values, then the code is the
// number of thresholds <= u. Norms: the fp16 norm must equal
// fp16(fp32(sqrt(sum w^2))) exactly (the sum of squares is the same on both
// sides of the rotation). A pairwise fp32 sum has relative error below
// 8 * 2^-24; when every value within 5e-7 of the fp32 estimate rounds to the
// same fp16 the result is certain, otherwise (about 0.2% of groups) the
// group recomputes the sum in fp64 from exact products.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <atomic>

#include "cq_internal.h"

namespace cq {
namespace {

constexpr int kEncThreads = 256;
constexpr int kEncWarps = kEncThreads / 32;                    // 8
constexpr int kEncWarpGroups = 16;                             // groups per warp tile (a thread pair each)
constexpr int kEncWarpFloats = kEncWarpGroups * kGroup;        // 2048 floats = 8 KB
constexpr int kEncTileFloats = kEncWarps * kEncWarpFloats;     // 64 KB of staging per CTA
constexpr float kInvSqrt128 = 0.08838834764831845f;            // 1/sqrt(128)

struct EncodeParams {
    const float *W;
    uint8_t *codes;
    __half *norms;
    unsigned int *status;  // device status word (bounded waits)
    long long n_groups;  // out * ng
    int in, ng;
    float cb[kMaxLevels];
};

// Order-preserving map from fp32 (non-NaN) to uint32 and back.
__device__ __forceinline__ uint32_t ord_key(float f) {
    uint32_t b = __float_as_uint(f);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float key_float(uint32_t k) {
    uint32_t b = (k & 0x80000000u) ? (k & 0x7fffffffu) : ~k;
    return __uint_as_float(b);
}

// First fp32 u in (a, b] at which level b is strictly nearer than level a
// under fp32 subtraction; below it the tie rule keeps the smaller index.
__device__ float decision_threshold(float a, float b) {
    uint32_t lo = ord_key(a), hi = ord_key(b);
    while (hi - lo > 1u) {
        uint32_t mid = lo + (hi - lo) / 2u;
        float u = key_float(mid);
        if (__fsub_rn(b, u) < __fsub_rn(u, a))
            hi = mid;
        else
            lo = mid;
    }
    return key_float(hi);
}

template <int L>
__device__ __forceinline__ int level_index(float u, const float (&T)[16]) {
    if (L == 4) {
        // two-step search over 3 thresholds
        return u >= T[1] ? (u >= T[2] ? 3 : 2) : (u >= T[0] ? 1 : 0);
    } else {
        int q = 0;
#pragma unroll
        for (int j = 0; j < L - 1; ++j) q += (u >= T[j]) ? 1 : 0;
        return q;
    }
}

// BITS: 2, 3, 4 or 5 (ternary). ALIGNED: in % 128 == 0 and W 16-byte aligned,
// so the groups of the matrix form one contiguous fp32 array.
//
// Every warp works on its own: it owns an 8 KB staging buffer and an
// mbarrier, takes tiles of 16 consecutive groups (one per thread pair) in a
// grid-stride order, and issues the next tile's copy as soon as its own 32
// threads hold the current one in registers. No barrier spans more than one
// warp, so a slow warp delays nobody else's copy.
template <int BITS, bool ALIGNED>
__global__ void __launch_bounds__(kEncThreads, 2) encode_kernel(const __grid_constant__ EncodeParams p) {
    constexpr int L = BITS == 5 ? 3 : (1 << BITS);
    constexpr int W = BITS == 5 ? 2 : BITS;  // code width
    extern __shared__ float4 smem4[];
    __shared__ float s_thr[16];
    __shared__ __align__(8) uint64_t s_bar[kEncWarps];  // aligned rows: each warp's bulk copy

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid < L - 1) s_thr[tid] = decision_threshold(p.cb[tid], p.cb[tid + 1]);
    const uint32_t bar = (uint32_t)__cvta_generic_to_shared(&s_bar[warp]);
    if (ALIGNED && lane == 0) {
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;\n" ::"r"(bar));
        asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    }
    __syncthreads();
    float T[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) T[j] = j < L - 1 ? s_thr[j] : 0.0f;

    const int pair = lane >> 1, h = lane & 1, f = pair & 3;
    float4 *buf = smem4 + warp * (kEncWarpFloats / 4);
    float *tile = reinterpret_cast<float *>(buf);
    const long long n_tiles = (p.n_groups + kEncWarpGroups - 1) / kEncWarpGroups;
    const long long first = (long long)blockIdx.x * kEncWarps + warp;
    const long long stride = (long long)gridDim.x * kEncWarps;

    // Aligned rows: the tile's groups are one contiguous block of W, staged by
    // one bulk copy (TMA engine) that completes on the warp's mbarrier.
    // Groups past the end of the matrix are not copied (their codes are
    // never stored).
    auto stage = [&](long long tt) {
        const long long gs = tt * kEncWarpGroups;
        const long long ngrp = p.n_groups - gs < kEncWarpGroups ? p.n_groups - gs : kEncWarpGroups;
        const uint32_t bytes = (uint32_t)ngrp * kGroup * 4;
        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(bar), "r"(bytes) : "memory");
        asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(
                         (uint32_t)__cvta_generic_to_shared(buf)),
                     "l"(p.W + gs * kGroup), "r"(bytes), "r"(bar)
                     : "memory");
    };
    if (ALIGNED && lane == 0 && first < n_tiles) stage(first);
    uint32_t phase = 0;  // parity of the bulk copy being waited for

    for (long long t = first; t < n_tiles; t += stride) {
        const long long g0 = t * kEncWarpGroups;
        // ---- stage 16 groups into the warp's buffer ----
        if (ALIGNED) {
            // bounded wait for the tile's bulk copy (on expiry the status word records it)
            bool done = false;
            for (unsigned i = 0; i < (1u << 24) && !done; ++i) {
                uint32_t ok;
                asm volatile(
                    "{\n .reg .pred q;\n mbarrier.try_wait.parity.shared::cta.b64 q, [%1], %2;\n selp.u32 %0, 1, 0, q;\n}\n"
                    : "=r"(ok)
                    : "r"(bar), "r"(phase)
                    : "memory");
                done = ok != 0;
            }
            if (!done && lane == 0 && p.status) atomicOr(p.status, 0x45430001u);
            phase ^= 1u;
        } else {
            for (int i = lane; i < kEncWarpFloats; i += 32) {
                const long long G = g0 + i / kGroup;
                float v = 0.0f;
                if (G < p.n_groups) {
                    const long long o = G / p.ng;
                    const int col = (int)(G - o * p.ng) * kGroup + (i % kGroup);
                    if (col < p.in) v = __ldcs(p.W + o * p.in + col);
                }
                tile[i] = v;
            }
            __syncwarp();
        }

        const long long G = g0 + pair;
        // ---- load: register 4j+e = coordinate c = 8(j^f)+4h+e after the
        // butterfly on coordinate bit 2, done here from both halves of the
        // group (the partner's half a second read of shared memory). The
        // transform's stages commute, so taking this one first leaves the
        // result exact up to rounding order. Squares use the original values.
        float x[64];
        float sq[32];
        const float sg = h ? -1.0f : 1.0f;  // h = 0: a + b;  h = 1: b - a  (fma by +-1 is exact)
        const float4 *grp = buf + pair * (kGroup / 4);
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            const float4 a = grp[2 * (j ^ f) + h];
            const float4 b = grp[2 * (j ^ f) + (h ^ 1)];
            sq[2 * j] = __fadd_rn(__fmul_rn(a.x, a.x), __fmul_rn(a.y, a.y));
            sq[2 * j + 1] = __fadd_rn(__fmul_rn(a.z, a.z), __fmul_rn(a.w, a.w));
            x[4 * j + 0] = __fmaf_rn(sg, a.x, b.x);
            x[4 * j + 1] = __fmaf_rn(sg, a.y, b.y);
            x[4 * j + 2] = __fmaf_rn(sg, a.z, b.z);
            x[4 * j + 3] = __fmaf_rn(sg, a.w, b.w);
        }
        __syncwarp();  // the warp's buffer may be overwritten from here on
        if (ALIGNED && lane == 0 && t + stride < n_tiles) stage(t + stride);

        // ---- sum of squares, pairwise in fp32 ----
#pragma unroll
        for (int w = 16; w >= 1; w >>= 1)
#pragma unroll
            for (int i = 0; i < w; ++i) sq[i] = __fadd_rn(sq[i], sq[i + w]);
        const float s32 = __fadd_rn(sq[0], __shfl_xor_sync(0xffffffffu, sq[0], 1));

        // ---- fast Walsh-Hadamard transform: the other 6 stages in registers ----
#pragma unroll
        for (int bit = 1; bit < 64; bit <<= 1)
#pragma unroll
            for (int r = 0; r < 64; ++r)
                if (!(r & bit)) {
                    float a = x[r], b = x[r | bit];
                    x[r] = __fadd_rn(a, b);
                    x[r | bit] = __fsub_rn(a, b);
                }

        // ---- fp32 group norm, exact fp16 storage ----
        float n32 = __fsqrt_rn(s32);
        bool sure = s32 >= 1e-30f && s32 <= 1e30f;
        if (sure) {
            __half lo = __float2half_rn(__fmul_rn(n32, 1.0f - 5e-7f));
            __half hi = __float2half_rn(__fmul_rn(n32, 1.0f + 5e-7f));
            sure = __half_as_ushort(lo) == __half_as_ushort(hi);
        }
        // Both threads of a pair hold the same s32, hence the same verdict.
        const bool need64 = !sure;
        if (__any_sync(0xffffffffu, need64)) {
            // Rare path: exact products and an fp64 sum over the group's
            // original values, reread from global memory.
            double d = 0.0;
            if (need64 && G < p.n_groups) {
                const long long o = G / p.ng;
                const int gcol = (int)(G - o * p.ng) * kGroup;
#pragma unroll 4
                for (int j = 0; j < 16; ++j)
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int col = gcol + 8 * (j ^ f) + 4 * h + e;
                        const double w = col < p.in ? (double)p.W[o * p.in + col] : 0.0;
                        d = __fma_rn(w, w, d);
                    }
            }
            d += __shfl_xor_sync(0xffffffffu, d, 1);
            if (need64) n32 = __double2float_rn(__dsqrt_rn(d));
        }

        // ---- directions and codes ----
        const float den = fmaxf(n32, 1e-12f);
        const float sc = __fdiv_rn(kInvSqrt128, den);
        float scale4[4];
#pragma unroll
        for (int b = 0; b < 4; ++b) scale4[b] = (__popc(f & b) & 1) ? -sc : sc;

        uint32_t chunk[16];  // 4 codes (4W bits) per j
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            uint32_t c = 0;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float u = __fmul_rn(x[4 * j + e], scale4[j & 3]);
                int q = level_index<L>(u, T);
                if (BITS == 5) q = (q - 1) & 3;  // ternary crumb
                c |= (uint32_t)q << (W * e);
            }
            chunk[j] = c;
        }

        // ---- exchange: thread h writes coordinates [64h, 64h+64) = j in [8h, 8h+8) ----
        // (register-indexed selects keep the chunk array out of local memory)
        uint32_t send[4], recv[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t lo = h ? chunk[2 * i] : chunk[8 + 2 * i];
            const uint32_t hi = h ? chunk[2 * i + 1] : chunk[8 + 2 * i + 1];
            send[i] = lo | (hi << 16);
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) recv[i] = __shfl_xor_sync(0xffffffffu, send[i], 1);

        // block i (8 coordinates, 8W bits) = [thread-0 chunk | thread-1 chunk]
        uint32_t outw[2 * W];
#pragma unroll
        for (int k = 0; k < 2 * W; ++k) outw[k] = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint32_t mine = h ? chunk[8 + i] : chunk[i];
            const uint32_t theirs = (recv[i >> 1] >> (16 * (i & 1))) & 0xffffu;
            const uint32_t lo = h ? theirs : mine;  // coordinates 8j'+0..3 come from thread 0
            const uint32_t hi = h ? mine : theirs;
            const uint64_t blk = (uint64_t)lo | ((uint64_t)hi << (4 * W));
            const int bitpos = 8 * W * i;
            outw[bitpos / 32] |= (uint32_t)(blk << (bitpos % 32));
            if ((bitpos % 32) + 8 * W > 32) outw[bitpos / 32 + 1] |= (uint32_t)(blk >> (32 - bitpos % 32));
        }

        if (G < p.n_groups) {
            uint8_t *dst = p.codes + G * (16 * W) + h * (8 * W);
            if (W == 3) {
                uint2 *d2 = reinterpret_cast<uint2 *>(dst);
#pragma unroll
                for (int k = 0; k < 3; ++k) __stcs(d2 + k, make_uint2(outw[2 * k], outw[2 * k + 1]));
            } else {
                uint4 *d4 = reinterpret_cast<uint4 *>(dst);
#pragma unroll
                for (int k = 0; k < W / 2; ++k)
                    __stcs(d4 + k, make_uint4(outw[4 * k], outw[4 * k + 1], outw[4 * k + 2], outw[4 * k + 3]));
            }
            if (h == 0) p.norms[G] = __float2half_rn(n32);
        }
    }
}

// ---------------------------------------------- group 64, one thread each --
// A group of 64 fits in one thread's registers, so each lane of a warp takes
// one group of the warp's 32-group (8 KB) tile and keeps the transform, the
// norm and the packing to itself: no shuffles. Staging as in encode_kernel:
// a warp-private buffer, filled by one bulk copy on an mbarrier when the
// rows are 64-aligned. Lane l reads its 16-byte chunks in the order
// j ^ m, m = l & 7 (the 8 lanes of a quarter-warp then hit 8 different
// bank groups), so register 4j+e holds coordinate 4(j^m)+e. The transform
// over the register index then yields, in register s, the rotation's
// coordinate s times (-1)^popc((s >> 2) & m), since the Sylvester matrix
// satisfies H[s][c ^ d] = H[s][c] H[s][d].
template <int BITS, bool ALIGNED>
__global__ void __launch_bounds__(kEncThreads, 2) encode_g64_kernel(const __grid_constant__ EncodeParams p) {
    constexpr int L = BITS == 5 ? 3 : (1 << BITS);
    constexpr int W = BITS == 5 ? 2 : BITS;
    constexpr int TG = 32;             // groups per warp tile
    constexpr int TF = TG * kGroup64;  // 2048 floats = 8 KB
    static_assert(TF == kEncWarpFloats, "warp tile size");
    extern __shared__ float4 smem4[];
    __shared__ float s_thr[16];
    __shared__ __align__(8) uint64_t s_bar[kEncWarps];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid < L - 1) s_thr[tid] = decision_threshold(p.cb[tid], p.cb[tid + 1]);
    const uint32_t bar = (uint32_t)__cvta_generic_to_shared(&s_bar[warp]);
    if (ALIGNED && lane == 0) {
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;\n" ::"r"(bar));
        asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    }
    __syncthreads();
    float T[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) T[j] = j < L - 1 ? s_thr[j] : 0.0f;

    const int m = lane & 7;
    float4 *buf = smem4 + warp * (TF / 4);
    float *tile = reinterpret_cast<float *>(buf);
    const long long n_tiles = (p.n_groups + TG - 1) / TG;
    const long long first = (long long)blockIdx.x * kEncWarps + warp;
    const long long stride = (long long)gridDim.x * kEncWarps;

    auto stage = [&](long long tt) {
        const long long gs = tt * TG;
        const long long ngrp = p.n_groups - gs < TG ? p.n_groups - gs : TG;
        const uint32_t bytes = (uint32_t)ngrp * kGroup64 * 4;
        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(bar), "r"(bytes) : "memory");
        asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(
                         (uint32_t)__cvta_generic_to_shared(buf)),
                     "l"(p.W + gs * kGroup64), "r"(bytes), "r"(bar)
                     : "memory");
    };
    if (ALIGNED && lane == 0 && first < n_tiles) stage(first);
    uint32_t phase = 0;

    for (long long t = first; t < n_tiles; t += stride) {
        const long long g0 = t * TG;
        if (ALIGNED) {
            bool done = false;
            for (unsigned i = 0; i < (1u << 24) && !done; ++i) {
                uint32_t ok;
                asm volatile(
                    "{\n .reg .pred q;\n mbarrier.try_wait.parity.shared::cta.b64 q, [%1], %2;\n selp.u32 %0, 1, 0, q;\n}\n"
                    : "=r"(ok)
                    : "r"(bar), "r"(phase)
                    : "memory");
                done = ok != 0;
            }
            if (!done && lane == 0 && p.status) atomicOr(p.status, 0x45430001u);
            phase ^= 1u;
        } else {
            for (int i = lane; i < TF; i += 32) {
                const long long Gx = g0 + i / kGroup64;
                float v = 0.0f;
                if (Gx < p.n_groups) {
                    const long long o = Gx / p.ng;
                    const int col = (int)(Gx - o * p.ng) * kGroup64 + (i % kGroup64);
                    if (col < p.in) v = __ldcs(p.W + o * p.in + col);
                }
                tile[i] = v;
            }
            __syncwarp();
        }

        const long long Gi = g0 + lane;
        float x[64];
        float sq[32];
        const float4 *grp = buf + lane * (kGroup64 / 4);
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            const float4 v = grp[j ^ m];
            sq[2 * j] = __fadd_rn(__fmul_rn(v.x, v.x), __fmul_rn(v.y, v.y));
            sq[2 * j + 1] = __fadd_rn(__fmul_rn(v.z, v.z), __fmul_rn(v.w, v.w));
            x[4 * j + 0] = v.x;
            x[4 * j + 1] = v.y;
            x[4 * j + 2] = v.z;
            x[4 * j + 3] = v.w;
        }
        __syncwarp();  // the warp's buffer may be overwritten from here on
        if (ALIGNED && lane == 0 && t + stride < n_tiles) stage(t + stride);

        // sum of squares, a tree in fp32
#pragma unroll
        for (int w = 16; w >= 1; w >>= 1)
#pragma unroll
            for (int i = 0; i < w; ++i) sq[i] = __fadd_rn(sq[i], sq[i + w]);
        const float s32 = sq[0];

        // the 6-stage transform in registers
#pragma unroll
        for (int bit = 1; bit < 64; bit <<= 1)
#pragma unroll
            for (int r = 0; r < 64; ++r)
                if (!(r & bit)) {
                    const float a = x[r], b = x[r | bit];
                    x[r] = __fadd_rn(a, b);
                    x[r | bit] = __fsub_rn(a, b);
                }

        // fp32 norm; exact fp64 recount when its fp16 rounding is in doubt
        float n32 = __fsqrt_rn(s32);
        bool sure = s32 >= 1e-30f && s32 <= 1e30f;
        if (sure) {
            const __half lo = __float2half_rn(__fmul_rn(n32, 1.0f - 5e-7f));
            const __half hi = __float2half_rn(__fmul_rn(n32, 1.0f + 5e-7f));
            sure = __half_as_ushort(lo) == __half_as_ushort(hi);
        }
        if (!sure && Gi < p.n_groups) {
            const long long o = Gi / p.ng;
            const int gcol = (int)(Gi - o * p.ng) * kGroup64;
            double d = 0.0;
            for (int c = 0; c < kGroup64; ++c) {
                const double w = gcol + c < p.in ? (double)p.W[o * p.in + gcol + c] : 0.0;
                d = __fma_rn(w, w, d);
            }
            n32 = __double2float_rn(__dsqrt_rn(d));
        }

        // codes, LSB-first: coordinate s at bit W*s of the group's stream
        const float sc = __fdiv_rn(0.125f, fmaxf(n32, 1e-12f));  // 1/sqrt(64) over the norm
        float scale8[8];
#pragma unroll
        for (int b = 0; b < 8; ++b) scale8[b] = (__popc(b & m) & 1) ? -sc : sc;
        uint32_t outw[2 * W];
#pragma unroll
        for (int k = 0; k < 2 * W; ++k) outw[k] = 0;
#pragma unroll
        for (int s = 0; s < 64; ++s) {
            const float u = __fmul_rn(x[s], scale8[(s >> 2) & 7]);
            int q = level_index<L>(u, T);
            if (BITS == 5) q = (q - 1) & 3;  // ternary crumb
            const int bp = W * s;
            outw[bp / 32] |= (uint32_t)q << (bp % 32);
            if (bp % 32 + W > 32) outw[bp / 32 + 1] |= (uint32_t)q >> (32 - bp % 32);
        }
        if (Gi < p.n_groups) {
            uint8_t *dst = p.codes + Gi * (8 * W);
            if (W % 2 == 0) {
                uint4 *d4 = reinterpret_cast<uint4 *>(dst);
#pragma unroll
                for (int k = 0; k < W / 2; ++k)
                    __stcs(d4 + k, make_uint4(outw[4 * k], outw[4 * k + 1], outw[4 * k + 2], outw[4 * k + 3]));
            } else {
                uint2 *d2 = reinterpret_cast<uint2 *>(dst);
#pragma unroll
                for (int k = 0; k < W; ++k) __stcs(d2 + k, make_uint2(outw[2 * k], outw[2 * k + 1]));
            }
            p.norms[Gi] = __float2half_rn(n32);
        }
    }
}

// ------------------------------------------- binary codes at group 128 --
// One warp per 128 positions: a group of 128 (binary codes), or two groups
// of 64 (lanes 0-15 and 16-31, whose transforms stop before the stage that
// would mix them; groups of 64 normally take encode_g64_kernel). Lane l holds coordinates 4l..4l+3. Same steps as encode_kernel:
// fp32 sum of squares in a tree (fp64 recount near an fp16 rounding
// boundary), FWHT, u = r / n, threshold search, LSB-first packing.
template <int G, int BITS>
__global__ void __launch_bounds__(256) encode_warp_kernel(const __grid_constant__ EncodeParams p) {
    constexpr int L = BITS == 5 ? 3 : (1 << BITS);
    constexpr int W = BITS == 5 ? 2 : BITS;
    constexpr int HALF = G == 128 ? 32 : 16;  // lanes per group
    constexpr int PER = 128 / G;              // groups per warp task
    constexpr int NW = G * W / 32;            // code words per group
    __shared__ float s_thr[16];
    __shared__ uint32_t s_words[8][PER][NW + 1];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid < L - 1) s_thr[tid] = decision_threshold(p.cb[tid], p.cb[tid + 1]);
    __syncthreads();
    float T[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) T[j] = j < L - 1 ? s_thr[j] : 0.0f;
    const int sub = lane / HALF, pos = 4 * (lane % HALF);  // group of the task, first coordinate
    const long long n_tasks = (p.n_groups + PER - 1) / PER;
    for (long long task = (long long)blockIdx.x * 8 + warp; task < n_tasks; task += (long long)gridDim.x * 8) {
        const long long Gi = task * PER + sub;
        const bool live = Gi < p.n_groups;
        const long long o = live ? Gi / p.ng : 0;
        const int col0 = (int)(Gi - o * p.ng) * G + pos;
        float x[4], w0[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            w0[e] = live && col0 + e < p.in ? __ldcs(p.W + o * p.in + col0 + e) : 0.0f;
            x[e] = w0[e];
        }
        // sum of squares, a tree in fp32
        float sq = __fadd_rn(__fadd_rn(__fmul_rn(x[0], x[0]), __fmul_rn(x[1], x[1])),
                             __fadd_rn(__fmul_rn(x[2], x[2]), __fmul_rn(x[3], x[3])));
#pragma unroll
        for (int m = 1; m < HALF; m <<= 1) sq = __fadd_rn(sq, __shfl_xor_sync(0xffffffffu, sq, m));
        // transform: coordinate bits 0, 1 in registers, bits 2.. across lanes
        const float a0 = __fadd_rn(x[0], x[1]), a1 = __fsub_rn(x[0], x[1]);
        const float a2 = __fadd_rn(x[2], x[3]), a3 = __fsub_rn(x[2], x[3]);
        x[0] = __fadd_rn(a0, a2);
        x[1] = __fadd_rn(a1, a3);
        x[2] = __fsub_rn(a0, a2);
        x[3] = __fsub_rn(a1, a3);
#pragma unroll
        for (int m = 1; m < HALF; m <<= 1)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float v = __shfl_xor_sync(0xffffffffu, x[e], m);
                x[e] = (lane & m) ? __fsub_rn(v, x[e]) : __fadd_rn(x[e], v);
            }
        // fp32 norm; exact fp64 recount when its fp16 rounding is in doubt
        float n32 = __fsqrt_rn(sq);
        bool sure = sq >= 1e-30f && sq <= 1e30f;
        if (sure) {
            const __half lo = __float2half_rn(__fmul_rn(n32, 1.0f - 5e-7f));
            const __half hi = __float2half_rn(__fmul_rn(n32, 1.0f + 5e-7f));
            sure = __half_as_ushort(lo) == __half_as_ushort(hi);
        }
        if (__any_sync(0xffffffffu, !sure)) {
            double d = 0.0;
#pragma unroll
            for (int e = 0; e < 4; ++e) d = __fma_rn((double)w0[e], (double)w0[e], d);
#pragma unroll
            for (int m = 1; m < HALF; m <<= 1) d += __shfl_xor_sync(0xffffffffu, d, m);
            if (!sure) n32 = __double2float_rn(__dsqrt_rn(d));
        }
        const float sc = __fdiv_rn(G == 128 ? 0.08838834764831845f : 0.125f, fmaxf(n32, 1e-12f));
        uint32_t bits = 0;  // my four codes, 4W bits
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            int q = level_index<L>(__fmul_rn(x[e], sc), T);
            if (BITS == 5) q = (q - 1) & 3;  // ternary crumb
            bits |= (uint32_t)q << (W * e);
        }
        // pack the group's LSB-first stream in shared memory, then store it
        uint32_t *sw = s_words[warp][sub];
        if (lane % HALF < NW) sw[lane % HALF] = 0u;
        __syncwarp();
        const int b0 = W * pos, wi = b0 >> 5, sh = b0 & 31;
        atomicOr(sw + wi, bits << sh);
        if (sh + 4 * W > 32) atomicOr(sw + wi + 1, bits >> (32 - sh));
        __syncwarp();
        if (live && lane % HALF < NW)
            reinterpret_cast<uint32_t *>(p.codes + Gi * (G * W / 8))[lane % HALF] = sw[lane % HALF];
        if (live && lane % HALF == 0) p.norms[Gi] = __float2half_rn(n32);
        __syncwarp();
    }
}

// ----------------------------------------------------- activation quant --
// One CTA per token: s = absmax/127 (IEEE division), q = rint(x/s) clamped.
__global__ void act_quant_kernel(const float *__restrict__ X, int M, int in, int8_t *__restrict__ Q,
                                 float *__restrict__ S) {
    __shared__ float red[32];
    for (int t = blockIdx.x; t < M; t += gridDim.x) {
        const float *x = X + (size_t)t * in;
        float amax = 0.0f;
        for (int k = threadIdx.x; k < in; k += blockDim.x) amax = fmaxf(amax, fabsf(x[k]));
#pragma unroll
        for (int o = 16; o; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
        __syncthreads();
        if (threadIdx.x < 32) {
            float v = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : 0.0f;
#pragma unroll
            for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
            if (threadIdx.x == 0) red[0] = v;
        }
        __syncthreads();
        amax = red[0];
        const float s = amax > 0.0f ? __fdiv_rn(amax, 127.0f) : 1.0f;
        for (int k = threadIdx.x; k < in; k += blockDim.x) {
            float v = rintf(__fdiv_rn(x[k], s));
            v = fminf(fmaxf(v, -128.0f), 127.0f);
            Q[(size_t)t * in + k] = (int8_t)(int)v;
        }
        if (threadIdx.x == 0) S[t] = s;
        __syncthreads();
    }
}

template <int BITS, bool ALIGNED>
int launch_encode_t(const EncodeParams &p, cudaStream_t st) {
    const size_t smem = kEncTileFloats * sizeof(float);
    auto k = encode_kernel<BITS, ALIGNED>;
    const int rc = ensure_smem(reinterpret_cast<const void *>(k), smem);
    if (rc) return rc;
    const long long tiles = (p.n_groups + kEncWarpGroups - 1) / kEncWarpGroups;
    const long long blocks = (tiles + kEncWarps - 1) / kEncWarps;
    const long long grid = std::min<long long>(blocks, (long long)sm_count() * 2);
    k<<<(unsigned)grid, kEncThreads, smem, st>>>(p);
    return CQ_OK;
}

}  // namespace

int sm_count() {
    static std::atomic<int> cache[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        cudaGetLastError();
        return 1;
    }
    int n = cache[dev].load(std::memory_order_relaxed);
    if (!n) {
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
            cudaGetLastError();
            n = 1;
        }
        cache[dev].store(n, std::memory_order_relaxed);  // every writer stores the same value
    }
    return n;
}

int launch_encode(const float *W, int out, int in, int group, int bits, const float *cb, uint8_t *blob,
                  void *stream) {
    const size_t rowBytes = (size_t)in_padded(in, group) * width_of(bits) / 8;
    return launch_encode_rows(W, out, in, group, bits, cb, blob, blob + (size_t)out * rowBytes, stream);
}

template <int BITS, bool ALIGNED>
int launch_encode_g64(const EncodeParams &p, cudaStream_t st) {
    const size_t smem = kEncTileFloats * sizeof(float);
    auto k = encode_g64_kernel<BITS, ALIGNED>;
    const int rc = ensure_smem(reinterpret_cast<const void *>(k), smem);
    if (rc) return rc;
    const long long tiles = (p.n_groups + 31) / 32;  // 32 groups per warp tile
    const long long blocks = (tiles + kEncWarps - 1) / kEncWarps;
    const long long grid = std::min<long long>(blocks, (long long)sm_count() * 2);
    k<<<(unsigned)grid, kEncThreads, smem, st>>>(p);
    return CQ_OK;
}

template <int G, int BITS>
void launch_encode_warp(const EncodeParams &p, cudaStream_t st) {
    const long long tasks = (p.n_groups + 128 / G - 1) / (128 / G);
    const long long grid = std::min<long long>((tasks + 7) / 8, (long long)sm_count() * 8);
    encode_warp_kernel<G, BITS><<<(unsigned)grid, 256, 0, st>>>(p);
}

int launch_encode_rows(const float *W, int out, int in, int group, int bits, const float *cb, uint8_t *codes,
                       uint8_t *nb, void *stream) {
    EncodeParams p;
    p.W = W;
    p.in = in;
    p.ng = in_padded(in, group) / group;
    p.n_groups = (long long)out * p.ng;
    p.codes = codes;
    if ((reinterpret_cast<uintptr_t>(codes) & 15) || (reinterpret_cast<uintptr_t>(nb) & 1))
        return set_error(CQ_ERR_ARG, "blob must be 16-byte aligned");
    p.norms = reinterpret_cast<__half *>(nb);
    p.status = device_status_ptr();
    const int L = levels_of(bits);
    for (int j = 0; j < kMaxLevels; ++j) p.cb[j] = j < L ? cb[j] : 0.0f;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    int rc = CQ_OK;
    if (group == kGroup64) {
        const bool aligned = (in % kGroup64 == 0) && !(reinterpret_cast<uintptr_t>(W) & 15);
        switch (bits) {
        case 1: rc = aligned ? launch_encode_g64<1, true>(p, st) : launch_encode_g64<1, false>(p, st); break;
        case 2: rc = aligned ? launch_encode_g64<2, true>(p, st) : launch_encode_g64<2, false>(p, st); break;
        case 3: rc = aligned ? launch_encode_g64<3, true>(p, st) : launch_encode_g64<3, false>(p, st); break;
        case 4: rc = aligned ? launch_encode_g64<4, true>(p, st) : launch_encode_g64<4, false>(p, st); break;
        case 5: rc = aligned ? launch_encode_g64<5, true>(p, st) : launch_encode_g64<5, false>(p, st); break;
        }
    } else if (bits == 1) {
        launch_encode_warp<128, 1>(p, st);
    } else {
        const bool aligned = (in % kGroup == 0) && !(reinterpret_cast<uintptr_t>(W) & 15);
        switch (bits) {
        case 2: rc = aligned ? launch_encode_t<2, true>(p, st) : launch_encode_t<2, false>(p, st); break;
        case 3: rc = aligned ? launch_encode_t<3, true>(p, st) : launch_encode_t<3, false>(p, st); break;
        case 4: rc = aligned ? launch_encode_t<4, true>(p, st) : launch_encode_t<4, false>(p, st); break;
        case 5: rc = aligned ? launch_encode_t<5, true>(p, st) : launch_encode_t<5, false>(p, st); break;
        }
    }
    if (rc) return rc;
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return set_error(CQ_ERR_CUDA, "encode launch: %s", cudaGetErrorString(e));
    return CQ_OK;
}

int launch_act_quant(const float *X, int M, int in, int8_t *Xq, float *s, void *stream) {
    const int grid = std::min(M, sm_count() * 8);
    act_quant_kernel<<<grid, 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(X, M, in, Xq, s);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return set_error(CQ_ERR_CUDA, "act_quant launch: %s", cudaGetErrorString(e));
    return CQ_OK;
}

}  // namespace cq
