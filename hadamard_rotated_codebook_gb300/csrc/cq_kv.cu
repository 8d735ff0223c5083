// cq_kv.cu -- decode-step attention over CQ key/value caches.
//
// A cache row is one token's head vectors side by side, stored as a CQ
// matrix row ("The .cact format", "How the kernel reads it": the weight path
// serves the KV cache at the header's kv_bits). For query head b, reading
// key/value head h, and group g of a row:
//   logit[b][t] = scale * sum_g n_k[t][g] * < c[q_k[t,g,:]], H x_{b,g} >
// where x_b is q_b placed at head h's columns of the row (zero elsewhere) --
// the rotated-domain identity of the weight GEMV (OpenNeedle
// docs/reference.md). The value sum stays in the rotated domain,
//   R[b][g] = sum_t p[b][t] n_v[t][g] c[q_v[t,g,:]],   o_b = slice_h(H R[b]) / l_b,
// so neither cache is ever expanded and H (its own inverse) is applied once
// per group and head at the end.
//
// GB300 mapping. A thread block owns a chunk of one sequence's tokens and
// walks it in sub-tiles of 128 tokens with an online softmax:
//  - key side: warp w takes tokens 16w..16w+15 of the sub-tile; their code
//    bits come straight from global memory into registers, a pair table in
//    shared memory (two codes -> two fp16 levels, one replica per bank)
//    turns them into A fragments of mma.sync m16n8k16, and the rotated
//    queries (fp16 hi + lo terms, two B columns per head) are the B operand;
//  - softmax statistics per head in fp32 (running max, sum, rescale factor);
//  - value side: the MMA contracts over tokens. Rows of A are value
//    coordinates (two neighbours per code pair), columns of A are tokens
//    (code pairs of two tokens interleaved with a byte permute), B holds the
//    weights p * n_v in fp16; each warp owns a few 16-coordinate slices and
//    keeps their accumulators in registers across the whole chunk.
// Sequences longer than one chunk write their partial (max, sum, R) to a
// workspace; the last block of the sequence to finish (an atomic ticket; no
// block waits for another) merges them and writes o.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <vector>

#include "cq_internal.h"

namespace cq {

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kTile = 128;      // tokens per sub-tile
constexpr int kMaxStages = 3;   // sub-tiles whose copies are in flight
constexpr int kMaxParts = 128;  // blocks sharing one sequence (the merge's factors fit the logits buffer)
constexpr int kSpRow = kTile + 8;  // logits [head][token]: the stride spreads a warp's heads over banks
constexpr int kMaxHeads = 16;   // query heads per call
constexpr int kMaxSeqs = 256;   // sequences per launch (the host splits larger calls)
constexpr float kInvSqrt128 = 0.08838834764831845f;

struct KvSeqDev {
    const uint8_t *kc, *vc;  // caches
    const float *q;
    float *o;
    int cap, n;              // rows allocated, rows attended
    int sub0;                // first sub-tile of the sequence in the launch's flat order
    int part_b0, n_parts;    // first block that works on it, and how many do
    int slot0;               // first workspace slot (n_parts > 1)
};

struct KvParams {
    int Hq, per, dk, dv;     // per = query heads per key/value head
    int in_k, in_v, ngk, ngv;
    int ntk, ntv;            // n-tiles of 8 columns: key side (hi, lo per head), value side
    float logit_scale;       // scale * log2(e) / sqrt(128): base-2 logits of the unnormalised rotation
    int n_seqs;
    int total_sub;           // sub-tiles of all sequences; block b takes [b T / G, (b + 1) T / G)
    int vrow;                // staged value-code row stride (bytes)
    int krow;                // staged key-code row stride (bytes)
    int cprk_magic, cprv_magic;  // ceil(65536 / (16-byte pieces per key / value row))
    int n_stages;            // sub-tiles in flight (1..3)
    // shared-memory byte offsets; a stage holds key codes at 0, value codes at
    // off_v, key norms at off_kn and value norms at off_vn
    int sm_tabk, sm_tabv, sm_zf, sm_isig, sm_p, sm_wf, sm_terms, sm_r, sm_stage;
    int stage_bytes, off_v, off_kn, off_vn;
    uint16_t lvk[16], lvv[16];  // fp16 level bits by code
    float *part;             // [slot][Hq][ngv*128] partial rotated value sums
    float *ml;               // [slot][Hq][2] running max and sum
    unsigned int *ticket;    // [seq] blocks finished
    KvSeqDev s[kMaxSeqs];
};

__device__ __forceinline__ void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                        uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// 16-byte asynchronous copy reading src_bytes (1..16) and zero-filling the rest.
__device__ __forceinline__ void cp_async16(void *dst, const void *src, int src_bytes) {
    const uint32_t d = (uint32_t)__cvta_generic_to_shared(dst);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(d), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory"); }

__device__ __forceinline__ uint32_t pack_h2(float lo, float hi) {
    return (uint32_t)__half_as_ushort(__float2half_rn(lo)) | ((uint32_t)__half_as_ushort(__float2half_rn(hi)) << 16);
}

// Largest power of two sigma with amax * sigma <= lim (1 for amax == 0).
__device__ __forceinline__ float pow2_scale(float amax, float lim) {
    if (!(amax > 0.0f)) return 1.0f;
    const float q = __fdiv_rn(lim, amax);
    const int E = min(max((__float_as_int(q) >> 23) & 0xff, 1), 254);
    float s = __int_as_float(E << 23);
    if (__fmul_rn(amax, s) > lim) s *= 0.5f;
    return s;
}

// Unnormalised 128-point transform of the values a warp holds (lane: 4*lane + i).
__device__ __forceinline__ void fwht128(float (&v)[4], int lane) {
    const float a0 = v[0] + v[1], a1 = v[0] - v[1], a2 = v[2] + v[3], a3 = v[2] - v[3];
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
}

// 2W code bits starting at bit `off` of a little-endian word array (W <= 4,
// so at most 8 bits, possibly straddling two words).
template <int W>
__device__ __forceinline__ uint32_t bits2(const uint32_t *w, int off) {
    const int i = off >> 5, sh = off & 31;
    if (W != 3) return (w[i] >> sh) & ((1u << (2 * W)) - 1u);
    return __funnelshift_r(w[i], w[i + 1], sh) & 63u;
}

// Code words of one key row's group (staged in shared memory) for lane
// quarter c: 4W bytes holding the thread's 32 coordinates 32c .. 32c+31.
template <int W>
__device__ __forceinline__ void load_key_words(const uint8_t *grp, int c, uint32_t (&w)[5]) {
    w[0] = w[1] = w[2] = w[3] = w[4] = 0u;
    if (W == 4) {
        const uint4 v = reinterpret_cast<const uint4 *>(grp)[c];
        w[0] = v.x;
        w[1] = v.y;
        w[2] = v.z;
        w[3] = v.w;
    } else {
        const uint32_t *q = reinterpret_cast<const uint32_t *>(grp) + 3 * c;
        w[0] = q[0];
        w[1] = q[1];
        w[2] = q[2];
    }
}

// Rotated-domain value sums R[b][k] in shared memory -> o[b] = slice of
// (H0 R[b]) / (sqrt(128) l_b) for the groups that overlap head b's columns.
__device__ void finish_heads(const KvParams &p, const float *sr, const float *sl, float *o, int warp, int lane) {
    const int ipv = p.ngv * kGroup;
    for (int task = warp; task < p.Hq * p.ngv; task += kWarps) {
        const int b = task / p.ngv, g = task % p.ngv;
        const int h = b / p.per, c0 = h * p.dv, c1 = c0 + p.dv;
        if (c1 <= g * kGroup || c0 >= (g + 1) * kGroup) continue;  // group outside the head
        float v[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) v[i] = sr[b * ipv + g * kGroup + 4 * lane + i];
        fwht128(v, lane);
        const float f = kInvSqrt128 / sl[b];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int col = g * kGroup + 4 * lane + i;
            if (col >= c0 && col < c1) o[(size_t)b * p.dv + col - c0] = v[i] * f;
        }
    }
}

// The block's queries as key-side B fragments: for head b and key group g,
// z = H0 x (x = q_b at its head's columns of the row) scaled by a power of
// two sigma and split into fp16 hi + lo terms; word (g, nu, nt, lane) of
// column n = 8 nt + lane/4 (head n/2, term n%2) holds positions
// 32 (lane%4) + 4 nu + {0,1} and {2,3}. isig[b][g] = 1/sigma. Ends with a
// block barrier (terms may be reused after it).
__device__ void rotate_queries(const KvParams &p, const float *qv, uint32_t *terms, float *isig, uint2 *zf) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, gq = lane >> 2, c = lane & 3;
    const int Hq = p.Hq, ngk = p.ngk, ntk = p.ntk;
    for (int task = warp; task < Hq * ngk; task += kWarps) {
        const int b = task / ngk, g = task - b * ngk;
        const int c0 = (b / p.per) * p.dk;
        float v[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int col = g * kGroup + 4 * lane + i;
            v[i] = (col >= c0 && col < c0 + p.dk) ? qv[(size_t)b * p.dk + col - c0] : 0.0f;
        }
        fwht128(v, lane);
        float mx = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
#pragma unroll
        for (int m = 16; m; m >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, m));
        const float sigma = pow2_scale(mx, 16384.0f);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float x = __fmul_rn(v[i], sigma);
            const __half hh = __float2half_rn(x);
            const __half ll = __float2half_rn(__fsub_rn(x, __half2float(hh)));
            terms[(b * ngk + g) * kGroup + 4 * lane + i] =
                (uint32_t)__half_as_ushort(hh) | ((uint32_t)__half_as_ushort(ll) << 16);
        }
        if (lane == 0) isig[b * ngk + g] = 1.0f / sigma;
    }
    __syncthreads();
    for (int g = 0; g < ngk; ++g)
        for (int nu = warp; nu < 8; nu += kWarps)
            for (int nt = 0; nt < ntk; ++nt) {
                const int n = 8 * nt + gq, b = n >> 1, tau = n & 1, k0 = 32 * c + 4 * nu;
                uint2 f = make_uint2(0u, 0u);
                if (b < Hq) {
                    const uint32_t *tw = terms + (b * ngk + g) * kGroup + k0;
                    f.x = ((tw[0] >> (16 * tau)) & 0xffffu) | (((tw[1] >> (16 * tau)) & 0xffffu) << 16);
                    f.y = ((tw[2] >> (16 * tau)) & 0xffffu) | (((tw[3] >> (16 * tau)) & 0xffffu) << 16);
                }
                zf[((g * 8 + nu) * ntk + nt) * 32 + lane] = f;
            }
    __syncthreads();
}

// The end of a segment, once sr[b][k] holds the rotated value sums and
// sM / sL the running max and sum per head: one part writes o directly;
// otherwise the part goes to workspace slot `slot` and the last block of the
// sequence to finish (atomic ticket) merges all parts into o. `scratch`
// holds n_parts * Hq floats. All threads of the block call this; it ends
// with a block barrier.
__device__ void emit_segment(const KvParams &p, float *sr, float *sM, float *sL, float *scratch, float *ov, int si,
                             int n_parts, int slot, int slot0, int *s_last) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, Hq = p.Hq, ipv = p.ngv * kGroup;
    if (n_parts == 1) {
        finish_heads(p, sr, sL, ov, warp, lane);
        __syncthreads();
        return;
    }
    float *pdst = p.part + (size_t)slot * Hq * ipv;
    for (int i = tid; i < Hq * ipv; i += kThreads) __stcg(pdst + i, sr[i]);
    if (tid < Hq) {
        __stcg(p.ml + ((size_t)slot * Hq + tid) * 2, sM[tid]);
        __stcg(p.ml + ((size_t)slot * Hq + tid) * 2 + 1, sL[tid]);
    }
    __threadfence();
    __syncthreads();
    if (tid == 0) *s_last = atomicAdd(p.ticket + si, 1u) == (unsigned)(n_parts - 1);
    __syncthreads();
    if (!*s_last) return;  // uniform; the caller's next segment starts after this barrier
    // the last block of the sequence merges the partials
    __threadfence();
    const float *ml0 = p.ml + (size_t)slot0 * Hq * 2;
    if (tid < Hq) {
        float mx = -INFINITY;
        for (int ch = 0; ch < n_parts; ++ch) mx = fmaxf(mx, __ldcg(ml0 + ((size_t)ch * Hq + tid) * 2));
        sM[tid] = mx;
    }
    __syncthreads();
    for (int i = tid; i < n_parts * Hq; i += kThreads) scratch[i] = exp2f(__ldcg(ml0 + 2 * (size_t)i) - sM[i % Hq]);
    __syncthreads();
    if (tid < Hq) {
        float l = 0.0f;
        for (int ch = 0; ch < n_parts; ++ch)
            l = fmaf(__ldcg(ml0 + ((size_t)ch * Hq + tid) * 2 + 1), scratch[ch * Hq + tid], l);
        sL[tid] = l;
    }
    const float *part0 = p.part + (size_t)slot0 * Hq * ipv;
    for (int i = tid; i < Hq * ipv; i += kThreads) {
        const int b = i / ipv;
        float r = 0.0f;
        for (int ch = 0; ch < n_parts; ++ch)
            r = fmaf(__ldcg(part0 + (size_t)ch * Hq * ipv + i), scratch[ch * Hq + b], r);
        sr[i] = r;
    }
    if (tid == 0) p.ticket[si] = 0u;  // ready for the next launch
    __syncthreads();
    finish_heads(p, sr, sL, ov, warp, lane);
    __syncthreads();
}

// Accumulator slot ms of a warp's value-side work: coordinate of its row
// gq (hi = 0) or gq + 8 (hi = 1). With 2-bit codes a unit is a pair of
// 16-coordinate slices fed by one byte lookup per token: slice A holds
// coordinates 4j, 4j+1 and slice B 4j+2, 4j+3 of bytes j = 8s + gq; with
// wider codes a unit is one slice of 16 neighbouring coordinates.
template <int WV>
__device__ __forceinline__ int slot_coord(int unit, int ms_in_unit, int gq, int hi) {
    if (WV == 2) return (unit >> 2) * kGroup + 4 * (8 * (unit & 3) + gq) + 2 * ms_in_unit + hi;
    return (unit >> 3) * kGroup + 16 * (unit & 7) + 2 * gq + hi;
}

template <int WK, int WV>
__global__ void __launch_bounds__(kThreads, 3) kv_attend_kernel(const __grid_constant__ KvParams p) {
    extern __shared__ __align__(16) uint8_t smem[];
    __shared__ float sM[kMaxHeads], sL[kMaxHeads], sF[kMaxHeads];
    __shared__ int s_last;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int gq = lane >> 2, c = lane & 3, r16 = lane & 15;

    const int Hq = p.Hq, ngk = p.ngk, ngv = p.ngv, ntk = p.ntk, ntv = p.ntv, vrow = p.vrow;

    uint32_t *tabk = reinterpret_cast<uint32_t *>(smem + p.sm_tabk);  // pair table [4^W][32], or quad table [256][16] (W = 2)
    uint32_t *tabv = reinterpret_cast<uint32_t *>(smem + p.sm_tabv);
    uint2 *zf = reinterpret_cast<uint2 *>(smem + p.sm_zf);             // [ngk][8][ntk][32]
    float *isig = reinterpret_cast<float *>(smem + p.sm_isig);         // [Hq][ngk]
    float *sp = reinterpret_cast<float *>(smem + p.sm_p);              // [16][kSpRow] logits, then weights
    uint2 *wf = reinterpret_cast<uint2 *>(smem + p.sm_wf);             // [ngv][8][ntv][32]
    uint32_t *terms = reinterpret_cast<uint32_t *>(smem + p.sm_terms); // [Hq][ngk][128] (setup only)
    float *sr = reinterpret_cast<float *>(smem + p.sm_r);              // [Hq][ngv*128] (end only)

    // ---- setup: level tables, rotated queries as B fragments ----
    if (WK == 2) {  // quad table: a code byte -> four fp16 levels, 16 replicas
        for (int i = tid; i < 256 * 16; i += kThreads) {
            const int e = i >> 4;
            tabk[2 * i] = (uint32_t)p.lvk[e & 3] | ((uint32_t)p.lvk[(e >> 2) & 3] << 16);
            tabk[2 * i + 1] = (uint32_t)p.lvk[(e >> 4) & 3] | ((uint32_t)p.lvk[e >> 6] << 16);
        }
    } else {  // pair table: two codes -> two fp16 levels, 32 replicas
        for (int i = tid; i < (1 << (2 * WK)) * 32; i += kThreads) {
            const int e = i >> 5;
            tabk[i] = (uint32_t)p.lvk[e & ((1 << WK) - 1)] | ((uint32_t)p.lvk[e >> WK] << 16);
        }
    }
    if (p.sm_tabv != p.sm_tabk) {
        if (WV == 2) {
            for (int i = tid; i < 256 * 16; i += kThreads) {
                const int e = i >> 4;
                tabv[2 * i] = (uint32_t)p.lvv[e & 3] | ((uint32_t)p.lvv[(e >> 2) & 3] << 16);
                tabv[2 * i + 1] = (uint32_t)p.lvv[(e >> 4) & 3] | ((uint32_t)p.lvv[e >> 6] << 16);
            }
        } else {
            for (int i = tid; i < (1 << (2 * WV)) * 32; i += kThreads) {
                const int e = i >> 5;
                tabv[i] = (uint32_t)p.lvv[e & ((1 << WV) - 1)] | ((uint32_t)p.lvv[e >> WV] << 16);
            }
        }
    }
    for (int q = blockIdx.x; q < p.n_seqs; q += gridDim.x)  // empty softmax: o = 0
        if (p.s[q].n == 0)
            for (int i = tid; i < Hq * p.dv; i += kThreads) p.s[q].o[i] = 0.0f;

    // This block's share of the flat sub-tile order, walked as segments of
    // consecutive sub-tiles of one sequence.
    const int G = gridDim.x, T = p.total_sub, bid = blockIdx.x;
    const int x_end = (int)(((long long)(bid + 1) * T) / G);
    for (int x = (int)(((long long)bid * T) / G); x < x_end;) {
    int lo = 0, hi = p.n_seqs - 1;  // the sequence holding sub-tile x
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (p.s[mid].sub0 <= x) lo = mid;
        else hi = mid - 1;
    }
    const int si = lo;
    // the sequence's fields in registers (indexed parameter reads would repeat in the loops)
    const uint8_t *const kc = p.s[si].kc;
    const uint8_t *const vc = p.s[si].vc;
    const float *const qv = p.s[si].q;
    float *const ov = p.s[si].o;
    const int cap = p.s[si].cap, n_tok = p.s[si].n, n_parts = p.s[si].n_parts, slot0 = p.s[si].slot0;
    const int sub0 = p.s[si].sub0, sub_end = sub0 + (n_tok + kTile - 1) / kTile;
    const int seg_end = min(x_end, sub_end), part = bid - p.s[si].part_b0;
    const int t_begin = (x - sub0) * kTile, t_end = min(n_tok, (seg_end - sub0) * kTile);
    x = seg_end;

    if (tid < kMaxHeads) {
        sM[tid] = -INFINITY;
        sL[tid] = 0.0f;
        sF[tid] = 1.0f;  // heads past Hq keep 1 (their accumulators stay 0)
    }
    rotate_queries(p, qv, terms, isig, zf);
    __syncthreads();  // terms (aliased by the value staging) are dead from here

    const int rbk = ngk * 16 * WK, rbv = ngv * 16 * WV, cprk = rbk >> 4, cprv = rbv >> 4;
    const int krow = p.krow;
    const uint8_t *const knorm_b = kc + (size_t)cap * rbk;  // fp16 norms [cap][ngk]
    const uint8_t *const vnorm_b = vc + (size_t)cap * rbv;
    // value-side work of this warp: its units, and its token tiles when two
    // warps share a unit (2-bit codes, one group: four units for eight warps)
    const int units = (WV == 2 ? 4 : 8) * ngv;
    const int split = units < kWarps ? kWarps / units : 1;
    const int unit0 = split > 1 ? warp % units : warp;
    const int tau0 = split > 1 ? (warp / units) * (8 / split) : 0;
    const int tau1 = split > 1 ? tau0 + 8 / split : 8;
    float acc[4][2][4];
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int i = 0; i < 4; ++i) acc[j][nt][i] = 0.0f;

    // Copies of sub-tile i into stage i % kStages, one commit group: key and
    // value code rows, then the two fp16 norm blocks (contiguous in the
    // cache; the last 16-byte piece reads only the rows that exist and
    // zero-fills the rest).
    const int nsub = (t_end - t_begin + kTile - 1) / kTile, NB = p.n_stages;
    auto issue = [&](int i) {
        uint8_t *stg = smem + p.sm_stage + (i % NB) * p.stage_bytes;
        const int t0 = t_begin + i * kTile, nv = min(kTile, t_end - t0);
        for (int x = tid; x < nv * cprk; x += kThreads) {
            const int r = (x * p.cprk_magic) >> 16, j = x - r * cprk;  // x / cprk, exact here
            cp_async16(stg + r * krow + 16 * j, kc + (size_t)(t0 + r) * rbk + 16 * j, 16);
        }
        for (int x = tid; x < nv * cprv; x += kThreads) {
            const int r = (x * p.cprv_magic) >> 16, j = x - r * cprv;
            cp_async16(stg + p.off_v + r * vrow + 16 * j, vc + (size_t)(t0 + r) * rbv + 16 * j, 16);
        }
        const int kb = nv * 2 * ngk, vb = nv * 2 * ngv, kp = (kb + 15) >> 4, vp = (vb + 15) >> 4;
        for (int x = tid; x < kp + vp; x += kThreads) {
            if (x < kp)
                cp_async16(stg + p.off_kn + 16 * x, knorm_b + (size_t)t0 * 2 * ngk + 16 * x, min(16, kb - 16 * x));
            else
                cp_async16(stg + p.off_vn + 16 * (x - kp), vnorm_b + (size_t)t0 * 2 * ngv + 16 * (x - kp),
                           min(16, vb - 16 * (x - kp)));
        }
        cp_async_commit();
    };
    for (int j = 0; j + 1 < NB; ++j) {
        if (j < nsub) issue(j);
        else cp_async_commit();  // empty groups keep the count of groups in flight uniform
    }
    for (int it = 0; it < nsub; ++it) {
        if (it + NB - 1 < nsub) issue(it + NB - 1);
        else cp_async_commit();
        // this sub-tile's copies have landed (NB - 1 younger groups may still fly)
        if (NB == 3) cp_async_wait<2>();
        else if (NB == 2) cp_async_wait<1>();
        else cp_async_wait<0>();
        __syncthreads();
        const int t0 = t_begin + it * kTile, nv = min(kTile, t_end - t0);
        const uint8_t *ks = smem + p.sm_stage + (it % NB) * p.stage_bytes;
        const uint8_t *vcodes = ks + p.off_v;
        const __half *kns = reinterpret_cast<const __half *>(ks + p.off_kn);
        const __half *vns = reinterpret_cast<const __half *>(ks + p.off_vn);
        // ---- B. logits of 16 tokens per warp (log2 units) ----
        {
            const int ra = 16 * warp + gq, rb = ra + 8;  // rows of the sub-tile
            const bool va = ra < nv, vb = rb < nv;
            float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
            for (int g = 0; g < ngk; ++g) {
                const float na = __half2float(kns[ra * ngk + g]), nb = __half2float(kns[rb * ngk + g]);
                float d[4][4];
#pragma unroll
                for (int nt = 0; nt < 4; ++nt)
#pragma unroll
                    for (int i = 0; i < 4; ++i) d[nt][i] = 0.0f;
                if (WK == 2) {
                    const uint2 ca = *reinterpret_cast<const uint2 *>(ks + ra * krow + g * 32 + 8 * c);
                    const uint2 cb = *reinterpret_cast<const uint2 *>(ks + rb * krow + g * 32 + 8 * c);
                    const uint2 *t4 = reinterpret_cast<const uint2 *>(tabk) + r16;
#pragma unroll
                    for (int nu = 0; nu < 8; ++nu) {
                        const uint32_t wa = nu < 4 ? ca.x : ca.y, wb = nu < 4 ? cb.x : cb.y;
                        const uint2 ea = t4[((wa >> (8 * (nu & 3))) & 0xffu) * 16];
                        const uint2 eb = t4[((wb >> (8 * (nu & 3))) & 0xffu) * 16];
                        const uint2 *zb = zf + ((g * 8 + nu) * ntk) * 32 + lane;
#pragma unroll
                        for (int nt = 0; nt < 4; ++nt)
                            if (nt < ntk) {
                                const uint2 bf = zb[nt * 32];
                                mma_f16(d[nt], ea.x, eb.x, ea.y, eb.y, bf.x, bf.y);
                            }
                    }
                } else {
                    uint32_t wa[5], wb[5];
                    load_key_words<WK>(ks + ra * krow + g * 16 * WK, c, wa);
                    load_key_words<WK>(ks + rb * krow + g * 16 * WK, c, wb);
#pragma unroll
                    for (int nu = 0; nu < 8; ++nu) {
                        const uint32_t a0 = tabk[bits2<WK>(wa, WK * 4 * nu) * 32 + lane];
                        const uint32_t a1 = tabk[bits2<WK>(wb, WK * 4 * nu) * 32 + lane];
                        const uint32_t a2 = tabk[bits2<WK>(wa, WK * (4 * nu + 2)) * 32 + lane];
                        const uint32_t a3 = tabk[bits2<WK>(wb, WK * (4 * nu + 2)) * 32 + lane];
                        const uint2 *zb = zf + ((g * 8 + nu) * ntk) * 32 + lane;
#pragma unroll
                        for (int nt = 0; nt < 4; ++nt)
                            if (nt < ntk) {
                                const uint2 bf = zb[nt * 32];
                                mma_f16(d[nt], a0, a1, a2, a3, bf.x, bf.y);
                            }
                    }
                }
#pragma unroll
                for (int nt = 0; nt < 4; ++nt) {
                    const int b = 4 * nt + c;
                    if (nt < ntk && b < Hq) {
                        const float is = isig[b * ngk + g];
                        sa[nt] = fmaf(na * is, d[nt][0] + d[nt][1], sa[nt]);
                        sb[nt] = fmaf(nb * is, d[nt][2] + d[nt][3], sb[nt]);
                    }
                }
            }
            // rows past the end hold stale bytes: their logits are -inf
#pragma unroll
            for (int nt = 0; nt < 4; ++nt) {
                const int b = 4 * nt + c;
                if (nt < ntk && b < Hq) {
                    sp[b * kSpRow + ra] = va ? sa[nt] * p.logit_scale : -INFINITY;
                    sp[b * kSpRow + rb] = vb ? sb[nt] * p.logit_scale : -INFINITY;
                }
            }
        }
        __syncthreads();
        // ---- C. online softmax per head (base 2: the logits carry log2(e)) ----
        for (int b = warp; b < Hq; b += kWarps) {
            float s[4], m = -INFINITY;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                s[i] = sp[b * kSpRow + lane + 32 * i];
                m = fmaxf(m, s[i]);
            }
#pragma unroll
            for (int o = 16; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
            const float m_old = sM[b], m_new = fmaxf(m_old, m);
            float sum = 0.0f;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float e = exp2f(s[i] - m_new);  // 0 for tokens past the end
                sp[b * kSpRow + lane + 32 * i] = e;
                sum += e;
            }
#pragma unroll
            for (int o = 16; o; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
            if (lane == 0) {
                const float f = exp2f(m_old - m_new);  // 0 on the first sub-tile
                sF[b] = f;
                sM[b] = m_new;
                sL[b] = fmaf(sL[b], f, sum);
            }
        }
        __syncthreads();
        // value-side B fragments of token tile `warp`: w[t][b] = p[t][b] * n_v[t][g] in fp16
        {
            const int t = 16 * warp + 2 * c;
            for (int g = 0; g < ngv; ++g) {
                const float n0 = t < nv ? __half2float(vns[t * ngv + g]) : 0.0f;
                const float n1 = t + 1 < nv ? __half2float(vns[(t + 1) * ngv + g]) : 0.0f;
                const float n8 = t + 8 < nv ? __half2float(vns[(t + 8) * ngv + g]) : 0.0f;
                const float n9 = t + 9 < nv ? __half2float(vns[(t + 9) * ngv + g]) : 0.0f;
                for (int nt = 0; nt < ntv; ++nt) {
                    const int b = 8 * nt + gq;
                    uint2 f = make_uint2(0u, 0u);
                    if (b < Hq) {
                        f.x = pack_h2(sp[b * kSpRow + t] * n0, sp[b * kSpRow + t + 1] * n1);
                        f.y = pack_h2(sp[b * kSpRow + t + 8] * n8, sp[b * kSpRow + t + 9] * n9);
                    }
                    wf[((g * 8 + warp) * ntv + nt) * 32 + lane] = f;
                }
            }
        }
        __syncthreads();
        // ---- D. rotated value sums: rows of A = coordinates, columns = tokens ----
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
                if (nt < ntv) {
                    const float f0 = sF[8 * nt + 2 * c], f1 = sF[8 * nt + 2 * c + 1];
                    acc[j][nt][0] *= f0;
                    acc[j][nt][1] *= f1;
                    acc[j][nt][2] *= f0;
                    acc[j][nt][3] *= f1;
                }
        if (WV == 2) {
            const uint2 *t4 = reinterpret_cast<const uint2 *>(tabv) + r16;
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                const int unit = unit0 + k * kWarps;
                if (unit >= units || (split > 1 && k > 0)) break;
                const int g = unit >> 2, boff = g * 32 + 8 * (unit & 3) + gq;
                for (int tau = tau0; tau < tau1; ++tau) {
                    const uint8_t *row = vcodes + (16 * tau + 2 * c) * vrow + boff;
                    const uint2 h0 = t4[(uint32_t)row[0] * 16], h1 = t4[(uint32_t)row[vrow] * 16];
                    const uint2 h2 = t4[(uint32_t)row[8 * vrow] * 16], h3 = t4[(uint32_t)row[9 * vrow] * 16];
                    const uint32_t aA0 = __byte_perm(h0.x, h1.x, 0x5410), aA1 = __byte_perm(h0.x, h1.x, 0x7632);
                    const uint32_t aA2 = __byte_perm(h2.x, h3.x, 0x5410), aA3 = __byte_perm(h2.x, h3.x, 0x7632);
                    const uint32_t aB0 = __byte_perm(h0.y, h1.y, 0x5410), aB1 = __byte_perm(h0.y, h1.y, 0x7632);
                    const uint32_t aB2 = __byte_perm(h2.y, h3.y, 0x5410), aB3 = __byte_perm(h2.y, h3.y, 0x7632);
                    const uint2 *wb = wf + ((g * 8 + tau) * ntv) * 32 + lane;
#pragma unroll
                    for (int nt = 0; nt < 2; ++nt)
                        if (nt < ntv) {
                            const uint2 bf = wb[nt * 32];
                            mma_f16(acc[2 * k][nt], aA0, aA1, aA2, aA3, bf.x, bf.y);
                            mma_f16(acc[2 * k + 1][nt], aB0, aB1, aB2, aB3, bf.x, bf.y);
                        }
                }
            }
        } else {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int unit = unit0 + k * kWarps;
                if (unit >= units) break;
                const int g = unit >> 3, mu = unit & 7;
                const int off = g * kGroup * WV + WV * (16 * mu + 2 * gq);  // bit offset of the code pair
                for (int tau = 0; tau < 8; ++tau) {
                    const int t = 16 * tau + 2 * c;
                    const uint32_t *r0 = reinterpret_cast<const uint32_t *>(vcodes + t * vrow);
                    const uint32_t *r1 = reinterpret_cast<const uint32_t *>(vcodes + (t + 1) * vrow);
                    const uint32_t *r2 = reinterpret_cast<const uint32_t *>(vcodes + (t + 8) * vrow);
                    const uint32_t *r3 = reinterpret_cast<const uint32_t *>(vcodes + (t + 9) * vrow);
                    const uint32_t h0 = tabv[bits2<WV>(r0, off) * 32 + lane];
                    const uint32_t h1 = tabv[bits2<WV>(r1, off) * 32 + lane];
                    const uint32_t h2 = tabv[bits2<WV>(r2, off) * 32 + lane];
                    const uint32_t h3 = tabv[bits2<WV>(r3, off) * 32 + lane];
                    const uint32_t a0 = __byte_perm(h0, h1, 0x5410), a1 = __byte_perm(h0, h1, 0x7632);
                    const uint32_t a2 = __byte_perm(h2, h3, 0x5410), a3 = __byte_perm(h2, h3, 0x7632);
                    const uint2 *wb = wf + ((g * 8 + tau) * ntv) * 32 + lane;
#pragma unroll
                    for (int nt = 0; nt < 2; ++nt)
                        if (nt < ntv) {
                            const uint2 bf = wb[nt * 32];
                            mma_f16(acc[k][nt], a0, a1, a2, a3, bf.x, bf.y);
                        }
                }
            }
        }
        __syncthreads();  // the stage is refilled two sub-tiles later; logits and fragments next one
    }
    cp_async_wait<0>();  // only empty groups remain; nothing may land after the block moves on

    // ---- E. rotated sums into shared memory: element i of slot (unit, m)
    // is row gq + 8 (i >> 1), head 8 nt + 2c + (i & 1); warps that split a
    // unit's tokens add into the same words ----
    const int ipv = ngv * kGroup;
    for (int i = tid; i < Hq * ipv; i += kThreads) sr[i] = 0.0f;
    __syncthreads();
#pragma unroll
    for (int k = 0; k < (WV == 2 ? 2 : 4); ++k) {
        const int unit = unit0 + k * kWarps;
        if (unit >= units || (split > 1 && k > 0)) break;
#pragma unroll
        for (int m = 0; m < (WV == 2 ? 2 : 1); ++m) {
            const int ms = WV == 2 ? 2 * k + m : k;
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
                if (nt < ntv)
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int b = 8 * nt + 2 * c + (i & 1);
                        if (b < Hq) atomicAdd(sr + b * ipv + slot_coord<WV>(unit, m, gq, i >> 1), acc[ms][nt][i]);
                    }
        }
    }
    __syncthreads();
    emit_segment(p, sr, sM, sL, sp, ov, si, n_parts, slot0 + part, slot0, &s_last);
    }  // segments
}

// ------------------------------------------- warp-autonomous variant --
// For 2-bit keys and values whose cache rows fit one group (at most 128
// values, e.g. two heads of 48 or 64): each warp owns every eighth 16-token
// tile of the block's segment and takes it through its own cp.async stages,
// the logits, an online softmax of its own (running max and sum per head in
// registers) and the rotated value sums (all 128 coordinates of its heads,
// 64 registers), without a block barrier in the loop. The warps' states
// merge once per segment.
constexpr int kWRows = 16;                        // tokens per warp tile
constexpr int kWKRow = 32;                        // staged key row (one group of 2-bit codes)
constexpr int kWVRow = 48;                        // staged value row: 32 bytes + 16 (the four rows a warp
                                                  // reads per byte position fall in distinct banks)
constexpr int kWOffV = kWRows * kWKRow;           // value rows
constexpr int kWOffN = kWOffV + kWRows * kWVRow;  // key norms (16 fp16), then value norms
constexpr int kWStage = kWOffN + 64;
constexpr int kWStages = 4;
constexpr int kWScr = 20;                         // scratch row stride (floats): conflict-free transposes

// 2^x by the hardware approximation (relative error about 2^-22; 2^-inf = 0).
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// NTK: key-side n-tiles (hi and lo columns of 4 heads each), ceil(Hq / 4).
template <int NTK>
__global__ void __launch_bounds__(kThreads, 2) kv_attend_warp_kernel(const __grid_constant__ KvParams p) {
    constexpr int ntk = NTK, ntv = (NTK + 1) / 2;  // value side: 8 heads per n-tile
    extern __shared__ __align__(16) uint8_t smem[];
    __shared__ float sMw[kWarps][kMaxHeads], sLw[kWarps][kMaxHeads], sFw[kWarps][kMaxHeads];
    __shared__ float sM[kMaxHeads], sL[kMaxHeads];
    __shared__ int s_last;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int gq = lane >> 2, c = lane & 3, r16 = lane & 15;
    const int Hq = p.Hq;

    const uint2 *tabk = reinterpret_cast<const uint2 *>(smem + p.sm_tabk) + r16;  // [256][16] levels of a byte
    const uint2 *tabv = reinterpret_cast<const uint2 *>(smem + p.sm_tabv) + r16;
    uint2 *zf = reinterpret_cast<uint2 *>(smem + p.sm_zf);
    float *isig = reinterpret_cast<float *>(smem + p.sm_isig);
    float *scr = reinterpret_cast<float *>(smem + p.sm_p) + warp * kWRows * kWScr;  // this warp's [16][kWScr]
    uint8_t *wst = smem + p.sm_stage + warp * kWStages * kWStage;                  // this warp's stages
    uint32_t *terms = reinterpret_cast<uint32_t *>(smem + p.sm_terms);  // setup only (aliases the stages)
    float *sr = reinterpret_cast<float *>(smem + p.sm_r);               // end only: [Hq][128], then merge factors

    for (int side = 0; side < 2; ++side) {  // byte -> four fp16 levels, 16 replicas
        if (side == 1 && p.sm_tabv == p.sm_tabk) break;
        const uint16_t *lv = side ? p.lvv : p.lvk;
        uint32_t *t = reinterpret_cast<uint32_t *>(smem + (side ? p.sm_tabv : p.sm_tabk));
        for (int i = tid; i < 256 * 16; i += kThreads) {
            const int e = i >> 4;
            t[2 * i] = (uint32_t)lv[e & 3] | ((uint32_t)lv[(e >> 2) & 3] << 16);
            t[2 * i + 1] = (uint32_t)lv[(e >> 4) & 3] | ((uint32_t)lv[e >> 6] << 16);
        }
    }
    for (int q = blockIdx.x; q < p.n_seqs; q += gridDim.x)  // empty softmax: o = 0
        if (p.s[q].n == 0)
            for (int i = tid; i < Hq * p.dv; i += kThreads) p.s[q].o[i] = 0.0f;

    const int G = gridDim.x, T = p.total_sub, bid = blockIdx.x;
    const int x_end = (int)(((long long)(bid + 1) * T) / G);
    for (int x = (int)(((long long)bid * T) / G); x < x_end;) {
        int lo = 0, hi = p.n_seqs - 1;  // the sequence holding sub-tile x
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (p.s[mid].sub0 <= x) lo = mid;
            else hi = mid - 1;
        }
        const int si = lo;
        const uint8_t *const kc = p.s[si].kc;
        const uint8_t *const vc = p.s[si].vc;
        float *const ov = p.s[si].o;
        const int cap = p.s[si].cap, n_tok = p.s[si].n, n_parts = p.s[si].n_parts, slot0 = p.s[si].slot0;
        const int sub0 = p.s[si].sub0, sub_end = sub0 + (n_tok + kTile - 1) / kTile;
        const int seg_end = min(x_end, sub_end), part = bid - p.s[si].part_b0;
        const int t_begin = (x - sub0) * kTile, t_end = min(n_tok, (seg_end - sub0) * kTile);
        x = seg_end;
        rotate_queries(p, p.s[si].q, terms, isig, zf);  // ends with a barrier: the stages are free

        const uint8_t *const knorm_b = kc + (size_t)cap * kWKRow;
        const uint8_t *const vnorm_b = vc + (size_t)cap * 32;
        const int ntiles = (t_end - t_begin + kWRows - 1) / kWRows;
        const int mine = warp < ntiles ? (ntiles - warp + kWarps - 1) / kWarps : 0;
        // Copies of this warp's k-th tile into stage k % kWStages (one commit
        // group per tile, empty past the end): lane l copies half l & 1 of key
        // and value row l >> 1; lanes 0-3 the two norm blocks.
        auto issue = [&](int k) {
            if (k < mine) {
                uint8_t *st = wst + (k % kWStages) * kWStage;
                const int t0 = t_begin + (warp + kWarps * k) * kWRows, nv = min(kWRows, t_end - t0);
                const int r = lane >> 1, h = lane & 1;
                const bool ok = r < nv;
                const size_t row = (size_t)(t0 + (ok ? r : 0));
                cp_async16(st + r * kWKRow + 16 * h, kc + row * kWKRow + 16 * h, ok ? 16 : 0);
                cp_async16(st + kWOffV + r * kWVRow + 16 * h, vc + row * 32 + 16 * h, ok ? 16 : 0);
                if (lane < 4) {
                    const int which = lane >> 1, piece = lane & 1;
                    const int bytes = min(16, max(0, 2 * nv - 16 * piece));
                    const uint8_t *src = (which ? vnorm_b : knorm_b) + (size_t)t0 * 2 + 16 * piece;
                    cp_async16(st + kWOffN + 32 * which + 16 * piece, bytes ? src : knorm_b, bytes);
                }
            }
            cp_async_commit();
        };

        float m_h[4], l_h[4];  // running max (base 2) and sum of heads 4 nt + c
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) {
            m_h[nt] = -INFINITY;
            l_h[nt] = 0.0f;
        }
        float acc[8][2][4];  // slot 2u + m: coordinates 4(8u + gq) + 2m + {0 (row gq), 1 (row gq + 8)}
#pragma unroll
        for (int j = 0; j < 8; ++j)
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int i = 0; i < 4; ++i) acc[j][nt][i] = 0.0f;

        for (int k = 0; k + 1 < kWStages; ++k) issue(k);
        for (int k = 0; k < mine; ++k) {
            issue(k + kWStages - 1);
            cp_async_wait<kWStages - 1>();
            __syncwarp();
            const uint8_t *st = wst + (k % kWStages) * kWStage;
            const int t0 = t_begin + (warp + kWarps * k) * kWRows, nv = min(kWRows, t_end - t0);
            const __half *kn = reinterpret_cast<const __half *>(st + kWOffN);
            const __half *vn = kn + kWRows;
            // ---- logits of rows gq and gq + 8 for heads 4 nt + c ----
            const bool va = gq < nv, vb = gq + 8 < nv;
            float sa[4], sb[4];
            {
                const uint2 ca = *reinterpret_cast<const uint2 *>(st + gq * kWKRow + 8 * c);
                const uint2 cb = *reinterpret_cast<const uint2 *>(st + (gq + 8) * kWKRow + 8 * c);
                float d[4][4];
#pragma unroll
                for (int nt = 0; nt < 4; ++nt)
#pragma unroll
                    for (int i = 0; i < 4; ++i) d[nt][i] = 0.0f;
#pragma unroll
                for (int nu = 0; nu < 8; ++nu) {
                    const uint32_t wa = nu < 4 ? ca.x : ca.y, wb = nu < 4 ? cb.x : cb.y;
                    const uint2 ea = tabk[((wa >> (8 * (nu & 3))) & 0xffu) * 16];
                    const uint2 eb = tabk[((wb >> (8 * (nu & 3))) & 0xffu) * 16];
                    const uint2 *zb = zf + (nu * ntk) * 32 + lane;
#pragma unroll
                    for (int nt = 0; nt < 4; ++nt)
                        if (nt < ntk) {
                            const uint2 bf = zb[nt * 32];
                            mma_f16(d[nt], ea.x, eb.x, ea.y, eb.y, bf.x, bf.y);
                        }
                }
                const float na = __half2float(kn[gq]), nb = __half2float(kn[gq + 8]);
#pragma unroll
                for (int nt = 0; nt < 4; ++nt) {
                    const int b = 4 * nt + c;
                    const float is = nt < ntk && b < Hq ? isig[b] * p.logit_scale : 0.0f;
                    sa[nt] = va && nt < ntk && b < Hq ? na * is * (d[nt][0] + d[nt][1]) : -INFINITY;
                    sb[nt] = vb && nt < ntk && b < Hq ? nb * is * (d[nt][2] + d[nt][3]) : -INFINITY;
                }
            }
            // ---- online softmax of the warp's heads; weights p * n_v to the scratch ----
            const float nva = __half2float(vn[gq]), nvb = __half2float(vn[gq + 8]);  // 0 past the end
            bool moved = false;  // some head's running max changed: the sums are rescaled
#pragma unroll
            for (int nt = 0; nt < 4; ++nt) {
                const int b = 4 * nt + c;
                if (nt >= ntk) break;  // uniform
                float mx = fmaxf(sa[nt], sb[nt]);
#pragma unroll
                for (int o = 4; o < 32; o <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
                const float mn = b < Hq ? fmaxf(m_h[nt], mx) : 0.0f;  // a tile has a live row: finite
                const float pa = ex2(sa[nt] - mn), pb = ex2(sb[nt] - mn);
                float sum = pa + pb;
#pragma unroll
                for (int o = 4; o < 32; o <<= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
                const float f = b < Hq && mn != m_h[nt] ? ex2(m_h[nt] - mn) : 1.0f;  // 0 on the warp's first tile
                moved |= f != 1.0f;
                l_h[nt] = fmaf(l_h[nt], f, sum);
                m_h[nt] = mn;
                if (b < Hq) {
                    scr[gq * kWScr + b] = pa * nva;
                    scr[(gq + 8) * kWScr + b] = pb * nvb;
                    if (gq == 0) sFw[warp][b] = f;
                }
            }
            moved = __any_sync(0xffffffffu, moved);
            __syncwarp();
            // ---- rotated value sums: rescale, then A = coordinates x tokens ----
            uint2 bw[2];  // B fragments: tokens 2c, 2c+1 | 2c+8, 2c+9 of column (head) 8 nt + gq
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                const int b = 8 * nt + gq;
                bw[nt] = make_uint2(0u, 0u);
                if (nt < ntv && b < Hq) {
                    bw[nt].x = pack_h2(scr[2 * c * kWScr + b], scr[(2 * c + 1) * kWScr + b]);
                    bw[nt].y = pack_h2(scr[(2 * c + 8) * kWScr + b], scr[(2 * c + 9) * kWScr + b]);
                }
                if (nt < ntv && moved) {
                    const int h0 = 8 * nt + 2 * c;
                    const float f0 = h0 < Hq ? sFw[warp][h0] : 1.0f, f1 = h0 + 1 < Hq ? sFw[warp][h0 + 1] : 1.0f;
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        acc[j][nt][0] *= f0;
                        acc[j][nt][1] *= f1;
                        acc[j][nt][2] *= f0;
                        acc[j][nt][3] *= f1;
                    }
                }
            }
            const uint8_t *vrow = st + kWOffV + 2 * c * kWVRow + gq;
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const uint8_t *q = vrow + 8 * u;
                const uint2 h0 = tabv[(uint32_t)q[0] * 16], h1 = tabv[(uint32_t)q[kWVRow] * 16];
                const uint2 h2 = tabv[(uint32_t)q[8 * kWVRow] * 16], h3 = tabv[(uint32_t)q[9 * kWVRow] * 16];
                const uint32_t aA0 = __byte_perm(h0.x, h1.x, 0x5410), aA1 = __byte_perm(h0.x, h1.x, 0x7632);
                const uint32_t aA2 = __byte_perm(h2.x, h3.x, 0x5410), aA3 = __byte_perm(h2.x, h3.x, 0x7632);
                const uint32_t aB0 = __byte_perm(h0.y, h1.y, 0x5410), aB1 = __byte_perm(h0.y, h1.y, 0x7632);
                const uint32_t aB2 = __byte_perm(h2.y, h3.y, 0x5410), aB3 = __byte_perm(h2.y, h3.y, 0x7632);
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
                    if (nt < ntv) {
                        mma_f16(acc[2 * u][nt], aA0, aA1, aA2, aA3, bw[nt].x, bw[nt].y);
                        mma_f16(acc[2 * u + 1][nt], aB0, aB1, aB2, aB3, bw[nt].x, bw[nt].y);
                    }
            }
            __syncwarp();  // the scratch and this stage are rewritten next
        }
        cp_async_wait<0>();  // only empty groups remain

        // ---- merge the warps: per head M = max over warps, factors 2^(m_w - M) ----
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) {
            const int b = 4 * nt + c;
            if (gq == 0 && nt < ntk && b < Hq) {
                sMw[warp][b] = m_h[nt];
                sLw[warp][b] = l_h[nt];
            }
        }
        __syncthreads();  // every warp is out of its stages: sr may reuse them
        if (tid < Hq) {
            float mx = -INFINITY;
            for (int w = 0; w < kWarps; ++w) mx = fmaxf(mx, sMw[w][tid]);
            float l = 0.0f;
            for (int w = 0; w < kWarps; ++w)
                if (sMw[w][tid] != -INFINITY) l = fmaf(sLw[w][tid], exp2f(sMw[w][tid] - mx), l);
            sM[tid] = mx;
            sL[tid] = l;
        }
        for (int i = tid; i < Hq * kGroup; i += kThreads) sr[i] = 0.0f;
        __syncthreads();
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            if (nt >= ntv) break;
            const int h0 = 8 * nt + 2 * c;
            const float f0 = h0 < Hq && sMw[warp][h0] != -INFINITY ? exp2f(sMw[warp][h0] - sM[h0]) : 0.0f;
            const float f1 = h0 + 1 < Hq && sMw[warp][h0 + 1] != -INFINITY ? exp2f(sMw[warp][h0 + 1] - sM[h0 + 1]) : 0.0f;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int k0 = 4 * (8 * (j >> 1) + gq) + 2 * (j & 1);
                if (h0 < Hq) {
                    atomicAdd(sr + h0 * kGroup + k0, acc[j][nt][0] * f0);
                    atomicAdd(sr + h0 * kGroup + k0 + 1, acc[j][nt][2] * f0);
                }
                if (h0 + 1 < Hq) {
                    atomicAdd(sr + (h0 + 1) * kGroup + k0, acc[j][nt][1] * f1);
                    atomicAdd(sr + (h0 + 1) * kGroup + k0 + 1, acc[j][nt][3] * f1);
                }
            }
        }
        __syncthreads();
        emit_segment(p, sr, sM, sL, sr + Hq * kGroup, ov, si, n_parts, slot0 + part, slot0, &s_last);
    }  // segments
}

// Resident blocks per SM of one instance at `smem` bytes (sets the
// shared-memory attribute first), or a negative CQ error.
template <int WK, int WV>
int occupancy_t(int smem) {
    auto k = kv_attend_kernel<WK, WV>;
    const int rc = ensure_smem(reinterpret_cast<const void *>(k), smem);
    if (rc) return rc;
    int nb = 0;
    const cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, k, kThreads, smem);
    if (e != cudaSuccess) return set_error(CQ_ERR_CUDA, "kv attention occupancy: %s", cudaGetErrorString(e));
    return std::max(nb, 1);
}

template <int WK, int WV>
void launch_t(const KvParams &p, int grid, int smem, cudaStream_t st) {
    kv_attend_kernel<WK, WV><<<grid, kThreads, smem, st>>>(p);
}

template <int WK, int WV>
int dispatch_t(bool occ, const KvParams &p, int grid, int smem, cudaStream_t st) {
    if (occ) return occupancy_t<WK, WV>(smem);
    launch_t<WK, WV>(p, grid, smem, st);
    return CQ_OK;
}

// Resident blocks per SM of the warp-autonomous kernel at `smem` bytes.
template <int NTK>
int occupancy_warp_t(int smem) {
    const int rc = ensure_smem(reinterpret_cast<const void *>(kv_attend_warp_kernel<NTK>), smem);
    if (rc) return rc;
    int nb = 0;
    const cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, kv_attend_warp_kernel<NTK>, kThreads, smem);
    if (e != cudaSuccess) return set_error(CQ_ERR_CUDA, "kv attention occupancy: %s", cudaGetErrorString(e));
    return std::max(nb, 1);
}

// occ: the occupancy of the warp kernel for ntk key n-tiles; else launch it.
int dispatch_warp(int ntk, bool occ, const KvParams &p, int grid, int smem, cudaStream_t st) {
    switch (ntk) {
    case 1: if (occ) return occupancy_warp_t<1>(smem); kv_attend_warp_kernel<1><<<grid, kThreads, smem, st>>>(p); break;
    case 2: if (occ) return occupancy_warp_t<2>(smem); kv_attend_warp_kernel<2><<<grid, kThreads, smem, st>>>(p); break;
    case 3: if (occ) return occupancy_warp_t<3>(smem); kv_attend_warp_kernel<3><<<grid, kThreads, smem, st>>>(p); break;
    default: if (occ) return occupancy_warp_t<4>(smem); kv_attend_warp_kernel<4><<<grid, kThreads, smem, st>>>(p); break;
    }
    return CQ_OK;
}

// occ: return the occupancy of the (WK, WV) instance; else launch it.
int dispatch(int WK, int WV, bool occ, const KvParams &p, int grid, int smem, cudaStream_t st) {
    switch (WK * 8 + WV) {
    case 2 * 8 + 2: return dispatch_t<2, 2>(occ, p, grid, smem, st);
    case 2 * 8 + 3: return dispatch_t<2, 3>(occ, p, grid, smem, st);
    case 2 * 8 + 4: return dispatch_t<2, 4>(occ, p, grid, smem, st);
    case 3 * 8 + 2: return dispatch_t<3, 2>(occ, p, grid, smem, st);
    case 3 * 8 + 3: return dispatch_t<3, 3>(occ, p, grid, smem, st);
    case 3 * 8 + 4: return dispatch_t<3, 4>(occ, p, grid, smem, st);
    case 4 * 8 + 2: return dispatch_t<4, 2>(occ, p, grid, smem, st);
    case 4 * 8 + 3: return dispatch_t<4, 3>(occ, p, grid, smem, st);
    default: return dispatch_t<4, 4>(occ, p, grid, smem, st);
    }
}

int align16(int x) { return (x + 15) & ~15; }

}  // namespace

int launch_kv_attend(const cq_kv_geom &g, const cq_kv_seq *seqs, int n, const float *lk, const float *lv,
                     void *stream) {
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const int Hq = g.n_q_heads, Hkv = g.n_kv_heads;
    const int WK = width_of(g.k_bits), WV = width_of(g.v_bits);
    KvParams p;  // large parameter block (about 15 KB): built here, copied into the launch
    p.Hq = Hq;
    p.per = Hq / Hkv;
    p.dk = g.head_dim_k;
    p.dv = g.head_dim_v;
    p.in_k = Hkv * g.head_dim_k;
    p.in_v = Hkv * g.head_dim_v;
    p.ngk = in_padded(p.in_k) / kGroup;
    p.ngv = in_padded(p.in_v) / kGroup;
    p.ntk = (2 * Hq + 7) / 8;
    p.ntv = (Hq + 7) / 8;
    p.logit_scale = (float)((double)g.scale * 1.4426950408889634 / std::sqrt(128.0));
    for (int j = 0; j < 16; ++j) {
        p.lvk[j] = __half_as_ushort(__float2half_rn(lk[j]));
        p.lvv[j] = __half_as_ushort(__float2half_rn(lv[j]));
    }
    const int rbv = p.ngv * 16 * WV;
    p.vrow = (rbv % 32 == 16) ? rbv : rbv + 16;  // stride = 16 mod 32 bytes: the four row pairs a warp reads hit distinct banks
    const int rbk = p.ngk * 16 * WK;
    // key rows: a half-warp's 8-byte (2-bit) or 16-byte (4-bit) reads of
    // four or two rows fall in distinct banks
    p.krow = rbk;
    if (WK == 2 && rbk % 64 == 0) p.krow = rbk + 32;
    if (WK == 4 && rbk % 128 == 0) p.krow = rbk + 64;
    if (WK == 3 && rbk % 32 == 0) p.krow = rbk + 16;
    p.cprk_magic = (65536 + rbk / 16 - 1) / (rbk / 16);
    p.cprv_magic = (65536 + rbv / 16 - 1) / (rbv / 16);
    bool same_levels = WK == WV;
    for (int j = 0; j < 16; ++j) same_levels = same_levels && p.lvk[j] == p.lvv[j];

    // shared memory: tables, rotated-query fragments, 1/sigma, then one region
    // used in turn by the query terms (setup), the value codes (sub-tiles) and
    // the rotated sums (end), then norms, logits and value fragments
    int off = 0;
    // level tables: 2-bit codes a byte -> four levels (256 x 16 replicas x 8 B),
    // else a code pair -> two levels (4^W x 32 replicas x 4 B); one table when
    // keys and values share their codes and levels
    const int tabk_b = WK == 2 ? 256 * 16 * 8 : (1 << (2 * WK)) * 32 * 4;
    const int tabv_b = WV == 2 ? 256 * 16 * 8 : (1 << (2 * WV)) * 32 * 4;
    p.sm_tabk = off;  off += align16(tabk_b);
    if (same_levels) {
        p.sm_tabv = p.sm_tabk;
    } else {
        p.sm_tabv = off;  off += align16(tabv_b);
    }
    p.sm_zf = off;    off += align16(p.ngk * 8 * p.ntk * 32 * 8);
    p.sm_isig = off;  off += align16(Hq * p.ngk * 4);
    p.sm_p = off;     off += align16(kSpRow * kMaxHeads * 4);
    p.sm_wf = off;    off += align16(p.ngv * 8 * p.ntv * 32 * 8);
    // one stage: key rows, value rows (+16 bytes: 3-bit pairs may read one word
    // past a row), key norms, value norms
    p.off_v = align16(kTile * p.krow);
    p.off_kn = p.off_v + align16(kTile * p.vrow + 16);
    p.off_vn = p.off_kn + align16(kTile * 2 * p.ngk);
    p.stage_bytes = p.off_vn + align16(kTile * 2 * p.ngv);
    const int fixed = off;
    auto union_bytes = [&](int nb) {
        return align16(std::max({Hq * p.ngk * kGroup * 4, nb * p.stage_bytes, Hq * p.ngv * kGroup * 4}));
    };
    // the most stages that keep three blocks on an SM (228 KB, 1 KB reserved
    // per block); failing that, the most that fit one block
    const int per3 = 228 * 1024 / 3 - 1024, limit = 227 * 1024;
    p.n_stages = kMaxStages;
    while (p.n_stages > 1 && fixed + union_bytes(p.n_stages) > per3) --p.n_stages;
    if (fixed + union_bytes(p.n_stages) > per3) {
        p.n_stages = kMaxStages;
        while (p.n_stages > 1 && fixed + union_bytes(p.n_stages) > limit) --p.n_stages;
    }
    // the union region is used in turn by the query terms (setup), the stages
    // (sub-tiles) and the rotated sums (end)
    p.sm_terms = p.sm_stage = p.sm_r = off;
    off += union_bytes(p.n_stages);
    int smem = off;

    // 2-bit keys and values in rows of one group: the warp-autonomous kernel,
    // with its own layout after the tables: query fragments, 1/sigma, the
    // warps' scratch rows, then one region for the query terms (setup), the
    // warps' stages (loop) and the rotated sums with the merge factors (end)
    const bool warp_path = WK == 2 && WV == 2 && p.ngk == 1 && p.ngv == 1;
    if (warp_path) {
        off = p.sm_zf;
        off += align16(8 * p.ntk * 32 * 8);
        p.sm_isig = off;  off += align16(Hq * 4);
        p.sm_p = off;     off += align16(kWarps * kWRows * kWScr * 4);
        p.sm_terms = p.sm_stage = p.sm_r = off;
        off += align16(std::max({kWarps * kWStages * kWStage, Hq * kGroup * 4, Hq * kGroup * 4 + kMaxParts * Hq * 4}));
        smem = off;
    }

    const int per_sm = warp_path ? dispatch_warp(p.ntk, true, p, 0, smem, st) : dispatch(WK, WV, true, p, 0, smem, st);
    if (per_sm < 0) return per_sm;
    const long long slots_gpu = (long long)per_sm * sm_count();
    for (int base = 0; base < n; base += kMaxSeqs) {
        const int cnt = std::min(kMaxSeqs, n - base);
        long long total = 0;
        for (int i = 0; i < cnt; ++i) total += (seqs[base + i].n_tokens + kTile - 1) / kTile;
        if (total > (1LL << 30)) return set_error(CQ_ERR_SHAPE, "too many cached tokens in one call");
        // one block per resident slot, each an equal run of the flat sub-tile order
        const int T = (int)total;
        int G = (int)std::max(1LL, std::min<long long>(slots_gpu, total));
        auto block_of = [&](long long x) { return (int)(((x + 1) * G - 1) / T); };  // block holding sub-tile x
        for (;;) {  // at most kMaxParts blocks per sequence (the merge keeps one factor per part and head)
            int worst = 0, s0 = 0;
            for (int i = 0; i < cnt; ++i) {
                const int ns = (seqs[base + i].n_tokens + kTile - 1) / kTile;
                if (ns) worst = std::max(worst, block_of(s0 + ns - 1) - block_of(s0) + 1);
                s0 += ns;
            }
            if (worst <= kMaxParts || G == 1) break;
            G = std::max(1, G * 3 / 4);
        }
        int slots = 0, sub = 0;
        for (int i = 0; i < cnt; ++i) {
            const cq_kv_seq &s = seqs[base + i];
            KvSeqDev &d = p.s[i];
            d.kc = s.k_cache;
            d.vc = s.v_cache;
            d.q = s.q;
            d.o = s.o;
            d.cap = s.cap;
            d.n = s.n_tokens;
            const int ns = (s.n_tokens + kTile - 1) / kTile;
            d.sub0 = sub;
            d.part_b0 = ns ? block_of(sub) : 0;
            d.n_parts = ns ? block_of(sub + ns - 1) - d.part_b0 + 1 : 0;
            d.slot0 = slots;
            if (d.n_parts > 1) slots += d.n_parts;
            sub += ns;
        }
        p.n_seqs = cnt;
        p.total_sub = T;
        p.part = nullptr;
        p.ml = nullptr;
        p.ticket = nullptr;
        if (slots > 0) {
            const size_t part_b = ((size_t)slots * Hq * p.ngv * kGroup * 4 + 255) & ~(size_t)255;
            const size_t ml_b = ((size_t)slots * Hq * 2 * 4 + 255) & ~(size_t)255;
            int err = CQ_OK;
            uint8_t *ws = static_cast<uint8_t *>(stream_workspace(stream, 1, part_b + ml_b + (size_t)cnt * 4, &err));
            if (!ws) return err;
            p.part = reinterpret_cast<float *>(ws);
            p.ml = reinterpret_cast<float *>(ws + part_b);
            p.ticket = reinterpret_cast<unsigned int *>(ws + part_b + ml_b);
            const cudaError_t e = cudaMemsetAsync(p.ticket, 0, (size_t)cnt * 4, st);
            if (e != cudaSuccess) return set_error(CQ_ERR_CUDA, "kv attention tickets: %s", cudaGetErrorString(e));
        }
        if (warp_path) dispatch_warp(p.ntk, false, p, G, smem, st);
        else dispatch(WK, WV, false, p, G, smem, st);
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return set_error(CQ_ERR_CUDA, "kv attention launch: %s", cudaGetErrorString(e));
    }
    return CQ_OK;
}

}  // namespace cq
