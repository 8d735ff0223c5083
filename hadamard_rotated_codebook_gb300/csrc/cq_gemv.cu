// cq_gemv.cu -- matrix-vector products over CQ-packed weights (batch 1..16),
// single and grouped.
//
// The rotated-domain identity (OpenNeedle docs/reference.md; "The .cact
// archive and Cactus Quants", "Reconstructing one group"): with H symmetric
// and orthogonal, <w_hat_g, x_g> = n_g * <c[q_g], H x_g>. Each activation
// group is rotated once by a fast Walsh-Hadamard transform in registers and
// reused for every output row; the codes are looked up, never expanded to a
// dense matrix ("The .cact format", "How the kernel reads it").
//
// Work decomposition: a work item is (matrix, tile of 32 rows, chunk of
// groups). A CTA rotates the activation chunk of its item into shared memory
// (fp32, one warp per group: four coordinates per lane, two butterfly stages
// in registers and five with shuffles), then its threads take (row, group)
// pairs: each loads the group's 16*width code bytes with 16-byte loads,
// accumulates level*z in fp32 for every batch column, scales by the group
// norm and adds into a per-row shared accumulator. Rows split over several
// chunks (long inputs with a large batch) accumulate into y atomically.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "cq_internal.h"

namespace cq {
namespace {

constexpr int kGemvThreads = 256;
constexpr int kRowsPerItem = 32;
constexpr int kZPad = kGroup + 1;            // padded group stride in shared memory
constexpr int kZBudgetFloats = 12288;        // 48 KB of rotated activations
constexpr float kInvSqrt128 = 0.08838834764831845f;

struct GemvMat {
    const uint8_t *codes;
    const __half *norms;
    const void *x;
    const float *xs;
    float *y;
    int out, in, ng, bits, xdt, B, lut, kcg, nchunks, row_tiles, items_before;
    int group;  // 128 or 64
};

struct GemvParams {
    int n, total_items, zfloats;
    float lut[kMaxLuts][16];
    GemvMat m[CQ_MAX_GROUPED];
};

// Rotates activation groups [gbeg, gend) of every batch row into zs:
// zs[(b*kcg + (g-gbeg))*kZPad + k] = (H x_{b,g})[k]. A warp task covers 128
// positions: one group of 128, or two groups of 64 (lanes 0-15 and 16-31,
// whose transforms stop before the stage that would mix the two halves).
__device__ void rotate_chunk(const GemvMat &M, int gbeg, int gend, int kcg, float *zs) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int ngc = gend - gbeg, per = kGroup / M.group, nspan = (ngc + per - 1) / per;
    const int half = M.group == kGroup ? 32 : 16;  // lanes per group
    for (int task = warp; task < M.B * nspan; task += kGemvThreads / 32) {
        const int b = task / nspan, gl = (task % nspan) * per + lane / half, g = gbeg + gl;
        const bool live = gl < ngc;
        float v[4];
        float scale = M.group == kGroup ? kInvSqrt128 : 0.125f;
        if (M.xdt == CQ_X_I8) {
            const int8_t *xq = static_cast<const int8_t *>(M.x) + (size_t)b * M.in;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int col = g * M.group + (4 * lane + i) % M.group;
                v[i] = live && col < M.in ? (float)xq[col] : 0.0f;
            }
            scale = __fmul_rn(M.xs[b], scale);
        } else {
            const float *xf = static_cast<const float *>(M.x) + (size_t)b * M.in;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int col = g * M.group + (4 * lane + i) % M.group;
                v[i] = live && col < M.in ? xf[col] : 0.0f;
            }
        }
        // coordinate bits 0,1 in registers
        float a0 = v[0] + v[1], a1 = v[0] - v[1], a2 = v[2] + v[3], a3 = v[2] - v[3];
        v[0] = a0 + a2;
        v[1] = a1 + a3;
        v[2] = a0 - a2;
        v[3] = a1 - a3;
        // coordinate bits 2..6 across lanes (bit 6 only within a group of 128)
#pragma unroll
        for (int m = 1; m < 32; m <<= 1)
            if (m < half)
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float o = __shfl_xor_sync(0xffffffffu, v[i], m);
                    v[i] = (lane & m) ? o - v[i] : v[i] + o;
                }
        if (live) {
            float *dst = zs + (size_t)(b * kcg + gl) * kZPad + (4 * lane) % M.group;
#pragma unroll
            for (int i = 0; i < 4; ++i) dst[i] = v[i] * scale;
        }
    }
}

template <int W>
__device__ __forceinline__ uint32_t code_at(const uint32_t (&w)[4 * W], int k) {  // code k of a group
    const int bit = k * W, word = bit >> 5, off = bit & 31;
    uint32_t v = w[word] >> off;
    if (off + W > 32) v |= w[word + 1] << (32 - off);
    return v & ((1u << W) - 1u);
}

template <int W, int BMAX>
__global__ void __launch_bounds__(kGemvThreads) gemv_kernel(const __grid_constant__ GemvParams p) {
    extern __shared__ float smem[];
    float *zs = smem;
    float *ys = smem + p.zfloats;  // [kRowsPerItem][16]
    __shared__ float lut_s[16];

    for (int item = blockIdx.x; item < p.total_items; item += gridDim.x) {
        // locate the matrix of this item
        int lo = 0, hi = p.n - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) / 2;
            if (p.m[mid].items_before <= item) lo = mid;
            else hi = mid - 1;
        }
        const GemvMat &M = p.m[lo];
        const int local = item - M.items_before;
        const int rt = local / M.nchunks, kc = local % M.nchunks;
        const int gbeg = kc * M.kcg, gend = min(M.ng, gbeg + M.kcg);
        const int row0 = rt * kRowsPerItem;
        const int B = M.B;

        if (threadIdx.x < 16) lut_s[threadIdx.x] = p.lut[M.lut][threadIdx.x];
        for (int i = threadIdx.x; i < kRowsPerItem * 16; i += kGemvThreads) ys[i] = 0.0f;
        rotate_chunk(M, gbeg, gend, M.kcg, zs);
        __syncthreads();

        const int ngc = gend - gbeg, G = M.group;
        const size_t grpBytes = (size_t)G * W / 8, rowBytes = (size_t)M.ng * grpBytes;
        for (int pr = threadIdx.x; pr < kRowsPerItem * ngc; pr += kGemvThreads) {
            const int r = pr / ngc, gl = pr % ngc, o = row0 + r;
            if (o >= M.out) continue;
            const int g = gbeg + gl;
            uint32_t w[4 * W];
            const uint8_t *gp = M.codes + (size_t)o * rowBytes + (size_t)g * grpBytes;
            if (G == kGroup) {  // 16 W bytes: W 16-byte loads
                const uint4 *src = reinterpret_cast<const uint4 *>(gp);
#pragma unroll
                for (int i = 0; i < W; ++i) {
                    const uint4 t = __ldg(src + i);
                    w[4 * i] = t.x;
                    w[4 * i + 1] = t.y;
                    w[4 * i + 2] = t.z;
                    w[4 * i + 3] = t.w;
                }
            } else {  // 8 W bytes: W 8-byte loads
                const uint2 *src = reinterpret_cast<const uint2 *>(gp);
#pragma unroll
                for (int i = 0; i < W; ++i) {
                    const uint2 t = __ldg(src + i);
                    w[2 * i] = t.x;
                    w[2 * i + 1] = t.y;
                }
#pragma unroll
                for (int i = 2 * W; i < 4 * W; ++i) w[i] = 0u;
            }
            float acc[BMAX];
#pragma unroll
            for (int b = 0; b < BMAX; ++b) acc[b] = 0.0f;
            const float *z = zs + (size_t)gl * kZPad;
#pragma unroll 8
            for (int k = 0; k < G; ++k) {
                const float lv = lut_s[code_at<W>(w, k)];
#pragma unroll
                for (int b = 0; b < BMAX; ++b)
                    if (b < B) acc[b] = fmaf(lv, z[(size_t)b * M.kcg * kZPad + k], acc[b]);
            }
            const float nrm = __half2float(M.norms[(size_t)o * M.ng + g]);
#pragma unroll
            for (int b = 0; b < BMAX; ++b)
                if (b < B) atomicAdd(&ys[r * 16 + b], acc[b] * nrm);
        }
        __syncthreads();
        for (int i = threadIdx.x; i < kRowsPerItem * B; i += kGemvThreads) {
            const int r = i / B, b = i % B, o = row0 + r;
            if (o >= M.out) continue;
            float *dst = M.y + (size_t)b * M.out + o;
            if (M.nchunks == 1) *dst = ys[r * 16 + b];
            else atomicAdd(dst, ys[r * 16 + b]);
        }
        __syncthreads();
    }
}

template <int W, int BMAX>
int launch_w(const GemvParams &p, size_t smem, int grid, cudaStream_t st) {
    auto k = gemv_kernel<W, BMAX>;
    const int rc = ensure_smem(reinterpret_cast<const void *>(k), 64 * 1024 + 4096);
    if (rc) return rc;
    k<<<grid, kGemvThreads, smem, st>>>(p);
    return CQ_OK;
}

template <int W>
int launch_b(int bmax, const GemvParams &p, size_t smem, int grid, cudaStream_t st) {
    if (bmax <= 1) return launch_w<W, 1>(p, smem, grid, st);
    if (bmax <= 4) return launch_w<W, 4>(p, smem, grid, st);
    if (bmax <= 8) return launch_w<W, 8>(p, smem, grid, st);
    return launch_w<W, 16>(p, smem, grid, st);
}

}  // namespace

namespace {

// Whether the descriptor takes the decode kernel (the routing below).
bool takes_fast(const cq_gemv_desc &d) {
    const bool g64w = d.group == kGroup64 && gemv_wide_eligible(d);
    return !g64w && !gemv_stream_eligible(d) && gemv_fast_eligible(d);
}

// CQ_X_F32Q activations of descriptors that the decode kernel does not take
// are quantised first (one quantiser launch per distinct activation, into a
// library workspace); their descriptors then read int8 and the scales. The
// decode kernel quantises its own. Returns the descriptors to route (d
// itself when nothing was quantised), or null with *err set.
const cq_gemv_desc *prequantize(const cq_gemv_desc *d, int n, void *stream, int *err) {
    bool any = false;
    for (int i = 0; i < n && !any; ++i) any = d[i].x_dtype == CQ_X_F32Q && d[i].out > 0 && d[i].in > 0 && !takes_fast(d[i]);
    if (!any) return d;
    static thread_local cq_gemv_desc dq[CQ_MAX_GROUPED];
    int src[CQ_MAX_GROUPED];  // descriptor whose activation another one shares (or itself)
    size_t off[CQ_MAX_GROUPED], bytes = 0;
    for (int i = 0; i < n; ++i) {
        dq[i] = d[i];
        src[i] = -1;
        if (d[i].x_dtype != CQ_X_F32Q || d[i].out <= 0 || d[i].in <= 0 || takes_fast(d[i])) continue;
        for (int j = 0; j < i && src[i] < 0; ++j)
            if (src[j] == j && d[j].x == d[i].x && d[j].in == d[i].in && d[j].B == d[i].B) src[i] = j;
        if (src[i] >= 0) continue;
        src[i] = i;
        off[i] = bytes;  // int8 [B][in], then fp32 scales [B], 256-byte aligned pieces
        bytes += ((size_t)d[i].B * d[i].in + 255) / 256 * 256 + ((size_t)d[i].B * 4 + 255) / 256 * 256;
    }
    uint8_t *ws = static_cast<uint8_t *>(stream_workspace(stream, 4, bytes, err));
    if (!ws) return nullptr;
    for (int i = 0; i < n; ++i) {
        if (src[i] < 0) continue;
        const int j = src[i];
        int8_t *q = reinterpret_cast<int8_t *>(ws + off[j]);
        float *sc = reinterpret_cast<float *>(ws + off[j] + ((size_t)d[j].B * d[j].in + 255) / 256 * 256);
        if (j == i) {
            const int rc = launch_act_quant(static_cast<const float *>(d[i].x), d[i].B, d[i].in, q, sc, stream);
            if (rc) {
                *err = rc;
                return nullptr;
            }
        }
        dq[i].x = q;
        dq[i].x_scale = sc;
        dq[i].x_dtype = CQ_X_I8;
    }
    return dq;
}

}  // namespace

int launch_gemv_grouped(const cq_gemv_desc *d_in, int n, void *stream) {
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    int qerr = CQ_OK;
    const cq_gemv_desc *d = prequantize(d_in, n, stream, &qerr);
    if (!d) return qerr;
    // The tensor-core kernels take what they can: one launch for all of the
    // matrices with inputs up to 15 groups, a streamed launch for 3-bit codes
    // of 16 to 32 groups, a rotation launch and split or sliced products for
    // the rest (groups of 64 go there first, and to the streamed kernel only
    // if no split launch takes them); what is left runs here.
    int fast_idx[CQ_MAX_GROUPED], nfast = 0, stream_idx[CQ_MAX_GROUPED], nstream = 0;
    int wide_idx[CQ_MAX_GROUPED], nwide = 0, rejected[CQ_MAX_GROUPED], nrej = 0;
    bool is_fast[CQ_MAX_GROUPED];
    for (int i = 0; i < n; ++i) {
        const bool g64w = d[i].group == kGroup64 && gemv_wide_eligible(d[i]);
        const bool sf = !g64w && gemv_stream_eligible(d[i]);
        const bool ff = !g64w && !sf && gemv_fast_eligible(d[i]);
        const bool wf = g64w || (!sf && !ff && gemv_wide_eligible(d[i]));
        is_fast[i] = sf || ff || wf;
        if (sf) stream_idx[nstream++] = i;
        else if (ff) fast_idx[nfast++] = i;
        else if (wf) wide_idx[nwide++] = i;
    }
    if (nfast) {
        int st2 = launch_gemv_fast(d, fast_idx, nfast, stream);
        if (st2) return st2;
    }
    if (nwide) {
        int st2 = launch_gemv_wide(d, wide_idx, nwide, stream, rejected, &nrej);
        if (st2) return st2;
        for (int r = 0; r < nrej; ++r) {
            const int i = rejected[r];
            if (gemv_stream_eligible(d[i])) stream_idx[nstream++] = i;
            else is_fast[i] = false;
        }
    }
    if (nstream) {
        int st2 = launch_gemv_stream(d, stream_idx, nstream, stream);
        if (st2) return st2;
    }
    // One launch per code width present; each launch walks all descriptors of
    // its width (matrices of other widths contribute no items).
    for (int W = 1; W <= 4; ++W) {
        static thread_local GemvParams p;  // large: off the stack, one per host thread
        p.n = 0;
        int bmax = 0, nlut = 0, items = 0, zfloats = 0;
        for (int i = 0; i < n; ++i) {
            if (is_fast[i] || width_of(d[i].bits) != W || d[i].out == 0) continue;
            if (d[i].in == 0) {  // empty reduction: the product is zero
                cudaMemsetAsync(d[i].y, 0, sizeof(float) * d[i].B * d[i].out, st);
                continue;
            }
            GemvMat &M = p.m[p.n];
            const int ip = in_padded(d[i].in, d[i].group);
            M.group = d[i].group;
            M.codes = d[i].blob;
            M.norms = reinterpret_cast<const __half *>(d[i].blob + (size_t)d[i].out * ip * W / 8);
            M.x = d[i].x;
            M.xs = d[i].x_scale;
            M.y = d[i].y;
            M.out = d[i].out;
            M.in = d[i].in;
            M.ng = ip / d[i].group;
            M.bits = d[i].bits;
            M.xdt = d[i].x_dtype;
            M.B = d[i].B;
            // level table for the stored codes (ternary crumbs sign-extend)
            float lut[16] = {0};
            if (d[i].bits == 5) {
                const float c = d[i].codebook[2];
                lut[0] = 0.0f;
                lut[1] = c;
                lut[2] = -2.0f * c;
                lut[3] = -c;
            } else {
                for (int j = 0; j < levels_of(d[i].bits); ++j) lut[j] = d[i].codebook[j];
            }
            int li = -1;
            for (int j = 0; j < nlut; ++j)
                if (std::equal(lut, lut + 16, p.lut[j])) li = j;
            if (li < 0) {
                if (nlut == kMaxLuts) return set_error(CQ_ERR_ARG, "more than %d distinct codebooks in one call", kMaxLuts);
                std::copy(lut, lut + 16, p.lut[nlut]);
                li = nlut++;
            }
            M.lut = li;
            const int bclass = M.B <= 1 ? 1 : M.B <= 4 ? 4 : M.B <= 8 ? 8 : 16;
            bmax = std::max(bmax, bclass);
            M.kcg = std::max(1, std::min(M.ng, kZBudgetFloats / (M.B * kZPad)));
            M.nchunks = (M.ng + M.kcg - 1) / M.kcg;
            M.row_tiles = (M.out + kRowsPerItem - 1) / kRowsPerItem;
            M.items_before = items;
            items += M.row_tiles * M.nchunks;
            zfloats = std::max(zfloats, M.B * M.kcg * kZPad);
            if (M.nchunks > 1) cudaMemsetAsync(M.y, 0, sizeof(float) * M.B * M.out, st);
            ++p.n;
        }
        if (p.n == 0) continue;
        p.total_items = items;
        p.zfloats = zfloats;
        const size_t smem = sizeof(float) * (zfloats + kRowsPerItem * 16);
        const int grid = std::min(items, sm_count() * 8);
        int rc = CQ_OK;
        switch (W) {
        case 1: rc = launch_b<1>(bmax, p, smem, grid, st); break;
        case 2: rc = launch_b<2>(bmax, p, smem, grid, st); break;
        case 3: rc = launch_b<3>(bmax, p, smem, grid, st); break;
        case 4: rc = launch_b<4>(bmax, p, smem, grid, st); break;
        }
        if (rc) return rc;
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return set_error(CQ_ERR_CUDA, "gemv launch: %s", cudaGetErrorString(e));
    }
    return CQ_OK;
}

}  // namespace cq

// Diagnostic (include/cq.h): the split products' tile counters of `stream`
// set to a nonzero pattern.
extern "C" int cq_selftest_dirty_counters(void *stream) {
    using namespace cq;
    clear_error();
    int err = CQ_OK;
    unsigned int *c = stream_counters(stream, 1024, &err);
    if (!c) return err;
    if (cudaMemsetAsync(c, 0x01, 1024 * sizeof(unsigned int), reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
        return set_error(CQ_ERR_CUDA, "counter fill: %s", cudaGetErrorString(cudaGetLastError()));
    return CQ_OK;
}
