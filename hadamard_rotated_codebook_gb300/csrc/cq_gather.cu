// cq_gather.cu -- row-gather dequantisation of a CQ table: only the rows a
// step indexes (token embeddings, engram rows) are rebuilt, each group as
//     w_hat[g*128 + k] = n[g] * (H c[q_g])[k],  H = H0 / sqrt(128)
// ("The .cact archive and Cactus Quants", "Reconstructing one group").
//
// GB300 mapping: a warp decodes two indexed rows, four groups at a time.
// Lane (grp, s) owns the positions 32t + 4s + j (t, j < 4) of a group: it
// loads their code bits itself (one to two bytes per t), takes the levels
// from registers (2-bit codes) or a 16-entry shared table, and the warp runs
// the 128-point transform as four butterfly stages in registers and three
// shuffle stages across the group's eight lanes; store t of those eight
// lanes then covers 128 contiguous output bytes. The two rows' indices, and
// then their code bytes, are requested together so that one latency covers
// both. The work is bound by HBM: the fp32 output is 8 to 16 times the code
// bytes it decodes.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "cq_internal.h"

namespace cq {

namespace {

constexpr int kWarps = 8;
constexpr int kRows = 2;  // indexed rows per warp
constexpr float kInvSqrt128 = 0.08838834764831845f;

struct GatherArgs {
    const uint8_t *codes;
    const __half *norms;
    const int32_t *idx;
    float *dst;
    unsigned int *status;
    int out, in, ng, n;  // ng: groups per row
    float lv[16];
};

// Zero row for an index out of range (the host learns of it from the status word).
__device__ __forceinline__ void zero_row(float *d, int in, bool vec, int lane) {
    for (int k = 4 * lane; k < in; k += 128) {
        if (vec) {
            *reinterpret_cast<float4 *>(d + k) = make_float4(0.f, 0.f, 0.f, 0.f);
        } else {
#pragma unroll
            for (int j = 0; j < 4; ++j)
                if (k + j < in) d[k + j] = 0.0f;
        }
    }
}

// The 4*W code bits of positions 32t + 4s .. 32t + 4s + 3 of a group whose
// codes start at `grp` (LSB-first packing).
template <int W>
__device__ __forceinline__ uint32_t load_codes4(const uint8_t *grp, int s, int t) {
    if (W == 1) return (__ldg(grp + 4 * t + (s >> 1)) >> (4 * (s & 1))) & 0xfu;
    if (W == 2) return __ldg(grp + 8 * t + s);
    if (W == 4) return __ldg(reinterpret_cast<const uint16_t *>(grp) + 8 * t + s);
    const int b = 96 * t + 12 * s;  // W == 3: twelve bits, two bytes
    return ((uint32_t)__ldg(grp + (b >> 3)) | ((uint32_t)__ldg(grp + (b >> 3) + 1) << 8)) >> (b & 7);
}

// A warp decodes four spans of 128 positions at once (a span is one group
// of 128, or two groups of 64). Lane (grp, s) = (lane / 8, lane % 8) owns
// the 16 positions 32t + 4s + j (t, j < 4) of span g0 + grp, so that store t
// of the span's eight lanes covers 128 contiguous bytes. The transform runs
// as butterfly stages in registers (position bits 0, 1, 5 and, for groups of
// 128, 6) and three shuffle stages across the eight lanes (bits 2, 3, 4).
template <int W, int G>
__global__ void __launch_bounds__(kWarps * 32) gather_rows_kernel(const __grid_constant__ GatherArgs a) {
    __shared__ float s_lv[16];
    if (threadIdx.x < 16) s_lv[threadIdx.x] = a.lv[threadIdx.x];
    __syncthreads();
    const int lane = threadIdx.x & 31, grp = lane >> 3, sl = lane & 7;
    const int i0 = (blockIdx.x * kWarps + (threadIdx.x >> 5)) * kRows;
    if (i0 >= a.n) return;
    const bool vec = (a.in & 3) == 0 && (reinterpret_cast<uintptr_t>(a.dst) & 15) == 0;
    const size_t gbytes = (size_t)16 * W;  // code bytes per span
    const int nspan = (a.ng * G + kGroup - 1) / kGroup;
    // 1- and 2-bit codes: the levels in registers (selects instead of table reads)
    const float l0 = a.lv[0], l1 = a.lv[1], l2 = a.lv[2], l3 = a.lv[3];
    int row[kRows];
#pragma unroll
    for (int r = 0; r < kRows; ++r) row[r] = i0 + r < a.n ? a.idx[i0 + r] : 0;
#pragma unroll
    for (int r = 0; r < kRows; ++r) {
        if (i0 + r < a.n && (row[r] < 0 || row[r] >= a.out)) {
            if (lane == 0 && a.status) atomicOr(a.status, kStatusIndex);
            zero_row(a.dst + (size_t)(i0 + r) * a.in, a.in, vec, lane);
            row[r] = -1;
        } else if (i0 + r >= a.n) {
            row[r] = -1;
        }
    }
    const size_t row_bytes = (size_t)a.ng * G * W / 8;
    for (int g0 = 0; g0 < nspan; g0 += 4) {
        const int g = g0 + grp;
        const bool live_g = g < nspan;
        uint32_t code[kRows][4];
        float nrm[kRows][2];  // per group of the span (one group of 128: both equal)
#pragma unroll
        for (int r = 0; r < kRows; ++r) {  // every row's codes and norms requested together
            const bool ok = row[r] >= 0 && live_g;
            const uint8_t *gp = a.codes + (size_t)(ok ? row[r] : 0) * row_bytes + (size_t)(live_g ? g : 0) * gbytes;
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                // a span of groups of 64 may hold only one group at the end of a row
                const bool has = G == kGroup || 2 * g + (t >> 1) < a.ng;
                code[r][t] = ok && has ? load_codes4<W>(gp, sl, t) : 0u;
            }
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int gi = G == kGroup ? g : 2 * g + h;
                nrm[r][h] = ok && gi < a.ng ? __half2float(a.norms[(size_t)row[r] * a.ng + gi]) *
                                                  (G == kGroup ? kInvSqrt128 : 0.125f)
                                            : 0.0f;
            }
        }
#pragma unroll
        for (int r = 0; r < kRows; ++r) {
            if (row[r] < 0) continue;  // uniform across the warp
            float v[16];  // v[4t + j]: position 32t + 4s + j
#pragma unroll
            for (int t = 0; t < 4; ++t)
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const uint32_t q = (code[r][t] >> (W * j)) & ((1u << W) - 1u);
                    v[4 * t + j] = W == 1   ? ((q & 1u) ? l1 : l0)
                                   : W == 2 ? ((q & 2u) ? ((q & 1u) ? l3 : l2) : ((q & 1u) ? l1 : l0))
                                            : s_lv[q];
                }
#pragma unroll
            for (int hb = 1; hb < (G == kGroup ? 16 : 8); hb <<= 1)
#pragma unroll
                for (int j = 0; j < 16; ++j)
                    if (!(j & hb)) {
                        const float x = v[j], y = v[j + hb];
                        v[j] = x + y;
                        v[j + hb] = x - y;
                    }
#pragma unroll
            for (int m = 1; m < 8; m <<= 1)
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const float o = __shfl_xor_sync(0xffffffffu, v[j], m);
                    v[j] = (sl & m) ? o - v[j] : v[j] + o;
                }
            if (!live_g) continue;
            float *d = a.dst + (size_t)(i0 + r) * a.in + g * kGroup + 4 * sl;
            const int k0 = g * kGroup + 4 * sl;
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                const float n = nrm[r][t >> 1];
                const int k = k0 + 32 * t;
                if (vec && k < a.in) {
                    __stcs(reinterpret_cast<float4 *>(d + 32 * t),
                           make_float4(v[4 * t] * n, v[4 * t + 1] * n, v[4 * t + 2] * n, v[4 * t + 3] * n));
                } else {
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        if (k + j < a.in) d[32 * t + j] = v[4 * t + j] * n;
                }
            }
        }
    }
}

}  // namespace

int launch_gather_rows(const uint8_t *blob, int out, int in, int group, int bits, const float *levels,
                       const int32_t *idx, int n, float *dst, void *stream) {
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const int W = width_of(bits), ip = in_padded(in, group), ng = ip / group;
    GatherArgs a;
    a.codes = blob;
    a.norms = reinterpret_cast<const __half *>(blob + (size_t)out * ip * W / 8);
    a.idx = idx;
    a.dst = dst;
    a.status = device_status_ptr();
    a.out = out;
    a.in = in;
    a.ng = ng;
    a.n = n;
    std::copy(levels, levels + 16, a.lv);
    const long long blocks = ((long long)n + kWarps * kRows - 1) / (kWarps * kRows);
    const unsigned nb = (unsigned)blocks;
    if (group == kGroup) {
        switch (W) {
        case 1: gather_rows_kernel<1, 128><<<nb, kWarps * 32, 0, st>>>(a); break;
        case 2: gather_rows_kernel<2, 128><<<nb, kWarps * 32, 0, st>>>(a); break;
        case 3: gather_rows_kernel<3, 128><<<nb, kWarps * 32, 0, st>>>(a); break;
        default: gather_rows_kernel<4, 128><<<nb, kWarps * 32, 0, st>>>(a); break;
        }
    } else {
        switch (W) {
        case 1: gather_rows_kernel<1, 64><<<nb, kWarps * 32, 0, st>>>(a); break;
        case 2: gather_rows_kernel<2, 64><<<nb, kWarps * 32, 0, st>>>(a); break;
        case 3: gather_rows_kernel<3, 64><<<nb, kWarps * 32, 0, st>>>(a); break;
        default: gather_rows_kernel<4, 64><<<nb, kWarps * 32, 0, st>>>(a); break;
        }
    }
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return set_error(CQ_ERR_CUDA, "gather launch: %s", cudaGetErrorString(e));
    return CQ_OK;
}

}  // namespace cq
