// cq_gemm.cu -- prefill products over CQ-packed weights with int8 per-token
// activations (OpenNeedle docs/reference.md, fake_quant_act: s = absmax/127
// per token), single and grouped.
//
//   Y[m][o] = s[m]/sqrt(128) * sum_g n[o][g] * sum_k c[q[o,g,k]] * (H0 Xq[m,g,:])[k]
//
// The activation rotation H0 Xq (H0 the +-1 Sylvester matrix) is an exact
// integer transform with |v| <= 128*128, done once per token and group by
// act_rotate_kernel and stored as fp16 (exact up to 2048, relative error
// <= 2^-11 above). The contraction is dense, so it runs on tensor cores:
// code tiles are expanded in shared memory only (W'[o][k] = c[q] * n[o][g]
// in fp16), never to a dense matrix in global memory ("The .cact format",
// "How the kernel reads it"; "The .cact archive and Cactus Quants", "Keep
// the quantized views"). Products of two fp16 values are exact in fp32 and
// accumulate in fp32.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <vector>

#include "cq_internal.h"

namespace cq {

// Status word written by this file's bounded device waits (see
// cq_device_status).
static __device__ unsigned int g_cq_device_status = 0;

int read_and_clear_device_status(void *stream) {
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    unsigned int v = 0;
    cudaError_t e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return set_error(CQ_ERR_CUDA, "stream synchronise: %s", cudaGetErrorString(e));
    e = cudaMemcpyFromSymbol(&v, g_cq_device_status, sizeof(v));
    if (e != cudaSuccess) return set_error(CQ_ERR_CUDA, "status read: %s", cudaGetErrorString(e));
    const unsigned int zero = 0;
    e = cudaMemcpyToSymbol(g_cq_device_status, &zero, sizeof(zero));
    if (e != cudaSuccess) return set_error(CQ_ERR_CUDA, "status clear: %s", cudaGetErrorString(e));
    if (v) return set_error(CQ_ERR_TIMEOUT, "a bounded device wait gave up (code 0x%08x)", v);
    return CQ_OK;
}

namespace {

constexpr float kInvSqrt128 = 0.08838834764831845f;

// ---------------------------------------------------------- act rotate --
// One warp per (token, group): Z[m][g*128 + k] = fp16((H0 q)[k]).
__global__ void act_rotate_kernel(const int8_t *__restrict__ Xq, int M, int in, int ng,
                                  __half *__restrict__ Z) {
    const int lane = threadIdx.x & 31;
    const long long warps = (long long)gridDim.x * (blockDim.x >> 5);
    for (long long task = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
         task < (long long)M * ng; task += warps) {
        const long long m = task / ng;
        const int g = (int)(task - m * ng);
        int v[4];
        const int col0 = g * kGroup + 4 * lane;
        if (col0 + 3 < in && !(((uintptr_t)(Xq + m * in + col0)) & 3)) {
            const char4 c = *reinterpret_cast<const char4 *>(Xq + m * in + col0);
            v[0] = c.x;
            v[1] = c.y;
            v[2] = c.z;
            v[3] = c.w;
        } else {
#pragma unroll
            for (int i = 0; i < 4; ++i) v[i] = col0 + i < in ? (int)Xq[m * in + col0 + i] : 0;
        }
        int a0 = v[0] + v[1], a1 = v[0] - v[1], a2 = v[2] + v[3], a3 = v[2] - v[3];
        v[0] = a0 + a2;
        v[1] = a1 + a3;
        v[2] = a0 - a2;
        v[3] = a1 - a3;
#pragma unroll
        for (int s = 1; s < 32; s <<= 1)
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int o = __shfl_xor_sync(0xffffffffu, v[i], s);
                v[i] = (lane & s) ? o - v[i] : v[i] + o;
            }
        __half2 *dst = reinterpret_cast<__half2 *>(Z + m * (long long)ng * kGroup + col0);
        dst[0] = __halves2half2(__int2half_rn(v[0]), __int2half_rn(v[1]));
        dst[1] = __halves2half2(__int2half_rn(v[2]), __int2half_rn(v[3]));
    }
}

// --------------------------------------------------------- GEMM (core) --
struct GemmMat {
    const uint8_t *codes;
    const __half *norms;
    const __half *Z;      // [M][in_pad] rotated activations
    const float *xs;      // [M]
    float *Y;             // [M][out]
    int out, ng, bits, M, lut, m_tiles, n_tiles, tiles_before;
};

struct GemmParams {
    int n, total_tiles;
    float lut[kMaxLuts][16];
    GemmMat m[CQ_MAX_GROUPED];
};

constexpr int kTM = 64, kTN = 64;  // tokens x output rows per CTA tile
constexpr int kSimtThreads = 256;

template <int W>
__device__ __forceinline__ uint32_t code_at(const uint32_t *w, int k) {
    const int bit = k * W, word = bit >> 5, off = bit & 31;
    uint32_t v = w[word] >> off;
    if (off + W > 32) v |= w[word + 1] << (32 - off);
    return v & ((1u << W) - 1u);
}

// Reference-quality tile kernel on the CUDA cores with the same operand
// precision as the tensor-core path (fp16 x fp16 products, fp32 sums).
template <int W>
__global__ void __launch_bounds__(kSimtThreads) gemm_simt_kernel(const __grid_constant__ GemmParams p) {
    __shared__ __half Ws[kTN][kGroup + 2];
    __shared__ __half Zs[kTM][kGroup + 2];
    __shared__ float lut_s[16];
    const int tid = threadIdx.x;
    const int tx = tid % 16, ty = tid / 16;  // 4x4 outputs per thread
    for (int tile = blockIdx.x; tile < p.total_tiles; tile += gridDim.x) {
        int lo = 0, hi = p.n - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) / 2;
            if (p.m[mid].tiles_before <= tile) lo = mid;
            else hi = mid - 1;
        }
        const GemmMat &G = p.m[lo];
        const int local = tile - G.tiles_before;
        const int mt = local % G.m_tiles, nt = local / G.m_tiles;
        const int m0 = mt * kTM, o0 = nt * kTN;
        if (tid < 16) lut_s[tid] = p.lut[G.lut][tid];
        float acc[4][4] = {};
        const size_t rowBytes = (size_t)G.ng * 16 * W;
        for (int g = 0; g < G.ng; ++g) {
            __syncthreads();
            // expand 64 rows x 128 codes: thread -> (row, 32-code quarter)
            {
                const int r = tid / 4, qtr = tid % 4, o = o0 + r;
                uint32_t w[4 * W + 1];
                float nrm = 0.0f;
                if (o < G.out) {
                    const uint32_t *src = reinterpret_cast<const uint32_t *>(G.codes + (size_t)o * rowBytes + (size_t)g * 16 * W);
#pragma unroll
                    for (int i = 0; i < 4 * W; ++i) w[i] = src[i];
                    nrm = __half2float(G.norms[(size_t)o * G.ng + g]);
                } else {
#pragma unroll
                    for (int i = 0; i < 4 * W; ++i) w[i] = 0;
                }
                w[4 * W] = 0;
                for (int k = qtr * 32; k < qtr * 32 + 32; ++k)
                    Ws[r][k] = __float2half_rn(lut_s[code_at<W>(w, k)] * nrm);
            }
            for (int i = tid; i < kTM * kGroup; i += kSimtThreads) {
                const int r = i / kGroup, k = i % kGroup, m = m0 + r;
                Zs[r][k] = m < G.M ? G.Z[(size_t)m * G.ng * kGroup + (size_t)g * kGroup + k] : __float2half_rn(0.0f);
            }
            __syncthreads();
#pragma unroll 4
            for (int k = 0; k < kGroup; ++k) {
                float a[4], b[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) a[i] = __half2float(Zs[ty * 4 + i][k]);
#pragma unroll
                for (int j = 0; j < 4; ++j) b[j] = __half2float(Ws[tx * 4 + j][k]);
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
            }
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int m = m0 + ty * 4 + i;
            if (m >= G.M) continue;
            const float sc = __fmul_rn(G.xs[m], kInvSqrt128);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int o = o0 + tx * 4 + j;
                if (o < G.out) G.Y[(size_t)m * G.out + o] = acc[i][j] * sc;
            }
        }
    }
}

// ------------------------------------------------------------ workspace --
struct Workspace {
    void *ptr = nullptr;
    size_t bytes = 0;
};
std::vector<Workspace> g_ws;

// Device workspace of at least `bytes`, grown on demand (cudaFree of the old
// buffer synchronises the device, so no kernel still reads it).
void *workspace(size_t bytes, int *err) {
    int dev = 0;
    cudaGetDevice(&dev);
    if ((int)g_ws.size() <= dev) g_ws.resize(dev + 1);
    Workspace &w = g_ws[dev];
    if (w.bytes >= bytes) return w.ptr;
    if (w.ptr) cudaFree(w.ptr);
    w.ptr = nullptr;
    w.bytes = 0;
    size_t want = std::max(bytes, (size_t)1 << 20);
    if (cudaMalloc(&w.ptr, want) != cudaSuccess) {
        cudaGetLastError();
        *err = set_error(CQ_ERR_NOMEM, "cannot allocate %zu bytes of GEMM workspace", want);
        return nullptr;
    }
    w.bytes = want;
    return w.ptr;
}

}  // namespace

// Distinct activations of a call and where their rotations go in a
// workspace (each rotated once: M * in_pad fp16, 256-byte aligned).
struct ActPlan {
    std::vector<const int8_t *> ptr;
    std::vector<size_t> off;
    std::vector<int> M, in;
    std::vector<int> act_of;  // per descriptor, -1 when it needs no product
    size_t total = 0;
};

static void plan_activations(const cq_gemm_desc *d, int n, cudaStream_t st, ActPlan &pl) {
    pl.act_of.assign(n, -1);
    for (int i = 0; i < n; ++i) {
        if (d[i].M == 0 || d[i].out == 0) continue;
        if (d[i].in == 0) {  // empty reduction: the product is zero
            cudaMemsetAsync(d[i].Y, 0, sizeof(float) * (size_t)d[i].M * d[i].out, st);
            continue;
        }
        int a = -1;
        for (size_t j = 0; j < pl.ptr.size(); ++j)
            if (pl.ptr[j] == d[i].Xq && pl.in[j] == d[i].in && pl.M[j] == d[i].M) a = (int)j;
        if (a < 0) {
            a = (int)pl.ptr.size();
            pl.ptr.push_back(d[i].Xq);
            pl.M.push_back(d[i].M);
            pl.in.push_back(d[i].in);
            pl.off.push_back(pl.total);
            pl.total += ((size_t)d[i].M * in_padded(d[i].in) * sizeof(__half) + 255) / 256 * 256;
        }
        pl.act_of[i] = a;
    }
}

// Rotations into `ws` (at least pl.total bytes), then the products.
static int run_gemm(const cq_gemm_desc *d, int n, const ActPlan &pl, uint8_t *ws, cudaStream_t st);

int launch_gemm_grouped(const cq_gemm_desc *d, int n, void *stream) {
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    ActPlan pl;
    plan_activations(d, n, st, pl);
    if (pl.ptr.empty()) return CQ_OK;
    int err = CQ_OK;
    uint8_t *ws = static_cast<uint8_t *>(workspace(pl.total, &err));
    if (!ws) return err;
    return run_gemm(d, n, pl, ws, st);
}

static int run_gemm(const cq_gemm_desc *d, int n, const ActPlan &pl, uint8_t *ws, cudaStream_t st) {
    for (size_t j = 0; j < pl.ptr.size(); ++j) {
        const int ng = in_padded(pl.in[j]) / kGroup;
        const long long tasks = (long long)pl.M[j] * ng;
        const int grid = (int)std::min<long long>((tasks + 7) / 8, (long long)sm_count() * 16);
        act_rotate_kernel<<<grid, 256, 0, st>>>(pl.ptr[j], pl.M[j], pl.in[j], ng,
                                                reinterpret_cast<__half *>(ws + pl.off[j]));
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return set_error(CQ_ERR_CUDA, "act_rotate launch: %s", cudaGetErrorString(e));

    for (int W = 2; W <= 4; ++W) {
        static GemmParams p;
        p.n = 0;
        int nlut = 0, tiles = 0;
        for (int i = 0; i < n; ++i) {
            if (pl.act_of[i] < 0 || width_of(d[i].bits) != W) continue;
            GemmMat &G = p.m[p.n];
            const int ip = in_padded(d[i].in);
            G.codes = d[i].blob;
            G.norms = reinterpret_cast<const __half *>(d[i].blob + (size_t)d[i].out * ip * W / 8);
            G.Z = reinterpret_cast<const __half *>(ws + pl.off[pl.act_of[i]]);
            G.xs = d[i].x_scale;
            G.Y = d[i].Y;
            G.out = d[i].out;
            G.ng = ip / kGroup;
            G.bits = d[i].bits;
            G.M = d[i].M;
            float lut[16] = {0};
            if (d[i].bits == 5) {
                const float c = d[i].codebook[2];
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
            G.lut = li;
            G.m_tiles = (G.M + kTM - 1) / kTM;
            G.n_tiles = (G.out + kTN - 1) / kTN;
            G.tiles_before = tiles;
            tiles += G.m_tiles * G.n_tiles;
            ++p.n;
        }
        if (!p.n) continue;
        p.total_tiles = tiles;
        const int grid = std::min(tiles, sm_count() * 4);
        switch (W) {
        case 2: gemm_simt_kernel<2><<<grid, kSimtThreads, 0, st>>>(p); break;
        case 3: gemm_simt_kernel<3><<<grid, kSimtThreads, 0, st>>>(p); break;
        case 4: gemm_simt_kernel<4><<<grid, kSimtThreads, 0, st>>>(p); break;
        }
        e = cudaGetLastError();
        if (e != cudaSuccess) return set_error(CQ_ERR_CUDA, "gemm launch: %s", cudaGetErrorString(e));
    }
    return CQ_OK;
}

// ------------------------------------------------- allocation-free GEMM --
// Some callers cannot allocate device memory while they run: an inference
// engine that reserves all device memory up front and hands the library only
// its inputs and outputs, or a host thread that must not touch the CUDA
// allocator (cudaMalloc synchronises the device and can fail under memory
// pressure). cq_gemm_noalloc serves them: the rotated activations that
// cq_gemm keeps in its grown-on-demand workspace live instead in the fixed
// array below, which every GPU that loads this library holds until the
// process exits.
static __device__ __align__(256) __half g_noalloc_scratch[CQ_GEMM_NOALLOC_MAX_ELEMS];

// Device address of the array, looked up once per device (host code cannot
// use the array's name as a device pointer).
static void *g_noalloc_ptr[64];

}  // namespace cq

extern "C" int cq_gemm_noalloc(const uint8_t *blob, int out, int in, int group, int bits, const float *codebook,
                               const int8_t *Xq, const float *x_scale, int M, float *Y, void *stream) {
    using namespace cq;
    clear_error();
    cq_gemm_desc d;
    d.blob = blob;
    d.Xq = Xq;
    d.x_scale = x_scale;
    d.Y = Y;
    d.codebook = codebook;
    d.out = out;
    d.in = in;
    d.group = group;
    d.bits = bits;
    d.M = M;
    int st = check_gemm_args(d);
    if (st) return st;
    if (M > 0 && in > 0 && (size_t)M * in_padded(in) > (size_t)CQ_GEMM_NOALLOC_MAX_ELEMS)
        return set_error(CQ_ERR_SHAPE,
                         "cq_gemm_noalloc: M*in_pad = %lld exceeds the fixed scratch of %d fp16 elements; "
                         "use cq_gemm or split M",
                         (long long)M * in_padded(in), (int)CQ_GEMM_NOALLOC_MAX_ELEMS);
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        cudaGetLastError();
        return set_error(CQ_ERR_CUDA, "cq_gemm_noalloc: no current CUDA device");
    }
    if (!g_noalloc_ptr[dev]) {
        void *ptr = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
        if (e != cudaSuccess || !ptr) {
            cudaGetLastError();
            return set_error(CQ_ERR_CUDA, "cq_gemm_noalloc: cannot resolve the scratch array: %s",
                             cudaGetErrorString(e));
        }
        g_noalloc_ptr[dev] = ptr;
    }
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    ActPlan pl;
    plan_activations(&d, 1, s, pl);
    if (pl.ptr.empty()) return CQ_OK;
    return run_gemm(&d, 1, pl, static_cast<uint8_t *>(g_noalloc_ptr[dev]), s);
}
