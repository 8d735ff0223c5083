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
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <map>
#include <mutex>
#include <vector>

#include "cq_internal.h"

namespace cq {

// Status word written by this file's bounded device waits (see
// cq_device_status).
static __device__ unsigned int g_cq_device_status = 0;

unsigned int *device_status_ptr() {
    // one slot per device; threads that race on an empty slot all store the
    // same address, and the slots are atomic so that the race is defined
    static std::atomic<unsigned int *> ptr[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        cudaGetLastError();
        return nullptr;
    }
    unsigned int *q = ptr[dev].load(std::memory_order_acquire);
    if (!q) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_cq_device_status) != cudaSuccess) {
            cudaGetLastError();
            return nullptr;
        }
        q = static_cast<unsigned int *>(p);
        ptr[dev].store(q, std::memory_order_release);
    }
    return q;
}

int ensure_smem(const void *func, size_t bytes) {
    static std::mutex mu;
    static std::map<std::pair<const void *, int>, size_t> raised;  // (kernel, device) -> bytes allowed
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return set_error(CQ_ERR_CUDA, "no current CUDA device: %s", cudaGetErrorString(e));
    }
    std::lock_guard<std::mutex> lock(mu);
    size_t &have = raised[{func, dev}];
    if (have >= bytes) return CQ_OK;
    e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return set_error(CQ_ERR_SHAPE, "kernel needs %zu bytes of shared memory: %s", bytes, cudaGetErrorString(e));
    }
    have = bytes;
    return CQ_OK;
}

static void reset_counters();

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
    if (v & ~kStatusIndex) {
        reset_counters();
        return set_error(CQ_ERR_TIMEOUT, "a bounded device wait gave up (code 0x%08x)", v);
    }
    if (v) return set_error(CQ_ERR_INDEX, "a gathered row index was out of range");
    return CQ_OK;
}

namespace {

constexpr float kInvSqrt128 = 0.08838834764831845f;

// ---------------------------------------------------------- act rotate --
// Z[m][g*128 + k] = fp16((H0 q)[k]): the exact integer transform of each
// 128-group of the int8 row, rounded once to fp16.
// One warp task is (token, four consecutive groups): lane l holds the 16
// consecutive elements of group 4*quad + l/8 at positions 16*(l%8) .. +15.
// The 128-point Sylvester butterfly runs over index bits 0-3 in registers and
// over bits 4-6 across lanes l^1, l^2, l^4 (all inside one 8-lane segment).
// All distinct activations of a call go in one launch: task t belongs to the
// activation whose task range holds it. Each warp keeps two tasks' loads in
// flight.
constexpr int kMaxRot = 256;
struct RotTable {
    int n;
    long long task_before[kMaxRot + 1];
    const int8_t *x[kMaxRot];
    __half *z[kMaxRot];
    int M[kMaxRot], in[kMaxRot];
};

struct RotSlot {
    uint4 raw;     // 16 int8 values
    __half *dst;   // where this lane's 16 outputs go, or null
};

__device__ __forceinline__ RotSlot rot_load(const RotTable &r, long long task, long long total, int lane) {
    RotSlot sl;
    sl.raw = make_uint4(0, 0, 0, 0);
    sl.dst = nullptr;
    if (task >= total) return sl;
    int lo = 0, hi = r.n - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) / 2;
        if (r.task_before[mid] <= task) lo = mid;
        else hi = mid - 1;
    }
    const int in = r.in[lo], ng = (in + kGroup - 1) / kGroup, nq = (ng + 3) / 4;
    const long long local = task - r.task_before[lo];
    const long long m = local / nq;
    const int g = 4 * (int)(local - m * nq) + (lane >> 3);
    if (g >= ng) return sl;
    const int col0 = g * kGroup + 16 * (lane & 7);
    const int8_t *src = r.x[lo] + m * in + col0;
    if (col0 + 16 <= in && !(reinterpret_cast<uintptr_t>(src) & 15)) {
        sl.raw = __ldg(reinterpret_cast<const uint4 *>(src));
    } else {
        uint32_t w[4] = {0, 0, 0, 0};
#pragma unroll
        for (int i = 0; i < 16; ++i)
            if (col0 + i < in) w[i >> 2] |= (uint32_t)(uint8_t)src[i] << (8 * (i & 3));
        sl.raw = make_uint4(w[0], w[1], w[2], w[3]);
    }
    sl.dst = r.z[lo] + m * (long long)ng * kGroup + col0;
    return sl;
}

__device__ __forceinline__ void rot_finish(const RotSlot &sl, int lane) {
    const uint32_t w[4] = {sl.raw.x, sl.raw.y, sl.raw.z, sl.raw.w};
    int v[16];
#pragma unroll
    for (int k = 0; k < 16; ++k) v[k] = (int)(int8_t)(uint8_t)(w[k >> 2] >> (8 * (k & 3)));
#pragma unroll
    for (int h = 1; h < 16; h <<= 1)
#pragma unroll
        for (int k = 0; k < 16; ++k)
            if (!(k & h)) {
                const int a = v[k], b = v[k + h];
                v[k] = a + b;
                v[k + h] = a - b;
            }
#pragma unroll
    for (int s = 1; s < 8; s <<= 1)
#pragma unroll
        for (int k = 0; k < 16; ++k) {
            const int o = __shfl_xor_sync(0xffffffffu, v[k], s);
            v[k] = (lane & s) ? o - v[k] : v[k] + o;
        }
    if (!sl.dst) return;
    uint32_t h2[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const __half2 t = __halves2half2(__int2half_rn(v[2 * k]), __int2half_rn(v[2 * k + 1]));
        h2[k] = *reinterpret_cast<const uint32_t *>(&t);
    }
    uint4 *d = reinterpret_cast<uint4 *>(sl.dst);
    d[0] = make_uint4(h2[0], h2[1], h2[2], h2[3]);
    d[1] = make_uint4(h2[4], h2[5], h2[6], h2[7]);
}

__global__ void __launch_bounds__(256, 4) act_rotate_many_kernel(const __grid_constant__ RotTable r) {
    // the GEMM that follows may launch now; it waits for this grid before it
    // reads Z (griddepcontrol.wait in its TMA producer)
    asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
    const int lane = threadIdx.x & 31;
    const long long warps = (long long)gridDim.x * (blockDim.x >> 5);
    const long long total = r.task_before[r.n];
    for (long long task = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); task < total;
         task += 2 * warps) {
        const RotSlot a = rot_load(r, task, total, lane);
        const RotSlot b = rot_load(r, task + warps, total, lane);
        rot_finish(a, lane);
        rot_finish(b, lane);
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

template <int W>
__device__ __forceinline__ uint32_t code_at(const uint32_t *w, int k) {
    const int bit = k * W, word = bit >> 5, off = bit & 31;
    uint32_t v = w[word] >> off;
    if (off + W > 32) v |= w[word + 1] << (32 - off);
    return v & ((1u << W) - 1u);
}

// ------------------------------------------------- GEMM on tcgen05/TMEM --
// One CTA (4 warps) computes a 128 (weight rows) x 128 (tokens) tile of
// Y^T = W' Z^T per step of a persistent loop: for each group of 128 inputs
// the threads expand the codes of their row into W' = c[q] * n in fp16 and
// copy the rotated activations of their token, both into shared memory in the
// canonical K-major layout with 128-byte swizzle; one thread then issues
// eight tcgen05.mma.kind::f16 (M=128, N=128, K=16) accumulating in fp32 in
// tensor memory and commits them to an mbarrier. The epilogue reads the
// accumulator with tcgen05.ld (warp w owns TMEM lanes 32w..32w+31, i.e. 32
// weight rows) and stores Y[m][o] * s[m] / sqrt(128), coalesced along o.
namespace tc {

constexpr int kThreads = 128;
constexpr int kTileRows = 128;   // MMA M: weight rows
constexpr int kTileTok = 128;    // MMA N: tokens
constexpr int kSegBytes = 128 * 128;  // one 64-wide K segment of a 128-row operand
constexpr int kOpBytes = 2 * kSegBytes;  // a 128-wide K group
constexpr unsigned kWaitIters = 1u << 22;

__device__ __forceinline__ uint32_t smem_u32(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

// Byte offset of 16-byte chunk `j` (0..15, 8 fp16 each) of row `r` in a
// K-major operand with 128-byte swizzle: two 64-wide K segments of 8-row
// atoms (1024 B), chunk index XORed with the row inside its atom.
__device__ __forceinline__ uint32_t sw128_off(int r, int j) {
    return (uint32_t)((j >> 3) * kSegBytes + (r >> 3) * 1024 + (r & 7) * 128 + (((j & 7) ^ (r & 7)) << 4));
}

// UMMA shared-memory descriptor: K-major, SWIZZLE_128B, 8-row groups 1024 B apart.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
    return (uint64_t)((saddr >> 4) & 0x3FFFu) | (1ull << 16) | ((uint64_t)(1024 >> 4) << 32) | (1ull << 46) |
           (2ull << 61);
}

// Instruction descriptor, kind::f16: fp16 A and B (both K-major), fp32 D.
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N) {
    return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(smem_u32(bar)), "r"(count));
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
}

// Test for completion of the phase with parity `phase`; a thread whose phase
// is not complete is suspended in hardware for up to ~1 us (suspend-time
// hint) instead of spinning, so waiting warps leave the issue slots to the
// warps that work.
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t phase) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(phase), "r"(1000u)
        : "memory");
    return ok != 0;
}

// Non-blocking test for completion of the phase with parity `phase`.
__device__ __forceinline__ bool mbar_test(uint64_t *bar, uint32_t phase) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(phase)
        : "memory");
    return ok != 0;
}

// Bounded wait; false (and the status word set) if the phase never completed.
__device__ bool mbar_wait(uint64_t *bar, uint32_t phase, unsigned int *status, unsigned code) {
    for (unsigned i = 0; i < kWaitIters; ++i)
        if (mbar_try_wait(bar, phase)) return true;
    atomicOr(status, code);
    return false;
}

__device__ __forceinline__ void mma_f16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(
            d_tmem),
        "l"(a), "l"(b), "r"(idesc), "r"(acc));
}

// The same with A read from tensor memory (a_tmem: lane = row, column c
// holding K elements 2c, 2c+1 as fp16 low | high).
__device__ __forceinline__ uint32_t h2_bits(__half2 h) { return *reinterpret_cast<uint32_t *>(&h); }
__device__ __forceinline__ __half2 bits_h2(uint32_t u) { return *reinterpret_cast<__half2 *>(&u); }
__device__ __forceinline__ void mma_f16_tA(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc,
                                           uint32_t acc) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(
            d_tmem),
        "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc));
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&v)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,"
        "%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};\n" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
        "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]),
        "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]),
        "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
        : "memory");
}

__device__ __forceinline__ void mma_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void fence_after() { asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory"); }
__device__ __forceinline__ void fence_before() { asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory"); }

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&v)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%"
        "19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]), "=r"(v[8]),
          "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]), "=r"(v[16]),
          "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]),
          "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
}

}  // namespace tc

template <int W>
__global__ void __launch_bounds__(tc::kThreads, 1) gemm_tc_kernel(const __grid_constant__ GemmParams p) {
    using namespace tc;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    uint8_t *sA = smem;             // W' tile: 128 rows x 128 k fp16, swizzled
    uint8_t *sB = smem + kOpBytes;  // Z tile: 128 tokens x 128 k fp16, swizzled
    __shared__ __align__(8) uint64_t bar;
    __shared__ uint32_t s_tmem;
    __shared__ float lut_s[16];
    __shared__ int s_abort;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    if (warp == 0) {  // 128 fp32 accumulator columns for a 128-token tile
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(smem_u32(&s_tmem)),
                     "r"(kTileTok));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::);
    }
    if (tid == 0) {
        mbar_init(&bar, 1);
        s_abort = 0;
    }
    fence_before();
    __syncthreads();
    fence_after();
    const uint32_t tmem = s_tmem;
    const uint32_t idesc = idesc_f16(kTileRows, kTileTok);
    uint32_t phase = 0;

    for (int tile = blockIdx.x; tile < p.total_tiles && !s_abort; tile += gridDim.x) {
        int lo = 0, hi = p.n - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) / 2;
            if (p.m[mid].tiles_before <= tile) lo = mid;
            else hi = mid - 1;
        }
        const GemmMat &G = p.m[lo];
        const int local = tile - G.tiles_before;
        const int m0 = (local % G.m_tiles) * kTileTok, o0 = (local / G.m_tiles) * kTileRows;
        if (tid < 16) lut_s[tid] = p.lut[G.lut][tid];
        __syncthreads();
        const int o = o0 + tid, m = m0 + tid;  // this thread's weight row and token
        const size_t rowBytes = (size_t)G.ng * 16 * W;

        for (int g = 0; g < G.ng; ++g) {
            // ---- expand W' for row o ----
            {
                uint32_t w[4 * W];
                float nrm = 0.0f;
                if (o < G.out) {
                    const uint4 *src = reinterpret_cast<const uint4 *>(G.codes + (size_t)o * rowBytes + (size_t)g * 16 * W);
#pragma unroll
                    for (int i = 0; i < W; ++i) {
                        const uint4 v = __ldg(src + i);
                        w[4 * i] = v.x, w[4 * i + 1] = v.y, w[4 * i + 2] = v.z, w[4 * i + 3] = v.w;
                    }
                    nrm = __half2float(G.norms[(size_t)o * G.ng + g]);
                } else {
#pragma unroll
                    for (int i = 0; i < 4 * W; ++i) w[i] = 0;
                }
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    uint32_t h[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const __half lo16 = __float2half_rn(lut_s[code_at<W>(w, 8 * j + 2 * e)] * nrm);
                        const __half hi16 = __float2half_rn(lut_s[code_at<W>(w, 8 * j + 2 * e + 1)] * nrm);
                        h[e] = (uint32_t)__half_as_ushort(lo16) | ((uint32_t)__half_as_ushort(hi16) << 16);
                    }
                    *reinterpret_cast<uint4 *>(sA + sw128_off(tid, j)) = make_uint4(h[0], h[1], h[2], h[3]);
                }
            }
            // ---- copy Z for token m ----
            {
                const uint4 *zrow = reinterpret_cast<const uint4 *>(G.Z + (size_t)m * G.ng * kGroup + (size_t)g * kGroup);
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const uint4 v = m < G.M ? __ldg(zrow + j) : make_uint4(0, 0, 0, 0);
                    *reinterpret_cast<uint4 *>(sB + sw128_off(tid, j)) = v;
                }
            }
            asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
            fence_before();
            __syncthreads();
            if (tid == 0) {
                fence_after();
                const uint32_t a0 = smem_u32(sA), b0 = smem_u32(sB);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint32_t off = (kk >> 2) * kSegBytes + (kk & 3) * 32;
                    mma_f16(tmem, sw128_desc(a0 + off), sw128_desc(b0 + off), idesc, (g | kk) != 0);
                }
                mma_commit(&bar);
            }
            const bool ok = mbar_wait(&bar, phase, &g_cq_device_status, 0x47470001u);
            phase ^= 1;
            if (!ok) s_abort = 1;
            fence_after();
            __syncthreads();
            if (s_abort) break;
        }
        if (s_abort) break;
        // ---- epilogue: warp w holds rows o0 + 32w + lane ----
        {
            const int orow = o0 + 32 * warp + lane;
#pragma unroll 1
            for (int c = 0; c < kTileTok / 32; ++c) {
                uint32_t v[32];
                tmem_ld32(tmem + ((uint32_t)(32 * warp) << 16) + 32 * c, v);
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const int mm = m0 + 32 * c + i;
                    if (mm < G.M && orow < G.out)
                        G.Y[(size_t)mm * G.out + orow] = __uint_as_float(v[i]) * __fmul_rn(G.xs[mm], kInvSqrt128);
                }
            }
        }
        fence_before();
        __syncthreads();
    }
    // a timed-out MMA may still be writing: give it one more bounded wait
    if (s_abort && tid == 0) mbar_wait(&bar, phase ^ 1, &g_cq_device_status, 0x47470002u);
    fence_before();
    __syncthreads();
    if (warp == 0) {
        fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(tmem), "r"(kTileTok));
    }
}

template <int W>
int launch_tc(const GemmParams &p, int grid, size_t smem, cudaStream_t st) {
    const int rc = ensure_smem(reinterpret_cast<const void *>(gemm_tc_kernel<W>), smem);
    if (rc) return rc;
    gemm_tc_kernel<W><<<grid, tc::kThreads, smem, st>>>(p);
    return CQ_OK;
}

// ------------------------------- pipelined GEMM for inputs up to 512 wide --
// Pieces of the persistent, warp-specialised GEMM below (gemm_x8_kernel):
// its parameter block, tile schedule and bounded mbarrier waits. Every wait
// is bounded; on expiry the status word records where, all roles drain, and
// TMEM is released.
namespace tc2 {

constexpr int kMaxActs = 64;     // distinct activations (tensor maps) per launch
constexpr int kMaxNg = 4;        // groups of the inputs kept resident
constexpr int kTok = 128;        // tokens of a tile
constexpr unsigned kSpin = 1u << 22;  // polls of one barrier (each may suspend ~1 us)
constexpr unsigned kDrainSpin = 1u << 20;

struct Mat {
    const uint8_t *codes;
    const __half *norms;
    const float *xs;
    float *Y;
    int out, ng, M, lut, act, n_tiles, m_tiles, tiles_before, runs_before;
    int w;  // code width in bits (1: binary, 2: CQ2 and ternary, 3, 4) | kG64 for groups of 64
};
constexpr int kG64 = 0x100;  // Mat::w flag: groups of 64 (two norms per 128-wide span)

struct Params {
    CUtensorMap tmap[kMaxActs];  // one per distinct rotated activation
    float lut[kMaxLuts][16];
    int n, total_tiles, ng_max;
    int full_rounds, tail_T0;    // schedule (see Cursor)
    Mat m[CQ_MAX_GROUPED];
};

// Output tiles are 128 rows x 128 tokens. Tiles are numbered matrix by
// matrix (matrices that share an activation are adjacent), weight-row tile by
// weight-row tile, token tile fastest; the tiles of one (matrix, row tile)
// form a run. The schedule works in rounds: in round k, CTA b takes the whole
// run k*G + b (G CTAs), so a CTA reuses the expanded weights W' in shared
// memory across the run, and the CTAs of a round move through the token tiles
// of the same activations together, which keeps each activation tile in L2
// while the row tiles that need it read it. The runs left after the full
// rounds are split into G equal contiguous ranges of tiles.
//
// The per-matrix numbers the schedule needs live in a shared-memory table
// (parameter reads with a runtime index miss the constant cache).
struct SchedTab {
    int4 m[CQ_MAX_GROUPED];          // tiles_before, runs_before, m_tiles, n_tiles
    uint16_t ngact[CQ_MAX_GROUPED];  // ng | act << 8
};

__device__ void load_sched(const Params &p, SchedTab *tab) {
    for (int i = threadIdx.x; i < p.n; i += blockDim.x) {
        tab->m[i] = make_int4(p.m[i].tiles_before, p.m[i].runs_before, p.m[i].m_tiles, p.m[i].n_tiles);
        tab->ngact[i] = (uint16_t)(p.m[i].ng | (p.m[i].act << 8));
    }
}

// Position in this CTA's sequence of tiles: segment k = [A, B), tile T =
// token tile t of row tile n of matrix mat. Advancing inside a segment is
// plain arithmetic; only a new segment searches the table.
struct Cursor {
    int k, A, B, T, mat, n, t, mt, nt;
    const SchedTab *tab;
    int nmat, full_rounds, total_tiles, tail_T0;

    __device__ int ng() const { return tab->ngact[mat] & 0xFF; }
    __device__ int act() const { return tab->ngact[mat] >> 8; }
    __device__ int o0() const { return n * tc::kTileRows; }
    __device__ bool first() const { return T == A || t == 0; }  // run starts here
    __device__ bool last() const { return T + 1 == B || t + 1 == mt; }  // run ends here
    __device__ void set_mat(int m) {
        mat = m;
        mt = tab->m[m].z;
        nt = tab->m[m].w;
    }
    // the matrix whose range of field f (0 tiles, 1 runs) holds v
    __device__ int find(int v, int f) const {
        int lo = 0, hi = nmat - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) / 2;
            const int4 e = tab->m[mid];
            if ((f ? e.y : e.x) <= v) lo = mid;
            else hi = mid - 1;
        }
        return lo;
    }
    __device__ bool segment(int kk) {
        for (k = kk; k <= full_rounds; ++k) {
            if (k < full_rounds) {
                const int r = k * (int)gridDim.x + (int)blockIdx.x;
                set_mat(find(r, 1));
                n = r - tab->m[mat].y;
                t = 0;
                A = T = tab->m[mat].x + n * mt;
                B = A + mt;
                return true;
            }
            const long long len = total_tiles - tail_T0;
            A = tail_T0 + (int)(blockIdx.x * len / gridDim.x);
            B = tail_T0 + (int)((blockIdx.x + 1) * len / gridDim.x);
            if (A < B) {
                T = A;
                set_mat(find(T, 0));
                const int local = T - tab->m[mat].x;
                n = local / mt;
                t = local - n * mt;
                return true;
            }
        }
        return false;
    }
    __device__ bool begin(const Params &p, const SchedTab *s) {
        tab = s;
        nmat = p.n;
        full_rounds = p.full_rounds;
        total_tiles = p.total_tiles;
        tail_T0 = p.tail_T0;
        return segment(0);
    }
    __device__ bool advance() {
        if (T + 1 < B) {
            ++T;
            if (++t == mt) {
                t = 0;
                if (++n == nt) {
                    n = 0;
                    set_mat(mat + 1);
                }
            }
            return true;
        }
        return segment(k + 1);
    }
};

// Copies matrix `mi` of the parameter block into `dst` with the lanes of the
// calling warp (all 32 must call) and returns it.
__device__ __forceinline__ const Mat &warp_mat(const Params &p, int mi, Mat *dst) {
    static_assert(sizeof(Mat) % 4 == 0 && sizeof(Mat) / 4 <= 32, "descriptor copy");
    const int lane = threadIdx.x & 31;
    __syncwarp();
    if (lane < (int)(sizeof(Mat) / 4))
        reinterpret_cast<uint32_t *>(dst)[lane] = reinterpret_cast<const uint32_t *>(&p.m[mi])[lane];
    __syncwarp();
    return *dst;
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(tc::smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(tc::smem_u32(bar)), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, int x, int y, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];\n" ::"r"(
            tc::smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(tc::smem_u32(bar))
        : "memory");
}
// Bounded wait for the phase of `bar` with parity `parity`; gives up when
// another role aborted or after kSpin polls (then records `code`).
__device__ bool wait(uint64_t *bar, uint32_t parity, volatile int *abort, unsigned code) {
    if (tc::mbar_test(bar, parity)) return true;  // fast path, cheaper than a suspending poll
    for (unsigned i = 0;; ++i) {
        if (tc::mbar_try_wait(bar, parity)) return true;
        if ((i & 255u) == 255u && *abort) return false;
        if (i >= kSpin) {
            atomicOr(&g_cq_device_status, code);
            *abort = 1;
            return false;
        }
    }
}

// After an abort: waits (bounded, without regard to the abort flag) for a
// phase that asynchronous work already in flight will complete.
__device__ void drain_wait(uint64_t *bar, uint32_t parity) {
    for (unsigned i = 0; i < kDrainSpin; ++i)
        if (tc::mbar_try_wait(bar, parity)) return;
}

}  // namespace tc2

// ------------------------ pipelined GEMM on int8 activations (in <= 512) --
// The rotated-domain product, with the rotation moved onto the weights:
// H is symmetric and orthonormal, so per group
//     n * <c[q], H x> = <n * H c[q], x>,
// and the weight tile W''[o][k] = n[o] * (H c[q[o]])[k] (fp16) meets the
// int8 activations q directly: Y[m][o] = s[m] * sum_k W''[o][k] q[m][k].
// The FWHT runs once per run of token tiles on 128 weight rows, instead of
// once per token on every activation, and the activations stay int8 until
// they reach tensor memory (exactly as fp16: |q| <= 128).
//   warp 0      TMA producer: int8 X groups (128 tokens x 128 inputs, 16 KB,
//               128-byte swizzle) into four stages
//   warp 1      MMA issuer: tcgen05.mma (M = 128 tokens, N = 128 weight
//               rows, K = 16; A = X from TMEM, B = W'' from shared memory),
//               sixteen MMAs (two groups) per commit, into two 128-column
//               TMEM accumulators D[token][row]
//   warps 2-5   conversion: each lane its token row of a stage, int8 -> fp16
//               pairs, tcgen05.st into one of two 128-column X slots
//   warps 6-9   epilogue: D -> registers, Y[m][o0..o0+127] = D * s[m];
//               32 x 32 blocks pass through shared memory so that eight
//               lanes store one 128-byte row segment of Y
//   warps 10-13 expansion: W'' rows of the next run into shared memory
//               (one thread per row), one group at a time, as soon as the
//               MMAs of the previous run are done with that group
namespace tc3 {

constexpr int kThreads = 448;
constexpr int kStages = 4;                            // X stages, one group each
constexpr int kStageBytes = tc2::kTok * kGroup;       // 128 tokens x 128 inputs int8
constexpr int kWGroupBytes = tc::kTileRows * kGroup * 2;  // W'' group: two 64-wide segments
constexpr int kAcc = 0;                               // TMEM columns of the accumulators (0, 128)
constexpr int kXcol = 256;                            // TMEM columns of the X slots (256, 384)
constexpr int kStageY = 32 * 128;                     // per epilogue warp: 32 rows x 32 fp32, transposed
constexpr int kSmem = tc2::kMaxNg * kWGroupBytes + kStages * kStageBytes + 4 * kStageY + 1024;

// 16-byte shared-memory accesses by 32-bit shared address. The dynamic
// shared memory is re-aligned through an integer, after which the compiler
// no longer knows that the pointers are shared (it would emit generic
// accesses, ordered against the global stores of the epilogue).
__device__ __forceinline__ uint4 lds128(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];\n" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
    return v;
}
__device__ __forceinline__ void sts128(uint32_t addr, uint4 v) {
    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};\n" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}

// Sylvester-ordered FWHT of 64 values in registers (no normalisation).
__device__ __forceinline__ void fwht64(float (&a)[64]) {
#pragma unroll
    for (int h = 1; h < 64; h <<= 1) {
#pragma unroll
        for (int k = 0; k < 64; ++k) {
            if (!(k & h)) {
                const float x = a[k], y = a[k + h];
                a[k] = x + y;
                a[k + h] = x - y;
            }
        }
    }
}

// One W'' row of one run (this thread's weight row o), group by group into
// shared memory, K-major with 128-byte swizzle (row e of the tile, segment
// s holds inputs 64 s .. 64 s + 63). H_128 = [[H_64, H_64], [H_64, -H_64]],
// so the first 64 outputs are H_64 (v_lo + v_hi) and the last 64 are
// H_64 (v_lo - v_hi), v = c[q] the group's levels; both are scaled by
// n / sqrt(128) and rounded once to fp16. Group g is written once the MMAs of
// the previous run are done with it (w_empty[g]) and handed over through
// w_full[g]. All 32 lanes of the warp call this. False if a wait gave up.
//
// Level tables (`tab`: this warp's 32 floats). CQ2 / ternary: the pairs of
// inputs k and k+64 that the first step of H_128 combines are read at once,
// tab[v] = c[v & 3] + c[v >> 2] and tab[16 + v] = c[v & 3] - c[v >> 2] for
// the nibble v = q[k] | q[k+64] << 2; other widths: tab[q] = c[q].
//
// Groups of 64 (G64): each 64-wide half of a span is a group of its own,
// with its own norm, so segment s holds H_64 c[q] of inputs 64 s .. 64 s + 63
// scaled by n[o][2g + s] / sqrt(64) ("Cactus Quants": the group is the unit
// of the rotation and of the norm).
template <int W, bool G64>
__device__ __forceinline__ bool expand_row(const tc2::Mat &G, const float *levels, float *tab, int o, int e,
                                           uint8_t *sW, uint64_t *w_empty, uint64_t *w_full, uint32_t &pe,
                                           volatile int *abort) {
    const int lane = threadIdx.x & 31;
    __syncwarp();  // the previous run's reads of the table are done
    if (W == 2 && !G64) {
        const int v = lane & 15;
        tab[lane] = lane < 16 ? levels[v & 3] + levels[v >> 2] : levels[v & 3] - levels[v >> 2];
    } else if (lane < 16) {
        tab[lane] = levels[lane];
    }
    __syncwarp();
    const bool orow = o < G.out;
    const int ng = G.ng;
    const uint4 *src = reinterpret_cast<const uint4 *>(G.codes + (size_t)o * ng * 16 * W);
    const int nper = G64 ? 2 : 1;  // norms per 128-wide span
    const __half *nsrc = G.norms + (size_t)o * ng * nper;
    uint32_t w[4 * W];
    float nrm = 0.0f, nrm1 = 0.0f;
#pragma unroll
    for (int i = 0; i < W; ++i) {
        const uint4 v = orow ? __ldg(src + i) : make_uint4(0, 0, 0, 0);
        w[4 * i] = v.x, w[4 * i + 1] = v.y, w[4 * i + 2] = v.z, w[4 * i + 3] = v.w;
    }
    if (orow) {
        nrm = __half2float(nsrc[0]);
        if (G64) nrm1 = __half2float(nsrc[1]);
    }
    for (int g = 0; g < ng; ++g) {
        uint32_t wn[4 * W];
        float nn = 0.0f, nn1 = 0.0f;
        const bool more = orow && g + 1 < ng;
#pragma unroll
        for (int i = 0; i < W; ++i) {
            const uint4 v = more ? __ldg(src + (g + 1) * W + i) : make_uint4(0, 0, 0, 0);
            wn[4 * i] = v.x, wn[4 * i + 1] = v.y, wn[4 * i + 2] = v.z, wn[4 * i + 3] = v.w;
        }
        if (more) {
            nn = __half2float(nsrc[(g + 1) * nper]);
            if (G64) nn1 = __half2float(nsrc[(g + 1) * nper + 1]);
        }
        if (!tc2::wait(&w_empty[g], (pe >> g) & 1u, abort, 0x47480016u)) return false;
        pe ^= 1u << g;
        const float sc = nrm * kInvSqrt128;
        const uint32_t row = tc::smem_u32(sW) + g * kWGroupBytes + (e >> 3) * 1024 + (e & 7) * 128;
#pragma unroll 1
        for (int pass = 0; pass < 2; ++pass) {
            // the codes are re-read by each pass (keeps the table addresses
            // from being computed once and held across the passes)
#pragma unroll
            for (int i = 0; i < 4 * W; ++i) asm volatile("" : "+r"(w[i]));
            // a = v_lo + v_hi (pass 0) or v_lo - v_hi (pass 1); groups of
            // 64: a = v_lo (pass 0) or v_hi (pass 1)
            float a[64];
            if (G64) {
#pragma unroll
                for (int k = 0; k < 64; ++k) a[k] = tab[code_at<W>(w, 64 * pass + k)];
            } else if (W == 2) {
                const float *t = tab + 16 * pass;
#pragma unroll
                for (int m = 0; m < 4; ++m) {  // word m: codes 16m .. 16m+15; word m+4: the same + 64
                    const uint32_t ev = (w[m] & 0x33333333u) | ((w[m + 4] & 0x33333333u) << 2);
                    const uint32_t od = ((w[m] >> 2) & 0x33333333u) | (w[m + 4] & 0xCCCCCCCCu);
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        a[16 * m + 2 * j] = t[(ev >> (4 * j)) & 15u];
                        a[16 * m + 2 * j + 1] = t[(od >> (4 * j)) & 15u];
                    }
                }
            } else {
                const float sgn = pass ? -1.0f : 1.0f;
#pragma unroll
                for (int k = 0; k < 64; ++k) a[k] = fmaf(sgn, tab[code_at<W>(w, k + 64)], tab[code_at<W>(w, k)]);
            }
            fwht64(a);
            const float scp = G64 ? (pass ? nrm1 : nrm) * 0.125f : sc;  // n / sqrt(64) per half
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                uint4 c;
                c.x = tc::h2_bits(__floats2half2_rn(a[8 * j] * scp, a[8 * j + 1] * scp));
                c.y = tc::h2_bits(__floats2half2_rn(a[8 * j + 2] * scp, a[8 * j + 3] * scp));
                c.z = tc::h2_bits(__floats2half2_rn(a[8 * j + 4] * scp, a[8 * j + 5] * scp));
                c.w = tc::h2_bits(__floats2half2_rn(a[8 * j + 6] * scp, a[8 * j + 7] * scp));
                sts128(row + pass * tc::kSegBytes + ((j ^ (e & 7)) << 4), c);
            }
        }
        // generic-proxy stores, read next by the tensor cores (async proxy)
        asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
        __syncwarp();
        if (lane == 0) tc2::mbar_arrive(&w_full[g]);
#pragma unroll
        for (int i = 0; i < 4 * W; ++i) w[i] = wn[i];
        nrm = nn;
        nrm1 = nn1;
    }
    return true;
}

// int8 x 4 (one word) -> two fp16 pairs, exactly: bias to unsigned, place
// each byte under the exponent of 1024 (0x64xx = 1024 + byte), subtract 1152.
__device__ __forceinline__ void i8x4_to_h2(uint32_t v, uint32_t &lo, uint32_t &hi) {
    const uint32_t u = v ^ 0x80808080u;
    const __half2 off = __floats2half2_rn(1152.0f, 1152.0f);
    lo = tc::h2_bits(__hsub2(tc::bits_h2(__byte_perm(u, 0x64646464u, 0x5140)), off));
    hi = tc::h2_bits(__hsub2(tc::bits_h2(__byte_perm(u, 0x64646464u, 0x5342)), off));
}

}  // namespace tc3

__global__ void __launch_bounds__(tc3::kThreads, 1) gemm_x8_kernel(const __grid_constant__ tc2::Params p) {
    using namespace tc;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    uint8_t *sW = smem;                                         // kMaxNg x 32 KB: W'' groups
    uint8_t *sX = smem + tc2::kMaxNg * tc3::kWGroupBytes;       // kStages x 16 KB: int8 X
    uint8_t *sY = sX + tc3::kStages * tc3::kStageBytes;         // 4 x 4 KB: epilogue transposes
    __shared__ __align__(8) uint64_t w_full[tc2::kMaxNg], w_empty[tc2::kMaxNg], x_full[tc3::kStages],
        x_empty[tc3::kStages], t_full[2], t_empty[2], acc_full[2], acc_empty[2], drain;
    __shared__ uint32_t s_tmem;
    __shared__ volatile int s_abort;
    __shared__ float s_lv[4][32];    // per expansion warp: level tables (see expand_row)
    __shared__ tc2::Mat s_mat[14];   // per warp: the current matrix
    __shared__ tc2::SchedTab s_tab;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // The next launch on the stream may start its blocks as this grid's
    // blocks retire (its weight expansion does not depend on this grid; its
    // producer waits for it before the first activation load).
    asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
    tc2::load_sched(p, &s_tab);

    if (warp == 0) {  // two 128-column fp32 accumulators and two 128-column X slots
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(smem_u32(&s_tmem)),
                     "r"(512));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::);
    }
    if (tid == 0) {
        for (int g = 0; g < tc2::kMaxNg; ++g) {
            mbar_init(&w_full[g], 4);
            mbar_init(&w_empty[g], 1);
        }
        for (int i = 0; i < tc3::kStages; ++i) {
            mbar_init(&x_full[i], 1);
            mbar_init(&x_empty[i], 4);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&t_full[i], 4);
            mbar_init(&t_empty[i], 1);
            mbar_init(&acc_full[i], 1);
            mbar_init(&acc_empty[i], 4);
        }
        mbar_init(&drain, 1);
        s_abort = 0;
    }
    fence_before();
    __syncthreads();
    fence_after();
    const uint32_t tmem = s_tmem;

    if (warp == 0) {
        // ------------------------------------------------ TMA producer --
        if (lane == 0) {
            // X may be written by the kernel this grid overlaps (padded copies)
            asm volatile("griddepcontrol.wait;\n" ::: "memory");
            uint32_t s = 0, pe = (1u << tc3::kStages) - 1u;  // empty-phase parity of stage s in bit s
            uint32_t loaded = 0, pfull = 0;  // stages ever loaded; parity their last load completes
            tc2::Cursor c;
            for (bool more = c.begin(p, &s_tab); more; more = c.advance()) {
                const int ng = c.ng();
                const CUtensorMap *map = &p.tmap[c.act()];
                for (int g = 0; g < ng; ++g) {
                    if (!tc2::wait(&x_empty[s], (pe >> s) & 1u, &s_abort, 0x47480011u)) goto done_prod;
                    pe ^= 1u << s;
                    tc2::mbar_expect_tx(&x_full[s], tc3::kStageBytes);
                    tc2::tma_load_2d(sX + s * tc3::kStageBytes, map, g * kGroup, c.t * tc2::kTok, &x_full[s]);
                    pfull = (pfull & ~(1u << s)) | (pe & (1u << s));
                    loaded |= 1u << s;
                    s = s + 1 == tc3::kStages ? 0 : s + 1;
                }
            }
        done_prod:
            if (s_abort)  // copies still in flight land before the CTA exits
                for (int i = 0; i < tc3::kStages; ++i)
                    if (loaded >> i & 1u) tc2::drain_wait(&x_full[i], (pfull >> i) & 1u);
        }
    } else if (warp == 1) {
        // ------------------------------------------------- MMA issuer --
        if (lane == 0) {
            const uint32_t idesc = idesc_f16(tc2::kTok, kTileRows);
            // parities in bit i: X slot full (ptf), accumulator empty (pae), W'' group full (pwf)
            uint32_t sl = 0, ptf = 0u, pae = 3u, pwf = 0u;
            int acc = 0;
            bool issued = false;
            tc2::Cursor c;
            for (bool more = c.begin(p, &s_tab); more; more = c.advance(), ++acc) {
                const int ng = c.ng();
                const bool first = c.first(), last = c.last();
                const int a = acc & 1;
                if (!tc2::wait(&acc_empty[a], (pae >> a) & 1u, &s_abort, 0x47480013u)) goto done_mma;
                pae ^= 1u << a;
                fence_after();
                const uint32_t da = tmem + tc3::kAcc + a * kTileRows;
                for (int g0 = 0; g0 < ng; g0 += 2) {  // X slot sl holds groups g0 and g0+1 (if g0+1 < ng)
                    const int n2 = ng - g0 >= 2 ? 2 : 1;
                    if (!tc2::wait(&t_full[sl], (ptf >> sl) & 1u, &s_abort, 0x47480014u)) goto done_mma;
                    ptf ^= 1u << sl;
                    fence_after();  // X written with tcgen05.st by the conversion warps
                    for (int h = 0; h < n2; ++h) {
                        const int g = g0 + h;
                        if (first) {  // a new run: W'' group g is being expanded
                            if (!tc2::wait(&w_full[g], (pwf >> g) & 1u, &s_abort, 0x47480012u)) goto done_mma;
                            pwf ^= 1u << g;
                            fence_after();
                        }
                        // K step kk: inputs 16kk .. 16kk+15 of group g; X: 8 TMEM columns;
                        // W'': 32 bytes into the rows of segment kk/4
                        const uint64_t db = sw128_desc(smem_u32(sW + g * tc3::kWGroupBytes));
                        const uint32_t xa = tmem + tc3::kXcol + 128 * sl + 64 * h;
#pragma unroll
                        for (int kk = 0; kk < 8; ++kk)
                            mma_f16_tA(da, xa + 8 * kk, db + (uint64_t)((kk >> 2) * (kSegBytes >> 4) + (kk & 3) * 2),
                                       idesc, (g | kk) != 0);
                        issued = true;
                    }
                    mma_commit(&t_empty[sl]);
                    sl ^= 1u;
                    if (last)
                        for (int h = 0; h < n2; ++h) mma_commit(&w_empty[g0 + h]);
                }
                mma_commit(&acc_full[a]);
            }
        done_mma:
            if (s_abort && issued) {  // MMAs in flight finish before TMEM is freed
                mma_commit(&drain);
                tc2::drain_wait(&drain, 0);
            }
        }
    } else if (warp < 6) {
        // ------------------------------------------------- conversion --
        const int q = warp & 3;          // TMEM lane quarter of this warp
        const int r = 32 * q + lane;     // token row of the tile
        const uint32_t lane_x = tmem + tc3::kXcol + ((uint32_t)(32 * q) << 16);
        uint32_t s = 0, pf = 0u, pte = 3u, sl = 0;
        tc2::Cursor c;
        for (bool more = c.begin(p, &s_tab); more && !s_abort; more = c.advance()) {
            const int ng = c.ng();
            bool ok = true;
            for (int g0 = 0; g0 < ng && ok; g0 += 2) {
                const int n2 = ng - g0 >= 2 ? 2 : 1;
                if (!tc2::wait(&t_empty[sl], (pte >> sl) & 1u, &s_abort, 0x47480015u)) {
                    ok = false;
                    break;
                }
                pte ^= 1u << sl;
                fence_after();  // the MMAs that read this slot are complete
                for (int h = 0; h < n2; ++h) {
                    if (!tc2::wait(&x_full[s], (pf >> s) & 1u, &s_abort, 0x47480017u)) {
                        ok = false;
                        break;
                    }
                    pf ^= 1u << s;
                    // row r of the stage: eight 16-byte chunks, chunk j at j ^ (r & 7)
                    const uint32_t row = smem_u32(sX) + s * tc3::kStageBytes + r * 128;
                    uint4 v[8];
#pragma unroll
                    for (int j = 0; j < 8; ++j) v[j] = tc3::lds128(row + ((j ^ (r & 7)) << 4));
                    asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");  // before TMA refills it
                    __syncwarp();
                    if (lane == 0) tc2::mbar_arrive(&x_empty[s]);
                    s = s + 1 == tc3::kStages ? 0 : s + 1;
                    // column c of the group holds inputs 2c (low half) and 2c+1
#pragma unroll
                    for (int hf = 0; hf < 2; ++hf) {
                        uint32_t hv[32];
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const uint4 x = v[4 * hf + j];
                            tc3::i8x4_to_h2(x.x, hv[8 * j], hv[8 * j + 1]);
                            tc3::i8x4_to_h2(x.y, hv[8 * j + 2], hv[8 * j + 3]);
                            tc3::i8x4_to_h2(x.z, hv[8 * j + 4], hv[8 * j + 5]);
                            tc3::i8x4_to_h2(x.w, hv[8 * j + 6], hv[8 * j + 7]);
                        }
                        tmem_st32(lane_x + 128 * sl + 64 * h + 32 * hf, hv);
                    }
                }
                asm volatile("tcgen05.wait::st.sync.aligned;\n" ::: "memory");
                if (!ok) break;
                fence_before();
                __syncwarp();
                if (lane == 0) tc2::mbar_arrive(&t_full[sl]);
                sl ^= 1u;
            }
            if (!ok) break;
        }
        asm volatile("tcgen05.wait::st.sync.aligned;\n" ::: "memory");
    } else if (warp < 10) {
        // --------------------------------------------------- epilogue --
        const int q = warp & 3;  // TMEM lane quarter of this warp
        const int r = 32 * q + lane;
        int cur = -1;
        uint32_t pfa = 0u;  // accumulator-full parity of buffer a in bit a
        int acc = 0;
        tc2::Cursor c;
        for (bool more = c.begin(p, &s_tab); more && !s_abort; more = c.advance(), ++acc) {
            if (c.mat != cur) {
                tc2::warp_mat(p, c.mat, &s_mat[warp]);
                cur = c.mat;
            }
            const tc2::Mat &G = s_mat[warp];
            const int out = G.out, m = c.t * tc2::kTok + r, o0 = c.o0();
            const bool mrow = m < G.M;
            const float sc = mrow ? G.xs[m] : 0.0f;
            const bool vec = ((out & 3) == 0) && ((reinterpret_cast<uintptr_t>(G.Y) & 15) == 0);
            const int a = acc & 1;
            if (!tc2::wait(&acc_full[a], (pfa >> a) & 1u, &s_abort, 0x47480018u)) break;
            pfa ^= 1u << a;
            fence_after();
            const uint32_t ty = smem_u32(sY) + (warp - 6) * tc3::kStageY;  // this warp's 32 x 128-byte block
            const int grp = lane >> 3, p = lane & 7;        // store phase: row group, 16-byte unit
#pragma unroll 1
            for (int ch = 0; ch < kTileRows / 32; ++ch) {
                uint32_t v[32];
                tmem_ld32(tmem + tc3::kAcc + a * kTileRows + 32 * ch + ((uint32_t)(32 * q) << 16), v);
                const int o = o0 + 32 * ch;
                if (o >= out) continue;  // uniform across the warp
                if (vec) {
                    // row `lane` of the block, unit u at u ^ (lane & 7)
#pragma unroll
                    for (int u = 0; u < 8; ++u)
                        tc3::sts128(ty + lane * 128 + ((u ^ (lane & 7)) << 4),
                                    make_uint4(__float_as_uint(__uint_as_float(v[4 * u]) * sc),
                                               __float_as_uint(__uint_as_float(v[4 * u + 1]) * sc),
                                               __float_as_uint(__uint_as_float(v[4 * u + 2]) * sc),
                                               __float_as_uint(__uint_as_float(v[4 * u + 3]) * sc)));
                    __syncwarp();
                    // store k: lanes 8 grp .. 8 grp + 7 write row 8 grp + k, floats 4p .. 4p + 3
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        const int rr = 8 * grp + k;
                        const int mm = c.t * tc2::kTok + 32 * q + rr;
                        const uint4 f = tc3::lds128(ty + rr * 128 + ((p ^ (rr & 7)) << 4));
                        // streaming (evict-first): Y is written once and would otherwise push
                        // the activations that other row tiles still read out of L2
                        if (mm < G.M && o + 4 * p < out)
                            __stcs(reinterpret_cast<int4 *>(G.Y + (size_t)mm * out + o + 4 * p),
                                   make_int4((int)f.x, (int)f.y, (int)f.z, (int)f.w));
                    }
                    __syncwarp();
                } else if (mrow) {
                    float *yr = G.Y + (size_t)m * out;
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        if (o + i < out) __stcs(yr + o + i, __uint_as_float(v[i]) * sc);
                }
            }
            fence_before();
            __syncwarp();
            if (lane == 0) tc2::mbar_arrive(&acc_empty[a]);
        }
    } else {
        // ------------------------------------------ weight expansion --
        const int e = 32 * (warp - 10) + lane;  // weight row of the tile
        float *lv = s_lv[warp - 10];
        uint32_t pe = (1u << tc2::kMaxNg) - 1u;  // w_empty parity of group g in bit g
        tc2::Cursor c;
        for (bool more = c.begin(p, &s_tab); more && !s_abort; more = c.advance()) {
            if (!c.first()) continue;
            const tc2::Mat &G = tc2::warp_mat(p, c.mat, &s_mat[warp]);
            const float *levels = p.lut[G.lut];
            const int o = c.o0() + e;
            bool ok;
            switch (G.w) {
            case 1: ok = tc3::expand_row<1, false>(G, levels, lv, o, e, sW, w_empty, w_full, pe, &s_abort); break;
            case 2: ok = tc3::expand_row<2, false>(G, levels, lv, o, e, sW, w_empty, w_full, pe, &s_abort); break;
            case 3: ok = tc3::expand_row<3, false>(G, levels, lv, o, e, sW, w_empty, w_full, pe, &s_abort); break;
            case 4: ok = tc3::expand_row<4, false>(G, levels, lv, o, e, sW, w_empty, w_full, pe, &s_abort); break;
            case 1 | tc2::kG64: ok = tc3::expand_row<1, true>(G, levels, lv, o, e, sW, w_empty, w_full, pe, &s_abort); break;
            case 2 | tc2::kG64: ok = tc3::expand_row<2, true>(G, levels, lv, o, e, sW, w_empty, w_full, pe, &s_abort); break;
            case 3 | tc2::kG64: ok = tc3::expand_row<3, true>(G, levels, lv, o, e, sW, w_empty, w_full, pe, &s_abort); break;
            default: ok = tc3::expand_row<4, true>(G, levels, lv, o, e, sW, w_empty, w_full, pe, &s_abort); break;
            }
            if (!ok) break;
        }
    }

    fence_before();
    __syncthreads();
    if (warp == 0) {
        fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(tmem), "r"(512));
    }
}

// `pdl`: launched as a programmatic dependent of the kernel before it (one of
// this library's that triggers early; only the TMA producer then waits for
// it, so every other input must be complete when that kernel started).
int launch_x8(const tc2::Params &p, int grid, bool pdl, cudaStream_t st) {
    const int rc = ensure_smem(reinterpret_cast<const void *>(gemm_x8_kernel), tc3::kSmem);
    if (rc) return rc;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(tc3::kThreads);
    cfg.dynamicSmemBytes = tc3::kSmem;
    cfg.stream = st;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = pdl ? 1 : 0;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, gemm_x8_kernel, p);
    if (e != cudaSuccess) return set_error(CQ_ERR_CUDA, "gemm launch: %s", cudaGetErrorString(e));
    return CQ_OK;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// 2-D tensor map over int8 activations X[M][in] with rows `ld` bytes apart
// (ld a multiple of 16, X 16-byte aligned): boxes of 128 inputs x 128
// tokens, 128-byte swizzle; inputs past `in` and tokens past M read as zero.
static int make_x_map(CUtensorMap *map, const void *X, int M, int in, int ld) {
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        cudaDriverEntryPointQueryResult q;
        void *f = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess || !f) {
            cudaGetLastError();
            return set_error(CQ_ERR_CUDA, "cuTensorMapEncodeTiled is not available");
        }
        fn = reinterpret_cast<EncodeTiledFn>(f);
    }
    const cuuint64_t dims[2] = {(cuuint64_t)in, (cuuint64_t)M};
    const cuuint64_t strides[1] = {(cuuint64_t)ld};
    const cuuint32_t box[2] = {(cuuint32_t)kGroup, (cuuint32_t)tc2::kTok};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(X), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return set_error(CQ_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
    return CQ_OK;
}

// Copy of int8 activations whose rows a tensor map cannot address (row
// length not a multiple of 16 bytes, or a base that is not 16-byte aligned)
// into rows of `ld` bytes (ld = in rounded up to 16; the tail is zero).
__global__ void __launch_bounds__(256) pad_rows_kernel(const int8_t *__restrict__ X, int M, int in, int ld,
                                                       int8_t *__restrict__ Y) {
    // the GEMM that follows may launch now; it waits for this grid before it reads Y
    asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
    const long long total = (long long)M * ld;
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (long long)gridDim.x * blockDim.x) {
        const long long m = i / ld;
        const int k = (int)(i - m * ld);
        Y[i] = k < in ? X[m * in + k] : (int8_t)0;
    }
}

}  // namespace

// ------------------------------------------------------------ workspace --
// Device scratch per (device, stream, kind), grown on demand. Grow-only: an
// outgrown buffer stays allocated until the process exits, because a CUDA
// graph captured earlier may still point at it (freeing it would leave the
// graph reading freed memory). Calls on one stream are ordered, so they may
// share its buffer; calls on different streams get different buffers.
namespace {
struct WsKey {
    int dev;
    cudaStream_t st;
    int kind;
    bool operator<(const WsKey &o) const {
        if (dev != o.dev) return dev < o.dev;
        if (st != o.st) return st < o.st;
        return kind < o.kind;
    }
};
struct WsBuf {
    void *ptr = nullptr;
    size_t bytes = 0;
};
std::mutex g_ws_mutex;
std::map<WsKey, WsBuf> g_ws;
std::vector<void *> g_ws_retired;
}  // namespace

void *stream_workspace(void *stream, int kind, size_t bytes, int *err) {
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    int dev = 0;
    cudaGetDevice(&dev);
    std::lock_guard<std::mutex> lock(g_ws_mutex);
    WsBuf &w = g_ws[WsKey{dev, st, kind}];
    if (w.bytes >= bytes) return w.ptr;
    size_t want = std::max(bytes, (size_t)1 << 20);
    void *p = nullptr;
    if (cudaMalloc(&p, want) != cudaSuccess) {
        cudaGetLastError();
        *err = set_error(CQ_ERR_NOMEM, "cannot allocate %zu bytes of workspace", want);
        return nullptr;
    }
    if (w.ptr) g_ws_retired.push_back(w.ptr);
    w.ptr = p;
    w.bytes = want;
    return w.ptr;
}

constexpr int kCounterKind = 3;  // stream_workspace kind of the zeroed counters

unsigned int *stream_counters(void *stream, size_t n, int *err) {
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    int dev = 0;
    cudaGetDevice(&dev);
    std::lock_guard<std::mutex> lock(g_ws_mutex);
    WsBuf &w = g_ws[WsKey{dev, st, kCounterKind}];
    const size_t bytes = n * sizeof(unsigned int);
    if (w.bytes >= bytes) return static_cast<unsigned int *>(w.ptr);
    const size_t want = std::max(bytes, (size_t)4096);
    void *p = nullptr;
    if (cudaMalloc(&p, want) != cudaSuccess) {
        cudaGetLastError();
        *err = set_error(CQ_ERR_NOMEM, "cannot allocate %zu bytes of counters", want);
        return nullptr;
    }
    if (cudaMemsetAsync(p, 0, want, st) != cudaSuccess) {
        cudaGetLastError();
        cudaFree(p);
        *err = set_error(CQ_ERR_CUDA, "cannot clear the counters");
        return nullptr;
    }
    if (w.ptr) g_ws_retired.push_back(w.ptr);
    w.ptr = p;
    w.bytes = want;
    return static_cast<unsigned int *>(w.ptr);
}

// After a device wait gave up: every counter buffer of this device back to zero.
static void reset_counters() {
    int dev = 0;
    cudaGetDevice(&dev);
    std::lock_guard<std::mutex> lock(g_ws_mutex);
    cudaDeviceSynchronize();
    for (auto &kv : g_ws)
        if (kv.first.dev == dev && kv.first.kind == kCounterKind && kv.second.ptr)
            cudaMemset(kv.second.ptr, 0, kv.second.bytes);
    cudaDeviceSynchronize();
}

// Distinct activations of a call and their workspace (256-byte aligned
// pieces). An activation read by matrices with in > 512 is rotated once
// into Z (M * in_pad fp16, at `off`); one with in <= 512 is read as int8 by
// a tensor map, in place when its rows allow it, else from a padded copy
// (M * ld bytes, at `off`).
struct ActPlan {
    std::vector<const int8_t *> ptr;
    std::vector<size_t> off;
    std::vector<int> M, in;
    std::vector<int> wide;    // 1: rotated into Z
    std::vector<int> ld;      // narrow: row pitch of the tensor map's rows
    std::vector<int> padded;  // narrow: 1 when the map reads the padded copy
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
            const int wide = in_padded(d[i].in) / kGroup > tc2::kMaxNg;
            const bool direct = !wide && d[i].in % 16 == 0 && (reinterpret_cast<uintptr_t>(d[i].Xq) & 15) == 0;
            const int ld = (d[i].in + 15) / 16 * 16;
            pl.ptr.push_back(d[i].Xq);
            pl.M.push_back(d[i].M);
            pl.in.push_back(d[i].in);
            pl.wide.push_back(wide);
            pl.ld.push_back(wide ? 0 : ld);
            pl.padded.push_back(!wide && !direct);
            pl.off.push_back(pl.total);
            size_t bytes = 0;
            if (wide) bytes = (size_t)d[i].M * in_padded(d[i].in) * sizeof(__half);
            else if (!direct) bytes = (size_t)d[i].M * ld;
            pl.total += (bytes + 255) / 256 * 256;
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
    uint8_t *ws = nullptr;
    if (pl.total) {
        ws = static_cast<uint8_t *>(stream_workspace(st, 0, pl.total, &err));
        if (!ws) return err;
    }
    return run_gemm(d, n, pl, ws, st);
}

// Level table of one descriptor (ternary crumbs sign-extend).
static void level_table(const cq_gemm_desc &d, float lut[16]) {
    for (int j = 0; j < 16; ++j) lut[j] = 0.0f;
    if (d.bits == 5) {
        const float c = d.codebook[2];
        lut[1] = c;
        lut[2] = -2.0f * c;
        lut[3] = -c;
    } else {
        for (int j = 0; j < levels_of(d.bits); ++j) lut[j] = d.codebook[j];
    }
}

// All matrices with in <= 512, whatever their code width, in one launch of
// gemm_x8_kernel (more only when a parameter block fills up). `pdl`: the
// first launch may overlap the kernel launched just before it.
static int run_gemm_x8(const cq_gemm_desc *d, int n, const ActPlan &pl, uint8_t *ws, bool pdl, cudaStream_t st) {
    static thread_local tc2::Params p;  // large: off the stack, one per host thread
    std::vector<int> map_of(pl.ptr.size(), -1);
    int nmaps = 0, nlut = 0, tiles = 0, runs = 0, ngmax = 0;
    p.n = 0;
    auto flush = [&]() -> int {
        if (!p.n) return CQ_OK;
        p.total_tiles = tiles;
        p.ng_max = ngmax;
        // rounds of whole runs, then the rest split by tiles
        const int grid = std::min(tiles, sm_count());
        p.full_rounds = runs / grid;
        const int r0 = p.full_rounds * grid;  // first run of the tail
        p.tail_T0 = tiles;
        for (int j = 0; j < p.n; ++j)
            if (r0 < p.m[j].runs_before + p.m[j].n_tiles) {
                p.tail_T0 = p.m[j].tiles_before + (r0 - p.m[j].runs_before) * p.m[j].m_tiles;
                break;
            }
        const int rc = launch_x8(p, grid, pdl, st);
        if (rc) return rc;
        pdl = false;
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return set_error(CQ_ERR_CUDA, "gemm launch: %s", cudaGetErrorString(e));
        p.n = 0;
        nmaps = nlut = tiles = runs = ngmax = 0;
        std::fill(map_of.begin(), map_of.end(), -1);
        return CQ_OK;
    };
    // matrices that share an activation next to each other (see the schedule)
    std::vector<int> order(n);
    for (int i = 0; i < n; ++i) order[i] = i;
    std::stable_sort(order.begin(), order.end(), [&](int x, int y) { return pl.act_of[x] < pl.act_of[y]; });
    for (int i : order) {
        if (pl.act_of[i] < 0) continue;
        const int ip = in_padded(d[i].in), ng = ip / kGroup, W = width_of(d[i].bits);
        if (ng > tc2::kMaxNg) continue;
        const int a = pl.act_of[i];
        float lut[16];
        level_table(d[i], lut);
        int li = -1;
        for (int j = 0; j < nlut; ++j)
            if (std::equal(lut, lut + 16, p.lut[j])) li = j;
        const bool need_map = map_of[a] < 0;
        if (p.n == CQ_MAX_GROUPED || (need_map && nmaps == tc2::kMaxActs) || (li < 0 && nlut == kMaxLuts)) {
            const int e = flush();
            if (e) return e;
            li = -1;
        }
        if (map_of[a] < 0) {
            const void *X = pl.padded[a] ? static_cast<const void *>(ws + pl.off[a]) : pl.ptr[a];
            const int e = make_x_map(&p.tmap[nmaps], X, pl.M[a], pl.in[a], pl.ld[a]);
            if (e) return e;
            map_of[a] = nmaps++;
        }
        if (li < 0) {
            std::copy(lut, lut + 16, p.lut[nlut]);
            li = nlut++;
        }
        tc2::Mat &G = p.m[p.n];
        G.codes = d[i].blob;
        G.norms = reinterpret_cast<const __half *>(d[i].blob + (size_t)d[i].out * ip * W / 8);
        G.xs = d[i].x_scale;
        G.Y = d[i].Y;
        G.out = d[i].out;
        G.ng = ng;
        G.M = d[i].M;
        G.lut = li;
        G.act = map_of[a];
        G.w = W | (d[i].group == kGroup64 ? tc2::kG64 : 0);
        G.n_tiles = (G.out + tc::kTileRows - 1) / tc::kTileRows;
        G.m_tiles = (G.M + tc2::kTok - 1) / tc2::kTok;
        G.tiles_before = tiles;
        G.runs_before = runs;
        tiles += G.n_tiles * G.m_tiles;
        runs += G.n_tiles;
        ngmax = std::max(ngmax, ng);
        ++p.n;
    }
    return flush();
}

static int run_gemm(const cq_gemm_desc *d, int n, const ActPlan &pl, uint8_t *ws, cudaStream_t st) {
    bool any_wide = false, any_narrow = false;
    for (size_t j = 0; j < pl.ptr.size(); ++j) (pl.wide[j] ? any_wide : any_narrow) = true;
    // The first kernel may overlap the kernel before it on the stream; that
    // one's early trigger (if any) decides how much. Every read of data a
    // previous grid may have written follows griddepcontrol.wait.
    bool pdl = true;
    // every distinct activation of the wide matrices rotated in one launch
    if (any_wide) {
        static thread_local RotTable rt;  // large: off the stack, one per host thread
        rt.n = 0;
        rt.task_before[0] = 0;
        for (size_t j = 0; j < pl.ptr.size(); ++j) {
            if (!pl.wide[j]) continue;
            const int k = rt.n++;
            rt.x[k] = pl.ptr[j];
            rt.z[k] = reinterpret_cast<__half *>(ws + pl.off[j]);
            rt.M[k] = pl.M[j];
            rt.in[k] = pl.in[j];
            const int ng = in_padded(pl.in[j]) / kGroup;
            rt.task_before[k + 1] = rt.task_before[k] + (long long)pl.M[j] * ((ng + 3) / 4);
        }
        const long long tasks = rt.task_before[rt.n];
        const int grid = (int)std::min<long long>((tasks + 15) / 16, (long long)sm_count() * 4);
        act_rotate_many_kernel<<<grid, 256, 0, st>>>(rt);
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return set_error(CQ_ERR_CUDA, "act_rotate launch: %s", cudaGetErrorString(e));
        pdl = true;
    }
    // narrow activations whose rows a tensor map cannot address: padded copies
    for (size_t j = 0; j < pl.ptr.size(); ++j) {
        if (pl.wide[j] || !pl.padded[j]) continue;
        const long long bytes = (long long)pl.M[j] * pl.ld[j];
        const int grid = (int)std::min<long long>((bytes + 255) / 256, (long long)sm_count() * 8);
        pad_rows_kernel<<<grid, 256, 0, st>>>(pl.ptr[j], pl.M[j], pl.in[j], pl.ld[j],
                                              reinterpret_cast<int8_t *>(ws + pl.off[j]));
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return set_error(CQ_ERR_CUDA, "pad launch: %s", cudaGetErrorString(e));
        pdl = true;
    }
    if (any_narrow) {
        const int e2 = run_gemm_x8(d, n, pl, ws, pdl, st);
        if (e2) return e2;
    }
    if (!any_wide) return CQ_OK;
    cudaError_t e;
    for (int W = 1; W <= 4; ++W) {
        static thread_local GemmParams p;  // large: off the stack, one per host thread
        p.n = 0;
        int nlut = 0, tiles = 0;
        for (int i = 0; i < n; ++i) {
            if (pl.act_of[i] < 0 || width_of(d[i].bits) != W) continue;
            if (in_padded(d[i].in) / kGroup <= tc2::kMaxNg) continue;  // taken by the pipelined kernel
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
            G.m_tiles = (G.M + tc::kTileTok - 1) / tc::kTileTok;
            G.n_tiles = (G.out + tc::kTileRows - 1) / tc::kTileRows;
            G.tiles_before = tiles;
            tiles += G.m_tiles * G.n_tiles;
            ++p.n;
        }
        if (!p.n) continue;
        p.total_tiles = tiles;
        const size_t smem = 2 * tc::kOpBytes + 1024;
        const int grid = std::min(tiles, sm_count() * 2);
        int rc = CQ_OK;
        switch (W) {
        case 1: rc = launch_tc<1>(p, grid, smem, st); break;
        case 2: rc = launch_tc<2>(p, grid, smem, st); break;
        case 3: rc = launch_tc<3>(p, grid, smem, st); break;
        case 4: rc = launch_tc<4>(p, grid, smem, st); break;
        }
        if (rc) return rc;
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
// pressure). cq_gemm_noalloc serves them: the scratch that cq_gemm keeps in
// its grown-on-demand workspace (rotated activations of inputs wider than
// 512, padded copies of activations a tensor map cannot address) lives
// instead in the fixed array below, which every GPU that loads this library holds until the
// process exits.
static __device__ __align__(256) __half g_noalloc_scratch[CQ_GEMM_NOALLOC_MAX_ELEMS];

// Device address of the array, looked up once per device (host code cannot
// use the array's name as a device pointer). Host threads that race on an
// empty slot all store the same address; the slots are atomic so that the
// race is a defined one.
static std::atomic<void *> g_noalloc_ptr[64];

}  // namespace cq

// ------------------------------------------------------------ self-test --
namespace cq {
// One warp polls (bounded) an mbarrier phase that nothing completes, then
// takes the same give-up path as the GEMM's waits: record a code in the
// status word and return.
__global__ void wait_timeout_probe_kernel(unsigned polls) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) tc::mbar_init(&bar, 1);
    __syncwarp();
    if (threadIdx.x == 0) {
        bool done = false;
        for (unsigned i = 0; i < polls && !done; ++i) done = tc::mbar_test(&bar, 0);
        if (!done) atomicOr(&g_cq_device_status, 0x4748FFFFu);
    }
}
}  // namespace cq

extern "C" int cq_selftest_wait_timeout(void *stream) {
    cq::wait_timeout_probe_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(1u << 16);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cq::set_error(CQ_ERR_CUDA, "self-test launch: %s", cudaGetErrorString(e));
    return CQ_OK;
}

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
    void *scratch = g_noalloc_ptr[dev].load(std::memory_order_acquire);
    if (!scratch) {
        const cudaError_t e = cudaGetSymbolAddress(&scratch, g_noalloc_scratch);
        if (e != cudaSuccess || !scratch) {
            cudaGetLastError();
            return set_error(CQ_ERR_CUDA, "cq_gemm_noalloc: cannot resolve the scratch array: %s",
                             cudaGetErrorString(e));
        }
        g_noalloc_ptr[dev].store(scratch, std::memory_order_release);
    }
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    ActPlan pl;
    plan_activations(&d, 1, s, pl);
    if (pl.ptr.empty()) return CQ_OK;
    return run_gemm(&d, 1, pl, static_cast<uint8_t *>(scratch), s);
}
