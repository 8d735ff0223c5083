// cq_internal.h -- declarations shared by the translation units of libcq.
// Host code (cq_host.cpp) validates arguments and calls the launchers below;
// each launcher lives in the .cu file of its kernel.
#pragma once

#include <cstddef>
#include <cstdint>

#include "../../include/cq.h"

namespace cq {

// Record an error for cq_last_error() and return `code`.
int set_error(int code, const char *fmt, ...);
void clear_error();

constexpr int kGroup = 128;          // the group size of the GEMM, the tensor-core GEMV and the KV cache
constexpr int kGroup64 = 64;         // the other group the encoder, the fp32 GEMV and the row gather take
constexpr int kMaxLevels = 16;
constexpr int kMaxLuts = 8;          // distinct codebooks per grouped launch

inline int levels_of(int bits) {
    switch (bits) {
    case 1: return 2;
    case 2: return 4;
    case 3: return 8;
    case 4: return 16;
    case 5: return 3;
    default: return -1;
    }
}
inline int width_of(int bits) {
    switch (bits) {
    case 1: return 1;
    case 2: return 2;
    case 3: return 3;
    case 4: return 4;
    case 5: return 2;
    default: return -1;
    }
}
inline int in_padded(int in, int group = kGroup) { return (in + group - 1) / group * group; }

// Checks a host codebook: non-null, finite, strictly increasing.
int check_codebook(const float *cb, int bits);

// ------------------------------------------------------------- encode --
int launch_encode(const float *W, int out, int in, int group, int bits, const float *cb,
                  uint8_t *blob, void *stream);
// Encodes W[n][in] into explicit code and norm regions (rows of a larger
// blob: codes at `codes`, fp16 norms at `norms`).
int launch_encode_rows(const float *W, int n, int in, int group, int bits, const float *cb, uint8_t *codes,
                       uint8_t *norms, void *stream);
int launch_act_quant(const float *X, int M, int in, int8_t *Xq, float *s,
                     void *stream);

// --------------------------------------------------------------- gemv --
int launch_gemv_grouped(const cq_gemv_desc *d, int n, void *stream);
// Tensor-core GEMV for small batches (cq_gemv_fast.cu): which descriptors it
// takes, and one launch over the descriptors d[idx[0..n)].
bool gemv_fast_eligible(const cq_gemv_desc &d);
int launch_gemv_fast(const cq_gemv_desc *d, const int *idx, int n, void *stream);
// Streamed tensor-core GEMV for inputs of 16..32 spans at group 64 (one
// block per SM, one activation rotation per block and matrix): the fallback
// for groups of 64 that no split launch takes. Which descriptors, and the
// launches over d[idx[0..n)].
bool gemv_stream_eligible(const cq_gemv_desc &d);
int launch_gemv_stream(const cq_gemv_desc *d, const int *idx, int n, void *stream);
// Tensor-core GEMV for the other shapes (cq_gemv_wide.cu): wide inputs,
// 3-bit codes and batches up to 16 at group 128, and groups of 64 in whole
// 128-spans at batches up to 4 (split products for batches up to 4, sliced
// products for 5 to 16). A rotation launch into a workspace, then the
// products; which descriptors, and the launches. Groups of 64 that no split
// launch can take are returned in rejected[0..*n_rejected) (descriptor
// indices; room for n) for the streamed or the fp32 kernel.
bool gemv_wide_eligible(const cq_gemv_desc &d);
int launch_gemv_wide(const cq_gemv_desc *d, const int *idx, int n, void *stream, int *rejected, int *n_rejected);


// --------------------------------------------------------------- gemm --
int launch_gemm_grouped(const cq_gemm_desc *d, int n, void *stream);
// Argument checks of one GEMM descriptor (as cq_gemm does them).
int check_gemm_args(const cq_gemm_desc &d);

// Number of SMs of the current device (cached per device).
int sm_count();

// Raises the dynamic shared-memory limit of kernel `func` to at least
// `bytes` on the current device. The attribute belongs to the device, so it
// is tracked per (kernel, device) and set under a lock; CQ_OK or CQ_ERR_CUDA.
int ensure_smem(const void *func, size_t bytes);

// Device scratch of at least `bytes` for work queued on `stream`; `kind`
// selects an independent buffer (0: GEMM rotated or padded activations).
// Grow-only; null with *err set if allocation fails.
void *stream_workspace(void *stream, int kind, size_t bytes, int *err);
// Zero-initialised device counters (at least n) for work queued on `stream`:
// grow-only, zeroed on the stream when (re)allocated. The kernels that use
// them leave them zero; read_and_clear_device_status zeroes them again
// after a device wait gave up (an aborted launch may leave some nonzero).
// Null with *err set if allocation fails.
unsigned int *stream_counters(void *stream, size_t n, int *err);

// Device status word shared by kernels with bounded waits (defined in
// cq_gemm.cu; kernels OR a nonzero code into it when a wait gives up).
int read_and_clear_device_status(void *stream);
// Device address of that word on the current device (null if unavailable),
// for kernels of other translation units. Bit 31 marks an index out of
// range; the other bits are the codes of waits that gave up.
unsigned int *device_status_ptr();
constexpr unsigned int kStatusIndex = 0x80000000u;

// ------------------------------------------------------------- gather --
// `levels`: the 16-entry level table by code (ternary crumbs sign-extend).
int launch_gather_rows(const uint8_t *blob, int out, int in, int group, int bits, const float *levels,
                       const int32_t *idx, int n, float *dst, void *stream);

// Level by code, 16 entries (ternary crumbs read as signed 2-bit values).
void level_table(int bits, const float *codebook, float lv[16]);

// ---------------------------------------------------------- KV cache --
// lk, lv: level tables of the key and value codes (level_table).
int launch_kv_attend(const cq_kv_geom &g, const cq_kv_seq *seqs, int n, const float *lk, const float *lv,
                     void *stream);

}  // namespace cq
