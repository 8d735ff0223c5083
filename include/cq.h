/*
 * cq.h -- C ABI of libcq: Cactus Quants (CQ) encode, GEMV and GEMM over
 * CQ-packed weights on one GB300 (sm_103a), plus a minimal .cact-shaped
 * container.
 *
 * Page citations give the page title and the section:
 *   [CF]  "The .cact format" (cactuscompute.com blog): "Five regions",
 *         "Cactus Quants", "How the kernel reads it", "Versions".
 *   [NJ]  "The .cact archive and Cactus Quants" (needle.js tutorial):
 *         "Shared codebooks", "Tensor directory", "Anatomy of a CQ matrix",
 *         "2-bit", "4-bit", "3-bit", "Reconstructing one group",
 *         "Keep the quantized views".
 *   [ON]  OpenNeedle docs/reference.md: CQ quantisation, file format,
 *         rotated-domain identity, fake_quant_act, SDOT kernels.
 *   [PN]  "Porting Needle 3" (cactuscompute.com blog): "2. The tensor order
 *         is the contract".
 *
 * Conventions for every entry point
 * ---------------------------------
 *  - Return value: CQ_OK (0) or a negative CQ_ERR_* code. On error the
 *    reason is available from cq_last_error() (thread-local, valid until the
 *    next call on the same thread). No entry point aborts the process.
 *  - Device entry points take caller-owned DEVICE pointers for tensors and
 *    are asynchronous on `stream` (a cudaStream_t passed as void*; NULL is
 *    the legacy default stream). They validate arguments on the host before
 *    launching and report launch failures as CQ_ERR_CUDA. Codebooks are
 *    HOST pointers: their values are copied into the launch parameters, so
 *    the caller may free them as soon as the call returns.
 *  - A CQ blob passed to a device entry point must start on a 16-byte
 *    boundary (the kernels read codes with 16-byte loads); CQ_ERR_ARG
 *    otherwise. cudaMalloc and torch allocations satisfy this.
 *  - Matrices are row-major [out][in], stored pre-transposed as in [CF]
 *    "Five regions": an output row is contiguous along the reduction axis.
 *  - Groups: cq_encode, cq_gemv* and cq_gather_rows take group 128 (what
 *    the pages ship) or 64 (which the OpenNeedle engine also tests);
 *    cq_gemm* take group 64 only on inputs that are a multiple of 128 and
 *    at most 512; the KV cache takes group 128. Other powers of two are valid
 *    in the format and container and are rejected by the device entry points
 *    with CQ_ERR_SHAPE.
 *  - bits: 2, 3, 4 (CQ2/CQ3/CQ4, 4/8/16 levels), 5, the ternary marker of
 *    [NJ] "Shared codebooks" (3 levels {-c, 0, +c}, stored as 2-bit crumbs),
 *    or 1, binary codes ([CF] "Cactus Quants": eight per byte, two
 *    closed-form levels +-sqrt(2/pi)/sqrt(group)). The KV cache does not
 *    take binary codes.
 *  - A codebook is cq_levels(bits) floats, strictly increasing, already
 *    divided by sqrt(group) ([NJ] "Shared codebooks"). For bits = 5 it is
 *    {-c, 0, +c}.
 */
#ifndef CQ_H
#define CQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define CQ_OK 0
#define CQ_ERR_ARG (-1)     /* null pointer, bad enum, bad codebook */
#define CQ_ERR_SHAPE (-2)   /* unsupported or inconsistent sizes */
#define CQ_ERR_FORMAT (-3)  /* malformed container */
#define CQ_ERR_IO (-4)      /* file system error */
#define CQ_ERR_CUDA (-5)    /* CUDA runtime or launch failure */
#define CQ_ERR_TIMEOUT (-6) /* a bounded device wait gave up (see cq_device_status) */
#define CQ_ERR_NOMEM (-7)   /* host or device allocation failed */
#define CQ_ERR_INDEX (-8)   /* a device-side index was out of range (see cq_device_status) */

/* Activation element types for cq_gemv. */
#define CQ_X_F32 0 /* fp32 activations x[B][in] */
#define CQ_X_I8 1  /* int8 activations q[B][in] with fp32 per-token scales s[B]: x = s*q */
/* fp32 activations x[B][in], quantised per token inside the call exactly as
 * cq_act_quant_int8 does (s = absmax/127, q = clamp(rint(x/s))) and then
 * multiplied as CQ_X_I8 with those scales: the same results, bit for bit, as
 * cq_act_quant_int8 followed by a CQ_X_I8 call. x_scale is ignored. */
#define CQ_X_F32Q 2

/* Largest batch accepted by cq_gemv / cq_gemv_grouped. */
#define CQ_GEMV_MAX_BATCH 16
/* Largest number of matrices in one grouped call. */
#define CQ_MAX_GROUPED 256

/* Thread-local description of the last error on this thread ("" if none). */
const char *cq_last_error(void);

/* Library version: major*10000 + minor*100 + patch. */
int cq_version(void);

/* ------------------------------------------------------------- host -- */

/* Number of codebook levels for `bits` (2 for binary codes, bits = 1;
 * 4, 8, 16 for bits 2-4; 3 for the ternary marker 5), or -1. */
int cq_levels(int bits);

/* Packed code width in bits per weight (1, 2, 3, 4; 2 for ternary), or -1. */
int cq_code_width(int bits);

/* Analytic codebook for `bits` and `group`.
 * [NJ] "Shared codebooks" and [CF] "Cactus Quants": Lloyd-Max levels of the
 * Gaussian, divided by sqrt(group). This computes them on the host by
 * iterating the Lloyd-Max centroid / midpoint conditions on the exact
 * standard normal density to a fixed point (the pages' own files carry an
 * empirical codebook instead; any strictly increasing codebook, such as one
 * read from a container, may be passed to the other entry points).
 * For bits = 5 the levels are {-1.2240064, 0, +1.2240064}/sqrt(group), the
 * constant printed in [NJ] "Shared codebooks".
 * levels: host buffer of `cap` floats, or NULL to query the count only
 *         (the convention of needle_embed in [PN]).
 * n_levels: receives cq_levels(bits); may be NULL.
 * Errors: CQ_ERR_ARG for bad bits/group or cap too small. */
int cq_codebook_init(int bits, int group, float *levels, size_t cap,
                     size_t *n_levels);

/* Bytes of one CQ blob ([NJ] "Anatomy of a CQ matrix"):
 * out*in_pad*width/8 + out*(in_pad/group)*2, in_pad = ceil(in/group)*group.
 * Returns 0 on invalid arguments (out or in < 0, group not a power of two
 * >= 8, unknown bits). */
uint64_t cq_packed_bytes(int out, int in, int group, int bits);

/* ----------------------------------------------------------- device -- */

/* Encode W[out][in] (fp32, device) into one CQ blob (device, exactly
 * cq_packed_bytes(out,in,group,bits) bytes): codes of all rows as an
 * LSB-first bitstream per row, then fp16 norms [out][in_pad/group].
 * Per group (128 or 64) along the input axis ([CF] "Cactus Quants", [ON] CQ
 * quantisation): zero-pad, rotate by the normalised Walsh-Hadamard matrix
 * (natural Sylvester order), fp32 norm n, direction u = r / max(n, 1e-12),
 * nearest level per coordinate with ties to the smaller index (decided in
 * fp32), fp16(n) stored. Ternary crumbs: 0 -> 00, +c -> 01, -c -> 11.
 * W and blob must not overlap. A W that is 16-byte aligned with `in` a
 * multiple of the group is staged by bulk copies (the fast path; binary
 * codes at group 128 are always read per thread); any other layout is read
 * per thread, with the same results. Errors: CQ_ERR_ARG, CQ_ERR_SHAPE,
 * CQ_ERR_CUDA. */
int cq_encode(const float *W, int out, int in, int group, int bits,
              const float *codebook, uint8_t *blob, void *stream);

/* Per-token int8 quantisation of activations ([ON] fake_quant_act):
 * s[t] = absmax(X[t,:])/127 in fp32 (1 for an all-zero row),
 * Xq[t,k] = clamp(rint(X[t,k]/s[t]), -128, 127). X fp32 [M][in], Xq int8
 * [M][in], s fp32 [M], all device. Errors: CQ_ERR_ARG, CQ_ERR_CUDA. */
int cq_act_quant_int8(const float *X, int M, int in, int8_t *Xq, float *s,
                      void *stream);

/* Matrix-vector product over one CQ blob, batch 1..16:
 *   y[b][o] = sum_g n[o][g] * < c[q[o,g,:]], H x_b,g >        ([ON], [NJ])
 * which equals W_hat x_b exactly in real arithmetic: the activation is
 * rotated once per group (in-register fast Walsh-Hadamard transform) and the
 * weights are never expanded to a dense matrix ([CF] "How the kernel reads
 * it"). Every shape at group 128 runs on the tensor cores (mma.sync, fp32
 * accumulation) with the codebook levels rounded to fp16:
 *  - B <= 4 with 1-, 2- and 4-bit codes and in < 2048: one launch whose
 *    blocks rotate their own activation (the decode step);
 *  - the other B <= 4 shapes (3-bit codes, inputs of 2048 up to 128
 *    groups), and groups of 64 whose input is a multiple of 128 (up to 16384)
 *    with 1-, 2- and 4-bit codes: one launch of per-warp pipelines over
 *    (matrix, k-slice, 16-row tile) units whose blocks rotate the activation
 *    groups they need, the k-slices of a tile summed in slice order (the
 *    results do not depend on scheduling); groups of 64 that no such plan
 *    fits take a streaming kernel;
 *  - batches of 5 to 16: a rotation launch, which writes each distinct
 *    activation's MMA fragments once, and block-wide slices.
 * The last two use library-owned device buffers (grown on demand: make one
 * untimed call before capturing a CUDA graph). z enters as fp16 hi + lo
 * terms for B <= 4 and as one fp16 term for B >= 5. The remaining shapes
 * (the rest of group 64, batches of 5 to 16 with too many groups for the
 * workspace's shared-memory stage) use fp32 arithmetic.
 * x: fp32 [B][in] (x_dtype = CQ_X_F32, x_scale ignored, may be NULL),
 *    int8 [B][in] with x_scale fp32 [B] (x_dtype = CQ_X_I8), or fp32 [B][in]
 *    quantised per token inside the call (x_dtype = CQ_X_F32Q: the decode
 *    kernel quantises as it rotates, in the same launch; other shapes first
 *    quantise into a library workspace with one more launch).
 * y: fp32 [B][out], fully overwritten.
 * x, x_scale and y are device memory or page-locked host memory that the
 * device can address (cudaHostAlloc / cudaHostRegister with unified
 * addressing): the kernels then read the activation and write the result
 * across the host link themselves, with no separate copy (on Grace-Blackwell
 * over NVLink-C2C). blob is device memory.
 * Errors: CQ_ERR_ARG, CQ_ERR_SHAPE (group other than 64 or 128, B out of range),
 * CQ_ERR_CUDA. */
int cq_gemv(const uint8_t *blob, int out, int in, int group, int bits,
            const float *codebook, const void *x, int x_dtype,
            const float *x_scale, int B, float *y, void *stream);

/* One matrix of a grouped GEMV. blob is a device pointer; x, x_scale and y
 * are device pointers or device-addressable page-locked host memory (as for
 * cq_gemv); the codebook is the host array `codebook` (cq_levels(bits)
 * floats). */
typedef struct cq_gemv_desc {
    const uint8_t *blob;
    const void *x;        /* [B][in], fp32 or int8 per x_dtype */
    const float *x_scale; /* [B] for CQ_X_I8, else ignored (may be NULL) */
    float *y;             /* [B][out] */
    const float *codebook;/* host pointer */
    int out, in, group, bits, x_dtype, B;
} cq_gemv_desc;

/* Runs n (1..CQ_MAX_GROUPED) independent GEMVs in one kernel launch: the
 * decode step of a Needle-shaped model, where many small matrices would
 * otherwise each pay a launch. On the tensor-core path each thread block
 * rotates the activation of its slice of output rows itself (a few FWHTs
 * per block; [ON]: Q/K/V/gate reuse one rotated input, here within a
 * block), so the launch has no prologue and no scratch memory. Results
 * are identical to n separate cq_gemv calls up to fp32 summation order.
 * Output buffers must not overlap. Errors as cq_gemv. */
int cq_gemv_grouped(const cq_gemv_desc *descs, int n, void *stream);

/* Shared-input products: y_j = W_j x for n_mats (1..CQ_MAX_GROUPED)
 * matrices that read the same activation, such as the Q, K, V and gate
 * projections of a layer ([ON]: "Q/K/V/gate reuse one rotated input";
 * out_proj reads a different one). One launch; on the tensor-core path every
 * thread block rotates x once for all the rows it holds. blobs, outs and ys
 * are host arrays of n_mats entries (device pointers in blobs and ys, as for
 * cq_gemv); in, group, bits, codebook, x, x_dtype, x_scale and B are shared
 * and mean what they mean for cq_gemv. Results are bit-identical to
 * cq_gemv_grouped over the same matrices. Errors as cq_gemv, CQ_ERR_ARG for
 * null arrays or n_mats out of range. */
int cq_gemv_shared(const uint8_t *const *blobs, const int *outs, int n_mats,
                   int in, int group, int bits, const float *codebook,
                   const void *x, int x_dtype, const float *x_scale, int B,
                   float *const *ys, void *stream);

/* Prefill product over one CQ blob with int8 per-token activations:
 *   Y[m][o] = s[m] * sum_k W_hat[o][k] Xq[m][k]
 * computed as a dense contraction on the tensor cores, the codes expanded
 * only tile by tile on chip, tcgen05 accumulating in fp32 in tensor memory.
 * The rotation of the rotated-domain identity is applied on whichever side
 * is cheaper ("Reconstructing one group": n <c[q], H x> = <n H c[q], x>):
 *  - in <= 512: per run of token tiles, the 128 weight rows of a tile are
 *    expanded and rotated back once, W''[o][k] = fp16(n[o][g] (H c[q])[k]),
 *    and meet the int8 activations directly (exact in fp16); groups of 64
 *    are rotated back half-span by half-span with H_64 and their own norms;
 *  - in > 512: the activations are rotated exactly in integers per group
 *    (H0 Xq, |v| <= 16384), stored in fp16, and meet W'[o][k] =
 *    fp16(c[q] n[o][g]).
 * Xq int8 [M][in], x_scale fp32 [M], Y fp32 [M][out]: device.
 * The library keeps one internal device workspace, grown on demand by the
 * first call that needs more (rotated activations for in > 512; padded
 * copies of activations whose rows are not a multiple of 16 bytes or not
 * 16-byte aligned); make one untimed call before capturing a CUDA graph.
 * Errors: CQ_ERR_ARG, CQ_ERR_SHAPE, CQ_ERR_NOMEM, CQ_ERR_CUDA,
 * CQ_ERR_TIMEOUT (a pipeline wait exceeded its bound; results invalid). */
int cq_gemm(const uint8_t *blob, int out, int in, int group, int bits,
            const float *codebook, const int8_t *Xq, const float *x_scale,
            int M, float *Y, void *stream);

/* One matrix of a grouped GEMM (device pointers; host codebook). */
typedef struct cq_gemm_desc {
    const uint8_t *blob;
    const int8_t *Xq;     /* [M][in] */
    const float *x_scale; /* [M] */
    float *Y;             /* [M][out] */
    const float *codebook;/* host pointer */
    int out, in, group, bits, M;
} cq_gemm_desc;

/* n independent GEMMs in as few launches as possible: one persistent GEMM
 * launch for all matrices with in <= 512 (whatever their code width), and
 * for wider inputs one rotation launch over their distinct activations plus
 * one GEMM launch per code width. Errors as cq_gemm. */
int cq_gemm_grouped(const cq_gemm_desc *descs, int n, void *stream);

/* Largest M * in_pad accepted by cq_gemm_noalloc (fp16 elements of its
 * fixed scratch array: 4 MiB of device memory per GPU). */
#define CQ_GEMM_NOALLOC_MAX_ELEMS (2 * 1024 * 1024)

/* cq_gemm without any device allocation.
 * The pages have no counterpart: this entry point exists for callers that
 * cannot allocate device memory while they run -- an engine that reserves
 * all device memory up front and passes the library only its inputs and
 * outputs, or a thread that must not enter the CUDA allocator (cudaMalloc
 * synchronises the device and may fail under memory pressure). cq_gemm keeps
 * its scratch (rotated or padded activations) in a workspace it grows with
 * cudaMalloc; this variant keeps it in a fixed array of
 * CQ_GEMM_NOALLOC_MAX_ELEMS fp16 values compiled into the library, which every GPU that loads the library
 * holds until the process exits. Arguments, layouts and results are those of
 * cq_gemm.
 *  - Sizes: M * in_pad must not exceed CQ_GEMM_NOALLOC_MAX_ELEMS
 *    (in_pad = in rounded up to 128); larger calls fail with CQ_ERR_SHAPE
 *    before anything is launched.
 *  - The first call on a device looks up the array's device address (with
 *    that device current) and caches it; make that first call before any
 *    stream capture.
 *  - The function allocates nothing: no cudaMalloc, no cudaFree, no
 *    allocating library call.
 *  - All calls share the one array. Each call overwrites every element it
 *    uses before reading it, so nothing needs clearing, but calls whose
 *    kernels overlap on the GPU (different streams, or several host threads)
 *    race on the array: serialise them, e.g. on one stream.
 * Errors: those of cq_gemm, and CQ_ERR_SHAPE for the size limit. */
int cq_gemm_noalloc(const uint8_t *blob, int out, int in, int group, int bits,
                    const float *codebook, const int8_t *Xq,
                    const float *x_scale, int M, float *Y, void *stream);

/* Row-gather dequantisation of a CQ table: an embedding or engram table
 * stored as one blob, of which a step needs a few rows.
 *   dst[i][k] = W_hat[idx[i]][k],  k < in
 * Each group of an indexed row is rebuilt as n * H c[q] ("The .cact archive
 * and Cactus Quants", "Reconstructing one group"; [ON] "rotated-domain
 * identity"), in fp32 (levels, transform and norm scaling; the fp16 norm is
 * exact in fp32). Only the indexed rows are read.
 * blob: device, 16-byte aligned; idx: int32 [n], device; dst: fp32 [n][in],
 * device, fully overwritten. n may be 0.
 * An index outside [0, out) yields a row of zeros and marks the device
 * status word, which a following cq_device_status reports as CQ_ERR_INDEX.
 * Errors: CQ_ERR_ARG, CQ_ERR_SHAPE (group other than 64 or 128), CQ_ERR_CUDA. */
int cq_gather_rows(const uint8_t *blob, int out, int in, int group, int bits,
                   const float *codebook, const int32_t *idx, int n,
                   float *dst, void *stream);

/* ------------------------------------------------------ CQ KV cache -- */
/*
 * A key or a value cache quantised with CQ: the header's kv_bits (2, 3 or 4;
 * 8 means int8 and is not this path) names the code width, and "the same
 * path" as the weights serves it ([CF] "Five regions": kv_bits field; "How
 * the kernel reads it"; [ON]: below 8 bits the KV cache goes through the CQ
 * quantiser). One cache holds `cap` token rows; row t is the concatenation
 * of the n_kv_heads head vectors of token t (width in = n_kv_heads *
 * head_dim), encoded exactly like a weight matrix with out = cap (groups of
 * 128 along the row, zero-padded tail): codes [cap][in_pad*width/8], then
 * fp16 norms [cap][in_pad/128], cq_packed_bytes(cap, in, 128, bits) bytes.
 * A cache of one head per row (n_kv_heads = 1) is the per-head layout.
 */

/* Encodes rows[n][in] (fp32, device) into cache rows t0 .. t0+n-1 of a cache
 * of `cap` rows (device, 16-byte aligned, cq_packed_bytes(cap, in, 128, bits)
 * bytes), as cq_encode would encode those rows; other rows are untouched.
 * 0 <= t0, t0 + n <= cap; n = 0 does nothing. A ring buffer over a sliding
 * window wraps by calling twice. Errors: CQ_ERR_ARG, CQ_ERR_SHAPE,
 * CQ_ERR_CUDA. */
int cq_kv_write(uint8_t *cache, int cap, int in, int bits,
                const float *codebook, const float *rows, int t0, int n,
                void *stream);

/* Geometry shared by the sequences of one cq_kv_attend call (one layer). */
typedef struct cq_kv_geom {
    int n_q_heads;        /* 1..16, a multiple of n_kv_heads */
    int n_kv_heads;       /* >= 1 */
    int head_dim_k;       /* query/key head width; n_kv_heads*head_dim_k <= 512 */
    int head_dim_v;       /* value head width;     n_kv_heads*head_dim_v <= 512 */
    int k_bits, v_bits;   /* 2, 3, 4 or 5 (ternary) */
    const float *k_codebook, *v_codebook; /* host, cq_levels(bits) floats */
    float scale;          /* logit scale, typically 1/sqrt(head_dim_k) */
} cq_kv_geom;

/* One sequence: its two caches (cq_kv_write layout, `cap` rows each; the key
 * cache of width n_kv_heads*head_dim_k, the value cache of width
 * n_kv_heads*head_dim_v), the query q[n_q_heads][head_dim_k] and the output
 * o[n_q_heads][head_dim_v] (fp32). All device pointers. */
typedef struct cq_kv_seq {
    const uint8_t *k_cache;
    const uint8_t *v_cache;
    const float *q;
    float *o;
    int cap;
    int n_tokens;         /* rows 0 .. n_tokens-1 are attended; 0..cap */
} cq_kv_seq;

/* Decode-step attention over CQ caches for n_seqs (>= 1) sequences:
 *   o[b] = sum_t p[b][t] v_hat[t][h], p[b] = softmax_t(scale * <q[b], k_hat[t][h]>)
 * with h = b / (n_q_heads / n_kv_heads) (consecutive query heads share a
 * key/value head) and k_hat, v_hat the head slices of the dequantised cache
 * rows. Neither cache is expanded: the logits use the rotated identity
 * n <c[q], H x> with x the query placed at its head's columns of the row
 * ([ON] rotated-domain identity), and the value sum is accumulated in the
 * rotated domain, sum_t p n_t c[q_t], and rotated back once per group at the
 * end (H is its own inverse). Rows outside 0 .. n_tokens-1 are never read
 * (they may hold anything); a sequence with n_tokens = 0 gets o = 0.
 * Arithmetic: levels and the rotated query (as fp16 hi + lo terms) meet on
 * the tensor cores with fp32 accumulation; softmax in fp32; the value
 * weights p*n enter the tensor cores in fp16.
 * The library keeps an internal device workspace for the partial results of
 * long sequences (grown on demand; make one untimed call before capturing a
 * CUDA graph). The o buffers must not overlap.
 * Errors: CQ_ERR_ARG, CQ_ERR_SHAPE, CQ_ERR_NOMEM, CQ_ERR_CUDA. */
int cq_kv_attend(const cq_kv_geom *geom, const cq_kv_seq *seqs, int n_seqs,
                 void *stream);

/* Reads and clears the device-side status word (synchronises `stream`).
 * CQ_OK; CQ_ERR_TIMEOUT if a bounded wait gave up (results of that call are
 * invalid); CQ_ERR_INDEX if a gather met an index out of range (and no wait
 * gave up). */
int cq_device_status(void *stream);

/* Diagnostic without a counterpart on the pages: exercises the give-up path
 * of a bounded device wait without faulting the GPU. Launches one warp on
 * `stream` that polls, a bounded number of times, an mbarrier phase that
 * nothing completes; the wait gives up, records code 0x4748FFFF in the
 * device status word and the kernel returns. A following cq_device_status
 * then reports CQ_ERR_TIMEOUT (and clears the word); the context stays
 * usable. Errors: CQ_ERR_CUDA if the launch fails. */
int cq_selftest_wait_timeout(void *stream);

/* Diagnostic without a counterpart on the pages: sets the split GEMV's tile
 * counters of `stream` (allocated if needed; at least 1024 of them) to a
 * nonzero pattern, as a launch whose waits gave up midway could leave them.
 * While they are dirty, k-sliced products of that stream do not write their
 * sums; the cq_device_status call that reports a give-up zeroes the counters
 * again. Errors: CQ_ERR_NOMEM, CQ_ERR_CUDA. */
int cq_selftest_dirty_counters(void *stream);

/* -------------------------------------------------------- container -- */
/*
 * Own .cact-shaped container (the pages disagree on the header: 196 bytes
 * and tag 0x05E12A84 in [CF] "Five regions" / "Versions", 120 bytes and tag
 * 0x05E12A83 in [NJ] "Header"; and on dtype codes: 1..4 in [CF], [NJ], [ON]
 * against 0..3 elsewhere). Layout, all little-endian:
 *   header 64 B: u32 tag 0x42475143 ("CQGB"), u32 version = 1,
 *                u32 header_bytes = 64, u32 n_tensors, u32 cb_len = 28,
 *                u32 default group, 10 x u32 reserved (0)
 *   codebook 28 x f32: CQ2[0..3], CQ3[4..11], CQ4[12..27] ([NJ] "Shared
 *                codebooks")
 *   directory n x 44 B ([NJ] "Tensor directory", [CF] "Five regions"):
 *                u8 dtype (1 FP16, 2 FP32, 3 CQ, 4 RAW), u8 ndim (<= 4),
 *                u16 pad, u32 shape[4], u64 offset, u64 nbytes, u32 group,
 *                u32 bits
 *   blobs at absolute offsets, each 64-byte aligned; tensors are nameless
 *                and positional ([PN]).
 * The reader refuses foreign tags with a message ([CF] "Versions") and
 * checks every record before exposing any byte: offset + nbytes within the
 * file (64-bit overflow-checked), 64-byte alignment, ndim <= 4, known
 * dtype, FP16/FP32 byte counts equal to the element count, and for CQ a
 * power-of-two group and nbytes equal to cq_packed_bytes(shape[0],
 * shape[1], group, bits) ([NJ] "Header", "Anatomy of a CQ matrix").
 */

#define CQ_CACT_TAG 0x42475143u
#define CQ_CACT_VERSION 1u
#define CQ_CACT_HEADER_BYTES 64u
#define CQ_CACT_CODEBOOK_LEN 28u
#define CQ_CACT_RECORD_BYTES 44u
#define CQ_CACT_ALIGN 64u

#define CQ_DTYPE_FP16 1
#define CQ_DTYPE_FP32 2
#define CQ_DTYPE_CQ 3
#define CQ_DTYPE_RAW 4

typedef struct cq_tensor_desc {
    uint8_t dtype;     /* CQ_DTYPE_* */
    uint8_t ndim;      /* 0..4; a CQ tensor is 2-D [out][in] */
    uint32_t shape[4]; /* unused dimensions are 0 */
    uint64_t nbytes;   /* blob length */
    uint32_t group;    /* CQ group, else 0 */
    uint32_t bits;     /* CQ bits (2,3,4,5), else 0 */
    const void *data;  /* host bytes: input to the writer; for the reader a
                          pointer into the handle's copy of the file */
} cq_tensor_desc;

typedef struct cq_cact cq_cact; /* opaque reader handle */

/* Writes n tensors (host data) and the 28-float codebook to `path`,
 * atomically (temporary file, then rename). default_group goes into the
 * header. Errors: CQ_ERR_ARG (bad descriptor, CQ nbytes inconsistent),
 * CQ_ERR_IO. */
int cq_cact_write(const char *path, const cq_tensor_desc *tensors, int n,
                  const float codebook[28], uint32_t default_group);

/* Opens and validates a container; on success *h owns one host copy of the
 * file. Errors: CQ_ERR_IO, CQ_ERR_FORMAT (with a message naming the first
 * failed check), CQ_ERR_NOMEM. */
int cq_cact_open(const char *path, cq_cact **h);

/* Same checks on an in-memory image (copied; `bytes` may be freed after). */
int cq_cact_open_memory(const void *bytes, uint64_t size, cq_cact **h);

int cq_cact_count(const cq_cact *h);            /* number of tensors, or -1 */
int cq_cact_codebook(const cq_cact *h, float out[28]);
uint32_t cq_cact_default_group(const cq_cact *h);
/* Descriptor of tensor i; d->data points into the handle (valid until
 * cq_cact_close). Errors: CQ_ERR_ARG for a bad index. */
int cq_cact_tensor(const cq_cact *h, int i, cq_tensor_desc *d);
void cq_cact_close(cq_cact *h);

#ifdef __cplusplus
}
#endif
#endif /* CQ_H */
