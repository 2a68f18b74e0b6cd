/*
 * qm.h -- C interface of libqm: weight-only quantized linear algebra over
 * packed block formats, computed by CUDA kernels on one GB300 (sm_103a).
 *
 * Formats (a weight W is a float matrix [..., n, k]: n outputs by k inputs,
 * stored along k in blocks of codes sharing a scale):
 *
 *   QM_AFFINE  MLX affine storage ("GPTQModel wiki: MLX Apple Silicon",
 *              sections "Concepts: method, checkpoint, runtime, and tensor
 *              layout" and "Packed layouts and exact transcoding"; "Quantized
 *              inference in tinygpt's HFModel", section "Problem").
 *              codes  uint32 [..., n, k*bits/32], bits 2, 3, 4, 5, 6 or 8: one
 *                     continuous little-endian bit stream per row, code i in
 *                     bits [i*bits, (i+1)*bits) (so a 4-bit word holds codes
 *                     8j..8j+7, lowest in bits 0..3; 3-, 5- and 6-bit codes
 *                     cross words);
 *              scales [..., n, k/group_size] and
 *              biases [..., n, k/group_size], both of scale_dtype, group g
 *                     covering inputs [g*group_size, (g+1)*group_size).
 *              value = code*scale + bias, rounded once to float32.
 *   QM_Q8_0    GGUF Q8_0 ("Nx_quant (raven-ml.dev API docs)", section
 *              "Weights", Q8_0): codes uint8 [..., n, k/32*34]; per 32 values
 *              a little-endian float16 d then 32 int8 quants; value = d*q.
 *   QM_MXFP4   MXFP4 with its scales apart (same page, "Weights", Mxfp4):
 *              codes  uint8 [..., n, k/2], value 2i in byte i's low nibble and
 *                     value 2i+1 in its high nibble, each an e2m1 code (sign
 *                     bit 3 over magnitudes 0, .5, 1, 1.5, 2, 3, 4, 6);
 *              scales uint8 [..., n, k/32] e8m0: 2^(s-127), s = 255 is NaN.
 *              value = e2m1(code) * 2^(s-127) (float32: infinite past its range).
 *   QM_MXFP4_BLOCKS  MXFP4 in GGUF's blocks (same page, "Weights",
 *              Mxfp4_blocks): codes uint8 [..., n, k/32*17]; per 32 values the
 *              e8m0 scale byte, then 16 bytes, byte j holding value j of the
 *              block in its low nibble and value j+16 in its high nibble.
 *              Values as QM_MXFP4.
 *   QM_Q4_K    GGUF Q4_K (same page, "Weights", Q4_K): codes uint8
 *              [..., n, k/256*144] (k a multiple of 256); per 256 values a
 *              block of float16 d, float16 dmin, 12 bytes of eight 6-bit
 *              scales and eight 6-bit mins (one each per sub-block of 32) and
 *              128 bytes of 4-bit quants, arranged as ggml's block_q4_K;
 *              value = d*sc*q - dmin*m, products exact, rounded once at the
 *              subtraction.
 *   QM_Q6_K    GGUF Q6_K (same page, "Weights", Q6_K): codes uint8
 *              [..., n, k/256*210]; per 256 values 128 bytes of the quants'
 *              low 4 bits, 64 bytes of their high 2 bits, sixteen int8 scales
 *              (sub-blocks of 16) and a float16 d, arranged as ggml's
 *              block_q6_K; value = d*sc*(q - 32), exact.
 *
 * Every part is contiguous, row-major, on the device, with a 16-byte aligned
 * base address. The caller owns every buffer and the stream. Entry points
 * validate on the host, enqueue their kernels on `stream` and return; they
 * allocate no device memory, hold no decoded copy of a weight, and may be
 * called from several host threads. The only state kept between calls is
 * host-side launch metadata: each calling thread memoizes the launch plan and
 * tensor-map descriptors of a (weight descriptor, M, device) it has seen,
 * which depend on nothing but those (results never depend on it).
 *
 * Errors: QM_EINVAL for a bad argument, with qm_last_error() (thread-local,
 * valid until the next call on the thread) naming the part: "w", "codes",
 * "scales", "biases", "x", "y", "out", "ids", "axis", "workspace". QM_ECUDA if
 * a launch fails. A device-side wait that runs past its limit (two seconds of
 * the GPU's global timer) abandons its work and raises a device flag;
 * qm_device_status() reads it. No entry point synchronizes the stream.
 */
#ifndef QM_H_
#define QM_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* The same type as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st* qm_stream_t;

typedef enum qm_status {
    QM_OK = 0,
    QM_EINVAL = 1,   /* invalid argument: shape, dtype, format, alignment, axis */
    QM_ECUDA = 2,    /* a CUDA runtime call or kernel launch failed */
    QM_ETIMEOUT = 3, /* a device-side wait gave up; results of that work undefined */
    QM_ENOTSUP = 4   /* a valid combination this library does not implement */
} qm_status;

typedef enum qm_format {
    QM_AFFINE = 0,
    QM_Q8_0 = 1,
    QM_MXFP4 = 2,
    QM_MXFP4_BLOCKS = 3,
    QM_Q4_K = 4,
    QM_Q6_K = 5
} qm_format;
typedef enum qm_dtype { QM_F32 = 0, QM_BF16 = 1, QM_F16 = 2 } qm_dtype;
typedef enum qm_itype { QM_I32 = 0, QM_I64 = 1 } qm_itype;

#define QM_MAX_NDIM 4

/* A packed weight: its format, logical shape [..., n, k] and device parts. */
typedef struct qm_weight {
    int32_t format;      /* qm_format */
    int32_t bits;        /* QM_AFFINE: 2, 3, 4, 5, 6 or 8. QM_Q8_0: 8 or 0. QM_MXFP4(_BLOCKS),
                            QM_Q4_K: 4 or 0. QM_Q6_K: 6 or 0 */
    int32_t group_size;  /* QM_AFFINE: 32, 64 or 128. QM_Q4_K, QM_Q6_K: 256 or 0. Otherwise 32 or 0 */
    int32_t scale_dtype; /* QM_AFFINE: QM_BF16 or QM_F16. Otherwise ignored */
    int32_t ndim;        /* 2 .. QM_MAX_NDIM */
    int64_t shape[QM_MAX_NDIM]; /* logical shape; shape[ndim-1] = k, a multiple of 32 */
    const void* codes;   /* see the formats above */
    const void* scales;  /* QM_AFFINE, QM_MXFP4; must be NULL otherwise */
    const void* biases;  /* QM_AFFINE only; must be NULL otherwise */
    uint32_t flags;      /* QM_WEIGHT_* bits; 0 for none */
} qm_weight;

/* The weight's parts are not written by any work that may still be running on
 * the stream when a call that reads them is enqueued -- as with the weights of
 * a deployed model. Products may then start reading the weight before the
 * preceding kernel on the stream has finished (its activations are still read
 * only after it). Leave it clear if the kernel just before the call writes the
 * weight (for example a qm_take producing it). */
#define QM_WEIGHT_STATIC 1u

/* dequant: out [..., n, k] of out_dtype (QM_F32, QM_BF16 or QM_F16) holds
 * every value of w rounded once to out_dtype (round to nearest even,
 * subnormals kept, overflow to infinity).
 * Defined by "Nx_quant (raven-ml.dev API docs)", section "Products", dequant. */
qm_status qm_dequant(const qm_weight* w, int32_t out_dtype, void* out, qm_stream_t stream);

/* quantize_q8_0: x [rows, k] (k a multiple of 32) of x_dtype (QM_F32,
 * QM_BF16 or QM_F16, read at float32) stored as GGUF Q8_0 blocks
 * [rows, k/32*34] in `blocks` (caller-allocated, must not overlap x). Per block
 * of 32 values: a NaN anywhere gives a NaN scale (0x7E00) and quants 0; else
 * an infinity gives the scale +inf and quants 0; else d = amax / 127 at
 * float32 (amax the largest magnitude), stored at float16 rounded to nearest
 * even (past float16's largest: infinity), and quant j = round(v_j * (1 / d)),
 * halves away from zero, the reciprocal and the products at float32 -- 1 / d
 * of the float32 d, 0 where d is 0, and a product that is not finite gives 0.
 * Defined by "Nx_quant (raven-ml.dev API docs)", section "Weights",
 * val quantize_q8_0. */
qm_status qm_quantize_q8_0(const void* x, int32_t x_dtype, int64_t rows, int64_t k, void* blocks,
                           qm_stream_t stream);

/* apply: y [M, n] = x [M, k] times W^T, summed at float32 and rounded once to
 * x's dtype, for a 2-d weight [n, k]. x_dtype must be QM_BF16. M = 0 is valid
 * and launches nothing. x and y must not overlap.
 * Defined by "Nx_quant (raven-ml.dev API docs)", section "Products", apply. */
qm_status qm_apply(const qm_weight* w, const void* x, int64_t M, int32_t x_dtype, void* y,
                   qm_stream_t stream);

/* Most weights qm_apply_many takes in one call. */
#define QM_MAX_MANY 8

/* apply_many: for `count` 2-d weights ws[i] [n_i, k] (1 <= count <= QM_MAX_MANY)
 * that read the same x [M, k], ys[i] [M, n_i] receives exactly what
 * qm_apply(ws[i], x, M, x_dtype, ys[i], stream) would write, bit for bit. The
 * weights must share format, bits, group_size and k (and scale_dtype for
 * QM_AFFINE). Each ys[i] must be 16-byte aligned and overlap neither x nor
 * another output; QM_EINVAL names the offending argument. ws and ys are host
 * arrays of count entries; the pointers in them are device pointers.
 * Each product is the one "Nx_quant (raven-ml.dev API docs)", section
 * "Products", apply, defines. The pages have no multi-weight call: it is this
 * library's, so that products reading the same activations (a decode step's
 * q/k/v projections, or gate and up) cost one launch instead of several. At
 * M = 1 weights of up to 24 MB each, and at M = 2..8 MLX affine 4-bit weights
 * whose k is a multiple of 256, run as one grid; otherwise the call makes the
 * qm_apply launches one after another. */
qm_status qm_apply_many(const qm_weight* const* ws, int32_t count, const void* x, int64_t M, int32_t x_dtype,
                        void* const* ys, qm_stream_t stream);

/* take: gathers the rows (or matrices) of w at positions ids[0..n_ids) along
 * `axis` (0 <= axis <= ndim-2; the last axis is refused because a gather along
 * it would cut blocks), from the packed parts, decoding nothing. A position
 * outside [0, shape[axis]) -- negative included -- gathers zero bytes.
 * Packed outputs: out_codes / out_scales / out_biases have w's part shapes
 * with shape[axis] replaced by n_ids (pass NULL for parts the format lacks).
 * If out_dense is not NULL it also receives the gathered values decoded and
 * rounded once to out_dtype, shape [..., n_ids, ..., k] (an out-of-range
 * position decodes its zero bytes: zeros, -0. in Q6_K). Either the packed
 * outputs or out_dense may be omitted (NULL), not both.
 * Defined by "Nx_quant (raven-ml.dev API docs)", section "Products", take. */
qm_status qm_take(const qm_weight* w, int32_t axis, const void* ids, int32_t id_type,
                  int64_t n_ids, void* out_codes, void* out_scales, void* out_biases,
                  int32_t out_dtype, void* out_dense, qm_stream_t stream);

/* Bytes of device workspace qm_apply_experts needs for weight w [E, n, k]
 * and T*topk positions (a multiple of 256; 0 if T*topk = 0 or w is not a
 * valid 3-d weight). It holds the routing tables and, where the experts
 * average more than 32 positions each, the routed activation rows (T*topk*k
 * bf16) that the tensor-core path reads. */
size_t qm_apply_experts_workspace(const qm_weight* w, int64_t T, int64_t topk);

/* Bytes of device workspace qm_experts_route needs for P positions over E
 * experts (a multiple of 256; 0 only if P = 0). */
size_t qm_experts_route_workspace(int64_t P, int64_t E);

/* apply_experts: for a weight [E, n, k] and ids [T, topk], y [T, topk, n]
 * holds, at each position p = t*topk + j, the product of expert ids[p]'s
 * matrix with p's row of x, or zeros where ids[p] is outside [0, E), whatever
 * that row holds. x is [x_rows, k] bf16 with x_rows = T (row t serves all topk
 * positions of token t) or T*topk (one row per position). The positions are
 * routed (a stable sort by expert) into `workspace`, then summed in one
 * segmented product: chunks of up to 16 positions of one expert through the
 * decode kernel where experts average at most 32 positions, else the routed
 * rows gathered expert by expert into `workspace` and multiplied on the tensor
 * cores. The path follows from the shapes alone, so a row's bits depend on the
 * shapes, its row and its expert, never on the other positions' experts.
 * workspace_bytes must be at least qm_apply_experts_workspace(w, T, topk).
 * Routing keeps positions as int32: T*topk past 2^31-1 is refused (QM_EINVAL
 * naming "ids") before any device work, and so is E past 2^31-2 ("w").
 * Defined by "Nx_quant (raven-ml.dev API docs)", section "Products",
 * apply_experts. */
qm_status qm_apply_experts(const qm_weight* w, const void* ids, int32_t id_type, int64_t T,
                           int64_t topk, const void* x, int64_t x_rows, int32_t x_dtype, void* y,
                           void* workspace, size_t workspace_bytes, qm_stream_t stream);

/* qm_apply_experts without a workspace argument, for callers that cannot
 * allocate device memory themselves: a plug-in living inside a host program
 * that owns every device allocation, or a latency-critical loop that must not
 * pay cudaMalloc's implicit synchronization. The routing tables go to a 1 MiB
 * array that the library reserves on every GPU that loads it, enough for, e.g.,
 * 245,760 positions over 32 experts; a larger T*topk*E is refused with
 * QM_EINVAL naming "workspace". The first call on a device looks up that
 * array's device address, so make the first call on each device before any
 * stream capture. The address is kept for the life of the process: after a
 * cudaDeviceReset on a device this entry point must not be called there again
 * (a launch that fails drops the kept address, so the next call looks it up
 * anew). All calls share the one array: calls that may overlap on the GPU
 * (other streams, other host threads) race, so serialize them. Nothing in the
 * array needs clearing between calls. The array holds no gathered
 * activations, so this entry point never takes the tensor-core path: it runs
 * the decode product (or, for shapes that one declines, the plain per-position
 * kernel). Where qm_apply_experts takes the same path the two give the same
 * bits; where qm_apply_experts uses the tensor cores (experts averaging more
 * than 32 positions) the two agree within the product's error bound.
 * Otherwise identical to qm_apply_experts; the pages have no counterpart to
 * this entry point. */
qm_status qm_apply_experts_static(const qm_weight* w, const void* ids, int32_t id_type, int64_t T,
                                  int64_t topk, const void* x, int64_t x_rows, int32_t x_dtype,
                                  void* y, qm_stream_t stream);

/* The routing step of qm_apply_experts on its own: for P flattened ids and E
 * experts, counts[E] (positions per expert), offsets[E+1] (exclusive prefix
 * sum; offsets[E] = positions in range) and perm[P]: first the in-range
 * positions by ascending expert, ties by ascending position, then (from
 * offsets[E] on) the out-of-range positions in ascending order. All three are
 * int32 device buffers; workspace is qm_experts_route_workspace(P, E) bytes. */
qm_status qm_experts_route(const void* ids, int32_t id_type, int64_t P, int64_t E,
                           int32_t* counts, int32_t* offsets, int32_t* perm, void* workspace,
                           size_t workspace_bytes, qm_stream_t stream);

/* Exercises the failure path of the bounded device waits without a fault:
 * enqueues one warp that waits on a barrier nothing will complete, with the
 * same bounded wait the pipelines use but a limit of limit_ns (1 ns .. 10 s,
 * else QM_EINVAL naming "limit"). The wait gives up, raises the device flag
 * and the warp exits; a later qm_device_status() reports QM_ETIMEOUT and
 * clears the flag. The context stays usable. The pages have no counterpart to
 * this call: it is a check of this library's own error reporting. */
qm_status qm_check_wait_timeout(uint64_t limit_ns, qm_stream_t stream);

/* Synchronizes `stream`, then reports and clears the device flag raised by a
 * device-side wait that gave up (QM_ETIMEOUT), or QM_ECUDA for an
 * asynchronous CUDA error, or QM_OK. */
qm_status qm_device_status(qm_stream_t stream);

/* The message of the calling thread's last failed call ("" if none). */
const char* qm_last_error(void);

/* Library version: major * 10000 + minor * 100 + patch. */
int32_t qm_version(void);

#ifdef __cplusplus
}
#endif

#endif /* QM_H_ */
