// qm_api.cu -- libqm's C entry points: host-side validation and dispatch.
//
// Every check here names the part it refuses, the way the constructors and
// products of "Nx_quant (raven-ml.dev API docs)" (sections "Weights" and
// "Products") raise Invalid_argument naming the part.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdio>
#include <cstring>
#include <limits>
#include <string>

#include "qm.h"
#include "qm_internal.h"

namespace qm {

static thread_local std::string g_last_error;

void set_error(const std::string& msg) { g_last_error = msg; }

qm_status fail(qm_status st, const std::string& msg) {
    set_error(msg);
    return st;
}

qm_status cuda_fail(cudaError_t e, const char* what) {
    std::string m = std::string(what) + ": " + cudaGetErrorName(e) + " (" + cudaGetErrorString(e) + ")";
    set_error(m);
    return QM_ECUDA;
}

int dtype_size(int dt) { return dt == QM_F32 ? 4 : 2; }

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

static bool mul_ok(int64_t a, int64_t b, int64_t* out) {
    if (a < 0 || b < 0) return false;
    if (a != 0 && b > std::numeric_limits<int64_t>::max() / a) return false;
    *out = a * b;
    return true;
}

static const int kMaxDevices = 64;

int num_sms() {
    static std::atomic<int> cache[kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 148;
    int v = cache[dev].load(std::memory_order_relaxed);
    if (v == 0) {
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0)
            v = 148;
        cache[dev].store(v, std::memory_order_relaxed);
    }
    return v;
}

int max_smem_optin() {
    static std::atomic<int> cache[kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 227 * 1024;
    int v = cache[dev].load(std::memory_order_relaxed);
    if (v == 0) {
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess ||
            v <= 0)
            v = 227 * 1024;
        cache[dev].store(v, std::memory_order_relaxed);
    }
    return v;
}

qm_status check_positions(int64_t T, int64_t topk, int64_t E) {
    if (T < 0 || topk < 0) return fail(QM_EINVAL, "ids: negative shape");
    // routing keeps positions, offsets and the permutation as int32
    if (T > 0 && topk > std::numeric_limits<int32_t>::max() / T)
        return fail(QM_EINVAL, "ids: T*topk = " + std::to_string(T) + "*" + std::to_string(topk) +
                                   " positions, more than 2^31-1");
    if (E > std::numeric_limits<int32_t>::max() - 1) return fail(QM_EINVAL, "w: more than 2^31-2 experts");
    return QM_OK;
}

qm_status validate_weight(const qm_weight* w, WDesc* d) {
    if (!w) return fail(QM_EINVAL, "w: NULL weight descriptor");
    if (w->format < QM_AFFINE || w->format > QM_Q6_K)
        return fail(QM_EINVAL, "w: unknown format " + std::to_string(w->format));
    if (w->ndim < 2 || w->ndim > QM_MAX_NDIM)
        return fail(QM_EINVAL, "w: ndim must be 2.." + std::to_string(QM_MAX_NDIM));
    d->fmt = w->format;
    d->ndim = w->ndim;
    int64_t rows = 1;
    for (int i = 0; i < w->ndim; ++i) {
        if (w->shape[i] < 0) return fail(QM_EINVAL, "w: negative shape[" + std::to_string(i) + "]");
        d->shape[i] = w->shape[i];
        if (i < w->ndim - 1 && !mul_ok(rows, w->shape[i], &rows))
            return fail(QM_EINVAL, "w: shape too large");
    }
    d->rows = rows;
    d->n = w->shape[w->ndim - 2];
    d->k = w->shape[w->ndim - 1];
    const int64_t k = d->k;
    if (k % 32 != 0) return fail(QM_EINVAL, "codes: k = " + std::to_string(k) + " is not a multiple of 32");

    if (w->format == QM_AFFINE) {
        if (w->bits != 2 && w->bits != 3 && w->bits != 4 && w->bits != 5 && w->bits != 6 && w->bits != 8)
            return fail(QM_EINVAL, "w: affine bits must be 2, 3, 4, 5, 6 or 8, got " + std::to_string(w->bits));
        if (w->group_size != 32 && w->group_size != 64 && w->group_size != 128)
            return fail(QM_EINVAL, "w: affine group_size must be 32, 64 or 128, got " +
                                       std::to_string(w->group_size));
        if (k % w->group_size != 0)
            return fail(QM_EINVAL, "scales: k is not a multiple of group_size");
        if (w->scale_dtype != QM_BF16 && w->scale_dtype != QM_F16)
            return fail(QM_EINVAL, "scales: affine scale_dtype must be QM_BF16 or QM_F16");
        d->bits = w->bits;
        d->gs = w->group_size;
        d->sdt = w->scale_dtype;
        d->code_row_bytes = k * w->bits / 8;
        d->scale_row_bytes = d->bias_row_bytes = (k / w->group_size) * 2;
    } else if (w->format == QM_Q8_0) {
        if (w->bits != 0 && w->bits != 8) return fail(QM_EINVAL, "w: Q8_0 bits must be 8 (or 0)");
        if (w->group_size != 0 && w->group_size != 32)
            return fail(QM_EINVAL, "w: Q8_0 group_size must be 32 (or 0)");
        if (w->scales) return fail(QM_EINVAL, "scales: Q8_0 keeps its scales in its blocks; pass NULL");
        if (w->biases) return fail(QM_EINVAL, "biases: Q8_0 has no biases; pass NULL");
        d->bits = 8;
        d->gs = 32;
        d->code_row_bytes = k / 32 * 34;
    } else if (w->format == QM_Q4_K || w->format == QM_Q6_K) {
        const bool q4 = w->format == QM_Q4_K;
        if (w->bits != 0 && w->bits != (q4 ? 4 : 6))
            return fail(QM_EINVAL, std::string("w: ") + (q4 ? "Q4_K bits must be 4 (or 0)" : "Q6_K bits must be 6 (or 0)"));
        if (w->group_size != 0 && w->group_size != 256)
            return fail(QM_EINVAL, "w: K-quant group_size must be 256 (or 0)");
        if (k % 256 != 0)
            return fail(QM_EINVAL, "codes: k = " + std::to_string(k) + " is not a multiple of 256 (K-quant blocks)");
        if (w->scales) return fail(QM_EINVAL, "scales: K-quant blocks hold their scales; pass NULL");
        if (w->biases) return fail(QM_EINVAL, "biases: K-quant blocks hold their mins; pass NULL");
        d->bits = q4 ? 4 : 6;
        d->gs = 256;
        d->code_row_bytes = k / 256 * (q4 ? 144 : 210);
    } else if (w->format == QM_MXFP4_BLOCKS) {
        if (w->bits != 0 && w->bits != 4) return fail(QM_EINVAL, "w: MXFP4 bits must be 4 (or 0)");
        if (w->group_size != 0 && w->group_size != 32)
            return fail(QM_EINVAL, "w: MXFP4 group_size must be 32 (or 0)");
        if (w->scales) return fail(QM_EINVAL, "scales: MXFP4 blocks keep their scales in the blocks; pass NULL");
        if (w->biases) return fail(QM_EINVAL, "biases: MXFP4 has no biases; pass NULL");
        d->bits = 4;
        d->gs = 32;
        d->code_row_bytes = k / 32 * 17;
    } else {
        if (w->bits != 0 && w->bits != 4) return fail(QM_EINVAL, "w: MXFP4 bits must be 4 (or 0)");
        if (w->group_size != 0 && w->group_size != 32)
            return fail(QM_EINVAL, "w: MXFP4 group_size must be 32 (or 0)");
        if (w->biases) return fail(QM_EINVAL, "biases: MXFP4 has no biases; pass NULL");
        d->bits = 4;
        d->gs = 32;
        d->code_row_bytes = k / 2;
        d->scale_row_bytes = k / 32;
    }
    int64_t tot = 0;
    if (!mul_ok(rows, d->code_row_bytes, &tot)) return fail(QM_EINVAL, "codes: size overflows");
    const bool empty = (rows == 0 || k == 0);
    d->codes = static_cast<const uint8_t*>(w->codes);
    d->scales = static_cast<const uint8_t*>(w->scales);
    d->biases = static_cast<const uint8_t*>(w->biases);
    if (w->flags & ~QM_WEIGHT_STATIC) return fail(QM_EINVAL, "w: unknown flags");
    d->is_static = (w->flags & QM_WEIGHT_STATIC) != 0;
    if (!empty) {
        if (!w->codes) return fail(QM_EINVAL, "codes: NULL");
        if (!aligned16(w->codes)) return fail(QM_EINVAL, "codes: base address must be 16-byte aligned");
        if (d->scale_row_bytes) {
            if (!w->scales) return fail(QM_EINVAL, "scales: NULL");
            if (!aligned16(w->scales)) return fail(QM_EINVAL, "scales: base address must be 16-byte aligned");
        }
        if (d->bias_row_bytes) {
            if (!w->biases) return fail(QM_EINVAL, "biases: NULL");
            if (!aligned16(w->biases)) return fail(QM_EINVAL, "biases: base address must be 16-byte aligned");
        }
    }
    return QM_OK;
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*,
                                   CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                   CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_tiled() {
    static std::atomic<EncodeTiledFn> fn{nullptr};
    EncodeTiledFn f = fn.load(std::memory_order_acquire);
    if (!f) {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess || !ptr)
            return nullptr;
        f = reinterpret_cast<EncodeTiledFn>(ptr);
        fn.store(f, std::memory_order_release);
    }
    return f;
}

bool make_tmap_2d(void* map, const void* base, uint64_t inner_bytes, uint64_t rows, uint64_t row_stride,
                  uint32_t box_inner, uint32_t box_rows, bool swizzle128, int elem_bytes) {
    EncodeTiledFn f = encode_tiled();
    if (!f) return false;
    if (elem_bytes != 1 && elem_bytes != 2) return false;
    const cuuint64_t dims[2] = {inner_bytes / elem_bytes, rows};
    const cuuint64_t strides[1] = {row_stride};
    const cuuint32_t box[2] = {box_inner / static_cast<uint32_t>(elem_bytes), box_rows};
    const cuuint32_t estr[2] = {1, 1};
    const CUtensorMapDataType dt = elem_bytes == 2 ? CU_TENSOR_MAP_DATA_TYPE_UINT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8;
    CUresult r = f(static_cast<CUtensorMap*>(map), dt, 2, const_cast<void*>(base), dims,
                   strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

static qm_status check_launch(cudaError_t e, const char* what) {
    if (e != cudaSuccess) return cuda_fail(e, what);
    return QM_OK;
}

}  // namespace qm

using namespace qm;

extern "C" {

const char* qm_last_error(void) { return g_last_error.c_str(); }

int32_t qm_version(void) { return 100; }

qm_status qm_dequant(const qm_weight* w, int32_t out_dtype, void* out, qm_stream_t stream) {
    set_error("");
    WDesc d;
    qm_status s = validate_weight(w, &d);
    if (s != QM_OK) return s;
    if (out_dtype != QM_F32 && out_dtype != QM_BF16 && out_dtype != QM_F16)
        return fail(QM_EINVAL, "out: dtype must be QM_F32, QM_BF16 or QM_F16");
    if (d.rows == 0 || d.k == 0) return QM_OK;
    if (!out) return fail(QM_EINVAL, "out: NULL");
    if (!aligned16(out)) return fail(QM_EINVAL, "out: base address must be 16-byte aligned");
    return check_launch(launch_dequant(d, out_dtype, out, reinterpret_cast<cudaStream_t>(stream)),
                        "dequant launch");
}

qm_status qm_quantize_q8_0(const void* x, int32_t x_dtype, int64_t rows, int64_t k, void* blocks,
                           qm_stream_t stream) {
    set_error("");
    if (x_dtype != QM_F32 && x_dtype != QM_BF16 && x_dtype != QM_F16)
        return fail(QM_EINVAL, "x: dtype must be QM_F32, QM_BF16 or QM_F16");
    if (rows < 0 || k < 0) return fail(QM_EINVAL, "x: negative shape");
    if (k % 32 != 0) return fail(QM_EINVAL, "x: k = " + std::to_string(k) + " is not a multiple of 32");
    int64_t n = 0;
    if (!mul_ok(rows, k, &n)) return fail(QM_EINVAL, "x: shape too large");
    if (n == 0) return QM_OK;
    if (!x) return fail(QM_EINVAL, "x: NULL");
    if (!aligned16(x)) return fail(QM_EINVAL, "x: base address must be 16-byte aligned");
    if (!blocks) return fail(QM_EINVAL, "out: NULL");
    if (!aligned16(blocks)) return fail(QM_EINVAL, "out: base address must be 16-byte aligned");
    const char* xb = static_cast<const char*>(x);
    const char* ob = static_cast<const char*>(blocks);
    if (xb < ob + n / 32 * 34 && ob < xb + n * dtype_size(x_dtype)) return fail(QM_EINVAL, "out: overlaps x");
    return check_launch(launch_quantize_q8_0(x, x_dtype, rows, k, static_cast<uint8_t*>(blocks),
                                             reinterpret_cast<cudaStream_t>(stream)),
                        "quantize launch");
}

static bool small_weight(const WDesc& d) {
    return d.n * d.code_row_bytes + d.n * (d.scale_row_bytes + d.bias_row_bytes) <= (int64_t(24) << 20);
}

// One token: the register kernel for weights up to 24 MB (a dependent chain of
// such products is latency-bound); larger weights stream through the
// tensor-map pipeline, which keeps more bytes in flight.
static bool one_token_register_path(const WDesc& d) {
    return gemv1_supported(d) && (small_weight(d) || !gemv_supported(d, 1));
}

// 2..8 tokens of affine 4-bit: weight tiles in registers on mma.sync (one
// token keeps the register FFMA kernel: 3.4 against 4.1 us per small layer).
// Weights of every size: an lm_head-sized weight alone streams faster through
// the tensor-map pipeline (32 against 50 us in a chain of them), but after the
// small layers of a decode step this kernel's CTAs start early and read ahead
// (M = 8 step 0.402 against 0.426 ms).
static bool few_token_register_path(const WDesc& d, int64_t M) {
    return M >= 2 && M <= 8 && gemvr_supported(d, M);
}

// The launches of a validated product (M >= 1, n >= 1, k >= 1).
static qm_status apply_launch(const WDesc& d, const void* x, int64_t M, void* y, cudaStream_t st) {
    if (M == 1 && one_token_register_path(d)) return check_launch(launch_gemv1(d, x, y, st), "gemv launch");
    if (few_token_register_path(d, M)) {
        void* ys[1] = {y};
        return check_launch(launch_gemvr_many(&d, 1, x, M, ys, st), "gemv launch");
    }
    if (M <= 16 && gemv_supported(d, M)) return launch_gemv(d, x, M, y, st);
    if (gemm_supported(d, M)) return launch_gemm(d, x, M, y, st);
    return check_launch(launch_apply_simple(d, x, M, y, st), "apply launch");
}

qm_status qm_apply(const qm_weight* w, const void* x, int64_t M, int32_t x_dtype, void* y,
                   qm_stream_t stream) {
    set_error("");
    WDesc d;
    qm_status s = validate_weight(w, &d);
    if (s != QM_OK) return s;
    if (d.ndim != 2) return fail(QM_ENOTSUP, "w: apply takes a 2-d weight [n, k]");
    if (M < 0) return fail(QM_EINVAL, "x: negative row count M");
    if (x_dtype != QM_BF16) return fail(QM_ENOTSUP, "x: apply takes bfloat16 activations");
    if (M == 0 || d.n == 0) return QM_OK;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (!y) return fail(QM_EINVAL, "y: NULL");
    if (!aligned16(y)) return fail(QM_EINVAL, "y: base address must be 16-byte aligned");
    if (d.k == 0) {  // an empty sum
        return check_launch(cudaMemsetAsync(y, 0, static_cast<size_t>(M * d.n * 2), st),
                            "apply memset");
    }
    if (!x) return fail(QM_EINVAL, "x: NULL");
    if (!aligned16(x)) return fail(QM_EINVAL, "x: base address must be 16-byte aligned");
    const char* xb = static_cast<const char*>(x);
    const char* yb = static_cast<const char*>(y);
    if (xb < yb + M * d.n * 2 && yb < xb + M * d.k * 2) return fail(QM_EINVAL, "y: overlaps x");
    return apply_launch(d, x, M, y, st);
}

qm_status qm_apply_many(const qm_weight* const* ws, int32_t count, const void* x, int64_t M, int32_t x_dtype,
                        void* const* ys, qm_stream_t stream) {
    set_error("");
    if (count < 1 || count > QM_MAX_MANY) return fail(QM_EINVAL, "count: must be 1 .. QM_MAX_MANY");
    if (!ws) return fail(QM_EINVAL, "ws: NULL");
    if (!ys) return fail(QM_EINVAL, "ys: NULL");
    WDesc d[QM_MAX_MANY];
    for (int i = 0; i < count; ++i) {
        qm_status s = validate_weight(ws[i], &d[i]);
        if (s != QM_OK) return fail(s, "ws[" + std::to_string(i) + "]: " + qm_last_error());
        if (d[i].ndim != 2) return fail(QM_ENOTSUP, "ws[" + std::to_string(i) + "]: apply takes a 2-d weight [n, k]");
        if (d[i].fmt != d[0].fmt || d[i].bits != d[0].bits || d[i].gs != d[0].gs ||
            (d[i].fmt == QM_AFFINE && d[i].sdt != d[0].sdt))
            return fail(QM_EINVAL, "ws[" + std::to_string(i) + "]: format, bits, group_size or scale_dtype differs from ws[0]");
        if (d[i].k != d[0].k) return fail(QM_EINVAL, "ws[" + std::to_string(i) + "]: k differs from ws[0]");
    }
    if (M < 0) return fail(QM_EINVAL, "x: negative row count M");
    if (x_dtype != QM_BF16) return fail(QM_ENOTSUP, "x: apply takes bfloat16 activations");
    const int64_t k = d[0].k;
    for (int i = 0; i < count; ++i) {
        if (M == 0 || d[i].n == 0) continue;
        const std::string name = "ys[" + std::to_string(i) + "]";
        if (!ys[i]) return fail(QM_EINVAL, name + ": NULL");
        if (!aligned16(ys[i])) return fail(QM_EINVAL, name + ": base address must be 16-byte aligned");
        const char* yb = static_cast<const char*>(ys[i]);
        if (k > 0) {
            if (!x) return fail(QM_EINVAL, "x: NULL");
            const char* xb = static_cast<const char*>(x);
            if (xb < yb + M * d[i].n * 2 && yb < xb + M * k * 2) return fail(QM_EINVAL, name + ": overlaps x");
        }
        for (int j = 0; j < i; ++j) {
            if (d[j].n == 0) continue;
            const char* ob = static_cast<const char*>(ys[j]);
            if (ob < yb + M * d[i].n * 2 && yb < ob + M * d[j].n * 2)
                return fail(QM_EINVAL, name + ": overlaps ys[" + std::to_string(j) + "]");
        }
    }
    if (M == 0) return QM_OK;
    if (k > 0 && !aligned16(x)) return fail(QM_EINVAL, "x: base address must be 16-byte aligned");
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    // one grid where every weight takes the one-token register kernel on its own
    WDesc live[QM_MAX_MANY];
    void* live_y[QM_MAX_MANY];
    int nlive = 0;
    bool fused = M == 1 && k > 0, fused_few = k > 0;
    for (int i = 0; i < count; ++i) {
        if (d[i].n == 0) continue;
        live[nlive] = d[i];
        live_y[nlive++] = ys[i];
        fused = fused && one_token_register_path(d[i]);
        fused_few = fused_few && few_token_register_path(d[i], M);
    }
    if (nlive == 0) return QM_OK;
    if (fused && gemv1_many_supported(live, nlive))
        return check_launch(launch_gemv1_many(live, nlive, x, live_y, st), "gemv launch");
    if (fused_few && gemvr_many_supported(live, nlive, M))
        return check_launch(launch_gemvr_many(live, nlive, x, M, live_y, st), "gemv launch");
    for (int i = 0; i < nlive; ++i) {
        qm_status s;
        if (k == 0)
            s = check_launch(cudaMemsetAsync(live_y[i], 0, static_cast<size_t>(M * live[i].n * 2), st), "apply memset");
        else
            s = apply_launch(live[i], x, M, live_y[i], st);
        if (s != QM_OK) return s;
    }
    return QM_OK;
}

qm_status qm_take(const qm_weight* w, int32_t axis, const void* ids, int32_t id_type,
                  int64_t n_ids, void* out_codes, void* out_scales, void* out_biases,
                  int32_t out_dtype, void* out_dense, qm_stream_t stream) {
    set_error("");
    WDesc d;
    qm_status s = validate_weight(w, &d);
    if (s != QM_OK) return s;
    if (axis < 0) axis += d.ndim;
    if (axis < 0 || axis >= d.ndim) return fail(QM_EINVAL, "axis: not an axis of w");
    if (axis == d.ndim - 1)
        return fail(QM_EINVAL, "axis: the last axis cannot be gathered (it would cut blocks)");
    if (id_type != QM_I32 && id_type != QM_I64) return fail(QM_EINVAL, "ids: id_type must be QM_I32 or QM_I64");
    if (n_ids < 0) return fail(QM_EINVAL, "ids: negative count");
    const bool has_scales = d.scale_row_bytes != 0, has_biases = d.bias_row_bytes != 0;
    if (!has_scales && out_scales) return fail(QM_EINVAL, "scales: this format has no scales part; pass NULL");
    if (!has_biases && out_biases) return fail(QM_EINVAL, "biases: this format has no biases part; pass NULL");
    const bool packed = out_codes || out_scales || out_biases;
    if (!packed && !out_dense) return fail(QM_EINVAL, "out: no output given");
    if (packed) {
        if (!out_codes) return fail(QM_EINVAL, "codes: packed output needs out_codes");
        if (has_scales && !out_scales) return fail(QM_EINVAL, "scales: packed output needs out_scales");
        if (has_biases && !out_biases) return fail(QM_EINVAL, "biases: packed output needs out_biases");
    }
    if (out_dense && out_dtype != QM_F32 && out_dtype != QM_BF16 && out_dtype != QM_F16)
        return fail(QM_EINVAL, "out: dtype must be QM_F32, QM_BF16 or QM_F16");
    int64_t outer = 1, inner_rows = 1;
    for (int i = 0; i < axis; ++i) outer *= d.shape[i];
    for (int i = axis + 1; i < d.ndim - 1; ++i) inner_rows *= d.shape[i];
    const int64_t len = d.shape[axis];
    if (n_ids == 0 || outer == 0 || inner_rows == 0 || d.k == 0) return QM_OK;
    if (!ids) return fail(QM_EINVAL, "ids: NULL");
    if ((reinterpret_cast<uintptr_t>(ids) & (id_type == QM_I64 ? 7u : 3u)) != 0)
        return fail(QM_EINVAL, "ids: misaligned");
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const int id64 = id_type == QM_I64;
    if (packed) {
        const void* outs[3] = {out_codes, out_scales, out_biases};
        const uint8_t* srcs[3] = {d.codes, d.scales, d.biases};
        const int64_t rb[3] = {d.code_row_bytes, d.scale_row_bytes, d.bias_row_bytes};
        const char* names[3] = {"codes", "scales", "biases"};
        for (int p = 0; p < 3; ++p) {
            if (!rb[p]) continue;
            if (!aligned16(outs[p])) return fail(QM_EINVAL, std::string(names[p]) + ": output must be 16-byte aligned");
        }
        TakeParts tp;
        for (int p = 0; p < 3; ++p) {
            if (!rb[p]) continue;
            tp.src[tp.n] = srcs[p];
            tp.dst[tp.n] = static_cast<uint8_t*>(const_cast<void*>(outs[p]));
            tp.inner[tp.n] = inner_rows * rb[p];
            ++tp.n;
        }
        cudaError_t e = launch_take_packed(tp, outer, len, ids, id64, n_ids, st);  // one launch for every part
        if (e != cudaSuccess) return cuda_fail(e, "take launch");
    }
    if (out_dense) {
        if (!aligned16(out_dense)) return fail(QM_EINVAL, "out: dense output must be 16-byte aligned");
        cudaError_t e = launch_take_dense(d, axis, ids, id64, n_ids, out_dtype, out_dense, st);
        if (e != cudaSuccess) return cuda_fail(e, "take launch");
    }
    return QM_OK;
}

size_t qm_apply_experts_workspace(const qm_weight* w, int64_t T, int64_t topk) {
    set_error("");
    WDesc d;
    if (validate_weight(w, &d) != QM_OK || d.ndim != 3 || T <= 0 || topk <= 0) return 0;
    if (check_positions(T, topk, d.shape[0]) != QM_OK) return 0;
    return experts_workspace_bytes(d, T * topk, true);
}

size_t qm_experts_route_workspace(int64_t P, int64_t E) {
    if (P <= 0 || E < 0) return 0;
    return route_workspace_bytes(P, E);
}

qm_status qm_apply_experts(const qm_weight* w, const void* ids, int32_t id_type, int64_t T,
                           int64_t topk, const void* x, int64_t x_rows, int32_t x_dtype, void* y,
                           void* workspace, size_t workspace_bytes, qm_stream_t stream) {
    return apply_experts_checked(w, ids, id_type, T, topk, x, x_rows, x_dtype, y, workspace,
                                 workspace_bytes, stream, true);
}

}  // extern "C"

qm_status qm::apply_experts_checked(const qm_weight* w, const void* ids, int32_t id_type, int64_t T,
                                    int64_t topk, const void* x, int64_t x_rows, int32_t x_dtype, void* y,
                                    void* workspace, size_t workspace_bytes, qm_stream_t stream,
                                    bool allow_tensor) {
    set_error("");
    WDesc d;
    qm_status s = validate_weight(w, &d);
    if (s != QM_OK) return s;
    if (d.ndim != 3) return fail(QM_EINVAL, "w: apply_experts takes a 3-d weight [E, n, k]");
    if (T < 0 || topk < 0) return fail(QM_EINVAL, "ids: negative shape");
    if (id_type != QM_I32 && id_type != QM_I64) return fail(QM_EINVAL, "ids: id_type must be QM_I32 or QM_I64");
    s = check_positions(T, topk, d.shape[0]);
    if (s != QM_OK) return s;
    if (x_dtype != QM_BF16) return fail(QM_ENOTSUP, "x: apply_experts takes bfloat16 activations");
    if (x_rows != T && x_rows != T * topk)
        return fail(QM_EINVAL, "x: rows must be T (broadcast over topk) or T*topk");
    const int64_t P = T * topk;
    if (P == 0 || d.n == 0) return QM_OK;
    if (!y) return fail(QM_EINVAL, "y: NULL");
    if (!aligned16(y)) return fail(QM_EINVAL, "y: base address must be 16-byte aligned");
    if (!ids) return fail(QM_EINVAL, "ids: NULL");
    if ((reinterpret_cast<uintptr_t>(ids) & (id_type == QM_I64 ? 7u : 3u)) != 0)
        return fail(QM_EINVAL, "ids: misaligned");
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (d.k == 0)
        return check_launch(cudaMemsetAsync(y, 0, static_cast<size_t>(P * d.n * 2), st), "experts memset");
    if (!x) return fail(QM_EINVAL, "x: NULL");
    if (!aligned16(x)) return fail(QM_EINVAL, "x: base address must be 16-byte aligned");
    const size_t need = experts_workspace_bytes(d, P, allow_tensor);
    if (!workspace || workspace_bytes < need)
        return fail(QM_EINVAL, "workspace: needs " + std::to_string(need) + " bytes");
    if (!aligned16(workspace)) return fail(QM_EINVAL, "workspace: must be 16-byte aligned");
    return launch_experts(d, ids, id_type == QM_I64, T, topk, x, x_rows, y, workspace,
                          workspace_bytes, st, allow_tensor);
}

extern "C" {

qm_status qm_experts_route(const void* ids, int32_t id_type, int64_t P, int64_t E,
                           int32_t* counts, int32_t* offsets, int32_t* perm, void* workspace,
                           size_t workspace_bytes, qm_stream_t stream) {
    set_error("");
    if (id_type != QM_I32 && id_type != QM_I64) return fail(QM_EINVAL, "ids: id_type must be QM_I32 or QM_I64");
    if (P < 0 || E < 0) return fail(QM_EINVAL, "ids: negative size");
    const qm_status cs = check_positions(P, 1, E);
    if (cs != QM_OK) return cs;
    if (!counts || !offsets) return fail(QM_EINVAL, "out: counts and offsets are required");
    if (P > 0 && (!ids || !perm)) return fail(QM_EINVAL, "ids: NULL");
    const size_t need = route_workspace_bytes(P, E);
    if (P > 0 && (!workspace || workspace_bytes < need))
        return fail(QM_EINVAL, "workspace: needs " + std::to_string(need) + " bytes");
    return check_launch(launch_route(ids, id_type == QM_I64, P, E, counts, offsets, perm, workspace,
                                     reinterpret_cast<cudaStream_t>(stream)),
                        "route launch");
}

qm_status qm_check_wait_timeout(uint64_t limit_ns, qm_stream_t stream) {
    set_error("");
    if (limit_ns == 0 || limit_ns > 10ull * 1000 * 1000 * 1000)
        return fail(QM_EINVAL, "limit: must be between 1 ns and 10 s");
    return check_launch(launch_wait_timeout(limit_ns, reinterpret_cast<cudaStream_t>(stream)), "wait check launch");
}

qm_status qm_device_status(qm_stream_t stream) {
    set_error("");
    cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "stream synchronize");
    uint32_t flags = elementwise_read_clear_error() | gemv_read_clear_error() |
                     gemm_read_clear_error() | experts_read_clear_error();
    if (flags) return fail(QM_ETIMEOUT, "device: a device-side wait gave up");
    return QM_OK;
}

}  // extern "C"
