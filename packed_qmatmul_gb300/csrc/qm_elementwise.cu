// qm_elementwise.cu -- dequant, take (packed gather and gather-then-decode)
// and the plain fallback product, all HBM-bound.
//
// Decoding follows "Nx_quant (raven-ml.dev API docs)", sections "Weights"
// (Q8_0 and Mxfp4 layouts, e2m1 / e8m0 values) and "Products" (dequant: every
// value a float32 rounded once to the output dtype; take: a gather of the
// packed rows, an out-of-range position gathering zero bytes), and the MLX
// affine rule of "GPTQModel wiki: MLX Apple Silicon" ("Concepts ..." and
// "Packed layouts and exact transcoding": value = code*scale + bias over a
// little-endian code stream).
#include <cuda_runtime.h>

#include <algorithm>

#include "qm_device.cuh"
#include "qm_internal.h"

namespace qm {

static __device__ uint32_t g_err_elementwise = 0;

uint32_t elementwise_read_clear_error() {
    uint32_t v = 0, z = 0;
    cudaMemcpyFromSymbol(&v, g_err_elementwise, sizeof(v));
    cudaMemcpyToSymbol(g_err_elementwise, &z, sizeof(z));
    return v;
}

namespace {

struct DecodeArgs {
    const uint8_t* codes;
    const uint8_t* scales;
    const uint8_t* biases;
    int64_t k;
    int64_t code_row_bytes;
    int64_t scale_row_bytes;  // bytes per row of scales (and of biases)
    int gs;
    int sdt;  // QM_BF16 / QM_F16 (affine)
};

QM_DEV float scale_val(const uint8_t* p, int64_t idx, int sdt) {
    const uint16_t h = reinterpret_cast<const uint16_t*>(p)[idx];
    return sdt == QM_F16 ? f16_bits_to_f32(h) : bf16_bits_to_f32(h);
}

// The 32 float32 values of unit u (inputs 32u .. 32u+31) of source row r.
template <int FMT, int BITS>
QM_DEV void decode_unit(const DecodeArgs& a, int64_t r, int64_t u, float (&v)[32]) {
    if constexpr (FMT == QM_AFFINE) {
        const int64_t g = (32 * u) / a.gs;  // the unit lies in one group (gs >= 32)
        const int64_t ng = a.k / a.gs;
        const float s = scale_val(a.scales, r * ng + g, a.sdt);
        const float b = scale_val(a.biases, r * ng + g, a.sdt);
        const uint4* src = reinterpret_cast<const uint4*>(a.codes + r * a.code_row_bytes + u * 4 * BITS);
        if constexpr (BITS != 4 && BITS != 8) {
            // 2, 3, 5, 6 bits: the unit's BITS words (4-byte aligned), codes read
            // across word boundaries from the little-endian bit stream
            const uint32_t* wp = reinterpret_cast<const uint32_t*>(a.codes + r * a.code_row_bytes + u * 4 * BITS);
            uint32_t w[BITS];
#pragma unroll
            for (int j = 0; j < BITS; ++j) w[j] = __ldg(wp + j);
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                const int bit = i * BITS, q = bit >> 5, sh = bit & 31;
                uint32_t c = w[q] >> sh;
                if (sh + BITS > 32) c |= w[q + 1] << (32 - sh);
                v[i] = fmaf(static_cast<float>(c & ((1u << BITS) - 1u)), s, b);
            }
        } else if constexpr (BITS == 4) {
            const uint4 q = __ldg(src);
            const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
            for (int j = 0; j < 4; ++j)
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    v[8 * j + i] = fmaf(static_cast<float>((w[j] >> (4 * i)) & 15u), s, b);
        } else {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const uint4 q = __ldg(src + h);
                const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
                for (int j = 0; j < 4; ++j)
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        v[16 * h + 4 * j + i] = fmaf(static_cast<float>((w[j] >> (8 * i)) & 255u), s, b);
            }
        }
    } else if constexpr (FMT == QM_Q8_0) {
        // A block: little-endian f16 d, then 32 int8 quants; 2-byte aligned.
        const uint16_t* blk = reinterpret_cast<const uint16_t*>(a.codes + r * a.code_row_bytes + u * 34);
        const float d = f16_bits_to_f32(__ldg(blk));
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const uint32_t two = __ldg(blk + 1 + i);
            v[2 * i] = d * static_cast<float>(static_cast<int8_t>(two & 0xFF));
            v[2 * i + 1] = d * static_cast<float>(static_cast<int8_t>(two >> 8));
        }
    } else if constexpr (FMT == QM_Q4_K) {
        // "Nx_quant", "Weights", Q4_K (ggml's block_q4_K): unit u is sub-block
        // j = u mod 8 of block u / 8; its 32 quants are the low (j even) or
        // high (j odd) nibbles of quant bytes 32(j/2) .. 32(j/2) + 31; its
        // 6-bit scale and min come from the 12 bytes after d and dmin. value
        // = (d * sc) * q - dmin * m: exact products, one rounding (fmaf).
        const uint8_t* blk = a.codes + r * a.code_row_bytes + (u / 8) * 144;
        const int j = static_cast<int>(u % 8);
        const uint4 hdr = __ldg(reinterpret_cast<const uint4*>(blk));
        const float d = f16_bits_to_f32(hdr.x & 0xFFFFu), dmin = f16_bits_to_f32(hdr.x >> 16);
        // byte i of the 12 scale/min bytes (header bytes 4 .. 15), by selects
        auto sb = [&](int i) -> int {
            const uint32_t wd = i < 4 ? hdr.y : (i < 8 ? hdr.z : hdr.w);
            return static_cast<int>((wd >> (8 * (i & 3))) & 0xFFu);
        };
        int sc, mn;
        if (j < 4) {
            sc = sb(j) & 63;
            mn = sb(4 + j) & 63;
        } else {
            sc = (sb(4 + j) & 15) | ((sb(j - 4) >> 6) << 4);
            mn = (sb(4 + j) >> 4) | ((sb(j) >> 6) << 4);
        }
        const float d1 = d * static_cast<float>(sc), m1 = dmin * static_cast<float>(mn);
        const uint4* qp = reinterpret_cast<const uint4*>(blk + 16 + 32 * (j / 2));
        const int sh = (j & 1) ? 4 : 0;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const uint4 q = __ldg(qp + h);
            const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
            for (int e = 0; e < 16; ++e)
                v[16 * h + e] = fmaf(d1, static_cast<float>((w[e / 4] >> (8 * (e % 4) + sh)) & 15u), -m1);
        }
    } else if constexpr (FMT == QM_Q6_K) {
        // "Nx_quant", "Weights", Q6_K (ggml's block_q6_K): unit u is quarter
        // t = u mod 4 of half h = (u / 4) mod 2 of block u / 8; value l of it
        // has its low 4 bits in ql[64h + l + 32(t mod 2)] (low nibble for
        // t < 2), its high 2 bits at bit 2t of qh[32h + l] and the int8 scale
        // scales[8h + 2t + l/16]; value = (d * sc) * (q - 32), exact.
        const uint8_t* blk = a.codes + r * a.code_row_bytes + (u / 8) * 210;  // 2-byte aligned
        const int h = static_cast<int>((u / 4) % 2), t = static_cast<int>(u % 4);
        const uint16_t* ql = reinterpret_cast<const uint16_t*>(blk + 64 * h + 32 * (t % 2));
        const uint16_t* qh = reinterpret_cast<const uint16_t*>(blk + 128 + 32 * h);
        const float d = f16_bits_to_f32(__ldg(reinterpret_cast<const uint16_t*>(blk + 208)));
        const uint32_t scw = __ldg(reinterpret_cast<const uint16_t*>(blk + 192 + 8 * h + 2 * t));
        const float d0 = d * static_cast<float>(static_cast<int8_t>(scw & 0xFF));
        const float d1 = d * static_cast<float>(static_cast<int8_t>(scw >> 8));
        const int lsh = t < 2 ? 0 : 4, hsh = 2 * t;
#pragma unroll
        for (int e = 0; e < 16; ++e) {
            const uint32_t lo2 = __ldg(ql + e), hi2 = __ldg(qh + e);  // values 2e and 2e + 1
#pragma unroll
            for (int b = 0; b < 2; ++b) {
                const int l = 2 * e + b;
                const int q = static_cast<int>(((lo2 >> (8 * b + lsh)) & 15u) | (((hi2 >> (8 * b + hsh)) & 3u) << 4));
                v[l] = (l < 16 ? d0 : d1) * static_cast<float>(q - 32);
            }
        }
    } else if constexpr (FMT == QM_MXFP4_BLOCKS) {
        // GGUF's 17-byte block: the e8m0 scale byte, then byte j holding value j
        // (low nibble) and value j + 16 (high nibble); blocks are byte-aligned
        const uint8_t* blk = a.codes + r * a.code_row_bytes + u * 17;
        const float sc = e8m0_to_f32(__ldg(blk));
#pragma unroll
        for (int j = 0; j < 16; j += 4) {
            const uint32_t w = static_cast<uint32_t>(__ldg(blk + 1 + j)) |
                               (static_cast<uint32_t>(__ldg(blk + 2 + j)) << 8) |
                               (static_cast<uint32_t>(__ldg(blk + 3 + j)) << 16) |
                               (static_cast<uint32_t>(__ldg(blk + 4 + j)) << 24);
            uint32_t h2[4];
            e2m1x8_to_f16x2(w, h2);  // byte i -> (its low nibble, its high nibble)
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h2[i]));
                v[j + i] = f.x * sc;
                v[j + i + 16] = f.y * sc;
            }
        }
    } else {  // MXFP4: 16 bytes of codes (value 2i low nibble, 2i+1 high), one e8m0 scale
        const uint4 q = __ldg(reinterpret_cast<const uint4*>(a.codes + r * a.code_row_bytes + u * 16));
        const float sc = e8m0_to_f32(__ldg(a.scales + r * a.scale_row_bytes + u));
        const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            uint32_t h2[4];
            e2m1x8_to_f16x2(w[j], h2);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h2[i]));
                v[8 * j + 2 * i] = f.x * sc;
                v[8 * j + 2 * i + 1] = f.y * sc;
            }
        }
    }
}

template <int OUT>
QM_DEV void store_unit(void* out, int64_t elem, const float (&v)[32]) {
    if constexpr (OUT == QM_F32) {
        float4* o = reinterpret_cast<float4*>(static_cast<float*>(out) + elem);
#pragma unroll
        for (int i = 0; i < 8; ++i) o[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
    } else {
        uint4* o = reinterpret_cast<uint4*>(static_cast<uint16_t*>(out) + elem);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            uint32_t p[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float lo = v[8 * i + 2 * j], hi = v[8 * i + 2 * j + 1];
                if constexpr (OUT == QM_BF16) {
                    __nv_bfloat162 t = __floats2bfloat162_rn(lo, hi);
                    p[j] = *reinterpret_cast<uint32_t*>(&t);
                } else {
                    __half2 t = __floats2half2_rn(lo, hi);
                    p[j] = *reinterpret_cast<uint32_t*>(&t);
                }
            }
            o[i] = make_uint4(p[0], p[1], p[2], p[3]);
        }
    }
}

// Output row -> source row (or -1 for zeros).
struct IdentityMap {
    QM_DEV int64_t operator()(int64_t r) const { return r; }
};

struct GatherMap {
    const void* ids;
    int id64;
    int64_t n_ids, len, inner_rows;
    QM_DEV int64_t operator()(int64_t r) const {
        const int64_t ii = r % inner_rows;
        const int64_t op = r / inner_rows;
        const int64_t p = op % n_ids, o = op / n_ids;
        const int64_t id = id64 ? __ldg(static_cast<const int64_t*>(ids) + p)
                                : static_cast<int64_t>(__ldg(static_cast<const int32_t*>(ids) + p));
        if (id < 0 || id >= len) return -1;
        return (o * len + id) * inner_rows + ii;
    }
};

// A warp's 32 consecutive units of 16-bit output (2 KB, contiguous) written
// as four coalesced 512-byte stores: lane l's four 16-byte pieces go to a
// shared-memory stage (piece j of lane l in slot 4l + (j ^ ((l >> 1) & 3)),
// so neither the writes nor the reads of a quarter warp share a bank group),
// then lane l stores pieces l, l + 32, l + 64 and l + 96 of the warp's run.
template <int OUT>
QM_DEV void store_warp_units(void* out, int64_t elem0, const float (&v)[32], uint4* stage, int lane) {
    uint4 p[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        uint32_t w[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float lo = v[8 * i + 2 * j], hi = v[8 * i + 2 * j + 1];
            if constexpr (OUT == QM_BF16) {
                __nv_bfloat162 t = __floats2bfloat162_rn(lo, hi);
                w[j] = *reinterpret_cast<uint32_t*>(&t);
            } else {
                __half2 t = __floats2half2_rn(lo, hi);
                w[j] = *reinterpret_cast<uint32_t*>(&t);
            }
        }
        p[i] = make_uint4(w[0], w[1], w[2], w[3]);
    }
    __syncwarp();
#pragma unroll
    for (int i = 0; i < 4; ++i) stage[4 * lane + (i ^ ((lane >> 1) & 3))] = p[i];
    __syncwarp();
    uint4* o = reinterpret_cast<uint4*>(static_cast<uint16_t*>(out) + elem0);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int q = 32 * i + lane, src = q >> 2, c = q & 3;
        o[q] = stage[4 * src + (c ^ ((src >> 1) & 3))];
    }
}

template <class Map>
constexpr bool kStaged = false;
template <>
constexpr bool kStaged<IdentityMap> = true;

template <int FMT, int BITS, int OUT, class Map>
__global__ void __launch_bounds__(256) decode_rows_kernel(DecodeArgs a, int64_t out_rows, Map map,
                                                          void* out) {
    grid_launch_dependents();
    grid_dependency_wait();  // the weight, ids or output may belong to the previous kernel
    __shared__ uint4 s_stage[kStaged<Map> ? 8 : 1][128];  // one 2 KB stage per warp (16-bit outputs)
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t upr = a.k / 32;
    const int64_t total = out_rows * upr;
    // the stride is a multiple of 32, so a warp's lanes hold 32 consecutive units
    // until the last, partial run
    for (int64_t t = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; t - lane < total;
         t += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const bool mine = t < total;
        float v[32];
        if (mine) {
            const int64_t r = t / upr, u = t - r * upr;
            const int64_t src = map(r);
            if (src >= 0) {
                decode_unit<FMT, BITS>(a, src, u, v);
            } else {
                // an out-of-range position gathers zero bytes: their values are
                // zeros, -0. in Q6_K ("Nx_quant", "Weights")
#pragma unroll
                for (int i = 0; i < 32; ++i) v[i] = FMT == QM_Q6_K ? -0.0f : 0.0f;
            }
        }
        // staged, coalesced stores for full dequant (2 % faster); a gather, short
        // and latency-bound, stores directly (its dense take measured slower staged)
        if (kStaged<Map> && OUT != QM_F32 && t - lane + 31 < total) {
            store_warp_units<OUT>(out, (t - lane) * 32, v, s_stage[warp], lane);
        } else if (mine) {
            store_unit<OUT>(out, t * 32, v);
        }
    }
}

template <class Map>
cudaError_t launch_decode_rows(const WDesc& w, int64_t out_rows, Map map, int out_dtype, void* out,
                               cudaStream_t st) {
    DecodeArgs a{w.codes, w.scales, w.biases, w.k, w.code_row_bytes, w.scale_row_bytes, w.gs, w.sdt};
    const int64_t total = out_rows * (w.k / 32);
    if (total == 0) return cudaSuccess;
    const int threads = 256;
    const int64_t blocks = std::min<int64_t>((total + threads - 1) / threads, int64_t(num_sms()) * 16);
#define QM_DECODE_CASE(F, B, O)                                                                  \
    if (w.fmt == F && (F != QM_AFFINE || w.bits == B) && out_dtype == O) {                        \
        return launch_pdl(decode_rows_kernel<F, B, O, Map>, static_cast<unsigned>(blocks), threads, 0, st, a, \
                          out_rows, map, out);                                                  \
    }
#define QM_DECODE_OUTS(F, B) QM_DECODE_CASE(F, B, QM_F32) QM_DECODE_CASE(F, B, QM_BF16) QM_DECODE_CASE(F, B, QM_F16)
    QM_DECODE_OUTS(QM_AFFINE, 2)
    QM_DECODE_OUTS(QM_AFFINE, 3)
    QM_DECODE_OUTS(QM_AFFINE, 4)
    QM_DECODE_OUTS(QM_AFFINE, 5)
    QM_DECODE_OUTS(QM_AFFINE, 6)
    QM_DECODE_OUTS(QM_AFFINE, 8)
    QM_DECODE_OUTS(QM_Q8_0, 8)
    QM_DECODE_OUTS(QM_MXFP4, 4)
    QM_DECODE_OUTS(QM_MXFP4_BLOCKS, 4)
    QM_DECODE_OUTS(QM_Q4_K, 4)
    QM_DECODE_OUTS(QM_Q6_K, 6)
#undef QM_DECODE_OUTS
#undef QM_DECODE_CASE
    return cudaErrorInvalidValue;
}

// ------------------------------------------------------------ packed gather
// dst[o, p, :] = src[o, ids[p], :] (inner bytes each), zero bytes out of range.
// One warp per gathered row (outer index o, position q): the id is read once
// and the row's bytes of every part are copied in V-sized pieces; positions
// outside [0, len) get zero bytes.
template <typename V>
__global__ void __launch_bounds__(256) take_packed_kernel(TakeParts tp, int64_t outer, int64_t len,
                                                          const void* ids, int id64, int64_t n_ids) {
    grid_launch_dependents();
    grid_dependency_wait();
    const int lane = threadIdx.x & 31;
    const int64_t rows = outer * n_ids;
    const int64_t nw = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    for (int64_t r = (blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x) >> 5; r < rows; r += nw) {
        const int64_t o = r / n_ids, q = r - o * n_ids;
        const int64_t id = id64 ? __ldg(static_cast<const int64_t*>(ids) + q)
                                : static_cast<int64_t>(__ldg(static_cast<const int32_t*>(ids) + q));
        const bool in = id >= 0 && id < len;
        if (tp.one_each) {
            // every part's row is at most 32 pieces: one piece per lane and part,
            // all loads issued before any store (one memory round trip, not three)
            V v[3];
#pragma unroll
            for (int part = 0; part < 3; ++part) {
                memset(&v[part], 0, sizeof(V));
                const int64_t vpr = tp.inner[part] / static_cast<int64_t>(sizeof(V));
                if (part < tp.n && in && lane < vpr)
                    v[part] = __ldg(reinterpret_cast<const V*>(tp.src[part] + (o * len + id) * tp.inner[part]) + lane);
            }
#pragma unroll
            for (int part = 0; part < 3; ++part) {
                const int64_t vpr = tp.inner[part] / static_cast<int64_t>(sizeof(V));
                if (part < tp.n && lane < vpr) reinterpret_cast<V*>(tp.dst[part] + r * tp.inner[part])[lane] = v[part];
            }
            continue;
        }
#pragma unroll 1
        for (int part = 0; part < tp.n; ++part) {
            const int64_t vpr = tp.inner[part] / static_cast<int64_t>(sizeof(V));
            const V* src = reinterpret_cast<const V*>(tp.src[part] + (o * len + (in ? id : 0)) * tp.inner[part]);
            V* dst = reinterpret_cast<V*>(tp.dst[part] + r * tp.inner[part]);
            for (int64_t c = lane; c < vpr; c += 32) {
                V v;
                if (in) v = __ldg(src + c);
                else memset(&v, 0, sizeof(V));
                dst[c] = v;
            }
        }
    }
}

}  // namespace

// ------------------------------------------------------------ quantize_q8_0
// "Nx_quant (raven-ml.dev API docs)", val quantize_q8_0: x read at float32,
// per block of 32 values d = amax / 127 (amax over the finite values) stored at
// float16 rounded to nearest, and quant j = round(v_j * (1 / d)), halves away
// from zero, the reciprocal and products at float32 (1 / d = 0 where d is 0,
// and a product that is not finite gives the quant 0). A block holding a NaN
// has a NaN scale and quants 0; else one holding an infinity has the scale +inf
// and quants 0. One warp per block, lane j holding value j: the loads of a
// block are one 128-byte line and its 34 bytes are one coalesced store.
namespace {
template <int XDT>
QM_DEV float load_f32(const void* x, int64_t i) {
    if constexpr (XDT == QM_F32) return __ldg(static_cast<const float*>(x) + i);
    else if constexpr (XDT == QM_BF16) return bf16_bits_to_f32(__ldg(static_cast<const uint16_t*>(x) + i));
    else return f16_bits_to_f32(__ldg(static_cast<const uint16_t*>(x) + i));
}

template <int XDT>
__global__ void __launch_bounds__(256) quantize_q8_0_kernel(const void* x, int64_t nblocks, uint8_t* blocks) {
    grid_launch_dependents();
    grid_dependency_wait();
    const int lane = threadIdx.x & 31;
    const int64_t nw = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    for (int64_t b = (blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x) >> 5; b < nblocks; b += nw) {
        const float v = load_f32<XDT>(x, b * 32 + lane);
        const bool has_nan = __any_sync(0xffffffffu, isnan(v));
        const bool has_inf = __any_sync(0xffffffffu, isinf(v));
        // amax over the finite values: magnitude bits of non-negative floats order as the values
        const uint32_t mag = isfinite(v) ? (__float_as_uint(v) & 0x7FFFFFFFu) : 0u;
        const float amax = __uint_as_float(__reduce_max_sync(0xffffffffu, mag));
        uint16_t h;
        int8_t q = 0;
        if (has_nan || has_inf) {
            h = has_nan ? 0x7E00 : 0x7C00;
        } else {
            const float d = __fdiv_rn(amax, 127.0f);
            const float id = d != 0.0f ? __fdiv_rn(1.0f, d) : 0.0f;
            h = __half_as_ushort(__float2half_rn(d));
            const float p = __fmul_rn(v, id);
            q = isfinite(p) ? static_cast<int8_t>(roundf(p)) : static_cast<int8_t>(0);
        }
        uint8_t* out = blocks + b * 34;
        if (lane < 2) out[lane] = static_cast<uint8_t>(lane == 0 ? (h & 0xFF) : (h >> 8));  // little-endian d
        out[2 + lane] = static_cast<uint8_t>(q);
    }
}
}  // namespace

cudaError_t launch_quantize_q8_0(const void* x, int x_dtype, int64_t rows, int64_t k, uint8_t* blocks,
                                 cudaStream_t st) {
    const int64_t nblocks = rows * (k / 32);
    if (nblocks == 0) return cudaSuccess;
    const int64_t grid = std::min<int64_t>((nblocks + 7) / 8, int64_t(num_sms()) * 16);
    if (x_dtype == QM_F32)
        return launch_pdl(quantize_q8_0_kernel<QM_F32>, static_cast<unsigned>(grid), 256, 0, st, x, nblocks, blocks);
    if (x_dtype == QM_BF16)
        return launch_pdl(quantize_q8_0_kernel<QM_BF16>, static_cast<unsigned>(grid), 256, 0, st, x, nblocks, blocks);
    return launch_pdl(quantize_q8_0_kernel<QM_F16>, static_cast<unsigned>(grid), 256, 0, st, x, nblocks, blocks);
}

// ------------------------------------------------------------ bounded-wait check
// One warp waits on an mbarrier that nothing arrives at, with the bounded wait
// every pipeline uses; it gives up after limit_ns, raises this file's device
// flag and exits. Nothing faults and nothing is left waiting.
namespace {
__global__ void __launch_bounds__(32) wait_timeout_kernel(uint64_t limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    const uint32_t b = smem_u32(&bar);
    if (threadIdx.x == 0) {
        mbar_init(b, 1);
        fence_mbar_init();
    }
    __syncwarp();
    if (threadIdx.x == 0 && !mbar_wait_slow(b, 0, limit_ns)) atomicOr(&g_err_elementwise, DEV_ERR_TIMEOUT);
}
}  // namespace

cudaError_t launch_wait_timeout(uint64_t limit_ns, cudaStream_t st) {
    wait_timeout_kernel<<<1, 32, 0, st>>>(limit_ns);
    return cudaGetLastError();
}

cudaError_t launch_dequant(const WDesc& w, int out_dtype, void* out, cudaStream_t st) {
    return launch_decode_rows(w, w.rows, IdentityMap{}, out_dtype, out, st);
}

cudaError_t launch_take_dense(const WDesc& w, int axis, const void* ids, int id64, int64_t n_ids,
                              int out_dtype, void* out, cudaStream_t st) {
    int64_t outer = 1, inner_rows = 1;
    for (int i = 0; i < axis; ++i) outer *= w.shape[i];
    for (int i = axis + 1; i < w.ndim - 1; ++i) inner_rows *= w.shape[i];
    GatherMap m{ids, id64, n_ids, w.shape[axis], inner_rows};
    return launch_decode_rows(w, outer * n_ids * inner_rows, m, out_dtype, out, st);
}

cudaError_t launch_take_packed(const TakeParts& tp, int64_t outer, int64_t len, const void* ids, int id64,
                               int64_t n_ids, cudaStream_t st) {
    const int64_t rows = outer * n_ids;
    if (rows == 0 || tp.n == 0) return cudaSuccess;
    const int64_t blocks = std::min<int64_t>((rows + 7) / 8, int64_t(num_sms()) * 16);
    int64_t common = 0;  // the widest piece that divides every part's row
    for (int part = 0; part < tp.n; ++part) common |= tp.inner[part];
    auto go = [&](auto vec) -> cudaError_t {
        using V = decltype(vec);
        TakeParts t2 = tp;
        t2.one_each = 1;
        for (int part = 0; part < tp.n; ++part)
            if (tp.inner[part] > 32 * static_cast<int64_t>(sizeof(V))) t2.one_each = 0;
        return launch_pdl(take_packed_kernel<V>, static_cast<unsigned>(blocks), 256, 0, st, t2, outer, len, ids,
                          id64, n_ids);
    };
    if (common % 16 == 0) return go(uint4{});
    if (common % 8 == 0) return go(uint2{});
    if (common % 4 == 0) return go(uint32_t{});
    if (common % 2 == 0) return go(uint16_t{});
    return go(uint8_t{});
}

// ------------------------------------------------------------ plain product
// One warp per (output row j, block of up to 8 rows of x): each lane decodes
// 32-value units in turn and forms their dot products with x; the warp then
// sums lanes in a fixed butterfly order. Used where the fast paths decline.
namespace {
template <int FMT, int BITS>
__global__ void __launch_bounds__(256) apply_simple_kernel(DecodeArgs a, int64_t n, const uint16_t* x,
                                                           int64_t M, uint16_t* y) {
    const int lane = threadIdx.x & 31;
    const int64_t warp = (blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x) >> 5;
    const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    const int64_t mblocks = (M + 7) / 8;
    const int64_t upr = a.k / 32;
    for (int64_t job = warp; job < n * mblocks; job += nwarps) {
        const int64_t j = job / mblocks, m0 = (job % mblocks) * 8;
        float acc[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
        for (int64_t u = lane; u < upr; u += 32) {
            float v[32];
            decode_unit<FMT, BITS>(a, j, u, v);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                if (m0 + i < M) {
                    const uint16_t* xr = x + (m0 + i) * a.k + 32 * u;
                    float s = 0.0f;
#pragma unroll
                    for (int e = 0; e < 32; ++e) s = fmaf(bf16_bits_to_f32(xr[e]), v[e], s);
                    acc[i] += s;
                }
            }
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            float s = acc[i];
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
            if (lane == 0 && m0 + i < M) {
                __nv_bfloat16 b = __float2bfloat16_rn(s);
                y[(m0 + i) * n + j] = *reinterpret_cast<uint16_t*>(&b);
            }
        }
    }
}
}  // namespace

cudaError_t launch_apply_simple(const WDesc& w, const void* x, int64_t M, void* y, cudaStream_t st) {
    DecodeArgs a{w.codes, w.scales, w.biases, w.k, w.code_row_bytes, w.scale_row_bytes, w.gs, w.sdt};
    const int64_t jobs = w.n * ((M + 7) / 8);
    const int64_t blocks = std::min<int64_t>((jobs * 32 + 255) / 256, int64_t(num_sms()) * 8);
    const uint16_t* xb = static_cast<const uint16_t*>(x);
    uint16_t* yb = static_cast<uint16_t*>(y);
#define QM_SIMPLE(B) apply_simple_kernel<QM_AFFINE, B><<<static_cast<unsigned>(blocks), 256, 0, st>>>(a, w.n, xb, M, yb)
    if (w.fmt == QM_AFFINE && w.bits == 2) QM_SIMPLE(2);
    else if (w.fmt == QM_AFFINE && w.bits == 3) QM_SIMPLE(3);
    else if (w.fmt == QM_AFFINE && w.bits == 4) QM_SIMPLE(4);
    else if (w.fmt == QM_AFFINE && w.bits == 5) QM_SIMPLE(5);
    else if (w.fmt == QM_AFFINE && w.bits == 6) QM_SIMPLE(6);
    else if (w.fmt == QM_AFFINE) QM_SIMPLE(8);
#undef QM_SIMPLE
    else if (w.fmt == QM_Q8_0)
        apply_simple_kernel<QM_Q8_0, 8><<<static_cast<unsigned>(blocks), 256, 0, st>>>(a, w.n, xb, M, yb);
    else if (w.fmt == QM_MXFP4_BLOCKS)
        apply_simple_kernel<QM_MXFP4_BLOCKS, 4><<<static_cast<unsigned>(blocks), 256, 0, st>>>(a, w.n, xb, M, yb);
    else if (w.fmt == QM_Q4_K)
        apply_simple_kernel<QM_Q4_K, 4><<<static_cast<unsigned>(blocks), 256, 0, st>>>(a, w.n, xb, M, yb);
    else if (w.fmt == QM_Q6_K)
        apply_simple_kernel<QM_Q6_K, 6><<<static_cast<unsigned>(blocks), 256, 0, st>>>(a, w.n, xb, M, yb);
    else
        apply_simple_kernel<QM_MXFP4, 4><<<static_cast<unsigned>(blocks), 256, 0, st>>>(a, w.n, xb, M, yb);
    return cudaGetLastError();
}

}  // namespace qm
