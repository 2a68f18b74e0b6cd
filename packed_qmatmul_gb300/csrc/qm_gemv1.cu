// qm_gemv1.cu -- the one-token product y[1, n] = x[1, k] * W^T over packed
// weights: the decode step's product, bound by launch latency for small
// layers and by HBM bandwidth for large ones.
//
// The product is the one "Nx_quant (raven-ml.dev API docs)", section
// "Products", val apply, defines: x times the weight's float32 values, summed
// at float32 and rounded once to x's dtype. Each lane sums the products of its
// own codes (exact small integers) with its activations, then scales the sum
// by its block's scale (and adds bias times the activations' sum): every
// product is exact, so the only roundings are float32 sums.
//
// Design (one GB300: 152 SMs):
//  * No shared memory, no barrier, no activation prologue: a warp owns R rows
//    and all of k; lane l holds inputs [1024c + 32l, 1024c + 32l + 32) of
//    every chunk c of 1024 inputs, reads its codes straight into registers
//    (16-byte loads where the layout allows) and its 32 activations, and the
//    warp adds its lanes' partial sums with shuffles.
//  * Codes become exact float32 integers with one byte permute into a float
//    of exponent 2^23 and one packed subtraction; products and sums run on the
//    packed float32 pairs of Blackwell's ALU (fma.rn.f32x2).
//  * Weights the caller marks static are read before the kernel waits on the
//    previous one (programmatic dependent launch), so a dependent chain of
//    small products pays for the activations' round trip only. The next
//    kernel is let start once this one's wait has returned.
//  * Warps stride over blocks of R rows, keeping the next two steps' codes in
//    flight (one for the formats with the largest lane data) while they work
//    on the current one: 3.39 -> 3.25 us per small layer at 4-bit.
//  * A lane whose partial sum is not finite, or whose block's scale could make
//    a value infinite (an MXFP4 scale byte of 253 or more, an affine scale or
//    bias of magnitude 2^119 or more), sums that block element by element
//    instead: each value decoded at float32 as dequant decodes it, times its
//    activation, in ascending k -- the infinities and NaNs IEEE arithmetic
//    gives a per-element sum ("Nx_quant", "Products": an MXFP4 value past
//    float32's range is infinite; a block whose float16 scale is infinite or
//    NaN gives infinite or NaN values).
//
// Layouts: MLX affine codes ("GPTQModel wiki: MLX Apple Silicon", "Packed
// layouts and exact transcoding": one little-endian bit stream per row, code i
// at bits [i*b, i*b + b)); Q8_0, MXFP4 and MXFP4 in GGUF's blocks ("Nx_quant",
// "Weights").
#include <cuda_runtime.h>

#include <algorithm>

#include "qm_device.cuh"
#include "qm_internal.h"

namespace qm {

namespace g1 {

constexpr int kWarps = 4;   // warps per CTA
constexpr int R = 2;        // rows per warp block
constexpr int kChunk = 1024;
constexpr int kMaxParts = 8;  // weights per launch (the C ABI's QM_MAX_MANY)

// One weight of a launch: several weights that read the same x (and share
// format, widths and k) run as one grid, their blocks of R rows numbered one
// after another.
struct Part {
    const uint8_t* codes;
    const uint8_t* scales;
    const uint8_t* biases;
    uint16_t* y;
    int64_t n;
};

struct Args {
    Part part[kMaxParts];
    int bstart[kMaxParts + 1];  // first block of each part; bstart[nparts]: all blocks
    int nparts;
    const uint16_t* x;
    int64_t k;
    int64_t code_row_bytes, scale_row_bytes;
    int gshift;          // log2(group_size): affine scales
    int sdt;             // affine scale dtype
    int nchunk;          // chunks of 1024 inputs: ceil(k / 1024)
    int static_w;        // the weights may be read before the previous kernel ends
    int ks;              // warps splitting one block's chunks (1: a warp takes all of k)
};

// Words of packed data a lane holds for one row and one chunk.
template <int FMT, int BITS>
struct Words {
    static constexpr int N = FMT == QM_AFFINE  ? BITS
                             : FMT == QM_Q8_0  ? 9
                             : FMT == QM_MXFP4 ? 4
                             : FMT == QM_Q4_K  ? 12
                             : FMT == QM_Q6_K  ? 20
                                               : 5;
};

// One lane's data for one row of one step: code words and the raw scale
// (and bias) of its block.
template <int FMT, int BITS>
struct Lane {
    uint32_t w[Words<FMT, BITS>::N];
    uint32_t s, b;   // affine: scale and bias bits; MXFP4: scale byte; others unused
    uint32_t off;    // Q8_0 / MXFP4 blocks: byte offset of the block in w[0]
};

// The aligned 32-bit word holding the byte at base + a (aligned as an address:
// a row of GGUF blocks may start at any even or odd byte).
QM_DEV uint32_t ldw(const uint8_t* base, int64_t a, uint64_t pol) {
    const uintptr_t p = reinterpret_cast<uintptr_t>(base + a) & ~uintptr_t(3);
    return ldg_stream(reinterpret_cast<const uint32_t*>(p), pol);
}

// Loads lane data for row `row` of weight P, inputs [i0, i0 + 32). Rows past n
// and inputs past k load nothing (the lane then contributes zero).
// Weights stream (ldg_stream, policy pol): each is read once per product.
template <int FMT, int BITS>
QM_DEV void load_lane(const Args& a, const Part& P, int64_t row, int64_t i0, uint64_t pol, Lane<FMT, BITS>& L) {
    constexpr int N = Words<FMT, BITS>::N;
    if (row >= P.n || i0 >= a.k) {
#pragma unroll
        for (int j = 0; j < N; ++j) L.w[j] = 0u;
        L.s = L.b = 0u;
        L.off = 0u;
        return;
    }
    const uint8_t* rp = P.codes + row * a.code_row_bytes;
    if constexpr (FMT == QM_AFFINE) {
        const int64_t byte0 = i0 * BITS / 8;  // 4*BITS-byte aligned
        if constexpr (BITS % 4 == 0) {
#pragma unroll
            for (int q = 0; q < BITS / 4; ++q) {
                const uint4 v = ldg_stream(reinterpret_cast<const uint4*>(rp + byte0) + q, pol);
                L.w[4 * q] = v.x; L.w[4 * q + 1] = v.y; L.w[4 * q + 2] = v.z; L.w[4 * q + 3] = v.w;
            }
        } else if constexpr (BITS % 2 == 0) {
#pragma unroll
            for (int q = 0; q < BITS / 2; ++q) {
                const uint2 v = ldg_stream(reinterpret_cast<const uint2*>(rp + byte0) + q, pol);
                L.w[2 * q] = v.x; L.w[2 * q + 1] = v.y;
            }
        } else {
#pragma unroll
            for (int q = 0; q < BITS; ++q) L.w[q] = ldg_stream(reinterpret_cast<const uint32_t*>(rp + byte0) + q, pol);
        }
        const int64_t gi = row * (a.scale_row_bytes / 2) + (i0 >> a.gshift);
        L.s = ldg_stream(reinterpret_cast<const uint16_t*>(P.scales) + gi, pol);
        L.b = ldg_stream(reinterpret_cast<const uint16_t*>(P.biases) + gi, pol);
        L.off = 0u;
    } else if constexpr (FMT == QM_Q8_0) {
        // 34 bytes at a 2-byte boundary: the nine aligned words holding them
        const int64_t a0 = (i0 / 32) * 34;
        L.off = static_cast<uint32_t>((reinterpret_cast<uintptr_t>(rp) + a0) & 3u);
#pragma unroll
        for (int j = 0; j < 9; ++j) L.w[j] = ldw(rp, a0 + 4 * j, pol);
        L.s = L.b = 0u;
    } else if constexpr (FMT == QM_MXFP4) {
        const uint4 v = ldg_stream(reinterpret_cast<const uint4*>(rp + i0 / 2), pol);
        L.w[0] = v.x; L.w[1] = v.y; L.w[2] = v.z; L.w[3] = v.w;
        L.s = ldg_stream(P.scales + row * a.scale_row_bytes + i0 / 32, pol);
        L.b = 0u;
        L.off = 0u;
    } else if constexpr (FMT == QM_Q4_K) {
        // sub-block j = (i0 / 32) mod 8 of block i0 / 256 (144 bytes, 16-byte aligned):
        // the 16-byte header (d, dmin, scales and mins), then the 32 quant bytes
        // whose low (j even) or high (j odd) nibbles are its values
        const uint8_t* blk = rp + (i0 / 256) * 144;
        const int j = static_cast<int>((i0 / 32) % 8);
        const uint4 h = ldg_stream(reinterpret_cast<const uint4*>(blk), pol);
        const uint4* qp = reinterpret_cast<const uint4*>(blk + 16 + 32 * (j / 2));
        const uint4 q0 = ldg_stream(qp, pol), q1 = ldg_stream(qp + 1, pol);
        L.w[0] = h.x; L.w[1] = h.y; L.w[2] = h.z; L.w[3] = h.w;
        L.w[4] = q0.x; L.w[5] = q0.y; L.w[6] = q0.z; L.w[7] = q0.w;
        L.w[8] = q1.x; L.w[9] = q1.y; L.w[10] = q1.z; L.w[11] = q1.w;
        L.off = static_cast<uint32_t>(j);
        L.s = L.b = 0u;
    } else if constexpr (FMT == QM_Q6_K) {
        // quarter t of half h (j = 4h + t = (i0 / 32) mod 8) of block i0 / 256 (210
        // bytes, 2-byte aligned): the aligned words holding its 32 ql bytes and 32
        // qh bytes, and those holding its two scales and d
        const int64_t a0 = (i0 / 256) * 210;
        const int j = static_cast<int>((i0 / 32) % 8), h = j / 4, t = j % 4;
        const int64_t aql = a0 + 64 * h + 32 * (t % 2), aqh = a0 + 128 + 32 * h;
#pragma unroll
        for (int q = 0; q < 9; ++q) {
            L.w[q] = ldw(rp, aql + 4 * q, pol);
            L.w[9 + q] = ldw(rp, aqh + 4 * q, pol);
        }
        L.w[18] = ldw(rp, a0 + 192 + 8 * h + 2 * t, pol);
        L.w[19] = ldw(rp, a0 + 208, pol);
        // bits 0-1: ql's byte offset within its word; bits 2-3: qh's; bits 4-5: the
        // scales'; bits 6-7: d's; bits 8-9: t
        const uintptr_t base = reinterpret_cast<uintptr_t>(rp);
        L.off = static_cast<uint32_t>(((base + aql) & 3) | (((base + aqh) & 3) << 2) |
                                      (((base + a0 + 192 + 8 * h + 2 * t) & 3) << 4) | (((base + a0 + 208) & 3) << 6) |
                                      (t << 8));
        L.s = L.b = 0u;
    } else {  // MXFP4 in GGUF's 17-byte blocks: the five aligned words holding them
        const int64_t a0 = (i0 / 32) * 17;
        L.off = static_cast<uint32_t>((reinterpret_cast<uintptr_t>(rp) + a0) & 3u);
#pragma unroll
        for (int j = 0; j < 5; ++j) L.w[j] = ldw(rp, a0 + 4 * j, pol);
        L.s = L.b = 0u;
    }
}

// A lane's 32 activations as float32 pairs, in the order its format pairs
// its codes, and their sum (affine bias).
template <int FMT, int BITS>
struct Acts {
    float2 p[16];
    float sum;
};

template <int FMT, int BITS>
QM_DEV void load_acts(const Args& a, int64_t i0, Acts<FMT, BITS>& X) {
    uint32_t w[16];
    if (i0 < a.k) {
        const uint4* src = reinterpret_cast<const uint4*>(a.x + i0);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const uint4 v = __ldca(src + q);  // written by the previous kernel: a coherent load
            w[4 * q] = v.x; w[4 * q + 1] = v.y; w[4 * q + 2] = v.z; w[4 * q + 3] = v.w;
        }
    } else {
#pragma unroll
        for (int q = 0; q < 16; ++q) w[q] = 0u;
    }
    // w[q] holds inputs 2q (low half) and 2q + 1 (high half), as bf16
    auto lo = [&](int i) { return __uint_as_float(w[i >> 1] << 16); };
    auto hi = [&](int i) { return __uint_as_float(w[i >> 1] & 0xFFFF0000u); };
    auto at = [&](int i) { return (i & 1) ? hi(i) : lo(i); };
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        if constexpr (FMT == QM_AFFINE && BITS == 4) {
            // word q of codes holds inputs 8q .. 8q + 7; its low nibbles are the
            // even inputs, its high nibbles the odd ones, paired byte by byte
            const int q = j >> 2, r = j & 3;
            const int base = 8 * q + ((r & 2) ? 1 : 0) + ((r & 1) ? 4 : 0);
            X.p[j] = make_float2(at(base), at(base + 2));
        } else if constexpr (FMT == QM_MXFP4_BLOCKS) {
            X.p[j] = make_float2(at(j), at(j + 16));  // byte j: inputs j and j + 16
        } else {
            X.p[j] = make_float2(lo(2 * j), hi(2 * j + 1));
        }
    }
    if constexpr (FMT == QM_AFFINE || FMT == QM_Q4_K) {  // for the bias (the Q4_K min) term
        float2 s = make_float2(0.0f, 0.0f);
#pragma unroll
        for (int j = 0; j < 16; ++j) s = add2(s, X.p[j]);
        X.sum = s.x + s.y;
    } else {
        X.sum = 0.0f;
    }
}

constexpr uint32_t kMagic = 0x4B000000u;  // float 2^23: 2^23 + u for a byte u in its low bits

QM_DEV float2 two_bytes(uint32_t w, uint32_t sel_lo, uint32_t sel_hi) {
    return make_float2(__uint_as_float(prmt(w, kMagic, sel_lo)), __uint_as_float(prmt(w, kMagic, sel_hi)));
}

// Code i (0..31) of a lane's affine chunk of BITS-bit codes.
template <int BITS>
QM_DEV uint32_t code_at(const uint32_t (&w)[BITS], int i) {
    const int bit = i * BITS, q = bit >> 5, sh = bit & 31;
    uint32_t v = w[q] >> sh;
    if (sh + BITS > 32) v |= w[q + 1] << (32 - sh);
    return v & ((1u << BITS) - 1u);
}

// sum over the lane's 32 inputs of code * x: the exact integer codes (or e2m1
// values) times the activations, float32 sums
template <int FMT, int BITS>
QM_DEV float lane_dot(const Lane<FMT, BITS>& L, const Acts<FMT, BITS>& X) {
    float2 acc = make_float2(0.0f, 0.0f);
    if constexpr (FMT == QM_AFFINE && BITS == 4) {
        const float2 neg = make_float2(-8388608.0f, -8388608.0f);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const uint32_t lo = L.w[q] & 0x0F0F0F0Fu, hi = (L.w[q] >> 4) & 0x0F0F0F0Fu;
            acc = fma2(add2(two_bytes(lo, 0x7540, 0x7541), neg), X.p[4 * q], acc);
            acc = fma2(add2(two_bytes(lo, 0x7542, 0x7543), neg), X.p[4 * q + 1], acc);
            acc = fma2(add2(two_bytes(hi, 0x7540, 0x7541), neg), X.p[4 * q + 2], acc);
            acc = fma2(add2(two_bytes(hi, 0x7542, 0x7543), neg), X.p[4 * q + 3], acc);
        }
    } else if constexpr (FMT == QM_AFFINE && BITS == 8) {
        const float2 neg = make_float2(-8388608.0f, -8388608.0f);
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            acc = fma2(add2(two_bytes(L.w[q], 0x7540, 0x7541), neg), X.p[2 * q], acc);
            acc = fma2(add2(two_bytes(L.w[q], 0x7542, 0x7543), neg), X.p[2 * q + 1], acc);
        }
    } else if constexpr (FMT == QM_AFFINE) {
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            const float2 c = make_float2(static_cast<float>(code_at<BITS>(L.w, 2 * j)),
                                         static_cast<float>(code_at<BITS>(L.w, 2 * j + 1)));
            acc = fma2(c, X.p[j], acc);
        }
    } else if constexpr (FMT == QM_Q8_0) {
        // quants from byte 2 of the block: word j of them is bytes 4j+2 .. 4j+5
        const float2 neg = make_float2(-8388736.0f, -8388736.0f);  // -(2^23 + 128)
        const uint32_t sh = 8u * (L.off + 2u);                     // 16 or 32
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const uint32_t qw =
                (sh == 32u ? L.w[j + 1] : __funnelshift_r(L.w[j], L.w[j + 1], 16)) ^ 0x80808080u;  // q + 128
            acc = fma2(add2(two_bytes(qw, 0x7540, 0x7541), neg), X.p[2 * j], acc);
            acc = fma2(add2(two_bytes(qw, 0x7542, 0x7543), neg), X.p[2 * j + 1], acc);
        }
    } else if constexpr (FMT == QM_Q4_K) {
        const float2 neg = make_float2(-8388608.0f, -8388608.0f);
        const uint32_t sh = (L.off & 1u) ? 4u : 0u;  // odd sub-blocks: the high nibbles
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const uint32_t c = (L.w[4 + q] >> sh) & 0x0F0F0F0Fu;  // values 4q .. 4q + 3
            acc = fma2(add2(two_bytes(c, 0x7540, 0x7541), neg), X.p[2 * q], acc);
            acc = fma2(add2(two_bytes(c, 0x7542, 0x7543), neg), X.p[2 * q + 1], acc);
        }
    } else if constexpr (FMT == QM_MXFP4) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            uint32_t h[4];
            e2m1x8_to_f16x2(L.w[q], h);  // byte i -> (input 2i, input 2i + 1)
#pragma unroll
            for (int i = 0; i < 4; ++i)
                acc = fma2(__half22float2(*reinterpret_cast<const __half2*>(&h[i])), X.p[4 * q + i], acc);
        }
    } else {  // MXFP4 blocks: 16 data bytes from byte 1 of the block
        const uint32_t sh = 8u * (L.off + 1u);  // 8 .. 32
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const uint32_t dw = sh == 32u ? L.w[q + 1] : __funnelshift_r(L.w[q], L.w[q + 1], sh);
            uint32_t h[4];
            e2m1x8_to_f16x2(dw, h);  // byte i -> (input j, input j + 16), j = 4q + i
#pragma unroll
            for (int i = 0; i < 4; ++i)
                acc = fma2(__half22float2(*reinterpret_cast<const __half2*>(&h[i])), X.p[4 * q + i], acc);
        }
    }
    return acc.x + acc.y;
}

QM_DEV float sval(uint32_t h, int sdt) { return sdt == QM_F16 ? f16_bits_to_f32(h) : bf16_bits_to_f32(h); }

// Q6_K: the lane's two sums over (q - 32) * x, values 0..15 and 16..31 (each
// half has its own sub-block scale).
QM_DEV float2 q6_k_dots(const uint32_t (&w)[20], uint32_t off, const float2 (&xp)[16]) {
    const uint32_t oql = 8u * (off & 3u), oqh = 8u * ((off >> 2) & 3u);
    const uint32_t t = (off >> 8) & 3u;
    const uint32_t lsh = t >= 2 ? 4u : 0u, hsh = 2u * t;
    const float2 neg = make_float2(-8388640.0f, -8388640.0f);  // -(2^23 + 32)
    float2 a0 = make_float2(0.0f, 0.0f), a1 = make_float2(0.0f, 0.0f);
#pragma unroll
    for (int q = 0; q < 8; ++q) {  // values 4q .. 4q + 3
        const uint32_t lw = oql ? __funnelshift_r(w[q], w[q + 1], oql) : w[q];
        const uint32_t hw = oqh ? __funnelshift_r(w[9 + q], w[10 + q], oqh) : w[9 + q];
        const uint32_t c = ((lw >> lsh) & 0x0F0F0F0Fu) | (((hw >> hsh) & 0x03030303u) << 4);  // 6-bit q per byte
        float2& a = q < 4 ? a0 : a1;
        a = fma2(add2(two_bytes(c, 0x7540, 0x7541), neg), xp[2 * q], a);
        a = fma2(add2(two_bytes(c, 0x7542, 0x7543), neg), xp[2 * q + 1], a);
    }
    return make_float2(a0.x + a0.y, a1.x + a1.y);
}

// Q4_K: sub-block j's 6-bit scale and min from the 12 bytes after d and dmin
// (header words 1..3): sub-blocks 0..3 from the low 6 bits of bytes j and
// j + 4, 4..7 from the nibbles of byte j + 4 with their top two bits from the
// top bits of bytes j - 4 and j.
QM_DEV void q4_k_scale_min(const uint32_t (&w)[12], int j, int& sc, int& mn) {
    auto sb = [&](int i) -> int {  // byte i of words 1..3, chosen by selects (no indexed array)
        const uint32_t wd = i < 4 ? w[1] : (i < 8 ? w[2] : w[3]);
        return static_cast<int>((wd >> (8 * (i & 3))) & 0xFFu);
    };
    if (j < 4) {
        sc = sb(j) & 63;
        mn = sb(4 + j) & 63;
    } else {
        sc = (sb(4 + j) & 15) | ((sb(j - 4) >> 6) << 4);
        mn = (sb(4 + j) >> 4) | ((sb(j) >> 6) << 4);
    }
}

// The e8m0 scale of a GGUF MXFP4 block held in the lane's words.
QM_DEV uint32_t blocks_scale_byte(const uint32_t (&w)[5], uint32_t off) { return (w[0] >> (8 * off)) & 0xFFu; }

// The lane's contribution for one row and chunk with its block's scale (and
// bias), and whether that block may hold a value the block-scaled sum does not
// reproduce exactly (non-finite values, or values that overflow float32).
template <int FMT, int BITS>
QM_DEV float lane_part(const Args& a, const Lane<FMT, BITS>& L, const Acts<FMT, BITS>& X, bool& exact) {
    if constexpr (FMT == QM_Q6_K) {
        const float2 dd = q6_k_dots(L.w, L.off, X.p);
        const uint32_t sw = L.w[18] >> (8 * ((L.off >> 4) & 3u));
        const float d = f16_bits_to_f32((L.w[19] >> (8 * ((L.off >> 6) & 3u))) & 0xFFFFu);
        exact = false;
        return fmaf(d * static_cast<float>(static_cast<int8_t>(sw & 0xFFu)), dd.x,
                    d * static_cast<float>(static_cast<int8_t>((sw >> 8) & 0xFFu)) * dd.y);
    } else if constexpr (FMT == QM_Q4_K) {
        int sc, mn;
        q4_k_scale_min(L.w, static_cast<int>(L.off), sc, mn);
        const float d = f16_bits_to_f32(L.w[0] & 0xFFFFu), dmin = f16_bits_to_f32(L.w[0] >> 16);
        exact = false;
        return fmaf(d * static_cast<float>(sc), lane_dot<FMT, BITS>(L, X), -(dmin * static_cast<float>(mn)) * X.sum);
    } else if constexpr (FMT == QM_AFFINE) {
        const float dot = lane_dot<FMT, BITS>(L, X);
        const float s = sval(L.s, a.sdt), b = sval(L.b, a.sdt);
        exact = fmaxf(fabsf(s), fabsf(b)) >= 0x1p119f;  // |code * s + b| may reach 2^128
        return fmaf(s, dot, b * X.sum);
    } else if constexpr (FMT == QM_Q8_0) {
        const float dot = lane_dot<FMT, BITS>(L, X);
        const uint32_t dbits = L.off ? (L.w[0] >> 16) : (L.w[0] & 0xFFFFu);
        exact = false;
        return f16_bits_to_f32(dbits) * dot;
    } else if constexpr (FMT == QM_MXFP4) {
        const float dot = lane_dot<FMT, BITS>(L, X);
        exact = L.s >= 253u;  // values of magnitude 4 (at 253) or 2 (at 254) pass float32's range
        return e8m0_to_f32(L.s) * dot;
    } else {  // MXFP4 in GGUF's blocks
        const float dot = lane_dot<FMT, BITS>(L, X);
        const uint32_t sb = blocks_scale_byte(L.w, L.off);
        exact = sb >= 253u;
        return e8m0_to_f32(sb) * dot;
    }
}

// Value i of row `row` of weight P, decoded at float32 from global memory as
// dequant decodes it.
template <int FMT, int BITS>
QM_DEV float value_g(const Args& a, const Part& P, int64_t row, int64_t i) {
    const uint8_t* rp = P.codes + row * a.code_row_bytes;
    if constexpr (FMT == QM_AFFINE) {
        const int64_t bit = i * BITS;
        const uint32_t lo = __ldg(rp + bit / 8), hi = (bit % 8 + BITS > 8) ? __ldg(rp + bit / 8 + 1) : 0u;
        const uint32_t c = ((lo | (hi << 8)) >> (bit % 8)) & ((1u << BITS) - 1u);
        const int64_t gi = row * (a.scale_row_bytes / 2) + (i >> a.gshift);
        return fmaf(static_cast<float>(c), sval(__ldg(reinterpret_cast<const uint16_t*>(P.scales) + gi), a.sdt),
                    sval(__ldg(reinterpret_cast<const uint16_t*>(P.biases) + gi), a.sdt));
    } else if constexpr (FMT == QM_Q8_0) {
        const uint8_t* blk = rp + (i / 32) * 34;
        const float d = f16_bits_to_f32(static_cast<uint32_t>(__ldg(blk)) | (static_cast<uint32_t>(__ldg(blk + 1)) << 8));
        return d * static_cast<float>(static_cast<int8_t>(__ldg(blk + 2 + i % 32)));
    } else if constexpr (FMT == QM_Q4_K) {
        const uint8_t* blk = rp + (i / 256) * 144;
        const int v = static_cast<int>(i % 256), c = v / 64, rr = v % 64, j = 2 * c + (rr >= 32);
        uint32_t w[12];
#pragma unroll
        for (int q = 0; q < 4; ++q) w[q] = __ldg(reinterpret_cast<const uint32_t*>(blk) + q);
        int sc, mn;
        q4_k_scale_min(w, j, sc, mn);
        const uint32_t byte = __ldg(blk + 16 + 32 * c + rr % 32);
        const float d = f16_bits_to_f32(w[0] & 0xFFFFu), dmin = f16_bits_to_f32(w[0] >> 16);
        return fmaf(d * static_cast<float>(sc), static_cast<float>(rr < 32 ? (byte & 15u) : (byte >> 4)),
                    -(dmin * static_cast<float>(mn)));
    } else if constexpr (FMT == QM_Q6_K) {
        const uint8_t* blk = rp + (i / 256) * 210;
        const int v = static_cast<int>(i % 256), h = v / 128, t = (v % 128) / 32, l = v % 32;
        const uint32_t lo = __ldg(blk + 64 * h + l + 32 * (t % 2));
        const uint32_t q = ((t < 2 ? lo : (lo >> 4)) & 15u) | (((static_cast<uint32_t>(__ldg(blk + 128 + 32 * h + l)) >> (2 * t)) & 3u) << 4);
        const float d = f16_bits_to_f32(static_cast<uint32_t>(__ldg(blk + 208)) | (static_cast<uint32_t>(__ldg(blk + 209)) << 8));
        return d * static_cast<float>(static_cast<int8_t>(__ldg(blk + 192 + 8 * h + 2 * t + l / 16))) *
               static_cast<float>(static_cast<int>(q) - 32);
    } else {
        uint32_t c, sb;
        if constexpr (FMT == QM_MXFP4) {
            const uint32_t byte = __ldg(rp + i / 2);
            c = (i & 1) ? (byte >> 4) : (byte & 15u);
            sb = __ldg(P.scales + row * a.scale_row_bytes + i / 32);
        } else {
            const uint8_t* blk = rp + (i / 32) * 17;
            const int t = static_cast<int>(i % 32);
            const uint32_t byte = __ldg(blk + 1 + (t & 15));
            c = t < 16 ? (byte & 15u) : (byte >> 4);
            sb = __ldg(blk);
        }
        uint32_t h[4];
        e2m1x8_to_f16x2(c, h);
        return __half2float(__ushort_as_half(static_cast<unsigned short>(h[0] & 0xFFFFu))) * e8m0_to_f32(sb);
    }
}

// The lane's contribution summed element by element: value times activation
// at float32, inputs in ascending order. Out of line: rarely taken.
template <int FMT, int BITS>
static __device__ __noinline__ float lane_exact(const Args& a, const Part& P, int64_t row, int64_t i0) {
    float acc = 0.0f;
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
        acc = fmaf(bf16_bits_to_f32(__ldca(a.x + i0 + i)), value_g<FMT, BITS>(a, P, row, i0 + i), acc);
    return acc;
}

template <int FMT, int BITS>
__global__ void __launch_bounds__(kWarps * 32) gemv1_kernel(const __grid_constant__ Args a) {
    const int lane = threadIdx.x & 31;
    // 32-bit block indices (a block is R rows; fewer than 2^31 blocks) and steps
    // walked incrementally: no integer division anywhere on the path.
    // ks == 1: warp w takes blocks w, w + nwarp, ... and all chunks of each.
    // ks > 1: the CTA is ks warps taking blocks blockIdx.x, + gridDim.x, ...;
    // warp kp takes chunks [kp * nchunk / ks, (kp + 1) * nchunk / ks) of each,
    // and the warps' sums meet in shared memory (added in warp order), so a
    // long row costs one warp's share of k, not all of it, after the wait.
    const int ks = a.ks, kp = static_cast<int>(threadIdx.x >> 5);
    const bool split = ks > 1;
    const int warp0 = split ? static_cast<int>(blockIdx.x)
                            : static_cast<int>((blockIdx.x * blockDim.x + threadIdx.x) >> 5);
    const int nwarp = split ? static_cast<int>(gridDim.x) : static_cast<int>((gridDim.x * blockDim.x) >> 5);
    const int nblocks = a.bstart[a.nparts];
    const int cpw = a.nchunk / ks, c_lo = split ? kp * cpw : 0, c_hi = c_lo + cpw;  // this warp's chunks
    __shared__ float s_red[kWarps][R];  // split: each warp's row sums of the current block
    if (warp0 >= nblocks) return;  // nothing to read or write (the whole CTA, when split)
    // the weight holding block b, and the block's index within that weight
    auto locate = [&](int b, int& g, int& lb) {
        g = 0;
        #pragma unroll 1
        while (g + 1 < a.nparts && b >= a.bstart[g + 1]) ++g;
        lb = b - a.bstart[g];
    };
    // two steps' codes in flight where the registers still leave 16 warps per
    // SM (four CTAs); one for the formats whose lane data is larger (8-bit
    // affine, Q4_K, Q6_K: with two, fewer CTAs fit and layers take two waves)
    constexpr bool kDeep = !(FMT == QM_AFFINE && BITS == 8) && FMT != QM_Q4_K && FMT != QM_Q6_K;
    Lane<FMT, BITS> cur[R], nxt[R], nx2[R];  // this step's codes and the next one's (two)
    const uint64_t pol = l2_evict_first_policy();
    auto load_step = [&](int g, int lb, int c, Lane<FMT, BITS> (&L)[R]) {
        const Part& P = a.part[g];
        const int64_t i0 = static_cast<int64_t>(c) * kChunk + 32 * lane;
#pragma unroll
        for (int r = 0; r < R; ++r) load_lane<FMT, BITS>(a, P, static_cast<int64_t>(lb) * R + r, i0, pol, L[r]);
    };
    // the (block, chunk) step after (b, c), and its block's weight and index there
    auto advance = [&](int& b, int& c, int& g, int& lb) {
        if (++c == c_hi) {
            c = c_lo;
            b += nwarp;
            if (b < nblocks) locate(b, g, lb);
        }
    };
    int cg, clb;  // the current block's weight and its block index there
    locate(warp0, cg, clb);
    int b1 = warp0, c1 = c_lo, g1 = cg, lb1 = clb;  // the next step
    advance(b1, c1, g1, lb1);
    if (a.static_w) {  // the weight is not written by the previous kernel: read it first
        load_step(cg, clb, c_lo, cur);
        if (kDeep && b1 < nblocks) load_step(g1, lb1, c1, nxt);
        grid_dependency_wait();
    } else {
        grid_dependency_wait();
        load_step(cg, clb, c_lo, cur);
        if (kDeep && b1 < nblocks) load_step(g1, lb1, c1, nxt);
    }
    // Let the next kernel start only now: it still has this kernel's whole
    // remaining run to read its own static weights, and only one kernel waits
    // ahead (triggered at entry, several later ones became resident at once
    // and each launch took about 0.2 us longer)
    grid_launch_dependents();
    Acts<FMT, BITS> X;
    float y[R];
#pragma unroll
    for (int r = 0; r < R; ++r) y[r] = 0.0f;
    bool have_x = false;
    // (block b, chunk c) steps, chunks fastest
    #pragma unroll 1
    for (int b = warp0, c = c_lo; b < nblocks;) {
        int b2 = b1, c2 = c1, g2 = g1, lb2 = lb1;  // the step after the next
        if (b2 < nblocks) advance(b2, c2, g2, lb2);
        if constexpr (kDeep) {
            if (b2 < nblocks) load_step(g2, lb2, c2, nx2);
        } else {
            if (b1 < nblocks) load_step(g1, lb1, c1, nxt);
        }
        const int64_t i0 = static_cast<int64_t>(c) * kChunk + 32 * lane;
        if (cpw > 1 || !have_x) {
            load_acts<FMT, BITS>(a, i0, X);
            have_x = true;
        }
        const Part& P = a.part[cg];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            bool exact;
            float part = lane_part<FMT, BITS>(a, cur[r], X, exact);
            const int64_t row = static_cast<int64_t>(clb) * R + r;
            if ((exact || !isfinite(part)) && row < P.n && i0 < a.k) part = lane_exact<FMT, BITS>(a, P, row, i0);
            y[r] += part;
        }
        if (c == c_hi - 1) {
            // the R rows' sums over the warp, in a fixed order: lanes first
            // exchange halves of their R values, then add down to one each
            static_assert(R == 2, "the exchange below pairs two rows");
            const float give = (lane & 1) ? y[0] : y[1];
            float v = ((lane & 1) ? y[1] : y[0]) + __shfl_xor_sync(0xffffffffu, give, 1);
#pragma unroll
            for (int o = 2; o < 32; o <<= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
            const int64_t row = static_cast<int64_t>(clb) * R + lane;  // lane 0: row 0 of the block, lane 1: row 1
            if (split) {  // the block's ks warps (every warp of the CTA, in step): their sums in warp order
                if (lane < R) s_red[kp][lane] = v;
                __syncthreads();
                if (kp == 0 && lane < R) {
                    float sum = s_red[0][lane];
                    #pragma unroll 1
                    for (int q = 1; q < ks; ++q) sum += s_red[q][lane];
                    v = sum;
                }
                __syncthreads();  // s_red is written again for the next block
            }
            if (kp == 0 || !split) {
                if (lane < R && row < P.n) {
                    __nv_bfloat16 bv = __float2bfloat16_rn(v);
                    P.y[row] = *reinterpret_cast<uint16_t*>(&bv);
                }
            }
#pragma unroll
            for (int r = 0; r < R; ++r) y[r] = 0.0f;
        }
#pragma unroll
        for (int r = 0; r < R; ++r) {
            cur[r] = nxt[r];
            if constexpr (kDeep) nxt[r] = nx2[r];
        }
        b = b1;
        c = c1;
        cg = g1;
        clb = lb1;
        b1 = b2;
        c1 = c2;
        g1 = g2;
        lb1 = lb2;
    }
}

template <int FMT, int BITS>
cudaError_t launch_t(const Args& a, cudaStream_t st) {
    // all warps resident at once where the rows allow: 16 warps per SM
    const int64_t nb = a.bstart[a.nparts], cap = int64_t(num_sms()) * 16;
    if (a.ks > 1)  // a CTA of ks warps per block
        return launch_pdl(gemv1_kernel<FMT, BITS>, static_cast<unsigned>(std::min<int64_t>(nb, cap / a.ks)),
                          a.ks * 32, 0, st, a);
    const int64_t warps = std::min<int64_t>(nb, cap);
    const unsigned grid = static_cast<unsigned>((warps + kWarps - 1) / kWarps);
    return launch_pdl(gemv1_kernel<FMT, BITS>, grid, kWarps * 32, 0, st, a);
}

}  // namespace g1

bool gemv1_supported(const WDesc& w) {
    if (w.ndim != 2 || w.n < 1 || w.k < 32 || w.n > (int64_t(1) << 31)) return false;
    if (w.fmt == QM_AFFINE) {
        if (w.gs < 32 || (w.gs & (w.gs - 1))) return false;
        return w.bits == 2 || w.bits == 3 || w.bits == 4 || w.bits == 5 || w.bits == 6 || w.bits == 8;
    }
    return w.fmt == QM_Q8_0 || w.fmt == QM_MXFP4 || w.fmt == QM_MXFP4_BLOCKS || w.fmt == QM_Q4_K || w.fmt == QM_Q6_K;
}

bool gemv1_many_supported(const WDesc* ws, int count) {
    if (count < 1 || count > g1::kMaxParts) return false;
    int64_t blocks = 0;
    for (int i = 0; i < count; ++i) {
        const WDesc& w = ws[i];
        if (!gemv1_supported(w)) return false;
        if (w.fmt != ws[0].fmt || w.bits != ws[0].bits || w.gs != ws[0].gs || w.k != ws[0].k ||
            w.code_row_bytes != ws[0].code_row_bytes || w.scale_row_bytes != ws[0].scale_row_bytes ||
            (w.fmt == QM_AFFINE && w.sdt != ws[0].sdt))
            return false;
        blocks += (w.n + g1::R - 1) / g1::R;
    }
    return blocks < (int64_t(1) << 31);
}

cudaError_t launch_gemv1_many(const WDesc* ws, int count, const void* x, void* const* ys, cudaStream_t st) {
    using namespace g1;
    const WDesc& w = ws[0];
    Args a{};
    a.nparts = count;
    a.bstart[0] = 0;
    bool all_static = true;
    for (int i = 0; i < count; ++i) {
        a.part[i].codes = ws[i].codes;
        a.part[i].scales = ws[i].scales;
        a.part[i].biases = ws[i].biases;
        a.part[i].y = static_cast<uint16_t*>(ys[i]);
        a.part[i].n = ws[i].n;
        a.bstart[i + 1] = a.bstart[i] + static_cast<int>((ws[i].n + R - 1) / R);
        all_static = all_static && ws[i].is_static;
    }
    a.x = static_cast<const uint16_t*>(x);
    a.k = w.k;
    a.code_row_bytes = w.code_row_bytes;
    a.scale_row_bytes = w.scale_row_bytes;
    a.gshift = 0;
    while ((1 << a.gshift) < w.gs) ++a.gshift;
    a.sdt = w.sdt;
    a.nchunk = static_cast<int>((w.k + kChunk - 1) / kChunk);
    a.static_w = all_static ? 1 : 0;
    // chunks split over 4, 3 or 2 warps where that divides them (k alone decides:
    // a row's sum order must not depend on the other weights of a launch)
    a.ks = 1;
    for (int d = kWarps; d >= 2; --d)
        if (a.nchunk % d == 0) {
            a.ks = d;
            break;
        }
    if (w.fmt == QM_AFFINE) {
        switch (w.bits) {
            case 2: return launch_t<QM_AFFINE, 2>(a, st);
            case 3: return launch_t<QM_AFFINE, 3>(a, st);
            case 4: return launch_t<QM_AFFINE, 4>(a, st);
            case 5: return launch_t<QM_AFFINE, 5>(a, st);
            case 6: return launch_t<QM_AFFINE, 6>(a, st);
            default: return launch_t<QM_AFFINE, 8>(a, st);
        }
    }
    if (w.fmt == QM_Q8_0) return launch_t<QM_Q8_0, 8>(a, st);
    if (w.fmt == QM_MXFP4) return launch_t<QM_MXFP4, 4>(a, st);
    if (w.fmt == QM_Q4_K) return launch_t<QM_Q4_K, 4>(a, st);
    if (w.fmt == QM_Q6_K) return launch_t<QM_Q6_K, 6>(a, st);
    return launch_t<QM_MXFP4_BLOCKS, 4>(a, st);
}

cudaError_t launch_gemv1(const WDesc& w, const void* x, void* y, cudaStream_t st) {
    void* ys[1] = {y};
    return launch_gemv1_many(&w, 1, x, ys, st);
}

}  // namespace qm
