// qm_gemm_kernel.cuh -- prefill product y[M, n] = x[M, k] * W^T for M >= 17 on the
// 5th-generation tensor cores (tcgen05), decoding the packed weight in the
// pipeline.
//
// The product is "Nx_quant (raven-ml.dev API docs)", section "Products", val
// apply: summed at float32, rounded once to x's dtype. Here each weight value
// (the float32 value of "Weights" / "Products", dequant) is rounded to bf16 to
// enter a kind::f16 MMA; the sums are float32 in TMEM. The rounding of the
// weights stays inside the product's error bound (a relative 2^-9 per value).
//
// One CTA per tile of 128 weight rows x NTOK tokens (NTOK 128 or 256; grid:
// token tiles fastest so x stays in L2 while each weight tile is read once;
// experts: weight tiles fastest within each expert's rows). The roles of the
// MMA operands are turned round from y = x W^T: the decoded weight tile is
// A (M = 128 rows, one TMEM lane each) and lives in tensor memory, written
// there by the decoders with tcgen05.st; the activation tile is B (N = NTOK)
// in shared memory. Decoded weights never pass through shared memory, whose
// bandwidth then serves only the TMA fills and the MMA's activation reads.
//  * warp 0, one lane: TMA producer. Activation tiles (NTOK tokens x 64 k,
//    bf16, 128B-swizzled: the canonical K-major layout) and raw packed chunks
//    of the weight tile (128 rows x 256 or 128 k values).
//  * warp 1, one lane: tcgen05.mma (M = 128, N = NTOK, K = 16, four per k
//    step, A from TMEM) into an NTOK-column accumulator, committing each stage
//    back to its producers through mbarriers; warp 1 also owns the TMEM
//    allocation (accumulator, then four 32-column weight stages).
//  * warps 2..9: decoders, two groups of four taking alternate k steps; warp w
//    owns TMEM lane quarter w % 4, so a thread decodes one weight row's 64
//    values per k step (scales fetched from global memory one chunk ahead).
//    After the k loop they read the accumulator back and store y.
// Plain products of at most 128 tokens use the dual layout instead: warp 0
// loads only the raw chunks; the even k steps have their own activation
// producer (warp 10) and MMA issuer (warp 1, accumulator 0), the odd steps
// theirs (warps 11 and 12, accumulator 1), and the epilogue adds the two
// accumulators. Each issuing thread completes about one TMA box per 0.39 us or
// one MMA per 0.14 us whatever their sizes (measured on GB300), so a single
// producer and a single issuer cap a 128-token tile; two pipes lift both caps.
// Every wait is bounded; a wait that gives up raises the device flag and the
// CTA winds down with its copies and MMAs drained.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "qm_device.cuh"
#include "qm_internal.h"

namespace qm {
namespace gemm {

// The device flag that a wait giving up raises. Every translation unit that
// includes this header has its own (internal linkage) and reads it back
// through read_clear_flag under its own name.
static __device__ uint32_t g_err_gemm = 0;

static inline uint32_t read_clear_flag() {
    uint32_t v = 0, z = 0;
    cudaMemcpyFromSymbol(&v, g_err_gemm, sizeof(v));
    cudaMemcpyToSymbol(g_err_gemm, &z, sizeof(z));
    return v;
}

constexpr int BK = 64;          // k values per step
constexpr int kDecWarps = 8;
// Roles by warp. Classic layout: warp 0 loads the raw weight chunks and the
// activation tiles, warp 1 issues the MMAs, warps 2..9 decode. Every issuing
// thread (of TMA copies or of MMAs) completes about one operation at a time
// at a fixed cost (about 0.39 us per TMA box, 0.14 us per MMA) whatever its
// size, so one producer and one issuer cap a 128-token tile. The dual layout
// (plain 128-token products) runs two pipelines by k-step parity, as the
// decoder groups already do: warp 0 loads the raw chunks only, warp 10 / warp 1
// load the activations of and issue the even steps into accumulator 0, warp 11
// / warp 12 the odd steps into accumulator 1; the epilogue adds the two.
constexpr int threads_for(bool dual) { return (dual ? 13 : 10) * 32; }
constexpr int NR = 2;           // raw chunk slots

// Raw chunk geometry per format: values per chunk, bytes per row per chunk,
// whether the TMA box is 128B-swizzled, and the tensor map's element size.
// Affine 2, 3, 5 and 6-bit codes (GEN) come as 128 inputs per row, 16 * BITS
// bytes, unswizzled (a row's codes then start on a 4-byte boundary).
// Q4_K comes as one 144-byte block (256 inputs) per row, unswizzled: rows 144
// bytes (nine 16-byte units) apart put consecutive rows in distinct bank groups.
// MXFP4 in GGUF's 17-byte blocks comes as 16 blocks (512 inputs, 272 bytes, a
// 16-byte multiple, as Q8_0's 8 blocks are) per row, unswizzled, read as
// 16-bit elements (the box's inner extent is then 136 elements).
template <int FMT, int BITS>
struct Raw {
    static constexpr bool GEN = FMT == QM_AFFINE && BITS != 4 && BITS != 8;
    static constexpr bool MXB = FMT == QM_MXFP4_BLOCKS;
    static constexpr int RAWK = (GEN || (FMT == QM_AFFINE && BITS == 8)) ? 128 : MXB ? 512 : 256;
    static constexpr int BYTES =
        GEN ? 16 * BITS : (FMT == QM_Q8_0 || MXB) ? 272 : (FMT == QM_Q4_K) ? 144 : 128;
    static constexpr bool SW = FMT != QM_Q8_0 && FMT != QM_Q4_K && !GEN && !MXB;
    static constexpr int ELEM = (FMT == QM_Q8_0 || MXB) ? 2 : 1;
    static constexpr int SPR = RAWK / BK;  // k steps per chunk
};

struct Params {
    CUtensorMap tm_x;    // x as bytes [M, 2k], boxes of 128 B x NTOK rows, 128B-swizzled
    CUtensorMap tm_raw;  // codes as [n, code_row_bytes], boxes of Raw::BYTES x 128 rows
    const uint8_t* scales;
    const uint8_t* biases;
    uint16_t* y;
    int64_t M, n, k;
    int64_t scale_row_bytes;
    int sdt;
    int gshift;  // log2(group_size) of an affine weight
    int ksteps, mtiles, ntiles;
    uint32_t off_x, off_raw, raw_stage_bytes;
    // split k (plain products with few tiles): a cluster of `splitk` CTAs takes
    // chunks [rank * cps, (rank + 1) * cps) of one tile; partial sums meet in
    // the receive areas at off_recv, each CTA adding one slice of the tokens
    int splitk, cps;
    uint32_t off_recv;
    // grouped mode (apply_experts), off when g_off is null: x holds the routed
    // activation rows expert by expert, the weight is [E, n, k], and m tile
    // slot t is the t-th BM-row tile of the experts' row ranges in order
    const int32_t* g_off;   // [E + 1] each expert's first row of x
    const int32_t* g_perm;  // row of x -> row of y
    int64_t g_E;
};

// Where 16-byte chunk c of row r of a 128B-swizzled, 128-byte-row tile sits.
QM_DEV uint32_t sw128(uint32_t r, uint32_t c) { return r * 128 + ((c ^ (r & 7)) << 4); }

QM_DEV float sval(uint32_t h, int sdt) { return sdt == QM_F16 ? f16_bits_to_f32(h) : bf16_bits_to_f32(h); }

QM_DEV uint32_t bf2(float lo, float hi) {
    __nv_bfloat162 t = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&t);
}

// 2^23 + u as a float32, for u < 2^23 already placed in the low bits.
QM_DEV float magic_f(uint32_t bits_or_u) { return __uint_as_float(bits_or_u | 0x4B000000u); }

// The scale (and bias) one decoder thread needs for one k step.
struct Sc {
    float s, b;
};

template <int FMT, int BITS, int GS>
QM_DEV Sc load_scale(const Params& p, int64_t grow, int64_t vidx) {
    Sc r{0.0f, 0.0f};
    if (vidx >= p.k) return r;
    if constexpr (FMT == QM_AFFINE) {
        const int64_t ng = p.k >> p.gshift;
        const int64_t g = vidx >> p.gshift;
        r.s = sval(__ldg(reinterpret_cast<const uint16_t*>(p.scales) + grow * ng + g), p.sdt);
        r.b = sval(__ldg(reinterpret_cast<const uint16_t*>(p.biases) + grow * ng + g), p.sdt);
    } else if constexpr (FMT == QM_MXFP4) {
        r.s = e8m0_to_f32(__ldg(p.scales + grow * p.scale_row_bytes + vidx / 32));
    }
    return r;
}

// Q8_0 block B (0..7) of a raw chunk row as 16 bf16 pairs. Rows are 272
// bytes apart; block B starts 2B bytes past the 16-byte boundary at 32B, so
// three aligned 16-byte loads cover it (and end inside the row). A warp's
// lanes take consecutive rows, whose 16-byte pieces then fall in distinct
// bank groups: 272 is 17 sixteen-byte units.
template <int B>
QM_DEV void decode_q8_block(const uint8_t* raw, int row, uint32_t (&o)[16]) {
    const uint4* src = reinterpret_cast<const uint4*>(raw + row * 272 + 32 * B);
    uint32_t w[12];
#pragma unroll
    for (int q = 0; q < 3; ++q) {
        const uint4 v = src[q];
        w[4 * q] = v.x; w[4 * q + 1] = v.y; w[4 * q + 2] = v.z; w[4 * q + 3] = v.w;
    }
    constexpr int kD = B / 2, kDs = (B & 1) * 16;              // f16 scale: word, shift
    constexpr int kQ = (B + 1) / 2, kQs = ((B + 1) & 1) * 16;  // first code byte: word, shift
    const float d = f16_bits_to_f32((w[kD] >> kDs) & 0xFFFFu);
    const float2 neg = make_float2(-8388736.0f, -8388736.0f);  // -(2^23 + 128)
    const float2 d2 = make_float2(d, d);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        uint32_t u;
        if constexpr (kQs == 0) u = w[kQ + j];
        else u = __funnelshift_r(w[kQ + j], w[kQ + j + 1], kQs);
        u ^= 0x80808080u;  // q + 128 per byte
#pragma unroll
        for (int i = 0; i < 4; i += 2) {
            const float2 f = make_float2(__uint_as_float(prmt(u, 0x4B000000u, 0x7540 + i)),
                                         __uint_as_float(prmt(u, 0x4B000000u, 0x7541 + i)));
            const float2 v = mul2(add2(f, neg), d2);
            o[(4 * j + i) / 2] = bf2(v.x, v.y);
        }
    }
}

// GGUF MXFP4 block B (0..15) of a raw chunk row as 16 bf16 pairs. Rows are 272
// bytes apart; block B's 17 bytes start B bytes into the row's 16-byte unit B,
// so units B and B + 1 hold them (and end inside the row). Data byte j holds
// values j (low nibble) and j + 16: each byte's decoded pair is split between
// output pairs j/2 and 8 + j/2 as the bf16 pairs are formed.
template <int B>
QM_DEV void decode_mxb_block(const uint8_t* raw, int row, uint32_t (&o)[16]) {
    const uint4* src = reinterpret_cast<const uint4*>(raw + row * 272 + 16 * B);
    const uint4 u0 = src[0], u1 = src[1];
    const uint32_t w[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
    const float s = e8m0_to_f32((w[B / 4] >> (8 * (B % 4))) & 0xFFu);
    constexpr int kW = (B + 1) / 4, kS = 8 * ((B + 1) % 4);  // data byte 0: word, shift
    const float2 s2 = make_float2(s, s);
    float2 p[16];  // p[j] = (value j, value j + 16)
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        uint32_t dw;
        if constexpr (kS == 0) dw = w[kW + q];
        else dw = __funnelshift_r(w[kW + q], w[kW + q + 1], kS);
        uint32_t h[4];
        e2m1x8_to_f16x2(dw, h);
#pragma unroll
        for (int i = 0; i < 4; ++i) p[4 * q + i] = mul2(__half22float2(*reinterpret_cast<const __half2*>(&h[i])), s2);
    }
#pragma unroll
    for (int m = 0; m < 8; ++m) {
        o[m] = bf2(p[2 * m].x, p[2 * m + 1].x);
        o[8 + m] = bf2(p[2 * m].y, p[2 * m + 1].y);
    }
}

// The 32 values of one decoder thread's half row (values kk*64 + half*32 .. of
// the chunk) as 16 bf16 pairs, from the raw chunk in shared memory.
template <int FMT, int BITS, int GS>
QM_DEV void decode32(const uint8_t* raw, int row, int kk, int half, Sc sc, uint32_t (&o)[16]) {
    if constexpr (Raw<FMT, BITS>::GEN) {
        // BITS words of a little-endian code stream; codes may cross words
        const uint32_t* wp = reinterpret_cast<const uint32_t*>(raw + row * (16 * BITS) + (kk * 64 + half * 32) * BITS / 8);
        uint32_t w[BITS];
#pragma unroll
        for (int j = 0; j < BITS; ++j) w[j] = wp[j];
        const float2 neg = make_float2(-8388608.0f, -8388608.0f);
        const float2 s2 = make_float2(sc.s, sc.s), b2 = make_float2(sc.b, sc.b);
        auto code = [&](int i) {
            const int bit = i * BITS, q = bit >> 5, sh = bit & 31;
            uint32_t c = w[q] >> sh;
            if (sh + BITS > 32) c |= w[q + 1] << (32 - sh);
            return c & ((1u << BITS) - 1u);
        };
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
            const float2 f = make_float2(magic_f(code(i)), magic_f(code(i + 1)));
            const float2 v = fma2(add2(f, neg), s2, b2);  // exact code, then one rounding
            o[i / 2] = bf2(v.x, v.y);
        }
    } else if constexpr (FMT == QM_AFFINE) {
        const float2 neg = make_float2(-8388608.0f, -8388608.0f);
        const float2 s2 = make_float2(sc.s, sc.s), b2 = make_float2(sc.b, sc.b);
        constexpr int PER = 32 / BITS;       // codes per word
        constexpr int WORDS = 32 / PER;      // words per half row: 4 (4-bit) or 8 (8-bit)
        uint32_t ws[WORDS];
#pragma unroll
        for (int q = 0; q < WORDS / 4; ++q) {
            const uint4 w = *reinterpret_cast<const uint4*>(raw + sw128(row, (kk * 64 + half * 32) * BITS / 128 + q));
            ws[4 * q] = w.x; ws[4 * q + 1] = w.y; ws[4 * q + 2] = w.z; ws[4 * q + 3] = w.w;
        }
#pragma unroll
        for (int j = 0; j < WORDS; ++j)
#pragma unroll
            for (int i = 0; i < PER; i += 2) {
                float2 f;
                if constexpr (BITS == 4) {
                    f = make_float2(magic_f((ws[j] >> (4 * i)) & 15u), magic_f((ws[j] >> (4 * i + 4)) & 15u));
                } else {
                    f = make_float2(__uint_as_float(prmt(ws[j], 0x4B000000u, 0x7540 + i)),
                                    __uint_as_float(prmt(ws[j], 0x4B000000u, 0x7541 + i)));
                }
                const float2 v = fma2(add2(f, neg), s2, b2);  // exact code, then one rounding
                o[(j * PER + i) / 2] = bf2(v.x, v.y);
            }
    } else if constexpr (FMT == QM_Q4_K) {
        // sub-block j = 2 kk + half of the row's block: 32 quant bytes from byte
        // 16 + 32 kk, their low (half 0) or high (half 1) nibbles; value =
        // (d * sc) * q - dmin * m, exact products and one rounding
        const uint8_t* blk = raw + row * 144;
        const uint4 h = *reinterpret_cast<const uint4*>(blk);
        const int j = 2 * kk + half;
        auto sb = [&](int i) -> int {
            const uint32_t wd = i < 4 ? h.y : (i < 8 ? h.z : h.w);
            return static_cast<int>((wd >> (8 * (i & 3))) & 0xFFu);
        };
        const int sc = j < 4 ? (sb(j) & 63) : ((sb(4 + j) & 15) | ((sb(j - 4) >> 6) << 4));
        const int mn = j < 4 ? (sb(4 + j) & 63) : ((sb(4 + j) >> 4) | ((sb(j) >> 6) << 4));
        const float d1 = f16_bits_to_f32(h.x & 0xFFFFu) * static_cast<float>(sc);
        const float m1 = f16_bits_to_f32(h.x >> 16) * static_cast<float>(mn);
        const float2 d2 = make_float2(d1, d1), nm2 = make_float2(-m1, -m1);
        const float2 neg = make_float2(-8388608.0f, -8388608.0f);
        const int sh = half ? 4 : 0;
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            const uint4 v = *reinterpret_cast<const uint4*>(blk + 16 + 32 * kk + 16 * q);
            const uint32_t ws[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const uint32_t c = (ws[e] >> sh) & 0x0F0F0F0Fu;  // four values, one per byte
#pragma unroll
                for (int i = 0; i < 4; i += 2) {
                    const float2 f = make_float2(__uint_as_float(prmt(c, 0x4B000000u, 0x7540 + i)),
                                                 __uint_as_float(prmt(c, 0x4B000000u, 0x7541 + i)));
                    const float2 val = fma2(add2(f, neg), d2, nm2);
                    o[(16 * q + 4 * e + i) / 2] = bf2(val.x, val.y);
                }
            }
        }
    } else if constexpr (FMT == QM_MXFP4) {
        const uint4 w = *reinterpret_cast<const uint4*>(raw + sw128(row, kk * 2 + half));
        const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
        const float2 s2 = make_float2(sc.s, sc.s);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            uint32_t h2[4];
            e2m1x8_to_f16x2(ws[j], h2);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float2 v = mul2(__half22float2(*reinterpret_cast<const __half2*>(&h2[i])), s2);
                o[4 * j + i] = bf2(v.x, v.y);
            }
        }
    } else if constexpr (FMT == QM_MXFP4_BLOCKS) {  // block kk*2 + half of the chunk
        switch (2 * kk + half) {
            case 0: decode_mxb_block<0>(raw, row, o); break;
            case 1: decode_mxb_block<1>(raw, row, o); break;
            case 2: decode_mxb_block<2>(raw, row, o); break;
            case 3: decode_mxb_block<3>(raw, row, o); break;
            case 4: decode_mxb_block<4>(raw, row, o); break;
            case 5: decode_mxb_block<5>(raw, row, o); break;
            case 6: decode_mxb_block<6>(raw, row, o); break;
            case 7: decode_mxb_block<7>(raw, row, o); break;
            case 8: decode_mxb_block<8>(raw, row, o); break;
            case 9: decode_mxb_block<9>(raw, row, o); break;
            case 10: decode_mxb_block<10>(raw, row, o); break;
            case 11: decode_mxb_block<11>(raw, row, o); break;
            case 12: decode_mxb_block<12>(raw, row, o); break;
            case 13: decode_mxb_block<13>(raw, row, o); break;
            case 14: decode_mxb_block<14>(raw, row, o); break;
            default: decode_mxb_block<15>(raw, row, o); break;
        }
    } else {  // Q8_0: block kk*2 + half of the chunk (kk is a constant once the k loop unrolls)
        switch (2 * kk + half) {
            case 0: decode_q8_block<0>(raw, row, o); break;
            case 1: decode_q8_block<1>(raw, row, o); break;
            case 2: decode_q8_block<2>(raw, row, o); break;
            case 3: decode_q8_block<3>(raw, row, o); break;
            case 4: decode_q8_block<4>(raw, row, o); break;
            case 5: decode_q8_block<5>(raw, row, o); break;
            case 6: decode_q8_block<6>(raw, row, o); break;
            default: decode_q8_block<7>(raw, row, o); break;
        }
    }
}

// ---------------------------------------------------------------- kernel
namespace ts {
constexpr int BW = 128;                // weight rows per CTA
constexpr int NA = 4;                  // decoded weight stages in TMEM
constexpr int NXT = 4;                 // activation tiles in flight
// TMEM columns of a CTA: the accumulator [0, NTOK) (dual: two, at [0, 128)
// and [128, 256)), then NA weight stages of 32 columns; classic 128-token tiles
// hold half the SM's 512 columns, so two CTAs share an SM (one's epilogue and
// setup overlap the other's main loop)
constexpr uint32_t acol(int ntok, bool dual) { return ntok <= 128 && !dual ? 128u : 256u; }
constexpr uint32_t cols(int ntok, bool dual) { return ntok <= 128 && !dual ? 256u : 512u; }
}  // namespace ts

// Grouped mode, one warp: which expert's rows of x m-tile slot `mt` covers
// (s_grp: found, expert, first row, end row), bm rows to a tile.
static __device__ __noinline__ void tile_lookup(const Params& p, int mt, int bm, int lane, int* s_grp) {
    int before = 0;  // tiles of the experts already passed
    int found = 0, ge = 0, gm0 = 0, gend = 0;
    for (int e0 = 0; e0 < p.g_E; e0 += 32) {
        const int e = e0 + lane;
        int o0 = 0, cnt = 0;
        if (e < p.g_E) {
            o0 = __ldg(p.g_off + e);
            cnt = __ldg(p.g_off + e + 1) - o0;
        }
        const int nch = (cnt + bm - 1) / bm;
        int inc = nch;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int t = __shfl_up_sync(0xffffffffu, inc, o);
            if (lane >= o) inc += t;
        }
        const int lo = before + inc - nch;
        const bool mine = e < p.g_E && mt >= lo && mt < lo + nch;
        const uint32_t hit = __ballot_sync(0xffffffffu, mine);
        if (mine) {
            found = 1;
            ge = e;
            gm0 = o0 + (mt - lo) * bm;
            gend = o0 + cnt;
        }
        if (hit) {
            const int src = __ffs(hit) - 1;
            found = __shfl_sync(0xffffffffu, found, src);
            ge = __shfl_sync(0xffffffffu, ge, src);
            gm0 = __shfl_sync(0xffffffffu, gm0, src);
            gend = __shfl_sync(0xffffffffu, gend, src);
            break;
        }
        before += __shfl_sync(0xffffffffu, inc, 31);
    }
    if (lane == 0) { s_grp[0] = found; s_grp[1] = ge; s_grp[2] = gm0; s_grp[3] = gend; }
}

template <int FMT, int BITS, int GS, int NTOK, bool DUAL>
__global__ void __launch_bounds__(threads_for(DUAL), (NTOK <= 128 && !DUAL) ? 2 : 1)
    gemm_kernel(const __grid_constant__ Params p) {
    using R = Raw<FMT, BITS>;
    using namespace ts;
    constexpr uint32_t kAcol = acol(NTOK, DUAL), kCols = cols(NTOK, DUAL);
    constexpr bool kDual = DUAL;
    static_assert(!DUAL || NTOK == 128, "two pipes fit TMEM at 128 tokens");
    constexpr int kPipes = kDual ? 2 : 1;  // k-step parities with their own producer, issuer, accumulator
    static_assert(kAcol + 32 * NA <= kCols && kPipes * NTOK <= kAcol, "TMEM columns");
    constexpr uint32_t kXBytes = NTOK * BK * 2;  // activation tile per k step
    extern __shared__ __align__(1024) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int S = p.splitk;
    const uint32_t rank = S > 1 ? cluster_ctarank() : 0;
    const int tile = static_cast<int>(blockIdx.x) / S;
    const int mt = p.g_off ? tile / p.ntiles : tile % p.mtiles;
    const int nt = p.g_off ? tile % p.ntiles : tile / p.mtiles;
    int64_t m0 = static_cast<int64_t>(mt) * NTOK, mend = p.M;  // this tile's rows of x
    int64_t wrow0 = 0;                                          // first row of the tile's matrix
    const int64_t n0 = static_cast<int64_t>(nt) * BW;
    const int ks_n = p.ksteps;
    const int nchunks = (ks_n + R::SPR - 1) / R::SPR;
    // this CTA's chunks and k steps (all of them without a split); ring slots
    // and parities count from the first
    const int c_lo = static_cast<int>(rank) * p.cps, c_hi = min(nchunks, c_lo + p.cps);
    const int ks_lo = c_lo * R::SPR, ks_hi = min(ks_n, c_hi * R::SPR);

    uint64_t* bars = reinterpret_cast<uint64_t*>(smem);
    const uint32_t b0 = smem_u32(bars);
    auto x_full = [&](int i) { return b0 + 8 * i; };
    auto x_empty = [&](int i) { return b0 + 8 * (NXT + i); };
    auto a_full = [&](int i) { return b0 + 8 * (2 * NXT + i); };
    auto a_empty = [&](int i) { return b0 + 8 * (2 * NXT + NA + i); };
    auto r_full = [&](int i) { return b0 + 8 * (2 * NXT + 2 * NA + i); };
    auto r_empty = [&](int i) { return b0 + 8 * (2 * NXT + 2 * NA + NR + i); };
    constexpr int kB = 2 * NXT + 2 * NA + 2 * NR;
    const uint32_t done = b0 + 8 * kB;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + 8 * (kB + 1));
    volatile int& s_abort = *reinterpret_cast<volatile int*>(smem + 8 * (kB + 2));
    int* s_grp = reinterpret_cast<int*>(smem + 8 * (kB + 3));  // [4], below 1 KB

    if (threadIdx.x == 0) {
        s_abort = 0;
        for (int i = 0; i < NXT; ++i) { mbar_init(x_full(i), 1); mbar_init(x_empty(i), 1); }
        for (int i = 0; i < NA; ++i) { mbar_init(a_full(i), 4); mbar_init(a_empty(i), 1); }
        for (int i = 0; i < NR; ++i) { mbar_init(r_full(i), 1); mbar_init(r_empty(i), kDecWarps); }
        mbar_init(done, kPipes);
        fence_mbar_init();
        prefetch_tmap(&p.tm_x);
        prefetch_tmap(&p.tm_raw);
    }
    if (p.g_off) {
        if (warp == 0) {
            grid_dependency_wait();  // the routing offsets come from an earlier kernel
            tile_lookup(p, mt, NTOK, lane, s_grp);
        }
        __syncthreads();
        if (!s_grp[0]) return;  // a slot past the last tile: nothing allocated yet
        wrow0 = static_cast<int64_t>(s_grp[1]) * p.n;
        m0 = s_grp[2];
        mend = s_grp[3];
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), kCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    grid_launch_dependents();
    grid_dependency_wait();

    auto give_up = [&]() {
        atomicOr(&g_err_gemm, DEV_ERR_TIMEOUT);
        s_abort = 1;
    };

    // pipe of an activation producer (warps 10, 11) or MMA issuer (warps 1, 12)
    const int x_pipe = warp == 11 ? 1 : 0, mma_pipe = warp == 12 ? 1 : 0;
    if (warp == 0 && !kDual) {
        // ------------------------------------------------------------ producer (classic)
        if (lane == 0) {
            int last_x = -1, last_r = -1;  // local indices
            for (int ks = ks_lo; ks < ks_hi && !s_abort; ++ks) {
                const int li = ks - ks_lo;
                if (li % R::SPR == 0) {
                    const int rc = ks / R::SPR, lc = rc - c_lo, sr = lc % NR;
                    if (!mbar_wait(r_empty(sr), ((lc / NR) & 1) ^ 1)) { give_up(); break; }
                    mbar_expect_tx(r_full(sr), R::BYTES * BW);
                    tma_load_2d(smem_u32(smem + p.off_raw + sr * p.raw_stage_bytes), &p.tm_raw,
                                rc * R::BYTES / R::ELEM, static_cast<int32_t>(wrow0 + n0), r_full(sr));
                    mbar_arrive(r_full(sr));
                    last_r = lc;
                }
                const int sx = li % NXT;
                if (!mbar_wait(x_empty(sx), ((li / NXT) & 1) ^ 1)) { give_up(); break; }
                mbar_expect_tx(x_full(sx), kXBytes);
                tma_load_2d(smem_u32(smem + p.off_x + sx * kXBytes), &p.tm_x, ks * 128, static_cast<int32_t>(m0),
                            x_full(sx));
                mbar_arrive(x_full(sx));
                last_x = li;
            }
            if (s_abort) {  // let issued copies land before the CTA winds down
                for (int li = std::max(0, last_x - NXT + 1); li <= last_x; ++li)
                    (void)mbar_wait(x_full(li % NXT), (li / NXT) & 1);
                for (int lc = std::max(0, last_r - NR + 1); lc <= last_r; ++lc)
                    (void)mbar_wait(r_full(lc % NR), (lc / NR) & 1);
            }
        }
    } else if (warp == 0) {
        // ------------------------------------------------------------ raw chunk producer (dual)
        if (lane == 0) {
            int last_r = -1;  // local chunk index
            for (int rc = c_lo; rc < c_hi && !s_abort; ++rc) {
                const int lc = rc - c_lo, sr = lc % NR;
                if (!mbar_wait(r_empty(sr), ((lc / NR) & 1) ^ 1)) { give_up(); break; }
                mbar_expect_tx(r_full(sr), R::BYTES * BW);
                tma_load_2d(smem_u32(smem + p.off_raw + sr * p.raw_stage_bytes), &p.tm_raw,
                            rc * R::BYTES / R::ELEM, static_cast<int32_t>(wrow0 + n0), r_full(sr));
                mbar_arrive(r_full(sr));
                last_r = lc;
            }
            if (s_abort) {  // let issued copies land before the CTA winds down
                for (int lc = std::max(0, last_r - NR + 1); lc <= last_r; ++lc)
                    (void)mbar_wait(r_full(lc % NR), (lc / NR) & 1);
            }
        }
    } else if (kDual && (warp == 10 || warp == 11)) {
        // ------------------------------------------------------------ activation producers (dual)
        if (lane == 0) {
            int last_x = -1;  // local index
            for (int ks = ks_lo + x_pipe; ks < ks_hi && !s_abort; ks += kPipes) {
                const int li = ks - ks_lo, sx = li % NXT;
                if (!mbar_wait(x_empty(sx), ((li / NXT) & 1) ^ 1)) { give_up(); break; }
                mbar_expect_tx(x_full(sx), kXBytes);
                tma_load_2d(smem_u32(smem + p.off_x + sx * kXBytes), &p.tm_x, ks * 128, static_cast<int32_t>(m0),
                            x_full(sx));
                mbar_arrive(x_full(sx));
                last_x = li;
            }
            if (s_abort) {
                for (int li = std::max(x_pipe, last_x - NXT + kPipes); li <= last_x; li += kPipes)
                    (void)mbar_wait(x_full(li % NXT), (li / NXT) & 1);
            }
        }
    } else if (warp == 1 || (kDual && warp == 12)) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = umma_idesc_bf16(BW, NTOK);
            const uint32_t acc = tmem + static_cast<uint32_t>(mma_pipe * NTOK);
            for (int ks = ks_lo + mma_pipe; ks < ks_hi && !s_abort; ks += kPipes) {
                const int li = ks - ks_lo;
                const int sx = li % NXT, sa = li % NA;
                if (!mbar_wait(x_full(sx), (li / NXT) & 1) || !mbar_wait(a_full(sa), (li / NA) & 1)) {
                    give_up();
                    break;
                }
                tc_fence_after();
                const uint64_t bd = umma_desc_sw128(smem_u32(smem + p.off_x + sx * kXBytes));
                const uint32_t ad = tmem + kAcol + 32 * sa;
#pragma unroll
                for (int kk = 0; kk < BK / 16; ++kk)  // 16 values: 8 TMEM columns of A, 32 bytes of B
                    umma_f16_ts(acc, ad + 8 * kk, bd + 2 * kk, idesc, li >= kPipes || kk > 0);
                umma_commit(x_empty(sx));
                umma_commit(a_empty(sa));
            }
            umma_commit(done);  // also drains whatever was issued when abandoning
        }
    } else if (warp >= 2 && warp < 2 + kDecWarps) {
        // ------------------------------------------------------------ decoders
        const int grp = (warp - 2) >> 2;           // k steps ks with ks % 2 == grp
        const int quarter = warp & 3;              // this warp's TMEM lanes
        const int row = 32 * quarter + lane;
        const uint32_t lane_addr = static_cast<uint32_t>(32 * quarter) << 16;
        const int64_t grow = n0 + row;
        const bool rowok = grow < p.n;
        Sc cur[R::SPR][2], nxt[R::SPR][2];
        // a chunk holds an even number of k steps, so this thread decodes steps
        // kk with kk % 2 == grp of every chunk: only their scales are fetched
        static_assert(R::SPR % 2 == 0, "k steps per chunk");
        // affine groups of 64 or more inputs: both halves of a k step share one
        // group, whose scale and bias are fetched once (entry [kk][0])
        constexpr bool kOneGroup = FMT == QM_AFFINE && GS >= 64;
        constexpr int kHalves = kOneGroup ? 1 : 2;
        auto fetch = [&](int rc, Sc (&dst)[R::SPR][2]) {
#pragma unroll
            for (int kk = 0; kk < R::SPR; ++kk)
#pragma unroll
                for (int h = 0; h < kHalves; ++h)
                    dst[kk][h] = rowok && (kk & 1) == grp
                                     ? load_scale<FMT, BITS, GS>(p, wrow0 + grow,
                                                                 static_cast<int64_t>(rc) * R::RAWK + kk * BK + h * 32)
                                     : Sc{0.0f, 0.0f};
        };
        fetch(c_lo, cur);
        for (int rc = c_lo; rc < c_hi; ++rc) {
            if (rc + 1 < c_hi) fetch(rc + 1, nxt);
            const int lc = rc - c_lo, sr = lc % NR;
            bool live = !s_abort && mbar_wait(r_full(sr), (lc / NR) & 1);
            const uint8_t* raw = smem + p.off_raw + sr * p.raw_stage_bytes;
#pragma unroll
            for (int kk = 0; kk < R::SPR; ++kk) {
                const int ks = rc * R::SPR + kk, li = ks - ks_lo;
                if (ks >= ks_hi) break;
                if ((li & 1) != grp) continue;
                const int sa = li % NA;
                if (live && !mbar_wait(a_empty(sa), ((li / NA) & 1) ^ 1)) live = false;
                if (!live) {
                    if (lane == 0) give_up();
                    break;
                }
                uint32_t o0[16], o1[16];
                if (rowok && static_cast<int64_t>(ks) * BK < p.k) {
                    decode32<FMT, BITS, GS>(raw, row, kk, 0, cur[kk][0], o0);
                } else {
#pragma unroll
                    for (int i = 0; i < 16; ++i) o0[i] = 0u;
                }
                if (rowok && static_cast<int64_t>(ks) * BK + 32 < p.k) {
                    decode32<FMT, BITS, GS>(raw, row, kk, 1, cur[kk][kHalves - 1], o1);
                } else {
#pragma unroll
                    for (int i = 0; i < 16; ++i) o1[i] = 0u;
                }
                const uint32_t ta = tmem + lane_addr + kAcol + 32 * sa;
                tmem_st16(ta, o0);
                tmem_st16(ta + 16, o1);
                tmem_wait_st();
                tc_fence_before();  // the MMA reads the stage after the barrier
                __syncwarp();
                if (lane == 0) mbar_arrive(a_full(sa));
            }
            __syncwarp();
            if (lane == 0 && live) mbar_arrive(r_empty(sr));
            if (!live) break;
#pragma unroll
            for (int kk = 0; kk < R::SPR; ++kk) {
                cur[kk][0] = nxt[kk][0];
                if constexpr (kHalves == 2) cur[kk][1] = nxt[kk][1];
            }
        }
        // ------------------------------------------------------------ epilogue
        const bool ok = mbar_wait(done, 0);
        if (!ok && lane == 0) give_up();
        tc_fence_after();
        // Each 32 x 32 block (this warp's rows x 32 tokens) turns round through
        // shared memory (the activation tiles are free now): lane pairs swap
        // values so each thread holds two adjacent rows of one token, rows are
        // written token-major (80-byte pitch: conflict-free both ways), then
        // lane t stores token t's 32 rows as four 16-byte pieces.
        const int part = grp;  // token columns [part * NTOK / 2, (part + 1) * NTOK / 2)
        uint8_t* stage = smem + p.off_x + (warp - 2) * (32 * 80);
        const int64_t row0 = n0 + 32 * quarter;  // this warp's first weight row
        const bool vec = (p.n & 7) == 0 && row0 + 32 <= p.n;
        const int odd = lane & 1;
        // tokens col .. col + 31 of this warp's 32 rows (r[c]: token col + c) to y
        auto store32 = [&](const uint32_t (&r)[32], int col) {
#pragma unroll
            for (int c = 0; c < 32; c += 2) {
                const float lo = __uint_as_float(r[c]), hi = __uint_as_float(r[c + 1]);
                const float got = __shfl_xor_sync(0xffffffffu, odd ? lo : hi, 1);
                const uint32_t pair = odd ? bf2(got, hi) : bf2(lo, got);  // rows (2i, 2i + 1) of token c + odd
                *reinterpret_cast<uint32_t*>(stage + (c + odd) * 80 + (lane >> 1) * 4) = pair;
            }
            __syncwarp();
            const int64_t m = m0 + col + lane;
            if (m < mend) {
                const int64_t ym = p.g_off ? static_cast<int64_t>(__ldg(p.g_perm + m)) : m;
                uint16_t* yr = p.y + ym * p.n + row0;
                const uint8_t* src = stage + lane * 80;
                if (vec) {
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        reinterpret_cast<uint4*>(yr)[q] = *reinterpret_cast<const uint4*>(src + 16 * q);
                } else {
                    for (int i = 0; i < 32 && row0 + i < p.n; ++i)
                        yr[i] = reinterpret_cast<const uint16_t*>(src)[i];
                }
            }
            __syncwarp();
        };
        // this warp's rows for tokens col .. col + 31: the accumulator, or the
        // sum of the two (the odd pipe's holds nothing when the CTA has one k step)
        const bool two = kDual && ks_hi - ks_lo >= 2;
        auto load_acc = [&](int col, uint32_t (&r)[32]) {
            tmem_ld32(tmem + lane_addr + col, r);
            if (two) {
                uint32_t r2[32];
                tmem_ld32(tmem + lane_addr + NTOK + col, r2);
                tmem_wait_ld();
#pragma unroll
                for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) + __uint_as_float(r2[i]));
            } else {
                tmem_wait_ld();
            }
        };
        if (S == 1) {
#pragma unroll 1
            for (int j = 0; j < NTOK / 64; ++j) {
                const int col = part * (NTOK / 2) + 32 * j;
                uint32_t r[32];
                load_acc(col, r);
                if (!ok || s_abort) continue;
                store32(r, col);
            }
        } else {
            // Split k. The tokens are cut into S slices of NTOK / S; CTA q adds
            // slice q. Every CTA puts its partial sums for slice q into CTA q's
            // receive area at [its rank][row][token] (pitch slice + 4 floats:
            // 16-byte rows that land in distinct bank groups), then, after the
            // cluster barrier, each CTA adds its S partials in rank order.
            const int slice = NTOK / S;
            const int pitch = slice + 4;
            const int row = 32 * quarter + lane;
            const uint32_t recv = smem_u32(smem + p.off_recv);
#pragma unroll 1
            for (int j = 0; j < NTOK / 64; ++j) {
                const int col = part * (NTOK / 2) + 32 * j;
                uint32_t r[32];
                load_acc(col, r);
                const int q = col / slice, cc = col - q * slice;
                const uint32_t dst = map_shared_rank(recv, static_cast<uint32_t>(q)) +
                                     4u * static_cast<uint32_t>((static_cast<int>(rank) * BW + row) * pitch + cc);
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    st_shared_cluster_v4(dst + 16 * i, r[4 * i], r[4 * i + 1], r[4 * i + 2], r[4 * i + 3]);
            }
        }
    }
    if (S > 1) {
        __syncthreads();
        cluster_sync();  // every partial sum has arrived; nothing is written remotely after this
        if (warp >= 2 && warp < 2 + kDecWarps) {
            const int quarter = warp & 3, part = (warp - 2) >> 2;
            const int slice = NTOK / S, pitch = slice + 4;
            const int row = 32 * quarter + lane;
            const float* recv = reinterpret_cast<const float*>(smem + p.off_recv);
            const int64_t row0 = n0 + 32 * quarter;
            const bool vec = (p.n & 7) == 0 && row0 + 32 <= p.n;
            const int odd = lane & 1;
            uint8_t* stage = smem + p.off_x + (warp - 2) * (32 * 80);
            // this warp's tokens of the slice: 32 when the slice has 64, else 16 (slice 32)
            const int cols = slice / 2;
            const int c0 = part * cols;
            const bool live = !s_abort;
            uint32_t r[32];
#pragma unroll
            for (int c = 0; c < 32; ++c) {
                float v = 0.0f;
                if (c < cols) {
                    for (int q = 0; q < S; ++q) v += recv[(q * BW + row) * pitch + c0 + c];
                }
                r[c] = __float_as_uint(v);
            }
            if (live) {
                // the store's tokens past `cols` belong to the next warp's part: keep them out
                const int64_t keep_end = mend;
                const int64_t first = m0 + static_cast<int64_t>(rank) * slice + c0;
#pragma unroll
                for (int c = 0; c < 32; c += 2) {
                    const float lo = __uint_as_float(r[c]), hi = __uint_as_float(r[c + 1]);
                    const float got = __shfl_xor_sync(0xffffffffu, odd ? lo : hi, 1);
                    const uint32_t pair = odd ? bf2(got, hi) : bf2(lo, got);
                    *reinterpret_cast<uint32_t*>(stage + (c + odd) * 80 + (lane >> 1) * 4) = pair;
                }
                __syncwarp();
                const int64_t m = first + lane;
                if (lane < cols && m < keep_end) {
                    uint16_t* yr = p.y + m * p.n + row0;
                    const uint8_t* src = stage + lane * 80;
                    if (vec) {
#pragma unroll
                        for (int qq = 0; qq < 4; ++qq)
                            reinterpret_cast<uint4*>(yr)[qq] = *reinterpret_cast<const uint4*>(src + 16 * qq);
                    } else {
                        for (int i = 0; i < 32 && row0 + i < p.n; ++i)
                            yr[i] = reinterpret_cast<const uint16_t*>(src)[i];
                    }
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kCols);
    }
}

template <int FMT, int BITS, int GS, int NTOK, bool DUAL>
static cudaError_t launch_t(Params& p, const WDesc& w, const void* x, cudaStream_t st) {
    using R = Raw<FMT, BITS>;
    p.mtiles = p.g_off ? static_cast<int>(std::min<int64_t>(p.M, p.M / NTOK + p.g_E))  // sum of ceil(count / NTOK)
                       : static_cast<int>((p.M + NTOK - 1) / NTOK);
    p.off_x = 1024;
    p.off_raw = p.off_x + ts::NXT * NTOK * BK * 2;
    p.raw_stage_bytes = (R::BYTES * ts::BW + 16 + 1023) / 1024 * 1024;  // 16 spare bytes after each slot
    p.off_recv = p.off_raw + NR * p.raw_stage_bytes;
    const int64_t ntiles = (w.n + ts::BW - 1) / ts::BW;
    const int nchunks = (p.ksteps + R::SPR - 1) / R::SPR;
    // split k while the tiles alone leave most SMs idle: 128-token tiles only
    // (slices of at least 32 tokens), at least two chunks per CTA
    int S = 1;
    if (!p.g_off && NTOK == 128) {
        const int64_t tiles = p.mtiles * ntiles;
        while (S < 4 && tiles * S * 2 <= num_sms() && nchunks >= 2 * S * 2) S *= 2;
    }
    p.splitk = S;
    p.cps = (nchunks + S - 1) / S;
    const size_t recv_bytes = S > 1 ? static_cast<size_t>(S) * ts::BW * (NTOK / S + 4) * 4 : 0;
    const size_t smem = p.off_recv + recv_bytes;
    if (!make_tmap_2d(&p.tm_x, x, static_cast<uint64_t>(w.k) * 2, p.M, static_cast<uint64_t>(w.k) * 2, 128, NTOK, true))
        return cudaErrorNotSupported;
    if (!make_tmap_2d(&p.tm_raw, w.codes, w.code_row_bytes, w.rows, w.code_row_bytes, R::BYTES, ts::BW, R::SW,
                      R::ELEM))
        return cudaErrorNotSupported;
    auto kern = gemm_kernel<FMT, BITS, GS, NTOK, DUAL>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    p.ntiles = static_cast<int>(ntiles);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(p.mtiles * ntiles * S));
    cfg.blockDim = dim3(threads_for(DUAL));
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attrs[2];
    attrs[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attrs[0].val.programmaticStreamSerializationAllowed = 1;
    int na = 1;
    if (S > 1) {
        attrs[1].id = cudaLaunchAttributeClusterDimension;
        attrs[1].val.clusterDim.x = S;
        attrs[1].val.clusterDim.y = 1;
        attrs[1].val.clusterDim.z = 1;
        na = 2;
    }
    cfg.attrs = attrs;
    cfg.numAttrs = na;
    return cudaLaunchKernelEx(&cfg, kern, p);
}


// The kernel instantiation for the weight's format: l.run<FMT, BITS, GS>().
// The group size reaches the kernel as p.gshift; the 4- and 8-bit kernels
// keep their per-size instantiations, the other widths share one.
template <class L>
static cudaError_t by_format(Params& p, const WDesc& w, const L& l) {
    p.gshift = 0;
    while ((1 << p.gshift) < w.gs) ++p.gshift;
    if (w.fmt == QM_AFFINE && w.bits == 2) return l.template run<QM_AFFINE, 2, 0>();
    if (w.fmt == QM_AFFINE && w.bits == 3) return l.template run<QM_AFFINE, 3, 0>();
    if (w.fmt == QM_AFFINE && w.bits == 5) return l.template run<QM_AFFINE, 5, 0>();
    if (w.fmt == QM_AFFINE && w.bits == 6) return l.template run<QM_AFFINE, 6, 0>();
    if (w.fmt == QM_AFFINE && w.bits == 4 && w.gs == 32) return l.template run<QM_AFFINE, 4, 32>();
    if (w.fmt == QM_AFFINE && w.bits == 4 && w.gs == 64) return l.template run<QM_AFFINE, 4, 64>();
    if (w.fmt == QM_AFFINE && w.bits == 4 && w.gs == 128) return l.template run<QM_AFFINE, 4, 128>();
    if (w.fmt == QM_AFFINE && w.bits == 8 && w.gs == 32) return l.template run<QM_AFFINE, 8, 32>();
    if (w.fmt == QM_AFFINE && w.bits == 8 && w.gs == 64) return l.template run<QM_AFFINE, 8, 64>();
    if (w.fmt == QM_AFFINE && w.bits == 8 && w.gs == 128) return l.template run<QM_AFFINE, 8, 128>();
    if (w.fmt == QM_Q8_0) return l.template run<QM_Q8_0, 8, 32>();
    if (w.fmt == QM_MXFP4) return l.template run<QM_MXFP4, 4, 32>();
    if (w.fmt == QM_Q4_K) return l.template run<QM_Q4_K, 4, 0>();
    if (w.fmt == QM_MXFP4_BLOCKS) return l.template run<QM_MXFP4_BLOCKS, 4, 32>();
    return cudaErrorInvalidValue;
}

// Grouped products with 128-token tiles (classic layout, two CTAs to an SM),
// instantiated in qm_gemm_grouped.cu so that they compile beside the rest.
cudaError_t dispatch_grouped_narrow(Params& p, const WDesc& w, const void* x, cudaStream_t st);
uint32_t grouped_read_clear_flag();

}  // namespace gemm
}  // namespace qm
