// qm_gemvr.cu -- decode product y[M, n] = x[M, k] * W^T for 1 <= M <= 8 tokens
// over MLX affine 4-bit weights, with the weight tiles in registers and the
// products on mma.sync tensor-core instructions: no shared-memory staging of
// weights, no activation prologue, no pipeline barriers. It serves decode
// steps of 2..8 tokens, where a chain of dependent launches is bound by each
// launch's latency.
//
// The product is the one "Nx_quant (raven-ml.dev API docs)", section
// "Products", val apply, defines (x times the weight's float32 values, summed
// at float32, rounded once to x's dtype); the affine value is code * scale +
// bias ("GPTQModel wiki: MLX Apple Silicon", "Concepts: method, checkpoint,
// runtime, and tensor layout"), codes little-endian in uint32 words ("Packed
// layouts and exact transcoding").
//
// Design (one GB300: 152 SMs):
//  * A warp owns a tile of 16 weight rows and a k range; KS warps of a CTA
//    split one tile's k and add their partial sums in warp order through
//    shared memory (deterministic).
//  * mma.sync m16n8k16 with bf16 operands and float32 accumulators: rows of W
//    on the M side, the (up to 8) tokens on the N side. A code c becomes the
//    bf16 value 128 + c, exact, with one mask-and-OR per pair of codes; the
//    activations enter as the bf16 values they are. Each 16-input MMA lies
//    inside one group (lane t takes words [t*V, t*V + V) of every group, V =
//    group_size / 32), so a group's sum is one accumulator.
//  * A second MMA against a matrix of ones gives each token's sum of x over
//    the group in the same fragment layout, so a group adds
//    s * sum((128 + c) x) + (b - 128 s) * sum(x) to each output: two fused
//    multiply-adds. The offset's cancellation costs a relative 2^-17 or so of
//    the largest term, far inside the product bound.
//  * Weights marked static are read before the kernel waits on the previous
//    one, with streaming loads (L1 not filled, L2 evict-first); every step
//    loads the next step's codes and scales before working on its own.
//  * A warp whose k range holds a scale or bias of magnitude 2^100 or more,
//    or whose partial sum for an output is not finite, recomputes that output
//    over its range element by element (each value decoded at float32 as
//    dequant decodes it, times its activation, in ascending k): the
//    infinities and NaNs IEEE arithmetic gives a per-element sum.
#include <cuda_runtime.h>

#include <algorithm>

#include "qm_device.cuh"
#include "qm_internal.h"

namespace qm {

namespace gr {

constexpr int kWarps = 4;       // warps per CTA where ks <= 2 (4 / ks tiles each)
constexpr int kMaxWarps = 12;   // the most warps a tile's k split takes (a CTA of ks warps)
constexpr int kStep = 256;      // inputs per step of a warp
constexpr int kMaxParts = 8;    // weights per launch (the C ABI's QM_MAX_MANY)
constexpr uint32_t kBf16Magic = 0x43004300u;  // bf16 pair (128, 128)
constexpr uint32_t kOnes = 0x3F803F80u;       // bf16 pair (1, 1)

struct Part {
    const uint8_t* codes;
    const uint16_t* scales;
    const uint16_t* biases;
    uint16_t* y;
    int64_t n;
};

struct Args {
    Part part[kMaxParts];
    int tstart[kMaxParts + 1];  // first 16-row tile of each part; tstart[nparts]: all tiles
    int nparts;
    const uint16_t* x;          // [M, k] bf16
    int M;
    int64_t k;
    int64_t code_row_bytes, scale_row_bytes;
    int sdt;                    // scale dtype (QM_BF16 or QM_F16)
    int ks;                     // warps splitting one tile's k (1 .. 12)
    int tpc;                    // tiles per CTA (4 / ks where ks <= 2, else 1)
    int nsteps;                 // steps of kStep inputs in one warp's k range
    int static_w;
};

QM_DEV void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

QM_DEV float sval(uint32_t h, int sdt) { return sdt == QM_F16 ? f16_bits_to_f32(h) : bf16_bits_to_f32(h); }

// One step of one lane: for rows g and g + 8 of the tile, the 8 code words it
// owns (two rows x kStep / GS groups x V words) and the step's scales and
// biases of those rows (kStep / GS values each, packed in 32-bit words).
template <int GS>
struct Step {
    static constexpr int G = kStep / GS;  // groups per step
    static constexpr int V = GS / 32;     // words per lane per group per row
    static constexpr int SW = (G + 1) / 2;  // 32-bit words of G 16-bit values
    uint32_t w0[G * V], w8[G * V];        // codes of rows g and g + 8
    uint32_t s0[SW], s8[SW], b0[SW], b8[SW];
};

// The 16-bit value i of a packed run.
template <int N>
QM_DEV uint32_t half_at(const uint32_t (&v)[N], int i) {
    return (v[i >> 1] >> (16 * (i & 1))) & 0xFFFFu;
}

// Loads one step: group j's words of this lane are [t*V, t*V + V) of the
// group's GS/8 words, i.e. bytes (j * GS + t * 8V) / 2 ... of the step.
template <int GS>
QM_DEV void load_step(const Args& a, const Part& P, int64_t r0, int64_t i0, int t, uint64_t pol, Step<GS>& S) {
    using St = Step<GS>;
    constexpr int G = St::G, V = St::V;
    const int64_t rg = r0, r8 = r0 + 8;
    const bool okg = rg < P.n, ok8 = r8 < P.n;
    const uint8_t* cg = P.codes + rg * a.code_row_bytes + i0 / 2;
    const uint8_t* c8 = P.codes + r8 * a.code_row_bytes + i0 / 2;
#pragma unroll
    for (int j = 0; j < G; ++j) {
        const int off = (j * GS) / 2 + t * 4 * V;  // bytes into the step's codes of a row
        if constexpr (V == 1) {
            S.w0[j] = okg ? ldg_stream(reinterpret_cast<const uint32_t*>(cg + off), pol) : 0u;
            S.w8[j] = ok8 ? ldg_stream(reinterpret_cast<const uint32_t*>(c8 + off), pol) : 0u;
        } else if constexpr (V == 2) {
            const uint2 z = make_uint2(0u, 0u);
            const uint2 u = okg ? ldg_stream(reinterpret_cast<const uint2*>(cg + off), pol) : z;
            const uint2 v = ok8 ? ldg_stream(reinterpret_cast<const uint2*>(c8 + off), pol) : z;
            S.w0[2 * j] = u.x; S.w0[2 * j + 1] = u.y;
            S.w8[2 * j] = v.x; S.w8[2 * j + 1] = v.y;
        } else {
            const uint4 z = make_uint4(0u, 0u, 0u, 0u);
            const uint4 u = okg ? ldg_stream(reinterpret_cast<const uint4*>(cg + off), pol) : z;
            const uint4 v = ok8 ? ldg_stream(reinterpret_cast<const uint4*>(c8 + off), pol) : z;
            S.w0[4 * j] = u.x; S.w0[4 * j + 1] = u.y; S.w0[4 * j + 2] = u.z; S.w0[4 * j + 3] = u.w;
            S.w8[4 * j] = v.x; S.w8[4 * j + 1] = v.y; S.w8[4 * j + 2] = v.z; S.w8[4 * j + 3] = v.w;
        }
    }
    // the step's G scales (and biases) of a row: G 16-bit values, 2G bytes
    // (8-byte aligned: the kernel runs only where k is a multiple of 4 GS)
    const int64_t so = i0 / GS;  // first group of the step
    const uint16_t* sg = P.scales + rg * (a.scale_row_bytes / 2) + so;
    const uint16_t* s8 = P.scales + r8 * (a.scale_row_bytes / 2) + so;
    const uint16_t* bg = P.biases + rg * (a.scale_row_bytes / 2) + so;
    const uint16_t* b8 = P.biases + r8 * (a.scale_row_bytes / 2) + so;
    if constexpr (G == 8) {
        const uint4 z = make_uint4(0u, 0u, 0u, 0u);
        uint4 q;
        q = okg ? ldg_stream(reinterpret_cast<const uint4*>(sg), pol) : z;
        S.s0[0] = q.x; S.s0[1] = q.y; S.s0[2] = q.z; S.s0[3] = q.w;
        q = ok8 ? ldg_stream(reinterpret_cast<const uint4*>(s8), pol) : z;
        S.s8[0] = q.x; S.s8[1] = q.y; S.s8[2] = q.z; S.s8[3] = q.w;
        q = okg ? ldg_stream(reinterpret_cast<const uint4*>(bg), pol) : z;
        S.b0[0] = q.x; S.b0[1] = q.y; S.b0[2] = q.z; S.b0[3] = q.w;
        q = ok8 ? ldg_stream(reinterpret_cast<const uint4*>(b8), pol) : z;
        S.b8[0] = q.x; S.b8[1] = q.y; S.b8[2] = q.z; S.b8[3] = q.w;
    } else if constexpr (G == 4) {
        const uint2 z = make_uint2(0u, 0u);
        uint2 q;
        q = okg ? ldg_stream(reinterpret_cast<const uint2*>(sg), pol) : z;
        S.s0[0] = q.x; S.s0[1] = q.y;
        q = ok8 ? ldg_stream(reinterpret_cast<const uint2*>(s8), pol) : z;
        S.s8[0] = q.x; S.s8[1] = q.y;
        q = okg ? ldg_stream(reinterpret_cast<const uint2*>(bg), pol) : z;
        S.b0[0] = q.x; S.b0[1] = q.y;
        q = ok8 ? ldg_stream(reinterpret_cast<const uint2*>(b8), pol) : z;
        S.b8[0] = q.x; S.b8[1] = q.y;
    } else {  // G == 2
        S.s0[0] = okg ? ldg_stream(reinterpret_cast<const uint32_t*>(sg), pol) : 0u;
        S.s8[0] = ok8 ? ldg_stream(reinterpret_cast<const uint32_t*>(s8), pol) : 0u;
        S.b0[0] = okg ? ldg_stream(reinterpret_cast<const uint32_t*>(bg), pol) : 0u;
        S.b8[0] = ok8 ? ldg_stream(reinterpret_cast<const uint32_t*>(b8), pol) : 0u;
    }
}

// Whether a scale or bias of the step may carry a group's terms past float32's
// range before they cancel (magnitude 2^100 or more; f16 values never do).
template <int GS>
QM_DEV bool step_big(const Step<GS>& S, int sdt) {
    if (sdt == QM_F16) return false;
    uint32_t m = 0u;
#pragma unroll
    for (int i = 0; i < Step<GS>::SW; ++i)
        m = max(m, max(__vmaxu2(S.s0[i] & 0x7FFF7FFFu, S.s8[i] & 0x7FFF7FFFu),
                       __vmaxu2(S.b0[i] & 0x7FFF7FFFu, S.b8[i] & 0x7FFF7FFFu)));
    m = max(m & 0xFFFFu, m >> 16);
    return m >= 0x7180u;  // bf16 2^100
}

// The step's activations of token g for this lane: for group j, its 8V inputs
// [j*GS + 8tV, j*GS + 8tV + 8V) as 4V words of bf16 pairs (zeros for tokens
// past M, or past k).
template <int GS>
QM_DEV void load_x(const Args& a, int g, int64_t i0, int t, uint32_t (&xw)[Step<GS>::G * 4 * Step<GS>::V]) {
    constexpr int G = Step<GS>::G, V = Step<GS>::V;
    const bool ok = g < a.M;
    const uint16_t* xr = a.x + static_cast<int64_t>(ok ? g : 0) * a.k + i0;
#pragma unroll
    for (int j = 0; j < G; ++j)
#pragma unroll
        for (int q = 0; q < V; ++q) {
            const uint4 v = ok ? __ldca(reinterpret_cast<const uint4*>(xr + j * GS + 8 * (t * V + q)))
                               : make_uint4(0u, 0u, 0u, 0u);
            uint32_t* d = xw + 4 * (j * V + q);
            d[0] = v.x; d[1] = v.y; d[2] = v.z; d[3] = v.w;
        }
}

// Row `row`'s (or token tok's) exact sum over inputs [i0, i1) of x * value,
// each value decoded at float32 (fmaf(code, scale, bias)), in ascending k.
static __device__ __noinline__ float exact_sum(const Args& a, const Part& P, int64_t row, int tok, int64_t i0,
                                               int64_t i1, int gshift) {
    float acc = 0.0f;
    const uint8_t* rp = P.codes + row * a.code_row_bytes;
    const uint16_t* xr = a.x + static_cast<int64_t>(tok) * a.k;
#pragma unroll 1
    for (int64_t i = i0; i < i1; ++i) {
        const uint32_t byte = __ldg(rp + i / 2);
        const uint32_t c = (i & 1) ? (byte >> 4) : (byte & 15u);
        const int64_t gi = row * (a.scale_row_bytes / 2) + (i >> gshift);
        const float v = fmaf(static_cast<float>(c), sval(__ldg(P.scales + gi), a.sdt), sval(__ldg(P.biases + gi), a.sdt));
        acc = fmaf(bf16_bits_to_f32(__ldca(xr + i)), v, acc);
    }
    return acc;
}

template <int GS>
__global__ void __launch_bounds__(kMaxWarps * 32) gemvr_kernel(const __grid_constant__ Args a) {
    using St = Step<GS>;
    constexpr int G = St::G, V = St::V;
    constexpr int GSHIFT = GS == 32 ? 5 : (GS == 64 ? 6 : 7);
    __shared__ float red[kMaxWarps][32][4];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t = lane & 3;
    const int ks = a.ks, tpc = a.tpc;   // tiles per CTA
    const int slot = warp / ks, kpart = warp % ks;
    const int ntiles = a.tstart[a.nparts];
    const int64_t krange = static_cast<int64_t>(a.nsteps) * kStep;  // k / ks
    const int64_t kbase = kpart * krange;
    const uint64_t pol = l2_evict_first_policy();
    // the weight holding tile tl, and the tile's first row within it
    auto locate = [&](int tl, int& pi, int64_t& r0) {
        pi = 0;
        #pragma unroll 1
        while (pi + 1 < a.nparts && tl >= a.tstart[pi + 1]) ++pi;
        r0 = static_cast<int64_t>(tl - a.tstart[pi]) * 16;
    };
    // CTA c takes tile groups c, c + gridDim.x, ...; group q holds tiles
    // [q*tpc, q*tpc + tpc), this warp the one at its slot
    const int tg_stride = static_cast<int>(gridDim.x) * tpc;
    int tl = static_cast<int>(blockIdx.x) * tpc + slot;
    int cpi = 0;
    int64_t cr0 = 0;
    St cur, nxt;
    if (tl < ntiles) locate(tl, cpi, cr0);
    if (a.static_w) {  // the weights are not written by the previous kernel: read them first
        if (tl < ntiles) load_step<GS>(a, a.part[cpi], cr0 + g, kbase, t, pol, cur);
        grid_dependency_wait();
    } else {
        grid_dependency_wait();
        if (tl < ntiles) load_step<GS>(a, a.part[cpi], cr0 + g, kbase, t, pol, cur);
    }
    grid_launch_dependents();  // one kernel waits ahead: it has this one's run to read its weights
    // every warp of the CTA runs the same number of tile groups (a barrier each when ks > 1)
    const int ngroups = (ntiles - static_cast<int>(blockIdx.x) * tpc + tg_stride - 1) / tg_stride;
    #pragma unroll 1
    for (int q = 0; q < ngroups; ++q) {
        const bool live = tl < ntiles;
        const int ntl = tl + tg_stride;
        const bool next_live = ntl < ntiles;
        int npi = cpi;
        int64_t nr0 = cr0;
        if (next_live) locate(ntl, npi, nr0);
        const Part& P = a.part[cpi];
        float y[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        bool big = false;
        #pragma unroll 1
        for (int s = 0; live && s < a.nsteps; ++s) {
            const int64_t i0 = kbase + static_cast<int64_t>(s) * kStep;
            // the next step: of this tile, or the first of the warp's next tile
            const bool last = s + 1 == a.nsteps;
            const bool have_next = !last || next_live;
            if (have_next)
                load_step<GS>(a, a.part[last ? npi : cpi], (last ? nr0 : cr0) + g, last ? kbase : i0 + kStep, t, pol,
                              nxt);
            uint32_t xw[G * 4 * V];
            load_x<GS>(a, g, i0, t, xw);
            big = big || step_big<GS>(cur, a.sdt);
#pragma unroll
            for (int j = 0; j < G; ++j) {
                float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
                float xs[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
                for (int v = 0; v < V; ++v) {
                    const uint32_t c0 = cur.w0[j * V + v], c8 = cur.w8[j * V + v];
                    const uint32_t* xq = xw + 4 * (j * V + v);  // the word's 8 inputs as 4 bf16 pairs
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        // codes (2h, 2h+4) and (2h+1, 2h+5) of the word as bf16 128 + c
                        const uint32_t sh = 8u * h;
                        const uint32_t a0 = ((c0 >> sh) & 0x000F000Fu) | kBf16Magic;
                        const uint32_t a2 = ((c0 >> (sh + 4)) & 0x000F000Fu) | kBf16Magic;
                        const uint32_t a1 = ((c8 >> sh) & 0x000F000Fu) | kBf16Magic;
                        const uint32_t a3 = ((c8 >> (sh + 4)) & 0x000F000Fu) | kBf16Magic;
                        // the same inputs' activations: (x[2h], x[2h+4]) and (x[2h+1], x[2h+5])
                        const uint32_t b0 = prmt(xq[h], xq[h + 2], 0x5410);
                        const uint32_t b1 = prmt(xq[h], xq[h + 2], 0x7632);
                        mma_bf16(acc, a0, a1, a2, a3, b0, b1);
                        mma_bf16(xs, kOnes, kOnes, kOnes, kOnes, b0, b1);
                    }
                }
                // y += s * acc + (b - 128 s) * sum(x): rows g (acc 0, 1) and g + 8 (acc 2, 3),
                // tokens 2t (acc 0, 2) and 2t + 1 (acc 1, 3); xs[0] and xs[1] are the two
                // tokens' sums of x over the group
                const float sg = sval(half_at(cur.s0, j), a.sdt), s8 = sval(half_at(cur.s8, j), a.sdt);
                const float bg = fmaf(-128.0f, sg, sval(half_at(cur.b0, j), a.sdt));
                const float b8 = fmaf(-128.0f, s8, sval(half_at(cur.b8, j), a.sdt));
                y[0] = fmaf(sg, acc[0], fmaf(bg, xs[0], y[0]));
                y[1] = fmaf(sg, acc[1], fmaf(bg, xs[1], y[1]));
                y[2] = fmaf(s8, acc[2], fmaf(b8, xs[0], y[2]));
                y[3] = fmaf(s8, acc[3], fmaf(b8, xs[1], y[3]));
            }
            if (have_next) cur = nxt;
        }
        // this lane's outputs: (row cr0 + g + 8*(i/2), token 2t + i%2); a big
        // scale in the range, or a sum that is not finite, is summed per element
        if (live) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int64_t row = cr0 + g + ((i & 2) ? 8 : 0);
                const int tok = 2 * t + (i & 1);
                if ((big || !isfinite(y[i])) && row < P.n && tok < a.M)
                    y[i] = exact_sum(a, P, row, tok, kbase, kbase + krange, GSHIFT);
            }
        }
        auto store = [&](const float (&v)[4]) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int64_t row = cr0 + g + ((i & 2) ? 8 : 0);
                const int tok = 2 * t + (i & 1);
                if (row < P.n && tok < a.M) {
                    __nv_bfloat16 bv = __float2bfloat16_rn(v[i]);
                    P.y[static_cast<int64_t>(tok) * P.n + row] = *reinterpret_cast<uint16_t*>(&bv);
                }
            }
        };
        if (ks == 1) {
            if (live) store(y);
        } else {
            // the tile's ks partial sums, added in warp order by its first warp
#pragma unroll
            for (int i = 0; i < 4; ++i) red[warp][lane][i] = y[i];
            __syncthreads();
            if (live && kpart == 0) {
                float v[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    v[i] = red[warp][lane][i];
                    #pragma unroll 1
                    for (int w = 1; w < ks; ++w) v[i] += red[warp + w][lane][i];
                }
                store(v);
            }
            __syncthreads();  // red is rewritten by the next tile group
        }
        tl = ntl;
        cpi = npi;
        cr0 = nr0;
    }
}

template <int GS>
static cudaError_t launch_t(const Args& a, cudaStream_t st) {
    const int wpc = a.ks * a.tpc;  // warps per CTA
    const int64_t ntiles = a.tstart[a.nparts];
    // all warps resident at once where the tiles allow: 16 warps per SM
    const int64_t ctas = std::min<int64_t>((ntiles + a.tpc - 1) / a.tpc, int64_t(num_sms()) * 16 / wpc);
    return launch_pdl(gemvr_kernel<GS>, static_cast<unsigned>(std::max<int64_t>(1, ctas)), wpc * 32, 0, st, a);
}

}  // namespace gr

bool gemvr_supported(const WDesc& w, int64_t M) {
    if (M < 1 || M > 8 || w.ndim != 2 || w.n < 1 || w.fmt != QM_AFFINE || w.bits != 4) return false;
    if (w.gs != 32 && w.gs != 64 && w.gs != 128) return false;
    if (w.k < gr::kStep || w.k % gr::kStep) return false;  // whole steps; scale loads aligned
    return w.n <= (int64_t(1) << 31) - 16;
}

bool gemvr_many_supported(const WDesc* ws, int count, int64_t M) {
    if (count < 1 || count > gr::kMaxParts) return false;
    int64_t tiles = 0;
    for (int i = 0; i < count; ++i) {
        if (!gemvr_supported(ws[i], M)) return false;
        if (ws[i].gs != ws[0].gs || ws[i].k != ws[0].k || ws[i].sdt != ws[0].sdt) return false;
        tiles += (ws[i].n + 15) / 16;
    }
    return tiles < (int64_t(1) << 31);
}

cudaError_t launch_gemvr_many(const WDesc* ws, int count, const void* x, int64_t M, void* const* ys,
                              cudaStream_t st) {
    using namespace gr;
    const WDesc& w = ws[0];
    Args a{};
    a.nparts = count;
    a.tstart[0] = 0;
    bool all_static = true;
    for (int i = 0; i < count; ++i) {
        a.part[i].codes = ws[i].codes;
        a.part[i].scales = static_cast<const uint16_t*>(static_cast<const void*>(ws[i].scales));
        a.part[i].biases = static_cast<const uint16_t*>(static_cast<const void*>(ws[i].biases));
        a.part[i].y = static_cast<uint16_t*>(ys[i]);
        a.part[i].n = ws[i].n;
        a.tstart[i + 1] = a.tstart[i] + static_cast<int>((ws[i].n + 15) / 16);
        all_static = all_static && ws[i].is_static;
    }
    a.x = static_cast<const uint16_t*>(x);
    a.M = static_cast<int>(M);
    a.k = w.k;
    a.code_row_bytes = w.code_row_bytes;
    a.scale_row_bytes = w.scale_row_bytes;
    a.sdt = w.sdt;
    a.static_w = all_static ? 1 : 0;
    // k split by k alone (the sum order of an output must not depend on the
    // other weights of a launch): as many warps per tile, up to 12, as divide
    // k's steps, so a long row (down_proj's 3072 inputs: 12 steps) costs one
    // step after the wait
    const int steps = static_cast<int>(w.k / kStep);
    a.ks = 1;
    for (int d = kMaxWarps; d >= 2; --d)
        if (steps % d == 0) {
            a.ks = d;
            break;
        }
    a.tpc = a.ks <= 2 ? kWarps / a.ks : 1;
    a.nsteps = steps / a.ks;
    if (w.gs == 32) return launch_t<32>(a, st);
    if (w.gs == 64) return launch_t<64>(a, st);
    return launch_t<128>(a, st);
}

}  // namespace qm
