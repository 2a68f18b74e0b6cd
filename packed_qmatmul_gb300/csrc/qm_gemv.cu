// qm_gemv.cu -- decode product y[M, n] = x[M, k] * W^T for M <= 16 over packed
// weights, HBM-bound.
//
// The product is the one "Nx_quant (raven-ml.dev API docs)", section
// "Products", val apply, defines: summed at float32 over the weight's float32
// values and rounded once to x's dtype. Like that page's block-scaled kernels,
// it scales each block's (group's) partial sum rather than every element: the
// codes enter the tensor cores as exact small integers, so the only roundings
// are float32 sums.
//
// Design (one GB300: 152 SMs, HBM3e):
//  * A CTA is 1 producer warp + 8 consumer warps, two CTAs to an SM where
//    shared memory allows (so the next launch's CTAs can start beside the
//    last ones of this launch), else 1 producer + 16 consumer warps alone on
//    the SM (large k with several tokens). The producer streams 32-row stages of the
//    packed weight into shared memory with 2-d TMA boxes (codes, 128B-
//    swizzled) and bulk copies (scales, biases), completing on mbarriers,
//    and bulk-copies the activation rows once.
//  * Consumer warps form teams of T. A team takes whole stages; its warps
//    split the stage's groups along k, so a stage is worked on by T warps at
//    once and each warp carries two independent 16-row MMA tiles. A warp
//    decodes codes in registers to f16 pairs that hold exact integers
//    (1024 + code, by a magic-exponent OR) and multiplies them with the
//    activations on mma.sync m16n8k16 (rows of W on the M side, tokens on
//    the N side); per group it applies scale (and bias) in float32. The team
//    adds its warps' partial sums in warp order through shared memory.
//  * Activations are rescaled per token by a power of two so that every bf16
//    value is exact in f16; each group's partial sum is taken back to its
//    true size (an exact power-of-two product) before its scale multiplies
//    it, so no intermediate is larger than the true partial product.
//  * A group whose values are, or may be, infinite (an MXFP4 scale byte of
//    253 or 254, a Q8_0 scale that is infinite, an affine scale or bias of
//    magnitude 2^119 or more) -- or any group, if an activation is infinite
//    or NaN -- is summed element by element instead: each value decoded at
//    float32 as dequant decodes it, times its activation, added in ascending
//    k. IEEE arithmetic then gives the infinities and NaNs that the
//    per-element definition of the product gives ("Nx_quant", "Products",
//    val apply and val dequant: an MXFP4 value past float32's range is
//    infinite; a block whose float16 scale is infinite gives infinite or NaN
//    values).
//  * Where one CTA per stage would leave SMs idle, a cluster of S CTAs splits
//    k; their partial sums meet through distributed shared memory and are
//    added in rank order (deterministic, no global scratch).
//
// MLX affine codes: "GPTQModel wiki: MLX Apple Silicon", "Packed layouts and
// exact transcoding" (little-endian code stream) and "Concepts ..."
// (value = code*scale + bias). Q8_0 and MXFP4 layouts: "Nx_quant", "Weights".
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstring>
#include <unordered_map>

#include "qm_device.cuh"
#include "qm_internal.h"

namespace qm {

static __device__ uint32_t g_err_gemv = 0;

uint32_t gemv_read_clear_error() {
    uint32_t v = 0, z = 0;
    cudaMemcpyFromSymbol(&v, g_err_gemv, sizeof(v));
    cudaMemcpyToSymbol(g_err_gemv, &z, sizeof(z));
    return v;
}

namespace gemv {

constexpr int kRows = 32;            // rows per stage (two MMA row tiles)
// consumer warps: 8 where two CTAs share an SM, 16 where one CTA has it alone
constexpr int kThreadsOf(int cw) { return (cw + 1) * 32; }
constexpr int kMaxTeams = 8;  // named barriers 2 .. 9
constexpr int kMaxStages = 16;
constexpr uint32_t kMagic = 0x64006400u;  // f16x2 (1024, 1024)

struct Params {
    CUtensorMap tm_codes;    // codes as a byte array [n, code_row_bytes], 128 B x 32-row boxes, swizzled
    CUtensorMap tm_scales;   // scales [n, scale_row_bytes], scale_seg x 32-row boxes (k split only)
    CUtensorMap tm_biases;
    const uint8_t* codes;
    const uint8_t* scales;
    const uint8_t* biases;
    const uint16_t* x;
    uint16_t* y;
    int64_t n, k;
    int M;
    int sdt;
    int64_t code_row_bytes, scale_row_bytes;
    // decomposition
    int S;                   // CTAs per cluster, splitting k
    int64_t krange;          // k values per CTA
    int stages_per_cluster;  // 32-row stages per cluster
    int64_t n_stages;        // 32-row stages in all
    int team;                // warps per team (1, 2, 4, 8 or 16)
    int static_w;            // weight may be read before the previous kernel ends
    // grouped mode (apply_experts), off when g_off is null: the weight is
    // [E, n, k] and each cluster slot is one chunk of up to g_Q routed positions
    // of one expert, times one share of that expert's rows
    const int32_t* g_off;    // [E + 1] start of each expert's positions in g_perm
    const int32_t* g_perm;   // routed order -> position
    int g_E;
    int g_Q;                 // positions per chunk
    int g_xdiv;              // activation row of position q: q / g_xdiv
    int g_wclusters;         // clusters per chunk
    // shared memory layout (byte offsets from the dynamic smem base)
    uint32_t nstage, stage_bytes;
    uint32_t code_seg, nbox;          // per row: bytes of codes; 128-byte boxes per stage
    uint32_t scale_seg;               // per row bytes of scales (and of biases) of this CTA's k range
    // scale_span: a stage holds whole rows of scales (and biases), copied as one
    // span, scale_row_bytes apart, this CTA's part at rank * scale_seg; else
    // (a k split whose part is a 16-byte multiple) one 2-d box of scale_seg-byte rows
    int scale_span;
    uint32_t scale_pitch;
    uint32_t off_scales, off_biases;  // within a stage
    uint32_t off_tokscale, off_tok, off_xfrag, off_red, off_xraw, off_recv, off_stages;
};

// ---------------------------------------------------------------- decoders
// Affine 4-bit word -> the A halves for MMA half h: (n[2h], n[4+2h]) and
// 16 * (n[1+2h], n[5+2h]), each as f16 (1024 + value).
QM_DEV void dec4(uint32_t w, int h, uint32_t& lo, uint32_t& hi) {
    const uint32_t s = h ? (w >> 8) : w;
    lo = (s & 0x000F000Fu) | kMagic;
    hi = (s & 0x00F000F0u) | kMagic;
}

// Four 8-bit codes -> f16 (1024 + u0, 1024 + u1), (1024 + u2, 1024 + u3).
QM_DEV void dec8(uint32_t w, uint32_t& lo, uint32_t& hi) {
    lo = prmt(w, 0x64646464u, 0x5140);
    hi = prmt(w, 0x64646464u, 0x7362);
}

template <int SDT>
QM_DEV float sval(uint32_t h) {
    if constexpr (SDT == QM_F16) return f16_bits_to_f32(h);
    else return bf16_bits_to_f32(h);
}

// A stage's codes are 128-byte boxes of 32 rows, each box 128B-swizzled by
// the TMA unit: byte b of row r sits in box b / 128, at row r's 128-byte
// line, 16-byte chunk ((b / 16) mod 8) XOR (r mod 8). Reads never straddle a
// 16-byte chunk, so one address per read suffices. Addresses are 32-bit
// shared-memory addresses; rows r, r + 8, r + 16 and r + 24 share the swizzle
// key, so their reads differ by whole 1 KB steps.
struct CodeRow {
    uint32_t line;  // shared address of stage + r * 128
    uint32_t key;   // (r mod 8) << 4
    QM_DEV uint32_t at(uint32_t b) const {
        return line + (b >> 7) * (kRows * 128) + (((b & 0x70u) ^ key) | (b & 15u));
    }
};

QM_DEV CodeRow code_row(uint32_t st, int r) {
    return CodeRow{st + r * 128, static_cast<uint32_t>(r & 7) << 4};
}

// One group of one 16-row tile: MMAs into acc, rows r0 (= g) and r8 (= g + 8).
template <int FMT, int BITS, int GS, int NT>
QM_DEV void tile_group(const CodeRow& r0, const CodeRow& r8, int gi, int t,
                       const uint32_t (&bf)[GS / 16][NT][2], float (&acc)[NT][4]) {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[nt][i] = 0.0f;
    if constexpr (FMT == QM_AFFINE && BITS == 4) {
        constexpr int V = GS / 32;  // words of a row per lane per group
        uint32_t w0[V], w8[V];
        const uint32_t off = gi * (GS / 2) + t * V * 4;
        const uint32_t a0_ = r0.at(off), a8_ = a0_ + (r8.line - r0.line);
        if constexpr (V == 1) {
            w0[0] = lds_u32(a0_);
            w8[0] = lds_u32(a8_);
        } else if constexpr (V == 2) {
            const uint2 a = lds_v2(a0_);
            const uint2 c = lds_v2(a8_);
            w0[0] = a.x; w0[1] = a.y; w8[0] = c.x; w8[1] = c.y;
        } else {
            const uint4 a = lds_v4(a0_);
            const uint4 c = lds_v4(a8_);
            w0[0] = a.x; w0[1] = a.y; w0[2] = a.z; w0[3] = a.w;
            w8[0] = c.x; w8[1] = c.y; w8[2] = c.z; w8[3] = c.w;
        }
#pragma unroll
        for (int v = 0; v < V; ++v)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                uint32_t a0, a2, a1, a3;
                dec4(w0[v], h, a0, a2);
                dec4(w8[v], h, a1, a3);
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
                    mma_f16(acc[nt], a0, a1, a2, a3, bf[2 * v + h][nt][0], bf[2 * v + h][nt][1]);
            }
    } else if constexpr (FMT == QM_AFFINE && BITS == 8) {
        constexpr int V = GS / 16;  // 2, 4 or 8 words
        const uint32_t off = gi * GS + t * V * 4;
        uint32_t wa[V], wc[V];
        const uint32_t d8 = r8.line - r0.line;
        if constexpr (V == 2) {
            const uint2 a = lds_v2(r0.at(off));
            const uint2 c = lds_v2(r0.at(off) + d8);
            wa[0] = a.x; wa[1] = a.y; wc[0] = c.x; wc[1] = c.y;
        } else {
#pragma unroll
            for (int q = 0; q < V / 4; ++q) {
                const uint4 a = lds_v4(r0.at(off + 16 * q));
                const uint4 c = lds_v4(r0.at(off + 16 * q) + d8);
                wa[4 * q] = a.x; wa[4 * q + 1] = a.y; wa[4 * q + 2] = a.z; wa[4 * q + 3] = a.w;
                wc[4 * q] = c.x; wc[4 * q + 1] = c.y; wc[4 * q + 2] = c.z; wc[4 * q + 3] = c.w;
            }
        }
#pragma unroll
        for (int v = 0; v < V; ++v) {
            uint32_t a0, a2, a1, a3;
            dec8(wa[v], a0, a2);
            dec8(wc[v], a1, a3);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) mma_f16(acc[nt], a0, a1, a2, a3, bf[v][nt][0], bf[v][nt][1]);
        }
    } else if constexpr (FMT == QM_Q8_0) {
        // codes of block gi at byte 34*gi + 2 + 8t (2-byte aligned when gi is even)
        const uint32_t o = 34 * gi + 2 + 8 * t;
        uint32_t c0[2], c8[2];
        auto w32 = [](const CodeRow& r, uint32_t b) { return lds_u32(r.at(b)); };
        if (o & 2) {
            const uint32_t x0 = w32(r0, o - 2), x1 = w32(r0, o + 2), x2 = w32(r0, o + 6);
            const uint32_t z0 = w32(r8, o - 2), z1 = w32(r8, o + 2), z2 = w32(r8, o + 6);
            c0[0] = prmt(x0, x1, 0x5432); c0[1] = prmt(x1, x2, 0x5432);
            c8[0] = prmt(z0, z1, 0x5432); c8[1] = prmt(z1, z2, 0x5432);
        } else {
            c0[0] = w32(r0, o); c0[1] = w32(r0, o + 4); c8[0] = w32(r8, o); c8[1] = w32(r8, o + 4);
        }
#pragma unroll
        for (int mm = 0; mm < 2; ++mm) {
            uint32_t a0, a2, a1, a3;
            dec8(c0[mm] ^ 0x80808080u, a0, a2);
            dec8(c8[mm] ^ 0x80808080u, a1, a3);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) mma_f16(acc[nt], a0, a1, a2, a3, bf[mm][nt][0], bf[mm][nt][1]);
        }
    } else if constexpr (FMT == QM_MXFP4_BLOCKS) {
        // data bytes 4t .. 4t+3 of 17-byte block gi (its scale byte, then byte j
        // holding values j and j + 16), from the aligned words around them. The
        // second word is read only when the bytes straddle two: a row holds a
        // multiple of 16 blocks, so its last block's data bytes are aligned and
        // no read passes the row's end.
        const uint32_t o = 17 * gi + 1 + 4 * t, a = o & ~3u, sh = 8u * (o & 3u);
        const uint32_t d8 = r8.line - r0.line;
        const uint32_t p0 = r0.at(a), p1 = sh ? r0.at(a + 4) : p0;
        const uint32_t w0 = __funnelshift_r(lds_u32(p0), lds_u32(p1), sh);
        const uint32_t w8 = __funnelshift_r(lds_u32(p0 + d8), lds_u32(p1 + d8), sh);
        uint32_t h0[4], h8[4];
        e2m1x8_to_f16x2(w0, h0);  // byte i -> (value 4t + i, value 4t + i + 16)
        e2m1x8_to_f16x2(w8, h8);
#pragma unroll
        for (int mm = 0; mm < 2; ++mm)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
                mma_f16(acc[nt], h0[2 * mm], h8[2 * mm], h0[2 * mm + 1], h8[2 * mm + 1], bf[mm][nt][0],
                        bf[mm][nt][1]);
    } else {  // MXFP4
        const uint32_t o = 16 * gi + 4 * t;
        uint32_t h0[4], h8[4];
        const uint32_t a = r0.at(o);
        e2m1x8_to_f16x2(lds_u32(a), h0);
        e2m1x8_to_f16x2(lds_u32(a + (r8.line - r0.line)), h8);
#pragma unroll
        for (int mm = 0; mm < 2; ++mm)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
                mma_f16(acc[nt], h0[2 * mm], h8[2 * mm], h0[2 * mm + 1], h8[2 * mm + 1], bf[mm][nt][0],
                        bf[mm][nt][1]);
    }
}

// Value i (0 .. GS-1) of group gi of one staged row, decoded at float32 as
// dequant decodes it: affine fmaf(code, s, b); Q8_0 d * q; MXFP4 e2m1 * scale.
template <int FMT, int BITS, int GS>
QM_DEV float elem_value(const CodeRow& r, int gi, int i, float s, float b) {
    if constexpr (FMT == QM_AFFINE) {
        const uint32_t bit = static_cast<uint32_t>(gi * GS + i) * BITS;
        const uint32_t c = (lds_u8(r.at(bit >> 3)) >> (bit & 7u)) & ((1u << BITS) - 1u);
        return fmaf(static_cast<float>(c), s, b);
    } else if constexpr (FMT == QM_Q8_0) {
        const int q = static_cast<int8_t>(lds_u8(r.at(34 * gi + 2 + i)));
        return s * static_cast<float>(q);
    } else {
        uint32_t code;
        if constexpr (FMT == QM_MXFP4_BLOCKS) {  // byte j of the block's data: values j and j + 16
            const uint32_t byte = lds_u8(r.at(17 * gi + 1 + (i & 15)));
            code = i < 16 ? (byte & 15u) : (byte >> 4);
        } else {
            const uint32_t byte = lds_u8(r.at(16 * gi + (i >> 1)));
            code = (i & 1) ? (byte >> 4) : (byte & 15u);
        }
        uint32_t h[4];
        e2m1x8_to_f16x2(code, h);
        return __half2float(__ushort_as_half(static_cast<unsigned short>(h[0] & 0xFFFFu))) * s;
    }
}

// Group gi's exact contribution to rows ra and rb of a tile for one token:
// the sums over the group's inputs of x * value at float32, in ascending k,
// x read from global memory (xrow: the token's activations at this group's
// first input). Kept out of line: it runs only for exceptional groups.
template <int FMT, int BITS, int GS>
static __device__ __noinline__ float2 group_exact(CodeRow ra, CodeRow rb, int gi, float sa, float ba, float sb,
                                                  float bb, const uint16_t* xrow) {
    float acc_a = 0.0f, acc_b = 0.0f;
#pragma unroll 1
    for (int i = 0; i < GS; ++i) {
        const float xv = bf16_bits_to_f32(__ldg(xrow + i));
        acc_a = fmaf(xv, elem_value<FMT, BITS, GS>(ra, gi, i, sa, ba), acc_a);
        acc_b = fmaf(xv, elem_value<FMT, BITS, GS>(rb, gi, i, sb, bb), acc_b);
    }
    return make_float2(acc_a, acc_b);
}

// Grouped mode, one warp: which chunk cluster slot `slot` is -- its size
// (s_grp[0], 0 past the last chunk), expert (s_grp[1]), positions and
// activation rows -- from the routing offsets, 32 experts per step.
static __device__ __noinline__ void group_lookup(const Params& p, int slot, int lane, int* s_grp, int* s_pos,
                                                 int* s_xrow) {
    int before = 0;  // chunks of the experts already passed
    int gm = 0, ge = 0, gb = 0;
    for (int e0 = 0; e0 < p.g_E; e0 += 32) {
        const int e = e0 + lane;
        int o0 = 0, cnt = 0;
        if (e < p.g_E) {
            o0 = __ldg(p.g_off + e);
            cnt = __ldg(p.g_off + e + 1) - o0;
        }
        const int nch = (cnt + p.g_Q - 1) / p.g_Q;
        int inc = nch;  // inclusive scan over the lanes
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int t = __shfl_up_sync(0xffffffffu, inc, o);
            if (lane >= o) inc += t;
        }
        const int lo = before + inc - nch;
        const bool mine = e < p.g_E && slot >= lo && slot < lo + nch;
        const uint32_t hit = __ballot_sync(0xffffffffu, mine);
        if (mine) {
            const int ch = slot - lo;
            gb = o0 + ch * p.g_Q;
            gm = min(p.g_Q, cnt - ch * p.g_Q);
            ge = e;
        }
        if (hit) {
            const int src = __ffs(hit) - 1;
            gm = __shfl_sync(0xffffffffu, gm, src);
            ge = __shfl_sync(0xffffffffu, ge, src);
            gb = __shfl_sync(0xffffffffu, gb, src);
            break;
        }
        before += __shfl_sync(0xffffffffu, inc, 31);
    }
    if (lane == 0) { s_grp[0] = gm; s_grp[1] = ge; }
    if (lane < gm) {
        const int q = __ldg(p.g_perm + gb + lane);
        s_pos[lane] = q;
        s_xrow[lane] = q / p.g_xdiv;
    }
}

// NTK: token tiles of 8 (1 for M <= 8, 2 for M <= 16), or 0 for exactly one
// token: the layout of NTK = 1, with the epilogue and the sums over a team
// restricted to the accumulator entries that hold token 0. SDT: the affine
// scale and bias dtype (QM_BF16 or QM_F16; unused by the other formats).
template <int FMT, int BITS, int GS, int NTK, int SDT, int CW>
__global__ void __launch_bounds__(kThreadsOf(CW), CW == 8 ? 2 : 1) gemv_kernel(const __grid_constant__ Params p) {
    constexpr int kWarps = CW;
    constexpr int NT = NTK == 0 ? 1 : NTK;
    constexpr bool ONE = NTK == 0;
    extern __shared__ __align__(1024) uint8_t smem[];
    constexpr int MM = GS / 16;  // MMAs per group
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int S = p.S;
    const uint32_t rank = (S > 1) ? cluster_ctarank() : 0;
    int cluster = static_cast<int>(blockIdx.x) / S;
    const int64_t kbase = rank * p.krange;
    const int groups = static_cast<int>(p.krange / GS);

    // barriers: full[16], empty[16], x, the abort flag, then slot_stage[16]:
    // the stage a slot was last filled with. Teams take stages round-robin,
    // so a consumer may reach a slot more than one fill ahead of the
    // producer; it waits for the slot's tag before trusting the parity.
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem);
    const uint32_t bar_full0 = smem_u32(bars), bar_empty0 = smem_u32(bars + kMaxStages);
    const uint32_t bar_x = smem_u32(bars + 2 * kMaxStages);
    const uint32_t bar_red = smem_u32(smem + 344);  // split k: the other CTAs' partial sums are in (rank 0)
    volatile int& s_abort = *reinterpret_cast<volatile int*>(smem + (2 * kMaxStages + 1) * 8);
    volatile int* slot_stage = reinterpret_cast<volatile int*>(smem + (2 * kMaxStages + 2) * 8);
    // grouped mode: the chunk's size and expert, its positions and activation rows
    int* s_grp = reinterpret_cast<int*>(smem + 360);        // [2]
    int* s_pos = reinterpret_cast<int*>(smem + 368);        // [16]
    int* s_xrow = reinterpret_cast<int*>(smem + 432);       // [16], ends at 496
    volatile int& s_xbad = *reinterpret_cast<volatile int*>(smem + 496);  // an activation is inf or NaN

    unsigned int* xmax = reinterpret_cast<unsigned int*>(smem + p.off_tokscale) + 32;  // [16] max |x| as bf16 bits
    if (threadIdx.x == 0) {
        s_abort = 0;
        s_xbad = 0;
        #pragma unroll 1
        for (int i = 0; i < kMaxStages; ++i) slot_stage[i] = -1;
        #pragma unroll 1
        for (int i = 0; i < 16; ++i) xmax[i] = 0u;
        prefetch_tmap(&p.tm_codes);
        #pragma unroll 1
        for (uint32_t i = 0; i < p.nstage; ++i) {
            mbar_init(bar_full0 + 8 * i, 32);      // the producer's lanes
            mbar_init(bar_empty0 + 8 * i, p.team);  // the warps of the team that read it
        }
        mbar_init(bar_x, 1);
        if (S > 1 && rank == 0) mbar_init(bar_red, 1);  // rank 0's own arrival; the pushes count bytes
        fence_mbar_init();
    }
    __syncthreads();
    // each thread lets the next kernel start once its own wait on the previous
    // one has returned: one kernel waits ahead, with this one's run to stream
    // its static weights
    auto wait_prev = [&]() {
        grid_dependency_wait();
        grid_launch_dependents();
    };
    int M = p.M;
    int64_t wrow0 = 0;  // first row of this CTA's matrix in the codes and scales
    if (p.g_off) {
        // which chunk of which expert: the routing tables come from the previous kernel
        if (warp == 0) {
            wait_prev();
            group_lookup(p, static_cast<int>(cluster / p.g_wclusters), lane, s_grp, s_pos, s_xrow);
        }
        __syncthreads();
        M = s_grp[0];
        if (M == 0) return;  // a slot past the last chunk; the same for every CTA of the cluster
        wrow0 = static_cast<int64_t>(s_grp[1]) * p.n;
        cluster = static_cast<int>(cluster % p.g_wclusters);
    }
    const int64_t stage0 = cluster * p.stages_per_cluster;
    const int nst = static_cast<int>(std::min<int64_t>(p.stages_per_cluster, p.n_stages - stage0));
    if (S > 1) cluster_arrive_relaxed();  // waited for before the first access to another CTA
    // x comes from the previous kernel; so may W, unless the caller marked it
    // static, in which case the producer streams its first stages before waiting
    if (!p.g_off && (!p.static_w || warp != kWarps)) wait_prev();
    else if (p.g_off && warp != 0) wait_prev();

    if (warp == kWarps) {
        // ------------------------------------------------------------ producer
        const uint32_t xbytes = static_cast<uint32_t>(p.krange * 2);
        auto copy_x = [&]() {  // after the first stage's copies are under way
            if (lane == 0) {
                mbar_expect_tx(bar_x, xbytes * M);
                mbar_arrive(bar_x);
            }
            __syncwarp();
            if (lane < M) {
                const int64_t xr = p.g_off ? s_xrow[lane] : lane;
                bulk_g2s(smem_u32(smem + p.off_xraw + lane * xbytes), p.x + xr * p.k + kbase, xbytes, bar_x);
            }
        };
        int issued = 0;
        bool xdone = false;
        const int npre = p.static_w ? std::min(nst, static_cast<int>(p.nstage)) : 0;
        uint32_t slot = 0, fill = 0;  // stage j goes to slot j mod nstage, fill j / nstage of it
        #pragma unroll 1
        for (int j = 0; j < nst; ++j, (++slot == p.nstage) ? (slot = 0, ++fill) : 0u) {
            if (p.static_w && !xdone && j == npre) {
                wait_prev();
                copy_x();
                xdone = true;
            }
            const uint32_t par = (fill & 1) ^ 1;
            if (!mbar_wait(bar_empty0 + 8 * slot, par) || s_abort) {
                if (lane == 0) { atomicOr(&g_err_gemv, DEV_ERR_TIMEOUT); s_abort = 1; }
                break;
            }
            issued = j + 1;
            const int64_t row0 = (stage0 + j) * kRows;
            const int rows = static_cast<int>(std::min<int64_t>(kRows, p.n - row0));
            uint8_t* st = smem + p.off_stages + slot * p.stage_bytes;
            const uint32_t bar = bar_full0 + 8 * slot;
            // whole boxes count in full (rows past n arrive as zeros); scales and
            // biases come as one span when k is whole, else as one box each
            uint32_t tx = p.nbox * kRows * 128;
            uint32_t span = 0, span_bulk = 0;
            if (p.scale_seg) {
                if (!p.scale_span) {
                    tx += kRows * p.scale_seg * (p.biases ? 2 : 1);
                } else {
                    span = rows * static_cast<uint32_t>(p.scale_row_bytes);
                    span_bulk = span & ~15u;
                    tx += span_bulk * (p.biases ? 2 : 1);
                }
            }
            if (lane == 0) {
                slot_stage[slot] = j;
                mbar_expect_tx(bar, tx);
            }
            __syncwarp();
            {
                // The stage's copies are spread over the warp's lanes: a thread
                // completes about one TMA copy per 0.39 us whatever its size, so
                // one lane issuing a stage's boxes in turn capped the stream.
                const int32_t x0 = static_cast<int32_t>(rank * p.code_seg), y0 = static_cast<int32_t>(wrow0 + row0);
                #pragma unroll 1
                for (uint32_t c = lane; c < p.nbox; c += 32)
                    tma_load_2d(smem_u32(st + c * kRows * 128), &p.tm_codes, x0 + 128 * c, y0, bar);
                if (p.scale_seg && !p.scale_span) {
                    const int32_t xs0 = static_cast<int32_t>(rank * p.scale_seg);
                    if (lane == 31) tma_load_2d(smem_u32(st + p.off_scales), &p.tm_scales, xs0, y0, bar);
                    if (p.biases && lane == 30) tma_load_2d(smem_u32(st + p.off_biases), &p.tm_biases, xs0, y0, bar);
                }
            }
            if (p.scale_seg && p.scale_span) {
                const int64_t off = (wrow0 + row0) * p.scale_row_bytes;
                if (span_bulk) {
                    if (lane == 31) bulk_g2s(smem_u32(st + p.off_scales), p.scales + off, span_bulk, bar);
                    if (p.biases && lane == 30) bulk_g2s(smem_u32(st + p.off_biases), p.biases + off, span_bulk, bar);
                }
                #pragma unroll 1
                for (uint32_t b = span_bulk + lane; b < span; b += 32) {  // ragged tail of the last stage
                    st[p.off_scales + b] = p.scales[off + b];
                    if (p.biases) st[p.off_biases + b] = p.biases[off + b];
                }
            }
            mbar_arrive(bar);
            if (!p.static_w && !xdone) {
                copy_x();
                xdone = true;
            }
        }
        if (!xdone) {  // every stage prefetched, or abandoned before the first
            if (p.static_w) wait_prev();
            copy_x();
        }
        if (s_abort) {
            // abandoned: let the copies already issued land before the CTA exits
            #pragma unroll 1
            for (int j = std::max(0, issued - static_cast<int>(p.nstage)); j < issued; ++j)
                (void)mbar_wait(bar_full0 + 8 * (j % p.nstage), (j / p.nstage) & 1);
            (void)mbar_wait(bar_x, 0);
        }
    } else {
        // ------------------------------------------------------------ consumers
        const int ctid = threadIdx.x;  // 0 .. 32 * kWarps - 1
        float* tokscale = reinterpret_cast<float*>(smem + p.off_tokscale);  // [16] 2^-E
        const uint16_t* xs = reinterpret_cast<const uint16_t*>(smem + p.off_xraw);  // [M][krange]
        if (!mbar_wait(bar_x, 0)) {
            if (lane == 0) { atomicOr(&g_err_gemv, DEV_ERR_TIMEOUT); s_abort = 1; }
        }
        // 1. per-token power-of-two scale over this CTA's k range (warp m: token m)
        {
            // max |x| per token as bf16 magnitude bits (integer order is value
            // order, and an infinity or NaN sorts above every finite value):
            // one pass over the staged rows, order-free (warp maxima first:
            // one shared atomic per warp and token)
            const int per_row = static_cast<int>(p.krange / 8);
            #pragma unroll 1
            for (int m = 0; m < M; ++m)
                #pragma unroll 1
                for (int i0 = 0; i0 < per_row; i0 += kWarps * 32) {
                    const int i = i0 + ctid;
                    uint32_t amax = 0u;
                    if (i < per_row) {
                        const uint4 q = *reinterpret_cast<const uint4*>(xs + m * p.krange + 8 * i);
                        amax = __vmaxu2(__vmaxu2(q.x & 0x7FFF7FFFu, q.y & 0x7FFF7FFFu),
                                        __vmaxu2(q.z & 0x7FFF7FFFu, q.w & 0x7FFF7FFFu));
                        amax = max(amax & 0xFFFFu, amax >> 16);
                    }
                    const uint32_t b = __reduce_max_sync(0xffffffffu, amax);
                    if (lane == 0 && b) atomicMax(&xmax[m], b);
                }
        }
        named_bar_sync(1, kWarps * 32);
        // x' = x * 2^E puts max |x'| in [2^14, 2^15): every bf16 value is then exact in f16
        auto token_exp = [&](int m) {
            const uint32_t bits = xmax[m];
            if (bits == 0u || bits >= 0x7F80u) return 0;  // zeros, or non-finite (summed per element)
            const int ex = static_cast<int>((bits >> 7) & 0xFF) - 127;
            return min(max(14 - ex, -126), 126);
        };
        if (ctid < 16) {
            const int E = token_exp(ctid);
            tokscale[ctid] = __uint_as_float(static_cast<uint32_t>(-E + 127) << 23);
            if (ctid < M && xmax[ctid] >= 0x7F80u) s_xbad = 1;
        }
        // 2. B fragments for every group of the k range; each quad of lanes
        //    also sums its token's B values (F) and x' (X) over the group
        uint32_t* xfrag = reinterpret_cast<uint32_t*>(smem + p.off_xfrag);
        float2* tok = reinterpret_cast<float2*>(smem + p.off_tok);  // [groups][16]
        if constexpr (ONE) {
            // One token: only lanes 0..3 (t) of a warp hold nonzero B values, so
            // the fragments are kept for those four lanes alone, [gi][t][MM][2].
            // A work item is one MMA's pair of registers (gi, mm, t): a group's
            // 4 MM items sit in adjacent lanes of one warp, which add its sums.
            const int items = (groups * MM * 4 + 31) / 32 * 32;
            const float mul = __uint_as_float(static_cast<uint32_t>(token_exp(0) + 127) << 23);
            #pragma unroll 1
            for (int it = ctid; it < items; it += kWarps * 32) {
                const int t = it & 3, mm = (it >> 2) % MM, gi = (it >> 2) / MM;
                const bool live = gi < groups;
                auto xv = [&](int kk) { return live ? bf16_bits_to_f32(xs[kk]) * mul : 0.0f; };
                float lo0, hi0, lo1, hi1, f1 = 1.0f;  // registers 2mm: (lo0, hi0), 2mm+1: f1 (lo1, hi1)
                if constexpr (FMT == QM_AFFINE && BITS == 4) {
                    constexpr int V = GS / 32;
                    const int v = mm >> 1, h = mm & 1;
                    const int k0 = 8 * (gi * (GS / 8) + t * V + v);
                    lo0 = xv(k0 + 2 * h);
                    hi0 = xv(k0 + 4 + 2 * h);
                    lo1 = xv(k0 + 1 + 2 * h);
                    hi1 = xv(k0 + 5 + 2 * h);
                    f1 = 0.0625f;
                } else if constexpr (FMT == QM_AFFINE && BITS == 8) {
                    constexpr int V = GS / 16;
                    const int k0 = 4 * (gi * (GS / 4) + t * V + mm);
                    lo0 = xv(k0); hi0 = xv(k0 + 1); lo1 = xv(k0 + 2); hi1 = xv(k0 + 3);
                } else if constexpr (FMT == QM_MXFP4_BLOCKS) {
                    // lane t holds values 4t .. 4t+3 and 4t+16 .. 4t+19 of the block,
                    // paired (j, j + 16) as its bytes pair them
                    const int k0 = 32 * gi + 4 * t + 2 * mm;
                    lo0 = xv(k0); hi0 = xv(k0 + 16); lo1 = xv(k0 + 1); hi1 = xv(k0 + 17);
                } else {  // Q8_0, MXFP4: lane t holds values 8t .. 8t+7 of the block
                    const int k0 = 32 * gi + 8 * t + 4 * mm;
                    lo0 = xv(k0); hi0 = xv(k0 + 1); lo1 = xv(k0 + 2); hi1 = xv(k0 + 3);
                }
                if (live) {
                    uint32_t* dst = xfrag + (gi * 4 + t) * MM * 2 + mm * 2;
                    dst[0] = pack_f16x2(lo0, hi0);
                    dst[1] = pack_f16x2(lo1 * f1, hi1 * f1);
                }
                if constexpr (FMT != QM_MXFP4 && FMT != QM_MXFP4_BLOCKS) {
                    // the offset the magic adds: magic * sum of the B values the MMAs see
                    float X = (lo0 + hi0) + (lo1 + hi1);
                    float F = (lo0 + hi0) + (lo1 * f1 + hi1 * f1);
#pragma unroll
                    for (int o = 1; o < 4 * MM; o <<= 1) {
                        X += __shfl_xor_sync(0xffffffffu, X, o);
                        F += __shfl_xor_sync(0xffffffffu, F, o);
                    }
                    const float magic = (FMT == QM_Q8_0) ? 1152.0f : 1024.0f;
                    if (t == 0 && mm == 0 && live) tok[gi * 16] = make_float2(magic * F, X);
                }
            }
        } else {
            const int items = groups * 32 * NT;  // a multiple of 32: a warp shares (gi, nt)
            #pragma unroll 1
            for (int it = ctid; it < items; it += kWarps * 32) {
                const int ln = it % 32, nt = (it / 32) % NT, gi = it / (32 * NT);
                const int tg = ln >> 2, t = ln & 3;
                const int m = nt * 8 + tg;
                const bool live = m < M;  // padding tokens get exact zeros
                const float mul = live ? __uint_as_float(static_cast<uint32_t>(token_exp(m) + 127) << 23) : 0.0f;
                const uint16_t* xr = xs + (live ? m : 0) * p.krange;
                uint32_t* dst = xfrag + ((gi * 32 + ln) * MM) * NT * 2 + nt * 2;
                float F = 0.0f, X = 0.0f;
                auto xv = [&](int kk) { return live ? bf16_bits_to_f32(xr[kk]) * mul : 0.0f; };
                auto put = [&](int idx, float lo, float hi, float flo, float fhi) {
                    dst[idx] = pack_f16x2(lo * flo, hi * fhi);
                    X += lo + hi;
                    F += lo * flo + hi * fhi;
                };
                if constexpr (FMT == QM_AFFINE && BITS == 4) {
                    constexpr int V = GS / 32;
#pragma unroll
                    for (int v = 0; v < V; ++v) {
                        const int k0 = 8 * (gi * (GS / 8) + t * V + v);
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            const int mm = 2 * v + h;
                            put(mm * NT * 2 + 0, xv(k0 + 2 * h), xv(k0 + 4 + 2 * h), 1.0f, 1.0f);
                            put(mm * NT * 2 + 1, xv(k0 + 1 + 2 * h), xv(k0 + 5 + 2 * h), 0.0625f, 0.0625f);
                        }
                    }
                } else if constexpr (FMT == QM_AFFINE && BITS == 8) {
                    constexpr int V = GS / 16;
#pragma unroll
                    for (int v = 0; v < V; ++v) {
                        const int k0 = 4 * (gi * (GS / 4) + t * V + v);
                        put(v * NT * 2 + 0, xv(k0), xv(k0 + 1), 1.0f, 1.0f);
                        put(v * NT * 2 + 1, xv(k0 + 2), xv(k0 + 3), 1.0f, 1.0f);
                    }
                } else if constexpr (FMT == QM_MXFP4_BLOCKS) {  // values (j, j + 16) as the bytes pair them
#pragma unroll
                    for (int mm = 0; mm < 2; ++mm) {
                        const int k0 = 32 * gi + 4 * t + 2 * mm;
                        put(mm * NT * 2 + 0, xv(k0), xv(k0 + 16), 1.0f, 1.0f);
                        put(mm * NT * 2 + 1, xv(k0 + 1), xv(k0 + 17), 1.0f, 1.0f);
                    }
                } else {  // Q8_0, MXFP4: lane t holds values 8t .. 8t+7 of the block
#pragma unroll
                    for (int mm = 0; mm < 2; ++mm) {
                        const int k0 = 32 * gi + 8 * t + 4 * mm;
                        put(mm * NT * 2 + 0, xv(k0), xv(k0 + 1), 1.0f, 1.0f);
                        put(mm * NT * 2 + 1, xv(k0 + 2), xv(k0 + 3), 1.0f, 1.0f);
                    }
                }
                if constexpr (FMT != QM_MXFP4 && FMT != QM_MXFP4_BLOCKS) {
                    // the offset the magic adds: magic * sum of the B values the MMAs see
                    X += __shfl_xor_sync(0xffffffffu, X, 1);
                    F += __shfl_xor_sync(0xffffffffu, F, 1);
                    X += __shfl_xor_sync(0xffffffffu, X, 2);
                    F += __shfl_xor_sync(0xffffffffu, F, 2);
                    const float magic = (FMT == QM_Q8_0) ? 1152.0f : 1024.0f;
                    if (t == 0) tok[gi * 16 + m] = make_float2(magic * F, X);
                }
            }
        }
        named_bar_sync(1, kWarps * 32);

        // 3. main loop: team `team` takes stages team, team + nteams, ...;
        //    warp wi of the team covers groups [gb, ge) of each.
        // the team size is a power of two: shifts, not divisions
        const int T = p.team, lt = __ffs(T) - 1, nteams = kWarps >> lt;
        const int team = warp >> lt, wi = warp & (T - 1);
        const int gb = (wi * groups) >> lt, ge = ((wi + 1) * groups) >> lt;
        const int g = lane >> 2, t = lane & 3;
        const uint32_t soff = p.scale_span ? rank * p.scale_seg : 0u;  // this CTA's part of a scale row
        float* partial = reinterpret_cast<float*>(smem + p.off_xraw);  // [stages][32 rows][16 tok]
        float* red = reinterpret_cast<float*>(smem + p.off_red);       // [teams][2][T][2][NT][4][32]
        int buf = 0;
        // 2^-E of the tokens of this lane's accumulator columns (2t and 2t + 1
        // of each token tile): a group's MMA sum times it is at its true size
        float tk[NT][2];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            tk[nt][0] = tokscale[ONE ? 0 : nt * 8 + 2 * t];
            tk[nt][1] = tokscale[ONE ? 0 : nt * 8 + 2 * t + 1];
        }
        const bool xbad = s_xbad != 0;
        const int64_t xk0 = kbase;  // this CTA's first input
        // Every warp of a team runs the same iterations and meets the team
        // barrier once per stage, abandoned or not, so no barrier is left waiting.
        // slot of stage j and how many times it was filled before, kept
        // incrementally (nteams <= nstage): j mod nstage and j / nstage
        uint32_t slot = team, fill = 0;
        while (slot >= p.nstage) { slot -= p.nstage; ++fill; }
        #pragma unroll 1
        for (int j = team; j < nst; j += nteams) {
            if (j != team) {
                slot += nteams;
                while (slot >= p.nstage) { slot -= p.nstage; ++fill; }
            }
            bool live = !s_abort;
            // A slot's first fill needs no tag: its barrier's first phase can only
            // be that fill. Later fills check that the producer has started stage j.
            if (fill > 0 && live && lane == 0 && slot_stage[slot] != j) {
                const uint64_t t0 = globaltimer();
                #pragma unroll 1
                for (int spin = 0; slot_stage[slot] != j && !s_abort; ++spin)
                    if ((spin & 63) == 63 && globaltimer() - t0 > kWaitLimitNs) {
                        atomicOr(&g_err_gemv, DEV_ERR_TIMEOUT);
                        s_abort = 1;
                        break;
                    }
                live = !s_abort;
            }
            live = __shfl_sync(0xffffffffu, live ? 1 : 0, 0) != 0;
            if (live && !mbar_wait(bar_full0 + 8 * slot, fill & 1)) {
                if (lane == 0) { atomicOr(&g_err_gemv, DEV_ERR_TIMEOUT); s_abort = 1; }
                live = false;
            }
            live = __shfl_sync(0xffffffffu, live ? 1 : 0, 0) != 0;
            const uint32_t st = smem_u32(smem) + p.off_stages + slot * p.stage_bytes;
            const CodeRow rows_[4] = {code_row(st, g), code_row(st, g + 8), code_row(st, 16 + g),
                                      code_row(st, 24 + g)};
            float y[2][NT][4];
#pragma unroll
            for (int tt = 0; tt < 2; ++tt)
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int i = 0; i < 4; ++i) y[tt][nt][i] = 0.0f;

            // one group of both tiles: MMAs, then scale (and bias) into y
            auto do_group = [&](int gi, float (&acc)[2][NT][4]) {
                uint32_t bf[MM][NT][2];
                {
                    const uint32_t src = smem_u32(smem) + p.off_xfrag +
                                         4u * (ONE ? (gi * 4 + t) * MM * 2 : ((gi * 32 + lane) * MM) * NT * 2);
                    uint32_t* bb = &bf[0][0][0];
#pragma unroll
                    for (int q = 0; q < MM * NT / 2; ++q) {
                        uint4 v = make_uint4(0u, 0u, 0u, 0u);
                        if (!ONE || g == 0) v = lds_v4(src + 16 * q);  // one token: the other lanes' columns are zero
                        bb[4 * q] = v.x; bb[4 * q + 1] = v.y; bb[4 * q + 2] = v.z; bb[4 * q + 3] = v.w;
                    }
                }
#pragma unroll
                for (int tt = 0; tt < 2; ++tt)
                    tile_group<FMT, BITS, GS, NT>(rows_[2 * tt], rows_[2 * tt + 1], gi, t, bf, acc[tt]);
            };
            // a group's scales (and biases) as raw bits, [tile][s0, s8, b0, b8]
            // (rows ra and ra + 8 of the tile), loaded ahead of the group's MMAs
            auto ep_load = [&](int gi, uint32_t (&raw)[2][4]) {
#pragma unroll
                for (int tt = 0; tt < 2; ++tt) {
                    const int ra = 16 * tt + g;
                    if constexpr (FMT == QM_AFFINE) {
                        // row ra, group gi; row rb = ra + 8 lies 8 rows of scale_pitch bytes on
                        const uint32_t sa = st + p.off_scales + ra * p.scale_pitch + soff + 2 * gi;
                        const uint32_t ba = sa + (p.off_biases - p.off_scales);
                        const uint32_t r8 = 8 * p.scale_pitch;
                        raw[tt][0] = lds_u16(sa);
                        raw[tt][1] = lds_u16(sa + r8);
                        raw[tt][2] = lds_u16(ba);
                        raw[tt][3] = lds_u16(ba + r8);
                    } else if constexpr (FMT == QM_Q8_0) {
                        const uint32_t da = rows_[2 * tt].at(34 * gi);
                        raw[tt][0] = lds_u16(da);
                        raw[tt][1] = lds_u16(da + (rows_[2 * tt + 1].line - rows_[2 * tt].line));
                    } else if constexpr (FMT == QM_MXFP4_BLOCKS) {  // the block's first byte
                        const uint32_t da = rows_[2 * tt].at(17 * gi);
                        raw[tt][0] = lds_u8(da);
                        raw[tt][1] = lds_u8(da + (rows_[2 * tt + 1].line - rows_[2 * tt].line));
                    } else {
                        const uint32_t sa = st + p.off_scales + ra * p.scale_pitch + soff + gi;
                        raw[tt][0] = lds_u8(sa);
                        raw[tt][1] = lds_u8(sa + 8 * p.scale_pitch);
                    }
                }
            };
            // a tile's scales (and biases) as float32 from their raw bits, and
            // whether the tile's rows must be summed element by element this stage:
            // a scale (or bias) so large that a group's sum at the activations'
            // 2^E scale could leave float32's range over a stage, or values that
            // are or may be infinite (an infinite Q8_0 d; MXFP4 bytes 253/254 and
            // affine magnitudes of 2^119 or more lie inside these bounds). Over a
            // stage a warp adds at most 2^9 groups, each at most 2^22.6 (MXFP4:
            // 6 * 32 * 2^15) or 2^30 (affine: 256 * 128 * 2^15) times its scale, so
            // scales below 2^93 (MXFP4) and 2^87 (affine) keep every sum below
            // 2^127. A NaN scale or bias needs no exception: it makes every value
            // of its group NaN, and the scaled sum NaN too.
            auto scales_of = [&](const uint32_t (&r)[4], float& s0, float& s8, float& b0, float& b8) -> bool {
                b0 = b8 = 0.0f;
                if constexpr (FMT == QM_AFFINE) {
                    s0 = sval<SDT>(r[0]);
                    s8 = sval<SDT>(r[1]);
                    b0 = sval<SDT>(r[2]);
                    b8 = sval<SDT>(r[3]);
                    return fmaxf(fmaxf(fabsf(s0), fabsf(s8)), fmaxf(fabsf(b0), fabsf(b8))) >= 0x1p87f;
                } else if constexpr (FMT == QM_Q8_0) {
                    s0 = f16_bits_to_f32(r[0]);
                    s8 = f16_bits_to_f32(r[1]);
                    return fmaxf(fabsf(s0), fabsf(s8)) > 0x1p127f;  // an infinite d
                } else {
                    e8m0x2_to_f32(r[0] | (r[1] << 8), s0, s8);
                    return max(r[0], r[1]) >= 220u;  // scales of 2^93 and more
                }
            };
            uint32_t big = xbad ? 3u : 0u;  // bit tt: tile tt is summed element by element this stage
            // the group's sums, at the activations' 2^E scale, into y
            auto epilogue = [&](int gi, const float (&acc)[2][NT][4], const uint32_t (&raw)[2][4]) {
                float4 td[NT];  // (O[2t], X[2t], O[2t+1], X[2t+1]) per token half
                if constexpr (FMT != QM_MXFP4 && FMT != QM_MXFP4_BLOCKS) {
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt)
                        td[nt] = *reinterpret_cast<const float4*>(tok + gi * 16 + nt * 8 + 2 * t);
                }
#pragma unroll
                for (int tt = 0; tt < 2; ++tt) {
                    float s0, s8, b0, b8;
                    if (scales_of(raw[tt], s0, s8, b0, b8)) big |= 1u << tt;
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) {
                        float* yv = y[tt][nt];
                        const float* c = acc[tt][nt];
                        if constexpr (FMT == QM_MXFP4 || FMT == QM_MXFP4_BLOCKS) {
                            yv[0] = fmaf(s0, c[0], yv[0]);
                            yv[2] = fmaf(s8, c[2], yv[2]);
                            if constexpr (!ONE) {
                                yv[1] = fmaf(s0, c[1], yv[1]);
                                yv[3] = fmaf(s8, c[3], yv[3]);
                            }
                        } else {
                            const float4 d = td[nt];
                            yv[0] = fmaf(s0, c[0] - d.x, fmaf(b0, d.y, yv[0]));
                            yv[2] = fmaf(s8, c[2] - d.x, fmaf(b8, d.y, yv[2]));
                            if constexpr (!ONE) {  // odd columns: tokens 2t + 1
                                yv[1] = fmaf(s0, c[1] - d.z, fmaf(b0, d.w, yv[1]));
                                yv[3] = fmaf(s8, c[3] - d.z, fmaf(b8, d.w, yv[3]));
                            }
                        }
                    }
                }
            };
            // tile tt's sums over the stage's groups [g0, g1), element by element
            // at float32 (rare: kept out of the streaming loop)
            auto exact_tile = [&](int tt, int g0, int g1) {
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int i = 0; i < 4; ++i) y[tt][nt][i] = 0.0f;
                #pragma unroll 1
                for (int gi = g0; gi < g1; ++gi) {
                    uint32_t raw[2][4];
                    ep_load(gi, raw);
                    float s0, s8, b0, b8;
                    (void)scales_of(raw[tt], s0, s8, b0, b8);
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            const int m = nt * 8 + 2 * t + h;
                            if ((ONE && (t != 0 || h != 0)) || m >= M) continue;
                            const int64_t xr = p.g_off ? s_xrow[m] : m;
                            const float2 e = group_exact<FMT, BITS, GS>(rows_[2 * tt], rows_[2 * tt + 1], gi, s0, b0,
                                                                        s8, b8, p.x + xr * p.k + xk0 + gi * GS);
                            y[tt][nt][h] += e.x;
                            y[tt][nt][2 + h] += e.y;
                        }
                }
            };
            // groups two at a time: four independent MMA chains in flight
            const int gend = live ? ge : gb;
            int gi = gb;
            #pragma unroll 1
            for (; gi + 1 < gend; gi += 2) {
                uint32_t raw0[2][4], raw1[2][4];
                ep_load(gi, raw0);
                ep_load(gi + 1, raw1);
                float acc0[2][NT][4], acc1[2][NT][4];
                do_group(gi, acc0);
                do_group(gi + 1, acc1);
                epilogue(gi, acc0, raw0);
                epilogue(gi + 1, acc1, raw1);
            }
            if (gi < gend) {
                uint32_t raw0[2][4];
                ep_load(gi, raw0);
                float acc0[2][NT][4];
                do_group(gi, acc0);
                epilogue(gi, acc0, raw0);
            }
            // the stage's sums at their true size: one power-of-two product per
            // output (exact), or the element-by-element sums of a big tile; both
            // before the stage's slot is released
#pragma unroll
            for (int tt = 0; tt < 2; ++tt) {
                if (big & (1u << tt)) {
                    exact_tile(tt, gb, gend);
                } else {
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) {
                        y[tt][nt][0] *= tk[nt][0];
                        y[tt][nt][2] *= tk[nt][0];
                        y[tt][nt][1] *= tk[nt][1];
                        y[tt][nt][3] *= tk[nt][1];
                    }
                }
            }
            __syncwarp();
            if (lane == 0 && live) mbar_arrive(bar_empty0 + 8 * slot);

            // ---- the team's sum in warp order, spread over the team's warps;
            //      then undo the token scale and store
            const int64_t row0 = (stage0 + j) * kRows;
            auto store = [&](int tt, int nt, int ln, int i, float v) {
                const int m = nt * 8 + 2 * (ln & 3) + (i & 1);
                const int r = 16 * tt + (ln >> 2) + ((i & 2) ? 8 : 0);
                if (S == 1) {
                    if (m < M && row0 + r < p.n) {
                        __nv_bfloat16 bv = __float2bfloat16_rn(v);
                        const int64_t yr = p.g_off ? s_pos[m] : m;
                        p.y[yr * p.n + row0 + r] = *reinterpret_cast<uint16_t*>(&bv);
                    }
                } else {
                    partial[(j * kRows + r) * 16 + m] = v;
                }
            };
            if constexpr (ONE) {
                // one token: a warp's partial is 32 floats, one per row of the
                // stage, held by the lanes with t = 0 (column 0 of each tile)
                float* base = red + ((team * 2 + buf) * T) * 32;
                if (t == 0) {
                    float* mine = base + wi * 32;
#pragma unroll
                    for (int tt = 0; tt < 2; ++tt) {
                        mine[16 * tt + g] = y[tt][0][0];
                        mine[16 * tt + g + 8] = y[tt][0][2];
                    }
                }
                named_bar_sync(2 + team, T * 32);
                if (live && !s_abort) {
                    const int e = wi * (32 / T) + lane;  // warp wi adds rows [wi*32/T, (wi+1)*32/T)
                    if (lane < 32 / T) {
                        float sum = 0.0f;
#pragma unroll 1
                        for (int q = 0; q < T; ++q) sum += base[q * 32 + e];
                        const float v = sum;
                        if (S == 1) {
                            if (row0 + e < p.n) {
                                __nv_bfloat16 bv = __float2bfloat16_rn(v);
                                const int64_t yr = p.g_off ? s_pos[0] : 0;
                                p.y[yr * p.n + row0 + e] = *reinterpret_cast<uint16_t*>(&bv);
                            }
                        } else {
                            partial[(j * kRows + e) * 16] = v;
                        }
                    }
                }
                buf ^= 1;
            } else {
                // red[team][buf][warp of team][tt][nt][lane][4] (a team of one
                // goes through it too: one store loop instead of an unrolled one)
                constexpr int E = 2 * NT * 32 * 4;  // floats per warp partial
                float* base = red + ((team * 2 + buf) * T) * E;
                float* mine = base + wi * E;
#pragma unroll
                for (int tt = 0; tt < 2; ++tt)
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt)
                        *reinterpret_cast<float4*>(mine + ((tt * NT + nt) * 32 + lane) * 4) =
                            make_float4(y[tt][nt][0], y[tt][nt][1], y[tt][nt][2], y[tt][nt][3]);
                named_bar_sync(2 + team, T * 32);
                if (live && !s_abort) {
                    // warp wi adds entries [wi*E/T, (wi+1)*E/T) over the team's warps in order
                    #pragma unroll 1
                    for (int e = wi * (E / T) + lane; e < (wi + 1) * (E / T); e += 32) {
                        float sum = 0.0f;
                        #pragma unroll 1
                        for (int q = 0; q < T; ++q) sum += base[q * E + e];
                        const int i = e & 3, ln = (e >> 2) & 31, tn = e >> 7;
                        store(tn / NT, tn % NT, ln, i, sum);
                    }
                }
                buf ^= 1;
            }
        }
    }

    // ---------------------------------------------------------------- split-k reduction
    // The CTAs of rank 1.. push their sums into rank 0's receive area with
    // asynchronous stores that count against rank 0's barrier, and leave;
    // rank 0 adds them in rank order and stores y.
    if (S > 1) {
        __syncthreads();  // this CTA's partial sums are complete
        cluster_wait();   // rank 0's barrier is initialized
        const int ent = nst * kRows * M;  // [row][token] of this cluster's stages
        const float* own = reinterpret_cast<const float*>(smem + p.off_xraw);  // [row][16]
        if (rank != 0) {
            const uint32_t dst = map_shared_rank(smem_u32(smem + p.off_recv), 0) + (rank - 1) * ent * 4u;
            const uint32_t rbar = map_shared_rank(bar_red, 0);
            #pragma unroll 1
            for (int e = threadIdx.x; e < ent; e += blockDim.x)
                st_async_f32(dst + 4u * e, own[(e / M) * 16 + e % M], rbar);
        } else {
            if (threadIdx.x == 0) {
                mbar_expect_tx(bar_red, static_cast<uint32_t>((S - 1) * ent * 4));
                mbar_arrive(bar_red);
            }
            const bool ok = mbar_wait(bar_red, 0);
            if (!ok && threadIdx.x == 0) atomicOr(&g_err_gemv, DEV_ERR_TIMEOUT);
            const float* recv = reinterpret_cast<const float*>(smem + p.off_recv);  // [rank - 1][ent]
            #pragma unroll 1
            for (int e = threadIdx.x; ok && e < ent; e += blockDim.x) {
                const int rr = e / M, m = e % M;
                const int64_t row = stage0 * kRows + rr;
                if (row >= p.n) continue;
                float sum = 0.0f;
                sum += own[rr * 16 + m];
                #pragma unroll 1
                for (int q = 1; q < S; ++q) sum += recv[(q - 1) * ent + e];
                __nv_bfloat16 b = __float2bfloat16_rn(sum);
                const int64_t yr = p.g_off ? s_pos[m] : m;
                p.y[yr * p.n + row] = *reinterpret_cast<uint16_t*>(&b);
            }
        }
    }
}

// ---------------------------------------------------------------- host planning
struct Plan {
    Params p;
    int S = 1;
    int cw = 8;  // consumer warps
    int64_t grid = 0;
    size_t smem = 0;
    bool ok = false;
};

static uint32_t round_up(uint64_t v, uint64_t a) { return static_cast<uint32_t>((v + a - 1) / a * a); }

// Bytes of codes for `kk` values of one row.
static int64_t code_bytes(const WDesc& w, int64_t kk) {
    if (w.fmt == QM_Q8_0) return kk / 32 * 34;
    if (w.fmt == QM_MXFP4_BLOCKS) return kk / 32 * 17;
    return kk * w.bits / 8;
}

__global__ void cluster_probe_kernel() {}

// Clusters of S CTAs (`threads` threads and `smem` bytes each) that can be
// resident at once; cached per (device, S, CTAs per SM), which fixes the other two.
static int max_clusters(int S, int per_sm, int threads, size_t smem) {
    static int cache[64][9][2];
    int dev = 0;
    cudaGetDevice(&dev);
    if (S <= 1) return num_sms();
    int* slot = (dev >= 0 && dev < 64) ? &cache[dev][S][per_sm - 1] : nullptr;
    if (slot && *slot > 0) return *slot;
    int n = 0;
    cudaFuncSetAttribute(cluster_probe_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         static_cast<int>(smem));
    cudaFuncSetAttribute(cluster_probe_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(S * 64);
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute a;
    a.id = cudaLaunchAttributeClusterDimension;
    a.val.clusterDim.x = S;
    a.val.clusterDim.y = 1;
    a.val.clusterDim.z = 1;
    cfg.attrs = &a;
    cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&n, cluster_probe_kernel, &cfg) != cudaSuccess || n <= 0) {
        cudaGetLastError();
        n = num_sms() / S;
    }
    if (slot) *slot = n;
    return n;
}

// A plan for S CTAs per cluster (splitting k) and `per_sm` CTAs per SM, the
// matrix getting `share` of the GPU's CTA slots (other chunks of a grouped
// product take the rest).
static bool plan_for(const WDesc& w, int64_t M, int S, int per_sm, Plan* out, double share = 1.0) {
    if (w.k % S) return false;
    const int64_t kr = w.k / S;
    if (kr % w.gs) return false;
    const int NT = M > 8 ? 2 : 1;
    const int64_t cseg = code_bytes(w, kr);
    if (cseg % 16 || w.code_row_bytes % 16) return false;
    int64_t sseg = 0;
    if (w.fmt == QM_AFFINE) sseg = kr / w.gs * 2;
    if (w.fmt == QM_MXFP4) sseg = kr / 32;
    // scales by 2-d boxes of this CTA's part, where a box can take it; else
    // whole rows as a span (k whole, or a part that is no 16-byte multiple)
    const bool boxes = S > 1 && sseg % 16 == 0 && sseg <= 256 && w.scale_row_bytes % 16 == 0;
    if (S > 1 && !boxes && M > 1) return false;  // whole scale rows per rank: measured slower with several tokens
    Params& p = out->p;
    p = Params{};
    p.code_seg = static_cast<uint32_t>(cseg);
    p.nbox = static_cast<uint32_t>((cseg + 127) / 128);
    p.scale_seg = static_cast<uint32_t>(sseg);
    p.scale_span = boxes ? 0 : 1;
    p.scale_pitch = static_cast<uint32_t>(boxes ? sseg : w.scale_row_bytes);
    const uint32_t codes_bytes = p.nbox * kRows * 128;
    const uint32_t sc_bytes = round_up(kRows * (sseg ? p.scale_pitch : 0), 128);
    p.off_scales = codes_bytes;
    p.off_biases = codes_bytes + sc_bytes;
    p.stage_bytes = round_up(codes_bytes + sc_bytes * (w.fmt == QM_AFFINE ? 2 : 1), 1024);  // swizzled boxes
    const int64_t groups = kr / w.gs;
    const int64_t budget = (per_sm == 2 ? (max_smem_optin() + 1024) / 2 : max_smem_optin()) - 1024;
    // work split: clusters of S CTAs, per_sm CTAs to an SM
    p.n_stages = (w.n + kRows - 1) / kRows;
    const int cw = per_sm == 1 ? 16 : 8;
    int64_t G = std::max<int64_t>(1, static_cast<int64_t>(num_sms() * per_sm * share) / S);
    if (S > 1) G = std::max<int64_t>(1, std::min<int64_t>(G, max_clusters(S, per_sm, kThreadsOf(cw), budget)));
    G = std::min<int64_t>(G, p.n_stages);
    const int64_t spc = (p.n_stages + G - 1) / G;
    G = (p.n_stages + spc - 1) / spc;
    // shared memory: fixed part, then as many stage slots as fit
    auto layout = [&]() -> int64_t {
        p.off_tokscale = 512;  // [16] 2^-E, [16] unused, [16] max |x| bits
        p.off_tok = p.off_tokscale + 256;
        p.off_xfrag = round_up(p.off_tok + groups * 16 * 8, 128);
        // B fragments: 16 bytes per k value and token tile, or 2 for exactly one token
        const uint64_t xfrag_bytes = M == 1 ? static_cast<uint64_t>(kr) * 2 : static_cast<uint64_t>(kr) * 16 * NT;
        const uint64_t red_bytes = M == 1 ? static_cast<uint64_t>(cw) * 2 * 32 * 4
                                          : static_cast<uint64_t>(cw) * 2 * 2 * NT * 32 * 4 * 4;
        const uint64_t partial_bytes = S > 1 ? static_cast<uint64_t>(spc) * kRows * 16 * 4 : 0;
        const uint64_t xraw_bytes = static_cast<uint64_t>(M) * kr * 2;
        // The raw activations are dead once the fragments are built (a barrier of
        // all consumers), so the team sums, which start after it, reuse their
        // room; with a k split the stages' partial sums take that room instead.
        p.off_xraw = round_up(p.off_xfrag + xfrag_bytes, 128);
        uint64_t end;
        if (S == 1) {
            p.off_red = p.off_xraw;
            end = p.off_xraw + std::max(xraw_bytes, red_bytes);
        } else {
            p.off_red = round_up(p.off_xraw + std::max(partial_bytes, xraw_bytes), 128);
            end = p.off_red + red_bytes;
        }
        // split k: rank 0 receives the other ranks' sums apart from everything it may still be reading
        const uint64_t recv_bytes = S > 1 ? static_cast<uint64_t>(S - 1) * spc * kRows * M * 4 : 0;
        p.off_recv = round_up(end, 128);
        p.off_stages = round_up(p.off_recv + recv_bytes, 1024);
        const int64_t room = budget - p.off_stages;
        return std::min<int64_t>(std::min<int64_t>(kMaxStages, room / p.stage_bytes), std::max<int64_t>(2, spc));
    };
    const int64_t nst = layout();
    if (nst < 2) return false;
    // teams: one per stage a CTA can hold in flight, each warp at least one group
    int teams = 1;
    while (teams * 2 <= kMaxTeams && teams * 2 <= spc && teams * 2 <= nst) teams *= 2;
    int T = cw / teams;
    while (T > 1 && T > groups && cw / (T / 2) <= kMaxTeams) T /= 2;
    p.team = T;
    p.nstage = static_cast<uint32_t>(nst);
    p.S = S;
    p.krange = kr;
    p.stages_per_cluster = static_cast<int>(spc);
    out->S = S;
    out->cw = cw;
    out->grid = G * S;
    out->smem = p.off_stages + nst * p.stage_bytes;
    out->ok = true;
    return true;
}

// Pick the k split and CTAs per SM: least per-CTA work (stages x k range,
// halved where two CTAs share an SM) plus a fixed cost per extra rank of a k
// split, then fewest splits; a plan that keeps three stages in flight beats
// one that cannot.
static Plan make_plan(const WDesc& w, int64_t M, double share = 1.0) {
    Plan best;
    double best_cost = 1e300;
    for (int per_sm = 2; per_sm >= 1; --per_sm)
        for (int S = 1; S <= 8; ++S) {
            Plan pl;
            if (!plan_for(w, M, S, per_sm, &pl, share)) continue;
            const bool shallow = pl.p.nstage < 3 && pl.p.stages_per_cluster >= 3;
            // one token: each extra rank of a k split costs a fixed hand-off
            // (its partial sums reach rank 0 through distributed shared memory),
            // measured on GB300 to be worth about 1024 k values of one stage; with
            // more tokens the activation work per CTA favors the wider splits
            const double cost = static_cast<double>(pl.p.stages_per_cluster) * pl.p.krange / per_sm *
                                    (1.0 + 0.03 * (S - 1)) * (shallow ? 2.0 : 1.0) +
                                (M == 1 ? 1024.0 * (S - 1) : 0.0);
            if (cost < best_cost * 0.999) {
                best_cost = cost;
                best = pl;
            }
        }
    return best;
}

template <int FMT, int BITS, int GS, int NTK, int SDT, int CW>
static cudaError_t launch_k(const Plan& pl, cudaStream_t st) {
    auto kern = gemv_kernel<FMT, BITS, GS, NTK, SDT, CW>;
    // the kernel's attributes, once per device: the most dynamic shared memory
    // any plan may ask for, and clusters past the portable size
    static std::atomic<uint64_t> configured{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = dev < 64 ? (uint64_t(1) << dev) : 0;
    if (!bit || !(configured.load(std::memory_order_acquire) & bit)) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem_optin());
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return e;
        configured.fetch_or(bit, std::memory_order_acq_rel);
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(pl.grid));
    cfg.blockDim = dim3(kThreadsOf(CW));
    cfg.dynamicSmemBytes = pl.smem;
    cfg.stream = st;
    cudaLaunchAttribute attrs[2];
    int na = 0;
    attrs[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attrs[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
    if (pl.S > 1) {
        attrs[na].id = cudaLaunchAttributeClusterDimension;
        attrs[na].val.clusterDim.x = pl.S;
        attrs[na].val.clusterDim.y = 1;
        attrs[na].val.clusterDim.z = 1;
        ++na;
    }
    cfg.attrs = attrs;
    cfg.numAttrs = na;
    return cudaLaunchKernelEx(&cfg, kern, pl.p);
}

template <int FMT, int BITS, int GS, int NTK, int CW>
static cudaError_t launch_c(const Plan& pl, cudaStream_t st) {
    if constexpr (FMT == QM_AFFINE) {
        if (pl.p.sdt == QM_F16) return launch_k<FMT, BITS, GS, NTK, QM_F16, CW>(pl, st);
    }
    return launch_k<FMT, BITS, GS, NTK, QM_BF16, CW>(pl, st);
}

template <int FMT, int BITS, int GS, int NTK>
static cudaError_t launch_t(const Plan& pl, cudaStream_t st) {
    return pl.cw == 16 ? launch_c<FMT, BITS, GS, NTK, 16>(pl, st) : launch_c<FMT, BITS, GS, NTK, 8>(pl, st);
}

}  // namespace gemv

namespace gemv {

// A plan with the weight's fields and tensor maps filled in: everything of a
// launch that depends only on the weight descriptor, M and the device.
struct Prepared {
    Plan pl;
    bool maps = false;  // the driver encoded the tensor maps (else the plain kernel runs)
};

static void prepare(const WDesc& w, int64_t M, Prepared* out) {
    out->pl = make_plan(w, M);
    out->maps = false;
    if (!out->pl.ok) return;
    Params& p = out->pl.p;
    p.codes = w.codes;
    p.scales = w.scales;
    p.biases = w.biases;
    p.n = w.n;
    p.k = w.k;
    p.M = static_cast<int>(M);
    p.sdt = w.sdt;
    p.code_row_bytes = w.code_row_bytes;
    p.scale_row_bytes = w.scale_row_bytes;
    p.static_w = w.is_static ? 1 : 0;
    bool maps = make_tmap_2d(&p.tm_codes, w.codes, w.code_row_bytes, w.n, w.code_row_bytes, 128, kRows, true);
    if (maps && !p.scale_span && p.scale_seg) {
        maps = make_tmap_2d(&p.tm_scales, w.scales, w.scale_row_bytes, w.n, w.scale_row_bytes, p.scale_seg,
                            kRows, false);
        if (maps && w.biases)
            maps = make_tmap_2d(&p.tm_biases, w.biases, w.scale_row_bytes, w.n, w.scale_row_bytes, p.scale_seg,
                                kRows, false);
    }
    out->maps = maps;
}

// What a prepared plan depends on, with no padding bytes (compared bytewise).
struct PlanKey {
    const void* codes;
    const void* scales;
    const void* biases;
    int64_t n, k, code_row_bytes, scale_row_bytes;
    int32_t fmt, bits, gs, sdt, M, is_static, dev, unused;
};
static_assert(sizeof(PlanKey) == 3 * 8 + 4 * 8 + 8 * 4, "PlanKey has padding");

struct PlanKeyHash {
    size_t operator()(const PlanKey& k) const {
        uint64_t h = 1469598103934665603ull;  // FNV-1a over the key's bytes
        const unsigned char* b = reinterpret_cast<const unsigned char*>(&k);
        for (size_t i = 0; i < sizeof k; ++i) h = (h ^ b[i]) * 1099511628211ull;
        return static_cast<size_t>(h);
    }
};
struct PlanKeyEq {
    bool operator()(const PlanKey& a, const PlanKey& b) const { return std::memcmp(&a, &b, sizeof a) == 0; }
};

// Prepared plans, memoized per calling thread: a decode step calls the same
// few hundred (weight, M) pairs over and over, and planning plus tensor-map
// encoding costs microseconds of host time per call. Only host-side launch
// metadata is kept (at most kMaxPlans entries, then the table starts over);
// no device memory is held.
static const Prepared* prepared(const WDesc& w, int64_t M, cudaError_t* err = nullptr) {
    PlanKey key;
    std::memset(&key, 0, sizeof key);
    key.codes = w.codes;
    key.scales = w.scales;
    key.biases = w.biases;
    key.n = w.n;
    key.k = w.k;
    key.code_row_bytes = w.code_row_bytes;
    key.scale_row_bytes = w.scale_row_bytes;
    key.fmt = w.fmt;
    key.bits = w.bits;
    key.gs = w.gs;
    key.sdt = w.sdt;
    key.M = static_cast<int32_t>(M);
    key.is_static = w.is_static ? 1 : 0;
    const cudaError_t e = cudaGetDevice(&key.dev);
    if (e != cudaSuccess) {
        if (err) *err = e;
        return nullptr;
    }
    constexpr size_t kMaxPlans = 4096;
    thread_local std::unordered_map<PlanKey, Prepared, PlanKeyHash, PlanKeyEq> table;
    auto it = table.find(key);
    if (it != table.end()) return &it->second;
    if (table.size() >= kMaxPlans) table.clear();
    Prepared& pr = table[key];
    prepare(w, M, &pr);
    return &pr;
}

}  // namespace gemv

bool gemv_supported(const WDesc& w, int64_t M) {
    if (M < 1 || M > 16 || w.ndim != 2 || !pipelined_format(w)) return false;
    const gemv::Prepared* pr = gemv::prepared(w, M);
    return pr && pr->pl.ok;
}

qm_status launch_gemv(const WDesc& w, const void* x, int64_t M, void* y, cudaStream_t st) {
    using namespace gemv;
    cudaError_t err = cudaSuccess;
    const Prepared* pr = prepared(w, M, &err);
    if (!pr) return cuda_fail(err, "cudaGetDevice");
    if (!pr->pl.ok) return fail(QM_ENOTSUP, "w: no decode plan for this shape");
    if (!pr->maps) {  // the driver refused a descriptor for this shape: the plain kernel
        cudaError_t e = launch_apply_simple(w, x, M, y, st);
        return e == cudaSuccess ? QM_OK : cuda_fail(e, "apply launch");
    }
    Plan pl = pr->pl;
    Params& p = pl.p;
    p.x = static_cast<const uint16_t*>(x);
    p.y = static_cast<uint16_t*>(y);
    const int ntk = M > 8 ? 2 : (M > 1 ? 1 : 0);
    cudaError_t e = cudaErrorInvalidValue;
#define QM_GEMV_CASE(F, B, G)                                                                  \
    if (w.fmt == F && (F != QM_AFFINE || (w.bits == B && w.gs == G))) {                         \
        e = ntk == 2 ? launch_t<F, B, G, 2>(pl, st)                                            \
                     : (ntk == 1 ? launch_t<F, B, G, 1>(pl, st) : launch_t<F, B, G, 0>(pl, st)); \
        goto done;                                                                             \
    }
    QM_GEMV_CASE(QM_AFFINE, 4, 32)
    QM_GEMV_CASE(QM_AFFINE, 4, 64)
    QM_GEMV_CASE(QM_AFFINE, 4, 128)
    QM_GEMV_CASE(QM_AFFINE, 8, 32)
    QM_GEMV_CASE(QM_AFFINE, 8, 64)
    QM_GEMV_CASE(QM_AFFINE, 8, 128)
    QM_GEMV_CASE(QM_Q8_0, 8, 32)
    QM_GEMV_CASE(QM_MXFP4, 4, 32)
    QM_GEMV_CASE(QM_MXFP4_BLOCKS, 4, 32)
#undef QM_GEMV_CASE
done:
    if (e != cudaSuccess) return cuda_fail(e, "gemv launch");
    return QM_OK;
}

// ---------------------------------------------------------------- grouped (apply_experts)
// Chunks of Q routed positions of one expert, each a decode product over that
// expert's [n, k] matrix. The chunk list lives on the device (the routing
// offsets), so the grid covers the most chunks P positions can make; slots
// past the last chunk exit at once.
namespace gemv {

static int grouped_q(int64_t P, int64_t E) { return P <= 8 * E ? 8 : 16; }

static bool grouped_plan(const WDesc& w, int64_t P, Plan* out, int64_t* slots) {
    const int64_t E = w.shape[0];
    if (w.ndim != 3 || E < 1 || P < 1 || E * w.n >= (int64_t(1) << 31) || !pipelined_format(w)) return false;
    if ((w.n * w.scale_row_bytes) % 16) return false;  // each expert's scales start 16-byte aligned
    const int Q = grouped_q(P, E);
    *slots = std::min<int64_t>(P, P / Q + E);  // sum over experts of ceil(count / Q) is below P/Q + E
    // chunks expected when ids spread evenly: every expert used, about half a chunk extra each
    const int64_t est = std::max<int64_t>(1, std::min<int64_t>(*slots, (P + Q - 1) / Q + std::min(E, P) / 2));
    *out = make_plan(w, Q, 1.0 / static_cast<double>(est));
    return out->ok;
}

}  // namespace gemv

bool gemv_grouped_supported(const WDesc& w, int64_t P) {
    gemv::Plan pl;
    int64_t slots = 0;
    return gemv::grouped_plan(w, P, &pl, &slots);
}

qm_status launch_gemv_grouped(const WDesc& w, const int32_t* offsets, const int32_t* perm, int64_t P,
                              int xdiv, const void* x, void* y, cudaStream_t st) {
    using namespace gemv;
    Plan pl;
    int64_t slots = 0;
    if (!grouped_plan(w, P, &pl, &slots)) return fail(QM_ENOTSUP, "w: no grouped decode plan for this shape");
    const int64_t E = w.shape[0];
    const int Q = grouped_q(P, E);
    Params& p = pl.p;
    p.codes = w.codes;
    p.scales = w.scales;
    p.biases = w.biases;
    p.x = static_cast<const uint16_t*>(x);
    p.y = static_cast<uint16_t*>(y);
    p.n = w.n;
    p.k = w.k;
    p.M = Q;
    p.sdt = w.sdt;
    p.code_row_bytes = w.code_row_bytes;
    p.scale_row_bytes = w.scale_row_bytes;
    p.static_w = 0;
    p.g_off = offsets;
    p.g_perm = perm;
    p.g_E = static_cast<int>(E);
    p.g_Q = Q;
    p.g_xdiv = xdiv;
    p.g_wclusters = static_cast<int>(pl.grid / pl.S);
    const int64_t rows = E * w.n;
    bool maps = make_tmap_2d(&p.tm_codes, w.codes, w.code_row_bytes, rows, w.code_row_bytes, 128, kRows, true);
    if (maps && !p.scale_span && p.scale_seg) {
        maps = make_tmap_2d(&p.tm_scales, w.scales, w.scale_row_bytes, rows, w.scale_row_bytes, p.scale_seg,
                            kRows, false);
        if (maps && w.biases)
            maps = make_tmap_2d(&p.tm_biases, w.biases, w.scale_row_bytes, rows, w.scale_row_bytes, p.scale_seg,
                                kRows, false);
    }
    if (!maps) return fail(QM_ENOTSUP, "w: no tensor map for the grouped decode product");
    if (pl.grid * slots >= (int64_t(1) << 31)) return fail(QM_ENOTSUP, "ids: too many positions for one launch");
    pl.grid *= slots;
    const bool two = Q > 8;
    cudaError_t e = cudaErrorInvalidValue;
#define QM_GEMV_CASE(F, B, G)                                                                  \
    if (w.fmt == F && (F != QM_AFFINE || (w.bits == B && w.gs == G))) {                         \
        e = two ? launch_t<F, B, G, 2>(pl, st) : launch_t<F, B, G, 1>(pl, st);                 \
        goto done;                                                                             \
    }
    QM_GEMV_CASE(QM_AFFINE, 4, 32)
    QM_GEMV_CASE(QM_AFFINE, 4, 64)
    QM_GEMV_CASE(QM_AFFINE, 4, 128)
    QM_GEMV_CASE(QM_AFFINE, 8, 32)
    QM_GEMV_CASE(QM_AFFINE, 8, 64)
    QM_GEMV_CASE(QM_AFFINE, 8, 128)
    QM_GEMV_CASE(QM_Q8_0, 8, 32)
    QM_GEMV_CASE(QM_MXFP4, 4, 32)
    QM_GEMV_CASE(QM_MXFP4_BLOCKS, 4, 32)
#undef QM_GEMV_CASE
done:
    if (e != cudaSuccess) return cuda_fail(e, "grouped gemv launch");
    return QM_OK;
}

}  // namespace qm
