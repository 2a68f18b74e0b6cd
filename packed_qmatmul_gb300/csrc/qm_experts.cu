// qm_experts.cu -- apply_experts: routing (a stable counting sort of the
// flattened positions by expert id) and the segmented product.
//
// "Nx_quant (raven-ml.dev API docs)", section "Products", val apply_experts:
// each position's row goes through the expert its id names, zeros where the
// id is outside [0, E) whatever the row holds; the positions in range are
// summed in one segmented contraction, and a row's bits do not depend on the
// other positions' experts. Routing order is ours: ascending expert, ties by
// ascending position, so the sort is deterministic.
#include <cuda_runtime.h>

#include <algorithm>
#include <mutex>
#include <string>

#include "qm_device.cuh"
#include "qm_internal.h"

namespace qm {

static __device__ uint32_t g_err_experts = 0;

uint32_t experts_read_clear_error() {
    uint32_t v = 0, z = 0;
    cudaMemcpyFromSymbol(&v, g_err_experts, sizeof(v));
    cudaMemcpyToSymbol(g_err_experts, &z, sizeof(z));
    return v;
}

namespace {

constexpr int kChunk = 1024;  // positions per routing CTA

QM_DEV int64_t load_id(const void* ids, int id64, int64_t p) {
    return id64 ? __ldg(static_cast<const int64_t*>(ids) + p)
                : static_cast<int64_t>(__ldg(static_cast<const int32_t*>(ids) + p));
}

size_t round256(size_t v) { return (v + 255) / 256 * 256; }

// Workspace layout for P positions over E experts, plus `xs_bytes` for the
// routed activation rows where the tensor-core path takes them.
struct WsLayout {
    size_t counts, offsets, perm, chunk_counts, xs, total;
};

WsLayout ws_layout(int64_t P, int64_t E, size_t xs_bytes = 0) {
    WsLayout l;
    const int64_t nchunks = (P + kChunk - 1) / kChunk;
    l.counts = 0;
    l.offsets = round256(static_cast<size_t>(E) * 4);
    l.perm = l.offsets + round256(static_cast<size_t>(E + 1) * 4);
    l.chunk_counts = l.perm + round256(static_cast<size_t>(P) * 4);
    l.xs = l.chunk_counts + round256(static_cast<size_t>(nchunks) * E * 4);
    l.total = l.xs + round256(xs_bytes);
    return l;
}

// How the segmented product runs, from the shapes alone (never from the ids,
// so a row's bits cannot depend on the other positions' experts).
enum class Path { kSimple, kDecode, kTensor };

Path experts_path(const WDesc& w, int64_t P, bool allow_tensor) {
    const int64_t E = w.shape[0];
    const bool decode = gemv_grouped_supported(w, P);
    if (decode && P <= 32 * E) return Path::kDecode;   // few positions per expert: HBM-bound
    if (allow_tensor && gemm_grouped_supported(w, P)) return Path::kTensor;
    return decode ? Path::kDecode : Path::kSimple;
}

// Routed activation rows: xs[i] = x[perm[i] / xdiv] for the n_in = offsets[E]
// positions in range, one warp per row in 16-byte pieces.
__global__ void __launch_bounds__(256) gather_rows_kernel(const int32_t* n_in_p, const int32_t* perm, int xdiv,
                                                          const uint4* x, int64_t row_vecs, uint4* xs) {
    grid_launch_dependents();
    grid_dependency_wait();
    const int64_t n_in = *n_in_p;
    const int lane = threadIdx.x & 31;
    const int64_t nw = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    for (int64_t i = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; i < n_in; i += nw) {
        const int64_t src = __ldg(perm + i) / xdiv;
        const uint4* a = x + src * row_vecs;
        uint4* b = xs + i * row_vecs;
        for (int64_t v = lane; v < row_vecs; v += 32) b[v] = __ldg(a + v);
    }
}

// Per-chunk histogram of in-range ids: chunk_counts[chunk][e].
__global__ void __launch_bounds__(256) route_count_kernel(const void* ids, int id64, int64_t P,
                                                          int64_t E, int32_t* chunk_counts) {
    grid_launch_dependents();
    grid_dependency_wait();  // ids may come from the previous kernel
    extern __shared__ int32_t cnt[];
    for (int64_t e = threadIdx.x; e < E; e += blockDim.x) cnt[e] = 0;
    __syncthreads();
    const int64_t c0 = static_cast<int64_t>(blockIdx.x) * kChunk;
    const int64_t c1 = std::min<int64_t>(c0 + kChunk, P);
    for (int64_t p = c0 + threadIdx.x; p < c1; p += blockDim.x) {
        const int64_t e = load_id(ids, id64, p);
        if (e >= 0 && e < E) atomicAdd(&cnt[e], 1);  // integer counts: order-free
    }
    __syncthreads();
    for (int64_t e = threadIdx.x; e < E; e += blockDim.x)
        chunk_counts[static_cast<int64_t>(blockIdx.x) * E + e] = cnt[e];
}

// One warp per chunk: scan the chunk counts into this chunk's start offsets,
// then place the chunk's positions 32 at a time, each step ranking equal ids
// by lane so the order stays stable. With zy set, the rows of zy [P, zn] at
// out-of-range positions are cleared on the way (their product is zero).
__global__ void __launch_bounds__(32) route_scatter_kernel(const void* ids, int id64, int64_t P,
                                                           int64_t E, const int32_t* chunk_counts,
                                                           int32_t* counts, int32_t* offsets,
                                                           int32_t* perm, uint16_t* zy, int64_t zn) {
    grid_launch_dependents();
    grid_dependency_wait();
    extern __shared__ int32_t sm[];
    int32_t* base = sm;           // [E + 1]: where this chunk's positions of expert e start
    int32_t* run = sm + E + 1;    // [E + 1]: how many of them are placed so far
    const int lane = threadIdx.x;
    const int64_t chunk = blockIdx.x, nchunks = gridDim.x;
    int32_t carry = 0, out_before = 0;
    for (int64_t e0 = 0; e0 < E; e0 += 32) {
        const int64_t e = e0 + lane;
        int32_t total = 0, before = 0;
        if (e < E) {
            for (int64_t c = 0; c < nchunks; ++c) {
                const int32_t v = chunk_counts[c * E + e];
                total += v;
                if (c < chunk) before += v;
            }
        }
        int32_t inc = total;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int32_t t = __shfl_up_sync(0xffffffffu, inc, o);
            if (lane >= o) inc += t;
        }
        if (e < E) {
            base[e] = carry + inc - total + before;
            run[e] = 0;
            if (chunk == 0) {
                counts[e] = total;
                offsets[e] = carry + inc - total;
            }
        }
        carry += __shfl_sync(0xffffffffu, inc, 31);
    }
    // out-of-range positions of earlier chunks
    for (int64_t c = lane; c < chunk; c += 32) {
        int32_t in = 0;
        for (int64_t e = 0; e < E; ++e) in += chunk_counts[c * E + e];
        const int64_t size = std::min<int64_t>(kChunk, P - c * kChunk);
        out_before += static_cast<int32_t>(size) - in;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) out_before += __shfl_xor_sync(0xffffffffu, out_before, o);
    if (lane == 0) {
        base[E] = carry + out_before;
        run[E] = 0;
        if (chunk == 0) offsets[E] = carry;
    }
    __syncwarp();
    const int64_t c0 = chunk * kChunk, c1 = std::min<int64_t>(c0 + kChunk, P);
    const uint32_t lt = (1u << lane) - 1u;
    for (int64_t s = c0; s < c1; s += 32) {
        const int64_t p = s + lane;
        const bool valid = p < c1;
        int32_t b = -1;
        if (valid) {
            const int64_t e = load_id(ids, id64, p);
            b = (e >= 0 && e < E) ? static_cast<int32_t>(e) : static_cast<int32_t>(E);
        }
        const uint32_t mask = __match_any_sync(0xffffffffu, b);
        const int32_t rank = __popc(mask & lt);
        if (valid) perm[base[b] + run[b] + rank] = static_cast<int32_t>(p);
        __syncwarp();
        if (valid && (mask & lt) == 0) run[b] += __popc(mask);
        __syncwarp();
        if (zy) {
            uint32_t out = __ballot_sync(0xffffffffu, valid && b == static_cast<int32_t>(E));
            while (out) {
                const int64_t q = s + (__ffs(out) - 1);
                out &= out - 1;
                for (int64_t j = lane; j < zn; j += 32) zy[q * zn + j] = 0;
            }
        }
    }
}

struct ExpArgs {
    const uint8_t* codes;
    const uint8_t* scales;
    const uint8_t* biases;
    int64_t E, n, k;
    int64_t code_row_bytes, scale_row_bytes;
    int gs, sdt;
};

QM_DEV float scale_val(const uint8_t* p, int64_t idx, int sdt) {
    const uint16_t h = reinterpret_cast<const uint16_t*>(p)[idx];
    return sdt == QM_F16 ? f16_bits_to_f32(h) : bf16_bits_to_f32(h);
}

// Float32 value of input i of weight row r (r indexes all E*n rows).
template <int FMT, int BITS>
QM_DEV float value_at(const ExpArgs& a, int64_t r, int64_t i) {
    if constexpr (FMT == QM_AFFINE) {
        const uint32_t* row = reinterpret_cast<const uint32_t*>(a.codes + r * a.code_row_bytes);
        const int64_t bit = i * BITS;
        const int sh = static_cast<int>(bit % 32);
        uint32_t c = row[bit / 32] >> sh;
        if (sh + BITS > 32) c |= row[bit / 32 + 1] << (32 - sh);  // a code across two words
        c &= (1u << BITS) - 1u;
        const int64_t ng = a.k / a.gs;
        return fmaf(static_cast<float>(c), scale_val(a.scales, r * ng + i / a.gs, a.sdt),
                    scale_val(a.biases, r * ng + i / a.gs, a.sdt));
    } else if constexpr (FMT == QM_Q8_0) {
        const uint8_t* blk = a.codes + r * a.code_row_bytes + (i / 32) * 34;
        const float d = f16_bits_to_f32(*reinterpret_cast<const uint16_t*>(blk));
        return d * static_cast<float>(static_cast<int8_t>(blk[2 + i % 32]));
    } else if constexpr (FMT == QM_Q4_K) {
        // ggml's block_q4_K: d, dmin, 12 bytes of 6-bit scales and mins, 128 quant bytes
        const uint8_t* blk = a.codes + r * a.code_row_bytes + (i / 256) * 144;
        const int v = static_cast<int>(i % 256), c = v / 64, rr = v % 64, j = 2 * c + (rr >= 32);
        const float d = f16_bits_to_f32(blk[0] | (blk[1] << 8)), dmin = f16_bits_to_f32(blk[2] | (blk[3] << 8));
        const uint8_t* sb = blk + 4;
        const int sc = j < 4 ? (sb[j] & 63) : ((sb[4 + j] & 15) | ((sb[j - 4] >> 6) << 4));
        const int mn = j < 4 ? (sb[4 + j] & 63) : ((sb[4 + j] >> 4) | ((sb[j] >> 6) << 4));
        const uint8_t byte = blk[16 + 32 * c + rr % 32];
        const int q = rr < 32 ? (byte & 15) : (byte >> 4);
        return fmaf(d * static_cast<float>(sc), static_cast<float>(q), -(dmin * static_cast<float>(mn)));
    } else if constexpr (FMT == QM_Q6_K) {
        // ggml's block_q6_K: 128 bytes of low 4 bits, 64 of high 2 bits, 16 int8 scales, d
        const uint8_t* blk = a.codes + r * a.code_row_bytes + (i / 256) * 210;
        const int v = static_cast<int>(i % 256), h = v / 128, t = (v % 128) / 32, l = v % 32;
        const uint8_t lo = blk[64 * h + l + 32 * (t % 2)];
        const int q = ((t < 2 ? lo : (lo >> 4)) & 15) | (((blk[128 + 32 * h + l] >> (2 * t)) & 3) << 4);
        const float d = f16_bits_to_f32(blk[208] | (blk[209] << 8));
        return d * static_cast<float>(static_cast<int8_t>(blk[192 + 8 * h + 2 * t + l / 16])) *
               static_cast<float>(q - 32);
    } else if constexpr (FMT == QM_MXFP4_BLOCKS) {
        // GGUF's 17-byte block: the scale byte, then byte j holding value j
        // (low nibble) and value j + 16 (high nibble)
        const uint8_t* blk = a.codes + r * a.code_row_bytes + (i / 32) * 17;
        const int t = static_cast<int>(i % 32);
        const uint8_t b = blk[1 + (t & 15)];
        const uint32_t c = t < 16 ? (b & 15) : (b >> 4);
        uint32_t f2[4];
        e2m1x8_to_f16x2(c, f2);  // byte 0 holds the code in its low nibble
        const float v = __half2float(__ushort_as_half(static_cast<unsigned short>(f2[0] & 0xFFFF)));
        return v * e8m0_to_f32(blk[0]);
    } else {
        const uint8_t b = a.codes[r * a.code_row_bytes + i / 2];
        const uint32_t c = (i & 1) ? (b >> 4) : (b & 15);
        uint32_t f2[4];
        e2m1x8_to_f16x2(c, f2);  // byte 0 holds the code in its low nibble
        const float v = __half2float(__ushort_as_half(static_cast<unsigned short>(f2[0] & 0xFFFF)));
        return v * e8m0_to_f32(a.scales[r * a.scale_row_bytes + i / 32]);
    }
}

// Plain segmented product: one warp per (routed position, output row).
template <int FMT, int BITS>
__global__ void __launch_bounds__(256) experts_simple_kernel(ExpArgs a, const void* ids, int id64,
                                                             int64_t P, int64_t topk, int64_t T,
                                                             const uint16_t* x, int64_t x_rows,
                                                             const int32_t* perm,
                                                             const int32_t* offsets, uint16_t* y) {
    const int lane = threadIdx.x & 31;
    const int64_t warp = (blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x) >> 5;
    const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    const int64_t n_in = offsets[a.E];
    for (int64_t job = warp; job < P * a.n; job += nwarps) {
        const int64_t q = job / a.n, j = job % a.n;
        const int64_t p = perm[q];
        float s = 0.0f;
        if (q < n_in) {
            const int64_t e = load_id(ids, id64, p);
            const int64_t xr = (x_rows == T) ? p / topk : p;
            const uint16_t* xp = x + xr * a.k;
            for (int64_t i = lane; i < a.k; i += 32)
                s = fmaf(bf16_bits_to_f32(xp[i]), value_at<FMT, BITS>(a, e * a.n + j, i), s);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
        }
        if (lane == 0) {
            __nv_bfloat16 b = __float2bfloat16_rn(s);
            y[p * a.n + j] = (q < n_in) ? *reinterpret_cast<uint16_t*>(&b) : uint16_t(0);
        }
    }
}

}  // namespace

size_t route_workspace_bytes(int64_t P, int64_t E) {
    if (P <= 0) return 0;
    return ws_layout(P, E).total;
}

size_t experts_workspace_bytes(const WDesc& w, int64_t P, bool allow_tensor) {
    if (P <= 0) return 0;
    const bool tensor = experts_path(w, P, allow_tensor) == Path::kTensor;
    return ws_layout(P, w.shape[0], tensor ? static_cast<size_t>(P) * w.k * 2 : 0).total;
}

cudaError_t launch_route(const void* ids, int id64, int64_t P, int64_t E, int32_t* counts,
                         int32_t* offsets, int32_t* perm, void* ws, cudaStream_t st, uint16_t* zy,
                         int64_t zn) {
    if (P == 0) {
        if (E > 0) {
            cudaError_t e = cudaMemsetAsync(counts, 0, E * 4, st);
            if (e != cudaSuccess) return e;
        }
        return cudaMemsetAsync(offsets, 0, (E + 1) * 4, st);
    }
    const WsLayout l = ws_layout(P, E);  // the routing part comes first whatever follows
    int32_t* chunk_counts = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(ws) + l.chunk_counts);
    const int64_t nchunks = (P + kChunk - 1) / kChunk;
    const size_t sm1 = static_cast<size_t>(E) * 4, sm2 = static_cast<size_t>(E + 1) * 8;
    if (sm2 > 48 * 1024) {
        cudaFuncSetAttribute(route_count_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(sm1));
        cudaFuncSetAttribute(route_scatter_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(sm2));
    }
    cudaError_t e = launch_pdl(route_count_kernel, static_cast<unsigned>(nchunks), 256, sm1, st, ids, id64, P, E,
                               chunk_counts);
    if (e != cudaSuccess) return e;
    return launch_pdl(route_scatter_kernel, static_cast<unsigned>(nchunks), 32, sm2, st, ids, id64, P, E,
                      static_cast<const int32_t*>(chunk_counts), counts, offsets, perm, zy, zn);
}

qm_status launch_experts(const WDesc& w, const void* ids, int id64, int64_t T, int64_t topk,
                         const void* x, int64_t x_rows, void* y, void* ws, size_t ws_bytes,
                         cudaStream_t st, bool allow_tensor) {
    (void)ws_bytes;
    const int64_t P = T * topk, E = w.shape[0];
    const Path path = experts_path(w, P, allow_tensor);
    const WsLayout l = ws_layout(P, E, path == Path::kTensor ? static_cast<size_t>(P) * w.k * 2 : 0);
    uint8_t* wb = static_cast<uint8_t*>(ws);
    int32_t* counts = reinterpret_cast<int32_t*>(wb + l.counts);
    int32_t* offsets = reinterpret_cast<int32_t*>(wb + l.offsets);
    int32_t* perm = reinterpret_cast<int32_t*>(wb + l.perm);
    const int xdiv = x_rows == T ? static_cast<int>(topk) : 1;
    cudaError_t e = launch_route(ids, id64, P, E, counts, offsets, perm, ws, st,
                                 path != Path::kSimple ? static_cast<uint16_t*>(y) : nullptr, w.n);
    if (e != cudaSuccess) return cuda_fail(e, "route launch");
    if (path == Path::kDecode)  // experts averaging few positions: chunks through the decode product
        return launch_gemv_grouped(w, offsets, perm, P, xdiv, x, y, st);
    if (path == Path::kTensor) {  // routed rows gathered expert by expert, then the tensor-core product
        uint4* xs = reinterpret_cast<uint4*>(wb + l.xs);
        const int64_t blocks = std::min<int64_t>((P + 7) / 8, int64_t(num_sms()) * 8);
        e = launch_pdl(gather_rows_kernel, static_cast<unsigned>(blocks), 256, 0, st,
                       static_cast<const int32_t*>(offsets + E), static_cast<const int32_t*>(perm), xdiv,
                       static_cast<const uint4*>(x), static_cast<int64_t>(w.k * 2 / 16), xs);
        if (e != cudaSuccess) return cuda_fail(e, "gather launch");
        return launch_gemm_grouped(w, offsets, perm, P, xs, y, st);
    }
    ExpArgs a{w.codes, w.scales, w.biases, E, w.n, w.k, w.code_row_bytes, w.scale_row_bytes, w.gs, w.sdt};
    const int64_t jobs = P * w.n;
    const int64_t blocks = std::min<int64_t>((jobs * 32 + 255) / 256, int64_t(num_sms()) * 8);
    const uint16_t* xb = static_cast<const uint16_t*>(x);
    uint16_t* yb = static_cast<uint16_t*>(y);
#define QM_EXP_CASE(F, B)                                                                         \
    experts_simple_kernel<F, B><<<static_cast<unsigned>(blocks), 256, 0, st>>>(a, ids, id64, P, topk, T, \
                                                                               xb, x_rows, perm, \
                                                                               offsets, yb)
    if (w.fmt == QM_AFFINE && w.bits == 2) QM_EXP_CASE(QM_AFFINE, 2);
    else if (w.fmt == QM_AFFINE && w.bits == 3) QM_EXP_CASE(QM_AFFINE, 3);
    else if (w.fmt == QM_AFFINE && w.bits == 4) QM_EXP_CASE(QM_AFFINE, 4);
    else if (w.fmt == QM_AFFINE && w.bits == 5) QM_EXP_CASE(QM_AFFINE, 5);
    else if (w.fmt == QM_AFFINE && w.bits == 6) QM_EXP_CASE(QM_AFFINE, 6);
    else if (w.fmt == QM_AFFINE) QM_EXP_CASE(QM_AFFINE, 8);
    else if (w.fmt == QM_Q8_0) QM_EXP_CASE(QM_Q8_0, 8);
    else if (w.fmt == QM_MXFP4_BLOCKS) QM_EXP_CASE(QM_MXFP4_BLOCKS, 4);
    else if (w.fmt == QM_Q4_K) QM_EXP_CASE(QM_Q4_K, 4);
    else if (w.fmt == QM_Q6_K) QM_EXP_CASE(QM_Q6_K, 6);
    else QM_EXP_CASE(QM_MXFP4, 4);
#undef QM_EXP_CASE
    e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "experts launch");
    return QM_OK;
}

}  // namespace qm

// ---------------------------------------------------------------- allocation-free variant
// qm_apply_experts_static: the same work as qm_apply_experts, with its routing
// tables kept in this file-scope device array instead of caller workspace.
// Every GPU that loads the library holds the array until the process exits.
namespace qm {

constexpr size_t kStaticScratchBytes = size_t(1) << 20;  // 1 MiB
static __device__ __align__(256) unsigned char g_experts_scratch[kStaticScratchBytes];

static std::mutex g_scratch_mu;
static void* g_scratch_ptr[64] = {};

// The array's device address on the current device, looked up once per
// device (host code only sees a host-side stand-in for the symbol).
static cudaError_t static_scratch(void** out) {
    std::mutex& mu = g_scratch_mu;
    void** ptr = g_scratch_ptr;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (!ptr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_experts_scratch);
        if (e != cudaSuccess) return e;
        ptr[dev] = p;
    }
    *out = ptr[dev];
    return cudaSuccess;
}

}  // namespace qm

extern "C" qm_status qm_apply_experts_static(const qm_weight* w, const void* ids, int32_t id_type,
                                             int64_t T, int64_t topk, const void* x, int64_t x_rows,
                                             int32_t x_dtype, void* y, qm_stream_t stream) {
    using namespace qm;
    set_error("");
    if (w && w->ndim == 3 && T > 0 && topk > 0 && w->shape[0] >= 0) {
        const qm_status s = check_positions(T, topk, w->shape[0]);
        if (s != QM_OK) return s;
        const size_t need = route_workspace_bytes(T * topk, w->shape[0]);
        if (need > kStaticScratchBytes)
            return fail(QM_EINVAL, "workspace: " + std::to_string(T * topk) + " positions over " +
                                       std::to_string(w->shape[0]) + " experts need " + std::to_string(need) +
                                       " bytes of routing scratch, more than the 1 MiB this entry point "
                                       "holds; use qm_apply_experts with caller workspace");
    }
    void* scratch = nullptr;
    cudaError_t e = static_scratch(&scratch);
    if (e != cudaSuccess) return cuda_fail(e, "static scratch address");
    // Every entry of the routing tables is written before it is read, so the
    // array needs no clearing between calls.
    const qm_status st = apply_experts_checked(w, ids, id_type, T, topk, x, x_rows, x_dtype, y, scratch,
                                               kStaticScratchBytes, stream, /*allow_tensor=*/false);
    if (st == QM_ECUDA) {  // the kept address may be stale (a reset device): look it up anew next time
        int dev = 0;
        if (cudaGetDevice(&dev) == cudaSuccess && dev >= 0 && dev < 64) {
            std::lock_guard<std::mutex> lock(g_scratch_mu);
            g_scratch_ptr[dev] = nullptr;
        }
    }
    return st;
}
