// qm_gemm.cu -- prefill product y[M, n] = x[M, k] * W^T for M >= 17 on the
// 5th-generation tensor cores: tile plans and the entry points. The kernel
// and its pipeline are in qm_gemm_kernel.cuh.
#include "qm_gemm_kernel.cuh"

namespace qm {

uint32_t gemm_read_clear_error() { return gemm::read_clear_flag() | gemm::grouped_read_clear_flag(); }

namespace gemm {

// Plain products: 256-token tiles (classic layout) above 128 tokens, else one
// 128-token tile row with the dual layout. Grouped products: 256-token tiles
// once experts average over 256 positions; below that, 128-token tiles in the
// classic layout, two CTAs to an SM (measured faster than the dual layout
// there, where many tiles queue: T = 1024 x top-4 over 32 experts 492 against
// 347 TFLOP/s; and faster than 256-token tiles even where an expert spills a
// second, nearly empty tile: 376 -> 392).
struct Launch {
    Params& p;
    const WDesc& w;
    const void* x;
    cudaStream_t st;
    bool wide;
    template <int FMT, int BITS, int GS>
    cudaError_t run() const {
        return wide ? launch_t<FMT, BITS, GS, 256, false>(p, w, x, st) : launch_t<FMT, BITS, GS, 128, true>(p, w, x, st);
    }
};

static cudaError_t dispatch(Params& p, const WDesc& w, const void* x, cudaStream_t st) {
    const bool wide = p.g_off ? p.M > 256 * std::max<int64_t>(1, p.g_E) : p.M > 128;
    if (p.g_off && !wide) return dispatch_grouped_narrow(p, w, x, st);
    return by_format(p, w, Launch{p, w, x, st, wide});
}

}  // namespace gemm

bool gemm_supported(const WDesc& w, int64_t M) {
    if (M < 1 || w.ndim != 2 || w.n < 1 || w.k < 64 || !gemm_format(w)) return false;
    if (w.code_row_bytes % 16) return false;  // TMA row stride
    if (M > (int64_t(1) << 31) || w.n > (int64_t(1) << 31)) return false;
    return true;
}

qm_status launch_gemm(const WDesc& w, const void* x, int64_t M, void* y, cudaStream_t st) {
    using namespace gemm;
    Params p{};
    p.scales = w.scales;
    p.biases = w.biases;
    p.y = static_cast<uint16_t*>(y);
    p.M = M;
    p.n = w.n;
    p.k = w.k;
    p.scale_row_bytes = w.scale_row_bytes;
    p.sdt = w.sdt;
    p.ksteps = static_cast<int>((w.k + BK - 1) / BK);
    cudaError_t e = dispatch(p, w, x, st);
    if (e == cudaErrorNotSupported) {  // no TMA descriptor for these operands: the plain kernel
        e = launch_apply_simple(w, x, M, y, st);
        return e == cudaSuccess ? QM_OK : cuda_fail(e, "apply launch");
    }
    if (e != cudaSuccess) return cuda_fail(e, "gemm launch");
    return QM_OK;
}

bool gemm_grouped_supported(const WDesc& w, int64_t P) {
    if (w.ndim != 3 || w.shape[0] < 1 || w.n < 1 || w.k < 64 || P < 1 || !gemm_format(w)) return false;
    if (w.code_row_bytes % 16 || (w.k * 2) % 16) return false;  // TMA row strides
    if (P >= (int64_t(1) << 31) || w.rows >= (int64_t(1) << 31)) return false;
    return true;
}

qm_status launch_gemm_grouped(const WDesc& w, const int32_t* offsets, const int32_t* perm, int64_t P,
                              const void* xs, void* y, cudaStream_t st) {
    using namespace gemm;
    if (!gemm_grouped_supported(w, P)) return fail(QM_ENOTSUP, "w: no grouped tensor-core plan for this shape");
    Params p{};
    p.scales = w.scales;
    p.biases = w.biases;
    p.y = static_cast<uint16_t*>(y);
    p.M = P;
    p.n = w.n;
    p.k = w.k;
    p.scale_row_bytes = w.scale_row_bytes;
    p.sdt = w.sdt;
    p.ksteps = static_cast<int>((w.k + BK - 1) / BK);
    p.g_off = offsets;
    p.g_perm = perm;
    p.g_E = w.shape[0];
    const cudaError_t e = dispatch(p, w, xs, st);
    if (e == cudaErrorNotSupported) return fail(QM_ENOTSUP, "w: no tensor map for the grouped product");
    if (e != cudaSuccess) return cuda_fail(e, "grouped gemm launch");
    return QM_OK;
}

}  // namespace qm
