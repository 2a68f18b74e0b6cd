// qm_gemm_grouped.cu -- the grouped products' 128-token tiles (classic
// layout), instantiated here so that they compile beside qm_gemm.cu.
#include "qm_gemm_kernel.cuh"

namespace qm {
namespace gemm {

uint32_t grouped_read_clear_flag() { return read_clear_flag(); }

namespace {
struct NarrowGrouped {
    Params& p;
    const WDesc& w;
    const void* x;
    cudaStream_t st;
    template <int FMT, int BITS, int GS>
    cudaError_t run() const {
        return launch_t<FMT, BITS, GS, 128, false>(p, w, x, st);
    }
};
}  // namespace

cudaError_t dispatch_grouped_narrow(Params& p, const WDesc& w, const void* x, cudaStream_t st) {
    return by_format(p, w, NarrowGrouped{p, w, x, st});
}

}  // namespace gemm
}  // namespace qm
