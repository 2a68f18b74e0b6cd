// qm_gemm.cu -- tensor-core product for M > 16 (tcgen05, TMEM, TMA).
#include <cuda_runtime.h>

#include "qm_device.cuh"
#include "qm_internal.h"

namespace qm {

static __device__ uint32_t g_err_gemm = 0;

uint32_t gemm_read_clear_error() {
    uint32_t v = 0, z = 0;
    cudaMemcpyFromSymbol(&v, g_err_gemm, sizeof(v));
    cudaMemcpyToSymbol(g_err_gemm, &z, sizeof(z));
    return v;
}

bool gemm_supported(const WDesc&, int64_t) { return false; }

qm_status launch_gemm(const WDesc&, const void*, int64_t, void*, cudaStream_t) {
    return fail(QM_ENOTSUP, "w: tensor-core path not available");
}

}  // namespace qm
