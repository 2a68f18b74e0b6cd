// qm_internal.h -- host-side declarations shared by libqm's translation units.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <string>

#include "qm.h"

namespace qm {

// A validated weight: the descriptor flattened to what the kernels read.
struct WDesc {
    int fmt = 0;          // qm_format
    int bits = 0;         // code width (affine 4/8; Q8_0 8; MXFP4 4)
    int gs = 32;          // values per scale group
    int sdt = QM_BF16;    // affine scale/bias dtype
    int ndim = 2;
    int64_t shape[QM_MAX_NDIM] = {0, 0, 0, 0};
    int64_t n = 0, k = 0;
    int64_t rows = 0;     // product of all axes but the last
    const uint8_t* codes = nullptr;
    const uint8_t* scales = nullptr;
    const uint8_t* biases = nullptr;
    int64_t code_row_bytes = 0;   // bytes of one row (k values) of codes
    int64_t scale_row_bytes = 0;  // bytes of one row of scales (0 if none)
    int64_t bias_row_bytes = 0;   // bytes of one row of biases (0 if none)
    bool is_static = false;       // QM_WEIGHT_STATIC: may be read before the previous kernel ends
};

// Thread-local error message of the calling thread (qm_last_error()).
void set_error(const std::string& msg);
qm_status fail(qm_status st, const std::string& msg);
qm_status cuda_fail(cudaError_t e, const char* what);

// Validates w and fills d. On failure sets the message and returns QM_EINVAL.
qm_status validate_weight(const qm_weight* w, WDesc* d);
// Refuses (QM_EINVAL naming "ids" or "w") T*topk positions past 2^31-1 or E
// experts past 2^31-2, before anything multiplies them: routing stores
// positions, offsets and the permutation as int32.
qm_status check_positions(int64_t T, int64_t topk, int64_t E);

int dtype_size(int dt);

// Encodes a 2-d tiled TMA descriptor (CUtensorMap, 128 bytes) over a byte
// array of `rows` rows of `inner_bytes` bytes at `row_stride` bytes apart; a
// box is `box_inner` bytes by `box_rows` rows, 128-byte swizzled if asked,
// out-of-range elements read as zeros. Returns false if the driver refuses.
bool make_tmap_2d(void* map, const void* base, uint64_t inner_bytes, uint64_t rows,
                  uint64_t row_stride, uint32_t box_inner, uint32_t box_rows, bool swizzle128,
                  int elem_bytes = 1);

// Number of SMs on the current device (cached per device).
int num_sms();
// Opt-in shared memory per block on the current device (cached per device).
int max_smem_optin();

// Weights the tensor-map decode GEMV (several tokens) decodes; the others take
// the plain kernels there.
inline bool pipelined_format(const WDesc& w) {
    return (w.fmt == QM_AFFINE && (w.bits == 4 || w.bits == 8)) || w.fmt == QM_Q8_0 || w.fmt == QM_MXFP4 ||
           w.fmt == QM_MXFP4_BLOCKS;
}
// Weights the tensor-core GEMM decodes: affine at every width, Q8_0, MXFP4,
// MXFP4 in GGUF's blocks, Q4_K (Q6_K's 210-byte blocks are no 16-byte
// multiple: no tensor-map tiles).
inline bool gemm_format(const WDesc& w) {
    return w.fmt == QM_AFFINE || w.fmt == QM_Q8_0 || w.fmt == QM_MXFP4 || w.fmt == QM_MXFP4_BLOCKS ||
           w.fmt == QM_Q4_K;
}

// ------------------------------------------------------------ launchers
// Each returns the CUDA error of its launch (cudaSuccess when nothing ran).
cudaError_t launch_dequant(const WDesc& w, int out_dtype, void* out, cudaStream_t st);
// x [rows, k] of x_dtype (QM_F32, QM_BF16, QM_F16) -> Q8_0 blocks [rows, k/32*34].
cudaError_t launch_quantize_q8_0(const void* x, int x_dtype, int64_t rows, int64_t k, uint8_t* blocks,
                                 cudaStream_t st);
// The parts of a packed take: up to three (codes, scales, biases), each a
// source of `len` rows of inner[part] bytes per outer index and a destination.
struct TakeParts {
    int n = 0;
    int one_each = 0;  // every part's row fits one piece per lane of a warp
    const uint8_t* src[3] = {nullptr, nullptr, nullptr};
    uint8_t* dst[3] = {nullptr, nullptr, nullptr};
    int64_t inner[3] = {0, 0, 0};
};
cudaError_t launch_take_packed(const TakeParts& tp, int64_t outer, int64_t len, const void* ids, int id64,
                               int64_t n_ids, cudaStream_t st);
cudaError_t launch_take_dense(const WDesc& w, int axis, const void* ids, int id64, int64_t n_ids,
                              int out_dtype, void* out, cudaStream_t st);

// y [1, n] = x [1, k] * W^T for a 2-d weight (one token), x and y bf16: a
// register-only kernel, no shared memory (qm_gemv1.cu). The _many form runs
// up to 8 weights that read the same x (same format, widths and k) as one
// grid, y_i for weight i.
bool gemv1_supported(const WDesc& w);
cudaError_t launch_gemv1(const WDesc& w, const void* x, void* y, cudaStream_t st);
bool gemv1_many_supported(const WDesc* ws, int count);
cudaError_t launch_gemv1_many(const WDesc* ws, int count, const void* x, void* const* ys, cudaStream_t st);
// y_i [M, n_i] = x [M, k] * W_i^T for up to 8 MLX affine 4-bit weights that
// read the same x, 1 <= M <= 8, k a multiple of 256: weight tiles in registers,
// products on mma.sync (qm_gemvr.cu).
bool gemvr_supported(const WDesc& w, int64_t M);
bool gemvr_many_supported(const WDesc* ws, int count, int64_t M);
cudaError_t launch_gemvr_many(const WDesc* ws, int count, const void* x, int64_t M, void* const* ys,
                              cudaStream_t st);
// y [M, n] = x [M, k] * W^T for a 2-d weight, M <= 16, x and y bf16.
qm_status launch_gemv(const WDesc& w, const void* x, int64_t M, void* y, cudaStream_t st);
bool gemv_supported(const WDesc& w, int64_t M);
// Grouped decode product over a weight [E, n, k]: chunks of routed positions
// (offsets [E+1] and perm from the routing step, on the device), activation
// row of position q is q / xdiv; y [P, n] by position.
qm_status launch_gemv_grouped(const WDesc& w, const int32_t* offsets, const int32_t* perm, int64_t P,
                              int xdiv, const void* x, void* y, cudaStream_t st);
bool gemv_grouped_supported(const WDesc& w, int64_t P);
// Tensor-core product for larger M (tcgen05); returns QM_ENOTSUP if the
// shape is outside what the kernel handles.
qm_status launch_gemm(const WDesc& w, const void* x, int64_t M, void* y, cudaStream_t st);
bool gemm_supported(const WDesc& w, int64_t M);
// Grouped tensor-core product over a weight [E, n, k]: xs holds the routed
// activation rows expert by expert (offsets [E+1]); row i of the result goes
// to row perm[i] of y [P, n].
qm_status launch_gemm_grouped(const WDesc& w, const int32_t* offsets, const int32_t* perm, int64_t P,
                              const void* xs, void* y, cudaStream_t st);
bool gemm_grouped_supported(const WDesc& w, int64_t P);
// Plain reference-order kernel for shapes the fast paths refuse.
cudaError_t launch_apply_simple(const WDesc& w, const void* x, int64_t M, void* y,
                                cudaStream_t st);

// Experts.
size_t route_workspace_bytes(int64_t P, int64_t E);
// allow_tensor: the tensor-core path may be chosen (it needs the routed rows
// of x in the workspace).
size_t experts_workspace_bytes(const WDesc& w, int64_t P, bool allow_tensor);
cudaError_t launch_route(const void* ids, int id64, int64_t P, int64_t E, int32_t* counts,
                         int32_t* offsets, int32_t* perm, void* ws, cudaStream_t st,
                         uint16_t* zero_y = nullptr, int64_t zero_n = 0);
qm_status launch_experts(const WDesc& w, const void* ids, int id64, int64_t T, int64_t topk,
                         const void* x, int64_t x_rows, void* y, void* ws, size_t ws_bytes,
                         cudaStream_t st, bool allow_tensor);
// qm_apply_experts's checks, then launch_experts.
qm_status apply_experts_checked(const qm_weight* w, const void* ids, int32_t id_type, int64_t T,
                                int64_t topk, const void* x, int64_t x_rows, int32_t x_dtype, void* y,
                                void* workspace, size_t workspace_bytes, qm_stream_t stream,
                                bool allow_tensor);

// One warp waiting on a barrier nothing arrives at, giving up after limit_ns.
cudaError_t launch_wait_timeout(uint64_t limit_ns, cudaStream_t st);

// Per-translation-unit device error flags: read-and-clear (after a sync).
uint32_t elementwise_read_clear_error();
uint32_t gemv_read_clear_error();
uint32_t gemm_read_clear_error();
uint32_t experts_read_clear_error();

}  // namespace qm
