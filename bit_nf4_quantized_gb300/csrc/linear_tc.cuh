// bf16 profile of the QLoRA linear: workspace sizes and the forward / backward
// sequences (tensor-core kernels for the base contraction).
#pragma once

#include "common.cuh"

namespace qnf4 {

size_t tc_fwd_ws_bytes(int64_t M, int64_t N, int64_t K, int r);
size_t tc_bwd_ws_bytes(int64_t M, int64_t N, int64_t K, int r);

cudaError_t tc_forward(const LinearArgs& a, const void* x, const float* A, const float* B, void* y,
                       float* T, void* ws, int* status, cudaStream_t st);
cudaError_t tc_backward(const LinearArgs& a, const void* dy, const void* x, const float* T,
                        const float* A, const float* B, void* dx, float* dA, float* dB, float* G,
                        void* ws, int* status, cudaStream_t st);

// adapter_tc.cu: skinny tcgen05 products Out[rows, r] = X[rows, red] . Q[red, r] for the
// rank-r contractions.  X is bf16 row-major with `x_inner` columns (the reduction runs
// along its rows when mn_major == false, down its columns otherwise); Q is bf16
// [nq][q_cols] (nq = r rounded up to 16).  Reduction slices write partial sums that
// adapter_finish adds in a fixed order.
int adapter_nq(int r);
size_t adapter_partial_bytes(int64_t rows, int64_t red, int r);
cudaError_t adapter_pass(const void* X, int64_t x_inner, int64_t x_outer, bool mn_major, const __nv_bfloat16* Q,
                         int64_t q_cols, int r, int64_t rows, int64_t red, float* partial, int* status, int* nsplit,
                         cudaStream_t st);
// Sum of the slices times `scale` into f32 ([rows][r], or [r][rows] when f32_t), and
// optionally bf16(scale_b * sum) into b_rows [rows][rp] and bf16(sum) into b_t [nq][ldt].
cudaError_t adapter_finish(const float* partial, int nsplit, int64_t rows, int r, float scale, float* f32, int f32_t,
                           __nv_bfloat16* b_rows, int rp, float scale_b, __nv_bfloat16* b_t, int64_t ldt,
                           cudaStream_t st);

}  // namespace qnf4
