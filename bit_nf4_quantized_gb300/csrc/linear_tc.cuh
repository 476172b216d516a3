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

// adapter_tc.cu: the rank-r contractions on tcgen05 (workspace sizes and sequences).
size_t adapter_fwd_ws_bytes(int64_t M, int64_t N, int64_t K, int r);
size_t adapter_bwd_ws_bytes(int64_t M, int64_t N, int64_t K, int r);
// T = x A^T (fp32) and sTp = bf16(s T) zero-padded to a multiple of 64 columns.
cudaError_t adapter_forward(const LinearArgs& a, const void* x, const float* A, float* T, __nv_bfloat16* sTp,
                            void* ws, int* status, cudaStream_t st);
// G = dY B (fp32), sGp = bf16(s G) padded, dB = s dY^T T; keeps bf16(G)^T in ws for the dA pass.
cudaError_t adapter_backward_pre(const LinearArgs& a, const void* dy, const float* T, const float* B, float* G,
                                 __nv_bfloat16* sGp, float* dB, void* ws, int* status, cudaStream_t st);
// dA = s G^T x, using the bf16(G)^T that adapter_backward_pre left in ws.
cudaError_t adapter_backward_post(const LinearArgs& a, const void* x, float* dA, void* ws, int* status,
                                  cudaStream_t st);

}  // namespace qnf4
