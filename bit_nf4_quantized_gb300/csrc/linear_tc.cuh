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

}  // namespace qnf4
