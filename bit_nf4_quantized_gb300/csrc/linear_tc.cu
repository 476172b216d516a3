// bf16 profile of the QLoRA linear.
#include "linear_tc.cuh"

namespace qnf4 {

size_t tc_fwd_ws_bytes(int64_t, int64_t, int64_t, int) { return 0; }
size_t tc_bwd_ws_bytes(int64_t, int64_t, int64_t, int) { return 0; }

cudaError_t tc_forward(const LinearArgs& a, const void* x, const float* A, const float* B, void* y,
                       float* T, void*, int*, cudaStream_t st) {
  cudaError_t e = launch_lora_down(a, NF4_BF16, x, A, T, st);
  if (e == cudaSuccess) e = launch_fwd_simt(a, NF4_BF16, x, T, B, y, st);
  return e;
}

cudaError_t tc_backward(const LinearArgs& a, const void* dy, const void* x, const float* T,
                        const float* A, const float* B, void* dx, float* dA, float* dB, float* G,
                        void*, int*, cudaStream_t st) {
  cudaError_t e = launch_lora_g(a, NF4_BF16, dy, B, G, st);
  if (e == cudaSuccess) e = launch_dx_simt(a, NF4_BF16, dy, G, A, dx, st);
  if (e == cudaSuccess) e = launch_lora_dA(a, NF4_BF16, G, x, dA, st);
  if (e == cudaSuccess) e = launch_lora_dB(a, NF4_BF16, dy, T, dB, st);
  return e;
}

}  // namespace qnf4
