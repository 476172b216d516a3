// QLoRA linear on CUDA cores: the fp32 profile (compute = NF4_F32).  The bf16 profile
// runs on the tensor cores (linear_tc.cu, adapter_tc.cu, stream_fwd.cu).
//
// Math ("Native model adaptation and NF4", sections "One model contract", "Packed
// NF4 and the portable QLoRA profile", "LoRA FA includes gradient preconditioning"):
//   T = x A^T;  y = x W^T + s T B^T;  G = dY B;  dX = dY W + s G A;
//   dA = s G^T x;  dB = s dY^T T.
// The fp32 profile follows the pages' FP32 path: fp32 operands and accumulation,
// the weight decoded inside the shared-memory tile (no global decoded copy), no
// TF32 and no atomics ("V100 accelerated qualification" record,
// jit.kernel_identity: shared-f32 tiles, global-decode-scratch-0, no-atomics).
#include "common.cuh"

namespace qnf4 {
namespace {

// ---- T = x A^T : one warp per (row m, 32 adapter columns) -----------------------------
__global__ void __launch_bounds__(256)
lora_down_kernel(const float* __restrict__ x, const float* __restrict__ A, float* __restrict__ T,
                 int64_t M, int64_t K, int r) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t m = static_cast<int64_t>(blockIdx.x) * 8 + warp;
  if (m >= M) return;
  for (int j = 0; j < r; ++j) {
    float acc = 0.0f;
    for (int64_t k = lane; k < K; k += 32)
      acc = fmaf(x[m * K + k], A[static_cast<int64_t>(j) * K + k], acc);
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (lane == 0) T[m * r + j] = acc;
  }
}

// ---- G = dY B : one warp per row m ------------------------------------------------------
__global__ void __launch_bounds__(256)
lora_g_kernel(const float* __restrict__ dy, const float* __restrict__ B, float* __restrict__ G,
              int64_t M, int64_t N, int r) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t m = static_cast<int64_t>(blockIdx.x) * 8 + warp;
  if (m >= M) return;
  for (int j = 0; j < r; ++j) {
    float acc = 0.0f;
    for (int64_t n = lane; n < N; n += 32)
      acc = fmaf(dy[m * N + n], B[n * r + j], acc);
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (lane == 0) G[m * r + j] = acc;
  }
}

// ---- dA[j][k] = s sum_m G[m][j] x[m][k] : one thread per (j, k), fixed order over m ---------
__global__ void __launch_bounds__(256)
lora_dA_kernel(const float* __restrict__ G, const float* __restrict__ x, float* __restrict__ dA,
               int64_t M, int64_t K, int r, float s) {
  const int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= static_cast<int64_t>(r) * K) return;
  const int j = static_cast<int>(idx / K);
  const int64_t k = idx % K;
  float acc = 0.0f;
  for (int64_t m = 0; m < M; ++m) acc = fmaf(G[m * r + j], x[m * K + k], acc);
  dA[idx] = s * acc;
}

// ---- dB[n][j] = s sum_m dY[m][n] T[m][j] : one thread per (n, j) ------------------------------
__global__ void __launch_bounds__(256)
lora_dB_kernel(const float* __restrict__ dy, const float* __restrict__ T, float* __restrict__ dB,
               int64_t M, int64_t N, int r, float s) {
  const int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= static_cast<int64_t>(r) * N) return;
  const int j = static_cast<int>(idx / N);
  const int64_t n = idx % N;
  float acc = 0.0f;
  for (int64_t m = 0; m < M; ++m) acc = fmaf(dy[m * N + n], T[m * r + j], acc);
  dB[n * r + j] = s * acc;
}

// ---- tiled GEMMs with the weight decoded into shared memory ---------------------------------
// CTA tile 64 x 64 outputs, 256 threads each owning 4 x 4, k-steps of 16.
constexpr int kTile = 64;
constexpr int kKStep = 16;

// Decoded weight element (n, k) of a row-major [N, K] NF4 matrix.
__device__ __forceinline__ float decode_w(const Nf4View& w, int64_t n, int64_t k, int64_t K,
                                          const float* nf4, const float* dyn8, float offset) {
  const int64_t i = n * K + k;
  return __fmul_rn(nf4[nf4_code_at(w.packed, i)], block_scale(w, i >> 6, dyn8, offset));
}

// y[m][n] = sum_k x[m][k] W[n][k] + s sum_j T[m][j] B[n][j]
__global__ void __launch_bounds__(256)
fwd_simt_kernel(const float* __restrict__ x, Nf4View w, const float* __restrict__ T,
                const float* __restrict__ B, float* __restrict__ y, int64_t M, int64_t N, int64_t K,
                int r, float s, DecodeTables tabs) {
  __shared__ float xs[kKStep][kTile + 4];
  __shared__ float ws[kKStep][kTile + 4];
  __shared__ float nf4[16];
  __shared__ float dyn8[256];
  if (threadIdx.x < 16) nf4[threadIdx.x] = tabs.nf4[threadIdx.x];
  dyn8[threadIdx.x] = tabs.dyn8[threadIdx.x];
  const float offset = w.dq ? *w.offset : 0.0f;
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const int64_t m0 = static_cast<int64_t>(blockIdx.y) * kTile;
  const int64_t n0 = static_cast<int64_t>(blockIdx.x) * kTile;
  float acc[4][4] = {};
  __syncthreads();
  for (int64_t k0 = 0; k0 < K; k0 += kKStep) {
    // 64 rows x 16 k of each operand: 1024 elements, 4 per thread
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const int e = threadIdx.x + t * 256;
      const int row = e >> 4, kk = e & 15;
      const int64_t k = k0 + kk;
      const int64_t m = m0 + row, n = n0 + row;
      xs[kk][row] = (m < M && k < K) ? x[m * K + k] : 0.0f;
      ws[kk][row] = (n < N && k < K) ? decode_w(w, n, k, K, nf4, dyn8, offset) : 0.0f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < kKStep; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = xs[kk][ty * 4 + i];
#pragma unroll
      for (int i = 0; i < 4; ++i) b[i] = ws[kk][tx * 4 + i];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) acc[i][jj] = fmaf(a[i], b[jj], acc[i][jj]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int64_t m = m0 + ty * 4 + i;
    if (m >= M) continue;
#pragma unroll
    for (int jj = 0; jj < 4; ++jj) {
      const int64_t n = n0 + tx * 4 + jj;
      if (n >= N) continue;
      float lora = 0.0f;
      for (int j = 0; j < r; ++j) lora = fmaf(s * T[m * r + j], B[n * r + j], lora);
      y[m * N + n] = acc[i][jj] + lora;
    }
  }
}

// dx[m][k] = sum_n dY[m][n] W[n][k] + s sum_j G[m][j] A[j][k]
__global__ void __launch_bounds__(256)
dx_simt_kernel(const float* __restrict__ dy, Nf4View w, const float* __restrict__ G,
               const float* __restrict__ A, float* __restrict__ dx, int64_t M, int64_t N, int64_t K,
               int r, float s, DecodeTables tabs) {
  __shared__ float ds[kKStep][kTile + 4];
  __shared__ float ws[kKStep][kTile + 4];
  __shared__ float nf4[16];
  __shared__ float dyn8[256];
  if (threadIdx.x < 16) nf4[threadIdx.x] = tabs.nf4[threadIdx.x];
  dyn8[threadIdx.x] = tabs.dyn8[threadIdx.x];
  const float offset = w.dq ? *w.offset : 0.0f;
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const int64_t m0 = static_cast<int64_t>(blockIdx.y) * kTile;
  const int64_t k0 = static_cast<int64_t>(blockIdx.x) * kTile;
  float acc[4][4] = {};
  __syncthreads();
  for (int64_t n0 = 0; n0 < N; n0 += kKStep) {
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const int e = threadIdx.x + t * 256;
      // dY tile: 64 m x 16 n (n fastest); W tile: 16 n x 64 k (k fastest)
      const int row = e >> 4, nn = e & 15;
      const int64_t m = m0 + row, n = n0 + nn;
      ds[nn][row] = (m < M && n < N) ? dy[m * N + n] : 0.0f;
      const int wn = e >> 6, wk = e & 63;
      const int64_t n2 = n0 + wn, k = k0 + wk;
      ws[wn][wk] = (n2 < N && k < K) ? decode_w(w, n2, k, K, nf4, dyn8, offset) : 0.0f;
    }
    __syncthreads();
#pragma unroll
    for (int nn = 0; nn < kKStep; ++nn) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = ds[nn][ty * 4 + i];
#pragma unroll
      for (int i = 0; i < 4; ++i) b[i] = ws[nn][tx * 4 + i];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) acc[i][jj] = fmaf(a[i], b[jj], acc[i][jj]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int64_t m = m0 + ty * 4 + i;
    if (m >= M) continue;
#pragma unroll
    for (int jj = 0; jj < 4; ++jj) {
      const int64_t k = k0 + tx * 4 + jj;
      if (k >= K) continue;
      float lora = 0.0f;
      for (int j = 0; j < r; ++j) lora = fmaf(s * G[m * r + j], A[static_cast<int64_t>(j) * K + k], lora);
      dx[m * K + k] = acc[i][jj] + lora;
    }
  }
}

unsigned blocks_for(int64_t n, int per) { return static_cast<unsigned>((n + per - 1) / per); }

}  // namespace

cudaError_t launch_lora_down(const LinearArgs& a, const float* x, const float* A, float* T, cudaStream_t st) {
  KernelTimer timer(NF4_TIME_ADAPTER, st);
  lora_down_kernel<<<blocks_for(a.M, 8), 256, 0, st>>>(x, A, T, a.M, a.K, a.r);
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_lora_g(const LinearArgs& a, const float* dy, const float* B, float* G, cudaStream_t st) {
  KernelTimer timer(NF4_TIME_ADAPTER, st);
  lora_g_kernel<<<blocks_for(a.M, 8), 256, 0, st>>>(dy, B, G, a.M, a.N, a.r);
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_lora_dA(const LinearArgs& a, const float* G, const float* x, float* dA, cudaStream_t st) {
  KernelTimer timer(NF4_TIME_ADAPTER, st);
  lora_dA_kernel<<<blocks_for(static_cast<int64_t>(a.r) * a.K, 256), 256, 0, st>>>(G, x, dA, a.M, a.K, a.r, a.s);
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_lora_dB(const LinearArgs& a, const float* dy, const float* T, float* dB, cudaStream_t st) {
  KernelTimer timer(NF4_TIME_ADAPTER, st);
  lora_dB_kernel<<<blocks_for(static_cast<int64_t>(a.r) * a.N, 256), 256, 0, st>>>(dy, T, dB, a.M, a.N, a.r, a.s);
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_fwd_simt(const LinearArgs& a, const float* x, const float* T, const float* B, float* y,
                            cudaStream_t st) {
  KernelTimer timer(NF4_TIME_FWD_GEMM, st);
  const dim3 grid(blocks_for(a.N, kTile), blocks_for(a.M, kTile));
  if (grid.y > 65535) return cudaErrorInvalidConfiguration;
  fwd_simt_kernel<<<grid, 256, 0, st>>>(x, a.W, T, B, y, a.M, a.N, a.K, a.r, a.s, decode_tables());
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_dx_simt(const LinearArgs& a, const float* dy, const float* G, const float* A, float* dx,
                           cudaStream_t st) {
  KernelTimer timer(NF4_TIME_DX_GEMM, st);
  const dim3 grid(blocks_for(a.K, kTile), blocks_for(a.M, kTile));
  if (grid.y > 65535) return cudaErrorInvalidConfiguration;
  dx_simt_kernel<<<grid, 256, 0, st>>>(dy, a.W, G, A, dx, a.M, a.N, a.K, a.r, a.s, decode_tables());
  note_launch();
  return cudaGetLastError();
}

}  // namespace qnf4
