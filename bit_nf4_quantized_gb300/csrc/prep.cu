// Per-call operand staging for the bf16 QLoRA linear, in one launch: the bf16 copies of
// the adapter factors in the layouts the tensor-core kernels read (rank side padded with
// zeros), and the zeroed flags and counters of the kernels that follow.
#include "prep.cuh"

namespace qnf4 {
namespace {

constexpr int kPrepThreads = 256;
constexpr int kPer = 8;           // outputs per thread: one 16-byte store

__device__ __forceinline__ void split_index(uint64_t idx, uint64_t width, uint64_t* hi, uint64_t* lo) {
  if (idx < (1ull << 32) && width < (1ull << 32)) {
    const uint32_t q = static_cast<uint32_t>(idx) / static_cast<uint32_t>(width);
    *hi = q;
    *lo = static_cast<uint32_t>(idx) - q * static_cast<uint32_t>(width);
  } else {
    *hi = idx / width;
    *lo = idx % width;
  }
}

__device__ __forceinline__ uint4 pack8(const float (&v)[kPer]) {
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t lo = __bfloat16_as_ushort(__float2bfloat16_rn(v[2 * i]));
    const uint32_t hi = __bfloat16_as_ushort(__float2bfloat16_rn(v[2 * i + 1]));
    w[i] = lo | (hi << 16);
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

__global__ void __launch_bounds__(kPrepThreads) prep_kernel(PrepJobs p) {
  pdl_allow_next();
  pdl_wait();
  int j = 0;
  while (j + 1 < p.n && blockIdx.x >= p.job[j + 1].first_block) ++j;
  const PrepJob& jb = p.job[j];
  const uint64_t t = static_cast<uint64_t>(blockIdx.x - jb.first_block) * kPrepThreads + threadIdx.x;
  if (jb.kind == kZeroWords) {
    if (4 * t < static_cast<uint64_t>(jb.count)) reinterpret_cast<uint4*>(jb.fdst)[t] = make_uint4(0u, 0u, 0u, 0u);
    return;
  }
  const uint64_t idx = kPer * t;   // first of the thread's 8 outputs (one row)
  if (idx >= static_cast<uint64_t>(jb.count)) return;
  const uint64_t r = static_cast<uint64_t>(jb.r);
  float v[kPer];
  uint64_t a, b;
  switch (jb.kind) {
    case kStageRows: {         // dst[row][c] = bf16(scale * src[row][c]) for c < r, 0 up to width
      split_index(idx, jb.width, &a, &b);
#pragma unroll
      for (int i = 0; i < kPer; ++i) v[i] = (b + i < r) ? jb.scale * jb.src[a * r + b + i] : 0.0f;
      break;
    }
    case kStageRowsDirect: {   // dst[j][c] = bf16(src[j][c]) for j < r, 0 for j in [r, width rows)
      split_index(idx, jb.cols, &a, &b);
#pragma unroll
      for (int i = 0; i < kPer; ++i) v[i] = (a < r) ? jb.src[idx + i] : 0.0f;
      break;
    }
    case kStageTransposed: {   // dst[j][c] = bf16(src[c][j]) for j < r, c < cols; row length width
      split_index(idx, jb.width, &a, &b);
      const uint64_t cols = static_cast<uint64_t>(jb.cols);
#pragma unroll
      for (int i = 0; i < kPer; ++i) v[i] = (a < r && b + i < cols) ? jb.src[(b + i) * r + a] : 0.0f;
      break;
    }
    case kStageColumns: {      // dst[c][j] = bf16(src[j][c]) for j < r; rows of width entries
      split_index(idx, jb.width, &a, &b);
      const uint64_t cols = static_cast<uint64_t>(jb.cols);
#pragma unroll
      for (int i = 0; i < kPer; ++i) v[i] = (b + i < r) ? jb.src[(b + i) * cols + a] : 0.0f;
      break;
    }
    default:
      return;
  }
  *reinterpret_cast<uint4*>(jb.dst + idx) = pack8(v);
}

}  // namespace

void PrepBuilder::add(const PrepJob& job) {
  if (jobs_.n == kMaxPrepJobs) {
    bad_ = true;
    return;
  }
  PrepJob j = job;
  const int64_t row = (j.kind == kStageRowsDirect) ? j.cols : j.width;
  if (j.kind == kZeroWords ? (j.count % 4 != 0) : (row % kPer != 0 || j.count % kPer != 0)) {
    bad_ = true;
    return;
  }
  j.first_block = blocks_;
  const int64_t per_thread = (j.kind == kZeroWords) ? 4 : kPer;
  blocks_ += static_cast<int>((j.count / per_thread + kPrepThreads - 1) / kPrepThreads);
  jobs_.job[jobs_.n++] = j;
}

cudaError_t PrepBuilder::launch(cudaStream_t st) {
  if (bad_) return cudaErrorInvalidValue;
  if (jobs_.n == 0 || blocks_ == 0) return cudaSuccess;
  KernelTimer timer(NF4_TIME_ADAPTER, st);
  const cudaError_t e = launch_pdl(prep_kernel, dim3(blocks_), dim3(kPrepThreads), 0, st, 1, jobs_);
  note_launch();
  return e;
}

}  // namespace qnf4
