// Per-call operand staging for the bf16 QLoRA linear, in one launch: the bf16 copies of
// the adapter factors in the layouts the tensor-core kernels read, and the fp32 block
// scales a' of the weight ("Native model adaptation and NF4", "Fused GPU NF4 decodes
// inside the matrix kernel": a' = dyn8[code] * nested + offset, two roundings).
#include "prep.cuh"

namespace qnf4 {
namespace {

constexpr int kPrepThreads = 256;

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

constexpr int kScaleTile = 32;   // block-scale transpose tile: 32 blocks x 32 weight rows

// a' of block `blk` (two roundings, as the dequantize kernel computes it)
__device__ __forceinline__ float block_scale(const PrepJobs& p, const float* dyn8, uint64_t blk) {
  if (!p.w.dq) return static_cast<const float*>(p.w.absmax)[blk];
  const uint32_t code = static_cast<const uint8_t*>(p.w.absmax)[blk];
  return __fadd_rn(__fmul_rn(dyn8[code], p.w.nested[blk >> 8]), *p.w.offset);
}

__global__ void __launch_bounds__(kPrepThreads) prep_kernel(PrepJobs p) {
  __shared__ float dyn8[256];
  __shared__ float tile[kScaleTile][kScaleTile + 1];
  dyn8[threadIdx.x] = p.dyn8[threadIdx.x];
  __syncthreads();
  pdl_allow_next();
  pdl_wait();
  int j = 0;
  while (j + 1 < p.n && blockIdx.x >= p.job[j + 1].first_block) ++j;
  const PrepJob& jb = p.job[j];
  if (jb.kind == kBlockScales) {
    // fdst[kb][n] = a'(n, kb) for n < N, 0 for n in [N, width): one 32 x 32 tile per CTA,
    // read along kb (the codes' order) and written along n, both coalesced
    const int64_t tiles_n = (jb.width + kScaleTile - 1) / kScaleTile;
    const int64_t t = blockIdx.x - jb.first_block;
    const int64_t n0 = (t % tiles_n) * kScaleTile, kb0 = (t / tiles_n) * kScaleTile;
    for (int e = threadIdx.x; e < kScaleTile * kScaleTile; e += kPrepThreads) {
      const int nl = e / kScaleTile, kl = e % kScaleTile;
      const int64_t n = n0 + nl, kb = kb0 + kl;
      tile[kl][nl] = (n < jb.cols && kb < p.kbn) ? block_scale(p, dyn8, static_cast<uint64_t>(n * p.kbn + kb)) : 0.0f;
    }
    __syncthreads();
    for (int e = threadIdx.x; e < kScaleTile * kScaleTile; e += kPrepThreads) {
      const int kl = e / kScaleTile, nl = e % kScaleTile;
      const int64_t n = n0 + nl, kb = kb0 + kl;
      if (n < jb.width && kb < p.kbn) jb.fdst[kb * jb.width + n] = tile[kl][nl];
    }
    return;
  }
  const uint64_t idx = static_cast<uint64_t>(blockIdx.x - jb.first_block) * kPrepThreads + threadIdx.x;
  if (idx >= static_cast<uint64_t>(jb.count)) return;
  uint64_t a, b;
  switch (jb.kind) {
    case kStageRows: {         // dst[row][c] = bf16(scale * src[row][c]) for c < r, 0 up to width
      split_index(idx, jb.width, &a, &b);
      jb.dst[idx] = __float2bfloat16_rn(b < static_cast<uint64_t>(jb.r) ? jb.scale * jb.src[a * jb.r + b] : 0.0f);
      break;
    }
    case kStageRowsDirect: {   // dst[j][c] = bf16(src[j][c]) for j < r, 0 for j in [r, width rows)
      split_index(idx, jb.cols, &a, &b);
      jb.dst[idx] = __float2bfloat16_rn(a < static_cast<uint64_t>(jb.r) ? jb.src[idx] : 0.0f);
      break;
    }
    case kStageTransposed: {   // dst[j][c] = bf16(src[c][j]) for j < r, c < cols; row length width
      split_index(idx, jb.width, &a, &b);
      const bool in = a < static_cast<uint64_t>(jb.r) && b < static_cast<uint64_t>(jb.cols);
      jb.dst[idx] = __float2bfloat16_rn(in ? jb.src[b * jb.r + a] : 0.0f);
      break;
    }
    case kStageColumns: {      // dst[c][j] = bf16(src[j][c]) for j < r; rows of width entries
      split_index(idx, jb.width, &a, &b);
      jb.dst[idx] = __float2bfloat16_rn(b < static_cast<uint64_t>(jb.r) ? jb.src[b * jb.cols + a] : 0.0f);
      break;
    }
    case kZeroWords:
      jb.fdst[idx] = 0.0f;
      break;
    default:
      break;
  }
}

}  // namespace

void PrepBuilder::add(const PrepJob& job) {
  if (jobs_.n == kMaxPrepJobs) {
    overflow_ = true;
    return;
  }
  PrepJob j = job;
  j.first_block = blocks_;
  if (j.kind == kBlockScales)   // one CTA per 32 x 32 tile
    blocks_ += static_cast<int>(((j.width + kScaleTile - 1) / kScaleTile) *
                                ((jobs_.kbn + kScaleTile - 1) / kScaleTile));
  else
    blocks_ += static_cast<int>((j.count + kPrepThreads - 1) / kPrepThreads);
  jobs_.job[jobs_.n++] = j;
}

cudaError_t PrepBuilder::launch(cudaStream_t st) {
  if (overflow_) return cudaErrorInvalidValue;
  if (jobs_.n == 0) return cudaSuccess;
  const DecodeTables& t = decode_tables();
  for (int i = 0; i < 256; ++i) jobs_.dyn8[i] = t.dyn8[i];
  KernelTimer timer(NF4_TIME_ADAPTER, st);
  const cudaError_t e = launch_pdl(prep_kernel, dim3(blocks_), dim3(kPrepThreads), 0, st, 1, jobs_);
  note_launch();
  return e;
}

}  // namespace qnf4
