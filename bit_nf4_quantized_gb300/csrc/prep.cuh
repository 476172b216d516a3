// Staging of the per-call operands of the 16-bit QLoRA linear (bf16, or IEEE half for the
// FP16 profile): jobs built on the host (PrepBuilder, prep.cu), run by extra CTAs of the
// weight-decode launch (prep_cta).
#pragma once

#include <cuda_fp16.h>

#include "common.cuh"

namespace qnf4 {

// Every 16-bit job writes rows whose length (`width`, or `cols` for kStageRowsDirect) is a
// multiple of 8, eight outputs per thread; kZeroWords clears a multiple of 4 words.
// T16 below is the call's 16-bit type (PrepJobs::f16 selects IEEE half over bf16).
enum PrepKind {
  kStageRows = 0,         // dst[row][c] = T16(scale * src[row][c]), c < r; zero up to `width`
  kStageRowsDirect = 1,   // dst[j][c] = T16(src[j][c]) for j < r; zero rows up to `width` rows
  kStageTransposed = 2,   // dst[j][c] = T16(src[c][j]), j < r, c < cols; rows of `width`
  kStageColumns = 3,      // dst[c][j] = T16(src[j][c]) (src rows of `cols`), j < r; rows of `width`
  kZeroWords = 4          // fdst[i] = 0 (as 32-bit words)
};

struct PrepJob {
  int kind;
  int r;
  int64_t width;
  float scale;
  const float* src;
  void* dst;              // 16-bit elements
  float* fdst;
  int64_t cols;
  int64_t count;          // elements (words for kZeroWords) written
  int first_block;        // set by PrepBuilder
};

constexpr int kMaxPrepJobs = 32;
constexpr int kPrepThreads = 256;   // threads of a prep CTA (the decode launch's CTA width)
constexpr int kPrepPer = 8;         // outputs per thread: one 16-byte store

struct PrepJobs {
  PrepJob job[kMaxPrepJobs];
  int n;
  int f16;                // 16-bit outputs are IEEE half (else bf16)
};

namespace prep_detail {

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

__device__ __forceinline__ uint4 pack8(const float (&v)[kPrepPer], int f16) {
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    if (f16) {
      const __half2 h = __floats2half2_rn(v[2 * i], v[2 * i + 1]);
      w[i] = *reinterpret_cast<const uint32_t*>(&h);
    } else {
      const __nv_bfloat162 b = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
      w[i] = *reinterpret_cast<const uint32_t*>(&b);
    }
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

}  // namespace prep_detail

// Prep CTA number `cta` of a launch over `p` (kPrepThreads threads).
__device__ __forceinline__ void prep_cta(const PrepJobs& p, unsigned cta) {
  using prep_detail::pack8;
  using prep_detail::split_index;
  pdl_allow_next();
  pdl_wait();
  int j = 0;
  while (j + 1 < p.n && cta >= static_cast<unsigned>(p.job[j + 1].first_block)) ++j;
  const PrepJob& jb = p.job[j];
  const uint64_t t = static_cast<uint64_t>(cta - jb.first_block) * kPrepThreads + threadIdx.x;
  if (jb.kind == kZeroWords) {
    if (4 * t < static_cast<uint64_t>(jb.count)) reinterpret_cast<uint4*>(jb.fdst)[t] = make_uint4(0u, 0u, 0u, 0u);
    return;
  }
  const uint64_t idx = kPrepPer * t;   // first of the thread's 8 outputs (one row)
  if (idx >= static_cast<uint64_t>(jb.count)) return;
  const uint64_t r = static_cast<uint64_t>(jb.r);
  float v[kPrepPer];
  uint64_t a, b;
  switch (jb.kind) {
    case kStageRows: {         // dst[row][c] = T16(scale * src[row][c]) for c < r, 0 up to width
      split_index(idx, jb.width, &a, &b);
#pragma unroll
      for (int i = 0; i < kPrepPer; ++i) v[i] = (b + i < r) ? jb.scale * jb.src[a * r + b + i] : 0.0f;
      break;
    }
    case kStageRowsDirect: {   // dst[j][c] = T16(src[j][c]) for j < r, 0 for j in [r, width rows)
      split_index(idx, jb.cols, &a, &b);
#pragma unroll
      for (int i = 0; i < kPrepPer; ++i) v[i] = (a < r) ? jb.src[idx + i] : 0.0f;
      break;
    }
    case kStageTransposed: {   // dst[j][c] = T16(src[c][j]) for j < r, c < cols; row length width
      split_index(idx, jb.width, &a, &b);
      const uint64_t cols = static_cast<uint64_t>(jb.cols);
#pragma unroll
      for (int i = 0; i < kPrepPer; ++i) v[i] = (a < r && b + i < cols) ? jb.src[(b + i) * r + a] : 0.0f;
      break;
    }
    case kStageColumns: {      // dst[c][j] = T16(src[j][c]) for j < r; rows of width entries
      split_index(idx, jb.width, &a, &b);
      const uint64_t cols = static_cast<uint64_t>(jb.cols);
#pragma unroll
      for (int i = 0; i < kPrepPer; ++i) v[i] = (b + i < r) ? jb.src[(b + i) * cols + a] : 0.0f;
      break;
    }
    default:
      return;
  }
  *reinterpret_cast<uint4*>(static_cast<uint16_t*>(jb.dst) + idx) = pack8(v, p.f16);
}

class PrepBuilder {
 public:
  explicit PrepBuilder(bool f16 = false) {
    jobs_.n = 0;
    jobs_.f16 = f16 ? 1 : 0;
  }
  void add(const PrepJob& job);   // at most kMaxPrepJobs; further jobs, or a job whose row
                                  // length breaks the rule above, make ok() false
  bool ok() const { return !bad_; }
  const PrepJobs& jobs() const { return jobs_; }
  unsigned ctas() const { return static_cast<unsigned>(blocks_); }

 private:
  PrepJobs jobs_{};
  int blocks_ = 0;
  bool bad_ = false;
};

}  // namespace qnf4
