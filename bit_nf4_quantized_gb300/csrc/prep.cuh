// One-launch staging of the per-call operands of the bf16 QLoRA linear (prep.cu).
#pragma once

#include "common.cuh"

namespace qnf4 {

// Every bf16 job writes rows whose length (`width`, or `cols` for kStageRowsDirect) is a
// multiple of 8, eight outputs per thread; kZeroWords clears a multiple of 4 words.
enum PrepKind {
  kStageRows = 0,         // dst[row][c] = bf16(scale * src[row][c]), c < r; zero up to `width`
  kStageRowsDirect = 1,   // dst[j][c] = bf16(src[j][c]) for j < r; zero rows up to `width` rows
  kStageTransposed = 2,   // dst[j][c] = bf16(src[c][j]), j < r, c < cols; rows of `width`
  kStageColumns = 3,      // dst[c][j] = bf16(src[j][c]) (src rows of `cols`), j < r; rows of `width`
  kZeroWords = 4          // fdst[i] = 0 (as 32-bit words)
};

struct PrepJob {
  int kind;
  int r;
  int64_t width;
  float scale;
  const float* src;
  __nv_bfloat16* dst;
  float* fdst;
  int64_t cols;
  int64_t count;          // elements (words for kZeroWords) written
  int first_block;        // set by PrepBuilder
};

constexpr int kMaxPrepJobs = 8;

struct PrepJobs {
  PrepJob job[kMaxPrepJobs];
  int n;
};

class PrepBuilder {
 public:
  PrepBuilder() { jobs_.n = 0; }
  void add(const PrepJob& job);   // at most kMaxPrepJobs; further jobs, or a job whose row
                                  // length breaks the rule above, make launch() fail
  cudaError_t launch(cudaStream_t st);

 private:
  PrepJobs jobs_{};
  int blocks_ = 0;
  bool bad_ = false;
};

}  // namespace qnf4
