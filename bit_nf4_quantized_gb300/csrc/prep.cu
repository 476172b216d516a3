// Per-call operand staging for the bf16 QLoRA linear: the job list whose CTAs run in the
// launch that decodes the call's weight (prep_cta in prep.cuh): the bf16 copies of the
// adapter factors in the layouts the tensor-core kernels read (rank side padded with
// zeros), and the zeroed flags of the kernels that follow.
#include "prep.cuh"

namespace qnf4 {

void PrepBuilder::add(const PrepJob& job) {
  if (jobs_.n == kMaxPrepJobs) {
    bad_ = true;
    return;
  }
  PrepJob j = job;
  const int64_t row = (j.kind == kStageRowsDirect) ? j.cols : j.width;
  if (j.kind == kZeroWords ? (j.count % 4 != 0) : (row % kPrepPer != 0 || j.count % kPrepPer != 0)) {
    bad_ = true;
    return;
  }
  j.first_block = blocks_;
  const int64_t per_thread = (j.kind == kZeroWords) ? 4 : kPrepPer;
  blocks_ += static_cast<int>((j.count / per_thread + kPrepThreads - 1) / kPrepThreads);
  jobs_.job[jobs_.n++] = j;
}

}  // namespace qnf4
