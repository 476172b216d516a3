// bf16 profile of the QLoRA linear: workspace sizes and the forward / backward
// sequences (tensor-core kernels for the base contraction).
#pragma once

#include "common.cuh"

namespace qnf4 {

// w16: the weight comes decoded (no room for a per-call decoded copy in the workspace).
size_t tc_fwd_ws_bytes(int64_t M, int64_t N, int64_t K, int r, bool w16 = false);
size_t tc_bwd_ws_bytes(int64_t M, int64_t N, int64_t K, int r, bool w16 = false);

// f16: the operands and outputs are IEEE half (the FP16 profile) instead of bf16.  w16, when
// given, is W already decoded to the 16-bit type ([N][K], as nf4_dequantize writes it): the
// call then runs its operand staging alone instead of decoding a.W first.
cudaError_t tc_forward(const LinearArgs& a, bool f16, const void* x, const float* A, const float* B, void* y,
                       float* T, void* ws, int* status, cudaStream_t st, const void* w16 = nullptr);
cudaError_t tc_backward(const LinearArgs& a, bool f16, const void* dy, const void* x, const float* T,
                        const float* A, const float* B, void* dx, float* dA, float* dB, float* G,
                        void* ws, int* status, cudaStream_t st, const void* w16 = nullptr);

// Runs of up to kTcGroupMax projections that share M (the tiled path of the batch calls).
// Consecutive items that read the same input x [M][K] (the same pointer and K; e.g. a
// layer's q, k and v, or gate and up) form an input set whose ranks, each rounded up to 16,
// add up to at most kTcGroupMaxRank: one skinny pass over x computes T for every item of a
// set (forward) and one computes dA (backward), with Q stacking the items' rank sides.  All
// sets' passes go in one launch, and so do all items' G and dB passes.  Each G/dB pair is
// split as the single call splits it (dX and dB are the single call's bits); the T or dA
// passes of a launch share the resident CTAs in proportion to the bytes each reads, so with
// one input set they are the single call's bits and with several their fp32 partial sums
// are added in another order (deterministic for a given run).  w16: the
// item's weight decoded to 16 bits, or nullptr (a.W is decoded, all such items of the run in
// one batched launch).  The run's workspace holds each item's single-call workspace
// (w16-aware) and each set's shared buffers.
constexpr int kTcGroupMax = 8;
constexpr int kTcGroupMaxRank = 256;
struct TcFwdItem {
  LinearArgs a;
  const void* x;
  const float* A;
  const float* B;
  void* y;
  float* T;
  const void* w16;
};
struct TcBwdItem {
  LinearArgs a;
  const void* x;
  const void* dy;
  const float* T;
  const float* A;
  const float* B;
  void* dx;
  float* dA;
  float* dB;
  const void* w16;
};
size_t tc_fwd_run_ws_bytes(const TcFwdItem* it, int n);
size_t tc_bwd_run_ws_bytes(const TcBwdItem* it, int n);
cudaError_t tc_forward_run(const TcFwdItem* it, int n, bool f16, void* ws, int* status, cudaStream_t st);
cudaError_t tc_backward_run(const TcBwdItem* it, int n, bool f16, void* ws, int* status, cudaStream_t st);

// stream_fwd.cu: the forward for at most kStreamMaxM tokens, for up to kStreamMaxGroup
// projections (sharing M) in two launches: T by lora_down_small, then one persistent pass that
// streams every projection's stored weight once, decodes it in registers straight into
// mma.sync fragments with the tokens as the 16-row operand, the LoRA term in the same
// accumulators.
constexpr int kStreamMaxM = 16;
constexpr int kStreamMaxGroup = 8;
struct StreamItem {
  LinearArgs a;
  const void* x;     // 16-bit [M, K]
  const float* A;    // [r, K]
  const float* B;    // [N, r]
  void* y;           // 16-bit [M, N]
  float* T;          // [M, r]
};
size_t stream_fwd_ws_bytes(const LinearArgs* a, int n);
// f16: x, y and every tensor-core operand are IEEE half (the FP16 profile) instead of bf16.
cudaError_t stream_forward(const StreamItem* items, int n, bool f16, void* ws, int* status, cudaStream_t st);

// small_fused.cu: the 16-bit profiles for small weights (K, N <= 1024, N*K <= 2^21, rank <= 32)
// and M > 16: the forward of up to kSmallMaxGroup projections sharing M in one launch, and
// their backward in one (the dX tiles with the adapter gradients' per-tile parts, whose ordered
// sums the last CTA of each column tile takes).
constexpr int kSmallMaxGroup = 8;
struct SmallItem {
  LinearArgs a;
  const void* x;     // 16-bit [M, K]
  const float* A;    // [r, K]
  const float* B;    // [N, r]
  void* y;           // forward: 16-bit [M, N]
  float* T;          // forward: written; backward: read [M, r]
  const void* dy;    // backward: 16-bit [M, N]
  const void* w16;   // W decoded to 16 bits [N, K], or null (decoded in the kernels)
  void* dx;          // backward: 16-bit [M, K]
  float* dA;         // backward: [r, K]
  float* dB;         // backward: [N, r]
};
bool small_fused_fits(int64_t N, int64_t K, int r);
cudaError_t small_fused_forward(const SmallItem* items, int n, int64_t M, bool f16, cudaStream_t st);
size_t small_fused_bwd_ws_bytes(const SmallItem* items, int n, int64_t M);
cudaError_t small_fused_backward(const SmallItem* items, int n, int64_t M, bool f16, void* ws, cudaStream_t st);

// adapter_tc.cu: skinny tcgen05 products Out[rows, r] = X[rows, red] . Q[red, r] for the
// rank-r contractions.  X is 16-bit (T16: bf16, or IEEE half when f16) row-major with
// `x_inner` columns (the reduction runs along its rows when mn_major == false, down its
// columns otherwise); Q is T16 [nq][q_cols] (nq = r rounded up to 16).  Reduction slices
// write partial sums to `partial` (adapter_partial_bytes) that a second launch adds in a
// fixed order, writing:
//   f32 = scale * sum as [rows][r] (or [r][rows] when f32_t), if f32 is set;
//   T16(scale_b * sum) as [rows][rp], zero past r, if b_rows is set;
//   T16(sum) as [r][ldt] (rows r.. of a [nq][ldt] buffer untouched), if b_t is set.
// A pass may instead serve several consumers that share X (the projections of a layer that
// read the same input): Q stacks their rank sides, and `outs` lists, for each consumer, its
// columns [col0, col0 + r) of the sums with its own outputs as above.
struct AdapterOut {
  int col0, r;
  float scale;
  float* f32;
  int f32_t;
  void* b_rows;
  int rp;
  float scale_b;
  void* b_t;
  int64_t ldt;
};
constexpr int kAdapterMaxOuts = 16;
constexpr int kAdapterMaxPasses = 16;
struct AdapterPassArgs {
  const void* X;
  int64_t x_inner, x_outer;
  bool mn_major;
  const void* Q;
  int64_t q_cols;
  int r;
  int64_t rows, red;
  float* partial;
  float scale;
  float* f32;
  int f32_t;
  void* b_rows;
  int rp;
  float scale_b;
  void* b_t;
  int64_t ldt;
  int f16;
  const AdapterOut* outs;   // nouts consumers (at most kAdapterMaxOuts in a launch); 0: the fields above
  int nouts;
  int target;               // CTAs the reduction split is planned for; 0: see adapter_run
};
int adapter_nq(int r);
// The CTAs a lone pass plans its split for, and the split of them between two passes in one
// launch (the single calls' G and dB passes).
int adapter_total_ctas();
void adapter_pair_targets(int64_t rows0, int64_t red0, int64_t rows1, int64_t red1, int* t0, int* t1);
size_t adapter_partial_bytes(int64_t rows, int64_t red, int r);
// Up to kAdapterMaxPasses independent passes (separate `partial` buffers) in one launch,
// then their finishes (at most kAdapterMaxOuts outputs in all) in one more.  A pass's
// reduction split (and so its sums' rounding order) depends only on its rows, reduction
// length and target: without targets one pass plans for every resident CTA and two passes
// share them in proportion to the bytes each reads.
cudaError_t adapter_run(const AdapterPassArgs* a, int n, int* status, cudaStream_t st);

}  // namespace qnf4
