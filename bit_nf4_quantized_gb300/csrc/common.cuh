// Internal declarations shared by the translation units of libqlora_nf4.so.
//
// The code tables reach the kernels as by-value kernel parameters (copied to
// shared memory at kernel start), so no __constant__ or __device__ state has to
// be shared between translation units.  The one piece of device state, the
// per-device status word, lives in abi.cu; kernels get its address as `status`.
#pragma once

#include <utility>

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "qlora_nf4.h"

namespace qnf4 {

constexpr int kBlock = 64;            // NF4 absmax block
constexpr int kNested = 256;          // absmax values per nested block
constexpr int kGroupElems = kBlock * kNested;
constexpr int kNf4ZeroCode = 7;       // nf4[7] == 0.0
constexpr int kDyn8ZeroCode = 127;    // dyn8[127] == 0.0

// The 16 NF4 values as published with QLoRA (Dettmers et al. 2023, appendix
// "NormalFloat 4-bit data type"), ascending.  A switch so that device code with a
// compile-time index folds it to an immediate.
__host__ __device__ constexpr float nf4_value(int i) {
  switch (i) {
    case 0: return -1.0f;
    case 1: return -0.6961928009986877f;
    case 2: return -0.5250730514526367f;
    case 3: return -0.39491748809814453f;
    case 4: return -0.28444138169288635f;
    case 5: return -0.18477343022823334f;
    case 6: return -0.09105003625154495f;
    case 7: return 0.0f;
    case 8: return 0.07958029955625534f;
    case 9: return 0.16093020141124725f;
    case 10: return 0.24611230194568634f;
    case 11: return 0.33791524171829224f;
    case 12: return 0.44070982933044434f;
    case 13: return 0.5626170039176941f;
    case 14: return 0.7229568362236023f;
    default: return 1.0f;
  }
}

// Decode tables: the 16 NF4 values and the 256 dynamic8 values, ascending.
struct DecodeTables {
  float nf4[16];
  float dyn8[256];
};

// Encode tables: thr[j] is the smallest float whose nearest code (ties to the
// lower index) is j + 1, so code(v) = #{ j : v >= thr[j] }.
struct EncodeTables {
  float nf4_thr[16];   // 15 used
  float dyn8_thr[256]; // 255 used
  // Bucketed NF4 search for a value q within a few ulp of v = x/a in [-1, 1].  The index
  // idx = (bits(q' ) >> 17) - 8191, q' = fl(x*r + 3) ~ q + 3, is 1 + the bucket k of
  // [-1 + k/32, -1 + (k+1)/32) (the top 6 mantissa bits of a value in [2, 4)), 0 for q
  // just below -1 and 65 for q >= 1.  Entry {lo, hi}: code(v) = base + (q >= hi) unless
  // lo <= q < hi (the band around the bucket's one threshold; lo = hi = 4 when none falls
  // inside); base sits in the low 4 bits of lo, which is moved away from the threshold to
  // make room (the band only widens).  Valid only when bucket_ok (at most one threshold per
  // bucket, none within 2^-18 of an edge, so an index off by one rounding near an edge
  // gives the same code).
  float nf4_band[66][2];
  int32_t bucket_ok;
  // bf16 input needs no band: with x and a bf16 values (a = max |x| of the block, so the
  // ratio is a quotient of two 8-bit significands times a power of two) and a in
  // [2^-126, 2^126) (1/a normal), the bits of q' = fl(x*r + 3) alone decide the code:
  // code(v) = sep_base[idx] + (bits(q') >= sep[idx]).  The host builds sep by running every
  // such pair through both formulas and sets sep_ok only if one cut per bucket separates
  // the codes (sep = ~0u where a bucket holds one code).
  uint32_t nf4_sep[66];
  uint32_t nf4_sep_base[66];
  int32_t sep_ok;
};

const DecodeTables& decode_tables();
const EncodeTables& encode_tables();

// Launch accounting (for the launch count reported by the ABI).
void note_launch(int n = 1);

// SM count of the current device (looked up once per device).
int device_sm_count();

// n zero ticket counters of the library's pool for one launch (which CTA of a group finishes
// last); the launch must put every counter it uses back to zero.
cudaError_t ticket_range(unsigned n, unsigned** out);

// Bounded-wait settings of one tensor-core launch: the wait limit, and whether the launch's
// first CTA leaves its first pipeline stage unissued (so that the waits for that stage run
// out).  Normally {4 s, 0}; qlora_debug_wait_timeout() arms {20 ms, 1} for the next launch.
struct WaitSettings {
  uint64_t wait_ns;
  int skip_stage0;
};
WaitSettings take_wait_settings();

// Programmatic dependent launch.  Kernels of the bf16 path are launched with
// programmatic stream serialization: a kernel may start while its predecessor in the
// stream is finishing.  Each kernel calls pdl_allow_next() once its prologue holds every
// resource it needs (shared memory set up, TMEM allocated), so the next kernel's CTAs can
// be placed as this one's retire, and pdl_wait() before it touches global memory, which
// returns once the predecessor has completed and its writes are visible.  Without a
// programmatic predecessor both are no-ops.
__device__ __forceinline__ void pdl_allow_next() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Launch `kernel` on `st` with programmatic stream serialization (and a cluster shape
// when cluster_x > 1).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       unsigned cluster_x, Args&&... args) {
  cudaLaunchConfig_t cfg{};
  cudaLaunchAttribute at[2];
  int n = 0;
  at[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[n].val.programmaticStreamSerializationAllowed = 1;
  ++n;
  if (cluster_x > 1) {
    at[n].id = cudaLaunchAttributeClusterDimension;
    at[n].val.clusterDim.x = cluster_x;
    at[n].val.clusterDim.y = 1;
    at[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = at;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Optional event timing of selected kernels (nf4_timing_enable): records a CUDA
// event pair on the launching stream around the scope when timing is on.
class KernelTimer {
 public:
  KernelTimer(int kind, cudaStream_t st);
  ~KernelTimer();
  KernelTimer(const KernelTimer&) = delete;
  KernelTimer& operator=(const KernelTimer&) = delete;

 private:
  int kind_;
  cudaStream_t st_;
  cudaEvent_t start_ = nullptr;
};

// Per-call view of an nf4_tensor for device code.
struct Nf4View {
  const uint8_t* packed;
  const void* absmax;      // uint8 codes (dq) or float
  const float* nested;
  const float* offset;     // device scalar (dq)
  int64_t numel;
  int dq;
};

// ---- quant.cu -----------------------------------------------------------------
cudaError_t launch_quantize(const void* x, nf4_dtype xd, int64_t numel, const nf4_tensor& out,
                            void* ws, int* status, cudaStream_t st);
// Up to kQuantBatchMax tensors of one input type in one block pass and one nested pass;
// each job's workspace slice holds quantize_ws_bytes(numel, dq) bytes.
constexpr int kQuantBatchMax = 8;
struct QuantJob {
  const void* x;
  int64_t numel;
  const nf4_tensor* out;
  void* ws;
};
cudaError_t launch_quantize_batch(const QuantJob* jobs, int n, nf4_dtype xd, int* status, cudaStream_t st);
size_t quantize_ws_bytes(int64_t numel, int dq);
cudaError_t launch_dequantize(const Nf4View& w, void* y, nf4_dtype od, cudaStream_t st);
// up to kQuantBatchMax tensors: one launch for those with double quantization, one for the rest
cudaError_t launch_dequantize_batch(const Nf4View* w, void* const* y, int n, nf4_dtype od, cudaStream_t st);
struct PrepJobs;
// quant.cu: the 16-bit decode of w into y (IEEE half when f16, else bf16) and `prep_ctas`
// CTAs of staging jobs, one launch.
cudaError_t launch_decode_with_prep(const Nf4View& w, void* y, bool f16, const PrepJobs& jobs, unsigned prep_ctas,
                                    cudaStream_t st);
// The prep jobs alone (a call whose weight comes already decoded).
cudaError_t launch_prep_only(bool f16, const PrepJobs& jobs, unsigned prep_ctas, cudaStream_t st);

// ---- export.cu: selected embedding rows and the merged LoRA weight ------------
cudaError_t launch_embedding_rows(const Nf4View& w, int64_t rows, int64_t dim, const int64_t* ids, int64_t n_ids,
                                  void* out, nf4_dtype od, int* status, cudaStream_t st);
cudaError_t launch_merge_lora(const Nf4View& w, int64_t N, int64_t K, int r, float s, const float* A,
                              const float* B, void* out, nf4_dtype od, cudaStream_t st);

// ---- linear_simt.cu (the fp32 profile) -----------------------------------------
struct LinearArgs {
  int64_t M, N, K;
  int r;
  float s;
  Nf4View W;
};
cudaError_t launch_lora_down(const LinearArgs& a, const float* x, const float* A, float* T, cudaStream_t st);
cudaError_t launch_fwd_simt(const LinearArgs& a, const float* x, const float* T, const float* B, float* y,
                            cudaStream_t st);
cudaError_t launch_lora_g(const LinearArgs& a, const float* dy, const float* B, float* G, cudaStream_t st);
cudaError_t launch_dx_simt(const LinearArgs& a, const float* dy, const float* G, const float* A, float* dx,
                           cudaStream_t st);
cudaError_t launch_lora_dA(const LinearArgs& a, const float* G, const float* x, float* dA, cudaStream_t st);
cudaError_t launch_lora_dB(const LinearArgs& a, const float* dy, const float* T, float* dB, cudaStream_t st);

// ---- device helpers -----------------------------------------------------------
// Round a float to the nearest bf16 value and return it as a float.
__device__ __forceinline__ float round_bf16(float v) {
  return __bfloat162float(__float2bfloat16_rn(v));
}

// a' of block b: dyn8[code] * nested + offset as two separately rounded operations
// (the decode the pages' kernels use: "decode-separate-rn"), or the fp32 absmax.
__device__ __forceinline__ float block_scale(const Nf4View& w, int64_t b, const float* dyn8_smem,
                                             float offset) {
  if (w.dq) {
    const uint8_t code = static_cast<const uint8_t*>(w.absmax)[b];
    return __fadd_rn(__fmul_rn(dyn8_smem[code], w.nested[b >> 8]), offset);
  }
  return static_cast<const float*>(w.absmax)[b];
}

// 4-bit code of flat element i (high nibble holds the even element).
__device__ __forceinline__ int nf4_code_at(const uint8_t* packed, int64_t i) {
  const uint8_t byte = packed[i >> 1];
  return (i & 1) ? (byte & 0x0F) : (byte >> 4);
}

}  // namespace qnf4
