// nf4_quantize for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc or hand out a workspace: code embedded in a
// host engine or framework that owns all device memory and gives its plugins only
// their input and output buffers, or a latency-critical loop where an allocation
// (and the implicit device synchronization cudaFree brings) is not allowed.  This
// entry point gives them double quantization anyway: the scratch nf4_quantize takes
// from its workspace (the fp32 block absmax values and the float64 group sums of the
// mean) lives here, in a fixed array in the library's own device memory.
//
// The array is a file-scope __device__ variable: every GPU that loads the library
// holds NF4_QUANTIZE_NOALLOC_SCRATCH_BYTES of it until the process exits.  In host
// code its name is only a host-side stand-in, so its device address is looked up
// with cudaGetSymbolAddress, once per device, with that device current, on the
// first call made on that device; make that first call before any stream capture.
//
// All calls share the one array and it keeps whatever the last call left there.
// Nothing in it has to start at zero (each call writes every entry it later reads),
// so nothing is cleared; calls that overlap on the GPU (different streams, or
// several host threads) race on it and must be serialized by the caller.
//
// The pages have no counterpart to this entry point; the computation is exactly
// nf4_quantize's (the same kernels, the same bytes).
#include <mutex>

#include "common.cuh"

namespace {

constexpr int64_t kMaxNumel = NF4_QUANTIZE_NOALLOC_MAX_NUMEL;
// block absmax fp32[2^20] (4 MiB) + group sums fp64[4096] padded to a power of two (32 KiB)
constexpr size_t kScratchBytes = NF4_QUANTIZE_NOALLOC_SCRATCH_BYTES;

static __device__ __align__(256) unsigned char g_quant_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
void* g_scratch_addr[kMaxDevices] = {};
std::mutex g_scratch_mu;

// Device address of g_quant_scratch on the current device (looked up once per device).
nf4_status scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return NF4_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_quant_scratch) != cudaSuccess || p == nullptr) return NF4_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return NF4_OK;
}

}  // namespace

extern "C" nf4_status nf4_quantize_noalloc(const void* x, nf4_dtype x_dtype, int64_t numel,
                                           const nf4_tensor* out, void* stream) {
  if (x == nullptr || out == nullptr || numel <= 0) return NF4_ERR_ARG;
  if (numel > kMaxNumel) return NF4_ERR_TOO_LARGE;
  if (qnf4::quantize_ws_bytes(numel, out->double_quant ? 1 : 0) > kScratchBytes) return NF4_ERR_TOO_LARGE;
  void* scratch = nullptr;
  const nf4_status st = scratch_address(&scratch);
  if (st != NF4_OK) return st;
  return nf4_quantize(x, x_dtype, numel, out, scratch, kScratchBytes, stream);
}
