// The C ABI of libqlora_nf4.so: argument validation, constant tables, the
// per-device status word, workspace layout and dispatch to the kernels.
//
// Contract ("Native model adaptation and NF4"): the NF4 base is frozen and needs an
// adapter ("One model contract"); storage is NF4 with or without double
// quantization ("Packed NF4 and the portable QLoRA profile"); rank is 1..256 and
// s = alpha / rank, rsLoRA a separate scale ("Adapter API", "LoRA FA includes
// gradient preconditioning"); no CPU fallback and no automatic precision change,
// unsupported values fail explicitly ("Explicit accelerated training profiles").
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstring>
#include <mutex>
#include <vector>

#include "common.cuh"
#include "linear_tc.cuh"

namespace qnf4 {

// ---- constant tables ---------------------------------------------------------------
namespace {

// Signed dynamic tree quantization (Dettmers et al. 2022, "8-bit Optimizers via
// Block-wise Quantization"): after the sign, E zero bits give the decade 10^-E, a
// 1 bit ends them and F = 6 - E bits pick one of 2^F equal bins of [0.1, 1]; the
// value is the bin midpoint.  The two all-zero patterns stand for 0 and +1.
// Magnitude of bin f in decade E: (2^(F+1) + 9(2f+1)) / (20 * 2^F * 10^E), an exact
// quotient of small integers, divided once in double and rounded once to float.
void build_dyn8(float out[256]) {
  float pos[127];
  int n = 0;
  for (int e = 6; e >= 0; --e) {           // ascending magnitude: smallest decade first
    const int f_bits = 6 - e;
    const int bins = 1 << f_bits;
    double pow10 = 1.0;
    for (int i = 0; i < e; ++i) pow10 *= 10.0;
    for (int f = 0; f < bins; ++f) {
      const double num = static_cast<double>((2 << f_bits) + 9 * (2 * f + 1));
      const double den = 20.0 * static_cast<double>(bins) * pow10;
      pos[n++] = static_cast<float>(num / den);
    }
  }
  for (int i = 0; i < 127; ++i) out[i] = -pos[126 - i];
  out[127] = 0.0f;
  for (int i = 0; i < 127; ++i) out[128 + i] = pos[i];
  out[255] = 1.0f;
}

// thr[j] = smallest float strictly above the exact midpoint of codes j and j+1, so
// that #{j : v >= thr[j]} is the nearest code with ties going to the lower index.
void build_thresholds(const float* codes, int n, float* thr) {
  for (int j = 0; j + 1 < n; ++j) {
    const double mid = (static_cast<double>(codes[j]) + static_cast<double>(codes[j + 1])) * 0.5;
    const float f = static_cast<float>(mid);
    thr[j] = (static_cast<double>(f) > mid) ? f : std::nextafter(f, INFINITY);
  }
  for (int j = n - 1; j < 16 && n == 16; ++j) thr[j] = INFINITY;
  if (n == 256) thr[255] = INFINITY;
}

// Bucket table for the quantizer's NF4 search: 64 buckets of width 1/32 over [-1, 1).
// lo moved down (toward -inf) by 1 to 31 ulps so that `code` fits in its low 4 bits; a lo of
// 4 (no band) stays at or above 4.
float band_lo_with_code(float lo, int code) {
  uint32_t b;
  std::memcpy(&b, &lo, 4);
  const uint32_t sign = b & 0x80000000u, mag = b & 0x7FFFFFFFu;
  uint32_t m;
  if (lo >= 4.0f) m = (mag & ~0xFu) + static_cast<uint32_t>(code);          // no band: stays >= 4
  else if (sign == 0) m = (mag & ~0xFu) - 0x10u + static_cast<uint32_t>(code);  // smaller positive
  else m = (mag & ~0xFu) + 0x10u + static_cast<uint32_t>(code);               // more negative
  const uint32_t out = sign | m;
  float f;
  std::memcpy(&f, &out, 4);
  return f;
}

void build_buckets(const float* thr, EncodeTables* e) {
  e->bucket_ok = 1;
  for (int idx = 0; idx < 66; ++idx) {
    int base = 0;
    float t_in = 4.0f;
    if (idx == 0) {
      base = 0;                       // q below -1: nearest is -1
    } else if (idx == 65) {
      base = 15;                      // q >= 1: nearest is 1
    } else {
      const int k = idx - 1;
      const double lo = -1.0 + k / 32.0, hi = lo + 1.0 / 32.0;
      int inner = 0;
      for (int j = 0; j < 15; ++j) {
        const double t = thr[j];
        if (t <= lo) ++base;
        else if (t < hi) { ++inner; t_in = thr[j]; }
        if (std::fabs(t - lo) < 1.0 / (1 << 18) || std::fabs(t - hi) < 1.0 / (1 << 18)) e->bucket_ok = 0;
      }
      if (inner > 1) e->bucket_ok = 0;
    }
    // band of +-2^-19 (relative) around the threshold: wider than the error of
    // x * RN(1/a) against RN(x / a) (a few ulp)
    const double t = t_in, w = std::fabs(t) / (1 << 19);
    const float lo = t_in == 4.0f ? 4.0f : static_cast<float>(t - w);
    const float hi = t_in == 4.0f ? 4.0f : static_cast<float>(t + w);
    e->nf4_band[idx][0] = band_lo_with_code(lo, base);
    e->nf4_band[idx][1] = hi;
  }
}

// The bf16 cut table (EncodeTables::nf4_sep): every pair x = s * mx * 2^-d, a = ma with mx, ma
// the 128 bf16 significands in [1, 2), d = 0..15 (below that |x/a| < 2^-15 and q' lands in
// the two buckets around 3, which hold code 7 alone), |x| <= a, and x = 0; scaling both by
// a power of two changes neither x/a nor fl(x*r) while 1/a stays normal.  The code of each
// pair is taken from RN(x/a) against the thresholds (the definition); its q' bits must then
// split each bucket into at most two codes with every lower-code q' below every
// higher-code q'.
void build_bf16_cuts(const float* thr, EncodeTables* e) {
  uint32_t lo_max[66], hi_min[66];
  int lo_code[66], hi_code[66];
  for (int i = 0; i < 66; ++i) lo_code[i] = 99, hi_code[i] = -1, lo_max[i] = 0, hi_min[i] = ~0u;
  bool ok = true;
  struct Pair { float x, a; };
  std::vector<Pair> pairs;
  pairs.reserve(128 * 128 * 32 + 128);
  for (int ia = 0; ia < 128; ++ia) {
    const float a = 1.0f + static_cast<float>(ia) / 128.0f;
    pairs.push_back({0.0f, a});
    for (int d = 0; d < 16; ++d)
      for (int ix = 0; ix < 128; ++ix) {
        const float m = std::ldexp(1.0f + static_cast<float>(ix) / 128.0f, -d);
        if (m > a) continue;
        pairs.push_back({m, a});
        pairs.push_back({-m, a});
      }
  }
  // two passes: the codes present in each bucket, then the cut between them
  for (int pass = 0; pass < 2 && ok; ++pass) {
    for (const Pair& p : pairs) {
      const float v = p.x / p.a;
      int code = 0;
      for (int j = 0; j < 15; ++j) code += (v >= thr[j]) ? 1 : 0;
      const float r = 1.0f / p.a;
      const float qp = std::fmaf(p.x, r, 3.0f);
      uint32_t qb;
      std::memcpy(&qb, &qp, 4);
      const int64_t idx = static_cast<int64_t>(qb >> 17) - 8191;
      if (idx < 0 || idx > 65) { ok = false; break; }
      if (pass == 0) {
        lo_code[idx] = std::min(lo_code[idx], code);
        hi_code[idx] = std::max(hi_code[idx], code);
      } else if (code == lo_code[idx]) {
        lo_max[idx] = std::max(lo_max[idx], qb);
      } else {
        hi_min[idx] = std::min(hi_min[idx], qb);
      }
    }
    if (pass == 0)
      for (int i = 0; i < 66; ++i)
        if (hi_code[i] - lo_code[i] > 1) ok = false;
  }
  for (int i = 0; i < 66 && ok; ++i) {
    if (hi_code[i] < 0) {                      // no bf16 pair lands here
      e->nf4_sep_base[i] = 0;
      e->nf4_sep[i] = ~0u;
    } else if (hi_code[i] == lo_code[i]) {
      e->nf4_sep_base[i] = static_cast<uint32_t>(lo_code[i]);
      e->nf4_sep[i] = ~0u;
    } else {
      if (!(lo_max[i] < hi_min[i])) ok = false;
      e->nf4_sep_base[i] = static_cast<uint32_t>(lo_code[i]);
      e->nf4_sep[i] = hi_min[i];
    }
  }
  e->sep_ok = ok ? 1 : 0;
}

struct Tables {
  DecodeTables dec;
  EncodeTables enc;
  Tables() {
    for (int i = 0; i < 16; ++i) dec.nf4[i] = nf4_value(i);
    build_dyn8(dec.dyn8);
    build_thresholds(dec.nf4, 16, enc.nf4_thr);
    build_thresholds(dec.dyn8, 256, enc.dyn8_thr);
    build_buckets(enc.nf4_thr, &enc);
    build_bf16_cuts(enc.nf4_thr, &enc);
  }
};

const Tables& tables() {
  static const Tables t;
  return t;
}

std::atomic<int64_t> g_launches{0};

// One status word per device (the module's copy on each device).
__device__ int g_device_status;

constexpr int kMaxDevices = 64;
int* g_status_addr[kMaxDevices] = {};
std::mutex g_status_mu;

nf4_status device_status_ptr(int** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return NF4_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_status_mu);
  if (g_status_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_status) != cudaSuccess) return NF4_ERR_CUDA;
    g_status_addr[dev] = static_cast<int*>(p);
  }
  *out = g_status_addr[dev];
  return NF4_OK;
}

}  // namespace

// ---- optional kernel timing ------------------------------------------------------
namespace {

struct TimingState {
  std::mutex mu;
  std::atomic<bool> enabled{false};
  std::vector<cudaEvent_t> pool;
  std::vector<std::pair<cudaEvent_t, cudaEvent_t>> pending[NF4_TIME_KINDS];
  double total_ms[NF4_TIME_KINDS] = {};
  int64_t count[NF4_TIME_KINDS] = {};
};

TimingState& timing() {
  static TimingState t;
  return t;
}

cudaEvent_t take_event(TimingState& t) {
  std::lock_guard<std::mutex> lock(t.mu);
  if (!t.pool.empty()) {
    cudaEvent_t e = t.pool.back();
    t.pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  return e;
}

}  // namespace

KernelTimer::KernelTimer(int kind, cudaStream_t st) : kind_(kind), st_(st) {
  TimingState& t = timing();
  if (!t.enabled.load(std::memory_order_relaxed)) return;
  start_ = take_event(t);
  if (start_ != nullptr && cudaEventRecord(start_, st_) != cudaSuccess) {
    std::lock_guard<std::mutex> lock(t.mu);
    t.pool.push_back(start_);
    start_ = nullptr;
  }
}

KernelTimer::~KernelTimer() {
  if (start_ == nullptr) return;
  TimingState& t = timing();
  cudaEvent_t stop = take_event(t);
  std::lock_guard<std::mutex> lock(t.mu);
  if (stop == nullptr || cudaEventRecord(stop, st_) != cudaSuccess) {
    t.pool.push_back(start_);
    if (stop != nullptr) t.pool.push_back(stop);
    return;
  }
  t.pending[kind_].emplace_back(start_, stop);
}

namespace {
std::atomic<int> g_wait_fault{0};
}  // namespace

WaitSettings take_wait_settings() {
  if (g_wait_fault.exchange(0) != 0) return WaitSettings{20000000ull, 1};
  return WaitSettings{4000000000ull, 0};
}

const DecodeTables& decode_tables() { return tables().dec; }
const EncodeTables& encode_tables() { return tables().enc; }

int device_sm_count() {
  constexpr int kMaxDev = 64;
  static std::atomic<int> cache[kMaxDev];
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < kMaxDev) {
    const int c = cache[dev].load(std::memory_order_relaxed);
    if (c > 0) return c;
  }
  int n = 0;
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  n = n > 0 ? n : 1;
  if (dev >= 0 && dev < kMaxDev) cache[dev].store(n, std::memory_order_relaxed);
  return n;
}
void note_launch(int n) { g_launches.fetch_add(n, std::memory_order_relaxed); }

}  // namespace qnf4

using namespace qnf4;

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t a256(size_t b) { return (b + 255) & ~static_cast<size_t>(255); }

nf4_status from_cuda(cudaError_t e) { return e == cudaSuccess ? NF4_OK : NF4_ERR_CUDA; }

// Checks an nf4_tensor descriptor against an expected element count.
nf4_status check_tensor(const nf4_tensor* t, int64_t numel) {
  if (t == nullptr) return NF4_ERR_ARG;
  if (t->numel != numel || t->numel <= 0) return NF4_ERR_CORRUPT;
  if ((t->double_quant != 0 && t->double_quant != 1) || t->reserved != 0) return NF4_ERR_CORRUPT;
  if (t->packed == nullptr || t->absmax == nullptr) return NF4_ERR_ARG;
  if (t->double_quant) {
    if (t->nested_absmax == nullptr || t->offset == nullptr) return NF4_ERR_CORRUPT;
  } else if (t->nested_absmax != nullptr || t->offset != nullptr) {
    return NF4_ERR_CORRUPT;
  }
  if (!aligned16(t->packed) || !aligned16(t->absmax)) return NF4_ERR_ALIGN;
  if (t->double_quant && (!aligned16(t->nested_absmax) || !aligned16(t->offset))) return NF4_ERR_ALIGN;
  return NF4_OK;
}

Nf4View view_of(const nf4_tensor* t) {
  Nf4View v;
  v.packed = t->packed;
  v.absmax = t->absmax;
  v.nested = t->nested_absmax;
  v.offset = t->offset;
  v.numel = t->numel;
  v.dq = t->double_quant;
  return v;
}

nf4_status check_linear(int64_t M, int64_t N, int64_t K, int32_t rank, float alpha,
                        qlora_scale_mode mode, nf4_dtype compute, float* s_out) {
  if (M < 0 || N <= 0 || K <= 0) return NF4_ERR_ARG;
  if (N > (int64_t(1) << 40) / K) return NF4_ERR_SHAPE;
  if (rank < 1 || rank > 256 || rank > N || rank > K) return NF4_ERR_ARG;
  if (!std::isfinite(alpha)) return NF4_ERR_ARG;
  if (mode != QLORA_SCALE_LORA && mode != QLORA_SCALE_RSLORA) return NF4_ERR_ARG;
  if (compute != NF4_F32 && compute != NF4_BF16 && compute != NF4_F16) return NF4_ERR_DTYPE;
  if (compute != NF4_F32 && (K % 64 != 0 || N % 8 != 0)) return NF4_ERR_SHAPE;
  *s_out = (mode == QLORA_SCALE_LORA)
               ? alpha / static_cast<float>(rank)
               : static_cast<float>(static_cast<double>(alpha) / std::sqrt(static_cast<double>(rank)));
  return NF4_OK;
}

// The two 16-bit compute dtypes run on the tensor cores; NF4_F32 on the CUDA cores.
bool is16(nf4_dtype cd) { return cd == NF4_BF16 || cd == NF4_F16; }

bool small_m(int64_t M, nf4_dtype cd) { return is16(cd) && M >= 1 && M <= kStreamMaxM; }

// Small weights at M > 16 run the fused small-shape kernels (one launch forward, one backward).
bool small_w(int64_t M, int64_t N, int64_t K, int32_t r, nf4_dtype cd) {
  return is16(cd) && M > kStreamMaxM && small_fused_fits(N, K, r);
}

size_t small_bwd_ws(int64_t M, int64_t N, int64_t K, int32_t r) {
  SmallItem it{};
  it.a = LinearArgs{M, N, K, r, 0.0f, Nf4View{}};
  return small_fused_bwd_ws_bytes(&it, 1, M);
}

// Workspace layouts.  bwd: G fp32 [M, r], then whatever the selected path needs.
size_t fwd_ws(int64_t M, int64_t N, int64_t K, int32_t r, nf4_dtype cd) {
  if (small_m(M, cd)) {
    LinearArgs la{M, N, K, r, 0.0f, Nf4View{}};
    return stream_fwd_ws_bytes(&la, 1);
  }
  if (small_w(M, N, K, r, cd)) return 0;
  if (is16(cd)) return tc_fwd_ws_bytes(M, N, K, r);
  return 0;
}

// Argument checks of one forward call (everything but the workspace); s receives the scale.
nf4_status check_fwd(int64_t M, int64_t N, int64_t K, int32_t rank, float alpha, qlora_scale_mode mode,
                     nf4_dtype compute, const void* x, const nf4_tensor* W, const float* A, const float* B,
                     const void* y, const float* T_out, float* s) {
  nf4_status st = check_linear(M, N, K, rank, alpha, mode, compute, s);
  if (st != NF4_OK) return st;
  if ((st = check_tensor(W, N * K)) != NF4_OK) return st;
  if (A == nullptr || B == nullptr) return NF4_ERR_ARG;
  if (M > 0 && (x == nullptr || y == nullptr || T_out == nullptr)) return NF4_ERR_ARG;
  if (!aligned16(A) || !aligned16(B) || (M > 0 && (!aligned16(x) || !aligned16(y) || !aligned16(T_out))))
    return NF4_ERR_ALIGN;
  return NF4_OK;
}

size_t bwd_ws(int64_t M, int64_t N, int64_t K, int32_t r, nf4_dtype cd) {
  if (small_w(M, N, K, r, cd)) return small_bwd_ws(M, N, K, r);
  size_t b = a256(sizeof(float) * static_cast<size_t>(M) * r);
  if (is16(cd)) b += tc_bwd_ws_bytes(M, N, K, r);
  return b;
}

// How a batch runs, as a list of runs in order; every run uses the whole workspace, one
// after another on the stream:
//   kRunStream: items given as NF4 at M <= 16 (16-bit), up to kStreamMaxGroup, one stream pass;
//   kRunSmall:  small weights, up to kSmallMaxGroup in one fused launch (a pair backward);
//   kRunGroup:  up to kTcGroupMax tiled items in a row: their adapter passes share launches,
//               and items that read the same x share a pass (a run of one item is the single
//               call);
//   kRunSingle: one single call (fp32 compute, or no tokens).
enum { kRunStream, kRunSmall, kRunGroup, kRunSingle };
struct BatchRun {
  int kind;
  std::vector<int> idx;
};

template <typename KindOf>
std::vector<BatchRun> plan_batch(int32_t count, KindOf kind_of) {
  std::vector<BatchRun> runs;
  BatchRun stream{kRunStream, {}}, small{kRunSmall, {}}, group{kRunGroup, {}};
  auto flush = [&](BatchRun& b) {
    if (!b.idx.empty()) runs.push_back(b);
    b.idx.clear();
  };
  for (int i = 0; i < count; ++i) {
    const int k = kind_of(i);
    if (k == kRunStream) {
      stream.idx.push_back(i);
      if (static_cast<int>(stream.idx.size()) == kStreamMaxGroup) flush(stream);
    } else if (k == kRunSmall) {
      small.idx.push_back(i);
      if (static_cast<int>(small.idx.size()) == kSmallMaxGroup) flush(small);
    } else if (k == kRunGroup) {
      group.idx.push_back(i);
      if (static_cast<int>(group.idx.size()) == kTcGroupMax) flush(group);
    } else {
      runs.push_back(BatchRun{kRunSingle, {i}});
    }
  }
  flush(group);
  flush(stream);
  flush(small);
  return runs;
}

std::vector<BatchRun> plan_fwd(int64_t M, int32_t count, const qlora_fwd_item* it, nf4_dtype cd) {
  return plan_batch(
      count,
      [&](int i) {
        if (!is16(cd) || M == 0) return static_cast<int>(kRunSingle);
        if (it[i].w16 == nullptr && small_m(M, cd)) return static_cast<int>(kRunStream);
        if (small_w(M, it[i].N, it[i].K, it[i].rank, cd)) return static_cast<int>(kRunSmall);
        return static_cast<int>(kRunGroup);
      });
}

std::vector<BatchRun> plan_bwd(int64_t M, int32_t count, const qlora_bwd_item* it, nf4_dtype cd) {
  return plan_batch(
      count,
      [&](int i) {
        if (!is16(cd) || M == 0) return static_cast<int>(kRunSingle);
        if (small_w(M, it[i].N, it[i].K, it[i].rank, cd)) return static_cast<int>(kRunSmall);
        return static_cast<int>(kRunGroup);
      });
}

// (the weight view only when `view`: workspace sizes are asked before any validation)
TcFwdItem tc_fwd_item(int64_t M, const qlora_fwd_item& it, float s, bool view = true) {
  TcFwdItem t{};
  t.a = LinearArgs{M, it.N, it.K, it.rank, s, (it.w16 != nullptr || !view) ? Nf4View{} : view_of(it.W)};
  t.x = it.x, t.A = it.A, t.B = it.B, t.y = it.y, t.T = it.T_out, t.w16 = it.w16;
  return t;
}

TcBwdItem tc_bwd_item(int64_t M, const qlora_bwd_item& it, float s, bool view = true) {
  TcBwdItem t{};
  t.a = LinearArgs{M, it.N, it.K, it.rank, s, (it.w16 != nullptr || !view) ? Nf4View{} : view_of(it.W)};
  t.x = it.x, t.dy = it.dy, t.T = it.T, t.A = it.A, t.B = it.B, t.dx = it.dx, t.dA = it.dA, t.dB = it.dB;
  t.w16 = it.w16;
  return t;
}

}  // namespace

extern "C" {

int32_t nf4_abi_version(void) { return QLORA_NF4_ABI_VERSION; }

const char* nf4_status_str(nf4_status s) {
  switch (s) {
    case NF4_OK: return "ok";
    case NF4_ERR_ARG: return "invalid argument";
    case NF4_ERR_SHAPE: return "unsupported shape";
    case NF4_ERR_ALIGN: return "device pointer not 16-byte aligned";
    case NF4_ERR_DTYPE: return "unsupported dtype";
    case NF4_ERR_NONFINITE: return "non-finite input";
    case NF4_ERR_CORRUPT: return "inconsistent NF4 descriptor";
    case NF4_ERR_CUDA: return "CUDA runtime error";
    case NF4_ERR_TIMEOUT: return "device-side wait timed out";
    case NF4_ERR_WORKSPACE: return "workspace missing or too small";
    case NF4_ERR_TOO_LARGE: return "numel above the fixed scratch limit of nf4_quantize_noalloc";
  }
  return "unknown status";
}

int64_t nf4_num_blocks(int64_t numel) { return numel <= 0 ? 0 : (numel + kBlock - 1) / kBlock; }
int64_t nf4_num_nested(int64_t numel) {
  return numel <= 0 ? 0 : (nf4_num_blocks(numel) + kNested - 1) / kNested;
}

size_t nf4_packed_bytes(int64_t numel, int32_t double_quant) {
  if (numel <= 0) return 0;
  const size_t packed = static_cast<size_t>((numel + 1) / 2);
  const size_t nb = static_cast<size_t>(nf4_num_blocks(numel));
  if (!double_quant) return packed + 4 * nb;
  return packed + nb + 4 * static_cast<size_t>(nf4_num_nested(numel));
}

void nf4_code_tables(float* nf4_out16, float* dyn8_out256) {
  const DecodeTables& t = decode_tables();
  if (nf4_out16) std::memcpy(nf4_out16, t.nf4, sizeof(t.nf4));
  if (dyn8_out256) std::memcpy(dyn8_out256, t.dyn8, sizeof(t.dyn8));
}

size_t nf4_quantize_workspace_bytes(int64_t numel, int32_t double_quant) {
  return numel <= 0 ? 0 : quantize_ws_bytes(numel, double_quant ? 1 : 0);
}

nf4_status nf4_quantize(const void* x, nf4_dtype x_dtype, int64_t numel, const nf4_tensor* out,
                        void* ws, size_t ws_bytes, void* stream) {
  if (x == nullptr || numel <= 0) return NF4_ERR_ARG;
  if (x_dtype != NF4_F32 && x_dtype != NF4_BF16) return NF4_ERR_DTYPE;
  nf4_status st = check_tensor(out, numel);
  if (st != NF4_OK) return st;
  if (!aligned16(x)) return NF4_ERR_ALIGN;
  const size_t need = quantize_ws_bytes(numel, out->double_quant);
  if (need > 0 && (ws == nullptr || ws_bytes < need)) return NF4_ERR_WORKSPACE;
  if (need > 0 && !aligned16(ws)) return NF4_ERR_ALIGN;
  int* status = nullptr;
  if ((st = device_status_ptr(&status)) != NF4_OK) return st;
  KernelTimer timer(NF4_TIME_QUANTIZE, static_cast<cudaStream_t>(stream));
  return from_cuda(launch_quantize(x, x_dtype, numel, *out, ws, status,
                                   static_cast<cudaStream_t>(stream)));
}

size_t nf4_quantize_batch_workspace_bytes(int32_t count, const nf4_quantize_item* items) {
  if (count < 1 || items == nullptr) return 0;
  size_t total = 0;
  for (int32_t i = 0; i < count; ++i) {
    if (items[i].numel <= 0 || items[i].out == nullptr) return 0;
    total += a256(quantize_ws_bytes(items[i].numel, items[i].out->double_quant ? 1 : 0));
  }
  return total;
}

nf4_status nf4_quantize_batch(int32_t count, const nf4_quantize_item* items, void* ws, size_t ws_bytes,
                              void* stream) {
  if (count < 1 || items == nullptr) return NF4_ERR_ARG;
  size_t need = 0;
  for (int32_t i = 0; i < count; ++i) {   // every item is checked before anything is enqueued
    const nf4_quantize_item& it = items[i];
    if (it.x == nullptr || it.numel <= 0 || it.out == nullptr) return NF4_ERR_ARG;
    if (it.x_dtype != NF4_F32 && it.x_dtype != NF4_BF16) return NF4_ERR_DTYPE;
    const nf4_status st = check_tensor(it.out, it.numel);
    if (st != NF4_OK) return st;
    if (!aligned16(it.x)) return NF4_ERR_ALIGN;
    need += a256(quantize_ws_bytes(it.numel, it.out->double_quant ? 1 : 0));
  }
  if (need > 0 && (ws == nullptr || ws_bytes < need)) return NF4_ERR_WORKSPACE;
  if (need > 0 && !aligned16(ws)) return NF4_ERR_ALIGN;
  int* status = nullptr;
  nf4_status st = device_status_ptr(&status);
  if (st != NF4_OK) return st;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  KernelTimer timer(NF4_TIME_QUANTIZE, cs);
  // runs of up to kQuantBatchMax items of one input type, in the items' order
  std::vector<QuantJob> jobs;
  char* w = static_cast<char*>(ws);
  for (int32_t i = 0; i < count;) {
    jobs.clear();
    const nf4_dtype xd = items[i].x_dtype;
    for (; i < count && items[i].x_dtype == xd && static_cast<int>(jobs.size()) < kQuantBatchMax; ++i) {
      jobs.push_back(QuantJob{items[i].x, items[i].numel, items[i].out, w});
      w += a256(quantize_ws_bytes(items[i].numel, items[i].out->double_quant ? 1 : 0));
    }
    const cudaError_t e = launch_quantize_batch(jobs.data(), static_cast<int>(jobs.size()), xd, status, cs);
    if (e != cudaSuccess) return from_cuda(e);
  }
  return NF4_OK;
}

nf4_status nf4_dequantize(const nf4_tensor* w, void* y, nf4_dtype out_dtype, void* stream) {
  if (w == nullptr || y == nullptr) return NF4_ERR_ARG;
  if (out_dtype != NF4_F32 && out_dtype != NF4_BF16 && out_dtype != NF4_F16) return NF4_ERR_DTYPE;
  nf4_status st = check_tensor(w, w->numel);
  if (st != NF4_OK) return st;
  if (!aligned16(y)) return NF4_ERR_ALIGN;
  KernelTimer timer(NF4_TIME_DEQUANTIZE, static_cast<cudaStream_t>(stream));
  return from_cuda(launch_dequantize(view_of(w), y, out_dtype, static_cast<cudaStream_t>(stream)));
}

nf4_status nf4_dequantize_batch(int32_t count, const nf4_dequantize_item* items, nf4_dtype out_dtype, void* stream) {
  if (count < 1 || items == nullptr) return NF4_ERR_ARG;
  if (out_dtype != NF4_F32 && out_dtype != NF4_BF16 && out_dtype != NF4_F16) return NF4_ERR_DTYPE;
  for (int32_t i = 0; i < count; ++i) {   // every item is checked before anything is enqueued
    const nf4_dequantize_item& it = items[i];
    if (it.w == nullptr || it.y == nullptr) return NF4_ERR_ARG;
    const nf4_status st = check_tensor(it.w, it.w->numel);
    if (st != NF4_OK) return st;
    if (!aligned16(it.y)) return NF4_ERR_ALIGN;
  }
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  KernelTimer timer(NF4_TIME_DEQUANTIZE, cs);
  // runs of up to kQuantBatchMax items, in the items' order
  for (int32_t i = 0; i < count;) {
    Nf4View views[kQuantBatchMax];
    void* ys[kQuantBatchMax];
    int n = 0;
    for (; i < count && n < kQuantBatchMax; ++i, ++n) {
      views[n] = view_of(items[i].w);
      ys[n] = items[i].y;
    }
    const cudaError_t e = launch_dequantize_batch(views, ys, n, out_dtype, cs);
    if (e != cudaSuccess) return from_cuda(e);
  }
  return NF4_OK;
}

nf4_status nf4_embedding_rows(const nf4_tensor* E, int64_t rows, int64_t dim, const int64_t* ids,
                              int64_t n_ids, void* out, nf4_dtype out_dtype, void* stream) {
  if (E == nullptr || rows <= 0 || dim <= 0 || n_ids < 0) return NF4_ERR_ARG;
  if (out_dtype != NF4_F32 && out_dtype != NF4_BF16) return NF4_ERR_DTYPE;
  if (rows > (int64_t(1) << 40) / dim) return NF4_ERR_SHAPE;
  nf4_status st = check_tensor(E, rows * dim);
  if (st != NF4_OK) return st;
  if (n_ids == 0) return NF4_OK;
  if (ids == nullptr || out == nullptr) return NF4_ERR_ARG;
  if (n_ids > (int64_t(1) << 40) / dim) return NF4_ERR_SHAPE;
  if (!aligned16(ids) || !aligned16(out)) return NF4_ERR_ALIGN;
  int* status = nullptr;
  if ((st = device_status_ptr(&status)) != NF4_OK) return st;
  KernelTimer timer(NF4_TIME_EMBEDDING, static_cast<cudaStream_t>(stream));
  return from_cuda(launch_embedding_rows(view_of(E), rows, dim, ids, n_ids, out, out_dtype, status,
                                         static_cast<cudaStream_t>(stream)));
}

nf4_status nf4_merge_lora(int64_t N, int64_t K, int32_t rank, float alpha, qlora_scale_mode mode,
                          const nf4_tensor* W, const float* A, const float* B, void* out,
                          nf4_dtype out_dtype, void* stream) {
  float s = 0.0f;
  // the scale rules of the linear; the dtype here is the output's
  if (out_dtype != NF4_F32 && out_dtype != NF4_BF16) return NF4_ERR_DTYPE;
  nf4_status st = check_linear(0, N, K, rank, alpha, mode, NF4_F32, &s);
  if (st != NF4_OK) return st;
  if (K % 8 != 0) return NF4_ERR_SHAPE;
  if (W == nullptr || A == nullptr || B == nullptr || out == nullptr) return NF4_ERR_ARG;
  if ((st = check_tensor(W, N * K)) != NF4_OK) return st;
  if (!aligned16(A) || !aligned16(B) || !aligned16(out)) return NF4_ERR_ALIGN;
  KernelTimer timer(NF4_TIME_MERGE, static_cast<cudaStream_t>(stream));
  return from_cuda(launch_merge_lora(view_of(W), N, K, rank, s, A, B, out, out_dtype,
                                     static_cast<cudaStream_t>(stream)));
}

size_t qlora_fwd_workspace_bytes(int64_t M, int64_t N, int64_t K, int32_t rank, nf4_dtype compute) {
  if (M < 0 || N <= 0 || K <= 0 || rank < 1 || rank > 256) return 0;
  return fwd_ws(M, N, K, rank, compute);
}

size_t qlora_bwd_workspace_bytes(int64_t M, int64_t N, int64_t K, int32_t rank, nf4_dtype compute) {
  if (M < 0 || N <= 0 || K <= 0 || rank < 1 || rank > 256) return 0;
  return bwd_ws(M, N, K, rank, compute);
}

nf4_status qlora_linear_fwd(int64_t M, int64_t N, int64_t K, int32_t rank, float alpha,
                            qlora_scale_mode mode, nf4_dtype compute,
                            const void* x, const nf4_tensor* W, const float* A, const float* B,
                            void* y, float* T_out, void* ws, size_t ws_bytes, void* stream) {
  float s = 0.0f;
  nf4_status st = check_fwd(M, N, K, rank, alpha, mode, compute, x, W, A, B, y, T_out, &s);
  if (st != NF4_OK) return st;
  const size_t need = fwd_ws(M, N, K, rank, compute);
  if (need > 0 && (ws == nullptr || ws_bytes < need)) return NF4_ERR_WORKSPACE;
  if (need > 0 && !aligned16(ws)) return NF4_ERR_ALIGN;
  if (M == 0) return NF4_OK;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  LinearArgs a{M, N, K, rank, s, view_of(W)};
  if (small_m(M, compute)) {
    int* status = nullptr;
    if ((st = device_status_ptr(&status)) != NF4_OK) return st;
    const StreamItem item{a, x, A, B, y, T_out};
    return from_cuda(stream_forward(&item, 1, compute == NF4_F16, ws, status, cs));
  }
  if (small_w(M, N, K, rank, compute)) {
    SmallItem it{};
    it.a = a;
    it.x = x, it.A = A, it.B = B, it.y = y, it.T = T_out;
    return from_cuda(small_fused_forward(&it, 1, M, compute == NF4_F16, cs));
  }
  if (is16(compute)) {
    int* status = nullptr;
    if ((st = device_status_ptr(&status)) != NF4_OK) return st;
    return from_cuda(tc_forward(a, compute == NF4_F16, x, A, B, y, T_out, ws, status, cs));
  }
  const float* xf = static_cast<const float*>(x);
  cudaError_t e = launch_lora_down(a, xf, A, T_out, cs);
  if (e == cudaSuccess) e = launch_fwd_simt(a, xf, T_out, B, static_cast<float*>(y), cs);
  return from_cuda(e);
}

size_t qlora_fwd_batch_workspace_bytes(int64_t M, int32_t count, const qlora_fwd_item* items, nf4_dtype compute) {
  if (M < 0 || count < 1 || items == nullptr) return 0;
  for (int32_t i = 0; i < count; ++i)
    if (items[i].N <= 0 || items[i].K <= 0 || items[i].rank < 1 || items[i].rank > 256) return 0;
  size_t need = 0;
  for (const BatchRun& r : plan_fwd(M, count, items, compute)) {
    const int n = static_cast<int>(r.idx.size());
    if (r.kind == kRunStream) {
      LinearArgs la[kStreamMaxGroup];
      for (int k = 0; k < n; ++k) {
        const qlora_fwd_item& it = items[r.idx[k]];
        la[k] = LinearArgs{M, it.N, it.K, it.rank, 0.0f, Nf4View{}};
      }
      need = std::max(need, stream_fwd_ws_bytes(la, n));
    } else if (r.kind == kRunGroup && n > 1) {
      TcFwdItem t[kTcGroupMax];
      for (int k = 0; k < n; ++k) t[k] = tc_fwd_item(M, items[r.idx[k]], 0.0f, false);
      need = std::max(need, tc_fwd_run_ws_bytes(t, n));
    } else if (r.kind != kRunSmall) {
      const qlora_fwd_item& it = items[r.idx[0]];
      need = std::max(need, it.w16 != nullptr ? qlora_fwd_w16_workspace_bytes(M, it.N, it.K, it.rank, compute)
                                              : fwd_ws(M, it.N, it.K, it.rank, compute));
    }
  }
  return need;
}

nf4_status qlora_linear_fwd_batch(int64_t M, int32_t count, const qlora_fwd_item* items, nf4_dtype compute,
                                  void* ws, size_t ws_bytes, void* stream) {
  if (count < 1 || items == nullptr) return NF4_ERR_ARG;
  std::vector<float> s(static_cast<size_t>(count));
  for (int32_t i = 0; i < count; ++i) {   // the single calls' checks, before anything is enqueued
    const qlora_fwd_item& it = items[i];
    nf4_status st;
    if (it.w16 != nullptr) {
      if ((st = check_linear(M, it.N, it.K, it.rank, it.alpha, it.mode, compute, &s[i])) != NF4_OK) return st;
      if (!is16(compute)) return NF4_ERR_DTYPE;
      if (it.A == nullptr || it.B == nullptr) return NF4_ERR_ARG;
      if (M > 0 && (it.x == nullptr || it.y == nullptr || it.T_out == nullptr)) return NF4_ERR_ARG;
      if (!aligned16(it.w16) || !aligned16(it.A) || !aligned16(it.B) ||
          (M > 0 && (!aligned16(it.x) || !aligned16(it.y) || !aligned16(it.T_out))))
        return NF4_ERR_ALIGN;
    } else if ((st = check_fwd(M, it.N, it.K, it.rank, it.alpha, it.mode, compute, it.x, it.W, it.A, it.B, it.y,
                               it.T_out, &s[i])) != NF4_OK) {
      return st;
    }
  }
  const size_t need = qlora_fwd_batch_workspace_bytes(M, count, items, compute);
  if (need > 0 && (ws == nullptr || ws_bytes < need)) return NF4_ERR_WORKSPACE;
  if (need > 0 && !aligned16(ws)) return NF4_ERR_ALIGN;
  if (M == 0) return NF4_OK;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  const bool f16 = compute == NF4_F16;
  int* status = nullptr;
  for (const BatchRun& r : plan_fwd(M, count, items, compute)) {
    const int n = static_cast<int>(r.idx.size());
    const int i0 = r.idx[0];
    if ((r.kind == kRunStream || (r.kind == kRunGroup && n > 1)) && status == nullptr) {
      const nf4_status st = device_status_ptr(&status);
      if (st != NF4_OK) return st;
    }
    cudaError_t e = cudaSuccess;
    if (r.kind == kRunStream) {
      StreamItem group[kStreamMaxGroup];
      for (int k = 0; k < n; ++k) {
        const qlora_fwd_item& it = items[r.idx[k]];
        group[k] = StreamItem{LinearArgs{M, it.N, it.K, it.rank, s[r.idx[k]], view_of(it.W)}, it.x, it.A, it.B, it.y,
                              it.T_out};
      }
      e = stream_forward(group, n, f16, ws, status, cs);
    } else if (r.kind == kRunSmall) {
      SmallItem small[kSmallMaxGroup];
      for (int k = 0; k < n; ++k) {
        const qlora_fwd_item& it = items[r.idx[k]];
        SmallItem& si = small[k];
        si = SmallItem{};
        si.a = LinearArgs{M, it.N, it.K, it.rank, s[r.idx[k]], it.w16 != nullptr ? Nf4View{} : view_of(it.W)};
        si.x = it.x, si.A = it.A, si.B = it.B, si.y = it.y, si.T = it.T_out, si.w16 = it.w16;
      }
      e = small_fused_forward(small, n, M, f16, cs);
    } else if (r.kind == kRunGroup && n > 1) {
      TcFwdItem t[kTcGroupMax];
      for (int k = 0; k < n; ++k) t[k] = tc_fwd_item(M, items[r.idx[k]], s[r.idx[k]]);
      e = tc_forward_run(t, n, f16, ws, status, cs);
    } else {
      const qlora_fwd_item& it = items[i0];
      const nf4_status st =
          it.w16 != nullptr
              ? qlora_linear_fwd_w16(M, it.N, it.K, it.rank, it.alpha, it.mode, compute, it.x, it.w16, it.A, it.B,
                                     it.y, it.T_out, ws, ws_bytes, stream)
              : qlora_linear_fwd(M, it.N, it.K, it.rank, it.alpha, it.mode, compute, it.x, it.W, it.A, it.B, it.y,
                                 it.T_out, ws, ws_bytes, stream);
      if (st != NF4_OK) return st;
    }
    if (e != cudaSuccess) return NF4_ERR_CUDA;
  }
  return NF4_OK;
}

nf4_status qlora_linear_bwd(int64_t M, int64_t N, int64_t K, int32_t rank, float alpha,
                            qlora_scale_mode mode, nf4_dtype compute,
                            const void* dy, const void* x, const float* T,
                            const nf4_tensor* W, const float* A, const float* B,
                            void* dx, float* dA, float* dB,
                            void* ws, size_t ws_bytes, void* stream) {
  float s = 0.0f;
  nf4_status st = check_linear(M, N, K, rank, alpha, mode, compute, &s);
  if (st != NF4_OK) return st;
  if ((st = check_tensor(W, N * K)) != NF4_OK) return st;
  if (A == nullptr || B == nullptr || dA == nullptr || dB == nullptr) return NF4_ERR_ARG;
  if (M > 0 && (dy == nullptr || x == nullptr || T == nullptr || dx == nullptr)) return NF4_ERR_ARG;
  if (!aligned16(A) || !aligned16(B) || !aligned16(dA) || !aligned16(dB)) return NF4_ERR_ALIGN;
  if (M > 0 && (!aligned16(dy) || !aligned16(x) || !aligned16(T) || !aligned16(dx))) return NF4_ERR_ALIGN;
  const size_t need = bwd_ws(M, N, K, rank, compute);
  if (ws == nullptr || ws_bytes < need) return NF4_ERR_WORKSPACE;
  if (!aligned16(ws)) return NF4_ERR_ALIGN;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  if (M == 0) {   // no tokens: the adapter gradients are zero
    cudaError_t e = cudaMemsetAsync(dA, 0, sizeof(float) * static_cast<size_t>(rank) * K, cs);
    if (e == cudaSuccess) e = cudaMemsetAsync(dB, 0, sizeof(float) * static_cast<size_t>(N) * rank, cs);
    return from_cuda(e);
  }
  LinearArgs a{M, N, K, rank, s, view_of(W)};
  if (small_w(M, N, K, rank, compute)) {
    SmallItem it{};
    it.a = a;
    it.x = x, it.A = A, it.B = B, it.T = const_cast<float*>(T), it.dy = dy, it.dx = dx, it.dA = dA, it.dB = dB;
    return from_cuda(small_fused_backward(&it, 1, M, compute == NF4_F16, ws, cs));
  }
  float* G = static_cast<float*>(ws);
  if (is16(compute)) {
    int* status = nullptr;
    if ((st = device_status_ptr(&status)) != NF4_OK) return st;
    void* tc_ws = static_cast<char*>(ws) + a256(sizeof(float) * static_cast<size_t>(M) * rank);
    return from_cuda(tc_backward(a, compute == NF4_F16, dy, x, T, A, B, dx, dA, dB, G, tc_ws, status, cs));
  }
  const float* dyf = static_cast<const float*>(dy);
  cudaError_t e = launch_lora_g(a, dyf, B, G, cs);
  if (e == cudaSuccess) e = launch_dx_simt(a, dyf, G, A, static_cast<float*>(dx), cs);
  if (e == cudaSuccess) e = launch_lora_dA(a, G, static_cast<const float*>(x), dA, cs);
  if (e == cudaSuccess) e = launch_lora_dB(a, dyf, T, dB, cs);
  return from_cuda(e);
}

size_t qlora_fwd_w16_workspace_bytes(int64_t M, int64_t N, int64_t K, int32_t rank, nf4_dtype compute) {
  if (M < 0 || N <= 0 || K <= 0 || rank < 1 || rank > 256 || !is16(compute)) return 0;
  if (small_w(M, N, K, rank, compute)) return 0;
  return tc_fwd_ws_bytes(M, N, K, rank, true);
}

size_t qlora_bwd_w16_workspace_bytes(int64_t M, int64_t N, int64_t K, int32_t rank, nf4_dtype compute) {
  if (M < 0 || N <= 0 || K <= 0 || rank < 1 || rank > 256 || !is16(compute)) return 0;
  if (small_w(M, N, K, rank, compute)) return small_bwd_ws(M, N, K, rank);
  return a256(sizeof(float) * static_cast<size_t>(M) * rank) + tc_bwd_ws_bytes(M, N, K, rank, true);
}

nf4_status qlora_linear_fwd_w16(int64_t M, int64_t N, int64_t K, int32_t rank, float alpha,
                                qlora_scale_mode mode, nf4_dtype compute,
                                const void* x, const void* w16, const float* A, const float* B,
                                void* y, float* T_out, void* ws, size_t ws_bytes, void* stream) {
  float s = 0.0f;
  nf4_status st = check_linear(M, N, K, rank, alpha, mode, compute, &s);
  if (st != NF4_OK) return st;
  if (!is16(compute)) return NF4_ERR_DTYPE;
  if (w16 == nullptr || A == nullptr || B == nullptr) return NF4_ERR_ARG;
  if (M > 0 && (x == nullptr || y == nullptr || T_out == nullptr)) return NF4_ERR_ARG;
  if (!aligned16(w16) || !aligned16(A) || !aligned16(B) ||
      (M > 0 && (!aligned16(x) || !aligned16(y) || !aligned16(T_out))))
    return NF4_ERR_ALIGN;
  const size_t need = qlora_fwd_w16_workspace_bytes(M, N, K, rank, compute);
  if (need > 0 && (ws == nullptr || ws_bytes < need)) return NF4_ERR_WORKSPACE;
  if (need > 0 && !aligned16(ws)) return NF4_ERR_ALIGN;
  if (M == 0) return NF4_OK;
  const LinearArgs a{M, N, K, rank, s, Nf4View{}};
  if (small_w(M, N, K, rank, compute)) {
    SmallItem it{};
    it.a = a;
    it.x = x, it.A = A, it.B = B, it.y = y, it.T = T_out, it.w16 = w16;
    return from_cuda(small_fused_forward(&it, 1, M, compute == NF4_F16, static_cast<cudaStream_t>(stream)));
  }
  int* status = nullptr;
  if ((st = device_status_ptr(&status)) != NF4_OK) return st;
  return from_cuda(tc_forward(a, compute == NF4_F16, x, A, B, y, T_out, ws, status,
                              static_cast<cudaStream_t>(stream), w16));
}

nf4_status qlora_linear_bwd_w16(int64_t M, int64_t N, int64_t K, int32_t rank, float alpha,
                                qlora_scale_mode mode, nf4_dtype compute,
                                const void* dy, const void* x, const float* T, const void* w16,
                                const float* A, const float* B, void* dx, float* dA, float* dB,
                                void* ws, size_t ws_bytes, void* stream) {
  float s = 0.0f;
  nf4_status st = check_linear(M, N, K, rank, alpha, mode, compute, &s);
  if (st != NF4_OK) return st;
  if (!is16(compute)) return NF4_ERR_DTYPE;
  if (w16 == nullptr || A == nullptr || B == nullptr || dA == nullptr || dB == nullptr) return NF4_ERR_ARG;
  if (M > 0 && (dy == nullptr || x == nullptr || T == nullptr || dx == nullptr)) return NF4_ERR_ARG;
  if (!aligned16(w16) || !aligned16(A) || !aligned16(B) || !aligned16(dA) || !aligned16(dB)) return NF4_ERR_ALIGN;
  if (M > 0 && (!aligned16(dy) || !aligned16(x) || !aligned16(T) || !aligned16(dx))) return NF4_ERR_ALIGN;
  const size_t need = qlora_bwd_w16_workspace_bytes(M, N, K, rank, compute);
  if (ws == nullptr || ws_bytes < need) return NF4_ERR_WORKSPACE;
  if (!aligned16(ws)) return NF4_ERR_ALIGN;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  if (M == 0) {   // no tokens: the adapter gradients are zero
    cudaError_t e = cudaMemsetAsync(dA, 0, sizeof(float) * static_cast<size_t>(rank) * K, cs);
    if (e == cudaSuccess) e = cudaMemsetAsync(dB, 0, sizeof(float) * static_cast<size_t>(N) * rank, cs);
    return from_cuda(e);
  }
  const LinearArgs a{M, N, K, rank, s, Nf4View{}};
  if (small_w(M, N, K, rank, compute)) {
    SmallItem it{};
    it.a = a;
    it.x = x, it.A = A, it.B = B, it.T = const_cast<float*>(T), it.dy = dy, it.dx = dx, it.dA = dA, it.dB = dB;
    it.w16 = w16;
    return from_cuda(small_fused_backward(&it, 1, M, compute == NF4_F16, ws, cs));
  }
  int* status = nullptr;
  if ((st = device_status_ptr(&status)) != NF4_OK) return st;
  float* G = static_cast<float*>(ws);
  void* tc_ws = static_cast<char*>(ws) + a256(sizeof(float) * static_cast<size_t>(M) * rank);
  return from_cuda(tc_backward(a, compute == NF4_F16, dy, x, T, A, B, dx, dA, dB, G, tc_ws, status, cs, w16));
}

size_t qlora_bwd_batch_workspace_bytes(int64_t M, int32_t count, const qlora_bwd_item* items, nf4_dtype compute) {
  if (M < 0 || count < 1 || items == nullptr) return 0;
  for (int32_t i = 0; i < count; ++i)
    if (items[i].N <= 0 || items[i].K <= 0 || items[i].rank < 1 || items[i].rank > 256) return 0;
  size_t need = 0;
  for (const BatchRun& r : plan_bwd(M, count, items, compute)) {
    const int n = static_cast<int>(r.idx.size());
    if (r.kind == kRunSmall) {
      SmallItem small[kSmallMaxGroup];
      for (int k = 0; k < n; ++k) {
        const qlora_bwd_item& it = items[r.idx[k]];
        small[k] = SmallItem{};
        small[k].a = LinearArgs{M, it.N, it.K, it.rank, 0.0f, Nf4View{}};
      }
      need = std::max(need, small_fused_bwd_ws_bytes(small, n, M));
    } else if (r.kind == kRunGroup && n > 1) {
      TcBwdItem t[kTcGroupMax];
      for (int k = 0; k < n; ++k) t[k] = tc_bwd_item(M, items[r.idx[k]], 0.0f, false);
      need = std::max(need, tc_bwd_run_ws_bytes(t, n));
    } else {
      const qlora_bwd_item& it = items[r.idx[0]];
      need = std::max(need, it.w16 != nullptr ? qlora_bwd_w16_workspace_bytes(M, it.N, it.K, it.rank, compute)
                                              : bwd_ws(M, it.N, it.K, it.rank, compute));
    }
  }
  return need;
}

nf4_status qlora_linear_bwd_batch(int64_t M, int32_t count, const qlora_bwd_item* items, nf4_dtype compute,
                                  void* ws, size_t ws_bytes, void* stream) {
  if (count < 1 || items == nullptr) return NF4_ERR_ARG;
  std::vector<float> s(static_cast<size_t>(count));
  for (int32_t i = 0; i < count; ++i) {   // the single calls' checks, before anything is enqueued
    const qlora_bwd_item& it = items[i];
    nf4_status st = check_linear(M, it.N, it.K, it.rank, it.alpha, it.mode, compute, &s[i]);
    if (st != NF4_OK) return st;
    if (it.w16 != nullptr) {
      if (!is16(compute)) return NF4_ERR_DTYPE;
      if (!aligned16(it.w16)) return NF4_ERR_ALIGN;
    } else if ((st = check_tensor(it.W, it.N * it.K)) != NF4_OK) {
      return st;
    }
    if (it.A == nullptr || it.B == nullptr || it.dA == nullptr || it.dB == nullptr) return NF4_ERR_ARG;
    if (M > 0 && (it.dy == nullptr || it.x == nullptr || it.T == nullptr || it.dx == nullptr)) return NF4_ERR_ARG;
    if (!aligned16(it.A) || !aligned16(it.B) || !aligned16(it.dA) || !aligned16(it.dB)) return NF4_ERR_ALIGN;
    if (M > 0 && (!aligned16(it.dy) || !aligned16(it.x) || !aligned16(it.T) || !aligned16(it.dx))) return NF4_ERR_ALIGN;
  }
  const size_t need = qlora_bwd_batch_workspace_bytes(M, count, items, compute);
  if (ws == nullptr || ws_bytes < need) return NF4_ERR_WORKSPACE;
  if (!aligned16(ws)) return NF4_ERR_ALIGN;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  const bool f16 = compute == NF4_F16;
  int* status = nullptr;
  for (const BatchRun& r : plan_bwd(M, count, items, compute)) {
    const int n = static_cast<int>(r.idx.size());
    const int i0 = r.idx[0];
    cudaError_t e = cudaSuccess;
    if (r.kind == kRunSmall) {
      SmallItem small[kSmallMaxGroup];
      for (int k = 0; k < n; ++k) {
        const qlora_bwd_item& it = items[r.idx[k]];
        SmallItem& si = small[k];
        si = SmallItem{};
        si.a = LinearArgs{M, it.N, it.K, it.rank, s[r.idx[k]], it.w16 != nullptr ? Nf4View{} : view_of(it.W)};
        si.x = it.x, si.A = it.A, si.B = it.B, si.T = const_cast<float*>(it.T), si.dy = it.dy, si.dx = it.dx;
        si.dA = it.dA, si.dB = it.dB, si.w16 = it.w16;
      }
      e = small_fused_backward(small, n, M, f16, ws, cs);
    } else if (r.kind == kRunGroup && n > 1) {
      if (status == nullptr) {
        const nf4_status st = device_status_ptr(&status);
        if (st != NF4_OK) return st;
      }
      TcBwdItem t[kTcGroupMax];
      for (int k = 0; k < n; ++k) t[k] = tc_bwd_item(M, items[r.idx[k]], s[r.idx[k]]);
      e = tc_backward_run(t, n, f16, ws, status, cs);
    } else {
      const qlora_bwd_item& it = items[i0];
      const nf4_status st =
          it.w16 != nullptr
              ? qlora_linear_bwd_w16(M, it.N, it.K, it.rank, it.alpha, it.mode, compute, it.dy, it.x, it.T, it.w16,
                                     it.A, it.B, it.dx, it.dA, it.dB, ws, ws_bytes, stream)
              : qlora_linear_bwd(M, it.N, it.K, it.rank, it.alpha, it.mode, compute, it.dy, it.x, it.T, it.W, it.A,
                                 it.B, it.dx, it.dA, it.dB, ws, ws_bytes, stream);
      if (st != NF4_OK) return st;
    }
    if (e != cudaSuccess) return NF4_ERR_CUDA;
  }
  return NF4_OK;
}

nf4_status qlora_last_device_status(void* stream, int32_t clear) {
  int* p = nullptr;
  nf4_status st = device_status_ptr(&p);
  if (st != NF4_OK) return st;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(cs) != cudaSuccess) return NF4_ERR_CUDA;
  int v = 0;
  if (cudaMemcpy(&v, p, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return NF4_ERR_CUDA;
  if (clear && v != 0) {
    const int zero = 0;
    if (cudaMemcpy(p, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess) return NF4_ERR_CUDA;
  }
  return static_cast<nf4_status>(v);
}

int64_t nf4_kernel_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

void qlora_debug_wait_timeout(int32_t on) { g_wait_fault.store(on != 0 ? 1 : 0); }

void nf4_timing_enable(int32_t on) { timing().enabled.store(on != 0); }

nf4_status nf4_timing_read(int32_t kind, double* total_ms, int64_t* launches, int32_t reset) {
  if (kind < 0 || kind >= NF4_TIME_KINDS) return NF4_ERR_ARG;
  TimingState& t = timing();
  std::lock_guard<std::mutex> lock(t.mu);
  nf4_status st = NF4_OK;
  for (auto& pr : t.pending[kind]) {
    float ms = 0.0f;
    if (cudaEventSynchronize(pr.second) != cudaSuccess ||
        cudaEventElapsedTime(&ms, pr.first, pr.second) != cudaSuccess) {
      st = NF4_ERR_CUDA;
    } else {
      t.total_ms[kind] += ms;
      t.count[kind] += 1;
    }
    t.pool.push_back(pr.first);
    t.pool.push_back(pr.second);
  }
  t.pending[kind].clear();
  if (total_ms) *total_ms = t.total_ms[kind];
  if (launches) *launches = t.count[kind];
  if (reset) {
    t.total_ms[kind] = 0.0;
    t.count[kind] = 0;
  }
  return st;
}

}  // extern "C"
