// Adapter-side contractions of the bf16 QLoRA linear on tcgen05:
//   T = x A^T,  G = dY B,  dB = s dY^T T,  dA = s G^T x
// ("Native model adaptation and NF4", "Mixed precision keeps stable state in FP32":
// adapter contractions accumulate in FP32; "Packed NF4 ...": no base-weight gradient).
//
// Each is a skinny product Out[rows, r] = X[rows, red] . Q[red, r] with a large bf16
// activation X (x or dY, read once, HBM-bound) and a small bf16 Q (the rank-r side).
// Kernel adapter_tc: one 128-row tile of Out per CTA and one slice of the reduction;
// X arrives by TMA as the MMA's A operand (K-major when the reduction runs along the
// activation's rows, MN-major when it runs down its columns), Q as the B operand
// (K-major, N = r rounded up to 16); the fp32 accumulator lives in TMEM.  Slices
// write partial sums that a second kernel adds in a fixed order (deterministic,
// no atomics) and scales.
#include <algorithm>
#include <mutex>

#include <cuda_fp16.h>

#include "linear_tc.cuh"
#include "tc_ptx.cuh"

namespace qnf4 {
namespace {

using namespace tc;

constexpr int kRowsT = 128;          // MMA M
constexpr int kBKa = 64;             // reduction per box
constexpr int kBoxes = 2;            // boxes per stage: 8 MMAs per commit
constexpr int kAThreads = 192;       // warp 0 TMA, warp 1 MMA + TMEM, warps 2..5 epilogue
constexpr int kATileBytes = kRowsT * kBKa * 2;
constexpr int kTargetCtas = 320;     // fixed, so workspace sizes do not depend on the device
constexpr int kMaxSplit = 64;

struct SkinnyParams {
  int64_t rows;     // rows of Out
  int tiles;        // ceil(rows / 128)
  int total_steps;  // ceil(red / 128): stages of the whole reduction
  int sps;          // steps per slice
  int a_mn_major;
  int n_mma;        // r rounded up to 16
  int r;
  int stages;
  uint32_t b_bytes; // n_mma * 128
  uint32_t stage_bytes;
  float* partial;   // [nsplit][rows][r]
  int* status;
  int ctas;         // tiles * nsplit: this pass's CTAs
  int f16;          // operands are IEEE half (else bf16)
};

// One launch runs up to kAdapterMaxPasses independent passes: CTAs [cta0[k], cta0[k + 1])
// take pass k.
struct AdapterLaunch {
  CUtensorMap tx[kAdapterMaxPasses];
  CUtensorMap tq[kAdapterMaxPasses];
  SkinnyParams p[kAdapterMaxPasses];
  int cta0[kAdapterMaxPasses + 1];
  int n;
};

__global__ void __launch_bounds__(kAThreads, 1)
adapter_tc(const __grid_constant__ AdapterLaunch L) {
  int k = 0;
  while (k + 1 < L.n && static_cast<int>(blockIdx.x) >= L.cta0[k + 1]) ++k;
  const SkinnyParams p = L.p[k];
  const CUtensorMap& tm_x = L.tx[k];
  const CUtensorMap& tm_q = L.tq[k];
  const int bid = static_cast<int>(blockIdx.x) - L.cta0[k];
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* base_ptr = smem_raw + (base - raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(base_ptr + p.stages * p.stage_bytes);
  // bars: full[stages], empty[stages], accfull
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 2 * p.stages + 1);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * p.stages + 1) + 1;
  auto bar = [&](int i) { return smem_u32(bars + i); };
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  uint32_t tmem_cols = 32;
  while (tmem_cols < static_cast<uint32_t>(p.n_mma)) tmem_cols <<= 1;

  const int tile = bid % p.tiles;
  const int slice = bid / p.tiles;
  const int k_begin = slice * p.sps;
  const int k_end = min(p.total_steps, k_begin + p.sps);
  const int nsteps = k_end - k_begin;

  if (threadIdx.x == 0) {
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(bar(s), 1);
      mbar_init(bar(p.stages + s), 1);
    }
    mbar_init(bar(2 * p.stages), 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  pdl_allow_next();
  pdl_wait();   // TMEM only after the preceding grid has completed (no hold-and-wait on TMEM)
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(tmem_cols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      // one stage = kBoxes boxes of 64 along the reduction; cursors instead of divisions
      bool ok = true;
      int s = 0, issued = 0;
      uint32_t ph = 0;
      for (int i = 0; i < nsteps; ++i) {
        if (!mbar_wait(bar(p.stages + s), ph ^ 1u, abort_flag, p.status)) { ok = false; break; }
        const uint32_t a_dst = base + s * p.stage_bytes;
        const uint32_t b_dst = a_dst + kBoxes * kATileBytes;
        mbar_expect_tx(bar(s), kBoxes * (kATileBytes + p.b_bytes));
#pragma unroll
        for (int h = 0; h < kBoxes; ++h) {
          const int k0 = ((k_begin + i) * kBoxes + h) * kBKa;
          const uint32_t ad = a_dst + h * kATileBytes;
          if (p.a_mn_major) {
            // activation [red rows, rows cols]: two 64-column boxes of 64 reduction rows
            tma_load_2d(ad, &tm_x, bar(s), tile * kRowsT, k0);
            tma_load_2d(ad + kATileBytes / 2, &tm_x, bar(s), tile * kRowsT + 64, k0);
          } else {
            tma_load_2d(ad, &tm_x, bar(s), k0, tile * kRowsT);
          }
          tma_load_2d(b_dst + h * p.b_bytes, &tm_q, bar(s), k0, 0);
        }
        ++issued;
        if (++s == p.stages) s = 0, ph ^= 1u;
      }
      if (!ok) {   // let the copies in flight land before the CTA exits
        for (int q = 0; q < issued && q < p.stages; ++q) {
          if (s == 0) s = p.stages - 1, ph ^= 1u;
          else --s;
          mbar_drain(bar(s), ph);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc = idesc_16(kRowsT, p.n_mma, p.a_mn_major ? 1u : 0u, p.f16 ? 1u : 0u);
      bool ok = true;
      int s = 0;
      uint32_t ph = 0;
      for (int i = 0; i < nsteps; ++i) {
        if (!mbar_wait(bar(s), ph, abort_flag, p.status)) { ok = false; break; }
        tc_fence_after();
        const uint32_t a_s = base + s * p.stage_bytes;
        const uint32_t b_s = a_s + kBoxes * kATileBytes;
#pragma unroll
        for (int h = 0; h < kBoxes; ++h) {
#pragma unroll
          for (int kk = 0; kk < kBKa / 16; ++kk) {
            const uint32_t ah = a_s + h * kATileBytes;
            const uint64_t adesc = p.a_mn_major ? smem_desc(ah + kk * 2048, 8192, 1024)
                                                : smem_desc(ah + kk * 32, 16, 1024);
            const uint64_t bdesc = smem_desc(b_s + h * p.b_bytes + kk * 32, 16, 1024);
            umma_bf16(tmem_base, adesc, bdesc, idesc, (i > 0 || h > 0 || kk > 0) ? 1u : 0u);
          }
        }
        umma_commit(bar(p.stages + s));
        if (++s == p.stages) s = 0, ph ^= 1u;
      }
      if (ok && nsteps > 0) umma_commit(bar(2 * p.stages));
    }
  } else {
    const int quarter = warp & 3;
    const int64_t row = static_cast<int64_t>(tile) * kRowsT + quarter * 32 + lane;
    const bool have = nsteps > 0 && __all_sync(0xffffffffu, mbar_wait(bar(2 * p.stages), 0, abort_flag, p.status));
    if (have) {
      tc_fence_after();
      float* dst = p.partial + (static_cast<int64_t>(slice) * p.rows + row) * p.r;
      for (int c0 = 0; c0 < p.n_mma; c0 += 16) {
        uint32_t v[16];
        tmem_ld16(tmem_base + c0 + (static_cast<uint32_t>(quarter * 32) << 16), v);
        tmem_ld_wait();
        if (row < p.rows) {
#pragma unroll
          for (int j = 0; j < 16; ++j)
            if (c0 + j < p.r) dst[c0 + j] = __uint_as_float(v[j]);
        }
      }
    } else if (nsteps == 0 && row < p.rows) {
      float* dst = p.partial + (static_cast<int64_t>(slice) * p.rows + row) * p.r;
      for (int j = 0; j < p.r; ++j) dst[j] = 0.0f;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(tmem_cols)
                 : "memory");
  }
}

// out = scale * sum over slices (fixed order), for up to kAdapterMaxOuts consumers of one or
// two passes in one launch; a consumer takes columns [col0, col0 + r) of its pass's sums
// (partial rows of pstride floats).  Optional outputs: f32 [rows][r] (or transposed
// [r][rows] when f32_t), T16(scale_b * v) [rows][rp] zero-padded, T16(v) transposed
// [nq][ldt] (entries past rows / r must already be zero); T16 is IEEE half when f16, else
// bf16.
struct FinishJob {
  const float* partial;
  int nsplit;
  int64_t rows;
  int col0, pstride;
  int r;
  float scale;
  float* f32;
  int f32_t;
  void* b_rows;
  int rp;
  float scale_b;
  void* b_t;
  int64_t ldt;
  unsigned first_block;
  int f16;
};

__device__ __forceinline__ void put16(void* base, int64_t i, float v, int f16) {
  if (f16) static_cast<__half*>(base)[i] = __float2half_rn(v);
  else static_cast<__nv_bfloat16*>(base)[i] = __float2bfloat16_rn(v);
}
struct FinishJobs {
  FinishJob job[kAdapterMaxOuts];
  int n;
};

// One thread per 4 consecutive columns of a row: the sums of its columns below r (the slices
// in order), and for b_rows the 4 16-bit values (zeros past r) as one 8-byte store.
__global__ void finish_partials(const FinishJobs jobs) {
  pdl_allow_next();
  pdl_wait();
  int k = 0;
  while (k + 1 < jobs.n && blockIdx.x >= jobs.job[k + 1].first_block) ++k;
  const FinishJob& f = jobs.job[k];
  const int64_t i = static_cast<int64_t>(blockIdx.x - f.first_block) * blockDim.x + threadIdx.x;
  const int chunks = ((f.b_rows ? f.rp : f.r) + 3) / 4;
  if (i >= f.rows * chunks) return;
  const int64_t row = i / chunks;
  const int j0 = static_cast<int>(i - row * chunks) * 4;
  const int nj = min(4, f.r - j0);   // columns of this chunk below r (none in the padding)
  float v[4];
#pragma unroll
  for (int u = 0; u < 4; ++u) v[u] = 0.0f;
  if (nj > 0) {
    const float* src = f.partial + row * f.pstride + f.col0 + j0;
    const int64_t stride = f.rows * f.pstride;
#pragma unroll 4
    for (int sp = 0; sp < f.nsplit; ++sp) {
      float t[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) t[u] = u < nj ? src[sp * stride + u] : 0.0f;
#pragma unroll
      for (int u = 0; u < 4; ++u) v[u] += t[u];
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      if (u >= nj) break;
      const int j = j0 + u;
      if (f.f32) {
        if (f.f32_t) f.f32[static_cast<int64_t>(j) * f.rows + row] = f.scale * v[u];
        else f.f32[row * f.r + j] = f.scale * v[u];
      }
      if (f.b_t) put16(f.b_t, static_cast<int64_t>(j) * f.ldt + row, v[u], f.f16);
    }
  }
  if (f.b_rows) {   // rp is a multiple of 64: the 4 values are one aligned 8-byte store
    uint32_t w[2];
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const float lo = 2 * q < nj ? f.scale_b * v[2 * q] : 0.0f;
      const float hi = 2 * q + 1 < nj ? f.scale_b * v[2 * q + 1] : 0.0f;
      if (f.f16) {
        const __half2 h = __floats2half2_rn(lo, hi);
        w[q] = *reinterpret_cast<const uint32_t*>(&h);
      } else {
        const __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
        w[q] = *reinterpret_cast<const uint32_t*>(&b);
      }
    }
    *reinterpret_cast<uint2*>(static_cast<uint16_t*>(f.b_rows) + row * f.rp + j0) = make_uint2(w[0], w[1]);
  }
}

int nq_of(int r) { return (r + 15) / 16 * 16; }
size_t al(size_t b) { return (b + 1023) & ~static_cast<size_t>(1023); }
unsigned blocks(int64_t n) { return static_cast<unsigned>((n + 255) / 256); }

struct Plan {
  int tiles, total_steps, sps, nsplit;
};

// Slices per row tile: as many as keep tiles * slices within `target` resident CTAs
// (two per SM fit); workspace is sized with the largest target any device uses.
Plan plan(int64_t rows, int64_t red, int target = kTargetCtas) {
  Plan pl;
  pl.tiles = static_cast<int>((rows + kRowsT - 1) / kRowsT);
  pl.total_steps = static_cast<int>((red + kBoxes * kBKa - 1) / (kBoxes * kBKa));
  int ns = target / pl.tiles;
  if (ns > kMaxSplit) ns = kMaxSplit;
  if (ns > pl.total_steps) ns = pl.total_steps;
  if (ns < 1) ns = 1;
  pl.sps = (pl.total_steps + ns - 1) / ns;
  pl.nsplit = (pl.total_steps + pl.sps - 1) / pl.sps;
  return pl;
}

int resident_ctas() {
  static int n = 0;
  if (n == 0) {
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    n = sms > 0 ? 2 * sms : 2;
    if (n > kTargetCtas) n = kTargetCtas;
  }
  return n;
}

size_t partial_bytes(int64_t rows, int64_t red, int r) {
  const Plan pl = plan(rows, red);
  return al(sizeof(float) * static_cast<size_t>(pl.nsplit) * rows * r);
}

// Parameters and tensor maps of one pass with `target` CTAs.
bool setup_pass(const AdapterPassArgs& a, int target, int* status, SkinnyParams* p, CUtensorMap* tx, CUtensorMap* tq) {
  const Plan pl = plan(a.rows, a.red, target);
  const int nq = nq_of(a.r);
  const CUtensorMapDataType dt = a.f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  bool ok = a.mn_major ? make_map(tx, dt, a.X, a.x_inner, a.x_outer, 2 * a.x_inner, 64, 64, CU_TENSOR_MAP_SWIZZLE_128B)
                       : make_map(tx, dt, a.X, a.x_inner, a.x_outer, 2 * a.x_inner, 64, kRowsT, CU_TENSOR_MAP_SWIZZLE_128B);
  ok = ok && make_map(tq, dt, a.Q, a.q_cols, nq, 2 * a.q_cols, 64, nq, CU_TENSOR_MAP_SWIZZLE_128B);
  *p = SkinnyParams{};
  p->rows = a.rows;
  p->tiles = pl.tiles;
  p->total_steps = pl.total_steps;
  p->sps = pl.sps;
  p->a_mn_major = a.mn_major ? 1 : 0;
  p->n_mma = nq;
  p->r = a.r;
  p->b_bytes = static_cast<uint32_t>(nq * 128);
  p->stage_bytes = static_cast<uint32_t>(al(kBoxes * (kATileBytes + p->b_bytes)));
  p->stages = nq <= 32 ? 3 : 2;
  p->partial = a.partial;
  p->status = status;
  p->ctas = pl.tiles * pl.nsplit;
  p->f16 = a.f16;
  return ok;
}

// The finish of consumer `o` of a pass (o < 0: the pass's own output fields, all columns).
FinishJob finish_job(const AdapterPassArgs& a, const SkinnyParams& p, int o) {
  FinishJob f{};
  f.partial = a.partial;
  f.nsplit = p.ctas / p.tiles;
  f.rows = a.rows;
  f.pstride = a.r;
  f.f16 = a.f16;
  if (o < 0) {
    f.col0 = 0;
    f.r = a.r;
    f.scale = a.scale;
    f.f32 = a.f32;
    f.f32_t = a.f32_t;
    f.b_rows = a.b_rows;
    f.rp = a.rp;
    f.scale_b = a.scale_b;
    f.b_t = a.b_t;
    f.ldt = a.ldt;
  } else {
    const AdapterOut& c = a.outs[o];
    f.col0 = c.col0;
    f.r = c.r;
    f.scale = c.scale;
    f.f32 = c.f32;
    f.f32_t = c.f32_t;
    f.b_rows = c.b_rows;
    f.rp = c.rp;
    f.scale_b = c.scale_b;
    f.b_t = c.b_t;
    f.ldt = c.ldt;
  }
  return f;
}

}  // namespace

int adapter_nq(int r) { return nq_of(r); }

int adapter_total_ctas() { return resident_ctas(); }

void adapter_pair_targets(int64_t rows0, int64_t red0, int64_t rows1, int64_t red1, int* t0, int* t1) {
  const int total = resident_ctas();
  const double b0 = static_cast<double>(rows0) * red0, b1 = static_cast<double>(rows1) * red1;
  *t0 = std::max(1, static_cast<int>(total * b0 / (b0 + b1)));
  *t1 = std::max(1, total - *t0);
}

size_t adapter_partial_bytes(int64_t rows, int64_t red, int r) { return partial_bytes(rows, red, r); }

cudaError_t adapter_run(const AdapterPassArgs* a, int n, int* status, cudaStream_t st) {
  KernelTimer timer(NF4_TIME_ADAPTER, st);
  if (n < 1 || n > kAdapterMaxPasses) return cudaErrorInvalidValue;
  int outs = 0;
  for (int i = 0; i < n; ++i) {
    if (a[i].nouts < 0 || (a[i].nouts > 0 && a[i].outs == nullptr)) return cudaErrorInvalidValue;
    outs += a[i].nouts > 0 ? a[i].nouts : 1;
    for (int o = 0; o < a[i].nouts; ++o)
      if (a[i].outs[o].col0 < 0 || a[i].outs[o].r < 1 || a[i].outs[o].col0 + a[i].outs[o].r > a[i].r)
        return cudaErrorInvalidValue;
  }
  if (outs > kAdapterMaxOuts) return cudaErrorInvalidValue;
  // each pass's reduction split: its own target if given; otherwise one pass takes every
  // resident CTA and two share them in proportion to the activation bytes each reads
  const int total = resident_ctas();
  int target[kAdapterMaxPasses];
  for (int i = 0; i < n; ++i) target[i] = a[i].target > 0 ? std::min(a[i].target, total) : total;
  if (n == 2 && a[0].target <= 0 && a[1].target <= 0)
    adapter_pair_targets(a[0].rows, a[0].red, a[1].rows, a[1].red, &target[0], &target[1]);
  AdapterLaunch L{};
  L.n = n;
  int ctas = 0, smem = 0;
  for (int i = 0; i < n; ++i) {
    if (!setup_pass(a[i], target[i], status, &L.p[i], &L.tx[i], &L.tq[i])) return cudaErrorInvalidValue;
    L.cta0[i] = ctas;
    ctas += L.p[i].ctas;
    smem = std::max(smem, 1024 + L.p[i].stages * static_cast<int>(L.p[i].stage_bytes) + 256);
  }
  L.cta0[n] = ctas;
  static std::once_flag once;
  static cudaError_t attr = cudaSuccess;
  std::call_once(once, [] {
    attr = cudaFuncSetAttribute(adapter_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, 1024 + 4 * 49152 + 256);
  });
  if (attr != cudaSuccess) return attr;
  cudaError_t e = launch_pdl(adapter_tc, dim3(ctas), dim3(kAThreads), static_cast<size_t>(smem), st, 1, L);
  note_launch();
  if (e != cudaSuccess) return e;
  FinishJobs jobs{};
  unsigned nblocks = 0;
  for (int i = 0; i < n; ++i) {
    for (int o = a[i].nouts > 0 ? 0 : -1; o < a[i].nouts; ++o) {
      FinishJob& f = jobs.job[jobs.n++];
      f = finish_job(a[i], L.p[i], o);
      f.first_block = nblocks;
      nblocks += blocks(f.rows * (((f.b_rows ? f.rp : f.r) + 3) / 4));
    }
  }
  e = launch_pdl(finish_partials, dim3(nblocks), dim3(256), 0, st, 1, jobs);
  note_launch();
  return e;
}

}  // namespace qnf4
