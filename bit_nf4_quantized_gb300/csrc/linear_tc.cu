// bf16 profile of the QLoRA linear on the 5th-generation tensor cores (tcgen05).
//
// Math ("Native model adaptation and NF4", sections "One model contract", "Packed
// NF4 and the portable QLoRA profile", "Fused GPU NF4 decodes inside the matrix
// kernel"): y = x W^T + s T B^T and dX = dY W + s G A, with W decoded from NF4 on
// the device and never written to global memory.
//
// Kernel nf4_tc_gemm (one CTA per SM, persistent over output tiles):
//   D[f, t] (TMEM, fp32) = sum_c Wdec[f, c] * Tok[t, c]  +  sum_j Slab_A[f, j] * Slab_B[t, j]
// with f = 128 output features per tile (the MMA's M), t = 256 tokens (the MMA's N):
//   forward: f = rows of W (output features), c = k, Tok = x,  slab (B, s*T)
//   dX:      f = columns of W (input features), c = n, Tok = dY, slab (A^T, s*G)
// Warp roles (480 threads):
//   warp 0      TMA producer: token tile (128B-swizzled) + packed NF4 tile per stage,
//               or the two adapter slab tiles for the last (rank / 64) stages;
//   warp 1      TMEM allocation; lane 0 issues tcgen05.mma and tcgen05.commit;
//   warps 2..9  decoders in two groups of four that take alternate stages; a thread
//               turns one 64-element NF4 block (one 128-byte row of the A tile) into
//               bf16 in the swizzled layout the MMA reads (K-major for the forward,
//               MN-major for dX), through a per-block scaled lookup table;
//   warps 10..13 epilogue: tcgen05.ld of the accumulator, bf16 stores.
// The per-block scales a' = dyn8[code] * nested + offset are computed once per call
// (prep.cu) into an fp32 [N][K/64 rounded up to 4] array and reach each stage by TMA
// next to the packed codes, so the decoders never wait on global memory.
// Two accumulators of 256 columns let the epilogue of one tile overlap the
// main loop of the next.  Every mbarrier wait is bounded in time; a wait that
// gives up sets NF4_ERR_TIMEOUT in the status word and the CTA winds down,
// freeing its TMEM.
#include <algorithm>

#include "linear_tc.cuh"
#include "decode.cuh"
#include "prep.cuh"
#include "tc_ptx.cuh"

namespace qnf4 {
namespace {

using namespace tc;

constexpr int kTileF = 128;                 // MMA M
constexpr int kTileT = 256;                 // MMA N
constexpr int kBK = 64;                     // contraction per stage (128 bytes of bf16)
constexpr int kStages = 4;
constexpr int kABytes = kTileF * kBK * 2;   // 16384
constexpr int kBBytes = kTileT * kBK * 2;   // 32768
constexpr int kPBytes = 4096;               // packed NF4 bytes per stage
constexpr int kStageBytes = kABytes + kBBytes + kPBytes;
constexpr int kThreads = 448;                // 14 warps, roles below
constexpr int kTmemCols = 512;
constexpr int kScaleSlot = 2048;              // fwd: 128 rows x 4 fp32; dX: 64 rows x 4 fp32
constexpr int kSmemBytes = 1024 + kStages * kStageBytes + kStages * kScaleSlot + 256;
static_assert(20 * 8 + 8 <= 256, "barrier block");

static_assert(kStageBytes % 1024 == 0, "stage buffers must stay 1024-byte aligned");
static_assert(kStages % 2 == 0, "the two decoder groups alternate stages");

struct GemmParams {
  int64_t M;           // tokens
  int64_t F;           // output features (N forward, K for dX)
  int64_t N, K;        // W is [N, K]
  int mode;            // 0 forward, 1 dX
  int red_steps;       // ceil(contraction / 64)
  int slab_steps;      // padded rank / 64
  int tiles_t, tiles_f;
  int f_fast;          // tile order: 1 = feature tiles vary fastest (dX), 0 = token tiles (forward)
  const void* absmax;  // uint8 codes (dq) or float
  const float* nested;
  const float* offset;
  int dq;
  __nv_bfloat16* out;  // [M, F]
  int* status;
};

// Warp roles:
//   0       TMA producer (lane 0)
//   1       TMEM allocation; MMA issue (lane 0)
//   2..9    decoders: warps 2..5 take the even stages, 6..9 the odd ones; thread =
//           one 128-byte row of the A tile (one 64-element NF4 block)
//   10..13  epilogue
__global__ void __launch_bounds__(kThreads, 1)
nf4_tc_gemm(const __grid_constant__ CUtensorMap tm_tok, const __grid_constant__ CUtensorMap tm_packed,
            const __grid_constant__ CUtensorMap tm_slab_f, const __grid_constant__ CUtensorMap tm_slab_t,
            const __grid_constant__ CUtensorMap tm_scale, const GemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* base_ptr = smem_raw + (base - raw);
  const float* scales = reinterpret_cast<const float*>(base_ptr + kStages * kStageBytes);
  uint64_t* bars = reinterpret_cast<uint64_t*>(base_ptr + kStages * kStageBytes + kStages * kScaleSlot);
  // bars: full_b[4] aready[4] empty[4] accfull[2] accempty[2] full_p[4]
  //   full_b: token tile (or both slab tiles) landed; full_p: packed codes + scales landed
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 20);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 20) + 1;
  auto bar = [&](int i) { return smem_u32(bars + i); };
  auto stage_a = [&](int s) { return base + s * kStageBytes; };
  auto stage_b = [&](int s) { return base + s * kStageBytes + kABytes; };
  auto stage_p = [&](int s) { return base + s * kStageBytes + kABytes + kBBytes; };
  auto stage_s = [&](int s) { return base + kStages * kStageBytes + s * kScaleSlot; };
  auto tile_t = [&](int64_t tile) { return p.f_fast ? tile / p.tiles_f : tile % p.tiles_t; };
  auto tile_f = [&](int64_t tile) { return p.f_fast ? tile % p.tiles_f : tile / p.tiles_t; };

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar(s), 1);                 // full_b: producer arrive + TMA bytes
      mbar_init(bar(16 + s), 1);            // full_p: producer arrive (+ TMA bytes on decode steps)
      mbar_init(bar(4 + s), 4);             // aready: the four warps of one decoder group
      mbar_init(bar(8 + s), 1);             // empty: tcgen05.commit
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(12 + b), 1);            // accfull: tcgen05.commit
      mbar_init(bar(14 + b), 4);            // accempty: one arrive per epilogue warp
    }
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  const int64_t total_tiles = static_cast<int64_t>(p.tiles_t) * p.tiles_f;
  const int steps = p.red_steps + p.slab_steps;
  const int64_t my_tiles =
      blockIdx.x < total_tiles ? (total_tiles - blockIdx.x + gridDim.x - 1) / gridDim.x : 0;
  const int64_t total_it = my_tiles * steps;    // every role walks the same step sequence

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      int last_phase[kStages];
      bool issued[kStages];
      for (int s = 0; s < kStages; ++s) issued[s] = false, last_phase[s] = 0;
      bool ok = true;
      for (int64_t it = 0; it < total_it; ++it) {
        const int64_t tile = blockIdx.x + (it / steps) * gridDim.x;
        const int step = static_cast<int>(it % steps);
        const int t0 = static_cast<int>(tile_t(tile) * kTileT);
        const int f0 = static_cast<int>(tile_f(tile) * kTileF);
        const int s = static_cast<int>(it % kStages);
        const uint32_t ph = static_cast<uint32_t>(it / kStages) & 1u;
        if (!mbar_wait(bar(8 + s), ph ^ 1u, abort_flag, p.status)) { ok = false; break; }
        if (step < p.red_steps) {
          // codes and scales first: the decoders start on them while the token tile streams
          mbar_expect_tx(bar(16 + s), kPBytes + (p.mode == 0 ? kTileF * 16 : 64 * 16));
          if (p.mode == 0) {
            tma_load_2d(stage_p(s), &tm_packed, bar(16 + s), step * (kBK / 2), f0);
            tma_load_2d(stage_s(s), &tm_scale, bar(16 + s), step & ~3, f0);
          } else {
            tma_load_2d(stage_p(s), &tm_packed, bar(16 + s), f0 / 2, step * kBK);
            tma_load_2d(stage_s(s), &tm_scale, bar(16 + s), (f0 / kBlock) & ~3, step * kBK);
          }
          mbar_expect_tx(bar(s), kBBytes);
          tma_load_2d(stage_b(s), &tm_tok, bar(s), step * kBK, t0);
        } else {
          const int j = (step - p.red_steps) * kBK;
          mbar_arrive(bar(16 + s));
          mbar_expect_tx(bar(s), kBBytes + kABytes);
          tma_load_2d(stage_b(s), &tm_slab_t, bar(s), j, t0);
          tma_load_2d(stage_a(s), &tm_slab_f, bar(s), j, f0);
        }
        issued[s] = true;
        last_phase[s] = ph;
      }
      if (!ok) {  // let copies already in flight land before the CTA exits
        for (int s = 0; s < kStages; ++s)
          if (issued[s]) {
            mbar_drain(bar(s), last_phase[s]);
            mbar_drain(bar(16 + s), last_phase[s]);
          }
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      const uint32_t idesc_main = idesc_bf16(kTileF, kTileT, p.mode == 1 ? 1u : 0u);
      const uint32_t idesc_slab = idesc_bf16(kTileF, kTileT, 0u);
      bool ok = true;
      for (int64_t it = 0; it < total_it && ok; ++it) {
        const int64_t lt = it / steps;
        const int step = static_cast<int>(it % steps);
        const uint32_t b = static_cast<uint32_t>(lt) & 1u;
        if (step == 0) {
          if (!mbar_wait(bar(14 + b), (static_cast<uint32_t>(lt >> 1) & 1u) ^ 1u, abort_flag, p.status)) break;
          tc_fence_after();
        }
        const int s = static_cast<int>(it % kStages);
        const uint32_t ph = static_cast<uint32_t>(it / kStages) & 1u;
        if (!mbar_wait(bar(s), ph, abort_flag, p.status) || !mbar_wait(bar(4 + s), ph, abort_flag, p.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const bool slab = step >= p.red_steps;
        const bool mn_major = (p.mode == 1) && !slab;
        const uint32_t d_tmem = tmem_base + b * kTileT;
#pragma unroll
        for (int kk = 0; kk < kBK / 16; ++kk) {
          // K-major: 32 bytes per 16-element k step inside the 128-byte row.
          // MN-major (dX): two 8-row groups of 1024 bytes per k step; the two
          // 64-feature halves of the tile are 8192 bytes apart.
          const uint64_t adesc = mn_major ? smem_desc(stage_a(s) + kk * 2048, 8192, 1024)
                                          : smem_desc(stage_a(s) + kk * 32, 16, 1024);
          const uint64_t bdesc = smem_desc(stage_b(s) + kk * 32, 16, 1024);
          umma_bf16(d_tmem, adesc, bdesc, slab ? idesc_slab : idesc_main, (step > 0 || kk > 0) ? 1u : 0u);
        }
        umma_commit(bar(8 + s));
        if (step == steps - 1) umma_commit(bar(12 + b));
      }
    }
  } else if (warp < 10) {
    // ---------------- NF4 decoders ----------------
    const int group = (warp - 2) >> 2;
    const int row = ((warp - 2) & 3) * 32 + lane;  // row of the A tile, 0..127
    const uint32_t sw = static_cast<uint32_t>(row & 7);
    const uint32_t poff = (p.mode == 0) ? row * 32 : (row & 63) * 64 + (row >> 6) * 32;
    for (int64_t it = group; it < total_it; it += 2) {
      const int step = static_cast<int>(it % steps);
      const int s = static_cast<int>(it % kStages);
      const uint32_t ph = static_cast<uint32_t>(it / kStages) & 1u;
      if (!__all_sync(0xffffffffu, mbar_wait(bar(16 + s), ph, abort_flag, p.status))) break;
      if (step < p.red_steps) {
        uint32_t L[4], H[4];
        // forward: scale of row `row`; dX: row (row & 63) of a 64 x 4 box whose first
        // column is the 128-feature tile's first block rounded down to a multiple of 4
        const int64_t f0 = tile_f(blockIdx.x + (it / steps) * gridDim.x) * kTileF;
        const float a = (p.mode == 0) ? scales[s * (kScaleSlot / 4) + row * 4 + (step & 3)]
                                      : scales[s * (kScaleSlot / 4) + (row & 63) * 4 +
                                               static_cast<int>((f0 / kBlock) & 3) + (row >> 6)];
        build_lut(a, L, H);
        const uint8_t* src = base_ptr + (stage_p(s) - base) + poff;
        const uint4 w0 = *reinterpret_cast<const uint4*>(src);
        const uint4 w1 = *reinterpret_cast<const uint4*>(src + 16);
        const uint32_t words[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
        const uint32_t arow = stage_a(s) + row * 128;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          uint32_t o[4];
          decode8(words[i], L, H, o);
          const uint32_t dst = arow + ((static_cast<uint32_t>(i) ^ sw) << 4);
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(dst), "r"(o[0]), "r"(o[1]), "r"(o[2]),
                       "r"(o[3])
                       : "memory");
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(4 + s));
    }
  } else {
    // ---------------- epilogue ----------------
    const int quarter = warp & 3;               // TMEM lanes 32*quarter .. +31
    for (int64_t lt = 0; lt < my_tiles; ++lt) {
      const int64_t tile = blockIdx.x + lt * gridDim.x;
      const uint32_t b = static_cast<uint32_t>(lt) & 1u;
      const uint32_t aph = static_cast<uint32_t>(lt >> 1) & 1u;
      if (!__all_sync(0xffffffffu, mbar_wait(bar(12 + b), aph, abort_flag, p.status))) break;
      tc_fence_after();
      const int64_t t0 = tile_t(tile) * kTileT;
      const int64_t f = tile_f(tile) * kTileF + quarter * 32 + lane;
      const uint32_t taddr = tmem_base + b * kTileT + (static_cast<uint32_t>(quarter * 32) << 16);
#pragma unroll 1
      for (int c0 = 0; c0 < kTileT; c0 += 16) {
        uint32_t v[16];
        tmem_ld16(taddr + c0, v);
        tmem_ld_wait();
        if (f < p.F) {
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int64_t m = t0 + c0 + j;
            if (m < p.M) p.out[m * p.F + f] = __float2bfloat16_rn(__uint_as_float(v[j]));
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(14 + b));
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(kTmemCols)
                 : "memory");
  }
}

// ---- host side --------------------------------------------------------------------------

int padded_rank(int r) { return (r + kBK - 1) / kBK * kBK; }
size_t a1024(size_t b) { return (b + 1023) & ~static_cast<size_t>(1023); }

int sm_count() {
  int dev = 0, n = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n > 0 ? n : 1;
}

cudaError_t launch_gemm(const GemmParams& p, const CUtensorMap& tok, const CUtensorMap& packed,
                        const CUtensorMap& slab_f, const CUtensorMap& slab_t, const CUtensorMap& scale,
                        cudaStream_t st) {
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    attr_err = cudaFuncSetAttribute(nf4_tc_gemm, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  });
  if (attr_err != cudaSuccess) return attr_err;
  const int64_t tiles = static_cast<int64_t>(p.tiles_t) * p.tiles_f;
  const int grid = static_cast<int>(tiles < sm_count() ? tiles : sm_count());
  KernelTimer timer(p.mode == 0 ? NF4_TIME_FWD_GEMM : NF4_TIME_DX_GEMM, st);
  nf4_tc_gemm<<<grid, kThreads, kSmemBytes, st>>>(tok, packed, slab_f, slab_t, scale, p);
  note_launch();
  return cudaGetLastError();
}

int64_t scale_ld(int64_t K) { return (K / kBlock + 3) / 4 * 4; }
int64_t pad8(int64_t v) { return (v + 7) / 8 * 8; }

// Block-scale job for the prep launch and the tensor map each GEMM stage reads it by.
PrepJob scales_job(const LinearArgs& a, float* out) {
  PrepJob j{};
  j.kind = kBlockScales;
  j.width = scale_ld(a.K);
  j.fdst = out;
  j.count = a.N * j.width;
  return j;
}

bool scales_map(const LinearArgs& a, int mode, const float* sc, CUtensorMap* map) {
  const int64_t ldk = scale_ld(a.K);
  return make_map(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, sc, ldk, a.N, 4 * ldk, 4, mode == 0 ? kTileF : 64,
                  CU_TENSOR_MAP_SWIZZLE_NONE);
}

// Workspace layouts (every part 1024-byte aligned).
struct FwdWs {
  size_t sTp, Bp, Aq, part, scale, total;
  FwdWs(int64_t M, int64_t N, int64_t K, int r) {
    const size_t rp = padded_rank(r), nq = adapter_nq(r);
    sTp = 0;
    Bp = sTp + a1024(2 * rp * M);
    Aq = Bp + a1024(2 * rp * N);
    part = Aq + a1024(2 * nq * K);
    scale = part + a1024(adapter_partial_bytes(M, K, r));
    total = scale + a1024(4 * static_cast<size_t>(N) * scale_ld(K));
  }
};

struct BwdWs {
  size_t sGp, ApT, Bt, Tt, Gt, part, scale, total;
  BwdWs(int64_t M, int64_t N, int64_t K, int r) {
    const size_t rp = padded_rank(r), nq = adapter_nq(r), Mp = pad8(M);
    size_t pb = adapter_partial_bytes(M, N, r);
    pb = std::max(pb, adapter_partial_bytes(N, M, r));
    pb = std::max(pb, adapter_partial_bytes(K, M, r));
    sGp = 0;
    ApT = sGp + a1024(2 * rp * M);
    Bt = ApT + a1024(2 * rp * K);
    Tt = Bt + a1024(2 * nq * N);
    Gt = Tt + a1024(2 * nq * Mp);
    part = Gt + a1024(2 * nq * Mp);
    scale = part + a1024(pb);
    total = scale + a1024(4 * static_cast<size_t>(N) * scale_ld(K));
  }
};

GemmParams base_params(const LinearArgs& a, int mode, void* out, int* status) {
  GemmParams p{};
  p.M = a.M;
  p.N = a.N;
  p.K = a.K;
  p.F = mode == 0 ? a.N : a.K;
  p.mode = mode;
  const int64_t red = mode == 0 ? a.K : a.N;
  p.red_steps = static_cast<int>((red + kBK - 1) / kBK);
  p.slab_steps = padded_rank(a.r) / kBK;
  p.tiles_t = static_cast<int>((a.M + kTileT - 1) / kTileT);
  p.tiles_f = static_cast<int>((p.F + kTileF - 1) / kTileF);
  p.f_fast = mode == 1 ? 1 : 0;
  p.absmax = a.W.absmax;
  p.nested = a.W.nested;
  p.offset = a.W.offset;
  p.dq = a.W.dq;
  p.out = static_cast<__nv_bfloat16*>(out);
  p.status = status;
  return p;
}

}  // namespace

size_t tc_fwd_ws_bytes(int64_t M, int64_t N, int64_t K, int r) { return FwdWs(M, N, K, r).total; }

size_t tc_bwd_ws_bytes(int64_t M, int64_t N, int64_t K, int r) { return BwdWs(M, N, K, r).total; }

// Forward: prep (A and B in bf16, block scales) -> T = x A^T (skinny tcgen05) ->
// T and bf16(s T) -> NF4 GEMM with the (s T) B^T slab.
cudaError_t tc_forward(const LinearArgs& a, const void* x, const float* A, const float* B, void* y, float* T,
                       void* ws, int* status, cudaStream_t st) {
  const FwdWs L(a.M, a.N, a.K, a.r);
  char* w = static_cast<char*>(ws);
  auto* sTp = reinterpret_cast<__nv_bfloat16*>(w + L.sTp);
  auto* Bp = reinterpret_cast<__nv_bfloat16*>(w + L.Bp);
  auto* Aq = reinterpret_cast<__nv_bfloat16*>(w + L.Aq);
  auto* part = reinterpret_cast<float*>(w + L.part);
  auto* sc = reinterpret_cast<float*>(w + L.scale);
  const int rp = padded_rank(a.r), nq = adapter_nq(a.r);
  PrepBuilder prep(a.W, a.K);
  {
    PrepJob j{};
    j.kind = kStageRowsDirect;   // A as the skinny pass's Q: [nq][K]
    j.r = a.r;
    j.src = A;
    j.dst = Aq;
    j.cols = a.K;
    j.count = static_cast<int64_t>(nq) * a.K;
    prep.add(j);
    PrepJob b{};
    b.kind = kStageRows;         // B as the slab's A operand: [N][rp]
    b.r = a.r;
    b.width = rp;
    b.scale = 1.0f;
    b.src = B;
    b.dst = Bp;
    b.count = a.N * rp;
    prep.add(b);
    prep.add(scales_job(a, sc));
  }
  cudaError_t e = prep.launch(st);
  if (e != cudaSuccess) return e;
  int ns = 0;
  if ((e = adapter_pass(x, a.K, a.M, false, Aq, a.K, a.r, a.M, a.K, part, status, &ns, st)) != cudaSuccess) return e;
  if ((e = adapter_finish(part, ns, a.M, a.r, 1.0f, T, 0, sTp, rp, a.s, nullptr, 0, st)) != cudaSuccess) return e;
  CUtensorMap tok, packed, slab_f, slab_t, scale;
  bool ok = make_map(&tok, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, x, a.K, a.M, 2 * a.K, kBK, kTileT,
                     CU_TENSOR_MAP_SWIZZLE_128B);
  ok = ok && make_map(&packed, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.W.packed, a.K / 2, a.N, a.K / 2, kBK / 2, kTileF,
                      CU_TENSOR_MAP_SWIZZLE_NONE);
  ok = ok && make_map(&slab_f, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, Bp, rp, a.N, 2 * rp, kBK, kTileF,
                      CU_TENSOR_MAP_SWIZZLE_128B);
  ok = ok && make_map(&slab_t, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, sTp, rp, a.M, 2 * rp, kBK, kTileT,
                      CU_TENSOR_MAP_SWIZZLE_128B);
  ok = ok && scales_map(a, 0, sc, &scale);
  if (!ok) return cudaErrorInvalidValue;
  return launch_gemm(base_params(a, 0, y, status), tok, packed, slab_f, slab_t, scale, st);
}

// Backward: prep (B^T, T^T, zeroed G^T, A^T in bf16, block scales) -> G = dY B ->
// G, bf16(s G), bf16(G)^T -> dB = s dY^T T -> NF4 GEMM for dX with the (s G) A slab ->
// dA = s G^T x.
cudaError_t tc_backward(const LinearArgs& a, const void* dy, const void* x, const float* T, const float* A,
                        const float* B, void* dx, float* dA, float* dB, float* G, void* ws, int* status,
                        cudaStream_t st) {
  const BwdWs L(a.M, a.N, a.K, a.r);
  char* w = static_cast<char*>(ws);
  auto* sGp = reinterpret_cast<__nv_bfloat16*>(w + L.sGp);
  auto* ApT = reinterpret_cast<__nv_bfloat16*>(w + L.ApT);
  auto* Bt = reinterpret_cast<__nv_bfloat16*>(w + L.Bt);
  auto* Tt = reinterpret_cast<__nv_bfloat16*>(w + L.Tt);
  auto* Gt = reinterpret_cast<__nv_bfloat16*>(w + L.Gt);
  auto* part = reinterpret_cast<float*>(w + L.part);
  auto* sc = reinterpret_cast<float*>(w + L.scale);
  const int rp = padded_rank(a.r), nq = adapter_nq(a.r);
  const int64_t Mp = pad8(a.M);
  PrepBuilder prep(a.W, a.K);
  {
    PrepJob j{};
    j.kind = kStageTransposed;   // B^T: [nq][N]
    j.r = a.r;
    j.width = a.N;
    j.src = B;
    j.dst = Bt;
    j.cols = a.N;
    j.count = static_cast<int64_t>(nq) * a.N;
    prep.add(j);
    PrepJob t = j;               // T^T: [nq][Mp]
    t.width = Mp;
    t.src = T;
    t.dst = Tt;
    t.cols = a.M;
    t.count = static_cast<int64_t>(nq) * Mp;
    prep.add(t);
    PrepJob g = t;               // G^T starts zero; the G finish fills rows < r, columns < M
    g.r = 0;
    g.dst = Gt;
    prep.add(g);
    PrepJob c{};
    c.kind = kStageColumns;      // A^T: [K][rp]
    c.r = a.r;
    c.width = rp;
    c.src = A;
    c.dst = ApT;
    c.cols = a.K;
    c.count = a.K * rp;
    prep.add(c);
    prep.add(scales_job(a, sc));
  }
  cudaError_t e = prep.launch(st);
  if (e != cudaSuccess) return e;
  int ns = 0;
  // G = dY B: rows M, reduction over N along dY's rows; also bf16(s G) and bf16(G)^T
  if ((e = adapter_pass(dy, a.N, a.M, false, Bt, a.N, a.r, a.M, a.N, part, status, &ns, st)) != cudaSuccess) return e;
  if ((e = adapter_finish(part, ns, a.M, a.r, 1.0f, G, 0, sGp, rp, a.s, Gt, Mp, st)) != cudaSuccess) return e;
  // dB = s dY^T T: rows N, reduction over M down dY's columns
  if ((e = adapter_pass(dy, a.N, a.M, true, Tt, Mp, a.r, a.N, a.M, part, status, &ns, st)) != cudaSuccess) return e;
  if ((e = adapter_finish(part, ns, a.N, a.r, a.s, dB, 0, nullptr, 0, 0.0f, nullptr, 0, st)) != cudaSuccess) return e;
  CUtensorMap tok, packed, slab_f, slab_t, scale;
  bool ok = make_map(&tok, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, dy, a.N, a.M, 2 * a.N, kBK, kTileT,
                     CU_TENSOR_MAP_SWIZZLE_128B);
  ok = ok && make_map(&packed, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.W.packed, a.K / 2, a.N, a.K / 2, kBK, kBK,
                      CU_TENSOR_MAP_SWIZZLE_NONE);
  ok = ok && make_map(&slab_f, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, ApT, rp, a.K, 2 * rp, kBK, kTileF,
                      CU_TENSOR_MAP_SWIZZLE_128B);
  ok = ok && make_map(&slab_t, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, sGp, rp, a.M, 2 * rp, kBK, kTileT,
                      CU_TENSOR_MAP_SWIZZLE_128B);
  ok = ok && scales_map(a, 1, sc, &scale);
  if (!ok) return cudaErrorInvalidValue;
  if ((e = launch_gemm(base_params(a, 1, dx, status), tok, packed, slab_f, slab_t, scale, st)) != cudaSuccess)
    return e;
  // dA = s G^T x: rows K, reduction over M down x's columns; written as [r][K]
  if ((e = adapter_pass(x, a.K, a.M, true, Gt, Mp, a.r, a.K, a.M, part, status, &ns, st)) != cudaSuccess) return e;
  return adapter_finish(part, ns, a.K, a.r, a.s, dA, 1, nullptr, 0, 0.0f, nullptr, 0, st);
}

}  // namespace qnf4
