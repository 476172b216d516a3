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
// Warp roles (320 threads):
//   warp 0      TMA producer: token tile (128B-swizzled) + packed NF4 tile per stage,
//               or the two adapter slab tiles for the last (rank / 64) stages;
//   warp 1      TMEM allocation; lane 0 issues tcgen05.mma and tcgen05.commit;
//   warps 2..5  decoders: 128 threads, one 64-element NF4 block (one 128-byte row of
//               the A tile) each per stage, written bf16 into the swizzled layout
//               the MMA reads (K-major for the forward, MN-major for dX);
//   warps 6..9  epilogue: tcgen05.ld of the accumulator, bf16 stores.
// Two accumulators of 256 columns let the epilogue of one tile overlap the
// main loop of the next.  Every mbarrier wait is bounded in time; a wait that
// gives up sets NF4_ERR_TIMEOUT in the status word and the CTA winds down,
// freeing its TMEM.
#include "linear_tc.cuh"
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
constexpr int kThreads = 320;
constexpr int kTmemCols = 512;
constexpr int kSmemBytes = 1024 + kStages * kStageBytes + 1024 /*dyn8*/ + 256 /*barriers, flags*/;

static_assert(kStageBytes % 1024 == 0, "stage buffers must stay 1024-byte aligned");

// ---- NF4 decode -------------------------------------------------------------------------

// Scaled lookup table of one block: entry i = bf16(nf4[i] * a'), split into low bytes
// (L, 4 registers of 4 entries) and high bytes (H), so prmt can index it by nibble.
__device__ __forceinline__ void build_lut(float a, uint32_t (&L)[4], uint32_t (&H)[4]) {
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    const __nv_bfloat162 p0 = __floats2bfloat162_rn(__fmul_rn(nf4_value(4 * t + 0), a),
                                                    __fmul_rn(nf4_value(4 * t + 1), a));
    const __nv_bfloat162 p1 = __floats2bfloat162_rn(__fmul_rn(nf4_value(4 * t + 2), a),
                                                    __fmul_rn(nf4_value(4 * t + 3), a));
    const uint32_t u0 = *reinterpret_cast<const uint32_t*>(&p0);
    const uint32_t u1 = *reinterpret_cast<const uint32_t*>(&p1);
    L[t] = prmt(u0, u1, 0x6420u);
    H[t] = prmt(u0, u1, 0x7531u);
  }
}

// Eight weights of one packed word (element 2i in the high nibble of byte i) to four
// bf16x2 registers in element order.
__device__ __forceinline__ void decode8(uint32_t w, const uint32_t (&L)[4], const uint32_t (&H)[4],
                                        uint32_t* out) {
  const uint32_t ws = ((w >> 4) & 0x0F0F0F0Fu) | ((w << 4) & 0xF0F0F0F0u);  // nibble i = element i
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const uint32_t q = ws >> (16 * h);
    const uint32_t s7 = q & 0x7777u;                      // index within a half table
    const uint32_t sb = 0x3210u | ((q >> 1) & 0x4444u);   // pick the half by bit 3
    const uint32_t lo = prmt(prmt(L[0], L[1], s7), prmt(L[2], L[3], s7), sb);
    const uint32_t hi = prmt(prmt(H[0], H[1], s7), prmt(H[2], H[3], s7), sb);
    out[2 * h] = prmt(lo, hi, 0x5140u);
    out[2 * h + 1] = prmt(lo, hi, 0x7362u);
  }
}

struct GemmParams {
  int64_t M;           // tokens
  int64_t F;           // output features (N forward, K for dX)
  int64_t N, K;        // W is [N, K]
  int mode;            // 0 forward, 1 dX
  int red_steps;       // ceil(contraction / 64)
  int slab_steps;      // padded rank / 64
  int tiles_t, tiles_f;
  const void* absmax;  // uint8 codes (dq) or float
  const float* nested;
  const float* offset;
  int dq;
  __nv_bfloat16* out;  // [M, F]
  int* status;
};

// Block scale inputs of one decode step, loaded one step ahead of use.
struct BlockMeta {
  float nested_or_absmax;
  uint32_t code;
  bool valid;
};

__device__ __forceinline__ BlockMeta fetch_meta(const GemmParams& p, int64_t tile, int step, int row) {
  BlockMeta m{0.0f, 0u, false};
  const int64_t f0 = (tile / p.tiles_t) * kTileF;
  int64_t n, kcol;
  if (p.mode == 0) {
    n = f0 + row;
    kcol = static_cast<int64_t>(step) * kBK;
  } else {
    n = static_cast<int64_t>(step) * kBK + (row & 63);
    kcol = f0 + 64 * (row >> 6);
  }
  if (n >= p.N || kcol >= p.K) return m;
  const int64_t blk = n * (p.K / kBlock) + kcol / kBlock;
  m.valid = true;
  if (p.dq) {
    m.code = static_cast<const uint8_t*>(p.absmax)[blk];
    m.nested_or_absmax = p.nested[blk >> 8];
  } else {
    m.nested_or_absmax = static_cast<const float*>(p.absmax)[blk];
  }
  return m;
}

__global__ void __launch_bounds__(kThreads, 1)
nf4_tc_gemm(const __grid_constant__ CUtensorMap tm_tok, const __grid_constant__ CUtensorMap tm_packed,
            const __grid_constant__ CUtensorMap tm_slab_f, const __grid_constant__ CUtensorMap tm_slab_t,
            const GemmParams p, const DecodeTables tabs) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* base_ptr = smem_raw + (base - raw);
  float* dyn8 = reinterpret_cast<float*>(base_ptr + kStages * kStageBytes);
  uint64_t* bars = reinterpret_cast<uint64_t*>(base_ptr + kStages * kStageBytes + 1024);
  // bars: full[4] aready[4] empty[4] accfull[2] accempty[2]
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 16);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 16) + 1;
  auto bar = [&](int i) { return smem_u32(bars + i); };
  auto stage_a = [&](int s) { return base + s * kStageBytes; };
  auto stage_b = [&](int s) { return base + s * kStageBytes + kABytes; };
  auto stage_p = [&](int s) { return base + s * kStageBytes + kABytes + kBBytes; };

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if (threadIdx.x < 256) dyn8[threadIdx.x] = tabs.dyn8[threadIdx.x];
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar(s), 1);                 // full: producer arrive + TMA bytes
      mbar_init(bar(4 + s), 4);             // aready: one arrive per decoder warp
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

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      uint32_t it = 0;
      int last_phase[kStages];
      bool issued[kStages];
      for (int s = 0; s < kStages; ++s) issued[s] = false, last_phase[s] = 0;
      bool ok = true;
      for (int64_t tile = blockIdx.x; tile < total_tiles && ok; tile += gridDim.x) {
        const int t0 = static_cast<int>((tile % p.tiles_t) * kTileT);
        const int f0 = static_cast<int>((tile / p.tiles_t) * kTileF);
        for (int step = 0; step < steps; ++step, ++it) {
          const int s = it % kStages;
          const uint32_t ph = (it / kStages) & 1u;
          if (!mbar_wait(bar(8 + s), ph ^ 1u, abort_flag, p.status)) { ok = false; break; }
          if (step < p.red_steps) {
            mbar_expect_tx(bar(s), kBBytes + kPBytes);
            tma_load_2d(stage_b(s), &tm_tok, bar(s), step * kBK, t0);
            if (p.mode == 0) tma_load_2d(stage_p(s), &tm_packed, bar(s), step * (kBK / 2), f0);
            else tma_load_2d(stage_p(s), &tm_packed, bar(s), f0 / 2, step * kBK);
          } else {
            const int j = (step - p.red_steps) * kBK;
            mbar_expect_tx(bar(s), kBBytes + kABytes);
            tma_load_2d(stage_b(s), &tm_slab_t, bar(s), j, t0);
            tma_load_2d(stage_a(s), &tm_slab_f, bar(s), j, f0);
          }
          issued[s] = true;
          last_phase[s] = ph;
        }
      }
      if (!ok) {  // let copies already in flight land before the CTA exits
        for (int s = 0; s < kStages; ++s)
          if (issued[s]) mbar_drain(bar(s), last_phase[s]);
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      const uint32_t idesc_main = idesc_bf16(kTileF, kTileT, p.mode == 1 ? 1u : 0u);
      const uint32_t idesc_slab = idesc_bf16(kTileF, kTileT, 0u);
      uint32_t it = 0;
      uint32_t lt = 0;
      bool ok = true;
      for (int64_t tile = blockIdx.x; tile < total_tiles && ok; tile += gridDim.x, ++lt) {
        const uint32_t b = lt & 1u;
        const uint32_t aph = (lt >> 1) & 1u;
        if (!mbar_wait(bar(14 + b), aph ^ 1u, abort_flag, p.status)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + b * kTileT;
        for (int step = 0; step < steps; ++step, ++it) {
          const int s = it % kStages;
          const uint32_t ph = (it / kStages) & 1u;
          if (!mbar_wait(bar(s), ph, abort_flag, p.status) || !mbar_wait(bar(4 + s), ph, abort_flag, p.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const bool slab = step >= p.red_steps;
          const bool mn_major = (p.mode == 1) && !slab;
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
        }
        if (!ok) break;
        umma_commit(bar(12 + b));
      }
    }
  } else if (warp < 6) {
    // ---------------- NF4 decoders ----------------
    const int row = threadIdx.x - 64;           // row of the A tile, 0..127
    uint32_t it = 0;
    bool ok = true;
    int64_t tile = blockIdx.x;
    BlockMeta cur = (tile < total_tiles) ? fetch_meta(p, tile, 0, row) : BlockMeta{0.0f, 0u, false};
    const float offset = p.dq ? *p.offset : 0.0f;
    for (; tile < total_tiles && ok; tile += gridDim.x) {
      for (int step = 0; step < steps; ++step, ++it) {
        const int s = it % kStages;
        const uint32_t ph = (it / kStages) & 1u;
        if (step < p.red_steps) {
          BlockMeta nxt{0.0f, 0u, false};
          if (step + 1 < p.red_steps) nxt = fetch_meta(p, tile, step + 1, row);
          else if (tile + gridDim.x < total_tiles) nxt = fetch_meta(p, tile + gridDim.x, 0, row);
          if (!__all_sync(0xffffffffu, mbar_wait(bar(s), ph, abort_flag, p.status))) { ok = false; break; }
          const uint32_t arow = stage_a(s) + row * 128;
          const uint32_t sw = static_cast<uint32_t>(row & 7);
          if (cur.valid) {
            const float a = p.dq ? __fadd_rn(__fmul_rn(dyn8[cur.code], cur.nested_or_absmax), offset)
                                 : cur.nested_or_absmax;
            uint32_t L[4], H[4];
            build_lut(a, L, H);
            const uint32_t poff = (p.mode == 0) ? row * 32 : (row & 63) * 64 + (row >> 6) * 32;
            const uint8_t* src = base_ptr + (stage_p(s) - base) + poff;
            const uint4 w0 = *reinterpret_cast<const uint4*>(src);
            const uint4 w1 = *reinterpret_cast<const uint4*>(src + 16);
            const uint32_t words[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              uint32_t o[4];
              decode8(words[i], L, H, o);
              const uint32_t dst = arow + ((static_cast<uint32_t>(i) ^ sw) << 4);
              asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(dst), "r"(o[0]), "r"(o[1]), "r"(o[2]),
                           "r"(o[3])
                           : "memory");
            }
          } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const uint32_t dst = arow + (static_cast<uint32_t>(i) << 4);
              asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};" ::"r"(dst), "r"(0u) : "memory");
            }
          }
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(4 + s));
          cur = nxt;
        } else {
          if (!__all_sync(0xffffffffu, mbar_wait(bar(s), ph, abort_flag, p.status))) { ok = false; break; }
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(4 + s));
        }
      }
    }
  } else {
    // ---------------- epilogue ----------------
    const int quarter = warp & 3;               // TMEM lanes 32*quarter .. +31
    uint32_t lt = 0;
    for (int64_t tile = blockIdx.x; tile < total_tiles; tile += gridDim.x, ++lt) {
      const uint32_t b = lt & 1u;
      const uint32_t aph = (lt >> 1) & 1u;
      if (!__all_sync(0xffffffffu, mbar_wait(bar(12 + b), aph, abort_flag, p.status))) break;
      tc_fence_after();
      const int64_t t0 = (tile % p.tiles_t) * kTileT;
      const int64_t f = (tile / p.tiles_t) * kTileF + quarter * 32 + lane;
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

// ---- adapter staging: bf16 operands of the LoRA slab, zero-padded to rp columns ------------

__global__ void stage_rows_bf16(const float* __restrict__ src, int64_t rows, int r, int rp, float scale,
                                __nv_bfloat16* __restrict__ dst) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= rows * rp) return;
  const int64_t row = i / rp;
  const int j = static_cast<int>(i % rp);
  dst[i] = __float2bfloat16_rn(j < r ? scale * src[row * r + j] : 0.0f);
}

__global__ void stage_transposed_bf16(const float* __restrict__ A, int64_t K, int r, int rp,
                                      __nv_bfloat16* __restrict__ dst) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= K * rp) return;
  const int64_t k = i / rp;
  const int j = static_cast<int>(i % rp);
  dst[i] = __float2bfloat16_rn(j < r ? A[static_cast<int64_t>(j) * K + k] : 0.0f);
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
                        const CUtensorMap& slab_f, const CUtensorMap& slab_t, cudaStream_t st) {
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    attr_err = cudaFuncSetAttribute(nf4_tc_gemm, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  });
  if (attr_err != cudaSuccess) return attr_err;
  const int64_t tiles = static_cast<int64_t>(p.tiles_t) * p.tiles_f;
  const int grid = static_cast<int>(tiles < sm_count() ? tiles : sm_count());
  KernelTimer timer(p.mode == 0 ? NF4_TIME_FWD_GEMM : NF4_TIME_DX_GEMM, st);
  nf4_tc_gemm<<<grid, kThreads, kSmemBytes, st>>>(tok, packed, slab_f, slab_t, p, decode_tables());
  note_launch();
  return cudaGetLastError();
}

cudaError_t stage_rows(const float* src, int64_t rows, int r, float scale, __nv_bfloat16* dst, cudaStream_t st) {
  const int rp = padded_rank(r);
  const int64_t n = rows * rp;
  stage_rows_bf16<<<static_cast<unsigned>((n + 255) / 256), 256, 0, st>>>(src, rows, r, rp, scale, dst);
  note_launch();
  return cudaGetLastError();
}

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
  p.absmax = a.W.absmax;
  p.nested = a.W.nested;
  p.offset = a.W.offset;
  p.dq = a.W.dq;
  p.out = static_cast<__nv_bfloat16*>(out);
  p.status = status;
  return p;
}

}  // namespace

size_t tc_fwd_ws_bytes(int64_t M, int64_t N, int64_t K, int r) {
  const size_t rp = padded_rank(r);
  return a1024(2 * rp * M) + a1024(2 * rp * N) + a1024(adapter_fwd_ws_bytes(M, N, K, r));
}

size_t tc_bwd_ws_bytes(int64_t M, int64_t N, int64_t K, int r) {
  const size_t rp = padded_rank(r);
  return a1024(2 * rp * M) + a1024(2 * rp * K) + a1024(adapter_bwd_ws_bytes(M, N, K, r));
}

cudaError_t tc_forward(const LinearArgs& a, const void* x, const float* A, const float* B, void* y, float* T,
                       void* ws, int* status, cudaStream_t st) {
  const int rp = padded_rank(a.r);
  auto* sTp = static_cast<__nv_bfloat16*>(ws);
  auto* Bp = reinterpret_cast<__nv_bfloat16*>(static_cast<char*>(ws) + a1024(2 * static_cast<size_t>(rp) * a.M));
  void* aws = static_cast<char*>(ws) + a1024(2 * static_cast<size_t>(rp) * a.M) +
              a1024(2 * static_cast<size_t>(rp) * a.N);
  cudaError_t e = adapter_forward(a, x, A, T, sTp, aws, status, st);
  if (e != cudaSuccess) return e;
  {
    KernelTimer timer(NF4_TIME_ADAPTER, st);
    if ((e = stage_rows(B, a.N, a.r, 1.0f, Bp, st)) != cudaSuccess) return e;
  }
  CUtensorMap tok, packed, slab_f, slab_t;
  bool ok = make_map(&tok, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, x, a.K, a.M, 2 * a.K, kBK, kTileT,
                     CU_TENSOR_MAP_SWIZZLE_128B);
  ok = ok && make_map(&packed, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.W.packed, a.K / 2, a.N, a.K / 2, kBK / 2, kTileF,
                      CU_TENSOR_MAP_SWIZZLE_NONE);
  ok = ok && make_map(&slab_f, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, Bp, rp, a.N, 2 * rp, kBK, kTileF,
                      CU_TENSOR_MAP_SWIZZLE_128B);
  ok = ok && make_map(&slab_t, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, sTp, rp, a.M, 2 * rp, kBK, kTileT,
                      CU_TENSOR_MAP_SWIZZLE_128B);
  if (!ok) return cudaErrorInvalidValue;
  return launch_gemm(base_params(a, 0, y, status), tok, packed, slab_f, slab_t, st);
}

cudaError_t tc_backward(const LinearArgs& a, const void* dy, const void* x, const float* T, const float* A,
                        const float* B, void* dx, float* dA, float* dB, float* G, void* ws, int* status,
                        cudaStream_t st) {
  const int rp = padded_rank(a.r);
  auto* sGp = static_cast<__nv_bfloat16*>(ws);
  auto* ApT = reinterpret_cast<__nv_bfloat16*>(static_cast<char*>(ws) + a1024(2 * static_cast<size_t>(rp) * a.M));
  void* aws = static_cast<char*>(ws) + a1024(2 * static_cast<size_t>(rp) * a.M) +
              a1024(2 * static_cast<size_t>(rp) * a.K);
  cudaError_t e = adapter_backward_pre(a, dy, T, B, G, sGp, dB, aws, status, st);
  if (e != cudaSuccess) return e;
  {
    KernelTimer timer(NF4_TIME_ADAPTER, st);
    const int64_t n = a.K * rp;
    stage_transposed_bf16<<<static_cast<unsigned>((n + 255) / 256), 256, 0, st>>>(A, a.K, a.r, rp, ApT);
    note_launch();
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  CUtensorMap tok, packed, slab_f, slab_t;
  bool ok = make_map(&tok, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, dy, a.N, a.M, 2 * a.N, kBK, kTileT,
                     CU_TENSOR_MAP_SWIZZLE_128B);
  ok = ok && make_map(&packed, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.W.packed, a.K / 2, a.N, a.K / 2, kBK, kBK,
                      CU_TENSOR_MAP_SWIZZLE_NONE);
  ok = ok && make_map(&slab_f, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, ApT, rp, a.K, 2 * rp, kBK, kTileF,
                      CU_TENSOR_MAP_SWIZZLE_128B);
  ok = ok && make_map(&slab_t, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, sGp, rp, a.M, 2 * rp, kBK, kTileT,
                      CU_TENSOR_MAP_SWIZZLE_128B);
  if (!ok) return cudaErrorInvalidValue;
  e = launch_gemm(base_params(a, 1, dx, status), tok, packed, slab_f, slab_t, st);
  if (e != cudaSuccess) return e;
  return adapter_backward_post(a, x, dA, aws, status, st);
}

}  // namespace qnf4
