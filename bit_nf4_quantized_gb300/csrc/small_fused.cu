// The 16-bit profiles of the QLoRA linear for small weights (K and N up to 1024, at most 2^21
// weights) and M > 16, in one launch for the forward and one for the backward, over the
// projections of a group at once.  Same operands and roundings as the tiled path: the weight
// decoded to T16(nf4[q] * a'), x or dY, T16(A) and T16(B), T16(s T) / T16(s G) for the adapter
// terms, T16(G) and T16(T) for the adapter gradients, fp32 accumulation; only the order of
// the fp32 sums differs.
//
// Math ("Native model adaptation and NF4", sections "One model contract", "Packed NF4 and
// the portable QLoRA profile", "Fused GPU NF4 decodes inside the matrix kernel"):
//   forward   T = x A^T,  y = x W^T + s T B^T
//   backward  G = dY B,   dX = dY W + s G A,  dA = s G^T x,  dB = s dY^T T.
//
// Why a separate path.  At these sizes (the SmolLM2-135M-shaped layers: K = 576, N = 576 or
// 192, M = 512) the tiled path's chain of about ten launches per call (decode and staging,
// skinny adapter passes and their finishes, the GEMM) costs more than the arithmetic, and its
// 256 x 256 tiles leave most SMs idle.  Here one CTA holds a 32-token x 64-feature output tile
// with the whole contraction in shared memory and does every step of the tile itself: the
// weight is decoded from the stored codes in registers straight into mma.sync fragments, the
// rank-r down-projection of its 32 tokens is recomputed by every feature tile (r = 16 columns
// against 64), and the adapter term is added from shared memory before the tile is stored.
// Tiles are sized so that two CTAs fit an SM (about 82 KB of shared memory each at K = 576)
// and a SmolLM2-shaped layer's q and v tiles (192 forward, 288 backward) run in one wave.
//
// Fragment order along the contraction.  Within each 32-deep slice, lane 4g + c of a warp
// takes contraction indices 8c .. 8c + 7 for both operands: one 16-byte shared load of x (or
// dY) per row and one packed code word of the weight (decoded to eight values in order) per
// row.  Two 16-deep mma.sync steps consume the slice, indices 8c .. 8c + 3 in the first and
// 8c + 4 .. 8c + 7 in the second; both operands follow the same permutation of the slice, so
// the products summed are exactly those of the plain order.
#include <algorithm>

#include <cuda_fp16.h>

#include "decode.cuh"
#include "linear_tc.cuh"
#include "mma_sync.cuh"

namespace qnf4 {
namespace {

constexpr int kTT = 32;          // tokens per forward tile
constexpr int kTF = 64;          // output features (forward) or input features (dX) per tile
constexpr int kWarps = 8;
constexpr int kThreads = 32 * kWarps;

// Row strides in shared memory (bytes), chosen so that the lanes of a quarter warp reading
// 16 bytes each, or a warp reading 4 bytes each, meet distinct banks.
__host__ __device__ constexpr int64_t row16(int64_t k) { return (2 * k + 127) / 128 * 128 + 64; }   // 16-byte reads
__host__ __device__ constexpr int64_t rowp(int64_t k) { return k / 2 + 16; }                        // packed codes
__host__ __device__ constexpr int64_t rowr(int64_t rp) { return 2 * rp + 16; }                      // rank rows

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async4(uint32_t dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_group1() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }

// One float rounded to T16 into shared memory.
template <typename T16>
__device__ __forceinline__ void st_shared16(uint32_t addr, float v) {
  const uint32_t p = pack2<T16>(v, 0.0f);
  asm volatile("st.shared.b16 [%0], %1;" ::"r"(addr), "h"(static_cast<unsigned short>(p & 0xFFFFu)) : "memory");
}

// Four 8 x 8 16-bit matrices; lane i gives the address of row i & 7 of matrix i >> 3.
__device__ __forceinline__ void ldsm4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}
__device__ __forceinline__ void ldsm4t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}

// Rows [r0, r0 + rows) of a 16-bit row-major matrix with `cols` columns (a multiple of 8) into
// shared memory at `dst`, row stride `stride`; rows past `valid` are zero.
template <typename T16>
__device__ __forceinline__ void stage_rows16(uint32_t dst, int64_t stride, const T16* src, int64_t r0, int rows,
                                             int64_t valid, int64_t cols) {
  const int chunks = static_cast<int>(cols / 8);   // 32-bit index arithmetic throughout
  for (int i = threadIdx.x; i < rows * chunks; i += kThreads) {
    const int r = i / chunks, c = i - r * chunks;
    const uint32_t d = dst + static_cast<uint32_t>(r * stride + c * 16);
    if (r0 + r < valid) cp_async16(d, src + (r0 + r) * cols + c * 8);
    else asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};" ::"r"(d), "r"(0u) : "memory");
  }
}

// fp32 rows [r0, r0 + rows) x columns [0, cols_pad) of a row-major matrix with `cols` columns,
// copied asynchronously into `raw` ([rows][cols_pad] fp32); entries outside rows < valid,
// cols < cols are zero.  vec: 16-byte copies, for rows that are 16-byte aligned and
// cols_pad <= cols, a multiple of 4 (the source's row stride is always `cols`).
__device__ __forceinline__ void stage_f32_raw(uint32_t raw, const float* src, int64_t r0, int rows, int64_t valid,
                                              int64_t cols, int64_t cols_pad, bool vec) {
  const int cp = static_cast<int>(cols_pad);
  if (vec) {
    const int q = cp / 4;
    for (int i = threadIdx.x; i < rows * q; i += kThreads) {
      const int r = i / q, c = 4 * (i - r * q);
      const uint32_t d = raw + static_cast<uint32_t>((r * cp + c) * 4);
      if (r0 + r < valid) cp_async16(d, src + (r0 + r) * cols + c);
      else asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};" ::"r"(d), "r"(0u) : "memory");
    }
    return;
  }
  for (int i = threadIdx.x; i < rows * cp; i += kThreads) {
    const int r = i / cp, c = i - r * cp;
    const uint32_t d = raw + static_cast<uint32_t>(i * 4);
    if (r0 + r < valid && c < cols) cp_async4(d, src + (r0 + r) * cols + c);
    else st_shared32(d, 0u);
  }
}

// The staged fp32 [rows][cols_pad] as T16 at `dst` (row stride `stride`), after the copies landed.
template <typename T16>
__device__ __forceinline__ void convert_raw(uint32_t dst, int64_t stride, const float* raw, int rows, int64_t cols_pad) {
  const int pairs = static_cast<int>(cols_pad / 2), cp = static_cast<int>(cols_pad);
  for (int i = threadIdx.x; i < rows * pairs; i += kThreads) {
    const int r = i / pairs, c = 2 * (i - r * pairs);
    const float2 v = *reinterpret_cast<const float2*>(raw + r * cp + c);
    st_shared32(dst + static_cast<uint32_t>(r * stride + c * 2), pack2<T16>(v.x, v.y));
  }
}

}  // namespace

// ---- forward ----------------------------------------------------------------------------

namespace {

struct FwdUnitItem {
  LinearArgs a;
  const void* x;     // [M, K] 16-bit
  const float* A;    // [r, K]
  const float* B;    // [N, r]
  void* y;           // [M, N] 16-bit
  float* T;          // [M, r]
  const void* w16;   // decoded weight [N, K], or null: decode the stored codes in registers
  int rp;            // r rounded up to 16
  int tiles_f;
  int64_t unit0;     // first unit of this item
};
struct FwdParams {
  FwdUnitItem it[kSmallMaxGroup];
  int n;
  int64_t M;
};

// Weight rows in shared memory: the packed codes, or the decoded 16-bit values.
__host__ __device__ inline int64_t wrow(int64_t K, bool w16) { return w16 ? row16(K) : rowp(K); }

// Shared memory of the forward: x rows, weight rows, T16(A) rows, T16(s T); with the stored
// codes also the block scales.
__host__ __device__ inline int64_t fwd_smem_bytes(int64_t K, int rp, bool w16) {
  const int64_t base = kTT * row16(K) + kTF * wrow(K, w16) + rp * row16(K) + kTT * rowr(rp);
  return w16 ? base : base + kTF * (K / 64) * 4;
}

template <typename T16>
__global__ void __launch_bounds__(kThreads, 2)
small_fused_fwd(FwdParams p, DecodeTables tabs) {
  constexpr bool F16 = std::is_same<T16, __half>::value;
  extern __shared__ __align__(16) unsigned char smem[];
  __shared__ float dyn8[256];
  __shared__ FwdUnitItem item;
  for (int i = threadIdx.x; i < 256; i += kThreads) dyn8[i] = tabs.dyn8[i];
  if (threadIdx.x == 0) {
    int k = 0;
    while (k + 1 < p.n && static_cast<int64_t>(blockIdx.x) >= p.it[k + 1].unit0) ++k;
    for (int j = 0; j < kSmallMaxGroup; ++j)
      if (j == k) item = p.it[j];
  }
  __syncthreads();
  pdl_allow_next();
  pdl_wait();
  const LinearArgs& a = item.a;
  const int64_t K = a.K, N = a.N, M = p.M;
  const int rp = item.rp;
  const int64_t local = blockIdx.x - item.unit0;
  const int64_t t0 = (local / item.tiles_f) * kTT, f0 = (local % item.tiles_f) * kTF;
  const int64_t nbr = K / 64;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, c = lane & 3;
  const int fw = 8 * warp;

  const uint32_t s_x = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
  const bool dec = item.w16 == nullptr;   // decode from the stored codes
  const int64_t wr = wrow(K, !dec);
  const uint32_t s_w = s_x + kTT * row16(K);
  const uint32_t s_a = s_w + kTF * wr;
  const uint32_t s_t = s_a + rp * row16(K);
  const uint32_t s_end = s_t + kTT * rowr(rp);
  float* s_sc = reinterpret_cast<float*>(smem + (s_end - s_x));              // stored codes: scales

  // every copy in flight at once: x rows, the weight rows (packed codes or decoded values), the
  // block scales; A straight from global memory into registers, in batches of 8 float4
  stage_rows16(s_x, row16(K), static_cast<const T16*>(item.x), t0, kTT, M, K);
  if (dec) {
    const int chunks = static_cast<int>(K / 32);   // 16-byte chunks of a packed row
    for (int i = threadIdx.x; i < kTF * chunks; i += kThreads) {
      const int r = i / chunks, cc = i - r * chunks;
      const uint32_t d = s_w + static_cast<uint32_t>(r * rowp(K) + cc * 16);
      if (f0 + r < N) cp_async16(d, a.W.packed + (f0 + r) * (K / 2) + cc * 16);
      else asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};" ::"r"(d), "r"(0u) : "memory");
    }
  } else {
    stage_rows16(s_w, row16(K), static_cast<const T16*>(item.w16), f0, kTF, N, K);
  }
  // B's fragments for the adapter term (8 values a lane), used after the main loop
  float bv[2][4];
  {
    const int64_t f = f0 + fw + g;
#pragma unroll
    for (int kk = 0; kk < 2; ++kk) {
      const int j0 = 16 * kk + 2 * c;
      const int js[4] = {j0, j0 + 1, j0 + 8, j0 + 9};
#pragma unroll
      for (int e = 0; e < 4; ++e) bv[kk][e] = (f < N && js[e] < a.r) ? __ldg(item.B + f * a.r + js[e]) : 0.0f;
    }
  }
  // the block scales' inputs and A's first 12 float4 a thread: every load issued before any is
  // used, so that the staging costs one round trip to memory
  constexpr int U = 1024 / kThreads;   // 64 rows x at most 16 blocks
  uint32_t scode[U];
  float snest[U];
  const float soff = (dec && a.W.dq) ? __ldg(a.W.offset) : 0.0f;
  const int nb32 = static_cast<int>(nbr);
#pragma unroll
  for (int u = 0; u < U; ++u) {
    const int i = threadIdx.x + u * kThreads, r = i / nb32, kb = i - r * nb32;
    scode[u] = 0, snest[u] = 0.0f;
    if (dec && i < kTF * nb32 && f0 + r < N) {
      const int64_t gi = (f0 + r) * nbr + kb;
      if (a.W.dq) {
        scode[u] = __ldg(static_cast<const uint8_t*>(a.W.absmax) + gi);
        snest[u] = __ldg(a.W.nested + (gi >> 8));
      } else {
        snest[u] = __ldg(static_cast<const float*>(a.W.absmax) + gi);
      }
    }
  }
  // T16(A) rows [rp][K]: rows past r are zero
  const int q4 = static_cast<int>(K / 4), atotal = rp * q4;
  const bool avec = (reinterpret_cast<uintptr_t>(item.A) & 15) == 0;
  constexpr int kAB = 12;   // float4 a thread per batch
  auto a_load = [&](int i0, float4 (&v)[kAB]) {
#pragma unroll
    for (int u = 0; u < kAB; ++u) {
      const int i = i0 + u * kThreads, j = i / q4, c4 = i - j * q4;
      v[u] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
      if (i < atotal && j < a.r) {
        const float* src = item.A + static_cast<int64_t>(j) * K + 4 * c4;
        v[u] = avec ? __ldg(reinterpret_cast<const float4*>(src))
                    : make_float4(__ldg(src), __ldg(src + 1), __ldg(src + 2), __ldg(src + 3));
      }
    }
  };
  auto a_store = [&](int i0, const float4 (&v)[kAB]) {
#pragma unroll
    for (int u = 0; u < kAB; ++u) {
      const int i = i0 + u * kThreads, j = i / q4, c4 = i - j * q4;
      if (i < atotal)
        asm volatile("st.shared.v2.b32 [%0], {%1, %2};" ::"r"(s_a + static_cast<uint32_t>(j * row16(K) + 8 * c4)),
                     "r"(pack2<T16>(v[u].x, v[u].y)), "r"(pack2<T16>(v[u].z, v[u].w))
                     : "memory");
    }
  };
  {
    float4 v[kAB];
    a_load(threadIdx.x, v);
    if (dec) {
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int i = threadIdx.x + u * kThreads;
        if (i < kTF * nb32)
          s_sc[i] = a.W.dq ? __fadd_rn(__fmul_rn(dyn8[scode[u]], snest[u]), soff) : snest[u];
      }
    }
    a_store(threadIdx.x, v);
    for (int i0 = threadIdx.x + kAB * kThreads; i0 < atotal; i0 += kAB * kThreads) {
      a_load(i0, v);
      a_store(i0, v);
    }
  }
  cp_async_wait_all();
  __syncthreads();

  // warp w: output features 8w .. 8w + 7 of the tile for both token blocks, and T of token
  // block tb = w & 1 for rank block q = w >> 1 (when 8 q < rp)
  const int tb = warp & 1, q = warp >> 1;
  const bool has_t = 8 * q < rp;
  const uint32_t R16 = static_cast<uint32_t>(row16(K));
  const uint32_t xrow = s_x + (g * R16 + 16 * c);           // + 16 mb R16 (+ 8 R16), + 64 ks
  const uint32_t wrow_ = dec ? s_w + static_cast<uint32_t>((fw + g) * rowp(K) + 4 * c)
                             : s_w + (fw + g) * R16 + 16 * c;
  const uint32_t arow = s_a + (8 * q + g) * R16 + 16 * c;   // + 64 ks
  float acc[2][4] = {};                  // [token block][fragment]
  float tac[4] = {};                     // T of token block tb, rank block q
  for (int kb = 0; kb < nb32; ++kb) {
    uint32_t L[4], H[4];
    if (dec) build_lut<T16>(s_sc[(fw + g) * nb32 + kb], L, H);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint32_t ks = static_cast<uint32_t>(2 * kb + h);   // 32-deep slice
      uint32_t bw[4];
      if (dec) {
        decode8(ld_shared32(wrow_ + ks * 16), L, H, bw);
      } else {
        const uint4 v = lds128(wrow_ + ks * 64);
        bw[0] = v.x, bw[1] = v.y, bw[2] = v.z, bw[3] = v.w;
      }
      uint4 xt0{}, xt1{};
#pragma unroll
      for (int mb = 0; mb < 2; ++mb) {
        const uint32_t xa_addr = xrow + static_cast<uint32_t>(16 * mb) * R16 + ks * 64;
        const uint4 xa = lds128(xa_addr);
        const uint4 xb = lds128(xa_addr + 8 * R16);
        mma16816<F16>(acc[mb], xa.x, xb.x, xa.y, xb.y, bw[0], bw[1]);
        mma16816<F16>(acc[mb], xa.z, xb.z, xa.w, xb.w, bw[2], bw[3]);
        if (mb == tb) xt0 = xa, xt1 = xb;
      }
      if (has_t) {
        const uint4 ta = lds128(arow + ks * 64);
        mma16816<F16>(tac, xt0.x, xt1.x, xt0.y, xt1.y, ta.x, ta.y);
        mma16816<F16>(tac, xt0.z, xt1.z, xt0.w, xt1.w, ta.z, ta.w);
      }
    }
  }
  // T (fp32, written by the first feature tile) and 16-bit s T for the adapter term
  if (has_t) {
    const int64_t tr0 = t0 + 16 * tb + g;
    const int j0 = 8 * q + 2 * c;
    if (f0 == 0) {
      if (tr0 < M && j0 < a.r) item.T[tr0 * a.r + j0] = tac[0];
      if (tr0 < M && j0 + 1 < a.r) item.T[tr0 * a.r + j0 + 1] = tac[1];
      if (tr0 + 8 < M && j0 < a.r) item.T[(tr0 + 8) * a.r + j0] = tac[2];
      if (tr0 + 8 < M && j0 + 1 < a.r) item.T[(tr0 + 8) * a.r + j0 + 1] = tac[3];
    }
    const uint32_t row = s_t + static_cast<uint32_t>((16 * tb + g) * rowr(rp) + j0 * 2);
    st_shared32(row, pack2<T16>(__fmul_rn(a.s, tac[0]), __fmul_rn(a.s, tac[1])));
    st_shared32(row + 8 * rowr(rp), pack2<T16>(__fmul_rn(a.s, tac[2]), __fmul_rn(a.s, tac[3])));
  }
  __syncthreads();
  // + (s T) B^T over the rank
  const uint32_t RR = static_cast<uint32_t>(rowr(rp));
#pragma unroll
  for (int kk = 0; kk < 2; ++kk) {
    if (16 * kk >= rp) break;
    const uint32_t b0 = pack2<T16>(bv[kk][0], bv[kk][1]), b1 = pack2<T16>(bv[kk][2], bv[kk][3]);
#pragma unroll
    for (int mb = 0; mb < 2; ++mb) {
      const uint32_t arow2 = s_t + (16 * mb + g) * RR + (16 * kk + 2 * c) * 2;
      const uint32_t a0 = ld_shared32(arow2), a1 = ld_shared32(arow2 + 8 * RR);
      const uint32_t a2 = ld_shared32(arow2 + 16), a3 = ld_shared32(arow2 + 8 * RR + 16);
      mma16816<F16>(acc[mb], a0, a1, a2, a3, b0, b1);
    }
  }
  // y through shared memory (the x rows are no longer read): [32 tokens][64 features] 16-bit
  constexpr int kYRow = 2 * kTF + 16;
#pragma unroll
  for (int mb = 0; mb < 2; ++mb) {
    const uint32_t yrow = s_x + static_cast<uint32_t>((16 * mb + g) * kYRow + (fw + 2 * c) * 2);
    st_shared32(yrow, pack2<T16>(acc[mb][0], acc[mb][1]));
    st_shared32(yrow + 8 * kYRow, pack2<T16>(acc[mb][2], acc[mb][3]));
  }
  __syncthreads();
  T16* y = static_cast<T16*>(item.y);
  for (int i = threadIdx.x; i < kTT * (kTF / 8); i += kThreads) {
    const int r = i / (kTF / 8), ch = i % (kTF / 8);
    if (t0 + r < M && f0 + 8 * ch < N)
      *reinterpret_cast<uint4*>(y + (t0 + r) * N + f0 + 8 * ch) = lds128(s_x + r * kYRow + ch * 16);
  }
}

// ---- backward ---------------------------------------------------------------------------
//
// Kernel small_fused_dx: one CTA per (projection, 32-token tile, 64-input-feature tile).
//   dX tile = dY[32, N] W[N, 64] + s G A[:, 64] with G = dY B over the whole N (recomputed by
//   every input-feature tile of the token tile).  N is taken in chunks of 128 rows: a chunk
//   of W's 64 columns is decoded into shared memory (or copied, when the caller gives the
//   decoded weight) together with its rows of T16(B), while the next chunk's packed codes and
//   B rows are in flight, and both products run over the chunk.
//   The token tile's shares of the adapter gradients go to fp32 workspace slices, unscaled:
//   dA part [r][K] (its 64 columns) = T16(G)^T x over the 32 tokens, and dB part [N][r] (an
//   equal share of W's rows per input-feature tile) = dY^T T16(T).
// The last CTA of each input-feature tile (a ticket counter per tile) then sums that tile's
//   share of dA and dB over the token tiles' parts, in tile order, times s.
// Warps: warp w takes token block w & 1 (16 tokens) and input features 16 (w >> 1) .. + 15.

constexpr int kBT = 32;           // tokens per backward tile
constexpr int kRow64 = 2 * kTF + 16;   // a row of 64 16-bit values, padded

struct BwdUnitItem {
  LinearArgs a;
  const void* dy;    // [M, N] 16-bit
  const void* x;     // [M, K] 16-bit
  const float* T;    // [M, r]
  const float* A;    // [r, K]
  const float* B;    // [N, r]
  const void* w16;   // decoded weight [N, K], or null: decode from a.W
  void* dx;          // [M, K] 16-bit
  float* dA_part;    // [tiles_t][r][K]
  float* dB_part;    // [tiles_t][N][r]
  float* dA;         // [r, K]
  float* dB;         // [N, r]
  unsigned* tickets; // one zero counter per input-feature tile
  int rp, tiles_k, tiles_t;
  int64_t unit0;
};
struct BwdParams {
  BwdUnitItem it[kSmallMaxGroup];
  int n;
  int64_t M;
};

// The contraction over N runs in steps of 16: the weight and B tiles hold N16 = N rounded up to
// 16 rows, and dY's columns N .. N16 - 1, all zero past N.  W's 64 columns and B are taken in
// chunks of kNC rows of N, so that two CTAs fit an SM at the SmolLM2 shapes.
__host__ __device__ inline int64_t n16(int64_t N) { return (N + 15) / 16 * 16; }
constexpr int kNC = 128;

// Shared memory of the backward: dY rows, a chunk of W's 64 columns (16-bit), a chunk of T16(B),
// T16(A) columns, x columns, G (fp32), T16(T), two chunks of B in flight (fp32), and with the
// stored codes all of N's packed columns and block scales.
__host__ __device__ inline int64_t bwd_smem_bytes(int64_t N, int rp, bool w16) {
  const int64_t N16 = n16(N);
  return kBT * row16(N16) + kNC * kRow64 + kNC * rowr(rp) + rp * kRow64 + kBT * kRow64 + kBT * (4 * rp + 16) +
         kBT * rowr(rp) + 2 * kNC * rp * 4 + (w16 ? 0 : N16 * 36);
}

// ldmatrix lane addresses.  A operand (m16 x k16) from [m][k] rows: row (i & 7) + 8 ((i >> 3) & 1),
// column 8 (i >> 4).  A operand from [k][m] rows (.trans): row 8 (i >> 4) + (i & 7), column
// 8 ((i >> 3) & 1).  B operand (k16 x two n8 blocks) from [k][n] rows (.trans): row (i & 7) +
// 8 ((i >> 3) & 1), column 8 (i >> 4).
template <typename T16>
__global__ void __launch_bounds__(kThreads, 2)
small_fused_dx(BwdParams p, DecodeTables tabs) {
  constexpr bool F16 = std::is_same<T16, __half>::value;
  extern __shared__ __align__(16) unsigned char smem[];
  __shared__ float dyn8[256];
  __shared__ BwdUnitItem item;
  for (int i = threadIdx.x; i < 256; i += kThreads) dyn8[i] = tabs.dyn8[i];
  if (threadIdx.x == 0) {
    int k = 0;
    while (k + 1 < p.n && static_cast<int64_t>(blockIdx.x) >= p.it[k + 1].unit0) ++k;
    for (int j = 0; j < kSmallMaxGroup; ++j)
      if (j == k) item = p.it[j];
  }
  __syncthreads();
  pdl_allow_next();
  pdl_wait();
  const LinearArgs& a = item.a;
  const int64_t K = a.K, N = a.N, M = p.M;
  const int rp = item.rp, r = a.r;
  const int64_t local = blockIdx.x - item.unit0;
  const int64_t tt = local / item.tiles_k, kt = local % item.tiles_k;
  const int64_t t0 = tt * kBT, k0 = kt * kTF;
  const int gstride = 4 * rp + 16;         // fp32 G rows
  const int64_t N16 = n16(N);
  const int64_t dys = row16(N16);          // dY row stride
  const int nch = static_cast<int>((N16 + kNC - 1) / kNC);

  const uint32_t s_dy = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
  const uint32_t s_w = s_dy + kBT * dys;                  // W[chunk rows, k0 .. k0 + 63], [kNC][64]
  const uint32_t s_b = s_w + kNC * kRow64;                // B chunk, [kNC][rp]
  const uint32_t s_a = s_b + kNC * rowr(rp);              // A[:, k0 .. +63], [rp][64]
  const uint32_t s_x = s_a + rp * kRow64;                 // x tile, [32][64]
  const uint32_t s_g = s_x + kBT * kRow64;                // G (fp32), [32][rp]
  const uint32_t s_t = s_g + kBT * gstride;               // T (16-bit), [32][rp]
  const uint32_t s_rawb = s_t + kBT * rowr(rp);           // two B chunks in flight, fp32 [2][kNC][rp]
  const uint32_t s_code = s_rawb + 2 * kNC * rp * 4;      // stored codes: packed columns [N16][32 bytes]
  float* s_sc = reinterpret_cast<float*>(smem + (s_code + N16 * 32 - s_dy));   // and block scales [N16]
  const bool dec = item.w16 == nullptr;
  const float* g_f = reinterpret_cast<const float*>(smem + (s_g - s_dy));
  auto raw = [&](uint32_t a) { return reinterpret_cast<const float*>(smem + (a - s_dy)); };
  const int64_t nbr = K / 64;
  auto rows_of = [&](int c) { return static_cast<int>(std::min<int64_t>(kNC, N16 - static_cast<int64_t>(c) * kNC)); };
  // B's rows of chunk c (fp32) into staging buffer c & 1, as one group of copies
  auto issue_b = [&](int c) {
    stage_f32_raw(s_rawb + static_cast<uint32_t>((c & 1) * kNC * rp * 4), item.B, static_cast<int64_t>(c) * kNC,
                  rows_of(c), N, r, rp, r == rp);
    cp_async_commit();
  };
  // with the decoded weight: chunk c's 16-bit columns straight into the chunk buffer
  auto issue_w16 = [&](int c) {
    const T16* w = static_cast<const T16*>(item.w16);
    const int64_t nb0 = static_cast<int64_t>(c) * kNC;
    for (int i = threadIdx.x; i < rows_of(c) * 8; i += kThreads) {
      const int rr = i >> 3, ch = i & 7;
      const uint32_t d = s_w + static_cast<uint32_t>(rr * kRow64 + ch * 16);
      if (nb0 + rr < N) cp_async16(d, w + (nb0 + rr) * K + k0 + 8 * ch);
      else asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};" ::"r"(d), "r"(0u) : "memory");
    }
    cp_async_commit();
  };

  // the copies: dY rows, x columns, all packed columns (or chunk 0 of the decoded weight), then
  // B's chunks 0 and 1; the block scales' inputs, A's columns and T straight into registers
  stage_rows16(s_dy, dys, static_cast<const T16*>(item.dy), t0, kBT, M, N);
  if (N16 > N)   // dY columns N .. N16 - 1 (8 of them) are zero
    for (int i = threadIdx.x; i < kBT; i += kThreads)
      asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};" ::"r"(s_dy + static_cast<uint32_t>(i * dys + 2 * N)),
                   "r"(0u)
                   : "memory");
  {
    const T16* x = static_cast<const T16*>(item.x);
    for (int i = threadIdx.x; i < kBT * 8; i += kThreads) {
      const int rr = i >> 3, ch = i & 7;
      const uint32_t d = s_x + rr * kRow64 + ch * 16;
      if (t0 + rr < M) cp_async16(d, x + (t0 + rr) * K + k0 + 8 * ch);
      else asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};" ::"r"(d), "r"(0u) : "memory");
    }
  }
  if (dec) {
    for (int i = threadIdx.x; i < static_cast<int>(N16) * 2; i += kThreads) {
      const int rr = i >> 1, h = i & 1;
      const uint32_t d = s_code + static_cast<uint32_t>(rr * 32 + h * 16);
      if (rr < N) cp_async16(d, a.W.packed + rr * (K / 2) + k0 / 2 + h * 16);
      else asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};" ::"r"(d), "r"(0u) : "memory");
    }
    cp_async_commit();
  } else {
    issue_w16(0);
  }
  issue_b(0);
  if (nch > 1) issue_b(1);
  constexpr int U = 1024 / kThreads;       // rows per thread (N16 <= 1024)
  uint32_t scode[U];
  float snest[U];
  const float soff = (dec && a.W.dq) ? __ldg(a.W.offset) : 0.0f;
#pragma unroll
  for (int u = 0; u < U; ++u) {
    const int64_t rr = threadIdx.x + u * kThreads;
    scode[u] = 0, snest[u] = 0.0f;
    if (dec && rr < N) {
      if (a.W.dq) {
        scode[u] = __ldg(static_cast<const uint8_t*>(a.W.absmax) + rr * nbr + kt);
        snest[u] = __ldg(a.W.nested + ((rr * nbr + kt) >> 8));
      } else {
        snest[u] = __ldg(static_cast<const float*>(a.W.absmax) + rr * nbr + kt);
      }
    }
  }
  // A's columns [rp][64] (8 a thread at most) and T [32][rp] (4 a thread at most), zero past r / M
  float av[8], tv[4];
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    const int ia = threadIdx.x + u * kThreads, ja = ia / kTF, ca = ia - ja * kTF;
    av[u] = (ia < rp * kTF && ja < r) ? __ldg(item.A + ja * K + k0 + ca) : 0.0f;
  }
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int it = threadIdx.x + u * kThreads, jt = it / rp, ct = it - jt * rp;
    tv[u] = (it < kBT * rp && t0 + jt < M && ct < r) ? __ldg(item.T + (t0 + jt) * r + ct) : 0.0f;
  }
  if (dec)
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int rr = threadIdx.x + u * kThreads;
      if (rr < N16) s_sc[rr] = rr >= N ? 0.0f : a.W.dq ? __fadd_rn(__fmul_rn(dyn8[scode[u]], snest[u]), soff) : snest[u];
    }
  // T16(A) and T16(T), one 16-bit value a store
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    const int ia = threadIdx.x + u * kThreads, ja = ia / kTF, ca = ia - ja * kTF;
    if (ia < rp * kTF) st_shared16<T16>(s_a + static_cast<uint32_t>(ja * kRow64 + 2 * ca), av[u]);
  }
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int it = threadIdx.x + u * kThreads, jt = it / rp, ct = it - jt * rp;
    if (it < kBT * rp) st_shared16<T16>(s_t + static_cast<uint32_t>(jt * rowr(rp) + 2 * ct), tv[u]);
  }
  if (nch > 1) cp_async_wait_group1();   // all but B's chunk 1
  else cp_async_wait_all();
  __syncthreads();

  // warp w: token block mb = w & 1 and input features 16 nq .. 16 nq + 15 (nq = w >> 1) of the
  // tile; G's rank block nq (when 8 nq < rp); the dA part's rank block w & 1 over the same 16
  // features; dB rows in 16-row blocks w, w + 8, ... of this tile's share
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, c = lane & 3;
  const int mb = warp & 1, nq = warp >> 1;
  const int ar = (lane & 7) + 8 * ((lane >> 3) & 1), ac = 8 * (lane >> 4);   // [m][k] A, and [k][n] B
  const int tr = 8 * (lane >> 4) + (lane & 7), tc = 8 * ((lane >> 3) & 1);   // [k][m] A (.trans)
  const uint32_t DYS = static_cast<uint32_t>(dys), RR = static_cast<uint32_t>(rowr(rp));
  const uint32_t dy_a = s_dy + (16 * mb + ar) * DYS + ac * 2;                 // + 2 n
  const uint32_t w_b = s_w + ar * kRow64 + (16 * nq + ac) * 2;                // + n0 kRow64 (chunk row)
  const bool has_g = 8 * nq < rp;
  const uint32_t b_b = s_b + ar * RR + (8 * nq + (ac & 8)) * 2;             // + n0 RR (chunk row)
  float acc[2][4] = {};                    // dX: [feature block of 8][fragment]
  float gac[4] = {};                       // G: rank block nq of the token block
  for (int ch = 0; ch < nch; ++ch) {
    const int64_t nb0 = static_cast<int64_t>(ch) * kNC;
    const int rows = rows_of(ch);
    // chunk ch into the chunk buffers: T16(B) from its staging buffer, and W's columns decoded
    // from the packed columns (two threads a row, the row's 64 columns being exactly one block)
    convert_raw<T16>(s_b, rowr(rp), raw(s_rawb + static_cast<uint32_t>((ch & 1) * kNC * rp * 4)), rows, rp);
    if (dec) {
      const int rr = threadIdx.x >> 1, h = threadIdx.x & 1;
      if (rr < rows) {
        const int64_t n = nb0 + rr;
        const uint32_t d = s_w + static_cast<uint32_t>(rr * kRow64 + h * 64);
        uint32_t L[4], H[4];
        build_lut<T16>(s_sc[n], L, H);   // scale 0 past N: those rows decode to zeros
        const uint4 cw = lds128(s_code + static_cast<uint32_t>(n * 32 + h * 16));
        const uint32_t cws[4] = {cw.x, cw.y, cw.z, cw.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint32_t o[4];
          decode8(cws[q], L, H, o);
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(d + q * 16), "r"(o[0]), "r"(o[1]), "r"(o[2]),
                       "r"(o[3])
                       : "memory");
        }
      }
    }
    __syncthreads();   // the chunk is in place; its B staging buffer is free
    if (ch + 2 < nch) issue_b(ch + 2);   // lands while this chunk and the next are contracted
    const int n16s = rows / 16;
    for (int st = 0; st < n16s; ++st) {
      const uint32_t n0 = static_cast<uint32_t>(16 * st);
      uint32_t a0, a1, a2, a3, b0, b1, b2, b3;
      ldsm4(dy_a + 2 * (static_cast<uint32_t>(nb0) + n0), a0, a1, a2, a3);
      ldsm4t(w_b + n0 * kRow64, b0, b1, b2, b3);
      mma16816<F16>(acc[0], a0, a1, a2, a3, b0, b1);
      mma16816<F16>(acc[1], a0, a1, a2, a3, b2, b3);
      if (has_g) {                           // the x4's second column pair is not used
        ldsm4t(b_b + n0 * RR, b0, b1, b2, b3);
        mma16816<F16>(gac, a0, a1, a2, a3, b0, b1);
      }
    }
    if (ch + 1 < nch) {
      __syncthreads();   // every warp is done with the chunk buffers
      if (!dec) {
        issue_w16(ch + 1);
        cp_async_wait_all();
      } else if (ch + 2 < nch) {
        cp_async_wait_group1();   // B's chunk ch + 1 has landed; chunk ch + 2 may be in flight
      } else {
        cp_async_wait_all();
      }
      __syncthreads();
    }
  }
  // G, fp32, to shared memory: every warp of a token block needs all of its ranks
  if (has_g) {
    float* row = reinterpret_cast<float*>(smem + (s_g - s_dy) + (16 * mb + g) * gstride) + 8 * nq + 2 * c;
    row[0] = gac[0];
    row[1] = gac[1];
    row[8 * gstride / 4] = gac[2];
    row[8 * gstride / 4 + 1] = gac[3];
  }
  __syncthreads();
  const int gs4 = gstride / 4;
  // dX += (s G) A over the rank (A operand: T16(s G) of the warp's 16 tokens)
#pragma unroll
  for (int kk = 0; kk < 2; ++kk) {
    if (16 * kk >= rp) break;
    const float* gr = g_f + (16 * mb + g) * gs4 + 16 * kk + 2 * c;
    const float* gr8 = gr + 8 * gs4;
    const uint32_t a0 = pack2<T16>(__fmul_rn(a.s, gr[0]), __fmul_rn(a.s, gr[1]));
    const uint32_t a1 = pack2<T16>(__fmul_rn(a.s, gr8[0]), __fmul_rn(a.s, gr8[1]));
    const uint32_t a2 = pack2<T16>(__fmul_rn(a.s, gr[8]), __fmul_rn(a.s, gr[9]));
    const uint32_t a3 = pack2<T16>(__fmul_rn(a.s, gr8[8]), __fmul_rn(a.s, gr8[9]));
    uint32_t b0, b1, b2, b3;
    ldsm4t(s_a + static_cast<uint32_t>((16 * kk + ar) * kRow64 + (16 * nq + ac) * 2), b0, b1, b2, b3);
    mma16816<F16>(acc[0], a0, a1, a2, a3, b0, b1);
    mma16816<F16>(acc[1], a0, a1, a2, a3, b2, b3);
  }
  // dA part [r][this tile's 64 columns] = T16(G)^T x over the 32 tokens: rank block w & 1, the
  // warp's 16 columns
  if (16 * mb < rp) {
    float da[2][4] = {};
#pragma unroll
    for (int kk = 0; kk < kBT / 16; ++kk) {   // tokens 16 kk .. + 15
      const float* gc = g_f + (16 * kk + 2 * c) * gs4 + 16 * mb + g;
      const uint32_t a0 = pack2<T16>(gc[0], gc[gs4]);
      const uint32_t a1 = pack2<T16>(gc[8], gc[gs4 + 8]);
      const uint32_t a2 = pack2<T16>(gc[8 * gs4], gc[9 * gs4]);
      const uint32_t a3 = pack2<T16>(gc[8 * gs4 + 8], gc[9 * gs4 + 8]);
      uint32_t b0, b1, b2, b3;
      ldsm4t(s_x + static_cast<uint32_t>((16 * kk + ar) * kRow64 + (16 * nq + ac) * 2), b0, b1, b2, b3);
      mma16816<F16>(da[0], a0, a1, a2, a3, b0, b1);
      mma16816<F16>(da[1], a0, a1, a2, a3, b2, b3);
    }
    float* part = item.dA_part + tt * r * K;
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int64_t col = k0 + 16 * nq + 8 * j + 2 * c;
      const int row = 16 * mb + g;
      if (row < r) part[row * K + col] = da[j][0], part[row * K + col + 1] = da[j][1];
      if (row + 8 < r) part[(row + 8) * K + col] = da[j][2], part[(row + 8) * K + col + 1] = da[j][3];
    }
  }
  // dB part [N][r], this tile's share of the rows: dY^T T16(T) over the 32 tokens
  {
    const int64_t blocks = N16 / 16;
    const int64_t per = (blocks + item.tiles_k - 1) / item.tiles_k;
    const int64_t b_lo = kt * per, b_hi = std::min<int64_t>(blocks, b_lo + per);
    float* part = item.dB_part + tt * N * r;
    for (int64_t bk = b_lo + warp; bk < b_hi; bk += kWarps) {
      float db[4][4] = {};                   // [rank block of 8][fragment]
#pragma unroll
      for (int kk = 0; kk < kBT / 16; ++kk) {
        uint32_t a0, a1, a2, a3;             // A[m = n][k = token] from dY [token][n]
        ldsm4t(s_dy + static_cast<uint32_t>((16 * kk + tr) * dys + (16 * bk + tc) * 2), a0, a1, a2, a3);
#pragma unroll
        for (int q2 = 0; q2 < 2; ++q2) {
          if (16 * q2 >= rp) break;
          uint32_t b0, b1, b2, b3;
          ldsm4t(s_t + static_cast<uint32_t>((16 * kk + ar) * rowr(rp) + (16 * q2 + ac) * 2), b0, b1, b2, b3);
          mma16816<F16>(db[2 * q2], a0, a1, a2, a3, b0, b1);
          mma16816<F16>(db[2 * q2 + 1], a0, a1, a2, a3, b2, b3);
        }
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        if (8 * q >= rp) break;
        const int64_t row = 16 * bk + g;
        const int col = 8 * q + 2 * c;
        if (row < N && col < r) part[row * r + col] = db[q][0];
        if (row < N && col + 1 < r) part[row * r + col + 1] = db[q][1];
        if (row + 8 < N && col < r) part[(row + 8) * r + col] = db[q][2];
        if (row + 8 < N && col + 1 < r) part[(row + 8) * r + col + 1] = db[q][3];
      }
    }
  }
  // the last CTA of this input-feature tile (over the token tiles) finishes the tile's share of
  // the adapter gradients: dA[:, k0 .. k0 + 63] and dB over its rows, s times the sum of the
  // parts in token-tile order (the pattern of a grid barrier's arrival: the CTA's threads meet,
  // thread 0 fences and counts)
  __shared__ unsigned s_last;
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    s_last = (atomicAdd(item.tickets + kt, 1u) == static_cast<unsigned>(item.tiles_t - 1)) ? 1u : 0u;
  }
  __syncthreads();
  if (s_last != 0) {
    __threadfence();
    const int64_t blocks = N16 / 16;
    const int64_t per = (blocks + item.tiles_k - 1) / item.tiles_k;
    const int64_t n_lo = std::min<int64_t>(N, kt * per * 16), n_hi = std::min<int64_t>(N, (kt * per + per) * 16);
    const int T = item.tiles_t;
    // dA's block: r rows of 64 columns as float4 groups; dB's rows: float4 groups when r % 4 == 0
    const bool vb = (r % 4) == 0;
    const int gA = r * (kTF / 4);
    const int gB = static_cast<int>(n_hi - n_lo) * (vb ? r / 4 : r);
    for (int e = threadIdx.x; e < gA + gB; e += kThreads) {
      const float* part;
      int64_t stride;
      float* out;
      bool v4 = true;
      if (e < gA) {
        const int j = e / (kTF / 4), c4 = e - j * (kTF / 4);
        part = item.dA_part + j * K + k0 + 4 * c4;
        stride = static_cast<int64_t>(r) * K;
        out = item.dA + j * K + k0 + 4 * c4;
      } else {
        const int64_t i = n_lo * r + (vb ? 4 * (e - gA) : (e - gA));
        part = item.dB_part + i;
        stride = N * r;
        out = item.dB + i;
        v4 = vb;
      }
      // the sums in token-tile order; each group of 16 tiles' loads is issued before its adds
      float4 sum = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
      for (int t0 = 0; t0 < T; t0 += 16) {
        float4 v[16];
#pragma unroll
        for (int u = 0; u < 16; ++u) {
          if (t0 + u >= T) break;
          const float* q = part + (t0 + u) * stride;
          v[u] = v4 ? __ldcg(reinterpret_cast<const float4*>(q)) : make_float4(__ldcg(q), 0.0f, 0.0f, 0.0f);
        }
#pragma unroll
        for (int u = 0; u < 16; ++u) {
          if (t0 + u >= T) break;
          sum.x += v[u].x, sum.y += v[u].y, sum.z += v[u].z, sum.w += v[u].w;
        }
      }
      if (v4) {
        *reinterpret_cast<float4*>(out) = make_float4(__fmul_rn(a.s, sum.x), __fmul_rn(a.s, sum.y),
                                                      __fmul_rn(a.s, sum.z), __fmul_rn(a.s, sum.w));
      } else {
        *out = __fmul_rn(a.s, sum.x);
      }
    }
    if (threadIdx.x == 0) item.tickets[kt] = 0u;
  }
  // dX through shared memory (the dY rows are no longer read after this barrier)
  __syncthreads();
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const uint32_t row = s_dy + static_cast<uint32_t>((16 * mb + g) * kRow64 + (16 * nq + 8 * j + 2 * c) * 2);
    st_shared32(row, pack2<T16>(acc[j][0], acc[j][1]));
    st_shared32(row + 8 * kRow64, pack2<T16>(acc[j][2], acc[j][3]));
  }
  __syncthreads();
  T16* dx = static_cast<T16*>(item.dx);
  for (int i = threadIdx.x; i < kBT * 8; i += kThreads) {
    const int rr = i >> 3, ch = i & 7;
    if (t0 + rr < M) *reinterpret_cast<uint4*>(dx + (t0 + rr) * K + k0 + 8 * ch) = lds128(s_dy + rr * kRow64 + ch * 16);
  }
}

}  // namespace

size_t small_fused_bwd_ws_bytes(const SmallItem* items, int n, int64_t M) {
  size_t b = 0;
  const int64_t tiles_t = (M + kBT - 1) / kBT;
  for (int i = 0; i < n; ++i) {
    const LinearArgs& a = items[i].a;
    b += (static_cast<size_t>(tiles_t) * (a.r * a.K + a.N * a.r) * sizeof(float) + 255) / 256 * 256;
  }
  return b;
}

cudaError_t small_fused_backward(const SmallItem* items, int n, int64_t M, bool f16, void* ws, cudaStream_t st) {
  if (n < 1 || n > kSmallMaxGroup || M < 1) return cudaErrorInvalidValue;
  BwdParams p{};
  p.n = n;
  p.M = M;
  const int64_t tiles_t = (M + kBT - 1) / kBT;
  int64_t units = 0, smem = 0;
  char* w = static_cast<char*>(ws);
  for (int i = 0; i < n; ++i) {
    const SmallItem& s = items[i];
    BwdUnitItem& it = p.it[i];
    it.a = s.a;
    it.dy = s.dy;
    it.x = s.x;
    it.T = s.T;
    it.A = s.A;
    it.B = s.B;
    it.w16 = s.w16;
    it.dx = s.dx;
    it.rp = (s.a.r + 15) / 16 * 16;
    it.tiles_k = static_cast<int>(s.a.K / kTF);
    it.unit0 = units;
    it.dA_part = reinterpret_cast<float*>(w);
    it.dB_part = it.dA_part + tiles_t * s.a.r * s.a.K;
    it.dA = s.dA;
    it.dB = s.dB;
    it.tiles_t = static_cast<int>(tiles_t);
    if (cudaError_t te = ticket_range(static_cast<unsigned>(s.a.K / kTF), &it.tickets); te != cudaSuccess) return te;
    w += (static_cast<size_t>(tiles_t) * (s.a.r * s.a.K + s.a.N * s.a.r) * sizeof(float) + 255) / 256 * 256;
    units += tiles_t * it.tiles_k;
    smem = std::max(smem, bwd_smem_bytes(s.a.N, it.rp, s.w16 != nullptr));
  }
  if (units > 0x7FFFFFFFLL) return cudaErrorInvalidValue;
  auto kern = f16 ? small_fused_dx<__half> : small_fused_dx<__nv_bfloat16>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  e = launch_pdl(kern, dim3(static_cast<unsigned>(units)), dim3(kThreads), static_cast<size_t>(smem), st, 1, p,
                 decode_tables());
  note_launch();
  return e;
}

bool small_fused_fits(int64_t N, int64_t K, int r) {
  const int rp = (r + 15) / 16 * 16;
  return K % 64 == 0 && N % 8 == 0 && K <= 1024 && N <= 1024 && N * K <= (int64_t(1) << 21) && rp <= 32 &&
         std::max(fwd_smem_bytes(K, rp, true), fwd_smem_bytes(K, rp, false)) <= 200 * 1024 &&
         std::max(bwd_smem_bytes(N, rp, true), bwd_smem_bytes(N, rp, false)) <= 200 * 1024;
}

cudaError_t small_fused_forward(const SmallItem* items, int n, int64_t M, bool f16, cudaStream_t st) {
  if (n < 1 || n > kSmallMaxGroup || M < 1) return cudaErrorInvalidValue;
  FwdParams p{};
  p.n = n;
  p.M = M;
  int64_t units = 0, smem = 0;
  for (int i = 0; i < n; ++i) {
    FwdUnitItem& it = p.it[i];
    it.a = items[i].a;
    it.x = items[i].x;
    it.A = items[i].A;
    it.B = items[i].B;
    it.y = items[i].y;
    it.T = items[i].T;
    it.w16 = items[i].w16;
    it.rp = (it.a.r + 15) / 16 * 16;
    it.tiles_f = static_cast<int>((it.a.N + kTF - 1) / kTF);
    it.unit0 = units;
    units += ((M + kTT - 1) / kTT) * it.tiles_f;
    smem = std::max(smem, fwd_smem_bytes(it.a.K, it.rp, it.w16 != nullptr));
  }
  if (units > 0x7FFFFFFFLL) return cudaErrorInvalidValue;
  auto kern = f16 ? small_fused_fwd<__half> : small_fused_fwd<__nv_bfloat16>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  e = launch_pdl(kern, dim3(static_cast<unsigned>(units)), dim3(kThreads), static_cast<size_t>(smem), st, 1, p,
                 decode_tables());
  note_launch();
  return e;
}

}  // namespace qnf4
