// Small-M forward of the bf16 QLoRA linear (M <= 16 tokens), for one projection or a group
// of up to 8 projections in two launches:
//     T = x A^T,   y = x deq(W)^T + s T B^T
// ("Native model adaptation and NF4", sections "Packed NF4 and the portable QLoRA profile"
// and "Fused GPU NF4 decodes inside the matrix kernel": the weight is decoded on the device
// inside the kernel that consumes it; "Mixed precision keeps stable state in FP32": adapter
// contractions accumulate in FP32.)
//
// With a handful of tokens the forward is bound by reading the stored weight (0.516 bytes per
// weight) and by decoding it; the weight is read exactly once and never written back decoded:
//
// lora_down_small (one CTA per rank row j of each projection): T[m][j] = sum_k x[m][k] *
//   bf16(A[j][k]) in fp32, per-thread partial sums reduced with warp shuffles and then across
//   warps in a fixed order; writes T and bf16(s T) (the LoRA term's token-side operand, padded
//   with zeros to 16 tokens and a multiple of 64 ranks).  It also clears the split-tile tickets.
//
// nf4_stream_fwd (persistent, one CTA per SM): the work is the list of units (projection,
//   256-row tile, 256-deep span of the contraction), cut into equal contiguous ranges, one per
//   CTA (stream-K), so every CTA streams the same number of weight bytes.  Warp 0 copies each
//   unit's packed codes (256 rows x 128 bytes) and the unit's slice of x (16 tokens x 256) into
//   a 4-stage ring by TMA (128-byte swizzled boxes).  Warps 1..8 each own 32 rows of the tile:
//   per 64-element block a thread builds the 16-entry table of bf16(nf4[q] * a') in registers
//   (a' = dyn8[code] * nested + offset, loaded one unit ahead), turns its code bytes into bf16
//   pairs with byte permutes and feeds them, without any further copy, as the A fragments of
//   mma.sync m16n8k16 (fp32 accumulation) against x fragments read from shared memory.
//   A tile's segment that holds its first span also adds the LoRA term as extra 16-rank MMA
//   steps into the same accumulators: bf16(B[row][j]) against bf16(s T).  A tile processed by
//   one CTA is stored from its accumulators; a tile split between CTAs leaves fp32 partial sums,
//   and after its last unit each CTA takes a ticket per split tile: the CTA that draws the last
//   ticket adds the parts in CTA order (deterministic) and stores the tile.  No CTA waits for
//   another.
//
// Why mma.sync and not tcgen05 here: a tcgen05.mma occupies an SM's tensor core for the same
// time whatever its N (measured on this GPU: ~97 ns for M = 128, K = 16 and any N from 16 to
// 256), so with 16 tokens a weight pass built on it is capped by the instruction count (one
// per 2048 weights); the warp-level MMA consumes the decoded fragments straight from registers
// at a cost that scales with the work, and the pass is bound by the byte-permute decode.
//
// The stream kernel is launched as a programmatic dependent of lora_down_small, which lets it
// start as soon as lora_down_small's CTAs have started: x and the weight are ready by then; the
// only data it takes from lora_down_small (bf16(s T) and the cleared tickets) is read after
// griddepcontrol.wait, at the end of a tile's first segment.  Every mbarrier wait is bounded; a
// timeout sets NF4_ERR_TIMEOUT in the status word and the CTA winds down.
#include <algorithm>
#include <mutex>
#include <type_traits>

#include <cuda_fp16.h>

#include "decode.cuh"
#include "mma_sync.cuh"
#include "linear_tc.cuh"
#include "tc_ptx.cuh"

namespace qnf4 {
namespace {

using namespace tc;

constexpr int kTok = 16;                          // tokens per unit: two 8-token MMA tiles
constexpr int kTileRows = 256;                    // weight rows per tile
constexpr int kBoxRows = 128;                     // rows per TMA box of codes
constexpr int kSpan = 256;                        // contraction per unit: four 64-element blocks
constexpr int kSpanBytes = kSpan / 2;             // packed code bytes per row per unit
constexpr int kCodeBox = kBoxRows * kSpanBytes;   // 16 KB
constexpr int kXBox = kTok * 64 * 2;              // 2 KB: [16 tokens][64] bf16
constexpr int kStageBytes = 2 * kCodeBox + 4 * kXBox;   // 40 KB
constexpr int kStages = 4;
constexpr int kDecWarps = 16;                     // 16 rows each
constexpr int kThreads = 32 * (1 + kDecWarps);    // warp 0 TMA, warps 1..16 decode + MMA
constexpr int kMaxGroup = kStreamMaxGroup;
constexpr int kMaxCtas = 256;
constexpr int kAccPerThread = 8;                  // 2 token tiles x 4
constexpr size_t kPartBytesPerCta = 2ull * kDecWarps * 32 * kAccPerThread * sizeof(float);   // 2 slots

constexpr int kBarFull = 0, kBarEmpty = kStages, kNumBars = 2 * kStages;
constexpr int kSmemBytes = 1024 + kStages * kStageBytes + 256 * 4 + kNumBars * 8 + 64;
static_assert(kSmemBytes <= 232448, "shared memory per CTA");
static_assert(kStageBytes % 1024 == 0, "swizzled boxes stay 1024-byte aligned");

struct StreamProj {
  const uint8_t* absmax;   // dq: uint8 codes, else float
  const float* nested;
  const float* offset;
  const float* B;          // [N][r] fp32
  const void* sT;          // [16][rp64] 16-bit s T, written by lora_down_small
  void* y;                 // [M][N] 16-bit
  int64_t N, K;
  int64_t unit0;           // first unit of this projection
  int r, rp64;
  int tiles, spans, nbr;   // ceil(N/256), ceil(K/256), K/64
  int tile0;               // first global tile (tickets)
  int dq;
};

struct StreamParams {
  StreamProj proj[kMaxGroup];
  float dyn8[256];
  int G;
  int M;
  int64_t units;
  int ctas;
  float* part;             // [ctas][slot 2][decoder thread 512][8] fp32
  int* tickets;            // [tiles]
  int* status;
  uint64_t wait_ns;
  int skip_stage0;
};

struct StreamMaps {
  CUtensorMap codes[kMaxGroup];   // uint8 [N][K/2], box [128 rows][128 bytes]
  CUtensorMap x[kMaxGroup];       // 16-bit [M][K], box [16][64]
};

struct Pos {
  int proj, tile, span;
};

__device__ __forceinline__ Pos pos_of(const StreamParams& p, int64_t u) {
  int i = 0;
  while (i + 1 < p.G && u >= p.proj[i + 1].unit0) ++i;
  const int64_t local = u - p.proj[i].unit0;
  Pos q;
  q.proj = i;
  q.tile = static_cast<int>(local / p.proj[i].spans);
  q.span = static_cast<int>(local - static_cast<int64_t>(q.tile) * p.proj[i].spans);
  return q;
}

// The unit after `q` in the work order (projection, tile, span).
__device__ __forceinline__ Pos advance(const StreamParams& p, Pos q) {
  if (++q.span == p.proj[q.proj].spans) {
    q.span = 0;
    if (++q.tile == p.proj[q.proj].tiles) q.tile = 0, ++q.proj;
  }
  return q;
}

// CTA whose range [floor(c U / P), floor((c+1) U / P)) holds unit u.
__device__ __forceinline__ int cta_of(int64_t u, int64_t U, int P) { return static_cast<int>((u * P + P - 1) / U); }
__device__ __forceinline__ int64_t range_begin(int c, int64_t U, int P) { return (static_cast<int64_t>(c) * U) / P; }

// The inputs of one block scale a' (one weight row, one 64-element block), loaded one unit
// ahead of their use: the absmax code (or fp32 maximum), the nested maximum and the offset.
struct ScaleIn {
  float nested_or_max;
  float offset;
  uint32_t code;
  int live;          // the block lies inside the tensor
};

__device__ __forceinline__ ScaleIn load_scale(const StreamProj& P, int64_t row, int64_t kb) {
  ScaleIn in{};
  in.live = row < P.N && kb < P.nbr;
  if (!in.live) return in;
  const int64_t g = row * P.nbr + kb;
  if (P.dq) {
    in.code = __ldg(P.absmax + g);
    in.nested_or_max = __ldg(P.nested + (g >> 8));
    in.offset = __ldg(P.offset);
  } else {
    in.nested_or_max = __ldg(reinterpret_cast<const float*>(P.absmax) + g);
  }
  return in;
}

// a' = dyn8[code] * nested + offset with two roundings, or the fp32 maximum; 0 outside.
__device__ __forceinline__ float scale_of(const ScaleIn& in, int dq, const float* dyn8) {
  if (!in.live) return 0.0f;
  if (!dq) return in.nested_or_max;
  return __fadd_rn(__fmul_rn(dyn8[in.code], in.nested_or_max), in.offset);
}

// Decoder thread layout.  Warp w (0..15) owns tile rows 16w .. 16w+15; in the mma.sync fragments
// thread (g = lane / 4, c = lane % 4) holds rows g and g+8 of them and, within every unit, the four contraction slots {2c, 2c+1, 2c+8, 2c+9} of each 16-deep
// step come from the unit's block c: at step pair j the thread decodes word (j + 2c) % 8 (eight
// weights) of block c of each of its rows, and takes x of its token g at the same eight
// positions (one 16-byte load, the two steps' b fragments).  The order of the contraction is
// thereby permuted identically for the weights and x.  The rotation by 2c keeps the eight lanes
// of each shared-memory phase on distinct banks.  One table of bf16(nf4[q] * a') serves each
// thread's 64 weights of one row and block.

template <int NT, typename T16>   // 8-token MMA tiles: 1 (M <= 8) or 2 (M <= 16); bf16 or IEEE half
__global__ void __launch_bounds__(kThreads, 1)
nf4_stream_fwd(const __grid_constant__ StreamMaps maps, const __grid_constant__ StreamParams p) {
  constexpr bool F16 = sizeof(T16) == 2 && !std::is_same<T16, __nv_bfloat16>::value;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* base_ptr = smem_raw + (base - raw);
  float* dyn8 = reinterpret_cast<float*>(base_ptr + kStages * kStageBytes);
  uint64_t* bars = reinterpret_cast<uint64_t*>(dyn8 + 256);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + kNumBars);
  volatile int* vote = abort_flag + 1;
  volatile int* ticket_flag = abort_flag + 2;
  auto bar = [&](int i) { return smem_u32(bars + i); };
  auto stage_code = [&](int s) { return base + s * kStageBytes; };
  auto stage_x = [&](int s) { return base + s * kStageBytes + 2 * kCodeBox; };

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  for (int i = threadIdx.x; i < 256; i += kThreads) dyn8[i] = p.dyn8[i];
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar(kBarFull + s), 1);
      mbar_init(bar(kBarEmpty + s), kDecWarps);
    }
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  pdl_allow_next();

  const int64_t U = p.units;
  const int nctas = p.ctas;
  const int cta = blockIdx.x;
  const int64_t ua = range_begin(cta, U, nctas), ub = range_begin(cta + 1, U, nctas);

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      bool ok = true;
      int s = 0, issued = 0;
      uint32_t ph = 0;
      Pos cur = pos_of(p, ua);
      for (int64_t u = ua; ok && u < ub; ++u) {
        if (!mbar_wait(bar(kBarEmpty + s), ph ^ 1u, abort_flag, p.status, p.wait_ns)) { ok = false; break; }
        if (!(p.skip_stage0 && cta == 0 && u == ua)) {   // (tests of the timeout path leave it unissued)
          mbar_expect_tx(bar(kBarFull + s), kStageBytes);
          for (int h = 0; h < 2; ++h)
            tma_load_2d(stage_code(s) + h * kCodeBox, &maps.codes[cur.proj], bar(kBarFull + s), cur.span * kSpanBytes,
                        cur.tile * kTileRows + h * kBoxRows);
          for (int c = 0; c < 4; ++c)
            tma_load_2d(stage_x(s) + c * kXBox, &maps.x[cur.proj], bar(kBarFull + s), cur.span * kSpan + c * 64, 0);
        }
        ++issued;
        if (++s == kStages) s = 0, ph ^= 1u;
        cur = advance(p, cur);
      }
      // every stage issued is consumed before the CTA exits; after a timeout, let the copies
      // in flight land first
      if (!ok || *abort_flag) {
        for (int q = 0; q < issued && q < kStages; ++q) {
          if (s == 0) s = kStages - 1, ph ^= 1u;
          else --s;
          mbar_drain(bar(kBarFull + s), ph);
        }
      }
    }
  } else {
    // ---------------- decoders: decode in registers, mma.sync ----------------
    const int w = warp - 1;
    const int g = lane >> 2, c = lane & 3;
    const int dthread = w * 32 + lane;               // 0..511 among the decoders
    bool ok = true;
    int s = 0, seg_s0 = 0;
    uint32_t ph = 0;
    bool waited = false;                             // griddepcontrol.wait done
    int n_pend = 0, pend_proj0 = 0, pend_tile0 = 0, pend_proj1 = 0, pend_tile1 = 0;
    float acc[NT][4];
    Pos cur = pos_of(p, ua);
    // rows of this thread within the tile: r8 = 0 (row g) or 1 (row g + 8) of the warp's 16
    auto trow = [&](int r8) { return 16 * w + 8 * r8 + g; };
    // byte offset of each of the thread's rows inside a stage's codes (box, row in box)
    uint32_t rowoff[2];
#pragma unroll
    for (int r8 = 0; r8 < 2; ++r8) {
      const uint32_t row = static_cast<uint32_t>(trow(r8));
      rowoff[r8] = (row >> 7) * kCodeBox + (row & 127u) * 128u;
    }
    // per step pair j: word (j + 2c) % 8 of block c, as an offset inside a row of codes (the
    // 16-byte chunk swizzled by the row, row & 7 == g) and as the x chunk of token g
    uint32_t coff[8], xoff[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const uint32_t wd = static_cast<uint32_t>((j + 2 * c) & 7);
      coff[j] = (((2u * c + (wd >> 2)) ^ static_cast<uint32_t>(g)) << 4) | ((wd & 3u) << 2);
      xoff[j] = (wd ^ static_cast<uint32_t>(g)) << 4;
    }
    ScaleIn nxt[2];
    {
      const StreamProj& P = p.proj[cur.proj];
#pragma unroll
      for (int r8 = 0; r8 < 2; ++r8)
        nxt[r8] = load_scale(P, static_cast<int64_t>(cur.tile) * kTileRows + trow(r8), static_cast<int64_t>(cur.span) * 4 + c);
    }
    for (int64_t u = ua; ok && u < ub; ++u) {
      const bool first = u == ua || cur.span == 0;
      const StreamProj& P = p.proj[cur.proj];
      const bool last = u + 1 == ub || cur.span == P.spans - 1;
      if (first) {
        seg_s0 = cur.span;
#pragma unroll
        for (int t = 0; t < NT; ++t)
#pragma unroll
          for (int i = 0; i < 4; ++i) acc[t][i] = 0.0f;
      }
      // this unit's tables from the scale inputs loaded one unit ago; the next unit's inputs
      uint32_t Lt[2][4], Ht[2][4];
#pragma unroll
      for (int r8 = 0; r8 < 2; ++r8) build_lut<T16>(scale_of(nxt[r8], P.dq, dyn8), Lt[r8], Ht[r8]);
      if (u + 1 < ub) {
        const Pos nx = advance(p, cur);
        const StreamProj& Q = p.proj[nx.proj];
#pragma unroll
        for (int r8 = 0; r8 < 2; ++r8)
          nxt[r8] = load_scale(Q, static_cast<int64_t>(nx.tile) * kTileRows + trow(r8), static_cast<int64_t>(nx.span) * 4 + c);
      }
      if (!mbar_wait(bar(kBarFull + s), ph, abort_flag, p.status, p.wait_ns)) { ok = false; break; }
      const uint32_t cb0 = stage_code(s) + rowoff[0], cb1 = stage_code(s) + rowoff[1];
      const uint32_t xbase = stage_x(s) + c * kXBox + g * 128;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        uint4 xb[NT];
#pragma unroll
        for (int t = 0; t < NT; ++t) xb[t] = ld_shared16(xbase + t * 1024 + xoff[j]);
        uint32_t o[2][4];
        decode8(ld_shared32(cb0 + coff[j]), Lt[0], Ht[0], o[0]);
        decode8(ld_shared32(cb1 + coff[j]), Lt[1], Ht[1], o[1]);
#pragma unroll
        for (int t = 0; t < NT; ++t) {
          mma16816<F16>(acc[t], o[0][0], o[1][0], o[0][1], o[1][1], xb[t].x, xb[t].y);
          mma16816<F16>(acc[t], o[0][2], o[1][2], o[0][3], o[1][3], xb[t].z, xb[t].w);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kBarEmpty + s));
      if (++s == kStages) s = 0, ph ^= 1u;
      if (last) {
        const int64_t row0 = static_cast<int64_t>(cur.tile) * kTileRows;
        if (seg_s0 == 0) {
          // the LoRA term, s T B^T: T16(B[row][j]) against T16(s T)[token][j] of
          // lora_down_small, 16 ranks per step
          if (!waited) {
            pdl_wait();
            waited = true;
          }
          for (int j0 = 0; j0 < P.r; j0 += 16) {
            uint32_t a[2][2];   // [r8][lo, hi slot pair]
#pragma unroll
            for (int r8 = 0; r8 < 2; ++r8) {
              const int64_t row = row0 + trow(r8);
              const float* brow = P.B + row * P.r;
              const bool live = row < P.N;
#pragma unroll
              for (int hp = 0; hp < 2; ++hp) {
                const int jj = j0 + 2 * c + 8 * hp;
                a[r8][hp] = pack2<T16>(live && jj < P.r ? __ldg(brow + jj) : 0.0f,
                                       live && jj + 1 < P.r ? __ldg(brow + jj + 1) : 0.0f);
              }
            }
#pragma unroll
            for (int t = 0; t < NT; ++t) {
              const uint32_t* st_row =
                  reinterpret_cast<const uint32_t*>(static_cast<const uint16_t*>(P.sT) + (8 * t + g) * P.rp64 + j0 + 2 * c);
              mma16816<F16>(acc[t], a[0][0], a[1][0], a[0][1], a[1][1], __ldcg(st_row), __ldcg(st_row + 4));
            }
          }
        }
        const bool whole = seg_s0 == 0 && cur.span == P.spans - 1;
        if (whole) {
#pragma unroll
          for (int r8 = 0; r8 < 2; ++r8) {
            const int64_t row = row0 + trow(r8);
            if (row < P.N) {
#pragma unroll
              for (int t = 0; t < NT; ++t)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                  const int m = 8 * t + 2 * c + e;
                  if (m < p.M) store16(static_cast<T16*>(P.y), static_cast<int64_t>(m) * P.N + row, acc[t][2 * r8 + e]);
                }
            }
          }
        } else {
          const int slot = (u - (cur.span - seg_s0) == ua) ? 0 : 1;   // the CTA's first segment, or not
          float4* dst = reinterpret_cast<float4*>(
              p.part + ((static_cast<int64_t>(cta) * 2 + slot) * (kDecWarps * 32) + dthread) * kAccPerThread);
#pragma unroll
          for (int t = 0; t < 2; ++t)
            dst[t] = t < NT ? make_float4(acc[t][0], acc[t][1], acc[t][2], acc[t][3]) : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
          if (n_pend == 0) pend_proj0 = cur.proj, pend_tile0 = cur.tile;
          else pend_proj1 = cur.proj, pend_tile1 = cur.tile;
          n_pend = min(n_pend + 1, 2);
        }
      }
      cur = advance(p, cur);
    }
    // tickets of the split tiles: every decoder warp reaches this point, whether its loop ended
    // normally or gave up, and all take the same path after the vote
    __threadfence();
    named_sync(1, kDecWarps * 32);
    if (dthread == 0) *vote = *abort_flag;
    named_sync(1, kDecWarps * 32);
    if (*vote == 0 && n_pend > 0) {
      if (!waited) pdl_wait();   // the tickets were cleared by lora_down_small
      for (int k = 0; k < n_pend; ++k) {
        const int pproj = k == 0 ? pend_proj0 : pend_proj1, ptile = k == 0 ? pend_tile0 : pend_tile1;
        const StreamProj& P = p.proj[pproj];
        int* ticket = p.tickets + P.tile0 + ptile;
        const int64_t u0 = P.unit0 + static_cast<int64_t>(ptile) * P.spans;
        const int c0 = cta_of(u0, U, nctas), c1 = cta_of(u0 + P.spans - 1, U, nctas);
        if (dthread == 0) *ticket_flag = (atomicAdd(ticket, 1) == c1 - c0) ? 1 : 0;
        named_sync(1, kDecWarps * 32);
        if (*ticket_flag == 1) {
          __threadfence();
          float v[kAccPerThread];
#pragma unroll
          for (int i = 0; i < kAccPerThread; ++i) v[i] = 0.0f;
          for (int jc = c0; jc <= c1; ++jc) {   // parts in CTA order = contraction order
            const int slot = (jc == c0 && range_begin(jc, U, nctas) < u0) ? 1 : 0;
            const float4* src = reinterpret_cast<const float4*>(
                p.part + ((static_cast<int64_t>(jc) * 2 + slot) * (kDecWarps * 32) + dthread) * kAccPerThread);
#pragma unroll
            for (int i = 0; i < 2; ++i) {
              const float4 t4 = __ldcg(src + i);
              v[4 * i] += t4.x, v[4 * i + 1] += t4.y, v[4 * i + 2] += t4.z, v[4 * i + 3] += t4.w;
            }
          }
          const int64_t row0 = static_cast<int64_t>(ptile) * kTileRows;
#pragma unroll
          for (int r8 = 0; r8 < 2; ++r8) {
            const int64_t row = row0 + trow(r8);
            if (row < P.N) {
#pragma unroll
              for (int t = 0; t < NT; ++t)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                  const int m = 8 * t + 2 * c + e;
                  if (m < p.M) store16(static_cast<T16*>(P.y), static_cast<int64_t>(m) * P.N + row, v[4 * t + 2 * r8 + e]);
                }
            }
          }
          if (dthread == 0) *ticket = 0;
        }
        named_sync(1, kDecWarps * 32);
      }
    }
  }
}

// ---- T = x A^T for the small-M forward ----------------------------------------------------

struct DownItem {
  const void* x;            // 16-bit [M][K]
  const float* A;           // [r][K]
  float* T;                 // [M][r]
  void* sT;                 // 16-bit [16][rp64]
  int64_t K;
  int r, rp64;
  float s;
  int cta0;                 // first CTA of this item
};

struct DownParams {
  DownItem item[kMaxGroup];
  int G;
  int M;
  int* tickets;
  int n_tickets;
};

constexpr int kDownThreads = 1024;   // at most two rounds of loads per thread for K <= 16384

template <typename T16>
__device__ __forceinline__ float round16(float v) {
  if constexpr (std::is_same<T16, __nv_bfloat16>::value) return round_bf16(v);
  else return __half2float(__float2half_rn(v));
}

template <typename T16>
__global__ void __launch_bounds__(kDownThreads)
lora_down_small(const __grid_constant__ DownParams p) {
  pdl_wait();         // x is written by the stream's earlier work
  pdl_allow_next();   // the stream kernel may start: it reads x and the weight, then waits for this grid
  int i = 0;
  while (i + 1 < p.G && static_cast<int>(blockIdx.x) >= p.item[i + 1].cta0) ++i;
  const DownItem& it = p.item[i];
  const int j = blockIdx.x - it.cta0;
  if (blockIdx.x == 0)
    for (int t = threadIdx.x; t < p.n_tickets; t += kDownThreads) p.tickets[t] = 0;
  float acc[kStreamMaxM];
#pragma unroll
  for (int m = 0; m < kStreamMaxM; ++m) acc[m] = 0.0f;
  const int64_t chunks = it.K / 8;
  const float* arow = it.A + static_cast<int64_t>(j) * it.K;
#pragma unroll 2
  for (int64_t c = threadIdx.x; c < chunks; c += kDownThreads) {
    const float4 a0 = __ldg(reinterpret_cast<const float4*>(arow) + 2 * c);
    const float4 a1 = __ldg(reinterpret_cast<const float4*>(arow) + 2 * c + 1);
    const float av[8] = {round16<T16>(a0.x), round16<T16>(a0.y), round16<T16>(a0.z), round16<T16>(a0.w),
                         round16<T16>(a1.x), round16<T16>(a1.y), round16<T16>(a1.z), round16<T16>(a1.w)};
#pragma unroll
    for (int m = 0; m < kStreamMaxM; ++m) {
      if (m < p.M) {
        const uint4 xv =
            __ldg(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(it.x) + static_cast<int64_t>(m) * it.K) + c);
        const uint32_t w[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          acc[m] = fmaf(from16<T16>(w[e]), av[2 * e], acc[m]);
          acc[m] = fmaf(from16<T16>(w[e] >> 16), av[2 * e + 1], acc[m]);
        }
      }
    }
  }
  // warp butterfly (fixed order), then the 8 warps' sums in warp order
  __shared__ float wsum[kDownThreads / 32][kStreamMaxM];
#pragma unroll
  for (int m = 0; m < kStreamMaxM; ++m) {
    float v = acc[m];
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    acc[m] = v;
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0)
#pragma unroll
    for (int m = 0; m < kStreamMaxM; ++m) wsum[warp][m] = acc[m];
  __syncthreads();
  if (threadIdx.x < kStreamMaxM) {
    const int m = threadIdx.x;
    float t = 0.0f;
    for (int w = 0; w < kDownThreads / 32; ++w) t += wsum[w][m];
    if (m < p.M) it.T[static_cast<int64_t>(m) * it.r + j] = t;
    store16(static_cast<T16*>(it.sT), m * it.rp64 + j, m < p.M ? it.s * t : 0.0f);
  }
  if (j == 0)   // the slab's padding columns r .. rp64-1
    for (int t = threadIdx.x; t < kStreamMaxM * (it.rp64 - it.r); t += kDownThreads)
      store16(static_cast<T16*>(it.sT), (t / (it.rp64 - it.r)) * it.rp64 + it.r + t % (it.rp64 - it.r), 0.0f);
}

size_t al1024(size_t b) { return (b + 1023) & ~static_cast<size_t>(1023); }

int rp64_of(int r) { return (r + 63) / 64 * 64; }

int tiles_of(int64_t N) { return static_cast<int>((N + kTileRows - 1) / kTileRows); }

struct StreamWs {
  size_t slab[kMaxGroup];
  size_t tickets, part, total;
  StreamWs(const LinearArgs* a, int n) {
    size_t off = 0;
    int tiles = 0;
    for (int i = 0; i < n; ++i) {
      slab[i] = off;
      off += al1024(static_cast<size_t>(kTok) * rp64_of(a[i].r) * 2);
      tiles += tiles_of(a[i].N);
    }
    tickets = off;
    off += al1024(static_cast<size_t>(tiles) * sizeof(int));
    part = off;
    off += al1024(kMaxCtas * kPartBytesPerCta);
    total = off;
  }
};

int sm_count_cached() {
  static int n = 0;
  if (n == 0) {
    int dev = 0, v = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
    n = v > 0 ? v : 1;
  }
  return n;
}

}  // namespace

size_t stream_fwd_ws_bytes(const LinearArgs* a, int n) { return StreamWs(a, n).total; }

template <typename T16>
cudaError_t launch_stream(int64_t M, int ctas_down, const DownParams& dp, const StreamMaps& maps,
                          const StreamParams& sp, cudaStream_t st) {
  static std::once_flag once;
  static cudaError_t attr = cudaSuccess;
  std::call_once(once, [] {
    attr = cudaFuncSetAttribute(nf4_stream_fwd<1, T16>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (attr == cudaSuccess)
      attr = cudaFuncSetAttribute(nf4_stream_fwd<2, T16>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  });
  if (attr != cudaSuccess) return attr;
  cudaError_t e = launch_pdl(lora_down_small<T16>, dim3(ctas_down), dim3(kDownThreads), 0, st, 1, dp);
  note_launch();
  if (e != cudaSuccess) return e;
  e = M <= 8 ? launch_pdl(nf4_stream_fwd<1, T16>, dim3(sp.ctas), dim3(kThreads), kSmemBytes, st, 1, maps, sp)
             : launch_pdl(nf4_stream_fwd<2, T16>, dim3(sp.ctas), dim3(kThreads), kSmemBytes, st, 1, maps, sp);
  note_launch();
  return e;
}

cudaError_t stream_forward(const StreamItem* items, int n, bool f16, void* ws, int* status, cudaStream_t st) {
  if (n < 1 || n > kMaxGroup) return cudaErrorInvalidValue;
  const int64_t M = items[0].a.M;
  if (M < 1 || M > kStreamMaxM) return cudaErrorInvalidValue;
  LinearArgs la[kMaxGroup];
  for (int i = 0; i < n; ++i) la[i] = items[i].a;
  const StreamWs L(la, n);
  char* w = static_cast<char*>(ws);

  DownParams dp{};
  StreamParams sp{};
  StreamMaps maps;
  dp.G = sp.G = n;
  dp.M = sp.M = static_cast<int>(M);
  const DecodeTables& dt = decode_tables();
  for (int k = 0; k < 256; ++k) sp.dyn8[k] = dt.dyn8[k];
  int ctas_down = 0, tiles = 0;
  int64_t units = 0;
  for (int i = 0; i < n; ++i) {
    const StreamItem& it = items[i];
    const LinearArgs& a = it.a;
    const int rp64 = rp64_of(a.r);
    void* sT = w + L.slab[i];
    DownItem& d = dp.item[i];
    d.x = it.x;
    d.A = it.A;
    d.T = it.T;
    d.sT = sT;
    d.K = a.K;
    d.r = a.r;
    d.rp64 = rp64;
    d.s = a.s;
    d.cta0 = ctas_down;
    ctas_down += a.r;
    StreamProj& q = sp.proj[i];
    q.absmax = static_cast<const uint8_t*>(a.W.absmax);
    q.nested = a.W.nested;
    q.offset = a.W.offset;
    q.dq = a.W.dq;
    q.B = it.B;
    q.sT = sT;
    q.y = it.y;
    q.N = a.N;
    q.K = a.K;
    q.r = a.r;
    q.rp64 = rp64;
    q.tiles = tiles_of(a.N);
    q.spans = static_cast<int>((a.K + kSpan - 1) / kSpan);
    q.nbr = static_cast<int>(a.K / kBlock);
    q.unit0 = units;
    q.tile0 = tiles;
    units += static_cast<int64_t>(q.tiles) * q.spans;
    tiles += q.tiles;
    bool ok = make_map(&maps.codes[i], CU_TENSOR_MAP_DATA_TYPE_UINT8, a.W.packed, a.K / 2, a.N, a.K / 2, kSpanBytes,
                       kBoxRows, CU_TENSOR_MAP_SWIZZLE_128B);
    ok = ok && make_map(&maps.x[i], f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, it.x,
                        a.K, M, 2 * a.K, 64, kTok, CU_TENSOR_MAP_SWIZZLE_128B);
    if (!ok) return cudaErrorInvalidValue;
  }
  for (int i = n; i < kMaxGroup; ++i) maps.codes[i] = maps.x[i] = maps.codes[0];
  dp.tickets = reinterpret_cast<int*>(w + L.tickets);
  dp.n_tickets = tiles;
  sp.tickets = dp.tickets;
  sp.part = reinterpret_cast<float*>(w + L.part);
  sp.status = status;
  sp.units = units;
  sp.ctas = static_cast<int>(std::min<int64_t>(units, std::min(sm_count_cached(), kMaxCtas)));
  const WaitSettings wsettings = take_wait_settings();
  sp.wait_ns = wsettings.wait_ns;
  sp.skip_stage0 = wsettings.skip_stage0;

  KernelTimer timer(NF4_TIME_STREAM_FWD, st);
  return f16 ? launch_stream<__half>(M, ctas_down, dp, maps, sp, st)
             : launch_stream<__nv_bfloat16>(M, ctas_down, dp, maps, sp, st);
}

}  // namespace qnf4
