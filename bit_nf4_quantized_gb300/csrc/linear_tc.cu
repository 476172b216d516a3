// bf16 profile of the QLoRA linear on the 5th-generation tensor cores (tcgen05).
//
// Math ("Native model adaptation and NF4", sections "One model contract", "Packed
// NF4 and the portable QLoRA profile", "Fused GPU NF4 decodes inside the matrix
// kernel"): y = x W^T + s T B^T and dX = dY W + s G A, with W decoded from NF4 on
// the device.
//
// W is decoded once per call into a bf16 copy in the workspace by the dequantize kernel
// (bit-exact bf16(nf4[q] * a'), as nf4_dequantize writes it) and the contraction runs as
// a bf16 GEMM fed entirely by TMA.  Decoding inside the matrix kernel would repeat the
// decode once per 256-token tile (16 times per call at 4096 tokens) on the CUDA cores,
// which cannot keep pace with the tensor cores; one decode pass costs 2.5 bytes per weight
// of HBM traffic instead.
//
// Kernel bf16_tc_gemm: clusters of two CTAs on neighbouring SMs, persistent over tiles of
// 256 output features x 256 tokens.  The pair runs 2-SM tcgen05.mma operations
// (M = 256, N = 256, K = 16):
//   D[f, t] (TMEM, fp32) = sum_c Wb[f, c] * Tok[t, c]  +  sum_j SlabA[f, j] * SlabB[t, j]
//   forward: f = rows of W (output features), c = k, Tok = x,  slab (B, s*T)
//   dX:      f = columns of W (input features), c = n, Tok = dY, slab (A^T, s*G)
// Each CTA loads its own 128 feature rows of A and one 128-token half of the token tile;
// the even CTA issues the MMAs, which read both CTAs' shared memory and write each CTA's
// 128 accumulator rows into its own TMEM.  The contraction advances 128 deep per step
// (two 64-deep, 128-byte-swizzled sub-blocks), then in 64-deep adapter slab steps.
// Warp roles (192 threads, in each CTA):
//   warp 0      TMA producer: A rows (K-major for the forward, MN-major for dX), the token
//               half, or the slab tiles, all completing on the even CTA's barrier;
//   warp 1      TMEM allocation (pair-wide); in the even CTA, lane 0 issues the MMAs;
//   warps 2..5  epilogue: tcgen05.ld of this CTA's accumulator rows, bf16 stores.
// Two accumulators of 256 columns let the epilogue of one tile overlap the main loop of
// the next.  A cluster's units alternate the direction of the contraction (even units
// forwards, odd ones backwards), so that a round of clusters starts where the previous one
// ended and finds those slices of the token operand still in L2.  Tiles left for a last,
// partial round of clusters are split along the
// contraction; the parts' fp32 partial sums are added in a fixed order.  Every mbarrier
// wait and the partial-sum flag wait is bounded in time; a wait that gives up sets
// NF4_ERR_TIMEOUT in the status word and the CTA winds down, freeing its TMEM.
#include <algorithm>
#include <vector>

#include <cuda_fp16.h>

#include "linear_tc.cuh"
#include "prep.cuh"
#include "tc_ptx.cuh"

namespace qnf4 {
namespace {

using namespace tc;

constexpr int kTileF = 128;                 // feature rows per CTA (the pair MMA's M is 256)
constexpr int kTileT = 256;                 // MMA N
constexpr int kSub = 64;                    // one sub-block: 64 deep, 128 bytes of bf16 per row
constexpr int kSubs = 2;                    // sub-blocks per step
constexpr int kStepK = kSub * kSubs;        // contraction per step
constexpr int kHalfT = kTileT / 2;          // token rows each CTA of a pair loads
constexpr int kCluster = 2;
constexpr int kSubBytes = 128 * kSub * 2;   // 16384: a 128-row sub-block of A or of the token half
constexpr int kHalfSub = kSubBytes / 2;     // 8192: one 64-feature half of an MN-major sub-block
constexpr int kStageBytes = 2 * kSubs * kSubBytes;   // A then B: 64 KB
constexpr int kStages = 3;
constexpr int kThreads = 192;               // 6 warps, roles above
constexpr int kWarpEpi = 2;                 // first of the 4 epilogue warps
constexpr int kTmemCols = 512;
// barriers: full[kStages] empty[kStages] accfull[2] accempty[2] done, then the abort flag
// and the TMEM address
constexpr int kBarFull = 0, kBarEmpty = kStages, kBarAccFull = 2 * kStages, kBarAccEmpty = kBarAccFull + 2,
              kBarDone = kBarAccEmpty + 2, kNumBars = kBarDone + 1;
constexpr int kOutRows = 32;                // tokens per epilogue store box
constexpr int kOutBytes = kOutRows * kTileF * 2;   // 8 KB: [32 tokens][128 features] bf16
constexpr int kSmemBytes = 1024 + kStages * kStageBytes + 2 * kOutBytes + kNumBars * 8 + 16;
static_assert(kStageBytes % 1024 == 0, "stage buffers must stay 1024-byte aligned");
static_assert(kSmemBytes <= 232448, "shared memory per CTA");

struct GemmParams {
  int64_t M;           // tokens
  int64_t F;           // output features (N forward, K for dX)
  int64_t N, K;        // W is [N, K]
  int mode;            // 0 forward, 1 dX
  int red_steps;       // ceil(contraction / 128)
  int slab_steps;      // padded rank / 64
  int tiles_t, tiles_f;
  int pairs_f;         // ceil(tiles_f / 2): feature-tile pairs; an odd count leaves the last pair's
                       // second tile past F (loads read zeros, the epilogue stores nothing)
  int f_fast;          // pair order: 1 = feature pairs vary fastest, 0 = token tiles
  int band;            // > 0: token tiles in bands of `band`, the band's tiles fastest within a
                       // feature pair, the feature pairs next, the bands slowest (overrides f_fast)
  int f16;             // operands and output are IEEE half (else bf16)
  void* out;           // [M, F] 16-bit
  int* status;
  // work units: tiles [0, full_units) whole, then the remaining tiles (fewer than one
  // round of clusters) in `split` parts along the contraction, `chunk` steps each (the
  // last part also runs the slab steps).  The leading parts leave their fp32 partial sums
  // in part_ws ([slot][part][rank][256 tokens][128 rows]) and take a ticket from
  // part_tickets[slot][rank] (zero at launch).  The last part, if it finds every ticket
  // taken, adds their sums to its own (still in TMEM) and stores the tile; otherwise it
  // leaves its sums too and takes a ticket, and the CTA that draws the last ticket stores
  // the tile.  The sum is always last part + parts 0, 1, ... in order.  Nothing waits for
  // another cluster, so a launch completes even when not all its clusters are resident.
  int64_t full_units, total_units;
  int split, chunk;
  float* part_ws;
  int* part_tickets;
  uint64_t wait_ns;    // bounded-wait limit of this launch
  int skip_stage0;     // CTA 0 leaves its first stage unissued (tests of the timeout path)
};

struct Unit {
  int64_t tile;      // tile pair index
  int red0, nred;    // contraction steps [red0, red0 + nred)
  int nslab;         // slab steps (last part only)
  int part;          // 0 .. split-1 (0 for a whole tile)
  int nparts;        // 1 for a whole tile
  int64_t slot;      // index of a split tile among the split tiles
};

__device__ __forceinline__ Unit unit_of(const GemmParams& p, int64_t u) {
  Unit x;
  if (u < p.full_units) {
    x.tile = u;
    x.red0 = 0;
    x.nred = p.red_steps;
    x.nslab = p.slab_steps;
    x.part = 0;
    x.nparts = 1;
    x.slot = 0;
  } else {
    const int64_t v = u - p.full_units;
    x.slot = v / p.split;
    x.part = static_cast<int>(v - x.slot * p.split);
    x.tile = p.full_units + x.slot;
    x.red0 = x.part * p.chunk;
    x.nred = min(p.chunk, p.red_steps - x.red0);
    x.nslab = x.part == p.split - 1 ? p.slab_steps : 0;
    x.nparts = p.split;
  }
  return x;
}

// Token tile (x) and feature pair (y) of tile pair `pair`, in the launch's order.
__device__ __forceinline__ longlong2 tile_pair_of(const GemmParams& p, int64_t pair) {
  if (p.band > 0) {
    const int64_t per = static_cast<int64_t>(p.band) * p.pairs_f;
    const int64_t bi = pair / per, t0 = bi * p.band;
    const int64_t bt = min(static_cast<int64_t>(p.band), static_cast<int64_t>(p.tiles_t) - t0);
    const int64_t idx = pair - bi * per;
    return make_longlong2(t0 + idx % bt, idx / bt);
  }
  if (p.f_fast) return make_longlong2(pair / p.pairs_f, pair % p.pairs_f);
  return make_longlong2(pair % p.tiles_t, pair / p.tiles_t);
}

// Slot and phase of the stage ring, advanced once per step by every role.
struct Ring {
  int s = 0;
  uint32_t ph = 0;
  __device__ __forceinline__ void advance() {
    if (++s == kStages) s = 0, ph ^= 1u;
  }
};

__global__ void __launch_bounds__(kThreads, 1)
bf16_tc_gemm(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_tok,
             const __grid_constant__ CUtensorMap tm_slab_f, const __grid_constant__ CUtensorMap tm_slab_t,
             const __grid_constant__ CUtensorMap tm_out, const GemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* base_ptr = smem_raw + (base - raw);
  const uint32_t out_stage = base + kStages * kStageBytes;   // two [32][128] bf16 store boxes
  uint64_t* bars = reinterpret_cast<uint64_t*>(base_ptr + kStages * kStageBytes + 2 * kOutBytes);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + kNumBars);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + kNumBars) + 1;
  auto bar = [&](int i) { return smem_u32(bars + i); };
  auto stage_a = [&](int s) { return base + s * kStageBytes; };
  auto stage_b = [&](int s) { return base + s * kStageBytes + kSubs * kSubBytes; };
  const uint32_t rank = cluster_ctarank();
  auto lead_bar = [&](int i) { return mapa_shared(bar(i), 0); };
  const int64_t cluster_id = blockIdx.x / kCluster;
  const int64_t n_clusters = gridDim.x / kCluster;
  auto tile_t = [&](int64_t pair) { return tile_pair_of(p, pair).x; };
  auto tile_f = [&](int64_t pair) { return 2 * tile_pair_of(p, pair).y + rank; };

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar(kBarFull + s), 1);      // even CTA: its producer's arrive + both CTAs' TMA bytes
      mbar_init(bar(kBarEmpty + s), 1);     // the pair MMAs' commit
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(kBarAccFull + b), 1);                  // the pair MMAs' commit
      mbar_init(bar(kBarAccEmpty + b), 4 * kCluster);      // the epilogue warps of both CTAs
    }
    mbar_init(bar(kBarDone), 1);                           // the issuer's last commit
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  pdl_allow_next();
  // TMEM is taken only after the preceding grid has completed: a CTA never holds TMEM while
  // it waits for another grid, so a CTA blocked in tcgen05.alloc always waits for one that
  // is running to its end
  pdl_wait();
  if (warp == 1) {   // one warp of each CTA of the pair allocates collectively
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    tc_fence_before();
  }
  cluster_sync();   // the peer's barriers are initialised before anything signals them
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  // every role walks the same units (cluster_id, + n_clusters, ...) and steps
  auto unit_at = [&](int64_t lt) { return cluster_id + lt * n_clusters; };

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      bool ok = true;
      Ring c;
      int64_t issued = 0;
      for (int64_t lt = 0; ok && unit_at(lt) < p.total_units; ++lt) {
        const Unit un = unit_of(p, unit_at(lt));
        const int th = static_cast<int>(tile_t(un.tile) * kTileT) + static_cast<int>(rank) * kHalfT;
        const int f0 = static_cast<int>(tile_f(un.tile) * kTileF);
        for (int st = 0; st < un.nred + un.nslab; ++st, c.advance()) {
          const int s = c.s;
          if (!mbar_wait(bar(kBarEmpty + s), c.ph ^ 1u, abort_flag, p.status, p.wait_ns)) { ok = false; break; }
          const uint32_t full = lead_bar(kBarFull + s);
          if (p.skip_stage0 && blockIdx.x == 0 && issued == 0) {   // the stage's waits will run out
            ++issued;
            continue;
          }
          if (st < un.nred) {
            // odd units walk the contraction backwards: the clusters of one round move through
            // it together, so the next round starts on the slices this one read last, which
            // are still in L2 when an operand is too large for L2 to hold whole
            const int kst = (lt & 1) ? un.nred - 1 - st : st;
            const int k0 = (un.red0 + kst) * kStepK;
            if (rank == 0) mbar_expect_tx(bar(kBarFull + s), kCluster * 2 * kSubs * kSubBytes);
#pragma unroll
            for (int u = 0; u < kSubs; ++u) {
              const uint32_t a = stage_a(s) + u * kSubBytes;
              if (p.mode == 0) {
                // forward: 128 rows of W (features f0..) x 64 of k, K-major
                tma_load_2d_pair(a, &tm_w, full, k0 + u * kSub, f0);
              } else {
                // dX: rows n of W are the contraction; two 64-feature halves, MN-major
                tma_load_2d_pair(a, &tm_w, full, f0, k0 + u * kSub);
                tma_load_2d_pair(a + kHalfSub, &tm_w, full, f0 + 64, k0 + u * kSub);
              }
              tma_load_2d_pair(stage_b(s) + u * kSubBytes, &tm_tok, full, k0 + u * kSub, th);
            }
          } else {
            const int j = (st - un.nred) * kSub;
            if (rank == 0) mbar_expect_tx(bar(kBarFull + s), kCluster * 2 * kSubBytes);
            tma_load_2d_pair(stage_a(s), &tm_slab_f, full, j, f0);
            tma_load_2d_pair(stage_b(s), &tm_slab_t, full, j, th);
          }
          ++issued;
        }
      }
      if (ok) {
        // the pair MMAs' commits arrive on this CTA's empty barriers: wait for the last
        // round of them so that none lands after the CTA has exited
        for (int k = 0; k < kStages; ++k) {
          if (!mbar_wait(bar(kBarEmpty + c.s), c.ph ^ 1u, abort_flag, p.status, p.wait_ns)) break;
          c.advance();
        }
      } else if (rank == 0) {  // let copies already in flight land before the CTA exits
        int ds = c.s;
        uint32_t dph = c.ph;
        for (int64_t k = 0; k < kStages && k < issued; ++k) {
          if (ds == 0) ds = kStages - 1, dph ^= 1u;
          else --ds;
          mbar_drain(bar(kBarFull + ds), dph);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      // ---------------- MMA issuer (even CTA) ----------------
      const uint32_t idesc_main = idesc_16(kCluster * kTileF, kTileT, p.mode == 1 ? 1u : 0u, p.f16 ? 1u : 0u);
      const uint32_t idesc_slab = idesc_16(kCluster * kTileF, kTileT, 0u, p.f16 ? 1u : 0u);
      bool ok = true;
      Ring c;
      for (int64_t lt = 0; ok && unit_at(lt) < p.total_units; ++lt) {
        const Unit un = unit_of(p, unit_at(lt));
        const int nsteps = un.nred + un.nslab;
        const uint32_t b = static_cast<uint32_t>(lt) & 1u;
        if (!mbar_wait(bar(kBarAccEmpty + b), (static_cast<uint32_t>(lt >> 1) & 1u) ^ 1u, abort_flag, p.status, p.wait_ns)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + b * kTileT;
        for (int st = 0; st < nsteps; ++st, c.advance()) {
          if (!mbar_wait(bar(kBarFull + c.s), c.ph, abort_flag, p.status, p.wait_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          if (st < un.nred) {
#pragma unroll
            for (int u = 0; u < kSubs; ++u)
#pragma unroll
              for (int kk = 0; kk < kSub / 16; ++kk) {
                // K-major: 32 bytes per 16-element k step inside the 128-byte row.
                // MN-major (dX): two 8-row groups of 1024 bytes per k step; the two
                // 64-feature halves of the sub-block are 8192 bytes apart.
                const uint32_t sa = stage_a(c.s) + u * kSubBytes;
                const uint64_t adesc = p.mode == 1 ? smem_desc(sa + kk * 2048, kHalfSub, 1024)
                                                   : smem_desc(sa + kk * 32, 16, 1024);
                const uint64_t bdesc = smem_desc(stage_b(c.s) + u * kSubBytes + kk * 32, 16, 1024);
                umma_bf16_pair(d_tmem, adesc, bdesc, idesc_main, (st > 0 || u > 0 || kk > 0) ? 1u : 0u);
              }
          } else {
#pragma unroll
            for (int kk = 0; kk < kSub / 16; ++kk)
              umma_bf16_pair(d_tmem, smem_desc(stage_a(c.s) + kk * 32, 16, 1024),
                             smem_desc(stage_b(c.s) + kk * 32, 16, 1024), idesc_slab, (st > 0 || kk > 0) ? 1u : 0u);
          }
          umma_commit_pair_mc(bar(kBarEmpty + c.s), 0x3);   // frees stage s in both CTAs
          if (st == nsteps - 1) umma_commit_pair_mc(bar(kBarAccFull + b), 0x3);
        }
      }
      // every pair MMA issued has completed before either CTA frees its TMEM (the final
      // cluster barrier holds the odd CTA until this drain is over)
      umma_commit_pair_mc(bar(kBarDone), 0x1);
      mbar_drain(bar(kBarDone), 0);
    }
  } else {
    // ---------------- epilogue ----------------
    // Output tiles go out through shared memory: each warp converts its 32 feature rows of
    // 32 tokens to bf16 in a [32 tokens][128 features] box, and one thread stores the box
    // with TMA (two boxes alternate).  The four warps meet at named barrier 1; whether to
    // go on is decided by a vote, so that all four always take the same path.
    __shared__ int votes[2][4];
    __shared__ int last_ticket;
    const int quarter = warp & 3;               // TMEM lanes 32*quarter .. +31
    const int lrow = quarter * 32 + lane;       // this thread's row of the CTA's 128
    const bool issuer = warp == kWarpEpi && lane == 0;
    uint32_t nst = 0;                           // boxes stored so far (picks the buffer)
    for (int64_t lt = 0; unit_at(lt) < p.total_units; ++lt) {
      const Unit un = unit_of(p, unit_at(lt));
      const uint32_t b = static_cast<uint32_t>(lt) & 1u;
      const uint32_t aph = static_cast<uint32_t>(lt >> 1) & 1u;
      const bool ok_w = __all_sync(0xffffffffu, mbar_wait(bar(kBarAccFull + b), aph, abort_flag, p.status, p.wait_ns));
      if (lane == 0) votes[b][quarter] = ok_w ? 1 : 0;
      named_sync(1, 128);
      if (!(votes[b][0] && votes[b][1] && votes[b][2] && votes[b][3])) break;
      tc_fence_after();
      const int64_t t0 = tile_t(un.tile) * kTileT;
      const int f0 = static_cast<int>(tile_f(un.tile) * kTileF);
      const uint32_t taddr = tmem_base + b * kTileT + (static_cast<uint32_t>(quarter * 32) << 16);
      // partial sums of a split tile: [slot][part][rank][256][128] fp32, coalesced along rows
      auto part_buf = [&](int part) {
        return p.part_ws + ((un.slot * p.split + part) * kCluster + rank) * (static_cast<int64_t>(kTileT) * 128);
      };
      bool store_tile = true;       // this CTA writes the tile's output
      bool last_in_tmem = true;     // the last part's sums are in this CTA's TMEM
      if (un.nparts > 1) {
        int* ticket = p.part_tickets + un.slot * kCluster + rank;
        bool fast = false;          // the last part, with every other part already done
        if (un.part == un.nparts - 1) {
          if (issuer) {
            int seen;
            asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(seen) : "l"(ticket) : "memory");
            last_ticket = (seen == un.nparts - 1) ? 1 : 0;
          }
          named_sync(1, 128);
          fast = last_ticket != 0;
          named_sync(1, 128);
        }
        if (!fast) {
          // this part's sums to the workspace, then a ticket; the last ticket finishes the tile
#pragma unroll 1
          for (int c0 = 0; c0 < kTileT; c0 += 16) {
            uint32_t v[16];
            tmem_ld16(taddr + c0, v);
            tmem_ld_wait();
            float* dst = part_buf(un.part) + static_cast<int64_t>(c0) * 128 + lrow;
#pragma unroll
            for (int j = 0; j < 16; ++j) dst[j * 128] = __uint_as_float(v[j]);
          }
          __threadfence();
          named_sync(1, 128);
          if (issuer) {
            const int t = atomicAdd(ticket, 1);
            last_ticket = (t == un.nparts - 1) ? 1 : 0;
          }
          named_sync(1, 128);
          store_tile = last_ticket != 0;
          last_in_tmem = false;
        }
        if (store_tile) __threadfence();
      }
      if (store_tile) {
#pragma unroll 1
        for (int c0 = 0; c0 < kTileT; c0 += kOutRows, ++nst) {
          const uint32_t box = out_stage + (nst & 1u) * kOutBytes;
          if (issuer) bulk_wait_read<1>();      // the store that last used this box has read it
          named_sync(1, 128);
#pragma unroll
          for (int h = 0; h < kOutRows; h += 16) {
            uint32_t v[16];
            if (last_in_tmem) {
              tmem_ld16(taddr + c0 + h, v);
              tmem_ld_wait();
            } else {               // the last part's sums from the workspace
              const float* src = part_buf(un.nparts - 1) + static_cast<int64_t>(c0 + h) * 128 + lrow;
#pragma unroll
              for (int j = 0; j < 16; ++j) v[j] = __float_as_uint(__ldcg(src + j * 128));
            }
            // then the other parts in part order: the same sums whichever CTA finishes
            for (int q = 0; q < un.nparts - 1; ++q) {
              const float* src = part_buf(q) + static_cast<int64_t>(c0 + h) * 128 + lrow;
#pragma unroll
              for (int j = 0; j < 16; ++j) v[j] = __float_as_uint(__uint_as_float(v[j]) + __ldcg(src + j * 128));
            }
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const float f = __uint_as_float(v[j]);
              const uint16_t o = p.f16 ? __half_as_ushort(__float2half_rn(f)) : __bfloat16_as_ushort(__float2bfloat16_rn(f));
              asm volatile("st.shared.b16 [%0], %1;" ::"r"(box + static_cast<uint32_t>(((h + j) * kTileF + lrow) * 2)),
                           "h"(o)
                           : "memory");
            }
          }
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          named_sync(1, 128);
          if (issuer) {   // rows past M and columns past F are not written
            tma_store_2d(&tm_out, box, f0, static_cast<int>(t0) + c0);
            bulk_commit();
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_remote(lead_bar(kBarAccEmpty + b));
    }
    if (issuer) bulk_wait_all();   // the last boxes are written before the CTA exits
  }

  tc_fence_before();
  cluster_sync();   // neither CTA exits while the other may still signal its barriers
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(kTmemCols)
                 : "memory");
  }
}

// ---- host side --------------------------------------------------------------------------

int padded_rank(int r) { return (r + kSub - 1) / kSub * kSub; }
size_t a1024(size_t b) { return (b + 1023) & ~static_cast<size_t>(1023); }

int sm_count() {
  int dev = 0, n = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n > 0 ? n : 1;
}

constexpr int kMaxPartTiles = 80;   // partial-sum tiles (of a cluster pair) a split may use (all parts)
constexpr int kMaxSplit = 4;
constexpr size_t kPartTileBytes = static_cast<size_t>(kCluster) * kTileT * 128 * sizeof(float);
constexpr size_t kPartFlagBytes = static_cast<size_t>(kMaxPartTiles) * kCluster * 4 * sizeof(int);

// Work units: whole tiles for every full round of clusters; the tiles of a last, partial
// round are split along the contraction into as many parts as idle clusters allow.
void split_tail(GemmParams* p, int64_t pairs, int64_t clusters) {
  const int64_t rounds = pairs / clusters, tail = pairs - rounds * clusters;
  p->full_units = pairs;
  p->total_units = pairs;
  p->split = 1;
  p->chunk = p->red_steps;
  if (rounds == 0 || tail == 0) return;
  int split = static_cast<int>(std::min<int64_t>(clusters / tail, kMaxSplit));
  split = std::min(split, p->red_steps);
  while (split > 1 && tail * split > kMaxPartTiles) --split;
  if (split < 2) return;
  const int chunk = (p->red_steps + split - 1) / split;
  split = (p->red_steps + chunk - 1) / chunk;   // every part keeps at least one contraction step
  if (split < 2) return;
  p->full_units = rounds * clusters;
  p->total_units = p->full_units + tail * split;
  p->split = split;
  p->chunk = chunk;
}

cudaError_t launch_gemm(const GemmParams& p, const CUtensorMap& w, const CUtensorMap& tok,
                        const CUtensorMap& slab_f, const CUtensorMap& slab_t, cudaStream_t st) {
  CUtensorMap out;   // [M][F] 16-bit, stored in [32 tokens][128 features] boxes
  if (!make_map(&out, p.f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, p.out, p.F, p.M,
                2 * p.F, kTileF, kOutRows, CU_TENSOR_MAP_SWIZZLE_NONE))
    return cudaErrorInvalidValue;
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  static int max_clusters = 0;
  cudaLaunchConfig_t cfg{};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kCluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;   // see pdl_allow_next
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  std::call_once(once, [&] {
    attr_err = cudaFuncSetAttribute(bf16_tc_gemm, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (attr_err != cudaSuccess) return;
    cfg.gridDim = dim3(static_cast<unsigned>(sm_count() / kCluster * kCluster));
    attr_err = cudaOccupancyMaxActiveClusters(&max_clusters, bf16_tc_gemm, &cfg);
    if (attr_err == cudaSuccess && max_clusters < 1) attr_err = cudaErrorInvalidConfiguration;
  });
  if (attr_err != cudaSuccess) return attr_err;
  const int64_t pairs = static_cast<int64_t>(p.tiles_t) * p.pairs_f;
  const int64_t clusters = pairs < max_clusters ? pairs : max_clusters;
  cfg.gridDim = dim3(static_cast<unsigned>(clusters * kCluster));
  GemmParams q = p;
  split_tail(&q, pairs, clusters);
  const WaitSettings ws = take_wait_settings();
  q.wait_ns = ws.wait_ns;
  q.skip_stage0 = ws.skip_stage0;
  KernelTimer timer(p.mode == 0 ? NF4_TIME_FWD_GEMM : NF4_TIME_DX_GEMM, st);
  cfg.numAttrs = 2;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, bf16_tc_gemm, w, tok, slab_f, slab_t, out, q);
  note_launch();
  return e != cudaSuccess ? e : cudaGetLastError();
}

int64_t pad8(int64_t v) { return (v + 7) / 8 * 8; }

PrepJob zero_flags_job(void* flags) {
  PrepJob j{};
  j.kind = kZeroWords;
  j.fdst = static_cast<float*>(flags);
  j.count = static_cast<int64_t>(kPartFlagBytes / sizeof(int));
  return j;
}

// The weight decoded to 16 bits [N][K] for this call (bit-exact with nf4_dequantize), in the
// same launch as the call's operand staging (extra CTAs run the prep jobs); with the weight
// given decoded (w16), the staging alone.
cudaError_t decode_weight(const LinearArgs& a, bool f16, void* wb, const PrepBuilder& prep, cudaStream_t st,
                          const void* w16) {
  if (!prep.ok()) return cudaErrorInvalidValue;
  if (w16 != nullptr) return launch_prep_only(f16, prep.jobs(), prep.ctas(), st);
  KernelTimer timer(NF4_TIME_WEIGHT_DECODE, st);
  return launch_decode_with_prep(a.W, wb, f16, prep.jobs(), prep.ctas(), st);
}

// Workspace layouts (every part 1024-byte aligned).  `part` holds the skinny passes'
// partial sums and, while the GEMM runs (never at the same time), its split tiles'
// partial sums; `wb` the bf16 weight; `flags` the GEMM's per-part flags.
struct FwdWs {
  size_t sTp, Bp, Aq, part, wb, flags, total;
  FwdWs(int64_t M, int64_t N, int64_t K, int r, bool w16 = false) {
    const size_t rp = padded_rank(r), nq = adapter_nq(r);
    sTp = 0;
    Bp = sTp + a1024(2 * rp * M);
    Aq = Bp + a1024(2 * rp * N);
    part = Aq + a1024(2 * nq * K);
    wb = part + a1024(std::max(adapter_partial_bytes(M, K, r), kMaxPartTiles * kPartTileBytes));
    flags = wb + (w16 ? 0 : a1024(2 * static_cast<size_t>(N) * K));
    total = flags + a1024(kPartFlagBytes);
  }
};

struct BwdWs {
  size_t sGp, ApT, Bt, Tt, Gt, part, wb, flags, total;
  BwdWs(int64_t M, int64_t N, int64_t K, int r, bool w16 = false) {
    const size_t rp = padded_rank(r), nq = adapter_nq(r), Mp = pad8(M);
    // G's and dB's partial sums side by side (one launch runs both), later dA's
    size_t pb = adapter_partial_bytes(M, N, r) + adapter_partial_bytes(N, M, r);
    pb = std::max(pb, adapter_partial_bytes(K, M, r));
    pb = std::max(pb, kMaxPartTiles * kPartTileBytes);
    sGp = 0;
    ApT = sGp + a1024(2 * rp * M);
    Bt = ApT + a1024(2 * rp * K);
    Tt = Bt + a1024(2 * nq * N);
    Gt = Tt + a1024(2 * nq * Mp);
    part = Gt + a1024(2 * nq * Mp);
    wb = part + a1024(pb);
    flags = wb + (w16 ? 0 : a1024(2 * static_cast<size_t>(N) * K));
    total = flags + a1024(kPartFlagBytes);
  }
};

GemmParams base_params(const LinearArgs& a, bool f16, int mode, void* out, int* status) {
  GemmParams p{};
  p.f16 = f16 ? 1 : 0;
  p.M = a.M;
  p.N = a.N;
  p.K = a.K;
  p.F = mode == 0 ? a.N : a.K;
  p.mode = mode;
  const int64_t red = mode == 0 ? a.K : a.N;
  p.red_steps = static_cast<int>((red + kStepK - 1) / kStepK);
  p.slab_steps = padded_rank(a.r) / kSub;
  p.tiles_t = static_cast<int>((a.M + kTileT - 1) / kTileT);
  p.tiles_f = static_cast<int>((p.F + kTileF - 1) / kTileF);
  p.pairs_f = (p.tiles_f + 1) / 2;
  // each round of clusters re-reads the whole operand along the fast dimension: run the
  // feature pairs fastest only when the weight panel set (F rows) is smaller than the tokens
  p.f_fast = p.F < a.M ? 1 : 0;
  // when neither operand fits in half of L2 (down's forward, gate's and up's dX at 4096
  // tokens), a round of clusters covers a block of 8 token tiles by about 76 / 8 feature pairs
  // (8 is near the square root of the 76 clusters): it reads 8 token panels and 9 or 10 weight
  // panels where the plain order reads every token panel, and the next round shares half of them
  const int64_t half_l2 = 64ll << 20;
  p.band = (2 * a.M * red > half_l2 && 2 * p.F * red > half_l2 && p.tiles_t > 8 && p.pairs_f > 8) ? 8 : 0;
  p.out = out;
  p.status = status;
  return p;
}

// The forward GEMM y = x W^T + (s T) B^T of one projection: W 16-bit [N][K] (wb), B's
// staged copy Bp [N][rp], 16-bit s T sTp [M][rp]; part / flags for split tiles.
cudaError_t fwd_gemm(const LinearArgs& a, bool f16, const void* x, const void* wb, const void* Bp, const void* sTp,
                     void* part, void* flags, void* y, int* status, cudaStream_t st) {
  const int rp = padded_rank(a.r);
  const CUtensorMapDataType dt16 = f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  CUtensorMap wm, tok, slab_f, slab_t;
  bool ok = make_map(&wm, dt16, wb, a.K, a.N, 2 * a.K, kSub, kTileF, CU_TENSOR_MAP_SWIZZLE_128B);
  ok = ok && make_map(&tok, dt16, x, a.K, a.M, 2 * a.K, kSub, kHalfT, CU_TENSOR_MAP_SWIZZLE_128B);
  ok = ok && make_map(&slab_f, dt16, Bp, rp, a.N, 2 * rp, kSub, kTileF, CU_TENSOR_MAP_SWIZZLE_128B);
  ok = ok && make_map(&slab_t, dt16, sTp, rp, a.M, 2 * rp, kSub, kHalfT, CU_TENSOR_MAP_SWIZZLE_128B);
  if (!ok) return cudaErrorInvalidValue;
  GemmParams gp = base_params(a, f16, 0, y, status);
  gp.part_ws = static_cast<float*>(part);
  gp.part_tickets = static_cast<int*>(flags);
  return launch_gemm(gp, wm, tok, slab_f, slab_t, st);
}

// The dX GEMM dX = dY W + (s G) A of one projection: A's staged copy ApT [K][rp], 16-bit
// s G sGp [M][rp].
cudaError_t dx_gemm(const LinearArgs& a, bool f16, const void* dy, const void* wb, const void* ApT, const void* sGp,
                    void* part, void* flags, void* dx, int* status, cudaStream_t st) {
  const int rp = padded_rank(a.r);
  const CUtensorMapDataType dt16 = f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  CUtensorMap wm, tok, slab_f, slab_t;
  // W [N][K] read as 64 features x 64 rows n (MN-major A: the features are the MMA's M)
  bool ok = make_map(&wm, dt16, wb, a.K, a.N, 2 * a.K, kSub, kSub, CU_TENSOR_MAP_SWIZZLE_128B);
  ok = ok && make_map(&tok, dt16, dy, a.N, a.M, 2 * a.N, kSub, kHalfT, CU_TENSOR_MAP_SWIZZLE_128B);
  ok = ok && make_map(&slab_f, dt16, ApT, rp, a.K, 2 * rp, kSub, kTileF, CU_TENSOR_MAP_SWIZZLE_128B);
  ok = ok && make_map(&slab_t, dt16, sGp, rp, a.M, 2 * rp, kSub, kHalfT, CU_TENSOR_MAP_SWIZZLE_128B);
  if (!ok) return cudaErrorInvalidValue;
  GemmParams gp = base_params(a, f16, 1, dx, status);
  gp.part_ws = static_cast<float*>(part);
  gp.part_tickets = static_cast<int*>(flags);
  return launch_gemm(gp, wm, tok, slab_f, slab_t, st);
}

// The backward's staging jobs of one projection (B^T, T^T, A^T and the GEMM's flags) and,
// when Gt_zero, the zeroed G^T [nq][Mp].
void bwd_prep_jobs(const LinearArgs& a, const float* T, const float* A, const float* B, const BwdWs& L, char* w,
                   bool Gt_zero, std::vector<PrepJob>* jobs) {
  const int rp = padded_rank(a.r), nq = adapter_nq(a.r);
  const int64_t Mp = pad8(a.M);
  PrepJob j{};
  j.kind = kStageTransposed;   // B^T: [nq][N]
  j.r = a.r;
  j.width = a.N;
  j.src = B;
  j.dst = w + L.Bt;
  j.cols = a.N;
  j.count = static_cast<int64_t>(nq) * a.N;
  jobs->push_back(j);
  PrepJob t = j;               // T^T: [nq][Mp]
  t.width = Mp;
  t.src = T;
  t.dst = w + L.Tt;
  t.cols = a.M;
  t.count = static_cast<int64_t>(nq) * Mp;
  jobs->push_back(t);
  if (Gt_zero) {
    PrepJob g = t;             // G^T starts zero; the G finish fills rows < r, columns < M
    g.r = 0;
    g.dst = w + L.Gt;
    jobs->push_back(g);
  }
  PrepJob c{};
  c.kind = kStageColumns;      // A^T as the slab's feature side: [K][rp]
  c.r = a.r;
  c.width = rp;
  c.src = A;
  c.dst = w + L.ApT;
  c.cols = a.K;
  c.count = a.K * rp;
  jobs->push_back(c);
  jobs->push_back(zero_flags_job(w + L.flags));
}

// The pair of passes G = dY B (rows M, reduction over N along dY's rows; G, 16-bit s G, 16-bit
// G^T into Gt with row stride ldt) and dB = s dY^T T (rows N, reduction over M down dY's
// columns), both reading only dY.
void gdb_args(const LinearArgs& a, bool f16, const void* dy, float* G, float* dB, const BwdWs& L, char* w, void* Gt,
              int64_t ldt, AdapterPassArgs* pa) {
  const int rp = padded_rank(a.r);
  const int64_t Mp = pad8(a.M);
  auto* part = reinterpret_cast<float*>(w + L.part);
  pa[0] = AdapterPassArgs{};
  pa[1] = AdapterPassArgs{};
  AdapterPassArgs& g = pa[0];
  g.X = dy;
  g.x_inner = a.N;
  g.x_outer = a.M;
  g.Q = w + L.Bt;
  g.q_cols = a.N;
  g.r = a.r;
  g.rows = a.M;
  g.red = a.N;
  g.partial = part;
  g.scale = 1.0f;
  g.f32 = G;
  g.b_rows = w + L.sGp;
  g.rp = rp;
  g.scale_b = a.s;
  g.b_t = Gt;
  g.ldt = ldt;
  AdapterPassArgs& d = pa[1];
  d.X = dy;
  d.x_inner = a.N;
  d.x_outer = a.M;
  d.mn_major = true;
  d.Q = w + L.Tt;
  d.q_cols = Mp;
  d.r = a.r;
  d.rows = a.N;
  d.red = a.M;
  d.partial = reinterpret_cast<float*>(reinterpret_cast<char*>(part) + adapter_partial_bytes(a.M, a.N, a.r));
  d.scale = a.s;
  d.f32 = dB;
  g.f16 = d.f16 = f16 ? 1 : 0;
}

// One launch for the pair, then one for both finishes.
cudaError_t gdb_pass(const LinearArgs& a, bool f16, const void* dy, float* G, float* dB, const BwdWs& L, char* w,
                     void* Gt, int64_t ldt, int* status, cudaStream_t st) {
  AdapterPassArgs pa[2];
  gdb_args(a, f16, dy, G, dB, L, w, Gt, ldt, pa);
  return adapter_run(pa, 2, status, st);
}

// Staging jobs in launches of at most kMaxPrepJobs each.
cudaError_t run_prep(const std::vector<PrepJob>& jobs, bool f16, cudaStream_t st) {
  for (size_t j0 = 0; j0 < jobs.size(); j0 += kMaxPrepJobs) {
    PrepBuilder b(f16);
    for (size_t j = j0; j < jobs.size() && j < j0 + kMaxPrepJobs; ++j) b.add(jobs[j]);
    if (!b.ok()) return cudaErrorInvalidValue;
    const cudaError_t e = launch_prep_only(f16, b.jobs(), b.ctas(), st);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

// The input sets of a run: maximal stretches of consecutive items that read the same x (the
// same pointer and K) whose ranks, each rounded up to 16, add up to at most kTcGroupMaxRank.
// Set g holds items [first[g], first[g + 1]); item i's rank side sits at rows col[i] of its
// set's stacked Q (nqt[g] rows).
struct XSets {
  int n = 0;
  int first[kTcGroupMax + 1] = {};
  int nqt[kTcGroupMax] = {};
  int col[kTcGroupMax] = {};
  template <typename Item>
  XSets(const Item* it, int m) {
    for (int i = 0; i < m; ++i) {
      const int nq = adapter_nq(it[i].a.r);
      const bool join = n > 0 && it[i].x == it[first[n - 1]].x && it[i].a.K == it[first[n - 1]].a.K &&
                        nqt[n - 1] + nq <= kTcGroupMaxRank;
      if (!join) {
        first[n] = i;
        nqt[n] = 0;
        ++n;
      }
      col[i] = nqt[n - 1];
      nqt[n - 1] += nq;
    }
    first[n] = m;
  }
};

// Run workspaces: each item's single-call layout (after its fp32 G, backward), then per input
// set its stacked rank side (A forward, G^T backward) and its shared pass's partial sums.
struct FwdRunWs {
  size_t item[kTcGroupMax] = {}, Aq[kTcGroupMax] = {}, part[kTcGroupMax] = {};
  size_t total = 0;
  FwdRunWs(const TcFwdItem* it, int n, const XSets& xs) {
    size_t off = 0;
    for (int i = 0; i < n; ++i) {
      const LinearArgs& a = it[i].a;
      item[i] = off;
      off += a1024(FwdWs(a.M, a.N, a.K, a.r, it[i].w16 != nullptr).total);
    }
    for (int g = 0; g < xs.n; ++g) {
      const LinearArgs& a = it[xs.first[g]].a;
      Aq[g] = off;
      part[g] = Aq[g] + a1024(2 * static_cast<size_t>(xs.nqt[g]) * a.K);
      off = part[g] + a1024(adapter_partial_bytes(a.M, a.K, xs.nqt[g]));
    }
    total = off;
  }
};

struct BwdRunWs {
  size_t G[kTcGroupMax] = {}, item[kTcGroupMax] = {}, Gt[kTcGroupMax] = {}, part[kTcGroupMax] = {};
  size_t total = 0;
  BwdRunWs(const TcBwdItem* it, int n, const XSets& xs) {
    size_t off = 0;
    for (int i = 0; i < n; ++i) {
      const LinearArgs& a = it[i].a;
      G[i] = off;
      off += a1024(sizeof(float) * static_cast<size_t>(a.M) * a.r);
      item[i] = off;
      off += a1024(BwdWs(a.M, a.N, a.K, a.r, it[i].w16 != nullptr).total);
    }
    for (int g = 0; g < xs.n; ++g) {
      const LinearArgs& a = it[xs.first[g]].a;
      Gt[g] = off;
      part[g] = Gt[g] + a1024(2 * static_cast<size_t>(xs.nqt[g]) * pad8(a.M));
      off = part[g] + a1024(adapter_partial_bytes(a.K, a.M, xs.nqt[g]));
    }
    total = off;
  }
};

// The resident CTAs shared between a launch's passes in proportion to the activation bytes
// each reads (the passes then hold about one wave of CTAs together).
void share_targets(AdapterPassArgs* a, int n) {
  const int total = adapter_total_ctas();
  double bytes = 0.0;
  for (int i = 0; i < n; ++i) bytes += static_cast<double>(a[i].rows) * a[i].red;
  for (int i = 0; i < n; ++i)
    a[i].target = std::max(1, static_cast<int>(total * (static_cast<double>(a[i].rows) * a[i].red) / bytes));
}

template <typename Item>
bool run_ok(const Item* it, int n) {
  if (n < 1 || n > kTcGroupMax) return false;
  for (int i = 0; i < n; ++i)
    if (it[i].a.M != it[0].a.M || adapter_nq(it[i].a.r) > kTcGroupMaxRank) return false;
  return true;
}

}  // namespace

size_t tc_fwd_ws_bytes(int64_t M, int64_t N, int64_t K, int r, bool w16) { return FwdWs(M, N, K, r, w16).total; }

size_t tc_bwd_ws_bytes(int64_t M, int64_t N, int64_t K, int r, bool w16) { return BwdWs(M, N, K, r, w16).total; }

// Forward: W in bf16 with prep (A and B in bf16) -> T = x A^T (skinny tcgen05) ->
// T and bf16(s T) -> GEMM with the (s T) B^T slab.
cudaError_t tc_forward(const LinearArgs& a, bool f16, const void* x, const float* A, const float* B, void* y,
                       float* T, void* ws, int* status, cudaStream_t st, const void* w16) {
  const FwdWs L(a.M, a.N, a.K, a.r, w16 != nullptr);
  char* w = static_cast<char*>(ws);
  void* sTp = w + L.sTp;
  void* Bp = w + L.Bp;
  void* Aq = w + L.Aq;
  auto* part = reinterpret_cast<float*>(w + L.part);
  const void* wb = w16 != nullptr ? w16 : w + L.wb;
  const int rp = padded_rank(a.r), nq = adapter_nq(a.r);
  PrepBuilder prep(f16);
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
    b.kind = kStageRows;         // B as the slab's feature side: [N][rp]
    b.r = a.r;
    b.width = rp;
    b.scale = 1.0f;
    b.src = B;
    b.dst = Bp;
    b.count = a.N * rp;
    prep.add(b);
    prep.add(zero_flags_job(w + L.flags));
  }
  cudaError_t e = decode_weight(a, f16, w + L.wb, prep, st, w16);
  if (e != cudaSuccess) return e;
  {  // T = x A^T: rows M, reduction over K along x's rows; T (fp32) and 16-bit s T for the slab
    AdapterPassArgs t{};
    t.X = x;
    t.x_inner = a.K;
    t.x_outer = a.M;
    t.Q = Aq;
    t.q_cols = a.K;
    t.r = a.r;
    t.rows = a.M;
    t.red = a.K;
    t.partial = part;
    t.scale = 1.0f;
    t.f32 = T;
    t.b_rows = sTp;
    t.rp = rp;
    t.scale_b = a.s;
    t.f16 = f16 ? 1 : 0;
    if ((e = adapter_run(&t, 1, status, st)) != cudaSuccess) return e;
  }
  return fwd_gemm(a, f16, x, wb, Bp, sTp, part, w + L.flags, y, status, st);
}

// Backward: W in bf16 with prep (B^T, T^T, zeroed G^T, A^T in bf16) -> G = dY B ->
// G, bf16(s G), bf16(G)^T -> dB = s dY^T T -> GEMM for dX with the (s G) A slab ->
// dA = s G^T x.
cudaError_t tc_backward(const LinearArgs& a, bool f16, const void* dy, const void* x, const float* T,
                        const float* A, const float* B, void* dx, float* dA, float* dB, float* G, void* ws,
                        int* status, cudaStream_t st, const void* w16) {
  const BwdWs L(a.M, a.N, a.K, a.r, w16 != nullptr);
  char* w = static_cast<char*>(ws);
  auto* part = reinterpret_cast<float*>(w + L.part);
  const void* wb = w16 != nullptr ? w16 : w + L.wb;
  PrepBuilder prep(f16);
  {
    std::vector<PrepJob> jobs;
    bwd_prep_jobs(a, T, A, B, L, w, true, &jobs);
    for (const PrepJob& j : jobs) prep.add(j);
  }
  cudaError_t e = decode_weight(a, f16, w + L.wb, prep, st, w16);
  if (e != cudaSuccess) return e;
  if ((e = gdb_pass(a, f16, dy, G, dB, L, w, w + L.Gt, pad8(a.M), status, st)) != cudaSuccess) return e;
  if ((e = dx_gemm(a, f16, dy, wb, w + L.ApT, w + L.sGp, part, w + L.flags, dx, status, st)) != cudaSuccess) return e;
  // dA = s G^T x: rows K, reduction over M down x's columns; written as [r][K]
  AdapterPassArgs da{};
  da.X = x;
  da.x_inner = a.K;
  da.x_outer = a.M;
  da.mn_major = true;
  da.Q = w + L.Gt;
  da.q_cols = pad8(a.M);
  da.r = a.r;
  da.rows = a.K;
  da.red = a.M;
  da.partial = part;
  da.scale = a.s;
  da.f32 = dA;
  da.f32_t = 1;
  da.f16 = f16 ? 1 : 0;
  return adapter_run(&da, 1, status, st);
}

size_t tc_fwd_run_ws_bytes(const TcFwdItem* it, int n) {
  if (!run_ok(it, n)) return 0;
  return FwdRunWs(it, n, XSets(it, n)).total;
}

size_t tc_bwd_run_ws_bytes(const TcBwdItem* it, int n) {
  if (!run_ok(it, n)) return 0;
  return BwdRunWs(it, n, XSets(it, n)).total;
}

// Forward of a run: the stored weights decoded by one batched launch, the staging of every
// item, one launch with a T pass per input set (Q = the set's A rows, each item's padded to
// 16, stacked) and one finish, then each item's GEMM.
cudaError_t tc_forward_run(const TcFwdItem* it, int n, bool f16, void* ws, int* status, cudaStream_t st) {
  if (!run_ok(it, n)) return cudaErrorInvalidValue;
  const XSets xs(it, n);
  const FwdRunWs Rw(it, n, xs);
  char* w = static_cast<char*>(ws);
  std::vector<PrepJob> jobs;
  Nf4View views[kTcGroupMax];
  void* outs[kTcGroupMax];
  AdapterOut tout[kTcGroupMax];
  int m = 0;
  for (int g = 0; g < xs.n; ++g) {
    for (int i = xs.first[g]; i < xs.first[g + 1]; ++i) {
      const LinearArgs& a = it[i].a;
      const FwdWs L(a.M, a.N, a.K, a.r, it[i].w16 != nullptr);
      char* wi = w + Rw.item[i];
      const int rp = padded_rank(a.r), nq = adapter_nq(a.r);
      PrepJob j{};
      j.kind = kStageRowsDirect;   // A as rows col .. col + nq of the set's stacked Q
      j.r = a.r;
      j.src = it[i].A;
      j.dst = w + Rw.Aq[g] + 2 * static_cast<size_t>(xs.col[i]) * a.K;
      j.cols = a.K;
      j.count = static_cast<int64_t>(nq) * a.K;
      jobs.push_back(j);
      PrepJob b{};
      b.kind = kStageRows;         // B as the slab's feature side: [N][rp]
      b.r = a.r;
      b.width = rp;
      b.scale = 1.0f;
      b.src = it[i].B;
      b.dst = wi + L.Bp;
      b.count = a.N * rp;
      jobs.push_back(b);
      jobs.push_back(zero_flags_job(wi + L.flags));
      if (it[i].w16 == nullptr) {
        views[m] = a.W;
        outs[m] = wi + L.wb;
        ++m;
      }
      AdapterOut& o = tout[i];
      o = AdapterOut{};
      o.col0 = xs.col[i];
      o.r = a.r;
      o.scale = 1.0f;
      o.f32 = it[i].T;
      o.b_rows = wi + L.sTp;
      o.rp = rp;
      o.scale_b = a.s;
    }
  }
  cudaError_t e = cudaSuccess;
  if (m > 0) {
    KernelTimer timer(NF4_TIME_WEIGHT_DECODE, st);
    e = launch_dequantize_batch(views, outs, m, f16 ? NF4_F16 : NF4_BF16, st);
  }
  if (e == cudaSuccess) e = run_prep(jobs, f16, st);
  if (e != cudaSuccess) return e;
  AdapterPassArgs t[kTcGroupMax] = {};
  for (int g = 0; g < xs.n; ++g) {
    const TcFwdItem& f = it[xs.first[g]];
    t[g].X = f.x;
    t[g].x_inner = f.a.K;
    t[g].x_outer = f.a.M;
    t[g].Q = w + Rw.Aq[g];
    t[g].q_cols = f.a.K;
    t[g].r = xs.nqt[g];
    t[g].rows = f.a.M;
    t[g].red = f.a.K;
    t[g].partial = reinterpret_cast<float*>(w + Rw.part[g]);
    t[g].f16 = f16 ? 1 : 0;
    t[g].outs = tout + xs.first[g];
    t[g].nouts = xs.first[g + 1] - xs.first[g];
  }
  share_targets(t, xs.n);
  if ((e = adapter_run(t, xs.n, status, st)) != cudaSuccess) return e;
  for (int i = 0; i < n; ++i) {
    const LinearArgs& a = it[i].a;
    const FwdWs L(a.M, a.N, a.K, a.r, it[i].w16 != nullptr);
    char* wi = w + Rw.item[i];
    const void* wb = it[i].w16 != nullptr ? it[i].w16 : wi + L.wb;
    e = fwd_gemm(a, f16, it[i].x, wb, wi + L.Bp, wi + L.sTp, wi + L.part, wi + L.flags, it[i].y, status, st);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

// Backward of a run: decode and staging as above (a zeroed G^T [nqt][Mp] per input set), one
// launch with every item's G and dB passes (each pair split as in the single call) and one
// finish (each item's 16-bit G^T into its rows of its set's G^T), each item's dX GEMM, then
// one launch with a dA pass per input set and one finish.
cudaError_t tc_backward_run(const TcBwdItem* it, int n, bool f16, void* ws, int* status, cudaStream_t st) {
  if (!run_ok(it, n)) return cudaErrorInvalidValue;
  const XSets xs(it, n);
  const BwdRunWs Rw(it, n, xs);
  char* w = static_cast<char*>(ws);
  std::vector<PrepJob> jobs;
  for (int g = 0; g < xs.n; ++g) {
    const int64_t M = it[xs.first[g]].a.M, Mp = pad8(M);
    PrepJob z{};                 // the set's G^T starts zero
    z.kind = kStageTransposed;
    z.r = 0;
    z.width = Mp;
    z.dst = w + Rw.Gt[g];
    z.cols = M;
    z.count = static_cast<int64_t>(xs.nqt[g]) * Mp;
    jobs.push_back(z);
  }
  Nf4View views[kTcGroupMax];
  void* outs[kTcGroupMax];
  AdapterOut aout[kTcGroupMax];
  AdapterPassArgs gd[2 * kTcGroupMax] = {};
  int m = 0;
  for (int g = 0; g < xs.n; ++g) {
    for (int i = xs.first[g]; i < xs.first[g + 1]; ++i) {
      const LinearArgs& a = it[i].a;
      const BwdWs L(a.M, a.N, a.K, a.r, it[i].w16 != nullptr);
      char* wi = w + Rw.item[i];
      const int64_t Mp = pad8(a.M);
      bwd_prep_jobs(a, it[i].T, it[i].A, it[i].B, L, wi, false, &jobs);
      if (it[i].w16 == nullptr) {
        views[m] = a.W;
        outs[m] = wi + L.wb;
        ++m;
      }
      gdb_args(a, f16, it[i].dy, reinterpret_cast<float*>(w + Rw.G[i]), it[i].dB, L, wi,
               w + Rw.Gt[g] + 2 * static_cast<size_t>(xs.col[i]) * Mp, Mp, &gd[2 * i]);
      adapter_pair_targets(gd[2 * i].rows, gd[2 * i].red, gd[2 * i + 1].rows, gd[2 * i + 1].red, &gd[2 * i].target,
                           &gd[2 * i + 1].target);
      AdapterOut& o = aout[i];
      o = AdapterOut{};
      o.col0 = xs.col[i];
      o.r = a.r;
      o.scale = a.s;
      o.f32 = it[i].dA;
      o.f32_t = 1;
    }
  }
  cudaError_t e = cudaSuccess;
  if (m > 0) {
    KernelTimer timer(NF4_TIME_WEIGHT_DECODE, st);
    e = launch_dequantize_batch(views, outs, m, f16 ? NF4_F16 : NF4_BF16, st);
  }
  if (e == cudaSuccess) e = run_prep(jobs, f16, st);
  if (e == cudaSuccess) e = adapter_run(gd, 2 * n, status, st);
  if (e != cudaSuccess) return e;
  for (int i = 0; i < n; ++i) {
    const LinearArgs& a = it[i].a;
    const BwdWs L(a.M, a.N, a.K, a.r, it[i].w16 != nullptr);
    char* wi = w + Rw.item[i];
    const void* wb = it[i].w16 != nullptr ? it[i].w16 : wi + L.wb;
    e = dx_gemm(a, f16, it[i].dy, wb, wi + L.ApT, wi + L.sGp, wi + L.part, wi + L.flags, it[i].dx, status, st);
    if (e != cudaSuccess) return e;
  }
  // dA of every item: rows K, reduction over M down x's columns, Q = its set's G^T
  AdapterPassArgs da[kTcGroupMax] = {};
  for (int g = 0; g < xs.n; ++g) {
    const TcBwdItem& f = it[xs.first[g]];
    const int64_t Mp = pad8(f.a.M);
    da[g].X = f.x;
    da[g].x_inner = f.a.K;
    da[g].x_outer = f.a.M;
    da[g].mn_major = true;
    da[g].Q = w + Rw.Gt[g];
    da[g].q_cols = Mp;
    da[g].r = xs.nqt[g];
    da[g].rows = f.a.K;
    da[g].red = f.a.M;
    da[g].partial = reinterpret_cast<float*>(w + Rw.part[g]);
    da[g].f16 = f16 ? 1 : 0;
    da[g].outs = aout + xs.first[g];
    da[g].nouts = xs.first[g + 1] - xs.first[g];
  }
  share_targets(da, xs.n);
  return adapter_run(da, xs.n, status, st);
}

}  // namespace qnf4
