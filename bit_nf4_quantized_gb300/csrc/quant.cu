// NF4 blockwise quantization with nested dynamic8 absmax, and dequantization.
//
// Format and decode: "Native model adaptation and NF4", section "Packed NF4 and the
// portable QLoRA profile" (64-element absmax blocks, the 16-value NF4 codebook, two
// codes per byte, block maxima centred by their global FP32 mean and quantized with
// dynamic8 in blocks of 256) and section "Fused GPU NF4 decodes inside the matrix
// kernel".  Deterministic, byte-identical requantization: "NF4 Layer Streaming --
// Gate results", section "P3 is solved".
//
// Lane mapping of the block and decode kernels: a warp walks rows of 1024 elements and lane
// l owns elements 32l .. 32l + 31 of a row, so a lane pair holds one 64-element block.
//
// quantize = two launches (a call, or a batch of up to 8 tensors):
//   1. nf4_encode_blocks: absmax, 4-bit codes, packing; with double quantization per 256-block
//      group the float64 pairwise-tree sum of the absmax values, and, by the CTA that counts a
//      tensor's last group, the tree over the group sums -> offset.
//   2. nf4_encode_nested (double quantization): centre, nested absmax per group, dynamic8 codes.
#include "common.cuh"
#include "decode.cuh"
#include "prep.cuh"

#include <algorithm>
#include <atomic>
#include <mutex>

namespace qnf4 {
namespace {

constexpr int kQuantThreads = 256;                 // 8 warps

__device__ __forceinline__ int nf4_encode(float v, const float* thr) {
  int c = (v >= thr[7]) ? 8 : 0;
  c += (v >= thr[c + 3]) ? 4 : 0;
  c += (v >= thr[c + 1]) ? 2 : 0;
  c += (v >= thr[c]) ? 1 : 0;
  return c;
}

__device__ __forceinline__ int dyn8_encode(float v, const float* thr) {
  int c = 0;
#pragma unroll
  for (int step = 128; step >= 1; step >>= 1) c += (v >= thr[c + step - 1]) ? step : 0;
  return c;
}

__device__ __forceinline__ uint32_t max_u16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.u16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// The raw bits of the lane's 32 elements from e0 (16 words of two bf16, or 32 fp32
// words), zero past numel.  The input is read once: read-only loads that allocate no L1
// line, 32 bytes per instruction when the input is 32-byte aligned (kV8), else 16.
template <typename Tin, bool kV8>
__device__ __forceinline__ void lane_words(const Tin* __restrict__ x, int64_t numel, int64_t e0,
                                           uint32_t (&w)[8 * sizeof(Tin)]) {
  constexpr int kW = 8 * sizeof(Tin);
  if (e0 + 32 <= numel) {
    const uint32_t* p = reinterpret_cast<const uint32_t*>(x + e0);
    if constexpr (kV8) {
#pragma unroll
      for (int i = 0; i < kW / 8; ++i)
        asm volatile("ld.global.nc.L1::no_allocate.v8.u32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                     : "=r"(w[8 * i]), "=r"(w[8 * i + 1]), "=r"(w[8 * i + 2]), "=r"(w[8 * i + 3]),
                       "=r"(w[8 * i + 4]), "=r"(w[8 * i + 5]), "=r"(w[8 * i + 6]), "=r"(w[8 * i + 7])
                     : "l"(p + 8 * i));
    } else {
#pragma unroll
      for (int i = 0; i < kW / 4; ++i)
        asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(w[4 * i]), "=r"(w[4 * i + 1]), "=r"(w[4 * i + 2]), "=r"(w[4 * i + 3])
                     : "l"(p + 4 * i));
    }
  } else {   // ragged tail
    const uint16_t* x16 = reinterpret_cast<const uint16_t*>(x);
    const uint32_t* x32 = reinterpret_cast<const uint32_t*>(x);
#pragma unroll
    for (int i = 0; i < kW; ++i) {
      if (sizeof(Tin) == 4) {
        w[i] = (e0 + i < numel) ? x32[e0 + i] : 0u;
      } else {
        const uint32_t lo = (e0 + 2 * i < numel) ? x16[e0 + 2 * i] : 0u;
        const uint32_t hi = (e0 + 2 * i + 1 < numel) ? x16[e0 + 2 * i + 1] : 0u;
        w[i] = lo | (hi << 16);
      }
    }
  }
}

// Element i of the lane as fp32.
template <typename Tin>
__device__ __forceinline__ float lane_elem(const uint32_t (&w)[8 * sizeof(Tin)], int i) {
  if (sizeof(Tin) == 4) return __uint_as_float(w[i]);
  return __uint_as_float((i & 1) ? (w[i >> 1] & 0xFFFF0000u) : (w[i >> 1] << 16));
}

// Largest |x| of the lane's elements as fp32 bits (bf16: an integer max over the 15-bit
// magnitudes, two at a time, which orders subnormals, Inf and NaN as the fp32 bit
// patterns do).
template <typename Tin>
__device__ __forceinline__ uint32_t lane_absmax_bits(const uint32_t (&w)[8 * sizeof(Tin)]) {
  if (sizeof(Tin) == 4) {
    uint32_t mb = 0;
#pragma unroll
    for (int i = 0; i < 32; ++i) mb = max(mb, w[i] & 0x7FFFFFFFu);
    return mb;
  }
  uint32_t m2 = 0;
#pragma unroll
  for (int k = 0; k < 16; ++k) m2 = max_u16x2(m2, w[k] & 0x7FFF7FFFu);
  return max(m2 & 0xFFFFu, m2 >> 16) << 16;
}

// Bucket row (bits(q') >> 17) of the lane's table copy; tab_base is the shared-memory address
// of row 0 of the copy minus 8191 rows.
__device__ __forceinline__ uint2 bucket_row(uint32_t tab_base, uint32_t qb) {
  uint2 e;
  asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(e.x), "=r"(e.y) : "r"(tab_base + ((qb >> 17) << 7)));
  return e;
}

// Codes of one lane (32 elements, one half block) with the block maximum a = bits mb.
// Words: element i sits in word i / 8, byte (i % 8) / 2, high nibble for even i; a word is
// built by shifting in elements 6, 7, 4, 5, 2, 3, 0, 1 of its eight.
//   bf16 input, a in [2^-126, 2^126), cut table valid: code = base + (bits(q') >= cut),
//     q' = fl(x*r + 3), r = RN(1/a), from the bucket row of q' (no band: see EncodeTables).
//   fp32 input: q = x*r and q' pick the bucket; code = base + (q >= hi); a q inside the
//     band [lo, hi) marks the lane unsure, and an unsure lane (or a, r not finite, or the
//     bucket table unusable) is redone with the IEEE quotient RN(x / a).
template <typename Tin>
__device__ __forceinline__ void lane_codes(const uint32_t (&w)[8 * sizeof(Tin)], uint32_t mb, uint32_t tab_base,
                                           bool fast_ok, const float* thr, uint32_t (&words)[4]) {
  const float a = __uint_as_float(mb);
  if (a == 0.0f) {
#pragma unroll
    for (int j = 0; j < 4; ++j) words[j] = 0x77777777u;     // every code is that of 0.0
    return;
  }
  const float r = __frcp_rn(a);
  bool exact;
  if (sizeof(Tin) == 2) {
    exact = !(fast_ok && mb >= 0x00800000u && mb < 0x7E800000u);
    if (!exact) {
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        uint32_t acc = 0;
#pragma unroll
        for (int t = 0; t < 8; ++t) {
          const int i = 8 * j + (6 - 2 * (t >> 1)) + (t & 1);
          const uint32_t qb = __float_as_uint(fmaf(lane_elem<Tin>(w, i), r, 3.0f));
          const uint2 e = bucket_row(tab_base, qb);
          acc = (acc << 4) + e.y + (qb >= e.x ? 1u : 0u);
        }
        words[j] = acc;
      }
    }
  } else {
    exact = !(fast_ok && isfinite(r) && mb < 0x7F800000u);
    if (!exact) {
      bool unsure = false;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        uint32_t acc = 0;
#pragma unroll
        for (int t = 0; t < 8; ++t) {
          const int i = 8 * j + (6 - 2 * (t >> 1)) + (t & 1);
          const float v = lane_elem<Tin>(w, i);
          const float q = v * r;
          const uint32_t qb = __float_as_uint(fmaf(v, r, 3.0f));
          const uint2 e = bucket_row(tab_base, qb);
          const float lo = __uint_as_float(e.x), hi = __uint_as_float(e.y);
          unsure |= (q >= lo) & (q < hi);
          acc = (acc << 4) + (e.x & 15u) + (q >= hi ? 1u : 0u);
        }
        words[j] = acc;
      }
      exact = unsure;
    }
  }
  if (exact) {  // rare: the lane again with the IEEE quotient
#pragma unroll
    for (int j = 0; j < 4; ++j) words[j] = 0u;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const uint32_t c = static_cast<uint32_t>(nf4_encode(__fdiv_rn(lane_elem<Tin>(w, i), a), thr));
      words[i >> 3] |= c << (((i >> 1) & 3) * 8 + ((i & 1) ? 0 : 4));
    }
  }
}

// One row of 1024 elements from the lane's words: block maxima, codes, the packed bytes and
// the fp32 maxima; the group's copy of each maximum goes to gs_slot.  Returns true if
// the lane's block holds a non-finite value.
template <typename Tin>
__device__ __forceinline__ bool encode_row(const uint32_t (&w)[8 * sizeof(Tin)], int64_t e0, int64_t numel,
                                           uint8_t* __restrict__ packed, float* __restrict__ absmax,
                                           float* gs_slot, uint32_t tab_base, bool fast_ok,
                                           const float* thr, int lane) {
  uint32_t mb = lane_absmax_bits<Tin>(w);
  mb = max(mb, __shfl_xor_sync(0xffffffffu, mb, 1));  // the lane pair holds one block
  uint32_t words[4];
  lane_codes<Tin>(w, mb, tab_base, fast_ok, thr, words);
  if (e0 + 31 >= numel) {  // ragged tail: codes past numel are 0 (the pad nibble of an odd tail)
    const int64_t vc = numel - e0;
#pragma unroll
    for (int i = 0; i < 32; ++i)
      if (i >= vc) words[i >> 3] &= ~(0xFu << (((i >> 1) & 3) * 8 + ((i & 1) ? 0 : 4)));
  }
  if (e0 + 31 < numel) {
    *reinterpret_cast<uint4*>(packed + (e0 >> 1)) = make_uint4(words[0], words[1], words[2], words[3]);
  } else if (e0 < numel) {
    const int64_t nbytes = (numel - e0 + 1) / 2;
#pragma unroll
    for (int b = 0; b < 16; ++b)
      if (b < nbytes) packed[(e0 >> 1) + b] = static_cast<uint8_t>(words[b >> 2] >> (8 * (b & 3)));
  }
  if ((lane & 1) == 0) {
    const float a = __uint_as_float(mb);
    if (e0 < numel) absmax[e0 >> 6] = a;
    *gs_slot = (e0 < numel) ? a : 0.0f;
  }
  return mb >= 0x7F800000u;
}

// Sum of a group's 256 block maxima (non-negative fp32, gs[0..255]) as the float64 pairwise
// tree s[i] += s[i + h], h = 128, 64, ..., 1 computes it, by one warp; the result is in lane 0.
// Write each maximum as M * 2^(E - 150) with an integer M < 2^24 and E = max(biased exponent, 1).
// When the group's E span at most 21 (and all are finite), every partial sum of the tree is a
// multiple of 2^(Emin - 150) below 2^53 of those units, so each float64 addition is exact and
// the tree's result is the exact sum: it is formed in integers (two 32-bit warp sums of the
// 24-bit halves) and scaled once by a power of two.  Otherwise the tree runs in float64, lane l
// holding s[l + 32 m]: the levels h >= 32 add within the lane, the rest across lanes.
__device__ __forceinline__ double group_sum(const float* gs, int lane) {
  uint32_t v[kNested / 32];
  uint32_t emin = 255u, emax = 0u;
#pragma unroll
  for (int m = 0; m < kNested / 32; ++m) {
    v[m] = __float_as_uint(gs[lane + 32 * m]);
    const uint32_t e = max(v[m] >> 23, 1u);
    if (v[m] != 0u) emin = min(emin, e), emax = max(emax, e);
  }
  emin = __reduce_min_sync(0xffffffffu, emin);
  emax = __reduce_max_sync(0xffffffffu, emax);
  if (emax == 0u) return 0.0;   // every maximum is +0
  if (emax < 255u && emax - emin <= 21u) {
    uint64_t acc = 0;
#pragma unroll
    for (int m = 0; m < kNested / 32; ++m) {
      const uint32_t be = v[m] >> 23;
      const uint64_t mant = (v[m] & 0x7FFFFFu) | (be != 0u ? 0x800000u : 0u);
      if (v[m] != 0u) acc += mant << (max(be, 1u) - emin);
    }
    const uint32_t lo = __reduce_add_sync(0xffffffffu, static_cast<uint32_t>(acc & 0xFFFFFFu));
    const uint32_t hi = __reduce_add_sync(0xffffffffu, static_cast<uint32_t>(acc >> 24));
    const uint64_t total = (static_cast<uint64_t>(hi) << 24) + lo;   // < 2^53: converts exactly
    const double unit = __longlong_as_double(static_cast<long long>(static_cast<int>(emin) - 150 + 1023) << 52);
    return __dmul_rn(__ull2double_rn(total), unit);
  }
  double t[kNested / 32];
#pragma unroll
  for (int m = 0; m < kNested / 32; ++m) t[m] = static_cast<double>(__uint_as_float(v[m]));
#pragma unroll
  for (int h = kNested / 64; h >= 1; h >>= 1)
#pragma unroll
    for (int m = 0; m < h; ++m) t[m] += t[m + h];
#pragma unroll
  for (int h = 16; h >= 1; h >>= 1) t[0] += __shfl_down_sync(0xffffffffu, t[0], h);
  return t[0];
}

// The offset: the float64 pairwise tree s[i] += s[i + h], h = p2/2, ..., 1, over the group
// sums gs padded with zeros to p2 entries, divided by nb and rounded once to fp32, by one CTA
// (the last of the block pass to finish).  Levels above 8192 entries run in place in gs (the
// workspace holds p2 entries); then each of the (at most) 1024 entries left after the next
// levels is summed from its column of up to 8 loads in registers, in the tree's own order; the
// levels down to 32 run in shared memory `sm` and the last five across the lanes of warp 0.
// Returns the offset in thread 0.
__device__ __forceinline__ float offset_tree(double* gs, int64_t ng, int64_t p2, int64_t nb, double* sm) {
  int64_t n = p2, valid = ng;   // live entries, of which the first `valid` hold data
  for (; n > 8192; n /= 2) {
    const int64_t h = n / 2;
    for (int64_t i = threadIdx.x; i < h; i += kQuantThreads) {
      const double a = i < valid ? gs[i] : 0.0;
      const double b = i + h < valid ? gs[i + h] : 0.0;
      gs[i] = a + b;
    }
    valid = valid < h ? valid : h;
    __syncthreads();
  }
  // entry i of the first w = min(n, 1024) entries is the tree over column j = 0 .. m-1 of
  // gs[i + w j] (m = n / w), whose pairs are (j, j + m/2), then (j, j + m/4), ...
  // (read from L2, where the other CTAs' writes are; with m <= 4 two entries a thread at a
  // time, so that 8 loads are in flight)
  const int64_t w = n < 1024 ? n : 1024, m = n / w;
  if (m <= 4) {
#pragma unroll 1
    for (int64_t i0 = threadIdx.x; i0 < w; i0 += 2 * kQuantThreads) {
      double c[2][4];
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int64_t i = i0 + e * kQuantThreads;
#pragma unroll
        for (int j = 0; j < 4; ++j) c[e][j] = (i < w && j < m && i + w * j < valid) ? __ldcg(gs + i + w * j) : 0.0;
      }
#pragma unroll
      for (int e = 0; e < 2; ++e) {
#pragma unroll
        for (int h = 2; h >= 1; h >>= 1)
          if (h < m)
#pragma unroll
            for (int j = 0; j < h; ++j) c[e][j] = c[e][j] + c[e][j + h];
        if (i0 + e * kQuantThreads < w) sm[i0 + e * kQuantThreads] = c[e][0];
      }
    }
  } else {
#pragma unroll 1
    for (int64_t i = threadIdx.x; i < w; i += kQuantThreads) {
      double c[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) c[j] = (i + w * j < valid) ? __ldcg(gs + i + w * j) : 0.0;
#pragma unroll
      for (int h = 4; h >= 1; h >>= 1)
#pragma unroll
        for (int j = 0; j < h; ++j) c[j] = c[j] + c[j + h];
      sm[i] = c[0];
    }
  }
  __syncthreads();
  for (n = w; n > 32; n /= 2) {
    const int64_t h = n / 2;
    for (int64_t i = threadIdx.x; i < h; i += kQuantThreads) sm[i] = sm[i] + sm[i + h];
    __syncthreads();
  }
  float offset = 0.0f;
  if (threadIdx.x < 32) {
    double t = threadIdx.x < n ? sm[threadIdx.x] : 0.0;
    for (int64_t h = n / 2; h >= 1; h /= 2) t += __shfl_down_sync(0xffffffffu, t, static_cast<int>(h));
    if (threadIdx.x == 0) offset = __double2float_rn(__ddiv_rn(t, static_cast<double>(nb)));
  }
  return offset;
}

// Nested quantization (per nested group of 256 maxima): c = a - offset, m = max |c| over the
// group, code = dyn8 code of RN(c / m), i.e. the number of thresholds at or below it.
// Rows of the dyn8 search: |q| in [2^-7, 1] split by sign and by the float's top six
// fraction bits (64 rows a binade, 449 rows a sign, the last holding 1.0).  Each CTA derives
// every row from the thresholds: with lo and hi the row's most negative and most positive
// floats, base = code(lo), and if code(hi) <= base + 1 then code(q) = base + (q >= thr[base])
// for every q of the row (code is a step function that crosses at most one threshold there);
// a row that crosses more (none does for the dyn8 values) is marked and searched in full.
constexpr uint32_t kDynRow0 = 7680u;          // bits(2^-7) >> 17
constexpr int kDynRows = 449;
constexpr uint32_t kDynAmbiguous = 0xFFFFFFFFu;

__device__ __forceinline__ uint32_t dyn8_code(float q, const uint2* rows, const float* thr) {
  const uint32_t qb = __float_as_uint(q), ab = qb & 0x7FFFFFFFu;
  if (ab >= (kDynRow0 << 17) && ab < ((kDynRow0 + kDynRows) << 17)) {
    const uint2 e = rows[(ab >> 17) - kDynRow0 + (qb >> 31) * kDynRows];
    if (e.y != kDynAmbiguous) return e.y + (q >= __uint_as_float(e.x) ? 1u : 0u);
  }
  return static_cast<uint32_t>(dyn8_encode(q, thr));   // small |q|, NaN, or a marked row
}

// One tensor of a block pass.  Its groups are numbers g0 .. g0 + ng - 1 of the launch's
// concatenated group list.
struct EncodeItem {
  const void* x;
  int64_t numel, ng, g0, p2;
  uint8_t* packed;
  float* absmax;          // fp32 maxima: the output, or (double quant) the workspace's copy
  double* group_sum;      // double quant: the workspace's group sums, p2 entries; else null
  unsigned* ticket;       // double quant: a zero counter of the library's ticket pool
  float* offset;          // double quant: the tensor's offset
};
constexpr int kEncodeBatch = kQuantBatchMax;
struct EncodeBatch {
  EncodeItem it[kEncodeBatch];
  int n;
  int64_t total;          // groups of all items
  unsigned* work;         // with any double-quant item: a zero counter handing out groups
};

__device__ __forceinline__ int item_of(const EncodeItem* items, int n, int64_t g) {
  int i = 0;
#pragma unroll 1
  while (i + 1 < n && g >= items[i + 1].g0) ++i;
  return i;
}

// Block pass: absmax, 4-bit codes and packing, one nested group (256 blocks, 16384
// elements) at a time, over the groups of up to 8 tensors of one input type; with double
// quantization also the float64 pairwise-tree sum of each group's absmax.  Persistent (the grid
// is the CTAs resident at once): CTA c takes group c first, then, without double quantization,
// c + G, c + 2G, ... (G = gridDim.x); with any double-quant item the further groups are handed
// out by a counter in the order CTAs ask, so that CTAs the warp schedulers serve less often take
// fewer groups and all finish together.  Warp w codes rows 2w and 2w + 1 of a group (1024
// elements each; lane l elements 32l .. 32l + 31, so a lane pair holds one block); after coding
// a row it loads the same row of its next group into the row's registers, so one row per warp
// is always in flight while the other is coded.  With the counter, thread 0 asks for the group
// after next while the CTA codes a group, and the CTA's threads meet once per group, which
// publishes the answer.  With double quantization the group's 256 maxima meet in shared memory
// (two buffers, by group parity) and one warp, rotating, sums them; it then fences and counts
// the group on its tensor's ticket, and the warp that counts a tensor's last group has its CTA
// sum the tensor's group sums into the offset after the CTA's next meeting, then put the
// counter back to zero (the arrival pattern of a grid barrier, without any waiting).
template <typename Tin, bool kV8>
__global__ void __launch_bounds__(kQuantThreads, sizeof(Tin) == 2 ? 3 : 2)
nf4_encode_blocks(EncodeBatch b, EncodeTables tabs, int* status) {
  __shared__ float thr[16];
  // bucket rows, 16 copies: the 8-byte lookups of a warp are served half a warp at a time,
  // and lanes l, l + 16 never meet in one bank access.  bf16: {cut, base}; fp32: {bits of
  // lo with the base code in its low 4 bits, bits of hi}
  __shared__ uint2 tab[66][16];
  __shared__ float gsum[2][kNested];
  __shared__ double tree[1024];      // the offset tree of a tensor this CTA finishes
  __shared__ EncodeItem items[kEncodeBatch];   // indexed at run time: kept out of the parameters
  __shared__ int s_next[2];          // the group after next, by group parity (counter mode)
  __shared__ int s_fin;              // item whose offset this CTA computes next, or -1
#pragma unroll
  for (int k = 0; k < kEncodeBatch; ++k)
    if (threadIdx.x == k) items[k] = b.it[k];   // static indices into the parameters
  if (threadIdx.x < 16) thr[threadIdx.x] = tabs.nf4_thr[threadIdx.x];
  for (int i = threadIdx.x; i < 66 * 16; i += kQuantThreads) {
    const int k = i >> 4;
    tab[k][i & 15] = (sizeof(Tin) == 2)
                         ? make_uint2(tabs.nf4_sep[k], tabs.nf4_sep_base[k])
                         : make_uint2(__float_as_uint(tabs.nf4_band[k][0]), __float_as_uint(tabs.nf4_band[k][1]));
  }
  __syncthreads();
  pdl_allow_next();
  pdl_wait();
  const bool fast_ok = (sizeof(Tin) == 2) ? tabs.sep_ok != 0 : tabs.bucket_ok != 0;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // row (bits(q') >> 17) of this lane's copy: q' in [2, 4] gives rows 8191 .. 8256 of the
  // shifted origin, i.e. table rows 0 .. 65 (rows are 128 bytes: 16 copies of 8)
  const uint32_t tab_base = static_cast<uint32_t>(__cvta_generic_to_shared(&tab[0][lane & 15])) - 8191u * 128u;
  constexpr int kW = 8 * sizeof(Tin);
  const int64_t lane_off = warp * 2048 + 32 * lane;
  const int slot = warp * 32 + (lane >> 1);    // block of the group held by the lane pair (row 2w)
  const bool dyn = b.work != nullptr;
  // the counter hands out groups G, G + 1, ...; every CTA asks until it is refused once, so
  // the counter ends at `total` and the CTA given total - 1 puts it back to zero
  // (group numbers fit in 31 bits: the host checks the total)
  const int total = static_cast<int>(b.total);
  auto ask = [&]() -> int {
    const unsigned v = atomicAdd(b.work, 1u);
    if (static_cast<int>(v) == total - 1) *b.work = 0u;
    return static_cast<int>(gridDim.x + v);
  };
  int g = blockIdx.x, gn = g + gridDim.x;
  if (dyn) {
    if (threadIdx.x == 0) {
      s_next[0] = ask();
      s_fin = -1;
    }
    __syncthreads();
    gn = s_next[0];
  }
  int ci = item_of(items, b.n, g);
  uint32_t wa[kW], wb[kW];
  {
    const EncodeItem& e = items[ci];
    const Tin* x = static_cast<const Tin*>(e.x);
    lane_words<Tin, kV8>(x, e.numel, (g - e.g0) * kGroupElems + lane_off, wa);
    lane_words<Tin, kV8>(x, e.numel, (g - e.g0) * kGroupElems + lane_off + 1024, wb);
  }
  // the offset of item f, by the whole CTA (its last group sum is written and counted)
  auto finish = [&](int f) {
    __syncthreads();   // every thread has read s_fin
    if (threadIdx.x == 0) s_fin = -1;
    __threadfence();
    const EncodeItem& e = items[f];
    const float off = offset_tree(e.group_sum, e.ng, e.p2, (e.numel + kBlock - 1) / kBlock, tree);
    if (threadIdx.x == 0) {
      *e.offset = off;
      *e.ticket = 0u;
    }
    __syncthreads();   // `tree` is free again
  };
  bool nonfinite = false;
#pragma unroll 1
  for (int it = 0; g < total; ++it) {
    const EncodeItem& e = items[ci];
    const int64_t gl = g - e.g0;                 // group within the tensor
    const int64_t e0 = gl * kGroupElems + lane_off;
    const int ni = gn < total ? item_of(items, b.n, gn) : ci;
    if (dyn && threadIdx.x == 0) s_next[(it + 1) & 1] = gn < total ? ask() : total;
    float* gs = gsum[it & 1];
    nonfinite |= encode_row<Tin>(wa, e0, e.numel, e.packed, e.absmax, gs + slot, tab_base, fast_ok, thr, lane);
    if (gn < total)
      lane_words<Tin, kV8>(static_cast<const Tin*>(items[ni].x), items[ni].numel,
                           (gn - items[ni].g0) * kGroupElems + lane_off, wa);
    nonfinite |= encode_row<Tin>(wb, e0 + 1024, e.numel, e.packed, e.absmax, gs + slot + 16, tab_base, fast_ok, thr,
                                 lane);
    if (gn < total)
      lane_words<Tin, kV8>(static_cast<const Tin*>(items[ni].x), items[ni].numel,
                           (gn - items[ni].g0) * kGroupElems + lane_off + 1024, wb);
    int gnn = gn + gridDim.x;
    if (dyn) {
      __syncthreads();
      gnn = s_next[(it + 1) & 1];
      const int f = s_fin;
      if (f >= 0) finish(f);
      if (e.group_sum != nullptr && warp == (it & 7)) {
        const double sum = group_sum(gs, lane);
        if (lane == 0) {
          e.group_sum[gl] = sum;
          __threadfence();
          if (atomicAdd(e.ticket, 1u) == static_cast<unsigned>(e.ng - 1)) s_fin = ci;
        }
      }
    }
    g = gn;
    gn = gnn;
    ci = ni;
  }
  if (dyn) {
    __syncthreads();
    const int f = s_fin;
    if (f >= 0) finish(f);
  }
  if (nonfinite) atomicCAS(status, 0, static_cast<int>(NF4_ERR_NONFINITE));
}

// Nested quantization of the block maxima: one warp per group of 256 maxima, eight per lane,
// over the groups of up to 8 tensors (numbered as in the block pass).
constexpr int kNestedWarps = 8;

struct NestedItem {
  const float* absmax;   // the fp32 maxima
  int64_t nb, ng, g0;
  const float* offset;
  uint8_t* codes;
  float* nested;
};
struct NestedBatch {
  NestedItem it[kEncodeBatch];
  int n;
  int64_t total;
};

// The lane's eight maxima of group gl of a tensor (zero past nb).
__device__ __forceinline__ void nested_load(const NestedItem& e, int64_t gl, int lane, float (&a)[8]) {
  const int64_t b0 = gl * kNested + 8 * lane;
  if (b0 + 8 <= e.nb && (reinterpret_cast<uintptr_t>(e.absmax + b0) & 15) == 0) {
    const float4 u = *reinterpret_cast<const float4*>(e.absmax + b0);
    const float4 v = *reinterpret_cast<const float4*>(e.absmax + b0 + 4);
    a[0] = u.x, a[1] = u.y, a[2] = u.z, a[3] = u.w, a[4] = v.x, a[5] = v.y, a[6] = v.z, a[7] = v.w;
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) a[i] = (b0 + i < e.nb) ? e.absmax[b0 + i] : 0.0f;
  }
}

// Persistent: warp w of CTA b takes groups b * 8 + w, then + 8 * gridDim.x, ...; while it codes
// one group the maxima of its next group are in flight.
__global__ void __launch_bounds__(kNestedWarps * 32)
nf4_encode_nested(NestedBatch b, EncodeTables tabs) {
  __shared__ float thr[256];
  __shared__ uint2 rows[2 * kDynRows];
  __shared__ NestedItem items[kEncodeBatch];
  thr[threadIdx.x] = tabs.dyn8_thr[threadIdx.x];
#pragma unroll
  for (int k = 0; k < kEncodeBatch; ++k)
    if (threadIdx.x == k) items[k] = b.it[k];
  __syncthreads();
  for (int i = threadIdx.x; i < 2 * kDynRows; i += kNestedWarps * 32) {
    const bool neg = i >= kDynRows;
    const uint32_t r0 = (kDynRow0 + static_cast<uint32_t>(neg ? i - kDynRows : i)) << 17;
    const float lo = neg ? -__uint_as_float(r0 | 0x1FFFFu) : __uint_as_float(r0);
    const float hi = neg ? -__uint_as_float(r0) : __uint_as_float(r0 | 0x1FFFFu);
    const int clo = dyn8_encode(lo, thr), chi = dyn8_encode(hi, thr);
    rows[i] = make_uint2(__float_as_uint(thr[clo]), chi - clo <= 1 ? static_cast<uint32_t>(clo) : kDynAmbiguous);
  }
  __syncthreads();
  pdl_allow_next();
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kNestedWarps;
  int64_t g = static_cast<int64_t>(blockIdx.x) * kNestedWarps + (threadIdx.x >> 5);
  if (g >= b.total) return;
  int ci = 0;
  while (ci + 1 < b.n && g >= items[ci + 1].g0) ++ci;
  float a[8];
  nested_load(items[ci], g - items[ci].g0, lane, a);
  int oi = -1;
  float offset = 0.0f;
  while (g < b.total) {
    const NestedItem& e = items[ci];
    if (oi != ci) offset = *e.offset, oi = ci;
    const int64_t gl = g - e.g0;
    float c[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) c[i] = __fsub_rn(a[i], offset);
    const int64_t gn = g + stride;
    int ni = ci;
    if (gn < b.total) {   // the next group's maxima, loaded while this one is coded
      while (ni + 1 < b.n && gn >= items[ni + 1].g0) ++ni;
      nested_load(items[ni], gn - items[ni].g0, lane, a);
    }
    const int64_t b0 = gl * kNested + 8 * lane;
    // maxima past nb do not count
    float m = b0 < e.nb ? fabsf(c[0]) : 0.0f;
#pragma unroll
    for (int i = 1; i < 8; ++i)
      if (b0 + i < e.nb) m = fmaxf(m, fabsf(c[i]));
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    uint32_t q[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) q[i] = (m > 0.0f) ? dyn8_code(__fdiv_rn(c[i], m), rows, thr) : kDyn8ZeroCode;
    if (b0 + 8 <= e.nb && (reinterpret_cast<uintptr_t>(e.codes + b0) & 7) == 0) {
      *reinterpret_cast<uint2*>(e.codes + b0) = make_uint2(q[0] | (q[1] << 8) | (q[2] << 16) | (q[3] << 24),
                                                           q[4] | (q[5] << 8) | (q[6] << 16) | (q[7] << 24));
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i)
        if (b0 + i < e.nb) e.codes[b0 + i] = static_cast<uint8_t>(q[i]);
    }
    if (lane == 0) e.nested[gl] = m;
    g = gn;
    ci = ni;
  }
}

// ---- dequantize -----------------------------------------------------------------
//
// A warp decodes 1024-element chunks: lane l takes elements 32l .. 32l+31 (one 16-byte
// load of packed codes, one block scale).  bf16 output goes through the register
// lookup table of decode.cuh (bf16(nf4[q] * a'), exact); fp32 output multiplies the
// code value by a' per element.  The lane's 64 or 128 output bytes are staged in a
// swizzled shared buffer so each global store instruction writes 512 contiguous bytes.

constexpr int kDeqThreads = 256;
constexpr int kDeqChunks = 2;                       // chunks per warp, loads issued together
constexpr int kDeqPerCta = (kDeqThreads / 32) * kDeqChunks * 1024;
static_assert(kDeqThreads == kPrepThreads, "prep jobs run in CTAs of the decode launch");

// One CTA's share of the decode: block `cta` of the dequantize grid.
template <typename Tout, bool kDQ>
__device__ __forceinline__ void decode_cta(const Nf4View& w, Tout* __restrict__ y, const DecodeTables& tabs,
                                           int64_t cta) {
  constexpr int kOutBytes = 32 * sizeof(Tout);      // per lane per chunk: 64 (bf16) or 128 (fp32)
  __shared__ float dyn8[256];
  __shared__ __align__(16) uint8_t stage[kDeqThreads / 32][32 * kOutBytes];
  for (int i = threadIdx.x; i < 256; i += kDeqThreads) dyn8[i] = tabs.dyn8[i];
  // code values replicated per lane (fp32 output only)
  float (*lut)[32] = nullptr;
  if constexpr (sizeof(Tout) == 4) {
    __shared__ float lut_f32[16][32];
    for (int i = threadIdx.x; i < 16 * 32; i += kDeqThreads) lut_f32[i >> 5][i & 31] = tabs.nf4[i >> 5];
    lut = lut_f32;
  }
  __syncthreads();
  pdl_allow_next();
  pdl_wait();
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int64_t n = w.numel;
  const float offset = kDQ ? *w.offset : 0.0f;
  uint8_t* buf = stage[warp];
  const uint32_t buf_s = static_cast<uint32_t>(__cvta_generic_to_shared(buf));
  const int64_t chunk0 = (cta * (kDeqThreads / 32) + warp) * kDeqChunks;

  uint4 pk[kDeqChunks];
  float sc[kDeqChunks];
#pragma unroll
  for (int u = 0; u < kDeqChunks; ++u) {           // all loads of the warp's chunks first
    const int64_t e0 = (chunk0 + u) * 1024 + 32 * lane;
    sc[u] = 0.0f;
    pk[u] = make_uint4(0, 0, 0, 0);
    if (e0 + 31 < n) pk[u] = __ldcs(reinterpret_cast<const uint4*>(w.packed + (e0 >> 1)));
    if (e0 < n) {
      const int64_t blk = e0 >> 6;
      if (kDQ) {
        const uint8_t c = static_cast<const uint8_t*>(w.absmax)[blk];
        sc[u] = __fadd_rn(__fmul_rn(dyn8[c], w.nested[blk >> 8]), offset);
      } else {
        sc[u] = static_cast<const float*>(w.absmax)[blk];
      }
    }
  }
#pragma unroll
  for (int u = 0; u < kDeqChunks; ++u) {
    const int64_t c0 = (chunk0 + u) * 1024;
    if (c0 >= n) break;
    const float a = sc[u];
    if (c0 + 1024 <= n) {
      const uint32_t words[4] = {pk[u].x, pk[u].y, pk[u].z, pk[u].w};
      if constexpr (sizeof(Tout) == 2) {
        uint32_t L[4], H[4];
        build_lut<Tout>(a, L, H);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          uint32_t o[4];
          decode8(words[i], L, H, o);
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(buf_s + stage_slot(4 * lane + i)),
                       "r"(o[0]), "r"(o[1]), "r"(o[2]), "r"(o[3])
                       : "memory");
        }
      } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const uint32_t wd = words[i];
          // nibbles low first: elements 1 0 3 2 5 4 7 6 of this word
          float v[8];
#pragma unroll
          for (int b = 0; b < 4; ++b) {
            v[2 * b] = __fmul_rn(lut[(wd >> (8 * b + 4)) & 15][lane], a);
            v[2 * b + 1] = __fmul_rn(lut[(wd >> (8 * b)) & 15][lane], a);
          }
#pragma unroll
          for (int h = 0; h < 2; ++h)
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(buf_s + stage_slot(8 * lane + 2 * i + h)),
                         "r"(__float_as_uint(v[4 * h])), "r"(__float_as_uint(v[4 * h + 1])),
                         "r"(__float_as_uint(v[4 * h + 2])), "r"(__float_as_uint(v[4 * h + 3]))
                         : "memory");
        }
      }
      __syncwarp();
      uint4* out = reinterpret_cast<uint4*>(y + c0);
#pragma unroll
      for (int j = 0; j < kOutBytes / 16; ++j) {
        const uint32_t g = 32 * j + lane;
        uint4 v;
        asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                     : "r"(buf_s + stage_slot(g)));
        __stcs(out + g, v);
      }
      __syncwarp();
    } else {
      // ragged last chunk: element by element
      const int64_t e0 = c0 + 32 * lane;
      for (int i = 0; i < 32; ++i) {
        const int64_t e = e0 + i;
        if (e >= n) break;
        const uint8_t byte = w.packed[e >> 1];
        const int q = (e & 1) ? (byte & 15) : (byte >> 4);
        const float v = __fmul_rn(tabs.nf4[q], a);
        if constexpr (sizeof(Tout) == 2) store16(y, e, v);
        else y[e] = v;
      }
    }
  }
}

template <typename Tout, bool kDQ>
__global__ void __launch_bounds__(kDeqThreads)
nf4_decode(Nf4View w, Tout* __restrict__ y, DecodeTables tabs) {
  decode_cta<Tout, kDQ>(w, y, tabs, blockIdx.x);
}

// Up to 8 tensors of one double-quant setting in one launch: CTA b decodes chunk b - cta0 of
// the item whose CTA range holds it.
struct DecodeItem {
  Nf4View w;
  void* y;
  int64_t cta0;
};
struct DecodeBatch {
  DecodeItem it[kEncodeBatch];
  int n;
};

template <typename Tout, bool kDQ>
__global__ void __launch_bounds__(kDeqThreads)
nf4_decode_batch(DecodeBatch b, DecodeTables tabs) {
  int i = 0;
#pragma unroll 1
  while (i + 1 < b.n && static_cast<int64_t>(blockIdx.x) >= b.it[i + 1].cta0) ++i;
  // static indices into the parameters (a run-time index would copy them to local memory)
  Nf4View w{};
  void* y = nullptr;
  int64_t cta0 = 0;
#pragma unroll
  for (int k = 0; k < kEncodeBatch; ++k)
    if (k == i) w = b.it[k].w, y = b.it[k].y, cta0 = b.it[k].cta0;
  decode_cta<Tout, kDQ>(w, static_cast<Tout*>(y), tabs, static_cast<int64_t>(blockIdx.x) - cta0);
}

// The 16-bit decode of the linear's weight and that call's operand staging in one launch:
// CTAs below `decode_ctas` decode, the rest run the prep jobs.
template <typename T16, bool kDQ>
__global__ void __launch_bounds__(kDeqThreads)
nf4_decode_prep(Nf4View w, T16* __restrict__ y, DecodeTables tabs, PrepJobs jobs, unsigned decode_ctas) {
  if (blockIdx.x < decode_ctas) decode_cta<T16, kDQ>(w, y, tabs, blockIdx.x);
  else prep_cta(jobs, blockIdx.x - decode_ctas);
}

int64_t pow2_at_least(int64_t v) {
  int64_t p = 1;
  while (p < v) p <<= 1;
  return p;
}

size_t align256(size_t b) { return (b + 255) & ~static_cast<size_t>(255); }

// Ticket counters (which CTA of a group finishes last), in the library's own device memory:
// zero at module load, and every kernel that counts on one puts it back to zero.  Calls draw
// ranges round-robin, so calls in flight at the same time (other streams, other host threads)
// use different counters unless more than kTicketSlots counters' worth of them overlap.
constexpr unsigned kTicketSlots = 16384;
__device__ unsigned g_tickets[kTicketSlots];

}  // namespace

cudaError_t ticket_range(unsigned n, unsigned** out) {
  constexpr int kMaxDev = 64;
  static unsigned* base[kMaxDev] = {};
  static std::mutex mu;
  static unsigned next = 0;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDev || n == 0 || n > kTicketSlots / 4) return cudaErrorInvalidValue;
  std::lock_guard<std::mutex> lock(mu);
  if (base[dev] == nullptr) {
    void* p = nullptr;
    if ((e = cudaGetSymbolAddress(&p, g_tickets)) != cudaSuccess) return e;
    base[dev] = static_cast<unsigned*>(p);
  }
  if (next + n > kTicketSlots) next = 0;   // a range never wraps
  *out = base[dev] + next;
  next += n;
  return cudaSuccess;
}

namespace {

cudaError_t ticket_slot(unsigned** out) { return ticket_range(1, out); }

// Resident CTAs per SM of an encode kernel (kind: input type and load width; 4 the nested
// pass), per device, looked up once (a racing first lookup stores the same value).
template <typename K>
cudaError_t encode_ctas_per_sm(K kernel, int kind, int* out) {
  constexpr int kMaxDev = 64;
  static std::atomic<int> cache[kMaxDev][5];
  int dev = 0;
  cudaGetDevice(&dev);
  const bool slot = dev >= 0 && dev < kMaxDev;
  if (slot) {
    const int c = cache[dev][kind].load(std::memory_order_relaxed);
    if (c > 0) return (*out = c), cudaSuccess;
  }
  int n = 0;
  const cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, kQuantThreads, 0);
  if (e != cudaSuccess) return e;
  n = n > 0 ? n : 1;
  if (slot) cache[dev][kind].store(n, std::memory_order_relaxed);
  *out = n;
  return cudaSuccess;
}

}  // namespace

size_t quantize_ws_bytes(int64_t numel, int dq) {
  if (!dq) return 0;
  const int64_t nb = (numel + kBlock - 1) / kBlock;
  const int64_t ng = (nb + kNested - 1) / kNested;
  return align256(sizeof(float) * nb) + align256(sizeof(double) * pow2_at_least(ng));
}

cudaError_t launch_quantize_batch(const QuantJob* jobs, int n, nf4_dtype xd, int* status, cudaStream_t st) {
  if (n < 1 || n > kEncodeBatch) return cudaErrorInvalidValue;
  const EncodeTables& et = encode_tables();
  bool v8 = true;
  for (int i = 0; i < n; ++i) v8 = v8 && (reinterpret_cast<uintptr_t>(jobs[i].x) & 31) == 0;
  int resident = 0;
  cudaError_t e;
  if (xd == NF4_F32)
    e = v8 ? encode_ctas_per_sm(nf4_encode_blocks<float, true>, 0, &resident)
           : encode_ctas_per_sm(nf4_encode_blocks<float, false>, 1, &resident);
  else
    e = v8 ? encode_ctas_per_sm(nf4_encode_blocks<__nv_bfloat16, true>, 2, &resident)
           : encode_ctas_per_sm(nf4_encode_blocks<__nv_bfloat16, false>, 3, &resident);
  if (e != cudaSuccess) return e;
  // the tensors' groups go largest tensor first: the last groups handed out belong to the
  // smallest tensor, whose offset tree (the tail after the last group) is the shortest
  QuantJob sorted[kEncodeBatch];
  for (int i = 0; i < n; ++i) sorted[i] = jobs[i];
  std::stable_sort(sorted, sorted + n, [](const QuantJob& a, const QuantJob& b) { return a.numel > b.numel; });
  jobs = sorted;
  EncodeBatch eb{};
  NestedBatch nbt{};
  eb.n = n;
  int64_t total = 0;
  for (int i = 0; i < n; ++i) {
    const int64_t nb = (jobs[i].numel + kBlock - 1) / kBlock;
    const int64_t ng = (nb + kNested - 1) / kNested;
    eb.it[i].x = jobs[i].x;
    eb.it[i].numel = jobs[i].numel;
    eb.it[i].ng = ng;
    eb.it[i].g0 = total;
    eb.it[i].p2 = pow2_at_least(ng);
    eb.it[i].packed = jobs[i].out->packed;
    total += ng;
  }
  eb.total = total;
  if (total + device_sm_count() * static_cast<int64_t>(resident) > 0x7FFFFFFFLL) return cudaErrorInvalidValue;
  const int64_t grid = std::min<int64_t>(total, static_cast<int64_t>(resident) * device_sm_count());
  for (int i = 0; i < n; ++i) {
    const nf4_tensor& out = *jobs[i].out;
    EncodeItem& it = eb.it[i];
    if (!out.double_quant) {
      it.absmax = static_cast<float*>(out.absmax);
      continue;
    }
    const int64_t nb = (jobs[i].numel + kBlock - 1) / kBlock;
    it.absmax = static_cast<float*>(jobs[i].ws);
    it.group_sum = reinterpret_cast<double*>(static_cast<char*>(jobs[i].ws) + align256(sizeof(float) * nb));
    it.offset = out.offset;
    if ((e = ticket_slot(&it.ticket)) != cudaSuccess) return e;
    NestedItem& ni = nbt.it[nbt.n++];
    ni.absmax = it.absmax;
    ni.nb = nb;
    ni.ng = it.ng;
    ni.g0 = nbt.total;
    ni.offset = out.offset;
    ni.codes = static_cast<uint8_t*>(out.absmax);
    ni.nested = out.nested_absmax;
    nbt.total += it.ng;
  }
  if (nbt.n > 0 && (e = ticket_slot(&eb.work)) != cudaSuccess) return e;
  const dim3 egrid(static_cast<unsigned>(grid)), block(kQuantThreads);
  if (xd == NF4_F32)
    e = v8 ? launch_pdl(nf4_encode_blocks<float, true>, egrid, block, 0, st, 1, eb, et, status)
           : launch_pdl(nf4_encode_blocks<float, false>, egrid, block, 0, st, 1, eb, et, status);
  else
    e = v8 ? launch_pdl(nf4_encode_blocks<__nv_bfloat16, true>, egrid, block, 0, st, 1, eb, et, status)
           : launch_pdl(nf4_encode_blocks<__nv_bfloat16, false>, egrid, block, 0, st, 1, eb, et, status);
  note_launch();
  if (e != cudaSuccess || nbt.n == 0) return e;
  int nres = 1;
  if ((e = encode_ctas_per_sm(nf4_encode_nested, 4, &nres)) != cudaSuccess) return e;
  const int64_t ngrid = std::min<int64_t>((nbt.total + kNestedWarps - 1) / kNestedWarps,
                                          static_cast<int64_t>(nres) * device_sm_count());
  e = launch_pdl(nf4_encode_nested, dim3(static_cast<unsigned>(ngrid)), dim3(kNestedWarps * 32), 0, st, 1, nbt, et);
  note_launch();
  return e;
}

cudaError_t launch_quantize(const void* x, nf4_dtype xd, int64_t numel, const nf4_tensor& out,
                            void* ws, int* status, cudaStream_t st) {
  const QuantJob job{x, numel, &out, ws};
  return launch_quantize_batch(&job, 1, xd, status, st);
}

cudaError_t launch_dequantize(const Nf4View& w, void* y, nf4_dtype od, cudaStream_t st) {
  const int64_t ctas = (w.numel + kDeqPerCta - 1) / kDeqPerCta;
  if (ctas > 0x7FFFFFFFLL) return cudaErrorInvalidValue;
  const dim3 grid(static_cast<unsigned>(ctas));
  const DecodeTables& dt = decode_tables();
  cudaError_t e;
  if (od == NF4_F32) {
    if (w.dq) e = launch_pdl(nf4_decode<float, true>, grid, dim3(kDeqThreads), 0, st, 1, w, static_cast<float*>(y), dt);
    else e = launch_pdl(nf4_decode<float, false>, grid, dim3(kDeqThreads), 0, st, 1, w, static_cast<float*>(y), dt);
  } else if (od == NF4_BF16) {
    auto* yb = static_cast<__nv_bfloat16*>(y);
    if (w.dq) e = launch_pdl(nf4_decode<__nv_bfloat16, true>, grid, dim3(kDeqThreads), 0, st, 1, w, yb, dt);
    else e = launch_pdl(nf4_decode<__nv_bfloat16, false>, grid, dim3(kDeqThreads), 0, st, 1, w, yb, dt);
  } else {
    auto* yh = static_cast<__half*>(y);
    if (w.dq) e = launch_pdl(nf4_decode<__half, true>, grid, dim3(kDeqThreads), 0, st, 1, w, yh, dt);
    else e = launch_pdl(nf4_decode<__half, false>, grid, dim3(kDeqThreads), 0, st, 1, w, yh, dt);
  }
  note_launch();
  return e;
}

// The items with double quantization in one launch, those without in another.
cudaError_t launch_dequantize_batch(const Nf4View* ws, void* const* ys, int n, nf4_dtype od, cudaStream_t st) {
  if (n < 1 || n > kEncodeBatch) return cudaErrorInvalidValue;
  const DecodeTables& dt = decode_tables();
  for (int dq = 1; dq >= 0; --dq) {
    DecodeBatch b{};
    int64_t ctas = 0;
    for (int i = 0; i < n; ++i) {
      if ((ws[i].dq != 0) != (dq != 0)) continue;
      DecodeItem& it = b.it[b.n++];
      it.w = ws[i];
      it.y = ys[i];
      it.cta0 = ctas;
      ctas += (ws[i].numel + kDeqPerCta - 1) / kDeqPerCta;
    }
    if (ctas == 0) continue;
    if (ctas > 0x7FFFFFFFLL) return cudaErrorInvalidValue;
    const dim3 grid(static_cast<unsigned>(ctas));
    cudaError_t e;
    if (od == NF4_F32)
      e = dq ? launch_pdl(nf4_decode_batch<float, true>, grid, dim3(kDeqThreads), 0, st, 1, b, dt)
             : launch_pdl(nf4_decode_batch<float, false>, grid, dim3(kDeqThreads), 0, st, 1, b, dt);
    else if (od == NF4_BF16)
      e = dq ? launch_pdl(nf4_decode_batch<__nv_bfloat16, true>, grid, dim3(kDeqThreads), 0, st, 1, b, dt)
             : launch_pdl(nf4_decode_batch<__nv_bfloat16, false>, grid, dim3(kDeqThreads), 0, st, 1, b, dt);
    else
      e = dq ? launch_pdl(nf4_decode_batch<__half, true>, grid, dim3(kDeqThreads), 0, st, 1, b, dt)
             : launch_pdl(nf4_decode_batch<__half, false>, grid, dim3(kDeqThreads), 0, st, 1, b, dt);
    note_launch();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t launch_decode_with_prep(const Nf4View& w, void* y, bool f16, const PrepJobs& jobs, unsigned prep_ctas,
                                    cudaStream_t st) {
  const int64_t ctas = (w.numel + kDeqPerCta - 1) / kDeqPerCta;
  if (ctas + prep_ctas > 0x7FFFFFFFLL) return cudaErrorInvalidValue;
  const dim3 grid(static_cast<unsigned>(ctas + prep_ctas));
  const DecodeTables& dt = decode_tables();
  const unsigned dc = static_cast<unsigned>(ctas);
  cudaError_t e;
  if (f16) {
    auto* yh = static_cast<__half*>(y);
    e = w.dq ? launch_pdl(nf4_decode_prep<__half, true>, grid, dim3(kDeqThreads), 0, st, 1, w, yh, dt, jobs, dc)
             : launch_pdl(nf4_decode_prep<__half, false>, grid, dim3(kDeqThreads), 0, st, 1, w, yh, dt, jobs, dc);
  } else {
    auto* yb = static_cast<__nv_bfloat16*>(y);
    e = w.dq ? launch_pdl(nf4_decode_prep<__nv_bfloat16, true>, grid, dim3(kDeqThreads), 0, st, 1, w, yb, dt, jobs, dc)
             : launch_pdl(nf4_decode_prep<__nv_bfloat16, false>, grid, dim3(kDeqThreads), 0, st, 1, w, yb, dt, jobs, dc);
  }
  note_launch();
  return e;
}

cudaError_t launch_prep_only(bool f16, const PrepJobs& jobs, unsigned prep_ctas, cudaStream_t st) {
  if (prep_ctas == 0) return cudaSuccess;
  const dim3 grid(prep_ctas);
  const DecodeTables& dt = decode_tables();
  const Nf4View none{};
  cudaError_t e = f16 ? launch_pdl(nf4_decode_prep<__half, false>, grid, dim3(kDeqThreads), 0, st, 1, none,
                                   static_cast<__half*>(nullptr), dt, jobs, 0u)
                      : launch_pdl(nf4_decode_prep<__nv_bfloat16, false>, grid, dim3(kDeqThreads), 0, st, 1, none,
                                   static_cast<__nv_bfloat16*>(nullptr), dt, jobs, 0u);
  note_launch();
  return e;
}

}  // namespace qnf4
