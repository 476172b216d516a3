// NF4 blockwise quantization with nested dynamic8 absmax, and dequantization.
//
// Format and decode: "Native model adaptation and NF4", section "Packed NF4 and the
// portable QLoRA profile" (64-element absmax blocks, the 16-value NF4 codebook, two
// codes per byte, block maxima centred by their global FP32 mean and quantized with
// dynamic8 in blocks of 256) and section "Fused GPU NF4 decodes inside the matrix
// kernel".  Deterministic, byte-identical requantization: "NF4 Layer Streaming --
// Gate results", section "P3 is solved".
//
// Lane mapping (all kernels here): a warp walks "quad rows" of 128 elements; lane l
// owns elements 4l..4l+3 of the row, so a half warp covers one 64-element block and
// every global access of a warp instruction is contiguous.
//
// quantize = three launches:
//   1. nf4_encode_blocks: absmax, 4-bit codes, packing; per 256-block group the
//      float64 pairwise-tree sum of the absmax values (double quant only).
//   2. nf4_absmax_mean: one CTA finishes the tree over the group sums -> offset.
//   3. nf4_encode_nested: centre, nested absmax per group, dynamic8 codes.
#include "common.cuh"
#include "decode.cuh"
#include "prep.cuh"

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

// Lane's 32 elements (from e0) as fp32, zero past numel, and the largest |x| among them
// as fp32 bits (bf16 input: an integer max over the 15-bit magnitudes, two at a time, which
// orders subnormals, Inf and NaN exactly as the fp32 bit patterns do).
__device__ __forceinline__ uint32_t max_u16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.u16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

template <typename Tin>
__device__ __forceinline__ uint32_t lane_load(const Tin* __restrict__ x, int64_t numel, int64_t e0, float (&v)[32]) {
  constexpr int kVec = 16 / sizeof(Tin);
  uint32_t w[32 / kVec * 4];
  if (e0 + 32 <= numel) {
#pragma unroll
    for (int i = 0; i < 32 / kVec; ++i) {
      const uint4 u = *reinterpret_cast<const uint4*>(x + e0 + i * kVec);
      w[4 * i] = u.x, w[4 * i + 1] = u.y, w[4 * i + 2] = u.z, w[4 * i + 3] = u.w;
    }
  } else {   // ragged tail: zero past numel
    const uint16_t* x16 = reinterpret_cast<const uint16_t*>(x);
    const uint32_t* x32 = reinterpret_cast<const uint32_t*>(x);
#pragma unroll
    for (int i = 0; i < 32 / kVec * 4; ++i) {
      if (sizeof(Tin) == 4) {
        w[i] = (e0 + i < numel) ? x32[e0 + i] : 0u;
      } else {
        const uint32_t lo = (e0 + 2 * i < numel) ? x16[e0 + 2 * i] : 0u;
        const uint32_t hi = (e0 + 2 * i + 1 < numel) ? x16[e0 + 2 * i + 1] : 0u;
        w[i] = lo | (hi << 16);
      }
    }
  }
  if (sizeof(Tin) == 4) {
    uint32_t mb = 0;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      v[i] = __uint_as_float(w[i]);
      mb = max(mb, w[i] & 0x7FFFFFFFu);
    }
    return mb;
  } else {
    uint32_t m2 = 0;   // two 16-bit maxima
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      v[2 * k] = __uint_as_float(w[k] << 16);
      v[2 * k + 1] = __uint_as_float(w[k] & 0xFFFF0000u);
      m2 = max_u16x2(m2, w[k] & 0x7FFF7FFFu);
    }
    return max(m2 & 0xFFFFu, m2 >> 16) << 16;
  }
}

// Block pass: absmax, 4-bit codes and packing for one nested group (256 blocks) per CTA;
// with double quantization also the float64 pairwise-tree sum of the group's absmax.
// Codes: q = x * RN(1/a), and fl(x * RN(1/a) + 3) picks an entry of the bucket table;
// when q lies in the entry's band around a threshold, or a or 1/a is not finite, the code
// is taken from the exact quotient RN(x / a) instead, so the result is always that of
// the IEEE division.
template <typename Tin>
__global__ void __launch_bounds__(kQuantThreads)
nf4_encode_blocks(const Tin* __restrict__ x, int64_t numel, uint8_t* __restrict__ packed,
                  float* __restrict__ absmax, double* __restrict__ group_sum, EncodeTables tabs,
                  int* status) {
  __shared__ float thr[16];
  // (lo with the base code in its low 4 bits, hi); 16 copies: the 8-byte lookups of a warp are
  // served half a warp at a time, so lanes l and l + 16 never meet in one bank access
  __shared__ float2 band[66][16];
  __shared__ double gsum[kNested];
  if (threadIdx.x < 16) thr[threadIdx.x] = tabs.nf4_thr[threadIdx.x];
  for (int i = threadIdx.x; i < 66 * 16; i += kQuantThreads)
    band[i >> 4][i & 15] = make_float2(tabs.nf4_band[i >> 4][0], tabs.nf4_band[i >> 4][1]);
  __syncthreads();
  pdl_allow_next();
  pdl_wait();
  const bool fast_ok = tabs.bucket_ok != 0;   // bucket table usable
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int64_t group_base = static_cast<int64_t>(blockIdx.x) * kGroupElems;
  // warp w handles elements [w*2048, (w+1)*2048) of the group: two 1024-element rows
  const int64_t wbase = group_base + warp * 2048;
  bool nonfinite = false;
#pragma unroll 1
  for (int u = 0; u < 2; ++u) {
    const int64_t e0 = wbase + u * 1024 + 32 * lane;    // lane's first element
    float v[32];
    uint32_t mb = lane_load<Tin>(x, numel, e0, v);
    mb = max(mb, __shfl_xor_sync(0xffffffffu, mb, 1));  // the lane pair holds one block
    nonfinite |= mb >= 0x7F800000u;
    const float a = __uint_as_float(mb);
    const float r = __frcp_rn(a);
    uint32_t words[4];
    if (a == 0.0f) {
#pragma unroll
      for (int w = 0; w < 4; ++w) words[w] = 0x77777777u;     // every code is that of 0.0
    } else {
      bool exact = !(fast_ok && isfinite(r) && mb < 0x7F800000u);
      if (!exact) {
        bool unsure = false;
#pragma unroll
        for (int w = 0; w < 4; ++w) words[w] = 0u;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const float q = v[i] * r;
          const uint32_t k = (__float_as_uint(fmaf(v[i], r, 3.0f)) >> 17) - 8191u;   // 0 .. 65
          const float2 b = band[k][lane & 15];
          unsure |= (q >= b.x) & (q < b.y);
          const uint32_t c = (__float_as_uint(b.x) & 15u) + (q >= b.y ? 1u : 0u);
          words[i >> 3] |= c << (((i >> 1) & 3) * 8 + ((i & 1) ? 0 : 4));
        }
        exact = unsure;
      }
      if (exact) {  // rare: redo the lane with the IEEE quotient
#pragma unroll
        for (int w = 0; w < 4; ++w) words[w] = 0u;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const uint32_t c = static_cast<uint32_t>(nf4_encode(__fdiv_rn(v[i], a), thr));
          words[i >> 3] |= c << (((i >> 1) & 3) * 8 + ((i & 1) ? 0 : 4));
        }
      }
    }
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
    const int block_in_group = warp * 32 + u * 16 + (lane >> 1);
    if ((lane & 1) == 0) {
      if (e0 < numel) absmax[e0 >> 6] = a;
      gsum[block_in_group] = (e0 < numel) ? static_cast<double>(a) : 0.0;
    }
  }
  if (nonfinite) atomicCAS(status, 0, static_cast<int>(NF4_ERR_NONFINITE));
  if (group_sum == nullptr) return;
  __syncthreads();
  if (warp != 0) return;
  // float64 pairwise tree s[i] += s[i + h], h = 128, 64, ..., 1, by one warp: lane l holds
  // s[l + 32 m]; the levels h >= 32 add within the lane, the rest across lanes
  double t[kNested / 32];
#pragma unroll
  for (int m = 0; m < kNested / 32; ++m) t[m] = gsum[lane + 32 * m];
#pragma unroll
  for (int h = kNested / 64; h >= 1; h >>= 1)
#pragma unroll
    for (int m = 0; m < h; ++m) t[m] += t[m + h];
#pragma unroll
  for (int h = 16; h >= 1; h >>= 1) t[0] += __shfl_down_sync(0xffffffffu, t[0], h);
  if (lane == 0) group_sum[blockIdx.x] = t[0];
}

// One CTA: the same pairwise tree over the group sums padded with zeros to p2
// entries, then offset = float(sum / nb).  The tree runs in shared memory when the p2
// entries fit (kMeanSmemEntries), in place in the workspace otherwise.
constexpr int kMeanSmemEntries = 16384;

__global__ void __launch_bounds__(1024)
nf4_absmax_mean(double* __restrict__ gs, int64_t ng, int64_t p2, int64_t nb, float* __restrict__ offset) {
  extern __shared__ double tree[];
  pdl_allow_next();
  pdl_wait();
  const bool in_smem = p2 >= 4 && p2 / 4 <= kMeanSmemEntries;
  double* s = in_smem ? tree : gs;
  int64_t valid = ng;
  int64_t h = p2 / 2;
  if (in_smem) {   // the first two levels straight from the workspace into p2 / 4 entries
    const int64_t q = p2 / 4;
    auto g = [&](int64_t i) { return i < ng ? gs[i] : 0.0; };
    for (int64_t i = threadIdx.x; i < q; i += blockDim.x)
      s[i] = (g(i) + g(i + 2 * q)) + (g(i + q) + g(i + 3 * q));
    __syncthreads();
    valid = q;
    h = q / 2;
  }
  for (; h >= 1; h /= 2) {
    for (int64_t i = threadIdx.x; i < h; i += blockDim.x) {
      const double a = (i < valid) ? s[i] : 0.0;
      const double b = (i + h < valid) ? s[i + h] : 0.0;
      s[i] = a + b;
    }
    valid = h;
    __syncthreads();
  }
  if (threadIdx.x == 0) *offset = __double2float_rn(__ddiv_rn(s[0], static_cast<double>(nb)));
}

// Nested quantization of the block maxima: one warp per group of 256 maxima, eight per
// lane.  c = a - offset; m = max |c| over the group; code = dyn8 code of RN(c / m).
constexpr int kNestedWarps = 8;

__global__ void __launch_bounds__(kNestedWarps * 32)
nf4_encode_nested(const float* __restrict__ absmax, int64_t nb, const float* __restrict__ offset_p,
                  uint8_t* __restrict__ codes, float* __restrict__ nested, EncodeTables tabs) {
  __shared__ float thr[256];
  thr[threadIdx.x] = tabs.dyn8_thr[threadIdx.x];
  __syncthreads();
  pdl_allow_next();
  pdl_wait();
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int64_t g = static_cast<int64_t>(blockIdx.x) * kNestedWarps + warp;
  if (g * kNested >= nb) return;
  const float offset = *offset_p;
  const int64_t b0 = g * kNested + 8 * lane;
  float c[8];
  const bool full = b0 + 8 <= nb && (reinterpret_cast<uintptr_t>(absmax + b0) & 15) == 0;
  if (full) {
    const float4 u = *reinterpret_cast<const float4*>(absmax + b0);
    const float4 v = *reinterpret_cast<const float4*>(absmax + b0 + 4);
    const float a[8] = {u.x, u.y, u.z, u.w, v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) c[i] = __fsub_rn(a[i], offset);
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) c[i] = (b0 + i < nb) ? __fsub_rn(absmax[b0 + i], offset) : 0.0f;
  }
  float m = fabsf(c[0]);
#pragma unroll
  for (int i = 1; i < 8; ++i) m = fmaxf(m, fabsf(c[i]));
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  uint32_t q[8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
    q[i] = static_cast<uint32_t>((m > 0.0f) ? dyn8_encode(__fdiv_rn(c[i], m), thr) : kDyn8ZeroCode);
  if (b0 + 8 <= nb && (reinterpret_cast<uintptr_t>(codes + b0) & 7) == 0) {
    *reinterpret_cast<uint2*>(codes + b0) =
        make_uint2(q[0] | (q[1] << 8) | (q[2] << 16) | (q[3] << 24), q[4] | (q[5] << 8) | (q[6] << 16) | (q[7] << 24));
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i)
      if (b0 + i < nb) codes[b0 + i] = static_cast<uint8_t>(q[i]);
  }
  if (lane == 0) nested[g] = m;
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

}  // namespace

size_t quantize_ws_bytes(int64_t numel, int dq) {
  if (!dq) return 0;
  const int64_t nb = (numel + kBlock - 1) / kBlock;
  const int64_t ng = (nb + kNested - 1) / kNested;
  return align256(sizeof(float) * nb) + align256(sizeof(double) * pow2_at_least(ng));
}

cudaError_t launch_quantize(const void* x, nf4_dtype xd, int64_t numel, const nf4_tensor& out,
                            void* ws, int* status, cudaStream_t st) {
  const int64_t nb = (numel + kBlock - 1) / kBlock;
  const int64_t ng = (nb + kNested - 1) / kNested;
  const EncodeTables& et = encode_tables();
  float* absmax_f = out.double_quant ? static_cast<float*>(ws) : static_cast<float*>(out.absmax);
  double* gsum = out.double_quant
                     ? reinterpret_cast<double*>(static_cast<char*>(ws) + align256(sizeof(float) * nb))
                     : nullptr;
  if (ng > 0x7FFFFFFFLL) return cudaErrorInvalidValue;
  const dim3 grid(static_cast<unsigned>(ng));
  cudaError_t e;
  if (xd == NF4_F32)
    e = launch_pdl(nf4_encode_blocks<float>, grid, dim3(kQuantThreads), 0, st, 1, static_cast<const float*>(x), numel,
                   out.packed, absmax_f, gsum, et, status);
  else
    e = launch_pdl(nf4_encode_blocks<__nv_bfloat16>, grid, dim3(kQuantThreads), 0, st, 1,
                   static_cast<const __nv_bfloat16*>(x), numel, out.packed, absmax_f, gsum, et, status);
  note_launch();
  if (e != cudaSuccess || !out.double_quant) return e;
  const int64_t p2 = pow2_at_least(ng);
  const size_t mean_smem = (p2 >= 4 && p2 / 4 <= kMeanSmemEntries) ? sizeof(double) * static_cast<size_t>(p2 / 4) : 0;
  static std::once_flag once;
  static cudaError_t attr = cudaSuccess;
  std::call_once(once, [] {
    attr = cudaFuncSetAttribute(nf4_absmax_mean, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                static_cast<int>(sizeof(double) * kMeanSmemEntries));
  });
  if (attr != cudaSuccess) return attr;
  e = launch_pdl(nf4_absmax_mean, dim3(1), dim3(1024), mean_smem, st, 1, gsum, ng, p2, nb, out.offset);
  note_launch();
  if (e != cudaSuccess) return e;
  const dim3 ngrid(static_cast<unsigned>((ng + kNestedWarps - 1) / kNestedWarps));
  e = launch_pdl(nf4_encode_nested, ngrid, dim3(kNestedWarps * 32), 0, st, 1, static_cast<const float*>(absmax_f), nb,
                 static_cast<const float*>(out.offset), static_cast<uint8_t*>(out.absmax), out.nested_absmax, et);
  note_launch();
  return e;
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

}  // namespace qnf4
