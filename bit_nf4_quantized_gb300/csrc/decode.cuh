// Register-table decode of packed NF4 codes to 16-bit values (bf16, or IEEE half for the
// FP16 profile), shared by the dequantize, selected-row and small-M forward kernels.  For a
// block with scale a', entry q of the table is T16(nf4[q] * a') -- the fp32 product rounded
// once -- so the decoded values are exactly what nf4_dequantize writes for that output type.
#pragma once

#include <cuda_fp16.h>

#include "common.cuh"

namespace qnf4 {

// Two floats rounded to nearest even and packed, the first in the low half.
template <typename T16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi);
template <>
__device__ __forceinline__ uint32_t pack2<__nv_bfloat16>(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}
template <>
__device__ __forceinline__ uint32_t pack2<__half>(float lo, float hi) {
  const __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// One float rounded to nearest even, stored as T16.
__device__ __forceinline__ void store16(__nv_bfloat16* p, int64_t i, float v) { p[i] = __float2bfloat16_rn(v); }
__device__ __forceinline__ void store16(__half* p, int64_t i, float v) { p[i] = __float2half_rn(v); }

// A 16-bit value (bf16 or half bits in the low half of `bits`) as a float.
template <typename T16>
__device__ __forceinline__ float from16(uint32_t bits);
template <>
__device__ __forceinline__ float from16<__nv_bfloat16>(uint32_t bits) { return __uint_as_float(bits << 16); }
template <>
__device__ __forceinline__ float from16<__half>(uint32_t bits) {
  return __half2float(__ushort_as_half(static_cast<unsigned short>(bits & 0xFFFFu)));
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

// Scaled lookup table of one block: entry i = T16(nf4[i] * a'), split into low bytes
// (L, 4 registers of 4 entries) and high bytes (H), so prmt can index it by nibble.
template <typename T16 = __nv_bfloat16>
__device__ __forceinline__ void build_lut(float a, uint32_t (&L)[4], uint32_t (&H)[4]) {
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    const uint32_t u0 = pack2<T16>(__fmul_rn(nf4_value(4 * t + 0), a), __fmul_rn(nf4_value(4 * t + 1), a));
    const uint32_t u1 = pack2<T16>(__fmul_rn(nf4_value(4 * t + 2), a), __fmul_rn(nf4_value(4 * t + 3), a));
    L[t] = prmt(u0, u1, 0x6420u);
    H[t] = prmt(u0, u1, 0x7531u);
  }
}

// Eight weights of one packed word to four registers of two 16-bit values, in element order.  The
// word's nibbles, low first, are elements 1 0 3 2 5 4 7 6 (element 2i is the high nibble
// of byte i); the final byte interleave puts them back in order.  The selectors (the low 3
// bits of each code, and bit 3 choosing the half table) are formed once for the whole word;
// prmt reads its selector from the low 16 bits, so the upper four codes take them shifted.
__device__ __forceinline__ void decode8(uint32_t w, const uint32_t (&L)[4], const uint32_t (&H)[4],
                                        uint32_t* out) {
  const uint32_t s7w = w & 0x77777777u;                            // index within a half table
  const uint32_t sbw = ((w >> 1) & 0x44444444u) | 0x32103210u;     // pick the half by bit 3
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const uint32_t s7 = h == 0 ? s7w : (s7w >> 16);
    const uint32_t sb = h == 0 ? sbw : (sbw >> 16);
    const uint32_t lo = prmt(prmt(L[0], L[1], s7), prmt(L[2], L[3], s7), sb);
    const uint32_t hi = prmt(prmt(H[0], H[1], s7), prmt(H[2], H[3], s7), sb);
    out[2 * h] = prmt(lo, hi, 0x4051u);
    out[2 * h + 1] = prmt(lo, hi, 0x6273u);
  }
}

// Output staging in shared memory: 16-byte slot g of a warp's buffer, rows of 8 slots
// XOR-swizzled by row, so that a warp writing each lane's consecutive slots and a warp
// reading slots 32j + lane both touch all 32 banks once per 8 lanes.
__device__ __forceinline__ uint32_t stage_slot(uint32_t g) {
  const uint32_t row = g >> 3, col = g & 7;
  return ((row << 3) | (col ^ (row & 7))) << 4;
}

__device__ __forceinline__ void st_shared16(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

__device__ __forceinline__ uint4 ld_shared16(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}

}  // namespace qnf4
