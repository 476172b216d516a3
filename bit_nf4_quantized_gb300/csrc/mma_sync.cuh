// Warp-level tensor-core products from registers (mma.sync m16n8k16, fp32 accumulate) and the
// shared-memory accesses that feed them; used by the passes whose tiles are too small for the
// tcgen05 pipeline (the small-M forward and the small-shape fused linear).
#pragma once

#include "common.cuh"

namespace qnf4 {

// D += A (16 x 16, row) * B (16 x 8, col), bf16 or (F16) IEEE half operands, fp32 accumulate,
// fragments per thread.  Lane l = 4g + c holds a0 = A[g][2c, 2c+1], a1 = A[g+8][2c, 2c+1],
// a2 = A[g][2c+8, 2c+9], a3 = A[g+8][2c+8, 2c+9], b0 = B[2c, 2c+1][g], b1 = B[2c+8, 2c+9][g],
// and d = D[g][2c], D[g][2c+1], D[g+8][2c], D[g+8][2c+1].
template <bool F16>
__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                         uint32_t b1) {
  if constexpr (F16)
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
                 "{%0, %1, %2, %3};"
                 : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                 : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  else
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
                 "{%0, %1, %2, %3};"
                 : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                 : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t ld_shared32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}

__device__ __forceinline__ void st_shared32(uint32_t addr, uint32_t v) {
  asm volatile("st.shared.b32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

}  // namespace qnf4
