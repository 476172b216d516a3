// Off the training step, two more consumers of the NF4 format:
//   * selected rows of an NF4 embedding table, decoded on the device ([ADAPT] "Packed NF4
//     and the portable QLoRA profile": embeddings decode only selected rows; "Fused GPU
//     NF4 decodes inside the matrix kernel": selected-row embedding kernels);
//   * the merged deployment weight W' = deq(W) + s B A ([ADAPT] "Checkpoints, exact
//     continuation and deployment": merged F32 deployment weights with the decoded base).
// Both decode with the arithmetic of nf4_dequantize: a' = dyn8[code] * nested + offset
// (two roundings) or the fp32 absmax, w = nf4[q] * a'.
#include <atomic>

#include "common.cuh"
#include "decode.cuh"

namespace qnf4 {
namespace {

constexpr int kThreads = 256;

constexpr int kMaxDevices = 64;

// Per-device launch facts, looked up once (a racing first lookup stores the same value).
int device_sms() {
  static std::atomic<int> cache[kMaxDevices];
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < kMaxDevices) {
    const int c = cache[dev].load(std::memory_order_relaxed);
    if (c > 0) return c;
  }
  int n = 0;
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  n = n > 0 ? n : 1;
  if (dev >= 0 && dev < kMaxDevices) cache[dev].store(n, std::memory_order_relaxed);
  return n;
}

// Resident CTAs per SM of `kernel` at kThreads threads (kind 0/1 selects the cache slot).
template <typename K>
cudaError_t resident_per_sm(K kernel, int kind, int* out) {
  static std::atomic<int> cache[kMaxDevices][2];
  int dev = 0;
  cudaGetDevice(&dev);
  const bool slot = dev >= 0 && dev < kMaxDevices;
  if (slot) {
    const int c = cache[dev][kind].load(std::memory_order_relaxed);
    if (c > 0) {
      *out = c;
      return cudaSuccess;
    }
  }
  int n = 0;
  const cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, kThreads, 0);
  if (e != cudaSuccess) return e;
  n = n > 0 ? n : 1;
  if (slot) cache[dev][kind].store(n, std::memory_order_relaxed);
  *out = n;
  return cudaSuccess;
}

struct Decoder {
  const Nf4View& w;
  const float* dyn8;   // shared copy
  const float* nf4v;   // shared copy
  float offset;
  __device__ __forceinline__ float scale(int64_t blk) const {
    if (!w.dq) return static_cast<const float*>(w.absmax)[blk];
    const uint8_t c = static_cast<const uint8_t*>(w.absmax)[blk];
    return __fadd_rn(__fmul_rn(dyn8[c], w.nested[blk >> 8]), offset);
  }
  __device__ __forceinline__ float element(int64_t e) const {
    const uint8_t byte = w.packed[e >> 1];
    const int q = (e & 1) ? (byte & 15) : (byte >> 4);
    return __fmul_rn(nf4v[q], scale(e >> 6));
  }
};

__device__ __forceinline__ void store1(float* p, float v) { *p = v; }
__device__ __forceinline__ void store1(__nv_bfloat16* p, float v) { *p = __float2bfloat16_rn(v); }

// ---- selected embedding rows --------------------------------------------------------
// Rows whose width is not a multiple of 32.
// CTA (chunk, rows i0 .. i0 + 8): thread t covers dims chunk*2048 + 8t .. +8 of each of the
// 8 rows.  When dim % 8 == 0 every thread's 8 elements lie in one 64-block and its output
// is 16-byte aligned: all 8 rows' ids, then all their code words and scales, are loaded
// before any decode, so a CTA waits for two memory latencies, not sixteen.  Otherwise
// each element is decoded on its own.

constexpr int kEmbedChunk = kThreads * 8;
constexpr int kEmbedRows = 8;

template <typename Tout>
__device__ __forceinline__ void store8(Tout* o, const float (&v)[8]) {
  if constexpr (sizeof(Tout) == 4) {
    reinterpret_cast<float4*>(o)[0] = make_float4(v[0], v[1], v[2], v[3]);
    reinterpret_cast<float4*>(o)[1] = make_float4(v[4], v[5], v[6], v[7]);
  } else {
    uint32_t u[4];
#pragma unroll
    for (int h = 0; h < 4; ++h)
      u[h] = static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(v[2 * h]))) |
             (static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(v[2 * h + 1]))) << 16);
    *reinterpret_cast<uint4*>(o) = make_uint4(u[0], u[1], u[2], u[3]);
  }
}

template <typename Tout>
__global__ void __launch_bounds__(kThreads)
nf4_embed_rows(Nf4View w, int64_t rows, int64_t dim, const int64_t* __restrict__ ids, int64_t n_ids,
               Tout* __restrict__ out, DecodeTables tabs, int* status) {
  __shared__ float dyn8[256];
  __shared__ float nf4v[16];
  dyn8[threadIdx.x] = tabs.dyn8[threadIdx.x];
  if (threadIdx.x < 16) nf4v[threadIdx.x] = tabs.nf4[threadIdx.x];
  __syncthreads();
  pdl_allow_next();
  pdl_wait();
  const Decoder dec{w, dyn8, nf4v, w.dq ? *w.offset : 0.0f};
  const int64_t d0 = static_cast<int64_t>(blockIdx.x) * kEmbedChunk + 8 * threadIdx.x;
  if (d0 >= dim) return;
  const int cnt = static_cast<int>(dim - d0 < 8 ? dim - d0 : 8);
  const bool vec = (dim & 7) == 0;   // grid-uniform
  for (int64_t i0 = static_cast<int64_t>(blockIdx.y) * kEmbedRows; i0 < n_ids;
       i0 += static_cast<int64_t>(gridDim.y) * kEmbedRows) {
    int64_t id[kEmbedRows];
#pragma unroll
    for (int u = 0; u < kEmbedRows; ++u) id[u] = i0 + u < n_ids ? ids[i0 + u] : 0;
    bool ok[kEmbedRows];
#pragma unroll
    for (int u = 0; u < kEmbedRows; ++u) {
      ok[u] = id[u] >= 0 && id[u] < rows;
      if (i0 + u < n_ids && !ok[u] && threadIdx.x == 0 && blockIdx.x == 0)
        atomicCAS(status, 0, static_cast<int>(NF4_ERR_ARG));
    }
    if (vec) {
      uint32_t word[kEmbedRows];
      float sc[kEmbedRows];
#pragma unroll
      for (int u = 0; u < kEmbedRows; ++u) {
        const int64_t e0 = ok[u] ? id[u] * dim + d0 : 0;
        word[u] = *reinterpret_cast<const uint32_t*>(w.packed + (e0 >> 1));
        sc[u] = dec.scale(e0 >> 6);
      }
#pragma unroll
      for (int u = 0; u < kEmbedRows; ++u) {
        if (i0 + u >= n_ids) break;
        float v[8];
#pragma unroll
        for (int b = 0; b < 4; ++b) {
          v[2 * b] = ok[u] ? __fmul_rn(nf4v[(word[u] >> (8 * b + 4)) & 15], sc[u]) : 0.0f;
          v[2 * b + 1] = ok[u] ? __fmul_rn(nf4v[(word[u] >> (8 * b)) & 15], sc[u]) : 0.0f;
        }
        store8(out + (i0 + u) * dim + d0, v);
      }
    } else {
#pragma unroll
      for (int u = 0; u < kEmbedRows; ++u) {
        if (i0 + u >= n_ids) break;
        Tout* o = out + (i0 + u) * dim + d0;
        for (int c = 0; c < cnt; ++c) store1(o + c, ok[u] ? dec.element(id[u] * dim + d0 + c) : 0.0f);
      }
    }
  }
}

// Rows whose width is a multiple of 32: warp w takes rows w, w + W, ... (W warps in the
// grid); lane l decodes pieces l, l + 32, ... of 32 elements, each inside one 64-block:
// one 16-byte load of codes and one scale per piece, then (bf16) the block's register
// lookup table of bf16(nf4[q] * a') and byte permutes, or (fp32) a lane-replicated table
// of the code values and one multiply per element.  A lane's 64 or 128 output bytes go
// through a swizzled warp buffer in shared memory, so each global store instruction
// writes 512 contiguous bytes.  The next row's id is loaded while this row is decoded.

constexpr int kEmbedPieces = 4;   // pieces per lane whose loads are issued together

template <typename Tout>
__global__ void __launch_bounds__(kThreads)
nf4_embed_rows32(Nf4View w, int64_t rows, int64_t dim, const int64_t* __restrict__ ids, int64_t n_ids,
                 Tout* __restrict__ out, DecodeTables tabs, int* status) {
  constexpr int kSlots = 2 * static_cast<int>(sizeof(Tout));   // 16-byte slots per lane and piece
  __shared__ float dyn8[256];
  __shared__ float lut[16][32];
  __shared__ __align__(16) uint8_t stage[kThreads / 32][32 * 16 * kSlots];
  dyn8[threadIdx.x] = tabs.dyn8[threadIdx.x];
  for (int i = threadIdx.x; i < 16 * 32; i += kThreads) lut[i >> 5][i & 31] = tabs.nf4[i >> 5];
  __syncthreads();
  pdl_allow_next();
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const uint32_t buf = static_cast<uint32_t>(__cvta_generic_to_shared(stage[threadIdx.x >> 5]));
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (kThreads / 32);
  const int64_t per_row = dim >> 5;
  const float offset = w.dq ? *w.offset : 0.0f;
  int64_t i = static_cast<int64_t>(blockIdx.x) * (kThreads / 32) + (threadIdx.x >> 5);
  int64_t id = i < n_ids ? ids[i] : 0;
  for (; i < n_ids; i += warps) {
    const int64_t id_next = i + warps < n_ids ? ids[i + warps] : 0;
    const bool ok = id >= 0 && id < rows;
    if (!ok && lane == 0) atomicCAS(status, 0, static_cast<int>(NF4_ERR_ARG));
    Tout* orow = out + i * dim;
    for (int64_t p0 = 0; p0 < per_row; p0 += 32 * kEmbedPieces) {
      uint4 pk[kEmbedPieces];
      float sc[kEmbedPieces];
#pragma unroll
      for (int u = 0; u < kEmbedPieces; ++u) {
        const int64_t p = p0 + 32 * u + lane;
        pk[u] = make_uint4(0x77777777u, 0x77777777u, 0x77777777u, 0x77777777u);   // code 7 is 0.0
        sc[u] = 0.0f;
        if (ok && p < per_row) {
          const int64_t e0 = id * dim + 32 * p;
          pk[u] = *reinterpret_cast<const uint4*>(w.packed + (e0 >> 1));
          const int64_t blk = e0 >> 6;
          sc[u] = w.dq ? __fadd_rn(__fmul_rn(dyn8[static_cast<const uint8_t*>(w.absmax)[blk]], w.nested[blk >> 8]),
                                   offset)
                       : static_cast<const float*>(w.absmax)[blk];
        }
      }
#pragma unroll
      for (int u = 0; u < kEmbedPieces; ++u) {
        const int64_t q0 = p0 + 32 * u;             // the warp's first piece this round
        if (q0 >= per_row) break;
        const int live = per_row - q0 < 32 ? static_cast<int>(per_row - q0) : 32;
        const uint32_t words[4] = {pk[u].x, pk[u].y, pk[u].z, pk[u].w};
        if constexpr (sizeof(Tout) == 2) {
          uint32_t L[4], H[4];
          build_lut(sc[u], L, H);   // an invalid id: scale 0 and code 7, +0.0 everywhere
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            uint32_t v[4];
            decode8(words[k], L, H, v);
            st_shared16(buf + stage_slot(kSlots * lane + k), v[0], v[1], v[2], v[3]);
          }
        } else {
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            float v[8];
#pragma unroll
            for (int b = 0; b < 4; ++b) {
              v[2 * b] = __fmul_rn(lut[(words[k] >> (8 * b + 4)) & 15][lane], sc[u]);
              v[2 * b + 1] = __fmul_rn(lut[(words[k] >> (8 * b)) & 15][lane], sc[u]);
            }
#pragma unroll
            for (int h = 0; h < 2; ++h)
              st_shared16(buf + stage_slot(kSlots * lane + 2 * k + h), __float_as_uint(v[4 * h]),
                          __float_as_uint(v[4 * h + 1]), __float_as_uint(v[4 * h + 2]), __float_as_uint(v[4 * h + 3]));
          }
        }
        __syncwarp();
        uint4* o = reinterpret_cast<uint4*>(orow + 32 * q0);
#pragma unroll
        for (int j = 0; j < kSlots; ++j) {
          const uint32_t g = 32 * j + lane;
          if (static_cast<int>(g) < kSlots * live) o[g] = ld_shared16(buf + stage_slot(g));
        }
        __syncwarp();
      }
    }
    id = id_next;
  }
}

// ---- merged weight ------------------------------------------------------------------
// Persistent CTAs over tiles of 32 rows x 256 columns; a CTA's tiles share one column
// range when the grid is a multiple of the column-tile count, so for r <= 16 its A chunk
// is staged once and the tile loop has no CTA-wide barrier.  Thread (tx, ty): rows
// ty*4 .. +4, columns tx*4 .. +4 and 128 + tx*4 .. +4 (each shared read of a warp is 512
// contiguous bytes).  Warp ty keeps the B entries of its own 4 rows in a private slice of
// shared memory.  The next tile's stored codes, scales and first B chunk are loaded
// during this tile's products and epilogue.  The rank-r product accumulates by fused
// multiply-adds in order j = 0, 1, ...

constexpr int kMTileN = 32, kMTileK = 256, kRankChunk = 16;

struct MergeFetch {
  uint32_t meta[4][2];   // packed codes of 4 columns (low 16 bits), dynamic8 code above
  float nest[4][2];      // nested maximum (or the fp32 absmax)
  float b[2];            // B chunk 0 of the warp's 4 rows: 2 of its 4 x 16 entries
};

__device__ __forceinline__ void merge_fetch(MergeFetch& f, const Nf4View& w, int64_t N, int64_t K, int r,
                                            const float* __restrict__ B, int64_t n0, int64_t k0, int tx,
                                            int ty) {
#pragma unroll
  for (int a = 0; a < 4; ++a)
#pragma unroll
    for (int g = 0; g < 2; ++g) {
      const int64_t n = n0 + ty * 4 + a, k = k0 + g * 128 + tx * 4;
      const bool in = n < N && k < K;             // K % 4 == 0: a group is all in or all out
      const int64_t e0 = in ? n * K + k : 0;      // four elements of one 64-block
      f.meta[a][g] = *reinterpret_cast<const uint16_t*>(w.packed + (e0 >> 1));
      const int64_t blk = e0 >> 6;
      if (w.dq) {
        f.meta[a][g] |= static_cast<uint32_t>(static_cast<const uint8_t*>(w.absmax)[blk]) << 16;
        f.nest[a][g] = w.nested[blk >> 8];
      } else {
        f.nest[a][g] = static_cast<const float*>(w.absmax)[blk];
      }
    }
#pragma unroll
  for (int u = 0; u < 2; ++u) {
    const int i = tx + 32 * u;
    const int a = i >> 4, jj = i & 15;
    const int64_t n = n0 + ty * 4 + a;
    f.b[u] = (jj < r && n < N) ? B[n * r + jj] : 0.0f;
  }
}

// One rank step of the thread's 4 x 8 outer product: acc[a][c] += B[row a][j] * A[j][col c]
// (Bw_j: B[row 0..3][j] of the warp's rows).
__device__ __forceinline__ void merge_step(const float* __restrict__ As_j, const float* __restrict__ Bw_j, int tx,
                                           float (&acc)[4][8]) {
  const float4 a0 = *reinterpret_cast<const float4*>(As_j + tx * 4);
  const float4 a1 = *reinterpret_cast<const float4*>(As_j + 128 + tx * 4);
  const float4 b0 = *reinterpret_cast<const float4*>(Bw_j);
  const float av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
  const float bv[4] = {b0.x, b0.y, b0.z, b0.w};
#pragma unroll
  for (int a = 0; a < 4; ++a)
#pragma unroll
    for (int c = 0; c < 8; ++c) acc[a][c] = fmaf(bv[a], av[c], acc[a][c]);
}

template <typename Tout>
__global__ void __launch_bounds__(kThreads, 2)
nf4_merge(Nf4View w, int64_t N, int64_t K, int64_t tiles_k, int64_t tiles, int r, float s,
          const float* __restrict__ A, const float* __restrict__ B, Tout* __restrict__ out, DecodeTables tabs) {
  __shared__ float dyn8[256];
  __shared__ float nf4v[16];
  __shared__ __align__(16) float As[kRankChunk][kMTileK];
  __shared__ __align__(16) float Bw[kThreads / 32][kRankChunk][4];
  dyn8[threadIdx.x] = tabs.dyn8[threadIdx.x];
  if (threadIdx.x < 16) nf4v[threadIdx.x] = tabs.nf4[threadIdx.x];
  pdl_allow_next();
  pdl_wait();
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
  const float offset = w.dq ? *w.offset : 0.0f;
  int64_t t = blockIdx.x;
  MergeFetch cur, nxt;
  merge_fetch(cur, w, N, K, r, B, (t / tiles_k) * kMTileN, (t % tiles_k) * kMTileK, tx, ty);
  int64_t a_tile = -1;
  for (; t < tiles; t += gridDim.x) {
    const int64_t n0 = (t / tiles_k) * kMTileN, tk = t % tiles_k, k0 = tk * kMTileK;
    const int64_t tn = t + gridDim.x;
    float acc[4][8];
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int c = 0; c < 8; ++c) acc[a][c] = 0.0f;
    for (int j0 = 0; j0 < r; j0 += kRankChunk) {
      const bool restage = tk != a_tile || r > kRankChunk;   // the same for the whole CTA
      if (restage) {
        __syncthreads();   // the previous chunk is consumed (and the tables are in place)
#pragma unroll
        for (int u = 0; u < kRankChunk * kMTileK / 4 / kThreads; ++u) {
          const int i = threadIdx.x + u * kThreads;
          const int jj = i / (kMTileK / 4), c4 = i % (kMTileK / 4);
          const int64_t k = k0 + 4 * c4;
          float4 v = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
          if (j0 + jj < r && k < K) v = *reinterpret_cast<const float4*>(A + static_cast<int64_t>(j0 + jj) * K + k);
          *reinterpret_cast<float4*>(&As[jj][4 * c4]) = v;
        }
      }
      __syncwarp();        // the warp's previous reads of its B slice are done
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int i = tx + 32 * u;
        const int a = i >> 4, jj = i & 15;
        const int64_t n = n0 + ty * 4 + a;
        Bw[ty][jj][a] = j0 == 0 ? cur.b[u] : ((j0 + jj < r && n < N) ? B[n * r + j0 + jj] : 0.0f);
      }
      if (restage) __syncthreads();
      else __syncwarp();
      if (j0 + kRankChunk >= r && tn < tiles)   // next tile's loads pass under this one's work
        merge_fetch(nxt, w, N, K, r, B, (tn / tiles_k) * kMTileN, (tn % tiles_k) * kMTileK, tx, ty);
      const int jn = r - j0 < kRankChunk ? r - j0 : kRankChunk;
      if (jn == kRankChunk) {
#pragma unroll
        for (int jj = 0; jj < kRankChunk; ++jj) merge_step(As[jj], Bw[ty][jj], tx, acc);
      } else {
        for (int jj = 0; jj < jn; ++jj) merge_step(As[jj], Bw[ty][jj], tx, acc);
      }
    }
    a_tile = tk;
#pragma unroll
    for (int a = 0; a < 4; ++a) {
      const int64_t n = n0 + ty * 4 + a;
#pragma unroll
      for (int g = 0; g < 2; ++g) {
        const int64_t k = k0 + g * 128 + tx * 4;
        if (n >= N || k >= K) continue;
        const uint32_t h = cur.meta[a][g];
        const float sc = w.dq ? __fadd_rn(__fmul_rn(dyn8[h >> 16], cur.nest[a][g]), offset) : cur.nest[a][g];
        const float wv[4] = {__fmul_rn(nf4v[(h >> 4) & 15], sc), __fmul_rn(nf4v[h & 15], sc),
                             __fmul_rn(nf4v[(h >> 12) & 15], sc), __fmul_rn(nf4v[(h >> 8) & 15], sc)};
        float m[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) m[c] = __fadd_rn(wv[c], __fmul_rn(s, acc[a][g * 4 + c]));
        Tout* o = out + n * K + k;
        if constexpr (sizeof(Tout) == 4) {
          *reinterpret_cast<float4*>(o) = make_float4(m[0], m[1], m[2], m[3]);
        } else {
          const uint32_t lo = static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(m[0]))) |
                              (static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(m[1]))) << 16);
          const uint32_t hi = static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(m[2]))) |
                              (static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(m[3]))) << 16);
          *reinterpret_cast<uint2*>(o) = make_uint2(lo, hi);
        }
      }
    }
    cur = nxt;
  }
}


}  // namespace

cudaError_t launch_embedding_rows(const Nf4View& w, int64_t rows, int64_t dim, const int64_t* ids, int64_t n_ids,
                                  void* out, nf4_dtype od, int* status, cudaStream_t st) {
  if (n_ids == 0 || dim == 0) return cudaSuccess;
  const DecodeTables& dt = decode_tables();
  cudaError_t e;
  if (dim % 32 == 0) {
    // one warp per row; no more CTAs than are resident at once
    int per_sm = 0;
    e = od == NF4_F32 ? resident_per_sm(nf4_embed_rows32<float>, 0, &per_sm)
                      : resident_per_sm(nf4_embed_rows32<__nv_bfloat16>, 1, &per_sm);
    if (e != cudaSuccess) return e;
    const int64_t ctas_max = static_cast<int64_t>(per_sm) * device_sms();
    const int64_t need = (n_ids + kThreads / 32 - 1) / (kThreads / 32);
    const dim3 grid(static_cast<unsigned>(need < ctas_max ? need : ctas_max));
    e = od == NF4_F32 ? launch_pdl(nf4_embed_rows32<float>, grid, dim3(kThreads), 0, st, 1, w, rows, dim, ids, n_ids,
                                   static_cast<float*>(out), dt, status)
                      : launch_pdl(nf4_embed_rows32<__nv_bfloat16>, grid, dim3(kThreads), 0, st, 1, w, rows, dim, ids,
                                   n_ids, static_cast<__nv_bfloat16*>(out), dt, status);
  } else {
    const int64_t chunks = (dim + kEmbedChunk - 1) / kEmbedChunk;
    const int64_t groups = (n_ids + kEmbedRows - 1) / kEmbedRows;
    if (chunks > 0x7FFFFFFFLL) return cudaErrorInvalidValue;
    const dim3 grid(static_cast<unsigned>(chunks), static_cast<unsigned>(groups < 65535 ? groups : 65535));
    e = od == NF4_F32 ? launch_pdl(nf4_embed_rows<float>, grid, dim3(kThreads), 0, st, 1, w, rows, dim, ids, n_ids,
                                   static_cast<float*>(out), dt, status)
                      : launch_pdl(nf4_embed_rows<__nv_bfloat16>, grid, dim3(kThreads), 0, st, 1, w, rows, dim, ids,
                                   n_ids, static_cast<__nv_bfloat16*>(out), dt, status);
  }
  note_launch();
  return e;
}

cudaError_t launch_merge_lora(const Nf4View& w, int64_t N, int64_t K, int r, float s, const float* A,
                              const float* B, void* out, nf4_dtype od, cudaStream_t st) {
  const int64_t tiles_k = (K + kMTileK - 1) / kMTileK, tiles_n = (N + kMTileN - 1) / kMTileN;
  if (tiles_n > (int64_t(1) << 62) / tiles_k) return cudaErrorInvalidValue;
  const int64_t tiles = tiles_n * tiles_k;
  // two resident CTAs per SM; a multiple of the column-tile count when that fits
  const int64_t slots = 2 * static_cast<int64_t>(device_sms());
  const int64_t grid = tiles <= slots ? tiles : (tiles_k <= slots ? slots / tiles_k * tiles_k : slots);
  const DecodeTables& dt = decode_tables();
  const cudaError_t e =
      od == NF4_F32 ? launch_pdl(nf4_merge<float>, dim3(static_cast<unsigned>(grid)), dim3(kThreads), 0, st, 1, w, N,
                                 K, tiles_k, tiles, r, s, A, B, static_cast<float*>(out), dt)
                    : launch_pdl(nf4_merge<__nv_bfloat16>, dim3(static_cast<unsigned>(grid)), dim3(kThreads), 0, st, 1,
                                 w, N, K, tiles_k, tiles, r, s, A, B, static_cast<__nv_bfloat16*>(out), dt);
  note_launch();
  return e;
}

}  // namespace qnf4
