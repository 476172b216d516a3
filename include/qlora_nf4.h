/*
 * qlora_nf4.h -- C ABI of the NF4 double-quantized frozen-base QLoRA linear for
 * one NVIDIA GB300 (sm_103a).  Library: libqlora_nf4.so (built in-tree).
 *
 * Sources, cited by page title and section:
 *   [ADAPT] "Native model adaptation and NF4" (anerlang.org/docs/gen-adaptation)
 *   [GATE]  "NF4 Layer Streaming -- Gate results" (Soup, gate-v0.72.2-nf4.md)
 *   [QUAL]  V100 accelerated qualification record (native_training_accelerated_20261031.json)
 *
 * Conventions for every call:
 *   - Pointers named "device" are CUDA device addresses on the current device; the
 *     caller owns every buffer.  The library keeps no pointer after a call returns
 *     and allocates no device memory: scratch comes from the caller's workspace.
 *   - Device buffers must be 16-byte aligned (NF4_ERR_ALIGN otherwise).
 *   - "stream" is a cudaStream_t (NULL = legacy default stream).  Work is enqueued
 *     asynchronously; argument, shape and alignment errors are reported
 *     synchronously by the return value and enqueue nothing.
 *   - Conditions only the device can see (a non-finite input found while
 *     quantizing, a bounded wait that gave up) set a per-device status word that
 *     qlora_last_device_status() reads.
 *   - There is no CPU fallback and no silent precision change ([ADAPT] "Explicit
 *     accelerated training profiles": "There is no automatic precision change or
 *     CPU fallback"; unsupported values "fail explicitly").
 *
 * NF4 format ([ADAPT] "Packed NF4 and the portable QLoRA profile"; sizes from
 * [GATE] "P3 is solved" and [QUAL] component_benchmarks.packed_gpu_bytes):
 *   A tensor of numel elements (row-major [N, K] for a weight, flattened) is cut
 *   into nb = ceil(numel/64) blocks.  Element i has a 4-bit code; two codes per
 *   byte, element 2j in the high nibble, 2j+1 in the low nibble (pad nibble 0).
 *   Without double quantization each block has an fp32 absmax.  With it, each
 *   block has a uint8 dynamic8 code of (absmax - offset), nnb = ceil(nb/256) fp32
 *   nested absmax values and one fp32 offset (the mean of all block absmax values).
 *   Decode: a' = dyn8[code] * nested + offset (two roundings, no FMA), then
 *   w = nf4[q] * a'.
 */
#ifndef QLORA_NF4_H
#define QLORA_NF4_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define QLORA_NF4_ABI_VERSION 5

typedef enum {
  NF4_OK = 0,
  NF4_ERR_ARG = 1,        /* null pointer, numel <= 0, bad enum, rank out of 1..256 */
  NF4_ERR_SHAPE = 2,      /* shape the selected path does not support */
  NF4_ERR_ALIGN = 3,      /* a device pointer is not 16-byte aligned */
  NF4_ERR_DTYPE = 4,      /* dtype not allowed for this call */
  NF4_ERR_NONFINITE = 5,  /* NaN or Inf in an input to nf4_quantize (device status) */
  NF4_ERR_CORRUPT = 6,    /* descriptor inconsistent with its numel / double_quant */
  NF4_ERR_CUDA = 7,       /* a CUDA runtime call failed (launch, no device, ...) */
  NF4_ERR_TIMEOUT = 8,    /* a device-side bounded wait gave up (device status) */
  NF4_ERR_WORKSPACE = 9,  /* workspace null or smaller than the size query returns */
  NF4_ERR_TOO_LARGE = 10  /* numel above NF4_QUANTIZE_NOALLOC_MAX_NUMEL (nf4_quantize_noalloc) */
} nf4_status;

/* Element types.  NF4_F16 (IEEE binary16) is the pages' reduced-precision profile ([ADAPT]
 * "Mixed precision keeps stable state in FP32": reconstructed weights rounded to FP16 before
 * multiplication); it is a compute dtype of the linear and an output type of nf4_dequantize. */
typedef enum { NF4_F32 = 0, NF4_BF16 = 1, NF4_F16 = 2 } nf4_dtype;

typedef enum {
  QLORA_SCALE_LORA = 0,   /* s = alpha / rank        ([ADAPT] "LoRA FA includes ...") */
  QLORA_SCALE_RSLORA = 1  /* s = alpha / sqrt(rank)  ([ADAPT] "Adapter API": rs_lora) */
} qlora_scale_mode;

/* One quantized tensor.  All pointers are device pointers owned by the caller. */
typedef struct {
  int64_t numel;          /* number of logical elements (> 0) */
  int32_t double_quant;   /* 1: nested dynamic8 absmax; 0: fp32 absmax */
  int32_t reserved;       /* must be 0 */
  uint8_t* packed;        /* [ceil(numel/2)] two 4-bit codes per byte */
  void* absmax;           /* double_quant: uint8[nb] codes; else float[nb] */
  float* nested_absmax;   /* double_quant: float[nnb]; else NULL */
  float* offset;          /* double_quant: float[1]; else NULL */
} nf4_tensor;

/* ABI version (QLORA_NF4_ABI_VERSION). */
int32_t nf4_abi_version(void);

/* Human-readable name of a status code (static string). */
const char* nf4_status_str(nf4_status s);

/* nb = ceil(numel/64) and nnb = ceil(nb/256); 0 when numel <= 0. */
int64_t nf4_num_blocks(int64_t numel);
int64_t nf4_num_nested(int64_t numel);

/* Device bytes of one quantized tensor without the offset scalar:
 *   double_quant: ceil(n/2) + nb + 4*nnb   ([QUAL] packed_gpu_bytes; [GATE] "P3 is solved")
 *   otherwise:    ceil(n/2) + 4*nb
 * Returns 0 when numel <= 0. */
size_t nf4_packed_bytes(int64_t numel, int32_t double_quant);

/* Copy the library's constant code tables to host memory: 16 NF4 values and 256
 * dynamic8 values, both ascending ([GATE] "P3 is solved": one shared constant copy
 * of each).  Either pointer may be NULL. */
void nf4_code_tables(float* nf4_out16, float* dyn8_out256);

/* Workspace (device bytes) nf4_quantize needs for numel elements. */
size_t nf4_quantize_workspace_bytes(int64_t numel, int32_t double_quant);

/* Quantize x (device, x_dtype NF4_F32 or NF4_BF16, numel elements, contiguous)
 * into *out, whose numel and double_quant select the format and whose pointers
 * receive the result ([ADAPT] "Packed NF4 ...": absmax blocks of 64, nearest of the
 * 16 NF4 codes; with double quantization the block maxima are centred by their
 * global FP32 mean and quantized with dynamic8 in blocks of 256).  Deterministic:
 * the same input gives the same bytes on every call ([GATE] "P3 is solved").
 * ws: device workspace of at least nf4_quantize_workspace_bytes() bytes.
 * A NaN/Inf input sets NF4_ERR_NONFINITE in the device status word; the output
 * bytes are then unspecified. */
nf4_status nf4_quantize(const void* x, nf4_dtype x_dtype, int64_t numel,
                        const nf4_tensor* out, void* ws, size_t ws_bytes, void* stream);

/* Several tensors in one call, e.g. the seven weights of one transformer layer: item i gets
 * exactly what nf4_quantize(items[i].x, items[i].x_dtype, items[i].numel, items[i].out, ...)
 * gives.  Consecutive items of one input dtype run together, up to 8 at a time, as one block
 * pass over all their 64-element blocks and one nested pass over all their maxima, so small
 * tensors share the GPU instead of running one after another.  ws: device workspace of
 * nf4_quantize_batch_workspace_bytes() bytes, 16-byte aligned (each item takes its own slice,
 * laid out in the items' order).  Every item is validated as nf4_quantize validates it; the
 * first failing item's status is returned and nothing is enqueued.  Items must not overlap
 * one another's outputs. */
typedef struct {
  const void* x;            /* device input, 16-byte aligned */
  nf4_dtype x_dtype;        /* NF4_F32 or NF4_BF16 */
  int64_t numel;
  const nf4_tensor* out;    /* preallocated for numel and its double_quant setting */
} nf4_quantize_item;
size_t nf4_quantize_batch_workspace_bytes(int32_t count, const nf4_quantize_item* items);
nf4_status nf4_quantize_batch(int32_t count, const nf4_quantize_item* items, void* ws, size_t ws_bytes,
                              void* stream);

/* nf4_quantize without a workspace, for callers that cannot allocate device
 * memory: code running inside a host engine or framework that owns all device
 * memory and hands it only input and output buffers, or a latency-critical loop
 * where cudaMalloc/cudaFree (and the device synchronization cudaFree implies) are
 * not allowed.  The pages have no counterpart to this entry point; it computes
 * exactly what nf4_quantize computes, with the same kernels.
 * Its scratch is a fixed array of NF4_QUANTIZE_NOALLOC_SCRATCH_BYTES in the
 * library's own device memory, held by every GPU that loads the library until the
 * process exits.  numel above NF4_QUANTIZE_NOALLOC_MAX_NUMEL returns
 * NF4_ERR_TOO_LARGE before any device work.  The first call on a device looks up
 * the array's device address (cudaGetSymbolAddress) with that device current; make
 * that first call before any stream capture.  All calls share the array: calls that
 * overlap on the GPU race on it, so serialize them.  No call allocates memory. */
#define NF4_QUANTIZE_NOALLOC_MAX_NUMEL (67108864LL)        /* 2^26 elements */
#define NF4_QUANTIZE_NOALLOC_SCRATCH_BYTES (4227072u)      /* 4 MiB + 32 KiB */
nf4_status nf4_quantize_noalloc(const void* x, nf4_dtype x_dtype, int64_t numel,
                                const nf4_tensor* out, void* stream);

/* Decode *w into y (device, out_dtype NF4_F32, NF4_BF16 or NF4_F16, w->numel elements).
 * fp32 output is exact nf4[q]*a'; bf16 and half outputs are that value rounded to nearest
 * even ([ADAPT] "Fused GPU NF4 decodes inside the matrix kernel"). */
nf4_status nf4_dequantize(const nf4_tensor* w, void* y, nf4_dtype out_dtype, void* stream);

/* Several tensors in one call, e.g. the seven weights of one transformer layer: item i gets
 * exactly what nf4_dequantize(items[i].w, items[i].y, out_dtype, stream) writes.  Up to 8
 * items at a time decode in one launch per double-quant setting, so small tensors share the
 * GPU instead of running one after another.  Every item is validated as nf4_dequantize
 * validates it; the first failing item's status is returned and nothing is enqueued.
 * Outputs must not overlap. */
typedef struct {
  const nf4_tensor* w;      /* the quantized tensor */
  void* y;                  /* device output, w->numel elements of out_dtype, 16-byte aligned */
} nf4_dequantize_item;
nf4_status nf4_dequantize_batch(int32_t count, const nf4_dequantize_item* items, nf4_dtype out_dtype,
                                void* stream);

/* Selected rows of an NF4-quantized embedding table ([ADAPT] "Packed NF4 and the portable
 * QLoRA profile": embeddings decode only selected rows; "Fused GPU NF4 decodes inside the
 * matrix kernel": selected-row embedding kernels decode on the device):
 *     out[i][d] = deq(E)[ids[i]][d],  i < n_ids, d < dim
 * E: an nf4_tensor of numel rows*dim holding [rows, dim] row-major.  ids: device int64
 * [n_ids].  out: device [n_ids, dim] in out_dtype, the same bits nf4_dequantize writes for
 * those elements.  Shapes and pointers are checked before any launch; an id outside
 * [0, rows) is found on the device: its output row is written as zeros and the device
 * status word is set to NF4_ERR_ARG (qlora_last_device_status). */
nf4_status nf4_embedding_rows(const nf4_tensor* E, int64_t rows, int64_t dim, const int64_t* ids,
                              int64_t n_ids, void* out, nf4_dtype out_dtype, void* stream);

/* Merged deployment weight of an NF4 base and a LoRA adapter ([ADAPT] "Checkpoints,
 * exact continuation and deployment": merged F32 deployment weights with the decoded NF4
 * base, one matrix at a time):
 *     W'[n][k] = deq(W)[n][k] + s * sum_j B[n][j] * A[j][k]
 * W: nf4_tensor of numel N*K holding [N, K] row-major; A fp32 [rank, K], B fp32 [N, rank];
 * s from alpha, rank and mode as for the linear (rank 1..256, rank <= min(N, K)).
 * out: device [N, K] row-major, NF4_F32 or NF4_BF16.  fp32 arithmetic: the decoded value
 * (exactly what nf4_dequantize writes for fp32), d = the rank-r dot product accumulated with
 * fused multiply-adds in order j = 0, 1, ..., then w + s*d with two roundings; bf16 output
 * rounds that fp32 value once (nearest even).  Needs K % 8 == 0 (NF4_ERR_SHAPE otherwise). */
nf4_status nf4_merge_lora(int64_t N, int64_t K, int32_t rank, float alpha, qlora_scale_mode mode,
                          const nf4_tensor* W, const float* A, const float* B, void* out,
                          nf4_dtype out_dtype, void* stream);

/* Workspace (device bytes) needed by qlora_linear_fwd / qlora_linear_bwd.  With
 * compute = NF4_BF16 it includes a bf16 copy of the decoded weight (2*N*K bytes): each
 * call decodes W once into it (the bits nf4_dequantize writes) before the contraction.
 * Calls on different streams need separate workspaces. */
size_t qlora_fwd_workspace_bytes(int64_t M, int64_t N, int64_t K, int32_t rank, nf4_dtype compute);
size_t qlora_bwd_workspace_bytes(int64_t M, int64_t N, int64_t K, int32_t rank, nf4_dtype compute);

/* Forward of the frozen-base QLoRA linear ([ADAPT] "One model contract": the NF4
 * base is frozen and needs an adapter; "Packed NF4 ...": linear operations decode
 * the weight; [ADAPT] "LoRA FA ...": s = alpha / rank):
 *     T = x A^T          (T_out, fp32 [M, rank], kept for the backward pass)
 *     y = x W^T + s T B^T
 * Shapes: x [M, K] row-major, W an nf4_tensor of numel N*K holding [N, K]
 * row-major, A fp32 [rank, K], B fp32 [N, rank], y [M, N].
 * compute = NF4_F32: x and y fp32, fp32 arithmetic, no TF32, any M, N, K >= 1.
 * compute = NF4_BF16: x and y bf16, bf16 tensor-core operands (the decoded weight
 *   rounded once to bf16, A and B rounded to bf16, s*T rounded to bf16) with fp32
 *   accumulation; needs K % 64 == 0 and N % 8 == 0 (NF4_ERR_SHAPE otherwise).
 * compute = NF4_F16: the same with IEEE half in place of bf16 everywhere (the pages' FP16
 *   profile, [ADAPT] "Mixed precision keeps stable state in FP32": reconstructed weights
 *   rounded to FP16 before multiplication; adapters, T and accumulation in fp32).
 *   With M <= 16 the stored weight is streamed once and decoded inside the contraction
 *   (no decoded copy; workspace of a few MB); larger M decodes W once per call into the
 *   workspace and runs the tiled tensor-core GEMM.
 * rank 1..256 ([ADAPT] "Adapter API") and rank <= min(N, K); alpha finite.
 * ws: device workspace of qlora_fwd_workspace_bytes() bytes. */
nf4_status qlora_linear_fwd(int64_t M, int64_t N, int64_t K, int32_t rank, float alpha,
                            qlora_scale_mode mode, nf4_dtype compute,
                            const void* x, const nf4_tensor* W, const float* A, const float* B,
                            void* y, float* T_out, void* ws, size_t ws_bytes, void* stream);

/* Forward of several projections that share M and the compute dtype, for example the seven
 * projections of one transformer layer ([GATE] "Shape-matched ceilings": q, k, v, o, gate, up,
 * down).  Item i computes what qlora_linear_fwd (w16 == NULL) or qlora_linear_fwd_w16
 * (w16 != NULL: W decoded as nf4_dequantize writes it; W may then be NULL) computes for its
 * arguments: the same operands and products, with some fp32 partial sums added in another
 * order where the item shares a pass's work split with other items (the M <= 16 pass; the T
 * passes of a run that reads more than one x), so y and T_out may differ from the single
 * call's in their last bits.  The results are deterministic for a given batch.
 *   - compute = NF4_BF16 or NF4_F16, M <= 16, items given as NF4: up to 8 run as one pair of
 *     launches (T for every item, then one persistent pass over all their stored weights).
 *   - 16-bit compute, small weights (M > 16, K and N at most 1024, N*K at most 2^21, rank at
 *     most 32): up to 8 at a time in one launch.
 *   - 16-bit compute, the other items (the tiled tensor-core path): up to 8 consecutive
 *     such items run together.  Their NF4 weights are decoded in one launch, and one launch
 *     computes T for all of them: items in a row that read the same x (the same pointer and
 *     K; a layer's q, k and v, or gate and up) share one pass over x as long as their ranks,
 *     each rounded up to 16, add up to at most 256.  Then each item's GEMM runs.  A run of
 *     one item is the single call.
 *   - anything else runs the single call.
 * Items must not write to memory another item reads.  ws: qlora_fwd_batch_workspace_bytes()
 * bytes.  Each item is validated as the single call validates it; the first failing item's
 * status is returned and nothing is enqueued. */
typedef struct {
  int64_t N, K;
  int32_t rank;
  float alpha;
  qlora_scale_mode mode;
  const nf4_tensor* W;    /* numel N*K, [N, K] row-major; or NULL with w16 */
  const float* A;         /* [rank, K] fp32 */
  const float* B;         /* [N, rank] fp32 */
  const void* x;          /* [M, K] in the compute dtype */
  void* y;                /* [M, N] in the compute dtype */
  float* T_out;           /* [M, rank] fp32 */
  const void* w16;        /* [N, K] decoded in the compute dtype (16-bit compute only), or NULL */
} qlora_fwd_item;

size_t qlora_fwd_batch_workspace_bytes(int64_t M, int32_t count, const qlora_fwd_item* items, nf4_dtype compute);
nf4_status qlora_linear_fwd_batch(int64_t M, int32_t count, const qlora_fwd_item* items, nf4_dtype compute,
                                  void* ws, size_t ws_bytes, void* stream);

/* Backward ([ADAPT] "Packed NF4 ...": input gradients through the frozen base, no
 * base-weight gradient; [GATE] "The TFLOPS back-check": no dL/dW), in the same three
 * compute dtypes as the forward:
 *     G  = dY B                    (internal, fp32 [M, rank])
 *     dX = dY W + s G A            [M, K], dtype of compute
 *     dA = s G^T x                 fp32 [rank, K]  (overwritten, not accumulated)
 *     dB = s dY^T T                fp32 [N, rank]  (overwritten, not accumulated)
 * dy [M, N] and x [M, K] in the compute dtype; T is the forward's T_out.
 * Shape rules as for the forward.  Reductions are deterministic (no atomics). */
nf4_status qlora_linear_bwd(int64_t M, int64_t N, int64_t K, int32_t rank, float alpha,
                            qlora_scale_mode mode, nf4_dtype compute,
                            const void* dy, const void* x, const float* T,
                            const nf4_tensor* W, const float* A, const float* B,
                            void* dx, float* dA, float* dB,
                            void* ws, size_t ws_bytes, void* stream);

/* The 16-bit profiles with the weight already decoded, so that one decode serves several
 * calls, e.g. the forward and the backward of one step ([ADAPT] "Fused GPU NF4 decodes inside
 * the matrix kernel": the reconstructed weight is what the contraction multiplies).
 * w16: device [N, K] row-major in the compute dtype (NF4_BF16 or NF4_F16; NF4_ERR_DTYPE
 * otherwise), holding the weight as nf4_dequantize writes it for that dtype; the library
 * cannot check that, and with any other contents the result is that of those contents.
 * Every other argument, the arithmetic and the results are those of qlora_linear_fwd /
 * qlora_linear_bwd for the weight w16 decodes, bit for bit on the tiled path (every M; the
 * small-M pass of qlora_linear_fwd, which decodes in registers, is not used here).  The
 * workspaces hold no decoded copy (2*N*K bytes smaller than the tiled path's).  w16 is read,
 * never written, and must stay unchanged until the call's work on the stream is done. */
size_t qlora_fwd_w16_workspace_bytes(int64_t M, int64_t N, int64_t K, int32_t rank, nf4_dtype compute);
size_t qlora_bwd_w16_workspace_bytes(int64_t M, int64_t N, int64_t K, int32_t rank, nf4_dtype compute);
nf4_status qlora_linear_fwd_w16(int64_t M, int64_t N, int64_t K, int32_t rank, float alpha,
                                qlora_scale_mode mode, nf4_dtype compute,
                                const void* x, const void* w16, const float* A, const float* B,
                                void* y, float* T_out, void* ws, size_t ws_bytes, void* stream);
nf4_status qlora_linear_bwd_w16(int64_t M, int64_t N, int64_t K, int32_t rank, float alpha,
                                qlora_scale_mode mode, nf4_dtype compute,
                                const void* dy, const void* x, const float* T, const void* w16,
                                const float* A, const float* B, void* dx, float* dA, float* dB,
                                void* ws, size_t ws_bytes, void* stream);

/* Backward of several projections that share M and the compute dtype, e.g. the projections of
 * one layer that read the same x (q, k and v): item i computes what qlora_linear_bwd
 * (w16 == NULL) or qlora_linear_bwd_w16 (w16 != NULL: W decoded as nf4_dequantize writes it)
 * computes for its arguments; W may be NULL when w16 is given.  dX and dB are the single
 * call's bits; dA's fp32 partial sums are added in another order when the run reads more
 * than one x (deterministic for a given batch).  Items with small
 * weights (16-bit compute, M > 16, K and N at most 1024, N*K at most 2^21, rank at most 32)
 * run up to 8 at a time in one pair of launches.  Other 16-bit items run up to 8 at a time
 * as in qlora_linear_fwd_batch: one launch for every item's G and dB passes, each item's dX
 * GEMM, then one launch for every item's dA, where items in a row that read the same x share
 * one pass over x.  The others run one call each.  Items must not write to memory another
 * item reads.  ws: qlora_bwd_batch_workspace_bytes() bytes.  Each item is validated as the
 * single call validates it; the first failing item's status is returned and nothing is
 * enqueued. */
typedef struct {
  int64_t N, K;
  int32_t rank;
  float alpha;
  qlora_scale_mode mode;
  const nf4_tensor* W;    /* numel N*K, [N, K] row-major; or NULL with w16 */
  const void* w16;        /* [N, K] decoded in the compute dtype, or NULL */
  const float* A;         /* [rank, K] fp32 */
  const float* B;         /* [N, rank] fp32 */
  const void* dy;         /* [M, N] in the compute dtype */
  const void* x;          /* [M, K] in the compute dtype */
  const float* T;         /* [M, rank] fp32, the forward's T_out */
  void* dx;               /* [M, K] in the compute dtype */
  float* dA;              /* [rank, K] fp32 */
  float* dB;              /* [N, rank] fp32 */
} qlora_bwd_item;

size_t qlora_bwd_batch_workspace_bytes(int64_t M, int32_t count, const qlora_bwd_item* items, nf4_dtype compute);
nf4_status qlora_linear_bwd_batch(int64_t M, int32_t count, const qlora_bwd_item* items, nf4_dtype compute,
                                  void* ws, size_t ws_bytes, void* stream);

/* Synchronize `stream`, then return the current device's status word (NF4_OK if no
 * device-side condition was recorded); clear != 0 resets it to NF4_OK. */
nf4_status qlora_last_device_status(void* stream, int32_t clear);

/* Test support for the timeout path of the library's bounded device waits.  After a call
 * with on != 0, the next tensor-core contraction launched (the bf16 GEMM of qlora_linear_fwd /
 * qlora_linear_bwd, or the small-M weight pass of the forward) runs with a 20 ms wait limit
 * instead of 4 s, and its first CTA does not issue the copies of its first pipeline stage, so
 * the waits for that stage run out.  That launch winds down (copies in flight land, TMEM is
 * freed), NF4_ERR_TIMEOUT is set in the device status word and its outputs are unspecified;
 * nothing faults or hangs, and later calls are unaffected.  on = 0 disarms a pending request. */
void qlora_debug_wait_timeout(int32_t on);

/* Number of kernels this library has launched in this process (all devices). */
int64_t nf4_kernel_launch_count(void);

/* Optional timing of the library's kernels, for benchmarks.  While enabled, each
 * timed kernel (or kernel sequence, for nf4_quantize) is bracketed by a pair of
 * CUDA events recorded on the stream it is launched on.  nf4_timing_read()
 * waits for the recorded pairs of one kind, returns the summed milliseconds and
 * the number of launches, and with reset != 0 clears that kind.  No device memory
 * is allocated; events are created once and reused. */
typedef enum {
  NF4_TIME_QUANTIZE = 0,    /* the kernels of one nf4_quantize call (two with double quantization) */
  NF4_TIME_DEQUANTIZE = 1,  /* the decode kernel */
  NF4_TIME_FWD_GEMM = 2,    /* base contraction of the forward (y) */
  NF4_TIME_DX_GEMM = 3,     /* base contraction of the input gradient (dX) */
  NF4_TIME_ADAPTER = 4,     /* adapter-side kernels (T, G, dA, dB) */
  NF4_TIME_WEIGHT_DECODE = 5, /* the bf16 profile's per-call decode of W before its GEMM,
                               * with the call's operand staging in the same launch */
  NF4_TIME_EMBEDDING = 6,   /* nf4_embedding_rows */
  NF4_TIME_MERGE = 7,       /* nf4_merge_lora */
  NF4_TIME_STREAM_FWD = 8,  /* the forward's small-M pair of launches (T, then the weight pass) */
  NF4_TIME_KINDS = 9
} nf4_timed_kernel;

void nf4_timing_enable(int32_t on);
nf4_status nf4_timing_read(int32_t kind, double* total_ms, int64_t* launches, int32_t reset);

#ifdef __cplusplus
}
#endif

#endif /* QLORA_NF4_H */
