/*
 * nf4gemm.h - C ABI of the GB300 (sm_103a) NF4 quantize / fused NF4-dequant
 * matmul library (libnf4gemm.so).
 *
 * The method (sources by page title and section):
 *  - "Zenbit" (pypi.org/project/zenbit), "What's inside", zenbit.nf4 bullet:
 *    NF4 blockwise quantization with double quantization of the scales.
 *  - same page, zenbit.pallas_nf4 bullet: fused NF4 dequant + matmul that
 *    streams the compressed weight and dequantizes on chip, never writing the
 *    full-precision weight to HBM; the backward computes dL/dX only (a frozen
 *    quantized base weight has no dL/dW).
 *  - "bitsandbytes" (unfragile.ai/artifact/bitsandbytes), NF4 paragraph: 16
 *    levels from the inverse normal CDF, mapped through a lookup table.
 *  - same page, double-quantization paragraph: one absmax per 64-weight block,
 *    the absmax vector quantized to 8 bits with its own scales; scales are
 *    dequantized first, then the weights.
 *  - same page, QuantState paragraph: a quantized weight is its codes, its
 *    scales, its data type and its shape (nf4_weight below).
 *  - same page, quantized-GEMM paragraph: fp32 outputs; int8 or 4-bit
 *    weights; float16/float32 activations.
 *  - same page, 4-bit paragraph: NF4 or FP4 (standard floating-point 4-bit)
 *    with double quantization; 4-bit weights dequantized to float16/float32
 *    and LoRA adapter outputs added to the layer's output.
 *  - "Zenbit", zenbit.int8 bullet: uniform int8 weight quantization.
 *
 * Storage format of the 4-bit data types, NF4 and FP4 (all buffers row-major
 * and contiguous):
 *  - W is [rows = N (out features), cols = K (in features)], fp32 or bf16.
 *  - Blocks of 64 and groups of 256 blocks run over W flattened row-major.
 *    cols is a multiple of 64, so a block never straddles a row; a group may.
 *  - codes:        uint8 [rows*cols/2]; element 2j in the high nibble of byte
 *                  j, element 2j+1 in the low nibble. Code q means level c[q]
 *                  of the NF4 table (nf4_codebook).
 *  - absmax_q:     uint8 [rows*cols/64]; a8 = round(255 * absmax / s2).
 *  - absmax_scale: fp32  [ceil(rows*cols/64/256)]; s2 = max absmax of the group.
 *  - Dequantized weight: ahat = fl32(fl32(a8 * s2) / 255),
 *                        w = fl32(c[q] * ahat).
 *  - NF4 levels: nf4_codebook. FP4 levels (nf4_codebook_of): the E2M1 code
 *    (sign bit 3, exponent bits 2-1 with bias 1, mantissa bit 0) of the
 *    magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6, divided by 6; code 8 is -0, and
 *    a weight that rounds to magnitude 0 gets code 0 whatever its sign.
 *
 * Storage format of the int8 data type (uniform symmetric, per block):
 *  - codes:        int8 [rows*cols]; q = round(127 * w / absmax), half to even.
 *  - absmax_q:     unused (NULL).
 *  - absmax_scale: fp32 [rows*cols/64]; absmax of each 64-weight block.
 *  - Dequantized weight: w = fl32(fl32(q * absmax) / 127).
 *
 * Conventions for every entry point:
 *  - Pointers marked "device" must be device-accessible (cudaMalloc'd or
 *    equivalent) and 16-byte aligned; the caller allocates and owns every
 *    buffer. The library allocates no device memory.
 *  - Calls are asynchronous on `stream` (a cudaStream_t; NULL means the legacy
 *    default stream) and do not synchronize, except nf4_poll_device_status.
 *  - Arguments are validated on the host before anything is launched; an
 *    invalid call returns a status other than NF4_OK and launches nothing.
 *  - A call with an empty extent (rows, cols or M equal to 0) returns NF4_OK
 *    and touches no pointer.
 *  - The kernels require an sm_103 device (NF4_ERR_DEVICE otherwise).
 *  - Every wait inside a kernel is bounded in time. A kernel that gives up
 *    records NF4_ERR_DEVICE_TIMEOUT in a device status word which
 *    nf4_poll_device_status reports; it never traps.
 *  - Thread-safe: no host-side mutable state except per-device set-up done
 *    once under a lock.
 */
#ifndef NF4GEMM_H
#define NF4GEMM_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum nf4_status {
  NF4_OK = 0,
  NF4_ERR_NULL = 1,            /* a required pointer is NULL                  */
  NF4_ERR_SHAPE = 2,           /* negative extent or unsupported shape        */
  NF4_ERR_ALIGN = 3,           /* a pointer is not 16-byte aligned            */
  NF4_ERR_BLOCKSIZE = 4,       /* blocksize != 64 or dq_group != 256          */
  NF4_ERR_DEVICE = 5,          /* no current device, or it is not sm_103      */
  NF4_ERR_LAUNCH = 6,          /* the CUDA runtime rejected a launch          */
  NF4_ERR_DEVICE_TIMEOUT = 7   /* a kernel's bounded wait ran out             */
} nf4_status;

/* Weight data types (the "data type (NF4/FP4/INT8)" of the bitsandbytes
 * page's QuantState paragraph). */
typedef enum nf4_dtype {
  NF4_DTYPE_NF4 = 0,           /* 4-bit NormalFloat codes, double-quantized absmax */
  NF4_DTYPE_FP4 = 1,           /* 4-bit E2M1 codes, double-quantized absmax        */
  NF4_DTYPE_INT8 = 2           /* int8 values, fp32 absmax per 64-weight block     */
} nf4_dtype;

/* Element types of activations, outputs and quantize inputs. */
typedef enum nf4_elem {
  NF4_F32 = 0,
  NF4_BF16 = 1,                /* raw bf16 bits in uint16 */
  NF4_F16 = 2                  /* raw IEEE half bits in uint16 */
} nf4_elem;

/* Flags of the fused matmuls. */
#define NF4_ACCUMULATE 1       /* add the product to the output's contents */

/* Most weights one nf4_matmul_fwd_group call takes. */
#define NF4_GROUP_MAX 4

/* A quantized weight (the QuantState of the bitsandbytes page, reduced to
 * plain device pointers). All arrays are device pointers owned by the
 * caller, in the storage format of `dtype` above. A zero-initialised dtype
 * is NF4. */
typedef struct nf4_weight {
  const uint8_t* codes;         /* 4-bit: [rows*cols/2]; int8: [rows*cols]        */
  const uint8_t* absmax_q;      /* 4-bit: [rows*cols/64]; int8: NULL              */
  const float* absmax_scale;    /* 4-bit: [ceil(rows*cols/16384)]; int8: [rows*cols/64] */
  int64_t rows;                 /* N: output features                             */
  int64_t cols;                 /* K: input features, % 64 == 0                   */
  int32_t blocksize;            /* must be 64                                     */
  int32_t dq_group;             /* 4-bit: must be 256; int8: must be 0            */
  int32_t dtype;                /* nf4_dtype                                      */
} nf4_weight;

/* NF4-quantize W with double-quantized absmax ("Zenbit", zenbit.nf4 bullet;
 * "bitsandbytes", NF4 and double-quantization paragraphs).
 *   W            device fp32 [rows, cols], finite, |W| <= 1e36.
 *   blocksize    must be 64 (NF4_ERR_BLOCKSIZE otherwise).
 *   codes        device uint8 [rows*cols/2]            (output)
 *   absmax_q     device uint8 [rows*cols/64]           (output)
 *   absmax_scale device fp32  [ceil(rows*cols/16384)]  (output)
 * Each weight is normalised by its block's fp32 absmax (IEEE quotient) and
 * given the code of the nearest level, ties to the lower code; an all-zero
 * block gets code 7 (level 0). cols % 64 != 0 -> NF4_ERR_SHAPE. */
nf4_status nf4_quantize(const float* W, int64_t rows, int64_t cols, int32_t blocksize,
                        uint8_t* codes, uint8_t* absmax_q, float* absmax_scale,
                        void* stream);

/* Quantize W of element type w_elem (NF4_F32, or NF4_BF16: real checkpoints
 * are bf16, whose values the fp32 path then sees exactly) into the data type
 * `dtype` ("bitsandbytes", 4-bit paragraph: NF4 or FP4 with double
 * quantization; "Zenbit", zenbit.int8 bullet: uniform int8).
 *   4-bit: as nf4_quantize, with the table of `dtype`.
 *   int8:  codes device int8 [rows*cols], absmax_q must be NULL,
 *          absmax_scale device fp32 [rows*cols/64]; q = round(fl32(fl32(127 w)
 *          / absmax)) half to even, 0 in an all-zero block.
 * Same validation and errors as nf4_quantize; an unknown dtype or element
 * type is NF4_ERR_SHAPE. */
nf4_status nf4_quantize_ex(const void* W, int32_t w_elem, int64_t rows, int64_t cols,
                           int32_t blocksize, int32_t dtype, uint8_t* codes, uint8_t* absmax_q,
                           float* absmax_scale, void* stream);

/* Dequantize to fp32 ("bitsandbytes", double-quantization paragraph: scales
 * first, then weights), for any dtype. W_out: device fp32 [rows, cols]
 * (output). The one entry point that writes a full-precision weight, for
 * checking and export. */
nf4_status nf4_dequantize(const nf4_weight* w, float* W_out, void* stream);

/* Dequantize to fp32, fp16 or bf16 ("bitsandbytes", 4-bit paragraph: 4-bit
 * weights dequantized to float16 or float32; bf16, the tensor-core operand
 * type of the fused kernels, is this library's addition). W_out: device
 * [rows, cols] of out_elem NF4_F32, NF4_F16 or NF4_BF16 (output, 16-byte
 * aligned). A 16-bit output is the fp32 value of nf4_dequantize rounded to
 * nearest even (fp16 overflows to infinity beyond 65504). NF4_ERR_SHAPE for
 * another out_elem, before any device access. */
nf4_status nf4_dequantize_ex(const nf4_weight* w, void* W_out, int32_t out_elem, void* stream);

/* Fused forward Y = X * dequant(W)^T ("Zenbit", zenbit.pallas_nf4 bullet;
 * "bitsandbytes", quantized-GEMM paragraph). The dequantized weight exists
 * only in registers, shared memory and tensor memory.
 *   X  device bf16 (raw uint16 bits) [M, cols]
 *   Y  device fp32 [M, rows] (output, overwritten)
 * Requires rows % 8 == 0; any cols that is a multiple of 64 is accepted.
 * M <= 16 with cols <= 49152 runs the streaming small-M kernel, every other
 * shape the tensor-core kernel. Accuracy against an fp64
 * dequantize-then-multiply: relative Frobenius error <= 2e-3 and max error
 * <= 5e-3 * max|Y_ref| (weights enter the tensor cores as bf16, or as fp16
 * levels with the block scale applied in fp32 on the small-M kernel).
 * Determinism: when the output tiles alone cannot fill the GPU, or would
 * leave its last round of tiles partly idle, the reduction is split across
 * CTAs and the partial sums are added into Y with fp32 atomics, in an order
 * that varies between runs, so the low bits of Y can differ between
 * identical calls. The small-M kernel reduces its splits in a fixed order
 * and is bitwise repeatable. */
nf4_status nf4_matmul_fwd(const uint16_t* X, int64_t M, const nf4_weight* w, float* Y,
                          void* stream);

/* Fused frozen-base backward dX = dY * dequant(W) ("Zenbit", zenbit.pallas_nf4
 * bullet: dL/dX without materialising the dequantized weight; dL/dW is not
 * computed).
 *   dY device bf16 (raw uint16 bits) [M, rows]
 *   dX device fp32 [M, cols] (output, overwritten)
 * Requires rows % 8 == 0. Same accuracy statement as nf4_matmul_fwd, and
 * the same determinism note: split reductions add partial sums with
 * atomics. */
nf4_status nf4_matmul_bwd_dx(const uint16_t* dY, int64_t M, const nf4_weight* w, float* dX,
                             void* stream);

/* The fused forward with a choice of element types and epilogue:
 *   X     device [M, cols], x_elem NF4_BF16 or NF4_F16 ("bitsandbytes",
 *         quantized-GEMM paragraph: float16 activations)
 *   Y     device [M, rows], y_elem NF4_F32 or NF4_BF16
 *   flags NF4_ACCUMULATE: Y = X * dequant(W)^T + Y (the LoRA output add of
 *         the bitsandbytes 4-bit paragraph, fused into the epilogue);
 *         otherwise Y is overwritten.
 * Weights of any dtype. With fp16 activations the dequantized weight enters
 * the tensor cores as fp16 and must lie within fp16's range (|w| < 65504;
 * weights below 2^-14 lose precision as fp16 subnormals). A bf16 output is
 * the fp32 result rounded to nearest even; its reduction is never split
 * across CTAs, so it is bitwise repeatable. With fp32 output and
 * NF4_ACCUMULATE a split reduction adds its partial sums into Y directly.
 * Accuracy as nf4_matmul_fwd, plus the bf16 rounding of the output. */
nf4_status nf4_matmul_fwd_ex(const void* X, int32_t x_elem, int64_t M, const nf4_weight* w,
                             void* Y, int32_t y_elem, int32_t flags, void* stream);

/* The frozen-base input gradient with the same choices:
 *   dY [M, rows] (dy_elem NF4_BF16 or NF4_F16), dX [M, cols] (dx_elem
 *   NF4_F32 or NF4_BF16), flags NF4_ACCUMULATE: dX += dY * dequant(W). */
nf4_status nf4_matmul_bwd_dx_ex(const void* dY, int32_t dy_elem, int64_t M, const nf4_weight* w,
                                void* dX, int32_t dx_elem, int32_t flags, void* stream);

/* The fused forward of up to NF4_GROUP_MAX weights that read the same
 * activations (the q, k and v projections of an attention layer, or the gate
 * and up projections of an MLP): Y_i = X * dequant(W_i)^T for i < count.
 * The method is nf4_matmul_fwd_ex's ("Zenbit", zenbit.pallas_nf4 bullet);
 * putting the weights in one launch is this library's choice, so that a
 * decode step pays the launch latency once per shared input.
 *   X      device [M, cols], x_elem NF4_BF16 or NF4_F16
 *   ws     host array of `count` weights, 1 <= count <= NF4_GROUP_MAX, all
 *          with the same cols and dtype (rows may differ)
 *   Ys     host array of `count` device outputs; Ys[i] is [M, ws[i].rows]
 *          of y_elem (NF4_F32 or NF4_BF16)
 *   flags  NF4_ACCUMULATE or 0, as nf4_matmul_fwd_ex
 * With M <= 16 and cols <= 49152 every weight runs in one launch of the
 * small-M kernel, one grid over all their row tiles; otherwise each weight
 * is one tensor-core launch, in order, on `stream`. The results are those of
 * count nf4_matmul_fwd_ex calls, up to the order of the fp32 sums (the
 * accuracy statement is the same). Every weight and output is validated as
 * nf4_matmul_fwd_ex does before anything is launched; ws or Ys NULL is
 * NF4_ERR_NULL; count out of range, or weights that differ in cols or dtype,
 * NF4_ERR_SHAPE. */
nf4_status nf4_matmul_fwd_group(const void* X, int32_t x_elem, int64_t M, const nf4_weight* ws,
                                int32_t count, void* const* Ys, int32_t y_elem, int32_t flags,
                                void* stream);

/* Synchronizes `stream`, then reports and clears the device status word of
 * the current device: NF4_ERR_DEVICE_TIMEOUT if any kernel's bounded wait ran
 * out since the last poll, NF4_ERR_LAUNCH if the stream holds a CUDA error,
 * NF4_OK otherwise. */
nf4_status nf4_poll_device_status(void* stream);

/* As nf4_poll_device_status, and if `site` is not NULL it receives where the
 * first timeout since the last poll happened (0 when there was none):
 *   bits 28-31  kernel: 1 small-M forward, 2 tensor-core forward,
 *               3 tensor-core input gradient
 *   bits 24-27  role: 1 copy producer, 2 MMA issuer, 3 dequantizing /
 *               computing warp, 4 epilogue
 *   bits  0-23  linear index of the CTA within its grid (low 24 bits).
 * Diagnostic only; the status value is the same. */
nf4_status nf4_poll_device_status_site(void* stream, int32_t* site);

/* Host-only: copies the 16 fp32 NF4 levels compiled into the library into
 * out16 (host memory). Needs no device. */
nf4_status nf4_codebook(float* out16);

/* Host-only: the 16 fp32 levels of a 4-bit dtype (NF4_DTYPE_NF4 or
 * NF4_DTYPE_FP4), by code, into out16 (host memory); NF4_ERR_SHAPE for any
 * other dtype. */
nf4_status nf4_codebook_of(int32_t dtype, float* out16);

/* Diagnostic, for testing the timeout path: from the next launch on, the
 * tensor-core kernels' MMA issuer gives up waiting for a dequantized stage
 * after `cycles` clock cycles (<= 0 restores the default of about a second)
 * and the kernel takes its abort path: it records NF4_ERR_DEVICE_TIMEOUT
 * with its site, lets its copies and MMAs in flight finish, frees its
 * tensor memory and returns; its output is then unspecified. Process-wide;
 * every other wait keeps its full limit. */
nf4_status nf4_set_mma_wait_limit(int64_t cycles);

/* Host-only: the CUDA runtime's description of the error behind the calling
 * thread's most recent NF4_ERR_LAUNCH ("no error" if there was none). */
const char* nf4_last_cuda_error(void);

/* Host-only: static description of a status code. */
const char* nf4_status_string(nf4_status status);

#ifdef __cplusplus
}
#endif

#endif /* NF4GEMM_H */
