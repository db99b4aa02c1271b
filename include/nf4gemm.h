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
 *  - same page, quantized-GEMM paragraph: fp32 outputs.
 *
 * Storage format (all buffers row-major and contiguous):
 *  - W is [rows = N (out features), cols = K (in features)], fp32.
 *  - Blocks of 64 and groups of 256 blocks run over W flattened row-major.
 *    cols is a multiple of 64, so a block never straddles a row; a group may.
 *  - codes:        uint8 [rows*cols/2]; element 2j in the high nibble of byte
 *                  j, element 2j+1 in the low nibble. Code q means level c[q]
 *                  of the NF4 table (nf4_codebook).
 *  - absmax_q:     uint8 [rows*cols/64]; a8 = round(255 * absmax / s2).
 *  - absmax_scale: fp32  [ceil(rows*cols/64/256)]; s2 = max absmax of the group.
 *  - Dequantized weight: ahat = fl32(fl32(a8 * s2) / 255),
 *                        w = fl32(c[q] * ahat).
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

/* A quantized weight (the QuantState of the bitsandbytes page, reduced to
 * plain device pointers). All three arrays are device pointers owned by the
 * caller, in the storage format above. */
typedef struct nf4_weight {
  const uint8_t* codes;         /* [rows*cols/2]                 */
  const uint8_t* absmax_q;      /* [rows*cols/64]                */
  const float* absmax_scale;    /* [ceil(rows*cols/64/256)]      */
  int64_t rows;                 /* N: output features            */
  int64_t cols;                 /* K: input features, % 64 == 0  */
  int32_t blocksize;            /* must be 64                    */
  int32_t dq_group;             /* must be 256                   */
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

/* Dequantize to fp32 ("bitsandbytes", double-quantization paragraph: scales
 * first, then weights). W_out: device fp32 [rows, cols] (output). The one
 * entry point that writes a full-precision weight, for checking and export. */
nf4_status nf4_dequantize(const nf4_weight* w, float* W_out, void* stream);

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
 * Determinism: when the output tiles alone cannot fill the GPU the reduction
 * is split across CTAs and the partial sums are added into Y with fp32
 * atomics, in an order that varies between runs, so the low bits of Y can
 * differ between identical calls. The small-M kernel reduces its splits in
 * a fixed order and is bitwise repeatable. */
nf4_status nf4_matmul_fwd(const uint16_t* X, int64_t M, const nf4_weight* w, float* Y,
                          void* stream);

/* Fused frozen-base backward dX = dY * dequant(W) ("Zenbit", zenbit.pallas_nf4
 * bullet: dL/dX without materialising the dequantized weight; dL/dW is not
 * computed).
 *   dY device bf16 (raw uint16 bits) [M, rows]
 *   dX device fp32 [M, cols] (output, overwritten)
 * Requires rows % 8 == 0. Same accuracy statement as nf4_matmul_fwd, and
 * the same determinism note: split reductions (small grids, and M <= 16)
 * add partial sums with atomics. */
nf4_status nf4_matmul_bwd_dx(const uint16_t* dY, int64_t M, const nf4_weight* w, float* dX,
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

/* Host-only: static description of a status code. */
const char* nf4_status_string(nf4_status status);

#ifdef __cplusplus
}
#endif

#endif /* NF4GEMM_H */
