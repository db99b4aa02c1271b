// Shared definitions of the NF4 CUDA library (device side and host side).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include <mutex>

#include "nf4gemm.h"

namespace nf4 {

constexpr int kBlock = 64;                    // weights per absmax block
constexpr int kGroup = 256;                   // blocks per second-level scale
constexpr int kGroupElems = kBlock * kGroup;  // 16384 weights per group
// Longest reduction the small-M forward takes: at most 8 K-slices (the
// portable cluster size) of at most 96 blocks each. Longer rows go to the
// tensor-core kernel.
constexpr int64_t kGemvMaxCols = 8 * 96 * kBlock;
// Most weights a grouped small-M forward takes in one launch.
constexpr int kGemvGroupMax = NF4_GROUP_MAX;

// The 16 NF4 levels: standard-normal quantiles at evenly spaced probabilities
// (8 on the positive side from delta = (1 - 1/30 + 1 - 1/32) / 2 to 1/2,
// 7 on the negative side), an exact 0, all divided by Phi^-1(delta) and
// rounded once to fp32 ("bitsandbytes", NF4 paragraph: levels derived from
// the inverse normal CDF). Stored as bit patterns.
constexpr uint32_t kLevelBits[16] = {
    0xbf800000u, 0xbf3239b1u, 0xbf066b2eu, 0xbeca329eu, 0xbe91a24bu, 0xbe3d353du,
    0xbdba7869u, 0x00000000u, 0x3da2fb01u, 0x3e24cadfu, 0x3e7c04dau, 0x3ead0336u,
    0x3ee1a4b5u, 0x3f1007a9u, 0x3f3913b0u, 0x3f800000u};

// Device copy of the levels for run-time indexing (one per translation unit).
static __constant__ uint32_t kLevelBitsDev[16] = {
    0xbf800000u, 0xbf3239b1u, 0xbf066b2eu, 0xbeca329eu, 0xbe91a24bu, 0xbe3d353du,
    0xbdba7869u, 0x00000000u, 0x3da2fb01u, 0x3e24cadfu, 0x3e7c04dau, 0x3ead0336u,
    0x3ee1a4b5u, 0x3f1007a9u, 0x3f3913b0u, 0x3f800000u};

// The 16 FP4 levels by code: E2M1 (sign bit 3, exponent bits 2-1 with bias 1,
// mantissa bit 0; exponent 0 subnormal), magnitudes 0, 0.5, 1, 1.5, 2, 3, 4,
// 6 divided by 6 and rounded once to fp32 ("bitsandbytes", 4-bit paragraph:
// NF4 or standard floating-point 4-bit). Code 8 is -0.
constexpr uint32_t kFp4LevelBits[16] = {
    0x00000000u, 0x3daaaaabu, 0x3e2aaaabu, 0x3e800000u, 0x3eaaaaabu, 0x3f000000u,
    0x3f2aaaabu, 0x3f800000u, 0x80000000u, 0xbdaaaaabu, 0xbe2aaaabu, 0xbe800000u,
    0xbeaaaaabu, 0xbf000000u, 0xbf2aaaabu, 0xbf800000u};

static __constant__ uint32_t kFp4LevelBitsDev[16] = {
    0x00000000u, 0x3daaaaabu, 0x3e2aaaabu, 0x3e800000u, 0x3eaaaaabu, 0x3f000000u,
    0x3f2aaaabu, 0x3f800000u, 0x80000000u, 0xbdaaaaabu, 0xbe2aaaabu, 0xbe800000u,
    0xbeaaaaabu, 0xbf000000u, 0xbf2aaaabu, 0xbf800000u};

// Weight formats (the nf4_dtype values of the C ABI).
constexpr int kFmtNf4 = NF4_DTYPE_NF4, kFmtFp4 = NF4_DTYPE_FP4, kFmtInt8 = NF4_DTYPE_INT8;

__host__ __device__ constexpr const uint32_t (&level_bits(int fmt))[16] {
  return fmt == kFmtFp4 ? kFp4LevelBits : kLevelBits;
}

// FP4 magnitude thresholds: t[i] is the largest fp32 value not above the
// exact midpoint of magnitudes i and i + 1 (of the fp32 levels). With ties to
// the lower code, a value of magnitude |x| gets magnitude #{i : |x| > t[i]};
// a magnitude of 0 is code 0 (+0) whatever the sign, since +0 comes first.
__host__ __device__ constexpr uint32_t fp4_threshold_bits(int i) {
  return i == 0 ? 0x3d2aaaabu : i == 1 ? 0x3e000000u : i == 2 ? 0x3e555555u
       : i == 3 ? 0x3e955555u : i == 4 ? 0x3ed55555u : i == 5 ? 0x3f155555u : 0x3f555555u;
}

// Decision thresholds between neighbouring levels: t[i] is the largest fp32
// value not above the exact midpoint (c[i] + c[i+1]) / 2. For an fp32 x the
// nearest level, ties to the lower index, is #{i : x > t[i]}. A constexpr
// function so that unrolled device loops see immediates.
__host__ __device__ constexpr uint32_t threshold_bits(int i) {
  return i == 0 ? 0xbf591cd9u : i == 1 ? 0xbf1c5270u : i == 2 ? 0xbeeb847du
       : i == 3 ? 0xbeadea75u : i == 4 ? 0xbe703ceau : i == 5 ? 0xbe0d38b9u
       : i == 6 ? 0xbd3a7869u : i == 7 ? 0x3d22fb01u : i == 8 ? 0x3df6485fu
       : i == 9 ? 0x3e5067dcu : i == 10 ? 0x3e9582d1u : i == 11 ? 0x3ec753f5u
       : i == 12 ? 0x3f006d01u : i == 13 ? 0x3f248dacu : 0x3f5c89d8u;
}

__host__ __device__ inline float bits_to_float(uint32_t b) {
#ifdef __CUDA_ARCH__
  return __uint_as_float(b);
#else
  union { uint32_t u; float f; } v;
  v.u = b;
  return v.f;
#endif
}

// fp32 -> fp16 round-to-nearest-even for the NF4 levels (all normal in fp16
// or zero), evaluated at compile time.
constexpr uint32_t level_to_f16(uint32_t b) {
  const uint32_t sign = (b >> 16) & 0x8000u;
  const uint32_t e = (b >> 23) & 0xffu;
  if (e == 0) return sign;
  const uint32_t m = b & 0x7fffffu;
  uint32_t h = ((e - 127u + 15u) << 10) | (m >> 13);
  const uint32_t rest = m & 0x1fffu;
  if (rest > 0x1000u || (rest == 0x1000u && (h & 1u))) h += 1u;
  return sign | h;
}

// Bytes of a shared-memory level pair table indexed by a code byte: fp16
// pairs in 32 copies (the GEMV's narrow table) or fp32 pairs in 16 copies
// (the tensor-core dequant), either way 8 KB per 256 entries x 32 words.
constexpr int kPairTableBytes = 256 * 32 * 4;

// Device status word values (the library's nf4_status codes).
constexpr int kStatusTimeout = NF4_ERR_DEVICE_TIMEOUT;

// Record a device-side failure without trapping.
// status[0] is the status word, status[1] the site of the first report:
// (kernel << 28) | (role << 24) | (linear CTA index & 0xffffff).
__device__ inline void report_status(int* status, int code, uint32_t kernel, uint32_t role) {
  if (!status) return;
  if (atomicCAS(status, 0, code) == 0) {
    const uint32_t cta = (blockIdx.z * gridDim.y + blockIdx.y) * gridDim.x + blockIdx.x;
    atomicExch(status + 1, static_cast<int>((kernel << 28) | (role << 24) | (cta & 0xffffffu)));
  }
}

// Kernel and role numbers of report_status (see nf4_poll_device_status_site).
constexpr uint32_t kSiteGemv = 1, kSiteTcFwd = 2, kSiteTcDx = 3;
constexpr uint32_t kRoleProducer = 1, kRoleMma = 2, kRoleCompute = 3, kRoleEpilogue = 4;

// x / D rounded to nearest for the constant divisors D = 255 and 127:
// q = RN(x r) with r = RN(1/D) is within one ulp of x / D, the remainder
// x - q D is exact in one FMA, and RN(q + rem r) is then the correctly
// rounded quotient (Markstein's theorem on division by reciprocal and
// remainder correction). For D = 255 and D = 127 this was also checked
// against the exact quotient for every positive fp32 x, subnormals
// included; the sign is symmetric. Three instructions, no division.
template <int D>
__device__ __forceinline__ float div_by_const(float x) {
  constexpr float r = 1.0f / static_cast<float>(D);
  const float q = __fmul_rn(x, r);
  const float rem = __fmaf_rn(-q, static_cast<float>(D), x);
  return __fmaf_rn(rem, r, q);
}

// Second-level dequant: ahat = fl32(fl32(a8 * s2) / 255), both IEEE RN.
__device__ __forceinline__ float dequant_absmax(uint32_t a8, float s2) {
  return div_by_const<255>(__fmul_rn(static_cast<float>(a8), s2));
}

// Element types of activations and outputs (the nf4_elem values of the C ABI).
constexpr int kElemF32 = NF4_F32, kElemBf16 = NF4_BF16, kElemF16 = NF4_F16;

// One fused matmul call, as the launchers take it. The activation operand is
// X [M, K] (forward) or dY [M, N] (input gradient), bf16 or fp16; the output
// Y [M, N] or dX [M, K], fp32 or bf16, overwritten or (accumulate) added to.
struct MatmulCall {
  const void* act;
  bool act_f16;
  int64_t M, N, K;
  int fmt;                 // kFmtNf4, kFmtFp4 or kFmtInt8
  const uint8_t* codes;    // packed 4-bit codes, or int8 values
  const uint8_t* a8;       // 4-bit formats: absmax codes [N*K/64]
  const float* scale;      // 4-bit formats: s2 [groups]; int8: absmax [N*K/64]
  void* out;
  bool out_bf16;
  bool accumulate;
  int num_sms;
  int* status;
  long long wait_limit;    // cycles before the MMA issuer's stage wait gives up
  int device;              // the current device's ordinal
  cudaStream_t st;
};

// Runs f once per device (a kernel's dynamic shared memory limit is an
// attribute of the function on each device); beyond the first 64 ordinals,
// on every call.
constexpr int kOnceDevices = 64;
template <typename F>
void once_per_device(std::once_flag (&flags)[kOnceDevices], int device, F&& f) {
  if (device >= 0 && device < kOnceDevices) std::call_once(flags[device], f);
  else f();
}

}  // namespace nf4

// Kernel launchers (each returns cudaGetLastError() of its launch).
namespace nf4 {
// Encodes a 2-D row-major tensor map [outer, inner] with the given row pitch
// (bytes), box and swizzle; zero fill out of bounds. False on failure.
bool encode_2d(CUtensorMap* map, CUtensorMapDataType dt, const void* base, uint64_t inner,
               uint64_t outer, uint64_t pitch_bytes, uint32_t box_inner, uint32_t box_outer,
               CUtensorMapSwizzle swizzle);

// W is fp32 or (w_bf16) bf16; fmt selects NF4 / FP4 (codes, a8, s2) or
// int8 (codes = int8 values, s2 = fp32 absmax per block, a8 unused).
cudaError_t launch_quantize(const void* W, bool w_bf16, int fmt, int64_t n_elems, uint8_t* codes,
                            uint8_t* a8, float* s2, cudaStream_t st);
// out: n_elems of out_elem (NF4_F32, NF4_BF16 or NF4_F16).
cudaError_t launch_dequantize(int fmt, const uint8_t* codes, const uint8_t* a8, const float* s2,
                              int64_t n_elems, void* out, int out_elem, cudaStream_t st);
cudaError_t launch_gemv_fwd(const MatmulCall& c);
// One launch for `count` (1 .. kGemvGroupMax) weights that share the
// activations, K, the data type, the element types, the flags and the
// stream; each call gives its own weight, N and output.
cudaError_t launch_gemv_group(const MatmulCall* cs, int count);
cudaError_t launch_tc_fwd(const MatmulCall& c);
cudaError_t launch_tc_dx(const MatmulCall& c);
}  // namespace nf4
