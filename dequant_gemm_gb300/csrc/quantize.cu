// Blockwise weight quantization and the stand-alone dequantization:
//  * NF4 and FP4 with 8-bit double-quantized absmax ("Zenbit", zenbit.nf4
//    bullet; "bitsandbytes", NF4, 4-bit and double-quantization paragraphs);
//  * uniform symmetric int8 with an fp32 absmax per 64-weight block
//    ("Zenbit", zenbit.int8 bullet).
// Weights come in as fp32 or bf16 (a bf16 value is exact in fp32, so both
// give the codes of the same fp32 weight).
//
// All kernels are HBM-bound streaming passes: the 4-bit quantize reads 4 (or
// 2) B and writes 0.516 B per weight, int8 writes 1.0625 B; dequantize reads
// the packed weight and writes 4 B per weight.
#include "common.cuh"

namespace nf4 {
namespace {

// Normalisation: the IEEE quotient x = fl32(w / a), computed as one
// Markstein correction of the product with the correctly rounded reciprocal:
// with r = RN(1/a), q0 = RN(w r) is within an ulp of w / a, the remainder
// w - a q0 is exact in one FMA, and RN(q0 + rem r) is the correctly rounded
// quotient (P. Markstein, "Computation of elementary functions on the IBM
// RISC System/6000 processor", IBM J. Res. Dev. 34(1), 1990). The theorem
// needs the intermediate values to stay normal: blocks whose absmax is below
// 2^-64 (and all-zero blocks) take the plain IEEE division instead, and
// |w| <= 1e36 keeps 1/a normal.
__device__ __forceinline__ float markstein_div(float w, float a, float r) {
  const float q0 = __fmul_rn(w, r);
  const float rem = __fmaf_rn(-q0, a, w);
  return __fmaf_rn(rem, r, q0);
}

constexpr float kMinFastAbsmax = 5.421010862427522e-20f;   // 2^-64

// Nearest level through buckets of width 1/16 centred on the multiples of
// 1/16: b = round(16 v + off), read from the low bits of
// fl32(16 v + off + 1.5 * 2^23). No decision threshold lies within 0.004 of a
// bucket edge (an odd multiple of 1/32) and neighbouring thresholds are more
// than 1/16 apart, so a bucket holds at most one threshold and a value
// rounded into the neighbouring bucket at an edge gets the same answer; the
// answer is lo[b] + (v > thr[b]) with lo[b] the number of thresholds below
// the bucket and thr[b] the threshold inside it (2 if none).
//  NF4: v = x in [-1, 1], 33 buckets (off = 16), 15 thresholds, the answer
//       is the code (ties to the lower code: x > t).
//  FP4: v = |x| in [0, 1], 17 buckets (off = 0), 7 magnitude thresholds, the
//       answer is the magnitude; the code adds the sign bit unless the
//       magnitude is 0 (+0 precedes -0, so ties at zero go to code 0).
struct Bucket {
  float thr;
  uint32_t lo;
};

template <int kFmt>
struct Buckets {
  static constexpr int kCount = kFmt == kFmtFp4 ? 17 : 33;
  static constexpr int kThresholds = kFmt == kFmtFp4 ? 7 : 15;
  static constexpr float kOff = kFmt == kFmtFp4 ? 0.0f : 16.0f;
  __device__ static float threshold(int i) {
    return __uint_as_float(kFmt == kFmtFp4 ? fp4_threshold_bits(i) : threshold_bits(i));
  }
};

template <int kFmt>
__device__ __forceinline__ void build_buckets(Bucket* tab) {
  using B = Buckets<kFmt>;
  const int b = threadIdx.x;
  if (b < B::kCount) {
    const float lo_edge = static_cast<float>(2 * b - 1) * 0.03125f - B::kOff * 0.0625f;
    const float hi_edge = lo_edge + 0.0625f;
    uint32_t lo = 0;
    float thr = 2.0f;
#pragma unroll
    for (int i = 0; i < B::kThresholds; ++i) {
      const float t = B::threshold(i);
      lo += (t < lo_edge) ? 1u : 0u;
      if (t > lo_edge && t < hi_edge) thr = t;
    }
    tab[b].thr = thr;
    tab[b].lo = lo;
  }
}

template <int kFmt>
__device__ __forceinline__ uint32_t nearest_code(float x, const Bucket* tab) {
  if constexpr (kFmt == kFmtFp4) {
    const float ax = fabsf(x);
    const uint32_t b = __float_as_uint(__fmaf_rn(ax, 16.0f, 12582912.0f)) & 31u;
    const Bucket e = tab[b];
    const uint32_t mag = e.lo + ((ax > e.thr) ? 1u : 0u);
    return (mag != 0u && x < 0.0f) ? (mag | 8u) : mag;
  } else {
    const uint32_t b = __float_as_uint(__fmaf_rn(x, 16.0f, 12582928.0f)) & 63u;
    const Bucket e = tab[b];
    return e.lo + ((x > e.thr) ? 1u : 0u);
  }
}

// Two bytes of codes for four consecutive weights (little-endian u16):
// element 4j in the high nibble of the first byte.
template <int kFmt>
__device__ __forceinline__ uint32_t pack4(const float* x, const Bucket* tab) {
  return (nearest_code<kFmt>(x[0], tab) << 4) | nearest_code<kFmt>(x[1], tab) |
         (nearest_code<kFmt>(x[2], tab) << 12) | (nearest_code<kFmt>(x[3], tab) << 8);
}

// 16 warps per group, 4 blocks a warp a step, 4 steps: 32 weights a thread.
// (Measured against 8 warps of 8 steps at three CTAs per SM: 4-8% faster on
// single weights, whose last partial wave of CTAs is then shorter; 32 warps
// of 2 steps at one CTA per SM were 20-40% slower.)
constexpr int kQThreads = 512;
constexpr int kQSteps = kGroup / (kQThreads / 32) / 4;

// Each lane of a block's 8 holds 8 of its weights in two runs of 4:
// fp32 input: float4 `sub` and `sub + 8` (elements 4 sub.. and 32 + 4 sub..);
// bf16 input: one 16-byte load of elements 8 sub .. 8 sub + 7.
template <bool kBf16>
struct LaneRuns {
  static __device__ int offset(int sub, int h) { return kBf16 ? 8 * sub + 4 * h : 4 * sub + 32 * h; }
};

template <bool kBf16>
__device__ __forceinline__ void load_lane(const void* W, int64_t blk, int sub, bool ok,
                                          float (&w)[2][4]) {
  if constexpr (kBf16) {
    uint4 r = make_uint4(0u, 0u, 0u, 0u);
    if (ok) r = __ldcs(reinterpret_cast<const uint4*>(W) + blk * 8 + sub);
    const uint32_t u[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      w[i >> 1][2 * (i & 1)] = __uint_as_float(u[i] << 16);
      w[i >> 1][2 * (i & 1) + 1] = __uint_as_float(u[i] & 0xffff0000u);
    }
  } else {
    const float4* src = reinterpret_cast<const float4*>(W) + blk * 16;
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f), b = a;
    if (ok) {
      a = __ldcs(src + sub);
      b = __ldcs(src + sub + 8);
    }
    w[0][0] = a.x; w[0][1] = a.y; w[0][2] = a.z; w[0][3] = a.w;
    w[1][0] = b.x; w[1][1] = b.y; w[1][2] = b.z; w[1][3] = b.w;
  }
}

__device__ __forceinline__ float lane_absmax(const float (&w)[2][4]) {
  float a = 0.0f;
#pragma unroll
  for (int h = 0; h < 2; ++h)
#pragma unroll
    for (int e = 0; e < 4; ++e) a = fmaxf(a, fabsf(w[h][e]));
#pragma unroll
  for (int off = 4; off >= 1; off >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, off));
  return a;
}

// One CTA per double-quant group of 256 blocks (16384 weights). Warp w owns
// blocks [16w, 16w + 16) of the group, 4 blocks per step: 8 lanes per block,
// so a lane's 8 weights share one absmax (3 shuffle steps) and one
// reciprocal. All loads of a lane are issued before any is used.
template <int kFmt, bool kBf16>
__global__ void __launch_bounds__(kQThreads, 2)
quantize_kernel(const void* __restrict__ W, int64_t n_blocks, uint8_t* __restrict__ codes,
                uint8_t* __restrict__ a8_out, float* __restrict__ s2_out) {
  __shared__ float s_absmax[kGroup];
  __shared__ float s_warp_max[kQThreads / 32];
  __shared__ Bucket s_buckets[33];
  build_buckets<kFmt>(s_buckets);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int sub = lane & 7;
  const int64_t blk0 = static_cast<int64_t>(blockIdx.x) * kGroup;
  const int nblk = static_cast<int>(min(static_cast<int64_t>(kGroup), n_blocks - blk0));

  float v[kQSteps][2][4];
#pragma unroll
  for (int j = 0; j < kQSteps; ++j) {
    const int b = warp * (4 * kQSteps) + 4 * j + (lane >> 3);
    load_lane<kBf16>(W, blk0 + b, sub, b < nblk, v[j]);
  }
  __syncthreads();   // bucket table ready

  uint16_t* dst = reinterpret_cast<uint16_t*>(codes + blk0 * (kBlock / 2));
#pragma unroll
  for (int j = 0; j < kQSteps; ++j) {
    const float a = lane_absmax(v[j]);
    const int b = warp * (4 * kQSteps) + 4 * j + (lane >> 3);
    float x[2][4];
    if (a >= kMinFastAbsmax) {   // fast exact quotient
      const float r = __frcp_rn(a);
#pragma unroll
      for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int e = 0; e < 4; ++e) x[h][e] = markstein_div(v[j][h][e], a, r);
    } else {
#pragma unroll
      for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int e = 0; e < 4; ++e) x[h][e] = (a > 0.0f) ? __fdiv_rn(v[j][h][e], a) : 0.0f;
    }
    if (b < nblk) {
      // run h of 4 elements at element offset o -> the u16 at byte o / 2
#pragma unroll
      for (int h = 0; h < 2; ++h)
        dst[b * 16 + LaneRuns<kBf16>::offset(sub, h) / 4] =
            static_cast<uint16_t>(pack4<kFmt>(x[h], s_buckets));
      if (sub == 0) s_absmax[b] = a;
    }
  }
  __syncthreads();

  // Second level: s2 = max absmax of the group, a8 = round(255 * a / s2).
  const int t = threadIdx.x;
  const float a = (t < nblk) ? s_absmax[t] : 0.0f;
  float m = a;
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
  if (lane == 0) s_warp_max[warp] = m;
  __syncthreads();
  float s2 = s_warp_max[0];
#pragma unroll
  for (int w = 1; w < kQThreads / 32; ++w) s2 = fmaxf(s2, s_warp_max[w]);
  if (t < nblk) {
    const uint32_t q =
        (s2 > 0.0f) ? __float2uint_rn(__fdiv_rn(__fmul_rn(255.0f, a), s2)) : 0u;
    a8_out[blk0 + t] = static_cast<uint8_t>(q);
  }
  if (t == 0) s2_out[blockIdx.x] = s2;
}

// Uniform int8: q = rint(fl32(fl32(127 w) / a)) with a the block's fp32
// absmax, kept as the block's scale. Same lane layout as the 4-bit kernel;
// the quotient is the exact IEEE one (Markstein correction of 127 w times
// RN(1/a)), and |q| <= 127 since 127 |w| <= 127 a.
template <bool kBf16>
__global__ void __launch_bounds__(kQThreads, 2)
quantize_int8_kernel(const void* __restrict__ W, int64_t n_blocks, int8_t* __restrict__ q_out,
                     float* __restrict__ absmax_out) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int sub = lane & 7;
  const int64_t blk0 = static_cast<int64_t>(blockIdx.x) * kGroup;
  const int nblk = static_cast<int>(min(static_cast<int64_t>(kGroup), n_blocks - blk0));
  float v[kQSteps][2][4];
#pragma unroll
  for (int j = 0; j < kQSteps; ++j) {
    const int b = warp * (4 * kQSteps) + 4 * j + (lane >> 3);
    load_lane<kBf16>(W, blk0 + b, sub, b < nblk, v[j]);
  }
#pragma unroll
  for (int j = 0; j < kQSteps; ++j) {
    const float a = lane_absmax(v[j]);
    const int b = warp * (4 * kQSteps) + 4 * j + (lane >> 3);
    const bool fast = a >= kMinFastAbsmax;
    const float r = fast ? __frcp_rn(a) : 0.0f;
    if (b < nblk) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t word = 0;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float y = __fmul_rn(127.0f, v[j][h][e]);
          const float t = fast ? markstein_div(y, a, r) : (a > 0.0f ? __fdiv_rn(y, a) : 0.0f);
          const int q = __float2int_rn(t);
          word |= (static_cast<uint32_t>(q) & 0xffu) << (8 * e);
        }
        *reinterpret_cast<uint32_t*>(q_out + (blk0 + b) * kBlock + LaneRuns<kBf16>::offset(sub, h)) =
            word;
      }
      if (sub == 0) absmax_out[blk0 + b] = a;
    }
  }
}

// Output element types of the stand-alone dequantize: fp32, or the fp32
// value rounded to nearest even in bf16 or fp16.
constexpr int kOutF32 = 0, kOutBf16 = 1, kOutF16 = 2;

// Four dequantized weights to out + 4 e (elements), as fp32 or rounded to
// 16 bits; streaming stores (the output is not read back here).
template <int kOut>
__device__ __forceinline__ void store4(void* out, int64_t e, float4 r) {
  if constexpr (kOut == kOutF32) {
    __stcs(reinterpret_cast<float4*>(out) + e, r);
  } else {
    uint2 v;
    if constexpr (kOut == kOutBf16) {
      const __nv_bfloat162 a = __floats2bfloat162_rn(r.x, r.y), b = __floats2bfloat162_rn(r.z, r.w);
      v = make_uint2(*reinterpret_cast<const uint32_t*>(&a), *reinterpret_cast<const uint32_t*>(&b));
    } else {
      const __half2 a = __floats2half2_rn(r.x, r.y), b = __floats2half2_rn(r.z, r.w);
      v = make_uint2(*reinterpret_cast<const uint32_t*>(&a), *reinterpret_cast<const uint32_t*>(&b));
    }
    __stcs(reinterpret_cast<uint2*>(out) + e, v);
  }
}

// Dequantize (4-bit): one thread per 32 weights (16 code bytes, half a block).
template <int kFmt, int kOut>
__global__ void __launch_bounds__(256)
dequantize_kernel(const uint8_t* __restrict__ codes, const uint8_t* __restrict__ a8,
                  const float* __restrict__ s2, int64_t n_chunks, void* __restrict__ out) {
  __shared__ float s_levels[16];
  if (threadIdx.x < 16)
    s_levels[threadIdx.x] = __uint_as_float(kFmt == kFmtFp4 ? kFp4LevelBitsDev[threadIdx.x]
                                                            : kLevelBitsDev[threadIdx.x]);
  __syncthreads();
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= n_chunks) return;
  const int64_t blk = i >> 1;
  const float ahat = dequant_absmax(a8[blk], s2[blk / kGroup]);
  const uint4 c = __ldg(reinterpret_cast<const uint4*>(codes) + i);
  const uint32_t words[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t w = words[j];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint32_t b0 = (w >> (16 * h)) & 0xffu, b1 = (w >> (16 * h + 8)) & 0xffu;
      float4 r;
      r.x = __fmul_rn(s_levels[b0 >> 4], ahat);
      r.y = __fmul_rn(s_levels[b0 & 15], ahat);
      r.z = __fmul_rn(s_levels[b1 >> 4], ahat);
      r.w = __fmul_rn(s_levels[b1 & 15], ahat);
      store4<kOut>(out, i * 8 + 2 * j + h, r);
    }
  }
}

// Dequantize (int8): w = fl32(fl32(q * a) / 127); one thread per 16 weights.
template <int kOut>
__global__ void __launch_bounds__(256)
dequantize_int8_kernel(const int8_t* __restrict__ q, const float* __restrict__ absmax,
                       int64_t n_chunks, void* __restrict__ out) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= n_chunks) return;
  const float a = absmax[i >> 2];
  const uint4 c = __ldg(reinterpret_cast<const uint4*>(q) + i);
  const uint32_t words[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    float r[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int v = static_cast<int8_t>((words[j] >> (8 * e)) & 0xffu);
      r[e] = div_by_const<127>(__fmul_rn(static_cast<float>(v), a));
    }
    store4<kOut>(out, i * 4 + j, make_float4(r[0], r[1], r[2], r[3]));
  }
}

template <int kOut>
void launch_dq(int fmt, const uint8_t* codes, const uint8_t* a8, const float* s2, int64_t n_elems,
               void* out, cudaStream_t st) {
  if (fmt == kFmtInt8) {
    const int64_t n_chunks = n_elems / 16;
    const unsigned grid = static_cast<unsigned>((n_chunks + 255) / 256);
    dequantize_int8_kernel<kOut><<<grid, 256, 0, st>>>(reinterpret_cast<const int8_t*>(codes), s2,
                                                       n_chunks, out);
    return;
  }
  const int64_t n_chunks = n_elems / 32;
  const unsigned grid = static_cast<unsigned>((n_chunks + 255) / 256);
  if (fmt == kFmtFp4)
    dequantize_kernel<kFmtFp4, kOut><<<grid, 256, 0, st>>>(codes, a8, s2, n_chunks, out);
  else
    dequantize_kernel<kFmtNf4, kOut><<<grid, 256, 0, st>>>(codes, a8, s2, n_chunks, out);
}

template <int kFmt, bool kBf16>
void launch_q4(const void* W, int64_t n_blocks, uint8_t* codes, uint8_t* a8, float* s2,
               cudaStream_t st) {
  const int64_t n_groups = (n_blocks + kGroup - 1) / kGroup;
  quantize_kernel<kFmt, kBf16><<<static_cast<unsigned>(n_groups), kQThreads, 0, st>>>(
      W, n_blocks, codes, a8, s2);
}

template <bool kBf16>
void launch_q8(const void* W, int64_t n_blocks, uint8_t* codes, float* absmax, cudaStream_t st) {
  const int64_t n_groups = (n_blocks + kGroup - 1) / kGroup;
  quantize_int8_kernel<kBf16><<<static_cast<unsigned>(n_groups), kQThreads, 0, st>>>(
      W, n_blocks, reinterpret_cast<int8_t*>(codes), absmax);
}

}  // namespace

cudaError_t launch_quantize(const void* W, bool w_bf16, int fmt, int64_t n_elems, uint8_t* codes,
                            uint8_t* a8, float* s2, cudaStream_t st) {
  const int64_t n_blocks = n_elems / kBlock;
  if (fmt == kFmtInt8) {
    if (w_bf16) launch_q8<true>(W, n_blocks, codes, s2, st);
    else launch_q8<false>(W, n_blocks, codes, s2, st);
  } else if (fmt == kFmtFp4) {
    if (w_bf16) launch_q4<kFmtFp4, true>(W, n_blocks, codes, a8, s2, st);
    else launch_q4<kFmtFp4, false>(W, n_blocks, codes, a8, s2, st);
  } else {
    if (w_bf16) launch_q4<kFmtNf4, true>(W, n_blocks, codes, a8, s2, st);
    else launch_q4<kFmtNf4, false>(W, n_blocks, codes, a8, s2, st);
  }
  return cudaGetLastError();
}

cudaError_t launch_dequantize(int fmt, const uint8_t* codes, const uint8_t* a8, const float* s2,
                              int64_t n_elems, void* out, int out_elem, cudaStream_t st) {
  if (out_elem == NF4_BF16) launch_dq<kOutBf16>(fmt, codes, a8, s2, n_elems, out, st);
  else if (out_elem == NF4_F16) launch_dq<kOutF16>(fmt, codes, a8, s2, n_elems, out, st);
  else launch_dq<kOutF32>(fmt, codes, a8, s2, n_elems, out, st);
  return cudaGetLastError();
}

}  // namespace nf4
