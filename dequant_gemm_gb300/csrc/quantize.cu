// NF4 blockwise quantization with 8-bit double-quantized absmax, and the
// stand-alone dequantization ("Zenbit", zenbit.nf4 bullet; "bitsandbytes",
// NF4 and double-quantization paragraphs).
//
// Both kernels are HBM-bound streaming passes: quantize reads 4 B and writes
// 0.516 B per weight, dequantize reads 0.516 B and writes 4 B per weight.
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

// Nearest level of x in [-1, 1], ties to the lower index, through 33 buckets
// of width 1/16 centred on the multiples of 1/16: b = round(16 x + 16), read
// from the low bits of fl32(16 x + 16 + 1.5 * 2^23). No decision threshold lies
// within 0.004 of a bucket edge (an odd multiple of 1/32) and neighbouring
// thresholds are more than 1/16 apart, so a bucket holds at most one
// threshold and an x rounded into the neighbouring bucket at an edge gets the
// same code; the code is lo[b] + (x > thr[b]) with lo[b] the number of
// thresholds below the bucket and thr[b] the threshold inside it (2 if none).
struct Bucket {
  float thr;
  uint32_t lo;
};

__device__ __forceinline__ void build_buckets(Bucket* tab) {
  const int b = threadIdx.x;
  if (b <= 32) {
    const float lo_edge = static_cast<float>(2 * b - 33) * 0.03125f;
    const float hi_edge = lo_edge + 0.0625f;
    uint32_t lo = 0;
    float thr = 2.0f;
#pragma unroll
    for (int i = 0; i < 15; ++i) {
      const float t = __uint_as_float(threshold_bits(i));
      lo += (t < lo_edge) ? 1u : 0u;
      if (t > lo_edge && t < hi_edge) thr = t;
    }
    tab[b].thr = thr;
    tab[b].lo = lo;
  }
}

__device__ __forceinline__ uint32_t nearest_code(float x, const Bucket* tab) {
  const uint32_t b = __float_as_uint(__fmaf_rn(x, 16.0f, 12582928.0f)) & 63u;
  const Bucket e = tab[b];
  return e.lo + ((x > e.thr) ? 1u : 0u);
}

// Two bytes of codes for four consecutive weights (little-endian u16):
// element 4j in the high nibble of the first byte.
__device__ __forceinline__ uint32_t pack4(const float (&x)[4], const Bucket* tab) {
  return (nearest_code(x[0], tab) << 4) | nearest_code(x[1], tab) |
         (nearest_code(x[2], tab) << 12) | (nearest_code(x[3], tab) << 8);
}

__device__ __forceinline__ float abs_max4(float4 v) {
  return fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
}

constexpr int kQThreads = 256;   // one thread per block of the group

// One CTA per double-quant group of 256 blocks (16384 weights). Warp w owns
// blocks [32w, 32w + 32) of the group, 4 blocks per step: 8 lanes per block,
// each holding float4 number `sub` and `sub + 8` of it (128 contiguous bytes
// per block per load), so a lane's 8 weights share one absmax (3 shuffle
// steps) and one reciprocal. All 16 loads of a lane are issued before any is
// used (64 KB in flight per CTA).
__global__ void __launch_bounds__(kQThreads, 3)
quantize_kernel(const float* __restrict__ W, int64_t n_blocks, uint8_t* __restrict__ codes,
                uint8_t* __restrict__ a8_out, float* __restrict__ s2_out) {
  __shared__ float s_absmax[kGroup];
  __shared__ float s_warp_max[kQThreads / 32];
  __shared__ Bucket s_buckets[33];
  build_buckets(s_buckets);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int sub = lane & 7;
  const int64_t blk0 = static_cast<int64_t>(blockIdx.x) * kGroup;
  const int nblk = static_cast<int>(min(static_cast<int64_t>(kGroup), n_blocks - blk0));

  const float4* src = reinterpret_cast<const float4*>(W) + blk0 * (kBlock / 4);
  float4 v[8][2];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int b = warp * 32 + 4 * j + (lane >> 3);
    const bool ok = b < nblk;
    v[j][0] = ok ? __ldcs(src + b * 16 + sub) : make_float4(0.f, 0.f, 0.f, 0.f);
    v[j][1] = ok ? __ldcs(src + b * 16 + sub + 8) : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  __syncthreads();   // bucket table ready

  uint16_t* dst = reinterpret_cast<uint16_t*>(codes + blk0 * (kBlock / 2));
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    float a = fmaxf(abs_max4(v[j][0]), abs_max4(v[j][1]));
#pragma unroll
    for (int off = 4; off >= 1; off >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, off));
    const int b = warp * 32 + 4 * j + (lane >> 3);
    float x[2][4];
    const float w[2][4] = {{v[j][0].x, v[j][0].y, v[j][0].z, v[j][0].w},
                           {v[j][1].x, v[j][1].y, v[j][1].z, v[j][1].w}};
    if (a >= 5.421010862427522e-20f) {   // 2^-64: fast exact quotient
      const float r = __frcp_rn(a);
#pragma unroll
      for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int e = 0; e < 4; ++e) x[h][e] = markstein_div(w[h][e], a, r);
    } else {
#pragma unroll
      for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int e = 0; e < 4; ++e) x[h][e] = (a > 0.0f) ? __fdiv_rn(w[h][e], a) : 0.0f;
    }
    if (b < nblk) {
      // block b's 32 code bytes: float4 `sub` -> bytes 2 sub, 2 sub + 1;
      // float4 `sub + 8` -> bytes 16 + 2 sub, 17 + 2 sub
      dst[b * 16 + sub] = static_cast<uint16_t>(pack4(x[0], s_buckets));
      dst[b * 16 + 8 + sub] = static_cast<uint16_t>(pack4(x[1], s_buckets));
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

// Dequantize: one thread per 32 weights (16 code bytes, half a block).
__global__ void __launch_bounds__(256)
dequantize_kernel(const uint8_t* __restrict__ codes, const uint8_t* __restrict__ a8,
                  const float* __restrict__ s2, int64_t n_chunks, float* __restrict__ out) {
  __shared__ float s_levels[16];
  if (threadIdx.x < 16) s_levels[threadIdx.x] = __uint_as_float(kLevelBitsDev[threadIdx.x]);
  __syncthreads();
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= n_chunks) return;
  const int64_t blk = i >> 1;
  const float ahat = dequant_absmax(a8[blk], s2[blk / kGroup]);
  const uint4 c = __ldg(reinterpret_cast<const uint4*>(codes) + i);
  const uint32_t words[4] = {c.x, c.y, c.z, c.w};
  float4* o = reinterpret_cast<float4*>(out) + i * 8;
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
      __stcs(o + 2 * j + h, r);
    }
  }
}

}  // namespace

cudaError_t launch_quantize(const float* W, int64_t n_elems, uint8_t* codes, uint8_t* a8,
                            float* s2, cudaStream_t st) {
  const int64_t n_blocks = n_elems / kBlock;
  const int64_t n_groups = (n_blocks + kGroup - 1) / kGroup;
  quantize_kernel<<<static_cast<unsigned>(n_groups), kQThreads, 0, st>>>(W, n_blocks, codes, a8,
                                                                         s2);
  return cudaGetLastError();
}

cudaError_t launch_dequantize(const uint8_t* codes, const uint8_t* a8, const float* s2,
                              int64_t n_elems, float* out, cudaStream_t st) {
  const int64_t n_chunks = n_elems / 32;
  const unsigned grid = static_cast<unsigned>((n_chunks + 255) / 256);
  dequantize_kernel<<<grid, 256, 0, st>>>(codes, a8, s2, n_chunks, out);
  return cudaGetLastError();
}

}  // namespace nf4
