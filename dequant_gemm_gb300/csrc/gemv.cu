// Small-M fused dequant matmul: Y = X * dequant(W)^T for M <= 16 tokens
// (decode shapes) ("Zenbit", zenbit.pallas_nf4 bullet: the compressed weight is streamed and
// dequantized on chip; the full-precision weight never reaches HBM).
// Weights are NF4 or FP4 (packed 4-bit codes, double-quantized absmax) or
// int8 ("bitsandbytes", 4-bit paragraph; "Zenbit", zenbit.int8 bullet);
// activations bf16 or fp16; outputs fp32 or bf16, overwritten or added to.
//
// Forward design (HBM-bound: 0.516 B of weight per 2*M flops):
//  * CTA = 16 warps = R row groups of 16 weight rows x 16 / R parts of one
//    K-slice (R = 8: 128 rows, 2 K-parts; R = 2: 32 rows, 8 K-parts), the
//    K-parts taking the slice's code boxes in turn and reducing through
//    shared memory. When the rows alone give too few CTAs, S K-slices of the
//    same rows form a thread-block cluster and reduce through distributed
//    shared memory. Every output is written once with a plain store (no
//    zeroing pass, no atomics). The launcher picks R, S, the n-tiles and the
//    table layout (see launch_gemv_group).
//  * Every warp streams its own codes: lane 0 issues 2-D TMA boxes of 16 rows
//    x 128 bytes (four 64-weight blocks, 128-byte swizzled) into two private
//    shared-memory slots with one mbarrier each, so warps never wait for one
//    another in the main loop, and the copies travel apart from the ordinary
//    loads of the prologue (activations, absmax codes, scales), which thus do
//    not queue behind the weight stream.
//  * The weight is the A operand of mma.sync.m16n8k16 (16 rows per warp), the
//    tokens are the N operand (8 per n-tile, one or two n-tiles): the "swap AB"
//    shape for skinny products. Each weight is dequantized once per CTA for
//    all of its tokens.
//  * Dequantization is factored as  sum_b ahat_b * (sum_{k in b} x_k c[q_k]):
//    the MMA consumes the raw levels c[q] and each 64-weight block's partial
//    sum is scaled by its dequantized absmax in fp32 afterwards. The levels
//    enter the tensor core as fp16 (relative error <= 2^-12), which needs the
//    activations in fp16 too: each token's slice of X is scaled by a power of
//    two that puts its max |x| in [2^14, 2^15) before conversion, and the
//    scale is removed from the fp32 result. The conversion keeps every bit of
//    a bf16 value that lands in fp16's normal range; values below about
//    2^-28 of the slice's max |x| become fp16 subnormals and lose low bits
//    (their share of the sum is below 2^-28 of the largest term).
//  * One packed byte (two adjacent weights) becomes one f16x2 fragment
//    register through a 256-entry table held in 32 copies, one per lane, so
//    that every lookup of a warp hits 32 distinct banks. Each CTA lays the
//    copies out itself, by shuffles from levels held in registers. Where the
//    shared memory allows (4-bit codes; the launcher decides) the table rows
//    are 256 bytes apart, so that a single byte permute of the code word and
//    the lane number gives the address of a lookup (a permute and a load per
//    two weights); that CTA takes an SM of its own and may use up to 128
//    registers a thread. Int8
//    weights need no table: two bytes become an f16x2 of 1024 + (q + 128)
//    by one byte permute with the fp16 exponent of 1024, less 1152, which is
//    q exactly; the block scale absmax / 127 is applied after the MMA like
//    the 4-bit one.
//  * Within a block the 4 threads of an MMA quad each own 16 contiguous k
//    (8 code bytes); the reduction order over k is permuted consistently in A
//    and B, which leaves the sum unchanged.
//  * The activation slice is staged by all 16 warps at once (one global round
//    trip), then scaled to fp16 in place after a block-wide max.
//  * Launched with programmatic stream serialization: the CTAs of the next
//    kernel in the stream can be resident and do their set-up while this one
//    drains. Before griddepcontrol.wait a CTA only prefetches its code boxes
//    and absmax codes into L2; every read comes after it.
#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "tc.cuh"

namespace nf4 {
namespace {

constexpr int kGemvWarps = 16;                  // row groups x K-parts
constexpr int kMaxRowGroups = 8;                // of 16 rows each
constexpr int kGemvRows = 16 * kMaxRowGroups;   // most weight rows per CTA
constexpr int kGemvThreads = 32 * kGemvWarps;
constexpr int kBoxBytes = 16 * 128;             // 16 rows x 128 bytes
constexpr int kWarpSlots = 2;                   // code boxes in flight per warp
constexpr int kTabBytes = kPairTableBytes;
constexpr int kMaxSliceBlocks = 96;
constexpr int kMaxCluster = 8;
static_assert(kMaxCluster * kMaxSliceBlocks * kBlock == kGemvMaxCols, "K limit");

// fp16 bits of level i (0 <= i < 16) of a 4-bit format as a select tree
// over immediates: no memory access, so the table set-up does not wait on a
// constant-cache miss.
template <int kFmt, int kLo, int kN>
__device__ __forceinline__ uint32_t level_f16(int i) {
  if constexpr (kN == 1) {
    return level_to_f16(kFmt == kFmtFp4 ? kFp4LevelBits[kLo] : kLevelBits[kLo]);
  } else {
    const uint32_t lo = level_f16<kFmt, kLo, kN / 2>(i);
    const uint32_t hi = level_f16<kFmt, kLo + kN / 2, kN / 2>(i);
    return (i & (kN / 2)) ? hi : lo;
  }
}

// Two int8 weights (bytes `sel` of w, sel = 0x4140 for bytes 0-1, 0x4342 for
// bytes 2-3) as an exact f16x2: the biased bytes q + 128 become the low
// mantissa bits of fp16 1024 (0x6400), giving 1024 + q + 128, and
// subtracting 1152 leaves q.
__device__ __forceinline__ uint32_t int8_pair_f16(uint32_t w_biased, uint32_t sel) {
  const uint32_t h = __byte_perm(w_biased, 0x64646464u, sel);
  const __half2 v = __hsub2(*reinterpret_cast<const __half2*>(&h),
                            __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480)));
  return *reinterpret_cast<const uint32_t*>(&v);
}

// Not volatile: independent MMA chains of different blocks may interleave.
__device__ __forceinline__ void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                        uint32_t a3, uint32_t b0, uint32_t b1) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Prefetch a tile of a tensor map into L2 (no shared memory, no barrier).
__device__ __forceinline__ void tma_prefetch_2d(const CUtensorMap* map, int32_t x, int32_t y) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y)
               : "memory");
}

__device__ __forceinline__ void prefetch_l2(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(reinterpret_cast<uint64_t>(p)) : "memory");
}

// Store a float into CTA `rank`'s shared memory at this CTA's address of
// `local` (made visible to that CTA by the next cluster barrier).
__device__ __forceinline__ void st_dsmem(float* local, uint32_t rank, float v) {
  const uint32_t remote = tc::mapa(tc::smem_addr(local), rank);
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(remote), "f"(v) : "memory");
}

// Up to kGemvGroupMax weights that share the activations (and K and the
// data type) run in one launch: the row tiles of weight i are blocks
// [tile0[i], tile0[i + 1]) of the grid's x dimension.
struct GemvMaps {
  CUtensorMap m[kGemvGroupMax];   // the codes of each weight
};
struct GemvArgs {
  const uint16_t* X;                   // bf16 or fp16 [M, K]
  const uint8_t* a8[kGemvGroupMax];    // 4-bit formats: [N*K/64]
  const float* scale[kGemvGroupMax];   // 4-bit formats: s2 [groups]; int8: absmax [N*K/64]
  void* Y[kGemvGroupMax];              // fp32 or bf16 [M, N]
  int64_t N[kGemvGroupMax];
  int tile0[kGemvGroupMax + 1];
  int count;
  int64_t M, K;
  int nblk;              // K / 64
  int slices;            // K-slices = cluster size along y
  int max_nb;            // largest slice, in blocks
  int out_bf16;
  int accumulate;
  int* status;
};

// One output element: Y[i] = v (+ Y[i] with accumulate), fp32 or bf16 (RN).
__device__ __forceinline__ void store_out(void* Y, int64_t i, float v, int out_bf16,
                                          int accumulate) {
  if (out_bf16) {
    __nv_bfloat16* y = reinterpret_cast<__nv_bfloat16*>(Y) + i;
    if (accumulate) v += __bfloat162float(*y);
    *y = __float2bfloat16_rn(v);
  } else {
    float* y = reinterpret_cast<float*>(Y) + i;
    if (accumulate) v += *y;
    *y = v;
  }
}

// Four consecutive outputs starting at i (a multiple of 4).
__device__ __forceinline__ void store_out4(void* Y, int64_t i, float4 v, int out_bf16,
                                           int accumulate) {
  if (out_bf16) {
    uint2* y = reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(Y) + i);
    if (accumulate) {
      const uint2 o = *y;
      const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&o.x));
      const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&o.y));
      v.x += a.x; v.y += a.y; v.z += b.x; v.w += b.y;
    }
    const __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y), hi = __floats2bfloat162_rn(v.z, v.w);
    *y = make_uint2(*reinterpret_cast<const uint32_t*>(&lo), *reinterpret_cast<const uint32_t*>(&hi));
  } else {
    float4* y = reinterpret_cast<float4*>(reinterpret_cast<float*>(Y) + i);
    if (accumulate) {
      const float4 o = *y;
      v.x += o.x; v.y += o.y; v.z += o.z; v.w += o.w;
    }
    *y = v;
  }
}

// First absmax block of K-slice s (nblk * slices stays far below 2^31).
__host__ __device__ constexpr int slice_begin(int nblk, int slices, int s) {
  return (nblk * s) / slices;
}

// Shared memory. The level table comes in two layouts. Narrow (where the
// wide one does not fit, or int8 without a table): rows of 128 bytes, one
// 4-byte copy per lane, at the start of the 1024-byte aligned region. Wide
// (4-bit formats, when the launcher finds room): rows of 256 bytes
// at the very start of the dynamic window, before the aligned region, so
// that the address of a lookup, (code byte) * 256 + lane * 4, is what one
// byte permute returns and the window offset folds into the load; the upper
// 128 bytes of each row stay unused. Then, from the aligned base: code slots
// (per warp, 1024-byte aligned for the swizzle; after the main loop a
// warp of K-part 1 and up hands its sums to K-part 0 through its first slot),
// mbarriers, token scales, per-warp max |x|, the cluster reduction inbox and
// the fp16 activation slice (rows of max_nb * 128 + 8 bytes: the 8 keeps the
// B fragment loads of 8 token rows on distinct banks).
constexpr int kWideTabBytes = 256 * 256;
__host__ __device__ constexpr int gemv_lead(bool wide) { return wide ? kWideTabBytes : 0; }
__host__ __device__ constexpr int gemv_off_slots(bool wide) { return wide ? 0 : kTabBytes; }
__host__ __device__ constexpr int gemv_off_bars(bool wide) {
  return gemv_off_slots(wide) + kGemvWarps * kWarpSlots * kBoxBytes;
}
__host__ __device__ constexpr int gemv_off_xinv(bool wide) { return gemv_off_bars(wide) + kGemvWarps * kWarpSlots * 8; }
__host__ __device__ constexpr int gemv_off_wmax(bool wide) { return gemv_off_xinv(wide) + 16 * 4; }
__host__ __device__ constexpr int gemv_off_inbox(bool wide) { return gemv_off_wmax(wide) + kGemvWarps * 4; }
__host__ __device__ constexpr int gemv_off_xs(int nt, bool wide) {
  return gemv_off_inbox(wide) + 8 * nt * kGemvRows * 4;
}
__host__ __device__ constexpr int gemv_xstride(int max_nb) { return max_nb * 128 + 8; }
// The wide table serves one n-tile of a 4-bit format.
__host__ __device__ constexpr bool gemv_wide(int nt, int fmt) { return nt <= 2 && fmt != kFmtInt8; }

// Per-format constants of the small-M forward: 64-weight blocks per 128-byte
// code box row (four of 32 bytes, or two of 64 for int8).
template <int kFmt>
struct GemvFmt {
  static constexpr bool kInt8 = kFmt == kFmtInt8;
  static constexpr int kBoxBlocks = kInt8 ? 2 : 4;
  static constexpr int kBlockBytes = kInt8 ? 64 : 32;   // code bytes of one block row
};

template <int NT, int kFmt, bool kF16, bool kWide, int kR>
__global__ void __launch_bounds__(kGemvThreads, kWide ? 1 : 2)
gemv_fwd_kernel(const __grid_constant__ GemvMaps maps, const __grid_constant__ GemvArgs p) {
  constexpr bool kInt8 = GemvFmt<kFmt>::kInt8;
  constexpr int kBoxBlocks = GemvFmt<kFmt>::kBoxBlocks;
  constexpr int kBlockBytes = GemvFmt<kFmt>::kBlockBytes;
  static_assert(!kWide || gemv_wide(NT, kFmt), "the wide table serves the 4-bit formats");
  extern __shared__ __align__(16) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw + gemv_lead(kWide)) + 1023) & ~static_cast<uintptr_t>(1023));
  uint32_t* tab = reinterpret_cast<uint32_t*>(kWide ? smem_raw : smem);
  float* xinv = reinterpret_cast<float*>(smem + gemv_off_xinv(kWide));    // [16]
  float* wmax = reinterpret_cast<float*>(smem + gemv_off_wmax(kWide));    // [kGemvWarps]
  float* inbox = reinterpret_cast<float*>(smem + gemv_off_inbox(kWide));
  uint8_t* xs = smem + gemv_off_xs(NT, kWide);
  const int xstride = gemv_xstride(p.max_nb);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, t = lane & 3;
  // warp = row group rgp of kR (16 rows each) x K-part kp of kP = 16 / kR
  constexpr int kP = kGemvWarps / kR, kRowsCta = 16 * kR;
  const int rgp = warp % kR, kp = warp / kR;
  // K-part hand-off: warp w's partial sums go through its own first code
  // slot, free once it has consumed its last box
  auto red_of = [&](int w) {
    return reinterpret_cast<float*>(smem + gemv_off_slots(kWide) + w * kWarpSlots * kBoxBytes);
  };
  // this CTA's weight of the group (selects on static indices, so the
  // parameter arrays stay in parameter space)
  int gi = 0;
#pragma unroll
  for (int q = 1; q < kGemvGroupMax; ++q)
    gi += (q < p.count && static_cast<int>(blockIdx.x) >= p.tile0[q]) ? 1 : 0;
  auto pick = [&](auto const (&arr)[kGemvGroupMax]) {
    auto v = arr[0];
#pragma unroll
    for (int q = 1; q < kGemvGroupMax; ++q)
      if (gi == q) v = arr[q];
    return v;
  };
  const int64_t N = pick(p.N);
  const uint8_t* const a8 = pick(p.a8);
  const float* const scale = pick(p.scale);
  void* const Y = pick(p.Y);
  const CUtensorMap* const tm_codes = &maps.m[gi];
  int tile_first = p.tile0[0];
#pragma unroll
  for (int q = 1; q < kGemvGroupMax; ++q)
    if (gi == q) tile_first = p.tile0[q];
  const int64_t row0 = static_cast<int64_t>(static_cast<int>(blockIdx.x) - tile_first) * kRowsCta;
  const int slice = blockIdx.y;
  const int kb0 = slice_begin(p.nblk, p.slices, slice);
  const int nb = slice_begin(p.nblk, p.slices, slice + 1) - kb0;
  const int nboxes = (nb + kBoxBlocks - 1) / kBoxBlocks;
  const int64_t m0 = static_cast<int64_t>(blockIdx.z) * 8 * NT;
  const int mt = static_cast<int>(min(static_cast<int64_t>(8 * NT), p.M - m0));
  // this warp's code slots and their mbarriers; it takes boxes kp, kp + kP, ...
  const uint32_t slots = tc::smem_addr(smem + gemv_off_slots(kWide)) + warp * kWarpSlots * kBoxBytes;
  const uint32_t bars = tc::smem_addr(smem + gemv_off_bars(kWide)) + warp * kWarpSlots * 8;

  // Programmatic dependent launch: the next kernel in the stream may start its
  // own set-up now; this one reads no global memory before the previous
  // kernel has completed (griddepcontrol.wait), beyond L2 prefetches.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // Warm L2 with this warp's code boxes and its rows' absmax codes while the
  // previous kernel drains. A prefetch returns nothing to the thread and L2 is
  // the point of coherence, so the loads after griddepcontrol.wait still see
  // everything the previous kernel wrote.
  {
    // Only for short slices (at most the boxes a warp keeps in flight),
    // where the launch is latency-bound: on long slices the prefetch competes
    // with demand loads and was measured slower (35 MB weights, 4% slower
    // even with the first four boxes only).
    const int nmine_pf = (nboxes - kp + kP - 1) / kP;
    if (lane == 0 && nmine_pf <= kWarpSlots && row0 + rgp * 16 < N)   // boxes inside the weight
      for (int i = 0; i < nmine_pf; ++i)
        tma_prefetch_2d(tm_codes, (kb0 + kBoxBlocks * (kp + kP * i)) * kBlockBytes,
                            static_cast<int32_t>(row0 + rgp * 16));
    const int64_t pr = row0 + rgp * 16 + lane;
    if (kp == 0 && lane < 16 && pr < N && nb > 0 && nmine_pf <= kWarpSlots) {
      const int64_t ia = pr * p.nblk + kb0;
      if constexpr (kInt8) {
        prefetch_l2(scale + ia);
        prefetch_l2(scale + ia + nb - 1);
      } else {
        prefetch_l2(a8 + ia);
        prefetch_l2(a8 + ia + nb - 1);
        prefetch_l2(scale + (ia >> 8));
      }
    }
  }
  // level table: entry e, copy l at word (32 or 64) e + l (one
  // conflict-free store per entry and warp); lane l holds level l & 15,
  // entries come by shuffles
  if constexpr (!kInt8) {
    const uint32_t lev = level_f16<kFmt, 0, 16>(lane & 15);
    for (int e = warp; e < 256; e += kGemvWarps) {
      const uint32_t hi = __shfl_sync(0xffffffffu, lev, e >> 4);
      const uint32_t lo = __shfl_sync(0xffffffffu, lev, e & 15);
      tab[e * (kWide ? 64 : 32) + lane] = hi | (lo << 16);
    }
  }
  if (lane == 0) {
    for (int s = 0; s < kWarpSlots; ++s) tc::mbar_init(bars + 8u * s, 1);
    tc::fence_barrier_init();
    tc::prefetch_tensormap(tm_codes);
  }
  __syncwarp();
  // First half of a split cluster barrier: the CTAs of a cluster store into
  // one another's shared memory at the end, which is only allowed once every
  // CTA of the cluster has started; the matching wait sits just before those
  // stores, so the barrier costs nothing on the way.
  if (p.slices > 1) asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");

  // Activations first, ahead of the code stream: every warp takes part.
  // Token xm = warp % mt of the tile is copied, as bf16, into its staging row
  // by the xparts = 16 / mt warps with that token, interleaved by 32 lanes,
  // each taking its max |x| on the way (one global round trip for short
  // slices); the conversion to fp16 happens in place below.
  auto to_f2 = [](uint32_t w) {
    if constexpr (kF16) return __half22float2(*reinterpret_cast<const __half2*>(&w));
    else return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w));
  };
  auto amax4 = [&](uint2 v) {
    const float2 f0 = to_f2(v.x), f1 = to_f2(v.y);
    return fmaxf(fmaxf(fabsf(f0.x), fabsf(f0.y)), fmaxf(fabsf(f1.x), fabsf(f1.y)));
  };
  const int nkv4 = nb * (kBlock / 4);      // uint2 (4 bf16) per token row
  const int xparts = kGemvWarps / mt, xm = warp % mt, xp = warp / mt;
  const bool xw = xp < xparts;             // warps past xparts * mt stage nothing
  uint2* xo = reinterpret_cast<uint2*>(xs + xm * xstride);
  float xmax = 0.0f;
  if (xw) {
    const uint2* xrow = reinterpret_cast<const uint2*>(p.X + (m0 + xm) * p.K +
                                                       static_cast<int64_t>(kb0) * kBlock);
#pragma unroll 4
    for (int i = xp * 32 + lane; i < nkv4; i += xparts * 32) {
      const uint2 v = __ldg(xrow + i);
      xo[i] = v;
      xmax = fmaxf(xmax, amax4(v));
    }
  }

  // Box i of this warp (the slice's box kp + kP i) goes into slot i % kWarpSlots, by
  // TMA; its absmax codes and scales travel alongside: lane e loads those of
  // row pair (e & 7, (e & 7) + 8) of block e >> 3 of the box.
  const int nmine = (nboxes - kp + kP - 1) / kP;   // boxes of this warp
  const int64_t ar = row0 + rgp * 16 + (lane & 7);
  const bool ar_ok = ar < N, br_ok = ar + 8 < N;
  auto issue_box = [&](int i) {
    if (lane == 0) {
      const int b = kp + kP * i;
      const uint32_t bar = bars + 8u * (i % kWarpSlots);
      tc::mbar_arrive_expect_tx(bar, kBoxBytes);
      tc::tma_load_2d(slots + (i % kWarpSlots) * kBoxBytes, tm_codes,
                      (kb0 + kBoxBlocks * b) * kBlockBytes, static_cast<int32_t>(row0 + rgp * 16),
                      bar);
    }
  };
  // 4-bit: absmax codes qa, qb and scales sa, sb; int8: the block absmax in
  // sa, sb (qa, qb unused)
  auto load_scales = [&](int i, uint32_t& qa, uint32_t& qb, float& sa, float& sb) {
    const int j = (kp + kP * i) * kBoxBlocks + (lane >> 3);
    const bool in = i < nmine && j < nb && (lane >> 3) < kBoxBlocks;
    const int64_t ia = ar * p.nblk + kb0 + j, ib = ia + 8 * p.nblk;
    if constexpr (kInt8) {
      qa = qb = 0u;
      sa = (in && ar_ok) ? __ldg(scale + ia) : 0.0f;
      sb = (in && br_ok) ? __ldg(scale + ib) : 0.0f;
    } else {
      qa = (in && ar_ok) ? static_cast<uint32_t>(__ldg(a8 + ia)) : 0u;
      qb = (in && br_ok) ? static_cast<uint32_t>(__ldg(a8 + ib)) : 0u;
      sa = (in && ar_ok) ? __ldg(scale + (ia >> 8)) : 0.0f;
      sb = (in && br_ok) ? __ldg(scale + (ib >> 8)) : 0.0f;
    }
  };
  uint32_t qa0, qb0, qa1, qb1;
  float sa0, sb0, sa1, sb1;
  load_scales(0, qa0, qb0, sa0, sb0);
  load_scales(1, qa1, qb1, sa1, sb1);
  for (int i = 0; i < kWarpSlots && i < nmine; ++i) issue_box(i);

  // max |x| over the slice -> power-of-two scale into [2^14, 2^15) -> fp16
  // (bit-preserving down to fp16's normal range, see the file comment)
  if (xw) {
    float mx = xmax;
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    if (lane == 0) wmax[warp] = mx;
  }
  __syncthreads();
  if (xw) {
    float mx = 0.0f;
    for (int q = 0; q < xparts; ++q) mx = fmaxf(mx, wmax[xm + q * mt]);
    int e = 0;
    if (mx > 0.0f) {
      const int E = max(1, static_cast<int>((__float_as_uint(mx) >> 23) & 0xffu));
      e = min(141 - E, 126);
    }
    const float scale = __uint_as_float(static_cast<uint32_t>(e + 127) << 23);
    if (xp == 0 && lane == 0) xinv[xm] = __uint_as_float(static_cast<uint32_t>(127 - e) << 23);
    auto convert = [&](uint2 v) {
      const float2 f0 = to_f2(v.x), f1 = to_f2(v.y);
      const __half2 h0 = __floats2half2_rn(f0.x * scale, f0.y * scale);
      const __half2 h1 = __floats2half2_rn(f1.x * scale, f1.y * scale);
      return make_uint2(*reinterpret_cast<const uint32_t*>(&h0),
                        *reinterpret_cast<const uint32_t*>(&h1));
    };
    for (int i = xp * 32 + lane; i < nkv4; i += xparts * 32) xo[i] = convert(xo[i]);   // own entries
  }
  __syncthreads();

  // Main loop: per block, 16 lookups and 4 MMA k-steps per n-tile, then the
  // block's partial sums scaled by the rows' dequantized absmax.
  float acc[NT][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[nt][i] = 0.0f;
  const uint8_t* tabl = smem + lane * 4;                 // this lane's narrow table copy
  const uint32_t lane_sel = static_cast<uint32_t>(lane) * 4u;   // byte 0: lane * 4, rest 0
  const uint8_t* xsl = xs + g * xstride + t * 32;        // token g, this lane's 16 k
  bool tok_ok[NT];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) tok_ok[nt] = nt * 8 + g < mt;
  auto lut = [&](uint32_t w, int b) {
    if constexpr (kWide) {
      // bytes (lane * 4, code byte b, 0, 0): the entry's offset in the window
      const uint32_t off = __byte_perm(w, lane_sel, 0x7604u + (static_cast<uint32_t>(b) << 4));
      return *reinterpret_cast<const uint32_t*>(smem_raw + off);
    } else {
      return *reinterpret_cast<const uint32_t*>(tabl + (__byte_perm(w, 0u, 0x4440u + b) << 7));
    }
  };
  // rows g and g + 8 of the box; 16-byte chunk c of row r sits at c ^ (r & 7)
  const uint8_t* slot_g = smem + gemv_off_slots(kWide) + warp * kWarpSlots * kBoxBytes + g * 128 +
                          (kInt8 ? 0 : (t & 1) * 8);
  bool ok = true;
  int waited = 0;
  // one box: lane e's row-pair scales (block e >> 3, rows (e & 7, + 8)),
  // then its four blocks, each taking its scales from lane 8 jj + g
  auto do_box = [&](int i, uint32_t qa, uint32_t qb, float sa, float sb) {
    const int sl = i % kWarpSlots;
    float aha, ahb;
    if constexpr (kInt8) {   // scale of the raw integer sums
      aha = div_by_const<127>(sa);
      ahb = div_by_const<127>(sb);
    } else {
      aha = dequant_absmax(qa, sa);
      ahb = dequant_absmax(qb, sb);
    }
    // warp-uniform outcome: the lanes leave together or go on together
    const bool got = tc::mbar_wait(bars + 8u * sl, (i / kWarpSlots) & 1);
    if (!__all_sync(0xffffffffu, got)) return false;
    const int b = kp + kP * i;
    const uint8_t* sg = slot_g + sl * kBoxBytes;
#pragma unroll
    for (int jj = 0; jj < kBoxBlocks; ++jj) {
      const int j = b * kBoxBlocks + jj;
      if (j < nb) {
        // this thread's 16 weights of the block in rows g and g + 8
        uint32_t ra[4], rb[4];
        if constexpr (kInt8) {
          const int chunk = ((4 * jj + t) ^ g) << 4;
          const uint4 wa = *reinterpret_cast<const uint4*>(sg + chunk);
          const uint4 wb = *reinterpret_cast<const uint4*>(sg + 8 * 128 + chunk);
          ra[0] = wa.x ^ 0x80808080u; ra[1] = wa.y ^ 0x80808080u;
          ra[2] = wa.z ^ 0x80808080u; ra[3] = wa.w ^ 0x80808080u;
          rb[0] = wb.x ^ 0x80808080u; rb[1] = wb.y ^ 0x80808080u;
          rb[2] = wb.z ^ 0x80808080u; rb[3] = wb.w ^ 0x80808080u;
        } else {
          const int chunk = ((2 * jj + (t >> 1)) ^ g) << 4;
          const uint2 wa = *reinterpret_cast<const uint2*>(sg + chunk);
          const uint2 wb = *reinterpret_cast<const uint2*>(sg + 8 * 128 + chunk);
          ra[0] = wa.x; ra[1] = wa.y; rb[0] = wb.x; rb[1] = wb.y;
          ra[2] = ra[3] = rb[2] = rb[3] = 0u;
        }
        float part[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int q = 0; q < 4; ++q) part[nt][q] = 0.0f;
#pragma unroll
        for (int s = 0; s < 4; ++s) {
          // step s covers weights 4s .. 4s + 3 of the thread's 16: logical k
          // (2t, 2t+1) then (2t+8, 2t+9) of the MMA fragment
          uint32_t a0, a1, a2, a3;
          if constexpr (kInt8) {
            a0 = int8_pair_f16(ra[s], 0x4140u);
            a2 = int8_pair_f16(ra[s], 0x4342u);
            a1 = int8_pair_f16(rb[s], 0x4140u);
            a3 = int8_pair_f16(rb[s], 0x4342u);
          } else {
            const uint32_t xa = s < 2 ? ra[0] : ra[1], xb = s < 2 ? rb[0] : rb[1];
            const int bs = 2 * (s & 1);
            a0 = lut(xa, bs);
            a2 = lut(xa, bs + 1);
            a1 = lut(xb, bs);
            a3 = lut(xb, bs + 1);
          }
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            uint2 bx = make_uint2(0u, 0u);
            if (tok_ok[nt])
              bx = *reinterpret_cast<const uint2*>(xsl + nt * 8 * xstride + j * 128 + 8 * s);
            mma_f16(part[nt], a0, a1, a2, a3, bx.x, bx.y);
          }
        }
        const float2 ah = make_float2(__shfl_sync(0xffffffffu, aha, jj * 8 + g),
                                      __shfl_sync(0xffffffffu, ahb, jj * 8 + g));
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          acc[nt][0] = fmaf(ah.x, part[nt][0], acc[nt][0]);
          acc[nt][1] = fmaf(ah.x, part[nt][1], acc[nt][1]);
          acc[nt][2] = fmaf(ah.y, part[nt][2], acc[nt][2]);
          acc[nt][3] = fmaf(ah.y, part[nt][3], acc[nt][3]);
        }
      }
    }
    // every lane is done with the slot: refill it with this warp's box i + 2
    __syncwarp();
    if (i + kWarpSlots < nmine) {
      if (lane == 0) asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      issue_box(i + kWarpSlots);
    }
    return true;
  };
  for (int i = 0; i < nmine && ok; i += 2) {
    // the registers of box i (slot 0) are refilled for box i + 2 right after use
    uint32_t qa = qa0, qb = qb0;
    float sa = sa0, sb = sb0;
    load_scales(i + 2, qa0, qb0, sa0, sb0);
    if (!do_box(i, qa, qb, sa, sb)) { ok = false; break; }
    waited = i + 1;
    if (i + 1 < nmine) {
      qa = qa1; qb = qb1; sa = sa1; sb = sb1;
      load_scales(i + 3, qa1, qb1, sa1, sb1);
      if (!do_box(i + 1, qa, qb, sa, sb)) { ok = false; break; }
      waited = i + 2;
    }
  }
  if (!ok) {
    report_status(p.status, kStatusTimeout, kSiteGemv, kRoleCompute);
    // copies still in flight land before the CTA may exit
    if (lane == 0)
      for (int i = waited; i < min(nmine, waited + kWarpSlots); ++i)
        tc::mbar_wait(bars + 8u * (i % kWarpSlots), (i / kWarpSlots) & 1);
  }

  // K-parts 1 .. kP-1 of each row group hand their sums to K-part 0.
  if (kp > 0) {
    float* red = red_of(warp);
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
      *reinterpret_cast<float4*>(red + (lane * NT + nt) * 4) =
          make_float4(acc[nt][0], acc[nt][1], acc[nt][2], acc[nt][3]);
  }
  __syncthreads();
  // Undo the token scales; K-part 0 holds the row group's sums.
  float inv0[NT], inv1[NT];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int tk0 = nt * 8 + 2 * t;
    inv0[nt] = tk0 < mt ? xinv[tk0] : 0.0f;
    inv1[nt] = tk0 + 1 < mt ? xinv[tk0 + 1] : 0.0f;
  }
  if (kp == 0) {
#pragma unroll
    for (int q = 1; q < kP; ++q) {
      const float* red = red_of(rgp + kR * q);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const float4 o = *reinterpret_cast<const float4*>(red + (lane * NT + nt) * 4);
        acc[nt][0] += o.x;
        acc[nt][1] += o.y;
        acc[nt][2] += o.z;
        acc[nt][3] += o.w;
      }
    }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      acc[nt][0] *= inv0[nt];
      acc[nt][1] *= inv1[nt];
      acc[nt][2] *= inv0[nt];
      acc[nt][3] *= inv1[nt];
    }
  }
  if (p.slices == 1) {
    // stage [8 NT tokens x 16 kR rows] over the level table, then float4 stores
    float* out_s = reinterpret_cast<float*>(tab);
    constexpr int kOutStride = kRowsCta + 4;   // floats, keeps rows 16-byte aligned
    if (kp == 0) {
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const int tk0 = nt * 8 + 2 * t, tk1 = tk0 + 1;
        const int rg = rgp * 16 + g;
        out_s[tk0 * kOutStride + rg] = acc[nt][0];
        out_s[tk1 * kOutStride + rg] = acc[nt][1];
        out_s[tk0 * kOutStride + rg + 8] = acc[nt][2];
        out_s[tk1 * kOutStride + rg + 8] = acc[nt][3];
      }
    }
    __syncthreads();
    for (int i = tid; i < 8 * NT * (kRowsCta / 4); i += kGemvThreads) {
      const int tk = i / (kRowsCta / 4), r4 = (i % (kRowsCta / 4)) * 4;
      if (tk < mt && row0 + r4 < N)
        store_out4(Y, (m0 + tk) * N + row0 + r4,
                   *reinterpret_cast<const float4*>(out_s + tk * kOutStride + r4), p.out_bf16,
                   p.accumulate);
    }
  } else {
    // Cluster reduction, push form: CTA `rank` owns rows [rank*rpc, (rank+1)*rpc)
    // of the row tile. Every CTA stores its partial of those rows into the
    // owner's inbox slot for its slice, one cluster barrier makes the stores
    // visible, and each owner sums its slots and writes Y once.
    const int rpc = kRowsCta / p.slices;           // rows owned per CTA (a power of two)
    const int rpc_shift = 31 - __clz(rpc);
    asm volatile("barrier.cluster.wait.aligned;" ::: "memory");   // every peer has started
    if (kp == 0) {
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const int tk0 = nt * 8 + 2 * t;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int tk = tk0 + (e & 1);
          const int rg = rgp * 16 + g + 8 * (e >> 1);
          const uint32_t owner = static_cast<uint32_t>(rg >> rpc_shift);
          st_dsmem(inbox + ((slice * 8 * NT + tk) << rpc_shift) + (rg & (rpc - 1)), owner,
                   acc[nt][e]);
        }
      }
    }
    tc::cluster_sync();
    const int rank = static_cast<int>(tc::cluster_ctarank());
    for (int i = tid; i < 8 * NT * rpc; i += kGemvThreads) {
      const int tk = i >> rpc_shift, rl = i & (rpc - 1), r = rank * rpc + rl;
      if (tk < mt && row0 + r < N) {
        float v = 0.0f;
        for (int c = 0; c < p.slices; ++c) v += inbox[((c * 8 * NT + tk) << rpc_shift) + rl];
        store_out(Y, (m0 + tk) * N + row0 + r, v, p.out_bf16, p.accumulate);
      }
    }
  }
}

}  // namespace

// Dynamic shared memory of one GEMV CTA (plus 1 KB to align the base).
constexpr size_t gemv_smem_bytes(int nt, int max_nb, int xrows, bool wide) {
  return static_cast<size_t>(gemv_lead(wide)) + static_cast<size_t>(gemv_off_xs(nt, wide)) +
         static_cast<size_t>(xrows) * gemv_xstride(max_nb) + 1024;
}
constexpr size_t kGemvSmemTwoPerSm = 112 * 1024;   // two CTAs per SM
constexpr size_t kGemvSmemLimit = 220 * 1024;

// The longest slices (96 blocks) of 8 tokens always fit one narrow n-tile:
// the small-M kernel has a launch shape for every K up to kGemvMaxCols.
static_assert(gemv_smem_bytes(1, kMaxSliceBlocks, 8, false) <= kGemvSmemLimit, "K limit shape");

// Row groups per CTA the kernel is built for: 8 (128 rows, 2 K-parts) or 2
// (32 rows, 8 K-parts).
template <int NT, int kFmt, bool kF16, bool kWide, int kR>
cudaError_t launch_gemv_kernel(const cudaLaunchConfig_t& cfg, const GemvMaps& tm,
                               const GemvArgs& a, int device) {
  static std::once_flag once[kOnceDevices];
  once_per_device(once, device, [] {
    cudaFuncSetAttribute(gemv_fwd_kernel<NT, kFmt, kF16, kWide, kR>,
                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                         static_cast<int>(kGemvSmemLimit));
  });
  return cudaLaunchKernelEx(&cfg, gemv_fwd_kernel<NT, kFmt, kF16, kWide, kR>, tm, a);
}

template <int NT, int kFmt, bool kF16, bool kWide>
cudaError_t launch_gemv_r(int r, int device, const cudaLaunchConfig_t& cfg, const GemvMaps& tm,
                          const GemvArgs& a) {
  return r == 2 ? launch_gemv_kernel<NT, kFmt, kF16, kWide, 2>(cfg, tm, a, device)
                : launch_gemv_kernel<NT, kFmt, kF16, kWide, kMaxRowGroups>(cfg, tm, a, device);
}

template <int kFmt, bool kF16>
cudaError_t launch_gemv_as(int nt, bool wide, int r, int device, const cudaLaunchConfig_t& cfg,
                           const GemvMaps& tm, const GemvArgs& a) {
  if constexpr (kFmt != kFmtInt8) {
    if (wide)
      return nt == 1 ? launch_gemv_r<1, kFmt, kF16, true>(r, device, cfg, tm, a)
                     : launch_gemv_r<2, kFmt, kF16, true>(r, device, cfg, tm, a);
  }
  return nt == 1 ? launch_gemv_r<1, kFmt, kF16, false>(r, device, cfg, tm, a)
                 : launch_gemv_r<2, kFmt, kF16, false>(r, device, cfg, tm, a);
}

cudaError_t launch_gemv_fwd(const MatmulCall& c) { return launch_gemv_group(&c, 1); }

cudaError_t launch_gemv_group(const MatmulCall* cs, int count) {
  if (count < 1 || count > kGemvGroupMax) return cudaErrorInvalidValue;
  const MatmulCall& c = cs[0];   // activations, M, K, formats, flags and stream are shared
  const int64_t M = c.M, K = c.K;
  const int num_sms = c.num_sms;
  GemvArgs a = {};
  a.X = static_cast<const uint16_t*>(c.act);
  a.count = count;
  for (int i = 0; i < kGemvGroupMax; ++i) {
    const MatmulCall& ci = cs[i < count ? i : 0];
    a.a8[i] = ci.a8;
    a.scale[i] = ci.scale;
    a.Y[i] = ci.out;
    a.N[i] = ci.N;
  }
  // row tiles of all weights for CTAs of r row groups (16 r rows)
  auto row_tiles = [&](int r) {
    int64_t n = 0;
    for (int i = 0; i < count; ++i) n += (cs[i].N + 16 * r - 1) / (16 * r);
    return n;
  };
  a.M = M;
  a.K = K;
  a.nblk = static_cast<int>(K / kBlock);
  a.out_bf16 = c.out_bf16 ? 1 : 0;
  a.accumulate = c.accumulate ? 1 : 0;
  a.status = c.status;
  // Launch shape: row groups per CTA (8: 128 rows whose 2 K-parts meet in
  // shared memory; 2: 32 rows, 8 K-parts), K-slices across a cluster (a
  // power of two <= 8, reducing through distributed shared memory), n-tiles
  // per CTA and the table layout (the wide one, for 4-bit codes, when its
  // shared memory fits, else the narrow one). In order: fewest waves (two
  // CTAs per SM when they fit in shared memory, else one); a code box for
  // every K-part; a grid that keeps 70% of the SMs busy over one that does
  // not; the fewest token tiles; the smaller activation slice per CTA, all
  // up to 16 KB counting alike (it is staged before the first MMA); no
  // cluster over a cluster (its barrier and remote stores cost about a
  // microsecond); the fewest CTAs (bigger CTAs pay the prologue and the
  // cluster barrier less often; measured faster than filling every SM with
  // smaller ones), else the most busy SMs; two n-tiles over one. (Measured:
  // one 32-row CTA per SM over the full K is 7-11% faster than 128-row CTAs
  // in 4-slice clusters for 3584 x 3584 and 4096 x 4096 at one token.)
  const int fmt = c.fmt;
  struct Shape {
    int s, nt, r;
    bool wide, parts_busy;
    int64_t mtiles, x_cost, ctas, waves, busy;
    size_t smem;
  };
  Shape best{0, 0, 0, false, false, 0, 0, 0, 0, 0, 0};
  const int64_t enough = (7 * static_cast<int64_t>(num_sms)) / 10;
  auto better = [&](const Shape& c) {
    if (best.s == 0) return true;
    if (c.waves != best.waves) return c.waves < best.waves;
    if (c.parts_busy != best.parts_busy) return c.parts_busy;
    const bool ce = c.busy >= enough, be = best.busy >= enough;
    if (ce != be) return ce;
    if (c.mtiles != best.mtiles) return c.mtiles < best.mtiles;
    if (c.x_cost != best.x_cost) return c.x_cost < best.x_cost;
    if (ce && (c.s > 1) != (best.s > 1)) return c.s == 1;
    if (ce && c.ctas != best.ctas) return c.ctas < best.ctas;
    if (!ce && c.busy != best.busy) return c.busy > best.busy;
    return c.nt > best.nt;
  };
  auto search = [&](int nt_lo, int nt_hi) {
   for (int r : {kMaxRowGroups, 2}) {
    const int64_t row_ctas = row_tiles(r);
    for (int sl = kMaxCluster; sl >= 1; sl /= 2) {
      if (sl > a.nblk) continue;
      const int nb = (a.nblk + sl - 1) / sl;
      if (nb > kMaxSliceBlocks && r == kMaxRowGroups) continue;
      for (int n = nt_hi; n >= nt_lo; --n) {
        // the wide table whenever it fits (two narrow CTAs sharing an SM
        // were measured slower than wide ones one after the other)
        bool wide_fits = false;
        for (int w = 1; w >= 0; --w) {
          const bool wide = w == 1;
          if (wide && !gemv_wide(n, fmt)) continue;
          if (!wide && wide_fits) continue;
          const size_t b = gemv_smem_bytes(n, nb, static_cast<int>(std::min<int64_t>(M, 8 * n)),
                                           wide);
          if (b > kGemvSmemLimit) continue;
          wide_fits = wide;
          Shape sh;
          sh.s = sl;
          sh.nt = n;
          sh.r = r;
          sh.wide = wide;
          sh.smem = b;
          sh.mtiles = (M + 8 * n - 1) / (8 * n);
          sh.ctas = row_ctas * sl * sh.mtiles;
          // every K-part has a code box; the activation slice a CTA stages
          // stays small (it is on the critical path before the first MMA)
          const int box_blocks = fmt == kFmtInt8 ? 2 : 4;
          sh.parts_busy = (nb + box_blocks - 1) / box_blocks >= kGemvWarps / r;
          sh.x_cost = std::max<int64_t>(std::min<int64_t>(M, 8 * n) * nb * 128, 16 * 1024);
          const int64_t cap = (b <= kGemvSmemTwoPerSm ? 2 : 1) * static_cast<int64_t>(num_sms);
          sh.waves = (sh.ctas + cap - 1) / cap;
          sh.busy = std::min(sh.ctas, static_cast<int64_t>(num_sms));
          if (better(sh)) best = sh;
        }
      }
    }
   }
  };
  // Up to 8 tokens take one n-tile; if no shape fits, two.
  search(1, M <= 8 ? 1 : 2);
  if (best.s == 0 && M <= 8) search(2, 2);
  const int best_s = best.s, best_nt = best.nt;
  const size_t best_smem = best.smem;
  if (best_s == 0) return cudaErrorInvalidValue;
  a.slices = best_s;
  a.max_nb = (a.nblk + best_s - 1) / best_s;
  a.tile0[0] = 0;
  for (int i = 0; i < kGemvGroupMax; ++i) {
    const int64_t rows_cta = 16 * best.r;
    const int64_t tiles = i < count ? (cs[i].N + rows_cta - 1) / rows_cta : 0;
    a.tile0[i + 1] = a.tile0[i] + static_cast<int>(tiles);
  }
  const int64_t row_ctas = a.tile0[count];   // row tiles of all weights
  const int nt = best_nt;
  const int64_t mtiles = (M + 8 * nt - 1) / (8 * nt);
  // A grid of at most one CTA per SM asks for more shared memory than two
  // CTAs can share, so that the early-launched CTAs of the next kernel in the
  // stream (programmatic dependent launch) cannot pile up two on one SM while
  // others stay idle.
  const size_t smem = best.ctas <= num_sms ? std::max(best_smem, kGemvSmemTwoPerSm + 4096) : best_smem;
  // codes [N, row bytes] (K/2 packed 4-bit, K int8), box 128 B x 16 rows,
  // 128-byte swizzle; one map per weight (unused entries repeat the first)
  const uint64_t row_bytes = static_cast<uint64_t>(c.fmt == kFmtInt8 ? K : K / 2);
  GemvMaps tm;
  for (int i = 0; i < kGemvGroupMax; ++i) {
    const MatmulCall& ci = cs[i < count ? i : 0];
    if (!encode_2d(&tm.m[i], CU_TENSOR_MAP_DATA_TYPE_UINT8, ci.codes, row_bytes,
                   static_cast<uint64_t>(ci.N), row_bytes, 128, 16, CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(row_ctas), static_cast<unsigned>(a.slices),
                     static_cast<unsigned>(mtiles));
  cfg.blockDim = dim3(kGemvThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = c.st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = static_cast<unsigned>(a.slices);
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  switch (c.fmt * 2 + (c.act_f16 ? 1 : 0)) {
    case kFmtNf4 * 2: return launch_gemv_as<kFmtNf4, false>(nt, best.wide, best.r, c.device, cfg, tm, a);
    case kFmtNf4 * 2 + 1: return launch_gemv_as<kFmtNf4, true>(nt, best.wide, best.r, c.device, cfg, tm, a);
    case kFmtFp4 * 2: return launch_gemv_as<kFmtFp4, false>(nt, best.wide, best.r, c.device, cfg, tm, a);
    case kFmtFp4 * 2 + 1: return launch_gemv_as<kFmtFp4, true>(nt, best.wide, best.r, c.device, cfg, tm, a);
    case kFmtInt8 * 2: return launch_gemv_as<kFmtInt8, false>(nt, best.wide, best.r, c.device, cfg, tm, a);
    case kFmtInt8 * 2 + 1: return launch_gemv_as<kFmtInt8, true>(nt, best.wide, best.r, c.device, cfg, tm, a);
  }
  return cudaErrorInvalidValue;
}

}  // namespace nf4
