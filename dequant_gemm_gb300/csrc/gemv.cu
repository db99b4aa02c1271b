// Small-M fused NF4-dequant matmul: Y = X * dequant(W)^T for M <= 16 tokens
// (decode shapes), and a plain fp32 input-gradient kernel for small M
// ("Zenbit", zenbit.pallas_nf4 bullet: the compressed weight is streamed and
// dequantized on chip; the full-precision weight never reaches HBM).
//
// Forward design (HBM-bound: 0.516 B of weight per 2*M flops):
//  * CTA = 8 warps = 128 weight rows (16 per warp) x one K-slice. The S
//    K-slices of the same rows form a thread-block cluster and reduce their
//    partial sums through distributed shared memory, so every output is
//    written once with a plain store (no zeroing pass, no atomics).
//  * A producer warp streams the CTA's packed codes with 2-D TMA boxes of
//    128 rows x 128 bytes (four absmax blocks), 128-byte swizzled, through a
//    ring of four shared-memory slots; the eight compute warps read them
//    bank-conflict free. The absmax codes, scales and activations of the
//    prologue are loaded with all requests issued before any is used.
//  * The weight is the A operand of mma.sync.m16n8k16 (16 rows per warp), the
//    tokens are the N operand (8 per n-tile, one or two n-tiles): the "swap AB"
//    shape for skinny products. Each weight is dequantized once per CTA for
//    all of its tokens.
//  * Dequantization is factored as  sum_b ahat_b * (sum_{k in b} x_k c[q_k]):
//    the MMA consumes the raw levels c[q] and each 64-weight block's partial
//    sum is scaled by its dequantized absmax in fp32 afterwards. The levels
//    enter the tensor core as fp16 (relative error <= 2^-12), which needs the
//    activations in fp16 too: each token's slice of X is scaled by a power of
//    two that puts its max |x| in [2^14, 2^15) before conversion (exact for
//    bf16 values), and the scale is removed from the fp32 result.
//  * One packed byte (two adjacent weights) becomes one f16x2 fragment
//    register through a 256-entry table held in 32 copies, one per lane, so
//    that every lookup of a warp hits 32 distinct banks. Each CTA lays the
//    copies out itself from a 1 KB constant array (no 32 KB copy from L2).
//  * Launched with programmatic stream serialization: the CTAs of the next
//    kernel in the stream can be resident and do their set-up while this one
//    drains; no global memory is touched before griddepcontrol.wait.
//  * Within a block the 4 threads of an MMA quad each own 16 contiguous k
//    (8 code bytes); the reduction order over k is permuted consistently in A
//    and B, which leaves the sum unchanged.
#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "tc.cuh"

namespace nf4 {
namespace {

constexpr int kGemvRows = 128;
constexpr int kTabBytes = kHalfPairTableBytes;
constexpr int kMaxSliceBlocks = 48;
constexpr int kMaxCluster = 8;
constexpr int kOutStride = kGemvRows + 4;     // floats, keeps rows 16-byte aligned

// The level pairs, read with warp-uniform addresses while each CTA lays out
// its 32 lane copies in shared memory.
__constant__ HalfPairs kPairConst = make_half_pairs();

// Not volatile: independent MMA chains of different blocks may interleave.
__device__ __forceinline__ void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                        uint32_t a3, uint32_t b0, uint32_t b1) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}

__device__ __forceinline__ uint2 lds64(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
  return v;
}

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}

// Store a float into CTA `rank`'s shared memory at this CTA's address of
// `local` (made visible to that CTA by the next cluster barrier).
__device__ __forceinline__ void st_dsmem(float* local, uint32_t rank, float v) {
  uint32_t remote;
  asm("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(tc::smem_addr(local)), "r"(rank));
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(remote), "f"(v) : "memory");
}

struct GemvArgs {
  const uint16_t* X;     // bf16 [M, K]
  const uint8_t* a8;     // [N*K/64]
  const float* s2;       // [groups]
  float* Y;              // fp32 [M, N]
  int64_t M, N, K;
  int nblk;              // K / 64
  int slices;            // K-slices = cluster size along y
  int max_nb;            // largest slice, in blocks
  int ring;              // code-box slots (1..kMaxRing)
  int* status;
};

// First absmax block of K-slice s (nblk * slices stays far below 2^31).
__host__ __device__ constexpr int slice_begin(int nblk, int slices, int s) {
  return (nblk * s) / slices;
}

constexpr int kComputeWarps = 8;
constexpr int kGemvThreads = 32 * (kComputeWarps + 1);   // + one TMA producer warp
constexpr int kMaxRing = 4;                 // code boxes in flight, at most
constexpr int kBoxBlocks = 4;               // absmax blocks per box (128 B of codes per row)
constexpr int kBoxBytes = kGemvRows * 128;  // 16 KB: 128 rows x 128 B

// Shared memory (offsets from a 1024-byte aligned base): level table, code
// ring, absmax table, token scales, mbarriers, fp16 activation slice.
constexpr int kOffRing = kTabBytes;
__host__ __device__ constexpr int gemv_off_ahat(int ring) { return kOffRing + ring * kBoxBytes; }
__host__ __device__ constexpr int gemv_off_xinv(int ring, int max_nb) {
  return gemv_off_ahat(ring) + kGemvRows * max_nb * 4;
}
__host__ __device__ constexpr int gemv_off_bars(int ring, int max_nb) {
  return gemv_off_xinv(ring, max_nb) + 64 * 4;
}
__host__ __device__ constexpr int gemv_off_xs(int ring, int max_nb) {
  return gemv_off_bars(ring, max_nb) + (1 + 2 * kMaxRing) * 8 + 8;
}
// Inbox of the cluster reduction: [slices][8 NT tokens][128 / slices rows].
__host__ __device__ constexpr int gemv_off_inbox(int ring, int max_nb, int nt) {
  return (gemv_off_xs(ring, max_nb) + 8 * nt * (max_nb * 128 + 8) + 15) & ~15;
}

template <int NT>
__global__ void __launch_bounds__(kGemvThreads)
gemv_fwd_kernel(const __grid_constant__ CUtensorMap tm_codes, const GemvArgs p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint32_t* tab = reinterpret_cast<uint32_t*>(smem);
  float* ahat_s = reinterpret_cast<float*>(smem + gemv_off_ahat(p.ring));   // [128][max_nb]
  float* xinv = reinterpret_cast<float*>(smem + gemv_off_xinv(p.ring, p.max_nb));  // [64]
  const uint32_t bars = tc::smem_addr(smem + gemv_off_bars(p.ring, p.max_nb));
  auto full_bar = [&](int s) { return bars + 8u * (1 + s); };
  auto empty_bar = [&](int s) { return bars + 8u * (1 + kMaxRing + s); };
  const int xstride_b = p.max_nb * 128 + 8;  // bytes per token row of the fp16 slice
  uint8_t* xs = smem + gemv_off_xs(p.ring, p.max_nb);
  const int nring = p.ring;
  const uint32_t ring = tc::smem_addr(smem + kOffRing);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, t = lane & 3;
  const int64_t row0 = static_cast<int64_t>(blockIdx.x) * kGemvRows;
  const int slice = blockIdx.y;
  const int kb0 = slice_begin(p.nblk, p.slices, slice);
  const int nb = slice_begin(p.nblk, p.slices, slice + 1) - kb0;
  const int nboxes = (nb + kBoxBlocks - 1) / kBoxBlocks;
  const int64_t m0 = static_cast<int64_t>(blockIdx.z) * 8 * NT;
  const int mt = static_cast<int>(min(static_cast<int64_t>(8 * NT), p.M - m0));

  // The prologue's own loads (activations, absmax codes, scales) are issued
  // before the producer starts streaming the code tile, so that they do not
  // queue behind it; the main loop then overlaps the stream.
  const int nkv4 = nb * (kBlock / 4);      // uint2 (4 bf16) per token row
  const uint2* xbase = reinterpret_cast<const uint2*>(p.X + m0 * p.K +
                                                      static_cast<int64_t>(kb0) * kBlock);
  const int64_t xrow4 = p.K / 4;
  uint2 xv[NT][4];
  auto load_x = [&](int c0) {
#pragma unroll
    for (int u = 0; u < NT; ++u) {
      const int tk = warp + 8 * u;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int i = c0 + lane + 32 * c;
        xv[u][c] = (tk < mt && i < nkv4) ? __ldg(xbase + tk * xrow4 + i) : make_uint2(0u, 0u);
      }
    }
  };
  // dequantized absmax: thread t owns row t / 2 and every other block of it
  constexpr int kAh = 4;
  const int ah_r = tid >> 1, ah_par = tid & 1;
  const bool ah_vrow = warp < kComputeWarps && row0 + ah_r < p.N;
  const int64_t ah_bi0 = (row0 + ah_r) * p.nblk + kb0;
  uint32_t av[kAh];
  float sv[kAh];
  auto load_ah = [&](int j0) {
#pragma unroll
    for (int u = 0; u < kAh; ++u) {
      const int j = j0 + 2 * u;
      const bool okj = ah_vrow && j < nb;
      av[u] = okj ? static_cast<uint32_t>(__ldg(p.a8 + ah_bi0 + j)) : 0u;
      sv[u] = okj ? __ldg(p.s2 + ((ah_bi0 + j) >> 8)) : 0.0f;
    }
  };
  // Programmatic dependent launch: the next kernel in the stream may start its
  // own set-up now; this one touches no global memory before the previous
  // kernel has completed (griddepcontrol.wait).
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // level table: entry e, copy l at word 32 e + l (one conflict-free store per
  // entry and warp)
  for (int e = warp; e < 256; e += kComputeWarps + 1) tab[e * 32 + lane] = kPairConst.w[e];
  asm volatile("griddepcontrol.wait;" ::: "memory");

  if (warp < kComputeWarps) {
    load_x(0);
    load_ah(ah_par);
  }

  if (tid == 0) {
    for (int s = 0; s < kMaxRing; ++s) {
      tc::mbar_init(full_bar(s), 1);
      tc::mbar_init(empty_bar(s), kComputeWarps);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();

  bool ok = true;
  // Producer (lane 0 of the last warp): level table and code boxes (128 rows
  // x 4 blocks each, 128-byte swizzled) through a ring of `nring` slots. The
  // first ring-full goes out before the prologue barrier; the rest, which
  // waits for slots to free, after it.
  const bool producer = warp == kComputeWarps && lane == 0;
  int issued = 0;
  auto issue_boxes = [&](int upto) {
    for (int b = issued; b < upto; ++b) {
      const int slot = b % nring;
      if (b >= nring && !tc::mbar_wait(empty_bar(slot), ((b / nring) - 1) & 1)) {
        report_status(p.status, kStatusTimeout, kSiteGemv, kRoleProducer);
        return;
      }
      tc::mbar_arrive_expect_tx(full_bar(slot), kBoxBytes);
      tc::tma_load_2d(ring + slot * kBoxBytes, &tm_codes, (kb0 + kBoxBlocks * b) * 32,
                      static_cast<int32_t>(row0), full_bar(slot));
      issued = b + 1;
    }
  };
  if (producer) {
    tc::prefetch_tensormap(&tm_codes);
    issue_boxes(min(nboxes, nring));
  }
  if (warp < kComputeWarps) {
    // Dequantized absmax (batches of kAh blocks; the first one is in flight).
    {
      float* arow = ahat_s + ah_r * p.max_nb;
      for (int j0 = ah_par; j0 < nb; j0 += 2 * kAh) {
        if (j0 != ah_par) load_ah(j0);
#pragma unroll
        for (int u = 0; u < kAh; ++u) {
          const int j = j0 + 2 * u;
          if (j < nb) arow[j] = dequant_absmax(av[u], sv[u]);
        }
      }
    }

    // Activations: warp w stages tokens w + 8u (u < NT) in chunks of 128 uint2
    // (8 blocks; the first one is in flight): per-token max |x| -> power-of-two
    // scale into [2^14, 2^15) -> fp16. A slice of at most 8 blocks is converted
    // straight from registers, longer slices are read a second time.
    {
      auto absmax4 = [](uint2 v) {
        const float2 f0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&v.x));
        const float2 f1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&v.y));
        return fmaxf(fmaxf(fabsf(f0.x), fabsf(f0.y)), fmaxf(fabsf(f1.x), fabsf(f1.y)));
      };
      auto convert = [](uint2 v, float scale) {
        const float2 f0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&v.x));
        const float2 f1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&v.y));
        const __half2 h0 = __floats2half2_rn(f0.x * scale, f0.y * scale);
        const __half2 h1 = __floats2half2_rn(f1.x * scale, f1.y * scale);
        return make_uint2(*reinterpret_cast<const uint32_t*>(&h0), *reinterpret_cast<const uint32_t*>(&h1));
      };
      float mx[NT];
#pragma unroll
      for (int u = 0; u < NT; ++u) mx[u] = 0.0f;
      for (int c0 = 0; c0 < nkv4; c0 += 128) {
        if (c0 > 0) load_x(c0);
#pragma unroll
        for (int u = 0; u < NT; ++u)
#pragma unroll
          for (int c = 0; c < 4; ++c) mx[u] = fmaxf(mx[u], absmax4(xv[u][c]));
      }
      float scale[NT];
#pragma unroll
      for (int u = 0; u < NT; ++u) {
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1)
          mx[u] = fmaxf(mx[u], __shfl_xor_sync(0xffffffffu, mx[u], off));
        int e = 0;
        if (mx[u] > 0.0f) {
          const int E = max(1, static_cast<int>((__float_as_uint(mx[u]) >> 23) & 0xffu));
          e = min(141 - E, 126);
        }
        scale[u] = __uint_as_float(static_cast<uint32_t>(e + 127) << 23);
        if (lane == 0) xinv[warp + 8 * u] = __uint_as_float(static_cast<uint32_t>(127 - e) << 23);
      }
      for (int c0 = 0; c0 < nkv4; c0 += 128) {
        if (nkv4 > 128) load_x(c0);
#pragma unroll
        for (int u = 0; u < NT; ++u) {
          const int tk = warp + 8 * u;
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const int i = c0 + lane + 32 * c;
            if (tk < mt && i < nkv4)
              reinterpret_cast<uint2*>(xs + tk * xstride_b)[i] = convert(xv[u][c], scale[u]);
          }
        }
      }
    }
  }
  __syncthreads();
  if (producer) {
    issue_boxes(nboxes);
    // copies still in flight land before the CTA may exit
    for (int b = max(0, issued - nring); b < issued; ++b)
      tc::mbar_wait(full_bar(b % nring), (b / nring) & 1);
  }

  float acc[NT][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[nt][i] = 0.0f;

  if (warp < kComputeWarps) {
    const uint32_t tab_b = tc::smem_addr(tab) + lane * 4;   // this lane's copy of the table
    const uint32_t xs_a = tc::smem_addr(xs) + g * xstride_b + t * 32;
    const float* ah_g = ahat_s + (warp * 16 + g) * p.max_nb;
    const float* ah_g8 = ah_g + 8 * p.max_nb;
    // swizzled offsets of this lane's 8 code bytes in rows g and g + 8 of the
    // warp: 16-byte chunk c of a box row r sits at chunk c ^ (r & 7)
    const uint32_t row_a = ring + (warp * 16 + g) * 128 + (t & 1) * 8;
    const uint32_t row_b = row_a + 8 * 128;
    bool tok_ok[NT];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) tok_ok[nt] = nt * 8 + g < mt;

    for (int b = 0; b < nboxes && ok; ++b) {
      const int slot = b % nring;
      if (!tc::mbar_wait(full_bar(slot), (b / nring) & 1)) {
        ok = false;
        break;
      }
#pragma unroll
      for (int jj = 0; jj < kBoxBlocks; ++jj) {
        const int j = b * kBoxBlocks + jj;
        if (j < nb) {
          const uint32_t chunk = static_cast<uint32_t>((2 * jj + (t >> 1)) ^ g) << 4;
          const uint2 cg = lds64(row_a + slot * kBoxBytes + chunk);
          const uint2 cg8 = lds64(row_b + slot * kBoxBytes + chunk);
          float part[NT][4];
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int i = 0; i < 4; ++i) part[nt][i] = 0.0f;
#pragma unroll
          for (int s = 0; s < 4; ++s) {
            const uint32_t wg = (s < 2) ? cg.x : cg.y;
            const uint32_t wg8 = (s < 2) ? cg8.x : cg8.y;
            const int sh = 16 * (s & 1);
            // byte 2s -> logical k (2t, 2t+1); byte 2s+1 -> logical k (2t+8, 2t+9)
            const uint32_t a0 = lds32(tab_b + (((wg >> sh) & 0xffu) << 7));
            const uint32_t a2 = lds32(tab_b + (((wg >> (sh + 8)) & 0xffu) << 7));
            const uint32_t a1 = lds32(tab_b + (((wg8 >> sh) & 0xffu) << 7));
            const uint32_t a3 = lds32(tab_b + (((wg8 >> (sh + 8)) & 0xffu) << 7));
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
              uint2 bx = make_uint2(0u, 0u);
              if (tok_ok[nt]) bx = lds64(xs_a + nt * 8 * xstride_b + j * 128 + 8 * s);
              mma_f16(part[nt], a0, a1, a2, a3, bx.x, bx.y);
            }
          }
          const float ag = ah_g[j], ag8 = ah_g8[j];
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            acc[nt][0] = fmaf(ag, part[nt][0], acc[nt][0]);
            acc[nt][1] = fmaf(ag, part[nt][1], acc[nt][1]);
            acc[nt][2] = fmaf(ag8, part[nt][2], acc[nt][2]);
            acc[nt][3] = fmaf(ag8, part[nt][3], acc[nt][3]);
          }
        }
      }
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(empty_bar(slot));   // slot free for the producer
    }
    if (!ok) report_status(p.status, kStatusTimeout, kSiteGemv, kRoleCompute);
  }

  // Epilogue: undo the token scales and stage this slice's partial
  // [8 NT tokens x 128 rows] in shared memory (over the level table).
  float inv0[NT], inv1[NT];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int tk0 = nt * 8 + 2 * t;
    inv0[nt] = tk0 < mt ? xinv[tk0] : 0.0f;
    inv1[nt] = tk0 + 1 < mt ? xinv[tk0 + 1] : 0.0f;
  }
  __syncthreads();
  float* out_s = reinterpret_cast<float*>(smem);
  if (p.slices == 1 && warp < kComputeWarps) {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int tk0 = nt * 8 + 2 * t, tk1 = tk0 + 1;
      const int rg = warp * 16 + g;
      out_s[tk0 * kOutStride + rg] = acc[nt][0] * inv0[nt];
      out_s[tk1 * kOutStride + rg] = acc[nt][1] * inv1[nt];
      out_s[tk0 * kOutStride + rg + 8] = acc[nt][2] * inv0[nt];
      out_s[tk1 * kOutStride + rg + 8] = acc[nt][3] * inv1[nt];
    }
  }
  if (p.slices == 1) {
    __syncthreads();
    for (int i = tid; i < 8 * NT * (kGemvRows / 4); i += kGemvThreads) {
      const int tk = i / (kGemvRows / 4), r4 = (i % (kGemvRows / 4)) * 4;
      if (tk < mt && row0 + r4 < p.N)
        *reinterpret_cast<float4*>(p.Y + (m0 + tk) * p.N + row0 + r4) =
            *reinterpret_cast<const float4*>(out_s + tk * kOutStride + r4);
    }
  } else {
    // Cluster reduction, push form: CTA `rank` owns rows [rank*rpc, (rank+1)*rpc)
    // of the row tile. Every CTA stores its scaled partial of those rows into
    // the owner's inbox slot for its slice, one cluster barrier makes the
    // stores visible, and each owner sums its slots and writes Y once.
    float* inbox = reinterpret_cast<float*>(smem + gemv_off_inbox(p.ring, p.max_nb, NT));
    const int rpc = kGemvRows / p.slices;          // rows owned per CTA (a power of two)
    const int rpc_shift = 31 - __clz(rpc);
    if (warp < kComputeWarps) {
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const int tk0 = nt * 8 + 2 * t;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int tk = tk0 + (e & 1);
          const int rg = warp * 16 + g + 8 * (e >> 1);
          const float v = acc[nt][e] * ((e & 1) ? inv1[nt] : inv0[nt]);
          const uint32_t owner = static_cast<uint32_t>(rg >> rpc_shift);
          st_dsmem(inbox + ((slice * 8 * NT + tk) << rpc_shift) + (rg & (rpc - 1)), owner, v);
        }
      }
    }
    cluster_sync();
    const int rank = static_cast<int>(cluster_ctarank());
    for (int i = tid; i < 8 * NT * rpc; i += kGemvThreads) {
      const int tk = i >> rpc_shift, rl = i & (rpc - 1), r = rank * rpc + rl;
      if (tk < mt && row0 + r < p.N) {
        float v = 0.0f;
        for (int c = 0; c < p.slices; ++c) v += inbox[((c * 8 * NT + tk) << rpc_shift) + rl];
        p.Y[(m0 + tk) * p.N + row0 + r] = v;
      }
    }
  }
}

// Input gradient for small M in plain fp32: dX[m, k] = sum_n dY[m, n] w[n, k].
// CTA = 256 consecutive k (4 absmax blocks) x a slice of rows n; one thread
// per k column; dY and the dequantized absmax of 64 rows at a time are staged
// in shared memory. Slices of n are summed with atomics into a zeroed dX.
constexpr int kDxThreads = 256;
constexpr int kDxRows = 64;
constexpr int kDxMaxM = 16;

__global__ void __launch_bounds__(kDxThreads)
simt_dx_kernel(const uint16_t* __restrict__ dY, int64_t M, const uint8_t* __restrict__ codes,
               const uint8_t* __restrict__ a8, const float* __restrict__ s2, int64_t N,
               int64_t K, float* __restrict__ dX, int64_t rows_per_slice, int atomic_out) {
  __shared__ float s_levels[16];
  __shared__ float s_ahat[kDxRows][4];
  __shared__ float s_dy[kDxMaxM][kDxRows];
  const int tid = threadIdx.x;
  if (tid < 16) s_levels[tid] = __uint_as_float(kLevelBitsDev[tid]);
  const int64_t k = static_cast<int64_t>(blockIdx.x) * kDxThreads + tid;
  const int64_t kb_base = (static_cast<int64_t>(blockIdx.x) * kDxThreads) / kBlock;
  const int64_t m0 = static_cast<int64_t>(blockIdx.z) * kDxMaxM;
  const int mt = static_cast<int>(min(static_cast<int64_t>(kDxMaxM), M - m0));
  const int64_t n_begin = blockIdx.y * rows_per_slice;
  const int64_t n_end = min(N, n_begin + rows_per_slice);
  const int64_t nblk = K / kBlock;
  float acc[kDxMaxM];
#pragma unroll
  for (int m = 0; m < kDxMaxM; ++m) acc[m] = 0.0f;

  for (int64_t n0 = n_begin; n0 < n_end; n0 += kDxRows) {
    __syncthreads();
    {
      const int r = tid >> 2, j = tid & 3;
      const int64_t n = n0 + r;
      float v = 0.0f;
      if (n < n_end && kb_base + j < nblk) {
        const int64_t bi = n * nblk + kb_base + j;
        v = dequant_absmax(a8[bi], s2[bi / kGroup]);
      }
      s_ahat[r][j] = v;
    }
    for (int i = tid; i < kDxMaxM * kDxRows; i += kDxThreads) {
      const int m = i / kDxRows, r = i % kDxRows;
      const int64_t n = n0 + r;
      float v = 0.0f;
      if (m < mt && n < n_end) {
        const uint16_t bits = dY[(m0 + m) * N + n];
        v = __bfloat162float(__ushort_as_bfloat16(bits));
      }
      s_dy[m][r] = v;
    }
    __syncthreads();
    if (k < K) {
      const int rows = static_cast<int>(min(static_cast<int64_t>(kDxRows), n_end - n0));
      for (int r = 0; r < rows; ++r) {
        const uint8_t byte = codes[((n0 + r) * K + k) >> 1];
        const uint32_t q = (k & 1) ? (byte & 15u) : (byte >> 4);
        const float w = __fmul_rn(s_levels[q], s_ahat[r][tid >> 6]);
#pragma unroll
        for (int m = 0; m < kDxMaxM; ++m) acc[m] = fmaf(s_dy[m][r], w, acc[m]);
      }
    }
  }
  if (k < K) {
#pragma unroll
    for (int m = 0; m < kDxMaxM; ++m) {
      if (m < mt) {
        float* dst = dX + (m0 + m) * K + k;
        if (atomic_out) atomicAdd(dst, acc[m]);
        else *dst = acc[m];
      }
    }
  }
}

}  // namespace

// Dynamic shared memory of one GEMV CTA (plus 1 KB to align the base).
constexpr size_t gemv_smem_bytes(int nt, int ring, int max_nb) {
  return static_cast<size_t>(gemv_off_inbox(ring, max_nb, nt)) + 8 * nt * kGemvRows * 4 + 1024;
}
constexpr size_t kGemvSmemLimit = 220 * 1024;

template <int NT>
cudaError_t launch_gemv_nt(const cudaLaunchConfig_t& cfg, const CUtensorMap& tm, const GemvArgs& a) {
  return cudaLaunchKernelEx(&cfg, gemv_fwd_kernel<NT>, tm, a);
}

cudaError_t launch_gemv_fwd(const uint16_t* X, int64_t M, const uint8_t* codes,
                            const uint8_t* a8, const float* s2, int64_t N, int64_t K, float* Y,
                            int num_sms, int* status, cudaStream_t st) {
  GemvArgs a;
  a.X = X;
  a.a8 = a8;
  a.s2 = s2;
  a.Y = Y;
  a.M = M;
  a.N = N;
  a.K = K;
  a.nblk = static_cast<int>(K / kBlock);
  a.status = status;
  // K-slices (cluster size): aim for about two CTAs per SM, at most 8, each
  // slice at least one block and at most kMaxSliceBlocks blocks.
  const int64_t row_ctas = (N + kGemvRows - 1) / kGemvRows;
  int slices = 1;
  while (slices < kMaxCluster && row_ctas * slices < 2 * static_cast<int64_t>(num_sms) &&
         slices * 2 <= a.nblk)
    slices *= 2;
  while (slices < kMaxCluster && (a.nblk + slices - 1) / slices > kMaxSliceBlocks) slices *= 2;
  if ((a.nblk + slices - 1) / slices > kMaxSliceBlocks) return cudaErrorInvalidValue;
  a.slices = slices;
  a.max_nb = (a.nblk + slices - 1) / slices;
  a.ring = std::min(kMaxRing, (a.max_nb + kBoxBlocks - 1) / kBoxBlocks);
  int nt = M <= 8 ? 1 : 2;
  while (nt > 1 && gemv_smem_bytes(nt, a.ring, a.max_nb) > kGemvSmemLimit) nt /= 2;
  const int64_t mtiles = (M + 8 * nt - 1) / (8 * nt);
  const size_t smem = gemv_smem_bytes(nt, a.ring, a.max_nb);
  if (smem > kGemvSmemLimit) return cudaErrorInvalidValue;
  // packed codes [N, K/2] bytes, box 128 B (4 absmax blocks) x 128 rows, 128-byte swizzle
  CUtensorMap tm;
  if (!encode_2d(&tm, CU_TENSOR_MAP_DATA_TYPE_UINT8, codes, static_cast<uint64_t>(K / 2),
                 static_cast<uint64_t>(N), static_cast<uint64_t>(K / 2), 128, kGemvRows,
                 CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  static std::once_flag once;
  std::call_once(once, [] {
    const int lim = static_cast<int>(kGemvSmemLimit);
    cudaFuncSetAttribute(gemv_fwd_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, lim);
    cudaFuncSetAttribute(gemv_fwd_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, lim);
  });
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(row_ctas), static_cast<unsigned>(slices),
                     static_cast<unsigned>(mtiles));
  cfg.blockDim = dim3(kGemvThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = static_cast<unsigned>(slices);
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return nt == 1 ? launch_gemv_nt<1>(cfg, tm, a) : launch_gemv_nt<2>(cfg, tm, a);
}

cudaError_t launch_simt_dx(const uint16_t* dY, int64_t M, const uint8_t* codes,
                           const uint8_t* a8, const float* s2, int64_t N, int64_t K, float* dX,
                           int num_sms, cudaStream_t st) {
  const int64_t kctas = (K + kDxThreads - 1) / kDxThreads;
  const int64_t mtiles = (M + kDxMaxM - 1) / kDxMaxM;
  int64_t slices = (2 * static_cast<int64_t>(num_sms) + kctas * mtiles - 1) / (kctas * mtiles);
  slices = std::max<int64_t>(1, std::min<int64_t>(slices, (N + kDxRows - 1) / kDxRows));
  int64_t rows_per_slice = (N + slices - 1) / slices;
  rows_per_slice = ((rows_per_slice + kDxRows - 1) / kDxRows) * kDxRows;
  slices = (N + rows_per_slice - 1) / rows_per_slice;
  if (slices > 1) {
    cudaError_t e = cudaMemsetAsync(dX, 0, static_cast<size_t>(M) * K * sizeof(float), st);
    if (e != cudaSuccess) return e;
  }
  dim3 grid(static_cast<unsigned>(kctas), static_cast<unsigned>(slices),
            static_cast<unsigned>(mtiles));
  simt_dx_kernel<<<grid, kDxThreads, 0, st>>>(dY, M, codes, a8, s2, N, K, dX, rows_per_slice,
                                              slices > 1 ? 1 : 0);
  return cudaGetLastError();
}

}  // namespace nf4
