// Large-M fused NF4-dequant matmuls on the sm_103a tensor cores (tcgen05):
//   forward   Y[m, n]  = sum_k X[m, k]  * w[n, k]
//   input grad dX[m, k] = sum_n dY[m, n] * w[n, k]      (no dW)
// ("Zenbit", zenbit.pallas_nf4 bullet: compressed weight tiles streamed in and
// dequantized on chip, full-precision weight never in HBM; dL/dX only.)
//
// One CTA computes a 128 x BN tile of D = A * B^T with the weight as the
// 128-row A operand and the tokens as the BN-column B operand (BN = 64, 128 or
// 256; 256 on CTA pairs that share one 256 x 256 MMA), looping over the
// reduction in stages of 64:
//   * warp 0 (one thread) TMA-loads the stage's activation tile (bf16,
//     128-byte swizzle, the K-major B operand) and its packed-code tile;
//   * the dequant warps, in groups of four (one per tensor-memory lane
//     quarter) that take the stages in turn, dequantize the codes (level *
//     dequantized absmax, rounded to bf16) and write them straight into
//     tensor memory, where the MMA reads its A operand: the dequantized
//     weight never touches shared memory;
//   * warp 1 issues tcgen05.mma (128 x BN x 16) from one elected lane into
//     an fp32 accumulator in tensor memory and commits each stage back to the
//     producer;
//   * the dequant warps then read the accumulator with tcgen05.ld and store
//     fp32 outputs (32 consecutive outputs of one token per warp store).
//
// Forward: the tile is 128 weight rows, one row per dequant thread, walked
// along K. Both levels of a code byte come from one lookup in a 256-entry
// fp16 level pair table kept in 32 lane-private copies (every lookup of a
// warp hits 32 distinct banks), are widened to fp32 and multiplied by the
// row's dequantized absmax, a register.
//
// Input gradient: the tile is 128 weight columns walked along N (the
// transposed walk), so a thread needs its column's nibbles down the stage's
// 64 rows. Each warp reads its 32 columns' codes as 32-bit words (8 columns
// of one row) and transposes 8 x 8 nibble blocks across lanes with three
// shuffle rounds, after which a byte of a thread's word holds the codes of
// two consecutive rows of its column: exactly one 32-bit tensor-memory word
// of the A operand. That byte indexes the same pair table; the two levels
// are multiplied by their rows' dequantized absmax, which the warp computes
// for its 64 rows and broadcasts through shared memory.
//
// When the output tiles alone cannot fill the GPU the reduction is split
// across CTAs and summed with atomics into a zeroed output.
//
// Every mbarrier wait is bounded; a CTA that gives up records a timeout in the
// device status word, skips the remaining work and still releases its tensor
// memory.
#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "tc.cuh"

namespace nf4 {
namespace {

constexpr int kTileRows = 128;               // MMA M
constexpr int kCodesStageBytes = 4096;       // 128 x 64 nibbles
constexpr uint32_t kTmemCols = 512;

// Per-direction and per-token-tile configuration and shared-memory layout.
// The token tile BN (MMA N) sets the stage size; smaller tiles get deeper
// rings, so that enough code bytes are in flight per SM to cover the memory
// latency. Tensor memory holds the BN fp32 accumulator columns, then one
// 32-column A-operand slot per stage.
//
// The forward with BN = 256 runs on CTA pairs (cta_group::2): the two CTAs of
// a cluster hold 128 weight rows each, and half of the token tile each; the
// MMA warp of the even CTA issues 256 x 256 x 16 MMAs over both SMs. Each SM
// then stages and reads only half of the activation tile, which is most of
// the shared-memory traffic of a stage. The dequant warps of
// both CTAs arrive on the issuing CTA's stage barrier. The arrival takes the
// instruction's default (CTA-scope) release: by then the warp's tensor-memory
// stores have retired (tcgen05.wait::st) and the stage's copies have been seen
// complete, and a cluster-scope release was measured to stall the arriving
// thread for 1-2.5K cycles on a busy SM, enough to halve the MMA rate.
template <bool kDx, int kBN>
struct Cfg {
  static constexpr bool kPair = kBN == 256 && !kDx;
  static constexpr int kCg = kPair ? 2 : 1;          // tcgen05 cta_group
  // dequant warp groups: a group needs several MMA stage times per stage;
  // four for the forward (72 registers a thread), three for the input
  // gradient, whose transposed walk runs best with ~120 registers a thread
  static constexpr int kGroups = kDx ? 3 : 4;
  static constexpr int kDqWarps = 4 * kGroups;
  static constexpr int kThreads = 64 + 32 * kDqWarps;
  static constexpr int kStages = kBN == 64 ? 12 : (kBN == 128 || kPair ? 8 : 5);
  static constexpr int kBRows = kPair ? kBN / 2 : kBN;   // tokens staged per CTA
  static constexpr int kActStageBytes = kBRows * 128;    // 64 bf16 per token row
  static constexpr uint32_t kTmemA0 = kBN;
  static constexpr int kLutBytes = kHalfPairTableBytes;
  static constexpr int kAhatBytes = kDx ? kDqWarps * 64 * 4 : 0;   // per-warp row scales
  static constexpr int kOffAct = 0;
  static constexpr int kOffCodes = kOffAct + kStages * kActStageBytes;
  static constexpr int kOffLut = kOffCodes + kStages * kCodesStageBytes;
  static constexpr int kOffAhat = kOffLut + kLutBytes;
  static constexpr int kOffBars = kOffAhat + kAhatBytes;
  static constexpr int kNumBars = 3 * kStages + 2;
  static constexpr int kOffMisc = kOffBars + kNumBars * 8;
  static constexpr int kSmemBytes = kOffMisc + 16 + 1024;   // + alignment slack
  static_assert(kTmemA0 + 32 * kStages <= kTmemCols, "tensor memory columns");
  static_assert(kBN == 64 || kBN == 128 || kBN == 256, "token tile");
  static_assert(kSmemBytes <= 227 * 1024, "shared memory");
};

struct TcArgs {
  const uint8_t* a8;
  const float* s2;
  float* out;        // Y [M, N] or dX [M, K]
  int64_t M, N, K;
  int nblk;          // K / 64
  int bn;            // token tile
  int stages_total;
  int stages_per_split;
  int atomic_out;
  int* status;
};

// Level pair table of both directions (fp16 levels, layout in common.cuh).
__device__ __align__(128) const HalfPairTable kHalfPairs = make_half_pair_table();

__device__ __forceinline__ void bulk_copy_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                              uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
      : "memory");
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}


template <bool kDx, int kBN>
__global__ void __launch_bounds__(Cfg<kDx, kBN>::kThreads, 1)
tc_gemm_kernel(const __grid_constant__ CUtensorMap tm_act, const __grid_constant__ CUtensorMap tm_codes,
               const TcArgs p) {
  using C = Cfg<kDx, kBN>;
  constexpr bool kPair = C::kPair;
  constexpr int kCg = C::kCg;
  constexpr int kStages = C::kStages;
  constexpr int kGroups = C::kGroups;
  constexpr int kActStageBytes = C::kActStageBytes;
  constexpr uint32_t kTmemA0 = C::kTmemA0;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t bars = tc::smem_addr(smem + C::kOffBars);
  auto full_bar = [&](int s) { return bars + 8u * s; };
  auto dq_bar = [&](int s) { return bars + 8u * (kStages + s); };
  auto empty_bar = [&](int s) { return bars + 8u * (2 * kStages + s); };
  const uint32_t accum_bar = bars + 8u * (3 * kStages);
  const uint32_t lut_bar = bars + 8u * (3 * kStages + 1);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // A pair is the cluster (2, 1, 1): CTA 2p + rank holds rows 128 (2p + rank),
  // the token half rank of the tile, and rank 0 issues the pair's MMAs.
  const uint32_t rank = kPair ? tc::cluster_ctarank() : 0u;
  const int64_t r0 = static_cast<int64_t>(blockIdx.x) * kTileRows;
  const int64_t m0 = static_cast<int64_t>(blockIdx.y) * p.bn;
  const int s_begin = blockIdx.z * p.stages_per_split;
  const int nst = min(p.stages_per_split, p.stages_total - s_begin);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      tc::mbar_init(full_bar(s), 1);
      // one arrival per warp of the stage's group, in both CTAs of a pair
      tc::mbar_init(dq_bar(s), 4 * kCg);
      tc::mbar_init(empty_bar(s), 1);
    }
    tc::mbar_init(accum_bar, 1);
    tc::mbar_init(lut_bar, 1);
    *abort_flag = 0;
    tc::fence_barrier_init();
    tc::mbar_arrive_expect_tx(lut_bar, C::kLutBytes);
    bulk_copy_g2s(tc::smem_addr(smem + C::kOffLut), &kHalfPairs, C::kLutBytes, lut_bar);
  }
  if (warp == 0 && lane == 0) {
    tc::prefetch_tensormap(&tm_act);
    tc::prefetch_tensormap(&tm_codes);
  }
  if (warp == 1) tc::tmem_alloc<kCg>(tc::smem_addr(tmem_slot), kTmemCols);
  tc::fence_before_sync();
  if constexpr (kPair) tc::cluster_sync();   // the peer's barriers exist before any arrival
  else __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  auto fail = [&](uint32_t role) {
    report_status(p.status, kStatusTimeout, kDx ? kSiteTcDx : kSiteTcFwd, role);
    *abort_flag = 1;
  };

  if (warp == 0) {
    // ------------------------------------------------------------ producer --
    if (lane == 0) {
      const uint32_t tx = static_cast<uint32_t>(kActStageBytes + kCodesStageBytes);
      const int32_t m_load = static_cast<int32_t>(m0) + static_cast<int32_t>(rank) * C::kBRows;
      int issued = 0;
      for (int i = 0; i < nst && !*abort_flag; ++i) {
        const int slot = i % kStages;
        const uint32_t ph = (i / kStages) & 1;
        if (!tc::mbar_wait(empty_bar(slot), ph ^ 1)) { fail(kRoleProducer); break; }
        const int s = s_begin + i;
        tc::mbar_arrive_expect_tx(full_bar(slot), tx);
        const uint32_t act = tc::smem_addr(smem + C::kOffAct + slot * kActStageBytes);
        const uint32_t cod = tc::smem_addr(smem + C::kOffCodes + slot * kCodesStageBytes);
        tc::tma_load_2d(act, &tm_act, s * 64, m_load, full_bar(slot));
        if (!kDx) {
          // 128 rows x 32 bytes
          tc::tma_load_2d(cod, &tm_codes, s * 32, static_cast<int32_t>(r0), full_bar(slot));
        } else {
          // four 16-byte x 64-row boxes, one per lane quarter: quarter c's
          // 32 columns land as a dense [64 rows][16 B] block at c * 1 KB
#pragma unroll
          for (int c = 0; c < 4; ++c)
            tc::tma_load_2d(cod + 1024u * c, &tm_codes, static_cast<int32_t>(r0 / 2 + 16 * c),
                            s * 64, full_bar(slot));
        }
        ++issued;
      }
      if (*abort_flag) {  // let copies in flight land before the CTA exits
        for (int i = max(0, issued - kStages); i < issued; ++i)
          tc::mbar_wait(full_bar(i % kStages), (i / kStages) & 1);
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA --
    // The whole warp runs the loop on warp-uniform values and one elected
    // lane issues, which lets the MMA operands stay uniform (a loop inside a
    // one-thread branch issued ~60% slower). The dequant warps arrive on
    // dq_bar only after they have seen the stage's copies land on full_bar,
    // so its completion orders both the tensor-memory A operand and the
    // shared-memory B tile before the MMAs; a failure elsewhere surfaces here
    // as a timeout. The wait is a spin on the non-blocking test: a suspending
    // try_wait on the issuing warp lets the MMAs already queued drain (about
    // 380 idle tensor cycles per wait, as measured). On a pair the peer's
    // dequant warps arrive here too, once they have stored the stage and
    // seen their own copies land.
    if (rank == 0) {
      const uint32_t idesc = tc::idesc_bf16_f32(kTileRows * kCg, static_cast<uint32_t>(p.bn));
      const uint64_t bdesc0 = tc::sw128_kmajor_desc(tc::smem_addr(smem + C::kOffAct));
      for (int i = 0; i < nst; ++i) {
        const int sl = i % kStages;
        const bool ok = tc::mbar_wait_spin<kPair>(dq_bar(sl), (i / kStages) & 1);
        if (!__all_sync(0xffffffffu, ok)) {
          if (lane == 0) fail(kRoleMma);
          break;
        }
        tc::fence_after_sync();
        const uint32_t a = tmem + kTmemA0 + 32u * sl;
        // the descriptor's start-address field counts 16-byte units
        const uint64_t bdesc = bdesc0 + static_cast<uint64_t>(sl * (kActStageBytes >> 4));
        if (tc::elect_one()) {
#pragma unroll
          for (int j = 0; j < 4; ++j)
            tc::mma_bf16_tmem_a<kCg>(tmem, a + 8u * j, bdesc + 2u * j, idesc,
                                     (i | j) != 0 ? 1u : 0u);
          tc::mma_commit<kCg>(empty_bar(sl));
        }
        __syncwarp();
      }
      if (tc::elect_one()) tc::mma_commit<kCg>(accum_bar);
      __syncwarp();
      // all MMAs done before teardown
      if (lane == 0 && !tc::mbar_wait(accum_bar, 0)) fail(kRoleMma);
    }
  } else {
    // ---------------------------------------------------- dequant + store --
    // the stage's A slot is written: tell the pair's MMA thread
    auto arrive_dq = [&](int slot) {
      if constexpr (kPair) tc::mbar_arrive_remote(tc::mapa(dq_bar(slot), 0));
      else tc::mbar_arrive(dq_bar(slot));
    };
    const int q = warp & 3;                 // TMEM lane quarter of this warp
    const int grp = (warp - 2) >> 2;        // takes the stages i % kGroups == grp
    const uint32_t lane_base = static_cast<uint32_t>(32 * q) << 16;
    // tile row (forward: weight row; input gradient: weight column) held by
    // this thread's accumulator lane
    int tile_row = 32 * q + lane;
    if (!kDx) {
      const int64_t n = r0 + tile_row;      // this thread's weight row
      const bool vrow = n < p.N;
      const uint8_t* tab = smem + C::kOffLut + 4 * lane;
      uint32_t a8v = 0;
      float s2v = 0.0f;
      auto load_scale = [&](int i) {
        if (vrow && i < nst) {
          const int64_t bi = n * p.nblk + s_begin + i;
          a8v = p.a8[bi];
          s2v = p.s2[bi >> 8];
        }
      };
      load_scale(grp);
      if (!tc::mbar_wait(lut_bar, 0)) fail(kRoleCompute);
      for (int i = grp; i < nst; i += kGroups) {
        const int slot = i % kStages;
        const uint32_t ph = (i / kStages) & 1;
        const float ahat = vrow ? dequant_absmax(a8v, s2v) : 0.0f;
        const float2 ahat2 = make_float2(ahat, ahat);
        load_scale(i + kGroups);
        // warp-uniform: the stage is done by all lanes or by none (the
        // arrival below follows a __syncwarp)
        bool go = !*abort_flag;
        if (go && !tc::mbar_wait(full_bar(slot), ph)) {
          fail(kRoleCompute);
          go = false;
        }
        if (!__all_sync(0xffffffffu, go)) continue;
        const uint8_t* crow = smem + C::kOffCodes + slot * kCodesStageBytes + tile_row * 32;
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          const uint4 c = *reinterpret_cast<const uint4*>(crow + 16 * hf);
          const uint32_t words[4] = {c.x, c.y, c.z, c.w};
          uint32_t v[16];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
#pragma unroll
            for (int b = 0; b < 4; ++b) {
              const uint32_t byte = __byte_perm(words[j], 0u, 0x4440u + b);
              const __half2 h2 = *reinterpret_cast<const __half2*>(tab + (byte << 7));
              const float2 lv = __fmul2_rn(__half22float2(h2), ahat2);
              v[4 * j + b] = pack_bf16x2(lv.x, lv.y);
            }
          }
          tc::tmem_st16(tmem + lane_base + kTmemA0 + 32u * slot + 16u * hf, v);
        }
        tc::tmem_wait_st();
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) arrive_dq(slot);
      }
    } else {
      // After the transpose below, lane t holds column 8 (t & 3) + (t >> 2)
      // of the warp's 32, and byte b of its word the codes of rows 2b (high
      // nibble) and 2b + 1 (low nibble) of an 8-row group. The three rounds
      // swap 4-bit, 8-bit and 16-bit blocks with the lanes 4, 8 and 16 away;
      // which half a lane keeps follows bit s of its row index (t >> 2) ^ 1.
      const int rho = lane >> 2;
      tile_row = 32 * q + 8 * (lane & 3) + rho;
      const bool h0 = ((rho & 1) ^ 1) != 0;
      const uint32_t keep0 = h0 ? 0xf0f0f0f0u : 0x0f0f0f0fu;
      const uint32_t rot0 = h0 ? 28u : 4u;
      const uint32_t sel1 = ((rho >> 1) & 1) ? 0x3715u : 0x6240u;
      const uint32_t sel2 = ((rho >> 2) & 1) ? 0x3276u : 0x5410u;
      // the warp's 32 columns share one absmax block per weight row
      const int64_t kb = (r0 >> 6) + (q >> 1);
      const bool kb_ok = kb < p.nblk;
      float* ah = reinterpret_cast<float*>(smem + C::kOffAhat) + (warp - 2) * 64;
      const uint8_t* tab = smem + C::kOffLut + 4 * lane;
      const uint8_t* cq = smem + C::kOffCodes + q * 1024 + rho * 16 + (lane & 3) * 4;
      uint32_t a8v[2] = {0u, 0u};
      float s2v[2] = {0.0f, 0.0f};
      bool rok[2] = {false, false};
      // this lane computes the dequantized absmax of rows lane and lane + 32
      auto load_scales = [&](int i) {
        if (i >= nst) return;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int64_t n = static_cast<int64_t>(s_begin + i) * 64 + lane + 32 * h;
          rok[h] = kb_ok && n < p.N;
          if (rok[h]) {
            const int64_t bi = n * p.nblk + kb;
            a8v[h] = p.a8[bi];
            s2v[h] = p.s2[bi >> 8];
          }
        }
      };
      load_scales(grp);
      if (!tc::mbar_wait(lut_bar, 0)) fail(kRoleCompute);
      for (int i = grp; i < nst; i += kGroups) {
        const int slot = i % kStages;
        const uint32_t ph = (i / kStages) & 1;
        const float ah0 = rok[0] ? dequant_absmax(a8v[0], s2v[0]) : 0.0f;
        const float ah1 = rok[1] ? dequant_absmax(a8v[1], s2v[1]) : 0.0f;
        load_scales(i + kGroups);
        __syncwarp();                       // last stage's reads of ah are done
        ah[lane] = ah0;
        ah[lane + 32] = ah1;
        __syncwarp();
        bool go = !*abort_flag;
        if (go && !tc::mbar_wait(full_bar(slot), ph)) {
          fail(kRoleCompute);
          go = false;
        }
        if (!__all_sync(0xffffffffu, go)) continue;
        const uint8_t* cw = cq + slot * kCodesStageBytes;
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          uint32_t v[16];
#pragma unroll
          for (int g8 = 0; g8 < 4; ++g8) {
            const int i8 = 4 * hf + g8;     // rows 8 i8 .. 8 i8 + 7
            uint32_t x = *reinterpret_cast<const uint32_t*>(cw + 128 * i8);
            uint32_t y = __shfl_xor_sync(0xffffffffu, x, 4);
            x = (x & keep0) | (__funnelshift_l(y, y, rot0) & ~keep0);
            y = __shfl_xor_sync(0xffffffffu, x, 8);
            x = __byte_perm(x, y, sel1);
            y = __shfl_xor_sync(0xffffffffu, x, 16);
            x = __byte_perm(x, y, sel2);
            const float4 sa = *reinterpret_cast<const float4*>(ah + 8 * i8);
            const float4 sb = *reinterpret_cast<const float4*>(ah + 8 * i8 + 4);
            const float2 sc[4] = {make_float2(sa.x, sa.y), make_float2(sa.z, sa.w),
                                  make_float2(sb.x, sb.y), make_float2(sb.z, sb.w)};
#pragma unroll
            for (int b = 0; b < 4; ++b) {
              const uint32_t byte = __byte_perm(x, 0u, 0x4440u + b);
              const __half2 h2 = *reinterpret_cast<const __half2*>(tab + (byte << 7));
              const float2 lv = __fmul2_rn(__half22float2(h2), sc[b]);
              v[4 * g8 + b] = pack_bf16x2(lv.x, lv.y);
            }
          }
          tc::tmem_st16(tmem + lane_base + kTmemA0 + 32u * slot + 16u * hf, v);
        }
        tc::tmem_wait_st();
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) arrive_dq(slot);
      }
    }

    // epilogue: accumulator lanes are tile rows, columns are tokens; the
    // groups share out the 16-column chunks
    if (!*abort_flag && !tc::mbar_wait(accum_bar, 0)) fail(kRoleEpilogue);
    tc::fence_after_sync();
    if (!*abort_flag) {
      const int64_t rg = r0 + tile_row;
      const int64_t nd = kDx ? p.K : p.N;
      const bool vrow = rg < nd;
      for (int c = 16 * grp; c < p.bn; c += 16 * kGroups) {
        uint32_t v[16];
        tc::tmem_ld16(tmem + lane_base + static_cast<uint32_t>(c), v);
        tc::tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int64_t m = m0 + c + j;
          if (vrow && m < p.M) {
            float* dst = p.out + m * nd + rg;
            if (p.atomic_out) atomicAdd(dst, __uint_as_float(v[j]));
            else *dst = __uint_as_float(v[j]);
          }
        }
      }
    }
  }

  // On a pair, neither CTA frees its tensor memory or leaves (its barriers
  // take the peer's arrivals) before both are done.
  tc::fence_before_sync();
  if constexpr (kPair) tc::cluster_sync();
  else __syncthreads();
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc<kCg>(tmem, kTmemCols);
  }
}

template <bool kDx, int kBN>
cudaError_t launch_tc(const uint16_t* act, int64_t M, const uint8_t* codes, const uint8_t* a8,
                      const float* s2, int64_t N, int64_t K, float* out, int num_sms, int* status,
                      cudaStream_t st) {
  using C = Cfg<kDx, kBN>;
  TcArgs a;
  a.a8 = a8;
  a.s2 = s2;
  a.out = out;
  a.M = M;
  a.N = N;
  a.K = K;
  a.nblk = static_cast<int>(K / kBlock);
  a.status = status;
  a.bn = kBN;
  const int64_t nd = kDx ? K : N;            // tile-row dimension
  const int64_t red = kDx ? N : K;           // reduction dimension
  // a pair's two CTAs take consecutive 128-row tiles
  const int64_t tile_rows = kTileRows * C::kCg;
  const int64_t row_tiles = (nd + tile_rows - 1) / tile_rows * C::kCg;
  const int64_t m_tiles = (M + a.bn - 1) / a.bn;
  a.stages_total = static_cast<int>((red + 63) / 64);
  int splits = 1;
  const int64_t ctas = row_tiles * m_tiles;
  if (ctas < num_sms) {   // each split fills the ring at least once
    splits = static_cast<int>(std::max<int64_t>(
        1, std::min<int64_t>(num_sms / ctas, a.stages_total / C::kStages)));
  }
  a.stages_per_split = (a.stages_total + splits - 1) / splits;
  splits = (a.stages_total + a.stages_per_split - 1) / a.stages_per_split;
  a.atomic_out = splits > 1 ? 1 : 0;

  CUtensorMap tm_act, tm_codes;
  // activations: [M, red] bf16, box 64 (reduction) x the tokens one CTA
  // stages, 128-byte swizzle
  if (!encode_2d(&tm_act, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, act, static_cast<uint64_t>(red),
                 static_cast<uint64_t>(M), static_cast<uint64_t>(red) * 2, 64,
                 static_cast<uint32_t>(C::kBRows), CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  // packed codes: [N, K/2] bytes; the forward takes 32 B x 128 rows, the input
  // gradient 16 B (32 columns) x 64 rows per box
  if (!encode_2d(&tm_codes, CU_TENSOR_MAP_DATA_TYPE_UINT8, codes, static_cast<uint64_t>(K / 2),
                 static_cast<uint64_t>(N), static_cast<uint64_t>(K / 2), kDx ? 16 : 32,
                 kDx ? 64 : 128, CU_TENSOR_MAP_SWIZZLE_NONE))
    return cudaErrorInvalidValue;

  static std::once_flag once;
  std::call_once(once, [] {
    cudaFuncSetAttribute(tc_gemm_kernel<kDx, kBN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         C::kSmemBytes);
  });
  if (a.atomic_out) {
    cudaError_t e = cudaMemsetAsync(out, 0, static_cast<size_t>(M) * nd * sizeof(float), st);
    if (e != cudaSuccess) return e;
  }
  dim3 grid(static_cast<unsigned>(row_tiles), static_cast<unsigned>(m_tiles),
            static_cast<unsigned>(splits));
  if constexpr (C::kPair) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(C::kThreads);
    cfg.dynamicSmemBytes = C::kSmemBytes;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, tc_gemm_kernel<kDx, kBN>, tm_act, tm_codes, a);
  } else {
    tc_gemm_kernel<kDx, kBN><<<grid, C::kThreads, C::kSmemBytes, st>>>(tm_act, tm_codes, a);
    return cudaGetLastError();
  }
}

}  // namespace

cudaError_t launch_tc_fwd(const uint16_t* X, int64_t M, const uint8_t* codes, const uint8_t* a8,
                          const float* s2, int64_t N, int64_t K, float* Y, int num_sms,
                          int* status, cudaStream_t st) {
  if (M <= 64) return launch_tc<false, 64>(X, M, codes, a8, s2, N, K, Y, num_sms, status, st);
  if (M <= 128) return launch_tc<false, 128>(X, M, codes, a8, s2, N, K, Y, num_sms, status, st);
  return launch_tc<false, 256>(X, M, codes, a8, s2, N, K, Y, num_sms, status, st);
}

cudaError_t launch_tc_dx(const uint16_t* dY, int64_t M, const uint8_t* codes, const uint8_t* a8,
                         const float* s2, int64_t N, int64_t K, float* dX, int num_sms,
                         int* status, cudaStream_t st) {
  if (M <= 64) return launch_tc<true, 64>(dY, M, codes, a8, s2, N, K, dX, num_sms, status, st);
  if (M <= 128) return launch_tc<true, 128>(dY, M, codes, a8, s2, N, K, dX, num_sms, status, st);
  return launch_tc<true, 256>(dY, M, codes, a8, s2, N, K, dX, num_sms, status, st);
}

}  // namespace nf4
