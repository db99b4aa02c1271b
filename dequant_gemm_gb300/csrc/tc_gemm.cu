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
//   * warp 0 TMA-loads the stage's activation tile (bf16, 128-byte swizzle,
//     the K-major B operand) and its packed-code tile from one elected lane;
//   * the dequant warps, in four groups of four that take the stages in
//     turn, dequantize the codes (level * dequantized absmax, rounded to
//     bf16) into the stage's A operand;
//   * warp 1 issues tcgen05.mma (128 x BN x 16) from one elected lane into
//     an fp32 accumulator in tensor memory and commits each stage back to the
//     producer;
//   * the dequant warps then read the accumulator with tcgen05.ld and store
//     fp32 outputs (32 consecutive outputs of one token per warp store).
//
// Both directions walk the weight along its rows, one thread per (row, 64
// columns) run, which is one absmax block: both levels of a code byte come
// from one lookup in a 256-entry fp16 level pair table kept in 32
// lane-private copies (every lookup of a warp hits 32 distinct banks), are
// widened to fp32 and multiplied by the block's dequantized absmax, a
// register.
//
// Forward: the tile is 128 weight rows, the reduction runs along a row, so a
// thread's run is K-contiguous and goes straight into tensor memory (one
// lane per weight row), where the MMA reads its A operand: the dequantized
// weight never touches shared memory.
//
// Input gradient: the tile is 128 weight columns and the reduction runs down
// the columns. A = w^T is then M-major in the weight's own row order, so a
// thread's run is one 128-byte row of a 128-byte-swizzled MN-major atom (64
// columns x 8 rows) of an A tile in shared memory, read by the MMA through
// an MN-major descriptor: no transposition and no per-row scale exchange
// between lanes.
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
  static constexpr bool kPair = kBN == 256;
  static constexpr int kCg = kPair ? 2 : 1;          // tcgen05 cta_group
  // dequant warp groups: a group needs several MMA stage times per stage
  static constexpr int kGroups = 4;
  static constexpr int kDqWarps = 4 * kGroups;
  static constexpr int kThreads = 64 + 32 * kDqWarps;
  // The input gradient stages its A tile in shared memory as well, in a ring
  // of its own: one slot per dequant group, freed by the stage's MMAs, while
  // the copies run further ahead (a shared 5-deep ring left the MMA waiting
  // on copy latency plus dequant every stage).
  static constexpr int kAStageBytes = kDx ? kTileRows * 64 * 2 : 0;
  static constexpr int kStages = kDx ? (kBN == 64 ? 8 : 6) : (kBN == 64 ? 12 : 8);
  static constexpr int kASlots = kDx ? 4 : kStages;   // forward: the TMEM slot of the stage
  static constexpr int kBRows = kPair ? kBN / 2 : kBN;   // tokens staged per CTA
  static constexpr int kActStageBytes = kBRows * 128;    // 64 bf16 per token row
  static constexpr uint32_t kTmemA0 = kBN;
  // the forward's A slots follow the accumulator; the input gradient holds
  // only the accumulator (BN columns, a power of two >= 32)
  static constexpr uint32_t kTmemAlloc = kDx ? static_cast<uint32_t>(kBN) : kTmemCols;
  static constexpr int kLutBytes = kHalfPairTableBytes;
  static constexpr int kOffAct = 0;
  static constexpr int kOffA = kOffAct + kStages * kActStageBytes;   // 1 KB aligned
  static constexpr int kOffCodes = kOffA + kASlots * kAStageBytes;
  static constexpr int kOffLut = kOffCodes + kStages * kCodesStageBytes;
  static constexpr int kOffBars = kOffLut + kLutBytes;
  static constexpr int kNumBars = 2 * kStages + 2 * kASlots + 2;
  static constexpr int kOffMisc = kOffBars + kNumBars * 8;
  static constexpr int kSmemBytes = kOffMisc + 16 + 1024;   // + alignment slack
  static_assert(kDx || kTmemA0 + 32 * kStages <= kTmemCols, "tensor memory columns");
  static_assert(kOffA % 1024 == 0 && kOffCodes % 1024 == 0, "swizzled tiles");
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
  constexpr int kASlots = C::kASlots;
  // copy ring: full / empty per stage slot; A ring: dq (written) / afree
  // (read by the MMAs; input gradient only) per A slot
  auto full_bar = [&](int s) { return bars + 8u * s; };
  auto empty_bar = [&](int s) { return bars + 8u * (kStages + s); };
  auto dq_bar = [&](int a) { return bars + 8u * (2 * kStages + a); };
  auto afree_bar = [&](int a) { return bars + 8u * (2 * kStages + kASlots + a); };
  const uint32_t accum_bar = bars + 8u * (2 * kStages + 2 * kASlots);
  const uint32_t lut_bar = accum_bar + 8u;
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
      tc::mbar_init(empty_bar(s), 1);
    }
    for (int a = 0; a < kASlots; ++a) {
      // one arrival per warp of the stage's group, in both CTAs of a pair
      tc::mbar_init(dq_bar(a), 4 * kCg);
      tc::mbar_init(afree_bar(a), 1);
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
  if (warp == 1) tc::tmem_alloc<kCg>(tc::smem_addr(tmem_slot), C::kTmemAlloc);
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
    // Like the MMA loop, the whole warp runs it on warp-uniform values and
    // one elected lane issues the copies: from a one-thread branch a stage's
    // expect_tx and two tensor copies took ~500 cycles, which paced the whole
    // pipeline.
    const uint32_t tx = static_cast<uint32_t>(kActStageBytes + kCodesStageBytes);
    const int32_t m_load = static_cast<int32_t>(m0) + static_cast<int32_t>(rank) * C::kBRows;
    int issued = 0;
    for (int i = 0; i < nst; ++i) {
      // one vote, so that the lanes leave together (a lane-wise read of the
      // flag could split the warp ahead of the vote below)
      if (__any_sync(0xffffffffu, *abort_flag != 0)) break;
      const int slot = i % kStages;
      const uint32_t ph = (i / kStages) & 1;
      if (!__all_sync(0xffffffffu, tc::mbar_wait(empty_bar(slot), ph ^ 1))) {
        if (lane == 0) fail(kRoleProducer);
        break;
      }
      const int s = s_begin + i;
      const uint32_t act = tc::smem_addr(smem + C::kOffAct + slot * kActStageBytes);
      const uint32_t cod = tc::smem_addr(smem + C::kOffCodes + slot * kCodesStageBytes);
      if (tc::elect_one()) {
        tc::mbar_arrive_expect_tx(full_bar(slot), tx);
        tc::tma_load_2d(act, &tm_act, s * 64, m_load, full_bar(slot));
        if (!kDx) {
          // 128 rows x 32 bytes
          tc::tma_load_2d(cod, &tm_codes, s * 32, static_cast<int32_t>(r0), full_bar(slot));
        } else {
          // one 64-byte (128 columns) x 64-row box with the 64-byte swizzle:
          // row r's 16-byte chunk c lands at r * 64 + 16 * (c ^ ((r >> 1) & 3))
          tc::tma_load_2d(cod, &tm_codes, static_cast<int32_t>(r0 / 2), s * 64, full_bar(slot));
        }
      }
      __syncwarp();
      ++issued;
    }
    if (*abort_flag && lane == 0) {  // let copies in flight land before the CTA exits
      for (int i = max(0, issued - kStages); i < issued; ++i)
        tc::mbar_wait(full_bar(i % kStages), (i / kStages) & 1);
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
      const uint32_t idesc =
          tc::idesc_bf16_f32(kTileRows * kCg, static_cast<uint32_t>(p.bn), kDx);
      const uint64_t bdesc0 = tc::sw128_kmajor_desc(tc::smem_addr(smem + C::kOffAct));
      // input gradient: A tile atoms (column half h, row group g) at
      // (2 g + h) KB, i.e. 1 KB apart along M and 2 KB along K
      const uint64_t adesc0 = tc::sw128_mnmajor_desc(tc::smem_addr(smem + C::kOffA), 1024, 2048);
      for (int i = 0; i < nst; ++i) {
        const int sl = i % kStages;
        const int as = i % kASlots;
        const bool ok = tc::mbar_wait_spin<kPair>(dq_bar(as), (i / kASlots) & 1);
        if (!__all_sync(0xffffffffu, ok)) {
          if (lane == 0) fail(kRoleMma);
          break;
        }
        tc::fence_after_sync();
        const uint32_t a = tmem + kTmemA0 + 32u * sl;
        // the descriptor's start-address field counts 16-byte units
        const uint64_t bdesc = bdesc0 + static_cast<uint64_t>(sl * (kActStageBytes >> 4));
        const uint64_t adesc = adesc0 + static_cast<uint64_t>(as * (C::kAStageBytes >> 4));
        if (tc::elect_one()) {
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            if constexpr (kDx)   // K rows 16 j .. 16 j + 15: row groups 2 j, 2 j + 1
              tc::mma_bf16_ss<kCg>(tmem, adesc + 256u * j, bdesc + 2u * j, idesc,
                                   (i | j) != 0 ? 1u : 0u);
            else
              tc::mma_bf16_tmem_a<kCg>(tmem, a + 8u * j, bdesc + 2u * j, idesc,
                                       (i | j) != 0 ? 1u : 0u);
          }
          tc::mma_commit<kCg>(empty_bar(sl));
          if constexpr (kDx) tc::mma_commit<kCg>(afree_bar(as));
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
    auto arrive_dq = [&](int a) {
      if constexpr (kPair) tc::mbar_arrive_remote(tc::mapa(dq_bar(a), 0));
      else tc::mbar_arrive(dq_bar(a));
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
      // Thread t of the group dequantizes weight row t % 64 of the stage over
      // the tile's columns 64 (t / 64) .. + 63, one absmax block, as the
      // forward walks a row. The 64 bf16 results are one 128-byte row of a
      // 128-byte-swizzled MN-major atom of the A tile (64 weight columns along
      // M x 8 weight rows along K per 1 KB atom; atom (column half h, row
      // group g) at (2 g + h) KB).
      const int t = ((warp - 2) & 3) * 32 + lane;
      const int rr = t & 63, h = t >> 6;
      const int64_t kb = (r0 >> 6) + h;
      const bool kb_ok = kb < p.nblk;
      const uint8_t* tab = smem + C::kOffLut + 4 * lane;
      // 16-byte code chunks 2 h and 2 h + 1 of row rr (64-byte swizzle)
      const int csw = (rr >> 1) & 3;
      const int co0 = rr * 64 + 16 * ((2 * h) ^ csw), co1 = rr * 64 + 16 * ((2 * h + 1) ^ csw);
      const int ao = (2 * (rr >> 3) + h) * 1024 + (rr & 7) * 128;
      const int asw = rr & 7;
      uint32_t a8v = 0;
      float s2v = 0.0f;
      bool rok = false;
      auto load_scale = [&](int i) {
        if (i >= nst) return;
        const int64_t n = static_cast<int64_t>(s_begin + i) * 64 + rr;
        rok = kb_ok && n < p.N;
        if (rok) {
          const int64_t bi = n * p.nblk + kb;
          a8v = p.a8[bi];
          s2v = p.s2[bi >> 8];
        }
      };
      load_scale(grp);
      if (!tc::mbar_wait(lut_bar, 0)) fail(kRoleCompute);
      for (int i = grp; i < nst; i += kGroups) {
        const int slot = i % kStages;
        const uint32_t ph = (i / kStages) & 1;
        const float ahat = rok ? dequant_absmax(a8v, s2v) : 0.0f;
        const float2 ahat2 = make_float2(ahat, ahat);
        load_scale(i + kGroups);
        bool go = !*abort_flag;
        if (go && !tc::mbar_wait(full_bar(slot), ph)) {
          fail(kRoleCompute);
          go = false;
        }
        // the A slot's previous tile (stage i - kASlots) has been read by its MMAs
        const int as = i % kASlots;
        if (go && i >= kASlots && !tc::mbar_wait(afree_bar(as), ((i / kASlots) - 1) & 1)) {
          fail(kRoleCompute);
          go = false;
        }
        if (!__all_sync(0xffffffffu, go)) continue;
        const uint8_t* cst = smem + C::kOffCodes + slot * kCodesStageBytes;
        uint8_t* arow = smem + C::kOffA + as * C::kAStageBytes + ao;
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          const uint4 c = *reinterpret_cast<const uint4*>(cst + (hf ? co1 : co0));
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
          // columns 32 hf + 8 j .. + 7 form chunk 4 hf + j of the atom row
#pragma unroll
          for (int j = 0; j < 4; ++j)
            *reinterpret_cast<uint4*>(arow + 16 * ((4 * hf + j) ^ asw)) =
                make_uint4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
        }
        tc::fence_proxy_async();   // the MMA reads the tile through the async proxy
        __syncwarp();
        if (lane == 0) arrive_dq(as);
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
    tc::tmem_dealloc<kCg>(tmem, C::kTmemAlloc);
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
  // gradient 64 B (128 columns) x 64 rows, 64-byte swizzled
  if (!encode_2d(&tm_codes, CU_TENSOR_MAP_DATA_TYPE_UINT8, codes, static_cast<uint64_t>(K / 2),
                 static_cast<uint64_t>(N), static_cast<uint64_t>(K / 2), kDx ? 64 : 32,
                 kDx ? 64 : 128, kDx ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_NONE))
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
