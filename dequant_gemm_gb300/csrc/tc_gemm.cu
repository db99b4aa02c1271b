// Large-M fused dequant matmuls on the sm_103a tensor cores (tcgen05):
//   forward   Y[m, n]  = sum_k X[m, k]  * w[n, k]
//   input grad dX[m, k] = sum_n dY[m, n] * w[n, k]      (no dW)
// ("Zenbit", zenbit.pallas_nf4 bullet: compressed weight tiles streamed in and
// dequantized on chip, full-precision weight never in HBM; dL/dX only.)
// Weights are NF4 or FP4 (4-bit codes, double-quantized absmax) or int8 with
// an fp32 absmax per block; activations bf16 or fp16 (the dequantized weight
// then enters the MMA in the same type); outputs fp32 or bf16, overwritten or
// added to ("bitsandbytes", quantized-GEMM and 4-bit paragraphs).
//
// The kernel is persistent: a CTA (or CTA pair) takes the output tile units
// c, c + G, c + 2G, ... of the launch (G = the number of CTAs or pairs, at
// most one per SM). A unit is a 128 x BN tile of D = A * B^T with the weight
// as the 128-row A operand and the tokens as the BN-column B operand (BN =
// 64, 128 or 256; 256 on CTA pairs that share one 256 x 256 MMA) over one
// reduction range, walked in stages of 64. One stage counter runs across the
// units, so the copy ring, the A slots and the dequant groups never restart:
//   * warp 0 TMA-loads the stage's activation tile (16-bit, 128-byte swizzle,
//     the K-major B operand) and its code tile from one elected lane;
//   * warps 2-17, in four groups of four that take the stages in turn,
//     dequantize the codes (level * dequantized absmax, rounded to the
//     activation type) into the stage's A operand;
//   * warp 1 issues tcgen05.mma (128 x BN x 16) from one elected lane into
//     an fp32 accumulator in tensor memory, commits each stage back to the
//     producer and each unit to the epilogue;
//   * warps 18-21 read a finished accumulator with tcgen05.ld and store the
//     outputs while the MMAs of the next unit run into the other of two
//     accumulator buffers. Where there is one accumulator only (the forward
//     at BN = 256, whose A operand slots take the other half of tensor
//     memory, and BN = 64, whose short units leave 4 warps too little time),
//     the dequant warps drain it between units instead, as the copies of the
//     next unit are already under way.
//
// Both directions walk the weight along its rows, one thread per (row, 64
// columns) run, which is one absmax block. Forward: a 4-bit code byte gives
// both levels from one 8-byte lookup in a 256-entry fp32 level pair table
// kept in 16 copies (each half-warp's lookups hit 32 distinct banks;
// measured 1% faster than fp16 pairs in 32 copies, which need widening, and
// the levels are then exact), multiplied in fp32 by the block's dequantized
// absmax, a register, and rounded to the operand type. Input gradient: the
// thread first scales and rounds the 16 levels for its run the same way and
// keeps them as byte planes in 8 registers, from which byte permutes pick
// the operands: no shared-memory lookups, whose wavefronts there compete
// with the A-tile stores and the tensor core's operand reads (7% faster
// alone, 5% in the decoder layer; the forward, with A in tensor memory,
// measured 2.5% slower with planes and keeps the table). Both give the same
// operand bits. An int8 byte is converted directly and scaled by absmax / 127.
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
// When the output tiles alone cannot fill the GPU, or (forward) leave the
// persistent grid a partial last round (112 tiles on 76 pairs run two
// rounds, the second 47% full; split in two, 224 half-length units run three
// full ones), and the output is fp32, the reduction is split across units
// and summed with atomics into a zeroed (or, accumulating, the caller's)
// output. A bf16 output is never split.
//
// Every mbarrier wait is bounded; a CTA that gives up records a timeout in the
// device status word and raises an abort flag (its own and, on a pair, the
// peer's); every role then stops at its next wait, the copies and MMAs in
// flight are waited for, and the tensor memory is freed before the CTA exits.
#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "tc.cuh"

namespace nf4 {
namespace {

constexpr int kTileRows = 128;               // MMA M
constexpr uint32_t kTmemCols = 512;

// Per-direction, per-token-tile and per-format configuration and shared-memory
// layout. The token tile BN (MMA N) sets the stage size; smaller tiles get
// deeper rings, so that enough code bytes are in flight per SM to cover the
// memory latency. Tensor memory holds the accumulator buffers (BN fp32
// columns each), then (forward) one 32-column A-operand slot per stage.
//
// The BN = 256 tiles run on CTA pairs (cta_group::2): the two CTAs of a
// cluster hold 128 weight rows (columns) each, and half of the token tile
// each; the MMA warp of the even CTA issues 256 x 256 x 16 MMAs over both
// SMs. Each SM then stages and reads only half of the activation tile, which
// is most of the shared-memory traffic of a stage. The dequant and epilogue
// warps of both CTAs arrive on the issuing CTA's barriers. The arrival takes
// the instruction's default (CTA-scope) release: by then the warp's
// tensor-memory accesses have retired and the stage's copies have been seen
// complete, and a cluster-scope release was measured to stall the arriving
// thread for 1-2.5K cycles on a busy SM, enough to halve the MMA rate.
template <bool kDx, int kBN, bool kInt8>
struct Cfg {
  static constexpr bool kPair = kBN == 256;
  static constexpr int kCg = kPair ? 2 : 1;          // tcgen05 cta_group
  // 16 dequant warps in 4 groups of 4 that take the stages in turn (measured:
  // 2 groups of 8 splitting each stage, 8-12% slower)
  static constexpr int kDqWarps = 16;
  static constexpr int kGroups = 4;
  // code bytes of a stage: 128 weight rows (forward) or 64 weight rows of 128
  // columns (input gradient) x 64 weights, at 4 or 8 bits
  static constexpr int kCodesStageBytes = kInt8 ? 8192 : 4096;
  // The input gradient stages its A tile in shared memory as well, in a ring
  // of its own: one slot per dequant group, freed by the stage's MMAs, while
  // the copies run further ahead (a shared 5-deep ring left the MMA waiting
  // on copy latency plus dequant every stage).
  static constexpr int kAStageBytes = kDx ? kTileRows * 64 * 2 : 0;
  // (the 4-bit input gradient takes a seventh copy slot in the space the
  // level table no longer uses: 0-1% faster)
  static constexpr int kStages = kDx ? (kBN == 64 ? 8 : kInt8 ? 6 : 7) : (kBN == 64 ? 12 : 8);
  static constexpr int kASlots = kDx ? 4 : kStages;   // forward: the TMEM slot of the stage
  static constexpr int kBRows = kPair ? kBN / 2 : kBN;   // tokens staged per CTA
  static constexpr int kActStageBytes = kBRows * 128;    // 64 16-bit values per token row
  // Two accumulator buffers where they fit next to the forward's A slots,
  // and where a unit is long enough for 4 epilogue warps to drain one while
  // the next fills the other: at BN = 64 (short, often split units whose
  // outputs go out as atomics) the 16 dequant warps drain a single buffer
  // between units instead (4 epilogue warps there measured 13% slower).
  static constexpr int kAccBufs = kBN >= 128 && 2 * kBN + (kDx ? 0 : 32 * kStages) <= 512 ? 2 : 1;
  // With two buffers, 4 epilogue warps, one per tensor-memory lane quarter
  // (22 warps leave 80 registers a thread; 18, without them, 96).
  static constexpr int kEpiWarps = kAccBufs == 2 ? 4 : 0;
  static constexpr int kFirstEpiWarp = 2 + kDqWarps;
  static constexpr int kThreads = 32 * (2 + kDqWarps + kEpiWarps);
  static constexpr uint32_t kTmemA0 = kAccBufs * kBN;
  // the input gradient holds only the accumulators (a power of two >= 32)
  static constexpr uint32_t kTmemAlloc = kDx ? static_cast<uint32_t>(kAccBufs * kBN) : kTmemCols;
  // arrivals that free an accumulator buffer: the epilogue warps, or with a
  // single buffer the dequant warps that drain it, of both CTAs of a pair
  static constexpr int kDrainWarps = kAccBufs == 2 ? kEpiWarps : kDqWarps;
  // 4-bit operands from per-run byte planes in registers (the 16 fp32 levels
  // in shared memory) instead of the pair table: the input gradient only
  static constexpr bool kPlanes = kDx && !kInt8;
  static constexpr int kLutBytes = kInt8 ? 0 : kPlanes ? 128 : kPairTableBytes;
  static constexpr int kOffAct = 0;
  static constexpr int kOffA = kOffAct + kStages * kActStageBytes;   // 1 KB aligned
  static constexpr int kOffCodes = kOffA + kASlots * kAStageBytes;
  static constexpr int kOffLut = kOffCodes + kStages * kCodesStageBytes;
  static constexpr int kOffBars = kOffLut + kLutBytes;
  // full, empty per stage; dq, afree per A slot; accumulator full, empty per
  // buffer; the level table; the final drain
  static constexpr int kNumBars = 2 * kStages + 2 * kASlots + 4 + 2;
  static constexpr int kOffMisc = kOffBars + kNumBars * 8;
  // epilogue staging: one 16-token x 32-row fp32 box per draining warp,
  // written out by TMA (not at 64 tokens, whose drains stay plain stores:
  // the boxes' 32 KB there cost more than the copy engine gained, 1.5%)
  static constexpr int kStageWarps = kBN == 64 ? 0 : kAccBufs == 2 ? kEpiWarps : kDqWarps;
  static constexpr int kStageBoxBytes = 16 * 32 * 4;
  static constexpr int kOffStage = (kOffMisc + 16 + 127) & ~127;
  static constexpr int kSmemBytes = kOffStage + kStageWarps * kStageBoxBytes + 1024;   // + slack
  static_assert(kDx || kTmemA0 + 32 * kStages <= kTmemCols, "tensor memory columns");
  static_assert(kOffA % 1024 == 0 && kOffCodes % 1024 == 0, "swizzled tiles");
  static_assert(kBN == 64 || kBN == 128 || kBN == 256, "token tile");
  static_assert(kSmemBytes <= 227 * 1024, "shared memory");
  // Every mbarrier a dequant group waits on with a parity test must not be
  // able to run a phase behind the one the group expects (the test cannot
  // tell them apart; a variant with 3 A slots for 4 groups deadlocked on
  // exactly that). Each A slot is therefore waited by one group only, in
  // order; the forward's copy slots likewise; the input gradient's copy
  // slots, shared between groups, are waited on only after the A slot,
  // which orders them (kStages >= kASlots).
  static_assert(kASlots % kGroups == 0, "A slots per dequant group");
  static_assert(kDx ? kStages >= kASlots : kStages % kGroups == 0, "copy slots per dequant group");
};

struct TcArgs {
  const uint8_t* a8;       // 4-bit formats: absmax codes
  const float* scale;      // 4-bit formats: s2 per group; int8: absmax per block
  void* out;               // Y [M, N] or dX [M, K], fp32 or bf16
  int64_t M, N, K;
  int nblk;                // K / 64
  int bn;                  // token tile
  int fmt;                 // 4-bit table: kFmtNf4 or kFmtFp4
  int stages_total;        // reduction stages of the whole product
  int stages_per_split;
  int row_units;           // tile units along the rows (one per CTA or pair)
  int m_tiles;             // token tiles
  int units;               // row_units * m_tiles * splits
  int atomic_out;
  int out_bf16;
  int accumulate;
  int out_mode;            // 0: TMA store; 1: TMA add (fp32, split or accumulating); 2: plain stores
  long long mma_wait_limit;
  int* status;
};

// One tile unit as a CTA sees it.
struct Unit {
  int64_t r0;              // first tile row (weight row or column) of this CTA
  int64_t m0;              // first token
  int s_begin, nst;        // reduction stages
};

// Level pair tables of the 4-bit formats: the fp32 levels of both nibbles
// of every code byte (the even element's level first), in 16 copies: entry
// (byte b, copy c) at (16 b + c) * 8 bytes.
struct FloatPairTable { uint32_t w[256 * 16 * 2]; };
constexpr FloatPairTable make_float_pair_table(int fmt) {
  FloatPairTable t{};
  const uint32_t (&lv)[16] = level_bits(fmt);
  for (int b = 0; b < 256; ++b)
    for (int c = 0; c < 16; ++c) {
      t.w[(b * 16 + c) * 2] = lv[b >> 4];
      t.w[(b * 16 + c) * 2 + 1] = lv[b & 15];
    }
  return t;
}
static_assert(sizeof(FloatPairTable) == kPairTableBytes, "table size");
__device__ __align__(128) const FloatPairTable kPairsNf4 = make_float_pair_table(kFmtNf4);
__device__ __align__(128) const FloatPairTable kPairsFp4 = make_float_pair_table(kFmtFp4);

__device__ __forceinline__ void bulk_copy_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                              uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
      : "memory");
}

// Two fp32 values rounded to the MMA operand type (bf16 or fp16), packed.
template <bool kF16>
__device__ __forceinline__ uint32_t pack_operand(float lo, float hi) {
  if constexpr (kF16) {
    const __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&v);
  } else {
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&v);
  }
}

// 16 code bytes of a 4-bit format (32 weights) -> 16 packed operand words.
// tab is this lane's copy of the level pair table (copy lane % 16; entries
// 128 bytes apart).
template <bool kF16>
__device__ __forceinline__ void dequant16_4bit(const uint4 c, const uint8_t* tab, float2 ahat2,
                                               uint32_t (&v)[16]) {
  const uint32_t words[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const uint32_t byte = __byte_perm(words[j], 0u, 0x4440u + b);
      const float2 lv = __fmul2_rn(*reinterpret_cast<const float2*>(tab + (byte << 7)), ahat2);
      v[4 * j + b] = pack_operand<kF16>(lv.x, lv.y);
    }
  }
}

// The 16 levels of a 4-bit format times one block's scale, rounded to the
// operand type, as byte planes: lo[q] holds the low bytes of levels 4 q ..
// 4 q + 3 (level 4 q in byte 0), hi[q] their high bytes. The products and
// roundings are those of the pair-table path, so the operands are the same.
template <bool kF16>
__device__ __forceinline__ void level_planes(const float* lev, float ahat, uint32_t (&lo)[4],
                                             uint32_t (&hi)[4]) {
  const float4* l4 = reinterpret_cast<const float4*>(lev);
  const float2 a2 = make_float2(ahat, ahat);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const float4 l = l4[q];
    const float2 p0 = __fmul2_rn(make_float2(l.x, l.y), a2);
    const float2 p1 = __fmul2_rn(make_float2(l.z, l.w), a2);
    const uint32_t w0 = pack_operand<kF16>(p0.x, p0.y), w1 = pack_operand<kF16>(p1.x, p1.y);
    lo[q] = __byte_perm(w0, w1, 0x6420u);
    hi[q] = __byte_perm(w0, w1, 0x7531u);
  }
}

// 16 code bytes (32 weights) -> 16 packed operand words from the byte planes
// of one block's scaled levels. Per 16-bit half of a code word (four codes),
// a byte permute indexed by the codes' low three bits picks among levels 0-7,
// a second among levels 8-15, and a third between the two by bit 3, for the
// low and the high bytes alike; two more interleave low and high bytes into
// operand pairs, the high nibble of a byte (the even element) in the low half.
template <bool kF16>
__device__ __forceinline__ void dequant16_4bit_planes(const uint4 c, const uint32_t (&lo)[4],
                                                      const uint32_t (&hi)[4], uint32_t (&v)[16]) {
  const uint32_t words[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t m = words[j] & 0x77777777u;
    const uint32_t s = ((words[j] >> 1) & 0x44444444u) | 0x32103210u;
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
      const uint32_t mh = m >> (16 * hf), sh = s >> (16 * hf);
      const uint32_t l =
          __byte_perm(__byte_perm(lo[0], lo[1], mh), __byte_perm(lo[2], lo[3], mh), sh);
      const uint32_t h =
          __byte_perm(__byte_perm(hi[0], hi[1], mh), __byte_perm(hi[2], hi[3], mh), sh);
      v[4 * j + 2 * hf] = __byte_perm(l, h, 0x4051u);
      v[4 * j + 2 * hf + 1] = __byte_perm(l, h, 0x6273u);
    }
  }
}

// 16 int8 weights -> 8 packed operand words.
template <bool kF16>
__device__ __forceinline__ void dequant16_int8(const uint4 c, float2 ahat2, uint32_t* v) {
  const uint32_t words[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t w = words[j];
    const float2 p0 = make_float2(static_cast<float>(static_cast<int8_t>(w & 0xffu)),
                                  static_cast<float>(static_cast<int8_t>((w >> 8) & 0xffu)));
    const float2 p1 = make_float2(static_cast<float>(static_cast<int8_t>((w >> 16) & 0xffu)),
                                  static_cast<float>(static_cast<int8_t>(w >> 24)));
    const float2 l0 = __fmul2_rn(p0, ahat2), l1 = __fmul2_rn(p1, ahat2);
    v[2 * j] = pack_operand<kF16>(l0.x, l0.y);
    v[2 * j + 1] = pack_operand<kF16>(l1.x, l1.y);
  }
}

// One output element: out[i] = v (+ out[i] with accumulate), fp32 or bf16.
__device__ __forceinline__ void store_out(void* out, int64_t i, float v, int out_bf16,
                                          int accumulate) {
  if (out_bf16) {
    __nv_bfloat16* y = reinterpret_cast<__nv_bfloat16*>(out) + i;
    if (accumulate) v += __bfloat162float(*y);
    *y = __float2bfloat16_rn(v);
  } else {
    float* y = reinterpret_cast<float*>(out) + i;
    if (accumulate) v += *y;
    *y = v;
  }
}

// The first nm of 16 consecutive tokens' outputs of one tile row (stride nd),
// bf16 or accumulating. Kept out of line: its registers would otherwise
// count against the whole kernel's budget of 80 or 96 a thread.
__device__ __noinline__ void store_out16(void* out, int64_t i0, int64_t nd, int nm, uint4 a,
                                         uint4 b, uint4 c, uint4 d, int out_bf16,
                                         int accumulate) {
  const uint32_t v[16] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w,
                          c.x, c.y, c.z, c.w, d.x, d.y, d.z, d.w};
#pragma unroll
  for (int j = 0; j < 16; ++j)
    if (j < nm) store_out(out, i0 + j * nd, __uint_as_float(v[j]), out_bf16, accumulate);
}

template <bool kDx, int kBN, bool kF16, bool kInt8>
__global__ void __launch_bounds__(Cfg<kDx, kBN, kInt8>::kThreads, 1)
tc_gemm_kernel(const __grid_constant__ CUtensorMap tm_act, const __grid_constant__ CUtensorMap tm_codes,
               const __grid_constant__ CUtensorMap tm_out, const TcArgs p) {
  using C = Cfg<kDx, kBN, kInt8>;
  constexpr bool kPair = C::kPair;
  constexpr int kCg = C::kCg;
  constexpr int kStages = C::kStages;
  constexpr int kASlots = C::kASlots;
  constexpr int kGroups = C::kGroups;
  constexpr int kAccBufs = C::kAccBufs;
  constexpr int kActStageBytes = C::kActStageBytes;
  constexpr int kCodesStageBytes = C::kCodesStageBytes;
  constexpr uint32_t kTmemA0 = C::kTmemA0;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t bars = tc::smem_addr(smem + C::kOffBars);
  // copy ring: full / empty per stage slot; A ring: dq (written) / afree
  // (read by the MMAs; input gradient only) per A slot; accumulator buffers:
  // accf (all MMAs of a unit done) / acce (drained by the epilogue)
  auto full_bar = [&](int s) { return bars + 8u * s; };
  auto empty_bar = [&](int s) { return bars + 8u * (kStages + s); };
  auto dq_bar = [&](int a) { return bars + 8u * (2 * kStages + a); };
  auto afree_bar = [&](int a) { return bars + 8u * (2 * kStages + kASlots + a); };
  auto accf_bar = [&](int b) { return bars + 8u * (2 * kStages + 2 * kASlots + b); };
  auto acce_bar = [&](int b) { return bars + 8u * (2 * kStages + 2 * kASlots + 2 + b); };
  const uint32_t lut_bar = bars + 8u * (2 * kStages + 2 * kASlots + 4);
  const uint32_t drain_bar = lut_bar + 8u;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // A pair is the cluster (2, 1, 1): its CTAs hold rows 128 (2 r + rank) of
  // a unit's 256, the token half rank of the tile, and rank 0 issues the MMAs.
  const uint32_t rank = kPair ? tc::cluster_ctarank() : 0u;
  const int cid = kPair ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
  const int ncl = kPair ? static_cast<int>(gridDim.x >> 1) : static_cast<int>(gridDim.x);
  // unit u: row unit fastest, then token tile, then reduction split
  auto unit_at = [&](int u) {
    Unit t;
    const int rt = u % p.row_units, rest = u / p.row_units;
    const int mt = rest % p.m_tiles, sp = rest / p.m_tiles;
    t.r0 = (static_cast<int64_t>(rt) * kCg + rank) * kTileRows;
    t.m0 = static_cast<int64_t>(mt) * p.bn;
    t.s_begin = sp * p.stages_per_split;
    t.nst = min(p.stages_per_split, p.stages_total - t.s_begin);
    return t;
  };

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
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(accf_bar(b), 1);
      tc::mbar_init(acce_bar(b), C::kDrainWarps * kCg);
    }
    tc::mbar_init(lut_bar, 1);
    tc::mbar_init(drain_bar, 1);
    *abort_flag = 0;
    tc::fence_barrier_init();
    if constexpr (C::kPlanes) {
      // level i is the first of the pair of byte 16 i (copy 0)
      const FloatPairTable* lut = p.fmt == kFmtFp4 ? &kPairsFp4 : &kPairsNf4;
      float* lev = reinterpret_cast<float*>(smem + C::kOffLut);
#pragma unroll
      for (int i = 0; i < 16; ++i) lev[i] = __uint_as_float(lut->w[i * 16 * 16 * 2]);
      tc::mbar_arrive(lut_bar);
    } else if constexpr (!kInt8) {
      const FloatPairTable* lut = p.fmt == kFmtFp4 ? &kPairsFp4 : &kPairsNf4;
      tc::mbar_arrive_expect_tx(lut_bar, C::kLutBytes);
      bulk_copy_g2s(tc::smem_addr(smem + C::kOffLut), lut, C::kLutBytes, lut_bar);
    }
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

  // A failure stops this CTA and, on a pair, the peer (whose barriers wait on
  // this CTA's MMAs or arrivals).
  auto fail = [&](uint32_t role) {
    report_status(p.status, kStatusTimeout, kDx ? kSiteTcDx : kSiteTcFwd, role);
    *abort_flag = 1;
    if constexpr (kPair) {
      const uint32_t peer = tc::mapa(tc::smem_addr(const_cast<int*>(abort_flag)), rank ^ 1u);
      asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(peer), "r"(1u) : "memory");
    }
  };
  // a wait that gave up because of a failure elsewhere is not a failure of its own
  auto waited = [&](int r, uint32_t role) {
    if (r == tc::kWaitTimeout) fail(role);
    return r == tc::kWaitDone;
  };
  // an arrival that frees accumulator buffer b (on the issuing CTA of a pair)
  auto arrive_acce = [&](int b) {
    if constexpr (kPair) tc::mbar_arrive_remote(tc::mapa(acce_bar(b), 0));
    else tc::mbar_arrive(acce_bar(b));
  };
  const int q = warp & 3;                      // TMEM lane quarter of this warp
  const uint32_t lane_base = static_cast<uint32_t>(32 * q) << 16;
  // tile row (forward: weight row; input gradient: weight column) held by
  // this thread's accumulator lane
  const int tile_row = 32 * q + lane;

  // Drain accumulator buffer b of unit t (16-column chunks c0, c0 + step, ...
  // of this warp's lane quarter) into the outputs. The TMA modes stage each
  // chunk (16 tokens x the quarter's 32 rows) in the warp's shared-memory
  // box and let one lane store (or add) it: the warp goes on while the copy
  // engine writes, rather than holding its stores in flight, and rows or
  // tokens past the output's end are dropped by the copy.
  const int stage_slot =
      C::kStageWarps > 0 ? max(0, warp - (kAccBufs == 2 ? C::kFirstEpiWarp : 2)) % C::kStageWarps : 0;
  uint8_t* stage_box = smem + C::kOffStage + stage_slot * C::kStageBoxBytes;
  const uint32_t stage_addr = tc::smem_addr(stage_box);
  auto drain = [&](const Unit& t, int b, int c0, int step) {
    const int64_t rg = t.r0 + tile_row;
    const int64_t nd = kDx ? p.K : p.N;
    const bool vrow = rg < nd;
    for (int c = c0; c < p.bn; c += step) {
      uint32_t v[16];
      tc::tmem_ld16(tmem + lane_base + static_cast<uint32_t>(b * kBN + c), v);
      tc::tmem_wait_ld();
      if (p.out_mode != 2) {
        // the box's previous contents have been read by their copy
        if (lane == 0) tc::bulk_wait_read_all();
        __syncwarp();
        if (p.out_bf16) {
          __nv_bfloat16* sb = reinterpret_cast<__nv_bfloat16*>(stage_box);
#pragma unroll
          for (int j = 0; j < 16; ++j) sb[j * 32 + lane] = __float2bfloat16_rn(__uint_as_float(v[j]));
        } else {
          float* sf = reinterpret_cast<float*>(stage_box);
#pragma unroll
          for (int j = 0; j < 16; ++j) sf[j * 32 + lane] = __uint_as_float(v[j]);
        }
        tc::fence_proxy_async();
        __syncwarp();
        if (lane == 0) {
          const int32_t x = static_cast<int32_t>(t.r0 + 32 * q);
          const int32_t y = static_cast<int32_t>(t.m0 + c);
          if (p.out_mode == 0) tc::tma_store_2d(&tm_out, stage_addr, x, y);
          else tc::tma_reduce_add_2d(&tm_out, stage_addr, x, y);
          tc::bulk_commit();
        }
        continue;
      }
      // one output mode per launch: the branch stays outside the stores
      const int nm = vrow ? static_cast<int>(min(static_cast<int64_t>(16), p.M - (t.m0 + c))) : 0;
      float* of = reinterpret_cast<float*>(p.out) + (t.m0 + c) * nd + rg;
      if (p.atomic_out) {
#pragma unroll
        for (int j = 0; j < 16; ++j)
          if (j < nm) atomicAdd(of + j * nd, __uint_as_float(v[j]));
      } else if (!p.out_bf16 && !p.accumulate) {
#pragma unroll
        for (int j = 0; j < 16; ++j)
          if (j < nm) of[j * nd] = __uint_as_float(v[j]);
      } else if (!p.accumulate) {
        __nv_bfloat16* ob = reinterpret_cast<__nv_bfloat16*>(p.out) + (t.m0 + c) * nd + rg;
#pragma unroll
        for (int j = 0; j < 16; ++j)
          if (j < nm) ob[j * nd] = __float2bfloat16_rn(__uint_as_float(v[j]));
      } else {
        store_out16(p.out, (t.m0 + c) * nd + rg, nd, nm, make_uint4(v[0], v[1], v[2], v[3]),
                    make_uint4(v[4], v[5], v[6], v[7]), make_uint4(v[8], v[9], v[10], v[11]),
                    make_uint4(v[12], v[13], v[14], v[15]), p.out_bf16, p.accumulate);
      }
    }
  };

  if (warp == 0) {
    // ------------------------------------------------------------ producer --
    // Like the MMA loop, the whole warp runs it on warp-uniform values and
    // one elected lane issues the copies: from a one-thread branch a stage's
    // expect_tx and two tensor copies took ~500 cycles, which paced the whole
    // pipeline. The ring runs on across units.
    const uint32_t tx = static_cast<uint32_t>(kActStageBytes + kCodesStageBytes);
    int gs = 0;                    // stages issued (across units)
    int slot = 0;                  // gs % kStages
    uint32_t ph = 0;               // (gs / kStages) & 1
    bool stop = false;
    for (int u = cid; u < p.units && !stop; u += ncl) {
      const Unit t = unit_at(u);
      const int32_t m_load = static_cast<int32_t>(t.m0) + static_cast<int32_t>(rank) * C::kBRows;
      for (int i = 0; i < t.nst; ++i, ++gs) {
        // one vote, so that the lanes leave together
        if (__any_sync(0xffffffffu, *abort_flag != 0)) { stop = true; break; }
        // every lane waits (a wait in lane 0 alone, the others parked at the
        // shuffle, was measured 4% slower on the prefill forward: the warp
        // reconverged late after each stage), then lane 0's outcome decides
        int r = tc::mbar_wait_abortable(empty_bar(slot), ph ^ 1, abort_flag);
        r = __shfl_sync(0xffffffffu, r, 0);
        if (r != tc::kWaitDone) {
          if (lane == 0 && r == tc::kWaitTimeout) fail(kRoleProducer);
          stop = true;
          break;
        }
        const int s = t.s_begin + i;
        const uint32_t act = tc::smem_addr(smem + C::kOffAct + slot * kActStageBytes);
        const uint32_t cod = tc::smem_addr(smem + C::kOffCodes + slot * kCodesStageBytes);
        if (tc::elect_one()) {
          tc::mbar_arrive_expect_tx(full_bar(slot), tx);
          tc::tma_load_2d(act, &tm_act, s * 64, m_load, full_bar(slot));
          if (!kDx) {
            // 128 rows x 32 (4-bit) or 64 (int8) bytes
            tc::tma_load_2d(cod, &tm_codes, s * (kInt8 ? 64 : 32), static_cast<int32_t>(t.r0),
                            full_bar(slot));
          } else {
            // 128 columns x 64 rows: 64 bytes with the 64-byte swizzle (4-bit,
            // row r's 16-byte chunk c at r * 64 + 16 * (c ^ ((r >> 1) & 3))) or
            // 128 bytes with the 128-byte swizzle (int8, chunk c at
            // r * 128 + 16 * (c ^ (r & 7)))
            tc::tma_load_2d(cod, &tm_codes, static_cast<int32_t>(kInt8 ? t.r0 : t.r0 / 2), s * 64,
                            full_bar(slot));
          }
        }
        __syncwarp();
        if (++slot == kStages) {
          slot = 0;
          ph ^= 1u;
        }
      }
    }
    if (*abort_flag && lane == 0) {  // let copies in flight land before the CTA exits
      for (int g = max(0, gs - kStages); g < gs; ++g)
        tc::mbar_wait(full_bar(g % kStages), (g / kStages) & 1);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA --
    // The whole warp runs the loop on warp-uniform values and one elected
    // lane issues, which lets the MMA operands stay uniform (a loop inside a
    // one-thread branch issued ~60% slower). The dequant warps arrive on
    // dq_bar only after they have seen the stage's copies land on full_bar,
    // so its completion orders both the A operand and the shared-memory B
    // tile before the MMAs; a failure elsewhere surfaces here through the
    // abort flag. The waits spin on the non-blocking test: a suspending
    // try_wait on the issuing warp lets the MMAs already queued drain (about
    // 380 idle tensor cycles per wait, as measured).
    if (rank == 0) {
      const uint32_t idesc =
          tc::idesc_f16kind_f32(kTileRows * kCg, static_cast<uint32_t>(p.bn), kDx, kF16);
      const uint64_t bdesc0 = tc::sw128_kmajor_desc(tc::smem_addr(smem + C::kOffAct));
      // input gradient: A tile atoms (column half h, row group g) at
      // (2 g + h) KB, i.e. 1 KB apart along M and 2 KB along K
      const uint64_t adesc0 = tc::sw128_mnmajor_desc(tc::smem_addr(smem + C::kOffA), 1024, 2048);
      int gs = 0, k = 0;
      // ring positions kept as counters, as in the producer: divisions by the
      // ring depth (12 at 64 tokens) on this warp's per-stage path cost the
      // forward 1-1.6%
      int sl = 0, as = 0;      // gs % kStages, gs % kASlots
      uint32_t aph = 0;        // (gs / kASlots) & 1
      bool stop = false;
      for (int u = cid; u < p.units && !stop; u += ncl, ++k) {
        const Unit t = unit_at(u);
        const int b = k % kAccBufs;
        const uint32_t acc = tmem + static_cast<uint32_t>(b * kBN);
        // the buffer's previous unit (k - kAccBufs) has been drained
        int r = tc::mbar_spin_abortable<kPair>(acce_bar(b), ((k / kAccBufs) & 1) ^ 1, abort_flag,
                                               1ll << 31);
        r = __shfl_sync(0xffffffffu, r, 0);
        if (r != tc::kWaitDone) {
          if (lane == 0 && r == tc::kWaitTimeout) fail(kRoleMma);
          break;
        }
        tc::fence_after_sync();
        for (int i = 0; i < t.nst; ++i, ++gs) {
          r = tc::mbar_spin_abortable<kPair>(dq_bar(as), aph, abort_flag, p.mma_wait_limit);
          r = __shfl_sync(0xffffffffu, r, 0);
          if (r != tc::kWaitDone) {
            if (lane == 0 && r == tc::kWaitTimeout) fail(kRoleMma);
            stop = true;
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
                tc::mma_bf16_ss<kCg>(acc, adesc + 256u * j, bdesc + 2u * j, idesc,
                                     (i | j) != 0 ? 1u : 0u);
              else
                tc::mma_bf16_tmem_a<kCg>(acc, a + 8u * j, bdesc + 2u * j, idesc,
                                         (i | j) != 0 ? 1u : 0u);
            }
            tc::mma_commit<kCg>(empty_bar(sl));
            if constexpr (kDx) tc::mma_commit<kCg>(afree_bar(as));
          }
          __syncwarp();
          if (++sl == kStages) sl = 0;
          if (++as == kASlots) {
            as = 0;
            aph ^= 1u;
          }
        }
        if (stop) break;
        if (tc::elect_one()) tc::mma_commit<kCg>(accf_bar(b));   // the unit's accumulator is done
        __syncwarp();
      }
      if (tc::elect_one()) tc::mma_commit<kCg>(drain_bar);
      __syncwarp();
      // all MMAs done before teardown (a drain: full limit, no abort exit)
      if (lane == 0 && !tc::mbar_wait(drain_bar, 0)) fail(kRoleMma);
    }
  } else if (warp < C::kFirstEpiWarp) {
    // ------------------------------------------------------------ dequant --
    // the stage's A slot is written: tell the pair's MMA thread
    auto arrive_dq = [&](int a) {
      if constexpr (kPair) tc::mbar_arrive_remote(tc::mapa(dq_bar(a), 0));
      else tc::mbar_arrive(dq_bar(a));
    };
    const int grp = (warp - 2) >> 2;        // takes the stages gs % kGroups == grp
    const uint8_t* tab = smem + C::kOffLut + 8 * (lane & 15);
    // block scale: 4-bit ahat = fl32(fl32(a8 s2) / 255); int8 absmax / 127
    auto block_scale = [&](uint32_t a8v, float sv) {
      return kInt8 ? div_by_const<127>(sv) : dequant_absmax(a8v, sv);
    };
    auto load_block = [&](int64_t bi, uint32_t& a8v, float& sv) {
      if constexpr (kInt8) {
        sv = p.scale[bi];
      } else {
        a8v = p.a8[bi];
        sv = p.scale[bi >> 8];
      }
    };
    // The level table's bulk copy is waited for in full even after an abort
    // (no copy may still be landing in this CTA's shared memory when it
    // exits), after the first scale loads have gone out so that their latency
    // overlaps the copy's.
    bool lut_ready = kInt8;
    auto wait_lut = [&] {
      if (!lut_ready) {
        if (!tc::mbar_wait(lut_bar, 0)) fail(kRoleCompute);
        lut_ready = true;
      }
    };
    // input gradient: thread t of the group dequantizes weight row t % 64 of
    // the stage over the tile's columns 64 (t / 64) .. + 63, one absmax
    // block, as the forward walks a row. The 64 results are one 128-byte row
    // of a 128-byte-swizzled MN-major atom of the A tile (64 weight columns
    // along M x 8 weight rows along K per 1 KB atom; atom (column half h, row
    // group g) at (2 g + h) KB).
    const int t4 = ((warp - 2) & 3) * 32 + lane;
    const int rr = t4 & 63, h = t4 >> 6;
    const int ao = (2 * (rr >> 3) + h) * 1024 + (rr & 7) * 128;
    const int asw = rr & 7;
    int gs = 0, k = 0;
    // With a single accumulator buffer these warps drain it, the four warps
    // of each lane quarter sharing out its 16-column chunks. Unit k's drain
    // waits until each group has dequantized its first stage of unit k + 1
    // (or found it has none): the MMAs of unit k + 1 then find four stages
    // ready when the buffer is free, instead of waiting for the dequant to
    // restart after the drain. Safe to defer: a group's first stage of a
    // unit needs only copies and slots freed by earlier units' MMAs.
    bool pend = false;
    Unit pend_t{};
    int pend_k = 0;
    auto drain_pending = [&]() {
      pend = false;
      if (*abort_flag) return false;
      if (!waited(tc::mbar_wait_abortable(accf_bar(0), pend_k & 1, abort_flag), kRoleEpilogue))
        return false;
      tc::fence_after_sync();
      drain(pend_t, 0, 16 * ((warp - 2) >> 2), 64);
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) arrive_acce(0);
      return true;
    };
    bool drained_ok = true;
    for (int u = cid; u < p.units; u += ncl, ++k) {
      if (*abort_flag) break;
      const Unit t = unit_at(u);
      // this thread's block of stage i of the unit: forward (weight row n,
      // block s_begin + i); input gradient (weight row (s_begin + i) 64 + rr,
      // block r0 / 64 + h)
      const int64_t n_fwd = t.r0 + tile_row;
      const int64_t kb = (t.r0 >> 6) + h;
      auto block_of = [&](int i, int64_t& bi) {
        if constexpr (kDx) {
          const int64_t n = static_cast<int64_t>(t.s_begin + i) * 64 + rr;
          bi = n * p.nblk + kb;
          return kb < p.nblk && n < p.N;
        } else {
          bi = n_fwd * p.nblk + t.s_begin + i;
          return n_fwd < p.N;
        }
      };
      uint32_t a8v = 0;
      float sv = 0.0f;
      bool ok = false;
      auto load_scale = [&](int i) {
        if (i >= t.nst) return;
        int64_t bi;
        ok = block_of(i, bi);
        if (ok) load_block(bi, a8v, sv);
      };
      int i = ((grp - gs % kGroups) + kGroups) % kGroups;   // this group's first stage of the unit
      load_scale(i);
      wait_lut();
      bool first = true;
      for (; i < t.nst; i += kGroups) {
        if constexpr (kAccBufs == 1) {
          if (!first && pend && !(drained_ok = drain_pending())) break;
          first = false;
        }
        const int g = gs + i;                 // the stage's index across units
        const int slot = g % kStages;
        const uint32_t ph = (g / kStages) & 1;
        const float ahat = ok ? block_scale(a8v, sv) : 0.0f;
        const float2 ahat2 = make_float2(ahat, ahat);
        uint32_t plo[4], phi[4];
        if constexpr (C::kPlanes)
          level_planes<kF16>(reinterpret_cast<const float*>(smem + C::kOffLut), ahat, plo, phi);
        load_scale(i + kGroups);
        if constexpr (!kDx) {
          // warp-uniform: the stage is done by all lanes or by none (the
          // arrival below follows a __syncwarp)
          const bool go = !*abort_flag &&
                          waited(tc::mbar_wait_abortable(full_bar(slot), ph, abort_flag),
                                 kRoleCompute);
          if (!__all_sync(0xffffffffu, go)) continue;
          const uint8_t* cst = smem + C::kOffCodes + slot * kCodesStageBytes;
          const uint32_t dst = tmem + lane_base + kTmemA0 + 32u * slot;
#pragma unroll
          for (int hf = 0; hf < 2; ++hf) {
            uint32_t v[16];
            if constexpr (kInt8) {
              // row tile_row's 64 bytes, 64-byte swizzle
              const int sw = (tile_row >> 1) & 3;
#pragma unroll
              for (int cc = 0; cc < 2; ++cc) {
                const int c = 2 * hf + cc;
                const uint4 w =
                    *reinterpret_cast<const uint4*>(cst + tile_row * 64 + 16 * (c ^ sw));
                dequant16_int8<kF16>(w, ahat2, v + 8 * cc);
              }
            } else {
              if constexpr (C::kPlanes)
                dequant16_4bit_planes<kF16>(
                    *reinterpret_cast<const uint4*>(cst + tile_row * 32 + 16 * hf), plo, phi, v);
              else
                dequant16_4bit<kF16>(
                    *reinterpret_cast<const uint4*>(cst + tile_row * 32 + 16 * hf), tab, ahat2, v);
            }
            tc::tmem_st16(dst + 16u * hf, v);
          }
          tc::tmem_wait_st();
          tc::fence_before_sync();
          __syncwarp();
          if (lane == 0) arrive_dq(slot);
        } else {
          // First the A slot: its previous tile (stage g - kASlots) has been
          // read by its MMAs. Only then the stage's copies: once MMA(g -
          // kASlots) is done, so is MMA(g - kStages), whose dequant saw the
          // copy slot's previous phase complete, so this parity wait cannot
          // pass a phase early (the copy slots are shared between groups, and
          // a parity wait cannot tell a phase still pending from the one
          // before it).
          const int as = g % kASlots;
          bool go = !*abort_flag;
          if (go && g >= kASlots)
            go = waited(tc::mbar_wait_abortable(afree_bar(as), ((g / kASlots) - 1) & 1, abort_flag),
                        kRoleCompute);
          go = go && waited(tc::mbar_wait_abortable(full_bar(slot), ph, abort_flag), kRoleCompute);
          if (!__all_sync(0xffffffffu, go)) continue;
          const uint8_t* cst = smem + C::kOffCodes + slot * kCodesStageBytes;
          uint8_t* arow = smem + C::kOffA + as * C::kAStageBytes + ao;
#pragma unroll
          for (int hf = 0; hf < 2; ++hf) {        // columns 32 hf .. + 31 of the run
            uint32_t v[16];
            if constexpr (kInt8) {
              // row rr's chunks 4 h + 2 hf, + 1 of 128 bytes, 128-byte swizzle
#pragma unroll
              for (int cc = 0; cc < 2; ++cc) {
                const uint4 w = *reinterpret_cast<const uint4*>(
                    cst + rr * 128 + 16 * ((4 * h + 2 * hf + cc) ^ (rr & 7)));
                dequant16_int8<kF16>(w, ahat2, v + 8 * cc);
              }
            } else {
              // row rr's chunk 2 h + hf of 64 bytes, 64-byte swizzle
              const int csw = (rr >> 1) & 3;
              if constexpr (C::kPlanes)
                dequant16_4bit_planes<kF16>(
                    *reinterpret_cast<const uint4*>(cst + rr * 64 + 16 * ((2 * h + hf) ^ csw)), plo,
                    phi, v);
              else
                dequant16_4bit<kF16>(
                    *reinterpret_cast<const uint4*>(cst + rr * 64 + 16 * ((2 * h + hf) ^ csw)), tab,
                    ahat2, v);
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
      gs += t.nst;
      if constexpr (kAccBufs == 1) {
        if (!drained_ok || (pend && !drain_pending())) break;   // fewer than two stages here
        pend = true;
        pend_t = t;
        pend_k = k;
      }
    }
    if constexpr (kAccBufs == 1)
      if (drained_ok && pend) drain_pending();   // the last unit
    wait_lut();   // a CTA with no unit still lets the table copy land
  } else if constexpr (kAccBufs == 2) {
    // ----------------------------------------------------------- epilogue --
    // Unit k's accumulator (buffer k % 2) goes out while the MMAs of unit
    // k + 1 fill the other buffer.
    int k = 0;
    for (int u = cid; u < p.units; u += ncl, ++k) {
      const Unit t = unit_at(u);
      const int b = k & 1;
      if (*abort_flag) break;
      if (!waited(tc::mbar_wait_abortable(accf_bar(b), (k >> 1) & 1, abort_flag), kRoleEpilogue))
        break;
      tc::fence_after_sync();
      drain(t, b, 0, 16);
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) arrive_acce(b);
    }
  }

  // The epilogue's output copies have landed before the CTA leaves.
  if (lane == 0) tc::bulk_wait_all();
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

template <bool kDx, int kBN, bool kF16, bool kInt8>
cudaError_t launch_tc(const MatmulCall& c) {
  using C = Cfg<kDx, kBN, kInt8>;
  const int64_t M = c.M, N = c.N, K = c.K;
  TcArgs a;
  a.a8 = c.a8;
  a.scale = c.scale;
  a.out = c.out;
  a.M = M;
  a.N = N;
  a.K = K;
  a.nblk = static_cast<int>(K / kBlock);
  a.fmt = c.fmt;
  a.status = c.status;
  a.bn = kBN;
  a.out_bf16 = c.out_bf16 ? 1 : 0;
  a.accumulate = c.accumulate ? 1 : 0;
  a.mma_wait_limit = c.wait_limit;
  const int64_t nd = kDx ? K : N;            // tile-row dimension
  const int64_t red = kDx ? N : K;           // reduction dimension
  // a unit covers 128 rows per CTA of a pair
  const int64_t row_units = (nd + kTileRows * C::kCg - 1) / (kTileRows * C::kCg);
  const int64_t m_tiles = (M + a.bn - 1) / a.bn;
  a.stages_total = static_cast<int>((red + 63) / 64);
  // Splits of the reduction, summed with atomics into the output (fp32 only):
  // when the tiles alone leave SMs idle, or (forward) leave the persistent
  // grid a partial last round. The estimate is the makespan in stages:
  // rounds of the grid x (stages a split + a unit's fixed cost). The fixed
  // cost, about 30 stages, was fitted to single launches of the
  // decoder-layer shapes at 2048 tokens, split and unsplit (3584 x 18944
  // forward 201 -> 168 us split in two, while 3584 x 3584 lost 2-7%). Each
  // split covers at least one ring of stages; a split is taken only when it
  // gains at least 10% (it adds the zeroing pass and atomic stores). The
  // input gradient splits only grids smaller than the GPU: splitting the
  // 18944 x 3584 gradient in two was 19% faster alone but slower inside the
  // decoder-layer step, where its output's atomics compete with the other
  // projections' traffic.
  const int64_t groups_max = std::max(1, c.num_sms / C::kCg);
  const int64_t tiles = row_units * m_tiles;
  int splits = 1;
  if (kDx) {
    const int64_t ctas = tiles * C::kCg;
    if (ctas < c.num_sms && !c.out_bf16)   // each split fills the ring at least once
      splits = static_cast<int>(std::max<int64_t>(
          1, std::min<int64_t>(c.num_sms / ctas, a.stages_total / C::kStages)));
  } else if (!c.out_bf16) {
    const int64_t smax = std::max<int64_t>(1, std::min<int64_t>(a.stages_total / C::kStages, 16));
    const int64_t ovh = 32;
    auto cost = [&](int64_t s) {
      return ((tiles * s + groups_max - 1) / groups_max) * ((a.stages_total + s - 1) / s + ovh);
    };
    int64_t best = cost(1), best_s = 1;
    for (int64_t s = 2; s <= smax; ++s)
      if (cost(s) < best) {
        best = cost(s);
        best_s = s;
      }
    if (best * 10 <= cost(1) * 9) splits = static_cast<int>(best_s);
  }
  a.stages_per_split = (a.stages_total + splits - 1) / splits;
  splits = (a.stages_total + a.stages_per_split - 1) / a.stages_per_split;
  a.atomic_out = splits > 1 ? 1 : 0;
  // outputs: TMA store, or TMA add (fp32) into a zeroed output for splits and
  // into the caller's for accumulate (2-5% faster than plain stores at 128
  // and 256 tokens); a bf16 output that accumulates keeps plain
  // read-modify-write stores, and so do 64-token tiles (no staging boxes)
  a.out_mode = C::kStageWarps == 0 ? 2 : (a.atomic_out || c.accumulate) ? (c.out_bf16 ? 2 : 1) : 0;
  a.row_units = static_cast<int>(row_units);
  a.m_tiles = static_cast<int>(m_tiles);
  const int64_t units = row_units * m_tiles * splits;
  a.units = static_cast<int>(units);
  // persistent: at most one CTA (or pair) per SM, each taking units in turn
  const int64_t groups = std::min<int64_t>(units, groups_max);

  CUtensorMap tm_act, tm_codes;
  // activations: [M, red] 16-bit, box 64 (reduction) x the tokens one CTA
  // stages, 128-byte swizzle
  if (!encode_2d(&tm_act, kF16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                 c.act, static_cast<uint64_t>(red), static_cast<uint64_t>(M),
                 static_cast<uint64_t>(red) * 2, 64, static_cast<uint32_t>(C::kBRows),
                 CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  // codes: [N, row bytes] (K/2 packed 4-bit, K int8). The forward takes 128
  // rows x one stage's bytes (32, or 64 with the 64-byte swizzle); the input
  // gradient 128 columns x 64 rows (64 bytes with the 64-byte swizzle, or 128
  // with the 128-byte swizzle).
  const uint64_t row_bytes = static_cast<uint64_t>(kInt8 ? K : K / 2);
  const uint32_t box_x = kDx ? (kInt8 ? 128u : 64u) : (kInt8 ? 64u : 32u);
  const uint32_t box_y = kDx ? 64u : 128u;
  const CUtensorMapSwizzle sw = kDx ? (kInt8 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B)
                                    : (kInt8 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_NONE);
  if (!encode_2d(&tm_codes, CU_TENSOR_MAP_DATA_TYPE_UINT8, c.codes, row_bytes,
                 static_cast<uint64_t>(N), row_bytes, box_x, box_y, sw))
    return cudaErrorInvalidValue;
  // outputs: [M, nd] fp32 or bf16, box 32 tile rows x 16 tokens, no swizzle
  CUtensorMap tm_out;
  const uint64_t out_elem = c.out_bf16 ? 2 : 4;
  if (!encode_2d(&tm_out, c.out_bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
                 c.out, static_cast<uint64_t>(nd), static_cast<uint64_t>(M),
                 static_cast<uint64_t>(nd) * out_elem, 32, 16, CU_TENSOR_MAP_SWIZZLE_NONE))
    return cudaErrorInvalidValue;

  static std::once_flag once[kOnceDevices];
  once_per_device(once, c.device, [] {
    cudaFuncSetAttribute(tc_gemm_kernel<kDx, kBN, kF16, kInt8>,
                         cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  });
  if (a.atomic_out && !c.accumulate) {
    cudaError_t e = cudaMemsetAsync(c.out, 0, static_cast<size_t>(M) * nd * sizeof(float), c.st);
    if (e != cudaSuccess) return e;
  }
  const dim3 grid(static_cast<unsigned>(groups * C::kCg));
  if constexpr (C::kPair) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(C::kThreads);
    cfg.dynamicSmemBytes = C::kSmemBytes;
    cfg.stream = c.st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, tc_gemm_kernel<kDx, kBN, kF16, kInt8>, tm_act, tm_codes, tm_out,
                              a);
  } else {
    tc_gemm_kernel<kDx, kBN, kF16, kInt8><<<grid, C::kThreads, C::kSmemBytes, c.st>>>(
        tm_act, tm_codes, tm_out, a);
    return cudaGetLastError();
  }
}

template <bool kDx, bool kF16, bool kInt8>
cudaError_t launch_tc_by_m(const MatmulCall& c) {
  if (c.M <= 64) return launch_tc<kDx, 64, kF16, kInt8>(c);
  if (c.M <= 128) return launch_tc<kDx, 128, kF16, kInt8>(c);
  return launch_tc<kDx, 256, kF16, kInt8>(c);
}

template <bool kDx>
cudaError_t launch_tc_any(const MatmulCall& c) {
  const bool i8 = c.fmt == kFmtInt8;
  if (c.act_f16) return i8 ? launch_tc_by_m<kDx, true, true>(c) : launch_tc_by_m<kDx, true, false>(c);
  return i8 ? launch_tc_by_m<kDx, false, true>(c) : launch_tc_by_m<kDx, false, false>(c);
}

}  // namespace

cudaError_t launch_tc_fwd(const MatmulCall& c) { return launch_tc_any<false>(c); }
cudaError_t launch_tc_dx(const MatmulCall& c) { return launch_tc_any<true>(c); }

}  // namespace nf4
