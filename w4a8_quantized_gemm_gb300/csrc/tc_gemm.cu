// tc_gemm.cu -- tcgen05 tensor-core GEMM for the W4A8, W4A16, W8A16 and W8A8
// linears.
//
// The pages describe the W4A8 linear only as prior art for other hardware (an
// AMX CPU kernel, "The 4-bit CPU path", section "W4A8 - _C::int4_scaled_mm_cpu";
// an optional CUTLASS large-prefill dispatch, "EgoPQ Real-Serving Handoff",
// section 1). This kernel is designed for sm_103a from the method itself:
//
//   y[m,n] = a_s[m] * sum_g s[n,g] * Q[m,n,g],
//   Q[m,n,g] = sum_{k in g} a_q[m,k] * (w_q[n,k] - z[n,g])
//
// sm_103a has no integer tcgen05.mma, so each group partial is formed EXACTLY
// on floating-point MMAs whose operands are exact small integers:
//  - token tiles of at most 64 (kind::f8f6f4, K = 32 per MMA): the weight
//    codes 0..15 are exact e4m3 (two PRMT table lookups per 4 codes), and each
//    activation code splits as a = 16 * (a >> 4) + (a & 15) into two exact
//    e4m3 rows of the B operand (N = 2 * tokens); z * sum(a) comes off in the
//    drain with the per-group activation sums;
//  - larger tiles (kind::f16, K = 16 per MMA): a_q (|a_q| <= 127) and w_q - z
//    (in [-15, 15]) as exact fp16, with z folded into the converted weights.
// Every product is exact and a 128-wide group sums to at most
// 128*127*15 = 243840 < 2^24 in magnitude, so fp32 accumulation of one group
// in Tensor Memory is exact. The accumulator is drained after every group,
// scaled by s[n,g] and accumulated in fp32 registers.
//
// Operand roles ("swap AB"): the 128 weight rows of a tile are the MMA's M
// dimension and live in TENSOR MEMORY as the A operand; the token tile (BT
// tokens, 16..192) is the MMA's N dimension and comes from shared memory as
// the B operand, staged by TMA with 128-byte swizzle. The dequantized weights
// therefore never touch shared memory: converter warps read the packed int4
// record (one 8512-byte bulk copy per 128 rows x 128 K: codes, scales, zero
// points), convert the codes and store them straight into TMEM with
// tcgen05.st.
//
// Warp roles (one CTA per SM; two lean CTAs per SM for 16-token e4m3 tiles):
//   drain warps      TMEM accumulator -> registers, *s, accumulate, epilogue;
//                    two warpgroups splitting the token columns (one warpgroup
//                    with all of them in the lean CTAs)
//   converter warps  packed int4 (or int8) smem tile -> e4m3/fp16/bf16 in TMEM
//                    (a second set of four takes every other group for token
//                    tiles of 32 and 128-token per-group tiles, and half of
//                    every group's K in 192-token tiles)
//   producer warp    TMA: activations tile + weight record per group (per-group
//                    tiles of 128 and 192 tokens: the records only, on a ring
//                    of their own, and a second producer warp for the
//                    activations; int8-weight tiles: both in one stage)
//   issuer warps     one MMA-issuing thread each (two for 32-token and
//                    per-group wide tiles, taking alternate groups); the
//                    first allocates TMEM
// (wide per-group tiles split the registers per warpgroup with setmaxnreg;
// a warp reaches TMEM lanes 32*(warp % 4) .. +31, so each role that touches
// TMEM is a whole warpgroup)
// Hand-offs: S shared-memory stages, kNumA TMEM A buffers, kNumD TMEM
// accumulators, on mbarriers with bounded waits; in the wide tiles the
// converters hand each group to its issuer on a hardware named barrier
// instead (see kNamedHandoff), which the drains of the 192-token tiles join
// too (see kDrainRendezvous). Every mbarrier test is a round trip of about a
// hundred cycles on the waiting thread, so an issuer waits on one barrier per
// group at most: the converters release it only after the stage has landed,
// the A buffer is free and the accumulator has been drained.
//
// Split-K for small grids: a cluster of up to 8 CTAs shares one output tile,
// each taking a contiguous range of groups; partial sums are reduced through
// distributed shared memory in rank order (deterministic, no global scratch).
//
// Variants: W4A16 uses bf16 operands (activations as given, w_q - z exact in
// bf16) and no a_s; W8A16 converts int8 weights to bf16 and accumulates all
// of K in TMEM, applying the per-channel scale once at the end; W8A8 converts
// int8 weights to fp16 against the fp16 activation codes, drains every 8
// groups (exact: 1024 * 127^2 < 2^24), adds the partials as int32 and scales
// by a_s[m] * s[n] at the end.

#include <type_traits>

#include "egopq_internal.h"

namespace egopq {

constexpr int kMaxSmem = 232448;      // dynamic shared memory of a CTA alone on its SM
constexpr int kMaxSmemHalf = 114688;  // each of two CTAs sharing an SM

// Wide tiles: the token tiles of the per-group (W4A8 fp16, W4A16) tensor-core
// path above kTcFp8MaxM tokens. With A in TMEM an MMA of N tokens costs
// max(~95, N/2) cycles per K = 16 step (measured on GB300: a 128-wide group
// takes 757 cycles at N = 128..176 and 4*N from N = 192 up, also with a CTA
// pair), so the tensor pipe reaches its full rate only from 192 tokens a tile.
//  - kWideBT (128 tokens): three 128-column accumulators and two 64-column A
//    buffers, weight records in a ring of their own, two converter sets, two
//    issuers (set q meets issuer q on a named barrier);
//  - kFullBT (192 tokens): two 192-column accumulators and two A buffers fill
//    the 512 TMEM columns, so the drain of group i gates the MMAs of group
//    i + 2; weight records in a ring of their own; two converter sets that
//    split each group's K between them (the first set's first warp also
//    waits for the drained accumulator and the landed activations), meeting
//    two alternating issuers on hardware named barriers (see kNamedHandoff).
// The int8-weight tiles (W8A16, W8A8) come in the same two widths, each
// accumulator holding several groups (two at 192 tokens, two A buffers).
// The launcher picks the width per linear from the grid it makes (192-token
// tiles quantise some grids into a short last wave).
constexpr int kWideBT = 128;
constexpr int kFullBT = 192;

// Output tensor maps of the linears (wide tiles' bulk-store epilogue): bf16
// y_j as 2-D {N_j, M}, box {128, drain columns}.
struct YMaps {
  CUtensorMap map[kMaxSegs];
};

struct TcParams {
  int64_t M, N, K;
  int G, ks;
  int m_tiles, n_tiles;
  // 1: CTAs stride over tiles [0, units) of the banded order with all of K;
  // 0: one tile (blockIdx.y, blockIdx.z) per cluster of ks CTAs splitting K;
  // 2: one tile tail_base + blockIdx.y of the banded order per cluster of ks
  //    CTAs (the short last round of a persistent grid, split so that it
  //    takes all SMs: run as a second launch after mode 1 over the rest)
  int persistent;
  int units, tail_base;
  int band;        // banded tile order: bands of `band` m-tiles, m fastest inside a band
  int act3d;       // 1: activation map is 3-D, one copy per 128-wide group; 0: 2-D, two copies
  const float* a_s;
  const int32_t* a_gsum;  // per-token group sums (e4m3 W4A8 form: zero points in the drain)
  const uint16_t* s8;
  int32_t* partials;
  uint64_t timeout_ns;
  SegTable seg;  // packed weight, output and N of each linear, by output tile
};

template <int VARIANT, int BT>
struct TcCfg {
  // W4A8 with token tiles of at most 64 runs kind::f8f6f4: an MMA costs the
  // same issue time for any N up to 64 (and K = 32 e4m3 per instruction
  // against K = 16 fp16), so the activation codes a = 16 * (a >> 4) + (a & 15)
  // enter as two exact e4m3 rows per token (N = 2*BT) and the weight codes
  // 0..15 as exact e4m3; a group takes 4 MMAs instead of 8, and the zero
  // points come off in the drain as z * sum(a).
  static constexpr bool kFp8 = (VARIANT == kW4A8) && BT <= kTcFp8MaxM;
  static constexpr int kDCols = kFp8 ? 2 * BT : BT;  // TMEM columns of one accumulator
  static constexpr int kACols = kFp8 ? 32 : 64;      // A operand columns of one group
  // Groups per accumulator drain: 1 where every group has its own scale
  // (W4A8, W4A16); 0 = the whole unit (W8A16: per-channel scale, fp32 sums);
  // W8A8 drains every 8 groups (1024 K: |partial| <= 1024 * 127^2 < 2^24,
  // so the fp32 accumulator holds it exactly) and adds the partials as int32
  // (a whole K row can exceed 2^24); its scales come only in the epilogue.
  static constexpr int kGroupsPerDrain = (VARIANT == kW8A16) ? 0 : (VARIANT == kW8A8 ? 8 : 1);
  static constexpr bool kCodes = (VARIANT == kW4A8 || VARIANT == kW8A8);  // per-token scales
  static constexpr bool kDrainPerGroup = (kGroupsPerDrain == 1);
  static constexpr bool kIntAcc = (VARIANT == kW8A8);
  // int8 weight tiles (W8A16, W8A8): staged by a 2-D TMA copy, no pack step
  static constexpr bool kW8 = (VARIANT == kW8A16 || VARIANT == kW8A8);
  // weights staged by a 2-D TMA copy (no pack step): int8 tiles, or the
  // dense bf16 tiles of the twin (two 64-column boxes a group)
  static constexpr bool kW16 = (VARIANT == kW16A16);
  static constexpr bool kTmaW = kW8 || kW16;
  // MMA issuers. An MMA instruction up to N = 64 costs its issuing thread
  // about as much as the tensor core, and every barrier test costs it a
  // round trip, so small token tiles use two issuing warps that take
  // alternate groups. Tiles that accumulate several groups in one
  // accumulator (W8A16, W8A8) keep one issuer, which orders those MMAs.
  // 16-token e4m3 tiles run two lean CTAs per SM (one drain warpgroup, one
  // converter set, one issuer each, half the shared memory and TMEM): their
  // per-group hand-off chain is latency-bound, so two independent pipelines
  // per SM carry twice the groups.
  static constexpr bool kLean = kFp8 && BT == 16;
  static constexpr int kCtasPerSm = kLean ? 2 : 1;
  static constexpr int kDrainWGs = kLean ? 1 : 2;
  static constexpr int kConvWarp0 = 4 * kDrainWGs;  // drain warps first
  static constexpr bool kWide = BT > 64 && kDrainPerGroup;
  static constexpr bool kFull = kWide && BT == kFullBT;  // full-rate tile (see kFullBT)
  static constexpr int kMmaWarps =
      kLean ? 1 : (kWide ? 2 : ((kDrainPerGroup && BT <= 32) ? 2 : 1));
  // Wide tiles hand each group from the converters to its issuer on a
  // hardware named barrier (one per A buffer and issuer), the converters'
  // first warp having waited for the drained accumulator and the landed
  // activations. The issuers then perform no mbarrier operation at all: an
  // mbarrier test queues behind the MMAs the issuing warp has just issued
  // (they wait for the tensor pipe in the same memory-instruction queue), so
  // a test between groups idled the pipe for ~400 cycles a group.
  static constexpr bool kNamedHandoff = kWide;
  static constexpr int kHandoffBar0 = 6;  // named barriers 6, 7 (A buffers 0, 1)
  // TMEM: kNumD accumulators of kDCols columns + kNumA A-operand buffers of
  // kACols columns (deep for small tiles: the converters run ahead of the
  // MMAs and the MMAs ahead of the drain).
  // (wide per-group tiles: three accumulators at 128 tokens -- with two the
  // MMAs of a group wait for the drain two back -- and two at 192, which is
  // all TMEM holds; two A buffers)
  static constexpr int kNumD =
      kLean ? 4 : (kWide ? (kFull ? 2 : 3) : (kFp8 ? (BT == 32 ? 4 : 2) : (BT <= 64 ? 4 : 2)));
  static constexpr int kNumA = kLean ? 4 : (kWide ? 2 : (kFp8 ? 8 : (BT > 128 ? 2 : 4)));
  static constexpr int kActBox = BT * 128;                        // one 64-wide K box, bytes
  static constexpr int kActBytes = 2 * kActBox;                   // a 128-wide group
  // weights of one group: the int8 tile, or one packed int4 record (8192 B of
  // codes, 256 B of scales, 64 B of zero nibbles), padded to keep stages
  // 1024-byte aligned
  static constexpr int kWCopyBytes = kW16 ? 32768 : (kW8 ? 16384 : 8512);
  static constexpr int kWBytes = kW16 ? 32768 : (kW8 ? 16384 : 9216);
  // 192-token tiles keep the weight records in a ring of their own: a
  // record's slot is free as soon as the converters have read it, while an
  // activation stage is held until its MMAs complete. (With one ring, only
  // three 57 KB stages fit, and each stage stayed held from its record's HBM
  // load through conversion, hand-offs and MMAs: ~5000 cycles, one group per
  // ~1700.) Each ring has its own producer thread.
  // (128-token per-group tiles likewise: their activation stage, held from
  // its copy through the MMAs, no longer also waits for the conversion, and
  // five stages fit instead of four; measured faster on every 128-token
  // W4A8 grid. The int8-weight tiles measured slower with a ring of int8
  // tiles, and the dense twin's weights come as two TMA boxes a stage.)
  static constexpr bool kSplitRings = (kFull || (BT == 128 && kWide)) && !kTmaW;
  static constexpr int kStageBytes = kSplitRings ? kActBytes : kActBytes + kWBytes;  // x 1024
  static constexpr int kTxBytes = kSplitRings ? kActBytes : kActBytes + kWCopyBytes;
  static constexpr int kSmemLimit = kCtasPerSm == 1 ? kMaxSmem : kMaxSmemHalf;
  // Wide tiles stage each finished tile in shared memory (bf16 [BT][128]) and
  // write it with TMA bulk stores, one per drain warpgroup, so that the drain
  // goes straight on to the next tile's groups; the tokens' scales of a tile
  // are staged at its start (two tiles' worth: double-buffered).
  static constexpr bool kTmaEpi = kWide;
  static constexpr int kEpiBytes = kTmaEpi ? BT * 128 * 2 : 0;
  static constexpr int kAsBytes = (kTmaEpi && kCodes) ? 2 * BT * 4 : 0;
  // record ring (split rings): kRecStages slots of one 8512-byte record
  static constexpr int kRecStages = kSplitRings ? 3 : 0;
  static constexpr int kRecBytes = (kRecStages * 8512 + 1023) / 1024 * 1024;
  static constexpr int kStagesRaw =
      (kSmemLimit - 3072 - kEpiBytes - kAsBytes - kRecBytes) / kStageBytes;
  // deep rings for small token tiles (decode streams weights: bytes in flight
  // hide HBM latency); larger tiles are bounded by shared memory
  static constexpr int kStageCap = BT <= 32 ? 16 : 8;
  static constexpr int kStages = kStagesRaw > kStageCap ? kStageCap : kStagesRaw;
  static constexpr int kRecOffset = kStages * kStageBytes;  // 1024-byte aligned
  static constexpr int kEpiOffset = kRecOffset + kRecBytes;
  static constexpr int kAsOffset = kEpiOffset + kEpiBytes;
  static constexpr int kBarOffset = kAsOffset + kAsBytes;
  static constexpr int kSmemBytes = kBarOffset + 1024 + 1024;    // + barriers + alignment slack
  static constexpr int kTmemColsRaw = kNumD * kDCols + kNumA * kACols;
  static constexpr int kTmemCols = kTmemColsRaw <= 32    ? 32
                                   : kTmemColsRaw <= 64  ? 64
                                   : kTmemColsRaw <= 128 ? 128
                                   : kTmemColsRaw <= 256 ? 256
                                                         : 512;
  // Converter warp sets: with small token tiles the MMA and drain per group are
  // short, so a second set of four converter warps takes every other group
  // (each set's store-to-arrive latency overlaps the other's conversion).
  static constexpr int kConvSets = kLean ? 1 : ((BT <= 32 || kWide) ? 2 : 1);
  // 192-token tiles: both converter sets work on every group, set q
  // converting K offsets [64q, 64q + 64) (A columns [32q, 32q + 32)), which
  // halves the conversion on each group's hand-off chain; elsewhere the sets
  // take alternate groups
  static constexpr bool kConvSplitK = kFull;
  // 192-token tiles (two accumulators): the drain warps join the rendezvous
  // of group i + 2 as soon as group i's accumulator is in their registers,
  // in place of an accumulator-free mbarrier the converters would test (with
  // two accumulators the current phase of that barrier is then always group
  // i + 2's: group i's completed before its MMAs were issued)
  static constexpr bool kDrainRendezvous = kNamedHandoff && kFull;
  // named hand-off participants: the converter warps meeting an issuer on a
  // group's barrier, the issuer warp, and (see above) the drain warps
  static constexpr int kHandoffCount = 32 * 4 * (kConvSplitK ? kConvSets : 1) + 32 +
                                       (kDrainRendezvous ? 32 * 4 * kDrainWGs : 0);
  static constexpr int kDrainCols = BT / kDrainWGs;  // token columns per drain thread
  static constexpr int kProducerWarp = kConvWarp0 + 4 * kConvSets;
  static constexpr int kMmaWarp = kProducerWarp + 1;  // first issuer; allocates TMEM
  // Register split (128-token per-group tiles): the drain threads hold 64
  // running sums each, so with an even split they can keep only 16 TMEM
  // columns in flight and the drain, latency-bound, paces the pipeline. The
  // block is padded to whole warpgroups (setmaxnreg acts per warpgroup) and
  // the drain warpgroups take registers from the producer/issuer warpgroup,
  // keeping 32 columns in flight. (Drains at 152 with all 64 columns in
  // flight, converters at 64 converting 16 words at a time after their
  // waits, measured slower: conversion then sits on the A-buffer hand-off.)
  static constexpr bool kRegSplit = kWide;
  static constexpr int kWarpsUsed = kMmaWarp + kMmaWarps;
  static constexpr int kWarps = kRegSplit ? (kWarpsUsed + 3) / 4 * 4 : kWarpsUsed;
  // split rings: the first padding warp loads the activations, the producer
  // warp the weight records
  static constexpr int kActWarp = kSplitRings ? kWarpsUsed : -1;
  static_assert(!kSplitRings || kWarps > kWarpsUsed, "activation producer warp");
  static constexpr int kThreads = 32 * kWarps;
  // (192-token tiles: five warpgroups of 96 registers at launch; the drains
  // hold 96 running sums and 48 TMEM columns in flight, the two converter
  // sets half a group's conversion each)
  static constexpr int kRegDrain = kFull ? 144 : 120, kRegConv = kFull ? 72 : 96,
                       kRegOther = 48;
  // (converters keep a whole converted group, 64 registers, in flight)
  static_assert(!kRegSplit || kConvSplitK || kRegConv >= 96, "converter registers");
  // registers every thread has at launch (ptxas holds a kernel that uses
  // setmaxnreg at its launch-bounds maximum; the launcher checks it)
  static constexpr int kRegLaunch = (65536 / kThreads) / 8 * 8;
  static constexpr int kBf16 = (VARIANT == kW4A8 || VARIANT == kW8A8) ? 0 : 1;  // fp16 codes
  static_assert(kStages >= 2, "shared memory too small for two stages");
  static_assert(kSmemBytes <= kSmemLimit, "shared memory");
  static_assert(!kLean || kTmemCols <= 256, "two CTAs share the SM's TMEM");
  static_assert(kTmemColsRaw <= 512, "TMEM budget");
  // Buffer reuse waits test the phase one use back, so the phase two uses back
  // must be known complete: for A buffers by the set's own previous wait
  // (kNumA a multiple of the sets); for accumulators either the same way, or
  // because the A-buffer wait (MMAs of group i - kNumA done, so drains up to
  // i - kNumA - kNumD done, drains run in order) covers i - 2*kNumD.
  static_assert(kNumA % kConvSets == 0 && (kNumD % kConvSets == 0 || kNumA <= kNumD),
                "buffer reuse waits");
  static_assert(8 * (2 * kStages + 2 * kNumA + 2 * kNumD + kMmaWarps + 2 * kRecStages) + 8 <= 1024,
                "barrier region");
  static_assert(BT % 16 == 0 && BT >= 16 && (BT <= 128 || kFull || (kW8 && BT == kFullBT)),
                "token tile");
  // the split hands out exactly the registers the block was launched with
  static_assert(!kRegSplit || (kWarps / 4 == kDrainWGs + kConvSets + 1 &&
                               kDrainWGs * kRegDrain + kConvSets * kRegConv + kRegOther <=
                                   (kWarps / 4) * kRegLaunch),
                "register split");
  static_assert(kStageBytes % 1024 == 0, "stage alignment");
};

// 32 packed int4 codes of one weight row (one 16-byte unit of the record:
// K offsets 0..31 of a 32-wide slice, nibble order as packed) -> 16 words of
// the tensor-core A operand, zero point folded in: fp16 (w - z) pairs for
// W4A8, bf16 pairs for W4A16; both exact.
template <int VARIANT>
__device__ __forceinline__ void cvt_w4_unit(const uint4& v, uint32_t z, uint32_t (&o)[16]) {
  const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
  if constexpr (VARIANT == kW4A8) {
    // fp16: 0x6400|e = 1024+e, 0x6400|(e<<4) = 1024+16e (exact)
    const __half2 zlo = __half2half2(__ushort_as_half((uint16_t)(0x6400u | z)));
    const __half2 nzhi = __half2half2(__float2half_rn(-64.0f - (float)z));
    const __half2 sixteenth = __float2half2_rn(0.0625f);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint32_t w = wv[j], w2 = wv[j] >> 8;
      uint32_t h0 = lop3_and_or(w, 0x000F000Fu, 0x64006400u);
      uint32_t h1 = lop3_and_or(w, 0x00F000F0u, 0x64006400u);
      uint32_t h2 = lop3_and_or(w2, 0x000F000Fu, 0x64006400u);
      uint32_t h3 = lop3_and_or(w2, 0x00F000F0u, 0x64006400u);
      __half2 r0 = __hsub2(*reinterpret_cast<__half2*>(&h0), zlo);
      __half2 r1 = __hfma2(*reinterpret_cast<__half2*>(&h1), sixteenth, nzhi);
      __half2 r2 = __hsub2(*reinterpret_cast<__half2*>(&h2), zlo);
      __half2 r3 = __hfma2(*reinterpret_cast<__half2*>(&h3), sixteenth, nzhi);
      o[j * 4 + 0] = *reinterpret_cast<uint32_t*>(&r0);
      o[j * 4 + 1] = *reinterpret_cast<uint32_t*>(&r1);
      o[j * 4 + 2] = *reinterpret_cast<uint32_t*>(&r2);
      o[j * 4 + 3] = *reinterpret_cast<uint32_t*>(&r3);
    }
  } else {
    // bf16: 0x4300|e = 128+e (exact for e < 128)
    const __nv_bfloat162 zz = __bfloat162bfloat162(__ushort_as_bfloat16((uint16_t)(0x4300u | z)));
#pragma unroll
    for (int j = 0; j < 4; ++j) {
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint32_t h = lop3_and_or(wv[j] >> (4 * q), 0x000F000Fu, 0x43004300u);
        __nv_bfloat162 rr = __hsub2(*reinterpret_cast<__nv_bfloat162*>(&h), zz);
        o[j * 4 + q] = *reinterpret_cast<uint32_t*>(&rr);
      }
    }
  }
}

// y[m0+t][n] = bf16(a_s[m0+t] * R[t]) (W4A8) or bf16(R[t]), t < HB, rows < M,
// into the output `o` of this tile's linear. Eight rows at a time, with a
// compiler barrier between chunks so the a_s loads are not all hoisted (they
// would cost a register each).
template <int VARIANT, int HB>
__device__ __forceinline__ void store_row(const float (&R)[HB], const TcParams& p,
                                          const TileRef& o, int64_t m0, int64_t n) {
  constexpr int CH = HB < 8 ? HB : 8;
#pragma unroll
  for (int c = 0; c < HB; c += CH) {
    asm volatile("" ::: "memory");
#pragma unroll
    for (int t = c; t < c + CH; ++t) {
      const int64_t m = m0 + t;
      if (m < p.M) {
        float v = R[t];
        if constexpr (VARIANT == kW4A8 || VARIANT == kW8A8) v = __ldg(p.a_s + m) * v;
        o.y[m * o.N + n] = f32_to_bf16_bits(v);
      }
    }
  }
}

// The same store with the tokens' scales already in registers (1 where the
// variant has none).
template <int HB>
__device__ __forceinline__ void store_row_scaled(const float (&R)[HB], const float (&asv)[HB],
                                                 const TcParams& p, const TileRef& o, int64_t m0,
                                                 int64_t n) {
#pragma unroll
  for (int t = 0; t < HB; ++t) {
    const int64_t m = m0 + t;
    if (m < p.M) o.y[m * o.N + n] = f32_to_bf16_bits(asv[t] * R[t]);
  }
}

template <int VARIANT, int BT, bool PARTIALS>
__global__ void __launch_bounds__(TcCfg<VARIANT, BT>::kThreads, TcCfg<VARIANT, BT>::kCtasPerSm)
tc_gemm_kernel(const __grid_constant__ CUtensorMap act_map,
               const __grid_constant__ CUtensorMap w8_map, const __grid_constant__ TcParams p,
               const __grid_constant__ YMaps ymaps) {
  using C = TcCfg<VARIANT, BT>;
  constexpr bool kCodes = (VARIANT == kW4A8 || VARIANT == kW8A8);  // per-token scales
  constexpr int S = C::kStages;
  constexpr int HB = C::kDrainCols;  // token columns per drain thread
  constexpr int kNumA = C::kNumA, kNumD = C::kNumD;
  constexpr int kConvWarp0 = C::kConvWarp0;
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte alignment for the 128-byte-swizzle atoms
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t base = (raw_addr + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw_addr);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = p.G;

  // ---- this CTA's work: a flat sequence of (tile, group) items ---------------
  // persistent: tiles blockIdx.x, +gridDim.x, ... each with all G groups;
  // split-K:    tile (blockIdx.y, blockIdx.z), or tail tile tail_base +
  //             blockIdx.y, groups of cluster rank blockIdx.x.
  int u_begin, u_step, n_units, g0, g1;
  if (p.persistent == 1) {
    const int total = p.units;
    u_begin = blockIdx.x;
    u_step = gridDim.x;
    n_units = u_begin < total ? (total - u_begin + u_step - 1) / u_step : 0;
    g0 = 0;
    g1 = G;
  } else {
    u_begin = p.persistent == 2 ? p.tail_base + (int)blockIdx.y
                                : (int)blockIdx.y + (int)blockIdx.z * p.m_tiles;
    u_step = 1;
    n_units = 1;
    g0 = (int)((int64_t)blockIdx.x * G / p.ks);
    g1 = (int)((int64_t)(blockIdx.x + 1) * G / p.ks);
  }
  const int ng = g1 - g0;
  const int n_items = n_units * ng;
  // accumulator drains per unit, and the drain that item i feeds
  constexpr int GPD = C::kGroupsPerDrain;
  const int nc = GPD == 0 ? 1 : (ng + GPD - 1) / GPD;
  auto drain_of = [&](int i) -> int {
    if constexpr (GPD == 1) return i;
    else if constexpr (GPD == 0) return i / ng;
    else return (i / ng) * nc + (i % ng) / (GPD > 1 ? GPD : 1);
  };
  // tile u -> (mt, nt). Persistent grids (and their split tails) walk bands
  // of p.band m-tiles, m fastest inside a band, so the tiles in flight at
  // once share a few activation tiles and a few weight tiles (both stay in L2).
  auto unit_tile = [&](int k, int& mt, int& nt) {
    const int u = u_begin + k * u_step;
    if (p.persistent != 0) {
      const int band_tiles = p.band * p.n_tiles;
      const int b = u / band_tiles;
      const int idx = u - b * band_tiles;
      const int m_base = b * p.band;
      const int bm = min(p.band, p.m_tiles - m_base);
      nt = idx / bm;
      mt = m_base + (idx - nt * bm);
    } else {
      mt = u % p.m_tiles;
      nt = u / p.m_tiles;
    }
  };

  // ---- barriers and flags ------------------------------------------------------
  const uint32_t bar0 = base + C::kBarOffset;
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (S + s); };
  auto afull_bar = [&](int i) { return bar0 + 8u * (2 * S + i); };
  auto aempty_bar = [&](int i) { return bar0 + 8u * (2 * S + kNumA + i); };
  auto dfull_bar = [&](int i) { return bar0 + 8u * (2 * S + 2 * kNumA + i); };
  auto dempty_bar = [&](int i) { return bar0 + 8u * (2 * S + 2 * kNumA + kNumD + i); };
  // one per issuer: its final commit, waited on before teardown
  auto fin_bar = [&](int i) { return bar0 + 8u * (2 * S + 2 * kNumA + 2 * kNumD + i); };
  // split rings: record slot r landed / read by the converters
  // (R is 1 without split rings, where nothing uses it: a divisor everywhere)
  constexpr int R = C::kRecStages > 0 ? C::kRecStages : 1;
  constexpr int kRecBar0 = 2 * S + 2 * kNumA + 2 * kNumD + C::kMmaWarps;
  auto wfull_bar = [&](int r) { return bar0 + 8u * (kRecBar0 + r); };
  auto wempty_bar = [&](int r) { return bar0 + 8u * (kRecBar0 + R + r); };
  uint8_t* misc = smem + C::kBarOffset + 8 * (kRecBar0 + 2 * C::kRecStages);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(misc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 4);
  auto stage_act = [&](int s) { return base + (uint32_t)(s * C::kStageBytes); };
  auto stage_w_ptr = [&](int s) { return smem + s * C::kStageBytes + C::kActBytes; };
  // the weight record of item i: its record-ring slot, or its stage
  auto rec_ptr = [&](int i) {
    if constexpr (C::kSplitRings) return smem + C::kRecOffset + (i % R) * 8512;
    else return stage_w_ptr(i % S);
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full_bar(s), 1);
      // released by the MMA commit and the 4 converter warps (and, in the
      // e4m3 form, the 8 drain warps, which read the record's scales and
      // zero points from the stage)
      mbar_init(empty_bar(s), 1 + (C::kSplitRings ? 0 : 4 * (C::kConvSplitK ? C::kConvSets : 1)) +
                                  (C::kFp8 ? 4 * C::kDrainWGs : 0));
    }
    for (int r = 0; r < C::kRecStages; ++r) {
      mbar_init(wfull_bar(r), 1);
      mbar_init(wempty_bar(r), 4 * (C::kConvSplitK ? C::kConvSets : 1));
    }
    for (int i = 0; i < kNumA; ++i) {
      mbar_init(afull_bar(i), 4);
      mbar_init(aempty_bar(i), 1);
    }
    for (int i = 0; i < kNumD; ++i) {
      mbar_init(dfull_bar(i), 1);
      mbar_init(dempty_bar(i), 4 * C::kDrainWGs);
    }
    for (int i = 0; i < C::kMmaWarps; ++i) mbar_init(fin_bar(i), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if ((warp == C::kProducerWarp || warp == C::kActWarp) && lane == 0) {
    prefetch_tensormap(&act_map);
    if constexpr (C::kTmaW) prefetch_tensormap(&w8_map);
  }
  if (warp == C::kMmaWarp) {
    tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t d_tmem = tmem;                  // accumulators: columns [0, kNumD*BT)
  const uint32_t a_tmem = tmem + kNumD * C::kDCols;  // A operand: kNumA buffers of kACols
  const uint64_t tmo = p.timeout_ns;
  const bool cluster_reduce = !PARTIALS && p.persistent != 1 && p.ks > 1;

  // Each role ends with the same named CTA barrier (every thread) and, for
  // split-K clusters, the same two cluster barriers, so the drain warps can
  // keep their accumulators in registers through the epilogue.
  auto teardown_sync = [&]() {
    tc_fence_before();
    asm volatile("bar.sync 1, %0;" ::"n"(C::kThreads) : "memory");
  };

  // kRecords / kActs: which copies this producer thread issues (both with one
  // ring; with split rings the producer warp the records, kActWarp the
  // activations)
  auto producer_role = [&](auto records_tag, auto acts_tag) {
    constexpr bool kRecords = decltype(records_tag)::value;
    constexpr bool kActs = decltype(acts_tag)::value;
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      // item i = (unit i / ng, group g0 + i % ng), walked with counters
      int w_k = 0, w_gi = 0, w_mt = 0, w_nt = 0;   // weights cursor
      int a_k = 0, a_gi = 0, a_mt = 0, a_nt = 0;   // activations cursor
      if (n_items > 0) {
        unit_tile(0, w_mt, w_nt);
        a_mt = w_mt;
        a_nt = w_nt;
      }
      auto advance = [&](int& k, int& gi, int& mt, int& nt) {
        if (++gi == ng) {
          gi = 0;
          if (++k < n_units) unit_tile(k, mt, nt);
        }
      };
      // weights of the next item into shared address dst, completing on bar
      auto load_weights_to = [&](uint32_t dst, uint32_t bar) {
        const int nt = w_nt, g = g0 + w_gi;
        advance(w_k, w_gi, w_mt, w_nt);
        const TileRef tr = tile_ref(p.seg, nt, G);
        const uint8_t* src = tr.rec0 + (int64_t)g * 8512;
        if (!dbg_record_ok((uint64_t)(src - p.seg.packed[tr.seg]), 8512,
                           packed_record_bytes(tr.N, G)))
          src = p.seg.packed[tr.seg];
        bulk_load(dst, src, 8512, bar);
      };
      auto load_weights = [&](int s) {
        if constexpr (C::kW16) {
          const int nt = w_nt, g = g0 + w_gi;
          advance(w_k, w_gi, w_mt, w_nt);
          tma_load_2d(stage_act(s) + C::kActBytes, &w8_map, full_bar(s), g * 128, nt * 128);
          tma_load_2d(stage_act(s) + C::kActBytes + 16384, &w8_map, full_bar(s), g * 128 + 64,
                      nt * 128);
        } else if constexpr (C::kW8) {
          const int nt = w_nt, g = g0 + w_gi;
          advance(w_k, w_gi, w_mt, w_nt);
          tma_load_2d(stage_act(s) + C::kActBytes, &w8_map, full_bar(s), g * 128, nt * 128);
        } else {
          load_weights_to(stage_act(s) + C::kActBytes, full_bar(s));
        }
      };
      auto load_act = [&](int s) {
        const int mt = a_mt, g = g0 + a_gi;
        advance(a_k, a_gi, a_mt, a_nt);
        if constexpr (C::kFp8) {
          // both e4m3 planes of BT tokens: [2][BT][128] bytes
          tma_load_3d(stage_act(s), &act_map, full_bar(s), g * 128, mt * BT, 0);
        } else if (p.act3d) {
          tma_load_3d(stage_act(s), &act_map, full_bar(s), 0, mt * BT, g * 2);
        } else {
          tma_load_2d(stage_act(s), &act_map, full_bar(s), g * 128, mt * BT);
          tma_load_2d(stage_act(s) + C::kActBox, &act_map, full_bar(s), g * 128 + 64, mt * BT);
        }
      };
      if constexpr (kRecords && !kActs) {
        // record ring: slot i % R is refilled once the converters of item
        // i - R have read it (weights do not depend on the preceding grid)
        int issued = 0;
        for (int i = 0; i < n_items; ++i) {
          const int r = i % R;
          if (i >= R && !mbar_wait(wempty_bar(r), ((i / R) & 1) ^ 1, abort_flag, tmo)) break;
          mbar_arrive_expect_tx(wfull_bar(r), 8512);
          load_weights_to(base + C::kRecOffset + (uint32_t)(r * 8512), wfull_bar(r));
          ++issued;
        }
        for (int i = (issued > R ? issued - R : 0); i < issued; ++i) {
          volatile int no_abort = 0;
          mbar_wait(wfull_bar(i % R), (i / R) & 1, &no_abort, tmo);
        }
      } else if constexpr (kActs && !kRecords) {
        // activation ring: stage i % S is refilled once the MMAs of item
        // i - S have completed
        griddep_wait();
        griddep_launch_dependents();
        int issued = 0;
        for (int i = 0; i < n_items; ++i) {
          const int s = i % S;
          if (i >= S && !mbar_wait(empty_bar(s), ((i / S) & 1) ^ 1, abort_flag, tmo)) break;
          mbar_arrive_expect_tx(full_bar(s), C::kTxBytes);
          load_act(s);
          ++issued;
        }
        for (int i = (issued > S ? issued - S : 0); i < issued; ++i) {
          volatile int no_abort = 0;
          mbar_wait(full_bar(i % S), (i / S) & 1, &no_abort, tmo);
        }
      } else {
        // weights do not depend on the preceding grid: start streaming them
        // before waiting for it; activations only after
        const int n_pre = n_items < S ? n_items : S;
        for (int i = 0; i < n_pre; ++i) {
          mbar_arrive_expect_tx(full_bar(i), C::kTxBytes);
          load_weights(i);
        }
        griddep_wait();
        griddep_launch_dependents();
        for (int i = 0; i < n_pre; ++i) load_act(i);
        int issued = n_pre;
        for (int i = n_pre; i < n_items; ++i) {
          const int s = i % S;
          if (!mbar_wait(empty_bar(s), ((i / S) & 1) ^ 1, abort_flag, tmo)) break;
          mbar_arrive_expect_tx(full_bar(s), C::kTxBytes);
          load_weights(s);
          load_act(s);
          ++issued;
        }
        // wait (bounded) for every copy this thread issued to land before exit
        for (int i = (issued > S ? issued - S : 0); i < issued; ++i) {
          volatile int no_abort = 0;
          mbar_wait(full_bar(i % S), (i / S) & 1, &no_abort, tmo);
        }
      }
    }
    __syncwarp();
    teardown_sync();
    if (cluster_reduce) {
      cluster_sync_all();
      cluster_sync_all();
    }
  };
  auto pad_role = [&]() {
    // ------------------------------------------------------------ padding warps
    teardown_sync();
    if (cluster_reduce) {
      cluster_sync_all();
      cluster_sync_all();
    }
  };
  auto mma_role = [&]() {
    // ------------------------------------------------------------ MMA issuers
    // issuer q takes groups q, q + kMmaWarps, ...
    const int q = warp - C::kMmaWarp;
    constexpr uint32_t idesc = idesc_f16(128, C::kFp8 ? 2 * BT : BT, C::kBf16);
    // (lane 0) the waits that let group i go: false once a wait gave up
    auto wait_group = [&](int i) -> bool {
      const int ab = i % kNumA;
      // one wait per group: the converters arrive on afull only once the
      // stage has landed, the A buffer is free and the accumulator drained
      return mbar_wait(afull_bar(ab), (i / kNumA) & 1, abort_flag, tmo);
    };
    // (lane 0) group i's MMAs and the commits that release its buffers
    auto issue_group = [&](int i) {
      const int s = i % S, ab = i % kNumA;
      const int gi = i % ng;
      const int di = drain_of(i);
      const int db = di % kNumD;
      // first group of its accumulator; last group of it
      constexpr int kGpd = GPD > 1 ? GPD : 1;  // (a divisor in every instantiation)
      const bool d_first = GPD == 1 || (GPD == 0 ? gi == 0 : gi % kGpd == 0);
      const bool d_last = GPD == 1 || gi == ng - 1 || (GPD > 1 && gi % kGpd == kGpd - 1);
      tc_fence_after();
      if constexpr (C::kFp8) {
        // 4 x K=32: B rows are the 2*BT e4m3 token rows of one 128-byte
        // swizzled box; K step j advances 32 bytes inside it
#pragma unroll
        for (int j = 0; j < 4; ++j)
          tc_mma_f8_ts(d_tmem + db * C::kDCols, a_tmem + ab * C::kACols + j * 8,
                       sdesc_kmajor_sw128(stage_act(s) + j * 32), idesc, j > 0);
      } else {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const uint32_t b_addr = stage_act(s) + (j >> 2) * C::kActBox + (j & 3) * 32;
          const uint32_t acc = (j > 0 || !d_first) ? 1u : 0u;
          tc_mma_f16_ts(d_tmem + db * C::kDCols, a_tmem + ab * 64 + j * 8,
                        sdesc_kmajor_sw128(b_addr), idesc, acc);
        }
      }
      tc_commit(empty_bar(s));
      tc_commit(aempty_bar(ab));
      if (d_last) tc_commit(dfull_bar(db));
    };
    bool any = false;
    if constexpr (C::kNamedHandoff) {
      // the whole warp meets the converters on each group's named barrier
      // (every group, also after an abort: see the converters); lane 0
      // issues unless a wait somewhere in the CTA gave up
      // (issuer q takes the groups i = q mod 2, whose A buffer and named
      // barrier are q; the two issuers' MMAs queue in the tensor pipe back to
      // back, so one issuer meets the converters while the other's MMAs are
      // still being accepted and the pipe does not drain between groups)
      static_assert(kNumA == 2 && C::kMmaWarps == 2, "named hand-off layout");
      for (int i = q; i < n_items; i += C::kMmaWarps) {
        asm volatile("bar.sync %0, %1;" ::"r"(C::kHandoffBar0 + i % kNumA), "n"(C::kHandoffCount)
                     : "memory");
        if (!__shfl_sync(0xffffffffu, *abort_flag != 0 ? 1 : 0, 0)) {
          if (lane == 0) issue_group(i);
          any = true;
        }
        __syncwarp();
      }
    } else if (lane == 0) {
      for (int i = q; i < n_items; i += C::kMmaWarps) {
        if (!wait_group(i)) break;
        issue_group(i);
        any = true;
      }
    }
    if (lane == 0 && any) {  // let this issuer's MMAs finish before teardown
      tc_commit(fin_bar(q));
      volatile int no_abort = 0;
      mbar_wait(fin_bar(q), 0, &no_abort, tmo);
    }
    __syncwarp();
    teardown_sync();
    if (warp == C::kMmaWarp) {
      tc_fence_after();
      tmem_dealloc(tmem, C::kTmemCols);
    }
    if (cluster_reduce) {
      cluster_sync_all();
      cluster_sync_all();
    }
  };
  auto conv_role = [&]() {
    // ------------------------------------------------------------ converters
    const int r = ((warp - kConvWarp0) & 3) * 32 + lane;  // weight row == TMEM lane
    const int set = (warp - kConvWarp0) >> 2;             // this set converts items set, +sets..
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    // item i: stage its weights as the A operand (false once a wait gave up)
    auto convert_item = [&](int i) -> bool {
      const int s = i % S, ab = i % kNumA;
      if constexpr (C::kSplitRings) {
        if (!mbar_wait(wfull_bar(i % R), (i / R) & 1, abort_flag, tmo)) return false;
      } else {
        if (!mbar_wait(full_bar(s), (i / S) & 1, abort_flag, tmo)) return false;
      }
      uint32_t out[64];
      if constexpr (C::kFp8) {
        const uint8_t* wt = stage_w_ptr(s) + r * 16;
        uint4 v[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) v[c] = *reinterpret_cast<const uint4*>(wt + c * 2048);
        __syncwarp();
        if (lane == 0) mbar_arrive(empty_bar(s));
        // codes 0..15 -> e4m3 by table: prmt picks byte (nibble & 7) of the
        // 8-byte half-table; a nibble with bit 3 set selects a sign fill,
        // which is 0x00 because every table byte is positive, so the two
        // half-table lookups (the second with bit 3 flipped) OR together.
        constexpr uint32_t kT0 = 0x44403800u, kT1 = 0x4E4C4A48u;  // 0,1,2,3 | 4,5,6,7
        constexpr uint32_t kT2 = 0x53525150u, kT3 = 0x57565554u;  // 8..11  | 12..15
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const uint32_t wv[4] = {v[c].x, v[c].y, v[c].z, v[c].w};
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const uint32_t w = wv[j], wx = wv[j] ^ 0x88888888u;
            // nibbles 0..3 (K offsets 0,2,4,6), then 4..7 (offsets 1,3,5,7)
            out[c * 8 + j * 2] = prmt(kT0, kT1, w) | prmt(kT2, kT3, wx);
            out[c * 8 + j * 2 + 1] = prmt(kT0, kT1, w >> 16) | prmt(kT2, kT3, wx >> 16);
          }
        }
      } else if constexpr (C::kW16) {
        // dense bf16 row r: two 128-byte-swizzled boxes of 64 K values, copied
        // as they are (K pairs per 32-bit word, the A operand's layout)
        // (K split between the sets: set q copies box q into out[0, 32))
#pragma unroll
        for (int bb = 0; bb < (C::kConvSplitK ? 1 : 2); ++bb) {
          const int b = C::kConvSplitK ? set : bb;
          const uint8_t* wt = stage_w_ptr(s) + b * 16384 + r * 128;
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const uint4 v = *reinterpret_cast<const uint4*>(wt + ((c ^ (r & 7)) * 16));
            out[bb * 32 + c * 4 + 0] = v.x;
            out[bb * 32 + c * 4 + 1] = v.y;
            out[bb * 32 + c * 4 + 2] = v.z;
            out[bb * 32 + c * 4 + 3] = v.w;
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(empty_bar(s));
      } else if constexpr (C::kW8) {
        const uint8_t* wt = stage_w_ptr(s) + r * 128;
        uint4 v[8];
#pragma unroll
        for (int c = 0; c < 8; ++c)
          v[c] = *reinterpret_cast<const uint4*>(wt + ((c ^ (r & 7)) * 16));
        __syncwarp();
        if (lane == 0) mbar_arrive(empty_bar(s));
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const uint32_t wv[4] = {v[c].x ^ 0x80808080u, v[c].y ^ 0x80808080u,
                                  v[c].z ^ 0x80808080u, v[c].w ^ 0x80808080u};
#pragma unroll
          for (int q = 0; q < 4; ++q) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              // 2^23 + (w + 128) as fp32 bits, minus 2^23 + 128: exactly w
              const float lo =
                  __uint_as_float(prmt(wv[q], 0x4B000000u, 0x7650u | (2 * h))) - 8388736.0f;
              const float hi =
                  __uint_as_float(prmt(wv[q], 0x4B000000u, 0x7650u | (2 * h + 1))) - 8388736.0f;
              if constexpr (VARIANT == kW8A8) {  // fp16 against fp16 activation codes
                __half2 h2 = __floats2half2_rn(lo, hi);
                out[c * 8 + q * 2 + h] = *reinterpret_cast<uint32_t*>(&h2);
              } else {
                __nv_bfloat162 b2 = __floats2bfloat162_rn(lo, hi);
                out[c * 8 + q * 2 + h] = *reinterpret_cast<uint32_t*>(&b2);
              }
            }
          }
        }
      } else {
        // (K split between the sets: set q converts the record's 32-wide
        // chunks 2q and 2q + 1 into out[0, 32))
        constexpr int NC = C::kConvSplitK ? 2 : 4;
        const int c0 = C::kConvSplitK ? 2 * set : 0;
        const uint8_t* rec = rec_ptr(i);
        const uint8_t* wt = rec + r * 16;
        uint4 v[NC];
#pragma unroll
        for (int c = 0; c < NC; ++c) v[c] = *reinterpret_cast<const uint4*>(wt + (c0 + c) * 2048);
        const uint8_t zb = rec[8448 + (r >> 1)];
        __syncwarp();
        if (lane == 0) mbar_arrive(C::kSplitRings ? wempty_bar(i % R) : empty_bar(s));
        const uint32_t z = (r & 1) ? (zb >> 4) : (zb & 0xF);
#pragma unroll
        for (int c = 0; c < NC; ++c) {
          uint32_t chunk[16];
          cvt_w4_unit<VARIANT>(v[c], z, chunk);
#pragma unroll
          for (int q = 0; q < 16; ++q) out[c * 16 + q] = chunk[q];
        }
      }
      // A buffer ab is free once the MMAs of item i - kNumA have completed
      if (!mbar_wait(aempty_bar(ab), ((i / kNumA) & 1) ^ 1, abort_flag, tmo)) return false;
      tc_fence_after();
      const uint32_t dst = a_tmem + lane_base + ab * C::kACols;
      // (K split: this set's half of the columns)
      constexpr int kStChunks = C::kConvSplitK ? C::kACols / 32 : C::kACols / 16;
      const int st0 = C::kConvSplitK ? set * kStChunks : 0;
#pragma unroll
      for (int c = 0; c < kStChunks; ++c) {
        uint32_t chunk[16];
#pragma unroll
        for (int q = 0; q < 16; ++q) chunk[q] = out[c * 16 + q];
        tmem_st16(dst + (st0 + c) * 16, chunk);
      }
      tmem_wait_st();
      // the accumulator this item feeds must have been drained before its
      // MMAs are released (the A operand is stored first: only the MMAs, not
      // the stores, wait for the drain); one warp of the set waits (afull
      // completes only with all four arrivals)
      // (K split: the first set's first warp)
      const bool gate_warp = C::kConvSplitK ? warp == kConvWarp0 : ((warp - kConvWarp0) & 3) == 0;
      if (!C::kDrainRendezvous && gate_warp) {
        const int di = drain_of(i);
        if (!mbar_wait(dempty_bar(di % kNumD), ((di / kNumD) & 1) ^ 1, abort_flag, tmo)) return false;
      }
      // split rings: the activation stage the MMAs read has landed (one warp
      // of the set waits; afull completes only with all four arrivals)
      if (C::kSplitRings && gate_warp) {
        if (!mbar_wait(full_bar(s), (i / S) & 1, abort_flag, tmo)) return false;
      }
      return true;
    };
    if constexpr (C::kNamedHandoff) {
      // rendezvous with the issuer on group i's named barrier, for every
      // group, also after a failed wait (the work is skipped then): both
      // sides always make exactly n_items rendezvous, so neither can wait
      // for ever, and no barrier phase can collect a second arrival early
      // (group i meets issuer i mod 2 on barrier i mod 2: one converter set
      // takes every group, two sets take one barrier each; bar.sync is the
      // .aligned form: each warp reaches it converged, and `ok` is kept
      // warp-uniform)
      static_assert(kNumA == 2 && (C::kConvSets == 1 || C::kConvSets == 2),
                    "named hand-off layout");
      // (with the K split every set takes every group)
      constexpr int kStep = C::kConvSplitK ? 1 : C::kConvSets;
      bool ok = true;
      for (int i = C::kConvSplitK ? 0 : set; i < n_items; i += kStep) {
        if (ok) ok = convert_item(i);
        ok = __all_sync(0xffffffffu, ok);
        tc_fence_before();
        __syncwarp();
        asm volatile("bar.sync %0, %1;" ::"r"(C::kHandoffBar0 + i % kNumA), "n"(C::kHandoffCount)
                     : "memory");
      }
    } else {
      for (int i = set; i < n_items; i += C::kConvSets) {
        if (!convert_item(i)) break;
        // hand group i to its issuer (A stored, accumulator drained,
        // activations landed)
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(afull_bar(i % kNumA));
      }
    }
    __syncwarp();
    teardown_sync();
    if (cluster_reduce) {
      cluster_sync_all();
      cluster_sync_all();
    }
  };
  auto drain_role = [&]() {
    // ------------------------------------------------------------ drain
    const int r = (warp & 3) * 32 + lane;
    const int col0 = (warp >> 2) * HB;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    // scale of row r, group g: half-word 4096 + r of record (tile, g), records
    // 4256 half-words apart
    // per-group scales of this thread's row, walked with a pointer and
    // prefetched one group ahead (the next tile's first one at a tile's end);
    // the e4m3 form reads scale and zero point from the staged record instead
    constexpr bool kScaleFromGlobal = C::kDrainPerGroup && !C::kFp8 && !C::kIntAcc && !C::kW16;
    constexpr bool kScaleCheck = kScaleFromGlobal;
    auto scale_ptr = [&](int tile, int g) {
      const TileRef tr = tile_ref(p.seg, tile, G);
      const uint8_t* base = p.seg.packed[tr.seg];
      const uint8_t* q = tr.rec0 + (int64_t)g * 8512 + 8192 + 2 * r;
      // (the release build reads every per-group scale through this pointer
      // plus multiples of 4256 half-words, one record per group, all within
      // the tile's G records)
      if (kScaleCheck && !dbg_record_ok((uint64_t)(q - base), 2u + (uint64_t)(G - 1 - g) * 8512u,
                                        packed_record_bytes(tr.N, G)))
        q = base + 8192;
      return reinterpret_cast<const uint16_t*>(q);
    };
    griddep_wait();  // a_s and y belong to the stream's order
    if constexpr (C::kTmaEpi && !PARTIALS) {
      if ((warp & 3) == 0 && lane < p.seg.count) prefetch_tensormap(&ymaps.map[lane]);
    }
    float R[HB];     // fp32 running sums for this thread's weight row
    const uint16_t* sp = nullptr;
    // (kept as raw fp16 bits until used, so that the load's latency overlaps
    // a whole group; W8A16 has no per-group scale: 1.0)
    uint16_t s_next = 0x3C00;
    int mt = 0, nt = 0;
    if (n_items > 0) {
      unit_tile(0, mt, nt);
      sp = scale_ptr(nt, g0);
      if constexpr (kScaleFromGlobal) s_next = __ldg(sp);
    }
    bool ok = true;
    TileRef out{};  // the current tile's linear: output, its rows, first row
    // bulk-store epilogue (wide tiles): the warpgroup's staging rows, its
    // token scales, and the one thread that issues its stores
    const int wg = warp >> 2;
    const bool epi_thread = (warp & 3) == 0 && lane == 0;
    uint16_t* ybuf = reinterpret_cast<uint16_t*>(smem + C::kEpiOffset) + col0 * 128;
    float* as_stage = reinterpret_cast<float*>(smem + C::kAsOffset);
    // y rows [m0 + col0, +HB) of tile k's linear `o`: scaled and rounded into
    // the warpgroup's staging rows, then one bulk store
    auto epilogue_tma = [&](const float (&Rv)[HB], int k, int64_t m0, const TileRef& o) {
      // the warpgroup's previous bulk store must have read its rows
      if (epi_thread) bulk_wait_group_read0();
      asm volatile("bar.sync %0, 128;" ::"r"(2 + wg) : "memory");
      // eight tokens at a time: their scales as two vector loads issued
      // before the chunk's stores (so that no load waits behind a store)
      const float* as_row = as_stage + (k & 1) * BT + col0;
#pragma unroll
      for (int c = 0; c < HB; c += 8) {
        float av[8] = {1.f, 1.f, 1.f, 1.f, 1.f, 1.f, 1.f, 1.f};
        if constexpr (kCodes) {
          const float4 a0 = *reinterpret_cast<const float4*>(as_row + c);
          const float4 a1 = *reinterpret_cast<const float4*>(as_row + c + 4);
          av[0] = a0.x; av[1] = a0.y; av[2] = a0.z; av[3] = a0.w;
          av[4] = a1.x; av[5] = a1.y; av[6] = a1.z; av[7] = a1.w;
        }
        uint16_t yv[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) yv[q] = f32_to_bf16_bits(Rv[c + q] * av[q]);
#pragma unroll
        for (int q = 0; q < 8; ++q) ybuf[(c + q) * 128 + r] = yv[q];
      }
      fence_proxy_async_smem();
      asm volatile("bar.sync %0, 128;" ::"r"(2 + wg) : "memory");
      if (epi_thread && ok && m0 + col0 < p.M) {
        tma_store_2d(&ymaps.map[o.seg], smem_u32(ybuf), (int)o.n0, (int)(m0 + col0));
        bulk_commit_group();
      }
    };
    // (drain rendezvous: the drain warps join the named barrier of every group
    // in order -- groups 0 and 1 at once, group i + 2 once group i's
    // accumulator is loaded, and any left after a failed wait at the end -- so
    // that they, too, make exactly n_items rendezvous)
    int next_join = 0;
    auto join = [&](int j) {
      tc_fence_before();
      __syncwarp();
      asm volatile("bar.sync %0, %1;" ::"r"(C::kHandoffBar0 + j % kNumA), "n"(C::kHandoffCount)
                   : "memory");
    };
    if constexpr (C::kDrainRendezvous) {
      while (next_join < 2 && next_join < n_items) join(next_join++);
    }
    // Wide tiles: after a failed wait a drain warp skips the work but keeps
    // the warpgroup's barrier sequence (the epilogue's named barriers, the
    // rendezvous joins) to the end, since its warpgroup's other warps may
    // have seen the same phase complete (a wait that finds the phase
    // complete on its first test returns at once, one that does not gives up
    // on the CTA's abort flag) and would otherwise wait for it for ever.
    constexpr bool kUniformDrain = C::kTmaEpi;
    for (int k = 0; k < n_units && (ok || kUniformDrain); ++k) {
      if (k > 0) unit_tile(k, mt, nt);
      out = tile_ref(p.seg, nt, G);
      const int64_t n = out.n0 + r;  // row of this thread in its linear's output
      const int64_t N = out.N;
      const int64_t m0 = (int64_t)mt * BT;
      // this tile's token scales for the bulk-store epilogue: loaded now,
      // staged in shared memory once the first group has been waited for
      // (the load's latency hides behind that wait)
      float as_pending = 0.f;
      if constexpr (C::kTmaEpi && kCodes && !PARTIALS) {
        const int64_t m = m0 + col0 + r;
        if (r < HB && m < p.M) as_pending = __ldg(p.a_s + m);
      }
      const uint16_t* sp_tile = scale_ptr(nt, g0);
      // the next tile's first scale, fetched now and used after this tile
      uint16_t s_first_next = 0;
      if (kScaleFromGlobal && k + 1 < n_units) {
        int mt2, nt2;
        unit_tile(k + 1, mt2, nt2);
        s_first_next = __ldg(scale_ptr(nt2, g0));
      }
#pragma unroll
      for (int t = 0; t < HB; ++t) R[t] = 0.f;
      // per-group drains (nc == ng) index groups with gi and items with i
      for (int gi = 0; gi < nc; ++gi) {
        const int i = k * ng + gi;
        const int di = k * nc + gi;
        const int db = di % kNumD;
        float s = f16_bits_to_f32(s_next);
        if constexpr (kScaleFromGlobal)
          s_next = (gi + 1 < ng) ? __ldg(sp_tile + (int64_t)(gi + 1) * 4256) : s_first_next;
        if (!(ok && mbar_wait(dfull_bar(db), (di / kNumD) & 1, abort_flag, tmo))) {
          ok = false;
          if constexpr (!kUniformDrain) {
            break;
          } else {
            if constexpr (C::kDrainRendezvous) {
              if (i + 2 < n_items) {
                join(i + 2);
                next_join = i + 3;
              }
            }
            continue;
          }
        }
        if constexpr (C::kTmaEpi && kCodes && !PARTIALS) {
          if (gi == 0 && r < HB) as_stage[(k & 1) * BT + col0 + r] = as_pending;
        }
        tc_fence_after();
        float nz = 0.f;
        if constexpr (C::kFp8) {
          // this group's scale and zero point from the staged record (the
          // stage is not refilled before the drain warps release it; the
          // full-barrier phase is checked so that the copy's bytes are
          // visible here)
          const int st = i % S;
          if (!mbar_wait(full_bar(st), (i / S) & 1, abort_flag, tmo)) {
            ok = false;
            break;
          }
          const uint8_t* rec = stage_w_ptr(st);
          s = f16_bits_to_f32(*reinterpret_cast<const uint16_t*>(rec + 8192 + 2 * r));
          const uint32_t zb = rec[8448 + (r >> 1)];
          nz = -(float)((r & 1) ? (zb >> 4) : (zb & 0xF));
          __syncwarp();
          if (lane == 0) mbar_arrive(empty_bar(st));
        }
        if constexpr (C::kFp8) {
          // accumulator columns [0, BT): sum w * (a >> 4); [BT, 2BT): sum w * (a & 15);
          // 8 columns per load keep the drain's registers in budget
          constexpr int CW = 8;
#pragma unroll
          for (int cb = 0; cb < HB / CW; ++cb) {
            asm volatile("" ::: "memory");  // keep the chunks' loads apart
            uint32_t vh[16], vl[16];
            const uint32_t src = d_tmem + lane_base + db * C::kDCols + col0 + cb * CW;
            if constexpr (CW == 16) {
              tmem_ld16(src, vh);
              tmem_ld16(src + BT, vl);
            } else {
              tmem_ld8(src, vh);
              tmem_ld8(src + BT, vl);
            }
            // the tokens' group sums (the same for every row: L1 hits), read
            // while the loads are in flight; tokens past M read the last row
            // (their columns are never stored)
            float asf[CW];
            {
              const int32_t* asum_g = p.a_gsum + (g0 + gi);
              const int mfirst = (int)(m0 + col0) + cb * CW, mlast = (int)(p.M - 1);
#pragma unroll
              for (int q = 0; q < CW; ++q) {
                const int64_t ai = (int64_t)min(mfirst + q, mlast) * G + g0 + gi;
                asf[q] = dbg_ok((uint64_t)ai, 1, (uint64_t)p.M * G)
                             ? (float)__ldg(asum_g + min(mfirst + q, mlast) * G)
                             : 0.f;
              }
            }
            tmem_wait_ld();
#pragma unroll
            for (int q = 0; q < CW; ++q) {
              const int t = cb * CW + q;
              // integers below 2^24, so exact: P = sum a*w, Q = P - z*sum(a)
              const float P = fmaf(16.f, __uint_as_float(vh[q]), __uint_as_float(vl[q]));
              const float Q = fmaf(nz, asf[q], P);
              if constexpr (PARTIALS) {
                const int64_t m = m0 + col0 + t;
                if (m < p.M) p.partials[(m * N + n) * G + g0 + gi] = __float2int_rn(Q);
              } else {
                R[t] = fmaf(s, Q, R[t]);
              }
            }
          }
        } else {
        // columns per tcgen05.ld (8 at 64 columns per thread without the
        // register split: the 64 running sums leave room for no more at 96
        // registers; with it, 16)
        constexpr int CW =
            HB < 16 ? HB : (((HB >= 64 && !C::kRegSplit) || HB % 16) ? 8 : 16);
        static_assert(HB % CW == 0, "drain columns");
        constexpr int NCH = HB / CW;  // loads per drain
        // loads in flight per wait (32 columns at most with the register
        // split -- 48 in the 192-token tiles -- two loads without it)
        constexpr int kInFlight = C::kFull ? 48 : 32;
        constexpr int PAIR =
            C::kRegSplit ? (NCH < kInFlight / CW ? NCH : kInFlight / CW) : (NCH >= 2 ? 2 : 1);
        static_assert(NCH % PAIR == 0, "drain batches");
#pragma unroll
        for (int cb = 0; cb < NCH; cb += PAIR) {
          uint32_t v[PAIR][16];
#pragma unroll
          for (int q2 = 0; q2 < PAIR; ++q2) {
            if (cb + q2 >= NCH) break;
            const uint32_t src = d_tmem + lane_base + db * C::kDCols + col0 + (cb + q2) * CW;
            if constexpr (CW == 16) tmem_ld16(src, v[q2]);
            else tmem_ld8(src, v[q2]);
          }
          tmem_wait_ld();
          if (cb + PAIR >= NCH) {
            // the whole accumulator is in registers: release it before the
            // last batch's arithmetic (the MMAs two groups on wait for it)
            if constexpr (C::kDrainRendezvous) {
              if (i + 2 < n_items) {
                join(i + 2);
                next_join = i + 3;
              }
            } else {
              tc_fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive(dempty_bar(db));
            }
          }
#pragma unroll
          for (int q2 = 0; q2 < PAIR; ++q2) {
            if (cb + q2 >= NCH) break;
            if constexpr (PARTIALS) {
              const int g = g0 + gi;
#pragma unroll
              for (int q = 0; q < CW; ++q) {
                const int64_t m = m0 + col0 + (cb + q2) * CW + q;
                if (m < p.M)
                  p.partials[(m * N + n) * G + g] = __float2int_rn(__uint_as_float(v[q2][q]));
              }
            } else if constexpr (C::kIntAcc) {
              // exact: the group partial is an integer below 2^24 in fp32; the
              // running sum is kept as int32 bits in R
#pragma unroll
              for (int q = 0; q < CW; ++q) {
                float& Rq = R[(cb + q2) * CW + q];
                Rq = __int_as_float(__float_as_int(Rq) + __float2int_rn(__uint_as_float(v[q2][q])));
              }
            } else if constexpr (C::kWide && CW % 2 == 0) {
              // two columns a packed FMA (the same rounding as fmaf, half the
              // issue slots of the drain's arithmetic)
              const uint64_t s2 = f32x2_splat(s);
#pragma unroll
              for (int q = 0; q < CW; q += 2)
                fma_f32x2(R[(cb + q2) * CW + q], R[(cb + q2) * CW + q + 1], s2, v[q2][q],
                          v[q2][q + 1]);
            } else {
#pragma unroll
              for (int q = 0; q < CW; ++q)
                R[(cb + q2) * CW + q] = fmaf(s, __uint_as_float(v[q2][q]), R[(cb + q2) * CW + q]);
            }
          }
        }
        }  // kind::f16 drain (released the accumulator after its last load)
        if constexpr (C::kFp8) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(dempty_bar(db));
        }
      }
      if (!ok && !kUniformDrain) break;
      if constexpr (VARIANT == kW8A16) {
        const float sc = f16_bits_to_f32(__ldg(p.s8 + n));
#pragma unroll
        for (int t = 0; t < HB; ++t) R[t] *= sc;
      }
      if constexpr (C::kIntAcc) {  // W8A8: int32 sums -> s[n] * sum (a_s in store_row)
        const float sc = f16_bits_to_f32(__ldg(p.s8 + n));
#pragma unroll
        for (int t = 0; t < HB; ++t) R[t] = sc * (float)__float_as_int(R[t]);
      }
      if constexpr (!PARTIALS) {
        if (!cluster_reduce) {
          if constexpr (C::kTmaEpi) {
            epilogue_tma(R, k, m0, out);
          } else {
            store_row<VARIANT, HB>(R, p, out, m0 + col0, n);
          }
        }
      }
    }
    if constexpr (C::kDrainRendezvous) {
      while (next_join < n_items) join(next_join++);
    }
    if constexpr (C::kTmaEpi && !PARTIALS) {
      if (epi_thread) bulk_wait_group0();  // the last tile's stores have landed
    }
    __syncwarp();
    teardown_sync();
    if (cluster_reduce) {
      // one tile per CTA; every copy and MMA of this CTA has completed, so the
      // stages are free for the partial sums
      const int64_t n = out.n0 + r;
      const int64_t m0 = (int64_t)mt * BT;
      float* red = reinterpret_cast<float*>(smem);  // [BT][128]
#pragma unroll
      for (int t = 0; t < HB; ++t) red[(col0 + t) * 128 + r] = R[t];
      if constexpr (HB <= 16) {  // decode-sized tiles: the epilogue is on the critical path
        cluster_sync_all();
        float asv[HB];  // the tokens' scales, loaded before the reduction so
                        // that their latency overlaps it
        if (cluster_ctarank() == 0) {
#pragma unroll
          for (int t = 0; t < HB; ++t)
            asv[t] = (kCodes && m0 + col0 + t < p.M) ? __ldg(p.a_s + m0 + col0 + t) : 1.f;
          // every rank's partials of 4 columns are loaded before any is added
          // (one DSMEM round trip per 4 columns, not one per rank); the sums
          // keep rank order
          const uint32_t local = smem_u32(red);
          constexpr int TC = HB < 4 ? HB : 4;
#pragma unroll
          for (int t0 = 0; t0 < HB; t0 += TC) {
            float v[7][TC];
#pragma unroll
            for (int rk = 1; rk < 8; ++rk) {
              if (rk < p.ks) {
                const uint32_t remote = map_to_rank(local, rk);
#pragma unroll
                for (int tt = 0; tt < TC; ++tt)
                  v[rk - 1][tt] = ld_dsmem_f32(remote + ((col0 + t0 + tt) * 128 + r) * 4);
              }
            }
#pragma unroll
            for (int rk = 1; rk < 8; ++rk) {
              if (rk < p.ks) {
#pragma unroll
                for (int tt = 0; tt < TC; ++tt) R[t0 + tt] += v[rk - 1][tt];
              }
            }
          }
        }
        cluster_sync_all();
        if (cluster_ctarank() == 0) {
          store_row_scaled<HB>(R, asv, p, out, m0 + col0, n);
        }
      } else {
        // wide tiles: reduce-scatter. Rank k sums the tile's columns
        // [k * sw, (k + 1) * sw) over every rank's partials, in rank order
        // (the order of a reduction by one rank), and stores them, so that
        // each SM takes in 1/ks of the partial sums through DSMEM.
        cluster_sync_all();
        const int ks = p.ks;
        const int sw = (BT + ks - 1) / ks;
        const int rank = (int)cluster_ctarank();
        const int c_lo = max(rank * sw, col0), c_hi = min(rank * sw + sw, col0 + HB);
        uint32_t rb[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) rb[j] = j < ks ? map_to_rank(smem_u32(red), j) : 0u;
        for (int c = c_lo; c < c_hi; ++c) {
          const uint32_t off = (uint32_t)((c * 128 + r) * 4);
          float v[8];
#pragma unroll
          for (int j = 0; j < 8; ++j) v[j] = j < ks ? ld_dsmem_f32(rb[j] + off) : 0.f;
          float acc = v[0];
#pragma unroll
          for (int j = 1; j < 8; ++j)
            if (j < ks) acc += v[j];
          const int64_t m = m0 + c;
          if (m < p.M) {
            if constexpr (kCodes) acc *= __ldg(p.a_s + m);
            out.y[m * out.N + n] = f32_to_bf16_bits(acc);
          }
        }
        cluster_sync_all();  // no rank leaves while another reads its partials
      }
    }
  };

  // Role dispatch. With the register split each warpgroup changes its budget
  // first, inside its own branch (so the budget covers all of the role's code).
  if constexpr (C::kRegSplit) {
    const int wg = warp >> 2;
    if (wg >= C::kDrainWGs + C::kConvSets) {
      setmaxnreg_dec<C::kRegOther>();
      if (warp == C::kProducerWarp) {
        if constexpr (C::kSplitRings) producer_role(std::true_type{}, std::false_type{});
        else producer_role(std::true_type{}, std::true_type{});
      } else if (warp == C::kActWarp) {
        producer_role(std::false_type{}, std::true_type{});
      } else if (warp >= C::kWarpsUsed) {
        pad_role();
      } else {
        mma_role();
      }
    } else if (wg >= C::kDrainWGs) {
      setmaxnreg_dec<C::kRegConv>();
      conv_role();
    } else {
      setmaxnreg_inc<C::kRegDrain>();
      drain_role();
    }
  } else {
    static_assert(!C::kSplitRings, "split rings run with the register split");
    if (warp == C::kProducerWarp) producer_role(std::true_type{}, std::true_type{});
    else if (warp >= C::kMmaWarp) mma_role();
    else if (warp >= kConvWarp0) conv_role();
    else drain_role();
  }
}

// ---- bounded-wait self test -----------------------------------------------------
__global__ void selftest_timeout_kernel(uint64_t timeout_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  // nothing ever arrives on `bar`: the wait must give up and flag a timeout
  if (threadIdx.x == 0) mbar_wait(smem_u32(&bar), 0, &abort_flag, timeout_ns);
  __syncthreads();
}

cudaError_t launch_selftest_timeout(uint64_t timeout_ns, cudaStream_t st) {
  selftest_timeout_kernel<<<1, 32, 0, st>>>(timeout_ns);
  return cudaGetLastError();
}

// ---- host side ----------------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  }
  return fn;
}

// 2-D row-major [rows][cols] tensor, box {box_cols, box_rows}, 128-byte swizzle.
static bool make_map(CUtensorMap* map, CUtensorMapDataType dt, int elem_bytes, const void* ptr,
                     int64_t rows, int64_t cols, int box_cols, int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)(cols * elem_bytes)};
  cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, dt, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Activations [rows][cols] seen as 3-D {64, rows, cols/64}: a box {64, box_rows,
// 2} lands as two [box_rows][64] swizzled tiles back to back, i.e. one copy per
// 128-wide group instead of two.
static bool make_act_map_3d(CUtensorMap* map, CUtensorMapDataType dt, const void* ptr, int64_t rows,
                            int64_t cols, int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn || cols % 64) return false;
  cuuint64_t dims[3] = {64, (cuuint64_t)rows, (cuuint64_t)(cols / 64)};
  cuuint64_t strides[2] = {(cuuint64_t)(cols * 2), 128};
  cuuint32_t box[3] = {64, (cuuint32_t)box_rows, 2};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, dt, 3, const_cast<void*>(ptr), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// The two e4m3 activation planes [2][rows][cols] bytes as a 3-D map {cols,
// rows, 2}; a box {128, box_rows, 2} lands as [2][box_rows][128] swizzled.
static bool make_act_map_planes(CUtensorMap* map, const void* ptr, int64_t rows, int64_t cols,
                                int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {(cuuint64_t)cols, (cuuint64_t)rows, 2};
  cuuint64_t strides[2] = {(cuuint64_t)cols, (cuuint64_t)(rows * cols)};
  cuuint32_t box[3] = {128, (cuuint32_t)box_rows, 2};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(ptr), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

static int tc_sm_count() {
  const int n = device_sm_count();
  return n > 0 ? n : 148;
}

// Split of the work over the GPU. With enough tiles, a persistent grid (one
// CTA per SM) strides over them with all of K; otherwise each tile's K groups
// are split over a cluster of ks CTAs. ks minimises rounds * groups-per-unit.
static void choose_split(int64_t tiles, int G, int sms, double split_cost, bool one_wave,
                         int* ks_out, int* persistent_out) {
  // enough tiles to fill the GPU: persistent, all of K per tile
  if (tiles >= sms) {
    *ks_out = 1;
    *persistent_out = 1;
    return;
  }
  // otherwise split K over a cluster, one round, as many SMs busy as possible
  // (a split costs `split_cost` groups of prologue and reduction per CTA)
  double best = 1e30;
  int best_ks = 1;
  for (int ks = 1; ks <= 8 && ks <= G; ++ks) {
    const int64_t units = tiles * ks;
    if (one_wave && ks > 1 && units > sms) break;
    const int64_t rounds = (units + sms - 1) / sms;
    const double cost = (double)rounds * ((G + ks - 1) / ks + (ks > 1 ? split_cost : 0.0));
    if (cost < best - 1e-9) {
      best = cost;
      best_ks = ks;
    }
  }
  *ks_out = best_ks;
  *persistent_out = 0;
}

// Grid plan of one GEMM: a persistent grid over the first `units` tiles of the
// banded order and, for wide tiles whose last round would leave most SMs idle,
// a second launch splitting the remaining `tail` tiles' K over clusters of
// `tail_ks` CTAs; or, with too few tiles to fill the GPU, one split-K grid
// over all tiles (persistent = 0, split ks).
struct GridPlan {
  int persistent = 0;
  int ks = 1;
  int64_t units = 0, tail = 0;
  int tail_ks = 1;
  double cost = 0.0;  // CTA time in groups of one unit of this width
};

// the second launch of a split tail, in groups of a full-grid CTA: its launch
// behind the first, pipeline fill, cluster reduction and stores (measured on
// GB300: ~14 us beside the split groups' own time, ~26 groups of 192 tokens;
// so the 3584 x 18944 linear at 4096 tokens takes a tail, 386 -> 334 us,
// and the 3584 x 3584 one, 28 groups a tile, does not)
constexpr double kTailLaunchCost = 24.0;

static GridPlan plan_grid(int64_t tiles, int G, int sms, bool wide) {
  GridPlan g;
  const double split_cost = wide ? 2.0 : 1.0;
  choose_split(tiles, G, sms, split_cost, wide, &g.ks, &g.persistent);
  if (!g.persistent) {
    const int64_t units = tiles * g.ks;
    g.cost = (double)((units + sms - 1) / sms) *
             ((G + g.ks - 1) / g.ks + (g.ks > 1 ? split_cost : 0.0));
    return g;
  }
  const int64_t rounds = (tiles + sms - 1) / sms;
  g.units = tiles;
  g.cost = (double)rounds * G;
  if (!wide || rounds < 2) return g;
  const int64_t tail = tiles - (rounds - 1) * sms;
  int ks = 1;
  for (int k = 2; k <= 8 && k <= G && tail * k <= sms; ++k) ks = k;
  if (ks < 2) return g;
  const double split = (double)(rounds - 1) * G + (G + ks - 1) / ks + split_cost + kTailLaunchCost;
  if (split < g.cost) {
    g.units = (rounds - 1) * sms;
    g.tail = tail;
    g.tail_ks = ks;
    g.cost = split;
  }
  return g;
}

// Band height (in m-tiles) for the persistent tile order, which walks bands of
// `band` m-tiles with m fastest inside a band: each weight tile is read from
// DRAM once per band, each activation tile once if the band's activations stay
// in L2. So DRAM traffic is lowest when one operand stays L2-resident while
// the other streams once: all m-tiles in one band when the whole activation
// matrix fits the L2 budget (weights stream once), one m-tile a band (n
// fastest) when the whole weight matrix fits (activations stream once),
// otherwise the tallest band whose activation tiles fit.
static int choose_band(int64_t m_tiles, int64_t n_tiles, double act_tile, double w_tile) {
  constexpr double kL2Budget = 48e6;  // bytes of one operand kept resident (129 MB L2)
  if (m_tiles * act_tile <= kL2Budget) return (int)m_tiles;
  if (n_tiles * w_tile <= kL2Budget) return 1;
  int band = (int)(kL2Budget / act_tile);
  if (band < 1) band = 1;
  if (band > m_tiles) band = (int)m_tiles;
  return band;
}

template <int VARIANT, int BT, bool PARTIALS>
static cudaError_t launch_tc(const GemmArgs& a, cudaStream_t st) {
  using C = TcCfg<VARIANT, BT>;
  CUtensorMap act_map, w8_map;
  memset(&w8_map, 0, sizeof(w8_map));
  constexpr bool kCodes = (VARIANT == kW4A8 || VARIANT == kW8A8);  // quantized activations
  const void* act_ptr = kCodes ? (const void*)a.a_tc : (const void*)a.x;
  const CUtensorMapDataType adt =
      kCodes ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  int act3d = 0;
  if constexpr (C::kFp8) {
    if (!make_act_map_planes(&act_map, act_ptr, a.M, a.K, BT)) return cudaErrorInvalidValue;
  } else {
    act3d = make_act_map_3d(&act_map, adt, act_ptr, a.M, a.K, BT) ? 1 : 0;
    if (!act3d && !make_map(&act_map, adt, 2, act_ptr, a.M, a.K, 64, BT))
      return cudaErrorInvalidValue;
  }
  if constexpr (C::kW16) {
    if (!make_map(&w8_map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.w16, a.N, a.K, 64, 128))
      return cudaErrorInvalidValue;
  } else if constexpr (C::kW8) {
    if (!make_map(&w8_map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, a.w8, a.N, a.K, 128, 128))
      return cudaErrorInvalidValue;
  }
  const int G = (int)(a.K / 128);
  const int64_t m_tiles = (a.M + BT - 1) / BT;
  const int64_t n_tiles = a.N / 128;
  const int64_t tiles = m_tiles * n_tiles;
  if (m_tiles > 65535 || n_tiles > 65535 || tiles >= (1LL << 31)) return cudaErrorInvalidValue;
  const int sms = tc_sm_count() * C::kCtasPerSm;  // CTA slots of one wave
  // (wide tiles reduce 128 x BT partial sums through DSMEM, about two groups'
  // worth, and split only while every CTA of the split fits one wave: a
  // second wave of split clusters measured slower than no split, e.g. the
  // 3584 x 3584 linear at 512 tokens 53 us split four ways against 23 us)
  const GridPlan plan = plan_grid(tiles, G, sms, C::kWide);
  const int ks = plan.ks, persistent = plan.persistent;
  TcParams p{};
  p.M = a.M;
  p.N = a.N;
  p.K = a.K;
  p.G = G;
  p.ks = ks;
  p.m_tiles = (int)m_tiles;
  p.n_tiles = (int)n_tiles;
  p.persistent = persistent;
  p.units = (int)plan.units;
  p.tail_base = (int)plan.units;
  p.act3d = act3d;
  p.band = persistent ? choose_band(m_tiles, n_tiles, (double)BT * a.K * 2.0,
                                    (double)128 * a.K * (C::kW16 ? 2.0 : (C::kW8 ? 1.0 : 0.5)))
                      : 1;
  p.a_s = a.a_s;
  p.a_gsum = a.a_gsum;
  p.s8 = a.s8;
  p.partials = a.partials;
  p.seg = seg_table(a);
  p.timeout_ns = a.timeout_ns;
  YMaps ymaps;
  memset(&ymaps, 0, sizeof(ymaps));
  if constexpr (C::kTmaEpi && !PARTIALS) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return cudaErrorInvalidValue;
    for (int j = 0; j < p.seg.count; ++j) {
      cuuint64_t dims[2] = {(cuuint64_t)p.seg.N[j], (cuuint64_t)a.M};
      cuuint64_t strides[1] = {(cuuint64_t)(p.seg.N[j] * 2)};
      cuuint32_t box[2] = {128, (cuuint32_t)C::kDrainCols};
      cuuint32_t estr[2] = {1, 1};
      if (fn(&ymaps.map[j], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p.seg.y[j], dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
             CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    }
  }
  auto kern = tc_gemm_kernel<VARIANT, BT, PARTIALS>;
  // opt-in to the large shared-memory carve-out, once per device
  static SmemOptIn opt_in;
  if (cudaError_t e = opt_in.ensure(kern, C::kSmemBytes); e != cudaSuccess) return e;
  if constexpr (C::kRegSplit) {
    // the warpgroups' register budgets must fit in what the block is launched
    // with, or a setmaxnreg increase would wait for ever (checked once: the
    // register count is a property of the compiled kernel)
    static std::atomic<int> regs_ok{0};  // 0 unchecked, 1 fits, 2 does not
    if (regs_ok.load(std::memory_order_relaxed) == 0) {
      cudaFuncAttributes fa;
      cudaError_t e = cudaFuncGetAttributes(&fa, kern);
      if (e != cudaSuccess) return e;
      regs_ok.store(C::kDrainWGs * C::kRegDrain + C::kConvSets * C::kRegConv + C::kRegOther <=
                            (C::kWarps / 4) * fa.numRegs
                        ? 1
                        : 2,
                    std::memory_order_relaxed);
    }
    if (regs_ok.load(std::memory_order_relaxed) != 1) return cudaErrorInvalidConfiguration;
  }
  cudaLaunchConfig_t cfg = {};
  if (persistent)
    cfg.gridDim = dim3((unsigned)(plan.units < sms ? plan.units : sms), 1, 1);
  else
    cfg.gridDim = dim3((unsigned)ks, (unsigned)m_tiles, (unsigned)n_tiles);
  cfg.blockDim = dim3(C::kThreads, 1, 1);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = persistent ? 1u : (unsigned)ks;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kern, act_map, w8_map, p, ymaps);
  if (e != cudaSuccess || plan.tail == 0) return e;
  // the split tail: the last tiles of the banded order, K over clusters
  p.persistent = 2;
  p.ks = plan.tail_ks;
  cfg.gridDim = dim3((unsigned)plan.tail_ks, (unsigned)plan.tail, 1);
  attr[0].val.clusterDim.x = (unsigned)plan.tail_ks;
  return cudaLaunchKernelEx(&cfg, kern, act_map, w8_map, p, ymaps);
}

// Time of a grid of `bt`-token wide tiles in units of one group of one
// 128-token tile: the cost of the grid plan_grid makes, times the relative
// cost of a group at that width.
static double wide_grid_cost(int64_t M, int64_t n_tiles, int G, int sms, int bt,
                             bool wide = true) {
  // one 192-token group against one 128-token group, CTA time in a full grid
  // (measured on GB300 over the 7B prefill shapes: 1.0-1.14 as the 192-token
  // kernel improved; every value in that range makes the same choices there)
  constexpr double kFullGroupCost = 1.12;
  const int64_t tiles = ((M + bt - 1) / bt) * n_tiles;
  return plan_grid(tiles, G, sms, wide).cost * (bt == kFullBT ? kFullGroupCost : 1.0);
}

int tc_token_tile(int variant, int64_t M, int64_t N, int64_t K) {
  if (M <= 16) return 16;
  if (M <= 32) return 32;
  if (M <= 64) return 64;
  // above 64 tokens every variant takes 192 tokens unless that grid costs
  // more (the int8-weight variants without the per-group tiles' split tails
  // and one-wave splits)
  if (variant == kW4A8 || variant == kW4A16 || variant == kW16A16 || variant == kW8A16 ||
      variant == kW8A8) {
    const int sms = tc_sm_count();
    const int G = (int)(K / 128);
    const int64_t n_tiles = N / 128;
    const bool wide = variant != kW8A16 && variant != kW8A8;  // (split tails, one-wave splits)
    return wide_grid_cost(M, n_tiles, G, sms, kFullBT, wide) <
                   wide_grid_cost(M, n_tiles, G, sms, kWideBT, wide)
               ? kFullBT
               : kWideBT;
  }
  return 128;
}

int tc_launches(int variant, int64_t M, int64_t N, int64_t K) {
  const int bt = tc_token_tile(variant, M, N, K);
  const bool per_group = (variant == kW4A8 || variant == kW4A16 || variant == kW16A16);
  if (bt <= 64 || !per_group) return 1;  // (only wide per-group tiles split a tail)
  const int64_t tiles = ((M + bt - 1) / bt) * (N / 128);
  return plan_grid(tiles, (int)(K / 128), tc_sm_count(), true).tail > 0 ? 2 : 1;
}

template <int VARIANT, bool PARTIALS>
static cudaError_t launch_tc_bt(const GemmArgs& a, cudaStream_t st) {
  constexpr bool kPerGroup = (VARIANT == kW4A8 || VARIANT == kW4A16 || VARIANT == kW16A16);
  switch (tc_token_tile(VARIANT, a.M, a.N, a.K)) {
    case 16:
      return launch_tc<VARIANT, 16, PARTIALS>(a, st);
    case 32:
      return launch_tc<VARIANT, 32, PARTIALS>(a, st);
    case 64:
      return launch_tc<VARIANT, 64, PARTIALS>(a, st);
    case kFullBT:
      if constexpr (kPerGroup || VARIANT == kW8A16 || VARIANT == kW8A8)
        return launch_tc<VARIANT, kFullBT, PARTIALS>(a, st);
      break;
    default:
      return launch_tc<VARIANT, 128, PARTIALS>(a, st);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_tc_gemm(const GemmArgs& a, cudaStream_t st) {
  if (a.M == 0) return cudaSuccess;
  switch (a.variant) {
    case kW4A8:
      return a.partials ? launch_tc_bt<kW4A8, true>(a, st) : launch_tc_bt<kW4A8, false>(a, st);
    case kW4A16:
      return launch_tc_bt<kW4A16, false>(a, st);
    case kW8A16:
      return launch_tc_bt<kW8A16, false>(a, st);
    case kW16A16:
      return launch_tc_bt<kW16A16, false>(a, st);
    case kW8A8:
      // the fp16 activation-code form exists for M > kTcFp8MaxM only (the
      // e4m3 planes below it are specific to 4-bit weights); smaller M run
      // on the GEMV
      if (a.M <= kTcFp8MaxM) return cudaErrorNotSupported;
      if (tc_token_tile(kW8A8, a.M, a.N, a.K) == kFullBT)
        return launch_tc<kW8A8, kFullBT, false>(a, st);
      return launch_tc<kW8A8, 128, false>(a, st);
  }
  return cudaErrorInvalidValue;
}

cudaError_t take_error_word_tc_gemm(unsigned* out) { return take_local_error_word(out); }
cudaError_t set_record_limit_tc_gemm(unsigned long long bytes) {
  return set_local_record_limit(bytes);
}

}  // namespace egopq
