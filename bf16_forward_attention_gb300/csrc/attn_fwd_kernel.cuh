// attn_fwd_kernel.cuh - fused bf16 forward attention for sm_103a (GB300).
//
// Computes O = softmax(Q K^T * scale) V for head_dim 128 (snilld.dk,
// "Open source attention-kernel i HIP slaar AITER v3 paa MI300X", sections
// "Hvordan kernen arbejder" and "Hvad er udgivet"), rounding the output to bf16
// per mode (same article, "Numerik samlet eet sted").
//
// One CTA owns two 128-row query tiles of one (batch, head) and streams every
// 128-key tile of K and V through a 4-stage shared-memory ring. Roles (warps):
//   warp 0      TMA producer: Q tiles once, then K_0, V_0, K_1, V_1, ...
//   warp 1      TMEM allocator and the single tcgen05.mma issuer
//   warps 2-3   causal and variable-length variants: check V of the key tiles
//               where some row hides keys for NaN / Inf (see "V check" below);
//               otherwise idle (they complete the first warpgroup)
//   warps 4-7   softmax + epilogue of query tile 0 (one TMEM lane = one row)
//   warps 8-11  softmax + epilogue of query tile 1
// The launch gives every thread 168 registers; the first warpgroup hands most of
// its share to the two softmax warpgroups (40 + 2 * 232 = 3 * 168), which each
// keep a 128-float output row per thread.
// Tensor memory (512 columns): O0 [0,128), O1 [128,256), S0/P0 [256,384),
// S1/P1 [384,512). The MMA order per key tile j is
//   PV0_j, S0_{j+1}, PV1_j, S1_{j+1}
// so the tensor pipe computes one tile's products while the other tile's
// softmax runs (the pages' "keep the matrix core busy while softmax and loads
// overlap", section "Hvordan kernen arbejder").
//
// The persistent variant (short key ranges) runs one CTA per SM over many such
// items with the same roles, carrying every barrier phase from item to item:
// the next item's Q loads as soon as the current item's last S MMAs are done,
// and each softmax warp stores its rows through a 4 KiB staging buffer of its
// own rather than through the Q buffer.
// Its short forms take items of one ragged key tile, or of 2 to 4 tiles ending
// in a ragged one: each S tile is read from TMEM once into registers for both
// softmax passes, the partial output stays in TMEM until the epilogue, and P V
// and the exponentials stop at the last 16-key chunk that holds a key.
//
// The pair variant (opt-in, for the last, partial wave of a launch) runs each
// item on a 2-CTA cluster, each CTA taking one half of the key tiles; the
// second CTA sends its unnormalised rows, running max and row sum to the first
// through distributed shared memory, and the first merges them and stores.
//
// Softmax is the online (running-max) form in base 2 with a lazy rescale: the
// running output and row sum are rescaled only when a tile's max exceeds the max
// in use by more than kTau (log2 units). P is written back into the S columns as
// two bf16 terms, P_hi = bf16(p) and P_lo = bf16(p - P_hi), and both products
// are accumulated, so the weights carry ~16 significant bits. With P in bf16
// alone only ~87% of outputs land within 1 bf16 ULP of the exact result on
// unit-normal inputs; the two-term P keeps ~99.98% there.
//
// The tensor pipe's fp32 accumulation truncates; summed over tens of thousands
// of keys that bias costs ~0.3% (32K keys) to ~1.5% (128K keys) of outputs their
// 1-ULP bound. So the PV products accumulate in TMEM over at most kFoldEvery
// key tiles (64 MMAs deep), after which each softmax thread adds that partial
// into its row's 128 fp32 registers, rounding to nearest, and the next partial
// starts fresh.
//
// Every wait is bounded in time. A wait that expires sets a device status word,
// raises a CTA-wide abort flag, and every role then stops, waits for its own
// asynchronous copies and MMAs, frees tensor memory and returns.
#pragma once
#include <cuda.h>
#include <stdint.h>

#include <utility>

#include "ptx.cuh"

namespace attn {

constexpr int kD = 128;                     // head dimension
constexpr int kBM = 128;                    // query rows per tile
constexpr int kBN = 128;                    // keys per tile
constexpr int kQTiles = 2;                  // query tiles per CTA
constexpr int kStages = 4;                  // K/V ring depth (K and V tiles share it)
constexpr int kTileBytes = kBM * kD * 2;    // 32 KiB: one 128 x 128 bf16 tile
constexpr int kHalfBytes = kTileBytes / 2;  // 16 KiB: 128 rows x 64 columns (one TMA box)
constexpr int kThreads = 384;
constexpr int kSoftmaxWarp0 = 4;
constexpr int kLaunchRegs = 168;     // per thread at launch: 65536 / 384, rounded to 8
constexpr uint32_t kRegsLow = 40;    // producer / MMA warpgroup after the split
constexpr uint32_t kRegsHigh = 232;  // each softmax warpgroup after the split
static_assert(kRegsLow + 2 * kRegsHigh == 3 * kLaunchRegs, "register split");
constexpr uint32_t kTmemCols = 512;
constexpr float kTau = 8.0f;  // lazy-rescale threshold (factor 256)
// The tensor pipe accumulates P V over kFoldEvery key tiles in TMEM; then the
// softmax threads fold that partial output into their fp32 registers (the
// pipe's fp32 accumulation truncates, so a partial must not grow too long).
// (The split-KV variant once folded every tile; every 4 tiles measured 3-5%
// faster on decode-like shapes.)
constexpr int kFoldEvery = 4;
// Items of at most this many key tiles never fold (the short persistent variant).
constexpr int kShortMaxKvTiles = kFoldEvery;
template <bool kPartial>
constexpr int kFoldOf = kFoldEvery;

enum : int {
  kBarQ = 0,
  kBarKvFull = 1,
  kBarKvEmpty = kBarKvFull + kStages,
  kBarSFull = kBarKvEmpty + kStages,
  kBarPFull = kBarSFull + kQTiles,
  kBarOFull = kBarPFull + kQTiles,
  kBarDrain = kBarOFull + kQTiles,
  kBarQFree = kBarDrain + 1,  // persistent: the Q buffer may be refilled (next item)
  kBarOFree = kBarQFree + 1,  // persistent, per query tile: the epilogue has read O
  kBarVChk = kBarOFree + kQTiles,  // key-limit variants: V of masked tile m checked (m < 3)
  kBarVLanded = kBarVChk + 3,      // key-limit variants: V of masked tile m is in the ring
  kBarPeerReady = kBarVLanded + 3,  // pair variant, rank 1: rank 0's ring is free for the exchange
  kBarReceived = kBarPeerReady + 1, // pair variant, rank 0: rank 1's partial rows have arrived
  kBarCount = kBarReceived + 1
};

constexpr int kOffQ = 0;
constexpr int kOffRing = kOffQ + kQTiles * kTileBytes;
constexpr int kOffBar = kOffRing + kStages * kTileBytes;
constexpr int kOffTmemSlot = kOffBar + kBarCount * 8;
constexpr int kOffAbort = kOffTmemSlot + 4;
constexpr int kSmemUsed = kOffAbort + 4;
constexpr int kSmemBytes = kSmemUsed + 1024;  // slack to align the base to 1024 B
static_assert(kSmemBytes <= 232448, "shared memory budget");
// Variants with a key limit per row (causal, variable-length batch): a record of
// the non-finite values found in V of each masked key tile (at most 3 per CTA):
// a flag word, a 128-bit mask of the keys that hold one, and per key three
// 128-bit column masks (NaN, +Inf, -Inf). 388 words per tile.
constexpr int kMaxMaskedTiles = 3;
constexpr int kVRecWords = 4 + 4 + 3 * kBN * 4;
constexpr int kVRecKeyMask = 4, kVRecNan = 8, kVRecPos = kVRecNan + kBN * 4,
              kVRecNeg = kVRecPos + kBN * 4;
constexpr int kOffVRec = (kSmemUsed + 15) & ~15;
constexpr int kSmemBytesRowLimit = kOffVRec + kMaxMaskedTiles * kVRecWords * 4 + 1024;
static_assert(kSmemBytesRowLimit <= 232448, "shared memory budget (key-limit variants)");
// Pair variant: rank 1 sends its 256 unnormalised rows into rank 0's K/V ring
// (256 x 512 bytes, the whole ring) and its (reference max, row sum) pairs here.
constexpr int kOffPairMl = (kSmemUsed + 15) & ~15;
constexpr int kSmemBytesPair = kOffPairMl + 2 * kBM * 8 + 1024;
static_assert(kSmemBytesPair <= 232448, "shared memory budget (pair variant)");
static_assert(kStages * kTileBytes == 2 * kBM * kD * 4, "the ring holds one CTA's fp32 rows");
// The persistent variant also stages its output: 4 KiB per softmax warp (32
// rows x 64 columns, one TMA box), so that the Q buffer can be refilled for the
// next item while the current one is being stored.
constexpr int kStageWarpBytes = 32 * 128;
constexpr int kOffStage = (kSmemUsed + 1023) & ~1023;
constexpr int kSmemBytesPersist = kOffStage + 8 * kStageWarpBytes + 1024;
static_assert(kSmemBytesPersist <= 232448, "shared memory budget (persistent)");

constexpr uint32_t kTmemO0 = 0, kTmemS0 = 256;

struct Params {
  int Sq, Sk, H;
  int n_qpairs;  // ceil(Sq / 256)
  int kv_tiles;  // ceil(Sk / 128)
  int kv_tail;   // valid keys in the last key tile, 1..128
  int n_splits;  // key-range splits (1: whole range per CTA, bf16 output)
  int BH;        // B * H
  int sq_pad;    // n_qpairs * 256: row pitch of the split workspace
  float* part_o;   // split workspace: [split][b*H + h][sq_pad][128] unnormalised O
  float* part_rl;  // split workspace: [split][b*H + h][sq_pad][2] (reference max, row sum)
  int layout;    // 0 = BHSD, 1 = BSHD
  int mode;      // 0 = RTNE, 1 = RTNA, 2 = RTZ
  float c;       // scale * log2(e)
  unsigned long long timeout_ns;
  int withhold_s0;  // self-test of the timeout path: never signal query tile 0's first S
  int group;        // query heads per key/value head (grouped-query attention)
  int causal;       // 1: key j visible to query i iff j <= i + Sk - Sq (per sequence)
  // Variable-length batch (packed tokens; the tensor maps then have B = 1 and
  // S = total tokens, and B above is the number of sequences):
  const int* cu_q;  // B + 1 query offsets (device memory)
  const int* cu_k;  // B + 1 key offsets
  int max_sq;       // bound on every sequence's query length (sizes the grid)
  uint16_t* out;    // output base, for rows stored without TMA
  int head_group;   // causal: (batch, head) items scheduled together, longest first
  int dbg_poison;   // debug build only: report one failed check (tests the reporting)
  int n_items;      // persistent variant: work items; CTA c takes c, c + gridDim.x, ...
  int item_base;    // pair variant: the work item of block 0 (CTA b takes item_base + b)
  int early_dependents;  // base variant: a pair launch follows and may start early
};

// Bit 0: some wait timed out. Bit 1: a variable-length batch's offsets were
// invalid (that sequence's output is left unwritten). Bit 2 (debug build): a
// bounds or protocol check failed.
__device__ unsigned int g_attn_status;

// Debug build (-DATTN_DEBUG=1): dbg_ok(cond) records a failed check in bit 2 of
// the status word and returns cond, so that the caller can skip the access it
// guards; no trap, no assert. In the release build it is the constant true and
// the checks compile away.
#ifndef ATTN_DEBUG
#define ATTN_DEBUG 0
#endif
__device__ __forceinline__ bool dbg_ok(bool cond) {
#if ATTN_DEBUG
  if (!cond) atomicOr(&g_attn_status, 4u);
  return cond;
#else
  (void)cond;
  return true;
#endif
}

// Shared-memory matrix descriptor, 128-byte swizzle (tcgen05 format: start,
// leading and stride byte offsets in 16-byte units, version 1, layout 2). Every
// operand here has a 1024-byte stride between 8-row groups, so the upper word is
// one constant and only the lower word (start address, leading offset) varies.
constexpr uint32_t kDescHi = (1024u >> 4) | (1u << 14) | (2u << 29);

__device__ __forceinline__ uint32_t desc_lo(uint32_t saddr, uint32_t lbo) {
  return ((saddr & 0x3FFFFu) >> 4) | ((lbo >> 4) << 16);
}

__device__ __forceinline__ uint64_t desc_of(uint32_t lo) {
  return (static_cast<uint64_t>(kDescHi) << 32) | lo;
}

// Instruction descriptor, kind::f16: fp32 accumulator, bf16 A and B, A K-major,
// B K-major (0) or MN-major (1), shape M x N.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, int b_mn_major) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(b_mn_major) << 16) |
         (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

// Waits for `parity` on `bar` for at most timeout_ns. On expiry: sets the abort
// flag and the device status, returns false. With honor_abort, also returns
// false as soon as another thread has raised the abort flag.
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          unsigned long long timeout_ns, bool honor_abort) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = ptx::globaltimer();
  while (true) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    if (honor_abort && *abort_flag) return false;
    if (ptx::globaltimer() - t0 > timeout_ns) {
      *abort_flag = 1;
      atomicOr(&g_attn_status, 1u);
      return false;
    }
  }
}

// The same for a barrier that a CTA of the cluster arrives on remotely (acquire
// at cluster scope); phase 0 only (each such barrier completes once).
__device__ __forceinline__ bool wait_bounded_cluster(uint32_t bar, volatile int* abort_flag,
                                                  unsigned long long timeout_ns) {
  if (ptx::mbar_try_wait_cluster(bar, 0)) return true;
  const uint64_t t0 = ptx::globaltimer();
  while (true) {
    if (ptx::mbar_try_wait_cluster(bar, 0)) return true;
    if (*abort_flag) return false;
    if (ptx::globaltimer() - t0 > timeout_ns) {
      *abort_flag = 1;
      atomicOr(&g_attn_status, 1u);
      return false;
    }
  }
}

__device__ __forceinline__ void tma_coords(int layout, int s, int h, int& c1, int& c2) {
  // BHSD maps are (d, S, H, B); BSHD maps are (d, H, S, B).
  if (layout == 0) {
    c1 = s;
    c2 = h;
  } else {
    c1 = h;
    c2 = s;
  }
}

// Moving an operand's start address by b bytes adds b >> 4 to the descriptor's
// lower word: the address field holds bits 4..17 and every shared address here
// is below 256 KiB, so the add never carries out of the field.

// S = Q K_j^T: 8 MMAs of K = 16 over head_dim; both operands K-major SW128.
// Step kk starts 32 bytes further into a 128-byte swizzle row; steps 4..7 use
// the second 64-column half, 16 KiB further.
template <int... kK>
__device__ __forceinline__ void issue_s_seq(uint32_t tmem_d, uint32_t q_lo, uint32_t k_lo,
                                            std::integer_sequence<int, kK...>) {
  constexpr uint32_t idesc = idesc_bf16(kBM, kBN, 0);
  (ptx::mma_ss_imm<((kK >> 2) << 10) + ((kK & 3) << 1), ((kK >> 2) << 10) + ((kK & 3) << 1)>(
       tmem_d, q_lo, k_lo, kDescHi, idesc, kK > 0 ? 1u : 0u),
   ...);
}

__device__ __forceinline__ void issue_s(uint32_t tmem_d, uint32_t q_lo, uint32_t k_lo) {
  issue_s_seq(tmem_d, q_lo, k_lo, std::make_integer_sequence<int, 8>{});
}

// O += P_hi V_j + P_lo V_j, into a fresh accumulator unless `accumulate`. P is
// in TMEM (A operand):
// the 16 columns of key chunk u (keys 16u..16u+15) hold P_hi in their first 8
// and P_lo in their last 8 columns, two bf16 per column. V_j (keys x head_dim,
// head_dim contiguous) is the B operand in MN-major SW128: 8-key groups 1024 B
// apart, the two 64-column halves 16 KiB apart (the leading offset); 16 keys
// are 2048 bytes.
template <int... kK>
__device__ __forceinline__ void issue_pv_seq(uint32_t tmem_o, uint32_t tmem_p, uint32_t v_lo,
                                             uint32_t accumulate,
                                             std::integer_sequence<int, kK...>) {
  constexpr uint32_t idesc = idesc_bf16(kBM, kD, 1);
  ((ptx::mma_ts_imm<16 * kK, (kK << 7)>(tmem_o, tmem_p, v_lo, kDescHi, idesc,
                                         kK == 0 ? accumulate : 1u),
    ptx::mma_ts_imm<16 * kK + 8, (kK << 7)>(tmem_o, tmem_p, v_lo, kDescHi, idesc, 1u)),
   ...);
}

__device__ __forceinline__ void issue_pv(uint32_t tmem_o, uint32_t tmem_p, uint32_t v_lo,
                                         uint32_t accumulate) {
  issue_pv_seq(tmem_o, tmem_p, v_lo, accumulate, std::make_integer_sequence<int, 8>{});
}

// The same over the first n key chunks only (1 <= n <= 8): the ragged last key
// tile of the short persistent forms, whose P is written for the chunks that
// hold keys. A rolled loop (a few instructions per chunk in the issuing thread).
__device__ __forceinline__ void issue_pv_chunks(uint32_t tmem_o, uint32_t tmem_p, uint32_t v_lo,
                                                uint32_t accumulate, int n) {
  constexpr uint32_t idesc = idesc_bf16(kBM, kD, 1);
#pragma unroll 1
  for (int k = 0; k < n; ++k) {
    const uint32_t a = tmem_p + 16u * static_cast<uint32_t>(k);
    const uint32_t b = v_lo + (static_cast<uint32_t>(k) << 7);
    ptx::mma_ts_imm<0, 0>(tmem_o, a, b, kDescHi, idesc, k == 0 ? accumulate : 1u);
    ptx::mma_ts_imm<8, 0>(tmem_o, a, b, kDescHi, idesc, 1u);
  }
}

__device__ __forceinline__ uint32_t round_bf16_bits(float x, int mode) {
  uint32_t u = __float_as_uint(x);
  if ((u & 0x7FFFFFFFu) > 0x7F800000u) return 0x7FC0u;  // NaN: one pattern
  if (mode == 0) {
    u += 0x7FFFu + ((u >> 16) & 1u);  // nearest, ties to even
  } else if (mode == 1) {
    u += 0x8000u;  // nearest, ties away from zero (sign-magnitude)
  }                // mode 2: toward zero = truncate
  return u >> 16;
}

// Two fp32 results of arithmetic -> packed bf16x2 (x0 in bits 0..15), rounded as
// round_bf16_bits does for RTNA (bias 0x8000) or RTZ (bias 0), the bias added
// before the upper halves are taken. A NaN produced by fp32 arithmetic on this
// GPU is the positive pattern 0x7FFFFFFF: as a signed integer it is above
// 0x7FC00000, so a signed min turns it (and only it: every other value, negative
// ones included, is not above) into 0x7FC00000, which both modes round to the one
// NaN pattern 0x7FC0.
__device__ __forceinline__ uint32_t round_pair_bf16(float x0, float x1, uint32_t bias) {
  const uint32_t u0 = static_cast<uint32_t>(min(__float_as_int(x0), 0x7FC00000));
  const uint32_t u1 = static_cast<uint32_t>(min(__float_as_int(x1), 0x7FC00000));
  return ptx::prmt_hi16(u0 + bias, u1 + bias);
}

// The same for RTNE, by the hardware conversion (round to nearest, ties to even;
// subnormals kept). It gives every NaN as the positive pattern 0x7FFF; a signed
// 16-bit min against 0x7FC0 makes that the one NaN pattern 0x7FC0 and leaves every
// other result (negative ones, +-Inf and finite values, all at most 0x7F80 as
// signed halves) as it is. Checked against the integer rounding on this GPU over
// every upper half with ties, neighbours of ties and random lower halves.
__device__ __forceinline__ uint32_t round_pair_bf16_rtne(float x0, float x1) {
  return ptx::min_s16x2(ptx::pack_bf16x2(x0, x1), 0x7FC07FC0u);
}

// The running output row of a softmax thread: 128 fp32 as 64 packed pairs
// (column 2i in the low half of pair i), updated with packed f32x2 arithmetic.
using Row = uint64_t[kD / 2];

// How a key tile is masked: not at all; per element (the ragged last tile); or,
// in pass A only, per element in the 16-column chunks that reach past the warp's
// least limit, writing the hidden logits back to TMEM as -Inf (the causal mask,
// whose limits rise row by row; pass B then needs no mask when c > 0).
enum MaskKind : int { kNoMask = 0, kElemMask = 1, kChunkMask = 2 };

// Pass A over one key tile. Folds the previous key tile's products (TMEM O)
// into the register row when kFold, and returns the row max of S (NaN if any
// element is NaN). Columns >= valid are skipped unless kMask is kNoMask; with
// kChunkMask, vmin is the least `valid` over the warp's lanes, so a chunk wholly
// below it needs no test (the branch on it is uniform over the warp), and a
// chunk that does is written back with its hidden columns set to -Inf. Both
// 16-column loads of a chunk are issued before one wait.
template <int kMask, bool kFold>
__device__ __forceinline__ float fold_and_max(uint32_t tS, uint32_t tO, Row& acc, int valid,
                                              int vmin) {
  const float neg_inf = -__int_as_float(0x7F800000);
  float e0 = neg_inf, e1 = neg_inf;
#pragma unroll
  for (int ch = 0; ch < 8; ++ch) {
    uint32_t r[16], o[16];
    ptx::tmem_ld16_nowait(tS + 16 * ch, r);
    if (kFold) ptx::tmem_ld16_nowait(tO + 16 * ch, o);
    ptx::tmem_wait_ld16(r);
    if (kFold) ptx::reg_fence16(o);
    if (kMask == kChunkMask)
      ptx::mask16_store_uniform(r, valid - 16 * ch, 16 * ch + 16 <= vmin,
                                __float_as_uint(neg_inf), tS + 16 * ch);
#pragma unroll
    for (int i = 0; i < 16; i += 4) {
      float s0 = __uint_as_float(r[i]), s1 = __uint_as_float(r[i + 1]);
      float s2 = __uint_as_float(r[i + 2]), s3 = __uint_as_float(r[i + 3]);
      if (kMask == kElemMask) {
        if (16 * ch + i >= valid) s0 = neg_inf;
        if (16 * ch + i + 1 >= valid) s1 = neg_inf;
        if (16 * ch + i + 2 >= valid) s2 = neg_inf;
        if (16 * ch + i + 3 >= valid) s3 = neg_inf;
      }
      e0 = ptx::max3_nan(e0, s0, s1);
      e1 = ptx::max3_nan(e1, s2, s3);
    }
    if (kFold) {
#pragma unroll
      for (int i = 0; i < 8; ++i)
        acc[8 * ch + i] = ptx::f2_add(
            acc[8 * ch + i], ptx::f2_pack(__uint_as_float(o[2 * i]), __uint_as_float(o[2 * i + 1])));
    }
  }
  return ptx::max_nan(e0, e1);
}

// Same for a negative scale, where the largest scaled logit comes from the
// smallest S: returns the row min (NaN-propagating). Kept simple (rare case).
template <bool kMasked>
__device__ __forceinline__ float fold_and_min(uint32_t tS, uint32_t tO, Row& acc, int valid,
                                              bool fold) {
  const float pos_inf = __int_as_float(0x7F800000);
  float e = pos_inf;
#pragma unroll
  for (int ch = 0; ch < 4; ++ch) {
    uint32_t r[32];
    ptx::tmem_ld32(tS + 32 * ch, r);
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      if (kMasked && 32 * ch + i >= valid) continue;
      e = ptx::min_nan(e, __uint_as_float(r[i]));
    }
    if (fold) {
      ptx::tmem_ld32(tO + 32 * ch, r);
#pragma unroll
      for (int i = 0; i < 16; ++i)
        acc[16 * ch + i] = ptx::f2_add(
            acc[16 * ch + i], ptx::f2_pack(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1])));
    }
  }
  return e;
}

// p = 2^(s*c - m_sub) for one 16-key chunk; writes P_hi (8 columns) and P_lo
// (8 columns) over the chunk's S columns; adds p into the pair sums l. Pairs of
// columns go through packed f32x2 instructions.
template <bool kMasked>
__device__ __forceinline__ void exp_chunk(uint32_t tS, int u, const uint32_t (&r)[16], int valid,
                                          uint64_t c2, uint64_t neg_m2, uint64_t (&l)[2]) {
  const float neg_inf = -__int_as_float(0x7F800000);
  uint32_t hi[8], lo[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint64_t x = ptx::f2_fma(
        ptx::f2_pack(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1])), c2, neg_m2);
    float x0, x1;
    ptx::f2_unpack(x, x0, x1);
    if (kMasked) {
      if (16 * u + 2 * i >= valid) x0 = neg_inf;
      if (16 * u + 2 * i + 1 >= valid) x1 = neg_inf;
    }
    const float p0 = ptx::ex2(x0);
    const float p1 = ptx::ex2(x1);
    const uint64_t p2 = ptx::f2_pack(p0, p1);
    l[i & 1] = ptx::f2_add(l[i & 1], p2);
    const uint32_t h = ptx::pack_bf16x2(p0, p1);
    // p - bf16(p) is exact in fp32; one packed subtraction per pair.
    const uint64_t res =
        ptx::f2_sub(p2, ptx::f2_pack(__uint_as_float(h << 16), __uint_as_float(h & 0xFFFF0000u)));
    float r0, r1;
    ptx::f2_unpack(res, r0, r1);
    hi[i] = h;
    lo[i] = ptx::pack_bf16x2(r0, r1);
  }
  ptx::tmem_st8(tS + 16 * u, hi);
  ptx::tmem_st8(tS + 16 * u + 8, lo);
}

// Pass B over one key tile: exp, P split, row sum. The load of chunk u+1 is in
// flight while chunk u is computed.
template <bool kMasked>
__device__ __forceinline__ float tile_exp(uint32_t tS, int valid, float c, float m_sub) {
  const uint64_t c2 = ptx::f2_pack(c, c);
  const uint64_t neg_m2 = ptx::f2_pack(-m_sub, -m_sub);
  uint64_t l[2] = {0, 0};
  uint32_t ra[16], rb[16];
  ptx::tmem_ld16_nowait(tS, ra);
#pragma unroll
  for (int u = 0; u < 8; u += 2) {
    ptx::tmem_wait_ld16(ra);
    ptx::tmem_ld16_nowait(tS + 16 * (u + 1), rb);
    exp_chunk<kMasked>(tS, u, ra, valid, c2, neg_m2, l);
    ptx::tmem_wait_ld16(rb);
    if (u + 2 < 8) ptx::tmem_ld16_nowait(tS + 16 * (u + 2), ra);
    exp_chunk<kMasked>(tS, u + 1, rb, valid, c2, neg_m2, l);
  }
  float a0, a1, b0, b1;
  ptx::f2_unpack(l[0], a0, a1);
  ptx::f2_unpack(l[1], b0, b1);
  return (a0 + a1) + (b0 + b1);
}

// acc *= f (the rare lazy rescale).
__device__ __forceinline__ void rescale_row(Row& acc, float f) {
  const uint64_t f2 = ptx::f2_pack(f, f);
#pragma unroll
  for (int i = 0; i < kD / 2; ++i) acc[i] = ptx::f2_mul(acc[i], f2);
}

// acc += O (the last key tile's products; epilogue).
// tO row *= f, 16 columns at a time (the stores complete before P_j is signalled).
__device__ __forceinline__ void rescale_tmem_row(uint32_t tO, float f) {
  const uint64_t f2 = ptx::f2_pack(f, f);
#pragma unroll 1
  for (int ch = 0; ch < 8; ++ch) {
    uint32_t r[16];
    ptx::tmem_ld16(tO + 16 * ch, r);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      float a, b;
      ptx::f2_unpack(ptx::f2_mul(ptx::f2_pack(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1])), f2),
                     a, b);
      r[2 * i] = __float_as_uint(a);
      r[2 * i + 1] = __float_as_uint(b);
    }
    ptx::tmem_st16(tO + 16 * ch, r);
  }
}

__device__ __forceinline__ void fold_last(uint32_t tO, Row& acc) {
#pragma unroll
  for (int ch = 0; ch < 4; ++ch) {
    uint32_t r[32];
    ptx::tmem_ld32(tO + 32 * ch, r);
#pragma unroll
    for (int i = 0; i < 16; ++i)
      acc[16 * ch + i] = ptx::f2_add(
          acc[16 * ch + i], ptx::f2_pack(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1])));
  }
}

// The same when the row holds nothing yet (an item of one key tile): a load.
__device__ __forceinline__ void load_last(uint32_t tO, Row& acc) {
#pragma unroll
  for (int ch = 0; ch < 4; ++ch) {
    uint32_t r[32];
    ptx::tmem_ld32(tO + 32 * ch, r);
#pragma unroll
    for (int i = 0; i < 16; ++i)
      acc[16 * ch + i] = ptx::f2_pack(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1]));
  }
}

// Both passes over one key tile of an item of a short persistent variant (at
// most 4 key tiles, so the output row stays in TMEM until the epilogue and its
// registers are free during the softmax). kMasked: the ragged last tile, valid =
// its keys (1..127, the same for every row, so every branch on it is uniform);
// only the 16-key chunks holding a key are read. The first five chunks (80 keys)
// are read from TMEM once and kept in registers for pass B; the others are read
// again (holding a sixth chunk made the variant spill registers). Updates the row's reference m_used by the lazy rule
// and sets f to the factor the row's earlier partial must take (1 if it did not
// move); returns the tile's row sum, relative to the new reference.
template <bool kMasked>
__device__ __forceinline__ float short_tile(uint32_t tS, int valid, float c, bool pos,
                                            float& m_used, float& f) {
  const float neg_inf = -__int_as_float(0x7F800000);
  const float pos_inf = __int_as_float(0x7F800000);
  uint32_t r[5][16];
  float e0 = pos ? neg_inf : pos_inf, e1 = e0;
#pragma unroll
  for (int ch = 0; ch < 8; ++ch) {
    if (kMasked && 16 * ch >= valid) continue;
    uint32_t q[16];
    uint32_t (&x)[16] = ch < 5 ? r[ch < 5 ? ch : 0] : q;  // held, or read again in pass B
    ptx::tmem_ld16_nowait(tS + 16 * ch, x);
    ptx::tmem_wait_ld16(x);
#pragma unroll
    for (int i = 0; i < 16; i += 2) {
      float s0 = __uint_as_float(x[i]), s1 = __uint_as_float(x[i + 1]);
      if (kMasked && 16 * ch + i >= valid) s0 = pos ? neg_inf : pos_inf;
      if (kMasked && 16 * ch + i + 1 >= valid) s1 = pos ? neg_inf : pos_inf;
      if (pos) {
        e0 = ptx::max_nan(e0, s0);
        e1 = ptx::max_nan(e1, s1);
      } else {
        e0 = ptx::min_nan(e0, s0);
        e1 = ptx::min_nan(e1, s1);
      }
    }
  }
  const float ext = pos ? ptx::max_nan(e0, e1) : ptx::min_nan(e0, e1);
  const float m_tile = ext * c;
  f = 1.f;
  if (m_tile > m_used + kTau) {  // false for NaN
    f = ptx::ex2(m_used - m_tile);  // 0 when m_used = -Inf
    m_used = m_tile;
  }
  const float m_sub = (m_used == neg_inf) ? 0.f : m_used;
  const uint64_t c2 = ptx::f2_pack(c, c);
  const uint64_t neg_m2 = ptx::f2_pack(-m_sub, -m_sub);
  uint64_t l[2] = {0, 0};
#pragma unroll
  for (int ch = 0; ch < 8; ++ch) {
    if (kMasked && 16 * ch >= valid) continue;
    if (ch < 5) {
      exp_chunk<kMasked>(tS, ch, r[ch < 5 ? ch : 0], valid, c2, neg_m2, l);
    } else {
      uint32_t q[16];
      ptx::tmem_ld16_nowait(tS + 16 * ch, q);
      ptx::tmem_wait_ld16(q);
      exp_chunk<kMasked>(tS, ch, q, valid, c2, neg_m2, l);
    }
  }
  float a0, a1, b0, b1;
  ptx::f2_unpack(l[0], a0, a1);
  ptx::f2_unpack(l[1], b0, b1);
  return (a0 + a1) + (b0 + b1);
}

__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          unsigned long long timeout_ns) {
  const bool ok = wait_bounded(bar, parity, abort_flag, timeout_ns, true);
  return __all_sync(0xFFFFFFFFu, ok);
}

// Merge of the key-range splits of one query row, four consecutive columns
// c0..c0+3. A split s left O_s = sum_j 2^(t_j - r_s) v_j and l_s = sum_j
// 2^(t_j - r_s) relative to its own reference r_s (t_j: scaled logits in log2
// units); the softmax over all keys is sum_s 2^(r_s - R) O_s / sum_s 2^(r_s - R)
// l_s for any R, here R = max_s r_s (r_s = -Inf for a split with no finite
// logit, which then weighs 0; R = 0 if every split is like that, and 0/0 gives
// NaN). The sums run over s in a fixed order, so the result is bit-identical
// from run to run. Returns the four outputs rounded per mode, two bf16 per word.
__device__ __forceinline__ uint2 merge_splits4(const float* part_o, const float* part_rl, size_t row0,
                                               size_t split_pitch, int n_splits, int c0, int mode) {
  const float2* rl = reinterpret_cast<const float2*>(part_rl);
  float R = -__int_as_float(0x7F800000);
#pragma unroll 8
  for (int s = 0; s < n_splits; ++s) R = fmaxf(R, rl[row0 + s * split_pitch].x);
  if (R == -__int_as_float(0x7F800000)) R = 0.f;
  float L = 0.f;
  float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 8
  for (int s = 0; s < n_splits; ++s) {
    const size_t r = row0 + s * split_pitch;
    const float2 ml = rl[r];
    const float w = ptx::ex2(ml.x - R);  // NaN only if R = +Inf: that row is NaN anyway
    const float4 x = *reinterpret_cast<const float4*>(part_o + r * kD + c0);
    L = fmaf(ml.y, w, L);
    o.x = fmaf(x.x, w, o.x);
    o.y = fmaf(x.y, w, o.y);
    o.z = fmaf(x.z, w, o.z);
    o.w = fmaf(x.w, w, o.w);
  }
  const float inv = __frcp_rn(L);
  return make_uint2(round_bf16_bits(o.x * inv, mode) | (round_bf16_bits(o.y * inv, mode) << 16),
                    round_bf16_bits(o.z * inv, mode) | (round_bf16_bits(o.w * inv, mode) << 16));
}

// The CTA's share of the work: (batch, head, query-tile pair, key split) and the
// split's key tiles. Splits of one pair are adjacent in the grid, pairs of one
// head are adjacent (so K/V of a head stay in L2); under the causal mask the
// pairs go longest first within groups of heads instead, which balances the
// SMs' loads while the blocks running at one time share their heads' K/V
// through L2.
// Recomputed by each role where it is needed, rather than kept live across the
// softmax loop.
struct Work {
  int split, pair, bh, head, kv_head, batch;
  int tile0, n_kv;  // key tiles [tile0, tile0 + n_kv)
  int q_base, k_base;  // first query / key token of the sequence (varlen; else 0)
  int sq, sk;          // the sequence's query / key lengths
  bool bad;            // varlen: the offsets of this sequence are invalid
};

template <bool kCausal, bool kVarlen>
__device__ __forceinline__ Work work_of(const Params& p, int work_item) {
  Work w;
  w.split = work_item % p.n_splits;
  const int item = work_item / p.n_splits;
  if (kCausal || kVarlen) {
    // Causal pairs differ in length: within each group of head_group (batch,
    // head) items, longest key ranges first (blocks start in index order, so
    // this is a greedy longest-first schedule); the group's K/V fit in L2. A
    // variable-length batch without the mask uses groups of one item: the pairs
    // of one (sequence, head) run together on its K/V.
    const int span = p.n_qpairs * p.head_group;
    const int g = item / span;
    const int r = item - g * span;
    const int gs = min(p.head_group, p.BH - g * p.head_group);
    w.pair = p.n_qpairs - 1 - r / gs;
    w.bh = g * p.head_group + r % gs;
  } else {
    w.pair = item % p.n_qpairs;
    w.bh = item / p.n_qpairs;
  }
  w.head = w.bh % p.H;
  w.kv_head = w.head / p.group;
  w.batch = w.bh / p.H;
  int kv_tiles = p.kv_tiles;
  if (kVarlen) {
    // The sequence's tokens within the packed tensors. At least one key tile
    // runs (fully masked if the sequence has no key, so its rows come out NaN).
    const int b = w.batch;
    w.q_base = __ldg(p.cu_q + b);
    w.sq = __ldg(p.cu_q + b + 1) - w.q_base;
    w.k_base = __ldg(p.cu_k + b);
    w.sk = __ldg(p.cu_k + b + 1) - w.k_base;
    w.bad = w.q_base < 0 || w.sq < 0 || w.sq > p.max_sq || w.q_base + w.sq > p.Sq ||
            w.k_base < 0 || w.sk < 0 || w.k_base + w.sk > p.Sk;
    w.batch = 0;
    kv_tiles = w.sk > 0 ? (w.sk + kBN - 1) / kBN : 1;
  } else {
    w.q_base = 0;
    w.k_base = 0;
    w.sq = p.Sq;
    w.sk = p.Sk;
    w.bad = false;
  }
  const int base = kv_tiles / p.n_splits, rem = kv_tiles % p.n_splits;
  w.tile0 = w.split * base + (w.split < rem ? w.split : rem);
  w.n_kv = base + (w.split < rem ? 1 : 0);
  if (kCausal) {
    // Key tiles up to the diagonal of the pair's last row (at least one, so that
    // a row with no visible key still runs and comes out NaN).
    const int last_row = min(w.sq, 2 * kBM * (w.pair + 1)) - 1;
    const int visible = last_row + (w.sk - w.sq) + 1;
    const int tiles = visible <= 0 ? 1 : (visible + kBN - 1) / kBN;
    w.n_kv = min(tiles, kv_tiles);
  }
  return w;
}

// The CTA's own work item (one item per CTA; the pair variant's grid starts at
// item_base).
template <bool kCausal, bool kVarlen, bool kPair = false>
__device__ __forceinline__ Work work_of(const Params& p) {
  return work_of<kCausal, kVarlen>(
      p, kPair ? p.item_base + static_cast<int>(blockIdx.x) : static_cast<int>(blockIdx.x));
}

// First key tile of a work item in which some row of the CTA does not see every
// key (the causal diagonal; the end of a variable-length sequence, where the tile
// runs into the next sequence's keys), or n_kv if there is none. The masked
// tiles [first, n_kv) are at most kMaxMaskedTiles: the CTA's 256 rows' key
// limits span at most 255 keys.
template <bool kCausal>
__device__ __forceinline__ int first_masked_tile(const Work& w) {
  const int min_lim = kCausal ? min(2 * kBM * w.pair + (w.sk - w.sq) + 1, w.sk) : w.sk;
  return min_lim <= 0 ? 0 : min(min_lim / kBN, w.n_kv);
}

// kPartial: the CTA covers one split of the key range and writes its fp32 partial
// result to the workspace (combined by attn_splitkv_combine); otherwise the CTA
// covers all keys and stores bf16 output. kCausal: the causal mask (p.causal
// must agree). kVarlen: a packed batch of variable-length sequences, one grid
// slot per (sequence, head, query-tile pair) up to the longest sequence.
// kPersist (whole key range, no mask only): each CTA loops over items c,
// c + gridDim.x, ... with the barrier phases carried from item to item, the next
// item's Q loaded as soon as the current item's last S MMAs are done, and the
// output stored through a staging area of its own; used for short key ranges,
// where an item's fixed latency (first loads, epilogue, store) would otherwise
// leave the SM idle. kPair (whole key range, no mask only): the grid's CTAs
// form 2-CTA clusters, each cluster one work item whose keys are split in two
// halves (n_splits = 2); rank 1 sends its unnormalised rows to rank 0 through
// distributed shared memory, and rank 0 merges them with its own and stores
// the output; used for the last, partial wave of a launch, which then takes half
// the time. kShort (with kPersist; the key range ends in a ragged tile): every
// item has one key tile (1) or 2 to 4 (2), so its partial stays in TMEM until the
// epilogue (no fold) and the softmax keeps S in the row's registers between its
// two passes; on the ragged last tile the P V MMAs and pass B stop at the last
// 16-key chunk holding a key.
// Each is compiled separately so that the other variants carry none of it.
template <bool kPartial, bool kCausal, bool kVarlen, bool kPersist = false, bool kPair = false,
          int kShort = 0>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                    const Params p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = ptx::smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (sbase - raw);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffAbort);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffTmemSlot);
  const uint32_t sQ = sbase + kOffQ;
  const uint32_t sRing = sbase + kOffRing;
  auto bar = [&](int i) -> uint32_t { return sbase + kOffBar + 8u * static_cast<uint32_t>(i); };

  static_assert(!kPersist || (!kPartial && !kCausal && !kVarlen), "persistent: base path only");
  static_assert(!kPair || (!kPartial && !kCausal && !kVarlen && !kPersist), "pair: base path only");
  static_assert(kShort == 0 || (kPersist && kShort <= 2), "short: a persistent variant");
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // A key limit per row (rising along the causal diagonal, or the sequence's
  // key count) selects pass-A masking in every tile.
  constexpr bool kRowLimit = kCausal || kVarlen;

  if constexpr (kVarlen) {
    // Grid slots past the sequence's queries, and sequences with invalid
    // offsets, leave before anything is set up (the decision is the same for
    // every thread of the CTA).
    const Work wk = work_of<kCausal, kVarlen, kPair>(p);
    if (wk.bad) {
      if (threadIdx.x == 0) atomicOr(&g_attn_status, 2u);
      return;
    }
    if (2 * kBM * wk.pair >= wk.sq) return;
  }
#if ATTN_DEBUG
  if (threadIdx.x == 0) {
    if (p.dbg_poison) dbg_ok(false);
    const Work wk = work_of<kCausal, kVarlen, kPair>(p);
    dbg_ok(wk.pair >= 0 && wk.pair < p.n_qpairs && wk.bh >= 0 && wk.bh < p.BH && wk.n_kv >= 1 &&
           wk.kv_head >= 0 && wk.kv_head * p.group < p.H);
    dbg_ok(kVarlen || wk.tile0 + wk.n_kv <= p.kv_tiles);
  }
#endif

  if (threadIdx.x == 0) {
    ptx::mbar_init(bar(kBarQ), 1);
    for (int s = 0; s < kStages; ++s) {
      ptx::mbar_init(bar(kBarKvFull + s), 1);
      ptx::mbar_init(bar(kBarKvEmpty + s), 1);
    }
    for (int t = 0; t < kQTiles; ++t) {
      ptx::mbar_init(bar(kBarSFull + t), 1);
      ptx::mbar_init(bar(kBarPFull + t), 128);
      ptx::mbar_init(bar(kBarOFull + t), 1);
    }
    ptx::mbar_init(bar(kBarDrain), 1);
    ptx::mbar_init(bar(kBarQFree), 1);
    for (int t = 0; t < kQTiles; ++t) ptx::mbar_init(bar(kBarOFree + t), 128);
    for (int m = 0; m < kMaxMaskedTiles; ++m) {
      ptx::mbar_init(bar(kBarVChk + m), 1);
      ptx::mbar_init(bar(kBarVLanded + m), 1);
    }
    ptx::mbar_init(bar(kBarPeerReady), 1);
    ptx::mbar_init(bar(kBarReceived), 2 * kBM);
    if (kRowLimit)
      for (int m = 0; m < kMaxMaskedTiles; ++m)
        reinterpret_cast<uint32_t*>(smem + kOffVRec)[m * kVRecWords] = 0;  // no non-finite V yet
    *abort_flag = 0;
    ptx::fence_mbar_init();
    ptx::fence_proxy_async_smem();
  }
  // The split variant's merge kernel may be scheduled as soon as every CTA of
  // this grid has started (it waits for the whole grid before reading); so may
  // the pair variant's launch after the base variant's full waves (it reads
  // nothing they write, and waits for them only before it completes).
  if constexpr (kPartial) {
    ptx::launch_dependents();
  } else if constexpr (!kCausal && !kVarlen && !kPersist && !kPair) {
    if (p.early_dependents) ptx::launch_dependents();
  }
  if (warp == 0 && lane == 0) {
    ptx::prefetch_tmap(&tm_q);
    ptx::prefetch_tmap(&tm_k);
    ptx::prefetch_tmap(&tm_v);
    ptx::prefetch_tmap(&tm_o);
  }
  if (warp == 1) {
    ptx::tmem_alloc(ptx::smem_u32(tmem_slot), kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // Pair variant: both CTAs' barriers are initialised before either arrives on
  // the other's. Every thread of both CTAs reaches this point unconditionally.
  if constexpr (kPair) ptx::cluster_sync();

  // Each role changes its register budget inside its own branch, so that the
  // budget of every instruction is known where it is compiled.
  if (warp < kSoftmaxWarp0) {
    ptx::setmaxnreg_dec<kRegsLow>();
    if (warp == 0) {
      // ------------------------------------------------------------ producer
      // L2 policies: query tiles are read once, key/value tiles by every CTA of
      // their head.
      const uint64_t pol_once = ptx::l2_policy_evict_first();
      const uint64_t pol_reuse = ptx::l2_policy_evict_last();
      if constexpr (kPersist) {
        if (lane == 0) {
          int issued = 0;   // ring fills started so far (fill i goes to stage i % kStages)
          int planned = 0;  // ring fills of the items started so far
          int q_loads = 0;  // Q loads started so far (load i completes phase i of kBarQ)
          int c1, c2;
          for (int item = blockIdx.x, iter = 0; item < p.n_items; item += gridDim.x, ++iter) {
            const Work wk = work_of<kCausal, kVarlen>(p, item);
            // The Q buffer is free once the previous item's last S MMAs are done.
            if (iter > 0 && !wait_bounded(bar(kBarQFree), (iter - 1) & 1, abort_flag, p.timeout_ns, true))
              break;
            dbg_ok(wk.q_base + 2 * wk.pair * kBM < p.Sq);  // the first query tile starts inside
            ptx::mbar_arrive_expect_tx(bar(kBarQ), kQTiles * kTileBytes);
            for (int t = 0; t < kQTiles; ++t) {
              tma_coords(p.layout, wk.q_base + (2 * wk.pair + t) * kBM, wk.head, c1, c2);
              for (int hf = 0; hf < 2; ++hf)
                ptx::tma_load_4d_hint(sQ + t * kTileBytes + hf * kHalfBytes, &tm_q, bar(kBarQ), 64 * hf,
                                      c1, c2, wk.batch, pol_once);
            }
            ++q_loads;
            planned += 2 * wk.n_kv;
            bool ok = true;
            for (int it = 0; it < 2 * wk.n_kv; ++it) {
              const int stage = issued % kStages;
              const uint32_t parity = ((issued / kStages) & 1) ^ 1;
              if (!(ok = wait_bounded(bar(kBarKvEmpty + stage), parity, abort_flag, p.timeout_ns, true)))
                break;
              const CUtensorMap* map = (it & 1) ? &tm_v : &tm_k;
              dbg_ok(wk.k_base + (wk.tile0 + (it >> 1)) * kBN < p.Sk + kBN);
              tma_coords(p.layout, wk.k_base + (wk.tile0 + (it >> 1)) * kBN, wk.kv_head, c1, c2);
              ptx::mbar_arrive_expect_tx(bar(kBarKvFull + stage), kTileBytes);
              for (int hf = 0; hf < 2; ++hf)
                ptx::tma_load_4d_hint(sRing + stage * kTileBytes + hf * kHalfBytes, map,
                                      bar(kBarKvFull + stage), 64 * hf, c1, c2, wk.batch, pol_reuse);
              ++issued;
            }
            if (!ok) break;
          }
          // Let every copy this thread started land before the CTA can exit. On
          // the normal path these phases have long completed; after an abort the
          // consumer may never have waited for them. (At most one Q load is ever
          // outstanding: the next waits for the S MMAs that consume it.)
          dbg_ok(issued == planned || *abort_flag);  // every fill of the plan was issued
          if (q_loads > 0) wait_bounded(bar(kBarQ), (q_loads - 1) & 1, abort_flag, p.timeout_ns, false);
          for (int s = 0; s < kStages && s < issued; ++s) {
            const int fills = (issued - 1 - s) / kStages + 1;  // fills of stage s so far
            wait_bounded(bar(kBarKvFull + s), (fills - 1) & 1, abort_flag, p.timeout_ns, false);
          }
        }
      } else {
        if (lane == 0) {
          const Work wk = work_of<kCausal, kVarlen, kPair>(p);
          const int pair = wk.pair, head = wk.head, batch = wk.batch, tile0 = wk.tile0, n_kv = wk.n_kv;
          const int kv_head = wk.kv_head, q_base = wk.q_base, k_base = wk.k_base;
          int issued = 0;  // ring fills started so far (fill i goes to stage i % kStages)
          int c1, c2;
          dbg_ok(q_base + 2 * pair * kBM < p.Sq);  // the first query tile starts inside
          ptx::mbar_arrive_expect_tx(bar(kBarQ), kQTiles * kTileBytes);
          for (int t = 0; t < kQTiles; ++t) {
            tma_coords(p.layout, q_base + (2 * pair + t) * kBM, head, c1, c2);
            for (int hf = 0; hf < 2; ++hf)
              ptx::tma_load_4d_hint(sQ + t * kTileBytes + hf * kHalfBytes, &tm_q, bar(kBarQ), 64 * hf, c1,
                                    c2, batch, pol_once);
          }
          for (int it = 0; it < 2 * n_kv; ++it) {
            const int stage = it % kStages;
            const uint32_t parity = ((it / kStages) & 1) ^ 1;
            if (!wait_bounded(bar(kBarKvEmpty + stage), parity, abort_flag, p.timeout_ns, true)) break;
            const CUtensorMap* map = (it & 1) ? &tm_v : &tm_k;
            dbg_ok(k_base + (tile0 + (it >> 1)) * kBN < p.Sk + kBN);
            tma_coords(p.layout, k_base + (tile0 + (it >> 1)) * kBN, kv_head, c1, c2);
            ptx::mbar_arrive_expect_tx(bar(kBarKvFull + stage), kTileBytes);
            for (int hf = 0; hf < 2; ++hf)
              ptx::tma_load_4d_hint(sRing + stage * kTileBytes + hf * kHalfBytes, map,
                                    bar(kBarKvFull + stage), 64 * hf, c1, c2, batch, pol_reuse);
            ++issued;
          }
          // Let every copy this thread started land before the CTA can exit. On
          // the normal path these phases have long completed; after an abort the
          // consumer may never have waited for them.
          dbg_ok(issued == 2 * n_kv || *abort_flag);  // every fill of the plan was issued
          wait_bounded(bar(kBarQ), 0, abort_flag, p.timeout_ns, false);
          for (int s = 0; s < kStages && s < issued; ++s) {
            const int fills = (issued - 1 - s) / kStages + 1;  // fills of stage s so far
            wait_bounded(bar(kBarKvFull + s), (fills - 1) & 1, abort_flag, p.timeout_ns, false);
          }
        }
      }
      __syncwarp();
    } else if (warp == 1) {
      // ------------------------------------------------------------ MMA issuer
      if (lane == 0) {
        if constexpr (kPersist) {
          auto ring_wait = [&](int it) -> bool {
            const bool r = wait_bounded(bar(kBarKvFull + it % kStages), (it / kStages) & 1, abort_flag,
                                        p.timeout_ns, true);
            ptx::tc_fence_after();
            return r;
          };
          // Ring stage descriptors: K tiles are K-major B operands, V tiles MN-major.
          auto k_desc = [&](int it) -> uint32_t {
            return desc_lo(sRing + (it % kStages) * kTileBytes, 16);
          };
          auto v_desc = [&](int it) -> uint32_t {
            return desc_lo(sRing + (it % kStages) * kTileBytes, kHalfBytes);
          };
          const uint32_t q0_desc = desc_lo(sQ, 16);
          const uint32_t q1_desc = desc_lo(sQ + kTileBytes, 16);
          bool ok = true;
          int fill = 0;   // ring fills consumed by the items before this one
          int ktile = 0;  // key tiles of the items before this one (S and P phases)
          for (int item = blockIdx.x, iter = 0; ok && item < p.n_items; item += gridDim.x, ++iter) {
            const int n_kv = work_of<kCausal, kVarlen>(p, item).n_kv;
            if (!(ok = wait_bounded(bar(kBarQ), iter & 1, abort_flag, p.timeout_ns, true))) break;
            ptx::tc_fence_after();
            if (!(ok = ring_wait(fill))) break;
            // S of the first key tile. The previous item's last P V MMAs, issued
            // before these on the same pipe, have read the S/P columns first.
            issue_s(tmem + kTmemS0, q0_desc, k_desc(fill));
            if (!p.withhold_s0) ptx::mma_commit(bar(kBarSFull + 0));
            issue_s(tmem + kTmemS0 + 128, q1_desc, k_desc(fill));
            ptx::mma_commit(bar(kBarSFull + 1));
            ptx::mma_commit(bar(kBarKvEmpty + fill % kStages));
            if (n_kv == 1) ptx::mma_commit(bar(kBarQFree));  // the item's last S MMAs
            for (int j = 0; ok && j < n_kv; ++j) {
              const int vit = fill + 2 * j + 1;
              const int kit = fill + 2 * j + 2;
              const bool more = j + 1 < n_kv;
              if (!(ok = ring_wait(vit))) break;
              if (!(ok = wait_bounded(bar(kBarPFull + 0), (ktile + j) & 1, abort_flag, p.timeout_ns, true)))
                break;
              // The first P V of an item starts a fresh partial in O: the previous
              // item's epilogue must have read it.
              if (j == 0 && iter > 0 &&
                  !(ok = wait_bounded(bar(kBarOFree + 0), (iter - 1) & 1, abort_flag, p.timeout_ns, true)))
                break;
              ptx::tc_fence_after();
              const uint32_t acc_o = (j % kFoldOf<kPartial>) != 0 ? 1u : 0u;  // partial continues
              // Short variants: P of the ragged last key tile was written for its first
              // n_pv chunks only (kShort 1: every tile is that tile).
              const int n_pv = (!more && p.kv_tail < kBN) ? (p.kv_tail + 15) >> 4 : 8;
              if (kShort == 1 || (kShort == 2 && n_pv < 8))
                issue_pv_chunks(tmem + kTmemO0, tmem + kTmemS0, v_desc(vit), acc_o, n_pv);
              else
                issue_pv(tmem + kTmemO0, tmem + kTmemS0, v_desc(vit), acc_o);
              if (!more) ptx::mma_commit(bar(kBarOFull + 0));
              if (more) {
                if (!(ok = ring_wait(kit))) break;
                issue_s(tmem + kTmemS0, q0_desc, k_desc(kit));
                ptx::mma_commit(bar(kBarSFull + 0));
              }
              if (!(ok = wait_bounded(bar(kBarPFull + 1), (ktile + j) & 1, abort_flag, p.timeout_ns, true)))
                break;
              if (j == 0 && iter > 0 &&
                  !(ok = wait_bounded(bar(kBarOFree + 1), (iter - 1) & 1, abort_flag, p.timeout_ns, true)))
                break;
              ptx::tc_fence_after();
              if (kShort == 1 || (kShort == 2 && n_pv < 8))
                issue_pv_chunks(tmem + kTmemO0 + 128, tmem + kTmemS0 + 128, v_desc(vit), acc_o, n_pv);
              else
                issue_pv(tmem + kTmemO0 + 128, tmem + kTmemS0 + 128, v_desc(vit), acc_o);
              ptx::mma_commit(bar(kBarKvEmpty + vit % kStages));
              if (!more) ptx::mma_commit(bar(kBarOFull + 1));
              if (more) {
                issue_s(tmem + kTmemS0 + 128, q1_desc, k_desc(kit));
                ptx::mma_commit(bar(kBarSFull + 1));
                ptx::mma_commit(bar(kBarKvEmpty + kit % kStages));
                if (j + 2 == n_kv) ptx::mma_commit(bar(kBarQFree));  // the item's last S MMAs
              }
            }
            fill += 2 * n_kv;
            ktile += n_kv;
          }
        } else {
          const Work wk = work_of<kCausal, kVarlen, kPair>(p);
          const int n_kv = wk.n_kv;
          // Masked key tiles (key-limit variants): V is checked first.
          const int jm = kRowLimit ? first_masked_tile<kCausal>(wk) : n_kv;
          bool ok = wait_bounded(bar(kBarQ), 0, abort_flag, p.timeout_ns, true);
          ptx::tc_fence_after();
          auto ring_wait = [&](int it) -> bool {
            const bool r = wait_bounded(bar(kBarKvFull + it % kStages), (it / kStages) & 1, abort_flag,
                                        p.timeout_ns, true);
            ptx::tc_fence_after();
            return r;
          };
          // Ring stage descriptors: K tiles are K-major B operands, V tiles MN-major.
          auto k_desc = [&](int it) -> uint32_t {
            return desc_lo(sRing + (it % kStages) * kTileBytes, 16);
          };
          auto v_desc = [&](int it) -> uint32_t {
            return desc_lo(sRing + (it % kStages) * kTileBytes, kHalfBytes);
          };
          const uint32_t q0_desc = desc_lo(sQ, 16);
          const uint32_t q1_desc = desc_lo(sQ + kTileBytes, 16);
          if (ok) ok = ring_wait(0);
          if (ok) {
            issue_s(tmem + kTmemS0, q0_desc, k_desc(0));
            if (!p.withhold_s0) ptx::mma_commit(bar(kBarSFull + 0));
            issue_s(tmem + kTmemS0 + 128, q1_desc, k_desc(0));
            ptx::mma_commit(bar(kBarSFull + 1));
            ptx::mma_commit(bar(kBarKvEmpty + 0));
          }
          // V of a masked key tile: tell the V check it has landed, one key tile
          // ahead of its P V products.
          if (kRowLimit && ok && jm == 0 && (ok = ring_wait(1))) ptx::mbar_arrive(bar(kBarVLanded + 0));
          for (int j = 0; ok && j < n_kv; ++j) {
            const int vit = 2 * j + 1;
            const int kit = 2 * j + 2;
            const bool more = j + 1 < n_kv;
            if (!(ok = ring_wait(vit))) break;
            if (kRowLimit && j >= jm && j - jm < kMaxMaskedTiles &&
                !(ok = wait_bounded(bar(kBarVChk + (j - jm)), 0, abort_flag, p.timeout_ns, true)))
              break;
            if (!(ok = wait_bounded(bar(kBarPFull + 0), j & 1, abort_flag, p.timeout_ns, true))) break;
            ptx::tc_fence_after();
            const uint32_t acc_o = (j % kFoldOf<kPartial>) != 0 ? 1u : 0u;  // partial continues
            issue_pv(tmem + kTmemO0, tmem + kTmemS0, v_desc(vit), acc_o);
            if (!more) ptx::mma_commit(bar(kBarOFull + 0));
            if (more) {
              if (!(ok = ring_wait(kit))) break;
              issue_s(tmem + kTmemS0, q0_desc, k_desc(kit));
              ptx::mma_commit(bar(kBarSFull + 0));
            }
            if (!(ok = wait_bounded(bar(kBarPFull + 1), j & 1, abort_flag, p.timeout_ns, true))) break;
            ptx::tc_fence_after();
            issue_pv(tmem + kTmemO0 + 128, tmem + kTmemS0 + 128, v_desc(vit), acc_o);
            ptx::mma_commit(bar(kBarKvEmpty + vit % kStages));
            if (!more) ptx::mma_commit(bar(kBarOFull + 1));
            if (more) {
              issue_s(tmem + kTmemS0 + 128, q1_desc, k_desc(kit));
              ptx::mma_commit(bar(kBarSFull + 1));
              ptx::mma_commit(bar(kBarKvEmpty + kit % kStages));
              const int mnext = j + 1 - jm;  // the next key tile's index among the masked ones
              if (kRowLimit && mnext >= 0 && mnext < kMaxMaskedTiles) {
                if (!(ok = ring_wait(vit + 2))) break;
                ptx::mbar_arrive(bar(kBarVLanded + mnext));
              }
            }
          }
        }
        // Wait until every MMA issued so far has finished (immediate on the normal
        // path, where the softmax warps have already waited for the last ones).
        ptx::mma_commit(bar(kBarDrain));
        const bool drained = wait_bounded(bar(kBarDrain), 0, abort_flag, p.timeout_ns, false);
        // Pair variant, rank 0: no MMA or copy uses the ring any more; rank 1 may
        // write its rows into it.
        if (kPair && drained && ptx::cluster_ctarank() == 0)
          ptx::mbar_arrive_cluster(ptx::map_to_rank(bar(kBarPeerReady), 1));
      }
      __syncwarp();
    } else if constexpr (kRowLimit) {
      // ------------------------------------------------------------ V check (warps 2-3)
      // In a masked key tile a row's hidden keys get P = 0, and the tensor pipe's
      // 0 * NaN or 0 * Inf would carry a non-finite V value at such a key into
      // that row. These two warps read each masked tile's V from the ring before
      // its first P V product. If it holds non-finite values they record each one
      // (key, column, kind) and set it to 0 in shared memory; the epilogue then
      // adds it back to exactly the rows that see its key. Decisions are taken
      // at barriers of both warps (with a reduction), so neither can leave while
      // the other waits.
      const int tid = static_cast<int>(threadIdx.x) - 64;  // 0..63
      const Work wk = work_of<kCausal, kVarlen, kPair>(p);
      const int jm = first_masked_tile<kCausal>(wk);
      dbg_ok(wk.n_kv - jm <= kMaxMaskedTiles);
      for (int m = 0; jm + m < wk.n_kv && m < kMaxMaskedTiles; ++m) {
        const int fill = 2 * (jm + m) + 1;  // ring fill that holds V of key tile jm + m
        // The MMA issuer, which follows the ring's phases in order, reports when
        // this fill has landed (a wait on the ring barrier itself could be more
        // than one phase ahead of it, which a parity wait cannot tell apart).
        const bool ok = wait_bounded(bar(kBarVLanded + m), 0, abort_flag, p.timeout_ns, true);
        if (ptx::named_barrier_or(1, 64, !ok)) break;
        const uint32_t vt = sRing + (fill % kStages) * kTileBytes;
        // 2048 chunks of 16 bytes; thread tid reads chunks tid, tid + 64, ...
        uint32_t acc0 = 0, acc1 = 0;
#pragma unroll 8
        for (int i = 0; i < 32; ++i) {
          const uint4 x = ptx::ld_shared_v4(vt + (tid + 64 * i) * 16);
          acc0 = ptx::bf16x2_nonfinite_acc(x.x, ptx::bf16x2_nonfinite_acc(x.y, acc0));
          acc1 = ptx::bf16x2_nonfinite_acc(x.z, ptx::bf16x2_nonfinite_acc(x.w, acc1));
        }
        const bool found = ptx::named_barrier_or(1, 64, (acc0 | acc1) != 0);
        uint32_t* rec = reinterpret_cast<uint32_t*>(smem + kOffVRec) + m * kVRecWords;
        if (found) {
          for (int i = tid; i < kVRecWords; i += 64) rec[i] = 0;
          ptx::named_barrier_sync(1, 64);
          for (int i = 0; i < 32; ++i) {
            const int ci = tid + 64 * i;
            uint32_t w[4];
            const uint4 x = ptx::ld_shared_v4(vt + ci * 16);
            w[0] = x.x; w[1] = x.y; w[2] = x.z; w[3] = x.w;
            bool dirty = false;
            const int key = (ci >> 3) & (kBN - 1);  // TMA box row
            // 128-byte swizzle: the row's 16-byte chunk c sits at position c ^ (row & 7).
            const int col0 = (ci >> 10) * 64 + (((ci & 7) ^ (key & 7)) << 3);
            for (int e = 0; e < 8; ++e) {
              const uint32_t h = (w[e >> 1] >> (16 * (e & 1))) & 0xFFFFu;
              if ((h & 0x7F80u) != 0x7F80u) continue;
              const int col = col0 + e;
              const int kind = (h & 0x7Fu) ? kVRecNan : ((h & 0x8000u) ? kVRecNeg : kVRecPos);
              atomicOr(&rec[kVRecKeyMask + (key >> 5)], 1u << (key & 31));
              atomicOr(&rec[kind + key * 4 + (col >> 5)], 1u << (col & 31));
              w[e >> 1] &= ~(0xFFFFu << (16 * (e & 1)));
              dirty = true;
            }
            if (dirty) ptx::st_shared_v4(vt + ci * 16, w[0], w[1], w[2], w[3]);
          }
          ptx::fence_proxy_async_smem();  // the zeros, before the tensor pipe reads V
          ptx::named_barrier_sync(1, 64);
        }
        if (tid == 0) {
          rec[0] = found ? 1u : 0u;
          ptx::mbar_arrive(bar(kBarVChk + m));
        }
      }
    }
  } else {
    ptx::setmaxnreg_inc<kRegsHigh>();
    // ------------------------------------------------------------ softmax + epilogue
    const int t = (warp - kSoftmaxWarp0) >> 2;  // query tile of this warpgroup
    const int wq = warp & 3;                    // TMEM lane quarter of this warp
    const int row = wq * 32 + lane;             // row within the query tile
    const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t tS = tmem + lane_base + kTmemS0 + 128 * t;
    const uint32_t tO = tmem + lane_base + kTmemO0 + 128 * t;
    const float c = p.c;
    const bool pos = c >= 0.f;
    const float neg_inf = -__int_as_float(0x7F800000);
    if constexpr (kPersist) {
      // One loop over every key tile of every item of this CTA (a loop over items
      // around a loop over their tiles makes the compiler spill the row
      // registers); an item's epilogue runs after its last tile.
      bool ok = true;
      int sp = 0;  // S and P phase parity (key tiles processed so far, mod 2)
      int item = blockIdx.x;
      int j = 0, n_kv = 0;
      const int row_lim = 0;  // no per-row key limit on this path
      float m_used = neg_inf, l = 0.f;
      Row acc;
      if (item < p.n_items) {
        m_used = neg_inf;
        l = 0.f;
        // (The short variant loads the row from O at the end: it holds nothing before.)
        if constexpr (!kShort) {
#pragma unroll
          for (int i = 0; i < kD / 2; ++i) acc[i] = 0;  // +0.0f in both halves
        }
        n_kv = work_of<kCausal, kVarlen>(p, item).n_kv;  // key tiles of this item
      }
      while (ok && item < p.n_items) {
        if constexpr (kShort == 1) {
          // The item's one key tile: both passes from one read of S.
          if (!(ok = warp_wait(bar(kBarSFull + t), sp, abort_flag, p.timeout_ns))) break;
          ptx::tc_fence_after();
          float f_row;
          l = short_tile<true>(tS, p.kv_tail, c, pos, m_used, f_row);
          ptx::tmem_wait_st();
          ptx::tc_fence_before();
          ptx::mbar_arrive(bar(kBarPFull + t));
        } else if constexpr (kShort == 2) {
          // A key tile of an item of 2 to 4: both passes from one read of S. The
          // item's partial stays in TMEM (no fold before the epilogue); when the
          // reference moves, the partial of the earlier tiles is scaled there.
          if (!(ok = warp_wait(bar(kBarSFull + t), sp, abort_flag, p.timeout_ns))) break;
          ptx::tc_fence_after();
          const bool last = (j == n_kv - 1) && (p.kv_tail < kBN);
          float f_row;
          const float l_tile = last ? short_tile<true>(tS, p.kv_tail, c, pos, m_used, f_row)
                                    : short_tile<false>(tS, kBN, c, pos, m_used, f_row);
          const bool need = f_row != 1.f;  // the reference moved (f < 2^-8, or 0)
          if (need) l *= f_row;
          l += l_tile;
          if (j > 0 && __any_sync(0xFFFFFFFFu, need)) rescale_tmem_row(tO, f_row);
          ptx::tmem_wait_st();
          ptx::tc_fence_before();
          ptx::mbar_arrive(bar(kBarPFull + t));
        } else {
            if (!(ok = warp_wait(bar(kBarSFull + t), sp, abort_flag, p.timeout_ns))) break;
            ptx::tc_fence_after();
            // The ragged key tile is the last tile of the last split. Written as tests
            // of kernel parameters and the item index, which keeps the compiler's
            // register allocation of this loop free of spills.
            const bool last = (j == n_kv - 1) && (p.kv_tail < kBN) &&
                              (!kPartial || item % p.n_splits == p.n_splits - 1);
            // Masked tile: the ragged last tile; with the causal mask every tile, each
            // row hiding the keys beyond its own limit (a tile it fully sees loses
            // nothing). One path for all tiles keeps the loop's registers spill-free.
            const bool masked = kRowLimit ? true : last;
            constexpr int kM = kRowLimit ? kChunkMask : kElemMask;
            const int valid = kRowLimit ? row_lim - kBN * j : p.kv_tail;
            // Least `valid` over the warp (lane 0 has the warp's first row).
            const int vmin = kRowLimit ? __shfl_sync(0xFFFFFFFFu, valid, 0) : p.kv_tail;
            // Pass A: take the row extreme of S_j and, on a fold tile, add the TMEM
            // partial into the row (it holds the tiles since the last fold, complete
            // because the MMA that wrote S_j was issued after PV_{j-1}, and PV_j waits
            // for P_j).
            float ext, m_tile;
            bool need;
            if constexpr (kFoldOf<kPartial> == 1) {
              if (pos) {
                if (j == 0) {
                  ext = masked ? fold_and_max<kM, false>(tS, tO, acc, valid, vmin)
                               : fold_and_max<kNoMask, false>(tS, tO, acc, kBN, kBN);
                } else {
                  ext = masked ? fold_and_max<kM, true>(tS, tO, acc, valid, vmin)
                               : fold_and_max<kNoMask, true>(tS, tO, acc, kBN, kBN);
                }
              } else {
                ext = masked ? fold_and_min<true>(tS, tO, acc, valid, j > 0)
                             : fold_and_min<false>(tS, tO, acc, kBN, j > 0);
              }
              m_tile = ext * c;
              need = m_tile > m_used + kTau;  // false for NaN
              if (need) {
                const float f = ptx::ex2(m_used - m_tile);  // 0 when m_used = -Inf
                if (j > 0) rescale_row(acc, f);
                l *= f;
                m_used = m_tile;
              }
            } else {
              // The TMEM partial (key tiles since the last fold) is folded into the
              // registers every kFoldOf<kPartial> tiles.
              const bool fold_now = j > 0 && (j % kFoldOf<kPartial>) == 0;
              if (pos) {
                if (!fold_now) {
                  ext = masked ? fold_and_max<kM, false>(tS, tO, acc, valid, vmin)
                               : fold_and_max<kNoMask, false>(tS, tO, acc, kBN, kBN);
                } else {
                  ext = masked ? fold_and_max<kM, true>(tS, tO, acc, valid, vmin)
                               : fold_and_max<kNoMask, true>(tS, tO, acc, kBN, kBN);
                }
              } else {
                ext = masked ? fold_and_min<true>(tS, tO, acc, valid, fold_now)
                             : fold_and_min<false>(tS, tO, acc, kBN, fold_now);
              }
              m_tile = ext * c;
              need = m_tile > m_used + kTau;  // false for NaN
              float f_row = 1.f;  // this row's rescale factor at this tile
              if (need) {
                const float f = ptx::ex2(m_used - m_tile);  // 0 when m_used = -Inf
                if (j > 0) rescale_row(acc, f);
                l *= f;
                m_used = m_tile;
                f_row = f;
              }
              // A partial still in TMEM is relative to the old reference: scale it in
              // place (the PV MMAs that wrote it are done, S_j being ready; the next one
              // waits for P_j). Warp-uniform: each lane rescales its own row, by 1 if its
              // reference did not move.
              if ((j % kFoldOf<kPartial>) != 0 && __any_sync(0xFFFFFFFFu, need))
                rescale_tmem_row(tO, f_row);
            }
            const float m_sub = (m_used == neg_inf) ? 0.f : m_used;
            // Causal, c > 0: pass A left -Inf in the hidden columns, so pass B needs
            // no mask; for c <= 0 (where -Inf * c is not -Inf) it masks per element.
            const bool masked_b = kRowLimit ? !(c > 0.f) : last;
            if (kRowLimit) ptx::tmem_wait_st();  // pass A's write-backs before pass B reads
            l += masked_b ? tile_exp<true>(tS, valid, c, m_sub) : tile_exp<false>(tS, kBN, c, m_sub);
            ptx::tmem_wait_st();
            ptx::tc_fence_before();
            ptx::mbar_arrive(bar(kBarPFull + t));
        }
        sp ^= 1;
        if (++j < n_kv) continue;
        // ---- the item's epilogue
        const int iter = (item - static_cast<int>(blockIdx.x)) / static_cast<int>(gridDim.x);
        if (!(ok = warp_wait(bar(kBarOFull + t), iter & 1, abort_flag, p.timeout_ns))) break;
        // Fold the last partial into the row, then hand O back to the tensor pipe
        // (the next item's first P V overwrites it) before the stores.
        ptx::tc_fence_after();
        if constexpr (kShort)
          load_last(tO, acc);
        else
          fold_last(tO, acc);
        ptx::tc_fence_before();
        ptx::mbar_arrive(bar(kBarOFree + t));
        // Normalise, round, and store this warp's 32 rows with two TMA boxes (one
        // per 64-column half) through its 4 KiB staging buffer, in the 128-byte
        // swizzle. A buffer is rewritten only after the previous box has been
        // read out of it; rows past Sq are clipped by the store.
        const Work wk = work_of<kCausal, kVarlen>(p, item);
        const uint32_t stage_w = sbase + kOffStage + (t * 4 + wq) * kStageWarpBytes;
        const int q_row0 = (2 * wk.pair + t) * kBM + wq * 32;
        const bool rtne = p.mode == 0;
        const uint32_t bias = p.mode == 1 ? 0x8000u : 0u;
        const float inv_l = __frcp_rn(l);  // 0 -> Inf, so an all -Inf row gives 0 * Inf = NaN
        const uint64_t inv2 = ptx::f2_pack(inv_l, inv_l);
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          if constexpr (kShort != 0) {
            // Short forms: round this half of the row first, then wait until the
            // previous box has been read out of the staging buffer (the rounding
            // hides that wait), then write it. (The general persistent variant keeps
            // the order below: its loop measured no gain from it.)
            uint32_t w[32];
            if (rtne) {
#pragma unroll
              for (int i = 0; i < 32; ++i) {
                float o0, o1;
                ptx::f2_unpack(ptx::f2_mul(acc[32 * hf + i], inv2), o0, o1);
                w[i] = round_pair_bf16_rtne(o0, o1);
              }
            } else {
#pragma unroll
              for (int i = 0; i < 32; ++i) {
                float o0, o1;
                ptx::f2_unpack(ptx::f2_mul(acc[32 * hf + i], inv2), o0, o1);
                w[i] = round_pair_bf16(o0, o1, bias);
              }
            }
            if (lane == 0) ptx::bulk_wait_group_read_0();
            __syncwarp();
#pragma unroll
            for (int u = 0; u < 8; ++u)
              ptx::st_shared_v4(stage_w + lane * 128 + ((u ^ (lane & 7)) << 4), w[4 * u],
                                w[4 * u + 1], w[4 * u + 2], w[4 * u + 3]);
          } else {
            if (lane == 0) ptx::bulk_wait_group_read_0();
            __syncwarp();
#pragma unroll
            for (int ch = 0; ch < 2; ++ch) {
              uint32_t w[16];
              if (rtne) {
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                  float o0, o1;
                  ptx::f2_unpack(ptx::f2_mul(acc[32 * hf + 16 * ch + i], inv2), o0, o1);
                  w[i] = round_pair_bf16_rtne(o0, o1);
                }
              } else {
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                  float o0, o1;
                  ptx::f2_unpack(ptx::f2_mul(acc[32 * hf + 16 * ch + i], inv2), o0, o1);
                  w[i] = round_pair_bf16(o0, o1, bias);
                }
              }
#pragma unroll
              for (int u = 0; u < 4; ++u) {
                const int chunk = ch * 4 + u;
                ptx::st_shared_v4(stage_w + lane * 128 + ((chunk ^ (lane & 7)) << 4), w[4 * u],
                                  w[4 * u + 1], w[4 * u + 2], w[4 * u + 3]);
              }
            }
          }
          ptx::fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0 && q_row0 < p.Sq && dbg_ok(q_row0 >= 0)) {
            int c1, c2;
            tma_coords(p.layout, q_row0, wk.head, c1, c2);
            ptx::tma_store_4d_hint(&tm_o, stage_w, 64 * hf, c1, c2, wk.batch,
                                   ptx::l2_policy_evict_first());
            ptx::bulk_commit_group();
          }
        }
        item += gridDim.x;
        j = 0;
        if (item < p.n_items) {
          m_used = neg_inf;
          l = 0.f;
          if constexpr (!kShort) {
#pragma unroll
            for (int i = 0; i < kD / 2; ++i) acc[i] = 0;  // +0.0f in both halves
          }
          n_kv = work_of<kCausal, kVarlen>(p, item).n_kv;  // key tiles of this item
        }
      }
      // Every store of this warp has completed before the CTA can exit.
      if (lane == 0) ptx::bulk_wait_group_0();
      __syncwarp();
    } else {
      float m_used = neg_inf;
      float l = 0.f;
      Row acc;
#pragma unroll
      for (int i = 0; i < kD / 2; ++i) acc[i] = 0;  // +0.0f in both halves
      bool ok = true;
      int n_kv, row_lim;
      {
        const Work wk = work_of<kCausal, kVarlen, kPair>(p);
        n_kv = wk.n_kv;  // key tiles of this CTA
        // Number of keys this row sees, counted from the sequence's key 0: the
        // causal limit (capped at Sk, which also hides the ragged tail from the
        // padding rows past Sq), or for a variable-length batch without the mask
        // the sequence's key count (hiding the next sequence's keys).
        row_lim = kCausal ? min((2 * wk.pair + t) * kBM + row + (wk.sk - wk.sq) + 1, wk.sk)
                          : (kVarlen ? wk.sk : 0);
      }

      for (int j = 0; j < n_kv; ++j) {
        if (!(ok = warp_wait(bar(kBarSFull + t), j & 1, abort_flag, p.timeout_ns))) break;
        ptx::tc_fence_after();
        // The ragged key tile is the last tile of the last split. Written as tests
        // of kernel parameters and the block index, which keeps the compiler's
        // register allocation of this loop free of spills.
        const bool last = (j == n_kv - 1) && (p.kv_tail < kBN) &&
                          (kPair ? (blockIdx.x & 1u) != 0
                                 : (!kPartial ||
                                    static_cast<int>(blockIdx.x % p.n_splits) == p.n_splits - 1));
        // Masked tile: the ragged last tile; with the causal mask every tile, each
        // row hiding the keys beyond its own limit (a tile it fully sees loses
        // nothing). One path for all tiles keeps the loop's registers spill-free.
        const bool masked = kRowLimit ? true : last;
        constexpr int kM = kRowLimit ? kChunkMask : kElemMask;
        const int valid = kRowLimit ? row_lim - kBN * j : p.kv_tail;
        // Least `valid` over the warp (lane 0 has the warp's first row).
        const int vmin = kRowLimit ? __shfl_sync(0xFFFFFFFFu, valid, 0) : p.kv_tail;
        // Pass A: take the row extreme of S_j and, on a fold tile, add the TMEM
        // partial into the row (it holds the tiles since the last fold, complete
        // because the MMA that wrote S_j was issued after PV_{j-1}, and PV_j waits
        // for P_j).
        float ext, m_tile;
        bool need;
        if constexpr (kFoldOf<kPartial> == 1) {
          if (pos) {
            if (j == 0) {
              ext = masked ? fold_and_max<kM, false>(tS, tO, acc, valid, vmin)
                           : fold_and_max<kNoMask, false>(tS, tO, acc, kBN, kBN);
            } else {
              ext = masked ? fold_and_max<kM, true>(tS, tO, acc, valid, vmin)
                           : fold_and_max<kNoMask, true>(tS, tO, acc, kBN, kBN);
            }
          } else {
            ext = masked ? fold_and_min<true>(tS, tO, acc, valid, j > 0)
                         : fold_and_min<false>(tS, tO, acc, kBN, j > 0);
          }
          m_tile = ext * c;
          need = m_tile > m_used + kTau;  // false for NaN
          if (need) {
            const float f = ptx::ex2(m_used - m_tile);  // 0 when m_used = -Inf
            if (j > 0) rescale_row(acc, f);
            l *= f;
            m_used = m_tile;
          }
        } else {
          // The TMEM partial (key tiles since the last fold) is folded into the
          // registers every kFoldOf<kPartial> tiles.
          const bool fold_now = j > 0 && (j % kFoldOf<kPartial>) == 0;
          if (pos) {
            if (!fold_now) {
              ext = masked ? fold_and_max<kM, false>(tS, tO, acc, valid, vmin)
                           : fold_and_max<kNoMask, false>(tS, tO, acc, kBN, kBN);
            } else {
              ext = masked ? fold_and_max<kM, true>(tS, tO, acc, valid, vmin)
                           : fold_and_max<kNoMask, true>(tS, tO, acc, kBN, kBN);
            }
          } else {
            ext = masked ? fold_and_min<true>(tS, tO, acc, valid, fold_now)
                         : fold_and_min<false>(tS, tO, acc, kBN, fold_now);
          }
          m_tile = ext * c;
          need = m_tile > m_used + kTau;  // false for NaN
          float f_row = 1.f;  // this row's rescale factor at this tile
          if (need) {
            const float f = ptx::ex2(m_used - m_tile);  // 0 when m_used = -Inf
            if (j > 0) rescale_row(acc, f);
            l *= f;
            m_used = m_tile;
            f_row = f;
          }
          // A partial still in TMEM is relative to the old reference: scale it in
          // place (the PV MMAs that wrote it are done, S_j being ready; the next one
          // waits for P_j). Warp-uniform: each lane rescales its own row, by 1 if its
          // reference did not move.
          if ((j % kFoldOf<kPartial>) != 0 && __any_sync(0xFFFFFFFFu, need))
            rescale_tmem_row(tO, f_row);
        }
        const float m_sub = (m_used == neg_inf) ? 0.f : m_used;
        // Causal, c > 0: pass A left -Inf in the hidden columns, so pass B needs
        // no mask; for c <= 0 (where -Inf * c is not -Inf) it masks per element.
        const bool masked_b = kRowLimit ? !(c > 0.f) : last;
        if (kRowLimit) ptx::tmem_wait_st();  // pass A's write-backs before pass B reads
        l += masked_b ? tile_exp<true>(tS, valid, c, m_sub) : tile_exp<false>(tS, kBN, c, m_sub);
        ptx::tmem_wait_st();
        ptx::tc_fence_before();
        ptx::mbar_arrive(bar(kBarPFull + t));
      }

      if (ok) ok = warp_wait(bar(kBarOFull + t), 0, abort_flag, p.timeout_ns);
      // The work item again, from an opaque copy of the block index: the compiler
      // then keeps none of its fields live across the loop above.
      int bx = static_cast<int>(blockIdx.x);
      asm volatile("" : "+r"(bx));
      const Work wk = work_of<kCausal, kVarlen>(p, kPair ? p.item_base + bx : bx);
      if (kPartial && ok) {
        // Split epilogue: this row's unnormalised fp32 output, the running max it is
        // relative to, and its row sum.
        ptx::tc_fence_after();
        fold_last(tO, acc);
        const int q = (2 * wk.pair + t) * kBM + row;
        if (q < p.Sq) {
          const size_t r = (static_cast<size_t>(wk.split) * p.BH + wk.bh) * p.sq_pad + q;
          if (dbg_ok(r < static_cast<size_t>(p.n_splits) * p.BH * p.sq_pad)) {
            // Each packed pair holds columns 2i (low word) and 2i + 1: stored as is,
            // two pairs per 16-byte store.
            ulonglong2* dst = reinterpret_cast<ulonglong2*>(p.part_o + r * kD);
#pragma unroll
            for (int i = 0; i < kD / 4; ++i) dst[i] = make_ulonglong2(acc[2 * i], acc[2 * i + 1]);
            // The products are relative to m_used, or to 0 while it is -Inf (then no
            // key had a finite logit and both sums are 0, or NaN).
            reinterpret_cast<float2*>(p.part_rl)[r] = make_float2(m_used, l);
          }
        }
      } else if (ok) {
        ptx::tc_fence_after();
        fold_last(tO, acc);
        if constexpr (kPair) {
          // The two halves of the key range: rank 1 sends, rank 0 merges. Row R of
          // the CTA (0..255) is 512 bytes of the ring at R * 512, its 16-byte chunk
          // i at position i ^ (R & 31), so that the 8 rows of a quarter-warp's
          // 16-byte accesses fall in distinct banks.
          const int R = t * kBM + row;
          const uint32_t row_s = sRing + static_cast<uint32_t>(R) * 512u;
          const uint32_t ml_s = sbase + kOffPairMl + static_cast<uint32_t>(R) * 8u;
          if (ptx::cluster_ctarank() == 1) {
            // Wait (bounded) until rank 0's ring is free, then write this row there.
            const bool ready = wait_bounded_cluster(bar(kBarPeerReady), abort_flag, p.timeout_ns);
            if (ready) {
              const uint32_t dst = ptx::map_to_rank(row_s, 0);
#pragma unroll
              for (int i = 0; i < kD / 4; ++i) {
                const uint64_t a = acc[2 * i], b = acc[2 * i + 1];
                ptx::st_cluster_v4(dst + ((static_cast<uint32_t>(i) ^ (R & 31)) << 4),
                                   static_cast<uint32_t>(a), static_cast<uint32_t>(a >> 32),
                                   static_cast<uint32_t>(b), static_cast<uint32_t>(b >> 32));
              }
              ptx::st_cluster_v2(ptx::map_to_rank(ml_s, 0), __float_as_uint(m_used),
                                 __float_as_uint(l));
              ptx::mbar_arrive_cluster(ptx::map_to_rank(bar(kBarReceived), 0));
            }
            ok = false;  // rank 1 stores nothing
          } else {
            // Wait (bounded) for rank 1's 256 rows, then merge row R: both halves'
            // sums are relative to their own reference m (0 while m = -Inf); with
            // M = the larger one, O = 2^(m0 - M) O0 + 2^(m1 - M) O1 and likewise l.
            const bool got = wait_bounded_cluster(bar(kBarReceived), abort_flag, p.timeout_ns);
            ok = got;
            if (got) {
              const uint2 ml = *reinterpret_cast<const uint2*>(smem + (ml_s - sbase));
              const float m1 = __uint_as_float(ml.x), l1 = __uint_as_float(ml.y);
              const float neg_inf_m = -__int_as_float(0x7F800000);
              float M = fmaxf(m_used, m1);
              if (M == neg_inf_m) M = 0.f;
              const float w0 = ptx::ex2(m_used - M), w1 = ptx::ex2(m1 - M);
              // The same operations in the same order as the split-key combine
              // (an fma onto +0 first, then one onto that), so that both give the
              // same bits.
              l = fmaf(l1, w1, fmaf(l, w0, 0.f));
              const uint64_t w0_2 = ptx::f2_pack(w0, w0), w1_2 = ptx::f2_pack(w1, w1);
              const uint64_t zero2 = 0;
#pragma unroll
              for (int i = 0; i < kD / 4; ++i) {
                const uint4 x =
                    ptx::ld_shared_v4(row_s + ((static_cast<uint32_t>(i) ^ (R & 31)) << 4));
                acc[2 * i] = ptx::f2_fma((static_cast<uint64_t>(x.y) << 32) | x.x, w1_2,
                                         ptx::f2_fma(acc[2 * i], w0_2, zero2));
                acc[2 * i + 1] = ptx::f2_fma((static_cast<uint64_t>(x.w) << 32) | x.z, w1_2,
                                             ptx::f2_fma(acc[2 * i + 1], w0_2, zero2));
              }
            }
          }
        }
      }
      if (!kPartial && ok) {
        // Normalise, round, stage in the (now free) Q tile buffer with the TMA
        // 128-byte swizzle, and store this warp's 32 rows with two TMA boxes.
        const uint32_t stage_base = sQ + t * kTileBytes;
        const int mode = p.mode;
        const float inv_l = __frcp_rn(l);  // 0 -> Inf, so an all -Inf row gives 0 * Inf = NaN
        uint64_t inv2 = ptx::f2_pack(inv_l, inv_l);
        if constexpr (kRowLimit) {
          // Non-finite V values the check took out of the masked tiles: each key
          // this row sees adds its value, times a positive weight, to the column
          // (NaN stays NaN; +Inf and -Inf together give NaN); keys the row does
          // not see add nothing. Applied after normalisation, so that a row that
          // is NaN already stays NaN.
          const int jm = first_masked_tile<kCausal>(wk);
          const int nm = min(wk.n_kv - jm, kMaxMaskedTiles);
          const uint32_t* rec0 = reinterpret_cast<const uint32_t*>(smem + kOffVRec);
          bool any = false;
          for (int m = 0; m < nm; ++m)
            if (wait_bounded(bar(kBarVChk + m), 0, abort_flag, p.timeout_ns, true))
              any |= rec0[m * kVRecWords] != 0;
          if (any) {
            // One 32-column word of the three masks at a time (few live registers
            // next to the 128-column row).
            const float pos_inf = __int_as_float(0x7F800000);
#pragma unroll
            for (int cw = 0; cw < 4; ++cw) {
              uint32_t pn = 0, pp = 0, pm = 0;
              for (int m = 0; m < nm; ++m) {
                const uint32_t* rec = rec0 + m * kVRecWords;
                if (!rec[0]) continue;
                const int vis = row_lim - kBN * (jm + m);  // keys of this tile the row sees
                for (int wd = 0; wd < 4; ++wd) {
                  const int lim = vis - 32 * wd;
                  uint32_t km = lim <= 0 ? 0u : rec[kVRecKeyMask + wd];
                  if (lim < 32) km &= (1u << (lim > 0 ? lim : 0)) - 1u;
                  while (km) {
                    const int key = 32 * wd + __ffs(km) - 1;
                    km &= km - 1;
                    pn |= rec[kVRecNan + key * 4 + cw];
                    pp |= rec[kVRecPos + key * 4 + cw];
                    pm |= rec[kVRecNeg + key * 4 + cw];
                  }
                }
              }
              auto special = [&](int b) -> float {
                if (((pn | (pp & pm)) >> b) & 1u) return __int_as_float(0x7FC00000);
                if ((pp >> b) & 1u) return pos_inf;
                if ((pm >> b) & 1u) return -pos_inf;
                return -0.0f;  // x + (-0) = x for every x, signed zeros included
              };
#pragma unroll
              for (int i = 0; i < 16; ++i)
                acc[16 * cw + i] = ptx::f2_add(ptx::f2_mul(acc[16 * cw + i], inv2),
                                               ptx::f2_pack(special(2 * i), special(2 * i + 1)));
            }
            inv2 = ptx::f2_pack(1.0f, 1.0f);
          }
        }
#pragma unroll
        for (int ch = 0; ch < 4; ++ch) {
          uint32_t w[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            float o0, o1;
            ptx::f2_unpack(ptx::f2_mul(acc[16 * ch + i], inv2), o0, o1);
            w[i] = round_bf16_bits(o0, mode) | (round_bf16_bits(o1, mode) << 16);
          }
          const uint32_t half_base = stage_base + (ch >> 1) * kHalfBytes + row * 128;
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int chunk = (ch & 1) * 4 + u;
            ptx::st_shared_v4(half_base + ((chunk ^ (row & 7)) << 4), w[4 * u], w[4 * u + 1],
                              w[4 * u + 2], w[4 * u + 3]);
          }
        }
        ptx::fence_proxy_async_smem();
        __syncwarp();
        const int q_row0 = (2 * wk.pair + t) * kBM + wq * 32;  // within the sequence
        if (!kVarlen || q_row0 + 32 <= wk.sq) {
          if (lane == 0 && q_row0 < wk.sq && dbg_ok(wk.q_base + q_row0 < p.Sq)) {
            int c1, c2;
            tma_coords(p.layout, wk.q_base + q_row0, wk.head, c1, c2);
            for (int hf = 0; hf < 2; ++hf)
              ptx::tma_store_4d_hint(&tm_o, stage_base + hf * kHalfBytes + wq * 32 * 128, 64 * hf, c1,
                                     c2, wk.batch, ptx::l2_policy_evict_first());
            ptx::bulk_commit_group();
            ptx::bulk_wait_group_0();
          }
        } else if (lane < wk.sq - q_row0 && dbg_ok(wk.q_base + q_row0 + lane < p.Sq)) {
          // The sequence ends inside this warp's rows: a TMA box would run into the
          // next sequence's rows, so each row up to the end is copied out of the
          // staging buffer with plain 16-byte stores (packed layout: token, head).
          const uint8_t* stage = smem + (stage_base - sbase);
          uint4* dst = reinterpret_cast<uint4*>(
              p.out + (static_cast<size_t>(wk.q_base + q_row0 + lane) * p.H + wk.head) * kD);
#pragma unroll
          for (int cix = 0; cix < 16; ++cix) {
            const int off = (cix >> 3) * kHalfBytes + row * 128 + (((cix & 7) ^ (row & 7)) << 4);
            dst[cix] = *reinterpret_cast<const uint4*>(stage + off);
          }
        }
        __syncwarp();
      }
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kTmemCols);
  }
  // Pair variant: the grid completes only after the launch it may overlap (the
  // full waves of the same call), so that later work on the stream sees both;
  // and neither CTA leaves while the other may still use its shared memory.
  // Every thread reaches this point (all waits above are bounded).
  if constexpr (kPair) {
    ptx::grid_dependency_wait();
    ptx::cluster_sync();
  }
}

}  // namespace attn
