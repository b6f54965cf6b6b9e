// fa_kernel.cuh -- FlashAttention-2 forward for sm_103a: TMA-fed shared-memory
// rings, tcgen05 MMAs accumulating in tensor memory (TMEM), and one softmax
// warpgroup per 128-row query tile (TMEM lane i = query row i).
//
// What it computes (per batch b, query head h, query row i):
//   O_i = softmax_j(scale * q_i . k_j + mask_ij) v_j,  L_i = m_i + ln(l_i)
// with causal (j <= i) masking, GQA (K/V head = h / (H_q / H_kv)), optional
// bool (nonzero keeps) or additive masks, and ragged tails; in the feature
// instantiations also a sliding window, a causal diagonal offset, a softcap
// and (its own instantiations) dropout.  Sources:
//  - mlx-native "ops/flash_attn_train.rs", module doc "Algorithm": FA-2
//    online softmax with the score pre-scaled by scale*log2(e) so the running
//    max and sum live in base 2, and L = m2 * ln2 + ln(l2) written per row;
//    "Buffer layout" ([B,H_q,qL,D] Q/O, [B,H_kv,kL,D] K/V, [B,H_q,qL] L).
//  - forge "flash_attention_mma.metal", header and kernel body: split-Q
//    (each row owned by one worker for the whole KV sweep), causal KV loop
//    bounded by the tile's last row, per-row rescale of O by exp(m_old -
//    m_new), and the epilogue O / l with l == 0 giving O = 0.
//  - ruDNN "dense_attention.rs", functions `forward` (mask kinds, -inf
//    exclusion) and `forward_flash` (exp2 domain, bf16 unnormalised P with
//    fp32 accumulation).
//  - oxibonsai "dit_attention_flash.rs", module doc: head-major input with
//    the transpose to token-major output folded into the epilogue.
//
// GB300 design (differs from the pages' Apple-GPU kernels):
//  - persistent grid: one CTA per SM walks a snake-ordered share of the
//    (query block, head, batch) work units, heavy causal blocks first; every
//    role carries its barrier phases across units, so the next unit's loads
//    and first MMAs overlap the current unit's last blocks and epilogue;
//  - warp 0 issues TMA loads: Q per unit, then K, V (and, for D = 256 bf16,
//    mask) tiles through mbarrier rings, in the order the tensor core reads
//    them;
//  - warp 1 (and warp 2 for two bf16 Q tiles, taking strict turns) issues
//    every tcgen05.mma from one thread: S = Q K^T (both operands in shared
//    memory, K-major, 128-byte swizzle) and O += P V (P read from TMEM, V
//    MN-major from shared memory for bf16, a transposed V^T for tf32);
//  - warps 2-3 (fp32 I/O without the pre-pass only) round Q and K tiles to
//    tf32 in place and transpose V; the pre-rounded fp32 plans load V^T tiles
//    from HBM instead;
//  - one softmax warpgroup per 128-row Q tile: thread r owns row r (TMEM lane
//    r), reads its S row with tcgen05.ld, applies masks, updates the base-2
//    running max/sum, writes P back to TMEM and rescales its O row in TMEM
//    only when the running max grows by more than 2^8 (exact: O and l share
//    the stale max; the epilogue divides it out);
//  - two Q tiles per CTA ping-pong on the tensor core where TMEM allows (P
//    over S); with one tile, S and P have their own columns and S_{j+1} is
//    computed while softmax j runs;
//  - epilogue: O / l -> I/O dtype -> 16-byte global stores straight from
//    registers (any {batch, head, row} strides, e.g. token-major), L in fp32;
//  - every wait is bounded; on expiry the kernel records kStatusTimeout,
//    drains its own copies and MMAs, frees TMEM and returns.
#pragma once

#include <cuda.h>
#include <stdint.h>

#include "fa_params.h"
#include "fa_ptx.cuh"

namespace fa {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
// The running max is only moved (and O rescaled) when it grows by more than
// this many powers of two; unnormalised p then stays below 2^8.
constexpr float kRescaleThreshold = 8.0f;
// Bound on the exit-time drains (copies and MMAs still in flight after an
// abort); independent of the configurable wait bound so a short bound never
// lets TMEM or shared memory go while the hardware still writes to them.
constexpr long long kDrainCycles = 1LL << 33;

template <bool kTf32_, int kD_, int kNQT_, int kBN_, int kKStages_, int kVStages_, int kVTStages_ = 0,
          bool kF16_ = false, bool kFeat_ = false, bool kDrop_ = false, bool kPre_ = false>
struct Cfg {
  static constexpr bool kTf32 = kTf32_;
  // fp32 I/O whose Q and K arrive already rounded to tf32 and whose V arrives
  // rounded and transposed ([B, H_kv, D, keys], from the pre-pass): the
  // producer loads the K-major V^T tiles straight into the V ring and no
  // helper warps run.  Otherwise fp32 I/O rounds and transposes in shared
  // memory with helper warps.
  static constexpr bool kPre = kPre_;
  static constexpr bool kHelpers = kTf32 && !kPre;
  // Sliding window, softcap and query offset compiled in (a separate
  // instantiation, so the plain forward keeps its exact code).
  static constexpr bool kFeat = kFeat_;
  // Dropout compiled in as well (its own instantiation again: its keep-bit
  // bookkeeping costs the other features 3-5%).
  static constexpr bool kDrop = kDrop_;
  // 16-bit I/O is bf16 unless kF16 (fp16): same kernel, other operand format.
  static constexpr bool kF16 = kF16_;
  static constexpr uint32_t kFmt = kTf32 ? kFmtTf32 : (kF16 ? kFmtF16 : kFmtBf16);
  static constexpr CUtensorMapDataType kTmaType =
      kTf32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : (kF16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16);
  static constexpr int kD = kD_;
  static constexpr int kEsz = kTf32 ? 4 : 2;          // bytes per stored element
  static constexpr int kChunk = 128 / kEsz;           // elements per 128-byte swizzle row
  static constexpr int kNChunk = kD / kChunk;         // swizzle column blocks per row
  static constexpr int kBM = 128;                     // rows per Q tile (= TMEM lanes)
  static constexpr int kNQT = kNQT_;                  // Q tiles per CTA
  static constexpr int kBN = kBN_;                    // keys per KV tile
  static constexpr int kKStages = kKStages_;
  static constexpr int kVStages = kVStages_;
  // TF32 MMAs take B only K-major, so fp32 I/O transposes each V tile into a
  // K-major V^T ring ([D rows x kBN keys]); bf16 reads V MN-major directly.
  static constexpr int kVTStages = kVTStages_;
  static constexpr int kKStep = kTf32 ? 8 : 16;       // MMA K per instruction (32 bytes)
  static constexpr bool kAliasP = (kNQT == 2);        // P over S; PV issued before the next S
  // K/V load order follows the tensor core's: with P over S it runs PV_j, S_{j+1}
  // (K_j, V_j, K_{j+1}, ...); otherwise S_{j+1} goes before PV_j, so V lags K by a block.
  static constexpr int kVLag = kAliasP ? 0 : 1;
  // MMA-issuing threads.  One warp issues at most one tcgen05.mma per ~54
  // cycles (measured), and anything else it does between MMAs adds to that,
  // while a 128x128x16 MMA is 64 cycles of work: with two bf16 Q tiles, tile
  // t's MMAs come from warp 1 + t and the two threads take strict turns, so
  // the tensor core still sees PV0 S0 PV1 S1 (the ping-pong order) while each
  // thread's waits and commits overlap the other's MMA issue.
  static constexpr int kIssuers = (kNQT == 2 && !kTf32) ? 2 : 1;
  static constexpr int kPCols = kTf32 ? kBN : kBN / 2;  // TMEM columns of one P tile
  static constexpr int kColO = kNQT * kBN;            // first O column
  static constexpr int kColP = kColO + kNQT * kD;     // P double buffer (non-aliased mode)
  static constexpr int kTmemUsed = kAliasP ? kNQT * (kBN + kD) : (kBN + kD + 2 * kPCols);
  static constexpr uint32_t kTmemCols =
      kTmemUsed <= 32 ? 32 : kTmemUsed <= 64 ? 64 : kTmemUsed <= 128 ? 128 : kTmemUsed <= 256 ? 256 : 512;
  // tf32 helper warps: warps 2-3, plus warps 8-11 when there is one Q tile
  // (rounding K and transposing V then keep pace with the tensor core).
  static constexpr bool kExtraHelpers = kHelpers && kNQT == 1;
  // One Q tile with 16-bit I/O (no dropout): two softmax warpgroups share the
  // tile, each taking 64 of a block's 128 keys for all 128 rows, so every SM
  // sub-partition runs two softmax warps (one alone leaves its latency bare).
  static constexpr bool kSplitRows = kNQT == 1 && !kTf32 && !kDrop;
  // Split-KV: the one-Q-tile 16-bit plans at D <= 128 without features may
  // cut a tile's key blocks into ranges (FaParams::kv_splits), each its own
  // work unit.
  static constexpr bool kSplitKV = kNQT == 1 && !kTf32 && !kFeat && !kDrop && kD <= 128;
  static constexpr int kCvtWarps = kHelpers ? (kExtraHelpers ? 6 : 2) : 1;
  static constexpr int kCvtThreads = 32 * kCvtWarps;
  static constexpr int kThreads = 128 * (1 + kNQT) + (kExtraHelpers || kSplitRows ? 128 : 0);
  // Per-thread registers at launch, and the split after setmaxnreg: the
  // control warpgroup (TMA, MMA, tf32 helpers) gives registers to the softmax
  // warpgroups.  Sums stay within the launch total (kThreads * kRegsLaunch).
  static constexpr int kRegsLaunch = kThreads == 384 ? 168 : 255;
  static constexpr int kRegsCtrl = 80;
  static constexpr int kRegsSoftmax = (kNQT == 2 || kSplitRows) ? 208 : 0;  // 0: no reallocation
  static_assert(kRegsSoftmax == 0 || 128 * kRegsCtrl + 256 * kRegsSoftmax <= kThreads * kRegsLaunch,
                "register split exceeds the launch allocation");
  static constexpr uint32_t kQTileBytes = kBM * kD * kEsz;
  static constexpr uint32_t kKVTileBytes = kBN * kD * kEsz;
  static constexpr uint32_t kOffK = kNQT * kQTileBytes;
  static constexpr uint32_t kOffV = kOffK + kKStages * kKVTileBytes;
  static constexpr uint32_t kOffVT = kOffV + kVStages * kKVTileBytes;
  // One shared-memory slot for a TMA-loaded mask tile [kBM rows x kBN keys]
  // (sized for a 2-byte additive mask; a 1-byte bool tile uses half).  Only
  // where shared memory allows: 16-bit I/O with one Q tile, except in the
  // dropout instantiation, whose keep bits take the room (its masks are read
  // from L2).
  static constexpr uint32_t kMaskSlotBytes = (!kTf32 && kNQT == 1 && !kDrop) ? kBM * kBN * 2 : 0;
  static constexpr uint32_t kOffM = kOffVT + kVTStages * kKVTileBytes;
  // Dropout keep bits of each row's next block (kBN / 8 bytes per row) in
  // shared memory for 16-bit I/O, whose softmax warps have no registers to
  // spare; in registers for fp32 I/O.
  static constexpr bool kDropSmem = kDrop && !kTf32;
  static constexpr uint32_t kDropBytes = kDropSmem ? kNQT * kBM * (kBN / 8) : 0;
  static constexpr uint32_t kOffDrop = kOffM + kMaskSlotBytes;
  static constexpr uint32_t kBarBytes = 512;
  // Two-tile 16-bit plans: each softmax warp stages its 32 rows of O, one
  // 128-byte column block at a time (4 KB), in shared memory, so the global
  // stores of the epilogue write whole 128-byte lines (four rows per warp
  // instruction) instead of 16 bytes of 32 different rows.  Only where the
  // 32 KB fit.
  static constexpr uint32_t kOStageBytes = 8 * 32 * 128;
  static constexpr bool kOStage =
      kAliasP && !kTf32 && 1024 + kOffDrop + kDropBytes + kOStageBytes + kBarBytes <= 232448;
  static constexpr uint32_t kOffOStage = kOffDrop + kDropBytes;
  static constexpr uint32_t kOffBar = kOffOStage + (kOStage ? kOStageBytes : 0);
  static_assert(!kOStage || kOffOStage % 1024 == 0, "the O staging slots are 128-byte-swizzled TMA boxes");
  static constexpr uint32_t kSmemBytes = 1024 + kOffBar + kBarBytes;  // + alignment slack

  static_assert(kD % kChunk == 0, "head dim must be a whole number of 128-byte rows");
  static_assert(kBN % 32 == 0 && kBN >= 32 && kBN <= 256, "KV tile must be 32..256, multiple of 32");
  static_assert(kD % 16 == 0 && kD <= 256, "PV MMA needs N = D in 16..256");
  static_assert(kTmemUsed <= 512, "TMEM overflow");
  static_assert(kSmemBytes <= 232448, "shared memory overflow");
  static_assert(kKStages >= 1 && kVStages >= 1 && kKStages <= 4 && kVStages <= 4, "ring size");
  static_assert(kHelpers ? (kVTStages >= 1 && kVTStages <= 4) : kVTStages == 0,
                "the V^T ring is for TF32 with helper warps only");
  static_assert(!kPre || kTf32, "pre-rounded inputs are fp32");
  static_assert(!(kTf32 && kF16), "fp16 I/O uses the 16-bit path");
  static_assert(!kDrop || kFeat, "the dropout instantiation includes the other features");
};

// Shared-memory control block (after the tiles).
template <class C>
struct Ctrl {
  uint64_t q_full[2];             // TMA -> Q tile t landed
  uint64_t q_empty[2];            // the unit's last S of tile t done: Q_t may be reloaded
  uint64_t q_ready[2];            // (tf32) Q tile t rounded in place
  uint64_t k_full[4], k_empty[4], k_ready[4];
  uint64_t v_full[4], v_empty[4];
  uint64_t vt_full[4], vt_empty[4];  // (tf32) transposed V tiles
  uint64_t m_full, m_empty;          // mask tile in shared memory
  uint64_t s_full[2];             // S_t computed (commit)
  uint64_t s_free[2];             // (one Q tile) softmax t holds S in registers: S may be overwritten
  uint64_t p_ready[2];            // softmax t wrote P (and rescaled O)
  uint64_t o_ready[2];            // PV_t completed (commit)
  uint64_t o_free[2];             // epilogue read O_t out of TMEM
  uint64_t drain[2];              // MMA drain at exit, one per issuing thread
  uint32_t tmem_base;
  int abort;
  uint64_t turn_bar[2];           // two issuers: issuer i may issue its next MMA group
};

// Two fp32 values -> the 16-bit I/O format's packed pair (`lo` in bits 0-15).
template <class C>
__device__ __forceinline__ uint32_t pack16x2(float lo, float hi) {
  if constexpr (C::kF16)
    return pack_f16x2(lo, hi);
  else
    return pack_bf16x2(lo, hi);
}

// Bounded wait: true once the phase of `parity` completed; false after the
// CTA-wide abort flag is raised or `timeout` cycles pass (then it raises the
// flag and records the timeout in the device status word).
__device__ __forceinline__ bool wait_bounded(uint64_t* bar, uint32_t parity, volatile int* abort,
                                             unsigned int* status, long long timeout, bool honour_abort = true) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64_now();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (honour_abort && *abort) return false;
    if (clock64_now() - t0 > timeout) {
      *abort = 1;
      atomicOr(status, kStatusTimeout);
      return false;
    }
  }
}

__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort, unsigned int* status,
                                          long long timeout) {
  const bool ok = wait_bounded(bar, parity, abort, status, timeout);
  return __all_sync(0xffffffffu, ok);
}

// KV tiles a 128-row Q tile starting at r0 visits: [tile_kv_begin, tile_kv_blocks).
// tile_kv_blocks is 0 when the tile has no rows, and at least 1 otherwise (a
// tile whose rows see no key still runs one fully masked block, which writes
// O = 0 and L = -inf).
template <class C>
__device__ __forceinline__ int tile_kv_blocks(const FaParams& p, int r0) {
  if (r0 >= p.qL) return 0;
  const int last = min(r0 + C::kBM, p.qL) - 1;
  if constexpr (!C::kFeat) {
    const int kv_end = p.causal ? min(p.kL, last + 1) : p.kL;
    return (kv_end + C::kBN - 1) / C::kBN;
  }
  const long long diag_end = (long long)last + 1 + (C::kFeat ? p.q_offset : 0);  // one past the last row's diagonal key
  const int kv_end = p.causal ? (int)max(0LL, min((long long)p.kL, diag_end)) : p.kL;
  return max(1, (kv_end + C::kBN - 1) / C::kBN);
}
// First KV tile any row of the tile starting at r0 can see (sliding window).
template <class C>
__device__ __forceinline__ int tile_kv_begin(const FaParams& p, int r0, int nblk) {
  if (!C::kFeat || p.window <= 0) return 0;
  const long long first = (long long)r0 + p.q_offset - p.window + 1;  // row r0's first key
  const int b0 = first <= 0 ? 0 : (int)min(first / C::kBN, (long long)0x7fffffff);
  return min(b0, max(nblk - 1, 0));
}

// Round a tile of fp32 values in shared memory to tf32 (round to nearest).
__device__ __forceinline__ void round_tf32_inplace(uint8_t* base, uint32_t bytes, int tid, int nthreads) {
  uint4* p4 = reinterpret_cast<uint4*>(base);
  const uint32_t n = bytes / 16;
  for (uint32_t i = tid; i < n; i += nthreads) {
    uint4 v = p4[i];
    v.x = to_tf32(__uint_as_float(v.x));
    v.y = to_tf32(__uint_as_float(v.y));
    v.z = to_tf32(__uint_as_float(v.z));
    v.w = to_tf32(__uint_as_float(v.w));
    p4[i] = v;
  }
}

// Transpose a landed V tile (rows = kBN keys, 128-byte swizzled rows of 32
// fp32, D/32 column blocks) into V^T (rows = D, 128-byte swizzled rows of 32
// keys, kBN/32 column blocks), rounding to tf32: the K-major B operand of
// O += P V for TF32.
// Each step moves a 4 keys x 4 d block with four 16-byte loads and stores.
// Within 8 consecutive threads both the d-group and the key-group run
// through 8 distinct values (diagonals of 8x8 block super-tiles), so the
// swizzled 16-byte units they touch are distinct: no bank conflicts.
template <class C>
__device__ __forceinline__ void transpose_v_tile(const uint8_t* src, uint8_t* dst, int tid, int nthreads) {
  constexpr int kKG = C::kBN / 32;  // key super-groups (8 groups of 4 keys each)
  constexpr int kBlocks = (C::kBN / 4) * (C::kD / 4);
  for (int blk = tid; blk < kBlocks; blk += nthreads) {
    const int t8 = blk & 7, diag = (blk >> 3) & 7, st = blk >> 6;
    const int kg = (st % kKG) * 8 + ((t8 + diag) & 7);  // group of keys 4kg .. 4kg+3
    const int dg = (st / kKG) * 8 + t8;                 // group of d 4dg .. 4dg+3
    float4 in[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int r = 4 * kg + i;
      in[i] = *reinterpret_cast<const float4*>(src + (dg >> 3) * (C::kBN * 128) + r * 128 +
                                               (((dg & 7) ^ (r & 7)) << 4));
    }
#pragma unroll
    for (int jd = 0; jd < 4; ++jd) {
      const int d = 4 * dg + jd;
      // Rounded to tf32 here: the tensor core would otherwise drop the low
      // mantissa bits, an error that rows with few allowed keys (O close to
      // a single V row) would see directly.
      uint4 o;
      o.x = to_tf32((&in[0].x)[jd]);
      o.y = to_tf32((&in[1].x)[jd]);
      o.z = to_tf32((&in[2].x)[jd]);
      o.w = to_tf32((&in[3].x)[jd]);
      *reinterpret_cast<uint4*>(dst + (kg >> 3) * (C::kD * 128) + d * 128 + (((kg & 7) ^ (d & 7)) << 4)) = o;
    }
  }
}

// Fold two additive mask values into a pair of scores: s += m * f, with
// f = 1 / scale while the scores are raw (the softmax's scale * log2(e)
// factor then covers mask and score alike) or f = log2(e) once they are
// scaled to base 2 (after a softcap, or for a non-positive scale).
__device__ __forceinline__ void fold_add2(float& s0, float& s1, float m0, float m1, float f) {
  ffma2(s0, s1, m0, m1, f, f, s0, s1);
}

// Load 32 mask entries [k0, k0+32) of one row and fold them into s[off .. off+32):
// additive: fold_add2; bool: s = -inf where the mask is zero.  Keys >= kL are
// left alone (cut by the tail limit).
template <class C, int kMaskKind>
__device__ __forceinline__ void fold_mask_chunk(float* s, const void* mrow_v, int k0, int kL, bool vec, float f) {
  if constexpr (kMaskKind == 1) {
    const uint8_t* mrow = static_cast<const uint8_t*>(mrow_v);
    if (vec && k0 + 32 <= kL) {
      const uint4* m4 = reinterpret_cast<const uint4*>(mrow + k0);
#pragma unroll
      for (int v = 0; v < 2; ++v) {
        const uint4 w = __ldg(m4 + v);
        const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const uint32_t byte = (ws[e >> 2] >> ((e & 3) * 8)) & 0xFFu;
          if (byte == 0u) s[v * 16 + e] = -INFINITY;
        }
      }
    } else {
#pragma unroll
      for (int e = 0; e < 32; ++e)
        if (k0 + e < kL && __ldg(mrow + k0 + e) == 0) s[e] = -INFINITY;
    }
  } else {
    if constexpr (C::kTf32) {
      const float* mrow = static_cast<const float*>(mrow_v);
      if (vec && k0 + 32 <= kL) {
        const float4* m4 = reinterpret_cast<const float4*>(mrow + k0);
#pragma unroll
        for (int v = 0; v < 8; ++v) {
          const float4 w = __ldg(m4 + v);
          fold_add2(s[v * 4 + 0], s[v * 4 + 1], w.x, w.y, f);
          fold_add2(s[v * 4 + 2], s[v * 4 + 3], w.z, w.w, f);
        }
      } else {
#pragma unroll
        for (int e = 0; e < 32; ++e)
          if (k0 + e < kL) s[e] = fmaf(__ldg(mrow + k0 + e), f, s[e]);
      }
    } else {
      const uint16_t* mrow = static_cast<const uint16_t*>(mrow_v);
      if (vec && k0 + 32 <= kL) {
        const uint4* m4 = reinterpret_cast<const uint4*>(mrow + k0);
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          const uint4 w = __ldg(m4 + v);
          const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
          for (int e = 0; e < 8; e += 2)
            fold_add2(s[v * 8 + e], s[v * 8 + e + 1], half_bits_to_f32<C::kF16>(ws[e >> 1]),
                      half_bits_to_f32<C::kF16>(ws[e >> 1] >> 16), f);
        }
      } else {
#pragma unroll
        for (int e = 0; e < 32; ++e)
          if (k0 + e < kL) s[e] = fmaf(half_bits_to_f32<C::kF16>(__ldg(mrow + k0 + e)), f, s[e]);
      }
    }
  }
}

// Fold one row of a TMA-loaded mask tile (128-byte swizzled rows; 2-byte
// additive values in kBN/64 column blocks, or 1-byte bool values in one) into
// s, like fold_mask_chunk does from global memory.
template <class C, int kCols = C::kBN>
__device__ __forceinline__ void fold_mask_smem(float (&s)[kCols], const uint8_t* tile, int kind, int tl, float f,
                                               int coff = 0) {  // coff: the tile column of s[0] (a multiple of 16)
  if (kind == 1) {
#pragma unroll
    for (int c = 0; c < kCols / 16; ++c) {  // 16 keys per 16-byte unit
      const int un = coff / 16 + c;
      const uint4 w = *reinterpret_cast<const uint4*>(tile + (un / 8) * (C::kBM * 128) + tl * 128 +
                                                      (((un % 8) ^ (tl & 7)) << 4));
      const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int e = 0; e < 16; ++e)
        if (((ws[e >> 2] >> ((e & 3) * 8)) & 0xFFu) == 0u) s[c * 16 + e] = -INFINITY;
    }
  } else {
#pragma unroll
    for (int c = 0; c < kCols / 8; ++c) {  // 8 bf16 keys per 16-byte unit
      const int un = coff / 8 + c;
      const uint4 w = *reinterpret_cast<const uint4*>(tile + (un / 8) * (C::kBM * 128) + tl * 128 +
                                                      (((un % 8) ^ (tl & 7)) << 4));
      const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int e = 0; e < 8; e += 2)
        fold_add2(s[c * 8 + e], s[c * 8 + e + 1], half_bits_to_f32<C::kF16>(ws[e >> 1]),
                  half_bits_to_f32<C::kF16>(ws[e >> 1] >> 16), f);
    }
  }
}

template <class C, int kCols = C::kBN>
__device__ __forceinline__ void apply_mask(float (&s)[kCols], const FaParams& p, int b, int h, int row, int kbase,
                                           const uint8_t* mask_tile, int tl, int coff = 0) {
  // s holds keys kbase .. kbase + kCols - 1; coff is their first column in the block's mask tile.
  // Scores to base 2 first when a softcap applies, the scale is not positive,
  // or an additive mask meets either.  The softcap c * tanh(y) (y = scale * s
  // / c) uses tanh(y) = 1 - 2 / (2^(2 log2(e) y) + 1): one ex2 and one
  // reciprocal, exact limits +-1 when the power overflows or underflows, and
  // an absolute error of a few fp32 ulps of 1 near y = 0 (what the capped
  // score needs).
  if (p.pre_scale) {
    if (C::kFeat && p.softcap_on) {
      const float kin = 2.0f * kLog2e * p.softcap_in, cout = p.softcap_out;
#pragma unroll
      for (int c = 0; c < kCols; ++c) s[c] = fmaf(-2.0f * cout, rcp_approx(ex2(s[c] * kin) + 1.0f), cout);
    } else {
#pragma unroll
      for (int c = 0; c < kCols; c += 2) fmul2(s[c], s[c + 1], s[c], s[c + 1], p.scale_log2, p.scale_log2);
    }
  }
  const float f = p.mask_natural ? p.inv_scale : kLog2e;  // additive mask factor
  if constexpr (C::kMaskSlotBytes > 0) {
    if (mask_tile) fold_mask_smem<C, kCols>(s, mask_tile, p.mask_kind, tl, f, coff);
  }
  if (p.mask_kind != 0 && row < p.qL && !(C::kMaskSlotBytes > 0 && mask_tile)) {
    const size_t esz = (p.mask_kind == 1) ? 1 : C::kEsz;
    const char* mrow = static_cast<const char*>(p.mask) +
                       ((long long)b * p.mask_sb + (long long)h * p.mask_sh + (long long)row * p.mask_ss) * esz;
    const bool vec = p.mask_vec != 0;
#pragma unroll
    for (int cc = 0; cc < kCols / 32; ++cc) {
      if (p.mask_kind == 1)
        fold_mask_chunk<C, 1>(s + cc * 32, mrow, kbase + cc * 32, p.kL, vec, f);
      else
        fold_mask_chunk<C, 2>(s + cc * 32, mrow, kbase + cc * 32, p.kL, vec, f);
    }
  }
  // Causal, tail and window limits: key kbase + c is allowed iff lo <= c < lim.
  const int diag = row + (C::kFeat ? p.q_offset : 0) - kbase;  // this row's diagonal key, relative to kbase
  int lim = p.kL - kbase;
  if (p.causal) lim = min(lim, diag + 1);
  const int lo = (C::kFeat && p.window > 0) ? diag - p.window + 1 : -1;
  if (lim < kCols || lo > 0) {  // most blocks lie wholly inside the limits
#pragma unroll
    for (int c = 0; c < kCols; ++c)
      if (c >= lim || c < lo) s[c] = -INFINITY;
  }
}

// Row max of s (raw or base-2 scores): three-input max, four chains.
template <class C, int kCols = C::kBN>
__device__ __forceinline__ float row_max(const float (&s)[kCols]) {
  float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
  for (int c = 0; c < kCols; c += 8) {
    mx4[0] = fmax3(mx4[0], s[c + 0], s[c + 1]);
    mx4[1] = fmax3(mx4[1], s[c + 2], s[c + 3]);
    mx4[2] = fmax3(mx4[2], s[c + 4], s[c + 5]);
    mx4[3] = fmax3(mx4[3], s[c + 6], s[c + 7]);
  }
  return fmax3(fmaxf(mx4[0], mx4[1]), mx4[2], mx4[3]);
}

// One pass over a row: p = 2^(s*sl - msub) stored to TMEM at tP (bf16 pairs,
// or tf32), the fp32 sum of p, and with kWithMax the row max of s on the
// side.  Pairs of scores go through packed fp32x2 FMA / add; the
// exponentials through the SFU one at a time.
template <class C, bool kWithMax, int kCols = C::kBN>
__device__ __forceinline__ void p_pass(const float (&s)[kCols], float sl, float msub, uint32_t tP, float& sum,
                                       float& mx) {
  float sum4[4] = {0.0f, 0.0f, 0.0f, 0.0f};
  float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
  for (int cc = 0; cc < kCols / 32; ++cc) {
    uint32_t pk[C::kTf32 ? 32 : 16];
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      const float s0 = s[cc * 32 + 2 * e], s1 = s[cc * 32 + 2 * e + 1];
      if constexpr (kWithMax) mx4[e & 3] = fmax3(mx4[e & 3], s0, s1);
      float x0, x1;
      ffma2(x0, x1, s0, s1, sl, sl, -msub, -msub);
      const float p0 = ex2(x0), p1 = ex2(x1);
      fadd2(sum4[(e & 1) * 2], sum4[(e & 1) * 2 + 1], p0, p1);
      if constexpr (C::kTf32) {
        pk[2 * e] = to_tf32(p0);
        pk[2 * e + 1] = to_tf32(p1);
      } else {
        pk[e] = pack16x2<C>(p0, p1);
      }
    }
    if constexpr (C::kTf32)
      tmem_st32(tP + cc * 32, pk);
    else
      tmem_st16(tP + cc * 16, pk);
  }
  sum = (sum4[0] + sum4[1]) + (sum4[2] + sum4[3]);
  if constexpr (kWithMax) mx = fmax3(fmaxf(mx4[0], mx4[1]), mx4[2], mx4[3]);
}

// One 32 x 32 -> 64-bit product as a single wide multiply: high and low words.
__device__ __forceinline__ void mul_wide(uint32_t a, uint32_t b, uint32_t& hi, uint32_t& lo) {
  asm("{\n\t.reg .b64 w;\n\tmul.wide.u32 w, %2, %3;\n\tmov.b64 {%1, %0}, w;\n\t}"
      : "=r"(hi), "=r"(lo)
      : "r"(a), "r"(b));
}

// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, SC11): ten rounds of the
// published round function on the counter (c0, c1, 0, 0) with key (k0, k1).
// The dropout path runs it once per 4 keys, between the softmax passes (the
// scores are dead there), so it is inlined.
__device__ __forceinline__ uint4 philox_10(uint32_t c0, uint32_t c1, uint32_t k0, uint32_t k1) {
  uint32_t x0 = c0, x1 = c1, x2 = 0u, x3 = 0u;
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    uint32_t hi0, lo0, hi2, lo2;
    mul_wide(0xD2511F53u, x0, hi0, lo0);
    mul_wide(0xCD9E8D57u, x2, hi2, lo2);
    x0 = hi2 ^ x1 ^ k0;
    x1 = lo2;
    x2 = hi0 ^ x3 ^ k1;
    x3 = lo0;
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
  return make_uint4(x0, x1, x2, x3);
}

// Keep bits of one row's block of 32 * kWords keys: bit i of word q is key
// kbase + 32 q + i.
// Position ((b H_q + h) qL + row) kL + key, counter = offset + position / 4,
// word = position % 4 (kL is a multiple of 4, so 4 keys share one counter);
// `ctr` is the counter of key kbase.  Computed for block j + 1 while the warp
// would otherwise wait for S_{j+1}, so the generator stays off the softmax's
// critical path.
// One keep word: 8 generator blocks of 4 keys from counter `ctr`.
__device__ __forceinline__ uint32_t drop_word(const FaParams& p, unsigned long long ctr) {
  uint32_t acc = 0;
#pragma unroll
  for (int g = 0; g < 8; ++g) {
    const unsigned long long c = ctr + (unsigned long long)g;
    const uint4 r = philox_10((uint32_t)c, (uint32_t)(c >> 32), p.seed_lo, p.seed_hi);
    acc |= ((r.x >> 8) >= p.drop_threshold ? 1u : 0u) << (4 * g);
    acc |= ((r.y >> 8) >= p.drop_threshold ? 1u : 0u) << (4 * g + 1);
    acc |= ((r.z >> 8) >= p.drop_threshold ? 1u : 0u) << (4 * g + 2);
    acc |= ((r.w >> 8) >= p.drop_threshold ? 1u : 0u) << (4 * g + 3);
  }
  return acc;
}
template <int kWords>
__device__ __forceinline__ void drop_bits(const FaParams& p, unsigned long long ctr, uint32_t (&kb)[kWords]) {
#pragma unroll
  for (int q = 0; q < kWords; ++q) kb[q] = drop_word(p, ctr + (unsigned long long)(q * 8));
}

// p_pass with dropout: the same P and sum, but the stored P (what P V
// reads) is zero for dropped keys; the sum (l) keeps them.  The 1 / (1 - p)
// of kept keys is applied to O in fp32 by the epilogue, so P carries no
// rounding of it.
template <class C, class KB>
__device__ __forceinline__ void p_pass_dropout(const float (&s)[C::kBN], float sl, float msub, uint32_t tP, float& sum,
                                               const KB& keep_word) {  // keep_word(cc): bits of keys 32 cc ..
  float sum4[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
  for (int cc = 0; cc < C::kBN / 32; ++cc) {
    uint32_t pk[C::kTf32 ? 32 : 16];
    const uint32_t kw = keep_word(cc);
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      float x0, x1;
      ffma2(x0, x1, s[cc * 32 + 2 * e], s[cc * 32 + 2 * e + 1], sl, sl, -msub, -msub);
      const float p0 = ex2(x0), p1 = ex2(x1);
      fadd2(sum4[(e & 1) * 2], sum4[(e & 1) * 2 + 1], p0, p1);
      if constexpr (C::kTf32) {
        pk[2 * e] = to_tf32((kw >> (2 * e)) & 1u ? p0 : 0.0f);
        pk[2 * e + 1] = to_tf32((kw >> (2 * e + 1)) & 1u ? p1 : 0.0f);
      } else {
        // the pair's two keep bits widened to a 16-bit lane mask
        const uint32_t t = (kw >> (2 * e)) & 3u;
        pk[e] = pack16x2<C>(p0, p1) & ((t & 1u) * 0x0000FFFFu + (t >> 1) * 0xFFFF0000u);
      }
    }
    if constexpr (C::kTf32)
      tmem_st32(tP + cc * 32, pk);
    else
      tmem_st16(tP + cc * 16, pk);
  }
  sum = (sum4[0] + sum4[1]) + (sum4[2] + sum4[3]);
}

// One work unit: kNQT 128-row Q tiles of one batch: consecutive row tiles of one
// head, or (head pairs) the same rows of two heads that share a K/V head.
struct Unit {
  int b, h, kvh, q0, N;
  int ks;            // key range (split-KV; 0 otherwise)
  int th[2], tr[2];  // head and first row of Q tile t
  int j0;       // first KV tile of the unit (the tiles share one K/V stream from j0 to N)
  int nblk[2];  // one past each Q tile's last KV tile (0: the tile has no rows)
};

// The unit's first KV tile: a compile-time 0 without a sliding window or
// key ranges.
template <class C>
__device__ __forceinline__ int unit_j0(const Unit& w) {
  if constexpr (C::kFeat || C::kSplitKV)
    return w.j0;
  else
    return 0;
}

template <class C>
__device__ __forceinline__ Unit decode_unit(const FaParams& p, int u) {
  // Heavy causal query blocks first; consecutive units are consecutive heads
  // (or head pairs), so the H_q / H_kv heads sharing a K/V head run side by
  // side (L2 reuse).  With head pairs both tiles cover the same rows, so they
  // visit the same K/V blocks and finish together (a causal row pair would
  // leave the second tile one block alone at the end of every unit).
  Unit w;
  // Split-KV: the key ranges of a query block come next to each other in the
  // order, between the query block and the (batch, head) units.
  const int per_bh = p.B * p.hq_units;
  const int splits = C::kSplitKV ? p.kv_splits : 1;
  const int per_q = per_bh * splits;
  const int qb_rev = u / per_q;
  int rem = u - qb_rev * per_q;
  w.ks = 0;
  if constexpr (C::kSplitKV) {
    w.ks = rem / per_bh;
    rem -= w.ks * per_bh;
  }
  const int qb = p.causal ? (p.n_qblocks - 1 - qb_rev) : qb_rev;
  w.b = rem / p.hq_units;
  const int hu = rem - w.b * p.hq_units;
  w.h = p.head_pairs ? 2 * hu : hu;
  w.kvh = w.h / p.group;
  w.q0 = qb * (p.head_pairs ? C::kBM : C::kBM * C::kNQT);
  w.th[0] = w.h;
  w.th[1] = p.head_pairs ? w.h + 1 : w.h;
  w.tr[0] = w.q0;
  w.tr[1] = p.head_pairs ? w.q0 : w.q0 + C::kBM;
  w.nblk[0] = tile_kv_blocks<C>(p, w.tr[0]);
  w.nblk[1] = (C::kNQT == 2) ? tile_kv_blocks<C>(p, w.tr[1]) : 0;
  w.N = max(w.nblk[0], w.nblk[1]);
  // Tile 0's rows come first (or equal), so its window starts first; tile 1
  // masks the (at most one) leading block it cannot see.
  w.j0 = tile_kv_begin<C>(p, w.tr[0], w.nblk[0]);
  if constexpr (C::kSplitKV) {
    if (splits > 1) {  // key blocks [j0, nblk) of range ks; an empty range is a unit without work
      const int jb = w.ks * p.kv_chunk;
      const int je = min(w.nblk[0], jb + p.kv_chunk);
      w.j0 = jb;
      w.nblk[0] = je > jb ? je : 0;
      w.N = w.nblk[0];
    }
  }
  return w;
}

// The r-th unit of this CTA: a boustrophedon ("snake") walk over the
// heavy-first unit list, so each CTA's total work stays balanced; -1 when done.
__device__ __forceinline__ int unit_of(int r, int num_units) {
  const int G = gridDim.x, c = blockIdx.x;
  const int idx = r * G + ((r & 1) ? (G - 1 - c) : c);
  return idx < num_units ? idx : -1;
}

// tf32 helper warps (fp32 I/O): round each landed Q and K tile to tf32 in
// place and transpose each V tile into the K-major V^T ring, in the order the
// producer loads them.  ct is this thread's index among the helper threads.
template <class C>
__device__ __forceinline__ void tf32_helpers(uint8_t* sQ, uint8_t* sK, uint8_t* sV, uint8_t* sVT, Ctrl<C>* ctl,
                                             const FaParams& p, volatile int* abort_flag, int num_units, int ct,
                                             int lane) {
  int q_seen[2] = {0, 0};
  int k_seen = 0, v_seen = 0;
  bool ok = true;
  for (int r = 0; ok; ++r) {
    const int u = unit_of(r, num_units);
    if (u < 0) break;
    const Unit w = decode_unit<C>(p, u);
#pragma unroll
    for (int t = 0; t < C::kNQT; ++t) {
      if (!ok || w.nblk[t] == 0) continue;
      ok = warp_wait(&ctl->q_full[t], q_seen[t] & 1, abort_flag, p.status, p.timeout_cycles);
      ++q_seen[t];
      if (!ok) continue;
      round_tf32_inplace(sQ + t * C::kQTileBytes, C::kQTileBytes, ct, C::kCvtThreads);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl->q_ready[t]);
    }
    // Same order as the producer: K_j, then V_{j - kVLag}.
    for (int j = unit_j0<C>(w); j < w.N + C::kVLag && ok; ++j) {
      if (j < w.N) {
        const int slot = k_seen % C::kKStages;
        ok = warp_wait(&ctl->k_full[slot], (k_seen / C::kKStages) & 1, abort_flag, p.status, p.timeout_cycles);
        ++k_seen;
        if (!ok) break;
        round_tf32_inplace(sK + slot * C::kKVTileBytes, C::kKVTileBytes, ct, C::kCvtThreads);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&ctl->k_ready[slot]);
      }
      if (j < unit_j0<C>(w) + C::kVLag) continue;
      // V -> V^T (K-major), then hand the V slot back to the producer.
      const int vs = v_seen % C::kVStages, ts = v_seen % C::kVTStages;
      ok = warp_wait(&ctl->v_full[vs], (v_seen / C::kVStages) & 1, abort_flag, p.status, p.timeout_cycles);
      if (!ok) break;
      ok = warp_wait(&ctl->vt_empty[ts], ((v_seen / C::kVTStages) & 1) ^ 1, abort_flag, p.status,
                     p.timeout_cycles);
      ++v_seen;
      if (!ok) break;
      transpose_v_tile<C>(sV + vs * C::kKVTileBytes, sVT + ts * C::kKVTileBytes, ct, C::kCvtThreads);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&ctl->vt_full[ts]);
        mbar_arrive(&ctl->v_empty[vs]);
      }
    }
  }
}

// Softmax of a one-Q-tile plan on two warpgroups (kSplitRows): warpgroup g
// (warps 4 + 4 g .. 7 + 4 g) owns keys 64 g .. 64 g + 63 of every block for
// all 128 rows (thread = TMEM lane = row), and half of O's columns in the
// epilogue.  The two halves of a row share one running max: each block's half
// maxima are exchanged through the block's P buffer in TMEM (free at that
// point: the P V that last read it has completed), each warpgroup writing its
// value into a column of the OTHER half, which that half reads before
// overwriting it with its P; the row sums meet the same way in the epilogue.
//
// Sync supplies the schedule and the hand-offs: next(r, b, h, r0, j0, nb, ks)
// (the r-th unit: batch, head, this CTA's first row, key blocks [j0, nb), key
// range ks; false when done), wait_s / wait_m / wait_o (bounded waits on S landed, the mask tile
// landed, P V landed) and the arrivals s_free / m_free / p_ready / o_free.
template <class C, class Sync>
__device__ __forceinline__ void softmax_split_rows(Sync& sy, uint8_t* sM, uint32_t tmem, const FaParams& p, int warp,
                                                   int lane) {
  constexpr int kHalf = C::kBN / 2;                 // keys per warpgroup
  constexpr int kHalfD = C::kD / 2;                 // O columns per warpgroup in the epilogue
  const int g = (warp - 4) >> 2;                    // 0: keys 0..63, 1: keys 64..127
  const int tl = threadIdx.x - 128 * (1 + g);       // row of the tile
  const uint32_t lane_addr = (uint32_t)((warp & 3) * 32) << 16;
  const uint32_t tS = tmem + lane_addr + g * kHalf;
  const uint32_t tO = tmem + lane_addr + C::kColO;
  const float sl = p.pre_scale ? 1.0f : p.scale_log2;
  // TMEM column (relative to a P buffer) this warpgroup writes for the other
  // half to read, and the one it reads: column 0 lies in half 0's P, column
  // kHalf / 2 in half 1's.
  const uint32_t x_put = g == 0 ? kHalf / 2 : 0, x_get = g == 0 ? 0 : kHalf / 2;
  int blocks_seen = 0, masks_seen = 0;
  bool ok = true;
  for (int r = 0; ok; ++r) {
    int b, h, r0, j0, nb, ks;
    if (!sy.next(r, b, h, r0, j0, nb, ks)) break;
    if (nb == 0) continue;
    const int row = r0 + tl;
    float m_run = -INFINITY;  // running max of the whole row, base 2 (scaled)
    float l_run = 0.0f;       // this half's running sum of 2^(s - m_run)
    for (int j = j0; j < nb; ++j) {
      ok = sy.wait_s(blocks_seen & 1);
      if (!ok) break;
      ++blocks_seen;
      tc_fence_after();
      float s[kHalf];
      {
        uint32_t rr[kHalf];
#pragma unroll
        for (int cc = 0; cc < kHalf / 32; ++cc)
          tmem_ld32(tS + cc * 32, *reinterpret_cast<uint32_t(*)[32]>(&rr[cc * 32]));
        tmem_wait_ld();
        reg_fence(rr);
#pragma unroll
        for (int c = 0; c < kHalf; ++c) s[c] = __uint_as_float(rr[c]);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) sy.s_free();

      const int kbase = j * C::kBN + g * kHalf;  // this half's first key
      const int q_off = C::kFeat ? p.q_offset : 0;
      const bool need_mask = p.pre_scale || p.mask_kind != 0 || kbase + kHalf > p.kL ||
                             (p.causal && kbase + kHalf - 1 > r0 + q_off) ||
                             (C::kFeat && p.window > 0 && kbase <= r0 + C::kBM - 1 + q_off - p.window);
      const uint8_t* mask_tile = nullptr;
      if (C::kMaskSlotBytes > 0 && p.mask_smem) {
        ok = sy.wait_m(masks_seen & 1);
        ++masks_seen;
        if (!ok) break;
        mask_tile = sM;
      }
      if (need_mask) apply_mask<C, kHalf>(s, p, b, h, row, kbase, mask_tile, tl, g * kHalf);
      if (mask_tile) {
        __syncwarp();
        if (lane == 0) sy.m_free();
      }

      // The row's block max from both halves.
      const uint32_t tP = tmem + lane_addr + C::kColP + (j & 1) * C::kPCols;
      const float mx_half = row_max<C, kHalf>(s);
      tmem_st1(tP + x_put, __float_as_uint(mx_half));
      tmem_wait_st();
      tc_fence_before();
      named_bar_sync(1, 256);
      tc_fence_after();
      const float mx_other = __uint_as_float(tmem_ld1(tP + x_get));
      tmem_wait_ld();
      const float mx = fmaxf(mx_half, mx_other);

      const float m_blk = mx * sl;  // -inf stays -inf (sl > 0 whenever it is not 1)
      const float m_new = fmaxf(m_run, m_blk);
      float corr = 1.0f;
      const bool resc = m_new > m_run + kRescaleThreshold;
      if (resc) {
        corr = ex2(m_run - m_new);  // 0 when m_run = -inf
        m_run = m_new;
      }
      const float msub = (m_run == -INFINITY) ? 0.0f : m_run;
      float sum, unused;
      p_pass<C, false, kHalf>(s, sl, msub, tP + g * (kHalf / 2), sum, unused);
      l_run = l_run * corr + sum;

      // PV_{j-1} has landed before this half's O columns are rescaled.
      if (j > j0) {
        ok = sy.wait_o((blocks_seen - 2) & 1);
        if (!ok) break;
      }
      if (j > j0 && __any_sync(0xffffffffu, resc)) {
        tc_fence_after();
#pragma unroll
        for (int cc = 0; cc < kHalfD / 32; ++cc) {
          uint32_t rr[32];
          tmem_ld32(tO + g * kHalfD + cc * 32, rr);
          tmem_wait_ld();
          reg_fence(rr);
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            float o0, o1;
            fmul2(o0, o1, __uint_as_float(rr[e]), __uint_as_float(rr[e + 1]), corr, corr);
            rr[e] = __float_as_uint(o0);
            rr[e + 1] = __float_as_uint(o1);
          }
          tmem_st32(tO + g * kHalfD + cc * 32, rr);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) sy.p_ready();
    }
    if (!ok) break;

    // ---- epilogue: this half's O columns / l -> I/O dtype -> global; L by half 0.
    ok = sy.wait_o((blocks_seen - 1) & 1);
    if (!ok) break;
    tc_fence_after();
    {  // the row sum of both halves (both P buffers are free: the last P V has completed)
      const uint32_t tX = tmem + lane_addr + C::kColP;
      tmem_st1(tX + x_put, __float_as_uint(l_run));
      tmem_wait_st();
      tc_fence_before();
      named_bar_sync(1, 256);
      tc_fence_after();
      l_run += __uint_as_float(tmem_ld1(tX + x_get));
      tmem_wait_ld();
      // the next unit's first exchange may write these columns only after both halves read them
      tc_fence_before();
      named_bar_sync(1, 256);
      tc_fence_after();
    }
    const float inv_l = (l_run > 0.0f) ? 1.0f / l_run : 0.0f;
    const bool store = row < p.qL;
    uint8_t* orow = static_cast<uint8_t*>(p.o) +
                    ((long long)b * p.o_sb + (long long)h * p.o_sh + (long long)(store ? row : 0) * p.o_ss) * C::kEsz +
                    g * kHalfD * C::kEsz;
    // Split-KV: this range's normalised O (fp32) and logsumexp go to the
    // partial buffers, row ((ks * B + b) * H_q + h) * qL + row.
    const bool part = C::kSplitKV && p.kv_splits > 1;
    const long long prow = (((long long)ks * p.B + b) * p.Hq + h) * p.qL + (store ? row : 0);
    constexpr int kBatch = kHalfD / 32 < 4 ? kHalfD / 32 : 4;
#pragma unroll
    for (int c0 = 0; c0 < kHalfD / 32; c0 += kBatch) {
      uint32_t rb[kBatch][32];
#pragma unroll
      for (int i = 0; i < kBatch; ++i) tmem_ld32(tO + g * kHalfD + (c0 + i) * 32, rb[i]);
      tmem_wait_ld();
#pragma unroll
      for (int i = 0; i < kBatch; ++i) reg_fence(rb[i]);
      if (c0 + kBatch == kHalfD / 32) {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) sy.o_free();
      }
      if (store && part) {
#pragma unroll
        for (int i = 0; i < kBatch; ++i) {
          uint4* dst = reinterpret_cast<uint4*>(p.part_o + prow * C::kD + g * kHalfD + (c0 + i) * 32);
#pragma unroll
          for (int u4 = 0; u4 < 8; ++u4) {
            float a0, a1, a2, a3;
            fmul2(a0, a1, __uint_as_float(rb[i][4 * u4]), __uint_as_float(rb[i][4 * u4 + 1]), inv_l, inv_l);
            fmul2(a2, a3, __uint_as_float(rb[i][4 * u4 + 2]), __uint_as_float(rb[i][4 * u4 + 3]), inv_l, inv_l);
            dst[u4] = make_uint4(__float_as_uint(a0), __float_as_uint(a1), __float_as_uint(a2), __float_as_uint(a3));
          }
        }
      } else if (store) {
#pragma unroll
        for (int i = 0; i < kBatch; ++i) {
          uint4* dst = reinterpret_cast<uint4*>(orow + (c0 + i) * 64);
#pragma unroll
          for (int u4 = 0; u4 < 4; ++u4) {
            uint32_t pk[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              float a0, a1;
              fmul2(a0, a1, __uint_as_float(rb[i][8 * u4 + 2 * e]), __uint_as_float(rb[i][8 * u4 + 2 * e + 1]),
                    inv_l, inv_l);
              pk[e] = pack16x2<C>(a0, a1);
            }
            dst[u4] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
          }
        }
      }
    }
    if (store && g == 0) {
      const float lse = (l_run > 0.0f) ? (m_run + lg2(l_run)) * kLn2 : -INFINITY;
      if (part)
        p.part_lse[prow] = lse;
      else
        p.lse[((long long)b * p.Hq + h) * p.qL + row] = lse;
    }
  }
}

// The one-CTA plans' hand-offs for softmax_split_rows.
template <class C>
struct LocalSync {
  Ctrl<C>* ctl;
  const FaParams& p;
  volatile int* abort;
  int num_units;
  __device__ bool next(int r, int& b, int& h, int& r0, int& j0, int& nb, int& ks) {
    const int u = unit_of(r, num_units);
    if (u < 0) return false;
    const Unit w = decode_unit<C>(p, u);
    b = w.b;
    h = w.th[0];
    r0 = w.tr[0];
    j0 = unit_j0<C>(w);
    nb = w.nblk[0];
    ks = w.ks;
    return true;
  }
  __device__ bool wait_s(uint32_t par) { return warp_wait(&ctl->s_full[0], par, abort, p.status, p.timeout_cycles); }
  __device__ bool wait_m(uint32_t par) { return warp_wait(&ctl->m_full, par, abort, p.status, p.timeout_cycles); }
  __device__ bool wait_o(uint32_t par) { return warp_wait(&ctl->o_ready[0], par, abort, p.status, p.timeout_cycles); }
  __device__ void s_free() { mbar_arrive(&ctl->s_free[0]); }
  __device__ void m_free() { mbar_arrive(&ctl->m_empty); }
  __device__ void p_ready() { mbar_arrive(&ctl->p_ready[0]); }
  __device__ void o_free() { mbar_arrive(&ctl->o_free[0]); }
};

// Split-KV combine pass: for each row, over the key ranges that ran a unit
// for the row's query tile (a range starting past the tile's last key block
// ran none), O = sum_s w_s O_s / sum_s w_s with w_s = exp(lse_s - max_s lse_s)
// and L = max_s lse_s + log(sum_s w_s) -- the softmax of the union of the
// ranges, since each O_s is its range's normalised output and lse_s its
// logsumexp.  A row none of whose ranges saw a key keeps O = 0, L = -inf.
// D / 8 threads per row, 8 columns each.
template <class C>
__global__ void __launch_bounds__(256) fa_splitkv_combine_kernel(const FaParams p) {
  constexpr int kT = C::kD / 8;
  const long long t = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const long long plane = (long long)p.B * p.Hq * p.qL;  // rows of one range
  if (t >= plane * kT) return;
  const long long row = t / kT;  // ((b * H_q + h) * qL + i)
  const int c8 = (int)(t - row * kT);
  const long long bh = row / p.qL;
  const int i = (int)(row - bh * p.qL);
  const int b = (int)(bh / p.Hq), h = (int)(bh - (long long)b * p.Hq);
  const int last = min((i / C::kBM) * C::kBM + C::kBM, p.qL) - 1;
  const int kv_end = p.causal ? min(p.kL, last + 1) : p.kL;
  const int nb = (kv_end + C::kBN - 1) / C::kBN;  // the tile's key blocks
  float m = -INFINITY;
  for (int s = 0; s < p.kv_splits && s * p.kv_chunk < nb; ++s) m = fmaxf(m, p.part_lse[s * plane + row]);
  float acc[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) acc[e] = 0.0f;
  float sum = 0.0f;
  if (m != -INFINITY) {
    for (int s = 0; s < p.kv_splits && s * p.kv_chunk < nb; ++s) {
      const float w = expf(p.part_lse[s * plane + row] - m);  // 0 for a range without keys for the row
      const float4* src = reinterpret_cast<const float4*>(p.part_o + (s * plane + row) * C::kD + c8 * 8);
      const float4 x0 = src[0], x1 = src[1];
      sum += w;
      acc[0] = fmaf(w, x0.x, acc[0]);
      acc[1] = fmaf(w, x0.y, acc[1]);
      acc[2] = fmaf(w, x0.z, acc[2]);
      acc[3] = fmaf(w, x0.w, acc[3]);
      acc[4] = fmaf(w, x1.x, acc[4]);
      acc[5] = fmaf(w, x1.y, acc[5]);
      acc[6] = fmaf(w, x1.z, acc[6]);
      acc[7] = fmaf(w, x1.w, acc[7]);
    }
  }
  const float inv = sum > 0.0f ? 1.0f / sum : 0.0f;
  uint8_t* dst = static_cast<uint8_t*>(p.o) +
                 ((long long)b * p.o_sb + (long long)h * p.o_sh + (long long)i * p.o_ss + c8 * 8) * C::kEsz;
  *reinterpret_cast<uint4*>(dst) = make_uint4(pack16x2<C>(acc[0] * inv, acc[1] * inv), pack16x2<C>(acc[2] * inv, acc[3] * inv),
                                              pack16x2<C>(acc[4] * inv, acc[5] * inv), pack16x2<C>(acc[6] * inv, acc[7] * inv));
  if (c8 == 0) p.lse[row] = sum > 0.0f ? m + logf(sum) : -INFINITY;
}

// Persistent forward kernel: each CTA walks its units; every role carries its
// barrier phase counters from one unit to the next, so the next unit's Q and
// K/V loads and its first S MMAs overlap the current unit's last blocks and
// epilogue.
template <class C>
__global__ void __launch_bounds__(C::kThreads, 1)
    fa_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmM,
                  const __grid_constant__ CUtensorMap tmO, const FaParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem;
  uint8_t* sK = smem + C::kOffK;
  uint8_t* sV = smem + C::kOffV;
  uint8_t* sVT = smem + C::kOffVT;
  uint8_t* sM = smem + C::kOffM;
  Ctrl<C>* ctl = reinterpret_cast<Ctrl<C>*>(smem + C::kOffBar);
  volatile int* abort_flag = &ctl->abort;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int num_units = p.n_qblocks * p.B * p.hq_units * p.kv_splits;

  if (threadIdx.x == 0) {
    for (int t = 0; t < 2; ++t) {
      mbar_init(&ctl->q_full[t], 1);
      mbar_init(&ctl->q_empty[t], 1);    // MMA commit after the unit's last S of tile t
      mbar_init(&ctl->q_ready[t], C::kCvtWarps);  // one arrival per tf32 helper warp
      mbar_init(&ctl->s_full[t], 1);
      mbar_init(&ctl->s_free[t], C::kSplitRows ? 8 : 4);   // one arrival per softmax warp
      mbar_init(&ctl->p_ready[t], C::kSplitRows ? 8 : 4);  // one arrival per softmax warp
      mbar_init(&ctl->o_ready[t], 1);
      mbar_init(&ctl->o_free[t], C::kSplitRows ? 8 : 4);   // one arrival per softmax warp after reading O
    }
    for (int s = 0; s < 4; ++s) {
      mbar_init(&ctl->k_full[s], 1);
      mbar_init(&ctl->k_empty[s], C::kIssuers);  // one commit per issuing thread
      mbar_init(&ctl->k_ready[s], C::kCvtWarps);
      mbar_init(&ctl->v_full[s], 1);
      mbar_init(&ctl->v_empty[s], C::kHelpers ? C::kCvtWarps : C::kIssuers);  // tf32: released by the helper warps
      mbar_init(&ctl->vt_full[s], C::kCvtWarps);
      mbar_init(&ctl->vt_empty[s], C::kIssuers);
    }
    mbar_init(&ctl->drain[0], 1);
    mbar_init(&ctl->drain[1], 1);
    mbar_init(&ctl->m_full, 1);
    mbar_init(&ctl->m_empty, C::kSplitRows ? 8 : 4);  // one arrival per softmax warp
    ctl->abort = 0;
    mbar_init(&ctl->turn_bar[0], 1);
    mbar_init(&ctl->turn_bar[1], 1);
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    if (p.mask_l2 || p.mask_smem) tma_prefetch_desc(&tmM);
  }
  if (warp == 1) {
    tmem_alloc(&ctl->tmem_base, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl->tmem_base;

  if (warp < 4) {
  // Control warpgroup: TMA producer, MMA issuer, tf32 helpers.
  if constexpr (C::kRegsSoftmax > 0) regs_dec<C::kRegsCtrl>();
  if (warp == 0) {
    // ===================================================== TMA producer
    if (lane == 0) {
      int k_issued = 0, v_issued = 0;  // ring items issued (all units)
      int m_issued = 0;                // mask tiles issued (shared-memory mask path)
      int q_issued[2] = {0, 0};        // Q loads issued per tile
      bool ok = true;
      for (int r = 0; ok; ++r) {
        const int u = unit_of(r, num_units);
        if (u < 0) break;
        const Unit w = decode_unit<C>(p, u);
#pragma unroll
        for (int t = 0; t < C::kNQT; ++t) {
          if (!ok || w.nblk[t] == 0) continue;
          // Q_t's shared memory is free once the previous unit's last S_t completed.
          if (q_issued[t] > 0)
            ok = wait_bounded(&ctl->q_empty[t], (q_issued[t] - 1) & 1, abort_flag, p.status, p.timeout_cycles);
          if (!ok) continue;
          mbar_arrive_expect_tx(&ctl->q_full[t], C::kQTileBytes);
#pragma unroll
          for (int c = 0; c < C::kNChunk; ++c)
            tma_load_4d(sQ + t * C::kQTileBytes + c * (C::kBM * 128), &tmQ, &ctl->q_full[t], c * C::kChunk,
                        t == 0 ? w.tr[0] : w.tr[1], t == 0 ? w.th[0] : w.th[1], w.b);
          ++q_issued[t];
        }
        // Mask tiles reach L2 two blocks ahead of their use (read by the
        // softmax from L2, or by the shared-memory mask load): block j + 2
        // while K_j is issued, reaching into the next unit near the end of this
        // one; a CTA's first unit prefetches its blocks 0 and 1 up front.
        const bool pf_mask = p.mask_l2 || p.mask_smem;
        auto prefetch_mask = [&](const Unit& uu, int j) {
          const int mesz = p.mask_kind == 1 ? 1 : C::kEsz;
#pragma unroll
          for (int t = 0; t < C::kNQT; ++t)
            for (int c = 0; c < (C::kBN * mesz) / 128; ++c)
              tma_prefetch_l2_4d(&tmM, j * C::kBN + c * (128 / mesz), t == 0 ? uu.tr[0] : uu.tr[1],
                                 t == 0 ? uu.th[0] : uu.th[1], uu.b);
        };
        const int u_next = unit_of(r + 1, num_units);
        const Unit w_next = decode_unit<C>(p, u_next < 0 ? u : u_next);
        if (pf_mask && r == 0) {
          for (int j = unit_j0<C>(w); j < min(unit_j0<C>(w) + 2, w.N); ++j) prefetch_mask(w, j);
        }
        for (int j = unit_j0<C>(w); j < w.N + C::kVLag && ok; ++j) {
          if (j < w.N) {
          if (pf_mask) {
            if (j + 2 < w.N)
              prefetch_mask(w, j + 2);
            else if (u_next >= 0 && unit_j0<C>(w_next) + j + 2 - w.N < w_next.N)
              prefetch_mask(w_next, unit_j0<C>(w_next) + j + 2 - w.N);
          }
          {  // K_j
            const int slot = k_issued % C::kKStages, use = k_issued / C::kKStages;
            ok = wait_bounded(&ctl->k_empty[slot], (use & 1) ^ 1, abort_flag, p.status, p.timeout_cycles);
            if (!ok) break;
            mbar_arrive_expect_tx(&ctl->k_full[slot], C::kKVTileBytes);
            uint8_t* dst = sK + slot * C::kKVTileBytes;
#pragma unroll
            for (int c = 0; c < C::kNChunk; ++c)
              tma_load_4d(dst + c * (C::kBN * 128), &tmK, &ctl->k_full[slot], c * C::kChunk, j * C::kBN, w.kvh,
                          w.b);
            ++k_issued;
          }
          if (C::kMaskSlotBytes > 0 && p.mask_smem) {  // M_j: the mask tile of block j
            ok = wait_bounded(&ctl->m_empty, (m_issued & 1) ^ 1, abort_flag, p.status, p.timeout_cycles);
            if (!ok) break;
            const int mesz = p.mask_kind == 1 ? 1 : 2;
            const int boxes = (C::kBN * mesz) / 128;  // 128-byte column blocks
            mbar_arrive_expect_tx(&ctl->m_full, (uint32_t)(C::kBM * C::kBN * mesz));
            for (int c = 0; c < boxes; ++c)
              tma_load_4d(sM + c * (C::kBM * 128), &tmM, &ctl->m_full, j * C::kBN + c * (128 / mesz), w.tr[0], w.th[0],
                          w.b);
            ++m_issued;
          }
          }
          const int jv = j - C::kVLag;
          if (jv >= unit_j0<C>(w)) {  // V_jv
            const int slot = v_issued % C::kVStages, use = v_issued / C::kVStages;
            ok = wait_bounded(&ctl->v_empty[slot], (use & 1) ^ 1, abort_flag, p.status, p.timeout_cycles);
            if (!ok) break;
            mbar_arrive_expect_tx(&ctl->v_full[slot], C::kKVTileBytes);
            uint8_t* dst = sV + slot * C::kKVTileBytes;
            if constexpr (C::kPre) {
              // V^T [.., D, keys]: 32-key column blocks of D rows (K-major B of O += P V)
#pragma unroll
              for (int c = 0; c < C::kBN / 32; ++c)
                tma_load_4d(dst + c * (C::kD * 128), &tmV, &ctl->v_full[slot], jv * C::kBN + c * 32, 0, w.kvh, w.b);
            } else {
#pragma unroll
              for (int c = 0; c < C::kNChunk; ++c)
                tma_load_4d(dst + c * (C::kBN * 128), &tmV, &ctl->v_full[slot], c * C::kChunk, jv * C::kBN, w.kvh,
                            w.b);
            }
            ++v_issued;
          }
        }
      }
      if (*abort_flag) {
        // Let every copy this thread started land before the CTA lets go of its memory.
        for (int t = 0; t < 2; ++t)
          if (q_issued[t] > 0)
            wait_bounded(&ctl->q_full[t], (q_issued[t] - 1) & 1, abort_flag, p.status, kDrainCycles, false);
        for (int it = max(0, k_issued - C::kKStages); it < k_issued; ++it)
          wait_bounded(&ctl->k_full[it % C::kKStages], (it / C::kKStages) & 1, abort_flag, p.status,
                       kDrainCycles, false);
        for (int it = max(0, v_issued - C::kVStages); it < v_issued; ++it)
          wait_bounded(&ctl->v_full[it % C::kVStages], (it / C::kVStages) & 1, abort_flag, p.status,
                       kDrainCycles, false);
        if (m_issued > 0) wait_bounded(&ctl->m_full, (m_issued - 1) & 1, abort_flag, p.status, kDrainCycles, false);
      }
    }
  } else if (warp == 1 || (C::kIssuers == 2 && warp == 2)) {
    // ===================================================== MMA issuer(s)
    // Issuer i handles Q tiles [t_begin, t_end).  Every issuer walks all
    // units and all K/V tiles in order and commits its own arrival on each
    // release barrier, so each release phase sees exactly kIssuers arrivals.
    const int issuer = warp - 1;
    const int t_begin = C::kIssuers == 1 ? 0 : issuer;
    const int t_end = C::kIssuers == 1 ? C::kNQT : issuer + 1;
    if (lane == 0) {
      constexpr uint32_t idS = make_idesc_fmt(C::kFmt, 128, C::kBN, false, false);
      constexpr uint32_t idPV = make_idesc_fmt(C::kFmt, 128, C::kD, false, !C::kTf32);
      // Descriptor halves of the first K-step of each operand ring; later
      // K-steps and slots only add to the start address in the low half.
      const uint64_t dQ = make_sdesc_sw128(smem_u32(sQ), 16, 1024);
      const uint64_t dK = make_sdesc_sw128(smem_u32(sK), 16, 1024);
      // tf32: V^T tile, rows = D (the MMA's N), keys along the 128-byte rows (K-major).
      // bf16: V tile, rows = keys (the MMA's K), 128 bytes of D per row; D column
      // blocks are kBN*128 bytes apart (LBO), 8-key groups 1024 apart (SBO).
      const uint64_t dV = C::kTf32 ? make_sdesc_sw128(smem_u32(C::kHelpers ? sVT : sV), 16, 1024)
                                   : make_sdesc_sw128(smem_u32(sV), C::kBN * 128, 1024);
      const uint32_t q_lo = (uint32_t)dQ, q_hi = (uint32_t)(dQ >> 32);
      const uint32_t k_lo = (uint32_t)dK, k_hi = (uint32_t)(dK >> 32);
      const uint32_t v_lo = (uint32_t)dV, v_hi = (uint32_t)(dV >> 32);

      auto issue_S = [&](int t, int kslot) {
        const uint32_t qa = q_lo + ((t * C::kQTileBytes) >> 4);
        const uint32_t ka = k_lo + ((kslot * C::kKVTileBytes) >> 4);
        const uint32_t dst = tmem + t * C::kBN;
        mma_ss_lh<C::kTf32, 0>(dst, qa, q_hi, ka, k_hi, idS, 0u);
#pragma unroll
        for (int kk = 1; kk < C::kD / C::kKStep; ++kk) {
          // 4 MMA K-steps of 32 bytes per 128-byte swizzle row, then the next column block
          constexpr int kQCol = (C::kBM * 128) >> 4, kKCol = (C::kBN * 128) >> 4;
          mma_ss_lh<C::kTf32, 1>(dst, qa + (kk / 4) * kQCol + (kk % 4) * 2, q_hi, ka + (kk / 4) * kKCol + (kk % 4) * 2,
                                 k_hi, idS, 1u);
        }
      };
      auto issue_PV = [&](int t, int j, int vslot, bool first) {
        const uint32_t pcol = C::kAliasP ? (uint32_t)(t * C::kBN) : (uint32_t)(C::kColP + (j & 1) * C::kPCols);
        const uint32_t va = v_lo + ((vslot * C::kKVTileBytes) >> 4);
        const uint32_t dst = tmem + C::kColO + t * C::kD;
        const uint32_t src = tmem + pcol;
        mma_ts_lh<C::kTf32, 0>(dst, src, va, v_hi, idPV, first ? 0u : 1u);
#pragma unroll
        for (int kk = 1; kk < C::kBN / C::kKStep; ++kk) {
          const uint32_t voff = C::kTf32 ? ((kk / 4) * (C::kD * 128) + (kk % 4) * 32) >> 4 : (kk * (C::kKStep * 128)) >> 4;
          mma_ts_lh<C::kTf32, 1>(dst, src + kk * 8, va + voff, v_hi, idPV, 1u);
        }
      };
      // Two issuers take turns, group by group: issuer 0's group g follows
      // issuer 1's group g - 1, and issuer 1's group g follows issuer 0's group
      // g.  Each hand-off is an mbarrier arrival, so the waiting thread sleeps
      // in try_wait instead of polling next to the softmax warps.
      int groups = 0;  // MMA groups this issuer has issued
      auto wait_turn = [&]() -> bool {
        if (C::kIssuers == 1 || (issuer == 0 && groups == 0)) return true;
        const int phase = issuer == 0 ? groups - 1 : groups;
        return wait_bounded(&ctl->turn_bar[issuer], phase & 1, abort_flag, p.status, p.timeout_cycles);
      };
      auto pass_turn = [&]() {
        if (C::kIssuers == 2) {
          mbar_arrive(&ctl->turn_bar[1 - issuer]);
          ++groups;
        }
      };

      int k_used = 0, v_used = 0;   // ring items consumed (all units)
      int q_used[2] = {0, 0};       // Q loads consumed per tile
      int p_seen[2] = {0, 0};       // p_ready phases consumed per tile
      int units_done[2] = {0, 0};   // units with a non-empty tile t (o_free phases to wait)
      int s_freed = 0;              // s_free phases consumed (one Q tile)
      bool ok = true;
      for (int r = 0; ok; ++r) {
        const int u = unit_of(r, num_units);
        if (u < 0) break;
        const Unit w = decode_unit<C>(p, u);
        if (w.N == 0) continue;  // an empty key range (split-KV): the producer loads nothing for it
#pragma unroll
        for (int t = 0; t < C::kNQT; ++t) {
          if (t < t_begin || t >= t_end || !ok || w.nblk[t] == 0) continue;
          const uint32_t par = q_used[t] & 1;
          ok = C::kHelpers ? wait_bounded(&ctl->q_ready[t], par, abort_flag, p.status, p.timeout_cycles)
                        : wait_bounded(&ctl->q_full[t], par, abort_flag, p.status, p.timeout_cycles);
          ++q_used[t];
        }
        // K_0 -> S_t,0 for every tile of this issuer
        int kslot = k_used % C::kKStages;
        if (ok) {
          const uint32_t par = (k_used / C::kKStages) & 1;
          ok = C::kHelpers ? wait_bounded(&ctl->k_ready[kslot], par, abort_flag, p.status, p.timeout_cycles)
                        : wait_bounded(&ctl->k_full[kslot], par, abort_flag, p.status, p.timeout_cycles);
        }
        if (ok) ok = wait_turn();
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int t = 0; t < C::kNQT; ++t) {
          if (t < t_begin || t >= t_end || w.nblk[t] == 0) continue;
          issue_S(t, kslot);
          mma_commit(&ctl->s_full[t]);
          if (w.nblk[t] == unit_j0<C>(w) + 1) mma_commit(&ctl->q_empty[t]);  // the unit's last S of tile t
        }
        pass_turn();
        mma_commit(&ctl->k_empty[kslot]);
        ++k_used;
        if constexpr (!C::kAliasP) {
          // One Q tile, one issuer, separate S and P columns: S_{j+1} goes to the
          // tensor core as soon as softmax j holds S_j in registers (and K_{j+1}
          // is ready), so it overlaps softmax j; PV_j follows once P_j is written.
          for (int j = unit_j0<C>(w); j < w.N && ok; ++j) {
            ok = wait_bounded(&ctl->s_free[0], s_freed & 1, abort_flag, p.status, p.timeout_cycles);
            ++s_freed;
            if (!ok) break;
            if (j + 1 < w.N) {
              kslot = k_used % C::kKStages;
              const uint32_t par = (k_used / C::kKStages) & 1;
              ok = C::kHelpers ? wait_bounded(&ctl->k_ready[kslot], par, abort_flag, p.status, p.timeout_cycles)
                            : wait_bounded(&ctl->k_full[kslot], par, abort_flag, p.status, p.timeout_cycles);
              if (!ok) break;
              tc_fence_after();
              issue_S(0, kslot);
              mma_commit(&ctl->s_full[0]);
              if (j + 2 == w.N) mma_commit(&ctl->q_empty[0]);  // the unit's last S
              mma_commit(&ctl->k_empty[kslot]);
              ++k_used;
            }
            const int vslot = C::kHelpers ? v_used % C::kVTStages : v_used % C::kVStages;
            const uint32_t vpar = (C::kHelpers ? v_used / C::kVTStages : v_used / C::kVStages) & 1;
            ok = C::kHelpers ? wait_bounded(&ctl->vt_full[vslot], vpar, abort_flag, p.status, p.timeout_cycles)
                          : wait_bounded(&ctl->v_full[vslot], vpar, abort_flag, p.status, p.timeout_cycles);
            if (!ok) break;
            ok = wait_bounded(&ctl->p_ready[0], p_seen[0] & 1, abort_flag, p.status, p.timeout_cycles);
            ++p_seen[0];
            // The unit's first PV overwrites O: the previous unit's epilogue must have read it.
            if (ok && j == unit_j0<C>(w) && units_done[0] > 0)
              ok = wait_bounded(&ctl->o_free[0], (units_done[0] - 1) & 1, abort_flag, p.status, p.timeout_cycles);
            if (!ok) break;
            tc_fence_after();
            issue_PV(0, j, vslot, j == unit_j0<C>(w));
            mma_commit(&ctl->o_ready[0]);
            mma_commit(C::kHelpers ? &ctl->vt_empty[vslot] : &ctl->v_empty[vslot]);
            ++v_used;
          }
        } else
        // P over S (two Q tiles): per block and tile, PV_j then S_{j+1}.
        for (int j = unit_j0<C>(w); j < w.N && ok; ++j) {
          // bf16: V ring slot; tf32: V^T ring slot
          const int vslot = C::kHelpers ? v_used % C::kVTStages : v_used % C::kVStages;
          const uint32_t vpar = (C::kHelpers ? v_used / C::kVTStages : v_used / C::kVStages) & 1;
          ok = C::kHelpers ? wait_bounded(&ctl->vt_full[vslot], vpar, abort_flag, p.status, p.timeout_cycles)
                        : wait_bounded(&ctl->v_full[vslot], vpar, abort_flag, p.status, p.timeout_cycles);
          if (!ok) break;
          const bool next = (j + 1 < w.N);
          kslot = k_used % C::kKStages;
          bool k_waited = false;
          auto wait_k = [&]() -> bool {
            if (k_waited) return true;
            k_waited = true;
            const uint32_t par = (k_used / C::kKStages) & 1;
            return C::kHelpers ? wait_bounded(&ctl->k_ready[kslot], par, abort_flag, p.status, p.timeout_cycles)
                            : wait_bounded(&ctl->k_full[kslot], par, abort_flag, p.status, p.timeout_cycles);
          };
          bool turn_taken = false;
#pragma unroll
          for (int t = 0; t < C::kNQT; ++t) {
            if (t < t_begin || t >= t_end || !ok || j >= w.nblk[t]) continue;
            ok = wait_bounded(&ctl->p_ready[t], p_seen[t] & 1, abort_flag, p.status, p.timeout_cycles);
            ++p_seen[t];
            // The unit's first PV overwrites O_t: the previous unit's epilogue must have read it.
            if (ok && j == unit_j0<C>(w) && units_done[t] > 0)
              ok = wait_bounded(&ctl->o_free[t], (units_done[t] - 1) & 1, abort_flag, p.status, p.timeout_cycles);
            if (!ok) break;
            const bool s_next = (j + 1 < w.nblk[t]);
            const bool s_last = (j + 2 == w.nblk[t]);  // S_{t,j+1} is the unit's last S of tile t
            if (s_next) {
              ok = wait_k();
              if (!ok) break;
            }
            if (!turn_taken) {
              ok = wait_turn();
              if (!ok) break;
              turn_taken = true;
            }
            tc_fence_after();
            issue_PV(t, j, vslot, j == unit_j0<C>(w));
            if (!s_next) mma_commit(&ctl->o_ready[t]);  // the tile's last PV of the unit
            if (s_next) {
              issue_S(t, kslot);
              mma_commit(&ctl->s_full[t]);
              if (s_last) mma_commit(&ctl->q_empty[t]);
            }
          }
          if (!ok) break;
          if (!turn_taken) {  // an empty group still takes its turn
            ok = wait_turn();
            if (!ok) break;
          }
          pass_turn();
          mma_commit(C::kHelpers ? &ctl->vt_empty[vslot] : &ctl->v_empty[vslot]);
          ++v_used;
          if (next) {
            // Tiles that stop earlier (causal) never waited on K_{j+1}; make sure
            // it landed before this issuer's release of its slot.
            ok = wait_k();
            if (!ok) break;
            mma_commit(&ctl->k_empty[kslot]);
            ++k_used;
          }
        }
#pragma unroll
        for (int t = 0; t < C::kNQT; ++t)
          if (t >= t_begin && t < t_end && w.nblk[t] > 0) ++units_done[t];
      }
      // Drain: every MMA this thread issued completes before TMEM is freed.
      mma_commit(&ctl->drain[issuer]);
      wait_bounded(&ctl->drain[issuer], 0, abort_flag, p.status, kDrainCycles, false);
    }
    __syncwarp();
  } else {
    // ===================================================== tf32 helpers (fp32 I/O only)
    if constexpr (C::kHelpers) tf32_helpers<C>(sQ, sK, sV, sVT, ctl, p, abort_flag, num_units, threadIdx.x - 64, lane);
  }
  } else if (C::kExtraHelpers && warp >= 8) {
    // ===================================================== more tf32 helpers (one Q tile)
    if constexpr (C::kExtraHelpers)
      tf32_helpers<C>(sQ, sK, sV, sVT, ctl, p, abort_flag, num_units, 64 + (threadIdx.x - 256), lane);
  } else if (C::kSplitRows) {
    // ===================================================== two softmax warpgroups of one Q tile
    if constexpr (C::kSplitRows) {
      regs_inc<C::kRegsSoftmax>();
      LocalSync<C> sy{ctl, p, abort_flag, num_units};
      softmax_split_rows<C>(sy, sM, tmem, p, warp, lane);
    }
  } else {
    // ===================================================== softmax warpgroup t
    if constexpr (C::kRegsSoftmax > 0) regs_inc<C::kRegsSoftmax>();
    const int t = (warp - 4) >> 2;
    const int tl = threadIdx.x - 128 * (1 + t);   // 0..127 = TMEM lane = tile row
    const uint32_t lane_addr = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_addr + t * C::kBN;
    const uint32_t tO = tmem + lane_addr + C::kColO + t * C::kD;
    const float sl = p.pre_scale ? 1.0f : p.scale_log2;
    int blocks_seen = 0;  // s_full phases consumed (all units)
    int masks_seen = 0;   // mask tiles consumed (shared-memory mask path)
    int units_seen = 0;   // units with rows in this tile (o_ready phases with P over S)
    bool ok = true;
    for (int r = 0; ok; ++r) {
      const int u = unit_of(r, num_units);
      if (u < 0) break;
      const Unit w = decode_unit<C>(p, u);
      const int nb = t == 0 ? w.nblk[0] : w.nblk[1];
      if (nb == 0) continue;
      const int b = w.b, h = t == 0 ? w.th[0] : w.th[1];
      const int r0 = t == 0 ? w.tr[0] : w.tr[1];
      const int row = r0 + tl;
      float m_run = -INFINITY;  // running max, base 2 (scaled)
      float l_run = 0.0f;       // running sum of 2^(s - m_run)
      // Dropout: the keep bits of the block the loop is about to process (the
      // generator counter of key kbase of this row, as a function).
      auto drop_ctr = [&](int jb) {
        return p.drop_offset + (((unsigned long long)b * p.Hq + h) * p.qL + row) * (unsigned long long)(p.kL / 4) +
               (unsigned long long)(jb * (C::kBN / 4));
      };
      constexpr int kKW = C::kBN / 32;  // keep words per row and block
      uint32_t kb[C::kDropSmem ? 1 : kKW];
#pragma unroll
      for (int q = 0; q < (C::kDropSmem ? 1 : kKW); ++q) kb[q] = 0u;
      uint32_t* kb_smem = reinterpret_cast<uint32_t*>(smem + C::kOffDrop) + (t * C::kBM + tl) * kKW;
      auto next_bits = [&](int jb) {
        if constexpr (C::kDropSmem) {
          // one word at a time (a fully unrolled row block interleaves 32
          // generator chains and runs out of registers)
          const unsigned long long c0 = drop_ctr(jb);
#pragma unroll 1
          for (int q = 0; q < kKW; ++q) kb_smem[q] = drop_word(p, c0 + (unsigned long long)(q * 8));
        } else {
          drop_bits(p, drop_ctr(jb), kb);
        }
      };
      auto keep_word = [&](int cc) -> uint32_t {
        if constexpr (C::kDropSmem)
          return kb_smem[cc];
        else
          return kb[cc];
      };
      if (C::kDrop) next_bits(unit_j0<C>(w));
      for (int j = unit_j0<C>(w); j < nb; ++j) {
        ok = warp_wait(&ctl->s_full[t], blocks_seen & 1, abort_flag, p.status, p.timeout_cycles);
        if (!ok) break;
        ++blocks_seen;
        tc_fence_after();

        float s[C::kBN];
        {
          uint32_t rr[C::kBN];
#pragma unroll
          for (int cc = 0; cc < C::kBN / 32; ++cc)
            tmem_ld32(tS + cc * 32, *reinterpret_cast<uint32_t(*)[32]>(&rr[cc * 32]));
          tmem_wait_ld();
          reg_fence(rr);
#pragma unroll
          for (int c = 0; c < C::kBN; ++c) s[c] = __uint_as_float(rr[c]);
        }
        if constexpr (!C::kAliasP) {  // S_t is in registers: the next S may overwrite it
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&ctl->s_free[t]);
        }

        const int kbase = j * C::kBN;
        const int q_off = C::kFeat ? p.q_offset : 0;
        const bool need_mask = p.pre_scale || p.mask_kind != 0 || kbase + C::kBN > p.kL ||
                               (p.causal && kbase + C::kBN - 1 > r0 + q_off) ||
                               (C::kFeat && p.window > 0 && kbase <= r0 + C::kBM - 1 + q_off - p.window);
        const uint8_t* mask_tile = nullptr;
        if (C::kMaskSlotBytes > 0 && p.mask_smem) {
          ok = warp_wait(&ctl->m_full, masks_seen & 1, abort_flag, p.status, p.timeout_cycles);
          ++masks_seen;
          if (!ok) break;
          mask_tile = sM;
        }
        if (need_mask) apply_mask<C>(s, p, b, h, row, kbase, mask_tile, tl);
        if (mask_tile) {  // the mask tile is folded in: the producer may load the next one
          __syncwarp();
          if (lane == 0) mbar_arrive(&ctl->m_empty);
        }

        const float mx = row_max<C>(s);
        const float m_blk = mx * sl;  // -inf stays -inf (sl > 0 whenever it is not 1)
        const float m_new = fmaxf(m_run, m_blk);
        float corr = 1.0f;
        const bool resc = m_new > m_run + kRescaleThreshold;
        if (resc) {
          corr = ex2(m_run - m_new);  // 0 when m_run = -inf
          m_run = m_new;
        }
        const float msub = (m_run == -INFINITY) ? 0.0f : m_run;

        // P = 2^(s*sl - m): fp32 sum, stored to TMEM as bf16 pairs or tf32.
        const uint32_t tP = C::kAliasP ? tS : (tmem + lane_addr + C::kColP + (j & 1) * C::kPCols);
        float sum, unused;
        if (C::kDrop) {
          p_pass_dropout<C>(s, sl, msub, tP, sum, keep_word);
        } else {
          p_pass<C, false>(s, sl, msub, tP, sum, unused);
        }
        l_run = l_run * corr + sum;

        // Without P over S, o_ready completes once per PV; every phase is
        // consumed here, in order (PV_{j-1}, issued as softmax j-1 ended), so a
        // parity wait never runs a phase behind.  With P over S, S_j's
        // completion already implies PV_{j-1}: it was issued first.
        if constexpr (!C::kAliasP) {
          if (j > unit_j0<C>(w)) {
            ok = warp_wait(&ctl->o_ready[t], (blocks_seen - 2) & 1, abort_flag, p.status, p.timeout_cycles);
            if (!ok) break;
          }
        }
        // Rescale this warp's O rows (the previous PV has landed).
        if (j > unit_j0<C>(w) && __any_sync(0xffffffffu, resc)) {
          tc_fence_after();
#pragma unroll
          for (int cc = 0; cc < C::kD / 32; ++cc) {
            uint32_t rr[32];
            tmem_ld32(tO + cc * 32, rr);
            tmem_wait_ld();
            reg_fence(rr);
#pragma unroll
            for (int e = 0; e < 32; e += 2) {
              float o0, o1;
              fmul2(o0, o1, __uint_as_float(rr[e]), __uint_as_float(rr[e + 1]), corr, corr);
              rr[e] = __float_as_uint(o0);
              rr[e + 1] = __float_as_uint(o1);
            }
            tmem_st32(tO + cc * 32, rr);
          }
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&ctl->p_ready[t]);
        if (C::kDrop && j + 1 < nb) next_bits(j + 1);
      }
      if (!ok) break;

      // ---- epilogue: O / l from TMEM -> I/O dtype -> global (any strides); L.
      // o_ready completes once per PV without P over S, once per unit with it.
      ok = warp_wait(&ctl->o_ready[t], C::kAliasP ? (uint32_t)(units_seen & 1) : (uint32_t)((blocks_seen - 1) & 1),
                     abort_flag, p.status, p.timeout_cycles);
      ++units_seen;
      if (!ok) break;
      tc_fence_after();
      // with dropout, kept weights also take 1 / (1 - p) here (0 when p = 1)
      const float inv_l = (l_run > 0.0f) ? (C::kDrop ? p.drop_scale : 1.0f) / l_run : 0.0f;
      const bool store = row < p.qL;
      uint8_t* orow = static_cast<uint8_t*>(p.o) +
                      ((long long)b * p.o_sb + (long long)h * p.o_sh + (long long)(store ? row : 0) * p.o_ss) * C::kEsz;
      // Up to 128 columns of O per TMEM wait (one latency instead of four), so
      // the next unit's first PV may overwrite O_t before the stores go out
      // (measured: 391 -> 385 us on a non-causal B2 H32 L4096 D128 problem).
      constexpr int kBatch = C::kD / 32 < 4 ? C::kD / 32 : 4;
#pragma unroll
      for (int c0 = 0; c0 < C::kD / 32; c0 += kBatch) {
        uint32_t rb[kBatch][32];
#pragma unroll
        for (int i = 0; i < kBatch; ++i) tmem_ld32(tO + (c0 + i) * 32, rb[i]);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < kBatch; ++i) reg_fence(rb[i]);
        if (c0 + kBatch == C::kD / 32) {
          // O_t is read: the next unit's first PV may overwrite it.
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&ctl->o_free[t]);
        }
        if constexpr (C::kOStage) {
          // Through this warp's staging slot, one 128-byte column block (64
          // columns) at a time: each lane writes its row's eight 16-byte pieces
          // (piece k of row r at r * 128 + (k ^ (r & 7)) * 16: conflict-free,
          // and the layout of a 128-byte-swizzled TMA box of 32 rows), then one
          // lane hands the block to a TMA store (rows past qL are clipped).
          uint8_t* slot = smem + C::kOffOStage + (warp - 4) * (32 * 128);
          const int wrow0 = row - lane;  // the warp's first row
#pragma unroll
          for (int hh = 0; hh < kBatch / 2; ++hh) {
            const int blk = c0 / 2 + hh;  // 128-byte column block of the row
            if (lane == 0) tma_store_wait_read0();  // the slot's previous store has read it
            __syncwarp();
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              const uint32_t(&rr)[32] = rb[2 * hh + k / 4];
              uint32_t pk[4];
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                float a0, a1;
                fmul2(a0, a1, __uint_as_float(rr[(k % 4) * 8 + 2 * e]), __uint_as_float(rr[(k % 4) * 8 + 2 * e + 1]),
                      inv_l, inv_l);
                pk[e] = pack16x2<C>(a0, a1);
              }
              *reinterpret_cast<uint4*>(slot + lane * 128 + ((k ^ (lane & 7)) << 4)) =
                  make_uint4(pk[0], pk[1], pk[2], pk[3]);
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0 && wrow0 < p.qL) {
              tma_store_4d(&tmO, slot, blk * C::kChunk, wrow0, h, b);
              tma_store_commit();
            }
          }
        } else {
#pragma unroll
        for (int i = 0; i < kBatch; ++i) {
          const int cc = c0 + i;
          const uint32_t (&rr)[32] = rb[i];
          if (store) {
            if constexpr (C::kTf32) {
              uint4* dst = reinterpret_cast<uint4*>(orow + cc * 128);
#pragma unroll
              for (int u4 = 0; u4 < 8; ++u4) {
                float a0, a1, a2, a3;
                fmul2(a0, a1, __uint_as_float(rr[4 * u4 + 0]), __uint_as_float(rr[4 * u4 + 1]), inv_l, inv_l);
                fmul2(a2, a3, __uint_as_float(rr[4 * u4 + 2]), __uint_as_float(rr[4 * u4 + 3]), inv_l, inv_l);
                dst[u4] = make_uint4(__float_as_uint(a0), __float_as_uint(a1), __float_as_uint(a2), __float_as_uint(a3));
              }
            } else {
              uint4* dst = reinterpret_cast<uint4*>(orow + cc * 64);
#pragma unroll
              for (int u4 = 0; u4 < 4; ++u4) {
                uint32_t pk[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                  float a0, a1;
                  fmul2(a0, a1, __uint_as_float(rr[8 * u4 + 2 * e]), __uint_as_float(rr[8 * u4 + 2 * e + 1]), inv_l,
                        inv_l);
                  pk[e] = pack16x2<C>(a0, a1);
                }
                dst[u4] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
              }
            }
          }
        }
        }
      }
      if (store) {
        const float lse = (l_run > 0.0f) ? (m_run + lg2(l_run)) * kLn2 : -INFINITY;
        p.lse[((long long)b * p.Hq + h) * p.qL + row] = lse;
      }
    }
  }

  if constexpr (C::kOStage) {
    if (warp >= 4 && lane == 0) tma_store_wait0();  // the epilogue's O stores are complete
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

}  // namespace fa
