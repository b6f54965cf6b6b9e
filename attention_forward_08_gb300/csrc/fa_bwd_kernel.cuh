// fa_bwd_kernel.cuh -- FlashAttention-2 backward for sm_103a (bf16 or fp16 I/O):
// dQ, dK, dV of O = softmax(scale * Q K^T) V given dO and the forward's L.
//
// What it computes (per batch b, query head h, kvh = h / (H_q / H_kv)):
//   P_ij  = exp(scale * q_i . k_j - L_i)            (L from the forward)
//   D_i   = rowsum(O_i * dO_i)
//   dP_ij = dO_i . v_j,  dS_ij = P_ij (dP_ij - D_i)
//   dQ_i  = scale * sum_j dS_ij k_j
//   dK_j  = scale * sum_{h in group, i} dS_ij q_i,  dV_j = sum_{h in group, i} P_ij dO_i
// with causal (j <= i) masking and ragged tails.  Sources:
//  - forge "flash_attention_mma.metal", section "backward (MMA)": no online
//    rescale (L fixes the normalisation); a query-parallel dQ kernel
//    (S = Q K^T, P = exp(S scale - L), dP = dO V^T, dS = P (dP - D), dQ += dS K)
//    and key-parallel dK/dV work on transposed operands (S^T = K Q^T,
//    dP^T = V dO^T, dV += P^T dO, dK += dS^T Q) whose accumulation stays
//    private to one K/V block: no atomics, deterministic results;
//  - mlx-native "ops/flash_attn_train.rs", section "Phase 2 -- FA-2 backward
//    kernel (dQ, dK, dV)": the D = rowsum(O * dO) pre-pass and its [B,H_q,qL]
//    f32 layout.
//
// GB300 design:
//  - three launches: the row-dot pre-pass (HBM-bound, 16-byte loads), the
//    dK/dV kernel (one CTA per 128-key tile of one (b, kvh); it walks every
//    query block of every query head of the GQA group, so the group sum stays
//    in TMEM), and the dQ kernel (one CTA per 128-row query tile);
//  - each CTA: warp 0 issues TMA loads (and stages L, D), warp 1 owns TMEM and
//    issues every tcgen05.mma from one thread, warps 4-7 are one elementwise
//    warpgroup with thread r owning TMEM lane r (a key row in dK/dV, a query
//    row in dQ);
//  - P and dS are rounded to the I/O format (bf16 or fp16) and written over the fp32 S and dP columns
//    of TMEM; the next block's S and dP MMAs are ordered behind the MMAs that
//    read them, so the elementwise work of one block overlaps the tensor core's
//    work on the previous one;
//  - every wait is bounded; on expiry the kernel records kStatusTimeout,
//    drains its copies and MMAs, frees TMEM and returns.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "fa_kernel.cuh"

namespace fa {

struct BwdParams {
  int B, Hq, Hkv, qL, kL;
  int group;          // Hq / Hkv
  int causal;
  int window;         // > 0: key j allowed only if j > i + q_offset - window (kFeat kernels)
  int q_offset;       // causal diagonal of row i is key i + q_offset (kFeat kernels)
  int softcap_on;     // kFeat kernels: scores t = c tanh(scale s / c) (as the forward)
  float softcap_kin;  // 2 log2(e) scale / c
  float softcap_out;  // c log2(e): t in base-2 units is softcap_out * tanh(...)
  float softcap_inv;  // 1 / softcap_out
  int dropout_on;     // kDrop kernels: the forward's weights were P_ij Z_ij, Z in {0, drop_scale}
  unsigned int drop_threshold;  // keep iff (word >> 8) >= threshold (ceil(p 2^24))
  float drop_scale;   // 1 / (1 - p), 0 when p = 1
  unsigned int seed_lo, seed_hi;
  unsigned long long drop_offset;  // generator counter of position 0
  // The forward's keep decisions, written by the keep-mask pre-pass: row
  // (b H_q + h) qL + i holds keep_row_words words; bit x of word w is key
  // 32 w + x.  Only the (128-row, 128-key) tiles some row of which can see
  // some key of are written; the others are never needed (P = 0 there).
  uint32_t* keep_mask;
  long long keep_row_words;  // a multiple of 4 (16-byte rows of 128-key blocks)
  // The forward's mask (kFeat kernels): 1 bool (uint8, nonzero keeps), 2
  // additive (I/O format, added to the scaled score); the dQ kernel reads its
  // rows, the dK/dV kernel a key-major copy (written by the transpose pre-pass,
  // zero past qL) whose rows hold mask_t_ld entries (a multiple of 128).
  int mask_kind;
  const void* mask;
  long long mask_sb, mask_sh, mask_ss;
  int mask_vec;
  const void* mask_t;
  long long mask_t_ld;
  // A bool mask reaches the kernels as keep bits written by the pre-pass (the
  // dropout keep words' layout): row-major for the dQ kernel, key-major for
  // the dK/dV kernel, 16 bytes per row (or key) and 128-entry block.
  const uint32_t* mask_tbits;
  long long mask_tbits_ld;
  const uint32_t* mask_rbits;
  long long mask_rbits_ld;
  int n_qt, n_kt;     // 128-row query tiles per (b, h), 128-key tiles per (b, kvh)
  float scale;        // softmax scale (applied to dQ and dK in the epilogue)
  float scale_log2;   // scale * log2(e)
  const float* lse;   // [B, Hq, qL] natural log
  float* dvec;        // [B, Hq, qL] D_i = rowsum(O_i * dO_i)
  void* dq;           // [B, Hq, qL, D] (I/O format)
  void* dk;           // [B, Hkv, kL, D]
  void* dv;           // [B, Hkv, kL, D]
  unsigned int* status;
  long long timeout_cycles;
};

template <int kD_, bool kF16_ = false, bool kFeat_ = false, bool kDrop_ = false, int kMask_ = 0,
          bool kCap_ = kFeat_ && kMask_ == 0>
struct BwdCfg {
  static constexpr int kD = kD_;
  // 16-bit I/O is bf16 unless kF16 (fp16): same kernels, other operand format.
  static constexpr bool kF16 = kF16_;
  // Sliding window and causal diagonal offset compiled in (their own
  // instantiations: the plain kernels keep their exact code).
  static constexpr bool kFeat = kFeat_;
  // Dropout as well (its own instantiations again; implies kFeat).
  static constexpr bool kDrop = kDrop_;
  static_assert(!kDrop || kFeat, "the dropout instantiation includes the other features");
  // The forward's mask, 1 bool or 2 additive (their own instantiations again:
  // the mask words cost registers that the other feature kernels keep free).
  // A mask excludes the softcap (the launch refuses the pair), so the mask
  // kernels carry no softcap code: one probability pass each.
  static constexpr int kMaskKind = kMask_;
  static constexpr bool kMask = kMask_ != 0;
  static_assert(kMask_ >= 0 && kMask_ <= 2, "mask kinds: 0 none, 1 bool, 2 additive");
  static_assert(!kMask || kFeat, "the mask instantiation includes the other features");
  // The softcap's code (a feature kernel's option; its own instantiations, so
  // that window, offset and dropout kernels without a softcap carry none).
  static constexpr bool kCap = kCap_;
  static_assert(!kCap || (kFeat && !kMask), "the softcap needs the feature kernels and no mask");
  static constexpr uint32_t kFmt = kF16 ? kFmtF16 : kFmtBf16;
  static constexpr CUtensorMapDataType kTmaType =
      kF16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  static constexpr int kTile = 128;                     // rows per tile (queries or keys)
  static constexpr int kNChunk = kD / 64;               // 128-byte column blocks per row
  static constexpr uint32_t kTileBytes = kTile * kD * 2;
  static constexpr int kStages = kD == 64 ? 4 : 2;      // streamed-tile ring depth
  static constexpr int kKStep = 16;                     // bf16 MMA K per instruction
  static constexpr int kThreads = 256;
  // TMEM columns: S (or S^T) 0..127, dP (or dP^T) 128..255, then the accumulators.
  static constexpr int kColS = 0, kColDP = 128, kColAcc0 = 256, kColAcc1 = 256 + kD;
  // dQ kernel: the tile's Q and dO rows as 16-bit pairs after dQ (the A
  // operands of S and dP, so those MMAs read only K_j or V_j from shared
  // memory), then, where TMEM has room (D = 64), a second dP buffer, so
  // dP_{j+1} need not wait for dQ_j to read dS_j.
  static constexpr int kColQT = kColAcc0 + kD, kColDOT = kColQT + kD / 2;
  static constexpr bool kDP2 = kColDOT + kD / 2 + 128 <= 512;
  static constexpr int kColDP2 = kDP2 ? kColDOT + kD / 2 : kColDP;
  static constexpr uint32_t kTmemCols = 512;
  // dK/dV kernel shared memory: K, V, then Q and dO rings, then L2 and D slots.
  static constexpr uint32_t kKVOffQ = 2 * kTileBytes;
  static constexpr uint32_t kKVOffDO = kKVOffQ + kStages * kTileBytes;
  static constexpr uint32_t kKVOffLD = kKVOffDO + kStages * kTileBytes;
  // dK/dV kernel with dropout: per stage, the block's 128 query rows' keep
  // words for this key tile (16 bytes a row, staged with L and D); then each
  // key row's transposed words for the current step (16 bytes a key).
  static constexpr uint32_t kKVOffKB = kKVOffLD + kStages * 2 * kTile * 4;
  static constexpr uint32_t kKVOffKeep = kKVOffKB + (kDrop ? kStages * kTile * 16 : 0);
  static constexpr uint32_t kKVOffBar = kKVOffKeep + (kDrop ? kTile * 16 : 0);
  static constexpr uint32_t kKVSmem = 1024 + kKVOffBar + 512;
  // dQ kernel shared memory: Q, dO, then K and V rings.
  static constexpr uint32_t kQOffK = 2 * kTileBytes;
  static constexpr int kQKStages = kD == 64 ? 4 : 3;  // dQ kernel K ring (K_j is read by S_j and dQ_j)
  static constexpr uint32_t kQOffV = kQOffK + kQKStages * kTileBytes;
  static constexpr uint32_t kQOffBar = kQOffV + kStages * kTileBytes;
  static constexpr uint32_t kQSmem = 1024 + kQOffBar + 512;
  static_assert(kD == 64 || kD == 128, "backward head dims: 64 or 128");
  static_assert(kKVSmem <= 232448 && kQSmem <= 232448, "shared memory overflow");
  static_assert(kColAcc1 + kD <= 512, "TMEM overflow");
  static_assert(kColDOT + kD / 2 <= 512 && (!kDP2 || kColDP2 + 128 <= 512), "dQ kernel TMEM overflow");
  // The epilogues stage their gradients in rings the finished MMAs no longer read.
  static_assert(kStages * kTileBytes >= kTile * kD * 2 && kQKStages * kTileBytes >= kTile * kD * 2,
                "epilogue staging space");
};

struct BwdKVCtrl {
  uint64_t kv_full;
  uint64_t q_full[4], q_empty[4], do_full[4], do_empty[4], ld_full[4], ld_empty[4];
  uint64_t s_full, dp_full, p_ready, ds_ready, done, drain;
  uint32_t tmem_base;
  int abort;
};

struct BwdQCtrl {
  uint64_t q_full;
  uint64_t k_full[4], k_empty[4], v_full[4], v_empty[4];
  // dp_full / ds_ready per dP buffer: a phase of buffer b can only complete
  // after its previous phase was waited for, so parity waits cannot skip one.
  uint64_t s_full, s_free, dp_full[2], ds_ready[2], done, drain;
  uint64_t qt_ready;  // Q and dO copied into TMEM
  uint32_t tmem_base;
  int abort;
};

static_assert(sizeof(BwdKVCtrl) <= 512 && sizeof(BwdQCtrl) <= 512, "barrier block overflow");

// ---------------------------------------------------------------- D pre-pass

// D_i = sum_d O_id dO_id for every row of a contiguous [rows, kD] 16-bit pair
// (bf16, or fp16 with kF16): kD / 8 threads per row, one 16-byte load of each
// operand per thread, fp32 products, a shuffle reduction within the row's threads.
template <int kD, bool kF16>
__global__ void __launch_bounds__(256) fa_bwd_rowdot_kernel(const uint4* __restrict__ o,
                                                            const uint4* __restrict__ dout,
                                                            float* __restrict__ dvec, long long rows) {
  constexpr int kLanes = kD / 8;            // threads per row
  constexpr int kRowsPerBlock = 256 / kLanes;
  const int sub = threadIdx.x % kLanes;
  const long long row = (long long)blockIdx.x * kRowsPerBlock + threadIdx.x / kLanes;
  float acc = 0.0f;
  if (row < rows) {
    const uint4 a = __ldg(o + row * kLanes + sub);
    const uint4 g = __ldg(dout + row * kLanes + sub);
    const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, gw[4] = {g.x, g.y, g.z, g.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      acc = fmaf(half_bits_to_f32<kF16>(aw[e]), half_bits_to_f32<kF16>(gw[e]), acc);
      acc = fmaf(half_bits_to_f32<kF16>(aw[e] >> 16), half_bits_to_f32<kF16>(gw[e] >> 16), acc);
    }
  }
#pragma unroll
  for (int off = kLanes / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (row < rows && sub == 0) dvec[row] = acc;
}

// ---------------------------------------------------------------- keep-mask pre-pass

// Arguments of the keep-mask pre-pass beyond BwdParams: the ten round keys of
// Philox4x32-10 for the seed (key words raised by the published constants
// each round), computed once on the host.
struct KeepMaskArgs {
  uint32_t rk0[10], rk1[10];
  uint32_t n_kb, n_units;  // 128-key blocks per row; (b, h, row tile, key block) units
};

// The published Philox4x32-10 round function (Salmon, Moraes, Dror, Shaw,
// SC11) with the round keys taken from the pre-pass arguments.
__device__ __forceinline__ uint4 philox_10_rk(uint32_t c0, uint32_t c1, const KeepMaskArgs& ka) {
  uint32_t x0 = c0, x1 = c1, x2 = 0u, x3 = 0u;
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    uint32_t hi0, lo0, hi2, lo2;
    mul_wide(0xD2511F53u, x0, hi0, lo0);
    mul_wide(0xCD9E8D57u, x2, hi2, lo2);
    x0 = hi2 ^ x1 ^ ka.rk0[r];
    x1 = lo2;
    x2 = hi0 ^ x3 ^ ka.rk1[r];
    x3 = lo0;
  }
  return make_uint4(x0, x1, x2, x3);
}

// The forward's dropout decisions for the backward: position ((b H_q + h) qL
// + i) kL + j, one Philox4x32-10 block per 4 keys at counter offset +
// position / 4 (kL is a multiple of 4), keep iff word >> 8 >= threshold;
// written as p.keep_mask's row words for every (128-row, 128-key) tile some
// row of which can see some key of.  A unit of work is one tile: warp w draws
// rows w, w + 8, ..., lane l the block of keys 4 l .. 4 l + 3, and the 4-bit
// results of 8 lanes become one word with three shuffles.  Throughput-bound
// on the integer pipes (the 32 x 32-bit multiplies): 8 CTAs of 256 threads
// per SM (32 registers), 32-bit unit decoding (the host keeps n_units below
// 2^31, so u + gridDim.x cannot wrap), counters and destinations advanced by
// adds.
// (static: each backward translation unit that launches it has its own copy)
static __global__ void __launch_bounds__(256, 8) fa_bwd_keep_mask_kernel(const BwdParams p, const KeepMaskArgs ka) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const unsigned long long row_ctr = (unsigned long long)(p.kL / 4);
  const uint32_t thr = p.drop_threshold, nqt = (uint32_t)p.n_qt;
  for (uint32_t u = blockIdx.x; u < ka.n_units; u += gridDim.x) {
    const uint32_t kb = u % ka.n_kb, rest = u / ka.n_kb;
    const int r0 = (int)(rest % nqt) * 128;
    const uint32_t bh = rest / nqt;
    const int r1 = min(r0 + 128, p.qL) - 1, c0 = (int)kb * 128, c1 = min(c0 + 128, p.kL) - 1;
    // Row i sees keys i + q_offset - window < j <= i + q_offset (the causal
    // and window limits); over rows r0 .. r1 those ranges join into one.
    if (p.causal && (long long)c0 > (long long)r1 + p.q_offset) continue;
    if (p.window > 0 && (long long)c1 < (long long)r0 + p.q_offset - p.window + 1) continue;
    const long long row = (long long)bh * p.qL + r0 + warp;
    unsigned long long c = p.drop_offset + (unsigned long long)row * row_ctr + (unsigned long long)(c0 / 4 + lane);
    uint32_t* dst = p.keep_mask + row * p.keep_row_words + c0 / 32 + (lane >> 3);
#pragma unroll 4
    for (int t = 0; t < 16; ++t) {
      const uint4 w = philox_10_rk((uint32_t)c, (uint32_t)(c >> 32), ka);
      const uint32_t nib = ((w.x >> 8) >= thr ? 1u : 0u) | ((w.y >> 8) >= thr ? 2u : 0u) |
                           ((w.z >> 8) >= thr ? 4u : 0u) | ((w.w >> 8) >= thr ? 8u : 0u);
      uint32_t x = nib << (4 * (lane & 7));
      x |= __shfl_xor_sync(0xffffffffu, x, 1);
      x |= __shfl_xor_sync(0xffffffffu, x, 2);
      x |= __shfl_xor_sync(0xffffffffu, x, 4);
      if (r0 + warp + 8 * t < p.qL && (lane & 7) == 0) *dst = x;
      c += 8 * row_ctr;
      dst += 8 * p.keep_row_words;
    }
  }
}

// ---------------------------------------------------------------- shared pieces

// S-like product: dst (+)= A[128 x kD] * B[128 x kD]^T, both K-major tiles of
// 128-byte swizzled rows (kD / 64 column blocks of 128 rows).
template <class C>
__device__ __forceinline__ void bwd_mma_kmajor(uint32_t dst, uint32_t a_lo, uint32_t a_hi, uint32_t b_lo,
                                               uint32_t b_hi, uint32_t idesc) {
  constexpr int kCol = (C::kTile * 128) >> 4;
  mma_ss_lh<false, 0>(dst, a_lo, a_hi, b_lo, b_hi, idesc, 0u);
#pragma unroll
  for (int kk = 1; kk < C::kD / C::kKStep; ++kk)
    mma_ss_lh<false, 1>(dst, a_lo + (kk / 4) * kCol + (kk % 4) * 2, a_hi, b_lo + (kk / 4) * kCol + (kk % 4) * 2,
                        b_hi, idesc, 1u);
}

// Accumulating product: dst (+)= A[128 x 128] (bf16 pairs in TMEM) * B[128 x kD]
// with B an MN-major tile in shared memory (rows = the MMA's K).
template <class C>
__device__ __forceinline__ void bwd_mma_tmem_a(uint32_t dst, uint32_t a_tmem, uint32_t b_lo, uint32_t b_hi,
                                               uint32_t idesc, uint32_t acc) {
  mma_ts_lh<false, 0>(dst, a_tmem, b_lo, b_hi, idesc, acc);
#pragma unroll
  for (int kk = 1; kk < C::kTile / C::kKStep; ++kk)
    mma_ts_lh<false, 1>(dst, a_tmem + kk * 8, b_lo + ((kk * C::kKStep * 128) >> 4), b_hi, idesc, 1u);
}

// S-like product with A in TMEM: dst = A[128 x kD] (16-bit pairs in TMEM) *
// B[128 x kD]^T, B a K-major tile of 128-byte swizzled rows.
template <class C>
__device__ __forceinline__ void bwd_mma_tmem_kmajor(uint32_t dst, uint32_t a_tmem, uint32_t b_lo, uint32_t b_hi,
                                                    uint32_t idesc) {
  constexpr int kCol = (C::kTile * 128) >> 4;
  mma_ts_lh<false, 0>(dst, a_tmem, b_lo, b_hi, idesc, 0u);
#pragma unroll
  for (int kk = 1; kk < C::kD / C::kKStep; ++kk)
    mma_ts_lh<false, 1>(dst, a_tmem + kk * 8, b_lo + (kk / 4) * kCol + (kk % 4) * 2, b_hi, idesc, 1u);
}

// Row r of a K-major tile (128-byte swizzled 64-column blocks, 128 rows
// each) into this lane's TMEM columns as 16-bit pairs: the layout of an MMA's
// A operand in TMEM (column c holds elements 2c and 2c + 1).
template <class C>
__device__ __forceinline__ void bwd_row_to_tmem(const uint8_t* tile, int r, uint32_t taddr) {
#pragma unroll
  for (int c = 0; c < C::kNChunk; ++c) {
    uint32_t w[32];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const uint4 v = *reinterpret_cast<const uint4*>(tile + c * (C::kTile * 128) + r * 128 + ((k ^ (r & 7)) << 4));
      w[4 * k] = v.x;
      w[4 * k + 1] = v.y;
      w[4 * k + 2] = v.z;
      w[4 * k + 3] = v.w;
    }
    tmem_st32(taddr + c * 32, w);
  }
}

// Read 64 fp32 TMEM columns of this lane.
__device__ __forceinline__ void tmem_ld64f(uint32_t taddr, float (&x)[64]) {
  uint32_t rr[64];
  tmem_ld32(taddr, *reinterpret_cast<uint32_t(*)[32]>(&rr[0]));
  tmem_ld32(taddr + 32, *reinterpret_cast<uint32_t(*)[32]>(&rr[32]));
  tmem_wait_ld();
  reg_fence(rr);
#pragma unroll
  for (int c = 0; c < 64; ++c) x[c] = __uint_as_float(rr[c]);
}

// Read 128 fp32 TMEM columns of this thread's lane.
__device__ __forceinline__ void tmem_ld128(uint32_t taddr, float (&x)[128]) {
  uint32_t rr[128];
#pragma unroll
  for (int cc = 0; cc < 4; ++cc) tmem_ld32(taddr + cc * 32, *reinterpret_cast<uint32_t(*)[32]>(&rr[cc * 32]));
  tmem_wait_ld();
  reg_fence(rr);
#pragma unroll
  for (int c = 0; c < 128; ++c) x[c] = __uint_as_float(rr[c]);
}

// dS = P (dP - d) chunk by chunk: read 32 fp32 dP columns, write 16 columns of
// 16-bit pairs over the part of the dP region already read.  dsub(c) gives the
// D term of column c.
template <class C, class F>
__device__ __forceinline__ void bwd_ds_pass(uint32_t tdp, const float (&p)[128], F dsub) {
#pragma unroll
  for (int cc = 0; cc < 4; ++cc) {
    uint32_t rr[32];
    tmem_ld32(tdp + cc * 32, rr);
    tmem_wait_ld();
    reg_fence(rr);
    uint32_t pk[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      const int c0 = cc * 32 + 2 * e;
      const float d0 = p[c0] * (__uint_as_float(rr[2 * e]) - dsub(c0));
      const float d1 = p[c0 + 1] * (__uint_as_float(rr[2 * e + 1]) - dsub(c0 + 1));
      pk[e] = pack16x2<C>(d0, d1);
    }
    tmem_st16(tdp + cc * 16, pk);
  }
}

// The softcap's factor dt/ds = 1 - tanh^2 of one probability p > 0 of a row
// whose logsumexp (base 2) is l2: t = log2(p) + l2 = softcap_out * tanh.
// Recovered from p instead of kept (no registers spare between the two
// passes); 0 where p = 0 (dS is 0 there anyway).
__device__ __forceinline__ float softcap_factor(float p, float l2, float inv_out) {
  const float th = (lg2(p) + l2) * inv_out;
  return p > 0.0f ? fmaf(-th, th, 1.0f) : 0.0f;
}

// Bit x set for the entries base + x (x < 32) inside [lo, hi).
__device__ __forceinline__ uint32_t range_bits32(int lo, int hi, int base) {
  const int a = min(max(lo - base, 0), 32), b = min(max(hi - base, 0), 32);
  return (uint32_t)((1ull << b) - 1ull) & ~(uint32_t)((1ull << a) - 1ull);
}

// The row's limits [lo, lim) over a 128-entry block as four words of
// allowed bits, ANDed with keep words when there are some: each entry then
// costs one bit test instead of two compares.
template <int N>
__device__ __forceinline__ void allowed_words(uint32_t (&aw)[4], const uint32_t (&mw)[N], bool keep, int lo, int lim) {
#pragma unroll
  for (int q = 0; q < 4; ++q) aw[q] = range_bits32(lo, lim, 32 * q) & (keep ? mw[q] : 0xFFFFFFFFu);
}

// Probabilities of 128 scores under a bool mask given as keep bits (bit c of
// mw[0..3] for entry c): p = 2^(s * sf - l2), 0 where the entry lies outside
// [lo, lim) (the row's limits) or its bit is clear.
template <class L2, int N>
__device__ __forceinline__ void bwd_p_keepbits(float (&pr)[128], float sf, L2 l2, const uint32_t (&mw)[N], int lo,
                                               int lim) {
  static_assert(N >= 4, "four keep words");
  uint32_t aw[4];
  allowed_words(aw, mw, true, lo, lim);
#pragma unroll
  for (int c = 0; c < 128; c += 2) {
    float x0, x1;
    ffma2(x0, x1, pr[c], pr[c + 1], sf, sf, -l2(c), -l2(c + 1));
    pr[c] = (aw[c >> 5] & (1u << (c & 31))) ? ex2(x0) : 0.0f;
    pr[c + 1] = (aw[c >> 5] & (2u << (c & 31))) ? ex2(x1) : 0.0f;
  }
}

// Probabilities of 128 scores with an additive mask read in 16-byte chunks
// from its row (`row`: 128 entries; prefetched into L1 before the scores
// landed): p = 2^(s * sf - l2 + m * log2(e)), 0 outside [lo, lim).  Without
// `vec` only the first `n` entries are read, one by one (the rest add 0).
template <class C, class L2>
__device__ __forceinline__ void bwd_p_additive(float (&pr)[128], float sf, L2 l2, const uint16_t* row, bool vec,
                                               int n, int lo, int lim) {
  uint32_t aw[4];
  allowed_words(aw, aw, false, lo, lim);
#pragma unroll
  for (int cc = 0; cc < 16; ++cc) {
    uint32_t w[4];
    if (vec) {
      const uint4 v = __ldg(reinterpret_cast<const uint4*>(row) + cc);
      w[0] = v.x;
      w[1] = v.y;
      w[2] = v.z;
      w[3] = v.w;
    } else {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int c = 8 * cc + 2 * e;
        w[e] = (c < n ? (uint32_t)__ldg(row + c) : 0u) | (c + 1 < n ? (uint32_t)__ldg(row + c + 1) << 16 : 0u);
      }
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int c = 8 * cc + 2 * e;
      float x0, x1;
      ffma2(x0, x1, pr[c], pr[c + 1], sf, sf, -l2(c), -l2(c + 1));
      ffma2(x0, x1, half_bits_to_f32<C::kF16>(w[e]), half_bits_to_f32<C::kF16>(w[e] >> 16), kLog2e, kLog2e, x0, x1);
      pr[c] = (aw[c >> 5] & (1u << (c & 31))) ? ex2(x0) : 0.0f;
      pr[c + 1] = (aw[c >> 5] & (2u << (c & 31))) ? ex2(x1) : 0.0f;
    }
  }
}

// An additive mask's 128 entries of a row as 64 packed words (16-byte loads
// with `vec`; otherwise the first `n` one by one, the rest 0).
__device__ __forceinline__ void bwd_load_additive128(uint32_t (&mw)[64], const uint16_t* row, bool vec, int n) {
  if (vec) {
#pragma unroll
    for (int v = 0; v < 16; ++v) {
      const uint4 w = __ldg(reinterpret_cast<const uint4*>(row) + v);
      mw[4 * v] = w.x;
      mw[4 * v + 1] = w.y;
      mw[4 * v + 2] = w.z;
      mw[4 * v + 3] = w.w;
    }
  } else {
#pragma unroll
    for (int v = 0; v < 64; ++v)  // every index compile-time: the words stay in registers
      mw[v] = (2 * v < n ? (uint32_t)__ldg(row + 2 * v) : 0u) |
              (2 * v + 1 < n ? (uint32_t)__ldg(row + 2 * v + 1) << 16 : 0u);
  }
}

// bwd_p_additive with the 128 entries already in registers (mw, as loaded by
// bwd_load_additive128).
template <class C, class L2>
__device__ __forceinline__ void bwd_p_additive_regs(float (&pr)[128], float sf, L2 l2, const uint32_t (&mw)[64],
                                                    int lo, int lim) {
  uint32_t aw[4];
  allowed_words(aw, mw, false, lo, lim);
#pragma unroll
  for (int c = 0; c < 128; c += 2) {
    float x0, x1;
    ffma2(x0, x1, pr[c], pr[c + 1], sf, sf, -l2(c), -l2(c + 1));
    const uint32_t w = mw[c >> 1];
    ffma2(x0, x1, half_bits_to_f32<C::kF16>(w), half_bits_to_f32<C::kF16>(w >> 16), kLog2e, kLog2e, x0, x1);
    pr[c] = (aw[c >> 5] & (1u << (c & 31))) ? ex2(x0) : 0.0f;
    pr[c + 1] = (aw[c >> 5] & (2u << (c & 31))) ? ex2(x1) : 0.0f;
  }
}

// Pull a 128-entry mask row (up to 256 bytes) into L1 ahead of its use.
__device__ __forceinline__ void prefetch_row_l1(const void* row, int bytes) {
  for (int o = 0; o < bytes; o += 128)
    asm volatile("prefetch.global.L1 [%0];" ::"l"(static_cast<const char*>(row) + o));
}

// The same into L2, a step before that (`bytes` within the row).
__device__ __forceinline__ void prefetch_row_l2(const void* row, int bytes) {
  for (int o = 0; o < bytes; o += 128)
    asm volatile("prefetch.global.L2 [%0];" ::"l"(static_cast<const char*>(row) + o));
}

// Key-major copy of the forward's mask for the key-parallel kernel:
// mask_t[(b H_q + h) kL + j][i] = mask[b, h, i, j] for i < qL, 0 for qL <= i <
// ld.  HBM-bound: a CTA moves a tile of kR query rows x 128 bytes of keys (kE
// entries to a 32-bit word, kR = 32 kE: 128 x 128 bool, 64 x 64 16-bit) with
// 16-byte loads into shared memory (rows 33 words apart: conflict-free
// stores), then each lane takes a word column of kE consecutive rows,
// transposes that kE x kE block in registers with byte permutes, and the warp
// writes whole 128-byte rows of the copy.  The grid walks (key tile, query
// tile, (b, h)), the last dimension in a loop.  `vec`: the mask's base and
// row strides are 16-byte multiples (else every entry is read on its own).
// Causal (diagonal of row i at key i + q_offset): a tile whose rows see none of
// its keys is skipped, as the gradient kernels zero its entries through their
// causal limits whatever the copy holds there.
template <class T>
__global__ void __launch_bounds__(256) fa_bwd_mask_transpose_kernel(const T* __restrict__ mask, long long sb,
                                                                    long long sh, long long ss, int Hq, int BH,
                                                                    int qL, int kL, long long ld, int vec,
                                                                    int causal, int q_offset,
                                                                    T* __restrict__ mask_t) {
  constexpr int kE = 4 / sizeof(T);  // entries per 32-bit word
  constexpr int kR = 32 * kE;        // query rows per tile (one 128-byte output row)
  constexpr int kK = 32 * kE;        // keys per tile (one 128-byte input row)
  __shared__ uint32_t tile[kR][33];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int j0 = blockIdx.x * kK, i0 = blockIdx.y * kR;
  if (causal && (long long)j0 > (long long)i0 + (kR - 1) + q_offset) return;
  const bool full = vec && j0 + kK <= kL;
  for (int bh = blockIdx.z; bh < BH; bh += gridDim.z) {
    const int b = bh / Hq, h = bh - b * Hq;
    const T* src = mask + (long long)b * sb + (long long)h * sh;
    // rows of the tile: 8 lanes per row, 16 bytes a lane
#pragma unroll
    for (int it = 0; it < kR / 32; ++it) {
      const int ch = threadIdx.x + it * 256, r = ch >> 3, c16 = ch & 7;
      const int i = i0 + r;
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      if (i < qL) {
        const T* row = src + (long long)i * ss + j0 + c16 * (4 * kE);
        if (full) {
          v = __ldg(reinterpret_cast<const uint4*>(row));
        } else {
          uint32_t w[4] = {0u, 0u, 0u, 0u};
#pragma unroll
          for (int e = 0; e < 4 * kE; ++e)
            if (j0 + c16 * (4 * kE) + e < kL) w[e / kE] |= (uint32_t)row[e] << (8 * sizeof(T) * (e % kE));
          v = make_uint4(w[0], w[1], w[2], w[3]);
        }
      }
      tile[r][c16 * 4 + 0] = v.x;
      tile[r][c16 * 4 + 1] = v.y;
      tile[r][c16 * 4 + 2] = v.z;
      tile[r][c16 * 4 + 3] = v.w;
    }
    __syncthreads();
    // word column c (keys j0 + kE c ..) of rows kE lane .. kE lane + kE - 1 -> kE output rows
    T* dst = mask_t + (long long)bh * kL * ld + i0;
#pragma unroll
    for (int cw = 0; cw < 4; ++cw) {
      const int c = warp * 4 + cw;
      uint32_t out[kE];
      if constexpr (kE == 4) {
        const uint32_t r0 = tile[4 * lane][c], r1 = tile[4 * lane + 1][c];
        const uint32_t r2 = tile[4 * lane + 2][c], r3 = tile[4 * lane + 3][c];
        const uint32_t t0 = __byte_perm(r0, r1, 0x5140), t1 = __byte_perm(r0, r1, 0x7362);
        const uint32_t t2 = __byte_perm(r2, r3, 0x5140), t3 = __byte_perm(r2, r3, 0x7362);
        out[0] = __byte_perm(t0, t2, 0x5410);
        out[1] = __byte_perm(t0, t2, 0x7632);
        out[2] = __byte_perm(t1, t3, 0x5410);
        out[3] = __byte_perm(t1, t3, 0x7632);
      } else {
        const uint32_t r0 = tile[2 * lane][c], r1 = tile[2 * lane + 1][c];
        out[0] = __byte_perm(r0, r1, 0x5410);
        out[1] = __byte_perm(r0, r1, 0x7632);
      }
#pragma unroll
      for (int e = 0; e < kE; ++e) {
        const int j = j0 + kE * c + e;
        if (j < kL) reinterpret_cast<uint32_t*>(dst + (long long)j * ld)[lane] = out[e];
      }
    }
    __syncthreads();
  }
}

// Transposes a 32 x 32 bit matrix held one row per lane (bit k of lane l's
// word = element (l, k)) so that lane k ends with column k (bit l = element
// (l, k)): five butterfly stages, each swapping the off-diagonal half-blocks
// of every 2j x 2j block between lanes l and l ^ j (the register form of the
// recursive block transpose, Hacker's Delight, section 7-3).
__device__ __forceinline__ uint32_t warp_transpose32(uint32_t x, int lane) {
  constexpr uint32_t kMask[5] = {0x0000FFFFu, 0x00FF00FFu, 0x0F0F0F0Fu, 0x33333333u, 0x55555555u};
#pragma unroll
  for (int st = 0; st < 5; ++st) {
    const int j = 16 >> st;
    const uint32_t y = __shfl_xor_sync(0xffffffffu, x, j);
    const uint32_t upper = ((y >> j) ^ x) & kMask[st];         // lanes with bit j set
    const uint32_t lower = (((x >> j) ^ y) & kMask[st]) << j;  // lanes with bit j clear
    x ^= (lane & j) ? upper : lower;
  }
  return x;
}

// Keep flags of four mask bytes as four bits (bit e: byte e nonzero): the
// high bit of each byte of ((w & 0x7f..) + 0x7f..) | w is set iff the byte is
// nonzero; one multiply gathers the four flags into bits 28..31 (the partial
// products of lower flags land below bit 28 without carries).
__device__ __forceinline__ uint32_t nonzero_bytes4(uint32_t w) {
  const uint32_t t = ((((w & 0x7F7F7F7Fu) + 0x7F7F7F7Fu) | w) >> 7) & 0x01010101u;
  return (t * 0x10204080u) >> 28;
}

// A bool mask as keep bits for both gradient kernels (one read of the mask):
//   rbits[((b H_q + h) qL + i) rld + w] bit x = mask[b, h, i, 32 w + x] != 0
//   tbits[((b H_q + h) kL + j) tld + w] bit x = mask[b, h, 32 w + x, j] != 0
// with 4 words per 128-entry block (rld = 4 ceil(kL / 128), tld = 4 ceil(qL /
// 128)); entries past qL or kL are 0.  A CTA loads a 128 x 128 tile as the
// transpose does (rows 144 bytes apart: conflict-free 16-byte accesses), then
// lane r of warp w turns half of tile row 32 (w % 4) + r (keys 64 (w / 4) ..
// + 63) into two keep words, stores them (row-major) and transposes the two
// 32 x 32 bit blocks of its warp's rows in registers (key-major).  Grid as the
// uint8 transpose: (key tile, query tile, (b, h) in a loop).  Causal: tiles
// whose rows see none of their keys are skipped, as in the transpose.
static __global__ void __launch_bounds__(256) fa_bwd_mask_bits_kernel(const uint8_t* __restrict__ mask, long long sb,
                                                                      long long sh, long long ss, int Hq, int BH,
                                                                      int qL, int kL, int vec, int causal, int q_offset,
                                                                      uint32_t* __restrict__ tbits, long long tld,
                                                                      uint32_t* __restrict__ rbits, long long rld) {
  __shared__ __align__(16) uint32_t tile[128][36];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int j0 = blockIdx.x * 128, i0 = blockIdx.y * 128;
  if (causal && (long long)j0 > (long long)i0 + 127 + q_offset) return;
  const bool full = vec && j0 + 128 <= kL;
  const int rg = warp & 3, r = 32 * rg + lane;  // this lane's tile row
  for (int bh = blockIdx.z; bh < BH; bh += gridDim.z) {
    const int b = bh / Hq, h = bh - b * Hq;
    const uint8_t* src = mask + (long long)b * sb + (long long)h * sh;
#pragma unroll
    for (int it = 0; it < 4; ++it) {
      const int ch = threadIdx.x + it * 256, rr = ch >> 3, c16 = ch & 7;
      const int i = i0 + rr;
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      if (i < qL) {
        const uint8_t* row = src + (long long)i * ss + j0 + c16 * 16;
        if (full) {
          v = __ldg(reinterpret_cast<const uint4*>(row));
        } else {
          uint32_t w[4] = {0u, 0u, 0u, 0u};
#pragma unroll
          for (int e = 0; e < 16; ++e)
            if (j0 + c16 * 16 + e < kL) w[e / 4] |= (uint32_t)row[e] << (8 * (e % 4));
          v = make_uint4(w[0], w[1], w[2], w[3]);
        }
      }
      *reinterpret_cast<uint4*>(&tile[rr][c16 * 4]) = v;
    }
    __syncthreads();
    const int hk = warp >> 2;  // this warp's half of the tile's keys
    uint32_t kw[2];            // bit x of kw[gg]: key 32 (2 hk + gg) + x of row r
#pragma unroll
    for (int gg = 0; gg < 2; ++gg) {
      const int g = 2 * hk + gg;
      uint32_t bits = 0u;
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const uint4 v = *reinterpret_cast<const uint4*>(&tile[r][8 * g + 4 * q]);
        bits |= (nonzero_bytes4(v.x) | nonzero_bytes4(v.y) << 4 | nonzero_bytes4(v.z) << 8 |
                 nonzero_bytes4(v.w) << 12) << (16 * q);
      }
      kw[gg] = bits;
    }
    if (i0 + r < qL)
      *reinterpret_cast<uint2*>(rbits + ((long long)bh * qL + i0 + r) * rld + j0 / 32 + 2 * hk) =
          make_uint2(kw[0], kw[1]);
#pragma unroll
    for (int gg = 0; gg < 2; ++gg) {
      const int g = 2 * hk + gg;
      // lane x: key 32 g + x, bit l = row 32 rg + l
      const uint32_t mine = warp_transpose32(kw[gg], lane);
      if (j0 + 32 * g + lane < kL) tbits[((long long)bh * kL + j0 + 32 * g + lane) * tld + i0 / 32 + rg] = mine;
    }
    __syncthreads();
  }
}

// Keep bits to masks in two steps.  keep_bytes spreads bits shift .. shift
// + 3 of a keep word into the sign bits of four bytes (byte k = 0x80 when bit
// shift + k is set): one multiply places bit k at 7 (k + 1) + k = 8 k + 7,
// and the shifted copies of the 4-bit field never overlap, so no carries
// reach those positions.  A byte permute with sign replication then turns
// byte k into a 32-bit mask (elem_mask) or bytes k, k + 1 into the mask of a
// packed 16-bit pair (pair_mask).
__device__ __forceinline__ uint32_t keep_bytes(uint32_t word, int shift) {
  return (((word >> shift) & 0xFu) * 0x10204080u) & 0x80808080u;
}
__device__ __forceinline__ uint32_t prmt_sign(uint32_t a, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, 0, %2;" : "=r"(d) : "r"(a), "r"(sel));
  return d;
}
__device__ __forceinline__ uint32_t elem_mask(uint32_t bytes, int k) {
  return prmt_sign(bytes, (uint32_t)(8 | k) * 0x1111u);
}
__device__ __forceinline__ uint32_t pair_mask(uint32_t bytes, int k) {
  return prmt_sign(bytes, (uint32_t)(8 | k) * 0x0011u | (uint32_t)(8 | (k + 1)) * 0x1100u);
}

// dS with dropout (and, with kCap, the softcap's factor): dS = P (Z dP - d)
// f; kword(cc) gives the keep word of columns 32 cc .. 32 cc + 31.  With
// kPerm, Z dP = scale * (dP masked through keep_bytes / elem_mask); without,
// Z = scale masked by the bit's negation.  (Measured on the causal GQA
// dropout workload: the byte permutes saved 75 us in the dK/dV kernel and
// cost 48 us in the dQ kernel, so each kernel takes its faster form.)
template <class C, bool kCap, bool kPerm, class F, class L, class K>
__device__ __forceinline__ void bwd_ds_pass_drop(uint32_t tdp, const float (&p)[128], F dsub, L l2, float inv_out,
                                                 K kword, float scale) {
#pragma unroll
  for (int cc = 0; cc < 4; ++cc) {
    uint32_t rr[32];
    tmem_ld32(tdp + cc * 32, rr);
    tmem_wait_ld();
    reg_fence(rr);
    uint32_t pk[16];
    const uint32_t kw = kword(cc);
    uint32_t kb4 = 0;
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      const int c0 = cc * 32 + 2 * e;
      float d0, d1;
      if constexpr (kPerm) {
        if ((e & 1) == 0) kb4 = keep_bytes(kw, 2 * e);
        const float z0 = __uint_as_float(rr[2 * e] & elem_mask(kb4, 2 * (e & 1)));
        const float z1 = __uint_as_float(rr[2 * e + 1] & elem_mask(kb4, 2 * (e & 1) + 1));
        d0 = p[c0] * fmaf(scale, z0, -dsub(c0));
        d1 = p[c0 + 1] * fmaf(scale, z1, -dsub(c0 + 1));
      } else {
        const float k0 = __int_as_float(__float_as_int(scale) & (0u - ((kw >> (2 * e)) & 1u)));
        const float k1 = __int_as_float(__float_as_int(scale) & (0u - ((kw >> (2 * e + 1)) & 1u)));
        d0 = p[c0] * fmaf(k0, __uint_as_float(rr[2 * e]), -dsub(c0));
        d1 = p[c0 + 1] * fmaf(k1, __uint_as_float(rr[2 * e + 1]), -dsub(c0 + 1));
      }
      if constexpr (kCap) {
        d0 *= softcap_factor(p[c0], l2(c0), inv_out);
        d1 *= softcap_factor(p[c0 + 1], l2(c0 + 1), inv_out);
      }
      pk[e] = pack16x2<C>(d0, d1);
    }
    tmem_st16(tdp + cc * 16, pk);
  }
}

// bwd_ds_pass with the softcap's factor: dS = P (dP - d) (1 - tanh^2);
// l2(c) gives the base-2 logsumexp of column c's row.
template <class C, class F, class L>
__device__ __forceinline__ void bwd_ds_pass_softcap(uint32_t tdp, const float (&p)[128], F dsub, L l2,
                                                    float inv_out) {
#pragma unroll
  for (int cc = 0; cc < 4; ++cc) {
    uint32_t rr[32];
    tmem_ld32(tdp + cc * 32, rr);
    tmem_wait_ld();
    reg_fence(rr);
    uint32_t pk[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      const int c0 = cc * 32 + 2 * e;
      const float d0 = p[c0] * (__uint_as_float(rr[2 * e]) - dsub(c0)) * softcap_factor(p[c0], l2(c0), inv_out);
      const float d1 =
          p[c0 + 1] * (__uint_as_float(rr[2 * e + 1]) - dsub(c0 + 1)) * softcap_factor(p[c0 + 1], l2(c0 + 1), inv_out);
      pk[e] = pack16x2<C>(d0, d1);
    }
    tmem_st16(tdp + cc * 16, pk);
  }
}

// Store a 128 x kD fp32 accumulator row (this thread's lane), times `mul`, in
// the 16-bit I/O format to a contiguous row of global memory (16-byte stores;
// the additive-mask kernels' epilogue, whose registers the staged one would
// push into spills).
template <class C>
__device__ __forceinline__ void bwd_store_row(uint32_t tacc, float mul, uint16_t* dst, bool store) {
#pragma unroll
  for (int cc = 0; cc < C::kD / 32; ++cc) {
    uint32_t rr[32];
    tmem_ld32(tacc + cc * 32, rr);
    tmem_wait_ld();
    reg_fence(rr);
    if (store) {
      uint4* d4 = reinterpret_cast<uint4*>(dst + cc * 32);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        uint32_t pk[4];
#pragma unroll
        for (int e = 0; e < 4; ++e)
          pk[e] = pack16x2<C>(__uint_as_float(rr[8 * u + 2 * e]) * mul, __uint_as_float(rr[8 * u + 2 * e + 1]) * mul);
        d4[u] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
      }
    }
  }
}

// The epilogue of one fp32 accumulator through TMA stores: kCols columns of
// this warp's 32 rows (its TMEM lanes), scaled and packed to the I/O format,
// staged as kCols / 64 boxes of 32 rows x 128 bytes with the 128-byte swizzle
// (row r's 16-byte piece k at r * 128 + (k ^ (r & 7)) * 16: conflict-free) in
// `slot` -- ring space that the finished MMAs no longer read, 1024-byte
// aligned -- then stored by lane 0 at columns x0 .., rows row0 .. row0 + 31 of
// (head, batch); rows past the tensor's extent are clipped.  One TMEM load
// wait per 64 columns.
template <class C, int kCols = C::kD>
__device__ __forceinline__ void bwd_store_tile_tma(uint32_t tacc, float mul, uint8_t* slot, const CUtensorMap* map,
                                                   int x0, int row0, int extent, int head, int batch, int lane) {
  constexpr int kBlk = kCols / 64;  // 128-byte column blocks
#pragma unroll
  for (int blk = 0; blk < kBlk; ++blk) {
    uint32_t rr[2][32];
    tmem_ld32(tacc + blk * 64, rr[0]);
    tmem_ld32(tacc + blk * 64 + 32, rr[1]);
    tmem_wait_ld();
    reg_fence(rr[0]);
    reg_fence(rr[1]);
    uint8_t* box = slot + blk * (32 * 128);
#pragma unroll
    for (int k = 0; k < 8; ++k) {  // piece k: columns 8k .. 8k + 7 of the block
      const uint32_t(&r)[32] = rr[k / 4];
      uint32_t pk[4];
#pragma unroll
      for (int e = 0; e < 4; ++e)
        pk[e] = pack16x2<C>(__uint_as_float(r[(k % 4) * 8 + 2 * e]) * mul,
                            __uint_as_float(r[(k % 4) * 8 + 2 * e + 1]) * mul);
      *reinterpret_cast<uint4*>(box + lane * 128 + ((k ^ (lane & 7)) << 4)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
    }
  }
  fence_proxy_async_smem();
  __syncwarp();
  if (lane == 0 && row0 < extent) {
#pragma unroll
    for (int blk = 0; blk < kBlk; ++blk) tma_store_4d(map, slot + blk * (32 * 128), x0 + blk * 64, row0, head, batch);
    tma_store_commit();
  }
}

// ---------------------------------------------------------------- dK / dV

// One CTA per (128-key tile, kvh, b), heavy (early) key tiles first.  It walks
// steps i = (query head r of the group, query block qb) and accumulates
//   dV += P^T dO and dK += dS^T Q   (scale applied in the epilogue)
// with S^T = K Q^T and dP^T = V dO^T recomputed per step.
template <class C>
__global__ void __launch_bounds__(C::kThreads, 1)
    fa_bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
                       const __grid_constant__ CUtensorMap tmDK, const __grid_constant__ CUtensorMap tmDV,
                       const BwdParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sK = smem;
  uint8_t* sV = smem + C::kTileBytes;
  uint8_t* sQ = smem + C::kKVOffQ;
  uint8_t* sDO = smem + C::kKVOffDO;
  float* sLD = reinterpret_cast<float*>(smem + C::kKVOffLD);  // per slot: 128 L2 values, then 128 D values
  BwdKVCtrl* ctl = reinterpret_cast<BwdKVCtrl*>(smem + C::kKVOffBar);
  volatile int* abort_flag = &ctl->abort;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int per_kt = p.Hkv * p.B;
  const int kt = blockIdx.x / per_kt;
  const int rem = blockIdx.x - kt * per_kt;
  const int b = rem / p.Hkv, kvh = rem - b * p.Hkv;
  const int k0 = kt * C::kTile;
  // Query blocks that see this tile's keys: causal, row i sees key j when
  // j <= i + q_offset, so rows from k0 - q_offset; with a window, row i sees
  // key j only while j > i + q_offset - window, so rows below
  // j_max - q_offset + window.
  int qb0, qb_end;
  if constexpr (C::kFeat) {
    const long long first = (long long)k0 - p.q_offset;
    qb0 = !p.causal || first <= 0 ? 0 : (int)min(first / C::kTile, (long long)p.n_qt);
    qb_end = p.n_qt;
    if (p.window > 0) {
      const long long jmax = min(k0 + C::kTile, p.kL) - 1;
      const long long last_row = jmax - p.q_offset + p.window - 1;  // the last row that sees key jmax
      qb_end = last_row < 0 ? 0 : (int)min(last_row / C::kTile + 1, (long long)p.n_qt);
    }
  } else {
    qb0 = p.causal ? min(k0 / C::kTile, p.n_qt) : 0;
    qb_end = p.n_qt;
  }
  const int per_head = max(0, qb_end - qb0);
  const int n_steps = p.group * per_head;

  if (threadIdx.x == 0) {
    mbar_init(&ctl->kv_full, 1);
    for (int s = 0; s < 4; ++s) {
      mbar_init(&ctl->q_full[s], 1);
      mbar_init(&ctl->q_empty[s], 1);
      mbar_init(&ctl->do_full[s], 1);
      mbar_init(&ctl->do_empty[s], 1);
      mbar_init(&ctl->ld_full[s], 32);   // every producer lane stages its 4 queries
      mbar_init(&ctl->ld_empty[s], 4);   // one arrival per elementwise warp
    }
    mbar_init(&ctl->s_full, 1);
    mbar_init(&ctl->dp_full, 1);
    mbar_init(&ctl->p_ready, 4);
    mbar_init(&ctl->ds_ready, 4);
    mbar_init(&ctl->done, 1);
    mbar_init(&ctl->drain, 1);
    ctl->abort = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    tma_prefetch_desc(&tmDO);
  }
  if (warp == 1) {
    tmem_alloc(&ctl->tmem_base, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl->tmem_base;

  auto step_of = [&](int i, int& h, int& q0) {
    const int r = i / per_head;
    h = kvh * p.group + r;
    q0 = (qb0 + (i - r * per_head)) * C::kTile;
  };

  if (warp == 0) {
    // ===================================================== producer: TMA + L, D staging
    int q_issued = 0, do_issued = 0;
    bool ok = true;
    if (lane == 0 && n_steps > 0) {
      mbar_arrive_expect_tx(&ctl->kv_full, 2 * C::kTileBytes);
#pragma unroll
      for (int c = 0; c < C::kNChunk; ++c) {
        tma_load_4d(sK + c * (C::kTile * 128), &tmK, &ctl->kv_full, c * 64, k0, kvh, b);
        tma_load_4d(sV + c * (C::kTile * 128), &tmV, &ctl->kv_full, c * 64, k0, kvh, b);
      }
    }
    for (int i = 0; i < n_steps && ok; ++i) {
      int h, q0;
      step_of(i, h, q0);
      const int s = i % C::kStages, use = i / C::kStages;
      if (lane == 0) {
        ok = wait_bounded(&ctl->q_empty[s], (use & 1) ^ 1, abort_flag, p.status, p.timeout_cycles);
        if (ok) {
          mbar_arrive_expect_tx(&ctl->q_full[s], C::kTileBytes);
#pragma unroll
          for (int c = 0; c < C::kNChunk; ++c)
            tma_load_4d(sQ + s * C::kTileBytes + c * (C::kTile * 128), &tmQ, &ctl->q_full[s], c * 64, q0, h, b);
          ++q_issued;
          ok = wait_bounded(&ctl->do_empty[s], (use & 1) ^ 1, abort_flag, p.status, p.timeout_cycles);
        }
        if (ok) {
          mbar_arrive_expect_tx(&ctl->do_full[s], C::kTileBytes);
#pragma unroll
          for (int c = 0; c < C::kNChunk; ++c)
            tma_load_4d(sDO + s * C::kTileBytes + c * (C::kTile * 128), &tmDO, &ctl->do_full[s], c * 64, q0, h, b);
          ++do_issued;
        }
      }
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      if (!ok) break;
      // L2 = L * log2(e) (+inf where the query is past qL or its row had no
      // allowed key, so P = 0 there) and D for the block's 128 queries.
      ok = warp_wait(&ctl->ld_empty[s], (use & 1) ^ 1, abort_flag, p.status, p.timeout_cycles);
      if (!ok) break;
      float* l2s = sLD + s * 2 * C::kTile;
      const long long base = ((long long)b * p.Hq + h) * p.qL;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int c = lane * 4 + e, iq = q0 + c;
        float l2 = __int_as_float(0x7f800000), dv = 0.0f;
        if (iq < p.qL) {
          const float L = __ldg(p.lse + base + iq);
          if (L != -INFINITY) l2 = L * kLog2e;
          dv = p.dvec[base + iq];
        }
        l2s[c] = l2;
        l2s[C::kTile + c] = dv;
        if constexpr (C::kDrop) {  // the row's keep words of this key tile
          uint4 kb = make_uint4(0u, 0u, 0u, 0u);
          if (iq < p.qL)
            kb = __ldg(reinterpret_cast<const uint4*>(p.keep_mask + (base + iq) * p.keep_row_words + k0 / 32));
          reinterpret_cast<uint4*>(smem + C::kKVOffKB)[s * C::kTile + c] = kb;
        }
      }
      mbar_arrive(&ctl->ld_full[s]);
    }
    if (lane == 0 && *abort_flag) {
      // Let every copy this thread started land before the CTA lets go of its memory.
      if (n_steps > 0) wait_bounded(&ctl->kv_full, 0, abort_flag, p.status, kDrainCycles, false);
      for (int it = max(0, q_issued - C::kStages); it < q_issued; ++it)
        wait_bounded(&ctl->q_full[it % C::kStages], (it / C::kStages) & 1, abort_flag, p.status, kDrainCycles,
                     false);
      for (int it = max(0, do_issued - C::kStages); it < do_issued; ++it)
        wait_bounded(&ctl->do_full[it % C::kStages], (it / C::kStages) & 1, abort_flag, p.status, kDrainCycles,
                     false);
    }
  } else if (warp == 1) {
    // ===================================================== MMA issuer
    if (lane == 0 && n_steps > 0) {
      constexpr uint32_t idS = make_idesc_fmt(C::kFmt, 128, 128, false, false);     // K-major A and B
      constexpr uint32_t idAcc = make_idesc_fmt(C::kFmt, 128, C::kD, false, true);  // B MN-major
      const uint64_t dK = make_sdesc_sw128(smem_u32(sK), 16, 1024);
      const uint64_t dV = make_sdesc_sw128(smem_u32(sV), 16, 1024);
      const uint64_t dQk = make_sdesc_sw128(smem_u32(sQ), 16, 1024);
      const uint64_t dOk = make_sdesc_sw128(smem_u32(sDO), 16, 1024);
      const uint64_t dQmn = make_sdesc_sw128(smem_u32(sQ), C::kTile * 128, 1024);
      const uint64_t dOmn = make_sdesc_sw128(smem_u32(sDO), C::kTile * 128, 1024);
      const uint32_t hi = (uint32_t)(dK >> 32), hi_mn = (uint32_t)(dQmn >> 32);
      const uint32_t slot = C::kTileBytes >> 4;
      auto issue_s = [&](int s) {  // S^T = K Q_s^T
        bwd_mma_kmajor<C>(tmem + C::kColS, (uint32_t)dK, hi, (uint32_t)dQk + s * slot, hi, idS);
      };
      auto issue_dp = [&](int s) {  // dP^T = V dO_s^T
        bwd_mma_kmajor<C>(tmem + C::kColDP, (uint32_t)dV, hi, (uint32_t)dOk + s * slot, hi, idS);
      };
      bool ok = wait_bounded(&ctl->kv_full, 0, abort_flag, p.status, p.timeout_cycles);
      if (ok) ok = wait_bounded(&ctl->q_full[0], 0, abort_flag, p.status, p.timeout_cycles);
      if (ok) {
        tc_fence_after();
        issue_s(0);
        mma_commit(&ctl->s_full);
        ok = wait_bounded(&ctl->do_full[0], 0, abort_flag, p.status, p.timeout_cycles);
      }
      if (ok) {
        tc_fence_after();
        issue_dp(0);
        mma_commit(&ctl->dp_full);
      }
      for (int i = 0; i < n_steps && ok; ++i) {
        const int s = i % C::kStages;
        const int s1 = (i + 1) % C::kStages, use1 = (i + 1) / C::kStages;
        const bool more = i + 1 < n_steps;
        ok = wait_bounded(&ctl->p_ready, i & 1, abort_flag, p.status, p.timeout_cycles);
        if (!ok) break;
        tc_fence_after();
        // dV += P^T dO_i (P^T: bf16 pairs over the S^T columns)
        bwd_mma_tmem_a<C>(tmem + C::kColAcc0, tmem + C::kColS, (uint32_t)dOmn + s * slot, hi_mn, idAcc,
                          i > 0 ? 1u : 0u);
        mma_commit(&ctl->do_empty[s]);
        if (more) {
          ok = wait_bounded(&ctl->q_full[s1], use1 & 1, abort_flag, p.status, p.timeout_cycles);
          if (!ok) break;
          tc_fence_after();
          issue_s(s1);
          mma_commit(&ctl->s_full);
        }
        ok = wait_bounded(&ctl->ds_ready, i & 1, abort_flag, p.status, p.timeout_cycles);
        if (!ok) break;
        tc_fence_after();
        // dK += dS^T Q_i (dS^T: bf16 pairs over the dP^T columns)
        bwd_mma_tmem_a<C>(tmem + C::kColAcc1, tmem + C::kColDP, (uint32_t)dQmn + s * slot, hi_mn, idAcc,
                          i > 0 ? 1u : 0u);
        mma_commit(&ctl->q_empty[s]);
        if (more) {
          ok = wait_bounded(&ctl->do_full[s1], use1 & 1, abort_flag, p.status, p.timeout_cycles);
          if (!ok) break;
          tc_fence_after();
          issue_dp(s1);
          mma_commit(&ctl->dp_full);
        }
      }
      if (ok) mma_commit(&ctl->done);
      // Drain: every MMA this thread issued completes before TMEM is freed.
      mma_commit(&ctl->drain);
      wait_bounded(&ctl->drain, 0, abort_flag, p.status, kDrainCycles, false);
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ===================================================== elementwise warpgroup: thread = key row
    const int tl = threadIdx.x - 128;
    const int j = k0 + tl;
    const uint32_t lane_addr = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_addr + C::kColS;
    const uint32_t tDP = tmem + lane_addr + C::kColDP;
    const float sl = p.scale_log2;
    // Dropout: this key row's keep bits for the step (bit c of word q: query
    // row q0 + 32 q + c), transposed from the staged row words while the MMA
    // warp computes S^T.
    uint4* keep_smem = reinterpret_cast<uint4*>(smem + C::kKVOffKeep) + tl;
    // The forward's mask for this key and a step's 128 queries: keep bits
    // (16 bytes) or the key-major copy's row (256 bytes; contiguous, 16-byte
    // aligned).  The next step's are fetched a step ahead (bits into
    // registers, a row into L2), so their DRAM latency hides behind this step.
    auto tbits_at = [&](int hh, int qq) {
      return reinterpret_cast<const uint4*>(p.mask_tbits + (((long long)b * p.Hq + hh) * p.kL + j) * p.mask_tbits_ld +
                                            qq / 32);
    };
    auto madd_at = [&](int hh, int qq) {
      return static_cast<const uint16_t*>(p.mask_t) + (((long long)b * p.Hq + hh) * p.kL + j) * p.mask_t_ld + qq;
    };
    uint4 kb_next = make_uint4(0u, 0u, 0u, 0u);
    if constexpr (C::kMask) {
      if (j < p.kL && n_steps > 0) {
        int h0, q00;
        step_of(0, h0, q00);
        if constexpr (C::kMaskKind == 1)
          kb_next = __ldg(tbits_at(h0, q00));
        else
          prefetch_row_l2(madd_at(h0, q00), 256);
      }
    }
    bool ok = true;
    for (int i = 0; i < n_steps && ok; ++i) {
      int h, q0;
      step_of(i, h, q0);
      const int s = i % C::kStages, use = i / C::kStages;
      const float* l2s = sLD + s * 2 * C::kTile;
      uint32_t mw[4];
      const uint16_t* madd = nullptr;
      if constexpr (C::kMask) {
        if (j < p.kL) {
          int hn = h, qn = q0;
          const bool more = i + 1 < n_steps;
          if (more) step_of(i + 1, hn, qn);
          if constexpr (C::kMaskKind == 1) {  // keep bits of the step's 128 queries
            mw[0] = kb_next.x;
            mw[1] = kb_next.y;
            mw[2] = kb_next.z;
            mw[3] = kb_next.w;
            if (more) kb_next = __ldg(tbits_at(hn, qn));
          } else {  // the row, read in the P pass
            madd = madd_at(h, q0);
            prefetch_row_l1(madd, 256);
            if (more) prefetch_row_l2(madd_at(hn, qn), 256);
          }
        }
      }
      ok = warp_wait(&ctl->ld_full[s], use & 1, abort_flag, p.status, p.timeout_cycles);
      if (!ok) break;
      if constexpr (C::kDrop) {
        // Lane l reads row 32 q + l's word for this warp's 32 keys; the
        // transpose hands lane k the column of key k0 + 32 (warp & 3) + k.
        const uint32_t* kb = reinterpret_cast<const uint32_t*>(smem + C::kKVOffKB) + s * C::kTile * 4 + (warp & 3);
        uint32_t kw[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) kw[q] = warp_transpose32(kb[(32 * q + lane) * 4], lane);
        *keep_smem = make_uint4(kw[0], kw[1], kw[2], kw[3]);
      }
      ok = warp_wait(&ctl->s_full, i & 1, abort_flag, p.status, p.timeout_cycles);
      if (!ok) break;
      tc_fence_after();
      float pr[128];
      tmem_ld128(tS, pr);
      // P^T_{j,c} = 2^(s * scale * log2e - L2_c); queries c < j - q0 are causally masked,
      // and a key row past kL gets no probability at all.  With the features:
      // queries c < j - q_offset - q0 (causal) or c >= j - q_offset + window - q0
      // (window) see no key j.
      if constexpr (C::kFeat) {
        int lim = p.causal ? j - p.q_offset - q0 : -(1 << 30);
        int hi = p.window > 0 ? j - p.q_offset + p.window - q0 : (1 << 30);
        if (j >= p.kL) lim = C::kTile;
        const bool capped = C::kCap && p.softcap_on;
        if (capped) {  // base-2 capped score, as the forward computes it
          const float kin = p.softcap_kin, cout = p.softcap_out;
#pragma unroll
          for (int c = 0; c < 128; ++c) pr[c] = fmaf(-2.0f * cout, rcp_approx(ex2(pr[c] * kin) + 1.0f), cout);
        }
        const float sf = capped ? 1.0f : sl;
        if (C::kMask && j < p.kL) {
          if constexpr (C::kMaskKind == 2)
            bwd_p_additive<C>(pr, sf, [&](int c) { return l2s[c]; }, madd, true, 128, lim, hi);
          else
            bwd_p_keepbits(pr, sf, [&](int c) { return l2s[c]; }, mw, lim, hi);
        } else {
          uint32_t aw[4];
          allowed_words(aw, aw, false, lim, hi);
#pragma unroll
          for (int c = 0; c < 128; c += 2) {
            float x0, x1;
            ffma2(x0, x1, pr[c], pr[c + 1], sf, sf, -l2s[c], -l2s[c + 1]);
            pr[c] = (aw[c >> 5] & (1u << (c & 31))) ? ex2(x0) : 0.0f;
            pr[c + 1] = (aw[c >> 5] & (2u << (c & 31))) ? ex2(x1) : 0.0f;
          }
        }
      } else {
        int lim = p.causal ? j - q0 : 0;
        if (j >= p.kL) lim = C::kTile;
#pragma unroll
        for (int c = 0; c < 128; c += 2) {
          float x0, x1;
          ffma2(x0, x1, pr[c], pr[c + 1], sl, sl, -l2s[c], -l2s[c + 1]);
          pr[c] = c < lim ? 0.0f : ex2(x0);
          pr[c + 1] = c + 1 < lim ? 0.0f : ex2(x1);
        }
      }
      const uint32_t* keep_words = reinterpret_cast<const uint32_t*>(keep_smem);
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) {
        uint32_t pk[16];
        const uint32_t kw = C::kDrop ? keep_words[cc] : 0u;
        uint32_t kb4 = 0;
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          pk[e] = pack16x2<C>(pr[cc * 32 + 2 * e], pr[cc * 32 + 2 * e + 1]);
          if constexpr (C::kDrop) {  // dV takes the dropped weights P Z (Z's scale in the epilogue)
            if ((e & 1) == 0) kb4 = keep_bytes(kw, 2 * e);
            pk[e] &= pair_mask(kb4, 2 * (e & 1));
          }
        }
        tmem_st16(tS + cc * 16, pk);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl->p_ready);
      // dS^T = P^T (dP^T - D_c)
      ok = warp_wait(&ctl->dp_full, i & 1, abort_flag, p.status, p.timeout_cycles);
      if (!ok) break;
      tc_fence_after();
      if constexpr (C::kDrop) {
        auto dsub = [&](int c) { return l2s[C::kTile + c]; };
        auto l2c = [&](int c) { return l2s[c]; };
        auto kword = [&](int cc) { return keep_words[cc]; };
        if (C::kCap && p.softcap_on)
          bwd_ds_pass_drop<C, C::kCap, true>(tDP, pr, dsub, l2c, p.softcap_inv, kword, p.drop_scale);
        else
          bwd_ds_pass_drop<C, false, true>(tDP, pr, dsub, l2c, 0.0f, kword, p.drop_scale);
      } else if (C::kCap && p.softcap_on) {
        bwd_ds_pass_softcap<C>(tDP, pr, [&](int c) { return l2s[C::kTile + c]; }, [&](int c) { return l2s[c]; },
                               p.softcap_inv);
      } else {
        bwd_ds_pass<C>(tDP, pr, [&](int c) { return l2s[C::kTile + c]; });
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&ctl->ds_ready);
        mbar_arrive(&ctl->ld_empty[s]);
      }

    }
    // ---- epilogue: dV and scale * dK rows (key j) as bf16
    if (ok) {
      const bool store = j < p.kL;
      const long long row = ((long long)b * p.Hkv + kvh) * p.kL + (store ? j : 0);
      uint16_t* dvp = static_cast<uint16_t*>(p.dv) + row * C::kD;
      uint16_t* dkp = static_cast<uint16_t*>(p.dk) + row * C::kD;
      if (n_steps == 0) {  // no query sees these keys: zero gradients
        if (store) {
          uint4* a4 = reinterpret_cast<uint4*>(dvp);
          uint4* b4 = reinterpret_cast<uint4*>(dkp);
          for (int u = 0; u < C::kD / 8; ++u) a4[u] = b4[u] = make_uint4(0, 0, 0, 0);
        }
      } else {
        ok = warp_wait(&ctl->done, 0, abort_flag, p.status, p.timeout_cycles);
        if (ok) {
          tc_fence_after();
          if constexpr (C::kMaskKind == 2) {
            bwd_store_row<C>(tmem + lane_addr + C::kColAcc0, C::kDrop ? p.drop_scale : 1.0f, dvp, store);
            bwd_store_row<C>(tmem + lane_addr + C::kColAcc1, p.scale, dkp, store);
          } else {  // staged in the Q and dO rings (every load of them consumed)
            constexpr int kSlot = (C::kD / 64) * 32 * 128;
            const int row0 = k0 + 32 * (warp & 3);
            bwd_store_tile_tma<C>(tmem + lane_addr + C::kColAcc0, C::kDrop ? p.drop_scale : 1.0f,
                                  sQ + (warp & 3) * kSlot, &tmDV, 0, row0, p.kL, kvh, b, lane);
            bwd_store_tile_tma<C>(tmem + lane_addr + C::kColAcc1, p.scale, sDO + (warp & 3) * kSlot, &tmDK, 0, row0,
                                  p.kL, kvh, b, lane);
            if (lane == 0) tma_store_wait0();
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

// ---------------------------------------------------------------- dQ

// One CTA per (128-row query tile, h, b), heavy (late, causal) tiles first.
// Per key block j: S = Q K_j^T, dP = dO V_j^T, dS = P (dP - D), dQ += dS K_j.
template <class C>
__global__ void __launch_bounds__(C::kThreads, 1)
    fa_bwd_dq_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                     const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
                     const __grid_constant__ CUtensorMap tmDQ,
                     const BwdParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem;
  uint8_t* sDO = smem + C::kTileBytes;
  uint8_t* sK = smem + C::kQOffK;
  uint8_t* sV = smem + C::kQOffV;
  BwdQCtrl* ctl = reinterpret_cast<BwdQCtrl*>(smem + C::kQOffBar);
  volatile int* abort_flag = &ctl->abort;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int per_qt = p.Hq * p.B;
  const int qt_rev = blockIdx.x / per_qt;
  const int rem = blockIdx.x - qt_rev * per_qt;
  const int b = rem / p.Hq, h = rem - b * p.Hq;
  const int qt = p.causal ? p.n_qt - 1 - qt_rev : qt_rev;
  const int q0 = qt * C::kTile;
  const int kvh = h / p.group;
  const int last = min(q0 + C::kTile, p.qL) - 1;
  // Key blocks [jb0, jb0 + n_blk) that the tile's rows see: up to the causal
  // diagonal (row i: key i + q_offset), from the window's first key of row q0.
  int jb0 = 0, n_blk;
  if constexpr (C::kFeat) {
    const long long diag_end = (long long)last + 1 + p.q_offset;
    const int kv_end = p.causal ? (int)max(0LL, min((long long)p.kL, diag_end)) : p.kL;
    const int nb = (kv_end + C::kTile - 1) / C::kTile;
    if (p.window > 0) {
      const long long first = (long long)q0 + p.q_offset - p.window + 1;
      jb0 = first <= 0 ? 0 : (int)min(first / C::kTile, (long long)nb);
    }
    n_blk = nb - jb0;
  } else {
    const int kv_end = p.causal ? min(p.kL, last + 1) : p.kL;
    n_blk = (kv_end + C::kTile - 1) / C::kTile;
  }

  if (threadIdx.x == 0) {
    mbar_init(&ctl->q_full, 1);
    for (int s = 0; s < 4; ++s) {
      mbar_init(&ctl->k_full[s], 1);
      mbar_init(&ctl->k_empty[s], 1);
      mbar_init(&ctl->v_full[s], 1);
      mbar_init(&ctl->v_empty[s], 1);
    }
    mbar_init(&ctl->s_full, 1);
    mbar_init(&ctl->s_free, 4);
    for (int d = 0; d < 2; ++d) {
      mbar_init(&ctl->dp_full[d], 1);
      mbar_init(&ctl->ds_ready[d], 4);
    }
    mbar_init(&ctl->qt_ready, 4);  // one arrival per elementwise warp
    mbar_init(&ctl->done, 1);
    mbar_init(&ctl->drain, 1);
    ctl->abort = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    tma_prefetch_desc(&tmDO);
  }
  if (warp == 1) {
    tmem_alloc(&ctl->tmem_base, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl->tmem_base;

  if (warp == 0) {
    // ===================================================== producer
    if (lane == 0 && n_blk > 0) {
      int k_issued = 0, v_issued = 0;
      bool ok = true;
      mbar_arrive_expect_tx(&ctl->q_full, 2 * C::kTileBytes);
#pragma unroll
      for (int c = 0; c < C::kNChunk; ++c) {
        tma_load_4d(sQ + c * (C::kTile * 128), &tmQ, &ctl->q_full, c * 64, q0, h, b);
        tma_load_4d(sDO + c * (C::kTile * 128), &tmDO, &ctl->q_full, c * 64, q0, h, b);
      }
      for (int j = 0; j < n_blk && ok; ++j) {
        const int sk = j % C::kQKStages, uk = j / C::kQKStages;
        const int sv = j % C::kStages, uv = j / C::kStages;
        ok = wait_bounded(&ctl->k_empty[sk], (uk & 1) ^ 1, abort_flag, p.status, p.timeout_cycles);
        if (!ok) break;
        mbar_arrive_expect_tx(&ctl->k_full[sk], C::kTileBytes);
#pragma unroll
        for (int c = 0; c < C::kNChunk; ++c)
          tma_load_4d(sK + sk * C::kTileBytes + c * (C::kTile * 128), &tmK, &ctl->k_full[sk], c * 64, (jb0 + j) * C::kTile,
                      kvh, b);
        ++k_issued;
        ok = wait_bounded(&ctl->v_empty[sv], (uv & 1) ^ 1, abort_flag, p.status, p.timeout_cycles);
        if (!ok) break;
        mbar_arrive_expect_tx(&ctl->v_full[sv], C::kTileBytes);
#pragma unroll
        for (int c = 0; c < C::kNChunk; ++c)
          tma_load_4d(sV + sv * C::kTileBytes + c * (C::kTile * 128), &tmV, &ctl->v_full[sv], c * 64, (jb0 + j) * C::kTile,
                      kvh, b);
        ++v_issued;
      }
      if (*abort_flag) {
        wait_bounded(&ctl->q_full, 0, abort_flag, p.status, kDrainCycles, false);
        for (int it = max(0, k_issued - C::kQKStages); it < k_issued; ++it)
          wait_bounded(&ctl->k_full[it % C::kQKStages], (it / C::kQKStages) & 1, abort_flag, p.status, kDrainCycles,
                       false);
        for (int it = max(0, v_issued - C::kStages); it < v_issued; ++it)
          wait_bounded(&ctl->v_full[it % C::kStages], (it / C::kStages) & 1, abort_flag, p.status, kDrainCycles,
                       false);
      }
    }
  } else if (warp == 1) {
    // ===================================================== MMA issuer
    if (lane == 0 && n_blk > 0) {
      constexpr uint32_t idS = make_idesc_fmt(C::kFmt, 128, 128, false, false);
      constexpr uint32_t idAcc = make_idesc_fmt(C::kFmt, 128, C::kD, false, true);
      const uint64_t dKk = make_sdesc_sw128(smem_u32(sK), 16, 1024);
      const uint64_t dVk = make_sdesc_sw128(smem_u32(sV), 16, 1024);
      const uint64_t dKmn = make_sdesc_sw128(smem_u32(sK), C::kTile * 128, 1024);
      const uint32_t hi = (uint32_t)(dKk >> 32), hi_mn = (uint32_t)(dKmn >> 32);
      const uint32_t slot = C::kTileBytes >> 4;
      // S = Q K_j^T and dP = dO V_j^T with Q and dO in TMEM
      auto issue_s = [&](int s) {
        bwd_mma_tmem_kmajor<C>(tmem + C::kColS, tmem + C::kColQT, (uint32_t)dKk + s * slot, hi, idS);
      };
      // dP_j goes to buffer j % 2 (kColDP or kColDP2) where there are two
      auto dp_col = [](int j) { return (uint32_t)((C::kDP2 && (j & 1)) ? C::kColDP2 : C::kColDP); };
      auto issue_dp = [&](int s, int j) {
        bwd_mma_tmem_kmajor<C>(tmem + dp_col(j), tmem + C::kColDOT, (uint32_t)dVk + s * slot, hi, idS);
      };
      bool ok = wait_bounded(&ctl->qt_ready, 0, abort_flag, p.status, p.timeout_cycles);
      if (ok) ok = wait_bounded(&ctl->k_full[0], 0, abort_flag, p.status, p.timeout_cycles);
      if (ok) {
        tc_fence_after();
        issue_s(0);
        mma_commit(&ctl->s_full);
        ok = wait_bounded(&ctl->v_full[0], 0, abort_flag, p.status, p.timeout_cycles);
      }
      if (ok) {
        tc_fence_after();
        issue_dp(0, 0);
        mma_commit(&ctl->dp_full[0]);
        mma_commit(&ctl->v_empty[0]);
      }
      // Tensor-core order per block: S_{j+1}, dP_{j+1}, dQ_j with two dP
      // buffers (dP_{j+1} overwrites the buffer of dS_{j-1}, which dQ_{j-1},
      // issued before it, has read); S_{j+1}, dQ_j, dP_{j+1} with one.
      for (int j = 0; j < n_blk && ok; ++j) {
        const int s = j % C::kQKStages;  // K slot of block j
        const int sk1 = (j + 1) % C::kQKStages, uk1 = (j + 1) / C::kQKStages;
        const int sv1 = (j + 1) % C::kStages, uv1 = (j + 1) / C::kStages;
        const bool more = j + 1 < n_blk;
        ok = wait_bounded(&ctl->s_free, j & 1, abort_flag, p.status, p.timeout_cycles);
        if (!ok) break;
        auto next_dp = [&]() {
          ok = wait_bounded(&ctl->v_full[sv1], uv1 & 1, abort_flag, p.status, p.timeout_cycles);
          if (!ok) return;
          tc_fence_after();
          issue_dp(sv1, j + 1);
          mma_commit(&ctl->dp_full[C::kDP2 ? (j + 1) & 1 : 0]);
          mma_commit(&ctl->v_empty[sv1]);
        };
        if (more) {
          ok = wait_bounded(&ctl->k_full[sk1], uk1 & 1, abort_flag, p.status, p.timeout_cycles);
          if (!ok) break;
          tc_fence_after();
          issue_s(sk1);
          mma_commit(&ctl->s_full);
          if constexpr (C::kDP2) {
            next_dp();
            if (!ok) break;
          }
        }
        const int x = C::kDP2 ? j & 1 : 0, par = C::kDP2 ? (j >> 1) & 1 : j & 1;
        ok = wait_bounded(&ctl->ds_ready[x], par, abort_flag, p.status, p.timeout_cycles);
        if (!ok) break;
        tc_fence_after();
        // dQ += dS K_j (dS: bf16 pairs over dP_j's columns; K_j read MN-major)
        bwd_mma_tmem_a<C>(tmem + C::kColAcc0, tmem + dp_col(j), (uint32_t)dKmn + s * slot, hi_mn, idAcc,
                          j > 0 ? 1u : 0u);
        mma_commit(&ctl->k_empty[s]);
        if constexpr (!C::kDP2) {
          if (more) {
            next_dp();
            if (!ok) break;
          }
        }
      }
      if (ok) mma_commit(&ctl->done);
      mma_commit(&ctl->drain);
      wait_bounded(&ctl->drain, 0, abort_flag, p.status, kDrainCycles, false);
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ===================================================== elementwise warpgroup: thread = query row
    const int tl = threadIdx.x - 128;
    const int i = q0 + tl;
    const uint32_t lane_addr = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_addr + C::kColS;
    const uint32_t tDP = tmem + lane_addr + C::kColDP;
    const uint32_t tDP2 = tmem + lane_addr + C::kColDP2;
    const float sl = p.scale_log2;
    const long long rowi = ((long long)b * p.Hq + h) * p.qL + (i < p.qL ? i : 0);
    float l2 = __int_as_float(0x7f800000), di = 0.0f;
    if (i < p.qL) {
      const float L = __ldg(p.lse + rowi);
      if (L != -INFINITY) l2 = L * kLog2e;
      di = p.dvec[rowi];
    }
    // The forward's mask on this row: keep bits of a 128-key block (16 bytes,
    // fetched a block ahead into registers) or the additive row (fetched a
    // block ahead into L2, then loaded into registers before S_j lands).
    auto rbits_at = [&](int kb) {
      return reinterpret_cast<const uint4*>(p.mask_rbits + (((long long)b * p.Hq + h) * p.qL + i) * p.mask_rbits_ld +
                                            kb / 32);
    };
    auto mrow_at = [&](int kb) {
      return static_cast<const uint16_t*>(p.mask) + (long long)b * p.mask_sb + (long long)h * p.mask_sh +
             (long long)i * p.mask_ss + kb;
    };
    uint4 rb_next = make_uint4(0u, 0u, 0u, 0u);
    if constexpr (C::kMask) {
      if (i < p.qL && n_blk > 0) {
        if constexpr (C::kMaskKind == 1)
          rb_next = __ldg(rbits_at(jb0 * C::kTile));
        else
          prefetch_row_l2(mrow_at(jb0 * C::kTile), 2 * min(128, p.kL - jb0 * C::kTile));
      }
    }
    bool ok = true;
    if (n_blk > 0) {  // this row of Q and of dO into TMEM, once the tiles have landed
      ok = warp_wait(&ctl->q_full, 0, abort_flag, p.status, p.timeout_cycles);
      if (ok) {
        bwd_row_to_tmem<C>(sQ, tl, tmem + lane_addr + C::kColQT);
        bwd_row_to_tmem<C>(sDO, tl, tmem + lane_addr + C::kColDOT);
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&ctl->qt_ready);
      }
    }
    for (int j = 0; j < n_blk && ok; ++j) {
      const int kbase = (jb0 + j) * C::kTile;
      // Dropout: this row's keep bits of block j (bit x of word q: key
      // kbase + 32 q + x), loaded while S_j is computed.
      uint32_t kw[4] = {0u, 0u, 0u, 0u};
      if constexpr (C::kDrop) {
        if (i < p.qL) {
          const uint4 k4 = __ldg(reinterpret_cast<const uint4*>(p.keep_mask + rowi * p.keep_row_words + kbase / 32));
          kw[0] = k4.x;
          kw[1] = k4.y;
          kw[2] = k4.z;
          kw[3] = k4.w;
        }
      }
      // The forward's mask on this row's keys of block j, loaded before S_j lands.
      // (the dQ kernel holds an additive mask's 64 words in registers: its rows
      // lie far apart in the mask, so reading them inside the P pass would
      // expose each load's latency)
      uint32_t mw[C::kMaskKind == 2 ? 64 : 4];
      if constexpr (C::kMask) {
        if (i < p.qL) {
          const bool more = j + 1 < n_blk;
          if constexpr (C::kMaskKind == 1) {  // keep bits of block j's 128 keys
            mw[0] = rb_next.x;
            mw[1] = rb_next.y;
            mw[2] = rb_next.z;
            mw[3] = rb_next.w;
            if (more) rb_next = __ldg(rbits_at(kbase + C::kTile));
          } else {
            bwd_load_additive128(mw, mrow_at(kbase), p.mask_vec != 0 && kbase + 128 <= p.kL, min(128, p.kL - kbase));
            if (more) prefetch_row_l2(mrow_at(kbase + C::kTile), 2 * min(128, p.kL - kbase - C::kTile));
          }
        }
      }
      ok = warp_wait(&ctl->s_full, j & 1, abort_flag, p.status, p.timeout_cycles);
      if (!ok) break;
      tc_fence_after();
      float pr[128];
      tmem_ld128(tS, pr);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl->s_free);
      // P = 2^(s * scale * log2e - L2_i) for keys below the causal and kL limits
      // (and, with the features, from the window's first key on).
      int lim = p.kL - kbase, lo = -(1 << 30);
      if constexpr (C::kFeat) {
        if (p.causal) lim = min(lim, i + p.q_offset + 1 - kbase);
        if (p.window > 0) lo = i + p.q_offset - p.window + 1 - kbase;
      } else {
        if (p.causal) lim = min(lim, i + 1 - kbase);
      }
      float sq = sl;
      if constexpr (C::kCap) {
        if (p.softcap_on) {  // base-2 capped score, as the forward computes it
          const float kin = p.softcap_kin, cout = p.softcap_out;
#pragma unroll
          for (int c = 0; c < 128; ++c) pr[c] = fmaf(-2.0f * cout, rcp_approx(ex2(pr[c] * kin) + 1.0f), cout);
          sq = 1.0f;
        }
      }
      if (C::kMask && i < p.qL) {
        if constexpr (C::kMaskKind == 2)
          bwd_p_additive_regs<C>(pr, sq, [&](int) { return l2; }, mw, lo, lim);
        else
          bwd_p_keepbits(pr, sq, [&](int) { return l2; }, mw, lo, lim);
      } else {
        uint32_t aw[4];
        if constexpr (C::kFeat) allowed_words(aw, aw, false, lo, lim);
#pragma unroll
        for (int c = 0; c < 128; c += 2) {
          float x0, x1;
          ffma2(x0, x1, pr[c], pr[c + 1], sq, sq, -l2, -l2);
          if constexpr (C::kFeat) {
            pr[c] = (aw[c >> 5] & (1u << (c & 31))) ? ex2(x0) : 0.0f;
            pr[c + 1] = (aw[c >> 5] & (2u << (c & 31))) ? ex2(x1) : 0.0f;
          } else {
            pr[c] = c < lim ? ex2(x0) : 0.0f;
            pr[c + 1] = c + 1 < lim ? ex2(x1) : 0.0f;
          }
        }
      }
      const int x = C::kDP2 ? j & 1 : 0, par = C::kDP2 ? (j >> 1) & 1 : j & 1;
      ok = warp_wait(&ctl->dp_full[x], par, abort_flag, p.status, p.timeout_cycles);
      if (!ok) break;
      tc_fence_after();
      const uint32_t tdp = x ? tDP2 : tDP;
      if constexpr (C::kDrop) {
        auto dsub = [&](int) { return di; };
        auto l2c = [&](int) { return l2; };
        auto kword = [&](int cc) { return kw[cc]; };
        if (C::kCap && p.softcap_on)
          bwd_ds_pass_drop<C, C::kCap, false>(tdp, pr, dsub, l2c, p.softcap_inv, kword, p.drop_scale);
        else
          bwd_ds_pass_drop<C, false, false>(tdp, pr, dsub, l2c, 0.0f, kword, p.drop_scale);
      } else if (C::kCap && p.softcap_on) {
        bwd_ds_pass_softcap<C>(tdp, pr, [&](int) { return di; }, [&](int) { return l2; }, p.softcap_inv);
      } else {
        bwd_ds_pass<C>(tdp, pr, [&](int) { return di; });
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl->ds_ready[x]);
    }
    if (ok) {
      const bool store = i < p.qL;
      uint16_t* dqp = static_cast<uint16_t*>(p.dq) + rowi * C::kD;
      if (n_blk == 0) {
        if (store) {
          uint4* a4 = reinterpret_cast<uint4*>(dqp);
          for (int u = 0; u < C::kD / 8; ++u) a4[u] = make_uint4(0, 0, 0, 0);
        }
      } else {
        ok = warp_wait(&ctl->done, 0, abort_flag, p.status, p.timeout_cycles);
        if (ok) {
          tc_fence_after();
          if constexpr (C::kMaskKind == 2) {
            bwd_store_row<C>(tmem + lane_addr + C::kColAcc0, p.scale, dqp, store);
          } else {  // staged in the K ring (every load of it consumed)
            constexpr int kSlot = (C::kD / 64) * 32 * 128;
            bwd_store_tile_tma<C>(tmem + lane_addr + C::kColAcc0, p.scale, sK + (warp & 3) * kSlot, &tmDQ, 0,
                                  q0 + 32 * (warp & 3), p.qL, h, b, lane);
            if (lane == 0) tma_store_wait0();
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

}  // namespace fa
