// fa_bwd256_kernel.cuh -- the FA-2 backward at head dim 256 (bf16 or fp16 I/O;
// causal or not, GQA): the products of fa_bwd_kernel.cuh on smaller tiles.
//
// At D = 256 a 128 x 256 tile takes 64 KB of shared memory and a 128 x 256
// fp32 accumulator 256 TMEM columns, so the D <= 128 kernels' tiling does not
// fit (mlx-native "ops/flash_attn_train.rs", "Phase 2 -- FA-2 backward
// kernel", ships a D = 256 variant of the same backward):
//  - dK/dV: two CTAs per 128-key tile of one (b, kvh), each owning half of D
//    for dK and dV (128 accumulator columns each).  Both compute the full
//    S^T = K Q^T and dP^T = V dO^T (K and V resident, 64 KB each), with the
//    queries streamed in 64-row steps (Q ring of 2, dO ring of 1, 32 KB a
//    tile); TMEM: S^T 64 + dP^T 64 + dV/2 128 + dK/2 128 columns.
//  - dQ: one CTA per 128-row query tile (Q and dO resident) with the keys in
//    64-key blocks (K ring of 2, V ring of 1); TMEM: S 64 + two dP buffers of
//    64 + dQ 256 columns.
// Warp roles, barrier protocol, issue order, bounded waits and the
// element-wise passes are those of fa_bwd_kernel.cuh with these tile sizes.
#pragma once

#include "fa_bwd_kernel.cuh"

namespace fa {

template <bool kF16_>
struct Bwd256Cfg {
  static constexpr int kD = 256;
  static constexpr bool kF16 = kF16_;
  static constexpr uint32_t kFmt = kF16 ? kFmtF16 : kFmtBf16;
  static constexpr CUtensorMapDataType kTmaType =
      kF16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  static constexpr int kNChunk = kD / 64;  // 128-byte column blocks of a row
  static constexpr int kKStep = 16;
  static constexpr int kThreads = 256;
  static constexpr uint32_t kTmemCols = 512;
  // dK / dV kernel
  static constexpr int kKT = 128;                              // keys per CTA (TMEM lanes)
  static constexpr int kQS = 64;                               // queries per step
  static constexpr int kHalfD = kD / 2;                        // dK, dV columns per CTA
  static constexpr uint32_t kKVBytes = kKT * kD * 2;           // 64 KB
  static constexpr uint32_t kQSBytes = kQS * kD * 2;           // 32 KB
  static constexpr int kQStages = 2, kDOStages = 1;
  static constexpr uint32_t kKVOffQ = 2 * kKVBytes;
  static constexpr uint32_t kKVOffDO = kKVOffQ + kQStages * kQSBytes;
  static constexpr uint32_t kKVOffLD = kKVOffDO + kDOStages * kQSBytes;  // per Q stage: 64 L2, 64 D values
  static constexpr uint32_t kKVOffBar = kKVOffLD + kQStages * 2 * kQS * 4;
  static constexpr uint32_t kKVSmem = 1024 + kKVOffBar + 512;
  static constexpr int kColST = 0, kColDPT = 64, kColDV = 128, kColDK = 128 + kHalfD;
  // dQ kernel
  static constexpr int kQT = 128;                              // queries per CTA
  static constexpr int kKB = 64;                               // keys per block
  static constexpr uint32_t kQTBytes = kQT * kD * 2;           // 64 KB
  static constexpr uint32_t kKBBytes = kKB * kD * 2;           // 32 KB
  static constexpr int kKStages = 2, kVStages = 1;
  static constexpr uint32_t kQOffK = 2 * kQTBytes;
  static constexpr uint32_t kQOffV = kQOffK + kKStages * kKBBytes;
  static constexpr uint32_t kQOffBar = kQOffV + kVStages * kKBBytes;
  static constexpr uint32_t kQSmem = 1024 + kQOffBar + 512;
  static constexpr int kColS = 0, kColDP = 64, kColDP2 = 128, kColDQ = 256;
  static_assert(kKVSmem <= 232448 && kQSmem <= 232448, "shared memory overflow");
  static_assert(kColDK + kHalfD <= 512 && kColDQ + kD <= 512, "TMEM overflow");
  // The epilogues stage their gradients in rings the finished MMAs no longer read.
  static_assert(kQStages * kQSBytes >= kKT * kHalfD * 2 && kDOStages * kQSBytes >= kKT * kHalfD * 2 &&
                    kKStages * kKBBytes >= kQT * kD * 2,
                "epilogue staging space");
};

struct Bwd256KVCtrl {
  uint64_t kv_full;
  uint64_t q_full[2], q_empty[2], do_full, do_empty, ld_full[2], ld_empty[2];
  uint64_t s_full, dp_full, p_ready, ds_ready, done, drain;
  uint32_t tmem_base;
  int abort;
};
struct Bwd256QCtrl {
  uint64_t q_full;
  uint64_t k_full[2], k_empty[2], v_full, v_empty;
  uint64_t s_full, s_free, dp_full[2], ds_ready[2], done, drain;
  uint32_t tmem_base;
  int abort;
};
static_assert(sizeof(Bwd256KVCtrl) <= 512 && sizeof(Bwd256QCtrl) <= 512, "barrier block overflow");

// dst (+)= A[128 rows x 256] * B[kBRows rows x 256]^T, both K-major 128-byte
// swizzled tiles of 64-column blocks (A's blocks 128 rows apart, B's kBRows).
template <class C, int kBRows>
__device__ __forceinline__ void bwd256_kmajor(uint32_t dst, uint32_t a_lo, uint32_t a_hi, uint32_t b_lo,
                                              uint32_t b_hi, uint32_t idesc) {
  constexpr int kACol = (128 * 128) >> 4, kBCol = (kBRows * 128) >> 4;
  mma_ss_lh<false, 0>(dst, a_lo, a_hi, b_lo, b_hi, idesc, 0u);
#pragma unroll
  for (int kk = 1; kk < C::kD / C::kKStep; ++kk)
    mma_ss_lh<false, 1>(dst, a_lo + (kk / 4) * kACol + (kk % 4) * 2, a_hi, b_lo + (kk / 4) * kBCol + (kk % 4) * 2,
                        b_hi, idesc, 1u);
}

// dst (+)= A[128 x kK] (16-bit pairs in TMEM) * B[kK rows x N] with B an
// MN-major tile (rows = the MMA's K, 128 bytes of N per row and column block).
template <class C, int kK>
__device__ __forceinline__ void bwd256_tmem_a(uint32_t dst, uint32_t a_tmem, uint32_t b_lo, uint32_t b_hi,
                                              uint32_t idesc, uint32_t acc) {
  mma_ts_lh<false, 0>(dst, a_tmem, b_lo, b_hi, idesc, acc);
#pragma unroll
  for (int kk = 1; kk < kK / C::kKStep; ++kk)
    mma_ts_lh<false, 1>(dst, a_tmem + kk * 8, b_lo + ((kk * C::kKStep * 128) >> 4), b_hi, idesc, 1u);
}

// dS = P (dP - d) over 64 columns: read 32 fp32 dP columns, write 16 columns of
// 16-bit pairs over the part already read.
template <class C, class F>
__device__ __forceinline__ void bwd256_ds_pass(uint32_t tdp, const float (&p)[64], F dsub) {
#pragma unroll
  for (int cc = 0; cc < 2; ++cc) {
    uint32_t rr[32];
    tmem_ld32(tdp + cc * 32, rr);
    tmem_wait_ld();
    reg_fence(rr);
    uint32_t pk[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      const int c0 = cc * 32 + 2 * e;
      pk[e] = pack16x2<C>(p[c0] * (__uint_as_float(rr[2 * e]) - dsub(c0)),
                          p[c0 + 1] * (__uint_as_float(rr[2 * e + 1]) - dsub(c0 + 1)));
    }
    tmem_st16(tdp + cc * 16, pk);
  }
}

// ---------------------------------------------------------------- dK / dV

// Grid: 2 CTAs (D halves) per (128-key tile, kvh, b), heavy (early) key tiles first.
template <class C>
__global__ void __launch_bounds__(C::kThreads, 1)
    fa_bwd256_dkdv_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                          const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
                          const __grid_constant__ CUtensorMap tmDK, const __grid_constant__ CUtensorMap tmDV,
                          const BwdParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sK = smem;
  uint8_t* sV = smem + C::kKVBytes;
  uint8_t* sQ = smem + C::kKVOffQ;
  uint8_t* sDO = smem + C::kKVOffDO;
  float* sLD = reinterpret_cast<float*>(smem + C::kKVOffLD);
  Bwd256KVCtrl* ctl = reinterpret_cast<Bwd256KVCtrl*>(smem + C::kKVOffBar);
  volatile int* abort_flag = &ctl->abort;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int half = blockIdx.x & 1;  // this CTA's half of D for dK and dV
  const int unit = blockIdx.x >> 1;
  const int per_kt = p.Hkv * p.B;
  const int kt = unit / per_kt;
  const int rem = unit - kt * per_kt;
  const int b = rem / p.Hkv, kvh = rem - b * p.Hkv;
  const int k0 = kt * C::kKT;
  const int n_qs = (p.qL + C::kQS - 1) / C::kQS;      // 64-row query steps per head
  const int qs0 = p.causal ? min(k0 / C::kQS, n_qs) : 0;  // causal: rows from k0 on
  const int per_head = max(0, n_qs - qs0);
  const int n_steps = p.group * per_head;

  if (threadIdx.x == 0) {
    mbar_init(&ctl->kv_full, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&ctl->q_full[s], 1);
      mbar_init(&ctl->q_empty[s], 1);
      mbar_init(&ctl->ld_full[s], 32);  // every producer lane stages its 2 queries
      mbar_init(&ctl->ld_empty[s], 4);  // one arrival per elementwise warp
    }
    mbar_init(&ctl->do_full, 1);
    mbar_init(&ctl->do_empty, 1);
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
    q0 = (qs0 + (i - r * per_head)) * C::kQS;
  };

  if (warp == 0) {
    // ===================================================== producer: TMA + L, D staging
    int q_issued = 0, do_issued = 0;
    bool ok = true;
    if (lane == 0 && n_steps > 0) {
      mbar_arrive_expect_tx(&ctl->kv_full, 2 * C::kKVBytes);
#pragma unroll
      for (int c = 0; c < C::kNChunk; ++c) {
        tma_load_4d(sK + c * (C::kKT * 128), &tmK, &ctl->kv_full, c * 64, k0, kvh, b);
        tma_load_4d(sV + c * (C::kKT * 128), &tmV, &ctl->kv_full, c * 64, k0, kvh, b);
      }
    }
    for (int i = 0; i < n_steps && ok; ++i) {
      int h, q0;
      step_of(i, h, q0);
      const int s = i % C::kQStages, use = i / C::kQStages;
      if (lane == 0) {
        ok = wait_bounded(&ctl->q_empty[s], (use & 1) ^ 1, abort_flag, p.status, p.timeout_cycles);
        if (ok) {
          mbar_arrive_expect_tx(&ctl->q_full[s], C::kQSBytes);
#pragma unroll
          for (int c = 0; c < C::kNChunk; ++c)
            tma_load_4d(sQ + s * C::kQSBytes + c * (C::kQS * 128), &tmQ, &ctl->q_full[s], c * 64, q0, h, b);
          ++q_issued;
          ok = wait_bounded(&ctl->do_empty, (i & 1) ^ 1, abort_flag, p.status, p.timeout_cycles);
        }
        if (ok) {
          mbar_arrive_expect_tx(&ctl->do_full, C::kQSBytes);
#pragma unroll
          for (int c = 0; c < C::kNChunk; ++c)
            tma_load_4d(sDO + c * (C::kQS * 128), &tmDO, &ctl->do_full, c * 64, q0, h, b);
          ++do_issued;
        }
      }
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      if (!ok) break;
      // L2 = L * log2(e) (+inf where the query is past qL or its row had no
      // allowed key, so P = 0 there) and D for the step's 64 queries.
      ok = warp_wait(&ctl->ld_empty[s], (use & 1) ^ 1, abort_flag, p.status, p.timeout_cycles);
      if (!ok) break;
      float* l2s = sLD + s * 2 * C::kQS;
      const long long base = ((long long)b * p.Hq + h) * p.qL;
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int c = lane * 2 + e, iq = q0 + c;
        float l2 = __int_as_float(0x7f800000), dv = 0.0f;
        if (iq < p.qL) {
          const float L = __ldg(p.lse + base + iq);
          if (L != -INFINITY) l2 = L * kLog2e;
          dv = p.dvec[base + iq];
        }
        l2s[c] = l2;
        l2s[C::kQS + c] = dv;
      }
      mbar_arrive(&ctl->ld_full[s]);
    }
    if (lane == 0 && *abort_flag) {
      if (n_steps > 0) wait_bounded(&ctl->kv_full, 0, abort_flag, p.status, kDrainCycles, false);
      for (int it = max(0, q_issued - C::kQStages); it < q_issued; ++it)
        wait_bounded(&ctl->q_full[it % C::kQStages], (it / C::kQStages) & 1, abort_flag, p.status, kDrainCycles,
                     false);
      if (do_issued > 0) wait_bounded(&ctl->do_full, (do_issued - 1) & 1, abort_flag, p.status, kDrainCycles, false);
    }
  } else if (warp == 1) {
    // ===================================================== MMA issuer
    if (lane == 0 && n_steps > 0) {
      constexpr uint32_t idS = make_idesc_fmt(C::kFmt, 128, C::kQS, false, false);      // K-major A and B
      constexpr uint32_t idAcc = make_idesc_fmt(C::kFmt, 128, C::kHalfD, false, true);  // B MN-major
      const uint64_t dK = make_sdesc_sw128(smem_u32(sK), 16, 1024);
      const uint64_t dV = make_sdesc_sw128(smem_u32(sV), 16, 1024);
      const uint64_t dQk = make_sdesc_sw128(smem_u32(sQ), 16, 1024);
      const uint64_t dOk = make_sdesc_sw128(smem_u32(sDO), 16, 1024);
      // MN-major views of this CTA's half of the Q and dO columns (two 64-column blocks, LBO apart)
      const uint64_t dQmn = make_sdesc_sw128(smem_u32(sQ + half * 2 * (C::kQS * 128)), C::kQS * 128, 1024);
      const uint64_t dOmn = make_sdesc_sw128(smem_u32(sDO + half * 2 * (C::kQS * 128)), C::kQS * 128, 1024);
      const uint32_t hi = (uint32_t)(dK >> 32), hi_mn = (uint32_t)(dQmn >> 32);
      const uint32_t slot = C::kQSBytes >> 4;
      auto issue_s = [&](int s) {  // S^T = K Q_s^T
        bwd256_kmajor<C, C::kQS>(tmem + C::kColST, (uint32_t)dK, hi, (uint32_t)dQk + s * slot, hi, idS);
      };
      auto issue_dp = [&]() {  // dP^T = V dO^T
        bwd256_kmajor<C, C::kQS>(tmem + C::kColDPT, (uint32_t)dV, hi, (uint32_t)dOk, hi, idS);
      };
      bool ok = wait_bounded(&ctl->kv_full, 0, abort_flag, p.status, p.timeout_cycles);
      if (ok) ok = wait_bounded(&ctl->q_full[0], 0, abort_flag, p.status, p.timeout_cycles);
      if (ok) {
        tc_fence_after();
        issue_s(0);
        mma_commit(&ctl->s_full);
        ok = wait_bounded(&ctl->do_full, 0, abort_flag, p.status, p.timeout_cycles);
      }
      if (ok) {
        tc_fence_after();
        issue_dp();
        mma_commit(&ctl->dp_full);
      }
      // Order per step: dV_i, S^T_{i+1}, dK_i, dP^T_{i+1} (dO_{i+1} lands in the slot dV_i freed).
      for (int i = 0; i < n_steps && ok; ++i) {
        const int s = i % C::kQStages;
        const int s1 = (i + 1) % C::kQStages, use1 = (i + 1) / C::kQStages;
        const bool more = i + 1 < n_steps;
        ok = wait_bounded(&ctl->p_ready, i & 1, abort_flag, p.status, p.timeout_cycles);
        if (!ok) break;
        tc_fence_after();
        // dV[:, half] += P^T dO_i[:, half] (P^T: 16-bit pairs over the S^T columns)
        bwd256_tmem_a<C, C::kQS>(tmem + C::kColDV, tmem + C::kColST, (uint32_t)dOmn, hi_mn, idAcc, i > 0 ? 1u : 0u);
        mma_commit(&ctl->do_empty);
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
        // dK[:, half] += dS^T Q_i[:, half] (dS^T: 16-bit pairs over the dP^T columns)
        bwd256_tmem_a<C, C::kQS>(tmem + C::kColDK, tmem + C::kColDPT, (uint32_t)dQmn + s * slot, hi_mn, idAcc,
                                 i > 0 ? 1u : 0u);
        mma_commit(&ctl->q_empty[s]);
        if (more) {
          ok = wait_bounded(&ctl->do_full, (i + 1) & 1, abort_flag, p.status, p.timeout_cycles);
          if (!ok) break;
          tc_fence_after();
          issue_dp();
          mma_commit(&ctl->dp_full);
        }
      }
      if (ok) mma_commit(&ctl->done);
      mma_commit(&ctl->drain);
      wait_bounded(&ctl->drain, 0, abort_flag, p.status, kDrainCycles, false);
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ===================================================== elementwise warpgroup: thread = key row
    const int tl = threadIdx.x - 128;
    const int j = k0 + tl;
    const uint32_t lane_addr = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_addr + C::kColST;
    const uint32_t tDP = tmem + lane_addr + C::kColDPT;
    const float sl = p.scale_log2;
    bool ok = true;
    for (int i = 0; i < n_steps && ok; ++i) {
      int h, q0;
      step_of(i, h, q0);
      const int s = i % C::kQStages, use = i / C::kQStages;
      const float* l2s = sLD + s * 2 * C::kQS;
      ok = warp_wait(&ctl->ld_full[s], use & 1, abort_flag, p.status, p.timeout_cycles);
      if (!ok) break;
      ok = warp_wait(&ctl->s_full, i & 1, abort_flag, p.status, p.timeout_cycles);
      if (!ok) break;
      tc_fence_after();
      float pr[64];
      tmem_ld64f(tS, pr);
      // P^T_{j,c} = 2^(s * scale * log2e - L2_c); queries c < j - q0 are causally masked,
      // and a key row past kL gets no probability at all.
      int lim = p.causal ? j - q0 : 0;
      if (j >= p.kL) lim = C::kQS;
#pragma unroll
      for (int c = 0; c < 64; c += 2) {
        float x0, x1;
        ffma2(x0, x1, pr[c], pr[c + 1], sl, sl, -l2s[c], -l2s[c + 1]);
        pr[c] = c < lim ? 0.0f : ex2(x0);
        pr[c + 1] = c + 1 < lim ? 0.0f : ex2(x1);
      }
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) pk[e] = pack16x2<C>(pr[cc * 32 + 2 * e], pr[cc * 32 + 2 * e + 1]);
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
      bwd256_ds_pass<C>(tDP, pr, [&](int c) { return l2s[C::kQS + c]; });
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&ctl->ds_ready);
        mbar_arrive(&ctl->ld_empty[s]);
      }
    }
    // ---- epilogue: this CTA's half of dV and scale * dK rows (key j)
    if (ok) {
      const bool store = j < p.kL;
      const long long row = ((long long)b * p.Hkv + kvh) * p.kL + (store ? j : 0);
      uint16_t* dvp = static_cast<uint16_t*>(p.dv) + row * C::kD + half * C::kHalfD;
      uint16_t* dkp = static_cast<uint16_t*>(p.dk) + row * C::kD + half * C::kHalfD;
      if (n_steps == 0) {  // no query sees these keys: zero gradients
        if (store) {
          uint4* a4 = reinterpret_cast<uint4*>(dvp);
          uint4* b4 = reinterpret_cast<uint4*>(dkp);
          for (int u = 0; u < C::kHalfD / 8; ++u) a4[u] = b4[u] = make_uint4(0, 0, 0, 0);
        }
      } else {
        ok = warp_wait(&ctl->done, 0, abort_flag, p.status, p.timeout_cycles);
        if (ok) {
          tc_fence_after();
          // this CTA's column half of dV and dK, staged in the Q and dO rings (every load consumed)
          constexpr int kSlot = (C::kHalfD / 64) * 32 * 128;
          const int row0 = k0 + 32 * (warp & 3);
          bwd_store_tile_tma<C, C::kHalfD>(tmem + lane_addr + C::kColDV, 1.0f, sQ + (warp & 3) * kSlot, &tmDV,
                                           half * C::kHalfD, row0, p.kL, kvh, b, lane);
          bwd_store_tile_tma<C, C::kHalfD>(tmem + lane_addr + C::kColDK, p.scale, sDO + (warp & 3) * kSlot, &tmDK,
                                           half * C::kHalfD, row0, p.kL, kvh, b, lane);
          if (lane == 0) tma_store_wait0();
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

// One CTA per (128-row query tile, h, b), heavy (late, causal) tiles first;
// keys in 64-key blocks: S = Q K_j^T, dP = dO V_j^T, dS = P (dP - D), dQ += dS K_j.
template <class C>
__global__ void __launch_bounds__(C::kThreads, 1)
    fa_bwd256_dq_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                        const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
                        const __grid_constant__ CUtensorMap tmDQ, const BwdParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem;
  uint8_t* sDO = smem + C::kQTBytes;
  uint8_t* sK = smem + C::kQOffK;
  uint8_t* sV = smem + C::kQOffV;
  Bwd256QCtrl* ctl = reinterpret_cast<Bwd256QCtrl*>(smem + C::kQOffBar);
  volatile int* abort_flag = &ctl->abort;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_qt = (p.qL + C::kQT - 1) / C::kQT;
  const int per_qt = p.Hq * p.B;
  const int qt_rev = blockIdx.x / per_qt;
  const int rem = blockIdx.x - qt_rev * per_qt;
  const int b = rem / p.Hq, h = rem - b * p.Hq;
  const int qt = p.causal ? n_qt - 1 - qt_rev : qt_rev;
  const int q0 = qt * C::kQT;
  const int kvh = h / p.group;
  const int last = min(q0 + C::kQT, p.qL) - 1;
  const int kv_end = p.causal ? min(p.kL, last + 1) : p.kL;
  const int n_blk = (kv_end + C::kKB - 1) / C::kKB;

  if (threadIdx.x == 0) {
    mbar_init(&ctl->q_full, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&ctl->k_full[s], 1);
      mbar_init(&ctl->k_empty[s], 1);
    }
    mbar_init(&ctl->v_full, 1);
    mbar_init(&ctl->v_empty, 1);
    mbar_init(&ctl->s_full, 1);
    mbar_init(&ctl->s_free, 4);
    for (int d = 0; d < 2; ++d) {
      mbar_init(&ctl->dp_full[d], 1);
      mbar_init(&ctl->ds_ready[d], 4);
    }
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
      mbar_arrive_expect_tx(&ctl->q_full, 2 * C::kQTBytes);
#pragma unroll
      for (int c = 0; c < C::kNChunk; ++c) {
        tma_load_4d(sQ + c * (C::kQT * 128), &tmQ, &ctl->q_full, c * 64, q0, h, b);
        tma_load_4d(sDO + c * (C::kQT * 128), &tmDO, &ctl->q_full, c * 64, q0, h, b);
      }
      for (int j = 0; j < n_blk && ok; ++j) {
        const int sk = j % C::kKStages, uk = j / C::kKStages;
        ok = wait_bounded(&ctl->k_empty[sk], (uk & 1) ^ 1, abort_flag, p.status, p.timeout_cycles);
        if (!ok) break;
        mbar_arrive_expect_tx(&ctl->k_full[sk], C::kKBBytes);
#pragma unroll
        for (int c = 0; c < C::kNChunk; ++c)
          tma_load_4d(sK + sk * C::kKBBytes + c * (C::kKB * 128), &tmK, &ctl->k_full[sk], c * 64, j * C::kKB, kvh, b);
        ++k_issued;
        ok = wait_bounded(&ctl->v_empty, (j & 1) ^ 1, abort_flag, p.status, p.timeout_cycles);
        if (!ok) break;
        mbar_arrive_expect_tx(&ctl->v_full, C::kKBBytes);
#pragma unroll
        for (int c = 0; c < C::kNChunk; ++c)
          tma_load_4d(sV + c * (C::kKB * 128), &tmV, &ctl->v_full, c * 64, j * C::kKB, kvh, b);
        ++v_issued;
      }
      if (*abort_flag) {
        wait_bounded(&ctl->q_full, 0, abort_flag, p.status, kDrainCycles, false);
        for (int it = max(0, k_issued - C::kKStages); it < k_issued; ++it)
          wait_bounded(&ctl->k_full[it % C::kKStages], (it / C::kKStages) & 1, abort_flag, p.status, kDrainCycles,
                       false);
        if (v_issued > 0) wait_bounded(&ctl->v_full, (v_issued - 1) & 1, abort_flag, p.status, kDrainCycles, false);
      }
    }
  } else if (warp == 1) {
    // ===================================================== MMA issuer
    if (lane == 0 && n_blk > 0) {
      constexpr uint32_t idS = make_idesc_fmt(C::kFmt, 128, C::kKB, false, false);
      constexpr uint32_t idAcc = make_idesc_fmt(C::kFmt, 128, C::kD, false, true);
      const uint64_t dQ = make_sdesc_sw128(smem_u32(sQ), 16, 1024);
      const uint64_t dO = make_sdesc_sw128(smem_u32(sDO), 16, 1024);
      const uint64_t dKk = make_sdesc_sw128(smem_u32(sK), 16, 1024);
      const uint64_t dVk = make_sdesc_sw128(smem_u32(sV), 16, 1024);
      const uint64_t dKmn = make_sdesc_sw128(smem_u32(sK), C::kKB * 128, 1024);
      const uint32_t hi = (uint32_t)(dQ >> 32), hi_mn = (uint32_t)(dKmn >> 32);
      const uint32_t slot = C::kKBBytes >> 4;
      auto issue_s = [&](int s) { bwd256_kmajor<C, C::kKB>(tmem + C::kColS, (uint32_t)dQ, hi, (uint32_t)dKk + s * slot, hi, idS); };
      auto dp_col = [](int j) { return (uint32_t)((j & 1) ? C::kColDP2 : C::kColDP); };
      auto issue_dp = [&](int j) { bwd256_kmajor<C, C::kKB>(tmem + dp_col(j), (uint32_t)dO, hi, (uint32_t)dVk, hi, idS); };
      bool ok = wait_bounded(&ctl->q_full, 0, abort_flag, p.status, p.timeout_cycles);
      if (ok) ok = wait_bounded(&ctl->k_full[0], 0, abort_flag, p.status, p.timeout_cycles);
      if (ok) {
        tc_fence_after();
        issue_s(0);
        mma_commit(&ctl->s_full);
        ok = wait_bounded(&ctl->v_full, 0, abort_flag, p.status, p.timeout_cycles);
      }
      if (ok) {
        tc_fence_after();
        issue_dp(0);
        mma_commit(&ctl->dp_full[0]);
        mma_commit(&ctl->v_empty);
      }
      // Tensor-core order per block: S_{j+1}, dP_{j+1}, dQ_j.
      for (int j = 0; j < n_blk && ok; ++j) {
        const int s = j % C::kKStages;
        const int sk1 = (j + 1) % C::kKStages, uk1 = (j + 1) / C::kKStages;
        const bool more = j + 1 < n_blk;
        ok = wait_bounded(&ctl->s_free, j & 1, abort_flag, p.status, p.timeout_cycles);
        if (!ok) break;
        if (more) {
          ok = wait_bounded(&ctl->k_full[sk1], uk1 & 1, abort_flag, p.status, p.timeout_cycles);
          if (!ok) break;
          tc_fence_after();
          issue_s(sk1);
          mma_commit(&ctl->s_full);
          ok = wait_bounded(&ctl->v_full, (j + 1) & 1, abort_flag, p.status, p.timeout_cycles);
          if (!ok) break;
          tc_fence_after();
          issue_dp(j + 1);
          mma_commit(&ctl->dp_full[(j + 1) & 1]);
          mma_commit(&ctl->v_empty);
        }
        ok = wait_bounded(&ctl->ds_ready[j & 1], (j >> 1) & 1, abort_flag, p.status, p.timeout_cycles);
        if (!ok) break;
        tc_fence_after();
        // dQ += dS K_j (dS: 16-bit pairs over dP_j's columns; K_j read MN-major)
        bwd256_tmem_a<C, C::kKB>(tmem + C::kColDQ, tmem + dp_col(j), (uint32_t)dKmn + s * slot, hi_mn, idAcc,
                                 j > 0 ? 1u : 0u);
        mma_commit(&ctl->k_empty[s]);
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
    const float sl = p.scale_log2;
    const long long rowi = ((long long)b * p.Hq + h) * p.qL + (i < p.qL ? i : 0);
    float l2 = __int_as_float(0x7f800000), di = 0.0f;
    if (i < p.qL) {
      const float L = __ldg(p.lse + rowi);
      if (L != -INFINITY) l2 = L * kLog2e;
      di = p.dvec[rowi];
    }
    bool ok = true;
    for (int j = 0; j < n_blk && ok; ++j) {
      const int kbase = j * C::kKB;
      ok = warp_wait(&ctl->s_full, j & 1, abort_flag, p.status, p.timeout_cycles);
      if (!ok) break;
      tc_fence_after();
      float pr[64];
      tmem_ld64f(tS, pr);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl->s_free);
      // P = 2^(s * scale * log2e - L2_i) for keys below the causal and kL limits
      int lim = p.kL - kbase;
      if (p.causal) lim = min(lim, i + 1 - kbase);
#pragma unroll
      for (int c = 0; c < 64; c += 2) {
        float x0, x1;
        ffma2(x0, x1, pr[c], pr[c + 1], sl, sl, -l2, -l2);
        pr[c] = c < lim ? ex2(x0) : 0.0f;
        pr[c + 1] = c + 1 < lim ? ex2(x1) : 0.0f;
      }
      ok = warp_wait(&ctl->dp_full[j & 1], (j >> 1) & 1, abort_flag, p.status, p.timeout_cycles);
      if (!ok) break;
      tc_fence_after();
      bwd256_ds_pass<C>(tmem + lane_addr + ((j & 1) ? C::kColDP2 : C::kColDP), pr, [&](int) { return di; });
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl->ds_ready[j & 1]);
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
          // staged in the K ring (every load consumed)
          constexpr int kSlot = (C::kD / 64) * 32 * 128;
          bwd_store_tile_tma<C, C::kD>(tmem + lane_addr + C::kColDQ, p.scale, sK + (warp & 3) * kSlot, &tmDQ, 0,
                                       q0 + 32 * (warp & 3), p.qL, h, b, lane);
          if (lane == 0) tma_store_wait0();
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
