// fa_bwd_tf32_kernel.cuh -- the FA-2 backward for fp32 I/O on the TF32
// tensor cores (head dims 64 and 128; causal or not; GQA).
//
// Same gradients as fa_bwd_kernel.cuh.  The split follows forge
// "flash_attention_mma.metal", section "backward (MMA)": a query-parallel dQ
// kernel and separate key-parallel dV and dK kernels (dV holds K and dV, dK
// holds K, V and dK; both recompute S^T = K Q^T), which keeps every
// accumulator private to one CTA.  One kernel template serves the three roles:
//
//   role  resident (128 rows)   streamed per 64-row step       accumulates
//   dV    K                     Q, dO^T                        P^T dO
//   dK    K, V                  Q, dO, Q^T                     dS^T Q
//   dQ    Q, dO                 K, V, K^T                      dS K
//
// A tf32 MMA takes its B operand K-major only, so the accumulating products
// read transposed copies (dO^T, Q^T, K^T: [B, H, D, L rounded up to 4]) that
// the launcher's pre-pass writes, together with tf32-rounded copies of Q, K,
// V and dO in their own layout (the tensor core would otherwise drop the low
// mantissa bits).  P and dS are rounded to tf32 (nearest) before their
// products.  Each streamed operand has its own ring, so a slot is refilled as
// soon as the one product that reads it has finished.
//
// Warps: 0 loads the resident tiles and the first ring, 1 issues every MMA
// from one thread, 2 the second ring and the per-query L and D values (dV, dK),
// 3 the transposed ring; 4-7 are the elementwise warpgroup (thread = resident
// row = TMEM lane).  S and dP have two TMEM buffers each, so step j + 1's
// products run while the elementwise warps work on step j.
#pragma once

#include "fa_bwd_kernel.cuh"

namespace fa {

enum : int { kT32DV = 0, kT32DK = 1, kT32DQ = 2 };

template <int kD_, int kRole_>
struct BwdT32Cfg {
  static constexpr int kD = kD_;
  static constexpr int kRole = kRole_;
  static constexpr bool kHasDP = kRole != kT32DV;  // dP (or dP^T) and the second resident tile
  static constexpr bool kColLD = kRole != kT32DQ;  // L and D belong to the columns (queries)
  static constexpr int kRows = 128;                // resident rows = TMEM lanes
  static constexpr int kStep = 64;                 // streamed rows per step
  static constexpr int kNChunk = kD / 32;          // 128-byte column blocks of a row (32 fp32)
  static constexpr int kThreads = 256;
  static constexpr uint32_t kResBytes = kRows * kD * 4;
  static constexpr uint32_t kTBytes = kStep * kD * 4;  // a streamed tile (either layout)
  static constexpr int kNRes = kHasDP ? 2 : 1;
  static constexpr uint32_t kLDBytes = kColLD ? 2 * kStep * 4 : 0;
  static constexpr uint32_t kPerStage = (kHasDP ? 3 : 2) * kTBytes + kLDBytes;
  static constexpr uint32_t kFixed = 1024 + kNRes * kResBytes + 512;
  static constexpr int kFit = (int)((232448 - kFixed) / kPerStage);
  static constexpr int kStages = kFit > 4 ? 4 : kFit;
  // shared memory: resident tiles, then the three rings, then L / D slots, then barriers
  static constexpr uint32_t kOffT0 = kNRes * kResBytes;
  static constexpr uint32_t kOffT1 = kOffT0 + kStages * kTBytes;
  static constexpr uint32_t kOffT2 = kOffT1 + (kHasDP ? kStages * kTBytes : 0);
  static constexpr uint32_t kOffLD = kOffT2 + kStages * kTBytes;
  static constexpr uint32_t kOffBar = kOffLD + kStages * kLDBytes;
  static constexpr uint32_t kSmem = 1024 + kOffBar + 512;
  // TMEM: two S buffers, two dP buffers, the accumulator
  static constexpr int kColS = 0, kColDP = 2 * kStep, kColAcc = 4 * kStep;
  static constexpr uint32_t kTmemCols = 512;
  static_assert(kD == 64 || kD == 128, "fp32 backward head dims: 64 or 128");
  static_assert(kStages >= 1 && kSmem <= 232448, "shared memory overflow");
  static_assert(kColAcc + kD <= 512, "TMEM overflow");
  // The epilogue stages the 128-row output tile in the streamed rings (idle by then).
  static_assert(kOffLD - kOffT0 >= kRows * kD * 4, "epilogue staging space");
};

struct BwdT32Ctrl {
  uint64_t res_full;
  uint64_t t_full[3][4], t_empty[3][4];
  uint64_t ld_full[4], ld_empty[4];
  uint64_t s_full[2], dp_full[2], ready[2];
  uint64_t done, drain;
  uint32_t tmem_base;
  int abort;
};
static_assert(sizeof(BwdT32Ctrl) <= 512, "barrier block overflow");

// dst (+)= A[128 x kD] * B[64 x kD]^T, both K-major 128-byte swizzled fp32
// tiles of 32-column blocks (A's blocks 128 rows apart, B's 64).
template <class C>
__device__ __forceinline__ void t32_mma_rows(uint32_t dst, uint32_t a_lo, uint32_t hi, uint32_t b_lo, uint32_t idesc) {
  constexpr int kACol = (C::kRows * 128) >> 4, kBCol = (C::kStep * 128) >> 4;
  mma_ss_lh<true, 0>(dst, a_lo, hi, b_lo, hi, idesc, 0u);
#pragma unroll
  for (int kk = 1; kk < C::kD / 8; ++kk)
    mma_ss_lh<true, 1>(dst, a_lo + (kk / 4) * kACol + (kk % 4) * 2, hi, b_lo + (kk / 4) * kBCol + (kk % 4) * 2, hi,
                       idesc, 1u);
}

// dst (+)= A[128 x 64] (tf32 in TMEM) * B with B a transposed tile: kD rows of
// 64 values (the MMA's K) in two 32-column blocks.
template <class C>
__device__ __forceinline__ void t32_mma_acc(uint32_t dst, uint32_t a_tmem, uint32_t b_lo, uint32_t hi, uint32_t idesc,
                                            uint32_t acc) {
  constexpr int kBCol = (C::kD * 128) >> 4;
  mma_ts_lh<true, 0>(dst, a_tmem, b_lo, hi, idesc, acc);
#pragma unroll
  for (int kk = 1; kk < C::kStep / 8; ++kk)
    mma_ts_lh<true, 1>(dst, a_tmem + kk * 8, b_lo + (kk / 4) * kBCol + (kk % 4) * 2, hi, idesc, 1u);
}

// Write 64 fp32 values, rounded to tf32, to this lane's TMEM columns.
__device__ __forceinline__ void t32_store64(uint32_t taddr, const float (&x)[64]) {
#pragma unroll
  for (int cc = 0; cc < 2; ++cc) {
    uint32_t pk[32];
#pragma unroll
    for (int e = 0; e < 32; ++e) pk[e] = to_tf32(x[cc * 32 + e]);
    tmem_st32(taddr + cc * 32, pk);
  }
}

// The epilogue through TMA stores: this warp's 32 rows (its TMEM lanes) of
// the kD-column fp32 accumulator, times `mul`, staged as kD / 32 boxes of 32
// rows x 128 bytes (32 floats) with the 128-byte swizzle (row r's 16-byte piece
// k at r * 128 + (k ^ (r & 7)) * 16) in `slot` -- the streamed rings, idle once
// every MMA has finished; 1024-byte aligned -- then stored by lane 0 at rows
// row0 .. row0 + 31 of (head, batch), clipped past the extent.  One TMEM load
// wait per 64 columns.
template <class C>
__device__ __forceinline__ void t32_store_tile_tma(uint32_t tacc, float mul, uint8_t* slot, const CUtensorMap* map,
                                                   int row0, int extent, int head, int batch, int lane) {
#pragma unroll
  for (int hh = 0; hh < C::kD / 64; ++hh) {
    uint32_t rr[2][32];
    tmem_ld32(tacc + hh * 64, rr[0]);
    tmem_ld32(tacc + hh * 64 + 32, rr[1]);
    tmem_wait_ld();
    reg_fence(rr[0]);
    reg_fence(rr[1]);
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      uint8_t* box = slot + (2 * hh + q) * (32 * 128);
#pragma unroll
      for (int k = 0; k < 8; ++k)  // piece k: columns 4k .. 4k + 3 of the box
        *reinterpret_cast<float4*>(box + lane * 128 + ((k ^ (lane & 7)) << 4)) =
            make_float4(__uint_as_float(rr[q][4 * k]) * mul, __uint_as_float(rr[q][4 * k + 1]) * mul,
                        __uint_as_float(rr[q][4 * k + 2]) * mul, __uint_as_float(rr[q][4 * k + 3]) * mul);
    }
  }
  fence_proxy_async_smem();
  __syncwarp();
  if (lane == 0 && row0 < extent) {
#pragma unroll
    for (int bx = 0; bx < C::kD / 32; ++bx) tma_store_4d(map, slot + bx * (32 * 128), bx * 32, row0, head, batch);
    tma_store_commit();
  }
}

// Grid: dV, dK -- one CTA per (128-key tile, kvh, b); dQ -- one CTA per
// (128-row query tile, h, b).  Causal: heavy tiles first; else head-major.
template <class C>
__global__ void __launch_bounds__(C::kThreads, 1)
    fa_bwd_tf32_kernel(const __grid_constant__ CUtensorMap tmR0, const __grid_constant__ CUtensorMap tmR1,
                       const __grid_constant__ CUtensorMap tmT0, const __grid_constant__ CUtensorMap tmT1,
                       const __grid_constant__ CUtensorMap tmT2, const __grid_constant__ CUtensorMap tmOut,
                       const BwdParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sR0 = smem;
  uint8_t* sR1 = smem + C::kResBytes;
  uint8_t* sT[3] = {smem + C::kOffT0, smem + C::kOffT1, smem + C::kOffT2};
  float* sLD = reinterpret_cast<float*>(smem + C::kOffLD);
  BwdT32Ctrl* ctl = reinterpret_cast<BwdT32Ctrl*>(smem + C::kOffBar);
  volatile int* abort_flag = &ctl->abort;
  constexpr int kS = C::kStages;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // ---- this CTA's work: (b, resident head, resident row 0) and its steps
  int b, rh, r0, n_steps, per_head = 1, s0 = 0;
  // Causal: tile-major, heavy tiles first (the longest CTAs start first).
  // Otherwise every CTA does the same work: head-major, so the CTAs running at
  // a time share few heads and the operands they stream stay in L2.
  if constexpr (C::kRole == kT32DQ) {
    const int n_qt = (p.qL + C::kRows - 1) / C::kRows;
    const int per_qt = p.Hq * p.B;
    int qt, rem;
    if (p.causal) {
      const int qt_rev = blockIdx.x / per_qt;
      rem = blockIdx.x - qt_rev * per_qt;
      qt = n_qt - 1 - qt_rev;
    } else {
      rem = blockIdx.x / n_qt;
      qt = blockIdx.x - rem * n_qt;
    }
    b = rem / p.Hq;
    rh = rem - b * p.Hq;
    r0 = qt * C::kRows;
    const int last = min(r0 + C::kRows, p.qL) - 1;
    const int kv_end = p.causal ? min(p.kL, last + 1) : p.kL;
    n_steps = (kv_end + C::kStep - 1) / C::kStep;
  } else {
    const int per_kt = p.Hkv * p.B;
    const int n_kt = (p.kL + C::kRows - 1) / C::kRows;
    int kt, rem;
    if (p.causal) {
      kt = blockIdx.x / per_kt;
      rem = blockIdx.x - kt * per_kt;
    } else {
      rem = blockIdx.x / n_kt;
      kt = blockIdx.x - rem * n_kt;
    }
    b = rem / p.Hkv;
    rh = rem - b * p.Hkv;
    r0 = kt * C::kRows;
    const int n_qs = (p.qL + C::kStep - 1) / C::kStep;
    s0 = p.causal ? min(r0 / C::kStep, n_qs) : 0;  // causal: query rows from r0 on
    per_head = max(0, n_qs - s0);
    n_steps = p.group * per_head;
  }
  // Step j streams rows row0 of head sh (queries for dV/dK, keys for dQ).
  auto step_of = [&](int j, int& sh, int& row0) {
    if constexpr (C::kRole == kT32DQ) {
      sh = rh / p.group;
      row0 = j * C::kStep;
    } else {
      const int r = j / per_head;
      sh = rh * p.group + r;
      row0 = (s0 + (j - r * per_head)) * C::kStep;
    }
  };

  if (threadIdx.x == 0) {
    mbar_init(&ctl->res_full, 1);
    for (int t = 0; t < 3; ++t)
      for (int s = 0; s < 4; ++s) {
        mbar_init(&ctl->t_full[t][s], 1);
        mbar_init(&ctl->t_empty[t][s], 1);
      }
    for (int s = 0; s < 4; ++s) {
      mbar_init(&ctl->ld_full[s], 32);  // every lane of warp 2 stages its 2 queries
      mbar_init(&ctl->ld_empty[s], 4);  // one arrival per elementwise warp
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(&ctl->s_full[x], 1);
      mbar_init(&ctl->dp_full[x], 1);
      mbar_init(&ctl->ready[x], 4);
    }
    mbar_init(&ctl->done, 1);
    mbar_init(&ctl->drain, 1);
    ctl->abort = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmR0);
    tma_prefetch_desc(&tmT0);
    tma_prefetch_desc(&tmT2);
    if (C::kHasDP) {
      tma_prefetch_desc(&tmR1);
      tma_prefetch_desc(&tmT1);
    }
  }
  if (warp == 1) {
    tmem_alloc(&ctl->tmem_base, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl->tmem_base;

  // Loads one streamed tile of ring t for step j into slot s.
  auto load_tile = [&](int t, int j, int s) {
    int sh, row0;
    step_of(j, sh, row0);
    uint64_t* bar = &ctl->t_full[t][s];
    uint8_t* dst = sT[t] + s * C::kTBytes;
    mbar_arrive_expect_tx(bar, C::kTBytes);
    if (t < 2) {
      const CUtensorMap* m = t == 0 ? &tmT0 : &tmT1;
#pragma unroll
      for (int c = 0; c < C::kNChunk; ++c) tma_load_4d(dst + c * (C::kStep * 128), m, bar, c * 32, row0, sh, b);
    } else {
#pragma unroll
      for (int c = 0; c < C::kStep / 32; ++c) tma_load_4d(dst + c * (C::kD * 128), &tmT2, bar, row0 + c * 32, 0, sh, b);
    }
  };
  // One producer thread's ring: waits for each slot to drain, then refills it.
  auto run_ring = [&](int t, bool& ok, int& issued) {
    for (int j = 0; j < n_steps && ok; ++j) {
      const int s = j % kS, use = j / kS;
      ok = wait_bounded(&ctl->t_empty[t][s], (use & 1) ^ 1, abort_flag, p.status, p.timeout_cycles);
      if (!ok) break;
      load_tile(t, j, s);
      ++issued;
    }
  };
  auto drain_ring = [&](int t, int issued) {
    for (int it = max(0, issued - kS); it < issued; ++it)
      wait_bounded(&ctl->t_full[t][it % kS], (it / kS) & 1, abort_flag, p.status, kDrainCycles, false);
  };

  if (warp == 0) {
    // ===================================================== resident tiles + ring 0
    if (lane == 0 && n_steps > 0) {
      mbar_arrive_expect_tx(&ctl->res_full, C::kNRes * C::kResBytes);
      const int res_h = rh;  // the resident head (kvh for dV / dK, h for dQ)
#pragma unroll
      for (int c = 0; c < C::kNChunk; ++c) {
        tma_load_4d(sR0 + c * (C::kRows * 128), &tmR0, &ctl->res_full, c * 32, r0, res_h, b);
        if (C::kHasDP) tma_load_4d(sR1 + c * (C::kRows * 128), &tmR1, &ctl->res_full, c * 32, r0, res_h, b);
      }
      bool ok = true;
      int issued = 0;
      run_ring(0, ok, issued);
      if (*abort_flag) {
        wait_bounded(&ctl->res_full, 0, abort_flag, p.status, kDrainCycles, false);
        drain_ring(0, issued);
      }
    }
  } else if (warp == 2) {
    // ===================================================== ring 1 and the per-query L2, D values
    bool ok = true;
    int issued = 0;
    for (int j = 0; j < n_steps && ok; ++j) {
      const int s = j % kS, use = j / kS;
      if (C::kHasDP && lane == 0) {
        ok = wait_bounded(&ctl->t_empty[1][s], (use & 1) ^ 1, abort_flag, p.status, p.timeout_cycles);
        if (ok) {
          load_tile(1, j, s);
          ++issued;
        }
      }
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      if (!ok) break;
      if constexpr (C::kColLD) {
        // L2 = L log2(e) (+inf past qL or for a row without keys, so P = 0 there) and D.
        ok = warp_wait(&ctl->ld_empty[s], (use & 1) ^ 1, abort_flag, p.status, p.timeout_cycles);
        if (!ok) break;
        int h, q0;
        step_of(j, h, q0);
        float* l2s = sLD + s * 2 * C::kStep;
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
          l2s[C::kStep + c] = dv;
        }
        mbar_arrive(&ctl->ld_full[s]);
      }
    }
    if (C::kHasDP && lane == 0 && *abort_flag) drain_ring(1, issued);
  } else if (warp == 3) {
    // ===================================================== ring 2 (transposed tiles)
    if (lane == 0 && n_steps > 0) {
      bool ok = true;
      int issued = 0;
      run_ring(2, ok, issued);
      if (*abort_flag) drain_ring(2, issued);
    }
  } else if (warp == 1) {
    // ===================================================== MMA issuer
    if (lane == 0 && n_steps > 0) {
      constexpr uint32_t idS = make_idesc_fmt(kFmtTf32, 128, C::kStep, false, false);
      constexpr uint32_t idAcc = make_idesc_fmt(kFmtTf32, 128, C::kD, false, false);
      const uint64_t dR0 = make_sdesc_sw128(smem_u32(sR0), 16, 1024);
      const uint32_t hi = (uint32_t)(dR0 >> 32);
      const uint32_t aR0 = (uint32_t)dR0, aR1 = (uint32_t)make_sdesc_sw128(smem_u32(sR1), 16, 1024);
      const uint32_t aT0 = (uint32_t)make_sdesc_sw128(smem_u32(sT[0]), 16, 1024);
      const uint32_t aT1 = (uint32_t)make_sdesc_sw128(smem_u32(sT[1]), 16, 1024);
      const uint32_t aT2 = (uint32_t)make_sdesc_sw128(smem_u32(sT[2]), 16, 1024);
      const uint32_t slot = C::kTBytes >> 4;
      // S (or S^T) and dP (or dP^T) of step j into buffer j & 1; each frees its ring slot.
      auto issue_rows = [&](int j) -> bool {
        const int s = j % kS, use = j / kS, x = j & 1;
        if (!wait_bounded(&ctl->t_full[0][s], use & 1, abort_flag, p.status, p.timeout_cycles)) return false;
        tc_fence_after();
        t32_mma_rows<C>(tmem + C::kColS + x * C::kStep, aR0, hi, aT0 + s * slot, idS);
        mma_commit(&ctl->s_full[x]);
        mma_commit(&ctl->t_empty[0][s]);
        if (C::kHasDP) {
          if (!wait_bounded(&ctl->t_full[1][s], use & 1, abort_flag, p.status, p.timeout_cycles)) return false;
          tc_fence_after();
          t32_mma_rows<C>(tmem + C::kColDP + x * C::kStep, aR1, hi, aT1 + s * slot, idS);
          mma_commit(&ctl->dp_full[x]);
          mma_commit(&ctl->t_empty[1][s]);
        }
        return true;
      };
      bool ok = wait_bounded(&ctl->res_full, 0, abort_flag, p.status, p.timeout_cycles);
      if (ok) ok = issue_rows(0);
      // Order: rows of step j + 1, then the accumulation of step j (its P or dS ready).
      for (int j = 0; j < n_steps && ok; ++j) {
        if (j + 1 < n_steps) {
          ok = issue_rows(j + 1);
          if (!ok) break;
        }
        const int s = j % kS, use = j / kS, x = j & 1;
        ok = wait_bounded(&ctl->ready[x], (j >> 1) & 1, abort_flag, p.status, p.timeout_cycles);
        if (!ok) break;
        ok = wait_bounded(&ctl->t_full[2][s], use & 1, abort_flag, p.status, p.timeout_cycles);
        if (!ok) break;
        tc_fence_after();
        const uint32_t src = C::kHasDP ? C::kColDP + x * C::kStep : C::kColS + x * C::kStep;
        t32_mma_acc<C>(tmem + C::kColAcc, tmem + src, aT2 + s * slot, hi, idAcc, j > 0 ? 1u : 0u);
        mma_commit(&ctl->t_empty[2][s]);
      }
      if (ok) mma_commit(&ctl->done);
      mma_commit(&ctl->drain);
      wait_bounded(&ctl->drain, 0, abort_flag, p.status, kDrainCycles, false);
    }
    __syncwarp();
  } else {
    // ===================================================== elementwise warpgroup: thread = resident row
    const int tl = threadIdx.x - 128;
    const int row = r0 + tl;  // key (dV, dK) or query (dQ)
    const uint32_t lane_addr = (uint32_t)((warp & 3) * 32) << 16;
    const float sl = p.scale_log2;
    float l2_row = __int_as_float(0x7f800000), d_row = 0.0f;
    long long qrow = 0;
    if constexpr (C::kRole == kT32DQ) {
      qrow = ((long long)b * p.Hq + rh) * p.qL + (row < p.qL ? row : 0);
      if (row < p.qL) {
        const float L = __ldg(p.lse + qrow);
        if (L != -INFINITY) l2_row = L * kLog2e;
        d_row = p.dvec[qrow];
      }
    }
    bool ok = true;
    for (int j = 0; j < n_steps && ok; ++j) {
      const int s = j % kS, use = j / kS, x = j & 1;
      int sh, c0;
      step_of(j, sh, c0);
      const float* l2s = sLD + s * 2 * C::kStep;
      if constexpr (C::kColLD) {
        ok = warp_wait(&ctl->ld_full[s], use & 1, abort_flag, p.status, p.timeout_cycles);
        if (!ok) break;
      }
      ok = warp_wait(&ctl->s_full[x], (j >> 1) & 1, abort_flag, p.status, p.timeout_cycles);
      if (!ok) break;
      tc_fence_after();
      const uint32_t tS = tmem + lane_addr + C::kColS + x * C::kStep;
      float pr[64];
      tmem_ld64f(tS, pr);
      // Columns c with c < lo or c >= hi get P = 0.
      int lo = 0, hi_c = C::kStep;
      if constexpr (C::kRole == kT32DQ) {
        hi_c = p.kL - c0;  // keys past kL
        if (p.causal) hi_c = min(hi_c, row + 1 - c0);
      } else {
        if (p.causal) lo = row - c0;  // queries before this key
        if (row >= p.kL) hi_c = 0;
      }
#pragma unroll
      for (int c = 0; c < 64; c += 2) {
        float x0, x1;
        if constexpr (C::kRole == kT32DQ)
          ffma2(x0, x1, pr[c], pr[c + 1], sl, sl, -l2_row, -l2_row);
        else
          ffma2(x0, x1, pr[c], pr[c + 1], sl, sl, -l2s[c], -l2s[c + 1]);
        pr[c] = (c >= lo && c < hi_c) ? ex2(x0) : 0.0f;
        pr[c + 1] = (c + 1 >= lo && c + 1 < hi_c) ? ex2(x1) : 0.0f;
      }
      if constexpr (C::kRole == kT32DV) {
        t32_store64(tS, pr);
      } else {
        ok = warp_wait(&ctl->dp_full[x], (j >> 1) & 1, abort_flag, p.status, p.timeout_cycles);
        if (!ok) break;
        tc_fence_after();
        const uint32_t tDP = tmem + lane_addr + C::kColDP + x * C::kStep;
        float dp[64];
        tmem_ld64f(tDP, dp);
#pragma unroll
        for (int c = 0; c < 64; ++c) {
          const float dsub = C::kRole == kT32DQ ? d_row : l2s[C::kStep + c];
          dp[c] = pr[c] * (dp[c] - dsub);
        }
        t32_store64(tDP, dp);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&ctl->ready[x]);
        if (C::kColLD) mbar_arrive(&ctl->ld_empty[s]);
      }
    }
    // ---- epilogue: this row of dV, scale * dK or scale * dQ (fp32)
    if (ok) {
      const int n_out = C::kRole == kT32DQ ? p.qL : p.kL;
      const bool store = row < n_out;
      float* out;
      float mul = p.scale;
      if constexpr (C::kRole == kT32DQ) {
        out = static_cast<float*>(p.dq) + qrow * C::kD;
      } else {
        const long long krow = ((long long)b * p.Hkv + rh) * p.kL + (store ? row : 0);
        out = static_cast<float*>(C::kRole == kT32DV ? p.dv : p.dk) + krow * C::kD;
        if (C::kRole == kT32DV) mul = 1.0f;
      }
      if (n_steps == 0) {  // no step reaches this row: zero gradient
        if (store)
          for (int u = 0; u < C::kD / 4; ++u) reinterpret_cast<float4*>(out)[u] = make_float4(0.f, 0.f, 0.f, 0.f);
      } else {
        ok = warp_wait(&ctl->done, 0, abort_flag, p.status, p.timeout_cycles);
        if (ok) {
          tc_fence_after();
          // staged in the streamed rings (every load of them consumed)
          constexpr int kSlot = (C::kD / 32) * 32 * 128;
          t32_store_tile_tma<C>(tmem + lane_addr + C::kColAcc, mul, smem + C::kOffT0 + (warp & 3) * kSlot, &tmOut,
                                r0 + 32 * (warp & 3), n_out, rh, b, lane);
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

// D_i = rowsum(O_i * dO_i) for fp32 rows: kD / 4 threads per row, 16-byte loads.
template <int kD>
__global__ void __launch_bounds__(256) fa_bwd_rowdot_f32_kernel(const float4* __restrict__ o,
                                                                const float4* __restrict__ dout,
                                                                float* __restrict__ dvec, long long rows) {
  constexpr int kLanes = kD / 4;
  constexpr int kRowsPerBlock = 256 / kLanes;
  const int sub = threadIdx.x % kLanes;
  const long long row = (long long)blockIdx.x * kRowsPerBlock + threadIdx.x / kLanes;
  float acc = 0.0f;
  if (row < rows) {
    const float4 a = __ldg(o + row * kLanes + sub);
    const float4 g = __ldg(dout + row * kLanes + sub);
    acc = fmaf(a.x, g.x, fmaf(a.y, g.y, fmaf(a.z, g.z, a.w * g.w)));
  }
#pragma unroll
  for (int off = kLanes / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (row < rows && sub == 0) dvec[row] = acc;
}

}  // namespace fa
