// fa_bwd_impl.cuh -- launcher template for the backward pass: tensor maps,
// grids and the launches (D pre-pass; keep-mask pre-pass with dropout; mask
// transpose with a mask; dK/dV; dQ) for one instantiation (head dim, bf16 or
// fp16 I/O, features, dropout, mask).  The translation units fa_bwd*.cu each
// instantiate a share of the plans (parallel compilation) and dispatch to it.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>

#include "fa_bwd_kernel.cuh"
#include "fa_bwd_launch.h"
#include "fa_launch.cuh"

namespace fa {

namespace bwd_impl {

template <class C>
int set_smem_once(const void* kern, uint32_t bytes, std::atomic<unsigned long long>& configured) {
  int dev = 0;
  cudaGetDevice(&dev);
  if (device_bit_set(configured, dev)) return 0;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e != cudaSuccess) {
    set_error("cudaFuncSetAttribute(max dynamic smem = %u): %s", (unsigned)bytes, cudaGetErrorString(e));
    return 4;
  }
  device_bit_mark(configured, dev);
  return 0;
}

template <int kD, bool kF16, bool kFeat, bool kDrop = false, int kMask = 0, bool kCap = false>
int launch_bwd_d(const BwdLaunchArgs& a) {
  using C = BwdCfg<kD, kF16, kFeat, kDrop, kMask, kCap>;
  if (a.mask_kind != kMask || (!kCap && a.softcap != 0.0f)) {
    set_error("backward plan for mask kind %d%s given mask kind %d, softcap %g", kMask, kCap ? " with a softcap" : "",
              a.mask_kind, (double)a.softcap);
    return 2;
  }
  // 1. D_i = rowsum(O_i * dO_i)
  const long long rows = (long long)a.B * a.Hq * a.qL;
  constexpr int kRowsPerBlock = 256 / (kD / 8);
  const long long blocks = (rows + kRowsPerBlock - 1) / kRowsPerBlock;
  fa_bwd_rowdot_kernel<kD, kF16><<<(unsigned)blocks, 256, 0, a.stream>>>(
      static_cast<const uint4*>(a.o), static_cast<const uint4*>(a.dout), a.dvec, rows);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    set_error("row-dot launch failed: %s", cudaGetErrorString(e));
    return 4;
  }

  // 2. Tensor maps: 128-row tiles of 128-byte swizzled column blocks.
  const long long qst[3] = {(long long)a.Hq * a.qL * kD, (long long)a.qL * kD, kD};
  const long long kst[3] = {(long long)a.Hkv * a.kL * kD, (long long)a.kL * kD, kD};
  CUtensorMap tq, tk, tv, tdo;
  if (!encode_bhsd(&tq, C::kTmaType, a.q, a.B, a.Hq, a.qL, kD, qst, 64, C::kTile)) return 4;
  if (!encode_bhsd(&tdo, C::kTmaType, a.dout, a.B, a.Hq, a.qL, kD, qst, 64, C::kTile)) return 4;
  if (!encode_bhsd(&tk, C::kTmaType, a.k, a.B, a.Hkv, a.kL, kD, kst, 64, C::kTile)) return 4;
  if (!encode_bhsd(&tv, C::kTmaType, a.v, a.B, a.Hkv, a.kL, kD, kst, 64, C::kTile)) return 4;
  // the gradients as 32-row, 128-byte boxes for the epilogues' TMA stores
  CUtensorMap tdq, tdk, tdv;
  if (!encode_bhsd(&tdq, C::kTmaType, a.dq, a.B, a.Hq, a.qL, kD, qst, 64, 32)) return 4;
  if (!encode_bhsd(&tdk, C::kTmaType, a.dk, a.B, a.Hkv, a.kL, kD, kst, 64, 32)) return 4;
  if (!encode_bhsd(&tdv, C::kTmaType, a.dv, a.B, a.Hkv, a.kL, kD, kst, 64, 32)) return 4;

  BwdParams p;
  p.B = a.B;
  p.Hq = a.Hq;
  p.Hkv = a.Hkv;
  p.qL = a.qL;
  p.kL = a.kL;
  p.group = a.Hq / a.Hkv;
  p.causal = a.causal;
  p.window = a.window;
  p.q_offset = a.q_offset;
  p.softcap_on = a.softcap > 0.0f ? 1 : 0;
  p.softcap_kin = p.softcap_on ? 2.0f * kLog2e * (a.scale / a.softcap) : 0.0f;
  p.softcap_out = p.softcap_on ? a.softcap * kLog2e : 0.0f;
  p.softcap_inv = p.softcap_on ? 1.0f / p.softcap_out : 0.0f;
  p.dropout_on = kDrop ? 1 : 0;
  p.drop_threshold = kDrop ? (unsigned int)std::ceil((double)a.dropout_p * 16777216.0) : 0u;
  p.drop_scale = kDrop && a.dropout_p < 1.0f ? (float)(1.0 / (1.0 - (double)a.dropout_p)) : 0.0f;
  p.seed_lo = (unsigned int)a.dropout_seed;
  p.seed_hi = (unsigned int)(a.dropout_seed >> 32);
  p.drop_offset = a.dropout_offset;
  p.keep_mask = a.keep_mask;
  p.keep_row_words = a.keep_row_words;
  p.mask_kind = a.mask_kind;
  p.mask = a.mask;
  p.mask_sb = a.ms[0];
  p.mask_sh = a.ms[1];
  p.mask_ss = a.ms[2];
  p.mask_vec = a.mask_vec;
  p.mask_t = a.mask_t;
  p.mask_t_ld = a.mask_t_ld;
  p.mask_tbits = a.mask_tbits;
  p.mask_tbits_ld = a.mask_tbits_ld;
  p.mask_rbits = a.mask_rbits;
  p.mask_rbits_ld = a.mask_rbits_ld;
  p.n_qt = (a.qL + C::kTile - 1) / C::kTile;
  p.n_kt = (a.kL + C::kTile - 1) / C::kTile;
  p.scale = a.scale;
  p.scale_log2 = a.scale * kLog2e;
  p.lse = a.lse;
  p.dvec = a.dvec;
  p.dq = a.dq;
  p.dk = a.dk;
  p.dv = a.dv;
  p.status = a.status;
  p.timeout_cycles = a.timeout_cycles;

  static std::atomic<unsigned long long> cfg_kv{0}, cfg_q{0};
  if (int rc = set_smem_once<C>((const void*)fa_bwd_dkdv_kernel<C>, C::kKVSmem, cfg_kv)) return rc;
  if (int rc = set_smem_once<C>((const void*)fa_bwd_dq_kernel<C>, C::kQSmem, cfg_q)) return rc;

  const long long n_kv = (long long)p.n_kt * a.Hkv * a.B;
  const long long n_q = (long long)p.n_qt * a.Hq * a.B;
  if (n_kv > 0x7fffffffLL || n_q > 0x7fffffffLL) {
    set_error("backward grid of %lld / %lld CTAs is out of range", n_kv, n_q);
    return 2;
  }

  // 3. Dropout: the forward's keep decisions, once for both kernels.
  if constexpr (kDrop) {
    const long long n_units = (long long)a.B * a.Hq * p.n_qt * p.n_kt;
    if (n_units > 0x7fffffffLL) {  // the kernel's 32-bit unit index u + gridDim.x must not wrap
      set_error("dropout keep mask of %lld tiles is out of range", n_units);
      return 2;
    }
    KeepMaskArgs ka;
    uint32_t k0 = (uint32_t)a.dropout_seed, k1 = (uint32_t)(a.dropout_seed >> 32);
    for (int r = 0; r < 10; ++r, k0 += 0x9E3779B9u, k1 += 0xBB67AE85u) {  // Philox4x32 key schedule
      ka.rk0[r] = k0;
      ka.rk1[r] = k1;
    }
    ka.n_kb = (uint32_t)p.n_kt;
    ka.n_units = (uint32_t)n_units;
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0) sms = 1;
    const unsigned grid = (unsigned)std::min<long long>(n_units, (long long)sms * 8);
    fa_bwd_keep_mask_kernel<<<grid, 256, 0, a.stream>>>(p, ka);
    e = cudaGetLastError();
    if (e != cudaSuccess) {
      set_error("keep-mask launch failed: %s", cudaGetErrorString(e));
      return 4;
    }
  }

  // 4. The forward's mask: bool as keep bits (row-major and key-major), additive
  // as a key-major copy for the dK/dV kernel.
  if constexpr (kMask != 0) {
    const int BH = a.B * a.Hq;
    constexpr int kSide = kMask == 1 ? 128 : 64;  // entries per tile side (128 bytes)
    dim3 grid((unsigned)((a.kL + kSide - 1) / kSide), (unsigned)(a.mask_t_ld / kSide), (unsigned)std::min(BH, 65535));
    if constexpr (kMask == 1)
      fa_bwd_mask_bits_kernel<<<grid, 256, 0, a.stream>>>(
          static_cast<const uint8_t*>(a.mask), a.ms[0], a.ms[1], a.ms[2], a.Hq, BH, a.qL, a.kL, a.mask_vec,
          a.causal, a.q_offset, a.mask_tbits, a.mask_tbits_ld, a.mask_rbits, a.mask_rbits_ld);
    else
      fa_bwd_mask_transpose_kernel<uint16_t><<<grid, 256, 0, a.stream>>>(
          static_cast<const uint16_t*>(a.mask), a.ms[0], a.ms[1], a.ms[2], a.Hq, BH, a.qL, a.kL, a.mask_t_ld,
          a.mask_vec, a.causal, a.q_offset, static_cast<uint16_t*>(a.mask_t));
    e = cudaGetLastError();
    if (e != cudaSuccess) {
      set_error("mask transpose launch failed: %s", cudaGetErrorString(e));
      return 4;
    }
  }

  // 5. dK, dV: one CTA per (128-key tile, kvh, b).
  fa_bwd_dkdv_kernel<C><<<(unsigned)n_kv, C::kThreads, C::kKVSmem, a.stream>>>(tq, tk, tv, tdo, tdk, tdv, p);
  e = cudaGetLastError();
  if (e != cudaSuccess) {
    set_error("dK/dV launch failed: %s", cudaGetErrorString(e));
    return 4;
  }
  // 6. dQ: one CTA per (128-row query tile, h, b).
  fa_bwd_dq_kernel<C><<<(unsigned)n_q, C::kThreads, C::kQSmem, a.stream>>>(tq, tk, tv, tdo, tdq, p);
  e = cudaGetLastError();
  if (e != cudaSuccess) {
    set_error("dQ launch failed: %s", cudaGetErrorString(e));
    return 4;
  }
  return 0;
}

}  // namespace bwd_impl

}  // namespace fa
