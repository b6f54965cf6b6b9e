// fa_bwd256.cu -- the backward plans at head dim 256 (bf16 or fp16 I/O,
// causal or not, GQA): the row-dot pre-pass, then the two-CTAs-per-key-tile
// dK/dV kernel and the 64-key-block dQ kernel of fa_bwd256_kernel.cuh.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstring>

#include "fa_bwd256_kernel.cuh"
#include "fa_bwd_impl.cuh"

namespace fa {

namespace {

template <bool kF16>
int launch_bwd256_t(const BwdLaunchArgs& a) {
  using C = Bwd256Cfg<kF16>;
  constexpr int kD = C::kD;
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

  // 2. Tensor maps.  dK/dV kernel: 128-row K and V tiles, 64-row Q and dO
  // steps; dQ kernel: 128-row Q and dO tiles, 64-row K and V blocks.
  const long long qst[3] = {(long long)a.Hq * a.qL * kD, (long long)a.qL * kD, kD};
  const long long kst[3] = {(long long)a.Hkv * a.kL * kD, (long long)a.kL * kD, kD};
  CUtensorMap kv_q, kv_k, kv_v, kv_do, q_q, q_k, q_v, q_do;
  if (!encode_bhsd(&kv_q, C::kTmaType, a.q, a.B, a.Hq, a.qL, kD, qst, 64, C::kQS)) return 4;
  if (!encode_bhsd(&kv_do, C::kTmaType, a.dout, a.B, a.Hq, a.qL, kD, qst, 64, C::kQS)) return 4;
  if (!encode_bhsd(&kv_k, C::kTmaType, a.k, a.B, a.Hkv, a.kL, kD, kst, 64, C::kKT)) return 4;
  if (!encode_bhsd(&kv_v, C::kTmaType, a.v, a.B, a.Hkv, a.kL, kD, kst, 64, C::kKT)) return 4;
  if (!encode_bhsd(&q_q, C::kTmaType, a.q, a.B, a.Hq, a.qL, kD, qst, 64, C::kQT)) return 4;
  if (!encode_bhsd(&q_do, C::kTmaType, a.dout, a.B, a.Hq, a.qL, kD, qst, 64, C::kQT)) return 4;
  if (!encode_bhsd(&q_k, C::kTmaType, a.k, a.B, a.Hkv, a.kL, kD, kst, 64, C::kKB)) return 4;
  if (!encode_bhsd(&q_v, C::kTmaType, a.v, a.B, a.Hkv, a.kL, kD, kst, 64, C::kKB)) return 4;
  // the gradients as 32-row, 128-byte boxes for the epilogues' TMA stores
  CUtensorMap t_dq, t_dk, t_dv;
  if (!encode_bhsd(&t_dq, C::kTmaType, a.dq, a.B, a.Hq, a.qL, kD, qst, 64, 32)) return 4;
  if (!encode_bhsd(&t_dk, C::kTmaType, a.dk, a.B, a.Hkv, a.kL, kD, kst, 64, 32)) return 4;
  if (!encode_bhsd(&t_dv, C::kTmaType, a.dv, a.B, a.Hkv, a.kL, kD, kst, 64, 32)) return 4;

  BwdParams p;
  std::memset(&p, 0, sizeof(p));
  p.B = a.B;
  p.Hq = a.Hq;
  p.Hkv = a.Hkv;
  p.qL = a.qL;
  p.kL = a.kL;
  p.group = a.Hq / a.Hkv;
  p.causal = a.causal;
  p.n_qt = (a.qL + C::kQT - 1) / C::kQT;
  p.n_kt = (a.kL + C::kKT - 1) / C::kKT;
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
  if (int rc = bwd_impl::set_smem_once<C>((const void*)fa_bwd256_dkdv_kernel<C>, C::kKVSmem, cfg_kv)) return rc;
  if (int rc = bwd_impl::set_smem_once<C>((const void*)fa_bwd256_dq_kernel<C>, C::kQSmem, cfg_q)) return rc;

  const long long n_kv = 2LL * p.n_kt * a.Hkv * a.B;
  const long long n_q = (long long)p.n_qt * a.Hq * a.B;
  if (n_kv > 0x7fffffffLL || n_q > 0x7fffffffLL) {
    set_error("backward grid of %lld / %lld CTAs is out of range", n_kv, n_q);
    return 2;
  }
  // 3. dK, dV: two CTAs (halves of D) per (128-key tile, kvh, b).
  fa_bwd256_dkdv_kernel<C><<<(unsigned)n_kv, C::kThreads, C::kKVSmem, a.stream>>>(kv_q, kv_k, kv_v, kv_do, t_dk, t_dv,
                                                                                 p);
  e = cudaGetLastError();
  if (e != cudaSuccess) {
    set_error("dK/dV launch failed: %s", cudaGetErrorString(e));
    return 4;
  }
  // 4. dQ: one CTA per (128-row query tile, h, b).
  fa_bwd256_dq_kernel<C><<<(unsigned)n_q, C::kThreads, C::kQSmem, a.stream>>>(q_q, q_k, q_v, q_do, t_dq, p);
  e = cudaGetLastError();
  if (e != cudaSuccess) {
    set_error("dQ launch failed: %s", cudaGetErrorString(e));
    return 4;
  }
  return 0;
}

}  // namespace

int launch_bwd256(const BwdLaunchArgs& a) {
  return a.f16 ? launch_bwd256_t<true>(a) : launch_bwd256_t<false>(a);
}

}  // namespace fa
