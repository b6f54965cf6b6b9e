// fa_bwd_tf32.cu -- the fp32 backward plans (head dims 64 and 128, causal or
// not, GQA): the D pre-pass, the tf32 rounding and transpose pre-pass into
// the workspace, then the dV, dK and dQ kernels of fa_bwd_tf32_kernel.cuh.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstring>

#include "fa_bwd_impl.cuh"
#include "fa_bwd_tf32_kernel.cuh"
#include "fa_tf32_ops.cuh"

namespace fa {

namespace {

int check(const char* what) {
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    set_error("%s launch failed: %s", what, cudaGetErrorString(e));
    return 4;
  }
  return 0;
}

// fp32 [B, H, rows, D] tiles of box_rows rows in 32-column (128-byte) blocks.
bool encode_rows(CUtensorMap* m, const void* ptr, int B, int H, int rows, int D, int box_rows) {
  const long long st[3] = {(long long)H * rows * D, (long long)rows * D, D};
  return encode_bhsd(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, ptr, B, H, rows, D, st, 32, box_rows);
}

template <class C>
int launch_role(const CUtensorMap& r0, const CUtensorMap& r1, const CUtensorMap& t0, const CUtensorMap& t1,
                const CUtensorMap& t2, const CUtensorMap& out, const BwdParams& p, long long grid, cudaStream_t stream,
                const char* what) {
  static std::atomic<unsigned long long> cfg{0};
  if (int rc = bwd_impl::set_smem_once<C>((const void*)fa_bwd_tf32_kernel<C>, C::kSmem, cfg)) return rc;
  if (grid <= 0) return 0;
  fa_bwd_tf32_kernel<C><<<(unsigned)grid, C::kThreads, C::kSmem, stream>>>(r0, r1, t0, t1, t2, out, p);
  return check(what);
}

template <int kD>
int launch_tf32_d(const BwdLaunchArgs& a) {
  const BwdTf32Layout l = bwd_tf32_layout(a.B, a.Hq, a.Hkv, a.qL, a.kL, kD);
  char* ws = static_cast<char*>(a.t32_ws);
  float* qr = reinterpret_cast<float*>(ws + l.qr);
  float* dor = reinterpret_cast<float*>(ws + l.dor);
  float* kr = reinterpret_cast<float*>(ws + l.kr);
  float* vr = reinterpret_cast<float*>(ws + l.vr);
  float* qt = reinterpret_cast<float*>(ws + l.qt);
  float* dot = reinterpret_cast<float*>(ws + l.dot);
  float* kt = reinterpret_cast<float*>(ws + l.kt);

  // 1. D_i = rowsum(O_i * dO_i)
  const long long rows = (long long)a.B * a.Hq * a.qL;
  constexpr int kRowsPerBlock = 256 / (kD / 4);
  fa_bwd_rowdot_f32_kernel<kD><<<(unsigned)((rows + kRowsPerBlock - 1) / kRowsPerBlock), 256, 0, a.stream>>>(
      static_cast<const float4*>(a.o), static_cast<const float4*>(a.dout), a.dvec, rows);
  if (int rc = check("row-dot")) return rc;

  // 2. tf32-rounded copies and transposes (HBM-bound, once per call).
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0) sms = 1;
  const long long cap = (long long)sms * 8;
  auto round_rows = [&](const void* src, float* dst, int H, int L) {
    const long long n4 = (long long)a.B * H * L * kD / 4;
    const long long st_b = (long long)H * L * kD, st_h = (long long)L * kD;
    tf32_round_rows_kernel<<<(unsigned)std::min<long long>((n4 + 255) / 256, cap), 256, 0, a.stream>>>(
        static_cast<const float*>(src), st_b, st_h, kD, dst, H, L, kD, n4);
    return check("tf32 rounding");
  };
  auto transpose = [&](const void* src, float* dst, int H, int L, long long row_len) {
    const long long BH = (long long)a.B * H, st_b = (long long)H * L * kD, st_h = (long long)L * kD;
    const dim3 grid((unsigned)((row_len + 31) / 32), (unsigned)(kD / 32), (unsigned)std::min<long long>(BH, 65535));
    tf32_transpose_v_kernel<<<grid, dim3(32, 8), 0, a.stream>>>(static_cast<const float*>(src), st_b, st_h, kD, dst,
                                                                H, BH, L, kD, row_len);
    return check("tf32 transpose");
  };
  if (int rc = round_rows(a.q, qr, a.Hq, a.qL)) return rc;
  if (int rc = round_rows(a.dout, dor, a.Hq, a.qL)) return rc;
  if (int rc = round_rows(a.k, kr, a.Hkv, a.kL)) return rc;
  if (int rc = round_rows(a.v, vr, a.Hkv, a.kL)) return rc;
  if (int rc = transpose(a.q, qt, a.Hq, a.qL, l.qt_row)) return rc;
  if (int rc = transpose(a.dout, dot, a.Hq, a.qL, l.qt_row)) return rc;
  if (int rc = transpose(a.k, kt, a.Hkv, a.kL, l.kt_row)) return rc;

  // 3. Tensor maps: resident 128-row tiles, streamed 64-row tiles, transposed 64-column tiles.
  using CV = BwdT32Cfg<kD, kT32DV>;
  using CK = BwdT32Cfg<kD, kT32DK>;
  using CQ = BwdT32Cfg<kD, kT32DQ>;
  CUtensorMap q128, do128, k128, v128, q64, do64, k64, v64, mqt, mdot, mkt;
  if (!encode_rows(&q128, qr, a.B, a.Hq, a.qL, kD, 128) || !encode_rows(&do128, dor, a.B, a.Hq, a.qL, kD, 128) ||
      !encode_rows(&k128, kr, a.B, a.Hkv, a.kL, kD, 128) || !encode_rows(&v128, vr, a.B, a.Hkv, a.kL, kD, 128) ||
      !encode_rows(&q64, qr, a.B, a.Hq, a.qL, kD, 64) || !encode_rows(&do64, dor, a.B, a.Hq, a.qL, kD, 64) ||
      !encode_rows(&k64, kr, a.B, a.Hkv, a.kL, kD, 64) || !encode_rows(&v64, vr, a.B, a.Hkv, a.kL, kD, 64) ||
      !encode_vt(&mqt, qt, a.B, a.Hq, (int)l.qt_row, kD, l.qt_row) ||
      !encode_vt(&mdot, dot, a.B, a.Hq, (int)l.qt_row, kD, l.qt_row) ||
      !encode_vt(&mkt, kt, a.B, a.Hkv, (int)l.kt_row, kD, l.kt_row))
    return 4;
  // the gradients as 32-row, 128-byte boxes for the epilogues' TMA stores
  CUtensorMap odq, odk, odv;
  if (!encode_rows(&odq, a.dq, a.B, a.Hq, a.qL, kD, 32) || !encode_rows(&odk, a.dk, a.B, a.Hkv, a.kL, kD, 32) ||
      !encode_rows(&odv, a.dv, a.B, a.Hkv, a.kL, kD, 32))
    return 4;

  BwdParams p;
  std::memset(&p, 0, sizeof(p));
  p.B = a.B;
  p.Hq = a.Hq;
  p.Hkv = a.Hkv;
  p.qL = a.qL;
  p.kL = a.kL;
  p.group = a.Hq / a.Hkv;
  p.causal = a.causal;
  p.n_qt = (a.qL + 127) / 128;
  p.n_kt = (a.kL + 127) / 128;
  p.scale = a.scale;
  p.scale_log2 = a.scale * kLog2e;
  p.lse = a.lse;
  p.dvec = a.dvec;
  p.dq = a.dq;
  p.dk = a.dk;
  p.dv = a.dv;
  p.status = a.status;
  p.timeout_cycles = a.timeout_cycles;

  const long long n_kv = (long long)p.n_kt * a.Hkv * a.B, n_q = (long long)p.n_qt * a.Hq * a.B;
  if (n_kv > 0x7fffffffLL || n_q > 0x7fffffffLL) {
    set_error("backward grid of %lld / %lld CTAs is out of range", n_kv, n_q);
    return 2;
  }
  // 4. dV (K resident; Q, dO^T streamed), dK (K, V; Q, dO, Q^T), dQ (Q, dO; K, V, K^T).
  if (int rc = launch_role<CV>(k128, k128, q64, q64, mdot, odv, p, n_kv, a.stream, "dV")) return rc;
  if (int rc = launch_role<CK>(k128, v128, q64, do64, mqt, odk, p, n_kv, a.stream, "dK")) return rc;
  return launch_role<CQ>(q128, do128, k64, v64, mkt, odq, p, n_q, a.stream, "dQ");
}

}  // namespace

int launch_bwd_tf32(const BwdLaunchArgs& a) { return a.D == 64 ? launch_tf32_d<64>(a) : launch_tf32_d<128>(a); }

}  // namespace fa
