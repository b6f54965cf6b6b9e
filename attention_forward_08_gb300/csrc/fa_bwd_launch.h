// fa_bwd_launch.h -- host-side interface between the C ABI layer and the
// backward launcher (fa_bwd.cu).  Arguments arrive already validated.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "fa.h"

namespace fa {

struct BwdLaunchArgs {
  const void *q, *k, *v, *o, *dout;  // bf16 (fp16 when f16), contiguous [B,H,L,D]
  const float* lse;                  // [B, H_q, qL]
  void *dq, *dk, *dv;                // outputs in the same format
  bool f16;                          // fp16 I/O instead of bf16
  bool f32;                          // fp32 I/O (TF32 products)
  void* t32_ws;                      // fp32: scratch for the rounded copies and transposes (BwdTf32Layout)
  float* dvec;                       // [B, H_q, qL] scratch for D = rowsum(O * dO)
  int B, Hq, Hkv, qL, kL, D;
  float scale;
  int causal;
  int window, q_offset;              // sliding window (0 = off) and causal diagonal offset
  float softcap;                     // 0 = off
  float dropout_p;                   // 0 = off: the forward's dropout, regenerated from
  unsigned long long dropout_seed;   //   the same seed and offset (counter-based keep
  unsigned long long dropout_offset; //   contract, as in the forward)
  uint32_t* keep_mask;               // dropout: [B, H_q, qL, keep_row_words] scratch for the
  long long keep_row_words;          //   keep decisions (4 * ceil(kL / 128) words a row)
  int mask_kind;                     // the forward's mask: 0 none, 1 bool (uint8), 2 additive (I/O format)
  const void* mask;                  // [B, H_q, qL, kL] through ms (element strides; key stride 1)
  long long ms[3];
  int mask_vec;                      // mask rows 16-byte aligned: vector loads
  void* mask_t;                      // additive: scratch key-major copy [B, H_q, kL, mask_t_ld]
  long long mask_t_ld;
  uint32_t* mask_tbits;              // bool: scratch keep bits, key-major [B, H_q, kL, mask_tbits_ld words]
  long long mask_tbits_ld;           //   (bit x of word w: query 32 w + x)
  uint32_t* mask_rbits;              // bool: scratch keep bits, row-major [B, H_q, qL, mask_rbits_ld words]
  long long mask_rbits_ld;           //   (bit x of word w: key 32 w + x)
  cudaStream_t stream;
  unsigned int* status;
  long long timeout_cycles;
};

// fp32 backward scratch (after the D vector; every part 256-byte aligned):
// tf32-rounded copies of Q, dO [B, H_q, qL, D] and K, V [B, H_kv, kL, D],
// then tf32-rounded transposes Q^T, dO^T [B, H_q, D, qt_row] and
// K^T [B, H_kv, D, kt_row], rows rounded up to 4 entries (16 bytes).
struct BwdTf32Layout {
  long long qr, dor, kr, vr, qt, dot, kt;  // byte offsets
  long long qt_row, kt_row;
  long long bytes;
};
inline BwdTf32Layout bwd_tf32_layout(int B, int Hq, int Hkv, int qL, int kL, int D) {
  auto al = [](long long n) { return (n + 255) / 256 * 256; };
  BwdTf32Layout l;
  l.qt_row = ((long long)qL + 3) / 4 * 4;
  l.kt_row = ((long long)kL + 3) / 4 * 4;
  const long long nq = al((long long)B * Hq * qL * D * 4), nk = al((long long)B * Hkv * kL * D * 4);
  const long long nqt = al((long long)B * Hq * D * l.qt_row * 4), nkt = al((long long)B * Hkv * D * l.kt_row * 4);
  l.qr = 0;
  l.dor = l.qr + nq;
  l.kr = l.dor + nq;
  l.vr = l.kr + nk;
  l.qt = l.vr + nk;
  l.dot = l.qt + nqt;
  l.kt = l.dot + nqt;
  l.bytes = l.kt + nkt;
  return l;
}

// Launches the D pre-pass, the dK/dV kernel and the dQ kernel on a.stream.
// Returns 0, or an fa_status code with the message set.
int launch_bwd(const BwdLaunchArgs& a);

// B * H * L > cap for positive B, H, L, computed without overflow.
bool rows_exceed(int B, int H, int L, long long cap);

// Checks a backward call's arguments other than its workspace; returns
// FA_OK or an fa_status code with the message set.
int validate_bwd(const fa_bwd_args* a);

}  // namespace fa
