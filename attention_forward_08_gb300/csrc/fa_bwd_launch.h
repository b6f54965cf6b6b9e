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
  void* mask_t;                      // scratch: key-major copy [B, H_q, kL, mask_t_ld]
  long long mask_t_ld;
  cudaStream_t stream;
  unsigned int* status;
  long long timeout_cycles;
};

// Launches the D pre-pass, the dK/dV kernel and the dQ kernel on a.stream.
// Returns 0, or an fa_status code with the message set.
int launch_bwd(const BwdLaunchArgs& a);

// B * H * L > cap for positive B, H, L, computed without overflow.
bool rows_exceed(int B, int H, int L, long long cap);

// Checks a backward call's arguments other than its workspace; returns
// FA_OK or an fa_status code with the message set.
int validate_bwd(const fa_bwd_args* a);

}  // namespace fa
