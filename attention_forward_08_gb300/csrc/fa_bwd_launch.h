// fa_bwd_launch.h -- host-side interface between the C ABI layer and the
// backward launcher (fa_bwd.cu).  Arguments arrive already validated.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

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
  cudaStream_t stream;
  unsigned int* status;
  long long timeout_cycles;
};

// Launches the D pre-pass, the dK/dV kernel and the dQ kernel on a.stream.
// Returns 0, or an fa_status code with the message set.
int launch_bwd(const BwdLaunchArgs& a);

// B * H * L > cap for positive B, H, L, computed without overflow.
bool rows_exceed(int B, int H, int L, long long cap);

// Checks a backward call's arguments other than its workspace (fa_bwd_ex's
// rules); returns FA_OK or an fa_status code with the message set.
int validate_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse,
                 const void* dq, const void* dk, const void* dv, int B, int H_q, int H_kv, int qL, int kL, int D,
                 float scale, int window, int q_offset, float softcap, float dropout_p, int dtype);

}  // namespace fa
