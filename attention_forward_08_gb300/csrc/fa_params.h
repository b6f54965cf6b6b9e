// fa_params.h -- the scalar parameter block the launcher hands to the forward
// kernel (passed by value as a kernel argument; tensor maps travel beside it).
#pragma once

#include <stdint.h>

namespace fa {

// Device status word bits (the library keeps one static word per device).
enum : unsigned int {
  kStatusTimeout = 1u << 0,  // a bounded wait ran out; the kernel unwound early
};

struct FaParams {
  int B, Hq, Hkv, qL, kL;
  int group;        // Hq / Hkv: query heads per K/V head
  int n_qblocks;    // query blocks per (b, head unit): 128 rows with head pairs, else tiles per CTA * 128
  int head_pairs;   // two Q tiles per unit are heads 2u and 2u + 1 (one K/V head) at the same rows
  int hq_units;     // head units per batch: H_q / 2 with head pairs, else H_q
  int causal;       // top-left aligned: key j allowed for row i iff j <= i
  int mask_kind;    // 0 none, 1 bool (uint8, nonzero keeps), 2 additive (I/O dtype)
  int pre_scale;    // scale scores before masking (additive mask, softcap, or scale <= 0)
  int mask_vec;     // mask rows 16-byte aligned: vector loads allowed
  int mask_l2;      // a tensor map describes the mask: prefetch its tiles into L2
  int mask_smem;    // the mask map is 128-byte swizzled: TMA-load its tiles into shared memory
  float scale_log2; // scale * log2(e)
  int dropout_on;       // weights of O kept with probability 1 - p (counter-based generator)
  unsigned int drop_threshold;  // keep iff (word >> 8) >= drop_threshold = ceil(p * 2^24)
  float drop_scale;     // 1 / (1 - p) (0 when p = 1)
  unsigned int seed_lo, seed_hi;
  unsigned long long drop_offset;  // counter of position 0
  int mask_natural; // additive mask, scale > 0, no softcap: fold s + mask / scale (raw score units)
  float inv_scale;  // 1 / scale (when mask_natural)
  int window;       // > 0: key j allowed only if j > i + q_offset - window (sliding window)
  int q_offset;     // causal diagonal of row i is key i + q_offset (0: top-left aligned)
  int softcap_on;   // scores become cap * tanh(scale * s / cap) before any mask
  float softcap_in;   // scale / cap
  float softcap_out;  // cap * log2(e)
  const void* mask;
  long long mask_sb, mask_sh, mask_ss;  // mask element strides: batch, head, query row
  void* o;                              // output, I/O dtype
  long long o_sb, o_sh, o_ss;           // O element strides: batch, head, query row
  float* lse;                           // [B, Hq, qL] fp32, natural log
  // Split-KV (one-Q-tile 16-bit plans without features): the key blocks of
  // each (query tile, head) are cut into kv_splits ranges of kv_chunk blocks,
  // one work unit each; a unit writes its range's normalised O in fp32 and
  // its logsumexp to part_o / part_lse instead of O and L, and a combine pass
  // merges the ranges.  kv_splits = 1: off.
  int kv_splits;
  int kv_chunk;
  float* part_o;                        // [kv_splits, B * Hq, qL, D]
  float* part_lse;                      // [kv_splits, B * Hq, qL]
  unsigned int* status;                 // device status word (kStatus* bits)
  long long timeout_cycles;             // bound on every wait, in SM clock cycles
};

}  // namespace fa
