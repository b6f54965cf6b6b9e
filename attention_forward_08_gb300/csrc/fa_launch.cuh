// fa_launch.cuh -- host launcher for one (I/O dtype, head dim) instantiation:
// encodes the four TMA tensor maps, sizes the grid and launches on the
// caller's stream.  Arguments arrive already validated by the C ABI layer.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstring>

#include "fa_kernel.cuh"

namespace fa {

struct LaunchArgs {
  const void *q, *k, *v;
  void* o;
  float* lse;
  const void* mask;
  int B, Hq, Hkv, qL, kL, D;
  float scale;
  int causal, mask_kind;
  int window, q_offset;  // sliding window (0 = off) and causal diagonal offset
  float softcap;         // 0 = off
  float dropout_p;       // 0 = off
  unsigned long long dropout_seed, dropout_offset;
  long long qs[3], ks[3], vs[3], os[3], ms[3];  // element strides: batch, head, row
  long long vt_row;      // pre-rounded fp32 plans: v is V^T [B, H_kv, D, vt_row] (keys innermost)
  int mask_vec;
  cudaStream_t stream;
  unsigned int* status;
  long long timeout_cycles;
  int num_sms;
  int max_ctas;  // 0: one CTA per SM
  // Split-KV (plans with Cfg::kSplitKV): key ranges per query tile (1: off)
  // and the partial buffers in the caller's workspace.
  int kv_splits;
  float* part_o;
  float* part_lse;
};

// cuTensorMapEncodeTiled, resolved from the driver at run time (the library
// does not link libcuda directly).
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn get_encode_tiled();  // defined in fa_api.cu
void set_error(const char* fmt, ...);

// One bit per device ordinal (0-63) recording that a per-kernel attribute has
// been set there.  Atomic, so host threads may launch concurrently; two
// threads racing on the first launch both set the (idempotent) attribute.
inline bool device_bit_set(const std::atomic<unsigned long long>& bits, int dev) {
  return dev >= 0 && dev < 64 && ((bits.load(std::memory_order_acquire) >> dev) & 1ull);
}
inline void device_bit_mark(std::atomic<unsigned long long>& bits, int dev) {
  if (dev >= 0 && dev < 64) bits.fetch_or(1ull << dev, std::memory_order_release);
}

// A [B, H, rows, D] view with element strides {sb, sh, sr} and unit inner
// stride, tiled as {chunk elements (128 bytes), box_rows, 1, 1} with 128-byte
// swizzle.  Rows past `rows` read as zero and are clipped on store.
inline bool encode_bhsd(CUtensorMap* map, CUtensorMapDataType dt, const void* ptr, int B, int H, int rows, int D,
                        const long long* st, int chunk, int box_rows) {
  const int esz = dt == CU_TENSOR_MAP_DATA_TYPE_FLOAT32 ? 4 : 2;
  cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)rows, (cuuint64_t)H, (cuuint64_t)B};
  // A stride of an extent-1 dimension is never used; give it a legal value.
  auto legal = [](long long bytes, int extent) -> cuuint64_t {
    return (extent <= 1 || bytes <= 0) ? (cuuint64_t)16 : (cuuint64_t)bytes;
  };
  cuuint64_t strides[3] = {legal(st[2] * esz, rows), legal(st[1] * esz, H), legal(st[0] * esz, B)};
  cuuint32_t box[4] = {(cuuint32_t)chunk, (cuuint32_t)box_rows, 1, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  EncodeTiledFn enc = get_encode_tiled();
  if (!enc) {
    set_error("cuTensorMapEncodeTiled is not available from the CUDA driver");
    return false;
  }
  CUresult r = enc(map, dt, 4,
                   const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    set_error("cuTensorMapEncodeTiled failed (CUresult %d)", (int)r);
    return false;
  }
  return true;
}

// The transposed, tf32-rounded V of the pre-rounded fp32 plans: V^T
// [B, H_kv, D, vt_row] fp32 (vt_row >= kL, a multiple of 4), tiled as
// {32 keys (128 bytes), D rows} with 128-byte swizzle: one K-major column block
// of the O += P V operand per load.  Keys past kL read as zero.
inline bool encode_vt(CUtensorMap* map, const void* ptr, int B, int H, int kL, int D, long long vt_row) {
  cuuint64_t dims[4] = {(cuuint64_t)kL, (cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)B};
  const long long row = vt_row * 4, head = row * D, batch = head * H;
  cuuint64_t strides[3] = {(cuuint64_t)row, (cuuint64_t)(H > 1 ? head : 16), (cuuint64_t)(B > 1 ? batch : 16)};
  cuuint32_t box[4] = {32, (cuuint32_t)D, 1, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  EncodeTiledFn enc = get_encode_tiled();
  if (!enc) {
    set_error("cuTensorMapEncodeTiled is not available from the CUDA driver");
    return false;
  }
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, const_cast<void*>(ptr), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    set_error("cuTensorMapEncodeTiled (V^T) failed (CUresult %d)", (int)r);
    return false;
  }
  return true;
}

// The mask tensor map (when the mask suits TMA) and the kernel's parameter
// block for instantiation C's tiling (its kBM, kNQT and element type).
template <class C>
void setup_params(const LaunchArgs& a, CUtensorMap& tm, FaParams& p) {
  // Mask tiles (128-byte column blocks x kBM rows, 128-byte swizzle) for the
  // L2 prefetch and the shared-memory mask path, when the mask's layout suits
  // TMA (aligned base, 16-byte multiple strides, no stride-0 broadcast).
  int mask_l2 = 0, mask_smem = 0;
  std::memset(&tm, 0, sizeof(tm));
  if (a.mask_kind != 0 && a.mask_vec) {
    const int mesz = a.mask_kind == 1 ? 1 : (C::kTf32 ? 4 : 2);
    const bool fits = a.ms[2] > 0 && (a.ms[1] > 0 || a.Hq == 1) && (a.ms[0] > 0 || a.B == 1);
    if (fits) {
      cuuint64_t dims[4] = {(cuuint64_t)a.kL, (cuuint64_t)a.qL, (cuuint64_t)a.Hq, (cuuint64_t)a.B};
      auto legal = [](long long bytes, int extent) -> cuuint64_t {
        return (extent <= 1 || bytes <= 0) ? (cuuint64_t)16 : (cuuint64_t)bytes;
      };
      cuuint64_t strides[3] = {legal(a.ms[2] * mesz, a.qL), legal(a.ms[1] * mesz, a.Hq), legal(a.ms[0] * mesz, a.B)};
      cuuint32_t box[4] = {(cuuint32_t)(128 / mesz), (cuuint32_t)C::kBM, 1, 1};
      cuuint32_t estr[4] = {1, 1, 1, 1};
      const CUtensorMapDataType dt = a.mask_kind == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                     : C::kTmaType;
      EncodeTiledFn enc = get_encode_tiled();
      if (enc && (C::kBN * mesz) % 128 == 0 &&
          enc(&tm, dt, 4, const_cast<void*>(a.mask), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
              CUDA_SUCCESS) {
        // otherwise the kernel simply reads the mask from global memory
        mask_smem = C::kMaskSlotBytes > 0 ? 1 : 0;
        mask_l2 = mask_smem ? 0 : 1;
      }
    }
  }

  p.B = a.B;
  p.Hq = a.Hq;
  p.Hkv = a.Hkv;
  p.qL = a.qL;
  p.kL = a.kL;
  p.group = a.Hq / a.Hkv;
  // Two Q tiles per unit: two consecutive row tiles of one head, or, with a
  // sliding window or dropout, two heads of one K/V head at the same 128 rows
  // when the query heads per K/V head come in pairs (both tiles then see the
  // same key blocks: measured 154 -> 136 us with a 1024-key window and 779 ->
  // 730 us with dropout 0.1 on the causal B2 H32/8 L4096 D128 workload; the
  // plain causal forward runs 1-2% faster with row pairs).
  p.head_pairs = (C::kNQT == 2 && (a.Hq / a.Hkv) % 2 == 0 && (a.window > 0 || a.dropout_p > 0.0f)) ? 1 : 0;
  p.hq_units = p.head_pairs ? a.Hq / 2 : a.Hq;
  const int unit_rows = p.head_pairs ? C::kBM : C::kBM * C::kNQT;
  p.n_qblocks = (a.qL + unit_rows - 1) / unit_rows;
  p.causal = a.causal;
  p.mask_kind = a.mask_kind;
  p.softcap_on = a.softcap > 0.0f ? 1 : 0;
  p.softcap_in = p.softcap_on ? a.scale / a.softcap : 0.0f;
  p.softcap_out = p.softcap_on ? a.softcap * kLog2e : 0.0f;
  p.dropout_on = a.dropout_p > 0.0f ? 1 : 0;
  p.drop_threshold = p.dropout_on ? (unsigned int)std::ceil((double)a.dropout_p * 16777216.0) : 0u;
  p.drop_scale = a.dropout_p < 1.0f ? (float)(1.0 / (1.0 - (double)a.dropout_p)) : 0.0f;
  p.seed_lo = (unsigned int)a.dropout_seed;
  p.seed_hi = (unsigned int)(a.dropout_seed >> 32);
  p.drop_offset = a.dropout_offset;
  p.window = a.window;
  p.q_offset = a.q_offset;
  // An additive mask with a positive scale may fold as s + mask / scale, so
  // the scores stay in raw units and the softmax's own scale * log2(e) factor
  // applies to both; otherwise scores go to base 2 before the mask.  The raw
  // fold is taken only when 1 / scale is finite and no mask value of the
  // type can overflow mask / scale (headroom 2^8 below the fp32 limit): in
  // practice fp16 masks at any normal scale, never bf16 or fp32 masks, whose
  // largest values (~2^128) would reach infinity.
  const double mask_max = C::kTf32 ? 3.4028234663852886e38 : (C::kF16 ? 65504.0 : 3.3895313892515355e38);
  const float inv_scale = a.scale > 0.0f ? 1.0f / a.scale : 0.0f;
  const bool natural_ok = a.scale > 0.0f && std::isfinite(inv_scale) && mask_max * (double)inv_scale < 0x1p120;
  p.mask_natural = (a.mask_kind == 2 && natural_ok && !p.softcap_on) ? 1 : 0;
  p.inv_scale = p.mask_natural ? inv_scale : 0.0f;
  p.pre_scale = ((a.mask_kind == 2 && !p.mask_natural) || !(a.scale > 0.0f) || p.softcap_on) ? 1 : 0;
  p.mask_vec = a.mask_vec;
  p.mask_l2 = mask_l2;
  p.mask_smem = mask_smem;
  p.scale_log2 = a.scale * kLog2e;
  p.mask = a.mask;
  p.mask_sb = a.ms[0];
  p.mask_sh = a.ms[1];
  p.mask_ss = a.ms[2];
  p.o = a.o;
  p.o_sb = a.os[0];
  p.o_sh = a.os[1];
  p.o_ss = a.os[2];
  p.lse = a.lse;
  p.status = a.status;
  p.timeout_cycles = a.timeout_cycles;
  p.kv_splits = (C::kSplitKV && a.kv_splits > 1) ? a.kv_splits : 1;
  p.kv_chunk = ((a.kL + C::kBN - 1) / C::kBN + p.kv_splits - 1) / p.kv_splits;
  p.part_o = p.kv_splits > 1 ? a.part_o : nullptr;
  p.part_lse = p.kv_splits > 1 ? a.part_lse : nullptr;
}

template <class C>
int launch_fa_fwd(const LaunchArgs& a) {
  CUtensorMap tq, tk, tv, tm;
  if (!encode_bhsd(&tq, C::kTmaType, a.q, a.B, a.Hq, a.qL, a.D, a.qs, C::kChunk, C::kBM)) return 4;
  if (!encode_bhsd(&tk, C::kTmaType, a.k, a.B, a.Hkv, a.kL, a.D, a.ks, C::kChunk, C::kBN)) return 4;
  if constexpr (C::kPre) {
    if (!encode_vt(&tv, a.v, a.B, a.Hkv, a.kL, a.D, a.vt_row)) return 4;
  } else {
    if (!encode_bhsd(&tv, C::kTmaType, a.v, a.B, a.Hkv, a.kL, a.D, a.vs, C::kChunk, C::kBN)) return 4;
  }
  // O as 32-row, 128-byte boxes for the staged epilogue's TMA stores.
  CUtensorMap to;
  std::memset(&to, 0, sizeof(to));
  if constexpr (C::kOStage) {
    if (!encode_bhsd(&to, C::kTmaType, a.o, a.B, a.Hq, a.qL, a.D, a.os, C::kChunk, 32)) return 4;
  }
  FaParams p;
  setup_params<C>(a, tm, p);
  auto kern = fa_fwd_kernel<C>;
  static std::atomic<unsigned long long> configured{0};  // attributes set, per device (per instantiation)
  int dev = 0;
  cudaGetDevice(&dev);
  if (!device_bit_set(configured, dev)) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::kSmemBytes);
    if (e != cudaSuccess) {
      set_error("cudaFuncSetAttribute(max dynamic smem = %u): %s", (unsigned)C::kSmemBytes, cudaGetErrorString(e));
      return 4;
    }
    // The setmaxnreg split inside the kernel assumes this launch register
    // count; a smaller allocation would make the softmax warps' increase wait
    // forever, so refuse to launch instead.
    if (C::kRegsSoftmax > 0) {
      cudaFuncAttributes fattr;
      e = cudaFuncGetAttributes(&fattr, kern);
      if (e != cudaSuccess || fattr.numRegs != C::kRegsLaunch) {
        set_error("kernel register count %d differs from the %d its register split assumes",
                  e == cudaSuccess ? fattr.numRegs : -1, C::kRegsLaunch);
        return 4;
      }
    }
    device_bit_mark(configured, dev);
  }
  // Persistent grid: one CTA per SM (or fewer when capped), each walking its
  // share of the (query block, batch, head) units.
  const long long units = (long long)p.n_qblocks * a.B * p.hq_units * p.kv_splits;
  if (units <= 0 || units > 0x7fffffffLL) {
    set_error("%lld work units are out of range", units);
    return 2;
  }
  long long grid = a.num_sms > 0 ? a.num_sms : 1;
  if (a.max_ctas > 0 && a.max_ctas < grid) grid = a.max_ctas;
  if (grid > units) grid = units;
  kern<<<(unsigned)grid, C::kThreads, C::kSmemBytes, a.stream>>>(tq, tk, tv, tm, to, p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    set_error("kernel launch failed: %s", cudaGetErrorString(e));
    return 4;
  }
  if constexpr (C::kSplitKV) {
    if (p.kv_splits > 1) {  // merge the key ranges into O and L
      const long long threads = (long long)a.B * a.Hq * a.qL * (C::kD / 8);
      fa_splitkv_combine_kernel<C><<<(unsigned)((threads + 255) / 256), 256, 0, a.stream>>>(p);
      e = cudaGetLastError();
      if (e != cudaSuccess) {
        set_error("split-KV combine launch failed: %s", cudaGetErrorString(e));
        return 4;
      }
    }
  }
  return 0;
}

// Per-instantiation configurations (dtype, D) -> tiles, rings and TMEM plan.
//                    tf32   D    Q tiles  BN  K ring  V ring
using CfgBf16D64  = Cfg<false, 64,  2, 128, 4, 4>;  // smem 160 KB, TMEM 384
using CfgBf16D128 = Cfg<false, 128, 2, 128, 2, 2>;  // smem 192 KB, TMEM 512
using CfgBf16D256 = Cfg<false, 256, 1, 128, 1, 1>;  // smem 192 KB, TMEM 512 (P double-buffered)
//                                                 V^T ring (tf32)
using CfgF32D64   = Cfg<true, 64,   2, 64, 2, 2, 2>;  // smem 160 KB, TMEM 256
using CfgF32D128  = Cfg<true, 128,  1, 64, 2, 1, 2>;  // smem 224 KB, TMEM 320
using CfgF32D256  = Cfg<true, 256,  1, 32, 1, 1, 1>;  // smem 224 KB, TMEM 352
// fp32 with the pre-pass (Q, K rounded, V rounded and transposed in HBM): no
// helper warps; the V ring holds K-major V^T tiles.
//                       tf32  D   Q tiles BN K   V  VT  f16    feat   drop   pre
using CfgF32PreD64  = Cfg<true, 64,  1, 64, 4, 4, 0, false, false, false, true>;  // smem 160 KB, TMEM 256
using CfgF32PreD128 = Cfg<true, 128, 1, 64, 3, 2, 0, false, false, false, true>;  // smem 224 KB, TMEM 320
using CfgF32PreD256 = Cfg<true, 256, 1, 32, 2, 1, 0, false, false, false, true>;  // smem 224 KB, TMEM 352
// fp16 I/O: the bf16 plans with the f16 operand format.
using CfgF16D64   = Cfg<false, 64,  2, 128, 4, 4, 0, true>;
using CfgF16D128  = Cfg<false, 128, 2, 128, 2, 2, 0, true>;
using CfgF16D256  = Cfg<false, 256, 1, 128, 1, 1, 0, true>;
// One Q tile per CTA (S and P in their own TMEM columns, S_{j+1} overlapping
// softmax j) for bf16 / fp16 D 64 and 128: chosen when two-tile work units
// cannot fill the GPU, since a one-tile unit's block chain is shorter.
using CfgBf16D64Q1  = Cfg<false, 64,  1, 128, 4, 4>;        // smem 176 KB (incl. mask slot), TMEM 320
using CfgBf16D128Q1 = Cfg<false, 128, 1, 128, 2, 2>;        // smem 192 KB, TMEM 384
using CfgF16D64Q1   = Cfg<false, 64,  1, 128, 4, 4, 0, true>;
using CfgF16D128Q1  = Cfg<false, 128, 1, 128, 2, 2, 0, true>;
// The same plans with sliding window, softcap and query offset compiled in.
template <class C>
using WithFeat = Cfg<C::kTf32, C::kD, C::kNQT, C::kBN, C::kKStages, C::kVStages, C::kVTStages, C::kF16, true>;
template <class C>
using WithDrop = Cfg<C::kTf32, C::kD, C::kNQT, C::kBN, C::kKStages, C::kVStages, C::kVTStages, C::kF16, true, true>;

int launch_bf16_d64(const LaunchArgs& a);
int launch_bf16_d128(const LaunchArgs& a);
int launch_bf16_d256(const LaunchArgs& a);
int launch_f32_d64(const LaunchArgs& a);
int launch_f32_d128(const LaunchArgs& a);
int launch_f32_d256(const LaunchArgs& a);
int launch_f16_d64(const LaunchArgs& a);
int launch_f16_d128(const LaunchArgs& a);
int launch_f16_d256(const LaunchArgs& a);
int launch_q1_bf16_d64(const LaunchArgs& a);
int launch_q1_bf16_d128(const LaunchArgs& a);
int launch_q1_f16_d64(const LaunchArgs& a);
int launch_q1_f16_d128(const LaunchArgs& a);
// Dispatch to the plain or the feature instantiation of a plan.
int launch_feat_bf16_d64(const LaunchArgs& a);
int launch_feat_bf16_d128(const LaunchArgs& a);
int launch_feat_bf16_d256(const LaunchArgs& a);
int launch_feat_f32_d64(const LaunchArgs& a);
int launch_feat_f32_d128(const LaunchArgs& a);
int launch_feat_f32_d256(const LaunchArgs& a);
int launch_feat_f16_d64(const LaunchArgs& a);
int launch_feat_f16_d128(const LaunchArgs& a);
int launch_feat_f16_d256(const LaunchArgs& a);
// ... and of the pre-rounded fp32 plans, with the pre-pass that feeds them
// (defined in fa_tf32_prep.cu).
int launch_pre_f32_d64(const LaunchArgs& a);
int launch_pre_f32_d128(const LaunchArgs& a);
int launch_pre_f32_d256(const LaunchArgs& a);
int launch_tf32_prep(const LaunchArgs& a, float* qr, float* kr, float* vt);
// ... and of the dropout instantiation (the features plus dropout).
int launch_drop_bf16_d64(const LaunchArgs& a);
int launch_drop_bf16_d128(const LaunchArgs& a);
int launch_drop_bf16_d256(const LaunchArgs& a);
int launch_drop_f32_d64(const LaunchArgs& a);
int launch_drop_f32_d128(const LaunchArgs& a);
int launch_drop_f32_d256(const LaunchArgs& a);
int launch_drop_f16_d64(const LaunchArgs& a);
int launch_drop_f16_d128(const LaunchArgs& a);
int launch_drop_f16_d256(const LaunchArgs& a);

}  // namespace fa
