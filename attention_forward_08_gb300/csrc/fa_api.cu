// fa_api.cu -- the C ABI (include/fa.h): argument validation, instantiation
// choice, the per-device status word, and error reporting.
//
// Validation follows mlx-native "ops/flash_attn_train.rs" (`validate_params`:
// every size positive, H_q divisible by H_kv; `dispatch_inner`: head_dim
// checked against the supported set and dtypes checked before dispatch),
// extended with the TMA alignment rules of this library.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "fa.h"
#include "fa_bwd_launch.h"
#include "fa_launch.cuh"

namespace fa {

namespace {

thread_local char g_err[512] = "";

// One status word per device (a static device variable: nothing is allocated).
__device__ unsigned int g_status_word;

constexpr int kMaxDevices = 64;
std::mutex g_mu;
unsigned int* g_status_ptr[kMaxDevices] = {nullptr};
int g_num_sms[kMaxDevices] = {0};
long long g_timeout_cycles = 0;  // 0: not yet initialised
int g_max_ctas = 0;              // 0: one CTA per SM
int g_q_tiles = 0;               // 0: choose per call; 1 or 2: Q tiles per CTA for bf16/fp16 D <= 128
int g_kv_splits = 0;             // 0: choose per call; >= 1: key ranges per query tile (1: no split-KV)
EncodeTiledFn g_encode = nullptr;
bool g_encode_tried = false;

constexpr long long kDefaultTimeout = 1LL << 31;

long long timeout_cycles() {
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_timeout_cycles == 0) {
    g_timeout_cycles = kDefaultTimeout;
    if (const char* s = std::getenv("FA_TIMEOUT_CYCLES")) {
      long long v = std::atoll(s);
      if (v > 0) g_timeout_cycles = v;
    }
  }
  return g_timeout_cycles;
}

// Per-device set-up with that device current: status word address, SM count.
int device_setup(int dev) {
  if (dev < 0 || dev >= kMaxDevices) {
    set_error("device ordinal %d is out of range", dev);
    return FA_ERR_CUDA;
  }
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_status_ptr[dev]) return FA_OK;
  void* ptr = nullptr;
  cudaError_t e = cudaGetSymbolAddress(&ptr, g_status_word);
  if (e != cudaSuccess) {
    set_error("cudaGetSymbolAddress(status word): %s", cudaGetErrorString(e));
    return FA_ERR_CUDA;
  }
  int sms = 0;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) {
    set_error("cudaDeviceGetAttribute(SM count): %s", cudaGetErrorString(e));
    return FA_ERR_CUDA;
  }
  g_num_sms[dev] = sms;
  g_status_ptr[dev] = static_cast<unsigned int*>(ptr);
  return FA_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

// B * H * L > cap for positive B, H, L, without forming the product (which
// can exceed the int64 range): B * H < 2^62 always fits, and
// L > floor(cap / (B * H)) holds exactly when L * B * H > cap.
bool rows_exceed(int B, int H, int L, long long cap) { return (long long)L > cap / ((long long)B * H); }

namespace {

// Words per row of the backward's keep mask: 4 (128 keys) per 128-key block.
long long keep_row_words(int kL) { return ((long long)kL + 127) / 128 * 4; }

// Bytes of a stride that TMA will use (extent-1 dimensions are never stepped).
bool stride_ok(long long elems, int extent, int esz) {
  if (extent <= 1) return true;
  const long long bytes = elems * esz;
  return bytes > 0 && (bytes % 16) == 0 && bytes < (1LL << 40);
}

int validate(const fa_fwd_args* a) {
  if (!a) {
    set_error("args is NULL");
    return FA_ERR_INVALID_ARGUMENT;
  }
  if (!a->q || !a->k || !a->v || !a->o || !a->lse) {
    set_error("q, k, v, o and lse must all be non-NULL");
    return FA_ERR_INVALID_ARGUMENT;
  }
  if (a->B <= 0 || a->H_q <= 0 || a->H_kv <= 0 || a->qL <= 0 || a->kL <= 0) {
    set_error("B (%d), H_q (%d), H_kv (%d), qL (%d) and kL (%d) must be > 0", a->B, a->H_q, a->H_kv, a->qL,
              a->kL);
    return FA_ERR_INVALID_ARGUMENT;
  }
  if (a->H_q % a->H_kv != 0) {
    set_error("H_q (%d) must be divisible by H_kv (%d)", a->H_q, a->H_kv);
    return FA_ERR_INVALID_ARGUMENT;
  }
  if (a->dtype != FA_DTYPE_F32 && a->dtype != FA_DTYPE_BF16 && a->dtype != FA_DTYPE_F16) {
    set_error("dtype %d is not FA_DTYPE_F32 (0), FA_DTYPE_BF16 (1) or FA_DTYPE_F16 (2)", a->dtype);
    return FA_ERR_INVALID_ARGUMENT;
  }
  if (a->mask_kind < FA_MASK_NONE || a->mask_kind > FA_MASK_ADDITIVE) {
    set_error("mask_kind %d is not 0 (none), 1 (bool) or 2 (additive)", a->mask_kind);
    return FA_ERR_INVALID_ARGUMENT;
  }
  if ((a->mask_kind != FA_MASK_NONE) != (a->mask != nullptr)) {
    set_error("mask must be non-NULL exactly when mask_kind != 0 (mask_kind %d, mask %p)", a->mask_kind, a->mask);
    return FA_ERR_INVALID_ARGUMENT;
  }
  if (!std::isfinite(a->scale)) {
    set_error("scale must be finite");
    return FA_ERR_INVALID_ARGUMENT;
  }
  if (a->window < 0) {
    set_error("window (%d) must be >= 0 (0 = no sliding window)", a->window);
    return FA_ERR_INVALID_ARGUMENT;
  }
  if (a->q_offset <= -(1 << 30) || a->q_offset >= (1 << 30)) {
    set_error("q_offset (%d) must lie in (-2^30, 2^30)", a->q_offset);
    return FA_ERR_INVALID_ARGUMENT;
  }
  if (!std::isfinite(a->softcap) || a->softcap < 0.0f) {
    set_error("softcap must be finite and >= 0 (0 = off)");
    return FA_ERR_INVALID_ARGUMENT;
  }
  if (!(a->dropout_p >= 0.0f && a->dropout_p <= 1.0f)) {
    set_error("dropout_p must lie in [0, 1]");
    return FA_ERR_INVALID_ARGUMENT;
  }
  if (a->workspace_bytes < 0 || (a->workspace && (reinterpret_cast<uintptr_t>(a->workspace) & 255u) != 0)) {
    set_error("workspace must be 256-byte aligned and workspace_bytes >= 0");
    return FA_ERR_INVALID_ARGUMENT;
  }
  if (a->dropout_p > 0.0f && a->kL % 4 != 0) {
    set_error("dropout needs kL (%d) to be a multiple of 4", a->kL);
    return FA_ERR_UNSUPPORTED;
  }
  if (a->D != 64 && a->D != 128 && a->D != 256) {
    set_error("head dim D = %d is not supported (64, 128 or 256)", a->D);
    return FA_ERR_UNSUPPORTED;
  }
  // Work units and flat L indices must fit the kernel's int32 arithmetic
  // (key rows too: no device holds a K of 2^31 rows, and the workspace sizes
  // below multiply them).
  if (rows_exceed(a->B, a->H_q, a->qL, 0x7fffffffLL) || rows_exceed(a->B, a->H_kv, a->kL, 0x7fffffffLL)) {
    set_error("B * H_q * qL or B * H_kv * kL exceeds 2^31 - 1");
    return FA_ERR_UNSUPPORTED;
  }
  const int esz = a->dtype == FA_DTYPE_F32 ? 4 : 2;
  if (!aligned16(a->q) || !aligned16(a->k) || !aligned16(a->v) || !aligned16(a->o)) {
    set_error("q, k, v and o must be 16-byte aligned");
    return FA_ERR_MISALIGNED;
  }
  if ((reinterpret_cast<uintptr_t>(a->lse) & 3u) != 0) {
    set_error("lse must be 4-byte aligned");
    return FA_ERR_MISALIGNED;
  }
  struct {
    const long long* s;
    int H, L;
    const char* name;
  } views[4] = {{a->q_strides, a->H_q, a->qL, "q"},
                {a->k_strides, a->H_kv, a->kL, "k"},
                {a->v_strides, a->H_kv, a->kL, "v"},
                {a->o_strides, a->H_q, a->qL, "o"}};
  for (auto& w : views) {
    if (!stride_ok(w.s[0], a->B, esz) || !stride_ok(w.s[1], w.H, esz) || !stride_ok(w.s[2], w.L, esz)) {
      set_error("%s strides {%lld, %lld, %lld} (elements) must be positive multiples of 16 bytes", w.name,
                w.s[0], w.s[1], w.s[2]);
      return FA_ERR_MISALIGNED;
    }
    if (w.s[2] < a->D && w.L > 1) {
      set_error("%s row stride %lld is smaller than D = %d", w.name, w.s[2], a->D);
      return FA_ERR_INVALID_ARGUMENT;
    }
  }
  if (a->mask_kind != FA_MASK_NONE) {
    for (int i = 0; i < 3; ++i)
      if (a->mask_strides[i] < 0) {
        set_error("mask strides must be >= 0");
        return FA_ERR_INVALID_ARGUMENT;
      }
  }
  return FA_OK;
}

long long align256(long long bytes) { return (bytes + 255) / 256 * 256; }

// Workspace of the pre-rounded fp32 plan (0: the plan does not apply).  It
// pays off once every work unit streams many key blocks, where rounding K and
// transposing V per tile in shared memory costs the kernel most; it covers
// the plain forward (masks allowed, no window, softcap, offset or dropout).
long long pre_workspace_bytes(const fa_fwd_args* a) {
  if (a->dtype != FA_DTYPE_F32 || a->window != 0 || a->q_offset != 0 || a->softcap != 0.0f ||
      a->dropout_p != 0.0f || a->kL < 1024 || (long long)a->B * a->H_kv > 65535)
    return 0;
  const long long vt_row = (a->kL + 3) / 4 * 4;
  return align256((long long)a->B * a->H_q * a->qL * a->D * 4) + align256((long long)a->B * a->H_kv * a->kL * a->D * 4) +
         align256((long long)a->B * a->H_kv * a->D * vt_row * 4);
}

// The plan choice for bf16 / fp16 I/O at D <= 128 without window, softcap,
// offset or dropout: one Q tile per CTA when the two-tile work units cannot
// occupy every SM (`sms`: the CTAs the launch may start), or as
// fa_set_q_tiles says.
bool one_tile_plan(const fa_fwd_args* a, int sms) {
  const bool feat = a->dropout_p != 0.0f || a->window != 0 || a->q_offset != 0 || a->softcap != 0.0f;
  if (feat || a->dtype == FA_DTYPE_F32 || a->D > 128) return false;
  int policy;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    policy = g_q_tiles;
  }
  const long long units2 = (long long)((a->qL + 255) / 256) * a->B * a->H_q;
  return policy == 1 || (policy == 0 && units2 < sms);
}

// Key ranges per query tile (split-KV; 1: none) for the one-tile plans:
// automatically when their units leave more than half of the SMs idle, as
// many ranges as fill the SMs with at least 4 key blocks each (at most 64);
// fa_set_kv_splits overrides the count.
int kv_splits_for(const fa_fwd_args* a, int sms) {
  if (sms <= 0 || !one_tile_plan(a, sms)) return 1;
  int forced;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    forced = g_kv_splits;
  }
  const long long units1 = (long long)((a->qL + 127) / 128) * a->B * a->H_q;
  const long long n_kb = (a->kL + 127) / 128;
  long long s = 1;
  if (forced >= 1)
    s = forced;
  else if (units1 * 2 <= sms)
    s = std::min<long long>(sms / units1, n_kb / 4);
  return (int)std::max<long long>(1, std::min<long long>(std::min<long long>(s, n_kb), 64));
}

// Workspace of split-KV with `splits` ranges: the partial O (fp32, D per row)
// and logsumexp of every (range, row).
long long split_rows(const fa_fwd_args* a, int splits) { return (long long)splits * a->B * a->H_q * a->qL; }
long long split_workspace_bytes(const fa_fwd_args* a, int splits) {
  if (splits <= 1) return 0;
  return align256(split_rows(a, splits) * a->D * 4) + align256(split_rows(a, splits) * 4);
}

}  // namespace

void set_error(const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  std::vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
}

EncodeTiledFn get_encode_tiled() {
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_encode_tried) {
    g_encode_tried = true;
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<EncodeTiledFn>(fn);
  }
  return g_encode;
}

int validate_bwd(const fa_bwd_args* a) {
  if (!(a->dropout_p >= 0.0f && a->dropout_p <= 1.0f)) {
    set_error("dropout_p must lie in [0, 1]");
    return FA_ERR_INVALID_ARGUMENT;
  }
  if (a->dropout_p > 0.0f && a->kL % 4 != 0) {
    set_error("dropout needs kL (%d) to be a multiple of 4", a->kL);
    return FA_ERR_UNSUPPORTED;
  }
  if (!(std::isfinite(a->softcap) && a->softcap >= 0.0f)) {
    set_error("softcap must be finite and >= 0 (0 = off)");
    return FA_ERR_INVALID_ARGUMENT;
  }
  if (a->window < 0) {
    set_error("window (%d) must be >= 0 (0 = no sliding window)", a->window);
    return FA_ERR_INVALID_ARGUMENT;
  }
  if (a->q_offset <= -(1 << 30) || a->q_offset >= (1 << 30)) {
    set_error("|q_offset| (%d) must be < 2^30", a->q_offset);
    return FA_ERR_INVALID_ARGUMENT;
  }
  if (!a->q || !a->k || !a->v || !a->o || !a->dout || !a->lse || !a->dq || !a->dk || !a->dv) {
    set_error("q, k, v, o, dout, lse, dq, dk and dv must all be non-NULL");
    return FA_ERR_INVALID_ARGUMENT;
  }
  if (a->B <= 0 || a->H_q <= 0 || a->H_kv <= 0 || a->qL <= 0 || a->kL <= 0) {
    set_error("B (%d), H_q (%d), H_kv (%d), qL (%d) and kL (%d) must be > 0", a->B, a->H_q, a->H_kv, a->qL, a->kL);
    return FA_ERR_INVALID_ARGUMENT;
  }
  if (a->H_q % a->H_kv != 0) {
    set_error("H_q (%d) must be divisible by H_kv (%d)", a->H_q, a->H_kv);
    return FA_ERR_INVALID_ARGUMENT;
  }
  if (!std::isfinite(a->scale)) {
    set_error("scale must be finite");
    return FA_ERR_INVALID_ARGUMENT;
  }
  if (a->mask_kind < FA_MASK_NONE || a->mask_kind > FA_MASK_ADDITIVE) {
    set_error("mask_kind %d is not 0 (none), 1 (bool) or 2 (additive)", a->mask_kind);
    return FA_ERR_INVALID_ARGUMENT;
  }
  if ((a->mask_kind != FA_MASK_NONE) != (a->mask != nullptr)) {
    set_error("mask must be non-NULL exactly when mask_kind != 0 (mask_kind %d, mask %p)", a->mask_kind, a->mask);
    return FA_ERR_INVALID_ARGUMENT;
  }
  if (a->mask_kind != FA_MASK_NONE) {
    for (int i = 0; i < 3; ++i)
      if (a->mask_strides[i] < 0) {
        set_error("mask strides must be >= 0");
        return FA_ERR_INVALID_ARGUMENT;
      }
  }
  if (a->dtype != FA_DTYPE_BF16 && a->dtype != FA_DTYPE_F16 && a->dtype != FA_DTYPE_F32) {
    set_error("dtype %d is not FA_DTYPE_F32 (0), FA_DTYPE_BF16 (1) or FA_DTYPE_F16 (2)", a->dtype);
    return FA_ERR_INVALID_ARGUMENT;
  }
  if (a->dtype == FA_DTYPE_F32 &&
      (a->D == 256 || a->mask_kind != FA_MASK_NONE || a->dropout_p != 0.0f || a->window != 0 || a->q_offset != 0 ||
       a->softcap != 0.0f)) {
    set_error("with fp32 I/O the backward pass takes D = 64 or 128 and causal or full attention only (no mask, "
              "window, q_offset, softcap or dropout)");
    return FA_ERR_UNSUPPORTED;
  }
  if (a->D != 64 && a->D != 128 && a->D != 256) {
    set_error("head dim D = %d is not supported by the backward pass (64, 128 or 256)", a->D);
    return FA_ERR_UNSUPPORTED;
  }
  if (a->D == 256 && (a->mask_kind != FA_MASK_NONE || a->dropout_p != 0.0f || a->window != 0 || a->q_offset != 0 ||
                      a->softcap != 0.0f)) {
    set_error("at D = 256 the backward pass takes causal or full attention only (no mask, window, q_offset, "
              "softcap or dropout)");
    return FA_ERR_UNSUPPORTED;
  }
  if (a->mask_kind != FA_MASK_NONE && a->softcap != 0.0f) {
    set_error("the backward pass does not combine a mask with a softcap");
    return FA_ERR_UNSUPPORTED;
  }
  if (rows_exceed(a->B, a->H_q, a->qL, 0x7fffffffLL) || rows_exceed(a->B, a->H_kv, a->kL, 0x7fffffffLL)) {
    set_error("row counts exceed 2^31 - 1");
    return FA_ERR_UNSUPPORTED;
  }
  const void* ptrs[9] = {a->q, a->k, a->v, a->o, a->dout, a->dq, a->dk, a->dv, a->lse};
  for (const void* ptr : ptrs)
    if (!aligned16(ptr)) {
      set_error("q, k, v, o, dout, lse, dq, dk, dv and workspace must be 16-byte aligned");
      return FA_ERR_MISALIGNED;
    }
  return FA_OK;
}

}  // namespace fa

extern "C" {

int fa_fwd_ex(const fa_fwd_args* a) {
  using namespace fa;
  g_err[0] = '\0';
  int rc = validate(a);
  if (rc != FA_OK) return rc;
  // fp32 with a workspace: round Q and K and transpose V once in HBM, then
  // run the plan that streams them by TMA (no helper warps).
  const long long pre_bytes = pre_workspace_bytes(a);
  if (a->workspace && pre_bytes > 0 && a->workspace_bytes < pre_bytes) {
    set_error("workspace of %lld bytes is smaller than the %lld this call needs (fa_fwd_workspace_bytes)",
              a->workspace_bytes, pre_bytes);
    return FA_ERR_INVALID_ARGUMENT;
  }

  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    set_error("cudaGetDevice: %s", cudaGetErrorString(e));
    return FA_ERR_CUDA;
  }
  rc = device_setup(dev);
  if (rc != FA_OK) return rc;

  LaunchArgs la;
  la.q = a->q;
  la.k = a->k;
  la.v = a->v;
  la.o = a->o;
  la.lse = a->lse;
  la.mask = a->mask;
  la.B = a->B;
  la.Hq = a->H_q;
  la.Hkv = a->H_kv;
  la.qL = a->qL;
  la.kL = a->kL;
  la.D = a->D;
  la.scale = a->scale;
  la.causal = a->causal ? 1 : 0;
  la.mask_kind = a->mask_kind;
  la.window = a->window;
  la.q_offset = a->q_offset;
  la.softcap = a->softcap;
  la.dropout_p = a->dropout_p;
  la.dropout_seed = a->dropout_seed;
  la.dropout_offset = a->dropout_offset;
  for (int i = 0; i < 3; ++i) {
    la.qs[i] = a->q_strides[i];
    la.ks[i] = a->k_strides[i];
    la.vs[i] = a->v_strides[i];
    la.os[i] = a->o_strides[i];
    la.ms[i] = a->mask_kind ? a->mask_strides[i] : 0;
  }
  la.vt_row = 0;
  la.mask_vec = 0;
  if (a->mask_kind != FA_MASK_NONE) {
    const int mesz = (a->mask_kind == FA_MASK_BOOL) ? 1 : (a->dtype == FA_DTYPE_F32 ? 4 : 2);
    bool vec = aligned16(a->mask);
    for (int i = 0; i < 3; ++i) vec = vec && ((la.ms[i] * mesz) % 16 == 0);
    la.mask_vec = vec ? 1 : 0;
  }
  la.stream = static_cast<cudaStream_t>(a->stream);
  la.status = g_status_ptr[dev];
  la.timeout_cycles = timeout_cycles();
  la.num_sms = g_num_sms[dev];
  {
    std::lock_guard<std::mutex> lk(g_mu);
    la.max_ctas = g_max_ctas;
  }

  const bool drop = a->dropout_p != 0.0f;
  const bool feat = drop || a->window != 0 || a->q_offset != 0 || a->softcap != 0.0f;
  // bf16 / fp16 at D <= 128 (no window, softcap or offset): one Q tile per CTA
  // when the two-tile work units cannot occupy every SM; with a workspace,
  // split-KV when even those leave most SMs idle.
  const int sms = la.max_ctas > 0 ? std::min(la.max_ctas, la.num_sms) : la.num_sms;
  const bool one_tile = one_tile_plan(a, sms);
  la.kv_splits = 1;
  la.part_o = nullptr;
  la.part_lse = nullptr;
  const int splits = one_tile ? kv_splits_for(a, sms) : 1;
  if (splits > 1 && a->workspace) {
    const long long need = split_workspace_bytes(a, splits);
    if (a->workspace_bytes < need) {
      set_error("workspace of %lld bytes is smaller than the %lld this call needs (fa_fwd_workspace_bytes)",
                a->workspace_bytes, need);
      return FA_ERR_INVALID_ARGUMENT;
    }
    la.kv_splits = splits;
    la.part_o = static_cast<float*>(a->workspace);
    la.part_lse = reinterpret_cast<float*>(static_cast<uint8_t*>(a->workspace) +
                                           align256(split_rows(a, splits) * a->D * 4));
  }
  if (a->workspace && pre_bytes > 0) {
    uint8_t* ws = static_cast<uint8_t*>(a->workspace);
    float* qr = reinterpret_cast<float*>(ws);
    float* kr = reinterpret_cast<float*>(ws + align256((long long)a->B * a->H_q * a->qL * a->D * 4));
    float* vt = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(kr) +
                                         align256((long long)a->B * a->H_kv * a->kL * a->D * 4));
    la.vt_row = (a->kL + 3) / 4 * 4;
    rc = launch_tf32_prep(la, qr, kr, vt);
    if (rc != FA_OK) return rc;
    const long long Dl = a->D;
    la.q = qr;
    la.qs[0] = (long long)a->H_q * a->qL * Dl;
    la.qs[1] = (long long)a->qL * Dl;
    la.qs[2] = Dl;
    la.k = kr;
    la.ks[0] = (long long)a->H_kv * a->kL * Dl;
    la.ks[1] = (long long)a->kL * Dl;
    la.ks[2] = Dl;
    la.v = vt;
    return a->D == 64 ? launch_pre_f32_d64(la) : a->D == 128 ? launch_pre_f32_d128(la) : launch_pre_f32_d256(la);
  }
  switch (a->dtype) {
    case FA_DTYPE_F32:
      if (drop)
        rc = a->D == 64 ? launch_drop_f32_d64(la) : a->D == 128 ? launch_drop_f32_d128(la) : launch_drop_f32_d256(la);
      else if (feat)
        rc = a->D == 64 ? launch_feat_f32_d64(la) : a->D == 128 ? launch_feat_f32_d128(la) : launch_feat_f32_d256(la);
      else
        rc = a->D == 64 ? launch_f32_d64(la) : a->D == 128 ? launch_f32_d128(la) : launch_f32_d256(la);
      break;
    case FA_DTYPE_F16:
      if (one_tile)
        rc = a->D == 64 ? launch_q1_f16_d64(la) : launch_q1_f16_d128(la);
      else if (drop)
        rc = a->D == 64 ? launch_drop_f16_d64(la) : a->D == 128 ? launch_drop_f16_d128(la) : launch_drop_f16_d256(la);
      else if (feat)
        rc = a->D == 64 ? launch_feat_f16_d64(la) : a->D == 128 ? launch_feat_f16_d128(la) : launch_feat_f16_d256(la);
      else
        rc = a->D == 64 ? launch_f16_d64(la) : a->D == 128 ? launch_f16_d128(la) : launch_f16_d256(la);
      break;
    default:
      if (one_tile)
        rc = a->D == 64 ? launch_q1_bf16_d64(la) : launch_q1_bf16_d128(la);
      else if (drop)
        rc = a->D == 64 ? launch_drop_bf16_d64(la) : a->D == 128 ? launch_drop_bf16_d128(la)
                                                                  : launch_drop_bf16_d256(la);
      else if (feat)
        rc = a->D == 64 ? launch_feat_bf16_d64(la) : a->D == 128 ? launch_feat_bf16_d128(la)
                                                                  : launch_feat_bf16_d256(la);
      else
        rc = a->D == 64 ? launch_bf16_d64(la) : a->D == 128 ? launch_bf16_d128(la) : launch_bf16_d256(la);
      break;
  }
  return rc;
}

long long fa_fwd_workspace_bytes(const fa_fwd_args* a) {
  using namespace fa;
  g_err[0] = '\0';
  if (validate(a) != FA_OK) return -1;
  const long long pre = pre_workspace_bytes(a);
  if (pre > 0) return pre;
  // Split-KV depends on the device's SM count; without a device no plan needs scratch.
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || device_setup(dev) != FA_OK) {
    cudaGetLastError();
    g_err[0] = '\0';
    return 0;
  }
  int max_ctas;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    max_ctas = g_max_ctas;
  }
  const int sms = max_ctas > 0 ? std::min(max_ctas, g_num_sms[dev]) : g_num_sms[dev];
  return split_workspace_bytes(a, kv_splits_for(a, sms));
}

int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H_q, int H_kv, int qL,
           int kL, int D, float scale, int causal, const void* mask, int mask_kind, int dtype, void* stream) {
  fa_fwd_args a;
  std::memset(&a, 0, sizeof(a));
  a.q = q;
  a.k = k;
  a.v = v;
  a.o = o;
  a.lse = lse;
  a.mask = mask;
  a.B = B;
  a.H_q = H_q;
  a.H_kv = H_kv;
  a.qL = qL;
  a.kL = kL;
  a.D = D;
  a.scale = scale;
  a.causal = causal;
  a.mask_kind = mask_kind;
  a.dtype = dtype;
  const long long Dl = D;
  a.q_strides[0] = (long long)H_q * qL * Dl;
  a.q_strides[1] = (long long)qL * Dl;
  a.q_strides[2] = Dl;
  a.o_strides[0] = a.q_strides[0];
  a.o_strides[1] = a.q_strides[1];
  a.o_strides[2] = a.q_strides[2];
  a.k_strides[0] = (long long)H_kv * kL * Dl;
  a.k_strides[1] = (long long)kL * Dl;
  a.k_strides[2] = Dl;
  a.v_strides[0] = a.k_strides[0];
  a.v_strides[1] = a.k_strides[1];
  a.v_strides[2] = a.k_strides[2];
  a.mask_strides[0] = (long long)H_q * qL * kL;
  a.mask_strides[1] = (long long)qL * kL;
  a.mask_strides[2] = kL;
  a.stream = stream;
  return fa_fwd_ex(&a);
}

const char* fa_last_error(void) { return fa::g_err; }

int fa_sync_status(void* stream) {
  using namespace fa;
  g_err[0] = '\0';
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) {
    set_error("stream synchronise: %s", cudaGetErrorString(e));
    return FA_ERR_CUDA;
  }
  int rc = device_setup(dev);
  if (rc != FA_OK) return rc;
  unsigned int word = 0;
  e = cudaMemcpy(&word, g_status_ptr[dev], sizeof(word), cudaMemcpyDeviceToHost);
  if (e == cudaSuccess && word != 0) {
    const unsigned int zero = 0;
    e = cudaMemcpy(g_status_ptr[dev], &zero, sizeof(zero), cudaMemcpyHostToDevice);
  }
  if (e != cudaSuccess) {
    set_error("status word read: %s", cudaGetErrorString(e));
    return FA_ERR_CUDA;
  }
  if (word & kStatusTimeout) {
    set_error("a kernel reached its wait bound and stopped early (status 0x%x)", word);
    return FA_ERR_DEVICE_TIMEOUT;
  }
  return FA_OK;
}

void fa_set_timeout_cycles(long long cycles) {
  std::lock_guard<std::mutex> lk(fa::g_mu);
  fa::g_timeout_cycles = cycles > 0 ? cycles : fa::kDefaultTimeout;
}

void fa_set_q_tiles(int n) {
  std::lock_guard<std::mutex> lk(fa::g_mu);
  fa::g_q_tiles = (n == 1 || n == 2) ? n : 0;
}

void fa_set_kv_splits(int n) {
  std::lock_guard<std::mutex> lk(fa::g_mu);
  fa::g_kv_splits = n >= 1 ? n : 0;
}

void fa_set_max_ctas(int n) {
  std::lock_guard<std::mutex> lk(fa::g_mu);
  fa::g_max_ctas = n > 0 ? n : 0;
}

long long fa_bwd_workspace_bytes(int B, int H_q, int qL) {
  if (B <= 0 || H_q <= 0 || qL <= 0 || fa::rows_exceed(B, H_q, qL, 0x7fffffffLL)) return -1;
  const long long bytes = (long long)B * H_q * qL * 4;
  return (bytes + 255) / 256 * 256;
}

namespace {
// Queries per key row of the backward's key-major mask copy: whole 128-row
// query blocks, so a block's 128 entries never leave the row.
long long mask_t_ld(int qL) { return ((long long)qL + 127) / 128 * 128; }
long long align256_ll(long long bytes) { return (bytes + 255) / 256 * 256; }
}  // namespace

long long fa_bwd_ex_workspace_bytes(int B, int H_q, int qL, int kL, float dropout_p) {
  const long long dvec = fa_bwd_workspace_bytes(B, H_q, qL);
  if (dvec < 0 || kL <= 0 || !(dropout_p >= 0.0f && dropout_p <= 1.0f)) return -1;
  if (dropout_p == 0.0f) return dvec;
  // keep mask: 4 words (128 keys) per row and 128-key block
  return dvec + (long long)B * H_q * qL * fa::keep_row_words(kL) * 4;
}

long long fa_bwd_full_workspace_bytes(const fa_bwd_args* a) {
  using namespace fa;
  g_err[0] = '\0';
  if (!a) {
    set_error("args is NULL");
    return -1;
  }
  if (validate_bwd(a) != FA_OK) return -1;
  const long long base = fa_bwd_ex_workspace_bytes(a->B, a->H_q, a->qL, a->kL, a->dropout_p);
  if (a->dtype == FA_DTYPE_F32)
    return align256_ll(base) + bwd_tf32_layout(a->B, a->H_q, a->H_kv, a->qL, a->kL, a->D).bytes;
  if (a->mask_kind == FA_MASK_NONE) return base;
  if (a->mask_kind == FA_MASK_BOOL)  // keep bits, key-major then row-major
    return align256_ll(base) + align256_ll((long long)a->B * a->H_q * a->kL * (mask_t_ld(a->qL) / 32) * 4) +
           align256_ll((long long)a->B * a->H_q * a->qL * keep_row_words(a->kL) * 4);
  return align256_ll(base) + align256_ll((long long)a->B * a->H_q * a->kL * mask_t_ld(a->qL) * 2);
}

int fa_bwd_full(const fa_bwd_args* args) {
  using namespace fa;
  g_err[0] = '\0';
  if (!args) {
    set_error("args is NULL");
    return FA_ERR_INVALID_ARGUMENT;
  }
  const fa_bwd_args& x = *args;
  int rc = validate_bwd(&x);
  if (rc != FA_OK) return rc;
  if (!x.workspace) {
    set_error("workspace must be non-NULL");
    return FA_ERR_INVALID_ARGUMENT;
  }
  const long long ws_need = fa_bwd_full_workspace_bytes(&x);
  if (x.workspace_bytes < ws_need) {
    set_error("workspace of %lld bytes is smaller than the %lld required", x.workspace_bytes, ws_need);
    return FA_ERR_INVALID_ARGUMENT;
  }
  if (!aligned16(x.workspace) || (x.mask_kind != FA_MASK_NONE && (reinterpret_cast<uintptr_t>(x.workspace) & 255u))) {
    set_error(x.mask_kind != FA_MASK_NONE ? "workspace must be 256-byte aligned" : "workspace must be 16-byte aligned");
    return FA_ERR_MISALIGNED;
  }
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    set_error("cudaGetDevice: %s", cudaGetErrorString(e));
    return FA_ERR_CUDA;
  }
  rc = device_setup(dev);
  if (rc != FA_OK) return rc;
  BwdLaunchArgs a;
  a.q = x.q;
  a.k = x.k;
  a.v = x.v;
  a.o = x.o;
  a.dout = x.dout;
  a.lse = x.lse;
  a.dq = x.dq;
  a.dk = x.dk;
  a.dv = x.dv;
  a.dvec = static_cast<float*>(x.workspace);
  a.f16 = x.dtype == FA_DTYPE_F16;
  a.f32 = x.dtype == FA_DTYPE_F32;
  a.t32_ws = a.f32 ? static_cast<char*>(x.workspace) + align256_ll(fa_bwd_workspace_bytes(x.B, x.H_q, x.qL)) : nullptr;
  a.B = x.B;
  a.Hq = x.H_q;
  a.Hkv = x.H_kv;
  a.qL = x.qL;
  a.kL = x.kL;
  a.D = x.D;
  a.scale = x.scale;
  a.causal = x.causal ? 1 : 0;
  a.window = x.window;
  a.q_offset = x.q_offset;
  a.softcap = x.softcap;
  a.dropout_p = x.dropout_p;
  a.dropout_seed = x.dropout_seed;
  a.dropout_offset = x.dropout_offset;
  a.keep_row_words = keep_row_words(x.kL);
  const long long base = fa_bwd_ex_workspace_bytes(x.B, x.H_q, x.qL, x.kL, x.dropout_p);
  a.keep_mask = x.dropout_p > 0.0f ? reinterpret_cast<uint32_t*>(static_cast<char*>(x.workspace) +
                                                                 fa_bwd_workspace_bytes(x.B, x.H_q, x.qL))
                                   : nullptr;
  a.mask_kind = x.mask_kind;
  a.mask = x.mask;
  for (int i = 0; i < 3; ++i) a.ms[i] = x.mask_kind ? x.mask_strides[i] : 0;
  char* mask_ws = static_cast<char*>(x.workspace) + align256_ll(base);
  a.mask_t = x.mask_kind == FA_MASK_ADDITIVE ? mask_ws : nullptr;
  a.mask_t_ld = mask_t_ld(x.qL);
  a.mask_tbits_ld = mask_t_ld(x.qL) / 32;
  a.mask_rbits_ld = keep_row_words(x.kL);
  a.mask_tbits = x.mask_kind == FA_MASK_BOOL ? reinterpret_cast<uint32_t*>(mask_ws) : nullptr;
  a.mask_rbits = x.mask_kind == FA_MASK_BOOL
                     ? reinterpret_cast<uint32_t*>(mask_ws + align256_ll((long long)x.B * x.H_q * x.kL *
                                                                          a.mask_tbits_ld * 4))
                     : nullptr;
  a.mask_vec = 0;
  if (x.mask_kind != FA_MASK_NONE) {
    const int mesz = x.mask_kind == FA_MASK_BOOL ? 1 : 2;
    bool vec = aligned16(x.mask);
    for (int i = 0; i < 3; ++i) vec = vec && ((a.ms[i] * mesz) % 16 == 0);
    a.mask_vec = vec ? 1 : 0;
  }
  a.stream = static_cast<cudaStream_t>(x.stream);
  a.status = g_status_ptr[dev];
  a.timeout_cycles = timeout_cycles();
  return launch_bwd(a);
}

int fa_bwd_ex(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse,
              void* dq, void* dk, void* dv, void* workspace, long long workspace_bytes, int B, int H_q, int H_kv,
              int qL, int kL, int D, float scale, int causal, int window, int q_offset, float softcap,
              float dropout_p, unsigned long long dropout_seed, unsigned long long dropout_offset, int dtype,
              void* stream) {
  if (dtype == FA_DTYPE_F32) {  // its workspace size depends on more than this entry's sizing function sees
    fa::set_error("fa_bwd and fa_bwd_ex take bf16 and fp16 I/O; fp32 goes through fa_bwd_full");
    return FA_ERR_UNSUPPORTED;
  }
  fa_bwd_args a;
  std::memset(&a, 0, sizeof(a));
  a.q = q;
  a.k = k;
  a.v = v;
  a.o = o;
  a.dout = dout;
  a.lse = lse;
  a.dq = dq;
  a.dk = dk;
  a.dv = dv;
  a.workspace = workspace;
  a.workspace_bytes = workspace_bytes;
  a.B = B;
  a.H_q = H_q;
  a.H_kv = H_kv;
  a.qL = qL;
  a.kL = kL;
  a.D = D;
  a.scale = scale;
  a.causal = causal;
  a.window = window;
  a.q_offset = q_offset;
  a.softcap = softcap;
  a.dropout_p = dropout_p;
  a.dropout_seed = dropout_seed;
  a.dropout_offset = dropout_offset;
  a.dtype = dtype;
  a.stream = stream;
  return fa_bwd_full(&a);
}

int fa_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse, void* dq,
           void* dk, void* dv, void* workspace, long long workspace_bytes, int B, int H_q, int H_kv, int qL, int kL,
           int D, float scale, int causal, int dtype, void* stream) {
  return fa_bwd_ex(q, k, v, o, dout, lse, dq, dk, dv, workspace, workspace_bytes, B, H_q, H_kv, qL, kL, D, scale,
                   causal, 0, 0, 0.0f, 0.0f, 0ull, 0ull, dtype, stream);
}

int fa_version(void) { return 111; }

}  // extern "C"
