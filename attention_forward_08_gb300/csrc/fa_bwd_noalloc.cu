// fa_bwd_noalloc.cu -- fa_bwd_noalloc: the backward pass with its scratch (the
// per-row D = rowsum(O * dO) vector) taken from a fixed device array compiled
// into the library instead of a caller workspace.  Nothing is allocated: the
// array's address is looked up once per device with cudaGetSymbolAddress.
#include <cuda_runtime.h>

#include <cstring>
#include <mutex>

#include "fa.h"
#include "fa_bwd_launch.h"
#include "fa_launch.cuh"

namespace {

// Largest B * H_q * qL the built-in scratch holds (one fp32 per query row: 8 MiB).
constexpr long long kNoAllocRows = 1LL << 21;

// The scratch: fully written by the D pre-pass before anything reads it, so it
// never needs clearing.
static __device__ __align__(256) float g_bwd_scratch[kNoAllocRows];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
float* g_scratch_ptr[kMaxDevices] = {nullptr};

}  // namespace

extern "C" int fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const void* dout,
                              const float* lse, void* dq, void* dk, void* dv, int B, int H_q, int H_kv, int qL,
                              int kL, int D, float scale, int causal, int dtype, void* stream) {
  // One factor at a time: B * H_q * qL itself may not fit in 64 bits.
  if (B > 0 && H_q > 0 && qL > 0 && fa::rows_exceed(B, H_q, qL, kNoAllocRows)) {
    fa::set_error("B * H_q * qL query rows exceed the %lld rows of fa_bwd_noalloc's built-in scratch; "
                  "call fa_bwd with a workspace instead",
                  kNoAllocRows);
    return FA_ERR_UNSUPPORTED;
  }
  // The remaining argument checks come before any CUDA call, as for fa_bwd.
  fa_bwd_args chk;
  std::memset(&chk, 0, sizeof(chk));
  chk.q = q;
  chk.k = k;
  chk.v = v;
  chk.o = o;
  chk.dout = dout;
  chk.lse = lse;
  chk.dq = dq;
  chk.dk = dk;
  chk.dv = dv;
  chk.B = B;
  chk.H_q = H_q;
  chk.H_kv = H_kv;
  chk.qL = qL;
  chk.kL = kL;
  chk.D = D;
  chk.scale = scale;
  chk.causal = causal;
  chk.dtype = dtype;
  int rc = fa::validate_bwd(&chk);
  if (rc != FA_OK) return rc;
  if (dtype == FA_DTYPE_F32) {  // the fp32 plans need a workspace for their rounded copies
    fa::set_error("fa_bwd_noalloc takes bf16 and fp16 I/O; fp32 goes through fa_bwd_full");
    return FA_ERR_UNSUPPORTED;
  }
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    fa::set_error("cudaGetDevice: %s", cudaGetErrorString(e));
    return FA_ERR_CUDA;
  }
  if (dev < 0 || dev >= kMaxDevices) {
    fa::set_error("device ordinal %d is out of range", dev);
    return FA_ERR_CUDA;
  }
  float* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (!g_scratch_ptr[dev]) {
      void* ptr = nullptr;
      e = cudaGetSymbolAddress(&ptr, g_bwd_scratch);
      if (e != cudaSuccess) {
        fa::set_error("cudaGetSymbolAddress(backward scratch): %s", cudaGetErrorString(e));
        return FA_ERR_CUDA;
      }
      g_scratch_ptr[dev] = static_cast<float*>(ptr);
    }
    scratch = g_scratch_ptr[dev];
  }
  return fa_bwd(q, k, v, o, dout, lse, dq, dk, dv, scratch, kNoAllocRows * (long long)sizeof(float), B, H_q,
                H_kv, qL, kL, D, scale, causal, dtype, stream);
}
