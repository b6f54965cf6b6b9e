/*
 * fa.h -- C ABI of the GB300 (sm_103a) FlashAttention-2 library: the forward
 * pass (fa_fwd, fa_fwd_ex) and its gradients (fa_bwd).
 *
 * The operation (per batch b, query head h, query row i):
 *
 *   kvh  = h / (H_q / H_kv)                                  GQA, no K/V copy
 *   S_ij = scale * q[b,h,i,:] . k[b,kvh,j,:] (+ mask[b,h,i,j] if additive)
 *   key j is excluded when causal and j > i (top-left aligned), when a bool
 *   mask entry is 0, or when an additive mask makes S_ij = -inf
 *   O[b,h,i,:] = sum_j softmax_j(S_i.) * v[b,kvh,j,:]
 *   L[b,h,i]   = m_i + ln(l_i)   (natural-log logsumexp of the allowed S_ij)
 *   a row with no allowed key gets O = 0 and L = -inf.
 *
 * Defined by: mlx-native "ops/flash_attn_train.rs" (module doc "Algorithm":
 * FA-2 forward emitting O and L = m + ln(l), the FA-2 Algorithm 1
 * logsumexp; "Buffer layout": Q/O [B,H_q,qL,D], K/V [B,H_kv,kL,D], mask
 * [B,H_q,qL,kL], L [B,H_q,qL] fp32; `FlashAttnTrainParams` and
 * `validate_params`), forge "flash_attention_mma.metal" (causal bound and
 * GQA map), ruDNN "dense_attention.rs" (`forward`: mask kind 1 keeps nonzero
 * entries, kind 2 adds the value, additive -inf excludes the key) and
 * oxibonsai "dit_attention_flash.rs" (head-major input, token-major output).
 *
 * Memory: every pointer is caller-owned DEVICE memory on the current CUDA
 * device.  The library allocates nothing per call and keeps no reference to
 * the buffers after the kernel finishes.  o and lse must not overlap any
 * input.  Calls are asynchronous on `stream` (a cudaStream_t; NULL = the
 * legacy default stream).
 *
 * Errors: arguments are validated before anything is launched; on error
 * nothing is written and a non-zero fa_status is returned, with a message
 * available from fa_last_error() on the calling thread.  A kernel that
 * hits its internal wait bound stops early and raises a device status bit
 * that fa_sync_status() reports as FA_ERR_DEVICE_TIMEOUT.
 */
#ifndef FA_GB300_FA_H
#define FA_GB300_FA_H

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FA_DTYPE_F32 = 0,  /* fp32 I/O, tensor-core products in TF32 (inputs rounded to nearest) */
  FA_DTYPE_BF16 = 1, /* bf16 I/O, fp32 accumulation, P rounded to bf16 before P.V */
  FA_DTYPE_F16 = 2   /* fp16 I/O, fp32 accumulation, P rounded to fp16 before P.V (forward only) */
} fa_dtype;

typedef enum {
  FA_MASK_NONE = 0,
  FA_MASK_BOOL = 1,     /* uint8, nonzero = keep the key */
  FA_MASK_ADDITIVE = 2  /* same dtype as q; added after scaling; -inf excludes the key */
} fa_mask_kind;

typedef enum {
  FA_OK = 0,
  FA_ERR_INVALID_ARGUMENT = 1, /* null pointer, non-positive size, H_q % H_kv != 0, bad enum, non-finite scale */
  FA_ERR_UNSUPPORTED = 2,      /* head dim not in {64, 128, 256}, or sizes beyond the kernel's index range */
  FA_ERR_MISALIGNED = 3,       /* q/k/v/o base or row/head/batch stride not a multiple of 16 bytes */
  FA_ERR_CUDA = 4,             /* a CUDA runtime/driver call failed (message says which) */
  FA_ERR_DEVICE_TIMEOUT = 5    /* a kernel stopped at its wait bound (reported by fa_sync_status) */
} fa_status;

/*
 * fa_fwd -- contiguous layouts:
 *   q, o   [B, H_q, qL, D]   (dtype)
 *   k, v   [B, H_kv, kL, D]  (dtype)
 *   lse    [B, H_q, qL]      fp32, natural-log logsumexp L
 *   mask   [B, H_q, qL, kL]  mask_kind 1: uint8; mask_kind 2: dtype; NULL when mask_kind 0
 * D must be 64, 128 or 256.  scale is typically 1/sqrt(D).
 * Returns an fa_status.
 */
int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H_q, int H_kv, int qL,
           int kL, int D, float scale, int causal, const void* mask, int mask_kind, int dtype, void* stream);

/*
 * fa_fwd_ex -- the same operation on strided views.  Each *_strides array
 * holds ELEMENT strides {batch, head, row}; the innermost (D, or key for the
 * mask) stride is 1.  q/k/v/o strides times the element size must be
 * multiples of 16 bytes (TMA).  Mask strides are free, and 0 broadcasts that
 * dimension.  lse stays contiguous [B, H_q, qL].
 * Example: head-major q/k/v [H, seq, D] with token-major output
 * o[seq, H*D] is B = 1 with o_strides = {seq*H*D, D, H*D}.
 * The last three fields extend the operation (all zero = the plain forward):
 *   window > 0  sliding window: key j allowed only if j > i + q_offset - window
 *               (forge "flash_attention_mma.metal" names the field `window`);
 *   q_offset    the causal diagonal of row i is key i + q_offset (mlx-native
 *               `ql_off`); kL - qL aligns the last query with the last key;
 *   softcap > 0 scores become softcap * tanh(scale * q.k / softcap) before
 *               any mask (mlx-native `softcapping`); L is the logsumexp of
 *               the capped scores.
 * window must be >= 0, |q_offset| < 2^30, softcap finite and >= 0.
 *   dropout_p   in [0, 1]; > 0 multiplies each weight P_ij of O by 0 or
 *               1 / (1 - p) (ruDNN "dense_attention.rs", `keep`): position
 *               ((b*H_q + h)*qL + i)*kL + j, Philox4x32-10 keyed by
 *               dropout_seed on the counter dropout_offset + position / 4,
 *               word position % 4, kept iff (word >> 8) * 2^-24 >= p.  L and
 *               the softmax normaliser are unaffected.  kL must be a
 *               multiple of 4 (else FA_ERR_UNSUPPORTED).
 */
typedef struct fa_fwd_args {
  const void* q;
  const void* k;
  const void* v;
  void* o;
  float* lse;
  const void* mask;
  int B, H_q, H_kv, qL, kL, D;
  float scale;
  int causal;
  int mask_kind;
  int dtype;
  long long q_strides[3];
  long long k_strides[3];
  long long v_strides[3];
  long long o_strides[3];
  long long mask_strides[3];
  void* stream; /* cudaStream_t */
  /* Added in ABI 1.03 (zero = off; zero-initialise the struct): */
  int window;    /* > 0: sliding window, key j allowed only if j > i + q_offset - window */
  int q_offset;  /* causal diagonal of row i is key i + q_offset (0: top-left; kL - qL: bottom-right) */
  float softcap; /* > 0: each scaled score s becomes softcap * tanh(s / softcap), before any mask */
  /* Added in ABI 1.04 (zero = off): */
  float dropout_p;                   /* keep each weight of O with probability 1 - p, scaled by 1/(1-p) */
  unsigned long long dropout_seed;   /* generator key */
  unsigned long long dropout_offset; /* generator counter of position 0 */
  /* Added in ABI 1.06 (NULL / 0 = none): */
  void* workspace;           /* optional caller-owned device scratch, 256-byte aligned */
  long long workspace_bytes; /* its size in bytes */
} fa_fwd_args;

int fa_fwd_ex(const fa_fwd_args* args);

/*
 * fa_fwd_workspace_bytes -- device scratch that lets fa_fwd_ex run the faster
 * plan for these arguments (all fields filled as for the call), or 0 when no
 * plan needs one; -1 (with the message set) when the arguments are invalid.
 * Split-KV (fa_set_kv_splits; it depends on the current device's SM count and
 * fa_set_max_ctas, so ask again after changing either): 4 * S * B*H_q*qL * D
 * bytes of partial O and 4 * S * B*H_q*qL of partial logsumexp, each rounded
 * up to 256, for S key ranges.  Also: fp32 I/O (TF32) without window, softcap, offset or dropout and with
 * kL >= 1024, where the library rounds Q and K to tf32 and transposes V once
 * into the workspace (one extra launch) instead of per tile inside the kernel:
 * 4 * (B*H_q*qL*D + B*H_kv*kL*D + B*H_kv*D*ceil4(kL)) bytes, each part rounded
 * up to 256.  Results are the same either way (both round to nearest before
 * the products).  fa_fwd_ex uses the workspace when workspace is non-NULL and
 * this function returns > 0; a non-NULL workspace smaller than that is
 * FA_ERR_INVALID_ARGUMENT.  The contents on entry do not matter; they are
 * clobbered, and the workspace must not overlap any argument.
 */
long long fa_fwd_workspace_bytes(const fa_fwd_args* args);

/* Message for the last non-FA_OK return on the calling thread ("" if none). */
const char* fa_last_error(void);

/*
 * fa_sync_status -- synchronise `stream`, then read and clear the device
 * status word of the current device.  FA_OK if no kernel stopped early since
 * the last call, FA_ERR_DEVICE_TIMEOUT if one did, FA_ERR_CUDA on a CUDA
 * error (including an earlier asynchronous kernel fault).
 */
int fa_sync_status(void* stream);

/*
 * fa_set_timeout_cycles -- bound (in SM clock cycles) on every wait inside
 * the kernel; <= 0 restores the default (2^31 cycles, about one second).
 * The environment variable FA_TIMEOUT_CYCLES sets the initial value.
 */
void fa_set_timeout_cycles(long long cycles);

/*
 * fa_set_max_ctas -- the forward kernel is persistent: by default it starts
 * one CTA per SM and each CTA walks a balanced share of the (query block,
 * batch, head) work units.  n > 0 caps the number of CTAs (for example to
 * leave SMs to work on other streams); n <= 0 restores one per SM.  Results
 * do not depend on it.
 */
void fa_set_max_ctas(int n);

/*
 * fa_set_q_tiles -- for bf16 / fp16 I/O at D <= 128 without window, softcap
 * or offset, each CTA owns two 128-row Q tiles (their softmax ping-pongs on
 * the tensor core) unless that leaves SMs without work, in which case it
 * owns one (shorter per-unit critical path).  n = 1 or 2 forces that choice,
 * any other value restores the automatic one.  Results do not depend on it.
 */
void fa_set_q_tiles(int n);

/*
 * fa_set_kv_splits -- split-KV for the one-Q-tile plans (bf16 / fp16 I/O,
 * D <= 128, masks allowed; no window, softcap, offset or dropout): each 128-row query
 * tile's key blocks are cut into n ranges, each its own work unit, which
 * writes its range's normalised O (fp32) and logsumexp to the workspace; a
 * second launch merges the ranges (O = sum_s w_s O_s / sum_s w_s, w_s =
 * exp(L_s - max L), L = max L + log sum_s w_s: the same softmax, rounded
 * once to the I/O type).  It applies only when fa_fwd_ex gets a workspace of
 * fa_fwd_workspace_bytes; without one the call runs unsplit.  n >= 1 forces
 * n ranges (at most one per key block, at most 64; 1: off); any other value
 * restores the automatic choice: split when the one-tile units would leave
 * more than half of the SMs idle (few, long query tiles: decoding-like
 * shapes), into as many ranges as fill the SMs with at least 4 key blocks
 * each.  Results agree with the unsplit plan to rounding.
 */
void fa_set_kv_splits(int n);

/*
 * fa_bwd_workspace_bytes -- bytes of device workspace fa_bwd needs for
 * B * H_q * qL query rows: one fp32 D_i = rowsum(O_i * dO_i) per row, rounded
 * up to 256 bytes.  Returns -1 for non-positive sizes.
 */
long long fa_bwd_workspace_bytes(int B, int H_q, int qL);

/*
 * fa_bwd -- gradients of the forward pass (FlashAttention-2 backward).
 *
 * Given dout = dLoss/dO, computes (kvh = h / (H_q / H_kv))
 *   P_ij  = exp(scale * q_i . k_j - L_i)        causal keys j > i excluded
 *   D_i   = rowsum(O_i * dO_i)
 *   dS_ij = P_ij * (dO_i . v_j - D_i)
 *   dq[b,h,i,:]   = scale * sum_j dS_ij k[b,kvh,j,:]
 *   dk[b,kvh,j,:] = scale * sum over the group's heads h and rows i of dS_ij q[b,h,i,:]
 *   dv[b,kvh,j,:] =         sum over the group's heads h and rows i of P_ij dout[b,h,i,:]
 * Defined by forge "flash_attention_mma.metal", section "backward (MMA)"
 * (dQ query-parallel; dK/dV key-parallel on transposed products, summed over
 * the query heads sharing a K/V head, no atomics) and mlx-native
 * "ops/flash_attn_train.rs", section "Phase 2 -- FA-2 backward kernel (dQ,
 * dK, dV)" (the D = rowsum(O * dO) pre-pass and the buffer shapes).
 *
 * Arguments: q, o, dout, dq [B,H_q,qL,D]; k, v, dk, dv [B,H_kv,kL,D]; all
 * contiguous bf16 or fp16 (dtype FA_DTYPE_BF16 or FA_DTYPE_F16; P and dS are
 * rounded to that format before their products), 16-byte aligned.  lse
 * [B,H_q,qL] fp32 is the forward's L (natural log; -inf rows get zero
 * gradients).  o is the forward's output.  workspace: caller-owned device
 * memory of at least fa_bwd_workspace_bytes(B, H_q, qL) bytes, 16-byte
 * aligned; its contents on entry do not matter and are clobbered.  D must be
 * 64, 128 or 256 (else FA_ERR_UNSUPPORTED); no mask here (fa_bwd_full takes
 * one).  At D = 256 the backward takes causal or full attention only: the
 * window, offset, softcap, dropout and mask of fa_bwd_ex and fa_bwd_full
 * return FA_ERR_UNSUPPORTED there.  dq, dk, dv are written in full (rows no
 * query or key reaches get zeros) and must not overlap any input or each
 * other.  Asynchronous on `stream`: three kernel launches (D pre-pass, dK/dV,
 * dQ); validation and errors as for fa_fwd.
 */
int fa_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse,
           void* dq, void* dk, void* dv, void* workspace, long long workspace_bytes, int B, int H_q, int H_kv,
           int qL, int kL, int D, float scale, int causal, int dtype, void* stream);

/*
 * fa_bwd_ex_workspace_bytes -- bytes of scratch fa_bwd_ex needs: those of
 * fa_bwd_workspace_bytes, plus, when dropout_p > 0, the keep decisions of
 * every (row, key) pair as a bit mask, 16 bytes per row and 128-key block
 * (B * H_q * qL * ceil(kL / 128) * 16 bytes).  -1 for non-positive sizes or
 * dropout_p outside [0, 1].  Pure function of its arguments.
 */
long long fa_bwd_ex_workspace_bytes(int B, int H_q, int qL, int kL, float dropout_p);

/*
 * fa_bwd_ex -- fa_bwd for a forward that used a sliding window, a causal
 * diagonal offset and/or a softcap (fa_fwd_args.window, .q_offset, .softcap,
 * same meaning and limits: window >= 0, |q_offset| < 2^30, softcap finite
 * and >= 0): key j takes part in row i's softmax only if j <= i + q_offset
 * (causal) and j > i + q_offset - window (window > 0); with softcap c > 0
 * the scores are t = c tanh(scale q.k / c), so dS carries the factor
 * 1 - tanh^2 (recovered from P and L).  dropout_p, dropout_seed and
 * dropout_offset are the forward's (the fa_fwd_args fields of the same names;
 * p outside [0, 1]: FA_ERR_INVALID_ARGUMENT; p > 0 with kL not a multiple of
 * 4: FA_ERR_UNSUPPORTED).  The backward regenerates the forward's keep
 * decisions Z_ij in {0, 1 / (1 - p)} from the same counter-based generator,
 * so that dV = (P Z)^T dO and dS = P (Z dP - D) with D = rowsum(dO O), O the
 * forward's (dropped) output: the chain rule through the forward's dropout
 * (ruDNN "dense_attention.rs", `keep`).  The workspace must hold
 * fa_bwd_ex_workspace_bytes(B, H_q, qL, kL, dropout_p) bytes (with dropout
 * the decisions are drawn once into it, by a fourth launch, and read by both
 * gradient kernels).  All zero is fa_bwd.  Arguments, results and errors
 * otherwise as fa_bwd.
 */
int fa_bwd_ex(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse,
              void* dq, void* dk, void* dv, void* workspace, long long workspace_bytes, int B, int H_q, int H_kv,
              int qL, int kL, int D, float scale, int causal, int window, int q_offset, float softcap,
              float dropout_p, unsigned long long dropout_seed, unsigned long long dropout_offset, int dtype,
              void* stream);

/*
 * fa_bwd_noalloc -- fa_bwd without a workspace argument (no counterpart on the
 * pages; a convenience of this library).  The D vector lives in a device array
 * compiled into the library, sized for B * H_q * qL <= 2^21 query rows (8 MiB
 * of fp32); larger problems return FA_ERR_UNSUPPORTED with a message, before
 * anything is launched.  Nothing is allocated: the array's address is looked
 * up once per device.  The array is fully written before it is read, so it
 * needs no clearing.  All calls on a device share that one array: calls that
 * overlap in time (on different streams or host threads) race and produce
 * wrong gradients.  Arguments, results and errors otherwise as fa_bwd.
 */
int fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse,
                   void* dq, void* dk, void* dv, int B, int H_q, int H_kv, int qL, int kL, int D, float scale,
                   int causal, int dtype, void* stream);

/*
 * fa_bwd_args / fa_bwd_full -- the backward pass with every option of the
 * forward in one argument block (ABI 1.09).  The fields mean what the fa_bwd
 * and fa_bwd_ex arguments of the same names mean; zero-initialise the struct
 * and fill what the forward used.  Added here:
 *   mask, mask_kind, mask_strides -- the forward's mask, with the
 *     fa_fwd_args conventions: mask_kind FA_MASK_BOOL (uint8, nonzero keeps
 *     the key) or FA_MASK_ADDITIVE (the I/O dtype, added to the scaled score,
 *     -inf excludes the key); element strides {batch, head, row} with unit key
 *     stride, 0 broadcasting that dimension; mask NULL exactly when mask_kind
 *     is FA_MASK_NONE.  The gradients are those of the masked softmax the
 *     forward computed (ruDNN "dense_attention.rs", `backward` and
 *     `backward_kv_owned`: mask kinds 1 and 2 with the same `allowed` and
 *     additive rules as its `forward`):
 *     P_ij = exp(scale q_i.k_j + m_ij - L_i), 0 where the key is excluded, so
 *     excluded keys and rows without any allowed key get zero gradient.  A
 *     mask together with a softcap is FA_ERR_UNSUPPORTED.
 *   dtype FA_DTYPE_F32 -- fp32 inputs and gradients, the products on the
 *     TF32 tensor cores (inputs, P and dS rounded to tf32, accumulation in
 *     fp32), following forge "flash_attention_mma.metal", section "backward
 *     (MMA)" (an fp32 backward with separate dQ, dV and dK kernels).  D 64 or
 *     128, causal or full attention, GQA; a mask, window, q_offset, softcap
 *     or dropout with fp32 is FA_ERR_UNSUPPORTED.  Only this entry point takes
 *     fp32 (fa_bwd, fa_bwd_ex and fa_bwd_noalloc return FA_ERR_UNSUPPORTED).
 * Scratch: fa_bwd_full_workspace_bytes(args) bytes, 256-byte aligned: the
 * D vector, the dropout keep decisions (dropout_p > 0) and, with a mask, a
 * key-major copy of the mask for the key-parallel kernel (B * H_q * kL *
 * ceil(qL / 128) * 128 elements), each part starting on a 256-byte boundary;
 * a fifth launch writes that copy.  fp32: after the D vector, tf32-rounded
 * copies of q, dout [B,H_q,qL,D] and k, v [B,H_kv,kL,D], then the rounded
 * transposes of q and dout [B,H_q,D,ceil(qL/4)*4] and of k
 * [B,H_kv,D,ceil(kL/4)*4] (each part 256-byte aligned; eight pre-pass
 * launches, then the dV, dK and dQ kernels).  Results and errors otherwise as
 * fa_bwd_ex.
 */
typedef struct fa_bwd_args {
  const void* q;
  const void* k;
  const void* v;
  const void* o;
  const void* dout;
  const float* lse;
  void* dq;
  void* dk;
  void* dv;
  void* workspace;           /* 256-byte aligned, fa_bwd_full_workspace_bytes(args) bytes */
  long long workspace_bytes;
  int B, H_q, H_kv, qL, kL, D;
  float scale;
  int causal;
  int window;
  int q_offset;
  float softcap;
  float dropout_p;
  unsigned long long dropout_seed;
  unsigned long long dropout_offset;
  const void* mask;
  int mask_kind;
  long long mask_strides[3];
  int dtype;
  void* stream; /* cudaStream_t */
} fa_bwd_args;

int fa_bwd_full(const fa_bwd_args* args);

/* Bytes of scratch fa_bwd_full needs for these arguments; -1 (with the message
 * set) when they are invalid. */
long long fa_bwd_full_workspace_bytes(const fa_bwd_args* args);

/* ABI version: major * 100 + minor (1.05: fa_bwd and fa_bwd_noalloc accept
 * FA_DTYPE_F16; 1.06: fa_fwd_args.workspace, fa_fwd_workspace_bytes; 1.07:
 * fa_bwd_ex; 1.08: fa_bwd_ex takes the forward's dropout arguments,
 * fa_bwd_ex_workspace_bytes; 1.09: fa_bwd_args, fa_bwd_full with masks;
 * 1.10: the backward at D = 256; 1.11: fa_set_kv_splits). */
int fa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FA_GB300_FA_H */
