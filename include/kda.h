/*
 * kda.h -- C ABI of the GB300 (sm_103a) Kimi Delta Attention forward.
 *
 * The operator (one independent chain per sequence n and head h):
 *
 *     S = h0[n,h]  (dk x dv, or zeros)
 *     for each token t of the sequence, in order:
 *         S   <- diag(exp(g_t)) S                   channel-wise forget gate
 *         S   <- S + beta_t k_t (v_t - S^T k_t)^T   delta-rule write
 *         o_t  = scale * S^T q_t                    read-out after the write
 *     hT[n,h] = S
 *
 * Sources: "Kimi K3 技术报告摘要" (gkm0120.cn/p/60370.html), section 1
 * 预训练 Recipe, 训练策略 table, KDA row (delta-rule recurrence with a
 * channel-wise forget gate, computed chunk-wise: parallel inside a chunk,
 * recurrent across chunks); "Kimi K3 NPU Training", section 模型结构 (L2
 * normalised q/k, per-channel decay and beta; a fixed matrix state per head
 * at decode) and section 定长与 TND (the state resets at every packed
 * sequence boundary; cu_seqlens).  g carries log(alpha) in natural-log units.
 *
 * Conventions shared by every entry point:
 *   - The caller owns every buffer.  The library allocates no memory.  Every
 *     entry point except kda_fwd_noalloc keeps no global state and is
 *     reentrant; kda_fwd_noalloc keeps its scratch in one fixed array per
 *     device (see there).
 *   - Tensor pointers are DEVICE pointers, 16-byte aligned, dense and
 *     row-major with the innermost dimension contiguous.  Activations are
 *     token-major [B, T, H, d]; a packed batch is [1, T_total, H, d] with
 *     int32 cu_seqlens[N+1].  States are float32 [N, H, dk, dv], dv fastest.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *     default stream).  No host synchronisation except in
 *     kda_read_device_status().
 *   - Host-checkable argument errors return before anything is launched.
 *     Launch failures return KDA_ERR_CUDA.  Errors found on the device
 *     (malformed cu_seqlens, a bounded wait that ran out) are latched in the
 *     workspace status word; read them with kda_read_device_status().
 *   - `out` must not alias any input.  `hT` may alias `h0`.
 */
#ifndef KDA_H_
#define KDA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  KDA_OK = 0,
  KDA_ERR_INVALID_ARG = 1,    /* null pointer, bad size, misalignment, B/T/H out of range */
  KDA_ERR_UNSUPPORTED = 2,    /* valid but not implemented (e.g. dk != dv, d not 64/128) */
  KDA_ERR_WORKSPACE = 3,      /* workspace missing, misaligned or smaller than kda_workspace_size */
  KDA_ERR_CUDA = 4,           /* a CUDA call or kernel launch failed */
  KDA_ERR_BAD_SEQLENS = 5,    /* device: cu_seqlens not non-decreasing from 0 to T */
  KDA_ERR_DEVICE_TIMEOUT = 6, /* device: a bounded wait inside a kernel ran out */
  KDA_ERR_DECAY_RANGE = 7     /* not raised: kept for compatibility (every gate in [-inf, 0]
                                 is supported; see kda_fwd) */
} kda_status;

typedef enum { KDA_F32 = 0, KDA_BF16 = 1 } kda_dtype;

typedef struct {
  int32_t B;            /* fixed length: batch size.  Packed: must be 1. */
  int32_t T;            /* tokens per sequence (fixed) or total tokens (packed), >= 0 */
  int32_t H;            /* heads, >= 1 */
  int32_t dk, dv;       /* head dims; supported: dk == dv in {64, 128} */
  int32_t num_seqs;     /* packed: N = number of sequences; ignored when cu_seqlens is NULL */
  kda_dtype in_dtype;   /* dtype of q, k, v, g, beta (all the same) */
  kda_dtype out_dtype;  /* dtype of o; KDA_F32 recommended (bf16 output rounding alone
                           costs about 2^-9 of each output) */
  float scale;          /* read-out scale, usually dk^-1/2 */
} kda_shape;

/* Bytes of workspace that let kda_fwd / kda_decode use every path for `s`
 * (always >= 256: the first 256 bytes hold the device status word; num_seqs > 0
 * counts as a packed call, which for a fixed-length call only over-estimates).
 * For a fixed-length bf16 batch with fewer (sequence, head) chains than SMs and
 * long sequences this includes the segment states of the long-chain split: each
 * chain is cut into up to 64 segments joined through their affine state maps (the
 * first up to 3 times as long as the others), as a model of the work items' schedule
 * on the current device's SMs favours (152, a GB300's count, when no device can be
 * queried), and 3 * nseg - 2 float32 dk x dv states per chain are reserved.  The minimum a call accepts is 256
 * bytes plus, for packed batches, 4 bytes per sequence rounded up to 64
 * sequences; with less than kda_workspace_size the split is skipped.  Returns 0
 * if `s` is NULL. */
size_t kda_workspace_size(const kda_shape* s);

/*
 * Chunkwise prefill over fixed-length or packed variable-length sequences.
 *
 *   q, k, g  [B,T,H,dk]   in_dtype.  q and k L2-normalised per (token, head);
 *                         g = log(alpha) <= 0; -inf (alpha = 0) is allowed.
 *   v        [B,T,H,dv]   in_dtype.
 *   beta     [B,T,H]      in_dtype, in [0, 1].
 *   cu_seqlens  device int32 [num_seqs+1] or NULL (fixed length, N = B).
 *   h0       device float32 [N,H,dk,dv] start states, or NULL for zeros.
 *   out      device [B,T,H,dv] out_dtype.
 *   hT       device float32 [N,H,dk,dv] final states, or NULL.
 *   workspace   device, 256-byte aligned, kda_workspace_size(s) bytes (or at
 *               least the minimum described there); contents on entry do not
 *               matter.
 * When B*T == 0 the activation pointers may be NULL (hT is still written).
 * Chunks of 64 tokens start at each sequence start; the last chunk of a
 * sequence may be partial.  A zero-length sequence writes hT = h0 (or 0).
 * The float32 path (in_dtype KDA_F32) evaluates every product in float32;
 * the bf16 path uses tensor cores with split bf16 operands and float32
 * accumulation.  A 64-token chunk in which some key channel decays by more
 * than about 160 nats (alpha near 0) cannot be factorised within float32's
 * exponent range; the bf16 path runs such a chunk token by token on the CUDA
 * cores (same results, about four times the time of a tensor-core chunk).
 */
kda_status kda_fwd(const kda_shape* s, const void* q, const void* k, const void* v,
                   const void* g, const void* beta, const int32_t* cu_seqlens,
                   const float* h0, void* out, float* hT, void* workspace,
                   size_t workspace_bytes, void* stream);

/*
 * kda_fwd plus prefix-cache checkpoints: the state of every (sequence, head)
 * after each `interval` tokens of its sequence ("Kimi K3 模型结构（7）：结构决定
 * 系统", section 前缀缓存: prefix hashes are cut into 512-token blocks and KDA state
 * checkpoints are kept at hash-block end points, so a cache hit can land on any
 * 512-token boundary).
 *
 * Same arguments and results as kda_fwd, plus:
 *   interval      tokens between checkpoints, a positive multiple of 64 (the
 *                 pages use 512).
 *   ckpt          device float32 [ckpt_rows, H, dk, dv], the same [dk][dv] layout
 *                 as hT.  Row base_n + j - 1 holds the state of sequence n after
 *                 its first j * interval tokens, j = 1 .. floor(len_n / interval).
 *   ckpt_offsets  device int32 [N+1] for packed batches: base_n = ckpt_offsets[n]
 *                 and ckpt_offsets[n+1] - ckpt_offsets[n] = floor(len_n / interval).
 *                 Ignored (may be NULL) for fixed-length batches, where
 *                 base_n = n * floor(T / interval).
 *   ckpt_rows     rows in ckpt.
 * Offsets that disagree with a sequence's length, or rows past ckpt_rows, latch
 * KDA_ERR_INVALID_ARG in the workspace status word; that sequence then writes no
 * checkpoints (its o and hT are still computed).  Each checkpoint adds 4*dk*dv
 * bytes of writes per (sequence, head).  Host-checkable errors: interval not a
 * positive multiple of 64, ckpt NULL or not 16-byte aligned, ckpt_rows < 0, a
 * packed batch without ckpt_offsets -> KDA_ERR_INVALID_ARG; otherwise those of
 * kda_fwd.
 */
kda_status kda_fwd_checkpoints(const kda_shape* s, const void* q, const void* k, const void* v,
                               const void* g, const void* beta, const int32_t* cu_seqlens,
                               const float* h0, void* out, float* hT, int32_t interval,
                               float* ckpt, const int32_t* ckpt_offsets, int64_t ckpt_rows,
                               void* workspace, size_t workspace_bytes, void* stream);

/*
 * Input preprocessing fused into the kernels ("Kimi K3 NPU Training", section
 * 模型结构, steps 1 and 3: q/k are L2 normalised and the channel-wise decay and
 * beta are built from the projected gate inputs).  Each enabled step is
 * computed in float32 from the values passed in.  The gate and beta are then
 * rounded to in_dtype, as a separate pass that stores in_dtype tensors would
 * (the bf16 path's cumulative sum takes a bf16 gate); the normalised q and k
 * enter the float32 products unrounded:
 *   qk_l2norm      q, k per (token, head):  x / max(||x||_2, 1e-12)
 *   gate_softplus  g holds the raw gate:    log(alpha) = -softplus(g),
 *                  softplus(x) = log(1 + e^x) (absolute error below 4e-7
 *                  before rounding; it equals x once log1p(e^-x) rounds away)
 *   beta_sigmoid   beta holds the raw value: beta = 1 / (1 + e^-beta)
 *                  (a few float32 ulp)
 *   gate_scale     device float32 [H] or NULL (= 1): with gate_softplus,
 *                  log(alpha) = -gate_scale[h] * softplus(g) (a per-head
 *                  scale of the decay rate); non-NULL without gate_softplus
 *                  is KDA_ERR_INVALID_ARG.  4-byte aligned.
 *   gate_per_head  the scalar-gate (Gated DeltaNet) variant: g is [.., H], one
 *                  gate per token and head (raw, or log(alpha) without
 *                  gate_softplus), shared by all dk key channels; g then needs
 *                  only in_dtype alignment.
 * The norm uses rsqrt (a few ulp).  A zero-initialised struct disables
 * everything (plain kda_fwd / kda_decode).
 */
typedef struct {
  int32_t qk_l2norm;
  int32_t gate_softplus;
  int32_t beta_sigmoid;
  int32_t gate_per_head;
  const float* gate_scale;
} kda_preproc;

/* kda_fwd with the preprocessing `pre` (NULL = none) applied to q, k, g, beta
 * inside the kernels.  Arguments, results and errors as kda_fwd. */
kda_status kda_fwd_preproc(const kda_shape* s, const kda_preproc* pre, const void* q,
                           const void* k, const void* v, const void* g, const void* beta,
                           const int32_t* cu_seqlens, const float* h0, void* out, float* hT,
                           void* workspace, size_t workspace_bytes, void* stream);

/* kda_decode with the preprocessing `pre` (NULL = none).  Arguments, results and
 * errors as kda_decode. */
kda_status kda_decode_preproc(const kda_shape* s, const kda_preproc* pre, const void* q,
                              const void* k, const void* v, const void* g, const void* beta,
                              float* state, void* out, void* workspace, size_t workspace_bytes,
                              void* stream);

/*
 * Backward of kda_fwd: the gradients of L = sum(o * dout) + sum(hT * dhT) with
 * respect to q, k, v, g (= log alpha), beta and h0 ("Kimi K3 NPU Training",
 * section NPU 算子支持度, row KDA 反向: dq, dk, dv, dbeta, dgate and dstate).
 * Shapes, dtypes and cu_seqlens as kda_fwd (scale included; out_dtype is not
 * used), and:
 *   dout     device float32 [B,T,H,dv]   cotangent of o
 *   dhT      device float32 [N,H,dk,dv]  cotangent of the final states, or NULL (0)
 *   h0       device float32 [N,H,dk,dv]  start states, or NULL (zeros)
 *   dq, dk, dg  device float32 [B,T,H,dk];  dv device float32 [B,T,H,dv];
 *   dbeta    device float32 [B,T,H];  dh0 device float32 [N,H,dk,dv] or NULL
 *   workspace   device, 256-byte aligned, at least kda_bwd_workspace_size(s)
 *               bytes: per 16-token sub-chunk and head it holds the start state
 *               (dk x dv), X and U (16 x dv) and T and P (16 x 16), float32.
 * Everything is computed in float32 (inputs converted exactly).  The forward
 * is recomputed inside the call, so the o and hT of a previous kda_fwd are not
 * needed.  Gates must be finite.  Device-detected errors (malformed
 * cu_seqlens) are latched as in kda_fwd.
 */
size_t kda_bwd_workspace_size(const kda_shape* s);
kda_status kda_bwd(const kda_shape* s, const void* q, const void* k, const void* v,
                   const void* g, const void* beta, const int32_t* cu_seqlens, const float* h0,
                   const float* dout, const float* dhT, float* dq, float* dk, float* dv,
                   float* dg, float* dbeta, float* dh0, void* workspace, size_t workspace_bytes,
                   void* stream);

/*
 * Decode step: T_step = s->T tokens (1..8) per sequence applied in order to a
 * state pool resident in device memory, updated in place (the replay form of
 * speculative-decode rollback: the cached inputs of the accepted tokens are
 * re-applied on chip; "Kimi K3 模型结构（7）：结构决定系统", section KDA 状态回滚).
 *
 *   q, k, g  [B,T_step,H,dk], v [B,T_step,H,dv], beta [B,T_step,H]   in_dtype
 *   state    device float32 [B,H,dk,dv], read and written in place
 *   out      device [B,T_step,H,dv] out_dtype (one output per token)
 * B is the number of sequences; cu_seqlens is not used.
 */
kda_status kda_decode(const kda_shape* s, const void* q, const void* k, const void* v,
                      const void* g, const void* beta, float* state, void* out,
                      void* workspace, size_t workspace_bytes, void* stream);

/*
 * Decode step with per-sequence commit counts, for speculative decoding: the
 * cached inputs of a step are replayed on chip, and only the state after the
 * accepted prefix is kept ("Kimi K3 模型结构（7）：结构决定系统", section KDA
 * 状态回滚: cache the small projected inputs instead of per-position state
 * snapshots, and rebuild the accepted tokens' state by replay; replay and
 * verification share one kernel).
 *
 * Same arguments as kda_decode, plus:
 *   num_commit  device int32 [B]; for sequence n, the state written back to
 *               `state` is the one after its first num_commit[n] tokens, each in
 *               0..T_step (0 leaves the state unchanged: a verification pass;
 *               T_step is kda_decode).  All T_step tokens are still applied in
 *               order to produce their outputs.
 *   out         device [B,T_step,H,dv] out_dtype, or NULL for no outputs (a pure
 *               replay).
 * A count outside 0..T_step latches KDA_ERR_INVALID_ARG in the workspace status
 * word and leaves that sequence's state unchanged; its outputs are still
 * written.  Host-checkable errors are those of kda_decode.
 */
kda_status kda_decode_commit(const kda_shape* s, const void* q, const void* k, const void* v,
                             const void* g, const void* beta, const int32_t* num_commit,
                             float* state, void* out, void* workspace, size_t workspace_bytes,
                             void* stream);

/*
 * kda_fwd without a workspace, for callers that cannot allocate device memory:
 * code whose device memory is planned in full by a host framework before it
 * runs and that may not request more at call time, or bindings that cannot
 * reach a device allocator at all.  The pages describe no such entry point;
 * it has no counterpart there.
 *
 * Same arguments and results as kda_fwd, minus the workspace.  The scratch
 * (status word and packed-batch sequence order) lives in a fixed array inside
 * the library: 256 + 4 * 16384 bytes of device memory per GPU that loads the
 * library, held until the process exits.  Limits and behaviour:
 *   - packed batches of more than 16384 sequences return KDA_ERR_UNSUPPORTED
 *     before anything is launched;
 *   - the first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current; make that first call
 *     before any stream capture;
 *   - nothing is allocated: no cudaMalloc, no cudaFree, no allocating library
 *     routine;
 *   - every call on a device shares the one array, and each call clears the
 *     status word it needs when it starts; calls whose work overlaps on the GPU
 *     (other streams, or other host threads) race on the array, so serialise
 *     them;
 *   - the array's address is looked up once per device and kept for the life
 *     of the process; do not use this entry point on a device after
 *     cudaDeviceReset (or any other teardown of its primary context);
 *   - a fixed-length batch whose few long chains kda_fwd would cut into
 *     segments (the segment states need a workspace of kda_workspace_size)
 *     runs every chain whole here: same results, but a batch like B=1,
 *     T=2^20, H=32 takes several times longer than through kda_fwd;
 *   - status_out: optional DEVICE pointer to one unsigned int; when non-NULL,
 *     the call's device status (KDA_OK or a device error code) is copied there
 *     in stream order after the kernels.
 */
kda_status kda_fwd_noalloc(const kda_shape* s, const void* q, const void* k, const void* v,
                           const void* g, const void* beta, const int32_t* cu_seqlens,
                           const float* h0, void* out, float* hT, unsigned int* status_out,
                           void* stream);

/* Synchronises `stream`, then returns (and clears) the status latched in the
 * workspace by the kernels of the latest kda_fwd / kda_decode call that used
 * it (each call clears the word when it starts): KDA_OK or a device error. */
kda_status kda_read_device_status(void* workspace, void* stream);

/* Self-test of the device-side bounded waits: launches one tiny kernel that
 * waits on a barrier nothing completes, gives up after about 1 ms and latches
 * KDA_ERR_DEVICE_TIMEOUT in the workspace status word (read it with
 * kda_read_device_status).  The wait never traps and the context stays
 * usable.  workspace: device, 256-byte aligned, >= 256 bytes. */
kda_status kda_selftest_bounded_wait(void* workspace, void* stream);

/* Static description of a status code; never NULL. */
const char* kda_status_string(kda_status st);

/* Library version, e.g. "kda-gb300 0.1". */
const char* kda_version(void);

#ifdef __cplusplus
}
#endif
#endif /* KDA_H_ */
