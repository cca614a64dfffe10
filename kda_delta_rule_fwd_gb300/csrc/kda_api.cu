// C ABI entry points: argument validation, workspace carving and dispatch.
// Every check that can be made on the host is made before anything is
// launched; nothing here allocates memory.
#include <stdio.h>

#include "kda_internal.cuh"

using namespace kda;

namespace {

bool aligned(const void* p, size_t a) { return ((uintptr_t)p % a) == 0; }

size_t dsize(kda_dtype t) { return t == KDA_F32 ? 4 : 2; }

// Shape checks shared by prefill and decode.
kda_status check_shape(const kda_shape* s, bool packed) {
  if (!s) return KDA_ERR_INVALID_ARG;
  if (s->H < 1 || s->T < 0 || s->dk < 1 || s->dv < 1) return KDA_ERR_INVALID_ARG;
  if (packed ? (s->B != 1 || s->num_seqs < 0) : s->B < 0) return KDA_ERR_INVALID_ARG;
  if ((s->in_dtype != KDA_F32 && s->in_dtype != KDA_BF16) ||
      (s->out_dtype != KDA_F32 && s->out_dtype != KDA_BF16))
    return KDA_ERR_INVALID_ARG;
  if (!(s->scale == s->scale)) return KDA_ERR_INVALID_ARG;  // NaN scale
  if (s->dk != s->dv || (s->dk != 64 && s->dk != 128)) return KDA_ERR_UNSUPPORTED;
  // the largest index used is (B*T*H) * d; keep it well inside int64 and the grid
  const int64_t toks = (int64_t)s->B * s->T;
  if (toks > ((int64_t)1 << 40) / ((int64_t)s->H * s->dk)) return KDA_ERR_INVALID_ARG;
  return KDA_OK;
}

// The minimum workspace: status header plus, for a packed call, the order list
// (num_seqs is ignored otherwise).  The long-chain segment states are optional
// (the split is skipped without them).
kda_status check_ws(const kda_shape* s, void* ws, size_t bytes, bool packed) {
  if (!ws || !aligned(ws, 256)) return KDA_ERR_WORKSPACE;
  size_t need = kWsHeader;
  if (packed && s->num_seqs > 0) need += ws_order_bytes(s->num_seqs);
  if (bytes < need) return KDA_ERR_WORKSPACE;
  return KDA_OK;
}

// SMs of the current device for the segment plan, looked up once per device;
// 152 (a GB300) when there is no device to ask, so sizes computed without a
// GPU match a GB300's.
int64_t device_sms() {
  constexpr int kMaxDev = 64;
  static int64_t cache[kMaxDev] = {};
  int dev = -1, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) {
    cudaGetLastError();  // clear the error a device-less host leaves behind
    return kGb300Sms;
  }
  if (dev < kMaxDev && cache[dev] > 0) return cache[dev];
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
    cudaGetLastError();
    return kGb300Sms;
  }
  if (dev < kMaxDev) cache[dev] = n;
  return n;
}

}  // namespace

extern "C" {

size_t kda_workspace_size(const kda_shape* s) {
  if (!s) return 0;
  size_t b = kWsHeader;
  const bool bf16_d128 = s->in_dtype == KDA_BF16 && s->dk == 128 && s->dv == 128;
  if (s->num_seqs > 0) {
    // packed: the order list, then (long enough batches) the split plan and states
    b += ws_order_bytes(s->num_seqs);
    if (s->H > 0 && packed_split_possible(bf16_d128, s->T)) {
      const int64_t nsx = packed_ns_max(s->T);
      b += packed_plan_bytes(s->num_seqs, nsx) + packed_state_bytes(nsx, s->H, s->dk);
    }
    return b;
  }
  // fixed-length batches of a few very long chains also keep segment states
  const int64_t chains = (int64_t)(s->B > 0 ? s->B : 0) * (s->H > 0 ? s->H : 0);
  b += seg_bytes(seg_plan(false, bf16_d128, chains, s->T, device_sms()), chains, s->dk);
  return b;
}

namespace {
// shared by kda_fwd and kda_fwd_checkpoints (ckpt == nullptr: no checkpoints)
Preproc to_preproc(const kda_preproc* p) {
  Preproc r{0, 0, 0, 0, nullptr};
  if (p) {
    r.l2 = p->qk_l2norm != 0;
    r.gate = p->gate_softplus != 0;
    r.beta = p->beta_sigmoid != 0;
    r.per_head = p->gate_per_head != 0;
    r.gate_scale = p->gate_scale;
  }
  return r;
}
// the preprocessing's own argument rules; g's alignment follows its layout
bool preproc_ok(const kda_preproc* p, const void* g, kda_dtype in_dtype) {
  const bool per_head = p && p->gate_per_head;
  if (g && !aligned(g, per_head ? dsize(in_dtype) : 16)) return false;
  if (p && p->gate_scale && (!p->gate_softplus || !aligned(p->gate_scale, 4))) return false;
  return true;
}

kda_status fwd_common(const kda_shape* s, const void* q, const void* k, const void* v,
                      const void* g, const void* beta, const int32_t* cu_seqlens,
                      const float* h0, void* out, float* hT, float* ckpt,
                      const int32_t* ckpt_offsets, int64_t ckpt_rows, int32_t ckpt_interval,
                      const kda_preproc* pre, void* workspace, size_t workspace_bytes,
                      void* stream) {
  const bool packed = cu_seqlens != nullptr;
  kda_status st = check_shape(s, packed);
  if (st != KDA_OK) return st;
  // with no tokens the activation buffers are empty and may be NULL
  const bool any_tokens = (int64_t)s->B * s->T > 0;
  if (any_tokens && (!q || !k || !v || !g || !beta || !out)) return KDA_ERR_INVALID_ARG;
  const void* ptrs[] = {q, k, v, out, h0, hT};
  for (const void* p : ptrs)
    if (p && !aligned(p, 16)) return KDA_ERR_INVALID_ARG;
  if (!aligned(beta, dsize(s->in_dtype)) || (packed && !aligned(cu_seqlens, 4)) ||
      !preproc_ok(pre, g, s->in_dtype))
    return KDA_ERR_INVALID_ARG;
  st = check_ws(s, workspace, workspace_bytes, packed);
  if (st != KDA_OK) return st;

  FwdArgs a{};
  a.q = q; a.k = k; a.v = v; a.g = g; a.beta = beta;
  a.cu = cu_seqlens; a.h0 = h0; a.out = out; a.hT = hT;
  a.T = s->T;
  a.N = packed ? s->num_seqs : s->B;
  a.H = s->H;
  a.D = s->dk;
  a.scale = s->scale;
  a.in_dtype = s->in_dtype;
  a.out_dtype = s->out_dtype;
  a.status = static_cast<unsigned int*>(workspace);
  a.ckpt = ckpt;
  a.ckpt_off = ckpt_offsets;
  a.ckpt_rows = ckpt_rows;
  a.ckpt_interval = ckpt_interval;
  a.pre = to_preproc(pre);
  a.stream = static_cast<cudaStream_t>(stream);
  a.sms = device_sms();

  // the status word and the kernels' work counters start at zero
  if (cudaMemsetAsync(workspace, 0, kWsHeader, a.stream) != cudaSuccess) return KDA_ERR_CUDA;
  if (packed) {
    char* w = static_cast<char*>(workspace);
    int32_t* order = reinterpret_cast<int32_t*>(w + kWsHeader);
    if (launch_schedule(a, order) != cudaSuccess) return KDA_ERR_CUDA;
    a.order = order;
    // long-chain split of the longest sequences, planned on the device, when the
    // workspace holds the plan and the segment states
    const bool bf16_d128 = s->in_dtype == KDA_BF16 && s->dk == 128;
    if (packed_split_possible(bf16_d128, s->T)) {
      const int64_t nsx = packed_ns_max(s->T);
      const size_t at = kWsHeader + ws_order_bytes(s->num_seqs);
      const size_t plan = packed_plan_bytes(s->num_seqs, nsx);
      if (workspace_bytes >= at + plan + packed_state_bytes(nsx, s->H, s->dk)) {
        a.pplan = w + at;
        a.ns_max = nsx;
        a.seg_ws = reinterpret_cast<float*>(w + at + plan);
        if (launch_plan_packed(a) != cudaSuccess) return KDA_ERR_CUDA;
      }
    }
  } else {
    // long-chain split: segment states follow the header when the plan asks for them
    const bool bf16_d128 = s->in_dtype == KDA_BF16 && s->dk == 128;
    const SegPlan pl = seg_plan(false, bf16_d128, (int64_t)s->B * s->H, s->T, device_sms());
    const size_t need = kWsHeader + seg_bytes(pl, (int64_t)s->B * s->H, s->dk);
    if (pl.nseg > 1 && workspace_bytes >= need) {
      a.seg_ws = reinterpret_cast<float*>(static_cast<char*>(workspace) + kWsHeader);
      a.plan = pl;
    }
  }
  cudaError_t e;
  if (s->in_dtype == KDA_BF16 && s->dk == 128)
    e = launch_prefill_bf16(a);
  else
    e = launch_prefill_f32(a);
  return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}
}  // namespace

kda_status kda_fwd(const kda_shape* s, const void* q, const void* k, const void* v,
                   const void* g, const void* beta, const int32_t* cu_seqlens,
                   const float* h0, void* out, float* hT, void* workspace,
                   size_t workspace_bytes, void* stream) {
  return fwd_common(s, q, k, v, g, beta, cu_seqlens, h0, out, hT, nullptr, nullptr, 0, 0,
                    nullptr, workspace, workspace_bytes, stream);
}

kda_status kda_fwd_preproc(const kda_shape* s, const kda_preproc* pre, const void* q,
                           const void* k, const void* v, const void* g, const void* beta,
                           const int32_t* cu_seqlens, const float* h0, void* out, float* hT,
                           void* workspace, size_t workspace_bytes, void* stream) {
  return fwd_common(s, q, k, v, g, beta, cu_seqlens, h0, out, hT, nullptr, nullptr, 0, 0, pre,
                    workspace, workspace_bytes, stream);
}

kda_status kda_fwd_checkpoints(const kda_shape* s, const void* q, const void* k, const void* v,
                               const void* g, const void* beta, const int32_t* cu_seqlens,
                               const float* h0, void* out, float* hT, int32_t interval,
                               float* ckpt, const int32_t* ckpt_offsets, int64_t ckpt_rows,
                               void* workspace, size_t workspace_bytes, void* stream) {
  if (interval <= 0 || interval % 64 != 0 || !ckpt || !aligned(ckpt, 16) || ckpt_rows < 0)
    return KDA_ERR_INVALID_ARG;
  if (cu_seqlens && (!ckpt_offsets || !aligned(ckpt_offsets, 4))) return KDA_ERR_INVALID_ARG;
  return fwd_common(s, q, k, v, g, beta, cu_seqlens, h0, out, hT, ckpt,
                    cu_seqlens ? ckpt_offsets : nullptr, ckpt_rows, interval, nullptr, workspace,
                    workspace_bytes, stream);
}

namespace {
// shared by kda_decode and kda_decode_commit; out may be NULL only with counts
kda_status decode_common(const kda_shape* s, const void* q, const void* k, const void* v,
                         const void* g, const void* beta, const int32_t* num_commit,
                         float* state, void* out, const kda_preproc* pre, void* workspace,
                         size_t workspace_bytes, void* stream) {
  kda_status st = check_shape(s, false);
  if (st != KDA_OK) return st;
  if (s->T < 1 || s->T > 8) return KDA_ERR_UNSUPPORTED;
  if (!q || !k || !v || !g || !beta || !state || (!out && !num_commit)) return KDA_ERR_INVALID_ARG;
  const void* ptrs[] = {q, k, v, state, out};
  for (const void* p : ptrs)
    if (p && !aligned(p, 16)) return KDA_ERR_INVALID_ARG;
  if (!aligned(beta, dsize(s->in_dtype)) || !preproc_ok(pre, g, s->in_dtype))
    return KDA_ERR_INVALID_ARG;
  if (num_commit && !aligned(num_commit, 4)) return KDA_ERR_INVALID_ARG;
  st = check_ws(s, workspace, workspace_bytes, false);
  if (st != KDA_OK) return st;

  DecodeArgs a{};
  a.q = q; a.k = k; a.v = v; a.g = g; a.beta = beta;
  a.state = state; a.out = out;
  a.B = s->B; a.Tstep = s->T; a.H = s->H; a.D = s->dk;
  a.scale = s->scale;
  a.in_dtype = s->in_dtype;
  a.out_dtype = s->out_dtype;
  a.num_commit = num_commit;
  a.status = static_cast<unsigned int*>(workspace);
  a.pre = to_preproc(pre);
  a.stream = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(workspace, 0, kWsHeader, a.stream) != cudaSuccess) return KDA_ERR_CUDA;
  return launch_decode(a) == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}
}  // namespace

kda_status kda_decode(const kda_shape* s, const void* q, const void* k, const void* v,
                      const void* g, const void* beta, float* state, void* out,
                      void* workspace, size_t workspace_bytes, void* stream) {
  if (!out) return KDA_ERR_INVALID_ARG;
  return decode_common(s, q, k, v, g, beta, nullptr, state, out, nullptr, workspace,
                       workspace_bytes, stream);
}

kda_status kda_decode_preproc(const kda_shape* s, const kda_preproc* pre, const void* q,
                              const void* k, const void* v, const void* g, const void* beta,
                              float* state, void* out, void* workspace, size_t workspace_bytes,
                              void* stream) {
  if (!out) return KDA_ERR_INVALID_ARG;
  return decode_common(s, q, k, v, g, beta, nullptr, state, out, pre, workspace,
                       workspace_bytes, stream);
}

kda_status kda_decode_commit(const kda_shape* s, const void* q, const void* k, const void* v,
                             const void* g, const void* beta, const int32_t* num_commit,
                             float* state, void* out, void* workspace, size_t workspace_bytes,
                             void* stream) {
  if (!num_commit) return KDA_ERR_INVALID_ARG;
  return decode_common(s, q, k, v, g, beta, num_commit, state, out, nullptr, workspace,
                       workspace_bytes, stream);
}

kda_status kda_read_device_status(void* workspace, void* stream) {
  if (!workspace || !aligned(workspace, 256)) return KDA_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  unsigned int code = 0;
  if (cudaMemcpyAsync(&code, workspace, sizeof(code), cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return KDA_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return KDA_ERR_CUDA;
  if (code != 0) {
    if (cudaMemsetAsync(workspace, 0, sizeof(code), s) != cudaSuccess) return KDA_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return KDA_ERR_CUDA;
  }
  return static_cast<kda_status>(code);
}

const char* kda_status_string(kda_status st) {
  switch (st) {
    case KDA_OK: return "ok";
    case KDA_ERR_INVALID_ARG: return "invalid argument";
    case KDA_ERR_UNSUPPORTED: return "unsupported shape or dtype";
    case KDA_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case KDA_ERR_CUDA: return "CUDA call or kernel launch failed";
    case KDA_ERR_BAD_SEQLENS: return "cu_seqlens is not non-decreasing from 0 to T";
    case KDA_ERR_DEVICE_TIMEOUT: return "a bounded wait inside a kernel ran out";
    case KDA_ERR_DECAY_RANGE: return "decay range (not raised by this version)";
  }
  return "unknown status";
}

// Backward workspace: status header, the packed order list, the packed state-row
// offsets, then one float32 dk x dv state per (16-token sub-chunk, head).
namespace {
size_t bwd_off_bytes(int64_t N) { return (size_t)((N * 8 + 255) / 256) * 256; }
size_t bwd_ws_bytes(const kda_shape* s) {
  const bool packed = s->num_seqs > 0;
  const int64_t N = packed ? s->num_seqs : s->B;
  size_t b = kWsHeader;
  if (packed) b += ws_order_bytes(N) + bwd_off_bytes(N);
  b = (b + 255) / 256 * 256;
  b += kda::bwd_state_rows(packed, N, s->T) * (size_t)s->H * kda::bwd_row_floats(s->dk) *
       sizeof(float);
  return b;
}
}  // namespace

size_t kda_bwd_workspace_size(const kda_shape* s) {
  if (!s || s->B < 0 || s->T < 0 || s->H < 0 || s->num_seqs < 0 || s->dk < 0 || s->dv < 0)
    return 0;
  return bwd_ws_bytes(s);
}

kda_status kda_bwd(const kda_shape* s, const void* q, const void* k, const void* v,
                   const void* g, const void* beta, const int32_t* cu_seqlens, const float* h0,
                   const float* dout, const float* dhT, float* dq, float* dk, float* dv,
                   float* dg, float* dbeta, float* dh0, void* workspace, size_t workspace_bytes,
                   void* stream) {
  const bool packed = cu_seqlens != nullptr;
  kda_status st = check_shape(s, packed);
  if (st != KDA_OK) return st;
  const bool any_tokens = (int64_t)s->B * s->T > 0;
  if (any_tokens && (!q || !k || !v || !g || !beta || !dout || !dq || !dk || !dv || !dg ||
                     !dbeta))
    return KDA_ERR_INVALID_ARG;
  const void* ptrs[] = {q, k, v, g, dout, h0, dhT, dq, dk, dv, dg, dh0};
  for (const void* p : ptrs)
    if (p && !aligned(p, 16)) return KDA_ERR_INVALID_ARG;
  if (!aligned(beta, dsize(s->in_dtype)) || !aligned(dbeta, 4) ||
      (packed && !aligned(cu_seqlens, 4)))
    return KDA_ERR_INVALID_ARG;
  if (!workspace || !aligned(workspace, 256)) return KDA_ERR_WORKSPACE;
  if (workspace_bytes < bwd_ws_bytes(s)) return KDA_ERR_WORKSPACE;

  kda::BwdArgs a{};
  a.q = q; a.k = k; a.v = v; a.g = g; a.beta = beta;
  a.dout = dout; a.dhT = dhT; a.h0 = h0;
  a.cu = cu_seqlens;
  a.T = s->T;
  a.N = packed ? s->num_seqs : s->B;
  a.H = s->H;
  a.D = s->dk;
  a.scale = s->scale;
  a.bf16 = s->in_dtype == KDA_BF16;
  a.dq = dq; a.dk = dk; a.dv = dv; a.dg = dg; a.dbeta = dbeta; a.dh0 = dh0;
  a.status = static_cast<unsigned int*>(workspace);
  a.stream = static_cast<cudaStream_t>(stream);
  char* w = static_cast<char*>(workspace);
  size_t at = kWsHeader;
  if (cudaMemsetAsync(workspace, 0, kWsHeader, a.stream) != cudaSuccess) return KDA_ERR_CUDA;
  if (packed) {
    int32_t* order = reinterpret_cast<int32_t*>(w + at);
    at += ws_order_bytes(a.N);
    int64_t* off = reinterpret_cast<int64_t*>(w + at);
    at += bwd_off_bytes(a.N);
    kda::FwdArgs f{};
    f.cu = cu_seqlens;
    f.T = s->T;
    f.N = a.N;
    f.status = a.status;
    f.stream = a.stream;
    if (kda::launch_schedule(f, order) != cudaSuccess) return KDA_ERR_CUDA;
    if (kda::launch_bwd_offsets(a, off) != cudaSuccess) return KDA_ERR_CUDA;
    a.order = order;
    a.sub_off = off;
  }
  at = (at + 255) / 256 * 256;
  a.states = reinterpret_cast<float*>(w + at);
  return kda::launch_backward(a) == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

const char* kda_version(void) { return "kda-gb300 0.1"; }

}  // extern "C"
