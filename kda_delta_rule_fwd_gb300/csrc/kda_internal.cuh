// Internal declarations shared by the CUDA translation units of the KDA library.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kda.h"

namespace kda {

// Device status word: first 4 bytes of the caller's workspace.  Kernels latch
// the first error with atomicCAS(0 -> code) and never trap.
struct DevStatus {
  unsigned int code;
};

__device__ __forceinline__ void latch_status(unsigned int* status, unsigned int code) {
  if (status) atomicCAS(status, 0u, code);
}

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

// Two float32 lanes per instruction (packed f32x2, IEEE round-to-nearest in each
// lane: the same results as two scalar operations, in half the issue slots).
union F2 {
  float2 f;
  unsigned long long u;
};
__device__ __forceinline__ float2 mul2(float2 a, float2 b) {
  F2 x{a}, y{b}, d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d.u) : "l"(x.u), "l"(y.u));
  return d.f;
}
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {  // a * b + c
  F2 x{a}, y{b}, z{c}, d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d.u) : "l"(x.u), "l"(y.u), "l"(z.u));
  return d.f;
}

template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

// Where a sequence's tokens live: global token offset and length.  A fixed
// batch (no cu_seqlens) puts sequence n at n*T.  Packed batches read the
// validated cu_seqlens.
struct SeqView {
  const int32_t* cu;   // device [N+1] or nullptr
  int64_t T;           // fixed: tokens per sequence; packed: total tokens
  __device__ __forceinline__ void get(int n, int64_t& start, int64_t& len) const {
    if (cu) {
      int64_t a = cu[n], b = cu[n + 1];
      a = a < 0 ? 0 : (a > T ? T : a);
      b = b < a ? a : (b > T ? T : b);
      start = a;
      len = b - a;
    } else {
      start = (int64_t)n * T;
      len = T;
    }
  }
};

// Workspace layout (bytes):
//   [0, 256)            status word (bytes 0-3) and the prefill launches' work
//                       counters (bytes 64-83), zeroed by every call
//   [256, 256 + 4*Npad) sequence order for the packed-batch scheduler
constexpr size_t kWsHeader = 256;
inline size_t ws_order_bytes(int64_t n) { return (size_t)((n + 63) / 64) * 64 * 4; }

// Long-chain split for fixed-length bf16 batches with few (sequence, head)
// chains: each chain is cut into nseg segments, so that the device has enough
// independent work (the segments are joined exactly through their affine state
// transitions).  Segment 0 has seg0_len tokens and segments 1 .. nseg-1 seg_len
// each (the last may be shorter).  A pure function of the shape, so that the
// workspace size can be computed without a device.
//
// The plan minimises a model of the critical path in chunk-steps (one 64-token
// chunk of one chain on one SM) on the device's `sms` SMs, one CTA per SM taking
// the next item as it frees up.  Per chain, the first launch runs segment 0 from
// the true start state (with its outputs) and 2 (nseg - 2) transition items, the
// segment-0 items first; the second launch runs the nseg - 1 output items; the
// scan costs about half a chunk-step per segment.  Segment 0 runs once while the
// others run in both launches, so it may be longer than the others: its length is
// seg_len times 1, 1.5, 2, 2.5 or 3, whichever models fastest.  A split is taken
// only when the model saves at least 10% over running every chain whole.
struct SegPlan {
  int nseg = 1;
  int64_t seg_len = 0;   // tokens of segments 1 .. nseg-1
  int64_t seg0_len = 0;  // tokens of segment 0 (at least seg_len)
};
constexpr int64_t kGb300Sms = 152;     // the plan's SM count when no device can be queried
constexpr int64_t kSegMinChunks = 64;  // at least this many 64-token chunks per segment
constexpr int64_t kSegMaxSegs = 64;
inline int64_t plan_waves(int64_t ctas, int64_t sms) { return (ctas + sms - 1) / sms; }
// Finishing time of n1 items of a chunk-steps, taken first, then n2 items of b <= a,
// on m CTAs that each take the next item when free (n1 < m): the n1 CTAs of the
// long items join the others at time a.
__host__ __device__ inline int64_t plan_makespan(int64_t n1, int64_t a, int64_t n2, int64_t b,
                                                 int64_t m) {
  int64_t last = n1 > 0 ? a : 0, tx = 0, ty = a, rem = n2;
  const int64_t gx = m - n1, gy = n1;
  while (rem > 0) {
    const bool x = gx > 0 && (tx <= ty || gy == 0);
    const int64_t g = x ? gx : gy;
    int64_t& t = x ? tx : ty;
    rem -= rem < g ? rem : g;
    if (t + b > last) last = t + b;
    t += b;
  }
  return last;
}
inline double plan_cost(int64_t chains, int64_t chunks, int64_t seg0_chunks, int64_t seg_chunks,
                        int64_t nseg, int64_t sms) {
  if (nseg < 2) return (double)plan_waves(chains, sms) * (double)chunks;
  return (double)plan_makespan(chains, seg0_chunks, chains * 2 * (nseg - 2), seg_chunks, sms) +
         (double)(plan_waves(chains * (nseg - 1), sms) * seg_chunks) + 0.5 * (double)nseg;
}
inline SegPlan seg_plan(bool packed, bool bf16_d128, int64_t chains, int64_t T, int64_t sms) {
  SegPlan pl;
  const int64_t chunks = (T + 63) / 64;
  if (sms < 1) sms = kGb300Sms;
  if (packed || !bf16_d128 || chains <= 0 || chains >= sms || chunks < 2 * kSegMinChunks)
    return pl;
  double best = 0.9 * plan_cost(chains, chunks, chunks, chunks, 1, sms);
  const int64_t max_ns = chunks / kSegMinChunks < kSegMaxSegs ? chunks / kSegMinChunks
                                                              : kSegMaxSegs;
  for (int64_t ns = 2; ns <= max_ns; ++ns) {
    for (int r2 = 2; r2 <= 6; ++r2) {  // segment 0 r2 / 2 times as long as the others
      int64_t seg, seg0, nseg;
      if (r2 == 2) {  // equal segments, the last one shorter
        seg = (chunks + ns - 1) / ns;
        nseg = (chunks + seg - 1) / seg;
        seg0 = seg;
      } else {  // segments 1 .. ns-1 of seg chunks, segment 0 the rest
        seg = (2 * chunks + r2 + 2 * (ns - 1) - 1) / (r2 + 2 * (ns - 1));
        nseg = ns;
        seg0 = chunks - (ns - 1) * seg;
        if (seg < kSegMinChunks || seg0 < seg) continue;
      }
      const double c = plan_cost(chains, chunks, seg0, seg, nseg, sms);
      if (c < best) {
        best = c;
        pl.nseg = (int)nseg;
        pl.seg_len = seg * 64;
        pl.seg0_len = seg0 * 64;
      }
    }
  }
  return pl;
}

// bytes of segment states: b and M for segments 0..nseg-2, start states for 0..nseg-1
inline size_t seg_bytes(const SegPlan& pl, int64_t chains, int D) {
  if (pl.nseg < 2) return 0;
  return (size_t)chains * (size_t)(3 * pl.nseg - 2) * (size_t)D * D * sizeof(float);
}

// Long-chain split for packed bf16 batches, the fixed-length split applied per
// sequence.  The lengths are only on the device, so a planner kernel (one CTA)
// reads the validated cu_seqlens, picks a segment length S (64-token chunks) and
// a ratio r for segment 0 from a cost model, and writes the plan into the
// workspace: every sequence of at least 2 S chunks is cut into up to 64
// segments, segments 1 .. nseg-1 of about S chunks and segment 0 about r times
// as long (r = 1: equal segments, the last one shorter); the others run whole.
// The transition pass runs each split sequence's segment 0 from its start state
// with its outputs (its end state is S_1) and the b and M items of segments
// 1 .. nseg-2; the output pass runs segments 1 .. nseg-1 and the whole
// sequences.  The passes (transitions, scan, outputs) launch over grids sized by
// an upper bound; CTAs past the plan's counts leave at once.
//
// Cost model, in chunk-steps on `sms` SMs with one CTA each: the transition pass
// as the list schedule of its segment-0 items (taken first) and then its b and M
// items (plan_makespan, with the longest of each); the output pass, whose items
// total W chunks, the longest L, about max(L, W / sms + L / 2); the scan about
// half a chunk-step per segment.  The split is taken when it saves at least 10%
// against running every chain whole.
struct PackedPlan {
  int32_t n_trans;   // transition entries (sequence, segment < nseg - 1), segment 0 first
  int32_t n_split;   // split sequences
  int32_t n_out;     // output items (sequence, segment >= 1, or whole), longest first
  int32_t seg_chunks;  // S, or 0 when nothing is split
};
struct PlanItem {
  int32_t n, seg;
};
// Bound on the segments of all split sequences together: each split sequence
// is at least 2 S >= 128 chunks long and its segments at least S >= 64 chunks.
inline int64_t packed_ns_max(int64_t T) { return T / 4096 + T / 524288 + 2; }
// packed split possible at all: some sequence may reach 2 * 64 chunks
inline bool packed_split_possible(bool bf16_d128, int64_t T) {
  return bf16_d128 && T >= 2 * 64 * 64;
}
// workspace bytes after the order list: the plan (header, per-sequence
// arrays, item tables; 256-byte aligned), then the segment states
inline size_t packed_plan_bytes(int64_t N, int64_t ns_max) {
  const size_t b = sizeof(PackedPlan) + (size_t)N * 4 * sizeof(int32_t) +
                   (size_t)ns_max * sizeof(PlanItem)            // transitions
                   + (size_t)ns_max * sizeof(int32_t)           // split sequences
                   + (size_t)(N + ns_max) * sizeof(PlanItem);   // outputs
  return (b + 255) / 256 * 256;
}
inline size_t packed_state_bytes(int64_t ns_max, int64_t H, int D) {
  return (size_t)(3 * ns_max) * (size_t)H * (size_t)D * D * sizeof(float);
}
// Views of the plan area (laid out in the order packed_plan_bytes counts it).
struct PlanView {
  PackedPlan* hdr;
  int32_t* nseg;      // [N] segments per sequence (1: whole)
  int32_t* seglen;    // [N] tokens per segment 1 .. nseg-1 (split sequences)
  int32_t* seg0len;   // [N] tokens of segment 0 (split sequences)
  int32_t* slot;      // [N] first state slot of a split sequence (x H heads)
  PlanItem* trans;    // [ns_max]
  int32_t* split;     // [ns_max]
  PlanItem* out;      // [N + ns_max]
  __host__ __device__ static PlanView at(void* base, int64_t N, int64_t ns_max) {
    PlanView v;
    char* p = static_cast<char*>(base);
    v.hdr = reinterpret_cast<PackedPlan*>(p);
    p += sizeof(PackedPlan);
    v.nseg = reinterpret_cast<int32_t*>(p);
    v.seglen = v.nseg + N;
    v.seg0len = v.seglen + N;
    v.slot = v.seg0len + N;
    p += (size_t)N * 4 * sizeof(int32_t);
    v.trans = reinterpret_cast<PlanItem*>(p);
    p += (size_t)ns_max * sizeof(PlanItem);
    v.split = reinterpret_cast<int32_t*>(p);
    p += (size_t)ns_max * sizeof(int32_t);
    v.out = reinterpret_cast<PlanItem*>(p);
    return v;
  }
};

// ---------------------------------------------------------------------------
// launchers (each returns cudaSuccess or the launch error)
// ---------------------------------------------------------------------------
// Fused input preprocessing (kda_preproc): each enabled step in float32, rounded
// to the input dtype, as a separate pass that stores input-dtype tensors would.
struct Preproc {
  int l2;                   // q, k: x / max(||x||, 1e-12) per (token, head)
  int gate;                 // log(alpha) = -gate_scale[h] * softplus(g)
  int beta;                 // beta = sigmoid(beta)
  int per_head;             // g holds one gate per (token, head), shared by the key channels
  const float* gate_scale;  // [H], or null for 1
};
template <typename T> __device__ __forceinline__ float round_to(float x);
template <> __device__ __forceinline__ float round_to<float>(float x) { return x; }
template <> __device__ __forceinline__ float round_to<__nv_bfloat16>(float x) {
  return __bfloat162float(__float2bfloat16_rn(x));
}
// -softplus(x) from softplus(x) = max(x, 0) + log1p(y), y = e^-|x| in (0, 1], on the
// special-function unit: y = 2^(-|x| log2 e); log1p(y) as ln 2 * log2(1 + y) for
// y >= 1/32 and as its Taylor series y - y^2/2 + y^3/3 - y^4/4 below (truncation
// under y^5/5, relative 2^-20; there 1 + y would lose y's low bits).  Absolute
// error below 4e-7 before the final rounding; log1p(y) rounds away above |x| ~ 17.
__device__ __forceinline__ float neg_softplus(float x) {
  float y, l2;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(-fabsf(x) * 1.4426950408889634f));
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(l2) : "f"(1.f + y));
  const float series = y * fmaf(y, fmaf(y, fmaf(y, -0.25f, 1.f / 3.f), -0.5f), 1.f);
  const float l = y < 0.03125f ? series : l2 * 0.6931471805599453f;
  return -(fmaxf(x, 0.f) + l);
}
// 1 / (1 + e^-x) with the fast exponential and division (a few ulp; 0 below x ~ -87)
__device__ __forceinline__ float sigmoid_f(float x) { return __fdividef(1.f, 1.f + __expf(-x)); }
// 1 / max(||x||, 1e-12) from the sum of squares, as rsqrt(max(sumsq, 1e-24))
__device__ __forceinline__ float inv_l2(float sumsq) { return rsqrtf(fmaxf(sumsq, 1e-24f)); }

struct FwdArgs {
  const void *q, *k, *v, *g, *beta;
  const int32_t* cu;
  const float* h0;
  void* out;
  float* hT;
  int64_t T;        // tokens per sequence (fixed) or total tokens (packed)
  int32_t N, H, D;  // sequences, heads, head dim (dk == dv)
  float scale;
  kda_dtype in_dtype, out_dtype;
  unsigned int* status;
  const int32_t* order;  // scheduler output: sequences longest first (packed), or nullptr
  float* seg_ws;         // segment-state area of the workspace (long-chain split), or nullptr
  SegPlan plan;          // the split seg_ws was sized for (nseg 1: none)
  void* pplan;           // packed batches: the plan area (long-chain split), or nullptr
  int64_t ns_max;        // packed batches: bound on the split sequences' segments
  int64_t sms;           // SMs of the device (the planner's cost model)
  // prefix-cache checkpoints (state after every ckpt_interval tokens), or ckpt == nullptr
  float* ckpt;              // [ckpt_rows, H, D, D]
  const int32_t* ckpt_off;  // [N+1] row offsets (packed batches), or nullptr (fixed length)
  int64_t ckpt_rows;
  int64_t ckpt_interval;    // tokens, a multiple of 64
  Preproc pre;              // all zero: the inputs are used as given
  cudaStream_t stream;
};

// First checkpoint row of sequence n (rows base .. base + seq_len / interval - 1
// hold the states after interval, 2 interval, ... tokens), or -1 when checkpoints
// are off or the caller's offsets disagree with the sequence length or the
// buffer (latched as KDA_ERR_INVALID_ARG by the leader thread; nothing written).
__device__ __forceinline__ int64_t ckpt_base(const float* ckpt, const int32_t* off, int64_t rows,
                                             int64_t interval, int n, int64_t seq_len,
                                             unsigned int* status, bool leader) {
  if (!ckpt) return -1;
  const int64_t cnt = seq_len / interval;
  const int64_t base = off ? (int64_t)off[n] : (int64_t)n * cnt;
  const bool bad = (off && (int64_t)off[n + 1] - base != cnt) || base < 0 || base + cnt > rows;
  if (bad) {
    if (leader) latch_status(status, KDA_ERR_INVALID_ARG);
    return -1;
  }
  return base;
}

cudaError_t launch_schedule(const FwdArgs& a, int32_t* order_out);
cudaError_t launch_plan_packed(const FwdArgs& a);
cudaError_t launch_prefill_f32(const FwdArgs& a);
// The segment scan of the long-chain split (kda_segment_scan.cu): per chain,
// S_{p+1} = M_p S_p + b_p, d = 128.  Fixed length: `chains` chains of nseg
// segments, b of all chains, then M, then the start states; segment 0 ran from
// the true start state, so S_1 = b_0 and the recursion starts at p = 1.
cudaError_t launch_segment_scan(const float* seg_m, const float* seg_b, float* seg_s,
                                int64_t chains, int nseg, cudaStream_t stream);
// Packed: the split sequences of the device-written plan, H heads each (segment
// 0 ran from the start state there too: S_1 = b_0).
cudaError_t launch_segment_scan_packed(PlanView pv, float* states, int H, int64_t ns_max,
                                       int64_t sms, cudaStream_t stream);
cudaError_t launch_prefill_bf16(const FwdArgs& a);

struct DecodeArgs {
  const void *q, *k, *v, *g, *beta;
  float* state;
  void* out;
  int32_t B, Tstep, H, D;
  float scale;
  kda_dtype in_dtype, out_dtype;
  const int32_t* num_commit;  // per-sequence commit counts, or nullptr (commit all)
  unsigned int* status;
  Preproc pre;                // all zero: the inputs are used as given
  cudaStream_t stream;
};

cudaError_t launch_decode(const DecodeArgs& a);

// Backward (kda_bwd): gradients of sum(o * dout) + sum(hT * dhT).
struct BwdArgs {
  const void *q, *k, *v, *g, *beta;
  const float* dout;
  const float* dhT;
  const float* h0;
  const int32_t* cu;
  int64_t T;
  int N, H, D;
  float scale;
  bool bf16;
  const int32_t* order;
  const int64_t* sub_off;
  float *dq, *dk, *dv, *dg, *dbeta, *dh0;
  float* states;
  unsigned int* status;
  cudaStream_t stream;
};
// state rows the backward keeps in the workspace (one per 16-token sub-chunk of
// every sequence, for each head)
size_t bwd_state_rows(bool packed, int64_t N, int64_t T);
// floats per row (state, then X and U [16][d], T and P [16][16] of the sub-chunk)
inline size_t bwd_row_floats(int d) { return (size_t)d * d + 2 * 16 * d + 2 * 16 * 16; }
cudaError_t launch_bwd_offsets(const BwdArgs& a, int64_t* off);
cudaError_t launch_backward(const BwdArgs& a);

}  // namespace kda
