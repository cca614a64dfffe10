// Packed-batch scheduler: validates cu_seqlens on the device and orders the
// sequences longest first, so that prefill CTAs (one per (sequence, head),
// dispatched in launch order) start the longest recurrent chains first.
//
// Packed sequences with a state reset at every boundary: "Kimi K3 NPU
// Training", section 定长与 TND (cu_seqlens; the recurrent state resets at
// each packed sequence boundary).
//
// A malformed cu_seqlens (cu[0] != 0, decreasing, or cu[N] != T) latches
// KDA_ERR_BAD_SEQLENS in the status word; the prefill kernels then skip all
// work, so no out-of-range token is ever read.
//
// For bf16 batches long enough, a planner then cuts the longest sequences into
// segments joined through their affine state maps (the long-chain split of
// fixed-length batches, applied per sequence): kda_plan_packed_split.
#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int kThreads = 256;

__global__ void kda_validate_seqlens(const int32_t* __restrict__ cu, int N, int64_t T,
                                     unsigned int* __restrict__ status) {
  for (int n = blockIdx.x * blockDim.x + threadIdx.x; n <= N; n += gridDim.x * blockDim.x) {
    const int64_t c = cu[n];
    bool bad = (n == 0 && c != 0) || (n == N && c != T) || c < 0 || c > T;
    if (n > 0 && cu[n - 1] > c) bad = true;
    if (bad) latch_status(status, KDA_ERR_BAD_SEQLENS);
  }
}

// rank(n) = number of sequences strictly longer, plus equal-length ones with a
// smaller index: a stable descending order.  O(N^2) compares spread over the
// grid; N is the number of sequences in one packed batch.
__global__ void kda_order_by_length(const int32_t* __restrict__ cu, int N,
                                    int32_t* __restrict__ order) {
  const int n = blockIdx.x * blockDim.x + threadIdx.x;
  if (n >= N) return;
  const int32_t ln = cu[n + 1] - cu[n];
  int rank = 0;
  for (int m = 0; m < N; ++m) {
    const int32_t lm = cu[m + 1] - cu[m];
    rank += (lm > ln) || (lm == ln && m < n);
  }
  order[rank] = n;
}

// Block-wide reductions of the planner (kPlanThreads threads).
constexpr int kPlanThreads = 256;
constexpr int kPlanWarps = kPlanThreads / 32;
__device__ __forceinline__ int64_t block_sum(int64_t x, int64_t* sh) {
  sh[threadIdx.x] = x;
  __syncthreads();
  for (int o = kPlanThreads / 2; o > 0; o >>= 1) {
    if ((int)threadIdx.x < o) sh[threadIdx.x] += sh[threadIdx.x + o];
    __syncthreads();
  }
  const int64_t r = sh[0];
  __syncthreads();
  return r;
}
__device__ __forceinline__ int64_t block_max(int64_t x, int64_t* sh) {
  sh[threadIdx.x] = x;
  __syncthreads();
  for (int o = kPlanThreads / 2; o > 0; o >>= 1) {
    if ((int)threadIdx.x < o && sh[threadIdx.x + o] > sh[threadIdx.x])
      sh[threadIdx.x] = sh[threadIdx.x + o];
    __syncthreads();
  }
  const int64_t r = sh[0];
  __syncthreads();
  return r;
}
// makespan estimate of one pass (chunk-steps): total work W, longest item L
__device__ __forceinline__ double pass_cost(int64_t W, int64_t L, int64_t sms) {
  const double lpt = (double)W / (double)sms + 0.5 * (double)L;
  return lpt > (double)L ? lpt : (double)L;
}
__device__ __forceinline__ int64_t seq_chunks(const int32_t* cu, int n) {
  return ((int64_t)cu[n + 1] - cu[n] + 63) / 64;
}
__device__ __forceinline__ int64_t imax(int64_t a, int64_t b) { return a > b ? a : b; }

// The segments of a sequence of c chunks for the candidate (S, r2): their count
// ns, the length s of segments 1 .. ns-1 and s0 of segment 0, in chunks.  With
// r2 > 2, segment 0 is about r2 / 2 times as long as the others and the last
// one is whole; with r2 = 2 (or where that leaves segments shorter than the
// minimum) the c / S segments are equal and the last one is shorter.  ns = 1:
// the sequence runs whole (fewer than 2 S chunks).
struct SegChoice {
  int64_t ns, s, s0;
};
__device__ __forceinline__ SegChoice seg_choice(int64_t c, int64_t S, int r2) {
  if (c < 2 * S) return SegChoice{1, 0, 0};
  if (r2 > 2) {
    int64_t ns = (2 * c - r2 * S) / (2 * S) + 1;
    ns = ns < 2 ? 2 : (ns < kSegMaxSegs ? ns : kSegMaxSegs);
    const int64_t den = r2 + 2 * (ns - 1), s = (2 * c + den - 1) / den, s0 = c - (ns - 1) * s;
    if (s >= kSegMinChunks && s0 >= s) return SegChoice{ns, s, s0};
  }
  int64_t ns = c / S;
  ns = ns < kSegMaxSegs ? ns : kSegMaxSegs;
  const int64_t s = (c + ns - 1) / ns;
  return SegChoice{ns, s, s};
}

// Per-candidate totals of the planner: sums (split sequences, b and M items per
// head, output work, segments) and maxima (segment 0, segments >= 1, longest
// output item, segments of one sequence).
struct PlanAcc {
  int64_t nsp, n2, w1, w2, tot, a, b, l2, nsm;
};
__device__ __forceinline__ void acc_combine(PlanAcc& x, const PlanAcc& y) {
  x.nsp += y.nsp;
  x.n2 += y.n2;
  x.w1 += y.w1;
  x.w2 += y.w2;
  x.tot += y.tot;
  x.a = imax(x.a, y.a);
  x.b = imax(x.b, y.b);
  x.l2 = imax(x.l2, y.l2);
  x.nsm = imax(x.nsm, y.nsm);
}
// the block's totals, the same in every thread (warp shuffles, then the warps)
__device__ PlanAcc block_reduce(PlanAcc x, PlanAcc* sh) {
  for (int o = 16; o > 0; o >>= 1) {
    PlanAcc y;
    y.nsp = __shfl_xor_sync(0xffffffffu, x.nsp, o);
    y.n2 = __shfl_xor_sync(0xffffffffu, x.n2, o);
    y.w1 = __shfl_xor_sync(0xffffffffu, x.w1, o);
    y.w2 = __shfl_xor_sync(0xffffffffu, x.w2, o);
    y.tot = __shfl_xor_sync(0xffffffffu, x.tot, o);
    y.a = __shfl_xor_sync(0xffffffffu, x.a, o);
    y.b = __shfl_xor_sync(0xffffffffu, x.b, o);
    y.l2 = __shfl_xor_sync(0xffffffffu, x.l2, o);
    y.nsm = __shfl_xor_sync(0xffffffffu, x.nsm, o);
    acc_combine(x, y);
  }
  if ((threadIdx.x & 31) == 0) sh[threadIdx.x / 32] = x;
  __syncthreads();
  PlanAcc r = sh[0];
  for (int w = 1; w < kPlanWarps; ++w) acc_combine(r, sh[w]);
  __syncthreads();
  return r;
}

// one sequence of c chunks into a candidate's totals
__device__ __forceinline__ void acc_add(PlanAcc& x, int64_t c, int64_t S, int r2) {
  const SegChoice g = seg_choice(c, S, r2);
  if (g.ns >= 2) {
    x.nsp += 1;
    x.n2 += 2 * (g.ns - 2);
    x.w1 += g.s0 + 2 * (g.ns - 2) * g.s;
    x.w2 += (g.ns - 1) * g.s;
    x.tot += g.ns;
    x.a = imax(x.a, g.s0);
    x.b = imax(x.b, g.s);
    x.l2 = imax(x.l2, g.s);
    x.nsm = imax(x.nsm, g.ns);
  } else {
    x.w2 += c;
    x.l2 = imax(x.l2, c);
  }
}
// modelled chunk-steps of a candidate from its totals (infinite past ns_max)
__device__ __forceinline__ double cand_cost(const PlanAcc& t, int H, int64_t sms, int64_t ns_max) {
  if (t.tot > ns_max) return 1e300;
  const int64_t n1 = t.nsp * H;
  const double c1 = n1 < sms ? (double)plan_makespan(n1, t.a, t.n2 * H, t.b, sms)
                             : pass_cost(t.w1 * H, t.a, sms);
  return c1 + 0.5 * (double)t.nsm + pass_cost(t.w2 * H, t.l2, sms);
}
// candidate k: S = 64, 80, 96, 128, 160, 192, ... (index k / 5), r2 = 2 + k % 5
__device__ __forceinline__ int64_t cand_S(int k) {
  const int i = k / 5;
  return (int64_t)(64 + 16 * (i % 3)) << (i / 3);
}
constexpr int kPlanSmallN = 512;  // up to this many sequences a thread costs a whole candidate

// The long-chain split plan of a packed batch (see PackedPlan).  One CTA.
// `order` holds the sequences longest first (kda_order_by_length).
__global__ void __launch_bounds__(kPlanThreads)
kda_plan_packed_split(const int32_t* __restrict__ cu, const int32_t* __restrict__ order, int N,
                      int H, int64_t sms, int64_t ns_max, void* plan_base,
                      unsigned int* __restrict__ status) {
  __shared__ int64_t sh[kPlanThreads];
  __shared__ PlanAcc sha[kPlanWarps];
  const int tid = threadIdx.x;
  PlanView pv = PlanView::at(plan_base, N, ns_max);
  if (status && *(volatile const unsigned int*)status == (unsigned)KDA_ERR_BAD_SEQLENS) {
    if (tid == 0) *pv.hdr = PackedPlan{0, 0, 0, 0};  // every pass leaves at once
    return;
  }
  int64_t mc = 0, w = 0;
  for (int n = tid; n < N; n += kPlanThreads) {
    const int64_t c = seq_chunks(cu, n);
    mc = c > mc ? c : mc;
    w += c;
  }
  const int64_t maxc = block_max(mc, sh), W0 = block_sum(w, sh) * H;
  const double cost0 = pass_cost(W0, maxc, sms);
  // candidates: S = 64, 80, 96, 128, 160, 192, ... while 2 S <= maxc, each with
  // segment 0 r2 / 2 = 1, 1.5, 2, 2.5 or 3 times as long; the cheapest (the first
  // of equals) is taken if it saves 10% against cost0
  int ncand = 0;
  while (2 * cand_S(ncand) <= maxc) ncand += 5;
  double best = 1e300;
  int bestk = -1;
  if (N <= kPlanSmallN) {
    // few sequences: each thread costs whole candidates, then one arg-min
    for (int k = tid; k < ncand; k += kPlanThreads) {
      PlanAcc x{0, 0, 0, 0, 0, 0, 0, 0, 0};
      const int64_t S = cand_S(k);
      for (int n = 0; n < N; ++n) acc_add(x, seq_chunks(cu, n), S, 2 + k % 5);
      const double c = cand_cost(x, H, sms, ns_max);
      if (c < best) {
        best = c;
        bestk = k;
      }
    }
    for (int o = 16; o > 0; o >>= 1) {
      const double ob = __shfl_xor_sync(0xffffffffu, best, o);
      const int ok = __shfl_xor_sync(0xffffffffu, bestk, o);
      if (ob < best || (ob == best && ok >= 0 && (bestk < 0 || ok < bestk))) {
        best = ob;
        bestk = ok;
      }
    }
    __shared__ double shb[kPlanWarps];
    __shared__ int shk[kPlanWarps];
    if ((tid & 31) == 0) {
      shb[tid / 32] = best;
      shk[tid / 32] = bestk;
    }
    __syncthreads();
    best = shb[0];
    bestk = shk[0];
    for (int w2 = 1; w2 < kPlanWarps; ++w2)
      if (shb[w2] < best || (shb[w2] == best && shk[w2] >= 0 && (bestk < 0 || shk[w2] < bestk))) {
        best = shb[w2];
        bestk = shk[w2];
      }
  } else {
    // many sequences: candidate by candidate, the totals by block reductions
    for (int k = 0; k < ncand; ++k) {
      PlanAcc x{0, 0, 0, 0, 0, 0, 0, 0, 0};
      for (int n = tid; n < N; n += kPlanThreads) acc_add(x, seq_chunks(cu, n), cand_S(k), 2 + k % 5);
      const double c = cand_cost(block_reduce(x, sha), H, sms, ns_max);
      if (c < best) {  // (uniform across the CTA: reduced values)
        best = c;
        bestk = k;
      }
    }
  }
  const bool split = bestk >= 0 && best < 0.9 * cost0;
  const int64_t bestS = split ? cand_S(bestk) : 0;
  const int bestR = split ? 2 + bestk % 5 : 2;
  // per-sequence segments; thread 0 then builds the tables (few split sequences)
  for (int n = tid; n < N; n += kPlanThreads) {
    const SegChoice g = bestS > 0 ? seg_choice(seq_chunks(cu, n), bestS, bestR)
                                  : SegChoice{1, 0, 0};
    pv.nseg[n] = (int32_t)g.ns;
    pv.seglen[n] = (int32_t)(g.s * 64);
    pv.seg0len[n] = (int32_t)(g.s0 * 64);
  }
  __syncthreads();
  if (tid != 0) return;
  // split sequences in order of decreasing segment length (insertion into the
  // split list; the sequences arrive longest first)
  int32_t n_split = 0, n_trans = 0, n_out = 0, slot = 0;
  for (int r = 0; r < N; ++r) {
    const int32_t n = order[r];
    if (pv.nseg[n] < 2) continue;
    int32_t j = n_split++;
    while (j > 0 && pv.seglen[pv.split[j - 1]] < pv.seglen[n]) {
      pv.split[j] = pv.split[j - 1];
      --j;
    }
    pv.split[j] = n;
  }
  // transition entries: every split sequence's segment 0 first, longest first
  // (insertion by segment-0 length), then segments 1 .. nseg-2
  for (int i = 0; i < n_split; ++i) {
    const int32_t n = pv.split[i];
    pv.slot[n] = slot;
    slot += 3 * pv.nseg[n] - 2;
    int32_t j = n_trans++;
    while (j > 0 && pv.seg0len[pv.trans[j - 1].n] < pv.seg0len[n]) {
      pv.trans[j] = pv.trans[j - 1];
      --j;
    }
    pv.trans[j] = PlanItem{n, 0};
  }
  for (int i = 0; i < n_split; ++i) {
    const int32_t n = pv.split[i];
    for (int32_t sg = 1; sg + 1 < pv.nseg[n]; ++sg) pv.trans[n_trans++] = PlanItem{n, sg};
  }
  // outputs longest first: merge the split sequences' segments 1 .. nseg-1 with the
  // whole sequences (both lists already in decreasing length)
  int i = 0, r = 0;
  while (true) {
    while (r < N && pv.nseg[order[r]] >= 2) ++r;  // split ones come from the other list
    const bool has_seg = i < n_split, has_seq = r < N;
    if (!has_seg && !has_seq) break;
    const int64_t lseg = has_seg ? pv.seglen[pv.split[i]] : -1;
    const int64_t lseq = has_seq ? (int64_t)cu[order[r] + 1] - cu[order[r]] : -1;
    if (has_seg && lseg >= lseq) {
      const int32_t n = pv.split[i++];
      for (int32_t sg = 1; sg < pv.nseg[n]; ++sg) pv.out[n_out++] = PlanItem{n, sg};
    } else {
      pv.out[n_out++] = PlanItem{order[r++], 0};
    }
  }
  *pv.hdr = PackedPlan{n_trans, n_split, n_out, (int32_t)bestS};
}

}  // namespace

cudaError_t launch_plan_packed(const FwdArgs& a) {
  kda_plan_packed_split<<<1, kPlanThreads, 0, a.stream>>>(a.cu, a.order, a.N, a.H, a.sms,
                                                          a.ns_max, a.pplan, a.status);
  return cudaGetLastError();
}

cudaError_t launch_schedule(const FwdArgs& a, int32_t* order_out) {
  const int N = a.N;
  const int blocks = (N + 1 + kThreads - 1) / kThreads;
  kda_validate_seqlens<<<blocks < 1024 ? blocks : 1024, kThreads, 0, a.stream>>>(a.cu, N, a.T,
                                                                              a.status);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || N == 0) return e;
  kda_order_by_length<<<(N + kThreads - 1) / kThreads, kThreads, 0, a.stream>>>(a.cu, N,
                                                                                 order_out);
  return cudaGetLastError();
}

}  // namespace kda
