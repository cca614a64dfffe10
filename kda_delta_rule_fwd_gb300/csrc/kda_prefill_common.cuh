// Device helpers of the bf16 prefill: the canonical operand layouts of the
// tensor-memory MMA, bf16 hi/lo splitting, shared-memory vector access, named
// barriers, the warp-level tf32 fragments of the blocked inverse, the CTA's
// bounded waits, the work items of a launch and the tensor-map encoder.
#pragma once

#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include <cstdint>
#include <mutex>

#include "kda_internal.cuh"
#include "kda_mma_sync.cuh"
#include "kda_sm100.cuh"

namespace kda {
namespace pf {

using namespace sm100;

// Canonical no-swizzle layouts (8 rows x 16 bytes per core matrix).  For an
// operand with `rows` (M or N) and K = `kdim`, core (rb, kb) sits at
// rb*(kdim/8)*128 + kb*128: LBO (K-adjacent cores) = 128 and SBO (M/N-adjacent
// cores) = (kdim/8)*128.  K-major cores hold 8 rows of 8 K-values; MN-major
// cores hold 8 K-rows of 8 M/N-values.
__device__ __forceinline__ uint32_t off_kmaj(int r, int k, int kdim) {
  return (r >> 3) * (kdim >> 3) * 128 + (k >> 3) * 128 + (r & 7) * 16 + (k & 7) * 2;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// 2^x on the special-function unit (relative error about 2^-22; tiny results
// flush to zero, which only drops terms far below the operands they join)
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// hi/lo split of two values, each part packed as bf16x2 (first value in the low half)
// (the remainder x - hi is exact in float32; one packed fma forms both)
__device__ __forceinline__ void split_pack2(float a, float b, uint32_t& hi, uint32_t& lo) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  const float2 r = fma2(__bfloat1622float2(h), make_float2(-1.f, -1.f), make_float2(a, b));
  const __nv_bfloat162 l = __floats2bfloat162_rn(r.x, r.y);
  hi = *reinterpret_cast<const uint32_t*>(&h);
  lo = *reinterpret_cast<const uint32_t*>(&l);
}
// 8 bf16 from a 16-byte shared-memory vector
__device__ __forceinline__ void ld8(const unsigned char* p, float (&x)[8]) {
  const uint4 u = *reinterpret_cast<const uint4*>(p);
  x[0] = bf16_lo(u.x); x[1] = bf16_hi(u.x); x[2] = bf16_lo(u.y); x[3] = bf16_hi(u.y);
  x[4] = bf16_lo(u.z); x[5] = bf16_hi(u.z); x[6] = bf16_lo(u.w); x[7] = bf16_hi(u.w);
}
__device__ __forceinline__ uint32_t pack2(float a, float b) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&h);
}
__device__ __forceinline__ void st8(unsigned char* p, const float (&x)[8]) {
  uint4 u;
  u.x = pack2(x[0], x[1]); u.y = pack2(x[2], x[3]);
  u.z = pack2(x[4], x[5]); u.w = pack2(x[6], x[7]);
  *reinterpret_cast<uint4*>(p) = u;
}
// store hi and lo parts of 8 values
__device__ __forceinline__ void st8_split(unsigned char* phi, unsigned char* plo,
                                          const float (&x)[8]) {
  uint4 h, l;
  split_pack2(x[0], x[1], h.x, l.x);
  split_pack2(x[2], x[3], h.y, l.y);
  split_pack2(x[4], x[5], h.z, l.z);
  split_pack2(x[6], x[7], h.w, l.w);
  *reinterpret_cast<uint4*>(phi) = h;
  *reinterpret_cast<uint4*>(plo) = l;
}
// CTA-local named barrier `id` for `count` threads (whole warps: the barrier
// counts arrivals, the callers choose which warps arrive; here 1 = warps 0-7,
// 2 = warps 8-15; each kernel documents its own ids)
__device__ __forceinline__ void named_bar_sync(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}
__device__ __forceinline__ void named_bar_arrive(int id, int count) {
  asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// m16n8k8 fragments (see mma_tf32x3) read from float matrices in shared memory:
// A rows r0.., columns k0.. of a row-major matrix (row stride ld), of A stored
// transposed (AT[k][r] = A[r][k], row stride ALDV), and B rows k0.., columns n0..
__device__ __forceinline__ void load_a(const float* M, int ld, int r0, int k0, int g, int t4,
                                       float (&a)[4]) {
  a[0] = M[(r0 + g) * ld + k0 + t4];
  a[1] = M[(r0 + g + 8) * ld + k0 + t4];
  a[2] = M[(r0 + g) * ld + k0 + t4 + 4];
  a[3] = M[(r0 + g + 8) * ld + k0 + t4 + 4];
}
template <int ALDV>
__device__ __forceinline__ void load_a_t(const float* AT, int r0, int k0, int g, int t4,
                                         float (&a)[4]) {
  a[0] = AT[(k0 + t4) * ALDV + r0 + g];
  a[1] = AT[(k0 + t4) * ALDV + r0 + g + 8];
  a[2] = AT[(k0 + t4 + 4) * ALDV + r0 + g];
  a[3] = AT[(k0 + t4 + 4) * ALDV + r0 + g + 8];
}
__device__ __forceinline__ void load_b(const float* M, int ld, int k0, int n0, int g, int t4,
                                       float (&b)[2]) {
  b[0] = M[(k0 + t4) * ld + n0 + g];
  b[1] = M[(k0 + t4 + 4) * ld + n0 + g];
}
// zero the three partial accumulators of mma_tf32x3
__device__ __forceinline__ void zero_acc(float (&acc)[3][4]) {
#pragma unroll
  for (int q = 0; q < 3; ++q)
#pragma unroll
    for (int r = 0; r < 4; ++r) acc[q][r] = 0.f;
}
// C fragment (16 x 8 at columns c0 of a row-major matrix with row stride ld),
// summed over the three partial products and scaled by `sign`
__device__ __forceinline__ void store_c(float* Cm, int ld, int c0, const float (&acc)[3][4], int g,
                                        int t4, float sign) {
  const int c = c0 + 2 * t4;
  Cm[g * ld + c] = sign * (acc[0][0] + acc[1][0] + acc[2][0]);
  Cm[g * ld + c + 1] = sign * (acc[0][1] + acc[1][1] + acc[2][1]);
  Cm[(g + 8) * ld + c] = sign * (acc[0][2] + acc[1][2] + acc[2][2]);
  Cm[(g + 8) * ld + c + 1] = sign * (acc[0][3] + acc[1][3] + acc[2][3]);
}

// -T diag(beta) in the K-major TB operand (rows = token i, K = token j, KDIM
// tokens per row), written
// by the producers of T: one value, or two values of adjacent columns (j even)
template <int KDIM>
__device__ __forceinline__ void store_tb1(unsigned char* tb_hi, unsigned char* tb_lo, int i, int j,
                                          float v) {
  const __nv_bfloat16 h = __float2bfloat16_rn(v);
  const uint32_t o = off_kmaj(i, j, KDIM);
  *reinterpret_cast<__nv_bfloat16*>(tb_hi + o) = h;
  *reinterpret_cast<__nv_bfloat16*>(tb_lo + o) = __float2bfloat16_rn(v - __bfloat162float(h));
}
template <int KDIM>
__device__ __forceinline__ void store_tb2(unsigned char* tb_hi, unsigned char* tb_lo, int i, int j,
                                          float v0, float v1) {
  uint32_t hi, lo;
  split_pack2(v0, v1, hi, lo);
  const uint32_t o = off_kmaj(i, j, KDIM);
  *reinterpret_cast<uint32_t*>(tb_hi + o) = hi;
  *reinterpret_cast<uint32_t*>(tb_lo + o) = lo;
}
// T block fragment of mma_tf32x3 (sign applied) to T32 and, scaled by -beta of
// its columns, to TB
template <int KDIM>
__device__ __forceinline__ void store_t_block(float* T32, int ld, int r0, int c0,
                                              const float (&acc)[3][4], int g, int t4, float sign,
                                              const float* beta, unsigned char* tb_hi,
                                              unsigned char* tb_lo) {
  const int c = c0 + 2 * t4;
  const float v00 = sign * (acc[0][0] + acc[1][0] + acc[2][0]);
  const float v01 = sign * (acc[0][1] + acc[1][1] + acc[2][1]);
  const float v10 = sign * (acc[0][2] + acc[1][2] + acc[2][2]);
  const float v11 = sign * (acc[0][3] + acc[1][3] + acc[2][3]);
  T32[(r0 + g) * ld + c] = v00;
  T32[(r0 + g) * ld + c + 1] = v01;
  T32[(r0 + g + 8) * ld + c] = v10;
  T32[(r0 + g + 8) * ld + c + 1] = v11;
  const float b0 = -beta[c], b1 = -beta[c + 1];
  store_tb2<KDIM>(tb_hi, tb_lo, r0 + g, c, v00 * b0, v01 * b1);
  store_tb2<KDIM>(tb_hi, tb_lo, r0 + g + 8, c, v10 * b0, v11 * b1);
}

// hi and lo parts of 16 values, packed two per 32-bit word
__device__ __forceinline__ void pack_split16(const float (&x)[16], uint32_t (&hi)[8],
                                             uint32_t (&lo)[8]) {
#pragma unroll
  for (int e = 0; e < 8; ++e) split_pack2(x[2 * e], x[2 * e + 1], hi[e], lo[e]);
}

// The CTA's bounded waits.  Every thread waits on the barrier itself; a thread
// whose wait runs out raises the shared flag, and the CTA barrier that follows
// each wait makes all threads see the same flag before they branch on it.
struct Waits {
  uint64_t* tma_bar;
  uint64_t* mma_bar;
  uint32_t mma_phase;
  uint32_t tma_waited;  // TMA phases consumed so far
  uint32_t* flag;       // nonzero once a wait ran out
  unsigned int* status;
  __device__ __forceinline__ void on_timeout() {
    atomicExch(flag, 1u);
    latch_status(status, KDA_ERR_DEVICE_TIMEOUT);
  }
  // wait for the MMAs committed last; returns true if the CTA must stop
  __device__ __forceinline__ bool wait_mma() {
    if (!mbar_wait(mma_bar, mma_phase)) on_timeout();
    mma_phase ^= 1u;
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    return *(volatile uint32_t*)flag != 0;
  }
  __device__ __forceinline__ bool wait_tma() {
    if (!mbar_wait(tma_bar, tma_waited & 1u)) on_timeout();
    ++tma_waited;
    __syncthreads();
    return *(volatile uint32_t*)flag != 0;
  }
};

// Work item modes.  CHAIN: one CTA per (sequence, head).  The two SEG modes
// split each chain of a fixed-length batch into nseg segments, segment 0 of
// seg0_len tokens and the others of seg_len (the associative affine form of the
// recurrence: a segment maps its start state S to M S + b):
//   SEG_TRANSITION: per chain, segment 0 from the chain's start state with its
//                   outputs (its end state, in b_0's slot, is S_1), and for
//                   segments 1 .. nseg-2 two items each: b = end state from
//                   S = 0; M = end state from S = I with v = 0 (no outputs).
//                   The segment-0 items of all chains come first (the longest
//                   items are taken first).
//   SEG_OUTPUT:     per (chain, segment >= 1) one item from the segment's true
//                   start state (computed by the scan kernel); writes o, and hT
//                   from the last segment.
// The two PSEG modes do the same for packed batches, item by item from the
// device-written plan (PackedPlan): PSEG_TRANSITION runs each split sequence's
// segment 0 from its start state with its outputs (one item per head), then the
// b and M items of segments 1 .. nseg-2; PSEG_OUTPUT runs segments 1 .. nseg-1
// and the sequences that are not split, whole (as CHAIN).  A CTA past the plan's
// count leaves at once.
enum ItemMode {
  MODE_CHAIN = 0,
  MODE_SEG_TRANSITION = 1,
  MODE_SEG_OUTPUT = 2,
  MODE_PSEG_TRANSITION = 3,
  MODE_PSEG_OUTPUT = 4
};

struct Bf16Params {
  const __nv_bfloat16* beta;
  SeqView seqs;
  const int32_t* order;
  const float* h0;
  void* out;
  float* hT;
  int H;
  int nchains;           // (sequence, head) chains of the batch
  float scale;
  int out_bf16;
  unsigned int* status;  // status word; words 16 + mode count each launch's taken items
  int mode;
  int nseg;
  int64_t seg_len;       // tokens per segment 1 .. nseg-1 (multiple of the chunk length)
  int64_t seg0_len;      // tokens of segment 0 (multiple of the chunk length)
  float* seg_b;          // [chains][nseg-1][D][D] zero-start end states
  float* seg_m;          // [chains][nseg-1][D][D] transitions
  const float* seg_s;    // [chains][nseg][D][D] segment start states (index 0 unused)
  float* ckpt;           // prefix-cache checkpoints [rows][H][D][D], or nullptr
  const int32_t* ckpt_off;
  int64_t ckpt_rows;
  int64_t ckpt_interval;
  Preproc pre;           // fused input preprocessing (kPre instantiation only)
  const __nv_bfloat16* g;  // the gate: [tokens, H, D], or [tokens, H] with pre.per_head
  PlanView pv;           // packed long-chain split: the plan (PSEG modes)
  float* pstates;        // packed long-chain split: segment states (PSEG modes)
};

// One work item: the tokens [t0, t0 + len) of sequence n, head h, from the start
// state s_in (nullptr: zeros, or the identity with ident) to the end state s_out
// (nullptr: not stored); rel0 is t0's offset within the sequence of seq_len
// tokens; zero_v runs the item with v = 0 and want_o = false stores no outputs.
struct ItemInfo {
  int n, h;
  int64_t t0, len, rel0, seq_len;
  const float* s_in;
  float* s_out;
  bool ident, zero_v, want_o;
};

__device__ __forceinline__ int64_t item_count(const Bf16Params& p) {
  return p.mode == MODE_CHAIN ? (int64_t)p.nchains
         : p.mode == MODE_SEG_TRANSITION ? (int64_t)p.nchains * (2 * p.nseg - 3)
         : p.mode == MODE_SEG_OUTPUT ? (int64_t)p.nchains * (p.nseg - 1)
         : p.mode == MODE_PSEG_TRANSITION
             ? (int64_t)p.H * (2 * (int64_t)p.pv.hdr->n_trans - p.pv.hdr->n_split)
                                          : (int64_t)p.H * p.pv.hdr->n_out;
}

__device__ __forceinline__ ItemInfo decode_item(const Bf16Params& p, int item) {
  constexpr int64_t DD = 128 * 128;  // floats per state (dk = dv = 128)
  ItemInfo r;
  r.rel0 = 0;
  r.s_in = nullptr;
  r.s_out = nullptr;
  r.ident = r.zero_v = false;
  r.want_o = true;
  if (p.mode == MODE_CHAIN) {
    r.n = p.order ? p.order[item / p.H] : item / p.H;
    r.h = item % p.H;
    p.seqs.get(r.n, r.t0, r.len);
    r.seq_len = r.len;
    r.s_in = p.h0 ? p.h0 + ((int64_t)r.n * p.H + r.h) * DD : nullptr;
    r.s_out = p.hT ? p.hT + ((int64_t)r.n * p.H + r.h) * DD : nullptr;
  } else if (p.mode == MODE_PSEG_TRANSITION || p.mode == MODE_PSEG_OUTPUT) {
    // transition items: H per segment-0 entry (the first n_split entries), then two
    // (b, M) per head for each later entry
    const bool trans = p.mode == MODE_PSEG_TRANSITION;
    const int n0 = trans ? p.H * p.pv.hdr->n_split : 0;
    int kind = 0, rest = item, it;
    if (trans && item >= n0) {
      kind = (item - n0) & 1;
      rest = (item - n0) >> 1;
      it = p.pv.hdr->n_split + rest / p.H;
    } else {
      it = rest / p.H;
    }
    r.h = rest % p.H;
    const PlanItem pi = trans ? p.pv.trans[it] : p.pv.out[it];
    r.n = pi.n;
    p.seqs.get(r.n, r.t0, r.len);
    r.seq_len = r.len;
    const int nseg = p.pv.nseg[r.n];
    if (nseg < 2) {  // an output item of a whole sequence
      r.s_in = p.h0 ? p.h0 + ((int64_t)r.n * p.H + r.h) * DD : nullptr;
      r.s_out = p.hT ? p.hT + ((int64_t)r.n * p.H + r.h) * DD : nullptr;
    } else {
      // this chain's states: b (segments 0..nseg-2; b_0 holds S_1), M (same; M_0 is
      // not formed), start states (0..nseg-1; S_0 is not stored)
      float* base = p.pstates + ((int64_t)p.pv.slot[r.n] * p.H + (int64_t)r.h * (3 * nseg - 2)) * DD;
      const int64_t s0 = p.pv.seg0len[r.n], sl = p.pv.seglen[r.n];
      const int64_t a0 = pi.seg == 0 ? 0 : s0 + (int64_t)(pi.seg - 1) * sl;
      const int64_t ln = pi.seg == 0 ? s0 : sl;
      if (trans && pi.seg == 0) {  // from the start state, with outputs; its end is S_1
        r.s_in = p.h0 ? p.h0 + ((int64_t)r.n * p.H + r.h) * DD : nullptr;
        r.s_out = base;
      } else if (trans) {
        r.ident = r.zero_v = kind == 1;
        r.want_o = false;
        r.s_out = base + (int64_t)(kind ? (nseg - 1) + pi.seg : pi.seg) * DD;
      } else {
        r.s_in = base + (int64_t)(2 * (nseg - 1) + pi.seg) * DD;
        if (pi.seg == nseg - 1 && p.hT) r.s_out = p.hT + ((int64_t)r.n * p.H + r.h) * DD;
      }
      r.rel0 = a0;
      r.t0 += a0;
      r.len = r.len - a0 < ln ? r.len - a0 : ln;
      if (r.len < 0) r.len = 0;
    }
  } else {
    int seg, chain;
    if (p.mode == MODE_SEG_TRANSITION) {
      // items 0 .. nchains-1: segment 0 of each chain from h0 with its outputs; then
      // per chain, items 2 (s - 1) + kind: segment s's b (kind 0) and M (kind 1),
      // s = 1 .. nseg-2
      if (item < p.nchains) {
        chain = item;
        seg = 0;
        r.s_in = p.h0 ? p.h0 + (int64_t)chain * DD : nullptr;
        r.s_out = p.seg_b + (int64_t)chain * (p.nseg - 1) * DD;
      } else {
        const int per = 2 * (p.nseg - 2), w = item - p.nchains;
        chain = w / per;
        const int kind = (w % per) & 1;
        seg = 1 + (w % per) / 2;
        r.ident = r.zero_v = kind == 1;
        r.want_o = false;
        r.s_out = (kind ? p.seg_m : p.seg_b) + ((int64_t)chain * (p.nseg - 1) + seg) * DD;
      }
    } else {
      seg = 1 + item % (p.nseg - 1);
      chain = item / (p.nseg - 1);
      // segments 1 .. nseg-1 start from the scan's states; hT (which may alias h0)
      // is written here, a launch after segment 0 has read h0
      r.s_in = p.seg_s + ((int64_t)chain * p.nseg + seg) * DD;
      if (seg == p.nseg - 1 && p.hT) r.s_out = p.hT + (int64_t)chain * DD;
    }
    r.n = chain / p.H;
    r.h = chain % p.H;
    int64_t st, ln;
    p.seqs.get(r.n, st, ln);
    const int64_t a = seg == 0 ? 0 : p.seg0_len + (int64_t)(seg - 1) * p.seg_len;
    const int64_t sl = seg == 0 ? p.seg0_len : p.seg_len;
    r.rel0 = a;
    r.seq_len = ln;
    r.t0 = st + a;
    r.len = ln - a < sl ? ln - a : sl;
    if (r.len < 0) r.len = 0;
  }
  return r;
}

// cuTensorMapEncodeTiled from the driver, looked up once
inline PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

}  // namespace pf
}  // namespace kda
