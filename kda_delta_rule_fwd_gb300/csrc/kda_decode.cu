// KDA decode: T_step (1..8) tokens applied in order to per-head float32 states
// resident in device memory, updated in place.
//
// Per token (one fixed matrix state per head at decode: "Kimi K3 NPU Training",
// section 模型结构, step 4; replay of cached inputs to rebuild the state:
// "Kimi K3 模型结构（7）：结构决定系统", section KDA 状态回滚):
//     S <- diag(alpha) S;  p = S^T k;  u = beta (v - p);  S <- S + k u^T;
//     o = scale S^T q = scale ((diag(alpha) S)^T q + u (k . q))
// The second form of o lets one reduction produce both S^T k and S^T q from
// the decayed state.
//
// Layout and work split: one CTA of 256 threads per (sequence, head).  The
// state S [D x D] (row = key channel, dv contiguous) lives in registers by
// column blocks: warp w owns the D/8 columns [w*D/8, (w+1)*D/8) over all D
// rows, and within it lane l = 4 rg + cq owns the D/32 columns starting at
// w*D/8 + cq*D/32 of rows [rg*D/8, (rg+1)*D/8).  The reductions over rows of
// S^T k and S^T q then stay inside a warp: a reduce-scatter over the 8 row
// groups (three shuffle levels) leaves each lane one column's sum, the lanes
// holding S^T k form u, and shuffles hand u to the lanes that own its column
// and to the lanes holding S^T q (which write o).  No CTA barrier runs in the
// token loop; the warps only share the step's staged inputs.  The arithmetic
// works on pairs of a lane's columns with packed f32x2 instructions.  One
// head-step reads and writes 4*D*D bytes of state: HBM-bound at T_step = 1,
// and bound by the per-token arithmetic as T_step grows.
#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int kDecodeThreads = 256;
constexpr int kMaxTstep = 8;

template <int N> struct VecF;
template <> struct VecF<2> { using T = float2; };
template <> struct VecF<4> { using T = float4; };


// 16 bytes of inputs (8 bf16 or 4 float32) from global memory as float32, and
// the float32 values to shared memory
__device__ __forceinline__ void ldg_chunk(const __nv_bfloat16* p, float (&x)[8]) {
  const uint4 u = __ldg(reinterpret_cast<const uint4*>(p));
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    x[2 * e] = __uint_as_float(w[e] << 16);
    x[2 * e + 1] = __uint_as_float(w[e] & 0xffff0000u);
  }
}
__device__ __forceinline__ void ldg_chunk(const float* p, float (&x)[4]) {
  const float4 u = __ldg(reinterpret_cast<const float4*>(p));
  x[0] = u.x; x[1] = u.y; x[2] = u.z; x[3] = u.w;
}
template <int N>
__device__ __forceinline__ void st_chunk(float* p, const float (&x)[N]) {
#pragma unroll
  for (int e = 0; e < N; e += 4)
    *reinterpret_cast<float4*>(p + e) = make_float4(x[e], x[e + 1], x[e + 2], x[e + 3]);
}

// One level of a reduce-scatter over the lanes that differ in bit `m`: the
// lane with that bit set keeps (and adds its partner's copy of) the upper
// HALF values, the other lane the lower ones; the kept sums move to v[0..HALF).
template <int HALF, int N>
__device__ __forceinline__ void rs_level(float (&v)[N], int lane, int m) {
  const bool up = (lane & m) != 0;
#pragma unroll
  for (int j = 0; j < HALF; ++j) {
    const float send = up ? v[j] : v[HALF + j];
    const float keep = up ? v[HALF + j] : v[j];
    v[j] = keep + __shfl_xor_sync(0xffffffffu, send, m);
  }
}

// kCommit: per-sequence commit counts (num_commit) decide which state is written
// back; otherwise the state after all Tstep tokens is.
// kPre: the fused input preprocessing `pre` is applied while the inputs are staged.
template <int D, typename TIn, typename TOut, bool kCommit, bool kPre>
__global__ void __launch_bounds__(kDecodeThreads, 2)
kda_decode_kernel(const TIn* __restrict__ q, const TIn* __restrict__ k,
                  const TIn* __restrict__ v, const TIn* __restrict__ g,
                  const TIn* __restrict__ beta, float* __restrict__ state,
                  TOut* __restrict__ out, int H, int Tstep, float scale,
                  const int32_t* __restrict__ num_commit, unsigned int* status,
                  Preproc pre) {
  constexpr int RPL = D / 8;   // state rows per lane (one row group)
  constexpr int CPL = D / 32;  // state columns per lane
  constexpr int P = CPL / 2;   // column pairs per lane (packed arithmetic)
  constexpr int WC = D / 8;    // columns per warp
  constexpr int DP = D + 32;   // staged row length: 4 pad floats after each row group
  using Vec = typename VecF<CPL>::T;

  // alpha, k and q are read by row group: padding each group of RPL channels by
  // 4 floats puts the 8 groups' 16-byte reads on distinct banks
  __shared__ __align__(16) float s_k[kMaxTstep][DP];
  __shared__ __align__(16) float s_q[kMaxTstep][DP];
  __shared__ __align__(16) float s_a[kMaxTstep][DP];   // alpha = exp(g)
  __shared__ __align__(16) float s_v[kMaxTstep][D];
  __shared__ float s_b[kMaxTstep];
  __shared__ float s_kq[kMaxTstep];
  auto pidx = [](int c) { return c + (c / RPL) * 4; };

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int rg = lane >> 2, cq = lane & 3;
  const int row0 = rg * RPL, col0 = warp * WC + cq * CPL;
  const int64_t nh = blockIdx.x;  // n * H + h
  const int64_t n = nh / H, h = nh % H;

  // Issue the state loads first: they are the HBM traffic that matters.
  float* Sg = state + nh * (int64_t)D * D;
  float2 S[RPL][P];
#pragma unroll
  for (int i = 0; i < RPL; ++i) {
    const Vec x = *reinterpret_cast<const Vec*>(Sg + (int64_t)(row0 + i) * D + col0);
    const float2* xf = reinterpret_cast<const float2*>(&x);
#pragma unroll
    for (int c = 0; c < P; ++c) S[i][c] = xf[c];
  }

  // Stage the step's inputs (Tstep tokens) in shared memory as float32, one
  // 16-byte chunk per lane: warps 0-3 take q and k, a group of CR lanes per
  // token row, and form that token's norms (fused preprocessing) and k . q by
  // shuffles inside the group; warps 4-7 take v, the gate (a scalar gate per
  // (token, head) is shared by the channels) and beta.
  constexpr int kE = 16 / (int)sizeof(TIn);  // elements per chunk
  constexpr int CR = D / kE;                 // chunks (lanes) per token row: 8 .. 32
  const float gsc = kPre && pre.gate_scale ? pre.gate_scale[h] : 1.f;
  const int rows = Tstep * CR;
  if (warp < 4) {
    for (int base = warp * 32; base < rows; base += 128) {  // warp-uniform trip count
      const int i = base + lane, t = i / CR, c0 = (i % CR) * kE;
      const bool on = i < rows;  // whole token rows are on or off
      float xk[kE], xq[kE];
      if (on) {
        const int64_t x = ((n * Tstep + t) * H + h) * D + c0;
        ldg_chunk(k + x, xk);
        ldg_chunk(q + x, xq);
      } else {
#pragma unroll
        for (int e = 0; e < kE; ++e) xk[e] = xq[e] = 0.f;
      }
      if (kPre && pre.l2) {
        float sk = 0.f, sq = 0.f;
#pragma unroll
        for (int e = 0; e < kE; ++e) {
          sk = fmaf(xk[e], xk[e], sk);
          sq = fmaf(xq[e], xq[e], sq);
        }
#pragma unroll
        for (int o = CR / 2; o > 0; o >>= 1) {
          sk += __shfl_xor_sync(0xffffffffu, sk, o);
          sq += __shfl_xor_sync(0xffffffffu, sq, o);
        }
        const float ik = inv_l2(sk), iq = inv_l2(sq);
#pragma unroll
        for (int e = 0; e < kE; ++e) {
          xk[e] *= ik;  // kept in float32 (the products take float32)
          xq[e] *= iq;
        }
      }
      float acc = 0.f;
#pragma unroll
      for (int e = 0; e < kE; ++e) acc = fmaf(xk[e], xq[e], acc);
#pragma unroll
      for (int o = CR / 2; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
      if (on) {
        st_chunk(&s_k[t][pidx(c0)], xk);  // a chunk lies inside one row group
        st_chunk(&s_q[t][pidx(c0)], xq);
        if (c0 == 0) s_kq[t] = acc;
      }
    }
  } else {
    // every load first (one memory round trip), then the conversions: v by
    // chunks; an activated or per-head gate one element per thread (the
    // activation is the longest work of the staging), a plain gate by chunks
    constexpr int kVmax = (kMaxTstep * CR + 127) / 128;  // chunks per thread
    constexpr int kGmax = kMaxTstep * D / 128;           // gate elements per thread
    const int j0 = tid - 128;
    const bool g_elems = kPre && (pre.gate || pre.per_head);
    float xv[kVmax][kE], xa[kVmax][kE], gr[kGmax];
#pragma unroll
    for (int jj = 0; jj < kVmax; ++jj) {
      const int i = j0 + 128 * jj;
      if (i < rows) {
        const int64_t x = ((n * Tstep + i / CR) * H + h) * D + (i % CR) * kE;
        ldg_chunk(v + x, xv[jj]);
        if (!g_elems) ldg_chunk(g + x, xa[jj]);
      }
    }
    if (g_elems) {
#pragma unroll
      for (int jj = 0; jj < kGmax; ++jj) {
        const int i = j0 + 128 * jj;
        if (i < Tstep * D) {
          const int64_t xt = (n * Tstep + i / D) * H + h;
          gr[jj] = to_f32(g[pre.per_head ? xt : xt * D + i % D]);
        }
      }
#pragma unroll
      for (int jj = 0; jj < kGmax; ++jj) {
        const int i = j0 + 128 * jj;
        if (i < Tstep * D) {
          float gv = gr[jj];
          if (pre.gate) gv = round_to<TIn>(gsc * neg_softplus(gv));
          s_a[i / D][pidx(i % D)] = expf(gv);
        }
      }
    }
#pragma unroll
    for (int jj = 0; jj < kVmax; ++jj) {
      const int i = j0 + 128 * jj;
      if (i < rows) {
        const int t = i / CR, c0 = (i % CR) * kE;
        st_chunk(&s_v[t][c0], xv[jj]);
        if (!g_elems) {
#pragma unroll
          for (int e = 0; e < kE; ++e) xa[jj][e] = expf(xa[jj][e]);
          st_chunk(&s_a[t][pidx(c0)], xa[jj]);
        }
      }
    }
    if (tid - 128 < Tstep) {
      const int t = tid - 128;
      float bv = to_f32(beta[(n * Tstep + t) * H + h]);
      if (kPre && pre.beta) bv = round_to<TIn>(sigmoid_f(bv));
      s_b[t] = bv;
    }
  }
  __syncthreads();

  // The state written back is the one after the first `commit` tokens (all of
  // them unless per-sequence counts are given); every token still produces its
  // output.  A count outside [0, Tstep] is latched and commits nothing.
  int commit = Tstep;
  if (kCommit) {
    commit = num_commit[n];
    if (commit < 0 || commit > Tstep) {
      if (tid == 0) latch_status(status, KDA_ERR_INVALID_ARG);
      commit = 0;
    }
  }
  auto store_state = [&]() {
#pragma unroll
    for (int i = 0; i < RPL; ++i) {
      Vec x;
      float2* xf = reinterpret_cast<float2*>(&x);
#pragma unroll
      for (int c = 0; c < P; ++c) xf[c] = S[i][c];
      *reinterpret_cast<Vec*>(Sg + (int64_t)(row0 + i) * D + col0) = x;
    }
  };
  // after the reduce-scatter: lanes of row groups 0-3 hold S^T k, lanes of row
  // groups 4-7 S^T q, of column col0 + my_c (row groups 4 + r and r pair up)
  const bool holds_k = rg < 4;
  const int my_c = CPL == 4 ? (rg & 3) : ((rg >> 1) & 1);
  const bool writes_o = !holds_k && (CPL == 4 || (rg & 1) == 0);
  const int pa = pidx(row0);

  for (int t = 0; t < Tstep; ++t) {
    // this lane's rows of alpha, k and q, read as 16-byte vectors (lanes of one
    // row group read the same addresses)
    float a[RPL], kr[RPL], qr[RPL];
#pragma unroll
    for (int r4 = 0; r4 < RPL / 4; ++r4) {
      const float4 av = *reinterpret_cast<const float4*>(&s_a[t][pa + 4 * r4]);
      const float4 kv = *reinterpret_cast<const float4*>(&s_k[t][pa + 4 * r4]);
      const float4 qv = *reinterpret_cast<const float4*>(&s_q[t][pa + 4 * r4]);
      a[4 * r4] = av.x; a[4 * r4 + 1] = av.y; a[4 * r4 + 2] = av.z; a[4 * r4 + 3] = av.w;
      kr[4 * r4] = kv.x; kr[4 * r4 + 1] = kv.y; kr[4 * r4 + 2] = kv.z; kr[4 * r4 + 3] = kv.w;
      qr[4 * r4] = qv.x; qr[4 * r4 + 1] = qv.y; qr[4 * r4 + 2] = qv.z; qr[4 * r4 + 3] = qv.w;
    }
    // decay and partial reductions over this lane's rows, two columns at a time
    float2 pk[P], pq[P];
#pragma unroll
    for (int c = 0; c < P; ++c) pk[c] = pq[c] = make_float2(0.f, 0.f);
#pragma unroll
    for (int i = 0; i < RPL; ++i) {
      const float2 a2 = make_float2(a[i], a[i]), k2 = make_float2(kr[i], kr[i]);
      const float2 q2 = make_float2(qr[i], qr[i]);
#pragma unroll
      for (int c = 0; c < P; ++c) {
        S[i][c] = mul2(S[i][c], a2);
        pk[c] = fma2(S[i][c], k2, pk[c]);
        pq[c] = fma2(S[i][c], q2, pq[c]);
      }
    }
    // sums over the 8 row groups, scattered: one (column, k or q) sum per lane
    float red;
    if constexpr (CPL == 4) {
      float vals[8] = {pk[0].x, pk[0].y, pk[1].x, pk[1].y, pq[0].x, pq[0].y, pq[1].x, pq[1].y};
      rs_level<4>(vals, lane, 16);
      rs_level<2>(vals, lane, 8);
      rs_level<1>(vals, lane, 4);
      red = vals[0];
    } else {
      float vals[4] = {pk[0].x, pk[0].y, pq[0].x, pq[0].y};
      rs_level<2>(vals, lane, 16);
      rs_level<1>(vals, lane, 8);
      red = vals[0] + __shfl_xor_sync(0xffffffffu, vals[0], 4);
    }
    const int col = col0 + my_c;
    const float u = holds_k ? s_b[t] * (s_v[t][col] - red) : 0.f;
    const float u_q = __shfl_xor_sync(0xffffffffu, u, 16);  // to the S^T q lane of the column
    if (writes_o && (!kCommit || out))
      out[((n * Tstep + t) * H + h) * D + col] = from_f32<TOut>(scale * fmaf(u_q, s_kq[t], red));
    // u of this lane's columns, from the lanes that formed them
    float uc[CPL];
#pragma unroll
    for (int c = 0; c < CPL; ++c) uc[c] = __shfl_sync(0xffffffffu, u, ((c * (4 / CPL)) << 2) | cq);
    // rank-1 write S <- S + k u^T
#pragma unroll
    for (int i = 0; i < RPL; ++i) {
      const float2 k2 = make_float2(kr[i], kr[i]);
#pragma unroll
      for (int c = 0; c < P; ++c) S[i][c] = fma2(k2, make_float2(uc[2 * c], uc[2 * c + 1]), S[i][c]);
    }
    if (kCommit && t + 1 == commit) store_state();
  }
  if (!kCommit) store_state();
}

template <int D, typename TIn, bool kPre>
cudaError_t launch_pre(const DecodeArgs& a) {
  const int64_t blocks = (int64_t)a.B * a.H;
  const TIn* q = static_cast<const TIn*>(a.q);
  const TIn* k = static_cast<const TIn*>(a.k);
  const TIn* v = static_cast<const TIn*>(a.v);
  const TIn* g = static_cast<const TIn*>(a.g);
  const TIn* b = static_cast<const TIn*>(a.beta);
  const bool f32 = a.out_dtype == KDA_F32;
  float* of = static_cast<float*>(a.out);
  __nv_bfloat16* ob = static_cast<__nv_bfloat16*>(a.out);
  const dim3 grid((unsigned)blocks);
  if (a.num_commit) {
    if (f32)
      kda_decode_kernel<D, TIn, float, true, kPre><<<grid, kDecodeThreads, 0, a.stream>>>(
          q, k, v, g, b, a.state, of, a.H, a.Tstep, a.scale, a.num_commit, a.status, a.pre);
    else
      kda_decode_kernel<D, TIn, __nv_bfloat16, true, kPre><<<grid, kDecodeThreads, 0, a.stream>>>(
          q, k, v, g, b, a.state, ob, a.H, a.Tstep, a.scale, a.num_commit, a.status, a.pre);
  } else {
    if (f32)
      kda_decode_kernel<D, TIn, float, false, kPre><<<grid, kDecodeThreads, 0, a.stream>>>(
          q, k, v, g, b, a.state, of, a.H, a.Tstep, a.scale, nullptr, a.status, a.pre);
    else
      kda_decode_kernel<D, TIn, __nv_bfloat16, false, kPre><<<grid, kDecodeThreads, 0, a.stream>>>(
          q, k, v, g, b, a.state, ob, a.H, a.Tstep, a.scale, nullptr, a.status, a.pre);
  }
  return cudaGetLastError();
}

template <int D, typename TIn>
cudaError_t launch_d_in(const DecodeArgs& a) {
  if ((int64_t)a.B * a.H == 0 || a.Tstep == 0) return cudaSuccess;
  if (a.pre.l2 || a.pre.gate || a.pre.beta || a.pre.per_head) return launch_pre<D, TIn, true>(a);
  return launch_pre<D, TIn, false>(a);
}

}  // namespace

cudaError_t launch_decode(const DecodeArgs& a) {
  if (a.D == 128)
    return a.in_dtype == KDA_F32 ? launch_d_in<128, float>(a) : launch_d_in<128, __nv_bfloat16>(a);
  return a.in_dtype == KDA_F32 ? launch_d_in<64, float>(a) : launch_d_in<64, __nv_bfloat16>(a);
}

}  // namespace kda
