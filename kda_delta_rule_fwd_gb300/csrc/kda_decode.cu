// KDA decode: T_step (1..8) tokens applied in order to per-head float32 states
// resident in device memory, updated in place.
//
// Per token (one fixed matrix state per head at decode: "Kimi K3 NPU Training",
// section 模型结构, step 4; replay of cached inputs to rebuild the state:
// "Kimi K3 模型结构（7）：结构决定系统", section KDA 状态回滚):
//     S <- diag(alpha) S;  p = S^T k;  u = beta (v - p);  S <- S + k u^T;
//     o = scale S^T q = scale ((diag(alpha) S)^T q + u (k . q))
// The second form of o lets one cross-warp reduction produce both S^T k and
// S^T q from the decayed state.
//
// Layout and work split: one CTA of 256 threads per (sequence, head).  The
// state S [D x D] (row = key channel, dv contiguous) lives in registers: warp w
// owns rows [w*D/8, (w+1)*D/8) and lane l owns columns [l*D/32, (l+1)*D/32), so
// every warp load/store of a state row is one contiguous, vectorised access.
// The token loop works on pairs of a lane's columns with packed f32x2 arithmetic.
// One head-step reads and writes 4*D*D bytes of state: HBM-bound at T_step = 1,
// and bound by the per-token arithmetic and barriers as T_step grows.
#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int kDecodeThreads = 256;
constexpr int kMaxTstep = 8;

template <int N> struct VecF;
template <> struct VecF<2> { using T = float2; };
template <> struct VecF<4> { using T = float4; };


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
  constexpr int R = D / 8;     // state rows per warp
  constexpr int CPL = D / 32;  // state columns per lane
  constexpr int P = CPL / 2;   // column pairs per lane (packed arithmetic)
  using Vec = typename VecF<CPL>::T;

  __shared__ __align__(16) float s_k[kMaxTstep][D];
  __shared__ __align__(16) float s_q[kMaxTstep][D];
  __shared__ __align__(16) float s_a[kMaxTstep][D];   // alpha = exp(g)
  __shared__ __align__(16) float s_v[kMaxTstep][D];
  __shared__ float s_b[kMaxTstep];
  __shared__ float s_kq[kMaxTstep];
  __shared__ __align__(16) float s_red[8][2][D];      // per-warp partial S^T k and S^T q
  __shared__ __align__(16) float s_u[D];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t nh = blockIdx.x;  // n * H + h
  const int64_t n = nh / H, h = nh % H;

  // Issue the state loads first: they are the HBM traffic that matters.
  float* Sg = state + nh * (int64_t)D * D;
  float2 S[R][P];
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const Vec x = *reinterpret_cast<const Vec*>(Sg + (int64_t)(warp * R + r) * D + lane * CPL);
    const float2* xf = reinterpret_cast<const float2*>(&x);
#pragma unroll
    for (int c = 0; c < P; ++c) S[r][c] = xf[c];
  }

  // Stage the step's inputs (Tstep tokens) in shared memory as float32 (with the
  // fused preprocessing: a scalar gate per (token, head) is shared by the channels).
  const float gsc = kPre && pre.gate_scale ? pre.gate_scale[h] : 1.f;
  for (int i = tid; i < Tstep * D; i += kDecodeThreads) {
    const int t = i / D, c = i % D;
    const int64_t x = ((n * Tstep + t) * H + h) * D + c;
    s_k[t][c] = to_f32(k[x]);
    s_q[t][c] = to_f32(q[x]);
    float gv = to_f32(g[kPre && pre.per_head ? (n * Tstep + t) * H + h : x]);
    if (kPre && pre.gate) gv = round_to<TIn>(gsc * neg_softplus(gv));
    s_a[t][c] = expf(gv);
    s_v[t][c] = to_f32(v[x]);
  }
  if (tid < Tstep) {
    float bv = to_f32(beta[(n * Tstep + tid) * H + h]);
    if (kPre && pre.beta) bv = round_to<TIn>(sigmoid_f(bv));
    s_b[tid] = bv;
  }
  __syncthreads();
  // k . q per token, one warp per token (which first normalises that token's q
  // and k when asked; each lane touches the same channels in both loops)
  if (warp < Tstep) {
    if (kPre && pre.l2) {
      float sk = 0.f, sq = 0.f;
      for (int c = lane; c < D; c += 32) {
        sk = fmaf(s_k[warp][c], s_k[warp][c], sk);
        sq = fmaf(s_q[warp][c], s_q[warp][c], sq);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        sk += __shfl_xor_sync(0xffffffffu, sk, o);
        sq += __shfl_xor_sync(0xffffffffu, sq, o);
      }
      const float ik = inv_l2(sk), iq = inv_l2(sq);
      for (int c = lane; c < D; c += 32) {
        s_k[warp][c] *= ik;  // kept in float32 (the products take float32)
        s_q[warp][c] *= iq;
      }
    }
    float acc = 0.f;
    for (int c = lane; c < D; c += 32) acc += s_k[warp][c] * s_q[warp][c];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (lane == 0) s_kq[warp] = acc;
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
    for (int r = 0; r < R; ++r) {
      Vec x;
      float2* xf = reinterpret_cast<float2*>(&x);
#pragma unroll
      for (int c = 0; c < P; ++c) xf[c] = S[r][c];
      *reinterpret_cast<Vec*>(Sg + (int64_t)(warp * R + r) * D + lane * CPL) = x;
    }
  };

  for (int t = 0; t < Tstep; ++t) {
    // this warp's rows of alpha, k and q, read as 16-byte vectors
    float a[R], kr[R], qr[R];
#pragma unroll
    for (int r4 = 0; r4 < R / 4; ++r4) {
      const float4 av = *reinterpret_cast<const float4*>(&s_a[t][warp * R + 4 * r4]);
      const float4 kv = *reinterpret_cast<const float4*>(&s_k[t][warp * R + 4 * r4]);
      const float4 qv = *reinterpret_cast<const float4*>(&s_q[t][warp * R + 4 * r4]);
      a[4 * r4] = av.x; a[4 * r4 + 1] = av.y; a[4 * r4 + 2] = av.z; a[4 * r4 + 3] = av.w;
      kr[4 * r4] = kv.x; kr[4 * r4 + 1] = kv.y; kr[4 * r4 + 2] = kv.z; kr[4 * r4 + 3] = kv.w;
      qr[4 * r4] = qv.x; qr[4 * r4 + 1] = qv.y; qr[4 * r4 + 2] = qv.z; qr[4 * r4 + 3] = qv.w;
    }
    // decay and partial reductions over this warp's rows, two columns at a time
    float2 pk[P], pq[P];
#pragma unroll
    for (int c = 0; c < P; ++c) pk[c] = pq[c] = make_float2(0.f, 0.f);
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const float2 a2 = make_float2(a[r], a[r]), k2 = make_float2(kr[r], kr[r]);
      const float2 q2 = make_float2(qr[r], qr[r]);
#pragma unroll
      for (int c = 0; c < P; ++c) {
        S[r][c] = mul2(S[r][c], a2);
        pk[c] = fma2(S[r][c], k2, pk[c]);
        pq[c] = fma2(S[r][c], q2, pq[c]);
      }
    }
    {
      Vec vk, vq;
      float2* fk = reinterpret_cast<float2*>(&vk);
      float2* fq = reinterpret_cast<float2*>(&vq);
#pragma unroll
      for (int c = 0; c < P; ++c) { fk[c] = pk[c]; fq[c] = pq[c]; }
      *reinterpret_cast<Vec*>(&s_red[warp][0][lane * CPL]) = vk;
      *reinterpret_cast<Vec*>(&s_red[warp][1][lane * CPL]) = vq;
    }
    __syncthreads();
    if (tid < D) {
      float sk = 0.f, sq = 0.f;
#pragma unroll
      for (int w = 0; w < 8; ++w) {
        sk += s_red[w][0][tid];
        sq += s_red[w][1][tid];
      }
      const float u = s_b[t] * (s_v[t][tid] - sk);
      s_u[tid] = u;
      const float o = scale * fmaf(u, s_kq[t], sq);
      if (!kCommit || out) out[((n * Tstep + t) * H + h) * D + tid] = from_f32<TOut>(o);
    }
    __syncthreads();
    // rank-1 write S <- S + k u^T
    float2 u[P];
    {
      const Vec uv = *reinterpret_cast<const Vec*>(&s_u[lane * CPL]);
      const float2* uf = reinterpret_cast<const float2*>(&uv);
#pragma unroll
      for (int c = 0; c < P; ++c) u[c] = uf[c];
    }
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const float2 k2 = make_float2(kr[r], kr[r]);
#pragma unroll
      for (int c = 0; c < P; ++c) S[r][c] = fma2(k2, u[c], S[r][c]);
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
