// KDA chunkwise prefill, float32 path (every product in float32 FFMA).
//
// Chunkwise form of the recurrence (parallel inside a chunk, recurrent across
// chunks: "Kimi K3 技术报告摘要", section 1, 训练策略 table, KDA row).  With
// Gam = inclusive per-channel prefix sum of g inside the chunk:
//   A[i][j]   = beta_i sum_c k_ic k_jc exp(Gam_ic - Gam_jc)     (j < i)
//   Aqk[i][j] =        sum_c q_ic k_jc exp(Gam_ic - Gam_jc)     (j <= i)
//   T  = (I + A)^-1                      forward substitution
//   W  = T diag(beta) (K * e^Gam),   U = T diag(beta) V - W S
//   O  = scale ((Q * e^Gam) S + Aqk U)
//   S <- diag(e^Gam_last) S + (K * e^(Gam_last - Gam))^T U
// The decayed products use exp of differences, which never exceed 1, so this
// path has no range limit on g.  Gam is summed in float64 and kept as a float
// hi + lo pair, so a difference of two nearby prefix sums stays exact even
// after a run of very large gates (g is floored at -1e4, where e^g is already
// 0 in float32; g = -inf, alpha = 0, is taken as that floor).  One CTA (256
// threads) per (sequence, head) chain, state S in shared memory.  Chunk: 64
// tokens at d = 64, 32 at d = 128 (the rearrangement is exact for any chunk
// length).
#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int kThreads = 256;

template <int D, int C>
struct F32Smem {
  static constexpr int LD = D + 1;  // padded row stride: row-per-thread reads hit distinct banks
  static constexpr size_t floats =
      (size_t)D * D                 // S
      + 8 * (size_t)C * LD          // q(->Qhat), k(->Khat), v, Gam (hi, lo), Kb, W, U
      + 3 * (size_t)C * C           // A, Aqk, T
      + C + 2 * D;                  // beta, Gam_last (hi, lo)
  static constexpr size_t bytes = floats * sizeof(float);
};

// kPre: the fused input preprocessing `pre` is applied while the chunk is loaded.
template <int D, int C, typename TIn, typename TOut, bool kPre>
__global__ void __launch_bounds__(kThreads, 1)
kda_prefill_f32_kernel(const TIn* __restrict__ q, const TIn* __restrict__ k,
                       const TIn* __restrict__ v, const TIn* __restrict__ g,
                       const TIn* __restrict__ beta, SeqView seqs,
                       const int32_t* __restrict__ order, const float* __restrict__ h0,
                       TOut* __restrict__ out, float* __restrict__ hT, int H, float scale,
                       unsigned int* __restrict__ status, float* __restrict__ ckpt,
                       const int32_t* __restrict__ ckpt_off, int64_t ckpt_rows,
                       int64_t ckpt_interval, Preproc pre) {
  using L = F32Smem<D, C>;
  constexpr int LD = L::LD;
  extern __shared__ float smem[];
  float* S = smem;
  float* sq = S + D * D;
  float* sk = sq + C * LD;
  float* sv = sk + C * LD;
  float* sG = sv + C * LD;
  float* sGlo = sG + C * LD;
  float* sKb = sGlo + C * LD;
  float* sW = sKb + C * LD;
  float* sU = sW + C * LD;
  float* sA = sU + C * LD;
  float* sAqk = sA + C * C;
  float* sT = sAqk + C * C;
  float* sb = sT + C * C;
  float* sGl = sb + C;
  float* sGllo = sGl + D;

  // a malformed cu_seqlens is latched by the scheduler before this kernel starts
  if (status && *(volatile const unsigned int*)status == (unsigned)KDA_ERR_BAD_SEQLENS) return;
  const int tid = threadIdx.x;
  const int item = blockIdx.x;
  const int n = order ? order[item / H] : item / H;
  const int h = item % H;
  int64_t t0, len;
  seqs.get(n, t0, len);

  const int64_t st = ((int64_t)n * H + h) * D * D;
  for (int i = tid; i < D * D; i += kThreads) S[i] = h0 ? h0[st + i] : 0.f;
  const int64_t ck_base =
      ckpt_base(ckpt, ckpt_off, ckpt_rows, ckpt_interval, n, len, status, tid == 0);

  const float gsc = kPre && pre.gate_scale ? pre.gate_scale[h] : 1.f;
  for (int64_t cs = 0; cs < len; cs += C) {
    const int nv = (int)(len - cs < C ? len - cs : C);
    __syncthreads();  // previous chunk finished with every buffer
    // 1. load the chunk; tokens past the sequence end act as g = 0, beta = 0
    for (int i = tid; i < C * D; i += kThreads) {
      const int t = i / D, c = i % D;
      float xq = 0.f, xk = 0.f, xv = 0.f, xg = 0.f;
      if (t < nv) {
        const int64_t x = ((t0 + cs + t) * H + h) * D + c;
        xq = to_f32(q[x]); xk = to_f32(k[x]); xv = to_f32(v[x]);
        xg = to_f32(g[kPre && pre.per_head ? (t0 + cs + t) * H + h : x]);  // scalar gate: shared
        if (kPre && pre.gate) xg = round_to<TIn>(gsc * neg_softplus(xg));
        xg = fmaxf(xg, -1e4f);
      }
      sq[t * LD + c] = xq; sk[t * LD + c] = xk; sv[t * LD + c] = xv; sG[t * LD + c] = xg;
    }
    for (int t = tid; t < C; t += kThreads) {
      float bt = t < nv ? to_f32(beta[(t0 + cs + t) * H + h]) : 0.f;
      if (kPre && pre.beta && t < nv) bt = round_to<TIn>(sigmoid_f(bt));
      sb[t] = bt;
    }
    __syncthreads();
    if (kPre && pre.l2) {  // q, k normalised per token, one warp per token
      const int warp = tid >> 5, lane = tid & 31;
      for (int t = warp; t < nv; t += kThreads / 32) {
        float s2k = 0.f, s2q = 0.f;
        for (int c = lane; c < D; c += 32) {
          s2k = fmaf(sk[t * LD + c], sk[t * LD + c], s2k);
          s2q = fmaf(sq[t * LD + c], sq[t * LD + c], s2q);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          s2k += __shfl_xor_sync(0xffffffffu, s2k, o);
          s2q += __shfl_xor_sync(0xffffffffu, s2q, o);
        }
        const float ik = inv_l2(s2k), iq = inv_l2(s2q);
        for (int c = lane; c < D; c += 32) {
          sk[t * LD + c] *= ik;  // kept in float32
          sq[t * LD + c] *= iq;
        }
      }
      __syncthreads();
    }
    // 2. inclusive log-decay prefix sums per channel (float64, kept as hi + lo)
    for (int c = tid; c < D; c += kThreads) {
      double run = 0.0;
      for (int t = 0; t < C; ++t) {
        run += (double)sG[t * LD + c];
        const float hi = (float)run;
        sG[t * LD + c] = hi;
        sGlo[t * LD + c] = (float)(run - (double)hi);
      }
      const float hi = (float)run;
      sGl[c] = hi;
      sGllo[c] = (float)(run - (double)hi);
    }
    __syncthreads();
    // 3. decayed key-key and query-key products (lower triangle)
    for (int p = tid; p < C * C; p += kThreads) {
      const int i = p / C, j = p % C;
      float ak = 0.f, aq = 0.f;
      if (j <= i) {
        for (int c = 0; c < D; ++c) {
          const float e = expf((sG[i * LD + c] - sG[j * LD + c]) +
                               (sGlo[i * LD + c] - sGlo[j * LD + c]));
          const float kj = sk[j * LD + c] * e;
          ak = fmaf(sk[i * LD + c], kj, ak);
          aq = fmaf(sq[i * LD + c], kj, aq);
        }
      }
      sA[p] = j < i ? sb[i] * ak : 0.f;
      sAqk[p] = aq;
    }
    __syncthreads();
    // 4. scaled operands: Kb = beta K e^Gam, Qhat = Q e^Gam (in place of q),
    //    Khat = K e^(Gam_last - Gam) (in place of k)
    for (int i = tid; i < C * D; i += kThreads) {
      const int t = i / D, c = i % D;
      const float G = sG[t * LD + c];
      const float e = expf(G);
      sKb[t * LD + c] = sb[t] * sk[t * LD + c] * e;
      sq[t * LD + c] *= e;
      sk[t * LD + c] *= expf((sGl[c] - G) + (sGllo[c] - sGlo[t * LD + c]));
    }
    // 5. T = (I + A)^-1 by forward substitution, one row at a time
    for (int i = 0; i < C; ++i) {
      for (int j = tid; j < C; j += kThreads) {
        float acc = 0.f;
        if (j < i)
          for (int m = j; m < i; ++m) acc = fmaf(sA[i * C + m], sT[m * C + j], acc);
        sT[i * C + j] = j < i ? -acc : (j == i ? 1.f : 0.f);
      }
      __syncthreads();
    }
    // 6. W = T Kb and U~ = T diag(beta) V
    for (int i = tid; i < C * D; i += kThreads) {
      const int r = i / D, c = i % D;
      float w = 0.f, u = 0.f;
      for (int j = 0; j <= r; ++j) {
        const float tij = sT[r * C + j];
        w = fmaf(tij, sKb[j * LD + c], w);
        u = fmaf(tij * sb[j], sv[j * LD + c], u);
      }
      sW[r * LD + c] = w;
      sU[r * LD + c] = u;
    }
    __syncthreads();
    // 7. U = U~ - W S
    for (int i = tid; i < C * D; i += kThreads) {
      const int r = i / D, c = i % D;
      float acc = sU[r * LD + c];
      for (int m = 0; m < D; ++m) acc = fmaf(-sW[r * LD + m], S[m * D + c], acc);
      sU[r * LD + c] = acc;
    }
    __syncthreads();
    // 8. O = scale (Qhat S + Aqk U)
    for (int i = tid; i < C * D; i += kThreads) {
      const int r = i / D, c = i % D;
      if (r >= nv) continue;
      float acc = 0.f;
      for (int m = 0; m < D; ++m) acc = fmaf(sq[r * LD + m], S[m * D + c], acc);
      for (int j = 0; j <= r; ++j) acc = fmaf(sAqk[r * C + j], sU[j * LD + c], acc);
      out[((t0 + cs + r) * H + h) * D + c] = from_f32<TOut>(scale * acc);
    }
    __syncthreads();
    // 9. S <- diag(e^Gam_last) S + Khat^T U; a checkpoint when cs + C tokens of
    // the sequence are done and that is a multiple of the interval
    const int64_t done = cs + C;
    float* ck = (ck_base >= 0 && done <= len && done % ckpt_interval == 0)
                    ? ckpt + ((ck_base + done / ckpt_interval - 1) * H + h) * D * D
                    : nullptr;
    for (int i = tid; i < D * D; i += kThreads) {
      const int m = i / D, c = i % D;
      float acc = expf(sGl[m]) * S[i];
      for (int j = 0; j < C; ++j) acc = fmaf(sk[j * LD + m], sU[j * LD + c], acc);
      S[i] = acc;
      if (ck) ck[i] = acc;
    }
  }
  __syncthreads();
  if (hT)
    for (int i = tid; i < D * D; i += kThreads) hT[st + i] = S[i];
}

template <int D, int C, typename TIn, typename TOut, bool kPre>
cudaError_t launch_p(const FwdArgs& a) {
  using L = F32Smem<D, C>;
  auto kern = kda_prefill_f32_kernel<D, C, TIn, TOut, kPre>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)L::bytes);
  if (e != cudaSuccess) return e;
  const int64_t items = (int64_t)a.N * a.H;
  if (items == 0) return cudaSuccess;
  SeqView sv{a.cu, a.T};
  kern<<<(unsigned)items, kThreads, L::bytes, a.stream>>>(
      static_cast<const TIn*>(a.q), static_cast<const TIn*>(a.k), static_cast<const TIn*>(a.v),
      static_cast<const TIn*>(a.g), static_cast<const TIn*>(a.beta), sv, a.order, a.h0,
      static_cast<TOut*>(a.out), a.hT, a.H, a.scale, a.status, a.ckpt, a.ckpt_off, a.ckpt_rows,
      a.ckpt_interval, a.pre);
  return cudaGetLastError();
}

template <int D, int C, typename TIn, typename TOut>
cudaError_t launch_t(const FwdArgs& a) {
  if (a.pre.l2 || a.pre.gate || a.pre.beta || a.pre.per_head) return launch_p<D, C, TIn, TOut, true>(a);
  return launch_p<D, C, TIn, TOut, false>(a);
}

template <int D, int C>
cudaError_t launch_d(const FwdArgs& a) {
  if (a.in_dtype == KDA_F32)
    return a.out_dtype == KDA_F32 ? launch_t<D, C, float, float>(a)
                                  : launch_t<D, C, float, __nv_bfloat16>(a);
  return a.out_dtype == KDA_F32 ? launch_t<D, C, __nv_bfloat16, float>(a)
                                : launch_t<D, C, __nv_bfloat16, __nv_bfloat16>(a);
}

}  // namespace

cudaError_t launch_prefill_f32(const FwdArgs& a) {
  return a.D == 128 ? launch_d<128, 32>(a) : launch_d<64, 64>(a);
}

}  // namespace kda
