// KDA backward: the gradients of L = sum(o * do) + sum(hT * dhT) with respect to
// q, k, v, g (log alpha), beta and h0, for the forward of kda_fwd ("Kimi K3 NPU
// Training", section NPU 算子支持度, row KDA 反向: dq, dk, dv, dbeta, dgate and
// dstate).
//
// One CTA of 512 threads per (sequence, head) chain, float32 throughout, in
// sub-chunks of C = 16 tokens (the M of the warp-level m16n8k8 products).
//   1. Forward sweep: the state at the start of every sub-chunk is recomputed
//      and stored in the workspace.
//   2. Backward sweep, last sub-chunk first, carrying dS = dL/dS at the current
//      sub-chunk's end (dhT at the start of the sweep).
//
// Per sub-chunk, with S its start state, Gam the in-sub-chunk prefix sum of g,
// Gl = Gam[C-1] (tokens past the sequence end carry zeros, so Gl is the last
// valid token's), Kb = K e^Gam, Qb = Q e^Gam, Kh = K e^(Gl - Gam),
//   P[i][j] = sum_c K_ic K_jc e^(Gam_ic - Gam_jc)  (j < i),  M likewise with Q_i
//   (j <= i),  T = (I + diag(beta) P)^-1,  X = V - Kb S,  U = T diag(beta) X,
//   O = scale (Qb S + M U),  S_end = diag(e^Gl) S + Kh^T U
// (the token recurrence unrolled over the sub-chunk; u_t are the rows of U).
// The backward applies the chain rule to these steps:
//   dU = scale M^T dO + Kh dS;  dY = T^T dU, dX = diag(beta) dY, dV = dX,
//   dbeta += rowsum(dY . X);  dT = dU (diag(beta) X)^T, dA = -T^T dT T^T
//   (strictly lower), dbeta_i += sum_j dA_ij P_ij, dP = diag(beta) dA;
//   dM = scale dO U^T (lower);  dKh = U dS^T, dQb = scale dO S^T, dKb = -dX S^T;
//   per channel, the pairwise factors give dq, dk and dGam; the elementwise
//   factors add dQb e^Gam, dKb e^Gam, dKh e^(Gl - Gam) and their dGam terms;
//   dGl = e^Gl rowsum(dS . S) + colsum(Kh . dKh);  dg = reverse prefix sum of dGam
//   (dGl added at the last row);  dS <- diag(e^Gl) dS + scale Qb^T dO - Kb^T dX.
// Pairwise factors are exponentials of differences (each at most 1), so finite
// gates of any size stay finite; a gate of -inf is not supported here.
//
// The seven products with S, dS or a 16 x d operand on both sides run on the
// warp-level tensor-core path with the three-way tf32 split (float32
// accuracy); the 16 x 16 pieces and the per-channel exponentials run on the
// CUDA cores.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "kda_internal.cuh"
#include "kda_mma_sync.cuh"

namespace kda {
namespace {

constexpr int kBT = 512;  // threads per CTA
constexpr int kBC = 16;   // sub-chunk length
constexpr int kSL = 17;   // row stride of the 16 x 16 matrices

// shared-memory layout in floats
template <int D>
struct BwdLayout {
  static constexpr int SLD = D + 4;  // D x D state matrices
  static constexpr int CLD = D + 4;  // 16 x D sub-chunk matrices
  static constexpr int CM = kBC * CLD;
  static constexpr int S = 0;
  static constexpr int DS = S + D * SLD;
  static constexpr int Q = DS + D * SLD;
  static constexpr int K = Q + CM;
  static constexpr int G = K + CM;    // g, then Gam log2(e)
  static constexpr int KB = G + CM;
  static constexpr int QB = KB + CM;
  static constexpr int KH = QB + CM;  // Kh, then dk
  static constexpr int X = KH + CM;   // v, then X, then dX
  static constexpr int DO = X + CM;
  static constexpr int U = DO + CM;   // U, then dq
  static constexpr int DU = U + CM;   // dU, then dGam
  static constexpr int TM = DU + CM;  // T
  static constexpr int PM = TM + kBC * kSL;
  static constexpr int MM = PM + kBC * kSL;
  static constexpr int DT = MM + kBC * kSL;  // dT, then dP
  static constexpr int DM = DT + kBC * kSL;
  static constexpr int SCR = DM + kBC * kSL;  // partial dT / dM tiles (8 x 16 x 8)
  static constexpr int SCG = SCR + 1024;      // partial row sums for dGl (2 x D)
  static constexpr int BETA = SCG + 2 * D;
  static constexpr int DB = BETA + kBC;     // dbeta
  static constexpr int GL = DB + kBC;       // Gl
  static constexpr int EGL = GL + D;        // e^Gl
  static constexpr int DGL = EGL + D;       // dGl
  static constexpr int FLAG = DGL + D;      // nonzero: a pairwise factor too large to split
  static constexpr int TOTAL = FLAG + 4;
  static constexpr size_t BYTES = (size_t)TOTAL * sizeof(float);
};
static_assert(BwdLayout<128>::BYTES <= 232448, "backward shared memory");

template <typename TIn>
struct BwdParams {
  const TIn *q, *k, *v, *g, *beta;
  const float* dout;
  const float* dhT;
  const float* h0;
  SeqView seqs;
  const int32_t* order;    // packed: longest first
  const int64_t* sub_off;  // packed: first sub-chunk state row of each sequence
  int H;
  float scale;
  float *dq, *dk, *dv, *dg, *dbeta, *dh0;
  float* states;  // [rows][H][D][D]
  unsigned int* status;
};

constexpr float kLog2e = 1.4426950408889634f;
// 2^x on the special-function unit (relative error about 2^-22; results below
// 2^-126 flush to zero, where they only drop terms far below the others)
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// acc += A(m0.., 0..Kd) B(0..Kd, n0..) for one m16n8 tile, with A(r, k) =
// A[r * ars + k * acs] and B(k, n) = B[k * bks + n * bns] in shared memory
template <int Kd>
__device__ __forceinline__ void tile_mma(float (&acc)[3][4], const float* A, int ars, int acs,
                                         int m0, const float* B, int bks, int bns, int n0,
                                         int g, int t4, float ascale) {
#pragma unroll
  for (int k0 = 0; k0 < Kd; k0 += 8) {
    float a[4], b[2];
    a[0] = ascale * A[(m0 + g) * ars + (k0 + t4) * acs];
    a[1] = ascale * A[(m0 + g + 8) * ars + (k0 + t4) * acs];
    a[2] = ascale * A[(m0 + g) * ars + (k0 + t4 + 4) * acs];
    a[3] = ascale * A[(m0 + g + 8) * ars + (k0 + t4 + 4) * acs];
    b[0] = B[(k0 + t4) * bks + (n0 + g) * bns];
    b[1] = B[(k0 + t4 + 4) * bks + (n0 + g) * bns];
    mma_tf32x3(acc, a, b);
  }
}
// as tile_mma, with A and B scaled by ks[k] at their K index (KS) and B by
// ns[n] at its column (NS)
template <int Kd, bool KS, bool NS>
__device__ __forceinline__ void tile_mma_sc(float (&acc)[3][4], const float* A, int ars, int acs,
                                            int m0, const float* B, int bks, int bns, int n0,
                                            int g, int t4, float ascale, const float* ks,
                                            const float* ns) {
  const float nsv = NS ? ns[n0 + g] : 1.f;
#pragma unroll 4
  for (int k0 = 0; k0 < Kd; k0 += 8) {
    const float k1 = KS ? ks[k0 + t4] : 1.f, k2 = KS ? ks[k0 + t4 + 4] : 1.f;
    float a[4], b[2];
    a[0] = ascale * k1 * A[(m0 + g) * ars + (k0 + t4) * acs];
    a[1] = ascale * k1 * A[(m0 + g + 8) * ars + (k0 + t4) * acs];
    a[2] = ascale * k2 * A[(m0 + g) * ars + (k0 + t4 + 4) * acs];
    a[3] = ascale * k2 * A[(m0 + g + 8) * ars + (k0 + t4 + 4) * acs];
    b[0] = nsv * k1 * B[(k0 + t4) * bks + (n0 + g) * bns];
    b[1] = nsv * k2 * B[(k0 + t4 + 4) * bks + (n0 + g) * bns];
    mma_tf32x3(acc, a, b);
  }
}
// two products sharing B: acc1 += s1 A1 B and acc2 += s2 A2 B (A1, A2 row-major with
// row stride ars; B(k, n) = B[k * bks + n * bns]); B is split once per K step
template <int Kd>
__device__ __forceinline__ void tile_mma2(float (&acc1)[3][4], float (&acc2)[3][4],
                                          const float* A1, float s1, const float* A2, float s2,
                                          int ars, const float* B, int bks, int bns, int n0,
                                          int g, int t4) {
#pragma unroll
  for (int k0 = 0; k0 < Kd; k0 += 8) {
    uint32_t bh[2], bl[2];
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const float x = B[(k0 + t4 + 4 * q) * bks + (n0 + g) * bns];
      bh[q] = tf32_hi(x);
      bl[q] = tf32_lo(x, bh[q]);
    }
#pragma unroll
    for (int which = 0; which < 2; ++which) {
      const float* A = which ? A2 : A1;
      const float sc = which ? s2 : s1;
      uint32_t ah[4], al[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float x = sc * A[(g + 8 * (e & 1)) * ars + k0 + t4 + 4 * (e >> 1)];
        ah[e] = tf32_hi(x);
        al[e] = tf32_lo(x, ah[e]);
      }
      float (&acc)[3][4] = which ? acc2 : acc1;
      mma_tf32(acc[0], ah, bh);
      mma_tf32(acc[1], ah, bl);
      mma_tf32(acc[2], al, bh);
    }
  }
}
// Dm[rows, n0..n0+7] = egl[row] Dm + sum over the products p < NP of s_p A_p^T B_p, for
// every 16-row tile this warp owns (K = the 16 tokens; A_p(c, t) = A_p[t * CLD + c],
// B_p(t, n) = B_p[t * CLD + n]); the B fragments, the same for all of the warp's
// tiles, are split once
template <int D, int NP>
__device__ __forceinline__ void dd_update(float* Dm, int sld, const float* egl, int cld,
                                          const float* A1, float s1, const float* B1,
                                          const float* A2, float s2, const float* B2, int warp,
                                          int g, int t4) {
  constexpr int NT = D / 8;  // 8-column tiles per row of tiles
  const int n0 = (warp % NT) * 8;
  uint32_t bh[NP][2][2], bl[NP][2][2];
#pragma unroll
  for (int pp = 0; pp < NP; ++pp)
#pragma unroll
    for (int ks = 0; ks < 2; ++ks)
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const float x = (pp ? B2 : B1)[(ks * 8 + t4 + 4 * q) * cld + n0 + g];
        bh[pp][ks][q] = tf32_hi(x);
        bl[pp][ks][q] = tf32_lo(x, bh[pp][ks][q]);
      }
  for (int tile = warp; tile < (D / 16) * NT; tile += kBT / 32) {
    const int m0 = (tile / NT) * 16;
    float acc[3][4];
#pragma unroll
    for (int q = 0; q < 3; ++q)
#pragma unroll
      for (int r = 0; r < 4; ++r) acc[q][r] = 0.f;
#pragma unroll
    for (int pp = 0; pp < NP; ++pp)
#pragma unroll
      for (int ks = 0; ks < 2; ++ks) {
        const float* A = pp ? A2 : A1;
        const float sc = pp ? s2 : s1;
        uint32_t ah[4], al[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float x = sc * A[(ks * 8 + t4 + 4 * (e >> 1)) * cld + m0 + g + 8 * (e & 1)];
          ah[e] = tf32_hi(x);
          al[e] = tf32_lo(x, ah[e]);
        }
        const uint32_t bhh[2] = {bh[pp][ks][0], bh[pp][ks][1]};
        const uint32_t bll[2] = {bl[pp][ks][0], bl[pp][ks][1]};
        mma_tf32(acc[0], ah, bhh);
        mma_tf32(acc[1], ah, bll);
        mma_tf32(acc[2], al, bhh);
      }
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int r = m0 + g + 8 * (e >> 1), c = n0 + 2 * t4 + (e & 1);
      Dm[r * sld + c] = fmaf(egl[r], Dm[r * sld + c], acc[0][e] + acc[1][e] + acc[2][e]);
    }
  }
}
__device__ __forceinline__ void acc_zero(float (&acc)[3][4]) {
#pragma unroll
  for (int q = 0; q < 3; ++q)
#pragma unroll
    for (int r = 0; r < 4; ++r) acc[q][r] = 0.f;
}
// four consecutive float32 elements (one 16-byte load)
__device__ __forceinline__ float4 ld4f(const float* p) { return *reinterpret_cast<const float4*>(p); }
__device__ __forceinline__ void st4(float* p, const float4& v) {
  p[0] = v.x; p[1] = v.y; p[2] = v.z; p[3] = v.w;
}
// four consecutive elements as loaded (8-byte bf16 or 16-byte float vectors), and
// their float32 values; a load's result is only converted when it is stored, so no
// instruction waits on it in between
template <typename TIn> struct Raw4;
template <> struct Raw4<float> {
  using type = float4;
  using scalar = float;
};
template <> struct Raw4<__nv_bfloat16> {
  using type = uint2;
  using scalar = unsigned short;
};
__device__ __forceinline__ float4 ldraw4(const float* p) { return *reinterpret_cast<const float4*>(p); }
__device__ __forceinline__ uint2 ldraw4(const __nv_bfloat16* p) {
  return *reinterpret_cast<const uint2*>(p);
}
__device__ __forceinline__ float4 cvt4(const float4& v) { return v; }
__device__ __forceinline__ float4 cvt4(const uint2& u) {
  return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xffff0000u),
                     __uint_as_float(u.y << 16), __uint_as_float(u.y & 0xffff0000u));
}
__device__ __forceinline__ float ldraw1(const float* p) { return *p; }
__device__ __forceinline__ unsigned short ldraw1(const __nv_bfloat16* p) {
  return __bfloat16_as_ushort(*p);
}
__device__ __forceinline__ float cvt1(float v) { return v; }
__device__ __forceinline__ float cvt1(unsigned short v) { return __uint_as_float((uint32_t)v << 16); }

// 16-byte asynchronous global -> shared copies (completion waited with cp_async_wait)
__device__ __forceinline__ void cp_async16(float* dst, const float* src) {
  const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(dst));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(d), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group 0;" ::: "memory");
}

// element e of the C fragment: row g + 8 (e >> 1), column 2 t4 + (e & 1)
__device__ __forceinline__ float acc_sum(const float (&acc)[3][4], int e) {
  return acc[0][e] + acc[1][e] + acc[2][e];
}

template <int D, typename TIn>
__global__ void __launch_bounds__(kBT, 1) kda_bwd_kernel(const BwdParams<TIn> p) {
  using L = BwdLayout<D>;
  constexpr int CLD = L::CLD, SLD = L::SLD;
  extern __shared__ __align__(16) float sm[];
  float* S = sm + L::S;
  float* dS = sm + L::DS;
  float* Q = sm + L::Q;
  float* K = sm + L::K;
  float* G = sm + L::G;
  float* KB = sm + L::KB;
  float* QB = sm + L::QB;
  float* KH = sm + L::KH;
  float* X = sm + L::X;
  float* DO = sm + L::DO;
  float* U = sm + L::U;
  float* DU = sm + L::DU;
  float* Tm = sm + L::TM;
  float* Pm = sm + L::PM;
  float* Mm = sm + L::MM;
  float* dTm = sm + L::DT;
  float* dMm = sm + L::DM;
  float* Wm = Mm;  // dT T^T, once M is consumed
  float* scr = sm + L::SCR;
  float* scg = sm + L::SCG;
  float* sbeta = sm + L::BETA;
  float* sdb = sm + L::DB;
  float* gl = sm + L::GL;
  float* egl = sm + L::EGL;
  float* dgl = sm + L::DGL;
  int* s_wide = reinterpret_cast<int*>(sm + L::FLAG);
  float* dK = KH;   // aliases (see the layout)
  float* dQ = U;
  float* dG = DU;

  // a malformed cu_seqlens is latched by the validation before this kernel
  if (p.status && *(volatile const unsigned int*)p.status == (unsigned)KDA_ERR_BAD_SEQLENS) return;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g8 = lane >> 2, t4 = lane & 3;
  const int H = p.H;
  const int n = p.order ? p.order[blockIdx.x / H] : (int)(blockIdx.x / H);
  const int h = blockIdx.x % H;
  int64_t t0, len;
  p.seqs.get(n, t0, len);
  const int64_t nsub = (len + kBC - 1) / kBC;
  const int64_t row0 = p.sub_off ? p.sub_off[n] : (int64_t)n * ((p.seqs.T + kBC - 1) / kBC);
  // workspace row of sub-chunk s: its start state S [D][D], then X and U [16][D],
  // T and P [16][16], all written by the forward sweep
  constexpr int64_t RF = (int64_t)D * D + 2 * kBC * D + 2 * kBC * kBC;
  auto state_row = [&](int64_t s) { return p.states + ((row0 + s) * H + h) * RF; };
  const int64_t sbase = ((int64_t)n * H + h) * D * D;

  // the sub-chunk's inputs, four channels per thread: fetch issues the loads (raw),
  // stash converts and stores them once the buffers are free (rows past the
  // sequence end are zero).  The next sub-chunk's loads are issued before the
  // current step's last phase, so they land while it runs.
  using RawT = typename Raw4<TIn>::type;
  struct InFlight {
    RawT k, g, x;  // x: v (forward sweep) or q (backward sweep)
    float4 o;      // dout (backward sweep)
    typename Raw4<TIn>::scalar b;
  };
  constexpr int G4 = D / 4;
  auto fetch = [&](int64_t cs, int nv, bool bwd) {
    InFlight f;
    f.k = f.g = f.x = RawT{};
    f.o = make_float4(0.f, 0.f, 0.f, 0.f);
    f.b = 0;
    const int t = tid / G4, c = (tid % G4) * 4;
    if (tid < kBC * G4 && t < nv) {
      const int64_t go = ((t0 + cs + t) * H + h) * D + c;
      f.k = ldraw4(p.k + go);
      f.g = ldraw4(p.g + go);
      if (bwd) {
        f.x = ldraw4(p.q + go);
        f.o = *reinterpret_cast<const float4*>(p.dout + go);
      } else {
        f.x = ldraw4(p.v + go);
      }
    }
    if (tid < nv && tid < kBC) f.b = ldraw1(p.beta + (t0 + cs + tid) * H + h);
    return f;
  };
  auto stash = [&](const InFlight& f, bool bwd) {
    if (tid < kBC * G4) {
      const int t = tid / G4, c = (tid % G4) * 4;
      st4(K + t * CLD + c, cvt4(f.k));
      st4(G + t * CLD + c, cvt4(f.g));
      if (bwd) {
        st4(Q + t * CLD + c, cvt4(f.x));
        st4(DO + t * CLD + c, f.o);
      } else {
        st4(X + t * CLD + c, cvt4(f.x));  // the backward sweep reads X itself
      }
    }
    if (tid < kBC) {
      sbeta[tid] = cvt1(f.b);
      sdb[tid] = 0.f;
    }
  };
  // a D x D state between global memory (dense) and shared memory (row stride SLD),
  // 16 bytes per access, all loads issued before the stores
  auto state_in = [&](float* dst, const float* src) {
    constexpr int NV = D * D / 4 / kBT;
    float4 r[NV];
#pragma unroll
    for (int m = 0; m < NV; ++m) r[m] = src ? ld4f(src + 4 * (tid + m * kBT)) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int m = 0; m < NV; ++m) {
      const int i = 4 * (tid + m * kBT);
      *reinterpret_cast<float4*>(dst + (i / D) * SLD + i % D) = r[m];
    }
  };
  // the forward sweep's X, U, T and P of a sub-chunk, after its state in the row
  auto row_out = [&](float* row) {
    float* xr = row + D * D;
    float* ur = xr + kBC * D;
    float* tr = ur + kBC * D;
    float* pr = tr + kBC * kBC;
    for (int i = 4 * tid; i < kBC * D; i += 4 * kBT) {
      const int o = (i / D) * CLD + i % D;
      *reinterpret_cast<float4*>(xr + i) = *reinterpret_cast<const float4*>(X + o);
      *reinterpret_cast<float4*>(ur + i) = *reinterpret_cast<const float4*>(U + o);
    }
    if (tid < kBC * kBC) {
      tr[tid] = Tm[(tid >> 4) * kSL + (tid & 15)];
      pr[tid] = Pm[(tid >> 4) * kSL + (tid & 15)];
    }
  };
  // the backward sweep's start: S (unless it is already on its way, see below), X,
  // U, T and P of sub-chunk s, every load issued before the first store
  auto row_in = [&](const float* row, bool with_s) {
    constexpr int NV = D * D / 4 / kBT;
    constexpr int NX = kBC * D / 4;  // float4 per 16 x D matrix
    float4 r[NV], rx = make_float4(0.f, 0.f, 0.f, 0.f), ru = rx;
    float vt = 0.f, vp = 0.f;
#pragma unroll
    for (int m = 0; m < NV; ++m)
      r[m] = with_s ? ld4f(row + 4 * (tid + m * kBT)) : make_float4(0.f, 0.f, 0.f, 0.f);
    if (tid < NX) {
      rx = ld4f(row + D * D + 4 * tid);
      ru = ld4f(row + D * D + kBC * D + 4 * tid);
    }
    if (tid < kBC * kBC) {
      vt = row[D * D + 2 * kBC * D + tid];
      vp = row[D * D + 2 * kBC * D + kBC * kBC + tid];
    }
    if (with_s) {
#pragma unroll
      for (int m = 0; m < NV; ++m) {
        const int i = 4 * (tid + m * kBT);
        *reinterpret_cast<float4*>(S + (i / D) * SLD + i % D) = r[m];
      }
    } else {
      cp_async_wait();  // this thread's part of S, requested during the previous step
    }
    if (tid < NX) {
      const int i = 4 * tid, o = (i / D) * CLD + i % D;
      *reinterpret_cast<float4*>(X + o) = rx;
      *reinterpret_cast<float4*>(U + o) = ru;
    }
    if (tid < kBC * kBC) {
      Tm[(tid >> 4) * kSL + (tid & 15)] = vt;
      Pm[(tid >> 4) * kSL + (tid & 15)] = vp;
    }
  };
  // the next (earlier) sub-chunk's state into S once this step is done with it
  auto s_prefetch = [&](const float* row) {
#pragma unroll
    for (int m = 0; m < D * D / 4 / kBT; ++m) {
      const int i = 4 * (tid + m * kBT);
      cp_async16(S + (i / D) * SLD + i % D, row + i);
    }
    cp_async_commit();
  };
  auto state_out = [&](float* dst, const float* src) {
#pragma unroll 4
    for (int m = 0; m < D * D / 4 / kBT; ++m) {
      const int i = 4 * (tid + m * kBT);
      *reinterpret_cast<float4*>(dst + i) = *reinterpret_cast<const float4*>(src + (i / D) * SLD + i % D);
    }
  };

  bool split = true;  // the pairwise factors of this sub-chunk are split (see prepare)
  // Gam (kept as Gam log2 e, so every factor is one ex2) and the decayed operands;
  // forward sweep: P, T, X = V - Kb S and U = T diag(beta) X; backward sweep: M
  // (P, T, X and U come back from the forward sweep's workspace row)
  auto prepare = [&](bool bwd) {
    if (tid == 0) *s_wide = 0;
    __syncthreads();
    if (tid < D) {
      float run = 0.f;
#pragma unroll
      for (int t = 0; t < kBC; ++t) {
        run += G[t * CLD + tid];
        G[t * CLD + tid] = run * kLog2e;
      }
      gl[tid] = run * kLog2e;
      egl[tid] = ex2(run * kLog2e);
      // e^(Gam_i - Gam_j) = e^(Gam_i - h) e^(h - Gam_j), h = Gl / 2; where some
      // factor would pass 2^86 the sub-chunk takes the explicit form instead
      const float h2 = 0.5f * run * kLog2e;
      bool ok = true;
#pragma unroll
      for (int t = 0; t < kBC; ++t) ok = ok && fabsf(G[t * CLD + tid] - h2) <= 86.f;
      if (!ok) atomicOr(s_wide, 1);
    }
    __syncthreads();
    split = *(volatile int*)s_wide == 0;
    for (int i = tid; i < kBC * D; i += kBT) {
      const int t = i / D, c = i % D, o = t * CLD + c;
      const float gm = G[o], e = ex2(gm);
      KB[o] = K[o] * e;
      if (bwd) QB[o] = Q[o] * e;
      KH[o] = K[o] * ex2(gl[c] - gm);
    }
    __syncthreads();  // the split products below read Kb, Qb and Kh
    float* Pt = bwd ? Mm : Pm;  // the pairwise matrix this sweep forms
    if (split) {
      // P = (K a)(K b)^T or M = (Q a)(K b)^T, with the factors a = e^(Gam - h),
      // b = e^(h - Gam) formed directly (not from Kb, which may have underflowed);
      // each of the first nw * parts warps takes one 8-column tile over a slice of
      // the channels, and the partial tiles meet in a 16 x D buffer that is free at
      // this point (parts is bounded by that buffer: 8 at D = 128, 4 at D = 64)
      constexpr int nw = 2;
      constexpr int parts = L::CM / (nw * 128) < 8 ? L::CM / (nw * 128) : 8;
      static_assert(nw * parts * 128 <= L::CM && D % (8 * parts) == 0, "partial tiles");
      const bool isM = bwd;
      float* part = bwd ? DU : U;
      if (warp < nw * parts) {
        const float* A = isM ? Q : K;
        const int n0 = (warp % nw) * 8, kc = D / parts, kb = (warp / nw) * kc;
        float acc[3][4];
        acc_zero(acc);
#pragma unroll 2
        for (int k0 = kb; k0 < kb + kc; k0 += 8) {
          float a[4], b[2];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int c = k0 + t4 + 4 * (e >> 1), o = (g8 + 8 * (e & 1)) * CLD + c;
            a[e] = A[o] * ex2(G[o] - 0.5f * gl[c]);
          }
#pragma unroll
          for (int q2 = 0; q2 < 2; ++q2) {
            const int c = k0 + t4 + 4 * q2, o = (n0 + g8) * CLD + c;
            b[q2] = K[o] * ex2(0.5f * gl[c] - G[o]);
          }
          mma_tf32x3(acc, a, b);
        }
#pragma unroll
        for (int e = 0; e < 4; ++e)
          part[warp * 128 + (g8 + 8 * (e >> 1)) * 8 + 2 * t4 + (e & 1)] = acc_sum(acc, e);
      }
      __syncthreads();
      {
        if (tid < nw * 128) {
          const int cb = tid >> 7, w = tid & 127, r = w >> 3, c = cb * 8 + (w & 7);
          float v = 0.f;
#pragma unroll
          for (int pp = 0; pp < parts; ++pp) v += part[(pp * nw + cb) * 128 + w];
          Pt[r * kSL + c] = (isM ? c <= r : c < r) ? v : 0.f;
        }
      }
    } else if (tid < 256) {  // explicit differences: P (j < i) or M (j <= i)
      const int pi = tid >> 4, pj = tid & 15;
      const bool isM = bwd;
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
      if (isM ? pj <= pi : pj < pi) {
        const float* A = isM ? Q : K;
#pragma unroll 4
        for (int cc = 0; cc < D; ++cc) {
          const int c = (cc + lane) & (D - 1);  // rotated so the lanes hit distinct banks
          acc[cc & 3] = fmaf(A[pi * CLD + c] * K[pj * CLD + c],
                             ex2(G[pi * CLD + c] - G[pj * CLD + c]), acc[cc & 3]);
        }
      }
      Pt[pi * kSL + pj] = (acc[0] + acc[1]) + (acc[2] + acc[3]);
    }
    __syncthreads();
    if (bwd) return;
    if (warp == 0 && lane < kBC) {  // T = (I + diag(beta) P)^-1, column jj per lane
      const int jj = lane;
      float x[kBC];
#pragma unroll
      for (int m = 0; m < kBC; ++m) {
        float vv = m == jj ? 1.f : 0.f;
#pragma unroll
        for (int l = 0; l < m; ++l)
          if (l >= jj) vv = fmaf(-sbeta[m] * Pm[m * kSL + l], x[l], vv);
        x[m] = m < jj ? 0.f : vv;
      }
      // T, and T diag(beta) for U below (M is the backward sweep's; free here)
      const float bj = sbeta[jj];
#pragma unroll
      for (int m = 0; m < kBC; ++m) {
        Tm[m * kSL + jj] = x[m];
        Mm[m * kSL + jj] = x[m] * bj;
      }
    }
    // X = V - Kb S (one n-tile of 8 columns per warp)
    for (int nt = warp; nt < D / 8; nt += kBT / 32) {
      float acc[3][4];
      acc_zero(acc);
      tile_mma<D>(acc, KB, CLD, 1, 0, S, SLD, 1, nt * 8, g8, t4, 1.f);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int r = g8 + 8 * (e >> 1), c = nt * 8 + 2 * t4 + (e & 1);
        X[r * CLD + c] -= acc_sum(acc, e);
      }
    }
    __syncthreads();
    // U = (T diag(beta)) X (one n-tile of 8 columns per warp; T is lower triangular)
    for (int nt = warp; nt < D / 8; nt += kBT / 32) {
      float acc[3][4];
      acc_zero(acc);
      tile_mma<kBC>(acc, Mm, kSL, 1, 0, X, CLD, 1, nt * 8, g8, t4, 1.f);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int r = g8 + 8 * (e >> 1), c = nt * 8 + 2 * t4 + (e & 1);
        U[r * CLD + c] = acc_sum(acc, e);
      }
    }
    __syncthreads();
  };

  // ---- 1. forward sweep: the start state of every sub-chunk
  state_in(S, p.h0 ? p.h0 + sbase : nullptr);
  __syncthreads();
  auto nv_of = [&](int64_t s) { return (int)(len - s * kBC < kBC ? len - s * kBC : kBC); };
  InFlight nxt = fetch(0, nsub > 0 ? nv_of(0) : 0, false);
  for (int64_t s = 0; s < nsub; ++s) {
    const int64_t cs = s * kBC;
    state_out(state_row(s), S);
    stash(nxt, false);
    __syncthreads();
    prepare(false);
    row_out(state_row(s));
    if (s + 1 < nsub) nxt = fetch(cs + kBC, nv_of(s + 1), false);
    // S <- diag(e^Gl) S + Kh^T U
    dd_update<D, 1>(S, SLD, egl, CLD, KH, 1.f, U, nullptr, 0.f, nullptr, warp, g8, t4);
    __syncthreads();
  }

  // ---- 2. backward sweep
  state_in(dS, p.dhT ? p.dhT + sbase : nullptr);
  if (nsub > 0) nxt = fetch((nsub - 1) * kBC, nv_of(nsub - 1), true);
  for (int64_t s = nsub - 1; s >= 0; --s) {
    const int64_t cs = s * kBC;
    const int nv = nv_of(s);
    row_in(state_row(s), s == nsub - 1);
    stash(nxt, true);
    __syncthreads();
    prepare(true);

    // dU = scale M^T dO + Kh dS
    for (int nt = warp; nt < D / 8; nt += kBT / 32) {
      float acc[3][4];
      acc_zero(acc);
      tile_mma<kBC>(acc, Mm, 1, kSL, 0, DO, CLD, 1, nt * 8, g8, t4, p.scale);
      tile_mma<D>(acc, KH, CLD, 1, 0, dS, SLD, 1, nt * 8, g8, t4, 1.f);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int r = g8 + 8 * (e >> 1), c = nt * 8 + 2 * t4 + (e & 1);
        DU[r * CLD + c] = acc_sum(acc, e);
      }
    }
    // dGl from the decay of the start state: e^Gl rowsum(dS . S); warp w takes rows
    // 8 w .. 8 w + 7 (D / 16 at D = 64), a lane four consecutive columns of each
    {
      float v[D / 16];
#pragma unroll
      for (int r = 0; r < D / 16; ++r) {  // the rows' loads and sums interleave
        const int c = warp * (D / 16) + r;
        v[r] = 0.f;
        if (4 * lane < D) {
          const float4 a = *reinterpret_cast<const float4*>(dS + c * SLD + 4 * lane);
          const float4 b = *reinterpret_cast<const float4*>(S + c * SLD + 4 * lane);
          v[r] = fmaf(a.x, b.x, fmaf(a.y, b.y, fmaf(a.z, b.z, a.w * b.w)));
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1)
#pragma unroll
        for (int r = 0; r < D / 16; ++r) v[r] += __shfl_xor_sync(0xffffffffu, v[r], o);
      if (lane < D / 16) {
        float w = v[0];
#pragma unroll
        for (int r = 1; r < D / 16; ++r) w = lane == r ? v[r] : w;
        scg[warp * (D / 16) + lane] = w;
      }
    }
    __syncthreads();
    // dT = dU (diag(beta) X)^T, dM = scale dO U^T (lower): warps 0..7 each take one
    // (matrix, 8-column tile) over half of the value channels
    if (warp < 8) {
      const int cb = warp & 3, kb = (warp >> 2) * (D / 2);
      const bool isM = cb >= 2;
      const int n0 = (cb & 1) * 8;
      float acc[3][4];
      acc_zero(acc);
      if (isM)
        tile_mma_sc<D / 2, false, false>(acc, DO + kb, CLD, 1, 0, U + kb, 1, CLD, n0, g8, t4,
                                         p.scale, nullptr, nullptr);
      else
        tile_mma_sc<D / 2, false, true>(acc, DU + kb, CLD, 1, 0, X + kb, 1, CLD, n0, g8, t4, 1.f,
                                        nullptr, sbeta);
#pragma unroll
      for (int e = 0; e < 4; ++e)
        scr[warp * 128 + (g8 + 8 * (e >> 1)) * 8 + 2 * t4 + (e & 1)] = acc_sum(acc, e);
    }
    __syncthreads();
    {  // the two halves of dT and dM; dGl's first term
      const int cb = tid >> 7, w = tid & 127, r = w >> 3, c = (cb & 1) * 8 + (w & 7);
      const float v = scr[cb * 128 + w] + scr[(4 + cb) * 128 + w];
      const bool isM = cb >= 2;
      (isM ? dMm : dTm)[r * kSL + c] = (!isM || c <= r) ? v : 0.f;
    }
    if (tid < D) dgl[tid] = egl[tid] * scg[tid];
    __syncthreads();  // the scratch area is read: the dY tiles' row sums take it
    // dY = T^T dU (one n-tile of 8 columns per warp; T is lower triangular);
    // dbeta += rowsum(dY . X), each tile's part to the scratch area and summed in a
    // fixed order below (so that dbeta does not depend on the warps' timing);
    // dX = diag(beta) dY in place of X (each thread reads and writes only its own
    // elements of X)
    for (int nt = warp; nt < D / 8; nt += kBT / 32) {
      float acc[3][4];
      acc_zero(acc);
      tile_mma<kBC>(acc, Tm, 1, kSL, 0, DU, CLD, 1, nt * 8, g8, t4, 1.f);
      float part[2] = {0.f, 0.f};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int r = g8 + 8 * (e >> 1), c = nt * 8 + 2 * t4 + (e & 1);
        const float dy = acc_sum(acc, e);
        part[e >> 1] = fmaf(dy, X[r * CLD + c], part[e >> 1]);
        const float dx = sbeta[r] * dy;
        X[r * CLD + c] = dx;
        if (r < nv) p.dv[((t0 + cs + r) * H + h) * D + c] = dx;
      }
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {  // the row's 8 columns of this tile: lanes t4 = 0..3
        part[hh] += __shfl_xor_sync(0xffffffffu, part[hh], 1);
        part[hh] += __shfl_xor_sync(0xffffffffu, part[hh], 2);
        if (t4 == 0) scr[nt * kBC + g8 + 8 * hh] = part[hh];
      }
    }
    __syncthreads();  // dU is consumed: dG may take its buffer; dT and dM are complete
    // W = dT T^T (threads 0..255; M is consumed, so W takes its place); threads
    // 256 .. 256 + 15 add the dY tiles' row sums to dbeta in tile order
    if (tid >= 256 && tid < 256 + kBC) {
      const int r = tid - 256;
      float a = 0.f;
#pragma unroll
      for (int nt = 0; nt < D / 8; ++nt) a += scr[nt * kBC + r];
      sdb[r] += a;
    }
    if (tid < 256) {
      const int wi = tid >> 4, wj = tid & 15;
      float acc = 0.f;
#pragma unroll
      for (int l = 0; l < kBC; ++l)
        if (l <= wj) acc = fmaf(dTm[wi * kSL + l], Tm[wj * kSL + l], acc);
      Wm[wi * kSL + wj] = acc;
    }
    // dKh = U dS^T: dk = dKh e^(Gl - Gam); dGam = -Kh dKh; dGl += colsum(Kh dKh)
    for (int nt = warp; nt < D / 8; nt += kBT / 32) {
      float acc[3][4];
      acc_zero(acc);
      tile_mma<D>(acc, U, CLD, 1, 0, dS, 1, SLD, nt * 8, g8, t4, 1.f);
      float col[2] = {0.f, 0.f};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int r = g8 + 8 * (e >> 1), c = nt * 8 + 2 * t4 + (e & 1), o = r * CLD + c;
        const float d = acc_sum(acc, e), kh = KH[o];
        col[e & 1] = fmaf(kh, d, col[e & 1]);
        dG[o] = -kh * d;
        dK[o] = d * ex2(gl[c] - G[o]);
      }
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) {
        col[0] += __shfl_xor_sync(0xffffffffu, col[0], o);
        col[1] += __shfl_xor_sync(0xffffffffu, col[1], o);
      }
      if (g8 == 0) {
        dgl[nt * 8 + 2 * t4] += col[0];
        dgl[nt * 8 + 2 * t4 + 1] += col[1];
      }
    }
    __syncthreads();
    // dA = -T^T W, strictly lower; dbeta_i += sum_j dA_ij P_ij; dP = diag(beta) dA
    if (tid < 256) {
      const int ai = tid >> 4, aj = tid & 15;
      float acc = 0.f;
      if (aj < ai) {
#pragma unroll
        for (int m = 0; m < kBC; ++m)
          if (m >= ai) acc = fmaf(-Tm[m * kSL + ai], Wm[m * kSL + aj], acc);
      }
      float part = acc * Pm[ai * kSL + aj];
#pragma unroll
      for (int o = 8; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
      if ((tid & 15) == 0) sdb[ai] += part;  // one thread per row
      dTm[ai * kSL + aj] = sbeta[ai] * acc;  // dP (dT is consumed by W)
    }
    // dQb = scale dO S^T: dq = dQb e^Gam; dGam += Qb dQb   (U is consumed: dq takes it)
    // dKb = -dX S^T: dk += dKb e^Gam; dGam += Kb dKb   (one pass: both read S^T)
    for (int nt = warp; nt < D / 8; nt += kBT / 32) {
      float aq[3][4], ak[3][4];
      acc_zero(aq);
      acc_zero(ak);
      tile_mma2<D>(aq, ak, DO, p.scale, X, -1.f, CLD, S, 1, SLD, nt * 8, g8, t4);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int r = g8 + 8 * (e >> 1), c = nt * 8 + 2 * t4 + (e & 1), o = r * CLD + c;
        const float dqb = acc_sum(aq, e), dkb = acc_sum(ak, e), eg = ex2(G[o]);
        dQ[o] = dqb * eg;
        dK[o] = fmaf(dkb, eg, dK[o]);
        dG[o] = fmaf(QB[o], dqb, fmaf(KB[o], dkb, dG[o]));
      }
    }
    __syncthreads();
    if (s > 0) s_prefetch(state_row(s - 1));  // S is not read again in this step
    // pairwise factors, per (token t, channel c):
    //   RK = sum_{j<t} dP_tj K_jc E_tj, RQ = sum_{j<=t} dM_tj K_jc E_tj,
    //   CK = sum_{i>t} dP_it K_ic E_it, CQ = sum_{i>=t} dM_it Q_ic E_it,
    //   E_ij = e^(Gam_ic - Gam_jc);  dq += RQ, dk += RK + CK + CQ,
    //   dGam += K RK + Q RQ - K CK - K CQ
    // Split (E_ij = a_i b_j, a = e^(Gam - h), b = e^(h - Gam)): RK = a (dP (K b)),
    // RQ = a (dM (K b)), CK = b (dP^T (K a)), CQ = b (dM^T (Q a)), the factors formed
    // from Gam directly; dP and dM are zero outside their triangles.
    if (split) {
      for (int nt = warp; nt < D / 8; nt += kBT / 32) {
        const int n0 = nt * 8;
        float rk[3][4], rq[3][4], ck[3][4], cq[3][4];
        acc_zero(rk);
        acc_zero(rq);
        acc_zero(ck);
        acc_zero(cq);
        const float hb = 0.5f * gl[n0 + g8];
#pragma unroll
        for (int k0 = 0; k0 < kBC; k0 += 8) {
          float kb[2], ka[2], qa[2], ap[4], am[4], apt[4], amt[4];
#pragma unroll
          for (int q2 = 0; q2 < 2; ++q2) {
            const int o = (k0 + t4 + 4 * q2) * CLD + n0 + g8;
            const float x = G[o] - hb;
            kb[q2] = K[o] * ex2(-x);
            ka[q2] = K[o] * ex2(x);
            qa[q2] = Q[o] * ex2(x);
          }
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int r = g8 + 8 * (e & 1), k = k0 + t4 + 4 * (e >> 1);
            ap[e] = dTm[r * kSL + k];
            am[e] = dMm[r * kSL + k];
            apt[e] = dTm[k * kSL + r];
            amt[e] = dMm[k * kSL + r];
          }
          mma_tf32x3(rk, ap, kb);
          mma_tf32x3(rq, am, kb);
          mma_tf32x3(ck, apt, ka);
          mma_tf32x3(cq, amt, qa);
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int t = g8 + 8 * (e >> 1), c = n0 + 2 * t4 + (e & 1), o = t * CLD + c;
          const float h2 = 0.5f * gl[c];
          const float a = ex2(G[o] - h2), b = ex2(h2 - G[o]);
          const float vrk = a * acc_sum(rk, e), vrq = a * acc_sum(rq, e);
          const float vck = b * acc_sum(ck, e), vcq = b * acc_sum(cq, e);
          const float kt = K[o];
          dQ[o] += vrq;
          dK[o] += vrk + vck + vcq;
          dG[o] += kt * (vrk - vck - vcq) + Q[o] * vrq;
        }
      }
    } else
    for (int i = tid; i < kBC * D; i += kBT) {
      const int t = i / D, c = i % D, o = t * CLD + c;
      const float gt = G[o], kt = K[o], qt = Q[o];
      float rk = 0.f, rq = 0.f, ck = 0.f, cq = 0.f;
#pragma unroll
      for (int j = 0; j < kBC; ++j) {
        const int oj = j * CLD + c;
        if (j <= t) {
          const float e = ex2(gt - G[oj]) * K[oj];
          rq = fmaf(dMm[t * kSL + j], e, rq);
          if (j < t) rk = fmaf(dTm[t * kSL + j], e, rk);
        }
        if (j >= t) {
          const float e = ex2(G[oj] - gt);
          cq = fmaf(dMm[j * kSL + t] * Q[oj], e, cq);
          if (j > t) ck = fmaf(dTm[j * kSL + t] * K[oj], e, ck);
        }
      }
      dQ[o] += rq;
      dK[o] += rk + ck + cq;
      dG[o] += kt * (rk - ck - cq) + qt * rq;
    }
    __syncthreads();
    // outputs of the sub-chunk; dS <- diag(e^Gl) dS + scale Qb^T dO - Kb^T dX
    for (int i = tid; i < kBC * D; i += kBT) {
      const int t = i / D, c = i % D;
      if (t < nv) {
        const int64_t go = ((t0 + cs + t) * H + h) * D + c;
        p.dq[go] = dQ[t * CLD + c];
        p.dk[go] = dK[t * CLD + c];
      }
    }
    if (tid < D) {  // dg: reverse prefix sum of dGam, dGl entering at the last row
      float run = dgl[tid];
#pragma unroll
      for (int t = kBC - 1; t >= 0; --t) {
        run += dG[t * CLD + tid];
        if (t < nv) p.dg[((t0 + cs + t) * H + h) * D + tid] = run;
      }
    }
    if (tid < nv) p.dbeta[(t0 + cs + tid) * H + h] = sdb[tid];
    if (s > 0) nxt = fetch(cs - kBC, nv_of(s - 1), true);
    dd_update<D, 2>(dS, SLD, egl, CLD, QB, p.scale, DO, KB, -1.f, X, warp, g8, t4);
    __syncthreads();
  }
  if (p.dh0) state_out(p.dh0 + sbase, dS);
}

// first state row of each packed sequence: exclusive prefix sum of
// ceil(len / 16), one block of 1024 threads stepping through the sequences
__global__ void __launch_bounds__(1024) kda_bwd_offsets(const int32_t* cu, int N, int64_t T,
                                                        int64_t* off) {
  __shared__ int64_t warp_tot[32];
  __shared__ int64_t carry;
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  if (tid == 0) carry = 0;
  __syncthreads();
  const SeqView sv{cu, T};
  for (int base = 0; base < N; base += 1024) {
    const int n = base + tid;
    int64_t x = 0;
    if (n < N) {
      int64_t a, l;
      sv.get(n, a, l);
      x = (l + kBC - 1) / kBC;
    }
    int64_t incl = x;  // inclusive scan within the warp
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int64_t y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane == 31) warp_tot[w] = incl;
    __syncthreads();
    if (w == 0) {
      int64_t wt = warp_tot[lane];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int64_t y = __shfl_up_sync(0xffffffffu, wt, o);
        if (lane >= o) wt += y;
      }
      warp_tot[lane] = wt;  // inclusive over warps
    }
    __syncthreads();
    const int64_t before = carry + (w > 0 ? warp_tot[w - 1] : 0);
    if (n < N) off[n] = before + incl - x;
    __syncthreads();
    if (tid == 1023) carry = before + incl;
    __syncthreads();
  }
}

template <int D, typename TIn>
cudaError_t launch_bwd_t(const BwdArgs& a) {
  using L = BwdLayout<D>;
  BwdParams<TIn> p;
  p.q = static_cast<const TIn*>(a.q);
  p.k = static_cast<const TIn*>(a.k);
  p.v = static_cast<const TIn*>(a.v);
  p.g = static_cast<const TIn*>(a.g);
  p.beta = static_cast<const TIn*>(a.beta);
  p.dout = a.dout;
  p.dhT = a.dhT;
  p.h0 = a.h0;
  p.seqs = SeqView{a.cu, a.T};
  p.order = a.order;
  p.sub_off = a.sub_off;
  p.H = a.H;
  p.scale = a.scale;
  p.dq = a.dq;
  p.dk = a.dk;
  p.dv = a.dv;
  p.dg = a.dg;
  p.dbeta = a.dbeta;
  p.dh0 = a.dh0;
  p.states = a.states;
  p.status = a.status;
  auto kern = kda_bwd_kernel<D, TIn>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)L::BYTES);
  if (e != cudaSuccess) return e;
  kern<<<(unsigned)((int64_t)a.N * a.H), kBT, L::BYTES, a.stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

size_t bwd_state_rows(bool packed, int64_t N, int64_t T) {
  return packed ? (size_t)((T + kBC - 1) / kBC + N) : (size_t)(N * ((T + kBC - 1) / kBC));
}

cudaError_t launch_bwd_offsets(const BwdArgs& a, int64_t* off) {
  if (a.N == 0) return cudaSuccess;
  kda_bwd_offsets<<<1, 1024, 0, a.stream>>>(a.cu, a.N, a.T, off);
  return cudaGetLastError();
}

cudaError_t launch_backward(const BwdArgs& a) {
  if ((int64_t)a.N * a.H == 0) return cudaSuccess;
  if (a.bf16)
    return a.D == 128 ? launch_bwd_t<128, __nv_bfloat16>(a) : launch_bwd_t<64, __nv_bfloat16>(a);
  return a.D == 128 ? launch_bwd_t<128, float>(a) : launch_bwd_t<64, float>(a);
}

}  // namespace kda
