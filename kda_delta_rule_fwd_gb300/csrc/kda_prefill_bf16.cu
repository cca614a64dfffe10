// KDA chunkwise prefill, bf16 inputs, on the sm_100-family tensor cores.
//
// Chunkwise form of the recurrence ("Kimi K3 技术报告摘要", section 1, 训练策略
// table, KDA row: parallel inside a chunk, recurrent across chunks; the
// transition (I - beta k k^T) diag(alpha) is diagonal-plus-low-rank: "Kimi K3
// NPU Training", section NPU 算子支持度, DPLR chunk kernel).  Per chunk of 64
// tokens with Gam = inclusive per-channel prefix sum of g and a per-channel
// reference c = 2^round(log2 e * Gam at token 31) (mid chunk, a power of two):
//
//   R_K = K e^Gam / c,  R_Q = Q e^Gam / c,  Ck = K c e^-Gam   (c cancels in R Ck^T)
//   [Akk; Aqk] = [R_K; R_Q] Ck^T
//   T   = (I + strict_lower(diag(beta) Akk))^-1  (forward substitution)
//   S'  = diag(c) S                              (exact: c is a power of two)
//   X'  = R_K S' - V   (= (K e^Gam) S - V)       U  = (-T diag(beta)) X' 
//   O   = scale (R_Q S' + lower(Aqk) U)          (R_Q S' = (Q e^Gam) S)
//   S  <- diag(e^Gam_last / c) (S' + Ck^T U)     (= diag(e^Gam_last) S + (K e^(Gam_last-Gam))^T U)
//
// The products with S' need nothing from the substitution, so they run on the
// tensor cores while the CUDA cores solve for T.
//
// Every product runs on tcgen05 with M = 128 and float32 accumulators in
// tensor memory.  The state products are taken transposed (rows = value
// channel) so that S^T lives in TMEM as the accumulator and as the A operand.
// Operands on the output path are split into bf16 hi + lo parts (x = hi + lo,
// products hi*hi + hi*lo + lo*hi), which keeps every product near float32
// accuracy: a single bf16 rounding of an operand on the dominant path
// already exceeds a 1e-2 max-error budget on heavy-tailed outputs.
//
// One CTA (512 threads) owns one (sequence, head) chain and walks its chunks
// in order; the inputs of chunk n+1 are fetched by TMA while chunk n's state
// update runs.  During the substitution (warps 0-7) warps 8-15 split X'.  Each
// mbarrier wait is bounded: on expiry the CTA latches KDA_ERR_DEVICE_TIMEOUT,
// drains its in-flight copies, frees TMEM and exits.
#include <cudaTypedefs.h>

#include <mutex>

#include "kda_prefill_common.cuh"

namespace kda {
namespace {

using namespace sm100;
using namespace pf;

constexpr int C = 64;            // chunk length (tokens)
constexpr int D = 128;           // head dim (dk == dv)
constexpr int kThreads = 512;
constexpr int NCOL = kThreads / 128;  // threads sharing one accumulator row (column slices)
constexpr int TCOL = 64 / NCOL;       // columns of a 64-wide accumulator per thread
constexpr int SCOL = 128 / NCOL;      // state columns per thread
constexpr int GPT = 16 / (2 * NCOL);  // 8-channel groups per thread in the elementwise passes
static_assert(TCOL == 16 && SCOL % 16 == 0 && GPT >= 1, "thread mapping");
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kMaxExp2 = 115.f;  // |log2 of a decay factor| beyond this: the exact token path
constexpr float kRefExp2 = 100.f;  // |log2 c| is clamped here (S' and its bf16 parts stay normal)

// ---- shared memory map (bytes) --------------------------------------------
constexpr uint32_t SM_IN_Q = 0;          // q, k tiles: two 64-channel halves, 128-byte swizzle
constexpr uint32_t SM_IN_K = 16384;      // (see off_sw128)
constexpr uint32_t SM_NRM = 32768;       // pass A: q/k sums of squares (fused normalisation)
constexpr uint32_t SM_GB = 40960;        // g tile, tokens 32..63: [group][32 tokens][8] bf16
constexpr uint32_t SM_IN_V = 49152;      // v and g tiles: [8-channel group][token][8] bf16
// forward-substitution scratch, over the q and k tiles once pass A has read them
constexpr uint32_t SV_AT = 0, SV_T32 = 17408, SV_M32 = 34304;
constexpr int ALD = 68;  // row stride of A^T (float): fragment loads hit distinct banks
constexpr int TLD = 66;  // row stride of T (float): 8-byte rows, few bank conflicts
static_assert(SV_M32 + 4 * 256 * 4 <= SM_GB, "substitution scratch overlaps the g tile");
constexpr uint32_t SM_X = 65536;         // 96 KB: [R_K; R_Q] hi, lo (K-major), Ck hi, lo
constexpr uint32_t X_R_HI = 0, X_R_LO = 32768, X_CK_HI = 65536, X_CK_LO = 81920;
constexpr uint32_t X_OUT = 0;  // output staging for the bulk store, [64 tokens][128] (32 KB)
constexpr uint32_t X_ALPHA = 32768;  // token path: alpha [64 tokens][128] float32
constexpr uint32_t SM_Y = 163840;        // 32 KB
constexpr uint32_t Y_TB_HI = 0, Y_TB_LO = 8192, Y_AQK_HI = 16384, Y_AQK_LO = 24576;
// token path scratch over the Aqk parts (rewritten in full by every tensor-core chunk)
constexpr uint32_t Y_RED = 16384, Y_KQ = 16384 + 8192;
constexpr uint32_t SM_LL = 196608;       // [L; L] 128 x 64 bf16 (lower-triangular ones)
constexpr uint32_t SM_MISC = 212992;
constexpr uint32_t MISC_PEND = 0, MISC_GL = 512, MISC_C = 1024, MISC_NRHO = 1536, MISC_GAMC = 2048,
                   MISC_BETA = 2560, MISC_BAR = 2816, MISC_TMEM = 2848, MISC_FLAG = 2852,
                   MISC_P12BAR = 2864;
// (MISC_FLAG + 4: the current work item, broadcast by thread 0; MISC_P12BAR: the
// output and state products, issued by two threads, each committing once)
constexpr uint32_t SM_NEGI = 216064;     // -I (64 x 64 bf16, K-major): adds -V^T on the tensor core
constexpr uint32_t SM_GA = SM_NEGI + 8192;  // g tile, tokens 0..31 (the two halves are
                                             // loaded a chunk ahead, outside the scratch)
constexpr uint32_t SMEM_BYTES = SM_GA + 8192;
static_assert(SM_MISC + MISC_P12BAR + 8 <= SM_NEGI && SMEM_BYTES <= 232448, "shared memory map");

// ---- tensor memory map (columns) -------------------------------------------
constexpr uint32_t TM_S = 0;       // S^T float32 (S'^T inside a chunk): lane = value channel
constexpr uint32_t TM_SHI = 128;   // S'^T bf16 hi, two key channels per column
constexpr uint32_t TM_SLO = 192;   // S'^T bf16 lo
constexpr uint32_t TM_ACC1 = 256;  // Gam (with TM_U) -> [Akk; Aqk]
constexpr uint32_t TM_U = 320;     // Gam (upper half) -> X'^T -> U^T
constexpr uint32_t TM_O = 384;     // O^T (adjacent to TM_U: one N=128 product feeds both)
constexpr uint32_t TM_UHI = 448;   // X'^T, then U^T, bf16 hi (two tokens per column)
constexpr uint32_t TM_ULO = 480;   // X'^T, then U^T, bf16 lo
constexpr uint32_t TM_COLS = 512;

// Byte offset of channels 8 cg .. 8 cg + 7 of token t in a q or k tile: each
// 64-channel half is 64 rows of 128 bytes (one per token) whose 16-byte chunks
// sit at chunk ^ (t & 7) (the 128-byte swizzle of the tile loads; lanes on
// consecutive tokens then read distinct banks).
__device__ __forceinline__ uint32_t off_sw128(int t, int cg) {
  return (cg >> 3) * 8192 + t * 128 + (((cg & 7) ^ (t & 7)) << 4);
}

// kPre: the fused input preprocessing p.pre is applied on chip (beta when it is
// staged, q and k in pass A, the gate on the g tile before its cumulative sum).
template <bool kPre>
__global__ void __launch_bounds__(kThreads, 1)
kda_prefill_bf16_kernel(const __grid_constant__ CUtensorMap tm_q,
                        const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_g,
                        const __grid_constant__ CUtensorMap tm_v,
                        const __grid_constant__ CUtensorMap tm_o, Bf16Params p) {
  extern __shared__ __align__(1024) unsigned char smem[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int qd = warp & 3;          // TMEM lane quarter of this warp
  const int cq = warp >> 2;         // which column slice of the accumulators this warp handles
  const int row = qd * 32 + lane;   // TMEM lane (accumulator row) of this thread

  // the factor e^Gam_last / c of the last tensor-core chunk, per key channel, that
  // the state in TMEM still owes (1 at an item's start and after a token chunk)
  float* s_pend = reinterpret_cast<float*>(smem + SM_MISC + MISC_PEND);
  float* s_gl = reinterpret_cast<float*>(smem + SM_MISC + MISC_GL);
  float* s_c = reinterpret_cast<float*>(smem + SM_MISC + MISC_C);
  float* s_nrho = reinterpret_cast<float*>(smem + SM_MISC + MISC_NRHO);
  float* s_gamc = reinterpret_cast<float*>(smem + SM_MISC + MISC_GAMC);
  float* s_beta = reinterpret_cast<float*>(smem + SM_MISC + MISC_BETA);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + SM_MISC + MISC_BAR);
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + SM_MISC + MISC_TMEM);
  uint32_t* s_flag = reinterpret_cast<uint32_t*>(smem + SM_MISC + MISC_FLAG);

  // A malformed cu_seqlens is latched by the scheduler before this kernel
  // starts; the value cannot change while it runs, so the test is CTA-uniform.
  if (p.status && *(volatile const unsigned int*)p.status == (unsigned)KDA_ERR_BAD_SEQLENS)
    return;
  // the swizzled tile layout assumes a 1024-byte aligned window (CTA-uniform test)
  if (smem_u32(smem) & 1023u) {
    if (tid == 0) latch_status(p.status, KDA_ERR_CUDA);
    return;
  }

  // The current work item: (sequence, head) chain, or a segment of one.
  int n = 0, h = 0;
  int64_t t0 = 0, len = 0;
  int64_t rel0 = 0, seq_len = 0;  // start of this item within its sequence; sequence length
  // start state (nullptr = zeros), identity start, end-state destination, flags
  const float* s_in = nullptr;
  float* s_out = nullptr;
  bool ident = false, zero_v = false, want_o = true;
  const int64_t n_items = item_count(p);
  auto decode = [&](int item) {
    const ItemInfo it = decode_item(p, item);
    n = it.n;
    h = it.h;
    t0 = it.t0;
    len = it.len;
    rel0 = it.rel0;
    seq_len = it.seq_len;
    s_in = it.s_in;
    s_out = it.s_out;
    ident = it.ident;
    zero_v = it.zero_v;
    want_o = it.want_o;
  };
  // nothing to do for this launch (a surplus pass of the packed split): leave
  // before any setup (CTA-uniform: the plan was written by an earlier launch)
  if ((int64_t)blockIdx.x >= n_items) return;

  if (tid == 0) {
    mbar_init(&bars[0], 1);
    mbar_init(&bars[1], 1);
    mbar_init(&bars[2], 1);
    mbar_init(&bars[3], 1);
    mbar_init(reinterpret_cast<uint64_t*>(smem + SM_MISC + MISC_P12BAR), 2);
    *s_flag = 0;
    fence_barrier_init();
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_g);
    tma_prefetch_desc(&tm_v);
  }
  if (warp == 0) {
    tmem_alloc(s_tmem, TM_COLS);
    tmem_relinquish();
  }
  // [L; L]: rows r and 64 + r hold row r of the 64 x 64 lower-triangular ones
  for (int i = tid; i < 128 * 8; i += kThreads) {
    const int r = i >> 3, kb = i & 7;
    float x[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) x[e] = (kb * 8 + e) <= (r & 63) ? 1.f : 0.f;
    st8(smem + SM_LL + off_kmaj(r, kb * 8, 64), x);
  }
  // TB parts start at zero: its blocks above the diagonal are never written
  for (int i = tid; i < 2 * 8192 / 16; i += kThreads)
    reinterpret_cast<uint4*>(smem + SM_Y + Y_TB_HI)[i] = make_uint4(0u, 0u, 0u, 0u);
  for (int i = tid; i < 64 * 8; i += kThreads) {  // -I, rows = N (token), K = token
    const int r = i >> 3, kb = i & 7;
    float x[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) x[e] = (kb * 8 + e) == r ? -1.f : 0.f;
    st8(smem + SM_NEGI + off_kmaj(r, kb * 8, 64), x);
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tb = *s_tmem;
  const uint32_t lane_base = (uint32_t)(qd * 32) << 16;
  Waits wt{&bars[0], &bars[1], 0u, 0u, s_flag, p.status};
  // Phase bookkeeping of the CTA's barriers carries over from item to item:
  // within an item every copy and product issued is also waited for.
  uint32_t tma_issued = 0;
  uint64_t* g_bar = &bars[3];
  uint32_t g_issued = 0, g_waited = 0;  // g_waited: thread 0's count
  uint64_t* xo_bar = &bars[2];          // completion of the products with S'
  uint32_t xo_issued = 0;
  uint64_t* p12_bar = reinterpret_cast<uint64_t*>(smem + SM_MISC + MISC_P12BAR);
  uint32_t p12_phase = 0;               // the output and state products, both issuers
  uint32_t* s_item = s_flag + 1;
  unsigned int* next_item = p.status + 16 + p.mode;  // zeroed with the status word

  // Persistent loop: the CTA takes items from the launch's counter, in order
  // (longest first where the items have different lengths), until none is left.
#pragma unroll 1
  for (;;) {
  if (tid == 0) *s_item = atomicAdd(next_item, 1u);
  __syncthreads();
  const int64_t item = *(volatile uint32_t*)s_item;
  __syncthreads();  // every thread has read it before thread 0 may fetch again
  if (item >= n_items) break;
  decode((int)item);

  const int nchunks = (int)((len + C - 1) / C);
  // one of the four tiles of a chunk (part 0 also arms the barrier); the four
  // parts are issued from different warps so their issue latencies overlap
  // (a tile's bytes may land before the barrier is armed: the transaction count
  // only has to balance when the arrival comes)
  // The g tile completes on its own barrier and travels as two 32-token halves
  // in buffers of their own: the next chunk's tile is loaded as soon as this
  // chunk's cumulative sum has read the previous one (a chunk ahead of the q, k
  // and v tiles, which share their buffers with the substitution scratch).
  // parts 0-3: the 64-channel halves of q and k (128-byte rows); 4: v
  auto issue_tma_part = [&](int chunk, int part) {
    const int32_t y = (int32_t)(t0 + (int64_t)chunk * C);
    if (part == 0) mbar_arrive_expect_tx(wt.tma_bar, 3 * 16384);
    if (part < 4)
      tma_load_2d(smem + SM_IN_Q + part * 8192, part < 2 ? &tm_q : &tm_k,
                  (int32_t)(h * D + (part & 1) * 64), y, wt.tma_bar);
    else
      tma_load_3d(smem + SM_IN_V, &tm_v, 0, y, h * (D / 8), wt.tma_bar);
  };
  // The scalar gate (one per token and head) has no tile to load: threads write
  // it, broadcast over the channels, into the g buffers (activate_gate below).
  const bool g_tma = !(kPre && p.pre.per_head);
  const bool g_fill = kPre && (p.pre.gate || p.pre.per_head);  // threads produce the g tile
  const float gsc = kPre && p.pre.gate_scale ? p.pre.gate_scale[h] : 1.f;
  auto issue_g_half = [&](int chunk, int half) {
    const int32_t y = (int32_t)(t0 + (int64_t)chunk * C + half * (C / 2));
    if (half == 0) mbar_arrive_expect_tx(g_bar, 16384);
    tma_load_3d(smem + (half ? SM_GB : SM_GA), &tm_g, 0, y, h * (D / 8), g_bar);
  };
  // the g barrier's phase of this item's chunk c is g_base + c
  const uint32_t g_base = g_issued;
  if (tid == 0 && nchunks > 0) {
    for (int part = 0; part < 5; ++part) issue_tma_part(0, part);
    if (g_tma) {
      issue_g_half(0, 0);
      issue_g_half(0, 1);
    }
  }
  if (nchunks > 0) {
    ++tma_issued;
    if (g_tma) ++g_issued;
  }
  // raw bf16 bits of beta for a chunk, loaded a chunk ahead and converted only
  // when used (no instruction waits on the load meanwhile); tokens past the
  // sequence end read as 0
  auto load_beta_bits = [&](int chunk) -> uint32_t {
    const int64_t tt = (int64_t)chunk * C + tid;
    uint32_t bits = 0u;
    if (tid < C && tt < len)
      bits = __bfloat16_as_ushort(p.beta[(t0 + tt) * p.H + h]);
    return bits;
  };
  uint32_t beta_bits = nchunks > 0 ? load_beta_bits(0) : 0u;

  // start state S^T (lane = value channel j, columns = key channels) from h0;
  // its bf16 parts are made per chunk, after the rescaling by c
  {
    const int j = row;
#pragma unroll 1
    for (int c0 = cq * SCOL; c0 < cq * SCOL + SCOL; c0 += 16) {
      uint32_t u[16];
#pragma unroll
      for (int e = 0; e < 16; ++e)
        u[e] = __float_as_uint(s_in ? s_in[(int64_t)(c0 + e) * D + j]
                                    : (ident && c0 + e == j ? 1.f : 0.f));
      tmem_st16(tb + lane_base + TM_S + c0, u);
    }
    tmem_wait_st();
    if (tid < D) s_pend[tid] = 1.f;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  const uint32_t idesc_cum = idesc_bf16(128, 128, 0, 1);
  const uint32_t idesc_kk = idesc_bf16(128, 64, 0, 0);
  const uint32_t idesc_mnk = idesc_bf16(128, 64, 1, 0);
  const uint32_t idesc_sq = idesc_bf16(128, 64, 0, 0);
  const uint32_t idesc_s = idesc_bf16(128, 128, 0, 1);
  const uint32_t sbase = smem_u32(smem);
  // prefix-cache checkpoints of this chain (output items only)
  const int64_t ck_base =
      want_o ? ckpt_base(p.ckpt, p.ckpt_off, p.ckpt_rows, p.ckpt_interval, n, seq_len, p.status,
                         tid == 0)
             : -1;
  // log2 of the chunk's per-channel reference c (an integer, clamped)
  auto ref_log2 = [](float rho) { return fminf(fmaxf(rintf(rho * kLog2e), -kRefExp2), kRefExp2); };
  // thread 0: once the g tile of `chunk` has landed, Gam (rows 0..63 and again
  // 64..127) = [L; L] G with G the g tile as an MN-major B (K steps 0, 1 on the
  // first half, 2, 3 on the second), committed to mma_bar; returns false if the
  // wait ran out
  auto issue_cumsum = [&](int chunk) -> bool {
    const bool ok = !g_tma || mbar_wait(g_bar, (g_base + (uint32_t)chunk) & 1u);
    if (g_tma) ++g_waited;
    if (!ok) return false;
    tc_fence_after();
#pragma unroll
    for (int kk = 0; kk < C / 16; ++kk)
      mma_ss(tb + TM_ACC1, (smem_desc(sbase + SM_LL, 128, 1024) + (uint64_t)(kk * 16)),
             (smem_desc(sbase + (kk < 2 ? SM_GA : SM_GB), 128, 512) + (uint64_t)((kk & 1) * 16)),
             idesc_cum, kk > 0);
    mma_commit(wt.mma_bar);
    return true;
  };
  // fused gate: log(alpha) = -gate_scale[h] softplus(raw) rounded to bf16, in
  // place on rows [i, end) of the g tile of `chunk` (16-byte rows of 8 channels;
  // 0..511 in the first half, 512..1023 in the second, each half [group][32
  // tokens]), stepping by `nthr`, once the tile has landed.  A scalar gate is
  // read per token from global memory and written to the 8 channels of the row.
  // The callers order these writes before the cumulative sum (a proxy fence and
  // a CTA barrier).
  constexpr int kHalfRows = (D / 8) * (C / 2);
  auto activate_gate = [&](int chunk, int i, int end, int nthr) {
    if (g_tma && !mbar_wait(g_bar, (g_base + (uint32_t)chunk) & 1u)) wt.on_timeout();
    for (; i < end; i += nthr) {
      uint8_t* r = smem + (i < kHalfRows ? SM_GA + i * 16 : SM_GB + (i - kHalfRows) * 16);
      float x[8];
      if (g_tma) {
        ld8(r, x);
#pragma unroll
        for (int e = 0; e < 8; ++e) x[e] = gsc * neg_softplus(x[e]);
      } else {
        const int64_t tt = (int64_t)chunk * C + (i < kHalfRows ? 0 : C / 2) + (i & (C / 2 - 1));
        float gv = tt < len ? __bfloat162float(p.g[(t0 + tt) * p.H + h]) : 0.f;
        if (p.pre.gate) gv = gsc * neg_softplus(gv);
#pragma unroll
        for (int e = 0; e < 8; ++e) x[e] = gv;
      }
      st8(r, x);
    }
  };
  // fused normalisation, warps 12-15: once the q and k tiles of `chunk` have
  // landed, the per-token sums of squares (s_nrm[token] for k, s_nrm[C + token]
  // for q); a lane per token (eight consecutive tokens cover all banks)
  float* s_nrm = reinterpret_cast<float*>(smem + SM_NRM);
  auto qk_sumsq = [&](uint32_t phase) {
    if (!mbar_wait(wt.tma_bar, phase & 1u)) wt.on_timeout();
    const int j = tid - 384, tt = j & (C - 1), isq = j >> 6;
    const uint8_t* base = smem + (isq ? SM_IN_Q : SM_IN_K);
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int cg = 0; cg < D / 8; ++cg) {
      float x[8];
      ld8(base + off_sw128(tt, cg), x);
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[e & 3] = fmaf(x[e], x[e], acc[e & 3]);
    }
    s_nrm[isq * C + tt] = (acc[0] + acc[1]) + (acc[2] + acc[3]);
  };
  // The exact token path for a chunk whose in-chunk decay span overflows the
  // factorisation (see pass A): the recurrence itself on the CUDA cores, with
  // the state read from and written back to TMEM, so the tensor-core path
  // continues from it.  Per token, for value channel j = row and key channels
  // cq*32 .. cq*32+31 of this thread:
  //   S <- diag(alpha) S;  p = S^T k, r = S^T q (one cross-warp sum);
  //   u = beta (v - p);    S <- S + k u^T;   o = scale (r + u (k . q))
  // alpha = e^g comes from global memory (the g tile buffers already hold the
  // next chunk's gate), activated exactly as the fused path does.  Costs about
  // four tensor-core chunks; ends with the same hand-over to chunk ci + 1.
  auto token_chunk = [&](int ci, int64_t cs, int nv) {
    float* s_al = reinterpret_cast<float*>(smem + SM_X + X_ALPHA);
    float2* s_red = reinterpret_cast<float2*>(smem + SM_Y + Y_RED);
    float* s_kq = reinterpret_cast<float*>(smem + SM_Y + Y_KQ);
    {  // alpha for (token tid / 8, channels 16 (tid % 8) ..); 1 past the sequence end
      const int tt = tid >> 3, c0 = (tid & 7) * 16;
      float a[16];
      if (tt < nv) {
        const int64_t tok = t0 + cs + tt;
        if (kPre && p.pre.per_head) {
          float gv = __bfloat162float(p.g[tok * p.H + h]);
          if (p.pre.gate) gv = round_to<__nv_bfloat16>(gsc * neg_softplus(gv));
#pragma unroll
          for (int e = 0; e < 16; ++e) a[e] = gv;
        } else {
          const uint4* src = reinterpret_cast<const uint4*>(p.g + (tok * p.H + h) * D + c0);
          const uint4 u0 = src[0], u1 = src[1];
          const uint32_t w[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            a[2 * e] = bf16_lo(w[e]);
            a[2 * e + 1] = bf16_hi(w[e]);
          }
          if (kPre && p.pre.gate)
#pragma unroll
            for (int e = 0; e < 16; ++e) a[e] = round_to<__nv_bfloat16>(gsc * neg_softplus(a[e]));
        }
#pragma unroll
        for (int e = 0; e < 16; ++e) a[e] = ex2(a[e] * kLog2e);  // e^-inf = 0
      } else {
#pragma unroll
        for (int e = 0; e < 16; ++e) a[e] = 1.f;
      }
      float4* dst = reinterpret_cast<float4*>(s_al + tt * D + c0);
#pragma unroll
      for (int e = 0; e < 4; ++e) dst[e] = make_float4(a[4 * e], a[4 * e + 1], a[4 * e + 2], a[4 * e + 3]);
    }
    {  // k . q per token: 16 lanes per token, two tokens per warp and pass
      const int half = lane >> 4, cg = lane & 15;
#pragma unroll
      for (int it = 0; it < 2; ++it) {
        const int tt = warp * 4 + it * 2 + half;
        float kx[8], qx[8];
        ld8(smem + SM_IN_K + off_sw128(tt, cg), kx);
        ld8(smem + SM_IN_Q + off_sw128(tt, cg), qx);
        float acc = 0.f;
#pragma unroll
        for (int e = 0; e < 8; ++e) acc = fmaf(kx[e], qx[e], acc);
#pragma unroll
        for (int o = 8; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
        if (kPre && p.pre.l2) acc *= inv_l2(s_nrm[tt]) * inv_l2(s_nrm[C + tt]);
        if (cg == 0) s_kq[tt] = acc;
      }
    }
    float sv[SCOL];  // S^T row j, key channels cq*32 ..
    {
      float a0[16], a1[16];
      tmem_ld16(tb + lane_base + TM_S + cq * SCOL, a0);
      tmem_ld16(tb + lane_base + TM_S + cq * SCOL + 16, a1);
      tmem_wait_ld();
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        sv[e] = a0[e] * s_pend[cq * SCOL + e];
        sv[16 + e] = a1[e] * s_pend[cq * SCOL + 16 + e];
      }
    }
    __syncthreads();  // alpha and k . q in place (and s_pend read)
    if (tid < D) s_pend[tid] = 1.f;  // the state goes back to TMEM owing nothing
    const int j = row;
    const uint8_t* vcol = smem + SM_IN_V + (j >> 3) * (C * 16) + (j & 7) * 2;
    const int64_t obase = ((t0 + cs) * p.H + h) * D + j, ostride = (int64_t)p.H * D;
#pragma unroll 1
    for (int tt = 0; tt < nv; ++tt) {
      float ik = 1.f, iq = 1.f;
      if (kPre && p.pre.l2) {
        ik = inv_l2(s_nrm[tt]);
        iq = inv_l2(s_nrm[C + tt]);
      }
      const float4* al4 = reinterpret_cast<const float4*>(s_al + tt * D + cq * SCOL);
      float2 pk = make_float2(0.f, 0.f), pq = make_float2(0.f, 0.f);
#pragma unroll
      for (int g4 = 0; g4 < SCOL / 8; ++g4) {
        float kx[8], qx[8];
        ld8(smem + SM_IN_K + off_sw128(tt, cq * (SCOL / 8) + g4), kx);
        ld8(smem + SM_IN_Q + off_sw128(tt, cq * (SCOL / 8) + g4), qx);
        const float4 a0 = al4[2 * g4], a1 = al4[2 * g4 + 1];
        const float al[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
#pragma unroll
        for (int e = 0; e < 8; e += 2) {
          float2 s2 = mul2(make_float2(sv[g4 * 8 + e], sv[g4 * 8 + e + 1]),
                           make_float2(al[e], al[e + 1]));
          sv[g4 * 8 + e] = s2.x;
          sv[g4 * 8 + e + 1] = s2.y;
          pk = fma2(s2, make_float2(kx[e] * ik, kx[e + 1] * ik), pk);
          pq = fma2(s2, make_float2(qx[e] * iq, qx[e + 1] * iq), pq);
        }
      }
      const int buf = tt & 1;
      s_red[(buf * NCOL + cq) * 128 + j] = make_float2(pk.x + pk.y, pq.x + pq.y);
      __syncthreads();  // double-buffered partial sums: one barrier per token
      float P = 0.f, Q = 0.f;
#pragma unroll
      for (int c = 0; c < NCOL; ++c) {
        const float2 r = s_red[(buf * NCOL + c) * 128 + j];
        P += r.x;
        Q += r.y;
      }
      const float vj = zero_v ? 0.f
                              : __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(
                                    vcol + tt * 16));
      const float u = s_beta[tt] * (vj - P);
      const float2 u2 = make_float2(u, u);
#pragma unroll
      for (int g4 = 0; g4 < SCOL / 8; ++g4) {
        float kx[8];
        ld8(smem + SM_IN_K + off_sw128(tt, cq * (SCOL / 8) + g4), kx);
#pragma unroll
        for (int e = 0; e < 8; e += 2) {
          const float2 s2 = fma2(make_float2(kx[e] * ik, kx[e + 1] * ik), u2,
                                 make_float2(sv[g4 * 8 + e], sv[g4 * 8 + e + 1]));
          sv[g4 * 8 + e] = s2.x;
          sv[g4 * 8 + e + 1] = s2.y;
        }
      }
      if (want_o && cq == 0) {
        const float o = p.scale * fmaf(u, s_kq[tt], Q);
        if (nv == C) {  // staged for the bulk store, as the tensor-core chunk does
          if (p.out_bf16)
            reinterpret_cast<__nv_bfloat16*>(smem + SM_X + X_OUT)[tt * D + j] =
                __float2bfloat16_rn(o);
          else
            reinterpret_cast<float*>(smem + SM_X + X_OUT)[tt * D + j] = o;
        } else if (p.out_bf16) {
          static_cast<__nv_bfloat16*>(p.out)[obase + tt * ostride] = __float2bfloat16_rn(o);
        } else {
          static_cast<float*>(p.out)[obase + tt * ostride] = o;
        }
      }
    }
    {  // the state back to TMEM, and the chunk's checkpoint
      uint32_t w0[16], w1[16];
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        w0[e] = __float_as_uint(sv[e]);
        w1[e] = __float_as_uint(sv[16 + e]);
      }
      tmem_st16(tb + lane_base + TM_S + cq * SCOL, w0);
      tmem_st16(tb + lane_base + TM_S + cq * SCOL + 16, w1);
      const int64_t done = rel0 + cs + C;
      if (ck_base >= 0 && nv == C && done % p.ckpt_interval == 0) {
        float* ck = p.ckpt + ((ck_base + done / p.ckpt_interval - 1) * p.H + h) * D * D + j;
#pragma unroll
        for (int e = 0; e < SCOL; ++e) ck[(int64_t)(cq * SCOL + e) * D] = sv[e];
      }
      tmem_wait_st();
    }
    fence_proxy_async_smem();  // staged outputs are read by the bulk store
    tc_fence_before();
    __syncthreads();  // every thread is done with the q, k, v tiles and the staging
    // hand-over to chunk ci + 1, as the tensor-core chunk does it: its q, k, v
    // tiles, this chunk's outputs, the fused preprocessing, its cumulative sum
    if (ci + 1 < nchunks) {
      if (lane == 0 && warp >= 1 && warp <= 5) issue_tma_part(ci + 1, warp - 1);
      ++tma_issued;
    }
    if (tid == 0 && want_o && nv == C) {
      tma_store_2d(&tm_o, h * D, (int32_t)(t0 + cs), smem + SM_X + X_OUT);
      bulk_commit();
    }
    if (kPre && ci + 1 < nchunks && (g_fill || p.pre.l2)) {
      if (g_fill) {
        activate_gate(ci + 1, tid, 2 * kHalfRows, kThreads);
        fence_proxy_async_smem();
      }
      if (p.pre.l2 && warp >= 12) qk_sumsq(tma_issued - 1);
      __syncthreads();
    }
    if (tid == 0 && ci + 1 < nchunks && !issue_cumsum(ci + 1)) wt.on_timeout();
  };
  if (kPre && nchunks > 0 && (g_fill || p.pre.l2)) {
    if (g_fill) activate_gate(0, tid, 2 * kHalfRows, kThreads);
    if (p.pre.l2 && warp >= 12) qk_sumsq(tma_issued - 1);  // chunk 0's tiles
    fence_proxy_async_smem();
    __syncthreads();
  }
  if (tid == 0 && nchunks > 0 && !issue_cumsum(0)) wt.on_timeout();

#pragma unroll 1
  for (int ci = 0; ci < nchunks; ++ci) {
    const int64_t cs = (int64_t)ci * C;
    const int nv = (int)(len - cs < C ? len - cs : C);
    const int rho_t = nv - 1 < 31 ? nv - 1 : 31;

    // ---- P1: beta; wait for the q, k, v tiles and for the cumulative log-decay
    // (issued at the end of the previous chunk, or before the loop)
    if (tid < C) {
      float bt = __uint_as_float(beta_bits << 16);
      if (kPre) {  // branch-free select
        const float sb = round_to<__nv_bfloat16>(sigmoid_f(bt));
        bt = p.pre.beta && tid < nv ? sb : bt;
      }
      s_beta[tid] = bt;
    }
    if (ci + 1 < nchunks) beta_bits = load_beta_bits(ci + 1);
    if (wt.wait_tma()) break;
    if (wt.wait_mma()) break;
    // the cumulative sum has read the g tile: load the next chunk's
    if (g_tma && ci + 1 < nchunks) {
      if (lane == 0 && (warp == 1 || warp == 2)) issue_g_half(ci + 1, warp - 1);
      ++g_issued;
    }

    // ---- P3 (pass A): per-channel reference, the decayed key/query operands,
    // in two halves of 64 key channels: the tensor core runs [Akk; Aqk]'s first
    // four K steps while the threads produce the second half (the previous
    // chunk's output store reads X until it completes)
    if (tid == 0) bulk_wait_read();
    const int t = row & 63;
    const int cgA = NCOL * (row >> 6) + cq;  // this thread's 8-channel groups: cgA, cgA + 8
    const bool valid = t < nv;
    float gam[2][8];
    tmem_ld8(tb + lane_base + TM_ACC1 + cgA * 8, gam[0]);
    tmem_ld8(tb + lane_base + TM_ACC1 + (cgA + 8) * 8, gam[1]);
    tmem_wait_ld();
    if (t == rho_t)  // log2 c per channel (s_nrho holds its negative from here on)
#pragma unroll
      for (int hf = 0; hf < 2; ++hf)
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float r = ref_log2(gam[hf][e]);
          s_nrho[(cgA + 8 * hf) * 8 + e] = -r;
        }
    if (t == nv - 1)
#pragma unroll
      for (int hf = 0; hf < 2; ++hf)
#pragma unroll
        for (int e = 0; e < 8; ++e) s_gl[(cgA + 8 * hf) * 8 + e] = gam[hf][e];
    tc_fence_before();
    __syncthreads();
    float inv_k = 1.f, inv_q = 1.f;
    if (kPre && p.pre.l2) {  // sums of squares from the previous chunk's last products
      inv_k = inv_l2(s_nrm[t]);
      inv_q = inv_l2(s_nrm[C + t]);
    }
    if (tid < D) {
      const float e2 = -s_nrho[tid];
      s_c[tid] = ldexpf(1.f, (int)e2);
      s_gamc[tid] = ex2(s_gl[tid] * kLog2e - e2);  // e^Gam_last / c
    }
    bool wide = false;  // a factor of this thread's slice leaves the exponent range (or is NaN)
    // thread 0: [Akk; Aqk] += R Ck^T over K steps 4 half .. 4 half + 3 (channels
    // 64 half .. 64 half + 63), three split products; the first step overwrites
    auto issue_akk = [&](int half) {
      const uint32_t r_hi = sbase + SM_X + X_R_HI, r_lo = sbase + SM_X + X_R_LO;
      const uint32_t c_hi = sbase + SM_X + X_CK_HI, c_lo = sbase + SM_X + X_CK_LO;
      const uint32_t as[3] = {r_hi, r_hi, r_lo}, bs[3] = {c_hi, c_lo, c_hi};
#pragma unroll
      for (int pr = 0; pr < 3; ++pr)
#pragma unroll
        for (int k4 = 0; k4 < 4; ++k4) {
          const int kk = 4 * half + k4;
          mma_ss(tb + TM_ACC1, (smem_desc(as[pr], 128, 2048) + (uint64_t)(kk * 16)),
                 (smem_desc(bs[pr], 128, 2048) + (uint64_t)(kk * 16)), idesc_kk, (pr | kk) != 0);
        }
    };
    // U^T (+)= X'^T (-TB)^T over K step kk (tokens j of column block kk of TB), three
    // split products; thread 256 issues step 3 once T's diagonal blocks are in TB,
    // step 2 once blocks (1,0) and (3,2) are, steps 1 and 0 after the join
    auto issue_u_step = [&](int kk) {
      const uint32_t tbh = sbase + SM_Y + Y_TB_HI, tbl = sbase + SM_Y + Y_TB_LO;
      const uint32_t xa[3] = {TM_UHI, TM_UHI, TM_ULO}, bt[3] = {tbh, tbl, tbh};
#pragma unroll
      for (int pr = 0; pr < 3; ++pr)
        mma_ts(tb + TM_U, tb + xa[pr] + kk * 8,
               (smem_desc(bt[pr], 128, 1024) + (uint64_t)(kk * 16)), idesc_sq,
               kk != 3 || pr != 0);
    };
    // R_K, R_Q and Ck of token t, channels 8 cg .. 8 cg + 7, split into the X operands;
    // rows past the sequence end are zero (their factors are never formed)
    auto decayed = [&](int cg, const float (&gm)[8]) {
      float rk[8], rq[8], ck[8];
      if (valid) {
        float kx[8], qx[8];
        ld8(smem + SM_IN_K + off_sw128(t, cg), kx);
        ld8(smem + SM_IN_Q + off_sw128(t, cg), qx);
        const float4 na = *reinterpret_cast<const float4*>(s_nrho + cg * 8);
        const float4 nb = *reinterpret_cast<const float4*>(s_nrho + cg * 8 + 4);
        const float nr[8] = {na.x, na.y, na.z, na.w, nb.x, nb.y, nb.z, nb.w};
#pragma unroll
        for (int e = 0; e < 8; e += 2) {
          // log2(e^Gam / c); an out-of-range chunk never uses its (infinite) operands
          const float2 d = fma2(make_float2(gm[e], gm[e + 1]), make_float2(kLog2e, kLog2e),
                                make_float2(nr[e], nr[e + 1]));
          wide |= !(fabsf(d.x) <= kMaxExp2) || !(fabsf(d.y) <= kMaxExp2);
          const float2 er = make_float2(ex2(d.x), ex2(d.y));
          const float2 ec = make_float2(ex2(-d.x), ex2(-d.y));
          float2 kv = make_float2(kx[e], kx[e + 1]), qv = make_float2(qx[e], qx[e + 1]);
          if (kPre && p.pre.l2) {  // normalised in float32, unrounded
            kv = mul2(kv, make_float2(inv_k, inv_k));
            qv = mul2(qv, make_float2(inv_q, inv_q));
          }
          const float2 a = mul2(kv, er), b = mul2(qv, er), c2 = mul2(kv, ec);
          rk[e] = a.x;
          rk[e + 1] = a.y;
          rq[e] = b.x;
          rq[e + 1] = b.y;
          ck[e] = c2.x;
          ck[e + 1] = c2.y;
        }
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) rk[e] = rq[e] = ck[e] = 0.f;
      }
      st8_split(smem + SM_X + X_R_HI + off_kmaj(t, cg * 8, 128),
                smem + SM_X + X_R_LO + off_kmaj(t, cg * 8, 128), rk);
      st8_split(smem + SM_X + X_R_HI + off_kmaj(64 + t, cg * 8, 128),
                smem + SM_X + X_R_LO + off_kmaj(64 + t, cg * 8, 128), rq);
      st8_split(smem + SM_X + X_CK_HI + off_kmaj(t, cg * 8, 128),
                smem + SM_X + X_CK_LO + off_kmaj(t, cg * 8, 128), ck);
    };
    decayed(cgA, gam[0]);
    fence_proxy_async_smem();
    const bool wide0 = __syncthreads_or(wide);
    if (!wide0 && tid == 0) {  // thread 0 issues both halves: its commit covers them
      tc_fence_after();
      issue_akk(0);
    }
    decayed(cgA + 8, gam[1]);
    fence_proxy_async_smem();
    // A factor beyond 2^+-115 (an in-chunk decay span of more than about 160
    // nats on some channel, alpha = 0 included) would overflow the
    // factorisation: the whole chunk then runs the recurrence token by token,
    // once the first half's products (if issued) have finished.
    // (A wait that ran out there is seen after the next chunk's first barrier.)
    if (__syncthreads_or(wide)) {
      if (!wide0) {
        if (tid == 0) mma_commit(wt.mma_bar);
        if (wt.wait_mma()) break;
      }
      token_chunk(ci, cs, nv);
      continue;
    }

    // ---- P4: the second half of [Akk; Aqk] (thread 0), while every thread
    // rescales its slice of the state: S = S_prev diag(e^Gam_last / c_prev), the
    // factor the previous chunk left owing, then S' = S diag(c) (exact: c is a power
    // of two), both transposed, with the bf16 parts of S'
    if (tid == 0) {
      tc_fence_after();
      issue_akk(1);
      mma_commit(wt.mma_bar);  // both halves
    }
    {
      float sv[SCOL / 16][16];
#pragma unroll
      for (int q4 = 0; q4 < SCOL / 16; ++q4)
        tmem_ld16(tb + lane_base + TM_S + cq * SCOL + q4 * 16, sv[q4]);
      tmem_wait_ld();
#pragma unroll
      for (int q4 = 0; q4 < SCOL / 16; ++q4) {
        const int c0 = cq * SCOL + q4 * 16;
        uint32_t w[16], hi[8], lo[8];
#pragma unroll
        for (int e = 0; e < 16; e += 4) {
          const float4 c4 = *reinterpret_cast<const float4*>(s_c + c0 + e);
          const float4 p4 = *reinterpret_cast<const float4*>(s_pend + c0 + e);
          // two roundings at most: the product with the owed factor, then the exact
          // power-of-two scaling (one combined factor could underflow)
          const float2 a = mul2(mul2(make_float2(sv[q4][e], sv[q4][e + 1]), make_float2(p4.x, p4.y)),
                                make_float2(c4.x, c4.y));
          const float2 b = mul2(mul2(make_float2(sv[q4][e + 2], sv[q4][e + 3]), make_float2(p4.z, p4.w)),
                                make_float2(c4.z, c4.w));
          sv[q4][e] = a.x;
          sv[q4][e + 1] = a.y;
          sv[q4][e + 2] = b.x;
          sv[q4][e + 3] = b.y;
        }
#pragma unroll
        for (int e = 0; e < 16; ++e) w[e] = __float_as_uint(sv[q4][e]);
        tmem_st16(tb + lane_base + TM_S + c0, w);
        pack_split16(sv[q4], hi, lo);
        tmem_st8(tb + lane_base + TM_SHI + c0 / 2, hi);
        tmem_st8(tb + lane_base + TM_SLO + c0 / 2, lo);
      }
      tmem_wait_st();
    }
    tc_fence_before();
    __syncthreads();
    ++xo_issued;  // thread 256 commits to xo_bar once per chunk (below)
    // From here to the join below the two halves of the CTA take different paths
    // (waits that run out only raise the flag; the CTA leaves after the join).
    //   warps 0-7:  P5 (A and Aqk from [Akk; Aqk]) and P6 (T = (I + A)^-1, whose
    //               producers also write -T diag(beta), split, into the TB operand)
    //   warps 8-15: thread 256 issues the products with S' once [Akk; Aqk] is done
    //               (the two streams then do not interleave on the tensor pipe),
    //               then the warps split X'
    if (warp < 8) {
      if (!mbar_wait(wt.mma_bar, wt.mma_phase)) wt.on_timeout();
      tc_fence_after();
      // ---- P5: A = strict_lower(beta Akk) (float32, for the substitution), Aqk split
      {
        float a[2][TCOL];
        tmem_ld16(tb + lane_base + TM_ACC1 + cq * 32, a[0]);
        tmem_ld16(tb + lane_base + TM_ACC1 + cq * 32 + 16, a[1]);
        tmem_wait_ld();
        if (row < 64) {
          const int i = row;
          const float bi = s_beta[i];
          float* AT = reinterpret_cast<float*>(smem + SV_AT);  // AT[j][i] = A[i][j]
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const int j = cq * 32 + e;
            AT[j * ALD + i] = j < i ? bi * a[e >> 4][e & 15] : 0.f;
          }
        } else if (want_o) {
          const int i = row - 64;
#pragma unroll
          for (int e8 = 0; e8 < 4; ++e8) {
            float x[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              const int j = cq * 32 + e8 * 8 + e;
              x[e] = j <= i ? a[e8 >> 1][(e8 & 1) * 8 + e] : 0.f;
            }
            const uint32_t o = off_kmaj(i, cq * 32 + e8 * 8, 64);
            st8_split(smem + SM_Y + Y_AQK_HI + o, smem + SM_Y + Y_AQK_LO + o, x);
          }
        }
      }
      named_bar_sync(1, 256);
      // ---- P6 (warps 0-7): T = (I + A)^-1 by blocks of 16 (named barrier 1)
      const float* AT = reinterpret_cast<const float*>(smem + SV_AT);  // AT[j][i]
      float* T32 = reinterpret_cast<float*>(smem + SV_T32);
      float* M32 = reinterpret_cast<float*>(smem + SV_M32);
      if (warp < 4 && lane < 16) {
        // diagonal block I = warp, column jj = lane: right-looking substitution, so
        // each of the 16 steps is a set of independent updates
        const int base = warp * 16, jj = lane;
        float acc[16], x[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) acc[i] = 0.f;
#pragma unroll
        for (int m = 0; m < 16; ++m) {
          x[m] = m < jj ? 0.f : (m == jj ? 1.f : acc[m]);
#pragma unroll
          for (int i = m + 1; i < 16; ++i)
            acc[i] = fmaf(-AT[(base + m) * ALD + base + i], x[m], acc[i]);
        }
        const float nb = -s_beta[base + jj];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          T32[(base + i) * TLD + base + jj] = x[i];
          store_tb1<64>(smem + SM_Y + Y_TB_HI, smem + SM_Y + Y_TB_LO, base + i, base + jj, x[i] * nb);
        }
      }
      named_bar_sync(1, 256);
      fence_proxy_async_smem();  // the diagonal blocks of TB: the U product's step 3
      named_bar_arrive(3, 288);
      // 32 x 32 diagonal blocks: T[I, J] = -T[I, I] A[I, J] T[J, J] for (I, J) = (1, 0)
      // and (3, 2), two warps per block (one per 8-column n-tile), as m16n8k8 tf32
      // products with 3-term splitting; each warp only reads back its own columns.
      const int g = lane >> 2, t4 = lane & 3;
      float af[4], bf[2], acc[3][4];
      if (warp < 4) {
        const int J = (warp >> 1) * 2, I = J + 1, nt = warp & 1;
        float* Mw = M32 + J * 256;
        zero_acc(acc);
#pragma unroll
        for (int ks = 0; ks < 2; ++ks) {
          const int k0 = J * 16 + ks * 8;
          load_a_t<ALD>(AT, I * 16, k0, g, t4, af);
          load_b(T32, TLD, k0, J * 16 + nt * 8, g, t4, bf);
          mma_tf32x3(acc, af, bf);
        }
        store_c(Mw, 16, nt * 8, acc, g, t4, 1.f);
        __syncwarp();
        zero_acc(acc);
#pragma unroll
        for (int ks = 0; ks < 2; ++ks) {
          load_a(T32, TLD, I * 16, I * 16 + ks * 8, g, t4, af);
          load_b(Mw, 16, ks * 8, nt * 8, g, t4, bf);
          mma_tf32x3(acc, af, bf);
        }
        store_t_block<64>(T32, TLD, I * 16, J * 16 + nt * 8, acc, g, t4, -1.f, s_beta,
                      smem + SM_Y + Y_TB_HI, smem + SM_Y + Y_TB_LO);
      }
      named_bar_sync(1, 256);
      fence_proxy_async_smem();  // blocks (1,0) and (3,2) of TB: the U product's step 2
      named_bar_arrive(4, 288);
      // lower-left 32 x 32 block: M = A[2..3, 0..1] T[0..1, 0..1], then
      // T[2..3, 0..1] = -T[2..3, 2..3] M; warp = (row block i, column block j, n-tile)
      {
        const int i = warp >> 2, j = (warp >> 1) & 1, nt = warp & 1;
        zero_acc(acc);
        for (int kb = j; kb < 2; ++kb)
#pragma unroll
          for (int ks = 0; ks < 2; ++ks) {
            const int k0 = kb * 16 + ks * 8;
            load_a_t<ALD>(AT, (2 + i) * 16, k0, g, t4, af);
            load_b(T32, TLD, k0, j * 16 + nt * 8, g, t4, bf);
            mma_tf32x3(acc, af, bf);
          }
        store_c(M32 + (i * 2 + j) * 256, 16, nt * 8, acc, g, t4, 1.f);
        named_bar_sync(1, 256);
        zero_acc(acc);
        for (int kb = 0; kb <= i; ++kb)
#pragma unroll
          for (int ks = 0; ks < 2; ++ks) {
            load_a(T32, TLD, (2 + i) * 16, (2 + kb) * 16 + ks * 8, g, t4, af);
            load_b(M32 + (kb * 2 + j) * 256, 16, ks * 8, nt * 8, g, t4, bf);
            mma_tf32x3(acc, af, bf);
          }
        store_t_block<64>(T32, TLD, (2 + i) * 16, j * 16 + nt * 8, acc, g, t4, -1.f, s_beta,
                      smem + SM_Y + Y_TB_HI, smem + SM_Y + Y_TB_LO);
      }
    } else {
      // thread 256: [X' | O]^T = S'^T [R_K; R_Q]^T as N = 128 products over the
      // adjacent U and O accumulators (K = key channel, three split products), then
      // X'^T -= V^T as V^T (-I) (V exact in bf16; A = the v tile as an MN-major
      // operand).  Committed even when the wait ran out, so xo_bar still arrives.
      if (tid == 256) {
        const bool ok = mbar_wait(wt.mma_bar, wt.mma_phase);
        if (!ok) wt.on_timeout();
        tc_fence_after();
        if (ok) {
          const uint32_t rh = sbase + SM_X + X_R_HI, rl = sbase + SM_X + X_R_LO;
          const uint32_t sa[3] = {TM_SHI, TM_SHI, TM_SLO};
          const uint32_t bk[3] = {rh, rl, rh};
          const uint32_t idesc_xo = want_o ? idesc_bf16(128, 128, 0, 0) : idesc_kk;
#pragma unroll
          for (int pr = 0; pr < 3; ++pr)
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk)
              mma_ts(tb + TM_U, tb + sa[pr] + kk * 8,
                     (smem_desc(bk[pr], 128, 2048) + (uint64_t)(kk * 16)), idesc_xo,
                     (pr | kk) != 0);
          if (!zero_v)
#pragma unroll
            for (int kk = 0; kk < C / 16; ++kk)
              mma_ss(tb + TM_U, (smem_desc(sbase + SM_IN_V, 128, 1024) + (uint64_t)(kk * 16)),
                     (smem_desc(sbase + SM_NEGI, 128, 1024) + (uint64_t)(kk * 16)), idesc_mnk, 1);
        }
        mma_commit(xo_bar);
      }
      // this warp: lane quarter qd, tokens h8 * 32 .. h8 * 32 + 31 of X'^T
      if (!mbar_wait(xo_bar, (xo_issued - 1) & 1u)) wt.on_timeout();
      tc_fence_after();
      const int h8 = (warp >> 2) - 2;
      float y[2][16];
      tmem_ld16(tb + lane_base + TM_U + h8 * 32, y[0]);
      tmem_ld16(tb + lane_base + TM_U + h8 * 32 + 16, y[1]);
      tmem_wait_ld();
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int tt0 = h8 * 32 + hh * 16;
        uint32_t hi[8], lo[8];
        pack_split16(y[hh], hi, lo);
        tmem_st8(tb + lane_base + TM_UHI + tt0 / 2, hi);
        tmem_st8(tb + lane_base + TM_ULO + tt0 / 2, lo);
      }
      tmem_wait_st();
      // all of X' split (and U read): the first steps of the U product, as soon as
      // their blocks of TB are ready
      tc_fence_before();
      named_bar_sync(2, 256);
      if (warp == 8) {
        named_bar_sync(3, 288);
        if (lane == 0) {
          tc_fence_after();
          issue_u_step(3);
        }
        __syncwarp();
        named_bar_sync(4, 288);
        if (lane == 0) {
          tc_fence_after();
          issue_u_step(2);
        }
        __syncwarp();
      } else if (g_fill && ci + 1 < nchunks) {
        // fused gate: the next chunk's g tile activated while warps 0-7 solve for T
        // (it was requested a chunk ahead); ordered before its cumulative sum by the
        // proxy fence and the join below
        activate_gate(ci + 1, tid - 288, 2 * kHalfRows, kThreads - 288);
        fence_proxy_async_smem();
      }
    }
    wt.mma_phase ^= 1u;  // [Akk; Aqk] consumed (waited above by warps 0-7 and thread 256)
    fence_proxy_async_smem();  // TB, written by the substitution, is an MMA operand next
    tc_fence_before();
    __syncthreads();
    // ---- P8: the rest of U^T = X'^T (-TB)^T (thread 256, whose commit covers all
    // four steps; committed also when the CTA leaves, so the drain sees them)
    {
      const bool leave = *(volatile uint32_t*)s_flag != 0;
      if (tid == 256) {
        tc_fence_after();
        if (!leave) {
          issue_u_step(1);
          issue_u_step(0);
        }
        mma_commit(wt.mma_bar);
      }
      if (leave) {
        wt.mma_phase ^= 1u;  // the drain waits for this commit
        break;
      }
    }
    // prefetch chunk ci+1 (the q, k, v tiles are consumed; warps 1-5 issue one part each)
    if (ci + 1 < nchunks) {
      if (lane == 0 && warp >= 1 && warp <= 5) issue_tma_part(ci + 1, warp - 1);
      ++tma_issued;
    }
    if (wt.wait_mma()) break;

    // ---- P11: U^T split into TMEM (A operand of the last products)
    {
      float u[TCOL];
      tmem_ld16(tb + lane_base + TM_U + cq * TCOL, u);
      tmem_wait_ld();
      uint32_t hi[8], lo[8];
      pack_split16(u, hi, lo);
      tmem_st8(tb + lane_base + TM_UHI + cq * (TCOL / 2), hi);
      tmem_st8(tb + lane_base + TM_ULO + cq * (TCOL / 2), lo);
      tmem_wait_st();
    }
    tc_fence_before();
    __syncthreads();

    // ---- P12: S'^T += U^T Ck (thread 0) and O^T += U^T Aqk^T (thread 256), two
    // accumulators issued side by side, each issuer committing once to p12_bar (all
    // split; Ck is an MN-major B with N = key channel)
    if (tid == 0) {
      tc_fence_after();
      const uint32_t kh = sbase + SM_X + X_CK_HI, kl = sbase + SM_X + X_CK_LO;
      const uint32_t ua[3] = {TM_UHI, TM_UHI, TM_ULO};
      const uint32_t bk[3] = {kh, kl, kh};
#pragma unroll
      for (int pr = 0; pr < 3; ++pr)
#pragma unroll
        for (int kk = 0; kk < C / 16; ++kk)
          mma_ts(tb + TM_S, tb + ua[pr] + kk * 8,
                 (smem_desc(bk[pr], 2048, 128) + (uint64_t)(kk * 256)), idesc_s, 1);
      mma_commit(p12_bar);
      // the next chunk's cumulative sum right behind them (ACC1 and U are free; a
      // fused gate was activated during the substitution)
      if (ci + 1 < nchunks && !issue_cumsum(ci + 1)) wt.on_timeout();
    } else if (tid == 256) {
      tc_fence_after();
      const uint32_t ah = sbase + SM_Y + Y_AQK_HI, al = sbase + SM_Y + Y_AQK_LO;
      const uint32_t ua[3] = {TM_UHI, TM_UHI, TM_ULO};
      const uint32_t bq[3] = {ah, al, ah};
      if (want_o)
#pragma unroll
        for (int pr = 0; pr < 3; ++pr)
#pragma unroll
          for (int kk = 0; kk < C / 16; ++kk)
            mma_ts(tb + TM_O, tb + ua[pr] + kk * 8,
                   (smem_desc(bq[pr], 128, 1024) + (uint64_t)(kk * 16)), idesc_sq, 1);
      mma_commit(p12_bar);  // (with no products it arrives at once)
    }
    // while these products run: the next chunk's q/k sums of squares (warps 12-15;
    // the tiles were requested in P8)
    if (kPre && ci + 1 < nchunks && p.pre.l2 && warp >= 12) qk_sumsq(tma_issued - 1);
    if (!mbar_wait(p12_bar, p12_phase)) wt.on_timeout();
    p12_phase ^= 1u;
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (*(volatile uint32_t*)s_flag) break;

    // ---- P13: outputs.  The state stays S'^T in TMEM, owing diag(e^Gam_last / c):
    // the next chunk's P4 (or token path, or the item's end) applies it.
    {
      const int j = row;
      float o[TCOL];
      tmem_ld16(tb + lane_base + TM_O + cq * TCOL, o);
      // a checkpoint when rel0 + (ci + 1) C tokens of the sequence are done and that
      // is a multiple of the interval: state [key channel][value channel]
      const int64_t done = rel0 + cs + C;
      if (ck_base >= 0 && nv == C && done % p.ckpt_interval == 0) {
        float* ck = p.ckpt + ((ck_base + done / p.ckpt_interval - 1) * p.H + h) * D * D + j;
#pragma unroll 1
        for (int c0 = cq * SCOL; c0 < cq * SCOL + SCOL; c0 += 16) {
          float sv[16];
          tmem_ld16(tb + lane_base + TM_S + c0, sv);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 16; ++e) ck[(int64_t)(c0 + e) * D] = sv[e] * s_gamc[c0 + e];
        }
      }
      tmem_wait_ld();
      if (tid < D) s_pend[tid] = s_gamc[tid];
      if (want_o && nv == C) {
        // full chunk: stage [token][value channel] in X, one bulk tensor store below
        if (p.out_bf16) {
          __nv_bfloat16* st = reinterpret_cast<__nv_bfloat16*>(smem + SM_X + X_OUT);
#pragma unroll
          for (int e = 0; e < TCOL; ++e)
            st[(cq * TCOL + e) * D + j] = __float2bfloat16_rn(p.scale * o[e]);
        } else {
          float* st = reinterpret_cast<float*>(smem + SM_X + X_OUT);
#pragma unroll
          for (int e = 0; e < TCOL; ++e) st[(cq * TCOL + e) * D + j] = p.scale * o[e];
        }
        fence_proxy_async_smem();
      } else if (want_o) {
        // partial last chunk: element stores, only for tokens of this sequence
        float* outf = static_cast<float*>(p.out);
        __nv_bfloat16* outb = static_cast<__nv_bfloat16*>(p.out);
        const int64_t obase = ((t0 + cs) * p.H + h) * D + j;
        const int64_t ostride = (int64_t)p.H * D;
#pragma unroll
        for (int e = 0; e < TCOL; ++e) {
          const int tt = cq * TCOL + e;
          if (tt < nv) {
            if (p.out_bf16)
              outb[obase + tt * ostride] = __float2bfloat16_rn(p.scale * o[e]);
            else
              outf[obase + tt * ostride] = p.scale * o[e];
          }
        }
      }
    }
    tc_fence_before();
    __syncthreads();
    if (tid == 0 && want_o && nv == C) {
      tma_store_2d(&tm_o, h * D, (int32_t)(t0 + cs), smem + SM_X + X_OUT);
      bulk_commit();
    }
  }

  if (tid == 0) bulk_wait_all();  // this item's outputs are complete
  const bool aborted = *(volatile uint32_t*)s_flag != 0;
  if (!aborted && s_out) {
    const int j = row;
    float* hTp = s_out;
    tc_fence_after();
#pragma unroll 1
    for (int c0 = cq * SCOL; c0 < cq * SCOL + SCOL; c0 += 16) {
      float s[16];
      tmem_ld16(tb + lane_base + TM_S + c0, s);
      tmem_wait_ld();
#pragma unroll
      for (int e = 0; e < 16; ++e) hTp[(int64_t)(c0 + e) * D + j] = s[e] * s_pend[c0 + e];
    }
  }
  if (aborted && tid == 0) {
    // drain what may still be in flight before the memory goes away (bounded)
    for (uint32_t ph = wt.tma_waited; ph < tma_issued; ++ph)
      mbar_wait(wt.tma_bar, ph & 1u, 20000000ll);
    mbar_wait(wt.mma_bar, wt.mma_phase ^ 1u, 20000000ll);
    mbar_wait(p12_bar, p12_phase ^ 1u, 20000000ll);
    if (xo_issued) mbar_wait(xo_bar, (xo_issued - 1) & 1u, 20000000ll);
    for (uint32_t ph = g_waited; ph < g_issued; ++ph) mbar_wait(g_bar, ph & 1u, 20000000ll);
  }
  tc_fence_before();
  __syncthreads();
  if (aborted) break;
  }  // items
  if (warp == 0) tmem_dealloc(tb, TM_COLS);
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
// Tile map over one activation tensor [tokens, H, D] (bf16): box = 64 tokens x
// 16 groups of 8 channels, written to shared memory as [group][token][8].
// Store map over the output [tokens, H, D] (float32 or bf16): box = 64 tokens x D
// channels of one head, read from shared memory as [token][channel].
bool make_out_map(CUtensorMap* m, void* base, int64_t tokens, int H, bool bf16) {
  auto enc = get_encode();
  if (!enc) return false;
  const cuuint64_t es = bf16 ? 2 : 4;
  cuuint64_t dims[2] = {(cuuint64_t)H * D, (cuuint64_t)tokens};
  cuuint64_t strides[1] = {(cuuint64_t)H * D * es};
  cuuint32_t box[2] = {D, C};
  cuuint32_t estr[2] = {1, 1};
  return enc(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, base,
             dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
             CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Map over q or k [tokens, H, D] (bf16) as [tokens][H * D]: box = 64 channels x 64
// tokens, one 128-byte row per token, 128-byte swizzle
bool make_map_sw128(CUtensorMap* m, const void* base, int64_t tokens, int H) {
  auto enc = get_encode();
  if (!enc) return false;
  cuuint64_t dims[2] = {(cuuint64_t)H * D, (cuuint64_t)tokens};
  cuuint64_t strides[1] = {(cuuint64_t)H * D * 2};
  cuuint32_t box[2] = {64, C};
  cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_map(CUtensorMap* m, const void* base, int64_t tokens, int H, int box_tokens = C) {
  auto enc = get_encode();
  if (!enc) return false;
  cuuint64_t dims[3] = {8, (cuuint64_t)tokens, (cuuint64_t)H * (D / 8)};
  cuuint64_t strides[2] = {(cuuint64_t)H * D * 2, 16};
  cuuint32_t box[3] = {8, (cuuint32_t)box_tokens, D / 8};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

namespace {
template <bool kPre>
cudaError_t run_bf16(const FwdArgs& a, const CUtensorMap& mq, const CUtensorMap& mk,
                     const CUtensorMap& mg, const CUtensorMap& mv, const CUtensorMap& mo,
                     Bf16Params p, int64_t items) {
  cudaError_t e = cudaFuncSetAttribute(kda_prefill_bf16_kernel<kPre>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
  if (e != cudaSuccess) return e;
  // Persistent CTAs, one per SM at most: each takes work items from its launch's
  // counter until none is left.
  const int64_t sms = a.sms > 0 ? a.sms : kGb300Sms;
  auto grid = [&](int64_t work) { return (unsigned)(work < sms ? work : sms); };
  auto run = [&](int64_t work) -> cudaError_t {
    kda_prefill_bf16_kernel<kPre><<<grid(work), kThreads, SMEM_BYTES, a.stream>>>(mq, mk, mg, mv,
                                                                                  mo, p);
    return cudaGetLastError();
  };
  if (a.pplan) {
    // packed batch with the device-written plan: transitions, scan, outputs (the
    // counts are on the device; a launch with nothing to do leaves at once)
    p.pv = PlanView::at(a.pplan, a.N, a.ns_max);
    p.pstates = a.seg_ws;
    p.mode = MODE_PSEG_TRANSITION;
    if ((e = run(2 * a.H * a.ns_max)) != cudaSuccess) return e;
    if ((e = launch_segment_scan_packed(p.pv, a.seg_ws, a.H, a.ns_max, sms, a.stream)) !=
        cudaSuccess)
      return e;
    p.mode = MODE_PSEG_OUTPUT;
    return run(a.H * (a.N + a.ns_max));
  }
  const SegPlan pl = a.plan;
  if (pl.nseg < 2 || !a.seg_ws) {
    return run(items);
  }
  // long chains: segment 0 from the start state (with its outputs) beside the
  // transitions of segments 1 .. nseg-2, the scan, then the outputs of segments
  // 1 .. nseg-1
  const int64_t per = (int64_t)D * D;
  p.nseg = pl.nseg;
  p.seg_len = pl.seg_len;
  p.seg0_len = pl.seg0_len;
  p.seg_b = a.seg_ws;
  p.seg_m = a.seg_ws + items * (pl.nseg - 1) * per;
  float* seg_s = a.seg_ws + 2 * items * (pl.nseg - 1) * per;
  p.seg_s = seg_s;
  p.mode = MODE_SEG_TRANSITION;
  if ((e = run(items * (2 * pl.nseg - 3))) != cudaSuccess) return e;
  if ((e = launch_segment_scan(p.seg_m, p.seg_b, seg_s, items, pl.nseg, a.stream)) !=
      cudaSuccess)
    return e;
  p.mode = MODE_SEG_OUTPUT;
  return run(items * (pl.nseg - 1));
}
}  // namespace

cudaError_t launch_prefill_bf16(const FwdArgs& a) {
  const int64_t items = (int64_t)a.N * a.H;
  if (items == 0) return cudaSuccess;
  const int64_t tokens = a.cu ? a.T : (int64_t)a.N * a.T;
  // A map needs a non-empty tensor.  With no tokens every chain is empty and no
  // tile is loaded; map a valid state pointer instead (or skip when none).
  const void* dummy = a.h0 ? (const void*)a.h0 : (const void*)a.hT;
  if (tokens == 0 && !dummy) return cudaSuccess;
  auto pick = [&](const void* x) { return tokens > 0 ? x : dummy; };
  const int64_t map_tokens = tokens > 0 ? tokens : 1;
  CUtensorMap mq, mk, mg, mv, mo;
  if (!make_map_sw128(&mq, pick(a.q), map_tokens, a.H) ||
      !make_map_sw128(&mk, pick(a.k), map_tokens, a.H) ||
      !make_map(&mg, pick(a.pre.per_head ? a.q : a.g), map_tokens, a.H, C / 2) ||
      !make_map(&mv, pick(a.v), map_tokens, a.H) ||
      !make_out_map(&mo, tokens > 0 ? a.out : const_cast<void*>(dummy), map_tokens, a.H,
                    tokens > 0 && a.out_dtype == KDA_BF16))
    return cudaErrorInvalidValue;
  Bf16Params p;
  p.beta = static_cast<const __nv_bfloat16*>(a.beta);
  p.seqs = SeqView{a.cu, a.T};
  p.order = a.order;
  p.h0 = a.h0;
  p.out = a.out;
  p.hT = a.hT;
  p.H = a.H;
  p.nchains = (int)items;
  p.scale = a.scale;
  p.out_bf16 = a.out_dtype == KDA_BF16;
  p.status = a.status;
  p.mode = MODE_CHAIN;
  p.nseg = 1;
  p.seg_len = p.seg0_len = 0;
  p.seg_b = p.seg_m = nullptr;
  p.seg_s = nullptr;
  p.ckpt = a.ckpt;
  p.ckpt_off = a.ckpt_off;
  p.ckpt_rows = a.ckpt_rows;
  p.ckpt_interval = a.ckpt_interval > 0 ? a.ckpt_interval : 1;
  p.pre = a.pre;
  p.g = static_cast<const __nv_bfloat16*>(a.g);
  p.pv = PlanView{};
  p.pstates = nullptr;
  if (a.pre.l2 || a.pre.gate || a.pre.beta || a.pre.per_head)
    return run_bf16<true>(a, mq, mk, mg, mv, mo, p, items);
  return run_bf16<false>(a, mq, mk, mg, mv, mo, p, items);
}

}  // namespace kda
