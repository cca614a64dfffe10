// Segment scan of the long-chain split: S_{p+1} = M_p S_p + b_p along each
// chain, in float32.  The state maps of a chain's segments compose
// associatively ("Kimi K3 模型结构（7）：结构决定系统", section 上下文并行: each
// part contributes a local transition matrix and a zero-start state, combined
// by a prefix scan); the segments here are on one GPU.
//
// The recursion is separable by state columns: column j of S_{p+1} is
// M_p (column j of S_p) + (column j of b_p).  Each CTA therefore owns 16 of
// the 128 columns of one chain's state for the whole scan, and a chain's eight
// column blocks run in parallel with no exchange.  Per step a CTA stages M_p in
// shared memory (rows padded to 129 floats, so the threads reading one column
// of it hit distinct banks) and each thread forms 8 entries of its block:
// 128 x 16 x 128 multiply-adds per CTA and step.
#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int D = 128;
constexpr int kCols = 16;               // state columns per CTA
constexpr int kBlocks = D / kCols;      // CTAs per chain
constexpr int kThreads = 256;           // thread t: row t / 2, columns 8 (t % 2) ..
constexpr int kMld = D + 1;             // padded row stride of M_p in shared memory
constexpr size_t kSmem = ((size_t)D * kMld + (size_t)D * kCols) * sizeof(float);
static_assert(kThreads == 2 * D && kCols == 16, "thread mapping");

// One chain's column block cb: S_0 = h0 (or 0) to Sp[0]; S_{p+1} = M_p S_p + b_p to
// Sp[p+1], with M_p = Mp + p D^2, b_p = bp + p D^2, S_p = Sp + p D^2 (row-major D x D).
__device__ void scan_block(const float* __restrict__ h0c, const float* __restrict__ Mp,
                           const float* __restrict__ bp, float* __restrict__ Sp, int nseg,
                           int cb, float* sm) {
  float* Ms = sm;             // M_p [D][kMld]
  float* Ss = sm + D * kMld;  // this block of S_p [D][kCols]
  const int tid = threadIdx.x, i = tid >> 1, j0 = (tid & 1) * 8;
  const int c0 = cb * kCols;
  for (int x = tid; x < D * kCols; x += kThreads) {
    const int r = x / kCols, c = x % kCols;
    const float v = h0c ? h0c[(int64_t)r * D + c0 + c] : 0.f;
    Ss[x] = v;
    Sp[(int64_t)r * D + c0 + c] = v;
  }
  for (int sp = 0; sp + 1 < nseg; ++sp) {
    const float* M = Mp + (int64_t)sp * D * D;
    const float* b = bp + (int64_t)sp * D * D;
    __syncthreads();  // the previous step is done with Ms
    for (int x = tid * 4; x < D * D; x += kThreads * 4) {
      const float4 m = *reinterpret_cast<const float4*>(M + x);
      float* dst = Ms + (x / D) * kMld + (x % D);
      dst[0] = m.x;
      dst[1] = m.y;
      dst[2] = m.z;
      dst[3] = m.w;
    }
    float acc[8];
    {
      const float4 b0 = *reinterpret_cast<const float4*>(b + (int64_t)i * D + c0 + j0);
      const float4 b1 = *reinterpret_cast<const float4*>(b + (int64_t)i * D + c0 + j0 + 4);
      acc[0] = b0.x; acc[1] = b0.y; acc[2] = b0.z; acc[3] = b0.w;
      acc[4] = b1.x; acc[5] = b1.y; acc[6] = b1.z; acc[7] = b1.w;
    }
    __syncthreads();  // M_p staged; S_p's block is in place
#pragma unroll 4
    for (int k = 0; k < D; ++k) {
      const float m = Ms[i * kMld + k];
      const float4 s0 = *reinterpret_cast<const float4*>(Ss + k * kCols + j0);
      const float4 s1 = *reinterpret_cast<const float4*>(Ss + k * kCols + j0 + 4);
      acc[0] = fmaf(m, s0.x, acc[0]);
      acc[1] = fmaf(m, s0.y, acc[1]);
      acc[2] = fmaf(m, s0.z, acc[2]);
      acc[3] = fmaf(m, s0.w, acc[3]);
      acc[4] = fmaf(m, s1.x, acc[4]);
      acc[5] = fmaf(m, s1.y, acc[5]);
      acc[6] = fmaf(m, s1.z, acc[6]);
      acc[7] = fmaf(m, s1.w, acc[7]);
    }
    __syncthreads();  // every thread is done reading S_p
    float* out = Sp + (int64_t)(sp + 1) * D * D + (int64_t)i * D + c0 + j0;
    *reinterpret_cast<float4*>(Ss + i * kCols + j0) = make_float4(acc[0], acc[1], acc[2], acc[3]);
    *reinterpret_cast<float4*>(Ss + i * kCols + j0 + 4) =
        make_float4(acc[4], acc[5], acc[6], acc[7]);
    *reinterpret_cast<float4*>(out) = make_float4(acc[0], acc[1], acc[2], acc[3]);
    *reinterpret_cast<float4*>(out + 4) = make_float4(acc[4], acc[5], acc[6], acc[7]);
  }
}

// Fixed-length batches: CTA (chain, column block); every chain nseg segments.
// Segment 0 ran from the chain's true start state, so b_0 is S_1 itself and the
// recursion starts there: S_{p+1} = M_p S_p + b_p for p = 1 .. nseg-2 (M_0 is not
// formed; S_0's slot is not used).
__global__ void __launch_bounds__(kThreads)
kda_segment_scan_kernel(const float* __restrict__ seg_m, const float* __restrict__ seg_b,
                        float* __restrict__ seg_s, int nseg) {
  extern __shared__ __align__(16) float sm[];
  const int64_t chain = blockIdx.x / kBlocks, per = (int64_t)(nseg - 1) * D * D;
  scan_block(seg_b + chain * per, seg_m + chain * per + D * D, seg_b + chain * per + D * D,
             seg_s + chain * nseg * D * D + D * D, nseg - 1, blockIdx.x % kBlocks, sm);
}

// Packed batches: (split sequence, head, column block) of the plan, grid-stride.
// As for fixed-length batches, segment 0 ran from the sequence's start state and
// b_0 is S_1: S_{p+1} = M_p S_p + b_p for p = 1 .. nseg-2.
__global__ void __launch_bounds__(kThreads)
kda_segment_scan_packed_kernel(PlanView pv, float* __restrict__ states, int H) {
  extern __shared__ __align__(16) float sm[];
  const int64_t work = (int64_t)pv.hdr->n_split * H * kBlocks;
  for (int64_t w = blockIdx.x; w < work; w += gridDim.x) {
    const int cb = (int)(w % kBlocks);
    const int64_t chain = w / kBlocks;
    const int h = (int)(chain % H), si = (int)(chain / H);
    const int n = pv.split[si], nseg = pv.nseg[n];
    float* base = states + ((int64_t)pv.slot[n] * H + (int64_t)h * (3 * nseg - 2)) * D * D;
    scan_block(base, base + (int64_t)nseg * D * D, base + (int64_t)D * D,
               base + (int64_t)(2 * (nseg - 1) + 1) * D * D, nseg - 1, cb, sm);
    __syncthreads();  // shared memory is reused by the next block
  }
}

}  // namespace

cudaError_t launch_segment_scan(const float* seg_m, const float* seg_b, float* seg_s,
                                int64_t chains, int nseg, cudaStream_t stream) {
  cudaError_t e = cudaFuncSetAttribute(kda_segment_scan_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmem);
  if (e != cudaSuccess) return e;
  kda_segment_scan_kernel<<<(unsigned)(chains * kBlocks), kThreads, kSmem, stream>>>(
      seg_m, seg_b, seg_s, nseg);
  return cudaGetLastError();
}

cudaError_t launch_segment_scan_packed(PlanView pv, float* states, int H, int64_t ns_max,
                                       int64_t sms, cudaStream_t stream) {
  cudaError_t e = cudaFuncSetAttribute(kda_segment_scan_packed_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmem);
  if (e != cudaSuccess) return e;
  // (at most ns_max / 2 sequences are split; three CTAs fit an SM)
  const int64_t work = (ns_max / 2 + 1) * H * kBlocks, cap = 3 * (sms > 0 ? sms : kGb300Sms);
  kda_segment_scan_packed_kernel<<<(unsigned)(work < cap ? work : cap), kThreads, kSmem,
                                   stream>>>(pv, states, H);
  return cudaGetLastError();
}

}  // namespace kda
