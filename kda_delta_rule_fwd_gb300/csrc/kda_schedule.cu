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

}  // namespace

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
