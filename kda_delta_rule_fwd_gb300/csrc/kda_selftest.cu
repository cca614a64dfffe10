// Self-test of the bounded device waits: a kernel waits on an mbarrier that
// nothing ever arrives at, gives up after a short budget, latches
// KDA_ERR_DEVICE_TIMEOUT in the caller's workspace status word and returns.
// It exercises the same wait helper the tensor-core prefill uses, so a test
// can check that a wait that runs out is reported to the host and leaves the
// CUDA context usable -- without faulting or hanging the GPU.
#include "kda_internal.cuh"
#include "kda_sm100.cuh"

namespace {

__global__ void kda_bounded_wait_selftest_kernel(unsigned int* status, long long budget) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    kda::sm100::mbar_init(&bar, 1);
    kda::sm100::fence_barrier_init();
  }
  __syncthreads();
  // phase 0 never completes: no thread arrives and no copy is attached
  if (threadIdx.x == 0 && !kda::sm100::mbar_wait(&bar, 0, budget))
    kda::latch_status(status, KDA_ERR_DEVICE_TIMEOUT);
}

}  // namespace

extern "C" kda_status kda_selftest_bounded_wait(void* workspace, void* stream) {
  if (!workspace || ((uintptr_t)workspace % 256) != 0) return KDA_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(workspace, 0, kda::kWsHeader, s) != cudaSuccess) return KDA_ERR_CUDA;
  // about 1 ms at 2 GHz
  kda_bounded_wait_selftest_kernel<<<1, 32, 0, s>>>(static_cast<unsigned int*>(workspace),
                                                    2000000ll);
  return cudaGetLastError() == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}
