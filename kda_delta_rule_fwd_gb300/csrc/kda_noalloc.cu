// kda_fwd_noalloc: the prefill entry point for callers that cannot allocate
// device memory themselves.
//
// kda_fwd needs a caller-provided workspace (a status word plus the packed-batch
// scheduler's sequence order).  Some callers have no way to provide one: code
// whose device memory is planned in full by a host framework before it runs
// and that may not request more at call time, or bindings that cannot reach a
// device allocator at all.  This variant runs the same kernels with their
// scratch in a fixed-size array that lives in the library's own device
// memory, so the caller passes only inputs and outputs.
//
// The array is a file-scope __device__ variable: every GPU that loads the
// library holds it until the process exits.  In host code its name is only a
// host-side stand-in, so its device address is looked up once per device with
// cudaGetSymbolAddress (on the first call made while that device is current)
// and cached.  All calls on a device share the one array.
#include <mutex>

#include "kda_internal.cuh"

namespace {

constexpr int kNoAllocMaxSeqs = 16384;
constexpr size_t kNoAllocBytes = kda::kWsHeader + (size_t)kNoAllocMaxSeqs * sizeof(int32_t);
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_kda_noalloc_scratch[kNoAllocBytes];

std::mutex g_mu;
void* g_scratch_addr[kMaxDevices];

}  // namespace

extern "C" kda_status kda_fwd_noalloc(const kda_shape* s, const void* q, const void* k,
                                      const void* v, const void* g, const void* beta,
                                      const int32_t* cu_seqlens, const float* h0, void* out,
                                      float* hT, unsigned int* status_out, void* stream) {
  if (!s) return KDA_ERR_INVALID_ARG;
  if (cu_seqlens && s->num_seqs > kNoAllocMaxSeqs) return KDA_ERR_UNSUPPORTED;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return KDA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return KDA_ERR_UNSUPPORTED;
  void* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_addr[dev]) {
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g_kda_noalloc_scratch) != cudaSuccess || !p)
        return KDA_ERR_CUDA;
      g_scratch_addr[dev] = p;
    }
    scratch = g_scratch_addr[dev];
  }
  const kda_status st = kda_fwd(s, q, k, v, g, beta, cu_seqlens, h0, out, hT, scratch,
                                kNoAllocBytes, stream);
  if (st != KDA_OK) return st;
  if (status_out &&
      cudaMemcpyAsync(status_out, scratch, sizeof(unsigned int), cudaMemcpyDeviceToDevice,
                      static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return KDA_ERR_CUDA;
  return KDA_OK;
}
