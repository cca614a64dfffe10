// Internal declarations shared by the CUDA translation units of the KDA library.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kda.h"

namespace kda {

// Device status word: first 4 bytes of the caller's workspace.  Kernels latch
// the first error with atomicCAS(0 -> code) and never trap.
struct DevStatus {
  unsigned int code;
};

__device__ __forceinline__ void latch_status(unsigned int* status, unsigned int code) {
  if (status) atomicCAS(status, 0u, code);
}

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

// Where a sequence's tokens live: global token offset and length.  A fixed
// batch (no cu_seqlens) puts sequence n at n*T.  Packed batches read the
// validated cu_seqlens.
struct SeqView {
  const int32_t* cu;   // device [N+1] or nullptr
  int64_t T;           // fixed: tokens per sequence; packed: total tokens
  __device__ __forceinline__ void get(int n, int64_t& start, int64_t& len) const {
    if (cu) {
      int64_t a = cu[n], b = cu[n + 1];
      a = a < 0 ? 0 : (a > T ? T : a);
      b = b < a ? a : (b > T ? T : b);
      start = a;
      len = b - a;
    } else {
      start = (int64_t)n * T;
      len = T;
    }
  }
};

// Workspace layout (bytes):
//   [0, 256)            status word and counters
//   [256, 256 + 4*Npad) sequence order for the packed-batch scheduler
constexpr size_t kWsHeader = 256;
inline size_t ws_order_bytes(int64_t n) { return (size_t)((n + 63) / 64) * 64 * 4; }

// ---------------------------------------------------------------------------
// launchers (each returns cudaSuccess or the launch error)
// ---------------------------------------------------------------------------
struct FwdArgs {
  const void *q, *k, *v, *g, *beta;
  const int32_t* cu;
  const float* h0;
  void* out;
  float* hT;
  int64_t T;        // tokens per sequence (fixed) or total tokens (packed)
  int32_t N, H, D;  // sequences, heads, head dim (dk == dv)
  float scale;
  kda_dtype in_dtype, out_dtype;
  unsigned int* status;
  const int32_t* order;  // scheduler output: sequences longest first (packed), or nullptr
  cudaStream_t stream;
};

cudaError_t launch_schedule(const FwdArgs& a, int32_t* order_out);
cudaError_t launch_prefill_f32(const FwdArgs& a);
cudaError_t launch_prefill_bf16(const FwdArgs& a);

struct DecodeArgs {
  const void *q, *k, *v, *g, *beta;
  float* state;
  void* out;
  int32_t B, Tstep, H, D;
  float scale;
  kda_dtype in_dtype, out_dtype;
  cudaStream_t stream;
};

cudaError_t launch_decode(const DecodeArgs& a);

}  // namespace kda
