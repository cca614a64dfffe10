// Placeholder until the tensor-core bf16 prefill lands: bf16 inputs run through
// the float32 SIMT chunk kernel.
#include "kda_internal.cuh"

namespace kda {
cudaError_t launch_prefill_bf16(const FwdArgs& a) { return launch_prefill_f32(a); }
}  // namespace kda
