// bf16 instances of the attention forward, head dim 64 (non-causal and causal).
#include "launch_impl.cuh"

namespace gb300 {
template cudaError_t launch_attn_fwd<64, false, false, false, false>(LaunchArgs&, cudaStream_t);
template cudaError_t launch_attn_fwd<64, true, false, false, false>(LaunchArgs&, cudaStream_t);
}  // namespace gb300
