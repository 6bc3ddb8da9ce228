// FP8 e4m3 instances of the attention forward, head dim 128 (non-causal and causal).
#include "launch_impl.cuh"

namespace gb300 {
template cudaError_t launch_attn_fwd<128, false, true, false, false>(LaunchArgs&, cudaStream_t);
template cudaError_t launch_attn_fwd<128, true, true, false, false>(LaunchArgs&, cudaStream_t);
}  // namespace gb300
