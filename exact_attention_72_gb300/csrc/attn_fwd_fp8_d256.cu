// FP8 e4m3 instances of the attention forward, head dim 256: non-causal and causal prefill, and
// split-KV decode.
#include "launch_impl.cuh"

namespace gb300 {
template cudaError_t launch_attn_fwd<256, false, true, false, false>(LaunchArgs&, cudaStream_t);
template cudaError_t launch_attn_fwd<256, true, true, false, false>(LaunchArgs&, cudaStream_t);
template cudaError_t launch_attn_fwd<256, false, true, true, false>(LaunchArgs&, cudaStream_t);
}  // namespace gb300
