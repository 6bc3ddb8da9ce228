// FP8 e4m3 instances of the attention forward, head dim 64 (non-causal and causal): 64-byte rows,
// stored and read with the 64-byte swizzle.
#include "launch_impl.cuh"

namespace gb300 {
template cudaError_t launch_attn_fwd<64, false, true, false, false>(LaunchArgs&, cudaStream_t);
template cudaError_t launch_attn_fwd<64, true, true, false, false>(LaunchArgs&, cudaStream_t);
}  // namespace gb300
