// Ragged-batch (varlen) instances of the attention forward, e4m3, head dim 64 (non-causal and
// causal).
#include "launch_impl.cuh"

namespace gb300 {
template cudaError_t launch_attn_fwd<64, false, true, false, true>(LaunchArgs&, cudaStream_t);
template cudaError_t launch_attn_fwd<64, true, true, false, true>(LaunchArgs&, cudaStream_t);
}  // namespace gb300
