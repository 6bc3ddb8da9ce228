// Ragged-batch (varlen) instances of the attention forward, head dim 128: bf16 and e4m3,
// non-causal and causal.
#include "launch_impl.cuh"

namespace gb300 {
template cudaError_t launch_attn_fwd<128, false, false, false, true>(LaunchArgs&, cudaStream_t);
template cudaError_t launch_attn_fwd<128, true, false, false, true>(LaunchArgs&, cudaStream_t);
template cudaError_t launch_attn_fwd<128, false, true, false, true>(LaunchArgs&, cudaStream_t);
template cudaError_t launch_attn_fwd<128, true, true, false, true>(LaunchArgs&, cudaStream_t);
}  // namespace gb300
