// Ragged-batch (varlen) instances of the attention forward, bf16 head dims 64 and 256,
// non-causal and causal.
#include "launch_impl.cuh"

namespace gb300 {
template cudaError_t launch_attn_fwd<64, false, false, false, true>(LaunchArgs&, cudaStream_t);
template cudaError_t launch_attn_fwd<64, true, false, false, true>(LaunchArgs&, cudaStream_t);
template cudaError_t launch_attn_fwd<256, false, false, false, true>(LaunchArgs&, cudaStream_t);
template cudaError_t launch_attn_fwd<256, true, false, false, true>(LaunchArgs&, cudaStream_t);
}  // namespace gb300
