// Split-KV (decode) instances of the attention forward: bf16 d = 64, 128, 256 and e4m3 d = 64 and
// 128 (e4m3 d = 256 is built with its prefill instances).
#include "launch_impl.cuh"

namespace gb300 {
template cudaError_t launch_attn_fwd<64, false, false, true, false>(LaunchArgs&, cudaStream_t);
template cudaError_t launch_attn_fwd<128, false, false, true, false>(LaunchArgs&, cudaStream_t);
template cudaError_t launch_attn_fwd<256, false, false, true, false>(LaunchArgs&, cudaStream_t);
template cudaError_t launch_attn_fwd<64, false, true, true, false>(LaunchArgs&, cudaStream_t);
template cudaError_t launch_attn_fwd<128, false, true, true, false>(LaunchArgs&, cudaStream_t);
}  // namespace gb300
