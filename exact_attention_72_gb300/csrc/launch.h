// Host-side launch plumbing shared by the C ABI and the kernel instantiation units.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include "attn_fwd_kernel.cuh"

namespace gb300 {

struct LaunchArgs {
  CUtensorMap tm_q, tm_k, tm_v;
  AttnParams params;
  int num_sms;
};

// Per-instance launcher: grid = min(work tiles, SMs), one persistent CTA per SM. SPLIT selects
// the split-KV (decode) mode of the kernel.
template <int D, bool CAUSAL, bool FP8, bool SPLIT = false>
cudaError_t launch_attn_fwd(LaunchArgs& a, cudaStream_t stream);

// Split-KV combine: merges the n_splits normalized partial results (part_o fp32
// [S, B, H, Nq, D], part_lse [S, B, H, Nq]) into o (bf16 [B, Nq, H, D]) and lse ([B, H, Nq]).
cudaError_t launch_splitkv_combine(const float* part_o, const float* part_lse, void* o, float* lse, int S, int B,
                                   int H, int Nq, int D, int num_sms, cudaStream_t stream);

// Rows of queries one CTA work tile covers for head dim d (two 128-row tiles for d <= 128).
inline int rows_per_work_tile(int d) { return d <= 128 ? 256 : 128; }

#define GB300_DECLARE_LAUNCH(D, CAUSAL, FP8) \
  extern template cudaError_t launch_attn_fwd<D, CAUSAL, FP8, false>(LaunchArgs&, cudaStream_t);
#define GB300_DECLARE_SPLIT(D, FP8) \
  extern template cudaError_t launch_attn_fwd<D, false, FP8, true>(LaunchArgs&, cudaStream_t);

GB300_DECLARE_LAUNCH(64, false, false)
GB300_DECLARE_LAUNCH(64, true, false)
GB300_DECLARE_LAUNCH(128, false, false)
GB300_DECLARE_LAUNCH(128, true, false)
GB300_DECLARE_LAUNCH(256, false, false)
GB300_DECLARE_LAUNCH(256, true, false)
GB300_DECLARE_LAUNCH(128, false, true)
GB300_DECLARE_LAUNCH(128, true, true)
GB300_DECLARE_SPLIT(64, false)
GB300_DECLARE_SPLIT(128, false)
GB300_DECLARE_SPLIT(256, false)
GB300_DECLARE_SPLIT(128, true)

}  // namespace gb300
