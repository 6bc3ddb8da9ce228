// Host-side launch plumbing shared by the C ABI and the kernel instantiation units.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include "attn_bwd_kernel.cuh"
#include "attn_fwd_kernel.cuh"

namespace gb300 {

struct LaunchArgs {
  CUtensorMap tm_q, tm_k, tm_v;
  AttnParams params;
  int num_sms;
  bool dependent;   // launch as a programmatic dependent of the previous kernel on the stream
};

// Per-instance launcher: grid = min(work tiles, SMs), one persistent CTA per SM. SPLIT selects
// the split-KV (decode) mode of the kernel, VARLEN the ragged-batch mode driven by a tile plan.
template <int D, bool CAUSAL, bool FP8, bool SPLIT = false, bool VARLEN = false>
cudaError_t launch_attn_fwd(LaunchArgs& a, cudaStream_t stream);

// Backward pass (attn_bwd.cu): preprocess, then the dK/dV and dQ kernels, on one stream.
struct BwdLaunchArgs {
  CUtensorMap tm_q, tm_k, tm_v, tm_do;
  BwdParams params;          // n_tiles is set per kernel
  const void* o;             // bf16 [B, N, H, D]
  const void* dout;          // bf16 [B, N, H, D]
  const float* lse;          // [B, H, N]
  float* nlse2;              // workspace [B, H, Np]
  float* dd;                 // workspace [B, H, Np]
  int num_sms;
};
cudaError_t launch_attn_bwd(BwdLaunchArgs& a, int d, bool causal, cudaStream_t stream);

// Builds the ragged-batch tile plan (varlen_plan.cu): one CTA on the stream.
cudaError_t launch_varlen_plan(const int* cu_q, const int* cu_k, int B, int H, int rows_per_tile, bool causal,
                               int total_q, int total_k, int capacity, int* plan, cudaStream_t stream);

// Split-KV combine: merges the n_splits normalized partial results (part_o fp32
// [S, B, H, Nq, D], part_lse [S, B, H, Nq]) into o (bf16 [B, Nq, H, D]) and lse ([B, H, Nq]).
cudaError_t launch_splitkv_combine(const float* part_o, const float* part_lse, void* o, float* lse, int S, int B,
                                   int H, int Nq, int D, int num_sms, cudaStream_t stream);

// e4m3 block quantisation of bf16 rows (fp8_quantize.cu). Rows of one (batch, head) are cut into
// spans of span rows (span = chunk_rows when blocks have at most 128 rows, else block_rows), and
// each span into cps chunks of up to chunk_rows rows; one chunk is one TMA load. A chunk holds
// chunk_rows / grp_rows groups of rows, each inside one block. tm_x: 4-D map of x (d, N, Hx, B),
// box (64, chunk_rows, 1, 1), 128-byte swizzle.
struct QuantLaunch {
  CUtensorMap tm_x;
  uint8_t* x8;              // [B, N, Hx, d] codes
  float* descale;           // [B, Hx, nblk]
  const float* signs;       // d values or null
  int B, N, Hx, d, block_rows, nblk;
  int span, cps, nspan, chunk_rows, grp_rows;
  uint32_t* status;
  unsigned long long timeout_ns;
  int num_sms;
};
cudaError_t launch_quantize_e4m3(const QuantLaunch& q, cudaStream_t stream);

// Rows of queries one CTA work tile covers for head dim d (two 128-row tiles for d <= 128).
inline int rows_per_work_tile(int d) { return d <= 128 ? 256 : 128; }

// Non-causal prefill: work tiles of the last wave whose KV range is halved across two launches
// (0: none). The last wave of `tiles` over `sms` persistent CTAs holds 1..sms tiles; when it would
// leave more than half of the SMs idle, its tiles are cut in two at KV tile n_kvt / 2, the second
// halves running as a dependent launch on the idle SMs. Each half keeps at least eight KV tiles,
// so the halves' own pipeline fill and the merge stay small beside what they save.
inline int halved_tail_tiles(long long tiles, int n_kvt, int sms, bool causal) {
  if (causal || n_kvt < 16 || sms < 2 || tiles < 1) return 0;
  const long long rem = tiles - (tiles - 1) / sms * sms;
  return rem <= sms / 2 ? (int)rem : 0;
}
// KV tile at which a halved tile is cut: the middle. The second launch starts cold and ends with
// the merge, which waits for the whole first grid; on the shapes measured (d = 64, 128, 256, bf16
// and e4m3) moving the cut by up to n_kvt / 6 either way saved at most 1% and mostly cost time.
inline int halved_tail_cut(int n_kvt) { return n_kvt / 2; }
// Split-KV mode always runs one 128-row Q tile per CTA.
inline int rows_per_split_work_tile(int) { return 128; }

#define GB300_DECLARE_LAUNCH(D, CAUSAL, FP8) \
  extern template cudaError_t launch_attn_fwd<D, CAUSAL, FP8, false, false>(LaunchArgs&, cudaStream_t);
#define GB300_DECLARE_SPLIT(D, FP8) \
  extern template cudaError_t launch_attn_fwd<D, false, FP8, true, false>(LaunchArgs&, cudaStream_t);
#define GB300_DECLARE_VARLEN(D, CAUSAL, FP8) \
  extern template cudaError_t launch_attn_fwd<D, CAUSAL, FP8, false, true>(LaunchArgs&, cudaStream_t);

GB300_DECLARE_LAUNCH(64, false, false)
GB300_DECLARE_LAUNCH(64, true, false)
GB300_DECLARE_LAUNCH(128, false, false)
GB300_DECLARE_LAUNCH(128, true, false)
GB300_DECLARE_LAUNCH(256, false, false)
GB300_DECLARE_LAUNCH(256, true, false)
GB300_DECLARE_LAUNCH(128, false, true)
GB300_DECLARE_LAUNCH(128, true, true)
GB300_DECLARE_LAUNCH(256, false, true)
GB300_DECLARE_LAUNCH(256, true, true)
GB300_DECLARE_SPLIT(64, false)
GB300_DECLARE_SPLIT(128, false)
GB300_DECLARE_SPLIT(256, false)
GB300_DECLARE_SPLIT(128, true)
GB300_DECLARE_SPLIT(256, true)
GB300_DECLARE_VARLEN(64, false, false)
GB300_DECLARE_VARLEN(64, true, false)
GB300_DECLARE_VARLEN(128, false, false)
GB300_DECLARE_VARLEN(128, true, false)
GB300_DECLARE_VARLEN(256, false, false)
GB300_DECLARE_VARLEN(256, true, false)
GB300_DECLARE_VARLEN(128, false, true)
GB300_DECLARE_VARLEN(128, true, true)
GB300_DECLARE_VARLEN(256, false, true)
GB300_DECLARE_VARLEN(256, true, true)

}  // namespace gb300
