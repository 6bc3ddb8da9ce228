// Host-side launch plumbing shared by the C ABI and the kernel instantiation units.
#pragma once
#include <algorithm>
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
  int x8_v8;                // x8 is 32-byte aligned: rows of codes go out in 32-byte stores
  uint32_t* status;
  unsigned long long timeout_ns;
  int num_sms;
};
cudaError_t launch_quantize_e4m3(const QuantLaunch& q, cudaStream_t stream);

// Rows of queries one CTA work tile covers for head dim d (two 128-row tiles for d <= 128).
inline int rows_per_work_tile(int d) { return d <= 128 ? 256 : 128; }

// Non-causal prefill over `tiles` work tiles of n_kvt KV tiles each on `sms` persistent CTAs:
// which tiles have their key range cut between the first launch and a dependent second launch
// (AttnParams::tail_mode). Sets tail_mode, tail_first, tail_kvt, bal_main, bal_wtail and the
// second launch's units (tail_tab) in p, and returns the unit count (0: one launch, tail_mode 0).
//  * shares (bf16 at d <= 128): more than one wave, not a whole number of waves, at least 8 KV
//    tiles: whole rounds of sms tiles go round-robin except the last whole one; the KV tiles of
//    the tiles after them are dealt in sms equal shares (tail_mode 3; each share is at least
//    n_kvt long). Every CTA then does the same number of KV tiles over the two launches instead
//    of some CTAs one tile more than others. A share boundary inside a tile makes a second-launch
//    unit (the rest of that tile). Units go longest first: the second launch's CTAs take SMs in
//    the order the first launch's CTAs leave them, and the CTA whose share begins with the
//    longest rest has the least work in the first launch. (e4m3 and d = 256 run their tiles in
//    fewer, cheaper steps; there the extra partial tile per CTA cost what the balance saved.)
//  * otherwise, a last wave that leaves more than half of the SMs idle, with at least 16 KV
//    tiles: its tiles are cut at the middle, n_kvt / 2 (tail_mode 1). Each half keeps at least
//    eight KV tiles, so the halves' own pipeline fill and the merge stay small beside what they
//    save; moving the cut by up to n_kvt / 6 either way saved at most 1% on the shapes measured.
inline int plan_tail(AttnParams& p, long long tiles, int n_kvt, int sms, bool causal, bool shares) {
  p.tail_mode = 0;
  p.tail_first = 0;
  p.tail_kvt = n_kvt;
  p.bal_main = 0;
  p.bal_wtail = 0;
  if (causal || sms < 2 || tiles < 1 || n_kvt < 1) return 0;
  if (!(shares && tiles > sms && tiles % sms != 0 && n_kvt >= 8 && sms - 1 <= kMaxTailUnits)) {
    if (n_kvt < 16) return 0;
    const long long rem = tiles - (tiles - 1) / sms * sms;   // tiles of the last wave
    if (rem > sms / 2 || rem > kMaxTailUnits) return 0;
    p.tail_mode = 1;
    p.tail_first = (int)(tiles - rem);
    p.tail_kvt = n_kvt / 2;
    for (int u = 0; u < (int)rem; ++u) p.tail_tab[u] = make_int2(p.tail_first + u, p.tail_kvt);
    return (int)rem;
  }
  const long long main_tiles = (tiles / sms - 1) * sms;
  const long long K = n_kvt, W = (tiles - main_tiles) * K;
  struct Unit { int tile, j0, share; };
  Unit u[kMaxTailUnits];
  int n = 0;
  for (int c = 1; c < sms; ++c) {
    const long long s0 = (long long)c * W / sms;
    if (s0 % K != 0) u[n++] = Unit{(int)(main_tiles + s0 / K), (int)(s0 % K), c};
  }
  std::sort(u, u + n, [&](const Unit& a, const Unit& b) {
    return a.j0 != b.j0 ? a.j0 < b.j0 : a.share < b.share;   // longest rest first
  });
  for (int i = 0; i < n; ++i) p.tail_tab[i] = make_int2(u[i].tile, u[i].j0);
  p.tail_mode = 3;
  p.bal_main = (int)main_tiles;
  p.bal_wtail = W;
  return n;
}
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
GB300_DECLARE_LAUNCH(64, false, true)
GB300_DECLARE_LAUNCH(64, true, true)
GB300_DECLARE_LAUNCH(128, false, true)
GB300_DECLARE_LAUNCH(128, true, true)
GB300_DECLARE_LAUNCH(256, false, true)
GB300_DECLARE_LAUNCH(256, true, true)
GB300_DECLARE_SPLIT(64, false)
GB300_DECLARE_SPLIT(128, false)
GB300_DECLARE_SPLIT(256, false)
GB300_DECLARE_SPLIT(64, true)
GB300_DECLARE_SPLIT(128, true)
GB300_DECLARE_SPLIT(256, true)
GB300_DECLARE_VARLEN(64, false, false)
GB300_DECLARE_VARLEN(64, true, false)
GB300_DECLARE_VARLEN(128, false, false)
GB300_DECLARE_VARLEN(128, true, false)
GB300_DECLARE_VARLEN(256, false, false)
GB300_DECLARE_VARLEN(256, true, false)
GB300_DECLARE_VARLEN(64, false, true)
GB300_DECLARE_VARLEN(64, true, true)
GB300_DECLARE_VARLEN(128, false, true)
GB300_DECLARE_VARLEN(128, true, true)
GB300_DECLARE_VARLEN(256, false, true)
GB300_DECLARE_VARLEN(256, true, true)

}  // namespace gb300
