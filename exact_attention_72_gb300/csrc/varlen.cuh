// Ragged batches (cumulative sequence offsets): the work-tile plan shared by the plan builder and
// the attention kernel's varlen mode.
//
// "flash-attention-3" (ai.thesatyajit.com), "Five schedulers" and "What is actually in the box":
// a varlen persistent scheduler exists because serving traffic is ragged, and the scheduler's
// metadata is computed once so a serving loop can reuse it across calls.
//
// Plan layout (32-bit words, device memory written by attn_varlen_plan):
//   [0] number of work tiles   [1] B (-1: invalid offsets)   [2] H   [3] query rows per work tile
//   [4] causal   [5] word offset of the tile list   [6] total query rows   [7] total key rows
//   [8 .. 8 + B]   tile prefix: work tiles of sequences 0 .. b-1 (builder scratch)
//   tile list: one (b, h << 16 | m) pair of words per work tile, longest first.
#pragma once
#include <cstdint>

namespace gb300 {

constexpr int kPlanHeaderWords = 8;
constexpr uint32_t kStatusBadPlan = 0x20000000u | 12u;   // device-side check of a plan failed

// 128-key KV tiles that the 128 query rows from pos0 of a sequence with nq queries and nk keys
// visit. Causal masking is bottom-right aligned: query i sees keys j <= i + (nk - nq).
__host__ __device__ inline int varlen_kv_tiles(int pos0, int nq, int nk, bool causal) {
  if (pos0 >= nq || nk <= 0) return 0;
  const int n_kvt = (nk + 127) / 128;
  if (!causal) return n_kvt;
  const int last_row = (pos0 + 127 < nq - 1 ? pos0 + 127 : nq - 1) + (nk - nq);
  if (last_row < 0) return 0;
  const int n = last_row / 128 + 1;
  return n < n_kvt ? n : n_kvt;
}

// Word offset of the tile list for B sequences (8-byte aligned).
__host__ __device__ inline int plan_tiles_offset(int B) { return (kPlanHeaderWords + B + 1 + 1) & ~1; }

}  // namespace gb300
