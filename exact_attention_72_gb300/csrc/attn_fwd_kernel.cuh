// Fused exact-attention forward for sm_103a: O = softmax(scale * Q K^T [+ causal mask]) V and
// the per-row log-sum-exp, computed tile by tile with the online softmax so the N x N score
// matrix never reaches global memory.
//
// The algorithm is the one the pages describe (tile the computation and keep a running max
// and sum per row: "flash-attention-3" (ai.thesatyajit.com), opening paragraph; the consumer
// does WGMMA(Q, K^T), rescale / exp / rowmax / rowsum, then WGMMA(P, V): "Lecture 9 — Hopper /
// FlashAttention-3 / FlashAttention-4", "Warp specialisation in FA3"). The schedule is new and
// written for Blackwell's tcgen05 tensor cores:
//
//   * one persistent CTA per SM walks work tiles (batch, head, block of NQ x 128 query rows);
//     causal work is ordered longest first ("flash-attention-3", "Five schedulers": the
//     longest-processing-time heuristic; "Hopper" tag page, section 9.2 title);
//   * warp LOAD issues TMA copies: Q once per work tile, then K_j and V_j through a ring of
//     NS shared-memory stages guarded by full/empty mbarriers ("FlashAttention-3 Deep Dive"
//     (mojostudio.in), section 2, the producer's multi-stage TMA pipeline with expected
//     transaction bytes);
//   * warp MMA (one thread) issues tcgen05.mma: S = Q K_j^T into tensor memory (TMEM), and
//     O += P V_j with P read from TMEM and V from shared memory. With two Q tiles a warp of its
//     own issues the S products: at d = 64 into three rotating TMEM buffers that P aliases
//     (AttnCfg::S3), at d = 128 (bf16 and e4m3) into one buffer both tiles share, P having a TMEM
//     area of its own (AttnCfg::S1);
//   * one softmax warpgroup per Q tile (one thread per query row) reads S from TMEM, masks,
//     takes the row max, evaluates exp2 with the scale folded in, accumulates the row sum,
//     writes P back to TMEM and rescales O in TMEM when the running max moves;
//   * the epilogue (same warpgroup) divides O by the row sum and writes O (bf16) and LSE.
//
// Two Q tiles per CTA share each K/V stage: while one warpgroup runs its softmax the tensor
// core works on the other tile's GEMMs (the role pingpong played on Hopper: "flash-attention-3",
// "Why a schedule, and not an algorithm"; "Lecture 9", "Ping-pong scheduling").
//
// Running-max reference: a row keeps its old max m as the exponent shift until a new tile's
// max exceeds it by more than 8 (log2 units). Until then p = exp2(s*x - m) <= 2^8, which fp32
// sums, bf16 and e4m3 all hold; O and l share the same shift, so the final O / l is exact.
// This skips almost every O rescale after the first few tiles.
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include "ptx.cuh"
#include "varlen.cuh"

namespace gb300 {

// Most units a second (dependent) launch of a non-causal prefill can take.
constexpr int kMaxTailUnits = 256;

struct AttnParams {
  void* o;                  // bf16 [B, N, H, D]
  float* lse;               // fp32 [B, H, N]
  // fp8 only. Descales are read at element offsets (all strides 0 = one value per tensor):
  //   q: b * dq_sb + h * dq_sh + (pos / 128) * dq_sm      (h query head, pos query position)
  //   k: b * dk_sb + kvh * dk_sh + (key / 64) * dk_sn     (kvh kv head, key key position)
  //   v: b * dv_sb + kvh * dv_sh
  const float* descale_q;
  const float* descale_k;
  const float* descale_v;
  int dq_sb, dq_sh, dq_sm, dk_sb, dk_sh, dk_sn, dv_sb, dv_sh;
  int B, H, Hkv, N;         // N: query rows per (batch, head) (prefill: also the key count)
  float scale_log2;         // |scale| * log2(e)
  // 0, or the instruction-descriptor bit that negates the A operand (Q) of S = Q K^T: with a
  // negative scale the kernel computes S = -Q K^T and scales it by |scale|, so every score the
  // softmax sees is scale * q . k and its row maximum is still a maximum.
  uint32_t qk_negate;
  int n_mb;                 // query blocks (NQ x 128 rows) per (batch, head) / per (batch, kv head)
  int n_tiles;              // work tiles in the launch
  // Split-KV (decode) mode: Nk keys in n_kvt tiles of 128, split into n_splits ranges; query
  // rows of a GQA group are packed G per position into the 128-row tiles; the normalized partial
  // O (fp32 [n_splits, B, H, N, D]) and LSE ([n_splits, B, H, N]) go to part_o / part_lse.
  int Nk, G, n_splits, n_kvt;
  float* part_o;
  float* part_lse;
  // Varlen mode (ragged batch): sequence b owns rows cu_q[b] .. cu_q[b+1]-1 of the packed q (the
  // maps and B = 1, N = total rows) and rows cu_k[b] .. of k and v; work tiles come from the plan.
  const int* cu_q;
  const int* cu_k;
  const int* plan;
  // Non-causal prefill whose last wave would leave SMs idle: some work tiles have their key range
  // cut in two. The first launch covers the first part of each such tile and writes its O and LSE
  // as usual; a second, dependent launch covers the rest of the keys and merges it into what the
  // first launch wrote.
  //   tail_mode 1, first launch (last wave halved): tiles t >= tail_first visit only KV tiles
  //     [0, tail_kvt); tail_mode 2, its second launch: unit u is tile tail_first + u from KV tile
  //     tail_kvt on.
  //   tail_mode 3, first launch (share deal, bf16 at d <= 128): tiles below bal_main go
  //     round-robin in whole rounds; the KV tiles of the rest, taken tile by tile, are dealt in
  //     gridDim.x equal shares (see bal_share), so every CTA ends the launch pair with the same
  //     number of KV tiles; tail_mode 4, its second launch: unit u is tile tail_tab[u].x from KV
  //     tile tail_tab[u].y on.
  // tail_mode 0: every tile visits all KV tiles.
  int tail_mode, tail_first, tail_kvt;
  int bal_main;             // tail_mode 3: tiles dealt in whole rounds (a multiple of gridDim.x)
  long long bal_wtail;      // tail_mode 3: KV tiles of the remaining tiles
  int2 tail_tab[kMaxTailUnits];   // tail_mode 4: (tile, first KV tile) per unit
  int o_v8;                 // o is 32-byte aligned: each lane writes its row 32 bytes at a time
  uint32_t* status;         // device status word (first failure)
  unsigned long long timeout_ns;
  int debug_skip_load;      // fault injection: CTA 0 never loads V_0 of its first tile
};

template <int D_, bool CAUSAL_, bool FP8_, bool SPLIT_ = false, bool VARLEN_ = false>
struct AttnCfg {
  static constexpr int D = D_;
  static constexpr bool CAUSAL = CAUSAL_;
  static constexpr bool FP8 = FP8_;
  static constexpr bool SPLIT = SPLIT_;                   // split-KV decode mode (no mask)
  static constexpr bool VARLEN = VARLEN_;                 // ragged batch from a tile plan
  static_assert(!(SPLIT && CAUSAL), "split-KV mode has no causal mask");
  static_assert(!(SPLIT && VARLEN), "split-KV and varlen modes are separate");
  static constexpr int ELT = FP8 ? 1 : 2;                 // bytes per q/k/v element
  // 128-row Q tiles per CTA. Split-KV (decode) units have few query rows, usually one tile, so
  // they take the one-tile pipeline, whose S double buffer lets S_{j+1} run during softmax j.
  static constexpr int NQ = (D <= 128 && !SPLIT_) ? 2 : 1;
  static constexpr int BM = 128, BN = 128;                // query rows per Q tile, keys per KV tile
  // Tiles are stored with the 128-byte swizzle, except e4m3 at d = 64, whose 64-byte rows take
  // the 64-byte swizzle (the TMA box and the MMA descriptors use the same one).
  static constexpr int SWZ = D * ELT < 128 ? 64 : 128;   // bytes per swizzle row
  static constexpr int CE = SWZ / ELT;                    // elements in one swizzle row
  static constexpr int NCH = D / CE;                      // swizzle-row column chunks per row
  static constexpr int CHUNK_BYTES = 128 * SWZ;           // 128 rows of one chunk (one TMA box)
  static constexpr int SBO = 8 * SWZ;                     // stride between 8-row groups
  static constexpr int TILE_BYTES = NCH * CHUNK_BYTES;    // one Q, K or V tile
  static constexpr int Q_BYTES = NQ * TILE_BYTES;
  // Non-causal bf16 prefill at d <= 128 may take the share deal of its last tiles (tail_mode 3).
  static constexpr bool SHARES = !CAUSAL_ && !SPLIT_ && !VARLEN_ && !FP8_ && D_ <= 128;
  static constexpr int SMEM_LIMIT = 232448;               // 227 KB per CTA
  static constexpr int RESERVE = 1024 + 1024;             // alignment slack + static shared
  static constexpr int NS_FIT = (SMEM_LIMIT - RESERVE - Q_BYTES) / TILE_BYTES;
  // K/V ring stages. With a dedicated S-issuer warp (two bf16 Q tiles) the count is even, so each
  // stage holds only K tiles or only V tiles: K stages are waited for by the S issuer alone and V
  // stages by the PV issuers alone, each of which has waited for the stage's previous load itself.
  // A parity wait cannot tell phases two apart, and with an odd count a PV issuer whose tile has
  // no keys in a work tile (a ragged sequence's end) would wait for a V stage whose previous load,
  // a K tile it never waits for, has not landed, and pass it two phases early.
  static constexpr int NS_CAP = NS_FIT > 8 ? 8 : NS_FIT;
  static constexpr int NS = (NQ == 2 && (NS_CAP & 1)) ? NS_CAP - 1 : NS_CAP;
  static constexpr int SMEM_BYTES = Q_BYTES + NS * TILE_BYTES + 1024;
  static constexpr int KSTEPS_QK = D * ELT / 32;          // one MMA k-step covers 32 bytes of K
  static constexpr int KSTEPS_PV = BN * ELT / 32;
  static constexpr int PV_ROWS = 32 / ELT;                // V rows consumed per PV k-step
  static constexpr int P_COLS = BN * ELT / 4;             // TMEM columns holding one P row
  static constexpr int S_COL0 = 0, S_COL1 = 128;          // two S buffers
  // Two Q tiles at d = 64 leave room in TMEM for a third 128-column S buffer. The S products of
  // both tiles then rotate through three buffers (the k-th S of the CTA in buffer k % 3), issued
  // by a warp of their own (the otherwise idle twelfth warp), so a tile's S_{j+1} is issued as
  // soon as a buffer is free, not behind its PV_j, and is ready when its softmax finishes step j.
  static constexpr bool S3 = (NQ == 2 && D == 64);
  // Two Q tiles at d = 128 fill TMEM with two O tiles, so P cannot alias a per-tile S buffer
  // without chaining S_{j+1} to PV_j. Instead both tiles share one 128-column S buffer and each
  // writes its P (P_COLS columns: 64 for bf16 pairs, 32 for e4m3 quadruples) to an area of its
  // own: the S issuer puts the next S into the buffer as soon as the softmax that owns the current
  // one has loaded it into registers, whatever the PVs are doing. TMEM: S at 0, P of tile q at
  // P_COL + P_COLS q, O at 256.
  static constexpr bool S1 = (NQ == 2 && D == 128);
  static constexpr bool SISS = S3 || S1;                  // a warp of its own issues every S
  static constexpr int NSB = S3 ? 3 : 1;                  // S buffers the S issuer rotates through
  static constexpr int P_COL = 128;
  // S-ready, P-ready and PV-done barriers: one per S buffer (one Q tile) or per Q tile (two); in
  // three-buffer mode three per Q tile, the tile's g-th S product using index g % 3. A tile can
  // then have up to three S products (or P halves, or PVs) outstanding without two of them
  // sharing a barrier phase window.
  static constexpr int N_SBAR = S3 ? 6 : 2;
  static constexpr int N_OBAR = S3 ? 6 : NQ;
  static constexpr int O_COL = S3 ? 384 : 256;            // O tile qt at O_COL + qt * D
  static constexpr int TMEM_COLS = 512;
  // Roles: warps [0, 4 NQ) softmax (one warpgroup per Q tile), then one MMA-issuer warp per Q
  // tile, then the TMA warp. With two Q tiles each tile's warp issues its PVs, so one issuer's
  // waits for its softmax never hold up the other tile's MMAs, and a warp of its own issues
  // every S.
  static constexpr int MMA_WARPS = NQ;
  static constexpr int SOFTMAX_WARPS = 4 * NQ;            // one warpgroup per Q tile
  static constexpr int WARP_MMA = SOFTMAX_WARPS, WARP_LOAD = SOFTMAX_WARPS + MMA_WARPS;
  static constexpr int WARP_S = WARP_LOAD + 1;            // two Q tiles: the S issuer
  // Two Q tiles: 12 warps (softmax x8, PV issuers x2, load, S issuer) so the
  // third warpgroup can hand registers to the softmax warpgroups with setmaxnreg. The launch gives
  // 384 x 168 = 64,512 registers; the split below takes 256 x 200 + 128 x 96 = 63,488 of them.
  // (256 x 216 + 128 x 72 at d = 64 was faster while the softmax took its row maximum with a
  // max chain; with the maximum from the TMEM loads it is 2.4% slower on the 16k-key workload.)
  // The host checks the compiled register count first (an over-subscribed increase never
  // returns).
  static constexpr bool REG_SPLIT = (NQ == 2);
  // With a two-stage ring (d = 256: 64 KB tiles) K_j always takes stage 0 and V_j stage 1. Then
  // K and V get a producer warp each (WARP_LOAD: Q and K, WARP_LOAD + 1: V), so the next K can
  // load as soon as S has read the last one, without queueing behind V's wait for PV.
  static constexpr bool TWO_LOADERS = (NS == 2);
  static constexpr int THREADS = REG_SPLIT ? 384 : (SOFTMAX_WARPS + MMA_WARPS + 1 + (TWO_LOADERS ? 1 : 0)) * 32;
  static constexpr uint32_t REGS_SOFTMAX = 200, REGS_OTHER = 96;
  static constexpr int REGS_NEEDED = SOFTMAX_WARPS * 32 * REGS_SOFTMAX + 128 * REGS_OTHER;
  static constexpr uint32_t FMT = FP8 ? kFmtE4M3 : kFmtBF16;
  static constexpr uint32_t IDESC_QK = make_idesc(FMT, 128, BN, false, false);
  static constexpr uint32_t IDESC_PV = make_idesc(FMT, 128, D, false, true);
  static_assert(NS >= 2, "K/V ring needs at least two stages");
  static_assert(!SISS || NS % 2 == 0, "an S-issuer warp needs an even number of K/V stages");
  static_assert(O_COL + NQ * D <= TMEM_COLS, "TMEM budget");
  static_assert(D % CE == 0, "head dim must fill whole swizzle rows");
};

// Wait-site codes recorded in the status word when a bounded wait gives up.
enum : uint32_t { SITE_Q_EMPTY = 1, SITE_KV_EMPTY = 2, SITE_Q_FULL = 3, SITE_KV_FULL = 4, SITE_P_FULL = 5,
                  SITE_S_FULL = 6, SITE_O_DONE = 7, SITE_DRAIN = 8, SITE_O_FULL = 9,
                  SITE_S_FREE = 12 };

struct TileCoord {
  int b, h, mb;     // h: query head (prefill) or kv head (split-KV)
  int s, j0, j1;    // split index and its KV tile range [j0, j1)
  int bo;           // batch coordinate of the maps and outputs (0 in varlen mode)
  int q_base, k_base;   // first q / k row of the sequence in the packed tensors (varlen)
  int nq, nk, n_kvt;    // query rows, keys and 128-key tiles of this sequence
};

// Balanced tail (tail_mode 3), this CTA's share of the W = bal_wtail KV tiles that follow the
// whole rounds: [s0, s1) with s0 = floor(c W / G), s1 = floor((c + 1) W / G), the KV tiles of tail
// tile i being i K .. i K + K - 1 (K = n_kvt). The first launch runs tail tiles ta .. te: those
// that start inside the share, whole, and tile te, cut at KV tile je when the share ends inside
// it (je = K otherwise). The part of a tile before s0 belongs to the previous share; the part
// from s0 on, when s0 falls inside a tile, is a second-launch unit. Every share is at least K
// long, so te >= ta and no tile is cut twice.
__device__ __forceinline__ void bal_share(const AttnParams& p, int& ta, int& te, int& je) {
  const long long G = gridDim.x, c = blockIdx.x, K = p.n_kvt;
  const long long s0 = c * p.bal_wtail / G, s1 = (c + 1) * p.bal_wtail / G;
  ta = (int)((s0 + K - 1) / K);
  te = (int)((s1 - 1) / K);
  je = (int)(s1 - (long long)te * K);
}

// Work tile t -> (batch, head, query block). Causal tiles go longest first: every head's last
// query block, then every head's second-to-last, and so on. Non-causal tiles keep a head's
// blocks together so concurrently running CTAs share K/V in L2.
template <class C>
__device__ __forceinline__ TileCoord decode_tile(int t, const AttnParams& p) {
  TileCoord c;
  if constexpr (C::VARLEN) {
    // Plan entry: (sequence, head << 16 | query block), longest first.
    const int2 e = reinterpret_cast<const int2*>(p.plan + p.plan[5])[t];
    c.b = e.x;
    c.h = (int)((uint32_t)e.y >> 16);
    c.mb = e.y & 0xFFFF;
    c.bo = 0;
    const bool b_ok = c.b >= 0 && c.b < p.B;
    c.q_base = b_ok ? __ldg(p.cu_q + c.b) : 0;
    c.nq = b_ok ? __ldg(p.cu_q + c.b + 1) - c.q_base : 0;
    c.k_base = b_ok ? __ldg(p.cu_k + c.b) : 0;
    c.nk = b_ok ? __ldg(p.cu_k + c.b + 1) - c.k_base : 0;
    // Rows outside the packed tensors (offsets that changed since the plan was built) make the
    // tile empty for every role, so nothing is read or written out of bounds.
    if (!(b_ok && c.h >= 0 && c.h < p.H && c.q_base >= 0 && c.nq >= 0 && c.q_base + c.nq <= p.N && c.k_base >= 0 && c.nk >= 0 &&
          c.k_base + c.nk <= p.Nk)) {
      atomicCAS(p.status, 0u, kStatusBadPlan);
      c.b = c.h = 0;
      c.q_base = c.k_base = c.nq = c.nk = 0;
    }
    c.n_kvt = (c.nk + C::BN - 1) / C::BN;
    c.s = 0;
    c.j0 = 0;
    c.j1 = c.n_kvt;
    return c;
  }
  c.q_base = 0;
  c.k_base = 0;
  c.nq = p.N;
  c.nk = C::SPLIT ? p.Nk : p.N;
  c.n_kvt = p.n_kvt;
  if (C::SPLIT) {
    // Split-KV: the query blocks of one (batch, kv head, split) are consecutive.
    c.mb = t % p.n_mb;
    const int rest = t / p.n_mb;
    c.s = rest % p.n_splits;
    const int bk = rest / p.n_splits;
    c.b = bk / p.Hkv;
    c.h = bk % p.Hkv;
    c.bo = c.b;
    c.j0 = (int)((long long)c.s * p.n_kvt / p.n_splits);
    c.j1 = (int)((long long)(c.s + 1) * p.n_kvt / p.n_splits);
    return c;
  }
  c.s = 0;
  c.j0 = 0;
  c.j1 = p.n_kvt;
  const int BH = p.B * p.H;
  int bh;
  if (C::CAUSAL) {
    c.mb = p.n_mb - 1 - t / BH;
    bh = t % BH;
  } else {
    int tile = t;
    if (p.tail_mode == 2) {
      tile += p.tail_first;
      c.j0 = p.tail_kvt;
    } else if (p.tail_mode == 1 && t >= p.tail_first) {
      c.j1 = p.tail_kvt;
    }
    if constexpr (C::SHARES) {
      if (p.tail_mode == 4) {
        const int2 e = p.tail_tab[t];
        tile = e.x;
        c.j0 = e.y;
      } else if (p.tail_mode == 3 && t >= p.bal_main) {
        int ta, te, je;
        bal_share(p, ta, te, je);
        if (t - p.bal_main == te) c.j1 = je;   // the tile this CTA's share ends in: its first part
      }
    }
    c.mb = tile % p.n_mb;
    bh = tile / p.n_mb;
  }
  c.b = bh / p.H;
  c.h = bh % p.H;
  c.bo = c.b;
  return c;
}

// First query position of Q tile qt (split-KV: G packed rows per position).
template <class C>
__device__ __forceinline__ int q_tile_pos0(const TileCoord& tc, int qt, const AttnParams& p) {
  const int row0 = (tc.mb * C::NQ + qt) * C::BM;
  return C::SPLIT ? row0 / p.G : row0;
}

// Number of KV tiles Q tile `qt` visits (0 if all its rows are past N), starting at tile tc.j0.
template <class C>
__device__ __forceinline__ int kv_tiles_for(const TileCoord& tc, int qt, const AttnParams& p) {
  const int pos0 = q_tile_pos0<C>(tc, qt, p);
  if constexpr (C::VARLEN) return varlen_kv_tiles(pos0, tc.nq, tc.nk, C::CAUSAL);
  if (pos0 >= p.N) return 0;
  if (C::SPLIT || !C::CAUSAL) return tc.j1 - tc.j0;
  return pos0 / C::BN + 1;
}

// S issuer modes: the position of Q tile qt's S_j among all S products of the CTA, in issue
// order, for a work tile whose two Q tiles visit n0 and n1 KV tiles, given the count issued before
// the work tile. The S issuer takes S0_j, then S1_j, skipping the S products a tile does not
// need, so that order is fixed. S number k lives in buffer k % NSB.
__device__ __forceinline__ uint32_t s_number(uint32_t sbase, int qt, int j, int n0, int n1) {
  return sbase + (uint32_t)(min(j, n0) + min(j, n1) + ((qt == 1 && j < n0) ? 1 : 0));
}

// Optional event trace for pipeline analysis (off unless compiled with -DGB300_ATTN_TRACE):
// in CTA 0, each warp's recording lane appends (event, a, b, clock64) to its own 1024-entry slot.
#ifdef GB300_ATTN_TRACE
__device__ unsigned long long g_attn_trace[2 * 32 * 1024];
#define ATTN_TRACE_DECL uint32_t trace_n_ = 0
#define ATTN_TRACE(ev, a, b)                                                                          \
  do {                                                                                               \
    if (blockIdx.x == 0 && trace_n_ < 1024u && (threadIdx.x >> 5) < 32u) {                           \
      const uint32_t i_ = (threadIdx.x >> 5) * 1024u + trace_n_++;                                   \
      g_attn_trace[2 * i_] =                                                                         \
          ((unsigned long long)(ev) << 48) | ((unsigned long long)(a) << 32) | (unsigned int)(b);    \
      g_attn_trace[2 * i_ + 1] = clock64();                                                          \
    }                                                                                                \
  } while (0)
#else
#define ATTN_TRACE_DECL \
  do {                  \
  } while (0)
#define ATTN_TRACE(ev, a, b) \
  do {                       \
  } while (0)
#endif

// Work tile of a CTA's turn-th turn: turn k deals tiles k G .. k G + G - 1 to the G persistent
// CTAs. With ZIGZAG (tiles sorted longest first: causal masks, varlen plans) the deal runs forward
// on even turns and backward on odd ones, so the CTA that took the longest tile of one turn takes
// the shortest of the next. Plain round-robin gives CTA 0 the longest tile of every turn. Tiles of
// equal cost keep the plain deal. Once a CTA's tile is past the end, so are all its later ones.
template <bool ZIGZAG>
__device__ __forceinline__ int deal_tile(int turn) {
  const int g = (int)gridDim.x, c = (int)blockIdx.x;
  return turn * g + ((ZIGZAG && (turn & 1)) ? g - 1 - c : c);
}

// Work tile of this CTA's turn-th turn; n_tiles or more once it has none left.
template <class C>
__device__ __forceinline__ int next_tile(int turn, const AttnParams& p) {
  if constexpr (C::SHARES) {
    if (p.tail_mode == 3) {
      const int rounds = p.bal_main / (int)gridDim.x;
      if (turn < rounds) return turn * (int)gridDim.x + (int)blockIdx.x;
      int ta, te, je;
      bal_share(p, ta, te, je);
      const int i = ta + (turn - rounds);
      return i <= te ? p.bal_main + i : p.n_tiles;
    }
  }
  return deal_tile<C::CAUSAL || C::VARLEN>(turn);
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// f16 pairs (low half = first element): packing from fp32 (round to nearest), 2^x per element,
// add, unpacking to fp32, and e4m3 (saturating, round to nearest) from f16 pairs.
__device__ __forceinline__ uint32_t f16x2_pack(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
__device__ __forceinline__ uint32_t ex2_f16x2(uint32_t h2) {
  uint32_t r;
  asm("ex2.approx.f16x2 %0, %1;" : "=r"(r) : "r"(h2));
  return r;
}
__device__ __forceinline__ uint32_t f16x2_add(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("add.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
__device__ __forceinline__ void f16x2_unpack(uint32_t h2, float& lo, float& hi) {
  asm("{\n .reg .b16 l, h;\n mov.b32 {l, h}, %2;\n cvt.f32.f16 %0, l;\n cvt.f32.f16 %1, h;\n}\n"
      : "=f"(lo), "=f"(hi)
      : "r"(h2));
}
// Four e4m3 values from two f16 pairs, the first pair in the low half: the two 16-bit results
// are joined by one move instead of a shift and an or.
__device__ __forceinline__ uint32_t e4m3x4_from_f16x2x2(uint32_t lo2, uint32_t hi2) {
  uint32_t r;
  asm("{\n .reg .b16 a, b;\n cvt.rn.satfinite.e4m3x2.f16x2 a, %1;\n cvt.rn.satfinite.e4m3x2.f16x2 b, %2;\n"
      " mov.b32 %0, {a, b};\n}\n"
      : "=r"(r)
      : "r"(lo2), "r"(hi2));
  return r;
}

// TMEM column of the S buffer S_j of Q tile qt uses (two Q tiles: one buffer each; one Q tile:
// the two buffers alternate).
template <class C>
__device__ __forceinline__ uint32_t s_buf_col(int qt, int j) {
  return (C::NQ == 2 ? qt : (j & 1)) ? (uint32_t)C::S_COL1 : (uint32_t)C::S_COL0;
}
template <class C>
__device__ __forceinline__ int s_buf_idx(int qt, int j) {
  return C::NQ == 2 ? qt : (j & 1);
}

// S = Q K^T for one 128 x 128 tile: KSTEPS_QK MMAs, each reading 32 bytes of every Q and K row.
// Descriptors are built once; a k-step only adds its byte offset (>> 4) to the start-address
// field, which cannot carry out because every shared-memory address is below 2^18.
// idesc: C::IDESC_QK, or (forward with a negative scale) that with the negate-A bit.
template <class C>
__device__ __forceinline__ void issue_qk(uint32_t d_tmem, uint32_t a_addr, uint32_t b_addr,
                                         uint32_t idesc = C::IDESC_QK) {
  const uint64_t a0 = make_sdesc_swz(a_addr, 16, C::SBO, C::SWZ);
  const uint64_t b0 = make_sdesc_swz(b_addr, 16, C::SBO, C::SWZ);
  constexpr int KPR = C::SWZ / 32;   // k-steps per swizzle row
#pragma unroll
  for (int kk = 0; kk < C::KSTEPS_QK; ++kk) {
    const uint64_t off = (uint64_t)(((kk / KPR) * C::CHUNK_BYTES + (kk % KPR) * 32) >> 4);
    mma_f16_or_f8<C::FP8>(d_tmem, a0 + off, b0 + off, idesc, kk > 0 ? 1u : 0u);
  }
}

// Half H of O += P V: the k-steps covering keys [64 H, 64 H + 64) of the tile. P comes from
// TMEM (8 columns per k-step), V from shared memory (MN-major, PV_ROWS rows per k-step).
template <class C, int H>
__device__ __forceinline__ void issue_pv_half(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_addr,
                                              bool accumulate_first) {
  constexpr int KH = C::KSTEPS_PV / 2;
  const uint64_t b0 = make_sdesc_swz(b_addr, C::CHUNK_BYTES, C::SBO, C::SWZ);
#pragma unroll
  for (int i = 0; i < KH; ++i) {
    const int kk = H * KH + i;
    const uint32_t acc = (H > 0 || i > 0) ? 1u : (accumulate_first ? 1u : 0u);
    mma_ts_f16_or_f8<C::FP8>(d_tmem, a_tmem + kk * 8, b0 + (uint64_t)((kk * C::PV_ROWS * C::SWZ) >> 4),
                             C::IDESC_PV, acc);
  }
}

template <class C>
__global__ void __launch_bounds__(C::THREADS, 1)
attn_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ AttnParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // kv_empty / q_empty take one arrival per MMA-issuer warp (a tcgen05.commit after the MMAs
  // that read the stage, or a plain arrive for a stage that warp's Q tile does not need).
  __shared__ __align__(8) uint64_t bar_q_full, bar_q_empty, bar_drain[C::MMA_WARPS + (C::SISS ? 1 : 0)];
  __shared__ __align__(8) uint64_t bar_kv_full[C::NS], bar_kv_empty[C::NS];
  // o_done: one phase per PV product (rescale waits); o_full: one phase per work tile, after its
  // last PV (epilogue waits). With one Q tile the S MMAs run a step ahead of the PVs, so at the
  // epilogue o_done can lag two phases and a parity wait on it would be ambiguous.
  // p_half[b][h]: the softmax has written half h of P (keys 64h .. 64h+63) into S buffer b.
  // One pair per S buffer: with one Q tile the softmax may run a step ahead of the MMA warp,
  // and per-buffer barriers keep each barrier within one phase of its waiter (a buffer is
  // reused only after the PV that read it has been issued).
  // s_free[b] (three-buffer mode): the PV that read S buffer b has completed, so b can take a new S.
  __shared__ __align__(8) uint64_t bar_s_full[C::N_SBAR], bar_p_half[C::N_SBAR][2], bar_o_done[C::N_OBAR], bar_o_full[C::NQ];
  // s_free[b] (S issuer modes): S buffer b may take a new S. Three S buffers: the PV that read P
  // from b has completed (one commit). Shared S buffer: the softmax warps that own the S in it
  // have loaded it (one arrival per warp).
  __shared__ __align__(8) uint64_t bar_s_free[C::SISS ? C::NSB : 1];
  __shared__ uint32_t tmem_slot;
  __shared__ volatile uint32_t abort_flag;

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  // Split mode: the combine kernel is launched as a programmatic dependent; a halved last wave:
  // the launch of the second halves is. Let its CTAs be scheduled now (they read this grid's
  // results only after waiting for it to finish).
  constexpr bool kDense = !C::CAUSAL && !C::SPLIT && !C::VARLEN;
  if (C::SPLIT || (kDense && (p.tail_mode == 1 || p.tail_mode == 3))) griddep_launch_dependents();
  const uint32_t smem_base = (smem_addr(smem_raw) + 1023u) & ~1023u;
  const uint32_t sQ = smem_base;
  const uint32_t sKV = smem_base + C::Q_BYTES;
  const WaitCtl ctl{&abort_flag, p.status, p.timeout_ns};

  if (tid == 0) {
    abort_flag = 0u;
    mbar_init(smem_addr(&bar_q_full), 1);
    mbar_init(smem_addr(&bar_q_empty), C::MMA_WARPS);
    for (int i = 0; i < C::MMA_WARPS + (C::SISS ? 1 : 0); ++i) mbar_init(smem_addr(&bar_drain[i]), 1);
    for (int i = 0; i < C::NS; ++i) {
      mbar_init(smem_addr(&bar_kv_full[i]), 1);
      mbar_init(smem_addr(&bar_kv_empty[i]), C::MMA_WARPS);
    }
    if constexpr (C::SISS)
      for (int i = 0; i < C::NSB; ++i) mbar_init(smem_addr(&bar_s_free[i]), C::S1 ? 4 : 1);
    for (int i = 0; i < C::N_SBAR; ++i) {
      mbar_init(smem_addr(&bar_s_full[i]), 1);
      // One arrival per softmax warp.
      mbar_init(smem_addr(&bar_p_half[i][0]), 4);
      mbar_init(smem_addr(&bar_p_half[i][1]), 4);
    }
    for (int i = 0; i < C::N_OBAR; ++i) mbar_init(smem_addr(&bar_o_done[i]), 1);
    for (int i = 0; i < C::NQ; ++i) mbar_init(smem_addr(&bar_o_full[i]), 1);
    fence_mbar_init();
  }
  if (warp == C::WARP_MMA) {
    tmem_alloc(smem_addr(&tmem_slot), C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  ATTN_TRACE_DECL;
  // Work tiles: a count fixed at launch, or (varlen) the plan's, once the plan is seen to have been
  // built for this launch's sequences, heads, tile height and mask.
  int n_tiles = p.n_tiles;
  if constexpr (C::VARLEN) {
    const bool good = __ldg(p.plan + 1) == p.B && __ldg(p.plan + 2) == p.H && __ldg(p.plan + 3) == C::NQ * C::BM &&
                      __ldg(p.plan + 4) == (C::CAUSAL ? 1 : 0) && __ldg(p.plan + 6) == p.N && __ldg(p.plan + 7) == p.Nk;
    n_tiles = good ? min(__ldg(p.plan), p.n_tiles) : 0;   // p.n_tiles: entries the plan buffer holds
    if (!good && tid == 0 && blockIdx.x == 0) atomicCAS(p.status, 0u, kStatusBadPlan);
  }

  if (C::TWO_LOADERS && (warp == C::WARP_LOAD || warp == C::WARP_LOAD + 1)) {
    // ------------------------------------------------------------------ TMA producers, K and V
    if (lane == 0) {
      const bool is_v = warp == C::WARP_LOAD + 1;   // stage 1: V tiles; stage 0: Q and K tiles
      const uint32_t slot = is_v ? 1u : 0u;
      if (!is_v) tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(is_v ? &tm_v : &tm_k);
      uint32_t cnt = 0;       // K (or V) tiles issued so far
      uint32_t nq_loads = 0;  // Q loads issued so far (K warp)
      bool ok = true;
      int iter = 0;
      for (int turn = 0, t = next_tile<C>(0, p); ok && t < n_tiles; t = next_tile<C>(++turn, p), ++iter) {
        const TileCoord tc = decode_tile<C>(t, p);
        const int kvh = C::SPLIT ? tc.h : tc.h / p.G;
        int nmax = 0, nq_valid = 0;
        for (int qt = 0; qt < C::NQ; ++qt) {
          const int n = kv_tiles_for<C>(tc, qt, p);
          nmax = n > nmax ? n : nmax;
          nq_valid += (n > 0);
        }
        if (C::VARLEN && nmax == 0) continue;   // every row sees no key: the softmax warps write it
        if (!is_v) {
          // Q: wait until the previous work tile's last S = Q K^T has completed.
          if (nq_loads > 0 && !mbar_wait(smem_addr(&bar_q_empty), (nq_loads - 1) & 1, ctl, SITE_Q_EMPTY)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(smem_addr(&bar_q_full), nq_valid * C::TILE_BYTES);
          for (int qt = 0; qt < C::NQ; ++qt) {
            const int pos0 = q_tile_pos0<C>(tc, qt, p);
            if (kv_tiles_for<C>(tc, qt, p) == 0) continue;
            for (int ch = 0; ch < C::NCH; ++ch) {
              const uint32_t dst = sQ + (qt * C::NCH + ch) * C::CHUNK_BYTES;
              if (C::SPLIT)
                tma_load_5d(dst, &tm_q, smem_addr(&bar_q_full), ch * C::CE, 0, pos0, tc.h, tc.b);
              else
                tma_load_4d(dst, &tm_q, smem_addr(&bar_q_full), ch * C::CE, tc.q_base + pos0, tc.h, tc.bo);
            }
          }
          ++nq_loads;
        }
        for (int j = 0; ok && j < nmax; ++j) {
          // load number cnt of this stage waits for the release of load cnt - 1
          if (cnt > 0 && !mbar_wait(smem_addr(&bar_kv_empty[slot]), (cnt - 1) & 1, ctl, SITE_KV_EMPTY)) {
            ok = false;
            break;
          }
          const bool skip = p.debug_skip_load && blockIdx.x == 0 && iter == 0 && j == 0 && is_v;
          if (!skip) {
            mbar_arrive_expect_tx(smem_addr(&bar_kv_full[slot]), C::TILE_BYTES);
            for (int ch = 0; ch < C::NCH; ++ch)
              tma_load_4d(sKV + slot * C::TILE_BYTES + ch * C::CHUNK_BYTES, is_v ? &tm_v : &tm_k,
                          smem_addr(&bar_kv_full[slot]), ch * C::CE, tc.k_base + (tc.j0 + j) * C::BN, kvh, tc.bo);
          }
          ++cnt;
        }
      }
      if (!ok) {
        // Unwinding: let the copy still in flight land before the CTA exits.
        if (cnt > 0) {
          const uint64_t t0 = global_timer_ns();
          while (!mbar_try_wait(smem_addr(&bar_kv_full[slot]), (cnt - 1) & 1) && global_timer_ns() - t0 < p.timeout_ns) {}
        }
        if (nq_loads > 0) {
          const uint64_t t0 = global_timer_ns();
          while (!mbar_try_wait(smem_addr(&bar_q_full), (nq_loads - 1) & 1) && global_timer_ns() - t0 < p.timeout_ns) {}
        }
      }
    }
  } else if (warp == C::WARP_LOAD) {
    // ------------------------------------------------------------------ TMA producer
    if constexpr (C::REG_SPLIT) setmaxnreg_dec<C::REGS_OTHER>();
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      uint32_t ring = 0;      // K/V tiles issued so far (ring position)
      uint32_t nq_loads = 0;  // Q loads issued so far
      bool ok = true;
      int iter = 0;
      for (int turn = 0, t = next_tile<C>(0, p); ok && t < n_tiles; t = next_tile<C>(++turn, p), ++iter) {
        const TileCoord tc = decode_tile<C>(t, p);
        const int kvh = C::SPLIT ? tc.h : tc.h / p.G;
        int nmax = 0, nq_valid = 0;
        for (int qt = 0; qt < C::NQ; ++qt) {
          const int n = kv_tiles_for<C>(tc, qt, p);
          nmax = n > nmax ? n : nmax;
          nq_valid += (n > 0);
        }
        if (C::VARLEN && nmax == 0) continue;   // every row sees no key: the softmax warps write it
        // Q: wait until the previous work tile's last S = Q K^T has completed.
        if (nq_loads > 0 && !mbar_wait(smem_addr(&bar_q_empty), (nq_loads - 1) & 1, ctl, SITE_Q_EMPTY)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(smem_addr(&bar_q_full), nq_valid * C::TILE_BYTES);
        for (int qt = 0; qt < C::NQ; ++qt) {
          const int pos0 = q_tile_pos0<C>(tc, qt, p);
          if (kv_tiles_for<C>(tc, qt, p) == 0) continue;
          for (int ch = 0; ch < C::NCH; ++ch) {
            const uint32_t dst = sQ + (qt * C::NCH + ch) * C::CHUNK_BYTES;
            if (C::SPLIT)   // (d, head in group, position, kv head, batch): G x 128/G packed rows
              tma_load_5d(dst, &tm_q, smem_addr(&bar_q_full), ch * C::CE, 0, pos0, tc.h, tc.b);
            else
              tma_load_4d(dst, &tm_q, smem_addr(&bar_q_full), ch * C::CE, tc.q_base + pos0, tc.h, tc.bo);
          }
        }
        ++nq_loads;
        for (int j = 0; ok && j < nmax; ++j) {
          for (int which = 0; which < 2; ++which) {  // 0: K_j, 1: V_j
            const uint32_t slot = ring % C::NS;
            if (ring >= (uint32_t)C::NS &&
                !mbar_wait(smem_addr(&bar_kv_empty[slot]), ((ring / C::NS) - 1) & 1, ctl, SITE_KV_EMPTY)) {
              ok = false;
              break;
            }
            const bool skip = p.debug_skip_load && blockIdx.x == 0 && iter == 0 && j == 0 && which == 1;
            if (!skip) {
              const CUtensorMap* tm = which ? &tm_v : &tm_k;
              mbar_arrive_expect_tx(smem_addr(&bar_kv_full[slot]), C::TILE_BYTES);
              for (int ch = 0; ch < C::NCH; ++ch)
                tma_load_4d(sKV + slot * C::TILE_BYTES + ch * C::CHUNK_BYTES, tm, smem_addr(&bar_kv_full[slot]),
                            ch * C::CE, tc.k_base + (tc.j0 + j) * C::BN, kvh, tc.bo);
            }
            ++ring;
          }
        }
      }
      if (!ok) {
        // Unwinding: let every copy still in flight land before the CTA exits.
        const uint32_t first = ring > (uint32_t)C::NS ? ring - C::NS : 0u;
        for (uint32_t pos = first; pos < ring; ++pos) {
          const uint32_t bar = smem_addr(&bar_kv_full[pos % C::NS]);
          const uint64_t t0 = global_timer_ns();
          while (!mbar_try_wait(bar, (pos / C::NS) & 1) && global_timer_ns() - t0 < p.timeout_ns) {}
        }
        if (nq_loads > 0) {
          const uint64_t t0 = global_timer_ns();
          while (!mbar_try_wait(smem_addr(&bar_q_full), (nq_loads - 1) & 1) && global_timer_ns() - t0 < p.timeout_ns) {}
        }
      }
    }
  } else if (C::NQ == 2 && warp >= C::WARP_MMA && warp < C::WARP_MMA + C::MMA_WARPS) {
    // ------------------------------------------------------------------ tcgen05 issuer, one per Q tile
    if constexpr (C::REG_SPLIT) setmaxnreg_dec<C::REGS_OTHER>();
    if (lane == 0) {
      const int myq = warp - C::WARP_MMA;   // Q tile (and S/P buffer) this warp issues for
      uint32_t ring = 0;
      bool ok = true;

      auto wait_kv = [&](uint32_t pos) -> bool {
        return mbar_wait(smem_addr(&bar_kv_full[pos % C::NS]), (pos / C::NS) & 1, ctl, SITE_KV_FULL);
      };
      // Release a ring stage: after this warp's MMAs that read it, or at once if none did.
      auto release = [&](uint64_t* bar, bool used) {
        if (used) tc_commit(smem_addr(bar));
        else mbar_arrive(smem_addr(bar));
      };
      const uint32_t d_o = tmem + C::O_COL + myq * C::D;
      {
        // The S issuer warp issues every S; this warp issues its Q tile's PVs. Three S buffers:
        // PV_j reads P_j from S buffer k % 3 (k: S number of S_j); its completion frees that
        // buffer (s_free) and is signalled on o_done for rescales. Barriers of this tile's g-th S
        // product: index 3 myq + g % 3, phase g / 3. Shared S buffer: PV_j reads P_j from this
        // tile's P area; its completion (o_done, index myq, phase g) lets the softmax write the
        // next P there.
        uint32_t sbase = 0;   // S products of both Q tiles before the current work tile
        uint32_t g = 0;       // S products of this Q tile before the current work tile
        for (int turn = 0, t = next_tile<C>(0, p); ok && t < n_tiles; t = next_tile<C>(++turn, p)) {
          const TileCoord tc = decode_tile<C>(t, p);
          const int n0 = kv_tiles_for<C>(tc, 0, p), n1 = kv_tiles_for<C>(tc, 1, p);
          const int n = myq ? n1 : n0;
          const int nmax = n0 > n1 ? n0 : n1;
          if (C::VARLEN && nmax == 0) continue;
          const uint32_t sb = sbase, gb = g;
          sbase += (uint32_t)(n0 + n1);
          g += (uint32_t)n;
          const uint32_t base = ring;  // K_j at base + 2j, V_j at base + 2j + 1
          for (int j = 0; ok && j < nmax; ++j) {
            const uint32_t pos_v = base + 2 * j + 1;
            if (!wait_kv(pos_v)) { ok = false; break; }
            if (j < n) {
              const uint32_t gj = gb + j;
              const uint32_t par = C::S3 ? (gj / 3u) & 1u : gj & 1u;
              const uint32_t bi = C::S3 ? 3u * myq + gj % 3u : (uint32_t)myq;
              const uint32_t b = C::S3 ? s_number(sb, myq, j, n0, n1) % 3u : 0u;
              const uint32_t a_p = C::S3 ? tmem + b * 128u : tmem + C::P_COL + (uint32_t)C::P_COLS * myq;
              const uint32_t b_v = sKV + (pos_v % C::NS) * C::TILE_BYTES;
              if (!mbar_wait(smem_addr(&bar_p_half[bi][0]), par, ctl, SITE_P_FULL)) { ok = false; break; }
              tc_fence_after();
              issue_pv_half<C, 0>(d_o, a_p, b_v, j > 0);
              if (!mbar_wait(smem_addr(&bar_p_half[bi][1]), par, ctl, SITE_P_FULL)) { ok = false; break; }
              tc_fence_after();
              issue_pv_half<C, 1>(d_o, a_p, b_v, true);
              if constexpr (C::S3) tc_commit(smem_addr(&bar_s_free[b]));
              tc_commit(smem_addr(&bar_o_done[bi]));
              if (j + 1 == n) tc_commit(smem_addr(&bar_o_full[myq]));
            }
            release(&bar_kv_empty[pos_v % C::NS], j < n);
          }
          ring = base + 2 * nmax;
        }
      }
      // Every MMA this warp issued must finish before TMEM is released.
      tc_commit(smem_addr(&bar_drain[myq]));
      const uint64_t t0 = global_timer_ns();
      while (!mbar_try_wait(smem_addr(&bar_drain[myq]), 0) && global_timer_ns() - t0 < p.timeout_ns) {}
    }
  } else if (C::SISS && warp == C::WARP_S) {
    // ------------------------------------------------------------------ S issuer
    if constexpr (C::REG_SPLIT) setmaxnreg_dec<C::REGS_OTHER>();
    if (lane == 0) {
      // S products in the order S0_0, S1_0, S0_1, S1_1, ... (skipping those a Q tile does not
      // need), the k-th into buffer k % NSB once that buffer is free of the (k - NSB)-th: three
      // buffers, its PV has read P from it; one shared buffer, its softmax has loaded it.
      uint32_t ring = 0, nq_loads = 0, sbase = 0, g0 = 0, g1 = 0;
      bool ok = true;
      for (int turn = 0, t = next_tile<C>(0, p); ok && t < n_tiles; t = next_tile<C>(++turn, p)) {
        const TileCoord tc = decode_tile<C>(t, p);
        const int n0 = kv_tiles_for<C>(tc, 0, p), n1 = kv_tiles_for<C>(tc, 1, p);
        const int nmax = n0 > n1 ? n0 : n1;
        if (C::VARLEN && nmax == 0) continue;
        const uint32_t sb = sbase, gb0 = g0, gb1 = g1;
        sbase += (uint32_t)(n0 + n1);
        g0 += (uint32_t)n0;
        g1 += (uint32_t)n1;
        if (!mbar_wait(smem_addr(&bar_q_full), nq_loads & 1, ctl, SITE_Q_FULL)) { ok = false; break; }
        ++nq_loads;
        const uint32_t base = ring;  // K_j at base + 2j
        for (int j = 0; ok && j < nmax; ++j) {
          const uint32_t pos_k = base + 2 * j;
          if (!mbar_wait(smem_addr(&bar_kv_full[pos_k % C::NS]), (pos_k / C::NS) & 1, ctl, SITE_KV_FULL)) { ok = false; break; }
          for (int qt = 0; ok && qt < 2; ++qt) {
            if (j >= (qt ? n1 : n0)) continue;
            const uint32_t k = s_number(sb, qt, j, n0, n1);
            const uint32_t b = k % (uint32_t)C::NSB;
            if (k >= (uint32_t)C::NSB &&
                !mbar_wait(smem_addr(&bar_s_free[b]), ((k / C::NSB) - 1u) & 1u, ctl, SITE_S_FREE)) {
              ok = false;
              break;
            }
            tc_fence_after();
            issue_qk<C>(tmem + b * 128u, sQ + qt * C::TILE_BYTES, sKV + (pos_k % C::NS) * C::TILE_BYTES,
                        C::IDESC_QK | p.qk_negate);
            const uint32_t gj = (qt ? gb1 : gb0) + j;
            tc_commit(smem_addr(&bar_s_full[C::S3 ? 3u * qt + gj % 3u : (uint32_t)qt]));
          }
          if (!ok) break;
          // K_j's stage and, after the last S, Q: both arrivals of each come from this warp.
          tc_commit(smem_addr(&bar_kv_empty[pos_k % C::NS]));
          tc_commit(smem_addr(&bar_kv_empty[pos_k % C::NS]));
          if (j + 1 == nmax) {
            tc_commit(smem_addr(&bar_q_empty));
            tc_commit(smem_addr(&bar_q_empty));
          }
        }
        ring = base + 2 * nmax;
      }
      tc_commit(smem_addr(&bar_drain[C::MMA_WARPS]));
      const uint64_t t0 = global_timer_ns();
      while (!mbar_try_wait(smem_addr(&bar_drain[C::MMA_WARPS]), 0) && global_timer_ns() - t0 < p.timeout_ns) {}
    }
  } else if (C::NQ == 1 && warp == C::WARP_MMA) {
    // ------------------------------------------------------------------ tcgen05 issuer, one Q tile
    if constexpr (C::REG_SPLIT) setmaxnreg_dec<C::REGS_OTHER>();
    if (lane == 0) {
      uint32_t ring = 0;        // K/V ring position (same sequence as the producer)
      uint32_t nq_loads = 0;
      uint32_t p_cnt[2] = {0u, 0u};   // P tiles consumed per S buffer
      bool ok = true;
      auto wait_kv = [&](uint32_t pos) -> bool {
        return mbar_wait(smem_addr(&bar_kv_full[pos % C::NS]), (pos / C::NS) & 1, ctl, SITE_KV_FULL);
      };
      // S_j into S buffer j % 2, then signal the softmax.
      auto qk = [&](int j, uint32_t k_slot) {
        issue_qk<C>(tmem + s_buf_col<C>(0, j), sQ, sKV + k_slot * C::TILE_BYTES, C::IDESC_QK | p.qk_negate);
        tc_commit(smem_addr(&bar_s_full[s_buf_idx<C>(0, j)]));
      };
      // O += P_j V_j, issued in two halves as the softmax hands P over.
      auto pv = [&](int j, uint32_t v_slot, bool last) -> bool {
        const uint32_t d_tmem = tmem + C::O_COL;
        const uint32_t a_tmem = tmem + s_buf_col<C>(0, j);
        const uint32_t b_addr = sKV + v_slot * C::TILE_BYTES;
        const int buf = s_buf_idx<C>(0, j);
        const uint32_t par = p_cnt[buf] & 1;
        if (!mbar_wait(smem_addr(&bar_p_half[buf][0]), par, ctl, SITE_P_FULL)) return false;
        tc_fence_after();
        issue_pv_half<C, 0>(d_tmem, a_tmem, b_addr, j > 0);
        if (!mbar_wait(smem_addr(&bar_p_half[buf][1]), par, ctl, SITE_P_FULL)) return false;
        tc_fence_after();
        issue_pv_half<C, 1>(d_tmem, a_tmem, b_addr, true);
        tc_commit(smem_addr(&bar_o_done[0]));
        if (last) tc_commit(smem_addr(&bar_o_full[0]));
        ++p_cnt[buf];
        return true;
      };
      for (int turn = 0, t = next_tile<C>(0, p); ok && t < n_tiles; t = next_tile<C>(++turn, p)) {
        const TileCoord tc = decode_tile<C>(t, p);
        const int nmax = kv_tiles_for<C>(tc, 0, p);
        if (nmax == 0) continue;
        if (!mbar_wait(smem_addr(&bar_q_full), nq_loads & 1, ctl, SITE_Q_FULL)) { ok = false; break; }
        ++nq_loads;
        const uint32_t base = ring;  // K_j at base + 2j, V_j at base + 2j + 1
        if (!wait_kv(base)) { ok = false; break; }
        tc_fence_after();
        qk(0, base % C::NS);
        // Release K_0 before waiting for anything else: with a two-stage ring the producer
        // needs this slot back to load K_1.
        tc_commit(smem_addr(&bar_kv_empty[base % C::NS]));
        if (nmax > 1) {
          // The second S buffer lets S_1 run while the softmax works on S_0.
          if (!wait_kv(base + 2)) { ok = false; break; }
          tc_fence_after();
          qk(1, (base + 2) % C::NS);
          tc_commit(smem_addr(&bar_kv_empty[(base + 2) % C::NS]));
        }
        if (nmax <= 2) tc_commit(smem_addr(&bar_q_empty));
        for (int j = 0; ok && j < nmax; ++j) {
          const uint32_t pos_v = base + 2 * j + 1;
          if (!wait_kv(pos_v)) { ok = false; break; }
          tc_fence_after();
          // S_{j+1} was issued a step ahead; issue S_{j+2} into the buffer P_j frees once PV_j
          // has been issued (one thread's MMAs run in issue order).
          if (!pv(j, pos_v % C::NS, j + 1 == nmax)) { ok = false; break; }
          tc_commit(smem_addr(&bar_kv_empty[pos_v % C::NS]));
          if (j + 2 < nmax) {
            const uint32_t pos_k = base + 2 * (j + 2);
            if (!wait_kv(pos_k)) { ok = false; break; }
            tc_fence_after();
            qk(j + 2, pos_k % C::NS);
            tc_commit(smem_addr(&bar_kv_empty[pos_k % C::NS]));
            if (j + 3 == nmax) tc_commit(smem_addr(&bar_q_empty));
          }
        }
        ring = base + 2 * nmax;
      }
      // Every MMA issued so far must finish before TMEM is released.
      tc_commit(smem_addr(&bar_drain[0]));
      const uint64_t t0 = global_timer_ns();
      while (!mbar_try_wait(smem_addr(&bar_drain[0]), 0) && global_timer_ns() - t0 < p.timeout_ns) {}
    }
  } else if (warp < C::SOFTMAX_WARPS) {
    // ------------------------------------------------------------------ softmax + epilogue
    if constexpr (C::REG_SPLIT) setmaxnreg_inc<C::REGS_SOFTMAX>();
    const int qt = warp >> 2;                  // Q tile of this warpgroup
    const int r = ((warp & 3) << 5) + lane;    // row within the Q tile == TMEM lane
    const uint32_t lane_base = (uint32_t)((warp & 3) << 5) << 16;
    // S tiles consumed per S buffer. Two Q tiles: one buffer per warpgroup, so a single counter
    // (an array indexed by the warpgroup's tile would live in local memory).
    uint32_t s_cnt0 = 0u, s_cnt1 = 0u;
    uint32_t pv_cnt = 0;            // PV products of this Q tile committed so far
    uint32_t tiles_done = 0;        // work tiles of this Q tile finished (o_full phases)
    uint32_t sbase = 0, g = 0;      // S issuer modes: S products of the CTA / of this Q tile so far
    bool ok = true;
    for (int turn = 0, t = next_tile<C>(0, p); ok && t < n_tiles; t = next_tile<C>(++turn, p)) {
      const TileCoord tc = decode_tile<C>(t, p);
      const int n = kv_tiles_for<C>(tc, qt, p);
      int n0 = 0, n1 = 0;
      uint32_t sb = 0, gb = 0;
      if constexpr (C::SISS) {
        n0 = kv_tiles_for<C>(tc, 0, p);
        n1 = kv_tiles_for<C>(tc, 1, p);
        sb = sbase;
        gb = g;
        sbase += (uint32_t)(n0 + n1);
        g += (uint32_t)n;
      }
      const int row0 = q_tile_pos0<C>(tc, qt, p);   // prefill: first query row of the tile
      const int Nk = tc.nk;                         // keys of this sequence
      if (n == 0) {
        // Varlen: rows that see no key at all get O = 0 and LSE = -inf.
        if constexpr (C::VARLEN) {
          const int row = row0 + r;
          if (row < tc.nq) {
            uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(p.o) +
                                                  ((size_t)(tc.q_base + row) * p.H + tc.h) * C::D);
#pragma unroll 1
            for (int v4 = 0; v4 < C::D / 8; ++v4) dst[v4] = make_uint4(0u, 0u, 0u, 0u);
            p.lse[(size_t)tc.h * p.N + tc.q_base + row] = -INFINITY;
          }
        }
        continue;
      }
      // Score scale (log2 units) and output scale of this row (FP8: descales per tensor, per head
      // or per block; split-KV rows of one tile belong to different query heads of the group).
      const int h_row = C::SPLIT ? tc.h * p.G + r % p.G : tc.h;
      const int kvh_row = C::SPLIT ? tc.h : tc.h / p.G;
      float s = p.scale_log2;        // bf16: the score scale; fp8: times the q (and k) descales
      float s_q = s;                 // fp8 with K blocks: scale_log2 * descale_q of this row
      float out_scale = 1.0f;
      const float* dk_row = nullptr;
      if (C::FP8) {
        const int pos = C::SPLIT ? min(row0 + r / p.G, p.N - 1) : row0;
        s_q = s * __ldg(p.descale_q + tc.b * p.dq_sb + h_row * p.dq_sh + (pos >> 7) * p.dq_sm);
        dk_row = p.descale_k + tc.b * p.dk_sb + kvh_row * p.dk_sh;
        s = p.dk_sn ? s_q : s_q * __ldg(dk_row);
        out_scale = __ldg(p.descale_v + tc.b * p.dv_sb + kvh_row * p.dv_sh);
      }
      const int n_kblk = (Nk + 63) >> 6;   // 64-key descale blocks
      float m = -INFINITY;   // running max of s * x (log2 units), used as the exponent shift
      float l = 0.0f;        // running sum of exp2(s * x - m)
      for (int j = 0; j < n; ++j) {
        // buf: index of this S's barriers; s_col: its TMEM buffer (three buffers: S number % 3)
        // buf: index of this S's barriers; s_col: its TMEM buffer (three buffers: S number % 3;
        // shared S buffer: column 0).
        const int buf = C::S3 ? 3 * qt + (int)((gb + j) % 3u) : (C::NQ == 2 ? qt : (j & 1));
        const uint32_t s_col = C::S3 ? (s_number(sb, qt, j, n0, n1) % 3u) * 128u
                                     : C::S1 ? 0u : (buf ? C::S_COL1 : C::S_COL0);
        // Scales of the two 64-key halves of this tile (they differ only with K block descales;
        // read before the wait so the load latency hides behind it).
        float s_lo = s, s_hi = s;
        if (C::FP8 && p.dk_sn) {
          const int kb = 2 * (tc.j0 + j);
          s_lo = s_q * __ldg(dk_row + kb * p.dk_sn);
          s_hi = s_q * __ldg(dk_row + min(kb + 1, n_kblk - 1) * p.dk_sn);
        }
        const uint32_t s_cnt = (C::NQ == 2 || buf == 0) ? s_cnt0 : s_cnt1;
        const uint32_t s_par = C::S3 ? ((gb + j) / 3u) & 1u : C::S1 ? (gb + j) & 1u : s_cnt & 1u;
        bool w = mbar_wait(smem_addr(&bar_s_full[buf]), s_par, ctl, SITE_S_FULL);
        if (!__all_sync(0xffffffffu, w)) { ok = false; break; }
        if (r == 0) ATTN_TRACE(4, qt, j);
        if constexpr (!C::SISS) {
          if (C::NQ == 2 || buf == 0) ++s_cnt0;
          else ++s_cnt1;
        }
        // Masking: keys past N (ragged tail) and, on the diagonal tile, keys after the query row.
        const int jk = tc.j0 + j;   // KV tile index within the sequence
        // Varlen causal masking is bottom-right aligned (query i sees keys <= i + Nk - Nq), so up
        // to two tiles can cross the diagonal; with equal lengths only the last one does.
        const int diag_off = C::VARLEN ? Nk - tc.nq : 0;
        const bool diag = C::CAUSAL && (C::VARLEN ? (jk * C::BN + C::BN - 1 > row0 + diag_off) : (j == n - 1));
        const bool tail = (jk == tc.n_kvt - 1) && (Nk % C::BN != 0);
        const bool masked = diag || tail;
        tc_fence_after();
        uint32_t sr[128];
        // The TMEM loads also give each lane's maximum per 32 columns: the row maximum of an
        // unmasked tile. A masked tile's maximum must skip its masked keys and is taken below.
        float mq0, mq1, mq2, mq3;
        const uint32_t tS = tmem + lane_base + s_col;
        tmem_ld_32cols_max(tS, sr, mq0);
        tmem_ld_32cols_max(tS + 32, sr + 32, mq1);
        tmem_ld_32cols_max(tS + 64, sr + 64, mq2);
        tmem_ld_32cols_max(tS + 96, sr + 96, mq3);
        tmem_ld_wait();
        reg_fence32(sr);
        reg_fence32(sr + 32);
        reg_fence32(sr + 64);
        reg_fence32(sr + 96);
        asm volatile("" : "+f"(mq0), "+f"(mq1), "+f"(mq2), "+f"(mq3));
        if constexpr (C::S1) {
          // S is in registers: the S issuer may put the next S into the shared buffer now.
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_addr(&bar_s_free[0]));
        }
        if (r == 0) ATTN_TRACE(5, qt, j);
        float x[128];
#pragma unroll
        for (int c = 0; c < 128; ++c) x[c] = __uint_as_float(sr[c]);
        if (masked) {
          int lim = Nk - jk * C::BN;
          if (diag) lim = min(lim, (row0 + r + diag_off) - jk * C::BN + 1);
#pragma unroll
          for (int c = 0; c < 128; ++c)
            if (c >= lim) x[c] = -INFINITY;
        }
        // P = exp2(s * x - m) in packed fp32 pairs, in two halves of 64 keys; each half is written
        // to TMEM (over the first columns of the S buffer) and handed to the MMA warp at once.
        // The first half is computed speculatively with the row's current shift m while the row
        // max of this tile is taken alongside it; only if some row's max moved by more than 8
        // (always on the first tile) is that half recomputed with the new shift.
        const uint64_t s2_lo = f2_pack(s_lo, s_lo), s2_hi = f2_pack(s_hi, s_hi);
        constexpr int PKN = C::FP8 ? 16 : 32;   // packed 32-bit P words per half
        auto exp_half = [&](int h, uint64_t nm2, uint32_t* pk, uint64_t& acc0, uint64_t& acc1) {
          const uint64_t s2 = h ? s2_hi : s2_lo;
          if constexpr (C::FP8) {
            // e4m3 P keeps 3 mantissa bits, so the exponentials run in f16 pairs (one exp-unit
            // operation per two scores; inputs to 11 bits, |t| <= 8 here) and P is packed from
            // f16. The half's 64 terms are summed per lane in f16 (16 terms of at most 2^8 each)
            // and then added to the fp32 row sum.
            uint32_t hs0 = 0u, hs1 = 0u;
#pragma unroll
            for (int c = 0; c < 64; c += 4) {
              const int cc = h * 64 + c;
              float t0, t1, t2, t3;
              f2_unpack(f2_fma(f2_pack(x[cc], x[cc + 1]), s2, nm2), t0, t1);
              f2_unpack(f2_fma(f2_pack(x[cc + 2], x[cc + 3]), s2, nm2), t2, t3);
              const uint32_t h01 = ex2_f16x2(f16x2_pack(t0, t1)), h23 = ex2_f16x2(f16x2_pack(t2, t3));
              hs0 = f16x2_add(hs0, h01);
              hs1 = f16x2_add(hs1, h23);
              pk[c >> 2] = e4m3x4_from_f16x2x2(h01, h23);
            }
            float a0, a1, b0, b1;
            f16x2_unpack(hs0, a0, a1);
            f16x2_unpack(hs1, b0, b1);
            acc0 = f2_add(acc0, f2_pack(a0, a1));
            acc1 = f2_add(acc1, f2_pack(b0, b1));
          } else {
#pragma unroll
            for (int c = 0; c < 64; c += 4) {
              const int cc = h * 64 + c;
              float t0, t1, t2, t3;
              f2_unpack(f2_fma(f2_pack(x[cc], x[cc + 1]), s2, nm2), t0, t1);
              f2_unpack(f2_fma(f2_pack(x[cc + 2], x[cc + 3]), s2, nm2), t2, t3);
              const float p0 = ex2(t0), p1 = ex2(t1), p2 = ex2(t2), p3 = ex2(t3);
              acc0 = f2_add(acc0, f2_pack(p0, p1));
              acc1 = f2_add(acc1, f2_pack(p2, p3));
              pk[c >> 1] = pack_bf16x2(p0, p1);
              pk[(c >> 1) + 1] = pack_bf16x2(p2, p3);
            }
          }
        };
        auto store_half = [&](int h, const uint32_t* pk) {
          {
            // P of this tile: its own P area (shared S buffer), else over the start of S.
            const uint32_t tP = C::S1 ? tmem + lane_base + C::P_COL + (uint32_t)C::P_COLS * qt : tS;
            if (C::FP8) tmem_st_16cols(tP + h * 16, pk);
            else tmem_st_32cols(tP + h * 32, pk);
            tmem_st_wait();
            tc_fence_before();
          }
          // Every lane's TMEM stores are complete and fenced; once the warp has converged, one
          // lane arrives for it.
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_addr(&bar_p_half[buf][h]));
          if (r == 0) ATTN_TRACE(7 + h, qt, j);
        };
        uint32_t pk[PKN];
        uint64_t acc0 = f2_pack(0.f, 0.f), acc1 = acc0;
        exp_half(0, f2_pack(-m, -m), pk, acc0, acc1);
        if (r == 0) ATTN_TRACE(16, qt, j);
        // Row max (per 64-key half for fp8, whose halves may carry different K descales; the scales
        // are positive, so max commutes with them): the loads' maxima on an unmasked tile, else
        // eight independent chains of 3-input max over the masked scores.
        float m_tile;
        if (!masked) {
          if constexpr (C::FP8) m_tile = fmaxf(fmaxf(mq0, mq1) * s_lo, fmaxf(mq2, mq3) * s_hi);
          else m_tile = fmaxf(fmaxf(mq0, mq1), fmaxf(mq2, mq3)) * s;
        } else if constexpr (C::FP8) {
          float mh[2];
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            float a8[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) a8[i] = x[h * 64 + i];
#pragma unroll
            for (int c = 8; c + 16 <= 64; c += 16)
#pragma unroll
              for (int i = 0; i < 8; ++i) a8[i] = fmax3(a8[i], x[h * 64 + c + i], x[h * 64 + c + 8 + i]);
#pragma unroll
            for (int i = 0; i < 8; ++i) a8[i] = fmaxf(a8[i], x[h * 64 + 56 + i]);
            mh[h] = fmax3(fmax3(a8[0], a8[1], a8[2]), fmax3(a8[3], a8[4], a8[5]), fmaxf(a8[6], a8[7]));
          }
          m_tile = fmaxf(mh[0] * s_lo, mh[1] * s_hi);
        } else {
          float a8[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) a8[i] = x[i];
#pragma unroll
          for (int c = 8; c + 16 <= 128; c += 16)
#pragma unroll
            for (int i = 0; i < 8; ++i) a8[i] = fmax3(a8[i], x[c + i], x[c + 8 + i]);
#pragma unroll
          for (int i = 0; i < 8; ++i) a8[i] = fmaxf(a8[i], x[120 + i]);
          m_tile = fmax3(fmax3(a8[0], a8[1], a8[2]), fmax3(a8[3], a8[4], a8[5]), fmaxf(a8[6], a8[7])) * s;
        }
        if (r == 0) ATTN_TRACE(6, qt, j);
        // e4m3 with the shared S buffer writes both P halves at once after the second half's
        // exponentials (its PVs are short, so an early first half buys little), and waits for
        // PV_{j-1} only there or before a rescale of O.
        constexpr bool LATE_P = C::S1 && C::FP8;
        if constexpr (C::S1 && !LATE_P) {
          // S_j may have been issued before PV_{j-1}: wait for that PV before P_j overwrites
          // P_{j-1} in this tile's P area and before any rescale of O.
          if (j > 0) {
            w = mbar_wait(smem_addr(&bar_o_done[qt]), (pv_cnt + j - 1) & 1, ctl, SITE_O_DONE);
            if (!__all_sync(0xffffffffu, w)) { ok = false; break; }
          }
        }
        float alpha = 1.0f;
        bool rescale = false;
        if (m_tile > m + 8.0f) {
          alpha = ex2(m - m_tile);   // 0 on the first tile (m = -inf)
          m = m_tile;
          rescale = true;
        }
        if (__any_sync(0xffffffffu, rescale)) {
          if (j > 0) {
            // Rescale O before any half of P_j is released: PV_j must accumulate onto the
            // rescaled O, and O must not be touched while PV_{j-1} is still accumulating into
            // it. Shared S buffer: PV_{j-1} was waited for above. One Q tile: S_j was issued
            // before PV_{j-1}; wait for that PV. Three S buffers: S_j comes from another warp,
            // so wait for PV_{j-1} as well.
            if constexpr (C::S3) {
              const uint32_t gp = gb + j - 1;   // this tile's PV_{j-1}
              w = mbar_wait(smem_addr(&bar_o_done[3 * qt + gp % 3u]), (gp / 3u) & 1u, ctl, SITE_O_DONE);
              if (!__all_sync(0xffffffffu, w)) { ok = false; break; }
            } else if constexpr (C::NQ == 1 || LATE_P) {
              w = mbar_wait(smem_addr(&bar_o_done[qt]), (pv_cnt + j - 1) & 1, ctl, SITE_O_DONE);
              if (!__all_sync(0xffffffffu, w)) { ok = false; break; }
            }
            tc_fence_after();
            const uint32_t tO = tmem + lane_base + C::O_COL + qt * C::D;
#pragma unroll 1
            for (int c0 = 0; c0 < C::D; c0 += 32) {
              uint32_t ov[32];
              tmem_ld_32cols(tO + c0, ov);
              tmem_ld_wait();
              reg_fence32(ov);
#pragma unroll
              for (int c = 0; c < 32; ++c) ov[c] = __float_as_uint(__uint_as_float(ov[c]) * alpha);
              tmem_st_32cols(tO + c0, ov);
            }
          }
          // The speculative half used the old shift: redo it with the new one.
          acc0 = f2_pack(0.f, 0.f);
          acc1 = acc0;
          exp_half(0, f2_pack(-m, -m), pk, acc0, acc1);
        }
        if constexpr (LATE_P) {
          uint32_t pk1[PKN];
          exp_half(1, f2_pack(-m, -m), pk1, acc0, acc1);
          if (r == 0) ATTN_TRACE(17, qt, j);
          // PV_{j-1} still reads P_{j-1} from this tile's P area. (After a rescale this phase has
          // completed already; o_done cannot complete another before P_j is handed over.)
          if (j > 0) {
            w = mbar_wait(smem_addr(&bar_o_done[qt]), (pv_cnt + j - 1) & 1, ctl, SITE_O_DONE);
            if (!__all_sync(0xffffffffu, w)) { ok = false; break; }
          }
          const uint32_t tP = tmem + lane_base + C::P_COL + (uint32_t)C::P_COLS * qt;
          tmem_st_16cols(tP, pk);
          tmem_st_16cols(tP + 16, pk1);
          tmem_st_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) {
            mbar_arrive(smem_addr(&bar_p_half[buf][0]));
            mbar_arrive(smem_addr(&bar_p_half[buf][1]));
          }
          if (r == 0) ATTN_TRACE(8, qt, j);
        } else {
          store_half(0, pk);
          exp_half(1, f2_pack(-m, -m), pk, acc0, acc1);
          if (r == 0) ATTN_TRACE(17, qt, j);
          store_half(1, pk);
        }
        float l0, l1, l2, l3;
        f2_unpack(acc0, l0, l1);
        f2_unpack(acc1, l2, l3);
        l = l * alpha + ((l0 + l1) + (l2 + l3));
      }
      if (!ok) break;
      // Epilogue: O / l -> bf16, LSE = (m + log2 l) * ln 2.
      bool w = mbar_wait(smem_addr(&bar_o_full[qt]), tiles_done & 1, ctl, SITE_O_FULL);
      if (!__all_sync(0xffffffffu, w)) { ok = false; break; }
      pv_cnt += n;
      ++tiles_done;
      tc_fence_after();
      const uint32_t tO = tmem + lane_base + C::O_COL + qt * C::D;
      const float lse_row = (m + log2f(l)) * 0.69314718055994531f;
      if constexpr (C::SPLIT) {
        // Partial result of this KV range: normalized O in fp32 and its LSE, row (position, head).
        const int pos = row0 + r / p.G;
        const int h = tc.h * p.G + r % p.G;
        const bool valid = pos < p.N;
        const float inv_l = out_scale / l;
        const size_t prow = (((size_t)tc.s * p.B + tc.b) * p.H + h) * p.N + (valid ? pos : 0);
        float* orow = p.part_o + prow * C::D;
#pragma unroll 1
        for (int c0 = 0; c0 < C::D; c0 += 32) {
          uint32_t ov[32];
          tmem_ld_32cols(tO + c0, ov);
          tmem_ld_wait();
          reg_fence32(ov);
          if (valid) {
            float4* dst = reinterpret_cast<float4*>(orow + c0);
#pragma unroll
            for (int v4 = 0; v4 < 8; ++v4)
              dst[v4] = make_float4(__uint_as_float(ov[4 * v4]) * inv_l, __uint_as_float(ov[4 * v4 + 1]) * inv_l,
                                    __uint_as_float(ov[4 * v4 + 2]) * inv_l, __uint_as_float(ov[4 * v4 + 3]) * inv_l);
          }
        }
        if (valid) p.part_lse[prow] = lse_row;
      } else {
        const int row = row0 + r;
        const bool valid = row < tc.nq;
        // Varlen: a row whose keys were all masked (its max never left -inf) gets O = 0 and
        // LSE = -inf; its accumulator holds no meaningful value.
        const bool empty_row = C::VARLEN && m == -INFINITY;
        float inv_l = out_scale / l;
        __nv_bfloat16* orow = reinterpret_cast<__nv_bfloat16*>(p.o) +
                              ((size_t)(tc.bo * p.N + tc.q_base + (valid ? row : 0)) * p.H + tc.h) * C::D;
        float* lse_dst = p.lse + ((size_t)tc.bo * p.H + tc.h) * p.N + tc.q_base + (valid ? row : 0);
        float lse_out = lse_row;
        // Second KV half of a halved tile: the first launch wrote this row's O_a (bf16) and LSE_a
        // over keys [0, tail_kvt). With this half's O_b and LSE_b over the rest, the row over all
        // keys is LSE = ln(e^LSE_a + e^LSE_b), O = e^(LSE_a - LSE) O_a + e^(LSE_b - LSE) O_b (the
        // split-KV combine for two ranges). Wait for the first grid to finish before reading.
        const bool merge = kDense && (p.tail_mode == 2 || p.tail_mode == 4);
        float w_a = 0.0f;
        if (merge) {
          griddep_wait();
          if (valid) {
            const float a2 = __ldcg(lse_dst) * 1.4426950408889634f;   // LSE_a in log2 units
            const float b2 = m + log2f(l);
            const float mx = fmaxf(a2, b2);
            const float ea = ex2(a2 - mx), eb = ex2(b2 - mx);
            const float inv = 1.0f / (ea + eb);
            w_a = ea * inv;
            inv_l *= eb * inv;
            lse_out = (mx + log2f(ea + eb)) * 0.69314718055994531f;
          }
        }
        // 64 columns per round: two TMEM loads behind one wait, then the row's 128 bytes of bf16
        // in 32-byte stores (one whole sector per lane) where o allows it.
#pragma unroll 1
        for (int c0 = 0; c0 < C::D; c0 += 64) {
          uint32_t ov[64];
          tmem_ld_32cols(tO + c0, ov);
          tmem_ld_32cols(tO + c0 + 32, ov + 32);
          tmem_ld_wait();
          reg_fence32(ov);
          reg_fence32(ov + 32);
          uint32_t pk[32];
          if (merge && valid) {
            // O_a of these 64 columns: 32 bf16 pairs, the lower-addressed element in the low half.
            const uint4* src = reinterpret_cast<const uint4*>(orow + c0);
#pragma unroll
            for (int v4 = 0; v4 < 8; ++v4) {
              const uint4 u = __ldcg(src + v4);
              const uint32_t wds[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                const int c = 8 * v4 + 2 * i;
                pk[c >> 1] = pack_bf16x2(fmaf(__uint_as_float(ov[c]), inv_l, __uint_as_float(wds[i] << 16) * w_a),
                                         fmaf(__uint_as_float(ov[c + 1]), inv_l,
                                              __uint_as_float(wds[i] & 0xFFFF0000u) * w_a));
              }
            }
          } else {
#pragma unroll
            for (int c = 0; c < 64; c += 2)
              pk[c >> 1] = empty_row ? 0u
                                     : pack_bf16x2(__uint_as_float(ov[c]) * inv_l, __uint_as_float(ov[c + 1]) * inv_l);
          }
          if (valid) {
            if (p.o_v8) {
#pragma unroll
              for (int v8 = 0; v8 < 4; ++v8) st_global_v8(orow + c0 + 16 * v8, pk + 8 * v8);
            } else {
              uint4* dst = reinterpret_cast<uint4*>(orow + c0);
#pragma unroll
              for (int v4 = 0; v4 < 8; ++v4)
                dst[v4] = make_uint4(pk[4 * v4], pk[4 * v4 + 1], pk[4 * v4 + 2], pk[4 * v4 + 3]);
            }
          }
        }
        if (valid) *lse_dst = empty_row ? -INFINITY : lse_out;
      }
    }
  }
  else {
    // Idle warps of the third warpgroup: give their registers back and wait for teardown.
    if constexpr (C::REG_SPLIT) setmaxnreg_dec<C::REGS_OTHER>();
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == C::WARP_MMA) tmem_dealloc(tmem, C::TMEM_COLS);
  // A second-half launch never finishes before the first launch, even where a failed wait kept
  // its epilogue from waiting, so work queued after it on the stream sees both.
  if (kDense && (p.tail_mode == 2 || p.tail_mode == 4)) griddep_wait();
}

}  // namespace gb300
