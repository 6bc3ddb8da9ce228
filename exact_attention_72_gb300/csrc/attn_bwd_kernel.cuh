// Backward pass of the fused attention forward on sm_103a: dQ, dK, dV from Q, K, V, dO, the
// forward's LSE and D = rowsum(dO * O).
//
// With S = scale Q K^T (+ causal mask), P = exp(S - LSE) row by row, dP = dO V^T and
// dS = P * (dP - D): dV = P^T dO, dK = scale dS^T Q, dQ = scale dS K. P is recomputed from the
// LSE the forward wrote; nothing else of the forward is kept. The pages name the pieces of the
// FA3 backward: recomputation, a preprocess that forms D and the base-2 LSE, dQ accumulation,
// the GQA path for dK and dV, and a longest-first scheduler for causal masking
// ("FlashAttention-3 Deep Dive" (mojostudio.in), its backward-pass sections; "flash-attention-3"
// (ai.thesatyajit.com), "Five schedulers").
//
// Two kernels, no atomics. Each recomputes S and dP on the tensor cores (tcgen05, fp32 in TMEM)
// and keeps one fp32 accumulator tile in TMEM for its whole loop:
//   * attn_bwd_dkdv_kernel: one CTA per (batch, kv head, 128-key tile j). It loops over every
//     query head of the kv head's group and every 128-row query tile i that sees tile j,
//     computing S^T = K_j Q_i^T and dP^T = V_j dO_i^T with keys as TMEM lanes, so P^T and dS^T
//     (bf16, written over S^T and dP^T in TMEM) are the A operands of dV += P^T dO_i and
//     dK += dS^T Q_i. The GQA sum over query heads happens inside the CTA.
//   * attn_bwd_dq_kernel: one CTA per (batch, query head, 128-row query tile i); it loops over
//     the key tiles j that tile i sees, computing S and dP with queries as lanes and
//     dQ += dS K_j with dS (bf16, written over S in TMEM) as the A operand. S is double-buffered
//     (TMEM has room here), so S_{j+1} runs while the elementwise warps work on step j, and K
//     and V stream through rings of their own (three and two stages).
// Both kernels are persistent; causal work tiles go longest first and are dealt to the CTAs in
// zig-zag turns (deal_tile).
// S and dP are computed twice in all (once per kernel): 7 tile GEMMs against 5 for a single
// kernel that accumulates dQ across CTAs, traded for deterministic results and no fp32 atomic
// traffic.
//
// Roles (576 threads): warps 0-15 elementwise, four warpgroups that split the 128 columns of a
// tile (thread = TMEM lane = one row, warpgroup g = columns 32g .. 32g+31); warp 16 issues the
// MMAs, warp 17 the TMA loads. In the dK/dV kernel the elementwise work of a step runs in two
// passes with their own barriers: P from S (the dV GEMM can start, while the dP GEMM may still
// run), then dS from dP. The dQ kernel forms dS in one pass.
// bf16 results are written in place over the fp32 columns they came from, so all warpgroups
// read their columns first and meet at a named barrier before any write: packed column c/2 of
// one group's columns lies in the fp32 columns of another. Every wait is bounded (status word + abort
// flag); on a failed wait the elementwise warps keep stepping through the named barriers without
// work, so no warp is left at a barrier.
#pragma once
#include "attn_fwd_kernel.cuh"

namespace gb300 {

struct BwdParams {
  __nv_bfloat16* dq;     // [B, N, H, D]
  __nv_bfloat16* dk;     // [B, N, Hkv, D]
  __nv_bfloat16* dv;     // [B, N, Hkv, D]
  const float* nlse2;    // [B, H, Np]: -LSE * log2(e); rows from N to Np: -inf
  const float* dd;       // [B, H, Np]: rowsum(dO * O); rows from N to Np: 0
  int B, H, Hkv, G, N, Np;   // Np: N rounded up to a multiple of 128
  int n_t;                   // 128-row tiles per sequence (queries and keys alike)
  float scale, scale_log2;
  int n_tiles;
  uint32_t* status;
  unsigned long long timeout_ns;
};

template <int D_, bool CAUSAL_>
struct BwdCfg {
  static constexpr int D = D_;
  static constexpr bool CAUSAL = CAUSAL_;
  static constexpr bool FP8 = false;
  static constexpr int BM = 128, BN = 128;
  static constexpr int CE = 64;                           // bf16 elements in one 128-byte row
  static constexpr int NCH = D / CE;
  static constexpr int CHUNK_BYTES = 128 * 128;
  static constexpr int SWZ = 128, SBO = 1024;             // 128-byte swizzle (issue_qk)
  static constexpr int TILE_BYTES = NCH * CHUNK_BYTES;    // 128 rows x D bf16
  static constexpr int KSTEPS_QK = D / 16;
  static constexpr int KSTEPS_PV = 8;                     // 128 rows of the MN-major B operand
  static constexpr int PV_ROWS = 16;
  static constexpr uint32_t IDESC_QK = make_idesc(kFmtBF16, 128, 128, false, false);
  static constexpr uint32_t IDESC_PV = make_idesc(kFmtBF16, 128, D, false, true);
  static constexpr int STAGES = 2;
  static constexpr int VEC_BYTES = 2 * 128 * 4;           // per stage: -LSE2 and D of 128 query rows
  // shared memory: two resident tiles, then STAGES x (two streamed tiles), then the vectors
  static constexpr int SMEM_USED = 2 * TILE_BYTES + STAGES * 2 * TILE_BYTES + STAGES * VEC_BYTES + 1024;
  // At least 116 KB so that one CTA holds an SM: each takes all 512 TMEM columns.
  static constexpr int SMEM_BYTES = SMEM_USED > 118784 ? SMEM_USED : 118784;
  // TMEM columns: S (or S^T, later P / dS in bf16) at 0, dP at 128, accumulators from 256
  static constexpr int S_COL = 0, DP_COL = 128, ACC0 = 256, ACC1 = 256 + D;
  static constexpr int TMEM_COLS = 512;
  // Elementwise warpgroups: each takes CPG of the tile's 128 columns for all 128 rows (lanes).
  static constexpr int EWG = 4;
  static constexpr int CPG = 128 / EWG;
  static constexpr int EW_THREADS = 128 * EWG;
  static constexpr int EW_WARPS = 4 * EWG;                 // arrivals on the elementwise barriers
  static constexpr int WARP_MMA = 4 * EWG, WARP_LOAD = 4 * EWG + 1;
  static constexpr int THREADS = (4 * EWG + 2) * 32;
  // dQ kernel shared memory: Q and dO, then a K ring and a V ring of their own
  static constexpr int DQ_KS = 3, DQ_VS = 2;
  static constexpr int DQ_SMEM_USED = 2 * TILE_BYTES + (DQ_KS + DQ_VS) * TILE_BYTES + 1024;
  static constexpr int DQ_SMEM_BYTES = DQ_SMEM_USED > 118784 ? DQ_SMEM_USED : 118784;
  // dQ kernel: S double buffer at 0 and 128, dP at 256, dQ at 384
  static constexpr int Q_S0 = 0, Q_S1 = 128, Q_DP = 256, Q_ACC = 384;
  static_assert(ACC1 + D <= TMEM_COLS, "TMEM budget: head dim up to 128");
  static_assert(Q_ACC + D <= TMEM_COLS, "TMEM budget (dQ kernel)");
  static_assert(SMEM_BYTES <= 232448, "shared memory budget");
  static_assert(DQ_SMEM_BYTES <= 232448 - 1024, "shared memory budget (dQ kernel; 1 KB static)");
};

// One arrival per warp: every lane has finished what precedes the call (its own tcgen05 waits and
// fences included) before lane 0 arrives. The barrier counts warps, not threads.
__device__ __forceinline__ void warp_arrive(uint32_t bar) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(bar);
}

enum : uint32_t { SITE_B_KV = 21, SITE_B_ST = 22, SITE_B_S = 23, SITE_B_P = 24, SITE_B_ACC = 25, SITE_B_EMPTY = 26 };

// dst (+)= A[tmem, bf16, 128 x 128] * B[smem, 128 x D, MN-major]: 8 k-steps of 16.
template <class C>
__device__ __forceinline__ void issue_ts_128(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_addr, bool accumulate) {
  const uint64_t b0 = make_sdesc_sw128(b_addr, C::CHUNK_BYTES, 1024);
#pragma unroll
  for (int kk = 0; kk < C::KSTEPS_PV; ++kk)
    mma_f16_ts(d_tmem, a_tmem + kk * 8, b0 + (uint64_t)((kk * C::PV_ROWS * 128) >> 4), C::IDESC_PV,
               (accumulate || kk > 0) ? 1u : 0u);
}

// Writes columns [c_begin, c_end) of the lane's row of an fp32 accumulator (at tcol) times `mul`
// as bf16 to dst (the row's first column).
__device__ __forceinline__ void store_acc_row(uint32_t tcol, int c_begin, int c_end, float mul, __nv_bfloat16* dst,
                                              bool valid) {
#pragma unroll 1
  for (int c0 = c_begin; c0 < c_end; c0 += 32) {
    uint32_t v[32];
    tmem_ld_32cols(tcol + c0, v);
    tmem_ld_wait();
    reg_fence32(v);
    uint32_t pk[16];
#pragma unroll
    for (int c = 0; c < 32; c += 2) pk[c >> 1] = pack_bf16x2(__uint_as_float(v[c]) * mul, __uint_as_float(v[c + 1]) * mul);
    if (valid) {
      uint4* d4 = reinterpret_cast<uint4*>(dst + c0);
#pragma unroll
      for (int i = 0; i < 4; ++i) d4[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
    }
  }
}

// Loads N (32 or 64) fp32 columns of the lane's row into x.
template <int N>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, float* x) {
  uint32_t a[N];
#pragma unroll
  for (int h = 0; h < N / 32; ++h) tmem_ld_32cols(taddr + 32 * h, a + 32 * h);
  tmem_ld_wait();
#pragma unroll
  for (int h = 0; h < N / 32; ++h) reg_fence32(a + 32 * h);
#pragma unroll
  for (int c = 0; c < N; ++c) x[c] = __uint_as_float(a[c]);
}

// Packs N values as bf16 pairs and writes them as N / 2 columns at taddr.
template <int N>
__device__ __forceinline__ void tmem_st_as_bf16(uint32_t taddr, const float* x) {
  uint32_t pk[16];
#pragma unroll
  for (int h = 0; h < N / 32; ++h) {
#pragma unroll
    for (int c = 0; c < 16; ++c) pk[c] = pack_bf16x2(x[32 * h + 2 * c], x[32 * h + 2 * c + 1]);
    tmem_st_16cols(taddr + 16 * h, pk);
  }
}

// ---------------------------------------------------------------------------------------------
// dK, dV: one CTA per (b, kv head, key tile j); steps over (query head g of the group, tile i).
// Causal: tile j is seen by query tiles i >= j; tiles go in ascending j (the longest first).
// ---------------------------------------------------------------------------------------------
template <class C>
__global__ void __launch_bounds__(C::THREADS, 1)
attn_bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                     const BwdParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bar_kv_full, bar_kv_empty, bar_st_full[C::STAGES], bar_st_empty[C::STAGES];
  __shared__ __align__(8) uint64_t bar_s_full, bar_dp_full, bar_p_ready, bar_ds_ready, bar_acc_full, bar_acc_empty;
  __shared__ __align__(8) uint64_t bar_drain;
  __shared__ uint32_t tmem_slot;
  __shared__ volatile uint32_t abort_flag;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sK = smem_addr(smem), sV = sK + C::TILE_BYTES;
  const uint32_t sStage = sV + C::TILE_BYTES;                          // stage s: Q at +0, dO at +TILE
  float* vec = reinterpret_cast<float*>(smem + 2 * C::TILE_BYTES + C::STAGES * 2 * C::TILE_BYTES);
  const WaitCtl ctl{&abort_flag, p.status, p.timeout_ns};
  if (tid == 0) {
    abort_flag = 0u;
    mbar_init(smem_addr(&bar_kv_full), 1);
    mbar_init(smem_addr(&bar_kv_empty), 1);
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(smem_addr(&bar_st_full[s]), 1);
      mbar_init(smem_addr(&bar_st_empty[s]), 1);
    }
    mbar_init(smem_addr(&bar_s_full), 1);
    mbar_init(smem_addr(&bar_dp_full), 1);
    mbar_init(smem_addr(&bar_p_ready), C::EW_WARPS);
    mbar_init(smem_addr(&bar_ds_ready), C::EW_WARPS);
    mbar_init(smem_addr(&bar_acc_full), 1);
    mbar_init(smem_addr(&bar_acc_empty), C::EW_WARPS);
    mbar_init(smem_addr(&bar_drain), 1);
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
  const int BHkv = p.B * p.Hkv;
  // work tile t -> (b, kv head, key tile j); steps of the tile
  auto decode = [&](int t, int& b, int& kvh, int& j, int& i0) {
    j = t / BHkv;
    const int bh = t % BHkv;
    b = bh / p.Hkv;
    kvh = bh % p.Hkv;
    i0 = C::CAUSAL ? j : 0;
  };

  if (warp == C::WARP_LOAD) {
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      tma_prefetch_desc(&tm_do);
      uint32_t tiles = 0, steps = 0;
      bool ok = true;
      for (int turn = 0, t = deal_tile<C::CAUSAL>(0); ok && t < p.n_tiles; t = deal_tile<C::CAUSAL>(++turn)) {
        int b, kvh, j, i0;
        decode(t, b, kvh, j, i0);
        if (tiles > 0 && !mbar_wait(smem_addr(&bar_kv_empty), (tiles - 1) & 1, ctl, SITE_B_EMPTY)) { ok = false; break; }
        mbar_arrive_expect_tx(smem_addr(&bar_kv_full), 2 * C::TILE_BYTES);
        for (int ch = 0; ch < C::NCH; ++ch) {
          tma_load_4d(sK + ch * C::CHUNK_BYTES, &tm_k, smem_addr(&bar_kv_full), ch * C::CE, j * 128, kvh, b);
          tma_load_4d(sV + ch * C::CHUNK_BYTES, &tm_v, smem_addr(&bar_kv_full), ch * C::CE, j * 128, kvh, b);
        }
        ++tiles;
        const int ni = p.n_t - i0;
        for (int k = 0; ok && k < p.G * ni; ++k) {
          const int h = kvh * p.G + k / ni, i = i0 + k % ni;
          const int s = steps % C::STAGES;
          if (steps >= (uint32_t)C::STAGES &&
              !mbar_wait(smem_addr(&bar_st_empty[s]), ((steps / C::STAGES) - 1) & 1, ctl, SITE_B_EMPTY)) {
            ok = false;
            break;
          }
          const uint32_t bar = smem_addr(&bar_st_full[s]);
          const uint32_t dst = sStage + s * 2 * C::TILE_BYTES;
          mbar_arrive_expect_tx(bar, 2 * C::TILE_BYTES + C::VEC_BYTES);
          for (int ch = 0; ch < C::NCH; ++ch) {
            tma_load_4d(dst + ch * C::CHUNK_BYTES, &tm_q, bar, ch * C::CE, i * 128, h, b);
            tma_load_4d(dst + C::TILE_BYTES + ch * C::CHUNK_BYTES, &tm_do, bar, ch * C::CE, i * 128, h, b);
          }
          const size_t row = ((size_t)b * p.H + h) * p.Np + (size_t)i * 128;
          bulk_load(smem_addr(vec + s * 256), p.nlse2 + row, 512, bar);
          bulk_load(smem_addr(vec + s * 256 + 128), p.dd + row, 512, bar);
          ++steps;
        }
      }
      if (!ok) {
        // let copies still in flight land before the CTA exits
        for (uint32_t q = steps > (uint32_t)C::STAGES ? steps - C::STAGES : 0u; q < steps; ++q) {
          const uint64_t t0 = global_timer_ns();
          while (!mbar_try_wait(smem_addr(&bar_st_full[q % C::STAGES]), (q / C::STAGES) & 1) &&
                 global_timer_ns() - t0 < p.timeout_ns) {}
        }
        if (tiles > 0) {
          const uint64_t t0 = global_timer_ns();
          while (!mbar_try_wait(smem_addr(&bar_kv_full), (tiles - 1) & 1) && global_timer_ns() - t0 < p.timeout_ns) {}
        }
      }
    }
  } else if (warp == C::WARP_MMA) {
    if (lane == 0) {
      uint32_t tiles = 0, steps = 0;
      bool ok = true;
      for (int turn = 0, t = deal_tile<C::CAUSAL>(0); ok && t < p.n_tiles; t = deal_tile<C::CAUSAL>(++turn)) {
        int b, kvh, j, i0;
        decode(t, b, kvh, j, i0);
        if (!mbar_wait(smem_addr(&bar_kv_full), tiles & 1, ctl, SITE_B_KV)) { ok = false; break; }
        // Issue order per step k: dV_k, S^T_{k+1}, dK_k, dP^T_{k+1}. S^T_{k+1} overwrites P^T_k and
        // dP^T_{k+1} overwrites dS^T_k, each after the GEMM that reads them (the MMAs of one thread
        // run in issue order), so the next step's S^T runs while the elementwise warps form dS^T_k.
        const int n = p.G * (p.n_t - i0);
        auto stage_q = [&](uint32_t st) { return sStage + (st % C::STAGES) * 2 * C::TILE_BYTES; };
        auto issue_st = [&](uint32_t st) -> bool {
          if (!mbar_wait(smem_addr(&bar_st_full[st % C::STAGES]), (st / C::STAGES) & 1, ctl, SITE_B_ST)) return false;
          tc_fence_after();
          issue_qk<C>(tmem + C::S_COL, sK, stage_q(st));     // S^T = K_j Q_i^T
          tc_commit(smem_addr(&bar_s_full));
          return true;
        };
        auto issue_dpt = [&](uint32_t st) {
          issue_qk<C>(tmem + C::DP_COL, sV, stage_q(st) + C::TILE_BYTES);   // dP^T = V_j dO_i^T
          tc_commit(smem_addr(&bar_dp_full));
        };
        if (!issue_st(steps)) { ok = false; break; }
        issue_dpt(steps);
        // K and V are read by the S^T and dP^T GEMMs only: free them after the tile's last dP^T.
        if (n == 1) tc_commit(smem_addr(&bar_kv_empty));
        for (int k = 0; k < n; ++k) {
          const uint32_t cur = steps + k;
          const uint32_t sQ = stage_q(cur), sdO = sQ + C::TILE_BYTES;
          if (!mbar_wait(smem_addr(&bar_p_ready), cur & 1, ctl, SITE_B_P)) { ok = false; break; }
          if (k == 0 && tiles > 0 &&
              !mbar_wait(smem_addr(&bar_acc_empty), (tiles - 1) & 1, ctl, SITE_B_ACC)) { ok = false; break; }
          tc_fence_after();
          issue_ts_128<C>(tmem + C::ACC0, tmem + C::S_COL, sdO, k > 0);    // dV += P^T dO_i
          if (k + 1 < n && !issue_st(cur + 1)) { ok = false; break; }
          if (!mbar_wait(smem_addr(&bar_ds_ready), cur & 1, ctl, SITE_B_P)) { ok = false; break; }
          tc_fence_after();
          issue_ts_128<C>(tmem + C::ACC1, tmem + C::DP_COL, sQ, k > 0);    // dK += dS^T Q_i
          tc_commit(smem_addr(&bar_st_empty[cur % C::STAGES]));
          if (k + 1 < n) {
            issue_dpt(cur + 1);
            if (k + 2 == n) tc_commit(smem_addr(&bar_kv_empty));
          }
        }
        if (!ok) break;
        steps += n;
        tc_commit(smem_addr(&bar_acc_full));
        ++tiles;
      }
      tc_commit(smem_addr(&bar_drain));
      const uint64_t t0 = global_timer_ns();
      while (!mbar_try_wait(smem_addr(&bar_drain), 0) && global_timer_ns() - t0 < p.timeout_ns) {}
    }
  } else if (warp < C::WARP_MMA) {
    // elementwise: thread = key row r of the tile (TMEM lane), warpgroup wg = query columns
    // CPG wg .. CPG wg + CPG - 1
    const int wg = warp >> 2;
    const int r = (warp & 3) * 32 + lane;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_base + C::S_COL, tP = tmem + lane_base + C::DP_COL;
    uint32_t tiles = 0, steps = 0;
    bool ok = true;
    for (int turn = 0, t = deal_tile<C::CAUSAL>(0); t < p.n_tiles; t = deal_tile<C::CAUSAL>(++turn)) {
      int b, kvh, j, i0;
      decode(t, b, kvh, j, i0);
      const int key = j * 128 + r;
      const int ni = p.n_t - i0;
      for (int k = 0; k < p.G * ni; ++k) {
        const int i = i0 + k % ni;
        const int s = steps % C::STAGES;
        // pass 1: P^T from S^T (this stage's LSE2 / D vectors are in shared memory; the stage is
        // not refilled before this step's ds_ready arrival)
        bool w = ok && mbar_wait(smem_addr(&bar_s_full), steps & 1, ctl, SITE_B_S);
        w = w && mbar_wait(smem_addr(&bar_st_full[s]), (steps / C::STAGES) & 1, ctl, SITE_B_ST);
        ok = __all_sync(0xffffffffu, w);
        // this group's query columns of -LSE2 and D, as float4 (broadcast reads)
        const float4* nl4 = reinterpret_cast<const float4*>(vec + s * 256 + wg * C::CPG);
        const float4* dd4 = reinterpret_cast<const float4*>(vec + s * 256 + 128 + wg * C::CPG);
        const bool diag = C::CAUSAL && i == j;
        float pf[C::CPG];
        if (ok) {
          tc_fence_after();
          tmem_ld_cols<C::CPG>(tS + wg * C::CPG, pf);
          const uint64_t sl2 = f2_pack(p.scale_log2, p.scale_log2);
#pragma unroll
          for (int c = 0; c < C::CPG; c += 4) {
            const float4 nl = nl4[c >> 2];
            float t0, t1, t2, t3;
            f2_unpack(f2_fma(f2_pack(pf[c], pf[c + 1]), sl2, f2_pack(nl.x, nl.y)), t0, t1);
            f2_unpack(f2_fma(f2_pack(pf[c + 2], pf[c + 3]), sl2, f2_pack(nl.z, nl.w)), t2, t3);
            pf[c] = ex2(t0);
            pf[c + 1] = ex2(t1);
            pf[c + 2] = ex2(t2);
            pf[c + 3] = ex2(t3);
          }
          if (diag) {
#pragma unroll
            for (int c = 0; c < C::CPG; ++c)
              if (wg * C::CPG + c < r) pf[c] = 0.0f;   // key after the query
          }
        }
        named_bar_sync(1, C::EW_THREADS);   // every S^T column read before any P^T write
        if (ok) {
          tmem_st_as_bf16<C::CPG>(tS + wg * (C::CPG / 2), pf);
          tmem_st_wait();
          tc_fence_before();
          warp_arrive(smem_addr(&bar_p_ready));
        }
        // pass 2: dS^T = P^T * (dP^T - D)
        w = ok && mbar_wait(smem_addr(&bar_dp_full), steps & 1, ctl, SITE_B_S);
        ok = __all_sync(0xffffffffu, w);
        if (ok) {
          float dp[C::CPG];
          tc_fence_after();
          tmem_ld_cols<C::CPG>(tP + wg * C::CPG, dp);
#pragma unroll
          for (int c = 0; c < C::CPG; c += 4) {
            const float4 d4 = dd4[c >> 2];
            f2_unpack(f2_mul(f2_pack(pf[c], pf[c + 1]), f2_sub(f2_pack(dp[c], dp[c + 1]), f2_pack(d4.x, d4.y))), pf[c],
                      pf[c + 1]);
            f2_unpack(f2_mul(f2_pack(pf[c + 2], pf[c + 3]), f2_sub(f2_pack(dp[c + 2], dp[c + 3]), f2_pack(d4.z, d4.w))),
                      pf[c + 2], pf[c + 3]);
          }
        }
        named_bar_sync(2, C::EW_THREADS);   // every dP^T column read before any dS^T write
        if (ok) {
          tmem_st_as_bf16<C::CPG>(tP + wg * (C::CPG / 2), pf);
          tmem_st_wait();
          tc_fence_before();
          warp_arrive(smem_addr(&bar_ds_ready));
        }
        ++steps;
      }
      // epilogue: the first half of the warpgroups write dV, the second half dK, each a range of
      // the D columns
      bool w = ok && mbar_wait(smem_addr(&bar_acc_full), tiles & 1, ctl, SITE_B_ACC);
      ok = __all_sync(0xffffffffu, w);
      if (ok) {
        tc_fence_after();
        const bool valid = key < p.N;
        const size_t orow = ((size_t)(b * p.N + (valid ? key : 0)) * p.Hkv + kvh) * C::D;
        constexpr int HALF = C::EWG / 2, W = C::D / HALF;
        const int part = wg % HALF;
        if (wg < HALF) store_acc_row(tmem + lane_base + C::ACC0, part * W, (part + 1) * W, 1.0f, p.dv + orow, valid);
        else store_acc_row(tmem + lane_base + C::ACC1, part * W, (part + 1) * W, p.scale, p.dk + orow, valid);
        tc_fence_before();
        warp_arrive(smem_addr(&bar_acc_empty));
      }
      ++tiles;
    }
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == C::WARP_MMA) tmem_dealloc(tmem, C::TMEM_COLS);
}

// ---------------------------------------------------------------------------------------------
// dQ: one CTA per (b, query head, query tile i); steps over the key tiles i sees.
// Causal: tile i sees key tiles j <= i; tiles go in descending i (the longest first).
// ---------------------------------------------------------------------------------------------
template <class C>
__global__ void __launch_bounds__(C::THREADS, 1)
attn_bwd_dq_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                   const BwdParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bar_q_full, bar_q_empty, bar_k_full[C::DQ_KS], bar_k_empty[C::DQ_KS];
  __shared__ __align__(8) uint64_t bar_v_full[C::DQ_VS], bar_v_empty[C::DQ_VS];
  __shared__ __align__(8) uint64_t bar_s_full2[2], bar_dp_full, bar_ds_ready, bar_acc_full, bar_acc_empty, bar_drain;
  __shared__ uint32_t tmem_slot;
  __shared__ volatile uint32_t abort_flag;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sQ = smem_addr(smem), sdO = sQ + C::TILE_BYTES;
  // K and V have rings of their own: K_j is read by S_j and, a step later, by dQ_j; V_j only by
  // dP_j. A third K stage lets K_{j+2} load while dQ_j still reads K_j.
  const uint32_t sK = sdO + C::TILE_BYTES, sV = sK + C::DQ_KS * C::TILE_BYTES;
  const WaitCtl ctl{&abort_flag, p.status, p.timeout_ns};
  if (tid == 0) {
    abort_flag = 0u;
    mbar_init(smem_addr(&bar_q_full), 1);
    mbar_init(smem_addr(&bar_q_empty), 1);
    for (int s = 0; s < C::DQ_KS; ++s) {
      mbar_init(smem_addr(&bar_k_full[s]), 1);
      mbar_init(smem_addr(&bar_k_empty[s]), 1);
    }
    for (int s = 0; s < C::DQ_VS; ++s) {
      mbar_init(smem_addr(&bar_v_full[s]), 1);
      mbar_init(smem_addr(&bar_v_empty[s]), 1);
    }
    mbar_init(smem_addr(&bar_s_full2[0]), 1);
    mbar_init(smem_addr(&bar_s_full2[1]), 1);
    mbar_init(smem_addr(&bar_dp_full), 1);
    mbar_init(smem_addr(&bar_ds_ready), C::EW_WARPS);
    mbar_init(smem_addr(&bar_acc_full), 1);
    mbar_init(smem_addr(&bar_acc_empty), C::EW_WARPS);
    mbar_init(smem_addr(&bar_drain), 1);
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
  const int BH = p.B * p.H;
  auto decode = [&](int t, int& b, int& h, int& i, int& nj) {
    i = C::CAUSAL ? p.n_t - 1 - t / BH : t / BH;
    const int bh = t % BH;
    b = bh / p.H;
    h = bh % p.H;
    nj = C::CAUSAL ? i + 1 : p.n_t;
  };

  if (warp == C::WARP_LOAD) {
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      tma_prefetch_desc(&tm_do);
      uint32_t tiles = 0, kq = 0, vq = 0;   // work tiles, K loads and V loads issued
      bool ok = true;
      for (int turn = 0, t = deal_tile<C::CAUSAL>(0); ok && t < p.n_tiles; t = deal_tile<C::CAUSAL>(++turn)) {
        int b, h, i, nj;
        decode(t, b, h, i, nj);
        const int kvh = h / p.G;
        if (tiles > 0 && !mbar_wait(smem_addr(&bar_q_empty), (tiles - 1) & 1, ctl, SITE_B_EMPTY)) { ok = false; break; }
        mbar_arrive_expect_tx(smem_addr(&bar_q_full), 2 * C::TILE_BYTES);
        for (int ch = 0; ch < C::NCH; ++ch) {
          tma_load_4d(sQ + ch * C::CHUNK_BYTES, &tm_q, smem_addr(&bar_q_full), ch * C::CE, i * 128, h, b);
          tma_load_4d(sdO + ch * C::CHUNK_BYTES, &tm_do, smem_addr(&bar_q_full), ch * C::CE, i * 128, h, b);
        }
        ++tiles;
        for (int jj = 0; ok && jj < nj; ++jj) {
          const int ks = kq % C::DQ_KS, vs = vq % C::DQ_VS;
          if (kq >= (uint32_t)C::DQ_KS &&
              !mbar_wait(smem_addr(&bar_k_empty[ks]), ((kq / C::DQ_KS) - 1) & 1, ctl, SITE_B_EMPTY)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(smem_addr(&bar_k_full[ks]), C::TILE_BYTES);
          for (int ch = 0; ch < C::NCH; ++ch)
            tma_load_4d(sK + ks * C::TILE_BYTES + ch * C::CHUNK_BYTES, &tm_k, smem_addr(&bar_k_full[ks]), ch * C::CE,
                        jj * 128, kvh, b);
          ++kq;
          if (vq >= (uint32_t)C::DQ_VS &&
              !mbar_wait(smem_addr(&bar_v_empty[vs]), ((vq / C::DQ_VS) - 1) & 1, ctl, SITE_B_EMPTY)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(smem_addr(&bar_v_full[vs]), C::TILE_BYTES);
          for (int ch = 0; ch < C::NCH; ++ch)
            tma_load_4d(sV + vs * C::TILE_BYTES + ch * C::CHUNK_BYTES, &tm_v, smem_addr(&bar_v_full[vs]), ch * C::CE,
                        jj * 128, kvh, b);
          ++vq;
        }
      }
      if (!ok) {
        // let copies still in flight land before the CTA exits
        for (uint32_t q = kq > (uint32_t)C::DQ_KS ? kq - C::DQ_KS : 0u; q < kq; ++q) {
          const uint64_t t0 = global_timer_ns();
          while (!mbar_try_wait(smem_addr(&bar_k_full[q % C::DQ_KS]), (q / C::DQ_KS) & 1) &&
                 global_timer_ns() - t0 < p.timeout_ns) {}
        }
        for (uint32_t q = vq > (uint32_t)C::DQ_VS ? vq - C::DQ_VS : 0u; q < vq; ++q) {
          const uint64_t t0 = global_timer_ns();
          while (!mbar_try_wait(smem_addr(&bar_v_full[q % C::DQ_VS]), (q / C::DQ_VS) & 1) &&
                 global_timer_ns() - t0 < p.timeout_ns) {}
        }
        if (tiles > 0) {
          const uint64_t t0 = global_timer_ns();
          while (!mbar_try_wait(smem_addr(&bar_q_full), (tiles - 1) & 1) && global_timer_ns() - t0 < p.timeout_ns) {}
        }
      }
    }
  } else if (warp == C::WARP_MMA) {
    if (lane == 0) {
      // Per step j: S_{j+1} into the other S buffer, then (once dS_j is in TMEM) dP_{j+1}, then
      // dQ_j. dP_{j+1} overwrites dP_j, which the elementwise warps read before writing dS_j; it
      // runs ahead of dQ_j so the next elementwise pass finds it done.
      uint32_t tiles = 0, steps = 0;
      bool ok = true;
      auto issue_s = [&](uint32_t st) -> bool {
        if (!mbar_wait(smem_addr(&bar_k_full[st % C::DQ_KS]), (st / C::DQ_KS) & 1, ctl, SITE_B_ST)) return false;
        tc_fence_after();
        issue_qk<C>(tmem + ((st & 1) ? C::Q_S1 : C::Q_S0), sQ, sK + (st % C::DQ_KS) * C::TILE_BYTES);   // S = Q_i K_j^T
        tc_commit(smem_addr(&bar_s_full2[st & 1]));
        return true;
      };
      auto issue_dp = [&](uint32_t st) -> bool {
        if (!mbar_wait(smem_addr(&bar_v_full[st % C::DQ_VS]), (st / C::DQ_VS) & 1, ctl, SITE_B_ST)) return false;
        tc_fence_after();
        issue_qk<C>(tmem + C::Q_DP, sdO, sV + (st % C::DQ_VS) * C::TILE_BYTES);           // dP = dO_i V_j^T
        tc_commit(smem_addr(&bar_dp_full));
        tc_commit(smem_addr(&bar_v_empty[st % C::DQ_VS]));
        return true;
      };
      for (int turn = 0, t = deal_tile<C::CAUSAL>(0); ok && t < p.n_tiles; t = deal_tile<C::CAUSAL>(++turn)) {
        int b, h, i, nj;
        decode(t, b, h, i, nj);
        if (!mbar_wait(smem_addr(&bar_q_full), tiles & 1, ctl, SITE_B_KV)) { ok = false; break; }
        if (!issue_s(steps) || !issue_dp(steps)) { ok = false; break; }
        // Q and dO are read by the S and dP GEMMs only: free them after the tile's last dP.
        if (nj == 1) tc_commit(smem_addr(&bar_q_empty));
        for (int jj = 0; jj < nj; ++jj) {
          const uint32_t cur = steps + jj;
          if (jj + 1 < nj && !issue_s(cur + 1)) { ok = false; break; }
          if (!mbar_wait(smem_addr(&bar_ds_ready), cur & 1, ctl, SITE_B_P)) { ok = false; break; }
          if (jj + 1 < nj) {
            if (!issue_dp(cur + 1)) { ok = false; break; }
            if (jj + 2 == nj) tc_commit(smem_addr(&bar_q_empty));
          }
          if (jj == 0 && tiles > 0 &&
              !mbar_wait(smem_addr(&bar_acc_empty), (tiles - 1) & 1, ctl, SITE_B_ACC)) { ok = false; break; }
          tc_fence_after();
          issue_ts_128<C>(tmem + C::Q_ACC, tmem + ((cur & 1) ? C::Q_S1 : C::Q_S0),
                          sK + (cur % C::DQ_KS) * C::TILE_BYTES, jj > 0);   // dQ += dS K_j
          tc_commit(smem_addr(&bar_k_empty[cur % C::DQ_KS]));
        }
        if (!ok) break;
        steps += nj;
        tc_commit(smem_addr(&bar_acc_full));
        ++tiles;
      }
      tc_commit(smem_addr(&bar_drain));
      const uint64_t t0 = global_timer_ns();
      while (!mbar_try_wait(smem_addr(&bar_drain), 0) && global_timer_ns() - t0 < p.timeout_ns) {}
    }
  } else if (warp < C::WARP_MMA) {
    // elementwise: thread = query row r of the tile (TMEM lane), warpgroup wg = key columns
    // CPG wg .. CPG wg + CPG - 1
    const int wg = warp >> 2;
    const int r = (warp & 3) * 32 + lane;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    uint32_t tiles = 0, steps = 0;
    bool ok = true;
    for (int turn = 0, t = deal_tile<C::CAUSAL>(0); t < p.n_tiles; t = deal_tile<C::CAUSAL>(++turn)) {
      int b, h, i, nj;
      decode(t, b, h, i, nj);
      const int qrow = i * 128 + r;
      const size_t vrow = ((size_t)b * p.H + h) * p.Np + qrow;   // padded rows: +inf / 0
      const float nlse2 = __ldg(p.nlse2 + vrow), dd = __ldg(p.dd + vrow);
      const uint64_t sl2 = f2_pack(p.scale_log2, p.scale_log2), nl2 = f2_pack(nlse2, nlse2), dd2 = f2_pack(dd, dd);
      for (int jj = 0; jj < nj; ++jj) {
        const uint32_t tS = tmem + lane_base + ((steps & 1) ? C::Q_S1 : C::Q_S0);
        const bool diag = C::CAUSAL && jj == i;
        const bool tail = jj == p.n_t - 1 && (p.N & 127) != 0;
        const int lim = diag ? r + 1 : (tail ? (p.N & 127) : 128);   // keys of this tile the row sees
        bool w = ok && mbar_wait(smem_addr(&bar_s_full2[steps & 1]), (steps >> 1) & 1, ctl, SITE_B_S);
        ok = __all_sync(0xffffffffu, w);
        float pf[C::CPG];
        if (ok) {
          tc_fence_after();
          tmem_ld_cols<C::CPG>(tS + wg * C::CPG, pf);
#pragma unroll
          for (int c = 0; c < C::CPG; c += 2) {
            float t0, t1;
            f2_unpack(f2_fma(f2_pack(pf[c], pf[c + 1]), sl2, nl2), t0, t1);
            pf[c] = wg * C::CPG + c < lim ? ex2(t0) : 0.0f;
            pf[c + 1] = wg * C::CPG + c + 1 < lim ? ex2(t1) : 0.0f;
          }
        }
        w = ok && mbar_wait(smem_addr(&bar_dp_full), steps & 1, ctl, SITE_B_S);
        ok = __all_sync(0xffffffffu, w);
        if (ok) {
          float dp[C::CPG];
          tc_fence_after();
          tmem_ld_cols<C::CPG>(tmem + lane_base + C::Q_DP + wg * C::CPG, dp);
#pragma unroll
          for (int c = 0; c < C::CPG; c += 2)
            f2_unpack(f2_mul(f2_pack(pf[c], pf[c + 1]), f2_sub(f2_pack(dp[c], dp[c + 1]), dd2)), pf[c], pf[c + 1]);
        }
        named_bar_sync(1, C::EW_THREADS);   // every S and dP column read before any dS write
        if (ok) {
          tmem_st_as_bf16<C::CPG>(tS + wg * (C::CPG / 2), pf);   // dS over this step's S buffer
          tmem_st_wait();
          tc_fence_before();
          warp_arrive(smem_addr(&bar_ds_ready));
        }
        ++steps;
      }
      bool w = ok && mbar_wait(smem_addr(&bar_acc_full), tiles & 1, ctl, SITE_B_ACC);
      ok = __all_sync(0xffffffffu, w);
      if (ok) {
        tc_fence_after();
        const bool valid = qrow < p.N;
        const size_t orow = ((size_t)(b * p.N + (valid ? qrow : 0)) * p.H + h) * C::D;
        constexpr int NG = (C::D / 32 < C::EWG) ? C::D / 32 : C::EWG;   // 32-column pieces per group
        if (wg < NG)
          store_acc_row(tmem + lane_base + C::Q_ACC, wg * (C::D / NG), (wg + 1) * (C::D / NG), p.scale, p.dq + orow,
                        valid);
        tc_fence_before();
        warp_arrive(smem_addr(&bar_acc_empty));
      }
      ++tiles;
    }
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == C::WARP_MMA) tmem_dealloc(tmem, C::TMEM_COLS);
}

// D = rowsum(dO * O) and -LSE * log2(e), per (b, h, row), rows padded to Np (D = 0, -LSE2 = -inf).
template <int D>
__global__ void __launch_bounds__(256) attn_bwd_preprocess_kernel(const __nv_bfloat16* o, const __nv_bfloat16* dout,
                                                                 const float* lse, float* nlse2, float* dd, int B,
                                                                 int H, int N, int Np) {
  const long long w = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);   // one warp per row
  const int lane = threadIdx.x & 31;
  if (w >= (long long)B * H * Np) return;
  const int row = (int)(w % Np);
  const long long bh = w / Np;
  const int h = (int)(bh % H), b = (int)(bh / H);
  float acc = 0.0f;
  if (row < N) {
    const size_t base = ((size_t)(b * N + row) * H + h) * D;
#pragma unroll
    for (int c = lane * 2; c < D; c += 64) {
      const float2 x = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(o + base + c));
      const float2 y = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(dout + base + c));
      acc = fmaf(x.x, y.x, fmaf(x.y, y.y, acc));
    }
  }
#pragma unroll
  for (int m = 16; m > 0; m >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, m);
  if (lane == 0) {
    dd[w] = acc;
    nlse2[w] = row < N ? lse[bh * N + row] * -1.4426950408889634f : -INFINITY;
  }
}

}  // namespace gb300
