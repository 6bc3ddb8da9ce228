// attn_quantize_e4m3: bf16 rows -> e4m3 codes with one fp32 descale per block of rows of one
// (batch, head), optionally after a random Hadamard rotation of every row.
//
// "FlashAttention-3 Deep Dive" (mojostudio.in), section 4 "FP8 Block Quantization & Numerical
// Incoherence Elimination": a separate fp32 scale per tile, codes = clip(x / s, -448, 448) in
// e4m3, and Q' = Q H, K' = K H with a random orthogonal Hadamard matrix so that one outlier is
// spread over the whole row before the scale is taken.
//
// The rotation is R = diag(sigma) H_d / sqrt(d) with H_d the Sylvester Hadamard matrix. Each row
// is multiplied by diag(sigma) H_d with the fast Walsh-Hadamard butterflies in fp32. The 1/sqrt(d)
// factor cancels in x'/descale, so codes come from the unnormalised product and only the stored
// descale carries it.
//
// HBM-bound: 2 bytes read and 1 byte written per element, plus 4 bytes per block. Work is cut
// into chunks of up to 128 rows of one (batch, head): 128 rows holding 128 / block_rows whole
// blocks when the block size divides 128, one whole block when it is another size below 128, or
// a 128-row piece of a longer block. Persistent CTAs walk the chunks; TMA copies the next chunks
// into a ring of shared-memory stages (128-byte swizzle) while the CTA converts the current one,
// so loads stay in flight throughout. Each lane holds a quarter of one row (8 rows per warp, 128
// per CTA of 16 warps), so two of the Walsh-Hadamard stages cross lanes and the rest stay in
// registers. Blocks of up to 128 rows take one launch that writes codes and descales; longer
// blocks take three: per-chunk maxima combined with an atomic max into the descale array
// (cleared by a memset first), then the codes, then each maximum's descale.
#include <algorithm>
#include <cstdint>

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include "launch.h"
#include "ptx.cuh"

namespace {

constexpr float kE4M3Max = 448.0f;
constexpr int kChunkRows = 128;          // most rows of one chunk (one smem stage)
constexpr uint32_t kSiteQuantFull = 11;  // wait site recorded in the status word on a timeout

template <int D, bool ROT>
struct QCfg {
  static constexpr int THREADS = 512;                // 16 warps x 8 rows = 128 rows
  static constexpr int WARPS = THREADS / 32;
  static constexpr int EPL = D / 4;                  // values per lane: a quarter of a row
  static constexpr int NP = EPL / 2;                 // packed fp32 pairs per lane
  static constexpr int SLAB_BYTES = kChunkRows * 128;   // one 64-column slab of a stage (128 rows)
  static constexpr int STAGE_BYTES = (D / 64) * SLAB_BYTES;
  // Loads in flight per CTA. The rotated d = 128 kernel holds one CTA per SM (registers), so it
  // takes a deep ring; the others fit two CTAs per SM with the shallower one.
  static constexpr int STAGES = D == 64 ? 4 : (D == 128 ? (ROT ? 6 : 3) : 3);
  static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024;
};

// The lane's quarter-row (EPL bf16 values, elements q * EPL ...) of row r in a stage, as EPL/2
// packed words. The stage holds D/64 slabs of 64 columns; a 128-byte line of a slab has its 16-byte
// pieces permuted by the 128-byte swizzle (piece c of row r sits at c ^ (r % 8)). The 8 lanes of a
// load phase hold 8 different rows, so they hit 8 different bank groups.
template <int D>
__device__ __forceinline__ void load_quarter_row(const uint8_t* stage, int r, int q, uint32_t* w) {
  constexpr int EPL = D / 4;
#pragma unroll
  for (int p = 0; p < EPL / 8; ++p) {
    const int off = q * (EPL * 2) + p * 16;      // byte offset of the piece within the row
    const int slab = off >> 7, c = (off & 127) >> 4;
    const uint4 t = *reinterpret_cast<const uint4*>(stage + slab * (kChunkRows * 128) + r * 128 + ((c ^ (r & 7)) << 4));
    w[4 * p] = t.x;
    w[4 * p + 1] = t.y;
    w[4 * p + 2] = t.z;
    w[4 * p + 3] = t.w;
  }
}

// Packed fp32 pairs p[j] = (v[2j], v[2j+1]) of the lane's values, from its bf16 words.
template <int NP>
__device__ __forceinline__ void unpack_pairs(const uint32_t* w, uint64_t* p) {
#pragma unroll
  for (int j = 0; j < NP; ++j) p[j] = gb300::f2_pack(__uint_as_float(w[j] << 16), __uint_as_float(w[j] & 0xFFFF0000u));
}

// p <- p diag(sigma) H_D over the row held by four lanes (lane bits 3 and 4 select the quarter; the
// element index is quarter * EPL + i). A butterfly on index bit b maps the pair (y_e, y_{e+2^b})
// with bit b of e clear to (y_e + y_{e+2^b}, y_e - y_{e+2^b}); applied for every bit it
// multiplies by the Sylvester matrix. Bits below log2(EPL) are inside the lane; the two above
// cross lanes, where each lane forms w + s v from its value v and its partner's w, with s = -1 on
// the upper lane of the pair.
template <int D>
__device__ __forceinline__ void rotate_quarter(uint64_t* p, const uint64_t* sg2, const uint64_t* lane_sgn2) {
  using namespace gb300;
  constexpr int NP = D / 8;
#pragma unroll
  for (int j = 0; j < NP; ++j) p[j] = f2_mul(p[j], sg2[j]);
#pragma unroll
  for (int j = 0; j < NP; ++j) {   // bit 0: the two halves of each pair
    float a, b;
    f2_unpack(p[j], a, b);
    p[j] = f2_pack(a + b, a - b);
  }
#pragma unroll
  for (int st = 1; st < NP; st <<= 1)   // bits 1 .. log2(EPL) - 1: pairs j and j + st
#pragma unroll
    for (int j = 0; j < NP; ++j)
      if (!(j & st)) {
        const uint64_t a = p[j], b = p[j + st];
        p[j] = f2_add(a, b);
        p[j + st] = f2_sub(a, b);
      }
#pragma unroll
  for (int k = 0; k < 2; ++k)   // the two quarter bits: lanes 8 and 16 apart
#pragma unroll
    for (int j = 0; j < NP; ++j) {
      float lo, hi;
      f2_unpack(p[j], lo, hi);
      const uint64_t w = f2_pack(__shfl_xor_sync(0xffffffffu, lo, 8 << k), __shfl_xor_sync(0xffffffffu, hi, 8 << k));
      p[j] = f2_fma(p[j], lane_sgn2[k], w);
    }
}

// Largest |value| of the lane's pairs.
template <int NP>
__device__ __forceinline__ float pairs_amax(const uint64_t* p) {
  float amax = 0.0f;
#pragma unroll
  for (int j = 0; j < NP; ++j) {
    float lo, hi;
    gb300::f2_unpack(p[j], lo, hi);
    amax = gb300::fmax3(amax, fabsf(lo), fabsf(hi));
  }
  return amax;
}

// Per-block constants of the division x / ds: r = 1/ds rounded to nearest, -ds, and -0.
struct DivConsts {
  uint64_t r2, nds2, nz2;
};
__device__ __forceinline__ DivConsts div_consts(float ds) {
  const float r = __frcp_rn(ds);
  return {gb300::f2_pack(r, r), gb300::f2_pack(-ds, -ds), gb300::f2_pack(-0.0f, -0.0f)};
}

// x / ds rounded to nearest fp32, for a pair, given r = 1/ds rounded to nearest: q0 = x r, then
// one correction with the exact residual x - q0 ds (an FMA). Markstein's theorem (P. Markstein,
// "Computation of elementary functions on the IBM RISC System/6000 processor", IBM J. Res. Dev.
// 34(1), 1990) makes the corrected quotient the correctly rounded one when r is within half an
// ulp of 1/ds, q0 within one ulp of x/ds, and nothing overflows or underflows. Here |x/ds| <= 448
// (ds is the block maximum over 448); quotients small enough to be fp32 subnormals round to an
// e4m3 zero whichever way their last bit falls. The product is formed as x r + (-0), which keeps
// the sign of a zero quotient.
__device__ __forceinline__ uint64_t div_by_descale(uint64_t x, const DivConsts& c) {
  using namespace gb300;
  const uint64_t q0 = f2_fma(x, c.r2, c.nz2);
  const uint64_t e = f2_fma(q0, c.nds2, x);
  return f2_fma(e, c.r2, q0);
}

// Codes of the lane's values / ds (round to nearest even, saturating to 448), EPL bytes at dst.
template <int D>
__device__ __forceinline__ void store_codes(uint8_t* dst, const uint64_t* p, const DivConsts& c) {
  constexpr int NP = D / 8;
  uint32_t h[NP];   // two codes in the low 16 bits
#pragma unroll
  for (int j = 0; j < NP; ++j) {
    float lo, hi;
    gb300::f2_unpack(div_by_descale(p[j], c), lo, hi);
    h[j] = (uint32_t)__nv_cvt_float2_to_fp8x2(make_float2(lo, hi), __NV_SATFINITE, __NV_E4M3);
  }
#pragma unroll
  for (int v = 0; v < NP / 8; ++v)
    reinterpret_cast<uint4*>(dst)[v] =
        make_uint4(__byte_perm(h[8 * v], h[8 * v + 1], 0x5410), __byte_perm(h[8 * v + 2], h[8 * v + 3], 0x5410),
                   __byte_perm(h[8 * v + 4], h[8 * v + 5], 0x5410), __byte_perm(h[8 * v + 6], h[8 * v + 7], 0x5410));
}

// Descale stored for a block: amax / 448 (1 for an all-zero block), divided by sqrt(D) when the
// rows were rotated (in fp64, rounded once to fp32).
template <int D>
__device__ __forceinline__ float stored_descale(float ds, bool rotated) {
  return rotated ? __double2float_rn(__ddiv_rn((double)ds, __dsqrt_rn((double)D))) : ds;
}

__device__ __forceinline__ float descale_of(float amax) { return amax > 0.0f ? __fdiv_rn(amax, kE4M3Max) : 1.0f; }

// Chunk c -> (batch, head, first row, end row). Heads vary fastest, so the chunks in flight at one
// time cover the same rows of many heads: whole rows of x in memory.
struct ChunkPos {
  int b, h, row_begin, row_end;
};
__device__ __forceinline__ ChunkPos chunk_pos(int c, const gb300::QuantLaunch& a) {
  ChunkPos p;
  p.h = c % a.Hx;
  c /= a.Hx;
  const int ci = c % a.cps;
  c /= a.cps;
  const int sp = c % a.nspan;
  p.b = c / a.nspan;
  const int span_begin = sp * a.span;
  p.row_begin = span_begin + ci * a.chunk_rows;
  p.row_end = min(a.N, min(span_begin + a.span, p.row_begin + a.chunk_rows));
  return p;
}

// MODE 0: a chunk holds whole blocks (codes + descales). MODE 1: chunk maximum into its block's
// descale slot with an atomic max. MODE 2: codes of the chunk from the block maximum in the slot.
// ROT: rows are rotated by diag(signs) H_D first.
template <int D, int MODE, bool ROT>
__global__ void __launch_bounds__(QCfg<D, ROT>::THREADS) quantize_kernel(const __grid_constant__ CUtensorMap tm,
                                                                   const gb300::QuantLaunch a, int n_chunks) {
  using C = QCfg<D, ROT>;
  using namespace gb300;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ __align__(8) uint64_t full[C::STAGES];
  __shared__ float red[2][C::WARPS];   // per-warp maxima, alternating between chunks
  __shared__ uint32_t abort_flag;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int r = 8 * warp + (lane & 7);   // row of the chunk this lane works on
  const int q = lane >> 3;               // its quarter of the row
  if (tid == 0) {
    for (int i = 0; i < C::STAGES; ++i) mbar_init(smem_addr(&full[i]), 1);
    fence_mbar_init();
    abort_flag = 0u;
    tma_prefetch_desc(&tm);
  }
  __syncthreads();
  const WaitCtl ctl{&abort_flag, a.status, a.timeout_ns};
  // One thread keeps up to STAGES chunks in flight, D/64 slab loads each. Boxes reaching past N
  // are filled with zeros and still count their full size.
  const uint32_t chunk_bytes = (uint32_t)a.chunk_rows * D * 2;
  auto issue = [&](int c, int stage) {
    const ChunkPos cp = chunk_pos(c, a);
    const uint32_t bar = smem_addr(&full[stage]);
    mbar_arrive_expect_tx(bar, chunk_bytes);
#pragma unroll
    for (int s = 0; s < D / 64; ++s)
      tma_load_4d(smem_addr(smem + stage * C::STAGE_BYTES + s * C::SLAB_BYTES), &tm, bar, 64 * s, cp.row_begin, cp.h,
                  cp.b);
  };
  if (tid == 0)
    for (int i = 0; i < C::STAGES; ++i) {
      const int c = blockIdx.x + i * gridDim.x;
      if (c < n_chunks) issue(c, i);
    }
  uint64_t sg2[ROT ? C::NP : 1], lane_sgn2[2];
  if constexpr (ROT) {
#pragma unroll
    for (int j = 0; j < C::NP; ++j)
      sg2[j] = f2_pack(__ldg(a.signs + q * C::EPL + 2 * j), __ldg(a.signs + q * C::EPL + 2 * j + 1));
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const float sgn = (q >> k) & 1 ? -1.0f : 1.0f;
      lane_sgn2[k] = f2_pack(sgn, sgn);
    }
  }
  // Rows of this lane's group (all inside one block) and the warps that hold them.
  const int grp = a.grp_rows >= 8 ? (8 * warp) / a.grp_rows : 0;
  const int gw0 = grp * a.grp_rows / 8;
  const int gw1 = min(C::WARPS, ((grp + 1) * a.grp_rows + 7) / 8);

  int k = 0;
  bool ok = true;
  for (int c = blockIdx.x; c < n_chunks; c += gridDim.x, ++k) {
    const int stage = k % C::STAGES;
    const bool w = mbar_wait(smem_addr(&full[stage]), (uint32_t)(k / C::STAGES) & 1u, ctl, kSiteQuantFull);
    if (!__syncthreads_and(w)) {
      ok = false;
      break;
    }
    const ChunkPos cp = chunk_pos(c, a);
    const bool valid = r < cp.row_end - cp.row_begin;
    const int grp_row0 = cp.row_begin + grp * a.grp_rows;       // first row of the group
    const bool grp_valid = grp_row0 < cp.row_end;
    float* ds_slot = a.descale + ((size_t)cp.b * a.Hx + cp.h) * a.nblk + (grp_valid ? grp_row0 / a.block_rows : 0);
    uint8_t* dst = a.x8 + ((size_t)(cp.b * a.N + cp.row_begin + r) * a.Hx + cp.h) * D + q * C::EPL;
    // Every lane computes (invalid rows on whatever the stage holds) so the shuffles see all 32.
    uint32_t raw[C::NP];
    uint64_t v[C::NP];
    load_quarter_row<D>(smem + stage * C::STAGE_BYTES, r, q, raw);
    unpack_pairs<C::NP>(raw, v);
    if constexpr (ROT) rotate_quarter<D>(v, sg2, lane_sgn2);
    if constexpr (MODE == 2) {
      const DivConsts dc = div_consts(descale_of(*ds_slot));   // the block maximum left by MODE 1
      if (valid) store_codes<D>(dst, v, dc);
    } else {
      float amax = valid ? pairs_amax<C::NP>(v) : 0.0f;
#pragma unroll
      for (int m = 16; m > 0; m >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, m));
      float* rk = red[k & 1];
      if (lane == 0) rk[warp] = amax;
      __syncthreads();
      // Every warp has read the stage: refill it while the codes are formed. (The next chunk
      // writes the other half of red; the one after waits at that chunk's barrier for every
      // warp, so no warp still reads this half then.)
      if (tid == 0) {
        const int next = c + C::STAGES * gridDim.x;
        if (next < n_chunks) issue(next, stage);
      }
      amax = rk[gw0];
      for (int i = gw0 + 1; i < gw1; ++i) amax = fmaxf(amax, rk[i]);
      const bool writer = lane == 0 && warp == gw0 && grp_valid;
      if constexpr (MODE == 1) {
        // non-negative floats order like their bit patterns
        if (writer) atomicMax(reinterpret_cast<unsigned int*>(ds_slot), __float_as_uint(amax));
      } else {
        const float ds = descale_of(amax);
        if (valid) store_codes<D>(dst, v, div_consts(ds));
        if (writer) *ds_slot = stored_descale<D>(ds, ROT);
      }
    }
    if constexpr (MODE == 2) {
      __syncthreads();   // the stage is read: refill it
      if (tid == 0) {
        const int next = c + C::STAGES * gridDim.x;
        if (next < n_chunks) issue(next, stage);
      }
    }
  }
  if (!ok && tid == 0) {
    // Copies this CTA issued and never consumed get a bounded time to land before it exits.
    for (int i = 0; i < C::STAGES; ++i) {
      const int kk = k + i;
      if (blockIdx.x + kk * gridDim.x >= n_chunks) break;
      const uint32_t bar = smem_addr(&full[kk % C::STAGES]);
      const uint64_t t0 = global_timer_ns();
      while (!mbar_try_wait(bar, (uint32_t)(kk / C::STAGES) & 1u) && global_timer_ns() - t0 < a.timeout_ns) {
      }
    }
  }
}

// One row per thread, for d = 64 and 128 and blocks of at most 128 rows. A CTA of 128 threads
// takes a chunk of up to 128 rows and thread r holds row r in registers (d fp32 values as pairs):
// the Walsh-Hadamard butterflies need no shuffles, and a block's maximum takes a warp reduction
// plus, for blocks of 64 or 128 rows, one exchange through shared memory at the chunk's single
// CTA barrier. Three CTAs share an SM, each with its own ring of TMA stages. Each thread writes
// its row of codes in 32-byte stores (one whole sector per lane) where x8 allows it.
template <int D>
struct RowCfg {
  static constexpr int THREADS = 128;
  static constexpr int NP = D / 2;                          // fp32 pairs per row
  static constexpr int SLAB_BYTES = kChunkRows * 128;       // one 64-column slab of a stage
  static constexpr int STAGE_BYTES = (D / 64) * SLAB_BYTES;
  static constexpr int STAGES = D == 64 ? 4 : 2;
  static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024;
};

// Row r of a stage (D bf16 values) as D/2 packed words; the 16-byte piece c of a 128-byte slab
// line sits at c ^ (r % 8) (128-byte swizzle).
template <int D>
__device__ __forceinline__ void load_row(const uint8_t* stage, int r, uint32_t* w) {
#pragma unroll
  for (int p = 0; p < D / 8; ++p) {
    const int slab = p >> 3, c = p & 7;
    const uint4 t = *reinterpret_cast<const uint4*>(stage + slab * (kChunkRows * 128) + r * 128 + ((c ^ (r & 7)) << 4));
    w[4 * p] = t.x;
    w[4 * p + 1] = t.y;
    w[4 * p + 2] = t.z;
    w[4 * p + 3] = t.w;
  }
}

// v <- v diag(sigma) H_D for a whole row in registers (pairs v[j] = (y_2j, y_2j+1)): a butterfly
// on index bit b maps (y_e, y_{e+2^b}) with bit b of e clear to (y_e + y_{e+2^b}, y_e - y_{e+2^b});
// bit 0 works inside each pair, bit b >= 1 on pairs j and j + 2^(b-1).
template <int D>
__device__ __forceinline__ void rotate_row(uint64_t* v, const float* sg) {
  using namespace gb300;
  constexpr int NP = D / 2;
#pragma unroll
  for (int j = 0; j < NP; j += 2) {
    const float4 s4 = *reinterpret_cast<const float4*>(sg + 2 * j);   // same address in every lane
    v[j] = f2_mul(v[j], f2_pack(s4.x, s4.y));
    v[j + 1] = f2_mul(v[j + 1], f2_pack(s4.z, s4.w));
  }
#pragma unroll
  for (int j = 0; j < NP; ++j) {
    float a, b;
    f2_unpack(v[j], a, b);
    v[j] = f2_pack(a + b, a - b);
  }
#pragma unroll
  for (int st = 1; st < NP; st <<= 1)
#pragma unroll
    for (int j = 0; j < NP; ++j)
      if (!(j & st)) {
        const uint64_t a = v[j], b = v[j + st];
        v[j] = f2_add(a, b);
        v[j + st] = f2_sub(a, b);
      }
}

// MODE as for quantize_kernel: 0 whole blocks per chunk (codes and descales), 1 chunk maxima of
// longer blocks (atomic max into the block's slot), 2 codes from the block maximum in the slot.
// Row r of chunk cp as codes x / ds (the division as div_by_descale), D bytes in 32-byte stores
// where x8 allows it.
template <int D>
__device__ __forceinline__ void store_row_codes(const gb300::QuantLaunch& a, const ChunkPos& cp, int r,
                                                const uint64_t* v, const DivConsts& dc) {
  using namespace gb300;
  uint32_t wd[D / 4];   // four codes per word, the lowest-addressed in the low byte
#pragma unroll
  for (int j = 0; j < D / 2; j += 2) {
    float a0, a1, b0, b1;
    f2_unpack(div_by_descale(v[j], dc), a0, a1);
    f2_unpack(div_by_descale(v[j + 1], dc), b0, b1);
    const uint32_t lo = (uint32_t)__nv_cvt_float2_to_fp8x2(make_float2(a0, a1), __NV_SATFINITE, __NV_E4M3);
    const uint32_t hi = (uint32_t)__nv_cvt_float2_to_fp8x2(make_float2(b0, b1), __NV_SATFINITE, __NV_E4M3);
    wd[j >> 1] = __byte_perm(lo, hi, 0x5410);
  }
  uint8_t* dst = a.x8 + ((size_t)(cp.b * a.N + cp.row_begin + r) * a.Hx + cp.h) * D;
  if (a.x8_v8) {
#pragma unroll
    for (int i = 0; i < D / 32; ++i) st_global_v8(dst + 32 * i, wd + 8 * i);
  } else {
#pragma unroll
    for (int i = 0; i < D / 16; ++i)
      reinterpret_cast<uint4*>(dst)[i] = make_uint4(wd[4 * i], wd[4 * i + 1], wd[4 * i + 2], wd[4 * i + 3]);
  }
}

template <int D, int MODE, bool ROT>
__global__ void __launch_bounds__(RowCfg<D>::THREADS, 3)
    quantize_rows_kernel(const __grid_constant__ CUtensorMap tm, const gb300::QuantLaunch a, int n_chunks) {
  using C = RowCfg<D>;
  using namespace gb300;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ __align__(8) uint64_t full[C::STAGES];
  __shared__ float red[2][4];                  // per-warp maxima, alternating between chunks
  __shared__ __align__(16) float sg[ROT ? D : 4];
  __shared__ uint32_t abort_flag;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int i = 0; i < C::STAGES; ++i) mbar_init(smem_addr(&full[i]), 1);
    fence_mbar_init();
    abort_flag = 0u;
    tma_prefetch_desc(&tm);
  }
  if constexpr (ROT)
    for (int i = tid; i < D; i += C::THREADS) sg[i] = __ldg(a.signs + i);
  __syncthreads();
  const WaitCtl ctl{&abort_flag, a.status, a.timeout_ns};
  const uint32_t chunk_bytes = (uint32_t)a.chunk_rows * D * 2;   // boxes past N count in full
  auto issue = [&](int c, int stage) {
    const ChunkPos cp = chunk_pos(c, a);
    const uint32_t bar = smem_addr(&full[stage]);
    mbar_arrive_expect_tx(bar, chunk_bytes);
#pragma unroll
    for (int sl = 0; sl < D / 64; ++sl)
      tma_load_4d(smem_addr(smem + stage * C::STAGE_BYTES + sl * C::SLAB_BYTES), &tm, bar, 64 * sl, cp.row_begin, cp.h,
                  cp.b);
  };
  if (tid == 0)
    for (int i = 0; i < C::STAGES; ++i) {
      const int c = blockIdx.x + i * gridDim.x;
      if (c < n_chunks) issue(c, i);
    }
  // Rows reduced together: a block of grp_rows rows (a power of two) inside a 128-row chunk, or
  // the whole chunk when the chunk is one block (rows past its end contribute 0).
  const int span_rows =
      (MODE == 0 && a.chunk_rows == kChunkRows && (a.grp_rows & (a.grp_rows - 1)) == 0) ? a.grp_rows : kChunkRows;
  const int r = tid;
  int k = 0;
  bool ok = true;
  for (int c = blockIdx.x; c < n_chunks; c += gridDim.x, ++k) {
    const int stage = k % C::STAGES;
    const bool w = mbar_wait(smem_addr(&full[stage]), (uint32_t)(k / C::STAGES) & 1u, ctl, kSiteQuantFull);
    if (!__all_sync(0xffffffffu, w)) {
      ok = false;
      break;
    }
    const ChunkPos cp = chunk_pos(c, a);
    const bool valid = r < cp.row_end - cp.row_begin;
    uint32_t raw[C::NP];
    uint64_t v[C::NP];
    load_row<D>(smem + stage * C::STAGE_BYTES, r, raw);
#pragma unroll
    for (int j = 0; j < C::NP; ++j) v[j] = f2_pack(__uint_as_float(raw[j] << 16), __uint_as_float(raw[j] & 0xFFFF0000u));
    if constexpr (ROT) rotate_row<D>(v, sg);
    if constexpr (MODE == 2) {
      // The block maximum the maxima launch left in the slot; the stage is read.
      __syncthreads();
      if (tid == 0) {
        const int next = c + C::STAGES * gridDim.x;
        if (next < n_chunks) issue(next, stage);
      }
      if (valid) {
        const float ds2 = descale_of(a.descale[((size_t)cp.b * a.Hx + cp.h) * a.nblk + cp.row_begin / a.block_rows]);
        store_row_codes<D>(a, cp, r, v, div_consts(ds2));
      }
      continue;
    }
    float amax = 0.0f;
    if (valid) {
#pragma unroll
      for (int j = 0; j < C::NP; ++j) {
        float lo, hi;
        f2_unpack(v[j], lo, hi);
        amax = fmax3(amax, fabsf(lo), fabsf(hi));
      }
    }
#pragma unroll
    for (int m = 1; m < 32; m <<= 1)
      if (m < span_rows) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, m));
    float* rk = red[k & 1];
    if (lane == 0) rk[warp] = amax;
    __syncthreads();   // every row of the stage is in registers, every warp's maximum is in rk
    if (tid == 0) {
      const int next = c + C::STAGES * gridDim.x;
      if (next < n_chunks) issue(next, stage);
    }
    if (span_rows > 32) {
      const int w0 = (warp * 32 / span_rows) * (span_rows / 32);
      for (int i = 0; i < span_rows / 32; ++i) amax = fmaxf(amax, rk[w0 + i]);
    }
    float* slot = a.descale + ((size_t)cp.b * a.Hx + cp.h) * a.nblk;
    if constexpr (MODE == 1) {
      // non-negative floats order like their bit patterns
      if (tid == 0 && cp.row_begin < cp.row_end)
        atomicMax(reinterpret_cast<unsigned int*>(slot + cp.row_begin / a.block_rows), __float_as_uint(amax));
      continue;
    }
    const float ds = descale_of(amax);
    const int grp_row0 = (r / span_rows) * span_rows;   // first row of this thread's group
    if (r == grp_row0 && grp_row0 < cp.row_end - cp.row_begin)
      slot[(cp.row_begin + grp_row0) / a.block_rows] = stored_descale<D>(ds, ROT);
    if (valid) store_row_codes<D>(a, cp, r, v, div_consts(ds));
  }
  if (!ok && tid == 0) {
    // Copies this CTA issued and never consumed get a bounded time to land before it exits.
    for (int i = 0; i < C::STAGES; ++i) {
      const int kk = k + i;
      if (blockIdx.x + kk * gridDim.x >= n_chunks) break;
      const uint32_t bar = smem_addr(&full[kk % C::STAGES]);
      const uint64_t t0 = global_timer_ns();
      while (!mbar_try_wait(bar, (uint32_t)(kk / C::STAGES) & 1u) && global_timer_ns() - t0 < a.timeout_ns) {
      }
    }
  }
}

// Block maxima -> descales, in place.
template <int D>
__global__ void finalize_descale_kernel(float* descale, int n, bool rotated) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) descale[i] = stored_descale<D>(descale_of(descale[i]), rotated);
}

template <int D, int MODE, bool ROT>
cudaError_t launch_mode(const gb300::QuantLaunch& q, int n_chunks, cudaStream_t s) {
  using C = QCfg<D, ROT>;
  auto kern = quantize_kernel<D, MODE, ROT>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, C::THREADS, C::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  const int grid = (int)std::min<long long>(n_chunks, (long long)std::max(per_sm, 1) * q.num_sms);
  kern<<<grid, C::THREADS, C::SMEM_BYTES, s>>>(q.tm_x, q, n_chunks);
  return cudaGetLastError();
}

template <int D, int MODE, bool ROT>
cudaError_t launch_rows(const gb300::QuantLaunch& q, int n_chunks, cudaStream_t s) {
  using C = RowCfg<D>;
  auto kern = quantize_rows_kernel<D, MODE, ROT>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, C::THREADS, C::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  const int grid = (int)std::min<long long>(n_chunks, (long long)std::max(per_sm, 1) * q.num_sms);
  kern<<<grid, C::THREADS, C::SMEM_BYTES, s>>>(q.tm_x, q, n_chunks);
  return cudaGetLastError();
}

template <int D, bool ROT>
cudaError_t launch_quantize(const gb300::QuantLaunch& q, cudaStream_t s) {
  const int n_chunks = q.B * q.Hx * q.nspan * q.cps;
  if (q.block_rows <= kChunkRows) {
    if constexpr (D <= 128) return launch_rows<D, 0, ROT>(q, n_chunks, s);
    else return launch_mode<D, 0, ROT>(q, n_chunks, s);
  }
  const size_t nds = (size_t)q.B * q.Hx * q.nblk;
  cudaError_t e = cudaMemsetAsync(q.descale, 0, nds * sizeof(float), s);
  if (e != cudaSuccess) return e;
  if constexpr (D <= 128) {
    if ((e = launch_rows<D, 1, ROT>(q, n_chunks, s)) != cudaSuccess) return e;
    if ((e = launch_rows<D, 2, ROT>(q, n_chunks, s)) != cudaSuccess) return e;
  } else {
    if ((e = launch_mode<D, 1, ROT>(q, n_chunks, s)) != cudaSuccess) return e;
    if ((e = launch_mode<D, 2, ROT>(q, n_chunks, s)) != cudaSuccess) return e;
  }
  finalize_descale_kernel<D><<<(unsigned)((nds + 255) / 256), 256, 0, s>>>(q.descale, (int)nds, ROT);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_quantize_d(const gb300::QuantLaunch& q, cudaStream_t s) {
  return q.signs ? launch_quantize<D, true>(q, s) : launch_quantize<D, false>(q, s);
}

}  // namespace

namespace gb300 {

cudaError_t launch_quantize_e4m3(const QuantLaunch& q, cudaStream_t stream) {
  switch (q.d) {
    case 64: return launch_quantize_d<64>(q, stream);
    case 128: return launch_quantize_d<128>(q, stream);
    case 256: return launch_quantize_d<256>(q, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace gb300
