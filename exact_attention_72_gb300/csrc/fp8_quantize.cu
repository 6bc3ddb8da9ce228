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

template <int D, bool ROT>
cudaError_t launch_quantize(const gb300::QuantLaunch& q, cudaStream_t s) {
  const int n_chunks = q.B * q.Hx * q.nspan * q.cps;
  if (q.block_rows <= kChunkRows) return launch_mode<D, 0, ROT>(q, n_chunks, s);
  const size_t nds = (size_t)q.B * q.Hx * q.nblk;
  cudaError_t e = cudaMemsetAsync(q.descale, 0, nds * sizeof(float), s);
  if (e != cudaSuccess) return e;
  if ((e = launch_mode<D, 1, ROT>(q, n_chunks, s)) != cudaSuccess) return e;
  if ((e = launch_mode<D, 2, ROT>(q, n_chunks, s)) != cudaSuccess) return e;
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
