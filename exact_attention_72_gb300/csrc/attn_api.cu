// C ABI of the attention forward library: argument checks, tensor-map encoding, dispatch to
// the kernel instance for (head dim, causal, dtype), device status word, host-buffer variant.
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <climits>
#include <cstring>
#include <mutex>

#include <cuda.h>
#include <cuda_runtime.h>

#include "attn.h"
#include "context_id.h"
#include "launch.h"

// First failure recorded by any kernel of this library on the device (0 = none).
static __device__ uint32_t g_attn_status;

namespace {

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

constexpr unsigned long long kDefaultTimeoutNs = 4000000000ull;
constexpr int kMaxDevices = 64;

unsigned long long g_timeout_ns = 0;  // 0: default
int g_skip_load = 0;

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static std::once_flag once;
  static EncodeTiledFn fn = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

constexpr int kMaxChunks = 10;   // eight even chunks, the first and last of them halved

// Per-device state, valid for one CUDA context (see context_id.h): the SM count, the device
// address of the status word and the host-buffer pipeline's streams and events. When the current
// context is not the one the state was made for (first use, or a new primary context after
// cudaDeviceReset) it is looked up again; a lookup that fails is not cached, so a later call retries.
struct DeviceInfo {
  std::mutex mu;
  unsigned long long ctx = 0;   // context id the fields below belong to (0: none yet)
  int num_sms = 0;
  uint32_t* status = nullptr;
  // Host-buffer pipeline (attn_fwd_host): created on first use in each context.
  bool pipe_made = false;
  unsigned long long pipe_ctx = 0;   // context id the pipeline was made in
  cudaStream_t s_in = nullptr, s_out = nullptr, s_comp[2] = {nullptr, nullptr};
  cudaEvent_t ev_start = nullptr, ev_end = nullptr, ev_in[kMaxChunks] = {}, ev_k[kMaxChunks] = {};
  std::mutex pipe_mutex;   // one host-buffer call at a time per device (shared streams/events)
};
DeviceInfo g_dev[kMaxDevices];

DeviceInfo* device_info() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  DeviceInfo* di = &g_dev[dev];
  const unsigned long long id = gb300::current_context_id();
  std::lock_guard<std::mutex> lock(di->mu);
  if (id != 0 && id == di->ctx) return di;
  int sms = 0;
  void* p = nullptr;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      cudaGetSymbolAddress(&p, g_attn_status) != cudaSuccess)
    return nullptr;
  di->num_sms = sms;
  di->status = static_cast<uint32_t*>(p);
  // The lookup has initialised the context if it did not exist yet; key the state on it. (With no
  // readable id the state is looked up again on every call.)
  di->ctx = gb300::current_context_id();
  return di;
}

// Streams and events of the host-buffer pipeline for the current context; called with
// di->pipe_mutex held. They are made once and made again only when the context id changes (with
// no readable id they are kept); handles made for an earlier context died with it and are not
// destroyed.
bool pipeline_ready(DeviceInfo* di) {
  if (di->pipe_made && di->pipe_ctx == di->ctx) return true;
  bool ok = true;
  ok = ok && cudaStreamCreateWithFlags(&di->s_in, cudaStreamNonBlocking) == cudaSuccess;
  ok = ok && cudaStreamCreateWithFlags(&di->s_out, cudaStreamNonBlocking) == cudaSuccess;
  for (int i = 0; i < 2; ++i) ok = ok && cudaStreamCreateWithFlags(&di->s_comp[i], cudaStreamNonBlocking) == cudaSuccess;
  ok = ok && cudaEventCreateWithFlags(&di->ev_start, cudaEventDisableTiming) == cudaSuccess;
  ok = ok && cudaEventCreateWithFlags(&di->ev_end, cudaEventDisableTiming) == cudaSuccess;
  for (int i = 0; i < kMaxChunks; ++i) {
    ok = ok && cudaEventCreateWithFlags(&di->ev_in[i], cudaEventDisableTiming) == cudaSuccess;
    ok = ok && cudaEventCreateWithFlags(&di->ev_k[i], cudaEventDisableTiming) == cudaSuccess;
  }
  di->pipe_made = ok;
  di->pipe_ctx = di->ctx;
  return ok;
}

// attn_fwd_host work split: chunks of whole batches (B >= kHostChunks) or, for fewer batches, one
// batch and a contiguous range of KV heads (with their query heads), so each chunk is a
// self-contained attention problem whose copies can overlap another chunk's kernel. The
// host-device link (about 210 GB/s each way) bounds the call; smaller chunks shorten the
// first upload and the last download that nothing overlaps.
constexpr int kHostChunks = 8;
static_assert(kHostChunks + 2 <= kMaxChunks, "chunk events");
struct HostChunk {
  int b0, nb;      // batches [b0, b0 + nb)
  int g0, ng;      // kv heads [g0, g0 + ng); query heads [g0 G, (g0 + ng) G)
  size_t off_q, off_k, off_v, off_o, off_lse;   // workspace offsets
};

int plan_host_chunks(int B, int H, int Hkv, int N, int d, size_t elt, HostChunk* ch, size_t* total) {
  const int G = H / Hkv;
  int nc = 0;
  auto add = [&](int b0, int nb, int g0, int ng) {
    HostChunk& c = ch[nc++];
    c.b0 = b0; c.nb = nb; c.g0 = g0; c.ng = ng;
    const size_t rows = (size_t)nb * N;
    size_t off = *total;
    c.off_q = off;   off += round_up(rows * ng * G * d * elt, 256);
    c.off_k = off;   off += round_up(rows * ng * d * elt, 256);
    c.off_v = off;   off += round_up(rows * ng * d * elt, 256);
    c.off_o = off;   off += round_up(rows * ng * G * d * 2, 256);
    c.off_lse = off; off += round_up(rows * ng * G * 4, 256);
    *total = off;
  };
  *total = 0;
  struct Spec {
    int b0, nb, g0, ng;
  };
  Spec spec[kMaxChunks];
  int ns = 0;
  if (B >= kHostChunks) {
    for (int i = 0; i < kHostChunks; ++i) {
      const int b0 = (int)((long long)B * i / kHostChunks), b1 = (int)((long long)B * (i + 1) / kHostChunks);
      if (b1 > b0) spec[ns++] = {b0, b1 - b0, 0, Hkv};
    }
  } else {
    const int S = std::min(Hkv, std::max(1, kHostChunks / B));   // B * S <= kHostChunks
    for (int b = 0; b < B; ++b)
      for (int i = 0; i < S; ++i) {
        const int g0 = (int)((long long)Hkv * i / S), g1 = (int)((long long)Hkv * (i + 1) / S);
        if (g1 > g0) spec[ns++] = {b, 1, g0, g1 - g0};
      }
  }
  // The first chunk's upload and the last chunk's kernel and download overlap nothing: halve
  // those two chunks (by batches, else by kv heads) when they can be halved.
  auto halves = [&](const Spec& x, Spec& lo, Spec& hi) -> bool {
    if (x.nb >= 2) {
      lo = {x.b0, x.nb / 2, x.g0, x.ng};
      hi = {x.b0 + x.nb / 2, x.nb - x.nb / 2, x.g0, x.ng};
      return true;
    }
    if (x.ng >= 2) {
      lo = {x.b0, x.nb, x.g0, x.ng / 2};
      hi = {x.b0, x.nb, x.g0 + x.ng / 2, x.ng - x.ng / 2};
      return true;
    }
    return false;
  };
  for (int i = 0; i < ns; ++i) {
    Spec lo, hi;
    if ((i == 0 || i == ns - 1) && ns > 1 && halves(spec[i], lo, hi)) {
      add(lo.b0, lo.nb, lo.g0, lo.ng);
      add(hi.b0, hi.nb, hi.g0, hi.ng);
    } else {
      add(spec[i].b0, spec[i].nb, spec[i].g0, spec[i].ng);
    }
  }
  *total += 256;   // fp8 descales
  return nc;
}

bool ranges_overlap(const void* a, size_t na, const void* b, size_t nb) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb && y < x + na;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// [B, N, heads, d] tensor -> 4-D map (d, N, heads, B), box (one swizzle row, 128 rows, 1, 1);
// rows past N read as zeros. The swizzle row is 128 bytes, or 64 where a whole row of d is 64
// bytes (e4m3 at d = 64), as the kernel's AttnCfg::SWZ.
bool make_map(CUtensorMap* m, const void* base, bool fp8, int d, int N, int heads, int B, int box_rows = 128) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t elt = fp8 ? 1 : 2;
  const bool swz64 = d * elt < 128;
  cuuint64_t dims[4] = {(cuuint64_t)d, (cuuint64_t)N, (cuuint64_t)heads, (cuuint64_t)B};
  cuuint64_t strides[3] = {(cuuint64_t)heads * d * elt, (cuuint64_t)d * elt, (cuuint64_t)N * heads * d * elt};
  cuuint32_t box[4] = {(cuuint32_t)((swz64 ? 64 : 128) / elt), (cuuint32_t)box_rows, 1, 1};
  cuuint32_t es[4] = {1, 1, 1, 1};
  return enc(m, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base),
             dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
             swz64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// bf16 [B, N, heads, d] tensor -> 4-D map (d, N, heads, B) whose box is 64 columns of box_rows
// rows of one (batch, head) with the 128-byte swizzle: the e4m3 quantiser's input, loaded as d/64
// boxes per chunk. Rows past N read as zeros.
bool make_rows_map(CUtensorMap* m, const void* base, int d, int N, int heads, int B, int box_rows) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[4] = {(cuuint64_t)d, (cuuint64_t)N, (cuuint64_t)heads, (cuuint64_t)B};
  cuuint64_t strides[3] = {(cuuint64_t)heads * d * 2, (cuuint64_t)d * 2, (cuuint64_t)N * heads * d * 2};
  cuuint32_t box[4] = {64, (cuuint32_t)box_rows, 1, 1};
  cuuint32_t es[4] = {1, 1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Packed GQA view of q [B, Nq, H, d] for split-KV decode: 5-D map (d, G, Nq, Hkv, B) so one box
// (one swizzle row, G heads, 128 / G positions, 1, 1) is 128 query rows of one kv head's group.
// The swizzle row is 128 bytes, or 64 for e4m3 at d = 64, as in make_map.
bool make_map_q_packed(CUtensorMap* m, const void* base, bool fp8, int d, int Nq, int H, int Hkv, int B) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t elt = fp8 ? 1 : 2;
  const bool swz64 = d * elt < 128;
  const int G = H / Hkv;
  cuuint64_t dims[5] = {(cuuint64_t)d, (cuuint64_t)G, (cuuint64_t)Nq, (cuuint64_t)Hkv, (cuuint64_t)B};
  cuuint64_t strides[4] = {(cuuint64_t)d * elt, (cuuint64_t)H * d * elt, (cuuint64_t)G * d * elt,
                           (cuuint64_t)Nq * H * d * elt};
  cuuint32_t box[5] = {(cuuint32_t)((swz64 ? 64 : 128) / elt), (cuuint32_t)G, (cuuint32_t)(128 / G), 1, 1};
  cuuint32_t es[5] = {1, 1, 1, 1, 1};
  return enc(m, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void*>(base),
             dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
             swz64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D>
cudaError_t dispatch_split(gb300::LaunchArgs& a, bool fp8, cudaStream_t s) {
  if constexpr (D == 64 || D == 128 || D == 256) {
    if (fp8) return gb300::launch_attn_fwd<D, false, true, true>(a, s);
  }
  return gb300::launch_attn_fwd<D, false, false, true>(a, s);
}

constexpr int kMaxSplits = 128;

size_t splitkv_part_o_bytes(int B, int H, int Nq, int d, int S) {
  return round_up((size_t)S * B * H * Nq * d * 4, 256);
}

bool supported_dim(int d, attn_dtype_t dtype) {
  if (dtype == ATTN_DTYPE_BF16) return d == 64 || d == 128 || d == 256;
  if (dtype == ATTN_DTYPE_FP8_E4M3) return d == 64 || d == 128 || d == 256;
  return false;
}

// Shape checks shared by attn_fwd and attn_fwd_host.
attn_status_t check_shape(int B, int H, int Hkv, int N, int d, float scale, attn_dtype_t dtype) {
  if (B < 1 || H < 1 || Hkv < 1 || N < 1 || d < 1) return ATTN_ERR_INVALID_ARG;
  if (H % Hkv != 0) return ATTN_ERR_INVALID_ARG;
  if (!std::isfinite(scale)) return ATTN_ERR_INVALID_ARG;
  if (dtype != ATTN_DTYPE_BF16 && dtype != ATTN_DTYPE_FP8_E4M3) return ATTN_ERR_INVALID_ARG;
  // Masked scores are -inf before scaling; scale == 0 would turn them into NaN (-inf * 0). A
  // negative scale is run as |scale| times -Q K^T (the MMA negates Q).
  if (scale == 0.0f) return ATTN_ERR_UNSUPPORTED;
  if (!supported_dim(d, dtype)) return ATTN_ERR_UNSUPPORTED;
  const long long rows = gb300::rows_per_work_tile(d);
  const long long tiles = (long long)B * H * ((N + rows - 1) / rows);
  if (tiles >= (1LL << 31)) return ATTN_ERR_UNSUPPORTED;
  if ((long long)B * N * H * d >= (1LL << 40)) return ATTN_ERR_UNSUPPORTED;
  return ATTN_OK;
}

template <int D>
cudaError_t dispatch_d(gb300::LaunchArgs& a, bool causal, bool fp8, cudaStream_t s) {
  if constexpr (D == 64 || D == 128 || D == 256) {
    if (fp8) return causal ? gb300::launch_attn_fwd<D, true, true>(a, s) : gb300::launch_attn_fwd<D, false, true>(a, s);
  }
  return causal ? gb300::launch_attn_fwd<D, true, false>(a, s) : gb300::launch_attn_fwd<D, false, false>(a, s);
}

}  // namespace

extern "C" {

}  // extern "C"

namespace {

template <int D>
cudaError_t dispatch_varlen(gb300::LaunchArgs& a, bool causal, bool fp8, cudaStream_t s) {
  if constexpr (D == 64 || D == 128 || D == 256) {
    if (fp8)
      return causal ? gb300::launch_attn_fwd<D, true, true, false, true>(a, s)
                    : gb300::launch_attn_fwd<D, false, true, false, true>(a, s);
  }
  return causal ? gb300::launch_attn_fwd<D, true, false, false, true>(a, s)
                : gb300::launch_attn_fwd<D, false, false, false, true>(a, s);
}

// Work tiles a ragged batch can have at most: sum_b ceil(Nq_b / R) <= total_q / R + B, per head.
long long varlen_tile_bound(int B, int H, int total_q, int d) {
  const long long R = gb300::rows_per_work_tile(d);
  return (long long)H * ((total_q + R - 1) / R + B);
}

// The prefill forward behind attn_fwd and the fp8 entries with finer descales. ds: descale
// element strides (q by batch, q by head, q by 128-row block, k by batch, k by kv head, k by
// 64-key block, v by batch, v by kv head); all 0 = one descale per tensor.
attn_status_t prefill_forward(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Hkv,
                              int N, int d, float scale, int causal, attn_dtype_t dtype, const float* descale_q,
                              const float* descale_k, const float* descale_v, const int* ds, cudaStream_t stream) {
  attn_status_t st = check_shape(B, H, Hkv, N, d, scale, dtype);
  if (st != ATTN_OK) return st;
  const bool fp8 = dtype == ATTN_DTYPE_FP8_E4M3;
  if (!q || !k || !v || !o || !lse) return ATTN_ERR_INVALID_ARG;
  if (fp8 && (!descale_q || !descale_k || !descale_v)) return ATTN_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) || !aligned(lse, 4))
    return ATTN_ERR_INVALID_ARG;
  const size_t elt = fp8 ? 1 : 2;
  const size_t nq = (size_t)B * N * H * d, nkv = (size_t)B * N * Hkv * d;
  const size_t o_bytes = nq * 2, lse_bytes = (size_t)B * H * N * 4;
  const void* ins[3] = {q, k, v};
  const size_t in_bytes[3] = {nq * elt, nkv * elt, nkv * elt};
  for (int i = 0; i < 3; ++i)
    if (ranges_overlap(o, o_bytes, ins[i], in_bytes[i]) || ranges_overlap(lse, lse_bytes, ins[i], in_bytes[i]))
      return ATTN_ERR_INVALID_ARG;
  if (ranges_overlap(o, o_bytes, lse, lse_bytes)) return ATTN_ERR_INVALID_ARG;

  DeviceInfo* di = device_info();
  if (!di) return ATTN_ERR_CUDA;
  gb300::LaunchArgs a;
  memset(&a, 0, sizeof(a));
  if (!make_map(&a.tm_q, q, fp8, d, N, H, B) || !make_map(&a.tm_k, k, fp8, d, N, Hkv, B) ||
      !make_map(&a.tm_v, v, fp8, d, N, Hkv, B))
    return ATTN_ERR_CUDA;
  const int rows = gb300::rows_per_work_tile(d);
  gb300::AttnParams& p = a.params;
  p.o = o;
  p.lse = lse;
  p.descale_q = descale_q;
  p.descale_k = descale_k;
  p.descale_v = descale_v;
  p.dq_sb = ds[0];
  p.dq_sh = ds[1];
  p.dq_sm = ds[2];
  p.dk_sb = ds[3];
  p.dk_sh = ds[4];
  p.dk_sn = ds[5];
  p.dv_sb = ds[6];
  p.dv_sh = ds[7];
  p.B = B;
  p.H = H;
  p.Hkv = Hkv;
  p.N = N;
  p.scale_log2 = std::fabs(scale) * 1.4426950408889634f;
  p.qk_negate = scale < 0.0f ? gb300::kIdescNegateA : 0u;
  p.o_v8 = aligned(o, 32) ? 1 : 0;
  p.n_mb = (N + rows - 1) / rows;
  p.n_tiles = B * H * p.n_mb;
  p.Nk = N;
  p.G = H / Hkv;
  p.n_splits = 1;
  p.n_kvt = (N + 127) / 128;
  p.part_o = nullptr;
  p.part_lse = nullptr;
  p.status = di->status;
  p.timeout_ns = g_timeout_ns ? g_timeout_ns : kDefaultTimeoutNs;
  p.debug_skip_load = g_skip_load;
  a.num_sms = di->num_sms;
  // A last wave that would leave SMs idle has its tiles' keys cut: the first launch takes the
  // first parts, a dependent launch the rest and the merge.
  const int halved = gb300::plan_tail(p, p.n_tiles, p.n_kvt, a.num_sms, causal != 0, !fp8 && d <= 128);
  auto launch = [&](gb300::LaunchArgs& x) -> cudaError_t {
    switch (d) {
      case 64: return dispatch_d<64>(x, causal != 0, fp8, stream);
      case 128: return dispatch_d<128>(x, causal != 0, fp8, stream);
      default: return dispatch_d<256>(x, causal != 0, fp8, stream);
    }
  };
  cudaError_t e = launch(a);
  if (e == cudaSuccess && halved) {
    gb300::LaunchArgs second = a;
    second.params.tail_mode = p.tail_mode == 3 ? 4 : 2;
    second.params.n_tiles = halved;
    second.dependent = true;
    e = launch(second);
  }
  return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

}  // namespace

extern "C" {

attn_status_t attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Hkv,
                       int N, int d, float scale, int causal, attn_dtype_t dtype, const float* descale_q,
                       const float* descale_k, const float* descale_v, cudaStream_t stream) {
  static const int per_tensor[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  return prefill_forward(q, k, v, o, lse, B, H, Hkv, N, d, scale, causal, dtype, descale_q, descale_k, descale_v,
                         per_tensor, stream);
}

attn_status_t attn_fwd_fp8_scaled(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                                  int Hkv, int N, int d, float scale, int causal, const float* descale_q,
                                  int q_stride_b, int q_stride_h, const float* descale_k, const float* descale_v,
                                  int kv_stride_b, int kv_stride_h, cudaStream_t stream) {
  if (q_stride_b < 0 || q_stride_h < 0 || kv_stride_b < 0 || kv_stride_h < 0) return ATTN_ERR_INVALID_ARG;
  const int ds[8] = {q_stride_b, q_stride_h, 0, kv_stride_b, kv_stride_h, 0, kv_stride_b, kv_stride_h};
  return prefill_forward(q, k, v, o, lse, B, H, Hkv, N, d, scale, causal, ATTN_DTYPE_FP8_E4M3, descale_q, descale_k,
                         descale_v, ds, stream);
}

attn_status_t attn_fwd_fp8_blockscaled(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                                       int H, int Hkv, int N, int d, float scale, int causal,
                                       const float* descale_q, const float* descale_k, const float* descale_v,
                                       cudaStream_t stream) {
  if (N < 1 || H < 1 || Hkv < 1) return ATTN_ERR_INVALID_ARG;
  const long long nqb = (N + ATTN_FP8_Q_BLOCK - 1) / ATTN_FP8_Q_BLOCK;
  const long long nkb = (N + ATTN_FP8_K_BLOCK - 1) / ATTN_FP8_K_BLOCK;
  if ((long long)B * H * nqb > INT_MAX || (long long)B * Hkv * nkb > INT_MAX) return ATTN_ERR_UNSUPPORTED;
  const int ds[8] = {(int)(H * nqb), (int)nqb, 1, (int)(Hkv * nkb), (int)nkb, 1, Hkv, 1};
  return prefill_forward(q, k, v, o, lse, B, H, Hkv, N, d, scale, causal, ATTN_DTYPE_FP8_E4M3, descale_q, descale_k,
                         descale_v, ds, stream);
}

size_t attn_fwd_host_workspace_bytes(int B, int H, int Hkv, int N, int d, attn_dtype_t dtype) {
  if (check_shape(B, H, Hkv, N, d, 1.0f, dtype) != ATTN_OK) return 0;
  HostChunk ch[kMaxChunks];
  size_t total = 0;
  plan_host_chunks(B, H, Hkv, N, d, dtype == ATTN_DTYPE_FP8_E4M3 ? 1 : 2, ch, &total);
  return total;
}

attn_status_t attn_fwd_host(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Hkv,
                            int N, int d, float scale, int causal, attn_dtype_t dtype, const float* descale_q,
                            const float* descale_k, const float* descale_v, void* workspace,
                            size_t workspace_bytes, cudaStream_t stream) {
  attn_status_t st = check_shape(B, H, Hkv, N, d, scale, dtype);
  if (st != ATTN_OK) return st;
  const bool fp8 = dtype == ATTN_DTYPE_FP8_E4M3;
  if (!q || !k || !v || !o || !lse || !workspace) return ATTN_ERR_INVALID_ARG;
  if (fp8 && (!descale_q || !descale_k || !descale_v)) return ATTN_ERR_INVALID_ARG;
  if (!aligned(workspace, 256) || workspace_bytes < attn_fwd_host_workspace_bytes(B, H, Hkv, N, d, dtype))
    return ATTN_ERR_INVALID_ARG;
  DeviceInfo* di = device_info();
  if (!di) return ATTN_ERR_CUDA;
  std::lock_guard<std::mutex> lock(di->pipe_mutex);
  if (!pipeline_ready(di)) return ATTN_ERR_CUDA;
  const size_t elt = fp8 ? 1 : 2;
  const int G = H / Hkv;
  HostChunk ch[kMaxChunks];
  size_t total = 0;
  const int nc = plan_host_chunks(B, H, Hkv, N, d, elt, ch, &total);
  uint8_t* w = static_cast<uint8_t*>(workspace);
  float* d_desc = reinterpret_cast<float*>(w + total - 256);
  const uint8_t* hq = static_cast<const uint8_t*>(q);
  const uint8_t* hk = static_cast<const uint8_t*>(k);
  const uint8_t* hv = static_cast<const uint8_t*>(v);
  uint8_t* ho = static_cast<uint8_t*>(o);
  uint8_t* hl = reinterpret_cast<uint8_t*>(lse);
  const size_t q_pitch = (size_t)H * d * elt, kv_pitch = (size_t)Hkv * d * elt, o_pitch = (size_t)H * d * 2;
  bool ok = cudaEventRecord(di->ev_start, stream) == cudaSuccess;
  for (cudaStream_t s : {di->s_in, di->s_out, di->s_comp[0], di->s_comp[1]})
    ok = ok && cudaStreamWaitEvent(s, di->ev_start, 0) == cudaSuccess;
  if (ok && fp8) {
    const float desc[3] = {*descale_q, *descale_k, *descale_v};
    ok = cudaMemcpyAsync(d_desc, desc, sizeof(desc), cudaMemcpyHostToDevice, di->s_in) == cudaSuccess;
  }
  // Uploads: rows [b0 N, (b0 + nb) N) of the [B N, heads, d] views, a head range of each row.
  for (int c = 0; ok && c < nc; ++c) {
    const HostChunk& x = ch[c];
    const size_t rows = (size_t)x.nb * N, row0 = (size_t)x.b0 * N;
    ok = cudaMemcpy2DAsync(w + x.off_q, (size_t)x.ng * G * d * elt, hq + row0 * q_pitch + (size_t)x.g0 * G * d * elt,
                           q_pitch, (size_t)x.ng * G * d * elt, rows, cudaMemcpyHostToDevice, di->s_in) == cudaSuccess &&
         cudaMemcpy2DAsync(w + x.off_k, (size_t)x.ng * d * elt, hk + row0 * kv_pitch + (size_t)x.g0 * d * elt,
                           kv_pitch, (size_t)x.ng * d * elt, rows, cudaMemcpyHostToDevice, di->s_in) == cudaSuccess &&
         cudaMemcpy2DAsync(w + x.off_v, (size_t)x.ng * d * elt, hv + row0 * kv_pitch + (size_t)x.g0 * d * elt,
                           kv_pitch, (size_t)x.ng * d * elt, rows, cudaMemcpyHostToDevice, di->s_in) == cudaSuccess &&
         cudaEventRecord(di->ev_in[c], di->s_in) == cudaSuccess;
  }
  // Kernels: each chunk is a [nb, N, ng G, d] problem, alternating between two streams so one
  // chunk's tail overlaps the next chunk's start.
  for (int c = 0; ok && c < nc; ++c) {
    const HostChunk& x = ch[c];
    cudaStream_t sc = di->s_comp[c & 1];
    ok = cudaStreamWaitEvent(sc, di->ev_in[c], 0) == cudaSuccess;
    if (!ok) break;
    st = attn_fwd(w + x.off_q, w + x.off_k, w + x.off_v, w + x.off_o, reinterpret_cast<float*>(w + x.off_lse), x.nb,
                  x.ng * G, x.ng, N, d, scale, causal, dtype, fp8 ? d_desc : nullptr, fp8 ? d_desc + 1 : nullptr,
                  fp8 ? d_desc + 2 : nullptr, sc);
    if (st != ATTN_OK) { ok = false; break; }
    ok = cudaEventRecord(di->ev_k[c], sc) == cudaSuccess;
  }
  // Downloads: O head ranges back into the strided host rows; LSE [B, H, N] rows are contiguous.
  for (int c = 0; ok && c < nc; ++c) {
    const HostChunk& x = ch[c];
    const size_t rows = (size_t)x.nb * N, row0 = (size_t)x.b0 * N;
    ok = cudaStreamWaitEvent(di->s_out, di->ev_k[c], 0) == cudaSuccess &&
         cudaMemcpy2DAsync(ho + row0 * o_pitch + (size_t)x.g0 * G * d * 2, o_pitch, w + x.off_o,
                           (size_t)x.ng * G * d * 2, (size_t)x.ng * G * d * 2, rows, cudaMemcpyDeviceToHost,
                           di->s_out) == cudaSuccess;
    for (int b = 0; ok && b < x.nb; ++b)
      ok = cudaMemcpyAsync(hl + (((size_t)(x.b0 + b) * H + (size_t)x.g0 * G) * N) * 4,
                           w + x.off_lse + (size_t)b * x.ng * G * N * 4, (size_t)x.ng * G * N * 4,
                           cudaMemcpyDeviceToHost, di->s_out) == cudaSuccess;
  }
  // The caller's stream resumes after the last download; the call returns when it is done.
  const bool joined = cudaEventRecord(di->ev_end, di->s_out) == cudaSuccess &&
                      cudaStreamWaitEvent(stream, di->ev_end, 0) == cudaSuccess;
  const bool synced = cudaStreamSynchronize(stream) == cudaSuccess;
  if (st != ATTN_OK) return st;
  return (ok && joined && synced) ? ATTN_OK : ATTN_ERR_CUDA;
}

int attn_fwd_tail_units(int B, int H, int N, int d, int causal, attn_dtype_t dtype, int* tiles, int* kv0,
                        int cap) {
  if (B < 1 || H < 1 || N < 1 || (d != 64 && d != 128 && d != 256)) return 0;
  if (dtype != ATTN_DTYPE_BF16 && dtype != ATTN_DTYPE_FP8_E4M3) return 0;
  int sms = 152;
  DeviceInfo* di = device_info();
  if (di) sms = di->num_sms;
  const long long rows = gb300::rows_per_work_tile(d);
  const long long n_tiles = (long long)B * H * ((N + rows - 1) / rows);
  if (n_tiles >= (1LL << 31)) return 0;
  gb300::AttnParams p;
  const int n = gb300::plan_tail(p, n_tiles, (N + 127) / 128, sms, causal != 0, dtype == ATTN_DTYPE_BF16 && d <= 128);
  for (int u = 0; u < n && u < cap; ++u) {
    if (tiles) tiles[u] = p.tail_tab[u].x;
    if (kv0) kv0[u] = p.tail_tab[u].y;
  }
  return n;
}

int attn_fwd_halved_tail_tiles(int B, int H, int N, int d, int causal) {
  return attn_fwd_tail_units(B, H, N, d, causal, ATTN_DTYPE_BF16, nullptr, nullptr, 0);
}

int attn_splitkv_num_splits(int B, int H, int Hkv, int Nq, int Nk, int d) {
  if (B < 1 || H < 1 || Hkv < 1 || H % Hkv != 0 || Nq < 1 || Nk < 1) return 1;
  int sms = 152;
  DeviceInfo* di = device_info();
  if (di) sms = di->num_sms;
  // The (batch, kv head, query block) units stream K and V at close to the HBM bandwidth once
  // about two thirds of the SMs or more take part. So split each unit as far as one wave of SMs
  // allows and no further: a second, partial wave, or more units per CTA, only adds Q loads,
  // partial-result writes and merge work.
  const long long units = (long long)B * Hkv * (((long long)Nq * (H / Hkv) + 127) / 128);
  const long long n_kvt = (Nk + 127) / 128;
  const long long s_max = std::min<long long>(n_kvt, kMaxSplits);
  const long long s = sms / units;
  return (int)std::max<long long>(1, std::min<long long>(s, s_max));
}

size_t attn_fwd_splitkv_workspace_bytes(int B, int H, int Nq, int d, int num_splits) {
  if (B < 1 || H < 1 || Nq < 1 || d < 1 || num_splits < 1 || num_splits > kMaxSplits) return 0;
  return splitkv_part_o_bytes(B, H, Nq, d, num_splits) + round_up((size_t)num_splits * B * H * Nq * 4, 256);
}

attn_status_t attn_fwd_splitkv(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                               int Hkv, int Nq, int Nk, int d, float scale, int num_splits, attn_dtype_t dtype,
                               const float* descale_q, const float* descale_k, const float* descale_v,
                               void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  if (Nq < 1 || Nk < 1 || num_splits < 1 || num_splits > kMaxSplits) return ATTN_ERR_INVALID_ARG;
  attn_status_t st = check_shape(B, H, Hkv, Nk, d, scale, dtype);
  if (st != ATTN_OK) return st;
  st = check_shape(B, H, Hkv, Nq, d, scale, dtype);
  if (st != ATTN_OK) return st;
  const int G = H / Hkv;
  if (G > 128 || (128 % G) != 0) return ATTN_ERR_UNSUPPORTED;   // G packed rows must tile 128
  const bool fp8 = dtype == ATTN_DTYPE_FP8_E4M3;
  if (!q || !k || !v || !o || !lse || !workspace) return ATTN_ERR_INVALID_ARG;
  if (fp8 && (!descale_q || !descale_k || !descale_v)) return ATTN_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) || !aligned(lse, 4) ||
      !aligned(workspace, 256))
    return ATTN_ERR_INVALID_ARG;
  if (workspace_bytes < attn_fwd_splitkv_workspace_bytes(B, H, Nq, d, num_splits)) return ATTN_ERR_INVALID_ARG;
  const size_t elt = fp8 ? 1 : 2;
  const size_t nq = (size_t)B * Nq * H * d, nkv = (size_t)B * Nk * Hkv * d;
  const size_t o_bytes = nq * 2, lse_bytes = (size_t)B * H * Nq * 4;
  const void* ins[3] = {q, k, v};
  const size_t in_bytes[3] = {nq * elt, nkv * elt, nkv * elt};
  for (int i = 0; i < 3; ++i)
    if (ranges_overlap(o, o_bytes, ins[i], in_bytes[i]) || ranges_overlap(lse, lse_bytes, ins[i], in_bytes[i]) ||
        ranges_overlap(workspace, workspace_bytes, ins[i], in_bytes[i]))
      return ATTN_ERR_INVALID_ARG;
  if (ranges_overlap(o, o_bytes, lse, lse_bytes) || ranges_overlap(workspace, workspace_bytes, o, o_bytes) ||
      ranges_overlap(workspace, workspace_bytes, lse, lse_bytes))
    return ATTN_ERR_INVALID_ARG;
  DeviceInfo* di = device_info();
  if (!di) return ATTN_ERR_CUDA;
  gb300::LaunchArgs a;
  memset(&a, 0, sizeof(a));
  if (!make_map_q_packed(&a.tm_q, q, fp8, d, Nq, H, Hkv, B) || !make_map(&a.tm_k, k, fp8, d, Nk, Hkv, B, 128) ||
      !make_map(&a.tm_v, v, fp8, d, Nk, Hkv, B, 128))
    return ATTN_ERR_CUDA;
  const int n_kvt = (Nk + 127) / 128;
  const int S = num_splits < n_kvt ? num_splits : n_kvt;   // every split gets at least one KV tile
  const int rows = gb300::rows_per_split_work_tile(d);
  float* part_o = static_cast<float*>(workspace);
  float* part_lse = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + splitkv_part_o_bytes(B, H, Nq, d, num_splits));
  gb300::AttnParams& p = a.params;
  p.o = o;
  p.lse = lse;
  p.descale_q = descale_q;
  p.descale_k = descale_k;
  p.descale_v = descale_v;
  p.B = B;
  p.H = H;
  p.Hkv = Hkv;
  p.N = Nq;
  p.Nk = Nk;
  p.G = G;
  p.n_splits = S;
  p.n_kvt = n_kvt;
  p.part_o = part_o;
  p.part_lse = part_lse;
  p.scale_log2 = std::fabs(scale) * 1.4426950408889634f;
  p.qk_negate = scale < 0.0f ? gb300::kIdescNegateA : 0u;
  p.n_mb = (int)(((long long)Nq * G + rows - 1) / rows);
  const long long tiles = (long long)B * Hkv * S * p.n_mb;
  if (tiles >= (1LL << 31)) return ATTN_ERR_UNSUPPORTED;
  p.n_tiles = (int)tiles;
  p.status = di->status;
  p.timeout_ns = g_timeout_ns ? g_timeout_ns : kDefaultTimeoutNs;
  p.debug_skip_load = g_skip_load;
  a.num_sms = di->num_sms;
  cudaError_t e;
  switch (d) {
    case 64: e = dispatch_split<64>(a, fp8, stream); break;
    case 128: e = dispatch_split<128>(a, fp8, stream); break;
    default: e = dispatch_split<256>(a, fp8, stream); break;
  }
  if (e != cudaSuccess) return ATTN_ERR_CUDA;
  e = gb300::launch_splitkv_combine(part_o, part_lse, o, lse, S, B, H, Nq, d, di->num_sms, stream);
  return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

size_t attn_varlen_plan_bytes(int B, int H, int total_q, int d) {
  if (B < 1 || H < 1 || total_q < 0 || (d != 64 && d != 128 && d != 256)) return 0;
  const long long tiles = varlen_tile_bound(B, H, total_q, d);
  if (tiles >= INT_MAX || B >= INT_MAX / 2) return 0;
  return (size_t)gb300::plan_tiles_offset(B) * 4 + (size_t)tiles * 8;
}

attn_status_t attn_varlen_plan(const int* cu_seqlens_q, const int* cu_seqlens_k, int B, int H, int total_q,
                               int total_k, int d, int causal, void* plan, size_t plan_bytes, cudaStream_t stream) {
  if (!cu_seqlens_q || !cu_seqlens_k || !plan) return ATTN_ERR_INVALID_ARG;
  if (B < 1 || H < 1 || total_q < 0 || total_k < 0) return ATTN_ERR_INVALID_ARG;
  if (d != 64 && d != 128 && d != 256) return ATTN_ERR_UNSUPPORTED;
  if (!aligned(plan, 16) || !aligned(cu_seqlens_q, 4) || !aligned(cu_seqlens_k, 4)) return ATTN_ERR_INVALID_ARG;
  const size_t need = attn_varlen_plan_bytes(B, H, total_q, d);
  if (need == 0) return ATTN_ERR_UNSUPPORTED;
  if (plan_bytes < need) return ATTN_ERR_INVALID_ARG;
  const size_t head = (size_t)gb300::plan_tiles_offset(B) * 4;
  const size_t cap = (plan_bytes - head) / 8;
  const int capacity = cap > (size_t)INT_MAX ? INT_MAX : (int)cap;
  const cudaError_t e = gb300::launch_varlen_plan(cu_seqlens_q, cu_seqlens_k, B, H, gb300::rows_per_work_tile(d),
                                                  causal != 0, total_q, total_k, capacity, static_cast<int*>(plan),
                                                  stream);
  return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

attn_status_t attn_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse,
                              const int* cu_seqlens_q, const int* cu_seqlens_k, const void* plan, size_t plan_bytes,
                              int B, int H, int Hkv, int total_q, int total_k, int d, float scale, int causal,
                              attn_dtype_t dtype, const float* descale_q, const float* descale_k,
                              const float* descale_v, cudaStream_t stream) {
  if (total_q < 0 || total_k < 0 || B < 1) return ATTN_ERR_INVALID_ARG;
  attn_status_t st = check_shape(1, H, Hkv, total_q > 0 ? total_q : 1, d, scale, dtype);
  if (st != ATTN_OK) return st;
  if (varlen_tile_bound(B, H, total_q, d) >= INT_MAX) return ATTN_ERR_UNSUPPORTED;
  const bool fp8 = dtype == ATTN_DTYPE_FP8_E4M3;
  if (!q || !k || !v || !o || !lse || !cu_seqlens_q || !cu_seqlens_k || !plan) return ATTN_ERR_INVALID_ARG;
  if (fp8 && (!descale_q || !descale_k || !descale_v)) return ATTN_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) || !aligned(lse, 4) ||
      !aligned(plan, 16) || !aligned(cu_seqlens_q, 4) || !aligned(cu_seqlens_k, 4))
    return ATTN_ERR_INVALID_ARG;
  if (plan_bytes < (size_t)gb300::plan_tiles_offset(B) * 4) return ATTN_ERR_INVALID_ARG;
  if (total_q == 0) return ATTN_OK;   // no query rows: nothing to write
  const size_t elt = fp8 ? 1 : 2;
  const size_t nq = (size_t)total_q * H * d, nkv = (size_t)total_k * Hkv * d;
  const size_t o_bytes = nq * 2, lse_bytes = (size_t)H * total_q * 4;
  const void* ins[3] = {q, k, v};
  const size_t in_bytes[3] = {nq * elt, nkv * elt, nkv * elt};
  for (int i = 0; i < 3; ++i)
    if (ranges_overlap(o, o_bytes, ins[i], in_bytes[i]) || ranges_overlap(lse, lse_bytes, ins[i], in_bytes[i]))
      return ATTN_ERR_INVALID_ARG;
  if (ranges_overlap(o, o_bytes, lse, lse_bytes)) return ATTN_ERR_INVALID_ARG;
  DeviceInfo* di = device_info();
  if (!di) return ATTN_ERR_CUDA;
  gb300::LaunchArgs a;
  memset(&a, 0, sizeof(a));
  // Packed tensors as one batch of total rows. With no keys at all the k/v maps are never read.
  const int kv_rows = total_k > 0 ? total_k : 1;
  if (!make_map(&a.tm_q, q, fp8, d, total_q, H, 1) || !make_map(&a.tm_k, k, fp8, d, kv_rows, Hkv, 1) ||
      !make_map(&a.tm_v, v, fp8, d, kv_rows, Hkv, 1))
    return ATTN_ERR_CUDA;
  gb300::AttnParams& p = a.params;
  p.o = o;
  p.lse = lse;
  p.descale_q = descale_q;
  p.descale_k = descale_k;
  p.descale_v = descale_v;
  p.B = B;
  p.H = H;
  p.Hkv = Hkv;
  p.N = total_q;
  p.Nk = total_k;
  p.G = H / Hkv;
  p.o_v8 = aligned(o, 32) ? 1 : 0;
  p.scale_log2 = std::fabs(scale) * 1.4426950408889634f;
  p.qk_negate = scale < 0.0f ? gb300::kIdescNegateA : 0u;
  // Launch bound and read limit: the tiles a valid plan can hold, and no more than the buffer has.
  const size_t held = (plan_bytes - (size_t)gb300::plan_tiles_offset(B) * 4) / 8;
  const long long bound = varlen_tile_bound(B, H, total_q, d);
  p.n_tiles = (int)std::min<long long>(bound, (long long)std::min<size_t>(held, (size_t)INT_MAX));
  if (p.n_tiles < 1) p.n_tiles = 1;
  p.n_splits = 1;
  p.cu_q = cu_seqlens_q;
  p.cu_k = cu_seqlens_k;
  p.plan = static_cast<const int*>(plan);
  p.status = di->status;
  p.timeout_ns = g_timeout_ns ? g_timeout_ns : kDefaultTimeoutNs;
  p.debug_skip_load = 0;
  a.num_sms = di->num_sms;
  cudaError_t e;
  switch (d) {
    case 64: e = dispatch_varlen<64>(a, causal != 0, fp8, stream); break;
    case 128: e = dispatch_varlen<128>(a, causal != 0, fp8, stream); break;
    default: e = dispatch_varlen<256>(a, causal != 0, fp8, stream); break;
  }
  return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

size_t attn_bwd_workspace_bytes(int B, int H, int N) {
  if (B < 1 || H < 1 || N < 1) return 0;
  const size_t np = ((size_t)N + 127) / 128 * 128;
  return 2 * round_up((size_t)B * H * np * 4, 256);
}

attn_status_t attn_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
                       const void* dout, void* dq, void* dk, void* dv, int B, int H, int Hkv, int N, int d,
                       float scale, int causal, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  attn_status_t st = check_shape(B, H, Hkv, N, d, scale, ATTN_DTYPE_BF16);
  if (st != ATTN_OK) return st;
  if (d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED;   // dK, dV, S, dP must fit TMEM's 512 columns
  if (!q || !k || !v || !o || !lse || !dout || !dq || !dk || !dv || !workspace) return ATTN_ERR_INVALID_ARG;
  const void* a16[8] = {q, k, v, o, dout, dq, dk, dv};
  for (const void* ptr : a16)
    if (!aligned(ptr, 16)) return ATTN_ERR_INVALID_ARG;
  if (!aligned(lse, 4) || !aligned(workspace, 256)) return ATTN_ERR_INVALID_ARG;
  if (workspace_bytes < attn_bwd_workspace_bytes(B, H, N)) return ATTN_ERR_INVALID_ARG;
  const size_t nq = (size_t)B * N * H * d * 2, nkv = (size_t)B * N * Hkv * d * 2, nl = (size_t)B * H * N * 4;
  // outputs (and the workspace) must not overlap any input or each other
  const void* outs[4] = {dq, dk, dv, workspace};
  const size_t out_bytes[4] = {nq, nkv, nkv, workspace_bytes};
  const void* ins[6] = {q, k, v, o, dout, lse};
  const size_t in_bytes[6] = {nq, nkv, nkv, nq, nq, nl};
  for (int i = 0; i < 4; ++i) {
    for (int j = 0; j < 6; ++j)
      if (ranges_overlap(outs[i], out_bytes[i], ins[j], in_bytes[j])) return ATTN_ERR_INVALID_ARG;
    for (int j = i + 1; j < 4; ++j)
      if (ranges_overlap(outs[i], out_bytes[i], outs[j], out_bytes[j])) return ATTN_ERR_INVALID_ARG;
  }
  DeviceInfo* di = device_info();
  if (!di) return ATTN_ERR_CUDA;
  gb300::BwdLaunchArgs a;
  memset(&a, 0, sizeof(a));
  if (!make_map(&a.tm_q, q, false, d, N, H, B) || !make_map(&a.tm_do, dout, false, d, N, H, B) ||
      !make_map(&a.tm_k, k, false, d, N, Hkv, B) || !make_map(&a.tm_v, v, false, d, N, Hkv, B))
    return ATTN_ERR_CUDA;
  const int np = (N + 127) / 128 * 128;
  a.o = o;
  a.dout = dout;
  a.lse = lse;
  a.nlse2 = static_cast<float*>(workspace);
  a.dd = reinterpret_cast<float*>(static_cast<char*>(workspace) + round_up((size_t)B * H * np * 4, 256));
  a.num_sms = di->num_sms;
  gb300::BwdParams& p = a.params;
  p.dq = static_cast<__nv_bfloat16*>(dq);
  p.dk = static_cast<__nv_bfloat16*>(dk);
  p.dv = static_cast<__nv_bfloat16*>(dv);
  p.nlse2 = a.nlse2;
  p.dd = a.dd;
  p.B = B;
  p.H = H;
  p.Hkv = Hkv;
  p.G = H / Hkv;
  p.N = N;
  p.Np = np;
  p.n_t = np / 128;
  p.scale = scale;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.status = di->status;
  p.timeout_ns = g_timeout_ns ? g_timeout_ns : kDefaultTimeoutNs;
  return gb300::launch_attn_bwd(a, d, causal != 0, stream) == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

size_t attn_quantize_e4m3_descale_count(int B, int N, int Hx, int block_rows) {
  if (B < 1 || N < 1 || Hx < 1 || block_rows < 1) return 0;
  return (size_t)B * Hx * (size_t)((N + (long long)block_rows - 1) / block_rows);
}

attn_status_t attn_quantize_e4m3(const void* x, void* x8, float* descale, int B, int N, int Hx, int d,
                                 int block_rows, const float* signs, cudaStream_t stream) {
  if (!x || !x8 || !descale) return ATTN_ERR_INVALID_ARG;
  if (B < 1 || N < 1 || Hx < 1 || block_rows < 1) return ATTN_ERR_INVALID_ARG;
  if (d != 64 && d != 128 && d != 256) return ATTN_ERR_UNSUPPORTED;
  if (!aligned(x, 16) || !aligned(x8, 16) || !aligned(descale, 4) || (signs && !aligned(signs, 4)))
    return ATTN_ERR_INVALID_ARG;
  const long long nblk = (N + (long long)block_rows - 1) / block_rows;
  // Chunks (one TMA load each, at most 128 rows of one batch and head): 128 rows holding whole
  // blocks when the block size is a power of two from 8 to 128; one block when it is another size
  // below 128; 128-row pieces of longer blocks. Rows split into spans of whole chunks.
  int chunk_rows, span, cps;
  if (block_rows <= 128) {
    chunk_rows = (block_rows >= 8 && 128 % block_rows == 0) ? 128 : block_rows;
    span = chunk_rows;
    cps = 1;
  } else {
    chunk_rows = 128;
    span = block_rows;
    cps = (block_rows + 127) / 128;
  }
  const long long nspan = (N + (long long)span - 1) / span;
  if ((long long)B * Hx * nspan * cps > INT_MAX || (long long)B * N * Hx > INT_MAX ||
      (long long)B * Hx * nblk > INT_MAX)
    return ATTN_ERR_UNSUPPORTED;
  // The codes and descales must not overlap x: other CTAs may still be reading it.
  const size_t elems = (size_t)B * N * Hx * d;
  const uintptr_t xb = (uintptr_t)x, xe = xb + elems * 2;
  const uintptr_t qb = (uintptr_t)x8, qe = qb + elems;
  const uintptr_t db = (uintptr_t)descale, de = db + (size_t)(B * Hx * nblk) * 4;
  if ((qb < xe && xb < qe) || (db < xe && xb < de) || (db < qe && qb < de)) return ATTN_ERR_INVALID_ARG;
  DeviceInfo* di = device_info();
  if (!di) return ATTN_ERR_CUDA;
  gb300::QuantLaunch q;
  memset(&q, 0, sizeof(q));
  if (!make_rows_map(&q.tm_x, x, d, N, Hx, B, chunk_rows)) return ATTN_ERR_CUDA;
  q.x8 = static_cast<uint8_t*>(x8);
  q.descale = descale;
  q.signs = signs;
  q.B = B;
  q.N = N;
  q.Hx = Hx;
  q.d = d;
  q.block_rows = block_rows;
  q.nblk = (int)nblk;
  q.span = span;
  q.cps = cps;
  q.nspan = (int)nspan;
  q.chunk_rows = chunk_rows;
  q.grp_rows = std::min(block_rows, chunk_rows);
  q.x8_v8 = aligned(x8, 32) ? 1 : 0;
  q.status = di->status;
  q.timeout_ns = g_timeout_ns ? g_timeout_ns : kDefaultTimeoutNs;
  q.num_sms = di->num_sms;
  return gb300::launch_quantize_e4m3(q, stream) == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

attn_status_t attn_get_status(cudaStream_t stream) { return attn_get_status_detail(stream, nullptr); }

attn_status_t attn_get_status_detail(cudaStream_t stream, uint32_t* detail) {
  if (detail) *detail = 0;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return ATTN_ERR_CUDA;
  uint32_t v = 0;
  if (cudaMemcpyFromSymbol(&v, g_attn_status, sizeof(v)) != cudaSuccess) return ATTN_ERR_CUDA;
  if (detail) *detail = v;
  if (!v) return ATTN_OK;
  return (v & 0x40000000u) ? ATTN_ERR_TIMEOUT : ATTN_ERR_INVALID_ARG;   // 0x20000000: bad varlen plan
}

attn_status_t attn_clear_status(void) {
  const uint32_t zero = 0;
  if (cudaMemcpyToSymbol(g_attn_status, &zero, sizeof(zero)) != cudaSuccess) return ATTN_ERR_CUDA;
  return cudaDeviceSynchronize() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

const char* attn_status_string(attn_status_t s) {
  switch (s) {
    case ATTN_OK: return "ok";
    case ATTN_ERR_INVALID_ARG: return "invalid argument";
    case ATTN_ERR_UNSUPPORTED: return "unsupported configuration";
    case ATTN_ERR_CUDA: return "CUDA error";
    case ATTN_ERR_TIMEOUT: return "kernel wait timed out";
  }
  return "unknown status";
}

void attn_debug_set(unsigned long long timeout_ns, int skip_load) {
  g_timeout_ns = timeout_ns;
  g_skip_load = skip_load;
}

int attn_version(void) { return 100; }

}  // extern "C"
