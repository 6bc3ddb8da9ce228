// Split-KV combine: each KV range s produced a normalized partial output O_s and its log-sum-exp
// LSE_s over the keys of that range. The full result over all keys is
//   LSE = ln sum_s exp(LSE_s),   O = sum_s exp(LSE_s - LSE) O_s,
// a direct consequence of the softmax definition (the "combine math" of split-KV decoding named in
// the "Hopper" tag page (l1-ca0.github.io), section 10.2.1 title).
// One warp per output row; each lane owns D/32 consecutive columns. Memory-bound: every partial
// row is read once and O is written once in bf16. The kernel is launched as a programmatic
// dependent of the split kernel: its CTAs may be scheduled while the split kernel runs and wait
// (griddepcontrol.wait) until that grid has finished and its writes are visible, so the launch
// latency of this short kernel overlaps the split kernel's tail.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cstdint>
#include "launch.h"

namespace gb300 {

template <int D>
__global__ void __launch_bounds__(256) splitkv_combine_kernel(const float* __restrict__ part_o,
                                                              const float* __restrict__ part_lse,
                                                              __nv_bfloat16* __restrict__ o, float* __restrict__ lse,
                                                              int S, int B, int H, int Nq) {
  constexpr int PER = D / 32;   // columns per lane
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int lane = threadIdx.x & 31;
  const long long rows = (long long)B * H * Nq;   // row = (b H + h) Nq + n, the layout of lse
  const long long nwarps = (long long)gridDim.x * (blockDim.x >> 5);
  for (long long row = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); row < rows; row += nwarps) {
    float mx = -INFINITY;
    for (int s = lane; s < S; s += 32) mx = fmaxf(mx, part_lse[(long long)s * rows + row]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    float sum = 0.f;
    for (int s = lane; s < S; s += 32) sum += expf(part_lse[(long long)s * rows + row] - mx);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
    const float lse_row = mx + logf(sum);
    float acc[PER];
#pragma unroll
    for (int i = 0; i < PER; ++i) acc[i] = 0.f;
    for (int s = 0; s < S; ++s) {
      const float wgt = expf(part_lse[(long long)s * rows + row] - lse_row);
      const float* src = part_o + ((long long)s * rows + row) * D + lane * PER;
#pragma unroll
      for (int i = 0; i < PER; i += 2) {
        const float2 x = *reinterpret_cast<const float2*>(src + i);
        acc[i] = fmaf(wgt, x.x, acc[i]);
        acc[i + 1] = fmaf(wgt, x.y, acc[i + 1]);
      }
    }
    const long long n = row % Nq, bh = row / Nq, h = bh % H, b = bh / H;
    __nv_bfloat16* dst = o + ((b * Nq + n) * H + h) * D + lane * PER;
#pragma unroll
    for (int i = 0; i < PER; i += 2)
      *reinterpret_cast<__nv_bfloat162*>(dst + i) = __floats2bfloat162_rn(acc[i], acc[i + 1]);
    if (lane == 0) lse[row] = lse_row;
  }
}

cudaError_t launch_splitkv_combine(const float* part_o, const float* part_lse, void* o, float* lse, int S, int B,
                                   int H, int Nq, int D, int num_sms, cudaStream_t stream) {
  const long long rows = (long long)B * H * Nq;
  long long blocks = (rows + 7) / 8;
  const long long cap = 8LL * num_sms;
  if (blocks > cap) blocks = cap;
  auto* ob = static_cast<__nv_bfloat16*>(o);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)blocks);
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  switch (D) {
    case 64: return cudaLaunchKernelEx(&cfg, splitkv_combine_kernel<64>, part_o, part_lse, ob, lse, S, B, H, Nq);
    case 128: return cudaLaunchKernelEx(&cfg, splitkv_combine_kernel<128>, part_o, part_lse, ob, lse, S, B, H, Nq);
    case 256: return cudaLaunchKernelEx(&cfg, splitkv_combine_kernel<256>, part_o, part_lse, ob, lse, S, B, H, Nq);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace gb300
