// Definition of the per-instance launcher; included by the instantiation units only.
#pragma once
#include "launch.h"

namespace gb300 {

template <int D, bool CAUSAL, bool FP8, bool SPLIT, bool VARLEN>
cudaError_t launch_attn_fwd(LaunchArgs& a, cudaStream_t stream) {
  using C = AttnCfg<D, CAUSAL, FP8, SPLIT, VARLEN>;
  auto kernel = attn_fwd_kernel<C>;
  // The attribute is per device; setting it on every call is cheap and keeps this stateless.
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  if constexpr (C::REG_SPLIT) {
    // setmaxnreg redistributes the registers the block was launched with; refuse to launch if the
    // compiled per-thread count leaves less than the split needs.
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, kernel);
    if (e != cudaSuccess) return e;
    if (fa.numRegs * C::THREADS < C::REGS_NEEDED) return cudaErrorInvalidConfiguration;
  }
  // Varlen: n_tiles is the host's upper bound; the kernel reads the plan's own count.
  const int grid = a.params.n_tiles < a.num_sms ? a.params.n_tiles : a.num_sms;
  if (!a.dependent) {
    kernel<<<grid, C::THREADS, C::SMEM_BYTES, stream>>>(a.tm_q, a.tm_k, a.tm_v, a.params);
    return cudaGetLastError();
  }
  // Programmatic dependent: its CTAs may start on SMs the previous grid has left, before that
  // grid ends; the kernel waits (griddepcontrol.wait) before reading the previous grid's output.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(C::THREADS);
  cfg.dynamicSmemBytes = C::SMEM_BYTES;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, a.tm_q, a.tm_k, a.tm_v, a.params);
}

}  // namespace gb300
