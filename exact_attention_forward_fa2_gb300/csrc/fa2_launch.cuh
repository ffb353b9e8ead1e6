// Launch side of the forward kernel: one instantiation unit per (dtype, D)
// includes this file and defines its entry through FA2_DEFINE_LAUNCH.
#pragma once

#include "fa2_fwd_kernel.cuh"

namespace fa2 {

// Sets the dynamic shared-memory limit once per device, then launches one CTA
// per work unit on the caller's stream.
template <class C>
cudaError_t launch_cfg(FwdLaunch& L) {
  static bool attr_done[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_done[dev]) {
    e = cudaFuncSetAttribute(fa2_fwd_kernel<C, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             C::kSmemBytes);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(fa2_fwd_kernel<C, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             C::kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_done[dev] = true;
  }
  L.params.units_per_head = (L.params.M + C::kQTiles * C::BM - 1) / (C::kQTiles * C::BM);
  L.params.num_units = L.params.units_per_head * L.params.BH;
  const dim3 grid(static_cast<unsigned>(L.params.num_units * L.params.num_splits));
  const dim3 block(C::kThreads);
  if (L.causal)
    fa2_fwd_kernel<C, true><<<grid, block, C::kSmemBytes, L.stream>>>(L.tmQ, L.tmK, L.tmV, L.tmO,
                                                                       L.params);
  else
    fa2_fwd_kernel<C, false><<<grid, block, C::kSmemBytes, L.stream>>>(L.tmQ, L.tmK, L.tmV, L.tmO,
                                                                        L.params);
  return cudaGetLastError();
}

}  // namespace fa2
