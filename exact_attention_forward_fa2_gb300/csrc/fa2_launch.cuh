// Launch side of the forward kernel: each instantiation unit (one per dtype and
// head dim) includes this file and calls launch_cfg with its tile configuration.
#pragma once

#include <atomic>

#include "fa2_fwd_kernel.cuh"

namespace fa2 {

// Sets the dynamic shared-memory limit once per device and kernel, then launches
// one CTA per (work unit, key split) on the caller's stream.  A work unit is C's
// kQTiles query tiles of one head, or the single query tile of kQTiles heads that
// share a key/value head (pair_heads, set by the host for two-tile configurations).
template <class C, bool kCausal, bool kMod, bool kWin>
cudaError_t launch_one(FwdLaunch& L, std::atomic<bool>& attr_done) {
  if (!attr_done.load(std::memory_order_acquire)) {
    // setting the limit is idempotent, so threads that race here only repeat it
    const cudaError_t e = cudaFuncSetAttribute(fa2_fwd_kernel<C, kCausal, kMod, kWin>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               C::kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_done.store(true, std::memory_order_release);
  }
  if (L.params.pair_heads) {  // one tile of each of two heads per unit
    L.params.units_per_head = 1;
    L.params.num_units = L.params.BH / 2;
  } else {
    L.params.units_per_head = (L.params.M + C::kQTiles * C::BM - 1) / (C::kQTiles * C::BM);
    L.params.num_units = L.params.units_per_head * L.params.BH;
  }
  const dim3 grid(static_cast<unsigned>(L.params.num_units * L.params.num_splits));
  const dim3 block(C::kThreads);
  fa2_fwd_kernel<C, kCausal, kMod, kWin><<<grid, block, C::kSmemBytes, L.stream>>>(L.tmQ, L.tmK, L.tmV,
                                                                                  L.tmO, L.params);
  return cudaGetLastError();
}

// C: the plain and ALiBi kernels; CW: the sliding-window kernels (both with one
// softmax warpgroup per query tile); CH: the softcap kernels.  The softcap spends
// two MUFU operations per score (the tanh and the exponential); there two softmax
// warpgroups per query tile, each owning 64 keys of a row, keep the MUFU pipe
// busier (+6% on bf16 D = 128, measured).  On every other path one warpgroup per
// tile is faster (the split costs an exchange per row and registers).  The host
// sizes the grid, the tensor maps' key tiles and the head pairing for the
// configuration that runs (qtiles_for and kv_tile_for with the same flags).
template <class C, class CW, class CH>
cudaError_t launch_cfg(FwdLaunch& L) {
  static_assert(CH::kHalves == 2 && C::kHalves == 1 && CW::kHalves == 1, "one and two warpgroups per query tile");
  static std::atomic<bool> attr_done[64][10] = {};
  int dev = 0;
  const cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::atomic<bool>* done = attr_done[dev];
  // kWin: spans and masks of a sliding window; kMod: softcap or ALiBi scores
  if (L.mod && L.params.cap_in > 0.f) {
    if (L.win)
      return L.causal ? launch_one<CH, true, true, true>(L, done[9]) : launch_one<CH, false, true, true>(L, done[8]);
    return L.causal ? launch_one<CH, true, true, false>(L, done[7]) : launch_one<CH, false, true, false>(L, done[6]);
  }
  if (L.win)
    return L.causal ? launch_one<CW, true, true, true>(L, done[5]) : launch_one<CW, false, true, true>(L, done[4]);
  if (L.mod)
    return L.causal ? launch_one<C, true, true, false>(L, done[3]) : launch_one<C, false, true, false>(L, done[2]);
  return L.causal ? launch_one<C, true, false, false>(L, done[1]) : launch_one<C, false, false, false>(L, done[0]);
}

}  // namespace fa2
