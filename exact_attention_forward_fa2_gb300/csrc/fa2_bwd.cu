// Instantiation and launch of the backward kernels (bf16, head dim 64 and 128),
// all on the caller's stream: preprocess, then either the dK/dV pass and the dQ
// pass, or (dQ by reduction, head dim 128) the dK/dV/dQ pass and the dQ convert.
#include <algorithm>
#include <atomic>

#include "fa2_bwd_kernel.cuh"

namespace fa2 {

namespace {

template <class C, bool kCausal>
cudaError_t launch_dkdv(BwdLaunch& L, std::atomic<bool>& attr_done) {
  using Lay = DkvLayout<C>;
  if (!attr_done.load(std::memory_order_acquire)) {  // idempotent: a race only repeats it
    const cudaError_t e = cudaFuncSetAttribute(bwd_dkdv_kernel<C, kCausal>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize, Lay::kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_done.store(true, std::memory_order_release);
  }
  const dim3 grid(static_cast<unsigned>(L.params.BHkv * L.params.n_ktiles));
  bwd_dkdv_kernel<C, kCausal><<<grid, C::kThreads, Lay::kSmemBytes, L.stream>>>(
      L.tmQ64, L.tmdO64, L.tmK128, L.tmV128, L.tmdK, L.tmdV, L.params);
  return cudaGetLastError();
}

template <class C, bool kCausal>
cudaError_t launch_dq(BwdLaunch& L, std::atomic<bool>& attr_done) {
  if (!attr_done.load(std::memory_order_acquire)) {  // idempotent: a race only repeats it
    const cudaError_t e = cudaFuncSetAttribute(bwd_dq_kernel<C, kCausal>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_done.store(true, std::memory_order_release);
  }
  const int pairs = (L.params.n_qtiles + C::kQT - 1) / C::kQT;
  const dim3 grid(static_cast<unsigned>(L.params.BH * pairs));
  bwd_dq_kernel<C, kCausal><<<grid, C::kThreads, C::kSmemBytes, L.stream>>>(L.tmQ128, L.tmdO128, L.tmK64,
                                                                           L.tmV64, L.tmdQ, L.params);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_all(BwdLaunch& L, int dev, int sms) {
  using C = BwdCfg<D, D == 64 ? 8 : 4>;  // deeper ring at D = 64 (keeps one CTA per SM)
  static std::atomic<bool> attr[64][6] = {};
  const int64_t rows_pad = static_cast<int64_t>(L.params.BH) * L.params.Mpad;
  const int64_t rows_per_block = 8 * (32 / (D / 8));  // 8 warps, 32 / (D / 8) rows each per pass
  const int64_t need = (rows_pad + rows_per_block - 1) / rows_per_block;
  const int blocks = static_cast<int>(need < 8LL * sms ? need : 8LL * sms);
  bwd_preprocess_kernel<D><<<blocks, 256, 0, L.stream>>>(
      static_cast<const __nv_bfloat16*>(L.o), static_cast<const __nv_bfloat16*>(L.dout), L.lse, L.nl2, L.dlt,
      L.dqacc, L.params.M, L.params.Mpad, rows_pad);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  std::atomic<bool>* a = attr[dev];
  if constexpr (D == 128) {
    if (L.dqacc) {  // dQ by reduction: dK, dV and the dQ accumulator in one pass, then dQ in bf16
      using CR = BwdCfg<D, 3, true>;  // three stages beside the two dS^T tiles
      e = L.causal ? launch_dkdv<CR, true>(L, a[5]) : launch_dkdv<CR, false>(L, a[4]);
      if (e != cudaSuccess) return e;
      const int64_t n8 = static_cast<int64_t>(L.params.BH) * L.params.M * (D / 8);
      const int64_t cblocks = std::min<int64_t>((n8 + 255) / 256, 16LL * sms);
      bwd_dq_convert_kernel<D><<<static_cast<unsigned>(cblocks), 256, 0, L.stream>>>(
          L.dqacc, static_cast<__nv_bfloat16*>(L.dq), L.params.scale, L.params.M, L.params.Mpad, n8);
      return cudaGetLastError();
    }
  }
  e = L.causal ? launch_dkdv<C, true>(L, a[1]) : launch_dkdv<C, false>(L, a[0]);
  if (e != cudaSuccess) return e;
  using CQ = DqCfg<D, D == 64 ? 4 : 3>;  // two query tiles per CTA; K/V ring as deep as fits
  return L.causal ? launch_dq<CQ, true>(L, a[3]) : launch_dq<CQ, false>(L, a[2]);
}

}  // namespace

cudaError_t launch_bwd(BwdLaunch& L, int D) {
  int dev = 0, sms = 148;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  return D == 64 ? launch_all<64>(L, dev, sms) : launch_all<128>(L, dev, sms);
}

}  // namespace fa2
