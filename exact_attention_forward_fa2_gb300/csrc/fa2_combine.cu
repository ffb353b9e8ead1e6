// Split-KV combine: merges the per-split partial results of the forward kernel.
//
// For one query row, split s saw a slice of the keys and wrote O_s (its softmax-
// weighted sum of V rows, already divided by its own row sum l_s) and
// L_s = m_s + ln l_s.  The whole row is then
//     L = ln sum_s exp(L_s),   O = sum_s exp(L_s - L) O_s,
// the same merge of partial softmax states that the online recurrence performs
// tile by tile ("From FlashAttention to FlashAttention 2", Online Softmax; the
// split-KV dispatch of Layer 2: C++ Entry Point).  A split with no visible key for
// the row has L_s = -inf and contributes nothing.
//
// Memory-bound: each row reads num_splits * (D + 1) fp32 values and writes D
// outputs plus L.  One warp per row, each lane owning D/32 consecutive columns
// (16-byte loads for D = 128), rows spread over a grid sized to the SM count.
#include <cuda_runtime.h>
#include <cuda_bf16.h>

#include <cstdint>

namespace fa2 {

template <int D, bool kBF16>
__global__ void __launch_bounds__(256) splitkv_combine_kernel(const float* __restrict__ o_part,
                                                              const float* __restrict__ l_part,
                                                              void* __restrict__ o,
                                                              float* __restrict__ lse, int64_t rows,
                                                              int num_splits) {
  constexpr int kPer = D / 32;  // columns per lane
  const int lane = static_cast<int>(threadIdx.x) % 32;
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x / 32);
  for (int64_t row = static_cast<int64_t>(blockIdx.x) * (blockDim.x / 32) + threadIdx.x / 32;
       row < rows; row += warps) {
    float lmax = -INFINITY;
    for (int s = 0; s < num_splits; ++s) lmax = fmaxf(lmax, l_part[s * rows + row]);
    float acc[kPer];
#pragma unroll
    for (int e = 0; e < kPer; ++e) acc[e] = 0.f;
    float denom = 0.f;
    if (lmax != -INFINITY) {
      for (int s = 0; s < num_splits; ++s) {
        const float ls = l_part[s * rows + row];
        if (ls == -INFINITY) continue;
        const float w = expf(ls - lmax);
        denom += w;
        const float* src = o_part + (s * rows + row) * D + lane * kPer;
#pragma unroll
        for (int e = 0; e < kPer; e += 2) {
          const float2 x = *reinterpret_cast<const float2*>(src + e);
          acc[e] = fmaf(w, x.x, acc[e]);
          acc[e + 1] = fmaf(w, x.y, acc[e + 1]);
        }
      }
    }
    const float inv = denom > 0.f ? 1.0f / denom : 0.f;
    if constexpr (kBF16) {
      __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(o) + row * D + lane * kPer;
#pragma unroll
      for (int e = 0; e < kPer; e += 2)
        *reinterpret_cast<__nv_bfloat162*>(dst + e) = __floats2bfloat162_rn(acc[e] * inv, acc[e + 1] * inv);
    } else {
      float* dst = static_cast<float*>(o) + row * D + lane * kPer;
#pragma unroll
      for (int e = 0; e < kPer; e += 2)
        *reinterpret_cast<float2*>(dst + e) = make_float2(acc[e] * inv, acc[e + 1] * inv);
    }
    if (lane == 0) lse[row] = denom > 0.f ? lmax + logf(denom) : -INFINITY;
  }
}

// Merges num_splits partials of `rows` = B*H*M rows into o (bf16 or fp32) and lse.
cudaError_t launch_splitkv_combine(const float* o_part, const float* l_part, void* o, float* lse,
                                   int64_t rows, int D, int num_splits, bool bf16,
                                   cudaStream_t stream) {
  int dev = 0, sms = 148;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const int threads = 256;  // 8 rows in flight per block
  const int64_t need = (rows + 7) / 8;
  const int blocks = static_cast<int>(need < 8LL * sms ? need : 8LL * sms);
  if (D == 64) {
    if (bf16)
      splitkv_combine_kernel<64, true><<<blocks, threads, 0, stream>>>(o_part, l_part, o, lse, rows, num_splits);
    else
      splitkv_combine_kernel<64, false><<<blocks, threads, 0, stream>>>(o_part, l_part, o, lse, rows, num_splits);
  } else {
    if (bf16)
      splitkv_combine_kernel<128, true><<<blocks, threads, 0, stream>>>(o_part, l_part, o, lse, rows, num_splits);
    else
      splitkv_combine_kernel<128, false><<<blocks, threads, 0, stream>>>(o_part, l_part, o, lse, rows, num_splits);
  }
  return cudaGetLastError();
}

}  // namespace fa2
