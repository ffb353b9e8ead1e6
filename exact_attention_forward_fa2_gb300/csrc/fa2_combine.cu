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
// (one 16-byte load per split for D = 128), rows spread over a grid sized to the
// SM count.  The loads are issued ahead of their use, so a row costs a few memory
// round trips instead of two per split: lane s loads L_s (splits in chunks of
// 32) and the lanes reduce their maximum; the O_s loads go out in groups of
// four splits, the first group together with the L_s loads, and the weights
// exp(L_s - max) reach every lane by shuffles.
// The sums still run over the splits in order.  At most 64 registers a thread
// (four blocks, 32 warps, per SM): the rows of a launch then run in one wave.
#include <cuda_runtime.h>
#include <cuda_bf16.h>

#include <cstdint>

namespace fa2 {

template <int D>
struct CombineVec;
template <>
struct CombineVec<64> {
  using T = float2;
  __device__ static void fma(float* acc, float w, const T& x) {
    acc[0] = fmaf(w, x.x, acc[0]);
    acc[1] = fmaf(w, x.y, acc[1]);
  }
};
template <>
struct CombineVec<128> {
  using T = float4;
  __device__ static void fma(float* acc, float w, const T& x) {
    acc[0] = fmaf(w, x.x, acc[0]);
    acc[1] = fmaf(w, x.y, acc[1]);
    acc[2] = fmaf(w, x.z, acc[2]);
    acc[3] = fmaf(w, x.w, acc[3]);
  }
};

constexpr int kCombineMaxSplits = 64;  // two chunks of 32 lanes
constexpr int kCombineGroup = 4;       // O_s loads in flight per lane

template <int D, bool kBF16>
__global__ void __launch_bounds__(256, 4) splitkv_combine_kernel(const float* __restrict__ o_part,
                                                              const float* __restrict__ l_part,
                                                              void* __restrict__ o,
                                                              float* __restrict__ lse, int64_t rows,
                                                              int num_splits) {
  constexpr int kPer = D / 32;  // columns per lane
  using V = CombineVec<D>;
  const int lane = static_cast<int>(threadIdx.x) % 32;
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x / 32);
  for (int64_t row = static_cast<int64_t>(blockIdx.x) * (blockDim.x / 32) + threadIdx.x / 32;
       row < rows; row += warps) {
    // L_s of split s sits in lane s % 32 of chunk s / 32; the first group's O_s
    // loads go out with them (a weight of 0 later leaves a loaded O_s unused)
    const float l_lo = lane < num_splits ? l_part[lane * rows + row] : -INFINITY;
    const float l_hi = 32 + lane < num_splits ? l_part[(32 + lane) * rows + row] : -INFINITY;
    typename V::T x[kCombineGroup];
#pragma unroll
    for (int u = 0; u < kCombineGroup; ++u)
      if (u < num_splits) x[u] = *reinterpret_cast<const typename V::T*>(o_part + (u * rows + row) * D + lane * kPer);
    float lmax = fmaxf(l_lo, l_hi);
#pragma unroll
    for (int sh = 16; sh > 0; sh >>= 1) lmax = fmaxf(lmax, __shfl_xor_sync(0xffffffffu, lmax, sh));
    float acc[kPer];
#pragma unroll
    for (int e = 0; e < kPer; ++e) acc[e] = 0.f;
    float denom = 0.f;
    if (lmax != -INFINITY) {
      // a split without visible keys (L_s = -inf) has weight 0 and adds nothing
      const float w_lo = l_lo == -INFINITY ? 0.f : expf(l_lo - lmax);
      const float w_hi = l_hi == -INFINITY ? 0.f : expf(l_hi - lmax);
      for (int s0 = 0; s0 < num_splits; s0 += kCombineGroup) {
        if (s0 > 0) {
#pragma unroll
          for (int u = 0; u < kCombineGroup; ++u) {
            const int s = s0 + u;
            if (s < num_splits)
              x[u] = *reinterpret_cast<const typename V::T*>(o_part + (s * rows + row) * D + lane * kPer);
          }
        }
#pragma unroll
        for (int u = 0; u < kCombineGroup; ++u) {
          const int s = s0 + u;
          const float w = __shfl_sync(0xffffffffu, s < 32 ? w_lo : w_hi, s & 31);
          if (s < num_splits && w > 0.f) {
            denom += w;
            V::fma(acc, w, x[u]);
          }
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
  if (num_splits < 1 || num_splits > kCombineMaxSplits) return cudaErrorInvalidValue;
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
