// Throughput probe of the special-function pipe's base-2 exponential (MUFU ex2),
// the instruction the softmax of both passes spends most of its issue time in.
// Measurement only: the caller times the launch and divides the exponentials it
// ran (blocks * 256 threads * 8 chains * iters) by the time.
#include <cuda_runtime.h>

#include "fa2.h"
#include "sm103_ptx.cuh"

namespace {

constexpr int kProbeThreads = 256;
constexpr int kProbeChains = 8;  // independent dependency chains per thread

// Each chain iterates a <- 2^a - 1.25, which maps (-1, 0) into (-0.75, -0.25):
// the values stay finite and normal, and every step is one ex2 and one add.
__global__ void __launch_bounds__(kProbeThreads) fa2_probe_ex2_kernel(float* out, int iters) {
  float a[kProbeChains];
#pragma unroll
  for (int i = 0; i < kProbeChains; ++i)
    a[i] = -1.0e-2f * static_cast<float>((static_cast<int>(threadIdx.x) + i) % 64 + 1);
  for (int it = 0; it < iters; ++it) {
#pragma unroll
    for (int i = 0; i < kProbeChains; ++i) a[i] = fa2::ptx::ex2_approx(a[i]) - 1.25f;
  }
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < kProbeChains; ++i) s += a[i];
  out[static_cast<size_t>(blockIdx.x) * kProbeThreads + threadIdx.x] = s;
}

}  // namespace

extern "C" int fa2_probe_ex2(float* out, int blocks, int iters, void* stream) {
  if (out == nullptr) return FA2_ERR_NULL;
  if (blocks < 1 || blocks > 65536 || iters < 1 || iters > (1 << 20)) return FA2_ERR_SHAPE;
  if ((reinterpret_cast<uintptr_t>(out) & 3u) != 0u) return FA2_ERR_ALIGN;
  int dev = 0, major = 0, minor = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return FA2_ERR_CUDA;
  if (major != 10 || minor != 3) return FA2_ERR_ARCH;
  fa2_probe_ex2_kernel<<<blocks, kProbeThreads, 0, static_cast<cudaStream_t>(stream)>>>(out, iters);
  return cudaGetLastError() == cudaSuccess ? FA2_OK : FA2_ERR_CUDA;
}
