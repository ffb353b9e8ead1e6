// Split-KV forward for callers that cannot allocate device memory.
//
// Some callers have no way to obtain scratch memory on the device: code running
// under an allocator that is already exhausted or locked down, plugins whose host
// framework owns every allocation, or a caller that must not call cudaMalloc or
// cudaFree because they synchronise the device and would stall other work.
// fa2_fwd_splitkv_noalloc serves them: the split-KV partial results go to a
// fixed buffer that lives in the library itself (a file-scope __device__ array,
// created when the library's device code is loaded on a GPU and held by every
// such GPU until the process exits).  Nothing is allocated per call.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "fa2.h"
#include "fa2_internal.h"

namespace {

// Capacity of the built-in split-KV scratch: 32 MiB per device.
constexpr size_t kScratchBytes = size_t(32) << 20;

static __device__ __align__(256) unsigned char g_splitkv_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of this device's copy of the scratch array.  In host code the
// array's name is only a stand-in for the symbol; the address must be asked for,
// once per device, with that device current.  It stays valid for the life of the
// device's primary context: a cudaDeviceReset ends that context, and with it the
// address cached here (and every other per-device state the library keeps).
int scratch_for_current_device(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FA2_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_splitkv_scratch) != cudaSuccess || p == nullptr)
      return FA2_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return FA2_OK;
}

}  // namespace

extern "C" int fa2_fwd_splitkv_noalloc(const void* q, const void* k, const void* v, void* o,
                                       float* lse, int B, int H, int H_kv, int M, int N, int D,
                                       float scale, int causal, int dtype, int num_splits,
                                       void* stream) {
  // the same argument checks as every forward entry, before any CUDA call
  int rc = fa2::check_forward_args(q, k, v, o, lse, B, H, H_kv, M, N, D, scale, dtype);
  if (rc != FA2_OK) return rc;
  void* scratch = nullptr;
  rc = scratch_for_current_device(&scratch);
  if (rc != FA2_OK) return rc;
  // fa2_fwd_splitkv lowers num_splits first (auto choice, the 64-slice cap, no
  // empty slice) and then refuses, with FA2_ERR_WORKSPACE, a split whose partials
  // need more than the buffer holds: exactly the calls that do not fit.  Every
  // slice writes each of its partial rows before the combine kernel reads it, so
  // nothing left in the buffer by an earlier call needs clearing.
  return fa2_fwd_splitkv(q, k, v, o, lse, B, H, H_kv, M, N, D, scale, causal, dtype, num_splits,
                         scratch, kScratchBytes, stream);
}
