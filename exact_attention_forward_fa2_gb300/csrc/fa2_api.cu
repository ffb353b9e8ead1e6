// C ABI of the forward pass (declared in include/fa2.h): argument checks,
// TMA tensor-map encoding and dispatch to the (dtype, head dim) instantiation.
#include <cuda.h>
#include <cuda_runtime.h>

#include <climits>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "fa2.h"
#include "fa2_config.h"
#include "fa2_fwd_kernel.cuh"

namespace fa2 {
cudaError_t launch_bf16_d64(FwdLaunch& L);
cudaError_t launch_bf16_d128(FwdLaunch& L);
cudaError_t launch_fp32_d64(FwdLaunch& L);
cudaError_t launch_fp32_d128(FwdLaunch& L);
}  // namespace fa2

// Sticky device status word; kernels receive its address and record the first
// wait that ran out.
__device__ int g_fa2_status;

namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

constexpr int kMaxDevices = 64;

struct DeviceState {
  bool checked = false;
  bool arch_ok = false;
  int* status = nullptr;  // device address of g_fa2_status
};

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];
EncodeTiledFn g_encode = nullptr;

int device_state(DeviceState** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FA2_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState& st = g_dev[dev];
  if (!st.checked) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return FA2_ERR_CUDA;
    st.arch_ok = (major == 10 && minor == 3);
    if (st.arch_ok) {
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g_fa2_status) != cudaSuccess) return FA2_ERR_CUDA;
      st.status = static_cast<int*>(p);
    }
    if (g_encode == nullptr) {
      void* fn = nullptr;
      cudaDriverEntryPointQueryResult qres;
      if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                           &qres) != cudaSuccess ||
          qres != cudaDriverEntryPointSuccess || fn == nullptr)
        return FA2_ERR_CUDA;
      g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    }
    st.checked = true;
  }
  if (!st.arch_ok) return FA2_ERR_ARCH;
  *out = &st;
  return FA2_OK;
}

// 3-D map over a [BH, rows, D] tensor: dims (D, rows, BH) innermost first, box of
// one 128-byte row segment x 128 rows x 1 head, 128-byte swizzle.  Rows past
// `rows` are zero-filled on load and dropped on store, per head.
int encode_map(CUtensorMap* map, const void* ptr, int dtype, int D, int rows, int64_t bh,
               CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B) {
  const int e = (dtype == FA2_BF16) ? 2 : 4;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(rows),
                              static_cast<cuuint64_t>(bh)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * e,
                                 static_cast<cuuint64_t>(rows) * D * e};
  const cuuint32_t box[3] = {static_cast<cuuint32_t>(128 / e), 128u, 1u};
  const cuuint32_t estr[3] = {1u, 1u, 1u};
  const CUresult r = g_encode(
      map, dtype == FA2_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3,
      const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
      CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? FA2_OK : FA2_ERR_CUDA;
}

}  // namespace

extern "C" int fa2_fwd_gqa(const void* q, const void* k, const void* v, void* o, float* lse,
                           int B, int H, int H_kv, int M, int N, int D, float scale, int causal,
                           int dtype, void* stream) {
  if (!q || !k || !v || !o || !lse) return FA2_ERR_NULL;
  if (B <= 0 || H <= 0 || M <= 0 || N <= 0) return FA2_ERR_SHAPE;
  if (H_kv <= 0 || H % H_kv != 0) return FA2_ERR_SHAPE;
  if (D != 64 && D != 128) return FA2_ERR_HEADDIM;
  if (dtype != FA2_BF16 && dtype != FA2_FP32) return FA2_ERR_DTYPE;
  if (!(scale > 0.f) || !std::isfinite(scale)) return FA2_ERR_SCALE;
  const auto addr = [](const void* p) { return reinterpret_cast<uintptr_t>(p); };
  if ((addr(q) | addr(k) | addr(v) | addr(o)) & 15u) return FA2_ERR_ALIGN;
  if (addr(lse) & 3u) return FA2_ERR_ALIGN;
  const int64_t bh = static_cast<int64_t>(B) * H;
  const int64_t bh_kv = static_cast<int64_t>(B) * H_kv;
  const int qt = fa2::qtiles_for(dtype == FA2_FP32, D);
  const int64_t units = bh * ((static_cast<int64_t>(M) + qt * 128 - 1) / (qt * 128));
  if (bh > INT_MAX || units > INT_MAX) return FA2_ERR_TOO_LARGE;

  DeviceState* st = nullptr;
  int rc = device_state(&st);
  if (rc != FA2_OK) return rc;

  fa2::FwdLaunch L;
  rc = encode_map(&L.tmQ, q, dtype, D, M, bh);
  if (rc == FA2_OK) rc = encode_map(&L.tmK, k, dtype, D, N, bh_kv);
  // fp32 V is read MN-major as TF32: 32-byte-chunk swizzle (see the kernel header)
  if (rc == FA2_OK)
    rc = encode_map(&L.tmV, v, dtype, D, N, bh_kv,
                    dtype == FA2_BF16 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_128B_ATOM_32B);
  if (rc == FA2_OK) rc = encode_map(&L.tmO, o, dtype, D, M, bh);
  if (rc != FA2_OK) return rc;
  L.params.lse = lse;
  L.params.status = st->status;
  L.params.M = M;
  L.params.N = N;
  L.params.BH = static_cast<int>(bh);
  L.params.H = H;
  L.params.group = H / H_kv;
  L.params.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  L.causal = causal ? 1 : 0;
  L.stream = static_cast<cudaStream_t>(stream);

  cudaError_t e;
  if (dtype == FA2_BF16)
    e = (D == 64) ? fa2::launch_bf16_d64(L) : fa2::launch_bf16_d128(L);
  else
    e = (D == 64) ? fa2::launch_fp32_d64(L) : fa2::launch_fp32_d128(L);
  return e == cudaSuccess ? FA2_OK : FA2_ERR_CUDA;
}

extern "C" int fa2_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                       int H, int M, int N, int D, float scale, int causal, int dtype,
                       void* stream) {
  return fa2_fwd_gqa(q, k, v, o, lse, B, H, H, M, N, D, scale, causal, dtype, stream);
}

extern "C" const char* fa2_strerror(int status) {
  switch (status) {
    case FA2_OK: return "ok";
    case FA2_ERR_NULL: return "a required pointer is NULL";
    case FA2_ERR_SHAPE: return "B, H, M, N and H_kv must be positive and H_kv must divide H";
    case FA2_ERR_HEADDIM: return "head dimension D must be 64 or 128";
    case FA2_ERR_DTYPE: return "dtype must be FA2_BF16 or FA2_FP32";
    case FA2_ERR_ALIGN: return "q, k, v, o must be 16-byte aligned and lse 4-byte aligned";
    case FA2_ERR_SCALE: return "scale must be finite and positive";
    case FA2_ERR_TOO_LARGE: return "sizes exceed the grid or tensor-map limits";
    case FA2_ERR_ARCH: return "the current device is not compute capability 10.3 (sm_103)";
    case FA2_ERR_CUDA: return "a CUDA runtime or driver call failed";
    case FA2_ERR_DEVICE_TIMEOUT: return "a kernel pipeline wait ran out of time";
    default: return "unknown status";
  }
}

extern "C" int fa2_device_status(int reset, int* raw_code) {
  DeviceState* st = nullptr;
  int rc = device_state(&st);
  if (rc != FA2_OK) return rc;
  if (cudaDeviceSynchronize() != cudaSuccess) return FA2_ERR_CUDA;
  int word = 0;
  if (cudaMemcpyFromSymbol(&word, g_fa2_status, sizeof(int)) != cudaSuccess) return FA2_ERR_CUDA;
  if (raw_code) *raw_code = word;
  if (reset && word != 0) {
    const int zero = 0;
    if (cudaMemcpyToSymbol(g_fa2_status, &zero, sizeof(int)) != cudaSuccess) return FA2_ERR_CUDA;
  }
  return word == 0 ? FA2_OK : FA2_ERR_DEVICE_TIMEOUT;
}

extern "C" int fa2_version(void) { return 100; }
