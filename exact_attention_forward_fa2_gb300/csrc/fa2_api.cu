// C ABI of the forward pass (declared in include/fa2.h): argument checks,
// TMA tensor-map encoding and dispatch to the (dtype, head dim) instantiation.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <climits>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "fa2.h"
#include "fa2_config.h"
#include "fa2_internal.h"
#include "fa2_bwd_kernel.cuh"
#include "fa2_fwd_kernel.cuh"

namespace fa2 {
cudaError_t launch_bwd(BwdLaunch& L, int D);
cudaError_t launch_bf16_d64(FwdLaunch& L);
cudaError_t launch_bf16_d128(FwdLaunch& L);
cudaError_t launch_fp32_d64(FwdLaunch& L);
cudaError_t launch_fp32_d128(FwdLaunch& L);
cudaError_t launch_splitkv_combine(const float* o_part, const float* l_part, void* o, float* lse,
                                   int64_t rows, int D, int num_splits, bool bf16,
                                   cudaStream_t stream);
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
// one 128-byte row segment x box_rows rows x 1 head, 128-byte swizzle.  Rows past
// `rows` are zero-filled on load and dropped on store, per head.
int encode_map(CUtensorMap* map, const void* ptr, int dtype, int D, int rows, int64_t bh,
               CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B, int box_rows = 128) {
  const int e = (dtype == FA2_BF16) ? 2 : 4;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(rows),
                              static_cast<cuuint64_t>(bh)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * e,
                                 static_cast<cuuint64_t>(rows) * D * e};
  const cuuint32_t box[3] = {static_cast<cuuint32_t>(128 / e), static_cast<cuuint32_t>(box_rows), 1u};
  const cuuint32_t estr[3] = {1u, 1u, 1u};
  const CUresult r = g_encode(
      map, dtype == FA2_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3,
      const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
      CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? FA2_OK : FA2_ERR_CUDA;
}

constexpr int kMaxSplits = 64;

// Key tiles of `bn` keys covering N keys.
int64_t kv_tiles_total(int N, int bn) { return (static_cast<int64_t>(N) + bn - 1) / bn; }

// Whether a unit pairs the single query tile of two heads that read the same
// key/value head (two tile slots per CTA, M <= 128, an even number of query
// heads per key/value head) instead of two query tiles of one head.
bool pair_heads(int H, int H_kv, int M, int qt) { return qt == 2 && M <= 128 && (H / H_kv) % 2 == 0; }

// Whether the query heads of each key/value head are computed as the rows of one
// problem with H_kv heads of (H / H_kv) * M rows.  Under grouped-query attention
// the heads of a group are contiguous in q, o and lse and read the same K and V,
// so without a causal mask or score modifiers that problem is the same attention
// computed on the same memory; with few query rows (decode) it fills 128-row
// tiles that would otherwise hold M rows each.
bool pack_heads(int H, int H_kv, int M, int causal, bool use_mod) {
  return !use_mod && !causal && H / H_kv >= 2 && M < 128;
}

// Query heads per group of the causal launch order.  When the keys and values of
// every head fit in half of L2 (kL2AllBytes) one group holds every head (the plain
// longest-first order); otherwise a group holds as many whole key/value heads
// (with their H / H_kv query heads) as fit in kL2GroupBytes, so that the CTAs in
// flight (one group, and the start of the next) read K and V from L2.  Measured:
// +0.8% on the 2 x 16 x 8192^2 x 128 causal workload (128 MiB of K/V, groups of
// 8 heads), -1.1% on 4 x 16 x 4096^2 x 64 causal (64 MiB) if grouped there too.
constexpr int64_t kL2AllBytes = int64_t(64) << 20;
constexpr int64_t kL2GroupBytes = int64_t(32) << 20;
int causal_head_group(int64_t bh, int group, int N, int D, int dtype) {
  const int64_t kv_head_bytes = 2 * static_cast<int64_t>(N) * D * (dtype == FA2_BF16 ? 2 : 4);
  if ((bh / group) * kv_head_bytes <= kL2AllBytes) return static_cast<int>(bh);
  const int64_t kv_heads = std::max<int64_t>(1, kL2GroupBytes / kv_head_bytes);
  return static_cast<int>(std::min<int64_t>(bh, kv_heads * group));
}

// CTAs of the forward before any key split.
int64_t forward_units(int B, int H, int H_kv, int M, int qt) {
  if (pair_heads(H, H_kv, M, qt)) return static_cast<int64_t>(B) * H / 2;
  return static_cast<int64_t>(B) * H * ((static_cast<int64_t>(M) + qt * 128 - 1) / (qt * 128));
}

// Split count that fills about one wave of CTAs when the query tiles alone do
// not: floor(#SMs / units), with at least 4 key tiles per split.
int auto_splits(int64_t units, int N, int bn, int sms) {
  if (units >= sms) return 1;
  int64_t s = sms / units;
  s = std::min<int64_t>(s, kv_tiles_total(N, bn) / 4);
  return static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(s, kMaxSplits)));
}

// Byte offset of the L partials inside the workspace (after the O partials).
size_t lpart_offset(int64_t rows, int D, int splits) {
  const size_t o_bytes = static_cast<size_t>(splits) * static_cast<size_t>(rows) * D * sizeof(float);
  return (o_bytes + 255) & ~static_cast<size_t>(255);
}

size_t workspace_bytes(int64_t rows, int D, int splits) {
  return lpart_offset(rows, D, splits) + static_cast<size_t>(splits) * rows * sizeof(float);
}

// Score modifiers of fa2_fwd_ext; the defaults leave the plain forward.
struct Modifiers {
  int window_left = -1;   // < 0: no left bound
  int window_right = -1;  // < 0: no right bound
  float softcap = 0.f;    // 0: no softcap
  const float* alibi = nullptr;
  int alibi_bstride = 0;
};

}  // namespace

int fa2::check_forward_args(const void* q, const void* k, const void* v, const void* o, const float* lse, int B,
                            int H, int H_kv, int M, int N, int D, float scale, int dtype) {
  if (!q || !k || !v || !o || !lse) return FA2_ERR_NULL;
  if (B <= 0 || H <= 0 || M <= 0 || N <= 0) return FA2_ERR_SHAPE;
  if (H_kv <= 0 || H % H_kv != 0) return FA2_ERR_SHAPE;
  if (D != 64 && D != 128) return FA2_ERR_HEADDIM;
  if (dtype != FA2_BF16 && dtype != FA2_FP32) return FA2_ERR_DTYPE;
  if (!(scale > 0.f) || !std::isfinite(scale)) return FA2_ERR_SCALE;
  const auto addr = [](const void* p) { return reinterpret_cast<uintptr_t>(p); };
  if ((addr(q) | addr(k) | addr(v) | addr(o)) & 15u) return FA2_ERR_ALIGN;
  if (addr(lse) & 3u) return FA2_ERR_ALIGN;
  return FA2_OK;
}

namespace {

// Shared by every entry point.  num_splits == 1: plain forward; > 1: split-KV
// partials into `workspace`, then the combine kernel.
int run_forward(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                int H_kv, int M, int N, int D, float scale, int causal, int dtype, int num_splits,
                void* workspace, size_t workspace_size, void* stream,
                const Modifiers& mods = Modifiers()) {
  const int arg_rc = fa2::check_forward_args(q, k, v, o, lse, B, H, H_kv, M, N, D, scale, dtype);
  if (arg_rc != FA2_OK) return arg_rc;
  const auto addr = [](const void* p) { return reinterpret_cast<uintptr_t>(p); };
  if (!(mods.softcap >= 0.f) || std::isinf(mods.softcap)) return FA2_ERR_MODIFIER;
  if (mods.alibi && mods.alibi_bstride != 0 && mods.alibi_bstride != H) return FA2_ERR_MODIFIER;
  if (addr(mods.alibi) & 3u) return FA2_ERR_ALIGN;
  // a causal right edge is the diagonal whatever window_right says
  const bool use_mod = mods.window_left >= 0 || (!causal && mods.window_right >= 0) ||
                       mods.softcap > 0.f || mods.alibi != nullptr;
  // the kernel forms row +- window and key - row in 32-bit ints and fp32
  if (use_mod && (M > (1 << 30) || N > (1 << 30))) return FA2_ERR_TOO_LARGE;
  // packed heads: the same memory seen as H_kv heads of (H / H_kv) * M rows
  if (pack_heads(H, H_kv, M, causal, use_mod)) {
    M = (H / H_kv) * M;
    H = H_kv;
  }
  const int64_t bh = static_cast<int64_t>(B) * H;
  const int64_t bh_kv = static_cast<int64_t>(B) * H_kv;
  // query tiles per CTA and keys per key/value tile of the kernel configuration that
  // will run: softcap, sliding window or plain (see fa2_config.h)
  const int cap_on = mods.softcap > 0.f ? 1 : 0;
  const int win_on = (mods.window_left >= 0 || (!causal && mods.window_right >= 0)) ? 1 : 0;
  const int qt = fa2::qtiles_for(dtype == FA2_FP32, D, cap_on, win_on);
  const int64_t units = forward_units(B, H, H_kv, M, qt);
  if (bh > INT_MAX || units > INT_MAX) return FA2_ERR_TOO_LARGE;
  const int bn = fa2::kv_tile_for(dtype == FA2_FP32, D, cap_on, win_on);
  const int64_t n_kv = kv_tiles_total(N, bn);
  int tiles_per_split = static_cast<int>(n_kv);
  if (num_splits > 1) {
    tiles_per_split = static_cast<int>((n_kv + num_splits - 1) / num_splits);
    num_splits = static_cast<int>((n_kv + tiles_per_split - 1) / tiles_per_split);
  }
  if (num_splits < 1) num_splits = 1;
  if (units * num_splits > INT_MAX) return FA2_ERR_TOO_LARGE;
  const int64_t rows = bh * M;
  if (num_splits > 1) {
    const auto wa = reinterpret_cast<uintptr_t>(workspace);
    if (!workspace || (wa & 255u) || workspace_size < workspace_bytes(rows, D, num_splits))
      return FA2_ERR_WORKSPACE;
  }

  DeviceState* st = nullptr;
  int rc = device_state(&st);
  if (rc != FA2_OK) return rc;

  fa2::FwdLaunch L;
  rc = encode_map(&L.tmQ, q, dtype, D, M, bh);
  if (rc == FA2_OK) rc = encode_map(&L.tmK, k, dtype, D, N, bh_kv, CU_TENSOR_MAP_SWIZZLE_128B, bn);
  // fp32 V is read MN-major as TF32: 32-byte-chunk swizzle (see the kernel header)
  if (rc == FA2_OK)
    rc = encode_map(&L.tmV, v, dtype, D, N, bh_kv,
                    dtype == FA2_BF16 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_128B_ATOM_32B, bn);
  if (rc == FA2_OK) rc = encode_map(&L.tmO, o, dtype, D, M, bh);
  if (rc != FA2_OK) return rc;
  L.params.lse = lse;
  L.params.status = st->status;
  L.params.M = M;
  L.params.N = N;
  L.params.BH = static_cast<int>(bh);
  L.params.H = H;
  L.params.group = H / H_kv;
  L.params.num_splits = num_splits;
  L.params.tiles_per_split = tiles_per_split;
  L.params.o_part = num_splits > 1 ? static_cast<float*>(workspace) : nullptr;
  L.params.l_part = num_splits > 1
                        ? reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                                   lpart_offset(rows, D, num_splits))
                        : nullptr;
  L.params.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  L.params.pair_heads = pair_heads(H, H_kv, M, qt) ? 1 : 0;
  L.params.head_group = causal_head_group(bh, H / H_kv, N, D, dtype);
  // window bounds: an absent side widens to cover every key (row - M <= 0 and
  // row + N >= N - 1 for every row); causal caps the right side at the diagonal
  L.params.win_left = (mods.window_left < 0 || mods.window_left > M) ? M : mods.window_left;
  L.params.win_right = (mods.window_right < 0 || mods.window_right > N) ? N : mods.window_right;
  if (causal) L.params.win_right = 0;
  L.params.cap_in = mods.softcap > 0.f ? static_cast<float>(static_cast<double>(scale) / mods.softcap) : 0.f;
  L.params.cap_out = static_cast<float>(static_cast<double>(mods.softcap) * 1.4426950408889634);
  L.params.alibi = mods.alibi;
  L.params.alibi_bstride = mods.alibi_bstride;
  L.causal = causal ? 1 : 0;
  L.win = win_on;
  L.mod = (mods.softcap > 0.f || mods.alibi != nullptr || L.win) ? 1 : 0;
  L.stream = static_cast<cudaStream_t>(stream);

  cudaError_t e;
  if (dtype == FA2_BF16)
    e = (D == 64) ? fa2::launch_bf16_d64(L) : fa2::launch_bf16_d128(L);
  else
    e = (D == 64) ? fa2::launch_fp32_d64(L) : fa2::launch_fp32_d128(L);
  if (e == cudaSuccess && num_splits > 1)
    e = fa2::launch_splitkv_combine(L.params.o_part, L.params.l_part, o, lse, rows, D, num_splits,
                                    dtype == FA2_BF16, L.stream);
  return e == cudaSuccess ? FA2_OK : FA2_ERR_CUDA;
}

// Key/value heads per group of the causal dK/dV order.  A group's CTAs run
// longest first and keep its Q, dO and dQ rows in L2; the groups are few (each
// at least kBwdGroupWaves full waves of CTAs), so the longest CTAs of the last
// group still start early enough not to stretch the end of the grid.
constexpr int64_t kBwdGroupWaves = 4;
int64_t bwd_head_group(int64_t bh_kv, int64_t n_ktiles) {
  int sms = 148, dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    sms = 148;
  const int64_t groups = std::max<int64_t>(1, bh_kv * n_ktiles / (kBwdGroupWaves * sms));
  return (bh_kv + groups - 1) / groups;
}

// Backward workspace: -L log2(e) and D = rowsum(dO o O), [B*H][M rounded up to
// 128] fp32 each, then the fp32 dQ accumulator of dQ by reduction, [B*H][Mpad][128].
constexpr int kBwdAccDim = 128;
size_t bwd_workspace_bytes(int64_t bh, int M) {
  const int64_t mpad = (static_cast<int64_t>(M) + 127) / 128 * 128;
  return (2 + kBwdAccDim) * static_cast<size_t>(bh * mpad) * sizeof(float);
}


// Streams and events of the host-buffer pipeline (fa2_fwd_host), created once
// per device; the whole enqueue sequence of one call holds the mutex.
constexpr int kHostMaxChunks = 32;
struct HostPipe {
  bool ready = false;
  cudaStream_t h2d = nullptr, d2h = nullptr;
  cudaEvent_t start = nullptr, out_done = nullptr;
  cudaEvent_t in[kHostMaxChunks] = {};
  cudaEvent_t done[kHostMaxChunks] = {};
};
std::mutex g_pipe_mu;
HostPipe g_pipe[kMaxDevices];

int host_pipe(int dev, HostPipe** out) {
  HostPipe& hp = g_pipe[dev];
  if (!hp.ready) {
    bool ok = cudaStreamCreateWithFlags(&hp.h2d, cudaStreamNonBlocking) == cudaSuccess &&
              cudaStreamCreateWithFlags(&hp.d2h, cudaStreamNonBlocking) == cudaSuccess &&
              cudaEventCreateWithFlags(&hp.start, cudaEventDisableTiming) == cudaSuccess &&
              cudaEventCreateWithFlags(&hp.out_done, cudaEventDisableTiming) == cudaSuccess;
    for (int c = 0; ok && c < kHostMaxChunks; ++c)
      ok = cudaEventCreateWithFlags(&hp.in[c], cudaEventDisableTiming) == cudaSuccess &&
           cudaEventCreateWithFlags(&hp.done[c], cudaEventDisableTiming) == cudaSuccess;
    if (!ok) return FA2_ERR_CUDA;
    hp.ready = true;
  }
  *out = &hp;
  return FA2_OK;
}

int sm_count(int* sms) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FA2_ERR_CUDA;
  if (cudaDeviceGetAttribute(sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return FA2_ERR_CUDA;
  return FA2_OK;
}

}  // namespace

extern "C" int fa2_fwd_gqa(const void* q, const void* k, const void* v, void* o, float* lse,
                           int B, int H, int H_kv, int M, int N, int D, float scale, int causal,
                           int dtype, void* stream) {
  return run_forward(q, k, v, o, lse, B, H, H_kv, M, N, D, scale, causal, dtype, 1, nullptr, 0,
                     stream);
}

extern "C" int fa2_splitkv_num_splits(int B, int H, int H_kv, int M, int N, int D, int dtype) {
  if (B <= 0 || H <= 0 || M <= 0 || N <= 0) return FA2_ERR_SHAPE;
  if (H_kv <= 0 || H % H_kv != 0) return FA2_ERR_SHAPE;
  if (D != 64 && D != 128) return FA2_ERR_HEADDIM;
  if (dtype != FA2_BF16 && dtype != FA2_FP32) return FA2_ERR_DTYPE;
  int sms = 0;
  const int rc = sm_count(&sms);
  if (rc != FA2_OK) return rc;
  const int qt = fa2::qtiles_for(dtype == FA2_FP32, D);
  // the CTAs of the forward as it will run (heads packed under the non-causal
  // rule; a causal problem, never packed, only gets more CTAs)
  if (pack_heads(H, H_kv, M, 0, false)) {
    M = (H / H_kv) * M;
    H = H_kv;
  }
  return auto_splits(forward_units(B, H, H_kv, M, qt), N, fa2::kv_tile_for(dtype == FA2_FP32, D), sms);
}

extern "C" size_t fa2_splitkv_workspace_bytes(int B, int H, int M, int D, int num_splits) {
  if (B <= 0 || H <= 0 || M <= 0 || (D != 64 && D != 128) || num_splits <= 1) return 0;
  return workspace_bytes(static_cast<int64_t>(B) * H * M, D, num_splits);
}

extern "C" int fa2_fwd_splitkv(const void* q, const void* k, const void* v, void* o, float* lse,
                               int B, int H, int H_kv, int M, int N, int D, float scale,
                               int causal, int dtype, int num_splits, void* workspace,
                               size_t workspace_size, void* stream) {
  if (num_splits <= 0) {
    num_splits = fa2_splitkv_num_splits(B, H, H_kv, M, N, D, dtype);
    if (num_splits < 0) return num_splits;
  }
  if (num_splits > kMaxSplits) num_splits = kMaxSplits;
  return run_forward(q, k, v, o, lse, B, H, H_kv, M, N, D, scale, causal, dtype, num_splits,
                     workspace, workspace_size, stream);
}

extern "C" int fa2_fwd_ext(const void* q, const void* k, const void* v, void* o, float* lse,
                           int B, int H, int H_kv, int M, int N, int D, float scale, int causal,
                           int window_left, int window_right, float softcap,
                           const float* alibi_slopes, int alibi_batch_stride, int dtype,
                           int num_splits, void* workspace, size_t workspace_size, void* stream) {
  if (num_splits <= 0) {
    num_splits = fa2_splitkv_num_splits(B, H, H_kv, M, N, D, dtype);
    if (num_splits < 0) return num_splits;
  }
  if (num_splits > kMaxSplits) num_splits = kMaxSplits;
  Modifiers mods;
  mods.window_left = window_left;
  mods.window_right = window_right;
  mods.softcap = softcap;
  mods.alibi = alibi_slopes;
  mods.alibi_bstride = alibi_batch_stride;
  return run_forward(q, k, v, o, lse, B, H, H_kv, M, N, D, scale, causal, dtype, num_splits,
                     workspace, workspace_size, stream, mods);
}

extern "C" int fa2_fwd_host(const void* q_host, const void* k_host, const void* v_host, void* o_host,
                            float* lse_host, void* q, void* k, void* v, void* o, float* lse, int B,
                            int H, int H_kv, int M, int N, int D, float scale, int causal, int dtype,
                            int chunks, void* stream) {
  if (!q_host || !k_host || !v_host || !o_host || !lse_host) return FA2_ERR_NULL;
  // every argument of the device-side call is checked once for the whole problem
  // (a call with num_splits = 1 that stops before any CUDA work on error)
  if (!q || !k || !v || !o || !lse) return FA2_ERR_NULL;
  if (B <= 0 || H <= 0 || M <= 0 || N <= 0 || H_kv <= 0 || H % H_kv != 0) return FA2_ERR_SHAPE;
  if (D != 64 && D != 128) return FA2_ERR_HEADDIM;
  if (dtype != FA2_BF16 && dtype != FA2_FP32) return FA2_ERR_DTYPE;
  if (!(scale > 0.f) || !std::isfinite(scale)) return FA2_ERR_SCALE;
  const auto addr = [](const void* p) { return reinterpret_cast<uintptr_t>(p); };
  if ((addr(q) | addr(k) | addr(v) | addr(o)) & 15u) return FA2_ERR_ALIGN;
  if (addr(lse) & 3u) return FA2_ERR_ALIGN;
  const int64_t bh = static_cast<int64_t>(B) * H;
  if (bh > INT_MAX) return FA2_ERR_TOO_LARGE;
  DeviceState* st = nullptr;
  int rc = device_state(&st);
  if (rc != FA2_OK) return rc;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FA2_ERR_CUDA;

  // chunk unit: one key/value head with the query heads that read it (flat
  // index b*H_kv + j; its query heads are the contiguous flat heads
  // [group*(b*H_kv + j), +group) of q, o and lse)
  const int group = H / H_kv;
  const int64_t kv_heads = static_cast<int64_t>(B) * H_kv;
  if (chunks <= 0) chunks = 4;
  chunks = static_cast<int>(std::min<int64_t>({static_cast<int64_t>(chunks), kv_heads, kHostMaxChunks}));
  const size_t e = dtype == FA2_BF16 ? 2 : 4;
  const size_t q_head = static_cast<size_t>(M) * D * e, kv_head = static_cast<size_t>(N) * D * e;
  const size_t l_head = static_cast<size_t>(M) * sizeof(float);
  const cudaStream_t s0 = static_cast<cudaStream_t>(stream);
  auto at = [](const void* p, size_t off) { return static_cast<const char*>(p) + off; };
  auto atw = [](void* p, size_t off) { return static_cast<char*>(p) + off; };

  std::lock_guard<std::mutex> lock(g_pipe_mu);
  HostPipe* hp = nullptr;
  rc = host_pipe(dev, &hp);
  if (rc != FA2_OK) return rc;
  bool ok = cudaEventRecord(hp->start, s0) == cudaSuccess &&  // after the caller's earlier work
            cudaStreamWaitEvent(hp->h2d, hp->start, 0) == cudaSuccess;
  for (int c = 0; ok && c < chunks; ++c) {
    const int64_t g0 = kv_heads * c / chunks, g1 = kv_heads * (c + 1) / chunks;
    const int64_t nq = (g1 - g0) * group, q0 = g0 * group;
    ok = cudaMemcpyAsync(atw(q, q0 * q_head), at(q_host, q0 * q_head), nq * q_head, cudaMemcpyHostToDevice,
                         hp->h2d) == cudaSuccess &&
         cudaMemcpyAsync(atw(k, g0 * kv_head), at(k_host, g0 * kv_head), (g1 - g0) * kv_head,
                         cudaMemcpyHostToDevice, hp->h2d) == cudaSuccess &&
         cudaMemcpyAsync(atw(v, g0 * kv_head), at(v_host, g0 * kv_head), (g1 - g0) * kv_head,
                         cudaMemcpyHostToDevice, hp->h2d) == cudaSuccess &&
         cudaEventRecord(hp->in[c], hp->h2d) == cudaSuccess &&
         cudaStreamWaitEvent(s0, hp->in[c], 0) == cudaSuccess;
    if (!ok) break;
    // these heads as a problem of their own: batch 1, nq query heads, g1 - g0 key/value heads
    rc = run_forward(at(q, q0 * q_head), at(k, g0 * kv_head), at(v, g0 * kv_head), atw(o, q0 * q_head),
                     lse + q0 * M, 1, static_cast<int>(nq), static_cast<int>(g1 - g0), M, N, D, scale, causal,
                     dtype, 1, nullptr, 0, s0);
    if (rc != FA2_OK) return rc;
    ok = cudaEventRecord(hp->done[c], s0) == cudaSuccess &&
         cudaStreamWaitEvent(hp->d2h, hp->done[c], 0) == cudaSuccess &&
         cudaMemcpyAsync(atw(o_host, q0 * q_head), at(o, q0 * q_head), nq * q_head, cudaMemcpyDeviceToHost,
                         hp->d2h) == cudaSuccess &&
         cudaMemcpyAsync(lse_host + q0 * M, lse + q0 * M, nq * l_head, cudaMemcpyDeviceToHost, hp->d2h) ==
             cudaSuccess;
  }
  // the caller's stream reaches its next work only after the last copy back
  ok = ok && cudaEventRecord(hp->out_done, hp->d2h) == cudaSuccess &&
       cudaStreamWaitEvent(s0, hp->out_done, 0) == cudaSuccess;
  return ok ? FA2_OK : FA2_ERR_CUDA;
}

extern "C" int fa2_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                       int H, int M, int N, int D, float scale, int causal, int dtype,
                       void* stream) {
  return fa2_fwd_gqa(q, k, v, o, lse, B, H, H, M, N, D, scale, causal, dtype, stream);
}

extern "C" size_t fa2_bwd_workspace_bytes(int B, int H, int M) {
  if (B <= 0 || H <= 0 || M <= 0) return 0;
  return bwd_workspace_bytes(static_cast<int64_t>(B) * H, M);
}

namespace {

int run_backward(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dout,
                 void* dq, void* dk, void* dv, int B, int H, int H_kv, int M, int N, int D, float scale,
                 int causal, int dtype, void* workspace, size_t workspace_size, void* stream, bool reduce_dq) {
  if (!q || !k || !v || !o || !lse || !dout || !dq || !dk || !dv) return FA2_ERR_NULL;
  if (B <= 0 || H <= 0 || M <= 0 || N <= 0) return FA2_ERR_SHAPE;
  if (H_kv <= 0 || H % H_kv != 0) return FA2_ERR_SHAPE;
  if (D != 64 && D != 128) return FA2_ERR_HEADDIM;
  if (dtype != FA2_BF16) return FA2_ERR_DTYPE;
  if (!(scale > 0.f) || !std::isfinite(scale)) return FA2_ERR_SCALE;
  const auto addr = [](const void* p) { return reinterpret_cast<uintptr_t>(p); };
  if ((addr(q) | addr(k) | addr(v) | addr(o) | addr(dout) | addr(dq) | addr(dk) | addr(dv)) & 15u)
    return FA2_ERR_ALIGN;
  if (addr(lse) & 3u) return FA2_ERR_ALIGN;
  const int64_t bh = static_cast<int64_t>(B) * H;
  const int64_t bh_kv = static_cast<int64_t>(B) * H_kv;
  const int64_t n_ktiles = (static_cast<int64_t>(N) + 127) / 128;
  const int64_t n_qtiles = (static_cast<int64_t>(M) + 127) / 128;
  if (M > (1 << 30) || N > (1 << 30) || bh * n_qtiles > INT_MAX || bh_kv * n_ktiles > INT_MAX)
    return FA2_ERR_TOO_LARGE;
  const size_t ws_need = bwd_workspace_bytes(bh, M);
  if (!workspace || (addr(workspace) & 255u) || workspace_size < ws_need) return FA2_ERR_WORKSPACE;

  DeviceState* st = nullptr;
  int rc = device_state(&st);
  if (rc != FA2_OK) return rc;
  fa2::BwdLaunch L;
  rc = encode_map(&L.tmQ64, q, dtype, D, M, bh, CU_TENSOR_MAP_SWIZZLE_128B, 64);
  if (rc == FA2_OK) rc = encode_map(&L.tmdO64, dout, dtype, D, M, bh, CU_TENSOR_MAP_SWIZZLE_128B, 64);
  if (rc == FA2_OK) rc = encode_map(&L.tmK128, k, dtype, D, N, bh_kv);
  if (rc == FA2_OK) rc = encode_map(&L.tmV128, v, dtype, D, N, bh_kv);
  if (rc == FA2_OK) rc = encode_map(&L.tmdK, dk, dtype, D, N, bh_kv);
  if (rc == FA2_OK) rc = encode_map(&L.tmdV, dv, dtype, D, N, bh_kv);
  if (rc == FA2_OK) rc = encode_map(&L.tmQ128, q, dtype, D, M, bh);
  if (rc == FA2_OK) rc = encode_map(&L.tmdO128, dout, dtype, D, M, bh);
  if (rc == FA2_OK) rc = encode_map(&L.tmK64, k, dtype, D, N, bh_kv, CU_TENSOR_MAP_SWIZZLE_128B, 64);
  if (rc == FA2_OK) rc = encode_map(&L.tmV64, v, dtype, D, N, bh_kv, CU_TENSOR_MAP_SWIZZLE_128B, 64);
  if (rc == FA2_OK) rc = encode_map(&L.tmdQ, dq, dtype, D, M, bh);
  if (rc != FA2_OK) return rc;
  const int64_t mpad = n_qtiles * 128;
  L.nl2 = static_cast<float*>(workspace);
  L.dlt = L.nl2 + bh * mpad;
  L.dqacc = (reduce_dq && D == kBwdAccDim) ? L.dlt + bh * mpad : nullptr;
  L.dq = dq;
  L.params.nl2 = L.nl2;
  L.params.dlt = L.dlt;
  L.params.dqacc = L.dqacc;
  L.params.head_group = static_cast<int>(bwd_head_group(bh_kv, n_ktiles));
  L.params.status = st->status;
  L.params.M = M;
  L.params.N = N;
  L.params.Mpad = static_cast<int>(mpad);
  L.params.H = H;
  L.params.group = H / H_kv;
  L.params.BH = static_cast<int>(bh);
  L.params.BHkv = static_cast<int>(bh_kv);
  L.params.n_ktiles = static_cast<int>(n_ktiles);
  L.params.n_qtiles = static_cast<int>(n_qtiles);
  L.params.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  L.params.scale = scale;
  L.o = o;
  L.dout = dout;
  L.lse = lse;
  L.causal = causal ? 1 : 0;
  L.stream = static_cast<cudaStream_t>(stream);
  return fa2::launch_bwd(L, D) == cudaSuccess ? FA2_OK : FA2_ERR_CUDA;
}

}  // namespace

extern "C" int fa2_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
                       const void* dout, void* dq, void* dk, void* dv, int B, int H, int H_kv, int M,
                       int N, int D, float scale, int causal, int dtype, void* workspace,
                       size_t workspace_size, void* stream) {
  return run_backward(q, k, v, o, lse, dout, dq, dk, dv, B, H, H_kv, M, N, D, scale, causal, dtype, workspace,
                      workspace_size, stream, true);
}

extern "C" int fa2_bwd_deterministic(const void* q, const void* k, const void* v, const void* o,
                                     const float* lse, const void* dout, void* dq, void* dk, void* dv, int B,
                                     int H, int H_kv, int M, int N, int D, float scale, int causal, int dtype,
                                     void* workspace, size_t workspace_size, void* stream) {
  return run_backward(q, k, v, o, lse, dout, dq, dk, dv, B, H, H_kv, M, N, D, scale, causal, dtype, workspace,
                      workspace_size, stream, false);
}

extern "C" int fa2_bwd_host(const void* q_host, const void* k_host, const void* v_host, const void* o_host,
                            const float* lse_host, const void* dout_host, void* dq_host, void* dk_host,
                            void* dv_host, void* q, void* k, void* v, void* o, float* lse, void* dout, void* dq,
                            void* dk, void* dv, int B, int H, int H_kv, int M, int N, int D, float scale,
                            int causal, int dtype, void* workspace, size_t workspace_size, int chunks,
                            void* stream) {
  if (!q_host || !k_host || !v_host || !o_host || !lse_host || !dout_host || !dq_host || !dk_host || !dv_host)
    return FA2_ERR_NULL;
  if (!q || !k || !v || !o || !lse || !dout || !dq || !dk || !dv) return FA2_ERR_NULL;
  if (B <= 0 || H <= 0 || M <= 0 || N <= 0 || H_kv <= 0 || H % H_kv != 0) return FA2_ERR_SHAPE;
  if (D != 64 && D != 128) return FA2_ERR_HEADDIM;
  if (dtype != FA2_BF16) return FA2_ERR_DTYPE;
  if (!(scale > 0.f) || !std::isfinite(scale)) return FA2_ERR_SCALE;
  const auto addr = [](const void* p) { return reinterpret_cast<uintptr_t>(p); };
  if ((addr(q) | addr(k) | addr(v) | addr(o) | addr(dout) | addr(dq) | addr(dk) | addr(dv)) & 15u)
    return FA2_ERR_ALIGN;
  if (addr(lse) & 3u) return FA2_ERR_ALIGN;
  const int64_t bh = static_cast<int64_t>(B) * H;
  if (bh > INT_MAX) return FA2_ERR_TOO_LARGE;
  // the whole problem's workspace serves every slice (a slice has fewer heads)
  if (!workspace || (addr(workspace) & 255u) || workspace_size < bwd_workspace_bytes(bh, M))
    return FA2_ERR_WORKSPACE;
  DeviceState* st = nullptr;
  int rc = device_state(&st);
  if (rc != FA2_OK) return rc;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FA2_ERR_CUDA;

  // slices of whole key/value heads with the query heads that read them, as in
  // fa2_fwd_host: copies in on one library stream, the backward on the caller's
  // stream, copies out on the other library stream
  const int group = H / H_kv;
  const int64_t kv_heads = static_cast<int64_t>(B) * H_kv;
  if (chunks <= 0) {
    // 8 slices while each still holds 1.5 waves of dK/dV CTAs (measured: +6-8%
    // end to end on the 2x16x8192x8192x128 backward), else 4 (fewer CTAs per
    // slice leave SMs idle: -38% at 8 slices on 2x32x8192x8192x128 grouped-query)
    int sms = 148;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) sms = 148;
    const int64_t ctas = kv_heads * ((static_cast<int64_t>(N) + 127) / 128);
    chunks = (2 * ctas >= 3 * 8 * static_cast<int64_t>(sms)) ? 8 : 4;
  }
  chunks = static_cast<int>(std::min<int64_t>({static_cast<int64_t>(chunks), kv_heads, kHostMaxChunks}));
  const size_t q_head = static_cast<size_t>(M) * D * 2, kv_head = static_cast<size_t>(N) * D * 2;
  const size_t l_head = static_cast<size_t>(M) * sizeof(float);
  const cudaStream_t s0 = static_cast<cudaStream_t>(stream);
  auto at = [](const void* p, size_t off) { return static_cast<const char*>(p) + off; };
  auto atw = [](void* p, size_t off) { return static_cast<char*>(p) + off; };

  std::lock_guard<std::mutex> lock(g_pipe_mu);
  HostPipe* hp = nullptr;
  rc = host_pipe(dev, &hp);
  if (rc != FA2_OK) return rc;
  bool ok = cudaEventRecord(hp->start, s0) == cudaSuccess && cudaStreamWaitEvent(hp->h2d, hp->start, 0) == cudaSuccess;
  for (int c = 0; ok && c < chunks; ++c) {
    const int64_t g0 = kv_heads * c / chunks, g1 = kv_heads * (c + 1) / chunks;
    const int64_t nq = (g1 - g0) * group, q0 = g0 * group;
    const size_t qo = q0 * q_head, ko = g0 * kv_head;
    ok = cudaMemcpyAsync(atw(q, qo), at(q_host, qo), nq * q_head, cudaMemcpyHostToDevice, hp->h2d) == cudaSuccess &&
         cudaMemcpyAsync(atw(k, ko), at(k_host, ko), (g1 - g0) * kv_head, cudaMemcpyHostToDevice, hp->h2d) ==
             cudaSuccess &&
         cudaMemcpyAsync(atw(v, ko), at(v_host, ko), (g1 - g0) * kv_head, cudaMemcpyHostToDevice, hp->h2d) ==
             cudaSuccess &&
         cudaMemcpyAsync(atw(o, qo), at(o_host, qo), nq * q_head, cudaMemcpyHostToDevice, hp->h2d) == cudaSuccess &&
         cudaMemcpyAsync(lse + q0 * M, lse_host + q0 * M, nq * l_head, cudaMemcpyHostToDevice, hp->h2d) ==
             cudaSuccess &&
         cudaMemcpyAsync(atw(dout, qo), at(dout_host, qo), nq * q_head, cudaMemcpyHostToDevice, hp->h2d) ==
             cudaSuccess &&
         cudaEventRecord(hp->in[c], hp->h2d) == cudaSuccess && cudaStreamWaitEvent(s0, hp->in[c], 0) == cudaSuccess;
    if (!ok) break;
    // these heads as a problem of their own: batch 1, nq query heads, g1 - g0 key/value heads
    rc = fa2_bwd(at(q, qo), at(k, ko), at(v, ko), at(o, qo), lse + q0 * M, at(dout, qo), atw(dq, qo), atw(dk, ko),
                 atw(dv, ko), 1, static_cast<int>(nq), static_cast<int>(g1 - g0), M, N, D, scale, causal, dtype,
                 workspace, workspace_size, s0);
    if (rc != FA2_OK) return rc;
    ok = cudaEventRecord(hp->done[c], s0) == cudaSuccess && cudaStreamWaitEvent(hp->d2h, hp->done[c], 0) == cudaSuccess &&
         cudaMemcpyAsync(atw(dq_host, qo), at(dq, qo), nq * q_head, cudaMemcpyDeviceToHost, hp->d2h) == cudaSuccess &&
         cudaMemcpyAsync(atw(dk_host, ko), at(dk, ko), (g1 - g0) * kv_head, cudaMemcpyDeviceToHost, hp->d2h) ==
             cudaSuccess &&
         cudaMemcpyAsync(atw(dv_host, ko), at(dv, ko), (g1 - g0) * kv_head, cudaMemcpyDeviceToHost, hp->d2h) ==
             cudaSuccess;
  }
  // the caller's stream reaches its next work only after the last copy back
  ok = ok && cudaEventRecord(hp->out_done, hp->d2h) == cudaSuccess &&
       cudaStreamWaitEvent(s0, hp->out_done, 0) == cudaSuccess;
  return ok ? FA2_OK : FA2_ERR_CUDA;
}

extern "C" const char* fa2_strerror(int status) {
  switch (status) {
    case FA2_OK: return "ok";
    case FA2_ERR_NULL: return "a required pointer is NULL";
    case FA2_ERR_SHAPE: return "B, H, M, N and H_kv must be positive and H_kv must divide H";
    case FA2_ERR_HEADDIM: return "head dimension D must be 64 or 128";
    case FA2_ERR_DTYPE: return "dtype must be FA2_BF16 or FA2_FP32 (FA2_BF16 for the backward)";
    case FA2_ERR_ALIGN: return "q, k, v, o must be 16-byte aligned and lse 4-byte aligned";
    case FA2_ERR_SCALE: return "scale must be finite and positive";
    case FA2_ERR_TOO_LARGE: return "sizes exceed the grid or tensor-map limits";
    case FA2_ERR_ARCH: return "the current device is not compute capability 10.3 (sm_103)";
    case FA2_ERR_CUDA: return "a CUDA runtime or driver call failed";
    case FA2_ERR_DEVICE_TIMEOUT: return "a kernel pipeline wait ran out of time";
    case FA2_ERR_WORKSPACE: return "workspace missing, not 256-byte aligned or too small";
    case FA2_ERR_MODIFIER: return "softcap must be finite and >= 0, alibi_batch_stride 0 or H";
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

// Self-test of the failure path: one thread waits, through the kernels' own
// bounded wait, on an mbarrier phase that nothing completes, gives up after
// limit_ns and records kStatusSelfTest in the device status word, exactly as a
// pipeline wait of a real kernel that ran out would.
__global__ void fa2_selftest_wait_kernel(int* status, uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ uint32_t abort_flag;
  if (threadIdx.x == 0) {
    abort_flag = 0u;
    fa2::ptx::mbar_init(fa2::ptx::smem_u32(&bar), 1);
    fa2::ptx::fence_mbar_init();
    const fa2::WaitCtx w{&abort_flag, status};
    (void)fa2::wait_bounded(fa2::ptx::smem_u32(&bar), 0, w, fa2::kStatusSelfTest, limit_ns);
  }
}

extern "C" int fa2_selftest_wait_timeout(int limit_ms, void* stream) {
  if (limit_ms < 1 || limit_ms > 2000) return FA2_ERR_SHAPE;
  DeviceState* st = nullptr;
  const int rc = device_state(&st);
  if (rc != FA2_OK) return rc;
  fa2_selftest_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
      st->status, static_cast<uint64_t>(limit_ms) * 1000000ull);
  return cudaGetLastError() == cudaSuccess ? FA2_OK : FA2_ERR_CUDA;
}

extern "C" int fa2_version(void) { return 200; }
