// FlashAttention-2 backward kernels for sm_103a (GB300), bf16 inputs.
//
// What they compute ("From FlashAttention to FlashAttention 2", Backward Pass:
// Recomputation and Layer 7: The Backward Kernel; "FlashAttention-2 from PyTorch
// to Triton", Known gaps item 5): for upstream gradient dO, with the forward's
// stored logsumexp L and output O,
//   P_ij  = exp(scale q_i.k_j - L_i)           (recomputed tile by tile, 0 if hidden)
//   D_i   = rowsum(dO_i o O_i)
//   dS_ij = P_ij (dO_i.v_j - D_i)
//   dV_j  = sum_i P_ij dO_i,   dK_j = scale sum_i dS_ij q_i,   dQ_i = scale sum_j dS_ij k_j
// The N x N matrices P and dS exist only tile by tile, in TMEM.
//
// The pages give dQ two ways, "by atomics or by a second pass"; both are here.
//
// dQ by a second pass (bitwise reproducible), three launches:
//   bwd_preprocess    D_i and -L_i log2(e) per query row into a padded workspace
//                     (rows past M get D = 0 and -L log2(e) = -inf, so their P is 0)
//   bwd_dkdv_kernel   one CTA per (batch, key/value head, 128-key tile): the pages'
//                     K/V-outer loop.  It streams 64-row tiles of Q and dO (over
//                     every query head of the group) and accumulates dV and dK
//                     in TMEM with four tcgen05 GEMMs per step:
//                       S^T = K Q^T, dP^T = V dO^T   (keys on TMEM lanes)
//                       dV += P^T dO, dK += dS^T Q   (P^T, dS^T read from TMEM)
//   bwd_dq_kernel     one CTA per (batch, head, 128-query tile): the second pass.
//                     It streams 64-row tiles of K and V: S = Q K^T, dP = dO V^T,
//                     dQ += dS K.
// Both GEMM kernels recompute S and dP.
//
// dQ by reduction (head dim 128; five GEMMs in all instead of seven):
//   bwd_preprocess    as above, and zeroes an fp32 dQ accumulator [B*H][Mpad][D]
//   bwd_dkdv_kernel   (kDq) a fifth GEMM per step, dQ^T = K^T dS^T (head dim on
//                     TMEM lanes, dS^T also written to shared memory), whose
//                     columns four more warps read out and add into the
//                     accumulator with fp32 reductions at L2.  The order of the
//                     adds varies from run to run, so dQ is not bitwise
//                     reproducible.
//   bwd_dq_convert    dQ = scale * accumulator, rounded to bf16.
//
// Warp roles per CTA: warps 0-3 compute P and dS (thread r owns TMEM lane r),
// warp 4 issues every tcgen05.mma from one thread, warp 5 issues the TMA copies,
// warps 6-9 (kDq) read dQ^T out of TMEM.  TMEM: two stages of {S or S^T: 64
// columns, dP or dP^T: 64 columns} so the tensor core computes step t+1 while
// the CUDA cores work on step t, then the fp32 accumulators (dV and dK, or dQ).
// Every mbarrier wait is bounded in time and winds the CTA down like the
// forward kernel.
#pragma once

#include <cuda_bf16.h>

#include "fa2_fwd_kernel.cuh"

namespace fa2 {

struct BwdParams {
  const float* nl2;   // [BH][Mpad]: -L * log2(e); rows >= M: -inf
  const float* dlt;   // [BH][Mpad]: rowsum(dO o O); rows >= M: 0
  float* dqacc;       // [BH][Mpad][D] fp32 dQ accumulator (dQ by reduction), else null
  int* status;        // sticky device status word
  int M, N, Mpad;     // Mpad = M rounded up to 128
  int head_group;     // causal dK/dV order: key/value heads per group (BHkv: one group)
  int H, group;       // query heads per batch entry; query heads per key/value head
  int BH, BHkv;       // B * H, B * H_kv
  int n_ktiles;       // ceil(N / 128): key tiles per key/value head
  int n_qtiles;       // ceil(M / 128): query tiles per head
  float scale_log2;   // scale * log2(e)
  float scale;        // dK and dQ carry one factor of scale
};

enum : int {
  kStatusBwdTimeoutTma = 20,
  kStatusBwdTimeoutMmaLoad = 21,
  kStatusBwdTimeoutMmaP = 22,
  kStatusBwdTimeoutSoftmax = 23,
  kStatusBwdTimeoutEpilogue = 24,
  kStatusBwdTimeoutDrain = 25,
  kStatusBwdTimeoutMmaDrain = 26,
};

// Instruction descriptor of the dQ^T = K^T dS^T product: bf16, fp32 accumulate,
// both operands MN-major (bits 15 and 16; the other fields as make_idesc).
__host__ __device__ constexpr uint32_t idesc_mn_mn(int m, int n) {
  return ptx::make_idesc(true, true, m, n) | (1u << 15);
}

// fp32 add into global memory, performed at L2 (no value returned).
__device__ __forceinline__ void red_add_f32(float* addr, float v) {
  asm volatile("red.global.add.f32 [%0], %1;" ::"l"(addr), "f"(v) : "memory");
}

// ------------------------------------------------------------------ preprocess
// Per query row: D_i = sum_d dO[i,d] O[i,d] in fp32 from bf16, and -L_i log2(e),
// the exponent offset of P = exp2(s scale log2(e) - L_i log2(e)).
// Rows in [M, Mpad) of every head get D = 0 and -inf.
// With dQ by reduction it also zeroes the row's D accumulator entries.  A row
// is D / 8 lanes with one 16-byte load of O and of dO each (32 / (D / 8) rows
// per warp per pass).
template <int D>
__global__ void __launch_bounds__(256) bwd_preprocess_kernel(const __nv_bfloat16* __restrict__ o,
                                                             const __nv_bfloat16* __restrict__ dout,
                                                             const float* __restrict__ lse,
                                                             float* __restrict__ nl2,
                                                             float* __restrict__ dlt,
                                                             float* __restrict__ dqacc, int M, int Mpad,
                                                             int64_t rows_pad) {
  constexpr int kLanes = D / 8;             // lanes per row
  constexpr int kRowsPerWarp = 32 / kLanes;
  const int lane = static_cast<int>(threadIdx.x) % 32;
  const int sub = lane % kLanes;
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x / 32);
  for (int64_t r0 = (static_cast<int64_t>(blockIdx.x) * (blockDim.x / 32) + threadIdx.x / 32) * kRowsPerWarp;
       r0 < rows_pad; r0 += warps * kRowsPerWarp) {
    const int64_t r = r0 + lane / kLanes;  // rows_pad is a multiple of 128: r < rows_pad
    const int64_t bh = r / Mpad;
    const int i = static_cast<int>(r % Mpad);
    float acc = 0.f;
    if (i < M) {
      const int64_t off = (bh * M + i) * D + sub * 8;
      const uint4 a = *reinterpret_cast<const uint4*>(o + off);
      const uint4 b = *reinterpret_cast<const uint4*>(dout + off);
      const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, bw[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const __nv_bfloat162 a2 = *reinterpret_cast<const __nv_bfloat162*>(&aw[e]);
        const __nv_bfloat162 b2 = *reinterpret_cast<const __nv_bfloat162*>(&bw[e]);
        acc = fmaf(__low2float(a2), __low2float(b2), acc);
        acc = fmaf(__high2float(a2), __high2float(b2), acc);
      }
    }
#pragma unroll
    for (int sh = kLanes / 2; sh > 0; sh >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, sh);
    if (sub == 0) {
      dlt[r] = acc;
      nl2[r] = i < M ? lse[bh * M + i] * -1.4426950408889634f : -INFINITY;
    }
    if (dqacc) {
      float4* z = reinterpret_cast<float4*>(dqacc + r * D + sub * 8);
      z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
      z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
}

// dQ[bh][i] = scale * accumulator[bh][i] rounded to bf16, for rows i < M; eight
// elements per thread.
template <int D>
__global__ void __launch_bounds__(256) bwd_dq_convert_kernel(const float* __restrict__ dqacc,
                                                             __nv_bfloat16* __restrict__ dq, float scale,
                                                             int M, int Mpad, int64_t n8) {
  for (int64_t x = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; x < n8;
       x += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t row = x / (D / 8);  // bh * M + i
    const int c8 = static_cast<int>(x % (D / 8)) * 8;
    const int64_t bh = row / M;
    const float* src = dqacc + (bh * Mpad + (row - bh * M)) * D + c8;
    const float4 a = *reinterpret_cast<const float4*>(src);
    const float4 b = *reinterpret_cast<const float4*>(src + 4);
    uint4 w;
    w.x = ptx::pack_bf16x2(a.x * scale, a.y * scale);
    w.y = ptx::pack_bf16x2(a.z * scale, a.w * scale);
    w.z = ptx::pack_bf16x2(b.x * scale, b.y * scale);
    w.w = ptx::pack_bf16x2(b.z * scale, b.w * scale);
    *reinterpret_cast<uint4*>(dq + row * D + c8) = w;
  }
}

// ------------------------------------------------------------------ shared configuration
template <int D_, int kStages_, bool kDq_ = false>
struct BwdCfg {
  static constexpr int D = D_;
  static constexpr int kStages = kStages_;  // depth of the ring of streamed tiles
  static constexpr bool kDq = kDq_;         // dK/dV kernel also forms dQ (by reduction)
  static constexpr int kDsBufs = 2;         // kDq: dS^T tiles in shared memory, one per step parity
  static constexpr int BF = 128;            // rows of the fixed tile (keys or queries)
  static constexpr int BS = 64;             // rows of a streamed tile per step
  static constexpr int kColBlocks = D / 64;  // 128-byte column blocks of a bf16 row
  static constexpr int kFixBlock = BF * 128;  // one column block of a 128-row tile
  static constexpr int kStrBlock = BS * 128;  // one column block of a 64-row tile
  static constexpr int kFixTile = kColBlocks * kFixBlock;
  static constexpr int kStrTile = kColBlocks * kStrBlock;
  static constexpr int kMmaK = 16;  // bf16 elements per MMA K step (32 bytes)
  static constexpr int kStepsD = D / kMmaK;
  static constexpr int kThreads = kDq ? 320 : 192;
  static constexpr int kMmaWarp = 4;
  static constexpr int kTmaWarp = 5;
  static constexpr int kDrainWarp0 = 6;  // kDq: warps 6-9 (one per TMEM lane quarter)
  static constexpr uint32_t kTmemCols = 512;
  // TMEM columns: stage s holds S (or S^T) at [128 s, +64) and dP (or dP^T) at
  // [128 s + 64, +64); P and dS overwrite them as packed bf16 (32 columns each):
  // P over the first half of S, dS over the first half of dP, or with kDq over
  // the second half of S, so that the step's dQ^T (64 fp32 columns, head dim on
  // the lanes) accumulates in the dP columns
  __host__ __device__ static constexpr int kColS(int s) { return 128 * s; }
  __host__ __device__ static constexpr int kColDP(int s) { return 128 * s + 64; }
  __host__ __device__ static constexpr int kColDS(int s) { return kDq ? 128 * s + 32 : 128 * s + 64; }
  static constexpr int kColAcc0 = 256;      // dV (dK/dV kernel) or dQ (dQ kernel)
  static constexpr int kColAcc1 = 256 + D;  // dK (dK/dV kernel)
  static constexpr uint32_t kIdescS = ptx::make_idesc(true, false, BF, BS);  // B K-major, N = 64
  static constexpr uint32_t kIdescAcc = ptx::make_idesc(true, true, BF, D);  // B MN-major, N = D
  static constexpr uint32_t kIdescDq = idesc_mn_mn(D, BS);  // dQ^T: M = D, N = 64 queries, K = keys
  static_assert(D == 64 || D == 128, "head dim");
  static_assert(kColAcc1 + D <= 512, "TMEM budget");
  static_assert(!kDq || D == 128, "dQ^T has the head dim on TMEM lanes: M = D = 128");
};

// Bounded waits shared by the roles; `ok` turns false on abort or timeout.
#define FA2_BWD_WAIT(bar_addr, parity, code) wait_bounded((bar_addr), (parity), wctx, (code))

// ------------------------------------------------------------------ dK, dV
template <class C>
struct DkvLayout {
  // shared memory: K, V (fixed, 128 rows), then kStages x {Q, dO (64 rows), L2, D vectors}
  static constexpr int kOffK = 0;
  static constexpr int kOffV = kOffK + C::kFixTile;
  static constexpr int kOffRing = kOffV + C::kFixTile;
  // (a stage starts on a 1024-byte boundary, as the 128-byte swizzle requires)
  static constexpr int kStageBytes = (2 * C::kStrTile + 2 * C::BS * 4 + 1023) / 1024 * 1024;
  // kDq: dS^T of the last two steps (tile t % 2), each [128 keys][64 queries]
  // bf16 in 128-byte swizzled rows
  static constexpr int kOffDS = kOffRing + C::kStages * kStageBytes;
  static constexpr int kDSTile = C::BF * 128;
  static constexpr int kDSBytes = C::kDq ? C::kDsBufs * kDSTile : 0;
  static constexpr int kOffBar = kOffDS + kDSBytes;
  // barriers: KV, full[S], empty[S], sfull[2], pfull[2], done, and with kDq
  // qfull[2] (dQ^T of the step complete) and qdrained[2] (read out of TMEM)
  static constexpr int kBarKV = 0;
  static constexpr int kBarFull = 1;
  static constexpr int kBarEmpty = kBarFull + C::kStages;
  static constexpr int kBarSFull = kBarEmpty + C::kStages;
  static constexpr int kBarPFull = kBarSFull + 2;
  static constexpr int kBarDone = kBarPFull + 2;
  static constexpr int kBarQFull = kBarDone + 1;
  static constexpr int kBarQDrained = kBarQFull + 2;
  static constexpr int kNumBars = C::kDq ? kBarQDrained + 2 : kBarDone + 1;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kSmemBytes = kOffMisc + 16 + 1024;
  static_assert(kSmemBytes <= 232448, "shared memory budget");
  __host__ __device__ static constexpr int q_off(int s) { return kOffRing + s * kStageBytes; }
  __host__ __device__ static constexpr int do_off(int s) { return q_off(s) + C::kStrTile; }
  __host__ __device__ static constexpr int l2_off(int s) { return q_off(s) + 2 * C::kStrTile; }
  __host__ __device__ static constexpr int dl_off(int s) { return l2_off(s) + C::BS * 4; }
};

// Work of one dK/dV CTA: query steps of 64 rows over every head of the group.
struct DkvUnit {
  int bhkv;   // flat batch * H_kv + key/value head
  int jt;     // key tile
  int i0;     // first 64-row query step that sees a key of this tile
  int nq;     // steps per query head
  int steps;  // group * nq
};

template <bool kCausal>
__device__ __forceinline__ DkvUnit dkv_unit(const BwdParams& p, int b) {
  DkvUnit u;
  if (kCausal) {
    // groups of head_group key/value heads one after another (their Q, dO and dQ
    // rows stay in L2); within a group the smallest key tile first, over the
    // group's heads (it has the most query steps)
    const int per = p.head_group * p.n_ktiles;
    const int g = b / per, rem = b - g * per;
    const int heads = min(p.head_group, p.BHkv - g * p.head_group);
    u.jt = rem / heads;
    u.bhkv = g * p.head_group + rem % heads;
  } else {  // tiles of one key/value head adjacent: Q and dO of its heads stay in L2
    u.bhkv = b / p.n_ktiles;
    u.jt = b % p.n_ktiles;
  }
  const int nsteps = (p.M + 63) / 64;
  u.i0 = kCausal ? min(u.jt * 2, nsteps) : 0;  // queries below the tile's first key see none of it
  u.nq = nsteps - u.i0;
  u.steps = u.nq * p.group;
  return u;
}

template <class C, bool kCausal>
__global__ void __launch_bounds__(C::kThreads, 1)
    bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmdO,
                    const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                    const __grid_constant__ CUtensorMap tmdK, const __grid_constant__ CUtensorMap tmdV,
                    const BwdParams p) {
  using namespace ptx;
  using Lay = DkvLayout<C>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  volatile uint32_t* misc = reinterpret_cast<volatile uint32_t*>(gbase + Lay::kOffMisc);
  const int warp = static_cast<int>(threadIdx.x) / 32;
  const int lane = static_cast<int>(threadIdx.x) % 32;
  auto bar = [&](int i) -> uint32_t { return base + Lay::kOffBar + 8u * static_cast<uint32_t>(i); };

  const DkvUnit u = dkv_unit<kCausal>(p, static_cast<int>(blockIdx.x));
  const int key0 = u.jt * C::BF;
  const int Hkv = p.H / p.group;
  // query head of step t and its first row
  auto step_head = [&](int t) { return (u.bhkv / Hkv) * p.H + (u.bhkv % Hkv) * p.group + t / u.nq; };
  auto step_row0 = [&](int t) { return (u.i0 + t % u.nq) * C::BS; };

  if (threadIdx.x == 0) {
    misc[1] = 0u;
    misc[2] = static_cast<uint32_t>(*reinterpret_cast<volatile int*>(p.status));
    mbar_init(bar(Lay::kBarKV), 1);
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(bar(Lay::kBarFull + s), 1);
      mbar_init(bar(Lay::kBarEmpty + s), 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(Lay::kBarSFull + s), 1);
      mbar_init(bar(Lay::kBarPFull + s), 128);
      if constexpr (C::kDq) {
        mbar_init(bar(Lay::kBarQFull + s), 1);
        mbar_init(bar(Lay::kBarQDrained + s), 128);
      }
    }
    mbar_init(bar(Lay::kBarDone), 1);
    fence_mbar_init();
  }
  if (warp == C::kTmaWarp && lane == 0) {
    prefetch_tensormap(&tmQ);
    prefetch_tensormap(&tmdO);
    prefetch_tensormap(&tmK);
    prefetch_tensormap(&tmV);
  }
  if (warp == C::kMmaWarp) {
    tmem_alloc(base + Lay::kOffMisc, C::kTmemCols);
    tmem_relinquish_alloc_permit();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = misc[0];
  const bool skip = misc[2] != 0u;
  const WaitCtx wctx{misc + 1, p.status};

  if (!skip && warp == C::kTmaWarp) {
    // ---------------------------------------------------------- TMA producer
    if (lane == 0) {
      const uint64_t pol_fix = l2_policy_evict_first();
      const uint64_t pol_str = l2_policy_evict_last();
      mbar_arrive_expect_tx(bar(Lay::kBarKV), 2 * C::kFixTile);
#pragma unroll
      for (int cb = 0; cb < C::kColBlocks; ++cb) {
        tma_load_3d_hint(base + Lay::kOffK + cb * C::kFixBlock, &tmK, bar(Lay::kBarKV), cb * 64, key0,
                         u.bhkv, pol_fix);
        tma_load_3d_hint(base + Lay::kOffV + cb * C::kFixBlock, &tmV, bar(Lay::kBarKV), cb * 64, key0,
                         u.bhkv, pol_fix);
      }
      int issued = 0;
      for (int t = 0; t < u.steps; ++t) {
        const int s = t % C::kStages;
        const uint32_t use = static_cast<uint32_t>(t / C::kStages);
        if (use > 0 && !FA2_BWD_WAIT(bar(Lay::kBarEmpty + s), (use - 1) & 1u, kStatusBwdTimeoutTma)) break;
        const int bh = step_head(t), row0 = step_row0(t);
        const uint32_t fb = bar(Lay::kBarFull + s);
        mbar_arrive_expect_tx(fb, 2 * C::kStrTile + 2 * C::BS * 4);
#pragma unroll
        for (int cb = 0; cb < C::kColBlocks; ++cb) {
          tma_load_3d_hint(base + Lay::q_off(s) + cb * C::kStrBlock, &tmQ, fb, cb * 64, row0, bh, pol_str);
          tma_load_3d_hint(base + Lay::do_off(s) + cb * C::kStrBlock, &tmdO, fb, cb * 64, row0, bh, pol_str);
        }
        const int64_t vec = static_cast<int64_t>(bh) * p.Mpad + row0;
        bulk_load_1d(base + Lay::l2_off(s), p.nl2 + vec, C::BS * 4, fb);
        bulk_load_1d(base + Lay::dl_off(s), p.dlt + vec, C::BS * 4, fb);
        issued = t + 1;
      }
      if (*wctx.abort_flag) {
        drain_bounded(bar(Lay::kBarKV), 0);
        for (int t = max(0, issued - C::kStages); t < issued; ++t)
          drain_bounded(bar(Lay::kBarFull + t % C::kStages), (t / C::kStages) & 1);
      }
    }
    __syncwarp();
  } else if (!skip && warp == C::kMmaWarp) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      // Descriptor words (K-major operands; MN-major B of the accumulating GEMMs):
      // a K step or a ring stage is one add to the low word, which keeps the
      // instructions between MMAs few (the issuing thread shares its scheduler
      // with the P/dS warps).
      const uint64_t dk = smem_desc_sw128(base, 16, 1024);
      const uint64_t dm = smem_desc(base, C::kStrBlock, 1024, kLayoutSw128);
      // kDq: K^T (A, MN-major: the head dim runs along the 128-byte rows of the
      // K tile's column blocks, kFixBlock apart) and dS^T (B, MN-major: one
      // 64-query block); both step along the keys by 8-row groups of 1024 bytes
      const uint64_t df = smem_desc(base, C::kFixBlock, 1024, kLayoutSw128);
      const uint32_t k_lo0 = static_cast<uint32_t>(dk), k_hi = static_cast<uint32_t>(dk >> 32);
      const uint32_t m_lo0 = static_cast<uint32_t>(dm), m_hi = static_cast<uint32_t>(dm >> 32);
      const uint32_t f_lo0 = static_cast<uint32_t>(df), f_hi = static_cast<uint32_t>(df >> 32);
      bool ok = FA2_BWD_WAIT(bar(Lay::kBarKV), 0, kStatusBwdTimeoutMmaLoad);
      for (int t = 0; ok && t <= u.steps; ++t) {
        if (t < u.steps) {
          const int s = t % C::kStages, ts = t % 2;
          ok = FA2_BWD_WAIT(bar(Lay::kBarFull + s), (t / C::kStages) & 1, kStatusBwdTimeoutMmaLoad);
          if (!ok) break;
          tc_fence_after_sync();
          const uint32_t q_lo = k_lo0 + (static_cast<uint32_t>(Lay::q_off(s)) >> 4);
          const uint32_t do_lo = k_lo0 + (static_cast<uint32_t>(Lay::do_off(s)) >> 4);
          // S^T = K Q^T and dP^T = V dO^T: M = 128 keys, N = 64 queries, K = D
#pragma unroll
          for (int kk = 0; kk < C::kStepsD; ++kk) {
            const uint32_t fo = ((kk / 4) * C::kFixBlock + (kk % 4) * 32) >> 4;
            const uint32_t so = ((kk / 4) * C::kStrBlock + (kk % 4) * 32) >> 4;
            mma_f16_ss(tmem + C::kColS(ts), desc_from_words(k_lo0 + (Lay::kOffK >> 4) + fo, k_hi),
                       desc_from_words(q_lo + so, k_hi), C::kIdescS, kk > 0 ? 1u : 0u);
          }
          if constexpr (C::kDq) {
            // dP^T of this step overwrites the dQ^T of step t - 2: wait until it was read out
            if (t >= 2) {
              ok = FA2_BWD_WAIT(bar(Lay::kBarQDrained + ts), ((t - 2) / 2) & 1, kStatusBwdTimeoutMmaDrain);
              if (!ok) break;
              tc_fence_after_sync();
            }
          }
#pragma unroll
          for (int kk = 0; kk < C::kStepsD; ++kk) {
            const uint32_t fo = ((kk / 4) * C::kFixBlock + (kk % 4) * 32) >> 4;
            const uint32_t so = ((kk / 4) * C::kStrBlock + (kk % 4) * 32) >> 4;
            mma_f16_ss(tmem + C::kColDP(ts), desc_from_words(k_lo0 + (Lay::kOffV >> 4) + fo, k_hi),
                       desc_from_words(do_lo + so, k_hi), C::kIdescS, kk > 0 ? 1u : 0u);
          }
          tc_commit(bar(Lay::kBarSFull + ts));
        }
        if (t >= 1) {
          const int tp = t - 1, sp = tp % C::kStages, tsp = tp % 2;
          ok = FA2_BWD_WAIT(bar(Lay::kBarPFull + tsp), (tp / 2) & 1, kStatusBwdTimeoutMmaP);
          if (!ok) break;
          tc_fence_after_sync();
          const uint32_t q_lo = m_lo0 + (static_cast<uint32_t>(Lay::q_off(sp)) >> 4);
          const uint32_t do_lo = m_lo0 + (static_cast<uint32_t>(Lay::do_off(sp)) >> 4);
          // dV += P^T dO and dK += dS^T Q: M = 128 keys, N = D, K = 64 queries;
          // A from TMEM (packed bf16), B = the 64-row tile read MN-major
#pragma unroll
          for (int kk = 0; kk < C::BS / C::kMmaK; ++kk) {
            const uint32_t bo = (kk * C::kMmaK * 128) >> 4;
            mma_f16_ts(tmem + C::kColAcc0, tmem + C::kColS(tsp) + kk * 8, desc_from_words(do_lo + bo, m_hi),
                       C::kIdescAcc, (tp > 0 || kk > 0) ? 1u : 0u);
            mma_f16_ts(tmem + C::kColAcc1, tmem + C::kColDS(tsp) + kk * 8, desc_from_words(q_lo + bo, m_hi),
                       C::kIdescAcc, (tp > 0 || kk > 0) ? 1u : 0u);
          }
          tc_commit(bar(Lay::kBarEmpty + sp));
          if constexpr (C::kDq) {
            // dQ^T = K^T dS^T: M = D, N = 64 queries, K = 128 keys, into the dP^T columns
#pragma unroll
            for (int kk = 0; kk < C::BF / C::kMmaK; ++kk) {
              const uint32_t ko = (kk * C::kMmaK * 128) >> 4;
              const uint32_t dso = (Lay::kOffDS + (tp % C::kDsBufs) * Lay::kDSTile) >> 4;
              mma_f16_ss(tmem + C::kColDP(tsp), desc_from_words(f_lo0 + (Lay::kOffK >> 4) + ko, f_hi),
                         desc_from_words(f_lo0 + dso + ko, f_hi), C::kIdescDq, kk > 0 ? 1u : 0u);
            }
            tc_commit(bar(Lay::kBarQFull + tsp));
          }
        }
      }
      tc_commit(bar(Lay::kBarDone));
      drain_bounded(bar(Lay::kBarDone), 0);
    }
    __syncwarp();
  } else if (!skip && warp < 4) {
    // ---------------------------------------------------------- P and dS
    const int r = warp * 32 + lane;  // key row of the tile = TMEM lane
    const int key = key0 + r;
    const bool key_ok = key < p.N;
    const uint32_t lane_addr = static_cast<uint32_t>(warp * 32) << 16;
    const float sl2 = p.scale_log2;
    bool ok = true;
    for (int t = 0; t < u.steps; ++t) {
      const int s = t % C::kStages, ts = t % 2;
      // S^T and dP^T of this step are in TMEM; the L and D vectors of the step
      // were copied by TMA with the stage (wait on both)
      ok = __all_sync(0xffffffffu, FA2_BWD_WAIT(bar(Lay::kBarSFull + ts), (t / 2) & 1, kStatusBwdTimeoutSoftmax));
      if (ok)
        ok = __all_sync(0xffffffffu,
                        FA2_BWD_WAIT(bar(Lay::kBarFull + s), (t / C::kStages) & 1, kStatusBwdTimeoutSoftmax));
      if (!ok) break;
      tc_fence_after_sync();
      uint32_t sv[64], dv[64];
      tmem_ld_x32(tmem + lane_addr + C::kColS(ts), *reinterpret_cast<uint32_t(*)[32]>(&sv[0]));
      tmem_ld_x32(tmem + lane_addr + C::kColS(ts) + 32, *reinterpret_cast<uint32_t(*)[32]>(&sv[32]));
      tmem_ld_x32(tmem + lane_addr + C::kColDP(ts), *reinterpret_cast<uint32_t(*)[32]>(&dv[0]));
      tmem_ld_x32(tmem + lane_addr + C::kColDP(ts) + 32, *reinterpret_cast<uint32_t(*)[32]>(&dv[32]));
      tmem_ld_wait();
      reg_fence_x32(*reinterpret_cast<uint32_t(*)[32]>(&sv[0]));
      reg_fence_x32(*reinterpret_cast<uint32_t(*)[32]>(&sv[32]));
      reg_fence_x32(*reinterpret_cast<uint32_t(*)[32]>(&dv[0]));
      reg_fence_x32(*reinterpret_cast<uint32_t(*)[32]>(&dv[32]));
      const int row0 = step_row0(t);
      uint32_t pk[32], dk[32];
      if ((!kCausal || row0 >= key0 + C::BF) && key0 + C::BF <= p.N) {
        // every query of the step sees every key of the tile: no mask, and the
        // arithmetic on packed pairs (one FFMA2, FSUB2 and FMUL2 per two scores)
        const uint64_t sl2x2 = pack_f32x2(sl2, sl2);
#pragma unroll
        for (int c4 = 0; c4 < C::BS; c4 += 4) {
          float l2[4], dl[4];
          ld_shared_v4(base + Lay::l2_off(s) + c4 * 4, l2[0], l2[1], l2[2], l2[3]);
          ld_shared_v4(base + Lay::dl_off(s) + c4 * 4, dl[0], dl[1], dl[2], dl[3]);
#pragma unroll
          for (int e = 0; e < 4; e += 2) {
            const int c = c4 + e;
            float x0, x1, d0, d1;
            unpack_f32x2(ffma2(pack_f32x2(__uint_as_float(sv[c]), __uint_as_float(sv[c + 1])), sl2x2,
                               pack_f32x2(l2[e], l2[e + 1])),
                         x0, x1);
            const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
            unpack_f32x2(fmul2(pack_f32x2(p0, p1),
                               fsub2(pack_f32x2(__uint_as_float(dv[c]), __uint_as_float(dv[c + 1])),
                                     pack_f32x2(dl[e], dl[e + 1]))),
                         d0, d1);
            pk[c / 2] = pack_bf16x2(p0, p1);
            dk[c / 2] = pack_bf16x2(d0, d1);
          }
        }
      } else {
        // causal: query row0 + c sees this key iff row0 + c >= key (diagonal steps only)
        const int lim = (kCausal && row0 < key0 + C::BF) ? key - row0 : -1;
#pragma unroll
        for (int c4 = 0; c4 < C::BS; c4 += 4) {
          float l2[4], dl[4];
          ld_shared_v4(base + Lay::l2_off(s) + c4 * 4, l2[0], l2[1], l2[2], l2[3]);
          ld_shared_v4(base + Lay::dl_off(s) + c4 * 4, dl[0], dl[1], dl[2], dl[3]);
          float pv[4], dsv[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int c = c4 + e;
            const bool vis = key_ok && c >= lim;
            const float pe = vis ? ex2_approx(fmaf(__uint_as_float(sv[c]), sl2, l2[e])) : 0.f;
            pv[e] = pe;
            dsv[e] = pe * (__uint_as_float(dv[c]) - dl[e]);
          }
          pk[c4 / 2] = pack_bf16x2(pv[0], pv[1]);
          pk[c4 / 2 + 1] = pack_bf16x2(pv[2], pv[3]);
          dk[c4 / 2] = pack_bf16x2(dsv[0], dsv[1]);
          dk[c4 / 2 + 1] = pack_bf16x2(dsv[2], dsv[3]);
        }
      }
      // kDq: dS^T tile t % 2 is free: the dQ^T product of step t - 2 that read it
      // was issued before this step's S^T, whose completion the wait on sfull saw
      tmem_st_x32(tmem + lane_addr + C::kColS(ts), pk);
      tmem_st_x32(tmem + lane_addr + C::kColDS(ts), dk);
      if constexpr (C::kDq) {
        // row r of dS^T (64 queries) as eight 16-byte chunks, chunk c at c ^ (r mod 8)
        const uint32_t row = base + Lay::kOffDS + (t % C::kDsBufs) * Lay::kDSTile + r * 128;
#pragma unroll
        for (int c = 0; c < 8; ++c)
          st_shared_v4(row + ((c ^ (r & 7)) << 4), dk[4 * c], dk[4 * c + 1], dk[4 * c + 2], dk[4 * c + 3]);
        fence_proxy_async_smem();
      }
      tmem_st_wait();
      tc_fence_before_sync();
      mbar_arrive(bar(Lay::kBarPFull + ts));
    }
    // ------------------------------------------------------------ epilogue
    // dV and scale * dK of this key row -> bf16 -> swizzled staging in the V and
    // K tiles (free once every MMA has completed) -> TMA store, clipped at N
    if (ok)
      ok = __all_sync(0xffffffffu, FA2_BWD_WAIT(bar(Lay::kBarDone), 0, kStatusBwdTimeoutEpilogue));
    if (ok) {
      tc_fence_after_sync();
#pragma unroll
      for (int which = 0; which < 2; ++which) {
        const uint32_t stage = base + (which == 0 ? Lay::kOffV : Lay::kOffK);
        const float mul = which == 0 ? 1.0f : p.scale;
#pragma unroll
        for (int ch = 0; ch < C::D / 32; ++ch) {
          uint32_t v[32];
          if (u.steps > 0) {
            tmem_ld_x32(tmem + lane_addr + (which == 0 ? C::kColAcc0 : C::kColAcc1) + ch * 32, v);
            tmem_ld_wait();
            reg_fence_x32(v);
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = 0u;  // no query sees these keys: zero gradients
          }
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            const int cidx = ch * 4 + q4;
            const int cb = cidx / 8, c = cidx % 8;
            const uint32_t addr = stage + cb * C::kFixBlock + r * 128 + ((c ^ (r & 7)) << 4);
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e)
              w[e] = pack_bf16x2(__uint_as_float(v[q4 * 8 + 2 * e]) * mul, __uint_as_float(v[q4 * 8 + 2 * e + 1]) * mul);
            st_shared_v4(addr, w[0], w[1], w[2], w[3]);
          }
        }
      }
    }
    fence_proxy_async_smem();
    named_barrier_sync(1, 128);
    if (r == 0 && ok && *wctx.abort_flag == 0u) {
#pragma unroll
      for (int cb = 0; cb < C::kColBlocks; ++cb) {
        tma_store_3d(&tmdV, base + Lay::kOffV + cb * C::kFixBlock, cb * 64, key0, u.bhkv);
        tma_store_3d(&tmdK, base + Lay::kOffK + cb * C::kFixBlock, cb * 64, key0, u.bhkv);
      }
      tma_store_commit();
      tma_store_wait_read_all();
    }
  } else if (!skip && C::kDq && warp >= C::kDrainWarp0) {
    // ---------------------------------------------------------- dQ read-out
    // thread d owns TMEM lane d (head-dim column d of dQ^T): per step it reads
    // the 64 query columns and adds them into rows row0 .. row0 + 63 of the
    // query head's accumulator, one 128-byte row segment per warp instruction
    const int quarter = warp % 4;
    const int d = quarter * 32 + lane;
    const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
    for (int t = 0; t < u.steps; ++t) {
      const int ts = t % 2;
      if (!__all_sync(0xffffffffu, FA2_BWD_WAIT(bar(Lay::kBarQFull + ts), (t / 2) & 1, kStatusBwdTimeoutDrain)))
        break;
      tc_fence_after_sync();
      uint32_t v[64];
      tmem_ld_x32(tmem + lane_addr + C::kColDP(ts), *reinterpret_cast<uint32_t(*)[32]>(&v[0]));
      tmem_ld_x32(tmem + lane_addr + C::kColDP(ts) + 32, *reinterpret_cast<uint32_t(*)[32]>(&v[32]));
      tmem_ld_wait();
      reg_fence_x32(*reinterpret_cast<uint32_t(*)[32]>(&v[0]));
      reg_fence_x32(*reinterpret_cast<uint32_t(*)[32]>(&v[32]));
      tc_fence_before_sync();
      mbar_arrive(bar(Lay::kBarQDrained + ts));
      float* dst = p.dqacc + (static_cast<int64_t>(step_head(t)) * p.Mpad + step_row0(t)) * C::D + d;
#pragma unroll
      for (int q = 0; q < C::BS; ++q) red_add_f32(dst + q * C::D, __uint_as_float(v[q]));
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == C::kMmaWarp) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

// ------------------------------------------------------------------ dQ
// Two 128-row query tiles per CTA share every streamed 64-row K/V step and
// ping-pong on the tensor core like the forward: while warpgroup t forms dS of
// tile t, the MMA thread runs the other tile's GEMMs.  TMEM per tile t (256
// columns): S_t [256 t, +64) (dS_t overwrites its first 32 as packed bf16),
// dP_t [256 t + 64, +64), dQ_t [256 t + 128, +D).
template <int D_, int kStages_>
struct DqCfg {
  static constexpr int D = D_;
  static constexpr int kStages = kStages_;
  static constexpr int kQT = 2;              // query tiles per CTA
  static constexpr int BF = 128;             // rows of a query tile
  static constexpr int BS = 64;              // keys per step
  static constexpr int kColBlocks = D / 64;
  static constexpr int kFixBlock = BF * 128;
  static constexpr int kStrBlock = BS * 128;
  static constexpr int kFixTile = kColBlocks * kFixBlock;
  static constexpr int kStrTile = kColBlocks * kStrBlock;
  static constexpr int kMmaK = 16;
  static constexpr int kStepsD = D / kMmaK;
  static constexpr int kSoftWarps = 4 * kQT;
  static constexpr int kThreads = (kSoftWarps + 2) * 32;
  static constexpr int kMmaWarp = kSoftWarps;
  static constexpr int kTmaWarp = kSoftWarps + 1;
  static constexpr uint32_t kTmemCols = 512;
  __host__ __device__ static constexpr int kColS(int t) { return 256 * t; }
  __host__ __device__ static constexpr int kColDP(int t) { return 256 * t + 64; }
  __host__ __device__ static constexpr int kColQ(int t) { return 256 * t + 128; }
  static constexpr uint32_t kIdescS = ptx::make_idesc(true, false, BF, BS);
  static constexpr uint32_t kIdescAcc = ptx::make_idesc(true, true, BF, D);
  // shared memory: Q[2], dO[2] (fixed), then kStages x {K, V} (64 rows)
  static constexpr int kOffQ = 0;
  static constexpr int kOffDO = kOffQ + kQT * kFixTile;
  static constexpr int kOffRing = kOffDO + kQT * kFixTile;
  static constexpr int kStageBytes = 2 * kStrTile;
  static constexpr int kOffBar = kOffRing + kStages * kStageBytes;
  // barriers: Q[2], full[S], empty[S], sfull[2], pfull[2], done
  static constexpr int kBarQ = 0;
  static constexpr int kBarFull = kBarQ + kQT;
  static constexpr int kBarEmpty = kBarFull + kStages;
  static constexpr int kBarSFull = kBarEmpty + kStages;
  static constexpr int kBarPFull = kBarSFull + kQT;
  static constexpr int kBarDone = kBarPFull + kQT;
  static constexpr int kNumBars = kBarDone + 1;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kSmemBytes = kOffMisc + 16 + 1024;
  __host__ __device__ static constexpr int k_off(int s) { return kOffRing + s * kStageBytes; }
  __host__ __device__ static constexpr int v_off(int s) { return k_off(s) + kStrTile; }
  static_assert(D == 64 || D == 128, "head dim");
  static_assert(kColQ(kQT - 1) + D <= 512, "TMEM budget");
  static_assert(kSmemBytes <= 232448, "shared memory budget");
  static_assert(kStageBytes % 1024 == 0 && kFixTile % 1024 == 0, "1024-byte aligned tiles");
};

// Keys [0, end) that some row of the query tile starting at row0 sees; 0 if the
// tile is past M.
template <bool kCausal>
__device__ __forceinline__ int dq_key_end(int row0, int M, int N) {
  if (row0 >= M) return 0;
  const int last_row = min(row0 + 128, M) - 1;
  return kCausal ? min(N, last_row + 1) : N;
}

template <class C, bool kCausal>
__global__ void __launch_bounds__(C::kThreads, 1)
    bwd_dq_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmdO,
                  const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                  const __grid_constant__ CUtensorMap tmdQ, const BwdParams p) {
  using namespace ptx;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  volatile uint32_t* misc = reinterpret_cast<volatile uint32_t*>(gbase + C::kOffMisc);
  const int warp = static_cast<int>(threadIdx.x) / 32;
  const int lane = static_cast<int>(threadIdx.x) % 32;
  auto bar = [&](int i) -> uint32_t { return base + C::kOffBar + 8u * static_cast<uint32_t>(i); };

  // unit: (head, pair of query tiles); causal pairs longest first, else one head's pairs adjacent
  const int pairs = (p.n_qtiles + C::kQT - 1) / C::kQT;
  const int b = static_cast<int>(blockIdx.x);
  int bh, pair;
  if (kCausal) {
    pair = pairs - 1 - b / p.BH;
    bh = b % p.BH;
  } else {
    bh = b / pairs;
    pair = b % pairs;
  }
  const int bh_kv = (bh / p.H) * (p.H / p.group) + (bh % p.H) / p.group;
  int row0[C::kQT], steps[C::kQT];
  int n_max = 0;
#pragma unroll
  for (int t = 0; t < C::kQT; ++t) {
    row0[t] = (pair * C::kQT + t) * C::BF;
    steps[t] = (dq_key_end<kCausal>(row0[t], p.M, p.N) + C::BS - 1) / C::BS;
    n_max = max(n_max, steps[t]);
  }

  if (threadIdx.x == 0) {
    misc[1] = 0u;
    misc[2] = static_cast<uint32_t>(*reinterpret_cast<volatile int*>(p.status));
    for (int t = 0; t < C::kQT; ++t) {
      mbar_init(bar(C::kBarQ + t), 1);
      mbar_init(bar(C::kBarSFull + t), 1);
      mbar_init(bar(C::kBarPFull + t), 128);
    }
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(bar(C::kBarFull + s), 1);
      mbar_init(bar(C::kBarEmpty + s), 1);
    }
    mbar_init(bar(C::kBarDone), 1);
    fence_mbar_init();
  }
  if (warp == C::kTmaWarp && lane == 0) {
    prefetch_tensormap(&tmQ);
    prefetch_tensormap(&tmdO);
    prefetch_tensormap(&tmK);
    prefetch_tensormap(&tmV);
  }
  if (warp == C::kMmaWarp) {
    tmem_alloc(base + C::kOffMisc, C::kTmemCols);
    tmem_relinquish_alloc_permit();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = misc[0];
  const bool skip = misc[2] != 0u;
  const WaitCtx wctx{misc + 1, p.status};

  if (!skip && warp == C::kTmaWarp) {
    if (lane == 0) {
      const uint64_t pol_fix = l2_policy_evict_first();
      const uint64_t pol_str = l2_policy_evict_last();
#pragma unroll
      for (int t = 0; t < C::kQT; ++t) {
        if (steps[t] == 0) continue;
        mbar_arrive_expect_tx(bar(C::kBarQ + t), 2 * C::kFixTile);
#pragma unroll
        for (int cb = 0; cb < C::kColBlocks; ++cb) {
          tma_load_3d_hint(base + C::kOffQ + t * C::kFixTile + cb * C::kFixBlock, &tmQ, bar(C::kBarQ + t), cb * 64,
                           row0[t], bh, pol_fix);
          tma_load_3d_hint(base + C::kOffDO + t * C::kFixTile + cb * C::kFixBlock, &tmdO, bar(C::kBarQ + t),
                           cb * 64, row0[t], bh, pol_fix);
        }
      }
      int issued = 0;
      for (int j = 0; j < n_max; ++j) {
        const int s = j % C::kStages;
        const uint32_t use = static_cast<uint32_t>(j / C::kStages);
        if (use > 0 && !FA2_BWD_WAIT(bar(C::kBarEmpty + s), (use - 1) & 1u, kStatusBwdTimeoutTma)) break;
        const uint32_t fb = bar(C::kBarFull + s);
        mbar_arrive_expect_tx(fb, 2 * C::kStrTile);
#pragma unroll
        for (int cb = 0; cb < C::kColBlocks; ++cb) {
          tma_load_3d_hint(base + C::k_off(s) + cb * C::kStrBlock, &tmK, fb, cb * 64, j * C::BS, bh_kv, pol_str);
          tma_load_3d_hint(base + C::v_off(s) + cb * C::kStrBlock, &tmV, fb, cb * 64, j * C::BS, bh_kv, pol_str);
        }
        issued = j + 1;
      }
      if (*wctx.abort_flag) {
        for (int t = 0; t < C::kQT; ++t)
          if (steps[t] > 0) drain_bounded(bar(C::kBarQ + t), 0);
        for (int j = max(0, issued - C::kStages); j < issued; ++j)
          drain_bounded(bar(C::kBarFull + j % C::kStages), (j / C::kStages) & 1);
      }
    }
    __syncwarp();
  } else if (!skip && warp == C::kMmaWarp) {
    if (lane == 0) {
      // descriptor words, as in the dK/dV issuer
      const uint64_t dk = smem_desc_sw128(base, 16, 1024);
      const uint64_t dm = smem_desc(base, C::kStrBlock, 1024, kLayoutSw128);
      const uint32_t k_lo0 = static_cast<uint32_t>(dk), k_hi = static_cast<uint32_t>(dk >> 32);
      const uint32_t m_lo0 = static_cast<uint32_t>(dm), m_hi = static_cast<uint32_t>(dm >> 32);
      bool ok = true;
#pragma unroll
      for (int t = 0; t < C::kQT; ++t)
        if (ok && steps[t] > 0) ok = FA2_BWD_WAIT(bar(C::kBarQ + t), 0, kStatusBwdTimeoutMmaLoad);
      for (int j = 0; ok && j <= n_max; ++j) {
        const int s = j % C::kStages;
        bool kv_ready = false;
#pragma unroll
        for (int t = 0; t < C::kQT; ++t) {
          if (j >= 1 && j - 1 < steps[t]) {
            // dQ_t += dS_t K_{j-1}: M = 128 queries, N = D, K = 64 keys; K tile MN-major
            const int jp = j - 1, sp = jp % C::kStages;
            ok = FA2_BWD_WAIT(bar(C::kBarPFull + t), jp & 1, kStatusBwdTimeoutMmaP);
            if (!ok) break;
            tc_fence_after_sync();
            const uint32_t kv_lo = m_lo0 + (static_cast<uint32_t>(C::k_off(sp)) >> 4);
#pragma unroll
            for (int kk = 0; kk < C::BS / C::kMmaK; ++kk)
              mma_f16_ts(tmem + C::kColQ(t), tmem + C::kColS(t) + kk * 8,
                         desc_from_words(kv_lo + ((kk * C::kMmaK * 128) >> 4), m_hi), C::kIdescAcc,
                         (jp > 0 || kk > 0) ? 1u : 0u);
          }
          if (j < steps[t]) {
            if (!kv_ready) {
              ok = FA2_BWD_WAIT(bar(C::kBarFull + s), (j / C::kStages) & 1, kStatusBwdTimeoutMmaLoad);
              if (!ok) break;
              kv_ready = true;
              tc_fence_after_sync();
            }
            // S_t = Q_t K_j^T and dP_t = dO_t V_j^T: M = 128 queries, N = 64 keys, K = D
            const uint32_t q_lo = k_lo0 + ((C::kOffQ + t * C::kFixTile) >> 4);
            const uint32_t o_lo = k_lo0 + ((C::kOffDO + t * C::kFixTile) >> 4);
            const uint32_t kk_lo = k_lo0 + (static_cast<uint32_t>(C::k_off(s)) >> 4);
            const uint32_t vv_lo = k_lo0 + (static_cast<uint32_t>(C::v_off(s)) >> 4);
#pragma unroll
            for (int kk = 0; kk < C::kStepsD; ++kk) {
              const uint32_t fo = ((kk / 4) * C::kFixBlock + (kk % 4) * 32) >> 4;
              const uint32_t so = ((kk / 4) * C::kStrBlock + (kk % 4) * 32) >> 4;
              mma_f16_ss(tmem + C::kColS(t), desc_from_words(q_lo + fo, k_hi), desc_from_words(kk_lo + so, k_hi),
                         C::kIdescS, kk > 0 ? 1u : 0u);
            }
#pragma unroll
            for (int kk = 0; kk < C::kStepsD; ++kk) {
              const uint32_t fo = ((kk / 4) * C::kFixBlock + (kk % 4) * 32) >> 4;
              const uint32_t so = ((kk / 4) * C::kStrBlock + (kk % 4) * 32) >> 4;
              mma_f16_ss(tmem + C::kColDP(t), desc_from_words(o_lo + fo, k_hi), desc_from_words(vv_lo + so, k_hi),
                         C::kIdescS, kk > 0 ? 1u : 0u);
            }
            tc_commit(bar(C::kBarSFull + t));
          }
        }
        if (!ok) break;
        // a K/V stage is handed back after every GEMM reading it was issued
        if (j >= 1) tc_commit(bar(C::kBarEmpty + (j - 1) % C::kStages));
      }
      tc_commit(bar(C::kBarDone));
      drain_bounded(bar(C::kBarDone), 0);
    }
    __syncwarp();
  } else if (!skip && warp < C::kSoftWarps) {
    const int t = warp / 4;
    const int r = (warp % 4) * 32 + lane;  // query row of tile t = TMEM lane
    const int tile_row0 = (pair * C::kQT + t) * C::BF;
    const int row = tile_row0 + r;
    const int n_t = (dq_key_end<kCausal>(tile_row0, p.M, p.N) + C::BS - 1) / C::BS;
    const uint32_t lane_addr = static_cast<uint32_t>((warp % 4) * 32) << 16;
    float l2 = -INFINITY, dl = 0.f;  // -L log2(e) and D of this row
    if (n_t > 0) {
      const int64_t vec = static_cast<int64_t>(bh) * p.Mpad + row;  // row < Mpad when the tile is in range
      l2 = p.nl2[vec];
      dl = p.dlt[vec];
    }
    const float sl2 = p.scale_log2;
    const uint64_t sl2x2 = pack_f32x2(sl2, sl2), l2x2 = pack_f32x2(l2, l2), dlx2 = pack_f32x2(dl, dl);
    bool ok = n_t > 0;
    for (int j = 0; ok && j < n_t; ++j) {
      ok = __all_sync(0xffffffffu, FA2_BWD_WAIT(bar(C::kBarSFull + t), j & 1, kStatusBwdTimeoutSoftmax));
      if (!ok) break;
      tc_fence_after_sync();
      uint32_t sv[64], dv[64];
      tmem_ld_x32(tmem + lane_addr + C::kColS(t), *reinterpret_cast<uint32_t(*)[32]>(&sv[0]));
      tmem_ld_x32(tmem + lane_addr + C::kColS(t) + 32, *reinterpret_cast<uint32_t(*)[32]>(&sv[32]));
      tmem_ld_x32(tmem + lane_addr + C::kColDP(t), *reinterpret_cast<uint32_t(*)[32]>(&dv[0]));
      tmem_ld_x32(tmem + lane_addr + C::kColDP(t) + 32, *reinterpret_cast<uint32_t(*)[32]>(&dv[32]));
      tmem_ld_wait();
      reg_fence_x32(*reinterpret_cast<uint32_t(*)[32]>(&sv[0]));
      reg_fence_x32(*reinterpret_cast<uint32_t(*)[32]>(&sv[32]));
      reg_fence_x32(*reinterpret_cast<uint32_t(*)[32]>(&dv[0]));
      reg_fence_x32(*reinterpret_cast<uint32_t(*)[32]>(&dv[32]));
      // keys past N (zero-filled rows of K) and, when causal, keys after this row
      const int kbase = j * C::BS;
      int lim = p.N - 1 - kbase;
      if (kCausal) lim = min(lim, row - kbase);
      uint32_t dk[32];
      if (__all_sync(0xffffffffu, lim >= C::BS - 1)) {
        // every key of the step is visible to every row of the warp: no mask, and
        // the arithmetic on packed pairs
#pragma unroll
        for (int c = 0; c < C::BS; c += 2) {
          float x0, x1, d0, d1;
          unpack_f32x2(ffma2(pack_f32x2(__uint_as_float(sv[c]), __uint_as_float(sv[c + 1])), sl2x2, l2x2), x0,
                       x1);
          unpack_f32x2(fmul2(pack_f32x2(ex2_approx(x0), ex2_approx(x1)),
                             fsub2(pack_f32x2(__uint_as_float(dv[c]), __uint_as_float(dv[c + 1])), dlx2)),
                       d0, d1);
          dk[c / 2] = pack_bf16x2(d0, d1);
        }
      } else {
#pragma unroll
        for (int c = 0; c < C::BS; c += 2) {
          float d2[2];
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const float pe = (c + e <= lim) ? ex2_approx(fmaf(__uint_as_float(sv[c + e]), sl2, l2)) : 0.f;
            d2[e] = pe * (__uint_as_float(dv[c + e]) - dl);
          }
          dk[c / 2] = pack_bf16x2(d2[0], d2[1]);
        }
      }
      tmem_st_x32(tmem + lane_addr + C::kColS(t), dk);
      tmem_st_wait();
      tc_fence_before_sync();
      mbar_arrive(bar(C::kBarPFull + t));
    }
    if (n_t > 0) {
      if (ok) ok = __all_sync(0xffffffffu, FA2_BWD_WAIT(bar(C::kBarDone), 0, kStatusBwdTimeoutEpilogue));
      const uint32_t stage = base + C::kOffQ + t * C::kFixTile;  // Q_t's tile, free once every MMA completed
      if (ok) {
        tc_fence_after_sync();
#pragma unroll
        for (int ch = 0; ch < C::D / 32; ++ch) {
          uint32_t v[32];
          tmem_ld_x32(tmem + lane_addr + C::kColQ(t) + ch * 32, v);
          tmem_ld_wait();
          reg_fence_x32(v);
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            const int cidx = ch * 4 + q4;
            const int cb = cidx / 8, c = cidx % 8;
            const uint32_t addr = stage + cb * C::kFixBlock + r * 128 + ((c ^ (r & 7)) << 4);
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e)
              w[e] = pack_bf16x2(__uint_as_float(v[q4 * 8 + 2 * e]) * p.scale,
                                 __uint_as_float(v[q4 * 8 + 2 * e + 1]) * p.scale);
            st_shared_v4(addr, w[0], w[1], w[2], w[3]);
          }
        }
      }
      fence_proxy_async_smem();
      named_barrier_sync(1 + t, 128);
      if (r == 0 && ok && *wctx.abort_flag == 0u) {
#pragma unroll
        for (int cb = 0; cb < C::kColBlocks; ++cb)
          tma_store_3d(&tmdQ, stage + cb * C::kFixBlock, cb * 64, tile_row0, bh);
        tma_store_commit();
        tma_store_wait_read_all();
      }
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == C::kMmaWarp) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

#undef FA2_BWD_WAIT

// Host-side launch description.
struct BwdLaunch {
  CUtensorMap tmQ64, tmdO64, tmK128, tmV128, tmdK, tmdV;  // dK/dV kernel
  CUtensorMap tmQ128, tmdO128, tmK64, tmV64, tmdQ;        // dQ kernel
  BwdParams params;
  const void* o;
  const void* dout;
  const float* lse;
  float* nl2;
  float* dlt;
  float* dqacc;    // non-null: dQ by reduction (head dim 128)
  void* dq;        // bf16 dQ, written by the convert kernel when dqacc is set
  int causal;
  cudaStream_t stream;
};

}  // namespace fa2
