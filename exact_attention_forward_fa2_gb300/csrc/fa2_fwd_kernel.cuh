// FlashAttention-2 forward kernel for sm_103a (GB300).
//
// What it computes: for one (batch, head) and a pair of 128-row query tiles,
// the score block S = Q K_j^T against every visible key tile K_j, folded into a
// running online softmax (row max m, row sum l, rescale of the unnormalised O by
// exp(m_old - m_new)), O += P V_j, one divide by l at the end, and the row
// logsumexp L = m + log l.  ("From FlashAttention to FlashAttention 2",
// FlashAttention 2: What Changed and Layers 5-6; "FlashAttention-2 from PyTorch
// to Triton", the Triton kernel's inner loop; "Writing FlashAttention 2 in
// Triton", Steps 3-5.)
//
// How it maps to the GB300 SM (one CTA per SM, warp-specialised):
//   warps 0..4*kQTiles-1  softmax warpgroups; warpgroup t owns query tile t,
//                         thread r owns row r = TMEM lane r (the pages' "warps
//                         split along Q rows only", taken to one row per thread)
//   warp  4*kQTiles       MMA issuer (one thread): tcgen05.mma S = Q K^T into TMEM
//                         and O += P V with P read from TMEM
//   warp  4*kQTiles+1     TMA producer (one thread): Q once, K/V through
//                         kStages-deep rings guarded by mbarriers
// Shared-memory tiles are written by TMA with a 128-byte swizzle; fp32 V tiles
// (the B operand of P V, read MN-major as TF32) use the swizzle of 32-byte chunks
// that the tensor core expects for 32-bit MN-major operands.
// TMEM columns: S_t at [t*BN, t*BN + BN) for key tiles of BN keys (P overwrites it
// in place), O_t at [kQTiles*BN + t*W, ... + W), where W = D, or D + 16 when the
// P V GEMM also forms the row sum from a ones block in V.  With two query tiles
// the MMA warp alternates between them, so one tile's softmax overlaps the other
// tile's two GEMMs.
//
// Every mbarrier wait is bounded in time; a wait that runs out records an error
// code in a device status word, sets a CTA-local abort flag, and all roles wind
// down: in-flight copies and MMAs are waited for (again bounded), TMEM is freed.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

#include "sm103_ptx.cuh"

namespace fa2 {

// Arguments that are not tensor maps.
struct FwdParams {
  float* lse;           // [BH, M] fp32, written for rows < M
  int* status;          // sticky device status word (0 = ok)
  int M, N, BH;         // BH = B * H query heads
  int H;                // query heads per batch entry
  int group;            // query heads per key/value head (H / H_kv)
  int num_units;        // BH * ceil(M / (kQTiles * 128))
  int units_per_head;   // ceil(M / (kQTiles * 128))
  float scale_log2;     // softmax scale * log2(e)
  // split-KV: the key range is cut into num_splits slices of tiles_per_split key
  // tiles; with more than one slice each CTA writes a partial (O_s = its P V / l_s
  // in fp32, L_s = m_s + ln l_s) instead of O and L, merged by the combine kernel
  int num_splits;
  int tiles_per_split;
  float* o_part;        // [num_splits][BH][M][D] fp32 (num_splits > 1)
  float* l_part;        // [num_splits][BH][M] fp32 (num_splits > 1)
  // 1: a unit is the single query tile of two heads that read the same key/value
  // head (M <= 128 under grouped-query attention), instead of two query tiles of one
  // head, so that both tile slots of a CTA work and share the streamed K/V tiles
  int pair_heads;
  // causal order: query heads per group (>= 1); a group's units all launch before
  // the next group's, longest first within the group (see unit_of_block)
  int head_group;
  // score modifiers.  Window (read by the kWin instantiations): key j is visible
  // to query row i iff i - win_left <= j <= i + win_right (the host folds the
  // causal bound into win_right and widens an unbounded side to cover every key).
  // Read by the kMod instantiations: s <- cap_out * tanh(s * cap_in) in log2 units
  // when cap_in > 0 (softcap); s <- s - log2(e) * slope * |i - j| when alibi is
  // not null (ALiBi)
  int win_left, win_right;
  float cap_in;         // scale / softcap, 0 = no softcap
  float cap_out;        // softcap * log2(e)
  const float* alibi;   // slopes, read at b * alibi_bstride + h; null = no ALiBi
  int alibi_bstride;
};

// The exponent base of a row moves only when the row max has grown by more than
// this many powers of two since the base was last set, so the O rescale (a TMEM
// load and store of the whole accumulator row, on the path to the next P V) is
// skipped on tiles where the max grows little.  Any base gives the same O and L in
// exact arithmetic, and it bounds P by 2^4, l by 16 N and the unnormalised O by
// 16 N max|v|.  The bound is kept small for precision: a P is rounded to bf16
// with a relative error of up to 2^-8 unless it is an exact power of two, and the
// base equal to the row max makes the largest weight exactly 1; a base lagging by
// up to 2^24 let the dominant weights of sharp rows (two keys of comparable score
// and far-apart values) carry that rounding, and the worst |dO| on rows with
// |O| < 2 of the sharp cross-attention workload rose from 8.7e-3 (bound 4) to
// 1.03e-2 (bound 24).  On N(0, 1) scores the row max rarely grows by more than 4
// after the first key tile, so the rescale stays rare there.
constexpr float kBaseLagLog2 = 4.0f;

// Device status codes (first failing wait site wins).
enum : int {
  kStatusOk = 0,
  kStatusTimeoutTmaK = 1,
  kStatusTimeoutTmaV = 2,
  kStatusTimeoutMmaQ = 3,
  kStatusTimeoutMmaK = 4,
  kStatusTimeoutMmaV = 5,
  kStatusTimeoutMmaP = 6,
  kStatusTimeoutSoftmaxS = 7,
  // 8 is retired: the O rescale needs no wait of its own (P_{j-1} V_{j-1} completed before S_j)
  kStatusTimeoutEpilogue = 9,
  kStatusTimeoutSoftmaxX = 10,  // the two halves of a score row exchanging max or sum
  kStatusSelfTest = 99,         // fa2_selftest_wait_timeout: a wait that was meant to run out
};

constexpr uint64_t kWaitTimeoutNs = 2000000000ull;  // 2 s; a real wait lasts microseconds

template <int D_, bool kBF16_, int kQTiles_, int kStages_, int kHalves_ = 1, int BN_ = 128>
struct FwdCfg {
  static constexpr int D = D_;
  static constexpr bool kBF16 = kBF16_;
  static constexpr int kQTiles = kQTiles_;
  static constexpr int kStages = kStages_;
  // softmax warpgroups per query tile: 1 (a thread owns a whole score row) or 2
  // (a thread owns 64 of its 128 keys; the two halves exchange the row max and
  // the row sum through shared memory)
  static constexpr int kHalves = kHalves_;
  static constexpr int BM = 128;  // query rows per tile = TMEM lanes = MMA M
  // keys per tile = MMA N of S: 128, or 112 at D = 128 so that the row-sum columns
  // fit in TMEM beside S and O of two query tiles (2 x (112 + 128 + 16) = 512)
  static constexpr int BN = BN_;
  static constexpr int kElem = kBF16 ? 2 : 4;
  static constexpr int kSwElems = 128 / kElem;              // elements in one 128-byte row
  static constexpr int kColBlocks = D / kSwElems;           // 128-byte column blocks per row
  static constexpr int kBlockBytes = 128 * 128;             // a query tile's block: 128 rows x 128 bytes
  static constexpr int kTileBytes = kColBlocks * kBlockBytes;  // a query (and O staging) tile
  static constexpr int kKVBlockBytes = BN * 128;            // a key/value tile's block: BN rows x 128 bytes
  static constexpr int kKTileBytes = kColBlocks * kKVBlockBytes;
  // D = 64, or D = 128 with 112-key tiles (one softmax warpgroup per tile): the
  // P V product also forms the row sum l.  Every V stage carries one more 128-byte
  // column block filled with ones, the P V GEMM runs with N = D + 16, and O_t holds
  // [O | 16 copies of l]: the sum of the rounded P the tensor core used, accumulated
  // in fp32 and rescaled with O, at no cost on the CUDA cores.  (With 128-key tiles
  // at D = 128 the 16 extra TMEM columns per tile do not fit beside S and O.)
  static constexpr bool kLOnes = kHalves == 1 && (D == 64 || BN < 128);
  static constexpr int kOW = kLOnes ? D + 16 : D;  // TMEM columns of O_t
  static constexpr int kVTileBytes = (kColBlocks + (kLOnes ? 1 : 0)) * kKVBlockBytes;
  static constexpr int kMmaK = 32 / kElem;                  // one MMA consumes 32 bytes of K
  static constexpr int kStepsS = D / kMmaK;
  static constexpr int kStepsPV = BN / kMmaK;
  static constexpr int kPCols = kBF16 ? BN / 2 : BN;        // TMEM columns holding P
  static constexpr int kSoftmaxWarps = 4 * kQTiles * kHalves;
  static constexpr int kMmaWarp = kSoftmaxWarps;
  static constexpr int kTmaWarp = kSoftmaxWarps + 1;
  static constexpr int kThreads = (kSoftmaxWarps + 2) * 32;
  static constexpr uint32_t kTmemCols = 512;
  __host__ __device__ static constexpr int kColS(int t) { return t * BN; }
  __host__ __device__ static constexpr int kColO(int t) { return kQTiles * BN + t * kOW; }
  // shared memory (offsets from a 1024-byte aligned base)
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kOffQ + kQTiles * kTileBytes;
  static constexpr int kOffV = kOffK + kStages * kKTileBytes;
  static constexpr int kOffBar = kOffV + kStages * kVTileBytes;
  static constexpr int kNumBars = 4 * kQTiles + 3 * kStages + 1 + (kHalves == 2 ? kQTiles : 0);
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  // exchange buffer of the two halves: [2 parities][kQTiles][2 halves][128 rows] floats
  static constexpr int kOffX = kOffMisc + 16;
  static constexpr int kXBytes = kHalves == 2 ? 2 * kQTiles * 2 * 128 * 4 : 0;
  static constexpr int kSmemBytes = kOffX + kXBytes + 1024;
  // barrier indices
  static constexpr int kBarQ = 0;
  static constexpr int kBarKFull = kBarQ + kQTiles;
  static constexpr int kBarFree = kBarKFull + kStages;
  static constexpr int kBarVFull = kBarFree + kStages;
  static constexpr int kBarSFull = kBarVFull + kStages;
  static constexpr int kBarPFull = kBarSFull + kQTiles;
  static constexpr int kBarOFull = kBarPFull + kQTiles;
  static constexpr int kBarMmaDone = kBarOFull + kQTiles;
  static constexpr int kBarX = kBarMmaDone + 1;  // per tile: both halves posted (kHalves == 2)
  static constexpr uint32_t kIdescS = ptx::make_idesc(kBF16, false, BM, BN);
  static constexpr uint32_t kIdescPV = ptx::make_idesc(kBF16, true, BM, kOW);

  static_assert(D % kSwElems == 0, "head dim must fill whole 128-byte rows");
  static_assert(kQTiles * (BN + kOW) <= 512, "TMEM budget");
  static_assert(BN == 128 || (BN == 112 && D == 128 && kBF16 && kHalves == 1),
                "112-key tiles: bf16, D = 128, one warpgroup per query tile");
  static_assert(kSmemBytes <= 232448, "shared memory budget");
  static_assert(kStepsS % 4 == 0 || kStepsS < 4, "K steps per 128-byte block");
  static_assert(kHalves == 1 || kHalves == 2, "one or two softmax warpgroups per query tile");
};

// Work decode and per-tile key-tile counts (shared by all roles).
struct Unit {
  int bh;    // flattened batch * heads index
  int pair;  // which group of kQTiles query tiles within the head
};

// Causal units are launched longest first (largest query offset, heads
// interleaved) so the tail of the grid holds the short ones, group of heads by
// group of heads: the host sizes a group so that its keys and values fit in a
// share of L2, so the CTAs in flight re-read K/V tiles from L2 instead of HBM.
// Non-causal units keep one head's query tiles adjacent so its K/V stay hot in L2.
__device__ __forceinline__ Unit unit_of_block(const FwdParams& p, bool causal, int b) {
  Unit u;
  if (p.pair_heads) {  // every unit is one tile long: any order
    u.bh = 2 * b;
    u.pair = 0;
    return u;
  }
  if (causal) {
    const int per_group = p.head_group * p.units_per_head;
    const int g = b / per_group;
    const int r = b - g * per_group;
    const int h0 = g * p.head_group;
    const int gh = min(p.head_group, p.BH - h0);  // heads in this group (the last may be short)
    u.pair = p.units_per_head - 1 - r / gh;
    u.bh = h0 + r % gh;
  } else {
    u.bh = b / p.units_per_head;
    u.pair = b % p.units_per_head;
  }
  return u;
}

// Number of key tiles of BN keys the query tile starting at row0 must visit (0 = tile empty).
template <int BN>
__device__ __forceinline__ int kv_tiles_for(int row0, int M, int N, bool causal) {
  if (row0 >= M) return 0;
  const int total = (N + BN - 1) / BN;
  if (!causal) return total;
  const int last_row = min(row0 + 128, M) - 1;
  return min(total, last_row / BN + 1);
}

// Query tile t of a unit: its flat head and first row.
__device__ __forceinline__ int tile_head(const FwdParams& p, const Unit& u, int t) {
  return u.bh + (p.pair_heads ? t : 0);
}
__device__ __forceinline__ int tile_first_row(const FwdParams& p, const Unit& u, int t, int tiles_per_unit) {
  return (u.pair * tiles_per_unit + (p.pair_heads ? 0 : t)) * 128;
}

// Key tiles [first, first + count) that the query tile starting at row0 visits
// inside split `split` (key tiles [split*tps, +tps)); count 0 = nothing to do.
// Plain: every key tile, or up to the diagonal when causal; the first is the
// split's first tile.  kWin: the tiles holding keys [row0 - win_left,
// last row + win_right] (a sliding window; the causal bound is in win_right).
struct KvSpan {
  int first, count;
};

template <bool kWin, int BN>
__device__ __forceinline__ KvSpan kv_span(int row0, const FwdParams& p, bool causal, int split) {
  const int s0 = split * p.tiles_per_split;
  if constexpr (!kWin) {
    const int n = kv_tiles_for<BN>(row0, p.M, p.N, causal) - s0;
    return KvSpan{s0, max(0, min(n, p.tiles_per_split))};
  } else {
    KvSpan r{s0, 0};
    if (row0 >= p.M) return r;
    const int last_row = min(row0 + 128, p.M) - 1;
    const int first_key = max(0, row0 - p.win_left);
    const int last_key = min(p.N - 1, last_row + p.win_right);
    if (first_key > last_key) return r;
    const int lo = max(first_key / BN, s0), hi = min(last_key / BN + 1, s0 + p.tiles_per_split);
    if (hi > lo) {
      r.first = lo;
      r.count = hi - lo;
    }
    return r;
  }
}

// tanh on the special-function unit (tanh.approx.f32): one instruction per score.
// Measured on GB300 against fp64 tanh over [-8, 8] (2^22 points): largest absolute
// error 7.9e-6, so a softcap c moves a capped score by at most c * 7.9e-6 (4e-4 at
// c = 50), inside the L tolerance with room; it measured 22% faster on the causal
// softcap-50 workload than tanh formed from ex2 and a reciprocal (two MUFU
// operations and four packed FMA-pipe operations per pair of scores).
__device__ __forceinline__ float tanh_mufu(float x) {
  float y;
  asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

struct WaitCtx {
  volatile uint32_t* abort_flag;  // CTA-local
  int* status;                    // device-wide sticky status
};

// Bounded mbarrier wait.  False if the CTA is aborting or the wait ran out.
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, const WaitCtx& w,
                                             int code, uint64_t limit_ns = kWaitTimeoutNs) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = ptx::globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    if ((it & 63u) == 0) {
      if (*w.abort_flag) return false;
      if (ptx::globaltimer_ns() - t0 > limit_ns) {
        *w.abort_flag = 1u;
        atomicCAS(w.status, 0, code);
        return false;
      }
    }
  }
}

// Wind-down wait: ignores the abort flag, bounded in time only.
__device__ __forceinline__ void drain_bounded(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = ptx::globaltimer_ns();
  while (!ptx::mbar_try_wait(bar, parity)) {
    if (ptx::globaltimer_ns() - t0 > kWaitTimeoutNs) return;
  }
}

// Softmax role with two warpgroups per query tile (kHalves == 2): thread (r, h)
// owns keys [64h, 64h + 64) of score row r and O columns [hD/2, hD/2 + D/2).  The
// two halves agree on the exponent base through a bounded exchange of their
// partial row maxima (shared memory + an mbarrier per tile), so P of one row is
// scaled consistently for the P V product; at the end they add their partial
// row sums the same way.
template <class C, bool kCausal, bool kMod, bool kWin>
__device__ __forceinline__ void softmax_halves(const FwdParams& p, const CUtensorMap& tmO, Unit unit,
                                               int split, int kb, uint32_t base, uint32_t tmem,
                                               int warp, int lane, const WaitCtx& wctx) {
  using namespace ptx;
  constexpr int kC = C::BN / 2;  // score columns (keys) of this thread
  constexpr int kOC = C::D / 2;  // O columns of this thread
  auto bar = [&](int i) -> uint32_t { return base + C::kOffBar + 8u * static_cast<uint32_t>(i); };
  const int g = warp / 4;
  const int t = g % C::kQTiles;
  const int h = g / C::kQTiles;
  const int r = (warp % 4) * 32 + lane;  // row within the tile = TMEM lane
  const int tile_row0 = tile_first_row(p, unit, t, C::kQTiles);
  const int bh_t = tile_head(p, unit, t);
  const int row = tile_row0 + r;
  const KvSpan span = kv_span<kWin, C::BN>(tile_row0, p, kCausal, split);
  const int n_t = span.count;
  const uint32_t lane_addr = static_cast<uint32_t>((warp % 4) * 32) << 16;
  const uint32_t tS = tmem + lane_addr + C::kColS(t) + h * kC;              // S of this half
  const uint32_t tP = tmem + lane_addr + C::kColS(t) + h * (C::kPCols / 2);  // P of this half
  const uint32_t tO = tmem + lane_addr + C::kColO(t) + h * kOC;
  const uint32_t xbar = bar(C::kBarX + t);
  int xphase = 0;
  // post `mine`, wait (bounded) until the other half has posted, read its value
  auto exchange = [&](float mine, float& other) -> bool {
    const uint32_t slot = base + C::kOffX + static_cast<uint32_t>((((xphase & 1) * C::kQTiles + t) * 2 + h) * 128 + r) * 4u;
    const uint32_t peer = base + C::kOffX + static_cast<uint32_t>((((xphase & 1) * C::kQTiles + t) * 2 + (1 - h)) * 128 + r) * 4u;
    st_shared_f32(slot, mine);
    tc_fence_before_sync();
    mbar_arrive(xbar);
    const bool got = wait_bounded(xbar, static_cast<uint32_t>(xphase & 1), wctx, kStatusTimeoutSoftmaxX);
    tc_fence_after_sync();
    if (got) other = ld_shared_f32(peer);
    ++xphase;
    return got;
  };
  // With a softcap S holds tanh(s * cap_in) and the exponent step multiplies by
  // cap_out (the softcap in log2 units); otherwise S stays in raw q.k units.  The
  // ALiBi penalty is applied in the units S is held in.
  const bool capped = kMod && p.cap_in > 0.f;
  const float sl2 = capped ? p.cap_out : p.scale_log2;
  float slope_s = 0.f;
  if constexpr (kMod) {
    if (p.alibi != nullptr) {
      const float a = p.alibi[(bh_t / p.H) * p.alibi_bstride + bh_t % p.H];
      slope_s = a * (1.4426950408889634f / sl2);
    }
  }
  const uint64_t sl2x2 = pack_f32x2(sl2, sl2);
  float m_run = -INFINITY;  // exponent base in use (the same in both halves)
  float l_run = 0.f;        // this half's running sum of the rounded P
  bool ok = n_t > 0;

  for (int j = 0; ok && j < n_t; ++j) {
    ok = __all_sync(0xffffffffu, wait_bounded(bar(C::kBarSFull + t), j & 1, wctx, kStatusTimeoutSoftmaxS));
    if (!ok) break;
    tc_fence_after_sync();
    uint32_t v[2][32];
    tmem_ld_x32(tS, v[0]);
    tmem_ld_x32(tS + 32, v[1]);
    tmem_ld_wait();
    reg_fence_x32(v[0]);
    reg_fence_x32(v[1]);
    float s[kC];
#pragma unroll
    for (int c = 0; c < kC; ++c) s[c] = __uint_as_float(v[c / 32][c % 32]);
    const int key0 = ((kWin ? span.first : kb) + j) * C::BN;
    const int keyh = key0 + h * kC;  // key of this thread's column 0
    if constexpr (kMod) {
      if (capped) {
#pragma unroll
        for (int c = 0; c < kC; c += 2) {
          ptx::unpack_f32x2(ptx::fmul2(ptx::pack_f32x2(s[c], s[c + 1]), ptx::pack_f32x2(p.cap_in, p.cap_in)),
                            s[c], s[c + 1]);
          s[c] = tanh_mufu(s[c]);
          s[c + 1] = tanh_mufu(s[c + 1]);
        }
      }
      if (slope_s != 0.f) {
        const float d0 = static_cast<float>(keyh - row);
#pragma unroll
        for (int c = 0; c < kC; ++c) s[c] = fmaf(-slope_s, fabsf(d0 + static_cast<float>(c)), s[c]);
      }
    }
    if constexpr (kWin) {
      const bool boundary = (key0 + C::BN > p.N) || (key0 + C::BN - 1 > tile_row0 + p.win_right) ||
                            (key0 < tile_row0 + C::BM - 1 - p.win_left);
      if (boundary) {
        const int hi = min(p.N - 1, row + p.win_right) - keyh;
        const int lo = row - p.win_left - keyh;
#pragma unroll
        for (int c = 0; c < kC; ++c) s[c] = (c >= lo && c <= hi) ? s[c] : -INFINITY;
      }
    } else {
      const bool boundary = (key0 + C::BN > p.N) || (kCausal && key0 + C::BN - 1 > tile_row0);
      if (boundary) {
        int lim = p.N - 1 - keyh;
        if (kCausal) lim = min(lim, row - keyh);
#pragma unroll
        for (int c = 0; c < kC; ++c) s[c] = (c <= lim) ? s[c] : -INFINITY;
      }
    }
    // max of this half (four chains), then of the whole row through the exchange
    float mx[4] = {s[0], s[1], s[2], s[3]};
#pragma unroll
    for (int c = 4; c + 8 <= kC; c += 8) {
#pragma unroll
      for (int q = 0; q < 4; ++q) mx[q] = fmax3(mx[q], s[c + q], s[c + 4 + q]);
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) mx[q] = fmaxf(mx[q], s[kC - 4 + q]);
    const float mh = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
    float mo = -INFINITY;
    ok = __all_sync(0xffffffffu, exchange(mh, mo));
    if (!ok) break;
    const float m_tile = fmaxf(mh, mo) * sl2;
    const float m_new = fmaxf(m_run, m_tile);
    const bool rescale = (m_new - m_run) > kBaseLagLog2;
    const float m_use = rescale ? m_new : m_run;
    const float alpha = rescale ? ex2_approx(m_run - m_new) : 1.0f;
    const float neg_base = (m_use == -INFINITY) ? 0.f : -m_use;
    const uint64_t nb2 = pack_f32x2(neg_base, neg_base);
    uint64_t acc[4] = {0ull, 0ull, 0ull, 0ull};
    uint32_t pk[32];
#pragma unroll
    for (int i = 0; i < kC / 2; ++i) {
      const int c = 2 * i;
      float x0, x1;
      unpack_f32x2(ffma2(pack_f32x2(s[c], s[c + 1]), sl2x2, nb2), x0, x1);
      const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
      if constexpr (C::kBF16) {
        const uint32_t w = pack_bf16x2(p0, p1);
        pk[i] = w;
        acc[i % 4] = fadd2(acc[i % 4], pack_f32x2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u)));
      } else {
        const uint32_t r0 = round_tf32(p0), r1 = round_tf32(p1);
        s[c] = __uint_as_float(r0);
        s[c + 1] = __uint_as_float(r1);
        acc[i % 4] = fadd2(acc[i % 4], pack_f32x2(s[c], s[c + 1]));
      }
    }
    if constexpr (C::kBF16) {
      tmem_st_x32(tP, pk);  // 64 keys -> 32 columns of bf16x2
    } else {
      uint32_t q0[32], q1[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        q0[i] = __float_as_uint(s[i]);
        q1[i] = __float_as_uint(s[32 + i]);
      }
      tmem_st_x32(tP, q0);
      tmem_st_x32(tP + 32, q1);
    }
    float a0, a1, a2, a3, a4, a5, a6, a7;
    unpack_f32x2(acc[0], a0, a1);
    unpack_f32x2(acc[1], a2, a3);
    unpack_f32x2(acc[2], a4, a5);
    unpack_f32x2(acc[3], a6, a7);
    l_run = l_run * alpha + (((a0 + a1) + (a2 + a3)) + ((a4 + a5) + (a6 + a7)));
    if (j > 0 && __any_sync(0xffffffffu, rescale)) {
      // P_{j-1} V_{j-1} completed before S_j, which this thread waited for
      tc_fence_after_sync();
#pragma unroll
      for (int ch = 0; ch < kOC / 32; ++ch) {
        uint32_t o[32];
        tmem_ld_x32(tO + ch * 32, o);
        tmem_ld_wait();
        reg_fence_x32(o);
#pragma unroll
        for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
        tmem_st_x32(tO + ch * 32, o);
      }
    }
    tmem_st_wait();
    tc_fence_before_sync();
    mbar_arrive(bar(C::kBarPFull + t));
    m_run = m_use;
  }

  // ------------------------------------------------------------ epilogue
  if (p.num_splits > 1) {
    if (tile_row0 < p.M) {
      if (n_t > 0 && ok)
        ok = __all_sync(0xffffffffu, wait_bounded(bar(C::kBarOFull + t), n_t > 0 ? 0 : 1, wctx, kStatusTimeoutEpilogue));
      float lo_sum = 0.f;
      if (n_t > 0 && ok) ok = __all_sync(0xffffffffu, exchange(l_run, lo_sum));
      const float l_tot = l_run + lo_sum;
      const int64_t prow = (static_cast<int64_t>(split) * p.BH + bh_t) * p.M + row;
      float4* op = reinterpret_cast<float4*>(p.o_part + prow * C::D + h * kOC);
      if (n_t > 0 && ok) {
        tc_fence_after_sync();
        const float inv_l = l_tot > 0.f ? 1.0f / l_tot : 0.f;
#pragma unroll
        for (int ch = 0; ch < kOC / 32; ++ch) {
          uint32_t v[32];
          tmem_ld_x32(tO + ch * 32, v);
          tmem_ld_wait();
          reg_fence_x32(v);
          if (row < p.M) {
#pragma unroll
            for (int q4 = 0; q4 < 8; ++q4)
              op[ch * 8 + q4] = make_float4(__uint_as_float(v[q4 * 4 + 0]) * inv_l, __uint_as_float(v[q4 * 4 + 1]) * inv_l,
                                            __uint_as_float(v[q4 * 4 + 2]) * inv_l, __uint_as_float(v[q4 * 4 + 3]) * inv_l);
          }
        }
        if (row < p.M && h == 0) p.l_part[prow] = (m_run + lg2_approx(l_tot)) * 0.69314718055994530942f;
      } else if (n_t == 0 && row < p.M) {
#pragma unroll
        for (int q4 = 0; q4 < kOC / 4; ++q4) op[q4] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (h == 0) p.l_part[prow] = -INFINITY;
      }
    }
  } else if (n_t > 0 || (kWin && tile_row0 < p.M)) {
    if (ok)
      ok = __all_sync(0xffffffffu, wait_bounded(bar(C::kBarOFull + t), n_t > 0 ? 0 : 1, wctx, kStatusTimeoutEpilogue));
    float lo_sum = 0.f;
    if (ok) ok = __all_sync(0xffffffffu, exchange(l_run, lo_sum));
    const float l_tot = l_run + lo_sum;
    const uint32_t stage = base + C::kOffQ + t * C::kTileBytes;
    constexpr int kChunks = C::kColBlocks * 8;  // 16-byte chunks of one O row
    if (kWin && n_t == 0) {
#pragma unroll
      for (int cidx = h * kChunks / 2; cidx < (h + 1) * kChunks / 2; ++cidx)
        st_shared_v4(stage + (cidx / 8) * C::kBlockBytes + r * 128 + (cidx % 8) * 16, 0u, 0u, 0u, 0u);
      if (row < p.M && h == 0) p.lse[static_cast<int64_t>(bh_t) * p.M + row] = -INFINITY;
    } else if (ok) {
      tc_fence_after_sync();
      const float inv_l = l_tot > 0.f ? 1.0f / l_tot : 0.f;
#pragma unroll
      for (int chl = 0; chl < kOC / 32; ++chl) {
        const int ch = h * (kOC / 32) + chl;  // 32-column group of the whole O row
        uint32_t v[32];
        tmem_ld_x32(tO + chl * 32, v);
        tmem_ld_wait();
        reg_fence_x32(v);
        if constexpr (C::kBF16) {
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            const int cidx = ch * 4 + q4;
            const int cb = cidx / 8, c = cidx % 8;
            const uint32_t addr = stage + cb * C::kBlockBytes + r * 128 + ((c ^ (r & 7)) << 4);
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e)
              w[e] = pack_bf16x2(__uint_as_float(v[q4 * 8 + 2 * e]) * inv_l, __uint_as_float(v[q4 * 8 + 2 * e + 1]) * inv_l);
            st_shared_v4(addr, w[0], w[1], w[2], w[3]);
          }
        } else {
#pragma unroll
          for (int q8 = 0; q8 < 8; ++q8) {
            const int cb = ch, c = q8;
            const uint32_t addr = stage + cb * C::kBlockBytes + r * 128 + ((c ^ (r & 7)) << 4);
            st_shared_v4(addr, __float_as_uint(__uint_as_float(v[q8 * 4 + 0]) * inv_l),
                         __float_as_uint(__uint_as_float(v[q8 * 4 + 1]) * inv_l),
                         __float_as_uint(__uint_as_float(v[q8 * 4 + 2]) * inv_l),
                         __float_as_uint(__uint_as_float(v[q8 * 4 + 3]) * inv_l));
          }
        }
      }
      if (row < p.M && h == 0)
        p.lse[static_cast<int64_t>(bh_t) * p.M + row] = (m_run + lg2_approx(l_tot)) * 0.69314718055994530942f;
    }
    fence_proxy_async_smem();
    named_barrier_sync(1 + t, 256);
    if (r == 0 && h == 0 && *wctx.abort_flag == 0u) {
#pragma unroll
      for (int cb = 0; cb < C::kColBlocks; ++cb)
        tma_store_3d(&tmO, stage + cb * C::kBlockBytes, cb * C::kSwElems, tile_row0, bh_t);
      tma_store_commit();
      tma_store_wait_read_all();
    }
  }
}

// One key tile of a query tile's online softmax, one warpgroup per tile (thread
// r owns row r = TMEM lane r): S row from TMEM, score modifiers, mask, row max, the
// exponent base (moved only past kBaseLagLog2), P = exp2(s*sl2 - base) rounded to
// the P V operand type and written over S, the row sum (when the softmax forms
// it), the rescale of O when the base moved, then the P barrier.  The caller has
// waited for S (and fenced); key0 is the tile's first key, not_first is false on
// a tile's first key tile of the item.
template <class C, bool kCausal, bool kMod, bool kWin>
__device__ __forceinline__ void softmax_step(const FwdParams& p, uint32_t tS, uint32_t tO, uint32_t pbar,
                                             int key0, int tile_row0, int row, bool capped, float slope_s,
                                             float sl2, uint64_t sl2x2, bool not_first, float& m_run,
                                             float& l_run) {
  using namespace ptx;
  tc_fence_after_sync();
  // the whole S row of this thread: every TMEM load in flight, one wait (32
  // columns per load; a 112-key row ends with a 16-column load)
  constexpr int kLd = (C::BN + 31) / 32;
  uint32_t v[kLd][32];
#pragma unroll
  for (int ch = 0; ch < C::BN / 32; ++ch) tmem_ld_x32(tS + ch * 32, v[ch]);
  if constexpr (C::BN % 32 == 16)
    tmem_ld_x16(tS + (C::BN / 32) * 32, *reinterpret_cast<uint32_t(*)[16]>(&v[kLd - 1][0]));
  tmem_ld_wait();
#pragma unroll
  for (int ch = 0; ch < C::BN / 32; ++ch) reg_fence_x32(v[ch]);
  if constexpr (C::BN % 32 == 16) reg_fence_x16(*reinterpret_cast<uint32_t(*)[16]>(&v[kLd - 1][0]));
  static_assert(C::BN % 32 == 0 || C::BN % 32 == 16, "S rows load in 32- and 16-column pieces");
  float s[C::BN];
#pragma unroll
  for (int c = 0; c < C::BN; ++c) s[c] = __uint_as_float(v[c / 32][c % 32]);
  if constexpr (kMod) {
    // score modifiers: softcap (into log2 units), then the ALiBi distance penalty
    if (capped) {
#pragma unroll
      for (int c = 0; c < C::BN; ++c) s[c] = p.cap_out * tanh_mufu(s[c] * p.cap_in);
    }
    if (slope_s != 0.f) {
      const float d0 = static_cast<float>(key0 - row);
#pragma unroll
      for (int c = 0; c < C::BN; ++c) s[c] = fmaf(-slope_s, fabsf(d0 + static_cast<float>(c)), s[c]);
    }
  }
  if constexpr (kWin) {
    // window mask, on tiles that cross N or either window edge of some row
    const bool boundary = (key0 + C::BN > p.N) || (key0 + C::BN - 1 > tile_row0 + p.win_right) ||
                          (key0 < tile_row0 + C::BM - 1 - p.win_left);
    if (boundary) {
      const int hi = min(p.N - 1, row + p.win_right) - key0;
      const int lo = row - p.win_left - key0;
#pragma unroll
      for (int c = 0; c < C::BN; ++c) s[c] = (c >= lo && c <= hi) ? s[c] : -INFINITY;
    }
  } else {
    // mask keys past N and, when causal, keys after this row (boundary tiles only)
    const bool boundary = (key0 + C::BN > p.N) || (kCausal && key0 + C::BN - 1 > tile_row0);
    if (boundary) {
      int lim = p.N - 1 - key0;
      if (kCausal) lim = min(lim, row - key0);
#pragma unroll
      for (int c = 0; c < C::BN; ++c) s[c] = (c <= lim) ? s[c] : -INFINITY;
    }
  }
  // row max: four independent chains of 3-input max over s[4..BN-5], then the
  // last four columns
  float mx[4] = {s[0], s[1], s[2], s[3]};
#pragma unroll
  for (int c = 4; c + 8 <= C::BN; c += 8) {
#pragma unroll
    for (int q = 0; q < 4; ++q) mx[q] = fmax3(mx[q], s[c + q], s[c + 4 + q]);
  }
  static_assert(C::BN % 8 == 0, "the max chains cover s[0..3], pairs of 4, then s[BN-4..BN-1]");
  static_assert(C::BN % 64 == 0 || C::BN % 64 == 48, "P is stored in pieces of 64 keys and one of 48");
#pragma unroll
  for (int q = 0; q < 4; ++q) mx[q] = fmaxf(mx[q], s[C::BN - 4 + q]);
  const float m_tile = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])) * sl2;
  const float m_new = fmaxf(m_run, m_tile);
  // Move the exponent base only when the max grew by more than kBaseLagLog2:
  // the result is exact for any base, and skipping the rescale keeps O in TMEM
  // untouched on most tiles.  (-inf) - (-inf) is NaN, so an empty row stays put.
  const bool rescale = (m_new - m_run) > kBaseLagLog2;
  const float m_use = rescale ? m_new : m_run;
  const float alpha = rescale ? ex2_approx(m_run - m_new) : 1.0f;
  const float neg_base = (m_use == -INFINITY) ? 0.f : -m_use;
  const uint64_t nb2 = pack_f32x2(neg_base, neg_base);
  // P = exp2(s*sl2 - base), rounded to the P.V operand type.  l sums the
  // rounded values, so O = sum(P v) / sum(P) is an exact convex combination
  // of V rows with the weights the tensor core actually used.
  uint64_t acc[4] = {0ull, 0ull, 0ull, 0ull};  // packed pairs of partial sums
#pragma unroll
  for (int h = 0; h < (C::BN + 63) / 64; ++h) {  // pieces of 64 keys (the last of a 112-key row: 48)
    uint32_t pk[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const int c = h * 64 + 2 * i;
      if (c >= C::BN) break;
      float x0, x1;
      unpack_f32x2(ffma2(pack_f32x2(s[c], s[c + 1]), sl2x2, nb2), x0, x1);
      const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
      if constexpr (C::kBF16) {
        const uint32_t w = pack_bf16x2(p0, p1);
        pk[i] = w;
        if constexpr (!C::kLOnes)
          acc[i % 4] = fadd2(acc[i % 4], pack_f32x2(__uint_as_float(w << 16),
                                                    __uint_as_float(w & 0xffff0000u)));
      } else if constexpr (C::kLOnes) {
        // fp32 P goes to TMEM as it is: the tensor core reads it as TF32 for the
        // P V product and for the ones columns alike, so l is the sum of exactly
        // the weights the product used (an explicit rounding measured 16% slower)
        s[c] = p0;
        s[c + 1] = p1;
      } else {
        const uint32_t r0 = round_tf32(p0), r1 = round_tf32(p1);
        s[c] = __uint_as_float(r0);
        s[c + 1] = __uint_as_float(r1);
        acc[i % 4] = fadd2(acc[i % 4], pack_f32x2(s[c], s[c + 1]));
      }
    }
    if constexpr (C::kBF16) {
      if (C::BN - h * 64 >= 64) {
        tmem_st_x32(tS + h * 32, pk);  // 64 keys -> 32 columns of bf16x2
      } else {                         // 48 keys -> 24 columns
        tmem_st_x16(tS + h * 32, *reinterpret_cast<const uint32_t(*)[16]>(&pk[0]));
        tmem_st_x8(tS + h * 32 + 16, *reinterpret_cast<const uint32_t(*)[8]>(&pk[16]));
      }
    } else {
      uint32_t q0[32], q1[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        q0[i] = __float_as_uint(s[h * 64 + i]);
        q1[i] = __float_as_uint(s[h * 64 + 32 + i]);
      }
      tmem_st_x32(tS + h * 64, q0);
      tmem_st_x32(tS + h * 64 + 32, q1);
    }
  }
  if constexpr (!C::kLOnes) {
    float a0, a1, a2, a3, a4, a5, a6, a7;
    unpack_f32x2(acc[0], a0, a1);
    unpack_f32x2(acc[1], a2, a3);
    unpack_f32x2(acc[2], a4, a5);
    unpack_f32x2(acc[3], a6, a7);
    l_run = l_run * alpha + (((a0 + a1) + (a2 + a3)) + ((a4 + a5) + (a6 + a7)));
  }
  if (not_first && __any_sync(0xffffffffu, rescale)) {
    // O_t *= alpha.  P_{j-1} V_{j-1} has landed: the MMA warp issued it before
    // S_j, and a commit completes only after every earlier MMA.
    tc_fence_after_sync();
    // every load of the row in flight at once, one wait
    uint32_t o[C::D / 32][32];
    uint32_t ol[16];  // the row sum columns, which scale with O
#pragma unroll
    for (int ch = 0; ch < C::D / 32; ++ch) tmem_ld_x32(tO + ch * 32, o[ch]);
    if constexpr (C::kLOnes) tmem_ld_x16(tO + C::D, ol);
    tmem_ld_wait();
    const uint64_t alpha2 = pack_f32x2(alpha, alpha);
#pragma unroll
    for (int ch = 0; ch < C::D / 32; ++ch) {
      reg_fence_x32(o[ch]);
#pragma unroll
      for (int i = 0; i < 32; i += 2) {
        float a, b;
        unpack_f32x2(fmul2(pack_f32x2(__uint_as_float(o[ch][i]), __uint_as_float(o[ch][i + 1])), alpha2), a, b);
        o[ch][i] = __float_as_uint(a);
        o[ch][i + 1] = __float_as_uint(b);
      }
      tmem_st_x32(tO + ch * 32, o[ch]);
    }
    if constexpr (C::kLOnes) {
      reg_fence_x16(ol);
#pragma unroll
      for (int i = 0; i < 16; ++i) ol[i] = __float_as_uint(__uint_as_float(ol[i]) * alpha);
      tmem_st_x16(tO + C::D, ol);
    }
  }
  tmem_st_wait();
  tc_fence_before_sync();
  mbar_arrive(pbar);
  m_run = m_use;}

template <class C, bool kCausal, bool kMod, bool kWin>
__global__ void __launch_bounds__(C::kThreads, 1)
  fa2_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                 const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                 const FwdParams p) {
  using namespace ptx;
extern __shared__ uint8_t smem_raw[];
const uint32_t raw = smem_u32(smem_raw);
const uint32_t base = (raw + 1023u) & ~1023u;
uint8_t* gbase = smem_raw + (base - raw);
volatile uint32_t* misc = reinterpret_cast<volatile uint32_t*>(gbase + C::kOffMisc);
// misc[0] TMEM base address, misc[1] abort flag, misc[2] status at CTA start

const int warp = static_cast<int>(threadIdx.x) / 32;
const int lane = static_cast<int>(threadIdx.x) % 32;
auto bar = [&](int i) -> uint32_t { return base + C::kOffBar + 8u * static_cast<uint32_t>(i); };

const int split = static_cast<int>(blockIdx.x) % p.num_splits;
const int kb = split * p.tiles_per_split;  // first key tile of this CTA's split
const Unit unit = unit_of_block(p, kCausal, static_cast<int>(blockIdx.x) / p.num_splits);
const int bh = unit.bh;
// key/value head read by this query head (grouped-query attention, "From
// FlashAttention to FlashAttention 2", Layer 8: h_kv = h / (H / H_kv))
const int bh_kv = (bh / p.H) * (p.H / p.group) + (bh % p.H) / p.group;
// Query tile t visits key tiles [kt0[t], kt0[t] + nkv[t]); the CTA streams key
// tiles ks, ks + 1, ..., ks + n_max - 1 and tile t uses stream positions
// [jb[t], jb[t] + nkv[t]).  Without a window every tile starts at the split's
// first key tile, so jb is 0.
int row0[C::kQTiles], kt0[C::kQTiles], nkv[C::kQTiles], jb[C::kQTiles];
int ks = kb, n_max = 0;
#pragma unroll
for (int t = 0; t < C::kQTiles; ++t) {
  row0[t] = tile_first_row(p, unit, t, C::kQTiles);
  const KvSpan sp = kv_span<kWin, C::BN>(row0[t], p, kCausal, split);
  kt0[t] = sp.first;
  nkv[t] = sp.count;
  jb[t] = 0;
  n_max = max(n_max, nkv[t]);
}
if constexpr (kWin) {
  int lo = 0x7fffffff, hi = 0;
#pragma unroll
  for (int t = 0; t < C::kQTiles; ++t)
    if (nkv[t] > 0) {
      lo = min(lo, kt0[t]);
      hi = max(hi, kt0[t] + nkv[t]);
    }
  ks = hi > 0 ? lo : 0;
  n_max = hi > 0 ? hi - lo : 0;
#pragma unroll
  for (int t = 0; t < C::kQTiles; ++t) jb[t] = kt0[t] - ks;
}

// ------------------------------------------------------------ set-up
// Thread 0 also issues the query tiles' loads, right after the barrier inits
// and before it reads the status word, so that they overlap that read, the
// TMEM allocation and the ones fill (measured: +1% on the causal
// 2x16x8192x8192x128 forward, +3% on the TF32 one), and with kEarlyKV the
// first K/V ring stage's as well, which otherwise waits for the CTA-wide
// barrier (measured: +1.4% at bf16 D = 64 causal, +1.3% on the sharp
// 1000 x 3000 cross-attention, +0.7% TF32; -0.3% at bf16 D = 128 causal, which
// keeps the later issue).  A CTA that then skips waits for them at the end,
// before its shared memory is released.
constexpr bool kEarlyKV = !(kCausal && C::D == 128);
if (threadIdx.x == 0) {
  for (int t = 0; t < C::kQTiles; ++t) {
    mbar_init(bar(C::kBarQ + t), 1);
    mbar_init(bar(C::kBarSFull + t), 1);
    mbar_init(bar(C::kBarPFull + t), 128 * C::kHalves);
    if (C::kHalves == 2) mbar_init(bar(C::kBarX + t), 256);
    mbar_init(bar(C::kBarOFull + t), 1);
  }
  for (int s = 0; s < C::kStages; ++s) {
    mbar_init(bar(C::kBarKFull + s), 1);
    mbar_init(bar(C::kBarFree + s), 1);
    mbar_init(bar(C::kBarVFull + s), 1);
  }
  mbar_init(bar(C::kBarMmaDone), 1);
  fence_mbar_init();
  {
    const uint64_t pol_q = l2_policy_evict_first();
#pragma unroll
    for (int t = 0; t < C::kQTiles; ++t) {
      if (nkv[t] == 0) continue;
      mbar_arrive_expect_tx(bar(C::kBarQ + t), C::kTileBytes);
#pragma unroll
      for (int cb = 0; cb < C::kColBlocks; ++cb)
        tma_load_3d_hint(base + C::kOffQ + t * C::kTileBytes + cb * C::kBlockBytes, &tmQ, bar(C::kBarQ + t),
                         cb * C::kSwElems, row0[t], tile_head(p, unit, t), pol_q);
    }
    if (kEarlyKV && n_max > 0) {  // stage 0 of the K/V ring
      const uint64_t pol_kv = l2_policy_evict_last();
      mbar_arrive_expect_tx(bar(C::kBarKFull), C::kKTileBytes);
#pragma unroll
      for (int cb = 0; cb < C::kColBlocks; ++cb)
        tma_load_3d_hint(base + C::kOffK + cb * C::kKVBlockBytes, &tmK, bar(C::kBarKFull), cb * C::kSwElems,
                         ks * C::BN, bh_kv, pol_kv);
      mbar_arrive_expect_tx(bar(C::kBarVFull), C::kKTileBytes);
#pragma unroll
      for (int cb = 0; cb < C::kColBlocks; ++cb)
        tma_load_3d_hint(base + C::kOffV + cb * C::kKVBlockBytes, &tmV, bar(C::kBarVFull), cb * C::kSwElems,
                         ks * C::BN, bh_kv, pol_kv);
    }
  }
  misc[1] = 0u;
  misc[2] = static_cast<uint32_t>(*reinterpret_cast<volatile int*>(p.status));
}
if (warp == C::kTmaWarp && lane == 0) {
  prefetch_tensormap(&tmQ);
  prefetch_tensormap(&tmK);
  prefetch_tensormap(&tmV);
  prefetch_tensormap(&tmO);
}
if (warp == C::kMmaWarp) {
  tmem_alloc(base + C::kOffMisc, C::kTmemCols);
  tmem_relinquish_alloc_permit();
}
if constexpr (C::kLOnes) {
  // the ones block of every V stage (TMA writes only the blocks before it)
  const uint32_t one2 = C::kBF16 ? 0x3F803F80u : 0x3F800000u;
  for (int i = static_cast<int>(threadIdx.x); i < C::kStages * (C::kKVBlockBytes / 16); i += C::kThreads) {
    const int st = i / (C::kKVBlockBytes / 16), o = i % (C::kKVBlockBytes / 16);
    st_shared_v4(base + C::kOffV + st * C::kVTileBytes + C::kColBlocks * C::kKVBlockBytes + o * 16, one2, one2,
                 one2, one2);
  }
  fence_proxy_async_smem();  // visible to the tensor core (async proxy)
}
tc_fence_before_sync();
__syncthreads();
tc_fence_after_sync();
const uint32_t tmem = misc[0];
const bool skip = misc[2] != 0u;  // an earlier launch failed: do nothing
const WaitCtx wctx{misc + 1, p.status};

if (!skip && warp == C::kTmaWarp) {
  // ---------------------------------------------------------- TMA producer
  if (lane == 0) {
    const uint64_t pol_kv = l2_policy_evict_last();
    // K/V tiles whose loads were issued (thread 0 issued the query tiles', and
    // with kEarlyKV stage 0's)
    int issued = kEarlyKV && n_max > 0 ? 1 : 0;
    for (int j = issued; j < n_max; ++j) {
      const int s = j % C::kStages;
      const uint32_t use = static_cast<uint32_t>(j / C::kStages);
      // K_j replaces K_{j-S}, free after MMA round j-S; V_j replaces V_{j-S}, free
      // after round j-S+1 (which ran P V on it).  One barrier per round.
      if (use > 0 && !wait_bounded(bar(C::kBarFree + s), (use - 1) & 1u, wctx, kStatusTimeoutTmaK))
        break;
      mbar_arrive_expect_tx(bar(C::kBarKFull + s), C::kKTileBytes);
#pragma unroll
      for (int cb = 0; cb < C::kColBlocks; ++cb)
        tma_load_3d_hint(base + C::kOffK + s * C::kKTileBytes + cb * C::kKVBlockBytes, &tmK,
                         bar(C::kBarKFull + s), cb * C::kSwElems, (ks + j) * C::BN, bh_kv, pol_kv);
      if (use > 0 && !wait_bounded(bar(C::kBarFree + (j - C::kStages + 1) % C::kStages),
                                   static_cast<uint32_t>((j - C::kStages + 1) / C::kStages) & 1u, wctx,
                                   kStatusTimeoutTmaV)) {
        issued = -(j + 1);  // K_j issued, V_j not
        break;
      }
      mbar_arrive_expect_tx(bar(C::kBarVFull + s), C::kKTileBytes);
#pragma unroll
      for (int cb = 0; cb < C::kColBlocks; ++cb)
        tma_load_3d_hint(base + C::kOffV + s * C::kVTileBytes + cb * C::kKVBlockBytes, &tmV,
                         bar(C::kBarVFull + s), cb * C::kSwElems, (ks + j) * C::BN, bh_kv, pol_kv);
      issued = j + 1;
    }
    if (*wctx.abort_flag) {
      // wind down: every issued copy must land before the CTA's smem is released
      const int k_done = issued >= 0 ? issued : -issued;
      const int v_done = issued >= 0 ? issued : -issued - 1;
      for (int t = 0; t < C::kQTiles; ++t)
        if (nkv[t] > 0) drain_bounded(bar(C::kBarQ + t), 0);
      for (int j = max(0, k_done - C::kStages); j < k_done; ++j)
        drain_bounded(bar(C::kBarKFull + j % C::kStages), (j / C::kStages) & 1);
      for (int j = max(0, v_done - C::kStages); j < v_done; ++j)
        drain_bounded(bar(C::kBarVFull + j % C::kStages), (j / C::kStages) & 1);
    }
  }
  __syncwarp();
} else if (!skip && warp == C::kMmaWarp) {
  // ---------------------------------------------------------- MMA issuer
  if (lane == 0) {
    // Descriptor words of the operand tiles.  The low word holds the start
    // address >> 4, so a K step or another ring stage is one 32-bit add to it;
    // fewer instructions between MMAs keep the tensor core's queue fed while
    // the softmax warps share this warp's scheduler.
    const uint64_t qk_desc = smem_desc_sw128(base, 16, 1024);
    const uint32_t qk_lo0 = static_cast<uint32_t>(qk_desc), qk_hi = static_cast<uint32_t>(qk_desc >> 32);
    const uint64_t v_desc = C::kBF16 ? smem_desc(base + C::kOffV, C::kKVBlockBytes, 1024, kLayoutSw128)
                                     : smem_desc(base + C::kOffV, C::kKVBlockBytes, 512, kLayoutSw128Atom32);
    const uint32_t v_lo0 = static_cast<uint32_t>(v_desc), v_hi = static_cast<uint32_t>(v_desc >> 32);
    bool ok = true;
#pragma unroll
    for (int t = 0; t < C::kQTiles; ++t)
      if (ok && nkv[t] > 0) ok = wait_bounded(bar(C::kBarQ + t), 0, wctx, kStatusTimeoutMmaQ);
    for (int j = 0; ok && j <= n_max; ++j) {
      const int s = j % C::kStages;
      bool v_ready = false, k_ready = false;
#pragma unroll
      for (int t = 0; t < C::kQTiles; ++t) {
        if ((kWin ? j - 1 >= jb[t] : j >= 1) && j - 1 < jb[t] + nkv[t]) {
          // O_t += P_t V_{j-1}
          const int jp = j - 1;
          const int sv = jp % C::kStages;
          // V first: it has normally landed long ago, and checking it while P is
          // still being written keeps that check off the path from P to the MMAs
          if (!v_ready) {
            ok = wait_bounded(bar(C::kBarVFull + sv), (jp / C::kStages) & 1, wctx, kStatusTimeoutMmaV);
            if (!ok) break;
            v_ready = true;
          }
          ok = wait_bounded(bar(C::kBarPFull + t), (kWin ? jp - jb[t] : jp) & 1, wctx, kStatusTimeoutMmaP);
          if (!ok) break;
          tc_fence_after_sync();
          const uint32_t v_lo = v_lo0 + static_cast<uint32_t>(sv) * (C::kVTileBytes >> 4);
          const int jp0 = kWin ? jb[t] : 0;  // first P V of this tile overwrites O
#pragma unroll
          for (int kk = 0; kk < C::kStepsPV; ++kk) {
            // B = V rows [kk*kMmaK, +kMmaK), all D columns, MN-major
            const uint64_t bdesc = desc_from_words(v_lo + (kk * C::kMmaK * 128 >> 4), v_hi);
            const uint32_t a_tmem = tmem + C::kColS(t) + kk * 8;
            if constexpr (C::kBF16)
              mma_f16_ts(tmem + C::kColO(t), a_tmem, bdesc, C::kIdescPV, (jp > jp0 || kk > 0) ? 1u : 0u);
            else
              mma_tf32_ts(tmem + C::kColO(t), a_tmem, bdesc, C::kIdescPV, (jp > jp0 || kk > 0) ? 1u : 0u);
          }
          // O_t is read by the epilogue after its last P V; a rescale on the way
          // needs no barrier of its own (it follows S_{jp+1}, issued after this)
          if (jp == jb[t] + nkv[t] - 1) tc_commit(bar(C::kBarOFull + t));
        }
        if ((kWin ? j >= jb[t] : true) && j < jb[t] + nkv[t]) {
          // S_t = Q_t K_j^T
          if (!k_ready) {
            ok = wait_bounded(bar(C::kBarKFull + s), (j / C::kStages) & 1, wctx, kStatusTimeoutMmaK);
            if (!ok) break;
            k_ready = true;
            tc_fence_after_sync();
          }
          const uint32_t q_lo = qk_lo0 + ((C::kOffQ + t * C::kTileBytes) >> 4);
          const uint32_t k_lo = qk_lo0 + ((C::kOffK >> 4) + static_cast<uint32_t>(s) * (C::kKTileBytes >> 4));
#pragma unroll
          for (int kk = 0; kk < C::kStepsS; ++kk) {
            const uint32_t off = ((kk / 4) * C::kBlockBytes + (kk % 4) * 32) >> 4;
            const uint32_t koff = ((kk / 4) * C::kKVBlockBytes + (kk % 4) * 32) >> 4;
            const uint64_t adesc = desc_from_words(q_lo + off, qk_hi);
            const uint64_t bdesc = desc_from_words(k_lo + koff, qk_hi);
            if constexpr (C::kBF16)
              mma_f16_ss(tmem + C::kColS(t), adesc, bdesc, C::kIdescS, kk > 0 ? 1u : 0u);
            else
              mma_tf32_ss(tmem + C::kColS(t), adesc, bdesc, C::kIdescS, kk > 0 ? 1u : 0u);
          }
          tc_commit(bar(C::kBarSFull + t));
        }
      }
      if (!ok) break;
      if constexpr (kWin) {
        // a ring slot is handed back only after its copy landed, even if no
        // query tile of this CTA read it
        if (j >= 1 && !v_ready)
          ok = wait_bounded(bar(C::kBarVFull + (j - 1) % C::kStages), ((j - 1) / C::kStages) & 1, wctx,
                            kStatusTimeoutMmaV);
        if (ok && j < n_max && !k_ready)
          ok = wait_bounded(bar(C::kBarKFull + s), (j / C::kStages) & 1, wctx, kStatusTimeoutMmaK);
        if (!ok) break;
      }
      // Round j's commit frees K_j (read by this round's S GEMMs) and V_{j-1}
      // (read by its P V GEMMs); the loader waits for round i - kStages before
      // loading K_i and for round i - kStages + 1 before loading V_i.
      if (j < n_max) tc_commit(bar(C::kBarFree + s));
    }
    // every MMA issued above must finish before TMEM is released
    tc_commit(bar(C::kBarMmaDone));
    drain_bounded(bar(C::kBarMmaDone), 0);
  }
  __syncwarp();
} else if (!skip && warp < C::kSoftmaxWarps && C::kHalves == 2) {
  softmax_halves<C, kCausal, kMod, kWin>(p, tmO, unit, split, kb, base, tmem, warp, lane, wctx);
} else if (!skip && warp < C::kSoftmaxWarps) {
  // ---------------------------------------------------------- softmax warpgroups
  const int t = warp / 4;
  const int r = (warp % 4) * 32 + lane;  // row within the tile = TMEM lane
  const int tile_row0 = tile_first_row(p, unit, t, C::kQTiles);
  const int bh_t = tile_head(p, unit, t);
  const int row = tile_row0 + r;
  const KvSpan span = kv_span<kWin, C::BN>(tile_row0, p, kCausal, split);
  const int n_t = span.count;
  const uint32_t lane_addr = static_cast<uint32_t>((warp % 4) * 32) << 16;
  const uint32_t tS = tmem + lane_addr + C::kColS(t);
  const uint32_t tO = tmem + lane_addr + C::kColO(t);
  // The exponent step computes s * sl2 - base.  With a softcap the kMod path
  // turns S into log2 units first (sl2 = 1); otherwise S stays in raw q.k units
  // and the ALiBi penalty is applied in those units (slope / scale).
  const bool capped = kMod && p.cap_in > 0.f;
  const float sl2 = capped ? 1.0f : p.scale_log2;
  float slope_s = 0.f;  // ALiBi slope of this head, in the units S is held in
  if constexpr (kMod) {
    if (p.alibi != nullptr) {
      const float a = p.alibi[(bh_t / p.H) * p.alibi_bstride + bh_t % p.H];
      slope_s = capped ? a * 1.4426950408889634f : a * (1.4426950408889634f / p.scale_log2);
    }
  }
  const uint64_t sl2x2 = pack_f32x2(sl2, sl2);
  float m_run = -INFINITY;  // exponent base in use: a running max of scale*log2e*s
  float l_run = 0.f;        // running sum of the rounded exp2(s*sl2 - m_run)
  bool ok = n_t > 0;

  for (int j = 0; ok && j < n_t; ++j) {
    ok = __all_sync(0xffffffffu, wait_bounded(bar(C::kBarSFull + t), j & 1, wctx, kStatusTimeoutSoftmaxS));
    if (!ok) break;
    softmax_step<C, kCausal, kMod, kWin>(p, tS, tO, bar(C::kBarPFull + t), ((kWin ? span.first : kb) + j) * C::BN,
                                         tile_row0, row, capped, slope_s, sl2, sl2x2, j > 0, m_run, l_run);
  }
  // With the ones column the row sum is read from O_t's column D once the last
  // P V has landed (the epilogue waits for it before using l_run).
  auto row_sum = [&]() -> float {
    if constexpr (C::kLOnes) {
      uint32_t lv[16];
      tmem_ld_x16(tO + C::D, lv);
      tmem_ld_wait();
      reg_fence_x16(lv);
      return __uint_as_float(lv[0]);
    } else {
      return l_run;
    }
  };

  // ------------------------------------------------------------ epilogue
  if (p.num_splits > 1) {
    // split-KV partial for the rows of this tile: O_s = O/l_s in fp32, L_s (natural
    // log); a split without visible keys for the tile contributes O_s = 0, L_s = -inf
    if (tile_row0 < p.M) {
      if (n_t > 0 && ok)
        ok = __all_sync(0xffffffffu, wait_bounded(bar(C::kBarOFull + t), n_t > 0 ? 0 : 1, wctx,
                                                  kStatusTimeoutEpilogue));
      const int64_t prow = (static_cast<int64_t>(split) * p.BH + bh_t) * p.M + row;
      float4* op = reinterpret_cast<float4*>(p.o_part + prow * C::D);
      if (n_t > 0 && ok) {
        tc_fence_after_sync();
        l_run = row_sum();
        const float inv_l = l_run > 0.f ? 1.0f / l_run : 0.f;
#pragma unroll
        for (int ch = 0; ch < C::D / 32; ++ch) {
          uint32_t v[32];
          tmem_ld_x32(tO + ch * 32, v);
          tmem_ld_wait();
          reg_fence_x32(v);
          if (row < p.M) {
#pragma unroll
            for (int q4 = 0; q4 < 8; ++q4)
              op[ch * 8 + q4] = make_float4(__uint_as_float(v[q4 * 4 + 0]) * inv_l,
                                            __uint_as_float(v[q4 * 4 + 1]) * inv_l,
                                            __uint_as_float(v[q4 * 4 + 2]) * inv_l,
                                            __uint_as_float(v[q4 * 4 + 3]) * inv_l);
          }
        }
        if (row < p.M)
          p.l_part[prow] = (m_run + lg2_approx(l_run)) * 0.69314718055994530942f;
      } else if (n_t == 0 && row < p.M) {
#pragma unroll
        for (int q4 = 0; q4 < C::D / 4; ++q4) op[q4] = make_float4(0.f, 0.f, 0.f, 0.f);
        p.l_part[prow] = -INFINITY;
      }
    }
  } else if (n_t > 0 || (kWin && tile_row0 < p.M)) {
    // (kWin: a window can leave every row of a tile without a visible key; the
    // tile is then written as O = 0, L = -inf)
    if (ok)
      ok = __all_sync(0xffffffffu, wait_bounded(bar(C::kBarOFull + t), n_t > 0 ? 0 : 1, wctx,
                                                kStatusTimeoutEpilogue));
    // Q_t's shared tile is free once the last GEMM of this tile completed: stage O there
    const uint32_t stage = base + C::kOffQ + t * C::kTileBytes;
    if (kWin && n_t == 0) {
#pragma unroll
      for (int cidx = 0; cidx < C::kColBlocks * 8; ++cidx)
        st_shared_v4(stage + (cidx / 8) * C::kBlockBytes + r * 128 + (cidx % 8) * 16, 0u, 0u, 0u, 0u);
      if (row < p.M) p.lse[static_cast<int64_t>(bh_t) * p.M + row] = -INFINITY;
    } else if (ok) {
      tc_fence_after_sync();
      l_run = row_sum();
      const float inv_l = l_run > 0.f ? 1.0f / l_run : 0.f;
#pragma unroll
      for (int ch = 0; ch < C::D / 32; ++ch) {
        uint32_t v[32];
        tmem_ld_x32(tO + ch * 32, v);
        tmem_ld_wait();
        reg_fence_x32(v);
        if constexpr (C::kBF16) {
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {  // 16-byte chunks of 8 bf16
            const int cidx = ch * 4 + q4;
            const int cb = cidx / 8, c = cidx % 8;
            const uint32_t addr = stage + cb * C::kBlockBytes + r * 128 + ((c ^ (r & 7)) << 4);
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e)
              w[e] = pack_bf16x2(__uint_as_float(v[q4 * 8 + 2 * e]) * inv_l,
                                 __uint_as_float(v[q4 * 8 + 2 * e + 1]) * inv_l);
            st_shared_v4(addr, w[0], w[1], w[2], w[3]);
          }
        } else {
#pragma unroll
          for (int q8 = 0; q8 < 8; ++q8) {  // 16-byte chunks of 4 fp32
            const int cb = ch, c = q8;
            const uint32_t addr = stage + cb * C::kBlockBytes + r * 128 + ((c ^ (r & 7)) << 4);
            st_shared_v4(addr, __float_as_uint(__uint_as_float(v[q8 * 4 + 0]) * inv_l),
                         __float_as_uint(__uint_as_float(v[q8 * 4 + 1]) * inv_l),
                         __float_as_uint(__uint_as_float(v[q8 * 4 + 2]) * inv_l),
                         __float_as_uint(__uint_as_float(v[q8 * 4 + 3]) * inv_l));
          }
        }
      }
      if (row < p.M) {
        // L = ln(2) * (m + log2 l): the base-2 running state converted to natural log
        const float L = (m_run + lg2_approx(l_run)) * 0.69314718055994530942f;
        p.lse[static_cast<int64_t>(bh_t) * p.M + row] = L;
      }
    }
    fence_proxy_async_smem();
    named_barrier_sync(1 + t, 128);
    if (r == 0 && *wctx.abort_flag == 0u) {
#pragma unroll
      for (int cb = 0; cb < C::kColBlocks; ++cb)
        tma_store_3d(&tmO, stage + cb * C::kBlockBytes, cb * C::kSwElems, tile_row0, bh_t);
      tma_store_commit();
      tma_store_wait_read_all();
    }
  }
}

// ------------------------------------------------------------ teardown
if (skip && threadIdx.x == 0) {  // the loads thread 0 issued land before the memory is released
#pragma unroll
  for (int t = 0; t < C::kQTiles; ++t)
    if (nkv[t] > 0) drain_bounded(bar(C::kBarQ + t), 0);
  if (kEarlyKV && n_max > 0) {
    drain_bounded(bar(C::kBarKFull), 0);
    drain_bounded(bar(C::kBarVFull), 0);
  }
}
tc_fence_before_sync();
__syncthreads();
if (warp == C::kMmaWarp) {
  tc_fence_after_sync();
  tmem_dealloc(tmem, C::kTmemCols);
}
}

// Host-side launch description shared by the instantiation units.
struct FwdLaunch {
  CUtensorMap tmQ, tmK, tmV, tmO;
  FwdParams params;
  int causal;
  int mod;  // softcap or ALiBi in use: the kernels with kMod
  int win;  // a sliding window in use: the kernels with kWin (spans and masks)
  cudaStream_t stream;
};

}  // namespace fa2
