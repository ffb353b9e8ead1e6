// Tile configurations of the forward kernel per (dtype, head dim), shared by the
// host API (grid sizing, validation) and the instantiation units.
#pragma once

namespace fa2 {

// Query tiles (of 128 rows) per CTA and K/V ring depth.  Shared memory per CTA is
// (kQTiles + 2 * kStages) tiles of 128 rows x D elements, at most ~192 KB here:
//   bf16 D=64   tile 16 KB: 2 query tiles, 3 stages (128 KB)
//   bf16 D=128  tile 32 KB: 2 query tiles, 2 stages (192 KB)
//   fp32 D=64   tile 32 KB: 2 query tiles, 2 stages (192 KB)
//   fp32 D=128  tile 64 KB: 1 query tile,  1 stage  (192 KB)
constexpr int qtiles_for(int is_fp32, int D) { return (is_fp32 && D == 128) ? 1 : 2; }

}  // namespace fa2

