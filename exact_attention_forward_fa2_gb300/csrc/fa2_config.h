// Tile configurations of the forward kernel per (dtype, head dim), shared by the
// host API (grid sizing, validation) and the instantiation units.
#pragma once

namespace fa2 {

// Three kernel configurations per (dtype, head dim), picked by the score modifiers
// in use (the instantiation units hold each one's K/V ring depth):
//   softcap          two softmax warpgroups per query tile, row sum on the CUDA
//                    cores, 128-key tiles
//   sliding window   one warpgroup per query tile, 128-key tiles (112-key tiles add
//                    masked tiles at the window edges: -4.4% measured)
//   otherwise        one warpgroup per query tile, with the key-tile sizes below
// Shared memory per CTA is kQTiles query tiles of 128 rows x D plus kStages K and
// V tiles of kv_tile_for() rows x D (V with one more 128-byte column block of ones
// where the tensor core forms the row sum), e.g. for the plain kernels:
//   bf16 D=64   2 query tiles, 128-key tiles, 3 stages (177 KB)
//   bf16 D=128  2 query tiles, 112-key tiles, 2 stages (205 KB)
//   fp32 D=64   2 query tiles, 128-key tiles, 2 stages (225 KB)
//   fp32 D=128  1 query tile,  128-key tiles, 1 stage  (193 KB)
// (Three query tiles of 80-key tiles at bf16 D=64, so that 3 x (80 + 80) TMEM
// columns hold S and [O | row sum], measured 14% slower than two of 128 keys: the
// smaller steps cost more MMA instructions and synchronisation per key.)
constexpr int qtiles_for(int is_fp32, int D, int softcap = 0, int window = 0) {
  (void)softcap;
  (void)window;
  return (is_fp32 && D == 128) ? 1 : 2;
}

// Keys per key/value tile.  bf16 at D = 128 uses 112-key tiles in the plain
// kernels: S then takes 112 TMEM columns and [O | row sum] 144, so both query
// tiles' S and O fit in the 512 columns with the row sum formed by the tensor core
// (a ones block in V) instead of the softmax warps.
constexpr int kv_tile_for(int is_fp32, int D, int softcap = 0, int window = 0) {
  return (!is_fp32 && D == 128 && !softcap && !window) ? 112 : 128;
}

}  // namespace fa2
