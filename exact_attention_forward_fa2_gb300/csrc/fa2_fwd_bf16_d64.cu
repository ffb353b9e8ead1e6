// Instantiation of the forward kernel for bf16 inputs, head dim 64.
#include "fa2_config.h"
#include "fa2_launch.cuh"

namespace fa2 {

// the plain and ALiBi kernels, the sliding-window kernels (one softmax warpgroup
// per query tile) and the softcap kernels (two per query tile)
using Cfg_bf16_d64 = FwdCfg<64, true, qtiles_for(0, 64), 3, 1, kv_tile_for(0, 64)>;
using CfgWin_bf16_d64 = FwdCfg<64, true, qtiles_for(0, 64, 0, 1), 3, 1, kv_tile_for(0, 64, 0, 1)>;
using CfgCap_bf16_d64 = FwdCfg<64, true, qtiles_for(0, 64, 1), 3, 2, kv_tile_for(0, 64, 1)>;

cudaError_t launch_bf16_d64(FwdLaunch& L) { return launch_cfg<Cfg_bf16_d64, CfgWin_bf16_d64, CfgCap_bf16_d64>(L); }

}  // namespace fa2
