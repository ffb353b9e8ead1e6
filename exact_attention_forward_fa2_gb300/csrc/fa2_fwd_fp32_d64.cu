// Instantiation of the forward kernel for fp32 inputs, head dim 64.
#include "fa2_config.h"
#include "fa2_launch.cuh"

namespace fa2 {

// the plain and ALiBi kernels, the sliding-window kernels (one softmax warpgroup
// per query tile) and the softcap kernels (two per query tile)
using Cfg_fp32_d64 = FwdCfg<64, false, qtiles_for(1, 64), 2, 1, kv_tile_for(1, 64)>;
using CfgWin_fp32_d64 = FwdCfg<64, false, qtiles_for(1, 64, 0, 1), 2, 1, kv_tile_for(1, 64, 0, 1)>;
using CfgCap_fp32_d64 = FwdCfg<64, false, qtiles_for(1, 64, 1), 2, 2, kv_tile_for(1, 64, 1)>;

cudaError_t launch_fp32_d64(FwdLaunch& L) { return launch_cfg<Cfg_fp32_d64, CfgWin_fp32_d64, CfgCap_fp32_d64>(L); }

}  // namespace fa2
