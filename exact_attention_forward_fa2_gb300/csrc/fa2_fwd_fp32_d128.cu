// Instantiation of the forward kernel for fp32 inputs, head dim 128.
#include "fa2_config.h"
#include "fa2_launch.cuh"

namespace fa2 {

// the plain and ALiBi kernels, the sliding-window kernels (one softmax warpgroup
// per query tile) and the softcap kernels (two per query tile)
using Cfg_fp32_d128 = FwdCfg<128, false, qtiles_for(1, 128), 1, 1, kv_tile_for(1, 128)>;
using CfgWin_fp32_d128 = FwdCfg<128, false, qtiles_for(1, 128, 0, 1), 1, 1, kv_tile_for(1, 128, 0, 1)>;
using CfgCap_fp32_d128 = FwdCfg<128, false, qtiles_for(1, 128, 1), 1, 2, kv_tile_for(1, 128, 1)>;

cudaError_t launch_fp32_d128(FwdLaunch& L) { return launch_cfg<Cfg_fp32_d128, CfgWin_fp32_d128, CfgCap_fp32_d128>(L); }

}  // namespace fa2
