// Instantiation of the forward kernel for bf16 inputs, head dim 128.
#include "fa2_config.h"
#include "fa2_launch.cuh"

namespace fa2 {

// the plain and ALiBi kernels, the sliding-window kernels (one softmax warpgroup
// per query tile) and the softcap kernels (two per query tile)
using Cfg_bf16_d128 = FwdCfg<128, true, qtiles_for(0, 128), 2, 1, kv_tile_for(0, 128)>;
using CfgWin_bf16_d128 = FwdCfg<128, true, qtiles_for(0, 128, 0, 1), 2, 1, kv_tile_for(0, 128, 0, 1)>;
using CfgCap_bf16_d128 = FwdCfg<128, true, qtiles_for(0, 128, 1), 2, 2, kv_tile_for(0, 128, 1)>;

cudaError_t launch_bf16_d128(FwdLaunch& L) { return launch_cfg<Cfg_bf16_d128, CfgWin_bf16_d128, CfgCap_bf16_d128>(L); }

}  // namespace fa2
