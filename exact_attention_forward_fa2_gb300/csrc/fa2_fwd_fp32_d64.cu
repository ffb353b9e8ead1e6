// Instantiation of the forward kernel for fp32 inputs, head dim 64.
#include "fa2_config.h"
#include "fa2_launch.cuh"

namespace fa2 {

using Cfg_fp32_d64 = FwdCfg<64, false, 2, 2>;
static_assert(qtiles_for(1, 64) == Cfg_fp32_d64::kQTiles, "host and kernel tile configs differ");

cudaError_t launch_fp32_d64(FwdLaunch& L) { return launch_cfg<Cfg_fp32_d64>(L); }

}  // namespace fa2
