// Instantiation of the forward kernel for bf16 inputs, head dim 64.
#include "fa2_config.h"
#include "fa2_launch.cuh"

namespace fa2 {

using Cfg_bf16_d64 = FwdCfg<64, true, 2, 3>;
static_assert(qtiles_for(0, 64) == Cfg_bf16_d64::kQTiles, "host and kernel tile configs differ");

cudaError_t launch_bf16_d64(FwdLaunch& L) { return launch_cfg<Cfg_bf16_d64>(L); }

}  // namespace fa2
