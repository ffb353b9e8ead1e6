// Instantiation of the forward kernel for fp32 inputs, head dim 128.
#include "fa2_config.h"
#include "fa2_launch.cuh"

namespace fa2 {

using Cfg_fp32_d128 = FwdCfg<128, false, 1, 1>;
static_assert(qtiles_for(1, 128) == Cfg_fp32_d128::kQTiles, "host and kernel tile configs differ");

cudaError_t launch_fp32_d128(FwdLaunch& L) { return launch_cfg<Cfg_fp32_d128>(L); }

}  // namespace fa2
