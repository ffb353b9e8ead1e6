// Instantiation of the forward kernel for bf16 inputs, head dim 128.
#include "fa2_config.h"
#include "fa2_launch.cuh"

namespace fa2 {

using Cfg_bf16_d128 = FwdCfg<128, true, 2, 2>;
static_assert(qtiles_for(0, 128) == Cfg_bf16_d128::kQTiles, "host and kernel tile configs differ");

cudaError_t launch_bf16_d128(FwdLaunch& L) { return launch_cfg<Cfg_bf16_d128>(L); }

}  // namespace fa2
