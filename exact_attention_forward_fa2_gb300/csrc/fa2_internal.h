// Declarations shared between the library's translation units; not part of the
// C ABI (include/fa2.h).
#pragma once

#include <cstddef>

namespace fa2 {

// The argument checks every forward entry makes before any CUDA call: pointers,
// sizes, head grouping, head dimension, element type, scale and alignment.
// FA2_OK or the FA2_ERR_* code of the first failing check.
int check_forward_args(const void* q, const void* k, const void* v, const void* o, const float* lse, int B,
                       int H, int H_kv, int M, int N, int D, float scale, int dtype);

}  // namespace fa2
