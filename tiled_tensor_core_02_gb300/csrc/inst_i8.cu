// Instantiations: int8 x int8 -> int32 kernels (fp16 tensor-core inputs).
#include "gemm_launch.cuh"

namespace ttc {
TTC_DEFINE_LAUNCH(128, kModeI8)
TTC_DEFINE_LAUNCH(64, kModeI8)
TTC_DEFINE_LAUNCH(32, kModeI8)
}  // namespace ttc
