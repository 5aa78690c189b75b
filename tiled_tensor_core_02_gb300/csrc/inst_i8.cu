// Instantiations: int8 x int8 -> int32 kernels (fp16 tensor-core inputs): plain-load
// producers for any pitch, TMA-staged int8 with converter warps for 16-byte pitches.
#include "gemm_launch.cuh"

namespace ttc {
TTC_DEFINE_LAUNCH(128, kModeI8)
TTC_DEFINE_LAUNCH(64, kModeI8)
TTC_DEFINE_LAUNCH(32, kModeI8)
TTC_DEFINE_LAUNCH(128, kModeI8Tma)
TTC_DEFINE_LAUNCH(64, kModeI8Tma)
TTC_DEFINE_LAUNCH(32, kModeI8Tma)
}  // namespace ttc
