// Instantiations: int8 x int8 -> int32 kernels (fp16 tensor-core inputs): plain-load
// producers for any pitch, TMA-staged int8 with converter warps for 16-byte pitches
// (an MN-major A widened into shared memory, a K-major A into tensor memory).
#include "gemm_launch.cuh"

namespace ttc {
TTC_DEFINE_LAUNCH(128, kModeI8)
TTC_DEFINE_LAUNCH(64, kModeI8)
TTC_DEFINE_LAUNCH(32, kModeI8)
TTC_DEFINE_LAUNCH(128, kModeI8Tma)
TTC_DEFINE_LAUNCH(64, kModeI8Tma)
TTC_DEFINE_LAUNCH(32, kModeI8Tma)
TTC_DEFINE_LAUNCH(128, kModeI8TmemA)
TTC_DEFINE_LAUNCH(64, kModeI8TmemA)
TTC_DEFINE_LAUNCH(32, kModeI8TmemA)
}  // namespace ttc
