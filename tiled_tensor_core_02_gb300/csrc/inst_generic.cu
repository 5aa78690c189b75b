// Instantiations: fp16/bf16 kernels whose operands are staged with plain loads.
#include "gemm_launch.cuh"

namespace ttc {
TTC_DEFINE_LAUNCH(256, kModeGenF16)
TTC_DEFINE_LAUNCH(128, kModeGenF16)
TTC_DEFINE_LAUNCH(64, kModeGenF16)
TTC_DEFINE_LAUNCH(32, kModeGenF16)
TTC_DEFINE_LAUNCH(256, kModeGenBF16)
TTC_DEFINE_LAUNCH(128, kModeGenBF16)
TTC_DEFINE_LAUNCH(64, kModeGenBF16)
TTC_DEFINE_LAUNCH(32, kModeGenBF16)
}  // namespace ttc
