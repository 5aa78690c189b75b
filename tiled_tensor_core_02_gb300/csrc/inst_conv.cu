// Instantiations: implicit-GEMM convolution kernels (A gathered from the NHWC
// input by plain loads, filters staged like a K-major B operand).
#include "gemm_launch.cuh"

namespace ttc {
TTC_DEFINE_LAUNCH(256, kModeConvF16)
TTC_DEFINE_LAUNCH(128, kModeConvF16)
TTC_DEFINE_LAUNCH(64, kModeConvF16)
TTC_DEFINE_LAUNCH(32, kModeConvF16)
TTC_DEFINE_LAUNCH(256, kModeConvBF16)
TTC_DEFINE_LAUNCH(128, kModeConvBF16)
TTC_DEFINE_LAUNCH(64, kModeConvBF16)
TTC_DEFINE_LAUNCH(32, kModeConvBF16)
}  // namespace ttc
