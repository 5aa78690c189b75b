// Instantiations: TMA-staged fp16/bf16 kernels.
#include "gemm_launch.cuh"

namespace ttc {
TTC_DEFINE_LAUNCH(256, kModeTmaF16)
TTC_DEFINE_LAUNCH(128, kModeTmaF16)
TTC_DEFINE_LAUNCH(64, kModeTmaF16)
TTC_DEFINE_LAUNCH(32, kModeTmaF16)
TTC_DEFINE_LAUNCH(256, kModeTmaBF16)
TTC_DEFINE_LAUNCH(128, kModeTmaBF16)
TTC_DEFINE_LAUNCH(64, kModeTmaBF16)
TTC_DEFINE_LAUNCH(32, kModeTmaBF16)
}  // namespace ttc
