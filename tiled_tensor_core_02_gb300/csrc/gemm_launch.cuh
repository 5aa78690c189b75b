// Launch wrapper for one (tile width, mode) instantiation of gemm_kernel.
// Each instantiation lives in its own translation unit (inst_*.cu) so the
// variants compile in parallel.
#pragma once
#include <cuda_runtime.h>

#include <atomic>

#include "gemm_kernel.cuh"

namespace ttc {

template <int BN, int MODE>
cudaError_t launch_gemm(const GemmParams& p, int grid, cudaStream_t stream);

// CTA-pair (2-SM) fp16/bf16 kernel, defined in inst_pair.cu.
// bn: the pair tile's width (256, 224, 192 or 128).
int pair_max_clusters(bool bf16, int bn);
cudaError_t launch_pair(bool bf16, int bn, const GemmParams& p, int clusters, cudaStream_t stream);
// 256-wide tiles with twelve epilogue warps, for outputs written with plain
// stores (p.d_tma == 0; cudaErrorInvalidValue otherwise).
int pair_max_clusters_ew12(bool bf16);
cudaError_t launch_pair_ew12(bool bf16, const GemmParams& p, int clusters, cudaStream_t stream);
// Its int8 variant: fp16 copies of int8 operands, exact int32 result, 256-wide tiles.
int pair_max_clusters_i8();
cudaError_t launch_pair_i8(const GemmParams& p, int clusters, cudaStream_t stream);

template <int BN, int MODE>
int gemm_smem_bytes() {
  return TileCfg<BN, MODE>::kSmemBytes;
}

#define TTC_DEFINE_LAUNCH(BN, MODE)                                                                  \
  template <>                                                                                        \
  cudaError_t launch_gemm<BN, MODE>(const GemmParams& p, int grid, cudaStream_t stream) {           \
    static std::atomic<bool> attr_done[64];                                                          \
    int dev = 0;                                                                                     \
    cudaError_t e = cudaGetDevice(&dev);                                                             \
    if (e != cudaSuccess) return e;                                                                  \
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;                                         \
    constexpr int smem = TileCfg<BN, MODE>::kSmemBytes;                                              \
    if (!attr_done[dev].load()) {                                                                    \
      e = cudaFuncSetAttribute(gemm_kernel<BN, MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize,    \
                               smem);                                                                \
      if (e != cudaSuccess) return e;                                                                \
      attr_done[dev].store(true);                                                                    \
    }                                                                                                \
    cudaLaunchConfig_t cfg = {};                                                                     \
    cfg.gridDim = dim3(grid, 1, 1);                                                                  \
    cfg.blockDim = dim3(ModeTraits<MODE>::kThreads, 1, 1);                                           \
    cfg.dynamicSmemBytes = smem;                                                                     \
    cfg.stream = stream;                                                                             \
    cudaLaunchAttribute attr[2];                                                                     \
    if (p.ksplit > 1) {                                                                              \
      attr[0].id = cudaLaunchAttributeClusterDimension;                                              \
      attr[0].val.clusterDim.x = p.ksplit;                                                           \
      attr[0].val.clusterDim.y = 1;                                                                  \
      attr[0].val.clusterDim.z = 1;                                                                  \
      cfg.attrs = attr;                                                                              \
      cfg.numAttrs = 1;                                                                              \
    }                                                                                                \
    add_pdl_attribute(cfg, attr);                                                                    \
    e = cudaLaunchKernelEx(&cfg, gemm_kernel<BN, MODE>, p);                                          \
    if (e != cudaSuccess) return e;                                                                  \
    return cudaGetLastError();                                                                       \
  }

}  // namespace ttc
