// Instantiations and launch of the CTA-pair (2-SM) fp16/bf16 kernel.
#include <cuda_runtime.h>

#include <atomic>

#include "gemm2sm_kernel.cuh"

namespace ttc {

namespace {
template <bool kBF16>
cudaError_t set_smem_attr() {
  static std::atomic<bool> done[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!done[dev].load()) {
    e = cudaFuncSetAttribute(gemm_pair_kernel<kBF16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             PairCfg::kSmemBytes);
    if (e != cudaSuccess) return e;
    done[dev].store(true);
  }
  return cudaSuccess;
}
}  // namespace

// Largest number of CTA pairs that can be resident at once (0 on error).
int pair_max_clusters(bool bf16) {
  cudaError_t e = bf16 ? set_smem_attr<true>() : set_smem_attr<false>();
  if (e != cudaSuccess) return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2, 1, 1);
  cfg.blockDim = dim3(kPairThreads, 1, 1);
  cfg.dynamicSmemBytes = PairCfg::kSmemBytes;
  int n = 0;
  e = bf16 ? cudaOccupancyMaxActiveClusters(&n, gemm_pair_kernel<true>, &cfg)
           : cudaOccupancyMaxActiveClusters(&n, gemm_pair_kernel<false>, &cfg);
  return e == cudaSuccess ? n : 0;
}

cudaError_t launch_pair(bool bf16, const GemmParams& p, int clusters, cudaStream_t stream) {
  cudaError_t e = bf16 ? set_smem_attr<true>() : set_smem_attr<false>();
  if (e != cudaSuccess) return e;
  if (bf16)
    gemm_pair_kernel<true><<<2 * clusters, kPairThreads, PairCfg::kSmemBytes, stream>>>(p);
  else
    gemm_pair_kernel<false><<<2 * clusters, kPairThreads, PairCfg::kSmemBytes, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace ttc
