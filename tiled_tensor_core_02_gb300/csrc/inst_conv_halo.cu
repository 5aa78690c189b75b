// Instantiations and launch of the unit-stride halo convolution kernel.
#include <cuda_runtime.h>

#include <atomic>

#include "conv_halo_kernel.cuh"

namespace ttc {

namespace {
constexpr int kHaloSmemLimit = 227 * 1024;

template <int BN, bool kBF16>
cudaError_t set_smem_attr() {
  static std::atomic<bool> done[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!done[dev].load()) {
    e = cudaFuncSetAttribute(conv_halo_kernel<BN, kBF16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kHaloSmemLimit);
    if (e != cudaSuccess) return e;
    done[dev].store(true);
  }
  return cudaSuccess;
}

template <int BN, bool kBF16>
int max_clusters() {
  if (set_smem_attr<BN, kBF16>() != cudaSuccess) return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2, 1, 1);
  cfg.blockDim = dim3(kHaloThreads, 1, 1);
  cfg.dynamicSmemBytes = kHaloSmemLimit;
  int n = 0;
  return cudaOccupancyMaxActiveClusters(&n, conv_halo_kernel<BN, kBF16>, &cfg) == cudaSuccess ? n : 0;
}

template <int BN, bool kBF16>
cudaError_t launch(const ConvHaloParams& hp, int smem_bytes, int clusters, cudaStream_t stream) {
  if (smem_bytes > kHaloSmemLimit) return cudaErrorInvalidValue;
  const cudaError_t e = set_smem_attr<BN, kBF16>();
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * clusters, 1, 1);  // clusters of 2 from the kernel's __cluster_dims__
  cfg.blockDim = dim3(kHaloThreads, 1, 1);
  cfg.dynamicSmemBytes = smem_bytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  add_pdl_attribute(cfg, attr);
  const cudaError_t le = cudaLaunchKernelEx(&cfg, conv_halo_kernel<BN, kBF16>, hp);
  if (le != cudaSuccess) return le;
  return cudaGetLastError();
}
}  // namespace

int conv_halo_max_clusters(bool bf16, int bn) {
  switch (bn) {
    case 256: return bf16 ? max_clusters<256, true>() : max_clusters<256, false>();
    case 128: return bf16 ? max_clusters<128, true>() : max_clusters<128, false>();
  }
  return 0;
}

cudaError_t launch_conv_halo(bool bf16, int bn, const ConvHaloParams& hp, int smem_bytes, int clusters,
                             cudaStream_t stream) {
  switch (bn) {
    case 256:
      return bf16 ? launch<256, true>(hp, smem_bytes, clusters, stream)
                  : launch<256, false>(hp, smem_bytes, clusters, stream);
    case 128:
      return bf16 ? launch<128, true>(hp, smem_bytes, clusters, stream)
                  : launch<128, false>(hp, smem_bytes, clusters, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace ttc
