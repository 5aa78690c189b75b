// Instantiations and launch of the CTA-pair (2-SM) fp16/bf16 kernel.
#include <cuda_runtime.h>

#include <atomic>

#include "gemm2sm_kernel.cuh"

namespace ttc {

namespace {
template <int BN, bool kBF16, bool kI8 = false, int kEW = 8>
cudaError_t set_smem_attr() {
  static std::atomic<bool> done[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!done[dev].load()) {
    e = cudaFuncSetAttribute(gemm_pair_kernel<BN, kBF16, kI8, kEW>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             PairCfg<BN, kI8, kEW>::kSmemBytes);
    if (e != cudaSuccess) return e;
    done[dev].store(true);
  }
  return cudaSuccess;
}

template <int BN, bool kBF16, bool kI8 = false, int kEW = 8>
int max_clusters() {
  if (set_smem_attr<BN, kBF16, kI8, kEW>() != cudaSuccess) return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2, 1, 1);
  cfg.blockDim = dim3(64 + 32 * kEW, 1, 1);
  cfg.dynamicSmemBytes = PairCfg<BN, kI8, kEW>::kSmemBytes;
  int n = 0;
  return cudaOccupancyMaxActiveClusters(&n, gemm_pair_kernel<BN, kBF16, kI8, kEW>, &cfg) == cudaSuccess ? n : 0;
}

template <int BN, bool kBF16, bool kI8 = false, int kEW = 8>
cudaError_t launch(const GemmParams& p, int clusters, cudaStream_t stream) {
  const cudaError_t e = set_smem_attr<BN, kBF16, kI8, kEW>();
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * clusters, 1, 1);  // clusters of 2 from the kernel's __cluster_dims__
  cfg.blockDim = dim3(64 + 32 * kEW, 1, 1);
  cfg.dynamicSmemBytes = PairCfg<BN, kI8, kEW>::kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  add_pdl_attribute(cfg, attr);
  const cudaError_t le = cudaLaunchKernelEx(&cfg, gemm_pair_kernel<BN, kBF16, kI8, kEW>, p);
  if (le != cudaSuccess) return le;
  return cudaGetLastError();
}
}  // namespace

// Largest number of CTA pairs that can be resident at once (0 on error).
int pair_max_clusters(bool bf16, int bn) {
  switch (bn) {
    case 256: return bf16 ? max_clusters<256, true>() : max_clusters<256, false>();
    case 224: return bf16 ? max_clusters<224, true>() : max_clusters<224, false>();
    case 192: return bf16 ? max_clusters<192, true>() : max_clusters<192, false>();
    case 128: return bf16 ? max_clusters<128, true>() : max_clusters<128, false>();
  }
  return 0;
}

// The int8 variant (fp16 copies of int8 operands, exact int32 sums): 256-wide tiles.
int pair_max_clusters_i8() { return max_clusters<256, false, true>(); }

cudaError_t launch_pair_i8(const GemmParams& p, int clusters, cudaStream_t stream) {
  return launch<256, false, true>(p, clusters, stream);
}

// 256-wide tiles with twelve epilogue warps and no staging buffers: only for
// outputs written with plain stores (p.d_tma == 0).
int pair_max_clusters_ew12(bool bf16) {
  return bf16 ? max_clusters<256, true, false, 12>() : max_clusters<256, false, false, 12>();
}

cudaError_t launch_pair_ew12(bool bf16, const GemmParams& p, int clusters, cudaStream_t stream) {
  if (p.d_tma) return cudaErrorInvalidValue;
  return bf16 ? launch<256, true, false, 12>(p, clusters, stream) : launch<256, false, false, 12>(p, clusters, stream);
}

cudaError_t launch_pair(bool bf16, int bn, const GemmParams& p, int clusters, cudaStream_t stream) {
  switch (bn) {
    case 256: return bf16 ? launch<256, true>(p, clusters, stream) : launch<256, false>(p, clusters, stream);
    case 224: return bf16 ? launch<224, true>(p, clusters, stream) : launch<224, false>(p, clusters, stream);
    case 192: return bf16 ? launch<192, true>(p, clusters, stream) : launch<192, false>(p, clusters, stream);
    case 128: return bf16 ? launch<128, true>(p, clusters, stream) : launch<128, false>(p, clusters, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace ttc
