// Parameters and launch of the unit-stride convolution kernel built from halo
// tiles (conv_halo_kernel.cuh, instantiated in inst_conv_halo.cu).
#pragma once
#include <cuda_runtime.h>

#include "gemm_kernel.cuh"

namespace ttc {

constexpr int kHaloThreads = 192;  // warp 0 producer, warp 1 TMEM + MMA, warps 2..5 epilogue
constexpr int kHaloMaxStages = 8;
// k-blocks (one filter tap of one 64-channel block each) per filter stage:
// one full/empty round trip per 8 MMAs keeps the tensor pipe fed, one per 4
// does not (measured on GB300)
constexpr int kHaloKPS = 2;
constexpr int kHaloEpiBufBytes = 32 * kEpiCols * 2;  // one warp's 32 x 32 staging block
constexpr int kHaloEpiBytes = kEpiWarps * kHaloEpiBufBytes;
constexpr int kHaloBarBytes = 256;

struct ConvHaloParams {
  GemmParams g;       // epilogue (alpha, beta, C, D, bias, act, N = output channels,
                      // M = N * P * Q), error word and timeouts; g.tmA is the halo
                      // map (C, W, H, N), g.tmB the filters (K-major)
  int n_img;          // images
  int img_pairs;      // ceil(n_img / 2)
  int tiles_per_img;  // 128-position tiles per image: ceil(P wp / 128)
  int n_blocks;       // output-channel blocks of the pair tile width
  int num_tiles;      // img_pairs * tiles_per_img * n_blocks
  int wp;             // positions per output row
  int p, q;           // output extent
  int c;              // input channels (a multiple of 64)
  int cblk;           // c / 64
  int taps;           // R * S
  int s;              // filter width
  int row_step;       // dil_h * wp: halo rows between filter rows
  int dw;             // dil_w
  int ph, pw;         // padding
  int halo_rows;      // input rows per halo box
  uint32_t halo_tx;   // bytes of one halo box
  uint32_t halo_bytes;  // its shared-memory footprint, a multiple of 1024
  int stages;         // filter ring depth in stages of kHaloKPS k-blocks (<= kHaloMaxStages)
  // work units [0, num_units) walk the tiles; units from tail_from on are
  // half tiles (the left or right half of the output channels of tile
  // tail_from + (u - tail_from) / 2): a last partial wave keeps twice as many
  // pairs busy for half as long.  tail_from == num_units: whole tiles.
  int tail_from, num_units;
};

// Bytes of dynamic shared memory the kernel needs (plus 1024 for alignment).
__host__ __device__ constexpr int conv_halo_smem_bytes(int halo_bytes, int stages, int b_half_bytes) {
  return 1024 + 2 * halo_bytes + stages * kHaloKPS * b_half_bytes + kHaloEpiBytes + kHaloBarBytes;
}

// Largest number of CTA pairs resident at once for tile width `bn` (0 on error).
int conv_halo_max_clusters(bool bf16, int bn);
// Launches `clusters` CTA pairs with `smem_bytes` of dynamic shared memory
// (conv_halo_smem_bytes of the plan).
cudaError_t launch_conv_halo(bool bf16, int bn, const ConvHaloParams& hp, int smem_bytes, int clusters,
                             cudaStream_t stream);

}  // namespace ttc
