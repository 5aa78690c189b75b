// Index maps the GEMM kernels read from their parameters.  The host derives
// every field from Shape/Stride layouts (index_maps.hpp: logical_divide,
// zipped_divide and local_partition of the operand, output and TMEM layouts);
// the kernels only evaluate the resulting affine maps.  Plain data, usable on
// both sides.
#pragma once
#include <stdint.h>

namespace ttc {

// One operand's k-block tile as TMA boxes.  The tile is the operand's
// (rows x 64 k) block as stored; a box lists the tile's contiguous mode first,
// and that mode is cut at the swizzle span (128 bytes) into `boxes` boxes.
struct BoxMap {
  int32_t k_inner;    // 1: the contiguous mode is K (K-major operand); 0: the M (or N) mode
  int32_t box_inner;  // box extent along the contiguous mode (elements)
  int32_t box_outer;  // box extent along the other mode
  int32_t boxes;      // boxes per k-block tile
  int32_t box_step;   // coordinate step along the contiguous mode from one box to the next
  int32_t smem_step;  // bytes from one box to the next in shared memory
};

struct TileMaps {
  // tile (mb, nb) of the output starts at row mb * tile_m, column nb * tile_n
  int32_t tile_m, tile_n;
  // CTA r of a cluster stages the A rows from r * cta_m and the B columns from
  // r * cta_n of its tile (0 when the cluster's CTAs share the tile's rows or
  // columns, as the CTAs of a split-K cluster do)
  int32_t cta_m, cta_n;
  BoxMap a, b;
  // CTA-pair kernel, half units: half h of a tile covers the columns from
  // h * half_n; CTA r stages its B columns from r * cta_n_half, boxed as b_half
  int32_t half_n, cta_n_half;
  BoxMap b_half;
  // epilogue: epilogue thread t (warp quarter q = t / 32, lane t mod 32) owns
  // accumulator row t * epi_row_step; TMEM holds accumulator (row, column) at
  // row * tmem_row_step + column; chunk c covers columns from c * epi_chunk
  int32_t epi_row_step;
  uint32_t tmem_row_step;
  int32_t epi_chunk;
};

}  // namespace ttc
