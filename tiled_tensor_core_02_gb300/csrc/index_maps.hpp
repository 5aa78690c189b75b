// Host-side derivation of the GEMM kernels' index maps (tile_maps.h) from
// Shape/Stride layouts, with the algebra of include/ttc_layout.hpp.
//
// Sources (restated): "Advanced CUTLASS Architecture and Kernel
// Optimization", section "Advanced Layout Operations" (oboe.com): a GEMM uses
// logical_divide to map the logical M, N and K dimensions onto its tiles;
// "4.21 What is CuTe?" (gpu-glossary-zh), transpose kernel: tiled_divide picks
// a block's tile, local_partition a thread's elements of it.
//
// Each map is read off a divided layout: the rest mode of a divide by the tile
// is the affine map from a tile index to the tile's origin, its stride is the
// step the kernel multiplies by.  Extents only need to hold two tiles for that
// stride to be defined, so coordinate layouts are built over max(extent, two
// tiles) (a mode of extent 1 has no stride of its own).
#pragma once

#include <cstdint>
#include <stdexcept>
#include <vector>

#include "tile_maps.h"
#include "ttc_layout.hpp"

namespace ttc {
namespace maps {

using layout::Layout;
using layout::tup;

// Stride of a layout of one leaf mode (or a one-mode tuple).
inline int64_t leaf_stride(const Layout& l) {
  const auto s = layout::flatten(l.shape), d = layout::flatten(l.stride);
  int64_t out = 0;
  int live = 0;
  for (size_t i = 0; i < s.size(); ++i)
    if (s[i] != 1) {
      out = d[i];
      ++live;
    }
  if (live > 1) throw std::invalid_argument("leaf_stride: more than one mode");
  return out;
}

inline int64_t two_tiles(int64_t extent, int64_t tile) { return extent > 2 * tile ? extent : 2 * tile; }

// Origins of the tiles of an M x N output: zipped_divide of the output's
// coordinate functions row(i, j) = i, i.e. (M, N):(1, 0), and col(i, j) = j,
// (M, N):(0, 1), by the (tile_m, tile_n) tiler.  Mode 1 of the result, the
// rest mode (mb, nb), maps a tile index to its origin row (column).
inline void tile_origins(int64_t M, int64_t N, int tile_m, int tile_n, TileMaps& tm) {
  const int64_t m = two_tiles(M, tile_m), n = two_tiles(N, tile_n);
  const std::vector<Layout> tiler{Layout(tile_m, 1), Layout(tile_n, 1)};
  const Layout row_rest = layout::mode(layout::zipped_divide(Layout(tup({m, n}), tup({1, 0})), tiler), 1);
  const Layout col_rest = layout::mode(layout::zipped_divide(Layout(tup({m, n}), tup({0, 1})), tiler), 1);
  tm.tile_m = (int32_t)leaf_stride(layout::mode(row_rest, 0));
  tm.tile_n = (int32_t)leaf_stride(layout::mode(col_rest, 1));
  if (leaf_stride(layout::mode(row_rest, 1)) != 0 || leaf_stride(layout::mode(col_rest, 0)) != 0)
    throw std::logic_error("tile origins: a row depends on the column index");
}

// The share of CTA r of a cluster of `ctas` in `extent` rows (columns) of a
// tile: logical_divide(extent:1, (extent / ctas):1) = ((extent / ctas):1,
// ctas:step); CTA r starts at r * step.  0 for one CTA.
inline int32_t cta_step(int extent, int ctas) {
  if (ctas <= 1) return 0;
  if (extent % ctas) throw std::invalid_argument("cta_step: CTAs do not divide the tile");
  const Layout d = layout::logical_divide(Layout(extent, 1), Layout(extent / ctas, 1));
  return (int32_t)leaf_stride(layout::mode(d, 1));
}

// TMA boxes of one operand's k-block tile.  The operand as stored is
// (rows, K):(ld, 1) when K-major and (rows, K):(1, ld) when MN-major; its tile
// is mode 0 of zipped_divide by (tile_rows, 64).  The tile's stride-1 mode is
// the box's inner dimension.  With the 128-byte swizzle a box spans 128 / esize
// elements of it (a slab of the swizzled layout the MMA reads), so
// logical_divide of that mode by the span gives the box (mode 0) and the boxes
// (mode 1: count and coordinate step); a mode shorter than the span still
// gets a whole slab, read past the operand's end as zeros.  Unswizzled (the
// raw int8 staging), the whole mode is one box.  The other mode is the box's
// outer extent.
inline BoxMap operand_boxes(bool k_major, int64_t rows, int64_t K, int64_t ld, int tile_rows, int esize,
                            bool swizzled = true) {
  const int64_t r = two_tiles(rows, tile_rows), k = two_tiles(K, 64);
  const Layout op = k_major ? Layout(tup({r, k}), tup({ld, 1})) : Layout(tup({r, k}), tup({1, ld}));
  const Layout tile = layout::mode(layout::zipped_divide(op, {Layout(tile_rows, 1), Layout(64, 1)}), 0);
  const Layout m_mode = layout::mode(tile, 0), k_mode = layout::mode(tile, 1);
  const bool k_inner = leaf_stride(k_mode) == 1;
  if (!k_inner && leaf_stride(m_mode) != 1) throw std::logic_error("operand_boxes: no contiguous mode");
  const Layout inner = k_inner ? k_mode : m_mode;
  const Layout outer = k_inner ? m_mode : k_mode;
  const int span = swizzled ? 128 / esize : (int)inner.size();
  const Layout cut = layout::logical_divide(inner, Layout(span, 1));
  BoxMap b;
  b.k_inner = k_inner ? 1 : 0;
  b.box_inner = (int32_t)layout::mode(cut, 0).size();
  b.boxes = (int32_t)layout::mode(cut, 1).size();
  b.box_step = b.boxes > 1 ? (int32_t)leaf_stride(layout::mode(cut, 1)) : b.box_inner;
  b.box_outer = (int32_t)outer.size();
  b.smem_step = b.box_inner * b.box_outer * esize;
  return b;
}

// The epilogue's thread -> accumulator maps.  The accumulator tile (128 rows
// x tile_n columns) sits in TMEM with row = TMEM lane: address(row, col) =
// row << 16 | col, the layout (128, tile_n):(65536, 1).  local_partition of
// that tile (and of the tile's row-coordinate function (128, tile_n):(1, 0))
// by the thread layout (128, 1):(1, 128) gives thread t row t: the
// partition's offset for thread 1 is the per-thread step.  The thread's own
// columns, divided by the 32-column chunk, give the chunk step (mode 1).
inline void epilogue_maps(int tile_n, TileMaps& tm) {
  const int n = tile_n > 32 ? tile_n : 64;  // at least two chunks, so the chunk step is defined
  const Layout thr(tup({128, 1}), tup({1, 128}));
  const Layout tmem(tup({128, n}), tup({65536, 1}));
  const Layout rows(tup({128, n}), tup({1, 0}));
  const auto pt = layout::local_partition(tmem, thr, 1);
  const auto pr = layout::local_partition(rows, thr, 1);
  tm.tmem_row_step = (uint32_t)(pt.offset - layout::local_partition(tmem, thr, 0).offset);
  tm.epi_row_step = (int32_t)(pr.offset - layout::local_partition(rows, thr, 0).offset);
  const Layout own_cols = layout::mode(pt.layout, 1);  // the thread's columns in TMEM: tile_n:1
  const Layout chunks = layout::logical_divide(own_cols, Layout(32, 1));
  tm.epi_chunk = (int32_t)leaf_stride(layout::mode(chunks, 1));
  if (layout::mode(chunks, 0).size() != tm.epi_chunk) throw std::logic_error("epilogue chunks overlap");
}

// Every map of one launch: an output in tiles of tile_m x tile_n shared by
// the `ctas` CTAs of a cluster (2 for the CTA-pair kernel, 1 otherwise); each
// CTA stages a_rows rows of A and its share of the tile's B columns per
// k-block; half_cols > 0: the pair kernel's half units, half_cols wide (their
// B share per CTA gets its own boxes).  The maps do not depend on the
// problem's extents or leading dimensions, only on which mode of each operand
// is contiguous: they are derived over a problem of two tiles each way with
// tight leading dimensions.
inline TileMaps derive(int tile_m, int tile_n, int ctas, int a_rows, bool a_mn, bool b_mn, int esize,
                       bool swizzled = true, int half_cols = 0) {
  const int64_t M = 2 * tile_m, N = 2 * tile_n, K = 128;
  const int64_t lda = a_mn ? M : K, ldb = b_mn ? N : K;
  TileMaps tm{};
  tile_origins(M, N, tile_m, tile_n, tm);
  tm.cta_m = cta_step(tile_m, ctas);
  tm.cta_n = cta_step(tile_n, ctas);
  const int b_cols = ctas > 1 ? tm.cta_n : tile_n;
  // B is K x N; stored column-major it is (N, K):(ldb, 1), K-major
  tm.a = operand_boxes(!a_mn, M, K, lda, a_rows, esize, swizzled);
  tm.b = operand_boxes(!b_mn, N, K, ldb, b_cols, esize, swizzled);
  if (half_cols > 0) {
    // the tile's columns in two halves, each shared by the cluster's CTAs
    tm.half_n = cta_step(tile_n, 2);
    tm.cta_n_half = cta_step(half_cols, ctas);
    tm.b_half = operand_boxes(!b_mn, N, K, ldb, ctas > 1 ? tm.cta_n_half : half_cols, esize, swizzled);
  }
  epilogue_maps(tile_n, tm);
  return tm;
}

}  // namespace maps
}  // namespace ttc
