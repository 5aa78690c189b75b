// ttc layout helper: Shape/Stride layouts and the few algebra operations the
// GEMM planner and kernels use to derive their index maps.
//
// Sources (restated in this code's own terms):
//   - "Advanced CUTLASS Architecture and Kernel Optimization", section "CuTe
//     Layout Algebra" (oboe.com): a layout is a (Shape, Stride) pair of integer
//     tuples; crd2idx is the dot product of coordinate and stride; layouts
//     compose as functions; logical_divide tiles a layout; logical_product
//     replicates one layout by another.
//   - "4.21 What is CuTe?" (gpu-glossary-zh): hierarchical shapes, and
//     tiled_divide's mode order (the tile first, the tile index after it).
//   - "ldmatrix and the CuTe TV layout" (hpc.payai.win/cutlass), Part 4: the
//     Swizzle<3,3,3> shared-memory layout that XORs the row into the 16-byte
//     chunk index; here as the byte-level Swizzle<B, 4, 3> family that TMA's
//     32/64/128-byte swizzle modes implement.
//   - PitchLinearStripminedThreadMap source walkthrough (lpnh.cn/news/2469163),
//     sections 2-4: the strip-mined thread map and its predicate.
//
// Conventions where the pages are silent: integer indices become coordinates
// colexicographically (leftmost mode fastest); complement() orders the gaps
// of a layout's image by stride; divides keep the within-tile mode first.
// Host code uses the dynamic IntTuple/Layout types; the swizzle and thread-map
// functions are constexpr and also callable from device code.
#pragma once

#include <cstdint>
#include <stdexcept>
#include <string>
#include <utility>
#include <vector>

#if defined(__CUDACC__)
#define TTC_HD __host__ __device__
#else
#define TTC_HD
#endif

namespace ttc {
namespace layout {

// ------------------------------------------------------------------ swizzle
// Byte-offset swizzle: bits [M+S, M+S+B) are XORed into bits [M, M+B).
// Swizzle<3,4,3> is TMA/UMMA's 128-byte swizzle (16-byte chunk index ^= row
// mod 8 for 128-byte rows); Swizzle<2,4,3> the 64-byte one; Swizzle<1,4,3>
// the 32-byte one.  On 2-byte elements Swizzle<3,4,3> of bytes equals the
// element-level Swizzle<3,3,3> the tutorial page draws.
template <int B, int M, int S>
struct Swizzle {
  static constexpr uint32_t kYMask = ((1u << B) - 1u) << (M + S);
  TTC_HD constexpr uint32_t operator()(uint32_t off) const { return off ^ ((off & kYMask) >> S); }
};
using SwizzleBytes128 = Swizzle<3, 4, 3>;
using SwizzleBytes64 = Swizzle<2, 4, 3>;
using SwizzleBytes32 = Swizzle<1, 4, 3>;

// ------------------------------------------------------------------ strip-mined thread map
// Tile of `rows` x `cols` elements (row-major, pitch = cols), `threads`
// threads, `vec` contiguous elements per access.  Columns are dealt out
// first: column group = tid mod (cols / vec), row anchor = tid div (cols /
// vec), iteration i moves down by row_stride = rows / iterations.
struct StripMined {
  int rows, cols, threads, vec;
  TTC_HD constexpr int iterations() const { return rows * cols / threads / vec; }
  TTC_HD constexpr int column_groups() const { return cols / vec; }
  TTC_HD constexpr int row_stride() const { return rows / iterations(); }
  // the invariant elements = threads * iterations * vec, and a whole number
  // of rows per iteration
  TTC_HD constexpr bool valid() const {
    return rows > 0 && cols > 0 && threads > 0 && vec > 0 && cols % vec == 0 &&
           (rows * cols) % (threads * vec) == 0 && iterations() > 0 && rows % iterations() == 0 &&
           threads % column_groups() == 0 && threads / column_groups() == row_stride();
  }
  TTC_HD constexpr int row(int tid, int it) const { return tid / column_groups() + it * row_stride(); }
  TTC_HD constexpr int col(int tid) const { return (tid % column_groups()) * vec; }
  // live iff the vector's first element lies inside the extent (the extent is
  // ragged; the stride above always comes from the tile)
  TTC_HD constexpr bool predicate(int tid, int it, int extent_rows, int extent_cols) const {
    return row(tid, it) < extent_rows && col(tid) < extent_cols;
  }
};

// ------------------------------------------------------------------ IntTuple
struct IntTuple {
  bool leaf = true;
  int64_t v = 0;
  std::vector<IntTuple> c;

  IntTuple() = default;
  IntTuple(int64_t x) : leaf(true), v(x) {}  // NOLINT: ints convert implicitly
  static IntTuple tuple(std::vector<IntTuple> elems) {
    IntTuple t;
    t.leaf = false;
    t.c = std::move(elems);
    return t;
  }
  size_t rank() const { return leaf ? 1 : c.size(); }
  const IntTuple& operator[](size_t i) const { return leaf ? *this : c.at(i); }
  bool operator==(const IntTuple& o) const {
    if (leaf != o.leaf) return false;
    return leaf ? v == o.v : c == o.c;
  }
  bool operator!=(const IntTuple& o) const { return !(*this == o); }
};

inline IntTuple tup(std::initializer_list<IntTuple> e) { return IntTuple::tuple(std::vector<IntTuple>(e)); }

inline void flatten_into(const IntTuple& t, std::vector<int64_t>& out) {
  if (t.leaf)
    out.push_back(t.v);
  else
    for (const auto& e : t.c) flatten_into(e, out);
}

inline std::vector<int64_t> flatten(const IntTuple& t) {
  std::vector<int64_t> out;
  flatten_into(t, out);
  return out;
}

inline int64_t product(const IntTuple& t) {
  int64_t p = 1;
  for (int64_t x : flatten(t)) p *= x;
  return p;
}

inline bool congruent(const IntTuple& a, const IntTuple& b) {
  if (a.leaf || b.leaf) return a.leaf == b.leaf;
  if (a.c.size() != b.c.size()) return false;
  for (size_t i = 0; i < a.c.size(); ++i)
    if (!congruent(a.c[i], b.c[i])) return false;
  return true;
}

inline std::string to_string(const IntTuple& t) {
  if (t.leaf) return std::to_string(t.v);
  std::string s = "(";
  for (size_t i = 0; i < t.c.size(); ++i) {
    if (i) s += ",";
    s += to_string(t.c[i]);
  }
  return s + ")";
}

// Parses "7", "(4,8)", "((4,8),(2,2,2))".
inline IntTuple parse_int_tuple(const std::string& s, size_t& pos) {
  while (pos < s.size() && s[pos] == ' ') ++pos;
  if (pos < s.size() && s[pos] == '(') {
    ++pos;
    std::vector<IntTuple> elems;
    while (true) {
      elems.push_back(parse_int_tuple(s, pos));
      while (pos < s.size() && s[pos] == ' ') ++pos;
      if (pos < s.size() && s[pos] == ',') {
        ++pos;
        while (pos < s.size() && s[pos] == ' ') ++pos;
        if (pos < s.size() && s[pos] == ')') {  // "(1,)": a one-element tuple
          ++pos;
          break;
        }
        continue;
      }
      if (pos < s.size() && s[pos] == ')') {
        ++pos;
        break;
      }
      throw std::invalid_argument("bad int tuple: " + s);
    }
    return IntTuple::tuple(std::move(elems));
  }
  size_t start = pos;
  if (pos < s.size() && s[pos] == '-') ++pos;
  while (pos < s.size() && s[pos] >= '0' && s[pos] <= '9') ++pos;
  if (start == pos) throw std::invalid_argument("bad int tuple: " + s);
  return IntTuple(std::stoll(s.substr(start, pos - start)));
}

inline IntTuple parse_int_tuple(const std::string& s) {
  size_t pos = 0;
  IntTuple t = parse_int_tuple(s, pos);
  return t;
}

// ------------------------------------------------------------------ Layout
struct Layout {
  IntTuple shape, stride;

  Layout() = default;
  Layout(IntTuple sh, IntTuple st) : shape(std::move(sh)), stride(std::move(st)) {
    if (!congruent(shape, stride)) throw std::invalid_argument("shape and stride are not congruent");
  }
  int64_t size() const { return product(shape); }

  // coordinate (hierarchical, or an integer for any sub-shape) -> index
  int64_t crd2idx(const IntTuple& crd) const { return crd2idx_rec(crd, shape, stride); }
  // flat integer index (colexicographic) -> index
  int64_t operator()(int64_t i) const { return crd2idx_rec(IntTuple(i), shape, stride); }

  int64_t cosize() const {
    int64_t m = 0;
    const auto s = flatten(shape), d = flatten(stride);
    for (size_t i = 0; i < s.size(); ++i)
      if (s[i] > 0) m += (s[i] - 1) * d[i];
    return size() ? m + 1 : 0;
  }

  static int64_t crd2idx_rec(const IntTuple& crd, const IntTuple& sh, const IntTuple& st) {
    if (sh.leaf) {
      if (!crd.leaf) throw std::invalid_argument("coordinate deeper than shape");
      if (crd.v < 0 || (sh.v > 0 && crd.v >= sh.v)) throw std::out_of_range("coordinate outside shape");
      return crd.v * st.v;
    }
    if (crd.leaf) {  // integer into a tuple shape: split colexicographically
      int64_t i = crd.v, acc = 0;
      if (i < 0 || i >= product(sh)) throw std::out_of_range("index outside shape");
      for (size_t m = 0; m < sh.c.size(); ++m) {
        const int64_t n = product(sh.c[m]);
        acc += crd2idx_rec(IntTuple(i % n), sh.c[m], st.c[m]);
        i /= n;
      }
      return acc;
    }
    if (crd.c.size() != sh.c.size()) throw std::invalid_argument("coordinate rank mismatch");
    int64_t acc = 0;
    for (size_t m = 0; m < sh.c.size(); ++m) acc += crd2idx_rec(crd.c[m], sh.c[m], st.c[m]);
    return acc;
  }
};

inline std::string to_string(const Layout& l) { return to_string(l.shape) + ":" + to_string(l.stride); }

inline Layout make_layout(std::vector<Layout> modes) {
  std::vector<IntTuple> s, d;
  for (auto& m : modes) {
    s.push_back(m.shape);
    d.push_back(m.stride);
  }
  return Layout(IntTuple::tuple(s), IntTuple::tuple(d));
}

// Colexicographic integer -> hierarchical coordinate of `shape`.
inline IntTuple idx2crd(int64_t i, const IntTuple& shape) {
  if (shape.leaf) return IntTuple(i);
  std::vector<IntTuple> out;
  for (const auto& s : shape.c) {
    const int64_t n = product(s);
    out.push_back(idx2crd(i % n, s));
    i /= n;
  }
  return IntTuple::tuple(out);
}

// Flat modes (extent, stride), dropping extent-1 modes and merging modes that
// continue one another (stride_{i+1} == extent_i * stride_i): same function.
inline std::vector<std::pair<int64_t, int64_t>> coalesce_modes(const Layout& l) {
  const auto s = flatten(l.shape), d = flatten(l.stride);
  std::vector<std::pair<int64_t, int64_t>> out;
  for (size_t i = 0; i < s.size(); ++i) {
    if (s[i] == 1) continue;
    if (!out.empty() && out.back().first * out.back().second == d[i]) {
      out.back().first *= s[i];
    } else {
      out.push_back({s[i], d[i]});
    }
  }
  if (out.empty()) out.push_back({1, 0});
  return out;
}

inline Layout from_modes(const std::vector<std::pair<int64_t, int64_t>>& m) {
  if (m.size() == 1) return Layout(IntTuple(m[0].first), IntTuple(m[0].second));
  std::vector<IntTuple> s, d;
  for (auto& p : m) {
    s.push_back(IntTuple(p.first));
    d.push_back(IntTuple(p.second));
  }
  return Layout(IntTuple::tuple(s), IntTuple::tuple(d));
}

// complement(L, m): the layout that enumerates, in increasing order, the
// positions L leaves out, repeated until the covered range reaches m.
inline Layout complement(const Layout& l, int64_t m) {
  std::vector<std::pair<int64_t, int64_t>> modes;  // (stride, extent), sorted by stride
  const auto s = flatten(l.shape), d = flatten(l.stride);
  for (size_t i = 0; i < s.size(); ++i)
    if (s[i] != 1 && d[i] != 0) modes.push_back({d[i], s[i]});
  for (size_t i = 1; i < modes.size(); ++i)  // insertion sort (few modes)
    for (size_t j = i; j > 0 && modes[j].first < modes[j - 1].first; --j) std::swap(modes[j], modes[j - 1]);
  std::vector<std::pair<int64_t, int64_t>> out;  // (extent, stride)
  int64_t cur = 1;
  for (auto& [stride, extent] : modes) {
    if (stride % cur != 0) throw std::invalid_argument("complement: layout is not a tiling");
    if (stride / cur > 1) out.push_back({stride / cur, cur});
    cur = extent * stride;
  }
  out.push_back({(m + cur - 1) / cur, cur});
  return from_modes(out);
}

// A o (s:d) for one leaf mode of the right operand.  Walks A's coalesced
// modes, first skipping d elements of A's domain (dividing d out of A's
// shape), then keeping s elements.  Throws when the division is not exact.
inline Layout compose_leaf(const Layout& a, int64_t s, int64_t d) {
  const auto am = coalesce_modes(a);
  if (s == 1) return Layout(IntTuple(1), IntTuple(0));
  if (d == 0) return Layout(IntTuple(s), IntTuple(0));
  std::vector<std::pair<int64_t, int64_t>> out;
  int64_t rest_stride = d, rest_shape = s;
  for (size_t i = 0; i < am.size(); ++i) {
    const int64_t ext = am[i].first, str = am[i].second;
    const bool last = i + 1 == am.size();
    if (last) {  // the last mode of A extends without bound
      out.push_back({rest_shape, rest_stride * str});
      rest_shape = 1;
      break;
    }
    // skip rest_stride elements of this mode
    if (rest_stride >= ext) {
      if (rest_stride % ext != 0) throw std::invalid_argument("composition: stride does not divide");
      rest_stride /= ext;
      continue;
    }
    if (ext % rest_stride != 0) throw std::invalid_argument("composition: stride does not divide");
    const int64_t avail = ext / rest_stride;
    const int64_t take = avail < rest_shape ? avail : rest_shape;
    out.push_back({take, str * rest_stride});
    if (rest_shape % take != 0) throw std::invalid_argument("composition: shape does not divide");
    rest_shape /= take;
    rest_stride = 1;
    if (take < avail) {  // the remaining shape fits inside this mode
      if (rest_shape != 1) throw std::invalid_argument("composition: shape does not divide");
      break;
    }
    if (rest_shape == 1) break;
  }
  if (rest_shape != 1) throw std::invalid_argument("composition: shape does not divide");
  return from_modes(out);
}

inline Layout compose_rec(const Layout& a, const IntTuple& bs, const IntTuple& bd) {
  if (bs.leaf) return compose_leaf(a, bs.v, bd.v);
  std::vector<Layout> modes;
  for (size_t i = 0; i < bs.c.size(); ++i) modes.push_back(compose_rec(a, bs.c[i], bd.c[i]));
  return make_layout(modes);
}

// composition(A, B): the layout R with R(i) = A(B(i)) over B's domain (R's
// shape refines B's shape mode by mode).
inline Layout composition(const Layout& a, const Layout& b) { return compose_rec(a, b.shape, b.stride); }

// logical_divide(L, T) = L o (T, complement(T, size(L))): mode 0 walks one
// tile, mode 1 picks the tile.
inline Layout logical_divide(const Layout& l, const Layout& tiler) {
  return composition(l, make_layout({tiler, complement(tiler, l.size())}));
}

// logical_product(A, B) = (A, complement(A, size(A) * cosize(B)) o B): B's
// pattern of copies of A.
inline Layout logical_product(const Layout& a, const Layout& b) {
  return make_layout({a, composition(complement(a, a.size() * b.cosize()), b)});
}

// ------------------------------------------------------------------ per-mode tiling
// Top-level mode i of a layout (the whole layout for a rank-1 leaf).
inline Layout mode(const Layout& l, size_t i) {
  if (l.shape.leaf) {
    if (i != 0) throw std::out_of_range("mode index");
    return l;
  }
  return Layout(l.shape.c.at(i), l.stride.c.at(i));
}

inline size_t rank(const Layout& l) { return l.shape.rank(); }

// logical_divide applied to each top-level mode with its own tiler:
// result mode i = (tile_i, rest_i).
inline Layout logical_divide_by_mode(const Layout& l, const std::vector<Layout>& tilers) {
  if (tilers.size() != rank(l)) throw std::invalid_argument("one tiler per mode");
  std::vector<Layout> out;
  for (size_t i = 0; i < tilers.size(); ++i) out.push_back(logical_divide(mode(l, i), tilers[i]));
  return make_layout(out);
}

// zipped_divide: the per-mode divide with the tile modes gathered first and
// the rest modes second: ((tile_0, tile_1, ...), (rest_0, rest_1, ...)).
// Mode 0 walks one tile, mode 1 picks the tile.
inline Layout zipped_divide(const Layout& l, const std::vector<Layout>& tilers) {
  const Layout d = logical_divide_by_mode(l, tilers);
  std::vector<Layout> tiles, rests;
  for (size_t i = 0; i < tilers.size(); ++i) {
    const Layout m = mode(d, i);
    tiles.push_back(mode(m, 0));
    rests.push_back(mode(m, 1));
  }
  return make_layout({make_layout(tiles), make_layout(rests)});
}

// tiled_divide: as zipped_divide, with the rest modes flattened into
// top-level modes: ((tile_0, tile_1, ...), rest_0, rest_1, ...), so a tile is
// picked by one index per mode (the way the transpose kernel of "4.21 What
// is CuTe?" indexes (make_coord(_, _), blockIdx.x, blockIdx.y)).
inline Layout tiled_divide(const Layout& l, const std::vector<Layout>& tilers) {
  const Layout z = zipped_divide(l, tilers);
  std::vector<Layout> out{mode(z, 0)};
  const Layout rests = mode(z, 1);
  for (size_t i = 0; i < rank(rests); ++i) out.push_back(mode(rests, i));
  return make_layout(out);
}

// The per-mode position of the thread whose index (thr's value) is `idx`:
// one flat (colexicographic) coordinate per top-level mode of `thr`.
inline std::vector<int64_t> thread_coordinate(const Layout& thr, int64_t idx) {
  for (int64_t i = 0; i < thr.size(); ++i) {
    if (thr(i) != idx) continue;
    std::vector<int64_t> c;
    int64_t rest = i;
    for (size_t m = 0; m < rank(thr); ++m) {
      const int64_t n = product(mode(thr, m).shape);
      c.push_back(rest % n);
      rest /= n;
    }
    return c;
  }
  throw std::invalid_argument("index not in the thread layout's image");
}

// local_partition(tile, thr, idx): the elements of `tile` thread `idx` of the
// thread layout `thr` owns when the tile is split into thr's shape, thread
// (i, j, ...) taking elements (i + T_0 a, j + T_1 b, ...).  Returned as the
// offset of the thread's first element plus the layout of its elements over
// (a, b, ...).  Needs tile extents that the thread extents divide.
struct Partition {
  int64_t offset;
  Layout layout;
};

inline Partition local_partition(const Layout& tile, const Layout& thr, int64_t idx) {
  if (rank(tile) != rank(thr)) throw std::invalid_argument("tile and thread layout ranks differ");
  std::vector<Layout> tilers;
  for (size_t i = 0; i < rank(thr); ++i) {
    const int64_t t = product(mode(thr, i).shape);
    if (product(mode(tile, i).shape) % t != 0) throw std::invalid_argument("thread extent does not divide tile");
    tilers.push_back(Layout(IntTuple(t), IntTuple(1)));
  }
  const Layout z = zipped_divide(tile, tilers);
  const std::vector<int64_t> c = thread_coordinate(thr, idx);
  // offset of the thread's element in tile 0: the tile mode evaluated at c
  const Layout tm = mode(z, 0);
  int64_t off = 0;
  for (size_t i = 0; i < rank(thr); ++i) off += mode(tm, i)(c[i]);
  return Partition{off, mode(z, 1)};
}

// The strip-mined thread map as a layout (thread, vector element, iteration)
// -> offset in a row-major tile of pitch `cols`:
//   ((column_groups, threads / column_groups), vec, iterations)
//   : ((vec, cols), 1, row_stride * cols)
inline Layout stripmined_layout(const StripMined& m) {
  if (!m.valid()) throw std::invalid_argument("strip-mined map: tile, threads and vector do not fit");
  const int64_t cg = m.column_groups();
  return Layout(tup({tup({cg, (int64_t)m.threads / cg}), (int64_t)m.vec, (int64_t)m.iterations()}),
                tup({tup({(int64_t)m.vec, (int64_t)m.cols}), 1, (int64_t)m.row_stride() * m.cols}));
}

}  // namespace layout
}  // namespace ttc
