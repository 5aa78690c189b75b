// Out-of-place transpose D = S^T: the layout-only transpose kernel of "4.21
// What is CuTe?" (gpu-glossary-zh), rebuilt for GB300.
//
// The page tiles the source into 32 x 32 blocks (tiled_divide), lets a
// row-major (8, 32) thread layout partition each block (local_partition:
// thread t holds rows t/32 + 8j of column t mod 32), copies the partition into
// registers and writes it back through the column-major view of the output.
// Its loads are coalesced, its stores are not (lanes of a warp write one
// element each to 32 different destination rows).
//
// Here both sides move 16-byte vectors.  A tile is TR source rows x 256 bytes
// (256/E columns for E-byte elements; TR = 64 for 4- and 8-byte elements, 128
// for 1- and 2-byte ones, so destination row segments are 128 bytes or more).
// Load phase: 16 lanes cover one 256-byte source row segment (V = 16/E
// elements per lane), 16 rows per pass, TR/16 passes.
// The tile goes to shared memory with an XOR swizzle at 16-byte granularity
// (chunk' = chunk ^ ((row / V) mod 16)), which keeps both the row-wise vector
// writes and the column-wise element reads of the store phase free of bank
// conflicts.  Store phase: a lane reads V consecutive source rows of one
// 4-byte word and transposes the V x (4/E) block in registers (byte
// permutes) into 4/E destination vectors of 16 bytes (8-byte elements: two
// element reads per vector).  The next tile's loads are issued (into
// registers) before the current tile's stores so their latency overlaps; a
// ring of asynchronous global-to-shared copies in place of the registers was
// measured slower (fewer resident warps to issue the stores).  Unaligned
// pitches or bases and ragged edges fall back to per-element accesses for the
// affected vectors.  Persistent grid over tiles, row-major tile order.
#include <cuda_runtime.h>

#include <cstdint>

#include "transpose.cuh"

namespace ttc {

namespace {
constexpr int kThreads = 256;
constexpr int kRowBytes = 256;     // source bytes per tile row

template <typename T>
struct Geom {
  static constexpr int E = sizeof(T);
  static constexpr int V = 16 / E;              // elements per 16-byte vector
  static constexpr int TR = E >= 4 ? 64 : 128;  // source rows per tile
  static constexpr int TC = kRowBytes / E;      // source columns per tile
  static constexpr int P = TR / 16;             // vectors per thread per phase
  static constexpr int L = TR * E / 16;         // lanes per destination row segment
  static constexpr int DR = kThreads / L;       // destination rows per store pass
  static_assert(DR * P == TC, "store passes cover the tile");
  static_assert((TR / V) <= 16 || E == 8, "swizzle keys distinct within a warp's reads");
};

template <typename T>
union Vec {
  uint4 v;
  T e[16 / sizeof(T)];
};

__device__ __forceinline__ uint32_t swz_offset(int row, int chunk, int key) {
  return (uint32_t)row * kRowBytes + (uint32_t)((chunk ^ key) << 4);
}

template <typename T>
__device__ __forceinline__ void load_tile(const T* __restrict__ src, int64_t lds, int64_t rows, int64_t cols,
                                          bool vec_ok, int64_t r0, int64_t c0, Vec<T> (&buf)[Geom<T>::P]) {
  using G = Geom<T>;
  const int q = threadIdx.x & 15, rr = threadIdx.x >> 4;
  const int64_t c = c0 + (int64_t)q * G::V;
#pragma unroll
  for (int p = 0; p < G::P; ++p) {
    const int64_t r = r0 + rr + 16 * p;
    buf[p].v = make_uint4(0, 0, 0, 0);
    if (r < rows) {
      const T* s = src + r * lds + c;
      if (vec_ok && c + G::V <= cols) {
        buf[p].v = __ldcs(reinterpret_cast<const uint4*>(s));
      } else {
#pragma unroll
        for (int k = 0; k < G::V; ++k)
          if (c + k < cols) buf[p].e[k] = s[k];
      }
    }
  }
}

template <typename T>
__device__ __forceinline__ void store_vec(T* __restrict__ dst, int64_t ldd, int64_t rows, int64_t cols, bool vec_ok,
                                          int64_t drow, int64_t dcol, const Vec<T>& out) {
  using G = Geom<T>;
  if (drow >= cols) return;
  T* d = dst + drow * ldd + dcol;
  if (vec_ok && dcol + G::V <= rows) {
    __stcs(reinterpret_cast<uint4*>(d), out.v);
  } else {
#pragma unroll
    for (int k = 0; k < G::V; ++k)
      if (dcol + k < rows) d[k] = out.e[k];
  }
}

// Store phase for 1-, 2- and 4-byte elements.  The unit of work is (g, w):
// source rows g*V .. g*V+V-1 of 4-byte word w (columns w*R .. w*R+R-1, R =
// 4/E), read as V words and transposed in registers into R destination
// vectors.  A warp takes 8 consecutive g by 4 consecutive w (one 16-byte
// chunk): with the swizzle key g mod 16 the 32 word reads hit 32 banks.
template <typename T>
__device__ __forceinline__ void store_tile_words(const unsigned char* tile, T* __restrict__ dst, int64_t ldd,
                                                 int64_t rows, int64_t cols, bool vec_ok, int64_t r0, int64_t c0) {
  using G = Geom<T>;
  constexpr int NG = G::TR / G::V;  // row groups per tile
  constexpr int NU = NG * (kRowBytes / 4) / kThreads;
  constexpr int R = 4 / G::E;
  static_assert(NG % 8 == 0 && NU >= 1, "warp covers 8 row groups");
#pragma unroll
  for (int p = 0; p < NU; ++p) {
    const int u = p * kThreads + threadIdx.x;
    const int wl = u & 3, gl = (u >> 2) & 7, rest = u >> 5;
    const int g = gl + 8 * (rest % (NG / 8));
    const int w = wl + 4 * (rest / (NG / 8));
    const uint32_t base = swz_offset(g * G::V, w >> 2, g & 15) + ((w & 3) << 2);
    uint32_t a[G::V];
#pragma unroll
    for (int i = 0; i < G::V; ++i) a[i] = *reinterpret_cast<const uint32_t*>(tile + base + i * kRowBytes);
    Vec<T> out[R];
    if constexpr (G::E == 4) {
      out[0].v = make_uint4(a[0], a[1], a[2], a[3]);
    } else if constexpr (G::E == 2) {
      // word k of destination row j pairs half j of rows 2k and 2k+1
      uint32_t lo[4], hi[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        lo[k] = __byte_perm(a[2 * k], a[2 * k + 1], 0x5410);
        hi[k] = __byte_perm(a[2 * k], a[2 * k + 1], 0x7632);
      }
      out[0].v = make_uint4(lo[0], lo[1], lo[2], lo[3]);
      out[1].v = make_uint4(hi[0], hi[1], hi[2], hi[3]);
    } else {
      // 4 x 4 byte transposes: word k of destination row j holds byte j of rows 4k .. 4k+3
      uint32_t y[4][4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint32_t t0 = __byte_perm(a[4 * k], a[4 * k + 1], 0x5140);
        const uint32_t t1 = __byte_perm(a[4 * k], a[4 * k + 1], 0x7362);
        const uint32_t t2 = __byte_perm(a[4 * k + 2], a[4 * k + 3], 0x5140);
        const uint32_t t3 = __byte_perm(a[4 * k + 2], a[4 * k + 3], 0x7362);
        y[0][k] = __byte_perm(t0, t2, 0x5410);
        y[1][k] = __byte_perm(t0, t2, 0x7632);
        y[2][k] = __byte_perm(t1, t3, 0x5410);
        y[3][k] = __byte_perm(t1, t3, 0x7632);
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) out[j].v = make_uint4(y[j][0], y[j][1], y[j][2], y[j][3]);
    }
#pragma unroll
    for (int j = 0; j < R; ++j)
      store_vec<T>(dst, ldd, rows, cols, vec_ok, c0 + (int64_t)w * R + j, r0 + (int64_t)g * G::V, out[j]);
  }
}

// Store phase for 8-byte elements: each lane gathers the V = 2 rows of one
// column with two 8-byte shared loads.
template <typename T>
__device__ __forceinline__ void store_tile_elems(const unsigned char* tile, T* __restrict__ dst, int64_t ldd,
                                                 int64_t rows, int64_t cols, bool vec_ok, int64_t r0, int64_t c0) {
  using G = Geom<T>;
  const int g = threadIdx.x % G::L, drr = threadIdx.x / G::L;
#pragma unroll
  for (int p = 0; p < G::P; ++p) {
    const int dr = drr + G::DR * p;  // destination row in the tile = source column
    const uint32_t base = swz_offset(g * G::V, (dr * G::E) >> 4, g & 15) + ((dr * G::E) & 15);
    Vec<T> out;
#pragma unroll
    for (int i = 0; i < G::V; ++i) out.e[i] = *reinterpret_cast<const T*>(tile + base + i * kRowBytes);
    store_vec<T>(dst, ldd, rows, cols, vec_ok, c0 + dr, r0 + (int64_t)g * G::V, out);
  }
}

template <typename T>
__global__ void __launch_bounds__(kThreads) transpose_kernel(const T* __restrict__ src, int64_t lds,
                                                             T* __restrict__ dst, int64_t ldd, int64_t rows,
                                                             int64_t cols, int src_vec, int dst_vec) {
  using G = Geom<T>;
  __shared__ __align__(128) unsigned char tile[G::TR * kRowBytes];
  const int64_t tiles_r = (rows + G::TR - 1) / G::TR;
  const int64_t tiles_c = (cols + G::TC - 1) / G::TC;
  const int64_t ntiles = tiles_r * tiles_c;
  const int q = threadIdx.x & 15, rr = threadIdx.x >> 4;  // load-phase chunk and row

  Vec<T> buf[G::P];
  int64_t t = blockIdx.x;
  if (t < ntiles) load_tile<T>(src, lds, rows, cols, src_vec, (t / tiles_c) * G::TR, (t % tiles_c) * G::TC, buf);
  for (; t < ntiles; t += gridDim.x) {
    const int64_t r0 = (t / tiles_c) * G::TR;
    const int64_t c0 = (t % tiles_c) * G::TC;
#pragma unroll
    for (int p = 0; p < G::P; ++p) {
      const int row = rr + 16 * p;
      *reinterpret_cast<uint4*>(tile + swz_offset(row, q, (row / G::V) & 15)) = buf[p].v;
    }
    __syncthreads();
    // the next tile's loads go out before this tile's stores
    const int64_t tn = t + gridDim.x;
    if (tn < ntiles)
      load_tile<T>(src, lds, rows, cols, src_vec, (tn / tiles_c) * G::TR, (tn % tiles_c) * G::TC, buf);
    if constexpr (G::E <= 4)
      store_tile_words<T>(tile, dst, ldd, rows, cols, dst_vec, r0, c0);
    else
      store_tile_elems<T>(tile, dst, ldd, rows, cols, dst_vec, r0, c0);
    __syncthreads();
  }
}

template <typename T>
cudaError_t launch_typed(const void* src, int64_t lds, void* dst, int64_t ldd, int64_t rows, int64_t cols,
                         int sm_count, cudaStream_t stream) {
  using G = Geom<T>;
  static int per_sm = 0;  // resident CTAs per SM, queried once per element type
  if (per_sm == 0) {
    int n = 0;
    const cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, transpose_kernel<T>, kThreads, 0);
    if (e != cudaSuccess) return e;
    per_sm = n < 1 ? 1 : n;
  }
  const int64_t tiles = ((rows + G::TR - 1) / G::TR) * ((cols + G::TC - 1) / G::TC);
  int64_t grid = (int64_t)sm_count * per_sm;
  if (grid > tiles) grid = tiles;
  if (grid < 1) grid = 1;
  const auto s = reinterpret_cast<uintptr_t>(src);
  const auto d = reinterpret_cast<uintptr_t>(dst);
  const int src_vec = (s % 16 == 0) && ((lds * G::E) % 16 == 0);
  const int dst_vec = (d % 16 == 0) && ((ldd * G::E) % 16 == 0);
  transpose_kernel<T><<<(unsigned)grid, kThreads, 0, stream>>>(static_cast<const T*>(src), lds, static_cast<T*>(dst),
                                                               ldd, rows, cols, src_vec, dst_vec);
  return cudaGetLastError();
}
}  // namespace

cudaError_t launch_transpose(const void* src, int64_t lds, void* dst, int64_t ldd, int64_t rows, int64_t cols,
                             int elem_bytes, int sm_count, cudaStream_t stream) {
  switch (elem_bytes) {
    case 1:
      return launch_typed<uint8_t>(src, lds, dst, ldd, rows, cols, sm_count, stream);
    case 2:
      return launch_typed<uint16_t>(src, lds, dst, ldd, rows, cols, sm_count, stream);
    case 4:
      return launch_typed<uint32_t>(src, lds, dst, ldd, rows, cols, sm_count, stream);
    case 8:
      return launch_typed<unsigned long long>(src, lds, dst, ldd, rows, cols, sm_count, stream);
    default:
      return cudaErrorInvalidValue;
  }
}

}  // namespace ttc
