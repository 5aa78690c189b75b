// Operand repacking for ttc_gemm_ws: copies a matrix whose pitch (or base)
// TMA cannot describe into a workspace with a 16-byte-multiple pitch, so the
// GEMM that follows can stage it with TMA (A, B; C into an aligned copy of D),
// and copies that aligned D back (launch_unpack).
//
// The matrix is taken in memory order: `rows` rows of `cols` contiguous
// elements, `src_ld` elements apart (for a column-major operand the "rows"
// are its columns).  Each thread writes one 16-byte chunk of a destination
// row; elements past `cols` in the last chunk are written as zero (they lie
// in the row's padding, which TMA never reads since the tensor map keeps the
// true extent).  Reads are element-wise (the source is only element-aligned)
// and coalesced across the warp.
#include <cuda_runtime.h>

#include <cstdint>

#include "repack.cuh"

namespace ttc {

template <typename T>
__global__ void __launch_bounds__(256) repack_rows_kernel(const T* __restrict__ src, int64_t src_ld, int64_t rows,
                                                          int64_t cols, T* __restrict__ dst, int64_t dst_ld) {
  constexpr int V = 16 / (int)sizeof(T);
  const int64_t chunks_per_row = (cols + V - 1) / V;
  const int64_t total = rows * chunks_per_row;
  for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = idx / chunks_per_row;
    const int64_t c0 = (idx - r * chunks_per_row) * V;
    const T* s = src + r * src_ld + c0;
    union {
      T e[V];
      uint4 u;
    } v;
#pragma unroll
    for (int j = 0; j < V; ++j) v.e[j] = (c0 + j < cols) ? __ldg(s + j) : T(0);
    *reinterpret_cast<uint4*>(dst + r * dst_ld + c0) = v.u;
  }
}

cudaError_t launch_repack(const void* src, int64_t src_ld, int64_t rows, int64_t cols, void* dst, int64_t dst_ld,
                          int elem_bytes, int sm_count, cudaStream_t stream) {
  const int64_t v = 16 / elem_bytes;
  const int64_t chunks = rows * ((cols + v - 1) / v);
  int64_t blocks = (chunks + 255) / 256;
  const int64_t cap = (int64_t)sm_count * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  if (elem_bytes == 4)
    repack_rows_kernel<uint32_t><<<(unsigned)blocks, 256, 0, stream>>>(
        static_cast<const uint32_t*>(src), src_ld, rows, cols, static_cast<uint32_t*>(dst), dst_ld);
  else if (elem_bytes == 2)
    repack_rows_kernel<uint16_t><<<(unsigned)blocks, 256, 0, stream>>>(
        static_cast<const uint16_t*>(src), src_ld, rows, cols, static_cast<uint16_t*>(dst), dst_ld);
  else
    repack_rows_kernel<uint8_t><<<(unsigned)blocks, 256, 0, stream>>>(
        static_cast<const uint8_t*>(src), src_ld, rows, cols, static_cast<uint8_t*>(dst), dst_ld);
  return cudaGetLastError();
}

// The reverse copy: rows of an aligned, padded-pitch matrix back to a
// destination whose rows are only element-aligned.  Element per thread, so
// each load and store instruction covers 32 consecutive elements of one row;
// blockIdx.x picks a 1024-element column block, blockIdx.y walks the rows.
template <typename T>
__global__ void __launch_bounds__(256) unpack_rows_kernel(const T* __restrict__ src, int64_t src_ld, int64_t rows,
                                                          int64_t cols, T* __restrict__ dst, int64_t dst_ld) {
  constexpr int kPer = 4;
  const int64_t c0 = (int64_t)blockIdx.x * (256 * kPer) + threadIdx.x;
  for (int64_t r = blockIdx.y; r < rows; r += gridDim.y) {
    const T* s = src + r * src_ld;
    T* d = dst + r * dst_ld;
    T v[kPer];
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      const int64_t c = c0 + j * 256;
      v[j] = c < cols ? s[c] : T(0);
    }
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      const int64_t c = c0 + j * 256;
      if (c < cols) d[c] = v[j];
    }
  }
}

cudaError_t launch_unpack(const void* src, int64_t src_ld, int64_t rows, int64_t cols, void* dst, int64_t dst_ld,
                          int elem_bytes, int sm_count, cudaStream_t stream) {
  const int64_t gx = (cols + 1023) / 1024;
  if (gx > 65535 || rows <= 0 || cols <= 0) return rows <= 0 || cols <= 0 ? cudaSuccess : cudaErrorInvalidValue;
  int64_t gy = (int64_t)sm_count * 16 / gx;
  if (gy < 1) gy = 1;
  if (gy > rows) gy = rows;
  if (gy > 65535) gy = 65535;
  const dim3 grid((unsigned)gx, (unsigned)gy);
  if (elem_bytes == 4)
    unpack_rows_kernel<uint32_t><<<grid, 256, 0, stream>>>(static_cast<const uint32_t*>(src), src_ld, rows, cols,
                                                           static_cast<uint32_t*>(dst), dst_ld);
  else if (elem_bytes == 2)
    unpack_rows_kernel<uint16_t><<<grid, 256, 0, stream>>>(static_cast<const uint16_t*>(src), src_ld, rows, cols,
                                                           static_cast<uint16_t*>(dst), dst_ld);
  else
    unpack_rows_kernel<uint8_t><<<grid, 256, 0, stream>>>(static_cast<const uint8_t*>(src), src_ld, rows, cols,
                                                          static_cast<uint8_t*>(dst), dst_ld);
  return cudaGetLastError();
}

}  // namespace ttc
