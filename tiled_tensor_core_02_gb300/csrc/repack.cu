// Operand repacking for ttc_gemm_ws: copies a matrix whose pitch (or base)
// TMA cannot describe into a workspace with a 16-byte-multiple pitch, so the
// GEMM that follows can stage it with TMA (A, B; C into an aligned copy of D),
// and copies that aligned D back (launch_unpack).
//
// The matrix is taken in memory order: `rows` rows of `cols` contiguous
// elements, `src_ld` elements apart (for a column-major operand the "rows"
// are its columns).  One launch copies up to two matrices (A and B).
#include <cuda_runtime.h>

#include <cstdint>

#include "gemm_kernel.cuh"
#include "repack.cuh"

namespace ttc {

// One matrix of a repack launch, in bytes.
struct RepackJob {
  const uint8_t* src;
  int64_t src_ld;  // bytes between source rows
  int64_t rows;
  int64_t cols;    // bytes per row
  uint8_t* dst;
  int64_t dst_ld;  // bytes between destination rows (a multiple of 16)
  int64_t chunks_per_row;
  int64_t first;   // index of the job's first 16-byte chunk among the launch's chunks
};

struct RepackParams {
  RepackJob job[2];
  int jobs;
  int64_t total;  // chunks of all jobs
};

// Bytes i + phase of the 8-word window go to i (phase 0..15), in stages of
// 8, 4, 2 and 1 bytes.
__device__ __forceinline__ void window8_shift_down(uint32_t (&x)[8], uint32_t phase) {
  const bool s8 = phase & 8, s4 = phase & 4, s2 = phase & 2, s1 = phase & 1;
#pragma unroll
  for (int k = 0; k < 6; ++k) x[k] = s8 ? x[k + 2] : x[k];
#pragma unroll
  for (int k = 0; k < 7; ++k) x[k] = s4 ? x[k + 1] : x[k];
#pragma unroll
  for (int k = 0; k < 7; ++k) x[k] = s2 ? __byte_perm(x[k], x[k + 1], 0x5432) : x[k];
#pragma unroll
  for (int k = 0; k < 7; ++k) x[k] = s1 ? __byte_perm(x[k], x[k + 1], 0x4321) : x[k];
}

// Destination chunk `idx` of the launch (a 16-byte piece of a destination
// row) and its source bytes, which start at any alignment: the one or two
// aligned 16-byte blocks that hold them (only blocks with at least one byte of
// the row's data, so never one outside the memory pages the matrix occupies).
struct RepackChunk {
  uint4 b0, b1;
  uint8_t* dst;
  uint32_t phase;  // source address mod 16
  int n;           // bytes of the row in this chunk (1..16)
};

__device__ __forceinline__ void repack_load(const RepackParams& p, int64_t idx, RepackChunk& c) {
  const RepackJob& j = (p.jobs > 1 && idx >= p.job[1].first) ? p.job[1] : p.job[0];
  // a job's chunk count is below 2^31 (checked on the host): 32-bit division
  const uint32_t q = (uint32_t)(idx - j.first);
  const uint32_t cpr = (uint32_t)j.chunks_per_row;
  const uint32_t r = q / cpr;
  const int64_t c0 = (int64_t)(q - r * cpr) * 16;
  c.n = j.cols - c0 < 16 ? (int)(j.cols - c0) : 16;
  const uint8_t* s = j.src + (int64_t)r * j.src_ld + c0;
  c.phase = (uint32_t)(reinterpret_cast<uintptr_t>(s) & 15u);
  const uint4* blk = reinterpret_cast<const uint4*>(s - c.phase);
  c.b0 = __ldg(blk);
  c.b1 = (int)c.phase + c.n > 16 ? __ldg(blk + 1) : make_uint4(0u, 0u, 0u, 0u);
  c.dst = j.dst + (int64_t)r * j.dst_ld + c0;
}

// Shifts the chunk's bytes into place, zeroes the bytes past the row's end
// (the padding, which TMA never reads since the tensor map keeps the true
// extent) and stores the 16 bytes.
__device__ __forceinline__ void repack_store(const RepackChunk& c) {
  uint32_t x[8] = {c.b0.x, c.b0.y, c.b0.z, c.b0.w, c.b1.x, c.b1.y, c.b1.z, c.b1.w};
  window8_shift_down(x, c.phase);
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int keep = c.n - 4 * k;  // bytes of word k inside the row
    x[k] = keep >= 4 ? x[k] : keep <= 0 ? 0u : (x[k] & ((1u << (8 * keep)) - 1u));
  }
  *reinterpret_cast<uint4*>(c.dst) = make_uint4(x[0], x[1], x[2], x[3]);
}

// Each thread writes destination chunks idx, idx + stride, ..., two per
// iteration with both chunks' loads in flight before either store.
// Launched with programmatic dependent launch: it waits for the previous grid
// before its first global access and lets the next grid (the GEMM, which
// waits for this one in turn) start its prologue.
__global__ void __launch_bounds__(256, 8) repack_rows_kernel(const __grid_constant__ RepackParams p) {
  grid_dependency_wait();
  grid_dependents_launch();
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  for (; idx + stride < p.total; idx += 2 * stride) {
    RepackChunk c0, c1;
    repack_load(p, idx, c0);
    repack_load(p, idx + stride, c1);
    repack_store(c0);
    repack_store(c1);
  }
  if (idx < p.total) {
    RepackChunk c0;
    repack_load(p, idx, c0);
    repack_store(c0);
  }
}

cudaError_t launch_repack2(const RepackSpec* specs, int count, int sm_count, cudaStream_t stream) {
  if (count < 1 || count > 2) return cudaErrorInvalidValue;
  RepackParams p{};
  p.jobs = count;
  int64_t total = 0;
  for (int i = 0; i < count; ++i) {
    const RepackSpec& sp = specs[i];
    RepackJob& j = p.job[i];
    j.src = static_cast<const uint8_t*>(sp.src);
    j.src_ld = sp.src_ld * sp.elem_bytes;
    j.rows = sp.rows;
    j.cols = sp.cols * sp.elem_bytes;
    j.dst = static_cast<uint8_t*>(sp.dst);
    j.dst_ld = sp.dst_ld * sp.elem_bytes;
    if (j.dst_ld % 16 || reinterpret_cast<uintptr_t>(j.dst) % 16 || j.dst_ld < j.cols) return cudaErrorInvalidValue;
    j.chunks_per_row = (j.cols + 15) / 16;
    if (j.rows * j.chunks_per_row >= (int64_t(1) << 31)) return cudaErrorInvalidValue;
    j.first = total;
    total += j.rows * j.chunks_per_row;
  }
  p.total = total;
  if (total == 0) return cudaSuccess;
  int64_t blocks = (total + 255) / 256;
  const int64_t cap = (int64_t)sm_count * 8;
  if (blocks > cap) blocks = cap;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)blocks, 1, 1);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  add_pdl_attribute(cfg, attr);
  const cudaError_t e = cudaLaunchKernelEx(&cfg, repack_rows_kernel, p);
  return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_repack(const void* src, int64_t src_ld, int64_t rows, int64_t cols, void* dst, int64_t dst_ld,
                          int elem_bytes, int sm_count, cudaStream_t stream) {
  const RepackSpec sp{src, src_ld, rows, cols, dst, dst_ld, elem_bytes};
  return launch_repack2(&sp, 1, sm_count, stream);
}

// ---------------------------------------------------------------- int8 -> fp16 widening
// For the CTA-pair int8 path: fp16 copies of the int8 operands, in their own
// layouts, rows padded to whole 16-element chunks.  A chunk is 16 int8 values
// read as one 16-byte vector (its row starts 16-byte aligned, so the vector
// lies inside the row's memory pages) and written as two; values past the
// row's end are written as zero.  Exact: with u = x + 128 (one byte), the fp16
// bit pattern 0x6400 | u is 1024 + u, and subtracting 1152 leaves x.
struct WidenJob {
  const uint8_t* src;
  int64_t src_ld;  // bytes
  int64_t rows, cols;
  uint16_t* dst;
  int64_t dst_ld;  // elements
  int64_t chunks_per_row;
  int64_t first;
};

struct WidenParams {
  WidenJob job[2];
  int jobs;
  int64_t total;
};

struct WidenChunk {
  uint4 v;
  uint16_t* dst;
  int n;  // values of the row in this chunk (1..16)
};

__device__ __forceinline__ void widen_load(const WidenParams& p, int64_t idx, WidenChunk& c) {
  const WidenJob& j = (p.jobs > 1 && idx >= p.job[1].first) ? p.job[1] : p.job[0];
  const uint32_t q = (uint32_t)(idx - j.first);
  const uint32_t cpr = (uint32_t)j.chunks_per_row;
  const uint32_t r = q / cpr;
  const int64_t c0 = (int64_t)(q - r * cpr) * 16;
  c.n = j.cols - c0 < 16 ? (int)(j.cols - c0) : 16;
  c.v = __ldg(reinterpret_cast<const uint4*>(j.src + (int64_t)r * j.src_ld + c0));
  c.dst = j.dst + (int64_t)r * j.dst_ld + c0;
}

__device__ __forceinline__ void widen_store(const WidenChunk& c) {
  const __half2 bias2 = __halves2half2(__ushort_as_half(0x6480u), __ushort_as_half(0x6480u));  // 1152
  const uint32_t ws[4] = {c.v.x, c.v.y, c.v.z, c.v.w};
  uint32_t h[8];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const uint32_t u = ws[k] ^ 0x80808080u;
    uint32_t lo = __byte_perm(u, 0x64646464u, 0x4140);
    uint32_t hi = __byte_perm(u, 0x64646464u, 0x4342);
    const __half2 l2 = __hsub2(*reinterpret_cast<__half2*>(&lo), bias2);
    const __half2 h2 = __hsub2(*reinterpret_cast<__half2*>(&hi), bias2);
    h[2 * k] = *reinterpret_cast<const uint32_t*>(&l2);
    h[2 * k + 1] = *reinterpret_cast<const uint32_t*>(&h2);
  }
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const int keep = c.n - 2 * k;  // values of word k inside the row
    h[k] = keep >= 2 ? h[k] : keep == 1 ? (h[k] & 0xFFFFu) : 0u;
  }
  uint4* d = reinterpret_cast<uint4*>(c.dst);
  d[0] = make_uint4(h[0], h[1], h[2], h[3]);
  d[1] = make_uint4(h[4], h[5], h[6], h[7]);
}

// Two chunks per thread per iteration, both loads in flight before either
// store; programmatic dependent launch as repack_rows_kernel.
__global__ void __launch_bounds__(256, 8) widen_i8_kernel(const __grid_constant__ WidenParams p) {
  grid_dependency_wait();
  grid_dependents_launch();
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  for (; idx + stride < p.total; idx += 2 * stride) {
    WidenChunk c0, c1;
    widen_load(p, idx, c0);
    widen_load(p, idx + stride, c1);
    widen_store(c0);
    widen_store(c1);
  }
  if (idx < p.total) {
    WidenChunk c0;
    widen_load(p, idx, c0);
    widen_store(c0);
  }
}

cudaError_t launch_widen_i8(const WidenSpec* specs, int count, int sm_count, cudaStream_t stream) {
  if (count < 1 || count > 2) return cudaErrorInvalidValue;
  WidenParams p{};
  p.jobs = count;
  int64_t total = 0;
  for (int i = 0; i < count; ++i) {
    const WidenSpec& sp = specs[i];
    WidenJob& j = p.job[i];
    j.src = static_cast<const uint8_t*>(sp.src);
    j.src_ld = sp.src_ld;
    j.rows = sp.rows;
    j.cols = sp.cols;
    j.dst = static_cast<uint16_t*>(sp.dst);
    j.dst_ld = sp.dst_ld;
    j.chunks_per_row = (j.cols + 15) / 16;
    if (reinterpret_cast<uintptr_t>(j.src) % 16 || j.src_ld % 16 || reinterpret_cast<uintptr_t>(j.dst) % 16 ||
        j.dst_ld % 16 || j.dst_ld < j.chunks_per_row * 16 || j.rows * j.chunks_per_row >= (int64_t(1) << 31))
      return cudaErrorInvalidValue;
    j.first = total;
    total += j.rows * j.chunks_per_row;
  }
  p.total = total;
  if (total == 0) return cudaSuccess;
  int64_t blocks = (total + 255) / 256;
  const int64_t cap = (int64_t)sm_count * 8;
  if (blocks > cap) blocks = cap;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)blocks, 1, 1);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  add_pdl_attribute(cfg, attr);
  const cudaError_t e = cudaLaunchKernelEx(&cfg, widen_i8_kernel, p);
  return e != cudaSuccess ? e : cudaGetLastError();
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
