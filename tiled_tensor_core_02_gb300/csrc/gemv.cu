// Matrix-vector path of the GEMM: D = act(alpha * A * B + beta * C + bias)
// when M == 1 or N == 1.  The problem is then a stream of the matrix operand
// with two FLOPs per element loaded, far below the tensor cores' ridge, so
// CUDA cores in fp32 do the arithmetic and the work is to keep HBM busy:
// no tiles, no TMEM, no cluster set-up on the common path.
//
// gemv_rows_kernel covers the case where the reduction runs along the
// matrix's contiguous dimension: one warp per output, each lane sixteen 16-byte
// vectors of the row and of x in flight, a shuffle reduction, the epilogue on
// lane 0.  gemv_cols_kernel covers the other one, where the outputs are
// contiguous in the matrix: a CTA per block of outputs and slice of K, the
// slices of one block in a cluster, added through distributed shared memory.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "gemm_kernel.cuh"
#include "gemv.cuh"

namespace ttc {

namespace {
constexpr int kThreads = 256;
constexpr int kRowsUnroll = 16;  // vectors in flight per lane

template <bool BF16>
__device__ __forceinline__ void epilogue_store(const GemvParams& p, int i, float acc) {
  float v = p.alpha * acc;
  if (p.beta != 0.0f) v = fmaf(p.beta, half_bits_to_float<BF16>(p.c[(int64_t)i * p.incc]), v);
  if (p.bias) v += p.bias[(int64_t)i * p.incb];
  v = apply_act(p.act, v);
  p.y[(int64_t)i * p.incy] = (uint16_t)(pack2<BF16>(v, 0.0f) & 0xFFFFu);
}

__device__ __forceinline__ float dot8(const uint4& a, const uint4& b, float acc, bool bf16) {
  const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, bw[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    float a0, a1, b0, b1;
    if (bf16) {
      a0 = __uint_as_float(aw[j] << 16);
      a1 = __uint_as_float(aw[j] & 0xFFFF0000u);
      b0 = __uint_as_float(bw[j] << 16);
      b1 = __uint_as_float(bw[j] & 0xFFFF0000u);
    } else {
      const float2 af = __half22float2(*reinterpret_cast<const __half2*>(&aw[j]));
      const float2 bf = __half22float2(*reinterpret_cast<const __half2*>(&bw[j]));
      a0 = af.x, a1 = af.y, b0 = bf.x, b1 = bf.y;
    }
    acc = fmaf(a0, b0, acc);
    acc = fmaf(a1, b1, acc);
  }
  return acc;
}

template <bool BF16>
__global__ void __launch_bounds__(kThreads) gemv_rows_kernel(const GemvParams p) {
  const int lane = threadIdx.x & 31;
  const int warps = kThreads / 32;
  grid_dependency_wait();  // every load and store after the previous grid on the stream
  grid_dependents_launch();
  for (int i = blockIdx.x * warps + (threadIdx.x >> 5); i < p.rows; i += gridDim.x * warps) {
    const uint16_t* row = p.mat + (int64_t)i * p.ldm;
    float acc = 0.0f;
    int k0 = 0;
    if (p.vec) {
      // whole 8-element groups, kRowsUnroll per lane in flight
      const int kv = p.K & ~7;
      for (; k0 + kRowsUnroll * 256 <= kv; k0 += kRowsUnroll * 256) {
        uint4 m[kRowsUnroll], x[kRowsUnroll];
#pragma unroll
        for (int u = 0; u < kRowsUnroll; ++u) {
          const int k = k0 + u * 256 + lane * 8;
          m[u] = __ldcs(reinterpret_cast<const uint4*>(row + k));
          x[u] = __ldg(reinterpret_cast<const uint4*>(p.x + k));
        }
#pragma unroll
        for (int u = 0; u < kRowsUnroll; ++u) acc = dot8(m[u], x[u], acc, BF16);
      }
      for (int k = k0 + lane * 8; k + 8 <= kv; k += 256)
        acc = dot8(__ldcs(reinterpret_cast<const uint4*>(row + k)), __ldg(reinterpret_cast<const uint4*>(p.x + k)),
                   acc, BF16);
      k0 = kv;
    }
    for (int k = k0 + lane; k < p.K; k += 32)
      acc = fmaf(half_bits_to_float<BF16>(row[k]), half_bits_to_float<BF16>(p.x[(int64_t)k * p.incx]), acc);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xFFFFFFFFu, acc, o);
    if (lane == 0) epilogue_store<BF16>(p, i, acc);
  }
}

// ---------------------------------------------------------------- outputs contiguous
// Line k of the matrix (k < K) holds the terms of consecutive outputs:
// y[i] = sum_k mat[k * ldm + i] x[k * incx].  A CTA takes kColsBlock outputs
// and one K slice; each half-warp reads 256 contiguous bytes of a line (8
// outputs per lane, one 16-byte vector), the CTA's 16 half-warps take lines
// 16 apart with kColsUnroll lines in flight each.  The half-warps' partial
// sums meet in shared memory; the cluster's CTAs (gridDim.y, the K slices of
// one output block) then hand theirs to the first CTA through distributed
// shared memory, which adds them in slice order and applies the epilogue.
constexpr int kColsBlock = 128;
constexpr int kColsUnroll = 16;

template <bool BF16>
__device__ __forceinline__ void fma8(uint4 w, float xv, float (&acc)[8]) {
  const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    acc[2 * j] = fmaf(half_bits_to_float<BF16>((uint16_t)(ws[j] & 0xFFFFu)), xv, acc[2 * j]);
    acc[2 * j + 1] = fmaf(half_bits_to_float<BF16>((uint16_t)(ws[j] >> 16)), xv, acc[2 * j + 1]);
  }
}

template <bool BF16>
__global__ void __launch_bounds__(kThreads) gemv_cols_kernel(const GemvParams p) {
  __shared__ float part[kThreads / 16][kColsBlock];
  __shared__ float tot[kColsBlock];
  const int tid = threadIdx.x;
  const int hw = tid >> 4;  // half-warp
  const int i0 = blockIdx.x * kColsBlock + (tid & 15) * 8;
  const int slices = gridDim.y;
  const int per = ((p.K + slices - 1) / slices + 15) / 16 * 16;
  const int k_lo = blockIdx.y * per;
  const int k_hi = min(p.K, k_lo + per);
  // whole 16-byte vectors: an aligned line pitch and all 8 outputs inside
  const bool vec = p.vec && i0 + 8 <= p.rows;
  grid_dependency_wait();  // every load and store after the previous grid on the stream
  grid_dependents_launch();
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  if (vec) {
    // every line's 16 bytes and its x issued before the first use
    const uint16_t* base = p.mat + i0;
    for (int k = k_lo + hw; k < k_hi; k += 16 * kColsUnroll) {
      uint4 w[kColsUnroll];
      float xv[kColsUnroll];
#pragma unroll
      for (int u = 0; u < kColsUnroll; ++u) {
        const int kk = k + 16 * u;
        const bool in = kk < k_hi;
        w[u] = in ? __ldcs(reinterpret_cast<const uint4*>(base + (int64_t)kk * p.ldm)) : make_uint4(0u, 0u, 0u, 0u);
        xv[u] = in ? half_bits_to_float<BF16>(p.x[(int64_t)kk * p.incx]) : 0.0f;
      }
#pragma unroll
      for (int u = 0; u < kColsUnroll; ++u) fma8<BF16>(w[u], xv[u], acc);
    }
  } else if (i0 < p.rows) {
    for (int k = k_lo + hw; k < k_hi; k += 16) {
      const uint16_t* line = p.mat + (int64_t)k * p.ldm + i0;
      const float xv = half_bits_to_float<BF16>(p.x[(int64_t)k * p.incx]);
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (i0 + j < p.rows) acc[j] = fmaf(half_bits_to_float<BF16>(line[j]), xv, acc[j]);
    }
  }
#pragma unroll
  for (int j = 0; j < 8; ++j) part[hw][(tid & 15) * 8 + j] = acc[j];
  __syncthreads();
  if (tid < kColsBlock) {
    float s = 0.0f;
#pragma unroll
    for (int h = 0; h < kThreads / 16; ++h) s += part[h][tid];
    tot[tid] = s;
  }
  if (slices == 1) {
    const int i = blockIdx.x * kColsBlock + tid;
    if (tid < kColsBlock && i < p.rows) epilogue_store<BF16>(p, i, tot[tid]);
    return;
  }
  cluster_sync();  // every slice's sums written (release / acquire across the cluster)
  if (blockIdx.y == 0 && tid < kColsBlock) {
    float s = 0.0f;
    for (int r = 0; r < slices; ++r) {
      const uint32_t a = mapa_shared(smem_u32(&tot[tid]), (uint32_t)r);
      float v;
      asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(a) : "memory");
      s += v;
    }
    const int i = blockIdx.x * kColsBlock + tid;
    if (i < p.rows) epilogue_store<BF16>(p, i, s);
  }
  cluster_sync();  // no CTA leaves while the first one may still read its sums
}

}  // namespace

cudaError_t launch_gemv_cols(const GemvParams& p, int sm_count, cudaStream_t stream) {
  const int blocks = (p.rows + kColsBlock - 1) / kColsBlock;
  // K slices per output block (a cluster): up to 8, while the CTAs fit about
  // two per SM and each slice keeps at least 128 lines
  int slices = 1;
  while (slices < 8 && (int64_t)blocks * slices * 2 <= 2 * (int64_t)sm_count && p.K / (slices * 2) >= 128) slices *= 2;
  if (blocks <= 0) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)blocks, (unsigned)slices, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  if (slices > 1) {
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = (unsigned)slices;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  add_pdl_attribute(cfg, attr);
  const cudaError_t le = p.bf16 ? cudaLaunchKernelEx(&cfg, gemv_cols_kernel<true>, p)
                                : cudaLaunchKernelEx(&cfg, gemv_cols_kernel<false>, p);
  if (le != cudaSuccess) return le;
  return cudaGetLastError();
}

cudaError_t launch_gemv_rows(const GemvParams& p, int sm_count, cudaStream_t stream) {
  const int warps = kThreads / 32;
  int64_t grid = (p.rows + warps - 1) / warps;
  const int64_t cap = (int64_t)sm_count * 8;
  if (grid > cap) grid = cap;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  add_pdl_attribute(cfg, attr);
  const cudaError_t le = p.bf16 ? cudaLaunchKernelEx(&cfg, gemv_rows_kernel<true>, p)
                                : cudaLaunchKernelEx(&cfg, gemv_rows_kernel<false>, p);
  if (le != cudaSuccess) return le;
  return cudaGetLastError();
}

}  // namespace ttc
