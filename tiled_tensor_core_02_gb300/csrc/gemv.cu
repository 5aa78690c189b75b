// Matrix-vector path of the GEMM: D = act(alpha * A * B + beta * C + bias)
// when M == 1 or N == 1.  The problem is then a stream of the matrix operand
// with two FLOPs per element loaded, far below the tensor cores' ridge, so
// CUDA cores in fp32 do the arithmetic and the work is to keep HBM busy:
// no tiles, no TMEM, no cluster set-up on the common path.
//
// The kernel covers the case where the reduction runs along the matrix's
// contiguous dimension: one warp per output, each lane eight 16-byte vectors
// of the row and of x in flight, a shuffle reduction, the epilogue on lane 0.
// (With the outputs contiguous instead, a CTA-per-output-block kernel with a
// cluster reduction over K slices measured slower than the tensor-core
// kernels at 1 x 4096 x 4096, so that case stays on them.)
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "gemm_kernel.cuh"
#include "gemv.cuh"

namespace ttc {

namespace {
constexpr int kThreads = 256;
constexpr int kRowsUnroll = 8;  // vectors in flight per lane

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

}  // namespace

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
