// Matrix-vector path of the GEMM (one output row or one output column): see gemv.cu.
#pragma once
#include <cuda_runtime.h>

#include <cstdint>

namespace ttc {

// y[i] = act(alpha * sum_k mat[i * ldm + k] x[k * incx] + beta * c[i * incc]
//            + bias[i * incb]),  i < rows,
// rounded to fp16/bf16 and stored at y[i * incy].  c is read only when
// beta != 0; bias may be null (incb = 0 broadcasts bias[0]).
struct GemvParams {
  const uint16_t* mat;
  int64_t ldm;
  const uint16_t* x;
  int64_t incx;
  const uint16_t* c;
  int64_t incc;
  uint16_t* y;
  int64_t incy;
  const float* bias;
  int64_t incb;
  float alpha, beta;
  int rows, K, act, bf16;
  int vec;  // 16-byte vector loads of mat and x are aligned (and incx == 1)
};

cudaError_t launch_gemv_rows(const GemvParams& p, int sm_count, cudaStream_t stream);

// The same sums with the outputs contiguous in the matrix: line k (k < K) at
// mat + k * ldm holds the terms of outputs 0 .. rows - 1,
//   y[i] = act(alpha * sum_k mat[k * ldm + i] x[k * incx] + beta * c[i * incc] + bias[i * incb]).
// vec: 16-byte vector loads of the lines are aligned (mat 16-byte aligned,
// ldm a multiple of 8).
cudaError_t launch_gemv_cols(const GemvParams& p, int sm_count, cudaStream_t stream);

}  // namespace ttc
