// Out-of-place transpose (see transpose.cu).
#pragma once
#include <cuda_runtime.h>

#include <cstdint>

namespace ttc {

// dst (cols x rows, pitch ldd) = src (rows x cols, pitch lds)^T; elements of
// elem_bytes (1, 2, 4 or 8) bytes, row-major.
cudaError_t launch_transpose(const void* src, int64_t lds, void* dst, int64_t ldd, int64_t rows, int64_t cols,
                             int elem_bytes, int sm_count, cudaStream_t stream);

}  // namespace ttc
