// Operand repacking into a padded-pitch workspace (see repack.cu).
#pragma once
#include <cuda_runtime.h>

#include <cstdint>

namespace ttc {

// Copies `rows` rows of `cols` elements (elem_bytes = 1, 2 or 4), `src_ld`
// elements apart, to `dst` with pitch `dst_ld` (a multiple of 16 bytes;
// `dst` 16-byte aligned).
struct RepackSpec {
  const void* src;
  int64_t src_ld, rows, cols;
  void* dst;
  int64_t dst_ld;
  int elem_bytes;
};

// One launch for one or two such copies (count 1 or 2).
cudaError_t launch_repack2(const RepackSpec* specs, int count, int sm_count, cudaStream_t stream);

cudaError_t launch_repack(const void* src, int64_t src_ld, int64_t rows, int64_t cols, void* dst, int64_t dst_ld,
                          int elem_bytes, int sm_count, cudaStream_t stream);

// Widens `rows` rows of `cols` int8 values (`src` and `src_ld` in bytes, both
// 16-byte aligned) into fp16 rows at `dst` with pitch `dst_ld` elements (a
// multiple of 16; `dst` 16-byte aligned).  Every int8 value is exact in fp16.
struct WidenSpec {
  const void* src;
  int64_t src_ld, rows, cols;
  void* dst;
  int64_t dst_ld;
};

// One launch for one or two such copies (count 1 or 2).
cudaError_t launch_widen_i8(const WidenSpec* specs, int count, int sm_count, cudaStream_t stream);

// Copies `rows` rows of `cols` elements (elem_bytes = 1, 2 or 4) from `src`
// (pitch `src_ld`) to `dst` (pitch `dst_ld`), element-aligned at both ends.
cudaError_t launch_unpack(const void* src, int64_t src_ld, int64_t rows, int64_t cols, void* dst, int64_t dst_ld,
                          int elem_bytes, int sm_count, cudaStream_t stream);

}  // namespace ttc
