// Host side of the ttc C ABI: argument validation, layout canonicalisation,
// TMA descriptor encoding, planning (tile width, grid, rasterization) and the
// kernel launch.  See include/ttc.h for the contract of each entry point.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <string>
#include <tuple>
#include <utility>

#include "conv_halo.cuh"
#include "gemm2sm_kernel.cuh"
#include "gemm_launch.cuh"
#include "gemv.cuh"
#include "index_maps.hpp"
#include "repack.cuh"
#include "transpose.cuh"
#include "ttc.h"
#include "ttc_layout.hpp"

namespace ttc {

__device__ uint32_t g_device_error;  // first failure code of any kernel on this device

namespace {

std::atomic<int64_t> g_timeout_ns{2000000000ll};
std::atomic<int> g_inject_stall{0};
std::atomic<int> g_force_generic_load{0};
std::atomic<int> g_force_generic_store{0};
std::atomic<int> g_force_tile_n{0};
std::atomic<int> g_pair_mode{0};
std::atomic<int> g_swap_mode{0};
std::atomic<int> g_split_k{0};
std::atomic<int> g_pair_tile_n{0};
std::atomic<int> g_group_m{0};
std::atomic<int> g_conv_halo{0};
std::atomic<int> g_pair_tail{0};
std::atomic<int> g_gemv_off{0};
std::atomic<int> g_pdl_off{0};
std::atomic<int> g_i8_wide{0};
std::atomic<int> g_pair_epi_warps{0};
std::atomic<int64_t> g_launches{0};

constexpr int kMaxDevices = 64;

// Largest size or leading dimension accepted (elements): the kernels index
// rows, columns and k in 32-bit integers and step past the end by up to a
// grid's stride (well under 2^24) before a loop test, which must not wrap.
constexpr int64_t kSizeLimit = (1ll << 31) - (1ll << 24);

struct DeviceInfo {
  bool ready = false;
  int sm_count = 0;
  int pair_clusters[2][4] = {{-1, -1, -1, -1}, {-1, -1, -1, -1}};  // resident CTA pairs [bf16][width 256/224/192/128]
  int halo_clusters[2][2] = {{-1, -1}, {-1, -1}};          // halo convolution pairs [bf16][width 256/128]
  int pair_clusters_i8 = -1;                                // resident CTA pairs of the int8 pair kernel
  int pair_clusters_ew12[2] = {-1, -1};                     // ... of the twelve-epilogue-warp variant [bf16]
  uint32_t* err = nullptr;
};
DeviceInfo g_dev[kMaxDevices];
std::mutex g_mu;

// Planning without a GPU (ttc_gemm_plan): while a thread plans, its calls
// see a device of t_plan_dev.sm_count SMs, skip tensor-map encoding and
// record each launch in *t_plan instead of making it.
thread_local std::string* t_plan = nullptr;
thread_local DeviceInfo t_plan_dev;

// Appends one launch to the plan ("; " between launches).  Returns true when
// the thread is planning, i.e. when the caller must not launch.
bool plan_note(const char* fmt, ...) {
  if (t_plan == nullptr) return false;
  char buf[256];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  if (!t_plan->empty()) *t_plan += "; ";
  *t_plan += buf;
  return true;
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

ttc_status device_info(DeviceInfo** out) {
  if (t_plan != nullptr) {
    *out = &t_plan_dev;
    return TTC_OK;
  }
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return TTC_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceInfo& d = g_dev[dev];
  if (!d.ready) {
    if (cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return TTC_ERR_CUDA;
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) return TTC_ERR_CUDA;
    d.err = static_cast<uint32_t*>(p);
    if (g_encode == nullptr) {
      void* fn = nullptr;
      cudaDriverEntryPointQueryResult q;
      if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
              cudaSuccess ||
          q != cudaDriverEntryPointSuccess || fn == nullptr)
        return TTC_ERR_CUDA;
      g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    }
    d.ready = true;
  }
  *out = &d;
  return TTC_OK;
}

// Batch layout of one operand for the 3-D tensor maps: `count` batches
// `stride` elements apart (count 1 for an unbatched or shared operand).
struct BatchDim {
  uint64_t count = 1;
  uint64_t stride = 0;
};

// 3-D tensor map over a row-major-in-memory view: `inner` contiguous
// elements, `outer` rows `pitch_elems` apart, and the batch dimension.  Boxes
// are box_inner x box_outer x 1.
bool encode_3d(CUtensorMap* m, CUtensorMapDataType dt, int esize, const void* base, uint64_t inner,
               uint64_t outer, uint64_t pitch_elems, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle sw,
               BatchDim bd = BatchDim()) {
  if (t_plan != nullptr) return true;
  const uint64_t pitch = pitch_elems * (uint64_t)esize;
  // one batch: a stride past the matrix (any 16-byte multiple is accepted)
  const uint64_t bstride = bd.count > 1 ? bd.stride * (uint64_t)esize : (pitch * outer + 15) / 16 * 16;
  cuuint64_t dims[3] = {inner, outer, bd.count};
  cuuint64_t strides[2] = {pitch, bstride};
  cuuint32_t box[3] = {box_inner, box_outer, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return g_encode(m, dt, 3, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Tensor map of one operand as its BoxMap describes it: the matrix as stored
// (`rows` x K with K contiguous when k_inner, rows contiguous otherwise), read
// in boxes of box_inner x box_outer.
bool encode_operand(CUtensorMap* m, CUtensorMapDataType dt, int esize, const void* base, int64_t rows, int64_t K,
                    int64_t ld, const BoxMap& bm, CUtensorMapSwizzle sw, BatchDim bd = BatchDim()) {
  return bm.k_inner ? encode_3d(m, dt, esize, base, K, rows, ld, bm.box_inner, bm.box_outer, sw, bd)
                    : encode_3d(m, dt, esize, base, rows, K, ld, bm.box_inner, bm.box_outer, sw, bd);
}

// The kernels' index maps for one tile configuration, derived from the
// layouts once (index_maps.hpp) and kept: they depend only on the key.
struct MapKey {
  int tile_m, tile_n, ctas, a_rows, a_mn, b_mn, esize, swizzled, half_cols;
  bool operator<(const MapKey& o) const {
    return std::tie(tile_m, tile_n, ctas, a_rows, a_mn, b_mn, esize, swizzled, half_cols) <
           std::tie(o.tile_m, o.tile_n, o.ctas, o.a_rows, o.a_mn, o.b_mn, o.esize, o.swizzled, o.half_cols);
  }
};
std::map<MapKey, TileMaps> g_maps;

// Fills `out` with the maps of `k`; false when the derivation fails or does
// not describe the tile the kernels were compiled for (chunk width, one row
// per epilogue thread, a lane per TMEM row).
bool tile_maps(const MapKey& k, TileMaps& out) {
  std::lock_guard<std::mutex> lk(g_mu);
  auto it = g_maps.find(k);
  if (it == g_maps.end()) {
    TileMaps tm;
    try {
      tm = maps::derive(k.tile_m, k.tile_n, k.ctas, k.a_rows, k.a_mn != 0, k.b_mn != 0, k.esize, k.swizzled != 0,
                        k.half_cols);
    } catch (...) {
      return false;
    }
    if (tm.epi_chunk != kEpiCols || tm.epi_row_step != 1 || tm.tmem_row_step != (1u << 16) ||
        tm.tile_m != k.tile_m || tm.tile_n != k.tile_n)
      return false;
    it = g_maps.emplace(k, tm).first;
  }
  out = it->second;
  return true;
}

// Bytes one k-block of an operand's boxes delivers (0 for more boxes than
// the kernels' producers issue: kMaxBoxes, two in the CTA-pair kernel).
int box_bytes(const BoxMap& b, int max_boxes = kMaxBoxes) {
  return b.boxes >= 1 && b.boxes <= max_boxes ? b.boxes * b.smem_step : 0;
}

bool tma_ok(const void* p, int64_t ld, int esize) {
  return (reinterpret_cast<uintptr_t>(p) % 16 == 0) && ((ld * esize) % 16 == 0) && ld * esize < (1ll << 40);
}

// A batch stride TMA can step by: none needed (one batch, or shared), or a
// 16-byte multiple.
bool tma_batch_ok(int64_t batch, int64_t stride, int esize) {
  return batch <= 1 || stride == 0 || ((stride * esize) % 16 == 0 && stride * esize < (1ll << 40));
}

int64_t round_up(int64_t x, int64_t m) { return (x + m - 1) / m * m; }

// Columns of a D row that TMA stores: the whole 16-byte granules.  A tiled
// TMA store clips at a row's end only to 16-byte granularity (measured: with
// N = 300 bf16 columns and a pitch of 304 it also wrote columns 300..303), so
// the tensor map ends at the last whole granule and the epilogue stores the
// rest of the row (under 16 bytes) itself.
int64_t tma_store_cols(int64_t N, int esize) { return N & ~(int64_t)(16 / esize - 1); }

// CTA-pair tile width for an M x N problem (times batch): the width whose
// tiles fill the resident pairs best, weighted by the width's measured
// relative rate (a narrower tile stages more A per column: 1, 0.95, 0.87,
// 0.64 for 256, 224, 192, 128 on bf16 8192^3) and by the share of its last
// column of tiles that lies inside N.  224 and 192 need a K-major B (their
// halves, 112 and 96 columns, are not whole 64-column MN-major slabs).
// bn == 0: no width fits.
struct PairChoice {
  int bn = 0;
  int clusters = 0;
};
PairChoice choose_pair(DeviceInfo* dev, bool bf16, int64_t M, int64_t N, int64_t batch, bool b_mn) {
  const int forced_pbn = g_pair_tile_n.load();
  PairChoice pc;
  double best = -1.0;
  const int widths[4] = {256, 224, 192, 128};
  const double rates[4] = {1.0, 0.95, 0.87, 0.64};
  for (int wi = 0; wi < 4; ++wi) {
    const int w = widths[wi];
    if ((forced_pbn != 0 && w != forced_pbn) || (b_mn && (w == 224 || w == 192))) continue;
    int& cl = dev->pair_clusters[bf16 ? 1 : 0][wi];
    if (cl < 0) {
      std::lock_guard<std::mutex> lk(g_mu);
      if (cl < 0) cl = pair_max_clusters(bf16, w);
    }
    if (cl <= 0) continue;
    const int64_t nb = (N + w - 1) / w;
    const int64_t tiles = batch * ((M + kPairBM - 1) / kPairBM) * nb;
    const int64_t waves = (tiles + cl - 1) / cl;
    const double fill = (double)tiles / (double)(waves * cl);
    const double inside = (double)N / (double)(nb * w);
    const double score = fill * inside * rates[wi];
    if (score > best + 1e-9) {
      best = score;
      pc.bn = w;
      pc.clusters = cl;
    }
  }
  return pc;
}

using EncodeIm2colFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                    const cuuint64_t*, const int*, const int*, cuuint32_t, cuuint32_t,
                                    const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                    CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeIm2colFn g_encode_im2col = nullptr;

// im2col map over an N x H x W x C tensor (16-bit elements, tightly packed):
// boxes of 128 output pixels x 64 channels, 128-byte swizzle.  The bounding
// box of window corners runs from -pad to pad - (taps - 1) dil past the last
// input row/column in each spatial mode, so it holds exactly P x Q corners,
// visited with the convolution's stride.
bool encode_im2col(CUtensorMap* m, CUtensorMapDataType dt, const void* X, int64_t N, int64_t H, int64_t W,
                   int64_t C, int64_t R, int64_t S, int64_t ph, int64_t pw, int64_t sh, int64_t sw, int64_t dh,
                   int64_t dw) {
  if (g_encode_im2col == nullptr) {
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_encode_im2col == nullptr) {
      void* fn = nullptr;
      cudaDriverEntryPointQueryResult q;
      if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeIm2col", &fn, 12000, cudaEnableDefault, &q) !=
              cudaSuccess ||
          q != cudaDriverEntryPointSuccess || fn == nullptr)
        return false;
      g_encode_im2col = reinterpret_cast<EncodeIm2colFn>(fn);
    }
  }
  cuuint64_t dims[4] = {(cuuint64_t)C, (cuuint64_t)W, (cuuint64_t)H, (cuuint64_t)N};
  cuuint64_t strides[3] = {(cuuint64_t)(C * 2), (cuuint64_t)(W * C * 2), (cuuint64_t)(H * W * C * 2)};
  int lower[2] = {(int)-pw, (int)-ph};
  int upper[2] = {(int)(pw - (S - 1) * dw), (int)(ph - (R - 1) * dh)};
  cuuint32_t estr[4] = {1, (cuuint32_t)sw, (cuuint32_t)sh, 1};
  return g_encode_im2col(m, dt, 4, const_cast<void*>(X), dims, strides, lower, upper, kBK, 128, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Tiled map over an N x H x W x C tensor (16-bit elements, tightly packed)
// for the halo convolution: boxes of 64 channels x `wp` pixels x `rows` rows of
// one image, 128-byte swizzle.  The kernel starts each box at pixel -pad_w of
// a row, so a box row is one zero-padded input row.
bool encode_halo(CUtensorMap* m, CUtensorMapDataType dt, const void* X, int64_t N, int64_t H, int64_t W, int64_t C,
                 int64_t wp, int64_t rows) {
  cuuint64_t dims[4] = {(cuuint64_t)C, (cuuint64_t)W, (cuuint64_t)H, (cuuint64_t)N};
  cuuint64_t strides[3] = {(cuuint64_t)(C * 2), (cuuint64_t)(W * C * 2), (cuuint64_t)(H * W * C * 2)};
  cuuint32_t box[4] = {(cuuint32_t)kBK, (cuuint32_t)wp, (cuuint32_t)rows, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  return g_encode(m, dt, 4, const_cast<void*>(X), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Plan of the halo convolution for a unit-stride problem, or ok == false when
// its shape does not fit the kernel: a padded output row of at most 256
// positions, a halo box of at most 256 rows, and two halo buffers plus at
// least two filter stages in shared memory.
struct HaloPlan {
  bool ok = false;
  int bn = 0, wp = 0, rows = 0, tiles_per_img = 0, stages = 0, smem = 0;
  uint32_t tx = 0, bytes = 0;
};
HaloPlan plan_halo(int64_t P, int64_t Q, int64_t K, int64_t R, int64_t S, int64_t dh, int64_t dw) {
  HaloPlan h;
  const int64_t wp = Q + (S - 1) * dw;
  if (wp > 256) return h;
  // rows a tile's taps reach: from its first position's row to its last
  // position shifted by the last tap; 128 j mod wp repeats with period <= wp
  const int64_t tiles_per_img = (P * wp + kBM - 1) / kBM;
  const int64_t reach = (kBM - 1) + (R - 1) * dh * wp + (S - 1) * dw;
  int64_t rows = 0;
  for (int64_t j = 0; j < tiles_per_img && j < 256; ++j) {
    const int64_t r = ((kBM * j) % wp + reach) / wp + 1;
    if (r > rows) rows = r;
  }
  if (rows > 256) return h;
  h.bn = (K % 256 == 0 || K % 256 > 128) ? 256 : 128;
  const int b_half = h.bn / 2 * kBK * 2;
  h.tx = (uint32_t)(rows * wp * kBK * 2);
  h.bytes = (h.tx + 1023u) / 1024u * 1024u;
  const int64_t room = 227 * 1024 - conv_halo_smem_bytes((int)h.bytes, 0, b_half);
  const int64_t stages = room / (kHaloKPS * b_half);
  if (stages < 2) return h;
  h.stages = (int)(stages < kHaloMaxStages ? stages : kHaloMaxStages);
  h.smem = conv_halo_smem_bytes((int)h.bytes, h.stages, b_half);
  h.wp = (int)wp;
  h.rows = (int)rows;
  h.tiles_per_img = (int)tiles_per_img;
  h.ok = true;
  return h;
}

// CTA pairs to launch for `tiles` tiles with `clusters` pairs resident, and
// the work units they walk: a last partial wave of R tiles whose halves fit
// in one wave (2 R <= pairs) runs as 2 R half tiles, as does a problem of at
// most half a wave.  Units from tail_from on are halves.
int split_last_wave(int tiles, int clusters, bool split, int& tail_from, int& num_units) {
  tail_from = tiles;
  num_units = tiles;
  split = split && g_pair_tail.load() == 0;
  if (tiles < clusters) {
    if (split && 2 * tiles <= clusters) {
      tail_from = 0;
      num_units = 2 * tiles;
      return 2 * tiles;
    }
    return tiles;
  }
  const int rest = tiles % clusters;
  if (split && rest > 0 && 2 * rest <= clusters) {
    tail_from = tiles - rest;
    num_units = tiles + rest;
  }
  return clusters;
}

// The GEMM pair kernel's walk.  Only 256-wide pair tiles are halved, so a
// CTA's half of B is one whole 64-column slab when B is MN-major.
int plan_pair_units(GemmParams& prm, int pbn, int clusters) {
  return split_last_wave(prm.num_tiles, clusters, pbn == 256, prm.tail_from, prm.num_units);
}

// int8 on the CTA-pair kernel: ttc_gemm_ws widens A and B into fp16 copies in
// the workspace (in their own layouts, rows padded to 16 elements) and runs
// the pair kernel's int8 variant on them.  Taken for problems of at least
// kI8WideMinTiles 256 x 256 tiles whose operand rows TMA could read as int8
// and whose int32 D TMA can write; the widening reads each operand once and
// writes twice its bytes.  Measured against the single-CTA int8 kernels
// (graph replay): 8192^3 679 vs 1318 us, 4096^3 110 vs 179 us, 2048 x 3000 x
// 1024 (96 tiles) 22.6 vs 24.3 us, but 1536 x 1536 x 4096 (36 tiles) 31.3 vs
// 29.6 us.
constexpr int64_t kI8WideMinTiles = 64;
struct I8Wide {
  bool on = false;
  int64_t a_rows = 0, a_cols = 0, a_ld = 0, b_rows = 0, b_cols = 0, b_ld = 0;
  size_t a_off = 0, b_off = 0, bytes = 0;
};

I8Wide plan_i8_wide(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, ttc_layout layoutA, const void* B,
                    int64_t ldb, ttc_layout layoutB, const void* D, int64_t ldd) {
  I8Wide w;
  const int mode = g_i8_wide.load();
  if (mode == 2 || K <= 0 || M < kPairBM || N < 256) return w;
  if (mode == 0 && ((M + kPairBM - 1) / kPairBM) * ((N + 255) / 256) < kI8WideMinTiles) return w;
  if (!tma_ok(A, lda, 1) || !tma_ok(B, ldb, 1) || !tma_ok(D, ldd, 4)) return w;
  w.a_rows = layoutA == TTC_ROW_MAJOR ? M : K;
  w.a_cols = layoutA == TTC_ROW_MAJOR ? K : M;
  w.b_rows = layoutB == TTC_ROW_MAJOR ? K : N;
  w.b_cols = layoutB == TTC_ROW_MAJOR ? N : K;
  w.a_ld = round_up(w.a_cols, 16);
  w.b_ld = round_up(w.b_cols, 16);
  w.a_off = 0;
  w.b_off = (size_t)round_up(w.a_rows * w.a_ld * 2, 256);
  w.bytes = w.b_off + (size_t)round_up(w.b_rows * w.b_ld * 2, 256);
  w.on = true;
  return w;
}

ttc_status gemm_i8_wide(DeviceInfo* dev, const I8Wide& w, int64_t M, int64_t N, int64_t K, const void* A,
                        int64_t lda, ttc_layout layoutA, const void* B, int64_t ldb, ttc_layout layoutB,
                        const void* C, int64_t ldc, void* D, int64_t ldd, float beta, void* workspace,
                        void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const bool a_mn = layoutA == TTC_COL_MAJOR;
  const bool b_mn = layoutB == TTC_ROW_MAJOR;
  if (dev->pair_clusters_i8 < 0) {
    std::lock_guard<std::mutex> lk(g_mu);
    if (dev->pair_clusters_i8 < 0) dev->pair_clusters_i8 = pair_max_clusters_i8();
  }
  const int clusters = dev->pair_clusters_i8;
  if (clusters <= 0) return TTC_ERR_CUDA;
  GemmParams prm;
  std::memset(&prm, 0, sizeof prm);
  // the maps of the fp16 pair path: 128 A rows and 128 B columns per CTA and
  // k-block, 64-column B boxes for the half units of a last wave
  if (!tile_maps({kPairBM, 256, 2, kBM, a_mn, b_mn, 2, 1, 128}, prm.maps)) return TTC_ERR_UNSUPPORTED;
  if (box_bytes(prm.maps.a, 2) != kABytes || box_bytes(prm.maps.b, 2) != 128 * kBK * 2 ||
      box_bytes(prm.maps.b_half, 2) != 64 * kBK * 2)
    return TTC_ERR_UNSUPPORTED;
  const void* A16 = ws + w.a_off;
  const void* B16 = ws + w.b_off;
  const CUtensorMapDataType f16 = CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  if (!encode_operand(&prm.tmA, f16, 2, A16, M, K, w.a_ld, prm.maps.a, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_operand(&prm.tmB, f16, 2, B16, N, K, w.b_ld, prm.maps.b, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_3d(&prm.tmD, CU_TENSOR_MAP_DATA_TYPE_INT32, 4, D, tma_store_cols(N, 4), M, ldd, kEpiCols, 32,
                 CU_TENSOR_MAP_SWIZZLE_128B))
    return TTC_ERR_CUDA;
  prm.A = A16;
  prm.B = B16;
  prm.lda = w.a_ld;
  prm.ldb = w.b_ld;
  prm.M = (int)M;
  prm.N = (int)N;
  prm.K = (int)K;
  prm.num_m_blocks = (int)((M + kPairBM - 1) / kPairBM);
  prm.num_n_blocks = (int)((N + 255) / 256);
  prm.num_k_blocks = (int)((K + kBK - 1) / kBK);
  prm.tiles_per_batch = prm.num_m_blocks * prm.num_n_blocks;
  prm.num_tiles = prm.tiles_per_batch;
  prm.batch = 1;
  const int gm = g_group_m.load() > 0 ? g_group_m.load() : 8;
  prm.group_m = prm.num_m_blocks < gm ? prm.num_m_blocks : gm;
  prm.ksplit = 1;
  prm.kb_split = prm.num_k_blocks;
  prm.a_mn = a_mn;
  prm.b_mn = b_mn;
  prm.alpha = 1.0f;
  prm.beta = beta;
  prm.C = beta != 0.0f ? C : nullptr;
  prm.ldc = ldc;
  prm.D = D;
  prm.ldd = ldd;
  prm.d_tma = 1;
  prm.err = dev->err;
  prm.timeout_ns = (uint64_t)g_timeout_ns.load();
  prm.inject_stall = g_inject_stall.load();
  const int nclus = plan_pair_units(prm, 256, clusters);
  if (!b_mn && prm.tail_from < prm.num_units) {
    // half units stage only their 64 columns of B per CTA
    if (!encode_operand(&prm.tmBh, f16, 2, B16, N, K, w.b_ld, prm.maps.b_half, CU_TENSOR_MAP_SWIZZLE_128B))
      return TTC_ERR_CUDA;
    prm.b_half_map = 1;
  }
  prm.a_stream = prm.num_n_blocks == 1;
  prm.b_stream = prm.num_m_blocks == 1;
  const WidenSpec specs[2] = {{A, lda, w.a_rows, w.a_cols, ws + w.a_off, w.a_ld},
                              {B, ldb, w.b_rows, w.b_cols, ws + w.b_off, w.b_ld}};
  if (!plan_note("widen_i8 a=%lldx%lld b=%lldx%lld", (long long)w.a_rows, (long long)w.a_cols,
                 (long long)w.b_rows, (long long)w.b_cols) &&
      launch_widen_i8(specs, 2, dev->sm_count, s) != cudaSuccess)
    return TTC_ERR_CUDA;
  g_launches.fetch_add(1);
  if (!plan_note("pair_i8 bn=256 clusters=%d tiles=%d units=%d", nclus, prm.num_tiles, prm.num_units) &&
      launch_pair_i8(prm, nclus, s) != cudaSuccess)
    return TTC_ERR_CUDA;
  g_launches.fetch_add(1);
  return TTC_OK;
}

const char* mode_name(int mode) {
  switch (mode) {
    case kModeTmaF16: return "tma_f16";
    case kModeTmaBF16: return "tma_bf16";
    case kModeGenF16: return "plain_f16";
    case kModeGenBF16: return "plain_bf16";
    case kModeI8: return "plain_i8";
    case kModeI8Tma: return "tma_i8";
    case kModeI8TmemA: return "tma_i8_tmem_a";
    case kModeConvF16: return "conv_f16";
    case kModeConvBF16: return "conv_bf16";
    default: return "?";
  }
}

template <int MODE>
cudaError_t launch_mode(int bn, const GemmParams& prm, int grid, cudaStream_t s) {
  switch (bn) {
    case 256:
      if constexpr (MODE != kModeI8 && MODE != kModeI8Tma && MODE != kModeI8TmemA)
        return launch_gemm<256, MODE>(prm, grid, s);
      return cudaErrorInvalidValue;
    case 128: return launch_gemm<128, MODE>(prm, grid, s);
    case 64: return launch_gemm<64, MODE>(prm, grid, s);
    case 32: return launch_gemm<32, MODE>(prm, grid, s);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch(int mode, int bn, const GemmParams& prm, int grid, cudaStream_t s) {
  switch (mode) {
    case kModeTmaF16: return launch_mode<kModeTmaF16>(bn, prm, grid, s);
    case kModeTmaBF16: return launch_mode<kModeTmaBF16>(bn, prm, grid, s);
    case kModeGenF16: return launch_mode<kModeGenF16>(bn, prm, grid, s);
    case kModeGenBF16: return launch_mode<kModeGenBF16>(bn, prm, grid, s);
    case kModeI8: return launch_mode<kModeI8>(bn, prm, grid, s);
    case kModeI8Tma: return launch_mode<kModeI8Tma>(bn, prm, grid, s);
    case kModeI8TmemA: return launch_mode<kModeI8TmemA>(bn, prm, grid, s);
    case kModeConvF16: return launch_mode<kModeConvF16>(bn, prm, grid, s);
    case kModeConvBF16: return launch_mode<kModeConvBF16>(bn, prm, grid, s);
    default: return cudaErrorInvalidValue;
  }
}

bool ranges_overlap(const void* a, int64_t a_bytes, const void* b, int64_t b_bytes) {
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
  return a0 < b0 + (uintptr_t)b_bytes && b0 < a0 + (uintptr_t)a_bytes;
}


// A size-1 mode leaves its stride free: a 1 x K column-major A with lda = 1
// is the same memory as a row-major one, and so on.  Rewrites such operands
// to the layout whose contiguous mode is the long one.
void canonicalise(int64_t M, int64_t N, int64_t K, ttc_layout& layoutA, int64_t& lda, ttc_layout& layoutB,
                  int64_t& ldb) {
  if (M == 1 && layoutA == TTC_COL_MAJOR && lda == 1) {
    layoutA = TTC_ROW_MAJOR;
    lda = round_up(K > 0 ? K : 1, 16);
  } else if (K == 1 && layoutA == TTC_ROW_MAJOR && lda == 1) {
    layoutA = TTC_COL_MAJOR;
    lda = round_up(M, 16);
  }
  if (N == 1 && layoutB == TTC_ROW_MAJOR && ldb == 1) {
    layoutB = TTC_COL_MAJOR;
    ldb = round_up(K > 0 ? K : 1, 16);
  } else if (K == 1 && layoutB == TTC_COL_MAJOR && ldb == 1) {
    layoutB = TTC_ROW_MAJOR;
    ldb = round_up(N, 16);
  }
}

// Problems the matrix-vector kernels take (after canonicalise): one output row
// (M == 1) or column (N == 1).  The reduction runs along the matrix operand's
// contiguous dimension (gemv_rows_kernel), or the outputs do (gemv_cols_kernel;
// taken when its K slices can fill the SMs, at least 1024 outputs, or K is at
// most 8192).  They read their operands with plain loads and use no workspace.
enum GemvKind { kGemvNone = 0, kGemvRows = 1, kGemvCols = 2 };
GemvKind gemv_kind(int64_t M, int64_t N, int64_t K, ttc_layout layoutA, ttc_layout layoutB, ttc_dtype dtype,
                   int64_t batch) {
  if (K <= 0 || dtype == TTC_I8 || batch != 1 || g_gemv_off.load()) return kGemvNone;
  if ((M == 1 && layoutB == TTC_COL_MAJOR) || (N == 1 && M > 1 && layoutA == TTC_ROW_MAJOR)) return kGemvRows;
  const int64_t outputs = M == 1 ? N : M;
  if (((M == 1 && layoutB == TTC_ROW_MAJOR) || (N == 1 && M > 1 && layoutA == TTC_COL_MAJOR)) &&
      (outputs >= 1024 || K <= 8192))
    return kGemvCols;
  return kGemvNone;
}

bool takes_gemv(int64_t M, int64_t N, int64_t K, ttc_layout layoutA, ttc_layout layoutB, ttc_dtype dtype,
                int64_t batch) {
  return gemv_kind(M, N, K, layoutA, layoutB, dtype, batch) != kGemvNone;
}

// Which operands ttc_gemm_ws copies into its workspace (those TMA cannot
// describe), with their memory-order shape and the padded pitch of the copy.
struct RepackPlan {
  bool a = false, b = false;
  int64_t a_rows = 0, a_cols = 0, a_ld = 0, b_rows = 0, b_cols = 0, b_ld = 0;
  size_t a_off = 0, b_off = 0, bytes = 0;
};

RepackPlan plan_repack(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, ttc_layout layoutA,
                       const void* B, int64_t ldb, ttc_layout layoutB, int esize) {
  RepackPlan r;
  if (K == 0) return r;
  const int64_t per16 = 16 / esize;
  if (!tma_ok(A, lda, esize)) {
    r.a = true;
    r.a_rows = layoutA == TTC_ROW_MAJOR ? M : K;
    r.a_cols = layoutA == TTC_ROW_MAJOR ? K : M;
    r.a_ld = round_up(r.a_cols, per16);
    r.a_off = 0;
    r.bytes = (size_t)round_up(r.a_rows * r.a_ld * esize, 256);
  }
  if (!tma_ok(B, ldb, esize)) {
    r.b = true;
    r.b_rows = layoutB == TTC_ROW_MAJOR ? K : N;
    r.b_cols = layoutB == TTC_ROW_MAJOR ? N : K;
    r.b_ld = round_up(r.b_cols, per16);
    r.b_off = r.bytes;
    r.bytes += (size_t)round_up(r.b_rows * r.b_ld * esize, 256);
  }
  return r;
}

// Aligned copy of D in the workspace, after the operand repack (`after`
// bytes): used when D's rows cannot take TMA stores (pitch or base not
// 16-byte aligned).  C is copied into it too, so the GEMM runs in place on
// aligned rows with TMA stores and vector C loads, and the result is copied
// back.  off/ld/bytes: its place, pitch (elements) and size.
struct DStage {
  bool on = false;
  int64_t ld = 0;
  size_t off = 0, bytes = 0;
};
// Only int32 outputs (int8 problems) are staged: the 16-bit epilogue stores
// rows at any 2-byte boundary itself (aligned 16-byte blocks shifted in
// registers), which measured faster than staging (4099 x 3001 x 1023 bf16,
// beta = 1, tight pitches: 38.6 us per step direct against 52.1 us staged).
DStage plan_dstage(int64_t M, int64_t N, const void* D, int64_t ldd, int esize, size_t after) {
  DStage d;
  if (esize != 4 || M <= 0 || N <= 0 || tma_ok(D, ldd, esize)) return d;
  d.on = true;
  d.ld = round_up(N, 16 / esize);
  d.off = after;
  d.bytes = (size_t)round_up(M * d.ld * esize, 256);
  return d;
}

}  // namespace

bool pdl_enabled() { return g_pdl_off.load() == 0; }

}  // namespace ttc

using namespace ttc;

extern "C" {

const char* ttc_status_string(ttc_status s) {
  switch (s) {
    case TTC_OK: return "TTC_OK";
    case TTC_ERR_INVALID_ARG: return "TTC_ERR_INVALID_ARG";
    case TTC_ERR_UNSUPPORTED: return "TTC_ERR_UNSUPPORTED";
    case TTC_ERR_CUDA: return "TTC_ERR_CUDA";
    case TTC_ERR_TIMEOUT: return "TTC_ERR_TIMEOUT";
    case TTC_ERR_SCRATCH_TOO_SMALL: return "TTC_ERR_SCRATCH_TOO_SMALL";
  }
  return "TTC_UNKNOWN_STATUS";
}

ttc_status ttc_set_knob(ttc_knob knob, int64_t value) {
  switch (knob) {
    case TTC_KNOB_TIMEOUT_NS: g_timeout_ns.store(value > 0 ? value : 2000000000ll); return TTC_OK;
    case TTC_KNOB_INJECT_STALL:
      if (value != 0 && value != 1) return TTC_ERR_INVALID_ARG;
      g_inject_stall.store((int)value);
      return TTC_OK;
    case TTC_KNOB_FORCE_GENERIC_LOAD:
      if (value != 0 && value != 1) return TTC_ERR_INVALID_ARG;
      g_force_generic_load.store((int)value);
      return TTC_OK;
    case TTC_KNOB_FORCE_GENERIC_STORE:
      if (value != 0 && value != 1) return TTC_ERR_INVALID_ARG;
      g_force_generic_store.store((int)value);
      return TTC_OK;
    case TTC_KNOB_TILE_N:
      if (value != 0 && value != 256 && value != 128 && value != 64 && value != 32 && value != 16)
        return TTC_ERR_INVALID_ARG;
      g_force_tile_n.store((int)value);
      return TTC_OK;
    case TTC_KNOB_PAIR:
      if (value < 0 || value > 2) return TTC_ERR_INVALID_ARG;
      g_pair_mode.store((int)value);
      return TTC_OK;
    case TTC_KNOB_SWAP_AB:
      if (value < 0 || value > 2) return TTC_ERR_INVALID_ARG;
      g_swap_mode.store((int)value);
      return TTC_OK;
    case TTC_KNOB_SPLIT_K:
      if (value < 0 || value > 8) return TTC_ERR_INVALID_ARG;
      g_split_k.store((int)value);
      return TTC_OK;
    case TTC_KNOB_GROUP_M:
      if (value < 0 || value > 64) return TTC_ERR_INVALID_ARG;
      g_group_m.store((int)value);
      return TTC_OK;
    case TTC_KNOB_GEMV:
      if (value < 0 || value > 1) return TTC_ERR_INVALID_ARG;
      g_gemv_off.store((int)value);
      return TTC_OK;
    case TTC_KNOB_PAIR_EPI_WARPS:
      if (value != 0 && value != 8 && value != 12) return TTC_ERR_INVALID_ARG;
      g_pair_epi_warps.store((int)value);
      return TTC_OK;
    case TTC_KNOB_I8_WIDE:
      if (value < 0 || value > 2) return TTC_ERR_INVALID_ARG;
      g_i8_wide.store((int)value);
      return TTC_OK;
    case TTC_KNOB_PAIR_TAIL:
      if (value < 0 || value > 1) return TTC_ERR_INVALID_ARG;
      g_pair_tail.store((int)value);
      return TTC_OK;
    case TTC_KNOB_PDL:
      if (value < 0 || value > 1) return TTC_ERR_INVALID_ARG;
      g_pdl_off.store((int)value);
      return TTC_OK;
    case TTC_KNOB_CONV_HALO:
      if (value < 0 || value > 2) return TTC_ERR_INVALID_ARG;
      g_conv_halo.store((int)value);
      return TTC_OK;
    case TTC_KNOB_PAIR_TILE_N:
      if (value != 0 && value != 256 && value != 224 && value != 192 && value != 128) return TTC_ERR_INVALID_ARG;
      g_pair_tile_n.store((int)value);
      return TTC_OK;
  }
  return TTC_ERR_INVALID_ARG;
}

int64_t ttc_launch_count(void) { return g_launches.load(); }

ttc_status ttc_get_device_error(void* stream) {
  DeviceInfo* dev = nullptr;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return TTC_ERR_CUDA;
  ttc_status st = device_info(&dev);
  if (st != TTC_OK) return st;
  uint32_t v = 0;
  if (cudaMemcpy(&v, dev->err, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess) return TTC_ERR_CUDA;
  if (v != 0) {
    const uint32_t zero = 0;
    if (cudaMemcpy(dev->err, &zero, sizeof zero, cudaMemcpyHostToDevice) != cudaSuccess) return TTC_ERR_CUDA;
    return TTC_ERR_TIMEOUT;
  }
  return TTC_OK;
}

static ttc_status gemm_impl(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, ttc_layout layoutA,
                            const void* B, int64_t ldb, ttc_layout layoutB, const void* C, int64_t ldc, void* D,
                            int64_t ldd, float alpha, float beta, const float* bias, ttc_act act, ttc_dtype dtype,
                            void* workspace, size_t workspace_bytes, void* stream, int64_t batch = 1,
                            int64_t sA = 0, int64_t sB = 0, int64_t sC = 0, int64_t sD = 0) {
  // ------------------------------------------------------------ validation
  if (M < 0 || N < 0 || K < 0 || batch < 0 || sA < 0 || sB < 0 || sC < 0 || sD < 0) return TTC_ERR_INVALID_ARG;
  if ((layoutA != TTC_ROW_MAJOR && layoutA != TTC_COL_MAJOR) ||
      (layoutB != TTC_ROW_MAJOR && layoutB != TTC_COL_MAJOR))
    return TTC_ERR_INVALID_ARG;
  if (act != TTC_ACT_NONE && act != TTC_ACT_RELU && act != TTC_ACT_GELU_TANH) return TTC_ERR_INVALID_ARG;
  if (dtype != TTC_F16 && dtype != TTC_BF16 && dtype != TTC_I8) return TTC_ERR_INVALID_ARG;
  if (M == 0 || N == 0 || batch == 0) return TTC_OK;
  const int64_t a_min = layoutA == TTC_ROW_MAJOR ? K : M;
  const int64_t b_min = layoutB == TTC_ROW_MAJOR ? N : K;
  if (lda < (a_min > 1 ? a_min : 1) || ldb < (b_min > 1 ? b_min : 1) || ldd < N) return TTC_ERR_INVALID_ARG;
  if (beta != 0.0f && (C == nullptr || ldc < N)) return TTC_ERR_INVALID_ARG;
  if (D == nullptr) return TTC_ERR_INVALID_ARG;
  if (K > 0 && (A == nullptr || B == nullptr)) return TTC_ERR_INVALID_ARG;
  const int out_esize = dtype == TTC_I8 ? 4 : 2;
  if (beta != 0.0f) {
    const int64_t c_bytes = ((M - 1) * ldc + N) * out_esize;
    const int64_t d_bytes = ((M - 1) * ldd + N) * out_esize;
    const bool in_place = (C == D) && (ldc == ldd) && (sC == sD);
    if (!in_place && ranges_overlap(C, c_bytes, D, d_bytes)) return TTC_ERR_INVALID_ARG;
  }
  // the batches of D may not overlap one another
  if (batch > 1 && sD < (M - 1) * ldd + N) return TTC_ERR_INVALID_ARG;
  if (dtype == TTC_I8 &&
      (bias != nullptr || act != TTC_ACT_NONE || alpha != 1.0f || (beta != 0.0f && beta != 1.0f)))
    return TTC_ERR_UNSUPPORTED;
  const int64_t lim = kSizeLimit;
  if (M > lim || N > lim || K > lim || lda > lim || ldb > lim || ldc > lim || ldd > lim || batch > 65535)
    return TTC_ERR_UNSUPPORTED;
  const int in_esize = dtype == TTC_I8 ? 1 : 2;
  // every pointer must be aligned to its element type
  if ((K > 0 && (reinterpret_cast<uintptr_t>(A) % in_esize || reinterpret_cast<uintptr_t>(B) % in_esize)) ||
      reinterpret_cast<uintptr_t>(D) % out_esize || (beta != 0.0f && reinterpret_cast<uintptr_t>(C) % out_esize) ||
      reinterpret_cast<uintptr_t>(bias) % 4)
    return TTC_ERR_INVALID_ARG;

  DeviceInfo* dev = nullptr;
  ttc_status st = device_info(&dev);
  if (st != TTC_OK) return st;

  // ------------------------------------------------------------ canonicalisation
  canonicalise(M, N, K, layoutA, lda, layoutB, ldb);
  if (M == 1 && !tma_ok(D, ldd, out_esize) && reinterpret_cast<uintptr_t>(D) % 16 == 0) ldd = round_up(N, 16);

  // ------------------------------------------------------------ matrix-vector problems
  // One output row (M == 1) or column (N == 1) whose reduction runs along the
  // matrix operand's contiguous dimension streams that operand with two FLOPs
  // per element: CUDA-core kernel, one warp per output, no tiles.
  const GemvKind gk = gemv_kind(M, N, K, layoutA, layoutB, dtype, batch);
  if (gk != kGemvNone) {
    GemvParams gp;
    std::memset(&gp, 0, sizeof gp);
    if (M == 1) {
      // D[0, n] = sum_k A[0, k] B[k, n]: column n of B is K-contiguous (rows
      // kernel), or row k of B is N-contiguous (cols kernel); same pointer and pitch
      gp.x = static_cast<const uint16_t*>(A);
      gp.incx = layoutA == TTC_ROW_MAJOR ? 1 : lda;
      gp.mat = static_cast<const uint16_t*>(B);
      gp.ldm = ldb;
      gp.rows = (int)N;
      gp.incy = 1;
      gp.incc = 1;
      gp.incb = 1;
    } else {
      // D[m, 0] = sum_k A[m, k] B[k, 0]: row m of A is K-contiguous (rows
      // kernel), or column k of A is M-contiguous (cols kernel)
      gp.x = static_cast<const uint16_t*>(B);
      gp.incx = layoutB == TTC_COL_MAJOR ? 1 : ldb;
      gp.mat = static_cast<const uint16_t*>(A);
      gp.ldm = lda;
      gp.rows = (int)M;
      gp.incy = ldd;
      gp.incc = ldc;
      gp.incb = 0;  // the bias is per output column: one value for the single column
    }
    gp.K = (int)K;
    gp.y = static_cast<uint16_t*>(D);
    gp.c = beta != 0.0f ? static_cast<const uint16_t*>(C) : nullptr;
    gp.bias = bias;
    gp.alpha = alpha;
    gp.beta = beta;
    gp.act = (int)act;
    gp.bf16 = dtype == TTC_BF16;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (gk == kGemvRows) {
      gp.vec = reinterpret_cast<uintptr_t>(gp.mat) % 16 == 0 && gp.ldm % 8 == 0 && gp.incx == 1 &&
               reinterpret_cast<uintptr_t>(gp.x) % 16 == 0;
      if (!plan_note("gemv_rows vec=%d", gp.vec) && launch_gemv_rows(gp, dev->sm_count, s) != cudaSuccess)
        return TTC_ERR_CUDA;
    } else {
      gp.vec = reinterpret_cast<uintptr_t>(gp.mat) % 16 == 0 && gp.ldm % 8 == 0;
      if (!plan_note("gemv_cols vec=%d", gp.vec) && launch_gemv_cols(gp, dev->sm_count, s) != cudaSuccess)
        return TTC_ERR_CUDA;
    }
    g_launches.fetch_add(1);
    return TTC_OK;
  }

  // ------------------------------------------------------------ int8 on the CTA-pair kernel (workspace)
  if (dtype == TTC_I8 && batch == 1 && workspace != nullptr && reinterpret_cast<uintptr_t>(workspace) % 256 == 0 &&
      !g_force_generic_load.load() && !g_force_generic_store.load()) {
    const I8Wide w = plan_i8_wide(M, N, K, A, lda, layoutA, B, ldb, layoutB, D, ldd);
    if (w.on && w.bytes <= workspace_bytes)
      return gemm_i8_wide(dev, w, M, N, K, A, lda, layoutA, B, ldb, layoutB, C, ldc, D, ldd, beta, workspace,
                          stream);
  }

  // ------------------------------------------------------------ workspace: repack what TMA cannot read
  if (batch == 1 && workspace != nullptr && reinterpret_cast<uintptr_t>(workspace) % 256 == 0 &&
      !g_force_generic_load.load()) {
    const RepackPlan rp = plan_repack(M, N, K, A, lda, layoutA, B, ldb, layoutB, in_esize);
    const bool use_rp = rp.bytes > 0 && rp.bytes <= workspace_bytes;
    const DStage ds = plan_dstage(M, N, D, ldd, out_esize, use_rp ? rp.bytes : 0);
    if (use_rp) {
      // one launch copies both operands
      uint8_t* ws = static_cast<uint8_t*>(workspace);
      RepackSpec specs[2];
      int n = 0;
      if (rp.a) specs[n++] = RepackSpec{A, lda, rp.a_rows, rp.a_cols, ws + rp.a_off, rp.a_ld, in_esize};
      if (rp.b) specs[n++] = RepackSpec{B, ldb, rp.b_rows, rp.b_cols, ws + rp.b_off, rp.b_ld, in_esize};
      if (!plan_note("repack a=%d b=%d", rp.a ? 1 : 0, rp.b ? 1 : 0) &&
          launch_repack2(specs, n, dev->sm_count, static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return TTC_ERR_CUDA;
      g_launches.fetch_add(1);
      if (rp.a) {
        A = ws + rp.a_off;
        lda = rp.a_ld;
      }
      if (rp.b) {
        B = ws + rp.b_off;
        ldb = rp.b_ld;
      }
    }
    if (ds.on && ds.off + ds.bytes <= workspace_bytes && !g_force_generic_store.load()) {
      // D staged: C copied in, the GEMM run in place on aligned rows (the
      // operands already repacked, so no workspace), the result copied out
      uint8_t* dst = static_cast<uint8_t*>(workspace) + ds.off;
      cudaStream_t s = static_cast<cudaStream_t>(stream);
      if (beta != 0.0f) {
        if (!plan_note("stage_c") && launch_repack(C, ldc, M, N, dst, ds.ld, out_esize, dev->sm_count, s) != cudaSuccess)
          return TTC_ERR_CUDA;
        g_launches.fetch_add(1);
      }
      st = gemm_impl(M, N, K, A, lda, layoutA, B, ldb, layoutB, beta != 0.0f ? dst : nullptr, ds.ld, dst, ds.ld,
                     alpha, beta, bias, act, dtype, nullptr, 0, stream);
      if (st != TTC_OK) return st;
      if (!plan_note("unstage_d") && launch_unpack(dst, ds.ld, M, N, D, ldd, out_esize, dev->sm_count, s) != cudaSuccess)
        return TTC_ERR_CUDA;
      g_launches.fetch_add(1);
      return TTC_OK;
    }
  }

  // ------------------------------------------------------------ orientation, tile width, K split
  // The kernel tile is 128 rows by bn columns.  Score each orientation (D
  // itself, or D^T = B^T A^T with a transposed store) and tile width by the
  // CTAs it can keep busy, counting a split of K over a cluster of up to 8
  // CTAs when the tiles alone cannot fill the SMs, weighted by how fast one
  // CTA runs at that width: a narrow tile re-reads its A operand from shared
  // memory for fewer columns, so it reaches a smaller share of the tensor rate
  // (relative rates 1, 0.7, 0.45, 0.3 for widths 256, 128, 64, 32).  Ties keep
  // the wider tile, then the untransposed orientation.
  const int forced_bn = g_force_tile_n.load();
  const int swap_mode = g_swap_mode.load();
  const int forced_split = g_split_k.load();
  const int max_bn = dtype == TTC_I8 ? 128 : 256;
  const int64_t nkb_total = (K + kBK - 1) / kBK;
  bool swap = swap_mode == 1;
  int bn = forced_bn;
  int ksplit = 1;
  // A split must keep at least 16 k-blocks per CTA: with fewer, the exchange
  // of partial sums costs more than the shorter main loop saves (measured on
  // 512^3 and 1024^3 under graph replay: 11.5 vs 7.1 us and 13.2 vs 9.3 us).
  auto split_for = [&](int64_t tiles, int cand) {
    int sp = 1;
    if (dtype == TTC_I8 || cand > 128) return sp;  // split-K exchange buffers exist up to width 128
    while (sp < 8 && tiles * sp * 2 <= dev->sm_count && nkb_total / (sp * 2) >= 16) sp *= 2;
    return sp;
  };
  {
    double best_score = -1.0;
    for (int sw = 0; sw < 2; ++sw) {
      if ((swap_mode == 1 && sw == 0) || (swap_mode == 2 && sw == 1)) continue;
      const int64_t mk = sw ? N : M, nk = sw ? M : N;
      // the kernel's B operand is MN-major when it is stored that way
      const bool bk_mn = sw ? layoutA == TTC_COL_MAJOR : layoutB == TTC_ROW_MAJOR;
      for (int cand = max_bn; cand >= 32; cand /= 2) {
        if (forced_bn != 0 && cand != forced_bn) continue;
        if (bk_mn && cand < 64) continue;
        // a tile wider than the padded N only wastes work (but an MN-major B
        // needs whole 64-column slabs, so 64 stays a candidate for it)
        if (forced_bn == 0 && cand > (bk_mn ? 64 : 32) && cand / 2 >= nk) continue;
        const int64_t tiles = batch * ((mk + kBM - 1) / kBM) * ((nk + cand - 1) / cand);
        const int sp = forced_bn == 0 ? split_for(tiles, cand) : 1;
        const double rate = cand == 256 ? 1.0 : cand == 128 ? 0.7 : cand == 64 ? 0.45 : 0.3;
        const double ctas = (double)(tiles * sp < dev->sm_count ? tiles * sp : dev->sm_count);
        const double score = ctas * rate;
        if (score > best_score + 1e-9) {
          best_score = score;
          bn = cand;
          swap = sw == 1;
          ksplit = sp;
        }
      }
    }
    if (best_score < 0) return TTC_ERR_UNSUPPORTED;
  }
  // HBM-bound skinny problems (one side at most 64): stream the long operand
  // through the 128-row side of the MMA, so every pipeline stage carries a
  // full 16 KB of it, and split K across the CTAs of a cluster until the
  // tiles fill the SMs.  Partial tiles are summed through distributed shared
  // memory, with no workspace.
  if (dtype != TTC_I8 && forced_bn == 0 && swap_mode == 0 && (M < N ? M : N) <= 64 && nkb_total >= 8) {
    swap = N > M;
    const int64_t mk = swap ? N : M, nk = swap ? M : N;
    const bool bk_mn = swap ? layoutA == TTC_COL_MAJOR : layoutB == TTC_ROW_MAJOR;
    bn = (bk_mn || nk > 32) ? 64 : 32;
    const int64_t tiles = batch * ((mk + kBM - 1) / kBM) * ((nk + bn - 1) / bn);
    ksplit = 1;
    while (ksplit < 8 && tiles * ksplit * 2 <= dev->sm_count && nkb_total / (ksplit * 2) >= 4) ksplit *= 2;
  }
  if (forced_split > 0) ksplit = dtype == TTC_I8 ? 1 : forced_split;
  if (ksplit > 1 && bn > 128) bn = 128;  // split-K exchange buffers exist for tiles up to 128 wide

  if (swap) {
    // D^T (N x M, stored as D with the roles of ldd's axes exchanged) = B^T A^T:
    // B^T is B read with the other layout, and likewise A^T
    std::swap(M, N);
    std::swap(A, B);
    std::swap(lda, ldb);
    std::swap(sA, sB);
    const ttc_layout la = layoutA;
    layoutA = layoutB == TTC_ROW_MAJOR ? TTC_COL_MAJOR : TTC_ROW_MAJOR;
    layoutB = la == TTC_ROW_MAJOR ? TTC_COL_MAJOR : TTC_ROW_MAJOR;
  }

  const bool a_mn = layoutA == TTC_COL_MAJOR;
  const bool b_mn = layoutB == TTC_ROW_MAJOR;

  // ------------------------------------------------------------ plan
  const bool load_tma = dtype != TTC_I8 && !g_force_generic_load.load() &&
                        (K == 0 || (tma_ok(A, lda, 2) && tma_ok(B, ldb, 2) && tma_batch_ok(batch, sA, 2) &&
                                    tma_batch_ok(batch, sB, 2)));
  const bool load_tma_i8 = dtype == TTC_I8 && !g_force_generic_load.load() &&
                           (K == 0 || (tma_ok(A, lda, 1) && tma_ok(B, ldb, 1) && tma_batch_ok(batch, sA, 1) &&
                                       tma_batch_ok(batch, sB, 1)));
  int mode;
  if (dtype == TTC_I8)
    // a K-major A is widened straight into tensor memory (less shared-memory
    // traffic per k-block than staging its fp16 copy in shared memory)
    mode = load_tma_i8 ? (a_mn ? kModeI8Tma : kModeI8TmemA) : kModeI8;
  else if (load_tma)
    mode = dtype == TTC_BF16 ? kModeTmaBF16 : kModeTmaF16;
  else
    mode = dtype == TTC_BF16 ? kModeGenBF16 : kModeGenF16;
  const bool store_tma = !swap && tma_ok(D, ldd, out_esize) && tma_batch_ok(batch, sD, out_esize) &&
                         tma_store_cols(N, out_esize) > 0 && !g_force_generic_store.load();
  // batch dimensions of the tensor maps: a shared operand (stride 0) keeps one batch
  const BatchDim bdA{batch > 1 && sA != 0 ? (uint64_t)batch : 1u, (uint64_t)sA};
  const BatchDim bdB{batch > 1 && sB != 0 ? (uint64_t)batch : 1u, (uint64_t)sB};
  const BatchDim bdD{batch > 1 ? (uint64_t)batch : 1u, (uint64_t)sD};
  if (bn == 16 || (b_mn && bn < 64) || bn > max_bn) return TTC_ERR_UNSUPPORTED;

  static_assert(sizeof(GemmParams) <= 4096, "kernel parameter space");
  GemmParams prm;
  std::memset(&prm, 0, sizeof prm);
  const CUtensorMapDataType dt = dtype == TTC_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  // rows of A worth loading per tile: all 128, or only those that exist (the
  // raw int8 staging always takes whole 128-row boxes)
  const bool staged_i8 = mode == kModeI8Tma || mode == kModeI8TmemA;
  const int a_rows = M >= kBM || staged_i8 ? kBM : (int)round_up(M, 8);
  // the kernel's index maps: tile origins, TMA boxes (128-byte swizzled slabs,
  // or the unswizzled int8 staging tiles) and the epilogue's thread maps
  if (!tile_maps({kBM, bn, 1, a_rows, a_mn, b_mn, in_esize, !staged_i8, 0}, prm.maps))
    return TTC_ERR_UNSUPPORTED;
  // the boxes must fit the kernel's shared-memory slots (raw int8 staging: one
  // byte per element)
  const int slot_esize = staged_i8 ? 1 : 2;
  const int a_bytes = box_bytes(prm.maps.a), b_bytes = box_bytes(prm.maps.b);
  if (a_bytes == 0 || a_bytes > kBM * kBK * slot_esize || b_bytes == 0 || b_bytes > bn * kBK * slot_esize)
    return TTC_ERR_UNSUPPORTED;
  if (K > 0 && staged_i8) {
    // the A tile that is widened into tensor memory row by row is written with
    // the 64-byte swizzle (64-byte rows), so the converters read it without
    // bank conflicts
    const CUtensorMapDataType d8 = CU_TENSOR_MAP_DATA_TYPE_UINT8;
    const CUtensorMapSwizzle swa = mode == kModeI8TmemA ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_NONE;
    const bool ok = encode_operand(&prm.tmA, d8, 1, A, M, K, lda, prm.maps.a, swa, bdA) &&
                    encode_operand(&prm.tmB, d8, 1, B, N, K, ldb, prm.maps.b, CU_TENSOR_MAP_SWIZZLE_NONE, bdB);
    if (!ok) return TTC_ERR_CUDA;
  }
  if (K > 0 && (mode == kModeTmaF16 || mode == kModeTmaBF16)) {
    const bool ok = encode_operand(&prm.tmA, dt, 2, A, M, K, lda, prm.maps.a, CU_TENSOR_MAP_SWIZZLE_128B, bdA) &&
                    encode_operand(&prm.tmB, dt, 2, B, N, K, ldb, prm.maps.b, CU_TENSOR_MAP_SWIZZLE_128B, bdB);
    if (!ok) return TTC_ERR_CUDA;
  }
  if (store_tma) {
    const bool ok = dtype == TTC_I8
                        ? encode_3d(&prm.tmD, CU_TENSOR_MAP_DATA_TYPE_INT32, 4, D, tma_store_cols(N, 4), M, ldd,
                                    kEpiCols, 32, CU_TENSOR_MAP_SWIZZLE_128B, bdD)
                        : encode_3d(&prm.tmD, dt, 2, D, tma_store_cols(N, 2), M, ldd, kEpiCols, 32,
                                    CU_TENSOR_MAP_SWIZZLE_64B, bdD);
    if (!ok) return TTC_ERR_CUDA;
  }

  // generic producers: 8-element groups load as one vector when every group
  // start is aligned (16 bytes for 16-bit types, 8 bytes for int8), in every
  // batch: the batch stride keeps each batch's start aligned too
  const int vec_bytes = 8 * in_esize;
  auto vec_ok = [&](const void* base, int64_t ld, int64_t bs) {
    return reinterpret_cast<uintptr_t>(base) % vec_bytes == 0 && (ld * in_esize) % vec_bytes == 0 &&
           (batch <= 1 || (bs * in_esize) % vec_bytes == 0);
  };
  prm.A = A;
  prm.B = B;
  prm.lda = lda;
  prm.ldb = ldb;
  prm.a_vec = vec_ok(A, lda, sA);
  prm.b_vec = vec_ok(B, ldb, sB);
  prm.M = (int)M;
  prm.N = (int)N;
  prm.K = (int)K;
  prm.num_m_blocks = (int)((M + kBM - 1) / kBM);
  prm.num_n_blocks = (int)((N + bn - 1) / bn);
  prm.num_k_blocks = (int)((K + kBK - 1) / kBK);
  prm.tiles_per_batch = prm.num_m_blocks * prm.num_n_blocks;
  prm.num_tiles = (int)batch * prm.tiles_per_batch;
  prm.batch = (int)batch;
  prm.a_bc = bdA.count > 1 ? 1 : 0;
  prm.b_bc = bdB.count > 1 ? 1 : 0;
  prm.a_bs = sA;
  prm.b_bs = sB;
  prm.c_bs = sC;
  prm.d_bs = sD;
  const int gm1 = g_group_m.load() > 0 ? g_group_m.load() : 16;
  prm.group_m = prm.num_m_blocks < gm1 ? prm.num_m_blocks : gm1;
  prm.ksplit = ksplit;
  prm.kb_split = (int)((prm.num_k_blocks + ksplit - 1) / ksplit);
  prm.a_mn = a_mn;
  prm.b_mn = b_mn;
  prm.alpha = alpha;
  prm.beta = beta;
  prm.C = beta != 0.0f ? C : nullptr;
  prm.ldc = ldc;
  prm.D = D;
  prm.ldd = ldd;
  prm.bias = bias;
  prm.act = (int)act;
  prm.stage_tx = (uint32_t)(box_bytes(prm.maps.a) + box_bytes(prm.maps.b));
  prm.d_tma = store_tma ? 1 : 0;
  prm.d_trans = swap ? 1 : 0;
  prm.err = dev->err;
  prm.timeout_ns = (uint64_t)g_timeout_ns.load();
  prm.inject_stall = g_inject_stall.load();

  // CTA-pair kernel: fp16/bf16 operands staged by TMA, a 256 x 256 tile per
  // pair of SMs; chosen for problems at least one pair tile in each direction
  const int pair_mode = g_pair_mode.load();
  const bool pair_ok = (mode == kModeTmaF16 || mode == kModeTmaBF16) && forced_bn == 0 && !swap && ksplit == 1;
  if (pair_ok && pair_mode != 2 && (pair_mode == 1 || (M >= kPairBM && N >= 256))) {
    const bool bf16 = dtype == TTC_BF16;
    const PairChoice pc = choose_pair(dev, bf16, M, N, batch, b_mn);
    const int pbn = pc.bn, clusters = pc.clusters;
    const int64_t pair_tiles = pbn ? batch * ((M + kPairBM - 1) / kPairBM) * ((N + pbn - 1) / pbn) : 0;
    if (pbn != 0 && (pair_mode == 1 || pair_tiles * 4 >= dev->sm_count)) {
      // each CTA of the pair stages 128 rows of A and its pbn / 2 columns of B
      // per k-block; only 256-wide tiles are halved for a last wave
      if (!tile_maps({kPairBM, pbn, 2, kBM, a_mn, b_mn, 2, 1, pbn == 256 ? pbn / 2 : 0}, prm.maps))
        return TTC_ERR_UNSUPPORTED;
      if (box_bytes(prm.maps.a, 2) != kABytes || box_bytes(prm.maps.b, 2) != pbn / 2 * kBK * 2 ||
          (pbn == 256 && box_bytes(prm.maps.b_half, 2) != pbn / 4 * kBK * 2))
        return TTC_ERR_UNSUPPORTED;
      if (K > 0) {
        const bool ok = encode_operand(&prm.tmA, dt, 2, A, M, K, lda, prm.maps.a, CU_TENSOR_MAP_SWIZZLE_128B, bdA) &&
                        encode_operand(&prm.tmB, dt, 2, B, N, K, ldb, prm.maps.b, CU_TENSOR_MAP_SWIZZLE_128B, bdB);
        if (!ok) return TTC_ERR_CUDA;
      }
      prm.num_m_blocks = (int)((M + kPairBM - 1) / kPairBM);
      prm.num_n_blocks = (int)((N + pbn - 1) / pbn);
      prm.tiles_per_batch = prm.num_m_blocks * prm.num_n_blocks;
      prm.num_tiles = (int)batch * prm.tiles_per_batch;
      const int gm = g_group_m.load() > 0 ? g_group_m.load() : 8;
      prm.group_m = prm.num_m_blocks < gm ? prm.num_m_blocks : gm;
      const int nclus = plan_pair_units(prm, pbn, clusters);
      if (K > 0 && !b_mn && prm.tail_from < prm.num_units) {
        // half units stage only their pbn / 4 columns of B per CTA
        if (!encode_operand(&prm.tmBh, dt, 2, B, N, K, ldb, prm.maps.b_half, CU_TENSOR_MAP_SWIZZLE_128B, bdB))
          return TTC_ERR_CUDA;
        prm.b_half_map = 1;
      }
      prm.a_stream = prm.num_n_blocks == 1;
      prm.b_stream = prm.num_m_blocks == 1;
      // rows TMA cannot store (written with plain stores, and C read from such
      // rows too): twelve epilogue warps instead of eight drain a tile sooner
      const int ew = g_pair_epi_warps.load();
      if (!store_tma && pbn == 256 && ew != 8) {
        int& cl12 = dev->pair_clusters_ew12[bf16 ? 1 : 0];
        if (cl12 < 0) {
          std::lock_guard<std::mutex> lk(g_mu);
          if (cl12 < 0) cl12 = pair_max_clusters_ew12(bf16);
        }
        if (cl12 >= nclus) {
          if (!plan_note("pair bn=256 ew=12 clusters=%d tiles=%d units=%d d_tma=0", nclus, prm.num_tiles,
                         prm.num_units) &&
              launch_pair_ew12(bf16, prm, nclus, static_cast<cudaStream_t>(stream)) != cudaSuccess)
            return TTC_ERR_CUDA;
          g_launches.fetch_add(1);
          return TTC_OK;
        }
      }
      if (!plan_note("pair bn=%d ew=8 clusters=%d tiles=%d units=%d d_tma=%d", pbn, nclus, prm.num_tiles,
                     prm.num_units, prm.d_tma) &&
          launch_pair(bf16, pbn, prm, nclus, static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return TTC_ERR_CUDA;
      g_launches.fetch_add(1);
      return TTC_OK;
    }
  }

  prm.a_stream = prm.num_n_blocks == 1;
  prm.b_stream = prm.num_m_blocks == 1;
  const int max_clusters = dev->sm_count / ksplit > 0 ? dev->sm_count / ksplit : 1;
  const int clusters = prm.num_tiles < max_clusters ? prm.num_tiles : max_clusters;
  if (!plan_note("single mode=%s bn=%d ksplit=%d swap=%d grid=%d tiles=%d d_tma=%d a_vec=%d b_vec=%d",
                 mode_name(mode), bn, ksplit, swap ? 1 : 0, clusters * ksplit, prm.num_tiles, prm.d_tma,
                 prm.a_vec, prm.b_vec) &&
      launch(mode, bn, prm, clusters * ksplit, static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return TTC_ERR_CUDA;
  g_launches.fetch_add(1);
  return TTC_OK;
}

ttc_status ttc_gemm(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, ttc_layout layoutA, const void* B,
                    int64_t ldb, ttc_layout layoutB, const void* C, int64_t ldc, void* D, int64_t ldd, float alpha,
                    float beta, const float* bias, ttc_act act, ttc_dtype dtype, void* stream) {
  return gemm_impl(M, N, K, A, lda, layoutA, B, ldb, layoutB, C, ldc, D, ldd, alpha, beta, bias, act, dtype, nullptr,
                   0, stream);
}

ttc_status ttc_gemm_ws(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, ttc_layout layoutA, const void* B,
                       int64_t ldb, ttc_layout layoutB, const void* C, int64_t ldc, void* D, int64_t ldd, float alpha,
                       float beta, const float* bias, ttc_act act, ttc_dtype dtype, void* workspace,
                       size_t workspace_bytes, void* stream) {
  return gemm_impl(M, N, K, A, lda, layoutA, B, ldb, layoutB, C, ldc, D, ldd, alpha, beta, bias, act, dtype, workspace,
                   workspace_bytes, stream);
}

ttc_status ttc_gemm_strided_batched(int64_t batch, int64_t M, int64_t N, int64_t K, const void* A, int64_t lda,
                                    int64_t strideA, ttc_layout layoutA, const void* B, int64_t ldb,
                                    int64_t strideB, ttc_layout layoutB, const void* C, int64_t ldc,
                                    int64_t strideC, void* D, int64_t ldd, int64_t strideD, float alpha, float beta,
                                    const float* bias, ttc_act act, ttc_dtype dtype, void* stream) {
  return gemm_impl(M, N, K, A, lda, layoutA, B, ldb, layoutB, C, ldc, D, ldd, alpha, beta, bias, act, dtype, nullptr,
                   0, stream, batch, strideA, strideB, strideC, strideD);
}

ttc_status ttc_gemm_plan(int64_t batch, int64_t M, int64_t N, int64_t K, const void* A, int64_t lda,
                         int64_t strideA, ttc_layout layoutA, const void* B, int64_t ldb, int64_t strideB,
                         ttc_layout layoutB, const void* C, int64_t ldc, int64_t strideC, void* D, int64_t ldd,
                         int64_t strideD, float alpha, float beta, const float* bias, ttc_act act, ttc_dtype dtype,
                         void* workspace, size_t workspace_bytes, int sm_count, char* out, size_t out_len) {
  if (sm_count < 2 || sm_count > 4096 || (out == nullptr && out_len > 0)) return TTC_ERR_INVALID_ARG;
  std::string plan;
  t_plan_dev = DeviceInfo();
  t_plan_dev.ready = true;
  t_plan_dev.sm_count = sm_count;
  // one CTA pair (or one twelve-warp pair, or one halo pair) per two SMs
  const int pairs = sm_count / 2;
  for (auto& row : t_plan_dev.pair_clusters)
    for (int& v : row) v = pairs;
  for (auto& row : t_plan_dev.halo_clusters)
    for (int& v : row) v = pairs;
  t_plan_dev.pair_clusters_i8 = pairs;
  t_plan_dev.pair_clusters_ew12[0] = t_plan_dev.pair_clusters_ew12[1] = pairs;
  t_plan = &plan;
  const ttc_status st = gemm_impl(M, N, K, A, lda, layoutA, B, ldb, layoutB, C, ldc, D, ldd, alpha, beta, bias, act,
                                  dtype, workspace, workspace_bytes, nullptr, batch, strideA, strideB, strideC,
                                  strideD);
  t_plan = nullptr;
  if (out_len > 0) {
    const size_t n = plan.size() < out_len - 1 ? plan.size() : out_len - 1;
    std::memcpy(out, plan.data(), n);
    out[n] = '\0';
  }
  return st;
}

ttc_status ttc_conv2d_fprop(int64_t N, int64_t H, int64_t W, int64_t C, int64_t K, int64_t R, int64_t S,
                            int64_t pad_h, int64_t pad_w, int64_t stride_h, int64_t stride_w, int64_t dil_h,
                            int64_t dil_w, const void* X, const void* Wt, const void* Cm, int64_t ldc, void* D,
                            int64_t ldd, float alpha, float beta, const float* bias, ttc_act act, ttc_dtype dtype,
                            void* stream) {
  // ------------------------------------------------------------ validation
  if (N < 0 || H < 1 || W < 1 || C < 0 || K < 0 || R < 1 || S < 1 || pad_h < 0 || pad_w < 0 || stride_h < 1 ||
      stride_w < 1 || dil_h < 1 || dil_w < 1)
    return TTC_ERR_INVALID_ARG;
  if (act != TTC_ACT_NONE && act != TTC_ACT_RELU && act != TTC_ACT_GELU_TANH) return TTC_ERR_INVALID_ARG;
  if (dtype == TTC_I8) return TTC_ERR_UNSUPPORTED;
  if (dtype != TTC_F16 && dtype != TTC_BF16) return TTC_ERR_INVALID_ARG;
  // every spatial quantity the kernel forms (p sh - ph + r dh, ...) must stay far inside int
  const int64_t small = 1ll << 24;
  if (H > small || W > small || pad_h > small || pad_w > small || stride_h > small || stride_w > small ||
      dil_h > small || dil_w > small || R > small || S > small || dil_h * (R - 1) > small || dil_w * (S - 1) > small)
    return TTC_ERR_UNSUPPORTED;
  const int64_t span_h = H + 2 * pad_h - dil_h * (R - 1) - 1, span_w = W + 2 * pad_w - dil_w * (S - 1) - 1;
  if (span_h < 0 || span_w < 0) return TTC_ERR_INVALID_ARG;  // the filter does not fit the padded input
  const int64_t P = span_h / stride_h + 1, Q = span_w / stride_w + 1;
  if (N == 0 || K == 0) return TTC_OK;
  const int64_t lim = kSizeLimit;
  if (N > lim / (P * Q) || N > lim / (H * W) || C > lim / (R * S) || K > lim || ldd > lim || ldc > lim)
    return TTC_ERR_UNSUPPORTED;
  const int64_t M = N * P * Q, Kg = R * S * C;
  if (D == nullptr || ldd < K) return TTC_ERR_INVALID_ARG;
  if (beta != 0.0f && (Cm == nullptr || ldc < K)) return TTC_ERR_INVALID_ARG;
  if (Kg > 0 && (X == nullptr || Wt == nullptr)) return TTC_ERR_INVALID_ARG;
  if ((Kg > 0 && (reinterpret_cast<uintptr_t>(X) % 2 || reinterpret_cast<uintptr_t>(Wt) % 2)) ||
      reinterpret_cast<uintptr_t>(D) % 2 || (beta != 0.0f && reinterpret_cast<uintptr_t>(Cm) % 2) ||
      reinterpret_cast<uintptr_t>(bias) % 4)
    return TTC_ERR_INVALID_ARG;
  if (beta != 0.0f) {
    const int64_t c_bytes = ((M - 1) * ldc + K) * 2, d_bytes = ((M - 1) * ldd + K) * 2;
    const bool in_place = Cm == D && ldc == ldd;
    if (!in_place && ranges_overlap(Cm, c_bytes, D, d_bytes)) return TTC_ERR_INVALID_ARG;
  }
  if (Kg > 0 && ranges_overlap(X, N * H * W * C * 2, D, ((M - 1) * ldd + K) * 2)) return TTC_ERR_INVALID_ARG;
  DeviceInfo* dev = nullptr;
  ttc_status st = device_info(&dev);
  if (st != TTC_OK) return st;

  // ------------------------------------------------------------ plan: 128-pixel tiles, tile width by SM fill
  const int forced_bn = g_force_tile_n.load();
  int bn = 0;
  double best = -1.0;
  for (int cand = 256; cand >= 32; cand /= 2) {
    if (forced_bn != 0 && cand != forced_bn) continue;
    if (forced_bn == 0 && cand > 32 && cand / 2 >= K) continue;
    const int64_t tiles = ((M + kBM - 1) / kBM) * ((K + cand - 1) / cand);
    const double rate = cand == 256 ? 1.0 : cand == 128 ? 0.7 : cand == 64 ? 0.45 : 0.3;
    const double score = (double)(tiles < dev->sm_count ? tiles : dev->sm_count) * rate;
    if (score > best + 1e-9) {
      best = score;
      bn = cand;
    }
  }
  if (bn == 0) return TTC_ERR_UNSUPPORTED;
  const int mode = dtype == TTC_BF16 ? kModeConvBF16 : kModeConvF16;
  const bool store_tma = tma_ok(D, ldd, 2) && tma_store_cols(K, 2) > 0 && !g_force_generic_store.load();

  GemmParams prm;
  std::memset(&prm, 0, sizeof prm);
  const CUtensorMapDataType dt = dtype == TTC_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  if (store_tma && !encode_3d(&prm.tmD, dt, 2, D, tma_store_cols(K, 2), M, ldd, kEpiCols, 32, CU_TENSOR_MAP_SWIZZLE_64B))
    return TTC_ERR_CUDA;
  // the im2col A and the filters are both K-major operands
  if (!tile_maps({kBM, bn, 1, kBM, 0, 0, 2, 1, 0}, prm.maps)) return TTC_ERR_UNSUPPORTED;
  prm.A = X;
  prm.lda = Kg;
  prm.B = Wt;  // B(kk, k) = Wt[k Kg + kk]: the K-major ("column-major") B operand
  prm.ldb = Kg > 0 ? Kg : 1;
  prm.a_vec = C % 8 == 0 && reinterpret_cast<uintptr_t>(X) % 16 == 0;
  prm.b_vec = reinterpret_cast<uintptr_t>(Wt) % 16 == 0 && (Kg * 2) % 16 == 0;
  prm.M = (int)M;
  prm.N = (int)K;
  prm.K = (int)Kg;
  prm.num_m_blocks = (int)((M + kBM - 1) / kBM);
  prm.num_n_blocks = (int)((K + bn - 1) / bn);
  prm.num_k_blocks = (int)((Kg + kBK - 1) / kBK);
  prm.tiles_per_batch = prm.num_m_blocks * prm.num_n_blocks;
  prm.num_tiles = prm.tiles_per_batch;
  prm.batch = 1;
  const int gm = g_group_m.load() > 0 ? g_group_m.load() : 16;
  prm.group_m = prm.num_m_blocks < gm ? prm.num_m_blocks : gm;
  prm.ksplit = 1;
  prm.kb_split = prm.num_k_blocks;
  prm.alpha = alpha;
  prm.beta = beta;
  prm.C = beta != 0.0f ? Cm : nullptr;
  prm.ldc = ldc;
  prm.D = D;
  prm.ldd = ldd;
  prm.bias = bias;
  prm.act = (int)act;
  prm.d_tma = store_tma ? 1 : 0;
  prm.err = dev->err;
  prm.timeout_ns = (uint64_t)g_timeout_ns.load();
  prm.inject_stall = g_inject_stall.load();
  prm.cv_h = (int)H;
  prm.cv_w = (int)W;
  prm.cv_c = (int)(C > 0 ? C : 1);
  prm.cv_p = (int)P;
  prm.cv_q = (int)Q;
  prm.cv_s = (int)S;
  prm.cv_ph = (int)pad_h;
  prm.cv_pw = (int)pad_w;
  prm.cv_sh = (int)stride_h;
  prm.cv_sw = (int)stride_w;
  prm.cv_dh = (int)dil_h;
  prm.cv_dw = (int)dil_w;

  // Unit stride: the halo kernel, when whole 64-channel blocks, output
  // channels in 32-column chunks and 16-byte aligned rows of X, D and C let it
  // run, and its plan fits
  const int halo_mode = g_conv_halo.load();
  const bool c_rows16 = beta == 0.0f || (reinterpret_cast<uintptr_t>(Cm) % 16 == 0 && ldc % 8 == 0);
  if (halo_mode != 2 && stride_h == 1 && stride_w == 1 && C > 0 && C % kBK == 0 && K % 32 == 0 &&
      reinterpret_cast<uintptr_t>(X) % 16 == 0 && tma_ok(Wt, Kg, 2) && reinterpret_cast<uintptr_t>(D) % 16 == 0 &&
      ldd % 8 == 0 && c_rows16 && !g_force_generic_load.load() && forced_bn == 0 &&
      (halo_mode == 1 || (M >= kPairBM && K >= 128))) {
    const HaloPlan hpn = plan_halo(P, Q, K, R, S, dil_h, dil_w);
    const int64_t img_pairs = (N + 1) / 2, n_blocks = (K + hpn.bn - 1) / (hpn.bn > 0 ? hpn.bn : 1);
    if (hpn.ok && img_pairs * hpn.tiles_per_img * n_blocks <= lim) {
      const bool bf16 = dtype == TTC_BF16;
      int& cl = dev->halo_clusters[bf16 ? 1 : 0][hpn.bn == 256 ? 0 : 1];
      if (cl < 0) {
        std::lock_guard<std::mutex> lk(g_mu);
        if (cl < 0) cl = conv_halo_max_clusters(bf16, hpn.bn);
      }
      if (cl > 0) {
        ConvHaloParams hp;
        std::memset(&hp, 0, sizeof hp);
        if (!encode_halo(&prm.tmA, dt, X, N, H, W, C, hpn.wp, hpn.rows) ||
            !encode_3d(&prm.tmB, dt, 2, Wt, Kg, K, Kg, kBK, hpn.bn / 2, CU_TENSOR_MAP_SWIZZLE_128B))
          return TTC_ERR_CUDA;
        hp.g = prm;
        hp.n_img = (int)N;
        hp.img_pairs = (int)img_pairs;
        hp.tiles_per_img = hpn.tiles_per_img;
        hp.n_blocks = (int)n_blocks;
        hp.num_tiles = (int)(img_pairs * hpn.tiles_per_img * n_blocks);
        hp.wp = hpn.wp;
        hp.p = (int)P;
        hp.q = (int)Q;
        hp.c = (int)C;
        hp.cblk = (int)(C / kBK);
        hp.taps = (int)(R * S);
        hp.s = (int)S;
        hp.row_step = (int)(dil_h * hpn.wp);
        hp.dw = (int)dil_w;
        hp.ph = (int)pad_h;
        hp.pw = (int)pad_w;
        hp.halo_rows = hpn.rows;
        hp.halo_tx = hpn.tx;
        hp.halo_bytes = hpn.bytes;
        hp.stages = hpn.stages;
        const int nclus = split_last_wave(hp.num_tiles, cl, hpn.bn == 256, hp.tail_from, hp.num_units);
        if (launch_conv_halo(bf16, hpn.bn, hp, hpn.smem, nclus, static_cast<cudaStream_t>(stream)) != cudaSuccess)
          return TTC_ERR_CUDA;
        g_launches.fetch_add(1);
        return TTC_OK;
      }
    }
  }

  // CTA-pair kernel with im2col TMA loads: whole 64-channel blocks per filter
  // tap, window corners and tap offsets inside the ranges an im2col map of two
  // spatial modes accepts ([-128, 127] and [0, 255]), strides up to 8, and at
  // least one 256-pixel pair tile
  const int pair_mode = g_pair_mode.load();
  const bool im2col_ok = C > 0 && C % kBK == 0 && reinterpret_cast<uintptr_t>(X) % 16 == 0 && tma_ok(Wt, Kg, 2) &&
                         pad_h <= 127 && pad_w <= 127 && pad_h - (R - 1) * dil_h >= -128 &&
                         pad_w - (S - 1) * dil_w >= -128 && (R - 1) * dil_h <= 255 && (S - 1) * dil_w <= 255 &&
                         stride_h <= 8 && stride_w <= 8 && !g_force_generic_load.load() && forced_bn == 0;
  if (im2col_ok && pair_mode != 2 && (pair_mode == 1 || (M >= kPairBM && K >= 128))) {
    const bool bf16 = dtype == TTC_BF16;
    const PairChoice pc = choose_pair(dev, bf16, M, K, 1, false);
    if (pc.bn != 0) {
      if (!tile_maps({kPairBM, pc.bn, 2, kBM, 0, 0, 2, 1, pc.bn == 256 ? pc.bn / 2 : 0}, prm.maps))
        return TTC_ERR_UNSUPPORTED;
      // filters: the K x Kg matrix of output channels, K-major
      if (!encode_im2col(&prm.tmA, dt, X, N, H, W, C, R, S, pad_h, pad_w, stride_h, stride_w, dil_h, dil_w) ||
          !encode_operand(&prm.tmB, dt, 2, Wt, K, Kg, Kg, prm.maps.b, CU_TENSOR_MAP_SWIZZLE_128B))
        return TTC_ERR_CUDA;
      prm.cv_tma = 1;
      prm.cv_cblk = (int)(C / kBK);
      prm.num_m_blocks = (int)((M + kPairBM - 1) / kPairBM);
      prm.num_n_blocks = (int)((K + pc.bn - 1) / pc.bn);
      prm.tiles_per_batch = prm.num_m_blocks * prm.num_n_blocks;
      prm.num_tiles = prm.tiles_per_batch;
      const int gmp = g_group_m.load() > 0 ? g_group_m.load() : 8;
      prm.group_m = prm.num_m_blocks < gmp ? prm.num_m_blocks : gmp;
      const int nclus = plan_pair_units(prm, pc.bn, pc.clusters);
      if (Kg > 0 && prm.tail_from < prm.num_units) {
        if (!encode_operand(&prm.tmBh, dt, 2, Wt, K, Kg, Kg, prm.maps.b_half, CU_TENSOR_MAP_SWIZZLE_128B))
          return TTC_ERR_CUDA;
        prm.b_half_map = 1;
      }
      if (launch_pair(bf16, pc.bn, prm, nclus, static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return TTC_ERR_CUDA;
      g_launches.fetch_add(1);
      return TTC_OK;
    }
  }

  const int grid = prm.num_tiles < dev->sm_count ? prm.num_tiles : dev->sm_count;
  if (launch(mode, bn, prm, grid, static_cast<cudaStream_t>(stream)) != cudaSuccess) return TTC_ERR_CUDA;
  g_launches.fetch_add(1);
  return TTC_OK;
}

ttc_status ttc_transpose(int64_t rows, int64_t cols, const void* src, int64_t lds, void* dst, int64_t ldd,
                         int elem_bytes, void* stream) {
  if (rows < 0 || cols < 0) return TTC_ERR_INVALID_ARG;
  if (elem_bytes != 1 && elem_bytes != 2 && elem_bytes != 4 && elem_bytes != 8) return TTC_ERR_INVALID_ARG;
  if (rows == 0 || cols == 0) return TTC_OK;
  if (src == nullptr || dst == nullptr || lds < cols || ldd < rows) return TTC_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(src) % elem_bytes || reinterpret_cast<uintptr_t>(dst) % elem_bytes)
    return TTC_ERR_INVALID_ARG;
  if (ranges_overlap(src, ((rows - 1) * lds + cols) * elem_bytes, dst, ((cols - 1) * ldd + rows) * elem_bytes))
    return TTC_ERR_INVALID_ARG;
  DeviceInfo* dev = nullptr;
  ttc_status st = device_info(&dev);
  if (st != TTC_OK) return st;
  if (launch_transpose(src, lds, dst, ldd, rows, cols, elem_bytes, dev->sm_count, static_cast<cudaStream_t>(stream)) !=
      cudaSuccess)
    return TTC_ERR_CUDA;
  g_launches.fetch_add(1);
  return TTC_OK;
}

size_t ttc_gemm_workspace_size(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, ttc_layout layoutA,
                               const void* B, int64_t ldb, ttc_layout layoutB, ttc_dtype dtype) {
  if (M <= 0 || N <= 0 || K <= 0) return 0;
  if ((layoutA != TTC_ROW_MAJOR && layoutA != TTC_COL_MAJOR) || (layoutB != TTC_ROW_MAJOR && layoutB != TTC_COL_MAJOR))
    return 0;
  if (dtype != TTC_F16 && dtype != TTC_BF16 && dtype != TTC_I8) return 0;
  canonicalise(M, N, K, layoutA, lda, layoutB, ldb);
  if (takes_gemv(M, N, K, layoutA, layoutB, dtype, 1)) return 0;
  return plan_repack(M, N, K, A, lda, layoutA, B, ldb, layoutB, dtype == TTC_I8 ? 1 : 2).bytes;
}

size_t ttc_gemm_workspace_size_staged(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda,
                                      ttc_layout layoutA, const void* B, int64_t ldb, ttc_layout layoutB,
                                      const void* D, int64_t ldd, ttc_dtype dtype) {
  if (M <= 0 || N <= 0 || K < 0 || ldd < N) return 0;
  if ((layoutA != TTC_ROW_MAJOR && layoutA != TTC_COL_MAJOR) || (layoutB != TTC_ROW_MAJOR && layoutB != TTC_COL_MAJOR))
    return 0;
  if (dtype != TTC_F16 && dtype != TTC_BF16 && dtype != TTC_I8) return 0;
  // matrix-vector problems take their own kernel and no workspace
  int64_t lda_c = lda, ldb_c = ldb;
  ttc_layout la = layoutA, lb = layoutB;
  canonicalise(M, N, K, la, lda_c, lb, ldb_c);
  if (takes_gemv(M, N, K, la, lb, dtype, 1)) return 0;
  if (dtype == TTC_I8) {
    // int8 problems the CTA-pair kernel takes: fp16 copies of A and B
    const I8Wide w = plan_i8_wide(M, N, K, A, lda_c, la, B, ldb_c, lb, D, ldd);
    if (w.on) return w.bytes;
  }
  const size_t ab = ttc_gemm_workspace_size(M, N, K, A, lda, layoutA, B, ldb, layoutB, dtype);
  return ab + plan_dstage(M, N, D, ldd, dtype == TTC_I8 ? 4 : 2, ab).bytes;
}

}  // extern "C"

// ---------------------------------------------------------------- no-allocation entry point
// Scratch for ttc_gemm_static_scratch: a fixed array in device memory that
// exists on every GPU that loads this library, for as long as the process
// lives.  Host code never dereferences the symbol itself (on the host it only
// names the array); the device address comes from cudaGetSymbolAddress, once
// per device, below.
static __device__ __align__(256) uint8_t g_static_scratch[TTC_STATIC_SCRATCH_BYTES];

namespace {
void* g_static_scratch_ptr[kMaxDevices] = {};
std::mutex g_static_scratch_mu;

// Device address of g_static_scratch on the current device (nullptr on error).
void* static_scratch_address() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lk(g_static_scratch_mu);
  if (g_static_scratch_ptr[dev] == nullptr) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_static_scratch) != cudaSuccess || ptr == nullptr) return nullptr;
    g_static_scratch_ptr[dev] = ptr;
  }
  return g_static_scratch_ptr[dev];
}
}  // namespace

extern "C" ttc_status ttc_gemm_static_scratch(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda,
                                              ttc_layout layoutA, const void* B, int64_t ldb, ttc_layout layoutB,
                                              const void* C, int64_t ldc, void* D, int64_t ldd, float alpha,
                                              float beta, const float* bias, ttc_act act, ttc_dtype dtype,
                                              void* stream) {
  // The scratch this call needs is a pure host computation; refuse before any
  // device work when it exceeds the fixed array.
  if (ttc_gemm_workspace_size(M, N, K, A, lda, layoutA, B, ldb, layoutB, dtype) > (size_t)TTC_STATIC_SCRATCH_BYTES)
    return TTC_ERR_SCRATCH_TOO_SMALL;
  void* scratch = static_scratch_address();
  if (scratch == nullptr) return TTC_ERR_CUDA;
  return gemm_impl(M, N, K, A, lda, layoutA, B, ldb, layoutB, C, ldc, D, ldd, alpha, beta, bias, act, dtype, scratch,
                   (size_t)TTC_STATIC_SCRATCH_BYTES, stream);
}
