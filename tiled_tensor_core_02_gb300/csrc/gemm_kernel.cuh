// Persistent, warp-specialized tiled GEMM for sm_103a:
//   D = act(alpha * A * B + beta * C + bias)
// fp16/bf16 operands with fp32 accumulation, or int8 operands with an exact
// int32 result.
//
// Structure (the tutorial's "Collective Mainloop + Collective Epilogue" split,
// hpc.payai.win/cutlass section 3, rebuilt for tcgen05/TMEM/TMA):
//   producer    fills a STAGES-deep ring of 128-byte-swizzled shared-memory
//               slots with the A and B tiles of each 64-wide k-block
//               (full/empty mbarrier pair per slot).  TMA modes: one thread
//               issues 2-D TMA boxes.  Generic modes (operands TMA cannot
//               describe, and int8): four warps load with plain predicated
//               loads along the strip-mined thread map of the
//               PitchLinearStripminedThreadMap walkthrough (lpnh.cn, sections
//               2-4) and write the same swizzled layout TMA would;
//   MMA issuer  allocates TMEM; one thread issues tcgen05.mma (M=128, N=BN,
//               K=16) into one of two TMEM accumulators and commits completion
//               back to the ring;
//   epilogue    4 warps; each owns the 32 TMEM lanes (= tile rows) its warp
//               index selects: tcgen05.ld, alpha / beta*C / bias / activation
//               in fp32, round, stage in swizzled shared memory, TMA store
//               (or predicated stores when TMA cannot describe D).
// The two accumulators let the epilogue of one unit overlap the mainloop of
// the next.  A unit is a whole tile for fp16/bf16; for int8 it is a chunk of
// at most 1024 k, whose exact fp32 partial sum the epilogue adds into int32
// registers (every partial is an integer below 2^24 in magnitude, so fp32
// holds it exactly).  Tiles are walked persistently in grouped order: group_m
// consecutive M-blocks share each N-block, so concurrent CTAs reuse A and B
// panels from L2.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "ptx.cuh"
#include "tile_maps.h"
#include "ttc_layout.hpp"

namespace ttc {

constexpr int kBM = 128;     // UMMA M (rows of the CTA tile = TMEM lanes)
constexpr int kBK = 64;      // k-block: 64 16-bit elements = one 128-byte swizzle row
constexpr int kUmmaK = 16;   // K of one tcgen05.mma for 16-bit inputs
constexpr int kEpiWarps = 4;
constexpr int kEpiCols = 32;  // columns per epilogue chunk
constexpr int kABytes = kBM * kBK * 2;  // 16 KiB
constexpr int kI8ChunkKBlocks = 16;     // int8: drain the accumulator every 1024 k
constexpr int kConvWarps = 8;           // int8 TMA staging: warps widening int8 tiles to fp16
constexpr int kConvGroups = 2;          // ... in groups that take alternate k-blocks
constexpr int kConvGroupWarps = kConvWarps / kConvGroups;

enum ActKind : int { kActNone = 0, kActRelu = 1, kActGelu = 2 };

// Kernel modes: how operands reach shared memory and what the element types are.
enum Mode : int {
  kModeTmaF16 = 0,   // TMA loads, fp16 in/out
  kModeTmaBF16 = 1,  // TMA loads, bf16 in/out
  kModeGenF16 = 2,   // plain loads, fp16
  kModeGenBF16 = 3,  // plain loads, bf16
  kModeI8 = 4,       // plain loads of int8, converted to fp16; int32 out
  kModeI8Tma = 5,    // TMA loads of int8 into a staging ring, converter warps widen to fp16; int32 out
  kModeConvF16 = 6,  // implicit-GEMM convolution: A gathered from the NHWC input (plain loads), fp16
  kModeConvBF16 = 7, // the same, bf16
  kModeI8TmemA = 8,  // as kModeI8Tma for a K-major A, whose converter warps widen A straight into
                     // tensor memory (the MMA reads A from there) and only B into shared memory
};

template <int MODE>
struct ModeTraits {
  static constexpr bool kTmaLoad = MODE == kModeTmaF16 || MODE == kModeTmaBF16;
  static constexpr bool kBF16 =
      MODE == kModeTmaBF16 || MODE == kModeGenBF16 || MODE == kModeConvBF16;  // tensor-core input type
  static constexpr bool kConv = MODE == kModeConvF16 || MODE == kModeConvBF16;
  static constexpr bool kStaged = MODE == kModeI8Tma || MODE == kModeI8TmemA;  // TMA int8 staging + converters
  static constexpr bool kATmem = MODE == kModeI8TmemA;  // the MMA's A operand lives in tensor memory
  static constexpr bool kI8 = MODE == kModeI8 || kStaged;
  // producer warps: 1 TMA thread; 4 plain-load warps; or 1 TMA warp + kConvWarps converter warps
  static constexpr int kProdWarps = kTmaLoad ? 1 : (kStaged ? 1 + kConvWarps : 4);
  static constexpr int kMmaWarp = kProdWarps;
  static constexpr int kEpiWarp0 = kProdWarps + 1;
  static constexpr int kThreads = 32 * (kProdWarps + 1 + kEpiWarps);
  static constexpr int kOutBytes = kI8 ? 4 : 2;
  static constexpr int kEpiBufBytes = 32 * kEpiCols * kOutBytes;  // 32 rows x (64 or 128) bytes
};

// Host: whether the GEMM, convolution and matrix-vector kernels are launched
// with programmatic dependent launch (on unless TTC_KNOB_PDL turns it off).
bool pdl_enabled();

// Host: appends the programmatic-stream-serialization attribute to `cfg`
// when it is enabled (`attrs` has room for it after cfg.numAttrs entries).
// The kernels so launched wait for the previous grid on the stream before
// their first global access (grid_dependency_wait).
inline void add_pdl_attribute(cudaLaunchConfig_t& cfg, cudaLaunchAttribute* attrs) {
  if (!pdl_enabled()) return;
  cudaLaunchAttribute& a = attrs[cfg.numAttrs];
  a = cudaLaunchAttribute{};
  a.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  a.val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attrs;
  cfg.numAttrs += 1;
}

struct GemmParams {
  CUtensorMap tmA;
  CUtensorMap tmB;
  CUtensorMap tmD;
  const void* A;  // generic modes: operand base pointers and leading dimensions
  const void* B;
  int64_t lda, ldb;
  int a_vec, b_vec;  // generic modes: 1 when 8-element groups may be read as one vector
  uint32_t stage_tx; // TMA modes: bytes the loads of one k-block deliver.  When M < 128
                     // only the rows that exist are loaded; the rest of the A tile keeps
                     // stale data, which only reaches accumulator rows that are never stored
  int M, N, K;
  int num_m_blocks, num_n_blocks, num_k_blocks, num_tiles, group_m;
  // strided batches: tiles [b * tiles_per_batch, (b + 1) * tiles_per_batch) belong
  // to batch b; operand x of batch b starts x_bs elements after batch 0 (plain
  // loads and stores); TMA boxes take batch coordinate b * a_bc (b_bc), 0 for an
  // operand shared by every batch
  int batch, tiles_per_batch, a_bc, b_bc;
  int64_t a_bs, b_bs, c_bs, d_bs;
  int ksplit;     // CTAs per cluster that split one tile's k-blocks (1 = no split)
  int kb_split;   // k-blocks per split (the last split may get fewer, or none)
  int a_mn, b_mn;  // operand stored MN-major (A column-major / B row-major)
  float alpha, beta;
  const void* C;
  int64_t ldc;
  void* D;
  int64_t ldd;
  const float* bias;
  int act;
  int d_tma;    // 1: D written by TMA store; 0: predicated st.global
  int d_trans;  // 1: the kernel computes D^T = B^T A^T: kernel element (i, j) is D[j * ldd + i],
                //    C likewise, and the bias is indexed by the kernel row
  uint32_t* err;
  uint64_t timeout_ns;
  int inject_stall;
  // implicit-GEMM convolution (kModeConv*): A is not a matrix in memory but
  // the im2col view of the NHWC input at A.  Row m is output pixel (n, p, q),
  // m = (n P + p) Q + q; column kk is filter tap (r, s) and channel c,
  // kk = (r S + s) C + c.  a_vec: C is a multiple of 8 and the input is 16-byte
  // aligned, so each 8-column group is one 16-byte load.
  int cv_h, cv_w, cv_c, cv_p, cv_q, cv_s;
  int cv_ph, cv_pw, cv_sh, cv_sw, cv_dh, cv_dw;
  // CTA-pair kernel, convolution by im2col TMA (tmA is an im2col map over the
  // NHWC input, 128 pixels x 64 channels per box): k-block kb is filter tap
  // kb / cv_cblk, channels 64 (kb mod cv_cblk) onwards (C = 64 cv_cblk)
  int cv_tma;
  int cv_cblk;
  // 1: the operand is read by one tile only (one tile column for A, one tile
  // row for B), so its TMA loads carry an evict-first L2 hint; otherwise
  // evict-last keeps it for the other tiles that read it
  int a_stream, b_stream;
  // CTA-pair kernel: work units [0, num_units) walk the tiles; units from
  // tail_from on are half tiles (the left or right half of the columns of tile
  // tail_from + (u - tail_from) / 2), so that a last, partial wave keeps twice
  // as many pairs busy for half as long.  tail_from == num_units: whole tiles.
  int tail_from, num_units;
  // tile origins, per-CTA shares, TMA boxes and the epilogue's thread maps,
  // derived on the host from the operand, output and TMEM layouts
  TileMaps maps;
  // CTA-pair kernel, K-major B: tmBh has boxes of a half unit's width per CTA
  // (BN / 4 columns), so that half units stage only the B columns they use
  // (b_half_map == 1; otherwise they load the whole box and read half of it)
  int b_half_map;
  CUtensorMap tmBh;
};

// Loads the k-block tile of an operand whose rows start at r0 and whose K
// starts at k0 as bm.boxes TMA boxes (see BoxMap; at most kMaxBoxes): box h
// starts h * box_step further along the contiguous mode and h * smem_step
// bytes further in shared memory.  Unrolled, with no loop: the producer
// thread is on the MMA's critical path (a runtime loop here measured 7 %
// slower on 8192^3).
constexpr int kMaxBoxes = 4;  // an MN-major B tile 256 wide: four 64-column slabs
template <int kMax = kMaxBoxes>
__device__ __forceinline__ void tma_load_boxes(uint8_t* dst, const CUtensorMap* m, const BoxMap bm, int r0, int k0,
                                               int z, uint64_t* bar, uint64_t pol) {
  const int x = bm.k_inner ? k0 : r0, y = bm.k_inner ? r0 : k0;
#pragma unroll
  for (int h = 0; h < kMax; ++h)
    if (h == 0 || h < bm.boxes) tma_load_3d(dst + h * bm.smem_step, m, x + h * bm.box_step, y, z, bar, pol);
}

// Tile and column offset of work unit u of the CTA-pair walk (see tail_from).
__device__ __forceinline__ void pair_unit(const GemmParams& p, int u, int half_cols, int& t, int& n_off, bool& half) {
  half = u >= p.tail_from;
  if (!half) {
    t = u;
    n_off = 0;
  } else {
    const int h = u - p.tail_from;
    t = p.tail_from + (h >> 1);
    n_off = (h & 1) * half_cols;
  }
}

template <int BN, int MODE>
struct TileCfg {
  using T = ModeTraits<MODE>;
  static constexpr int kBBytes = BN * kBK * 2;
  static constexpr int kAStageBytes = T::kATmem ? 0 : kABytes;  // fp16 A in shared memory per stage
  static constexpr int kStageBytes = kAStageBytes + kBBytes;
  static constexpr int kEpiBytes = kEpiWarps * 2 * T::kEpiBufBytes;
  static constexpr int kBarBytes = 512;
  static constexpr int kSmemLimit = 227 * 1024;  // opt-in dynamic shared memory per block
  // split-K partial-sum exchange (fp16/bf16 modes, tiles up to 128 wide): per
  // epilogue warp two slots of 32 rows x 32 fp32 columns
  static constexpr bool kSplitK = !T::kI8 && BN <= 128;
  static constexpr int kRedSlotBytes = 32 * kEpiCols * 4;
  static constexpr int kRedBytes = kSplitK ? kEpiWarps * 2 * kRedSlotBytes : 0;
  static constexpr int kStageBudget = kSmemLimit - 1024 - kBarBytes - kEpiBytes - kRedBytes;
  // int8 staging ring (staged mode): the raw int8 A and B tiles of one k-block
  static constexpr int kStage8Bytes = T::kStaged ? (kBM + BN) * kBK : 0;
  static constexpr int kStagesRaw = kStageBudget / (kStageBytes + kStage8Bytes);
  // with A in tensor memory, a stage also takes 32 TMEM columns (64 k of fp16)
  static constexpr int kStageCap = T::kATmem ? 4 : 12;
  static constexpr int kStages = kStagesRaw > kStageCap ? kStageCap : kStagesRaw;
  // int8 staging ring: as deep as the fp16 ring, or, with A in tensor memory
  // (whose fp16 ring holds only B), as deep as the rest of shared memory
  // allows: the raw tiles in flight are what hides the load latency
  static constexpr int kStages8Raw = (kStageBudget - kStages * kStageBytes) / (kStage8Bytes > 0 ? kStage8Bytes : 1);
  static constexpr int kStages8 = !T::kStaged ? 0 : !T::kATmem ? kStages : kStages8Raw > 12 ? 12 : kStages8Raw;
  // two accumulators of BN columns; int8 adds BN columns of exact int32 running
  // sums after them; allocations are powers of two of at least 32 columns
  static constexpr int kATmemCol0 = 3 * BN;  // kATmem: stage s of A in columns [kATmemCol0 + 32 s, + 32)
  static constexpr int kTmemUsed = (T::kI8 ? 3 : 2) * BN + (T::kATmem ? 32 * kStages : 0);
  static constexpr int kTmemCols = kTmemUsed <= 32 ? 32 : kTmemUsed <= 64 ? 64 : kTmemUsed <= 128 ? 128
                                   : kTmemUsed <= 256 ? 256 : 512;
  static_assert(kTmemUsed <= 512, "TMEM columns");
  static constexpr int kSmemBytes =
      1024 /*align slack*/ + kStages * kStageBytes + kStages8 * kStage8Bytes + kEpiBytes + kRedBytes + kBarBytes;
  static_assert(BN % 32 == 0 && BN >= 32 && BN <= 256, "UMMA N for M=128, whole epilogue chunks");
  static_assert(kStages >= 2, "pipeline depth");
  static_assert(kSmemBytes <= kSmemLimit, "shared memory budget");
  static_assert((2 * BN & (2 * BN - 1)) == 0, "TMEM allocation is a power of two");
};

__device__ __forceinline__ void tile_coords(int t, const GemmParams& p, int& bz, int& mb, int& nb) {
  bz = t / p.tiles_per_batch;
  t -= bz * p.tiles_per_batch;
  const int per_group = p.group_m * p.num_n_blocks;
  const int g = t / per_group;
  const int first_m = g * p.group_m;
  const int gsize = min(p.num_m_blocks - first_m, p.group_m);
  const int r = t - g * per_group;
  mb = first_m + r % gsize;
  nb = r / gsize;
}

__device__ __forceinline__ float apply_act(int act, float x) {
  if (act == kActRelu) return fmaxf(x, 0.0f);
  if (act == kActGelu) {
    const float k0 = 0.7978845608028654f;  // sqrt(2/pi)
    const float inner = k0 * fmaf(0.044715f * x, x * x, x);
    return 0.5f * x * (1.0f + tanh_approx(inner));
  }
  return x;
}

template <bool BF16>
__device__ __forceinline__ float half_bits_to_float(uint16_t h) {
  if constexpr (BF16) {
    return __bfloat162float(__ushort_as_bfloat16(h));
  } else {
    return __half2float(__ushort_as_half(h));
  }
}

template <bool BF16>
__device__ __forceinline__ uint32_t pack2(float a, float b) {
  if constexpr (BF16) {
    __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&v);
  } else {
    __half2 v = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&v);
  }
}

// Waits for a barrier phase during shutdown, ignoring errors raised by other
// threads: used only to let copies this thread started land before exit.
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity, uint64_t budget_ns) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > budget_ns) return;
  }
}

// ------------------------------------------------------------------ generic operand loads
// One operand tile in memory order: ROWS rows ("outer": M/N rows of a K-major
// operand, k rows of an MN-major one) of COLS contiguous elements.  The 128
// producer threads walk it with the strip-mined map (8 contiguous elements per
// access), load with predicates (zero outside the extents) and store each
// 8-element group as one 16-byte chunk of the 128-byte-swizzled layout the
// tensor core reads: element (r, c) sits at
//   Swizzle<3,4,3>((c / 64) * ROWS * 128 + r * 128 + (c % 64) * 2),
// i.e. 64-column slabs of ROWS 128-byte rows, the layout TMA writes for the
// same tile.
template <int ROWS, int COLS, bool kI8>
__device__ __forceinline__ void generic_load_tile(uint8_t* sdst, const void* gsrc, int64_t ld, int outer0,
                                                  int inner0, int outer_ext, int inner_ext, bool vec_ok, int tid) {
  constexpr layout::StripMined map{ROWS, COLS, 128, 8};
  static_assert(map.valid(), "strip-mined map must tile the operand tile");
  constexpr int kIters = map.iterations();
  constexpr layout::SwizzleBytes128 swz{};
  const int c = map.col(tid);
  const int gi = inner0 + c;
  const bool inner_full = gi + 7 < inner_ext;
  constexpr int kBatch = kIters < 4 ? kIters : 4;
#pragma unroll
  for (int i0 = 0; i0 < kIters; i0 += kBatch) {
    uint4 w[kBatch];
#pragma unroll
    for (int b = 0; b < kBatch; ++b) {
      const int r = map.row(tid, i0 + b);
      const int go = outer0 + r;
      const bool row_ok = go < outer_ext;
      if constexpr (kI8) {
        const int8_t* src = reinterpret_cast<const int8_t*>(gsrc) + (int64_t)go * ld + gi;
        int8_t e[8];
        if (row_ok && inner_full && vec_ok) {
          const uint2 u = __ldg(reinterpret_cast<const uint2*>(src));
          *reinterpret_cast<uint2*>(e) = u;
        } else {
#pragma unroll
          for (int j = 0; j < 8; ++j) e[j] = (row_ok && gi + j < inner_ext) ? __ldg(src + j) : (int8_t)0;
        }
        uint32_t h[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          // int8 values are exact in fp16
          __half2 v = __halves2half2(__int2half_rn(e[2 * j]), __int2half_rn(e[2 * j + 1]));
          h[j] = *reinterpret_cast<uint32_t*>(&v);
        }
        w[b] = make_uint4(h[0], h[1], h[2], h[3]);
      } else {
        const uint16_t* src = reinterpret_cast<const uint16_t*>(gsrc) + (int64_t)go * ld + gi;
        if (row_ok && inner_full && vec_ok) {
          w[b] = __ldg(reinterpret_cast<const uint4*>(src));
        } else {
          uint16_t e[8];
#pragma unroll
          for (int j = 0; j < 8; ++j) e[j] = (row_ok && gi + j < inner_ext) ? __ldg(src + j) : (uint16_t)0;
          w[b] = make_uint4(e[0] | ((uint32_t)e[1] << 16), e[2] | ((uint32_t)e[3] << 16),
                            e[4] | ((uint32_t)e[5] << 16), e[6] | ((uint32_t)e[7] << 16));
        }
      }
    }
#pragma unroll
    for (int b = 0; b < kBatch; ++b) {
      const int r = map.row(tid, i0 + b);
      const uint32_t off = swz((uint32_t)((c / 64) * ROWS * 128 + r * 128 + (c % 64) * 2));
      *reinterpret_cast<uint4*>(sdst + off) = w[b];
    }
  }
}

// ------------------------------------------------------------------ implicit-GEMM convolution
// One im2col row as the producer threads need it across a tile's k-blocks.
struct ConvRow {
  int pix;  // n H W: index of the first pixel of the row's image
  int h0;   // p sh - ph; a large negative value for rows past M (always outside)
  int w0;   // q sw - pw
};

__device__ __forceinline__ ConvRow conv_row(const GemmParams& p, int m) {
  ConvRow cr;
  if (m >= p.M) {
    cr.pix = 0;
    cr.h0 = -(1 << 29);
    cr.w0 = 0;
    return cr;
  }
  const int pq = p.cv_p * p.cv_q;
  const int n = m / pq;
  const int rem = m - n * pq;
  const int pp = rem / p.cv_q;
  const int qq = rem - pp * p.cv_q;
  cr.pix = n * p.cv_h * p.cv_w;
  cr.h0 = pp * p.cv_sh - p.cv_ph;
  cr.w0 = qq * p.cv_sw - p.cv_pw;
  return cr;
}

// The A tile of k-block k0 (kBM rows x kBK columns of the im2col matrix),
// written with the placement generic_load_tile<kBM, kBK> uses.  Element
// (m, kk) is x[n, h0 + r dh, w0 + s dw, c], zero where the tap is outside the
// input or kk >= K.  rows[i] describes map row i of this thread.
template <int ITERS>
__device__ __forceinline__ void im2col_load_tile(uint8_t* sdst, const GemmParams& p, const ConvRow (&rows)[ITERS],
                                                 int k0, int tid) {
  constexpr layout::StripMined map{kBM, kBK, 128, 8};
  static_assert(map.iterations() == ITERS, "one ConvRow per map row");
  constexpr layout::SwizzleBytes128 swz{};
  const uint16_t* X = static_cast<const uint16_t*>(p.A);
  const int col = map.col(tid);
  const int kk = k0 + col;
  const unsigned H = (unsigned)p.cv_h, W = (unsigned)p.cv_w;
  const int C = p.cv_c;
  if (p.a_vec) {
    // the group's 8 columns are channels c .. c + 7 of one tap
    const bool k_ok = kk < p.K;
    const int rs = kk / C;
    const int c = kk - rs * C;
    const int rr = rs / p.cv_s;
    const int ss = rs - rr * p.cv_s;
    const int dh = rr * p.cv_dh, dw = ss * p.cv_dw;
#pragma unroll
    for (int i = 0; i < ITERS; ++i) {
      const int h = rows[i].h0 + dh, w = rows[i].w0 + dw;
      uint4 v = make_uint4(0, 0, 0, 0);
      if (k_ok && (unsigned)h < H && (unsigned)w < W)
        v = __ldg(reinterpret_cast<const uint4*>(X + ((int64_t)rows[i].pix + (int64_t)h * p.cv_w + w) * C + c));
      const int r = map.row(tid, i);
      *reinterpret_cast<uint4*>(sdst + swz((uint32_t)(r * 128 + col * 2))) = v;
    }
  } else {
    // every column decomposed on its own (C not a multiple of 8, or unaligned input)
    int dh[8], dw[8], cc[8];
    bool ok[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int k = kk + j;
      ok[j] = k < p.K;
      const int rs = k / C;
      cc[j] = k - rs * C;
      const int rr = rs / p.cv_s;
      dh[j] = rr * p.cv_dh;
      dw[j] = (rs - rr * p.cv_s) * p.cv_dw;
    }
#pragma unroll
    for (int i = 0; i < ITERS; ++i) {
      uint16_t e[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int h = rows[i].h0 + dh[j], w = rows[i].w0 + dw[j];
        e[j] = (ok[j] && (unsigned)h < H && (unsigned)w < W)
                   ? __ldg(X + ((int64_t)rows[i].pix + (int64_t)h * p.cv_w + w) * C + cc[j])
                   : (uint16_t)0;
      }
      const int r = map.row(tid, i);
      *reinterpret_cast<uint4*>(sdst + swz((uint32_t)(r * 128 + col * 2))) =
          make_uint4(e[0] | ((uint32_t)e[1] << 16), e[2] | ((uint32_t)e[3] << 16), e[4] | ((uint32_t)e[5] << 16),
                     e[6] | ((uint32_t)e[7] << 16));
    }
  }
}

// ------------------------------------------------------------------ int8 -> fp16 conversion
// Widens one raw int8 tile (ROWS rows of COLS bytes, as TMA wrote it, no
// swizzle) into the fp16 128-byte-swizzled layout the tensor core reads (the
// same placement as generic_load_tile).  Exact: with u = x + 128 (a byte),
// the fp16 bit pattern 0x6400 | u is 1024 + u, and subtracting 1152 leaves x.
// Raw chunks a thread widens: chunk tid + NT i of the tile, i < kIters.
template <int ROWS, int COLS, int NT>
struct I8Tile {
  static constexpr int kPerRow = COLS / 16;
  static constexpr int kChunks = ROWS * kPerRow;
  static constexpr int kIters = (kChunks + NT - 1) / NT;
};

// convert_i8_tile in two steps, so a caller can put other work between the
// loads and the stores: the compiler may not move a shared-memory load above
// a store to the same space, so loads interleaved with stores would each wait
// out their own latency.
template <int ROWS, int COLS, int NT>
__device__ __forceinline__ void i8_tile_load(const uint8_t* s8, uint4 (&w)[I8Tile<ROWS, COLS, NT>::kIters], int tid) {
  using T = I8Tile<ROWS, COLS, NT>;
#pragma unroll
  for (int i = 0; i < T::kIters; ++i) {
    const int q = tid + NT * i;
    if (T::kChunks % NT == 0 || q < T::kChunks)
      w[i] = *reinterpret_cast<const uint4*>(s8 + (q / T::kPerRow) * COLS + (q % T::kPerRow) * 16);
  }
}

template <int ROWS, int COLS, int NT>
__device__ __forceinline__ void i8_tile_widen_store(uint8_t* s16, const uint4 (&w)[I8Tile<ROWS, COLS, NT>::kIters],
                                                    int tid) {
  using T = I8Tile<ROWS, COLS, NT>;
  constexpr layout::SwizzleBytes128 swz{};
  const __half2 bias2 = __halves2half2(__ushort_as_half(0x6480u), __ushort_as_half(0x6480u));  // 1152
#pragma unroll
  for (int i = 0; i < T::kIters; ++i) {
    const int q = tid + NT * i;
    if (T::kChunks % NT != 0 && q >= T::kChunks) break;
    const int r = q / T::kPerRow;
    const int c = (q % T::kPerRow) * 16;
    const uint32_t ws[4] = {w[i].x, w[i].y, w[i].z, w[i].w};
    uint32_t h[8];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint32_t u = ws[j] ^ 0x80808080u;
      uint32_t lo = __byte_perm(u, 0x64646464u, 0x4140);
      uint32_t hi = __byte_perm(u, 0x64646464u, 0x4342);
      __half2 l2 = __hsub2(*reinterpret_cast<__half2*>(&lo), bias2);
      __half2 h2 = __hsub2(*reinterpret_cast<__half2*>(&hi), bias2);
      h[2 * j] = *reinterpret_cast<uint32_t*>(&l2);
      h[2 * j + 1] = *reinterpret_cast<uint32_t*>(&h2);
    }
    const uint32_t base = (uint32_t)((c / 64) * ROWS * 128 + r * 128 + (c % 64) * 2);
    *reinterpret_cast<uint4*>(s16 + swz(base)) = make_uint4(h[0], h[1], h[2], h[3]);
    *reinterpret_cast<uint4*>(s16 + swz(base + 16)) = make_uint4(h[4], h[5], h[6], h[7]);
  }
}

template <int ROWS, int COLS, int NT>
__device__ __forceinline__ void convert_i8_tile(const uint8_t* s8, uint8_t* s16, int tid) {
  uint4 w[I8Tile<ROWS, COLS, NT>::kIters];
  i8_tile_load<ROWS, COLS, NT>(s8, w, tid);
  i8_tile_widen_store<ROWS, COLS, NT>(s16, w, tid);
}

// Widens row `r` of a raw K-major int8 tile (rows of 64 bytes, written by TMA
// with the 64-byte swizzle: 16-byte chunk c of a row stored at chunk
// c ^ (address bits 7-8)) into 32 words of exact fp16 pairs in k order, the
// layout of one tensor-memory lane of an A operand.  Row r's four chunks sit
// in different banks from those of rows r + 1 .. r + 7, so a warp reading 32
// rows has no bank conflicts.  The tile must start on a 512-byte boundary.
__device__ __forceinline__ void convert_i8_row_sw64(const uint8_t* s8, int r, uint32_t (&w)[32]) {
  constexpr layout::SwizzleBytes64 swz{};
  const __half2 bias2 = __halves2half2(__ushort_as_half(0x6480u), __ushort_as_half(0x6480u));  // 1152
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const uint4 v = *reinterpret_cast<const uint4*>(s8 + swz((uint32_t)(r * 64 + c * 16)));
    const uint32_t ws[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint32_t u = ws[j] ^ 0x80808080u;
      uint32_t lo = __byte_perm(u, 0x64646464u, 0x4140);
      uint32_t hi = __byte_perm(u, 0x64646464u, 0x4342);
      __half2 l2 = __hsub2(*reinterpret_cast<__half2*>(&lo), bias2);
      __half2 h2 = __hsub2(*reinterpret_cast<__half2*>(&hi), bias2);
      w[8 * c + 2 * j] = *reinterpret_cast<uint32_t*>(&l2);
      w[8 * c + 2 * j + 1] = *reinterpret_cast<uint32_t*>(&h2);
    }
  }
}

// ------------------------------------------------------------------ epilogue helpers
// How one 32-column chunk of fp16/bf16 C is read (the same for the whole warp).
enum CPath : int {
  kCNone = 0,   // beta == 0: C is not read
  kCVec = 1,    // each thread loads its own row's 64 bytes as four 16-byte vectors
  kCRow = 2,    // C's rows are not 16-byte aligned: each thread loads the five aligned
                // 16-byte blocks that cover its row's 64 bytes and shifts them into place
  kCTrans = 3,  // D^T orientation: lanes already hold consecutive elements of a C row
};

// ------------------------------------------------------------------ rows at any 2-byte boundary
// A 32-element segment of a 16-bit row (64 bytes) that starts at an address
// a with phase = a mod 16 lies in the 80-byte window of five aligned 16-byte
// blocks from a - phase.  The window is held as 20 words; the shifts move its
// bytes by `phase` (even, 0..14) in three conditional stages of 8, 4 and 2
// bytes, so no register is indexed at run time.  Only an aligned block that
// holds at least one byte of the segment is ever loaded or stored: such a
// block lies in the same memory page as that byte.

// Moves the window's bytes up by `phase`: byte i goes to i + phase.
__device__ __forceinline__ void window_shift_up(uint32_t (&x)[20], uint32_t phase) {
  const bool s8 = phase & 8, s4 = phase & 4, s2 = phase & 2;
#pragma unroll
  for (int k = 19; k >= 2; --k) x[k] = s8 ? x[k - 2] : x[k];
  x[1] = s8 ? 0u : x[1];
  x[0] = s8 ? 0u : x[0];
#pragma unroll
  for (int k = 19; k >= 1; --k) x[k] = s4 ? x[k - 1] : x[k];
  x[0] = s4 ? 0u : x[0];
#pragma unroll
  for (int k = 19; k >= 1; --k) x[k] = s2 ? __byte_perm(x[k - 1], x[k], 0x5432) : x[k];
  x[0] = s2 ? x[0] << 16 : x[0];
}

// Moves the window's bytes down by `phase`: byte i + phase goes to i.
__device__ __forceinline__ void window_shift_down(uint32_t (&x)[20], uint32_t phase) {
  const bool s8 = phase & 8, s4 = phase & 4, s2 = phase & 2;
#pragma unroll
  for (int k = 0; k < 18; ++k) x[k] = s8 ? x[k + 2] : x[k];
#pragma unroll
  for (int k = 0; k < 19; ++k) x[k] = s4 ? x[k + 1] : x[k];
#pragma unroll
  for (int k = 0; k < 19; ++k) x[k] = s2 ? __byte_perm(x[k], x[k + 1], 0x5432) : x[k];
}

// Writes bytes [s, e) (even offsets, 0 <= s < e <= 16) of the aligned 16-byte
// block v to `blk` with aligned 8-, 4- and 2-byte stores.
__device__ __forceinline__ void store_block_part(uint8_t* blk, const uint4 v, int s, int e) {
  int b = s;
#pragma unroll 1
  while (b < e) {
    const int wi = b >> 2;
    const uint32_t word = wi == 0 ? v.x : wi == 1 ? v.y : wi == 2 ? v.z : v.w;
    if ((b & 7) == 0 && b + 8 <= e) {
      *reinterpret_cast<uint2*>(blk + b) = make_uint2(word, wi == 0 ? v.y : v.w);
      b += 8;
    } else if ((b & 3) == 0 && b + 4 <= e) {
      *reinterpret_cast<uint32_t*>(blk + b) = word;
      b += 4;
    } else {
      *reinterpret_cast<uint16_t*>(blk + b) = (uint16_t)(word >> ((b & 2) * 8));
      b += 2;
    }
  }
}

// Stores bytes [s, e) of the aligned block v at blk: one 16-byte vector when
// whole, pieces otherwise, nothing when empty.
__device__ __forceinline__ void store_block(uint8_t* blk, const uint4 v, int s, int e) {
  if (s == 0 && e >= 16)
    *reinterpret_cast<uint4*>(blk) = v;
  else if (s < e)
    store_block_part(blk, v, s, min(e, 16));
}

// The aligned block a thread's row segment shares with the next 32-column
// chunk of the same row: consecutive chunks of a row have the same phase, so
// the last block of one chunk's window is the first block of the next one's,
// each holding the bytes the other lacks (zeros elsewhere).  Carried over, it
// is stored once, whole, with the next chunk.
struct RowCarry {
  uint4 v;
  int on;
};

// The C and D of the batch a tile belongs to, and its batch index (the TMA
// store's third coordinate).
struct EpiPtrs {
  const void* C;
  void* D;
  int bz;
};

__device__ __forceinline__ EpiPtrs epi_ptrs(const GemmParams& p, int bz, int out_bytes) {
  EpiPtrs e;
  e.C = p.C ? static_cast<const void*>(static_cast<const char*>(p.C) + (int64_t)bz * p.c_bs * out_bytes) : nullptr;
  e.D = static_cast<char*>(p.D) + (int64_t)bz * p.d_bs * out_bytes;
  e.bz = bz;
  return e;
}

__device__ __forceinline__ int c_path(const GemmParams& p, const EpiPtrs& e, int gcol0) {
  if (p.beta == 0.0f) return kCNone;
  if (p.d_trans) return kCTrans;
  const bool vec =
      ((p.ldc & 7) == 0) && ((reinterpret_cast<uintptr_t>(e.C) & 15) == 0) && (gcol0 + 32 <= p.N);
  return vec ? kCVec : kCRow;
}

// Pulls row `grow` of a tile's C, columns [n0, n0 + ncols), toward L2 ahead of
// the tile's epilogue (16-bit C in the row-major orientation).  The range is
// trimmed inward to 16-byte boundaries, so it never leaves the row.
__device__ __forceinline__ void c_prefetch_row(const GemmParams& p, const EpiPtrs& e, int grow, int n0, int ncols) {
  if (p.beta == 0.0f || p.d_trans || grow >= p.M) return;
  const int n1 = min(n0 + ncols, p.N);
  if (n1 <= n0) return;
  const uint16_t* row = static_cast<const uint16_t*>(e.C) + (int64_t)grow * p.ldc;
  const uintptr_t a0 = (reinterpret_cast<uintptr_t>(row + n0) + 15) & ~uintptr_t(15);
  const uintptr_t a1 = reinterpret_cast<uintptr_t>(row + n1) & ~uintptr_t(15);
  if (a1 > a0) prefetch_l2_bulk(reinterpret_cast<const void*>(a0), (uint32_t)(a1 - a0));
}

// D^T orientation: pulls the tile's C toward L2 ahead of its epilogue.  Kernel
// row i, column j is C[j * ldc + i]: the tile's columns n0 .. n0 + ncols - 1
// are C rows, each holding the 128 contiguous elements of rows m0 .. m0 + 127;
// epilogue thread t takes C row n0 + t.
__device__ __forceinline__ void c_prefetch_trans(const GemmParams& p, const EpiPtrs& e, int m0, int n0, int ncols,
                                                 int t) {
  if (p.beta == 0.0f || !p.d_trans || t >= ncols || n0 + t >= p.N || m0 >= p.M) return;
  const uint16_t* row = static_cast<const uint16_t*>(e.C) + (int64_t)(n0 + t) * p.ldc;
  const int i1 = min(m0 + kBM, p.M);
  const uintptr_t a0 = (reinterpret_cast<uintptr_t>(row + m0) + 15) & ~uintptr_t(15);
  const uintptr_t a1 = reinterpret_cast<uintptr_t>(row + i1) & ~uintptr_t(15);
  if (a1 > a0) prefetch_l2_bulk(reinterpret_cast<const void*>(a0), (uint32_t)(a1 - a0));
}

// C values of one chunk, fetched one chunk ahead of their use so that the
// load latency overlaps the previous chunk's work.
struct CChunk16 {
  uint4 v[5];      // kCVec: this thread's row, 32 values in v[0..3]; kCRow: the five aligned
                   // blocks that cover them
  uint32_t phase;  // kCRow: the row segment's address mod 16
};

__device__ __forceinline__ void c_fetch16(const GemmParams& p, const EpiPtrs& e, int path, int grow, int gcol0,
                                          int lane, CChunk16& cc) {
  if (path == kCVec) {
    if (grow < p.M) {
      const uint4* src = reinterpret_cast<const uint4*>(reinterpret_cast<const uint16_t*>(e.C) +
                                                        (int64_t)grow * p.ldc + gcol0);
#pragma unroll
      for (int u = 0; u < 4; ++u) cc.v[u] = __ldg(src + u);
    } else {
#pragma unroll
      for (int u = 0; u < 4; ++u) cc.v[u] = make_uint4(0u, 0u, 0u, 0u);
    }
  } else if (path == kCRow) {
    cc.phase = 0;
#pragma unroll
    for (int u = 0; u < 5; ++u) cc.v[u] = make_uint4(0u, 0u, 0u, 0u);
    if (grow < p.M && gcol0 < p.N) {
      const uint8_t* a = reinterpret_cast<const uint8_t*>(e.C) + ((int64_t)grow * p.ldc + gcol0) * 2;
      const uint32_t ph = (uint32_t)(reinterpret_cast<uintptr_t>(a) & 15u);
      const int hi = (int)ph + 2 * min(32, p.N - gcol0);  // the segment's bytes in the window
      const uint4* base = reinterpret_cast<const uint4*>(a - ph);
      cc.phase = ph;
#pragma unroll
      for (int u = 0; u < 5; ++u)
        if (16 * u < hi) cc.v[u] = __ldg(base + u);
    }
  }
}

// fp16/bf16 epilogue of one 32-column chunk of the calling thread's row:
// v = alpha * acc (+ beta * C) (+ bias), activation, round to nearest even.
// `cc` holds this chunk's C as fetched by c_fetch16 for `cpath`.
template <bool kBF16>
__device__ __forceinline__ void epi_f16_values(const GemmParams& p, const uint32_t (&r)[32], bool row_ok,
                                               int grow, int gcol0, uint32_t (&packed)[16], int cpath,
                                               const CChunk16& cc, const EpiPtrs& e) {
  float v[32];
#pragma unroll
  for (int j = 0; j < 32; ++j) v[j] = p.alpha * __uint_as_float(r[j]);
  if (cpath == kCTrans) {
    if (row_ok) {
      const uint16_t* ccol = reinterpret_cast<const uint16_t*>(e.C) + grow;
#pragma unroll
      for (int j = 0; j < 32; ++j)
        if (gcol0 + j < p.N)
          v[j] = fmaf(p.beta, half_bits_to_float<kBF16>(__ldg(ccol + (int64_t)(gcol0 + j) * p.ldc)), v[j]);
    }
  } else if (cpath == kCVec) {
    if (row_ok) {
#pragma unroll
      for (int u4 = 0; u4 < 4; ++u4) {
        const uint32_t ws[4] = {cc.v[u4].x, cc.v[u4].y, cc.v[u4].z, cc.v[u4].w};
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          v[u4 * 8 + 2 * h] =
              fmaf(p.beta, half_bits_to_float<kBF16>((uint16_t)(ws[h] & 0xFFFFu)), v[u4 * 8 + 2 * h]);
          v[u4 * 8 + 2 * h + 1] =
              fmaf(p.beta, half_bits_to_float<kBF16>((uint16_t)(ws[h] >> 16)), v[u4 * 8 + 2 * h + 1]);
        }
      }
    }
  } else if (cpath == kCRow) {
    if (row_ok) {
      uint32_t x[20];
#pragma unroll
      for (int u = 0; u < 5; ++u) {
        x[4 * u] = cc.v[u].x;
        x[4 * u + 1] = cc.v[u].y;
        x[4 * u + 2] = cc.v[u].z;
        x[4 * u + 3] = cc.v[u].w;
      }
      window_shift_down(x, cc.phase);
#pragma unroll
      for (int h = 0; h < 16; ++h) {
        v[2 * h] = fmaf(p.beta, half_bits_to_float<kBF16>((uint16_t)(x[h] & 0xFFFFu)), v[2 * h]);
        v[2 * h + 1] = fmaf(p.beta, half_bits_to_float<kBF16>((uint16_t)(x[h] >> 16)), v[2 * h + 1]);
      }
    }
  }
  if (p.bias != nullptr) {
    if (p.d_trans) {
      if (row_ok) {
        const float b = __ldg(p.bias + grow);
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] += b;
      }
    } else {
#pragma unroll
      for (int j = 0; j < 32; ++j)
        if (gcol0 + j < p.N) v[j] += __ldg(p.bias + gcol0 + j);
    }
  }
  if (p.act != kActNone) {
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] = apply_act(p.act, v[j]);
  }
#pragma unroll
  for (int j = 0; j < 16; ++j) packed[j] = pack2<kBF16>(v[2 * j], v[2 * j + 1]);
}

// Writes one 32-column chunk of the calling thread's row: through a swizzled
// shared-memory staging buffer and a TMA store of the warp's 32 x 32 block
// (rows tile_row .. tile_row + 31), or with predicated stores when TMA cannot
// describe D.  `buf` alternates between the warp's two staging buffers.
// `carry` and `last` serve the unaligned 16-bit path: the block shared with
// the calling thread's next chunk (see RowCarry) and whether this is the last
// chunk the thread stores of this row.
template <int kOutBytes, int kPacked>
__device__ __forceinline__ void epi_store_chunk(const GemmParams& p, const uint32_t (&packed)[kPacked], bool row_ok,
                                                int grow, int gcol0, int tile_row, uint8_t* stage_buf,
                                                int buf_bytes, int& buf, RowCarry& carry, bool last, int lane,
                                                const EpiPtrs& e) {
  if (p.d_tma) {
    // staging buffer `buf` was last used two chunks ago; its store must
    // have finished reading shared memory
    if (lane == 0) bulk_wait_read<1>();
    __syncwarp();
    uint8_t* sb = stage_buf + buf * buf_bytes;
    if constexpr (kOutBytes == 2) {
      // 64-byte rows, 64-byte swizzle
      constexpr layout::SwizzleBytes64 swz{};
#pragma unroll
      for (int ch = 0; ch < 4; ++ch)
        *reinterpret_cast<uint4*>(sb + swz((uint32_t)(lane * 64 + ch * 16))) =
            make_uint4(packed[4 * ch], packed[4 * ch + 1], packed[4 * ch + 2], packed[4 * ch + 3]);
    } else {
      // 128-byte rows, 128-byte swizzle
      constexpr layout::SwizzleBytes128 swz{};
#pragma unroll
      for (int ch = 0; ch < 8; ++ch)
        *reinterpret_cast<uint4*>(sb + swz((uint32_t)(lane * 128 + ch * 16))) =
            make_uint4(packed[4 * ch], packed[4 * ch + 1], packed[4 * ch + 2], packed[4 * ch + 3]);
    }
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      tma_store_3d(&p.tmD, gcol0, tile_row, e.bz, sb);
      bulk_commit();
    }
    buf ^= 1;
    // The tensor map ends at the row's last whole 16-byte granule (a TMA
    // store clips only to granules); the columns after it, fewer than one
    // granule, are stored here from the thread's own row.
    constexpr int kGran = 16 / kOutBytes;  // elements per granule
    const int n_full = p.N & ~(kGran - 1);
    if (row_ok && n_full < p.N && gcol0 <= n_full && n_full < gcol0 + 32) {
      const int g = (n_full - gcol0) / kGran;  // the chunk's granule holding the tail
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
      for (int q = 0; q < kPacked / 4; ++q)
        if (q == g) v = make_uint4(packed[4 * q], packed[4 * q + 1], packed[4 * q + 2], packed[4 * q + 3]);
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
      uint8_t* dst = static_cast<uint8_t*>(e.D) + ((int64_t)grow * p.ldd + n_full) * kOutBytes;
      const int cnt = p.N - n_full;
#pragma unroll
      for (int t = 0; t < kGran - 1; ++t) {
        if (t < cnt) {
          if constexpr (kOutBytes == 4)
            reinterpret_cast<uint32_t*>(dst)[t] = w[t];
          else
            reinterpret_cast<uint16_t*>(dst)[t] = (uint16_t)((w[t >> 1] >> ((t & 1) * 16)) & 0xFFFFu);
        }
      }
    }
  } else if (kOutBytes == 2 && !p.d_trans) {
    // 16-bit rows TMA cannot describe: each thread stores its own row's
    // 64 bytes as the aligned blocks that cover them; the block it shares with
    // its next chunk is carried over and stored whole with that chunk
    if (row_ok && gcol0 < p.N) {
      uint8_t* a = reinterpret_cast<uint8_t*>(e.D) + ((int64_t)grow * p.ldd + gcol0) * 2;
      const uint32_t ph = (uint32_t)(reinterpret_cast<uintptr_t>(a) & 15u);
      uint8_t* base = a - ph;
      uint32_t x[20];
#pragma unroll
      for (int j = 0; j < 16; ++j) x[j] = packed[j];
#pragma unroll
      for (int j = 16; j < 20; ++j) x[j] = 0u;
      window_shift_up(x, ph);
      const int ncols = min(32, p.N - gcol0);
      const int hi = (int)ph + 2 * ncols;  // the chunk's bytes in the window: [ph, hi)
      uint4 b0 = make_uint4(x[0], x[1], x[2], x[3]);
      if (carry.on) b0 = make_uint4(b0.x | carry.v.x, b0.y | carry.v.y, b0.z | carry.v.z, b0.w | carry.v.w);
      store_block(base, b0, carry.on ? 0 : (int)ph, hi);
#pragma unroll
      for (int blk = 1; blk < 4; ++blk)
        store_block(base + 16 * blk, make_uint4(x[4 * blk], x[4 * blk + 1], x[4 * blk + 2], x[4 * blk + 3]), 0,
                    hi - 16 * blk);
      const uint4 b4 = make_uint4(x[16], x[17], x[18], x[19]);
      carry.on = 0;
      if (hi > 64) {
        // carried only when this thread's next chunk has columns to store,
        // so it is merged there
        if (ncols == 32 && !last && gcol0 + 32 < p.N) {
          carry.v = b4;
          carry.on = 1;
        } else {
          store_block(base + 64, b4, 0, hi - 64);
        }
      }
    } else {
      carry.on = 0;
    }
  } else if (!p.d_trans) {
    // plain stores, coalesced through the warp's staging area (both buffers):
    // each thread writes its row, then lane l stores column gcol0 + l of the
    // warp's 32 rows
    uint32_t* w = reinterpret_cast<uint32_t*>(stage_buf);
    constexpr int kPitch = kOutBytes == 4 ? 33 : 17;  // words per staged row
#pragma unroll
    for (int j = 0; j < kPacked; ++j) w[lane * kPitch + j] = packed[j];
    __syncwarp();
    const int row0 = grow - lane;
    const int col = gcol0 + lane;
    if (col < p.N) {
#pragma unroll 8
      for (int rr = 0; rr < 32; ++rr) {
        const int gr = row0 + rr;
        if (gr < p.M) {
          if constexpr (kOutBytes == 4)
            reinterpret_cast<int32_t*>(e.D)[(int64_t)gr * p.ldd + col] = (int32_t)w[rr * 33 + lane];
          else
            reinterpret_cast<uint16_t*>(e.D)[(int64_t)gr * p.ldd + col] =
                reinterpret_cast<const uint16_t*>(w)[rr * 34 + lane];
        }
      }
    }
    __syncwarp();
  } else if (row_ok) {
    // lanes hold consecutive kernel rows = consecutive elements of a D row
    if constexpr (kOutBytes == 4) {
      int32_t* dst = reinterpret_cast<int32_t*>(e.D) + grow;
#pragma unroll
      for (int j = 0; j < 32; ++j)
        if (gcol0 + j < p.N) dst[(int64_t)(gcol0 + j) * p.ldd] = (int32_t)packed[j];
    } else {
      uint16_t* dst = reinterpret_cast<uint16_t*>(e.D) + grow;
#pragma unroll
      for (int j = 0; j < 32; ++j)
        if (gcol0 + j < p.N)
          dst[(int64_t)(gcol0 + j) * p.ldd] = (uint16_t)((packed[j >> 1] >> ((j & 1) * 16)) & 0xFFFFu);
    }
  }
}

template <int BN, int MODE>
__global__ void __launch_bounds__(ModeTraits<MODE>::kThreads, 1) gemm_kernel(const __grid_constant__ GemmParams p) {
  using Cfg = TileCfg<BN, MODE>;
  using Tr = ModeTraits<MODE>;
  constexpr int S = Cfg::kStages;
  constexpr bool kBF16 = Tr::kBF16;
  constexpr bool kI8 = Tr::kI8;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = sA + S * Cfg::kAStageBytes;
  uint8_t* s8 = sB + S * Cfg::kBBytes;  // int8 staging ring (staged mode only)
  constexpr int S8 = Cfg::kStages8;
  uint8_t* sEpi = s8 + S8 * Cfg::kStage8Bytes;
  uint8_t* sRed = sEpi + Cfg::kEpiBytes;  // split-K partial sums (kSplitK only)
  uint64_t* bars = reinterpret_cast<uint64_t*>(sRed + Cfg::kRedBytes);
  uint64_t* full = bars;
  uint64_t* empty = bars + S;
  uint64_t* tmem_full = bars + 2 * S;
  uint64_t* tmem_empty = bars + 2 * S + 2;
  uint64_t* stall_bar = bars + 2 * S + 4;
  uint64_t* drain_bar = bars + 2 * S + 5;
  uint64_t* full8 = bars + 2 * S + 6;
  uint64_t* empty8 = full8 + S8;
  uint64_t* red_full = empty8 + S8;       // [warp][slot], in the leader: peers' partials written
  uint64_t* red_empty = red_full + 2 * kEpiWarps;  // [warp][slot], in each peer: leader done reading
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(red_empty + 2 * kEpiWarps);
  static_assert((2 * S + 6 + 2 * S8 + 4 * kEpiWarps) * 8 + 4 <= Cfg::kBarBytes, "barrier area");

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const WaitCtx wc{p.err, p.timeout_ns};
  // split-K: the CTAs of a cluster share each tile, CTA `rank` taking k-blocks [k_lo, k_hi)
  const uint32_t rank = p.ksplit > 1 ? cluster_ctarank() : 0u;
  const int cluster_id = blockIdx.x / p.ksplit;
  const int num_clusters = gridDim.x / p.ksplit;
  const int k_lo = min(p.num_k_blocks, (int)rank * p.kb_split);
  const int k_hi = min(p.num_k_blocks, k_lo + p.kb_split);
  const int nkb = k_hi - k_lo;
  // units per tile: int8 drains its accumulator every kI8ChunkKBlocks k-blocks
  const int chunk_kb = kI8 ? kI8ChunkKBlocks : (nkb > 0 ? nkb : 1);
  const int units_per_tile = nkb > 0 ? (nkb + chunk_kb - 1) / chunk_kb : 1;

  if (warp == 0) {
    // the lanes of warp 0 initialise the barriers between them
    for (int s = lane; s < S; s += 32) {
      // generic: one arrive per plain-load warp; staged: one per converter warp
      mbar_init(&full[s], Tr::kTmaLoad ? 1 : (Tr::kStaged ? kConvGroupWarps : 4));
      mbar_init(&empty[s], 1);
    }
    for (int s = lane; s < S8; s += 32) {
      mbar_init(&full8[s], 1);
      mbar_init(&empty8[s], kConvGroupWarps);
    }
    if (lane < 2 * kEpiWarps) {
      mbar_init(&red_full[lane], 32 * (p.ksplit > 1 ? p.ksplit - 1 : 1));
      mbar_init(&red_empty[lane], 1);
    }
    if (lane < 2) {
      mbar_init(&tmem_full[lane], 1);
      mbar_init(&tmem_empty[lane], kEpiWarps);
    }
    if (lane == 0) {
      mbar_init(stall_bar, 1);
      mbar_init(drain_bar, 1);
    }
    fence_barrier_init();
  }
  if (threadIdx.x == 0) {
    if constexpr (Tr::kTmaLoad || Tr::kStaged) {
      prefetch_tmap(&p.tmA);
      prefetch_tmap(&p.tmB);
    }
    if (p.d_tma) prefetch_tmap(&p.tmD);
  }
  if (warp == Tr::kMmaWarp) {
    tmem_alloc(tmem_slot, Cfg::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  if (p.ksplit > 1)
    cluster_sync();  // every CTA's barriers initialised before any remote arrival
  else
    __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // the prologue above touched only shared and tensor memory and the kernel
  // parameters; global memory comes after the previous grid on the stream
  grid_dependency_wait();
  grid_dependents_launch();

  if (warp < Tr::kProdWarps) {
    // ---------------------------------------------------------------- producer
    if constexpr (Tr::kTmaLoad) {
      if (lane == 0) {
        // operands re-read by other tiles stay in L2; one read once goes first
        const uint64_t pol_a = p.a_stream ? policy_evict_first() : policy_evict_last();
        const uint64_t pol_b = p.b_stream ? policy_evict_first() : policy_evict_last();
        int stage = 0;
        uint32_t phase = 0;
        uint32_t issued_mask = 0, issued_parity = 0;
        bool ok = true;
        for (int t = cluster_id; ok && t < p.num_tiles; t += num_clusters) {
          int bz, mb, nb;
          tile_coords(t, p, bz, mb, nb);
          const int m0 = mb * p.maps.tile_m, n0 = nb * p.maps.tile_n;
          const int za = bz * p.a_bc, zb = bz * p.b_bc;
          const BoxMap am = p.maps.a, bmp = p.maps.b;
          for (int kb = k_lo; kb < k_hi; ++kb) {
            if (!mbar_wait(&empty[stage], phase ^ 1u, wc)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(&full[stage], p.stage_tx);
            uint8_t* a = sA + stage * kABytes;
            uint8_t* b = sB + stage * Cfg::kBBytes;
            const int k0 = kb * kBK;
            tma_load_boxes(a, &p.tmA, am, m0, k0, za, &full[stage], pol_a);
            tma_load_boxes(b, &p.tmB, bmp, n0, k0, zb, &full[stage], pol_b);
            issued_mask |= 1u << stage;
            issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
            if (++stage == S) {
              stage = 0;
              phase ^= 1u;
            }
          }
        }
        if (!ok) {
          // Let every load this thread started land before the CTA exits.
          for (int s = 0; s < S; ++s)
            if (issued_mask & (1u << s)) drain_wait(&full[s], (issued_parity >> s) & 1u, 100000000ull);
        }
      }
    } else if constexpr (Tr::kStaged) {
      if (warp == 0) {
        // TMA thread: raw int8 tiles into the staging ring
        if (lane == 0) {
          // operands re-read by other tiles stay in L2; one read once goes first
          const uint64_t pol_a = p.a_stream ? policy_evict_first() : policy_evict_last();
          const uint64_t pol_b = p.b_stream ? policy_evict_first() : policy_evict_last();
          int st8 = 0;
          uint32_t ph8 = 0;
          uint32_t issued_mask = 0, issued_parity = 0;
          bool ok = true;
          for (int t = cluster_id; ok && t < p.num_tiles; t += num_clusters) {
            int bz, mb, nb;
            tile_coords(t, p, bz, mb, nb);
            const int m0 = mb * p.maps.tile_m, n0 = nb * p.maps.tile_n;
            const int za = bz * p.a_bc, zb = bz * p.b_bc;
            const BoxMap am = p.maps.a, bmp = p.maps.b;
            for (int kb = k_lo; kb < k_hi; ++kb) {
              if (!mbar_wait(&empty8[st8], ph8 ^ 1u, wc)) {
                ok = false;
                break;
              }
              mbar_arrive_expect_tx(&full8[st8], Cfg::kStage8Bytes);
              uint8_t* a = s8 + st8 * Cfg::kStage8Bytes;
              uint8_t* b = a + kBM * kBK;
              const int k0 = kb * kBK;
              tma_load_boxes(a, &p.tmA, am, m0, k0, za, &full8[st8], pol_a);
              tma_load_boxes(b, &p.tmB, bmp, n0, k0, zb, &full8[st8], pol_b);
              issued_mask |= 1u << st8;
              issued_parity = (issued_parity & ~(1u << st8)) | (ph8 << st8);
              if (++st8 == S8) {
                st8 = 0;
                ph8 ^= 1u;
              }
            }
          }
          if (!ok) {
            for (int s2 = 0; s2 < S8; ++s2)
              if (issued_mask & (1u << s2)) drain_wait(&full8[s2], (issued_parity >> s2) & 1u, 100000000ull);
          }
        }
      } else {
        // converter warps: int8 staging slot -> fp16 MMA slot.  Group g widens
        // the k-blocks at positions j = g (mod kConvGroups) of the CTA's
        // k-block sequence, so the groups' conversions overlap.
        const int ctid = threadIdx.x - 32;  // 0 .. 32 kConvWarps - 1
        const int grp = ctid / (32 * kConvGroupWarps);
        const int gtid = ctid % (32 * kConvGroupWarps);
        bool ok = true;
        int j = 0;  // position in the k-block sequence
        for (int t = cluster_id; ok && t < p.num_tiles; t += num_clusters) {
          for (int kb = k_lo; kb < k_hi; ++kb, ++j) {
            if (j % kConvGroups != grp) continue;
            const int st8 = j % S8, stage = j % S;
            const uint32_t ph8 = (uint32_t)(j / S8) & 1u, phase = (uint32_t)(j / S) & 1u;
            if (!mbar_wait(&full8[st8], ph8, wc) || !mbar_wait(&empty[stage], phase ^ 1u, wc)) {
              ok = false;
              break;
            }
            const uint8_t* a8 = s8 + st8 * Cfg::kStage8Bytes;
            const uint8_t* b8 = a8 + kBM * kBK;
            uint8_t* b = sB + stage * Cfg::kBBytes;
            if constexpr (Tr::kATmem) {
              // the group's four warps cover the four TMEM lane quarters: lane l
              // of the warp in quarter q widens A row 32 q + l into that lane.
              // B's raw chunks are read first and its fp16 stores overlap the
              // tensor-memory store of A
              constexpr int kNT = 32 * kConvGroupWarps;
              constexpr int kBIt = I8Tile<BN, kBK, kNT>::kIters;
              static_assert(kBIt == I8Tile<kBK, BN, kNT>::kIters, "B chunks per thread, either majorness");
              uint4 wb[kBIt];
              if (!p.b_mn)
                i8_tile_load<BN, kBK, kNT>(b8, wb, gtid);
              else
                i8_tile_load<kBK, BN, kNT>(b8, wb, gtid);
              const int qa = warp & 3;
              uint32_t w[32];
              convert_i8_row_sw64(a8, qa * 32 + lane, w);
              tmem_st_32x32b_x32(tmem_base + ((uint32_t)(qa * 32) << 16) + Cfg::kATmemCol0 + stage * 32, w);
              if (!p.b_mn)
                i8_tile_widen_store<BN, kBK, kNT>(b, wb, gtid);
              else
                i8_tile_widen_store<kBK, BN, kNT>(b, wb, gtid);
              tmem_st_wait();
            } else {
              uint8_t* a = sA + stage * kABytes;
              if (!p.a_mn)
                convert_i8_tile<kBM, kBK, 32 * kConvGroupWarps>(a8, a, gtid);
              else
                convert_i8_tile<kBK, kBM, 32 * kConvGroupWarps>(a8, a, gtid);
              if (!p.b_mn)
                convert_i8_tile<BN, kBK, 32 * kConvGroupWarps>(b8, b, gtid);
              else
                convert_i8_tile<kBK, BN, 32 * kConvGroupWarps>(b8, b, gtid);
            }
            fence_proxy_async_smem();
            if constexpr (Tr::kATmem) tc_fence_before();  // the tensor-memory stores, before the arrive
            __syncwarp();
            if (lane == 0) {
              mbar_arrive(&full[stage]);
              mbar_arrive(&empty8[st8]);
            }
          }
        }
      }
    } else {
      const int tid = threadIdx.x;  // 0..127
      int stage = 0;
      uint32_t phase = 0;
      for (int t = cluster_id; t < p.num_tiles; t += num_clusters) {
        int bz, mb, nb;
        tile_coords(t, p, bz, mb, nb);
        const int m0 = mb * p.maps.tile_m, n0 = nb * p.maps.tile_n;
        constexpr int kInBytes = kI8 ? 1 : 2;
        const void* Ab = static_cast<const char*>(p.A) + (int64_t)bz * p.a_bs * kInBytes;
        const void* Bb = static_cast<const char*>(p.B) + (int64_t)bz * p.b_bs * kInBytes;
        constexpr int kConvIters = layout::StripMined{kBM, kBK, 128, 8}.iterations();
        ConvRow crow[Tr::kConv ? kConvIters : 1];
        if constexpr (Tr::kConv) {
          constexpr layout::StripMined cmap{kBM, kBK, 128, 8};
#pragma unroll
          for (int i = 0; i < kConvIters; ++i) crow[i] = conv_row(p, m0 + cmap.row(tid, i));
        }
        bool ok = true;
        for (int kb = k_lo; kb < k_hi; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1u, wc)) {
            ok = false;
            break;
          }
          uint8_t* a = sA + stage * kABytes;
          uint8_t* b = sB + stage * Cfg::kBBytes;
          const int k0 = kb * kBK;
          if constexpr (Tr::kConv)
            im2col_load_tile<kConvIters>(a, p, crow, k0, tid);
          else if (!p.a_mn)
            generic_load_tile<kBM, kBK, kI8>(a, Ab, p.lda, m0, k0, p.M, p.K, p.a_vec, tid);
          else
            generic_load_tile<kBK, kBM, kI8>(a, Ab, p.lda, k0, m0, p.K, p.M, p.a_vec, tid);
          if (!p.b_mn) {
            generic_load_tile<BN, kBK, kI8>(b, Bb, p.ldb, n0, k0, p.N, p.K, p.b_vec, tid);
          } else {
            if constexpr (BN >= 64) generic_load_tile<kBK, BN, kI8>(b, Bb, p.ldb, k0, n0, p.K, p.N, p.b_vec, tid);
          }
          // generic-proxy writes must be visible to the tensor core (async proxy)
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(&full[stage]);
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
      }
    }
  } else if (warp == Tr::kMmaWarp) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t idesc = idesc_f16(kBF16, p.a_mn != 0, p.b_mn != 0, kBM, BN);
      bool ok = true;
      bool any_mma = false;
      if (p.inject_stall) ok = mbar_wait(stall_bar, 0, wc);  // nothing arrives here
      int stage = 0;
      uint32_t phase = 0;
      int unit = 0;
      // descriptors are built once and stepped: the start address is a 14-bit
      // field at bit 0 (address >> 4) that no shared-memory offset overflows
      const uint64_t a_desc0 = smem_desc_sw128(smem_u32(sA), p.a_mn ? 8192u : 16u, 1024);
      const uint64_t b_desc0 = smem_desc_sw128(smem_u32(sB), p.b_mn ? 8192u : 16u, 1024);
      const uint64_t a_kstep = p.a_mn ? 2048u >> 4 : 32u >> 4, b_kstep = p.b_mn ? 2048u >> 4 : 32u >> 4;
      for (int t = cluster_id; ok && t < p.num_tiles; t += num_clusters) {
        for (int u = 0; ok && u < units_per_tile; ++u, ++unit) {
          const int acc = unit & 1;
          const uint32_t acc_phase = (unit >> 1) & 1;
          if (!mbar_wait(&tmem_empty[acc], acc_phase ^ 1u, wc)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d_tmem = tmem_base + acc * BN;
          const int kb0 = k_lo + u * chunk_kb;
          const int kb1 = min(k_hi, kb0 + chunk_kb);
          for (int kb = kb0; kb < kb1; ++kb) {
            if (!mbar_wait(&full[stage], phase, wc)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint64_t bd = b_desc0 + (uint32_t)stage * (Cfg::kBBytes >> 4);
            if constexpr (Tr::kATmem) {
              // A from tensor memory: 16 k of fp16 = 8 columns per MMA
              const uint32_t at = tmem_base + Cfg::kATmemCol0 + (uint32_t)stage * 32;
              mma_f16_ta(d_tmem, at, bd, idesc, kb != kb0);
#pragma unroll
              for (int k = 1; k < kBK / kUmmaK; ++k) mma_f16_ta(d_tmem, at + 8 * k, bd + k * b_kstep, idesc, 1u);
            } else {
              const uint64_t ad = a_desc0 + (uint32_t)stage * (kABytes >> 4);
              mma_f16(d_tmem, ad, bd, idesc, kb != kb0);
#pragma unroll
              for (int k = 1; k < kBK / kUmmaK; ++k) mma_f16(d_tmem, ad + k * a_kstep, bd + k * b_kstep, idesc, 1u);
            }
            any_mma = true;
            mma_commit(&empty[stage]);
            if (++stage == S) {
              stage = 0;
              phase ^= 1u;
            }
          }
          if (!ok) break;
          if (kb1 <= kb0)
            mbar_arrive(&tmem_full[acc]);
          else
            mma_commit(&tmem_full[acc]);
        }
      }
      if (any_mma) {
        // Every MMA must have finished with TMEM before it is freed.
        mma_commit(drain_bar);
        drain_wait(drain_bar, 0, 100000000ull);
      }
    }
  } else {
    // ---------------------------------------------------------------- epilogue
    const int ew = warp - Tr::kEpiWarp0;  // epilogue warp 0..3 (owns a staging area)
    const int q = warp & 3;               // TMEM lane quarter this warp may access
    const int row_in_tile = (q * 32 + lane) * p.maps.epi_row_step;
    uint8_t* stage_buf = sEpi + ew * 2 * Tr::kEpiBufBytes;
    int buf = 0;
    int unit = 0;
    const bool has_k = nkb > 0;
    const uint32_t lane_base = (uint32_t)(q * 32) * p.maps.tmem_row_step;
    const int chunk = p.maps.epi_chunk;
    bool ok = true;
    int red_it = 0;  // split-K: partial-sum chunks exchanged so far
    for (int t = cluster_id; ok && t < p.num_tiles; t += num_clusters) {
      int bz, mb, nb;
      tile_coords(t, p, bz, mb, nb);
      const int m0 = mb * p.maps.tile_m, n0 = nb * p.maps.tile_n;
      const int grow = m0 + row_in_tile;
      const bool row_ok = grow < p.M;
      const EpiPtrs ep = epi_ptrs(p, bz, Tr::kOutBytes);

      // int8: exact int32 sums of the per-chunk partials, kept in TMEM columns
      // [2 BN, 3 BN) of this warp's lanes (each partial is an integer below
      // 2^24 in magnitude, exact in fp32)
      const uint32_t sum_cols = tmem_base + lane_base + 2 * BN;
      if constexpr (kI8) {
        for (int u = 0; u < units_per_tile; ++u, ++unit) {
          const int acc = unit & 1;
          if (!mbar_wait(&tmem_full[acc], (unit >> 1) & 1, wc)) {
            ok = false;
            break;
          }
          tc_fence_after();
          if (has_k) {
#pragma unroll 1
            for (int c = 0; c < BN / kEpiCols; ++c) {
              uint32_t r[32], sm[32];
              tmem_ld_32x32b_x32(tmem_base + lane_base + acc * BN + c * chunk, r);
              if (u > 0) tmem_ld_32x32b_x32(sum_cols + c * chunk, sm);
              tmem_ld_wait();
#pragma unroll
              for (int j = 0; j < 32; ++j)
                sm[j] = (uint32_t)((u > 0 ? (int32_t)sm[j] : 0) + __float2int_rn(__uint_as_float(r[j])));
              tmem_st_32x32b_x32(sum_cols + c * chunk, sm);
            }
            tmem_st_wait();
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&tmem_empty[acc]);
        }
        if (!ok) break;
      }
      // fp16/bf16: the first chunk's C is fetched before waiting for the
      // accumulator, so its latency overlaps the mainloop
      const bool writes_out = p.ksplit == 1 || rank == 0;
      CChunk16 cc;
      if constexpr (!kI8) {
        if (writes_out) {
          c_prefetch_trans(p, ep, m0, n0, BN, row_in_tile);
          c_fetch16(p, ep, c_path(p, ep, n0), grow, n0, lane, cc);
        }
        if (!mbar_wait(&tmem_full[unit & 1], (unit >> 1) & 1, wc)) break;
        tc_fence_after();
      }
      const int acc = unit & 1;  // fp16/bf16: the unit being drained below

      RowCarry carry{};
#pragma unroll 1
      for (int c = 0; c < BN / kEpiCols; ++c) {
        const int gcol0 = n0 + c * chunk;
        uint32_t packed[Tr::kOutBytes == 4 ? 32 : 16];
        if constexpr (kI8) {
          // D = sum (+ C when beta == 1); alpha == 1 (checked on the host)
          int32_t v[32];
          if (has_k) {
            uint32_t sm[32];
            tmem_ld_32x32b_x32(sum_cols + c * chunk, sm);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = (int32_t)sm[j];
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = 0;
          }
          if (p.beta != 0.0f && row_ok && p.d_trans) {
            const int32_t* ccol = reinterpret_cast<const int32_t*>(ep.C) + grow;
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (gcol0 + j < p.N) v[j] += __ldg(ccol + (int64_t)(gcol0 + j) * p.ldc);
          } else if (p.beta != 0.0f && row_ok) {
            const int32_t* crow = reinterpret_cast<const int32_t*>(ep.C) + (int64_t)grow * p.ldc + gcol0;
            const bool vec = ((p.ldc & 3) == 0) && ((reinterpret_cast<uintptr_t>(ep.C) & 15) == 0) &&
                             (gcol0 + 32 <= p.N);
            if (vec) {
#pragma unroll
              for (int u4 = 0; u4 < 8; ++u4) {
                const int4 w = __ldg(reinterpret_cast<const int4*>(crow) + u4);
                v[4 * u4] += w.x;
                v[4 * u4 + 1] += w.y;
                v[4 * u4 + 2] += w.z;
                v[4 * u4 + 3] += w.w;
              }
            } else {
#pragma unroll
              for (int j = 0; j < 32; ++j)
                if (gcol0 + j < p.N) v[j] += __ldg(crow + j);
            }
          }
#pragma unroll
          for (int j = 0; j < 32; ++j) packed[j] = (uint32_t)v[j];
        } else {
          uint32_t r[32];
          if (has_k) {
            tmem_ld_32x32b_x32(tmem_base + lane_base + acc * BN + c * chunk, r);
            tmem_ld_wait();
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) r[j] = 0u;
          }
          if (c == BN / kEpiCols - 1) {
            // accumulator fully read: hand it back to the MMA issuer
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tmem_empty[acc]);
          }
          if constexpr (Cfg::kSplitK) {
            if (p.ksplit > 1) {
              // split-K: peers hand their fp32 partial chunk to the leader (rank 0)
              // through their own shared memory; the leader sums in rank order
              const int slot = red_it & 1;
              const uint32_t ph = (red_it >> 1) & 1;
              ++red_it;
              uint64_t* rf = &red_full[ew * 2 + slot];
              uint64_t* re = &red_empty[ew * 2 + slot];
              uint8_t* row = sRed + (ew * 2 + slot) * Cfg::kRedSlotBytes + lane * 128;
              if (rank != 0) {
                if (!mbar_wait_cluster(re, ph ^ 1u, wc)) {
                  ok = false;
                  break;
                }
#pragma unroll
                for (int ch = 0; ch < 8; ++ch)  // 16-byte chunk ch of the row, rotated by lane
                  *reinterpret_cast<uint4*>(row + ((ch ^ (lane & 7)) << 4)) =
                      make_uint4(r[4 * ch], r[4 * ch + 1], r[4 * ch + 2], r[4 * ch + 3]);
                mbar_arrive_cluster(mapa_shared(smem_u32(rf), 0));
                continue;
              }
              if (!mbar_wait_cluster(rf, ph, wc)) {
                ok = false;
                break;
              }
              for (int pr = 1; pr < p.ksplit; ++pr) {
                const uint32_t src = mapa_shared(smem_u32(row), (uint32_t)pr);
                // all eight remote loads in flight before the first use
                uint4 w[8];
#pragma unroll
                for (int ch = 0; ch < 8; ++ch) w[ch] = ld_shared_cluster_v4(src + ((ch ^ (lane & 7)) << 4));
#pragma unroll
                for (int ch = 0; ch < 8; ++ch) {
                  r[4 * ch] = __float_as_uint(__uint_as_float(r[4 * ch]) + __uint_as_float(w[ch].x));
                  r[4 * ch + 1] = __float_as_uint(__uint_as_float(r[4 * ch + 1]) + __uint_as_float(w[ch].y));
                  r[4 * ch + 2] = __float_as_uint(__uint_as_float(r[4 * ch + 2]) + __uint_as_float(w[ch].z));
                  r[4 * ch + 3] = __float_as_uint(__uint_as_float(r[4 * ch + 3]) + __uint_as_float(w[ch].w));
                }
              }
              // the peers' slots may be reused: every lane's loads above have
              // returned (their values are summed), so one relaxed arrive per
              // warp and peer suffices; a release here would fence each arrive
              __syncwarp();
              if (lane == 0)
                for (int pr = 1; pr < p.ksplit; ++pr) mbar_arrive_cluster_relaxed(mapa_shared(smem_u32(re), (uint32_t)pr));
            }
          }
          epi_f16_values<kBF16>(p, r, row_ok, grow, gcol0, packed, c_path(p, ep, gcol0), cc, ep);
          if (c + 1 < BN / kEpiCols) c_fetch16(p, ep, c_path(p, ep, gcol0 + chunk), grow, gcol0 + chunk, lane, cc);
        }

        epi_store_chunk<Tr::kOutBytes>(p, packed, row_ok, grow, gcol0, grow - lane * p.maps.epi_row_step, stage_buf,
                                       Tr::kEpiBufBytes, buf, carry, c == BN / kEpiCols - 1, lane, ep);
      }
      if constexpr (!kI8) ++unit;
      if (!ok) break;
    }
    if (p.d_tma && lane == 0) bulk_wait_all();
  }

  __syncthreads();
  if (p.ksplit > 1) cluster_sync();  // no CTA leaves while a peer may still read its partials
  if (warp == Tr::kMmaWarp) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, Cfg::kTmemCols);
  }
}

}  // namespace ttc
