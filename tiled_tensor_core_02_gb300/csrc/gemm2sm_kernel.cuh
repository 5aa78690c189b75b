// CTA-pair (2-SM) variant of the fp16/bf16 TMA GEMM: one cluster of two CTAs
// computes a 256 x 256 output tile with tcgen05.mma.cta_group::2 (M = 256,
// N = 256, K = 16).
//
// Each CTA stages only its own half of the operands: rows [128 r, 128 r + 128)
// of the A tile and columns [128 r, 128 r + 128) of the B tile (r = the CTA's
// rank in the pair), at the same shared-memory offsets in both CTAs.  One
// thread of the even CTA issues the pair MMA, which reads A and B halves from
// both CTAs and writes rows [128 r, 128 r + 128) of the accumulator into CTA
// r's TMEM.  Per SM this halves the B operand traffic of the single-CTA
// 128 x 256 tile while keeping the same per-SM work.
//
// Synchronisation (barrier -> who arrives -> who waits):
//   full[s]      even CTA only; its producer arms it with both CTAs' bytes, both
//                CTAs' TMA loads complete on it (.cta_group::2); MMA waits.
//   empty[s]     both CTAs; the MMA's commit is multicast to both; producers wait.
//   tmem_full[a] both CTAs; multicast commit after a tile's last k-block;
//                epilogue warps wait.
//   tmem_empty[a] even CTA only; all 16 epilogue warps of the pair arrive (the
//                odd CTA's remotely); the MMA waits before reusing accumulator a.
//                The arrive is relaxed: it follows tcgen05.wait::ld, so the
//                warp's reads of the accumulator are complete, and it publishes
//                no memory writes (a release arrive would also wait for the
//                warp's outstanding C loads and stores).
// Epilogue: eight warps, two per TMEM lane quarter; the first four drain the
// left half of a tile's 32-column chunks, the other four the right half.  For
// outputs written with plain stores (rows TMA cannot store) a variant has
// twelve, three per quarter, each draining a third of the chunks.
// The layout of a CTA's half tiles, the epilogue and the error handling are
// those of gemm_kernel (one CTA); every wait is bounded.
//
// The pairs walk work units (GemmParams::num_units): whole tiles, then, for
// a last partial wave, half tiles of N = BN / 2 columns.  A half unit issues
// MMAs with N = BN / 2, and each CTA uses the first BN / 4 columns of its
// usual B box, which it loads starting at its own columns.
//
// int8 (kI8): the operands are fp16 copies of int8 matrices (every int8 value
// is exact in fp16, every product exact in fp32).  The issuer starts a fresh
// accumulator every kI8ChunkKBlocks k-blocks (1024 of K), so each partial sum
// is an integer below 2^24 in magnitude and exact in fp32; the epilogue warps
// add the partials as int32 into running sums held in their registers (a
// thread's row, its half of the tile's columns) and store the int32 tile once
// per unit, after the last partial.
#pragma once
#include "gemm_kernel.cuh"

namespace ttc {

constexpr int kPairBM = 256;
constexpr int kPairEpiWarps = 8;   // by default two per TMEM lane quarter, each taking half of a tile's columns
constexpr int kPairThreads = 64 + 32 * kPairEpiWarps;  // warp 0 producer, warp 1 TMEM + MMA, then the epilogue

// Pair tile 256 x BN (BN = 256, 224, 192 or 128): each CTA stages 128 A rows and
// BN / 2 B columns per k-block.  A pipeline stage holds kKPS = 2 k-blocks
// (128 of K, 8 MMAs per barrier round trip): measured on GB300, one full/empty
// round trip per 4 MMAs holds the pair to ~85 ns per N = 256 MMA, one per 8
// MMAs to the tensor pipe's own ~67 ns, with as few as 2 stages.
// kEW: epilogue warps, 8 (two per TMEM lane quarter, each draining half of a
// tile's columns) or 12 (three per quarter, a third each) for outputs whose
// rows TMA cannot store, written with plain stores and no staging buffers.
template <int BN, bool kI8 = false, int kEW = 8>
struct PairCfg {
  static constexpr int kBHalf = BN / 2;
  static constexpr int kKPS = 2;                        // k-blocks per stage
  static constexpr int kAHalfBytes = 128 * kBK * 2;     // one k-block of A rows: 16 KiB
  static constexpr int kBHalfBytes = kBHalf * kBK * 2;  // one k-block of B columns: 16 / 14 / 12 / 8 KiB
  static constexpr int kKBlockBytes = kAHalfBytes + kBHalfBytes;
  static constexpr int kStageBytes = kKPS * kKBlockBytes;
  static constexpr int kOutBytes = kI8 ? 4 : 2;
  static constexpr int kEpiBufBytes = 32 * kEpiCols * kOutBytes;
  // staging buffers per epilogue warp: two, or one for int8, whose warps
  // store their chunks once per tile, or none with 12 epilogue warps
  static constexpr int kEpiBufs = kI8 ? 1 : kEW == 8 ? 2 : 0;
  static constexpr int kEpiBytes = kEW * kEpiBufs * kEpiBufBytes;
  static constexpr int kBarBytes = 256;
  static constexpr int kSmemLimit = 227 * 1024;
  static constexpr int kStagesRaw = (kSmemLimit - 1024 - kBarBytes - kEpiBytes) / kStageBytes;
  static constexpr int kStages = kStagesRaw > 8 ? 8 : kStagesRaw;
  static constexpr int kTmemCols = 2 * BN > 256 ? 512 : 256;  // two accumulators, a power of two
  static constexpr int kSmemBytes = 1024 + kStages * kStageBytes + kEpiBytes + kBarBytes;
  static_assert(BN == 256 || BN == 224 || BN == 192 || BN == 128, "pair tile width");
  static_assert(!kI8 || BN == 256, "int8: 256-wide tiles (a warp's running sums cover at most 4 chunks)");
  static_assert(kEW == 8 || (kEW == 12 && !kI8), "epilogue warps: 8, or 12 for 16-bit plain-store outputs");
  static_assert(kStages >= 2, "pipeline depth");
  static_assert(kSmemBytes <= kSmemLimit, "shared memory budget");
};

// tma_load_boxes for the pair kernel: completion counted on the even CTA's
// barrier (.cta_group::2).
// A CTA's share of a pair tile is at most 128 rows (columns): one or two boxes.
__device__ __forceinline__ void tma_load_boxes_pair(uint8_t* dst, const CUtensorMap* m, const BoxMap bm, int r0,
                                                    int k0, int z, uint32_t bar_leader, uint64_t pol) {
  const int x = bm.k_inner ? k0 : r0, y = bm.k_inner ? r0 : k0;
  tma_load_3d_pair(dst, m, x, y, z, bar_leader, pol);
  if (bm.boxes > 1) tma_load_3d_pair(dst + bm.smem_step, m, x + bm.box_step, y, z, bar_leader, pol);
}

template <int BN, bool kBF16, bool kI8 = false, int kEW = 8>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(64 + 32 * kEW, 1)
    gemm_pair_kernel(const __grid_constant__ GemmParams p) {
  static_assert(!(kI8 && kBF16), "int8 runs on fp16 copies");
  using PairCfg = ttc::PairCfg<BN, kI8, kEW>;
  constexpr int kPairBN = BN;
  constexpr int S = PairCfg::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  constexpr int KPS = PairCfg::kKPS;
  uint8_t* sA = smem;  // [stage][k-block of the stage][128 rows x 64]
  uint8_t* sB = sA + S * KPS * PairCfg::kAHalfBytes;
  uint8_t* sEpi = sB + S * KPS * PairCfg::kBHalfBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sEpi + PairCfg::kEpiBytes);
  uint64_t* full = bars;
  uint64_t* empty = bars + S;
  uint64_t* tmem_full = bars + 2 * S;
  uint64_t* tmem_empty = bars + 2 * S + 2;
  uint64_t* stall_bar = bars + 2 * S + 4;
  uint64_t* drain_bar = bars + 2 * S + 5;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * S + 6);
  static_assert((2 * S + 6) * 8 + 4 <= PairCfg::kBarBytes, "barrier area");

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int pair = blockIdx.x >> 1;
  const int num_pairs = gridDim.x >> 1;
  const WaitCtx wc{p.err, p.timeout_ns};

  if (warp == 0) {
    // the lanes of warp 0 initialise the barriers between them
    for (int s = lane; s < S; s += 32) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    if (lane < 2) {
      mbar_init(&tmem_full[lane], 1);
      mbar_init(&tmem_empty[lane], 2 * kEW);
    }
    if (lane == 0) {
      mbar_init(stall_bar, 1);
      mbar_init(drain_bar, 1);
    }
    fence_barrier_init();
  }
  if (threadIdx.x == 0) {
    prefetch_tmap(&p.tmA);
    prefetch_tmap(&p.tmB);
    if (p.b_half_map) prefetch_tmap(&p.tmBh);
    if (p.d_tma) prefetch_tmap(&p.tmD);
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_slot, PairCfg::kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync();  // barrier initialisation and the TMEM address visible to both CTAs
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // the prologue above touched only shared and tensor memory and the kernel
  // parameters; global memory comes after the previous grid on the stream
  grid_dependency_wait();
  grid_dependents_launch();

  if (warp == 0) {
    // ---------------------------------------------------------------- producer (both CTAs)
    if (lane == 0) {
      // operands re-read by other tiles stay in L2; one read once goes first
      const uint64_t pol_a = p.a_stream ? policy_evict_first() : policy_evict_last();
      const uint64_t pol_b = p.b_stream ? policy_evict_first() : policy_evict_last();
      int stage = 0;
      uint32_t phase = 0;
      uint32_t armed_mask = 0, armed_parity = 0;
      bool ok = true;
      for (int u = pair; ok && u < p.num_units; u += num_pairs) {
        int t, n_off;
        bool half;
        pair_unit(p, u, p.maps.half_n, t, n_off, half);
        int bz, mb, nb;
        tile_coords(t, p, bz, mb, nb);
        const int za = bz * p.a_bc, zb = bz * p.b_bc;
        const int m0 = mb * p.maps.tile_m + (int)rank * p.maps.cta_m;  // this CTA's A rows
        // this CTA's B columns: a half unit uses the first cta_n_half of the
        // usual box, and loads only those where it can (MN-major slabs of 64
        // columns, or the half-width map of a K-major B); otherwise it loads the
        // whole box and the rest is not read
        const int n0 = nb * p.maps.tile_n + n_off + (int)rank * (half ? p.maps.cta_n_half : p.maps.cta_n);
        const bool b_half_box = half && (p.b_mn || p.b_half_map);
        const BoxMap amap = p.maps.a;
        const BoxMap bmap = b_half_box ? p.maps.b_half : p.maps.b;
        const CUtensorMap* tmb = b_half_box && !p.b_mn ? &p.tmBh : &p.tmB;
        const int kblock_tx = amap.boxes * amap.smem_step + bmap.boxes * bmap.smem_step;
        // convolution: window corner of output pixel m0 (rows past the end start
        // beyond the last image, where the im2col box reads zeros)
        int cv_n = 0, cv_h0 = 0, cv_w0 = 0;
        if (p.cv_tma) {
          const int pq = p.cv_p * p.cv_q;
          cv_n = m0 / pq;
          const int rem = m0 - cv_n * pq;
          const int pp = rem / p.cv_q;
          cv_h0 = pp * p.cv_sh - p.cv_ph;
          cv_w0 = (rem - pp * p.cv_q) * p.cv_sw - p.cv_pw;
        }
        for (int kb0 = 0; kb0 < p.num_k_blocks; kb0 += KPS) {
          const int nkb = min(KPS, p.num_k_blocks - kb0);
          if (!mbar_wait(&empty[stage], phase ^ 1u, wc)) {
            ok = false;
            break;
          }
          const uint32_t full_leader = mapa_shared(smem_u32(&full[stage]), 0);
          if (leader) {
            mbar_arrive_expect_tx(&full[stage], 2 * nkb * kblock_tx);
            armed_mask |= 1u << stage;
            armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
          }
          for (int j = 0; j < nkb; ++j) {
            const int kb = kb0 + j;
            uint8_t* a = sA + (stage * KPS + j) * PairCfg::kAHalfBytes;
            uint8_t* b = sB + (stage * KPS + j) * PairCfg::kBHalfBytes;
            const int k0 = kb * kBK;
            if (p.cv_tma) {
              const int tap = kb / p.cv_cblk;
              const int c0 = (kb - tap * p.cv_cblk) * kBK;
              const int rr = tap / p.cv_s;
              const int ss = tap - rr * p.cv_s;
              tma_load_im2col_4d_pair(a, &p.tmA, c0, cv_w0, cv_h0, cv_n, (uint16_t)(ss * p.cv_dw),
                                      (uint16_t)(rr * p.cv_dh), full_leader, pol_a);
            } else {
              tma_load_boxes_pair(a, &p.tmA, amap, m0, k0, za, full_leader, pol_a);
            }
            tma_load_boxes_pair(b, tmb, bmap, n0, k0, zb, full_leader, pol_b);
          }
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok && leader) {
        // every stage this CTA armed completes once both CTAs' loads for it
        // have landed; wait for them before the pair may exit
        for (int s = 0; s < S; ++s)
          if (armed_mask & (1u << s)) drain_wait(&full[s], (armed_parity >> s) & 1u, 100000000ull);
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer (even CTA)
    if (leader && lane == 0) {
      const uint32_t idesc_full = idesc_f16(kBF16, p.a_mn != 0, p.b_mn != 0, kPairBM, kPairBN);
      const uint32_t idesc_half = idesc_f16(kBF16, p.a_mn != 0, p.b_mn != 0, kPairBM, kPairBN / 2);
      bool ok = true;
      bool any_mma = false;
      if (p.inject_stall) ok = mbar_wait(stall_bar, 0, wc);  // nothing arrives here
      int stage = 0;
      uint32_t phase = 0;
      int it = 0;
      // descriptors are built once and stepped: the start address is a 14-bit
      // field at bit 0 (address >> 4) that no shared-memory offset overflows
      const uint64_t a_desc0 = smem_desc_sw128(smem_u32(sA), p.a_mn ? 8192u : 16u, 1024);
      const uint64_t b_desc0 = smem_desc_sw128(smem_u32(sB), p.b_mn ? 8192u : 16u, 1024);
      const uint64_t a_kstep = p.a_mn ? 2048u >> 4 : 32u >> 4, b_kstep = p.b_mn ? 2048u >> 4 : 32u >> 4;
      // k-blocks per accumulator: a unit's all, or for int8 1024-deep chunks
      // (a multiple of KPS, so the stages of a unit never straddle two)
      const int nkbt = p.num_k_blocks;
      const int chunk_kb = kI8 ? kI8ChunkKBlocks : (nkbt > 0 ? nkbt : 1);
      const int chunks_per_unit = nkbt > 0 ? (nkbt + chunk_kb - 1) / chunk_kb : 1;
      static_assert(!kI8 || kI8ChunkKBlocks % KPS == 0, "accumulator chunks hold whole stages");
      for (int u = pair; ok && u < p.num_units; u += num_pairs) {
        const uint32_t idesc = u >= p.tail_from ? idesc_half : idesc_full;
        for (int kc = 0; ok && kc < chunks_per_unit; ++kc, ++it) {
          const int acc = it & 1;
          const uint32_t acc_phase = (it >> 1) & 1;
          if (!mbar_wait_cluster(&tmem_empty[acc], acc_phase ^ 1u, wc)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d_tmem = tmem_base + acc * kPairBN;
          const int kbeg = kc * chunk_kb, kend = min(nkbt, kbeg + chunk_kb);
          for (int kb0 = kbeg; kb0 < kend; kb0 += KPS) {
            const int nkb = min(KPS, kend - kb0);
            if (!mbar_wait(&full[stage], phase, wc)) {
              ok = false;
              break;
            }
            tc_fence_after();
#pragma unroll
            for (int j = 0; j < KPS; ++j) {
              if (j < nkb) {
                const uint64_t ad = a_desc0 + (uint32_t)(stage * KPS + j) * (PairCfg::kAHalfBytes >> 4);
                const uint64_t bd = b_desc0 + (uint32_t)(stage * KPS + j) * (PairCfg::kBHalfBytes >> 4);
                mma_f16_pair(d_tmem, ad, bd, idesc, ((kb0 - kbeg) | j) != 0);
#pragma unroll
                for (int k = 1; k < kBK / kUmmaK; ++k)
                  mma_f16_pair(d_tmem, ad + k * a_kstep, bd + k * b_kstep, idesc, 1u);
              }
            }
            any_mma = true;
            mma_commit_pair(&empty[stage], 0x3);
            if (++stage == S) {
              stage = 0;
              phase ^= 1u;
            }
          }
          if (!ok) break;
          if (kend <= kbeg) {
            mbar_arrive(&tmem_full[acc]);
            mbar_arrive_cluster(mapa_shared(smem_u32(&tmem_full[acc]), 1));
          } else {
            mma_commit_pair(&tmem_full[acc], 0x3);
          }
        }
      }
      if (any_mma) {
        // every MMA must have finished with both CTAs' TMEM before it is freed
        mma_commit_pair(drain_bar, 0x1);
        drain_wait(drain_bar, 0, 100000000ull);
      }
    }
  } else {
    // ---------------------------------------------------------------- epilogue (both CTAs)
    const int ew = warp - 2;
    const int q = warp & 3;
    const int part = ew >> 2;  // which half (third) of a tile's columns this warp drains
    constexpr int kParts = kEW / 4;
    uint8_t* stage_buf = sEpi + ew * PairCfg::kEpiBufs * PairCfg::kEpiBufBytes;
    int buf = 0;
    int it = 0;
    const bool has_k = p.num_k_blocks > 0;
    // this thread's accumulator row within the CTA's half of a tile, and the
    // TMEM address of its warp's first row
    const int row_in_tile = (q * 32 + lane) * p.maps.epi_row_step;
    const uint32_t lane_base = (uint32_t)(q * 32) * p.maps.tmem_row_step;
    const int chunk = p.maps.epi_chunk;
    // this thread's row of a tile's C, toward L2 one tile ahead of its epilogue
    // (the first tile's during the first mainloop)
    auto prefetch_c = [&](int unit) {
      if (unit >= p.num_units || p.beta == 0.0f) return;
      int pt, pn_off;
      bool phalf;
      pair_unit(p, unit, p.maps.half_n, pt, pn_off, phalf);
      int pbz, pmb, pnb;
      tile_coords(pt, p, pbz, pmb, pnb);
      c_prefetch_row(p, epi_ptrs(p, pbz, 2), pmb * p.maps.tile_m + (int)rank * p.maps.cta_m + row_in_tile,
                     pnb * p.maps.tile_n + pn_off, phalf ? p.maps.half_n : p.maps.tile_n);
    };
    if constexpr (kI8) {
      // int8: running int32 sums of this thread's row over its part's (at most
      // four) 32-column chunks, one accumulator chunk (1024 of K) at a time
      const int nkbt = p.num_k_blocks;
      const int chunks_per_unit = nkbt > 0 ? (nkbt + kI8ChunkKBlocks - 1) / kI8ChunkKBlocks : 1;
      bool ok = true;
      for (int u = pair; ok && u < p.num_units; u += num_pairs) {
        int t, n_off;
        bool half;
        pair_unit(p, u, p.maps.half_n, t, n_off, half);
        const int chunks = (half ? kPairBN / 2 : kPairBN) / kEpiCols;
        int bz, mb, nb;
        tile_coords(t, p, bz, mb, nb);
        const int m0 = mb * p.maps.tile_m + (int)rank * p.maps.cta_m;
        const int n0 = nb * p.maps.tile_n + n_off;
        const int grow = m0 + row_in_tile;
        const bool row_ok = grow < p.M;
        const EpiPtrs ep = epi_ptrs(p, bz, 4);
        const int c_lo = part == 0 ? 0 : (chunks + 1) / 2;
        const int c_hi = part == 0 ? (chunks + 1) / 2 : chunks;
        int32_t sums[4][32];
#pragma unroll
        for (int cc = 0; cc < 4; ++cc)
#pragma unroll
          for (int j = 0; j < 32; ++j) sums[cc][j] = 0;
        for (int kc = 0; kc < chunks_per_unit; ++kc, ++it) {
          const int acc = it & 1;
          if (!mbar_wait(&tmem_full[acc], (it >> 1) & 1, wc)) {
            ok = false;
            break;
          }
          tc_fence_after();
          if (has_k) {
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) {
              if (c_lo + cc < c_hi) {
                uint32_t r[32];
                tmem_ld_32x32b_x32(tmem_base + lane_base + acc * kPairBN + (c_lo + cc) * chunk, r);
                tmem_ld_wait();
                // an integer below 2^24 in magnitude: exact in fp32 and in the conversion
#pragma unroll
                for (int j = 0; j < 32; ++j) sums[cc][j] += __float2int_rn(__uint_as_float(r[j]));
              }
            }
          }
          // this warp's accumulator columns are read: tell the even CTA's issuer
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive_cluster_relaxed(mapa_shared(smem_u32(&tmem_empty[acc]), 0));
        }
        if (!ok) break;
        RowCarry carry{};
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          const int c = c_lo + cc;
          if (c < c_hi) {
            const int gcol0 = n0 + c * chunk;
            uint32_t packed[32];
            if (p.beta != 0.0f && row_ok) {
              // D = sums + C (beta == 1, checked on the host)
              const int32_t* crow = reinterpret_cast<const int32_t*>(ep.C) + (int64_t)grow * p.ldc + gcol0;
              const bool vec = ((p.ldc & 3) == 0) && ((reinterpret_cast<uintptr_t>(ep.C) & 15) == 0) &&
                               (gcol0 + 32 <= p.N);
              if (vec) {
#pragma unroll
                for (int u4 = 0; u4 < 8; ++u4) {
                  const int4 w = __ldg(reinterpret_cast<const int4*>(crow) + u4);
                  packed[4 * u4] = (uint32_t)(sums[cc][4 * u4] + w.x);
                  packed[4 * u4 + 1] = (uint32_t)(sums[cc][4 * u4 + 1] + w.y);
                  packed[4 * u4 + 2] = (uint32_t)(sums[cc][4 * u4 + 2] + w.z);
                  packed[4 * u4 + 3] = (uint32_t)(sums[cc][4 * u4 + 3] + w.w);
                }
              } else {
#pragma unroll
                for (int j = 0; j < 32; ++j)
                  packed[j] = (uint32_t)(sums[cc][j] + (gcol0 + j < p.N ? __ldg(crow + j) : 0));
              }
            } else {
#pragma unroll
              for (int j = 0; j < 32; ++j) packed[j] = (uint32_t)sums[cc][j];
            }
            // one staging buffer per warp: the previous chunk's store must have read it
            if (lane == 0) bulk_wait_read<0>();
            __syncwarp();
            epi_store_chunk<4>(p, packed, row_ok, grow, gcol0, grow - lane * p.maps.epi_row_step, stage_buf, 0, buf,
                               carry, c == c_hi - 1, lane, ep);
          }
        }
      }
    } else {
      if (part == 0) prefetch_c(pair);
      for (int u = pair; u < p.num_units; u += num_pairs, ++it) {
        int t, n_off;
        bool half;
        pair_unit(p, u, p.maps.half_n, t, n_off, half);
        const int chunks = (half ? kPairBN / 2 : kPairBN) / kEpiCols;
        const int acc = it & 1;
        int bz, mb, nb;
        tile_coords(t, p, bz, mb, nb);
        const int m0 = mb * p.maps.tile_m + (int)rank * p.maps.cta_m;
        const int n0 = nb * p.maps.tile_n + n_off;
        const int grow = m0 + row_in_tile;
        const bool row_ok = grow < p.M;
        const EpiPtrs ep = epi_ptrs(p, bz, 2);
        if (part == 0) prefetch_c(u + num_pairs);
        const int c_lo = (part * chunks + kParts - 1) / kParts;
        const int c_hi = ((part + 1) * chunks + kParts - 1) / kParts;
        // the first chunk's C is fetched before waiting for the accumulator
        CChunk16 cc;
        c_fetch16(p, ep, c_path(p, ep, n0 + c_lo * chunk), grow, n0 + c_lo * chunk, lane, cc);
        if (!mbar_wait(&tmem_full[acc], (it >> 1) & 1, wc)) break;
        tc_fence_after();
        if (c_lo == c_hi) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive_cluster_relaxed(mapa_shared(smem_u32(&tmem_empty[acc]), 0));
        }
        RowCarry carry{};
  #pragma unroll 1
        for (int c = c_lo; c < c_hi; ++c) {
          const int gcol0 = n0 + c * chunk;
          uint32_t r[32];
          if (has_k) {
            tmem_ld_32x32b_x32(tmem_base + lane_base + acc * kPairBN + c * chunk, r);
            tmem_ld_wait();
          } else {
  #pragma unroll
            for (int j = 0; j < 32; ++j) r[j] = 0u;
          }
          if (c == c_hi - 1) {
            // this warp's accumulator columns are read: tell the even CTA's issuer
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster_relaxed(mapa_shared(smem_u32(&tmem_empty[acc]), 0));
          }
          uint32_t packed[16];
          epi_f16_values<kBF16>(p, r, row_ok, grow, gcol0, packed, c_path(p, ep, gcol0), cc, ep);
          if (c + 1 < c_hi) c_fetch16(p, ep, c_path(p, ep, gcol0 + chunk), grow, gcol0 + chunk, lane, cc);
          epi_store_chunk<2>(p, packed, row_ok, grow, gcol0, grow - lane * p.maps.epi_row_step, stage_buf,
                             PairCfg::kEpiBufBytes, buf, carry, c == c_hi - 1, lane, ep);
        }
      }
    }
    if (p.d_tma && lane == 0) bulk_wait_all();
  }

  __syncthreads();
  cluster_sync();  // the pair's MMAs, remote arrivals and loads are all finished
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, PairCfg::kTmemCols);
  }
}

}  // namespace ttc
