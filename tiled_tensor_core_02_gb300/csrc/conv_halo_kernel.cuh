// Implicit-GEMM convolution with unit stride, built from halo tiles: the
// CTA-pair tcgen05 kernel of gemm2sm_kernel.cuh with a different A operand.
//
// Output positions are numbered along rows of `wp` = Q + (S - 1) dil_w
// positions (the Q outputs of an output row, then S - 1 positions that are
// computed and dropped).  In that numbering the input pixel that filter tap
// (r, s) multiplies with output position L sits at L + r dil_h wp + s dil_w of
// the zero-padded input, for every tap.  So one 4-D tiled TMA box per 64-channel
// block (`halo_rows` padded input rows of wp pixels x 64 channels, zeros
// outside the image) holds the A operand of all R x S taps: tap (r, s) is the
// 128 rows starting r dil_h wp + s dil_w rows into the box.  The im2col
// formulation loads every input pixel R x S times per channel block; this one
// loads it about halo_rows x wp / 128 times.
//
// A CTA tile is 128 consecutive positions of one image; a pair computes the
// same tile of two images (2u and 2u + 1), so both CTAs place their halo at the
// same shared-memory offsets and one MMA descriptor serves both halves.  An odd
// last image pairs with an image past the end, whose box reads zeros and whose
// rows are not stored.
//
// Filter stages hold kHaloKPS taps (a block's 9 taps as 2, 2, 2, 2, 1 for a
// 3 x 3 filter, never spanning two halos), so one barrier round trip covers 8
// MMAs.  The pairs walk work units: whole tiles, then, for a last partial
// wave, half tiles of BN / 2 output channels (MMAs with N = BN / 2; each CTA
// uses the first rows of its usual filter box).
//
// Synchronisation, in addition to the pair kernel's (full/empty ring for the
// filter operand, tmem_full/tmem_empty for the two accumulators):
//   hfull[h]   even CTA only; its producer arms it with both CTAs' halo bytes.
//   hempty[h]  both CTAs; the MMA commit after a channel block's last tap.
// Every wait is bounded; on an error the CTA drains its loads and MMAs.
#pragma once
#include "conv_halo.cuh"
#include "gemm2sm_kernel.cuh"

namespace ttc {

struct HaloTile {
  int nb;   // output-channel block
  int j;    // position tile inside the image
  int img;  // this CTA's image
};

// Tile of work unit u (see ConvHaloParams::tail_from); n_off and half give the
// unit's first output channel inside the tile and whether it is a half.
__device__ __forceinline__ HaloTile halo_tile(const ConvHaloParams& hp, int u, uint32_t rank, int half_cols,
                                              int& n_off, bool& half) {
  half = u >= hp.tail_from;
  int t = u;
  n_off = 0;
  if (half) {
    t = hp.tail_from + ((u - hp.tail_from) >> 1);
    n_off = ((u - hp.tail_from) & 1) * half_cols;
  }
  HaloTile h;
  h.nb = t % hp.n_blocks;
  const int rest = t / hp.n_blocks;
  h.j = rest % hp.tiles_per_img;
  h.img = 2 * (rest / hp.tiles_per_img) + (int)rank;
  return h;
}

// Output row index of position `pos` of image `img`, or -1 for a dropped one.
__device__ __forceinline__ int halo_out_row(const ConvHaloParams& hp, int img, int pos) {
  const int op = pos / hp.wp;
  const int oq = pos - op * hp.wp;
  if (img >= hp.n_img || op >= hp.p || oq >= hp.q) return -1;
  return (img * hp.p + op) * hp.q + oq;
}

// Writes one 32-column chunk of the warp's 32 positions: each thread stages
// its row's 64 bytes (16-byte words XOR-swizzled by row pair, so the writes
// and the reads are free of bank conflicts), then each store instruction
// writes 8 rows x 64 bytes.  out_row[it] is the output row (or -1: dropped)
// of the position this thread stores in step it, row it * 8 + lane / 4 of the
// warp's 32.
__device__ __forceinline__ void halo_store_chunk(const ConvHaloParams& hp, const uint32_t (&packed)[16],
                                                 uint8_t* sbuf, int lane, const int (&out_row)[4], int gcol0) {
#pragma unroll
  for (int ch = 0; ch < 4; ++ch)
    *reinterpret_cast<uint4*>(sbuf + lane * 64 + ((ch ^ ((lane >> 1) & 3)) * 16)) =
        make_uint4(packed[4 * ch], packed[4 * ch + 1], packed[4 * ch + 2], packed[4 * ch + 3]);
  __syncwarp();
  const int ch = lane & 3;
#pragma unroll
  for (int it = 0; it < 4; ++it) {
    const int r = it * 8 + (lane >> 2);
    const int m = out_row[it];
    if (m >= 0 && gcol0 + ch * 8 < hp.g.N) {
      const uint4 v = *reinterpret_cast<const uint4*>(sbuf + r * 64 + ((ch ^ ((r >> 1) & 3)) * 16));
      *reinterpret_cast<uint4*>(static_cast<uint16_t*>(hp.g.D) + (int64_t)m * hp.g.ldd + gcol0 + ch * 8) = v;
    }
  }
  __syncwarp();
}

template <int BN, bool kBF16>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kHaloThreads, 1)
    conv_halo_kernel(const __grid_constant__ ConvHaloParams hp) {
  const GemmParams& p = hp.g;
  constexpr int kBHalf = BN / 2;
  constexpr int kBHalfBytes = kBHalf * kBK * 2;
  constexpr int kTmemCols = 2 * BN > 256 ? 512 : 256;
  const int S = hp.stages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sH = smem;  // two halo buffers of hp.halo_bytes
  uint8_t* sB = sH + 2 * hp.halo_bytes;
  uint8_t* sEpi = sB + S * kHaloKPS * kBHalfBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sEpi + kHaloEpiBytes);
  uint64_t* full = bars;
  uint64_t* empty = bars + kHaloMaxStages;
  uint64_t* hfull = bars + 2 * kHaloMaxStages;
  uint64_t* hempty = hfull + 2;
  uint64_t* tmem_full = hempty + 2;
  uint64_t* tmem_empty = tmem_full + 2;
  uint64_t* stall_bar = tmem_empty + 2;
  uint64_t* drain_bar = stall_bar + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain_bar + 1);
  static_assert((2 * kHaloMaxStages + 10) * 8 + 4 <= kHaloBarBytes, "barrier area");

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int pair = blockIdx.x >> 1;
  const int num_pairs = gridDim.x >> 1;
  const WaitCtx wc{p.err, p.timeout_ns};

  if (warp == 0) {
    for (int s = lane; s < S; s += 32) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    if (lane < 2) {
      mbar_init(&hfull[lane], 1);
      mbar_init(&hempty[lane], 1);
      mbar_init(&tmem_full[lane], 1);
      mbar_init(&tmem_empty[lane], 2 * kEpiWarps);
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
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_slot, kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // global memory only after the previous grid on the stream (see ptx.cuh)
  grid_dependency_wait();
  grid_dependents_launch();

  if (warp == 0) {
    // ---------------------------------------------------------------- producer (both CTAs)
    if (lane == 0) {
      const uint64_t pol_x = policy_evict_last();  // every tap of R x S channel blocks re-reads it
      const uint64_t pol_w = policy_evict_last();  // filters: re-read by every tile
      int stage = 0, hb = 0;
      uint32_t phase = 0, hphase = 0;
      uint32_t armed_mask = 0, armed_parity = 0, harmed_mask = 0, harmed_parity = 0;
      bool ok = true;
      for (int u = pair; ok && u < hp.num_units; u += num_pairs) {
        int n_off;
        bool half;
        const HaloTile ht = halo_tile(hp, u, rank, BN / 2, n_off, half);
        const int l0 = ht.j * kBM;
        const int hrow = l0 / hp.wp;  // first output row of the tile
        // this CTA's filters: a half unit uses the first kBHalf / 2 rows of the usual box
        const int n0 = ht.nb * BN + n_off + (int)rank * (half ? kBHalf / 2 : kBHalf);
        for (int cb = 0; ok && cb < hp.cblk; ++cb) {
          if (!mbar_wait(&hempty[hb], hphase ^ 1u, wc)) {
            ok = false;
            break;
          }
          if (leader) {
            mbar_arrive_expect_tx(&hfull[hb], 2 * hp.halo_tx);
            harmed_mask |= 1u << hb;
            harmed_parity = (harmed_parity & ~(1u << hb)) | (hphase << hb);
          }
          tma_load_4d_pair(sH + hb * hp.halo_bytes, &p.tmA, cb * kBK, -hp.pw, hrow - hp.ph, ht.img,
                           mapa_shared(smem_u32(&hfull[hb]), 0), pol_x);
          if (++hb == 2) {
            hb = 0;
            hphase ^= 1u;
          }
          // the block's taps, kHaloKPS per stage (the last stage may hold fewer)
          for (int t0 = 0; t0 < hp.taps; t0 += kHaloKPS) {
            const int nkb = min(kHaloKPS, hp.taps - t0);
            if (!mbar_wait(&empty[stage], phase ^ 1u, wc)) {
              ok = false;
              break;
            }
            if (leader) {
              mbar_arrive_expect_tx(&full[stage], 2 * nkb * kBHalfBytes);
              armed_mask |= 1u << stage;
              armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
            }
            for (int j = 0; j < nkb; ++j)
              tma_load_3d_pair(sB + (stage * kHaloKPS + j) * kBHalfBytes, &p.tmB, (t0 + j) * hp.c + cb * kBK, n0, 0,
                               mapa_shared(smem_u32(&full[stage]), 0), pol_w);
            if (++stage == S) {
              stage = 0;
              phase ^= 1u;
            }
          }
        }
      }
      if (!ok && leader) {
        // every box this CTA armed for completes once both CTAs' loads have landed
        for (int s = 0; s < S; ++s)
          if (armed_mask & (1u << s)) drain_wait(&full[s], (armed_parity >> s) & 1u, 100000000ull);
        for (int h = 0; h < 2; ++h)
          if (harmed_mask & (1u << h)) drain_wait(&hfull[h], (harmed_parity >> h) & 1u, 100000000ull);
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer (even CTA)
    if (leader && lane == 0) {
      const uint32_t idesc_full = idesc_f16(kBF16, false, false, 2 * kBM, BN);
      const uint32_t idesc_half = idesc_f16(kBF16, false, false, 2 * kBM, BN / 2);
      // descriptors are built once and stepped: the start address is a 14-bit
      // field at bit 0 (address >> 4) that no shared-memory offset overflows,
      // so +2 is one 16-deep k-step (32 bytes), +8 one 128-byte row
      const uint64_t desc0 = smem_desc_sw128(0u, 16, 1024);
      const uint64_t b_desc0 = desc0 + (smem_u32(sB) >> 4);
      const uint64_t a_tap_step = (uint64_t)hp.dw * 8u;
      const uint64_t a_row_step = (uint64_t)(hp.row_step - hp.s * hp.dw) * 8u;
      bool ok = true;
      bool any_mma = false;
      if (p.inject_stall) ok = mbar_wait(stall_bar, 0, wc);  // nothing arrives here
      int stage = 0, hb = 0;
      uint32_t phase = 0, hphase = 0;
      int it = 0;
      for (int u = pair; ok && u < hp.num_units; u += num_pairs, ++it) {
        const int acc = it & 1;
        if (!mbar_wait_cluster(&tmem_empty[acc], ((it >> 1) & 1) ^ 1u, wc)) {
          ok = false;
          break;
        }
        tc_fence_after();
        int n_off;
        bool half;
        const HaloTile ht = halo_tile(hp, u, rank, BN / 2, n_off, half);
        const uint32_t idesc = half ? idesc_half : idesc_full;
        const int l0 = ht.j * kBM;
        const int off = l0 - (l0 / hp.wp) * hp.wp;  // the tile's first position inside its halo row
        const uint32_t d_tmem = tmem_base + acc * BN;
        for (int cb = 0; ok && cb < hp.cblk; ++cb) {
          if (!mbar_wait(&hfull[hb], hphase, wc)) {
            ok = false;
            break;
          }
          tc_fence_after();
          // tap (r, s) starts r row_step + s dw rows past the tile's first position
          uint64_t ad = desc0 + ((smem_u32(sH + hb * hp.halo_bytes) + (uint32_t)off * 128u) >> 4);
          int fs = 0;
          for (int t0 = 0; t0 < hp.taps; t0 += kHaloKPS) {
            const int nkb = min(kHaloKPS, hp.taps - t0);
            if (!mbar_wait(&full[stage], phase, wc)) {
              ok = false;
              break;
            }
            tc_fence_after();
#pragma unroll
            for (int j = 0; j < kHaloKPS; ++j) {
              if (j < nkb) {
                const uint64_t bd = b_desc0 + (uint32_t)(stage * kHaloKPS + j) * (kBHalfBytes >> 4);
                mma_f16_pair(d_tmem, ad, bd, idesc, (cb | t0 | j) != 0);
#pragma unroll
                for (int k = 1; k < kBK / kUmmaK; ++k) mma_f16_pair(d_tmem, ad + 2 * k, bd + 2 * k, idesc, 1u);
                ad += a_tap_step;
                if (++fs == hp.s) {
                  fs = 0;
                  ad += a_row_step;
                }
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
          mma_commit_pair(&hempty[hb], 0x3);  // every tap of this block has read the halo
          if (++hb == 2) {
            hb = 0;
            hphase ^= 1u;
          }
        }
        if (!ok) break;
        mma_commit_pair(&tmem_full[acc], 0x3);
      }
      if (any_mma) {
        mma_commit_pair(drain_bar, 0x1);
        drain_wait(drain_bar, 0, 100000000ull);
      }
    }
  } else {
    // ---------------------------------------------------------------- epilogue (both CTAs)
    const int q = warp & 3;
    uint8_t* sbuf = sEpi + (warp - 2) * kHaloEpiBufBytes;
    int it = 0;
    const uint32_t lane_base = (uint32_t)(q * 32) << 16;
    for (int u = pair; u < hp.num_units; u += num_pairs, ++it) {
      const int acc = it & 1;
      int n_off;
      bool half;
      const HaloTile ht = halo_tile(hp, u, rank, BN / 2, n_off, half);
      const int pos0 = ht.j * kBM + q * 32;  // the warp's first position
      const int m = halo_out_row(hp, ht.img, pos0 + lane);
      const bool row_ok = m >= 0;
      int out_row[4];
#pragma unroll
      for (int s4 = 0; s4 < 4; ++s4) out_row[s4] = halo_out_row(hp, ht.img, pos0 + s4 * 8 + (lane >> 2));
      const int grow = row_ok ? m : p.M;  // past the end: C reads nothing for it
      const int n0 = ht.nb * BN + n_off;
      const int chunks = max(0, min(half ? BN / 2 : BN, p.N - n0)) / kEpiCols;
      const EpiPtrs ep = epi_ptrs(p, 0, 2);
      const int cpath = p.beta != 0.0f ? kCVec : kCNone;
      CChunk16 cc;
      c_fetch16(p, ep, cpath, grow, n0, lane, cc);
      if (!mbar_wait(&tmem_full[acc], (it >> 1) & 1, wc)) break;
      tc_fence_after();
      if (chunks == 0) {
        // nothing of this unit is stored: release the accumulator at once
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster_relaxed(mapa_shared(smem_u32(&tmem_empty[acc]), 0));
        continue;
      }
#pragma unroll 1
      for (int c = 0; c < chunks; ++c) {
        const int gcol0 = n0 + c * kEpiCols;
        uint32_t r[32];
        tmem_ld_32x32b_x32(tmem_base + lane_base + acc * BN + c * kEpiCols, r);
        tmem_ld_wait();
        if (c == chunks - 1) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive_cluster_relaxed(mapa_shared(smem_u32(&tmem_empty[acc]), 0));
        }
        uint32_t packed[16];
        epi_f16_values<kBF16>(p, r, row_ok, grow, gcol0, packed, cpath, cc, ep);
        if (c + 1 < chunks) c_fetch16(p, ep, cpath, grow, gcol0 + kEpiCols, lane, cc);
        halo_store_chunk(hp, packed, sbuf, lane, out_row, gcol0);
      }
    }
  }

  __syncthreads();
  cluster_sync();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, kTmemCols);
  }
}

}  // namespace ttc
