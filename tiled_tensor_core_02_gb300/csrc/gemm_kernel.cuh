// Persistent, warp-specialized tiled GEMM for sm_103a:
//   D = act(alpha * A * B + beta * C + bias), fp16/bf16 operands, fp32 accumulation.
//
// Structure (the CUTLASS tutorial's "Collective Mainloop + Collective Epilogue"
// split on hpc.payai.win/cutlass, section 3, rebuilt for tcgen05/TMEM/TMA):
//   warp 0      producer: one thread issues TMA loads of the A and B tiles of
//               each k-block into a STAGES-deep ring of 128-byte-swizzled
//               shared-memory slots (full/empty mbarrier pair per slot);
//   warp 1      tensor-core issuer: allocates TMEM, one thread issues
//               tcgen05.mma (M=128, N=BN, K=16) into one of two TMEM
//               accumulators and commits completion back to the ring;
//   warps 2..5  epilogue: tcgen05.ld of the accumulator (each warp owns the
//               32 TMEM lanes = tile rows its warp index selects), then
//               alpha / beta*C / bias / activation in fp32, round to the
//               output type, stage in swizzled shared memory and TMA-store.
// The two TMEM accumulators let the epilogue of tile i overlap the mainloop
// of tile i+1.  Tiles are walked persistently (tile = blockIdx.x + j*gridDim.x)
// in grouped order: group_m consecutive M-blocks share each N-block, so a
// wave of CTAs reuses the same A and B panels from L2.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "ptx.cuh"

namespace ttc {

constexpr int kBM = 128;          // UMMA M (rows of the CTA tile = TMEM lanes)
constexpr int kBK = 64;           // k-block: 64 16-bit elements = one 128-byte swizzle row
constexpr int kUmmaK = 16;        // K of one tcgen05.mma for 16-bit inputs
constexpr int kEpiWarps = 4;
constexpr int kThreads = 64 + 32 * kEpiWarps;
constexpr int kEpiCols = 32;      // columns per epilogue chunk
constexpr int kEpiBufBytes = 32 * kEpiCols * 2;  // 32 rows x 64 bytes
constexpr int kABytes = kBM * kBK * 2;           // 16 KiB

enum ActKind : int { kActNone = 0, kActRelu = 1, kActGelu = 2 };

struct GemmParams {
  CUtensorMap tmA;
  CUtensorMap tmB;
  CUtensorMap tmD;
  int M, N, K;
  int num_m_blocks, num_n_blocks, num_k_blocks, num_tiles, group_m;
  int a_mn, b_mn;  // operand stored MN-major (A column-major / B row-major)
  float alpha, beta;
  const void* C;
  int64_t ldc;
  void* D;
  int64_t ldd;
  const float* bias;
  int act;
  int d_tma;  // 1: D written by TMA store; 0: predicated st.global
  uint32_t* err;
  uint64_t timeout_ns;
  int inject_stall;
};

template <int BN>
struct TileCfg {
  static constexpr int kBBytes = BN * kBK * 2;
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kEpiBytes = kEpiWarps * 2 * kEpiBufBytes;
  static constexpr int kBarBytes = 256;
  static constexpr int kSmemLimit = 227 * 1024;  // opt-in dynamic shared memory per block
  static constexpr int kStageBudget = kSmemLimit - 1024 - kBarBytes - kEpiBytes;
  static constexpr int kStages = kStageBudget / kStageBytes > 8 ? 8 : kStageBudget / kStageBytes;
  static constexpr int kTmemCols = 2 * BN < 32 ? 32 : 2 * BN;
  static constexpr int kSmemBytes = 1024 /*align slack*/ + kStages * kStageBytes + kEpiBytes + kBarBytes;
  static_assert(BN % 16 == 0 && BN >= 16 && BN <= 256, "UMMA N for M=128");
  static_assert(kStages >= 2, "pipeline depth");
  static_assert(kSmemBytes <= kSmemLimit, "shared memory budget");
  static_assert((2 * BN & (2 * BN - 1)) == 0, "TMEM allocation is a power of two");
};

__device__ __forceinline__ void tile_coords(int t, const GemmParams& p, int& mb, int& nb) {
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
__device__ __forceinline__ float load_elem16(const void* base, int64_t idx) {
  const uint16_t h = reinterpret_cast<const uint16_t*>(base)[idx];
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

template <int BN, bool BF16>
__global__ void __launch_bounds__(kThreads, 1) gemm_f16_kernel(const __grid_constant__ GemmParams p) {
  using Cfg = TileCfg<BN>;
  constexpr int S = Cfg::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = sA + S * kABytes;
  uint8_t* sEpi = sB + S * Cfg::kBBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sEpi + Cfg::kEpiBytes);
  uint64_t* full = bars;
  uint64_t* empty = bars + S;
  uint64_t* tmem_full = bars + 2 * S;
  uint64_t* tmem_empty = bars + 2 * S + 2;
  uint64_t* stall_bar = bars + 2 * S + 4;
  uint64_t* drain_bar = bars + 2 * S + 5;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * S + 6);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const WaitCtx wc{p.err, p.timeout_ns};

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tmem_full[a], 1);
      mbar_init(&tmem_empty[a], kEpiWarps);
    }
    mbar_init(stall_bar, 1);
    mbar_init(drain_bar, 1);
    fence_barrier_init();
    prefetch_tmap(&p.tmA);
    prefetch_tmap(&p.tmB);
    if (p.d_tma) prefetch_tmap(&p.tmD);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, Cfg::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      const uint64_t pol = policy_evict_last();
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued_mask = 0, issued_parity = 0;
      bool ok = true;
      for (int t = blockIdx.x; ok && t < p.num_tiles; t += gridDim.x) {
        int mb, nb;
        tile_coords(t, p, mb, nb);
        const int m0 = mb * kBM, n0 = nb * BN;
        for (int kb = 0; kb < p.num_k_blocks; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1u, wc)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&full[stage], Cfg::kStageBytes);
          uint8_t* a = sA + stage * kABytes;
          uint8_t* b = sB + stage * Cfg::kBBytes;
          const int k0 = kb * kBK;
          if (!p.a_mn) {
            tma_load_2d(a, &p.tmA, k0, m0, &full[stage], pol);
          } else {
            tma_load_2d(a, &p.tmA, m0, k0, &full[stage], pol);
            tma_load_2d(a + kABytes / 2, &p.tmA, m0 + 64, k0, &full[stage], pol);
          }
          if (!p.b_mn) {
            tma_load_2d(b, &p.tmB, k0, n0, &full[stage], pol);
          } else {
#pragma unroll
            for (int h = 0; h < BN / 64; ++h) tma_load_2d(b + h * 8192, &p.tmB, n0 + 64 * h, k0, &full[stage], pol);
          }
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
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t idesc = idesc_f16(BF16, p.a_mn != 0, p.b_mn != 0, kBM, BN);
      bool ok = true;
      bool any_mma = false;
      if (p.inject_stall) ok = mbar_wait(stall_bar, 0, wc);  // nothing arrives here
      int stage = 0;
      uint32_t phase = 0;
      int it = 0;
      const uint32_t a_lbo = p.a_mn ? 8192u : 16u, b_lbo = p.b_mn ? 8192u : 16u;
      const uint32_t a_kstep = p.a_mn ? 2048u : 32u, b_kstep = p.b_mn ? 2048u : 32u;
      for (int t = blockIdx.x; ok && t < p.num_tiles; t += gridDim.x, ++it) {
        const int acc = it & 1;
        const uint32_t acc_phase = (it >> 1) & 1;
        if (!mbar_wait(&tmem_empty[acc], acc_phase ^ 1u, wc)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * BN;
        for (int kb = 0; kb < p.num_k_blocks; ++kb) {
          if (!mbar_wait(&full[stage], phase, wc)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_addr = smem_u32(sA + stage * kABytes);
          const uint32_t b_addr = smem_u32(sB + stage * Cfg::kBBytes);
#pragma unroll
          for (int k = 0; k < kBK / kUmmaK; ++k) {
            const uint64_t ad = smem_desc_sw128(a_addr + k * a_kstep, a_lbo, 1024);
            const uint64_t bd = smem_desc_sw128(b_addr + k * b_kstep, b_lbo, 1024);
            mma_f16(d_tmem, ad, bd, idesc, (kb | k) != 0);
          }
          any_mma = true;
          mma_commit(&empty[stage]);
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        if (p.num_k_blocks == 0)
          mbar_arrive(&tmem_full[acc]);
        else
          mma_commit(&tmem_full[acc]);
      }
      if (any_mma) {
        // Every MMA must have finished with TMEM before it is freed.
        mma_commit(drain_bar);
        drain_wait(drain_bar, 0, 100000000ull);
      }
    }
  } else {
    // ---------------------------------------------------------------- epilogue
    const int ew = warp - 2;      // epilogue warp 0..3 (owns a staging area)
    const int q = warp & 3;       // TMEM lane quarter this warp may access
    const int row_in_tile = q * 32 + lane;
    uint8_t* stage_buf = sEpi + ew * 2 * kEpiBufBytes;
    int buf = 0;
    int it = 0;
    const bool has_k = p.num_k_blocks > 0;
    for (int t = blockIdx.x; t < p.num_tiles; t += gridDim.x, ++it) {
      const int acc = it & 1;
      const uint32_t acc_phase = (it >> 1) & 1;
      if (!mbar_wait(&tmem_full[acc], acc_phase, wc)) break;
      tc_fence_after();
      int mb, nb;
      tile_coords(t, p, mb, nb);
      const int m0 = mb * kBM, n0 = nb * BN;
      const int grow = m0 + row_in_tile;
      const bool row_ok = grow < p.M;
#pragma unroll 1
      for (int c = 0; c < BN / kEpiCols; ++c) {
        uint32_t r[32];
        if (has_k) {
          tmem_ld_32x32b_x32(tmem_base + ((uint32_t)(q * 32) << 16) + acc * BN + c * kEpiCols, r);
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
        const int gcol0 = n0 + c * kEpiCols;
        float v[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = p.alpha * __uint_as_float(r[j]);
        if (p.beta != 0.0f && row_ok) {
          const int64_t rbase = (int64_t)grow * p.ldc;
          const bool vec = ((p.ldc & 7) == 0) && ((reinterpret_cast<uintptr_t>(p.C) & 15) == 0) &&
                           (gcol0 + 32 <= p.N);
          if (vec) {
            const uint4* src = reinterpret_cast<const uint4*>(reinterpret_cast<const uint16_t*>(p.C) + rbase + gcol0);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const uint4 w = __ldg(src + u);
              const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
              for (int h = 0; h < 4; ++h) {
                float lo, hi;
                if constexpr (BF16) {
                  lo = __bfloat162float(__ushort_as_bfloat16((uint16_t)(ws[h] & 0xFFFFu)));
                  hi = __bfloat162float(__ushort_as_bfloat16((uint16_t)(ws[h] >> 16)));
                } else {
                  lo = __half2float(__ushort_as_half((uint16_t)(ws[h] & 0xFFFFu)));
                  hi = __half2float(__ushort_as_half((uint16_t)(ws[h] >> 16)));
                }
                v[u * 8 + 2 * h] = fmaf(p.beta, lo, v[u * 8 + 2 * h]);
                v[u * 8 + 2 * h + 1] = fmaf(p.beta, hi, v[u * 8 + 2 * h + 1]);
              }
            }
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (gcol0 + j < p.N) v[j] = fmaf(p.beta, load_elem16<BF16>(p.C, rbase + gcol0 + j), v[j]);
          }
        }
        if (p.bias != nullptr) {
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (gcol0 + j < p.N) v[j] += __ldg(p.bias + gcol0 + j);
        }
        if (p.act != kActNone) {
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] = apply_act(p.act, v[j]);
        }
        uint32_t packed[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) packed[j] = pack2<BF16>(v[2 * j], v[2 * j + 1]);

        if (p.d_tma) {
          // staging buffer `buf` was last used two chunks ago; its store must
          // have finished reading shared memory
          if (lane == 0) bulk_wait_read<1>();
          __syncwarp();
          uint8_t* sb = stage_buf + buf * kEpiBufBytes;
          // 64-byte rows, 64-byte swizzle: 16-byte chunk index ^= (row >> 1) & 3
          const uint32_t xr = (uint32_t)(lane >> 1) & 3u;
#pragma unroll
          for (int ch = 0; ch < 4; ++ch) {
            uint4 w = make_uint4(packed[4 * ch], packed[4 * ch + 1], packed[4 * ch + 2], packed[4 * ch + 3]);
            *reinterpret_cast<uint4*>(sb + lane * 64 + ((ch ^ xr) << 4)) = w;
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_2d(&p.tmD, gcol0, m0 + q * 32, sb);
            bulk_commit();
          }
          buf ^= 1;
        } else if (row_ok) {
          uint16_t* dst = reinterpret_cast<uint16_t*>(p.D) + (int64_t)grow * p.ldd + gcol0;
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            if (gcol0 + j < p.N) {
              const uint32_t h = (packed[j >> 1] >> ((j & 1) * 16)) & 0xFFFFu;
              dst[j] = (uint16_t)h;
            }
          }
        }
      }
    }
    if (p.d_tma && lane == 0) bulk_wait_all();
  }

  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, Cfg::kTmemCols);
  }
}

}  // namespace ttc
