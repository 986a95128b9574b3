// rlk_gemm.cuh -- the one tcgen05 tile engine behind every contraction of
// linear_logp, specialised by epilogue:
//
//   MODE_FWD  z = h W^T over the 256-column tiles of one 1024-column leaf; the
//             epilogue keeps per-row running max / sum-exp / target logit in
//             registers and writes one (m, s, zt) triple per (token, leaf)
//             ("Announcing RL-Kernel for vime", "Why the Fused Path Wins",
//             second reason: statistics maintained during tiled GEMM work).
//   MODE_DZ   the same z tiles, recomputed with the same K order; the epilogue
//             forms dz = g (onehot - exp(z - lse)) and writes it as bf16
//             (fourth reason: tiled logits / dlogits in a controlled workspace).
//   MODE_DH   dH = dz W    (K = vocab, ascending), bf16 or fp32 output.
//   MODE_DW   dW = dz^T h  (K = tokens, ascending), fp32 output.
//
// Kernel structure (one persistent CTA per SM, 192 threads):
//   warp 0     TMA producer: 4-stage shared-memory ring of 48 KiB stages
//              (A 128x64 + B 256x64 bf16, 128-byte swizzle)
//   warp 1     allocates 512 TMEM columns; one thread issues tcgen05.mma
//              (M=128, N=256, K=16; four per stage) into one of two fp32
//              accumulators, releasing stages and accumulators by tcgen05.commit
//   warps 2-5  epilogue: tcgen05.ld (thread = token row, lane quarter = warp % 4)
//              -> registers -> mode-specific math -> global memory
// Work items are assigned statically (item = blockIdx.x + i * gridDim.x), so
// numerics never depend on the grid: each output element is produced by one
// fixed instruction sequence regardless of T, batch composition or SM count.
#pragma once

#include "rlk_internal.h"
#include "rlk_ptx.cuh"

namespace rlk {

template <int MODE>
struct Operands {
  static constexpr bool A_MN = (MODE == MODE_DW);
  static constexpr bool B_MN = (MODE == MODE_DH || MODE == MODE_DW);
  static constexpr uint32_t IDESC = make_idesc_bf16(BM, BN, A_MN, B_MN);
};

// Number of 256-wide tiles in a work item.
template <int MODE>
__device__ __forceinline__ int item_tiles(const GemmArgs& a, int item) {
  if constexpr (MODE == MODE_FWD) {
    const int leaf_local = item / a.n_tt;
    const int col0 = (a.leaf0 + leaf_local) * LEAF;
    const int end = min(col0 + LEAF, a.V_true);
    return (end - col0 + BN - 1) / BN;
  } else {
    return 1;
  }
}

// Tile origin: m0 = first row of the A operand's M extent, n0 = first row of
// the B operand's N extent (fwd/dz: local W row; dH/dW: output column).
template <int MODE>
__device__ __forceinline__ void tile_origin(const GemmArgs& a, int item, int j, int& m0, int& n0) {
  if constexpr (MODE == MODE_FWD) {
    const int leaf_local = item / a.n_tt, tt = item % a.n_tt;
    m0 = tt * BM;
    n0 = (a.leaf0 + leaf_local) * LEAF + j * BN - a.vocab_start;
  } else if constexpr (MODE == MODE_DZ) {
    const int vt = item / a.n_tt, tt = item % a.n_tt;
    m0 = tt * BM;
    n0 = vt * BN;
  } else {
    const int mt = item / a.n_nt, nt = item % a.n_nt;
    m0 = mt * BM;
    n0 = nt * BN;
  }
}

// A wait that ignores the abort flag (used only to drain work already in flight).
__device__ __forceinline__ bool mbar_wait_timeout(uint64_t* bar, uint32_t parity) {
  const uint32_t a = smem_u32(bar);
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(a, parity)) {
    if (global_timer_ns() - t0 > kWaitLimitNs) return false;
  }
  return true;
}

// ---------------------------------------------------------------------------
// warp 0: TMA producer (one thread)
// ---------------------------------------------------------------------------
template <int MODE>
__device__ void producer_loop(const CUtensorMap* tmA, const CUtensorMap* tmB, const GemmArgs& a,
                              uint8_t* smem, uint64_t* full, uint64_t* empty,
                              volatile int* abort_flag) {
  uint32_t issued = 0;
  bool ok = true;
  for (int item = blockIdx.x; ok && item < a.n_items; item += gridDim.x) {
    const int ntiles = item_tiles<MODE>(a, item);
    for (int j = 0; ok && j < ntiles; ++j) {
      int m0, n0;
      tile_origin<MODE>(a, item, j, m0, n0);
      for (int kb = 0; kb < a.n_kb; ++kb) {
        const uint32_t s = issued % STAGES, ph = (issued / STAGES) & 1u;
        if (!mbar_wait_bounded(&empty[s], ph ^ 1u, abort_flag)) {
          ok = false;
          break;
        }
        uint8_t* sA = smem + s * STAGE_BYTES;
        uint8_t* sB = sA + A_STAGE_BYTES;
        mbar_arrive_expect_tx(&full[s], STAGE_BYTES);
        const int k0 = kb * BK;
        if constexpr (MODE == MODE_FWD || MODE == MODE_DZ) {
          tma_load_2d(sA, tmA, &full[s], k0, m0);  // h rows m0.., K-major box 64 x 128
          tma_load_2d(sB, tmB, &full[s], k0, n0);  // W rows n0.., K-major box 64 x 256
        } else if constexpr (MODE == MODE_DH) {
          tma_load_2d(sA, tmA, &full[s], k0, m0);  // dz rows m0.., K-major box 64 x 128
#pragma unroll
          for (int q = 0; q < BN / 64; ++q)        // W[k0.., n0+64q..] MN-major boxes 64 x 64
            tma_load_2d(sB + q * MN_ATOM_BYTES, tmB, &full[s], n0 + q * 64, k0);
        } else {
#pragma unroll
          for (int q = 0; q < BM / 64; ++q)        // dz[k0.., m0+64q..] MN-major boxes 64 x 64
            tma_load_2d(sA + q * MN_ATOM_BYTES, tmA, &full[s], m0 + q * 64, k0);
#pragma unroll
          for (int q = 0; q < BN / 64; ++q)        // h[k0.., n0+64q..] MN-major boxes 64 x 64
            tma_load_2d(sB + q * MN_ATOM_BYTES, tmB, &full[s], n0 + q * 64, k0);
        }
        ++issued;
      }
    }
  }
  if (ok) {
    // Tail: every stage must have been released by the MMA warp (all its
    // commits have landed) before the CTA may exit.
    for (uint32_t i = 0; i < STAGES; ++i) {
      const uint32_t it = issued + i;
      if (!mbar_wait_bounded(&empty[it % STAGES], ((it / STAGES) & 1u) ^ 1u, abort_flag)) break;
    }
  } else {
    // Abort: wait for the copies already in flight so no TMA write lands after exit.
    const uint32_t first = issued > STAGES ? issued - STAGES : 0;
    for (uint32_t it = first; it < issued; ++it)
      mbar_wait_timeout(&full[it % STAGES], (it / STAGES) & 1u);
  }
}

// ---------------------------------------------------------------------------
// warp 1: tcgen05.mma issuer (one thread)
// ---------------------------------------------------------------------------
template <int MODE>
__device__ void mma_loop(const GemmArgs& a, uint8_t* smem, uint64_t* full, uint64_t* empty,
                         uint64_t* acc_full, uint64_t* acc_empty, uint64_t* drain,
                         uint32_t tmem_base, volatile int* abort_flag) {
  using Ops = Operands<MODE>;
  uint32_t it = 0, tile = 0;
  bool ok = true;
  for (int item = blockIdx.x; ok && item < a.n_items; item += gridDim.x) {
    const int ntiles = item_tiles<MODE>(a, item);
    for (int j = 0; ok && j < ntiles; ++j) {
      const uint32_t buf = tile & 1u, use = tile >> 1;
      if (!mbar_wait_bounded(&acc_empty[buf], (use & 1u) ^ 1u, abort_flag)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + buf * BN;
      for (int kb = 0; kb < a.n_kb; ++kb, ++it) {
        const uint32_t s = it % STAGES, ph = (it / STAGES) & 1u;
        if (!mbar_wait_bounded(&full[s], ph, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t a_base = smem_u32(smem + s * STAGE_BYTES);
        const uint32_t b_base = a_base + A_STAGE_BYTES;
#pragma unroll
        for (int k = 0; k < BK / UMMA_K; ++k) {
          const uint64_t ad = Ops::A_MN ? make_smem_desc(a_base + k * 2048, MN_ATOM_BYTES, 1024)
                                        : make_smem_desc(a_base + k * 32, 16, 1024);
          const uint64_t bd = Ops::B_MN ? make_smem_desc(b_base + k * 2048, MN_ATOM_BYTES, 1024)
                                        : make_smem_desc(b_base + k * 32, 16, 1024);
          umma_bf16(d_tmem, ad, bd, Ops::IDESC, (kb | k) != 0 ? 1u : 0u);
        }
        umma_commit(&empty[s]);  // stage s is free once these MMAs have read it
      }
      if (!ok) break;
      umma_commit(&acc_full[buf]);  // accumulator complete
      ++tile;
    }
  }
  // Every issued MMA must have finished before TMEM is released.
  umma_commit(drain);
  mbar_wait_timeout(drain, 0);
}

// ---------------------------------------------------------------------------
// warps 2-5: epilogues (128 threads; thread = one accumulator row)
// ---------------------------------------------------------------------------

__device__ __forceinline__ float max64(const float (&v)[64]) {
  float m[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) m[i] = fmaxf(fmaxf(v[i], v[i + 16]), fmaxf(v[i + 32], v[i + 48]));
#pragma unroll
  for (int w = 8; w >= 1; w >>= 1)
#pragma unroll
    for (int i = 0; i < w; ++i) m[i] = fmaxf(m[i], m[i + w]);
  return m[0];
}

// Sum of e(v[i] - b) over 64 values in a fixed order: eight interleaved running
// sums (i mod 8), then a fixed pairwise combination.
__device__ __forceinline__ float sum_exp64(const float (&v)[64], float nb) {
  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = exp_shifted(v[i], nb);
#pragma unroll
  for (int i = 8; i < 64; ++i) acc[i & 7] = __fadd_rn(acc[i & 7], exp_shifted(v[i], nb));
  const float a01 = __fadd_rn(acc[0], acc[1]), a23 = __fadd_rn(acc[2], acc[3]);
  const float a45 = __fadd_rn(acc[4], acc[5]), a67 = __fadd_rn(acc[6], acc[7]);
  return __fadd_rn(__fadd_rn(a01, a23), __fadd_rn(a45, a67));
}

struct RowStats {
  float m, s, zt, nb;  // running max, sum of e(z - m), target logit, -rn(m log2 e)
};

// Online update of one row's statistics with one 64-column chunk (forward).
// `valid` = number of leading columns of the chunk below V_true (warp-uniform),
// `tl` = the target's column inside the chunk or outside [0, 64).
__device__ __forceinline__ void fwd_chunk(float (&v)[64], int valid, int tl, RowStats& st) {
  if (valid < 64) {
#pragma unroll
    for (int i = 0; i < 64; ++i)
      if (i >= valid) v[i] = neg_inf();
  }
  if (__any_sync(0xffffffffu, tl >= 0 && tl < 64)) {
#pragma unroll
    for (int i = 0; i < 64; ++i)
      if (i == tl) st.zt = v[i];
  }
  const float cm = max64(v);
  if (cm > st.m) {
    const float nb = neg_scaled(cm);
    st.s = __fmul_rn(st.s, exp_shifted(st.m, nb));
    st.m = cm;
    st.nb = nb;
  }
  st.s = __fadd_rn(st.s, sum_exp64(v, st.nb));
}

template <int MODE>
__device__ void epilogue_loop(const GemmArgs& a, uint64_t* acc_full, uint64_t* acc_empty,
                              uint32_t tmem_base, volatile int* abort_flag) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int quarter = warp & 3;  // TMEM lane quarter this warp may access
  const int row = quarter * 32 + lane;
  const uint32_t lane_base = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16);
  uint32_t tile = 0;
  bool ok = true;

  for (int item = blockIdx.x; ok && item < a.n_items; item += gridDim.x) {
    const int ntiles = item_tiles<MODE>(a, item);
    int m0, n0;
    tile_origin<MODE>(a, item, 0, m0, n0);

    // ---- per-item setup
    RowStats st{neg_inf(), 0.f, neg_inf(), 0.f};
    int64_t yt = -1;
    float g_t = 0.f, nl = 0.f;
    bool yvalid = false;
    const int t = m0 + row;  // token row (fwd, dz, dH) or vocab row (dW)
    if constexpr (MODE == MODE_FWD) {
      if (t < a.T) yt = a.y[t];
    } else if constexpr (MODE == MODE_DZ) {
      if (t < a.T) {
        yt = a.y[t];
        g_t = a.g[t];
        nl = neg_scaled(a.lse[t]);
        yvalid = yt >= 0 && yt < a.V_true;
        if (!yvalid && n0 == 0 && a.err_flag) atomicOr(a.err_flag, 1);
      }
    }

    for (int j = 0; j < ntiles; ++j) {
      const uint32_t buf = tile & 1u, use = tile >> 1;
      bool got = mbar_wait_bounded(&acc_full[buf], use & 1u, abort_flag);
      got = __all_sync(0xffffffffu, got);
      if (!got) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t taddr = lane_base + buf * BN;

      if constexpr (MODE == MODE_FWD) {
        const int c0 = n0 + a.vocab_start + j * BN;  // global column of the tile's first column
        const int vcols = min(BN, a.V_true - c0);
        const int tl = (yt >= c0 && yt < static_cast<int64_t>(c0) + vcols) ? static_cast<int>(yt - c0) : -1;
#pragma unroll 1
        for (int ch = 0; ch < BN; ch += 64) {
          float v[64];
          tmem_ld64(taddr + ch, v);
          fwd_chunk(v, vcols - ch, tl - ch, st);
        }
      } else if constexpr (MODE == MODE_DZ) {
        const int gc0 = a.vocab_start + n0;
        const int vcols = max(0, min(min(BN, a.V_true - gc0), a.V_local - n0));
        const int tl = (yvalid && yt >= gc0 && yt < static_cast<int64_t>(gc0) + vcols)
                           ? static_cast<int>(yt - gc0) : -1;
        uint16_t* dst = a.dz + static_cast<size_t>(t) * a.dz_ld + n0;
        const float ng = -g_t;
#pragma unroll 1
        for (int ch = 0; ch < BN; ch += 64) {
          float v[64];
          tmem_ld64(taddr + ch, v);
          const int tli = tl - ch;
          float d_target = 0.f;
          const bool any_target = __any_sync(0xffffffffu, tli >= 0 && tli < 64);
          if (any_target) {
#pragma unroll
            for (int i = 0; i < 64; ++i)
              if (i == tli) d_target = __fmul_rn(g_t, __fsub_rn(1.f, exp_shifted(v[i], nl)));
          }
#pragma unroll
          for (int i = 0; i < 64; ++i) v[i] = __fmul_rn(ng, exp_shifted(v[i], nl));
          if (any_target) {
#pragma unroll
            for (int i = 0; i < 64; ++i)
              if (i == tli) v[i] = d_target;
          }
          const int valid = yvalid ? vcols - ch : 0;
          if (valid < 64) {
#pragma unroll
            for (int i = 0; i < 64; ++i)
              if (i >= valid) v[i] = 0.f;
          }
          if (t < a.T) {
            uint4* p = reinterpret_cast<uint4*>(dst + ch);
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              uint4 w;
              w.x = pack_bf16x2(v[8 * q + 0], v[8 * q + 1]);
              w.y = pack_bf16x2(v[8 * q + 2], v[8 * q + 3]);
              w.z = pack_bf16x2(v[8 * q + 4], v[8 * q + 5]);
              w.w = pack_bf16x2(v[8 * q + 6], v[8 * q + 7]);
              p[q] = w;
            }
          }
        }
      } else {
        // dH / dW: plain stores of the fp32 accumulator (bf16 for dH unless partial)
        const bool row_ok = t < a.out_rows;
#pragma unroll 1
        for (int ch = 0; ch < BN; ch += 64) {
          float v[64];
          tmem_ld64(taddr + ch, v);
          const int col = n0 + ch;
          if (row_ok && col < a.out_cols) {
            if (a.out_f32) {
              float* p = static_cast<float*>(a.out) + static_cast<size_t>(t) * a.out_ld + col;
#pragma unroll
              for (int q = 0; q < 16; ++q)
                if (col + 4 * q < a.out_cols)
                  *reinterpret_cast<float4*>(p + 4 * q) =
                      make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
            } else {
              uint16_t* p = static_cast<uint16_t*>(a.out) + static_cast<size_t>(t) * a.out_ld + col;
#pragma unroll
              for (int q = 0; q < 8; ++q)
                if (col + 8 * q < a.out_cols) {
                  uint4 w;
                  w.x = pack_bf16x2(v[8 * q + 0], v[8 * q + 1]);
                  w.y = pack_bf16x2(v[8 * q + 2], v[8 * q + 3]);
                  w.z = pack_bf16x2(v[8 * q + 4], v[8 * q + 5]);
                  w.w = pack_bf16x2(v[8 * q + 6], v[8 * q + 7]);
                  *reinterpret_cast<uint4*>(p + 8 * q) = w;
                }
            }
          }
        }
      }

      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[buf]);
      ++tile;
    }

    if constexpr (MODE == MODE_FWD) {
      if (ok && t < a.T) {
        const int leaf_local = item / a.n_tt;
        const size_t o = static_cast<size_t>(leaf_local) * a.T + t;
        a.ws_m[o] = st.m;
        a.ws_s[o] = st.s;
        a.ws_zt[o] = st.zt;
      }
    }
  }
}

// ---------------------------------------------------------------------------
// the kernel
// ---------------------------------------------------------------------------
template <int MODE>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                const GemmArgs a) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
  uint8_t* smem = smem_raw + pad;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + STAGES * STAGE_BYTES);
  uint64_t* empty = full + STAGES;
  uint64_t* acc_full = empty + STAGES;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* drain = acc_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], 4);  // one arrival per epilogue warp
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) producer_loop<MODE>(&tmA, &tmB, a, smem, full, empty, abort_flag);
  } else if (warp == 1) {
    if (lane == 0)
      mma_loop<MODE>(a, smem, full, empty, acc_full, acc_empty, drain, tmem_base, abort_flag);
  } else {
    epilogue_loop<MODE>(a, acc_full, acc_empty, tmem_base, abort_flag);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
  if (threadIdx.x == 0 && *abort_flag && a.err_flag) atomicOr(a.err_flag, 2);
}

template <int MODE>
cudaError_t launch_gemm(const CUtensorMap& tmA, const CUtensorMap& tmB, const GemmArgs& a,
                        int grid, cudaStream_t stream) {
  auto kernel = gemm_kernel<MODE>;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
  if (e != cudaSuccess) return e;
  kernel<<<grid, NUM_THREADS, SMEM_BYTES, stream>>>(tmA, tmB, a);
  return cudaGetLastError();
}

}  // namespace rlk
