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
//   MODE_FWD8 / MODE_DZ8  MODE_FWD / MODE_DZ on E4M3 operands with one power-of-two
//             scale per row: the accumulator of hq Wq^T is multiplied by
//             h_scale[t] * W_scale[v] before the same epilogue (an FP8 LM head
//             whose training forward re-quantizes its weights every step; AREX
//             feed article on vLLM's bitwise-consistent RL training, section
//             "对齐的代价：逐算子拆解").
//
// Kernel structure: clusters of two CTAs (one per SM, persistent) compute
// 256 x 256 tiles with tcgen05 cta_group::2. Per CTA, 192 threads:
//   warp 0     TMA producer: 6-stage shared-memory ring of 32 KiB stages (this
//              CTA's 128 x 64 slice of A and 128 x 64 slice of B, 128-byte
//              swizzle). Both CTAs' copies signal the even CTA's "full" barriers.
//   warp 1     allocates 512 TMEM columns in both CTAs (two fp32 accumulators of
//              128 rows x 256 columns each); in the even CTA one thread issues
//              tcgen05.mma.cta_group::2 (M = 256, N = 256, K = 16; four per stage)
//              and releases stages / publishes accumulators in BOTH CTAs with
//              multicast tcgen05.commit.
//   warps 2-5  epilogue in each CTA: tcgen05.ld of its own 128 accumulator rows
//              (thread = row, lane quarter = warp % 4) -> registers -> mode math ->
//              global memory (dz, dH, dW: staged per warp in shared memory and written
//              by TMA stores, BoxStager); releases the accumulator on the even CTA's
//              barrier.
// Work items are handed out at run time in ascending index order (ItemRing below).
// Which cluster computes an item, and when, never changes its arithmetic: each output
// element is produced by one fixed instruction sequence regardless of T, batch
// composition, SM count or scheduling.
#pragma once

#include <atomic>

#include "rlk_internal.h"
#include "rlk_ptx.cuh"

namespace rlk {

template <int MODE>
constexpr bool is_fwd = (MODE == MODE_FWD || MODE == MODE_FWDP || MODE == MODE_FWD8);
template <int MODE>
constexpr bool is_dz = (MODE == MODE_DZ || MODE == MODE_DZ8);
template <int MODE>
constexpr bool is_e4m3 = (MODE == MODE_FWD8 || MODE == MODE_DZ8);

template <int MODE>
struct Operands {
  static constexpr bool A_MN = (MODE == MODE_DW);
  static constexpr bool B_MN = (MODE == MODE_DH || MODE == MODE_DW);
  static constexpr uint32_t IDESC =
      is_e4m3<MODE> ? make_idesc_e4m3(PAIR_M, BN) : make_idesc_bf16(PAIR_M, BN, A_MN, B_MN);
  static constexpr int K_PER_STAGE = is_e4m3<MODE> ? BK8 : BK;  // K elements of one stage
};

// Work-item order of the forward and dz kernels: items are (vocab unit, token pair-tile)
// pairs, vocab unit = leaf (forward) or DZ_UNIT 256-column tiles (dz). Token pair-tiles
// are taken in groups of TOKEN_GROUP; inside a group the items run vocab-unit-major, so
// the clusters working at one time touch at most TOKEN_GROUP token tiles of h (32 MiB of
// bf16 h at H = 4096), and W is streamed once per group. Measured at T = 8192 (GB300, items handed
// out in order): groups of 16 read 3.4 GB (forward) and 2.6 GB (dz) from DRAM; one group of
// all 32 token tiles read 9.4 / 7.7 GB (64 MiB of h does not stay in L2) and made the
// power-capped fwd+bwd step 3 % slower. The order changes only which cluster computes a
// tile and when, never a tile's arithmetic.
constexpr int TOKEN_GROUP = 16;
// dH / dW work order: items are (row tile, column tile) pairs of the output, column tiles
// taken in groups of COL_GROUP, row-tile-major inside a group. Measured at T = 8192,
// H = 4096 (16 column tiles): groups of 8 read 15.3 GB (dH) and 6.3 GB (dW) from DRAM,
// all 16 in one group 23.3 / 8.8 GB, groups of 4 15.4 / 10.1 GB; groups of 8 made the
// power-capped fwd+bwd step 1.6 % faster than one group.
constexpr int COL_GROUP = 8;

__device__ __forceinline__ void item_unit_pm(const GemmArgs& a, int n_units, int item, int& unit, int& pm) {
  const int g0 = (item / (TOKEN_GROUP * n_units)) * TOKEN_GROUP;  // first token tile of the group
  const int gsize = min(TOKEN_GROUP, a.n_pm - g0);
  const int r = item - g0 * n_units;
  unit = r / gsize;
  pm = g0 + r % gsize;
}

// Number of 256-wide tiles in a work item.
template <int MODE>
__device__ __forceinline__ int item_tiles(const GemmArgs& a, int item) {
  if constexpr (is_fwd<MODE>) {
    int leaf_local, pm;
    item_unit_pm(a, a.n_leaves, item, leaf_local, pm);
    const int col0 = (a.leaf0 + leaf_local) * LEAF;
    const int end = min(col0 + LEAF, a.V_true);
    return (end - col0 + BN - 1) / BN;
  } else if constexpr (is_dz<MODE>) {
    int vu, pm;
    item_unit_pm(a, a.n_items / a.n_pm, item, vu, pm);
    return min(DZ_UNIT, a.n_vt - vu * DZ_UNIT);
  } else {
    return 1;
  }
}

// Accumulator chunks per tile: dH / dW split K into KC_BLOCKS-block chunks.
template <int MODE>
__device__ __forceinline__ int tile_chunks(const GemmArgs& a) {
  if constexpr (MODE == MODE_DH || MODE == MODE_DW) return (a.n_kb + KC_BLOCKS - 1) / KC_BLOCKS;
  return 1;
}

// Pair-tile origin: m0 = first of the pair's 256 A / accumulator rows, n0 = first
// of its 256 B rows (fwd/dz: local W row; dH/dW: output column).
template <int MODE>
__device__ __forceinline__ void tile_origin(const GemmArgs& a, int item, int j, int& m0, int& n0) {
  if constexpr (is_fwd<MODE>) {
    int leaf_local, pm;
    item_unit_pm(a, a.n_leaves, item, leaf_local, pm);
    m0 = pm * PAIR_M;
    n0 = (a.leaf0 + leaf_local) * LEAF + j * BN - a.vocab_start;
  } else if constexpr (is_dz<MODE>) {
    int vu, pm;
    item_unit_pm(a, a.n_items / a.n_pm, item, vu, pm);
    m0 = pm * PAIR_M;
    n0 = (vu * DZ_UNIT + j) * BN;
  } else {
    // dH / dW: output column tiles in groups of COL_GROUP, row-tile-major inside a group
    const int g0 = (item / (COL_GROUP * a.n_mt)) * COL_GROUP;  // first column tile of the group
    const int gsize = min(COL_GROUP, a.n_nt - g0);
    const int r = item - g0 * a.n_mt;
    m0 = (r / gsize) * PAIR_M;
    n0 = (g0 + r % gsize) * BN;
  }
}

// Shared state of one CTA of the pair.
struct PairCtx {
  uint32_t rank;           // 0 = even CTA (issues the MMAs), 1 = odd CTA
  volatile int* abort_flag;
  uint32_t peer_abort;     // shared::cluster address of the peer CTA's abort flag
};

// Bounded wait; on expiry it also raises the peer CTA's abort flag.
__device__ __forceinline__ bool pair_wait(uint64_t* bar, uint32_t parity, const PairCtx& c) {
  if (mbar_wait_bounded(bar, parity, c.abort_flag)) return true;
  st_cluster_u32(c.peer_abort, 1u);
  return false;
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

__device__ __forceinline__ void spin_ns(uint64_t ns) {
  const uint64_t t0 = global_timer_ns();
  while (global_timer_ns() - t0 < ns) {
  }
}

// ---------------------------------------------------------------------------
// Work-item hand-out. The even CTA's producer draws the next item index from a
// counter in global memory (zeroed before the launch) each time it is ready to load
// another item, so the items in flight across all clusters always form one
// contiguous window of the work order, and the operand tiles they share are fetched
// while they are still in L2 however far the clusters drift apart in speed. (With a
// fixed round-robin assignment, clusters that run slightly faster move ahead into
// items whose operands no other cluster is reading, and the shared tiles are fetched
// from DRAM several times.) The index reaches the other roles of both CTAs through a
// ring of shared-memory slots: `full[s]` (in each CTA, one arrival from the even
// producer) publishes slot s, `empty[s]` (in the even CTA) collects one release from
// every reader: the odd producer, the MMA issuer and the eight epilogue warps. An
// index of -1 ends the work.
// ---------------------------------------------------------------------------
constexpr uint32_t ITEM_READERS = 1 + 1 + 4 * PAIR;

struct ItemRing {
  uint64_t* full;   // [ITEM_RING]
  uint64_t* empty;  // [ITEM_RING], used in the even CTA only
  int* slot;        // [ITEM_RING]
  uint32_t seq = 0;
};

// Even producer: draw the next item and publish it to both CTAs. False on abort.
__device__ __forceinline__ bool ring_publish(const GemmArgs& a, ItemRing& q, const PairCtx& c, int& item) {
  const uint32_t s = q.seq % ITEM_RING, ph = (q.seq / ITEM_RING) & 1u;
  if (!pair_wait(&q.empty[s], ph ^ 1u, c)) return false;  // every reader took the slot's last index
  int v = atomicAdd(a.sched, 1);
  if (v >= a.n_items) v = -1;
  const uint32_t slot_addr = smem_u32(&q.slot[s]);
  const uint32_t full_addr = smem_u32(&q.full[s]);
  st_cluster_u32(map_to_cta(slot_addr, 0u), static_cast<uint32_t>(v));
  st_cluster_u32(map_to_cta(slot_addr, 1u), static_cast<uint32_t>(v));
  mbar_arrive_cluster(map_to_cta(full_addr, 0u));  // release: the stores above come first
  mbar_arrive_cluster(map_to_cta(full_addr, 1u));
  ++q.seq;
  item = v;
  return true;
}

// Any other reader (one thread): take the next published item and release its slot.
__device__ __forceinline__ bool ring_take(ItemRing& q, const PairCtx& c, int& item) {
  const uint32_t s = q.seq % ITEM_RING, ph = (q.seq / ITEM_RING) & 1u;
  if (!pair_wait(&q.full[s], ph, c)) return false;
  item = *reinterpret_cast<volatile int*>(&q.slot[s]);
  mbar_arrive_cluster(map_to_cta(smem_u32(&q.empty[s]), 0u));
  ++q.seq;
  return true;
}

// An epilogue warp: every lane takes the item; lane 0 releases the slot once the whole
// warp has read it. False (in every lane) on abort.
__device__ __forceinline__ bool ring_take_warp(ItemRing& q, const PairCtx& c, int& item) {
  const uint32_t s = q.seq % ITEM_RING, ph = (q.seq / ITEM_RING) & 1u;
  bool got = pair_wait(&q.full[s], ph, c);
  got = __all_sync(0xffffffffu, got);
  if (!got) return false;
  item = *reinterpret_cast<volatile int*>(&q.slot[s]);
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive_cluster(map_to_cta(smem_u32(&q.empty[s]), 0u));
  ++q.seq;
  return true;
}

// ---------------------------------------------------------------------------
// warp 0: TMA producer (one thread per CTA)
// ---------------------------------------------------------------------------
constexpr int A_BOX_ROWS = 64;                    // K-major A boxes: 64 rows x 64 K
constexpr int A_BOX_BYTES = A_BOX_ROWS * BK * 2;  // 8 KiB

// 64-row A boxes needed for a CTA whose first A row leaves `rows_left` valid rows.
__device__ __forceinline__ int a_boxes(int rows_left) {
  return rows_left <= 0 ? 0 : min(BM / A_BOX_ROWS, (rows_left + A_BOX_ROWS - 1) / A_BOX_ROWS);
}

// One 128(MN) x 64(K) MN-major tile: two 64 x 64 swizzle atoms at dst and dst + 8 KiB,
// fetched by one copy of the 3-D view when `wide`, else by two 2-D copies. mn is a
// multiple of 128.
__device__ __forceinline__ void load_mn_tile(uint8_t* dst, const CUtensorMap* m, int32_t wide,
                                             uint32_t bar, int mn, int k0, uint64_t pol,
                                             int32_t* err_flag) {
  // the innermost coordinate of a tensor copy must be a multiple of 16 bytes (8 bf16)
  if (!dbg_ok((mn & 7) == 0, err_flag)) mn &= ~7;
  if (wide) {
    tma_load_3d_pair(dst, m, bar, 0, k0, mn / 64, pol);
  } else {
#pragma unroll
    for (int q = 0; q < 2; ++q) tma_load_2d_pair(dst + q * MN_ATOM_BYTES, m, bar, mn + q * 64, k0, pol);
  }
}

template <int MODE>
__device__ void producer_loop(const TileMaps& maps, const GemmArgs& a, uint8_t* smem, uint64_t* full,
                              uint64_t* empty, ItemRing ring, const PairCtx& c) {
  // L2 policy per operand: h is re-read by every leaf / vocab tile (fwd, dz) or by
  // every vocab tile of dW, so it is kept; the W tiles of fwd / dz are used by all
  // token tiles within a short window and then never again, so they go first.
  const uint64_t pol_keep = policy_evict_last();
  const uint64_t pol_norm = policy_evict_normal();
  const uint64_t pol_first = policy_evict_first();
  constexpr bool kZ = (is_fwd<MODE> || is_dz<MODE>);
  constexpr bool kAPerRow = (MODE != MODE_DW);  // A rows are tokens (independent outputs)
  const uint64_t polA = kZ ? pol_keep : pol_norm;
  const uint64_t polB = (MODE == MODE_DW) ? pol_keep : (kZ ? pol_first : pol_norm);
  const uint32_t r = c.rank;
  uint32_t issued = 0;
  bool ok = true;
  while (ok) {
    int item;
    ok = (r == 0) ? ring_publish(a, ring, c, item) : ring_take(ring, c, item);
    if (!ok || item < 0) break;
    const int ntiles = item_tiles<MODE>(a, item);
    for (int j = 0; ok && j < ntiles; ++j) {
      int m0, n0;
      tile_origin<MODE>(a, item, j, m0, n0);
      const int am = m0 + r * BM;      // this CTA's A rows
      const int bn = n0 + r * B_HALF;  // this CTA's B rows
      // Token-row A operands (fwd, dz, dH) load as one 128-row box when all of this CTA's
      // rows lie below T; otherwise in 64-row boxes, skipping those wholly at or beyond T:
      // accumulator rows are independent dot products, rows past T are never stored, and
      // the zero fill would otherwise cost as much load bandwidth as real data (small
      // batches). The byte count is the same either way.
      const int boxes_mine = kAPerRow ? a_boxes(a.T - am) : 0;
      const int boxes_pair = kAPerRow ? a_boxes(a.T - m0) + a_boxes(a.T - m0 - BM) : 0;
      const uint32_t tx = kAPerRow ? static_cast<uint32_t>(boxes_pair * A_BOX_BYTES + PAIR * B_STAGE_BYTES)
                                   : static_cast<uint32_t>(PAIR * STAGE_BYTES);
      for (int kb = 0; kb < a.n_kb; ++kb) {
        const uint32_t s = issued % STAGES, ph = (issued / STAGES) & 1u;
        if (!pair_wait(&empty[s], ph ^ 1u, c)) {
          ok = false;
          break;
        }
        uint8_t* sA = smem + s * STAGE_BYTES;
        uint8_t* sB = sA + A_STAGE_BYTES;
        const uint32_t bar = map_to_cta(smem_u32(&full[s]), 0);  // the even CTA's barrier
        if (r == 0) mbar_arrive_expect_tx(&full[s], tx);
        if (r == 0 && static_cast<int32_t>(issued) == a.stall_stage) {
          ++issued;  // self-test: this stage's bytes never arrive
          continue;
        }
        int k0 = kb * Operands<MODE>::K_PER_STAGE;
        // K-major copies start at k0 along their innermost axis: 16-byte aligned (E4M3 codes
        // are 1 byte, bf16 2); a failed check copies from the aligned coordinate below
        if (!dbg_ok(((k0 * (is_e4m3<MODE> ? 1 : 2)) & 15) == 0, a.err_flag)) k0 &= ~15;
        if constexpr (kAPerRow) {
          if (boxes_mine == BM / A_BOX_ROWS) {            // h / dz, K-major box 64 x 128
            tma_load_2d_pair(sA, &maps.a_full, bar, k0, am, polA);
          } else {
            for (int q = 0; q < boxes_mine; ++q)          // ragged tail: boxes 64 x 64
              tma_load_2d_pair(sA + q * A_BOX_BYTES, &maps.a, bar, k0, am + q * A_BOX_ROWS, polA);
          }
        } else {                                          // dz[k0.., am..], MN-major 128 x 64
          load_mn_tile(sA, &maps.a, a.a_mn_wide, bar, am, k0, polA, a.err_flag);
        }
        if constexpr (kZ) {
          tma_load_2d_pair(sB, &maps.b, bar, k0, bn, polB);   // W, K-major box 128 rows x 128 B
        } else {                                          // W (dH) / h (dW)[k0.., bn..], MN-major
          load_mn_tile(sB, &maps.b, a.b_mn_wide, bar, bn, k0, polB, a.err_flag);
        }
        ++issued;
      }
    }
  }
  if (ok) {
    // Tail: every stage must have been released by the MMAs (their multicast
    // commits have landed here) before the CTA may exit.
    for (uint32_t i = 0; i < STAGES; ++i) {
      const uint32_t it = issued + i;
      if (!pair_wait(&empty[it % STAGES], ((it / STAGES) & 1u) ^ 1u, c)) break;
    }
  } else if (c.rank == 0) {
    // Abort: wait for the copies already in flight (the even CTA's full barriers
    // also count the odd CTA's bytes) so no TMA write lands after exit.
    const uint32_t first = issued > STAGES ? issued - STAGES : 0;
    for (uint32_t it = first; it < issued; ++it)
      mbar_wait_timeout(&full[it % STAGES], (it / STAGES) & 1u);
  } else {
    spin_ns(1000000);  // odd CTA: its copies signal the peer; give them 1 ms to land
  }
}

// ---------------------------------------------------------------------------
// warp 1 of the even CTA: tcgen05.mma issuer (one thread)
// ---------------------------------------------------------------------------
template <int MODE>
__device__ void mma_loop(const GemmArgs& a, uint8_t* smem, uint64_t* full, uint64_t* empty,
                         uint64_t* acc_full, uint64_t* acc_empty, uint64_t* drain,
                         uint32_t tmem_base, ItemRing ring, const PairCtx& c) {
  using Ops = Operands<MODE>;
  uint32_t it = 0, tile = 0;
  bool ok = true;
  const int nchunks = tile_chunks<MODE>(a);
  while (ok) {
    int item;
    ok = ring_take(ring, c, item);
    if (!ok || item < 0) break;
    const int ntiles = item_tiles<MODE>(a, item) * nchunks;  // accumulator fills of this item
    for (int j = 0; ok && j < ntiles; ++j) {
      const uint32_t buf = tile & 1u, use = tile >> 1;
      if (!pair_wait(&acc_empty[buf], (use & 1u) ^ 1u, c)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + buf * BN;
      const int chunk = j % nchunks;
      const int kb_begin = chunk * KC_BLOCKS;
      const int kb_end = nchunks == 1 ? a.n_kb : min(a.n_kb, kb_begin + KC_BLOCKS);
      for (int kb = kb_begin; kb < kb_end; ++kb, ++it) {
        const uint32_t s = it % STAGES, ph = (it / STAGES) & 1u;
        if (!pair_wait(&full[s], ph, c)) {
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
          const uint32_t acc = (kb != kb_begin || k != 0) ? 1u : 0u;
          if constexpr (is_e4m3<MODE>)
            umma_e4m3_pair(d_tmem, ad, bd, Ops::IDESC, acc);
          else
            umma_bf16_pair(d_tmem, ad, bd, Ops::IDESC, acc);
        }
        umma_commit_pair_multicast(&empty[s], 0x3);  // stage s free in both CTAs
      }
      if (!ok) break;
      umma_commit_pair_multicast(&acc_full[buf], 0x3);  // accumulator complete in both CTAs
      ++tile;
    }
  }
  // Every issued MMA must have finished before TMEM is released.
  umma_commit_pair_local(drain);
  mbar_wait_timeout(drain, 0);
}

// ---------------------------------------------------------------------------
// warps 2-5: epilogues (128 threads per CTA; thread = one accumulator row)
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

// The same update, also leaving e(z - m) of the 64 values in v (m = the running max
// after this chunk) so they can be saved. The sum is formed in the same order as
// sum_exp64, so the statistics are identical to fwd_chunk's.
__device__ __forceinline__ void fwd_chunk_keep_exps(float (&v)[64], int valid, int tl, RowStats& st) {
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
#pragma unroll
  for (int i = 0; i < 64; ++i) v[i] = exp_shifted(v[i], st.nb);
  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = v[i];
#pragma unroll
  for (int i = 8; i < 64; ++i) acc[i & 7] = __fadd_rn(acc[i & 7], v[i]);
  const float a01 = __fadd_rn(acc[0], acc[1]), a23 = __fadd_rn(acc[2], acc[3]);
  const float a45 = __fadd_rn(acc[4], acc[5]), a67 = __fadd_rn(acc[6], acc[7]);
  st.s = __fadd_rn(st.s, __fadd_rn(__fadd_rn(a01, a23), __fadd_rn(a45, a67)));
}

__device__ __forceinline__ uint4 pack8_bf16(const float* v) {
  uint4 w;
  w.x = pack_bf16x2(v[0], v[1]);
  w.y = pack_bf16x2(v[2], v[3]);
  w.z = pack_bf16x2(v[4], v[5]);
  w.w = pack_bf16x2(v[6], v[7]);
  return w;
}

// E4M3 modes: z = acc * (s_row * s_col) for the 64 columns starting at local column
// `col` (s_col = W_scale; columns at or beyond V_local take 0, their accumulator is 0).
// Both scales are powers of two, so the products are exact while they stay normal.
__device__ __forceinline__ void apply_row_col_scales(float (&v)[64], float s_row, const float* s_col,
                                                     int col, int V_local) {
  if (col + 64 <= V_local) {  // warp-uniform: every row of the warp shares the columns
    const float4* p = reinterpret_cast<const float4*>(s_col + col);
#pragma unroll
    for (int q = 0; q < 16; ++q) {
      const float4 c4 = __ldg(p + q);
      v[4 * q] = __fmul_rn(v[4 * q], __fmul_rn(s_row, c4.x));
      v[4 * q + 1] = __fmul_rn(v[4 * q + 1], __fmul_rn(s_row, c4.y));
      v[4 * q + 2] = __fmul_rn(v[4 * q + 2], __fmul_rn(s_row, c4.z));
      v[4 * q + 3] = __fmul_rn(v[4 * q + 3], __fmul_rn(s_row, c4.w));
    }
  } else {
#pragma unroll
    for (int i = 0; i < 64; ++i) {
      const float c1 = (col + i < V_local) ? __ldg(s_col + col + i) : 0.f;
      v[i] = __fmul_rn(v[i], __fmul_rn(s_row, c1));
    }
  }
}

// Epilogue stores through shared memory and TMA (dz, and the final values of dH / dW):
// each epilogue warp writes a box of its 32 rows x 128 bytes into one of its two staging
// buffers (128-byte swizzle: 16-byte chunk j of row r goes to chunk position j ^ (r & 7),
// the layout the output tensor map expects), and lane 0 stores the box with one TMA copy,
// which writes whole 128-byte row segments instead of each thread's scattered 16-byte
// pieces. A buffer is refilled only after the copy that read it two boxes earlier has
// finished reading it.
struct BoxStager {
  uint32_t base;  // shared address of this warp's two buffers
  uint32_t seq;   // boxes staged so far
};

__device__ __forceinline__ uint32_t stage_begin(BoxStager& S, int lane) {
  if (S.seq >= 2) {
    if (lane == 0) bulk_wait_group_read<1>();
    __syncwarp();
  }
  return S.base + (S.seq & 1u) * STORE_BOX_BYTES;
}

__device__ __forceinline__ void stage_chunk(uint32_t buf, int lane, int j, uint4 v) {
  st_shared_v4(buf + static_cast<uint32_t>(lane * 128 + ((j ^ (lane & 7)) << 4)), v);
}

// Every lane of the warp calls it after staging its row; (x, y) = the box's first column
// and row in the output.
__device__ __forceinline__ void stage_store(BoxStager& S, uint32_t buf, int lane, const CUtensorMap* m,
                                            int x, int y, uint64_t pol, int32_t* err_flag) {
  fence_proxy_async_smem();
  __syncwarp();
  // a store starts at a non-negative, 16-byte aligned innermost coordinate (x is in
  // elements of 2 or 4 bytes: a multiple of 8 is aligned for both)
  if (lane == 0 && dbg_ok(x >= 0 && y >= 0 && (x & 7) == 0, err_flag)) {
    tma_store_2d(m, buf, x, y, pol);
    bulk_commit_group();
  }
  ++S.seq;
}

__device__ __forceinline__ uint4 f32x4_bits(const float* v) {
  return make_uint4(__float_as_uint(v[0]), __float_as_uint(v[1]), __float_as_uint(v[2]), __float_as_uint(v[3]));
}

template <int MODE>
__device__ void epilogue_loop(const GemmArgs& a, uint64_t* acc_full, uint64_t* acc_empty,
                              uint32_t tmem_base, ItemRing ring, const PairCtx& c,
                              const CUtensorMap* out_map, uint8_t* stage_smem) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int quarter = warp & 3;  // TMEM lane quarter this warp may access
  const int row = quarter * 32 + lane;
  const uint32_t lane_base = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16);
  const uint64_t pol_out = policy_evict_first();  // outputs are streamed, never re-read here
  uint32_t tile = 0;
  bool ok = true;
  BoxStager stg{smem_u32(stage_smem + (warp - 2) * 2 * STORE_BOX_BYTES), 0u};
  const int row0_off = static_cast<int>(c.rank) * BM + quarter * 32;  // warp's first row in a tile

  const int nchunks = tile_chunks<MODE>(a);
  while (ok) {
    int item;
    ok = ring_take_warp(ring, c, item);
    if (!ok || item < 0) break;
    const int ntiles = item_tiles<MODE>(a, item) * nchunks;  // accumulator fills of this item
    int m0, n0;
    tile_origin<MODE>(a, item, 0, m0, n0);

    // ---- per-item setup
    RowStats st{neg_inf(), 0.f, neg_inf(), 0.f};
    int64_t yt = -1;
    float g_t = 0.f, nl = 0.f;
    bool yvalid = false;
    const int t = m0 + static_cast<int>(c.rank) * BM + row;  // token row (fwd, dz, dH) or vocab row (dW)
    float s_row = 0.f;  // E4M3 modes: this token's scale
    if constexpr (is_e4m3<MODE>) {
      if (t < a.T) s_row = a.a_scale[t];
    }
    if constexpr (is_fwd<MODE>) {
      if (t < a.T) yt = a.y[t];
    } else if constexpr (is_dz<MODE>) {
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
      bool got = pair_wait(&acc_full[buf], use & 1u, c);
      got = __all_sync(0xffffffffu, got);
      if (!got) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t taddr = lane_base + buf * BN;

      if constexpr (is_fwd<MODE>) {
        const int c0 = n0 + a.vocab_start + j * BN;  // global column of the tile's first column
        const int vcols = min(BN, a.V_true - c0);
        const int tl = (yt >= c0 && yt < static_cast<int64_t>(c0) + vcols) ? static_cast<int>(yt - c0) : -1;
        const int lc = n0 + j * BN;  // local column of the tile
        constexpr bool keep_p = (MODE == MODE_FWDP);
#pragma unroll 1
        for (int ch = 0; ch < BN; ch += 64) {
          float v[64];
          tmem_ld64(taddr + ch, v);
          if constexpr (is_e4m3<MODE>) apply_row_col_scales(v, s_row, a.b_scale, lc + ch, a.V_local);
          if (a.z_out) {  // saved logits: the accumulator exactly as computed, two fp32 boxes
#pragma unroll
            for (int b = 0; b < 2; ++b) {
              const uint32_t buf = stage_begin(stg, lane);
#pragma unroll
              for (int q = 0; q < 8; ++q) stage_chunk(buf, lane, q, f32x4_bits(v + 32 * b + 4 * q));
              stage_store(stg, buf, lane, out_map, lc + ch + 32 * b, m0 + row0_off, pol_out, a.err_flag);
            }
          }
          if constexpr (keep_p) {  // saved probabilities: bf16 e(z - m) and the fp32 running max m
            fwd_chunk_keep_exps(v, vcols - ch, tl - ch, st);
            const uint32_t buf = stage_begin(stg, lane);
#pragma unroll
            for (int q = 0; q < 8; ++q) stage_chunk(buf, lane, q, pack8_bf16(v + 8 * q));
            stage_store(stg, buf, lane, out_map, lc + ch, m0 + row0_off, pol_out, a.err_flag);
            if (t < a.T) {
              const size_t i = static_cast<size_t>(t) * (a.z_ld / 64) + (lc + ch) / 64;
              if (dbg_ok(i < static_cast<size_t>(a.pm_elems), a.err_flag)) a.pm_out[i] = st.m;
            }
          } else {
            fwd_chunk(v, vcols - ch, tl - ch, st);
          }
        }
      } else if constexpr (is_dz<MODE>) {
        const int nt0 = n0 + j * BN;  // local column of this tile
        const int gc0 = a.vocab_start + nt0;
        const int vcols = max(0, min(min(BN, a.V_true - gc0), a.V_local - nt0));
        const int tl = (yvalid && yt >= gc0 && yt < static_cast<int64_t>(gc0) + vcols)
                           ? static_cast<int>(yt - gc0) : -1;
        const float ng = -g_t;
#pragma unroll 1
        for (int ch = 0; ch < BN; ch += 64) {
          float v[64];
          tmem_ld64(taddr + ch, v);
          if constexpr (is_e4m3<MODE>) apply_row_col_scales(v, s_row, a.b_scale, nt0 + ch, a.V_local);
          const int tli = tl - ch;
          float d_target = 0.f;
          const bool any_target = __any_sync(0xffffffffu, tli >= 0 && tli < 64);
          if (any_target) {
#pragma unroll
            for (int i = 0; i < 64; ++i)
              if (i == tli) d_target = dz_target(v[i], nl, g_t);
          }
#pragma unroll
          for (int i = 0; i < 64; ++i) v[i] = dz_other(v[i], nl, ng);
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
          {  // one box: this warp's 32 rows x 64 bf16 columns (rows at or past T are clipped)
            const uint32_t buf = stage_begin(stg, lane);
#pragma unroll
            for (int q = 0; q < 8; ++q) stage_chunk(buf, lane, q, pack8_bf16(v + 8 * q));
            stage_store(stg, buf, lane, out_map, nt0 + ch, m0 + row0_off, pol_out, a.err_flag);
          }
        }
      } else {
        // dH / dW: chunk j of nchunks. With one chunk the accumulator is stored directly
        // (bf16 for dH unless partial); otherwise chunk sums go to an fp32 running sum
        // (the fp32 output itself, or the scratch for a bf16 dH), folded in ascending
        // chunk order with round-to-nearest adds, and the last chunk writes the output.
        const bool row_ok = t < a.out_rows;
        const bool first = j == 0, last = j == nchunks - 1;
        float* run = a.out_f32 ? static_cast<float*>(a.out) : a.acc_scratch;
#pragma unroll 1
        for (int ch = 0; ch < BN; ch += 64) {
          float v[64];
          tmem_ld64(taddr + ch, v);
          const int col = n0 + ch;
          if (row_ok && col < a.out_cols && nchunks > 1) {
            const size_t off = static_cast<size_t>(t) * a.out_ld + col;
            float* p = run + off;
            if (!first) {
#pragma unroll
              for (int q = 0; q < 16; ++q)
                if (col + 4 * q < a.out_cols &&
                    dbg_ok(off + 4 * q + 4 <= static_cast<size_t>(a.run_elems), a.err_flag)) {
                  const float4 r = *reinterpret_cast<const float4*>(p + 4 * q);
                  v[4 * q] = __fadd_rn(r.x, v[4 * q]);
                  v[4 * q + 1] = __fadd_rn(r.y, v[4 * q + 1]);
                  v[4 * q + 2] = __fadd_rn(r.z, v[4 * q + 2]);
                  v[4 * q + 3] = __fadd_rn(r.w, v[4 * q + 3]);
                }
            }
            if (!last) {
#pragma unroll
              for (int q = 0; q < 16; ++q)
                if (col + 4 * q < a.out_cols &&
                    dbg_ok(off + 4 * q + 4 <= static_cast<size_t>(a.run_elems), a.err_flag))
                  *reinterpret_cast<float4*>(p + 4 * q) =
                      make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
              continue;
            }
          }
          if (a.out_tma && last) {
            // the final values (one chunk, or the last chunk folded into the running sum;
            // `last` is the same for every lane, so the whole warp takes this branch): all
            // lanes stage their rows, and the copy clips rows and columns past the output
            if (col < a.out_cols) {
              if (a.out_f32) {
#pragma unroll
                for (int b = 0; b < 2; ++b) {
                  if (col + 32 * b >= a.out_cols) break;
                  const uint32_t buf = stage_begin(stg, lane);
#pragma unroll
                  for (int q = 0; q < 8; ++q) stage_chunk(buf, lane, q, f32x4_bits(v + 32 * b + 4 * q));
                  stage_store(stg, buf, lane, out_map, col + 32 * b, m0 + row0_off, pol_out, a.err_flag);
                }
              } else {
                const uint32_t buf = stage_begin(stg, lane);
#pragma unroll
                for (int q = 0; q < 8; ++q) stage_chunk(buf, lane, q, pack8_bf16(v + 8 * q));
                stage_store(stg, buf, lane, out_map, col, m0 + row0_off, pol_out, a.err_flag);
              }
            }
          } else if (!a.out_tma && row_ok && col < a.out_cols) {
            const size_t off = static_cast<size_t>(t) * a.out_ld + col;
            if (a.out_f32) {
              float* p = static_cast<float*>(a.out) + off;
#pragma unroll
              for (int q = 0; q < 16; ++q)
                if (col + 4 * q < a.out_cols &&
                    dbg_ok(off + 4 * q + 4 <= static_cast<size_t>(a.out_elems), a.err_flag))
                  st_global_v4_hint(p + 4 * q,
                                    make_uint4(__float_as_uint(v[4 * q]), __float_as_uint(v[4 * q + 1]),
                                               __float_as_uint(v[4 * q + 2]), __float_as_uint(v[4 * q + 3])),
                                    pol_out);
            } else {
              uint16_t* p = static_cast<uint16_t*>(a.out) + off;
#pragma unroll
              for (int q = 0; q < 8; ++q)
                if (col + 8 * q < a.out_cols &&
                    dbg_ok(off + 8 * q + 8 <= static_cast<size_t>(a.out_elems), a.err_flag))
                  st_global_v4_hint(p + 8 * q, pack8_bf16(v + 8 * q), pol_out);
            }
          }
        }
      }

      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(map_to_cta(smem_u32(&acc_empty[buf]), 0));
      ++tile;
    }

    if constexpr (is_fwd<MODE>) {
      if (ok && t < a.T) {
        int leaf_local, pm;
        item_unit_pm(a, a.n_leaves, item, leaf_local, pm);
        const size_t i = (static_cast<size_t>(t) * a.n_leaves + leaf_local) * 3;
        if (dbg_ok(i + 3 <= static_cast<size_t>(a.ws_elems), a.err_flag)) {
          float* o = a.ws + i;
          o[0] = st.m;
          o[1] = st.s;
          o[2] = st.zt;
        }
      }
    }
  }
  // Every TMA store of this warp completes before the CTA may exit: its staging buffers
  // stay valid while they are read, and its writes are performed.
  if (lane == 0) bulk_wait_group_all();
  __syncwarp();
}

// ---------------------------------------------------------------------------
// the kernel (launched as clusters of 2 CTAs)
// ---------------------------------------------------------------------------
template <int MODE>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    gemm_kernel(const __grid_constant__ TileMaps maps, const GemmArgs a) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
  uint8_t* smem = smem_raw + pad;
  uint8_t* stage_smem = smem + STAGES * STAGE_BYTES;  // epilogue store staging (BoxStager)
  uint64_t* full = reinterpret_cast<uint64_t*>(stage_smem + STORE_STAGE_BYTES);
  uint64_t* empty = full + STAGES;
  uint64_t* acc_full = empty + STAGES;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* drain = acc_empty + 2;
  ItemRing ring;
  ring.full = drain + 1;
  ring.empty = ring.full + ITEM_RING;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(ring.empty + ITEM_RING);
  int* abort_word = reinterpret_cast<int*>(tmem_slot + 1);
  ring.slot = abort_word + 1;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  PairCtx c;
  c.rank = cluster_ctarank();
  c.abort_flag = abort_word;
  c.peer_abort = map_to_cta(smem_u32(abort_word), c.rank ^ 1u);

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);   // used in the even CTA: its producer's expect_tx arrival
      mbar_init(&empty[s], 1);  // one multicast commit per use
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], PAIR * 4);  // one arrival per epilogue warp of both CTAs
    }
    mbar_init(drain, 1);
    for (int i = 0; i < ITEM_RING; ++i) {
      mbar_init(&ring.full[i], 1);              // the even producer's publication
      mbar_init(&ring.empty[i], ITEM_READERS);  // even CTA: one release per reader
    }
    *abort_word = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&maps.a);
    if (MODE != MODE_DW) tma_prefetch_desc(&maps.a_full);
    tma_prefetch_desc(&maps.b);
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_slot, TMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // both CTAs' barriers exist before any cross-CTA arrival
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // The kernel that follows in the stream (the forward's leaf-tree merge, the backward's next
  // product) may be scheduled now; it waits for this grid's completion before it reads
  // anything.
  griddep_launch_dependents();
  // Launched as such a dependent (GemmArgs::chained), this grid has only done its setup so far
  // (barriers, tensor memory, descriptor prefetch): wait here until the kernel before it has
  // completed and its writes are visible. Otherwise this returns at once.
  griddep_wait();

  if (warp == 0) {
    if (lane == 0) producer_loop<MODE>(maps, a, smem, full, empty, ring, c);
  } else if (warp == 1) {
    if (lane == 0 && c.rank == 0)
      mma_loop<MODE>(a, smem, full, empty, acc_full, acc_empty, drain, tmem_base, ring, c);
  } else {
    epilogue_loop<MODE>(a, acc_full, acc_empty, tmem_base, ring, c, &maps.out, stage_smem);
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();  // all MMAs of the pair drained, all cross-CTA arrivals done
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, TMEM_COLS);
  }
  if (threadIdx.x == 0 && *c.abort_flag && a.err_flag) atomicOr(a.err_flag, 2);
  cluster_sync();  // neither CTA exits while its peer may still address its shared memory
}

template <int MODE>
cudaError_t launch_gemm(const TileMaps& maps, const GemmArgs& a,
                        cudaStream_t stream) {
  auto kernel = gemm_kernel<MODE>;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = PAIR;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(NUM_THREADS, 1, 1);
  cfg.dynamicSmemBytes = SMEM_BYTES;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;  // the occupancy query takes the cluster shape only
  // Shared-memory opt-in and resident pairs of this kernel, once per device (both
  // are properties of the device; racing first calls compute the same values).
  static std::atomic<int> resident[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  int clusters = (dev >= 0 && dev < 64) ? resident[dev].load(std::memory_order_relaxed) : 0;
  if (clusters <= 0) {
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return e;
    cfg.gridDim = dim3(PAIR, 1, 1);
    e = cudaOccupancyMaxActiveClusters(&clusters, kernel, &cfg);
    if (e != cudaSuccess) return e;
    if (clusters <= 0) return cudaErrorInvalidConfiguration;
    if (dev >= 0 && dev < 64) resident[dev].store(clusters, std::memory_order_relaxed);
  }
  clusters = min(clusters, a.n_items);
  cfg.gridDim = dim3(PAIR * clusters, 1, 1);
  if (!a.sched) return cudaErrorInvalidValue;
  if (!a.sched_zeroed) {
    e = cudaMemsetAsync(a.sched, 0, sizeof(int32_t), stream);  // the work-item counter
    if (e != cudaSuccess) return e;
  }
  cfg.numAttrs = a.chained ? 2 : 1;
  e = cudaLaunchKernelEx(&cfg, kernel, maps, a);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace rlk
