// rlk_internal.h -- host/device shared definitions of the rlk library
// (not part of the public ABI; see include/rlk.h for that).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

// Device-side index and tensor-copy coordinate checks (debug-checks builds only; see
// rlk_debug_checks in rlk.h). Off, every check below compiles to nothing.
#ifndef RLK_DEBUG_CHECKS
#define RLK_DEBUG_CHECKS 0
#endif

namespace rlk {

constexpr bool kDebugChecks = RLK_DEBUG_CHECKS != 0;
constexpr int32_t kFlagBounds = 8;  // RLK_FLAG_BOUNDS

// True when the access may go ahead. In a debug-checks build a failed check ORs the bounds
// flag into the caller's flag (if any) and returns false; otherwise it is always true.
__device__ __forceinline__ bool dbg_ok(bool cond, int32_t* err_flag) {
  if constexpr (kDebugChecks) {
    if (!cond) {
      if (err_flag) atomicOr(err_flag, kFlagBounds);
      return false;
    }
  }
  return true;
}

// Tile constants: part of the numerical contract (they fix the K steps and the
// vocab walk), identical for every shape.
constexpr int BM = 128;      // tokens per tile (tcgen05 M)
constexpr int BN = 256;      // vocab columns / output columns per tile (tcgen05 N)
constexpr int BK = 64;       // K per pipeline stage: one 128-byte swizzle atom of bf16
constexpr int UMMA_K = 16;   // K of one tcgen05.mma kind::f16
constexpr int LEAF = 1024;   // vocab columns per leaf of the merge tree
constexpr int TILES_PER_LEAF = LEAF / BN;
constexpr int MAX_SHARDS = 8;
// dH / dW reduce over the vocabulary / the tokens, which can be very long. The tensor
// core accumulates with truncation, a bias that grows with the number of accumulation
// steps (measured: ~1e-4 relative after K = 65536), so these two contractions restart
// the TMEM accumulator every KC_BLOCKS k-blocks (K = 65536) and the epilogue folds the
// chunk results in ascending order with round-to-nearest fp32 adds. The chunking
// depends only on K.
constexpr int KC_BLOCKS = 1024;
// dz work items: DZ_UNIT consecutive 256-column tiles of one token pair-tile, like the
// forward's leaves, so that the per-item costs (drawing the item, handing it to the other
// roles, the epilogue's per-row loads of y, g and lse) are paid once per four tiles. Each
// tile's arithmetic is independent of the others. With one tile per item, dz ran 12 %
// slower than the forward at T = 16384, H = 2048 (32 k-blocks per tile) and 4.5 % at
// H = 4096; with four, the T = 8192, H = 4096 dz kernel took 5.12 instead of 5.25 ms.
constexpr int DZ_UNIT = 4;

// A CTA pair (cluster of 2, tcgen05 cta_group::2) computes one 256 x 256 tile: CTA r
// holds rows [128 r, 128 r + 128) of A and of the accumulator, and rows
// [128 r, 128 r + 128) of the 256-row B tile.
constexpr int PAIR = 2;
constexpr int PAIR_M = BM * PAIR;           // 256 accumulator rows per pair
constexpr int B_HALF = BN / PAIR;           // 128 B rows per CTA
constexpr int STAGES = 6;
constexpr int A_STAGE_BYTES = BM * BK * 2;      // 16 KiB
constexpr int B_STAGE_BYTES = B_HALF * BK * 2;  // 16 KiB
constexpr int STAGE_BYTES = A_STAGE_BYTES + B_STAGE_BYTES;
constexpr int MN_ATOM_BYTES = 64 * BK * 2;  // one 64(MN) x 64(K) TMA box, 8 KiB
constexpr int NUM_THREADS = 192;            // warp 0 TMA, warp 1 MMA, warps 2-5 epilogue
constexpr int TMEM_COLS = 512;              // two fp32 128x256 accumulators per CTA
// Work items reach the roles of a pair through a ring of ITEM_RING shared-memory slots
// (the even CTA's producer draws them from a counter in global memory).
constexpr int ITEM_RING = 8;
// Epilogue store staging: each of the four epilogue warps owns two 4 KiB buffers, each one
// TMA store box of 32 rows x 128 bytes (128-byte swizzle).
constexpr int STORE_BOX_BYTES = 32 * 128;
constexpr int STORE_STAGE_BYTES = 4 * 2 * STORE_BOX_BYTES;
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + STORE_STAGE_BYTES + 1024 /* alignment slack */ +
                           512 /* barriers, slots */;

enum GemmMode : int {
  MODE_FWD = 0,  // z = h W^T per (token tile, leaf): online max / sum-exp / target
  MODE_DZ = 1,   // z = h W^T per tile: dz = g (onehot - p) -> bf16 workspace
  MODE_DH = 2,   // dH = dz W      (A K-major, B MN-major)
  MODE_DW = 3,   // dW = dz^T h    (A MN-major, B MN-major)
  MODE_FWDP = 4, // MODE_FWD that also saves bf16 e(z - m) and the running maxima
  MODE_FWD8 = 5, // MODE_FWD on E4M3 operands: z = (hq Wq^T) * h_scale[t] * W_scale[v]
  MODE_DZ8 = 6,  // MODE_DZ on E4M3 operands (the straight-through backward's logits)
};

// E4M3 modes: one 128-byte swizzle atom holds 128 K elements, so a stage spans
// BK8 = 128 of K (the same bytes as BK bf16 elements); one tcgen05.mma kind::f8f6f4
// takes K = 32 (the same 32-byte step through the atom as K = 16 of bf16).
constexpr int BK8 = 128;

// The tensor maps of one GEMM launch, passed as one __grid_constant__ parameter.
//  a       K-major A (h or dz): 64-row boxes, for tiles whose rows run past T; MN-major A
//          (dz of dW): see a_mn_wide
//  a_full  K-major A: the same tensor in 128-row boxes, for tiles with all rows below T
//  b       W or h: K-major 64 x 128 boxes (fwd, dz), or MN-major (dH, dW): see b_mn_wide
//  out     the output of dz / dH / dW for TMA stores: boxes of 128 bytes x 32 rows (64 bf16
//          or 32 fp32 columns), 128-byte swizzle; used when GemmArgs::out_tma is set
// An MN-major operand is either a 2-D map with 64 x 64 boxes (two copies per 128-wide
// tile) or, when its row length is a multiple of 64 elements, a 3-D view
// {64 elements, K rows, row / 64 atoms} that fetches both 64-wide swizzle atoms of the
// tile in one copy; the shared-memory image is the same.
struct TileMaps {  // CUtensorMap is 128-byte aligned, as TMA descriptors must be (64 B at least)
  CUtensorMap a, a_full, b, out;
};

struct GemmArgs {
  int32_t T = 0, H = 0;
  int32_t n_items = 0;
  int32_t n_kb = 0;  // k-blocks of BK per tile
  int32_t* sched = nullptr;  // work-item counter in global memory; the launcher zeroes it
  int32_t sched_zeroed = 0;  // ... unless the caller zeroed it on the stream already
  int32_t chained = 0;       // launch as a programmatic dependent of the previous kernel on the
                             // stream: its setup overlaps that kernel's tail, then it waits for it
  int32_t* err_flag = nullptr;
  // forward / dz
  int32_t V_local = 0, vocab_start = 0, V_true = 0;
  int32_t n_pm = 0;                // fwd / dz: 256-token pair tiles
  int32_t n_vt = 0;                // dz: 256-column tiles of the dz workspace
  int32_t leaf0 = 0, n_leaves = 0; // fwd: global index of the shard's first leaf, leaf count
  const int64_t* y = nullptr;
  float* ws = nullptr;             // fwd: (m, s, zt) per (token, leaf), [T][n_leaves][3]
  float* z_out = nullptr;          // fwd, optional: fp32 logits [T][z_ld] (local columns)
  int64_t z_ld = 0;
  uint16_t* p_out = nullptr;       // fwd, optional: bf16 e(z - m) [T][z_ld] with m the row's
  float* pm_out = nullptr;         //   running max after each 64-column chunk, fp32 [T][z_ld / 64]
  const float* lse = nullptr;      // dz
  const float* g = nullptr;
  uint16_t* dz = nullptr;          // dz: bf16 bits [T][dz_ld]
  int64_t dz_ld = 0;
  // dH / dW stores
  void* out = nullptr;
  int64_t out_ld = 0;
  int32_t out_rows = 0, out_cols = 0;
  int32_t out_f32 = 0;
  int32_t out_tma = 0;             // dz / dH / dW: the final values go out by TMA stores (TileMaps::out)
  float* acc_scratch = nullptr;    // dH with bf16 output and several K chunks: fp32 running sum, ld = out_ld
  int32_t a_mn_wide = 0, b_mn_wide = 0;  // MN-major maps are 3-D 128-wide views (TileMaps)
  // E4M3 modes: per-token scale of hq [T] and per-local-row scale of Wq [V_local]
  const float* a_scale = nullptr;
  const float* b_scale = nullptr;
  int32_t n_mt = 0, n_nt = 0;      // dH / dW: 256-row pair tiles along M, 256-column tiles along N
  // Extents (in elements) of the buffers the epilogue addresses by index, for the checks of
  // debug-checks builds: fwd statistics, saved running maxima, the running sum of several K
  // chunks (the fp32 output or acc_scratch), the plain-store output.
  int64_t ws_elems = 0, pm_elems = 0, run_elems = 0, out_elems = 0;
  // Self-test only (rlk_selftest_wait_timeout): the even CTA arms its `stall_stage`-th
  // stage but issues none of its copies, so the wait on that stage cannot complete.
  int32_t stall_stage = -1;
};

// Launchers (one translation unit each): enqueue one cluster launch (pairs of CTAs,
// as many pairs as can be resident, at most one per work item) on `stream`.
cudaError_t launch_gemm_fwd(const TileMaps& maps, const GemmArgs& a,
                            cudaStream_t stream);  // MODE_FWDP when a.p_out is set
cudaError_t launch_gemm_dz(const TileMaps& maps, const GemmArgs& a,
                           cudaStream_t stream);
cudaError_t launch_gemm_dh(const TileMaps& maps, const GemmArgs& a,
                           cudaStream_t stream);
cudaError_t launch_gemm_fwd8(const TileMaps& maps, const GemmArgs& a, cudaStream_t stream);
cudaError_t launch_gemm_dz8(const TileMaps& maps, const GemmArgs& a, cudaStream_t stream);
cudaError_t launch_gemm_dw(const TileMaps& maps, const GemmArgs& a,
                           cudaStream_t stream);

}  // namespace rlk
