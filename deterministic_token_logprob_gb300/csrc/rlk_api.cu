// rlk_api.cu -- the C ABI of include/rlk.h: argument validation, workspace
// carve-up, tensor-map encoding and kernel launches, plus the small kernels
// of the fixed merge tree (leaf tree, shard merge, shard sum).
//
// Nothing here allocates device or host memory, synchronises the host, or
// keeps state between calls beyond a cached driver entry point.
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "rlk.h"
#include "rlk_internal.h"
#include "rlk_ptx.cuh"

namespace rlk {
namespace {

// ---------------------------------------------------------------------------
// The merge operator of the statistics triples and the final step.
// ("Why the Fused Path Wins", third reason: shards combine only the statistics
// needed for the global selected logprob; fixed merge order, item 3 of "The
// Numerical Execution Contract".)
// ---------------------------------------------------------------------------
struct Triple {
  float m, s, zt;
};

__device__ __forceinline__ Triple identity_triple() { return Triple{neg_inf(), 0.f, neg_inf()}; }

__device__ __forceinline__ float merge_target(float a, float b) {
  // exactly one shard owns a valid target, the others hold -inf; NaN marks an invalid target
  return (isnan(a) || isnan(b)) ? __int_as_float(0x7fc00000) : fmaxf(a, b);
}

// a (+) b, operand a's term first. An operand with s == 0 is the identity (an
// empty shard or a padding slot) and leaves the other unchanged, bit for bit.
__device__ __noinline__ Triple merge_pair(Triple a, Triple b) {
  Triple r;
  if (a.s == 0.f) {
    r.m = b.m;
    r.s = b.s;
  } else if (b.s == 0.f) {
    r.m = a.m;
    r.s = a.s;
  } else if (a.m >= b.m) {
    r.m = a.m;
    r.s = __fadd_rn(a.s, __fmul_rn(b.s, exp_shifted(b.m, neg_scaled(a.m))));
  } else {
    r.m = b.m;
    r.s = __fadd_rn(__fmul_rn(a.s, exp_shifted(a.m, neg_scaled(b.m))), b.s);
  }
  r.zt = merge_target(a.zt, b.zt);
  return r;
}

// lse = m + log(s); logp = zt - lse.
__device__ __noinline__ void finalize(Triple x, float* logp, float* lse) {
  const float l = __fadd_rn(x.m, logf(x.s));
  *lse = l;
  *logp = __fsub_rn(x.zt, l);
}

constexpr int kMaxTreeDepth = 16;  // log2(max slots = 8 * 2048) + 1

struct TreeArgs {
  const float* ws;     // [T][n_leaves_local][3]: (m, s, zt) of each (token, leaf)
  int64_t ws_elems;    // its extent in floats (index checks of debug-checks builds)
  int32_t T;
  int32_t n_leaves_local, leaf0, n_leaves_global;
  int32_t L_ss, P;                // leaves per super-shard, slots per super-shard
  int32_t slot_begin, slot_count; // this shard's aligned slot range (slot_count a power of two)
  const int64_t* y;
  int32_t V_true;
  rlk_lse_partial* partial;
  float* logp;
  float* lse;
  int32_t* err_flag;
};

__device__ __forceinline__ Triple load_slot(const TreeArgs& a, int t, int q) {
  const int slot = a.slot_begin + q;
  const int ss = slot / a.P, jj = slot - ss * a.P;
  const int leaf = ss * a.L_ss + jj;
  const int ll = leaf - a.leaf0;
  if (jj < a.L_ss && leaf < a.n_leaves_global && ll >= 0 && ll < a.n_leaves_local) {
    const size_t i = (static_cast<size_t>(t) * a.n_leaves_local + ll) * 3;
    if (dbg_ok(i + 3 <= static_cast<size_t>(a.ws_elems), a.err_flag)) {
      const float* p = a.ws + i;
      return Triple{p[0], p[1], p[2]};
    }
  }
  return identity_triple();
}

__device__ __forceinline__ Triple shfl_xor_triple(const Triple& x, int d) {
  return Triple{__shfl_xor_sync(0xffffffffu, x.m, d), __shfl_xor_sync(0xffffffffu, x.s, d),
                __shfl_xor_sync(0xffffffffu, x.zt, d)};
}

// One warp per token: the balanced pairwise tree over the shard's slot_count slots
// (a power of two). Lane L merges its run of consecutive slots with a binary-counter
// walk (after slot q, merge once per trailing one bit of q) -- the tree's lower
// levels -- then the lanes combine pairwise by xor-shuffles, the lower lane's
// subtree always the left operand: the same tree, node for node, as a sequential
// walk over all slots.

__global__ void leaf_tree_kernel(const TreeArgs a) {
  // Launched as a programmatic dependent of the forward tile kernel: wait until that grid
  // has completed and its leaf statistics are visible (returns at once otherwise).
  griddep_wait();
  const int t = static_cast<int>((static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  if (t >= a.T) return;  // warp-uniform
  const int per = a.slot_count >= 32 ? a.slot_count >> 5 : 1;
  const int lanes = a.slot_count >= 32 ? 32 : a.slot_count;
  Triple node = identity_triple();
  if (lane < lanes) {
    Triple stack[kMaxTreeDepth];
    int sp = 0;
    for (int q0 = 0; q0 < per; q0 += 8) {
      Triple buf[8];
#pragma unroll
      for (int i = 0; i < 8; ++i)
        buf[i] = (q0 + i < per) ? load_slot(a, t, lane * per + q0 + i) : identity_triple();
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int q = q0 + i;
        if (q >= per) break;
        Triple n = buf[i];
        for (int idx = q; idx & 1; idx >>= 1) n = merge_pair(stack[--sp], n);
        stack[sp++] = n;
      }
    }
    node = stack[0];
  }
  for (int d = 1; d < lanes; d <<= 1) {
    const Triple other = shfl_xor_triple(node, d);
    node = (lane & d) ? merge_pair(other, node) : merge_pair(node, other);
  }
  if (lane != 0) return;
  Triple r = node;
  const int64_t y = a.y[t];
  if (y < 0 || y >= a.V_true) {
    r.zt = __int_as_float(0x7fc00000);
    if (a.err_flag) atomicOr(a.err_flag, RLK_FLAG_BAD_TARGET);
  }
  if (a.partial) {
    a.partial[t] = rlk_lse_partial{r.m, r.s, r.zt};
  } else {
    float lp, l;
    finalize(r, &lp, &l);
    if (a.logp) a.logp[t] = lp;
    if (a.lse) a.lse[t] = l;
  }
}

// Top levels of the same tree over S shard triples, then the final step.
__global__ void lse_merge_kernel(const rlk_lse_partial* p, int S, int T, float* logp, float* lse) {
  const int t = blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= T) return;
  Triple stack[4];
  int sp = 0;
  for (int q = 0; q < S; ++q) {
    const rlk_lse_partial x = p[static_cast<size_t>(q) * T + t];
    Triple node{x.m, x.s, x.zt};
    for (int idx = q; idx & 1; idx >>= 1) node = merge_pair(stack[--sp], node);
    stack[sp++] = node;
  }
  float lp, l;
  finalize(stack[0], &lp, &l);
  logp[t] = lp;
  lse[t] = l;
}

// out = bf16(((p0 + p1) + p2) + ...), four elements per thread. The vector path
// needs every shard's row start 16-byte aligned, i.e. n % 4 == 0.
__global__ void shard_sum_kernel(const float* p, int S, int64_t n, uint16_t* out) {
  const int64_t i4 = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) * 4;
  if (i4 >= n) return;
  if (i4 + 4 <= n && (n & 3) == 0) {
    float4 acc = *reinterpret_cast<const float4*>(p + i4);
    for (int s = 1; s < S; ++s) {
      const float4 x = *reinterpret_cast<const float4*>(p + static_cast<size_t>(s) * n + i4);
      acc.x = __fadd_rn(acc.x, x.x);
      acc.y = __fadd_rn(acc.y, x.y);
      acc.z = __fadd_rn(acc.z, x.z);
      acc.w = __fadd_rn(acc.w, x.w);
    }
    uint2 w;
    w.x = pack_bf16x2(acc.x, acc.y);
    w.y = pack_bf16x2(acc.z, acc.w);
    *reinterpret_cast<uint2*>(out + i4) = w;
  } else {
    for (int64_t i = i4; i < n; ++i) {
      float acc = p[i];
      for (int s = 1; s < S; ++s) acc = __fadd_rn(acc, p[static_cast<size_t>(s) * n + i]);
      out[i] = static_cast<uint16_t>(pack_bf16x2(acc, 0.f) & 0xFFFFu);
    }
  }
}

// dz from saved fp32 logits. One block per token row: the row's target, gradient and lse
// are read once, and each thread takes eight consecutive columns per step, UNROLL steps
// at a time with all of their loads issued first (a streaming pass: fp32 z read, bf16 dz
// written). Same arithmetic as the recompute epilogue (dz_target / dz_other), so the two
// backward paths produce identical bits.
constexpr int DZS_THREADS = 256;
constexpr int DZS_UNROLL = 4;

__global__ void __launch_bounds__(DZS_THREADS)
    dz_from_logits_kernel(const float* __restrict__ z, int64_t z_ld, const int64_t* __restrict__ y,
                          const float* __restrict__ lse, const float* __restrict__ g, int Vd,
                          int V_valid, int vocab_start, int V_true, uint16_t* __restrict__ dz,
                          int64_t dz_ld, int32_t* err_flag, int64_t z_elems, int64_t dz_elems) {
  const int t = blockIdx.x;
  const int64_t yt = y[t];
  const bool yvalid = yt >= 0 && yt < V_true;
  if (!yvalid && threadIdx.x == 0 && err_flag) atomicOr(err_flag, RLK_FLAG_BAD_TARGET);
  const float gt = g[t];
  const float nl = neg_scaled(lse[t]);
  const float ng = -gt;
  const int64_t tcol = yt - vocab_start;  // the target's local column
  const float* zr = z + static_cast<size_t>(t) * z_ld;
  uint16_t* dr = dz + static_cast<size_t>(t) * dz_ld;
  const int n_valid = yvalid ? V_valid : 0;  // columns with a nonzero gradient
  for (int base = threadIdx.x * 8; base < Vd; base += DZS_THREADS * 8 * DZS_UNROLL) {
    float4 zv[DZS_UNROLL][2];
#pragma unroll
    for (int u = 0; u < DZS_UNROLL; ++u) {
      const int c0 = base + u * DZS_THREADS * 8;
      if (c0 < n_valid &&
          dbg_ok(static_cast<size_t>(t) * z_ld + c0 + 8 <= static_cast<size_t>(z_elems), err_flag)) {
        const float4* zp = reinterpret_cast<const float4*>(zr + c0);
        zv[u][0] = zp[0];
        zv[u][1] = zp[1];
      } else {
        zv[u][0] = zv[u][1] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
#pragma unroll
    for (int u = 0; u < DZS_UNROLL; ++u) {
      const int c0 = base + u * DZS_THREADS * 8;
      if (c0 >= Vd) break;
      float d[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) d[i] = 0.f;
      if (c0 < n_valid) {
        const float v8[8] = {zv[u][0].x, zv[u][0].y, zv[u][0].z, zv[u][0].w,
                             zv[u][1].x, zv[u][1].y, zv[u][1].z, zv[u][1].w};
        const int64_t tl = tcol - c0;  // target column inside this group, if any
#pragma unroll
        for (int i = 0; i < 8; ++i)
          if (c0 + i < n_valid) d[i] = (i == tl) ? dz_target(v8[i], nl, gt) : dz_other(v8[i], nl, ng);
      }
      uint4 w;
      w.x = pack_bf16x2(d[0], d[1]);
      w.y = pack_bf16x2(d[2], d[3]);
      w.z = pack_bf16x2(d[4], d[5]);
      w.w = pack_bf16x2(d[6], d[7]);
      if (dbg_ok(static_cast<size_t>(t) * dz_ld + c0 + 8 <= static_cast<size_t>(dz_elems), err_flag))
        *reinterpret_cast<uint4*>(dr + c0) = w;
    }
  }
}

// dz from saved bf16 probabilities: p = e(z - m) (bf16) x e(m - lse), m the row's running
// max recorded per 64-column chunk. Same block-per-row structure as dz_from_logits_kernel.
__global__ void __launch_bounds__(DZS_THREADS)
    dz_from_probs_kernel(const uint16_t* __restrict__ pb, const float* __restrict__ pm, int64_t ld,
                         const int64_t* __restrict__ y, const float* __restrict__ lse,
                         const float* __restrict__ g, int Vd, int V_valid, int vocab_start,
                         int V_true, uint16_t* __restrict__ dz, int64_t dz_ld, int32_t* err_flag,
                         int64_t p_elems, int64_t pm_elems, int64_t dz_elems) {
  const int t = blockIdx.x;
  const int64_t yt = y[t];
  const bool yvalid = yt >= 0 && yt < V_true;
  if (!yvalid && threadIdx.x == 0 && err_flag) atomicOr(err_flag, RLK_FLAG_BAD_TARGET);
  const float gt = g[t];
  const float nls = neg_scaled(lse[t]);
  const int64_t tcol = yt - vocab_start;
  const uint16_t* pr = pb + static_cast<size_t>(t) * ld;
  const float* pmr = pm + static_cast<size_t>(t) * (ld / 64);
  uint16_t* dr = dz + static_cast<size_t>(t) * dz_ld;
  const int n_valid = yvalid ? V_valid : 0;
  for (int base = threadIdx.x * 8; base < Vd; base += DZS_THREADS * 8 * DZS_UNROLL) {
    uint4 raw[DZS_UNROLL];
    float mx[DZS_UNROLL];
#pragma unroll
    for (int u = 0; u < DZS_UNROLL; ++u) {
      const int c0 = base + u * DZS_THREADS * 8;
      if (c0 < n_valid &&
          dbg_ok(static_cast<size_t>(t) * ld + c0 + 8 <= static_cast<size_t>(p_elems) &&
                     static_cast<size_t>(t) * (ld / 64) + c0 / 64 < static_cast<size_t>(pm_elems),
                 err_flag)) {
        raw[u] = *reinterpret_cast<const uint4*>(pr + c0);
        mx[u] = pmr[c0 / 64];
      } else {
        raw[u] = make_uint4(0u, 0u, 0u, 0u);
        mx[u] = 0.f;
      }
    }
#pragma unroll
    for (int u = 0; u < DZS_UNROLL; ++u) {
      const int c0 = base + u * DZS_THREADS * 8;
      if (c0 >= Vd) break;
      float d[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) d[i] = 0.f;
      if (c0 < n_valid) {
        const uint32_t w[4] = {raw[u].x, raw[u].y, raw[u].z, raw[u].w};
        const float scale = exp_shifted(mx[u], nls);
        const int64_t tl = tcol - c0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const uint32_t bits = (i & 1) ? (w[i >> 1] & 0xFFFF0000u) : (w[i >> 1] << 16);
          const float p = __fmul_rn(__uint_as_float(bits), scale);
          if (c0 + i < n_valid) d[i] = (i == tl) ? __fmul_rn(gt, __fsub_rn(1.f, p)) : __fmul_rn(-gt, p);
        }
      }
      uint4 o;
      o.x = pack_bf16x2(d[0], d[1]);
      o.y = pack_bf16x2(d[2], d[3]);
      o.z = pack_bf16x2(d[4], d[5]);
      o.w = pack_bf16x2(d[6], d[7]);
      if (dbg_ok(static_cast<size_t>(t) * dz_ld + c0 + 8 <= static_cast<size_t>(dz_elems), err_flag))
        *reinterpret_cast<uint4*>(dr + c0) = o;
    }
  }
}

// ---------------------------------------------------------------------------
// host helpers
// ---------------------------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode;
}

// 2-D tensor [outer][inner] (inner contiguous) of bf16 (elem_bytes 2) or E4M3 codes
// (elem_bytes 1), 128-byte swizzled boxes of box_inner x box_outer elements;
// out-of-range elements read as zero.
bool encode_2d(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint64_t row_elems,
               uint32_t box_inner, uint32_t box_outer, int elem_bytes = 2) {
  auto enc = encoder();
  if (!enc) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {row_elems * static_cast<uint64_t>(elem_bytes)};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  const CUtensorMapDataType dt = elem_bytes == 1   ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                 : elem_bytes == 4 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                                   : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  CUresult r = enc(m, dt, 2, const_cast<void*>(base), dims, strides, box,
                   estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// MN-major operand [K rows][row_elems] (row_elems contiguous, the MN axis) whose tiles are
// 128 wide in MN and 64 deep in K. With row_elems a multiple of 64 it is viewed as
// {64 elements, K rows, row_elems / 64 atoms} with 3-D boxes {64, 64, 2}: one copy fetches
// both 128-byte swizzle atoms of a tile, in the layout two 2-D 64 x 64 boxes give. Other
// row lengths keep the 2-D map (the view's last atom would run past the row). *wide says
// which one was made.
bool encode_mn(CUtensorMap* m, const void* base, uint64_t row_elems, uint64_t k_rows, int32_t* wide) {
  if (row_elems % 64 != 0) {
    *wide = 0;
    return encode_2d(m, base, row_elems, k_rows, row_elems, 64, 64);
  }
  auto enc = encoder();
  if (!enc) return false;
  cuuint64_t dims[3] = {64, k_rows, row_elems / 64};
  cuuint64_t strides[2] = {row_elems * 2, 128};
  cuuint32_t box[3] = {64, 64, 2};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
                   estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  *wide = 1;
  return r == CUDA_SUCCESS;
}

// K-major token-row operand [T][row_elems] as the two A maps of TileMaps (boxes of one
// 128-byte swizzle atom along K: 64 bf16 or 128 E4M3 codes).
bool encode_rows(TileMaps* m, const void* base, uint64_t row_elems, uint64_t T, int elem_bytes = 2) {
  const uint32_t k_box = 128u / static_cast<uint32_t>(elem_bytes);
  return encode_2d(&m->a, base, row_elems, T, row_elems, k_box, 64, elem_bytes) &&
         encode_2d(&m->a_full, base, row_elems, T, row_elems, k_box, BM, elem_bytes);
}

// Output [rows][cols] (row length cols, contiguous) as TileMaps::out: boxes of 128 bytes
// (64 bf16 or 32 fp32 columns) x 32 rows, 128-byte swizzle, for the epilogue's TMA stores.
bool encode_out(TileMaps* m, const void* base, uint64_t cols, uint64_t rows, int elem_bytes) {
  return encode_2d(&m->out, base, cols, rows, cols, 128u / static_cast<uint32_t>(elem_bytes), 32, elem_bytes);
}

// E4M3 operands of the FP8 entry points: codes in place of h / W plus their scales.
struct Fp8In {
  const float* h_scale;  // [T]
  const float* W_scale;  // [V_local], 16-byte aligned
};

inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
inline int64_t round_up(int64_t a, int64_t b) { return ceil_div(a, b) * b; }
inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool is_pow2(int64_t x) { return x > 0 && (x & (x - 1)) == 0; }
inline int64_t next_pow2(int64_t x) {
  int64_t p = 1;
  while (p < x) p <<= 1;
  return p;
}

// Geometry of the fixed merge tree for a given V_true, and the part of it a
// shard [vocab_start, vocab_start + V_local) owns.
struct ShardGeom {
  int64_t n_leaves, L_ss, P, ss_width;  // tree
  int64_t ss0, n_ss;                    // shard's super-shards
  int64_t leaf0, n_leaves_local;        // shard's leaves (global index of the first)
  int64_t slot_begin, slot_count;
  bool reaches_end;
};

rlk_status shard_geometry(int64_t V_local, int64_t vocab_start, int64_t V_true, ShardGeom* g) {
  g->n_leaves = ceil_div(V_true, LEAF);
  g->L_ss = ceil_div(g->n_leaves, MAX_SHARDS);
  g->P = next_pow2(g->L_ss);
  g->ss_width = g->L_ss * LEAF;
  if (vocab_start % g->ss_width != 0) return RLK_ERR_UNSUPPORTED;
  g->ss0 = vocab_start / g->ss_width;
  if (g->ss0 >= MAX_SHARDS) return RLK_ERR_UNSUPPORTED;
  g->reaches_end = vocab_start + V_local >= V_true;
  if (!g->reaches_end && V_local % g->ss_width != 0) return RLK_ERR_UNSUPPORTED;
  int64_t n = ceil_div(V_local, g->ss_width);
  if (n > MAX_SHARDS - g->ss0) n = MAX_SHARDS - g->ss0;
  if (g->reaches_end) n = next_pow2(n);
  if (!is_pow2(n) || g->ss0 % n != 0 || g->ss0 + n > MAX_SHARDS) return RLK_ERR_UNSUPPORTED;
  g->n_ss = n;
  g->leaf0 = g->ss0 * g->L_ss;
  const int64_t leaf_end = std::min((g->ss0 + n) * g->L_ss, g->n_leaves);
  g->n_leaves_local = std::max<int64_t>(0, leaf_end - g->leaf0);
  g->slot_begin = g->ss0 * g->P;
  g->slot_count = n * g->P;
  return RLK_OK;
}

rlk_status common_checks(const void* h, const void* W, const int64_t* y, int64_t T, int64_t H,
                         int64_t V_local, int64_t vocab_start, int64_t V_true) {
  // per-token inputs may be NULL for an empty batch (an empty tensor has no storage)
  if (!W || (T > 0 && (!h || !y))) return RLK_ERR_INVALID_ARG;
  if (T < 0 || H <= 0 || V_local <= 0 || vocab_start < 0 || V_true <= 0) return RLK_ERR_INVALID_ARG;
  if (H % 8 != 0 || !aligned16(h) || !aligned16(W)) return RLK_ERR_INVALID_ARG;
  if (V_true > RLK_MAX_VOCAB || V_local > RLK_MAX_VOCAB || vocab_start > RLK_MAX_VOCAB ||
      H > RLK_MAX_HIDDEN || T > INT32_MAX - BM)
    return RLK_ERR_UNSUPPORTED;
  return RLK_OK;
}

size_t fwd_ws_array_bytes(int64_t T, int64_t V_local) {
  return static_cast<size_t>(round_up(ceil_div(V_local, LEAF) * T * 4, 256));
}

// Work-item counters of the tile kernels (one int32 per launch of a call; each launch
// zeroes its own before it starts), at the end of either workspace.
constexpr size_t SCHED_BYTES = 256;

// Backward workspace: the bf16 dz tiles, then (when dH's K = vocab spans several
// accumulation chunks) an fp32 running sum for a bf16 dH.
size_t bwd_dz_bytes(int64_t T, int64_t V_local) {
  return static_cast<size_t>(round_up(T * round_up(V_local, BN) * 2, 256));
}

size_t bwd_run_bytes(int64_t T, int64_t H, int64_t V_local) {
  return V_local > static_cast<int64_t>(KC_BLOCKS) * BK ? static_cast<size_t>(T) * H * 4 : 0;
}

// Saved probabilities: bf16 [T][round_up(V_local, 256)], then fp32 chunk maxima
// [T][round_up(V_local, 256) / 64] at a 256-byte aligned offset.
size_t saved_probs_offset(int64_t T, int64_t V_local) {
  return static_cast<size_t>(round_up(T * round_up(V_local, BN) * 2, 256));
}

size_t saved_probs_bytes(int64_t T, int64_t V_local) {
  if (T <= 0 || V_local <= 0) return 0;
  return saved_probs_offset(T, V_local) + static_cast<size_t>(T) * (round_up(V_local, BN) / 64) * 4;
}

size_t saved_logits_bytes(int64_t T, int64_t V_local) {
  if (T <= 0 || V_local <= 0) return 0;
  return static_cast<size_t>(T) * static_cast<size_t>(round_up(V_local, BN)) * 4;
}

}  // namespace
}  // namespace rlk

using namespace rlk;

extern "C" {

const char* rlk_version(void) { return "rlk 0.1.0 sm_103a"; }

const char* rlk_status_string(rlk_status s) {
  switch (s) {
    case RLK_OK: return "ok";
    case RLK_ERR_INVALID_ARG: return "invalid argument";
    case RLK_ERR_UNSUPPORTED: return "unsupported shape or shard split";
    case RLK_ERR_WORKSPACE: return "workspace missing or too small";
    case RLK_ERR_CUDA: return "CUDA error";
  }
  return "unknown status";
}

size_t rlk_linear_logp_fwd_workspace(int64_t T, int64_t H, int64_t V_local) {
  (void)H;
  if (T <= 0 || V_local <= 0) return 0;
  return 3 * fwd_ws_array_bytes(T, V_local) + SCHED_BYTES;
}

}  // extern "C"

namespace rlk {
namespace {

// The forward; z_saved (optional) receives the fp32 logits of the shard's columns.
rlk_status fwd_impl(const void* h, const void* W, const int64_t* y, int64_t T, int64_t H,
                    int64_t V_local, int64_t vocab_start, int64_t V_true, float* logp, float* lse,
                    rlk_lse_partial* partial, float* z_saved, size_t z_saved_bytes,
                    int32_t* err_flag, void* workspace, size_t workspace_bytes, void* stream,
                    int32_t stall_stage = -1, void* p_saved = nullptr, size_t p_saved_bytes = 0,
                    const Fp8In* f8 = nullptr, int64_t ws_entries_short = 0) {
  rlk_status st = common_checks(h, W, y, T, H, V_local, vocab_start, V_true);
  if (st != RLK_OK) return st;
  if (f8 && (H % 16 != 0 || !f8->W_scale || !aligned16(f8->W_scale) || (T > 0 && !f8->h_scale)))
    return RLK_ERR_INVALID_ARG;
  if (T > 0 && !partial && !logp && !lse) return RLK_ERR_INVALID_ARG;
  ShardGeom g;
  st = shard_geometry(V_local, vocab_start, V_true, &g);
  if (st != RLK_OK) return st;
  if (!partial && (vocab_start != 0 || !g.reaches_end)) return RLK_ERR_INVALID_ARG;
  if (z_saved && (!aligned16(z_saved) || z_saved_bytes < saved_logits_bytes(T, V_local)))
    return RLK_ERR_INVALID_ARG;
  if (z_saved && p_saved) return RLK_ERR_INVALID_ARG;  // the forward saves one of the two
  if (p_saved && ((reinterpret_cast<uintptr_t>(p_saved) & 255u) != 0 ||
                  p_saved_bytes < saved_probs_bytes(T, V_local)))
    return RLK_ERR_INVALID_ARG;
  if (T == 0) return RLK_OK;
  const size_t arr = fwd_ws_array_bytes(T, V_local);
  if (g.n_leaves_local > 0) {
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return RLK_ERR_WORKSPACE;
    if (workspace_bytes < 3 * arr + SCHED_BYTES) return RLK_ERR_WORKSPACE;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  float* ws = static_cast<float*>(workspace);  // [T][n_leaves_local][3] (fits in 3 * arr)
  // its extent for the index checks (the bounds self-test understates it by whole entries)
  const int64_t ws_elems = (T * g.n_leaves_local - ws_entries_short) * 3;

  if (g.n_leaves_local > 0) {
    const int eb = f8 ? 1 : 2;  // element bytes of h / W
    TileMaps maps{};
    if (!encode_rows(&maps, h, H, T, eb)) return RLK_ERR_CUDA;
    if (!encode_2d(&maps.b, W, H, V_local, H, 128 / eb, B_HALF, eb)) return RLK_ERR_CUDA;
    GemmArgs a;
    a.T = static_cast<int32_t>(T);
    a.H = static_cast<int32_t>(H);
    a.V_local = static_cast<int32_t>(V_local);
    a.vocab_start = static_cast<int32_t>(vocab_start);
    a.V_true = static_cast<int32_t>(V_true);
    a.n_pm = static_cast<int32_t>(ceil_div(T, PAIR_M));
    a.leaf0 = static_cast<int32_t>(g.leaf0);
    a.n_leaves = static_cast<int32_t>(g.n_leaves_local);
    if (static_cast<int64_t>(a.n_pm) * a.n_leaves > INT32_MAX) return RLK_ERR_UNSUPPORTED;
    a.n_items = a.n_pm * a.n_leaves;
    a.n_kb = static_cast<int32_t>(ceil_div(H, f8 ? BK8 : BK));
    if (f8) {
      a.a_scale = f8->h_scale;
      a.b_scale = f8->W_scale;
    }
    a.y = y;
    a.ws = ws;
    a.ws_elems = ws_elems;
    a.z_out = z_saved;
    a.z_ld = round_up(V_local, BN);
    if (z_saved && !encode_out(&maps, z_saved, a.z_ld, T, 4)) return RLK_ERR_CUDA;
    if (p_saved) {
      a.p_out = static_cast<uint16_t*>(p_saved);
      a.pm_out = reinterpret_cast<float*>(static_cast<char*>(p_saved) + saved_probs_offset(T, V_local));
      a.pm_elems = T * (a.z_ld / 64);
      if (!encode_out(&maps, p_saved, a.z_ld, T, 2)) return RLK_ERR_CUDA;
    }
    a.err_flag = err_flag;
    a.sched = reinterpret_cast<int32_t*>(static_cast<char*>(workspace) + 3 * arr);
    a.stall_stage = stall_stage;
    if ((f8 ? launch_gemm_fwd8(maps, a, s) : launch_gemm_fwd(maps, a, s)) != cudaSuccess) return RLK_ERR_CUDA;
  }

  TreeArgs ta;
  ta.ws = ws;
  ta.ws_elems = ws_elems;
  ta.T = static_cast<int32_t>(T);
  ta.n_leaves_local = static_cast<int32_t>(g.n_leaves_local);
  ta.leaf0 = static_cast<int32_t>(g.leaf0);
  ta.n_leaves_global = static_cast<int32_t>(g.n_leaves);
  ta.L_ss = static_cast<int32_t>(g.L_ss);
  ta.P = static_cast<int32_t>(g.P);
  ta.slot_begin = static_cast<int32_t>(g.slot_begin);
  ta.slot_count = static_cast<int32_t>(g.slot_count);
  ta.y = y;
  ta.V_true = static_cast<int32_t>(V_true);
  ta.partial = partial;
  ta.logp = logp;
  ta.lse = lse;
  ta.err_flag = err_flag;
  const int warps_per_block = 8;  // one warp per token
  // Programmatic stream serialization: the tree kernel's launch overlaps the tail of the
  // tile kernel (it waits for the tile kernel's completion inside, griddep_wait).
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(ceil_div(T, warps_per_block)), 1, 1);
  cfg.blockDim = dim3(32 * warps_per_block, 1, 1);
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, leaf_tree_kernel, ta) != cudaSuccess) return RLK_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? RLK_OK : RLK_ERR_CUDA;
}

}  // namespace
}  // namespace rlk

extern "C" {

rlk_status rlk_linear_logp_fwd(const void* h, const void* W, const int64_t* y, int64_t T,
                               int64_t H, int64_t V_local, int64_t vocab_start, int64_t V_true,
                               float* logp, float* lse, rlk_lse_partial* partial,
                               int32_t* err_flag, void* workspace, size_t workspace_bytes,
                               void* stream) {
  return fwd_impl(h, W, y, T, H, V_local, vocab_start, V_true, logp, lse, partial, nullptr, 0,
                  err_flag, workspace, workspace_bytes, stream);
}

size_t rlk_saved_logits_bytes(int64_t T, int64_t V_local) { return saved_logits_bytes(T, V_local); }

size_t rlk_saved_probs_bytes(int64_t T, int64_t V_local) { return saved_probs_bytes(T, V_local); }

rlk_status rlk_linear_logp_fwd_save_probs(const void* h, const void* W, const int64_t* y,
                                          int64_t T, int64_t H, int64_t V_local,
                                          int64_t vocab_start, int64_t V_true, float* logp,
                                          float* lse, rlk_lse_partial* partial, void* p_saved,
                                          size_t p_saved_bytes, int32_t* err_flag,
                                          void* workspace, size_t workspace_bytes, void* stream) {
  if (T > 0 && !p_saved) return RLK_ERR_INVALID_ARG;
  return fwd_impl(h, W, y, T, H, V_local, vocab_start, V_true, logp, lse, partial, nullptr, 0,
                  err_flag, workspace, workspace_bytes, stream, -1, p_saved, p_saved_bytes);
}

int32_t rlk_debug_checks(void) { return kDebugChecks ? 1 : 0; }

rlk_status rlk_selftest_bounds_check(const void* h, const void* W, const int64_t* y, int64_t T,
                                     int64_t H, int64_t V, int64_t V_true, float* logp, float* lse,
                                     int32_t* err_flag, void* workspace, size_t workspace_bytes,
                                     void* stream) {
  if (!kDebugChecks) return RLK_ERR_UNSUPPORTED;
  if (!err_flag || T <= 0) return RLK_ERR_INVALID_ARG;
  return fwd_impl(h, W, y, T, H, V, 0, V_true, logp, lse, nullptr, nullptr, 0, err_flag, workspace,
                  workspace_bytes, stream, -1, nullptr, 0, nullptr, /*ws_entries_short=*/1);
}

rlk_status rlk_selftest_wait_timeout(const void* h, const void* W, const int64_t* y, int64_t T,
                                     int64_t H, int64_t V, int64_t V_true, float* logp, float* lse,
                                     int32_t* err_flag, void* workspace, size_t workspace_bytes,
                                     void* stream) {
  if (!err_flag || T <= 0) return RLK_ERR_INVALID_ARG;
  return fwd_impl(h, W, y, T, H, V, 0, V_true, logp, lse, nullptr, nullptr, 0, err_flag, workspace,
                  workspace_bytes, stream, /*stall_stage=*/0);
}

rlk_status rlk_linear_logp_fwd_save(const void* h, const void* W, const int64_t* y, int64_t T,
                                    int64_t H, int64_t V_local, int64_t vocab_start,
                                    int64_t V_true, float* logp, float* lse,
                                    rlk_lse_partial* partial, float* z_saved,
                                    size_t z_saved_bytes, int32_t* err_flag, void* workspace,
                                    size_t workspace_bytes, void* stream) {
  if (T > 0 && !z_saved) return RLK_ERR_INVALID_ARG;
  return fwd_impl(h, W, y, T, H, V_local, vocab_start, V_true, logp, lse, partial, z_saved,
                  z_saved_bytes, err_flag, workspace, workspace_bytes, stream);
}

rlk_status rlk_lse_merge(const rlk_lse_partial* partials, int32_t S, int64_t T, float* logp,
                         float* lse, void* stream) {
  if (T < 0 || (T > 0 && (!partials || !logp || !lse))) return RLK_ERR_INVALID_ARG;
  if (S != 1 && S != 2 && S != 4 && S != 8) return RLK_ERR_UNSUPPORTED;
  if (T > INT32_MAX) return RLK_ERR_UNSUPPORTED;
  if (T == 0) return RLK_OK;
  const int threads = 128;
  lse_merge_kernel<<<static_cast<unsigned>(ceil_div(T, threads)), threads, 0,
                     static_cast<cudaStream_t>(stream)>>>(partials, S, static_cast<int>(T), logp, lse);
  return cudaGetLastError() == cudaSuccess ? RLK_OK : RLK_ERR_CUDA;
}

size_t rlk_linear_logp_bwd_workspace(int64_t T, int64_t H, int64_t V_local) {
  if (T <= 0 || V_local <= 0) return 0;
  return bwd_dz_bytes(T, V_local) + bwd_run_bytes(T, H, V_local) + SCHED_BYTES;
}

}  // extern "C"

namespace rlk {
namespace {

// The backward; with z_saved the dz tiles come from the saved logits instead of
// a recomputed GEMM.
rlk_status bwd_impl(const void* h, const void* W, const int64_t* y, const float* lse,
                    const float* g, const float* z_saved, int64_t T, int64_t H, int64_t V_local,
                    int64_t vocab_start, int64_t V_true, void* dH, int32_t dH_fp32_partial,
                    float* dW, int32_t* err_flag, void* workspace, size_t workspace_bytes,
                    void* stream, const void* p_saved = nullptr, const void* hq = nullptr,
                    const void* Wq = nullptr, const Fp8In* f8 = nullptr,
                    int32_t stages = RLK_BWD_DZ | RLK_BWD_DH | RLK_BWD_DW) {
  rlk_status st = common_checks(h, W, y, T, H, V_local, vocab_start, V_true);
  if (st != RLK_OK) return st;
  if (f8) {  // straight-through: dz from the E4M3 logits, dH / dW with the bf16 operands
    st = common_checks(hq, Wq, y, T, H, V_local, vocab_start, V_true);
    if (st != RLK_OK) return st;
    if (H % 16 != 0 || !f8->W_scale || !aligned16(f8->W_scale) || (T > 0 && !f8->h_scale))
      return RLK_ERR_INVALID_ARG;
  }
  if (T > 0 && (!lse || !g)) return RLK_ERR_INVALID_ARG;
  if ((dH && !aligned16(dH)) || (dW && !aligned16(dW))) return RLK_ERR_INVALID_ARG;
  if (T == 0) return RLK_OK;
  const int64_t Vd = round_up(V_local, BN);
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return RLK_ERR_WORKSPACE;
  if (workspace_bytes < rlk_linear_logp_bwd_workspace(T, H, V_local)) return RLK_ERR_WORKSPACE;
  if (Vd > INT32_MAX / 2) return RLK_ERR_UNSUPPORTED;
  // every launch's work-item count fits int32 (checked before anything is enqueued)
  {
    const int64_t pm = ceil_div(T, PAIR_M), nt = ceil_div(H, BN);
    if ((Vd / BN) * pm > INT32_MAX || pm * nt > INT32_MAX || ceil_div(V_local, PAIR_M) * nt > INT32_MAX)
      return RLK_ERR_UNSUPPORTED;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint16_t* dz = static_cast<uint16_t*>(workspace);
  const int32_t n_pm = static_cast<int32_t>(ceil_div(T, PAIR_M));
  int32_t* sched = reinterpret_cast<int32_t*>(static_cast<char*>(workspace) + bwd_dz_bytes(T, V_local) +
                                              bwd_run_bytes(T, H, V_local));  // dz, dH, dW
  // The work-item counters of this call's tile kernels are zeroed first, each stage's own only
  // (the dH and dW stages may run at once on two streams), so that the kernels follow one
  // another directly: dH and dW start as programmatic dependents of the kernel before them.
  {
    const bool run[3] = {(stages & RLK_BWD_DZ) != 0 && !p_saved && !z_saved,
                         (stages & RLK_BWD_DH) != 0 && dH != nullptr,
                         (stages & RLK_BWD_DW) != 0 && dW != nullptr};
    for (int i = 0; i < 3;) {
      if (!run[i]) {
        ++i;
        continue;
      }
      int j = i;
      while (j < 3 && run[j]) ++j;
      if (cudaMemsetAsync(sched + i, 0, (j - i) * sizeof(int32_t), s) != cudaSuccess) return RLK_ERR_CUDA;
      i = j;
    }
  }
  bool after_kernel = false;  // the last operation this call enqueued is a kernel

  // 1. dz (bf16) workspace: from saved probabilities, saved logits, or recomputed z tiles
  if (!(stages & RLK_BWD_DZ)) {
    // the workspace already holds this shard's dz (rlk_linear_logp_bwd_stages)
  } else if (p_saved) {
    const int64_t V_valid = std::max<int64_t>(0, std::min<int64_t>(V_true - vocab_start, V_local));
    dz_from_probs_kernel<<<static_cast<unsigned>(T), DZS_THREADS, 0, s>>>(  // one block per row
        static_cast<const uint16_t*>(p_saved),
        reinterpret_cast<const float*>(static_cast<const char*>(p_saved) + saved_probs_offset(T, V_local)),
        Vd, y, lse, g, static_cast<int>(Vd), static_cast<int>(V_valid),
        static_cast<int>(vocab_start), static_cast<int>(V_true), dz, Vd, err_flag, T * Vd,
        T * (Vd / 64), T * Vd);
    if (cudaGetLastError() != cudaSuccess) return RLK_ERR_CUDA;
    after_kernel = true;
  } else if (z_saved) {
    const int64_t V_valid = std::max<int64_t>(0, std::min<int64_t>(V_true - vocab_start, V_local));
    dz_from_logits_kernel<<<static_cast<unsigned>(T), DZS_THREADS, 0, s>>>(  // one block per row
        z_saved, Vd, y, lse, g, static_cast<int>(Vd), static_cast<int>(V_valid),
        static_cast<int>(vocab_start), static_cast<int>(V_true), dz, Vd, err_flag, T * Vd, T * Vd);
    if (cudaGetLastError() != cudaSuccess) return RLK_ERR_CUDA;
    after_kernel = true;
  } else {
    const int eb = f8 ? 1 : 2;  // element bytes of the logit operands
    TileMaps maps{};
    if (!encode_rows(&maps, f8 ? hq : h, H, T, eb)) return RLK_ERR_CUDA;
    if (!encode_2d(&maps.b, f8 ? Wq : W, H, V_local, H, 128 / eb, B_HALF, eb)) return RLK_ERR_CUDA;
    GemmArgs a;
    a.T = static_cast<int32_t>(T);
    a.H = static_cast<int32_t>(H);
    a.V_local = static_cast<int32_t>(V_local);
    a.vocab_start = static_cast<int32_t>(vocab_start);
    a.V_true = static_cast<int32_t>(V_true);
    a.n_pm = n_pm;
    a.n_vt = static_cast<int32_t>(Vd / BN);
    a.n_items = static_cast<int32_t>(ceil_div(a.n_vt, DZ_UNIT)) * n_pm;  // checked above
    a.n_kb = static_cast<int32_t>(ceil_div(H, f8 ? BK8 : BK));
    if (f8) {
      a.a_scale = f8->h_scale;
      a.b_scale = f8->W_scale;
    }
    a.y = y;
    a.lse = lse;
    a.g = g;
    a.dz = dz;
    a.dz_ld = Vd;
    if (!encode_out(&maps, dz, Vd, T, 2)) return RLK_ERR_CUDA;
    a.out_tma = 1;
    a.err_flag = err_flag;
    a.sched = sched;
    a.sched_zeroed = 1;
    if ((f8 ? launch_gemm_dz8(maps, a, s) : launch_gemm_dz(maps, a, s)) != cudaSuccess) return RLK_ERR_CUDA;
    after_kernel = true;
  }

  // 2. dH = dz W over this shard's valid columns
  if (dH && (stages & RLK_BWD_DH)) {
    const int64_t V_valid = std::max<int64_t>(0, std::min<int64_t>(V_true - vocab_start, V_local));
    const size_t elem = dH_fp32_partial ? 4 : 2;
    if (V_valid == 0) {
      if (cudaMemsetAsync(dH, 0, static_cast<size_t>(T) * H * elem, s) != cudaSuccess) return RLK_ERR_CUDA;
      after_kernel = false;
    } else {
      TileMaps maps{};
      GemmArgs a;
      if (!encode_rows(&maps, dz, Vd, T)) return RLK_ERR_CUDA;
      if (!encode_mn(&maps.b, W, H, V_local, &a.b_mn_wide)) return RLK_ERR_CUDA;
      a.T = static_cast<int32_t>(T);
      a.H = static_cast<int32_t>(H);
      a.n_mt = n_pm;
      a.n_nt = static_cast<int32_t>(ceil_div(H, BN));
      if (static_cast<int64_t>(a.n_mt) * a.n_nt > INT32_MAX) return RLK_ERR_UNSUPPORTED;
      a.n_items = a.n_mt * a.n_nt;
      a.n_kb = static_cast<int32_t>(ceil_div(V_valid, BK));
      a.out = dH;
      a.out_ld = H;
      a.out_rows = static_cast<int32_t>(T);
      a.out_cols = static_cast<int32_t>(H);
      a.out_f32 = dH_fp32_partial ? 1 : 0;
      if (!dH_fp32_partial && a.n_kb > KC_BLOCKS)
        a.acc_scratch = reinterpret_cast<float*>(static_cast<char*>(workspace) + bwd_dz_bytes(T, V_local));
      a.out_elems = T * H;
      a.run_elems = (dH_fp32_partial || a.acc_scratch) ? T * H : 0;
      // TMA stores of the final values, unless the fp32 output is itself the running sum
      // of several K chunks (then every chunk updates it with plain loads and stores)
      if (!dH_fp32_partial || a.n_kb <= KC_BLOCKS) {
        if (!encode_out(&maps, dH, H, T, dH_fp32_partial ? 4 : 2)) return RLK_ERR_CUDA;
        a.out_tma = 1;
      }
      a.err_flag = err_flag;
      a.sched = sched + 1;
      a.sched_zeroed = 1;
      a.chained = after_kernel ? 1 : 0;
      if (launch_gemm_dh(maps, a, s) != cudaSuccess) return RLK_ERR_CUDA;
      after_kernel = true;
    }
  }

  // 3. dW = dz^T h (rows at or above V_true come out exactly zero: their dz is zero)
  if (dW && (stages & RLK_BWD_DW)) {
    TileMaps maps{};
    GemmArgs a;
    if (!encode_mn(&maps.a, dz, Vd, T, &a.a_mn_wide)) return RLK_ERR_CUDA;
    maps.a_full = maps.a;  // unused: dW's A is MN-major
    if (!encode_mn(&maps.b, h, H, T, &a.b_mn_wide)) return RLK_ERR_CUDA;
    a.T = static_cast<int32_t>(T);
    a.H = static_cast<int32_t>(H);
    a.n_mt = static_cast<int32_t>(ceil_div(V_local, PAIR_M));
    a.n_nt = static_cast<int32_t>(ceil_div(H, BN));
    if (static_cast<int64_t>(a.n_mt) * a.n_nt > INT32_MAX) return RLK_ERR_UNSUPPORTED;
    a.n_items = a.n_mt * a.n_nt;
    a.n_kb = static_cast<int32_t>(ceil_div(T, BK));
    a.out = dW;
    a.out_ld = H;
    a.out_rows = static_cast<int32_t>(V_local);
    a.out_cols = static_cast<int32_t>(H);
    a.out_f32 = 1;
    a.out_elems = a.run_elems = V_local * H;
    if (a.n_kb <= KC_BLOCKS) {  // one K chunk: TMA stores (several: dW is the running sum)
      if (!encode_out(&maps, dW, H, V_local, 4)) return RLK_ERR_CUDA;
      a.out_tma = 1;
    }
    a.err_flag = err_flag;
    a.sched = sched + 2;
    a.sched_zeroed = 1;
    a.chained = after_kernel ? 1 : 0;
    if (launch_gemm_dw(maps, a, s) != cudaSuccess) return RLK_ERR_CUDA;
  }
  return RLK_OK;
}

}  // namespace
}  // namespace rlk

extern "C" {

rlk_status rlk_linear_logp_bwd(const void* h, const void* W, const int64_t* y, const float* lse,
                               const float* g, int64_t T, int64_t H, int64_t V_local,
                               int64_t vocab_start, int64_t V_true, void* dH,
                               int32_t dH_fp32_partial, float* dW, int32_t* err_flag,
                               void* workspace, size_t workspace_bytes, void* stream) {
  return bwd_impl(h, W, y, lse, g, nullptr, T, H, V_local, vocab_start, V_true, dH,
                  dH_fp32_partial, dW, err_flag, workspace, workspace_bytes, stream);
}

rlk_status rlk_linear_logp_bwd_stages(const void* h, const void* W, const int64_t* y,
                                      const float* lse, const float* g, int64_t T, int64_t H,
                                      int64_t V_local, int64_t vocab_start, int64_t V_true,
                                      void* dH, int32_t dH_fp32_partial, float* dW,
                                      int32_t stages, int32_t* err_flag, void* workspace,
                                      size_t workspace_bytes, void* stream) {
  constexpr int32_t all = RLK_BWD_DZ | RLK_BWD_DH | RLK_BWD_DW;
  if (stages == 0 || (stages & ~all) != 0) return RLK_ERR_INVALID_ARG;
  if (((stages & RLK_BWD_DH) && !dH) || ((stages & RLK_BWD_DW) && !dW)) return RLK_ERR_INVALID_ARG;
  return bwd_impl(h, W, y, lse, g, nullptr, T, H, V_local, vocab_start, V_true, dH,
                  dH_fp32_partial, dW, err_flag, workspace, workspace_bytes, stream, nullptr,
                  nullptr, nullptr, nullptr, stages);
}

rlk_status rlk_linear_logp_bwd_saved(const void* h, const void* W, const int64_t* y,
                                     const float* lse, const float* g, const float* z_saved,
                                     size_t z_saved_bytes, int64_t T, int64_t H, int64_t V_local,
                                     int64_t vocab_start, int64_t V_true, void* dH,
                                     int32_t dH_fp32_partial, float* dW, int32_t* err_flag,
                                     void* workspace, size_t workspace_bytes, void* stream) {
  if (T > 0 && (!z_saved || !aligned16(z_saved) || z_saved_bytes < saved_logits_bytes(T, V_local)))
    return RLK_ERR_INVALID_ARG;
  return bwd_impl(h, W, y, lse, g, z_saved, T, H, V_local, vocab_start, V_true, dH,
                  dH_fp32_partial, dW, err_flag, workspace, workspace_bytes, stream);
}

rlk_status rlk_linear_logp_bwd_saved_probs(const void* h, const void* W, const int64_t* y,
                                           const float* lse, const float* g, const void* p_saved,
                                           size_t p_saved_bytes, int64_t T, int64_t H,
                                           int64_t V_local, int64_t vocab_start, int64_t V_true,
                                           void* dH, int32_t dH_fp32_partial, float* dW,
                                           int32_t* err_flag, void* workspace,
                                           size_t workspace_bytes, void* stream) {
  if (T > 0 && (!p_saved || (reinterpret_cast<uintptr_t>(p_saved) & 255u) != 0 ||
                p_saved_bytes < saved_probs_bytes(T, V_local)))
    return RLK_ERR_INVALID_ARG;
  return bwd_impl(h, W, y, lse, g, nullptr, T, H, V_local, vocab_start, V_true, dH,
                  dH_fp32_partial, dW, err_flag, workspace, workspace_bytes, stream, p_saved);
}

rlk_status rlk_linear_logp_fwd_fp8(const void* hq, const float* h_scale, const void* Wq,
                                   const float* W_scale, const int64_t* y, int64_t T, int64_t H,
                                   int64_t V_local, int64_t vocab_start, int64_t V_true, float* logp,
                                   float* lse, rlk_lse_partial* partial, int32_t* err_flag,
                                   void* workspace, size_t workspace_bytes, void* stream) {
  const Fp8In f8{h_scale, W_scale};
  return fwd_impl(hq, Wq, y, T, H, V_local, vocab_start, V_true, logp, lse, partial, nullptr, 0,
                  err_flag, workspace, workspace_bytes, stream, -1, nullptr, 0, &f8);
}

rlk_status rlk_linear_logp_bwd_fp8(const void* h, const void* W, const void* hq,
                                   const float* h_scale, const void* Wq, const float* W_scale,
                                   const int64_t* y, const float* lse, const float* g, int64_t T,
                                   int64_t H, int64_t V_local, int64_t vocab_start, int64_t V_true,
                                   void* dH, int32_t dH_fp32_partial, float* dW, int32_t* err_flag,
                                   void* workspace, size_t workspace_bytes, void* stream) {
  const Fp8In f8{h_scale, W_scale};
  return bwd_impl(h, W, y, lse, g, nullptr, T, H, V_local, vocab_start, V_true, dH,
                  dH_fp32_partial, dW, err_flag, workspace, workspace_bytes, stream, nullptr, hq, Wq,
                  &f8);
}

rlk_status rlk_shard_sum_bf16(const float* partials, int32_t S, int64_t n, void* out, void* stream) {
  if (!partials || !out || S < 1 || n < 0) return RLK_ERR_INVALID_ARG;
  if (!aligned16(partials) || !aligned16(out)) return RLK_ERR_INVALID_ARG;
  if (n == 0) return RLK_OK;
  const int threads = 256;
  const int64_t blocks = ceil_div(ceil_div(n, 4), threads);
  if (blocks > INT32_MAX) return RLK_ERR_UNSUPPORTED;
  shard_sum_kernel<<<static_cast<unsigned>(blocks), threads, 0, static_cast<cudaStream_t>(stream)>>>(
      partials, S, n, static_cast<uint16_t*>(out));
  return cudaGetLastError() == cudaSuccess ? RLK_OK : RLK_ERR_CUDA;
}

}  // extern "C"
