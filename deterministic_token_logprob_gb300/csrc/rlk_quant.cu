// rlk_quant.cu -- E4M3 quantization with one power-of-two scale per row, the input
// step of the FP8 LM head (the training forward quantizes its weights again at every
// step, with the same rounding rule as the inference side; AREX feed article on vLLM's
// bitwise-consistent RL training, section "对齐的代价：逐算子拆解").
//
// Per row r: e = the smallest integer with max_k |x[r][k]| <= 448 * 2^e (0 for an
// all-zero row), scale[r] = 2^e, q[r][k] = E4M3(x[r][k] / 2^e) rounded to nearest
// even. The division by 2^e is exact (a power-of-two multiply that never leaves the
// normal range for a value whose code is non-zero), so the codes are exactly those
// of the definition.
#include <cuda_runtime.h>

#include <cstdint>

#include "rlk.h"
#include "rlk_ptx.cuh"

namespace rlk {
namespace {

constexpr int kRowsPerBlock = 8;  // one warp per row

__device__ __forceinline__ float bf16_to_f32(uint16_t b) { return __uint_as_float(static_cast<uint32_t>(b) << 16); }

__global__ void __launch_bounds__(32 * kRowsPerBlock)
    quantize_rows_e4m3_kernel(const uint16_t* __restrict__ x, int64_t rows, int64_t cols,
                              uint8_t* __restrict__ q, float* __restrict__ scale, int32_t* err_flag) {
  const int lane = threadIdx.x & 31;
  const int64_t r = static_cast<int64_t>(blockIdx.x) * kRowsPerBlock + (threadIdx.x >> 5);
  if (r >= rows) return;  // warp-uniform
  const uint16_t* xr = x + r * cols;
  uint8_t* qr = q + r * cols;
  const bool vec = (cols % 16) == 0;  // rows are then 32-byte aligned (x) and 16-byte aligned (q)

  // pass 1: largest magnitude (bf16 magnitude bits order like the values) and finiteness
  uint32_t mag = 0;
  bool bad = false;
  if (vec) {
#pragma unroll 4
    for (int64_t c = static_cast<int64_t>(lane) * 16; c < cols; c += 32 * 16) {
      const uint4 u0 = *reinterpret_cast<const uint4*>(xr + c);
      const uint4 u1 = *reinterpret_cast<const uint4*>(xr + c + 8);
      const uint32_t w[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const uint32_t lo = w[i] & 0x7FFFu, hi = (w[i] >> 16) & 0x7FFFu;
        bad |= (lo >= 0x7F80u) | (hi >= 0x7F80u);
        mag = max(mag, max(lo, hi));
      }
    }
  } else {
    for (int64_t c = lane; c < cols; c += 32) {
      const uint32_t m = xr[c] & 0x7FFFu;
      bad |= m >= 0x7F80u;
      mag = max(mag, m);
    }
  }
  mag = __reduce_max_sync(0xffffffffu, mag);
  bad = __any_sync(0xffffffffu, bad);

  if (bad) {  // outside the definition: NaN scale, zero codes, flag
    if (lane == 0) {
      scale[r] = __int_as_float(0x7fc00000);
      if (err_flag) atomicOr(err_flag, RLK_FLAG_NONFINITE);
    }
    for (int64_t c = lane; c < cols; c += 32) qr[c] = 0;
    return;
  }

  int e = 0;
  if (mag != 0) {
    int k2;
    const float f = frexpf(bf16_to_f32(static_cast<uint16_t>(mag)), &k2);  // amax = f 2^k2, f in [0.5, 1)
    e = (f <= 0.875f) ? k2 - 9 : k2 - 8;  // 448 = 0.875 * 2^9
  }
  // 2^-e as one or two normal fp32 factors (e >= -142 for bf16 inputs)
  const int s1 = min(-e, 127);
  const float p1 = ldexpf(1.f, s1), p2 = ldexpf(1.f, -e - s1);
  if (lane == 0) scale[r] = ldexpf(1.f, e);

  // pass 2: codes (the row was just read: these loads mostly hit in L1 / L2)
  if (vec) {
#pragma unroll 4
    for (int64_t c = static_cast<int64_t>(lane) * 16; c < cols; c += 32 * 16) {
      const uint4 u0 = *reinterpret_cast<const uint4*>(xr + c);
      const uint4 u1 = *reinterpret_cast<const uint4*>(xr + c + 8);
      const uint32_t w[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
      uint32_t o[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint32_t a = w[2 * i], b = w[2 * i + 1];
        const float v0 = __fmul_rn(__fmul_rn(__uint_as_float(a << 16), p1), p2);
        const float v1 = __fmul_rn(__fmul_rn(__uint_as_float(a & 0xFFFF0000u), p1), p2);
        const float v2 = __fmul_rn(__fmul_rn(__uint_as_float(b << 16), p1), p2);
        const float v3 = __fmul_rn(__fmul_rn(__uint_as_float(b & 0xFFFF0000u), p1), p2);
        o[i] = static_cast<uint32_t>(cvt_e4m3x2(v1, v0)) | (static_cast<uint32_t>(cvt_e4m3x2(v3, v2)) << 16);
      }
      *reinterpret_cast<uint4*>(qr + c) = make_uint4(o[0], o[1], o[2], o[3]);
    }
  } else {
    for (int64_t c = lane; c < cols; c += 32) {
      const float v = __fmul_rn(__fmul_rn(bf16_to_f32(xr[c]), p1), p2);
      qr[c] = static_cast<uint8_t>(cvt_e4m3x2(0.f, v) & 0xFFu);
    }
  }
}

}  // namespace
}  // namespace rlk

extern "C" {

rlk_status rlk_quantize_rows_e4m3(const void* x, int64_t rows, int64_t cols, void* q, float* scale,
                                  int32_t* err_flag, void* stream) {
  if (rows < 0 || cols < 0) return RLK_ERR_INVALID_ARG;
  if (rows == 0 || cols == 0) return RLK_OK;
  if (!x || !q || !scale || cols % 8 != 0) return RLK_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(x) & 15u) != 0 || (reinterpret_cast<uintptr_t>(q) & 15u) != 0)
    return RLK_ERR_INVALID_ARG;
  if (rows > (static_cast<int64_t>(1) << 30)) return RLK_ERR_UNSUPPORTED;
  const int64_t blocks = (rows + rlk::kRowsPerBlock - 1) / rlk::kRowsPerBlock;
  rlk::quantize_rows_e4m3_kernel<<<static_cast<unsigned>(blocks), 32 * rlk::kRowsPerBlock, 0,
                                   static_cast<cudaStream_t>(stream)>>>(
      static_cast<const uint16_t*>(x), rows, cols, static_cast<uint8_t*>(q), scale, err_flag);
  return cudaGetLastError() == cudaSuccess ? RLK_OK : RLK_ERR_CUDA;
}

}  // extern "C"
