// mx.cuh - MXFP8 (OCP MX v1.0: E4M3 elements, E8M0 scale per 32 values)
// device helpers shared by the fused FC1 epilogue and the standalone
// quantisers.
//
// Block rule: e = clamp(floor(log2 amax) - 8, -127, 127) (8 = exponent of
// E4M3's largest normal), scale code = e + 127, element code =
// E4M3(v * 2^-e) rounded to nearest even with saturation to +-448.
//
// Scale layout consumed by tcgen05.mma.kind::mxf8f6f4.block_scale ("MMA
// tiled"): 128 rows (or B columns) x 4 consecutive 32-blocks of K form one
// 512-byte chunk; the scale of row r (0..127) and block kb (0..3) sits at
// byte (r % 32) * 16 + (r / 32) * 4 + kb.  tcgen05.cp .32x128b.warpx4 moves
// one chunk into 4 TMEM columns of every lane quadrant.
#pragma once

#include <cstdint>

namespace moe {

// e + 127 for a block maximum amax >= 0 (read from the float's exponent
// field: amax = 1.m * 2^(be-127), so floor(log2 amax) = be - 127; zero and
// float32 subnormals give the clamped minimum).
__device__ __forceinline__ uint32_t mx_scale_code(float amax) {
  const uint32_t be = (__float_as_uint(amax) >> 23) & 0xFFu;
  return be > 8u ? be - 8u : 0u;
}

// 2^-(code - 127) as a float (always a normal number for code <= 246)
__device__ __forceinline__ float mx_inv_scale(uint32_t code) {
  return __uint_as_float((254u - code) << 23);
}

// two floats -> two E4M3 codes (lo in the low byte), RNE, saturating
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// 32 values (already bf16-representable) -> 32 codes in 8 words, scale code
__device__ __forceinline__ uint32_t mx_quant32(const float (&v)[32], uint32_t (&q)[8]) {
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(v[i]));
  const uint32_t code = mx_scale_code(amax);
  const float inv = mx_inv_scale(code);
#pragma unroll
  for (int w = 0; w < 8; ++w) {
    const uint32_t lo = e4m3x2(v[4 * w + 0] * inv, v[4 * w + 1] * inv);
    const uint32_t hi = e4m3x2(v[4 * w + 2] * inv, v[4 * w + 3] * inv);
    q[w] = lo | (hi << 16);
  }
  return code;
}

// column-wise over the 32 lanes of a warp (one value per lane): scale code
// of the 32-row block and this lane's code
__device__ __forceinline__ uint32_t mx_quant_lanes(float v, uint32_t& code_out) {
  const uint32_t amax_bits = __reduce_max_sync(0xffffffffu, __float_as_uint(fabsf(v)));
  const uint32_t sc = mx_scale_code(__uint_as_float(amax_bits));
  code_out = e4m3x2(v * mx_inv_scale(sc), 0.f) & 0xFFu;
  return sc;
}

// byte offset of (row r in 0..127, block kb in 0..3) inside a 512-byte chunk
__device__ __forceinline__ uint32_t mx_chunk_off(int r, int kb) {
  return static_cast<uint32_t>((r & 31) * 16 + (r >> 5) * 4 + kb);
}

}  // namespace moe
