// Device helpers shared by the libdsv4 kernels: format conversions, reductions.
//
// Storage formats (vibecoco.ai, "DeepSeek V4 agent architecture", section
// "混合注意力：两种压缩，交替使用"): KV entries in FP8 with the RoPE dims in
// BF16, indexer keys in FP4. Bit layouts are OCP e4m3fn and OCP MX e2m1.
// Every conversion rounds to nearest-even and saturates (the hardware cvt
// with .rn.satfinite); divisions that decide a code use __fdiv_rn so that the
// quantised bytes follow IEEE fp32 exactly.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/dsv4.h"

#define DSV4_DEV __device__ __forceinline__

namespace dsv4 {

DSV4_DEV float bf16_to_f32(uint16_t b) { return __uint_as_float(static_cast<uint32_t>(b) << 16); }

// round-to-nearest-even fp32 -> bf16 (finite inputs; overflow gives inf)
DSV4_DEV uint16_t f32_to_bf16(float f) {
  uint16_t r;
  asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(r) : "f"(f));
  return r;
}

// exact e4m3 -> fp32: move the 7 magnitude bits under the fp32 exponent/mantissa
// boundary (a value 2^-120 times too small, fp32 subnormal for e4m3 subnormals)
// and rescale by 2^120. Exact because the scaled value is representable.
DSV4_DEV float e4m3_to_f32(uint32_t code) {
  const uint32_t bits = ((code & 0x7Fu) << 20) | ((code & 0x80u) << 24);
  return __uint_as_float(bits) * 1.329227995784916e36f;  // 2^120
}

// fp32 pair -> packed e4m3 pair, RNE, saturating: `lo` lands in bits 0..7.
DSV4_DEV uint32_t f32x2_to_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

DSV4_DEV uint32_t f32_to_e4m3(float x) { return f32x2_to_e4m3x2(x, 0.f) & 0xFFu; }

// e2m1 nibble -> fp32 (exact)
DSV4_DEV float e2m1_to_f32(uint32_t nib) {
  const float mag[8] = {0.f, 0.5f, 1.f, 1.5f, 2.f, 3.f, 4.f, 6.f};
  const float m = mag[nib & 7u];
  return (nib & 8u) ? -m : m;
}

// 8 fp32 values -> 8 e2m1 nibbles packed into 32 bits, element 0 in the low nibble.
DSV4_DEV uint32_t f32x8_to_e2m1x8(const float* v) {
  uint32_t out;
  asm("{\n"
      ".reg .b8 b0, b1, b2, b3;\n"
      "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n"
      "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n"
      "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n"
      "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n"
      "mov.b32 %0, {b0, b1, b2, b3};\n"
      "}"
      : "=r"(out)
      : "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]));
  return out;
}

// Order-preserving map of a float score to an unsigned key (larger score ->
// larger key); -0 and +0 map to the same key.
DSV4_DEV uint32_t score_key(float s) {
  const uint32_t u = __float_as_uint(s + 0.0f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

DSV4_DEV float warp_max(float v) {
  for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
DSV4_DEV float warp_sum(float v) {
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Quantise one FP8 row held in shared memory (y[0..d_nope) fp32) with the whole
// block: scale = amax/448, code = e4m3(y/scale). `red` is >= 32 floats of
// scratch shared memory. Returns the scale (in every thread).
DSV4_DEV float block_quant_fp8_row(const float* y, int d_nope, uint8_t* codes, float* red) {
  float amax = 0.f;
  for (int c = threadIdx.x; c < d_nope; c += blockDim.x) amax = fmaxf(amax, fabsf(y[c]));
  amax = warp_max(amax);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) red[warp] = amax;
  __syncthreads();
  if (warp == 0) {
    float a = lane < (int)(blockDim.x >> 5) ? red[lane] : 0.f;
    a = warp_max(a);
    if (lane == 0) red[0] = a;
  }
  __syncthreads();
  amax = red[0];
  __syncthreads();
  const float s = __fdiv_rn(amax, 448.f);
  for (int c = 2 * threadIdx.x; c < d_nope; c += 2 * blockDim.x) {
    uint32_t pair = 0;
    if (s > 0.f) pair = f32x2_to_e4m3x2(__fdiv_rn(y[c], s), __fdiv_rn(y[c + 1], s));
    codes[c] = static_cast<uint8_t>(pair & 0xFF);
    codes[c + 1] = static_cast<uint8_t>(pair >> 8);
  }
  return s;
}

// Quantise 16 fp32 values to FP4 with one e4m3 scale: scale = e4m3(amax/6),
// codes = e2m1(v/scale). Writes 8 code bytes; returns the scale byte.
DSV4_DEV uint32_t quant_fp4_block16(const float* v, uint8_t* codes8) {
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(v[i]));
  const uint32_t sc = f32_to_e4m3(__fdiv_rn(amax, 6.f));
  const float s = e4m3_to_f32(sc);
  float q[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) q[i] = s > 0.f ? __fdiv_rn(v[i], s) : 0.f;
  const uint32_t w0 = s > 0.f ? f32x8_to_e2m1x8(q) : 0u;
  const uint32_t w1 = s > 0.f ? f32x8_to_e2m1x8(q + 8) : 0u;
  reinterpret_cast<uint32_t*>(codes8)[0] = w0;
  reinterpret_cast<uint32_t*>(codes8)[1] = w1;
  return sc;
}

}  // namespace dsv4
