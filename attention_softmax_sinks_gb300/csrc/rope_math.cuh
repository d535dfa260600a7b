// Per-element arithmetic of the QKV bias + rotary step, shared by the kernel that
// writes rotated q/k (rope.cu) and the prefill that rotates q on chip (prefill.cu),
// so both produce the same bf16 values from the same (cos, sin) table.
#pragma once
#include <cstdint>

#include "ptx.cuh"

namespace sa {

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// eight bf16 values (one 16-byte vector) -> fp32
__device__ __forceinline__ void widen8(const uint4& v, float (&f)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = bf16_lo(w[i]);
    f[2 * i + 1] = bf16_hi(w[i]);
  }
}

// y += bias, eight bf16 bias values widened one word at a time
__device__ __forceinline__ void add_bias8(float (&y)[8], const uint4& b) {
  const uint32_t w[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    y[2 * i] += bf16_lo(w[i]);
    y[2 * i + 1] += bf16_hi(w[i]);
  }
}

// eight fp32 values -> bf16 (round to nearest even), one 16-byte vector
__device__ __forceinline__ uint4 pack8(const float (&f)[8]) {
  return make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]), pack_bf16x2(f[4], f[5]),
                    pack_bf16x2(f[6], f[7]));
}

// Rotation of one feature pair (a, b) = (x_i, x_{i+32}) by (c, s) = temperature x
// (cos, sin) of its angle, in place:  (a, b) -> (a c - b s, b c + a s).
__device__ __forceinline__ void rotate_pair(float& a, float& b, float c, float s) {
  const float a0 = a, b0 = b;
  a = fmaf(a0, c, -b0 * s);
  b = fmaf(b0, c, a0 * s);
}

// Pairs (y1[2i], y2[2i]) and (y1[2i+1], y2[2i+1]), where y1 holds features
// [8j, 8j + 8) of a head row and y2 their partners [8j + 32, 8j + 40); r holds
// (cos, sin, cos, sin) of pairs 8j + 2i and 8j + 2i + 1.
__device__ __forceinline__ void rotate2(float (&y1)[8], float (&y2)[8], int i, const float4& r) {
  rotate_pair(y1[2 * i], y2[2 * i], r.x, r.y);
  rotate_pair(y1[2 * i + 1], y2[2 * i + 1], r.z, r.w);
}

}  // namespace sa
