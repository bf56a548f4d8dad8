// OCP FP8 E4M3 (e4m3fn) codes -> bfloat16, exactly.
//
// Every finite E4M3 value is a bfloat16 value: 3 mantissa bits fit in 7, and
// the E4M3 range (2^-9 .. 448) lies inside bfloat16's.  So the conversion is a
// change of bit layout plus one exact power-of-two scaling.  Code c = s eeee mmm
// placed as the bfloat16 bits s 0000eeee mmm0000 reads as c's value times
// 2^-120 (exponent bias 127 instead of 7; a subnormal code lands on a bfloat16
// subnormal with the same mantissa), and one bf16x2 multiply by 2^120 (exact,
// bfloat16 arithmetic keeps subnormal inputs) restores the value.  The two NaN
// codes (0x7F, 0xFF) are not preserved: they come out as +-480.
#pragma once
#include <cstdint>

namespace akp {

// q holds two codes as [0, b1, 0, b0] (bytes, high to low); returns the two
// bfloat16 values, b0 in the low half.
__device__ __forceinline__ uint32_t e4m3_pair_to_bf16x2(uint32_t q) {
  const uint32_t sign = q & 0x00800080u;
  // each half: code << 4 puts the sign at bit 11; adding sign * 240 (0x7800 per
  // set sign) carries it to bit 15 and leaves bits 11-14 clear
  const uint32_t bits = (q << 4) + sign * 240u;
  uint32_t r;
  asm("mul.rn.bf16x2 %0, %1, %2;\n" : "=r"(r) : "r"(bits), "r"(0x7B807B80u));   // x 2^120
  return r;
}

// 16 E4M3 codes (byte k = element k) -> 16 bfloat16 values as two 16-byte chunks
// (elements 0-7 in lo, 8-15 in hi; element 2j in the low half of word j).
__device__ __forceinline__ void e4m3x16_to_bf16(const uint4 raw, uint4 &lo, uint4 &hi) {
  const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
  uint32_t h[8];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    h[2 * q] = e4m3_pair_to_bf16x2(__byte_perm(w[q], 0u, 0x4140));
    h[2 * q + 1] = e4m3_pair_to_bf16x2(__byte_perm(w[q], 0u, 0x4342));
  }
  lo = make_uint4(h[0], h[1], h[2], h[3]);
  hi = make_uint4(h[4], h[5], h[6], h[7]);
}

// 16 E4M3 codes -> 16 fp16 values, also exact (every E4M3 value is an fp16
// value); one cvt.rn.f16x2.e4m3x2 per pair of codes, low byte to low half.
// The NaN codes stay NaN here.
__device__ __forceinline__ void e4m3x16_to_f16(const uint4 raw, uint4 &lo, uint4 &hi) {
  const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
  uint32_t h[8];
#pragma unroll
  for (int q = 0; q < 4; ++q)
    asm("{\n .reg .b16 l, u;\n mov.b32 {l, u}, %2;\n cvt.rn.f16x2.e4m3x2 %0, l;\n"
        " cvt.rn.f16x2.e4m3x2 %1, u;\n}\n"
        : "=r"(h[2 * q]), "=r"(h[2 * q + 1])
        : "r"(w[q]));
  lo = make_uint4(h[0], h[1], h[2], h[3]);
  hi = make_uint4(h[4], h[5], h[6], h[7]);
}

}  // namespace akp
