// Device helpers of the online activation quantizer, shared by the standalone
// activation kernel and the GEMM that quantizes its activations on chip, so
// that both produce the same codes bit for bit.
//
// Method: "FoldQuantVLA" abstract (block Hadamard transform of the
// activations, then per-token quantization) and the "Omega-QVLA" technical
// summary (normalised Hadamard matrix applied block-wise over channels;
// per-step static activation scales as the alternative to dynamic ones).
#pragma once

#include "common.cuh"

namespace vqlin_dev {

__device__ __forceinline__ void butterfly(float& a, float& b) {
  const float s = a + b, d = a - b;
  a = s;
  b = d;
}

// Normalised Walsh-Hadamard transform of blocks of HB channels (64 or 128)
// held as "units" of 32 channels per thread: a block is spread over LPG =
// HB/32 consecutive lanes, lane l of the block holding the four 8-channel
// chunks l, l + LPG, l + 2 LPG, l + 3 LPG (channel 8 (l + LPG j) + e of the
// block in v[j][e]).  The stages run in a fixed order: the 3 index bits
// inside a chunk, the 2 bits that pick the chunk, then the lane bits with
// warp shuffles; the result is scaled by 1/sqrt(HB).
template <int HB>
__device__ __forceinline__ void hadamard_unit(float (&v)[4][8], int lane) {
  constexpr int LPG = HB / 32;
#pragma unroll
  for (int j = 0; j < 4; ++j)
#pragma unroll
    for (int h = 1; h < 8; h <<= 1)
#pragma unroll
      for (int e = 0; e < 8; ++e)
        if ((e & h) == 0) butterfly(v[j][e], v[j][e + h]);
#pragma unroll
  for (int h = 1; h < 4; h <<= 1)
#pragma unroll
    for (int j = 0; j < 4; ++j)
      if ((j & h) == 0)
#pragma unroll
        for (int e = 0; e < 8; ++e) butterfly(v[j][e], v[j + h][e]);
#pragma unroll
  for (int mk = 1; mk < LPG; mk <<= 1) {
    // the partner lane holds the other half of each butterfly
    const float sg = (lane & mk) ? -1.0f : 1.0f;
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float p = __shfl_xor_sync(0xffffffffu, v[j][e], mk);
        v[j][e] = fmaf(v[j][e], sg, p);
      }
  }
  const float c = HB == 64 ? 0.125f : 0.08838834764831845f;  // 1/sqrt(HB)
#pragma unroll
  for (int j = 0; j < 4; ++j)
#pragma unroll
    for (int e = 0; e < 8; ++e) v[j][e] *= c;
}

// Codes of one 8-channel chunk, c = clamp(rint(v / s), -qmax, qmax), in the
// integer GEMM's operand encoding:
//   int4: one byte per code, s<<7 | |c| (the e4m3 bits of c * 2^-9) -> w[0..1];
//   int8: one 16-bit word per code, s<<15 | |c| (the f16 bits of c * 2^-24)
//         -> w[0..3].
// A zero scale gives zero codes.
template <int BITS>
__device__ __forceinline__ void quantize_chunk(const float (&v)[8], float s, float inv_s, uint32_t (&w)[4]) {
  constexpr int qmax = (1 << (BITS - 1)) - 1;
  w[0] = w[1] = w[2] = w[3] = 0;
  if (s == 0.0f) return;
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    // Fast quotient; near a rounding tie, redo with the IEEE division so the
    // code equals rint(v / s) exactly (|t| <= 130 gives an error < 2^-10).
    const float t = v[e] * inv_s;
    float rt = rintf(t);
    if (fabsf(t - rt) > 0.4990234375f) rt = rintf(__fdiv_rn(v[e], s));
    rt = fminf(fmaxf(rt, (float)(-qmax)), (float)qmax);
    const uint32_t mag = (uint32_t)fabsf(rt);
    const uint32_t neg = rt < 0.0f ? 1u : 0u;
    if (BITS == 4) {
      w[e >> 2] |= ((neg << 7) | mag) << (8 * (e & 3));
    } else {
      w[e >> 1] |= ((neg << 15) | mag) << (16 * (e & 1));
    }
  }
}

// The same codes from the hardware's float -> e4m3 / f16 conversions, for
// rotated activations: c * 2^-9 (int4) and c * 2^-24 (int8) are the
// subnormals of those formats, so converting clamp(v * inv_s, +-qmax) scaled
// by that power of two rounds half to even straight into the operand
// encoding, two codes per instruction (the exact path above spends a round
// and a float -> integer conversion on every code, on a conversion unit a
// quarter as wide as the arithmetic units).  The decision is taken on the
// float32 product v * inv_s, which differs from the IEEE quotient v / s only
// within 2^-22 (relative) of a half-integer.  k = inv_s * 2^-9 (int4) or
// inv_s * 2^-24 (int8).  A zero is encoded +0.
template <int BITS>
__device__ __forceinline__ void quantize_chunk_fast(const float (&v)[8], float k, uint32_t (&w)[4]) {
  constexpr float lim = BITS == 4 ? 7.0f / 512.0f : 127.0f / 16777216.0f;  // qmax times the unit
  float c[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) c[e] = fminf(fmaxf(v[e] * k, -lim), lim);
  if (BITS == 4) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      uint32_t lo, hi;
      asm("{\n\t.reg .b16 a, b;\n\t"
          "cvt.rn.satfinite.e4m3x2.f32 a, %3, %2;\n\t"
          "cvt.rn.satfinite.e4m3x2.f32 b, %5, %4;\n\t"
          "cvt.u32.u16 %0, a;\n\tcvt.u32.u16 %1, b;\n\t}"
          : "=r"(lo), "=r"(hi)
          : "f"(c[4 * h]), "f"(c[4 * h + 1]), "f"(c[4 * h + 2]), "f"(c[4 * h + 3]));
      uint32_t x = lo | (hi << 16);
      // clear the sign of zero codes: bit 7 of (b & 0x7F) + 0x7F is set iff b & 0x7F != 0
      const uint32_t mag = x & 0x7F7F7F7Fu;
      x = mag | (x & (mag + 0x7F7F7F7Fu) & 0x80808080u);
      w[h] = x;
    }
    w[2] = w[3] = 0;
  } else {
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      uint32_t x;
      asm("cvt.rn.f16x2.f32 %0, %2, %1;" : "=r"(x) : "f"(c[2 * h]), "f"(c[2 * h + 1]));
      const uint32_t mag = x & 0x7FFF7FFFu;
      x = mag | (x & (mag + 0x7FFF7FFFu) & 0x80008000u);
      w[h] = x;
    }
  }
}

}  // namespace vqlin_dev
