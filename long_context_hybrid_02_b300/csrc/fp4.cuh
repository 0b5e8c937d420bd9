// The FP4 indexer format on the device ("DeepSeek-V4 深度研究剖析" §8: the
// Lightning Indexer computes in FP4): rows of 80 bytes, d_I = 128 e2m1 codes two
// per byte (element 2i in the low nibble), then 8 e4m3fn scales (one per 16
// elements), then 8 unused bytes.  scale = e4m3(amax / 6), code = e2m1(x / scale),
// both rounded to nearest even with saturation, the divisions in float32.
// Quantization uses the hardware cvt instructions; widening uses byte permutes and
// an f16 multiply (exact: an e2m1 value times an e4m3 scale has at most 6
// significant bits and stays in the half range).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

namespace ha {
namespace fp4 {

constexpr int kRowBytes = 80;     // one row of d_I = 128
constexpr int kGroup = 16;        // elements per scale

// e4m3fn byte of x (nearest even, saturating at +-448).
__device__ __forceinline__ uint32_t to_e4m3(float x) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.f), "f"(x));
  return r & 0xffu;
}

// Value of an e4m3fn byte as a half (exact).
__device__ __forceinline__ __half e4m3_to_half(uint32_t byte) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(uint16_t(byte)));
  return __ushort_as_half(uint16_t(h2 & 0xffffu));
}

// Byte of two e2m1 codes: lo -> low nibble, hi -> high nibble (nearest even,
// saturating at +-6).
__device__ __forceinline__ uint32_t to_e2m1x2(float lo, float hi) {
  uint16_t r;
  asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\tcvt.u16.u8 %0, t;\n\t}"
      : "=h"(r)
      : "f"(hi), "f"(lo));
  return r & 0xffu;
}

// Two e2m1 codes of a byte as a half2 (low nibble in .x).
__device__ __forceinline__ __half2 e2m1x2_to_half2(uint32_t byte) {
  uint32_t h2;
  asm("{\n\t.reg .b8 t;\n\tcvt.u8.u16 t, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, t;\n\t}"
      : "=r"(h2)
      : "h"(uint16_t(byte)));
  return *reinterpret_cast<__half2*>(&h2);
}

// Eight e2m1 codes (4 bytes, element 0 in the lowest nibble) times their scale, as
// 8 halves in a uint4 (element order kept), without conversion instructions: the
// half of an e2m1 magnitude has a zero low byte, so a byte permute over an 8-entry
// table of high bytes gives the magnitudes; the sign bits are moved to bit 7 of
// the same bytes; the product with the scale is exact (at most 6 significant bits,
// within the half range for e4m3 scales).
__device__ __forceinline__ uint4 decode8_half(uint32_t codes, __half2 scale2) {
  constexpr uint32_t kLo = 0x3E3C3800u;              // magnitudes 0, .5, 1, 1.5
  constexpr uint32_t kHi = 0x46444240u;              // magnitudes 2, 3, 4, 6
  const uint32_t m03 = __byte_perm(kLo, kHi, codes & 0x7777u);           // e0..e3
  const uint32_t m47 = __byte_perm(kLo, kHi, (codes >> 16) & 0x7777u);   // e4..e7
  const uint32_t se = (codes << 4) & 0x80808080u;    // signs of e0, e2, e4, e6
  const uint32_t so = codes & 0x80808080u;           // signs of e1, e3, e5, e7
  const uint32_t h03 = m03 | __byte_perm(se, so, 0x5140u);
  const uint32_t h47 = m47 | __byte_perm(se, so, 0x7362u);
  uint32_t w[4] = {__byte_perm(h03, 0u, 0x1404u), __byte_perm(h03, 0u, 0x3424u),
                   __byte_perm(h47, 0u, 0x1404u), __byte_perm(h47, 0u, 0x3424u)};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __half2 v = __hmul2(*reinterpret_cast<const __half2*>(&w[i]), scale2);
    w[i] = *reinterpret_cast<const uint32_t*>(&v);
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// Quantization of 8 values whose 16-element group has absolute maximum amax16:
// the scale byte and the 4 code bytes (as one word, element 0 in the lowest
// nibble).  Also returns the decoded scale (0 for a zero group: codes 0).
__device__ __forceinline__ uint32_t quantize8(const float (&x)[8], float amax16,
                                              uint32_t& scale_byte, float& scale) {
  scale_byte = to_e4m3(__fdiv_rn(amax16, 6.f));
  scale = __half2float(e4m3_to_half(scale_byte));
  uint32_t codes = 0;
  if (scale > 0.f) {
#pragma unroll
    for (int i = 0; i < 4; ++i)
      codes |= to_e2m1x2(__fdiv_rn(x[2 * i], scale), __fdiv_rn(x[2 * i + 1], scale)) << (8 * i);
  }
  return codes;
}

}  // namespace fp4
}  // namespace ha
