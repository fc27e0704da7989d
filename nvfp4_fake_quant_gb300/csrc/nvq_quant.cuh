// NVFP4 block quantization device functions (16 elements, E4M3 scale, E2M1 codes).
//
// Definition (FastVideo "nvfp4_qad.py", module docstring; "vsqa-preview-1.3b
// metadata.json", attention.precision): s = E4M3(amax*gsf/6), code =
// E2M1(|x|*gsf/s), value = sign(x)*code*s/gsf, both roundings to nearest even
// and saturating.  The two decisions are taken on IEEE fp32 values of
// amax*gsf/6 and |x|*gsf/s.
//
// Three variants:
//  * quant16_unit   exact for bf16 input and unit gsf, cheap: the scale uses a
//                   product snapped to 17 bits; each code uses a hardware
//                   reciprocal, a product and one fma residual correction.
//                   Why that equals the exact decision: x (8-bit significand)
//                   and s (<= 4 bits) make x/s either exactly a tie point t of
//                   the E2M1 grid (then x == t*s and the corrected quotient is
//                   exactly t) or at relative distance >= 2^-13 from every tie
//                   (x - t*s is a non-zero multiple of 2^min(ex-7, es-5) while
//                   t*s < 2^(es+4)), which an error of one ulp cannot cross.
//  * quant16_static IEEE fp32 products and quotients (mul.rn / div.rn) in the
//                   order of the definition: bit-identical to any IEEE fp32
//                   evaluation of the same steps.  quant16_static_fast gets
//                   the same quotients from correctly rounded reciprocals and
//                   one FMA correction each (Markstein), and sends a block
//                   whose outputs leave the normal fp32 range to quant16_static.
//  * pquant16       the softmax probabilities inside attention (fp32 inputs):
//                   reciprocal and product without snapping.  The forward and
//                   the dK/dV kernel run this same code on S from the same FP4
//                   UMMA on the same codes and scales.
#pragma once
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

namespace nvq {

// RNE(v) to E4M3FN with saturation; v >= 0 finite.  Returns the bit pattern.
__device__ __forceinline__ uint32_t e4m3_rn_sat(float v) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.0f), "f"(v));
  return r & 0xFFu;
}

// E4M3FN bit pattern (low byte of `b`) to its value, as a packed f16x2 whose
// low half holds the value.
__device__ __forceinline__ uint32_t e4m3_to_f16x2(uint32_t b) {
  uint32_t h;
  const uint16_t in = static_cast<uint16_t>(b & 0xFFu);
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"(in));
  return h;
}

__device__ __forceinline__ float f16lo_to_f32(uint32_t h2) {
  return __half2float(__ushort_as_half(static_cast<unsigned short>(h2 & 0xFFFFu)));
}

// Eight non-negative fp32 values -> eight E2M1 codes (RNE, satfinite), element
// i in nibble i of the result.
__device__ __forceinline__ uint32_t e2m1x8(const float (&v)[8]) {
  uint32_t out;
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
      "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
      : "=r"(out)
      : "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]),
        "f"(v[7]));
  return out;
}

// Eight packed E2M1 codes -> four f16x2 values (element 2j in the low half of h[j]).
__device__ __forceinline__ void e2m1x8_to_f16x2(uint32_t codes, uint32_t (&h)[4]) {
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
      "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
      "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
      : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
      : "r"(codes));
}

__device__ __forceinline__ float rcp_approx(float x) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

__device__ __forceinline__ float snap17(float q) {
  return __uint_as_float((__float_as_uint(q) + 0x40u) & 0xFFFFFF80u);
}

__device__ __forceinline__ float bf16_bits_to_f32(uint32_t b16) { return __uint_as_float(b16 << 16); }

// Result of quantizing one 16-element block of bf16 values.
struct Q16 {
  uint32_t sbyte;      // E4M3FN scale byte
  uint32_t codes[2];   // 16 four-bit codes, signed (element i in nibble i%8 of codes[i/8])
  uint32_t out[8];     // 16 dequantized values as bf16x2 or f16x2 (element 2j low half of out[j])
};

__device__ __forceinline__ uint32_t bmax2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("max.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// max |x| over 16 bf16 values (exact: bf16 maxima of magnitudes), as fp32.
__device__ __forceinline__ float amax16_bf16(const uint32_t (&x)[8]) {
  constexpr uint32_t kAbs = 0x7FFF7FFFu;
  const uint32_t m01 = bmax2(x[0] & kAbs, x[1] & kAbs), m23 = bmax2(x[2] & kAbs, x[3] & kAbs);
  const uint32_t m45 = bmax2(x[4] & kAbs, x[5] & kAbs), m67 = bmax2(x[6] & kAbs, x[7] & kAbs);
  uint32_t m = bmax2(bmax2(m01, m23), bmax2(m45, m67));
  m = bmax2(m, m >> 16);  // low half: max of both halves
  return __uint_as_float(m << 16);
}

// The sign bit of every code from the sign bit of its input element, so that a
// code rounded to zero keeps the sign of x.
__device__ __forceinline__ void code_signs(const uint32_t (&x)[8], uint32_t (&codes)[2]) {
#pragma unroll
  for (int j = 0; j < 8; ++j)
    codes[j >> 2] |= (((x[j] >> 12) & 0x8u) | ((x[j] >> 24) & 0x80u)) << (8 * (j & 3));
}

__device__ __forceinline__ uint64_t qpk2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void qup2(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}

// x/s for a pair of fp32 values (signed), from inv = rcp.approx(s) and one
// residual correction: r = x - q0*s is exact (fma), and q0 + r*inv lands on
// x/s exactly whenever x/s is a short number (a tie of the E2M1 grid), and
// within an ulp of it otherwise.  s = 0 (inv = 0) gives signed zeros.
__device__ __forceinline__ uint64_t quot2(uint64_t x2, uint64_t neg_s2, uint64_t inv2) {
  uint64_t q0, r, q;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(q0) : "l"(x2), "l"(inv2));
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(q0), "l"(neg_s2), "l"(x2));
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(q) : "l"(r), "l"(inv2), "l"(q0));
  return q;
}

// x: 16 bf16 values packed as 8 u32 (element 2j in the low half of x[j]).
// OUT_F16: dequantized values as f16 (exact for unit gsf) instead of bf16.
// The scale decision: amax*fp32(1/6) is within 2 ulp of amax/6 and snapped to
// 17 bits.  amax/6 with an 8-bit amax is either a short number (the snap
// restores it exactly) or at relative distance >= 2^-8 from every E4M3 tie
// (3 does not divide the significand), so the E4M3 rounding equals that of
// the IEEE quotient.  Codes: E2M1 of the signed quotient x/s (quot2).
template <bool OUT_F16>
__device__ __forceinline__ Q16 quant16_unit(const uint32_t (&x)[8]) {
  Q16 r;
  const float amax = amax16_bf16(x);
  r.sbyte = e4m3_rn_sat(snap17(amax * (1.0f / 6.0f)));
  const uint32_t s_h = e4m3_to_f16x2(r.sbyte) & 0xFFFFu;
  const float s = f16lo_to_f32(s_h);
  const float inv = s > 0.f ? rcp_approx(s) : 0.f;
  const uint64_t inv2 = qpk2(inv, inv), neg_s2 = qpk2(-s, -s);
  const uint32_t s_h2 = s_h | (s_h << 16);
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    float q[8];
#pragma unroll
    for (int jj = 0; jj < 4; ++jj) {
      const uint32_t w = x[4 * h + jj];
      qup2(quot2(qpk2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u)), neg_s2, inv2),
           q[2 * jj], q[2 * jj + 1]);
    }
    const uint32_t c = e2m1x8(q);
    r.codes[h] = c;
    uint32_t hv[4];
    e2m1x8_to_f16x2(c, hv);
#pragma unroll
    for (int jj = 0; jj < 4; ++jj) {
      const uint32_t m = hmul2(hv[jj], s_h2);  // exact: <= 7 significant bits, f16 normal range
      const uint32_t sg = x[4 * h + jj] & 0x80008000u;  // zeros keep the sign of x
      if (OUT_F16) {
        r.out[4 * h + jj] = m | sg;
      } else {
        __nv_bfloat162 b = __floats2bfloat162_rn(f16lo_to_f32(m), f16lo_to_f32(m >> 16));  // exact
        r.out[4 * h + jj] = *reinterpret_cast<uint32_t*>(&b) | sg;
      }
    }
  }
  return r;
}

// Static global scale g (fp32): IEEE products and quotients in the order of the
// definition, on signed values (round to nearest even is symmetric).  Output
// values are bf16 (RNE of the fp32 quotient code*s/g).
__device__ __forceinline__ Q16 quant16_static(const uint32_t (&x)[8], float g) {
  Q16 r;
  const float amax = amax16_bf16(x);
  const float t = __fdiv_rn(__fmul_rn(amax, g), 6.0f);
  r.sbyte = e4m3_rn_sat(t);
  const float s = f16lo_to_f32(e4m3_to_f16x2(r.sbyte));
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    float q[8];
#pragma unroll
    for (int jj = 0; jj < 4; ++jj) {
      const uint32_t w = x[4 * h + jj];
      const float lo = __uint_as_float(w << 16), hi = __uint_as_float(w & 0xFFFF0000u);
      q[2 * jj] = s > 0.f ? __fdiv_rn(__fmul_rn(lo, g), s) : lo * 0.f;
      q[2 * jj + 1] = s > 0.f ? __fdiv_rn(__fmul_rn(hi, g), s) : hi * 0.f;
    }
    const uint32_t c = e2m1x8(q);
    r.codes[h] = c;
    uint32_t hv[4];
    e2m1x8_to_f16x2(c, hv);
#pragma unroll
    for (int jj = 0; jj < 4; ++jj) {
      const float lo = __fdiv_rn(__fmul_rn(f16lo_to_f32(hv[jj]), s), g);
      const float hi = __fdiv_rn(__fmul_rn(f16lo_to_f32(hv[jj] >> 16), s), g);
      __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
      r.out[4 * h + jj] = *reinterpret_cast<uint32_t*>(&b) | (x[4 * h + jj] & 0x80008000u);
    }
  }
  return r;
}

}  // namespace nvq

namespace nvq {

// ---------------------------------------------------------------------------
// Softmax probabilities inside attention (forward and backward run this same
// code, so P~ agrees between them up to the S values they are given).
//
// Every rounding decision is taken on fp32 values: O is an incoherent sum of
// P~V~ terms, so even rare decision flips (from an f16 P or an f16 q = P/s)
// move it by sqrt(flip rate) x one grid step, about 1e-2 with f16 precision.
// Packed f32x2 arithmetic halves the FP32 instruction count; the E2M1 decode
// and the product code*s stay in packed halves, where they are exact.
__device__ __forceinline__ uint64_t pk2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void up2(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ float ex2_f32(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float max3f(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}
__device__ __forceinline__ uint32_t pack_f16x2_rn(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
__device__ __forceinline__ float f16hi_to_f32(uint32_t h2) {
  return __half2float(__ushort_as_half(static_cast<unsigned short>(h2 >> 16)));
}
// E2M1 code (RNE, satfinite) of two fp32 values, decoded to an f16x2 pair.
__device__ __forceinline__ uint32_t e2m1_pair_f16x2(float lo, float hi) {
  uint32_t r;
  asm("{\n\t.reg .b8 b;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b, %2, %1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b;\n\t}"
      : "=r"(r)
      : "f"(lo), "f"(hi));
  return r;
}

// amax of P over a 16-key block, max_i 2^x_i, as 2^(max_i x_i): equal bit for
// bit because ex2.approx.ftz.f32 is non-decreasing (nvq_selftest_ex2_monotone
// checks every float in [-200, 2] on the device; below -200 it returns 0, and
// a NaN argument is skipped by the maximum either way).  Taking the maximum
// of the arguments lets the block's scale be formed while its sixteen
// exponentials are still in flight.
__device__ __forceinline__ float block_amax_p(const float* x) {
  float a = max3f(x[0], x[1], x[2]);
  a = max3f(a, x[3], x[4]);
  a = max3f(a, x[5], x[6]);
  a = max3f(a, x[7], x[8]);
  a = max3f(a, x[9], x[10]);
  a = max3f(a, x[11], x[12]);
  a = max3f(a, x[13], x[14]);
  return ex2_f32(fmaxf(a, x[15]));
}

// One 16-key block.  x: exponent arguments log2(e)*(scale*S - m) (-inf for
// masked keys).  Out: p = 2^x (fp32) and P~ = E2M1(p/s)*s as f16x2 pairs,
// s = E4M3(amax/6).  Returns nothing else; the caller sums p.
__device__ __forceinline__ void pquant16(const float* x, float (&p)[16], uint32_t (&pt)[8]) {
  const uint32_t sb = e4m3_rn_sat(block_amax_p(x) * (1.0f / 6.0f));
#pragma unroll
  for (int i = 0; i < 16; ++i) p[i] = ex2_f32(x[i]);
  const uint32_t s_h = e4m3_to_f16x2(sb);
  const uint32_t s_h2 = (s_h & 0xFFFFu) | (s_h << 16);
  const float s = f16lo_to_f32(s_h);
  const float inv = s > 0.f ? rcp_approx(s) : 0.f;
  const uint64_t inv2 = pk2(inv, inv);
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    float q0, q1;
    up2(mul2(pk2(p[2 * j], p[2 * j + 1]), inv2), q0, q1);
    pt[j] = hmul2(e2m1_pair_f16x2(q0, q1), s_h2);
  }
}

__device__ __forceinline__ uint32_t prmt_b32(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
  return r;
}
__device__ __forceinline__ uint32_t mul_bf16x2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
__device__ __forceinline__ uint32_t bf16x2_splat(float v) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %1;" : "=r"(r) : "f"(v));
  return r;
}

// Eight non-negative E2M1 codes (element i in nibble i, the 3-bit magnitude
// index in its low bits) decoded to bf16 by byte lookup and multiplied by the
// bf16x2 factor f2: four bf16x2 pairs, element 2j in the low half of out[j].
// The bf16 patterns of the magnitudes 0, .5, 1, 1.5, 2, 3, 4, 6 have high
// bytes 00 3F 3F 3F 40 40 40 40 and low bytes 00 00 80 C0 00 40 80 C0; prmt
// looks up four codes per instruction (one code nibble selects one byte).
__device__ __forceinline__ void e2m1x8_bf16_mul(uint32_t codes, uint32_t f2, uint32_t* out) {
  constexpr uint32_t kLo0 = 0xC0800000u, kLo1 = 0xC0804000u;
  constexpr uint32_t kHi0 = 0x3F3F3F00u, kHi1 = 0x40404040u;
#pragma unroll
  for (int hv = 0; hv < 2; ++hv) {
    const uint32_t sel = codes >> (16 * hv);  // four code nibbles in the low 16 bits
    const uint32_t lo = prmt_b32(kLo0, kLo1, sel), hi = prmt_b32(kHi0, kHi1, sel);
    out[2 * hv] = mul_bf16x2(prmt_b32(lo, hi, 0x5140u), f2);      // elements 0, 1
    out[2 * hv + 1] = mul_bf16x2(prmt_b32(lo, hi, 0x7362u), f2);  // elements 2, 3
  }
}

// The backward's P~ / l for one 16-key block.  The quantization decisions are
// pquant16's (p = 2^x, s = E4M3(amax/6), codes = E2M1(p * rcp(s))), so the
// codes and scale equal the forward's bit for bit; the codes are then decoded
// to bf16 and multiplied by bf16(s * inv_l).  Also returns p (fp32).
__device__ __forceinline__ void pquant16_scaled_bf16(const float* x, float inv_l, float (&p)[16],
                                                     uint32_t (&out)[8]) {
  const uint32_t sb = e4m3_rn_sat(block_amax_p(x) * (1.0f / 6.0f));
#pragma unroll
  for (int i = 0; i < 16; ++i) p[i] = ex2_f32(x[i]);
  const float s = f16lo_to_f32(e4m3_to_f16x2(sb));
  const float inv = s > 0.f ? rcp_approx(s) : 0.f;
  const uint64_t inv2 = pk2(inv, inv);
  float q0[8], q1[8];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    up2(mul2(pk2(p[2 * j], p[2 * j + 1]), inv2), q0[2 * j], q0[2 * j + 1]);
    up2(mul2(pk2(p[8 + 2 * j], p[8 + 2 * j + 1]), inv2), q1[2 * j], q1[2 * j + 1]);
  }
  const uint32_t f2 = bf16x2_splat(s * inv_l);
  e2m1x8_bf16_mul(e2m1x8(q0), f2, out);
  e2m1x8_bf16_mul(e2m1x8(q1), f2, out + 4);
}

// Static global scale, fast form.  The same decisions as quant16_static, without
// per-element IEEE divisions.  Codes: y = RN(x*g) and the correctly rounded
// quotient RN(y / s) from the correctly rounded reciprocal v = RN(1/s) by one
// FMA correction: q0 = RN(y v) is within an ulp of y / s, the remainder
// y - q0 s is then exact in one FMA, and RN(q0 + (y - q0 s) v) = RN(y / s)
// (Markstein's theorem on division by FMA; y / s is far from the fp32
// underflow range wherever the E2M1 code is not 0).
// Output values: a code magnitude is 2^k * b with b in {1, 1.5}, and code * s
// is exact, so RN(code * s / g) = 2^k * RN(b * s / g) and its bf16 rounding is
// 2^k times that of RN(b * s / g) (no fp32 or bf16 range limit is near: checked).
// So each block needs two values, bf16(RN(s / g)) and bf16(RN(1.5 s / g)), the
// quotients again by one FMA correction of a product with inv_g = RN(1/g); the
// eight possible outputs are then looked up per code.  A block outside that
// range is redone by quant16_static.  The IEEE path as a call of its own, so that its registers
// stay out of the fast path's allocation.
static __device__ __noinline__ Q16 quant16_static_cold(const uint32_t (&x)[8], float g) {
  return quant16_static(x, g);
}

// bf16 bits of RN(v) (low 16 bits).
__device__ __forceinline__ uint32_t bf16_bits(float v) {
  uint16_t r;
  asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(r) : "f"(v));
  return r;
}

template <bool OUT>
__device__ __forceinline__ Q16 quant16_static_fast(const uint32_t (&x)[8], float g, float inv_g) {
  Q16 r;
  const float amax = amax16_bf16(x);
  // t = RN(RN(amax g) / 6), by the same FMA correction with RN(1/6)
  const float a = __fmul_rn(amax, g), t0 = __fmul_rn(a, 1.0f / 6.0f);
  const float t = __fmaf_rn(__fmaf_rn(-t0, 6.0f, a), 1.0f / 6.0f, t0);
  r.sbyte = e4m3_rn_sat(t);
  const float s = f16lo_to_f32(e4m3_to_f16x2(r.sbyte));
  const float inv = s > 0.f ? __frcp_rn(s) : 0.f;
  const uint64_t g2 = pk2(g, g), inv2 = pk2(inv, inv), ns2 = pk2(-s, -s);
  bool ok = true;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    float q[8];
#pragma unroll
    for (int jj = 0; jj < 4; ++jj) {
      const uint32_t w = x[4 * h + jj];
      const uint64_t y2 = mul2(pk2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u)), g2);
      const uint64_t q0 = mul2(y2, inv2);
      up2(fma2(fma2(q0, ns2, y2), inv2, q0), q[2 * jj], q[2 * jj + 1]);
    }
    r.codes[h] = e2m1x8(q);
  }
  if constexpr (OUT) {
    // f1 = RN(s / g), f15 = RN(1.5 s / g)
    const uint64_t n2 = pk2(s, 1.5f * s), ig2 = pk2(inv_g, inv_g);
    const uint64_t p0 = mul2(n2, ig2);
    float f1, f15;
    up2(fma2(fma2(p0, pk2(-g, -g), n2), ig2, p0), f1, f15);
    const uint32_t v2 = bf16_bits(f1), v3 = bf16_bits(f15);
    // 2^k scaling must stay exact: f1 / 2 and 4 f15 inside the normal range
    ok = s == 0.f || (f1 >= 0x1p-120f && f15 <= 0x1p124f);
    // bf16 bits of the eight magnitudes {0, .5, 1, 1.5, 2, 3, 4, 6} * s / g:
    // index 2, 3 are v2, v3; +-0x80 per factor of two in the exponent field
    const uint32_t nz = s > 0.f ? 0xFFFFFFFFu : 0u;
    const uint32_t w01 = ((v2 - 0x80u) << 16) & nz;                     // 0, v2 / 2
    const uint32_t w23 = (v2 | (v3 << 16)) & nz;                        // v2, v3
    const uint32_t w45 = ((v2 + 0x80u) | ((v3 + 0x80u) << 16)) & nz;    // 2 v2, 2 v3
    const uint32_t w67 = ((v2 + 0x100u) | ((v3 + 0x100u) << 16)) & nz;  // 4 v2, 4 v3
    // byte tables: low bytes of entries 0-3 / 4-7, high bytes of entries 0-3 / 4-7
    const uint32_t lo03 = prmt_b32(w01, w23, 0x6420u), hi03 = prmt_b32(w01, w23, 0x7531u);
    const uint32_t lo47 = prmt_b32(w45, w67, 0x6420u), hi47 = prmt_b32(w45, w67, 0x7531u);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
#pragma unroll
      for (int hv = 0; hv < 2; ++hv) {
        const uint32_t sel = (r.codes[h] >> (16 * hv)) & 0x7777u;  // four code magnitudes
        const uint32_t lo = prmt_b32(lo03, lo47, sel), hi = prmt_b32(hi03, hi47, sel);
        const int j = 4 * h + 2 * hv;
        r.out[j] = prmt_b32(lo, hi, 0x5140u) | (x[j] & 0x80008000u);          // elements 0, 1
        r.out[j + 1] = prmt_b32(lo, hi, 0x7362u) | (x[j + 1] & 0x80008000u);  // elements 2, 3
      }
    }
  }
  if (!ok) r = quant16_static_cold(x, g);
  return r;
}

}  // namespace nvq
