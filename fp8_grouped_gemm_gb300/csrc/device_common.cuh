// Device-side helpers shared by the kernels of libmgq: bf16 access, the
// saturating round-to-nearest casts to the 8- and 4-bit formats, the E8M0
// block-scale exponent, and the device error word.
#pragma once
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "mgq.h"

namespace mgq {

// ---------------------------------------------------------------------------
// error word (one per device, see abi.cu); kernels receive its address.

__device__ __forceinline__ void report(int* err, int code) {
  if (err) atomicCAS(err, 0, code);
}

// ---------------------------------------------------------------------------
// bf16

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);   // .x = lo, .y = hi
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ float round_bf16(float x) {
  return __bfloat162float(__float2bfloat16_rn(x));
}

// SwiGLU pieces with the fast intrinsics (their float32 error is far below the
// bf16 rounding of every result they feed). Every kernel that evaluates SwiGLU
// or its derivative uses these, so fused and separate paths agree bit for bit.
__device__ __forceinline__ float silu_fast(float g) { return __fdividef(g, 1.0f + __expf(-g)); }
__device__ __forceinline__ float sigmoid_fast(float g) { return __fdividef(1.0f, 1.0f + __expf(-g)); }
// h = bf16(silu(g) u)
__device__ __forceinline__ float swiglu_bf16(float g, float u) { return round_bf16(__fmul_rn(silu_fast(g), u)); }
// silu(g) u in float32, before the bf16 rounding
__device__ __forceinline__ float swiglu_f32(float g, float u) { return __fmul_rn(silu_fast(g), u); }
// dSwiGLU of one element with s = sigmoid(g): dG = dh u s (1 + g (1 - s)),
// dU = dh g s in float32 (before the bf16 rounding), every operation spelled
// out so no kernel contracts it differently
__device__ __forceinline__ void dswiglu_f32(float d, float g, float u, float& dg, float& du) {
  const float s = sigmoid_fast(g);
  const float t = __fmaf_rn(g, __fsub_rn(1.0f, s), 1.0f);
  dg = __fmul_rn(__fmul_rn(__fmul_rn(d, u), s), t);
  du = __fmul_rn(__fmul_rn(d, g), s);
}
// Packed float32 pairs (sm_100 f32x2 forms): each lane is one IEEE operation
// with round-to-nearest, the same result as the scalar __fadd_rn / __fsub_rn /
// __fmul_rn / __fmaf_rn.
struct f32x2 {
  float x, y;
};
// a pair rounded to bf16 and packed (.x in the low half)
__device__ __forceinline__ uint32_t pack_bf16x2x2(f32x2 v) { return pack_bf16x2(v.x, v.y); }
__device__ __forceinline__ f32x2 mul2(f32x2 a, f32x2 b) {
  f32x2 r;
  asm("{\n\t.reg .b64 p, q, d;\n\tmov.b64 p, {%2, %3};\n\tmov.b64 q, {%4, %5};\n\t"
      "mul.rn.f32x2 d, p, q;\n\tmov.b64 {%0, %1}, d;\n\t}"
      : "=f"(r.x), "=f"(r.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return r;
}
__device__ __forceinline__ f32x2 add2(f32x2 a, f32x2 b) {
  f32x2 r;
  asm("{\n\t.reg .b64 p, q, d;\n\tmov.b64 p, {%2, %3};\n\tmov.b64 q, {%4, %5};\n\t"
      "add.rn.f32x2 d, p, q;\n\tmov.b64 {%0, %1}, d;\n\t}"
      : "=f"(r.x), "=f"(r.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return r;
}
__device__ __forceinline__ f32x2 sub2(f32x2 a, f32x2 b) {
  f32x2 r;
  asm("{\n\t.reg .b64 p, q, d;\n\tmov.b64 p, {%2, %3};\n\tmov.b64 q, {%4, %5};\n\t"
      "sub.rn.f32x2 d, p, q;\n\tmov.b64 {%0, %1}, d;\n\t}"
      : "=f"(r.x), "=f"(r.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return r;
}
__device__ __forceinline__ f32x2 fma2(f32x2 a, f32x2 b, f32x2 c) {
  f32x2 r;
  asm("{\n\t.reg .b64 p, q, s, d;\n\tmov.b64 p, {%2, %3};\n\tmov.b64 q, {%4, %5};\n\t"
      "mov.b64 s, {%6, %7};\n\tfma.rn.f32x2 d, p, q, s;\n\tmov.b64 {%0, %1}, d;\n\t}"
      : "=f"(r.x), "=f"(r.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return r;
}
// swiglu_f32 of two elements: the same operations in the same order, paired
__device__ __forceinline__ f32x2 swiglu_f32x2(f32x2 g, f32x2 u) {
  const f32x2 den = add2(f32x2{1.0f, 1.0f}, f32x2{__expf(-g.x), __expf(-g.y)});
  return mul2(f32x2{__fdividef(g.x, den.x), __fdividef(g.y, den.y)}, u);
}
// dswiglu_f32 of two elements: the same operations in the same order, paired
__device__ __forceinline__ void dswiglu_f32x2(f32x2 d, f32x2 g, f32x2 u, f32x2& dg, f32x2& du) {
  const f32x2 one{1.0f, 1.0f};
  const f32x2 den = add2(one, f32x2{__expf(-g.x), __expf(-g.y)});
  const f32x2 s{__fdividef(1.0f, den.x), __fdividef(1.0f, den.y)};
  const f32x2 t = fma2(g, sub2(one, s), one);
  dg = mul2(mul2(mul2(d, u), s), t);
  du = mul2(mul2(d, g), s);
}
__device__ __forceinline__ void dswiglu_bf16(float d, float g, float u, float& dg, float& du) {
  dswiglu_f32(d, g, u, dg, du);
  dg = round_bf16(dg);
  du = round_bf16(du);
}
// dswiglu_bf16 of elements i, i + 1 of d, g, u (paired)
__device__ __forceinline__ void dswiglu_bf16x2(const float* d, const float* g, const float* u, float* dg, float* du) {
  f32x2 a, b;
  dswiglu_f32x2(f32x2{d[0], d[1]}, f32x2{g[0], g[1]}, f32x2{u[0], u[1]}, a, b);
  dg[0] = round_bf16(a.x);
  dg[1] = round_bf16(a.y);
  du[0] = round_bf16(b.x);
  du[1] = round_bf16(b.y);
}

// ---------------------------------------------------------------------------
// Saturating round-to-nearest-even casts (PTX cvt .rn.satfinite). The first
// source operand of the x2 forms lands in the upper half of the result.

__device__ __forceinline__ uint32_t cvt_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}
__device__ __forceinline__ uint32_t cvt_e5m2x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e5m2x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}
// four values -> four codes in one word, element 0 in the low byte
template <int DT>
__device__ __forceinline__ uint32_t cvt_fp8x4(float a, float b, float c, float d) {
  if (DT == MGQ_E4M3) return cvt_e4m3x2(a, b) | (cvt_e4m3x2(c, d) << 16);
  return cvt_e5m2x2(a, b) | (cvt_e5m2x2(c, d) << 16);
}
// four values times m -> four codes in one word, element 0 in the low byte.
// The products are float32 round-to-nearest (packed f32x2 multiplies, the
// same IEEE rounding as four __fmul_rn), then cast like cvt_fp8x4.
template <int DT>
__device__ __forceinline__ uint32_t cvt_fp8x4_mul(float a, float b, float c, float d, float m) {
  uint32_t r;
  if (DT == MGQ_E4M3)
    asm("{\n\t.reg .b64 p, q, s;\n\t.reg .b32 a, b, c, d;\n\t.reg .b16 lo, hi;\n\t"
        "mov.b64 s, {%5, %5};\n\t"
        "mov.b64 p, {%1, %2};\n\tmul.rn.f32x2 p, p, s;\n\tmov.b64 {a, b}, p;\n\t"
        "mov.b64 q, {%3, %4};\n\tmul.rn.f32x2 q, q, s;\n\tmov.b64 {c, d}, q;\n\t"
        "cvt.rn.satfinite.e4m3x2.f32 lo, b, a;\n\tcvt.rn.satfinite.e4m3x2.f32 hi, d, c;\n\t"
        "mov.b32 %0, {lo, hi};\n\t}"
        : "=r"(r)
        : "r"(__float_as_uint(a)), "r"(__float_as_uint(b)), "r"(__float_as_uint(c)), "r"(__float_as_uint(d)),
          "r"(__float_as_uint(m)));
  else
    asm("{\n\t.reg .b64 p, q, s;\n\t.reg .b32 a, b, c, d;\n\t.reg .b16 lo, hi;\n\t"
        "mov.b64 s, {%5, %5};\n\t"
        "mov.b64 p, {%1, %2};\n\tmul.rn.f32x2 p, p, s;\n\tmov.b64 {a, b}, p;\n\t"
        "mov.b64 q, {%3, %4};\n\tmul.rn.f32x2 q, q, s;\n\tmov.b64 {c, d}, q;\n\t"
        "cvt.rn.satfinite.e5m2x2.f32 lo, b, a;\n\tcvt.rn.satfinite.e5m2x2.f32 hi, d, c;\n\t"
        "mov.b32 %0, {lo, hi};\n\t}"
        : "=r"(r)
        : "r"(__float_as_uint(a)), "r"(__float_as_uint(b)), "r"(__float_as_uint(c)), "r"(__float_as_uint(d)),
          "r"(__float_as_uint(m)));
  return r;
}
// four bf16 values (two packed pairs, element 0 in the low half of w0) times m
template <int DT>
__device__ __forceinline__ uint32_t cvt_fp8x4_bf16_mul(uint32_t w0, uint32_t w1, float m) {
  return cvt_fp8x4_mul<DT>(bf16_lo(w0), bf16_hi(w0), bf16_lo(w1), bf16_hi(w1), m);
}
// eight values times m -> one word of e2m1 codes, element 2i in the low nibble
// of byte i (float32 round-to-nearest products, packed f32x2 multiplies)
__device__ __forceinline__ uint32_t cvt_e2m1x8_mul(const float* v, float m) {
  uint32_t r;
  asm("{\n\t.reg .b64 p0, p1, p2, p3, s;\n\t.reg .b32 a<8>;\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "mov.b64 s, {%9, %9};\n\t"
      "mov.b64 p0, {%1, %2};\n\tmul.rn.f32x2 p0, p0, s;\n\tmov.b64 {a0, a1}, p0;\n\t"
      "mov.b64 p1, {%3, %4};\n\tmul.rn.f32x2 p1, p1, s;\n\tmov.b64 {a2, a3}, p1;\n\t"
      "mov.b64 p2, {%5, %6};\n\tmul.rn.f32x2 p2, p2, s;\n\tmov.b64 {a4, a5}, p2;\n\t"
      "mov.b64 p3, {%7, %8};\n\tmul.rn.f32x2 p3, p3, s;\n\tmov.b64 {a6, a7}, p3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b0, a1, a0;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b1, a3, a2;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b2, a5, a4;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b3, a7, a6;\n\t"
      "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
      : "=r"(r)
      : "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
        "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
        "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(m)));
  return r;
}
// eight e2m1 values -> one word, element 2i in the low nibble of byte i
__device__ __forceinline__ uint32_t cvt_e2m1x8(const float* v) {
  uint32_t r;
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
      "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
      : "=r"(r)
      : "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]));
  return r;
}
// one non-negative value -> ue4m3 code (e4m3 with the sign bit clear)
__device__ __forceinline__ uint32_t cvt_ue4m3(float x) { return cvt_e4m3x2(x, 0.0f) & 0xFFu; }
__device__ __forceinline__ float ue4m3_value(uint32_t code) {
  // exact decode: exponent field e (bias 7), mantissa m (3 bits)
  uint32_t e = (code >> 3) & 0xF, m = code & 7;
  if (e == 0) return (float)m * 0.001953125f;             // m * 2^-9
  return __uint_as_float(((e + 120u) << 23) | (m << 20));  // 2^(e-7) * (1 + m/8)
}

template <int DT> struct FmtInfo;
template <> struct FmtInfo<MGQ_E4M3> { static constexpr float fmax = 448.0f;   static constexpr int emax = 8; };
template <> struct FmtInfo<MGQ_E5M2> { static constexpr float fmax = 57344.0f; static constexpr int emax = 15; };

// ---------------------------------------------------------------------------
// E8M0 block-scale exponent from the float32 bits of a non-negative amax.
// rceil: smallest e with amax <= fmax * 2^e (fmax = 1.75 * 2^emax), i.e.
// floor(log2 amax) - emax, plus one when the significand exceeds 1.75.
// floor: floor(log2 amax) - emax. amax == 0 -> -127. Clamped to [-127, 127].
// Returns 128 for a NaN / infinite amax (scale code 0xFF).
__device__ __forceinline__ int mx_exponent(uint32_t amax_bits, int emax, bool rceil) {
  if (amax_bits >= 0x7F800000u) return 128;
  if (amax_bits == 0) return -127;
  int eb = (int)(amax_bits >> 23);
  uint32_t m = amax_bits & 0x7FFFFFu;
  int p;
  if (eb == 0) {                       // subnormal amax: normalise
    int lz = __clz(m) - 8;
    m = (m << lz) & 0x7FFFFFu;
    p = -126 - lz;
  } else {
    p = eb - 127;
  }
  int e = p - emax + ((rceil && m > 0x600000u) ? 1 : 0);
  return max(-127, min(127, e));
}
// 2^-e as a float32 multiplier (NaN for the NaN/inf marker)
__device__ __forceinline__ float mx_multiplier(int e) {
  if (e == 128) return __uint_as_float(0x7FC00000u);
  int b = 127 - e;                     // e in [-127, 126] -> normal float
  if (b >= 1) return __uint_as_float((uint32_t)b << 23);
  return 0x1p-127f;                    // e == 127 (unreachable for finite fp8 inputs)
}
__device__ __forceinline__ uint32_t mx_scale_code(int e) { return e == 128 ? 255u : (uint32_t)(e + 127); }

// Byte offset of the block scale of (row r, block b) in the 128x4-tiled
// layout, for a matrix whose row pitch holds `kblocks4` groups of 4 blocks.
__device__ __forceinline__ int64_t tiled_scale_offset(int64_t r, int64_t b, int64_t kblocks4) {
  return ((r >> 7) * kblocks4 + (b >> 2)) * 512 + (r & 31) * 16 + ((r >> 5) & 3) * 4 + (b & 3);
}

// |x| maximum of packed bf16 pairs as integers: NaN > inf > finite values
__device__ __forceinline__ uint32_t absmax_bf16x2(uint32_t acc, uint32_t w) {
  return __vmaxu2(acc, w & 0x7FFF7FFFu);
}
// running |x| maximum of packed bf16 pairs in the bf16 unit: the magnitude of
// each half is max(|acc|, |w|), a NaN operand gives NaN; the sign bits are
// garbage (clear them with absmax_bf16x2_final)
__device__ __forceinline__ uint32_t absmax_acc_bf16x2(uint32_t acc, uint32_t w) {
  uint32_t r;
  asm("max.NaN.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(acc), "r"(w));
  return r;
}
__device__ __forceinline__ uint32_t absmax_bf16x2_final(uint32_t acc) { return acc & 0x7FFF7FFFu; }
__device__ __forceinline__ uint32_t fold_bf16x2(uint32_t w) {   // max of the halves, as float bits
  uint32_t a = w & 0xFFFFu, b = w >> 16;
  return (a > b ? a : b) << 16;
}

__device__ __forceinline__ void atomic_max_nonneg(float* p, float v) {
  // valid for non-negative floats (and +NaN, which then sticks)
  atomicMax(reinterpret_cast<unsigned int*>(p), __float_as_uint(v));
}

}  // namespace mgq
