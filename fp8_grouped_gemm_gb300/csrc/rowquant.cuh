// Lane-level row-wise block quantiser shared by the fused elementwise kernels.
// A warp covers a 1024-element slice of one row; lane l owns the 32 elements
// [32 l, 32 l + 32), which is exactly one MX block (1x32) and a quarter of a
// 1x128 block. All 32 lanes must call quantize32 (it shuffles).
#pragma once
#include "device_common.cuh"

namespace mgq {

struct Block32 {
  uint32_t cw[8];   // 32 codes
  uint32_t s4;      // MX: the 4 scale bytes of lanes 4j..4j+3 (valid in lane 4j)
  float sinv;       // 1x128: float32 scale_inv of the 128-element block
};

__device__ __forceinline__ uint32_t absmax_bits_f32(const float* v, int n) {
  uint32_t m = 0;
  for (int i = 0; i < n; ++i) m = max(m, __float_as_uint(v[i]) & 0x7FFFFFFFu);
  return m;
}

// Blockwise (1x128, 128x1, 128x128) scale of a block from the float bits of its
// amax: s = max_finite / amax (IEEE division), 1 for an all-zero block, the
// largest float32 when the quotient overflows. The stored scale_inv is 1 / s.
template <int DT>
__device__ __forceinline__ float blk_scale(uint32_t amax_bits) {
  const float s = (amax_bits == 0) ? 1.0f : __fdiv_rn(FmtInfo<DT>::fmax, __uint_as_float(amax_bits));
  return isinf(s) ? 3.40282347e38f : s;
}

// v: the lane's 32 values; amax_bits: float bits of max |v| of this lane's
// 32 values; ts: per-tensor scale (MGQ_TENSOR_F32)
template <int SC, int DT>
__device__ __forceinline__ void quantize32(const float* v, uint32_t amax_bits, float ts, bool rceil, Block32& o) {
  float mult = ts;
  o.s4 = 0;
  o.sinv = 0.0f;
  if (SC == MGQ_MX32_E8M0) {
    const int e = mx_exponent(amax_bits, FmtInfo<DT>::emax, rceil);
    mult = mx_multiplier(e);
    const uint32_t sc = mx_scale_code(e);
    const uint32_t b1 = __shfl_down_sync(0xFFFFFFFFu, sc, 1);
    const uint32_t b2 = __shfl_down_sync(0xFFFFFFFFu, sc, 2);
    const uint32_t b3 = __shfl_down_sync(0xFFFFFFFFu, sc, 3);
    o.s4 = sc | (b1 << 8) | (b2 << 16) | (b3 << 24);
  } else if (SC == MGQ_BLK_1x128_F32) {
    uint32_t m = amax_bits;
    m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));
    m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 2));
    float s = (m == 0) ? 1.0f : __fdiv_rn(FmtInfo<DT>::fmax, __uint_as_float(m));
    if (isinf(s)) s = 3.40282347e38f;
    mult = s;
    o.sinv = __fdiv_rn(1.0f, s);
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) o.cw[i] = cvt_fp8x4_mul<DT>(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3], mult);
}

// Stores the lane's block of row r, columns [c, c + 32), of a matrix with row
// pitch ld (elements) and rows_cap rows (1x128 scales are k-block major).
template <int SC>
__device__ __forceinline__ void store32(const Block32& o, uint8_t* codes, uint8_t* scales, int64_t r, int64_t c,
                                        int64_t ld, int64_t rows_cap, uint32_t lane) {
  uint4* dst = reinterpret_cast<uint4*>(codes + r * ld + c);
  dst[0] = make_uint4(o.cw[0], o.cw[1], o.cw[2], o.cw[3]);
  dst[1] = make_uint4(o.cw[4], o.cw[5], o.cw[6], o.cw[7]);
  if (SC == MGQ_MX32_E8M0) {
    if ((lane & 3) == 0) *reinterpret_cast<uint32_t*>(scales + tiled_scale_offset(r, c / 32, ld / 128)) = o.s4;
  } else if (SC == MGQ_BLK_1x128_F32) {
    if ((lane & 3) == 0) reinterpret_cast<float*>(scales)[(c / 128) * rows_cap + r] = o.sinv;
  }
}

__device__ __forceinline__ void load_bf16x32(const uint16_t* src, float* v) {
  const uint4* p = reinterpret_cast<const uint4*>(src);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const uint4 w = __ldg(p + q);
    v[8 * q + 0] = bf16_lo(w.x); v[8 * q + 1] = bf16_hi(w.x);
    v[8 * q + 2] = bf16_lo(w.y); v[8 * q + 3] = bf16_hi(w.y);
    v[8 * q + 4] = bf16_lo(w.z); v[8 * q + 5] = bf16_hi(w.z);
    v[8 * q + 6] = bf16_lo(w.w); v[8 * q + 7] = bf16_hi(w.w);
  }
}

__device__ __forceinline__ void store_bf16x32(uint16_t* dst, const float* v) {
  uint4* p = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int q = 0; q < 4; ++q)
    p[q] = make_uint4(pack_bf16x2(v[8 * q], v[8 * q + 1]), pack_bf16x2(v[8 * q + 2], v[8 * q + 3]),
                      pack_bf16x2(v[8 * q + 4], v[8 * q + 5]), pack_bf16x2(v[8 * q + 6], v[8 * q + 7]));
}

__device__ __forceinline__ uint32_t warp_max_u32(uint32_t v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  return v;
}

}  // namespace mgq

namespace mgq {

// ---- NVFP4: e2m1 elements, ue4m3 scale per 16 elements, float32 global scale --

// s_g = 6 * 448 / amax of the tensor (float32 IEEE division); 1 for an
// all-zero tensor; the largest float32 on overflow.
__device__ __forceinline__ float nv_global_scale(float amax) {
  if (amax == 0.0f) return 1.0f;
  const float s = __fdiv_rn(2688.0f, amax);
  return isinf(s) ? 3.40282347e38f : s;
}

struct Block32nv {
  uint32_t cw[4];   // 32 e2m1 codes, element 2i in the low nibble of byte i
  uint32_t s4;      // the 4 ue4m3 scale bytes of lanes 2j, 2j+1 (valid in lane 2j)
};

// Lane's 32 elements = two 16-element blocks. Block scale code =
// ue4m3(float32(amax_b / 6) * s_g); with sc its value, r = s_g / sc (0 when
// sc is 0) and each element is e2m1(x * r). All 32 lanes must call it.
__device__ __forceinline__ void quantize32_nv(const float* v, float s_g, Block32nv& o) {
  uint32_t sc2 = 0;
#pragma unroll
  for (int blk = 0; blk < 2; ++blk) {
    const float* vb = v + 16 * blk;
    const float amax_b = __uint_as_float(absmax_bits_f32(vb, 16));
    const float t = __fmul_rn(__fdiv_rn(amax_b, 6.0f), s_g);
    const uint32_t code = cvt_ue4m3(t);
    const float sc = ue4m3_value(code);
    const float r = (sc == 0.0f) ? 0.0f : __fdiv_rn(s_g, sc);
    o.cw[2 * blk] = cvt_e2m1x8_mul(vb, r);
    o.cw[2 * blk + 1] = cvt_e2m1x8_mul(vb + 8, r);
    sc2 |= code << (8 * blk);
  }
  const uint32_t nb = __shfl_down_sync(0xFFFFFFFFu, sc2, 1);
  o.s4 = sc2 | (nb << 16);
}

// row r, elements [c, c + 32) of a matrix with `ld` elements per row (ld/2 bytes)
__device__ __forceinline__ void store32_nv(const Block32nv& o, uint8_t* codes, uint8_t* scales, int64_t r, int64_t c,
                                           int64_t ld, uint32_t lane) {
  *reinterpret_cast<uint4*>(codes + r * (ld / 2) + c / 2) = make_uint4(o.cw[0], o.cw[1], o.cw[2], o.cw[3]);
  if ((lane & 1) == 0) *reinterpret_cast<uint32_t*>(scales + tiled_scale_offset(r, c / 16, ld / 64)) = o.s4;
}

}  // namespace mgq
