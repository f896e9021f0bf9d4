// Row-wise and column-wise quantisation in one pass over 128 x 128 tiles.
//
// The backward GEMMs need every quantised activation and weight twice: blocks
// along the rows for one GEMM and along the columns (written transposed) for
// the other ("Numerical fix for moe single grouped weight with fp8 fp4
// primary weight and grad norm spikes", Megatron-LM PR #5487: rowwise and
// columnwise data and scales of one grouped tensor; "FP8BlockQuantizer not
// work on TE", TransformerEngine issue #2393: 128x1 backward blocks with the
// transpose done in shared memory, transpose(colwise(x)) = rowwise(x^T)).
//
// A CTA reads its tile once from its source functor (a plain bf16 matrix,
// SwiGLU of the gate/up output, or dSwiGLU), keeps the float values in shared
// memory, and writes
//   row-wise codes [rows, C] (blocks of 32 along C for MX), and
//   column-wise codes [C, M] per group of M rows (blocks of 32 along the rows),
// with per-tensor scales (the column copy is then the transposed cast) or
// E8M0 block scales in the 128x4-tiled layout.
#include "mgq_internal.h"
#include "rowquant.cuh"

namespace mgq {
namespace {

constexpr int TR = 128, TC = 128;  // tile rows x columns (per part)

// Source kinds (kKind):
//  kPlain    the tile is a block of a bf16 matrix (load_raw: 16-byte copies)
//  kGather   row r of the tile is a gathered bf16 row (row_offset), optionally
//            multiplied by a per-row float32 factor; the row offsets are
//            resolved once per tile into shared memory
//  kComputed the values are computed elementwise from kLoads bf16 operands
//            (fetch, then make), loads of several chunks in flight at once
// kExactBf16: every value the source produces is a bf16 value, so the tile
// keeps it as 2 bytes in shared memory.
enum SrcKind { kPlain, kGather, kComputed };

struct SrcPlain {
  static constexpr int kKind = kPlain;
  static constexpr int kParts = 1;
  static constexpr bool kExactBf16 = true;
  const uint16_t* x;
  int64_t ld;
  __device__ __forceinline__ uint4 load_raw(int64_t r, int64_t c) const {
    return __ldg(reinterpret_cast<const uint4*>(x + r * ld + c));
  }
};

__device__ __forceinline__ void unpack8_bf16(const uint4 w, float* v) {
  v[0] = bf16_lo(w.x); v[1] = bf16_hi(w.x); v[2] = bf16_lo(w.y); v[3] = bf16_hi(w.y);
  v[4] = bf16_lo(w.z); v[5] = bf16_hi(w.z); v[6] = bf16_lo(w.w); v[7] = bf16_hi(w.w);
}
__device__ __forceinline__ void store8_bf16(uint16_t* p, const float* v) {
  *reinterpret_cast<uint4*>(p) = make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]),
                                            pack_bf16x2(v[4], v[5]), pack_bf16x2(v[6], v[7]));
}

// h = bf16(silu(g) * u), g = gu[:, :F], u = gu[:, F:]; h optionally written out
struct SrcSwiglu {
  static constexpr int kKind = kComputed;
  static constexpr int kParts = 1;
  static constexpr bool kExactBf16 = true;
  static constexpr int kLoads = 2;
  const uint16_t* gu;
  int64_t F;
  uint16_t* h_out;
  __device__ __forceinline__ void fetch(int64_t r, int64_t c, uint4* w) const {
    w[0] = __ldg(reinterpret_cast<const uint4*>(gu + r * 2 * F + c));
    w[1] = __ldg(reinterpret_cast<const uint4*>(gu + r * 2 * F + F + c));
  }
  __device__ __forceinline__ void make(const uint4* w, int64_t r, int64_t c, bool valid, float* v, float*) const {
    float g[8], u[8];
    unpack8_bf16(w[0], g);
    unpack8_bf16(w[1], u);
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = swiglu_bf16(g[i], u[i]);
    if (h_out && valid) store8_bf16(h_out + r * F + c, v);
  }
};

// dSwiGLU: for ffn columns f..f+7 of row r, part 0 = dG = dh u s (1 + g (1 - s))
// and part 1 = dU = dh silu(g), s = sigmoid(g); both written to [dG | dU]
// (columns f and F + f) when requested. One read of dh, g, u serves both.
struct SrcDswiglu {
  static constexpr int kKind = kComputed;
  static constexpr int kParts = 2;
  static constexpr bool kExactBf16 = true;
  static constexpr int kLoads = 3;
  const uint16_t* dh;
  const uint16_t* gu;
  int64_t F;
  uint16_t* out;
  __device__ __forceinline__ void fetch(int64_t r, int64_t f, uint4* w) const {
    w[0] = __ldg(reinterpret_cast<const uint4*>(dh + r * F + f));
    w[1] = __ldg(reinterpret_cast<const uint4*>(gu + r * 2 * F + f));
    w[2] = __ldg(reinterpret_cast<const uint4*>(gu + r * 2 * F + F + f));
  }
  __device__ __forceinline__ void make(const uint4* w, int64_t r, int64_t f, bool valid, float* dg,
                                       float* du) const {
    float d[8], g[8], u[8];
    unpack8_bf16(w[0], d);
    unpack8_bf16(w[1], g);
    unpack8_bf16(w[2], u);
#pragma unroll
    for (int i = 0; i < 8; ++i) dswiglu_bf16(d[i], g[i], u[i], dg[i], du[i]);
    if (out && valid) {
      store8_bf16(out + r * 2 * F + f, dg);
      store8_bf16(out + r * 2 * F + F + f, du);
    }
  }
};

// row r of the permuted matrix: X[t] for the (token, slot) entry e = src_row[r]
// (t = e / k), zeros for filler rows
struct SrcGatherX {
  static constexpr int kKind = kGather;
  static constexpr int kParts = 1;
  static constexpr bool kExactBf16 = true;
  const uint16_t* x;
  const int32_t* src_row;
  int k;
  int64_t H;
  // element offset of the source row of r (-1: zero row) and its factor
  __device__ __forceinline__ int64_t row_offset(int64_t r, float&) const {
    const int e = src_row[r];
    return e < 0 ? -1 : (int64_t)(e / k) * H;
  }
  __device__ __forceinline__ const uint16_t* base() const { return x; }
};

// row r of dY = float32(probs[e] * dout[t]) for the entry e = src_row[r]
// (the unpermute backward), zeros for filler rows
struct SrcGatherDy {
  static constexpr int kKind = kGather;
  static constexpr int kParts = 1;
  static constexpr bool kExactBf16 = false;   // float32 products
  const uint16_t* dout;
  const float* probs;
  const int32_t* src_row;
  int k;
  int64_t H;
  __device__ __forceinline__ int64_t row_offset(int64_t r, float& p) const {
    const int e = src_row[r];
    if (e < 0) return -1;
    p = probs[e];
    return (int64_t)(e / k) * H;
  }
  __device__ __forceinline__ const uint16_t* base() const { return dout; }
};

struct RowColArgs {
  int64_t rows_cap;          // rows of the row-wise output
  const int32_t* rows_used;  // device row count or null (= rows_cap)
  int64_t C;                 // columns of the output rows
  int64_t part_off;          // column offset of part 1 (two-part sources)
  int64_t M;                 // rows per group (column-wise output [G][C][M])
  uint8_t* row_codes;        // [rows, C]
  uint8_t* row_scales;       // MX: tiled over [rows, C]
  uint8_t* col_codes;        // [G][C][M] or null
  uint8_t* col_scales;       // MX: tiled over [G*C, M]
  const float* tensor_scale; // per group (TENSOR)
  float* amax_out;           // per group, optional
  int rceil;
};

// shared-memory tile element: bf16 bits (exact sources) or float
template <bool B16> struct TileT;
template <> struct TileT<true> {
  using T = uint16_t;
  static constexpr int kPad = 8;             // rows stay 16-byte aligned
  __device__ static T put(float v) { return (T)(__float_as_uint(v) >> 16); }
  __device__ static float get(T v) { return __uint_as_float((uint32_t)v << 16); }
};
template <> struct TileT<false> {
  using T = float;
  static constexpr int kPad = 4;             // rows stay 16-byte aligned
  __device__ static T put(float v) { return v; }
  __device__ static float get(T v) { return v; }
};

template <class Src>
constexpr size_t rowcol_smem() {
  return (size_t)Src::kParts * TR * (TC + TileT<Src::kExactBf16>::kPad) * sizeof(typename TileT<Src::kExactBf16>::T);
}

template <class Src, int SC, int DT>
__global__ void __launch_bounds__(256, (Src::kParts == 2 || !Src::kExactBf16) ? 3 : 4)
    quant_rowcol_kernel(const Src src, const RowColArgs a) {
  using TT = TileT<Src::kExactBf16>;
  using T = typename TT::T;
  constexpr int P = Src::kParts;
  constexpr int LD = TC + TT::kPad;
  extern __shared__ uint8_t smem_raw[];
  T* tile = reinterpret_cast<T*>(smem_raw);                 // [P][TR][LD]
  __shared__ uint32_t s_amax[8];
  const int tid = threadIdx.x, warp = tid >> 5;
  const uint32_t lane = tid & 31;
  const int64_t c0 = (int64_t)blockIdx.x * TC, r0 = (int64_t)blockIdx.y * TR;
  const int64_t nrows = a.rows_used ? (int64_t)*a.rows_used : a.rows_cap;
  if (r0 >= nrows) return;
  const int64_t g = r0 / a.M;
  const float ts = (SC == MGQ_TENSOR_F32) ? a.tensor_scale[g] : 1.0f;
  // ---- load: TR rows x 16 chunks of 8 columns, 8 chunks per thread
  uint32_t am = 0;
  if constexpr (Src::kKind == kPlain || Src::kKind == kGather) {
    // gathered rows: the source offsets (and factors) of the tile's rows first
    __shared__ int64_t s_off[Src::kKind == kGather ? TR : 1];
    __shared__ float s_fac[Src::kKind == kGather ? TR : 1];
    if constexpr (Src::kKind == kGather) {
      if (tid < TR) {
        float f = 0.0f;
        const int64_t off = (r0 + tid < nrows) ? src.row_offset(r0 + tid, f) : -1;
        s_off[tid] = off;
        s_fac[tid] = f;
      }
      __syncthreads();
    }
    // all eight 16-byte loads in flight, then copied into the tile
    uint4 w[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int chunk = tid + 256 * i;
      const int rr = chunk >> 4, cc = (chunk & 15) * 8;
      if constexpr (Src::kKind == kGather) {
        const int64_t off = s_off[rr];
        w[i] = off >= 0 ? __ldg(reinterpret_cast<const uint4*>(src.base() + off + c0 + cc)) : make_uint4(0, 0, 0, 0);
      } else {
        w[i] = (r0 + rr < nrows) ? src.load_raw(r0 + rr, c0 + cc) : make_uint4(0, 0, 0, 0);
      }
    }
    if constexpr (Src::kExactBf16) {
      uint32_t am2 = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int chunk = tid + 256 * i;
        const int rr = chunk >> 4, cc = (chunk & 15) * 8;
        am2 = absmax_bf16x2(absmax_bf16x2(absmax_bf16x2(absmax_bf16x2(am2, w[i].x), w[i].y), w[i].z), w[i].w);
        *reinterpret_cast<uint4*>(&tile[rr * LD + cc]) = w[i];
      }
      am = fold_bf16x2(am2);
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int chunk = tid + 256 * i;
        const int rr = chunk >> 4, cc = (chunk & 15) * 8;
        const float f = Src::kKind == kGather ? s_fac[rr] : 1.0f;
        float v[8];
        unpack8_bf16(w[i], v);
#pragma unroll
        for (int j = 0; j < 8; ++j) v[j] = __fmul_rn(f, v[j]);
        am = max(am, absmax_bits_f32(v, 8));
        float4* d = reinterpret_cast<float4*>(&tile[rr * LD + cc]);
        d[0] = make_float4(v[0], v[1], v[2], v[3]);
        d[1] = make_float4(v[4], v[5], v[6], v[7]);
      }
    }
  } else {
    // computed values: the operands of kBatch chunks loaded together
    constexpr int kBatch = 4;
#pragma unroll 1
    for (int b = 0; b < 8; b += kBatch) {
      uint4 w[kBatch][Src::kLoads];
#pragma unroll
      for (int j = 0; j < kBatch; ++j) {
        const int chunk = tid + 256 * (b + j);
        const int rr = chunk >> 4, cc = (chunk & 15) * 8;
        if (r0 + rr < nrows) {
          src.fetch(r0 + rr, c0 + cc, w[j]);
        } else {
#pragma unroll
          for (int l = 0; l < Src::kLoads; ++l) w[j][l] = make_uint4(0, 0, 0, 0);
        }
      }
#pragma unroll
      for (int j = 0; j < kBatch; ++j) {
        const int chunk = tid + 256 * (b + j);
        const int rr = chunk >> 4, cc = (chunk & 15) * 8;
        float v[P][8];
        src.make(w[j], r0 + rr, c0 + cc, r0 + rr < nrows, v[0], v[P - 1]);
#pragma unroll
        for (int p = 0; p < P; ++p) {
          am = max(am, absmax_bits_f32(v[p], 8));
#pragma unroll
          for (int q = 0; q < 8; ++q) tile[(p * TR + rr) * LD + cc + q] = TT::put(v[p][q]);
        }
      }
    }
  }
  __syncthreads();
  // ---- row-wise: the P*TR (part, row) pairs, 4 per warp at a time; 8 lanes
  // per row, lane takes 16 columns (half an MX block: the pair l, l^1 shares one)
  {
    const int seg = lane & 7;
    for (int pr0 = warp * P * 16; a.row_codes && pr0 < (warp + 1) * P * 16; pr0 += 4) {
      const int pr = pr0 + (int)(lane >> 3);
      const int p = pr / TR, rr = pr % TR;
      const int64_t r = r0 + rr;
      const int64_t cb = c0 + p * a.part_off;     // first output column of this part
      float v[16];
      uint32_t m = 0;   // |v| maximum as float bits (MX)
      const T* src = &tile[(p * TR + rr) * LD + 16 * seg];
      if constexpr (Src::kExactBf16) {
        const uint4 w0 = reinterpret_cast<const uint4*>(src)[0], w1 = reinterpret_cast<const uint4*>(src)[1];
        const uint32_t ww[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
        uint32_t m2 = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          v[2 * i] = bf16_lo(ww[i]);
          v[2 * i + 1] = bf16_hi(ww[i]);
          m2 = absmax_bf16x2(m2, ww[i]);
        }
        m = fold_bf16x2(m2);
      } else {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float4 f = reinterpret_cast<const float4*>(src)[q];
          v[4 * q] = f.x; v[4 * q + 1] = f.y; v[4 * q + 2] = f.z; v[4 * q + 3] = f.w;
        }
        if (SC == MGQ_MX32_E8M0) m = absmax_bits_f32(v, 16);
      }
      float mult = ts;
      uint32_t scode = 0;
      if (SC == MGQ_MX32_E8M0) {
        m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));        // the other half of the block
        const int e = mx_exponent(m, FmtInfo<DT>::emax, a.rceil != 0);
        mult = mx_multiplier(e);
        scode = mx_scale_code(e);
      }
      uint32_t cw[4];
#pragma unroll
      for (int i = 0; i < 4; ++i)
        cw[i] = cvt_fp8x4<DT>(__fmul_rn(v[4 * i], mult), __fmul_rn(v[4 * i + 1], mult),
                              __fmul_rn(v[4 * i + 2], mult), __fmul_rn(v[4 * i + 3], mult));
      if (SC == MGQ_MX32_E8M0) {
        // the row's 4 block scales (lanes seg 0, 2, 4, 6 of its 8) into seg 0
        const uint32_t s1 = __shfl_down_sync(0xFFFFFFFFu, scode, 2), s2 = __shfl_down_sync(0xFFFFFFFFu, scode, 4),
                       s3 = __shfl_down_sync(0xFFFFFFFFu, scode, 6);
        if (seg == 0 && r < nrows)
          *reinterpret_cast<uint32_t*>(a.row_scales + tiled_scale_offset(r, cb / 32, a.C / 128)) =
              scode | (s1 << 8) | (s2 << 16) | (s3 << 24);
      }
      if (r < nrows)
        *reinterpret_cast<uint4*>(a.row_codes + r * a.C + cb + 16 * seg) = make_uint4(cw[0], cw[1], cw[2], cw[3]);
    }
  }
  // ---- column-wise: thread takes 2 adjacent columns of one 32-row block (one
  // MX block each); its 32 output bytes per column are contiguous
  if (a.col_codes) {
    const int cp = tid & 63, rb = (tid >> 6) & 3;
#pragma unroll 1
    for (int p = 0; p < P; ++p) {
      const int cc = 2 * cp;
      const int64_t crow = g * a.C + c0 + p * a.part_off + cc;  // row of the column-wise output
      const int64_t rg = r0 - g * a.M + 32 * rb;                // row inside the group
      // the two columns' 32 values: bf16 pairs (exact sources) or floats
      uint32_t w[32];
      float v0[Src::kExactBf16 ? 1 : 32], v1[Src::kExactBf16 ? 1 : 32];
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const T* src = &tile[(p * TR + 32 * rb + i) * LD + cc];
        if constexpr (Src::kExactBf16) {
          w[i] = *reinterpret_cast<const uint32_t*>(src);
        } else {
          const float2 f = *reinterpret_cast<const float2*>(src);
          v0[i] = f.x;
          v1[i] = f.y;
        }
      }
      uint32_t amh[2];
      if constexpr (Src::kExactBf16) {
        uint32_t m2 = 0;
#pragma unroll
        for (int i = 0; i < 32; ++i) m2 = absmax_bf16x2(m2, w[i]);
        amh[0] = m2 << 16;
        amh[1] = m2 & 0xFFFF0000u;
      } else {
        amh[0] = absmax_bits_f32(v0, 32);
        amh[1] = absmax_bits_f32(v1, 32);
      }
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        auto val = [&](int i) {
          if constexpr (Src::kExactBf16) return h ? bf16_hi(w[i]) : bf16_lo(w[i]);
          else return h ? v1[i] : v0[i];
        };
        float mult = ts;
        if (SC == MGQ_MX32_E8M0) {
          const int e = mx_exponent(amh[h], FmtInfo<DT>::emax, a.rceil != 0);
          mult = mx_multiplier(e);
          a.col_scales[tiled_scale_offset(crow + h, rg / 32, a.M / 128)] = (uint8_t)mx_scale_code(e);
        }
        uint32_t cw[8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
          cw[i] = cvt_fp8x4<DT>(__fmul_rn(val(4 * i), mult), __fmul_rn(val(4 * i + 1), mult),
                                __fmul_rn(val(4 * i + 2), mult), __fmul_rn(val(4 * i + 3), mult));
        uint4* dst = reinterpret_cast<uint4*>(a.col_codes + (crow + h) * a.M + rg);
        dst[0] = make_uint4(cw[0], cw[1], cw[2], cw[3]);
        dst[1] = make_uint4(cw[4], cw[5], cw[6], cw[7]);
      }
    }
  }
  if (SC == MGQ_TENSOR_F32 && a.amax_out) {
    am = warp_max_u32(am);
    if (lane == 0) s_amax[warp] = am;
    __syncthreads();
    if (tid == 0) {
      for (int i = 1; i < 8; ++i) am = max(am, s_amax[i]);
      atomic_max_nonneg(a.amax_out + g, __uint_as_float(am));
    }
  }
}

template <class Src, int SC, int DT>
int launch_rowcol_t(const Src& src, const RowColArgs& a, dim3 grid, cudaStream_t s) {
  constexpr size_t smem = rowcol_smem<Src>();
  auto kern = quant_rowcol_kernel<Src, SC, DT>;
  static bool attr_set[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (smem > 48 * 1024 && dev < 64 && !attr_set[dev]) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
      return MGQ_ERR_CUDA;
    attr_set[dev] = true;
  }
  kern<<<grid, 256, smem, s>>>(src, a);
  MGQ_LAUNCH_CHECK();
  return MGQ_OK;
}

template <class Src>
int launch_rowcol(const Src& src, const mgq_qdesc* q, RowColArgs a, cudaStream_t s) {
  const dim3 grid((unsigned)(a.C / Src::kParts / TC), (unsigned)((a.rows_cap + TR - 1) / TR));
  const int sc = q->scaling, dt = q->dtype;
  if (sc == MGQ_MX32_E8M0 && dt == MGQ_E4M3) return launch_rowcol_t<Src, MGQ_MX32_E8M0, MGQ_E4M3>(src, a, grid, s);
  if (sc == MGQ_MX32_E8M0 && dt == MGQ_E5M2) return launch_rowcol_t<Src, MGQ_MX32_E8M0, MGQ_E5M2>(src, a, grid, s);
  // per-tensor column copies of gathered rows are transposed casts of the row codes
  if constexpr (Src::kKind == kGather) {
    return MGQ_ERR_UNSUPPORTED;
  } else {
    if (sc == MGQ_TENSOR_F32 && dt == MGQ_E4M3) return launch_rowcol_t<Src, MGQ_TENSOR_F32, MGQ_E4M3>(src, a, grid, s);
    if (sc == MGQ_TENSOR_F32 && dt == MGQ_E5M2) return launch_rowcol_t<Src, MGQ_TENSOR_F32, MGQ_E5M2>(src, a, grid, s);
    return MGQ_ERR_UNSUPPORTED;
  }
}

RowColArgs make_args(const mgq_qdesc* q, int64_t rows_cap, const int32_t* rows_used, int64_t C, int64_t M,
                     int64_t part_off = 0) {
  RowColArgs a;
  a.rows_cap = rows_cap;
  a.rows_used = rows_used;
  a.C = C;
  a.part_off = part_off;
  a.M = M;
  a.row_codes = static_cast<uint8_t*>(q->row.data);
  a.row_scales = static_cast<uint8_t*>(q->row.scale);
  a.col_codes = static_cast<uint8_t*>(q->col.data);
  a.col_scales = static_cast<uint8_t*>(q->col.scale);
  a.tensor_scale = q->tensor_scale;
  a.amax_out = q->amax_out;
  a.rceil = q->e8m0_mode == MGQ_E8M0_RCEIL;
  return a;
}

}  // namespace

int rowcol_plain(const uint16_t* x, int64_t G, int64_t M, int64_t K, const mgq_qdesc* q, cudaStream_t s) {
  return launch_rowcol(SrcPlain{x, K}, q, make_args(q, G * M, nullptr, K, M), s);
}

int rowcol_swiglu(const uint16_t* gu, int64_t R_cap, int64_t F, const int32_t* rows_used, uint16_t* h_out,
                  const mgq_qdesc* q, cudaStream_t s) {
  return launch_rowcol(SrcSwiglu{gu, F, h_out}, q, make_args(q, R_cap, rows_used, F, R_cap), s);
}

int rowcol_dswiglu(const uint16_t* dh, const uint16_t* gu, int64_t R_cap, int64_t F, const int32_t* rows_used,
                   uint16_t* out, const mgq_qdesc* q, cudaStream_t s) {
  return launch_rowcol(SrcDswiglu{dh, gu, F, out}, q, make_args(q, R_cap, rows_used, 2 * F, R_cap, F), s);
}

int gather_x_rowcol(const uint16_t* x, const int32_t* src_row, int k, int64_t H, int64_t R_cap,
                    const int32_t* rows_used, bool with_rows, const mgq_qdesc* q, cudaStream_t s) {
  RowColArgs a = make_args(q, R_cap, rows_used, H, R_cap);
  if (!with_rows) a.row_codes = nullptr;   // the row-wise codes come from the permute kernel
  return launch_rowcol(SrcGatherX{x, src_row, k, H}, q, a, s);
}

int col_gather_dy(const uint16_t* dout, const float* probs, const int32_t* src_row, int k, int64_t H, int64_t R_cap,
                  const int32_t* rows_used, const mgq_qdesc* q, cudaStream_t s) {
  RowColArgs a = make_args(q, R_cap, rows_used, H, R_cap);
  a.row_codes = nullptr;       // the row-wise codes come from the unpermute-backward kernel
  return launch_rowcol(SrcGatherDy{dout, probs, src_row, k, H}, q, a, s);
}

}  // namespace mgq
