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
// A tile is read once from its source (a plain bf16 matrix, SwiGLU of the
// gate/up output, dSwiGLU, or rows gathered through the routing), held as bf16
// in shared memory, and written as
//   row-wise codes [rows, C] (MX blocks of 32 along C, NVFP4 blocks of 16,
//   blockwise 1x128 blocks), and
//   column-wise codes [C, M] per group of M rows (blocks along the rows: MX 32,
//   NVFP4 16, blockwise 128x1),
// with per-tensor scales (the column copy is then the transposed cast), E8M0
// block scales or NVFP4 ue4m3 block scales with s_g from an amax pre-pass (both
// in the 128x4-tiled scale layout), or blockwise float32 scale_inv stored
// block-major: row-wise [C/128][rows], column-wise [M/128][G*C]. Weights with
// 128x128 tiles (one scale per tile) get both copies from one pass, the
// column-wise copy the transposed codes with the transposed tile scales
// ([G][M/128][C/128] and [G][C/128][M/128]).
// Kernels: quant_rowcol_kernel (one tile per CTA: plain sources, SwiGLU, and
// dSwiGLU with blockwise 128x1 blocks), quant_rowcol_pipe_kernel (dSwiGLU with
// MX or per-tensor scaling: a persistent CTA whose operands arrive by TMA in
// half tiles while it quantises the previous tile), quant_rowcol_stream_kernel
// (gathered rows: a CTA walks a range of tiles and stages the next with
// cp.async; the FP8 column codes of dY = probs * dout go out through a staged
// tile and one TMA store per item), quant_nv2d_kernel (NVFP4 weights with 16x16
// blocks: both copies share the block scales). Tiles are XOR-swizzled (tix).
#include "mgq_internal.h"
#include "ptx_sm100.cuh"
#include "rowquant.cuh"

#include <algorithm>
#include <cstring>
#include <type_traits>

namespace mgq {
namespace {

constexpr int TR = 128, TC = 128;  // tile rows x columns (per part)
constexpr int LD = TC + 8;          // bf16 tile row pitch in elements (rows stay 16-byte aligned)
constexpr int kStgBytes = TC * TR;  // one part's staged column codes (FP8): 128 rows of 128 bytes

// Tile layout: element (row, col) of a bf16 tile [rows][LD] sits in 16-byte
// unit (col / 8) ^ sw(row) of its row, sw(row) = 2 * ((row / 32) % 4). With
// the padded pitch alone, lanes reading one column in the four 32-row blocks
// hit the same bank; the swizzle moves the blocks 0, 32, 64 and 96 bytes apart,
// so the column reads are conflict-free whichever lanes share an instruction.
// Row reads and the 16-byte tile writes stay conflict-free (a row's units are
// only permuted).
__device__ __forceinline__ int tile_sw(int row) { return (row >> 4) & 6; }
// element offset of (row, col); col a multiple of 8 for a 16-byte unit
__device__ __forceinline__ int tix(int row, int col) {
  return row * LD + ((((col >> 3) ^ tile_sw(row))) << 3) + (col & 7);
}

// Staged column-wise codes (FP8 kinds, gathered sources): the CTA's writes to the staging tiles
// become visible to the TMA unit, then one thread stores each part's tile
// ([128 output rows][128 bytes] at output row y0 + p * part_off, byte x0).
template <int P>
__device__ __forceinline__ void store_col_tiles(const CUtensorMap* tm, const uint8_t* stg, int32_t x0, int32_t y0,
                                                int64_t part_off, int tid) {
  ptx::fence_proxy_async_smem();
  __syncthreads();
  if (tid == 0) {
#pragma unroll
    for (int p = 0; p < P; ++p) ptx::tma_store_2d(tm, stg + p * kStgBytes, x0, y0 + (int32_t)(p * part_off));
    ptx::bulk_commit();
  }
}
// before the staging tiles are written again: the previous stores have read them
__device__ __forceinline__ void wait_col_tiles(int tid) {
  if (tid == 0) ptx::bulk_wait_read0();
  __syncthreads();
}

// Sources. Every value a source produces is a bf16 value, or (kFactor) a bf16
// value times a per-row float32 factor, so tiles hold bf16 in shared memory.
//  plain (SrcPlain): a block of a bf16 matrix, one tile per CTA
//  streamed (SrcGatherX, SrcGatherDy, kStream): row r of the tile is the bf16
//    row at element offset row_offset(r) of base() (-1: a zero row); these run
//    on the pipelined kernel, which stages tiles with cp.async
//  computed (SrcSwiglu, SrcDswiglu): values computed elementwise from kLoads
//    bf16 operands (fetch, then make), loads of several chunks in flight
struct SrcPlain {
  static constexpr bool kComputed = false;
  static constexpr bool kFactor = false;
  static constexpr bool kStream = false;      // one tile per CTA (4 CTAs per SM) is faster for dense rows
  static constexpr int kParts = 1;
  const uint16_t* x;
  int64_t ld;
};

__device__ __forceinline__ void unpack8_bf16(const uint4 w, float* v) {
  v[0] = bf16_lo(w.x); v[1] = bf16_hi(w.x); v[2] = bf16_lo(w.y); v[3] = bf16_hi(w.y);
  v[4] = bf16_lo(w.z); v[5] = bf16_hi(w.z); v[6] = bf16_lo(w.w); v[7] = bf16_hi(w.w);
}

// h = bf16(silu(g) * u), g = gu[:, :F], u = gu[:, F:]; h optionally written out
struct SrcSwiglu {
  static constexpr bool kComputed = true;
  static constexpr bool kFactor = false;
  static constexpr bool kStream = false;
  static constexpr int kParts = 1;
  static constexpr int kLoads = 2;
  const uint16_t* gu;
  int64_t F;
  uint16_t* h_out;
  __device__ __forceinline__ void fetch(int64_t r, int64_t c, uint4* w) const {
    w[0] = __ldg(reinterpret_cast<const uint4*>(gu + r * 2 * F + c));
    w[1] = __ldg(reinterpret_cast<const uint4*>(gu + r * 2 * F + F + c));
  }
  // out[0]: the 8 values of h as packed bf16
  __device__ __forceinline__ void make(const uint4* w, int64_t r, int64_t c, bool valid, uint4* out) const {
    float g[8], u[8];
    unpack8_bf16(w[0], g);
    unpack8_bf16(w[1], u);
    uint32_t hw[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
      hw[i] = pack_bf16x2x2(swiglu_f32x2(f32x2{g[2 * i], g[2 * i + 1]}, f32x2{u[2 * i], u[2 * i + 1]}));
    out[0] = make_uint4(hw[0], hw[1], hw[2], hw[3]);
    if (h_out && valid) *reinterpret_cast<uint4*>(h_out + r * F + c) = out[0];
  }
};

// dSwiGLU: for ffn columns f..f+7 of row r, part 0 = dG = dh u s (1 + g (1 - s))
// and part 1 = dU = dh silu(g), s = sigmoid(g); both written to [dG | dU]
// (columns f and F + f) when requested. One read of dh, g, u serves both.
struct SrcDswiglu {
  static constexpr bool kComputed = true;
  static constexpr bool kFactor = false;
  static constexpr bool kStream = false;
  static constexpr int kParts = 2;
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
  // o[0], o[1]: the 8 values of dG and of dU as packed bf16
  __device__ __forceinline__ void make(const uint4* w, int64_t r, int64_t f, bool valid, uint4* o) const {
    float d[8], g[8], u[8], dg[8], du[8];
    unpack8_bf16(w[0], d);
    unpack8_bf16(w[1], g);
    unpack8_bf16(w[2], u);
#pragma unroll
    for (int i = 0; i < 8; i += 2) {
      f32x2 a, b;
      dswiglu_f32x2(f32x2{d[i], d[i + 1]}, f32x2{g[i], g[i + 1]}, f32x2{u[i], u[i + 1]}, a, b);
      dg[i] = a.x;
      dg[i + 1] = a.y;
      du[i] = b.x;
      du[i + 1] = b.y;
    }
    o[0] = make_uint4(pack_bf16x2(dg[0], dg[1]), pack_bf16x2(dg[2], dg[3]), pack_bf16x2(dg[4], dg[5]),
                      pack_bf16x2(dg[6], dg[7]));
    o[1] = make_uint4(pack_bf16x2(du[0], du[1]), pack_bf16x2(du[2], du[3]), pack_bf16x2(du[4], du[5]),
                      pack_bf16x2(du[6], du[7]));
    if (out && valid) {
      *reinterpret_cast<uint4*>(out + r * 2 * F + f) = o[0];
      *reinterpret_cast<uint4*>(out + r * 2 * F + F + f) = o[1];
    }
  }
};

// row r of the permuted matrix: X[t] for the (token, slot) entry e = src_row[r]
// (t = e / k), zeros for filler rows
struct SrcGatherX {
  static constexpr bool kStream = true;
  static constexpr bool kComputed = false;
  static constexpr int kParts = 1;
  static constexpr bool kFactor = false;
  static constexpr bool kColumnsOnly = false;
  const uint16_t* x;
  const int32_t* src_row;
  int k;
  int64_t H;
  __device__ __forceinline__ int64_t row_offset(int64_t r, float&) const {
    const int e = src_row[r];
    return e < 0 ? -1 : (int64_t)(e / k) * H;
  }
  __device__ __forceinline__ const uint16_t* base() const { return x; }
};

// row r of dY = float32(probs[e] * dout[t]) for the entry e = src_row[r]
// (the unpermute backward), zeros for filler rows; column-wise codes only
// (the row-wise codes come from the token-major kernel)
struct SrcGatherDy {
  static constexpr bool kStream = true;
  static constexpr bool kComputed = false;
  static constexpr int kParts = 1;
  static constexpr bool kFactor = true;
  static constexpr bool kColumnsOnly = true;
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
  float* amax_out;           // per group: TENSOR optional output; NVFP4 the pre-pass amax (input)
  float* s_out;              // NVFP4: s_g per group (output)
  int rceil;
  int col_tma;               // FP8 column copies: staged in shared memory, one TMA store per tile and part
  int* err;                  // device error word (a wait that ran out of time)
  uint64_t wait_ns;          // limit of every mbarrier wait
};

// ---- the quantisation of one tile (shared by both kernels) -----------------

// One NVFP4 block of 16 values: scale code =
// ue4m3(float32(amax_b / 6) * s_g); with sc its value, r = s_g / sc (0 when sc
// is 0) and each element is e2m1(v * r). Returns the scale code.
__device__ __forceinline__ uint32_t nv_block16(float* v, float amax_b, float s_g, uint2& codes) {
  const float t = __fmul_rn(__fdiv_rn(amax_b, 6.0f), s_g);
  const uint32_t code = cvt_ue4m3(t);
  const float sc = ue4m3_value(code);
  const float r = (sc == 0.0f) ? 0.0f : __fdiv_rn(s_g, sc);
  codes = make_uint2(cvt_e2m1x8_mul(v, r), cvt_e2m1x8_mul(v + 8, r));
  return code;
}

// one column-wise block: the 32 values of output row crow, rows rg..rg+31 of
// its group (amax_bits: float bits of their |v| maximum, MX)
// stg (FP8, when staging): this part's staging tile [128 tile columns][128
// tile rows] of code bytes in the 128-byte-swizzled layout a TMA store reads
// (16-byte chunk k of row c at chunk k ^ (c & 7)); cl: the tile column, rl:
// the block's first tile row
template <int SC, int DT>
__device__ __forceinline__ void col_block_out(float* v, uint32_t amax_bits, float ts, const RowColArgs& a,
                                              int64_t crow, int64_t rg, uint8_t* stg = nullptr, int cl = 0,
                                              int rl = 0) {
  if constexpr (SC == MGQ_NV16_UE4M3) {
    // two 16-row blocks, e2m1 packed along the rows; ts is s_g
    uint2 c0, c1;
    const uint32_t s0 = nv_block16(v, __uint_as_float(absmax_bits_f32(v, 16)), ts, c0);
    const uint32_t s1 = nv_block16(v + 16, __uint_as_float(absmax_bits_f32(v + 16, 16)), ts, c1);
    *reinterpret_cast<uint4*>(a.col_codes + crow * (a.M / 2) + rg / 2) = make_uint4(c0.x, c0.y, c1.x, c1.y);
    *reinterpret_cast<uint16_t*>(a.col_scales + tiled_scale_offset(crow, rg / 16, a.M / 64)) =
        (uint16_t)(s0 | (s1 << 8));
  } else {
    float mult = ts;
    if constexpr (SC == MGQ_MX32_E8M0) {
      const int e = mx_exponent(amax_bits, FmtInfo<DT>::emax, a.rceil != 0);
      mult = mx_multiplier(e);
      a.col_scales[tiled_scale_offset(crow, rg / 32, a.M / 128)] = (uint8_t)mx_scale_code(e);
    }
    uint32_t cw[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) cw[i] = cvt_fp8x4_mul<DT>(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3], mult);
    if (stg) {
      uint4* row = reinterpret_cast<uint4*>(stg + cl * 128);
      const int k0 = rl / 16;
      row[k0 ^ (cl & 7)] = make_uint4(cw[0], cw[1], cw[2], cw[3]);
      row[(k0 + 1) ^ (cl & 7)] = make_uint4(cw[4], cw[5], cw[6], cw[7]);
    } else {
      uint4* dst = reinterpret_cast<uint4*>(a.col_codes + crow * a.M + rg);
      dst[0] = make_uint4(cw[0], cw[1], cw[2], cw[3]);
      dst[1] = make_uint4(cw[4], cw[5], cw[6], cw[7]);
    }
  }
}

// Row-wise codes of a bf16 tile [P][TR][LD]: the P*TR (part, row) pairs, 8 per
// warp at a time; 4 lanes per row, lane takes one 32-column block. The lane
// reads its four 16-byte chunks in the order q ^ sw (sw = 0 for blocks 0, 1 and
// 2 for blocks 2, 3), so the 8 lanes of a quarter warp hit 8 different bank groups.
// srow (gathered sources): the tile rows' source offsets, negative for filler
// rows, whose blockwise scale_inv is written as 0 like their codes (zero
// codes and zero scales for padding)
template <int P, int SC, int DT, int RPW = P * 16>
__device__ __forceinline__ void row_phase(const uint16_t* tile, int64_t r0, int64_t nrows, int64_t c0, float ts,
                                          const RowColArgs& a, int warp, uint32_t lane,
                                          const int64_t* srow = nullptr) {
  // RPW: (part, row) pairs per warp (P * TR over the CTA's warps)
  const int seg = lane & 3;
  const int sw = (seg >> 1) * 2;
#pragma unroll 1
  for (int pr0 = warp * RPW; pr0 < (warp + 1) * RPW; pr0 += 8) {
    const int pr = pr0 + (int)(lane >> 2);
    const int p = pr / TR, rr = pr % TR;
    const int64_t r = r0 + rr;
    const int64_t cb = c0 + p * a.part_off + 32 * seg;   // first output column of the block
    const uint4* src = reinterpret_cast<const uint4*>(&tile[(p * TR + rr) * LD]);
    const int usw = tile_sw(rr);
    uint32_t ww[16];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint4 w = src[(4 * seg + (q ^ sw)) ^ usw];
      ww[4 * q] = w.x; ww[4 * q + 1] = w.y; ww[4 * q + 2] = w.z; ww[4 * q + 3] = w.w;
    }
    if constexpr (SC == MGQ_NV16_UE4M3) {
      // two 16-column blocks: ww[0..7] hold block sw / 2 of the lane's 32
      // columns, ww[8..15] the other; ts is s_g
      uint32_t sc2 = 0;
#pragma unroll
      for (int hb = 0; hb < 2; ++hb) {
        uint32_t acc = 0;
        float y[16];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          acc = absmax_acc_bf16x2(acc, ww[8 * hb + i]);
          y[2 * i] = bf16_lo(ww[8 * hb + i]);
          y[2 * i + 1] = bf16_hi(ww[8 * hb + i]);
        }
        uint2 c;
        const uint32_t code = nv_block16(y, __uint_as_float(fold_bf16x2(absmax_bf16x2_final(acc))), ts, c);
        const int blk = (sw >> 1) ^ hb;
        if (r < nrows) *reinterpret_cast<uint2*>(a.row_codes + r * (a.C / 2) + (cb + 16 * blk) / 2) = c;
        sc2 |= code << (8 * blk);
      }
      if (r < nrows)
        *reinterpret_cast<uint16_t*>(a.row_scales + tiled_scale_offset(r, cb / 16, a.C / 64)) = (uint16_t)sc2;
    } else {
    float mult = ts;
    if constexpr (SC == MGQ_MX32_E8M0) {
      uint32_t acc = 0;
#pragma unroll
      for (int i = 0; i < 16; ++i) acc = absmax_acc_bf16x2(acc, ww[i]);
      const int e = mx_exponent(fold_bf16x2(absmax_bf16x2_final(acc)), FmtInfo<DT>::emax, a.rceil != 0);
      mult = mx_multiplier(e);
      if (r < nrows) a.row_scales[tiled_scale_offset(r, cb / 32, a.C / 128)] = (uint8_t)mx_scale_code(e);
    } else if constexpr (SC == MGQ_BLK_1x128_F32) {
      // the row's 128 tile columns are one block: the 4 lanes of the row agree on its amax
      uint32_t acc = 0;
#pragma unroll
      for (int i = 0; i < 16; ++i) acc = absmax_acc_bf16x2(acc, ww[i]);
      uint32_t m = fold_bf16x2(absmax_bf16x2_final(acc));
      m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));
      m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 2));
      mult = blk_scale<DT>(m);
      if (seg == 0 && r < nrows)
        reinterpret_cast<float*>(a.row_scales)[((c0 + p * a.part_off) / 128) * a.rows_cap + r] =
            (srow && srow[rr] < 0) ? 0.0f : __fdiv_rn(1.0f, mult);
    }
    uint32_t cw[8];        // codes in the order held (chunk q ^ sw in cw[2q], cw[2q + 1])
#pragma unroll
    for (int i = 0; i < 8; ++i) cw[i] = cvt_fp8x4_bf16_mul<DT>(ww[2 * i], ww[2 * i + 1], mult);
    if (r < nrows) {
      uint8_t* dst = a.row_codes + r * a.C + cb;
      *reinterpret_cast<uint4*>(dst + 8 * sw) = make_uint4(cw[0], cw[1], cw[2], cw[3]);
      *reinterpret_cast<uint4*>(dst + (16 - 8 * sw)) = make_uint4(cw[4], cw[5], cw[6], cw[7]);
    }
    }
  }
}

// Column-wise codes of a bf16 tile [P][TR][LD]: thread takes 2 adjacent
// columns of one 32-row block (one MX block each); its 32 output bytes per
// column are contiguous. FAC: values are fac[row] * tile (float32 products).
// am: running |v| maximum (float bits) for the per-tensor amax.
// Blockwise (128x1 blocks: the tile's 128 rows): the four 32-row partial
// maxima of each column meet in s_cm [4][TC]; every thread of the CTA calls.
template <int DT>
__device__ __forceinline__ float col_blk_scale(uint32_t* s_cm, int rb, int col, uint32_t part_max,
                                               const RowColArgs& a, int64_t crow, int64_t rtile) {
  s_cm[rb * TC + col] = part_max;
  __syncthreads();
  const uint32_t m = max(max(s_cm[col], s_cm[TC + col]), max(s_cm[2 * TC + col], s_cm[3 * TC + col]));
  const float s = blk_scale<DT>(m);
  if (rb == 0) reinterpret_cast<float*>(a.col_scales)[rtile * ((a.rows_cap / a.M) * a.C) + crow] = __fdiv_rn(1.0f, s);
  return s;
}

template <int P, int SC, int DT, bool FAC>
__device__ __forceinline__ void col_phase(const uint16_t* tile, const float* fac, int64_t g, int64_t r0, int64_t c0,
                                          float ts, const RowColArgs& a, int tid, uint32_t& am, uint32_t* s_cm,
                                          uint8_t* stg0 = nullptr) {
  // thread -> (column pair cp, 32-row block rb). A warp takes 8 column pairs
  // x the 4 row blocks, so each direct store instruction covers whole output
  // rows of the tile (128 FP8 bytes or 64 NVFP4 bytes, 8 of them) instead of
  // pieces of 32 rows; the tile swizzle keeps its column reads conflict-free.
  // The factor pass (dY = probs * dout) is the exception: there a warp takes
  // 32 column pairs of one row block, which measured faster for it (with the
  // FP8 column codes staged for one TMA store), while the whole-row mapping
  // measured faster for every other source and format.
  const bool by_rows = stg0 == nullptr && !FAC;
  const int cp = by_rows ? (tid >> 2) : (tid & 63), rb = by_rows ? (tid & 3) : ((tid >> 6) & 3);
  const int cc = 2 * cp;
  // the thread's column pair inside a swizzled tile row of its row block
  const int cx = (((cc >> 3) ^ (2 * rb)) << 3) + (cc & 7);
  const int64_t rg = r0 - g * a.M + 32 * rb;                 // row inside the group
#pragma unroll 1
  for (int p = 0; p < P; ++p) {
    const int64_t crow = g * a.C + c0 + p * a.part_off + cc;  // row of the column-wise output
    uint8_t* stg = stg0 ? stg0 + p * kStgBytes : nullptr;     // this part's staging tile
    if constexpr (SC == MGQ_BLK_1x128_F32) {
      // 128x1 blocks: per column the amax of the tile's 128 rows, then the
      // column's codes with its scale (two columns per thread)
      const int64_t rtile = (r0 - g * a.M) / TR;
      auto val = [&](int i, int h) {
        const float x = __uint_as_float((uint32_t)tile[(p * TR + 32 * rb + i) * LD + cx + h] << 16);
        if constexpr (FAC) return __fmul_rn(fac[32 * rb + i], x);
        else return x;
      };
      uint32_t m2[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t m = 0;
#pragma unroll
        for (int i = 0; i < 32; ++i) m = max(m, __float_as_uint(val(i, h)) & 0x7FFFFFFFu);
        m2[h] = m;
      }
      float sc[2];
      sc[0] = col_blk_scale<DT>(s_cm, rb, cc, m2[0], a, crow, rtile);
      __syncthreads();
      sc[1] = col_blk_scale<DT>(s_cm, rb, cc + 1, m2[1], a, crow + 1, rtile);
#pragma unroll 1
      for (int h = 0; h < 2; ++h) {
        float v[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = val(i, h);
        col_block_out<MGQ_TENSOR_F32, DT>(v, 0u, sc[h], a, crow + h, rg, stg, cc + h, 32 * rb);
      }
      __syncthreads();     // s_cm is reused by the next part / tile
    } else if constexpr (FAC) {
      // one column at a time (32 products live)
#pragma unroll 1
      for (int h = 0; h < 2; ++h) {
        float v[32];
#pragma unroll
        for (int i = 0; i < 32; ++i)
          v[i] = __fmul_rn(fac[32 * rb + i], __uint_as_float((uint32_t)tile[(p * TR + 32 * rb + i) * LD + cx + h] << 16));
        const uint32_t m = absmax_bits_f32(v, 32);
        am = max(am, m);
        col_block_out<SC, DT>(v, m, ts, a, crow + h, rg, stg, cc + h, 32 * rb);
      }
    } else {
      uint32_t w[32];      // the two columns' 32 values as bf16 pairs
#pragma unroll
      for (int i = 0; i < 32; ++i) w[i] = *reinterpret_cast<const uint32_t*>(&tile[(p * TR + 32 * rb + i) * LD + cx]);
      uint32_t amh[2] = {0, 0};
      if (SC == MGQ_MX32_E8M0 || (SC == MGQ_TENSOR_F32 && a.amax_out)) {
        uint32_t acc = 0;
#pragma unroll
        for (int i = 0; i < 32; ++i) acc = absmax_acc_bf16x2(acc, w[i]);
        acc = absmax_bf16x2_final(acc);
        amh[0] = acc << 16;
        amh[1] = acc & 0xFFFF0000u;
        am = max(am, max(amh[0], amh[1]));
      }
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        float v[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = h ? bf16_hi(w[i]) : bf16_lo(w[i]);
        col_block_out<SC, DT>(v, amh[h], ts, a, crow + h, rg, stg, cc + h, 32 * rb);
      }
    }
  }
}

// the scale a tile's codes are made with: per-tensor s of the group, NVFP4 s_g
// of the group from its amax (pre-pass), else unused
template <int SC>
__device__ __forceinline__ float tile_scale(const RowColArgs& a, int64_t g) {
  if (SC == MGQ_TENSOR_F32) return a.tensor_scale[g];
  if (SC == MGQ_NV16_UE4M3) return nv_global_scale(a.amax_out[g]);
  return 1.0f;
}

// per-tensor amax of group g: CTA reduction (NW warps), one atomic
template <int NW = 8>
__device__ __forceinline__ void flush_amax(uint32_t am, float* amax_out, int64_t g, uint32_t* s_amax, int tid) {
  am = warp_max_u32(am);
  if ((tid & 31) == 0) s_amax[tid >> 5] = am;
  __syncthreads();
  if (tid == 0) {
    for (int i = 1; i < NW; ++i) am = max(am, s_amax[i]);
    atomic_max_nonneg(amax_out + g, __uint_as_float(am));
  }
  __syncthreads();
}

// ---- plain and computed sources: one tile per CTA ---------------------------

template <class Src, int SC, int DT>
__global__ void __launch_bounds__(256, Src::kParts == 2 ? 3 : 4)
    quant_rowcol_kernel(const Src src, const RowColArgs a, const __grid_constant__ CUtensorMap tmc) {
  constexpr int P = Src::kParts;
  // 128x128 weight tiles: one scale per tile, then both copies cast like a
  // per-tensor scale (the column-wise copy is the transposed cast)
  constexpr bool T128 = SC == MGQ_BLK_128x128_F32;
  constexpr int SCC = T128 ? MGQ_TENSOR_F32 : SC;
  extern __shared__ __align__(16) uint8_t smem_raw[];
  uint16_t* tile = reinterpret_cast<uint16_t*>(smem_raw);   // [P][TR][LD]
  // staged column codes [P][128][128] (1024-byte aligned for the swizzled TMA store)
  uint8_t* stg = nullptr;
  if (a.col_tma) {
    const uint32_t raw = ptx::smem_u32(smem_raw) + P * TR * LD * 2;
    stg = smem_raw + P * TR * LD * 2 + (((raw + 1023u) & ~1023u) - raw);
  }
  __shared__ uint32_t s_amax[8];
  __shared__ uint32_t s_cm[SC == MGQ_BLK_1x128_F32 ? 4 * TC : 1];
  const int tid = threadIdx.x, warp = tid >> 5;
  const uint32_t lane = tid & 31;
  const int64_t nrows = a.rows_used ? (int64_t)*a.rows_used : a.rows_cap;
  const int n_rt = (int)((nrows + TR - 1) / TR);     // fewer than 2^31 rows
  const int64_t c0 = (int64_t)blockIdx.x * TC;
#pragma unroll 1
  for (int rt = blockIdx.y; rt < n_rt; rt += gridDim.y) {
    const int64_t r0 = (int64_t)rt * TR;
    const int64_t g = (int)r0 / (int)a.M;
    const float ts = tile_scale<SC>(a, g);
    if (SC == MGQ_NV16_UE4M3 && blockIdx.x == 0 && r0 == g * a.M && tid == 0) a.s_out[g] = ts;
    // ---- load: TR rows x 16 chunks of 8 columns, 8 chunks per thread
    uint32_t am2 = 0;
    if constexpr (!Src::kComputed) {
      // plain: all eight 16-byte loads in flight, then copied into the tile
      uint4 w[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int chunk = tid + 256 * i;
        const int rr = chunk >> 4, cc = (chunk & 15) * 8;
        w[i] = (r0 + rr < nrows) ? __ldg(reinterpret_cast<const uint4*>(src.x + (r0 + rr) * src.ld + c0 + cc))
                                 : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int chunk = tid + 256 * i;
        const int rr = chunk >> 4, cc = (chunk & 15) * 8;
        if (SC == MGQ_TENSOR_F32 || T128)
          am2 = absmax_bf16x2(absmax_bf16x2(absmax_bf16x2(absmax_bf16x2(am2, w[i].x), w[i].y), w[i].z), w[i].w);
        *reinterpret_cast<uint4*>(&tile[tix(rr, cc)]) = w[i];
      }
    } else {
    // the operands of kBatch chunks loaded together
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
        uint4 o[P];
        src.make(w[j], r0 + rr, c0 + cc, r0 + rr < nrows, o);
#pragma unroll
        for (int p = 0; p < P; ++p) {
          if (SC == MGQ_TENSOR_F32)
            am2 = absmax_bf16x2(absmax_bf16x2(absmax_bf16x2(absmax_bf16x2(am2, o[p].x), o[p].y), o[p].z), o[p].w);
          *reinterpret_cast<uint4*>(&tile[p * TR * LD + tix(rr, cc)]) = o[p];
        }
      }
    }
    }
    __syncthreads();
    float tsc = ts;
    if constexpr (T128) {
      // the tile's amax (CTA reduction) sets its scale; scale_inv of both copies
      uint32_t m = warp_max_u32(fold_bf16x2(am2));
      if (lane == 0) s_amax[warp] = m;
      __syncthreads();
      m = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) m = max(m, s_amax[i]);
      tsc = blk_scale<DT>(m);
      if (tid == 0) {
        const float sinv = __fdiv_rn(1.0f, tsc);
        const int64_t mt = (r0 - g * a.M) / TR, ct = c0 / TC;
        reinterpret_cast<float*>(a.row_scales)[(r0 / TR) * (a.C / TC) + ct] = sinv;
        if (a.col_codes) reinterpret_cast<float*>(a.col_scales)[(g * (a.C / TC) + ct) * (a.M / TR) + mt] = sinv;
      }
      __syncthreads();   // s_amax is reused by the next row tile
    }
    if (a.row_codes) row_phase<P, SCC, DT>(tile, r0, nrows, c0, tsc, a, warp, lane);
    uint32_t am_unused = 0;
    if (a.col_codes) {
      if (stg) wait_col_tiles(tid);
      col_phase<P, SCC, DT, false>(tile, nullptr, g, r0, c0, tsc, a, tid, am_unused, s_cm, stg);
      if (stg) store_col_tiles<P>(&tmc, stg, (int32_t)(r0 - g * a.M), (int32_t)(g * a.C + c0), a.part_off, tid);
    }
    if (SC == MGQ_TENSOR_F32 && a.amax_out) flush_amax(fold_bf16x2(am2), a.amax_out, g, s_amax, tid);
    __syncthreads();   // the tile is reused by the next row tile
  }
  // the staged stores have read shared memory before the CTA exits (their
  // global writes complete with the grid)
  if (stg && tid == 0) ptx::bulk_wait_read0();
}

// ---- dSwiGLU: persistent, operands brought in by TMA ---------------------------

constexpr int kHalf = TR / 2;                                 // rows of a half tile
constexpr uint32_t kOpHalfBytes = kHalf * TC * 2;             // one operand's half tile (bf16)

// The operands of the dSwiGLU source (dh, g, u) arrive by TMA in 64-row half
// tiles, three copies a half, into two half buffers with an mbarrier each. A
// CTA of 512 threads walks a contiguous range of (row tile, column tile)
// items. For each half it waits for the copies, makes the half's dG and dU
// into the tile, and then requests the same half of its next item, so those
// copies are in flight while the CTA makes the other half and quantises the
// tile (row phase over all 16 warps, column phase one part per 256 threads).
// tmA: gu [R_cap, 2F] (g at column f, u at F + f); tmB: dh [R_cap, F]. Rows at
// or past the row count are made from zeros, as in the one-tile kernel.
template <class Src, int SC, int DT>
__global__ void __launch_bounds__(512, 1)
    quant_rowcol_pipe_kernel(const Src src, const RowColArgs a, const __grid_constant__ CUtensorMap tmA,
                             const __grid_constant__ CUtensorMap tmB) {
  constexpr int P = Src::kParts, L = Src::kLoads, NT = P * 256, NW = NT / 32;
  static_assert(P == 2 && L == 3 && SC != MGQ_BLK_1x128_F32, "the dSwiGLU source, MX or per-tensor scaling");
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_a = ptx::smem_u32(smem_raw);
  uint8_t* base = smem_raw + (((raw_a + 1023u) & ~1023u) - raw_a);
  uint16_t* ops = reinterpret_cast<uint16_t*>(base);                         // [2 halves][L][kHalf][TC]
  uint16_t* tile = reinterpret_cast<uint16_t*>(base + 2 * L * kOpHalfBytes);  // [P][TR][LD]
  __shared__ __align__(8) uint64_t s_full[2];
  __shared__ uint32_t s_amax[NW];
  __shared__ uint32_t s_cm[1];   // (blockwise column maxima: not used)
  const int tid = threadIdx.x, warp = tid >> 5;
  const uint32_t lane = tid & 31;
  const int64_t nrows = a.rows_used ? (int64_t)*a.rows_used : a.rows_cap;
  const int64_t n_ct = a.C / P / TC;
  const int64_t n_items = (nrows + TR - 1) / TR * n_ct;
  const int64_t i0 = n_items * blockIdx.x / gridDim.x, i1 = n_items * (blockIdx.x + 1) / gridDim.x;
  if (i0 >= i1) return;
  // the copies of one half of an item: L operands of kHalf rows x TC columns
  auto request = [&](int64_t item, int h) {
    const int64_t rt = item / n_ct, ct = item - rt * n_ct;
    const int32_t y = (int32_t)(rt * TR + h * kHalf), f = (int32_t)(ct * TC);
    uint16_t* dst = ops + (size_t)h * L * (kOpHalfBytes / 2);
    ptx::mbar_arrive_expect_tx(&s_full[h], L * kOpHalfBytes);
    ptx::tma_load_2d(dst, &tmB, &s_full[h], f, y);                                   // dh
    ptx::tma_load_2d(dst + kOpHalfBytes / 2, &tmA, &s_full[h], f, y);                // g
    ptx::tma_load_2d(dst + kOpHalfBytes, &tmA, &s_full[h], (int32_t)src.F + f, y);   // u
  };
  if (tid == 0) {
    ptx::mbar_init(&s_full[0], 1);
    ptx::mbar_init(&s_full[1], 1);
    ptx::fence_mbar_init();
    ptx::prefetch_tmap(&tmA);
    ptx::prefetch_tmap(&tmB);
    request(i0, 0);
    request(i0, 1);
  }
  __syncthreads();
#pragma unroll 1
  for (int64_t item = i0; item < i1; ++item) {
    const int64_t rt = item / n_ct, ct = item - rt * n_ct;
    const int64_t r0 = rt * TR, c0 = ct * TC;
    const int64_t g = r0 / a.M;
    const float ts = tile_scale<SC>(a, g);
    const uint32_t ph = (uint32_t)((item - i0) & 1);
    uint32_t am2 = 0;
#pragma unroll 1
    for (int h = 0; h < 2; ++h) {
      const bool ok = ptx::mbar_wait(&s_full[h], ph, a.wait_ns);
      if (__syncthreads_or(!ok)) {
        // a copy ran out of time: report it, let the copies still in flight
        // (this half's, and the other half's request) land, and leave
        if (tid == 0) {
          report(a.err, MGQ_ERR_TIMEOUT);
          ptx::mbar_wait(&s_full[h], ph, a.wait_ns);
          if (h == 0) ptx::mbar_wait(&s_full[1], ph, a.wait_ns);
          else if (item + 1 < i1) ptx::mbar_wait(&s_full[0], ph ^ 1u, a.wait_ns);
        }
        __syncthreads();
        return;
      }
      const uint16_t* src_h = ops + (size_t)h * L * (kOpHalfBytes / 2);
      // make: kHalf rows x 16 chunks of 8 columns, NT threads
#pragma unroll
      for (int j = 0; j < kHalf * 16 / NT; ++j) {
        const int chunk = tid + NT * j;
        const int rr = chunk >> 4, cc = (chunk & 15) * 8;
        const int64_t r = r0 + h * kHalf + rr;
        const bool valid = r < nrows;
        uint4 w[L];
#pragma unroll
        for (int l = 0; l < L; ++l)
          w[l] = valid ? *reinterpret_cast<const uint4*>(src_h + (size_t)l * (kOpHalfBytes / 2) + rr * TC + cc)
                       : make_uint4(0, 0, 0, 0);
        uint4 o[P];
        src.make(w, r, c0 + cc, valid, o);
#pragma unroll
        for (int pp = 0; pp < P; ++pp) {
          if (SC == MGQ_TENSOR_F32)
            am2 = absmax_bf16x2(absmax_bf16x2(absmax_bf16x2(absmax_bf16x2(am2, o[pp].x), o[pp].y), o[pp].z), o[pp].w);
          *reinterpret_cast<uint4*>(&tile[pp * TR * LD + tix(h * kHalf + rr, cc)]) = o[pp];
        }
      }
      __syncthreads();   // the half buffer is read (and this half of the tile written)
      if (tid == 0 && item + 1 < i1) request(item + 1, h);
    }
    if (a.row_codes) row_phase<P, SC, DT, 16>(tile, r0, nrows, c0, ts, a, warp, lane);
    if (a.col_codes) {
      // one part per 256 threads
      const int pp = tid >> 8;
      uint32_t am_unused = 0;
      col_phase<1, SC, DT, false>(tile + pp * TR * LD, nullptr, g, r0, c0 + pp * a.part_off, ts, a, tid & 255,
                                  am_unused, s_cm);
    }
    if (SC == MGQ_TENSOR_F32 && a.amax_out) flush_amax<NW>(fold_bf16x2(am2), a.amax_out, g, s_amax, tid);
    __syncthreads();   // the tile is made again for the next item
  }
}

// ---- streamed sources: pipelined over the CTA's items -----------------------

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem, bool valid) {
  const uint32_t s = (uint32_t)__cvta_generic_to_shared(smem);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(s), "l"(gmem), "r"(valid ? 16 : 0) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N> __device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// The items (row tile, column tile) in row-major order are split into one
// contiguous range per CTA. A CTA resolves the source offsets (and factors) of
// a row tile once, into the slot of the row tile's parity, and stages the
// next item's tile with cp.async (zero fill for zero rows) while it quantises
// the current one: two tile buffers, two offset slots.
template <class Src, int SC, int DT>
__global__ void __launch_bounds__(256, 3)
    quant_rowcol_stream_kernel(const Src src, const RowColArgs a, const __grid_constant__ CUtensorMap tmc) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  uint16_t* tiles = reinterpret_cast<uint16_t*>(smem_raw);   // [2][TR][LD]
  uint8_t* stg = nullptr;                                     // staged column codes [128][128]
  if (a.col_tma) {
    const uint32_t raw = ptx::smem_u32(smem_raw) + 2 * TR * LD * 2;
    stg = smem_raw + 2 * TR * LD * 2 + (((raw + 1023u) & ~1023u) - raw);
  }
  __shared__ int64_t s_off[2][TR];
  __shared__ float s_fac[2][TR];
  __shared__ uint32_t s_amax[8];
  __shared__ uint32_t s_cm[SC == MGQ_BLK_1x128_F32 ? 4 * TC : 1];
  const int tid = threadIdx.x, warp = tid >> 5;
  const uint32_t lane = tid & 31;
  const int64_t nrows = a.rows_used ? (int64_t)*a.rows_used : a.rows_cap;
  const int64_t n_ct = a.C / TC;
  const int64_t n_items = (nrows + TR - 1) / TR * n_ct;
  const int64_t i0 = n_items * blockIdx.x / gridDim.x, i1 = n_items * (blockIdx.x + 1) / gridDim.x;
  if (i0 >= i1) return;
  auto resolve = [&](int rt) {                    // offsets of row tile rt, slot rt & 1
    if (tid < TR) {
      const int64_t r = (int64_t)rt * TR + tid;
      float f = 0.0f;
      const int64_t off = r < nrows ? src.row_offset(r, f) : -1;
      s_off[rt & 1][tid] = off;
      s_fac[rt & 1][tid] = f;
    }
  };
  auto issue = [&](int rt, int ct, int buf) {     // cp.async of the item's tile
    uint16_t* t = tiles + buf * TR * LD;
    const int64_t c0 = (int64_t)ct * TC;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int chunk = tid + 256 * j;
      const int rr = chunk >> 4, cc = (chunk & 15) * 8;
      const int64_t off = s_off[rt & 1][rr];
      cp_async16(&t[tix(rr, cc)], src.base() + (off >= 0 ? off + c0 + cc : 0), off >= 0);
    }
    cp_async_commit();
  };
  // item coordinates advance incrementally (row tile, column tile)
  int rt = (int)(i0 / n_ct), ct = (int)(i0 - (int64_t)rt * n_ct);
  resolve(rt);
  __syncthreads();
  issue(rt, ct, 0);
  int64_t g = (int)((int64_t)rt * TR) / (int)a.M;
  float ts = tile_scale<SC>(a, g);
  uint32_t am = 0;
#pragma unroll 1
  for (int64_t item = i0; item < i1; ++item) {
    const int buf = (int)((item - i0) & 1);
    int rt_n = rt, ct_n = ct + 1;
    if (ct_n == (int)n_ct) {
      ct_n = 0;
      ++rt_n;
    }
    if (item + 1 < i1) {
      if (rt_n != rt) {
        resolve(rt_n);
        __syncthreads();
      }
      issue(rt_n, ct_n, buf ^ 1);
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    const int64_t r0 = (int64_t)rt * TR, c0 = (int64_t)ct * TC;
    const uint16_t* t = tiles + buf * TR * LD;
    if (SC == MGQ_NV16_UE4M3 && ct == 0 && r0 == g * a.M && tid == 0) a.s_out[g] = ts;
    if (!Src::kColumnsOnly && a.row_codes) row_phase<1, SC, DT>(t, r0, nrows, c0, ts, a, warp, lane, s_off[rt & 1]);
    if (stg) wait_col_tiles(tid);
    col_phase<1, SC, DT, Src::kFactor>(t, s_fac[rt & 1], g, r0, c0, ts, a, tid, am, s_cm, stg);
    if (stg) store_col_tiles<1>(&tmc, stg, (int32_t)(r0 - g * a.M), (int32_t)(g * a.C + c0), 0, tid);
    __syncthreads();   // the buffer is refilled two items on
    if (rt_n != rt || item + 1 == i1) {
      if (SC == MGQ_TENSOR_F32 && a.amax_out) flush_amax(am, a.amax_out, g, s_amax, tid);
      am = 0;
      g = (int)((int64_t)rt_n * TR) / (int)a.M;
      if (item + 1 < i1) ts = tile_scale<SC>(a, g);
    }
    rt = rt_n;
    ct = ct_n;
  }
  // the staged stores have read shared memory before the CTA exits (their
  // global writes complete with the grid)
  if (stg && tid == 0) ptx::bulk_wait_read0();
}

// the dynamic shared memory limit of one kernel, set once per device
// (attr_set: a flag array owned by the kernel's launcher)
template <class Kern>
int set_smem(Kern kern, size_t smem, bool* attr_set) {
  int dev = 0;
  cudaGetDevice(&dev);
  if (smem > 48 * 1024 && dev < 64 && !attr_set[dev]) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
      return MGQ_ERR_CUDA;
    attr_set[dev] = true;
  }
  return MGQ_OK;
}

template <class Src, int SC, int DT>
int launch_rowcol_t(const Src& src, RowColArgs a, cudaStream_t s) {
  static bool attr_set[64] = {false};   // one per instantiation
  // FP8 column copies of the factor pass go out through staged TMA stores: a
  // map of the column output [G * C rows, M bytes], 128 x 128-byte boxes
  CUtensorMap tmc;
  memset(&tmc, 0, sizeof(tmc));
  a.col_tma = 0;
  // (measured: the factor pass gains from the staging; the gathered X with
  // whole-row column stores and three CTAs an SM, and the one-tile CTAs of
  // plain and computed sources, do not)
  if (SC != MGQ_NV16_UE4M3 && Src::kStream && Src::kFactor && a.col_codes) {
    if (!encode_tmap_u8_2d(&tmc, a.col_codes, (uint64_t)a.M, (uint64_t)((a.rows_cap / a.M) * a.C), (uint64_t)a.M,
                           128, 128))
      return MGQ_ERR_CUDA;
    a.col_tma = 1;
  }
  constexpr int P = Src::kParts;
  constexpr size_t stg_max = (SC == MGQ_NV16_UE4M3 || !Src::kStream || !Src::kFactor) ? 0 : 1024 + (size_t)kStgBytes;
  const size_t stg = a.col_tma ? stg_max : 0;
  // dSwiGLU with MX or per-tensor scaling: the persistent kernel fed by TMA
  // (measured: MX 1.09 -> 1.03 ms on the Mixtral training shape; SwiGLU and
  // the blockwise 128x1 column blocks, whose column phase synchronises the
  // CTA twice a part, ran 3-4% slower on it than on one-tile CTAs)
  constexpr bool kPipe = !Src::kStream && Src::kComputed && Src::kParts == 2 && SC != MGQ_BLK_1x128_F32;
  if constexpr (kPipe) {
    // operand maps: gu [R_cap, 2F] and dh [R_cap, F], boxes of 128 columns x
    // 64 rows (the callers keep F and R_cap multiples of 128)
    CUtensorMap tma, tmb;
    memset(&tma, 0, sizeof(tma));
    memset(&tmb, 0, sizeof(tmb));
    if (!encode_tmap_2d(&tma, src.gu, 2, (uint64_t)(2 * src.F), (uint64_t)a.rows_cap, (uint64_t)(4 * src.F), TC,
                        kHalf, false))
      return MGQ_ERR_CUDA;
    if (!encode_tmap_2d(&tmb, src.dh, 2, (uint64_t)src.F, (uint64_t)a.rows_cap, (uint64_t)(2 * src.F), TC, kHalf,
                        false))
      return MGQ_ERR_CUDA;
    constexpr size_t smem = 1024 + 2 * (size_t)Src::kLoads * kOpHalfBytes + (size_t)P * TR * LD * sizeof(uint16_t);
    auto kern = quant_rowcol_pipe_kernel<Src, SC, DT>;
    if (set_smem(kern, smem, attr_set) != MGQ_OK) return MGQ_ERR_CUDA;
    const int64_t items = (a.rows_cap + TR - 1) / TR * (a.C / P / TC);
    const int64_t ctas = std::max<int64_t>(1, std::min<int64_t>(items, (int64_t)num_sms()));   // one an SM
    kern<<<(unsigned)ctas, 512, smem, s>>>(src, a, tma, tmb);
  } else if constexpr (!Src::kStream) {
    constexpr size_t tiles = (size_t)P * TR * LD * sizeof(uint16_t);
    auto kern = quant_rowcol_kernel<Src, SC, DT>;
    if (set_smem(kern, tiles + stg_max, attr_set) != MGQ_OK) return MGQ_ERR_CUDA;
    const dim3 grid((unsigned)(a.C / P / TC), (unsigned)std::min<int64_t>((a.rows_cap + TR - 1) / TR, 65535));
    kern<<<grid, 256, tiles + stg, s>>>(src, a, tmc);
  } else {
    constexpr size_t tiles = 2 * TR * LD * sizeof(uint16_t);
    auto kern = quant_rowcol_stream_kernel<Src, SC, DT>;
    if (set_smem(kern, tiles + stg_max, attr_set) != MGQ_OK) return MGQ_ERR_CUDA;
    const int64_t items = (a.rows_cap + TR - 1) / TR * (a.C / TC);
    // resident CTAs per SM: 3 with the tile buffers alone, 2 with the staging
    const int64_t ctas = std::max<int64_t>(1, std::min<int64_t>(items, (int64_t)num_sms() * (stg ? 2 : 3)));
    kern<<<(unsigned)ctas, 256, tiles + stg, s>>>(src, a, tmc);
  }
  MGQ_LAUNCH_CHECK();
  return MGQ_OK;
}

template <class Src>
int launch_rowcol(const Src& src, const mgq_qdesc* q, RowColArgs a, cudaStream_t s) {
  if (a.rows_cap >= (1ll << 31) || a.M >= (1ll << 31)) return MGQ_ERR_UNSUPPORTED;
  if (Src::kStream && !a.col_codes) return MGQ_ERR_UNSUPPORTED;   // a row + column pass
  const int sc = q->scaling, dt = q->dtype;
  // NVFP4 (s_g from the amax pre-pass in amax_out): streamed and plain sources
  constexpr bool kComputedSrc = std::is_same<Src, SrcSwiglu>::value || std::is_same<Src, SrcDswiglu>::value;
  if (sc == MGQ_NV16_UE4M3) {
    if constexpr (kComputedSrc) {
      return MGQ_ERR_UNSUPPORTED;
    } else {
      if (dt != MGQ_E2M1 || !a.amax_out || !a.s_out) return MGQ_ERR_INVALID_ARG;
      return launch_rowcol_t<Src, MGQ_NV16_UE4M3, MGQ_E2M1>(src, a, s);
    }
  }
  if (sc == MGQ_MX32_E8M0 && dt == MGQ_E4M3) return launch_rowcol_t<Src, MGQ_MX32_E8M0, MGQ_E4M3>(src, a, s);
  if (sc == MGQ_MX32_E8M0 && dt == MGQ_E5M2) return launch_rowcol_t<Src, MGQ_MX32_E8M0, MGQ_E5M2>(src, a, s);
  // blockwise: 1x128 rows / 128x1 columns inside 128-row groups; 128x128
  // tiles for plain matrices (weights)
  if (sc == MGQ_BLK_1x128_F32 || sc == MGQ_BLK_128x128_F32) {
    // (the gathered dY source writes column-wise codes only)
    if (a.M % TR != 0 || (a.row_codes && !a.row_scales) || (a.col_codes && !a.col_scales)) return MGQ_ERR_INVALID_ARG;
    if (sc == MGQ_BLK_1x128_F32 && dt == MGQ_E4M3) return launch_rowcol_t<Src, MGQ_BLK_1x128_F32, MGQ_E4M3>(src, a, s);
    if (sc == MGQ_BLK_1x128_F32 && dt == MGQ_E5M2) return launch_rowcol_t<Src, MGQ_BLK_1x128_F32, MGQ_E5M2>(src, a, s);
    if constexpr (std::is_same<Src, SrcPlain>::value) {
      if (dt == MGQ_E4M3) return launch_rowcol_t<Src, MGQ_BLK_128x128_F32, MGQ_E4M3>(src, a, s);
      if (dt == MGQ_E5M2) return launch_rowcol_t<Src, MGQ_BLK_128x128_F32, MGQ_E5M2>(src, a, s);
    }
    return MGQ_ERR_UNSUPPORTED;
  }
  // per-tensor column copies of gathered rows are transposed casts of the row codes
  if constexpr (std::is_same<Src, SrcGatherX>::value || std::is_same<Src, SrcGatherDy>::value) {
    return MGQ_ERR_UNSUPPORTED;
  } else {
    if (sc == MGQ_TENSOR_F32 && dt == MGQ_E4M3) return launch_rowcol_t<Src, MGQ_TENSOR_F32, MGQ_E4M3>(src, a, s);
    if (sc == MGQ_TENSOR_F32 && dt == MGQ_E5M2) return launch_rowcol_t<Src, MGQ_TENSOR_F32, MGQ_E5M2>(src, a, s);
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
  a.s_out = q->tensor_scale;
  a.rceil = q->e8m0_mode == MGQ_E8M0_RCEIL;
  a.col_tma = 0;
  a.err = error_word();
  a.wait_ns = 2000000000ull;   // 2 s: far beyond any tile
  return a;
}

// ---- NVFP4 weights with 16x16 blocks ------------------------------------------
// One 128x128 tile of a group's [M, K] weight per CTA, staged in shared
// memory (swizzled like the row/column tiles): the 64 block amaxes (4 threads
// per 16x16 block), then the ue4m3 scale code and multiplier r = s_g / sc of
// each block by the 1x16 rule, then the row-wise copy ([G*M, K/2], one 1x16
// block per thread step) and the column-wise copy ([G*K, M/2]). Both copies'
// 1x16 blocks carry the scale of their 16x16 block. In the column-wise copy a
// thread takes two adjacent columns of one 32-row quarter, and the four
// quarters of a column are adjacent lanes, so one store instruction writes
// the whole 64-byte piece of 8 output rows.
__global__ void __launch_bounds__(256) quant_nv2d_kernel(const uint16_t* x, int64_t M, int64_t K, uint8_t* row_codes,
                                                         uint8_t* row_scales, uint8_t* col_codes, uint8_t* col_scales,
                                                         const float* amax, float* s_out) {
  __shared__ __align__(16) uint16_t tile[TR * LD];
  __shared__ __align__(16) uint8_t s_code[64];
  __shared__ float s_r[64];
  const int tid = threadIdx.x;
  const uint32_t lane = tid & 31;
  const int64_t c0 = (int64_t)blockIdx.x * TC, r0 = (int64_t)blockIdx.y * TR;
  const int64_t g = r0 / M, m0 = r0 - g * M;    // group, first row inside it
  const float s_g = nv_global_scale(amax[g]);
  if (blockIdx.x == 0 && m0 == 0 && tid == 0) s_out[g] = s_g;
  {
    uint4 w[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int chunk = tid + 256 * i;
      w[i] = __ldg(reinterpret_cast<const uint4*>(x + (r0 + (chunk >> 4)) * K + c0 + (chunk & 15) * 8));
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int chunk = tid + 256 * i;
      *reinterpret_cast<uint4*>(&tile[tix(chunk >> 4, (chunk & 15) * 8)]) = w[i];
    }
  }
  __syncthreads();
  {
    // block b = (br, bc); this thread's quarter: rows 16 br + 4 q .. + 3
    const int b = tid >> 2, q = tid & 3, br = b >> 3, bc = b & 7;
    uint32_t acc = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int row = 16 * br + 4 * q + j;
      const uint4 w0 = *reinterpret_cast<const uint4*>(&tile[tix(row, 16 * bc)]);
      const uint4 w1 = *reinterpret_cast<const uint4*>(&tile[tix(row, 16 * bc + 8)]);
      acc = absmax_acc_bf16x2(absmax_acc_bf16x2(absmax_acc_bf16x2(absmax_acc_bf16x2(acc, w0.x), w0.y), w0.z), w0.w);
      acc = absmax_acc_bf16x2(absmax_acc_bf16x2(absmax_acc_bf16x2(absmax_acc_bf16x2(acc, w1.x), w1.y), w1.z), w1.w);
    }
    uint32_t m = fold_bf16x2(absmax_bf16x2_final(acc));
    m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));
    m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 2));
    if (q == 0) {
      const float t = __fmul_rn(__fdiv_rn(__uint_as_float(m), 6.0f), s_g);
      const uint32_t code = cvt_ue4m3(t);
      const float sc = ue4m3_value(code);
      s_code[b] = (uint8_t)code;
      s_r[b] = (sc == 0.0f) ? 0.0f : __fdiv_rn(s_g, sc);
    }
  }
  __syncthreads();
  // row-wise copy: items (row, 16-column block), 4 per thread; the lane of
  // blocks 0 and 4 of a row stores the row's four scale codes of its half
#pragma unroll 1
  for (int j = 0; j < 4; ++j) {
    const int item = tid + 256 * j, row = item >> 3, blk = item & 7;
    const int b = (row >> 4) * 8 + blk;
    const float r = s_r[b];
    const uint4 w0 = *reinterpret_cast<const uint4*>(&tile[tix(row, 16 * blk)]);
    const uint4 w1 = *reinterpret_cast<const uint4*>(&tile[tix(row, 16 * blk + 8)]);
    float y[16];
    unpack8_bf16(w0, y);
    unpack8_bf16(w1, y + 8);
    const int64_t grow = r0 + row, c = c0 + 16 * blk;
    *reinterpret_cast<uint2*>(row_codes + grow * (K / 2) + c / 2) = make_uint2(cvt_e2m1x8_mul(y, r),
                                                                                cvt_e2m1x8_mul(y + 8, r));
    if ((blk & 3) == 0)
      *reinterpret_cast<uint32_t*>(row_scales + tiled_scale_offset(grow, c / 16, K / 64)) =
          *reinterpret_cast<const uint32_t*>(&s_code[b]);
  }
  if (!col_codes) return;
  // column-wise copy: columns 2 cp, 2 cp + 1, rows 32 qr .. 32 qr + 31 (the
  // 16x16 blocks 2 qr and 2 qr + 1 of the columns' block column)
  {
    const int qr = lane & 3, cp = (tid >> 5) * 8 + (int)(lane >> 2);
    const int cc = 2 * cp;
    const int cx = (((cc >> 3) ^ (2 * qr)) << 3) + (cc & 7);   // swizzled column offset (tile_sw of rows 32 qr..)
    uint32_t w[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) w[i] = *reinterpret_cast<const uint32_t*>(&tile[(32 * qr + i) * LD + cx]);
    const int b0 = (2 * qr) * 8 + (cc >> 4), b1 = b0 + 8;
    const float rk[2] = {s_r[b0], s_r[b1]};
    const uint16_t sc2 = (uint16_t)(s_code[b0] | (s_code[b1] << 8));
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      uint32_t out[4];
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        float y[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) y[i] = h ? bf16_hi(w[16 * k + i]) : bf16_lo(w[16 * k + i]);
        out[2 * k] = cvt_e2m1x8_mul(y, rk[k]);
        out[2 * k + 1] = cvt_e2m1x8_mul(y + 8, rk[k]);
      }
      const int64_t crow = g * K + c0 + cc + h;                  // row of the column-wise copy
      *reinterpret_cast<uint4*>(col_codes + crow * (M / 2) + (m0 + 32 * qr) / 2) =
          make_uint4(out[0], out[1], out[2], out[3]);
      *reinterpret_cast<uint16_t*>(col_scales + tiled_scale_offset(crow, (m0 + 32 * qr) / 16, M / 64)) = sc2;
    }
  }
}

}  // namespace

int rowcol_plain(const uint16_t* x, int64_t G, int64_t M, int64_t K, const mgq_qdesc* q, cudaStream_t s) {
  return launch_rowcol(SrcPlain{x, K}, q, make_args(q, G * M, nullptr, K, M), s);
}

int rowcol_rows(const uint16_t* x, int64_t rows_cap, const int32_t* rows_used, int64_t C, const mgq_qdesc* q,
                cudaStream_t s) {
  return launch_rowcol(SrcPlain{x, C}, q, make_args(q, rows_cap, rows_used, C, rows_cap), s);
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

int col_gather_dy(const uint16_t* dout, const float* probs, const int32_t* src_row, int k, int64_t H,
                  int64_t R_cap, const int32_t* rows_used, const mgq_qdesc* q, cudaStream_t s) {
  RowColArgs a = make_args(q, R_cap, rows_used, H, R_cap);
  a.row_codes = nullptr;       // the row-wise codes come from the unpermute-backward kernel
  return launch_rowcol(SrcGatherDy{dout, probs, src_row, k, H}, q, a, s);
}

int quant_nv2d(const uint16_t* x, int64_t G, int64_t M, int64_t K, uint8_t* row_codes, uint8_t* row_scales,
               uint8_t* col_codes, uint8_t* col_scales, const float* amax, float* s_out, cudaStream_t s) {
  if ((G * M) / TR > 65535) return MGQ_ERR_UNSUPPORTED;
  const dim3 grid((unsigned)(K / TC), (unsigned)(G * M / TR));
  quant_nv2d_kernel<<<grid, 256, 0, s>>>(x, M, K, row_codes, row_scales, col_codes, col_scales, amax, s_out);
  MGQ_LAUNCH_CHECK();
  return MGQ_OK;
}

}  // namespace mgq
