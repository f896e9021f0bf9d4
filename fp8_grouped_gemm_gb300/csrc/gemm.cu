// Grouped FP8 GEMM on the Blackwell tensor cores (tcgen05), one launch for
// all experts over variable per-expert row counts.
//
// The grouped GEMM of the routed-expert layer ("--moe-grouped-gemm",
// TEGroupedMLP: "[BUG] Loss difference when training with FP8 vs. BF16 MoE",
// Megatron-LM issue #1152), fed by dynamic quantisation ("float8 moe training
// conversion API prototype", pytorch/ao PR #2275), with MXFP8 block scales or
// per-tensor scales ("Numerical fix for moe single grouped weight with fp8 fp4
// primary weight and grad norm spikes", Megatron-LM PR #5487, coverage
// matrix), and the backward GEMMs on the column-wise copies ("FP8BlockQuantizer
// not work on TE", TransformerEngine issue #2393, 128x1 blocks for backward).
//
// Design (one CTA per SM, persistent):
//   warp 0     TMA producer: 128x128 A tile + 256x128 B tile per stage (128-byte
//              swizzle), plus the 512-byte E8M0 scale chunks (bulk copies)
//   warp 1     allocates tensor memory; lane 0 issues tcgen05.cp (scales to
//              tensor memory) and tcgen05.mma (M=128, N=256, K=32 each)
//   warps 2-9  epilogue: tcgen05.ld of the f32 accumulator into registers, release
//              of the accumulator, then scale, convert, store
// The tile scheduler walks the expert offset array; every role derives the
// same tile sequence from it. Every mbarrier wait is bounded: on a timeout the
// kernel records MGQ_ERR_TIMEOUT, all roles leave their loops, tensor memory is
// freed and the kernel returns.
// The dSwiGLU instantiations leave the plain epilogue after their `continue`
// unreachable by design.
#pragma nv_diag_suppress 128
#include <atomic>
#include <cstdlib>

#include "device_common.cuh"
#include "mgq_internal.h"
#include "ptx_sm100.cuh"

namespace mgq {
namespace {

constexpr int BM = 128, BN = 256, BK = 128;     // BK: bytes = fp8 elements
constexpr int STAGES = 4;
constexpr int kThreads = 320;     // warp 0 TMA, warp 1 MMA, warps 2-9 epilogue
// The 1-CTA kernel with float32 block scales (kind 2) runs 384 threads: warp 0
// TMA, warp 1 MMA, warps 2-3 idle, warps 4-11 epilogue. After the prologue the
// first warpgroup gives up registers (setmaxnreg) to the two epilogue
// warpgroups, whose promotion keeps a 128-column float32 accumulator plus two
// tensor-memory loads in flight. The split needs kBlkRegLaunch registers a
// thread at launch (128 x kBlkRegLow + 256 x kBlkRegHigh <= 384 x that); the
// launch checks the compiled kernel's count first.
__host__ __device__ constexpr int threads_of(int kind) { return kind == 2 ? 384 : kThreads; }
__host__ __device__ constexpr int epi_warp0(int kind) { return kind == 2 ? 4 : 2; }
constexpr int kBlkRegLow = 40, kBlkRegHigh = 208, kBlkRegLaunch = 152;
static_assert(128 * kBlkRegLow + 256 * kBlkRegHigh <= 384 * kBlkRegLaunch, "register split");
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kSfaCol = 256;
// scale bytes and tensor-memory scale columns per stage (MX: one chunk per
// 128 rows; NVFP4: four)
__host__ __device__ constexpr uint32_t sfa_bytes(int kind) { return kind == 3 ? 2048u : 512u; }
__host__ __device__ constexpr uint32_t sfa_cols(int kind) { return kind == 3 ? 16u : 4u; }
__host__ __device__ constexpr uint32_t sfb_col0(int kind) { return kSfaCol + sfa_cols(kind) * 4; }
constexpr uint64_t kWaitNs = 2000000000ull;     // default wait limit, 2 s: far beyond any tile
constexpr int kMaxE = 1024;

constexpr uint32_t kABytes = BM * BK, kBBytes = BN * BK;
// B scale bytes per stage: MX the two 512-byte chunks of the 256 B rows;
// NVFP4 room for the stage's slice of a scale image (its 8 chunks, two row
// blocks x the stage's 4 MMAs, each four times over: mgq_nv_scale_image),
// of which the compact chunks use the first 4 KB; none for the other kinds
__host__ __device__ constexpr uint32_t sfb_bytes(int kind) {
  return kind == 3 ? 2 * 4 * 4 * 512u : kind == 0 ? 2 * 512u : 0u;
}
// per stage: A + B tiles and the scale chunks (MX 512 + 1024 bytes, NVFP4 2048 + 16384)
__host__ __device__ constexpr uint32_t sf_stage_bytes(int kind) {
  return kind == 0 || kind == 3 ? sfa_bytes(kind) + sfb_bytes(kind) : 0u;
}
// epilogue staging for TMA stores: per warp 32 rows x 64 bytes, in two slots
// for NVFP4 read with compact B scales (whose short contractions leave little
// mainloop to hide each store's read-out behind); one slot otherwise (NVFP4
// with a B scale image gives the room to the image's 16 KB a stage; the other
// kinds have no shared memory to spare)
constexpr uint32_t kStageOut = 32 * 64;
__host__ __device__ constexpr uint32_t staging_slots(int kind, bool img = true) {
  return kind == 3 && !img ? 2u : 1u;
}
// NVFP4 B scale bytes a stage actually used: the image slice or the compact chunks
__host__ __device__ constexpr uint32_t nv_sfb_stage(bool img) { return img ? 8 * 4 * 512u : 8 * 512u; }
// float32 block scales (kind 2) in contract mode (wgrad): the accumulator
// lives in the epilogue's registers, so the MMA can run only two stages ahead
// while a tile's 128 KB of float32 output is stored; each warp stages half its
// tile slice at once in 8 KB, swizzled, and moves on while the TMA stores
// drain it. That takes the shared memory of one pipeline stage; in rows mode
// (bf16 output, long contractions) the fourth stage is worth more.
constexpr uint32_t kStageWide = 32 * 256;
__host__ __device__ constexpr bool wide_staging(int kind, int mode) { return kind == 2 && mode == 1; }
__host__ __device__ constexpr uint32_t staging_bytes(int kind, int mode) {
  return wide_staging(kind, mode) ? 8 * kStageWide : 8 * kStageOut * staging_slots(kind);
}
// pipeline depth: NVFP4's larger scale chunks leave room for 3 stages next to
// the staging buffers (its 128-byte stages hold 256 elements of K); so do the
// wide staging buffers
__host__ __device__ constexpr int stages_of(int kind, int mode) {
  return kind == 3 || wide_staging(kind, mode) ? 3 : STAGES;
}
// float32 block scales (kind 2): a ring of kBlkSlots slots, one per contraction
// stage, each with the stage's 128 A row scales and (contract mode) the 256
// B column scales of the tile, bulk-copied by the producer and read by the
// epilogue warps from shared memory. The ring is deeper than the operand ring
// plus the two tensor-memory buffers, so its slots are always free in time.
constexpr uint32_t kBlkSlots = 8, kBlkSlotFloats = 128 + BN;
__host__ __device__ constexpr uint32_t blk_ring_bytes(int kind) { return kind == 2 ? kBlkSlots * kBlkSlotFloats * 4 : 0u; }
__host__ __device__ constexpr size_t smem_bytes(int kind, int mode) {
  return 1024 /*align slack*/ + stages_of(kind, mode) * (size_t)(kABytes + kBBytes + sf_stage_bytes(kind)) +
         staging_bytes(kind, mode) + blk_ring_bytes(kind) + 256 /*barriers*/ + (kMaxE + 8) * 4;
}
// NVFP4 with compact B scales: 4 KB of B scales a stage and two staging slots
__host__ __device__ constexpr size_t smem_bytes_nv_compact(int mode) {
  return 1024 + stages_of(3, mode) * (size_t)(kABytes + kBBytes + sfa_bytes(3) + nv_sfb_stage(false)) +
         8 * kStageOut * staging_slots(3, false) + 256 + (kMaxE + 8) * 4;
}
static_assert(smem_bytes(2, 0) <= 232448 && smem_bytes(2, 1) <= 232448, "blockwise kernel exceeds the shared memory");
static_assert(smem_bytes(3, 0) <= 232448 && smem_bytes(3, 1) <= 232448, "NVFP4 kernel exceeds the shared memory");
static_assert(smem_bytes_nv_compact(0) <= smem_bytes(3, 0) && smem_bytes_nv_compact(1) <= smem_bytes(3, 1),
              "the compact NVFP4 layout fits the launch's shared-memory limit");
static_assert((3 * nv_sfb_stage(false)) % 1024 == 0, "the compact B scale stages keep the tiles aligned");
static_assert(smem_bytes(0, 0) <= 232448 && smem_bytes(0, 1) <= 232448, "MX kernel exceeds the shared memory");
static_assert((STAGES * sfb_bytes(0)) % 1024 == 0 && (3 * sfb_bytes(3)) % 1024 == 0,
              "the B scale stages keep the operand tiles 1024-byte aligned");
static_assert(kBlkSlots >= STAGES + 2, "the scale ring must cover the operand ring and both partial buffers");

enum { kModeRows = 0, kModeContract = 1 };
// operand scaling handled by the kernel: E8M0 block scales in the MMA, one
// float32 scale per tensor (epilogue), or float32 1x128 x 128x128 block scales
// (promotion: one 128-deep partial product per stage, scaled and summed in
// registers by the epilogue warps)
enum { kKindMX = 0, kKindTensor = 1, kKindBlock = 2, kKindNV = 3 };
// NVFP4 (kKindNV): a 128-byte stage holds 256 e2m1 elements = 4 MMAs of K=64,
// each with 4 ue4m3 scales per row (one 512-byte scale chunk per 128 rows)

struct GemmParams {
  const int32_t* offsets;
  int E;
  int64_t N;          // rows: output columns; contract: output rows
  int64_t K;          // rows: contraction length; contract: output columns
  int64_t R_cap;
  const uint8_t* sfa;
  int64_t sfa_kb4;    // 512-byte scale chunks per 128-row tile of A
  const uint8_t* sfb;
  int64_t sfb_kb4;
  const uint8_t* sfb_img;  // NVFP4: B's scale image (mgq_nv_scale_image), or null
  const float* sa;    // tensor: s_a; block: scale_inv_a [K/128][sa_ld]; NVFP4: s_g of A
  const float* sb;    // tensor: s_b per expert; block rows mode: scale_inv_b [E][N/128][K/128], block
                      // contract mode: scale_inv_b [R_cap/128][sb_ld] (one per column and 128 rows);
                      // NVFP4: s_g per expert
  int64_t sa_ld;
  int64_t sb_ld;
  void* out;
  int64_t ldo;
  int out_f32;
  float beta;
  uint32_t idesc;
  int tma_store;      // write the output through TMA stores
  int a_mn, b_mn;     // pair kernel: operand stored MN-major (contraction down the rows)
  int kdiv;           // contract mode: group rows per byte of the operands (2: e2m1)
  int64_t b_half2;    // rows from the first to the second 128-row half of a B tile
                      // (128; SwiGLU: F, the up rows matching the gate rows)
  // SwiGLU epilogue (gate/up GEMM): h = bf16(silu(g) u) of the bf16-rounded
  // accumulator columns, quantised row-wise; the plain output (g | u) only
  // when `out` is set
  int swiglu;
  int64_t F;
  uint8_t* h_codes;   // [R_cap, F]
  uint8_t* h_scales;  // MX: tiled E8M0 scales of [R_cap, F]
  const float* h_scale;  // per-tensor: the scale multiplying h
  float* h_amax;      // per-tensor: max |h| (atomically raised), or null
  uint16_t* h_bf16;   // [R_cap, F] or null (dSwiGLU: [R_cap, 2F])
  int h_dtype, h_rceil;
  // dSwiGLU epilogue (down-projection dgrad, per-tensor): [dG | dU] from
  // dh = bf16(acc) and the forward's g | u, quantised row-wise into h_codes
  // [R_cap, 2F] with h_scale; dh itself only when `out` is set
  int dswiglu;
  const uint16_t* gu_in;   // [R_cap, 2F]
  // MX column-wise copy of h (SwiGLU) or of [dG | dU] (dSwiGLU), written by
  // the epilogue: codes [C, c_ld] (C = F or 2F, c_ld = R_cap) with E8M0 scales
  // per 32 rows (the 32 rows of one epilogue warp), tiled; null = none
  uint8_t* c_codes;
  uint8_t* c_scales;
  int64_t c_ld;
  int debug_stall;    // failure-detection test: the producer issues no loads, so
                      // every consumer wait runs out and reports MGQ_ERR_TIMEOUT
  uint64_t wait_ns;   // limit of every mbarrier wait
  int* err;
};

struct Tile {
  int e;
  int nst;            // contraction stages (128 each)
  int64_t row_a, row_b, kx0, out_row, out_col;
};

// Order of an expert's (N tile, M tile) pairs in rows mode: bands of kBandN N
// tiles; inside a band the N tiles run fastest, then the M tiles. A wave of
// consecutive tiles then covers a block about kBandN wide and a few M tiles
// high, and the waves of one band reuse its B tiles from L2, so A is read
// once per band instead of once per wave (the operand that re-streamed when
// the M tiles ran fastest over a whole expert: the down forward's h and the
// gate/up dgrad's dY, larger than L2 per expert).
constexpr int64_t kBandN = 8;
__device__ __forceinline__ void band_order(int64_t local, int64_t mt, int64_t nN, int64_t& n, int64_t& m) {
  const int64_t band = local / (kBandN * mt), r = local - band * (kBandN * mt);
  const int64_t gn = min(kBandN, nN - band * kBandN);    // the last band may be narrower
  m = r / gn;
  n = band * kBandN + (r - m * gn);
}

// Tile t of the sequence. kModeRows: tiles ordered expert, then N bands
// (band_order); kModeContract (wgrad): expert, output-row tile, output-column
// tile (columns fastest).
template <int MODE>
__device__ __forceinline__ bool get_tile(const int32_t* s_off, int E, const GemmParams& p, int64_t t, int& ecur,
                                         Tile& tl) {
  if (MODE == kModeRows) {
    const int64_t nN = p.N / BN;
    const int64_t total = (int64_t)(s_off[E] / BM) * nN;
    if (t >= total) return false;
    while (ecur < E - 1 && (int64_t)(s_off[ecur + 1] / BM) * nN <= t) ++ecur;
    const int e = ecur;
    const int64_t mt = (s_off[e + 1] - s_off[e]) / BM;
    const int64_t local = t - (int64_t)(s_off[e] / BM) * nN;
    int64_t n, m;
    band_order(local, mt, nN, n, m);
    tl.e = e;
    tl.nst = (int)(p.K / BK);
    tl.row_a = s_off[e] + BM * m;
    // SwiGLU: gate rows 128 n.. and (b_half2 = F later) the matching up rows
    tl.row_b = (int64_t)e * p.N + (p.swiglu ? 128 : BN) * n;
    tl.kx0 = 0;
    tl.out_row = tl.row_a;
    tl.out_col = (p.swiglu ? 128 : BN) * n;
  } else {
    const int64_t mN = p.N / BM, nK = p.K / BN;
    const int64_t tpe = mN * nK;
    if (t >= tpe * E) return false;
    const int e = (int)(t / tpe);
    const int64_t local = t % tpe;
    const int64_t m = local / nK, n = local % nK;
    tl.e = e;
    // a stage covers BK bytes of the group's rows (2 BK rows for e2m1)
    tl.nst = (s_off[e + 1] - s_off[e]) / (BK * p.kdiv);
    tl.row_a = BM * m;
    tl.row_b = BN * n;
    tl.kx0 = s_off[e] / p.kdiv;
    tl.out_row = (int64_t)e * p.N + BM * m;
    tl.out_col = BN * n;
  }
  return true;
}

// A warp's TMA-store staging: `nslots` buffers of 32 rows x 64 bytes used in
// turn. A row of `rowbytes` (32 or 64) per lane is filled 16 bytes at a time;
// after its last piece the whole 32-row box goes out as one TMA store. Before a
// buffer is refilled, the store that last used it has finished reading it.
// Every lane of the warp calls put (the counter stays warp-uniform).
struct Stager {
  uint8_t* base;
  uint32_t nslots;
  uint32_t n;
  __device__ __forceinline__ void put(uint32_t lane, int j, uint4 v, const CUtensorMap* m, int64_t x, int32_t y,
                                      int rowbytes) {
    uint8_t* buf = base + (nslots > 1 ? (n & 1u) * kStageOut : 0u);
    if (j == 0) {
      if (lane == 0) {
        if (nslots > 1) ptx::bulk_wait_read1();
        else ptx::bulk_wait_read0();
      }
      __syncwarp();
    }
    reinterpret_cast<uint4*>(buf + lane * rowbytes)[j] = v;
    if (j == rowbytes / 16 - 1) {
      ptx::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        ptx::tma_store_2d(m, buf, (int32_t)x, y);
        ptx::bulk_commit();
      }
      ++n;
    }
  }
};

// Stores one thread's 128 accumulator columns (its row `orow`, columns col0..)
// scaled by alpha: through TMA (the warp stages 32 rows x 64 bytes at a time in
// `stg`; whole lines reach memory) or, when accumulating into float32 (beta) or
// without staging, directly from registers.
__device__ __forceinline__ void epilogue_store(const GemmParams& p, const uint32_t (&r)[4][32], float alpha,
                                               int64_t orow, int64_t col0, bool use_tma, Stager& sg,
                                               const CUtensorMap* tmO, int32_t y0, uint32_t lane) {
  if (use_tma) {
    // 64-byte column chunks: 8 (float32) or 4 (bf16); fully unrolled so the
    // accumulator registers are indexed statically
    auto put = [&](int ch, int j, uint4 v, int ncols) { sg.put(lane, j, v, tmO, col0 + ch * ncols, y0, 64); };
    if (p.out_f32) {
#pragma unroll
      for (int ch = 0; ch < 8; ++ch)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int c = ch >> 1, i0 = (ch & 1) * 16 + 4 * j;
          put(ch, j,
              make_uint4(__float_as_uint(__uint_as_float(r[c][i0]) * alpha),
                         __float_as_uint(__uint_as_float(r[c][i0 + 1]) * alpha),
                         __float_as_uint(__uint_as_float(r[c][i0 + 2]) * alpha),
                         __float_as_uint(__uint_as_float(r[c][i0 + 3]) * alpha)),
              16);
        }
    } else {
#pragma unroll
      for (int ch = 0; ch < 4; ++ch)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int i0 = 8 * j;
          uint4 v;
          v.x = pack_bf16x2(__uint_as_float(r[ch][i0]) * alpha, __uint_as_float(r[ch][i0 + 1]) * alpha);
          v.y = pack_bf16x2(__uint_as_float(r[ch][i0 + 2]) * alpha, __uint_as_float(r[ch][i0 + 3]) * alpha);
          v.z = pack_bf16x2(__uint_as_float(r[ch][i0 + 4]) * alpha, __uint_as_float(r[ch][i0 + 5]) * alpha);
          v.w = pack_bf16x2(__uint_as_float(r[ch][i0 + 6]) * alpha, __uint_as_float(r[ch][i0 + 7]) * alpha);
          put(ch, j, v, 32);
        }
    }
    return;
  }
  if (p.out_f32) {
    float* o = static_cast<float*>(p.out) + orow * p.ldo + col0;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
#pragma unroll
      for (int i = 0; i < 32; i += 4) {
        float4 v = make_float4(__uint_as_float(r[c][i]) * alpha, __uint_as_float(r[c][i + 1]) * alpha,
                               __uint_as_float(r[c][i + 2]) * alpha, __uint_as_float(r[c][i + 3]) * alpha);
        if (p.beta != 0.0f) {
          const float4 old = *reinterpret_cast<const float4*>(o + c * 32 + i);
          v.x += p.beta * old.x; v.y += p.beta * old.y; v.z += p.beta * old.z; v.w += p.beta * old.w;
        }
        *reinterpret_cast<float4*>(o + c * 32 + i) = v;
      }
    }
  } else {
    uint16_t* o = static_cast<uint16_t*>(p.out) + orow * p.ldo + col0;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
#pragma unroll
      for (int i = 0; i < 32; i += 8) {
        uint4 v;
        v.x = pack_bf16x2(__uint_as_float(r[c][i]) * alpha, __uint_as_float(r[c][i + 1]) * alpha);
        v.y = pack_bf16x2(__uint_as_float(r[c][i + 2]) * alpha, __uint_as_float(r[c][i + 3]) * alpha);
        v.z = pack_bf16x2(__uint_as_float(r[c][i + 4]) * alpha, __uint_as_float(r[c][i + 5]) * alpha);
        v.w = pack_bf16x2(__uint_as_float(r[c][i + 6]) * alpha, __uint_as_float(r[c][i + 7]) * alpha);
        *reinterpret_cast<uint4*>(o + c * 32 + i) = v;
      }
    }
  }
}

// Stores one warp's 32 rows x 128 accumulator columns (kind 2: alpha is 1)
// through its 8 KB staging buffer `stg` and TMA stores of 32 rows x 128 bytes
// with the 128-byte swizzle (16-byte chunk j of row l at chunk j ^ (l % 8):
// the eight lanes of each shared-memory phase hit distinct banks). bf16 goes
// out in one round of two boxes, float32 in two; a round first waits until
// the stores that last read the buffer have read it.
__device__ __forceinline__ void epilogue_store_wide(const GemmParams& p, const uint32_t (&r)[4][32], uint8_t* stg,
                                                    const CUtensorMap* tmO, int64_t col0, int32_t y0, uint32_t lane) {
  auto chunk = [&](int b, int j) -> uint4* {
    return reinterpret_cast<uint4*>(stg + b * 4096 + lane * 128 + ((j ^ (lane & 7)) << 4));
  };
  auto issue = [&](int x0, int ncols) {
    ptx::fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      ptx::tma_store_2d(tmO, stg, (int32_t)(col0 + x0), y0);
      ptx::tma_store_2d(tmO, stg + 4096, (int32_t)(col0 + x0 + ncols), y0);
      ptx::bulk_commit();
    }
  };
  auto wait_buffer = [&]() {
    if (lane == 0) ptx::bulk_wait_read0();
    __syncwarp();
  };
  if (p.out_f32) {
#pragma unroll
    for (int rd = 0; rd < 2; ++rd) {
      wait_buffer();
#pragma unroll
      for (int b = 0; b < 2; ++b)
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int c = 2 * rd + b;      // columns 32 c .. 32 c + 31
          *chunk(b, j) = make_uint4(r[c][4 * j], r[c][4 * j + 1], r[c][4 * j + 2], r[c][4 * j + 3]);
        }
      issue(64 * rd, 32);
    }
  } else {
    wait_buffer();
#pragma unroll
    for (int b = 0; b < 2; ++b)
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int c = 2 * b + j / 4, i = (j % 4) * 8;     // columns 64 b + 8 j ..
        *chunk(b, j) = make_uint4(
            pack_bf16x2(__uint_as_float(r[c][i]), __uint_as_float(r[c][i + 1])),
            pack_bf16x2(__uint_as_float(r[c][i + 2]), __uint_as_float(r[c][i + 3])),
            pack_bf16x2(__uint_as_float(r[c][i + 4]), __uint_as_float(r[c][i + 5])),
            pack_bf16x2(__uint_as_float(r[c][i + 6]), __uint_as_float(r[c][i + 7])));
      }
    issue(0, 64);
  }
}

// Accumulator column of a thread's chunk c (of 4 x 32): the 128-column half
// `half` of the tile, or for SwiGLU the gate columns half*64.. (c = 0, 1) and
// the matching up columns 128 + half*64.. (c = 2, 3).
__device__ __forceinline__ uint32_t acc_col(int swiglu, uint32_t half, int c) {
  return swiglu ? (c < 2 ? half * 64 + 32 * c : 128 + half * 64 + 32 * (c - 2)) : half * 128 + 32 * c;
}

// 32 x 32 transpose of 16-bit values across a warp. On entry lane l holds
// row l as 16 words (word j: columns 2j and 2j + 1, the first in the low
// half); on exit lane l holds column l (word j: rows 2j and 2j + 1). Round k
// exchanges, with lane l ^ 2^k, the elements whose row and column indices
// differ in bit k (whole words for k >= 1, half words for k = 0); after the
// five rounds element (r, c) has moved to lane c, position r.
__device__ __forceinline__ void warp_transpose32_b16(uint32_t (&w)[16], uint32_t lane) {
#pragma unroll
  for (int k = 4; k >= 1; --k) {
    const int m = 1 << (k - 1);               // the word-index bit of column bit k
    const bool up = (lane >> k) & 1u;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      if (j & m) continue;
      const uint32_t send = up ? w[j] : w[j | m];
      const uint32_t recv = __shfl_xor_sync(0xFFFFFFFFu, send, 1 << k);
      if (up) w[j] = recv;
      else w[j | m] = recv;
    }
  }
  // round 0: an even lane trades its odd columns (high halves) for the odd
  // lane's even columns (low halves), two words per exchange
  const bool odd = lane & 1u;
#pragma unroll
  for (int j = 0; j < 16; j += 2) {
    const uint32_t send = odd ? __byte_perm(w[j], w[j + 1], 0x5410) : __byte_perm(w[j], w[j + 1], 0x7632);
    const uint32_t recv = __shfl_xor_sync(0xFFFFFFFFu, send, 1);
    if (odd) {
      w[j] = __byte_perm(w[j], recv, 0x3254);
      w[j + 1] = __byte_perm(w[j + 1], recv, 0x3276);
    } else {
      w[j] = __byte_perm(w[j], recv, 0x5410);
      w[j + 1] = __byte_perm(w[j + 1], recv, 0x7610);
    }
  }
}

// E8M0 block quantisation of 32 bf16 values held as pairs: the block's
// exponent from max |x| (NaN and infinity give the NaN marker), the codes
// cast(x * 2^-e) as eight words (element 0 in the low byte of word 0)
__device__ __forceinline__ uint32_t mx_block32(const uint32_t (&w)[16], bool e5, bool rceil, uint32_t (&cw)[8]) {
  uint32_t acc = 0;
#pragma unroll
  for (int i = 0; i < 16; ++i) acc = absmax_acc_bf16x2(acc, w[i]);
  const int e = mx_exponent(fold_bf16x2(absmax_bf16x2_final(acc)),
                            e5 ? FmtInfo<MGQ_E5M2>::emax : FmtInfo<MGQ_E4M3>::emax, rceil);
  const float mult = mx_multiplier(e);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float a0 = __fmul_rn(bf16_lo(w[2 * i]), mult), a1 = __fmul_rn(bf16_hi(w[2 * i]), mult);
    const float a2 = __fmul_rn(bf16_lo(w[2 * i + 1]), mult), a3 = __fmul_rn(bf16_hi(w[2 * i + 1]), mult);
    cw[i] = e5 ? cvt_fp8x4<MGQ_E5M2>(a0, a1, a2, a3) : cvt_fp8x4<MGQ_E4M3>(a0, a1, a2, a3);
  }
  return mx_scale_code(e);
}

// Column-wise MX copy of a warp's 32 rows (row0..row0+31, one per lane) and 32
// columns (col..col+31, one 32-bit pair of each per word of `w`, the lane's own
// row): after the warp transpose lane l holds column col + l, one E8M0 block of
// 32 rows, whose codes (32 bytes) go to c_codes[col + l][row0..] and whose
// scale to the tiled scales of [C, c_ld]. `w` is clobbered. Warp-collective.
__device__ __forceinline__ void col_copy_mx32(const GemmParams& p, uint32_t (&w)[16], int64_t col, int64_t row0,
                                              uint32_t lane) {
  warp_transpose32_b16(w, lane);
  uint32_t cw[8];
  const uint32_t code = mx_block32(w, p.h_dtype == MGQ_E5M2, p.h_rceil != 0, cw);
  const int64_t c = col + lane;
  p.c_scales[tiled_scale_offset(c, row0 / 32, p.c_ld / 128)] = (uint8_t)code;
  uint4* dst = reinterpret_cast<uint4*>(p.c_codes + c * p.c_ld + row0);
  dst[0] = make_uint4(cw[0], cw[1], cw[2], cw[3]);
  dst[1] = make_uint4(cw[4], cw[5], cw[6], cw[7]);
}

// SwiGLU epilogue of the gate/up GEMM for one thread's row `orow` and ffn
// columns f0..f0+63: g, u = bf16(acc * alpha) (the values the plain GEMM would
// write), h = bf16(silu(g) u), quantised with the GEMM's scaling kind (MX:
// E8M0 per 32 columns; per-tensor: *p.h_scale, max |h| into tam). The codes,
// and (p.out set) g and u, go out through TMA stores from the warp's staging
// buffer; MX scales and the optional bf16 h by plain stores. MX with
// p.c_codes: also the column-wise copy of h (blocks of the warp's 32 rows).
template <int KIND, bool COL = true>
__device__ __forceinline__ void epilogue_swiglu(const GemmParams& p, const uint32_t (&r)[4][32], float alpha,
                                                int64_t orow, int64_t f0, Stager& sg, const CUtensorMap* tmO,
                                                const CUtensorMap* tmH, int32_t y0, uint32_t lane, uint32_t& tam) {
  auto stage = [&](int j, uint4 v, const CUtensorMap* m, int64_t x) { sg.put(lane, j, v, m, x, y0, 64); };
  auto bf = [&](uint32_t bits) { return round_bf16(__uint_as_float(bits) * alpha); };
  if (p.out) {
    // g and u as bf16: columns f0 + 32c and F + f0 + 32c of [R_cap, 2F]
#pragma unroll
    for (int c = 0; c < 4; ++c)
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint32_t* v = &r[c][8 * j];
        stage(j,
              make_uint4(pack_bf16x2(bf(v[0]), bf(v[1])), pack_bf16x2(bf(v[2]), bf(v[3])),
                         pack_bf16x2(bf(v[4]), bf(v[5])), pack_bf16x2(bf(v[6]), bf(v[7]))),
              tmO, (c < 2 ? 0 : p.F) + f0 + 32 * (c & 1));
      }
  }
  const float ts = KIND == kKindTensor ? *p.h_scale : 1.0f;   // (NVFP4: h_scale receives s_g later)
  const bool e5 = p.h_dtype == MGQ_E5M2;
  uint32_t hw[16];        // the 64 codes
  uint32_t sc2 = 0;       // MX: the two block scales
#pragma unroll
  for (int c = 0; c < 2; ++c) {
    uint32_t hp[16];      // h as bf16 pairs (exact)
    uint32_t am2 = 0;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      // (the pair conversion rounds each value to bf16 once)
      hp[i] = pack_bf16x2(swiglu_f32(bf(r[c][2 * i]), bf(r[2 + c][2 * i])),
                          swiglu_f32(bf(r[c][2 * i + 1]), bf(r[2 + c][2 * i + 1])));
      am2 = absmax_bf16x2(am2, hp[i]);
    }
    if (KIND == kKindNV) {
      // NVFP4 needs the amax of all of h before any block is cast: h goes out
      // in bf16 (tmH maps h_bf16) for the second pass, and into tam
#pragma unroll
      for (int q = 0; q < 4; ++q) stage(q, make_uint4(hp[4 * q], hp[4 * q + 1], hp[4 * q + 2], hp[4 * q + 3]), tmH,
                                        f0 + 32 * c);
      tam = max(tam, fold_bf16x2(am2));
    } else {
      if (p.h_bf16) {
        uint4* d = reinterpret_cast<uint4*>(p.h_bf16 + orow * p.F + f0 + 32 * c);
#pragma unroll
        for (int q = 0; q < 4; ++q) d[q] = make_uint4(hp[4 * q], hp[4 * q + 1], hp[4 * q + 2], hp[4 * q + 3]);
      }
      const uint32_t am = fold_bf16x2(am2);
      float mult = ts;
      if (KIND == kKindMX) {
        const int e = mx_exponent(am, e5 ? FmtInfo<MGQ_E5M2>::emax : FmtInfo<MGQ_E4M3>::emax, p.h_rceil != 0);
        mult = mx_multiplier(e);
        sc2 |= mx_scale_code(e) << (8 * c);
      } else {
        tam = max(tam, am);
      }
#pragma unroll
      for (int w = 0; w < 8; ++w) {
        const float a0 = __fmul_rn(bf16_lo(hp[2 * w]), mult), a1 = __fmul_rn(bf16_hi(hp[2 * w]), mult);
        const float a2 = __fmul_rn(bf16_lo(hp[2 * w + 1]), mult), a3 = __fmul_rn(bf16_hi(hp[2 * w + 1]), mult);
        hw[8 * c + w] = e5 ? cvt_fp8x4<MGQ_E5M2>(a0, a1, a2, a3) : cvt_fp8x4<MGQ_E4M3>(a0, a1, a2, a3);
      }
      // MX column-wise copy of these 32 columns over the warp's 32 rows
      if (COL && KIND == kKindMX && p.c_codes) col_copy_mx32(p, hp, f0 + 32 * c, y0, lane);
    }
  }
  if (KIND != kKindNV) {
#pragma unroll
    for (int j = 0; j < 4; ++j) stage(j, make_uint4(hw[4 * j], hw[4 * j + 1], hw[4 * j + 2], hw[4 * j + 3]), tmH, f0);
    if (KIND == kKindMX)
      *reinterpret_cast<uint16_t*>(p.h_scales + tiled_scale_offset(orow, f0 / 32, p.F / 128)) = (uint16_t)sc2;
  }
}

// g and u of 16 columns (col0 + 16 c ..) of one row of the forward's gu
__device__ __forceinline__ void dswiglu_load_gu(const GemmParams& p, int64_t orow, int64_t col0, int c,
                                                uint4 (&gq)[2], uint4 (&uq)[2]) {
  const uint16_t* grow = p.gu_in + orow * 2 * p.F + col0 + 16 * c;
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    gq[q] = __ldg(reinterpret_cast<const uint4*>(grow) + q);
    uq[q] = __ldg(reinterpret_cast<const uint4*>(grow + p.F) + q);
  }
}

// g / u staging of the per-tensor dSwiGLU epilogue (2-CTA kernel): a warp's
// 4 KB slot holds, for its 32 rows and 32 columns, g (bytes 0..63 of a row's
// 128) and u (64..127) in 16-byte units, unit j of row r at r * 128 + 16 (j ^
// (r & 7)). Each copy instruction moves four whole row segments (8 lines, 64
// bytes each) where a lane-per-row load would touch 32 lines for 16 bytes each;
// the swizzle keeps both the copies and the lanes' row reads free of bank
// conflicts.
constexpr uint32_t kGuSlot = 4096;
__device__ __forceinline__ void gu_stage_issue(const GemmParams& p, uint32_t slot, int64_t row0, int64_t col,
                                               uint32_t lane) {
  const uint32_t j = lane & 7;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint32_t r = 4 * i + (lane >> 3);
    const uint16_t* src = p.gu_in + (row0 + r) * 2 * p.F + col + (j >> 2) * p.F + (j & 3) * 8;
    ptx::cp_async16(slot + r * 128 + 16 * (j ^ (r & 7)), src);
  }
  ptx::cp_async_commit();
}
// the lane's row of a landed slot: g and u of columns 0..15 and 16..31
__device__ __forceinline__ void gu_stage_read(const uint8_t* slot, uint32_t lane, uint4 (&g0)[2], uint4 (&u0)[2],
                                              uint4 (&g1)[2], uint4 (&u1)[2]) {
  const uint8_t* row = slot + lane * 128;
  auto unit = [&](uint32_t jj) { return *reinterpret_cast<const uint4*>(row + 16 * (jj ^ (lane & 7))); };
  g0[0] = unit(0); g0[1] = unit(1); g1[0] = unit(2); g1[1] = unit(3);
  u0[0] = unit(4); u0[1] = unit(5); u1[0] = unit(6); u1[1] = unit(7);
}

// dSwiGLU epilogue of the down-projection dgrad (per-tensor) for one thread's
// row `orow` and columns col0..col0+127, in 8 chunks of 16: each reads its
// accumulator columns from tensor memory (`tcol` = the first) and the matching
// g and u of the forward's gu (chunk 0 already in gq / uq, requested by the
// caller before the accumulator was ready; further chunks in pairs, 32 columns
// per request), or with `gslot` (a warp's staging slot, shared-memory address;
// its first 32 columns already requested by the caller) through the slot;
// dh = bf16(acc * alpha), [dG | dU] = dswiglu_bf16, quantised with *p.h_scale
// (max |.| into tam). Codes and (p.out set) dh go out through TMA stores from
// the warp's staging buffer; the optional bf16 dG | dU by plain stores.
// Warp-collective (tensor-memory loads).
__device__ __forceinline__ void epilogue_dswiglu(const GemmParams& p, uint32_t tcol, float alpha, int64_t orow,
                                                 int64_t col0, Stager& sg, const CUtensorMap* tmO,
                                                 const CUtensorMap* tmH, int32_t y0, uint32_t lane, uint32_t& tam,
                                                 uint4 (&gq)[2], uint4 (&uq)[2], uint8_t* gslot = nullptr) {
  auto stage = [&](int j, uint4 v, const CUtensorMap* m, int64_t x) { sg.put(lane, j, v, m, x, y0, 64); };
  const int64_t F = p.F;
  const float ts = *p.h_scale;
  const bool e5 = p.h_dtype == MGQ_E5M2;
  uint32_t cg[16], cu[16];    // codes of four 16-column chunks: dG, dU
  uint32_t dhw[16];           // dh of two chunks as bf16 pairs (the 64-byte rows of its stores)
  uint4 g2[2], u2[2];          // the odd chunk of a pair, requested with the even one
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    if (gslot) {
      if ((c & 1) == 0) {
        // this pair of chunks from the slot, then the next pair into it
        ptx::cp_async_wait_all();
        __syncwarp();
        gu_stage_read(gslot, lane, gq, uq, g2, u2);
        __syncwarp();
        if (c < 6) gu_stage_issue(p, ptx::smem_u32(gslot), orow - lane, col0 + 16 * (c + 2), lane);
      }
    } else {
      if (c > 0 && (c & 1) == 0) dswiglu_load_gu(p, orow, col0, c, gq, uq);
      if ((c & 1) == 0) dswiglu_load_gu(p, orow, col0, c + 1, g2, u2);
    }
    if (c & 1) {
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        gq[q] = g2[q];
        uq[q] = u2[q];
      }
    }
    uint32_t v[16];
    ptx::tmem_ld_32x32b_x16(tcol + 16 * c, v);
    ptx::tmem_ld_wait();
    float d[16];   // dh = bf16(acc * alpha), as float
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const f32x2 pr = mul2(f32x2{__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1])}, f32x2{alpha, alpha});
      const uint32_t w = pack_bf16x2(pr.x, pr.y);
      dhw[8 * (c & 1) + i] = w;
      d[2 * i] = bf16_lo(w);
      d[2 * i + 1] = bf16_hi(w);
    }
    if (p.out && (c & 1)) {   // dh: 32 columns at col0 + 16 (c - 1)
#pragma unroll
      for (int j = 0; j < 4; ++j) stage(j, make_uint4(dhw[4 * j], dhw[4 * j + 1], dhw[4 * j + 2], dhw[4 * j + 3]),
                                        tmO, col0 + 16 * (c - 1));
    }
    uint32_t dgp[8], dup[8];   // bf16 pairs (exact)
    uint32_t am2 = 0;
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const uint32_t gw[4] = {gq[q].x, gq[q].y, gq[q].z, gq[q].w};
      const uint32_t uw[4] = {uq[q].x, uq[q].y, uq[q].z, uq[q].w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int k = 8 * q + 2 * i;
        f32x2 dg, du;
        dswiglu_f32x2(f32x2{d[k], d[k + 1]}, f32x2{bf16_lo(gw[i]), bf16_hi(gw[i])},
                      f32x2{bf16_lo(uw[i]), bf16_hi(uw[i])}, dg, du);
        dgp[4 * q + i] = pack_bf16x2(dg.x, dg.y);
        dup[4 * q + i] = pack_bf16x2(du.x, du.y);
        am2 = absmax_bf16x2(absmax_bf16x2(am2, dgp[4 * q + i]), dup[4 * q + i]);
      }
    }
    tam = max(tam, fold_bf16x2(am2));
    if (p.h_bf16) {
      uint4* og = reinterpret_cast<uint4*>(p.h_bf16 + orow * 2 * F + col0 + 16 * c);
      uint4* ou = reinterpret_cast<uint4*>(p.h_bf16 + orow * 2 * F + F + col0 + 16 * c);
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        og[q] = make_uint4(dgp[4 * q], dgp[4 * q + 1], dgp[4 * q + 2], dgp[4 * q + 3]);
        ou[q] = make_uint4(dup[4 * q], dup[4 * q + 1], dup[4 * q + 2], dup[4 * q + 3]);
      }
    }
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      cg[4 * (c & 3) + w] = e5 ? cvt_fp8x4_bf16_mul<MGQ_E5M2>(dgp[2 * w], dgp[2 * w + 1], ts)
                               : cvt_fp8x4_bf16_mul<MGQ_E4M3>(dgp[2 * w], dgp[2 * w + 1], ts);
      cu[4 * (c & 3) + w] = e5 ? cvt_fp8x4_bf16_mul<MGQ_E5M2>(dup[2 * w], dup[2 * w + 1], ts)
                               : cvt_fp8x4_bf16_mul<MGQ_E4M3>(dup[2 * w], dup[2 * w + 1], ts);
    }
    if ((c & 3) == 3) {   // 64 columns of codes: dG at col0 + 16 (c - 3), dU F further
#pragma unroll
      for (int j = 0; j < 4; ++j) stage(j, make_uint4(cg[4 * j], cg[4 * j + 1], cg[4 * j + 2], cg[4 * j + 3]), tmH,
                                        col0 + 16 * (c - 3));
#pragma unroll
      for (int j = 0; j < 4; ++j) stage(j, make_uint4(cu[4 * j], cu[4 * j + 1], cu[4 * j + 2], cu[4 * j + 3]), tmH,
                                        F + col0 + 16 * (c - 3));
    }

  }
}

// dSwiGLU epilogue of the down-projection dgrad with MX scaling, for one
// thread's row `orow` and dh columns col0..col0+127. dhp holds dh = bf16(acc)
// as pairs (consumed), read from tensor memory before the accumulator was released (so
// this work overlaps the next tile's MMAs). Per 32-column chunk: g and u of
// the forward's gu (the next chunk's requested before this one is worked
// on), [dG | dU] = dswiglu_bf16, the row-wise E8M0 blocks (codes [R_cap, 2F]
// through `tmR`, tiled scales into h_scales), with p.c_codes the column-wise
// blocks of the warp's 32 rows from row0 (codes [2F, R_cap] through `tmC`,
// tiled scales into c_scales), and the optional bf16 dh (p.out) and dG | dU
// (p.h_bf16), all by plain stores (32 bytes of a row per lane).
// Warp-collective.
__device__ __forceinline__ void epilogue_dswiglu_mx(const GemmParams& p, uint32_t (&dhp)[64], int64_t orow,
                                                    int64_t col0, int64_t row0, uint32_t lane) {
  const int64_t F = p.F;
  const bool e5 = p.h_dtype == MGQ_E5M2, rceil = p.h_rceil != 0;
  const uint16_t* grow = p.gu_in + orow * 2 * F + col0;
  uint4 gq[4], uq[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    gq[q] = __ldg(reinterpret_cast<const uint4*>(grow) + q);
    uq[q] = __ldg(reinterpret_cast<const uint4*>(grow + F) + q);
  }
  // a rolled loop keeps the code small: chunk c works on dhp[0..15], then the
  // words of the later chunks move down (static register indices throughout)
#pragma unroll 1
  for (int c = 0; c < 4; ++c) {
    uint32_t dg[16], du[16];   // bf16 pairs (exact)
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint32_t gw[4] = {gq[q].x, gq[q].y, gq[q].z, gq[q].w};
      const uint32_t uw[4] = {uq[q].x, uq[q].y, uq[q].z, uq[q].w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint32_t d = dhp[4 * q + i];
        float g0, g1, u0, u1;
        dswiglu_f32(bf16_lo(d), bf16_lo(gw[i]), bf16_lo(uw[i]), g0, u0);
        dswiglu_f32(bf16_hi(d), bf16_hi(gw[i]), bf16_hi(uw[i]), g1, u1);
        dg[4 * q + i] = pack_bf16x2(g0, g1);
        du[4 * q + i] = pack_bf16x2(u0, u1);
      }
    }
    if (c < 3) {
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        gq[q] = __ldg(reinterpret_cast<const uint4*>(grow + 32 * (c + 1)) + q);
        uq[q] = __ldg(reinterpret_cast<const uint4*>(grow + F + 32 * (c + 1)) + q);
      }
    }
    const int64_t col = col0 + 32 * c;
    if (p.out) {
      uint4* o = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.out) + orow * p.ldo + col);
#pragma unroll
      for (int q = 0; q < 4; ++q) o[q] = make_uint4(dhp[4 * q], dhp[4 * q + 1], dhp[4 * q + 2], dhp[4 * q + 3]);
    }
#pragma unroll
    for (int i = 0; i < 48; ++i) dhp[i] = dhp[i + 16];
    if (p.h_bf16) {
      uint4* og = reinterpret_cast<uint4*>(p.h_bf16 + orow * 2 * F + col);
      uint4* ou = reinterpret_cast<uint4*>(p.h_bf16 + orow * 2 * F + F + col);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        og[q] = make_uint4(dg[4 * q], dg[4 * q + 1], dg[4 * q + 2], dg[4 * q + 3]);
        ou[q] = make_uint4(du[4 * q], du[4 * q + 1], du[4 * q + 2], du[4 * q + 3]);
      }
    }
    uint32_t cw[8];
    const uint32_t sg = mx_block32(dg, e5, rceil, cw);
    uint4* dst = reinterpret_cast<uint4*>(p.h_codes + orow * 2 * F + col);
    dst[0] = make_uint4(cw[0], cw[1], cw[2], cw[3]);
    dst[1] = make_uint4(cw[4], cw[5], cw[6], cw[7]);
    const uint32_t su = mx_block32(du, e5, rceil, cw);
    dst = reinterpret_cast<uint4*>(p.h_codes + orow * 2 * F + F + col);
    dst[0] = make_uint4(cw[0], cw[1], cw[2], cw[3]);
    dst[1] = make_uint4(cw[4], cw[5], cw[6], cw[7]);
    p.h_scales[tiled_scale_offset(orow, col / 32, 2 * F / 128)] = (uint8_t)sg;
    p.h_scales[tiled_scale_offset(orow, (F + col) / 32, 2 * F / 128)] = (uint8_t)su;
    if (p.c_codes) {
      col_copy_mx32(p, dg, col, row0, lane);
      col_copy_mx32(p, du, F + col, row0, lane);
    }
  }
}

// DSW: the down-projection dgrad with the dSwiGLU epilogue (a separate
// instantiation, so the other epilogues keep their registers)
template <int MODE, int KIND, bool DSW = false, bool IMG = false>
__global__ void __launch_bounds__(threads_of(KIND), 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                        const __grid_constant__ CUtensorMap tmO, const __grid_constant__ CUtensorMap tmH,
                        const GemmParams p) {
  constexpr int STG = stages_of(KIND, MODE);
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = ptx::smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  constexpr uint32_t kSfaBytes = sfa_bytes(KIND), kSfbBytes = sfb_bytes(KIND);
  constexpr uint32_t kSfbCol = sfb_col0(KIND);
  // [B scale stages][A stages][B stages][A scale stages][staging]...: the B
  // scale stages (multiples of 1024 bytes) come first, so the operand tiles
  // stay 1024-byte aligned
  // NVFP4: B scales a stage and staging slots follow the kind of B scales
  // (IMG: B's scale image, p.sfb_img; else the compact chunks)
  constexpr bool img = KIND == kKindNV && IMG;
  constexpr uint32_t sfb_stage = KIND == kKindNV ? nv_sfb_stage(img) : kSfbBytes;
  constexpr uint32_t nslots = staging_slots(KIND, img);
  constexpr uint32_t stage_out_bytes = wide_staging(KIND, MODE) ? staging_bytes(KIND, MODE) : 8 * kStageOut * nslots;
  uint8_t* sSFB = smem;
  uint8_t* sA = sSFB + STG * sfb_stage;
  uint8_t* sB = sA + STG * kABytes;
  uint8_t* sSFA = sB + STG * kBBytes;
  uint8_t* sOut = sSFA + STG * (sf_stage_bytes(KIND) - kSfbBytes);   // epilogue staging (TMA stores)
  float* sRing = reinterpret_cast<float*>(sOut + stage_out_bytes);   // block scales
  uint64_t* bars = reinterpret_cast<uint64_t*>(sOut + stage_out_bytes + blk_ring_bytes(KIND));
  uint64_t* full = bars;
  uint64_t* empty = bars + STG;
  uint64_t* tmem_full = bars + 2 * STG;        // [2]
  uint64_t* tmem_empty = bars + 2 * STG + 2;   // [2]
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(bars + 2 * STG + 4);
  volatile int* s_abort = reinterpret_cast<volatile int*>(s_tmem + 1);
  int* s_bad = reinterpret_cast<int*>(s_tmem + 2);
  uint64_t* s_full = bars + 14;                // [kBlkSlots] block-scale slot loaded
  uint64_t* s_empty = bars + 14 + kBlkSlots;   // [kBlkSlots] block-scale slot read by the epilogue
  static_assert(2 * STG + 4 + 2 <= 14 && 14 + 2 * kBlkSlots <= 32, "barrier region");
  int32_t* s_off = reinterpret_cast<int32_t*>(bars + 32);

  const int warp = threadIdx.x >> 5;
  const uint32_t lane = threadIdx.x & 31;
  const int E = p.E;
  constexpr bool NV = KIND == kKindNV;
  constexpr bool MX = KIND == kKindMX || NV;     // block scales through tensor memory
  constexpr bool BLOCK = KIND == kKindBlock;
  // accumulator buffers in tensor memory: two 256-column tiles when no
  // scale-factor columns are needed, else one (columns 256.. hold the scales).
  // In block mode the two buffers hold per-stage partial products.
  constexpr uint32_t kAcc = MX ? 1 : 2;

  constexpr int NT = threads_of(KIND), EW0 = epi_warp0(KIND);
  for (int i = threadIdx.x; i <= E; i += NT) s_off[i] = p.offsets[i];
  if (threadIdx.x == 0) {
    for (int s = 0; s < STG; ++s) {
      ptx::mbar_init(&full[s], 1);
      ptx::mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      ptx::mbar_init(&tmem_full[a], 1);
      ptx::mbar_init(&tmem_empty[a], 8 * 32);
    }
    if (KIND == kKindBlock) {
      for (uint32_t i = 0; i < kBlkSlots; ++i) {
        ptx::mbar_init(&s_full[i], 1);
        ptx::mbar_init(&s_empty[i], 8 * 32);
      }
    }
    *s_abort = 0;
    *s_bad = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    ptx::prefetch_tmap(&tmA);
    ptx::prefetch_tmap(&tmB);
  }
  if (warp == 1) {
    ptx::tmem_alloc(s_tmem, kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  if (threadIdx.x == 0) {
    // the group layout must be 128-row aligned and inside the buffers
    bool bad = s_off[0] != 0;
    // (contract mode over e2m1: whole 256-row stages)
    const int align = MODE == kModeContract ? BM * p.kdiv : BM;
    for (int e = 0; e < E; ++e) bad |= (s_off[e + 1] < s_off[e]) || (s_off[e + 1] % align) != 0;
    bad |= (int64_t)s_off[E] > p.R_cap;
    if (bad) {
      *s_bad = 1;
      report(p.err, MGQ_ERR_INVALID_ARG);
    }
  }
  __syncthreads();
  const uint32_t tmem = *s_tmem;
  const bool run = (*s_bad == 0);

  if (warp < EW0) {
  // (the register budget changes inside each role's branch: code after a
  // setmaxnreg is compiled for that budget only where no other path joins it)
  if (KIND == kKindBlock) ptx::setmaxnreg_dec<kBlkRegLow>();   // to the epilogue warpgroups
  if (run && warp == 0 && lane == 0 && !p.debug_stall) {
    // ------------------------------------------------------------ producer
    int ecur = 0;
    uint32_t it = 0;
    Tile tl;
    for (int64_t t = blockIdx.x; get_tile<MODE>(s_off, E, p, t, ecur, tl); t += gridDim.x) {
      for (int s = 0; s < tl.nst; ++s, ++it) {
        const uint32_t st = it % STG, ph = (it / STG) & 1;
        if (*s_abort) break;
        if (!ptx::mbar_wait(&empty[st], ph ^ 1, p.wait_ns)) {
          report(p.err, MGQ_ERR_TIMEOUT);
          *s_abort = 1;
          break;
        }
        if (BLOCK) {
          // this stage's float32 scales into ring slot it % kBlkSlots (free once
          // the epilogue has promoted stage it - kBlkSlots)
          const uint32_t sl = it % kBlkSlots;
          if (!ptx::mbar_wait(&s_empty[sl], ((it / kBlkSlots) & 1) ^ 1, p.wait_ns)) {
            report(p.err, MGQ_ERR_TIMEOUT);
            *s_abort = 1;
            break;
          }
          const int64_t kb = tl.kx0 / BK + s;
          float* dst = sRing + sl * kBlkSlotFloats;
          ptx::mbar_arrive_expect_tx(&s_full[sl], MODE == kModeContract ? kBlkSlotFloats * 4 : 128 * 4);
          ptx::bulk_load(dst, p.sa + kb * p.sa_ld + tl.row_a, 128 * 4, &s_full[sl]);
          if (MODE == kModeContract) ptx::bulk_load(dst + 128, p.sb + kb * p.sb_ld + tl.out_col, BN * 4, &s_full[sl]);
        }
        // (NVFP4 B scales: the image slice, 16 KB, or the compact chunks, 4 KB)
        const uint32_t bytes = kABytes + kBBytes + (MX ? kSfaBytes + sfb_stage : 0);
        ptx::mbar_arrive_expect_tx(&full[st], bytes);
        const int32_t kx = (int32_t)(tl.kx0 + (int64_t)s * BK);
        ptx::tma_load_2d(sA + st * kABytes, &tmA, &full[st], kx, (int32_t)tl.row_a);
        // B in two 128-row halves (contiguous, or gate and up rows for SwiGLU)
        ptx::tma_load_2d(sB + st * kBBytes, &tmB, &full[st], kx, (int32_t)tl.row_b);
        ptx::tma_load_2d(sB + st * kBBytes + kBBytes / 2, &tmB, &full[st], kx, (int32_t)(tl.row_b + p.b_half2));
        if (MX) {
          // scale chunks of this stage: MX one 512-byte chunk per 128 rows,
          // NVFP4 four consecutive chunks (the 4 MMAs of the stage)
          const int64_t kt = (tl.kx0 / BK + s) * (kSfaBytes / 512);
          const uint8_t* fa = p.sfa + ((tl.row_a / BM) * p.sfa_kb4 + kt) * 512;
          const uint8_t* fb = p.sfb + ((tl.row_b / BM) * p.sfb_kb4 + kt) * 512;
          const uint8_t* fb2 = p.sfb + (((tl.row_b + p.b_half2) / BM) * p.sfb_kb4 + kt) * 512;
          ptx::bulk_load(sSFA + st * kSfaBytes, fa, kSfaBytes, &full[st]);
          if (img) {
            // the stage's 8 KB slice of the image for each B row block
            const int64_t ks = kt / 4, nks = p.sfb_kb4 / 4;
            ptx::bulk_load(sSFB + st * sfb_stage, p.sfb_img + ((tl.row_b / BM) * nks + ks) * 8192, 8192, &full[st]);
            ptx::bulk_load(sSFB + st * sfb_stage + 8192,
                           p.sfb_img + (((tl.row_b + p.b_half2) / BM) * nks + ks) * 8192, 8192, &full[st]);
          } else {
            ptx::bulk_load(sSFB + st * sfb_stage, fb, kSfaBytes, &full[st]);
            ptx::bulk_load(sSFB + st * sfb_stage + kSfaBytes, fb2, kSfaBytes, &full[st]);
          }
        }
      }
      if (*s_abort) break;
    }
  } else if (run && warp == 1 && lane == 0) {
    // ------------------------------------------------------------ MMA issuer
    int ecur = 0;
    uint32_t it = 0, tc = 0;
    Tile tl;
    const uint32_t sA0 = ptx::smem_u32(sA), sB0 = ptx::smem_u32(sB);
    const uint32_t sSFA0 = ptx::smem_u32(sSFA), sSFB0 = ptx::smem_u32(sSFB);
    for (int64_t t = blockIdx.x; get_tile<MODE>(s_off, E, p, t, ecur, tl); t += gridDim.x) {
      if (tl.nst == 0) continue;
      if (*s_abort) break;
      bool ok = true;
      uint32_t a = tc % kAcc;
      if (!BLOCK) {
        const uint32_t aph = (tc / kAcc) & 1;
        if (!ptx::mbar_wait(&tmem_empty[a], aph ^ 1, p.wait_ns)) {
          report(p.err, MGQ_ERR_TIMEOUT);
          *s_abort = 1;
          break;
        }
        ptx::tc_fence_after();
      }
      for (int s = 0; s < tl.nst; ++s, ++it) {
        const uint32_t st = it % STG, ph = (it / STG) & 1;
        if (BLOCK) {
          // every stage gets a fresh partial buffer
          a = tc % kAcc;
          if (!ptx::mbar_wait(&tmem_empty[a], ((tc / kAcc) & 1) ^ 1, p.wait_ns)) {
            report(p.err, MGQ_ERR_TIMEOUT);
            *s_abort = 1;
            ok = false;
            break;
          }
        }
        if (*s_abort || !ptx::mbar_wait(&full[st], ph, p.wait_ns)) {
          report(p.err, MGQ_ERR_TIMEOUT);
          *s_abort = 1;
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t d_tmem = tmem + a * BN;
        const uint32_t sfa_t = tmem + kSfaCol + st * sfa_cols(KIND), sfb_t = tmem + kSfbCol + st * 2 * sfa_cols(KIND);
        if (MX) {
#pragma unroll
          for (uint32_t ch = 0; ch < kSfaBytes / 512; ++ch) {
            ptx::tmem_cp_32x128b_x4(sfa_t + ch * 4, ptx::sdesc_sf(sSFA0 + st * kSfaBytes + ch * 512));
            if (img) {
              // both B row blocks of MMA ch in one copy: 128 rows of 2 x 16
              // bytes, the second 16 bytes 8192 bytes on (the other row block)
              ptx::tmem_cp_128x256b(sfb_t + ch * 8, ptx::sdesc(sSFB0 + st * sfb_stage + ch * 2048, 8192, 128,
                                                                ptx::kSwizzleNone));
            } else {
              ptx::tmem_cp_32x128b_x4(sfb_t + ch * 8, ptx::sdesc_sf(sSFB0 + st * sfb_stage + ch * 512));
              ptx::tmem_cp_32x128b_x4(sfb_t + ch * 8 + 4,
                                      ptx::sdesc_sf(sSFB0 + st * sfb_stage + kSfaBytes + ch * 512));
            }
          }
        }
        const uint64_t ad = ptx::sdesc_kmajor_sw128(sA0 + st * kABytes);
        const uint64_t bd = ptx::sdesc_kmajor_sw128(sB0 + st * kBBytes);
#pragma unroll
        for (int kk = 0; kk < BK / 32; ++kk) {
          // advance 32 bytes (one K=32 step) inside the 128-byte swizzle atom
          const uint64_t adk = ad + (uint64_t)(kk * 2), bdk = bd + (uint64_t)(kk * 2);
          const uint32_t acc = ((BLOCK ? 0 : s) > 0 || kk > 0) ? 1u : 0u;
          if (NV)
            ptx::mma_mxf4nvf4(d_tmem, adk, bdk, p.idesc, sfa_t + kk * 4, sfb_t + kk * 8, acc);
          else if (MX)
            ptx::mma_mxf8f6f4(d_tmem, adk, bdk, p.idesc | ptx::idesc_sf_ids(kk, kk), sfa_t, sfb_t, acc);
          else
            ptx::mma_f8f6f4(d_tmem, adk, bdk, p.idesc, acc);
        }
        ptx::mma_commit(&empty[st]);   // frees the smem stage once these MMAs finish
        if (BLOCK) {
          ptx::mma_commit(&tmem_full[a]);  // partial product of this stage complete
          ++tc;
        }
      }
      if (!ok) break;
      if (!BLOCK) {
        ptx::mma_commit(&tmem_full[a]);  // accumulator complete
        ++tc;
      }
    }
  }
  } else {
    if (KIND == kKindBlock) ptx::setmaxnreg_inc<kBlkRegHigh>();
    // ------------------------------------------------------------ epilogue
    // 8 warps: warp w reads tensor-memory lane quadrant w % 4 (the hardware
    // rule) and the column half (w - EW0) / 4 of the 256-column accumulator. The
    // whole accumulator is moved to registers first and released to the MMA
    // issuer; the scaling, conversion and stores overlap the next tile.
    const uint32_t q = warp & 3;
    const uint32_t half = (uint32_t)(warp - EW0) >> 2;
    const int64_t row_in_tile = q * 32 + lane;
    Stager sg{sOut + (warp - EW0) * kStageOut * nslots, nslots, 0u};
    uint32_t h_tam = 0;    // per-tensor SwiGLU: this thread's max |h| (float bits)
    int ecur = 0;
    uint32_t tc = 0;
    uint32_t it_e = 0;     // block scales: stage count, as the producer's `it`
    Tile tl;
    for (int64_t t = blockIdx.x; run && get_tile<MODE>(s_off, E, p, t, ecur, tl); t += gridDim.x) {
      const int64_t orow = tl.out_row + row_in_tile;
      const int64_t col0 = tl.out_col + half * (BN / 2);
      if (tl.nst == 0) {
        // empty group (wgrad): dW_e = 0, or unchanged when accumulating
        if (p.beta == 0.0f) {
          if (p.out_f32) {
            float* o = static_cast<float*>(p.out) + orow * p.ldo + col0;
            for (int c = 0; c < BN / 2; c += 4) *reinterpret_cast<float4*>(o + c) = make_float4(0, 0, 0, 0);
          } else {
            uint16_t* o = static_cast<uint16_t*>(p.out) + orow * p.ldo + col0;
            for (int c = 0; c < BN / 2; c += 8) *reinterpret_cast<uint4*>(o + c) = make_uint4(0, 0, 0, 0);
          }
        }
        continue;
      }
      uint32_t r[4][32];
      if (BLOCK) {
        // promotion: acc += partial(stage) * s_a[row, kb] * s_b[n block, kb];
        // contract mode (wgrad, 128x1 blocks of both operands along the
        // group's rows): acc += partial(stage) * s_a[row, kb] * s_b[column, kb].
        // The stage's row (and column) scales come from the shared ring slot
        // the producer filled; rows mode's B tile scale is one float per
        // stage and 128-column half, loaded one stage ahead.
        const float* sb_blk = MODE == kModeRows
                                  ? p.sb + ((int64_t)tl.e * (p.N / 128) + (col0 / 128)) * (p.K / 128)
                                  : nullptr;
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int i = 0; i < 32; ++i) r[c][i] = 0u;   // +0.0f
        float sb_next = MODE == kModeRows ? __ldg(sb_blk + tl.kx0 / 128) : 1.0f;
        bool alive = true;
        for (int s = 0; s < tl.nst; ++s, ++it_e) {
          const uint32_t a = tc % kAcc, aph = (tc / kAcc) & 1;
          const uint32_t sl = it_e % kBlkSlots;
          const float sb_cur = sb_next;
          if (MODE == kModeRows && s + 1 < tl.nst) sb_next = __ldg(sb_blk + tl.kx0 / 128 + s + 1);
          if (__any_sync(0xFFFFFFFFu, *s_abort != 0)) { alive = false; break; }
          const bool got = __all_sync(0xFFFFFFFFu, ptx::mbar_wait(&s_full[sl], (it_e / kBlkSlots) & 1, p.wait_ns) &&
                                                       ptx::mbar_wait(&tmem_full[a], aph, p.wait_ns));
          if (!got) {
            report(p.err, MGQ_ERR_TIMEOUT);
            *s_abort = 1;
            alive = false;
            break;
          }
          ptx::tc_fence_after();
          const float* slot = sRing + sl * kBlkSlotFloats;
          const float f = slot[row_in_tile] * sb_cur;     // rows: s_a * s_b; contract: s_a
          const float4* sbc = reinterpret_cast<const float4*>(slot + 128 + half * (BN / 2));
          const uint32_t taddr = tmem + a * BN + ((q * 32) << 16) + half * (BN / 2);
          // 16 columns per load, two loads in flight: chunk c + 1 is read
          // while chunk c is scaled and added
          uint32_t vb[2][16];
          ptx::tmem_ld_32x32b_x16(taddr, vb[0]);
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            uint32_t (&v)[16] = vb[c & 1];
            ptx::tmem_ld_wait_regs(v);
            if (c + 1 < 8) ptx::tmem_ld_32x32b_x16(taddr + (c + 1) * 16, vb[(c + 1) & 1]);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              uint32_t* acc = &r[c / 2][(c & 1) * 16 + 4 * j];
              if (MODE == kModeContract) {
                // columns 16 c + 4 j .. + 3: their scales (the same for every
                // lane: one broadcast read) times this row's s_a
                const float4 cs = sbc[4 * c + j];
                uint32_t f0, f1, f2, f3;
                ptx::fmul2(f0, f1, __float_as_uint(cs.x), __float_as_uint(cs.y), __float_as_uint(f), __float_as_uint(f));
                ptx::fmul2(f2, f3, __float_as_uint(cs.z), __float_as_uint(cs.w), __float_as_uint(f), __float_as_uint(f));
                ptx::ffma2(acc[0], acc[1], v[4 * j], v[4 * j + 1], f0, f1);
                ptx::ffma2(acc[2], acc[3], v[4 * j + 2], v[4 * j + 3], f2, f3);
              } else {
                ptx::ffma2(acc[0], acc[1], v[4 * j], v[4 * j + 1], __float_as_uint(f), __float_as_uint(f));
                ptx::ffma2(acc[2], acc[3], v[4 * j + 2], v[4 * j + 3], __float_as_uint(f), __float_as_uint(f));
              }
            }
          }
          ptx::tc_fence_before();
          ptx::mbar_arrive(&tmem_empty[a]);
          ptx::mbar_arrive(&s_empty[sl]);     // this thread's reads of the slot are done
          ++tc;
        }
        if (!alive) break;
      } else {
        const uint32_t a = tc % kAcc, aph = (tc / kAcc) & 1;
        uint4 gq[2], uq[2];    // dSwiGLU: the first g / u chunk, requested before the accumulator is ready
        if (DSW && KIND == kKindTensor) dswiglu_load_gu(p, orow, col0, 0, gq, uq);
        // the whole warp agrees before the .sync.aligned tensor-memory loads
        if (__any_sync(0xFFFFFFFFu, *s_abort != 0)) break;
        const bool got = __all_sync(0xFFFFFFFFu, ptx::mbar_wait(&tmem_full[a], aph, p.wait_ns));
        if (!got) {
          report(p.err, MGQ_ERR_TIMEOUT);
          *s_abort = 1;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t tbase = tmem + a * BN + ((q * 32) << 16);
        if (DSW && KIND == kKindTensor) {
          epilogue_dswiglu(p, tbase + half * (BN / 2), 1.0f / (p.sa[0] * p.sb[tl.e]), orow, col0,
                           sg, &tmO, &tmH, (int32_t)(tl.out_row + q * 32), lane, h_tam,
                           gq, uq);
          ptx::tc_fence_before();
          ptx::mbar_arrive(&tmem_empty[a]);
          ++tc;
          continue;
        }
#pragma unroll
        for (int c = 0; c < 4; ++c) ptx::tmem_ld_32x32b_x32(tbase + acc_col(MODE == kModeRows && p.swiglu, half, c), r[c]);
        ptx::tmem_ld_wait();
        ptx::tc_fence_before();
        ptx::mbar_arrive(&tmem_empty[a]);       // accumulator free for the next tile
        ++tc;
        if (DSW && KIND == kKindMX) {
          // MX dSwiGLU: dh = bf16(acc) packed, then the epilogue from registers
          uint32_t dhp[64];
#pragma unroll
          for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int i = 0; i < 16; ++i)
              dhp[16 * c + i] = pack_bf16x2(__uint_as_float(r[c][2 * i]), __uint_as_float(r[c][2 * i + 1]));
          epilogue_dswiglu_mx(p, dhp, orow, col0, tl.out_row + q * 32, lane);
          continue;
        }
      }
      float alpha = 1.0f;
      if (KIND == kKindTensor || NV) alpha = 1.0f / (p.sa[0] * p.sb[MODE == kModeRows ? tl.e : 0]);
      if (wide_staging(KIND, MODE) && p.tma_store)
        epilogue_store_wide(p, r, sOut + (warp - EW0) * kStageWide, &tmO, col0, (int32_t)(tl.out_row + q * 32),
                            lane);
      else if (MODE == kModeRows && KIND != kKindBlock && p.swiglu)
        epilogue_swiglu<KIND == kKindBlock ? kKindTensor : KIND>(p, r, alpha, orow, tl.out_col + half * 64,
                                                                 sg, &tmO, &tmH,
                                                                 (int32_t)(tl.out_row + q * 32), lane, h_tam);
      else
        epilogue_store(p, r, alpha, orow, col0, p.tma_store != 0, sg, &tmO,
                       (int32_t)(tl.out_row + q * 32), lane);
    }
    if (MODE == kModeRows && (KIND == kKindTensor || KIND == kKindNV) && (p.swiglu || DSW) && p.h_amax) {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) h_tam = max(h_tam, __shfl_xor_sync(0xFFFFFFFFu, h_tam, o));
      if (lane == 0) atomic_max_nonneg(p.h_amax, __uint_as_float(h_tam));
    }
  }
  if (warp >= EW0 && lane == 0) ptx::bulk_wait0();   // this warp's TMA stores are complete
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kTmemCols);
  }
}

template <int MODE, int KIND, bool DSW = false, bool IMG = false>
int launch_gemm_t(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& to, const CUtensorMap& th,
                const GemmParams& p, cudaStream_t s) {
  auto kern = grouped_gemm_kernel<MODE, KIND, DSW, IMG>;
  // (NVFP4 with compact B scales: the smaller layout)
  constexpr size_t kSmemBytes = KIND == kKindNV && !IMG ? smem_bytes_nv_compact(MODE) : smem_bytes(KIND, MODE);
  static bool attr_set[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_set[dev]) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes) != cudaSuccess)
      return MGQ_ERR_CUDA;
    if (KIND == kKindBlock) {
      // the register split must fit in what the block is launched with, or
      // setmaxnreg.inc would never return: never launch such a build
      cudaFuncAttributes fa;
      if (cudaFuncGetAttributes(&fa, kern) != cudaSuccess || fa.numRegs < kBlkRegLaunch) return MGQ_ERR_CUDA;
    }
    attr_set[dev] = true;
  }
  kern<<<num_sms(), threads_of(KIND), kSmemBytes, s>>>(ta, tb, to, th, p);
  MGQ_LAUNCH_CHECK();
  return MGQ_OK;
}

// NVFP4 calls with a B scale image run the IMG instantiation
template <int MODE, int KIND, bool DSW = false>
int launch_gemm(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& to, const CUtensorMap& th,
                const GemmParams& p, cudaStream_t s) {
  if constexpr (KIND == kKindNV && !DSW) {
    if (p.sfb_img) return launch_gemm_t<MODE, KIND, DSW, true>(ta, tb, to, th, p, s);
  }
  return launch_gemm_t<MODE, KIND, DSW, false>(ta, tb, to, th, p, s);
}


// ============================================================================
// 2-CTA variant (cta_group::2) for per-tensor FP8: a cluster of two CTAs on two
// SMs computes 256 x 256 tiles. Each CTA loads its 128 rows of A and its 128
// rows (N half) of B; one thread of CTA 0 issues M=256 MMAs that read both
// CTAs' shared memory, and each CTA's tensor memory receives its 128 rows of
// the accumulator. Half of the B tile per SM means 32 KB per stage, so the
// pipeline is 6 stages deep in the same shared memory.
//   - TMA loads of both CTAs complete on CTA 0's `full` barrier (which CTA 0
//     arms with the pair's byte count); the MMA commit is multicast to both
//     CTAs' `empty` and `tmem_full` barriers; both CTAs' epilogue warps arrive
//     on CTA 0's `tmem_empty`.
//   - MX (E8M0 block scales): each CTA also loads, per stage, the 512-byte
//     scale chunk of its own 128 rows of A and the two chunks of all 256 rows
//     of B (the scales of B are needed whole in both CTAs); CTA 0 copies them
//     into both CTAs' tensor memory with pair scale copies. Tensor memory then
//     has no room for a second accumulator: the epilogue moves it to registers
//     and releases it before storing.
constexpr int PSTAGES = 6;                                     // per-tensor and MX; NVFP4 5
// (the per-tensor dSwiGLU instantiation gives one stage to its g / u staging slots)
__host__ __device__ constexpr int pstages_of(int kind, bool dsw = false) {
  return (kind == kKindNV || dsw) ? 5 : PSTAGES;
}
constexpr uint32_t kPairTile = 128 * 128;                      // bytes of one A or B half tile
// block-scale bytes per stage for this CTA's A rows (B: twice, both halves):
// MX one 512-byte chunk per 128 rows, NVFP4 four (the 4 MMAs of a 256-element stage)
__host__ __device__ constexpr uint32_t pair_sfa_bytes(int kind) {
  return kind == kKindMX ? 512u : (kind == kKindNV ? 2048u : 0u);
}
__host__ __device__ constexpr uint32_t pair_sf_bytes(int kind) { return 3 * pair_sfa_bytes(kind); }
__host__ __device__ constexpr size_t pair_smem(int kind, bool dsw = false) {
  return 1024 + pstages_of(kind, dsw) * (2 * kPairTile + pair_sf_bytes(kind)) + 8 * kStageOut +
         (dsw ? 8 * kGuSlot : 0) + 256 + (2 * kMaxE + 16) * 4;
}
// tensor-memory columns: accumulator(s), then the scale slots of every stage
// (4 columns per chunk of A, 8 per chunk pair of B; NVFP4: 496 columns in all)
constexpr uint32_t kPairSfaCol = 256;
__host__ __device__ constexpr uint32_t pair_sfb_col(int kind) {
  return kPairSfaCol + pstages_of(kind) * 4 * (pair_sfa_bytes(kind) / 512);
}

template <int MODE>
__device__ __forceinline__ bool get_pair_tile(const int32_t* s_off, const int32_t* s_cum, int E, const GemmParams& p,
                                              int64_t t, int& ecur, Tile& tl) {
  if (MODE == kModeRows) {
    // pair tiles of 256 rows per expert (the last may reach past the group;
    // those rows are computed on whatever follows and never stored)
    const int64_t nN = p.N / BN;
    const int64_t total = (int64_t)s_cum[E] * nN;
    if (t >= total) return false;
    while (ecur < E - 1 && (int64_t)s_cum[ecur + 1] * nN <= t) ++ecur;
    const int e = ecur;
    const int64_t mt = s_cum[e + 1] - s_cum[e];
    const int64_t local = t - (int64_t)s_cum[e] * nN;
    int64_t n, m;
    band_order(local, mt, nN, n, m);
    tl.e = e;
    tl.nst = (int)(p.K / BK);
    tl.row_a = s_off[e] + 256 * m;
    tl.row_b = (int64_t)e * p.N + (p.swiglu ? 128 : BN) * n;
    tl.kx0 = 0;
    tl.out_row = tl.row_a;
    tl.out_col = (p.swiglu ? 128 : BN) * n;
  } else {
    const int64_t mN = p.N / 256, nK = p.K / BN;
    const int64_t tpe = mN * nK;
    if (t >= tpe * E) return false;
    const int e = (int)(t / tpe);
    const int64_t local = t % tpe;
    const int64_t m = local / nK, n = local % nK;
    tl.e = e;
    tl.nst = (s_off[e + 1] - s_off[e]) / (BK * p.kdiv);     // (e2m1: 2 BK rows a stage)
    tl.row_a = 256 * m;
    tl.row_b = BN * n;
    tl.kx0 = s_off[e] / p.kdiv;
    tl.out_row = (int64_t)e * p.N + 256 * m;
    tl.out_col = BN * n;
  }
  return true;
}

template <int MODE, int KIND, bool DSW = false>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    grouped_gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                             const __grid_constant__ CUtensorMap tmO, const __grid_constant__ CUtensorMap tmSFA,
                             const __grid_constant__ CUtensorMap tmSFB, const __grid_constant__ CUtensorMap tmH,
                             const GemmParams p) {
  constexpr bool MX = KIND == kKindMX;
  constexpr bool NV = KIND == kKindNV;
  constexpr bool BS = MX || NV;                    // block scales through tensor memory
  constexpr int PST = pstages_of(KIND, DSW);
  constexpr uint32_t kSfa = pair_sfa_bytes(KIND), kSfb = 2 * kSfa, kCh = kSfa / 512;   // chunks per 128 rows
  constexpr uint32_t kSfbCol = pair_sfb_col(KIND);
  constexpr int kAccBufs = BS ? 1 : 2;             // block scales: their slots leave room for one accumulator
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = ptx::smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  uint8_t* sA = smem;
  uint8_t* sB = sA + PST * kPairTile;
  uint8_t* sOut = sB + PST * kPairTile;            // [8 warps][32 rows][64 bytes] epilogue staging
  uint8_t* sSFA = sOut + 8 * kStageOut;            // block scales: [stage] chunks of this CTA's A rows
  uint8_t* sSFB = sSFA + PST * kSfa;               // block scales: [stage] chunks of both B halves
  uint8_t* sGU = sOut + 8 * kStageOut + PST * pair_sf_bytes(KIND);   // dSwiGLU: [8 warps] g / u slots
  uint64_t* bars = reinterpret_cast<uint64_t*>(sGU + (DSW ? 8 * kGuSlot : 0));
  uint64_t* full = bars;
  uint64_t* empty = bars + PST;
  uint64_t* tmem_full = bars + 2 * PST;            // [2]
  uint64_t* tmem_empty = bars + 2 * PST + 2;       // [2]
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(bars + 2 * PST + 4);
  volatile int* s_abort = reinterpret_cast<volatile int*>(s_tmem + 1);
  int* s_bad = reinterpret_cast<int*>(s_tmem + 2);
  int32_t* s_off = reinterpret_cast<int32_t*>(bars + 32);
  int32_t* s_cum = s_off + (kMaxE + 8);

  const int warp = threadIdx.x >> 5;
  const uint32_t lane = threadIdx.x & 31;
  const int E = p.E;
  const uint32_t rank = ptx::cluster_ctarank();
  const bool leader = rank == 0;
  const int64_t pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;

  for (int i = threadIdx.x; i <= E; i += kThreads) s_off[i] = p.offsets[i];
  if (threadIdx.x == 0) {
    for (int s = 0; s < PST; ++s) {
      ptx::mbar_init(&full[s], 1);
      ptx::mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      ptx::mbar_init(&tmem_full[a], 1);
      ptx::mbar_init(&tmem_empty[a], 2 * 8);      // one arrival per epilogue warp of each CTA
    }
    *s_abort = 0;
    *s_bad = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    ptx::prefetch_tmap(&tmA);
    ptx::prefetch_tmap(&tmB);
    if (BS) {
      ptx::prefetch_tmap(&tmSFA);
      ptx::prefetch_tmap(&tmSFB);
    }
  }
  if (warp == 1) {
    ptx::tmem_alloc_pair(s_tmem, kTmemCols);
    ptx::tmem_relinquish_pair();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    bool bad = s_off[0] != 0;
    int cum = 0;
    for (int e = 0; e < E; ++e) {
      // (contract mode over e2m1: whole 256-row stages)
      bad |= (s_off[e + 1] < s_off[e]) || (s_off[e + 1] % (MODE == kModeContract ? BM * p.kdiv : BM)) != 0;
      s_cum[e] = cum;
      cum += (s_off[e + 1] - s_off[e] + 255) / 256;
    }
    s_cum[E] = cum;
    bad |= (int64_t)s_off[E] > p.R_cap;
    if (bad) {
      *s_bad = 1;
      report(p.err, MGQ_ERR_INVALID_ARG);
    }
  }
  ptx::tc_fence_before();
  ptx::cluster_sync();                 // both CTAs' barriers initialised, tensor memory allocated
  ptx::tc_fence_after();
  const uint32_t tmem = *s_tmem;
  const bool run = (*s_bad == 0);

  if (run && warp == 0 && lane == 0 && !p.debug_stall) {
    // ------------------------------------------------------------ producer (both CTAs)
    int ecur = 0;
    uint32_t it = 0;
    Tile tl;
    for (int64_t t = pair; get_pair_tile<MODE>(s_off, s_cum, E, p, t, ecur, tl); t += npairs) {
      for (int s = 0; s < tl.nst; ++s, ++it) {
        const uint32_t st = it % PST, ph = (it / PST) & 1;
        if (*s_abort) break;
        if (!ptx::mbar_wait(&empty[st], ph ^ 1, p.wait_ns)) {
          report(p.err, MGQ_ERR_TIMEOUT);
          *s_abort = 1;
          break;
        }
        // both CTAs' A and B halves (and the scale chunks)
        if (leader) ptx::mbar_arrive_expect_tx(&full[st], 4 * kPairTile + 2 * pair_sf_bytes(KIND));
        const uint32_t bar0 = ptx::mapa_shared(ptx::smem_u32(&full[st]), 0);
        const int32_t kx = (int32_t)(tl.kx0 + (int64_t)s * BK);
        // K-major: box (128 contraction bytes, 128 rows); MN-major: box (128
        // columns of M/N, 128 contraction rows)
        const int32_t am = (int32_t)(tl.row_a + 128 * rank);
        if (p.a_mn) ptx::tma_load_2d_pair(sA + st * kPairTile, &tmA, bar0, am, kx);
        else ptx::tma_load_2d_pair(sA + st * kPairTile, &tmA, bar0, kx, am);
        if (p.b_mn)
          ptx::tma_load_2d_pair(sB + st * kPairTile, &tmB, bar0, (int32_t)(tl.out_col + 128 * rank),
                                (int32_t)((MODE == kModeRows ? (int64_t)tl.e * p.K : 0) + kx));
        else
          ptx::tma_load_2d_pair(sB + st * kPairTile, &tmB, bar0, kx, (int32_t)(tl.row_b + p.b_half2 * rank));
        if (BS) {
          // the stage's chunks (row tile, chunk) start at row tile * kb4 + kt in
          // the [chunks][128 words] view of the scales (boxes of kCh chunks):
          // MX one chunk per 128-element k tile, NVFP4 four per 256-element stage
          const int32_t kt = (kx / BK) * (int32_t)kCh;
          ptx::tma_load_2d_pair(sSFA + st * kSfa, &tmSFA, bar0, 0,
                                (int32_t)(((tl.row_a + 128 * rank) / 128) * p.sfa_kb4 + kt));
          ptx::tma_load_2d_pair(sSFB + st * kSfb, &tmSFB, bar0, 0, (int32_t)((tl.row_b / 128) * p.sfb_kb4 + kt));
          ptx::tma_load_2d_pair(sSFB + st * kSfb + kSfa, &tmSFB, bar0, 0,
                                (int32_t)(((tl.row_b + p.b_half2) / 128) * p.sfb_kb4 + kt));
        }
      }
      if (*s_abort) break;
    }
  } else if (run && leader && warp == 1 && lane == 0) {
    // ------------------------------------------------------------ MMA issuer (CTA 0)
    int ecur = 0;
    uint32_t it = 0, tc = 0;
    Tile tl;
    const uint32_t sA0 = ptx::smem_u32(sA), sB0 = ptx::smem_u32(sB);
    const uint32_t sSFA0 = ptx::smem_u32(sSFA), sSFB0 = ptx::smem_u32(sSFB);
    for (int64_t t = pair; get_pair_tile<MODE>(s_off, s_cum, E, p, t, ecur, tl); t += npairs) {
      if (tl.nst == 0) continue;
      if (*s_abort) break;
      const uint32_t a = tc % kAccBufs, aph = (tc / kAccBufs) & 1;
      if (!ptx::mbar_wait(&tmem_empty[a], aph ^ 1, p.wait_ns)) {
        report(p.err, MGQ_ERR_TIMEOUT);
        *s_abort = 1;
        break;
      }
      ptx::tc_fence_after();
      bool ok = true;
      for (int s = 0; s < tl.nst; ++s, ++it) {
        const uint32_t st = it % PST, ph = (it / PST) & 1;
        if (*s_abort || !ptx::mbar_wait(&full[st], ph, p.wait_ns)) {
          report(p.err, MGQ_ERR_TIMEOUT);
          *s_abort = 1;
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        // a K=32 step: 32 bytes along a K-major row, 32 rows (4096 bytes) of
        // an MN-major tile; descriptor addresses count 16-byte units
        const uint64_t ad = p.a_mn ? ptx::sdesc_mnmajor_sw128(sA0 + st * kPairTile)
                                   : ptx::sdesc_kmajor_sw128(sA0 + st * kPairTile);
        const uint64_t bd = p.b_mn ? ptx::sdesc_mnmajor_sw128(sB0 + st * kPairTile)
                                   : ptx::sdesc_kmajor_sw128(sB0 + st * kPairTile);
        const uint64_t astep = p.a_mn ? 256 : 2, bstep = p.b_mn ? 256 : 2;
        if constexpr (BS) {
          // this stage's scales into both CTAs' tensor memory (ordered before
          // the MMAs below, which read them): chunk ch of A at 4 ch columns,
          // of the two B halves at 8 ch and 8 ch + 4
          const uint32_t sfa_t = tmem + kPairSfaCol + st * 4 * kCh, sfb_t = tmem + kSfbCol + st * 8 * kCh;
#pragma unroll
          for (uint32_t ch = 0; ch < kCh; ++ch) {
            ptx::tmem_cp_32x128b_x4_pair(sfa_t + ch * 4, ptx::sdesc_sf(sSFA0 + st * kSfa + ch * 512));
            ptx::tmem_cp_32x128b_x4_pair(sfb_t + ch * 8, ptx::sdesc_sf(sSFB0 + st * kSfb + ch * 512));
            ptx::tmem_cp_32x128b_x4_pair(sfb_t + ch * 8 + 4, ptx::sdesc_sf(sSFB0 + st * kSfb + kSfa + ch * 512));
          }
#pragma unroll
          for (int kk = 0; kk < BK / 32; ++kk) {
            // a 32-byte step: K=32 of e4m3/e5m2 or K=64 of e2m1 (one chunk each)
            if constexpr (NV)
              ptx::mma_mxf4nvf4_pair(tmem + a * BN, ad + kk * astep, bd + kk * bstep, p.idesc, sfa_t + kk * 4,
                                     sfb_t + kk * 8, (s > 0 || kk > 0) ? 1u : 0u);
            else
              ptx::mma_mxf8f6f4_pair(tmem + a * BN, ad + kk * astep, bd + kk * bstep,
                                     p.idesc | ptx::idesc_sf_ids(kk, kk), sfa_t, sfb_t, (s > 0 || kk > 0) ? 1u : 0u);
          }
        } else {
#pragma unroll
          for (int kk = 0; kk < BK / 32; ++kk)
            ptx::mma_f8f6f4_pair(tmem + a * BN, ad + kk * astep, bd + kk * bstep, p.idesc,
                                 (s > 0 || kk > 0) ? 1u : 0u);
        }
        ptx::mma_commit_pair(&empty[st], 0x3);        // frees the stage in both CTAs
      }
      if (!ok) break;
      ptx::mma_commit_pair(&tmem_full[a], 0x3);       // both halves of the accumulator complete
      ++tc;
    }
  } else if (warp >= 2) {
    // ------------------------------------------------------------ epilogue (both CTAs)
    const uint32_t q = warp & 3;
    const uint32_t half = (uint32_t)(warp - 2) >> 2;
    const int64_t row_in_tile = 128 * rank + q * 32 + lane;
    Stager sg{sOut + (warp - 2) * kStageOut, 1u, 0u};
    uint32_t h_tam = 0;    // per-tensor SwiGLU: this thread's max |h| (float bits)
    const uint32_t empty_remote0 = ptx::mapa_shared(ptx::smem_u32(&tmem_empty[0]), 0);
    const uint32_t empty_remote1 = ptx::mapa_shared(ptx::smem_u32(&tmem_empty[1]), 0);
    int ecur = 0;
    uint32_t tc = 0;
    Tile tl;
    for (int64_t t = pair; run && get_pair_tile<MODE>(s_off, s_cum, E, p, t, ecur, tl); t += npairs) {
      const int64_t orow = tl.out_row + row_in_tile;
      const int64_t col0 = tl.out_col + half * (BN / 2);
      // rows of the last pair tile past the expert's group are not stored
      const bool store = MODE == kModeContract || orow < s_off[tl.e + 1];
      if (tl.nst == 0) {
        if (p.beta == 0.0f && store) {
          if (p.out_f32) {
            float* o = static_cast<float*>(p.out) + orow * p.ldo + col0;
            for (int c = 0; c < BN / 2; c += 4) *reinterpret_cast<float4*>(o + c) = make_float4(0, 0, 0, 0);
          } else {
            uint16_t* o = static_cast<uint16_t*>(p.out) + orow * p.ldo + col0;
            for (int c = 0; c < BN / 2; c += 8) *reinterpret_cast<uint4*>(o + c) = make_uint4(0, 0, 0, 0);
          }
        }
        continue;
      }
      const uint32_t a = tc % kAccBufs, aph = (tc / kAccBufs) & 1;
      uint4 gq[2], uq[2];    // dSwiGLU: the first g / u chunk, requested before the accumulator is ready
      uint8_t* gslot = sGU + (warp - 2) * kGuSlot;
      if (DSW && store) gu_stage_issue(p, ptx::smem_u32(gslot), orow - lane, col0, lane);
      if (__any_sync(0xFFFFFFFFu, *s_abort != 0)) break;
      const bool got = __all_sync(0xFFFFFFFFu, ptx::mbar_wait(&tmem_full[a], aph, p.wait_ns));
      if (!got) {
        report(p.err, MGQ_ERR_TIMEOUT);
        *s_abort = 1;
        break;
      }
      ptx::tc_fence_after();
      const uint32_t tbase = tmem + a * BN + ((q * 32) << 16);
      if (DSW) {
        // tensor memory read chunk by chunk beside the gu loads, released after
        // (the other accumulator buffer keeps the MMAs going meanwhile)
        if (store)
          epilogue_dswiglu(p, tbase + half * (BN / 2), 1.0f / (p.sa[0] * p.sb[tl.e]), orow, col0,
                           sg, &tmO, &tmH, (int32_t)(tl.out_row + 128 * rank + q * 32),
                           lane, h_tam, gq, uq, gslot);
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive_cluster(a ? empty_remote1 : empty_remote0);
        ++tc;
        continue;
      }
      uint32_t r[4][32];
#pragma unroll
      for (int c = 0; c < 4; ++c) ptx::tmem_ld_32x32b_x32(tbase + acc_col(MODE == kModeRows && p.swiglu, half, c), r[c]);
      ptx::tmem_ld_wait();
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive_cluster(a ? empty_remote1 : empty_remote0);
      ++tc;
      if (!store) continue;    // the warp's 32 rows lie wholly inside or past the group
      const float alpha = MX ? 1.0f : 1.0f / (p.sa[0] * p.sb[MODE == kModeRows ? tl.e : 0]);
      if (MODE == kModeRows && p.swiglu)
        epilogue_swiglu<KIND, false>(p, r, alpha, orow, tl.out_col + half * 64, sg, &tmO, &tmH,
                              (int32_t)(tl.out_row + 128 * rank + q * 32), lane, h_tam);
      else
        epilogue_store(p, r, alpha, orow, col0, p.tma_store != 0, sg, &tmO,
                       (int32_t)(tl.out_row + 128 * rank + q * 32), lane);
    }
    if (MODE == kModeRows && (KIND == kKindTensor || KIND == kKindNV) && (p.swiglu || DSW) && p.h_amax) {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) h_tam = max(h_tam, __shfl_xor_sync(0xFFFFFFFFu, h_tam, o));
      if (lane == 0) atomic_max_nonneg(p.h_amax, __uint_as_float(h_tam));
    }
    if (DSW) ptx::cp_async_wait_all();   // (a timeout can leave a g / u copy in flight)
  }
  if (warp >= 2 && lane == 0) ptx::bulk_wait0();   // this warp's TMA stores are complete
  __syncthreads();
  ptx::tc_fence_before();
  ptx::cluster_sync();                 // the peer's MMAs and reads are finished before freeing
  ptx::tc_fence_after();
  if (warp == 1) {
    __syncwarp();
    ptx::tmem_dealloc_pair(tmem, kTmemCols);
  }
}

template <int MODE, int KIND, bool DSW = false>
int launch_gemm_pair(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& to, const CUtensorMap& tsfa,
                     const CUtensorMap& tsfb, const CUtensorMap& th, const GemmParams& p, cudaStream_t s) {
  auto kern = grouped_gemm_pair_kernel<MODE, KIND, DSW>;
  constexpr size_t kSmem = pair_smem(KIND, DSW);
  static bool attr_set[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_set[dev]) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmem) != cudaSuccess)
      return MGQ_ERR_CUDA;
    attr_set[dev] = true;
  }
  kern<<<num_sms() / 2 * 2, kThreads, kSmem, s>>>(ta, tb, to, tsfa, tsfb, th, p);
  MGQ_LAUNCH_CHECK();
  return MGQ_OK;
}

// Process-wide GEMM options (mgq_set_gemm_option): which kernel serves a call,
// how the pair kernel stores, and the failure-detection test hooks. Each launch
// reads them with relaxed atomic loads; nothing is taken from the environment.
//  - The 2-CTA kernel serves per-tensor FP8 (wgrad needs output rows in
//    multiples of 256); MGQ_GEMM_OPT_FORCE_1CTA puts every call on the 1-CTA
//    kernel (both compute the same values).
//  - MX goes to the 1-CTA kernel unless MGQ_GEMM_OPT_MX_PAIR is set: measured
//    on the Mixtral gate/up and down shapes, the pair scale copies (three
//    32x128b.warpx4 copies per 128-deep stage, executed in order with the
//    MMAs) cost the pair kernel about a fifth of its MMA rate, which leaves it
//    behind the 1-CTA kernel.
//  - NVFP4 on the 2-CTA kernel with MGQ_GEMM_OPT_NV_PAIR: correct, but
//    measured slower than the 1-CTA kernel (the pair form of the four scale
//    copies a stage costs more than the copies it saves), so not the default.
//  - MGQ_GEMM_OPT_DEBUG_STALL makes the producer issue no loads, so the
//    pipeline waits run out and the kernel reports MGQ_ERR_TIMEOUT and exits
//    cleanly; MGQ_GEMM_OPT_WAIT_MS sets the wait limit (0: 2000 ms).
std::atomic<int64_t> g_gemm_opt[MGQ_GEMM_OPT_COUNT];

int64_t gemm_opt(int o) { return g_gemm_opt[o].load(std::memory_order_relaxed); }

void debug_knobs(int* stall, uint64_t* wait_ns) {
  *stall = gemm_opt(MGQ_GEMM_OPT_DEBUG_STALL) ? 1 : 0;
  const int64_t ms = gemm_opt(MGQ_GEMM_OPT_WAIT_MS);
  *wait_ns = ms > 0 ? (uint64_t)ms * 1000000ull : kWaitNs;
}

bool direct_store_forced() { return gemm_opt(MGQ_GEMM_OPT_DIRECT_STORE) != 0; }

bool use_pair_kernel(int mode, int64_t N) {
  if (gemm_opt(MGQ_GEMM_OPT_FORCE_1CTA)) return false;
  return mode == kModeRows || N % 256 == 0;
}

bool mx_pair_selected() { return gemm_opt(MGQ_GEMM_OPT_MX_PAIR) != 0; }
bool nv_pair_selected() { return gemm_opt(MGQ_GEMM_OPT_NV_PAIR) != 0; }

int check_operand(const mgq_operand* o) {
  if (!o || !o->data || !aligned16(o->data)) return MGQ_ERR_INVALID_ARG;
  if (o->dtype != MGQ_E4M3 && o->dtype != MGQ_E5M2 && o->dtype != MGQ_E2M1) return MGQ_ERR_UNSUPPORTED;
  return MGQ_OK;
}

// Shared driver of the three entry points.
//  mode rows:     A [rowsA, Kc] (ld), B [E*Nout, Kc] (ld); out [rowsA, Nout]
//  mode contract: A [Nout_rows, R_cap], B [Kout, R_cap]; out [E*Nout_rows, Kout]
// SwiGLU epilogue request of the gate/up GEMM (N = 2F)
struct SwigluOut {
  const mgq_qdesc* qh;
  void* h_bf16;
};
// dSwiGLU epilogue request of the down-projection dgrad (N = F)
struct DswigluOut {
  const void* gu;
  const mgq_qdesc* q;
  void* dgu_bf16;
};

// NVFP4 SwiGLU: the epilogue wrote h (bf16) and its amax; cast h with s_g,
// row-wise (and column-wise when qh->col is set) (N = 2F)
int nv_swiglu_second_pass(const SwigluOut* sw, int64_t R_cap, const int32_t* offsets, int E, int64_t N,
                          cudaStream_t s) {
  if (sw->qh->col.data)   // row-wise and column-wise copies in one tile pass
    return rowcol_rows(static_cast<const uint16_t*>(sw->h_bf16), R_cap, offsets + E, N / 2, sw->qh, s);
  return launch_quant_rows_nv(static_cast<const uint16_t*>(sw->h_bf16), R_cap, offsets + E, N / 2,
                              static_cast<uint8_t*>(sw->qh->row.data), static_cast<uint8_t*>(sw->qh->row.scale),
                              sw->qh->amax_out, sw->qh->tensor_scale, s);
}

int run_grouped(int mode, const mgq_operand* A, const mgq_operand* B, int scaling, const int32_t* offsets, int E,
                int64_t R_cap, int64_t N, int64_t K, float beta, void* out, int out_dtype, void* stream,
                const SwigluOut* sw = nullptr, const DswigluOut* dsw = nullptr) {
  int rc;
  if ((rc = check_operand(A)) != MGQ_OK) return rc;
  if ((rc = check_operand(B)) != MGQ_OK) return rc;
  MGQ_CHECK_ARG(offsets && (out || sw || dsw) && aligned16(out) && E >= 1 && E <= kMaxE && R_cap > 0 && R_cap % BM == 0);
  MGQ_CHECK_ARG(out_dtype == MGQ_OUT_BF16 || out_dtype == MGQ_OUT_F32);
  MGQ_CHECK_ARG(beta == 0.0f || (mode == kModeContract && out_dtype == MGQ_OUT_F32));
  MGQ_CHECK_ARG(R_cap < (1ll << 31));
  int kind;
  if (scaling == MGQ_MX32_E8M0) kind = kKindMX;
  else if (scaling == MGQ_TENSOR_F32) kind = kKindTensor;
  else if (scaling == MGQ_BLK_1x128_F32) kind = kKindBlock;
  else if (scaling == MGQ_NV16_UE4M3) kind = kKindNV;
  else return MGQ_ERR_UNSUPPORTED;
  const bool mx = kind == kKindMX;
  const bool nv = kind == kKindNV;
  if ((A->layout != MGQ_LAYOUT_K && A->layout != MGQ_LAYOUT_MN) ||
      (B->layout != MGQ_LAYOUT_K && B->layout != MGQ_LAYOUT_MN))
    return MGQ_ERR_INVALID_ARG;
  // MN-major operands: per-tensor FP8 on the 2-CTA kernel; A only in wgrad
  const bool a_mn = A->layout == MGQ_LAYOUT_MN, b_mn = B->layout == MGQ_LAYOUT_MN;
  if ((a_mn || b_mn) && (kind != kKindTensor || !use_pair_kernel(mode, N) || (a_mn && mode != kModeContract)))
    return MGQ_ERR_UNSUPPORTED;
  if (nv != (A->dtype == MGQ_E2M1) || nv != (B->dtype == MGQ_E2M1)) return MGQ_ERR_UNSUPPORTED;
  MGQ_CHECK_ARG(A->scale && B->scale);
  if (mx || nv || kind == kKindBlock) MGQ_CHECK_ARG(aligned16(A->scale) && aligned16(B->scale));
  if (nv) MGQ_CHECK_ARG(A->global_scale && B->global_scale && K % 256 == 0 && A->ld % 256 == 0 && B->ld % 256 == 0);
  // operand bytes per element: e2m1 codes are packed two per byte
  const int64_t ebytes_den = nv ? 2 : 1;
  GemmParams p;
  CUtensorMap ta, tb;
  // K-major operands here; MN-major ones (2-CTA kernel) get their maps below
  MGQ_CHECK_ARG(A->ld % 128 == 0 && B->ld % 128 == 0);
  if (mode == kModeRows) {
    MGQ_CHECK_ARG(N > 0 && K > 0 && N % BN == 0 && K % BK == 0);
    MGQ_CHECK_ARG(A->ld >= K && (b_mn || B->ld >= K));
    MGQ_CHECK_ARG((int64_t)E * N < (1ll << 31));
    if (!encode_tmap_u8_2d(&ta, A->data, (uint64_t)(K / ebytes_den), (uint64_t)R_cap,
                           (uint64_t)(A->ld / ebytes_den), 128, BM) ||
        (!b_mn && !encode_tmap_u8_2d(&tb, B->data, (uint64_t)(K / ebytes_den), (uint64_t)E * N,
                                     (uint64_t)(B->ld / ebytes_den), 128, 128)))
      return MGQ_ERR_CUDA;
    // 512-byte scale chunks per 128-row tile: MX 32x4-element blocks, NVFP4 16x4
    p.sfa_kb4 = A->ld / (nv ? 64 : 128);
    p.sfb_kb4 = B->ld / (nv ? 64 : 128);
  } else {
    MGQ_CHECK_ARG(N > 0 && K > 0 && N % BM == 0 && K % BN == 0);
    MGQ_CHECK_ARG((a_mn || A->ld >= R_cap) && (b_mn || B->ld >= R_cap));
    if (nv) MGQ_CHECK_ARG(R_cap % 256 == 0);
    if ((!a_mn && !encode_tmap_u8_2d(&ta, A->data, (uint64_t)(R_cap / ebytes_den), (uint64_t)N,
                                     (uint64_t)(A->ld / ebytes_den), 128, BM)) ||
        (!b_mn && !encode_tmap_u8_2d(&tb, B->data, (uint64_t)(R_cap / ebytes_den), (uint64_t)K,
                                     (uint64_t)(B->ld / ebytes_den), 128, 128)))
      return MGQ_ERR_CUDA;
    p.sfa_kb4 = A->ld / (nv ? 64 : 128);
    p.sfb_kb4 = B->ld / (nv ? 64 : 128);
  }
  int* err = error_word();
  if (!err) return MGQ_ERR_CUDA;
  p.offsets = offsets;
  p.E = E;
  p.N = N;
  // rows: contraction length in bytes of the operand rows (128 per stage);
  // contract: output columns
  p.K = mode == kModeRows ? K / ebytes_den : K;
  p.R_cap = R_cap;
  p.sfa = static_cast<const uint8_t*>(A->scale);
  p.sfb = static_cast<const uint8_t*>(B->scale);
  p.sfb_img = nv ? static_cast<const uint8_t*>(B->scale_image) : nullptr;
  if (p.sfb_img) MGQ_CHECK_ARG(aligned16(p.sfb_img));
  p.sa = nv ? A->global_scale : static_cast<const float*>(A->scale);
  p.sb = nv ? B->global_scale : static_cast<const float*>(B->scale);
  // block scales: A's scale_inv [k block][rows of A]; contract mode B's
  // [k block][rows of B = output columns]
  p.sa_ld = mode == kModeRows ? R_cap : N;
  p.sb_ld = mode == kModeRows ? 0 : K;
  p.out = out;
  p.ldo = (mode == kModeRows) ? N : K;
  p.out_f32 = out_dtype == MGQ_OUT_F32;
  p.beta = beta;
  p.tma_store = 0;
  p.a_mn = 0;
  p.b_mn = 0;
  p.kdiv = (nv && mode == kModeContract) ? 2 : 1;
  p.b_half2 = 128;
  p.swiglu = 0;
  p.F = 0;
  p.h_codes = nullptr;
  p.h_scales = nullptr;
  p.h_scale = nullptr;
  p.h_amax = nullptr;
  p.h_bf16 = nullptr;
  p.h_dtype = MGQ_E4M3;
  p.h_rceil = 1;
  p.dswiglu = 0;
  p.gu_in = nullptr;
  p.c_codes = nullptr;
  p.c_scales = nullptr;
  p.c_ld = R_cap;
  CUtensorMap th = ta;    // SwiGLU / dSwiGLU codes map (unused otherwise)
  if (sw) {
    // gate/up tiles: gate rows 128 n.. and up rows F + 128 n..; h quantised
    // row-wise with the GEMM's own scaling (MX or per-tensor)
    const mgq_qdesc* qh = sw->qh;
    const int64_t F = N / 2;
    if (mode != kModeRows || kind == kKindBlock || b_mn) return MGQ_ERR_UNSUPPORTED;
    MGQ_CHECK_ARG(qh && qh->row.data && aligned16(qh->row.data) && N % 256 == 0 && aligned16(sw->h_bf16));
    // a column-wise copy of h with NVFP4 (written by the second pass) or MX
    // (written by the epilogue); not per tensor
    if (qh->scaling != scaling || (qh->col.data && !nv && !mx)) return MGQ_ERR_UNSUPPORTED;
    if (nv) {
      // h in bf16 and its amax from the epilogue, then the NVFP4 cast
      if (qh->dtype != MGQ_E2M1) return MGQ_ERR_UNSUPPORTED;
      MGQ_CHECK_ARG(qh->row.scale && aligned16(qh->row.scale) && qh->amax_out && qh->tensor_scale && sw->h_bf16);
      if (qh->col.data) MGQ_CHECK_ARG(aligned16(qh->col.data) && qh->col.scale && aligned16(qh->col.scale));
    } else {
      if (qh->dtype != MGQ_E4M3 && qh->dtype != MGQ_E5M2) return MGQ_ERR_UNSUPPORTED;
      if (mx) MGQ_CHECK_ARG(qh->row.scale && aligned16(qh->row.scale));
      else MGQ_CHECK_ARG(qh->tensor_scale != nullptr);
      if (mx && qh->col.data) {
        MGQ_CHECK_ARG(aligned16(qh->col.data) && qh->col.scale && aligned16(qh->col.scale));
        p.c_codes = static_cast<uint8_t*>(qh->col.data);
        p.c_scales = static_cast<uint8_t*>(qh->col.scale);
      }
    }
    MGQ_CHECK_ARG(out_dtype == MGQ_OUT_BF16);
    p.swiglu = 1;
    p.F = F;
    p.b_half2 = F;
    p.h_codes = static_cast<uint8_t*>(qh->row.data);
    p.h_scales = static_cast<uint8_t*>(qh->row.scale);
    p.h_scale = qh->tensor_scale;
    p.h_amax = qh->amax_out;
    p.h_bf16 = static_cast<uint16_t*>(sw->h_bf16);
    p.h_dtype = qh->dtype;
    p.h_rceil = qh->e8m0_mode == MGQ_E8M0_RCEIL;
    const bool ok = nv ? encode_tmap_2d(&th, sw->h_bf16, 2, (uint64_t)F, (uint64_t)R_cap, (uint64_t)F * 2, 32, 32)
                       : encode_tmap_2d(&th, qh->row.data, 1, (uint64_t)F, (uint64_t)R_cap, (uint64_t)F, 64, 32);
    if (!ok) return MGQ_ERR_CUDA;
  }
  if (dsw) {
    // down-projection dgrad (N = F output columns): [dG | dU] quantised
    // row-wise into dsw->q ([R_cap, 2F] codes): per tensor, or MX (E8M0
    // blocks of 32 columns, and optionally the column-wise copy [2F, R_cap]
    // with blocks of 32 rows)
    const mgq_qdesc* q = dsw->q;
    const bool dsw_mx = kind == kKindMX && q->scaling == MGQ_MX32_E8M0;
    const bool dsw_pt = kind == kKindTensor && q->scaling == MGQ_TENSOR_F32 && !q->col.data;
    if (mode != kModeRows || !(dsw_mx || dsw_pt)) return MGQ_ERR_UNSUPPORTED;
    if (q->dtype != MGQ_E4M3 && q->dtype != MGQ_E5M2) return MGQ_ERR_UNSUPPORTED;
    MGQ_CHECK_ARG(q->row.data && aligned16(q->row.data) && dsw->gu && aligned16(dsw->gu) &&
                  aligned16(dsw->dgu_bf16) && N % 128 == 0 && out_dtype == MGQ_OUT_BF16);
    if (dsw_mx) {
      MGQ_CHECK_ARG(q->row.scale && aligned16(q->row.scale));
      if (q->col.data) {
        MGQ_CHECK_ARG(aligned16(q->col.data) && q->col.scale && aligned16(q->col.scale));
        p.c_codes = static_cast<uint8_t*>(q->col.data);
        p.c_scales = static_cast<uint8_t*>(q->col.scale);
      }
    } else {
      MGQ_CHECK_ARG(q->tensor_scale != nullptr);
    }
    p.dswiglu = 1;
    p.F = N;
    p.gu_in = static_cast<const uint16_t*>(dsw->gu);
    p.h_codes = static_cast<uint8_t*>(q->row.data);
    p.h_scales = static_cast<uint8_t*>(q->row.scale);
    p.h_scale = q->tensor_scale;
    p.h_amax = q->amax_out;
    p.h_bf16 = static_cast<uint16_t*>(dsw->dgu_bf16);
    p.h_dtype = q->dtype;
    p.h_rceil = q->e8m0_mode == MGQ_E8M0_RCEIL;
    if (!encode_tmap_2d(&th, q->row.data, 1, (uint64_t)(2 * N), (uint64_t)R_cap, (uint64_t)(2 * N), 64, 32))
      return MGQ_ERR_CUDA;
  }
  debug_knobs(&p.debug_stall, &p.wait_ns);
  p.idesc = nv   ? ptx::idesc_mxf4nvf4_ue4m3(BM, BN)
            : mx ? ptx::idesc_mxf8f6f4(A->dtype, B->dtype, BM, BN)
                 : ptx::idesc_f8f6f4(A->dtype, B->dtype, BM, BN);
  p.err = err;
  cudaStream_t s = as_stream(stream);
  // (the epilogue's MX column-wise copies and MX dSwiGLU run on the 1-CTA kernel)
  const bool mx_pair = kind == kKindMX && mx_pair_selected() && !p.c_codes && !p.dswiglu;
  if ((kind == kKindTensor || mx_pair || (nv && nv_pair_selected())) && use_pair_kernel(mode, N)) {
    // the pair kernel loads 128-row halves of B (K-major) or 128-column
    // halves (MN-major); MN-major operands are stored with the contraction
    // index down the rows:
    //   rows mode, B: W [E, Kc, ld >= N]; contract mode, A: dY [R_cap, ld >= N],
    //   B: X [R_cap, ld >= K]
    CUtensorMap tb2;
    bool ok;
    if (a_mn) {
      MGQ_CHECK_ARG(A->ld >= N);
      if (!encode_tmap_u8_2d(&ta, A->data, (uint64_t)N, (uint64_t)R_cap, (uint64_t)A->ld, 128, 128))
        return MGQ_ERR_CUDA;
    }
    if (b_mn && mode == kModeRows) {
      MGQ_CHECK_ARG(B->ld >= N && (int64_t)E * K < (1ll << 31));
      ok = encode_tmap_u8_2d(&tb2, B->data, (uint64_t)N, (uint64_t)E * K, (uint64_t)B->ld, 128, 128);
    } else if (b_mn) {
      MGQ_CHECK_ARG(B->ld >= K);
      ok = encode_tmap_u8_2d(&tb2, B->data, (uint64_t)K, (uint64_t)R_cap, (uint64_t)B->ld, 128, 128);
    } else {
      // (e2m1: the contraction extent and pitch in bytes)
      ok = mode == kModeRows
               ? encode_tmap_u8_2d(&tb2, B->data, (uint64_t)(K / ebytes_den), (uint64_t)E * N,
                                   (uint64_t)(B->ld / ebytes_den), 128, 128)
               : encode_tmap_u8_2d(&tb2, B->data, (uint64_t)(R_cap / ebytes_den), (uint64_t)K,
                                   (uint64_t)(B->ld / ebytes_den), 128, 128);
    }
    if (!ok) return MGQ_ERR_CUDA;
    p.a_mn = a_mn;
    p.b_mn = b_mn;
    p.idesc = nv   ? ptx::idesc_mxf4nvf4_ue4m3(256, BN)
              : mx ? ptx::idesc_mxf8f6f4(A->dtype, B->dtype, 256, BN)
                   : ptx::idesc_f8f6f4(A->dtype, B->dtype, 256, BN) | ptx::idesc_mn_major(a_mn, b_mn);
    // block scales as [chunks][128 words]: chunk (row tile, k chunk) = row tile * kb4 + k chunk;
    // a stage's box holds its chunks (MX 1, NVFP4 4)
    CUtensorMap tsfa = ta, tsfb = ta;
    if (mx || nv) {
      const int64_t rows_a = mode == kModeRows ? R_cap : N, rows_b = mode == kModeRows ? (int64_t)E * N : K;
      const uint32_t box = nv ? 4 : 1;
      if (!encode_tmap_2d(&tsfa, A->scale, 4, 128, (uint64_t)(rows_a / 128 * p.sfa_kb4), 512, 128, box) ||
          !encode_tmap_2d(&tsfb, B->scale, 4, 128, (uint64_t)(rows_b / 128 * p.sfb_kb4), 512, 128, box))
        return MGQ_ERR_CUDA;
    }
    // output map: [rows, ldo] elements, boxes of 64 bytes x 32 rows
    CUtensorMap to = th;
    const int eb = p.out_f32 ? 4 : 2;
    const uint64_t orows = mode == kModeRows ? (uint64_t)R_cap : (uint64_t)E * N;
    p.tma_store = (beta == 0.0f && !direct_store_forced()) ? 1 : 0;
    if (out && !encode_tmap_2d(&to, out, eb, (uint64_t)p.ldo, orows, (uint64_t)p.ldo * eb, 64 / eb, 32))
      return MGQ_ERR_CUDA;
    if (mx)
      return mode == kModeRows ? launch_gemm_pair<kModeRows, kKindMX>(ta, tb2, to, tsfa, tsfb, th, p, s)
                               : launch_gemm_pair<kModeContract, kKindMX>(ta, tb2, to, tsfa, tsfb, th, p, s);
    if (nv) {
      if (mode == kModeContract) return launch_gemm_pair<kModeContract, kKindNV>(ta, tb2, to, tsfa, tsfb, th, p, s);
      if (sw && cudaMemsetAsync(sw->qh->amax_out, 0, sizeof(float), s) != cudaSuccess) return MGQ_ERR_CUDA;
      rc = launch_gemm_pair<kModeRows, kKindNV>(ta, tb2, to, tsfa, tsfb, th, p, s);
      return (rc != MGQ_OK || !sw) ? rc : nv_swiglu_second_pass(sw, R_cap, offsets, E, N, s);
    }
    if (p.dswiglu) return launch_gemm_pair<kModeRows, kKindTensor, true>(ta, tb2, to, tsfa, tsfb, th, p, s);
    return mode == kModeRows ? launch_gemm_pair<kModeRows, kKindTensor>(ta, tb2, to, tsfa, tsfb, th, p, s)
                             : launch_gemm_pair<kModeContract, kKindTensor>(ta, tb2, to, tsfa, tsfb, th, p, s);
  }
  CUtensorMap to = th;
  {
    const int eb = p.out_f32 ? 4 : 2;
    const uint64_t orows = mode == kModeRows ? (uint64_t)R_cap : (uint64_t)E * N;
    // float32 block scales in contract mode: 128-byte swizzled boxes (the wide staging)
    const bool wide = wide_staging(kind, mode);
    if (out && !encode_tmap_2d(&to, out, eb, (uint64_t)p.ldo, orows, (uint64_t)p.ldo * eb, (wide ? 128 : 64) / eb,
                               32, wide))
      return MGQ_ERR_CUDA;
    p.tma_store = (beta == 0.0f && !direct_store_forced()) ? 1 : 0;
  }
  if (mode == kModeRows) {
    if (kind == kKindMX)
      return p.dswiglu ? launch_gemm<kModeRows, kKindMX, true>(ta, tb, to, th, p, s)
                       : launch_gemm<kModeRows, kKindMX>(ta, tb, to, th, p, s);
    if (kind == kKindTensor)
      return p.dswiglu ? launch_gemm<kModeRows, kKindTensor, true>(ta, tb, to, th, p, s)
                       : launch_gemm<kModeRows, kKindTensor>(ta, tb, to, th, p, s);
    if (kind == kKindNV) {
      if (sw && cudaMemsetAsync(sw->qh->amax_out, 0, sizeof(float), s) != cudaSuccess) return MGQ_ERR_CUDA;
      rc = launch_gemm<kModeRows, kKindNV>(ta, tb, to, th, p, s);
      if (rc != MGQ_OK || !sw) return rc;
      return nv_swiglu_second_pass(sw, R_cap, offsets, E, N, s);
    }
    return launch_gemm<kModeRows, kKindBlock>(ta, tb, to, th, p, s);
  }
  if (kind == kKindMX) return launch_gemm<kModeContract, kKindMX>(ta, tb, to, th, p, s);
  if (kind == kKindNV) return launch_gemm<kModeContract, kKindNV>(ta, tb, to, th, p, s);
  if (kind == kKindBlock) return launch_gemm<kModeContract, kKindBlock>(ta, tb, to, th, p, s);
  return launch_gemm<kModeContract, kKindTensor>(ta, tb, to, th, p, s);
}

}  // namespace
}  // namespace mgq

using namespace mgq;

namespace mgq {
namespace {
// The scale image of an NVFP4 operand: its 512-byte chunks in order, each
// written four times (chunk c at image chunks 4c .. 4c + 3). One thread per
// 16 bytes of the source; a warp moves one chunk.
__global__ void __launch_bounds__(256) nv_scale_image_kernel(const uint4* __restrict__ src, int64_t units,
                                                             uint4* __restrict__ dst) {
  const int64_t t = (int64_t)blockIdx.x * 256 + threadIdx.x;
  if (t >= units) return;
  const uint4 v = __ldg(src + t);
  uint4* d = dst + (t >> 5) * 128 + (t & 31);
#pragma unroll
  for (int q = 0; q < 4; ++q) d[32 * q] = v;
}
}  // namespace
}  // namespace mgq

extern "C" {

int mgq_grouped_gemm_fwd(const mgq_operand* A, const mgq_operand* W, int scaling, const int32_t* offsets, int E,
                         int64_t R_cap, int64_t N, int64_t K, void* Y, int out_dtype, void* stream) {
  return run_grouped(kModeRows, A, W, scaling, offsets, E, R_cap, N, K, 0.0f, Y, out_dtype, stream);
}

int mgq_grouped_gemm_dgrad(const mgq_operand* dY, const mgq_operand* Wcol, int scaling, const int32_t* offsets,
                           int E, int64_t R_cap, int64_t N, int64_t K, void* dA, int out_dtype, void* stream) {
  // dA [R_cap, K] = dY [R_cap, N] x Wcol_e [K, N]^T: a row-grouped GEMM with
  // contraction N and K output columns
  return run_grouped(kModeRows, dY, Wcol, scaling, offsets, E, R_cap, K, N, 0.0f, dA, out_dtype, stream);
}

int mgq_grouped_gemm_wgrad(const mgq_operand* dYcol, const mgq_operand* Acol, int scaling, const int32_t* offsets,
                           int E, int64_t R_cap, int64_t N, int64_t K, float beta, void* dW, int out_dtype,
                           void* stream) {
  return run_grouped(kModeContract, dYcol, Acol, scaling, offsets, E, R_cap, N, K, beta, dW, out_dtype, stream);
}

int mgq_grouped_gemm_dgrad_dswiglu(const mgq_operand* dY, const mgq_operand* W2, int scaling,
                                   const int32_t* offsets, int E, int64_t R_cap, int64_t H, int64_t F,
                                   const void* gu_bf16, const mgq_qdesc* q, void* dh_bf16, void* dgu_bf16,
                                   void* stream) {
  if (!q) return MGQ_ERR_INVALID_ARG;
  const DswigluOut dsw{gu_bf16, q, dgu_bf16};
  return run_grouped(kModeRows, dY, W2, scaling, offsets, E, R_cap, F, H, 0.0f, dh_bf16, MGQ_OUT_BF16, stream,
                     nullptr, &dsw);
}

int mgq_grouped_gemm_fwd_swiglu(const mgq_operand* A, const mgq_operand* W1, int scaling, const int32_t* offsets,
                                int E, int64_t R_cap, int64_t F, int64_t K, const mgq_qdesc* qh, void* gu_bf16,
                                void* h_bf16, void* stream) {
  if (F <= 0 || F % 128 != 0) return MGQ_ERR_INVALID_ARG;
  const SwigluOut sw{qh, h_bf16};
  return run_grouped(kModeRows, A, W1, scaling, offsets, E, R_cap, 2 * F, K, 0.0f, gu_bf16, MGQ_OUT_BF16, stream,
                     &sw);
}

int mgq_set_gemm_option(int option, int64_t value) {
  if (option < 0 || option >= MGQ_GEMM_OPT_COUNT) return MGQ_ERR_INVALID_ARG;
  if (value < 0 || (option != MGQ_GEMM_OPT_WAIT_MS && value > 1) ||
      (option == MGQ_GEMM_OPT_WAIT_MS && value > 600000))
    return MGQ_ERR_INVALID_ARG;
  g_gemm_opt[option].store(value, std::memory_order_relaxed);
  return MGQ_OK;
}

int mgq_get_gemm_option(int option, int64_t* value) {
  if (option < 0 || option >= MGQ_GEMM_OPT_COUNT || !value) return MGQ_ERR_INVALID_ARG;
  *value = g_gemm_opt[option].load(std::memory_order_relaxed);
  return MGQ_OK;
}

int mgq_nv_scale_image(const void* scale, int64_t rows, int64_t ld, void* image, void* stream) {
  using namespace mgq;
  MGQ_CHECK_ARG(scale && image && aligned16(scale) && aligned16(image));
  MGQ_CHECK_ARG(rows > 0 && rows % 128 == 0 && ld > 0 && ld % 256 == 0);
  const int64_t units = rows / 128 * (ld / 64) * 32;   // 16-byte units of the scales
  MGQ_CHECK_ARG((units + 255) / 256 < (1ll << 31));
  nv_scale_image_kernel<<<(unsigned)((units + 255) / 256), 256, 0, as_stream(stream)>>>(
      static_cast<const uint4*>(scale), units, static_cast<uint4*>(image));
  MGQ_LAUNCH_CHECK();
  return MGQ_OK;
}

}  // extern "C"
