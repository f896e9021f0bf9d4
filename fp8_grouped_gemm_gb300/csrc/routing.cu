// Token dispatch: routing (stable counting sort of the (token, slot) entries
// by expert) and the fused permute + amax + scale + cast of the token rows.
//
// Grouping rows by expert so that one grouped GEMM covers all experts, with
// expert inputs padded for FP8: "[BUG] Loss difference when training with FP8
// vs. BF16 MoE" (Megatron-LM issue #1152, repro steps and additional
// context); padding to the quantisation block as the required layout: "FP8BlockQuantizer
// not work on TE" (TransformerEngine issue #2393, maintainer replies);
// dynamic quantisation in front of the scaled grouped mm: "float8 moe
// training conversion API prototype" (pytorch/ao PR #2275, description).
#include <algorithm>

#include "device_common.cuh"
#include "mgq_internal.h"
#include "rowquant.cuh"

namespace mgq {
namespace {

constexpr int kChunk = 1024;        // routing entries per chunk
constexpr int kRouteThreads = 256;
constexpr int kMaxExperts = 1024;

// ---- routing pass 1: per-chunk histogram and stable rank inside the chunk ----
// Entries of a chunk are taken in order, 256 per round; within a warp,
// __match_any_sync finds the lanes with the same expert and the rank is the
// number of such lanes before this one; warps and rounds before it add their
// counts. The rank inside the chunk is parked in row_id_map (the permute
// kernel adds the chunk's base row); the chunk's counts go to cnt[chunk][e].
__global__ void route_count_rank_kernel(const int32_t* __restrict__ idx, int64_t n, int E,
                                        int32_t* __restrict__ cnt, int32_t* __restrict__ row_id_map, int* err) {
  extern __shared__ int smem[];
  int* s_run = smem;                 // [E] entries of this chunk already ranked
  int* s_w = smem + E;               // [8][E] per-warp counts of this round
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int e = threadIdx.x; e < E; e += blockDim.x) s_run[e] = 0;
  const int64_t cbase = (int64_t)blockIdx.x * kChunk;
  for (int round = 0; round < kChunk / kRouteThreads; ++round) {
    for (int i = threadIdx.x; i < 8 * E; i += blockDim.x) s_w[i] = 0;
    __syncthreads();
    const int64_t g = cbase + round * kRouteThreads + threadIdx.x;
    int key = -1;
    if (g < n) {
      key = idx[g];
      if (key < 0 || key >= E) {
        report(err, MGQ_ERR_DEVICE_INDEX);
        key = -1;
      }
    }
    const unsigned peers = __match_any_sync(0xFFFFFFFFu, key);
    const int rank = __popc(peers & ((1u << lane) - 1u));
    if (key >= 0 && rank == 0) s_w[warp * E + key] = __popc(peers);
    __syncthreads();
    if (key >= 0) {
      int r = s_run[key] + rank;
      for (int w = 0; w < warp; ++w) r += s_w[w * E + key];
      row_id_map[g] = r;
    } else if (g < n) {
      row_id_map[g] = -1;
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
      int sum = 0;
      for (int w = 0; w < 8; ++w) sum += s_w[w * E + e];
      s_run[e] += sum;
    }
    __syncthreads();
  }
  for (int e = threadIdx.x; e < E; e += blockDim.x) cnt[(int64_t)blockIdx.x * E + e] = s_run[e];
}

// inclusive warp scan
__device__ __forceinline__ int warp_incl_scan(int v, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int u = __shfl_up_sync(0xFFFFFFFFu, v, o);
    if (lane >= o) v += u;
  }
  return v;
}

// ---- routing pass 2 (one CTA of 1024 threads): totals, padded exclusive
// scan over experts, and the first destination row of every (chunk, expert)
// pair (in place in cnt); filler rows of every group get src_row -1 ----------
__global__ void __launch_bounds__(1024) route_scan_kernel(int32_t* __restrict__ cnt, int nchunks, int E, int align,
                                                          int32_t* __restrict__ offsets, int32_t* __restrict__ counts,
                                                          int32_t* __restrict__ src_row) {
  __shared__ int s_tot[kMaxExperts];
  __shared__ int s_off[kMaxExperts + 1];
  __shared__ int s_wsum[32];
  __shared__ int s_seg[32][33];      // [warp = chunk segment][lane = expert of the block]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // Blocks of 32 experts (lane = expert); warp w takes the contiguous chunk
  // segment [w S, (w + 1) S), so every load reads 32 consecutive experts of
  // one chunk. Pass 1: per-segment sums -> expert totals.
  const int S = (nchunks + 31) / 32;
  const int c_lo = warp * S, c_hi = min(nchunks, c_lo + S);
  for (int eb = 0; eb < E; eb += 32) {
    const int e = eb + lane;
    int t = 0;
    if (e < E)
      for (int c = c_lo; c < c_hi; ++c) t += cnt[(int64_t)c * E + e];
    s_seg[warp][lane] = t;
    __syncthreads();
    if (warp == 0 && e < E) {
      int tot = 0;
      for (int w = 0; w < 32; ++w) tot += s_seg[w][lane];
      s_tot[e] = tot;
    }
    __syncthreads();
  }
  // exclusive scan of the padded totals (E <= 1024: one per thread)
  const int e0 = threadIdx.x;
  const int pad = e0 < E ? (s_tot[e0] + align - 1) / align * align : 0;
  const int incl = warp_incl_scan(pad, lane);
  if (lane == 31) s_wsum[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int v = warp_incl_scan(s_wsum[lane], lane);
    s_wsum[lane] = v;
  }
  __syncthreads();
  const int excl = incl - pad + (warp > 0 ? s_wsum[warp - 1] : 0);
  if (e0 < E) {
    s_off[e0] = excl;
    offsets[e0] = excl;
    counts[e0] = s_tot[e0];
  }
  if (e0 == 0) {
    s_off[E] = s_wsum[31];
    offsets[E] = s_wsum[31];
  }
  __syncthreads();
  // Pass 2: per-(chunk, expert) base rows (in place): the expert's offset plus
  // the segments before this warp's, then a running sum along the segment.
  for (int eb = 0; eb < E; eb += 32) {
    const int e = eb + lane;
    int t = 0;
    if (e < E)
      for (int c = c_lo; c < c_hi; ++c) t += cnt[(int64_t)c * E + e];
    s_seg[warp][lane] = t;
    __syncthreads();
    if (e < E) {
      int run = s_off[e];
      for (int w = 0; w < warp; ++w) run += s_seg[w][lane];
      for (int c = c_lo; c < c_hi; ++c) {
        const int v = cnt[(int64_t)c * E + e];
        cnt[(int64_t)c * E + e] = run;
        run += v;
      }
    }
    __syncthreads();
  }
  // filler rows of every group
  for (int e = warp; e < E; e += 32)
    for (int r = s_off[e] + s_tot[e] + lane; r < s_off[e + 1]; r += 32) src_row[r] = -1;
}

// Final destination row of routing entry g (lane-level): the chunk's base row
// for the entry's expert plus the entry's rank inside the chunk; written back
// to row_id_map with the inverse map src_row. -1 for an invalid entry.
__device__ __forceinline__ int resolve_row(const int32_t* __restrict__ idx, int32_t* row_id_map,
                                           const int32_t* __restrict__ base, int32_t* src_row, int E, int64_t g) {
  const int local = row_id_map[g];
  if (local < 0) return -1;
  const int e = idx[g];
  const int r = base[(g / kChunk) * E + e] + local;
  row_id_map[g] = r;
  src_row[r] = (int32_t)g;
  return r;
}

// ---- fused permute + quantise ---------------------------------------------------
// One warp per token row, in 1024-element chunks: per tensor, lane l takes
// 8-element runs 256 apart (fully coalesced loads); with block scales,
// 16-element runs 512 apart (half an MX block, an eighth of a 1x128 block).
// The row is read once and its codes and scales are written to the k
// destination rows.

struct PermuteArgs {
  const uint16_t* x;
  int T, H, k, E;
  const int32_t* offsets;
  const int32_t* counts;
  uint8_t* codes;          // [R_cap, H]
  uint8_t* scales;         // layout per scaling mode
  uint16_t* out_bf16;      // [R_cap, H] or null
  const float* tensor_scale;
  float* amax_out;
  float* s_out;            // NVFP4: receives s_g
  int64_t R_cap;
  int e8m0_rceil;
  int token_blocks;        // CTAs that process tokens; the rest fill padding
  int* err;
  const int32_t* idx;      // [T, k] expert ids
  const int32_t* base;     // [chunks][E] first row of each (chunk, expert)
  int32_t* rim;            // row_id_map: rank inside the chunk in, final row out
  int32_t* src_row;
  int resolve;             // 0: rim already holds the final rows
  int nv_rowmajor;         // NVFP4: write the scales row-major ([R_cap][H/16]) for retile_nv_scales
};

// ---- routing pass 3 (standalone routing only): final rows and src_row -------
__global__ void route_finalize_kernel(const int32_t* __restrict__ idx, int64_t n, int E,
                                      const int32_t* __restrict__ base, int32_t* __restrict__ row_id_map,
                                      int32_t* __restrict__ src_row) {
  const int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (g < n) resolve_row(idx, row_id_map, base, src_row, E, g);
}

// Every lane gets the k destination rows of token t (lane j resolves entry j,
// or reads it when the routing is already final).
__device__ __forceinline__ void token_rows(const PermuteArgs& a, int t, uint32_t lane, int (&dest)[8]) {
  int mine = -1;
  if ((int)lane < a.k)
    mine = a.resolve ? resolve_row(a.idx, a.rim, a.base, a.src_row, a.E, (int64_t)t * a.k + lane)
                     : a.rim[(int64_t)t * a.k + lane];
#pragma unroll
  for (int j = 0; j < 8; ++j) dest[j] = __shfl_sync(0xFFFFFFFFu, mine, j);
}

template <int SC, int DT>
__global__ void __launch_bounds__(256, 4) permute_quant_kernel(PermuteArgs a) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int H = a.H;
  if ((int)blockIdx.x >= a.token_blocks) {
    // ---- padding rows of expert e: zero codes (and zero scales) -------------
    int e = blockIdx.x - a.token_blocks;
    if (e >= a.E) return;
    int64_t lo = a.offsets[e] + a.counts[e], hi = a.offsets[e + 1];
    for (int64_t r = lo + warp; r < hi; r += 8) {
      for (int c = lane * 16; c < H; c += 32 * 16)
        *reinterpret_cast<uint4*>(a.codes + r * H + c) = make_uint4(0, 0, 0, 0);
      if (a.out_bf16)
        for (int c = lane * 8; c < H; c += 32 * 8)
          *reinterpret_cast<uint4*>(a.out_bf16 + r * H + c) = make_uint4(0, 0, 0, 0);
      if (SC == MGQ_MX32_E8M0) {
        const int64_t kb4 = H / 128;
        for (int b4 = lane; b4 < H / 128; b4 += 32)
          *reinterpret_cast<uint32_t*>(a.scales + tiled_scale_offset(r, (int64_t)b4 * 4, kb4)) = 0u;
      } else if (SC == MGQ_BLK_1x128_F32) {
        float* s = reinterpret_cast<float*>(a.scales);
        for (int b = lane; b < H / 128; b += 32) s[(int64_t)b * a.R_cap + r] = 0.0f;
      }
    }
    return;
  }
  // token CTAs stride over the tokens (a few waves' worth of CTAs, no tail
  // wave); a warp keeps the next 1024-element chunk in flight, across token
  // boundaries too. Lane l holds the runs of G elements at 32 G q + G l
  // (q < 32 / G). G = 8 (per tensor): each 16-byte load of the warp covers 512
  // contiguous bytes. G = 16 (block scales): a 32-block spans 2 lanes (a 1x128
  // block 8), so a chunk needs two scale computations per lane, against four
  // with G = 8; the warp's loads cover 1 KB (8 lines) each.
  constexpr int G = SC == MGQ_TENSOR_F32 ? 8 : 16;
  constexpr int NQ = 32 / G;          // runs per lane and chunk
  constexpr int WQ = G / 2;           // bf16-pair words per run
  constexpr int LB = 32 / G;          // lanes per 32-element block
  const int tstride = a.token_blocks * 8;
  auto load_chunk = [&](int tt, int c0, uint32_t (&w)[16]) {
    const uint16_t* row = a.x + (int64_t)tt * H + c0 + lane * G;
#pragma unroll
    for (int q = 0; q < NQ; ++q) {
      const bool in = c0 + 32 * G * q + (int)lane * G < H;
#pragma unroll
      for (int u = 0; u < G / 8; ++u) {
        uint4 v = make_uint4(0, 0, 0, 0);
        if (in) v = __ldg(reinterpret_cast<const uint4*>(row + 32 * G * q + 8 * u));
        uint32_t* d = &w[WQ * q + 4 * u];
        d[0] = v.x; d[1] = v.y; d[2] = v.z; d[3] = v.w;
      }
    }
  };
  const float ts = (SC == MGQ_TENSOR_F32) ? a.tensor_scale[0] : 1.0f;
  uint32_t tamax = 0;   // per-tensor amax (bf16 bits in the high half)
  int t = blockIdx.x * 8 + warp;
  uint32_t wnext[16];
  if (t < a.T) load_chunk(t, 0, wnext);
  for (; t < a.T; t += tstride) {
  int dest[8];
  token_rows(a, t, lane, dest);
  for (int c0 = 0; c0 < H; c0 += 1024) {
    uint32_t w[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) w[i] = wnext[i];
    if (c0 + 1024 < H) load_chunk(t, c0 + 1024, wnext);
    else if (t + tstride < a.T) load_chunk(t + tstride, 0, wnext);
#pragma unroll
    for (int q = 0; q < NQ; ++q) {
      const int c = c0 + 32 * G * q + lane * G;
      const bool active = c < H;     // every lane stays in the loop (shuffles below)
      const uint32_t* wq = &w[WQ * q];
      uint32_t am2 = 0;
#pragma unroll
      for (int i = 0; i < WQ; ++i) am2 = absmax_bf16x2(am2, wq[i]);
      uint32_t amax_bits = fold_bf16x2(am2);
      float mult;
      uint32_t scode = 0;
      float sinv = 0.0f;
      if (SC == MGQ_MX32_E8M0) {
#pragma unroll
        for (int o = 1; o < LB; o <<= 1) amax_bits = max(amax_bits, __shfl_xor_sync(0xFFFFFFFFu, amax_bits, o));
        const int e = mx_exponent(amax_bits, FmtInfo<DT>::emax, a.e8m0_rceil != 0);
        mult = mx_multiplier(e);
        scode = mx_scale_code(e);
      } else if (SC == MGQ_BLK_1x128_F32) {
        // amax over 128 elements = 4 LB lanes
        uint32_t m = amax_bits;
#pragma unroll
        for (int o = 1; o < 4 * LB; o <<= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
        const float am = __uint_as_float(m);
        float sc = (m == 0) ? 1.0f : __fdiv_rn(FmtInfo<DT>::fmax, am);
        if (isinf(sc)) sc = 3.40282347e38f;
        mult = sc;
        sinv = __fdiv_rn(1.0f, sc);
      } else {  // MGQ_TENSOR_F32
        mult = ts;
        tamax = max(tamax, amax_bits);
      }
      uint32_t cw[G / 4];
#pragma unroll
      for (int i = 0; i < G / 4; ++i) cw[i] = cvt_fp8x4_bf16_mul<DT>(wq[2 * i], wq[2 * i + 1], mult);
      // MX: the 4 scale bytes of 4 consecutive blocks (lanes 4 LB j, + LB, ..) into lane 4 LB j
      uint32_t s4 = 0;
      if (SC == MGQ_MX32_E8M0) {
        const uint32_t b1 = __shfl_down_sync(0xFFFFFFFFu, scode, LB);
        const uint32_t b2 = __shfl_down_sync(0xFFFFFFFFu, scode, 2 * LB);
        const uint32_t b3 = __shfl_down_sync(0xFFFFFFFFu, scode, 3 * LB);
        s4 = scode | (b1 << 8) | (b2 << 16) | (b3 << 24);
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        if (j >= a.k || !active) break;
        const int r = dest[j];
        if (r < 0) continue;
        uint8_t* dst = a.codes + (int64_t)r * H + c;
        if (G == 8) {
          *reinterpret_cast<uint2*>(dst) = make_uint2(cw[0], cw[1]);
        } else {
#pragma unroll
          for (int u = 0; u < G / 16; ++u)
            reinterpret_cast<uint4*>(dst)[u] = make_uint4(cw[4 * u], cw[4 * u + 1], cw[4 * u + 2], cw[4 * u + 3]);
        }
        if (a.out_bf16) {
          uint4* ob = reinterpret_cast<uint4*>(a.out_bf16 + (int64_t)r * H + c);
#pragma unroll
          for (int u = 0; u < G / 8; ++u) ob[u] = make_uint4(wq[4 * u], wq[4 * u + 1], wq[4 * u + 2], wq[4 * u + 3]);
        }
        if (SC == MGQ_MX32_E8M0) {
          if ((lane & (4 * LB - 1)) == 0)
            *reinterpret_cast<uint32_t*>(a.scales + tiled_scale_offset(r, c / 32, H / 128)) = s4;
        } else if (SC == MGQ_BLK_1x128_F32) {
          if ((lane & (4 * LB - 1)) == 0) reinterpret_cast<float*>(a.scales)[(int64_t)(c / 128) * a.R_cap + r] = sinv;
        }
      }
    }
  }
  }
  if (SC == MGQ_TENSOR_F32 && a.amax_out) {
    // one atomic per CTA (every warp of a token CTA gets here): thousands of
    // same-address atomics would queue at one L2 slice
    __shared__ uint32_t s_am[8];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) tamax = max(tamax, __shfl_xor_sync(0xFFFFFFFFu, tamax, o));
    if (lane == 0) s_am[warp] = tamax;
    __syncthreads();
    if (threadIdx.x == 0) {
      for (int w = 1; w < 8; ++w) tamax = max(tamax, s_am[w]);
      atomic_max_nonneg(a.amax_out, __uint_as_float(tamax));
    }
  }
}

// ---- fused permute + NVFP4 quantisation (after the amax pass over X) -----------
__global__ void __launch_bounds__(256) permute_quant_nv_kernel(PermuteArgs a) {
  const int warp = threadIdx.x >> 5;
  const uint32_t lane = threadIdx.x & 31;
  const int H = a.H;
  if ((int)blockIdx.x >= a.token_blocks) {
    const int e = blockIdx.x - a.token_blocks;
    if (e >= a.E) return;
    const int64_t lo = a.offsets[e] + a.counts[e], hi = a.offsets[e + 1];
    for (int64_t r = lo + warp; r < hi; r += 8) {
      for (int c = lane * 32; c < H; c += 32 * 32)
        *reinterpret_cast<uint4*>(a.codes + r * (H / 2) + c / 2) = make_uint4(0, 0, 0, 0);
      for (int b4 = lane; b4 < H / 64; b4 += 32)
        *reinterpret_cast<uint32_t*>(a.scales + (a.nv_rowmajor ? r * (H / 16) + b4 * 4
                                                                : tiled_scale_offset(r, (int64_t)b4 * 4, H / 64))) = 0u;
    }
    return;
  }
  const float s_g = nv_global_scale(*a.amax_out);
  if (blockIdx.x == 0 && warp == 0 && lane == 0) *a.s_out = s_g;
  // token CTAs stride over the tokens
  for (int t = blockIdx.x * 8 + warp; t < a.T; t += a.token_blocks * 8) {
  int dest[8];
  token_rows(a, t, lane, dest);
  for (int c0 = 0; c0 < H; c0 += 1024) {
    const int c = c0 + lane * 32;
    const bool act = c < H;
    float v[32];
    if (act) {
      load_bf16x32(a.x + (int64_t)t * H + c, v);
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i) v[i] = 0.0f;
    }
    Block32nv o;
    quantize32_nv(v, s_g, o);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (j >= a.k || !act) break;
      const int r = dest[j];
      if (r < 0) continue;
      if (a.nv_rowmajor) {
        // codes as usual; the lane pair's 4 scale bytes at their row-major place
        *reinterpret_cast<uint4*>(a.codes + (int64_t)r * (H / 2) + c / 2) = make_uint4(o.cw[0], o.cw[1], o.cw[2], o.cw[3]);
        if ((lane & 1) == 0) *reinterpret_cast<uint32_t*>(a.scales + (int64_t)r * (H / 16) + c / 16) = o.s4;
      } else {
        store32_nv(o, a.codes, a.scales, r, c, H, lane);
      }
    }
  }
  }
}

// ---- NVFP4 scales: row-major -> 128x4-tiled, in place ------------------------
// A token row's scales go to k scattered destination rows; in the tiled
// layout each row owns only 4 contiguous bytes of every 512-byte tile, so the
// permute writes them row-major (64 contiguous bytes per warp and destination)
// and this pass re-tiles them. The 128 rows of a row group occupy the same
// 128 x H/16 bytes in both layouts, so each CTA loads its group's block into
// shared memory (row stride kb4 + 1 words: conflict-free column reads) and
// writes it back tiled. Groups past the used rows (offsets[E]) are left alone.
__global__ void __launch_bounds__(256) retile_nv_scales_kernel(uint8_t* scales, int kb4, const int32_t* rows_used) {
  extern __shared__ uint32_t rt_words[];          // [128][kb4 + 1]
  const int64_t g = blockIdx.x;
  if (g * 128 >= (int64_t)*rows_used) return;
  uint8_t* blk = scales + g * (int64_t)kb4 * 512;
  const int ld = kb4 + 1;
  const int nvec = 128 * kb4 / 4;                 // 16-byte pieces of the block
  for (int v = threadIdx.x; v < nvec; v += blockDim.x) {
    const uint4 x = reinterpret_cast<const uint4*>(blk)[v];
    const int w = 4 * v, row = w / kb4, jj = w - row * kb4;   // kb4 is a multiple of 4 (H % 256 == 0)
    uint32_t* d = rt_words + row * ld + jj;
    d[0] = x.x; d[1] = x.y; d[2] = x.z; d[3] = x.w;
  }
  __syncthreads();
  // tile j, line l (16 bytes): word j of rows l, l + 32, l + 64, l + 96
  for (int line = threadIdx.x; line < kb4 * 32; line += blockDim.x) {
    const int jj = line >> 5, l = line & 31;
    reinterpret_cast<uint4*>(blk)[line] = make_uint4(rt_words[l * ld + jj], rt_words[(l + 32) * ld + jj],
                                                     rt_words[(l + 64) * ld + jj], rt_words[(l + 96) * ld + jj]);
  }
}

// ---- byte transpose of the used rows: dst[c, r] = src[r, c] -----------------
// 64x64 tiles through shared memory; rows >= *rows_used are skipped.
__global__ void transpose_u8_kernel(const uint8_t* __restrict__ src, int64_t src_ld, uint8_t* __restrict__ dst,
                                    int64_t dst_ld, const int32_t* __restrict__ rows_used, int64_t rows_cap,
                                    int64_t cols) {
  __shared__ uint32_t tile[64][17];   // 64 rows x 64 bytes, padded
  const int64_t r0 = (int64_t)blockIdx.x * 64, c0 = (int64_t)blockIdx.y * 64;
  const int64_t nrows = rows_used ? (int64_t)*rows_used : rows_cap;
  if (r0 >= nrows) return;
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;   // 256 threads: 16 x 16
  for (int rr = ty; rr < 64; rr += 16) {
    int64_t r = r0 + rr;
    tile[rr][tx] = (r < nrows) ? *reinterpret_cast<const uint32_t*>(src + r * src_ld + c0 + tx * 4) : 0u;
  }
  __syncthreads();
  // thread writes 4 consecutive rows (bytes) of one output row (column c)
  for (int cc = ty; cc < 64; cc += 16) {
    int64_t c = c0 + cc;
    if (c >= cols) continue;
    uint32_t v = 0;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      int rr = tx * 4 + q;
      uint32_t word = tile[rr][cc >> 2];
      v |= ((word >> ((cc & 3) * 8)) & 0xFFu) << (8 * q);
    }
    if (r0 + tx * 4 < nrows) *reinterpret_cast<uint32_t*>(dst + c * dst_ld + r0 + tx * 4) = v;
  }
}

}  // namespace

// launched by other translation units (per-tensor column-wise copies)
int launch_transpose_u8(const uint8_t* src, int64_t src_ld, uint8_t* dst, int64_t dst_ld, const int32_t* rows_used,
                        int64_t rows_cap, int64_t cols, cudaStream_t s) {
  dim3 grid((unsigned)((rows_cap + 63) / 64), (unsigned)((cols + 63) / 64));
  transpose_u8_kernel<<<grid, 256, 0, s>>>(src, src_ld, dst, dst_ld, rows_used, rows_cap, cols);
  MGQ_LAUNCH_CHECK();
  return MGQ_OK;
}

}  // namespace mgq

using namespace mgq;

extern "C" {

size_t mgq_permute_workspace_size(int T, int k, int E) {
  if (T < 0 || k <= 0 || E <= 0) return 0;
  int64_t n = (int64_t)T * k;
  int64_t nchunks = (n + kChunk - 1) / kChunk;
  if (nchunks == 0) nchunks = 1;
  return (size_t)(nchunks * E * sizeof(int32_t));
}

}  // extern "C"

namespace mgq {
namespace {

int check_permute_q(const mgq_qdesc* q, int align) {
  if (!q) return MGQ_ERR_UNSUPPORTED;   // bf16-only dispatch is not needed by the layer
  MGQ_CHECK_ARG(q->row.data && aligned16(q->row.data));
  if (q->scaling == MGQ_NV16_UE4M3) {
    MGQ_CHECK_ARG(q->dtype == MGQ_E2M1 && q->row.scale && aligned16(q->row.scale) && q->amax_out &&
                  q->tensor_scale);
    if (q->col.data) MGQ_CHECK_ARG(aligned16(q->col.data) && q->col.scale && aligned16(q->col.scale) && align % 32 == 0);
    return MGQ_OK;
  }
  MGQ_CHECK_ARG(q->dtype == MGQ_E4M3 || q->dtype == MGQ_E5M2);
  if (q->scaling == MGQ_MX32_E8M0 || q->scaling == MGQ_BLK_1x128_F32)
    MGQ_CHECK_ARG(q->row.scale && aligned16(q->row.scale));
  else if (q->scaling == MGQ_TENSOR_F32)
    MGQ_CHECK_ARG(q->tensor_scale != nullptr);
  else
    return MGQ_ERR_UNSUPPORTED;
  if (q->col.data) {
    // column blocks run inside the groups: groups padded to the block (MX 32, blockwise 128)
    MGQ_CHECK_ARG(aligned16(q->col.data) && align % (q->scaling == MGQ_BLK_1x128_F32 ? 128 : 32) == 0);
    if (q->scaling != MGQ_TENSOR_F32) MGQ_CHECK_ARG(q->col.scale && aligned16(q->col.scale));
  }
  return MGQ_OK;
}

int check_route_args(int T, int k, int E, int align, int64_t R_cap, const void* rim, const void* src_row,
                     const void* offsets, const void* counts) {
  MGQ_CHECK_ARG(T >= 0 && k >= 1 && k <= 8 && E >= 1 && E <= kMaxExperts && k <= E);
  MGQ_CHECK_ARG(align >= 1 && (align % 32 == 0 || align == 1));
  MGQ_CHECK_ARG((T == 0 || rim) && src_row && offsets && counts);   // no entries: row_id_map may be null
  const int64_t n = (int64_t)T * k;
  const int64_t need = ((n + (int64_t)E * (align - 1)) + 127) / 128 * 128;
  MGQ_CHECK_ARG(R_cap >= need && R_cap % 128 == 0 && R_cap < (1ll << 31));
  return MGQ_OK;
}

// routing passes 1 and 2 (and 3 when `finalize`; otherwise the permute
// kernel resolves the rows itself from the chunk ranks and bases)
int route_impl(const int32_t* topk_idx, int T, int k, int E, int align, int32_t* row_id_map, int32_t* src_row,
               int32_t* offsets, int32_t* counts, int32_t* cnt, bool finalize, int* err, cudaStream_t s) {
  const int64_t n = (int64_t)T * k;
  const int64_t nchunks = (n + kChunk - 1) / kChunk;
  if (nchunks > 0) {
    route_count_rank_kernel<<<(unsigned)nchunks, kRouteThreads, 9 * E * sizeof(int), s>>>(topk_idx, n, E, cnt,
                                                                                           row_id_map, err);
    MGQ_LAUNCH_CHECK();
  }
  route_scan_kernel<<<1, 1024, 0, s>>>(cnt, (int)nchunks, E, align, offsets, counts, src_row);
  MGQ_LAUNCH_CHECK();
  if (finalize && n > 0) {
    route_finalize_kernel<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(topk_idx, n, E, cnt, row_id_map, src_row);
    MGQ_LAUNCH_CHECK();
  }
  return MGQ_OK;
}

// block scales (MX, NVFP4, blockwise) with a column-wise copy and no bf16
// copy: one tile pass over the permuted rows writes both copies (needs the
// final src_row)
bool permute_fused_rowcol(const mgq_qdesc* q, const void* out_bf16) {
  return (q->scaling == MGQ_MX32_E8M0 || q->scaling == MGQ_NV16_UE4M3 || q->scaling == MGQ_BLK_1x128_F32) &&
         q->col.data && !out_bf16;
}

// permute + quantise of the token rows to their routed rows (row_id_map final,
// or chunk ranks to resolve with `idx` and the chunk bases `cnt`)
int permute_impl(const void* x_bf16, int T, int H, int k, int E, const mgq_qdesc* q, void* out_bf16, int64_t R_cap,
                 int32_t* row_id_map, int32_t* src_row, const int32_t* offsets, const int32_t* counts,
                 const int32_t* idx, const int32_t* cnt, bool resolve, int* err, cudaStream_t s) {
  if (!resolve && permute_fused_rowcol(q, out_bf16)) {
    if (q->scaling == MGQ_NV16_UE4M3) {   // s_g needs the amax of X first
      const int rc = launch_amax_groups(static_cast<const uint16_t*>(x_bf16), (int64_t)T * H, 1, q->amax_out, s);
      if (rc != MGQ_OK) return rc;
    }
    return gather_x_rowcol(static_cast<const uint16_t*>(x_bf16), src_row, k, H, R_cap, offsets + E, true, q, s);
  }
  PermuteArgs a;
  a.x = static_cast<const uint16_t*>(x_bf16);
  a.T = T; a.H = H; a.k = k; a.E = E;
  a.offsets = offsets; a.counts = counts;
  a.idx = idx; a.base = cnt; a.rim = row_id_map; a.src_row = src_row;
  a.resolve = resolve ? 1 : 0;
  a.codes = static_cast<uint8_t*>(q->row.data);
  a.scales = static_cast<uint8_t*>(q->row.scale);
  a.out_bf16 = static_cast<uint16_t*>(out_bf16);
  a.tensor_scale = q->tensor_scale;
  a.amax_out = q->amax_out;
  a.s_out = q->tensor_scale;
  a.R_cap = R_cap;
  a.e8m0_rceil = q->e8m0_mode == MGQ_E8M0_RCEIL;
  a.nv_rowmajor = 0;
  // token CTAs: FP8 kernels stride over the tokens from at most four resident
  // waves (keeping the next chunk in flight across tokens); the NVFP4 kernel,
  // whose tokens fan out to many destinations, runs one token per warp
  a.token_blocks = q->scaling == MGQ_NV16_UE4M3 ? (T + 7) / 8
                                                : (int)std::min<int64_t>((T + 7) / 8, (int64_t)num_sms() * 4);
  a.err = err;
  dim3 grid((unsigned)(a.token_blocks + E));
  const int sc = q->scaling, dt = q->dtype;
  if (sc == MGQ_NV16_UE4M3) {
    int rc = launch_amax_groups(a.x, (int64_t)T * H, 1, q->amax_out, s);
    if (rc != MGQ_OK) return rc;
    // row-major scales and a re-tiling pass, when a row group's scales fit a
    // CTA's shared memory
    const int kb4 = H / 64;
    const size_t rt_smem = (size_t)128 * (kb4 + 1) * 4;
    a.nv_rowmajor = (H % 256 == 0 && rt_smem <= 200 * 1024) ? 1 : 0;
    if (a.nv_rowmajor && rt_smem > 48 * 1024) {
      if (cudaFuncSetAttribute(retile_nv_scales_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)rt_smem) !=
          cudaSuccess)
        return MGQ_ERR_CUDA;
    }
    permute_quant_nv_kernel<<<grid, 256, 0, s>>>(a);
    MGQ_LAUNCH_CHECK();
    if (a.nv_rowmajor) {
      retile_nv_scales_kernel<<<(unsigned)(R_cap / 128), 256, rt_smem, s>>>(static_cast<uint8_t*>(q->row.scale), kb4,
                                                                          offsets + E);
      MGQ_LAUNCH_CHECK();
    }
    // column-wise copy (16-row blocks along the permuted rows) from the gathered rows
    if (q->col.data) return gather_x_rowcol(a.x, src_row, k, H, R_cap, offsets + E, false, q, s);
    return MGQ_OK;
  }
#define MGQ_PERMUTE_LAUNCH(SC, DT) permute_quant_kernel<SC, DT><<<grid, 256, 0, s>>>(a)
  if (sc == MGQ_MX32_E8M0 && dt == MGQ_E4M3) MGQ_PERMUTE_LAUNCH(MGQ_MX32_E8M0, MGQ_E4M3);
  else if (sc == MGQ_MX32_E8M0 && dt == MGQ_E5M2) MGQ_PERMUTE_LAUNCH(MGQ_MX32_E8M0, MGQ_E5M2);
  else if (sc == MGQ_BLK_1x128_F32 && dt == MGQ_E4M3) MGQ_PERMUTE_LAUNCH(MGQ_BLK_1x128_F32, MGQ_E4M3);
  else if (sc == MGQ_BLK_1x128_F32 && dt == MGQ_E5M2) MGQ_PERMUTE_LAUNCH(MGQ_BLK_1x128_F32, MGQ_E5M2);
  else if (sc == MGQ_TENSOR_F32 && dt == MGQ_E4M3) MGQ_PERMUTE_LAUNCH(MGQ_TENSOR_F32, MGQ_E4M3);
  else if (sc == MGQ_TENSOR_F32 && dt == MGQ_E5M2) MGQ_PERMUTE_LAUNCH(MGQ_TENSOR_F32, MGQ_E5M2);
  else return MGQ_ERR_UNSUPPORTED;
#undef MGQ_PERMUTE_LAUNCH
  MGQ_LAUNCH_CHECK();
  if (q->col.data) {
    // per-tensor: the column copy is the transposed cast of the row codes;
    // MX: blocks of 32 along the permuted rows, from the gathered bf16 rows
    int rc = q->scaling == MGQ_TENSOR_F32
                 ? launch_transpose_u8(static_cast<const uint8_t*>(q->row.data), H,
                                       static_cast<uint8_t*>(q->col.data), R_cap, offsets + E, R_cap, H, s)
                 : gather_x_rowcol(a.x, src_row, k, H, R_cap, offsets + E, false, q, s);
    if (rc != MGQ_OK) return rc;
  }
  return MGQ_OK;
}

}  // namespace
}  // namespace mgq

extern "C" {

int mgq_moe_permute(const void* x_bf16, int T, int H, const int32_t* topk_idx, int k, int E, int align,
                    const mgq_qdesc* q, void* out_bf16, int64_t R_cap, int32_t* row_id_map, int32_t* src_row,
                    int32_t* offsets, int32_t* counts, void* workspace, size_t ws_bytes, void* stream) {
  int rc = check_route_args(T, k, E, align, R_cap, row_id_map, src_row, offsets, counts);
  if (rc != MGQ_OK) return rc;
  MGQ_CHECK_ARG(H > 0 && H % 128 == 0 && workspace && (T == 0 || (x_bf16 && topk_idx)));
  MGQ_CHECK_ARG(ws_bytes >= mgq_permute_workspace_size(T, k, E));
  MGQ_CHECK_ARG(aligned16(x_bf16) && aligned16(out_bf16));
  if ((rc = check_permute_q(q, align)) != MGQ_OK) return rc;
  int* err = error_word();
  if (!err) return MGQ_ERR_CUDA;
  cudaStream_t s = as_stream(stream);
  int32_t* cnt = static_cast<int32_t*>(workspace);
  // two routing launches and the permute kernel resolving the final rows, or
  // (fused row + column copies) three routing launches and the tile pass
  const bool fused = permute_fused_rowcol(q, out_bf16);
  if ((rc = route_impl(topk_idx, T, k, E, align, row_id_map, src_row, offsets, counts, cnt, fused, err, s)) != MGQ_OK)
    return rc;
  return permute_impl(x_bf16, T, H, k, E, q, out_bf16, R_cap, row_id_map, src_row, offsets, counts, topk_idx, cnt,
                      !fused, err, s);
}

int mgq_moe_route(const int32_t* topk_idx, int T, int k, int E, int align, int64_t R_cap, int32_t* row_id_map,
                  int32_t* src_row, int32_t* offsets, int32_t* counts, void* workspace, size_t ws_bytes,
                  void* stream) {
  int rc = check_route_args(T, k, E, align, R_cap, row_id_map, src_row, offsets, counts);
  if (rc != MGQ_OK) return rc;
  MGQ_CHECK_ARG(workspace && (T == 0 || topk_idx) && ws_bytes >= mgq_permute_workspace_size(T, k, E));
  int* err = error_word();
  if (!err) return MGQ_ERR_CUDA;
  return route_impl(topk_idx, T, k, E, align, row_id_map, src_row, offsets, counts,
                    static_cast<int32_t*>(workspace), true, err, as_stream(stream));
}

int mgq_moe_permute_routed(const void* x_bf16, int T, int H, int k, int E, const mgq_qdesc* q, void* out_bf16,
                           int64_t R_cap, const int32_t* row_id_map, const int32_t* src_row,
                           const int32_t* offsets, const int32_t* counts, void* stream) {
  int rc = check_route_args(T, k, E, 1, R_cap, row_id_map, src_row, offsets, counts);
  if (rc != MGQ_OK) return rc;
  MGQ_CHECK_ARG(H > 0 && H % 128 == 0 && (T == 0 || x_bf16) && aligned16(x_bf16) && aligned16(out_bf16));
  // (the group alignment a column copy needs is the routing's, stated by the caller)
  if ((rc = check_permute_q(q, 128)) != MGQ_OK) return rc;
  int* err = error_word();
  if (!err) return MGQ_ERR_CUDA;
  // the kernels only read row_id_map and src_row when the rows are final
  return permute_impl(x_bf16, T, H, k, E, q, out_bf16, R_cap, const_cast<int32_t*>(row_id_map),
                      const_cast<int32_t*>(src_row), offsets, counts, nullptr, nullptr, false, err,
                      as_stream(stream));
}

}  // extern "C"
