// HBM-bound steps of the routed-expert layer, each fused with the
// quantisation of its output: SwiGLU (+ its derivative), unpermute / combine
// and its backward, permute backward, block quantisation of grouped weights,
// and the delayed-scaling amax history.
//
// Sources: the SwiGLU experts of the Mixtral / Llama4 layers ("[BUG] Loss
// difference when training with FP8 vs. BF16 MoE", Megatron-LM issue #1152;
// "float8 moe training conversion API prototype", pytorch/ao PR #2275, testing:
// outputs, input gradients and parameter gradients); row-wise and column-wise
// copies with their own scales ("Numerical fix for moe single grouped weight
// with fp8 fp4 primary weight and grad norm spikes", Megatron-LM PR #5487;
// "FP8BlockQuantizer not work on TE", TransformerEngine issue #2393, transpose
// identity); delayed scaling with a 1024-long history and max (issue #1152,
// repro steps).
#include <algorithm>

#include "mgq_internal.h"
#include "rowquant.cuh"

namespace mgq {
namespace {

constexpr int kWarps = 8;

// CTA-wide max of the warps' per-tensor amax (float bits), one atomic per CTA.
// Every thread of the CTA must call it.
__device__ __forceinline__ void cta_amax_atomic(uint32_t tam, float* out) {
  __shared__ uint32_t s_am[kWarps];
  tam = warp_max_u32(tam);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) s_am[warp] = tam;
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t m = 0;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) m = max(m, s_am[w]);
    atomic_max_nonneg(out, __uint_as_float(m));
  }
}

// ---- SwiGLU + quantise: warp per row ----------------------------------------
struct SwigluArgs {
  const uint16_t* gu;   // [R_cap, 2F]
  const int32_t* rows_used;
  int64_t R_cap;
  int F;
  uint8_t* codes;       // [R_cap, F]
  uint8_t* scales;
  uint16_t* h_out;      // [R_cap, F] or null
  const float* tensor_scale;
  float* amax_out;
  int rceil;
};


template <int SC, int DT>
__global__ void __launch_bounds__(256) swiglu_quant_kernel(SwigluArgs a) {
  const int warp = threadIdx.x >> 5;
  const uint32_t lane = threadIdx.x & 31;
  const int64_t r = (int64_t)blockIdx.x * kWarps + warp;
  const bool row_ok = r < *a.rows_used;
  const int F = a.F;
  const float ts = (SC == MGQ_TENSOR_F32) ? a.tensor_scale[0] : 1.0f;
  uint32_t tam = 0;
  for (int c0 = 0; row_ok && c0 < F; c0 += 1024) {
    const int c = c0 + 32 * lane;
    const bool act = c < F;
    float h[32];
    if (act) {
      float g[32], u[32];
      load_bf16x32(a.gu + r * 2 * F + c, g);
      load_bf16x32(a.gu + r * 2 * F + F + c, u);
#pragma unroll
      for (int i = 0; i < 32; ++i) h[i] = swiglu_bf16(g[i], u[i]);
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i) h[i] = 0.0f;
    }
    const uint32_t am = absmax_bits_f32(h, 32);
    tam = max(tam, am);
    Block32 o;
    quantize32<SC, DT>(h, am, ts, a.rceil != 0, o);
    if (act) {
      store32<SC>(o, a.codes, a.scales, r, c, F, a.R_cap, lane);
      if (a.h_out) store_bf16x32(a.h_out + r * F + c, h);
    }
  }
  if (SC == MGQ_TENSOR_F32 && a.amax_out) cta_amax_atomic(tam, a.amax_out);
}

// ---- dSwiGLU + quantise: warp per row ---------------------------------------
struct DswigluArgs {
  const uint16_t* dh;   // [R_cap, F]
  const uint16_t* gu;   // [R_cap, 2F]
  const int32_t* rows_used;
  int64_t R_cap;
  int F;
  uint8_t* codes;       // [R_cap, 2F]
  uint8_t* scales;
  uint16_t* dgu_out;    // [R_cap, 2F] or null
  const float* tensor_scale;
  float* amax_out;
  int rceil;
};

template <int SC, int DT>
__global__ void __launch_bounds__(256) dswiglu_quant_kernel(DswigluArgs a) {
  const int warp = threadIdx.x >> 5;
  const uint32_t lane = threadIdx.x & 31;
  const int64_t r = (int64_t)blockIdx.x * kWarps + warp;
  const bool row_ok = r < *a.rows_used;
  const int F = a.F;
  const float ts = (SC == MGQ_TENSOR_F32) ? a.tensor_scale[0] : 1.0f;
  uint32_t tam = 0;
  for (int c0 = 0; row_ok && c0 < F; c0 += 1024) {
    const int c = c0 + 32 * lane;
    const bool act = c < F;
    float dg[32], du[32];
    if (act) {
      float d[32], g[32], u[32];
      load_bf16x32(a.dh + r * F + c, d);
      load_bf16x32(a.gu + r * 2 * F + c, g);
      load_bf16x32(a.gu + r * 2 * F + F + c, u);
#pragma unroll
      for (int i = 0; i < 32; i += 2) dswiglu_bf16x2(d + i, g + i, u + i, dg + i, du + i);
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i) dg[i] = du[i] = 0.0f;
    }
    const uint32_t amg = absmax_bits_f32(dg, 32), amu = absmax_bits_f32(du, 32);
    tam = max(tam, max(amg, amu));
    Block32 og, ou;
    quantize32<SC, DT>(dg, amg, ts, a.rceil != 0, og);
    quantize32<SC, DT>(du, amu, ts, a.rceil != 0, ou);
    if (act) {
      store32<SC>(og, a.codes, a.scales, r, c, 2 * F, a.R_cap, lane);
      store32<SC>(ou, a.codes, a.scales, r, F + c, 2 * F, a.R_cap, lane);
      if (a.dgu_out) {
        store_bf16x32(a.dgu_out + r * 2 * F + c, dg);
        store_bf16x32(a.dgu_out + r * 2 * F + F + c, du);
      }
    }
  }
  if (SC == MGQ_TENSOR_F32 && a.amax_out) cta_amax_atomic(tam, a.amax_out);
}

// ---- combine: out[t] = sum_j w_j * y[row(t, j)] (w = probs, or 1) -----------
// CTAs of the combine kernels: at most three resident waves
unsigned combine_grid(int T, int k) {
  return (unsigned)std::min<int64_t>((T + kWarps - 1) / kWarps, (int64_t)num_sms() * (k <= 2 ? 3 : 2));
}

// KMAX: the largest k the instance serves (2 or 8)
template <int KMAX>
__global__ void __launch_bounds__(256) combine_kernel(const uint16_t* __restrict__ y, const int32_t* __restrict__ rim,
                                                      const float* __restrict__ probs, int T, int k, int H,
                                                      uint16_t* __restrict__ out) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // CTAs stride over the tokens (a few resident waves, no tail wave)
  for (int t = blockIdx.x * kWarps + warp; t < T; t += gridDim.x * kWarps) {
  int rows[KMAX];
  float w[KMAX];
#pragma unroll
  for (int j = 0; j < KMAX; ++j) {
    rows[j] = j < k ? rim[(int64_t)t * k + j] : -1;
    w[j] = (j < k && probs) ? probs[(int64_t)t * k + j] : 1.0f;
  }
  // four 256-element column blocks per iteration, rows in pairs: every lane
  // keeps 8 independent 16-byte loads in flight
  for (int c0 = 0; c0 < H; c0 += 1024) {
    float acc[4][8];
#pragma unroll
    for (int q = 0; q < 4; ++q)
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[q][i] = 0.0f;
#pragma unroll
    for (int j0 = 0; j0 < KMAX; j0 += 2) {
      if (j0 >= k) break;
      uint4 v[2][4];
#pragma unroll
      for (int jj = 0; jj < 2; ++jj) {
        const int j = j0 + jj;
        const int r = j < k ? rows[j] : -1;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int c = c0 + q * 256 + lane * 8;
          v[jj][q] = (r >= 0 && c < H) ? __ldg(reinterpret_cast<const uint4*>(y + (int64_t)r * H + c))
                                       : make_uint4(0, 0, 0, 0);
        }
      }
#pragma unroll
      for (int jj = 0; jj < 2; ++jj) {
        const int j = j0 + jj;
        if (j >= k || rows[j] < 0) continue;    // a missing row adds nothing (not even -0.0)
        const float wj = w[j];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint4 u = v[jj][q];
          acc[q][0] = fmaf(wj, bf16_lo(u.x), acc[q][0]); acc[q][1] = fmaf(wj, bf16_hi(u.x), acc[q][1]);
          acc[q][2] = fmaf(wj, bf16_lo(u.y), acc[q][2]); acc[q][3] = fmaf(wj, bf16_hi(u.y), acc[q][3]);
          acc[q][4] = fmaf(wj, bf16_lo(u.z), acc[q][4]); acc[q][5] = fmaf(wj, bf16_hi(u.z), acc[q][5]);
          acc[q][6] = fmaf(wj, bf16_lo(u.w), acc[q][6]); acc[q][7] = fmaf(wj, bf16_hi(u.w), acc[q][7]);
        }
      }
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int c = c0 + q * 256 + lane * 8;
      if (c < H)
        *reinterpret_cast<uint4*>(out + (int64_t)t * H + c) =
            make_uint4(pack_bf16x2(acc[q][0], acc[q][1]), pack_bf16x2(acc[q][2], acc[q][3]),
                       pack_bf16x2(acc[q][4], acc[q][5]), pack_bf16x2(acc[q][6], acc[q][7]));
    }
  }
}
}

// ---- unpermute backward + quantise of dY, and dprobs ------------------------
struct UnpermBwdArgs {
  const uint16_t* dout;  // [T, H]
  const uint16_t* y;     // [R_cap, H]
  const int32_t* rim;
  const int32_t* src_row;
  const float* probs;
  const int32_t* offsets;
  int T, k, H, E;
  int64_t R_cap;
  uint8_t* codes;        // [R_cap, H]
  uint8_t* scales;
  const float* tensor_scale;
  float* amax_out;       // per-tensor: max |dY| (optional); NVFP4: the pre-pass amax (input)
  float* s_out;          // NVFP4: s_g (output)
  float* dprobs;
  int rceil;
  int token_blocks;
};

// amax of dY = probs[t, j] * dout[t] over the routed entries (row_id_map >= 0):
// float32 products round monotonically, so the maximum of |fl(p d)| over a
// token's row is fl(|p| max |d|). One warp per token (strided), one atomic per CTA.
__global__ void __launch_bounds__(256) dy_amax_kernel(const uint16_t* dout, const float* probs, const int32_t* rim,
                                                      int T, int k, int H, float* amax) {
  const int warp = threadIdx.x >> 5;
  const uint32_t lane = threadIdx.x & 31;
  uint32_t tam = 0;
  for (int64_t t = (int64_t)blockIdx.x * kWarps + warp; t < T; t += (int64_t)gridDim.x * kWarps) {
    uint32_t acc = 0;
    for (int c = 8 * lane; c < H; c += 256) {
      const uint4 w = __ldg(reinterpret_cast<const uint4*>(dout + t * H + c));
      acc = absmax_acc_bf16x2(absmax_acc_bf16x2(absmax_acc_bf16x2(absmax_acc_bf16x2(acc, w.x), w.y), w.z), w.w);
    }
    const float dmax = __uint_as_float(warp_max_u32(fold_bf16x2(absmax_bf16x2_final(acc))));
    if (lane < (uint32_t)k && rim[t * k + lane] >= 0)
      tam = max(tam, __float_as_uint(__fmul_rn(fabsf(probs[t * k + lane]), dmax)));
  }
  cta_amax_atomic(tam, amax);
}

// One warp per routing entry (t, j): row r = row_id_map[t, j] receives the
// codes of probs[t, j] * dout[t] and dprobs[t, j] = <dout[t], Y[r]>. Lane l
// covers elements [32 l, 32 l + 32) of each 1024-element chunk; the loads of
// the next chunk are issued before the current one is processed, so every
// warp keeps two chunks of dout and Y in flight.
template <int SC, int DT>
__global__ void __launch_bounds__(256, SC == MGQ_TENSOR_F32 ? 3 : 2) unpermute_bwd_kernel(UnpermBwdArgs a) {
  const int warp = threadIdx.x >> 5;
  const uint32_t lane = threadIdx.x & 31;
  const int H = a.H;
  if ((int)blockIdx.x >= a.token_blocks) {
    // filler rows of expert e (the tail of its group, where src_row < 0;
    // found by binary search): zero codes and scales
    const int e = blockIdx.x - a.token_blocks;
    if (e >= a.E) return;
    int64_t lo = a.offsets[e], hi = a.offsets[e + 1];
    while (lo < hi) {
      const int64_t mid = (lo + hi) >> 1;
      if (a.src_row[mid] >= 0) lo = mid + 1;
      else hi = mid;
    }
    constexpr int kBytesDen = SC == MGQ_NV16_UE4M3 ? 2 : 1;     // e2m1: two codes per byte
    constexpr int kBlk = SC == MGQ_NV16_UE4M3 ? 16 : 32;          // elements per scale byte
    for (int64_t r = lo + warp; r < a.offsets[e + 1]; r += kWarps) {
      for (int c = lane * 16; c < H / kBytesDen; c += 512)
        *reinterpret_cast<uint4*>(a.codes + r * (H / kBytesDen) + c) = make_uint4(0, 0, 0, 0);
      if (SC == MGQ_MX32_E8M0 || SC == MGQ_NV16_UE4M3)
        for (int b4 = lane; b4 < H / (4 * kBlk); b4 += 32)
          *reinterpret_cast<uint32_t*>(a.scales + tiled_scale_offset(r, (int64_t)b4 * 4, H / (4 * kBlk))) = 0u;
      else if (SC == MGQ_BLK_1x128_F32)
        for (int b = lane; b < H / 128; b += 32) reinterpret_cast<float*>(a.scales)[(int64_t)b * a.R_cap + r] = 0.0f;
    }
    return;
  }
  // NVFP4: s_g from the dY amax pre-pass, published by the first warp
  const float s_g = SC == MGQ_NV16_UE4M3 ? nv_global_scale(a.amax_out[0]) : 1.0f;
  if (SC == MGQ_NV16_UE4M3 && blockIdx.x == 0 && threadIdx.x == 0) a.s_out[0] = s_g;
  uint32_t tam = 0;
  // the entry CTAs stride over the routing entries t * k + j
  for (int64_t g = (int64_t)blockIdx.x * kWarps + warp; g < (int64_t)a.T * a.k; g += (int64_t)a.token_blocks * kWarps) {
  const int r = a.rim[g];
  if (r >= 0) {
    const float ts = (SC == MGQ_TENSOR_F32) ? a.tensor_scale[0] : 1.0f;
    const float pr = a.probs[g];
    const uint16_t* drow = a.dout + (g / a.k) * H;
    const uint16_t* yrow = a.y + (int64_t)r * H;
    float dp = 0.0f;
    // per tensor (codes element by element), lane l takes the 8-element runs
    // 256 q + 8 l of a 1024-element chunk, so each 16-byte load of the warp
    // covers 512 contiguous bytes; with block scales it takes its own block(s)
    constexpr bool kRuns = SC == MGQ_TENSOR_F32;
    auto load = [&](int c0, uint4 (&d)[4], uint4 (&y)[4]) {
      const int c = c0 + 32 * (int)lane;
      if (kRuns) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int cq = c0 + 256 * q + 8 * (int)lane;
          d[q] = y[q] = make_uint4(0, 0, 0, 0);
          if (cq < H) {
            d[q] = __ldg(reinterpret_cast<const uint4*>(drow + cq));
            y[q] = __ldg(reinterpret_cast<const uint4*>(yrow + cq));
          }
        }
      } else if (c < H) {
        const uint4* pd = reinterpret_cast<const uint4*>(drow + c);
        const uint4* py = reinterpret_cast<const uint4*>(yrow + c);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          d[q] = __ldg(pd + q);
          y[q] = __ldg(py + q);
        }
      } else {
#pragma unroll
        for (int q = 0; q < 4; ++q) d[q] = y[q] = make_uint4(0, 0, 0, 0);
      }
    };
    auto process = [&](int c0, const uint4 (&d)[4], const uint4 (&y)[4]) {
      const int c = c0 + 32 * (int)lane;
      float v[32];
      float s = 0.0f;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint32_t dw[4] = {d[q].x, d[q].y, d[q].z, d[q].w};
        const uint32_t yw[4] = {y[q].x, y[q].y, y[q].z, y[q].w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float d0 = bf16_lo(dw[i]), d1 = bf16_hi(dw[i]);
          s = fmaf(d0, bf16_lo(yw[i]), s);
          s = fmaf(d1, bf16_hi(yw[i]), s);
          v[8 * q + 2 * i] = __fmul_rn(pr, d0);
          v[8 * q + 2 * i + 1] = __fmul_rn(pr, d1);
        }
      }
      dp += s;
      if constexpr (SC == MGQ_NV16_UE4M3) {
        Block32nv o;
        quantize32_nv(v, s_g, o);
        if (c < H) store32_nv(o, a.codes, a.scales, r, c, H, lane);
      } else {
        const uint32_t am = absmax_bits_f32(v, 32);
        tam = max(tam, am);
        Block32 o;
        quantize32<SC, DT>(v, am, ts, a.rceil != 0, o);
        if (kRuns) {
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int cq = c0 + 256 * q + 8 * (int)lane;
            if (cq < H) *reinterpret_cast<uint2*>(a.codes + (int64_t)r * H + cq) = make_uint2(o.cw[2 * q], o.cw[2 * q + 1]);
          }
        } else if (c < H) {
          store32<SC>(o, a.codes, a.scales, r, c, H, a.R_cap, lane);
        }
      }
    };
    uint4 d0[4], y0[4], d1[4], y1[4];
    load(0, d0, y0);
    for (int c0 = 0; c0 < H; c0 += 2048) {
      load(c0 + 1024, d1, y1);
      process(c0, d0, y0);
      if (c0 + 1024 >= H) break;
      load(c0 + 2048, d0, y0);
      process(c0 + 1024, d1, y1);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) dp += __shfl_xor_sync(0xFFFFFFFFu, dp, o);
    if (lane == 0) a.dprobs[g] = dp;
  } else if (lane == 0) {
    a.dprobs[g] = 0.0f;
  }
  }
  if (SC == MGQ_TENSOR_F32 && a.amax_out) cta_amax_atomic(tam, a.amax_out);
}

// ---- row-wise quantisation of [G*M, K] (grouped weights) ---------------------
struct QuantRowsArgs {
  const uint16_t* x;
  int64_t rows, M, K;
  uint8_t* codes;
  uint8_t* scales;
  const float* tensor_scale;   // per group
  float* amax_out;             // per group
  int rceil;
};

template <int SC, int DT>
__global__ void __launch_bounds__(256) quant_rows_kernel(QuantRowsArgs a) {
  const int warp = threadIdx.x >> 5;
  const uint32_t lane = threadIdx.x & 31;
  // a CTA's 8 rows lie in one group (M is a multiple of 128)
  const int64_t r = (int64_t)blockIdx.x * kWarps + warp;
  const int64_t g = ((int64_t)blockIdx.x * kWarps) / a.M;
  const float ts = (SC == MGQ_TENSOR_F32) ? a.tensor_scale[g] : 1.0f;
  uint32_t tam = 0;
  for (int64_t c0 = 0; r < a.rows && c0 < a.K; c0 += 1024) {
    const int64_t c = c0 + 32 * lane;
    const bool act = c < a.K;
    float v[32];
    if (act) {
      load_bf16x32(a.x + r * a.K + c, v);
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i) v[i] = 0.0f;
    }
    const uint32_t am = absmax_bits_f32(v, 32);
    tam = max(tam, am);
    Block32 o;
    quantize32<SC, DT>(v, am, ts, a.rceil != 0, o);
    if (act) store32<SC>(o, a.codes, a.scales, r, c, a.K, a.rows, lane);
  }
  if (SC == MGQ_TENSOR_F32 && a.amax_out) cta_amax_atomic(tam, a.amax_out + g);
}


// ---- 128x128 tile quantisation of grouped weights [G, N, K] ------------------
// One CTA per tile; 256 threads, thread i covers row i/2, 64 columns. The tile
// amax gives s = fmax / amax (float32, IEEE division; 1 for an all-zero tile;
// FLT_MAX on overflow); codes = cast(x * s); scale_inv = 1 / s at
// [(g * N/128 + n/128) * K/128 + k/128].
template <int DT>
__global__ void __launch_bounds__(256, 4) quant_tile128_kernel(const uint16_t* __restrict__ x, int64_t N, int64_t K,
                                                               uint8_t* __restrict__ codes, float* __restrict__ sinv) {
  // one tile per CTA; a thread's 64 values stay packed bf16 pairs (32
  // registers), so four CTAs fit an SM. Each load instruction of a warp
  // covers two whole 256-byte tile rows, so every sector it requests is used
  // in full (16-byte lanes at a wider stride leave each request's sectors
  // half used)
  __shared__ uint32_t s_max[8];
  const int64_t nb = N / 128, kb = K / 128;
  const int64_t tile = blockIdx.x;
  const int64_t g = tile / (nb * kb), rem = tile % (nb * kb);
  // chunk q of this thread: tile row 16 q + t / 16, 16-byte column chunk t % 16
  // (a warp's load covers two whole 256-byte rows)
  const int64_t base = (g * N + (rem / kb) * 128 + threadIdx.x / 16) * K + (rem % kb) * 128 + (threadIdx.x % 16) * 8;
  uint4 w[8];
#pragma unroll
  for (int q = 0; q < 8; ++q) w[q] = __ldg(reinterpret_cast<const uint4*>(x + base + (int64_t)q * 16 * K));
  uint32_t acc = 0;
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    acc = absmax_acc_bf16x2(acc, w[q].x);
    acc = absmax_acc_bf16x2(acc, w[q].y);
    acc = absmax_acc_bf16x2(acc, w[q].z);
    acc = absmax_acc_bf16x2(acc, w[q].w);
  }
  uint32_t m = warp_max_u32(fold_bf16x2(absmax_bf16x2_final(acc)));
  if ((threadIdx.x & 31) == 0) s_max[threadIdx.x >> 5] = m;
  __syncthreads();
  m = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) m = max(m, s_max[i]);
  const float sc = blk_scale<DT>(m);
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    const uint4 a = w[q];
    *reinterpret_cast<uint2*>(codes + base + (int64_t)q * 16 * K) = make_uint2(
        cvt_fp8x4<DT>(__fmul_rn(bf16_lo(a.x), sc), __fmul_rn(bf16_hi(a.x), sc), __fmul_rn(bf16_lo(a.y), sc),
                      __fmul_rn(bf16_hi(a.y), sc)),
        cvt_fp8x4<DT>(__fmul_rn(bf16_lo(a.z), sc), __fmul_rn(bf16_hi(a.z), sc), __fmul_rn(bf16_lo(a.w), sc),
                      __fmul_rn(bf16_hi(a.w), sc)));
  }
  if (threadIdx.x == 0) sinv[tile] = __fdiv_rn(1.0f, sc);
}


// ---- NVFP4 support: per-group amax, then row quantisation with s_g -------------

// amax[g] = max |x| over group g ([G][per_group] bf16, per_group % 8 == 0).
// amax must hold +0 (or a smaller value) before the launch.
__global__ void __launch_bounds__(256) amax_groups_kernel(const uint16_t* __restrict__ x, int64_t per_group,
                                                          float* __restrict__ amax) {
  __shared__ uint32_t s_m[8];
  const int64_t g = blockIdx.y;
  const uint16_t* base = x + g * per_group;
  uint32_t m2 = 0;
  for (int64_t i = ((int64_t)blockIdx.x * 256 + threadIdx.x) * 8; i < per_group; i += (int64_t)gridDim.x * 256 * 8) {
    const uint4 w = __ldg(reinterpret_cast<const uint4*>(base + i));
    m2 = absmax_bf16x2(m2, w.x);
    m2 = absmax_bf16x2(m2, w.y);
    m2 = absmax_bf16x2(m2, w.z);
    m2 = absmax_bf16x2(m2, w.w);
  }
  uint32_t m = warp_max_u32(fold_bf16x2(m2));
  if ((threadIdx.x & 31) == 0) s_m[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int i = 1; i < 8; ++i) m = max(m, s_m[i]);
    atomic_max_nonneg(amax + g, __uint_as_float(m));
  }
}

// NVFP4 row quantisation of [rows, K] bf16 in groups of M rows: warp per row;
// s_g from the group's amax (also written to s_out[g] by the group's first row).
struct QuantRowsNvArgs {
  const uint16_t* x;
  int64_t rows, M, K;
  const int32_t* rows_used;    // device row count or null
  uint8_t* codes;              // [rows, K/2]
  uint8_t* scales;             // tiled ue4m3
  const float* amax;           // per group
  float* s_out;                // per group
};

__global__ void __launch_bounds__(256) quant_rows_nv_kernel(QuantRowsNvArgs a) {
  const int warp = threadIdx.x >> 5;
  const uint32_t lane = threadIdx.x & 31;
  const int64_t r = (int64_t)blockIdx.x * kWarps + warp;
  const int64_t nrows = a.rows_used ? (int64_t)*a.rows_used : a.rows;
  if (r >= nrows) return;
  const int64_t g = r / a.M;
  const float s_g = nv_global_scale(a.amax[g]);
  if (r % a.M == 0 && lane == 0) a.s_out[g] = s_g;
  for (int64_t c0 = 0; c0 < a.K; c0 += 1024) {
    const int64_t c = c0 + 32 * lane;
    const bool act = c < a.K;
    float v[32];
    if (act) {
      load_bf16x32(a.x + r * a.K + c, v);
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i) v[i] = 0.0f;
    }
    Block32nv o;
    quantize32_nv(v, s_g, o);
    if (act) store32_nv(o, a.codes, a.scales, r, c, a.K, lane);
  }
}

// SwiGLU pass of the NVFP4 path: h = bf16(silu(g) * u) written out, and the
// tensor amax of h accumulated (the quantisation needs it first).
__global__ void __launch_bounds__(256) swiglu_h_kernel(const uint16_t* __restrict__ gu, const int32_t* rows_used, int F,
                                                       uint16_t* __restrict__ h, float* amax) {
  const int warp = threadIdx.x >> 5;
  const uint32_t lane = threadIdx.x & 31;
  const int64_t r = (int64_t)blockIdx.x * kWarps + warp;
  const bool live = r < *rows_used;      // (all warps stay for the CTA's amax reduction)
  uint32_t tam = 0;
  for (int c0 = 0; live && c0 < F; c0 += 1024) {
    const int c = c0 + 32 * lane;
    if (c < F) {
      float g[32], u[32], hv[32];
      load_bf16x32(gu + r * 2 * F + c, g);
      load_bf16x32(gu + r * 2 * F + F + c, u);
#pragma unroll
      for (int i = 0; i < 32; ++i) hv[i] = swiglu_bf16(g[i], u[i]);
      tam = max(tam, absmax_bits_f32(hv, 32));
      store_bf16x32(h + r * F + c, hv);
    }
  }
  cta_amax_atomic(tam, amax);
}

// [dG | dU] = dSwiGLU(dh, g, u) (bf16, as the quantising kernels round them)
// and its amax: the first pass of the NVFP4 dSwiGLU quantisation
__global__ void __launch_bounds__(256) dswiglu_dgu_kernel(const uint16_t* __restrict__ dh,
                                                          const uint16_t* __restrict__ gu, const int32_t* rows_used,
                                                          int F, uint16_t* __restrict__ dgu, float* amax) {
  const int warp = threadIdx.x >> 5;
  const uint32_t lane = threadIdx.x & 31;
  const int64_t r = (int64_t)blockIdx.x * kWarps + warp;
  const bool live = r < *rows_used;      // (all warps stay for the CTA's amax reduction)
  uint32_t tam = 0;
  for (int c0 = 0; live && c0 < F; c0 += 1024) {
    const int c = c0 + 32 * lane;
    if (c < F) {
      float d[32], g[32], u[32], dg[32], du[32];
      load_bf16x32(dh + r * F + c, d);
      load_bf16x32(gu + r * 2 * F + c, g);
      load_bf16x32(gu + r * 2 * F + F + c, u);
#pragma unroll
      for (int i = 0; i < 32; i += 2) dswiglu_bf16x2(d + i, g + i, u + i, dg + i, du + i);
      tam = max(tam, max(absmax_bits_f32(dg, 32), absmax_bits_f32(du, 32)));
      store_bf16x32(dgu + r * 2 * F + c, dg);
      store_bf16x32(dgu + r * 2 * F + F + c, du);
    }
  }
  cta_amax_atomic(tam, amax);
}

// max |x| over the rows [0, *rows_used) of a bf16 [rows, C] matrix: one warp
// per row (strided), one atomic per CTA (amax zeroed by the caller)
__global__ void __launch_bounds__(256) amax_rows_kernel(const uint16_t* __restrict__ x, const int32_t* rows_used,
                                                        int64_t C, float* amax) {
  const int warp = threadIdx.x >> 5;
  const uint32_t lane = threadIdx.x & 31;
  const int64_t n = *rows_used;
  uint32_t tam = 0;
  for (int64_t r = (int64_t)blockIdx.x * kWarps + warp; r < n; r += (int64_t)gridDim.x * kWarps) {
    uint32_t acc = 0;
    for (int64_t c = 8 * lane; c < C; c += 256) {
      const uint4 w = __ldg(reinterpret_cast<const uint4*>(x + r * C + c));
      acc = absmax_acc_bf16x2(absmax_acc_bf16x2(absmax_acc_bf16x2(absmax_acc_bf16x2(acc, w.x), w.y), w.z), w.w);
    }
    tam = max(tam, warp_max_u32(fold_bf16x2(absmax_bf16x2_final(acc))));
  }
  cta_amax_atomic(tam, amax);
}

// a group layout whose starts are not multiples of `blk` rows (or that is not
// monotone, or runs past R_cap) is reported in the error word
__global__ void group_layout_check_kernel(const int32_t* off, int E, int64_t R_cap, int blk, int* err) {
  for (int e = threadIdx.x; e <= E; e += blockDim.x) {
    const int64_t o = off[e];
    const bool bad = (o % blk) != 0 || o > R_cap || (e == 0 && o != 0) || (e > 0 && off[e - 1] > o);
    if (bad) report(err, MGQ_ERR_INVALID_ARG);
  }
}

// ---- delayed scaling ------------------------------------------------------------
// One warp per role: the lanes read the ring coalesced (entry h already
// replaced by this step's amax) and reduce the max with shuffles; fmaxf drops
// NaN entries in any order, so the result equals a serial scan.
__global__ void amax_history_kernel(float* hist, int32_t* head, float* amax, float* scale, int n, int L, float fmax) {
  const int h = *head;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nwarps = blockDim.x >> 5;
  for (int i = warp; i < n; i += nwarps) {
    float* ring = hist + (int64_t)i * L;
    const float a = amax[i];
    float m = 0.0f;
    for (int j = lane; j < L; j += 32) m = fmaxf(m, j == h ? a : ring[j]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
    __syncwarp();
    if (lane == 0) {
      ring[h] = a;
      if (m > 0.0f && isfinite(m)) scale[i] = __fdiv_rn(fmax, m);
      amax[i] = 0.0f;
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) *head = (h + 1) % L;
}

bool dtype_ok(int dt) { return dt == MGQ_E4M3 || dt == MGQ_E5M2; }

int check_q(const mgq_qdesc* q) {
  if (!q || !q->row.data || !aligned16(q->row.data)) return MGQ_ERR_INVALID_ARG;
  if (q->scaling == MGQ_NV16_UE4M3) {
    // e2m1 codes, tiled ue4m3 scales, the amax pre-pass output and s_g
    if (q->dtype != MGQ_E2M1 || !q->row.scale || !aligned16(q->row.scale) || !q->amax_out || !q->tensor_scale)
      return MGQ_ERR_INVALID_ARG;
    if (q->col.data && (!aligned16(q->col.data) || !q->col.scale || !aligned16(q->col.scale)))
      return MGQ_ERR_INVALID_ARG;
    return MGQ_OK;
  }
  if (!dtype_ok(q->dtype)) return MGQ_ERR_UNSUPPORTED;
  if (q->scaling == MGQ_MX32_E8M0 || q->scaling == MGQ_BLK_1x128_F32) {
    if (!q->row.scale || !aligned16(q->row.scale)) return MGQ_ERR_INVALID_ARG;
  } else if (q->scaling == MGQ_TENSOR_F32) {
    if (!q->tensor_scale) return MGQ_ERR_INVALID_ARG;
  } else {
    return MGQ_ERR_UNSUPPORTED;
  }
  if (q->col.data && !aligned16(q->col.data)) return MGQ_ERR_INVALID_ARG;
  if (q->col.data && (q->scaling == MGQ_MX32_E8M0 || q->scaling == MGQ_BLK_1x128_F32) &&
      (!q->col.scale || !aligned16(q->col.scale)))
    return MGQ_ERR_INVALID_ARG;
  return MGQ_OK;
}

}  // namespace

// NVFP4 row-wise quantisation of a bf16 matrix whose amax is already in
// *amax (s_g written to *s_out): the second pass of the fused SwiGLU GEMM
int launch_quant_rows_nv(const uint16_t* x, int64_t rows, const int32_t* rows_used, int64_t K, uint8_t* codes,
                         uint8_t* scales, const float* amax, float* s_out, cudaStream_t s) {
  QuantRowsNvArgs a{x, rows, rows, K, rows_used, codes, scales, amax, s_out};
  quant_rows_nv_kernel<<<(unsigned)((rows + kWarps - 1) / kWarps), 256, 0, s>>>(a);
  MGQ_LAUNCH_CHECK();
  return MGQ_OK;
}

int launch_amax_groups(const uint16_t* x, int64_t per_group, int64_t G, float* amax, cudaStream_t s) {
  if (cudaMemsetAsync(amax, 0, (size_t)G * sizeof(float), s) != cudaSuccess) return MGQ_ERR_CUDA;
  int64_t blocks = (per_group + 256 * 8 * 8 - 1) / (256 * 8 * 8);     // >= 8 loads per thread
  blocks = blocks < 1 ? 1 : (blocks > 2048 ? 2048 : blocks);
  amax_groups_kernel<<<dim3((unsigned)blocks, (unsigned)G), 256, 0, s>>>(x, per_group, amax);
  MGQ_LAUNCH_CHECK();
  return MGQ_OK;
}

}  // namespace mgq

using namespace mgq;

#define MGQ_DISPATCH_Q(q, KERNEL, GRID, ARGS)                                                         \
  do {                                                                                               \
    const int sc_ = (q)->scaling, dt_ = (q)->dtype;                                                  \
    if (sc_ == MGQ_MX32_E8M0 && dt_ == MGQ_E4M3) KERNEL<MGQ_MX32_E8M0, MGQ_E4M3><<<GRID, 256, 0, s>>>(ARGS); \
    else if (sc_ == MGQ_MX32_E8M0 && dt_ == MGQ_E5M2) KERNEL<MGQ_MX32_E8M0, MGQ_E5M2><<<GRID, 256, 0, s>>>(ARGS); \
    else if (sc_ == MGQ_BLK_1x128_F32 && dt_ == MGQ_E4M3) KERNEL<MGQ_BLK_1x128_F32, MGQ_E4M3><<<GRID, 256, 0, s>>>(ARGS); \
    else if (sc_ == MGQ_BLK_1x128_F32 && dt_ == MGQ_E5M2) KERNEL<MGQ_BLK_1x128_F32, MGQ_E5M2><<<GRID, 256, 0, s>>>(ARGS); \
    else if (sc_ == MGQ_TENSOR_F32 && dt_ == MGQ_E4M3) KERNEL<MGQ_TENSOR_F32, MGQ_E4M3><<<GRID, 256, 0, s>>>(ARGS); \
    else if (sc_ == MGQ_TENSOR_F32 && dt_ == MGQ_E5M2) KERNEL<MGQ_TENSOR_F32, MGQ_E5M2><<<GRID, 256, 0, s>>>(ARGS); \
    else return MGQ_ERR_UNSUPPORTED;                                                                  \
    MGQ_LAUNCH_CHECK();                                                                              \
  } while (0)

extern "C" {

int mgq_swiglu_quantize(const void* gu_bf16, int64_t R_cap, int F, const int32_t* offsets, int E,
                        const mgq_qdesc* q, void* h_bf16, void* stream) {
  if (q && q->scaling == MGQ_NV16_UE4M3) {
    // two passes: h (materialised) and its amax, then the quantisation with s_g
    MGQ_CHECK_ARG(q->dtype == MGQ_E2M1 && q->row.data && q->row.scale && q->amax_out && q->tensor_scale);
    MGQ_CHECK_ARG(h_bf16 && aligned16(h_bf16) && gu_bf16 && aligned16(gu_bf16) && offsets && E >= 1);
    MGQ_CHECK_ARG(aligned16(q->row.data) && aligned16(q->row.scale));
    MGQ_CHECK_ARG(F > 0 && F % 128 == 0 && R_cap > 0 && R_cap % 128 == 0);
    if (q->col.data) MGQ_CHECK_ARG(q->col.scale && aligned16(q->col.data) && aligned16(q->col.scale));
    cudaStream_t s = as_stream(stream);
    if (cudaMemsetAsync(q->amax_out, 0, sizeof(float), s) != cudaSuccess) return MGQ_ERR_CUDA;
    const unsigned grid = (unsigned)((R_cap + kWarps - 1) / kWarps);
    swiglu_h_kernel<<<grid, 256, 0, s>>>(static_cast<const uint16_t*>(gu_bf16), offsets + E, F,
                                         static_cast<uint16_t*>(h_bf16), q->amax_out);
    MGQ_LAUNCH_CHECK();
    // row-wise and column-wise copies of h in one tile pass
    if (q->col.data) return rowcol_rows(static_cast<const uint16_t*>(h_bf16), R_cap, offsets + E, F, q, s);
    QuantRowsNvArgs a{static_cast<const uint16_t*>(h_bf16), R_cap, R_cap, F, offsets + E,
                      static_cast<uint8_t*>(q->row.data), static_cast<uint8_t*>(q->row.scale), q->amax_out,
                      q->tensor_scale};
    quant_rows_nv_kernel<<<grid, 256, 0, s>>>(a);
    MGQ_LAUNCH_CHECK();
    return MGQ_OK;
  }
  int rc = check_q(q);
  if (rc != MGQ_OK) return rc;
  MGQ_CHECK_ARG(gu_bf16 && aligned16(gu_bf16) && aligned16(h_bf16) && offsets && E >= 1);
  MGQ_CHECK_ARG(F > 0 && F % 128 == 0 && R_cap > 0 && R_cap % 128 == 0);
  cudaStream_t s = as_stream(stream);
  if (q->col.data)
    return rowcol_swiglu(static_cast<const uint16_t*>(gu_bf16), R_cap, F, offsets + E, static_cast<uint16_t*>(h_bf16),
                         q, s);
  SwigluArgs a{static_cast<const uint16_t*>(gu_bf16), offsets + E, R_cap, F,
               static_cast<uint8_t*>(q->row.data), static_cast<uint8_t*>(q->row.scale),
               static_cast<uint16_t*>(h_bf16), q->tensor_scale, q->amax_out, q->e8m0_mode == MGQ_E8M0_RCEIL};
  const unsigned grid = (unsigned)((R_cap + kWarps - 1) / kWarps);
  MGQ_DISPATCH_Q(q, swiglu_quant_kernel, grid, a);
  return MGQ_OK;
}

int mgq_dswiglu_quantize(const void* dh_bf16, const void* gu_bf16, int64_t R_cap, int F, const int32_t* offsets,
                         int E, const mgq_qdesc* q, void* dgu_bf16, void* stream) {
  int rc = check_q(q);
  if (rc != MGQ_OK) return rc;
  MGQ_CHECK_ARG(dh_bf16 && gu_bf16 && aligned16(dh_bf16) && aligned16(gu_bf16) && aligned16(dgu_bf16));
  MGQ_CHECK_ARG(offsets && E >= 1 && F > 0 && F % 128 == 0 && R_cap > 0 && R_cap % 128 == 0);
  cudaStream_t s = as_stream(stream);
  if (q->scaling == MGQ_NV16_UE4M3) {
    // two passes: [dG | dU] (materialised, dgu_bf16 required) and its amax,
    // then the quantisation with s_g (rows, or rows and columns)
    MGQ_CHECK_ARG(dgu_bf16 != nullptr);
    if (cudaMemsetAsync(q->amax_out, 0, sizeof(float), s) != cudaSuccess) return MGQ_ERR_CUDA;
    const unsigned grid = (unsigned)((R_cap + kWarps - 1) / kWarps);
    dswiglu_dgu_kernel<<<grid, 256, 0, s>>>(static_cast<const uint16_t*>(dh_bf16),
                                            static_cast<const uint16_t*>(gu_bf16), offsets + E, F,
                                            static_cast<uint16_t*>(dgu_bf16), q->amax_out);
    MGQ_LAUNCH_CHECK();
    if (q->col.data) return rowcol_rows(static_cast<const uint16_t*>(dgu_bf16), R_cap, offsets + E, 2 * (int64_t)F, q, s);
    return launch_quant_rows_nv(static_cast<const uint16_t*>(dgu_bf16), R_cap, offsets + E, 2 * (int64_t)F,
                                static_cast<uint8_t*>(q->row.data), static_cast<uint8_t*>(q->row.scale), q->amax_out,
                                q->tensor_scale, s);
  }
  if (q->col.data)
    return rowcol_dswiglu(static_cast<const uint16_t*>(dh_bf16), static_cast<const uint16_t*>(gu_bf16), R_cap, F,
                          offsets + E, static_cast<uint16_t*>(dgu_bf16), q, s);
  DswigluArgs a{static_cast<const uint16_t*>(dh_bf16), static_cast<const uint16_t*>(gu_bf16), offsets + E, R_cap, F,
                static_cast<uint8_t*>(q->row.data), static_cast<uint8_t*>(q->row.scale),
                static_cast<uint16_t*>(dgu_bf16), q->tensor_scale, q->amax_out, q->e8m0_mode == MGQ_E8M0_RCEIL};
  const unsigned grid = (unsigned)((R_cap + kWarps - 1) / kWarps);
  MGQ_DISPATCH_Q(q, dswiglu_quant_kernel, grid, a);
  return MGQ_OK;
}

int mgq_moe_unpermute(const void* y_bf16, const int32_t* row_id_map, const float* probs, int T, int k, int H,
                      void* out_bf16, void* stream) {
  MGQ_CHECK_ARG(T >= 0 && k >= 1 && k <= 8 && H > 0 && H % 8 == 0);
  MGQ_CHECK_ARG(T == 0 || (y_bf16 && row_id_map && probs && out_bf16));
  MGQ_CHECK_ARG(aligned16(y_bf16) && aligned16(out_bf16));
  if (T == 0) return MGQ_OK;
  (k <= 2 ? combine_kernel<2> : combine_kernel<8>)<<<combine_grid(T, k), 256, 0, as_stream(stream)>>>(
      static_cast<const uint16_t*>(y_bf16), row_id_map, probs, T, k, H, static_cast<uint16_t*>(out_bf16));
  MGQ_LAUNCH_CHECK();
  return MGQ_OK;
}

int mgq_moe_permute_bwd(const void* da_bf16, const int32_t* row_id_map, int T, int k, int H, void* dx_bf16,
                        void* stream) {
  MGQ_CHECK_ARG(T >= 0 && k >= 1 && k <= 8 && H > 0 && H % 8 == 0);
  MGQ_CHECK_ARG(T == 0 || (da_bf16 && row_id_map && dx_bf16));
  MGQ_CHECK_ARG(aligned16(da_bf16) && aligned16(dx_bf16));
  if (T == 0) return MGQ_OK;
  (k <= 2 ? combine_kernel<2> : combine_kernel<8>)<<<combine_grid(T, k), 256, 0, as_stream(stream)>>>(
      static_cast<const uint16_t*>(da_bf16), row_id_map, nullptr, T, k, H, static_cast<uint16_t*>(dx_bf16));
  MGQ_LAUNCH_CHECK();
  return MGQ_OK;
}

int mgq_moe_unpermute_bwd(const void* dout_bf16, const void* y_bf16, const int32_t* row_id_map,
                          const int32_t* src_row, const float* probs, int T, int k, int H, int64_t R_cap,
                          const int32_t* offsets, int E, const mgq_qdesc* q, float* dprobs, void* stream) {
  int rc = check_q(q);
  if (rc != MGQ_OK) return rc;
  MGQ_CHECK_ARG(T >= 0 && k >= 1 && k <= 8 && H > 0 && H % 128 == 0 && E >= 1 && offsets && src_row);
  MGQ_CHECK_ARG(T == 0 || (dout_bf16 && y_bf16 && row_id_map && probs && dprobs));   // no entries: may be null
  MGQ_CHECK_ARG(aligned16(dout_bf16) && aligned16(y_bf16) && R_cap > 0 && R_cap % 128 == 0);
  cudaStream_t s = as_stream(stream);
  const bool nv = q->scaling == MGQ_NV16_UE4M3;
  if (nv) {
    if (T > 0) {
      if (cudaMemsetAsync(q->amax_out, 0, sizeof(float), s) != cudaSuccess) return MGQ_ERR_CUDA;
      const int blocks = (int)std::min<int64_t>((T + kWarps - 1) / kWarps, (int64_t)num_sms() * 4);
      dy_amax_kernel<<<blocks, 256, 0, s>>>(static_cast<const uint16_t*>(dout_bf16), probs, row_id_map, T, k, H,
                                            q->amax_out);
      MGQ_LAUNCH_CHECK();
    } else if (cudaMemsetAsync(q->amax_out, 0, sizeof(float), s) != cudaSuccess) {
      return MGQ_ERR_CUDA;
    }
  }
  UnpermBwdArgs a;
  a.dout = static_cast<const uint16_t*>(dout_bf16);
  a.y = static_cast<const uint16_t*>(y_bf16);
  a.rim = row_id_map;
  a.src_row = src_row;
  a.probs = probs;
  a.offsets = offsets;
  a.T = T; a.k = k; a.H = H; a.E = E;
  a.R_cap = R_cap;
  a.codes = static_cast<uint8_t*>(q->row.data);
  a.scales = static_cast<uint8_t*>(q->row.scale);
  a.tensor_scale = q->tensor_scale;
  a.amax_out = q->amax_out;
  a.s_out = q->tensor_scale;
  a.dprobs = dprobs;
  a.rceil = q->e8m0_mode == MGQ_E8M0_RCEIL;
  // entry CTAs: at most a few resident waves (they stride over the entries)
  a.token_blocks = (int)std::min<int64_t>(((int64_t)T * k + kWarps - 1) / kWarps,
                                          (int64_t)num_sms() * (q->scaling == MGQ_TENSOR_F32 ? 3 : 2));
  const unsigned grid = (unsigned)(a.token_blocks + E);
  if (q->col.data && q->scaling != MGQ_TENSOR_F32 && q->scaling != MGQ_MX32_E8M0 &&
      q->scaling != MGQ_BLK_1x128_F32 && !nv)
    return MGQ_ERR_UNSUPPORTED;
  if (nv) {
    unpermute_bwd_kernel<MGQ_NV16_UE4M3, MGQ_E2M1><<<grid, 256, 0, s>>>(a);
    MGQ_LAUNCH_CHECK();
  } else {
    MGQ_DISPATCH_Q(q, unpermute_bwd_kernel, grid, a);
  }
  if (q->col.data && q->scaling == MGQ_TENSOR_F32)
    return launch_transpose_u8(static_cast<const uint8_t*>(q->row.data), H, static_cast<uint8_t*>(q->col.data),
                               R_cap, offsets + E, R_cap, H, s);
  if (q->col.data)
    return col_gather_dy(static_cast<const uint16_t*>(dout_bf16), probs, src_row, k, H, R_cap, offsets + E, q, s);
  return MGQ_OK;
}

int mgq_block_quantize(const void* x_bf16, int64_t G, int64_t M, int64_t K, const mgq_qdesc* q, void* stream) {
  if (q && q->scaling == MGQ_NV16_UE4M3) {
    MGQ_CHECK_ARG(q->dtype == MGQ_E2M1 && q->row.data && q->row.scale && q->amax_out && q->tensor_scale);
    MGQ_CHECK_ARG(aligned16(q->row.data) && aligned16(q->row.scale) && x_bf16 && aligned16(x_bf16));
    MGQ_CHECK_ARG(G >= 1 && M > 0 && K > 0 && M % 128 == 0 && K % 128 == 0);
    if (q->col.data) MGQ_CHECK_ARG(q->col.scale && aligned16(q->col.data) && aligned16(q->col.scale));
    cudaStream_t s = as_stream(stream);
    int rc = launch_amax_groups(static_cast<const uint16_t*>(x_bf16), M * K, G, q->amax_out, s);
    if (rc != MGQ_OK) return rc;
    // 1x16 blocks both ways: rows along K, columns along each group's M rows
    if (q->col.data) return rowcol_plain(static_cast<const uint16_t*>(x_bf16), G, M, K, q, s);
    QuantRowsNvArgs a{static_cast<const uint16_t*>(x_bf16), G * M, M, K, nullptr,
                      static_cast<uint8_t*>(q->row.data), static_cast<uint8_t*>(q->row.scale), q->amax_out,
                      q->tensor_scale};
    quant_rows_nv_kernel<<<(unsigned)((G * M + kWarps - 1) / kWarps), 256, 0, s>>>(a);
    MGQ_LAUNCH_CHECK();
    return MGQ_OK;
  }
  if (q && q->scaling == MGQ_NV16x16_UE4M3) {
    MGQ_CHECK_ARG(q->dtype == MGQ_E2M1 && q->row.data && q->row.scale && q->amax_out && q->tensor_scale);
    MGQ_CHECK_ARG(aligned16(q->row.data) && aligned16(q->row.scale) && x_bf16 && aligned16(x_bf16));
    MGQ_CHECK_ARG(!q->col.data || (q->col.scale && aligned16(q->col.data) && aligned16(q->col.scale)));
    MGQ_CHECK_ARG(G >= 1 && M > 0 && K > 0 && M % 128 == 0 && K % 128 == 0);
    cudaStream_t s = as_stream(stream);
    int rc = launch_amax_groups(static_cast<const uint16_t*>(x_bf16), M * K, G, q->amax_out, s);
    if (rc != MGQ_OK) return rc;
    return quant_nv2d(static_cast<const uint16_t*>(x_bf16), G, M, K, static_cast<uint8_t*>(q->row.data),
                      static_cast<uint8_t*>(q->row.scale), static_cast<uint8_t*>(q->col.data),
                      static_cast<uint8_t*>(q->col.scale), q->amax_out, q->tensor_scale, s);
  }
  if (q && q->scaling == MGQ_BLK_128x128_F32) {
    MGQ_CHECK_ARG(q->row.data && q->row.scale && aligned16(q->row.data) && x_bf16 && aligned16(x_bf16));
    MGQ_CHECK_ARG(G >= 1 && M > 0 && K > 0 && M % 128 == 0 && K % 128 == 0);
    if (q->col.data) {
      // both copies in one tile pass: the column-wise copy holds the
      // transposed codes and the transposed tile scales
      MGQ_CHECK_ARG(aligned16(q->col.data) && q->col.scale);
      if (q->dtype != MGQ_E4M3 && q->dtype != MGQ_E5M2) return MGQ_ERR_UNSUPPORTED;
      return rowcol_plain(static_cast<const uint16_t*>(x_bf16), G, M, K, q, as_stream(stream));
    }
    const unsigned grid = (unsigned)(G * (M / 128) * (K / 128));
    cudaStream_t s = as_stream(stream);
    if (q->dtype == MGQ_E4M3)
      quant_tile128_kernel<MGQ_E4M3><<<grid, 256, 0, s>>>(static_cast<const uint16_t*>(x_bf16), M, K,
                                                          static_cast<uint8_t*>(q->row.data),
                                                          static_cast<float*>(q->row.scale));
    else if (q->dtype == MGQ_E5M2)
      quant_tile128_kernel<MGQ_E5M2><<<grid, 256, 0, s>>>(static_cast<const uint16_t*>(x_bf16), M, K,
                                                          static_cast<uint8_t*>(q->row.data),
                                                          static_cast<float*>(q->row.scale));
    else
      return MGQ_ERR_UNSUPPORTED;
    MGQ_LAUNCH_CHECK();
    return MGQ_OK;
  }
  int rc = check_q(q);
  if (rc != MGQ_OK) return rc;
  MGQ_CHECK_ARG(x_bf16 && aligned16(x_bf16) && G >= 1 && M > 0 && K > 0 && M % 128 == 0 && K % 128 == 0);
  cudaStream_t s = as_stream(stream);
  if (q->col.data) return rowcol_plain(static_cast<const uint16_t*>(x_bf16), G, M, K, q, s);
  QuantRowsArgs a{static_cast<const uint16_t*>(x_bf16), G * M, M, K, static_cast<uint8_t*>(q->row.data),
                  static_cast<uint8_t*>(q->row.scale), q->tensor_scale, q->amax_out,
                  q->e8m0_mode == MGQ_E8M0_RCEIL};
  const unsigned grid = (unsigned)((G * M + kWarps - 1) / kWarps);
  MGQ_DISPATCH_Q(q, quant_rows_kernel, grid, a);
  return MGQ_OK;
}

int mgq_grouped_quantize(const void* x_bf16, int64_t R_cap, int64_t C, const int32_t* offsets, int E,
                         const mgq_qdesc* q, void* stream) {
  int rc = check_q(q);
  if (rc != MGQ_OK) return rc;
  MGQ_CHECK_ARG(x_bf16 && aligned16(x_bf16) && offsets && E >= 1 && E <= 1024);
  MGQ_CHECK_ARG(C > 0 && C % 128 == 0 && R_cap > 0 && R_cap % 128 == 0 && R_cap < (1ll << 31));
  const int sc = q->scaling;
  if (sc != MGQ_MX32_E8M0 && sc != MGQ_TENSOR_F32 && sc != MGQ_NV16_UE4M3 && sc != MGQ_BLK_1x128_F32)
    return MGQ_ERR_UNSUPPORTED;
  int* err = error_word();
  if (!err) return MGQ_ERR_CUDA;
  cudaStream_t s = as_stream(stream);
  // column blocks run inside the groups: group starts on block boundaries
  const int blk = sc == MGQ_MX32_E8M0 ? 32 : (sc == MGQ_NV16_UE4M3 ? 16 : (sc == MGQ_BLK_1x128_F32 ? 128 : 1));
  group_layout_check_kernel<<<1, 256, 0, s>>>(offsets, E, R_cap, blk, err);
  MGQ_LAUNCH_CHECK();
  if (sc == MGQ_NV16_UE4M3) {   // s_g needs the amax of the rows in use first
    if (cudaMemsetAsync(q->amax_out, 0, sizeof(float), s) != cudaSuccess) return MGQ_ERR_CUDA;
    const int blocks = (int)std::min<int64_t>((R_cap + kWarps - 1) / kWarps, (int64_t)num_sms() * 4);
    amax_rows_kernel<<<blocks, 256, 0, s>>>(static_cast<const uint16_t*>(x_bf16), offsets + E, C, q->amax_out);
    MGQ_LAUNCH_CHECK();
  }
  // one tile pass over the rows in use: the groups are whole column blocks, so
  // treating the matrix as one group gives every group's own column blocks
  return rowcol_rows(static_cast<const uint16_t*>(x_bf16), R_cap, offsets + E, C, q, s);
}

int mgq_amax_history_update(float* history, int32_t* head, float* amax, float* scale, int n, int L, float fmax,
                            void* stream) {
  MGQ_CHECK_ARG(history && head && amax && scale && n >= 1 && L >= 1 && fmax > 0.0f);
  amax_history_kernel<<<1, 1024, 0, as_stream(stream)>>>(history, head, amax, scale, n, L, fmax);
  MGQ_LAUNCH_CHECK();
  return MGQ_OK;
}

}  // extern "C"
