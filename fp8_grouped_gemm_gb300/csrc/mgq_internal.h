// Host-side internals shared by the translation units of libmgq.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "mgq.h"

namespace mgq {

// Device address of the current device's error word (cached per device).
// Returns nullptr if it cannot be resolved.
int* error_word();

// Encodes a 2D row-major tiled tensor map of unsigned bytes: `inner` bytes per
// row (contiguous), `outer` rows with a pitch of `pitch` bytes; the box is
// box_inner x box_outer with 128-byte swizzling (box_inner == 128).
bool encode_tmap_u8_2d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer, uint64_t pitch,
                       uint32_t box_inner, uint32_t box_outer);

// 2D row-major tensor map of 8-, 16- or 32-bit elements (elem_bytes 1, 2 or 4):
// `inner` elements per row, `outer` rows, pitch bytes; no swizzle, or with
// sw128 the 128-byte swizzle (box_inner * elem_bytes == 128).
bool encode_tmap_2d(CUtensorMap* map, const void* base, int elem_bytes, uint64_t inner, uint64_t outer,
                    uint64_t pitch, uint32_t box_inner, uint32_t box_outer, bool sw128 = false);

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }

// Number of SMs of the current device (cached).
int num_sms();

// dst[c, r] = src[r, c] for r < *rows_used (or rows_cap when rows_used is
// null), c < cols; 64x64 byte tiles (routing.cu).
int launch_transpose_u8(const uint8_t* src, int64_t src_ld, uint8_t* dst, int64_t dst_ld, const int32_t* rows_used,
                        int64_t rows_cap, int64_t cols, cudaStream_t s);

// amax[g] = max |x| over each of G groups of per_group bf16 values (zeroes
// amax first; elementwise.cu).
int launch_amax_groups(const uint16_t* x, int64_t per_group, int64_t G, float* amax, cudaStream_t s);
// NVFP4 row-wise codes of x [rows, K] (rows_used on the device, or null) with
// s_g = 2688 / *amax, written to *s_out
int launch_quant_rows_nv(const uint16_t* x, int64_t rows, const int32_t* rows_used, int64_t K, uint8_t* codes,
                         uint8_t* scales, const float* amax, float* s_out, cudaStream_t s);

// Row-wise + column-wise quantisation in one pass (quant_tile.cu); q->col.data
// must be set. Per-tensor or MX scaling.
int rowcol_plain(const uint16_t* x, int64_t G, int64_t M, int64_t K, const mgq_qdesc* q, cudaStream_t s);
// row-wise and column-wise copies of a bf16 [rows_cap, C] matrix whose rows in
// use are *rows_used (one group: column copy [C, rows_cap]) (quant_tile.cu)
int rowcol_rows(const uint16_t* x, int64_t rows_cap, const int32_t* rows_used, int64_t C, const mgq_qdesc* q,
                cudaStream_t s);
int rowcol_swiglu(const uint16_t* gu, int64_t R_cap, int64_t F, const int32_t* rows_used, uint16_t* h_out,
                  const mgq_qdesc* q, cudaStream_t s);
int rowcol_dswiglu(const uint16_t* dh, const uint16_t* gu, int64_t R_cap, int64_t F, const int32_t* rows_used,
                   uint16_t* out, const mgq_qdesc* q, cudaStream_t s);

// Column-wise copies (MX or per-tensor) of the permuted X rows, with the
// row-wise codes too when `with_rows`, and column-wise copies only of
// dY = probs * dout rows, gathered through src_row (quant_tile.cu).
int gather_x_rowcol(const uint16_t* x, const int32_t* src_row, int k, int64_t H, int64_t R_cap,
                    const int32_t* rows_used, bool with_rows, const mgq_qdesc* q, cudaStream_t s);
int col_gather_dy(const uint16_t* dout, const float* probs, const int32_t* src_row, int k, int64_t H,
                  int64_t R_cap, const int32_t* rows_used, const mgq_qdesc* q, cudaStream_t s);

// NVFP4 weights with 16x16 blocks: row-wise [G*M, K/2] and (when col_codes
// is set) column-wise [G*K, M/2] codes with tiled ue4m3 scales; s_g per group
// from amax (written to s_out) (quant_tile.cu)
int quant_nv2d(const uint16_t* x, int64_t G, int64_t M, int64_t K, uint8_t* row_codes, uint8_t* row_scales,
               uint8_t* col_codes, uint8_t* col_scales, const float* amax, float* s_out, cudaStream_t s);

}  // namespace mgq

#define MGQ_CHECK_ARG(cond)                 \
  do {                                      \
    if (!(cond)) return MGQ_ERR_INVALID_ARG; \
  } while (0)

#define MGQ_LAUNCH_CHECK()                           \
  do {                                               \
    if (cudaPeekAtLastError() != cudaSuccess) {      \
      (void)cudaGetLastError();                      \
      return MGQ_ERR_CUDA;                           \
    }                                                \
  } while (0)
