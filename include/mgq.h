/*
 * mgq.h — C ABI of the GB300 (sm_103a) low-precision MoE routed-expert layer.
 *
 * One GPU, stream-ordered, stateless. The caller owns every buffer: the
 * library never allocates device memory (the only device-resident state is a
 * per-device error word read by mgq_get_error). Pointers marked "device" must
 * be device (or managed) memory of the current device; "host" pointers are
 * read during the call only. `stream` is a cudaStream_t (NULL = legacy
 * default stream). Every call returns an mgq_status synchronously:
 * argument errors are detected on the host before anything is launched;
 * errors found by a kernel (an expert id out of range, a pipeline wait that
 * timed out) are recorded in the device error word and reported by
 * mgq_get_error. No call traps, aborts or throws. The error word's device
 * address is looked up once per device and kept for the life of the process,
 * so using the library after cudaDeviceReset in the same process is not
 * supported.
 *
 * What the operations compute comes from four pages on low-precision MoE
 * training:
 *  [MOE-FP8]  "[BUG] Loss difference when training with FP8 vs. BF16 MoE"
 *             (Megatron-LM issue #1152): grouped GEMM over experts
 *             (--moe-grouped-gemm, TEGroupedMLP), padding of expert inputs
 *             for FP8, the hybrid format (e4m3 forward, e5m2 gradients) and
 *             delayed scaling with a 1024-long amax history reduced by max.
 *  [GROUPED]  "Numerical fix for moe single grouped weight with fp8 fp4
 *             primary weight and grad norm spikes" (Megatron-LM PR #5487):
 *             the MXFP8 and NVFP4 recipes, one contiguous grouped weight for
 *             all experts, row-wise and column-wise data + scales, gradient
 *             accumulation fusion, e2m1 packed two per byte.
 *  [BLOCK]    "FP8BlockQuantizer not work on TE" (TransformerEngine issue
 *             #2393): 1x128 forward / 128x1 backward block scaling, the
 *             transpose identity colwise(x) = transpose(rowwise(x^T)), zero
 *             fill of partial blocks, block-aligned shapes as a hard error.
 *  [AO-MOE]   "float8 moe training conversion API prototype" (pytorch/ao PR
 *             #2275): dynamic quantisation followed by a scaled grouped mm;
 *             SQNR of outputs and gradients against bf16.
 * Number formats follow OCP OFP8 (e4m3, e5m2) and OCP MX v1.0 (e2m1, E8M0).
 *
 * Notation: T tokens, k experts per token, E experts, H hidden, F ffn.
 * R_cap = capacity (rows) of permuted buffers; the rows in use are
 * [0, offsets[E]), a device value, so no call needs a host sync.
 *
 * Quantised storage (codes: 1 byte per element, e2m1: 2 elements per byte,
 * element 2i in the low nibble). For a row-major matrix with `rows` rows and
 * row pitch `ld` elements (the contraction dimension K):
 *  MGQ_MX32_E8M0     E8M0 scale per 32 consecutive elements of a row, stored
 *                    in 128x4 tiles: byte of (row r, block b) at
 *                      ((r/128)*(ld/128) + b/4)*512 + (r%32)*16 + ((r/32)%4)*4 + b%4
 *                    (ld a multiple of 128; rows padded to 128).
 *  MGQ_NV16_UE4M3    ue4m3 scale per 16 elements, same tiling with b the
 *                    16-element block (ld a multiple of 64 elements);
 *                    plus one float32 global scale s_g per tensor (weights:
 *                    per expert) in tensor_scale; value = e2m1 * sc / s_g.
 *  MGQ_NV16x16_UE4M3 weights only (mgq_block_quantize): one ue4m3 scale per
 *                    16x16 block of each group's [M, K], by the NVFP4 rule
 *                    on the block's amax; written as MGQ_NV16_UE4M3 row-wise
 *                    and column-wise copies whose 1x16 blocks carry their
 *                    16x16 block's scale, so both copies hold the same
 *                    element codes, transposed. Reading of [GROUPED]'s NVFP4
 *                    primary-weight path (one grouped weight with row-wise
 *                    and column-wise data); the page fixes no block shape.
 *  MGQ_BLK_1x128_F32 float32 scale_inv per 128 elements of a row, stored
 *                    k-block major: scale_inv[b * rows_cap + r].
 *  MGQ_BLK_128x128_F32 float32 scale_inv per 128x128 tile of each expert's
 *                    weight: scale_inv[(g * (N/128) + n/128) * (K/128) + k/128].
 *  MGQ_TENSOR_F32    one float32 scale s per tensor (weights: per expert),
 *                    code = cast(x * s), value = code / s.
 * Column-wise ("col") copies hold the transposed matrix quantised with its
 * own blocks along the old row dimension (transpose identity of [BLOCK]).
 */
#ifndef MGQ_H
#define MGQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MGQ_OK = 0,
  MGQ_ERR_INVALID_ARG = 1,   /* bad pointer, size, alignment or combination */
  MGQ_ERR_UNSUPPORTED = 2,   /* valid but not implemented (format / mode)   */
  MGQ_ERR_CUDA = 3,          /* a CUDA runtime or driver call failed        */
  MGQ_ERR_TIMEOUT = 4,       /* device: a pipeline wait gave up             */
  MGQ_ERR_DEVICE_INDEX = 5   /* device: an expert index out of range        */
} mgq_status;

typedef enum { MGQ_E4M3 = 0, MGQ_E5M2 = 1, MGQ_E2M1 = 2 } mgq_dtype;

typedef enum {
  MGQ_MX32_E8M0 = 0,
  MGQ_NV16_UE4M3 = 1,
  MGQ_BLK_1x128_F32 = 2,
  MGQ_BLK_128x128_F32 = 3,
  MGQ_TENSOR_F32 = 4,
  MGQ_NV16x16_UE4M3 = 5
} mgq_scaling;

/* Exponent of an E8M0 block scale. RCEIL: the smallest power of two that
 * keeps the block amax at or below the format's largest value (no element
 * saturates). FLOOR: floor(log2 amax) - emax (OCP MX v1.0). */
typedef enum { MGQ_E8M0_RCEIL = 0, MGQ_E8M0_FLOOR = 1 } mgq_e8m0_mode;

typedef enum { MGQ_OUT_BF16 = 0, MGQ_OUT_F32 = 1 } mgq_out_dtype;

/* Quantised output buffers of one layout (device pointers). */
typedef struct {
  void* data;     /* codes                                  */
  void* scale;    /* block scales (NULL for MGQ_TENSOR_F32) */
} mgq_qbuf;

/* How to quantise, and where to. */
typedef struct {
  int dtype;                 /* mgq_dtype                                       */
  int scaling;               /* mgq_scaling                                     */
  int e8m0_mode;             /* mgq_e8m0_mode (MX only)                         */
  mgq_qbuf row;              /* row-wise output; row.data required              */
  mgq_qbuf col;              /* column-wise (transposed) output; col.data NULL = none */
  float* tensor_scale;       /* device, per group: MGQ_TENSOR_F32: the scale s to
                                apply (read); MGQ_NV16_UE4M3: receives s_g
                                = 2688 / amax (written)                        */
  float* amax_out;           /* device, per group: max |x| (MGQ_TENSOR_F32:
                                optional, atomically raised; MGQ_NV16_UE4M3:
                                required, computed by the call)                 */
} mgq_qdesc;

/* Which dimension of a GEMM operand is contiguous in memory. */
typedef enum {
  MGQ_LAYOUT_K = 0,          /* rows are the operand's M (or N) index, the
                                contraction index runs along each row          */
  MGQ_LAYOUT_MN = 1          /* rows are the contraction index (the transposed
                                storage); per-tensor FP8 dgrad / wgrad only     */
} mgq_layout;

/* A quantised GEMM operand (device pointers). */
typedef struct {
  const void* data;          /* codes, row-major, row pitch `ld` elements      */
  const void* scale;         /* block scales, or device float s per tensor/group */
  int64_t ld;                /* row pitch in elements                          */
  int dtype;                 /* mgq_dtype                                       */
  const float* global_scale; /* NVFP4: device s_g per tensor (A) / per expert (W); else NULL */
  int layout;                /* mgq_layout; 0 (MGQ_LAYOUT_K) unless stated      */
  const void* scale_image;   /* NVFP4 second operand (W, Wcol, Acol) only: the
                                image of `scale` from mgq_nv_scale_image, or
                                NULL (the GEMM then reads `scale` alone)       */
} mgq_operand;

/* ---- status --------------------------------------------------------------- */

const char* mgq_status_string(int status);
/* The interface version: 2 since mgq_operand gained scale_image (callers
 * built against version 1 pass the shorter struct and must be rebuilt). */
#define MGQ_VERSION 2
int mgq_version(void);

/* Reads and clears the device error word of the current device after
 * synchronising `stream`. *device_status receives MGQ_OK or the first device
 * error recorded since the last call. */
int mgq_get_error(void* stream, int* device_status);

/* ---- a2: permute + quantise (dispatch) -------------------------------------
 * [MOE-FP8] grouped GEMM over experts with padded expert inputs; [AO-MOE]
 * dynamic quantisation before the scaled grouped mm; [BLOCK] padding to the
 * block is required.
 *
 * Routes T tokens to experts and writes each token's row to its k expert
 * groups. Group e occupies rows [offsets[e], offsets[e]+counts[e]) in token
 * order (stable), padded with zero rows (codes 0, scales 0) up to a multiple
 * of `align`: offsets[e+1] = offsets[e] + roundup(counts[e], align).
 *  x_bf16      device [T, H] bf16
 *  topk_idx    device [T, k] int32, distinct experts per token in [0, E)
 *              (out of range: the entry is skipped, MGQ_ERR_DEVICE_INDEX set)
 *  q           quantisation of the permuted rows (row: [R_cap, H]; col:
 *              [H, R_cap], MX / NVFP4 / blockwise 128x1 blocks along the rows
 *              of each group (blockwise: align a multiple of 128, scale_inv
 *              [R_cap/128][H]), per-tensor the transposed row codes; e2m1:
 *              [R_cap, H/2] and [H, R_cap/2] bytes, s_g from an amax
 *              pre-pass); NULL = no quantised output
 *  out_bf16    device [R_cap, H] bf16 permuted copy, or NULL
 *  row_id_map  device [T, k] int32: destination row of (t, j)
 *  src_row     device [R_cap] int32: t*k + j of the row, -1 for padding
 *  offsets     device [E+1] int32; counts device [E] int32
 *  workspace   device scratch of mgq_permute_workspace_size() bytes
 * Requires: align a multiple of 128 when a GEMM consumes the result (32 is
 * accepted for quantise-only use), H a multiple of 128,
 * R_cap >= T*k + E*(align-1) rounded up to 128. */
size_t mgq_permute_workspace_size(int T, int k, int E);
int mgq_moe_permute(const void* x_bf16, int T, int H, const int32_t* topk_idx, int k,
                    int E, int align, const mgq_qdesc* q, void* out_bf16, int64_t R_cap,
                    int32_t* row_id_map, int32_t* src_row, int32_t* offsets,
                    int32_t* counts, void* workspace, size_t ws_bytes, void* stream);

/* ---- the two halves of mgq_moe_permute -------------------------------------
 * mgq_moe_route does the routing alone: it writes row_id_map, src_row,
 * offsets and counts exactly as mgq_moe_permute does (same arguments and
 * requirements, no x and no quantisation).
 * mgq_moe_permute_routed then does the permute + quantise on those final
 * routing arrays (read only): the codes and scales equal those of
 * mgq_moe_permute with the same routing. It requires the arrays from
 * mgq_moe_route (or mgq_moe_permute) for this T, k, E, and, for a column-wise
 * copy, an `align` that was a multiple of the column block (MX and NVFP4 32,
 * blockwise 128).
 * Splitting lets a caller route once and permute several tensors, or run the
 * routing (index work, latency-bound) beside other work. */
int mgq_moe_route(const int32_t* topk_idx, int T, int k, int E, int align, int64_t R_cap,
                  int32_t* row_id_map, int32_t* src_row, int32_t* offsets, int32_t* counts,
                  void* workspace, size_t ws_bytes, void* stream);
int mgq_moe_permute_routed(const void* x_bf16, int T, int H, int k, int E, const mgq_qdesc* q,
                           void* out_bf16, int64_t R_cap, const int32_t* row_id_map,
                           const int32_t* src_row, const int32_t* offsets,
                           const int32_t* counts, void* stream);

/* ---- permute + quantise without a workspace --------------------------------
 * The pages have no counterpart of this call: it exists for callers that
 * cannot allocate device memory, such as a plugin whose host framework owns
 * every device allocation and passes it only inputs and outputs, or a runtime
 * that forbids allocation while it runs. It computes exactly what
 * mgq_moe_permute computes (same arguments, same results) but takes the
 * routing scratch from a fixed 1 MiB device array inside the library instead
 * of a caller workspace; it allocates nothing.
 *  - Limit: mgq_permute_workspace_size(T, k, E) must not exceed 1048576 bytes
 *    (ceil(T*k/1024) * E <= 262144), else MGQ_ERR_INVALID_ARG, nothing launched.
 *  - The first call on a device looks up the array's device address (with
 *    that device current) and caches it; make that first call before any
 *    stream capture.
 *  - All calls share the one array: calls whose kernels can overlap on the
 *    GPU (different streams or host threads) race and must be serialised by
 *    the caller. Every scratch entry is written before it is read, so the
 *    previous call's contents need no clearing.
 *  - Every GPU that loads the library holds the array until the process exits.
 *  - The looked-up address is kept for the life of the process: calling this
 *    entry point after cudaDeviceReset in the same process is not supported. */
int mgq_moe_permute_noalloc(const void* x_bf16, int T, int H, const int32_t* topk_idx, int k,
                            int E, int align, const mgq_qdesc* q, void* out_bf16, int64_t R_cap,
                            int32_t* row_id_map, int32_t* src_row, int32_t* offsets,
                            int32_t* counts, void* stream);

/* ---- a3/a4: block quantise, row-wise and column-wise -----------------------
 * [BLOCK] 1x128 forward / 128x1 backward with the transpose identity;
 * [GROUPED] row-wise and column-wise data and scales of one grouped weight.
 *  x_bf16  device [G, M, K] bf16 (G groups, e.g. experts)
 *  q->row  [G, M, K] codes (+ scales); q->col [G, K, M] codes (+ scales)
 *  per-tensor mode reads one scale per group from q->tensor_scale.
 *  blockwise: MGQ_BLK_1x128_F32 row-wise scale_inv [K/128][G*M] and, with
 *    q->col, 128x1 column blocks (the transpose identity: the 1x128
 *    quantisation of each group's transpose) with scale_inv [M/128][G*K];
 *    MGQ_BLK_128x128_F32 (weights) one scale per 128x128 tile, row-wise
 *    scale_inv [G][M/128][K/128] and, with q->col, the transposed codes with
 *    the transposed tile scales [G][K/128][M/128] from the same pass.
 *  NVFP4 (MGQ_NV16_UE4M3, row-wise only; MGQ_NV16x16_UE4M3, row-wise and
 *    optionally column-wise, dtype MGQ_E2M1): an amax pre-pass writes each
 *    group's amax to q->amax_out [G] and s_g = 6*448/amax to
 *    q->tensor_scale [G]; codes [G, M, K/2] / [G, K, M/2] bytes. (Every
 *    NVFP4 call writes s_g with the first row it quantises: with no rows in
 *    use it writes the amax, 0, and leaves q->tensor_scale as it was.)
 * Requires M and K multiples of 128. */
int mgq_block_quantize(const void* x_bf16, int64_t G, int64_t M, int64_t K,
                       const mgq_qdesc* q, void* stream);

/* Row-wise and column-wise quantisation of a bf16 matrix over ragged groups
 * ([GROUPED]'s grouped tensor with row-wise and column-wise data; [BLOCK]'s
 * 128x1 backward blocks inside each group): x_bf16 device [R_cap, C]; rows
 * [0, offsets[E]) are in use, group e = rows [offsets[e], offsets[e+1]).
 *  q->row  [R_cap, C] codes (+ scales over [R_cap, C]) for the rows in use
 *  q->col  [C, R_cap] codes (+ scales over [C, R_cap]) or NULL; column blocks
 *          (MX 32, NVFP4 16, blockwise 128 rows) run inside each group
 * scaling: MGQ_TENSOR_F32 (q->tensor_scale[0]; the column copy is the
 * transposed cast; q->amax_out optional), MGQ_MX32_E8M0, MGQ_BLK_1x128_F32
 * (row-wise scale_inv [C/128][R_cap], column-wise [R_cap/128][C]), or
 * MGQ_NV16_UE4M3 (an amax pre-pass over the rows in use into q->amax_out[0],
 * s_g into q->tensor_scale[0]; e2m1 codes [R_cap, C/2] / [C, R_cap/2] bytes).
 * Group starts must be multiples of the column block (MX 32, NVFP4 16,
 * blockwise 128): a
 * layout that is not (or not monotone, or past R_cap) is reported as
 * MGQ_ERR_INVALID_ARG in the device error word, and the codes are then
 * unspecified. Requires C and R_cap multiples of 128, E <= 1024. */
int mgq_grouped_quantize(const void* x_bf16, int64_t R_cap, int64_t C, const int32_t* offsets,
                         int E, const mgq_qdesc* q, void* stream);

/* ---- a5/a9/a11: grouped GEMMs ------------------------------------------------
 * [MOE-FP8] one grouped GEMM for all experts; [AO-MOE] scaled grouped mm;
 * [GROUPED] single grouped weight [E, N, K], gradient accumulation fusion.
 * tcgen05 block-scaled MMA with float32 accumulation in tensor memory.
 *
 * fwd:   Y[r, :]  = sum_k A[r, k] W_e[:, k]  for rows r of group e
 *        A [R_cap, K] (ld >= K), W [E, N, K], Y [R_cap, N] (out_dtype)
 * dgrad: dA[r, :] = sum_n dY[r, n] W_e[n, :]: pass dY [R_cap, N] and the
 *        column-wise weight copy Wcol [E, K, N]; dA [R_cap, K]
 * wgrad: dW_e = beta * dW_e + sum_{r in e} dY[r, :]^T A[r, :]: pass the
 *        column-wise copies dYcol [N, R_cap] and Acol [K, R_cap];
 *        dW [E, N, K] (out_dtype); an empty group gives zeros (beta 0) or
 *        leaves dW_e unchanged (beta 1).
 * scaling: MGQ_MX32_E8M0 (e4m3/e5m2 codes with blocked E8M0 scales),
 *        MGQ_TENSOR_F32 (scale = device float s: one for A / dY, E for the
 *        weight; the product is multiplied by 1/(s_a s_b)), or
 *        MGQ_BLK_1x128_F32 ([BLOCK]'s DeepSeek-style recipe; each 128-deep
 *        partial product is scaled and summed in float32): for fwd and dgrad
 *        A (dY) with 1x128 float32 scale_inv [K/128][R_cap] and W (Wcol)
 *        with 128x128 float32 scale_inv [E][N/128][K/128]; for wgrad the
 *        column-wise copies with 128x1 blocks along each group's rows,
 *        scale_inv [R_cap/128][N] for dYcol and [R_cap/128][K] for Acol
 *        (one per column and 128 rows). The blockwise kernel needs at
 *        least 152 registers a thread in its compiled form (its register
 *        split); a build below that returns MGQ_ERR_CUDA instead of
 *        launching. Or MGQ_NV16_UE4M3 (fwd, dgrad and
 *        wgrad): e2m1 codes packed two per byte along the contraction (ld and
 *        the contraction length in elements, multiples of 256), 16-element
 *        ue4m3 block scales, and each operand's global_scale s_g (A / dY /
 *        the column-wise copies: one per tensor; W, Wcol: one per expert);
 *        the product is multiplied by 1/(s_g,a s_g,b). NVFP4 wgrad contracts
 *        in 256-row stages: offsets[e] multiples of 256 (otherwise
 *        MGQ_ERR_INVALID_ARG in the device error word, nothing written) and
 *        R_cap a multiple of 256. The second operand may carry scale_image
 *        (built by mgq_nv_scale_image from its scales, 16-byte aligned): the
 *        same values, one tensor-memory copy per MMA instead of two; the
 *        results are identical. scale_image is ignored for other scalings.
 * Operand layout (MGQ_TENSOR_F32 only): with per-tensor scales the
 *        column-wise copy holds the same codes as the row-wise one,
 *        transposed, so dgrad accepts the forward weight W [E, N, K] (ld >= K)
 *        in place of Wcol with layout MGQ_LAYOUT_MN, and wgrad accepts dY
 *        [R_cap, N] (ld >= N) and A [R_cap, K] (ld >= K) in place of dYcol and
 *        Acol with layout MGQ_LAYOUT_MN: the tensor cores read them
 *        transposed. Requires the 2-CTA kernel (wgrad: N a multiple of 256);
 *        MGQ_ERR_UNSUPPORTED otherwise and for every other scaling.
 * Requires offsets[e] multiples of 128, N a multiple of 256 (fwd/dgrad) or
 * 128, K a multiple of 128, 16-byte aligned pointers. */
int mgq_grouped_gemm_fwd(const mgq_operand* A, const mgq_operand* W, int scaling,
                         const int32_t* offsets, int E, int64_t R_cap, int64_t N,
                         int64_t K, void* Y, int out_dtype, void* stream);
int mgq_grouped_gemm_dgrad(const mgq_operand* dY, const mgq_operand* Wcol, int scaling,
                           const int32_t* offsets, int E, int64_t R_cap, int64_t N,
                           int64_t K, void* dA, int out_dtype, void* stream);
int mgq_grouped_gemm_wgrad(const mgq_operand* dYcol, const mgq_operand* Acol, int scaling,
                           const int32_t* offsets, int E, int64_t R_cap, int64_t N,
                           int64_t K, float beta, void* dW, int out_dtype, void* stream);

/* Scale image of an NVFP4 GEMM operand for the grouped GEMMs above ([GROUPED]:
 * NVFP4 e2m1 elements with ue4m3 scales per 16 along the contraction). The
 * same scale bytes, rearranged: for each 128-row block rb and each 256-element
 * stage s of the contraction, its four 512-byte chunks c = 4 s + i (the 128x4
 * tiled layout: 128 rows x 4 blocks of 16), each written four times,
 *   image[(((rb * (ld / 256) + s) * 4 + i) * 4 + q) * 512 + b]
 *       = scale[(rb * (ld / 64) + 4 s + i) * 512 + b],   q = 0..3,
 * one copy per tensor-memory lane quadrant.
 * scale: device, the operand's scales (rows x ld / 16 bytes); rows: the
 * operand's rows (a multiple of 128); ld: its row pitch in elements (a
 * multiple of 256); image: device, caller-owned, rows * ld / 4 bytes, 16-byte
 * aligned. Enqueued on `stream`; MGQ_ERR_INVALID_ARG for bad sizes or
 * pointers. */
int mgq_nv_scale_image(const void* scale, int64_t rows, int64_t ld, void* image, void* stream);

/* Process-wide options of the grouped GEMMs (every entry point above and
 * below). They change which kernel runs or how it stores, never the values it
 * computes, except the two test hooks. They start at 0 (the defaults), apply
 * to calls made after they are set, and are never read from the environment.
 *  MGQ_GEMM_OPT_FORCE_1CTA    1: every call on the one-SM kernel (per-tensor
 *                             calls otherwise run on the 2-SM pair kernel)
 *  MGQ_GEMM_OPT_MX_PAIR       1: MX calls on the pair kernel (slower on the
 *                             Mixtral shapes; the default is the one-SM kernel)
 *  MGQ_GEMM_OPT_NV_PAIR       1: NVFP4 calls on the pair kernel (likewise)
 *  MGQ_GEMM_OPT_DIRECT_STORE  1: the pair kernel stores from registers
 *                             instead of through TMA
 *  MGQ_GEMM_OPT_DEBUG_STALL   failure-detection test hook: 1 makes the
 *                             producer issue no loads, so the pipeline waits
 *                             run out and the call reports MGQ_ERR_TIMEOUT
 *                             through mgq_get_error with nothing stored
 *  MGQ_GEMM_OPT_WAIT_MS       limit of every pipeline wait in ms (0: 2000;
 *                             at most 600000)
 * Values outside {0, 1} (WAIT_MS: outside [0, 600000]) or an unknown option
 * give MGQ_ERR_INVALID_ARG. Setting an option while another host thread
 * launches a GEMM is safe; which setting that launch sees is unspecified. */
typedef enum {
  MGQ_GEMM_OPT_FORCE_1CTA = 0,
  MGQ_GEMM_OPT_MX_PAIR = 1,
  MGQ_GEMM_OPT_NV_PAIR = 2,
  MGQ_GEMM_OPT_DIRECT_STORE = 3,
  MGQ_GEMM_OPT_DEBUG_STALL = 4,
  MGQ_GEMM_OPT_WAIT_MS = 5,
  MGQ_GEMM_OPT_COUNT = 6
} mgq_gemm_option;
int mgq_set_gemm_option(int option, int64_t value);
int mgq_get_gemm_option(int option, int64_t* value);

/* ---- f1: gate/up GEMM with SwiGLU + quantisation in its epilogue ------------
 * The forward gate/up GEMM of mgq_grouped_gemm_fwd (A [R_cap, K], W1 [E, 2F, K]
 * with the gate rows 0..F-1 and the up rows F..2F-1 of each expert) whose
 * epilogue applies SwiGLU: for every row, g and u are the GEMM outputs rounded
 * to bf16 (the values mgq_grouped_gemm_fwd writes), h = bf16(silu(g) u), and h
 * is quantised row-wise into qh exactly as mgq_swiglu_quantize would quantise
 * it (same codes, scales and amax). The tiles pair gate rows f.. with the up
 * rows F + f.., so each tile holds both halves of 128 ffn columns.
 *  scaling  MGQ_MX32_E8M0 or MGQ_TENSOR_F32 (qh->scaling must match), or
 *           MGQ_NV16_UE4M3: the epilogue writes h (h_bf16 required) and its
 *           amax, and a second pass casts h as mgq_swiglu_quantize does, rows
 *           and (qh->col set) columns.
 *           qh->col: MX only (NULL for MGQ_TENSOR_F32): the epilogue also
 *           writes the column-wise copy of h exactly as mgq_swiglu_quantize
 *           would: codes [F, R_cap] (row f holds column f of h, one E8M0
 *           block per 32 rows of a group) and their tiled scales
 *           (mgq_mx_scale_bytes(F, R_cap) bytes)
 *  gu_bf16  [R_cap, 2F] receives g | u when not NULL (the backward's
 *           dSwiGLU input); h_bf16 [R_cap, F] receives h when not NULL
 * Requirements as mgq_grouped_gemm_fwd with N = 2F, F a multiple of 128.
 * MGQ_ERR_UNSUPPORTED for other scalings. */
int mgq_grouped_gemm_fwd_swiglu(const mgq_operand* A, const mgq_operand* W1, int scaling,
                                const int32_t* offsets, int E, int64_t R_cap, int64_t F,
                                int64_t K, const mgq_qdesc* qh, void* gu_bf16, void* h_bf16,
                                void* stream);

/* ---- f1: down-projection dgrad with dSwiGLU + quantisation in its epilogue --
 * The dgrad of the down projection (as mgq_grouped_gemm_dgrad with N = H and
 * K = F: dh = dY W2_e, dY [R_cap, H], W2 as the Wcol operand there or the
 * forward weight [E, H, F] with MGQ_LAYOUT_MN) whose epilogue rounds dh to
 * bf16 and applies the SwiGLU derivative with the forward's gu_bf16 [R_cap, 2F]
 * (g | u), then quantises [dG | dU] row-wise into q exactly as
 * mgq_dswiglu_quantize would (same codes, scales and amax).
 *  scaling  MGQ_TENSOR_F32 (q->scaling too; q->col must be NULL) or
 *           MGQ_MX32_E8M0 (q->scaling too; q->row.scale required): E8M0
 *           blocks of 32 along the 2F columns, and with q->col set the
 *           column-wise copy [2F, R_cap] with blocks of 32 rows of a group
 *           and tiled scales, as mgq_dswiglu_quantize writes it
 *  dh_bf16  [R_cap, F] receives dh when not NULL; dgu_bf16 [R_cap, 2F]
 *           receives dG | dU when not NULL
 * MGQ_ERR_UNSUPPORTED for other scalings. */
int mgq_grouped_gemm_dgrad_dswiglu(const mgq_operand* dY, const mgq_operand* W2, int scaling,
                                   const int32_t* offsets, int E, int64_t R_cap, int64_t H,
                                   int64_t F, const void* gu_bf16, const mgq_qdesc* q,
                                   void* dh_bf16, void* dgu_bf16, void* stream);

/* ---- a6/a10: SwiGLU and its derivative, fused with quantisation -------------
 * h = silu(g) * u, g = gu[:, :F], u = gu[:, F:2F] (float32, rounded to bf16,
 * then quantised). dG = dh u s (1 + g (1 - s)), dU = dh silu(g), s = sigmoid(g),
 * rounded to bf16 then quantised ([dG | dU] is one [R_cap, 2F] matrix).
 * Rows [0, offsets[E]) are processed. q->col (when set) receives the
 * column-wise copy [C, R_cap] with blocks along the rows of each group (MX
 * 32, blockwise 128 with scale_inv [R_cap/128][C]; blockwise row-wise
 * scale_inv [C/128][R_cap]).
 * NVFP4 (q->scaling MGQ_NV16_UE4M3): two passes, the bf16 result (h_bf16 /
 * dgu_bf16 required) with its amax in q->amax_out, then the cast with s_g =
 * 6*448/amax written to q->tensor_scale. */
int mgq_swiglu_quantize(const void* gu_bf16, int64_t R_cap, int F, const int32_t* offsets,
                        int E, const mgq_qdesc* q, void* h_bf16, void* stream);
int mgq_dswiglu_quantize(const void* dh_bf16, const void* gu_bf16, int64_t R_cap, int F,
                         const int32_t* offsets, int E, const mgq_qdesc* q,
                         void* dgu_bf16, void* stream);

/* ---- a7: unpermute / combine -------------------------------------------------
 * out[t] = sum_j probs[t, j] * Y[row_id_map[t, j]] (float32, j ascending) -> bf16. */
int mgq_moe_unpermute(const void* y_bf16, const int32_t* row_id_map, const float* probs,
                      int T, int k, int H, void* out_bf16, void* stream);

/* ---- a8: unpermute backward, fused with quantisation of dY -----------------
 * dY[row(t, j)] = float32(probs[t, j] * dout[t]) quantised into q (row and
 * col; the column-wise copy [H, R_cap] with blocks along each group's rows:
 * MX 32, NVFP4 16, blockwise 128), filler rows zero;
 * dprobs[t, j] = <dout[t], Y[row(t, j)]> (float32).
 * NVFP4: an amax pre-pass over dY (max |fl(p d)| over a row is
 * fl(|p| max |d|)) into q->amax_out, s_g into q->tensor_scale. */
int mgq_moe_unpermute_bwd(const void* dout_bf16, const void* y_bf16,
                          const int32_t* row_id_map, const int32_t* src_row,
                          const float* probs, int T, int k, int H, int64_t R_cap,
                          const int32_t* offsets, int E, const mgq_qdesc* q,
                          float* dprobs, void* stream);

/* ---- a12: permute backward ----------------------------------------------------
 * dX[t] = sum_j dA[row_id_map[t, j]] (float32, j ascending) -> bf16. */
int mgq_moe_permute_bwd(const void* da_bf16, const int32_t* row_id_map, int T, int k,
                        int H, void* dx_bf16, void* stream);

/* ---- a13: delayed scaling ------------------------------------------------------
 * [MOE-FP8] --fp8-amax-history-len 1024 --fp8-amax-compute-algo max.
 * For each of n roles: history[i*L + head] = amax[i]; m = max(history[i*L ..]);
 * if m > 0 and finite, scale[i] = fmax / m (float32); amax[i] is reset to 0.
 * head (device int32) advances by one (mod L) after all roles. */
int mgq_amax_history_update(float* history, int32_t* head, float* amax, float* scale,
                            int n, int L, float fmax, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* MGQ_H */
