/*
 * moeq: grouped mixture-of-experts low-precision kernels for one GB300 GPU
 * (sm_103a).  C ABI.
 *
 * Conventions shared by every call below
 * --------------------------------------
 * - Every pointer is a DEVICE pointer the caller owns (allocated with
 *   cudaMalloc, PyTorch, ...).  The library never allocates, frees or
 *   synchronises inside a compute call; each call only enqueues kernels on
 *   `stream` (a cudaStream_t; NULL = the legacy default stream) and returns.
 *   Pointers must be 16-byte aligned unless stated otherwise.
 * - Ragged expert groups ("grouped_matmul_rowwise_dynamic_scaled_fp8", Args
 *   a_offsets / expert_ids): group g = 0..num_active_experts-1 owns rows
 *   [offsets[g], offsets[g+1]) and uses expert expert_ids[g] (any order,
 *   need not be sorted or unique).  offsets are uint32 [G+1], expert_ids are
 *   int32 [G].  Empty groups write nothing.  Rows outside every group are
 *   never written.
 * - Padded scale rows ("max.nn.moe.NvMxf4f8Strategy", grouped_quantize:
 *   per-expert padding of the scales; "grouped_quantize_dynamic_scaled_fp4_async_kernel",
 *   scales_offsets): the block scales of group g live in logical scale rows
 *   [scales_offsets[g], scales_offsets[g+1]); scales_offsets[g] must be a
 *   multiple of 128 and leave room for ceil(r_g / 128) * 128 rows.
 *   moeq_padded_scale_offsets() builds the tightest such offsets.
 * - Block-scale layout (the tensor core's tiled layout; the pages leave it
 *   open): logical scales [rows, Kv] (Kv = K / block) are stored as 512-byte
 *   atoms of 128 rows x 4 columns; byte (r, c) of an atom is at
 *   (r % 32) * 16 + (r / 32) * 4 + c; atom (rb, kb) starts at
 *   (rb * ceil(Kv / 4) + kb) * 512.  Weight scales are one such buffer per
 *   expert, each ceil(N / 128) * ceil(Kv / 4) * 512 bytes.
 * - FP4 elements are packed two per byte, the lower-k element in the low
 *   nibble.
 * - Routed tokens ("Struct_ep_dispatch_mxfp4", execute, on one rank):
 *   moeq_route_topk turns per-token top-k expert ids into the group layout
 *   above (group e = expert e, every expert, stable order);
 *   moeq_grouped_amax_scale_topk and moeq_quantize_topk then read each token
 *   once and give the bytes of the row-level calls on the routed rows.
 * - Host threads.  Calls may be made concurrently from several host threads,
 *   on the same or different streams.  The only host state the library
 *   keeps is per-device launch set-up (SM count, kernel attributes applied,
 *   occupancy answers), computed once per device under an internal lock.
 *   moeq_last_cuda_error() is per host thread.  The device error word is
 *   shared by every call on a device.
 * - num_active_experts == 0 (or zero total rows) is MOEQ_OK and launches
 *   nothing.  max_tokens_per_expert is a sizing hint (the largest token
 *   count of any active expert): it picks launch shapes only, and groups larger than
 *   it are still computed in full.
 * - Errors.  Bad host arguments return MOEQ_ERR_INVALID_ARG before anything
 *   is launched (this includes a missing NVFP4 scale tensor, the pages'
 *   ValueError of prepare_swiglu_operands).  A shape or format that is not
 *   built returns MOEQ_ERR_UNSUPPORTED.  A launch failure returns
 *   MOEQ_ERR_CUDA (see moeq_last_cuda_error()).  Bad device-side data
 *   (non-monotone offsets, an expert id outside [0, num_experts), offsets
 *   past the buffers, a wait that timed out) never faults the GPU: the
 *   affected group is skipped and a sticky bit is set in the device error
 *   word, read with moeq_get_device_error().
 */
#ifndef MOEQ_H
#define MOEQ_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *moeq_stream_t; /* == cudaStream_t */

typedef enum {
    MOEQ_OK = 0,
    MOEQ_ERR_INVALID_ARG = 1,
    MOEQ_ERR_UNSUPPORTED = 2,
    MOEQ_ERR_CUDA = 3,
    MOEQ_ERR_DEVICE = 4
} moeq_status;

/* Quantized formats ("max.nn.moe.NvMxf4f8Strategy", is_nvfp4; the kernel of
 * "grouped_quantize_dynamic_scaled_fp4_async_kernel" quantizes to
 * NVFP4 / MXFP4 / MXFP8).
 *   NVFP4: E2M1 elements, 16-element blocks, E4M3 block scale, fp32
 *          per-expert tensor scale.
 *   MXFP4: E2M1 elements, 32-element blocks, E8M0 block scale.
 *   MXFP8: E4M3 elements, 32-element blocks, E8M0 block scale. */
typedef enum { MOEQ_NVFP4 = 0, MOEQ_MXFP4 = 1, MOEQ_MXFP8 = 2 } moeq_format;

/* Device error word bits (sticky until moeq_clear_device_error). */
#define MOEQ_DEVERR_BAD_OFFSETS 0x1u /* non-monotone or out-of-range offsets */
#define MOEQ_DEVERR_BAD_EXPERT 0x2u  /* expert id outside [0, num_experts)   */
#define MOEQ_DEVERR_SCALE_ROWS 0x4u  /* scale offsets unaligned / too small  */
#define MOEQ_DEVERR_TIMEOUT 0x8u     /* a pipeline wait gave up (~1 s)       */
#define MOEQ_DEVERR_BAD_INDEX 0x10u  /* gather index outside the input rows  */
#define MOEQ_DEVERR_BOUNDS 0x20u     /* debug builds: a store outside its buffer was skipped */

/* Per-expert NVFP4 tensor scale of the activations
 * ("grouped_quantize_dynamic_scaled_fp4_async_kernel": sf_tensor, the
 * per-expert tensor-wise scale factor, is a read-only input; this call
 * produces it).  tensor_scale_out[e] = fp32(amax_e / 2688), 2688 = 6 * 448,
 * amax_e = max |in| over all rows of all groups routed to expert e; experts
 * with no rows or an all-zero input get 1.0.
 *   in            bf16 [total_rows, K], row stride in_row_stride elements.
 *   row_offsets   uint32 [G+1]; expert_ids int32 [G].
 *   tensor_scale_out  fp32 [num_experts], fully overwritten.
 * K must be a multiple of 8; in_row_stride a multiple of 8, >= K. */
moeq_status moeq_grouped_amax_scale(const void *in, int64_t in_row_stride,
                                    int64_t total_rows, int64_t K,
                                    const uint32_t *row_offsets,
                                    const int32_t *expert_ids,
                                    float *tensor_scale_out,
                                    int32_t num_experts,
                                    int32_t num_active_experts,
                                    moeq_stream_t stream);

/* Grouped activation quantizer ("grouped_quantize_dynamic_scaled_fp4_async_kernel":
 * each block of work finds its expert by binary search on row_offsets /
 * scales_offsets and quantizes that expert's BF16 rows; "max.nn.moe.NvMxf4f8Strategy",
 * grouped_quantize).
 *   in            bf16 [total_rows, K], row stride in_row_stride elements.
 *   out           NVFP4 / MXFP4: [total_rows, K/2] packed; MXFP8: [total_rows, K].
 *   scales        tiled block-scale buffer of scale_rows_total logical rows
 *                 x K/16 (NVFP4) or K/32 (MX) columns.  For group g the rows
 *                 [scales_offsets[g], scales_offsets[g] + r_g) get the scales of
 *                 its rows and the rows up to scales_offsets[g] + ceil(r_g/128)*128
 *                 are zeroed; any further rows and rows >= scales_offsets[G]
 *                 are untouched.
 *   tensor_scale  fp32 [num_experts] raw (dequantization-direction) scale s_e
 *                 (NVFP4 only, required; ignored for MX).
 * Per block (NVFP4): inv = 1/s_e; sb = E4M3((amax * inv) / 6);
 * q = E2M1(x * (inv / sb)), all zero when sb == 0.  MX: scale code
 * c = clamp(floor(log2 amax) - emax + 127, 0, 254) (emax 8 for E4M3, 2 for
 * E2M1); q = elem(x * 2^(127-c)); an all-zero block is all +0 with c = 0.
 * All rounding is to nearest even, saturating.  K must be a multiple of 128;
 * scale_rows_total a multiple of 128. */
moeq_status moeq_grouped_quantize(moeq_format fmt, const void *in,
                                  int64_t in_row_stride, int64_t total_rows,
                                  int64_t K, uint8_t *out, uint8_t *scales,
                                  int64_t scale_rows_total,
                                  const uint32_t *row_offsets,
                                  const uint32_t *scales_offsets,
                                  const int32_t *expert_ids,
                                  const float *tensor_scale,
                                  int32_t num_experts,
                                  int32_t max_tokens_per_expert,
                                  int32_t num_active_experts,
                                  moeq_stream_t stream);

/* Gather-fused variants ("max.nn.moe.NvMxf4f8Strategy", grouped_quantize:
 * the indices and indices_divisor arguments).  Reading adopted: the rows
 * being quantized are gathered from the input, quantized row t reading input
 * row indices[t] / indices_divisor (e.g. indices = the expert-sorted
 * positions token * top_k + slot and indices_divisor = top_k, so the MoE
 * permutation needs no separate copy).  Everything else is exactly
 * moeq_grouped_amax_scale / moeq_grouped_quantize on the gathered rows.
 *   in          bf16 [in_rows, K], row stride in_row_stride elements.
 *   indices     int32 [total_rows] (device); indices_divisor >= 1.
 *   total_rows  number of quantized rows (row_offsets index these).
 * An index whose input row falls outside [0, in_rows) skips that row and
 * sets MOEQ_DEVERR_BAD_INDEX. */
moeq_status moeq_grouped_amax_scale_gather(const void *in, int64_t in_row_stride,
                                           int64_t in_rows, int64_t K,
                                           const int32_t *indices, int32_t indices_divisor,
                                           int64_t total_rows, const uint32_t *row_offsets,
                                           const int32_t *expert_ids, float *tensor_scale_out,
                                           int32_t num_experts, int32_t num_active_experts,
                                           moeq_stream_t stream);

moeq_status moeq_grouped_quantize_gather(moeq_format fmt, const void *in, int64_t in_row_stride,
                                         int64_t in_rows, int64_t K, const int32_t *indices,
                                         int32_t indices_divisor, int64_t total_rows,
                                         uint8_t *out, uint8_t *scales, int64_t scale_rows_total,
                                         const uint32_t *row_offsets,
                                         const uint32_t *scales_offsets,
                                         const int32_t *expert_ids, const float *tensor_scale,
                                         int32_t num_experts, int32_t max_tokens_per_expert,
                                         int32_t num_active_experts, moeq_stream_t stream);

/* scales_offsets[g] = sum_{h<g} ceil((row_offsets[h+1]-row_offsets[h]) / 128) * 128,
 * g = 0..G (uint32 [G+1], device).  The tightest padding accepted by the
 * calls above. */
moeq_status moeq_padded_scale_offsets(const uint32_t *row_offsets,
                                      uint32_t *scales_offsets,
                                      int32_t num_active_experts,
                                      moeq_stream_t stream);

/* Grouped rowwise-scaled FP8 matmul ("grouped_matmul_rowwise_dynamic_scaled_fp8",
 * description and Args):
 *   c[t, n] = bf16( (sum_k a[t,k] * b[expert_ids[g], n, k]) * a_scales[t]
 *                   * b_scales[expert_ids[g], n] )
 * accumulated in fp32 by the tensor cores, the two scales applied once after
 * the reduction (acc * a_scale first, then * b_scale), round to nearest even.
 *   c         bf16 [total_tokens, N]
 *   a         E4M3 [total_tokens, K]
 *   b         E4M3 [num_experts, N, K] (K innermost: the page accepts only transposed b)
 *   a_scales  fp32 [total_tokens];  b_scales fp32 [num_experts, N]
 * K % 128 == 0, N % 16 == 0. */
moeq_status moeq_grouped_matmul_rowwise_fp8(
    void *c, const uint8_t *a, const uint8_t *b, const float *a_scales,
    const float *b_scales, const uint32_t *a_offsets,
    const int32_t *expert_ids, int64_t total_tokens, int64_t N, int64_t K,
    int32_t num_experts, int32_t max_tokens_per_expert,
    int32_t num_active_experts, moeq_stream_t stream);

/* Grouped block-scaled matmul with per-expert epilogue scales
 * ("max.nn.moe.NvMxf4f8Strategy", grouped_matmul: a grouped block-scaled
 * matmul with one scale per expert, applied in the matmul epilogue):
 *   c[t, n] = bf16( expert_scales[e] * sum_k (qa[t,k] * sa[t,k/v]) * (qb[e,n,k] * sb[e,n,k/v]) )
 * with e = expert_ids[g], v = 16 (NVFP4) or 32 (MXFP8, MXFP4).
 *   a      NVFP4 / MXFP4: packed [total_tokens, K/2]; MXFP8: [total_tokens, K]
 *   a_sf   tiled scales, scale_rows_total rows; row t of group g uses
 *          scale row a_scales_offsets[g] + (t - a_offsets[g])
 *   b      NVFP4 / MXFP4: packed [num_experts, N, K/2]; MXFP8: [num_experts, N, K]
 *   b_sf   per-expert tiled scales (see the layout above)
 *   expert_scales  fp32 [num_experts]; required for NVFP4, NULL means 1 for MX.
 * NVFP4 and MXFP4: K % 256 == 0; MXFP8: K % 128 == 0; N % 128 == 0. */
moeq_status moeq_grouped_matmul_blockscaled(
    moeq_format fmt, void *c, const uint8_t *a, const uint8_t *a_sf,
    const uint8_t *b, const uint8_t *b_sf, const float *expert_scales,
    const uint32_t *a_offsets, const uint32_t *a_scales_offsets,
    const int32_t *expert_ids, int64_t total_tokens, int64_t scale_rows_total,
    int64_t N, int64_t K, int32_t num_experts, int32_t max_tokens_per_expert,
    int32_t num_active_experts, moeq_stream_t stream);

/* Chained SwiGLU + NVFP4 requantization ("max.nn.moe.NvMxf4f8Strategy",
 * fused_silu_quantize: the gated activation, then quantization; the
 * SiLU-output scale is passed raw and inverted inside, as
 * prepare_swiglu_operands requires).
 *   y      bf16 [total_tokens, 2I]: column 2j = gate_j, 2j+1 = up_j
 *   h_j    = silu(gate_j) * up_j in fp32, silu(g) = g * sigma(g) with the
 *            library's own deterministic sigma, each step one IEEE fp32
 *            operation or one fused multiply-add:
 *              e = exp(-|g|): Cody-Waite reduction (ln 2 split into a
 *                  16-bit head and an fp32 tail, n from one FMA with the
 *                  1.5 * 2^23 shift), degree-7 Taylor polynomial by Horner
 *                  in FMAs, times 2^n (2^n taken as 0 for n < -126);
 *              d = 1 + e;  r = 1 / d by three Newton steps in FMAs
 *                  (q = 1 - d r, r = r + r q) from 24/17 - 8/17 d;
 *              sigma = r for g >= 0, e * r otherwise.
 *            CUDA's expf and IEEE division are not used.
 *   c_packed  NVFP4 [total_tokens, I/2];  c_sf tiled scales [scale_rows_total
 *            rows x I/16], padded per expert exactly like moeq_grouped_quantize
 *   out_tensor_scale  fp32 [num_experts] raw s_e (required).
 * I % 64 == 0. */
moeq_status moeq_swiglu_quantize(uint8_t *c_packed, uint8_t *c_sf,
                                 const void *y, const float *out_tensor_scale,
                                 const uint32_t *a_offsets,
                                 const uint32_t *a_scales_offsets,
                                 const int32_t *expert_ids,
                                 int64_t total_tokens,
                                 int64_t scale_rows_total, int64_t I,
                                 int32_t num_experts,
                                 int32_t max_tokens_per_expert,
                                 int32_t num_active_experts,
                                 moeq_stream_t stream);

/* Chained SwiGLU + MX requantization ("max.nn.moe.NvMxf4f8Strategy": the
 * strategy handles NVFP4, MXFP4 or MXFP8; fused_silu_quantize applies the
 * gated activation and then quantizes, read here as quantizing in the
 * strategy's format; MX formats carry no tensor scale).
 *   h as in moeq_swiglu_quantize, then per 32-element block of h the MX rule
 *   of moeq_grouped_quantize: c = clamp(floor(log2 amax) - emax + 127, 0, 254)
 *   (amax of the fp32 h values), q = elem(h * 2^(127-c)), an all-zero block
 *   all +0 with c = 0.
 *   fmt     MOEQ_MXFP4 (E2M1, c_q [total_tokens, I/2] packed) or MOEQ_MXFP8
 *           (E4M3, c_q [total_tokens, I]).
 *   c_sf    tiled E8M0 scales [scale_rows_total rows x I/32], padded per
 *           expert like moeq_grouped_quantize.
 * I % 128 == 0. */
moeq_status moeq_swiglu_quantize_mx(moeq_format fmt, uint8_t *c_q, uint8_t *c_sf,
                                    const void *y, const uint32_t *a_offsets,
                                    const uint32_t *a_scales_offsets,
                                    const int32_t *expert_ids, int64_t total_tokens,
                                    int64_t scale_rows_total, int64_t I,
                                    int32_t num_experts, int32_t max_tokens_per_expert,
                                    int32_t num_active_experts, moeq_stream_t stream);

/* Fused grouped NVFP4 matmul + SwiGLU + NVFP4 requantization in one kernel
 * ("max.nn.moe.NvMxf4f8Strategy", grouped_matmul_swiglu: equivalent to
 * grouped_matmul followed by fused_silu_quantize; its (c_packed,
 * c_swiglu_scales) match the chained path byte for byte with a bf16
 * rounding where the chained path has a bf16 tensor).
 * Computes, with no bf16 tensor in memory, exactly
 *   moeq_grouped_matmul_blockscaled(NVFP4, y, ...) ; moeq_swiglu_quantize(..., y, ...)
 * and writes the same bytes.  b is [num_experts, 2I, K/2] with gate/up rows
 * interleaved (row 2j = gate_j, row 2j+1 = up_j); b_sf its per-expert tiled
 * scales.  expert_scales and out_tensor_scale are required.
 *   a_row_scales  optional bf16 [total_tokens] (NULL = none; grouped_matmul_swiglu:
 *            one bf16 scale per row, applied with the expert scale ahead
 *            of the SwiGLU): gate and up become
 *            bf16((acc * expert_scale) * a_row_scale[t]), two fp32 multiplies
 *            in that order.  With row scales there is no chained counterpart.
 * K % 256 == 0, I % 64 == 0. */
moeq_status moeq_grouped_matmul_swiglu(
    uint8_t *c_packed, uint8_t *c_sf, const uint8_t *a, const uint8_t *a_sf,
    const uint8_t *b, const uint8_t *b_sf, const float *expert_scales,
    const float *out_tensor_scale, const void *a_row_scales, const uint32_t *a_offsets,
    const uint32_t *a_scales_offsets, const int32_t *expert_ids,
    int64_t total_tokens, int64_t scale_rows_total, int64_t I, int64_t K,
    int32_t num_experts, int32_t max_tokens_per_expert,
    int32_t num_active_experts, moeq_stream_t stream);

/* Fused grouped MX matmul + SwiGLU + MX requantization in one kernel: the
 * MX counterpart of moeq_grouped_matmul_swiglu (same reading of the
 * strategy: MXFP4 or MXFP8 throughout).  Computes, with no bf16 tensor in
 * memory, exactly
 *   moeq_grouped_matmul_blockscaled(fmt, y, ...) ; moeq_swiglu_quantize_mx(fmt, ..., y, ...)
 * and writes the same bytes.  a / a_sf / b / b_sf as for
 * moeq_grouped_matmul_blockscaled(fmt) with N = 2I (gate/up rows of b
 * interleaved); expert_scales optional (NULL = 1).
 * MXFP4: K % 256 == 0; MXFP8: K % 128 == 0; I % 128 == 0. */
moeq_status moeq_grouped_matmul_swiglu_mx(
    moeq_format fmt, uint8_t *c_q, uint8_t *c_sf, const uint8_t *a, const uint8_t *a_sf,
    const uint8_t *b, const uint8_t *b_sf, const float *expert_scales,
    const uint32_t *a_offsets, const uint32_t *a_scales_offsets, const int32_t *expert_ids,
    int64_t total_tokens, int64_t scale_rows_total, int64_t I, int64_t K,
    int32_t num_experts, int32_t max_tokens_per_expert, int32_t num_active_experts,
    moeq_stream_t stream);

/* ---- weight preparation ("max.nn.moe.NvMxf4f8Strategy", prepare_weight_scales:
 * block scales rearranged into the kernel's layout).  Run once per weight,
 * off the per-step path.  Every pointer is a caller-owned device pointer;
 * the calls only enqueue work on `stream`.  batch, rows, kv / row_bytes == 0
 * is MOEQ_OK and a no-op; negative sizes or NULL pointers (with a non-empty
 * call) return MOEQ_ERR_INVALID_ARG before any launch. */

/* Logical -> tiled block-scale layout, for `batch` independent matrices
 * (e.g. one per expert).
 *   logical  uint8 [batch, rows, kv], row-major, kv = K / block size
 *   tiled    uint8 [batch, ceil(rows / 128) * ceil(kv / 4) * 512]: matrix b starts at byte
 *            b * ceil(rows / 128) * ceil(kv / 4) * 512; inside it scale (r, c)
 *            sits in the 512-byte atom (r / 128, c / 4) (atoms row-block-major)
 *            at byte (r % 32) * 16 + ((r / 32) % 4) * 4 + c % 4 -- the layout
 *            every block-scaled call reads and writes.
 * Bytes of the tiled buffer that hold no logical scale are written 0. */
moeq_status moeq_sf_swizzle(uint8_t *tiled, const uint8_t *logical, int64_t batch,
                            int64_t rows, int64_t kv, moeq_stream_t stream);

/* Tiled -> logical (the inverse of moeq_sf_swizzle; padding is not read
 * into the output, which holds exactly batch * rows * kv bytes). */
moeq_status moeq_sf_unswizzle(uint8_t *logical, const uint8_t *tiled, int64_t batch,
                              int64_t rows, int64_t kv, moeq_stream_t stream);

/* Gate/up interleave of the fused SwiGLU GEMM's weight: out[b, 2j, :] =
 * gate[b, j, :] and out[b, 2j + 1, :] = up[b, j, :] for rows of row_bytes
 * bytes (packed weight rows, K / 2 bytes for E2M1; or logical scale rows,
 * kv bytes, then moeq_sf_swizzle with 2 * rows rows).
 *   gate, up uint8 [batch, rows, row_bytes];  out uint8 [batch, 2 * rows, row_bytes]
 * out must not overlap the inputs. */
moeq_status moeq_interleave_gate_up(uint8_t *out, const uint8_t *gate, const uint8_t *up,
                                    int64_t batch, int64_t rows, int64_t row_bytes,
                                    moeq_stream_t stream);

/* Expert dispatch on one rank ("Struct_ep_dispatch_mxfp4", execute: the
 * row_offsets, expert_ids and src_info outputs and the MXFP4 tokens; with a
 * single rank the all-to-all exchange is the identity and is not built).
 *
 * moeq_route_topk routes every choice i = t * top_k + k of topk_ids to the
 * group of its expert.  Group e is expert e for all e in [0, num_experts),
 * empty groups included; a group's rows hold its choices in increasing i
 * (a stable order: the page's atomic counters leave the order open).
 *   topk_ids        int32 [num_tokens, top_k] (device), expert of each choice.
 *   row_offsets     u32 [num_experts + 1] (out)
 *   expert_ids      int32 [num_experts] (out): 0 .. num_experts - 1
 *   src_info        int32 [num_tokens * top_k] (out): row r holds choice
 *                   src_info[r] (token src_info[r] / top_k); entries past
 *                   row_offsets[num_experts] are not written.
 *   dst_info        int32 [num_tokens * top_k] (out, may be NULL): the row of
 *                   choice i (the inverse of src_info), -1 for a dropped
 *                   choice.
 *   scales_offsets  u32 [num_experts + 1] (out, may be NULL): with
 *                   slot_rows == 0 the padded prefix of ceil(r_e / 128) * 128
 *                   (as moeq_padded_scale_offsets); with slot_rows > 0 (a
 *                   multiple of 128) the fixed-stride slots e * slot_rows of
 *                   the page's scale-slot fusion (fuse_a_scale_preshuffle,
 *                   slot stride max_padded_M).
 * A choice whose expert id lies outside [0, num_experts) is dropped and sets
 * MOEQ_DEVERR_BAD_EXPERT.  Limits: 1 <= num_experts <= 1024 (else
 * MOEQ_ERR_UNSUPPORTED), num_tokens * top_k < 2^31.  One CTA on one SM; no
 * memory besides the outputs. */
moeq_status moeq_route_topk(const int32_t *topk_ids, int64_t num_tokens, int32_t top_k,
                            int32_t num_experts, uint32_t *row_offsets, int32_t *expert_ids,
                            int32_t *src_info, int32_t *dst_info, uint32_t *scales_offsets,
                            int32_t slot_rows, moeq_stream_t stream);

/* Token-major quantization of routed tokens: the bytes of
 * moeq_grouped_quantize_gather(fmt, tokens, indices = src_info,
 * indices_divisor = top_k, groups = all num_experts experts, row_offsets,
 * scales_offsets, expert_ids = 0..E-1, tensor_scale) -- the same NVFP4 /
 * MXFP4 / MXFP8 rule per routed row, padding scale rows zero -- but each
 * token row is read once and written to its routed rows dst_info[t * top_k
 * + j] (MX formats quantize it once; NVFP4 shares the loads and block amax
 * across the choices' tensor scales).
 *   tokens       bf16 [num_tokens, K], row stride token_stride; K % 128 == 0.
 *   topk_ids, dst_info  int32 [num_tokens * top_k] (from moeq_route_topk).
 *   row_offsets, scales_offsets  u32 [num_experts + 1] (from moeq_route_topk).
 *   tensor_scale fp32 [num_experts] raw per-expert scales (NVFP4 only).
 *   out          [num_tokens * top_k, K / 2] (FP4) or [.., K] (MXFP8).
 *   scales       tiled block scales of scale_rows_total logical rows.
 * top_k <= 8 (else MOEQ_ERR_UNSUPPORTED).  A group whose scale rows do not
 * fit is skipped and sets MOEQ_DEVERR_SCALE_ROWS. */
moeq_status moeq_quantize_topk(moeq_format fmt, const void *tokens, int64_t token_stride,
                               int64_t num_tokens, int64_t K, const int32_t *topk_ids,
                               int32_t top_k, const int32_t *dst_info,
                               const uint32_t *row_offsets, const uint32_t *scales_offsets,
                               const float *tensor_scale, int32_t num_experts, uint8_t *out,
                               uint8_t *scales, int64_t scale_rows_total, moeq_stream_t stream);

/* Per-expert NVFP4 tensor scales from tokens and their top-k expert ids:
 * tensor_scale_out[e] = amax_e / (6 * 448) (1 when amax_e == 0), amax_e the
 * max |x| over the tokens with a choice of expert e -- the value
 * moeq_grouped_amax_scale gives over the routed rows
 * ("grouped_quantize_dynamic_scaled_fp4_async_kernel": the per-expert tensor
 * scale), but each token row is read once instead of once per choice.
 *   tokens      bf16 [num_tokens, K], row stride token_stride elements.
 *   topk_ids    int32 [num_tokens, top_k] (device).
 *   tensor_scale_out  fp32 [num_experts] (out).
 * An id outside [0, num_experts) is skipped and sets MOEQ_DEVERR_BAD_EXPERT. */
moeq_status moeq_grouped_amax_scale_topk(const void *tokens, int64_t token_stride,
                                         int64_t num_tokens, int64_t K, const int32_t *topk_ids,
                                         int32_t top_k, float *tensor_scale_out,
                                         int32_t num_experts, moeq_stream_t stream);

/* Scale rows that moeq_dispatch_mxfp4 needs: num_experts * slot_rows with
 * slot_rows > 0, else the largest possible padded total,
 * floor((num_tokens * top_k + 127 * num_experts) / 128) * 128.  Host only. */
int64_t moeq_dispatch_scale_rows(int64_t num_tokens, int32_t top_k, int32_t num_experts,
                                 int32_t slot_rows);

/* moeq_route_topk, then MXFP4 quantization of the routed rows (routed row r
 * is token src_info[r] / top_k), token-major (moeq_quantize_topk: each
 * token quantized once and stored to its top_k rows), in stream order.
 *   tokens          bf16 [num_tokens, hidden], row stride token_stride
 *                   elements; hidden a multiple of 128.
 *   out             uint8 [num_tokens * top_k, hidden / 2] packed E2M1
 *                   (rows past the routed count are not written).
 *   scales          tiled E8M0 block scales of scale_rows_total logical rows
 *                   of hidden / 32 scales; scale_rows_total >=
 *                   moeq_dispatch_scale_rows(...) and a multiple of 128.
 *   row_offsets, expert_ids, src_info, dst_info, scales_offsets: as
 *                   moeq_route_topk (dst_info and scales_offsets required
 *                   here).  top_k <= 8.
 * With slot_rows > 0 a group larger than slot_rows is not quantized and
 * sets MOEQ_DEVERR_SCALE_ROWS. */
moeq_status moeq_dispatch_mxfp4(const void *tokens, int64_t token_stride, int64_t num_tokens,
                                int64_t hidden, const int32_t *topk_ids, int32_t top_k,
                                int32_t num_experts, uint8_t *out, uint8_t *scales,
                                int64_t scale_rows_total, uint32_t *row_offsets,
                                int32_t *expert_ids, int32_t *src_info, int32_t *dst_info,
                                uint32_t *scales_offsets, int32_t slot_rows,
                                moeq_stream_t stream);

/* Reads the sticky device error word of the current device (MOEQ_DEVERR_*
 * bits) after synchronising `stream`.  Returns MOEQ_ERR_DEVICE when any bit
 * is set, MOEQ_OK otherwise. */
moeq_status moeq_get_device_error(moeq_stream_t stream, uint32_t *bits);

/* Clears the device error word of the current device (enqueued on stream). */
moeq_status moeq_clear_device_error(moeq_stream_t stream);

/* The cudaError_t of the last MOEQ_ERR_CUDA on this thread (0 if none). */
int moeq_last_cuda_error(void);

/* Static string naming a status. */
const char *moeq_status_string(moeq_status s);

#ifdef __cplusplus
}
#endif

#endif /* MOEQ_H */
