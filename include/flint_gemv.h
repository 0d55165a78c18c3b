/* Small-batch dense GEMV on weight-only NVFP4 (or BF16) matrices: C ABI.
 *
 * "Day-0 Support for Flint on vLLM", section "Optimisation": besides the MoE
 * kernels, small-batch dense GEMVs serve the dense MLPs of the first layers
 * and the projections, on the same NVFP4 weights with BF16 activations. For
 * every token row x (bf16) and output n:
 *   y[n] = bf16(G * sum_k c[n][k] * x[k])     (FP32 accumulation)
 * with c = E2M1(code) * E4M3(scale), one E4M3 scale per 16 consecutive values
 * of a row, and G the FP32 tensor scale (c the bf16 weight and G = 1 for a
 * BF16 matrix). With a norm weight the rows are first normalised like the
 * MoE pre-norm block: x = bf16(x * w / sqrt(mean(x^2) + eps)).
 *
 * Conventions as in flint_moe.h: device pointers, caller-owned memory,
 * asynchronous on `stream`, status codes, 16-byte alignment (FLINT_MOE_EALIGN).
 * Shapes: N a multiple of 16, K a multiple of 256 up to 8192 (and of 2048
 * above 2048), 0 <= B <= 32 (B = 0 is a no-op), else FLINT_MOE_EUNSUPPORTED
 * (shape) or FLINT_MOE_EINVAL (B). For K > 2048 the K / 2048 column slices of
 * a 16-row tile go to the CTAs of one thread-block cluster, whose partial sums
 * are added in distributed shared memory in a fixed order.
 */
#ifndef FLINT_GEMV_H
#define FLINT_GEMV_H

#include "flint_moe.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Canonical source of one matrix W [N][K]: NVFP4 codes uint8 [N][K/2]
 * (element 2j the low nibble of byte j), E4M3 scales uint8 [N][K/16] and a
 * float32 tensor scale, or bf16 values [N][K] (weight_fmt FLINT_MOE_BF16). */
typedef struct flint_gemv_src {
  const uint8_t* codes;
  const uint8_t* scales;
  const float* global_;
  const uint16_t* bf16;
} flint_gemv_src;

/* Bytes of a packed matrix; 0 for an unsupported shape or format. */
size_t flint_gemv_packed_bytes(int32_t N, int32_t K, int32_t weight_fmt);

/* Lossless repack of W into the tile layout the GEMV kernel reads (the same
 * fragment order as a MoE expert's down matrix). dst: flint_gemv_packed_bytes
 * bytes (dst_bytes is checked), 16-byte aligned. A NaN scale code sets
 * FLINT_MOE_DEV_ERR_NAN_SCALE in *dev_status (device int32, may be NULL). */
flint_moe_status flint_gemv_pack(const flint_gemv_src* src, int32_t N, int32_t K, int32_t weight_fmt, void* dst,
                                 size_t dst_bytes, int32_t* dev_status, cudaStream_t stream);

/* Inverse of flint_gemv_pack, into the arrays named in dst (same shapes as the
 * source); proves the repack is a bijection. */
flint_moe_status flint_gemv_unpack_debug(const void* packed, int32_t N, int32_t K, int32_t weight_fmt,
                                         const flint_gemv_src* dst, cudaStream_t stream);

/* y bf16 [B][N] = x bf16 [B][K] times W^T as above. norm_weight: bf16 [K]
 * RMSNorm weight applied to the rows of x first, or NULL. dev_status: device
 * int32 for the device status bits (FLINT_MOE_DEV_ERR_TIMEOUT when a bounded
 * wait gave up), may be NULL. Launched with programmatic dependent launch:
 * the weights are fetched before the wait for the previous kernel's x. x and y
 * must not overlap. */
flint_moe_status flint_gemv(const void* packed, int32_t N, int32_t K, int32_t weight_fmt, const uint16_t* x,
                            int32_t B, uint16_t* y, const uint16_t* norm_weight, float eps, int32_t* dev_status,
                            cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* FLINT_GEMV_H */
