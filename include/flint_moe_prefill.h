/*
 * flint_moe_prefill.h - C ABI of the expert-grouped tensor-core path of the
 * Flint-style W4A16 MoE layer, for batches of many tokens (prefill, or decode
 * batches past the low-latency path's 32 tokens).
 *
 * "Day-0 Support for Flint on vLLM", section "Optimisation": the new MoE
 * kernels gave the largest gain in prefill as well as in small-batch decode.
 * With many tokens every expert is selected by several tokens, so its weights
 * are dequantised once into shared memory and multiplied against all of its
 * tokens on the tensor cores (tcgen05.mma, FP32 accumulation in tensor
 * memory), instead of once per token tile in registers. Experts that few
 * tokens chose (up to 16, in calls of up to 512 tokens; the shared expert
 * while a call has at most 256 tokens) are multiplied on mma.sync tiles of up
 * to 16 tokens with the weights dequantised in registers instead, where the
 * tensor-core staging would serve too few columns per weight.
 *
 * Same computation and rounding points as flint_moe_decode (flint_moe.h):
 *   logit = x Wr^T (FP32); sigmoid top-k (ties to the lower index),
 *   renormalised weights; per selected and shared expert
 *   h = bf16(silu(G_g c_g x) * (G_u c_u x)), y = G_d c_d h (FP32);
 *   out = bf16(sum_j w_j y_j + sum_shared y_s), summed in a fixed order
 *   (shared experts first, then the token's top-k in rank order).
 *
 * Conventions as in flint_moe.h: device pointers, caller-owned memory, no
 * allocation, asynchronous on `stream`, errors as flint_moe_status; device-side
 * wait timeouts set bits of the workspace status word (flint_moe_read_status).
 */
#ifndef FLINT_MOE_PREFILL_H_
#define FLINT_MOE_PREFILL_H_

#include "flint_moe.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Largest token count of one flint_moe_prefill call. */
#define FLINT_MOE_PREFILL_MAX_TOKENS 65536

/* Bytes of the prefill workspace for calls of up to max_tokens tokens
 * (1..FLINT_MOE_PREFILL_MAX_TOKENS); 0 if the configuration or count is not
 * supported (NVFP4 expert weights only). It holds the logits, the routing, the
 * expert-grouped token lists and tile lists, the normalised (pre-norm block)
 * and f16 token rows, h (bf16) of every (token, expert) pair and the FP32
 * expert outputs y [B][S + k][H] that the combine sums. */
size_t flint_moe_prefill_workspace_bytes(const flint_moe_config* cfg, int32_t max_tokens);

/* Zeroes a prefill workspace's header and per-expert counters; call once
 * after allocating it. Asynchronous on stream. */
flint_moe_status flint_moe_prefill_workspace_init(const flint_moe_config* cfg, int32_t max_tokens,
                                                  void* workspace, cudaStream_t stream);

/* The MoE layer for B tokens, 0 <= B <= FLINT_MOE_PREFILL_MAX_TOKENS (B = 0 is
 * a no-op). x: bf16 [B][H]; out: bf16 [B][H] (must not overlap x); workspace:
 * workspace_bytes >= flint_moe_prefill_workspace_bytes(cfg, B), 256-byte
 * aligned, initialised once with flint_moe_prefill_workspace_init, not shared
 * with another call in flight. Seven kernels in stream order (nine in calls of
 * up to 512 tokens, with the small-tile kernels of steps 5 and 6):
 *   1. router GEMM on the tensor cores (bf16 router rows x tokens, FP32),
 *      split along H into up to 8 ranges while its tiles are fewer than the
 *      SMs (the partial sums live in the y region until step 6);
 *   2. the partial logits added in split order (a fixed order: the result does
 *      not depend on timing), sigmoid top-k per token, counting the tokens of
 *      every expert;
 *   3. plan: slots, the first grouped row of every expert, and the (expert,
 *      128-row tile, token tile) work lists of both tile kinds;
 *   4. per token: its entries of the expert-grouped row lists, and its row in
 *      f16 (times a power of two that keeps every bf16 value exact) at its
 *      grouped rows;
 *   5. gate/up grouped GEMM: NVFP4 tiles dequantised to f16 in shared memory,
 *      tcgen05.mma against the expert's token rows (loaded by TMA), SiLU * up
 *      epilogue writing h (bf16); then the small tiles the same way on
 *      mma.sync;
 *   6. down grouped GEMM on h (bf16 products), epilogue writing w_j * y into
 *      y[B][S + k][H]; then its small tiles;
 *   7. combine: out = bf16(sum over the S + k rows of y), in that fixed order.
 * NVFP4 layers only (FLINT_MOE_EUNSUPPORTED for BF16 weights). Inputs must be
 * finite. x and out 16-byte aligned. */
flint_moe_status flint_moe_prefill(const flint_moe_layer* layer, const uint16_t* x_bf16, int32_t B,
                                   uint16_t* out_bf16, void* workspace, size_t workspace_bytes,
                                   cudaStream_t stream);

/* The layer as a pre-norm sublayer of the residual stream, for B tokens, with
 * the same definition as flint_moe_decode_prenorm ("Day-0 Support for Flint on
 * vLLM", section "Model architecture": a pre-norm MoE): for every row r,
 *   x  = bf16(r * w / sqrt(mean(r^2) + eps))   (RMSNorm, w = the layer's norm weight)
 *   r' = bf16(r + flint_moe_prefill(x))
 * One more kernel normalises the rows into the workspace first; the combine
 * adds the residual. residual_out may be residual_in (in-place update) but must
 * not overlap it otherwise. FLINT_MOE_EINVAL if the layer has no norm weight
 * (flint_moe_layer_set_norm). Otherwise as flint_moe_prefill. */
flint_moe_status flint_moe_prefill_prenorm(const flint_moe_layer* layer, const uint16_t* residual_in_bf16,
                                           int32_t B, uint16_t* residual_out_bf16, void* workspace,
                                           size_t workspace_bytes, cudaStream_t stream);

/* Copies the routing of the last flint_moe_prefill of B tokens on this
 * workspace: idx int32 [B][k], w float32 [B][k], and (if logits is not NULL)
 * the router logits float32 [B][E]. Device pointers. For tests. */
flint_moe_status flint_moe_prefill_debug_routing(const flint_moe_config* cfg, const void* workspace,
                                                 int32_t B, int32_t* idx, float* w, float* logits,
                                                 cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* FLINT_MOE_PREFILL_H_ */
