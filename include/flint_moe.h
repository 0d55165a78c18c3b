/*
 * flint_moe.h - C ABI of the GB300 (sm_103a) small-batch decode step of a
 * Flint-style mixture-of-experts FFN layer with weight-only NVFP4 (W4A16)
 * weights and BF16 activations.
 *
 * The method is described on the page "Day-0 Support for Flint on vLLM"
 * (vLLM blog, in Chinese, Japanese, French and Korean versions):
 *   - section "Model architecture": 256 experts, sigmoid top-6, plus one
 *     shared expert; the NVFP4 checkpoint stores NVIDIA's NVFP4 format in a
 *     different byte order, is repacked losslessly at load and runs
 *     weight-only (W4A16) with BF16 activations, following the reference
 *     implementation's rounding points;
 *   - section "Optimisation": small-batch MoE kernels whose router and expert
 *     GEMVs read only the selected experts' weights; SiLU with the reference
 *     rounding; for up to 8 requests routing and the expert combine are fused
 *     into the adjacent GEMV kernels, and every kernel uses programmatic
 *     dependent launch so it loads its weights while the previous one runs.
 *
 * What one decode computes, per token x (bf16 [H]):
 *   logit_e = sum_h x_h Wr[e,h]           FP32 accumulation, bf16 router Wr [E,H]
 *   s_e = sigmoid(logit_e);  key_e = s_e + sel_bias_e
 *   top-k experts by key (descending; ties go to the lower expert index)
 *   w_j = s_j / sum_top-k s (if renormalize) * routed_scale
 *   for every selected expert and every shared expert:
 *     g = G_g * (c_g x),  u = G_u * (c_u x)   FP32 accumulation
 *     h = bf16(silu(g) * u)                    BF16 rounding point
 *     y = G_d * (c_d h)                        FP32 accumulation
 *   out = bf16(sum_j w_j y_j + sum_shared y_s) BF16 rounding point
 * with c = E2M1(code) * E4M3(block scale) (exact) and G the FP32 tensor scale.
 *
 * Conventions (every entry point):
 *   - All tensor pointers are DEVICE pointers unless stated otherwise; the
 *     caller allocates and owns all memory. Nothing here allocates device
 *     memory or synchronises, except flint_moe_read_status, which says so.
 *   - Every call is asynchronous on `stream` (0 = legacy default stream) and
 *     returns a flint_moe_status; no C++ exception crosses this boundary.
 *   - Pointers that feed 16-byte vector or bulk-copy loads must be 16-byte
 *     aligned, else FLINT_MOE_EALIGN.
 *   - Inputs must be finite. Errors found on the device (a wait that timed out,
 *     a NaN scale code at pack time) are recorded as bits of a device status
 *     word; they never fault or trap the GPU.
 */
#ifndef FLINT_MOE_H_
#define FLINT_MOE_H_

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FLINT_MOE_OK = 0,
  FLINT_MOE_EINVAL = 1,       /* bad argument: null pointer, size out of range */
  FLINT_MOE_EALIGN = 2,       /* pointer not 16-byte aligned */
  FLINT_MOE_ECUDA = 3,        /* a CUDA runtime call failed */
  FLINT_MOE_ETIMEOUT = 4,     /* a device-side bounded wait gave up (status word) */
  FLINT_MOE_EUNSUPPORTED = 5  /* shape or format this build does not handle */
} flint_moe_status;

/* Device status word bits (see flint_moe_read_status). */
#define FLINT_MOE_DEV_ERR_TIMEOUT   0x1  /* an mbarrier wait ran past its limit */
#define FLINT_MOE_DEV_ERR_NAN_SCALE 0x2  /* pack met an E4M3 NaN scale (0x7F/0xFF) */
#define FLINT_MOE_DEV_ERR_SLOTS     0x4  /* inconsistent routing slots (internal) */

typedef enum { FLINT_MOE_NVFP4 = 0, FLINT_MOE_BF16 = 1 } flint_moe_weight_fmt;

/* Layer shape and routing options.
 * hidden H: multiple of 256 up to 2048, or of 2048 up to 8192 (Flint: 2048).
 * num_experts E: 1..512 (Flint: 256).  top_k: 1..min(E, 16) (Flint: 6).
 * inter I: routed and shared expert intermediate size, multiple of 64, <= 4096
 *   (512 for the Flint-shape workload; the pages give only ~40B total /
 *   ~2.5B active parameters).
 * n_shared S: 0..4 always-on experts, unweighted (Flint: 1).
 * weight_fmt: FLINT_MOE_NVFP4 or FLINT_MOE_BF16 expert weights (router is bf16).
 * renormalize: nonzero -> w = s / sum(top-k s); zero -> w = s.
 * routed_scale: multiplies every routed weight (1.0 for Flint). */
typedef struct flint_moe_config {
  int32_t hidden;
  int32_t num_experts;
  int32_t top_k;
  int32_t inter;
  int32_t n_shared;
  int32_t weight_fmt;
  int32_t renormalize;
  float routed_scale;
} flint_moe_config;

/* Canonical (source) weights of one layer, device pointers, experts stacked
 * [E + S] with the S shared experts last.
 * NVFP4 matrix [rows, cols]: codes uint8 [rows][cols/2] (element 2j is the
 *   low nibble of byte j), scales uint8 E4M3 [rows][cols/16] (one per 16
 *   consecutive elements of a row), global float32 (one per matrix).
 * gate, up: [I, H] each; down: [H, I].
 * For FLINT_MOE_BF16 only the *_bf16 pointers are read: [E+S][I][H] (gate,
 * up) and [E+S][H][I] (down), bf16 bit patterns. */
typedef struct flint_moe_nvfp4_src {
  const uint8_t* codes;
  const uint8_t* scales;
  const float* global;
} flint_moe_nvfp4_src;

typedef struct flint_moe_src {
  flint_moe_nvfp4_src gate, up, down;
  const uint16_t* gate_bf16;
  const uint16_t* up_bf16;
  const uint16_t* down_bf16;
} flint_moe_src;

/* A packed layer: plain device pointers, no ownership, no allocation. */
typedef struct flint_moe_layer {
  flint_moe_config cfg;
  const void* packed;        /* flint_moe_pack output, 16-byte aligned */
  const uint16_t* router;    /* bf16 [E][H], row-major, 16-byte aligned */
  const float* sel_bias;     /* float32 [E] added to the keys for selection only; may be NULL */
  const uint16_t* norm_weight; /* bf16 [H] pre-norm RMSNorm weight (flint_moe_layer_set_norm), or NULL */
  float norm_eps;              /* RMSNorm epsilon */
} flint_moe_layer;

/* Checks a configuration; FLINT_MOE_OK if this build supports it. */
flint_moe_status flint_moe_check_config(const flint_moe_config* cfg);

/* Bytes of one packed layer (all E + S experts plus their tensor scales).
 * 0 if the configuration is not supported. */
size_t flint_moe_packed_bytes(const flint_moe_config* cfg);

/* Bytes of the decode workspace for batches up to max_batch (1..32).
 * 0 if the arguments are not supported. */
size_t flint_moe_workspace_bytes(const flint_moe_config* cfg, int32_t max_batch);

/* Zeroes a workspace (counters, status word); call once after allocating it,
 * before its first decode. Asynchronous on stream. */
flint_moe_status flint_moe_workspace_init(const flint_moe_config* cfg, int32_t max_batch,
                                          void* workspace, cudaStream_t stream);

/* Lossless repack of canonical weights into the GB300 layout read by the
 * decode kernels ("repacked losslessly at load": page "Day-0 Support for Flint
 * on vLLM", section "Model architecture"). The layout is a byte permutation:
 * per expert, the gate/up rows are tiled 16 rows (8 gate + 8 up rows of the
 * same intermediate indices) by 64 columns, each tile holding the codes in the
 * order one warp's tensor-core fragments consume them, followed by the tile's
 * 16 x 4 scale bytes; the down rows are tiled the same way, 16 rows by 64
 * columns; tensor scales follow all experts. dst must hold
 * flint_moe_packed_bytes(cfg) bytes (dst_bytes is checked). A NaN scale code sets
 * FLINT_MOE_DEV_ERR_NAN_SCALE in *dev_status (device int32, may be NULL).
 * src and dst must not overlap. */
flint_moe_status flint_moe_pack(const flint_moe_config* cfg, const flint_moe_src* src,
                                void* dst, size_t dst_bytes, int32_t* dev_status,
                                cudaStream_t stream);

/* Inverse of flint_moe_pack: writes the canonical arrays named in dst (device
 * pointers, same shapes as flint_moe_src) from a packed layer. Used to prove
 * the repack is a bijection. */
flint_moe_status flint_moe_unpack_debug(const flint_moe_config* cfg, const void* packed,
                                        const flint_moe_src* dst, cudaStream_t stream);

/* Fills a layer handle (host struct) after checking shapes and alignment. */
flint_moe_status flint_moe_layer_init(const flint_moe_config* cfg, const void* packed,
                                      const uint16_t* router_bf16, const float* sel_bias,
                                      flint_moe_layer* out_layer);

/* Gives a layer its pre-norm RMSNorm (needed by flint_moe_decode_prenorm):
 * norm_weight bf16 [H] (device, 16-byte aligned, not owned), eps >= 0 and
 * finite, else FLINT_MOE_EINVAL / FLINT_MOE_EALIGN. */
flint_moe_status flint_moe_layer_set_norm(flint_moe_layer* layer, const uint16_t* norm_weight_bf16,
                                          float eps);

/* One decode step of the MoE layer for B tokens (0 <= B <= 32; B = 0 is a
 * no-op). x: bf16 [B][H]; out: bf16 [B][H]. x and out may be device memory or
 * pinned host memory (cudaHostAlloc / cudaMallocHost, addressable by the
 * device under unified addressing): with x in host memory a first kernel
 * copies it across the host link into the workspace, once, and the layer's
 * kernels read that copy; out in host memory is written by the down kernel
 * across the link; there is no copy-engine operation before or after. Any
 * other host memory is refused with FLINT_MOE_EINVAL. workspace: flint_moe_workspace_bytes
 * (cfg, >= B) bytes, initialised once with flint_moe_workspace_init, not shared
 * by decodes in flight at the same time. Three kernels: the router GEMV
 * (logits); gate/up GEMV with SiLU*up over the selected and shared experts;
 * down GEMV with the routing-weighted combine. Every block of the last two
 * computes the sigmoid top-k it needs from the logits itself. They are
 * chained with programmatic dependent launch, so each loads its
 * routing-independent weights (the shared expert, the router) while the
 * previous kernel, or the previous layer, still runs.
 * x and out must not overlap. Sections "Model architecture" and "Optimisation"
 * of "Day-0 Support for Flint on vLLM". */
flint_moe_status flint_moe_decode(const flint_moe_layer* layer, const uint16_t* x_bf16,
                                  int32_t B, uint16_t* out_bf16, void* workspace,
                                  cudaStream_t stream);

/* The layer as a pre-norm sublayer of the residual stream ("Day-0 Support for
 * Flint on vLLM", section "Model architecture": a pre-norm MoE; section
 * "Optimisation": norm kernels with the reference rounding). For every token
 * row r (bf16 [B][H]):
 *   x  = bf16(r * w / sqrt(mean(r^2) + eps))   (RMSNorm, w = norm_weight)
 *   r' = bf16(r + flint_moe_decode(x))          (the layer output is bf16)
 * The norm runs inside the router and gate/up kernels, the residual add inside
 * the down kernel: still three kernels, no extra pass over memory.
 * residual_out may be residual_in (in-place update) but must not overlap it
 * otherwise. FLINT_MOE_EINVAL if the layer has no norm weight. Otherwise as
 * flint_moe_decode. */
flint_moe_status flint_moe_decode_prenorm(const flint_moe_layer* layer, const uint16_t* residual_in_bf16,
                                          int32_t B, uint16_t* residual_out_bf16, void* workspace,
                                          cudaStream_t stream);

/* Copies the routing of the last decode from the workspace: idx int32 [B][k]
 * and w float32 [B][k] (device pointers), in selection order. */
flint_moe_status flint_moe_debug_routing(const flint_moe_config* cfg, const void* workspace,
                                         int32_t B, int32_t* idx, float* w, cudaStream_t stream);

/* Dequantised weights of one matrix of one packed expert, read back through
 * the decode kernels' own dequantisation: out float32 [rows][cols] = c * G in
 * canonical row-major order. mat: 0 gate, 1 up, 2 down. expert: 0..E+S-1. */
flint_moe_status flint_moe_debug_dequant(const flint_moe_config* cfg, const void* packed,
                                         int32_t expert, int32_t mat, float* out,
                                         cudaStream_t stream);

/* Phase trace of the decode kernels, for profiling. Only a library built with
 * -DFLINT_MOE_TRACE records it; otherwise returns FLINT_MOE_EUNSUPPORTED.
 * op 0: clear the trace (asynchronous on stream). op 1: copy it to
 * host_events, uint64 [64 calls][24 events][2] = earliest and latest
 * %globaltimer (ns) over all blocks, and SYNCHRONISE the stream. Call n of
 * flint_moe_decode records into slot n % 64. Events: router start 0, after
 * its wait 1, x arrived 2, end 3; gate/up start 8, after its wait 9, routed
 * 10, operands arrived 11, products done 12, end 13, routing published to
 * the block 14, keys sorted 21, top-k selected 22, top-k written 23; down
 * start 16, routed 17, after its wait 18, first item ready 19, end 20. */
flint_moe_status flint_moe_trace(int32_t op, uint64_t* host_events, cudaStream_t stream);

/* Self-check of the reciprocal the routing sigmoid uses (the hardware
 * approximation refined by one Newton-Raphson step): compares it, bit for bit,
 * with the IEEE quotient 1.0f / y for every FP32 y whose bit pattern lies in
 * [lo_bits, hi_bits) with 1 <= y < 2^125, and writes the number of
 * mismatches to *host_mismatches. SYNCHRONISES the stream. Returns
 * FLINT_MOE_EINVAL for a range outside [1, 2^125). */
flint_moe_status flint_moe_debug_rcp_check(uint32_t lo_bits, uint32_t hi_bits,
                                           uint64_t* host_mismatches, cudaStream_t stream);

/* Self-check of the failure path every kernel wait takes: one block waits on
 * an mbarrier that nothing completes, gives up after the same bounded wait
 * (about 200 ms of %globaltimer), sets FLINT_MOE_DEV_ERR_TIMEOUT in
 * *dev_status (device int32) and returns, leaving the context usable.
 * Asynchronous on stream. */
flint_moe_status flint_moe_debug_wait_timeout(int32_t* dev_status, cudaStream_t stream);

/* Reads the workspace status word into *host_status and clears it.
 * SYNCHRONISES the stream. Returns FLINT_MOE_ETIMEOUT if the timeout bit
 * was set, FLINT_MOE_OK otherwise (other bits are reported in *host_status). */
flint_moe_status flint_moe_read_status(const void* workspace, int32_t* host_status,
                                       cudaStream_t stream);

/* Bytes of the scratch array behind flint_moe_decode_noalloc. */
#define FLINT_MOE_NOALLOC_SCRATCH_BYTES (8u << 20)

/* flint_moe_decode for callers that cannot allocate device memory for a
 * workspace: a plugin whose host application owns every device allocation and
 * offers it no allocator, or a latency-critical loop in which cudaMalloc and
 * cudaFree could synchronise the device. No counterpart on the pages: it is a
 * variant of flint_moe_decode with the same arguments minus the workspace.
 * The scratch is one array of FLINT_MOE_NOALLOC_SCRATCH_BYTES bytes (8 MiB)
 * in this library's device memory, held by every GPU that loads the library
 * until the process exits. It allocates nothing and calls no allocating
 * routine. The first call on a device looks up the array's device address
 * (with that device current); make that first call before any stream capture:
 * while `stream` is being captured that first call returns FLINT_MOE_EINVAL.
 * Every call shares the array and leaves its contents behind; the call clears
 * what must start at zero. Calls whose work overlaps on the GPU (other streams,
 * other threads) race on the array: serialise them. Returns
 * FLINT_MOE_EUNSUPPORTED when the workspace this shape and batch need
 * (flint_moe_workspace_bytes) exceeds FLINT_MOE_NOALLOC_SCRATCH_BYTES (the
 * Flint-shape layer needs 6.1 MiB at B = 32, 0.78 MiB at B = 8), checked before
 * anything else touches the device. dev_status (device int32, 4-byte aligned,
 * may be NULL): the device status bits of this call (FLINT_MOE_DEV_ERR_*) are
 * ORed into it by one more small kernel after the decode. */
flint_moe_status flint_moe_decode_noalloc(const flint_moe_layer* layer, const uint16_t* x_bf16,
                                          int32_t B, uint16_t* out_bf16, int32_t* dev_status,
                                          cudaStream_t stream);

/* ---- loading helpers (checkpoint side, off the decode path) ---- */

/* Quantises n_mat float32 matrices [n_mat][rows][cols] to canonical NVFP4
 * (codes [n_mat][rows][cols/2], scales [n_mat][rows][cols/16], global
 * [n_mat]) with the two-level recipe: G = amax / (6 * 448); per 16-block
 * s = E4M3_rn(amax_blk / (6 G)); code = E2M1_rn(w / (E4M3(s) G)), all FP32,
 * round to nearest even, saturating; G = 0 or a zero scale gives zero codes.
 * cols must be a multiple of 16. The pages describe no quantiser (their
 * checkpoint was trained quantisation-aware); this one produces test and
 * benchmark weights from BF16/FP32 weights. */
flint_moe_status flint_moe_quantize_nvfp4(const float* w, int32_t n_mat, int32_t rows, int32_t cols,
                                          uint8_t* codes, uint8_t* scales, float* global,
                                          cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* FLINT_MOE_H_ */
