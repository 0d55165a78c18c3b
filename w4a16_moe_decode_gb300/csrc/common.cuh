// Shared device helpers of the Flint-style W4A16 MoE decode library (sm_103a).
//
// Contents: the packed weight layout, the workspace layout, inline PTX for
// bulk copies, mbarriers, programmatic dependent launch and mma.sync, and the
// NVFP4 -> f16 tensor-core fragment dequantiser.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "flint_moe.h"

namespace flint {

// ---------------------------------------------------------------------------
// Packed layout (the result of flint_moe_pack).
//
// A "tile" is 16 matrix rows by the full reduction length, cut into k-groups of
// 64 columns (4 tensor-core k-steps of 16). Within a k-group (NVFP4, 576 B):
//   bytes [0, 512): lane L = 4g + t of the consuming warp owns bytes
//     [16L, 16L + 16): for k-step ks = 0..3 the four A-fragment bytes
//     b = 0..3 of mma.m16n8k16, byte b holding rows r = g + 8 (b & 1),
//     columns c = 2t + 8 (b >> 1) and c + 1 of that k-step (low nibble = c).
//   bytes [512, 576): the E4M3 scales, [row 16][ks 4].
// BF16 k-groups (2048 B): lane L owns 64 B = for ks 0..3, registers a0..a3
//   (2 bf16 each, lower column in the lower half) with the same row/column map.
// Per expert: I/8 gate/up tiles (rows 0..7 gate rows, 8..15 up rows of the
// same 8 intermediate indices; reduction length H), then H/16 down tiles
// (reduction length I). After all E + S experts: float32 globals [E+S][4] =
// {G_gate, G_up, G_down, 0}.
// ---------------------------------------------------------------------------
constexpr int KG_COLS = 64;
constexpr int KG_NVFP4 = 576;
constexpr int KG_BF16 = 2048;
constexpr int KG_CODE_BYTES = 512;
constexpr int MAX_BATCH = 32;
constexpr int MAX_TOPK = 16;
constexpr int MAX_EXPERTS = 512;
constexpr int MAX_SHARED = 4;

struct Layout {
  int64_t kg_bytes;      // 576 (NVFP4) or 2048 (BF16)
  int64_t gu_tile;       // bytes of one gate/up tile
  int64_t dn_tile;       // bytes of one down tile
  int64_t gu_bytes;      // all gate/up tiles of one expert
  int64_t expert_bytes;  // one expert
  int64_t globals_off;   // offset of the float32 globals
  int64_t total;         // packed bytes of the layer
};

__host__ __device__ inline Layout make_layout(int H, int I, int E, int S, int fmt) {
  Layout L;
  L.kg_bytes = fmt == FLINT_MOE_NVFP4 ? KG_NVFP4 : KG_BF16;
  L.gu_tile = (int64_t)(H / KG_COLS) * L.kg_bytes;
  L.dn_tile = (int64_t)(I / KG_COLS) * L.kg_bytes;
  L.gu_bytes = (int64_t)(I / 8) * L.gu_tile;
  L.expert_bytes = L.gu_bytes + (int64_t)(H / 16) * L.dn_tile;
  L.globals_off = (int64_t)(E + S) * L.expert_bytes;
  L.total = L.globals_off + (((int64_t)(E + S) * 16 + 255) / 256) * 256;
  return L;
}

// A dense matrix W [N][K] for the small-batch GEMV: laid out like one
// expert's down matrix (N / 16 tiles of 16 rows x K / 64 k-groups), then its
// tensor scale (float32 words [G, G, G, 0]).
__host__ __device__ inline Layout make_dense_layout(int N, int K, int fmt) {
  Layout L;
  L.kg_bytes = fmt == FLINT_MOE_NVFP4 ? KG_NVFP4 : KG_BF16;
  L.gu_tile = 0;
  L.gu_bytes = 0;
  L.dn_tile = (int64_t)(K / KG_COLS) * L.kg_bytes;
  L.expert_bytes = (int64_t)(N / 16) * L.dn_tile;
  L.globals_off = L.expert_bytes;
  L.total = L.globals_off + 256;
  return L;
}

// ---------------------------------------------------------------------------
// Workspace layout. Header words, then 256-byte aligned regions.
// ---------------------------------------------------------------------------
// HDR_HBIG: nonzero when some |h| of the call is 2^15 or more (its f16 copy
// is then not exact); set by the gate/up kernel, cleared by the router.
enum : int { HDR_STATUS = 1, HDR_HBIG = 2 };

// Regions: router logits [B][E] and the selection keys the router derives
// from them ([B][E], order-preserving unsigned form); the routing of the last decode ([B][k]
// indices and weights, for read-back); the largest |h| per (slot, token) row;
// h in bf16 [rows][I] in fragment order, and the same values in f16 (exact
// for 2^-14 <= |h| < 2^15, on the f16 grid of 2^-24 below) for the
// small-batch down kernel's f16 products. Slot s (shared experts first, then
// the distinct selected experts in ascending id) owns rows s * B .. s * B + B - 1.
struct WsLayout {
  size_t logits, keys, topk_idx, topk_w, hmax, h, h16, xs, xn, total;
  int max_slots, max_rows;
  int has_h16;  // the f16 copy of h exists (calls of up to 8 tokens, NVFP4 weights)
};

__host__ __device__ inline size_t ws_align(size_t x) { return (x + 255) & ~(size_t)255; }

// The f16 copy of h serves the small-batch down kernel only: calls of up to
// 8 tokens with NVFP4 weights.
__host__ __device__ inline bool ws_wants_h16(int B, int fmt) { return B <= 8 && fmt == FLINT_MOE_NVFP4; }

__host__ __device__ inline WsLayout make_ws_layout(int H, int E, int k, int I, int S, int maxB, bool with_h16) {
  WsLayout W;
  W.has_h16 = with_h16 ? 1 : 0;
  W.max_slots = S + (E < maxB * k ? E : maxB * k);
  W.max_rows = W.max_slots * maxB;
  size_t o = 256;
  W.logits = o;   o = ws_align(o + sizeof(float) * maxB * E);
  W.keys = o;     o = ws_align(o + sizeof(uint32_t) * maxB * E);
  W.topk_idx = o; o = ws_align(o + sizeof(int) * maxB * k);
  W.topk_w = o;   o = ws_align(o + sizeof(float) * maxB * k);
  W.hmax = o;     o = ws_align(o + sizeof(unsigned) * W.max_rows);
  W.h = o;        o = ws_align(o + (size_t)2 * W.max_rows * I);
  W.h16 = o;      o = ws_align(o + (with_h16 ? (size_t)2 * W.max_rows * I : 0));
  W.xs = o;       o = ws_align(o + (size_t)2 * maxB * H);  // x staged from host memory
  W.xn = o;       o = ws_align(o + (size_t)2 * maxB * H);  // the pre-norm block's normalised x
  W.total = o;
  return W;
}

// ---------------------------------------------------------------------------
// Inline PTX.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

// Makes initialised mbarriers visible to the async (bulk-copy) proxy.
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Orders this thread's earlier shared-memory accesses before later bulk-copy
// (async proxy) writes to the same bytes.
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
               : "memory");
}

// Bulk (non-tensor) copy global -> this CTA's shared memory, completing on bar.
// dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

// The same for data read once per decode (expert weights): an L2 evict-first
// policy, so the weight stream does not push out what the next kernels reuse
// (logits, h, activations, router rows, code).
__device__ __forceinline__ void bulk_g2s_stream(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "{\n\t.reg .b64 pol;\n\t"
      "createpolicy.fractional.L2::evict_first.b64 pol, 1.0;\n\t"
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], pol;\n\t}"
      ::"r"(smem_addr(dst)), "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

// Bounded wait on an mbarrier phase: gives up after ~limit_ns of wall time,
// setting FLINT_MOE_DEV_ERR_TIMEOUT in *status. Never spins forever.
constexpr uint64_t WAIT_LIMIT_NS = 200ull * 1000ull * 1000ull;  // 200 ms

__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, int* status) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  for (uint32_t it = 0;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 63) == 63 && global_ns() - t0 > WAIT_LIMIT_NS) {
      atomicOr(status, FLINT_MOE_DEV_ERR_TIMEOUT);
      return false;
    }
  }
}

// After a failed wait the CTA may still have bulk copies in flight into its
// shared memory; give them a second bounded wait before the CTA exits.
__device__ __forceinline__ void mbar_drain(uint64_t* bar, uint32_t parity) {
  const uint64_t t0 = global_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_ns() - t0 > WAIT_LIMIT_NS) return;
  }
}

// Thread-block clusters: rank, barrier and distributed shared memory.
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// All threads of every CTA of the cluster; orders their earlier shared-memory
// writes before the other CTAs' reads after it.
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// A float at the same shared-memory offset in CTA `rank` of this cluster.
__device__ __forceinline__ float ld_dsmem_f32(const void* p, uint32_t rank) {
  uint32_t remote;
  float v;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_addr(p)), "r"(rank));
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(remote) : "memory");
  return v;
}

// Programmatic dependent launch.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Loads of data written by an earlier kernel of the stream: L2 (".cg").
__device__ __forceinline__ uint4 ld_cg_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.cg.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}
__device__ __forceinline__ int ld_cg_s32(const int* p) { return __ldcg(p); }
__device__ __forceinline__ float ld_cg_f32(const float* p) { return __ldcg(p); }

__device__ __forceinline__ uint4 lds128(const void* p) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(smem_addr(p)));
  return v;
}
__device__ __forceinline__ uint32_t lds32(const void* p) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(smem_addr(p)));
  return v;
}

// D += A * B, m16n8k16, f16 inputs, f32 accumulate.
__device__ __forceinline__ void mma_f16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// ---------------------------------------------------------------------------
// NVFP4 dequantisation into mma.m16n8k16 A fragments (f16).
//
// codes: the 4 fragment bytes of one k-step (byte b -> register a[b]);
// scales: low byte = E4M3 scale of row g, high byte = scale of row g + 8.
// a[b] = E2M1 pair * scale, an exact f16 product: |E2M1| <= 6 and
// E4M3 in [2^-9, 448] give at most 6 significant bits in [2^-10, 2688], all
// f16 normals, so the tensor core sees the exact dequantised weight c.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void e2m1x4_to_f16x2(uint32_t w, uint32_t (&q)[4]) {
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
      "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
      "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
      : "=r"(q[0]), "=r"(q[1]), "=r"(q[2]), "=r"(q[3])
      : "r"(w));
}

__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two_bytes) {
  uint32_t r;
  uint16_t s = static_cast<uint16_t>(two_bytes);
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(s));
  return r;
}

__device__ __forceinline__ uint32_t hmul2_bcast_lo(uint32_t q, uint32_t s) {
  __half2 qq = *reinterpret_cast<__half2*>(&q);
  __half2 ss = *reinterpret_cast<__half2*>(&s);
  __half2 r = __hmul2(qq, __low2half2(ss));
  return *reinterpret_cast<uint32_t*>(&r);
}
__device__ __forceinline__ uint32_t hmul2_bcast_hi(uint32_t q, uint32_t s) {
  __half2 qq = *reinterpret_cast<__half2*>(&q);
  __half2 ss = *reinterpret_cast<__half2*>(&s);
  __half2 r = __hmul2(qq, __high2half2(ss));
  return *reinterpret_cast<uint32_t*>(&r);
}

// f16x2 holding two values exactly representable in bf16 -> bf16x2 (exact):
// the dequantised NVFP4 weights (at most 6 significant bits, in [2^-10, 2688]).
__device__ __forceinline__ uint32_t f16x2_to_bf16x2(uint32_t h) {
  const __half2 hv = *reinterpret_cast<const __half2*>(&h);
  const float2 f = __half22float2(hv);
  const __nv_bfloat162 b = __float22bfloat162_rn(f);
  return *reinterpret_cast<const uint32_t*>(&b);
}

// codes_word: the 4 fragment bytes of one k-step; sg, sg8: the 4-byte scale
// words of rows g and g + 8 in this k-group; ks selects the k-step's byte.
__device__ __forceinline__ void nvfp4_afrag(uint32_t codes_word, uint32_t sg, uint32_t sg8, int ks,
                                            uint32_t (&a)[4]) {
  const uint32_t pair = __byte_perm(sg, sg8, (uint32_t)ks | ((uint32_t)(ks + 4) << 4));
  const uint32_t s = e4m3x2_to_f16x2(pair);  // lo half: row g, hi half: row g + 8
  uint32_t q[4];
  e2m1x4_to_f16x2(codes_word, q);
  a[0] = hmul2_bcast_lo(q[0], s);
  a[1] = hmul2_bcast_hi(q[1], s);
  a[2] = hmul2_bcast_lo(q[2], s);
  a[3] = hmul2_bcast_hi(q[3], s);
}

// ---------------------------------------------------------------------------
// Activation fragments. Per token row, per k-group of 64 columns: 128 bytes,
// [t 4][ks 4][4 halves] with halves (2t, 2t+1, 2t+8, 2t+9) of the k-step, so
// thread (g, t) of mma.m16n8k16 reads its B fragments for 4 k-steps as 32
// contiguous bytes. Row strides in shared memory are padded by 16 bytes.
// ---------------------------------------------------------------------------
__host__ __device__ inline int frag_offset_elems(int col) {
  const int kg = col >> 6, ks = (col >> 4) & 3, c = col & 15;
  const int t = (c & 7) >> 1, idx = (c & 1) | ((c >> 3) << 1);
  return kg * 64 + t * 16 + ks * 4 + idx;
}

// Power-of-two prescale that maps the largest magnitude m into [2^14, 2^15),
// so values fit f16 without overflow and keep full precision down to 2^-29 m.
__device__ __forceinline__ int prescale_exp(float maxabs) {
  const int e = (int)((__float_as_uint(maxabs) >> 23) & 0xFF) - 127;
  int k = maxabs > 0.f ? 14 - e : 0;
  k = k > 126 ? 126 : (k < -126 ? -126 : k);
  return k;
}
__device__ __forceinline__ float exp2i(int k) { return __uint_as_float((uint32_t)(k + 127) << 23); }

__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// RMSNorm pieces (pre-norm sublayer), used identically by every kernel that
// normalises a row, so all of them derive bit-identical normalised
// activations: lane l owns the 16-byte chunks l, l + 32, ... of a row; its sum
// of squares runs over them in that order, the warp total is a butterfly (the
// same value in every lane), then 1 / sqrt(mean + eps) with IEEE square root
// and division, and each value becomes bf16((x * inv) * w); a row whose sum
// of squares overflows FP32 takes the scaled path below.
__device__ __forceinline__ float sumsq8(const uint4 u, float acc) {
  acc = fmaf(bf16lo(u.x), bf16lo(u.x), acc);
  acc = fmaf(bf16hi(u.x), bf16hi(u.x), acc);
  acc = fmaf(bf16lo(u.y), bf16lo(u.y), acc);
  acc = fmaf(bf16hi(u.y), bf16hi(u.y), acc);
  acc = fmaf(bf16lo(u.z), bf16lo(u.z), acc);
  acc = fmaf(bf16hi(u.z), bf16hi(u.z), acc);
  acc = fmaf(bf16lo(u.w), bf16lo(u.w), acc);
  acc = fmaf(bf16hi(u.w), bf16hi(u.w), acc);
  return acc;
}


__device__ __forceinline__ uint32_t norm2(uint32_t x, uint32_t w, float inv) {
  const __nv_bfloat162 r = __floats2bfloat162_rn((bf16lo(x) * inv) * bf16lo(w), (bf16hi(x) * inv) * bf16hi(w));
  return *reinterpret_cast<const uint32_t*>(&r);
}

__device__ __forceinline__ uint4 norm8(const uint4 x, const uint4 w, float inv) {
  return make_uint4(norm2(x.x, w.x, inv), norm2(x.y, w.y, inv), norm2(x.z, w.z, inv), norm2(x.w, w.w, inv));
}

// Largest finite FP32 value: a warp's sum of squares above it has overflowed.
constexpr float FP32_MAX = 3.40282347e38f;

// Rows whose sum of squares overflows FP32 (|r| beyond about 2^58; bf16
// reaches 2^128). Such a row is first scaled by an exact power of two
// pre = 2^-e (e from its largest magnitude), so that
//   1 / sqrt(mean(r^2) + eps) = pre / sqrt(mean((pre r)^2) + pre^2 eps)
// comes from a finite sum; each value becomes bf16(((r pre) inv) w). This path
// is out of line, so the common one carries none of its code.
__device__ __forceinline__ float absmax8(const uint4 u, float m) {
  const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int q = 0; q < 4; ++q) m = fmaxf(m, fmaxf(fabsf(bf16lo(w4[q])), fabsf(bf16hi(w4[q]))));
  return m;
}

// The factor inv (x) and the scale pre (y) of such a row: lane l re-reads its
// 16-byte chunks l, l + 32, ... (H / 256 of them) from shared memory or,
// written by an earlier kernel, through L2.
static __device__ __noinline__ float2 rms_factor_huge(const uint8_t* row, int row_in_smem, int lane, int H,
                                                      float eps) {
  const int nch = H / 256;
  float m = 0.f;
  for (int c = 0; c < nch; ++c) {
    const uint8_t* p = row + (lane + 32 * c) * 16;
    m = absmax8(row_in_smem ? lds128(p) : ld_cg_v4(p), m);
  }
  m = warp_max(m);
  int e = (int)((__float_as_uint(m) >> 23) & 0xFF) - 127;
  e = e < 0 ? 0 : (e > 120 ? 120 : e);
  const float pre = exp2i(-e);
  float acc = 0.f;
  for (int c = 0; c < nch; ++c) {
    const uint8_t* p = row + (lane + 32 * c) * 16;
    const uint4 u = row_in_smem ? lds128(p) : ld_cg_v4(p);
    const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
    for (int q = 0; q < 4; ++q) {
      const float a = bf16lo(w4[q]) * pre, b = bf16hi(w4[q]) * pre;
      acc = fmaf(a, a, acc);
      acc = fmaf(b, b, acc);
    }
  }
  const float ss = warp_sum(acc);
  return make_float2(1.0f / sqrtf(ss / (float)H + (eps * pre) * pre), pre);
}

// One chunk of such a row, normalised with f = rms_factor_huge(...).
static __device__ __noinline__ uint4 norm8_huge(const uint4 x, const uint4 w, const float2 f) {
  const uint32_t xs[4] = {x.x, x.y, x.z, x.w}, ws[4] = {w.x, w.y, w.z, w.w};
  uint32_t o[4];
  for (int q = 0; q < 4; ++q) {
    const __nv_bfloat162 r = __floats2bfloat162_rn(((bf16lo(xs[q]) * f.y) * f.x) * bf16lo(ws[q]),
                                                   ((bf16hi(xs[q]) * f.y) * f.x) * bf16hi(ws[q]));
    o[q] = *reinterpret_cast<const uint32_t*>(&r);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}


}  // namespace flint
