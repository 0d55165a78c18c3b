// Decode step of the Flint-style W4A16 MoE layer on sm_103a: three kernels
// chained with programmatic dependent launch (PDL), plus the dense GEMV.
//
//   k_stage_x     (x in pinned host memory only) copies x once into the
//                 workspace, where the other kernels read it.
//   k_router      logits = x Wr^T (FP32 accumulation), optionally on the
//                 RMS-normalised x; a block's router rows arrive by one bulk
//                 copy before the wait, its warps split the tokens.
//   k_gateup      persistent, one block per SM; warp groups take units (slot,
//                 8 intermediate rows). A slot is one of the always-on shared
//                 experts or one of the distinct experts the batch selected
//                 (ascending id). Every block derives the selection itself from
//                 the 1 KB-per-token logits, streams its units' packed gate/up
//                 tiles into shared memory, dequantises into mma fragments and
//                 writes h = bf16(silu(g) * u).
//   k_down_items  (up to 8 tokens) / k_down (more): one block per 16 output
//                 rows; routes and prefetches its down tiles *before* waiting
//                 for k_gateup, then, once h exists, multiplies and accumulates
//                 w * y per warp, adds the warps in a fixed order and writes
//                 out = bf16(sum) (plus the residual for the pre-norm block).
//   k_gemv        dense y = x W^T on the same packed layout.
//
// Launch order inside a layer and across layers (same stream):
//   k_router waits for the previous layer, then lets k_gateup launch;
//   k_gateup fetches the shared expert before its wait and lets the down kernel
//   launch right after its wait (so the router has finished when it starts);
//   the down kernel routes and fetches its weights while k_gateup runs, and
//   waits only for h. Each kernel's routing-independent bytes therefore move
//   while the previous kernel runs.
//
// "Day-0 Support for Flint on vLLM", section "Optimisation": the small-batch
// MoE kernels read only the selected experts' weights; routing and the expert
// combine are fused into the adjacent GEMV kernels; every kernel uses PDL so it
// loads its weights while the previous kernel still runs.
#include <algorithm>
#include <atomic>
#include <cmath>

#include "common.cuh"
#include "flint_gemv.h"

namespace flint {

struct DecodeArgs {
  int H, I, E, S, k, B, fmt, renorm;
  float routed_scale;
  const uint16_t* x;
  uint16_t* out;
  const uint16_t* router;
  const float* bias;
  const uint8_t* packed;
  const float* globals;
  Layout L;
  uint8_t* ws;
  WsLayout W;
  int gu_nb;      // gate/up weight buffers in flight per warp group (1..3)
  int trace_seq;  // decode call number, used only by trace builds
  // Pre-norm sublayer: x is the residual stream, normalised (RMSNorm with
  // weight gamma) on the way in, added to the layer output on the way out.
  int prenorm;
  const uint16_t* gamma;
  float eps;
  int router_epb;  // experts per router block; the block's warps split its tokens into nw / epb groups
  int dn_nbuf;     // down tiles in flight per warp
  int dn_hcap;     // h rows the down kernel stages at a time
};

__device__ __forceinline__ int* ws_hdr(const DecodeArgs& a) { return reinterpret_cast<int*>(a.ws); }
__device__ __forceinline__ float* ws_logits(const DecodeArgs& a) { return reinterpret_cast<float*>(a.ws + a.W.logits); }
__device__ __forceinline__ uint32_t* ws_keys(const DecodeArgs& a) { return reinterpret_cast<uint32_t*>(a.ws + a.W.keys); }
__device__ __forceinline__ int* ws_topk_idx(const DecodeArgs& a) { return reinterpret_cast<int*>(a.ws + a.W.topk_idx); }
__device__ __forceinline__ float* ws_topk_w(const DecodeArgs& a) { return reinterpret_cast<float*>(a.ws + a.W.topk_w); }
__device__ __forceinline__ unsigned* ws_hmax(const DecodeArgs& a) { return reinterpret_cast<unsigned*>(a.ws + a.W.hmax); }
__device__ __forceinline__ uint16_t* ws_h(const DecodeArgs& a) { return reinterpret_cast<uint16_t*>(a.ws + a.W.h); }
__device__ __forceinline__ uint16_t* ws_h16(const DecodeArgs& a) { return reinterpret_cast<uint16_t*>(a.ws + a.W.h16); }

// ---------------------------------------------------------------------------
// Optional phase trace (built with -DFLINT_MOE_TRACE): per decode call, the
// earliest and latest %globaltimer over all blocks at each phase boundary of
// each kernel. Off by default; it adds no work to the decode itself.
// ---------------------------------------------------------------------------
#ifdef FLINT_MOE_TRACE
constexpr int TRACE_CALLS = 64, TRACE_EVENTS = 24;
__device__ unsigned long long g_trace[TRACE_CALLS][TRACE_EVENTS][2];
#define FLINT_TRACE(a, ev)                                                          \
  do {                                                                              \
    if (threadIdx.x == 0 && (ev) >= 0) {                                            \
      const unsigned long long t_ = global_ns();                                    \
      atomicMin(&g_trace[(a).trace_seq % TRACE_CALLS][(ev)][0], t_);                \
      atomicMax(&g_trace[(a).trace_seq % TRACE_CALLS][(ev)][1], t_);                \
    }                                                                               \
  } while (0)
#else
#define FLINT_TRACE(a, ev) \
  do {                     \
  } while (0)
#endif

__device__ __forceinline__ float dot8_bf16(const uint4 w, const uint4 x, float acc) {
  acc = fmaf(bf16lo(w.x), bf16lo(x.x), acc);
  acc = fmaf(bf16hi(w.x), bf16hi(x.x), acc);
  acc = fmaf(bf16lo(w.y), bf16lo(x.y), acc);
  acc = fmaf(bf16hi(w.y), bf16hi(x.y), acc);
  acc = fmaf(bf16lo(w.z), bf16lo(x.z), acc);
  acc = fmaf(bf16hi(w.z), bf16hi(x.z), acc);
  acc = fmaf(bf16lo(w.w), bf16lo(x.w), acc);
  acc = fmaf(bf16hi(w.w), bf16hi(x.w), acc);
  return acc;
}

// ===========================================================================
// Routing: sigmoid, top-k, renormalised weights, slots and rows. Computed by
// every block that needs it from the logits in the workspace; the result is
// a deterministic function of the logits, so all blocks agree.
// ===========================================================================
constexpr int MAX_WARPS = 20;
constexpr int USED_WORDS = MAX_EXPERTS / 32;

// Routing result in shared memory. Slots are the S shared experts, then the
// distinct selected experts in ascending id; slot s holds all B token rows
// s * B .. s * B + B - 1 of h (a token that did not select the expert has a
// row that is computed and never combined). The r-th selected expert is the
// r-th set bit of `used`, which the selection also lists in slot_e, and the
// tokens of expert e are the bits of mask[e].
struct __align__(16) RouteSmem {
  uint32_t mask[MAX_EXPERTS];       // bit t: token t selected expert e
  uint32_t used[USED_WORDS];        // bit e % 32 of word e / 32: some token selected e
  int idx[MAX_BATCH * MAX_TOPK];    // full routing only: per token, (key desc, index asc)
  float w[MAX_BATCH * MAX_TOPK];
  int sel_e[MAX_WARPS][MAX_TOPK];   // per warp scratch for the token being routed
  float sel_l[MAX_WARPS][MAX_TOPK];
  uint16_t slot_e[MAX_EXPERTS];     // expert of routed slot S + r (built by route_select)
};

// Clears the selection bitmaps; the caller synchronises the block afterwards.
// Needs nothing from the previous kernel, so it runs before the dependency wait.
__device__ __forceinline__ void route_clear(RouteSmem& R, int E) {
  for (int i = threadIdx.x; i < E; i += blockDim.x) R.mask[i] = 0u;
  if (threadIdx.x < USED_WORDS) R.used[threadIdx.x] = 0u;
}

// Order-preserving map of a float key to an unsigned integer; 0 means "none".
__device__ __forceinline__ uint32_t ordered_key(float f) {
  const uint32_t b = __float_as_uint(f);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// Inverse of ordered_key.
__device__ __forceinline__ float unordered_key(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// 1 / y rounded to nearest for y in [1, 2^125): the hardware approximation
// (max error 1 ulp) refined by one Newton-Raphson step r + r (1 - y r) with
// fused multiply-adds. An exhaustive GPU check over every FP32 y in that range
// found it equal, bit for bit, to the IEEE quotient 1.0f / y, at a fraction of
// the division's cost (no slow-path branch, so eight of them interleave).
__device__ __forceinline__ float rcp_nr(float y) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(y));
  return fmaf(r, fmaf(-y, r, 1.0f), r);
}
constexpr float RCP_NR_MAX = 0x1p125f;

// The IEEE quotient 1 / y, out of line, for values outside rcp_nr's range:
// the common path then carries none of the division's code.
__device__ __noinline__ float rcp_ieee(float y) { return 1.0f / y; }
__device__ __noinline__ float div_ieee(float x, float y) { return x / y; }

// Routing score 1 / (1 + e^-l) in FP32: the IEEE quotient, computed through
// rcp_nr except for l below about -86.6 (y >= 2^125) or NaN.
__device__ __forceinline__ float sigmoid_f32(float l) {
  const float y = 1.0f + expf(-l);
  return y < RCP_NR_MAX ? rcp_nr(y) : rcp_ieee(y);
}

// Key of expert e: sigmoid of its logit plus its selection bias, in FP32.
__device__ __forceinline__ float route_key(float l, const float* bias, int e) {
  const float s = sigmoid_f32(l);
  return bias ? s + __ldg(bias + e) : s;
}

// Publishes one token's k winners (lanes 0..k-1 hold my_e) and, for full
// routing, their renormalised weights in (key desc, index asc) order. Lane r
// holds the r-th winner in selection order, which is (key desc, index asc).
__device__ __forceinline__ void route_publish(const DecodeArgs& a, RouteSmem& R, int t, int lane, int my_e, float s,
                                              bool full, bool write_debug) {
  const bool act = lane < a.k;
  if (act) {
    atomicOr(&R.mask[my_e], 1u << t);
    atomicOr(&R.used[my_e >> 5], 1u << (my_e & 31));
  }
  if (!full) return;
  // Sum of the k scores in selection order (a fixed order: deterministic).
  float ssum = 0.f;
  for (int q = 0; q < a.k; ++q) ssum += __shfl_sync(0xffffffffu, s, q);
  if (act) {
    float w = a.renorm ? s / ssum : s;
    w *= a.routed_scale;
    R.idx[t * a.k + lane] = my_e;
    R.w[t * a.k + lane] = w;
    if (write_debug) {
      ws_topk_idx(a)[t * a.k + lane] = my_e;
      ws_topk_w(a)[t * a.k + lane] = w;
    }
  }
}

// Arg-max of two (key, index) pairs whose indices increase left to right: the
// right one wins only when strictly greater, so equal keys keep the lower index.
__device__ __forceinline__ void argmax2(uint32_t k0, int j0, uint32_t k1, int j1, uint32_t& k, int& j) {
  const bool hi = k1 > k0;
  k = hi ? k1 : k0;
  j = hi ? j1 : j0;
}

// Top-k of one token by one warp, any E <= 512: lane l holds experts l, l+32,
// ...; k rounds of a 16-key arg-max tree and two warp reductions.
__device__ void topk_token_wide(const DecodeArgs& a, int t, int warp, int lane, RouteSmem& R, bool full,
                                bool write_debug, int tb, const float* logits) {
  constexpr int EPL = MAX_EXPERTS / 32;
  static_assert(EPL == 16, "the arg-max tree below is written for 16 keys per lane");
  const float* lg = logits + (size_t)t * a.E;
  float lv[EPL];
#pragma unroll
  for (int j = 0; j < EPL; ++j) lv[j] = 32 * j < a.E ? __ldcg(lg + min(lane + 32 * j, a.E - 1)) : 0.f;
  uint32_t key[EPL];
#pragma unroll
  for (int j = 0; j < EPL; ++j) {
    const int e = lane + 32 * j;
    key[j] = e < a.E ? ordered_key(route_key(lv[j], a.bias, e)) : 0u;
  }
  if (t == 0) FLINT_TRACE(a, tb);
  for (int r = 0; r < a.k; ++r) {
    uint32_t k8[8], k4[4], k2[2], best;
    int j8[8], j4[4], j2[2], bj;
#pragma unroll
    for (int p = 0; p < 8; ++p) argmax2(key[2 * p], 2 * p, key[2 * p + 1], 2 * p + 1, k8[p], j8[p]);
#pragma unroll
    for (int p = 0; p < 4; ++p) argmax2(k8[2 * p], j8[2 * p], k8[2 * p + 1], j8[2 * p + 1], k4[p], j4[p]);
#pragma unroll
    for (int p = 0; p < 2; ++p) argmax2(k4[2 * p], j4[2 * p], k4[2 * p + 1], j4[2 * p + 1], k2[p], j2[p]);
    argmax2(k2[0], j2[0], k2[1], j2[1], best, bj);
    const uint32_t wmax = __reduce_max_sync(0xffffffffu, best);
    const int cand = (best == wmax && best != 0u) ? lane + 32 * bj : 0x7fffffff;
    int win = __reduce_min_sync(0xffffffffu, cand);
    if (win == 0x7fffffff) {  // only with non-finite logits: keep every index in range
      if (lane == 0) atomicOr(ws_hdr(a) + HDR_STATUS, FLINT_MOE_DEV_ERR_SLOTS);
      win = r;
    }
    if (lane == (win & 31)) {
      const int wj = win >> 5;
      float l = 0.f;
#pragma unroll
      for (int j = 0; j < EPL; ++j)
        if (j == wj) {
          l = lv[j];
          key[j] = 0u;
        }
      R.sel_e[warp][r] = win;
      R.sel_l[warp][r] = l;
    }
  }
  __syncwarp();
  if (t == 0) FLINT_TRACE(a, tb < 0 ? -1 : tb + 1);
  const bool act = lane < a.k;
  const int my_e = act ? R.sel_e[warp][lane] : 0;
  const float s = act ? sigmoid_f32(R.sel_l[warp][lane]) : 0.f;
  __syncwarp();  // the warp's scratch is reused by its next token
  route_publish(a, R, t, lane, my_e, s, full, write_debug);
  if (t == 0) FLINT_TRACE(a, tb < 0 ? -1 : tb + 2);
}

__device__ __forceinline__ void ce_desc(uint64_t& x, uint64_t& y) {  // x >= y afterwards
  const uint64_t hi = x > y ? x : y, lo = x > y ? y : x;
  x = hi;
  y = lo;
}

// Top-k of one token by one warp for E <= 256 (the Flint shape), the same
// result as topk_token_wide with a fraction of the instructions. Lane l holds
// experts 8l .. 8l+7, each as one 64-bit word (order-preserving key << 32 |
// 0xFFFF - e, so a larger word is a larger key or, on equal keys, a lower
// index), sorts them once with a 19-comparator network, and each round is two
// warp reductions and a shift of the winning lane's list. Winners come out in
// (key desc, index asc) order.
__device__ void topk_token_narrow(const DecodeArgs& a, int t, int warp, int lane, RouteSmem& R, bool full,
                                  bool write_debug, int tb, const float* logits) {
  constexpr int EPL = 8;
  const float* lg = logits + (size_t)t * a.E;
  const uint32_t* kt = ws_keys(a) + (size_t)t * a.E;  // keys the router derived from the logits
  const int e0 = lane * EPL;
  uint32_t kv[EPL];
  if (a.E == 256) {  // 32 contiguous, 16-byte aligned bytes per lane
    const uint4 p = ld_cg_v4(kt + e0), q = ld_cg_v4(kt + e0 + 4);
    kv[0] = p.x; kv[1] = p.y; kv[2] = p.z; kv[3] = p.w; kv[4] = q.x; kv[5] = q.y; kv[6] = q.z; kv[7] = q.w;
  } else {
#pragma unroll
    for (int j = 0; j < EPL; ++j) kv[j] = __ldcg(kt + min(e0 + j, a.E - 1));  // clamped: all issue at once
  }
#ifdef FLINT_MOE_TRACE
  if (t == 0 && tb >= 0 && kv[0] != 1u && kv[7] != 1u) {
    FLINT_TRACE(a, 4);  // keys arrived (the condition makes the timer wait for them)
    FLINT_TRACE(a, 5);
  }
#endif
  // (key, complemented index) words: larger word = larger key, then lower index.
  uint64_t v[EPL];
#pragma unroll
  for (int j = 0; j < EPL; ++j) {
    const int e = e0 + j;
    v[j] = e < a.E ? ((uint64_t)kv[j] << 32) | (uint32_t)(0xFFFF - e) : 0ull;
  }
  ce_desc(v[0], v[2]); ce_desc(v[1], v[3]); ce_desc(v[4], v[6]); ce_desc(v[5], v[7]);
  ce_desc(v[0], v[4]); ce_desc(v[1], v[5]); ce_desc(v[2], v[6]); ce_desc(v[3], v[7]);
  ce_desc(v[0], v[1]); ce_desc(v[2], v[3]); ce_desc(v[4], v[5]); ce_desc(v[6], v[7]);
  ce_desc(v[2], v[4]); ce_desc(v[3], v[5]);
  ce_desc(v[1], v[4]); ce_desc(v[3], v[6]);
  ce_desc(v[1], v[2]); ce_desc(v[3], v[4]); ce_desc(v[5], v[6]);
  if (t == 0 && v[0] != 1ull) FLINT_TRACE(a, tb);
  uint32_t my_hi = 0u, my_lo = 0xFFFFu;
  for (int r = 0; r < a.k; ++r) {
    const uint32_t hi = (uint32_t)(v[0] >> 32), lo = (uint32_t)v[0];
    const uint32_t whi = __reduce_max_sync(0xffffffffu, hi);
    const uint32_t wlo = __reduce_max_sync(0xffffffffu, hi == whi ? lo : 0u);
    if (hi == whi && lo == wlo) {  // the winning lane drops its head
#pragma unroll
      for (int j = 0; j < EPL - 1; ++j) v[j] = v[j + 1];
      v[EPL - 1] = 0ull;
    }
    if (lane == r) {
      my_hi = whi;
      my_lo = wlo;
    }
  }
  if (t == 0) FLINT_TRACE(a, tb < 0 ? -1 : tb + 1);
  const bool act = lane < a.k;
  int my_e = min(0xFFFF - (int)my_lo, a.E - 1);
  if (act && my_hi == 0u) {  // fewer than k finite keys: only with non-finite logits
    atomicOr(ws_hdr(a) + HDR_STATUS, FLINT_MOE_DEV_ERR_SLOTS);
    my_e = lane;
  }
  float s = 0.f;
  if (full && act) s = a.bias ? sigmoid_f32(__ldcg(lg + my_e)) : unordered_key(my_hi);  // key = score unbiased
  route_publish(a, R, t, lane, my_e, s, full, write_debug);
  if (t == 0) FLINT_TRACE(a, tb < 0 ? -1 : tb + 2);
}

// Rank of selected expert e among the selected experts (its routed slot is
// S + rank): the set bits of `used` below e.
template <bool NARROW>
__device__ __forceinline__ int used_rank(const DecodeArgs& a, const RouteSmem& R, int e) {
  const int w = e >> 5;
  int r = __popc(R.used[w] & ((1u << (e & 31)) - 1u));
  if (NARROW) {  // 8 words, loaded at once
#pragma unroll
    for (int q = 0; q < 8; ++q)
      if (q < w) r += __popc(R.used[q]);
  } else {
    for (int q = 0; q < w; ++q) r += __popc(R.used[q]);
  }
  return r;
}

// Whole block, after route_clear and a barrier: selects every token's experts
// (one warp per token) from logits [B][E] and ends with a barrier. Without
// `full` only the selection bitmaps are built; with it also the weights. tb:
// first trace event id, or -1.
// NARROW: the kernel was instantiated for the Flint shape (E = 256 experts,
// hidden H = 2048, intermediate I = 512, top-6, one shared expert), so it
// carries only the narrow top-k and the short-row staging, with the sizes
// known at compile time (a kernel's cold code still costs instruction
// fetches on this latency-bound path, and its index arithmetic becomes
// shifts and unrolled loops).
template <bool NARROW>
__device__ __forceinline__ DecodeArgs flint_shape(const DecodeArgs& a_in) {
  DecodeArgs a = a_in;
  if (NARROW) {
    a.H = 2048;
    a.E = 256;
    a.I = 512;
    a.k = 6;
    a.S = 1;
  }
  return a;
}

template <bool NARROW>
__device__ void route_select(const DecodeArgs& a, RouteSmem& R, bool full, bool write_debug, int tb,
                             const float* logits) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  if (NARROW || a.E <= 256) {
    for (int t = warp; t < a.B; t += nw) topk_token_narrow(a, t, warp, lane, R, full, write_debug, tb, logits);
  } else {
    for (int t = warp; t < a.B; t += nw) topk_token_wide(a, t, warp, lane, R, full, write_debug, tb, logits);
  }
  __syncthreads();
  // The slot table: routed slot S + r is the r-th set bit of `used`.
  for (int e = threadIdx.x; e < a.E; e += blockDim.x)
    if ((R.used[e >> 5] >> (e & 31)) & 1u) R.slot_e[used_rank<NARROW>(a, R, e)] = (uint16_t)e;
  __syncthreads();
  FLINT_TRACE(a, tb < 0 ? -1 : 14);
}

// Position of the n-th (from 0) set bit of m; n < popc(m).
__device__ __forceinline__ int nth_set_bit(uint32_t m, int n) {
  int pos = 0;
#pragma unroll
  for (int width = 16; width >= 1; width >>= 1) {
    const uint32_t low = m & ((1u << width) - 1u);
    const int c = __popc(low);
    if (n >= c) {
      n -= c;
      m >>= width;
      pos += width;
    } else {
      m = low;
    }
  }
  return pos;
}

// Number of slots: the shared experts plus the distinct selected experts.
__device__ __forceinline__ int route_slots(const DecodeArgs& a, const RouteSmem& R) {
  int c = a.S;
  for (int w = 0; w < (a.E + 31) >> 5; ++w) c += __popc(R.used[w]);
  return c;
}

struct SlotInfo {
  int expert;      // packed expert index (shared experts follow the E routed ones)
  uint32_t tmask;  // tokens whose output takes this expert
};

__device__ __forceinline__ SlotInfo slot_info(const DecodeArgs& a, const RouteSmem& R, int slot) {
  SlotInfo si;
  if (slot < a.S) {
    si.expert = a.E + slot;
    si.tmask = a.B >= 32 ? 0xFFFFFFFFu : (1u << a.B) - 1u;
    return si;
  }
  si.expert = R.slot_e[slot - a.S];  // slot < route_slots
  si.tmask = R.mask[si.expert];
  return si;
}

// ===========================================================================
// K1: router GEMV (logits in the workspace); also clears the per-row |h|
// maxima that k_gateup accumulates. Block b computes experts epb*b ..
// epb*b + epb - 1 (epb = 4, 2 or 1 as the batch grows); warp w takes expert
// w % epb for tokens w / epb, w / epb + 4 / epb, ..., so every warp has about
// as many dot products at any batch size. The block's router rows are
// contiguous: one bulk copy brings them into shared memory before the
// dependency wait (they do not depend on x).
// NCH: 16-byte chunks of a router row per lane (H / 256).
// ===========================================================================
// NT tokens' dot products with one router row: lane l takes 16-byte chunks
// l, l + 32, ...; all NT sums are independent, so their latencies overlap.
// Tokens t0, t0 + ts, ... (NT of them) of the x chunk.
template <int NCH, int NT>
__device__ __forceinline__ void router_dots(const uint8_t* wrow, const uint8_t* xsm, int H, int lane, float* lg,
                                            uint32_t* kc, float bias_e, int E, int e, int t0, int ts, bool dry) {
  float acc[NT];
#pragma unroll
  for (int t = 0; t < NT; ++t) acc[t] = 0.f;
#pragma unroll
  for (int c = 0; c < NCH; ++c) {
    const uint4 w = lds128(wrow + (lane + 32 * c) * 16);
#pragma unroll
    for (int t = 0; t < NT; ++t)
      acc[t] = dot8_bf16(w, lds128(xsm + (size_t)(t0 + t * ts) * H * 2 + (lane + 32 * c) * 16), acc[t]);
  }
  // Lane t stores token t's logit and its selection key (sigmoid + bias, in
  // the order-preserving unsigned form the top-k compares), so the blocks that
  // route after the dependency wait only compare.
// The key is computed in the warm-up pass too (only the stores are skipped),
  // so its code is hot when the real pass runs.
#pragma unroll
  for (int t = 0; t < NT; ++t) {
    const float v = warp_sum(acc[t]);
    if (lane == t) {
      const uint32_t key = ordered_key(sigmoid_f32(v) + bias_e);  // bias_e: 0 without a selection bias
      if (!dry) {
        lg[(t0 + t * ts) * E + e] = v;
        kc[(t0 + t * ts) * E + e] = key;
      }
    }
  }
}

// One token's logit of expert e for the pre-norm block of 2 tokens: the
// warp normalises the token's row (in shared memory, as loaded) itself, the
// same steps in the same order as every kernel that normalises a row, and
// feeds each normalised chunk to the dot product as it goes; no warp writes
// the row back, so no barrier separates the norm from the dot products (the
// block's warps each do this for their own expert).
template <int NCH>
__device__ __forceinline__ void router_dot_normed(const uint8_t* wrow, const uint8_t* xrow, const uint8_t* gsm, int H,
                                                  float eps, int lane, float* lg, uint32_t* kc, float bias_e, int E,
                                                  int e, int t, bool dry) {
  uint4 xv[NCH];
  float part = 0.f;
#pragma unroll
  for (int c = 0; c < NCH; ++c) {
    xv[c] = lds128(xrow + (lane + 32 * c) * 16);
    part = sumsq8(xv[c], part);
  }
  const float ss = warp_sum(part);
  float acc = 0.f;
  if (ss <= FP32_MAX) {
    const float inv = 1.0f / sqrtf(ss / (float)H + eps);
#pragma unroll
    for (int c = 0; c < NCH; ++c) {
      const int off = (lane + 32 * c) * 16;
      acc = dot8_bf16(lds128(wrow + off), norm8(xv[c], lds128(gsm + off), inv), acc);
    }
  } else {  // the sum of squares overflowed: the scaled path
    const float2 f = rms_factor_huge(xrow, 1, lane, H, eps);
    for (int c = 0; c < NCH; ++c) {
      const int off = (lane + 32 * c) * 16;
      acc = dot8_bf16(lds128(wrow + off), norm8_huge(xv[c], lds128(gsm + off), f), acc);
    }
  }
  const float v = warp_sum(acc);
  if (lane == 0) {
    const uint32_t key = ordered_key(sigmoid_f32(v) + bias_e);  // bias_e: 0 without a selection bias
    if (!dry) {
      lg[t * E + e] = v;
      kc[t * E + e] = key;
    }
  }
}

// Pre-norm calls of NORM_KERNEL_MIN_B tokens or more: one warp per row
// computes the RMSNorm once (the same steps, in the same order, as every
// kernel that normalises a row: bit-identical results) and writes the
// normalised bf16 rows to the workspace, which the router and gate/up kernels
// then read as plain activations; otherwise each router block normalises
// every row of the batch itself, on the critical path. Measured on the
// 47-layer pre-norm stack (us per layer): 8 tokens 29.6 -> 29.0, 16 59.9 ->
// 55.4, 32 140.8 -> 126.8; below 8 tokens the extra launch costs more
// (4 tokens 21.3 -> 22.1, 1 token 10.8 -> 12.1).
constexpr int NORM_KERNEL_MIN_B = 8;

__global__ void __launch_bounds__(128) k_norm_x(const DecodeArgs a) {
  pdl_wait();  // x is the previous layer's output
  pdl_trigger();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * 4 + warp;
  if (t >= a.B) return;
  const uint8_t* row = reinterpret_cast<const uint8_t*>(a.x + (size_t)t * a.H);
  uint8_t* dst = a.ws + a.W.xn + (size_t)t * a.H * 2;
  const uint8_t* g8 = reinterpret_cast<const uint8_t*>(a.gamma);
  const int nch = a.H / 256;  // 16-byte chunks per lane
  float part = 0.f;
#pragma unroll 8
  for (int c = 0; c < nch; ++c) part = sumsq8(ld_cg_v4(row + (lane + 32 * c) * 16), part);
  const float ss = warp_sum(part);
  if (ss <= FP32_MAX) {
    const float inv = 1.0f / sqrtf(ss / (float)a.H + a.eps);
#pragma unroll 8
    for (int c = 0; c < nch; ++c) {
      const int off = (lane + 32 * c) * 16;
      *reinterpret_cast<uint4*>(dst + off) =
          norm8(ld_cg_v4(row + off), __ldg(reinterpret_cast<const uint4*>(g8 + off)), inv);
    }
  } else {  // the sum of squares overflowed: the scaled path
    const float2 f = rms_factor_huge(row, 0, lane, a.H, a.eps);
    for (int c = 0; c < nch; ++c) {
      const int off = (lane + 32 * c) * 16;
      *reinterpret_cast<uint4*>(dst + off) =
          norm8_huge(ld_cg_v4(row + off), __ldg(reinterpret_cast<const uint4*>(g8 + off)), f);
    }
  }
}

// Calls whose x is pinned host memory: its rows are copied once, by this
// kernel, into the workspace, and the layer's kernels read that copy (the
// 16-byte loads cross the host link once, not once per block that needs x).
__global__ void __launch_bounds__(256) k_stage_x(const DecodeArgs a) {
  pdl_wait();  // x may be written by earlier work in the stream
  pdl_trigger();
  const int n = a.B * a.H / 8;  // 16-byte words
  uint4* dst = reinterpret_cast<uint4*>(a.ws + a.W.xs);
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x)
    dst[i] = ld_cg_v4(reinterpret_cast<const uint8_t*>(a.x) + (size_t)i * 16);
}

template <int NCH, int PRE>
__global__ void __launch_bounds__(512) k_router(DecodeArgs a) {
  const int prenorm = PRE < 0 ? a.prenorm : PRE;
  // 2 pre-norm tokens normalised inside the dot products (rows of up to 2048:
  // a lane keeps its NCH chunks in registers)
  constexpr bool FUSED_NORM2 = NCH <= 8;
  extern __shared__ __align__(128) uint8_t dsm[];  // router rows [4][H], norm weight [H], x chunk [<= 8][H]
  __shared__ __align__(8) uint64_t bars[2];        // 0: router rows, 1: x
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nw = blockDim.x >> 5;
  const int epb = a.router_epb, G = nw / epb;  // experts per block, token groups
  const int e0 = blockIdx.x * epb, e = e0 + warp % epb, tg = warp / epb;
  const int nrows = min(epb, a.E - e0);
  uint8_t* wsm = dsm;
  uint8_t* gsm = dsm + (size_t)epb * a.H * 2;
  uint8_t* xsm = gsm + (size_t)a.H * 2;
  FLINT_TRACE(a, 0);
  if (threadIdx.x == 0) {
    mbar_init(&bars[0], 1);
    mbar_init(&bars[1], 1);
    fence_mbar_init();
    const uint32_t bytes = (uint32_t)nrows * a.H * 2;
    mbar_arrive_expect_tx(&bars[0], bytes + (prenorm ? (uint32_t)a.H * 2 : 0u));
    bulk_g2s(wsm, a.router + (size_t)e0 * a.H, bytes, &bars[0]);
    if (prenorm) bulk_g2s(gsm, a.gamma, (uint32_t)a.H * 2, &bars[0]);
  }
  // Two passes at one call site: a dry one on zeroed activations before the
  // dependency wait (no stores), which brings the dot-product code into this
  // SM's instruction caches, then the real one on x.
  int* status = ws_hdr(a) + HDR_STATUS;
  float* lg = ws_logits(a);
  const uint8_t* wrow = wsm + (size_t)(warp % epb) * a.H * 2;
  // the selection bias of this warp's expert, read before the dependency wait
  const float bias_e = a.bias && e < a.E ? __ldg(a.bias + e) : 0.f;
  {
    const int n = (a.B < 8 ? a.B : 8) * a.H / 8;  // 16-byte words of the first x chunk
    for (int i = threadIdx.x; i < n; i += blockDim.x) reinterpret_cast<uint4*>(xsm)[i] = make_uint4(0, 0, 0, 0);
  }
  __syncthreads();  // the barriers are initialised (thread 0) before any thread waits on them
  const bool okw = mbar_wait(&bars[0], 0, status);
  uint32_t phase = 0;
  bool ok = okw;
#pragma unroll 1
  for (int pass = 0; pass < 2 && ok; ++pass) {
    const bool dry = pass == 0;
    if (!dry) {
      pdl_wait();  // x is the previous kernel's output
      pdl_trigger();
      FLINT_TRACE(a, 1);
      if (blockIdx.x == 0) {
        for (int i = threadIdx.x; i < a.W.max_slots * a.B; i += blockDim.x) ws_hmax(a)[i] = 0u;
        if (threadIdx.x == 0) ws_hdr(a)[HDR_HBIG] = 0;
      }
    }
    for (int t0 = 0; t0 < a.B; t0 += 8) {
      const int nt = min(8, a.B - t0);
      if (!dry) {
        if (threadIdx.x == 0) {
          const uint32_t bytes = (uint32_t)nt * a.H * 2;
          mbar_arrive_expect_tx(&bars[1], bytes);
          bulk_g2s(xsm, a.x + (size_t)t0 * a.H, bytes, &bars[1]);
        }
        ok = __syncthreads_and(mbar_wait(&bars[1], phase, status));  // block-uniform
        phase ^= 1;
        if (!ok) break;
        FLINT_TRACE(a, 2);
        // RMSNorm of the chunk's rows, in place (8 and more tokens arrive
        // normalised by k_norm_x); 2 tokens: inside the dot products, which
        // measured faster there (pre-norm stack 16.8 -> 16.2 us per layer) but
        // not at 1 token (10.8 -> 11.3)
        if (prenorm && (nt != 2 || !FUSED_NORM2)) {
          for (int t = warp; t < nt; t += nw) {
            uint8_t* row = xsm + (size_t)t * a.H * 2;
            float part = 0.f;
#pragma unroll
            for (int c = 0; c < NCH; ++c) part = sumsq8(lds128(row + (lane + 32 * c) * 16), part);
            const float ss = warp_sum(part);
            if (ss <= FP32_MAX) {
              const float inv = 1.0f / sqrtf(ss / (float)a.H + a.eps);
#pragma unroll
              for (int c = 0; c < NCH; ++c) {
                const int off = (lane + 32 * c) * 16;
                *reinterpret_cast<uint4*>(row + off) = norm8(lds128(row + off), lds128(gsm + off), inv);
              }
            } else {  // the sum of squares overflowed: the scaled path (the whole row is read first)
              const float2 f = rms_factor_huge(row, 1, lane, a.H, a.eps);
              for (int c = 0; c < NCH; ++c) {
                const int off = (lane + 32 * c) * 16;
                *reinterpret_cast<uint4*>(row + off) = norm8_huge(lds128(row + off), lds128(gsm + off), f);
              }
            }
          }
          __syncthreads();
        }
      }
      const int ntw = tg < nt ? (nt - tg + G - 1) / G : 0;  // this warp's tokens in the chunk
      if (e < a.E && ntw > 0) {
        float* lgc = lg + (size_t)t0 * a.E;
        uint32_t* kcc = ws_keys(a) + (size_t)t0 * a.E;
        // One code path per token count, no predicated-off work. A warp has at
        // most 2 tokens of a chunk (at least 4 token groups from 3 tokens on).
        bool done = false;
        if constexpr (FUSED_NORM2) {
          if (prenorm && nt == 2) {  // one token per warp
            router_dot_normed<NCH>(wrow, xsm + (size_t)tg * a.H * 2, gsm, a.H, a.eps, lane, lgc, kcc, bias_e, a.E,
                                   e, tg, dry);
            done = true;
          }
        }
        if (done) {
        } else if (ntw == 1)
          router_dots<NCH, 1>(wrow, xsm, a.H, lane, lgc, kcc, bias_e, a.E, e, tg, G, dry);
        else
          router_dots<NCH, 2>(wrow, xsm, a.H, lane, lgc, kcc, bias_e, a.E, e, tg, G, dry);
        if (!dry) FLINT_TRACE(a, 7);
      }
      fence_proxy_async();  // the zeroing stores and these reads come before the copy into the buffer
      __syncthreads();      // the x chunk buffer is reused by the next copy
      if (dry) break;       // one chunk warms the code
    }
  }
  if (!okw) mbar_drain(&bars[0], 0);
  FLINT_TRACE(a, 3);
}

// One k-group (64 columns) of a 16-row tile against NTMAX token tiles.
// Even and odd k-groups accumulate into separate registers (cs) so that
// consecutive mma.sync need not wait for one another. BF16B: the token
// fragments are bf16 (the NVFP4 weights, exact in f16, are converted to bf16
// exactly), so bf16 activations need no prescale or conversion.
template <int FMT, int NTMAX, bool BF16B = false>
__device__ __forceinline__ void tile_kgroup(const uint8_t* kp, const uint4 (&bx)[NTMAX][2], int nt_used, int lane,
                                            float (&acc)[NTMAX][4]) {
  const int g = lane >> 2;
  if (FMT == FLINT_MOE_NVFP4) {
    const uint4 codes = lds128(kp + lane * 16);
    const uint32_t sg = lds32(kp + KG_CODE_BYTES + g * 4);
    const uint32_t sg8 = lds32(kp + KG_CODE_BYTES + (g + 8) * 4);
    const uint32_t cw[4] = {codes.x, codes.y, codes.z, codes.w};
#pragma unroll
    for (int ks = 0; ks < 4; ++ks) {
      uint32_t af[4];
      nvfp4_afrag(cw[ks], sg, sg8, ks, af);
      if (BF16B) {
#pragma unroll
        for (int j = 0; j < 4; ++j) af[j] = f16x2_to_bf16x2(af[j]);
      }
#pragma unroll
      for (int nt = 0; nt < NTMAX; ++nt) {
        if (NTMAX == 1 || nt < nt_used) {
          const uint4& q = bx[nt][ks >> 1];
          if (BF16B)
            mma_bf16(acc[nt], af, (ks & 1) ? q.z : q.x, (ks & 1) ? q.w : q.y);
          else
            mma_f16(acc[nt], af, (ks & 1) ? q.z : q.x, (ks & 1) ? q.w : q.y);
        }
      }
    }
  } else {
#pragma unroll
    for (int ks = 0; ks < 4; ++ks) {
      const uint4 v = lds128(kp + lane * 64 + ks * 16);
      const uint32_t af[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int nt = 0; nt < NTMAX; ++nt) {
        if (NTMAX == 1 || nt < nt_used) {
          const uint4& q = bx[nt][ks >> 1];
          mma_bf16(acc[nt], af, (ks & 1) ? q.z : q.x, (ks & 1) ? q.w : q.y);
        }
      }
    }
  }
}

// ===========================================================================
// K2: gate/up GEMV + SiLU * up. A unit is (slot, tile of 8 intermediate rows);
// units are numbered slot-major. A block has ng groups of 4 warps; group gi
// works through units blockIdx.x + (gi + ng * jj) * gridDim.x, jj = 0, 1, ...,
// with nb of them in flight, and synchronises on its own named barrier, so the
// groups of a block proceed independently. The 4 warps of a group split a
// unit's reduction (H) into contiguous k-group ranges.
//
// Before waiting for the router the block copies the bf16 activations of all
// tokens, prescales them and stores them in fragment order: they are the
// previous layer's output, which had completed before the router (which lets
// this kernel launch only after its own wait) started.
// ===========================================================================
struct GateupPlan {
  size_t wbuf_off, xs_off, red_off, inv_off, bar_off, total;
};

__host__ __device__ inline GateupPlan gateup_plan(int H, int B, int fmt, int ntmax, int ng, int nb) {
  const int kgb = fmt == FLINT_MOE_NVFP4 ? KG_NVFP4 : KG_BF16;
  const size_t kslice = (size_t)(H / 256) * kgb;
  GateupPlan p;
  size_t o = 0;
  p.wbuf_off = o;   o += (size_t)ng * nb * 4 * kslice;
  p.xs_off = o;     o += (size_t)B * (H * 2 + 16);
  p.red_off = o;    o += sizeof(float) * ng * 2 * 4 * ntmax * 128;
  p.inv_off = o;    o += sizeof(float) * MAX_BATCH;
  o = (o + 15) & ~(size_t)15;
  p.bar_off = o;    o += sizeof(uint64_t) * ng * nb * 4;
  p.total = o;
  return p;
}

// Barrier of one 4-warp group (named barrier 1 + gi); returns the AND of v.
__device__ __forceinline__ bool group_sync_and(int gi, bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, %2, 128, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)v), "r"(gi + 1)
      : "memory");
  return r != 0;
}

// Activations for the gate/up kernels: warp w takes tokens w, w + nwarps, ...,
// applies the RMSNorm if asked, a per-token power-of-two prescale (NVFP4
// layers) and stores the row in mma B-fragment order (f16, or bf16 as is).
// Read straight from global memory (L2): a row of up to 2048 columns stays in
// registers between the max and the conversion; wider rows are read twice.
// PRE: 0 or 1 when the kernel was instantiated for one case of the pre-norm
// block, -1 to follow `prenorm` at run time.
template <int FMT, bool NARROW = false, int PRE = -1>
__device__ void stage_rows(const uint16_t* x, int B, int K, int prenorm_rt, const uint16_t* gamma, float eps,
                           uint8_t* xs, int xstride, float* s_inv, int warp, int nwarps, int lane) {
  const int prenorm = PRE < 0 ? prenorm_rt : PRE;
  for (int t = warp; t < B; t += nwarps) {
    const uint8_t* src = reinterpret_cast<const uint8_t*>(x + (size_t)t * K);
    const int nch = K / 256;  // 16-byte chunks per lane
    uint8_t* dst = xs + (size_t)t * xstride;
    auto absmax = [&](const uint4& u, float m) {
      const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int q = 0; q < 4; ++q) m = fmaxf(m, fmaxf(fabsf(bf16lo(w4[q])), fabsf(bf16hi(w4[q]))));
      return m;
    };
    auto store = [&](const uint4& u, int c, float sc) {
      const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
      const int col = 8 * (lane + 32 * c);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint32_t bits = w4[q];
        if (FMT == FLINT_MOE_NVFP4) {
          const __half2 hv = __floats2half2_rn(bf16lo(w4[q]) * sc, bf16hi(w4[q]) * sc);
          bits = *reinterpret_cast<const uint32_t*>(&hv);
        }
        *reinterpret_cast<uint32_t*>(dst + 2 * frag_offset_elems(col + 2 * q)) = bits;
      }
    };
    const uint8_t* gw8 = reinterpret_cast<const uint8_t*>(gamma);
    float mx = 0.f;
    int kx = 0;
    if (NARROW || nch <= 8) {
      uint4 v[8];
#pragma unroll
      for (int c = 0; c < 8; ++c)
        if (c < nch) v[c] = ld_cg_v4(src + (lane + 32 * c) * 16);
      if (prenorm) {  // RMSNorm, as the router computes it
        auto wv = [&](int c) { return __ldg(reinterpret_cast<const uint4*>(gw8 + (lane + 32 * c) * 16)); };
        float part = 0.f;
#pragma unroll
        for (int c = 0; c < 8; ++c)
          if (c < nch) part = sumsq8(v[c], part);
        const float ss = warp_sum(part);
        if (ss <= FP32_MAX) {
          const float inv = 1.0f / sqrtf(ss / (float)K + eps);
#pragma unroll
          for (int c = 0; c < 8; ++c)
            if (c < nch) v[c] = norm8(v[c], wv(c), inv);
        } else {  // the sum of squares overflowed: the scaled path
          const float2 f = rms_factor_huge(src, 0, lane, K, eps);
#pragma unroll
          for (int c = 0; c < 8; ++c)
            if (c < nch) v[c] = norm8_huge(v[c], wv(c), f);
        }
      }
      if (FMT == FLINT_MOE_NVFP4) {
#pragma unroll
        for (int c = 0; c < 8; ++c)
          if (c < nch) mx = absmax(v[c], mx);
        kx = prescale_exp(warp_max(mx));
      }
      const float sc = exp2i(kx);
#pragma unroll
      for (int c = 0; c < 8; ++c)
        if (c < nch) store(v[c], c, sc);
    } else {
      float inv = 1.f;
      float2 huge = make_float2(0.f, 0.f);  // the scaled path's factor and scale, if taken (y != 0)
      if (prenorm) {
        float part = 0.f;
#pragma unroll 8
        for (int c = 0; c < nch; ++c) part = sumsq8(ld_cg_v4(src + (lane + 32 * c) * 16), part);
        const float ss = warp_sum(part);
        if (ss <= FP32_MAX)
          inv = 1.0f / sqrtf(ss / (float)K + eps);
        else
          huge = rms_factor_huge(src, 0, lane, K, eps);
      }
      auto chunk = [&](int c) {
        const uint4 u = ld_cg_v4(src + (lane + 32 * c) * 16);
        if (!prenorm) return u;
        const uint4 w = __ldg(reinterpret_cast<const uint4*>(gw8 + (lane + 32 * c) * 16));
        return huge.y == 0.f ? norm8(u, w, inv) : norm8_huge(u, w, huge);
      };
      // unrolled by 8, so that 8 chunks' loads are in flight together
      if (FMT == FLINT_MOE_NVFP4) {
#pragma unroll 8
        for (int c = 0; c < nch; ++c) mx = absmax(chunk(c), mx);
        kx = prescale_exp(warp_max(mx));
      }
      const float sc = exp2i(kx);
#pragma unroll 8
      for (int c = 0; c < nch; ++c) store(chunk(c), c, sc);
    }
    if (lane == 0) s_inv[t] = exp2i(-kx);
  }
}

template <int FMT, bool NARROW, int PRE>
__device__ __forceinline__ void stage_x(const DecodeArgs& a, uint8_t* xs, int xstride, float* s_inv, int warp,
                                        int nwarps, int lane) {
  stage_rows<FMT, NARROW, PRE>(a.x, a.B, a.H, a.prenorm, a.gamma, a.eps, xs, xstride, s_inv, warp, nwarps, lane);
}

// Registers per thread of the gate/up kernel in its three-group shape (1 and 2
// tokens), which shares each SM with a down block of 8 warps at 64.
constexpr int GATEUP_SMALL_REGS = 112;

// REGS: registers per thread; 96 lets five groups fill the register file,
// GATEUP_SMALL_REGS is for three groups beside a down block (1 and 2 tokens).
template <int FMT, int NTMAX, bool NARROW, int PRE, int REGS = 96>
__global__ void __maxnreg__(REGS) k_gateup(const DecodeArgs a_in) {
  const DecodeArgs a = flint_shape<NARROW>(a_in);
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ RouteSmem R;
  constexpr int KGB = FMT == FLINT_MOE_NVFP4 ? KG_NVFP4 : KG_BF16;
  const int NG = blockDim.x >> 7, NB = a.gu_nb;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t4 = lane & 3;
  const int gi = warp >> 2, gw = warp & 3;
  const int TILES = a.I / 8;
  const int KGW = a.H / (KG_COLS * 4);
  const int kslice = KGW * KGB;
  const int xstride = a.H * 2 + 16;
  const GateupPlan P = gateup_plan(a.H, a.B, FMT, NTMAX, NG, NB);
  uint8_t* xs = smem + P.xs_off;
  // Partial sums of the group's four warps, double-buffered by unit parity:
  // the finalising warps read one buffer while the next unit fills the other.
  float* red = reinterpret_cast<float*>(smem + P.red_off) + gi * 2 * 4 * NTMAX * 128;
  float* s_inv = reinterpret_cast<float*>(smem + P.inv_off);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + P.bar_off);  // [NG][NB][4] weight slices
  auto wbar = [&](int b) { return &bars[(gi * NB + b) * 4 + gw]; };
  auto wbuf = [&](int b) { return smem + P.wbuf_off + ((size_t)(gi * NB + b) * 4 + gw) * kslice; };
  int* status = ws_hdr(a) + HDR_STATUS;
  const int G = gridDim.x;
  auto unit_of = [&](int jj) { return (int)blockIdx.x + (gi + NG * jj) * G; };

  FLINT_TRACE(a, 8);
  if (threadIdx.x < NG * NB * 4) mbar_init(&bars[threadIdx.x], 1);
  fence_mbar_init();
  __syncthreads();
  auto issue_w = [&](int b, int expert, int tile) {
    if (lane == 0) {
      const uint8_t* src = a.packed + (int64_t)expert * a.L.expert_bytes + (int64_t)tile * a.L.gu_tile +
                           (int64_t)gw * kslice;
      mbar_arrive_expect_tx(wbar(b), (uint32_t)kslice);
      bulk_g2s_stream(wbuf(b), src, (uint32_t)kslice, wbar(b));
    }
  };
  // The shared experts' units come first and need no routing: fetch them now.
  int pre = 0;
  while (pre < NB && unit_of(pre) < a.S * TILES) {
    const int u = unit_of(pre);
    issue_w(pre, a.E + u / TILES, u % TILES);
    ++pre;
  }
  route_clear(R, a.E);
  stage_x<FMT, NARROW, PRE>(a, xs, xstride, s_inv, warp, blockDim.x >> 5, lane);
  __syncthreads();  // route_clear before the selection's atomics
  pdl_wait();
  pdl_trigger();
  FLINT_TRACE(a, 9);
  route_select<NARROW>(a, R, false, false, 21, ws_logits(a));  // its barrier also publishes xs and s_inv
  FLINT_TRACE(a, 10);
  const int n_units = route_slots(a, R) * TILES;
  for (int jj = pre; jj < NB; ++jj) {
    const int u = unit_of(jj);
    if (u < n_units) issue_w(jj, slot_info(a, R, u / TILES).expert, u % TILES);
  }
  const float* glob = a.globals;
  int b = 0;          // jj % NB
  uint32_t par = 0u;  // (jj / NB) & 1
  for (int jj = 0;; ++jj) {
    const int u = unit_of(jj);
    if (u >= n_units) break;  // the same for the 4 warps of the group
    const int slot = u / TILES, tile = u % TILES;
    const SlotInfo si = slot_info(a, R, slot);
    const int expert = si.expert;
    const float Gg = glob[expert * 4 + 0];  // loaded while the weights are on their way
    const float Gu = glob[expert * 4 + 1];
    // One token tile (B <= 8): column c is token c. More: column c is the
    // slot's c-th selecting token, so a slot chosen by few tokens needs one tile.
    const int T = NTMAX == 1 ? a.B : __popc(si.tmask);
    const int nt_used = (T + 7) >> 3;
    float acc[2][NTMAX][4];
#pragma unroll
    for (int c = 0; c < 2; ++c)
#pragma unroll
      for (int nt = 0; nt < NTMAX; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[c][nt][i] = 0.f;
    const bool ok = mbar_wait(wbar(b), par, status);
    if (jj == 0) FLINT_TRACE(a, 11);
    // After a failed wait the buffer's copy is let land and the products run on
    // it all the same (the group stops after them): the loop is not under a
    // branch, so its mma.sync need no reconvergence of the warp first.
    if (!ok) mbar_drain(wbar(b), par);
    {
      int tok[NTMAX];  // column 8 nt + g (past T: a repeat of the last selecting token)
#pragma unroll
      for (int nt = 0; nt < NTMAX; ++nt)
        tok[nt] = NTMAX == 1 ? min(g, a.B - 1) : nth_set_bit(si.tmask, min(nt * 8 + g, T - 1));
      const uint8_t* wb = wbuf(b);
#pragma unroll 4
      for (int kl = 0; kl < KGW; ++kl) {
        const int kg = gw * KGW + kl;
        uint4 bx[NTMAX][2];
#pragma unroll
        for (int nt = 0; nt < NTMAX; ++nt) {
          if (NTMAX == 1 || nt < nt_used) {  // columns past the slot's tokens repeat a valid row
            const uint8_t* rp = xs + (size_t)tok[nt] * xstride + kg * 128 + t4 * 32;
            bx[nt][0] = lds128(rp);
            bx[nt][1] = lds128(rp + 16);
          }
        }
        if (kl & 1)
          tile_kgroup<FMT, NTMAX>(wb + kl * KGB, bx, nt_used, lane, acc[1]);
        else
          tile_kgroup<FMT, NTMAX>(wb + kl * KGB, bx, nt_used, lane, acc[0]);
      }
    }
    // Every warp's partial sums go to the group's reduction buffer
    // (double-buffered by unit parity); after the barrier the 2 * nt_used
    // (token tile, column parity) pairs are finalised by warps p % 4, each
    // adding the four partials in warp order.
    float* rb = red + (jj & 1) * 4 * NTMAX * 128;
#pragma unroll
    for (int nt = 0; nt < NTMAX; ++nt)
#pragma unroll
      for (int i = 0; i < 4; ++i) rb[(gw * NTMAX + nt) * 128 + lane * 4 + i] = acc[0][nt][i] + acc[1][nt][i];
    if (!group_sync_and(gi, ok)) {  // a copy timed out: let the next buffer's copies land, then stop
      if (unit_of(jj + 1) < n_units && NB > 1) mbar_drain(wbar((jj + 1) % NB), (uint32_t)(((jj + 1) / NB) & 1));
      break;
    }
    if (jj == 0) FLINT_TRACE(a, 12);
    // This warp's weight slice is free again: fetch its slice of unit jj + NB.
    {
      const int u2 = unit_of(jj + NB);
      if (u2 < n_units) issue_w(b, slot_info(a, R, u2 / TILES).expert, u2 % TILES);
    }
    const int hoff = frag_offset_elems(tile * 8 + g);
    uint16_t* h = ws_h(a);
    uint16_t* h16 = ws_h16(a);
    unsigned* hmax = ws_hmax(a);
    // (token tile, column parity) pairs; one token has no odd column
    const int npairs = NTMAX == 1 && T == 1 ? 1 : 2 * nt_used;
    for (int pr = gw; pr < npairs; pr += 4) {
      const int nt = pr >> 1, hh = pr & 1;
      float gs = 0.f, us = 0.f;
#pragma unroll
      for (int w2 = 0; w2 < 4; ++w2) {
        gs += rb[(w2 * NTMAX + nt) * 128 + lane * 4 + hh];
        us += rb[(w2 * NTMAX + nt) * 128 + lane * 4 + 2 + hh];
      }
      const int n = nt * 8 + 2 * t4 + hh;  // column
      const bool sel = n < T && (NTMAX > 1 || ((si.tmask >> n) & 1u));
      const int tk = NTMAX == 1 ? n : (sel ? nth_set_bit(si.tmask, n) : 0);  // its token
      const size_t row = (size_t)slot * a.B + tk;
      float hv = 0.f;
      if (sel) {
        const float inv = s_inv[tk];
        const float gv = (gs * inv) * Gg;
        const float uv = (us * inv) * Gu;
        const float ey = 1.0f + expf(-gv);
        const float sv = ey < RCP_NR_MAX ? gv * rcp_nr(ey) : div_ieee(gv, ey);  // SiLU
        const __nv_bfloat16 hb = __float2bfloat16_rn(sv * uv);
        h[row * a.I + hoff] = *reinterpret_cast<const uint16_t*>(&hb);
        hv = fabsf(__bfloat162float(hb));
        if (a.W.has_h16) {
          const __half hh = __float2half_rn(__bfloat162float(hb));
          h16[row * a.I + hoff] = *reinterpret_cast<const uint16_t*>(&hh);
        }
      }
      hv = fmaxf(hv, __shfl_xor_sync(0xffffffffu, hv, 4));
      hv = fmaxf(hv, __shfl_xor_sync(0xffffffffu, hv, 8));
      hv = fmaxf(hv, __shfl_xor_sync(0xffffffffu, hv, 16));
      if (g == 0 && sel && hv > 0.f) {
        atomicMax(hmax + row, __float_as_uint(hv));
        if (!(hv < 32768.f)) atomicOr(ws_hdr(a) + HDR_HBIG, 1);  // its f16 copy is not exact
      }
    }
    if (++b == NB) {
      b = 0;
      par ^= 1u;
    }
  }
  FLINT_TRACE(a, 13);
}

// One row of I bf16 values (row stride >= 2 I) to f16 times 2^kh, in place:
// each lane converts 16-byte words lane, lane + 32, ..., two at a time so
// that their shared-memory latencies overlap.
__device__ __forceinline__ uint32_t bf16x2_to_f16x2_scaled(uint32_t w, float sc) {
  const __half2 hv = __floats2half2_rn(bf16lo(w) * sc, bf16hi(w) * sc);
  return *reinterpret_cast<const uint32_t*>(&hv);
}
__device__ __forceinline__ void row_to_f16(uint8_t* row, int I, int kh, int lane) {
  const float sc = exp2i(kh);
  for (int q = lane; q < I / 8; q += 64) {
    const bool two = q + 32 < I / 8;
    uint4 u0 = lds128(row + q * 16), u1 = two ? lds128(row + (q + 32) * 16) : make_uint4(0, 0, 0, 0);
    u0 = make_uint4(bf16x2_to_f16x2_scaled(u0.x, sc), bf16x2_to_f16x2_scaled(u0.y, sc),
                    bf16x2_to_f16x2_scaled(u0.z, sc), bf16x2_to_f16x2_scaled(u0.w, sc));
    *reinterpret_cast<uint4*>(row + q * 16) = u0;
    if (two) {
      u1 = make_uint4(bf16x2_to_f16x2_scaled(u1.x, sc), bf16x2_to_f16x2_scaled(u1.y, sc),
                      bf16x2_to_f16x2_scaled(u1.z, sc), bf16x2_to_f16x2_scaled(u1.w, sc));
      *reinterpret_cast<uint4*>(row + (q + 32) * 16) = u1;
    }
  }
}

// ===========================================================================
// K3 for small batches (at most 8 tokens, NVFP4): each warp keeps nbuf items
// in flight, each buffer holding the item's down tile and its h rows, so a
// warp copies and consumes its own items with no block barrier before the
// final sum. The products run in bf16 (the dequantised weights are exact in
// bf16), so h is used as stored, without the prescale pass of the staged
// kernel. Measured faster than the staged kernel below at batch 1 (fewer
// instructions on the cold path after the wait).
// ===========================================================================
// The rare path of the small-batch down kernel, when some |h| of the call
// reached 2^15 (its f16 copy is not exact): the item's selected token rows
// (h rows r0 + n, n < 8, bit n of bits) are rebuilt in the buffer from the
// bf16 h, each times a power of two that puts its largest |h| in
// [2^14, 2^15) (exact down to 2^-29 of it). Whole warp; returns, in lane
// n < 8, the inverse of column n's scale (1 elsewhere). Out of line: the
// common path carries none of it.
static __device__ __noinline__ float h_rows_prescaled(const unsigned* hmax, const uint16_t* h, int I, uint8_t* hb,
                                                      int hstride, int r0, uint32_t bits, int lane) {
  float inv = 1.0f;
  for (int n = 0; n < 8; ++n) {
    if (!((bits >> n) & 1u)) continue;
    const int kh = prescale_exp(__uint_as_float(__ldcg(hmax + r0 + n)));
    const float sc = exp2i(kh);
    const uint8_t* src = reinterpret_cast<const uint8_t*>(h + (size_t)(r0 + n) * I);
    uint8_t* dst = hb + n * hstride;
    for (int q = lane; q < I / 8; q += 32) {
      const uint4 u = ld_cg_v4(src + q * 16);
      *reinterpret_cast<uint4*>(dst + q * 16) =
          make_uint4(bf16x2_to_f16x2_scaled(u.x, sc), bf16x2_to_f16x2_scaled(u.y, sc),
                     bf16x2_to_f16x2_scaled(u.z, sc), bf16x2_to_f16x2_scaled(u.w, sc));
    }
    if (lane == n) inv = exp2i(-kh);
  }
  __syncwarp();
  return inv;
}

// The small-batch down kernel's two shapes: 8 warps with 2 tiles in flight
// each (1 and 2 tokens, beside a gate/up block), or 16 warps with 1.
constexpr int DOWN_ITEMS_NW = 8, DOWN_ITEMS_NBUF = 2, DOWN_ITEMS_WIDE_NW = 16, DOWN_ITEMS_WIDE_NBUF = 1;
__host__ __device__ constexpr int down_items_warps(int nbuf) { return nbuf == DOWN_ITEMS_NBUF ? DOWN_ITEMS_NW : DOWN_ITEMS_WIDE_NW; }

// A compile-time flag as a value (selects a copy of a generic lambda's body).
template <bool V>
struct BoolTag {
  static constexpr bool value = V;
};

struct DownItemsPlan {
  int buf_bytes, hrows, hstride;
  size_t acc_off, sw_off, bar_off, total;
};

__host__ __device__ inline DownItemsPlan down_items_plan(int H, int I, int B, int max_slots, int fmt, int nbuf, int nw) {
  DownItemsPlan p;
  const int kgb = fmt == FLINT_MOE_NVFP4 ? KG_NVFP4 : KG_BF16;
  p.hrows = B < 8 ? B : 8;
  p.hstride = I * 2 + 16;
  p.buf_bytes = (I / KG_COLS) * kgb + p.hrows * p.hstride;
  size_t o = (size_t)nw * nbuf * p.buf_bytes;
  p.acc_off = o;    o += sizeof(float) * nw * B * 16;
  p.sw_off = o;     o += sizeof(float) * 8 * max_slots;  // routing weights [slot][token]
  o = (o + 15) & ~(size_t)15;
  p.bar_off = o;    o += sizeof(uint64_t) * nw * nbuf;
  p.total = o;
  return p;
}

// ===========================================================================
// Small-batch down kernel (up to 8 tokens, NVFP4 weights): one block per 16
// output rows. Up to 8 tokens a slot is one work item; warp w takes slots
// w, w + NW, ... with NBUF buffers, each holding the slot's 4.6 KB down tile
// and the f16 rows of h of the tokens that selected its expert. Before its
// dependency wait the block fetches the down tiles (the shared experts' at
// once, the routed ones after routing) while k_gateup runs; after it, the h
// rows. Per-warp partial sums are added in warp order at the end.
// ===========================================================================
template <int FMT, int NBUF, bool NARROW, int PRE>
__global__ void __launch_bounds__(512) k_down_items(const DecodeArgs a_in) {
  const DecodeArgs a = flint_shape<NARROW>(a_in);
  const int prenorm = PRE < 0 ? a.prenorm : PRE;
  constexpr int NW = down_items_warps(NBUF);
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ RouteSmem R;
  __shared__ uint16_t s_res[8 * 16];  // residual values (pre-norm block)
  constexpr int KGB = FMT == FLINT_MOE_NVFP4 ? KG_NVFP4 : KG_BF16;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t4 = lane & 3;
  const int tile = blockIdx.x;
  const DownItemsPlan P = down_items_plan(a.H, a.I, a.B, a.W.max_slots, FMT, NBUF, NW);
  const int dn_bytes = (int)a.L.dn_tile;
  float* acc_s = reinterpret_cast<float*>(smem + P.acc_off);
  float* s_sw = reinterpret_cast<float*>(smem + P.sw_off);  // [slot][8]: routing weight of token n
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + P.bar_off) + warp * NBUF;
  auto buf = [&](int b) { return smem + (size_t)(warp * NBUF + b) * P.buf_bytes; };
  int* status = ws_hdr(a) + HDR_STATUS;

  // The next layer's router may launch now (it waits for this grid to
  // complete): its row fetch and warm-up pass then finish before that. Not
  // for the pre-norm block, where launching the router early measured slower
  // (the stack at batch 1: 10.89 -> 11.40 us per layer; the rotation gains
  // 0.04-0.09).
  if (!prenorm) pdl_trigger();
  FLINT_TRACE(a, 16);
  if (lane < NBUF) mbar_init(&bars[lane], 2);  // one arrival for the weights, one for the h rows
  fence_mbar_init();
  for (int i = threadIdx.x; i < NW * a.B * 16; i += blockDim.x) acc_s[i] = 0.f;
  route_clear(R, a.E);
  __syncthreads();

  auto issue_weights = [&](int j, int expert) {
    if (lane == 0) {
      const uint8_t* src = a.packed + (int64_t)expert * a.L.expert_bytes + a.L.gu_bytes + (int64_t)tile * dn_bytes;
      mbar_arrive_expect_tx(&bars[j % NBUF], (uint32_t)dn_bytes);
      bulk_g2s_stream(buf(j % NBUF), src, (uint32_t)dn_bytes, &bars[j % NBUF]);
    }
  };
  // Up to 8 tokens (one token tile) a slot is one work item: warp w takes
  // slots w, w + NW, .... The shared experts' slots come first and are known
  // before routing.
  int w_issued = 0;
  for (int i = warp; i < a.S && w_issued < NBUF; i += NW, ++w_issued) issue_weights(w_issued, a.E + i);

  // k_gateup lets this kernel launch only after its own wait, so the router has
  // finished: route now and fetch the routed down tiles while k_gateup runs.
  route_select<NARROW>(a, R, true, blockIdx.x == 0, -1, ws_logits(a));
  FLINT_TRACE(a, 17);
  const int n_items = route_slots(a, R);
  auto item_of = [&](int j, int& s, uint32_t& bits, int& expert) {
    s = warp + NW * j;
    const SlotInfo si = slot_info(a, R, s);
    expert = si.expert;
    bits = si.tmask & 0xFFu;
  };
  for (int j = w_issued; j < NBUF && warp + NW * j < n_items; ++j) {
    int s, e;
    uint32_t bits;
    item_of(j, s, bits, e);
    issue_weights(j, e);
  }
  // The combine's routing weights, by slot and token: entry (slot of the
  // r-th pick of token t, t) = the pick's weight (entries of tokens that did
  // not select the slot's expert are never read; shared slots weigh 1).
  for (int i = threadIdx.x; i < a.B * a.k; i += blockDim.x)
    s_sw[(a.S + used_rank<NARROW>(a, R, R.idx[i])) * 8 + i / a.k] = R.w[i];

  // Slot s is h rows s * B + n, n < B; only the rows of tokens that selected
  // the expert are copied (column n of the product is token n, and the other
  // columns are never combined).
  auto issue_h = [&](int j) {
    int s, e;
    uint32_t bits;
    item_of(j, s, bits, e);
    const int r0 = s * a.B;
    const int b = j % NBUF;
    if (lane == 0) mbar_arrive_expect_tx(&bars[b], (uint32_t)(__popc(bits) * a.I * 2));
    __syncwarp();
    if (lane < 8 && ((bits >> lane) & 1u))
      bulk_g2s(buf(b) + dn_bytes + lane * P.hstride, ws_h16(a) + (size_t)(r0 + lane) * a.I, (uint32_t)(a.I * 2),
               &bars[b]);
  };
  const int KG = a.I / KG_COLS;
  // The residual rows of this tile (the layer's input, final before the
  // router ran) are read now, while the wait is pending.
  if (prenorm)
    for (int p = threadIdx.x; p < a.B * 16; p += blockDim.x)
      s_res[p] = __ldcg(a.x + (size_t)(p >> 4) * a.H + tile * 16 + (p & 15));
  __syncthreads();  // the weight table is complete
  pdl_wait();       // h comes from k_gateup
  if (prenorm) pdl_trigger();
  FLINT_TRACE(a, 18);
  for (int j = 0; j < NBUF && warp + NW * j < n_items; ++j) issue_h(j);
  // h is consumed in its f16 copy, exact for |h| < 2^15, so the products run
  // in f16 with the dequantised weights as they are (exact in f16): no
  // conversion, no per-row prescale, no block barrier between the wait and
  // the products. Only if some |h| of the call reached 2^15 (the flag is read
  // while the copies are on their way) does each item rebuild its rows from
  // the bf16 h with a per-row power-of-two prescale: a second copy of the
  // item loop, so that the common one carries no call.
  const bool hbig = __ldcg(ws_hdr(a) + HDR_HBIG) != 0;
  auto run_items = [&](auto hbig_tag) {
    constexpr bool HBIG = decltype(hbig_tag)::value;
    for (int j = 0; warp + NW * j < n_items; ++j) {
      int s, expert;
      uint32_t bits;
      item_of(j, s, bits, expert);
      const int b = j % NBUF;
      const uint32_t parity = (uint32_t)((j / NBUF) & 1);
      const float Gd = a.globals[expert * 4 + 2];  // loaded while the copies are on their way
      if (!mbar_wait(&bars[b], parity, status)) {
        for (int jj = j; jj < j + NBUF && warp + NW * jj < n_items; ++jj)
          mbar_drain(&bars[jj % NBUF], (uint32_t)((jj / NBUF) & 1));
        break;
      }
      if (j == 0) FLINT_TRACE(a, 19);
      uint8_t* wb = buf(b);
      uint8_t* hb = wb + dn_bytes;
      float hinv = 1.0f;  // this lane's column's inverse prescale (fallback only)
      if constexpr (HBIG) hinv = h_rows_prescaled(ws_hmax(a), ws_h(a), a.I, hb, P.hstride, s * a.B, bits, lane);
      float acc[2][1][4];
#pragma unroll
      for (int c = 0; c < 2; ++c)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[c][0][i] = 0.f;
      const int nrow = g < a.B ? g : a.B - 1;
#pragma unroll 4
      for (int kg = 0; kg < KG; ++kg) {
        const uint8_t* rp = hb + nrow * P.hstride + kg * 128 + t4 * 32;
        uint4 bx[1][2];
        bx[0][0] = lds128(rp);
        bx[0][1] = lds128(rp + 16);
        if (kg & 1)
          tile_kgroup<FMT, 1>(wb + kg * KGB, bx, 1, lane, acc[1]);
        else
          tile_kgroup<FMT, 1>(wb + kg * KGB, bx, 1, lane, acc[0]);
      }
      float inv0 = 1.0f, inv1 = 1.0f;
      if constexpr (HBIG) {  // columns 2 t4 and 2 t4 + 1: their inverse prescales, from lanes n
        inv0 = __shfl_sync(0xffffffffu, hinv, 2 * t4);
        inv1 = __shfl_sync(0xffffffffu, hinv, 2 * t4 + 1);
      }
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int n = 2 * t4 + hh;  // the column's token
        if (n < a.B && ((bits >> n) & 1u)) {
          const float wt = s < a.S ? 1.0f : s_sw[s * 8 + n];  // the shared experts are unweighted
          const float inv = hh ? inv1 : inv0;
          float* dst = acc_s + (warp * a.B + n) * 16;
          dst[g] += wt * (((acc[0][0][hh] + acc[1][0][hh]) * inv) * Gd);
          dst[g + 8] += wt * (((acc[0][0][2 + hh] + acc[1][0][2 + hh]) * inv) * Gd);
        }
      }
      __syncwarp();
      if (warp + NW * (j + NBUF) < n_items) {
        fence_proxy_async();  // this warp's accesses to the buffer come before the copies into it
        int s2, e2;
        uint32_t bits2;
        item_of(j + NBUF, s2, bits2, e2);
        issue_weights(j + NBUF, e2);
        issue_h(j + NBUF);
      }
    }
  };
  if (hbig)
    run_items(BoolTag<true>{});
  else
    run_items(BoolTag<false>{});
  __syncthreads();
  for (int p = threadIdx.x; p < a.B * 16; p += blockDim.x) {
    const int t = p >> 4, r = p & 15;
    float v = 0.f;
#pragma unroll
    for (int w2 = 0; w2 < NW; ++w2) v += acc_s[(w2 * a.B + t) * 16 + r];
    __nv_bfloat16 o = __float2bfloat16_rn(v);
    if (prenorm) {  // residual stream: r + bf16(layer output), rounded to bf16
      const uint32_t rb = (uint32_t)s_res[p] << 16;
      o = __float2bfloat16_rn(__uint_as_float(rb) + __bfloat162float(o));
    }
    a.out[(size_t)t * a.H + tile * 16 + r] = *reinterpret_cast<const uint16_t*>(&o);
  }
  FLINT_TRACE(a, 20);
}

// ===========================================================================
// K3: down GEMV + routing-weighted combine for one tile of 16 output rows.
// Work items are (slot, token tile) pairs with at least one selecting token,
// slot-major; warp w of nw takes items w, w + nw, ... in order with nbuf down
// tiles in flight (routing-independent: fetched while k_gateup still runs).
// The h rows the items read (one per selecting token) are staged once per
// block, converted to prescaled f16 once, and shared by all warps: in rounds
// of consecutive items when they do not all fit. Per-warp partial sums are
// added in warp order at the end, so the result does not depend on timing.
// ===========================================================================
struct DownPlan {
  int nw, nbuf, hcap, hstride;
  size_t wbuf_off, h_off, acc_off, items_off, hsc_off, hinv_off, bar_off, total;
};

__host__ __device__ inline DownPlan down_plan(int I, int B, int max_slots, int fmt, int nw, int nbuf, int hcap) {
  DownPlan p;
  const int kgb = fmt == FLINT_MOE_NVFP4 ? KG_NVFP4 : KG_BF16;
  const int dn = (I / KG_COLS) * kgb;
  const int nt = (B + 7) / 8;
  p.nw = nw;
  p.nbuf = nbuf;
  p.hcap = hcap;
  p.hstride = I * 2 + 16;
  size_t o = 0;
  p.wbuf_off = o;   o += (size_t)nw * nbuf * dn;
  p.h_off = o;      o += (size_t)hcap * p.hstride;
  p.acc_off = o;    o += sizeof(float) * nw * B * 16;
  p.items_off = o;  o += sizeof(int) * 4 * max_slots * nt;
  p.hsc_off = o;    o += sizeof(float) * hcap;
  p.hinv_off = o;   o += sizeof(float) * hcap;
  o = (o + 15) & ~(size_t)15;
  p.bar_off = o;    o += sizeof(uint64_t) * nw * (nbuf + 1);
  p.total = o;
  return p;
}

template <int FMT, bool NARROW>
__global__ void __launch_bounds__(512) k_down(const DecodeArgs a_in) {
  const DecodeArgs a = flint_shape<NARROW>(a_in);
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ RouteSmem R;
  __shared__ int s_wsum[MAX_WARPS];
  __shared__ uint16_t s_res[MAX_BATCH * 16];  // residual values (pre-norm block)
  constexpr int KGB = FMT == FLINT_MOE_NVFP4 ? KG_NVFP4 : KG_BF16;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t4 = lane & 3;
  const int nw = blockDim.x >> 5;
  const int tile = blockIdx.x;
  const int NT = (a.B + 7) / 8;  // token tiles
  const DownPlan P = down_plan(a.I, a.B, a.W.max_slots, FMT, nw, a.dn_nbuf, a.dn_hcap);
  const int NBUF = P.nbuf;
  const int dn_bytes = (int)a.L.dn_tile;
  float* acc_s = reinterpret_cast<float*>(smem + P.acc_off);
  // per item: slot << 16 | chunk << 8 | count, expert, first staged row, token mask
  int* s_items = reinterpret_cast<int*>(smem + P.items_off);
  float* s_hsc = reinterpret_cast<float*>(smem + P.hsc_off);  // staged row's max |h|
  float* s_hinv = reinterpret_cast<float*>(smem + P.hinv_off);  // staged row's inverse prescale
  uint8_t* hsm = smem + P.h_off;
  uint64_t* wbars = reinterpret_cast<uint64_t*>(smem + P.bar_off) + warp * NBUF;
  uint64_t* hbar = reinterpret_cast<uint64_t*>(smem + P.bar_off) + nw * NBUF + warp;  // this warp's h rows
  auto wbuf = [&](int b) { return smem + P.wbuf_off + (size_t)(warp * NBUF + b) * dn_bytes; };
  int* status = ws_hdr(a) + HDR_STATUS;

  FLINT_TRACE(a, 16);
  if (lane < NBUF) mbar_init(&wbars[lane], 1);
  if (lane == 0) mbar_init(hbar, 1);
  fence_mbar_init();
  for (int i = threadIdx.x; i < nw * a.B * 16; i += blockDim.x) acc_s[i] = 0.f;
  route_clear(R, a.E);
  __syncthreads();

  auto issue_weights = [&](int j, int expert) {
    if (lane == 0) {
      const uint8_t* src = a.packed + (int64_t)expert * a.L.expert_bytes + a.L.gu_bytes + (int64_t)tile * dn_bytes;
      mbar_arrive_expect_tx(&wbars[j % NBUF], (uint32_t)dn_bytes);
      bulk_g2s_stream(wbuf(j % NBUF), src, (uint32_t)dn_bytes, &wbars[j % NBUF]);
    }
  };
  // The shared experts' items come first and cover every token tile, so they
  // are known before routing.
  int w_issued = 0;
  for (int i = warp; i < a.S * NT && w_issued < NBUF; i += nw, ++w_issued) issue_weights(w_issued, a.E + i / NT);

  // k_gateup lets this kernel launch only after its own wait, so the router has
  // finished: route now and fetch the routed down tiles while k_gateup runs.
  route_select<NARROW>(a, R, true, blockIdx.x == 0, -1, ws_logits(a));
  FLINT_TRACE(a, 17);
  const int n_slots = route_slots(a, R);
  {  // item list: chunks of up to 8 of a slot's selecting tokens; items and
     // staged rows counted in one packed prefix sum
    const int spt = (n_slots + blockDim.x - 1) / blockDim.x;
    const int s0 = threadIdx.x * spt;
    int local = 0;
    for (int s = s0; s < s0 + spt && s < n_slots; ++s) {
      const int T = __popc(slot_info(a, R, s).tmask);
      local += (((T + 7) >> 3) << 16) | T;
    }
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += n;
    }
    if (lane == 31) s_wsum[warp] = incl;
    __syncthreads();
    int run = incl - local;
    for (int w2 = 0; w2 < warp; ++w2) run += s_wsum[w2];
    for (int s = s0; s < s0 + spt && s < n_slots; ++s) {
      const SlotInfo si = slot_info(a, R, s);
      const int T = __popc(si.tmask);
      for (int c = 0; 8 * c < T; ++c) {
        const int it = run >> 16, cnt = min(8, T - 8 * c);
        s_items[4 * it] = (s << 16) | (c << 8) | cnt;
        s_items[4 * it + 1] = si.expert;
        s_items[4 * it + 2] = run & 0xFFFF;
        s_items[4 * it + 3] = (int)si.tmask;
        run += (1 << 16) | cnt;
      }
    }
  }
  __syncthreads();
  int tot = 0;
  for (int w2 = 0; w2 < nw; ++w2) tot += s_wsum[w2];
  const int n_items = tot >> 16, n_rows = tot & 0xFFFF;
  auto rowbase = [&](int i) { return i < n_items ? s_items[4 * i + 2] : n_rows; };
  for (int j = w_issued; j < NBUF && warp + nw * j < n_items; ++j) issue_weights(j, s_items[4 * (warp + nw * j) + 1]);

  const int KG = a.I / KG_COLS;
  // Round r stages the h rows of items i0 .. i1 - 1, as many as fit.
  auto round_end = [&](int i0) {
    const int rb0 = rowbase(i0);
    int lo = i0 + 1, hi = n_items;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (rowbase(mid) - rb0 <= P.hcap) lo = mid;
      else hi = mid - 1;
    }
    return lo;
  };
  int i1 = n_items > 0 ? round_end(0) : 0;

  // The residual rows of this tile (the layer's input, final before the
  // router ran) are read now, while the wait is pending.
  if (a.prenorm)
    for (int p = threadIdx.x; p < a.B * 16; p += blockDim.x)
      s_res[p] = __ldcg(a.x + (size_t)(p >> 4) * a.H + tile * 16 + (p & 15));
  pdl_wait();  // h comes from k_gateup
  pdl_trigger();
  FLINT_TRACE(a, 18);

  uint16_t* h = ws_h(a);
  const unsigned* hmax = ws_hmax(a);
  int j = 0;           // this warp's next item is warp + nw * j
  bool dead = false;   // a weight copy of this warp timed out
  uint32_t hphase = 0;
  for (int i0 = 0; i0 < n_items; i0 = i1, i1 = i0 < n_items ? round_end(i0) : i0) {
    const int rb0 = rowbase(i0);
    // This warp's items of the round are warp + nw * jj, j <= jj < jend; it
    // stages their rows (disjoint slices of the shared area) on its own
    // barrier and converts them itself: no block barrier inside a round.
    const int jend = i1 > warp ? (i1 - warp + nw - 1) / nw : 0;
    if (j < jend && !dead) {
      int myrows = 0;
      for (int jj = j + lane; jj < jend; jj += 32) myrows += s_items[4 * (warp + nw * jj)] & 0xFF;
      myrows = __reduce_add_sync(0xffffffffu, myrows);
      if (lane == 0) mbar_arrive_expect_tx(hbar, (uint32_t)(myrows * a.I * 2));
      __syncwarp();
      for (int jj = j + lane; jj < jend; jj += 32) {
        const int it = warp + nw * jj;
        const int code = s_items[4 * it], s = code >> 16, c = (code >> 8) & 0xFF, cnt = code & 0xFF;
        const uint32_t tm = (uint32_t)s_items[4 * it + 3];
        const int r0 = rowbase(it) - rb0;
        unsigned hv[8];
#pragma unroll
        for (int n = 0; n < 8; ++n) {  // copies first, then all the maxima in flight together
          if (n < cnt) {
            const int src = s * a.B + nth_set_bit(tm, 8 * c + n);
            bulk_g2s(hsm + (size_t)(r0 + n) * P.hstride, h + (size_t)src * a.I, (uint32_t)(a.I * 2), hbar);
            hv[n] = __ldcg(hmax + src);
          }
        }
#pragma unroll
        for (int n = 0; n < 8; ++n)
          if (n < cnt) s_hsc[r0 + n] = __uint_as_float(hv[n]);
      }
      const bool okh = mbar_wait(hbar, hphase, status);
      hphase ^= 1;
      __syncwarp();
      if (!okh) {
        mbar_drain(hbar, hphase ^ 1);
        dead = true;
      } else {
        if (i0 == 0 && warp == 0) FLINT_TRACE(a, 19);
        for (int jj = j; jj < jend; ++jj) {  // prescaled f16 (NVFP4) or kept (BF16)
          const int it = warp + nw * jj;
          const int r0 = rowbase(it) - rb0, nrow = s_items[4 * it] & 0xFF;
          for (int r = r0; r < r0 + nrow; ++r) {
            int kh = 0;
            if (FMT == FLINT_MOE_NVFP4) {
              kh = prescale_exp(s_hsc[r]);
              row_to_f16(hsm + (size_t)r * P.hstride, a.I, kh, lane);
            }
            if (lane == 0) s_hinv[r] = exp2i(-kh);
          }
        }
        __syncwarp();
        if (i0 == 0 && warp == 0) FLINT_TRACE(a, 6);
      }
    }
    for (; !dead && warp + nw * j < i1; ++j) {
      const int it = warp + nw * j;
      const int code = s_items[4 * it], s = code >> 16, c = (code >> 8) & 0xFF, cnt = code & 0xFF;
      const uint32_t tm = (uint32_t)s_items[4 * it + 3];
      const int expert = s_items[4 * it + 1], rb = rowbase(it) - rb0;
      const int b = j % NBUF;
      const float Gd = a.globals[expert * 4 + 2];  // loaded while the copies are on their way
      if (!mbar_wait(&wbars[b], (uint32_t)((j / NBUF) & 1), status)) {
        for (int jj = j; jj < j + NBUF && warp + nw * jj < n_items; ++jj)
          mbar_drain(&wbars[jj % NBUF], (uint32_t)((jj / NBUF) & 1));
        dead = true;
        break;
      }
      if (j == 0 && warp == 0) FLINT_TRACE(a, 15);
      const uint8_t* wb = wbuf(b);
      // Column n < cnt is the item's n-th token (staged row rb + n); the
      // other columns read row rb and are never combined.
      const int grow = rb + (g < cnt ? g : 0);
      float acc[2][1][4];
#pragma unroll
      for (int c = 0; c < 2; ++c)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[c][0][i] = 0.f;
#pragma unroll 4
      for (int kg = 0; kg < KG; ++kg) {
        const uint8_t* rp = hsm + (size_t)grow * P.hstride + kg * 128 + t4 * 32;
        uint4 bx[1][2];
        bx[0][0] = lds128(rp);
        bx[0][1] = lds128(rp + 16);
        if (kg & 1)
          tile_kgroup<FMT, 1>(wb + kg * KGB, bx, 1, lane, acc[1]);
        else
          tile_kgroup<FMT, 1>(wb + kg * KGB, bx, 1, lane, acc[0]);
      }
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int n = 2 * t4 + hh;
        if (n < cnt) {
          const int tok = nth_set_bit(tm, 8 * c + n);
          float wt = 1.0f;  // the shared experts are unweighted
          if (s >= a.S)
            for (int r = 0; r < a.k; ++r)
              if (R.idx[tok * a.k + r] == expert) wt = R.w[tok * a.k + r];
          const float inv = s_hinv[rb + n];
          float* dst = acc_s + (warp * a.B + tok) * 16;
          dst[g] += wt * (((acc[0][0][hh] + acc[1][0][hh]) * inv) * Gd);
          dst[g + 8] += wt * (((acc[0][0][2 + hh] + acc[1][0][2 + hh]) * inv) * Gd);
        }
      }
      __syncwarp();
      if (warp + nw * (j + NBUF) < n_items) issue_weights(j + NBUF, s_items[4 * (warp + nw * (j + NBUF)) + 1]);
    }
    if (i1 < n_items) {     // another round reuses the staging area
      fence_proxy_async();  // reads of it come before the next round's copies into it
      if (!__syncthreads_and(!dead)) {
        dead = true;
        break;
      }
    }
  }
  dead = __syncthreads_or(dead);
  if (dead)  // let this warp's weight copies in flight land before the block exits
    for (int jj = j; jj < j + NBUF && warp + nw * jj < n_items; ++jj)
      mbar_drain(&wbars[jj % NBUF], (uint32_t)((jj / NBUF) & 1));
  __syncthreads();
  if (dead) return;
  for (int p = threadIdx.x; p < a.B * 16; p += blockDim.x) {
    const int t = p >> 4, r = p & 15;
    float v = 0.f;
    for (int w2 = 0; w2 < nw; ++w2) v += acc_s[(w2 * a.B + t) * 16 + r];
    __nv_bfloat16 o = __float2bfloat16_rn(v);
    if (a.prenorm) {  // residual stream: r + bf16(layer output), rounded to bf16
      const uint32_t rb = (uint32_t)s_res[p] << 16;
      o = __float2bfloat16_rn(__uint_as_float(rb) + __bfloat162float(o));
    }
    a.out[(size_t)t * a.H + tile * 16 + r] = *reinterpret_cast<const uint16_t*>(&o);
  }
  FLINT_TRACE(a, 20);
}

// ===========================================================================
// Small-batch dense GEMV: y [B][N] = x [B][K] W^T for a packed NVFP4 or BF16
// matrix (16-row tiles of 64-column k-groups). One block per 16 output rows;
// its nw warps split K into contiguous k-group ranges, each fetching its slice
// of the tile with one bulk copy before the dependency wait (the weights do
// not depend on the previous kernel), and the warps' partial sums are added
// in warp order.
// ===========================================================================
struct GemvArgs {
  int N, K, B, fmt, prenorm;
  const uint16_t* x;
  uint16_t* y;
  const uint8_t* packed;
  const float* G;  // the tensor scale word after the tiles
  Layout L;
  const uint16_t* gamma;
  float eps;
  int* status;
};

__host__ __device__ inline size_t gemv_smem(int K, int B, int fmt, int nw, int ntmax, size_t* xs_off,
                                            size_t* inv_off, size_t* wbuf_off, size_t* red_off, size_t* bar_off) {
  const int kgb = fmt == FLINT_MOE_NVFP4 ? KG_NVFP4 : KG_BF16;
  size_t o = 0;
  *wbuf_off = o;  o += (size_t)(K / KG_COLS) * kgb;
  *xs_off = o;    o += (size_t)B * (K * 2 + 16);
  *inv_off = o;   o += sizeof(float) * MAX_BATCH;
  *red_off = o;   o += sizeof(float) * nw * ntmax * 128;
  o = (o + 15) & ~(size_t)15;
  *bar_off = o;   o += sizeof(uint64_t) * nw;
  return o;
}

template <int FMT, int NTMAX>
__global__ void __launch_bounds__(256) k_gemv(GemvArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  constexpr int KGB = FMT == FLINT_MOE_NVFP4 ? KG_NVFP4 : KG_BF16;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t4 = lane & 3;
  const int nw = blockDim.x >> 5;
  const int KGW = (a.K / KG_COLS) / nw;  // k-groups per warp
  size_t xs_off, inv_off, wbuf_off, red_off, bar_off;
  gemv_smem(a.K, a.B, FMT, nw, NTMAX, &xs_off, &inv_off, &wbuf_off, &red_off, &bar_off);
  uint8_t* wb = smem + wbuf_off + (size_t)warp * KGW * KGB;
  uint8_t* xs = smem + xs_off;
  float* s_inv = reinterpret_cast<float*>(smem + inv_off);
  float* red = reinterpret_cast<float*>(smem + red_off);
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + bar_off) + warp;
  const int xstride = a.K * 2 + 16;
  if (lane == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
    const uint32_t bytes = (uint32_t)KGW * KGB;
    mbar_arrive_expect_tx(bar, bytes);
    bulk_g2s_stream(wb, a.packed + (int64_t)blockIdx.x * a.L.dn_tile + (int64_t)warp * bytes, bytes, bar);
  }
  pdl_wait();  // x may be the previous kernel's output
  pdl_trigger();
  stage_rows<FMT>(a.x, a.B, a.K, a.prenorm, a.gamma, a.eps, xs, xstride, s_inv, warp, nw, lane);
  __syncthreads();
  const int nt_used = (a.B + 7) >> 3;
  float acc[2][NTMAX][4];
#pragma unroll
  for (int c = 0; c < 2; ++c)
#pragma unroll
    for (int nt = 0; nt < NTMAX; ++nt)
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[c][nt][i] = 0.f;
  const bool ok = mbar_wait(bar, 0, a.status);
  // after a failed wait the copy is let land and the products run on it (the
  // block stops after them): no branch around the loop's mma.sync
  if (!ok) mbar_drain(bar, 0);
  {
    int tok[NTMAX];  // column g of token tile nt is token 8 nt + g (past B: a repeat of token B - 1)
#pragma unroll
    for (int nt = 0; nt < NTMAX; ++nt) tok[nt] = min(nt * 8 + g, a.B - 1);
#pragma unroll 4
    for (int kl = 0; kl < KGW; ++kl) {
      const int kg = warp * KGW + kl;
      uint4 bx[NTMAX][2];
#pragma unroll
      for (int nt = 0; nt < NTMAX; ++nt) {
        if (NTMAX == 1 || nt < nt_used) {
          const uint8_t* rp = xs + (size_t)tok[nt] * xstride + kg * 128 + t4 * 32;
          bx[nt][0] = lds128(rp);
          bx[nt][1] = lds128(rp + 16);
        }
      }
      if (kl & 1)
        tile_kgroup<FMT, NTMAX>(wb + kl * KGB, bx, nt_used, lane, acc[1]);
      else
        tile_kgroup<FMT, NTMAX>(wb + kl * KGB, bx, nt_used, lane, acc[0]);
    }
  }
#pragma unroll
  for (int nt = 0; nt < NTMAX; ++nt)
#pragma unroll
    for (int i = 0; i < 4; ++i) red[((warp * NTMAX + nt) * 32 + lane) * 4 + i] = acc[0][nt][i] + acc[1][nt][i];
  if (!__syncthreads_and(ok)) return;
  // Output (row r of the tile, token t): token tile t / 8, fragment lane
  // 4 (r % 8) + (t % 8) / 2, element 2 (r / 8) + t % 2.
  const float G = FMT == FLINT_MOE_NVFP4 ? a.G[0] : 1.0f;
  for (int p = threadIdx.x; p < 16 * a.B; p += blockDim.x) {
    const int r = p & 15, t = p >> 4, nt = t >> 3, c = t & 7;
    const int ln = 4 * (r & 7) + (c >> 1), i = 2 * (r >> 3) + (c & 1);
    float v = 0.f;
    for (int w2 = 0; w2 < nw; ++w2) v += red[((w2 * NTMAX + nt) * 32 + ln) * 4 + i];
    const __nv_bfloat16 o = __float2bfloat16_rn((v * s_inv[t]) * G);
    a.y[(size_t)t * a.N + blockIdx.x * 16 + r] = *reinterpret_cast<const uint16_t*>(&o);
  }
}

// ===========================================================================
// The same GEMV split along K over a thread-block cluster, for K > 2048: the
// S = K / 2048 CTAs of a cluster share one tile of 16 output rows, each taking
// 2048 columns (its weights, its slice of x). Their partial sums meet in
// distributed shared memory and CTA 0 adds them in rank order (a fixed order,
// so the result does not depend on timing) and writes y. With a norm weight
// the rows' sums of squares are shared the same way before normalising.
// Each slice of x is staged from registers (8 16-byte chunks per lane): no
// serial passes over long rows.
// ===========================================================================
constexpr int GEMV_SLICE = 2048;

struct GemvSplitPlan {
  size_t wbuf_off, xs_off, red_off, part_off, ss_off, inv_off, bar_off, total;
};

__host__ __device__ inline GemvSplitPlan gemv_split_plan(int B, int fmt, int nw, int ntmax) {
  const int kgb = fmt == FLINT_MOE_NVFP4 ? KG_NVFP4 : KG_BF16;
  GemvSplitPlan p;
  size_t o = 0;
  p.wbuf_off = o;  o += (size_t)(GEMV_SLICE / KG_COLS) * kgb;
  p.xs_off = o;    o += (size_t)B * (GEMV_SLICE * 2 + 16);
  p.red_off = o;   o += sizeof(float) * nw * ntmax * 128;
  p.part_off = o;  o += sizeof(float) * MAX_BATCH * 16;
  p.ss_off = o;    o += sizeof(float) * MAX_BATCH;
  p.inv_off = o;   o += sizeof(float) * MAX_BATCH;
  o = (o + 15) & ~(size_t)15;
  p.bar_off = o;   o += sizeof(uint64_t) * nw;
  p.total = o;
  return p;
}

// SOLO (one token): at most 64 registers, four CTAs per SM, so that the grid
// (N / 16 row tiles x K / 2048 slices: 512 CTAs for 2048 x 8192) runs in one
// wave instead of two at three per SM (2048 x 8192: 7.4 -> 6.3 us per call).
template <int FMT, int NTMAX, bool SOLO = false>
__global__ void __launch_bounds__(256, SOLO ? 4 : 0) k_gemv_split(GemvArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  constexpr int KGB = FMT == FLINT_MOE_NVFP4 ? KG_NVFP4 : KG_BF16;
  constexpr int NCH = GEMV_SLICE / 256;  // 16-byte chunks per lane of a slice row
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t4 = lane & 3;
  const int nw = blockDim.x >> 5;
  const uint32_t rank = cluster_rank(), S = gridDim.y;
  const int KGW = (GEMV_SLICE / KG_COLS) / nw;  // k-groups per warp
  const GemvSplitPlan P = gemv_split_plan(a.B, FMT, nw, NTMAX);
  uint8_t* wb = smem + P.wbuf_off + (size_t)warp * KGW * KGB;
  uint8_t* xs = smem + P.xs_off;
  float* red = reinterpret_cast<float*>(smem + P.red_off);
  float* part = reinterpret_cast<float*>(smem + P.part_off);  // [B][16] this CTA's partial y
  float* s_ss = reinterpret_cast<float*>(smem + P.ss_off);    // [B] this slice's sums of squares
  float* s_inv = reinterpret_cast<float*>(smem + P.inv_off);  // [B] inverse prescale
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + P.bar_off) + warp;
  const int xstride = GEMV_SLICE * 2 + 16;
  const size_t col0 = (size_t)rank * GEMV_SLICE;
  if (lane == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
    const uint32_t bytes = (uint32_t)KGW * KGB;
    const int64_t off = (int64_t)blockIdx.x * a.L.dn_tile + (int64_t)rank * (GEMV_SLICE / KG_COLS) * KGB +
                        (int64_t)warp * bytes;
    mbar_arrive_expect_tx(bar, bytes);
    bulk_g2s_stream(wb, a.packed + off, bytes, bar);
  }
  pdl_wait();  // x may be the previous kernel's output
  pdl_trigger();
  // Stage this CTA's slice of every token row: warp w takes tokens w, w + nw, ...
  const int ntw = (a.B - warp + nw - 1) / nw;  // tokens of this warp: at most NTMAX with 8 warps
  uint4 v[NTMAX][NCH];
  float sq[NTMAX];
#pragma unroll
  for (int i = 0; i < NTMAX; ++i) {
    const int t = warp + i * nw;
    sq[i] = 0.f;
    if (i < ntw) {
      const uint8_t* src = reinterpret_cast<const uint8_t*>(a.x + (size_t)t * a.K + col0);
#pragma unroll
      for (int c = 0; c < NCH; ++c) v[i][c] = ld_cg_v4(src + (lane + 32 * c) * 16);
      if (a.prenorm) {
#pragma unroll
        for (int c = 0; c < NCH; ++c) sq[i] = sumsq8(v[i][c], sq[i]);
        sq[i] = warp_sum(sq[i]);
        if (lane == 0) s_ss[t] = sq[i];
      }
    }
  }
  if (a.prenorm) cluster_sync();  // every slice's sums of squares are published
#pragma unroll
  for (int i = 0; i < NTMAX; ++i) {
    const int t = warp + i * nw;
    if (i < ntw) {
      if (a.prenorm) {
        float ss = 0.f;
        for (uint32_t r = 0; r < S; ++r) ss += ld_dsmem_f32(s_ss + t, r);  // rank order
        const uint8_t* gw8 = reinterpret_cast<const uint8_t*>(a.gamma) + col0 * 2;
        if (ss <= FP32_MAX) {
          const float inv = 1.0f / sqrtf(ss / (float)a.K + a.eps);
#pragma unroll
          for (int c = 0; c < NCH; ++c)
            v[i][c] = norm8(v[i][c], __ldg(reinterpret_cast<const uint4*>(gw8 + (lane + 32 * c) * 16)), inv);
        } else {  // the sum of squares overflowed: the scaled path over the whole row
          const float2 f = rms_factor_huge(reinterpret_cast<const uint8_t*>(a.x + (size_t)t * a.K), 0, lane, a.K,
                                           a.eps);
#pragma unroll
          for (int c = 0; c < NCH; ++c)
            v[i][c] = norm8_huge(v[i][c], __ldg(reinterpret_cast<const uint4*>(gw8 + (lane + 32 * c) * 16)), f);
        }
      }
      int kx = 0;
      if (FMT == FLINT_MOE_NVFP4) {
        float mx = 0.f;
#pragma unroll
        for (int c = 0; c < NCH; ++c) mx = absmax8(v[i][c], mx);
        kx = prescale_exp(warp_max(mx));
      }
      const float sc = exp2i(kx);
      uint8_t* dst = xs + (size_t)t * xstride;
#pragma unroll
      for (int c = 0; c < NCH; ++c) {
        const uint32_t w4[4] = {v[i][c].x, v[i][c].y, v[i][c].z, v[i][c].w};
        const int col = 8 * (lane + 32 * c);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint32_t bits = w4[q];
          if (FMT == FLINT_MOE_NVFP4) {
            const __half2 hv = __floats2half2_rn(bf16lo(w4[q]) * sc, bf16hi(w4[q]) * sc);
            bits = *reinterpret_cast<const uint32_t*>(&hv);
          }
          *reinterpret_cast<uint32_t*>(dst + 2 * frag_offset_elems(col + 2 * q)) = bits;
        }
      }
      if (lane == 0) s_inv[t] = exp2i(-kx);
    }
  }
  __syncthreads();
  const int nt_used = (a.B + 7) >> 3;
  float acc[2][NTMAX][4];
#pragma unroll
  for (int c = 0; c < 2; ++c)
#pragma unroll
    for (int nt = 0; nt < NTMAX; ++nt)
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[c][nt][i] = 0.f;
  const bool ok = mbar_wait(bar, 0, a.status);
  // after a failed wait the copy is let land and the products run on it (the
  // block stops after them): no branch around the loop's mma.sync
  if (!ok) mbar_drain(bar, 0);
  {
    int tok[NTMAX];
#pragma unroll
    for (int nt = 0; nt < NTMAX; ++nt) tok[nt] = min(nt * 8 + g, a.B - 1);
#pragma unroll 4
    for (int kl = 0; kl < KGW; ++kl) {
      const int kg = warp * KGW + kl;
      uint4 bx[NTMAX][2];
#pragma unroll
      for (int nt = 0; nt < NTMAX; ++nt) {
        if (NTMAX == 1 || nt < nt_used) {
          const uint8_t* rp = xs + (size_t)tok[nt] * xstride + kg * 128 + t4 * 32;
          bx[nt][0] = lds128(rp);
          bx[nt][1] = lds128(rp + 16);
        }
      }
      if (kl & 1)
        tile_kgroup<FMT, NTMAX>(wb + kl * KGB, bx, nt_used, lane, acc[1]);
      else
        tile_kgroup<FMT, NTMAX>(wb + kl * KGB, bx, nt_used, lane, acc[0]);
    }
  }
#pragma unroll
  for (int nt = 0; nt < NTMAX; ++nt)
#pragma unroll
    for (int i = 0; i < 4; ++i) red[((warp * NTMAX + nt) * 32 + lane) * 4 + i] = acc[0][nt][i] + acc[1][nt][i];
  __syncthreads();
  // This CTA's partial sums (prescale undone), output (row r, token t) at [t][r].
  for (int p = threadIdx.x; p < 16 * a.B; p += blockDim.x) {
    const int r = p & 15, t = p >> 4, nt = t >> 3, c = t & 7;
    const int ln = 4 * (r & 7) + (c >> 1), i = 2 * (r >> 3) + (c & 1);
    float v2 = 0.f;
    for (int w2 = 0; w2 < nw; ++w2) v2 += red[((w2 * NTMAX + nt) * 32 + ln) * 4 + i];
    part[t * 16 + r] = v2 * s_inv[t];
  }
  cluster_sync();  // every CTA's partial sums are published
  if (rank == 0) {
    const float G = FMT == FLINT_MOE_NVFP4 ? a.G[0] : 1.0f;
    for (int p = threadIdx.x; p < 16 * a.B; p += blockDim.x) {
      float v2 = 0.f;
      for (uint32_t r = 0; r < S; ++r) v2 += ld_dsmem_f32(part + p, r);  // rank order
      const int rr = p & 15, t = p >> 4;
      const __nv_bfloat16 o = __float2bfloat16_rn(v2 * G);
      a.y[(size_t)t * a.N + blockIdx.x * 16 + rr] = *reinterpret_cast<const uint16_t*>(&o);
    }
  }
  cluster_sync();  // the other CTAs' shared memory stays until CTA 0 has read it
}

}  // namespace flint

using namespace flint;

// ===========================================================================
// Host side
// ===========================================================================
namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

constexpr size_t SMEM_LIMIT = 227 * 1024;

// Experts per router block: the four warps of a block split its tokens.
int router_epb(int B) { return B <= 1 ? 4 : (B == 2 ? 2 : 1); }
// Warps per router block: 4, so that a warp has at most 2 tokens of a chunk
// of 8 (nw / epb >= 4 token groups from 3 tokens on).
int router_warps(int B) { return 4; }

// Router rows of one block, the norm weight and one x chunk of up to 8 tokens.
size_t router_smem(int H, int B) { return (size_t)(router_epb(B) + 1 + (B < 8 ? B : 8)) * H * 2; }

// Down kernel shape: 8 warps with 3 or 2 tiles in flight each if they fit,
// else 4 warps; the rest of the budget stages h rows (all B (k + S) of them if
// possible). Small batches keep the block small enough to run beside a
// gate/up block, which lets it prefetch while k_gateup works.
bool down_shape(int I, int B, int k, int S, int max_slots, int fmt, size_t budget, DownPlan& out) {
  const int need = B * (k + S);
  // Up to 2 tokens the block must fit beside a gate/up block (8 warps at
  // most); from 3 tokens on it runs alone on its SM and takes 16 warps (20
  // measured slower: batch 8 42.6 against 37.0 us).
  const int cand[][2] = {{16, 2}, {8, 3}, {8, 2}, {4, 2}, {4, 1}};
  for (int i = B <= 2 ? 1 : 0; i < 5; ++i) {
    const auto& c = cand[i];
    const size_t base = down_plan(I, B, max_slots, fmt, c[0], c[1], 0).total;
    const size_t per_row = (size_t)(I * 2 + 16) + 8;
    if (base + 8 * per_row > budget) continue;
    const int fit = (int)((budget - base) / per_row);
    out = down_plan(I, B, max_slots, fmt, c[0], c[1], fit < need ? fit : need);
    if (out.total <= budget) return true;
  }
  return false;
}

// Static shared memory of a kernel (its __shared__ variables), from the runtime.
template <typename K>
size_t static_smem(K kernel) {
  cudaFuncAttributes at;
  if (cudaFuncGetAttributes(&at, kernel) != cudaSuccess) return 16 * 1024;
  return at.sharedSizeBytes;
}

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      n < 1)
    n = 148;
  return n;
}

template <typename K, typename Args>
cudaError_t launch_any(K kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t stream, const Args& a);

// The same launch with a cluster of (1, cy, 1) CTAs.
template <typename K, typename Args>
cudaError_t launch_cluster(K kernel, dim3 grid, dim3 block, size_t smem, int cy, cudaStream_t stream, const Args& a) {
  if (smem > 32 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = 1;
  attr[1].val.clusterDim.y = cy;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kernel, a);
}

template <typename K>
cudaError_t launch_pdl(K kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t stream, const DecodeArgs& a) {
  return launch_any(kernel, grid, block, smem, stream, a);
}

template <typename K, typename Args>
cudaError_t launch_any(K kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t stream, const Args& a) {
  // Above 48 KB of static plus dynamic shared memory a kernel must opt in; the
  // decode kernels' static shared memory stays under 16 KB, so opting in from
  // 32 KB of dynamic memory covers every case.
  if (smem > 32 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  // Every decode kernel asks for the largest shared-memory carveout: an SM runs
  // blocks of different kernels side by side only under one carveout, and the
  // early (programmatic) launch of the next kernel is only useful if its blocks
  // can be resident while the current kernel's blocks still run.
  {
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                         (int)cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, a);
}

// Warp groups (ng) and buffers per group (nb) of k_gateup: as many units in
// flight as fit, and for 1 and 2 tokens of NVFP4 weights a footprint that
// leaves room on each SM for a down block, which launches early and prefetches
// meanwhile (a BF16 unit is 3.6 times larger: there the gate/up block takes
// the SM's shared memory, as more units in flight measured faster).
void gateup_shape(int H, int B, int fmt, int units_per_block, int& ng, int& nb) {
  // static shared memory of the gate/up kernels, as laid out by the compiler
  static const size_t route =
      std::max({static_smem(k_gateup<FLINT_MOE_NVFP4, 1, false, -1>), static_smem(k_gateup<FLINT_MOE_NVFP4, 4, false, -1>),
                static_smem(k_gateup<FLINT_MOE_BF16, 1, false, -1>), static_smem(k_gateup<FLINT_MOE_BF16, 4, false, -1>),
                static_smem(k_gateup<FLINT_MOE_NVFP4, 1, true, 0>), static_smem(k_gateup<FLINT_MOE_NVFP4, 1, true, 1>),
                static_smem(k_gateup<FLINT_MOE_NVFP4, 1, true, 0, GATEUP_SMALL_REGS>),
                static_smem(k_gateup<FLINT_MOE_NVFP4, 1, true, 1, GATEUP_SMALL_REGS>),
                static_smem(k_gateup<FLINT_MOE_NVFP4, 4, true, -1>)});
  const int ntmax = (B + 7) / 8;
  const size_t budget = B <= 2 && fmt == FLINT_MOE_NVFP4 ? 110 * 1024 : SMEM_LIMIT;
  const int want_nb = units_per_block <= 3 ? 1 : 2;
  // Up to 2 tokens a gate/up block stays small (3 groups) so that a down block
  // runs beside it; larger batches take a fourth and fifth group of warps
  // (five groups of 4 warps at 96 registers fill the register file).
  const int first = B <= 2 && fmt == FLINT_MOE_NVFP4 ? 4 : 0;
  const int cand[][2] = {{5, want_nb}, {5, 1}, {4, want_nb}, {4, 1}, {3, want_nb}, {3, 1}, {2, 2}, {2, 1},
                         {1, 3},       {1, 2}, {1, 1}};
  for (int i = first; i < (int)(sizeof(cand) / sizeof(cand[0])); ++i) {
    const auto& c = cand[i];
    if (gateup_plan(H, B, fmt, ntmax, c[0], c[1]).total + route <= budget) {
      ng = c[0];
      nb = c[1];
      return;
    }
  }
  for (int i = first; i < (int)(sizeof(cand) / sizeof(cand[0])); ++i) {
    const auto& c = cand[i];
    if (gateup_plan(H, B, fmt, ntmax, c[0], c[1]).total + route <= SMEM_LIMIT) {
      ng = c[0];
      nb = c[1];
      return;
    }
  }
  ng = 0;
  nb = 0;
}

// The kernels for the Flint shape (E = 256, H = 2048, I = 512, top-6, one
// shared expert) are separate instantiations that carry no code for other shapes.
bool narrow_shape(const DecodeArgs& a) { return a.E == 256 && a.H == 2048 && a.I == 512 && a.k == 6 && a.S == 1; }

template <int FMT, bool NARROW>
cudaError_t launch_gateup_n(const DecodeArgs& a, cudaStream_t stream, int ng) {
  const int ntmax = (a.B + 7) / 8;
  const size_t smem = gateup_plan(a.H, a.B, FMT, ntmax, ng, a.gu_nb).total;
  const int units = a.W.max_slots * (a.I / 8);
  const int blocks = units < sm_count() ? units : sm_count();
  const dim3 block(128 * ng);
  switch (ntmax) {
    case 1:  // up to 8 tokens, the low-latency path: one instantiation per pre-norm case
      if constexpr (NARROW) {
        if (ng <= 3)
          return a.prenorm
                     ? launch_pdl(k_gateup<FMT, 1, NARROW, 1, GATEUP_SMALL_REGS>, dim3(blocks), block, smem, stream, a)
                     : launch_pdl(k_gateup<FMT, 1, NARROW, 0, GATEUP_SMALL_REGS>, dim3(blocks), block, smem, stream, a);
        return a.prenorm ? launch_pdl(k_gateup<FMT, 1, NARROW, 1>, dim3(blocks), block, smem, stream, a)
                         : launch_pdl(k_gateup<FMT, 1, NARROW, 0>, dim3(blocks), block, smem, stream, a);
      } else {
        return launch_pdl(k_gateup<FMT, 1, NARROW, -1>, dim3(blocks), block, smem, stream, a);
      }
    case 2: return launch_pdl(k_gateup<FMT, 2, NARROW, -1>, dim3(blocks), block, smem, stream, a);
    case 3: return launch_pdl(k_gateup<FMT, 3, NARROW, -1>, dim3(blocks), block, smem, stream, a);
    default: return launch_pdl(k_gateup<FMT, 4, NARROW, -1>, dim3(blocks), block, smem, stream, a);
  }
}

template <int FMT>
cudaError_t launch_gateup(const DecodeArgs& a, cudaStream_t stream, int ng) {
  return narrow_shape(a) ? launch_gateup_n<FMT, true>(a, stream, ng) : launch_gateup_n<FMT, false>(a, stream, ng);
}

template <int FMT>
cudaError_t launch_down(const DecodeArgs& a, cudaStream_t stream, const DownPlan& P) {
  return narrow_shape(a) ? launch_pdl(k_down<FMT, true>, dim3(a.H / 16), dim3(32 * P.nw), P.total, stream, a)
                         : launch_pdl(k_down<FMT, false>, dim3(a.H / 16), dim3(32 * P.nw), P.total, stream, a);
}

// Up to 2 tokens the block shares its SM with a gate/up block: 8 warps, two
// buffers each. From 3 tokens on it runs alone: 16 warps, one buffer each.
size_t down_items_smem(const DecodeArgs& a) {
  const bool wide = a.B >= 3;
  return down_items_plan(a.H, a.I, a.B, a.W.max_slots, a.fmt, wide ? DOWN_ITEMS_WIDE_NBUF : DOWN_ITEMS_NBUF,
                         wide ? DOWN_ITEMS_WIDE_NW : DOWN_ITEMS_NW)
      .total;
}

cudaError_t launch_router(const DecodeArgs& a, cudaStream_t stream) {
  const dim3 grid((a.E + a.router_epb - 1) / a.router_epb), block(32 * router_warps(a.B));
  const size_t smem = router_smem(a.H, a.B);
  switch (a.H / 256) {
    case 1: return launch_pdl(k_router<1, -1>, grid, block, smem, stream, a);
    case 2: return launch_pdl(k_router<2, -1>, grid, block, smem, stream, a);
    case 3: return launch_pdl(k_router<3, -1>, grid, block, smem, stream, a);
    case 4: return launch_pdl(k_router<4, -1>, grid, block, smem, stream, a);
    case 5: return launch_pdl(k_router<5, -1>, grid, block, smem, stream, a);
    case 6: return launch_pdl(k_router<6, -1>, grid, block, smem, stream, a);
    case 7: return launch_pdl(k_router<7, -1>, grid, block, smem, stream, a);
    case 8:  // the Flint shape: one instantiation per pre-norm case
      return a.prenorm ? launch_pdl(k_router<8, 1>, grid, block, smem, stream, a)
                       : launch_pdl(k_router<8, 0>, grid, block, smem, stream, a);
    case 16: return launch_pdl(k_router<16, -1>, grid, block, smem, stream, a);
    case 24: return launch_pdl(k_router<24, -1>, grid, block, smem, stream, a);
    case 32: return launch_pdl(k_router<32, -1>, grid, block, smem, stream, a);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

extern "C" size_t flint_moe_workspace_bytes(const flint_moe_config* c, int32_t max_batch) {
  if (flint_moe_check_config(c) != FLINT_MOE_OK || max_batch < 1 || max_batch > MAX_BATCH) return 0;
  // A call of B <= max_batch tokens lays the workspace out for its own B: the
  // largest layout is that of max_batch, or of 8 tokens where those carry the
  // f16 copy of h and max_batch does not.
  const int b8 = max_batch < 8 ? max_batch : 8;
  const size_t t1 = make_ws_layout(c->hidden, c->num_experts, c->top_k, c->inter, c->n_shared, max_batch,
                                   ws_wants_h16(max_batch, c->weight_fmt)).total;
  const size_t t2 = make_ws_layout(c->hidden, c->num_experts, c->top_k, c->inter, c->n_shared, b8,
                                   ws_wants_h16(b8, c->weight_fmt)).total;
  return t1 > t2 ? t1 : t2;
}

extern "C" flint_moe_status flint_moe_workspace_init(const flint_moe_config* c, int32_t max_batch, void* ws,
                                                     cudaStream_t stream) {
  const size_t bytes = flint_moe_workspace_bytes(c, max_batch);
  if (!bytes || !ws) return FLINT_MOE_EINVAL;
  if (!aligned16(ws)) return FLINT_MOE_EALIGN;
  return cudaMemsetAsync(ws, 0, bytes, stream) == cudaSuccess ? FLINT_MOE_OK : FLINT_MOE_ECUDA;
}

extern "C" flint_moe_status flint_moe_layer_init(const flint_moe_config* c, const void* packed,
                                                 const uint16_t* router, const float* sel_bias,
                                                 flint_moe_layer* out) {
  const flint_moe_status st = flint_moe_check_config(c);
  if (st != FLINT_MOE_OK) return st;
  if (!packed || !router || !out) return FLINT_MOE_EINVAL;
  if (!aligned16(packed) || !aligned16(router)) return FLINT_MOE_EALIGN;
  out->cfg = *c;
  out->packed = packed;
  out->router = router;
  out->sel_bias = sel_bias;
  out->norm_weight = nullptr;
  out->norm_eps = 0.f;
  return FLINT_MOE_OK;
}

extern "C" flint_moe_status flint_moe_layer_set_norm(flint_moe_layer* layer, const uint16_t* w, float eps) {
  if (!layer || !w || !(eps >= 0.f) || !(eps <= 3.0e38f)) return FLINT_MOE_EINVAL;
  if (!aligned16(w)) return FLINT_MOE_EALIGN;
  layer->norm_weight = w;
  layer->norm_eps = eps;
  return FLINT_MOE_OK;
}

namespace {
flint_moe_status decode_impl(const flint_moe_layer* layer, const uint16_t* x, int32_t B, uint16_t* out, void* ws,
                             cudaStream_t stream, bool prenorm);
}  // namespace

extern "C" flint_moe_status flint_moe_decode(const flint_moe_layer* layer, const uint16_t* x, int32_t B,
                                             uint16_t* out, void* ws, cudaStream_t stream) {
  return decode_impl(layer, x, B, out, ws, stream, false);
}

extern "C" flint_moe_status flint_moe_decode_prenorm(const flint_moe_layer* layer, const uint16_t* r_in, int32_t B,
                                                     uint16_t* r_out, void* ws, cudaStream_t stream) {
  if (!layer || !layer->norm_weight) return FLINT_MOE_EINVAL;
  return decode_impl(layer, r_in, B, r_out, ws, stream, true);
}

namespace {
flint_moe_status decode_impl(const flint_moe_layer* layer, const uint16_t* x, int32_t B, uint16_t* out, void* ws,
                             cudaStream_t stream, bool prenorm) {
  if (!layer) return FLINT_MOE_EINVAL;
  const flint_moe_config* c = &layer->cfg;
  const flint_moe_status st = flint_moe_check_config(c);
  if (st != FLINT_MOE_OK) return st;
  if (B < 0 || B > MAX_BATCH) return FLINT_MOE_EINVAL;
  if (B == 0) return FLINT_MOE_OK;
  if (!x || !out || !ws || !layer->packed || !layer->router) return FLINT_MOE_EINVAL;
  if (!aligned16(x) || !aligned16(out) || !aligned16(ws) || !aligned16(layer->packed) || !aligned16(layer->router))
    return FLINT_MOE_EALIGN;
  DecodeArgs a;
  a.H = c->hidden;
  a.I = c->inter;
  a.E = c->num_experts;
  a.S = c->n_shared;
  a.k = c->top_k;
  a.B = B;
  a.fmt = c->weight_fmt;
  a.renorm = c->renormalize != 0;
  a.routed_scale = c->routed_scale;
  a.x = x;
  a.out = out;
  a.router = layer->router;
  a.bias = layer->sel_bias;
  a.packed = static_cast<const uint8_t*>(layer->packed);
  a.L = make_layout(a.H, a.I, a.E, a.S, a.fmt);
  a.globals = reinterpret_cast<const float*>(a.packed + a.L.globals_off);
  a.ws = static_cast<uint8_t*>(ws);
  // The workspace is laid out for the batch of this call; callers size it for
  // their largest batch, which is at least as large.
  a.W = make_ws_layout(a.H, a.E, a.k, a.I, a.S, B, ws_wants_h16(B, a.fmt));
  a.prenorm = prenorm ? 1 : 0;
  a.router_epb = router_epb(B);
  // x and out may be device memory or pinned (device-mapped) host memory;
  // memory the device cannot address is refused before any launch.
  bool x_host = false;
  {
    cudaPointerAttributes px, po;
    if (cudaPointerGetAttributes(&px, x) != cudaSuccess || cudaPointerGetAttributes(&po, out) != cudaSuccess)
      return FLINT_MOE_EINVAL;
    auto addressable = [](const cudaPointerAttributes& p) {
      return p.type == cudaMemoryTypeDevice || p.type == cudaMemoryTypeManaged ||
             (p.type == cudaMemoryTypeHost && p.devicePointer == p.hostPointer);
    };
    if (!addressable(px) || !addressable(po)) return FLINT_MOE_EINVAL;
    x_host = px.type == cudaMemoryTypeHost;
  }
  a.gamma = prenorm ? layer->norm_weight : nullptr;
  a.eps = prenorm ? layer->norm_eps : 0.f;
  if (prenorm && !aligned16(a.gamma)) return FLINT_MOE_EALIGN;
#ifdef FLINT_MOE_TRACE
  static std::atomic<int> trace_calls{0};
  a.trace_seq = trace_calls.fetch_add(1);
#else
  a.trace_seq = 0;
#endif
  // Static shared memory of the down kernels (the routing, the warp sums, the
  // residual values), as the compiler laid it out: static plus dynamic must
  // stay within the per-block limit.
  static const size_t route_smem =
      std::max({static_smem(k_down<FLINT_MOE_NVFP4, false>), static_smem(k_down<FLINT_MOE_BF16, false>),
                static_smem(k_down<FLINT_MOE_NVFP4, true>),
                static_smem(k_down_items<FLINT_MOE_NVFP4, DOWN_ITEMS_NBUF, false, -1>),
                static_smem(k_down_items<FLINT_MOE_NVFP4, DOWN_ITEMS_WIDE_NBUF, false, -1>),
                static_smem(k_down_items<FLINT_MOE_NVFP4, DOWN_ITEMS_NBUF, true, 0>),
                static_smem(k_down_items<FLINT_MOE_NVFP4, DOWN_ITEMS_NBUF, true, 1>),
                static_smem(k_down_items<FLINT_MOE_NVFP4, DOWN_ITEMS_WIDE_NBUF, true, 0>),
                static_smem(k_down_items<FLINT_MOE_NVFP4, DOWN_ITEMS_WIDE_NBUF, true, 1>)});
  int gu_ng = 0;
  {
    const int units = a.W.max_slots * (a.I / 8), sms = sm_count();
    gateup_shape(a.H, B, a.fmt, (units + sms - 1) / sms, gu_ng, a.gu_nb);
  }
  DownPlan dp;
  const size_t down_budget = (B <= 2 && a.fmt == FLINT_MOE_NVFP4 ? 110 * 1024 : SMEM_LIMIT) - route_smem;
  if (gu_ng == 0 || !down_shape(a.I, B, a.k, a.S, a.W.max_slots, a.fmt, down_budget, dp) ||
      router_smem(a.H, B) > SMEM_LIMIT)
    return FLINT_MOE_EUNSUPPORTED;
  a.dn_nbuf = dp.nbuf;
  a.dn_hcap = dp.hcap;
  const bool small_down = B <= 8 && a.fmt == FLINT_MOE_NVFP4 && down_items_smem(a) <= down_budget;
  cudaError_t e = cudaSuccess;
  if (x_host) {  // one copy of x into the workspace, which the layer's kernels read
    const int words = B * a.H / 8;
    e = launch_pdl(k_stage_x, dim3((words + 255) / 256), dim3(256), 0, stream, a);
    a.x = reinterpret_cast<const uint16_t*>(a.ws + a.W.xs);
  }
  // The router and gate/up kernels' arguments: from NORM_KERNEL_MIN_B
  // pre-norm tokens they read the rows k_norm_x normalised, as plain
  // activations; the down kernel keeps x as the residual it adds.
  DecodeArgs an = a;
  if (e == cudaSuccess && prenorm && B >= NORM_KERNEL_MIN_B) {
    e = launch_pdl(k_norm_x, dim3((B + 3) / 4), dim3(128), 0, stream, a);
    an.x = reinterpret_cast<const uint16_t*>(a.ws + a.W.xn);
    an.prenorm = 0;
    an.gamma = nullptr;
  }
  if (e == cudaSuccess) e = launch_router(an, stream);
  if (e == cudaSuccess) e = a.fmt == FLINT_MOE_NVFP4 ? launch_gateup<FLINT_MOE_NVFP4>(an, stream, gu_ng)
                                                       : launch_gateup<FLINT_MOE_BF16>(an, stream, gu_ng);
  if (e == cudaSuccess) {
    const bool nar = narrow_shape(a);
    const size_t dsm = down_items_smem(a);
    const dim3 grid(a.H / 16), wide_blk(32 * DOWN_ITEMS_WIDE_NW), blk(32 * DOWN_ITEMS_NW);
    if (small_down && B >= 3)
      e = !nar     ? launch_pdl(k_down_items<FLINT_MOE_NVFP4, DOWN_ITEMS_WIDE_NBUF, false, -1>, grid, wide_blk, dsm,
                                stream, a)
          : prenorm ? launch_pdl(k_down_items<FLINT_MOE_NVFP4, DOWN_ITEMS_WIDE_NBUF, true, 1>, grid, wide_blk, dsm,
                                 stream, a)
                    : launch_pdl(k_down_items<FLINT_MOE_NVFP4, DOWN_ITEMS_WIDE_NBUF, true, 0>, grid, wide_blk, dsm,
                                 stream, a);
    else if (small_down)
      e = !nar     ? launch_pdl(k_down_items<FLINT_MOE_NVFP4, DOWN_ITEMS_NBUF, false, -1>, grid, blk, dsm, stream, a)
          : prenorm ? launch_pdl(k_down_items<FLINT_MOE_NVFP4, DOWN_ITEMS_NBUF, true, 1>, grid, blk, dsm, stream, a)
                    : launch_pdl(k_down_items<FLINT_MOE_NVFP4, DOWN_ITEMS_NBUF, true, 0>, grid, blk, dsm, stream, a);
    else
      e = a.fmt == FLINT_MOE_NVFP4 ? launch_down<FLINT_MOE_NVFP4>(a, stream, dp)
                                   : launch_down<FLINT_MOE_BF16>(a, stream, dp);
  }
  return e == cudaSuccess ? FLINT_MOE_OK : FLINT_MOE_ECUDA;
}
}  // namespace

extern "C" flint_moe_status flint_moe_trace(int32_t op, uint64_t* host_events, cudaStream_t stream) {
#ifdef FLINT_MOE_TRACE
  if (op == 0) {
    static unsigned long long init[TRACE_CALLS][TRACE_EVENTS][2];
    for (int c = 0; c < TRACE_CALLS; ++c)
      for (int e = 0; e < TRACE_EVENTS; ++e) {
        init[c][e][0] = ~0ull;
        init[c][e][1] = 0ull;
      }
    return cudaMemcpyToSymbolAsync(g_trace, init, sizeof(init), 0, cudaMemcpyHostToDevice, stream) == cudaSuccess
               ? FLINT_MOE_OK
               : FLINT_MOE_ECUDA;
  }
  if (op == 1 && host_events) {
    if (cudaMemcpyFromSymbolAsync(host_events, g_trace, sizeof(g_trace), 0, cudaMemcpyDeviceToHost, stream) !=
            cudaSuccess ||
        cudaStreamSynchronize(stream) != cudaSuccess)
      return FLINT_MOE_ECUDA;
    return FLINT_MOE_OK;
  }
  return FLINT_MOE_EINVAL;
#else
  (void)op;
  (void)host_events;
  (void)stream;
  return FLINT_MOE_EUNSUPPORTED;
#endif
}

extern "C" flint_moe_status flint_moe_debug_routing(const flint_moe_config* c, const void* ws, int32_t B,
                                                    int32_t* idx, float* w, cudaStream_t stream) {
  if (flint_moe_check_config(c) != FLINT_MOE_OK || !ws || !idx || !w || B < 1 || B > MAX_BATCH)
    return FLINT_MOE_EINVAL;
  const WsLayout W = make_ws_layout(c->hidden, c->num_experts, c->top_k, c->inter, c->n_shared, B,
                                    ws_wants_h16(B, c->weight_fmt));
  const uint8_t* base = static_cast<const uint8_t*>(ws);
  const size_t n = (size_t)B * c->top_k;
  if (cudaMemcpyAsync(idx, base + W.topk_idx, n * sizeof(int), cudaMemcpyDeviceToDevice, stream) != cudaSuccess)
    return FLINT_MOE_ECUDA;
  if (cudaMemcpyAsync(w, base + W.topk_w, n * sizeof(float), cudaMemcpyDeviceToDevice, stream) != cudaSuccess)
    return FLINT_MOE_ECUDA;
  return FLINT_MOE_OK;
}

namespace {
__global__ void k_rcp_check(uint32_t lo, uint32_t hi, unsigned long long* bad) {
  unsigned long long nb = 0;
  for (uint64_t i = lo + (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; i < hi; i += (uint64_t)gridDim.x * blockDim.x) {
    const float y = __uint_as_float((uint32_t)i);
    if (__float_as_uint(rcp_nr(y)) != __float_as_uint(1.0f / y)) ++nb;
  }
  if (nb) atomicAdd(bad, nb);
}
}  // namespace

extern "C" flint_moe_status flint_moe_debug_rcp_check(uint32_t lo_bits, uint32_t hi_bits,
                                                      uint64_t* host_mismatches, cudaStream_t stream) {
  const uint32_t one = 0x3F800000u, top = (127u + 125u) << 23;  // 1.0f, 2^125
  if (!host_mismatches || lo_bits < one || hi_bits > top || lo_bits > hi_bits) return FLINT_MOE_EINVAL;
  unsigned long long* d = nullptr;
  if (cudaMallocAsync(&d, sizeof(*d), stream) != cudaSuccess) return FLINT_MOE_ECUDA;
  cudaError_t e = cudaMemsetAsync(d, 0, sizeof(*d), stream);
  if (e == cudaSuccess && hi_bits > lo_bits) {
    k_rcp_check<<<sm_count() * 8, 256, 0, stream>>>(lo_bits, hi_bits, d);
    e = cudaGetLastError();
  }
  unsigned long long h = 0;
  if (e == cudaSuccess) e = cudaMemcpyAsync(&h, d, sizeof(h), cudaMemcpyDeviceToHost, stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  cudaFreeAsync(d, stream);
  *host_mismatches = h;
  return e == cudaSuccess ? FLINT_MOE_OK : FLINT_MOE_ECUDA;
}

// One block waits on an mbarrier that nothing completes: the bounded wait of
// every kernel gives up, records the timeout and the block returns.
__global__ void k_wait_timeout(int* status) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  mbar_wait(&bar, 0, status);
}

extern "C" flint_moe_status flint_moe_debug_wait_timeout(int32_t* dev_status, cudaStream_t stream) {
  if (!dev_status) return FLINT_MOE_EINVAL;
  k_wait_timeout<<<1, 64, 0, stream>>>(dev_status);
  return cudaGetLastError() == cudaSuccess ? FLINT_MOE_OK : FLINT_MOE_ECUDA;
}

extern "C" flint_moe_status flint_gemv(const void* packed, int32_t N, int32_t K, int32_t fmt, const uint16_t* x,
                                       int32_t B, uint16_t* y, const uint16_t* norm_weight, float eps,
                                       int32_t* dev_status, cudaStream_t stream) {
  if (flint_gemv_packed_bytes(N, K, fmt) == 0) return FLINT_MOE_EUNSUPPORTED;
  if (B < 0 || B > MAX_BATCH || !(eps >= 0.f) || !(eps <= 3.0e38f)) return FLINT_MOE_EINVAL;
  if (B == 0) return FLINT_MOE_OK;
  if (!packed || !x || !y) return FLINT_MOE_EINVAL;
  if (!aligned16(packed) || !aligned16(x) || !aligned16(y) || (norm_weight && !aligned16(norm_weight)))
    return FLINT_MOE_EALIGN;
  GemvArgs a;
  a.N = N;
  a.K = K;
  a.B = B;
  a.fmt = fmt;
  a.prenorm = norm_weight != nullptr;
  a.x = x;
  a.y = y;
  a.packed = static_cast<const uint8_t*>(packed);
  a.L = make_dense_layout(N, K, fmt);
  a.G = reinterpret_cast<const float*>(a.packed + a.L.globals_off + 8);  // [G, G, G, 0]: the third word
  a.gamma = norm_weight;
  a.eps = eps;
  a.status = dev_status;
  const int kg = K / KG_COLS, nw = kg % 8 == 0 ? 8 : 4, ntmax = (B + 7) / 8;
  if (K > GEMV_SLICE) {  // split along K over a cluster of K / 2048 CTAs
    const int S = K / GEMV_SLICE;
    const size_t smem = gemv_split_plan(B, fmt, 8, ntmax).total;
    if (smem > SMEM_LIMIT) return FLINT_MOE_EUNSUPPORTED;
    const dim3 grid(N / 16, S), block(256);
    cudaError_t e;
    if (fmt == FLINT_MOE_NVFP4) {
      switch (B == 1 ? 0 : ntmax) {
        case 0: e = launch_cluster(k_gemv_split<FLINT_MOE_NVFP4, 1, true>, grid, block, smem, S, stream, a); break;
        case 1: e = launch_cluster(k_gemv_split<FLINT_MOE_NVFP4, 1>, grid, block, smem, S, stream, a); break;
        case 2: e = launch_cluster(k_gemv_split<FLINT_MOE_NVFP4, 2>, grid, block, smem, S, stream, a); break;
        case 3: e = launch_cluster(k_gemv_split<FLINT_MOE_NVFP4, 3>, grid, block, smem, S, stream, a); break;
        default: e = launch_cluster(k_gemv_split<FLINT_MOE_NVFP4, 4>, grid, block, smem, S, stream, a); break;
      }
    } else {
      switch (B == 1 ? 0 : ntmax) {
        case 0: e = launch_cluster(k_gemv_split<FLINT_MOE_BF16, 1, true>, grid, block, smem, S, stream, a); break;
        case 1: e = launch_cluster(k_gemv_split<FLINT_MOE_BF16, 1>, grid, block, smem, S, stream, a); break;
        case 2: e = launch_cluster(k_gemv_split<FLINT_MOE_BF16, 2>, grid, block, smem, S, stream, a); break;
        case 3: e = launch_cluster(k_gemv_split<FLINT_MOE_BF16, 3>, grid, block, smem, S, stream, a); break;
        default: e = launch_cluster(k_gemv_split<FLINT_MOE_BF16, 4>, grid, block, smem, S, stream, a); break;
      }
    }
    return e == cudaSuccess ? FLINT_MOE_OK : FLINT_MOE_ECUDA;
  }
  size_t o1, o2, o3, o4, o5;
  const size_t smem = gemv_smem(K, B, fmt, nw, ntmax, &o1, &o2, &o3, &o4, &o5);
  if ((size_t)B * (K * 2 + 16) > 160 * 1024 || smem > SMEM_LIMIT) return FLINT_MOE_EUNSUPPORTED;
  const dim3 grid(N / 16), block(32 * nw);
  cudaError_t e;
  if (fmt == FLINT_MOE_NVFP4) {
    switch (ntmax) {
      case 1: e = launch_any(k_gemv<FLINT_MOE_NVFP4, 1>, grid, block, smem, stream, a); break;
      case 2: e = launch_any(k_gemv<FLINT_MOE_NVFP4, 2>, grid, block, smem, stream, a); break;
      case 3: e = launch_any(k_gemv<FLINT_MOE_NVFP4, 3>, grid, block, smem, stream, a); break;
      default: e = launch_any(k_gemv<FLINT_MOE_NVFP4, 4>, grid, block, smem, stream, a); break;
    }
  } else {
    switch (ntmax) {
      case 1: e = launch_any(k_gemv<FLINT_MOE_BF16, 1>, grid, block, smem, stream, a); break;
      case 2: e = launch_any(k_gemv<FLINT_MOE_BF16, 2>, grid, block, smem, stream, a); break;
      case 3: e = launch_any(k_gemv<FLINT_MOE_BF16, 3>, grid, block, smem, stream, a); break;
      default: e = launch_any(k_gemv<FLINT_MOE_BF16, 4>, grid, block, smem, stream, a); break;
    }
  }
  return e == cudaSuccess ? FLINT_MOE_OK : FLINT_MOE_ECUDA;
}

extern "C" flint_moe_status flint_moe_read_status(const void* ws, int32_t* host_status, cudaStream_t stream) {
  if (!ws || !host_status) return FLINT_MOE_EINVAL;
  int32_t v = 0;
  int32_t* dev = static_cast<int32_t*>(const_cast<void*>(ws)) + HDR_STATUS;
  if (cudaMemcpyAsync(&v, dev, sizeof(int32_t), cudaMemcpyDeviceToHost, stream) != cudaSuccess) return FLINT_MOE_ECUDA;
  if (cudaMemsetAsync(dev, 0, sizeof(int32_t), stream) != cudaSuccess) return FLINT_MOE_ECUDA;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return FLINT_MOE_ECUDA;
  *host_status = v;
  return (v & FLINT_MOE_DEV_ERR_TIMEOUT) ? FLINT_MOE_ETIMEOUT : FLINT_MOE_OK;
}

// ===========================================================================
// Decode without a caller-provided workspace.
//
// Some callers cannot allocate device memory for a workspace: a plugin whose
// host application owns every device allocation and exposes no allocator, or
// a latency-critical loop where cudaMalloc / cudaFree could synchronise the
// device and stall other work. For them the decode's scratch lives in one
// file-scope device array instead. Every GPU that loads this library keeps
// the array (FLINT_MOE_NOALLOC_SCRATCH_BYTES bytes) until the process exits.
// ===========================================================================
#include <mutex>

static __device__ __align__(256) uint8_t g_noalloc_scratch[FLINT_MOE_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mutex;
void* g_noalloc_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device. The host-side
// symbol is only a stand-in; the address is looked up once per device. The
// lookup is not a stream operation, so it is refused (EINVAL) while `stream`
// is being captured into a CUDA graph.
flint_moe_status noalloc_scratch(cudaStream_t stream, void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FLINT_MOE_ECUDA;
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  if (!g_noalloc_ptr[dev]) {
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cap) != cudaSuccess) return FLINT_MOE_ECUDA;
    if (cap != cudaStreamCaptureStatusNone) return FLINT_MOE_EINVAL;
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return FLINT_MOE_ECUDA;
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return FLINT_MOE_OK;
}

// Moves the status word of the scratch header into the caller's word (OR),
// then clears it. Device code names the array directly.
__global__ void k_noalloc_status(int32_t* dev_status) {
  int* hdr = reinterpret_cast<int*>(g_noalloc_scratch);
  const int v = hdr[HDR_STATUS];
  if (v) atomicOr(dev_status, v);
  hdr[HDR_STATUS] = 0;
}

}  // namespace

extern "C" flint_moe_status flint_moe_decode_noalloc(const flint_moe_layer* layer, const uint16_t* x, int32_t B,
                                                     uint16_t* out, int32_t* dev_status, cudaStream_t stream) {
  if (!layer) return FLINT_MOE_EINVAL;
  const flint_moe_config* c = &layer->cfg;
  const flint_moe_status st = flint_moe_check_config(c);
  if (st != FLINT_MOE_OK) return st;
  if (B < 0 || B > MAX_BATCH) return FLINT_MOE_EINVAL;
  if (B == 0) return FLINT_MOE_OK;
  if (make_ws_layout(c->hidden, c->num_experts, c->top_k, c->inter, c->n_shared, B, ws_wants_h16(B, c->weight_fmt))
          .total >
      FLINT_MOE_NOALLOC_SCRATCH_BYTES)
    return FLINT_MOE_EUNSUPPORTED;
  if (!x || !out) return FLINT_MOE_EINVAL;
  if (dev_status && (reinterpret_cast<uintptr_t>(dev_status) & 3)) return FLINT_MOE_EALIGN;
  void* scratch = nullptr;
  const flint_moe_status sst = noalloc_scratch(stream, &scratch);
  if (sst != FLINT_MOE_OK) return sst;
  // The header (routing counter, status word) must start at zero.
  if (cudaMemsetAsync(scratch, 0, 256, stream) != cudaSuccess) return FLINT_MOE_ECUDA;
  const flint_moe_status dst = flint_moe_decode(layer, x, B, out, scratch, stream);
  if (dst != FLINT_MOE_OK || !dev_status) return dst;
  k_noalloc_status<<<1, 1, 0, stream>>>(dev_status);
  return cudaGetLastError() == cudaSuccess ? FLINT_MOE_OK : FLINT_MOE_ECUDA;
}
