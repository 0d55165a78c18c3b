// Decode step of the Flint-style W4A16 MoE layer on sm_103a: three kernels
// chained with programmatic dependent launch.
//
//   k_router   logits = x Wr^T (FP32 accumulation), then the last block to
//              finish computes sigmoid, top-k, the routing weights and the
//              "slots": the distinct experts the batch selected (ascending
//              expert id) after the always-on shared experts, each with its
//              list of (token, weight) rows.
//   k_gateup   one block per (slot, 8 intermediate rows): bulk-copies the
//              slot's packed gate/up tile into shared memory, dequantises it
//              into tensor-core fragments and writes h = bf16(silu(g) * u).
//   k_down     one block per 16 output rows: for every slot, bulk-copies the
//              down tile and the slot's h rows, multiplies, and accumulates
//              w * y in a fixed slot order; writes out = bf16(sum).
//
// "Day-0 Support for Flint on vLLM", section "Optimisation": the small-batch
// MoE kernels read only the selected experts' weights; routing and the expert
// combine are fused into the adjacent GEMV kernels; every kernel is launched
// with programmatic dependent launch so it fetches its routing-independent
// weights (router rows, shared expert) while the previous kernel still runs.
#include <cmath>

#include "common.cuh"

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
};

__device__ __forceinline__ int* ws_hdr(const DecodeArgs& a) { return reinterpret_cast<int*>(a.ws); }
__device__ __forceinline__ float* ws_logits(const DecodeArgs& a) { return reinterpret_cast<float*>(a.ws + a.W.logits); }
__device__ __forceinline__ int* ws_topk_idx(const DecodeArgs& a) { return reinterpret_cast<int*>(a.ws + a.W.topk_idx); }
__device__ __forceinline__ float* ws_topk_w(const DecodeArgs& a) { return reinterpret_cast<float*>(a.ws + a.W.topk_w); }
__device__ __forceinline__ int* ws_slot_expert(const DecodeArgs& a) { return reinterpret_cast<int*>(a.ws + a.W.slot_expert); }
__device__ __forceinline__ int* ws_slot_off(const DecodeArgs& a) { return reinterpret_cast<int*>(a.ws + a.W.slot_off); }
__device__ __forceinline__ int* ws_row_tok(const DecodeArgs& a) { return reinterpret_cast<int*>(a.ws + a.W.row_tok); }
__device__ __forceinline__ float* ws_row_w(const DecodeArgs& a) { return reinterpret_cast<float*>(a.ws + a.W.row_w); }
__device__ __forceinline__ unsigned* ws_hmax(const DecodeArgs& a) { return reinterpret_cast<unsigned*>(a.ws + a.W.hmax); }
__device__ __forceinline__ uint16_t* ws_h(const DecodeArgs& a) { return reinterpret_cast<uint16_t*>(a.ws + a.W.h); }

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
// Routing: sigmoid, top-k, weights and slots. Run by the last router block.
// ===========================================================================
struct RouteSmem {
  uint32_t mask[MAX_EXPERTS];   // token bitmask per expert
  int rank[MAX_EXPERTS];        // slot rank of a used expert
  int rowoff[MAX_EXPERTS];      // first row of its token list (relative)
  int idx[MAX_BATCH * MAX_TOPK];
  float w[MAX_BATCH * MAX_TOPK];
  int scan[4];
};

__device__ void route_and_slots(const DecodeArgs& a, RouteSmem& sm) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int B = a.B, E = a.E, k = a.k, S = a.S;
  for (int i = threadIdx.x; i < E; i += blockDim.x) sm.mask[i] = 0;
  __syncthreads();
  const float* lg = ws_logits(a);
  for (int t = warp; t < B; t += 4) {
    float key[MAX_EXPERTS / 32], sc[MAX_EXPERTS / 32];
#pragma unroll
    for (int j = 0; j < MAX_EXPERTS / 32; ++j) {
      const int e = lane + 32 * j;
      key[j] = -INFINITY;
      sc[j] = 0.f;
      if (e < E) {
        const float l = __ldcg(lg + t * E + e);
        const float s = 1.0f / (1.0f + expf(-l));
        sc[j] = s;
        key[j] = a.bias ? s + a.bias[e] : s;
      }
    }
    int my_e = 0;
    float my_s = 0.f, ssum = 0.f;
    for (int r = 0; r < k; ++r) {
      float bk = -INFINITY, bs = 0.f;
      int be = 0x7fffffff;
#pragma unroll
      for (int j = 0; j < MAX_EXPERTS / 32; ++j) {
        if (key[j] > bk) {  // strictly greater: the lowest index wins ties
          bk = key[j];
          be = lane + 32 * j;
          bs = sc[j];
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float ok = __shfl_xor_sync(0xffffffffu, bk, o);
        const int oe = __shfl_xor_sync(0xffffffffu, be, o);
        const float os = __shfl_xor_sync(0xffffffffu, bs, o);
        if (ok > bk || (ok == bk && oe < be)) {
          bk = ok;
          be = oe;
          bs = os;
        }
      }
#pragma unroll
      for (int j = 0; j < MAX_EXPERTS / 32; ++j)
        if (lane + 32 * j == be) key[j] = -INFINITY;
      if (be >= E) {  // only reachable with non-finite logits; keep every index in range
        if (lane == 0) atomicOr(ws_hdr(a) + HDR_STATUS, FLINT_MOE_DEV_ERR_SLOTS);
        be = r;
        bs = 0.f;
      }
      if (lane == r) {
        my_e = be;
        my_s = bs;
      }
      ssum += bs;
    }
    if (lane < k) {
      float w = a.renorm ? my_s / ssum : my_s;
      w *= a.routed_scale;
      ws_topk_idx(a)[t * k + lane] = my_e;
      ws_topk_w(a)[t * k + lane] = w;
      sm.idx[t * k + lane] = my_e;
      sm.w[t * k + lane] = w;
      atomicOr(&sm.mask[my_e], 1u << t);
    }
  }
  __syncthreads();

  // Exclusive scan over experts of (used << 16 | token count): slot rank and row offset.
  const int ept = (E + blockDim.x - 1) / blockDim.x;
  const int e0 = threadIdx.x * ept;
  int local = 0;
  for (int e = e0; e < e0 + ept && e < E; ++e) {
    const uint32_t m = sm.mask[e];
    local += m ? (1 << 16) | __popc(m) : 0;
  }
  int incl = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += n;
  }
  if (lane == 31) sm.scan[warp] = incl;
  __syncthreads();
  int warp_off = 0;
  for (int w2 = 0; w2 < warp; ++w2) warp_off += sm.scan[w2];
  const int total = sm.scan[0] + sm.scan[1] + sm.scan[2] + sm.scan[3];
  int run = warp_off + incl - local;
  int* slot_expert = ws_slot_expert(a);
  int* slot_off = ws_slot_off(a);
  for (int e = e0; e < e0 + ept && e < E; ++e) {
    const uint32_t m = sm.mask[e];
    if (m) {
      const int rank = run >> 16, roff = run & 0xFFFF;
      sm.rank[e] = rank;
      sm.rowoff[e] = roff;
      slot_expert[S + rank] = e;
      slot_off[S + rank] = S * B + roff;
      run += (1 << 16) | __popc(m);
    }
  }
  const int D = total >> 16, R = total & 0xFFFF;
  const int n_slots = S + D, n_rows = S * B + R;
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      slot_expert[s] = E + s;
      slot_off[s] = s * B;
    }
    slot_off[n_slots] = n_rows;
    int* hdr = ws_hdr(a);
    hdr[HDR_NSLOTS] = n_slots;
    hdr[HDR_NROWS] = n_rows;
    hdr[HDR_BATCH] = B;
  }
  __syncthreads();
  int* row_tok = ws_row_tok(a);
  float* row_w = ws_row_w(a);
  for (int p = threadIdx.x; p < B * k; p += blockDim.x) {
    const int t = p / k, e = sm.idx[p];
    const int pos = __popc(sm.mask[e] & ((1u << t) - 1u));
    const int row = S * B + sm.rowoff[e] + pos;
    row_tok[row] = t;
    row_w[row] = sm.w[p];
  }
  for (int p = threadIdx.x; p < S * B; p += blockDim.x) {
    row_tok[p] = p % B;
    row_w[p] = 1.0f;
  }
  unsigned* hmax = ws_hmax(a);
  for (int p = threadIdx.x; p < n_rows; p += blockDim.x) hmax[p] = 0u;
  if (threadIdx.x == 0) ws_hdr(a)[HDR_COUNTER] = 0;
}

// ===========================================================================
// K1: router GEMV (+ routing by the last block).
// NCH: 16-byte chunks of a router row per lane per pass (H / 256 capped at 8).
// ===========================================================================
template <int NCH>
__global__ void __launch_bounds__(128) k_router(DecodeArgs a) {
  extern __shared__ __align__(128) uint8_t dsm[];  // x chunk: up to 8 tokens x H bf16
  __shared__ RouteSmem rs;
  __shared__ __align__(8) uint64_t bar;
  __shared__ int s_last;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int e = blockIdx.x * 4 + warp;
  const int passes = a.H / (256 * NCH);
  uint4 w[NCH];
  if (e < a.E) {
    const uint8_t* row = reinterpret_cast<const uint8_t*>(a.router + (size_t)e * a.H);
#pragma unroll
    for (int c = 0; c < NCH; ++c) w[c] = ld_weights_v4(row + (size_t)(lane + 32 * c) * 16);
  }
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  pdl_trigger();
  pdl_wait();
  __syncthreads();
  int* status = ws_hdr(a) + HDR_STATUS;
  float* lg = ws_logits(a);
  uint32_t phase = 0;
  for (int t0 = 0; t0 < a.B; t0 += 8) {
    const int nt = min(8, a.B - t0);
    if (threadIdx.x == 0) {
      const uint32_t bytes = (uint32_t)nt * a.H * 2;
      mbar_arrive_expect_tx(&bar, bytes);
      bulk_g2s(dsm, a.x + (size_t)t0 * a.H, bytes, &bar);
    }
    const bool ok = mbar_wait(&bar, phase, status);
    phase ^= 1;
    if (e < a.E && ok) {
      for (int t = 0; t < nt; ++t) {
        const uint8_t* xr = dsm + (size_t)t * a.H * 2;
        float acc = 0.f;
        for (int p = 0; p < passes; ++p) {
          if (p > 0) {
            const uint8_t* row = reinterpret_cast<const uint8_t*>(a.router + (size_t)e * a.H) + (size_t)p * NCH * 512;
#pragma unroll
            for (int c = 0; c < NCH; ++c) w[c] = ld_weights_v4(row + (size_t)(lane + 32 * c) * 16);
          }
#pragma unroll
          for (int c = 0; c < NCH; ++c)
            acc = dot8_bf16(w[c], lds128(xr + (size_t)p * NCH * 512 + (lane + 32 * c) * 16), acc);
        }
        acc = warp_sum(acc);
        if (lane == 0) lg[(t0 + t) * a.E + e] = acc;
        if (passes > 1 && t + 1 < nt) {  // reload the first pass for the next token
          const uint8_t* row = reinterpret_cast<const uint8_t*>(a.router + (size_t)e * a.H);
#pragma unroll
          for (int c = 0; c < NCH; ++c) w[c] = ld_weights_v4(row + (size_t)(lane + 32 * c) * 16);
        }
      }
    }
    __syncthreads();  // the x chunk is reused by the next copy
  }
  if (threadIdx.x == 0) {
    __threadfence();
    const int ticket = atomicAdd(ws_hdr(a) + HDR_COUNTER, 1);
    s_last = ticket == (int)gridDim.x - 1;
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  route_and_slots(a, rs);
}

// ===========================================================================
// Activation rows -> fragment order in shared memory.
// NVFP4 path: f16 with a per-row power-of-two prescale (exact for values
// within 2^29 of the row's largest magnitude); *inv gets 2^-prescale.
// BF16 path: bf16 unchanged, *inv = 1.
// ===========================================================================
template <int FMT>
__device__ __forceinline__ void stage_x_row(const uint16_t* src, int len, uint8_t* dst, float* inv, int lane) {
  float mx = 0.f;
  if (FMT == FLINT_MOE_NVFP4) {
    for (int c = lane; c < len / 8; c += 32) {
      const uint4 v = ld_cg_v4(src + 8 * c);
      const uint32_t ws[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int p = 0; p < 4; ++p) mx = fmaxf(mx, fmaxf(fabsf(bf16lo(ws[p])), fabsf(bf16hi(ws[p]))));
    }
    mx = warp_max(mx);
  }
  const int kx = FMT == FLINT_MOE_NVFP4 ? prescale_exp(mx) : 0;
  const float sc = exp2i(kx);
  for (int c = lane; c < len / 8; c += 32) {
    const uint4 v = ld_cg_v4(src + 8 * c);
    const uint32_t ws[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int p = 0; p < 4; ++p) {
      uint32_t bits = ws[p];
      if (FMT == FLINT_MOE_NVFP4) {
        const __half2 hv = __floats2half2_rn(bf16lo(ws[p]) * sc, bf16hi(ws[p]) * sc);
        bits = *reinterpret_cast<const uint32_t*>(&hv);
      }
      *reinterpret_cast<uint32_t*>(dst + 2 * frag_offset_elems(8 * c + 2 * p)) = bits;
    }
  }
  if (lane == 0) *inv = exp2i(-kx);
}

// ===========================================================================
// K2: gate/up GEMV + SiLU * up for one (slot, tile of 8 intermediate rows).
// 4 warps split the reduction (H) into contiguous k-group ranges.
// ===========================================================================
template <int FMT, int NTMAX>
__global__ void __launch_bounds__(128) k_gateup(DecodeArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  constexpr int KGB = FMT == FLINT_MOE_NVFP4 ? KG_NVFP4 : KG_BF16;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t4 = lane & 3;
  const int tile = blockIdx.x, slot = blockIdx.y;
  const int KGW = a.H / (KG_COLS * 4);
  const int kslice = KGW * KGB;
  const int xstride = a.H * 2 + 16;
  uint8_t* wbuf = smem + warp * kslice;
  uint8_t* xs = smem + 4 * kslice;
  float* red = reinterpret_cast<float*>(xs + (size_t)a.B * xstride);
  float* s_inv = red + 3 * NTMAX * 128;
  uint64_t* bars = reinterpret_cast<uint64_t*>(s_inv + MAX_BATCH);

  if (threadIdx.x < 4) mbar_init(&bars[threadIdx.x], 1);
  fence_mbar_init();
  __syncthreads();
  const bool shared_slot = slot < a.S;
  auto issue = [&](int expert) {
    if (lane == 0) {
      const uint8_t* src = a.packed + (int64_t)expert * a.L.expert_bytes + (int64_t)tile * a.L.gu_tile +
                           (int64_t)warp * kslice;
      mbar_arrive_expect_tx(&bars[warp], (uint32_t)kslice);
      bulk_g2s(wbuf, src, (uint32_t)kslice, &bars[warp]);
    }
  };
  if (shared_slot) issue(a.E + slot);  // routing-independent: fetch before waiting
  pdl_trigger();
  pdl_wait();
  int* hdr = ws_hdr(a);
  const int n_slots = __ldcg(hdr + HDR_NSLOTS);
  if (slot >= n_slots) return;  // a routed slot this batch does not use; nothing in flight
  const int expert = __ldcg(ws_slot_expert(a) + slot);
  const int off = __ldcg(ws_slot_off(a) + slot);
  const int T = __ldcg(ws_slot_off(a) + slot + 1) - off;
  if (expert < 0 || expert >= a.E + a.S || T < 1 || T > a.B || off < 0 || off + T > a.W.max_rows) {
    if (threadIdx.x == 0) atomicOr(hdr + HDR_STATUS, FLINT_MOE_DEV_ERR_SLOTS);
    if (shared_slot) mbar_drain(&bars[warp], 0);
    return;
  }
  if (!shared_slot) issue(expert);
  for (int n = warp; n < T; n += 4) {
    const int tok = __ldcg(ws_row_tok(a) + off + n);
    stage_x_row<FMT>(a.x + (size_t)tok * a.H, a.H, xs + (size_t)n * xstride, s_inv + n, lane);
  }
  __syncthreads();

  float acc[NTMAX][4];
#pragma unroll
  for (int nt = 0; nt < NTMAX; ++nt)
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[nt][i] = 0.f;
  const int nt_used = (T + 7) >> 3;
  const bool ok = mbar_wait(&bars[warp], 0, hdr + HDR_STATUS);
  if (ok) {
    for (int kl = 0; kl < KGW; ++kl) {
      const int kg = warp * KGW + kl;
      const uint8_t* kp = wbuf + kl * KGB;
      uint4 bx[NTMAX][2];
#pragma unroll
      for (int nt = 0; nt < NTMAX; ++nt) {
        if (nt < nt_used) {
          int n = nt * 8 + g;
          n = n < T ? n : T - 1;  // columns past the slot's tokens repeat a valid row
          const uint8_t* rp = xs + (size_t)n * xstride + kg * 128 + t4 * 32;
          bx[nt][0] = lds128(rp);
          bx[nt][1] = lds128(rp + 16);
        }
      }
      if (FMT == FLINT_MOE_NVFP4) {
        const uint4 codes = lds128(kp + lane * 16);
        const uint32_t sg = lds32(kp + KG_CODE_BYTES + g * 4);
        const uint32_t sg8 = lds32(kp + KG_CODE_BYTES + (g + 8) * 4);
        const uint32_t cw[4] = {codes.x, codes.y, codes.z, codes.w};
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
          uint32_t af[4];
          nvfp4_afrag(cw[ks], sg, sg8, ks, af);
#pragma unroll
          for (int nt = 0; nt < NTMAX; ++nt) {
            if (nt < nt_used) {
              const uint4& q = bx[nt][ks >> 1];
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
            if (nt < nt_used) {
              const uint4& q = bx[nt][ks >> 1];
              mma_bf16(acc[nt], af, (ks & 1) ? q.z : q.x, (ks & 1) ? q.w : q.y);
            }
          }
        }
      }
    }
  } else {
    mbar_drain(&bars[warp], 0);
  }
  if (warp > 0) {
#pragma unroll
    for (int nt = 0; nt < NTMAX; ++nt)
#pragma unroll
      for (int i = 0; i < 4; ++i) red[((warp - 1) * NTMAX + nt) * 128 + lane * 4 + i] = acc[nt][i];
  }
  __syncthreads();
  if (warp != 0) return;
#pragma unroll
  for (int w2 = 0; w2 < 3; ++w2)
#pragma unroll
    for (int nt = 0; nt < NTMAX; ++nt)
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[nt][i] += red[(w2 * NTMAX + nt) * 128 + lane * 4 + i];

  const float Gg = a.globals[expert * 4 + 0];
  const float Gu = a.globals[expert * 4 + 1];
  const int i_row = tile * 8 + g;
  const int hoff = frag_offset_elems(i_row);
  uint16_t* h = ws_h(a);
  unsigned* hmax = ws_hmax(a);
#pragma unroll
  for (int nt = 0; nt < NTMAX; ++nt) {
    if (nt >= nt_used) break;
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const int n = nt * 8 + 2 * t4 + hh;
      float hv = 0.f;
      if (n < T) {
        const float inv = s_inv[n];
        const float gv = (acc[nt][hh] * inv) * Gg;
        const float uv = (acc[nt][2 + hh] * inv) * Gu;
        const float sv = gv / (1.0f + expf(-gv));
        const __nv_bfloat16 hb = __float2bfloat16_rn(sv * uv);
        h[(size_t)(off + n) * a.I + hoff] = *reinterpret_cast<const uint16_t*>(&hb);
        hv = fabsf(__bfloat162float(hb));
      }
      hv = fmaxf(hv, __shfl_xor_sync(0xffffffffu, hv, 4));
      hv = fmaxf(hv, __shfl_xor_sync(0xffffffffu, hv, 8));
      hv = fmaxf(hv, __shfl_xor_sync(0xffffffffu, hv, 16));
      if (g == 0 && n < T && hv > 0.f) atomicMax(hmax + off + n, __float_as_uint(hv));
    }
  }
}

// ===========================================================================
// K3: down GEMV + routing-weighted combine for one tile of 16 output rows.
// Work items are (slot, chunk of up to 8 of its rows); warp w takes items
// w, w+4, ... in order, NBUF of them in flight; per-warp partial sums are
// added in warp order at the end, so the result does not depend on timing.
// ===========================================================================
struct DownSmemPlan {
  int buf_bytes, hrows, hstride;
  size_t acc_off, off_off, rowtok_off, roww_off, items_off, inv_off, bar_off, total;
};

__host__ __device__ inline DownSmemPlan down_plan(int H, int I, int B, int max_slots, int max_rows, int fmt, int nbuf) {
  DownSmemPlan p;
  const int kgb = fmt == FLINT_MOE_NVFP4 ? KG_NVFP4 : KG_BF16;
  p.hrows = B < 8 ? B : 8;
  p.hstride = I * 2 + 16;
  p.buf_bytes = (I / KG_COLS) * kgb + p.hrows * p.hstride;
  size_t o = (size_t)4 * nbuf * p.buf_bytes;
  p.acc_off = o;     o += sizeof(float) * 4 * B * 16;
  p.off_off = o;     o += sizeof(int) * (max_slots + 1);
  p.rowtok_off = o;  o += sizeof(int) * max_rows;
  p.roww_off = o;    o += sizeof(float) * max_rows;
  p.items_off = o;   o += sizeof(int) * (max_slots + max_rows / 8 + 8);
  o = (o + 15) & ~(size_t)15;
  p.inv_off = o;     o += sizeof(float) * 4 * nbuf * 8;
  o = (o + 15) & ~(size_t)15;
  p.bar_off = o;     o += sizeof(uint64_t) * 4 * nbuf;
  p.total = o;
  return p;
}

template <int FMT, int NBUF>
__global__ void __launch_bounds__(128) k_down(DecodeArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  constexpr int KGB = FMT == FLINT_MOE_NVFP4 ? KG_NVFP4 : KG_BF16;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t4 = lane & 3;
  const int tile = blockIdx.x;
  const DownSmemPlan P = down_plan(a.H, a.I, a.B, a.W.max_slots, a.W.max_rows, FMT, NBUF);
  const int dn_bytes = (int)a.L.dn_tile;
  float* acc_s = reinterpret_cast<float*>(smem + P.acc_off);
  int* s_off = reinterpret_cast<int*>(smem + P.off_off);
  int* s_rowtok = reinterpret_cast<int*>(smem + P.rowtok_off);
  float* s_roww = reinterpret_cast<float*>(smem + P.roww_off);
  int* s_items = reinterpret_cast<int*>(smem + P.items_off);
  float* s_inv = reinterpret_cast<float*>(smem + P.inv_off) + warp * NBUF * 8;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + P.bar_off) + warp * NBUF;
  auto buf = [&](int b) { return smem + (size_t)(warp * NBUF + b) * P.buf_bytes; };
  __shared__ int s_wsum[4];

  if (lane < NBUF) mbar_init(&bars[lane], 2);  // one arrival for the weights, one for the h rows
  fence_mbar_init();
  for (int i = threadIdx.x; i < 4 * a.B * 16; i += blockDim.x) acc_s[i] = 0.f;
  __syncthreads();

  // Items of the shared slots are known before routing: T = B for each.
  const int cps = (a.B + 7) / 8;
  int pre = 0;
  for (int i = warp; i < a.S * cps && pre < NBUF; i += 4, ++pre) {
    if (lane == 0) {
      const int s = i / cps;
      const uint8_t* src = a.packed + (int64_t)(a.E + s) * a.L.expert_bytes + a.L.gu_bytes + (int64_t)tile * dn_bytes;
      mbar_arrive_expect_tx(&bars[pre], (uint32_t)dn_bytes);
      bulk_g2s(buf(pre), src, (uint32_t)dn_bytes, &bars[pre]);
    }
  }
  pdl_trigger();
  pdl_wait();

  int* hdr = ws_hdr(a);
  int n_slots = __ldcg(hdr + HDR_NSLOTS);
  int n_rows = __ldcg(hdr + HDR_NROWS);
  if (n_slots < a.S || n_slots > a.W.max_slots || n_rows < 0 || n_rows > a.W.max_rows) {
    if (threadIdx.x == 0) atomicOr(hdr + HDR_STATUS, FLINT_MOE_DEV_ERR_SLOTS);
    for (int j = 0; j < pre; ++j) mbar_drain(&bars[j], 0);  // let pre-issued copies land, then stop
    return;
  }
  for (int i = threadIdx.x; i <= n_slots; i += blockDim.x) s_off[i] = __ldcg(ws_slot_off(a) + i);
  for (int i = threadIdx.x; i < n_rows; i += blockDim.x) {
    s_rowtok[i] = __ldcg(ws_row_tok(a) + i);
    s_roww[i] = __ldcg(ws_row_w(a) + i);
  }
  __syncthreads();
  // Item list: slot s contributes ceil(T_s / 8) items; exclusive prefix over slots.
  {
    const int spt = (n_slots + blockDim.x - 1) / blockDim.x;
    const int s0 = threadIdx.x * spt;
    int local = 0;
    for (int s = s0; s < s0 + spt && s < n_slots; ++s) local += (s_off[s + 1] - s_off[s] + 7) >> 3;
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
      const int nc = (s_off[s + 1] - s_off[s] + 7) >> 3;
      for (int c = 0; c < nc; ++c) s_items[run + c] = (s << 8) | c;
      run += nc;
    }
  }
  __syncthreads();
  const int n_items = s_wsum[0] + s_wsum[1] + s_wsum[2] + s_wsum[3];
  const int* slot_expert = ws_slot_expert(a);

  // Issue item j of this warp into buffer j % NBUF.
  auto issue = [&](int j) {
    const int item = warp + 4 * j;
    if (item >= n_items) return;
    const int s = s_items[item] >> 8, c = s_items[item] & 0xFF;
    const int r0 = s_off[s] + 8 * c;
    const int Tc = min(8, s_off[s + 1] - r0);
    const int b = j % NBUF;
    if (lane == 0) {
      if (j >= pre) {
        int expert = __ldcg(slot_expert + s);
        if (expert < 0 || expert >= a.E + a.S) {
          atomicOr(hdr + HDR_STATUS, FLINT_MOE_DEV_ERR_SLOTS);
          expert = 0;
        }
        const uint8_t* src = a.packed + (int64_t)expert * a.L.expert_bytes + a.L.gu_bytes + (int64_t)tile * dn_bytes;
        mbar_arrive_expect_tx(&bars[b], (uint32_t)dn_bytes);
        bulk_g2s(buf(b), src, (uint32_t)dn_bytes, &bars[b]);
      }
      mbar_arrive_expect_tx(&bars[b], (uint32_t)(Tc * a.I * 2));
    }
    __syncwarp();
    if (lane < Tc)
      bulk_g2s(buf(b) + dn_bytes + lane * P.hstride, ws_h(a) + (size_t)(r0 + lane) * a.I, (uint32_t)(a.I * 2),
               &bars[b]);
  };
  for (int j = 0; j < NBUF; ++j) issue(j);

  const int KG = a.I / KG_COLS;
  for (int j = 0;; ++j) {
    const int item = warp + 4 * j;
    if (item >= n_items) break;
    const int s = s_items[item] >> 8, c = s_items[item] & 0xFF;
    const int r0 = s_off[s] + 8 * c;
    const int Tc = min(8, s_off[s + 1] - r0);
    const int b = j % NBUF;
    const uint32_t parity = (uint32_t)((j / NBUF) & 1);
    if (!mbar_wait(&bars[b], parity, hdr + HDR_STATUS)) {
      // give every copy this warp has in flight a bounded chance to land
      for (int jj = j; jj < j + NBUF && warp + 4 * jj < n_items; ++jj)
        mbar_drain(&bars[jj % NBUF], (uint32_t)((jj / NBUF) & 1));
      break;
    }
    uint8_t* wb = buf(b);
    uint8_t* hb = wb + dn_bytes;
    if (FMT == FLINT_MOE_NVFP4) {
      for (int n = 0; n < Tc; ++n) {
        const float mx = __uint_as_float(__ldcg(ws_hmax(a) + r0 + n));
        const int kh = prescale_exp(mx);
        const float sc = exp2i(kh);
        uint32_t* rowp = reinterpret_cast<uint32_t*>(hb + n * P.hstride);
        for (int q = lane; q < a.I / 2; q += 32) {
          const uint32_t wv = rowp[q];
          const __half2 hv = __floats2half2_rn(bf16lo(wv) * sc, bf16hi(wv) * sc);
          rowp[q] = *reinterpret_cast<const uint32_t*>(&hv);
        }
        if (lane == 0) s_inv[b * 8 + n] = exp2i(-kh);
      }
    } else if (lane < Tc) {
      s_inv[b * 8 + lane] = 1.0f;
    }
    __syncwarp();
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    const int nrow = g < Tc ? g : Tc - 1;
    for (int kg = 0; kg < KG; ++kg) {
      const uint8_t* kp = wb + kg * KGB;
      const uint8_t* rp = hb + nrow * P.hstride + kg * 128 + t4 * 32;
      const uint4 b01 = lds128(rp), b23 = lds128(rp + 16);
      if (FMT == FLINT_MOE_NVFP4) {
        const uint4 codes = lds128(kp + lane * 16);
        const uint32_t sg = lds32(kp + KG_CODE_BYTES + g * 4);
        const uint32_t sg8 = lds32(kp + KG_CODE_BYTES + (g + 8) * 4);
        const uint32_t cw[4] = {codes.x, codes.y, codes.z, codes.w};
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
          uint32_t af[4];
          nvfp4_afrag(cw[ks], sg, sg8, ks, af);
          const uint4& q = ks < 2 ? b01 : b23;
          mma_f16(acc, af, (ks & 1) ? q.z : q.x, (ks & 1) ? q.w : q.y);
        }
      } else {
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
          const uint4 v = lds128(kp + lane * 64 + ks * 16);
          const uint32_t af[4] = {v.x, v.y, v.z, v.w};
          const uint4& q = ks < 2 ? b01 : b23;
          mma_bf16(acc, af, (ks & 1) ? q.z : q.x, (ks & 1) ? q.w : q.y);
        }
      }
    }
    const int expert = min(max(__ldcg(slot_expert + s), 0), a.E + a.S - 1);
    const float Gd = a.globals[expert * 4 + 2];
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const int n = 2 * t4 + hh;
      if (n < Tc) {
        const int row = r0 + n;
        const int tok = min(max(s_rowtok[row], 0), a.B - 1);
        const float wt = s_roww[row];
        const float inv = s_inv[b * 8 + n];
        float* dst = acc_s + (warp * a.B + tok) * 16;
        dst[g] += wt * ((acc[hh] * inv) * Gd);
        dst[g + 8] += wt * ((acc[2 + hh] * inv) * Gd);
      }
    }
    __syncwarp();
    issue(j + NBUF);
  }
  __syncthreads();
  for (int p = threadIdx.x; p < a.B * 16; p += blockDim.x) {
    const int t = p >> 4, r = p & 15;
    const float v = acc_s[(0 * a.B + t) * 16 + r] + acc_s[(1 * a.B + t) * 16 + r] + acc_s[(2 * a.B + t) * 16 + r] +
                    acc_s[(3 * a.B + t) * 16 + r];
    const __nv_bfloat16 o = __float2bfloat16_rn(v);
    a.out[(size_t)t * a.H + tile * 16 + r] = *reinterpret_cast<const uint16_t*>(&o);
  }
}

}  // namespace flint

using namespace flint;

// ===========================================================================
// Host side
// ===========================================================================
namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

constexpr int DOWN_NBUF = 2;

size_t gateup_smem(int H, int B, int fmt, int ntmax) {
  const int kgb = fmt == FLINT_MOE_NVFP4 ? KG_NVFP4 : KG_BF16;
  return (size_t)4 * (H / 256) * kgb + (size_t)B * (H * 2 + 16) + sizeof(float) * (3 * ntmax * 128 + MAX_BATCH) +
         sizeof(uint64_t) * 4;
}

template <typename K>
cudaError_t launch_pdl(K kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t stream, const DecodeArgs& a) {
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
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

template <int FMT>
cudaError_t launch_gateup(const DecodeArgs& a, cudaStream_t stream) {
  const int ntmax = (a.B + 7) / 8;
  const dim3 grid(a.I / 8, a.S + (a.E < a.B * a.k ? a.E : a.B * a.k));
  const size_t smem = gateup_smem(a.H, a.B, FMT, ntmax);
  switch (ntmax) {
    case 1: return launch_pdl(k_gateup<FMT, 1>, grid, dim3(128), smem, stream, a);
    case 2: return launch_pdl(k_gateup<FMT, 2>, grid, dim3(128), smem, stream, a);
    case 3: return launch_pdl(k_gateup<FMT, 3>, grid, dim3(128), smem, stream, a);
    default: return launch_pdl(k_gateup<FMT, 4>, grid, dim3(128), smem, stream, a);
  }
}

template <int FMT>
cudaError_t launch_down(const DecodeArgs& a, cudaStream_t stream) {
  const DownSmemPlan P = down_plan(a.H, a.I, a.B, a.W.max_slots, a.W.max_rows, FMT, DOWN_NBUF);
  return launch_pdl(k_down<FMT, DOWN_NBUF>, dim3(a.H / 16), dim3(128), P.total, stream, a);
}

cudaError_t launch_router(const DecodeArgs& a, cudaStream_t stream) {
  const dim3 grid((a.E + 3) / 4);
  const size_t smem = (size_t)(a.B < 8 ? a.B : 8) * a.H * 2;
  switch (a.H) {
    case 256: return launch_pdl(k_router<1>, grid, dim3(128), smem, stream, a);
    case 512: return launch_pdl(k_router<2>, grid, dim3(128), smem, stream, a);
    case 768: return launch_pdl(k_router<3>, grid, dim3(128), smem, stream, a);
    case 1024: return launch_pdl(k_router<4>, grid, dim3(128), smem, stream, a);
    case 1280: return launch_pdl(k_router<5>, grid, dim3(128), smem, stream, a);
    case 1536: return launch_pdl(k_router<6>, grid, dim3(128), smem, stream, a);
    case 1792: return launch_pdl(k_router<7>, grid, dim3(128), smem, stream, a);
    default:
      if (a.H % 2048) return cudaErrorInvalidValue;
      return launch_pdl(k_router<8>, grid, dim3(128), smem, stream, a);
  }
}

}  // namespace

extern "C" size_t flint_moe_workspace_bytes(const flint_moe_config* c, int32_t max_batch) {
  if (flint_moe_check_config(c) != FLINT_MOE_OK || max_batch < 1 || max_batch > MAX_BATCH) return 0;
  return make_ws_layout(c->num_experts, c->top_k, c->inter, c->n_shared, max_batch).total;
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
  return FLINT_MOE_OK;
}

extern "C" flint_moe_status flint_moe_decode(const flint_moe_layer* layer, const uint16_t* x, int32_t B,
                                             uint16_t* out, void* ws, cudaStream_t stream) {
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
  a.W = make_ws_layout(a.E, a.k, a.I, a.S, B);
  constexpr size_t SMEM_LIMIT = 227 * 1024;
  if (gateup_smem(a.H, B, a.fmt, (B + 7) / 8) > SMEM_LIMIT ||
      down_plan(a.H, a.I, B, a.W.max_slots, a.W.max_rows, a.fmt, DOWN_NBUF).total > SMEM_LIMIT ||
      (size_t)(B < 8 ? B : 8) * a.H * 2 > SMEM_LIMIT - 16 * 1024)
    return FLINT_MOE_EUNSUPPORTED;
  cudaError_t e = launch_router(a, stream);
  if (e == cudaSuccess) e = a.fmt == FLINT_MOE_NVFP4 ? launch_gateup<FLINT_MOE_NVFP4>(a, stream)
                                                       : launch_gateup<FLINT_MOE_BF16>(a, stream);
  if (e == cudaSuccess) e = a.fmt == FLINT_MOE_NVFP4 ? launch_down<FLINT_MOE_NVFP4>(a, stream)
                                                       : launch_down<FLINT_MOE_BF16>(a, stream);
  return e == cudaSuccess ? FLINT_MOE_OK : FLINT_MOE_ECUDA;
}

extern "C" flint_moe_status flint_moe_debug_routing(const flint_moe_config* c, const void* ws, int32_t B,
                                                    int32_t* idx, float* w, cudaStream_t stream) {
  if (flint_moe_check_config(c) != FLINT_MOE_OK || !ws || !idx || !w || B < 1 || B > MAX_BATCH)
    return FLINT_MOE_EINVAL;
  const WsLayout W = make_ws_layout(c->num_experts, c->top_k, c->inter, c->n_shared, B);
  const uint8_t* base = static_cast<const uint8_t*>(ws);
  const size_t n = (size_t)B * c->top_k;
  if (cudaMemcpyAsync(idx, base + W.topk_idx, n * sizeof(int), cudaMemcpyDeviceToDevice, stream) != cudaSuccess)
    return FLINT_MOE_ECUDA;
  if (cudaMemcpyAsync(w, base + W.topk_w, n * sizeof(float), cudaMemcpyDeviceToDevice, stream) != cudaSuccess)
    return FLINT_MOE_ECUDA;
  return FLINT_MOE_OK;
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
// symbol is only a stand-in; the address is looked up once per device.
flint_moe_status noalloc_scratch(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FLINT_MOE_ECUDA;
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  if (!g_noalloc_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return FLINT_MOE_ECUDA;
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return FLINT_MOE_OK;
}

}  // namespace

extern "C" flint_moe_status flint_moe_decode_noalloc(const flint_moe_layer* layer, const uint16_t* x, int32_t B,
                                                     uint16_t* out, cudaStream_t stream) {
  if (!layer) return FLINT_MOE_EINVAL;
  const flint_moe_config* c = &layer->cfg;
  const flint_moe_status st = flint_moe_check_config(c);
  if (st != FLINT_MOE_OK) return st;
  if (B < 0 || B > MAX_BATCH) return FLINT_MOE_EINVAL;
  if (B == 0) return FLINT_MOE_OK;
  if (make_ws_layout(c->num_experts, c->top_k, c->inter, c->n_shared, B).total > FLINT_MOE_NOALLOC_SCRATCH_BYTES)
    return FLINT_MOE_EUNSUPPORTED;
  void* scratch = nullptr;
  const flint_moe_status sst = noalloc_scratch(&scratch);
  if (sst != FLINT_MOE_OK) return sst;
  // The routing counter must start at zero; the status word is not reported
  // by this entry point, so both header words are cleared on every call.
  if (cudaMemsetAsync(scratch, 0, 256, stream) != cudaSuccess) return FLINT_MOE_ECUDA;
  return flint_moe_decode(layer, x, B, out, scratch, stream);
}
