// Expert-grouped tensor-core path of the Flint-style W4A16 MoE layer for many
// tokens ("Day-0 Support for Flint on vLLM", section "Optimisation": the MoE
// kernels were also the largest prefill gain).
//
// With many tokens per expert the weights are worth staging: every 128-row x
// 64-column weight block is dequantised once (E2M1 x E4M3 products are exact in
// bf16) into shared memory in the 128-byte-swizzled K-major layout that
// tcgen05.mma reads, the expert's tokens are gathered into the same layout with
// cp.async, and one thread issues the tensor-core MMAs (M = 128 weight rows,
// N = up to 128 tokens, K = 16 per instruction) that accumulate in FP32 in
// tensor memory. The epilogue reads the accumulators back with tcgen05.ld.
//
//   k_pf_gemm<ROUTER>  logits = Wr x^T      (bf16 router rows, cp.async)
//   k_pf_topk          sigmoid top-k per token; tokens counted per expert
//   k_pf_plan          expert-grouped token lists, tile lists
//   k_pf_gemm<GATEUP>  h = bf16(silu(G_g g) * G_u u) per (token, expert)
//   k_pf_gemm<DOWN>    y[t][q] = w * G_d (c_d h) per (token, expert)
//   k_pf_combine       out = bf16(sum_q y[t][q]) in slot order
#include <algorithm>
#include <atomic>
#include <cmath>

#include "common.cuh"
#include "flint_moe_prefill.h"

namespace flint {
namespace pf {

constexpr int BM = 128;       // weight rows per tile (MMA M)
constexpr int BK = 64;        // k per pipeline stage: one 128-byte swizzle row of bf16
constexpr int NT = 128;       // tokens per tile at most (MMA N)
constexpr int STAGES = 4;     // shared-memory stages
constexpr int PREF = 2;       // k-blocks loaded ahead of the one being consumed
constexpr int THREADS = 256;  // 8 warps: each dequantises one 16-row packed tile per stage
constexpr uint32_t TMEM_COLS = 2 * NT;  // N <= NT columns are used; the margin costs nothing at one CTA per SM
constexpr int A_STAGE = BM * BK * 2;              // 16 KiB
constexpr int B_STAGE = NT * BK * 2;              // 16 KiB
constexpr int RAW_STAGE = (BM / 16) * KG_NVFP4;   // 4608 B: eight packed k-groups
constexpr int MAX_E = 512;

enum Mode : int { ROUTER = 0, GATEUP = 1, DOWN = 2 };
enum : int { PF_STATUS = HDR_STATUS, PF_NSLOTS = 2, PF_NGU = 3, PF_NDN = 4 };

// Workspace: header words, then 256-byte aligned regions sized for T tokens.
struct PfLayout {
  size_t counts, logits, idx, w, pos, slot_expert, slot_row0, slot_count, list_tok, list_q, list_w, gu_tiles,
      dn_tiles, h, y, total;
  int max_slots, max_rows, max_gu, max_dn;
};

__host__ __device__ inline PfLayout make_pf_layout(int H, int E, int k, int I, int S, int T) {
  PfLayout W;
  W.max_slots = S + (E < T * k ? E : T * k);
  W.max_rows = T * (S + k);
  // sum over slots of ceil(count / NT) <= rows / NT + slots
  const int max_nt = W.max_rows / NT + W.max_slots + 1;
  W.max_gu = max_nt * (2 * I / BM);
  W.max_dn = max_nt * (H / BM);
  size_t o = 256;
  W.counts = o;      o = ws_align(o + sizeof(int) * E);
  W.logits = o;      o = ws_align(o + sizeof(float) * (size_t)T * E);
  W.idx = o;         o = ws_align(o + sizeof(int) * (size_t)T * k);
  W.w = o;           o = ws_align(o + sizeof(float) * (size_t)T * k);
  W.pos = o;         o = ws_align(o + sizeof(int) * (size_t)T * k);
  W.slot_expert = o; o = ws_align(o + sizeof(int) * W.max_slots);
  W.slot_row0 = o;   o = ws_align(o + sizeof(int) * W.max_slots);
  W.slot_count = o;  o = ws_align(o + sizeof(int) * W.max_slots);
  W.list_tok = o;    o = ws_align(o + sizeof(int) * (size_t)W.max_rows);
  W.list_q = o;      o = ws_align(o + sizeof(int) * (size_t)W.max_rows);
  W.list_w = o;      o = ws_align(o + sizeof(float) * (size_t)W.max_rows);
  W.gu_tiles = o;    o = ws_align(o + sizeof(int4) * (size_t)W.max_gu);
  W.dn_tiles = o;    o = ws_align(o + sizeof(int4) * (size_t)W.max_dn);
  W.h = o;           o = ws_align(o + (size_t)2 * W.max_rows * I);
  W.y = o;           o = ws_align(o + sizeof(float) * (size_t)W.max_rows * H);
  W.total = o;
  return W;
}

struct PfArgs {
  int H, I, E, S, k, B, renorm;
  float routed_scale;
  const uint16_t* x;       // [B][H]
  const uint16_t* router;  // [E][H]
  const float* bias;       // [E] or null
  const uint8_t* packed;
  const float* globals;    // [E + S][4]: G_gate, G_up, G_down, 0
  Layout L;
  uint8_t* ws;
  PfLayout W;
  uint16_t* out;           // [B][H]
};

template <typename T>
__device__ __forceinline__ T* ws_at(const PfArgs& a, size_t off) {
  return reinterpret_cast<T*>(a.ws + off);
}

// ---------------------------------------------------------------------------
// tcgen05 / cp.async helpers.
// ---------------------------------------------------------------------------

// Shared-memory matrix descriptor for a K-major operand in the 128-byte
// swizzle layout: 8-row x 128-byte atoms (row r of an atom at r * 128, its
// 16-byte chunk c at chunk position c ^ r), atoms stacked along M/N every
// 1024 bytes (stride byte offset). Fields: start address >> 4 (bits 0-13),
// leading byte offset >> 4 (16-29; unused for swizzled K-major, set to 1),
// stride byte offset >> 4 (32-45), descriptor version 1 (46-47), base offset 0
// (atoms are 1024-byte aligned), layout type 2 = 128-byte swizzle (61-63).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)1 << 16;
  d |= (uint64_t)(1024 >> 4) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

// Instruction descriptor of kind::f16: D f32 (bits 4-5 = 1), A and B bf16
// (bits 7-9 = 1, 10-12 = 1), both K-major (bits 15, 16 = 0), N >> 3 in bits
// 17-22, M >> 4 in bits 24-28.
__device__ __forceinline__ uint32_t idesc_bf16_f32(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                       uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrives once on bar when every tcgen05 operation this thread issued so far has completed.
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_addr(bar))
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// 16 consecutive 32-bit columns of this warp's 32 tensor-memory lanes.
__device__ __forceinline__ void tc_ld16(uint32_t taddr, uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
        "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// 16-byte copy global -> shared; src_bytes 0 fills the 16 bytes with zeros.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Byte offset of element (row r, column c) of a 64-column bf16 block stored
// K-major with the 128-byte swizzle.
__device__ __forceinline__ uint32_t sw128_off(int r, int c) {
  return (uint32_t)((r >> 3) * 1024 + (r & 7) * 128 + ((((c * 2) >> 4) ^ (r & 7)) << 4) + ((c * 2) & 15));
}

// f16x2 holding two values exactly representable in bf16 -> bf16x2 (exact).
__device__ __forceinline__ uint32_t f16x2_to_bf16x2(uint32_t h) {
  const __half2 hv = *reinterpret_cast<const __half2*>(&h);
  const float2 f = __half22float2(hv);
  const __nv_bfloat162 b = __float22bfloat162_rn(f);
  return *reinterpret_cast<const uint32_t*>(&b);
}

// ---------------------------------------------------------------------------
// The grouped GEMM. A tile is (slot, m-tile of 128 weight rows, first grouped
// row, token count n <= NT); the kernel is persistent over its tile list.
// ---------------------------------------------------------------------------
struct GemmSmem {
  uint64_t raw_full[STAGES];
  uint64_t mma_done[STAGES];
  uint32_t tmem_base;
  const uint16_t* src[NT];  // activation row of each tile column
  int col_tok[NT];
  int col_q[NT];
  float col_w[NT];
};

constexpr size_t gemm_dyn_smem() { return 1024 + (size_t)STAGES * (A_STAGE + B_STAGE + RAW_STAGE); }

template <int MODE>
__global__ void __launch_bounds__(THREADS, 1) k_pf_gemm(PfArgs a) {
  extern __shared__ uint8_t dsmem[];
  __shared__ GemmSmem G;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t base = (smem_addr(dsmem) + 1023u) & ~1023u;
  uint8_t* const base_ptr = dsmem + (base - smem_addr(dsmem));
  const uint32_t a_op = base;                                   // STAGES x 16 KiB
  const uint32_t b_op = base + STAGES * A_STAGE;                // STAGES x 16 KiB
  uint8_t* const raw = base_ptr + STAGES * (A_STAGE + B_STAGE);  // STAGES x 4608 B
  int* status = ws_at<int>(a, 0) + PF_STATUS;

  const int K = MODE == DOWN ? a.I : a.H;
  const int KB = K / BK;
  int n_tiles, mt_count = 0, nt_count = 0;
  if (MODE == ROUTER) {
    mt_count = (a.E + BM - 1) / BM;
    nt_count = (a.B + NT - 1) / NT;
    n_tiles = mt_count * nt_count;
  } else {
    n_tiles = __ldcg(ws_at<int>(a, 0) + (MODE == GATEUP ? PF_NGU : PF_NDN));
  }
  if ((int)blockIdx.x >= n_tiles) return;  // uniform: no tensor memory taken

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&G.raw_full[s], 1);
      mbar_init(&G.mma_done[s], 1);
    }
    fence_mbar_init();
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(&G.tmem_base)),
                 "r"(TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = G.tmem_base;

  const int* slot_expert = ws_at<int>(a, a.W.slot_expert);
  const int4* tiles = ws_at<int4>(a, MODE == GATEUP ? a.W.gu_tiles : a.W.dn_tiles);
  const int* list_tok = ws_at<int>(a, a.W.list_tok);
  const int* list_q = ws_at<int>(a, a.W.list_q);
  const float* list_w = ws_at<float>(a, a.W.list_w);
  uint16_t* hbuf = ws_at<uint16_t>(a, a.W.h);

  uint32_t gk = 0;  // k-blocks this CTA has started, over all its tiles (stage = gk % STAGES)
  bool failed = false;
  for (int tile = blockIdx.x; tile < n_tiles && !failed; tile += gridDim.x) {
    int slot = 0, mt, row0, n;
    if (MODE == ROUTER) {
      mt = tile % mt_count;
      row0 = (tile / mt_count) * NT;
      n = min(NT, a.B - row0);
    } else {
      const int4 t = __ldcg(tiles + tile);
      slot = t.x;
      mt = t.y;
      row0 = t.z;
      n = t.w;
    }
    const int expert = MODE == ROUTER ? 0 : __ldcg(slot_expert + slot);
    for (int i = threadIdx.x; i < NT; i += THREADS) {
      const uint16_t* s = nullptr;
      if (i < n) {
        if (MODE == ROUTER) s = a.x + (size_t)(row0 + i) * a.H;
        if (MODE == GATEUP) s = a.x + (size_t)__ldcg(list_tok + row0 + i) * a.H;
        if (MODE == DOWN) {
          s = hbuf + (size_t)(row0 + i) * a.I;
          G.col_tok[i] = __ldcg(list_tok + row0 + i);
          G.col_q[i] = __ldcg(list_q + row0 + i);
          G.col_w[i] = __ldcg(list_w + row0 + i);
        }
      }
      G.src[i] = s;
    }
    __syncthreads();

    // Packed weight tiles of this m-tile: tile p of the expert's gate/up or down run.
    const uint8_t* wbase = nullptr;
    int64_t wtile = 0;
    if (MODE == GATEUP) {
      wbase = a.packed + (int64_t)expert * a.L.expert_bytes + (int64_t)(mt * 8) * a.L.gu_tile;
      wtile = a.L.gu_tile;
    } else if (MODE == DOWN) {
      wbase = a.packed + (int64_t)expert * a.L.expert_bytes + a.L.gu_bytes + (int64_t)(mt * 8) * a.L.dn_tile;
      wtile = a.L.dn_tile;
    }

    // Loads of k-block kb of this tile into stage s.
    auto issue = [&](int kb, int s) {
      if (MODE == ROUTER) {
        for (int c = threadIdx.x; c < BM * 8; c += THREADS) {
          const int r = c >> 3, ch = c & 7, e = mt * BM + r;
          const uint16_t* src = a.router + (size_t)(e < a.E ? e : 0) * a.H + kb * BK + ch * 8;
          cp_async16(a_op + s * A_STAGE + sw128_off(r, ch * 8), src, e < a.E ? 16u : 0u);
        }
      } else if (threadIdx.x == 0) {
        mbar_arrive_expect_tx(&G.raw_full[s], (uint32_t)RAW_STAGE);
        for (int p = 0; p < BM / 16; ++p)
          bulk_g2s_stream(raw + s * RAW_STAGE + p * KG_NVFP4, wbase + p * wtile + (int64_t)kb * KG_NVFP4,
                          (uint32_t)KG_NVFP4, &G.raw_full[s]);
      }
      for (int c = threadIdx.x; c < n * 8; c += THREADS) {
        const int r = c >> 3, ch = c & 7;
        cp_async16(b_op + s * B_STAGE + sw128_off(r, ch * 8), G.src[r] + kb * BK + ch * 8, 16u);
      }
    };

    const uint32_t g0 = gk;
    bool ok = true;
    for (int p = 0; p < PREF; ++p) {
      const uint32_t gq = g0 + p;
      if (p < KB) {
        if (gq >= STAGES) ok &= mbar_wait(&G.mma_done[gq % STAGES], ((gq / STAGES) - 1) & 1, status);
        if (ok) issue(p, gq % STAGES);
      }
      cp_async_commit();
    }
    const uint32_t idesc = idesc_bf16_f32(BM, (n + 15) & ~15);
    for (int kb = 0; kb < KB; ++kb) {
      const uint32_t g = g0 + kb, s = g % STAGES;
      cp_async_wait<PREF - 1>();
      if (MODE != ROUTER && ok) {
        ok = mbar_wait(&G.raw_full[s], (g / STAGES) & 1, status);
        if (ok) {
          // Warp w dequantises packed tile w: rows 16 w .. 16 w + 15 of the block.
          const uint8_t* kp = raw + s * RAW_STAGE + warp * KG_NVFP4;
          const uint4 codes = lds128(kp + lane * 16);
          const int gr = lane >> 2, t4 = lane & 3;
          const uint32_t sg = lds32(kp + KG_CODE_BYTES + gr * 4);
          const uint32_t sg8 = lds32(kp + KG_CODE_BYTES + (gr + 8) * 4);
          const uint32_t cw[4] = {codes.x, codes.y, codes.z, codes.w};
          uint8_t* ap = base_ptr + s * A_STAGE;
          const int r0 = warp * 16 + gr;
#pragma unroll
          for (int ks = 0; ks < 4; ++ks) {
            uint32_t af[4];
            nvfp4_afrag(cw[ks], sg, sg8, ks, af);
            const int c0 = ks * 16 + 2 * t4;
            *reinterpret_cast<uint32_t*>(ap + sw128_off(r0, c0)) = f16x2_to_bf16x2(af[0]);
            *reinterpret_cast<uint32_t*>(ap + sw128_off(r0 + 8, c0)) = f16x2_to_bf16x2(af[1]);
            *reinterpret_cast<uint32_t*>(ap + sw128_off(r0, c0 + 8)) = f16x2_to_bf16x2(af[2]);
            *reinterpret_cast<uint32_t*>(ap + sw128_off(r0 + 8, c0 + 8)) = f16x2_to_bf16x2(af[3]);
          }
        }
      }
      fence_proxy_async();  // this thread's cp.async and st.shared data -> visible to the tensor core
      if (__syncthreads_or(!ok)) {
        failed = true;
        break;
      }
      if (threadIdx.x == 0) {
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < BK / 16; ++ks)
          tc_mma(tmem, sw128_desc(a_op + s * A_STAGE + ks * 32), sw128_desc(b_op + s * B_STAGE + ks * 32), idesc,
                 (kb > 0 || ks > 0) ? 1u : 0u);
        tc_commit(&G.mma_done[s]);
      }
      // Prefetch k-block kb + PREF once the MMAs that last read its stage are done.
      const int kn = kb + PREF;
      if (kn < KB) {
        const uint32_t gq = g0 + kn;
        if (gq >= STAGES) ok &= mbar_wait(&G.mma_done[gq % STAGES], ((gq / STAGES) - 1) & 1, status);
        if (ok) issue(kn, gq % STAGES);
      }
      cp_async_commit();
    }
    gk = g0 + KB;
    if (failed) break;
    // All MMAs of the tile: the commit of its last k-block covers them.
    ok = mbar_wait(&G.mma_done[(gk - 1) % STAGES], ((gk - 1) / STAGES) & 1, status);
    if (__syncthreads_or(!ok)) {
      failed = true;
      break;
    }
    tc_fence_after();

    // Epilogue: warp w reads tensor-memory lanes 32 (w % 4) .. + 31 (weight
    // rows), columns 64 (w / 4) .. + 63 (tokens), 16 at a time.
    const int q4 = warp & 3, chalf = warp >> 2;
    const int r = q4 * 32 + lane;  // weight row within the m-tile
    for (int c0 = chalf * 64; c0 < chalf * 64 + 64 && c0 < n; c0 += 16) {
      uint32_t v[16];
      tc_ld16(tmem + ((uint32_t)(q4 * 32) << 16) + (uint32_t)c0, v);
      if (MODE == ROUTER) {
        const int e = mt * BM + r;
        float* logits = ws_at<float>(a, a.W.logits);
#pragma unroll
        for (int j = 0; j < 16; ++j)
          if (e < a.E && c0 + j < n) logits[(size_t)(row0 + c0 + j) * a.E + e] = __uint_as_float(v[j]);
      } else if (MODE == GATEUP) {
        // Rows 16 t .. 16 t + 7 of packed tile t are gate rows, the next 8 the
        // up rows of the same intermediate indices (8 (8 mt + t) + r % 8).
        const float Gg = a.globals[expert * 4 + 0], Gu = a.globals[expert * 4 + 1];
        const bool gate = (lane & 8) == 0;
        const int i = (mt * 8 + q4 * 2 + (lane >> 4)) * 8 + (lane & 7);
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const float up = __shfl_down_sync(0xffffffffu, __uint_as_float(v[j]), 8);
          if (gate && c0 + j < n) {
            const float gv = __uint_as_float(v[j]) * Gg;
            const float uv = up * Gu;
            const float sv = gv / (1.0f + expf(-gv));
            const __nv_bfloat16 hb = __float2bfloat16_rn(sv * uv);
            hbuf[(size_t)(row0 + c0 + j) * a.I + i] = *reinterpret_cast<const uint16_t*>(&hb);
          }
        }
      } else {
        const float Gd = a.globals[expert * 4 + 2];
        float* y = ws_at<float>(a, a.W.y);
        const int jrow = mt * BM + r;
        const int q_per_tok = a.S + a.k;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int c = c0 + j;
          if (c < n)
            y[((size_t)G.col_tok[c] * q_per_tok + G.col_q[c]) * a.H + jrow] =
                G.col_w[c] * (__uint_as_float(v[j]) * Gd);
        }
      }
    }
    tc_fence_before();
    __syncthreads();  // tensor memory and the column tables are free for the next tile
    tc_fence_after();
  }

  if (failed) {  // let in-flight copies and MMAs land before the memory goes away
    cp_async_wait<0>();
    for (uint32_t g = (gk >= STAGES ? gk - STAGES : 0); g < gk; ++g) {
      mbar_drain(&G.mma_done[g % STAGES], (g / STAGES) & 1);
      if (MODE != ROUTER) mbar_drain(&G.raw_full[g % STAGES], (g / STAGES) & 1);
    }
  }
  cp_async_wait<0>();
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS) : "memory");
  }
}

// ---------------------------------------------------------------------------
// Sigmoid top-k per token: one warp per token. key = sigmoid(logit) + bias;
// larger key first, equal keys to the lower expert index.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t order_f32(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__global__ void __launch_bounds__(256) k_pf_topk(PfArgs a) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * 8 + warp;
  if (t >= a.B) return;
  constexpr int PER = MAX_E / 32;
  const float* logits = ws_at<float>(a, a.W.logits) + (size_t)t * a.E;
  float s[PER];
  uint32_t key[PER];
  uint32_t taken = 0;
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    const int e = lane + 32 * i;
    s[i] = 0.f;
    key[i] = 0u;
    if (e < a.E) {
      const float l = __ldcg(logits + e);
      s[i] = 1.0f / (1.0f + expf(-l));
      key[i] = order_f32(s[i] + (a.bias ? a.bias[e] : 0.f));
    } else {
      taken |= 1u << i;
    }
  }
  int sel_e[MAX_TOPK];
  float sel_s[MAX_TOPK];
  for (int j = 0; j < a.k; ++j) {
    uint64_t best = 0;
#pragma unroll
    for (int i = 0; i < PER; ++i) {
      const uint64_t c = ((uint64_t)key[i] << 32) | (uint32_t)(0xFFFFFFFFu - (uint32_t)(lane + 32 * i));
      if (!((taken >> i) & 1u) && c > best) best = c;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const uint64_t other = __shfl_xor_sync(0xffffffffu, best, o);
      best = other > best ? other : best;
    }
    const int e = (int)(0xFFFFFFFFu - (uint32_t)best);
    const int owner = e & 31, slot_i = e >> 5;
    float se = 0.f;
#pragma unroll
    for (int i = 0; i < PER; ++i)
      if (i == slot_i) se = s[i];
    se = __shfl_sync(0xffffffffu, se, owner);
    if (lane == owner) taken |= 1u << slot_i;
    sel_e[j] = e;
    sel_s[j] = se;
  }
  if (lane == 0) {
    float sum = 0.f;
    for (int j = 0; j < a.k; ++j) sum += sel_s[j];
    int* idx = ws_at<int>(a, a.W.idx) + (size_t)t * a.k;
    float* w = ws_at<float>(a, a.W.w) + (size_t)t * a.k;
    int* pos = ws_at<int>(a, a.W.pos) + (size_t)t * a.k;
    int* counts = ws_at<int>(a, a.W.counts);
    for (int j = 0; j < a.k; ++j) {
      const float wj = a.renorm ? sel_s[j] / sum : sel_s[j];
      idx[j] = sel_e[j];
      w[j] = wj * a.routed_scale;
      pos[j] = atomicAdd(counts + sel_e[j], 1);
    }
  }
}

// ---------------------------------------------------------------------------
// Plan (one block): slots = the S shared experts (every token), then the
// experts with tokens in ascending id; grouped rows = shared slots' B rows each,
// then each routed expert's tokens; tile lists (slot, m-tile, first row, n).
// ---------------------------------------------------------------------------
constexpr int PLAN_THREADS = 1024;

__device__ int block_exclusive_scan(int v, int* sh) {  // sh: 32 ints
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int u = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += u;
  }
  __syncthreads();
  if (lane == 31) sh[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = lane < (int)(blockDim.x >> 5) ? sh[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += u;
    }
    sh[lane] = w;  // inclusive over warps
  }
  __syncthreads();
  return incl - v + (warp > 0 ? sh[warp - 1] : 0);
}

__global__ void __launch_bounds__(PLAN_THREADS) k_pf_plan(PfArgs a) {
  __shared__ int sh[32];
  __shared__ int s_rowbase[MAX_E];
  __shared__ int s_slot_cnt[PLAN_THREADS], s_slot_row0[PLAN_THREADS];
  __shared__ int s_nslots, s_ntiles;
  int* counts = ws_at<int>(a, a.W.counts);
  const int e = threadIdx.x;
  const int c = e < a.E ? __ldcg(counts + e) : 0;
  // Grouped rows and slot numbers of the routed experts (ascending id).
  const int rb = block_exclusive_scan(c, sh);
  const int sl = block_exclusive_scan(c > 0 ? 1 : 0, sh);
  if (e < a.E) s_rowbase[e] = a.S * a.B + rb;
  if (e < a.E && c > 0) {
    s_slot_cnt[a.S + sl] = c;
    s_slot_row0[a.S + sl] = a.S * a.B + rb;
    ws_at<int>(a, a.W.slot_expert)[a.S + sl] = e;
  }
  if (e < a.S) {
    s_slot_cnt[e] = a.B;
    s_slot_row0[e] = e * a.B;
    ws_at<int>(a, a.W.slot_expert)[e] = a.E + e;
  }
  if (e == PLAN_THREADS - 1) s_nslots = a.S + sl + (c > 0 ? 1 : 0);
  __syncthreads();
  const int nslots = s_nslots;
  // Token tiles per slot (one slot per thread: S + E <= PLAN_THREADS).
  const int s = threadIdx.x;
  const int cnt = s < nslots ? s_slot_cnt[s] : 0;
  const int ntl = (cnt + NT - 1) / NT;
  const int tb = block_exclusive_scan(ntl, sh);
  if (s == PLAN_THREADS - 1) s_ntiles = tb + ntl;
  const int mgu = 2 * a.I / BM, mdn = a.H / BM;
  if (s < nslots) {
    const int row0 = s_slot_row0[s];
    ws_at<int>(a, a.W.slot_row0)[s] = row0;
    ws_at<int>(a, a.W.slot_count)[s] = cnt;
    int4* gu = ws_at<int4>(a, a.W.gu_tiles);
    int4* dn = ws_at<int4>(a, a.W.dn_tiles);
    for (int q = 0; q < ntl; ++q) {
      const int n = min(NT, cnt - q * NT);
      for (int m = 0; m < mgu; ++m) gu[(size_t)(tb + q) * mgu + m] = make_int4(s, m, row0 + q * NT, n);
      for (int m = 0; m < mdn; ++m) dn[(size_t)(tb + q) * mdn + m] = make_int4(s, m, row0 + q * NT, n);
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int* hdr = ws_at<int>(a, 0);
    hdr[PF_NSLOTS] = nslots;
    hdr[PF_NGU] = s_ntiles * mgu;
    hdr[PF_NDN] = s_ntiles * mdn;
  }
  // Token lists: grouped row -> (token, slot rank q, routing weight).
  int* list_tok = ws_at<int>(a, a.W.list_tok);
  int* list_q = ws_at<int>(a, a.W.list_q);
  float* list_w = ws_at<float>(a, a.W.list_w);
  for (int p = threadIdx.x; p < a.S * a.B; p += PLAN_THREADS) {
    list_tok[p] = p % a.B;
    list_q[p] = p / a.B;
    list_w[p] = 1.0f;
  }
  const int* idx = ws_at<int>(a, a.W.idx);
  const float* w = ws_at<float>(a, a.W.w);
  const int* pos = ws_at<int>(a, a.W.pos);
  for (int p = threadIdx.x; p < a.B * a.k; p += PLAN_THREADS) {
    const int ex = __ldcg(idx + p);
    const int row = s_rowbase[ex] + __ldcg(pos + p);
    list_tok[row] = p / a.k;
    list_q[row] = a.S + p % a.k;
    list_w[row] = __ldcg(w + p);
  }
  if (e < a.E) counts[e] = 0;  // ready for the next call (every read of counts is above)
}

// out[t][j] = bf16(sum over q of y[t][q][j]), q = shared experts, then top-k ranks.
__global__ void __launch_bounds__(256) k_pf_combine(PfArgs a) {
  const int Q = a.S + a.k;
  const size_t n4 = (size_t)a.B * a.H / 4;
  const float* y = ws_at<float>(a, a.W.y);
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n4; i += (size_t)gridDim.x * blockDim.x) {
    const size_t t = i / (a.H / 4), j4 = i % (a.H / 4);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int q = 0; q < Q; ++q) {
      const float4 v = __ldcg(reinterpret_cast<const float4*>(y + (t * Q + q) * a.H) + j4);
      acc.x += v.x;
      acc.y += v.y;
      acc.z += v.z;
      acc.w += v.w;
    }
    const __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y), hi = __floats2bfloat162_rn(acc.z, acc.w);
    uint2 o;
    o.x = *reinterpret_cast<const uint32_t*>(&lo);
    o.y = *reinterpret_cast<const uint32_t*>(&hi);
    *reinterpret_cast<uint2*>(a.out + t * a.H + j4 * 4) = o;
  }
}

__global__ void k_pf_debug_routing(const int* idx, const float* w, const float* logits, int n, int nl, int* oi,
                                   float* ow, float* ol) {
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n || i < nl; i += gridDim.x * blockDim.x) {
    if (i < n) {
      oi[i] = idx[i];
      ow[i] = w[i];
    }
    if (ol && i < nl) ol[i] = logits[i];
  }
}

// ---------------------------------------------------------------------------
// Host side.
// ---------------------------------------------------------------------------
static flint_moe_status cfg_supported(const flint_moe_config* c) {
  const flint_moe_status st = flint_moe_check_config(c);
  if (st != FLINT_MOE_OK) return st;
  if (c->weight_fmt != FLINT_MOE_NVFP4) return FLINT_MOE_EUNSUPPORTED;
  if (c->hidden % BM || (2 * c->inter) % BM || c->num_experts > MAX_E || c->top_k > MAX_TOPK)
    return FLINT_MOE_EUNSUPPORTED;
  if (c->n_shared + c->num_experts > PLAN_THREADS) return FLINT_MOE_EUNSUPPORTED;
  return FLINT_MOE_OK;
}

static int sm_count() {
  static std::atomic<int> n{0};
  int v = n.load();
  if (v == 0) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0)
      v = 148;
    n.store(v);
  }
  return v;
}

template <int MODE>
static cudaError_t launch_gemm(const PfArgs& a, int grid, cudaStream_t stream) {
  static std::atomic<int> attr_set{0};
  const size_t smem = gemm_dyn_smem();
  if (!attr_set.load()) {
    cudaError_t e = cudaFuncSetAttribute(k_pf_gemm<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    attr_set.store(1);
  }
  k_pf_gemm<MODE><<<grid, THREADS, smem, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace pf
}  // namespace flint

using namespace flint;
using namespace flint::pf;

extern "C" size_t flint_moe_prefill_workspace_bytes(const flint_moe_config* c, int32_t max_tokens) {
  if (cfg_supported(c) != FLINT_MOE_OK) return 0;
  if (max_tokens < 1 || max_tokens > FLINT_MOE_PREFILL_MAX_TOKENS) return 0;
  return make_pf_layout(c->hidden, c->num_experts, c->top_k, c->inter, c->n_shared, max_tokens).total;
}

extern "C" flint_moe_status flint_moe_prefill_workspace_init(const flint_moe_config* c, int32_t max_tokens,
                                                             void* ws, cudaStream_t stream) {
  const flint_moe_status st = cfg_supported(c);
  if (st != FLINT_MOE_OK) return st;
  if (!ws || max_tokens < 1 || max_tokens > FLINT_MOE_PREFILL_MAX_TOKENS) return FLINT_MOE_EINVAL;
  if ((uintptr_t)ws % 256) return FLINT_MOE_EALIGN;
  const PfLayout W = make_pf_layout(c->hidden, c->num_experts, c->top_k, c->inter, c->n_shared, max_tokens);
  if (cudaMemsetAsync(ws, 0, W.counts + sizeof(int) * c->num_experts, stream) != cudaSuccess)
    return FLINT_MOE_ECUDA;
  return FLINT_MOE_OK;
}

extern "C" flint_moe_status flint_moe_prefill(const flint_moe_layer* layer, const uint16_t* x, int32_t B,
                                              uint16_t* out, void* ws, size_t ws_bytes, cudaStream_t stream) {
  if (!layer) return FLINT_MOE_EINVAL;
  const flint_moe_config* c = &layer->cfg;
  const flint_moe_status st = cfg_supported(c);
  if (st != FLINT_MOE_OK) return st;
  if (B < 0 || B > FLINT_MOE_PREFILL_MAX_TOKENS) return FLINT_MOE_EINVAL;
  if (B == 0) return FLINT_MOE_OK;
  if (!x || !out || !ws || !layer->packed || !layer->router) return FLINT_MOE_EINVAL;
  if ((uintptr_t)x % 16 || (uintptr_t)out % 16 || (uintptr_t)ws % 256 || (uintptr_t)layer->packed % 16 ||
      (uintptr_t)layer->router % 16)
    return FLINT_MOE_EALIGN;
  const size_t xb = (size_t)B * c->hidden * 2;
  const uintptr_t xa = (uintptr_t)x, oa = (uintptr_t)out;
  if (xa < oa + xb && oa < xa + xb) return FLINT_MOE_EINVAL;
  PfArgs a;
  a.H = c->hidden;
  a.I = c->inter;
  a.E = c->num_experts;
  a.S = c->n_shared;
  a.k = c->top_k;
  a.B = B;
  a.renorm = c->renormalize;
  a.routed_scale = c->routed_scale;
  a.x = x;
  a.router = layer->router;
  a.bias = layer->sel_bias;
  a.packed = static_cast<const uint8_t*>(layer->packed);
  a.L = make_layout(a.H, a.I, a.E, a.S, FLINT_MOE_NVFP4);
  a.globals = reinterpret_cast<const float*>(a.packed + a.L.globals_off);
  a.ws = static_cast<uint8_t*>(ws);
  a.W = make_pf_layout(a.H, a.E, a.k, a.I, a.S, B);
  a.out = out;
  if (ws_bytes < a.W.total) return FLINT_MOE_EINVAL;

  const int nsm = sm_count();
  const int router_tiles = ((a.E + BM - 1) / BM) * ((B + NT - 1) / NT);
  if (launch_gemm<ROUTER>(a, std::min(nsm, router_tiles), stream) != cudaSuccess) return FLINT_MOE_ECUDA;
  k_pf_topk<<<(B + 7) / 8, 256, 0, stream>>>(a);
  if (cudaGetLastError() != cudaSuccess) return FLINT_MOE_ECUDA;
  k_pf_plan<<<1, PLAN_THREADS, 0, stream>>>(a);
  if (cudaGetLastError() != cudaSuccess) return FLINT_MOE_ECUDA;
  if (launch_gemm<GATEUP>(a, std::min(nsm, a.W.max_gu), stream) != cudaSuccess) return FLINT_MOE_ECUDA;
  if (launch_gemm<DOWN>(a, std::min(nsm, a.W.max_dn), stream) != cudaSuccess) return FLINT_MOE_ECUDA;
  const int cgrid = (int)std::min<size_t>((size_t)nsm * 8, ((size_t)B * a.H / 4 + 255) / 256);
  k_pf_combine<<<cgrid, 256, 0, stream>>>(a);
  if (cudaGetLastError() != cudaSuccess) return FLINT_MOE_ECUDA;
  return FLINT_MOE_OK;
}

extern "C" flint_moe_status flint_moe_prefill_debug_routing(const flint_moe_config* c, const void* ws, int32_t B,
                                                            int32_t* idx, float* w, float* logits,
                                                            cudaStream_t stream) {
  const flint_moe_status st = cfg_supported(c);
  if (st != FLINT_MOE_OK) return st;
  if (!ws || !idx || !w || B < 1 || B > FLINT_MOE_PREFILL_MAX_TOKENS) return FLINT_MOE_EINVAL;
  const PfLayout W = make_pf_layout(c->hidden, c->num_experts, c->top_k, c->inter, c->n_shared, B);
  const uint8_t* b = static_cast<const uint8_t*>(ws);
  const int n = B * c->top_k, nl = logits ? B * c->num_experts : 0;
  k_pf_debug_routing<<<64, 256, 0, stream>>>(reinterpret_cast<const int*>(b + W.idx),
                                              reinterpret_cast<const float*>(b + W.w),
                                              reinterpret_cast<const float*>(b + W.logits), n, nl, idx, w, logits);
  return cudaGetLastError() == cudaSuccess ? FLINT_MOE_OK : FLINT_MOE_ECUDA;
}
