// Expert-grouped tensor-core path of the Flint-style W4A16 MoE layer for many
// tokens ("Day-0 Support for Flint on vLLM", section "Optimisation": the MoE
// kernels were also the largest prefill gain).
//
// With many tokens per expert the weights are worth staging: every 128-row x
// 64-column weight block is dequantised once (E2M1 x E4M3 products are exact in
// f16 and in bf16) into shared memory in the 128-byte-swizzled K-major layout
// that tcgen05.mma reads, the expert's token rows arrive in the same layout by
// TMA, and one elected thread issues the tensor-core MMAs (M = 128 weight rows,
// N = up to 128 tokens, K = 16 per instruction) that accumulate in FP32 in
// tensor memory. The epilogue reads the accumulators back with tcgen05.ld.
//
//   k_pf_gemm<ROUTER>  logits = Wr x^T      (bf16 router rows and tokens by TMA;
//                      split along H into up to 8 k-ranges while the tiles are
//                      fewer than the SMs)
//   k_pf_topk          adds the splits' partial logits in split order; sigmoid
//                      top-k per token; tokens counted per expert
//   k_pf_plan          slots, grouped-row bases, tile lists (one block)
//   k_pf_token_rows    per token: its grouped-list entries, its f16 rows
//   k_pf_gemm<GATEUP>  h = bf16(silu(G_g g) * G_u u) per (token, expert), f16 MMA
//   k_pf_small<GATEUP> the same for slots of few rows (up to 512-token calls):
//                      tiles of up to 16 tokens on mma.sync, dequantised in registers
//   k_pf_gemm<DOWN>    y[t][q] = w * G_d (c_d h) per (token, expert), bf16 MMA
//   k_pf_small<DOWN>   the same for the small tiles
//   k_pf_combine       out = bf16(sum_q y[t][q]) in slot order
#include <algorithm>
#include <atomic>
#include <cmath>

#include <cuda.h>  // CUtensorMap and its enums (types only; the encoder comes through the runtime)

#include "common.cuh"
#include "flint_moe_prefill.h"

namespace flint {
namespace pf {

constexpr int BM = 128;       // weight rows per tile (MMA M)
constexpr int BK = 64;        // k per pipeline stage: one 128-byte swizzle row of bf16
constexpr int NT = 128;       // tokens per tile at most (MMA N)
constexpr int SN = 16;                 // tokens per small tile (two 8-column groups of mma.sync)
constexpr int SMALL_MAX = 16;          // routed slots of up to this many rows take small tiles (when they fit)
constexpr int SMALL_SHARED_MAX = 256;  // shared-expert slots (B rows) likewise
constexpr int SMALL_B_MAX = 512;       // calls of more tokens use the tensor-core tiles only
constexpr int NPIPE = 2;      // independent GEMM pipelines per CTA (one CTA per SM)
constexpr int KPS = 1;        // k-blocks per operand stage
constexpr int STAGES = 2;     // operand stages per pipeline
constexpr uint32_t TMEM_COLS = 512;  // per pipeline two accumulator buffers of NT columns
constexpr int A_KBLK = BM * BK * 2;               // 16 KiB: one k-block of the weight operand
constexpr int B_KBLK = NT * BK * 2;               // 16 KiB: one k-block of the token operand
constexpr int A_STAGE = KPS * A_KBLK;
constexpr int B_STAGE = KPS * B_KBLK;
constexpr int MAX_E = 512;

enum Mode : int { ROUTER = 0, GATEUP = 1, DOWN = 2 };
enum : int { PF_STATUS = HDR_STATUS, PF_NSLOTS = 2, PF_NGU = 3, PF_NDN = 4, PF_NGUS = 5, PF_NDNS = 6 };

// Workspace: header words, then 256-byte aligned regions sized for T tokens.
struct PfLayout {
  size_t counts, logits, idx, w, pos, slot_expert, slot_row0, slot_count, list_tok, list_q, list_w, gu_tiles,
      dn_tiles, gus_tiles, dns_tiles, rowbase, kx, xn, x16, xg, h, y, total;
  int max_slots, max_rows, max_gu, max_dn, max_gus, max_dns;
};

__host__ __device__ inline PfLayout make_pf_layout(int H, int E, int k, int I, int S, int T) {
  PfLayout W;
  W.max_slots = S + (E < T * k ? E : T * k);
  W.max_rows = T * (S + k);
  // sum over slots of ceil(count / NT) <= rows / NT + slots
  const int max_nt = W.max_rows / NT + W.max_slots + 1;
  W.max_gu = max_nt * (2 * I / BM);
  W.max_dn = max_nt * (H / BM);
  // small token tiles: the shared slots' B <= SMALL_SHARED_MAX rows, the routed slots' <= SMALL_MAX rows
  const int max_nts = S * (SMALL_SHARED_MAX / SN) + W.max_slots * (SMALL_MAX / SN);
  W.max_gus = max_nts * (2 * I / BM);
  W.max_dns = max_nts * (H / BM);
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
  W.gus_tiles = o;   o = ws_align(o + sizeof(int4) * (size_t)W.max_gus);
  W.dns_tiles = o;   o = ws_align(o + sizeof(int4) * (size_t)W.max_dns);
  W.rowbase = o;     o = ws_align(o + sizeof(int) * E);                // first grouped row of each routed expert
  W.kx = o;          o = ws_align(o + sizeof(int) * (size_t)T);       // per-token power-of-two prescale
  W.xn = o;          o = ws_align(o + (size_t)2 * T * H);             // RMS-normalised x (pre-norm block)
  W.x16 = o;         o = ws_align(o + (size_t)2 * T * H);             // x * 2^kx in f16
  W.xg = o;          o = ws_align(o + (size_t)2 * T * k * H);         // the same rows grouped by routed expert
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
  // Pre-norm block: x is the normalised residual stream (in the workspace),
  // res the residual stream itself, added to the output by the combine.
  int prenorm;
  const uint16_t* res;     // [B][H]
  const uint16_t* gamma;   // [H]
  float eps;
  // Router GEMM split along H into rsplit k-ranges (1, 2, 4 or 8): split s
  // writes its partial logits [B][E] at y + s B E (the expert outputs y are
  // written only later, by the down GEMM), and k_pf_topk adds the splits in
  // order and stores the logits.
  int rsplit;
  // Routed slots with at most small_max grouped rows, and shared slots with at
  // most small_shared (0: none), take small tiles of up to SN tokens, multiplied
  // on the mma.sync path (k_pf_small); the others take the tensor-core tiles
  // of up to NT tokens.
  int small_max, small_shared;
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

// Instruction descriptor of kind::f16: D f32 (bits 4-5 = 1), A and B both
// bf16 (bits 7-9 = 1, 10-12 = 1) or both f16 (0, 0), both K-major (bits 15,
// 16 = 0), N >> 3 in bits 17-22, M >> 4 in bits 24-28.
__device__ __forceinline__ uint32_t idesc_f32acc(int M, int N, bool bf16) {
  const uint32_t t = bf16 ? 1u : 0u;
  return (1u << 4) | (t << 7) | (t << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
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

// bf16x2 -> f16x2 of the values times sc (a power of two).
__device__ __forceinline__ uint32_t bf16x2_to_f16x2_scaled(uint32_t w, float sc) {
  const __half2 hv = __floats2half2_rn(bf16lo(w) * sc, bf16hi(w) * sc);
  return *reinterpret_cast<const uint32_t*>(&hv);
}


// ---------------------------------------------------------------------------
// The grouped GEMM. A tile is (slot, m-tile of 128 weight rows, first grouped
// row, token count n <= NT); the kernel is persistent over its tiles
// blockIdx.x, blockIdx.x + gridDim.x, ..., and treats their k-blocks as one
// stream: k-block g of the CTA is k-block g % KB of its tile g / KB.
//
// Warp roles, handing off through mbarriers only (no block-wide barrier in
// the main loop):
//   warp 16  streams the packed weights into a ring of RAW_SL slots of RAW_KB
//            k-blocks (lane p copies packed tile p's run of k-groups: few,
//            large bulk copies), as far ahead as the ring allows, across tiles;
//   warp 17  loads each stage's 128 activation rows per k-block (and the
//            router's weight rows) with TMA in the 128-byte swizzle;
//   warp 18  issues the MMAs of a stage (KPS k-blocks x 4 k-steps) once its
//            single mbarrier reports both operands in, commits them to the
//            stage's mbarrier, and after a tile's last k-block to the
//            accumulator buffer's mbarrier;
//   warps 0-15 dequantise the packed k-blocks into the stages' operands, two
//            groups of 8 warps taking alternate stages (warp w: packed tile
//            w % 8), and run the epilogue of each tile from tensor memory. Two
//            accumulator buffers (columns 0-127, 128-255) let the MMAs of the
//            next tile start before the epilogue of this one has finished.
// ---------------------------------------------------------------------------
constexpr int PCW = 8;                      // dequantising warps per pipeline
constexpr int W_PROD0 = NPIPE * PCW;         // producer warp of pipeline p: W_PROD0 + p
constexpr int W_MMA0 = W_PROD0 + NPIPE;      // MMA-issue warp of pipeline p: W_MMA0 + p
constexpr int GEMM_THREADS = (W_MMA0 + NPIPE) * 32;
constexpr int RAW_KB = 4;   // k-blocks of one packed weight slot (eight copies of RAW_KB k-groups)
constexpr int RAW_SL = 2;   // slots per pipeline: up to 8 k-blocks in flight
constexpr int RAW_SLOT = (BM / 16) * RAW_KB * KG_NVFP4;  // 18 KiB
constexpr int PIPE_BYTES = STAGES * (A_STAGE + B_STAGE) + RAW_SL * RAW_SLOT;  // 100 KiB

struct PfMaps {  // TMA descriptors, bf16, 64-column x 128-row boxes, 128-byte swizzle
  CUtensorMap a;   // router rows (router GEMM)
  CUtensorMap b0;  // activations: x (router GEMM, shared experts' gate/up), h (down)
  CUtensorMap b1;  // the routed pairs' grouped activation rows (gate/up)
};

struct GemmSmem {  // per pipeline
  uint64_t raw_full[NPIPE][RAW_SL];
  uint64_t raw_empty[NPIPE][RAW_SL];
  uint64_t full[NPIPE][STAGES];      // the stage's token rows landed (TMA) and its weights are dequantised
  uint64_t mma_done[NPIPE][STAGES];
  uint64_t acc_full[NPIPE][2];
  uint64_t acc_empty[NPIPE][2];
  uint32_t tmem_base;
  int abort;
};

constexpr size_t gemm_dyn_smem() { return 1024 + (size_t)NPIPE * PIPE_BYTES; }

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// One lane of the (fully active) warp returns true.
__device__ __forceinline__ bool elect_one() {
  uint32_t pred = 0;
  asm volatile(
      "{\n\t.reg .b32 rx;\n\t.reg .pred px;\n\telect.sync rx|px, %1;\n\t@px mov.s32 %0, 1;\n\t}"
      : "+r"(pred)
      : "r"(0xffffffffu));
  return pred != 0;
}

__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// Bulk copy global -> shared with an L2 cache policy, completing on bar.
__device__ __forceinline__ void bulk_g2s_pol(uint32_t dst, const void* src, uint32_t bytes, uint64_t* bar,
                                             uint64_t pol) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          dst),
      "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(pol)
      : "memory");
}

// 2-D TMA tile load (box from the descriptor) into shared memory, completing on bar.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::
          "r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar))
      : "memory");
}

// Bounded wait that also gives up as soon as another warp of the CTA has given up.
__device__ __forceinline__ bool wait_ab(uint64_t* bar, uint32_t parity, volatile int* abort, int* status) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  for (uint32_t it = 0;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 63) == 63) {
      if (*abort) return false;
      if (global_ns() - t0 > WAIT_LIMIT_NS) {
        atomicOr(status, FLINT_MOE_DEV_ERR_TIMEOUT);
        *abort = 1;
        return false;
      }
    }
  }
}

struct TileInfo {
  int slot, mt, row0, n, expert;
};

template <int MODE>
__device__ __forceinline__ TileInfo tile_info(const PfArgs& a, int tile) {
  TileInfo t;
  if (MODE == ROUTER) {  // tile = (split * ntc + token tile) * mtc + m-tile; slot = the split
    const int mtc = (a.E + BM - 1) / BM, ntc = (a.B + NT - 1) / NT;
    t.mt = tile % mtc;
    t.slot = tile / mtc / ntc;
    t.row0 = (tile / mtc % ntc) * NT;
    t.n = min(NT, a.B - t.row0);
    t.expert = 0;
  } else {
    const int4 v = __ldcg(ws_at<const int4>(a, MODE == GATEUP ? a.W.gu_tiles : a.W.dn_tiles) + tile);
    t.slot = v.x;
    t.mt = v.y;
    t.row0 = v.z;
    t.n = v.w;
    t.expert = __ldcg(ws_at<const int>(a, a.W.slot_expert) + v.x);
  }
  return t;
}

template <int MODE>
__global__ void __launch_bounds__(GEMM_THREADS, 1) k_pf_gemm(const PfArgs a, const __grid_constant__ PfMaps maps) {
  extern __shared__ uint8_t dsmem[];
  __shared__ GemmSmem G;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // Pipeline of this warp, its shared memory and tensor-memory columns.
  const int p = warp < W_PROD0 ? warp / PCW : (warp < W_MMA0 ? warp - W_PROD0 : warp - W_MMA0);
  const uint32_t base = ((smem_addr(dsmem) + 1023u) & ~1023u) + (uint32_t)(p * PIPE_BYTES);
  uint8_t* const base_ptr = dsmem + (base - smem_addr(dsmem));
  const uint32_t a_op = base;                                   // STAGES x 16 KiB
  const uint32_t b_op = base + STAGES * A_STAGE;                // STAGES x 16 KiB
  uint8_t* const raw = base_ptr + STAGES * (A_STAGE + B_STAGE);  // RAW_SL x 18 KiB
  int* status = ws_at<int>(a, 0) + PF_STATUS;
  volatile int* abort = &G.abort;

  const int K = MODE == DOWN ? a.I : a.H;
  const int KB = K / BK / (MODE == ROUTER ? a.rsplit : 1);  // k-blocks per tile
  const int n_tiles = MODE == ROUTER ? ((a.E + BM - 1) / BM) * ((a.B + NT - 1) / NT) * a.rsplit
                                     : __ldcg(ws_at<int>(a, 0) + (MODE == GATEUP ? PF_NGU : PF_NDN));
  if ((int)blockIdx.x >= n_tiles) return;  // uniform: no tensor memory taken
  const int cta_tiles = (n_tiles - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x;
  // Pipeline p takes the CTA's tiles p, p + NPIPE, ...
  const int my_tiles = cta_tiles > p ? (cta_tiles - p + NPIPE - 1) / NPIPE : 0;
  const int total = my_tiles * KB;  // k-blocks of this pipeline
  auto tile_of = [&](int i) { return (int)blockIdx.x + (p + NPIPE * i) * (int)gridDim.x; };
  // Packed weights travel in slots of up to RAW_KB k-blocks of one tile.
  const int SPT = (KB + RAW_KB - 1) / RAW_KB;
  const int n_slots = my_tiles * SPT;

  if (threadIdx.x == 0) {
    for (int q = 0; q < NPIPE; ++q) {
      for (int s = 0; s < RAW_SL; ++s) {
        mbar_init(&G.raw_full[q][s], 1);
        mbar_init(&G.raw_empty[q][s], PCW);
      }
      for (int s = 0; s < STAGES; ++s) {
        // the TMA lane's expect-tx arrival, plus one arrival per dequantising warp
        mbar_init(&G.full[q][s], MODE == ROUTER ? 1 : 1 + PCW);
        mbar_init(&G.mma_done[q][s], 1);
      }
      for (int b = 0; b < 2; ++b) {
        mbar_init(&G.acc_full[q][b], 1);
        mbar_init(&G.acc_empty[q][b], PCW);
      }
    }
    G.abort = 0;
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
  const uint32_t tmem = G.tmem_base + (uint32_t)(p * 2 * NT);  // this pipeline's two accumulators

  if (warp >= W_PROD0 && warp < W_MMA0) {
    if (lane == 0 && MODE != ROUTER) {
      // ---------------- packed weights -> raw ring (one lane issues the slot's eight copies) ----------------
      const uint64_t pol = l2_evict_first_policy();
      const int64_t wtile = MODE == GATEUP ? a.L.gu_tile : a.L.dn_tile;
      int u = 0;
      TileInfo nxt = my_tiles > 0 ? tile_info<MODE>(a, tile_of(0)) : TileInfo{};
      const uint8_t* wsrc = nullptr;
      for (; u < n_slots; ++u) {
        const int sl = u % RAW_SL, i = u / SPT, kb0 = (u % SPT) * RAW_KB;
        const int nk = min(RAW_KB, KB - kb0);
        if (u >= RAW_SL && !wait_ab(&G.raw_empty[p][sl], ((u / RAW_SL) - 1) & 1, abort, status)) break;
        if (kb0 == 0) {
          const TileInfo t = nxt;
          if (i + 1 < my_tiles) nxt = tile_info<MODE>(a, tile_of(i + 1));
          wsrc = a.packed + (int64_t)t.expert * a.L.expert_bytes + (MODE == GATEUP ? 0 : a.L.gu_bytes) +
                 (int64_t)(t.mt * 8) * wtile;
        }
        mbar_arrive_expect_tx(&G.raw_full[p][sl], (uint32_t)((BM / 16) * nk * KG_NVFP4));
        for (int q = 0; q < BM / 16; ++q)
          bulk_g2s_pol(smem_addr(raw + sl * RAW_SLOT + q * RAW_KB * KG_NVFP4), wsrc + q * wtile + (int64_t)kb0 * KG_NVFP4,
                       (uint32_t)(nk * KG_NVFP4), &G.raw_full[p][sl], pol);
      }
      // The CTA's memory must outlive every copy this lane started.
      for (int r = (u > RAW_SL ? u - RAW_SL : 0); r < u; ++r) mbar_drain(&G.raw_full[p][r % RAW_SL], (r / RAW_SL) & 1);
    } else if (lane == 1) {
      // ---------------- token rows (and router weight rows) -> stages, TMA ----------------
      int v = 0;
      TileInfo nxt = my_tiles > 0 ? tile_info<MODE>(a, tile_of(0)) : TileInfo{}, t = nxt;
      for (; v < total; ++v) {
        const int s = v % STAGES, i = v / KB, kb = v % KB;
        if (v >= STAGES && !wait_ab(&G.mma_done[p][s], ((v / STAGES) - 1) & 1, abort, status)) break;
        if (kb == 0) {
          t = nxt;
          if (i + 1 < my_tiles) nxt = tile_info<MODE>(a, tile_of(i + 1));
        }
        mbar_arrive_expect_tx(&G.full[p][s], (uint32_t)(MODE == ROUTER ? A_KBLK + B_KBLK : B_KBLK));
        const int x = ((MODE == ROUTER ? t.slot * KB : 0) + kb) * BK;
        const uint32_t bdst = b_op + s * B_STAGE;
        if (MODE == ROUTER) {
          tma_load_2d(a_op + s * A_STAGE, &maps.a, x, t.mt * BM, &G.full[p][s]);
          tma_load_2d(bdst, &maps.b0, x, t.row0, &G.full[p][s]);
        } else if (MODE == GATEUP) {
          if (t.slot < a.S)  // a shared expert's rows are the tokens in order
            tma_load_2d(bdst, &maps.b0, x, t.row0 - t.slot * a.B, &G.full[p][s]);
          else
            tma_load_2d(bdst, &maps.b1, x, t.row0 - a.S * a.B, &G.full[p][s]);
        } else {
          tma_load_2d(bdst, &maps.b0, x, t.row0, &G.full[p][s]);
        }
      }
      for (int r = (v > STAGES ? v - STAGES : 0); r < v; ++r) mbar_drain(&G.full[p][r % STAGES], (r / STAGES) & 1);
    }
  } else if (warp >= W_MMA0) {
    // ---------------- tensor-core issue (one elected lane) ----------------
    int g = 0;
    TileInfo nxt = my_tiles > 0 ? tile_info<MODE>(a, tile_of(0)) : TileInfo{};
    uint32_t idesc = 0, acc = tmem;

    int s = 0, phase = 0, i = 0, kb = 0;  // stage, its phase parity, tile, k-block
    for (; g < total; ++g) {
      bool ok = true;
      if (kb == 0) {
        const TileInfo t = nxt;
        if (i + 1 < my_tiles) nxt = tile_info<MODE>(a, tile_of(i + 1));
        idesc = idesc_f32acc(BM, (t.n + 15) & ~15, MODE != GATEUP);  // gate/up runs in f16
        acc = tmem + (uint32_t)((i & 1) * NT);
        ok = i < 2 || wait_ab(&G.acc_empty[p][i & 1], ((i / 2) - 1) & 1, abort, status);
      }
      ok = ok && wait_ab(&G.full[p][s], (uint32_t)phase, abort, status);
      if (!__all_sync(0xffffffffu, ok)) break;
      tc_fence_after();
      const uint64_t ad = sw128_desc(a_op + s * A_STAGE), bd = sw128_desc(b_op + s * B_STAGE);
      if (elect_one()) {
#pragma unroll
        for (int ks = 0; ks < BK / 16; ++ks)
          tc_mma(acc, ad + (uint64_t)((ks * 32) >> 4), bd + (uint64_t)((ks * 32) >> 4), idesc, (kb > 0 || ks > 0) ? 1u : 0u);
        tc_commit(&G.mma_done[p][s]);
        if (kb == KB - 1) tc_commit(&G.acc_full[p][i & 1]);
      }
      __syncwarp();
      if (++kb == KB) {
        kb = 0;
        ++i;
      }
      if (++s == STAGES) {
        s = 0;
        phase ^= 1;
      }
    }
    // Let the MMAs in flight finish before the memory goes away.
    if (lane == 0)
      for (int r = (g > STAGES ? g - STAGES : 0); r < g; ++r) mbar_drain(&G.mma_done[p][r % STAGES], (r / STAGES) & 1);
  } else {
    // ---------------- consumers: dequantise, epilogue ----------------
    // Warp lw of the pipeline dequantises packed tile lw (all four k-steps) of
    // every k-block and reads tensor-memory lanes 32 (lw % 4) .., columns
    // 64 (lw / 4) .. of each tile's accumulator.
    const int lw = warp - p * PCW;
    TileInfo nxt = my_tiles > 0 ? tile_info<MODE>(a, tile_of(0)) : TileInfo{}, t = nxt;
    const int dq_p = lw, dq_g = lane >> 2;
    const int q4 = lw & 3, cg = lw >> 2;
    // The k-step's 16 x 16 fragment goes to shared memory with one
    // stmatrix.x4: lanes 8 i .. 8 i + 7 address the rows of 8 x 8 matrix i
    // (rows 8 (i & 1) .., columns 8 (i >> 1) .. of the fragment, the order of
    // the mma A registers), each a 16-byte swizzled chunk.
    uint32_t soff[4];
#pragma unroll
    for (int ks = 0; ks < 4; ++ks)
      soff[ks] = sw128_off(dq_p * 16 + (lane & 7) + ((lane >> 3) & 1) * 8, ks * 16 + (lane >> 4) * 8);
    const uint32_t tile_off = (uint32_t)(dq_p * RAW_KB * KG_NVFP4);
    int ctok[2] = {0, 0}, cq[2] = {0, 0};  // this lane's two epilogue columns: 64 cg + lane, + 32
    float cw[2] = {0.f, 0.f}, cinv[2] = {1.f, 1.f};
    // Deferred epilogue: once all k-blocks of a tile are dequantised, its
    // accumulator is read out one 16-column chunk after each k-block of the
    // next tile (in time this warp would otherwise spend waiting for a free
    // stage), and the rest after the last tile. The MMAs of the tile after
    // next wait for this buffer, so a tile's epilogue always ends before the
    // dequantisation of the following tile does.
    bool pend = false;
    TileInfo pt{};
    int pi = 0, pc = 0;  // the pending tile's index and next chunk column
    int pctok[2] = {0, 0}, pcq[2] = {0, 0};
    float pcw[2] = {0.f, 0.f}, pcinv[2] = {1.f, 1.f};
    auto epi_chunk = [&]() -> bool {  // false: a wait gave up
      const int ab = pi & 1;
      if (pc == cg * 64) {  // before the first chunk: the tile's MMAs are complete
        const bool ok = wait_ab(&G.acc_full[p][ab], (pi / 2) & 1, abort, status);
        if (!__all_sync(0xffffffffu, ok)) return false;
        tc_fence_after();
      }
      const int r = q4 * 32 + lane;  // weight row within the m-tile
      const uint32_t tacc = tmem + (uint32_t)(ab * NT) + ((uint32_t)(q4 * 32) << 16);
      const int c0 = pc;
      if (c0 < cg * 64 + 64 && c0 < pt.n) {
        const int hcol = (c0 - cg * 64) >> 5;  // which of the lane's two column registers
        uint32_t v[16];
        tc_ld16(tacc + (uint32_t)c0, v);
        if (MODE == ROUTER) {
          const int e = pt.mt * BM + r;
          float* logits = a.rsplit > 1 ? ws_at<float>(a, a.W.y) + (size_t)pt.slot * a.B * a.E : ws_at<float>(a, a.W.logits);
#pragma unroll
          for (int j = 0; j < 16; ++j)
            if (e < a.E && c0 + j < pt.n) logits[(size_t)(pt.row0 + c0 + j) * a.E + e] = __uint_as_float(v[j]);
        } else if (MODE == GATEUP) {
          // Rows 16 u .. 16 u + 7 of packed tile u are gate rows, the next 8 the
          // up rows of the same intermediate indices 8 (8 mt + u) + r % 8: lane
          // L and lane L ^ 8 hold (gate, up) of one index. The gate lane
          // finishes the even columns, the up lane the odd ones.
          const float Gg = a.globals[pt.expert * 4 + 0], Gu = a.globals[pt.expert * 4 + 1];
          const bool gate = (lane & 8) == 0;
          const int ii = (pt.mt * 8 + q4 * 2 + (lane >> 4)) * 8 + (lane & 7);
          uint16_t* hbuf = ws_at<uint16_t>(a, a.W.h);
          const float cinv_h = hcol ? pcinv[1] : pcinv[0];
#pragma unroll
          for (int j = 0; j < 16; j += 2) {
            const float v0 = __uint_as_float(v[j]), v1 = __uint_as_float(v[j + 1]);
            const float mine = gate ? v0 : v1;
            const float other = __shfl_xor_sync(0xffffffffu, gate ? v1 : v0, 8);
            const int c = c0 + j + (gate ? 0 : 1);
            const float inv = __shfl_sync(0xffffffffu, cinv_h, c & 31);
            const float gv = (gate ? mine : other) * inv * Gg;
            const float uv = (gate ? other : mine) * inv * Gu;
            const float sv = __fdividef(gv, 1.0f + __expf(-gv));
            if (c < pt.n) {
              const __nv_bfloat16 hb = __float2bfloat16_rn(sv * uv);
              hbuf[(size_t)(pt.row0 + c) * a.I + ii] = *reinterpret_cast<const uint16_t*>(&hb);
            }
          }
        } else {
          const float Gd = a.globals[pt.expert * 4 + 2];
          float* y = ws_at<float>(a, a.W.y);
          const int jrow = pt.mt * BM + r;
          const int q_per_tok = a.S + a.k;
          const int ctok_h = hcol ? pctok[1] : pctok[0], cq_h = hcol ? pcq[1] : pcq[0];
          const float cw_h = hcol ? pcw[1] : pcw[0];
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int c = c0 + j, src = c & 31;
            const int tok = __shfl_sync(0xffffffffu, ctok_h, src);
            const int qq = __shfl_sync(0xffffffffu, cq_h, src);
            const float wv = __shfl_sync(0xffffffffu, cw_h, src);
            if (c < pt.n) y[((size_t)tok * q_per_tok + qq) * a.H + jrow] = wv * (__uint_as_float(v[j]) * Gd);
          }
        }
        pc = c0 + 16;
      }
      if (!(pc < cg * 64 + 64 && pc < pt.n)) {  // the warp's columns are done: the buffer is free for it
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&G.acc_empty[p][ab]);
        pend = false;
      }
      return true;
    };
    bool failed = false;
    for (int u = 0; u < n_slots && !failed; ++u) {
      const int i = u / SPT, kb0 = (u % SPT) * RAW_KB, nk = min(RAW_KB, KB - kb0);
      if (kb0 == 0) {
        t = nxt;
        if (i + 1 < my_tiles) nxt = tile_info<MODE>(a, tile_of(i + 1));
#pragma unroll
        for (int hcol = 0; hcol < 2; ++hcol) {
          const int c = cg * 64 + hcol * 32 + lane;
          if (MODE == GATEUP && c < t.n) {  // 2^-kx of its token
            const int tok = t.slot < a.S ? t.row0 - t.slot * a.B + c : __ldcg(ws_at<const int>(a, a.W.list_tok) + t.row0 + c);
            cinv[hcol] = exp2i(-__ldcg(ws_at<const int>(a, a.W.kx) + tok));
          }
          if (MODE == DOWN && c < t.n) {
            const int row = t.row0 + c;
            ctok[hcol] = __ldcg(ws_at<const int>(a, a.W.list_tok) + row);
            cq[hcol] = __ldcg(ws_at<const int>(a, a.W.list_q) + row);
            cw[hcol] = __ldcg(ws_at<const float>(a, a.W.list_w) + row);
          }
        }
      }
      if (MODE != ROUTER) {
        const uint8_t* slot_p = raw + (u % RAW_SL) * RAW_SLOT + tile_off;
        bool ok = wait_ab(&G.raw_full[p][u % RAW_SL], (u / RAW_SL) & 1, abort, status);
        for (int j = 0; j < nk; ++j) {
          const int g = i * KB + kb0 + j, s = g % STAGES;
          ok = ok && (g < STAGES || wait_ab(&G.mma_done[p][s], ((g / STAGES) - 1) & 1, abort, status));
          if (!__all_sync(0xffffffffu, ok)) {
            failed = true;
            break;
          }
          const uint8_t* kp = slot_p + j * KG_NVFP4;
          const uint4 codes = lds128(kp + lane * 16);
          const uint32_t sg = lds32(kp + KG_CODE_BYTES + dq_g * 4);
          const uint32_t sg8 = lds32(kp + KG_CODE_BYTES + (dq_g + 8) * 4);
          const uint32_t cw4[4] = {codes.x, codes.y, codes.z, codes.w};
          const uint32_t ap = a_op + s * A_STAGE;
#pragma unroll
          for (int ks = 0; ks < 4; ++ks) {
            uint32_t af[4];
            nvfp4_afrag(cw4[ks], sg, sg8, ks, af);
            if (MODE != GATEUP) {
#pragma unroll
              for (int q = 0; q < 4; ++q) af[q] = f16x2_to_bf16x2(af[q]);
            }
            asm volatile("stmatrix.sync.aligned.m8n8.x4.shared.b16 [%0], {%1, %2, %3, %4};" ::"r"(ap + soff[ks]),
                         "r"(af[0]), "r"(af[1]), "r"(af[2]), "r"(af[3])
                         : "memory");
          }
          fence_proxy_async();  // these st.shared -> visible to the tensor core
          __syncwarp();
          if (lane == 0) mbar_arrive(&G.full[p][s]);
          if (pend && !epi_chunk()) {
            failed = true;
            break;
          }
        }
        if (failed || !__all_sync(0xffffffffu, ok)) {
          failed = true;
          break;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&G.raw_empty[p][u % RAW_SL]);  // this warp is done with the slot
      }
      if (kb0 + nk == KB) {  // all k-blocks of the tile are dequantised: its epilogue is next
        while (pend && !failed) failed = !epi_chunk();
        if (failed) break;
        pend = true;
        pt = t;
        pi = i;
        pc = cg * 64;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          pctok[h] = ctok[h];
          pcq[h] = cq[h];
          pcw[h] = cw[h];
          pcinv[h] = cinv[h];
        }
        if (MODE == ROUTER)  // no dequantisation to interleave with: now
          while (pend && !failed) failed = !epi_chunk();
      }
    }
    while (pend && !failed) failed = !epi_chunk();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(G.tmem_base), "r"(TMEM_COLS) : "memory");
  }
}

// ---------------------------------------------------------------------------
// Small tiles: a slot with few grouped rows (a routed expert that few tokens
// chose) gives the tensor-core tiles little to multiply per dequantised weight,
// so its tiles of up to SN tokens go through registers instead: each of the 8
// warps of a block takes one packed tile (16 weight rows) of the tile's m-tile,
// streams its k-groups from global memory, dequantises each k-step into the
// mma.sync A fragment (the layout the packed bytes are stored in) and
// multiplies it with the tile's token rows, which the block stages in shared
// memory (row pitch K + 8 elements, so the 8 rows an ldmatrix reads fall in
// distinct banks; rows n..SN-1 are zero). Same epilogues, arithmetic and
// rounding points as k_pf_gemm; only the FP32 summation order of the products
// differs. Persistent over the small tiles blockIdx.x, + gridDim.x, ...
// ---------------------------------------------------------------------------
constexpr int SMALL_THREADS = 256;
constexpr int SMALL_PF = 4;  // k-groups of packed weights loaded ahead per warp

__host__ __device__ constexpr size_t small_smem_bytes(int K) { return (size_t)SN * (K * 2 + 16); }

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

__device__ __forceinline__ uint4 ldg_stream_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}
__device__ __forceinline__ uint32_t ldg_stream_u32(const void* p) {
  uint32_t v;
  asm volatile("ld.global.nc.L1::no_allocate.u32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}

// NKG > 0: the k-groups per packed tile (K / 64) fixed at compile time (the
// Flint shape: 32 for gate/up, 8 for down); 0: read from the arguments.
template <int MODE, int NKG>
__global__ void __launch_bounds__(SMALL_THREADS, 3) k_pf_small(const PfArgs a) {
  extern __shared__ __align__(16) uint8_t srows[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, tq = lane & 3;
  const int K = NKG ? NKG * 64 : (MODE == DOWN ? a.I : a.H);
  const int pitch = K * 2 + 16, nkg = K / 64, cpr = K / 8;
  const int n_tiles = __ldcg(ws_at<int>(a, 0) + (MODE == GATEUP ? PF_NGUS : PF_NDNS));
  const int4* tiles = ws_at<const int4>(a, MODE == GATEUP ? a.W.gus_tiles : a.W.dns_tiles);
  const int64_t wtile = MODE == GATEUP ? a.L.gu_tile : a.L.dn_tile;
  const uint32_t sbase = smem_addr(srows);
  // ldmatrix.x4 rows of this lane: matrix lane / 8 = (token half, k half) of a k-step
  const uint32_t bl = sbase + (uint32_t)(((lane >> 4) * 8 + (lane & 7)) * pitch + ((lane >> 3) & 1) * 16);
  for (int tile = blockIdx.x; tile < n_tiles; tile += gridDim.x) {
    const int4 tv = __ldcg(tiles + tile);
    const int slot = tv.x, mt = tv.y, row0 = tv.z, n = tv.w;
    const int expert = __ldcg(ws_at<const int>(a, a.W.slot_expert) + slot);
    const uint16_t* src;
    if (MODE == GATEUP)  // a shared expert's rows are the tokens in order; the routed pairs' are grouped
      src = slot < a.S ? ws_at<const uint16_t>(a, a.W.x16) + (size_t)(row0 - slot * a.B) * K
                       : ws_at<const uint16_t>(a, a.W.xg) + (size_t)(row0 - a.S * a.B) * K;
    else
      src = ws_at<const uint16_t>(a, a.W.h) + (size_t)row0 * K;
    __syncthreads();  // the previous tile's rows are no longer read
#pragma unroll 4
    for (int r = 0; r < SN; ++r)
      for (int c = threadIdx.x; c < cpr; c += SMALL_THREADS)
        cp_async16(sbase + (uint32_t)(r * pitch + c * 16), src + (size_t)(r < n ? r : 0) * K + c * 8, r < n ? 16u : 0u);
    cp_async_commit();
    // Packed tile (8 mt + warp) of the expert's gate/up or down matrix.
    const uint8_t* wp = a.packed + (int64_t)expert * a.L.expert_bytes + (MODE == GATEUP ? 0 : a.L.gu_bytes) +
                        (int64_t)(mt * 8 + warp) * wtile;
    uint4 cw[SMALL_PF];
    uint32_t sg[SMALL_PF], sg8[SMALL_PF];
#pragma unroll
    for (int j = 0; j < SMALL_PF; ++j)
      if (j < nkg) {
        const uint8_t* kp = wp + j * KG_NVFP4;
        cw[j] = ldg_stream_v4(kp + lane * 16);
        sg[j] = ldg_stream_u32(kp + KG_CODE_BYTES + g * 4);
        sg8[j] = ldg_stream_u32(kp + KG_CODE_BYTES + (g + 8) * 4);
      }
    cp_async_wait<0>();
    __syncthreads();
    float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    // k-group kg0 + j sits in register set j; once multiplied, the set takes
    // k-group kg0 + j + SMALL_PF, so SMALL_PF k-groups stay in flight.
    for (int kg0 = 0; kg0 < nkg; kg0 += SMALL_PF) {
#pragma unroll
      for (int j = 0; j < SMALL_PF; ++j) {
        if (kg0 + j < nkg) {
          const uint32_t w4[4] = {cw[j].x, cw[j].y, cw[j].z, cw[j].w};
#pragma unroll
          for (int ks = 0; ks < 4; ++ks) {
            uint32_t af[4];
            nvfp4_afrag(w4[ks], sg[j], sg8[j], ks, af);
            uint32_t b[4];
            ldsm_x4(bl + (uint32_t)(((kg0 + j) * 64 + ks * 16) * 2), b);
            if (MODE == GATEUP) {
              mma_f16(acc[0], af, b[0], b[1]);
              mma_f16(acc[1], af, b[2], b[3]);
            } else {
#pragma unroll
              for (int q = 0; q < 4; ++q) af[q] = f16x2_to_bf16x2(af[q]);
              mma_bf16(acc[0], af, b[0], b[1]);
              mma_bf16(acc[1], af, b[2], b[3]);
            }
          }
        }
        if (kg0 + SMALL_PF + j < nkg) {
          const uint8_t* kp = wp + (kg0 + SMALL_PF + j) * KG_NVFP4;
          cw[j] = ldg_stream_v4(kp + lane * 16);
          sg[j] = ldg_stream_u32(kp + KG_CODE_BYTES + g * 4);
          sg8[j] = ldg_stream_u32(kp + KG_CODE_BYTES + (g + 8) * 4);
        }
      }
    }
    // Epilogue: lane (g, tq) holds rows g, g + 8 of the packed tile for token
    // columns 8 jn + 2 tq + {0, 1}.
    if (MODE == GATEUP) {
      // rows g and g + 8 are the gate and up rows of intermediate index 8 (8 mt + warp) + g
      const float Gg = a.globals[expert * 4 + 0], Gu = a.globals[expert * 4 + 1];
      const int ii = (mt * 8 + warp) * 8 + g;
      uint16_t* hbuf = ws_at<uint16_t>(a, a.W.h);
#pragma unroll
      for (int jn = 0; jn < 2; ++jn)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int c = jn * 8 + tq * 2 + e;
          if (c < n) {
            const int tok = slot < a.S ? row0 - slot * a.B + c : __ldcg(ws_at<const int>(a, a.W.list_tok) + row0 + c);
            const float inv = exp2i(-__ldcg(ws_at<const int>(a, a.W.kx) + tok));
            const float gv = acc[jn][e] * inv * Gg;
            const float uv = acc[jn][2 + e] * inv * Gu;
            const float sv = __fdividef(gv, 1.0f + __expf(-gv));
            const __nv_bfloat16 hb = __float2bfloat16_rn(sv * uv);
            hbuf[(size_t)(row0 + c) * a.I + ii] = *reinterpret_cast<const uint16_t*>(&hb);
          }
        }
    } else {
      const float Gd = a.globals[expert * 4 + 2];
      float* y = ws_at<float>(a, a.W.y);
      const int jrow = mt * BM + warp * 16 + g;
      const int q_per_tok = a.S + a.k;
#pragma unroll
      for (int jn = 0; jn < 2; ++jn)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int c = jn * 8 + tq * 2 + e;
          if (c < n) {
            const int row = row0 + c;
            const int tok = __ldcg(ws_at<const int>(a, a.W.list_tok) + row);
            const int qq = __ldcg(ws_at<const int>(a, a.W.list_q) + row);
            const float wv = __ldcg(ws_at<const float>(a, a.W.list_w) + row);
            float* yr = y + ((size_t)tok * q_per_tok + qq) * a.H + jrow;
            yr[0] = wv * (acc[jn][e] * Gd);
            yr[8] = wv * (acc[jn][2 + e] * Gd);
          }
        }
    }
  }
}

// One warp per token, after the plan: the token's entries of the grouped row
// lists (token, slot rank, routing weight), and its gate/up activations in
// f16 for the tensor cores: a power of two 2^kx maps the row's largest |x|
// into [2^14, 2^15), so every bf16 value is exact in f16 (down to 2^-24 of
// that bound, below which the tail flushes; the epilogue multiplies by
// 2^-kx). The row goes to x16 and to the grouped rows of its k routed pairs.
__global__ void __launch_bounds__(256) k_pf_token_rows(PfArgs a) {
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (t >= a.B) return;
  const uint4* src = reinterpret_cast<const uint4*>(a.x + (size_t)t * a.H);
  const int nw = a.H / 8;
  // Lane q < S + k: list row q of the token (its S shared rows s B + t, then
  // its k routed rows rowbase[e_j] + pos_j, the token's place in e_j's list).
  int row = 0;
  if (lane < a.S + a.k) {
    float w = 1.0f;
    if (lane < a.S) {
      row = lane * a.B + t;
    } else {
      const size_t p = (size_t)t * a.k + (lane - a.S);
      const int e = __ldcg(ws_at<const int>(a, a.W.idx) + p);
      row = __ldcg(ws_at<const int>(a, a.W.rowbase) + e) + __ldcg(ws_at<const int>(a, a.W.pos) + p);
      w = __ldcg(ws_at<const float>(a, a.W.w) + p);
    }
    ws_at<int>(a, a.W.list_tok)[row] = t;
    ws_at<int>(a, a.W.list_q)[row] = lane;
    ws_at<float>(a, a.W.list_w)[row] = w;
  }
  float m = 0.f;
#pragma unroll 4
  for (int i = lane; i < nw; i += 32) {
    const uint4 v = __ldg(src + i);
    const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) m = fmaxf(m, fmaxf(fabsf(bf16lo(w4[j])), fabsf(bf16hi(w4[j]))));
  }
  const int kx = prescale_exp(warp_max(m));
  const float sc = exp2i(kx);
  if (lane == 0) ws_at<int>(a, a.W.kx)[t] = kx;
  uint4* x16 = ws_at<uint4>(a, a.W.x16) + (size_t)t * nw;
  uint4* xg = ws_at<uint4>(a, a.W.xg);
  for (int i = lane; i < nw; i += 32) {
    const uint4 v = __ldg(src + i);
    uint4 o;
    o.x = bf16x2_to_f16x2_scaled(v.x, sc);
    o.y = bf16x2_to_f16x2_scaled(v.y, sc);
    o.z = bf16x2_to_f16x2_scaled(v.z, sc);
    o.w = bf16x2_to_f16x2_scaled(v.w, sc);
    x16[i] = o;
    for (int j = 0; j < a.k; ++j) {  // grouped routed row (activation copy)
      const int r = __shfl_sync(0xffffffffu, row, a.S + j) - a.S * a.B;
      xg[(size_t)r * nw + i] = o;
    }
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

template <int PER>
__global__ void __launch_bounds__(256) k_pf_topk(PfArgs a) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * 8 + warp;
  if (t >= a.B) return;
  float* logits = ws_at<float>(a, a.W.logits) + (size_t)t * a.E;
  const float* part = ws_at<const float>(a, a.W.y) + (size_t)t * a.E;  // split partials (rsplit > 1)
  const size_t plane = (size_t)a.B * a.E;
  float s[PER];
  uint32_t key[PER];
  uint32_t taken = 0;
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    const int e = lane + 32 * i;
    s[i] = 0.f;
    key[i] = 0u;
    if (e < a.E) {
      float l;
      if (a.rsplit > 1) {  // the splits' partial sums, all loaded at once, added in split order
        float pq[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) pq[q] = q < a.rsplit ? __ldcg(part + q * plane + e) : 0.f;
        l = pq[0];
#pragma unroll
        for (int q = 1; q < 8; ++q)
          if (q < a.rsplit) l += pq[q];
        logits[e] = l;
      } else {
        l = __ldcg(logits + e);
      }
      s[i] = 1.0f / (1.0f + expf(-l));
      key[i] = order_f32(s[i] + (a.bias ? __ldg(a.bias + e) : 0.f));
    } else {
      taken |= 1u << i;
    }
  }
  // k rounds of a warp arg-max; every lane ends with every rank's expert and sigmoid.
  int sel_e[MAX_TOPK];
  float sel_s[MAX_TOPK];
#pragma unroll
  for (int j = 0; j < MAX_TOPK; ++j) {
    sel_e[j] = 0;
    sel_s[j] = 0.f;
    if (j < a.k) {
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
  }
  // Lane j finishes rank j: the same sum in rank order on every lane.
  float sum = 0.f;
#pragma unroll
  for (int j = 0; j < MAX_TOPK; ++j)
    if (j < a.k) sum += sel_s[j];
  if (lane < a.k) {
    int ej = 0;
    float sj = 0.f;
#pragma unroll
    for (int j = 0; j < MAX_TOPK; ++j)
      if (j == lane) {
        ej = sel_e[j];
        sj = sel_s[j];
      }
    const size_t p = (size_t)t * a.k + lane;
    const float wj = a.renorm ? sj / sum : sj;
    ws_at<int>(a, a.W.idx)[p] = ej;
    ws_at<float>(a, a.W.w)[p] = wj * a.routed_scale;
    ws_at<int>(a, a.W.pos)[p] = atomicAdd(ws_at<int>(a, a.W.counts) + ej, 1);
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
  __shared__ int s_slot_cnt[PLAN_THREADS], s_slot_row0[PLAN_THREADS], s_slot_tb[PLAN_THREADS],
      s_slot_tbs[PLAN_THREADS];
  __shared__ int s_nslots, s_ntiles, s_nstiles;
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
  // Token tiles per slot (one slot per thread: S + E <= PLAN_THREADS): NT-token
  // tiles for the tensor cores, or SN-token tiles for slots of few rows.
  const int s = threadIdx.x;
  const int cnt = s < nslots ? s_slot_cnt[s] : 0;
  const bool small = cnt <= (s < a.S ? a.small_shared : a.small_max);
  const int ntl = small ? 0 : (cnt + NT - 1) / NT;
  const int nts = small ? (cnt + SN - 1) / SN : 0;
  const int tb = block_exclusive_scan(ntl, sh);
  const int tbs = block_exclusive_scan(nts, sh);
  if (s == PLAN_THREADS - 1) {
    s_ntiles = tb + ntl;
    s_nstiles = tbs + nts;
  }
  const int mgu = 2 * a.I / BM, mdn = a.H / BM;
  if (s < nslots) {
    s_slot_tb[s] = tb;
    s_slot_tbs[s] = tbs;
    ws_at<int>(a, a.W.slot_row0)[s] = s_slot_row0[s];
    ws_at<int>(a, a.W.slot_count)[s] = cnt;
  }
  __syncthreads();
  // Tile lists, spread over the block: entry i of the token tiles x (gate/up
  // m-tiles + down m-tiles). A token tile's slot is the last one whose first
  // tile is <= it: the first tiles are non-decreasing in slot order, and a slot
  // without tiles of the kind shares its first tile with the next slot that has some.
  auto slot_of = [&](const int* first, int tile) {
    int lo = 0, hi = nslots - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (first[mid] <= tile) lo = mid; else hi = mid - 1;
    }
    return lo;
  };
  const int per = mgu + mdn;
  for (int kind = 0; kind < 2; ++kind) {
    const int* first = kind ? s_slot_tbs : s_slot_tb;
    const int tsz = kind ? SN : NT;
    int4* gu = ws_at<int4>(a, kind ? a.W.gus_tiles : a.W.gu_tiles);
    int4* dn = ws_at<int4>(a, kind ? a.W.dns_tiles : a.W.dn_tiles);
    const int n_ent = (kind ? s_nstiles : s_ntiles) * per;
    for (int i = threadIdx.x; i < n_ent; i += PLAN_THREADS) {
      const int tile = i / per, m = i % per;
      const int sl = slot_of(first, tile);
      const int q = tile - first[sl], row0 = s_slot_row0[sl] + q * tsz;
      const int n = min(tsz, s_slot_cnt[sl] - q * tsz);
      if (m < mgu) gu[(size_t)tile * mgu + m] = make_int4(sl, m, row0, n);
      else dn[(size_t)tile * mdn + (m - mgu)] = make_int4(sl, m - mgu, row0, n);
    }
  }
  if (threadIdx.x == 0) {
    int* hdr = ws_at<int>(a, 0);
    hdr[PF_NSLOTS] = nslots;
    hdr[PF_NGU] = s_ntiles * mgu;
    hdr[PF_NDN] = s_ntiles * mdn;
    hdr[PF_NGUS] = s_nstiles * mgu;
    hdr[PF_NDNS] = s_nstiles * mdn;
  }
  if (e < a.E) ws_at<int>(a, a.W.rowbase)[e] = s_rowbase[e];
  if (e < a.E) counts[e] = 0;  // ready for the next call (every read of counts is above)
}

// Pre-norm block: xn = bf16(r * gamma / sqrt(mean(r^2) + eps)), one warp per
// token, with the same lane order and arithmetic as the decode kernels.
__global__ void __launch_bounds__(256) k_pf_norm(PfArgs a) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * 8 + warp;
  if (t >= a.B) return;
  const uint4* r = reinterpret_cast<const uint4*>(a.res + (size_t)t * a.H);
  const uint4* w = reinterpret_cast<const uint4*>(a.gamma);
  uint4* xn = ws_at<uint4>(a, a.W.xn) + (size_t)t * (a.H / 8);
  const int nch = a.H / 256;  // 16-byte chunks per lane
  float part = 0.f;
  for (int c = 0; c < nch; ++c) part = sumsq8(__ldg(r + lane + 32 * c), part);
  const float ss = warp_sum(part);
  if (ss <= FP32_MAX) {
    const float inv = 1.0f / sqrtf(ss / (float)a.H + a.eps);
    for (int c = 0; c < nch; ++c) xn[lane + 32 * c] = norm8(__ldg(r + lane + 32 * c), __ldg(w + lane + 32 * c), inv);
  } else {  // the sum of squares overflowed: the scaled path
    const float2 f = rms_factor_huge(reinterpret_cast<const uint8_t*>(r), 0, lane, a.H, a.eps);
    for (int c = 0; c < nch; ++c)
      xn[lane + 32 * c] = norm8_huge(__ldg(r + lane + 32 * c), __ldg(w + lane + 32 * c), f);
  }
}

// out[t][j] = bf16(sum over q of y[t][q][j]), q = shared experts, then top-k ranks;
// for the pre-norm block out = bf16(r + that).
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
    __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y), hi = __floats2bfloat162_rn(acc.z, acc.w);
    if (a.prenorm) {  // residual stream: r + bf16(layer output), rounded to bf16
      const uint2 rv = *reinterpret_cast<const uint2*>(a.res + t * a.H + j4 * 4);
      lo = __floats2bfloat162_rn(bf16lo(rv.x) + __low2float(lo), bf16hi(rv.x) + __high2float(lo));
      hi = __floats2bfloat162_rn(bf16lo(rv.y) + __low2float(hi), bf16hi(rv.y) + __high2float(hi));
    }
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
template <int MODE, int NKG>
static cudaError_t launch_small_k(const PfArgs& a, int grid, cudaStream_t stream) {
  static std::atomic<int> attr_set{0};
  const size_t smem = small_smem_bytes(MODE == DOWN ? a.I : a.H);
  if (smem > 48 * 1024 && !attr_set.load()) {
    cudaError_t e = cudaFuncSetAttribute(k_pf_small<MODE, NKG>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    attr_set.store(1);
  }
  k_pf_small<MODE, NKG><<<grid, SMALL_THREADS, smem, stream>>>(a);
  return cudaGetLastError();
}

template <int MODE>
static cudaError_t launch_small(const PfArgs& a, int grid, cudaStream_t stream) {
  const int K = MODE == DOWN ? a.I : a.H;
  constexpr int FLINT_K = MODE == DOWN ? 512 : 2048;  // the Flint shape's I and H
  return K == FLINT_K ? launch_small_k<MODE, FLINT_K / 64>(a, grid, stream) : launch_small_k<MODE, 0>(a, grid, stream);
}

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

// cuTensorMapEncodeTiled, reached through the runtime (no link against the driver library).
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn tensor_map_encoder() {
  static std::atomic<void*> fn{nullptr};
  void* f = fn.load();
  if (!f) {
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !f)
      return nullptr;
    fn.store(f);
  }
  return reinterpret_cast<EncodeTiledFn>(f);
}

// bf16 matrix [rows][cols] (row stride cols * 2 bytes), boxes of 64 columns x
// 128 rows written in the 128-byte swizzle; rows past the end read as zero.
static bool encode_rows(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows, bool f16 = false) {
  const EncodeTiledFn enc = tensor_map_encoder();
  if (!enc || rows == 0) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * 2};
  const cuuint32_t box[2] = {(cuuint32_t)BK, (cuuint32_t)NT};
  const cuuint32_t estr[2] = {1, 1};
  return enc(m, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int MODE>
static cudaError_t launch_gemm(const PfArgs& a, const PfMaps& maps, int grid, cudaStream_t stream) {
  static std::atomic<int> attr_set{0};
  const size_t smem = gemm_dyn_smem();
  if (!attr_set.load()) {
    cudaError_t e = cudaFuncSetAttribute(k_pf_gemm<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    attr_set.store(1);
  }
  k_pf_gemm<MODE><<<grid, GEMM_THREADS, smem, stream>>>(a, maps);
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

static flint_moe_status prefill_impl(const flint_moe_layer* layer, const uint16_t* x, int32_t B, uint16_t* out,
                                     void* ws, size_t ws_bytes, cudaStream_t stream, bool prenorm) {
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
  // the pre-norm block may update the residual stream in place; otherwise x and out are disjoint
  if (xa < oa + xb && oa < xa + xb && !(prenorm && xa == oa)) return FLINT_MOE_EINVAL;
  if (prenorm && (!layer->norm_weight || (uintptr_t)layer->norm_weight % 16)) return FLINT_MOE_EINVAL;
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
  a.prenorm = prenorm ? 1 : 0;
  a.res = x;
  a.gamma = layer->norm_weight;
  a.eps = layer->norm_eps;
  // Small tiles while three blocks' token rows fit one SM's shared memory, for
  // calls of up to SMALL_B_MAX tokens: beyond, most routed experts have more
  // than SMALL_MAX tokens, and the few small tiles would only add a launch
  // after the tensor-core tiles.
  const bool small_fits = 3 * small_smem_bytes(a.H) <= (size_t)227 * 1024 && B <= SMALL_B_MAX;
  a.small_max = small_fits ? SMALL_MAX : 0;
  a.small_shared = small_fits ? SMALL_SHARED_MAX : 0;
  if (ws_bytes < a.W.total) return FLINT_MOE_EINVAL;
  if (prenorm) {  // the layer runs on the normalised rows
    k_pf_norm<<<(B + 7) / 8, 256, 0, stream>>>(a);
    if (cudaGetLastError() != cudaSuccess) return FLINT_MOE_ECUDA;
    a.x = reinterpret_cast<const uint16_t*>(static_cast<uint8_t*>(ws) + a.W.xn);
  }

  // TMA descriptors of the three GEMMs (host-side encoding, passed by value).
  PfMaps m_router, m_gateup, m_down;
  uint8_t* wsb = static_cast<uint8_t*>(ws);
  if (!encode_rows(&m_router.a, a.router, a.H, a.E) || !encode_rows(&m_router.b0, a.x, a.H, B) ||
      !encode_rows(&m_gateup.b0, wsb + a.W.x16, a.H, B, true) ||
      !encode_rows(&m_gateup.b1, wsb + a.W.xg, a.H, (uint64_t)B * a.k, true) ||
      !encode_rows(&m_down.b0, wsb + a.W.h, a.I, (uint64_t)a.W.max_rows))
    return FLINT_MOE_ECUDA;
  m_router.b1 = m_router.b0;
  m_gateup.a = m_gateup.b0;
  m_down.a = m_down.b1 = m_down.b0;

  const int nsm = sm_count();
  const int router_tiles = ((a.E + BM - 1) / BM) * ((B + NT - 1) / NT);
  // Few router tiles (up to a few hundred tokens) leave most SMs idle and each
  // tile's k-loop latency-bound: split H so that the tiles fill the SMs, while
  // every split keeps at least STAGES k-blocks and the partials fit in y.
  a.rsplit = 1;
  while (a.rsplit < 8 && router_tiles * a.rsplit * 2 <= nsm && (a.H / BK) % (a.rsplit * 2) == 0 &&
         a.H / BK / (a.rsplit * 2) >= STAGES && (size_t)a.rsplit * 2 * a.E <= (size_t)(a.S + a.k) * a.H)
    a.rsplit *= 2;
  if (launch_gemm<ROUTER>(a, m_router, std::min(nsm, router_tiles * a.rsplit), stream) != cudaSuccess)
    return FLINT_MOE_ECUDA;
  if (a.E <= 256)  // experts per lane: 8 (up to 256 experts) or 16
    k_pf_topk<8><<<(B + 7) / 8, 256, 0, stream>>>(a);
  else
    k_pf_topk<MAX_E / 32><<<(B + 7) / 8, 256, 0, stream>>>(a);
  if (cudaGetLastError() != cudaSuccess) return FLINT_MOE_ECUDA;
  k_pf_plan<<<1, PLAN_THREADS, 0, stream>>>(a);
  if (cudaGetLastError() != cudaSuccess) return FLINT_MOE_ECUDA;
  k_pf_token_rows<<<(B + 7) / 8, 256, 0, stream>>>(a);
  if (cudaGetLastError() != cudaSuccess) return FLINT_MOE_ECUDA;
  if (launch_gemm<GATEUP>(a, m_gateup, std::min(nsm, a.W.max_gu), stream) != cudaSuccess) return FLINT_MOE_ECUDA;
  if (small_fits && launch_small<GATEUP>(a, std::min(3 * nsm, a.W.max_gus), stream) != cudaSuccess)
    return FLINT_MOE_ECUDA;
  if (launch_gemm<DOWN>(a, m_down, std::min(nsm, a.W.max_dn), stream) != cudaSuccess) return FLINT_MOE_ECUDA;
  if (small_fits && launch_small<DOWN>(a, std::min(3 * nsm, a.W.max_dns), stream) != cudaSuccess)
    return FLINT_MOE_ECUDA;
  const int cgrid = (int)std::min<size_t>((size_t)nsm * 8, ((size_t)B * a.H / 4 + 255) / 256);
  k_pf_combine<<<cgrid, 256, 0, stream>>>(a);
  if (cudaGetLastError() != cudaSuccess) return FLINT_MOE_ECUDA;
  return FLINT_MOE_OK;
}

extern "C" flint_moe_status flint_moe_prefill(const flint_moe_layer* layer, const uint16_t* x, int32_t B,
                                              uint16_t* out, void* ws, size_t ws_bytes, cudaStream_t stream) {
  return prefill_impl(layer, x, B, out, ws, ws_bytes, stream, false);
}

extern "C" flint_moe_status flint_moe_prefill_prenorm(const flint_moe_layer* layer, const uint16_t* residual_in,
                                                      int32_t B, uint16_t* residual_out, void* ws, size_t ws_bytes,
                                                      cudaStream_t stream) {
  return prefill_impl(layer, residual_in, B, residual_out, ws, ws_bytes, stream, true);
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
