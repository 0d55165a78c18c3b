// Load-time side of the library: configuration checks, the lossless repack
// into the GB300 layout (and its inverse), the NVFP4 quantiser and the
// dequantisation read-back used to check the decode kernels' dequantiser.
//
// "Day-0 Support for Flint on vLLM", section "Model architecture": the NVFP4
// checkpoint holds NVIDIA's NVFP4 blocks in another byte order and is repacked
// losslessly at load. Here the source is a canonical row-major layout and the
// target is the tensor-core fragment order documented in common.cuh.
#include <cuda_fp8.h>

#include "common.cuh"
#include "flint_gemv.h"

namespace flint {

// Where a packed 32-bit word comes from. For an NVFP4 code word the four bytes
// come from four canonical bytes (src_idx[0..3]); for scale and BF16 words the
// four bytes are one aligned canonical word (src_idx[0], whole = true).
struct WordSrc {
  int mat;          // 0 gate, 1 up, 2 down (of byte 0; a code word mixes gate and up rows)
  int mat_b[4];     // matrix of each byte of a code word
  int64_t expert;
  bool is_scale;
  bool whole;
  int64_t idx[4];   // byte offsets into the canonical array of `mat` (per expert)
};

__host__ __device__ inline void map_word(const Layout& L, int H, int I, int fmt, int64_t w, WordSrc& s) {
  const int64_t byte = w * 4;
  s.expert = byte / L.expert_bytes;
  int64_t o = byte - s.expert * L.expert_bytes;
  int row_base, mat_lo, mat_hi, cols;
  int64_t tile_bytes;
  if (o < L.gu_bytes) {
    tile_bytes = L.gu_tile;
    const int64_t tile = o / tile_bytes;
    o -= tile * tile_bytes;
    row_base = (int)tile * 8;
    mat_lo = 0;
    mat_hi = 1;
    cols = H;
  } else {
    o -= L.gu_bytes;
    tile_bytes = L.dn_tile;
    const int64_t tile = o / tile_bytes;
    o -= tile * tile_bytes;
    row_base = (int)tile * 16;
    mat_lo = 2;
    mat_hi = 2;
    cols = I;
  }
  const int kg = (int)(o / L.kg_bytes);
  const int q = (int)(o - (int64_t)kg * L.kg_bytes);  // byte within the k-group, multiple of 4
  auto row_of = [&](int r, int& mat) -> int {
    if (mat_lo != mat_hi) {  // gate/up tile: rows 0..7 gate, 8..15 up
      mat = r < 8 ? mat_lo : mat_hi;
      return row_base + (r & 7);
    }
    mat = mat_lo;
    return row_base + r;
  };
  if (fmt == FLINT_MOE_NVFP4) {
    if (q < KG_CODE_BYTES) {
      const int lane = q >> 4, ks = (q >> 2) & 3, g = lane >> 2, t = lane & 3;
      s.is_scale = false;
      s.whole = false;
      for (int b = 0; b < 4; ++b) {
        const int r = g + 8 * (b & 1);  // b & 1 selects row g + 8: the up row in a gate/up tile
        const int c = kg * KG_COLS + ks * 16 + 2 * t + 8 * (b >> 1);
        int mat;
        const int row = row_of(r, mat);
        s.mat_b[b] = mat;
        s.idx[b] = (int64_t)row * (cols / 2) + c / 2;
      }
    } else {
      const int r = (q - KG_CODE_BYTES) >> 2;  // 4 scale bytes per row: blocks kg*4 .. kg*4+3
      int mat;
      const int row = row_of(r, mat);
      s.mat = mat;
      s.is_scale = true;
      s.whole = true;
      s.idx[0] = (int64_t)row * (cols / 16) + kg * 4;
    }
  } else {
    const int lane = q >> 6, ks = (q >> 4) & 3, reg = (q >> 2) & 3, g = lane >> 2, t = lane & 3;
    const int r = g + 8 * (reg & 1);
    const int c = kg * KG_COLS + ks * 16 + 2 * t + 8 * (reg >> 1);
    int mat;
    const int row = row_of(r, mat);
    s.mat = mat;
    s.is_scale = false;
    s.whole = true;
    s.idx[0] = ((int64_t)row * cols + c) * 2;  // byte offset into the bf16 matrix
  }
}

struct PackArgs {
  Layout L;
  int H, I, fmt;
  int64_t n_words;  // words of expert data
  const uint8_t* codes[3];
  const uint8_t* scales[3];
  const uint8_t* bf16[3];
  int64_t codes_per_expert[3], scales_per_expert[3], bf16_per_expert[3];
  uint8_t* dst;
  int* status;
};

__global__ void k_pack(PackArgs a) {
  for (int64_t w = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; w < a.n_words;
       w += (int64_t)gridDim.x * blockDim.x) {
    WordSrc s;
    map_word(a.L, a.H, a.I, a.fmt, w, s);
    uint32_t v;
    if (a.fmt == FLINT_MOE_NVFP4) {
      if (s.is_scale) {
        const uint8_t* p = a.scales[s.mat] + s.expert * a.scales_per_expert[s.mat] + s.idx[0];
        v = (uint32_t)p[0] | ((uint32_t)p[1] << 8) | ((uint32_t)p[2] << 16) | ((uint32_t)p[3] << 24);
        bool nan = false;
        for (int b = 0; b < 4; ++b) nan |= ((v >> (8 * b)) & 0x7F) == 0x7F;
        if (nan && a.status) atomicOr(a.status, FLINT_MOE_DEV_ERR_NAN_SCALE);
      } else {
        v = 0;
        for (int b = 0; b < 4; ++b) {
          const int m = s.mat_b[b];
          v |= (uint32_t)a.codes[m][s.expert * a.codes_per_expert[m] + s.idx[b]] << (8 * b);
        }
      }
    } else {
      const uint8_t* p = a.bf16[s.mat] + s.expert * a.bf16_per_expert[s.mat] + s.idx[0];
      v = *reinterpret_cast<const uint32_t*>(p);
    }
    reinterpret_cast<uint32_t*>(a.dst)[w] = v;
  }
}

struct GlobalsArgs {
  const float* g[3];
  float* dst;
  int n;
  int fmt;
};

__global__ void k_pack_globals(GlobalsArgs a) {
  const int e = blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= a.n) return;
  for (int m = 0; m < 3; ++m) a.dst[e * 4 + m] = a.fmt == FLINT_MOE_NVFP4 ? a.g[m][e] : 1.0f;
  a.dst[e * 4 + 3] = 0.f;
}

struct UnpackArgs {
  Layout L;
  int H, I, fmt;
  int64_t n_words;
  const uint8_t* src;
  uint8_t* codes[3];
  uint8_t* scales[3];
  uint8_t* bf16[3];
  float* global[3];
  int64_t codes_per_expert[3], scales_per_expert[3], bf16_per_expert[3];
};

__global__ void k_unpack(UnpackArgs a) {
  for (int64_t w = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; w < a.n_words;
       w += (int64_t)gridDim.x * blockDim.x) {
    WordSrc s;
    map_word(a.L, a.H, a.I, a.fmt, w, s);
    const uint32_t v = reinterpret_cast<const uint32_t*>(a.src)[w];
    if (a.fmt == FLINT_MOE_NVFP4) {
      if (s.is_scale) {
        uint8_t* p = a.scales[s.mat] + s.expert * a.scales_per_expert[s.mat] + s.idx[0];
        for (int b = 0; b < 4; ++b) p[b] = (uint8_t)(v >> (8 * b));
      } else {
        for (int b = 0; b < 4; ++b) {
          const int m = s.mat_b[b];
          a.codes[m][s.expert * a.codes_per_expert[m] + s.idx[b]] = (uint8_t)(v >> (8 * b));
        }
      }
    } else {
      uint8_t* p = a.bf16[s.mat] + s.expert * a.bf16_per_expert[s.mat] + s.idx[0];
      *reinterpret_cast<uint32_t*>(p) = v;
    }
  }
}

__global__ void k_unpack_globals(const float* src, float* g0, float* g1, float* g2, int n) {
  const int e = blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= n) return;
  if (g0) g0[e] = src[e * 4 + 0];
  if (g1) g1[e] = src[e * 4 + 1];
  if (g2) g2[e] = src[e * 4 + 2];
}

// ---------------------------------------------------------------------------
// Dequantisation read-back through the decode kernels' own fragment path.
// One warp per (tile, k-group); writes c * G as float32 in canonical order.
// ---------------------------------------------------------------------------
struct DeqArgs {
  Layout L;
  int H, I, fmt, mat;
  const uint8_t* expert_base;
  const float* G;  // tensor scale in the packed globals, or nullptr (BF16: 1)
  float* out;
  int n_tiles, n_kg;
};

__global__ void k_debug_dequant(DeqArgs a) {
  const int lane = threadIdx.x & 31;
  const int job = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (job >= a.n_tiles * a.n_kg) return;
  const int tile = job / a.n_kg, kg = job % a.n_kg;
  const bool gu = a.mat < 2;
  const uint8_t* tp = a.expert_base + (gu ? (int64_t)tile * a.L.gu_tile : a.L.gu_bytes + (int64_t)tile * a.L.dn_tile) +
                      (int64_t)kg * a.L.kg_bytes;
  const int cols = gu ? a.H : a.I;
  const int g = lane >> 2, t = lane & 3;
  const float G = a.G ? *a.G : 1.0f;
  for (int ks = 0; ks < 4; ++ks) {
    uint32_t af[4];
    if (a.fmt == FLINT_MOE_NVFP4) {
      const uint4 codes = *reinterpret_cast<const uint4*>(tp + lane * 16);
      const uint32_t sg = *reinterpret_cast<const uint32_t*>(tp + KG_CODE_BYTES + g * 4);
      const uint32_t sg8 = *reinterpret_cast<const uint32_t*>(tp + KG_CODE_BYTES + (g + 8) * 4);
      const uint32_t cw = ks == 0 ? codes.x : ks == 1 ? codes.y : ks == 2 ? codes.z : codes.w;
      nvfp4_afrag(cw, sg, sg8, ks, af);
    } else {
      const uint4 v = *reinterpret_cast<const uint4*>(tp + lane * 64 + ks * 16);
      af[0] = v.x;
      af[1] = v.y;
      af[2] = v.z;
      af[3] = v.w;
    }
    for (int b = 0; b < 4; ++b) {
      const int r = g + 8 * (b & 1);
      int row;
      if (gu) {
        if ((r < 8) != (a.mat == 0)) continue;
        row = tile * 8 + (r & 7);
      } else {
        row = tile * 16 + r;
      }
      const int c = kg * KG_COLS + ks * 16 + 2 * t + 8 * (b >> 1);
      float lo, hi;
      if (a.fmt == FLINT_MOE_NVFP4) {
        const __half2 h = *reinterpret_cast<const __half2*>(&af[b]);
        lo = __low2float(h);
        hi = __high2float(h);
      } else {
        lo = bf16lo(af[b]);
        hi = bf16hi(af[b]);
      }
      a.out[(int64_t)row * cols + c] = lo * G;
      a.out[(int64_t)row * cols + c + 1] = hi * G;
    }
  }
}

// ---------------------------------------------------------------------------
// NVFP4 quantiser (two-level recipe, all float32, nearest even, saturating).
// ---------------------------------------------------------------------------
__global__ void k_amax(const float* w, int64_t per_mat, int n_mat, unsigned* amax_bits) {
  const int m = blockIdx.y;
  const float* p = w + (int64_t)m * per_mat;
  float mx = 0.f;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < per_mat; i += (int64_t)gridDim.x * blockDim.x)
    mx = fmaxf(mx, fabsf(p[i]));
  mx = warp_max(mx);
  if ((threadIdx.x & 31) == 0 && mx > 0.f) atomicMax(amax_bits + m, __float_as_uint(mx));
}

// E2M1 nearest-even from the magnitude thresholds of the grid {0,.5,1,1.5,2,3,4,6}:
// midpoints 0.25, 1.25, 2.5 and 5 round down (to an even code), 0.75, 1.75 and
// 3.5 round up (to an even code).
__device__ __forceinline__ uint32_t e2m1_rn(float r) {
  const float m = fabsf(r);
  uint32_t c = (m > 0.25f) + (m >= 0.75f) + (m > 1.25f) + (m >= 1.75f) + (m > 2.5f) + (m >= 3.5f) + (m > 5.0f);
  return c | (signbit(r) ? 8u : 0u);
}

__global__ void k_quant(const float* w, int64_t per_mat, int cols, int n_mat, const unsigned* amax_bits,
                        uint8_t* codes, uint8_t* scales) {
  const int64_t blocks_per_mat = per_mat / 16;
  const int64_t total = blocks_per_mat * n_mat;
  for (int64_t b = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; b < total; b += (int64_t)gridDim.x * blockDim.x) {
    const int m = (int)(b / blocks_per_mat);
    const float amax = __uint_as_float(amax_bits[m]);
    const float G = amax / 2688.0f;
    const float4* src = reinterpret_cast<const float4*>(w + b * 16);
    float v[16];
    for (int i = 0; i < 4; ++i) {
      const float4 q = src[i];
      v[4 * i] = q.x;
      v[4 * i + 1] = q.y;
      v[4 * i + 2] = q.z;
      v[4 * i + 3] = q.w;
    }
    uint8_t sc = 0;
    uint32_t packed[2] = {0, 0};
    if (G != 0.f) {
      float ab = 0.f;
      for (int i = 0; i < 16; ++i) ab = fmaxf(ab, fabsf(v[i]));
      const float six_g = 6.0f * G;
      const float sf = ab / six_g;
      sc = (uint8_t)__nv_cvt_float_to_fp8(sf, __NV_SATFINITE, __NV_E4M3);
      const __half_raw hs = __nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)sc, __NV_E4M3);
      const float ds = __half2float(*reinterpret_cast<const __half*>(&hs));
      const float t = ds * G;
      if (t != 0.f) {
        for (int i = 0; i < 16; ++i) {
          const uint32_t c = e2m1_rn(v[i] / t);
          packed[i >> 3] |= c << (4 * (i & 7));
        }
      }
    }
    scales[b] = sc;
    uint2* dst = reinterpret_cast<uint2*>(codes + b * 8);
    *dst = make_uint2(packed[0], packed[1]);
  }
}

__global__ void k_quant_globals(const unsigned* amax_bits, float* global, int n_mat) {
  const int m = blockIdx.x * blockDim.x + threadIdx.x;
  if (m < n_mat) global[m] = __uint_as_float(amax_bits[m]) / 2688.0f;
}

}  // namespace flint

using namespace flint;

// ---------------------------------------------------------------------------
// C ABI
// ---------------------------------------------------------------------------
static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

extern "C" flint_moe_status flint_moe_check_config(const flint_moe_config* c) {
  if (!c) return FLINT_MOE_EINVAL;
  if (c->hidden < 256 || c->hidden > 8192 || c->hidden % 256) return FLINT_MOE_EUNSUPPORTED;
  if (c->hidden > 2048 && c->hidden % 2048) return FLINT_MOE_EUNSUPPORTED;
  if (c->inter < 64 || c->inter > 4096 || c->inter % 64) return FLINT_MOE_EUNSUPPORTED;
  if (c->num_experts < 1 || c->num_experts > MAX_EXPERTS) return FLINT_MOE_EUNSUPPORTED;
  if (c->top_k < 1 || c->top_k > MAX_TOPK || c->top_k > c->num_experts) return FLINT_MOE_EUNSUPPORTED;
  if (c->n_shared < 0 || c->n_shared > MAX_SHARED) return FLINT_MOE_EUNSUPPORTED;
  if (c->weight_fmt != FLINT_MOE_NVFP4 && c->weight_fmt != FLINT_MOE_BF16) return FLINT_MOE_EUNSUPPORTED;
  if (!(c->routed_scale == c->routed_scale)) return FLINT_MOE_EINVAL;
  return FLINT_MOE_OK;
}

extern "C" size_t flint_moe_packed_bytes(const flint_moe_config* c) {
  if (flint_moe_check_config(c) != FLINT_MOE_OK) return 0;
  return (size_t)make_layout(c->hidden, c->inter, c->num_experts, c->n_shared, c->weight_fmt).total;
}

static void fill_src_strides(const flint_moe_config* c, int64_t* codes_pe, int64_t* scales_pe, int64_t* bf16_pe) {
  const int64_t H = c->hidden, I = c->inter;
  const int64_t rows[3] = {I, I, H}, cols[3] = {H, H, I};
  for (int m = 0; m < 3; ++m) {
    codes_pe[m] = rows[m] * cols[m] / 2;
    scales_pe[m] = rows[m] * cols[m] / 16;
    bf16_pe[m] = rows[m] * cols[m] * 2;
  }
}

static int grid_for(int64_t n, int block) {
  int64_t g = (n + block - 1) / block;
  if (g > 152 * 32) g = 152 * 32;
  return (int)(g < 1 ? 1 : g);
}

extern "C" flint_moe_status flint_moe_pack(const flint_moe_config* c, const flint_moe_src* src, void* dst,
                                           size_t dst_bytes, int32_t* dev_status, cudaStream_t stream) {
  flint_moe_status st = flint_moe_check_config(c);
  if (st != FLINT_MOE_OK) return st;
  if (!src || !dst) return FLINT_MOE_EINVAL;
  const Layout L = make_layout(c->hidden, c->inter, c->num_experts, c->n_shared, c->weight_fmt);
  if (dst_bytes < (size_t)L.total) return FLINT_MOE_EINVAL;
  if (!aligned16(dst)) return FLINT_MOE_EALIGN;
  PackArgs a;
  a.L = L;
  a.H = c->hidden;
  a.I = c->inter;
  a.fmt = c->weight_fmt;
  a.n_words = L.globals_off / 4;
  const flint_moe_nvfp4_src* m3[3] = {&src->gate, &src->up, &src->down};
  const uint16_t* b3[3] = {src->gate_bf16, src->up_bf16, src->down_bf16};
  for (int m = 0; m < 3; ++m) {
    if (c->weight_fmt == FLINT_MOE_NVFP4) {
      if (!m3[m]->codes || !m3[m]->scales || !m3[m]->global) return FLINT_MOE_EINVAL;
      if (!aligned16(m3[m]->scales)) return FLINT_MOE_EALIGN;
    } else {
      if (!b3[m]) return FLINT_MOE_EINVAL;
      if (!aligned16(b3[m])) return FLINT_MOE_EALIGN;
    }
    a.codes[m] = m3[m]->codes;
    a.scales[m] = m3[m]->scales;
    a.bf16[m] = reinterpret_cast<const uint8_t*>(b3[m]);
  }
  fill_src_strides(c, a.codes_per_expert, a.scales_per_expert, a.bf16_per_expert);
  a.dst = static_cast<uint8_t*>(dst);
  a.status = dev_status;
  k_pack<<<grid_for(a.n_words, 256), 256, 0, stream>>>(a);
  GlobalsArgs ga;
  for (int m = 0; m < 3; ++m) ga.g[m] = m3[m]->global;
  ga.dst = reinterpret_cast<float*>(static_cast<uint8_t*>(dst) + L.globals_off);
  ga.n = c->num_experts + c->n_shared;
  ga.fmt = c->weight_fmt;
  k_pack_globals<<<(ga.n + 127) / 128, 128, 0, stream>>>(ga);
  return cudaGetLastError() == cudaSuccess ? FLINT_MOE_OK : FLINT_MOE_ECUDA;
}

extern "C" flint_moe_status flint_moe_unpack_debug(const flint_moe_config* c, const void* packed,
                                                   const flint_moe_src* dst, cudaStream_t stream) {
  flint_moe_status st = flint_moe_check_config(c);
  if (st != FLINT_MOE_OK) return st;
  if (!packed || !dst) return FLINT_MOE_EINVAL;
  if (!aligned16(packed)) return FLINT_MOE_EALIGN;
  const Layout L = make_layout(c->hidden, c->inter, c->num_experts, c->n_shared, c->weight_fmt);
  UnpackArgs a;
  a.L = L;
  a.H = c->hidden;
  a.I = c->inter;
  a.fmt = c->weight_fmt;
  a.n_words = L.globals_off / 4;
  a.src = static_cast<const uint8_t*>(packed);
  const flint_moe_nvfp4_src* m3[3] = {&dst->gate, &dst->up, &dst->down};
  const uint16_t* b3[3] = {dst->gate_bf16, dst->up_bf16, dst->down_bf16};
  for (int m = 0; m < 3; ++m) {
    if (c->weight_fmt == FLINT_MOE_NVFP4) {
      if (!m3[m]->codes || !m3[m]->scales) return FLINT_MOE_EINVAL;
    } else if (!b3[m]) {
      return FLINT_MOE_EINVAL;
    }
    a.codes[m] = const_cast<uint8_t*>(m3[m]->codes);
    a.scales[m] = const_cast<uint8_t*>(m3[m]->scales);
    a.bf16[m] = reinterpret_cast<uint8_t*>(const_cast<uint16_t*>(b3[m]));
    a.global[m] = const_cast<float*>(m3[m]->global);
  }
  fill_src_strides(c, a.codes_per_expert, a.scales_per_expert, a.bf16_per_expert);
  k_unpack<<<grid_for(a.n_words, 256), 256, 0, stream>>>(a);
  if (c->weight_fmt == FLINT_MOE_NVFP4) {
    const int n = c->num_experts + c->n_shared;
    k_unpack_globals<<<(n + 127) / 128, 128, 0, stream>>>(
        reinterpret_cast<const float*>(static_cast<const uint8_t*>(packed) + L.globals_off), a.global[0], a.global[1],
        a.global[2], n);
  }
  return cudaGetLastError() == cudaSuccess ? FLINT_MOE_OK : FLINT_MOE_ECUDA;
}

extern "C" flint_moe_status flint_moe_debug_dequant(const flint_moe_config* c, const void* packed, int32_t expert,
                                                    int32_t mat, float* out, cudaStream_t stream) {
  flint_moe_status st = flint_moe_check_config(c);
  if (st != FLINT_MOE_OK) return st;
  if (!packed || !out || mat < 0 || mat > 2 || expert < 0 || expert >= c->num_experts + c->n_shared)
    return FLINT_MOE_EINVAL;
  if (!aligned16(packed)) return FLINT_MOE_EALIGN;
  const Layout L = make_layout(c->hidden, c->inter, c->num_experts, c->n_shared, c->weight_fmt);
  DeqArgs a;
  a.L = L;
  a.H = c->hidden;
  a.I = c->inter;
  a.fmt = c->weight_fmt;
  a.mat = mat;
  a.expert_base = static_cast<const uint8_t*>(packed) + (int64_t)expert * L.expert_bytes;
  a.out = out;
  a.n_tiles = mat < 2 ? c->inter / 8 : c->hidden / 16;
  a.n_kg = (mat < 2 ? c->hidden : c->inter) / KG_COLS;
  a.G = c->weight_fmt == FLINT_MOE_NVFP4
            ? reinterpret_cast<const float*>(static_cast<const uint8_t*>(packed) + L.globals_off) + expert * 4 + mat
            : nullptr;
  const int jobs = a.n_tiles * a.n_kg;
  k_debug_dequant<<<(jobs + 3) / 4, 128, 0, stream>>>(a);
  return cudaGetLastError() == cudaSuccess ? FLINT_MOE_OK : FLINT_MOE_ECUDA;
}

extern "C" flint_moe_status flint_moe_quantize_nvfp4(const float* w, int32_t n_mat, int32_t rows, int32_t cols,
                                                     uint8_t* codes, uint8_t* scales, float* global,
                                                     cudaStream_t stream) {
  if (!w || !codes || !scales || !global || n_mat < 1 || rows < 1 || cols < 16 || cols % 16) return FLINT_MOE_EINVAL;
  if (!aligned16(w) || (reinterpret_cast<uintptr_t>(codes) & 7)) return FLINT_MOE_EALIGN;
  const int64_t per_mat = (int64_t)rows * cols;
  // the global scale array doubles as the amax accumulator (uint bits of a non-negative float)
  unsigned* amax_bits = reinterpret_cast<unsigned*>(global);
  if (cudaMemsetAsync(amax_bits, 0, sizeof(unsigned) * n_mat, stream) != cudaSuccess) return FLINT_MOE_ECUDA;
  dim3 ag((unsigned)grid_for(per_mat, 256) > 512 ? 512 : (unsigned)grid_for(per_mat, 256), (unsigned)n_mat);
  k_amax<<<ag, 256, 0, stream>>>(w, per_mat, n_mat, amax_bits);
  k_quant<<<grid_for(per_mat / 16 * n_mat, 256), 256, 0, stream>>>(w, per_mat, cols, n_mat, amax_bits, codes, scales);
  k_quant_globals<<<(n_mat + 127) / 128, 128, 0, stream>>>(amax_bits, global, n_mat);
  return cudaGetLastError() == cudaSuccess ? FLINT_MOE_OK : FLINT_MOE_ECUDA;
}

// ---------------------------------------------------------------------------
// Dense matrices for the small-batch GEMV: the MoE repack with a layout of one
// down matrix (H = N rows, I = K columns) and no gate/up tiles.
// ---------------------------------------------------------------------------
static bool gemv_shape_ok(int32_t N, int32_t K, int32_t fmt) {
  if (N < 16 || N % 16 || N > (1 << 20)) return false;
  if (K < 256 || K > 8192 || K % 256 || (K > 2048 && K % 2048)) return false;
  return fmt == FLINT_MOE_NVFP4 || fmt == FLINT_MOE_BF16;
}

extern "C" size_t flint_gemv_packed_bytes(int32_t N, int32_t K, int32_t fmt) {
  return gemv_shape_ok(N, K, fmt) ? (size_t)make_dense_layout(N, K, fmt).total : 0;
}

extern "C" flint_moe_status flint_gemv_pack(const flint_gemv_src* src, int32_t N, int32_t K, int32_t fmt, void* dst,
                                            size_t dst_bytes, int32_t* dev_status, cudaStream_t stream) {
  if (!gemv_shape_ok(N, K, fmt)) return FLINT_MOE_EUNSUPPORTED;
  if (!src || !dst) return FLINT_MOE_EINVAL;
  const Layout L = make_dense_layout(N, K, fmt);
  if (dst_bytes < (size_t)L.total) return FLINT_MOE_EINVAL;
  if (!aligned16(dst)) return FLINT_MOE_EALIGN;
  if (fmt == FLINT_MOE_NVFP4) {
    if (!src->codes || !src->scales || !src->global_) return FLINT_MOE_EINVAL;
    if (!aligned16(src->scales)) return FLINT_MOE_EALIGN;
  } else {
    if (!src->bf16) return FLINT_MOE_EINVAL;
    if (!aligned16(src->bf16)) return FLINT_MOE_EALIGN;
  }
  PackArgs a = {};
  a.L = L;
  a.H = N;
  a.I = K;
  a.fmt = fmt;
  a.n_words = L.globals_off / 4;
  a.codes[2] = src->codes;
  a.scales[2] = src->scales;
  a.bf16[2] = reinterpret_cast<const uint8_t*>(src->bf16);
  a.dst = static_cast<uint8_t*>(dst);
  a.status = dev_status;
  k_pack<<<grid_for(a.n_words, 256), 256, 0, stream>>>(a);
  GlobalsArgs ga;
  for (int m = 0; m < 3; ++m) ga.g[m] = src->global_;
  ga.dst = reinterpret_cast<float*>(static_cast<uint8_t*>(dst) + L.globals_off);
  ga.n = 1;
  ga.fmt = fmt;
  k_pack_globals<<<1, 32, 0, stream>>>(ga);
  return cudaGetLastError() == cudaSuccess ? FLINT_MOE_OK : FLINT_MOE_ECUDA;
}

extern "C" flint_moe_status flint_gemv_unpack_debug(const void* packed, int32_t N, int32_t K, int32_t fmt,
                                                    const flint_gemv_src* dst, cudaStream_t stream) {
  if (!gemv_shape_ok(N, K, fmt)) return FLINT_MOE_EUNSUPPORTED;
  if (!packed || !dst) return FLINT_MOE_EINVAL;
  const Layout L = make_dense_layout(N, K, fmt);
  UnpackArgs a = {};
  a.L = L;
  a.H = N;
  a.I = K;
  a.fmt = fmt;
  a.n_words = L.globals_off / 4;
  a.src = static_cast<const uint8_t*>(packed);
  if (fmt == FLINT_MOE_NVFP4) {
    if (!dst->codes || !dst->scales || !dst->global_) return FLINT_MOE_EINVAL;
    a.codes[2] = const_cast<uint8_t*>(dst->codes);
    a.scales[2] = const_cast<uint8_t*>(dst->scales);
  } else {
    if (!dst->bf16) return FLINT_MOE_EINVAL;
    a.bf16[2] = reinterpret_cast<uint8_t*>(const_cast<uint16_t*>(dst->bf16));
  }
  k_unpack<<<grid_for(a.n_words, 256), 256, 0, stream>>>(a);
  if (fmt == FLINT_MOE_NVFP4) {
    float* g = const_cast<float*>(dst->global_);
    k_unpack_globals<<<1, 32, 0, stream>>>(reinterpret_cast<const float*>(a.src + L.globals_off), nullptr, nullptr,
                                          g, 1);
  }
  return cudaGetLastError() == cudaSuccess ? FLINT_MOE_OK : FLINT_MOE_ECUDA;
}
