// step_kernel.cuh -- the fused AdamW / AdEMAMix step over a plan's chunk
// table (one launch per gradient-dtype bucket).
//
// Per element, with the per-step scalars formed once on the host
// ("Investigate SM103 bias-correction broadcast in 32-bit optimizers",
// 'Problem': those scalars are uniform, so no thread evaluates powf):
//   g' = g * clip_coef
//   m  = b1 m + (1-b1) g'              v = b2 v + (1-b2) g'^2
//   m2 = b3 m2 + (1-b3) g'             (AdEMAMix)
//   u  = (m / bc1 [+ alpha m2]) / (sqrt(v / bc2) + eps)
//   p  = p (1 - lr wd) - lr u          decay-first: both terms from the old p
// ("Fix decoupled weight decay ordering in the CUDA Adam/AdEMAMix kernels",
// body).  Every operation is one IEEE round-to-nearest fp32 operation in the
// order written (no FMA contraction), so m and v before write-back are
// reproducible bit for bit.  Low-precision states are decoded exactly to fp32
// and re-encoded with nearest or stochastic rounding, each tensor read and
// written once ("When Small Updates Disappear", sec. 8.1).
//
// Layout: a persistent grid strides over the bucket's chunks; inside a chunk
// each thread owns groups of 8 consecutive elements, moved with 16-byte
// streaming loads and stores (p, m, v, m2: evict-first; g: read-only path).
// The group start is a multiple of 8 elements and every base pointer is
// 16-byte aligned, so each stream's vector is naturally aligned (E4M3: 8
// bytes, E2M2: 4 bytes).  The one ragged group of a tensor is handled
// element by element.  Stochastic-rounding draws: two Philox4x32-10 calls
// per group (counters q = e0/4 and e0/4 + 1), so each draw depends only on
// (seed, step, tensor, element).
#pragma once

#include "common.cuh"
#include "internal.h"

namespace psopt {

constexpr int kStepThreads = 256;

template <int COMBO>
struct Combo;
template <> struct Combo<SC_F32>       { static constexpr int M = OPT_F32,  V = OPT_F32;  };
template <> struct Combo<SC_BF16_BF16> { static constexpr int M = OPT_BF16, V = OPT_BF16; };
template <> struct Combo<SC_BF16_E4M3> { static constexpr int M = OPT_BF16, V = OPT_E4M3; };
template <> struct Combo<SC_BF16_E2M2> { static constexpr int M = OPT_BF16, V = OPT_E2M2; };

__device__ __forceinline__ void u4_to_f4(uint4 w, float* f) {
  f[0] = u2f(w.x); f[1] = u2f(w.y); f[2] = u2f(w.z); f[3] = u2f(w.w);
}
__device__ __forceinline__ uint4 f4_to_u4(const float* f) {
  return make_uint4(f2u(f[0]), f2u(f[1]), f2u(f[2]), f2u(f[3]));
}
__device__ __forceinline__ void bf16x8_to_f(uint4 w, float* f) {
  const uint32_t a[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int k = 0; k < 4; ++k) { f[2 * k] = u2f(a[k] << 16); f[2 * k + 1] = u2f(a[k] & 0xFFFF0000u); }
}

template <int GT, int COMBO, int ALGO, bool SR>
__device__ __forceinline__ uint32_t step_group(const TensorDesc& td, int64_t e0, int cnt,
                                               float coef, const opt_step_scalars& sc,
                                               uint32_t tensor, uint32_t seed_lo,
                                               uint32_t seed_hi, uint32_t step32) {
  constexpr int MD = Combo<COMBO>::M, VD = Combo<COMBO>::V;
  constexpr bool LOWP = COMBO != SC_F32;
  const bool full = cnt == 8;

  float p[8], g[8], m[8], v[8], m2[8];
  uint32_t vold[8];

  // ------------------------------------------------------------- loads
  if (full) {
    u4_to_f4(ld_cs_u4(td.p + e0), p);
    u4_to_f4(ld_cs_u4(td.p + e0 + 4), p + 4);
    if (GT == OPT_BF16) {
      bf16x8_to_f(ld_nc_u4(static_cast<const uint16_t*>(td.g) + e0), g);
    } else {
      u4_to_f4(ld_nc_u4(static_cast<const float*>(td.g) + e0), g);
      u4_to_f4(ld_nc_u4(static_cast<const float*>(td.g) + e0 + 4), g + 4);
    }
    if (MD == OPT_F32) {
      u4_to_f4(ld_cs_u4(static_cast<float*>(td.m) + e0), m);
      u4_to_f4(ld_cs_u4(static_cast<float*>(td.m) + e0 + 4), m + 4);
    } else {
      bf16x8_to_f(ld_cs_u4(static_cast<uint16_t*>(td.m) + e0), m);
    }
    if (VD == OPT_F32) {
      const uint4 a = ld_cs_u4(static_cast<float*>(td.v) + e0);
      const uint4 b = ld_cs_u4(static_cast<float*>(td.v) + e0 + 4);
      vold[0] = a.x; vold[1] = a.y; vold[2] = a.z; vold[3] = a.w;
      vold[4] = b.x; vold[5] = b.y; vold[6] = b.z; vold[7] = b.w;
#pragma unroll
      for (int j = 0; j < 8; ++j) v[j] = u2f(vold[j]);
    } else if (VD == OPT_BF16) {
      const uint4 w = ld_cs_u4(static_cast<uint16_t*>(td.v) + e0);
      const uint32_t a[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) { vold[2 * k] = a[k] & 0xFFFFu; vold[2 * k + 1] = a[k] >> 16; }
#pragma unroll
      for (int j = 0; j < 8; ++j) v[j] = bf16_dec(vold[j]);
    } else if (VD == OPT_E4M3) {
      const uint2 w = ld_cs_u2(static_cast<uint8_t*>(td.v) + e0);
#pragma unroll
      for (int j = 0; j < 4; ++j) { vold[j] = (w.x >> (8 * j)) & 0xFFu; vold[4 + j] = (w.y >> (8 * j)) & 0xFFu; }
#pragma unroll
      for (int j = 0; j < 8; ++j) v[j] = e4m3_dec(vold[j]);
    } else {
      const uint32_t w = ld_cs_u1(static_cast<uint8_t*>(td.v) + (e0 >> 1));
#pragma unroll
      for (int j = 0; j < 8; ++j) vold[j] = (w >> (4 * j)) & 0xFu;
#pragma unroll
      for (int j = 0; j < 8; ++j) v[j] = e2m2_dec(vold[j]);
    }
    if (ALGO == ALGO_ADEMAMIX) {
      u4_to_f4(ld_cs_u4(td.m2 + e0), m2);
      u4_to_f4(ld_cs_u4(td.m2 + e0 + 4), m2 + 4);
    }
  } else {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const bool in = j < cnt;
      const int64_t e = e0 + j;
      p[j] = in ? td.p[e] : 0.0f;
      g[j] = !in ? 0.0f
                 : (GT == OPT_BF16 ? bf16_dec(static_cast<const uint16_t*>(td.g)[e])
                                   : static_cast<const float*>(td.g)[e]);
      m[j] = !in ? 0.0f
                 : (MD == OPT_F32 ? static_cast<const float*>(td.m)[e]
                                  : bf16_dec(static_cast<const uint16_t*>(td.m)[e]));
      uint32_t code = 0;
      if (in) {
        if (VD == OPT_F32) code = f2u(static_cast<const float*>(td.v)[e]);
        else if (VD == OPT_BF16) code = static_cast<const uint16_t*>(td.v)[e];
        else if (VD == OPT_E4M3) code = static_cast<const uint8_t*>(td.v)[e];
        else code = (static_cast<const uint8_t*>(td.v)[e >> 1] >> (4 * (e & 1))) & 0xFu;
      }
      vold[j] = code;
      v[j] = VD == OPT_F32 ? u2f(code)
           : VD == OPT_BF16 ? bf16_dec(code)
           : VD == OPT_E4M3 ? e4m3_dec(code) : e2m2_dec(code);
      if (ALGO == ALGO_ADEMAMIX) m2[j] = in ? td.m2[e] : 0.0f;
    }
  }

  // ------------------------------------------------------------- draws
  uint32_t words[8];
  if (LOWP && SR) {
    const uint4 d0 = draw_words((uint64_t)e0 >> 2, tensor, step32, seed_lo, seed_hi);
    const uint4 d1 = draw_words(((uint64_t)e0 >> 2) + 1, tensor, step32, seed_lo, seed_hi);
    words[0] = d0.x; words[1] = d0.y; words[2] = d0.z; words[3] = d0.w;
    words[4] = d1.x; words[5] = d1.y; words[6] = d1.z; words[7] = d1.w;
  }

  // ----------------------------------------------------------- compute
  uint32_t mcode[8], vcode[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const float ge = __fmul_rn(g[j], coef);
    const float mn = __fadd_rn(__fmul_rn(sc.beta1, m[j]), __fmul_rn(sc.omb1, ge));
    const float vn = __fadd_rn(__fmul_rn(sc.beta2, v[j]), __fmul_rn(sc.omb2, __fmul_rn(ge, ge)));
    float num = __fmul_rn(mn, sc.inv_bc1);
    if (ALGO == ALGO_ADEMAMIX) {
      const float m2n = __fadd_rn(__fmul_rn(sc.beta3, m2[j]), __fmul_rn(sc.omb3, ge));
      num = __fadd_rn(num, __fmul_rn(sc.alpha, m2n));
      m2[j] = m2n;
    }
    const float den = __fadd_rn(__fsqrt_rn(__fmul_rn(vn, sc.inv_bc2)), sc.eps);
    const float u = __fdiv_rn(num, den);
    p[j] = __fsub_rn(__fmul_rn(p[j], sc.decay), __fmul_rn(sc.lr, u));
    if (MD == OPT_F32) m[j] = mn;
    else mcode[j] = bf16_enc<SR>(mn, SR ? (words[j] & 0xFFFFu) : 0u);
    if (VD == OPT_F32) { v[j] = vn; vcode[j] = f2u(vn); }
    else if (VD == OPT_BF16) vcode[j] = bf16_enc<SR>(vn, SR ? (words[j] >> 16) : 0u);
    else if (VD == OPT_E2M2) vcode[j] = e2m2_enc<SR>(vn, SR ? (words[j] >> 16) : 0u);
    else if (SR) vcode[j] = e4m3_enc_sr(vn, words[j] >> 16);
    else v[j] = vn;   // E4M3 nearest: converted in pairs below
  }
  if (VD == OPT_E4M3 && !SR) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint32_t pair = e4m3x2_rn(v[2 * k], v[2 * k + 1]);
      vcode[2 * k] = pair & 0xFFu;
      vcode[2 * k + 1] = pair >> 8;
    }
  }
  uint32_t same = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) same += (j < cnt && vcode[j] == vold[j]) ? 1u : 0u;

  // ------------------------------------------------------------ stores
  if (full) {
    st_cs_u4(td.p + e0, f4_to_u4(p));
    st_cs_u4(td.p + e0 + 4, f4_to_u4(p + 4));
    if (MD == OPT_F32) {
      st_cs_u4(static_cast<float*>(td.m) + e0, f4_to_u4(m));
      st_cs_u4(static_cast<float*>(td.m) + e0 + 4, f4_to_u4(m + 4));
    } else {
      st_cs_u4(static_cast<uint16_t*>(td.m) + e0,
               make_uint4(mcode[0] | (mcode[1] << 16), mcode[2] | (mcode[3] << 16),
                          mcode[4] | (mcode[5] << 16), mcode[6] | (mcode[7] << 16)));
    }
    if (VD == OPT_F32) {
      st_cs_u4(static_cast<float*>(td.v) + e0, f4_to_u4(v));
      st_cs_u4(static_cast<float*>(td.v) + e0 + 4, f4_to_u4(v + 4));
    } else if (VD == OPT_BF16) {
      st_cs_u4(static_cast<uint16_t*>(td.v) + e0,
               make_uint4(vcode[0] | (vcode[1] << 16), vcode[2] | (vcode[3] << 16),
                          vcode[4] | (vcode[5] << 16), vcode[6] | (vcode[7] << 16)));
    } else if (VD == OPT_E4M3) {
      st_cs_u2(static_cast<uint8_t*>(td.v) + e0,
               make_uint2(vcode[0] | (vcode[1] << 8) | (vcode[2] << 16) | (vcode[3] << 24),
                          vcode[4] | (vcode[5] << 8) | (vcode[6] << 16) | (vcode[7] << 24)));
    } else {
      uint32_t w = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) w |= vcode[j] << (4 * j);
      st_cs_u1(static_cast<uint8_t*>(td.v) + (e0 >> 1), w);
    }
    if (ALGO == ALGO_ADEMAMIX) {
      st_cs_u4(td.m2 + e0, f4_to_u4(m2));
      st_cs_u4(td.m2 + e0 + 4, f4_to_u4(m2 + 4));
    }
  } else {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (j >= cnt) break;
      const int64_t e = e0 + j;
      td.p[e] = p[j];
      if (MD == OPT_F32) static_cast<float*>(td.m)[e] = m[j];
      else static_cast<uint16_t*>(td.m)[e] = (uint16_t)mcode[j];
      if (VD == OPT_F32) static_cast<float*>(td.v)[e] = v[j];
      else if (VD == OPT_BF16) static_cast<uint16_t*>(td.v)[e] = (uint16_t)vcode[j];
      else if (VD == OPT_E4M3) static_cast<uint8_t*>(td.v)[e] = (uint8_t)vcode[j];
      if (ALGO == ALGO_ADEMAMIX) td.m2[e] = m2[j];
    }
    if (VD == OPT_E2M2) {
      // whole bytes: e0 is even, so byte k holds elements 2k and 2k+1 of the
      // group; an element past the end contributes a zero nibble
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        if (2 * k >= cnt) break;
        const uint32_t hi = (2 * k + 1 < cnt) ? vcode[2 * k + 1] : 0u;
        static_cast<uint8_t*>(td.v)[(e0 >> 1) + k] = (uint8_t)(vcode[2 * k] | (hi << 4));
      }
    }
  }
  return same;
}

template <int GT, int COMBO, int ALGO, bool SR>
__global__ void __launch_bounds__(kStepThreads)
step_kernel(const StepArgs a) {
  float coef = 1.0f;
  if (a.d_norm != nullptr) {
    if (a.d_norm->status != OPT_OK) return;     // non-finite norm: leave all untouched
    coef = a.d_norm->clip_coef;
  }
  uint32_t same = 0;
  for (int64_t c = a.chunk_begin + blockIdx.x; c < a.chunk_end; c += gridDim.x) {
    const opt_chunk ch = a.chunks[c];
    const TensorDesc td = a.tensors[ch.tensor];
    const int len = (int)ch.len;
    for (int base = threadIdx.x * 8; base < len; base += kStepThreads * 8) {
      same += step_group<GT, COMBO, ALGO, SR>(td, ch.start + base, min(8, len - base), coef, a.sc,
                                              ch.tensor, a.seed_lo, a.seed_hi, a.step32);
    }
  }
  if (a.unchanged != nullptr) {
    // integer sums: the total does not depend on the order of the atomics
    same = __reduce_add_sync(0xFFFFFFFFu, same);
    if ((threadIdx.x & 31) == 0 && same) atomicAdd(a.unchanged, (unsigned long long)same);
  }
}

// Persistent launch: as many CTAs as fit on the GPU at once (occupancy is
// a property of the kernel, cached), but no more than there are chunks.
template <int GT, int COMBO, int ALGO, bool SR>
cudaError_t launch_one(const StepArgs& a, int sm_count, cudaStream_t s) {
  const int64_t n = a.chunk_end - a.chunk_begin;
  if (n <= 0) return cudaSuccess;
  auto k = step_kernel<GT, COMBO, ALGO, SR>;
  static int cached_grid_per_sm = 0;
  if (cached_grid_per_sm == 0) {
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, kStepThreads, 0) != cudaSuccess ||
        per_sm < 1)
      per_sm = 1;
    cached_grid_per_sm = per_sm;
  }
  const int64_t full = (int64_t)cached_grid_per_sm * sm_count;
  const int grid = (int)(n < full ? n : full);
  k<<<grid, kStepThreads, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace psopt
