// common.cuh -- device-side building blocks shared by the library's kernels:
// table layouts, the per-step scalar block, Philox4x32-10, the BF16 / E4M3 /
// unsigned-E2M2 state codecs, and streaming vector loads and stores.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "opt.h"

namespace psopt {

// ---------------------------------------------------------------- tables
// One entry per tensor of a plan, uploaded once at plan creation.
struct TensorDesc {
  float* p;
  const void* g;
  void* m;
  void* v;
  float* m2;
  int64_t numel;
};
static_assert(sizeof(TensorDesc) == 48, "TensorDesc layout");
static_assert(sizeof(opt_chunk) == 16, "opt_chunk layout");

// One fixed slot of the gradient-norm pass: the slot's chunks are
// c = bucket_begin + slot + k * OPT_NORM_SLOTS, summed in that order.
struct NormSlot {
  double sum;          // sum of finite squares
  uint64_t nan_count;
  uint64_t inf_count;
  float maxabs;        // max |g| over finite elements
  uint32_t pad;
};
static_assert(sizeof(NormSlot) == 32, "NormSlot layout");

// Everything a step kernel needs besides the tables.
struct StepArgs {
  const TensorDesc* tensors;
  const opt_chunk* chunks;
  int64_t chunk_begin, chunk_end;     // this bucket's range of the chunk table
  opt_step_scalars sc;
  uint32_t seed_lo, seed_hi, step32;
  const opt_norm_result* d_norm;      // NULL: no clipping
  unsigned long long* unchanged;      // NULL: do not count
};

// ------------------------------------------------------------- bit views
__device__ __forceinline__ uint32_t f2u(float x) { return __float_as_uint(x); }
__device__ __forceinline__ float u2f(uint32_t x) { return __uint_as_float(x); }

// ------------------------------------------------------------------ Philox
// Philox4x32 with 10 rounds (Salmon, Moraes, Dror, Shaw, "Parallel Random
// Numbers: As Easy as 1, 2, 3", SC'11, sec. 3).  A round multiplies counter
// words 0 and 2 by the two round multipliers and recombines the product
// halves with words 1 and 3 and the round key; the key advances by the two
// Weyl increments between rounds.
__device__ __forceinline__ uint4 philox10(uint4 c, uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    if (r) { k0 += 0x9E3779B9u; k1 += 0xBB67AE85u; }
    const uint32_t lo0 = 0xD2511F53u * c.x, hi0 = __umulhi(0xD2511F53u, c.x);
    const uint32_t lo1 = 0xCD9E8D57u * c.z, hi1 = __umulhi(0xCD9E8D57u, c.z);
    c = make_uint4(hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0);
  }
  return c;
}

// The four draw words for elements 4q .. 4q+3 of tensor `tensor` at a step.
__device__ __forceinline__ uint4 draw_words(uint64_t q, uint32_t tensor, uint32_t step32,
                                            uint32_t seed_lo, uint32_t seed_hi) {
  return philox10(make_uint4((uint32_t)q, (uint32_t)(q >> 32), tensor, step32), seed_lo, seed_hi);
}

// -------------------------------------------------------------- BF16 codec
// Decode is exact: the code is the top half of an fp32 word.
__device__ __forceinline__ float bf16_dec(uint32_t code) { return u2f(code << 16); }

// Nearest-even on the 16 dropped bits; Inf kept, NaN kept quiet.
__device__ __forceinline__ uint32_t bf16_enc_rn(float x) {
  const uint32_t w = f2u(x);
  if ((w & 0x7F800000u) == 0x7F800000u)
    return (w >> 16) | ((w & 0x007FFFFFu) ? 0x40u : 0u);
  return (w + 0x7FFFu + ((w >> 16) & 1u)) >> 16;
}

// Stochastic: add the 16-bit draw to the word and keep the top half; the
// kept part moves away from zero exactly when the dropped 16 bits plus the
// draw carry ("When Small Updates Disappear", sec. 6.1).
__device__ __forceinline__ uint32_t bf16_enc_sr(float x, uint32_t r16) {
  const uint32_t w = f2u(x);
  if ((w & 0x7F800000u) == 0x7F800000u)
    return (w >> 16) | ((w & 0x007FFFFFu) ? 0x40u : 0u);
  return (w + r16) >> 16;
}

template <bool SR>
__device__ __forceinline__ uint32_t bf16_enc(float x, uint32_t r16) {
  return SR ? bf16_enc_sr(x, r16) : bf16_enc_rn(x);
}

// ------------------------------------------------- small-grid rounding core
// Rounds a >= 0 onto a grid with P fraction bits whose binades start at
// 2^EMIN (spacing 2^(EMIN-P) below it), saturating at vmax.  With
// ulp = 2^(e-P), t = a/ulp, k = floor(t): stochastic rounding takes k+1 iff
// the first 16 fraction bits of t plus the draw carry past 2^16; nearest
// takes k+1 iff frac(t) > 1/2, or = 1/2 with k odd.  Every operation below is
// exact (power-of-two scalings, floor, and the subtraction of the floor).
template <int P, int EMIN, bool SR>
__device__ __forceinline__ float grid_round(float a, uint32_t r16, float vmax) {
  if (a >= vmax) return vmax;
  const int eb = (int)(f2u(a) >> 23);               // a >= 0: biased exponent
  const int e = max(eb - 127, EMIN);
  const float ulp = u2f((uint32_t)(e - P + 127) << 23);
  const float inv_ulp = u2f((uint32_t)(P - e + 127) << 23);
  const float t = __fmul_rn(a, inv_ulp);
  const float k = floorf(t);
  const float f = __fsub_rn(t, k);
  uint32_t up;
  if (SR) {
    const uint32_t l16 = __float2uint_rz(__fmul_rn(f, 65536.0f));
    up = (l16 + r16) >> 16;
  } else {
    up = (f > 0.5f || (f == 0.5f && (__float2uint_rz(k) & 1u))) ? 1u : 0u;
  }
  return fminf(__fmul_rn(__fadd_rn(k, (float)up), ulp), vmax);
}

// ------------------------------------------------------- E4M3 (FP8) codec
__device__ __forceinline__ float e4m3_dec(uint32_t c) {
  const uint32_t mag = c & 0x7Fu;
  float r = (mag < 8u) ? __fmul_rn((float)mag, 0.001953125f)          // k * 2^-9
                       : u2f((mag << 20) + (120u << 23));             // (1+k/8) 2^(e-7)
  if (mag == 0x7Fu) r = u2f(0x7FC00000u);
  return (c & 0x80u) ? -r : r;
}

// code of a magnitude that lies exactly on the E4M3 grid, 0 <= q <= 448
__device__ __forceinline__ uint32_t e4m3_code_exact(float q) {
  if (q < 0.015625f) return __float2uint_rz(__fmul_rn(q, 512.0f));   // 0..8
  const uint32_t b = f2u(q);
  return (((b >> 23) - 120u) << 3) | ((b >> 20) & 7u);
}

// Nearest (saturating) conversion of two values by the hardware converter:
// the first operand lands in the upper byte.
__device__ __forceinline__ uint32_t e4m3x2_rn(float lo, float hi) {
  unsigned short r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return (uint32_t)r;
}

__device__ __forceinline__ uint32_t e4m3_enc_sr(float x, uint32_t r16) {
  if (x != x) return 0x7Fu;
  const uint32_t sign = (f2u(x) >> 24) & 0x80u;
  return sign | e4m3_code_exact(grid_round<3, -6, true>(fabsf(x), r16, 448.0f));
}

// ------------------------------------------------ unsigned E2M2 (FP4) codec
__device__ __forceinline__ float e2m2_dec(uint32_t c) {
  return (c < 4u) ? __fmul_rn((float)c, 0.25f)
                  : u2f((((c >> 2) + 126u) << 23) | ((c & 3u) << 21));
}

__device__ __forceinline__ uint32_t e2m2_code_exact(float q) {   // 0 <= q <= 7 on grid
  if (q < 1.0f) return __float2uint_rz(__fmul_rn(q, 4.0f));      // 0..4
  const uint32_t b = f2u(q);
  return (((b >> 23) - 126u) << 2) | ((b >> 21) & 3u);
}

template <bool SR>
__device__ __forceinline__ uint32_t e2m2_enc(float x, uint32_t r16) {
  if (x != x) return 15u;
  if (!(x > 0.0f)) return 0u;
  return e2m2_code_exact(grid_round<2, 0, SR>(x, r16, 7.0f));
}

// -------------------------------------------------- streaming memory access
// Read-only gradient stream: non-coherent path, no L1 allocation.
__device__ __forceinline__ uint4 ld_nc_u4(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
  return r;
}
// Read-modify-write streams (p, m, v): evict-first loads and stores.
__device__ __forceinline__ uint4 ld_cs_u4(const void* p) {
  uint4 r;
  asm volatile("ld.global.cs.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
  return r;
}
__device__ __forceinline__ uint2 ld_cs_u2(const void* p) {
  uint2 r;
  asm volatile("ld.global.cs.v2.u32 {%0,%1}, [%2];" : "=r"(r.x), "=r"(r.y) : "l"(p));
  return r;
}
__device__ __forceinline__ uint32_t ld_cs_u1(const void* p) {
  uint32_t r;
  asm volatile("ld.global.cs.u32 %0, [%1];" : "=r"(r) : "l"(p));
  return r;
}
__device__ __forceinline__ void st_cs_u4(void* p, uint4 v) {
  asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};"
               :: "l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w) : "memory");
}
__device__ __forceinline__ void st_cs_u2(void* p, uint2 v) {
  asm volatile("st.global.cs.v2.u32 [%0], {%1,%2};" :: "l"(p), "r"(v.x), "r"(v.y) : "memory");
}
__device__ __forceinline__ void st_cs_u1(void* p, uint32_t v) {
  asm volatile("st.global.cs.u32 [%0], %1;" :: "l"(p), "r"(v) : "memory");
}

}  // namespace psopt
