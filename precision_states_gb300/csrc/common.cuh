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
  float v_scale;       // stored v code holds v / v_scale (power of two)
  float v_inv_scale;   // 1 / v_scale, exact
  uint32_t a32;        // kA32* bits: the FP32 streams whose base is 32-byte aligned
  uint32_t pad;
};
static_assert(sizeof(TensorDesc) == 64, "TensorDesc layout");
enum : uint32_t { kA32P = 1u, kA32M = 2u, kA32V = 4u };
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

// One chunk as the norm kernel reads it: the address of its first gradient
// element (the tensor's base plus the chunk start) and its element count.
// Resolved when the table is built, so a chunk costs one 16-byte load.
struct NormChunk {
  const void* ptr;
  uint32_t len;
  uint32_t pad;
};
static_assert(sizeof(NormChunk) == 16, "NormChunk layout");

// Everything a step kernel needs besides the tables.
struct StepArgs {
  const TensorDesc* tensors;
  const opt_chunk* tiles;             // the step's work table (kTileElems per entry)
  int64_t tile_begin, tile_end;       // this bucket's range of it
  opt_step_scalars sc;
  uint32_t step32;
  uint32_t rk[20];                    // Philox round keys of the seed (philox_round_keys)
  unsigned long long neg_zero2;       // -0.0 in both f32 lanes (kNegZero2), for mulr2
  const opt_norm_result* d_norm;      // NULL: no clipping
  unsigned long long* unchanged;      // NULL: do not count
  int reset;                          // nonzero: start from zero moments
  int* err;                           // kernel error flags (OPT_FLAG_*)
  const opt_step_scalars* d_sc;       // non-NULL: use these scalars (device memory), not sc
  unsigned long long wait_ns;         // limit of each wait of the staged step (opt_plan_set_wait_limit)
  int drill;                          // nonzero: the staged step's waits run out on purpose
  unsigned long long* dyn;            // the FP32 AdamW step's tile counter and finished-warp count
                                      // (0 between launches: the last warp resets them)
};

// A short bucket passed whole in a kernel's parameters (the short-list step,
// step_small.cu): at most kSmallMaxTensors non-empty tensors in list order,
// each with its descriptor, its index in the plan's list and the end of its
// tiles in the bucket (tiles of kTileElems; an inclusive prefix sum).
constexpr int kSmallMaxTensors = 8;
constexpr int64_t kSmallMaxTiles = 4096;
struct SmallList {
  int n;
  uint32_t tensor[kSmallMaxTensors];
  int64_t tile_end[kSmallMaxTensors];
  TensorDesc td[kSmallMaxTensors];
};

// ------------------------------------------------------------- bit views
__device__ __forceinline__ uint32_t f2u(float x) { return __float_as_uint(x); }
__device__ __forceinline__ float u2f(uint32_t x) { return __uint_as_float(x); }

// ------------------------------------------------- packed f32x2 arithmetic
// sm_100+ executes two independent IEEE fp32 operations per instruction on a
// pair of lanes held in one 64-bit register; each lane rounds exactly as the
// scalar operation would.
typedef unsigned long long f2_t;   // two fp32 lanes in one 64-bit register

__device__ __forceinline__ f2_t pk(float a, float b) {
  f2_t r;
  asm("mov.b64 %0, {%1,%2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void unpk(f2_t v, float& a, float& b) {
  asm("mov.b64 {%0,%1}, %2;" : "=f"(a), "=f"(b) : "l"(v));
}
__device__ __forceinline__ f2_t add2(f2_t a, f2_t b) {
  f2_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ f2_t sub2(f2_t a, f2_t b) {
  f2_t r;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ f2_t mul2(f2_t a, f2_t b) {
  f2_t r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ f2_t fma2(f2_t a, f2_t b, f2_t c) {
  f2_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}

// The rounded products a*b of both lanes, written as fma(a, b, z) with z
// -0.0 in both lanes: adding -0 changes no bit (the sign of a zero product
// included), and the result of a fused multiply-add cannot be fused again.
// For products that feed an addition whose result must be the definition's
// bits.  Measured on GB300: a packed mul.rn.f32x2 used once, by an
// add.rn.f32x2, was fused into it in spite of the .rn (and of --fmad=false),
// so that about half of the sums b1 m + (1 - b1) g of BF16 inputs came out
// 1 ulp or more off.  z must come from outside the compiler's view (a kernel
// argument): with a literal -0 the fma was turned back into a multiply
// and fused all the same.
constexpr unsigned long long kNegZero2 = 0x8000000080000000ull;
__device__ __forceinline__ f2_t mulr2(f2_t a, f2_t b, unsigned long long z) {
  f2_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(z));
  return r;
}

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

// The same generator with its ten round keys given: rk[2r], rk[2r+1] are
// the key words of round r (the seed advanced r times by the Weyl
// increments).  They depend on the seed alone, so a kernel receives them
// formed once (philox_round_keys on the host) in its arguments, where each
// round reads them as operands instead of recomputing them per call.
__device__ __forceinline__ uint4 philox10_rk(uint4 c, const uint32_t* rk) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    const uint32_t lo0 = 0xD2511F53u * c.x, hi0 = __umulhi(0xD2511F53u, c.x);
    const uint32_t lo1 = 0xCD9E8D57u * c.z, hi1 = __umulhi(0xCD9E8D57u, c.z);
    c = make_uint4(hi1 ^ c.y ^ rk[2 * r], lo1, hi0 ^ c.w ^ rk[2 * r + 1], lo0);
  }
  return c;
}
__device__ __forceinline__ uint4 draw_words_rk(uint64_t q, uint32_t tensor, uint32_t step32, const uint32_t* rk) {
  return philox10_rk(make_uint4((uint32_t)q, (uint32_t)(q >> 32), tensor, step32), rk);
}

// Round keys of Philox4x32-10 for a 64-bit seed (host side).
inline void philox_round_keys(uint64_t seed, uint32_t rk[20]) {
  uint32_t k0 = (uint32_t)seed, k1 = (uint32_t)(seed >> 32);
  for (int r = 0; r < 10; ++r) {
    if (r) { k0 += 0x9E3779B9u; k1 += 0xBB67AE85u; }
    rk[2 * r] = k0;
    rk[2 * r + 1] = k1;
  }
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

// ------------------------------------------------- small-grid rounding core
// Stochastic rounding of a (finite, 0 <= a below the grid's largest value)
// onto a grid with P fraction bits whose binades start at 2^EMIN (constant
// spacing 2^(EMIN-P) below it); returns the code (binade index << P | the P
// fraction bits, counting the spacing below 2^EMIN as binade 0).
// The rule ("When Small Updates Disappear", sec. 6.1, applied at the target
// grid's spacing): round up iff the 16 bits just below the kept bits plus the
// 16-bit draw carry past 2^16.  In the grid's normal range the kept bits are
// the top P of the fp32 mantissa, so this is the BF16 bit trick at a shifted
// position: add r16 << (7 - P) to the word and drop the low 23 - P bits (the
// bits below the 16 examined cannot carry into them).  Below 2^EMIN the
// spacing is constant: adding 2^EMIN with round-toward-zero moves a into the
// first binade without disturbing any of the 16 examined bits (they all lie
// at or above that binade's last place), and the same trick applies.
template <int P, int EMIN>
__device__ __forceinline__ uint32_t grid_code_sr(float a, uint32_t r16) {
  constexpr uint32_t kMinNormal = (uint32_t)(EMIN + 127) << 23;   // the word of 2^EMIN
  constexpr int kDrop = 23 - P;
  const bool sub = f2u(a) < kMinNormal;
  const float y = sub ? __fadd_rz(a, u2f(kMinNormal)) : a;
  const uint32_t w = (f2u(y) + (r16 << (kDrop - 16))) >> kDrop;  // biased exponent << P | fraction
  return w - ((uint32_t)(EMIN + 126) << P) - (sub ? (1u << P) : 0u);
}

// ------------------------------------------------------- E4M3 (FP8) codec
// Decode: as if normal with exponent field max(E, 1), minus 2^-6 for the
// subnormal codes (E = 0), which gives k 2^-9 exactly.
__device__ __forceinline__ float e4m3_dec(uint32_t c) {
  const uint32_t mag = c & 0x7Fu;
  const uint32_t E = mag >> 3;
  float r = u2f(((max(E, 1u) + 120u) << 23) | ((mag & 7u) << 20));
  if (E == 0u) r = __fsub_rn(r, 0.015625f);
  if (mag == 0x7Fu) r = u2f(0x7FC00000u);
  return (c & 0x80u) ? -r : r;
}

// Nearest (saturating) conversion of two values by the hardware converter:
// the first operand lands in the upper byte.
__device__ __forceinline__ uint32_t e4m3x2_rn(float lo, float hi) {
  unsigned short r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return (uint32_t)r;
}

// Stochastic: sign kept, magnitudes at or above 448 (and Inf) saturate, NaN
// stays NaN.  Branch-free: 448 itself lies on the grid, so clamping to it
// yields its code whatever the draw.
__device__ __forceinline__ uint32_t e4m3_enc_sr(float x, uint32_t r16) {
  const uint32_t sign = (f2u(x) >> 24) & 0x80u;
  const uint32_t code = sign | min(grid_code_sr<3, -6>(fminf(fabsf(x), 448.0f), r16), 0x7Eu);
  return (x != x) ? 0x7Fu : code;
}

// Decode of two E4M3 codes (the low byte is the first element) by the
// hardware converter to f16, then f16 to fp32; every E4M3 value, NaN
// included, is an f16 value, so both steps are exact.
__device__ __forceinline__ float h2f(unsigned short h) {
  float f;
  asm("cvt.f32.f16 %0, %1;" : "=f"(f) : "h"(h));
  return f;
}
__device__ __forceinline__ void e4m3x2_dec(uint32_t pair16, float& first, float& second) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"((unsigned short)pair16));
  first = h2f((unsigned short)(h2 & 0xFFFFu));
  second = h2f((unsigned short)(h2 >> 16));
}

// ------------------------------------------------ unsigned E2M2 (FP4) codec
// Decode: codes 0-3 are k/4 = (1 + k/4) - 1; codes 4-15 are normal.
__device__ __forceinline__ float e2m2_dec(uint32_t c) {
  const uint32_t E = c >> 2;
  const float r = u2f(((max(E, 1u) + 126u) << 23) | ((c & 3u) << 21));
  return E == 0u ? __fsub_rn(r, 1.0f) : r;
}

// Decode of two E2M2 codes held in the low 4 bits of the two bytes of
// pair16 (low byte first): as FP6 E3M2 codes (exponent field 0-3) they are
// the E2M2 values over 4, which the hardware converts exactly to f16.
// e2m2x2_dec_q returns those quarter values (callers fold the factor 4 into
// a power-of-two scale), e2m2x2_dec the E2M2 values themselves.
__device__ __forceinline__ void e2m2x2_dec_q(uint32_t pair16, float& first, float& second) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e3m2x2 %0, %1;" : "=r"(h2) : "h"((unsigned short)pair16));
  first = h2f((unsigned short)(h2 & 0xFFFFu));
  second = h2f((unsigned short)(h2 >> 16));
}
__device__ __forceinline__ void e2m2x2_dec(uint32_t pair16, float& first, float& second) {
  e2m2x2_dec_q(pair16, first, second);
  first = __fmul_rn(first, 4.0f);
  second = __fmul_rn(second, 4.0f);
}

// The converters see E2M2 values over 4 (the E3M2 grid) clamped to
// [0, 7/4]: NaN stores 7 (fminf returns its non-NaN operand), negative
// values store 0, values at or above 7 saturate.  Callers pass x/4.
__device__ __forceinline__ float e2m2_clamp_q(float x4) { return fmaxf(fminf(x4, 1.75f), 0.0f); }
// The step's v is never negative (b2 v + (1 - b2) g^2 with v, b2, 1 - b2 >= 0,
// or NaN), so there only the upper clamp is needed.
template <bool NONNEG>
__device__ __forceinline__ float e2m2_clamp_q(float x4) { return NONNEG ? fminf(x4, 1.75f) : e2m2_clamp_q(x4); }

// Nearest, two values at a time: unsigned E2M2 is the FP6 E3M2 grid scaled
// by 4 (E3M2 subnormals k/16 are E2M2's k/4 over 4; its binades with
// exponent field 1-3 are E2M2's), so the hardware's nearest-even E3M2
// conversion of x/4 (exact scaling), for 0 <= x <= 7, yields the E2M2 code
// in the low bits of each byte (sign and exponent bits above are 0).
// Arguments are the quarter values lo4 = lo/4, hi4 = hi/4; returns the pair
// (lo | hi << 8).
template <bool NONNEG = false>
__device__ __forceinline__ uint32_t e2m2x2_rn_q(float lo4, float hi4) {
  unsigned short r;
  asm("cvt.rn.satfinite.e3m2x2.f32 %0, %1, %2;"
      : "=h"(r) : "f"(e2m2_clamp_q<NONNEG>(hi4)), "f"(e2m2_clamp_q<NONNEG>(lo4)));
  return (uint32_t)r;
}

// ----------------------------------------- paired hardware encoders
// Blackwell's converters round two fp32 values per instruction, and their
// stochastic forms (cvt.rs, with a 32-bit operand of random bits) apply the
// rule the software encoders above apply: a lane rounds away from zero
// exactly when its 16 dropped bits plus its 16-bit draw carry past 2^16.
// Lane layout: the BF16 form takes bits 31:16 for the upper result and bits
// 15:0 for the lower; the four-lane FP8/FP6 forms were matched bit for bit
// to the software rule (every code of 2^21 seeded values, NaN, Inf,
// saturation, subnormals and negatives included) in their second and fourth
// lanes only, which take bits 31:16 and 15:0 -- so the first and third lanes
// are fed zeros and their results dropped.  Each encoder returns a pair
// word with `lo` in the low half (16-bit codes) or the low byte (8-bit).
// NaN inputs, rare, take the software encoders so that NaN codes stay those
// of the codec definitions (the converters emit a canonical NaN).
// The NaN paths, out of line: they are rare, and inlined they would hold
// registers across the whole update.
static __device__ __noinline__ uint32_t bf16x2_rn_soft(float lo, float hi) {
  return bf16_enc_rn(lo) | (bf16_enc_rn(hi) << 16);
}
static __device__ __noinline__ uint32_t bf16x2_sr_soft(float lo, float hi, uint32_t rbits) {
  return bf16_enc_sr(lo, rbits & 0xFFFFu) | (bf16_enc_sr(hi, rbits >> 16) << 16);
}
static __device__ __noinline__ uint32_t e4m3x2_sr_soft(float lo, float hi, uint32_t rbits) {
  return e4m3_enc_sr(lo, rbits & 0xFFFFu) | (e4m3_enc_sr(hi, rbits >> 16) << 8);
}

__device__ __forceinline__ uint32_t bf16x2_rn(float lo, float hi) {
  uint32_t d;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  if (__builtin_expect(lo != lo || hi != hi, 0)) d = bf16x2_rn_soft(lo, hi);
  return d;
}

// rbits: bits 15:0 draw for lo, bits 31:16 for hi.
__device__ __forceinline__ uint32_t bf16x2_sr(float lo, float hi, uint32_t rbits) {
  uint32_t d;
  asm("cvt.rs.bf16x2.f32 %0, %1, %2, %3;" : "=r"(d) : "f"(hi), "f"(lo), "r"(rbits));
  if (__builtin_expect(lo != lo || hi != hi, 0)) d = bf16x2_sr_soft(lo, hi, rbits);
  return d;
}

template <bool SR>
__device__ __forceinline__ uint32_t bf16x2_enc(float lo, float hi, uint32_t rbits) {
  return SR ? bf16x2_sr(lo, hi, rbits) : bf16x2_rn(lo, hi);
}

// E4M3, stochastic, saturating: the pair (lo | hi << 8).
__device__ __forceinline__ uint32_t e4m3x2_sr(float lo, float hi, uint32_t rbits) {
  uint32_t d;
  asm("cvt.rs.satfinite.e4m3x4.f32 %0, {%1, %2, %3, %4}, %5;"
      : "=r"(d) : "f"(0.0f), "f"(hi), "f"(0.0f), "f"(lo), "r"(rbits));
  uint32_t pair = __byte_perm(d, 0u, 0x4420);          // byte 0 (lo), byte 2 (hi)
  if (__builtin_expect(lo != lo || hi != hi, 0)) pair = e4m3x2_sr_soft(lo, hi, rbits);
  return pair;
}
// The same, as the converter leaves it: lo in byte 0, hi in byte 2, so that
// the step can gather eight codes with two byte permutes (one per 4-element
// word) instead of one per pair and the shifts.  Bytes 1 and 3 come from
// the lanes fed zeros and are never read.
__device__ __forceinline__ uint32_t e4m3x2_sr_wide(float lo, float hi, uint32_t rbits) {
  uint32_t d;
  asm("cvt.rs.satfinite.e4m3x4.f32 %0, {%1, %2, %3, %4}, %5;"
      : "=r"(d) : "f"(0.0f), "f"(hi), "f"(0.0f), "f"(lo), "r"(rbits));
  if (__builtin_expect(lo != lo || hi != hi, 0)) d = __byte_perm(e4m3x2_sr_soft(lo, hi, rbits), 0u, 0x4140);
  return d;
}

// Unsigned E2M2, stochastic: the E3M2 grid of the quarter values (as in
// e2m2x2_rn_q), after the clamp (7/4 lies on the grid, so no draw moves a
// saturated value).  The pair (lo | hi << 8), codes 0-15.
template <bool NONNEG = false>
__device__ __forceinline__ uint32_t e2m2x2_sr_q(float lo4, float hi4, uint32_t rbits) {
  uint32_t d;
  asm("cvt.rs.satfinite.e3m2x4.f32 %0, {%1, %2, %3, %4}, %5;"
      : "=r"(d)
      : "f"(0.0f), "f"(e2m2_clamp_q<NONNEG>(hi4)), "f"(0.0f), "f"(e2m2_clamp_q<NONNEG>(lo4)), "r"(rbits));
  return __byte_perm(d, 0u, 0x4420);
}
// The same, as the converter leaves it: lo in byte 0, hi in byte 2 (bytes 1
// and 3, from the lanes fed zeros, are never read).
template <bool NONNEG = false>
__device__ __forceinline__ uint32_t e2m2x2_sr_wide_q(float lo4, float hi4, uint32_t rbits) {
  uint32_t d;
  if constexpr (NONNEG) {
    // v >= 0 (or NaN): convert unclamped and clamp the codes instead, both
    // at once as 16-bit lanes (each lane holds one code, its upper byte from
    // a lane fed zero).  The converter saturates at the E3M2 maximum, above
    // 7/4, and a stochastic rounding of a value at or above 7/4 lands on a
    // code of 7/4 or above: min(code, 15) is the code of the clamped value.
    asm("cvt.rs.satfinite.e3m2x4.f32 %0, {%1, %2, %3, %4}, %5;"
        : "=r"(d) : "f"(0.0f), "f"(hi4), "f"(0.0f), "f"(lo4), "r"(rbits));
    asm("min.u16x2 %0, %1, %2;" : "=r"(d) : "r"(d), "r"(0x000F000Fu));
  } else {
    asm("cvt.rs.satfinite.e3m2x4.f32 %0, {%1, %2, %3, %4}, %5;"
        : "=r"(d)
        : "f"(0.0f), "f"(e2m2_clamp_q<NONNEG>(hi4)), "f"(0.0f), "f"(e2m2_clamp_q<NONNEG>(lo4)), "r"(rbits));
  }
  return d;
}

// ------------------------------------------ arithmetic for the update term
// The parameter update is not a stored code, so it may use the hardware
// approximations (relative error about 2^-22, far inside the tolerance the
// update is checked to); the moments, which are, use exact fp32 operations.
// The division is div.approx (a reciprocal, then a multiply; its
// denominator sqrt(v_hat) + eps lies far inside the range where that is
// accurate) or div.full, whichever measured faster for the state
// combination: against div.full, div.approx made stochastic E2M2 states
// 2 % faster, E4M3 1 %, the Llama-3-8B FP32-state step 0.5 %, and both
// BF16-v steps 2 % slower.
__device__ __forceinline__ float sqrt_approx(float x) {
  float r;
  asm("sqrt.approx.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}
__device__ __forceinline__ float div_approx(float a, float b) {
  float r;
  asm("div.approx.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ float rcp_approx(float x) {
  float r;
  asm("rcp.approx.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}
__device__ __forceinline__ float div_full(float a, float b) {
  float r;
  asm("div.full.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
  return r;
}

// -------------------------------------------------- streaming memory access
// Read-only gradient stream: non-coherent path, no L1 allocation.
__device__ __forceinline__ uint4 ld_nc_u4(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
  return r;
}
// 32 bytes in one evict-first load (sm_100+); the address must be 32-byte
// aligned.
__device__ __forceinline__ void ld_cs_v8(const void* p, uint32_t* r) {
  asm volatile("ld.global.cs.v8.u32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
                 "=r"(r[7])
               : "l"(p));
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
