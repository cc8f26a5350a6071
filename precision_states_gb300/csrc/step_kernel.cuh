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
// written once ("When Small Updates Disappear", sec. 8.1); both directions
// go through the hardware converters, two values per instruction (their
// stochastic forms apply the same 16-bit carry rule as the codec
// definitions; see the paired encoders in common.cuh).
//
// Layout: a persistent grid strides over the bucket's tiles of 2048 elements
// (a finer table than the norm's chunks, so that short lists and lists of
// uneven tensors still spread evenly over every SM); in a tile thread t owns
// the 8 consecutive elements 8t .. 8t+7, moved with 16-byte
// streaming loads and stores (p, m, v, m2: evict-first; g: read-only path).
// The group start is a multiple of 8 elements and every base pointer is
// 16-byte aligned, so each stream's vector is naturally aligned (E4M3: 8
// bytes, E2M2: 4 bytes).  The one ragged group of a tensor is loaded and
// stored element by element.
//
// The kernel is bound by HBM latency x bytes in flight, so each thread runs a
// two-deep software pipeline: the raw words of its group in the CTA's next
// tile are requested before the current group is decoded, updated, encoded
// and stored.
//
// Stochastic-rounding draws: two Philox4x32-10 calls per group (counters
// q = e0/4 and e0/4 + 1), so each draw depends only on (seed, step, tensor,
// element); the round keys come formed in the kernel arguments.
#pragma once

#include "common.cuh"
#include "internal.h"

namespace psopt {

constexpr int kStepThreads = 256;

// Launch shape per instantiation, chosen by measurement on GB300 (GPT-2
// list, 124M params):
// - CTAs per SM: 2 (<= 128 registers, no spills) everywhere, except the
//   nearest-rounding E4M3 and E2M2 v states with BF16 gradients.  Those fit
//   3 CTAs (<= 80 registers) without spilling, and the extra warps lift them
//   from 0.93 / 0.90 to 1.00 of the measured copy bandwidth.  Every other
//   instantiation spills at 3 CTAs and runs slower there.
// - Grid: persistent (as many CTAs as are resident), CTA c taking tiles
//   c, c + G, ... -- except for AdEMAMix, whose five fp32 streams ran faster
//   with one CTA per tile here (0.993 against 0.944 of measured).  The
//   FP32-state steps (AdamW and AdEMAMix) now run step_dyn_kernel
//   (step_dyn.cuh) instead, whose warps take tiles from a counter, and the
//   stochastic and BF16-v states are staged (below); this kernel runs the
//   nearest E4M3 / E2M2 states (3 CTAs per SM with BF16 gradients).
// - Staging: the low-precision AdamW instantiations with stochastic rounding,
//   and BF16 v with nearest rounding, take their input tiles through shared
//   memory from a producer warp's bulk copies (step_bulk.cuh): 0.956 / 0.917
//   / 0.869 -> 0.980 / 0.970 / 0.948 (stochastic BF16 / E4M3 / E2M2 v) and
//   0.964 -> 0.989 (nearest BF16 v).  Nearest E4M3 and E2M2 stay on the
//   3-CTA register pipeline, which measured equal or better.
// - Entry lookahead: where registers allow (2 CTAs per SM), a thread
//   requests the table entry of the tile after its next one a whole tile
//   ahead, so that only the descriptor load stands between a tile's entry
//   and its data requests.
template <int GT, int COMBO, int ALGO, bool SR>
struct StepShape {
  static constexpr int kMinBlocks =
      (GT == OPT_BF16 && !SR && (COMBO == SC_BF16_E4M3 || COMBO == SC_BF16_E2M2)) ? 3 : 2;
  static constexpr bool kPersistent = ALGO != ALGO_ADEMAMIX;
  static constexpr bool kBulk = ALGO == ALGO_ADAMW && step_is_staged(COMBO, SR);
  static constexpr bool kLookahead = kPersistent && kMinBlocks == 2;
};

template <int COMBO>
struct Combo;
template <> struct Combo<SC_F32>       { static constexpr int M = OPT_F32,  V = OPT_F32;  };
template <> struct Combo<SC_BF16_BF16> { static constexpr int M = OPT_BF16, V = OPT_BF16; };
template <> struct Combo<SC_BF16_E4M3> { static constexpr int M = OPT_BF16, V = OPT_E4M3; };
template <> struct Combo<SC_BF16_E2M2> { static constexpr int M = OPT_BF16, V = OPT_E2M2; };

// Raw 32-bit words of one 8-element group, as they sit in memory.
template <int GT, int COMBO, int ALGO>
struct Frag {
  static constexpr int MD = Combo<COMBO>::M, VD = Combo<COMBO>::V;
  static constexpr int NG = GT == OPT_BF16 ? 4 : 8;
  static constexpr int NM = MD == OPT_F32 ? 8 : 4;
  static constexpr int NV = VD == OPT_F32 ? 8 : VD == OPT_BF16 ? 4 : VD == OPT_E4M3 ? 2 : 1;
  static constexpr int NM2 = ALGO == ALGO_ADEMAMIX ? 8 : 1;
  uint32_t p[8], g[NG], m[NM], v[NV], m2[NM2];
};

__device__ __forceinline__ void put4(uint32_t* w, uint4 x) { w[0] = x.x; w[1] = x.y; w[2] = x.z; w[3] = x.w; }

// Eight consecutive FP32 words of a read-modify-write stream at an
// 8-element group: one 32-byte load when the stream's base is 32-byte
// aligned (then so is every group, which starts a multiple of 8 elements
// in), else two 16-byte loads.  Measured on GB300 (bench CUDA events):
//  - AdamW, FP32 p, m, v: the Llama-3-8B step (norm + step) went from 33.54
//    to 33.17 ms; the 740-tensor list and the low-precision states did not
//    change.  32-byte stores gained nothing and slowed the norm that
//    follows, so stores stay 16 bytes.
//  - AdEMAMix on the GPT-2 list (one CTA per tile, FP32 gradients): 32-byte
//    loads cost 0.4 %, and 6 % with the gradient stream included, so the
//    wide loads are AdamW's only and never the gradient's.
__device__ __forceinline__ void ld_cs_x8(const void* p, bool a32, uint32_t* r) {
  if (a32) {
    ld_cs_v8(p, r);
  } else {
    put4(r, ld_cs_u4(p));
    put4(r + 4, ld_cs_u4(static_cast<const char*>(p) + 16));
  }
}

// Element j of a word array holding `bits`-wide codes (16, 8 or 4 bits).
template <int BITS>
__device__ __forceinline__ uint32_t code_at(const uint32_t* w, int j) {
  if constexpr (BITS == 32) {
    return w[j];
  } else {
    constexpr int PER = 32 / BITS;
    return (w[j / PER] >> (BITS * (j % PER))) & ((1u << BITS) - 1u);
  }
}

// Loads the group's words; with `reset` the moments are not read: they
// start from zero (every format's code 0 is the value 0).
template <int GT, int COMBO, int ALGO>
__device__ __forceinline__ void load_full(const TensorDesc& td, int64_t e0, bool reset,
                                          Frag<GT, COMBO, ALGO>& f) {
  using F = Frag<GT, COMBO, ALGO>;
  const uint32_t a32 = ALGO == ALGO_ADAMW ? td.a32 : 0u;
  ld_cs_x8(td.p + e0, a32 & kA32P, f.p);
  if constexpr (F::NG == 4) {
    put4(f.g, ld_nc_u4(static_cast<const uint16_t*>(td.g) + e0));
  } else {
    put4(f.g, ld_nc_u4(static_cast<const float*>(td.g) + e0));
    put4(f.g + 4, ld_nc_u4(static_cast<const float*>(td.g) + e0 + 4));
  }
  if (reset) {
#pragma unroll
    for (int k = 0; k < F::NM; ++k) f.m[k] = 0u;
#pragma unroll
    for (int k = 0; k < F::NV; ++k) f.v[k] = 0u;
#pragma unroll
    for (int k = 0; k < F::NM2; ++k) f.m2[k] = 0u;
    return;
  }
  if constexpr (F::NM == 8) {
    ld_cs_x8(static_cast<const float*>(td.m) + e0, a32 & kA32M, f.m);
  } else {
    put4(f.m, ld_cs_u4(static_cast<const uint16_t*>(td.m) + e0));
  }
  if constexpr (F::NV == 8) {
    ld_cs_x8(static_cast<const float*>(td.v) + e0, a32 & kA32V, f.v);
  } else if constexpr (F::NV == 4) {
    put4(f.v, ld_cs_u4(static_cast<const uint16_t*>(td.v) + e0));
  } else if constexpr (F::NV == 2) {
    const uint2 w = ld_cs_u2(static_cast<const uint8_t*>(td.v) + e0);
    f.v[0] = w.x;
    f.v[1] = w.y;
  } else {
    f.v[0] = ld_cs_u1(static_cast<const uint8_t*>(td.v) + (e0 >> 1));
  }
  if constexpr (ALGO == ALGO_ADEMAMIX) {
    put4(f.m2, ld_cs_u4(td.m2 + e0));
    put4(f.m2 + 4, ld_cs_u4(td.m2 + e0 + 4));
  }
}

// The ragged group of a tensor: element-wise loads packed into the same
// words, zero past the end (an E2M2 byte is read whole: both nibbles belong
// to the tensor's ceil(n/2) bytes).
template <int GT, int COMBO, int ALGO>
__device__ __forceinline__ void load_partial(const TensorDesc& td, int64_t e0, int cnt, bool reset,
                                             Frag<GT, COMBO, ALGO>& f) {
  using F = Frag<GT, COMBO, ALGO>;
#pragma unroll
  for (int k = 0; k < 8; ++k) f.p[k] = 0u;
#pragma unroll
  for (int k = 0; k < F::NG; ++k) f.g[k] = 0u;
#pragma unroll
  for (int k = 0; k < F::NM; ++k) f.m[k] = 0u;
#pragma unroll
  for (int k = 0; k < F::NV; ++k) f.v[k] = 0u;
#pragma unroll
  for (int k = 0; k < F::NM2; ++k) f.m2[k] = 0u;
  // unrolled with an exit, so that the word arrays stay in registers
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    if (j >= cnt) break;
    const int64_t e = e0 + j;
    f.p[j] = f2u(td.p[e]);
    if constexpr (F::NG == 8) f.g[j] = f2u(static_cast<const float*>(td.g)[e]);
    else f.g[j >> 1] |= (uint32_t)static_cast<const uint16_t*>(td.g)[e] << (16 * (j & 1));
    if (reset) continue;
    if constexpr (F::NM == 8) f.m[j] = f2u(static_cast<const float*>(td.m)[e]);
    else f.m[j >> 1] |= (uint32_t)static_cast<const uint16_t*>(td.m)[e] << (16 * (j & 1));
    if constexpr (F::NV == 8) {
      f.v[j] = f2u(static_cast<const float*>(td.v)[e]);
    } else if constexpr (F::NV == 4) {
      f.v[j >> 1] |= (uint32_t)static_cast<const uint16_t*>(td.v)[e] << (16 * (j & 1));
    } else if constexpr (F::NV == 2) {
      f.v[j >> 2] |= (uint32_t)static_cast<const uint8_t*>(td.v)[e] << (8 * (j & 3));
    } else if ((j & 1) == 0) {
      uint32_t byte = static_cast<const uint8_t*>(td.v)[e >> 1];
      if (j + 1 >= cnt) byte &= 0xFu;
      f.v[0] |= byte << (4 * j);
    }
    if constexpr (ALGO == ALGO_ADEMAMIX) f.m2[j] = f2u(td.m2[e]);
  }
}

template <int GT, int COMBO, int ALGO, bool SR, int N = 8>
__device__ __forceinline__ uint32_t update_store(const TensorDesc& td, int64_t e0, int cnt,
                                                 const Frag<GT, COMBO, ALGO>& f, float coef,
                                                 const opt_step_scalars& sc, uint32_t tensor,
                                                 const uint32_t* rk, uint32_t step32, bool count,
                                                 unsigned long long neg_zero2) {
  using F = Frag<GT, COMBO, ALGO>;
  constexpr int MD = F::MD, VD = F::VD;
  constexpr bool LOWP = COMBO != SC_F32;
  constexpr int VBITS = VD == OPT_F32 ? 32 : VD == OPT_BF16 ? 16 : VD == OPT_E4M3 ? 8 : 4;
  // N: the elements of the group the lanes hold, 8, or 4 with FP32 states
  // (the short-list kernel's quarter groups: only elements 0..3 are touched)
  static_assert(N == 8 || (N == 4 && COMBO == SC_F32), "four-element groups: FP32 states only");

  uint32_t words[8];
  if constexpr (LOWP && SR) {
    const uint4 d0 = draw_words_rk((uint64_t)e0 >> 2, tensor, step32, rk);
    const uint4 d1 = draw_words_rk(((uint64_t)e0 >> 2) + 1, tensor, step32, rk);
    words[0] = d0.x; words[1] = d0.y; words[2] = d0.z; words[3] = d0.w;
    words[4] = d1.x; words[5] = d1.y; words[6] = d1.z; words[7] = d1.w;
  }

  // decode to fp32 (exact)
  float g[8], m[8], v[8];
#pragma unroll
  for (int j = 0; j < N; ++j) {
    g[j] = GT == OPT_BF16 ? bf16_dec(code_at<16>(f.g, j)) : u2f(f.g[j]);
    m[j] = MD == OPT_F32 ? u2f(f.m[j]) : bf16_dec(code_at<16>(f.m, j));
    if constexpr (VD == OPT_F32) v[j] = u2f(f.v[j]);
    if constexpr (VD == OPT_BF16) v[j] = bf16_dec(code_at<16>(f.v, j));
  }
  if constexpr (VD == OPT_E4M3) {
    // byte pairs straight from the loaded words
#pragma unroll
    for (int k = 0; k < 4; ++k)
      e4m3x2_dec((k & 1) ? (f.v[k >> 1] >> 16) : (f.v[k >> 1] & 0xFFFFu), v[2 * k], v[2 * k + 1]);
  }
  if constexpr (VD == OPT_E2M2) {
    // spread the nibbles into bytes: even elements, odd elements; decoded
    // as quarter values (the factor 4 joins v_scale below)
    const uint32_t even = f.v[0] & 0x0F0F0F0Fu, odd = (f.v[0] >> 4) & 0x0F0F0F0Fu;
#pragma unroll
    for (int k = 0; k < 4; ++k)
      e2m2x2_dec_q(__byte_perm(even, odd, (uint32_t)k | ((uint32_t)(4 + k) << 4)), v[2 * k], v[2 * k + 1]);
  }
  float pn[8], mnv[8], vnv[8], m2n[8], vs[8];
  if constexpr (StepShape<GT, COMBO, ALGO, SR>::kBulk && COMBO != SC_BF16_BF16) {
    // Stochastic E4M3 / E2M2 v, where the issue slots are the scarce
    // resource: everything from the decoded values to the value the v code
    // stores runs two elements per packed f32x2 instruction.  The moments
    // keep the scalar path's operations and order, each lane rounding as
    // the scalar operation does, so their bits are the definition's; the
    // products that feed an addition are mulr2, which no compiler fusion
    // can merge into it.  The update term is
    // p' = fma(-lr, u, p decay) with a reciprocal then a multiply for the
    // division.  Measured on GB300 (GPT-2 list, A/B/A/B), the packed update
    // term alone took stochastic E2M2 from 0.938-0.940 to 0.954-0.956 of
    // the measured copy bandwidth and E4M3 from 0.974 to 0.979-0.981; BF16 v
    // lost 0.15-0.35 % with it and the 3-CTA/SM nearest E4M3 / E2M2 kernels
    // spill with it, so they keep the scalar form.
    const float vsc = VD == OPT_E2M2 ? __fmul_rn(td.v_scale, 4.0f) : td.v_scale;
    const float vinv = VD == OPT_E2M2 ? __fmul_rn(td.v_inv_scale, 0.25f) : td.v_inv_scale;
    const f2_t vsc2 = pk(vsc, vsc), vinv2 = pk(vinv, vinv), c2 = pk(coef, coef);
    const f2_t b1p = pk(sc.beta1, sc.beta1), o1p = pk(sc.omb1, sc.omb1);
    const f2_t b2p = pk(sc.beta2, sc.beta2), o2p = pk(sc.omb2, sc.omb2);
    const f2_t ib1 = pk(sc.inv_bc1, sc.inv_bc1), ib2 = pk(sc.inv_bc2, sc.inv_bc2);
    const f2_t eps2 = pk(sc.eps, sc.eps), dec2 = pk(sc.decay, sc.decay), nlr2 = pk(-sc.lr, -sc.lr);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const f2_t ge = mul2(pk(g[2 * k], g[2 * k + 1]), c2);
      const f2_t mp = add2(mulr2(b1p, pk(m[2 * k], m[2 * k + 1]), neg_zero2), mulr2(o1p, ge, neg_zero2));
      const f2_t vp = add2(mulr2(b2p, mul2(pk(v[2 * k], v[2 * k + 1]), vsc2), neg_zero2),
                           mulr2(o2p, mul2(ge, ge), neg_zero2));
      unpk(mp, mnv[2 * k], mnv[2 * k + 1]);
      unpk(mul2(vp, vinv2), vs[2 * k], vs[2 * k + 1]);
      float a0, a1, d0, d1;
      unpk(mul2(vp, ib2), a0, a1);
      unpk(add2(pk(sqrt_approx(a0), sqrt_approx(a1)), eps2), d0, d1);
      const f2_t u = mul2(mul2(mp, ib1), pk(rcp_approx(d0), rcp_approx(d1)));
      unpk(fma2(nlr2, u, mul2(pk(u2f(f.p[2 * k]), u2f(f.p[2 * k + 1])), dec2)), pn[2 * k], pn[2 * k + 1]);
    }
  } else {
    // a low-precision v code holds v / v_scale (a power of two: exact; for
    // E2M2 the decoded quarter value times 4 v_scale, also a power of two)
    if constexpr (VD != OPT_F32) {
      const float vsc = VD == OPT_E2M2 ? __fmul_rn(td.v_scale, 4.0f) : td.v_scale;
#pragma unroll
      for (int j = 0; j < 8; ++j) v[j] = __fmul_rn(v[j], vsc);
    }
    // the moments: scalar IEEE fp32 operations in the order of the
    // definition (no contraction), so the values before rounding match bit
    // for bit
#pragma unroll
    for (int j = 0; j < N; ++j) {
      const float ge = __fmul_rn(g[j], coef);
      mnv[j] = __fadd_rn(__fmul_rn(sc.beta1, m[j]), __fmul_rn(sc.omb1, ge));
      vnv[j] = __fadd_rn(__fmul_rn(sc.beta2, v[j]), __fmul_rn(sc.omb2, __fmul_rn(ge, ge)));
      if constexpr (ALGO == ALGO_ADEMAMIX)
        m2n[j] = __fadd_rn(__fmul_rn(sc.beta3, u2f(f.m2[j])), __fmul_rn(sc.omb3, ge));
    }
    // the update term (not a stored code)
#pragma unroll
    for (int j = 0; j < N; ++j) {
      float num = __fmul_rn(mnv[j], sc.inv_bc1);
      if constexpr (ALGO == ALGO_ADEMAMIX) num = __fadd_rn(num, __fmul_rn(sc.alpha, m2n[j]));
      const float den = __fadd_rn(sqrt_approx(__fmul_rn(vnv[j], sc.inv_bc2)), sc.eps);
      const float u = COMBO == SC_BF16_BF16 ? div_full(num, den) : div_approx(num, den);
      pn[j] = __fsub_rn(__fmul_rn(u2f(f.p[j]), sc.decay), __fmul_rn(sc.lr, u));
    }
    // the value the v code stores: v / v_scale, exact (E2M2: a quarter of
    // it, the converters' E3M2 grid, in the same one multiplication)
    const float vinv = VD == OPT_E2M2 ? __fmul_rn(td.v_inv_scale, 0.25f) : td.v_inv_scale;
#pragma unroll
    for (int j = 0; j < N; ++j) vs[j] = VD == OPT_F32 ? vnv[j] : __fmul_rn(vnv[j], vinv);
  }
  // encode, two elements per converter instruction: pair k holds elements
  // 2k (low half / low byte) and 2k+1 -- for stochastic E4M3 / E2M2 v in
  // bytes 0 and 2, as the four-lane converter leaves them (WIDE), so that
  // the store gathers them with a few byte permutes.  Element j's m draw is
  // the low half of draw word j and its v draw the high half, so the
  // random-bits operand of pair k gathers those halves of words 2k and 2k+1.
  constexpr bool WIDE = SR && (VD == OPT_E4M3 || VD == OPT_E2M2);
  constexpr int HI = WIDE ? 16 : 8;            // bit position of element 2k+1 in an 8-bit-code pair
  uint32_t mpair[4], vpair[4];
#pragma unroll
  for (int k = 0; k < N / 2; ++k) {
    const uint32_t rm = SR ? __byte_perm(words[2 * k], words[2 * k + 1], 0x5410) : 0u;
    const uint32_t rv = SR ? __byte_perm(words[2 * k], words[2 * k + 1], 0x7632) : 0u;
    const float v0 = vs[2 * k], v1 = vs[2 * k + 1];
    if constexpr (MD == OPT_BF16) mpair[k] = bf16x2_enc<SR>(mnv[2 * k], mnv[2 * k + 1], rm);
    if constexpr (VD == OPT_BF16) vpair[k] = bf16x2_enc<SR>(v0, v1, rv);
    if constexpr (VD == OPT_E4M3) vpair[k] = SR ? e4m3x2_sr_wide(v0, v1, rv) : e4m3x2_rn(v0, v1);
    if constexpr (VD == OPT_E2M2) vpair[k] = SR ? e2m2x2_sr_wide_q<true>(v0, v1, rv) : e2m2x2_rn_q<true>(v0, v1);
  }
  // code of element j in the pair words
  auto vcode_at = [&](int j) -> uint32_t {
    if constexpr (VD == OPT_F32) return f2u(vnv[j]);
    else if constexpr (VD == OPT_BF16) return (vpair[j >> 1] >> (16 * (j & 1))) & 0xFFFFu;
    else return (vpair[j >> 1] >> (HI * (j & 1))) & 0xFFu;
  };
  uint32_t same = 0;
  if (count) {
#pragma unroll
    for (int j = 0; j < N; ++j)
      same += (j < cnt && vcode_at(j) == (VBITS == 32 ? f.v[j] : code_at<VBITS>(f.v, j))) ? 1u : 0u;
  }

  if (N == 8 && cnt == 8) {
    st_cs_u4(td.p + e0, make_uint4(f2u(pn[0]), f2u(pn[1]), f2u(pn[2]), f2u(pn[3])));
    st_cs_u4(td.p + e0 + 4, make_uint4(f2u(pn[4]), f2u(pn[5]), f2u(pn[6]), f2u(pn[7])));
    if constexpr (MD == OPT_F32) {
      st_cs_u4(static_cast<float*>(td.m) + e0, make_uint4(f2u(mnv[0]), f2u(mnv[1]), f2u(mnv[2]), f2u(mnv[3])));
      st_cs_u4(static_cast<float*>(td.m) + e0 + 4,
               make_uint4(f2u(mnv[4]), f2u(mnv[5]), f2u(mnv[6]), f2u(mnv[7])));
    } else {
      st_cs_u4(static_cast<uint16_t*>(td.m) + e0, make_uint4(mpair[0], mpair[1], mpair[2], mpair[3]));
    }
    if constexpr (VD == OPT_F32) {
      st_cs_u4(static_cast<float*>(td.v) + e0, make_uint4(f2u(vnv[0]), f2u(vnv[1]), f2u(vnv[2]), f2u(vnv[3])));
      st_cs_u4(static_cast<float*>(td.v) + e0 + 4,
               make_uint4(f2u(vnv[4]), f2u(vnv[5]), f2u(vnv[6]), f2u(vnv[7])));
    } else if constexpr (VD == OPT_BF16) {
      st_cs_u4(static_cast<uint16_t*>(td.v) + e0, make_uint4(vpair[0], vpair[1], vpair[2], vpair[3]));
    } else if constexpr (VD == OPT_E4M3) {
      if constexpr (WIDE)
        st_cs_u2(static_cast<uint8_t*>(td.v) + e0,
                 make_uint2(__byte_perm(vpair[0], vpair[1], 0x6420), __byte_perm(vpair[2], vpair[3], 0x6420)));
      else
        st_cs_u2(static_cast<uint8_t*>(td.v) + e0,
                 make_uint2(vpair[0] | (vpair[1] << 16), vpair[2] | (vpair[3] << 16)));
    } else {
      // byte k holds element 2k in its low nibble and 2k+1 in its high one:
      // gather the eight codes into a word of even elements and one of odd
      // elements (one code per byte), then w = even | odd << 4
      uint32_t w;
      if constexpr (WIDE) {
        const uint32_t p01 = __byte_perm(vpair[0], vpair[1], 0x6240), p23 = __byte_perm(vpair[2], vpair[3], 0x6240);
        w = __byte_perm(p01, p23, 0x5410) | (__byte_perm(p01, p23, 0x7632) << 4);
      } else {
        w = 0;
#pragma unroll
        for (int k = 0; k < 4; ++k) w |= ((vpair[k] | (vpair[k] >> 4)) & 0xFFu) << (8 * k);
      }
      st_cs_u1(static_cast<uint8_t*>(td.v) + (e0 >> 1), w);
    }
    if constexpr (ALGO == ALGO_ADEMAMIX) {
      st_cs_u4(td.m2 + e0, make_uint4(f2u(m2n[0]), f2u(m2n[1]), f2u(m2n[2]), f2u(m2n[3])));
      st_cs_u4(td.m2 + e0 + 4, make_uint4(f2u(m2n[4]), f2u(m2n[5]), f2u(m2n[6]), f2u(m2n[7])));
    }
  } else if (COMBO == SC_F32 && cnt == 4) {
    // four FP32-state elements (the short-list kernel's quarter groups, or a
    // tensor's last group of exactly four): e0 is a multiple of 4, so 16 bytes
    st_cs_u4(td.p + e0, make_uint4(f2u(pn[0]), f2u(pn[1]), f2u(pn[2]), f2u(pn[3])));
    st_cs_u4(static_cast<float*>(td.m) + e0, make_uint4(f2u(mnv[0]), f2u(mnv[1]), f2u(mnv[2]), f2u(mnv[3])));
    st_cs_u4(static_cast<float*>(td.v) + e0, make_uint4(f2u(vnv[0]), f2u(vnv[1]), f2u(vnv[2]), f2u(vnv[3])));
    if constexpr (ALGO == ALGO_ADEMAMIX)
      st_cs_u4(td.m2 + e0, make_uint4(f2u(m2n[0]), f2u(m2n[1]), f2u(m2n[2]), f2u(m2n[3])));
  } else {
#pragma unroll
    for (int j = 0; j < N; ++j) {
      if (j >= cnt) break;
      const int64_t e = e0 + j;
      td.p[e] = pn[j];
      if constexpr (MD == OPT_F32) static_cast<float*>(td.m)[e] = mnv[j];
      else static_cast<uint16_t*>(td.m)[e] = (uint16_t)((mpair[j >> 1] >> (16 * (j & 1))) & 0xFFFFu);
      if constexpr (VD == OPT_F32) static_cast<float*>(td.v)[e] = vnv[j];
      else if constexpr (VD == OPT_BF16) static_cast<uint16_t*>(td.v)[e] = (uint16_t)vcode_at(j);
      else if constexpr (VD == OPT_E4M3) static_cast<uint8_t*>(td.v)[e] = (uint8_t)vcode_at(j);
      if constexpr (ALGO == ALGO_ADEMAMIX) td.m2[e] = m2n[j];
    }
    if constexpr (VD == OPT_E2M2) {
      // whole bytes: e0 is even, so byte k holds elements 2k and 2k+1 of the
      // group; an element past the end contributes a zero nibble
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        if (2 * k >= cnt) break;
        const uint32_t hi = (2 * k + 1 < cnt) ? vcode_at(2 * k + 1) : 0u;
        static_cast<uint8_t*>(td.v)[(e0 >> 1) + k] = (uint8_t)(vcode_at(2 * k) | (hi << 4));
      }
    }
  }
  return same;
}

// The next tile (from index i, stepping by the grid) in which this thread
// owns a group: thread t owns elements 8t .. 8t+7 of every tile; the last
// tile of a tensor may be shorter than kTileElems.
__device__ __forceinline__ bool next_tile(int64_t& i, const StepArgs& a, int off, opt_chunk& tl) {
  for (; i < a.tile_end; i += gridDim.x) {
    tl = a.tiles[i];
    if (off < (int)tl.len) return true;
  }
  return false;
}

// DEVSC: the step's scalars come from device memory (a.d_sc, written by
// the device step counter's kernel just before), so that a captured CUDA
// graph can replay the step with a new step number; otherwise they are a
// kernel argument.
template <int GT, int COMBO, int ALGO, bool SR, bool DEVSC = false>
__global__ void __launch_bounds__(kStepThreads, (StepShape<GT, COMBO, ALGO, SR>::kMinBlocks))
step_kernel(const StepArgs a) {
  float coef = 1.0f;
  if (a.d_norm != nullptr) {
    if (a.d_norm->status != OPT_OK) return;     // non-finite norm: leave all untouched
    coef = a.d_norm->clip_coef;
  }
  opt_step_scalars sc_dev;
  if constexpr (DEVSC) sc_dev = *a.d_sc;
  const opt_step_scalars& sc = DEVSC ? sc_dev : a.sc;
  const bool count = a.unchanged != nullptr;
  const bool reset = a.reset != 0;
  constexpr bool LA = StepShape<GT, COMBO, ALGO, SR>::kLookahead;
  const int off = threadIdx.x * 8;
  int64_t i = a.tile_begin + blockIdx.x;
  opt_chunk tl, la;     // la: with LA, the entry of tile i + gridDim.x, requested a tile early
  if (LA && i + gridDim.x < a.tile_end) la = a.tiles[i + gridDim.x];
  const int64_t i0 = i;
  bool have = next_tile(i, a, off, tl);
  if (LA && have && i != i0 && i + gridDim.x < a.tile_end) la = a.tiles[i + gridDim.x];   // rare: skipped

  Frag<GT, COMBO, ALGO> cur, nxt;
  TensorDesc ctd;
  int64_t ce0 = 0;
  int ccnt = 0;
  uint32_t ctensor = 0;
  if (have) {
    ctd = a.tensors[tl.tensor];
    ctensor = tl.tensor;
    ce0 = tl.start + off;
    ccnt = min(8, (int)tl.len - off);
    if (ccnt == 8) load_full(ctd, ce0, reset, cur);
    else load_partial(ctd, ce0, ccnt, reset, cur);
  }
  uint32_t same = 0;
  while (have) {
    // request the next group before working on the current one
    int64_t j = i + gridDim.x;
    opt_chunk ntl;
    bool have_next;
    if constexpr (LA) {
      have_next = false;
      if (j < a.tile_end) {
        ntl = la;
        if (j + gridDim.x < a.tile_end) la = a.tiles[j + gridDim.x];
        have_next = off < (int)ntl.len;
        if (!have_next) {
          // rare: no group of this thread in that tile (a tensor's short last tile)
          j += gridDim.x;
          have_next = next_tile(j, a, off, ntl);
          if (have_next && j + gridDim.x < a.tile_end) la = a.tiles[j + gridDim.x];
        }
      }
    } else {
      have_next = next_tile(j, a, off, ntl);
    }
    TensorDesc ntd;
    int64_t ne0 = 0;
    int ncnt = 0;
    if (have_next) {
      // consecutive tiles usually share a tensor; reusing its descriptor pays
      // off where the ALU is busy (low-precision states), not elsewhere
      if constexpr (COMBO != SC_F32) ntd = ntl.tensor == ctensor ? ctd : a.tensors[ntl.tensor];
      else ntd = a.tensors[ntl.tensor];
      ne0 = ntl.start + off;
      ncnt = min(8, (int)ntl.len - off);
      if (ncnt == 8) load_full(ntd, ne0, reset, nxt);
      else load_partial(ntd, ne0, ncnt, reset, nxt);
    }
    same += update_store<GT, COMBO, ALGO, SR>(ctd, ce0, ccnt, cur, coef, sc, ctensor, a.rk, a.step32, count,
                                              a.neg_zero2);
    cur = nxt;
    ctd = ntd;
    ce0 = ne0;
    ccnt = ncnt;
    ctensor = ntl.tensor;
    i = j;
    have = have_next;
  }
  if (a.unchanged != nullptr) {
    // integer sums: the total does not depend on the order of the atomics
    same = __reduce_add_sync(0xFFFFFFFFu, same);
    if ((threadIdx.x & 31) == 0 && same) atomicAdd(a.unchanged, (unsigned long long)same);
  }
}

// Persistent launch: as many CTAs as fit on the GPU at once (occupancy is
// a property of the kernel, cached), but no more than there are tiles.
// Non-persistent shapes launch one CTA per tile (the tile loop then runs
// once; it still covers any tiles past the grid-size limit).
template <int GT, int COMBO, int ALGO, bool SR, bool DEVSC = false>
cudaError_t launch_one(const StepArgs& a, int sm_count, cudaStream_t s) {
  const int64_t n = a.tile_end - a.tile_begin;
  if (n <= 0) return cudaSuccess;
  auto k = step_kernel<GT, COMBO, ALGO, SR, DEVSC>;
  static OccupancyCache occ;
  const int per_sm = cached_occupancy(k, occ, kStepThreads, 0);
  constexpr int64_t kMaxGrid = 0x7FFFFFFF;
  const int64_t full = StepShape<GT, COMBO, ALGO, SR>::kPersistent ? (int64_t)per_sm * sm_count : kMaxGrid;
  const int grid = (int)(n < full ? n : full);
  k<<<grid, kStepThreads, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace psopt
