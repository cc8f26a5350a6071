/*
 * oracle.c -- plain CPU oracle (TEST INFRASTRUCTURE ONLY; see oracle.h).
 *
 * Scalar loops, no SIMD, built with -O2 -ffp-contract=off and no fast-math so
 * that every float operation is a single IEEE round-to-nearest operation in
 * the order written.
 */
#include "oracle.h"

#include <math.h>
#include <string.h>

static uint32_t f2u(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }
static float    u2f(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }

/* ======================================================================
 * BF16 codec.  A BF16 code is the top 16 bits of an FP32 word, so decoding
 * is exact [SMALL sec. 1.1: reading the stored value into FP32 is exact].
 * Nearest: round-to-nearest-even on the 16 dropped bits (what x.to(bfloat16)
 * does).  Stochastic: add a 16-bit draw r to the FP32 word and drop the low
 * 16 bits; a carry into the kept bits happens exactly when l + r >= 2^16,
 * where l is the dropped part [SMALL sec. 6.1].  Inf and NaN are kept.
 * ====================================================================== */
float oracle_bf16_decode(uint16_t code) { return u2f((uint32_t)code << 16); }

uint16_t oracle_bf16_encode(float x, int stochastic, uint32_t r16) {
  uint32_t w = f2u(x);
  uint32_t kept = w >> 16;
  uint32_t dropped = w & 0xFFFFu;
  if ((w & 0x7F800000u) == 0x7F800000u) {         /* Inf or NaN: keep */
    if (w & 0x007FFFFFu) kept |= 0x0040u;           /* NaN stays a (quiet) NaN */
    return (uint16_t)kept;
  }
  int up;
  if (stochastic) {
    up = (dropped + (r16 & 0xFFFFu)) >= 0x10000u;
  } else {
    up = dropped > 0x8000u || (dropped == 0x8000u && (kept & 1u));
  }
  /* incrementing the sign-magnitude word moves away from zero, carrying into
     the exponent (next binade, or Inf past the largest finite value) */
  return (uint16_t)(kept + (uint32_t)up);
}

/* ======================================================================
 * Rounding onto a small floating-point grid with p fraction bits, smallest
 * binade exponent emin (below it the spacing stays 2^(emin-p): subnormals)
 * and largest finite magnitude vmax.  [SMALL sec. 2.1]: the spacing near
 * a = m 2^e is 2^(e-p).  Nearest is round-half-to-even, saturating at vmax.
 * Stochastic follows the same carry rule as the BF16 trick, applied at the
 * target grid's spacing: with t = a / ulp, k = floor(t) and l the first 16
 * bits of the fraction t - k, round up iff l + r >= 2^16 [SMALL sec. 3 and
 * 6.1].  For a BF16 normal this is exactly the BF16 rule.  All steps are
 * exact in double.
 * ====================================================================== */
static double grid_round(double a, int p, int emin, double vmax, int stochastic,
                         uint32_t r16) {
  if (a >= vmax) return vmax;
  if (a == 0.0) return 0.0;
  int e2;
  (void)frexp(a, &e2);           /* a = f 2^e2, f in [0.5, 1) */
  int e = e2 - 1;                /* floor(log2 a) */
  if (e < emin) e = emin;
  double ulp = ldexp(1.0, e - p);
  double t = a / ulp;            /* exact: power-of-two scaling */
  double k = floor(t);
  double frac = t - k;           /* exact */
  int up;
  if (stochastic) {
    uint32_t l16 = (uint32_t)floor(frac * 65536.0);
    up = (l16 + (r16 & 0xFFFFu)) >= 65536u;
  } else {
    up = frac > 0.5 || (frac == 0.5 && fmod(k, 2.0) == 1.0);
  }
  double q = (k + (double)up) * ulp;
  if (q > vmax) q = vmax;
  return q;
}

/* ----- E4M3 (OCP FP8 E4M3FN): bias 7, 3 fraction bits, subnormal spacing
 * 2^-9, largest finite 448, no infinities, NaN = S.1111.111.
 * [SMALL sec. 2.1]: FP8 is 16x coarser than BF16 at the same scale. */
float oracle_e4m3_decode(uint8_t code) {
  int s = code >> 7, e = (code >> 3) & 0xF, k = code & 7;
  double mag;
  if (e == 15 && k == 7) return s ? -NAN : NAN;
  if (e == 0) mag = ldexp((double)k, -9);
  else        mag = ldexp(1.0 + k / 8.0, e - 7);
  return (float)(s ? -mag : mag);
}

static uint8_t e4m3_mag_code(double q) {
  if (q < ldexp(1.0, -6)) return (uint8_t)(q / ldexp(1.0, -9)); /* 0..8 */
  int e2; (void)frexp(q, &e2);
  int e = e2 - 1;
  int k = (int)(q / ldexp(1.0, e - 3)) - 8;
  return (uint8_t)(((e + 7) << 3) | k);
}

uint8_t oracle_e4m3_encode(float x, int stochastic, uint32_t r16) {
  if (isnan(x)) return 0x7F;
  uint8_t sign = signbit(x) ? 0x80 : 0x00;
  double q = grid_round(fabs((double)x), 3, -6, 448.0, stochastic, r16);
  return (uint8_t)(sign | e4m3_mag_code(q));
}

/* ----- unsigned E2M2 (4 bits): 2 exponent bits with bias 1, 2 fraction
 * bits, no sign; codes 0-3 are 0, 1/4, 1/2, 3/4; largest value 7; no NaN or
 * Inf.  [SMALL sec. 2.1]: unsigned E2M2 (not E2M1), 32x coarser than BF16.
 * Negative inputs become 0; NaN becomes the largest code (lossy). */
float oracle_e2m2_decode(uint8_t code) {
  int e = (code >> 2) & 3, k = code & 3;
  if (e == 0) return (float)(k / 4.0);
  return (float)ldexp(1.0 + k / 4.0, e - 1);
}

uint8_t oracle_e2m2_encode(float x, int stochastic, uint32_t r16) {
  if (isnan(x)) return 0xF;
  if (!(x > 0.0f)) return 0;
  double q = grid_round((double)x, 2, 0, 7.0, stochastic, r16);
  if (q < 1.0) return (uint8_t)(q / 0.25);          /* 0..4 */
  int e2; (void)frexp(q, &e2);
  int e = e2 - 1;                                    /* 0..2 */
  int k = (int)(q / ldexp(1.0, e - 2)) - 4;
  return (uint8_t)(((e + 1) << 2) | k);
}

/* ======================================================================
 * Philox-4x32 with 10 rounds [PHILOX sec. 3]: each round multiplies counter
 * words 0 and 2 by the two round multipliers, splits each 64-bit product
 * into high and low halves, and forms the next counter by crossing the
 * halves and XOR-ing the other two words with the round key; the key is
 * advanced by the two Weyl increments between rounds.
 * ====================================================================== */
void oracle_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2],
                          uint32_t out[4]) {
  const uint32_t M0 = 0xD2511F53u, M1 = 0xCD9E8D57u;
  const uint32_t W0 = 0x9E3779B9u, W1 = 0xBB67AE85u;
  uint32_t c0 = ctr[0], c1 = ctr[1], c2 = ctr[2], c3 = ctr[3];
  uint32_t k0 = key[0], k1 = key[1];
  for (int round = 0; round < 10; ++round) {
    if (round > 0) { k0 += W0; k1 += W1; }
    uint64_t prod0 = (uint64_t)M0 * c0;
    uint64_t prod1 = (uint64_t)M1 * c2;
    uint32_t hi0 = (uint32_t)(prod0 >> 32), lo0 = (uint32_t)prod0;
    uint32_t hi1 = (uint32_t)(prod1 >> 32), lo1 = (uint32_t)prod1;
    uint32_t n0 = hi1 ^ c1 ^ k0;
    uint32_t n1 = lo1;
    uint32_t n2 = hi0 ^ c3 ^ k1;
    uint32_t n3 = lo0;
    c0 = n0; c1 = n1; c2 = n2; c3 = n3;
  }
  out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

/* The draw for an element is tied to the element, never to a thread block
 * [SMALL sec. 7.3]: key = seed, counter = (element index / 4, tensor, step);
 * word (index mod 4) of the output gives the m draw (low half) and the v
 * draw (high half). */
void oracle_draws(uint64_t seed, int64_t step, uint32_t tensor_index,
                  int64_t index, uint32_t* r16_m, uint32_t* r16_v) {
  uint64_t q = (uint64_t)index >> 2;
  uint32_t ctr[4] = {(uint32_t)q, (uint32_t)(q >> 32), tensor_index,
                     (uint32_t)step};
  uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
  uint32_t out[4];
  oracle_philox4x32_10(ctr, key, out);
  uint32_t word = out[index & 3];
  *r16_m = word & 0xFFFFu;
  *r16_v = word >> 16;
}

/* The standalone cast draws one 16-bit value per element and no more, so it
 * uses every bit of each Philox output [SMALL sec. 7.3, the same generator
 * and key]: counter = (element index / 8, tensor, step); element i takes
 * word (i / 2) mod 4, its low half for an even i and its high half for an
 * odd one. */
uint32_t oracle_cast_draw(uint64_t seed, int64_t step, uint32_t tensor_index,
                          int64_t index) {
  uint64_t q = (uint64_t)index >> 3;
  uint32_t ctr[4] = {(uint32_t)q, (uint32_t)(q >> 32), tensor_index,
                     (uint32_t)step};
  uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
  uint32_t out[4];
  oracle_philox4x32_10(ctr, key, out);
  uint32_t word = out[(index >> 1) & 3];
  return (index & 1) ? (word >> 16) : (word & 0xFFFFu);
}

/* ======================================================================
 * Gradient norm [NORM "Correctness properties"]: every element is widened to
 * double (exact for BF16 and FP32, and so is its square), the finite squares
 * are summed with Neumaier's compensated summation, tensor by tensor and then
 * across tensors in list order.  The inf-norm is max |g|.  NaN anywhere makes
 * both norms NaN (the NaN is counted, never skipped); otherwise any +-Inf
 * makes both +Inf.  The clip coefficient is min(1, max_norm/(norm + 1e-6)),
 * computed in double and cast once to float; max_norm <= 0 means no clipping.
 * ====================================================================== */
static double load_grad(const void* g, int dtype, int64_t i) {
  if (dtype == ORC_BF16) return (double)oracle_bf16_decode(((const uint16_t*)g)[i]);
  if (dtype == ORC_F64) return ((const double*)g)[i];
  return (double)((const float*)g)[i];
}

static void neumaier_add(double* s, double* c, double x) {
  double t = *s + x;
  if (fabs(*s) >= fabs(x)) *c += (*s - t) + x;
  else                     *c += (x - t) + *s;
  *s = t;
}

void oracle_tensor_sumsq(int64_t n, const void* g, int dtype, oracle_sumsq* out) {
  double s = 0.0, c = 0.0;
  double mx = 0.0;
  uint64_t nans = 0, infs = 0;
  for (int64_t i = 0; i < n; ++i) {
    double x = load_grad(g, dtype, i);
    if (isnan(x)) { ++nans; continue; }
    if (isinf(x)) { ++infs; continue; }
    neumaier_add(&s, &c, x * x);
    if (fabs(x) > mx) mx = fabs(x);
  }
  out->sum = s;
  out->comp = c;
  out->maxabs = (float)mx;
  out->nan_count = nans;
  out->inf_count = infs;
}

float oracle_clip_coef(double norm2, double max_norm) {
  if (!(max_norm > 0.0)) return 1.0f;
  double coef = max_norm / (norm2 + 1e-6);
  if (coef > 1.0) coef = 1.0;
  return (float)coef;
}

void oracle_norm_finish(int32_t n, const oracle_sumsq* parts, double max_norm,
                        oracle_norm* out) {
  double s = 0.0, c = 0.0;
  float mx = 0.0f;
  uint64_t nans = 0, infs = 0;
  for (int32_t i = 0; i < n; ++i) {
    neumaier_add(&s, &c, parts[i].sum);
    neumaier_add(&s, &c, parts[i].comp);
    if (parts[i].maxabs > mx) mx = parts[i].maxabs;
    nans += parts[i].nan_count;
    infs += parts[i].inf_count;
  }
  out->nan_count = nans;
  out->inf_count = infs;
  if (nans > 0) {
    out->sumsq = NAN; out->norm2 = NAN; out->norm_inf = NAN;
    out->clip_coef = 1.0f; out->status = 1;
  } else if (infs > 0) {
    out->sumsq = INFINITY; out->norm2 = INFINITY; out->norm_inf = INFINITY;
    out->clip_coef = 1.0f; out->status = 1;
  } else {
    out->sumsq = s + c;
    out->norm2 = sqrt(out->sumsq);
    out->norm_inf = (double)mx;
    out->clip_coef = oracle_clip_coef(out->norm2, max_norm);
    out->status = 0;
  }
}

void oracle_grad_norm(int32_t n, const int64_t* numel, const void* const* grads,
                      const int32_t* dtypes, double max_norm, oracle_norm* out) {
  oracle_sumsq part, acc;
  double s = 0.0, c = 0.0;
  acc.maxabs = 0.0f; acc.nan_count = 0; acc.inf_count = 0;
  for (int32_t i = 0; i < n; ++i) {
    oracle_tensor_sumsq(numel[i], grads[i], dtypes[i], &part);
    neumaier_add(&s, &c, part.sum);
    neumaier_add(&s, &c, part.comp);
    if (part.maxabs > acc.maxabs) acc.maxabs = part.maxabs;
    acc.nan_count += part.nan_count;
    acc.inf_count += part.inf_count;
  }
  acc.sum = s; acc.comp = c;
  oracle_norm_finish(1, &acc, max_norm, out);
}

/* ======================================================================
 * Optimizer step.
 *
 * AdamW [PR2040 body; Loshchilov & Hutter Alg. 2] and AdEMAMix [PR2040 body;
 * Pagliardini et al.]:
 *   m  <- b1 m  + (1-b1) g
 *   m2 <- b3 m2 + (1-b3) g                 (AdEMAMix only, no bias correction)
 *   v  <- b2 v  + (1-b2) g^2
 *   u  <- (m/(1-b1^t) [+ alpha m2]) / (sqrt(v/(1-b2^t)) + eps)
 *   p  <- p (1 - lr wd) - lr u             decay-first: both terms from old p
 * The wrong decay-after ordering, p <- (p - lr u)(1 - lr wd), and three
 * plausible mistakes in the low-precision update (ORC_MUT_* in oracle.h) are
 * selectable only so that tests can show the pins reject them.
 *
 * FP32 (and F64) states: every step is done in double from the stored values
 * and the results are rounded once to the storage type.
 *
 * Low-precision states: the stored codes are decoded exactly to FP32 and the
 * new moments are formed in FP32 -- the precision the pages call "full
 * precision" for the value before write-back [SMALL sec. 1.1] -- one rounded
 * operation at a time in this order, with no fused multiply-add:
 *   g' = g * coef;  m' = b1*m + omb1*g';  v' = b2*v + omb2*(g'*g')
 * where omb = (float)(1 - (double)b).  m' and v' are then encoded (nearest or
 * stochastic) and the parameter update is done in double from m' and v',
 * the values before rounding: the fused step forms the update and the
 * write-back from the same in-register value ("When Small Updates
 * Disappear", sec. 8.1), never from the codes it has just rounded.
 * ====================================================================== */
static double load_state(const void* s, int dtype, int64_t i) {
  switch (dtype) {
    case ORC_F32:  return (double)((const float*)s)[i];
    case ORC_F64:  return ((const double*)s)[i];
    case ORC_BF16: return (double)oracle_bf16_decode(((const uint16_t*)s)[i]);
    case ORC_E4M3: return (double)oracle_e4m3_decode(((const uint8_t*)s)[i]);
    case ORC_E2M2: {
      uint8_t byte = ((const uint8_t*)s)[i >> 1];
      return (double)oracle_e2m2_decode((i & 1) ? (byte >> 4) : (byte & 0xF));
    }
  }
  return NAN;
}

/* returns the new code (or the f32 bit pattern) so callers can count */
static uint32_t store_state(void* s, int dtype, int64_t i, int64_t n, double val,
                            int stochastic, uint32_t r16) {
  switch (dtype) {
    case ORC_F32: {
      float f = (float)val;
      ((float*)s)[i] = f;
      return f2u(f);
    }
    case ORC_F64: ((double*)s)[i] = val; return 0;
    case ORC_BF16: {
      uint16_t c = oracle_bf16_encode((float)val, stochastic, r16);
      ((uint16_t*)s)[i] = c;
      return c;
    }
    case ORC_E4M3: {
      uint8_t c = oracle_e4m3_encode((float)val, stochastic, r16);
      ((uint8_t*)s)[i] = c;
      return c;
    }
    case ORC_E2M2: {
      uint8_t c = oracle_e2m2_encode((float)val, stochastic, r16);
      uint8_t* b = (uint8_t*)s + (i >> 1);
      if (i & 1) *b = (uint8_t)((*b & 0x0F) | (c << 4));
      else {
        *b = (uint8_t)((*b & 0xF0) | c);
        if (i + 1 == n) *b &= 0x0F;   /* odd length: unused high nibble is 0 */
      }
      return c;
    }
  }
  return 0;
}

static uint32_t state_code(const void* s, int dtype, int64_t i) {
  switch (dtype) {
    case ORC_F32:  return f2u(((const float*)s)[i]);
    case ORC_BF16: return ((const uint16_t*)s)[i];
    case ORC_E4M3: return ((const uint8_t*)s)[i];
    case ORC_E2M2: {
      uint8_t byte = ((const uint8_t*)s)[i >> 1];
      return (i & 1) ? (byte >> 4) : (byte & 0xF);
    }
  }
  return 0;
}

int oracle_adam_tensor(int algo, int64_t n,
                       void* p, int p_dtype,
                       const void* g, int g_dtype,
                       void* m, void* m2, int m_dtype,
                       void* v, int v_dtype,
                       const oracle_hparams* hp, int64_t step, float coef,
                       int stochastic, uint64_t seed, uint32_t tensor_index,
                       int64_t index_base, double v_scale, int mutation,
                       int64_t* unchanged) {
  if (step < 1 || index_base < 0) return -1;
  if (v_dtype == ORC_E2M2 && (index_base & 1)) return -1;
  if (algo == ORC_ADEMAMIX && m2 == 0) return -1;
  int wide = (p_dtype == ORC_F64);
  if (wide && (g_dtype != ORC_F64 || m_dtype != ORC_F64 || v_dtype != ORC_F64)) return -1;
  if (!wide && p_dtype != ORC_F32) return -1;
  if (!wide && g_dtype != ORC_F32 && g_dtype != ORC_BF16) return -1;
  if (!wide && m_dtype != ORC_F32 && m_dtype != ORC_BF16) return -1;
  int lowp = (m_dtype == ORC_BF16) || (v_dtype == ORC_BF16) ||
             (v_dtype == ORC_E4M3) || (v_dtype == ORC_E2M2);
  if (algo == ORC_ADEMAMIX && lowp) return -1;   /* AdEMAMix: FP32 states only */
  if (!(v_scale > 0.0) || (!lowp && v_scale != 1.0)) return -1;

  const double b1 = hp->beta1, b2 = hp->beta2, b3 = hp->beta3;
  const double lr = hp->lr, wd = hp->weight_decay, eps = hp->eps, alpha = hp->alpha;
  const double bc1 = 1.0 - pow(b1, (double)step);
  const double bc2 = 1.0 - pow(b2, (double)step);
  const double decay = 1.0 - lr * wd;

  /* FP32 mirror constants for the low-precision path */
  const float b1f = hp->beta1, b2f = hp->beta2;
  const float omb1f = (float)(1.0 - (double)hp->beta1);
  const float omb2f = (float)(1.0 - (double)hp->beta2);

  int64_t same = 0;
  for (int64_t i = 0; i < n; ++i) {
    double pi = wide ? ((double*)p)[i] : (double)((float*)p)[i];
    double gi = load_grad(g, g_dtype, i);
    uint32_t old_code = wide ? 0 : state_code(v, v_dtype, i);
    double m_new, v_new, m2_new = 0.0;
    uint32_t r16_m = 0, r16_v = 0;
    if (!lowp) {
      double ge = gi * (double)coef;
      m_new = b1 * load_state(m, m_dtype, i) + (1.0 - b1) * ge;
      v_new = b2 * load_state(v, v_dtype, i) + (1.0 - b2) * ge * ge;
      if (algo == ORC_ADEMAMIX)
        m2_new = b3 * load_state(m2, m_dtype, i) + (1.0 - b3) * ge;
    } else {
      float ge = (float)gi * coef;
      float md = (float)load_state(m, m_dtype, i);
      /* a scaled low-precision v code holds v / v_scale (a power of two) */
      float vd = (float)(load_state(v, v_dtype, i) * v_scale);
      float t1 = b1f * md;
      float t2 = omb1f * ge;
      float mf = t1 + t2;
      float t3 = b2f * vd;
      float gg = ge * ge;
      float t4 = omb2f * gg;
      float vf = t3 + t4;
      m_new = mf;
      v_new = vf;
      if (stochastic)
        oracle_draws(seed, step, tensor_index, index_base + i, &r16_m, &r16_v);
    }
    store_state(m, m_dtype, i, n, m_new, stochastic, r16_m);
    uint32_t new_code = store_state(v, v_dtype, i, n, lowp ? v_new / v_scale : v_new, stochastic, r16_v);
    if (algo == ORC_ADEMAMIX)
      store_state(m2, m_dtype, i, n, m2_new, stochastic, r16_m);
    if (!wide && new_code == old_code) ++same;

    /* the update, from the new moments before rounding */
    double mu = m_new, vu = v_new, c1 = bc1, c2 = bc2;
    if (lowp && (mutation & ORC_MUT_U_FROM_CODES)) {
      mu = load_state(m, m_dtype, i);
      vu = load_state(v, v_dtype, i) * v_scale;
    }
    if (lowp && (mutation & ORC_MUT_SCALE_IN_SQRT)) vu = vu / v_scale;
    if (lowp && (mutation & ORC_MUT_NO_BIAS_CORR)) c1 = c2 = 1.0;
    double num = mu / c1;
    if (algo == ORC_ADEMAMIX) num += alpha * m2_new;
    double u = num / (sqrt(vu / c2) + eps);
    double pn = (mutation & ORC_MUT_DECAY_AFTER) ? (pi - lr * u) * decay : pi * decay - lr * u;

    if (wide) ((double*)p)[i] = pn;
    else      ((float*)p)[i] = (float)pn;
  }
  if (unchanged) *unchanged = same;
  return 0;
}

/* ======================================================================
 * LAMB-style update-norm clipping ("Investigate SM103 bias-correction
 * broadcast in 32-bit optimizers", 'Problem' and 'B300 result': the 2-state
 * optimizers' max_unorm > 0 path measures the norm of the whole update of a
 * tensor before applying it).  Reading (the pages give no formula): with the
 * AdamW direction u of every element of the tensor (computed from the new
 * moments as in oracle_adam_tensor, FP32 states), ratio = max_unorm |p| / |u|
 * when |u| > max_unorm |p| (norms over the tensor, |p| of the parameters
 * before the step), else 1; then p <- p (1 - lr wd) - lr ratio u, decay-first.
 * Norms are summed in double with Neumaier's compensation.
 * ====================================================================== */
int oracle_lamb_tensor(int64_t n, float* p, const void* g, int g_dtype, float* m,
                       float* v, const oracle_hparams* hp, int64_t step, float coef,
                       float max_unorm, double* ratio_out) {
  if (step < 1 || n < 0) return -1;
  if (g_dtype != ORC_F32 && g_dtype != ORC_BF16) return -1;
  const double b1 = hp->beta1, b2 = hp->beta2;
  const double lr = hp->lr, wd = hp->weight_decay, eps = hp->eps;
  const double bc1 = 1.0 - pow(b1, (double)step);
  const double bc2 = 1.0 - pow(b2, (double)step);
  const double decay = 1.0 - lr * wd;
  double su = 0.0, cu = 0.0, sp = 0.0, cp = 0.0;
  /* first pass: the new moments (stored as FP32, as the buffers hold) and
     the norms of the update and of the old parameters */
  for (int64_t i = 0; i < n; ++i) {
    double ge = load_grad(g, g_dtype, i) * (double)coef;
    float mf = (float)(b1 * (double)m[i] + (1.0 - b1) * ge);
    float vf = (float)(b2 * (double)v[i] + (1.0 - b2) * ge * ge);
    m[i] = mf;
    v[i] = vf;
    double u = ((double)mf / bc1) / (sqrt((double)vf / bc2) + eps);
    neumaier_add(&su, &cu, u * u);
    neumaier_add(&sp, &cp, (double)p[i] * (double)p[i]);
  }
  const double un = sqrt(su + cu), pn = sqrt(sp + cp);
  double ratio = 1.0;
  if (max_unorm > 0.0f && un > (double)max_unorm * pn && un > 0.0)
    ratio = (double)max_unorm * pn / un;
  /* second pass: the update from the stored moments */
  for (int64_t i = 0; i < n; ++i) {
    double u = ((double)m[i] / bc1) / (sqrt((double)v[i] / bc2) + eps);
    p[i] = (float)((double)p[i] * decay - lr * ratio * u);
  }
  if (ratio_out) *ratio_out = ratio;
  return 0;
}
