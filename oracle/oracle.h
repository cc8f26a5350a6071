/*
 * oracle.h -- plain CPU oracle for the fused optimizer step (TEST INFRASTRUCTURE).
 *
 * This library is test infrastructure only.  It is the slow, obviously-correct
 * definition that the CUDA library is checked against.  Only the tests, the
 * smoke check and the benchmark's CPU-baseline leg may load it; the product
 * path never calls it.  It shares no code, header, table or constant with the
 * CUDA library under precision_states_gb300/.
 *
 * Sources (cited by page title and section):
 *  [PR2040]  "Fix decoupled weight decay ordering in the CUDA Adam/AdEMAMix
 *            kernels" (bitsandbytes PR #2040): body (decay-first ordering),
 *            "Why the current tests do not catch it" (step-1 closed form).
 *  [SMALL]   "When Small Updates Disappear" (Topollai): sec. 1.1 (EMA update,
 *            exact FP32 read-back), sec. 2-2.1 (ULP, FP8/FP4 grids), sec. 3
 *            (stochastic rounding), sec. 6.1 (BF16 carry rule), sec. 7.2-7.3
 *            (counter-based hash tied to the element).
 *  [NORM]    "perf(training): fused multi-tensor gradient-norm reduction"
 *            (NeMo Automodel PR #3685): "Numerics", "Correctness properties".
 *  [PHILOX]  Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As Easy as
 *            1, 2, 3", SC'11, sec. 3 (Philox-4x32, 10 rounds).
 *
 * Parity pins: every function here is pinned by tests/test_oracle_*.py
 * against closed forms, brute force, library routines or values printed on
 * the pages: the codecs against torch's casts, brute force over every code
 * and the carry rule; the norm against exact rational arithmetic; the step,
 * FP32 and low-precision states alike, against the one-step closed form and
 * torch.optim.AdamW in float64, with planted mistakes (the `mutation` bits)
 * shown to fail those pins; the Philox generator against cuRAND's host-side
 * Philox4_32_10 generator.
 */
#ifndef PS_ORACLE_H
#define PS_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* storage types understood by the oracle */
enum { ORC_F32 = 0, ORC_BF16 = 1, ORC_E4M3 = 2, ORC_E2M2 = 3, ORC_F64 = 4 };

/* ---- codecs ---------------------------------------------------------- */
float    oracle_bf16_decode(uint16_t code);
uint16_t oracle_bf16_encode(float x, int stochastic, uint32_t r16);
float    oracle_e4m3_decode(uint8_t code);
uint8_t  oracle_e4m3_encode(float x, int stochastic, uint32_t r16);
float    oracle_e2m2_decode(uint8_t code);            /* code in 0..15 */
uint8_t  oracle_e2m2_encode(float x, int stochastic, uint32_t r16);

/* ---- counter-based generator ------------------------------------------ */
void oracle_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2],
                          uint32_t out[4]);
/* The two 16-bit draws (for m and for v) of element `index` of tensor
 * `tensor_index` at step `step` under `seed`. */
void oracle_draws(uint64_t seed, int64_t step, uint32_t tensor_index,
                  int64_t index, uint32_t* r16_m, uint32_t* r16_v);
/* The single 16-bit draw of element `index` in the standalone cast: eight
 * elements per generator call (counter index / 8, word (index / 2) mod 4,
 * low half for even index, high half for odd). */
uint32_t oracle_cast_draw(uint64_t seed, int64_t step, uint32_t tensor_index,
                          int64_t index);

/* ---- gradient norm ---------------------------------------------------- */
typedef struct {
  double   sum;       /* Neumaier running sum of finite squares */
  double   comp;      /* its compensation term                  */
  float    maxabs;    /* max |g| over finite elements           */
  uint64_t nan_count;
  uint64_t inf_count;
} oracle_sumsq;

typedef struct {
  double   sumsq, norm2, norm_inf;
  uint64_t nan_count, inf_count;
  float    clip_coef;
  int32_t  status;   /* 0 finite, 1 non-finite */
} oracle_norm;

void oracle_tensor_sumsq(int64_t n, const void* g, int dtype, oracle_sumsq* out);
void oracle_norm_finish(int32_t n, const oracle_sumsq* parts, double max_norm,
                        oracle_norm* out);
void oracle_grad_norm(int32_t n, const int64_t* numel, const void* const* grads,
                      const int32_t* dtypes, double max_norm, oracle_norm* out);
float oracle_clip_coef(double norm2, double max_norm);

/* ---- optimizer step (one tensor, in place) ---------------------------- */
typedef struct {
  float lr, beta1, beta2, beta3, alpha, eps, weight_decay;
} oracle_hparams;

enum { ORC_ADAMW = 0, ORC_ADEMAMIX = 1 };

/* Applies one step t (1-based) to one tensor.  p is f32 (or f64 when
 * p_dtype == ORC_F64, then every state is f64 too).  g is f32 or bf16 (f64
 * with p_dtype == ORC_F64).  m is f32 or bf16 (AdEMAMix: m, m2, v all f32); v is f32, bf16, e4m3
 * or e2m2 (two codes per byte, low nibble = even element).  `coef` is the
 * clip coefficient (1 = none).  Element i of the arrays is element
 * index_base + i of the tensor (it selects the stochastic-rounding draws; it
 * must be even for E2M2).  v_scale (1 unless v is low precision): the v
 * code holds v / v_scale ("When Small Updates Disappear", sec. 2.3 and 5:
 * a coarse grid flushes a small second moment; a power-of-two scale moves v
 * onto the grid without changing the rounding rule).  `mutation` is 0 for
 * the oracle itself; its ORC_MUT_* bits each plant one plausible mistake,
 * and exist only so that tests can show the pins catch it.  *unchanged (if
 * non-NULL) receives the count of v codes (or f32 words) left bitwise
 * unchanged by this step.  Returns 0, or -1 on an unsupported combination. */
enum {
  ORC_MUT_DECAY_AFTER = 1,    /* p <- (p - lr u)(1 - lr wd): the ordering the
                                 decay-ordering PR fixed */
  ORC_MUT_U_FROM_CODES = 2,   /* low-precision states: u from the re-decoded
                                 stored codes, not the values before rounding */
  ORC_MUT_NO_BIAS_CORR = 4,   /* low-precision states: u without 1/(1-b1^t) and
                                 1/(1-b2^t) */
  ORC_MUT_SCALE_IN_SQRT = 8   /* low-precision states: u from v / v_scale (the
                                 stored value) instead of v */
};
int oracle_adam_tensor(int algo, int64_t n,
                       void* p, int p_dtype,
                       const void* g, int g_dtype,
                       void* m, void* m2, int m_dtype,
                       void* v, int v_dtype,
                       const oracle_hparams* hp, int64_t step, float coef,
                       int stochastic, uint64_t seed, uint32_t tensor_index,
                       int64_t index_base, double v_scale, int mutation,
                       int64_t* unchanged);

/* LAMB-style update-norm clipping of one tensor (FP32 states), in place:
 * the new moments, u = m_hat / (sqrt(v_hat) + eps) per element,
 * ratio = min(1, max_unorm |p| / |u|) over the tensor (1 when max_unorm <= 0),
 * p <- p (1 - lr wd) - lr ratio u.  *ratio_out receives the ratio. */
int oracle_lamb_tensor(int64_t n, float* p, const void* g, int g_dtype, float* m,
                       float* v, const oracle_hparams* hp, int64_t step, float coef,
                       float max_unorm, double* ratio_out);

#ifdef __cplusplus
}
#endif
#endif
