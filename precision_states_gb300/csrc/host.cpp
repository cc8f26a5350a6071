// host.cpp -- host-only parts of the C ABI (no CUDA calls): status strings,
// the chunk table, the per-step scalars and the cross-rank norm combine.
#include <cmath>
#include <cstdint>
#include <cstring>
#include <limits>

#include "opt.h"

extern "C" {

int opt_version(void) { return OPT_ABI_VERSION; }

const char* opt_strerror(int status) {
  switch (status) {
    case OPT_OK: return "ok";
    case OPT_ENONFINITE: return "gradient norm is not finite (step skipped)";
    case OPT_EINVAL: return "invalid argument";
    case OPT_EUNSUPPORTED: return "unsupported dtype combination";
    case OPT_EALIGN: return "device pointer not 16-byte aligned";
    case OPT_ECUDA: return "CUDA runtime error";
    case OPT_ENOMEM: return "out of device memory";
    case OPT_ELIMIT: return "list exceeds a fixed limit of the norm";
    default: return "unknown status";
  }
}

}  // extern "C"

namespace psopt {
// A table of pieces of at most `elems` elements, from sizes and gradient
// dtypes only ("perf(training): fused multi-tensor gradient-norm reduction",
// 'Correctness properties': host-side decomposition from sizes, no atomics;
// 'What': one launch per dtype bucket).  FP32-gradient tensors first, then
// BF16; list order within a bucket; element order within a tensor.
int64_t build_table(int32_t n, const int64_t* numel, const int32_t* grad_dtype, const int64_t elems[2],
                    opt_chunk* out, int64_t cap, int64_t bucket_begin[3]) {
  if (n < 0 || (n > 0 && (numel == nullptr || grad_dtype == nullptr))) return OPT_EINVAL;
  for (int32_t i = 0; i < n; ++i) {
    if (numel[i] < 0) return OPT_EINVAL;
    if (grad_dtype[i] != OPT_F32 && grad_dtype[i] != OPT_BF16) return OPT_EUNSUPPORTED;
  }
  const int buckets[2] = {OPT_F32, OPT_BF16};
  int64_t count = 0;
  for (int b = 0; b < 2; ++b) {
    if (bucket_begin) bucket_begin[b] = count;
    for (int32_t i = 0; i < n; ++i) {
      if (grad_dtype[i] != buckets[b]) continue;
      for (int64_t start = 0; start < numel[i]; start += elems[b]) {
        if (out != nullptr && count < cap) {
          const int64_t left = numel[i] - start;
          out[count].tensor = (uint32_t)i;
          out[count].len = (uint32_t)(left < elems[b] ? left : elems[b]);
          out[count].start = start;
        }
        ++count;
      }
    }
  }
  if (bucket_begin) bucket_begin[2] = count;
  return count;
}

// The norm's chunk size for one dtype bucket (the rule stated at
// OPT_NORM_CHUNK_MIN in opt.h).  Measured on GB300 with the norm's
// one-CTA-per-SM kernel: on the 740-tensor list (197M elements), each norm
// right after an AdamW step whose dirty L2 lines it evicts, 4K-element
// chunks took 0.080 ms against 0.084 with 8K and 0.088 with 16K, and the
// whole step ran 0.45 % faster (with L2 clean first 8K was faster, 0.0705
// against 0.073 ms); 32K chunks were fastest on the Llama-3-8B list (8.03e9;
// 16K 1 % slower).
int64_t norm_chunk_elems(int32_t n, const int64_t* numel, const int32_t* grad_dtype, int bucket) {
  if (n < 0 || (n > 0 && (numel == nullptr || grad_dtype == nullptr)) || bucket < 0 || bucket > 1)
    return OPT_EINVAL;
  const int want = bucket == 0 ? OPT_F32 : OPT_BF16;
  int64_t elems = 0;
  for (int32_t i = 0; i < n; ++i) {
    if (numel[i] < 0) return OPT_EINVAL;
    if (grad_dtype[i] != OPT_F32 && grad_dtype[i] != OPT_BF16) return OPT_EUNSUPPORTED;
    if (grad_dtype[i] == want) elems += numel[i];
  }
  int64_t ce = elems < (int64_t(1) << 28) ? OPT_NORM_CHUNK_MIN
             : elems < (int64_t(1) << 29) ? 2 * OPT_NORM_CHUNK_MIN
             : elems < (int64_t(1) << 31) ? 4 * OPT_NORM_CHUNK_MIN : OPT_CHUNK_ELEMS;
  for (; ce <= (int64_t(1) << 31); ce *= 2) {
    int64_t chunks = 0;
    for (int32_t i = 0; i < n; ++i)
      if (grad_dtype[i] == want) chunks += (numel[i] + ce - 1) / ce;
    if ((chunks + OPT_NORM_SLOTS - 1) / OPT_NORM_SLOTS <= OPT_NORM_MAX_PART) return ce;
  }
  return OPT_ELIMIT;     // more tensors than the slots can hold chunks
}
}  // namespace psopt

extern "C" {

int64_t opt_chunk_table(int32_t n, const int64_t* numel, const int32_t* grad_dtype,
                        opt_chunk* out, int64_t cap, int64_t bucket_begin[3]) {
  int64_t ce[2];
  for (int b = 0; b < 2; ++b) {
    ce[b] = psopt::norm_chunk_elems(n, numel, grad_dtype, b);
    if (ce[b] < 0) return ce[b];
  }
  return psopt::build_table(n, numel, grad_dtype, ce, out, cap, bucket_begin);
}

int64_t opt_norm_chunk_elems(int32_t n, const int64_t* numel, const int32_t* grad_dtype, int32_t bucket) {
  return psopt::norm_chunk_elems(n, numel, grad_dtype, bucket);
}

// Per-step scalars, formed in double and rounded once ("Investigate SM103
// bias-correction broadcast in 32-bit optimizers", 'Problem': the
// bias-correction terms are uniform across threads).
int opt_step_scalars_compute(const opt_hparams* hp, int64_t step, opt_step_scalars* out) {
  if (hp == nullptr || out == nullptr || step < 1) return OPT_EINVAL;
  const double lr = hp->lr, wd = hp->weight_decay;
  const double b1 = hp->beta1, b2 = hp->beta2, b3 = hp->beta3;
  // the ranges torch.optim.AdamW accepts, and finite: beta1, beta2 < 1 keep
  // the bias corrections 1 - beta^t positive; beta3 = 1 freezes m2
  const double vals[7] = {lr, wd, b1, b2, b3, (double)hp->alpha, (double)hp->eps};
  for (double x : vals)
    if (!std::isfinite(x)) return OPT_EINVAL;
  if (lr < 0.0 || wd < 0.0 || hp->eps < 0.0f) return OPT_EINVAL;
  if (!(b1 >= 0.0 && b1 < 1.0) || !(b2 >= 0.0 && b2 < 1.0) || !(b3 >= 0.0 && b3 <= 1.0)) return OPT_EINVAL;
  out->lr = hp->lr;
  out->decay = (float)(1.0 - lr * wd);
  out->beta1 = hp->beta1;
  out->omb1 = (float)(1.0 - b1);
  out->beta2 = hp->beta2;
  out->omb2 = (float)(1.0 - b2);
  out->beta3 = hp->beta3;
  out->omb3 = (float)(1.0 - b3);
  out->alpha = hp->alpha;
  out->eps = hp->eps;
  out->inv_bc1 = (float)(1.0 / (1.0 - std::pow(b1, (double)step)));
  out->inv_bc2 = (float)(1.0 / (1.0 - std::pow(b2, (double)step)));
  return OPT_OK;
}

int opt_norm_combine(const opt_norm_result* parts, int32_t n, double max_norm,
                     opt_norm_result* out) {
  if (n < 0 || (n > 0 && parts == nullptr) || out == nullptr) return OPT_EINVAL;
  double sum = 0.0, mx = 0.0;
  uint64_t nans = 0, infs = 0;
  for (int32_t i = 0; i < n; ++i) {
    nans += parts[i].nan_count;
    infs += parts[i].inf_count;
    if (parts[i].nan_count == 0 && parts[i].inf_count == 0) {
      sum += parts[i].sumsq;
      if (parts[i].norm_inf > mx) mx = parts[i].norm_inf;
    }
  }
  opt_norm_result r;
  std::memset(&r, 0, sizeof r);
  r.nan_count = nans;
  r.inf_count = infs;
  r.clip_coef = 1.0f;
  if (nans > 0) {
    r.sumsq = r.norm2 = r.norm_inf = std::numeric_limits<double>::quiet_NaN();
    r.status = OPT_ENONFINITE;
  } else if (infs > 0) {
    r.sumsq = r.norm2 = r.norm_inf = std::numeric_limits<double>::infinity();
    r.status = OPT_ENONFINITE;
  } else {
    r.sumsq = sum;
    r.norm2 = std::sqrt(sum);
    r.norm_inf = mx;
    if (max_norm > 0.0) {
      double coef = max_norm / (r.norm2 + 1e-6);
      r.clip_coef = (float)(coef > 1.0 ? 1.0 : coef);
    }
    r.status = OPT_OK;
  }
  *out = r;
  return OPT_OK;
}

}  // extern "C"
