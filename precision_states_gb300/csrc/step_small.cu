// step_small.cu -- the fused step for short lists: a launch shape in which
// no dependent global load stands before a tile's data.
//
// The persistent step kernel reaches each tile through two dependent global
// loads -- its table entry, then its tensor's descriptor -- before it can
// request the tile's data, and on a list of one or a few tensors (the
// 1M-parameter AdamW workload: 512 tiles over 304 resident CTAs) those
// chains are most of the launch: the SMs were busy 56 % of a 12 us launch,
// stalled on them.  Here a bucket of at most kSmallMaxTensors tensors and
// kSmallMaxTiles tiles travels in the kernel's parameters (descriptors and
// the tile count of each tensor), every CTA takes exactly one 2048-element
// tile, finds its tensor by scanning at most eight parameter words, and
// requests its data first; the norm's status and clip coefficient, a
// dependent load of their own, are read while the data are on the way.
// The per-element work is update_store, so the results are the same bits as
// the persistent kernel's.
#include "common.cuh"
#include "internal.h"
#include "step_kernel.cuh"

namespace psopt {
namespace {

template <int GT, int COMBO, int ALGO, bool SR>
__global__ void __launch_bounds__(kStepThreads, 2)
step_small_kernel(const StepArgs a, const __grid_constant__ SmallList L) {
  using F = Frag<GT, COMBO, ALGO>;
  const int64_t tile = blockIdx.x;
  int k = 0;
  while (k + 1 < L.n && tile >= L.tile_end[k]) ++k;
  const TensorDesc& td = L.td[k];
  const int64_t e0 = (tile - (k ? L.tile_end[k - 1] : 0)) * kTileElems + threadIdx.x * 8;
  const int64_t left = td.numel - e0;
  const int cnt = left < 8 ? (int)left : 8;
  const bool reset = a.reset != 0;
  F f;
  if (cnt == 8) load_full(td, e0, reset, f);
  else if (cnt > 0) load_partial(td, e0, cnt, reset, f);
  float coef = 1.0f;
  if (a.d_norm != nullptr) {
    if (a.d_norm->status != OPT_OK) return;     // non-finite norm: leave all untouched
    coef = a.d_norm->clip_coef;
  }
  const bool count = a.unchanged != nullptr;
  uint32_t same = 0;
  if (cnt > 0)
    same = update_store<GT, COMBO, ALGO, SR>(td, e0, cnt, f, coef, a.sc, L.tensor[k], a.rk, a.step32, count,
                                             a.neg_zero2);
  if (count) {
    // integer sums: the total does not depend on the order of the atomics
    same = __reduce_add_sync(0xFFFFFFFFu, same);
    if ((threadIdx.x & 31) == 0 && same) atomicAdd(a.unchanged, (unsigned long long)same);
  }
}

template <int GT, int COMBO, int ALGO, bool SR>
cudaError_t launch_small(const StepArgs& a, const SmallList& L, cudaStream_t s) {
  const int64_t n = L.n > 0 ? L.tile_end[L.n - 1] : 0;
  if (n <= 0) return cudaSuccess;
  step_small_kernel<GT, COMBO, ALGO, SR><<<(unsigned)n, kStepThreads, 0, s>>>(a, L);
  return cudaGetLastError();
}

template <int GT>
cudaError_t dispatch(int combo, int algo, bool stochastic, const StepArgs& a, const SmallList& L, cudaStream_t s) {
  if (combo == SC_F32)
    return algo == ALGO_ADEMAMIX ? launch_small<GT, SC_F32, ALGO_ADEMAMIX, false>(a, L, s)
                                 : launch_small<GT, SC_F32, ALGO_ADAMW, false>(a, L, s);
  switch (combo) {
    case SC_BF16_BF16:
      return stochastic ? launch_small<GT, SC_BF16_BF16, ALGO_ADAMW, true>(a, L, s)
                        : launch_small<GT, SC_BF16_BF16, ALGO_ADAMW, false>(a, L, s);
    case SC_BF16_E4M3:
      return stochastic ? launch_small<GT, SC_BF16_E4M3, ALGO_ADAMW, true>(a, L, s)
                        : launch_small<GT, SC_BF16_E4M3, ALGO_ADAMW, false>(a, L, s);
    case SC_BF16_E2M2:
      return stochastic ? launch_small<GT, SC_BF16_E2M2, ALGO_ADAMW, true>(a, L, s)
                        : launch_small<GT, SC_BF16_E2M2, ALGO_ADAMW, false>(a, L, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_step_small(int grad_dtype, int combo, int algo, int stochastic, const StepArgs& a,
                              const SmallList& L, cudaStream_t s) {
  if (grad_dtype == OPT_BF16) return dispatch<OPT_BF16>(combo, algo, stochastic != 0, a, L, s);
  return dispatch<OPT_F32>(combo, algo, stochastic != 0, a, L, s);
}

}  // namespace psopt
