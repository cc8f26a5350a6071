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
// tile (half a tile with FP32 states, below), finds its tensor by scanning
// at most eight parameter words, and requests its data first; the norm's
// status and clip coefficient, a dependent load of their own, are read
// while the data are on the way.  The per-element work is update_store, so
// the results are the same bits as the persistent kernel's.
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

// FP32 states: each thread takes 4 elements, two CTAs per tile (CTA 2i + h
// takes elements h * 1024 .. h * 1024 + 1023 of tile i), so twice the threads
// hold half the words each.  Same update_store arithmetic, on four lanes.
// The read-only gradient's 8 BF16 bytes come through the non-coherent path.
__device__ __forceinline__ uint2 ld_nc_u2(const void* p) {
  uint2 r;
  asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];" : "=r"(r.x), "=r"(r.y) : "l"(p));
  return r;
}

template <int GT, int ALGO>
__global__ void __launch_bounds__(kStepThreads)
step_small4_kernel(const StepArgs a, const __grid_constant__ SmallList L) {
  using F = Frag<GT, SC_F32, ALGO>;
  const int64_t tile = blockIdx.x >> 1;
  int k = 0;
  while (k + 1 < L.n && tile >= L.tile_end[k]) ++k;
  const TensorDesc& td = L.td[k];
  const int64_t e0 = (tile - (k ? L.tile_end[k - 1] : 0)) * kTileElems + (int64_t)(blockIdx.x & 1) * (kTileElems / 2) +
                     threadIdx.x * 4;
  const int64_t left = td.numel - e0;
  const int cnt = left < 4 ? (int)left : 4;
  const bool reset = a.reset != 0;
  F f;
  if (cnt == 4) {
    put4(f.p, ld_cs_u4(td.p + e0));
    if constexpr (GT == OPT_BF16) {
      const uint2 w = ld_nc_u2(static_cast<const uint16_t*>(td.g) + e0);
      f.g[0] = w.x;
      f.g[1] = w.y;
    } else {
      put4(f.g, ld_nc_u4(static_cast<const float*>(td.g) + e0));
    }
    if (reset) {
#pragma unroll
      for (int q = 0; q < 4; ++q) f.m[q] = f.v[q] = 0u;
      if constexpr (ALGO == ALGO_ADEMAMIX) {
#pragma unroll
        for (int q = 0; q < 4; ++q) f.m2[q] = 0u;
      }
    } else {
      put4(f.m, ld_cs_u4(static_cast<const float*>(td.m) + e0));
      put4(f.v, ld_cs_u4(static_cast<const float*>(td.v) + e0));
      if constexpr (ALGO == ALGO_ADEMAMIX) put4(f.m2, ld_cs_u4(td.m2 + e0));
    }
  } else if (cnt > 0) {
    load_partial(td, e0, cnt, reset, f);
  }
  float coef = 1.0f;
  if (a.d_norm != nullptr) {
    if (a.d_norm->status != OPT_OK) return;     // non-finite norm: leave all untouched
    coef = a.d_norm->clip_coef;
  }
  const bool count = a.unchanged != nullptr;
  uint32_t same = 0;
  if (cnt > 0)
    same = update_store<GT, SC_F32, ALGO, false, 4>(td, e0, cnt, f, coef, a.sc, L.tensor[k], a.rk, a.step32, count,
                                                    a.neg_zero2);
  if (count) {
    same = __reduce_add_sync(0xFFFFFFFFu, same);
    if ((threadIdx.x & 31) == 0 && same) atomicAdd(a.unchanged, (unsigned long long)same);
  }
}

template <int GT, int COMBO, int ALGO, bool SR>
cudaError_t launch_small(const StepArgs& a, const SmallList& L, cudaStream_t s) {
  const int64_t n = L.n > 0 ? L.tile_end[L.n - 1] : 0;
  if (n <= 0) return cudaSuccess;
  if constexpr (COMBO == SC_F32)
    step_small4_kernel<GT, ALGO><<<(unsigned)(2 * n), kStepThreads, 0, s>>>(a, L);
  else
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
