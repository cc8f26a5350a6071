// step_dyn.cuh -- the fused AdamW and AdEMAMix steps with FP32 states, their
// tiles handed to warps as they free up.
//
// The same per-element work as step_kernel (update_store, so the same bits),
// scheduled differently.  In the persistent step_kernel, CTA c takes tiles
// c, c + G, ... fixed in advance, and CTAs whose share of an SM's bandwidth
// is smaller finish later: per-CTA %globaltimer stamps on GB300 showed the
// CTAs ending over 1.3 % of the launch on the Llama-3-8B list and 3.5 % on
// the 740-tensor list, the SMs idling meanwhile.  Here every warp takes whole
// tiles from a counter (one atomic per 2048-element tile, requested a tile
// ahead), and its lanes cover a tile in eight passes of 256 elements (lane l:
// elements pass * 256 + 8 l .. + 7), keeping the register pipeline of
// step_kernel: the words of the lane's next group -- the next pass, or the
// first of the next tile -- are requested before the current group is
// updated.  Each tile's update is independent of which warp does it, so the
// result does not depend on the order.  The counter and a count of finished
// warps live in the plan's workspace; the last warp of a launch to finish
// returns both to 0 for the next launch.
//
// Measured on GB300 against the fixed shares (A/B/A/B): Llama-3-8B AdamW
// step 30.41 -> 29.76 ms (1.024 -> 1.047 of the measured copy bandwidth),
// 740-tensor list 1.005 -> 1.024, AdEMAMix on the GPT-2 list 1.001 -> 1.012
// (1.025-1.027 once it took its next tile at the switch, without spills),
// FP32-state AdamW on the GPT-2 list 1.018 -> 1.013.  The nearest E4M3 /
// E2M2 states keep step_kernel: at their 3 CTAs per SM this loop spills
// (60-76 bytes) and ran at 0.88 / 0.96 against 1.00 / 1.01.
#pragma once

#include "step_kernel.cuh"

namespace psopt {

// The next tile index from the counter (lane 0's atomic, broadcast).
__device__ __forceinline__ int64_t dyn_take(unsigned long long* ctr, int lane) {
  unsigned long long v = 0ull;
  if (lane == 0) v = atomicAdd(ctr, 1ull);
  return (int64_t)__shfl_sync(0xFFFFFFFFu, v, 0);
}

// A warp that has taken its last index (>= the tile count) counts itself;
// once every warp of the launch has, no one reads the counter again, and the
// last one returns both counts to 0.
__device__ __forceinline__ void dyn_done(unsigned long long* ctr, int lane) {
  if (lane != 0) return;
  const unsigned long long warps = (unsigned long long)gridDim.x * (blockDim.x / 32);
  __threadfence();                     // this warp's last take comes before its count
  if (atomicAdd(ctr + 1, 1ull) == warps - 1) {
    __threadfence();                   // and every warp's, before the reset
    ctr[0] = 0ull;
    ctr[1] = 0ull;
  }
}

template <int GT, int COMBO, int ALGO, bool SR, bool DEVSC>
__global__ void __launch_bounds__(kStepThreads, (StepShape<GT, COMBO, ALGO, SR>::kMinBlocks))
step_dyn_kernel(const StepArgs a) {
  using F = Frag<GT, COMBO, ALGO>;
  float coef = 1.0f;
  if (a.d_norm != nullptr) {
    if (a.d_norm->status != OPT_OK) return;     // non-finite norm: leave all untouched (counters stay 0)
    coef = a.d_norm->clip_coef;
  }
  opt_step_scalars sc_dev;
  if constexpr (DEVSC) sc_dev = *a.d_sc;
  const opt_step_scalars& sc = DEVSC ? sc_dev : a.sc;
  const bool count = a.unchanged != nullptr;
  const bool reset = a.reset != 0;
  const int lane = threadIdx.x & 31;
  const int64_t n = a.tile_end - a.tile_begin;
  unsigned long long* ctr = a.dyn;
  uint32_t same = 0;
  // AHEAD: the next tile is taken, and its entry requested, a tile early.
  // AdEMAMix, whose five streams fill the registers, takes it when it
  // switches tiles instead, which keeps it from spilling.
  constexpr bool AHEAD = ALGO != ALGO_ADEMAMIX;

  int64_t u = dyn_take(ctr, lane);
  if (u < n) {
    opt_chunk tl = a.tiles[a.tile_begin + u];
    int64_t un = AHEAD ? dyn_take(ctr, lane) : 0;
    opt_chunk tln{};
    if (AHEAD && un < n) tln = a.tiles[a.tile_begin + un];
    TensorDesc ctd = a.tensors[tl.tensor];
    uint32_t ctensor = tl.tensor;
    int pass = 0;
    int64_t ce0 = tl.start + lane * 8;
    int ccnt = min(8, (int)tl.len - lane * 8);
    F cur, nxt;
    if (ccnt == 8) load_full(ctd, ce0, reset, cur);
    else if (ccnt > 0) load_partial(ctd, ce0, ccnt, reset, cur);
    bool have = true;
    while (have) {
      // request the lane's next group before working on the current one
      TensorDesc ntd = ctd;
      uint32_t ntensor = ctensor;
      int64_t ne0 = 0;
      int ncnt = 0;
      bool have_next = true;
      if ((pass + 1) * 256 < (int)tl.len) {
        ++pass;
        const int o = pass * 256 + lane * 8;
        ne0 = tl.start + o;
        ncnt = min(8, (int)tl.len - o);
      } else if (AHEAD ? un < n : (un = dyn_take(ctr, lane)) < n) {
        tl = AHEAD ? tln : a.tiles[a.tile_begin + un];
        ntensor = tl.tensor;
        ntd = a.tensors[ntensor];   // (reusing ctd for the same tensor cost 2-6 % on FP32 paths)
        if constexpr (AHEAD) {
          un = dyn_take(ctr, lane);
          if (un < n) tln = a.tiles[a.tile_begin + un];
        }
        pass = 0;
        ne0 = tl.start + lane * 8;
        ncnt = min(8, (int)tl.len - lane * 8);
      } else {
        have_next = false;
      }
      if (have_next) {
        if (ncnt == 8) load_full(ntd, ne0, reset, nxt);
        else if (ncnt > 0) load_partial(ntd, ne0, ncnt, reset, nxt);
      }
      if (ccnt > 0)
        same += update_store<GT, COMBO, ALGO, SR>(ctd, ce0, ccnt, cur, coef, sc, ctensor, a.rk, a.step32, count,
                                                  a.neg_zero2);
      cur = nxt;
      ctd = ntd;
      ctensor = ntensor;
      ce0 = ne0;
      ccnt = ncnt;
      have = have_next;
    }
  }
  if (count) {
    // integer sums: the total does not depend on the order of the atomics
    same = __reduce_add_sync(0xFFFFFFFFu, same);
    if (lane == 0 && same) atomicAdd(a.unchanged, (unsigned long long)same);
  }
  dyn_done(ctr, lane);
}

// As many CTAs as are resident (occupancy cached), but no more than the
// tiles need at one tile per warp.
template <int GT, int COMBO, int ALGO, bool SR, bool DEVSC>
cudaError_t launch_dyn(const StepArgs& a, int sm_count, cudaStream_t s) {
  const int64_t n = a.tile_end - a.tile_begin;
  if (n <= 0) return cudaSuccess;
  if (a.dyn == nullptr) return cudaErrorInvalidValue;     // the kernel needs the counter
  auto k = step_dyn_kernel<GT, COMBO, ALGO, SR, DEVSC>;
  static OccupancyCache occ;
  const int per_sm = cached_occupancy(k, occ, kStepThreads, 0);
  if (per_sm < 1) return cudaGetLastError();
  const int64_t full = (int64_t)per_sm * sm_count;
  const int64_t need = (n + kStepThreads / 32 - 1) / (kStepThreads / 32);
  const int grid = (int)(need < full ? need : full);
  k<<<grid, kStepThreads, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace psopt
