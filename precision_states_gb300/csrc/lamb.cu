// lamb.cu -- deterministic update-norm clipping (the LAMB / max_unorm path)
// over a plan's tiles, FP32 states.
//
// "Investigate SM103 bias-correction broadcast in 32-bit optimizers",
// 'Problem' and 'B300 result': the 2-state optimizers' max_unorm > 0 path
// measures the norm of a tensor's whole update before applying it, and its
// cross-CTA atomicAdd made that norm -- and every step after it -- differ from
// run to run.  Here the norms come from fixed slots reduced in a fixed order,
// so the result is bit-identical run to run:
//   pass 1 (lamb_stats_kernel): per tile, update m and v (stored), form the
//     AdamW direction u and write the tile's sums of u^2 and p^2 (old p) to
//     the tile's own slot;
//   pass 2 (lamb_ratio_kernel): one CTA per segment of at most
//     kLambSegTiles of a tensor's tiles sums their slots in a fixed order;
//     the last of the tensor's segments to finish (a per-tensor ticket) sums
//     the segments in order and sets ratio = max_unorm |p| / |u| when
//     |u| > max_unorm |p|, else 1 (one CTA per tensor took 0.27 ms on the
//     Llama-3-8B list, whose embedding and head have 256K tiles each; with
//     segments the LAMB step fell from 45.66 to 45.42 ms there, GB300);
//   pass 3 (lamb_apply_kernel): per element, u again from the stored m and v
//     (the same operations, so the same bits), p <- p (1 - lr wd) - lr ratio u.
// Traffic: pass 1 reads p, g, m, v and writes m, v; pass 3 reads p, m, v and
// writes p: 38 B per parameter with BF16 gradients.
#include "step_dyn.cuh"
#include "step_kernel.cuh"

namespace psopt {
namespace {

constexpr int kLambThreads = kStepThreads;
constexpr int kLambMinBlocks = 2;     // <= 128 registers per thread

struct TileSums {
  double su, sp;   // sum of u^2 and of p^2 over the tile
};

// the AdamW direction of one element from its new moments (shared by both passes)
__device__ __forceinline__ float lamb_dir(float mn, float vn, const opt_step_scalars& sc) {
  const float num = __fmul_rn(mn, sc.inv_bc1);
  const float den = __fadd_rn(sqrt_approx(__fmul_rn(vn, sc.inv_bc2)), sc.eps);
  return div_approx(num, den);
}

// The streaming passes take their tiles as warps free up: a warp takes whole
// tiles from the plan's counter (one atomic per tile, a tile ahead) and
// covers each in passes of 256 elements, lane l taking elements
// base + 8 l .. + 7 of each pass.  body(td, e0, cnt) works on the lane's
// group (cnt <= 0: none in this pass); tile_done(i) runs, warp-wide, after
// tile i's last pass, so pass 1 reduces each tile within one warp and needs
// no CTA barrier.  Measured on GB300 against fixed shares per CTA (pass 1
// with one CTA barrier per tile), A/B/A/B: the LAMB step on the Llama-3-8B
// list went from 45.40 to 42.40 ms (1.003 -> 1.074 of the measured copy
// bandwidth), on the 740-tensor list from 1.028 to 1.022.
template <typename Body, typename TileDone>
__device__ __forceinline__ void warp_tiles(const StepArgs& a, int lane, Body body, TileDone tile_done) {
  const int64_t n = a.tile_end - a.tile_begin;
  unsigned long long* ctr = a.dyn;
  int64_t u = dyn_take(ctr, lane);
  if (u < n) {
    opt_chunk tl = a.tiles[a.tile_begin + u];
    int64_t un = dyn_take(ctr, lane);
    opt_chunk tln{};
    if (un < n) tln = a.tiles[a.tile_begin + un];
    for (;;) {
      const TensorDesc td = a.tensors[tl.tensor];
      for (int base = 0; base < (int)tl.len; base += 256) {
        const int o = base + lane * 8;
        body(td, tl.tensor, tl.start + o, min(8, (int)tl.len - o));
      }
      tile_done(a.tile_begin + u);
      if (un >= n) break;
      u = un;
      tl = tln;
      un = dyn_take(ctr, lane);
      if (un < n) tln = a.tiles[a.tile_begin + un];
    }
  }
  dyn_done(ctr, lane);
}

template <int GT>
__global__ void __launch_bounds__(kLambThreads, kLambMinBlocks)
lamb_stats_kernel(const StepArgs a, TileSums* __restrict__ sums) {
  float coef = 1.0f;
  if (a.d_norm != nullptr) {
    if (a.d_norm->status != OPT_OK) return;
    coef = a.d_norm->clip_coef;
  }
  const int lane = threadIdx.x & 31;
  float su = 0.0f, sp = 0.0f;          // this lane's sums over its groups of the tile
  auto body = [&](const TensorDesc& td, uint32_t, int64_t e0, int cnt) {
    if (cnt <= 0) return;
    Frag<GT, SC_F32, ALGO_ADAMW> f;
    if (cnt == 8) load_full(td, e0, false, f);
    else load_partial(td, e0, cnt, false, f);
    float mn[8], vn[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float g = GT == OPT_BF16 ? bf16_dec(code_at<16>(f.g, j)) : u2f(f.g[j]);
      const float ge = __fmul_rn(g, coef);
      mn[j] = __fadd_rn(__fmul_rn(a.sc.beta1, u2f(f.m[j])), __fmul_rn(a.sc.omb1, ge));
      vn[j] = __fadd_rn(__fmul_rn(a.sc.beta2, u2f(f.v[j])), __fmul_rn(a.sc.omb2, __fmul_rn(ge, ge)));
      if (j < cnt) {
        const float u = lamb_dir(mn[j], vn[j], a.sc);
        su = __fadd_rn(su, __fmul_rn(u, u));
        sp = __fadd_rn(sp, __fmul_rn(u2f(f.p[j]), u2f(f.p[j])));
      }
    }
    if (cnt == 8) {
      st_cs_u4(static_cast<float*>(td.m) + e0, make_uint4(f2u(mn[0]), f2u(mn[1]), f2u(mn[2]), f2u(mn[3])));
      st_cs_u4(static_cast<float*>(td.m) + e0 + 4, make_uint4(f2u(mn[4]), f2u(mn[5]), f2u(mn[6]), f2u(mn[7])));
      st_cs_u4(static_cast<float*>(td.v) + e0, make_uint4(f2u(vn[0]), f2u(vn[1]), f2u(vn[2]), f2u(vn[3])));
      st_cs_u4(static_cast<float*>(td.v) + e0 + 4, make_uint4(f2u(vn[4]), f2u(vn[5]), f2u(vn[6]), f2u(vn[7])));
    } else {
      for (int j = 0; j < cnt; ++j) {
        static_cast<float*>(td.m)[e0 + j] = mn[j];
        static_cast<float*>(td.v)[e0 + j] = vn[j];
      }
    }
  };
  // the tile's sums: the lanes' fp32 sums in double, a fixed butterfly
  auto tile_done = [&](int64_t i) {
    double tu = (double)su, tp = (double)sp;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      tu += __shfl_xor_sync(0xFFFFFFFFu, tu, o);
      tp += __shfl_xor_sync(0xFFFFFFFFu, tp, o);
    }
    if (lane == 0) sums[i] = TileSums{tu, tp};
    su = 0.0f;
    sp = 0.0f;
  };
  warp_tiles(a, lane, body, tile_done);
}

// One CTA per segment (a tensor's tiles are contiguous in the table, its
// segments consecutive).  Thread k sums the segment's tiles k, k + T, ... in
// order, then a fixed tree; the CTA that takes a tensor's last ticket sums
// the tensor's segments in order (warp 0: lane-strided, then a butterfly),
// writes the ratio and returns the ticket to 0.
__global__ void __launch_bounds__(kLambThreads)
lamb_ratio_kernel(LambWork w, float max_unorm, const opt_norm_result* d_norm) {
  if (d_norm != nullptr && d_norm->status != OPT_OK) return;
  __shared__ double s_u[kLambThreads], s_p[kLambThreads];
  __shared__ unsigned int s_ticket;
  const TileSums* __restrict__ sums = static_cast<const TileSums*>(w.tile_sums);
  TileSums* __restrict__ segs = static_cast<TileSums*>(w.seg_sums);
  const int sg = blockIdx.x;
  const int t = w.seg_tensor[sg];
  const int64_t first = w.seg_first[sg];
  const int count = w.seg_count[sg];
  double su = 0.0, sp = 0.0;
  for (int k = threadIdx.x; k < count; k += kLambThreads) {
    su += sums[first + k].su;
    sp += sums[first + k].sp;
  }
  s_u[threadIdx.x] = su;
  s_p[threadIdx.x] = sp;
  __syncthreads();
  for (int h = kLambThreads / 2; h > 0; h >>= 1) {
    if ((int)threadIdx.x < h) {
      s_u[threadIdx.x] += s_u[threadIdx.x + h];
      s_p[threadIdx.x] += s_p[threadIdx.x + h];
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    TileSums r;
    r.su = s_u[0];
    r.sp = s_p[0];
    segs[sg] = r;
    __threadfence();                         // the segment's sums are visible before the ticket
    s_ticket = atomicAdd(&w.tickets[t], 1u);
  }
  __syncthreads();
  const int nseg = w.tensor_nseg[t];
  if (s_ticket != (unsigned int)(nseg - 1) || threadIdx.x >= 32) return;
  __threadfence();                           // every other segment's sums are visible now
  const int lane = threadIdx.x;
  const int s0 = w.tensor_seg0[t];
  su = 0.0;
  sp = 0.0;
  for (int k = lane; k < nseg; k += 32) {
    su += __ldcg(&segs[s0 + k].su);
    sp += __ldcg(&segs[s0 + k].sp);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    su += __shfl_xor_sync(0xFFFFFFFFu, su, o);
    sp += __shfl_xor_sync(0xFFFFFFFFu, sp, o);
  }
  if (lane == 0) {
    const double un = sqrt(su), pn = sqrt(sp);
    double r = 1.0;
    if (max_unorm > 0.0f && un > (double)max_unorm * pn && un > 0.0) r = (double)max_unorm * pn / un;
    w.ratio[t] = (float)r;
    w.tickets[t] = 0u;
  }
}

template <int GT>
__global__ void __launch_bounds__(kLambThreads, kLambMinBlocks)
lamb_apply_kernel(const StepArgs a, const float* __restrict__ ratio) {
  if (a.d_norm != nullptr && a.d_norm->status != OPT_OK) return;
  const int lane = threadIdx.x & 31;
  auto body = [&](const TensorDesc& td, uint32_t tensor, int64_t e0, int cnt) {
    if (cnt <= 0) return;
    const float r = ratio[tensor];
    float p[8], m[8], v[8];
    if (cnt == 8) {
      uint32_t w[8];
      ld_cs_x8(td.p + e0, td.a32 & kA32P, w);
      for (int j = 0; j < 8; ++j) p[j] = u2f(w[j]);
      ld_cs_x8(static_cast<const float*>(td.m) + e0, td.a32 & kA32M, w);
      for (int j = 0; j < 8; ++j) m[j] = u2f(w[j]);
      ld_cs_x8(static_cast<const float*>(td.v) + e0, td.a32 & kA32V, w);
      for (int j = 0; j < 8; ++j) v[j] = u2f(w[j]);
    } else {
      for (int j = 0; j < 8; ++j) {
        const bool in = j < cnt;
        p[j] = in ? td.p[e0 + j] : 0.0f;
        m[j] = in ? static_cast<const float*>(td.m)[e0 + j] : 0.0f;
        v[j] = in ? static_cast<const float*>(td.v)[e0 + j] : 0.0f;
      }
    }
    float pn[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float u = lamb_dir(m[j], v[j], a.sc);
      pn[j] = __fsub_rn(__fmul_rn(p[j], a.sc.decay), __fmul_rn(a.sc.lr, __fmul_rn(r, u)));
    }
    if (cnt == 8) {
      st_cs_u4(td.p + e0, make_uint4(f2u(pn[0]), f2u(pn[1]), f2u(pn[2]), f2u(pn[3])));
      st_cs_u4(td.p + e0 + 4, make_uint4(f2u(pn[4]), f2u(pn[5]), f2u(pn[6]), f2u(pn[7])));
    } else {
      for (int j = 0; j < cnt; ++j) td.p[e0 + j] = pn[j];
    }
  };
  warp_tiles(a, lane, body, [](int64_t) {});
}

// Persistent grid: CTAs resident at once (occupancy cached per kernel
// instance and device), at most one per unit of work.
template <typename K>
int grid_for_kernel(K k, OccupancyCache& occ, int sm_count, int64_t work) {
  const int64_t full = (int64_t)cached_occupancy(k, occ, kLambThreads, 0) * sm_count;
  return (int)(work < full ? work : full);
}

}  // namespace

cudaError_t launch_lamb(int grad_dtype, const StepArgs& a, const LambWork& w, float max_unorm, int sm_count,
                        cudaStream_t s, int phase) {
  const int64_t tiles = a.tile_end - a.tile_begin;
  if (a.dyn == nullptr) return cudaErrorInvalidValue;     // the streaming passes need the counter
  TileSums* ts = static_cast<TileSums*>(w.tile_sums);
  float* ratio = w.ratio;
  // one occupancy slot per kernel instance
  static OccupancyCache occ_stats[2], occ_apply[2];
  const int b = grad_dtype == OPT_BF16 ? 1 : 0;
  if (phase == 0) {
    if (tiles <= 0) return cudaSuccess;
    if (b) {
      auto k = lamb_stats_kernel<OPT_BF16>;
      k<<<grid_for_kernel(k, occ_stats[b], sm_count, tiles), kLambThreads, 0, s>>>(a, ts);
    } else {
      auto k = lamb_stats_kernel<OPT_F32>;
      k<<<grid_for_kernel(k, occ_stats[b], sm_count, tiles), kLambThreads, 0, s>>>(a, ts);
    }
  } else if (phase == 1) {
    if (w.n_segs <= 0) return cudaSuccess;
    lamb_ratio_kernel<<<w.n_segs, kLambThreads, 0, s>>>(w, max_unorm, a.d_norm);
  } else {
    if (tiles <= 0) return cudaSuccess;
    if (b) {
      auto k = lamb_apply_kernel<OPT_BF16>;
      k<<<grid_for_kernel(k, occ_apply[b], sm_count, tiles), kLambThreads, 0, s>>>(a, ratio);
    } else {
      auto k = lamb_apply_kernel<OPT_F32>;
      k<<<grid_for_kernel(k, occ_apply[b], sm_count, tiles), kLambThreads, 0, s>>>(a, ratio);
    }
  }
  return cudaGetLastError();
}

}  // namespace psopt
