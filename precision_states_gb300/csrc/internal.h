// internal.h -- host-side declarations shared by the API layer and the
// kernel launch files.
#pragma once

#include <atomic>
#include <cstdint>
#include <cuda_runtime.h>

#include "opt.h"

namespace psopt {

struct TensorDesc;
struct NormSlot;
struct NormChunk;
struct StepArgs;
struct SmallList;

// Resident CTAs per SM of one kernel, cached per device and safe to fill
// from several host threads.  The value is a property of the kernel and the
// architecture, but a dynamic shared-memory size above the default has to be
// enabled on each device, so the first launch on a device does that too.
constexpr int kMaxDevices = 64;
struct OccupancyCache {
  std::atomic<int> per_sm[kMaxDevices];
};

template <typename K>
inline int cached_occupancy(K kernel, OccupancyCache& cache, int threads, int smem_bytes) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) dev = -1;
  int v = dev >= 0 ? cache.per_sm[dev].load(std::memory_order_relaxed) : 0;
  if (v > 0) return v;
  if (smem_bytes > 48 * 1024 &&
      cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes) != cudaSuccess)
    return 0;      // the launch reports the error
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&v, kernel, threads, smem_bytes) != cudaSuccess || v < 1)
    v = 1;
  if (dev >= 0) cache.per_sm[dev].store(v, std::memory_order_relaxed);
  return v;
}

// state combinations (m_dtype, v_dtype) built into the library
enum StateCombo { SC_F32 = 0, SC_BF16_BF16 = 1, SC_BF16_E4M3 = 2, SC_BF16_E2M2 = 3 };
enum Algo { ALGO_ADAMW = 0, ALGO_ADEMAMIX = 1 };

int state_combo(int32_t m_dtype, int32_t v_dtype);   // -1 if not built
// whether the AdamW step of a state combination runs the staged kernel
// (tiles through shared memory by bulk copies, bounded waits)
__host__ __device__ constexpr inline bool step_is_staged(int combo, bool stochastic) {
  return combo != SC_F32 && (stochastic || combo == SC_BF16_BF16);
}

// Elements per tile of the step's work table: one 8-element group for each
// of the step kernel's 256 threads.
constexpr int64_t kTileElems = 2048;

// Table of pieces of at most elems[b] elements in bucket b (the norm's
// chunks, the step's tiles), bucketed by gradient dtype; see opt_chunk_table.
int64_t build_table(int32_t n, const int64_t* numel, const int32_t* grad_dtype, const int64_t elems[2],
                    opt_chunk* out, int64_t cap, int64_t bucket_begin[3]);
// the norm's chunk size for a dtype bucket (see OPT_NORM_CHUNK_MIN)
int64_t norm_chunk_elems(int32_t n, const int64_t* numel, const int32_t* grad_dtype, int bucket);

// The gradient norm: one pass-1 launch per non-empty dtype bucket b (chunks
// [bucket_begin[b], bucket_begin[b + 1]) into slots[b * OPT_NORM_SLOTS ...]),
// the last CTA to complete finishing into `out`.  `done` is a counter that is
// 0 between norms (the finishing CTA resets it).
cudaError_t launch_norm(const NormChunk* chunks, const int64_t bucket_begin[3], NormSlot* slots,
                        unsigned int* done, double max_norm, opt_norm_result* out, cudaStream_t s);

// fused step for one bucket (persistent grid of sm_count x occupancy CTAs)
cudaError_t launch_step_fp32_states(int grad_dtype, int algo, const StepArgs& args, int sm_count,
                                    cudaStream_t s);
// device step counter: advance it and write the step's scalars (base with
// the bias corrections of the new step) to `out`; or set it to `value`
cudaError_t launch_step_scalars(const opt_step_scalars& base, int64_t* counter, opt_step_scalars* out,
                                cudaStream_t s);
cudaError_t launch_set_step(int64_t* counter, int64_t value, cudaStream_t s);
cudaError_t launch_step_lowp_states(int grad_dtype, int combo, int stochastic, const StepArgs& args,
                                    int sm_count, cudaStream_t s);
// fused step for a short bucket (SmallList): one CTA per tile, descriptors
// in the kernel parameters; every state combination and algorithm
cudaError_t launch_step_small(int grad_dtype, int combo, int algo, int stochastic, const StepArgs& args,
                              const SmallList& list, cudaStream_t s);

// update-norm clipping (LAMB / max_unorm): the workspace, device pointers.
// A tensor's tiles are cut into segments of at most kLambSegTiles tiles;
// each segment's sums are reduced by one CTA of the ratio pass, and the last
// of a tensor's segments to finish (a per-tensor ticket) sums them in order.
constexpr int64_t kLambSegTiles = 2048;
struct LambWork {
  void* tile_sums;                 // per tile: sums of u^2 and p^2
  const int32_t* seg_tensor;       // per segment: its tensor
  const int64_t* seg_first;        // per segment: first tile
  const int32_t* seg_count;        // per segment: tiles (0 for an empty tensor)
  void* seg_sums;                  // per segment: sums of u^2 and p^2
  const int32_t* tensor_seg0;      // per tensor: first segment
  const int32_t* tensor_nseg;      // per tensor: segments (at least 1)
  unsigned int* tickets;           // per tensor: 0 between calls
  float* ratio;                    // per tensor: the trust ratio
  int n_segs;
};
// phase 0 = per-tile sums (one bucket), 1 = per-tensor ratios (all
// tensors), 2 = apply (one bucket)
cudaError_t launch_lamb(int grad_dtype, const StepArgs& args, const LambWork& w, float max_unorm,
                        int sm_count, cudaStream_t s, int phase);

// standalone codecs
cudaError_t launch_encode(const float* in, void* out, int64_t n, int dtype, int stochastic,
                          uint32_t seed_lo, uint32_t seed_hi, uint32_t tensor,
                          uint32_t step32, int sm_count, cudaStream_t s);
cudaError_t launch_decode(const void* in, float* out, int64_t n, int dtype, int sm_count,
                          cudaStream_t s);

}  // namespace psopt
