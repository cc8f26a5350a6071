// step_bulk.cuh -- the fused AdamW step for low-precision states with its
// input tiles staged in shared memory by bulk copies from a producer warp.
//
// The same per-element work as step_kernel (update_store, so the same bits),
// fed differently.  In step_kernel every thread holds the raw words of its
// next group in registers; with the Philox draws and the encoders also live,
// the stochastic-rounding instantiations need ~120 registers, so only 16
// warps fit on an SM and few bytes are in flight per warp.  Here the words
// in flight live in shared memory:
//   - a CTA has kStepThreads consumer threads (8 warps) and one producer
//     warp, and a ring of S stages (4 or 5), each holding one whole tile
//     (2048 elements of p, g, m, v) and a header (the tile's table entry and
//     its tensor's descriptor);
//   - the producer (lane 0 of the last warp) runs up to S tiles
//     ahead: it waits for a stage to be released, writes the header, and
//     requests the tile with four cp.async.bulk copies completing on the
//     stage's "full" mbarrier (expect_tx with the byte count);
//   - the consumers wait on "full", take everything from shared memory
//     (header, then their 8 elements' words), release the stage (one arrive
//     per warp on its "empty" mbarrier) and run update_store, which stores to
//     global memory directly.
// The producer's dependent loads of the tile table and descriptors are thus
// hidden behind the ring.  A tile shorter than 2048 elements (the last tile
// of a tensor) is not copied: the producer completes "full" with a plain
// arrive and the consumers load it from global memory as step_kernel does.
//
// Every wait is bounded in time by %globaltimer: the producer's and the
// consumers' waits by a.wait_ns (the plan's limit, 2 s unless set).  A wait
// that runs out sets OPT_FLAG_WAIT_TIMEOUT in *a.err and the thread stops
// working.  Before a consumer warp leaves, it makes sure no copy still
// targets the stages: the producer, when it stops (at the end of its tiles,
// or when one of its own waits runs out), publishes in shared memory how
// many tiles it issued; the warp waits for that, then for every issued tile
// it has not consumed.  Those waits have their own, much longer limit
// (kDrainNs: issued copies land in microseconds), and if one of them runs
// out too, OPT_FLAG_DRAIN_TIMEOUT is set as well.  The host reads the flags
// with opt_plan_status.
//
// A wait drill (a.drill, OPT_STEP_WAIT_DRILL) makes the waits run out on
// purpose, with no fault: each CTA's producer withholds its first tile --
// no copy, no arrive, so nothing ever completes that stage's "full" phase --
// and issues the next S - 1 as usual.  Every consumer warp's first wait then
// runs out, the producer's wait for the withheld stage's release runs out
// too, and the consumers drain the S - 1 issued tiles (never the withheld
// one) before leaving.  No tile is processed: the step changes nothing.
#pragma once

#include "step_kernel.cuh"

namespace psopt {

constexpr int kSmemPerSm = 228 * 1024;                      // shared memory per SM
constexpr int kSmemReservedPerCta = 1024;                   // the runtime's share of each CTA
constexpr int kBulkConsumers = kStepThreads / 32;          // consumer warps
constexpr int kBulkThreads = kStepThreads + 32;            // + the producer warp
constexpr unsigned long long kDrainNs = 10000000000ull;    // 10 s beyond the wait limits

// Shared-memory layout: barriers, then S stages of {header, p, g, m, v};
// every part a multiple of 16 bytes.  S is 4, or 5 for BF16 v with nearest
// rounding where two CTAs still fit on an SM.  Measured on GB300 (GPT-2
// list, A/B/A/B on two boxes): a fifth stage lifted nearest BF16 v by
// 0.8-1.8 %, to 0.991-1.003 of the measured copy bandwidth; for the
// stochastic modes five or six stages cost 2-3 % (E2M2 0.927 -> 0.900, E4M3
// 0.967 -> 0.943, BF16 0.997 -> 0.981).
struct BulkHeader {
  opt_chunk tl;
  TensorDesc td;
};
static_assert(sizeof(BulkHeader) == 80, "BulkHeader layout");

template <int GT, int COMBO, bool SR>
struct BulkLayout {
  static constexpr int VD = Combo<COMBO>::V;
  static constexpr int N = (int)kTileElems;
  static constexpr int HDR = 128;
  static constexpr int P = 4 * N;
  static constexpr int G = (GT == OPT_BF16 ? 2 : 4) * N;
  static constexpr int M = 2 * N;                          // BF16 m
  static constexpr int V = VD == OPT_BF16 ? 2 * N : VD == OPT_E4M3 ? N : N / 2;
  static constexpr int OFF_P = HDR, OFF_G = OFF_P + P, OFF_M = OFF_G + G, OFF_V = OFF_M + M;
  static constexpr int STAGE = OFF_V + V;
  static constexpr int CTRL = 16;                          // producer's issued count, done flag
  static constexpr bool fits(int s) { return 2 * (16 * s + CTRL + STAGE * s + kSmemReservedPerCta) <= kSmemPerSm; }
  static constexpr int S = (!SR && COMBO == SC_BF16_BF16 && fits(5)) ? 5 : 4;
  static_assert(fits(S), "two CTAs per SM");
  static constexpr int OFF_CTRL = 16 * S;
  static constexpr int BAR_BYTES = 16 * S + CTRL;           // full[S], empty[S], control
  static constexpr int BYTES = BAR_BYTES + STAGE * S;
  static_assert(STAGE % 16 == 0 && BAR_BYTES % 16 == 0, "bulk copy alignment");
  static_assert(kStepThreads * 8 == N, "one tile per stage");
};

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
// Wait for the phase with the given parity to complete, at most limit_ns.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, unsigned long long limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_ns();
  while (!mbar_try_wait(bar, parity))
    if (global_ns() - t0 > limit_ns) return false;
  return true;
}
__device__ __forceinline__ void sts_volatile_u64(uint32_t a, unsigned long long v) {
  asm volatile("st.volatile.shared.u64 [%0], %1;" ::"r"(a), "l"(v) : "memory");
}
__device__ __forceinline__ unsigned long long lds_volatile_u64(uint32_t a) {
  unsigned long long v;
  asm volatile("ld.volatile.shared.u64 %0, [%1];" : "=l"(v) : "r"(a) : "memory");
  return v;
}
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}
__device__ __forceinline__ uint4 lds_u4(uint32_t a) {
  uint4 r;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "r"(a));
  return r;
}
__device__ __forceinline__ uint2 lds_u2(uint32_t a) {
  uint2 r;
  asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(r.x), "=r"(r.y) : "r"(a));
  return r;
}
__device__ __forceinline__ uint32_t lds_u1(uint32_t a) {
  uint32_t r;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(r) : "r"(a));
  return r;
}

template <int GT, int COMBO, bool SR>
__global__ void __launch_bounds__(kBulkThreads, 2)
step_bulk_kernel(const StepArgs a) {
  using L = BulkLayout<GT, COMBO, SR>;
  using F = Frag<GT, COMBO, ALGO_ADAMW>;
  constexpr int S = L::S;
  extern __shared__ __align__(128) unsigned char smem[];
  if (a.d_norm != nullptr && a.d_norm->status != OPT_OK) return;   // non-finite norm: leave all untouched
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t sbase = smem_u32(smem);
  const uint32_t full0 = sbase, empty0 = sbase + 8 * S;             // barrier of stage s: + 8 * s
  const uint32_t issued_at = sbase + L::OFF_CTRL, done_at = issued_at + 8;
  const uint32_t stage0 = sbase + L::BAR_BYTES;                     // stage s: + s * STAGE
  const bool reset = a.reset != 0;
  if (threadIdx.x == 0) {
    for (int st = 0; st < S; ++st) {
      mbar_init(full0 + 8 * st, 1);
      mbar_init(empty0 + 8 * st, kBulkConsumers);
    }
    sts_volatile_u64(issued_at, 0ull);
    sts_volatile_u64(done_at, 0ull);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();

  // The CTA's k-th tile is first + k * gridDim.x.
  const int64_t first = a.tile_begin + blockIdx.x;
  const int64_t stride = gridDim.x;
  const int64_t ntiles = first < a.tile_end ? (a.tile_end - 1 - first) / stride + 1 : 0;

  if (warp == kBulkConsumers) {
    // ---------------------------------------------------------- producer
    if (lane != 0) return;
    int64_t k = 0;
    for (; k < ntiles; ++k) {
      const int st = (int)(k % S);
      if (k >= S && !mbar_wait(empty0 + 8 * st, (uint32_t)(k / S - 1) & 1u, a.wait_ns)) {
        atomicOr(a.err, OPT_FLAG_WAIT_TIMEOUT);
        break;
      }
      if (k == 0 && a.drill) continue;     // withheld: no copy, no arrive
      BulkHeader h;
      h.tl = a.tiles[first + k * stride];
      h.td = a.tensors[h.tl.tensor];
      unsigned char* stage = smem + L::BAR_BYTES + st * L::STAGE;
      *reinterpret_cast<BulkHeader*>(stage) = h;
      const uint32_t bar = full0 + 8 * st, dst = stage0 + (uint32_t)st * L::STAGE;
      if ((int64_t)h.tl.len == kTileElems) {
        const int64_t e = h.tl.start;
        mbar_expect_tx(bar, L::P + L::G + (reset ? 0 : L::M + L::V));
        bulk_g2s(dst + L::OFF_P, h.td.p + e, L::P, bar);
        bulk_g2s(dst + L::OFF_G, static_cast<const char*>(h.td.g) + e * (L::G / L::N), L::G, bar);
        if (!reset) {
          bulk_g2s(dst + L::OFF_M, static_cast<const uint16_t*>(h.td.m) + e, L::M, bar);
          bulk_g2s(dst + L::OFF_V, static_cast<const char*>(h.td.v) + e * L::V / L::N, L::V, bar);
        }
      } else {
        mbar_arrive(bar);     // a short tile: nothing copied, the consumers load it directly
      }
    }
    // Tiles 0 .. k-1 are issued and no more will be: say so, for a consumer
    // warp that stopped early and must let those copies land before it
    // leaves (read only on that path).
    sts_volatile_u64(issued_at, (unsigned long long)k);
    __threadfence_block();
    sts_volatile_u64(done_at, 1ull);
    return;
  }

  // ------------------------------------------------------------ consumers
  float coef = 1.0f;
  if (a.d_norm != nullptr) coef = a.d_norm->clip_coef;
  const bool count = a.unchanged != nullptr;
  const int off = threadIdx.x * 8;
  uint32_t same = 0;
  int64_t k = 0;
  bool ok = true;
  for (; k < ntiles; ++k) {
    const int st = (int)(k % S);
    // one verdict for the warp, so that its lanes never part ways
    if (!__all_sync(0xFFFFFFFFu, mbar_wait(full0 + 8 * st, (uint32_t)(k / S) & 1u, a.wait_ns))) {
      ok = false;
      break;
    }
    const unsigned char* stage = smem + L::BAR_BYTES + st * L::STAGE;
    const BulkHeader h = *reinterpret_cast<const BulkHeader*>(stage);
    const int64_t e0 = h.tl.start + off;
    const int cnt = min(8, (int)h.tl.len - off);
    F f;
    if ((int64_t)h.tl.len == kTileElems) {
      const uint32_t base = stage0 + (uint32_t)st * L::STAGE;
      put4(f.p, lds_u4(base + L::OFF_P + 4 * off));
      put4(f.p + 4, lds_u4(base + L::OFF_P + 4 * off + 16));
      if constexpr (F::NG == 4) {
        put4(f.g, lds_u4(base + L::OFF_G + 2 * off));
      } else {
        put4(f.g, lds_u4(base + L::OFF_G + 4 * off));
        put4(f.g + 4, lds_u4(base + L::OFF_G + 4 * off + 16));
      }
      if (reset) {
#pragma unroll
        for (int q = 0; q < F::NM; ++q) f.m[q] = 0u;
#pragma unroll
        for (int q = 0; q < F::NV; ++q) f.v[q] = 0u;
      } else {
        put4(f.m, lds_u4(base + L::OFF_M + 2 * off));
        if constexpr (F::NV == 4) {
          put4(f.v, lds_u4(base + L::OFF_V + 2 * off));
        } else if constexpr (F::NV == 2) {
          const uint2 w = lds_u2(base + L::OFF_V + off);
          f.v[0] = w.x;
          f.v[1] = w.y;
        } else {
          f.v[0] = lds_u1(base + L::OFF_V + off / 2);
        }
      }
    } else if (cnt > 0) {
      if (cnt == 8) load_full(h.td, e0, reset, f);
      else load_partial(h.td, e0, cnt, reset, f);
    }
    // the stage is read: release it to the producer
    __syncwarp();
    if (lane == 0) mbar_arrive(empty0 + 8 * st);
    if (cnt > 0)
      same += update_store<GT, COMBO, ALGO_ADAMW, SR>(h.td, e0, cnt, f, coef, a.sc, h.tl.tensor, a.rk, a.step32,
                                                      count, a.neg_zero2);
  }
  if (!ok) {
    // A wait ran out: flag it, then let every copy that may still target a
    // stage land before leaving.  This warp released tiles 0 .. k-1 only, so
    // the producer issued at most tiles up to k + S - 1 (each needs every
    // warp's release of the tile S before it): one pending phase per stage.
    // Its own waits are bounded by wait_ns each, at most S + 1 of them after
    // this warp's last release.
    if (lane == 0) atomicOr(a.err, OPT_FLAG_WAIT_TIMEOUT);
    const unsigned long long t0 = global_ns();
    bool drained;
    while (!(drained = lds_volatile_u64(done_at) != 0ull))
      if (global_ns() - t0 > (unsigned long long)(S + 1) * a.wait_ns + kDrainNs) break;
    if (drained) {
      __threadfence_block();
      const int64_t issued = (int64_t)lds_volatile_u64(issued_at);
      for (int64_t q = (a.drill && k == 0) ? 1 : k; q < issued && drained; ++q)
        drained = mbar_wait(full0 + 8 * (int)(q % S), (uint32_t)(q / S) & 1u, kDrainNs);
    }
    if (!drained && lane == 0) atomicOr(a.err, OPT_FLAG_DRAIN_TIMEOUT);
    return;
  }
  if (count) {
    // integer sums: the total does not depend on the order of the atomics
    same = __reduce_add_sync(0xFFFFFFFFu, same);
    if (lane == 0 && same) atomicAdd(a.unchanged, (unsigned long long)same);
  }
}

// Persistent grid: as many CTAs as fit at once with this shared memory.
template <int GT, int COMBO, bool SR>
cudaError_t launch_bulk(const StepArgs& a, int sm_count, cudaStream_t s) {
  const int64_t n = a.tile_end - a.tile_begin;
  if (n <= 0) return cudaSuccess;
  auto k = step_bulk_kernel<GT, COMBO, SR>;
  constexpr int bytes = BulkLayout<GT, COMBO, SR>::BYTES;
  static OccupancyCache occ;
  const int per_sm = cached_occupancy(k, occ, kBulkThreads, bytes);
  if (per_sm < 1) return cudaGetLastError();
  const int64_t full = (int64_t)per_sm * sm_count;
  const int grid = (int)(n < full ? n : full);
  k<<<grid, kBulkThreads, bytes, s>>>(a);
  return cudaGetLastError();
}

}  // namespace psopt
