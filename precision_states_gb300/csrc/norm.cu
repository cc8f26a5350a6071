// norm.cu -- deterministic global gradient norm in one launch per gradient
// dtype.
//
// "perf(training): fused multi-tensor gradient-norm reduction" (NeMo
// Automodel PR #3685), 'Correctness properties': values are widened in
// registers (never squared in BF16), the decomposition into chunks comes from
// sizes only and there are no atomics, so the norm is bit-identical run to
// run; NaNs are counted because a max that ignores NaN would hide them.
//
// GB300 design.  Blackwell Ultra's FP64 rate is a small fraction of its FP32
// rate, so one fp64 operation per element would make this streaming pass
// compute-bound.  Instead each thread accumulates squares in error-free
// float-float form (Knuth's TwoSum, exact; BF16 squares are exact in fp32 and
// FP32 squares are split exactly with an FMA), two lanes at a time with the
// packed f32x2 instructions.  The per-chunk float-float sums are merged into
// a per-thread float-float accumulator, converted to double once per thread,
// and reduced across the CTA in double in a fixed tree.  Only a thread whose
// elements in a chunk hold a NaN, an Inf, or a magnitude outside
// [2^-40, 2^40] (where fp32 squares could overflow or lose bits) re-reads
// those elements and accumulates them in double -- a rare, exact slow path.
//
// Pass 1 runs OPT_NORM_SLOTS CTAs per dtype bucket; slot s sums chunks
// s, s + OPT_NORM_SLOTS, ... of the bucket in that order, each chunk's
// first element resolved to an address in the table.  (Giving each slot one
// contiguous, equal span of the bucket instead balanced the slots exactly
// but measured 2-4 % slower on GB300: in this order all CTAs stream one
// window of memory together.)  Pass 2, the finish, reduces all slots in a
// fixed order and derives norm2, the inf-norm, the NaN/Inf status and the
// clip coefficient.  It runs in whichever CTA of the last pass-1 launch
// completes last: every CTA publishes its slot, then takes a ticket from a
// completion counter; the CTA holding the last ticket finishes and resets
// the counter.  Which CTA that is varies from run to run, but the order of
// the reduction does not, so neither do the bits of the result.  Fusing the
// finish into pass 1 saves a launch and the gap before it: 2.5 % of the
// norm on the 740-tensor list, where the finish is a visible share; on the
// Llama-3-8B list it measured 0.2 % slower, with one counter or with
// sixteen (so not from contention on the counter).
#include "common.cuh"
#include "internal.h"

namespace psopt {
namespace {

// 128 threads and 6 CTAs per SM: the 912 slots are one wave on GB300's 152
// SMs, and each thread may hold 85 registers -- enough for eight 16-byte
// loads in flight that rotate (each register refilled as soon as its vector
// is summed) and two float-float chains (alternate vectors), so that the
// additions of one vector need not wait for the previous vector's.  Per-CTA
// timestamps on GB300 showed the pass bound by each SM's throughput (every
// SM finishing at the same time however the work was split), so the lever
// is bytes in flight per SM, not balance.  Measured against 8 CTAs per SM
// with four loads each (in a loop with the AdamW step between norms):
// Llama-3-8B list 2.453 -> 2.380 ms, 740-tensor list 0.0850 -> 0.0818 ms;
// with L2 clean before the norm, 0.0773 -> 0.0746 ms.  (Also measured: 608
// CTAs of 256 threads with six loads, 456 of 256 with eight -- close
// behind; a ring of 16 KB stages filled by one producer lane's bulk copies,
// 1 to 3 CTAs per SM -- 3-27 % slower on the 740-tensor list; chunks of 16K
// or 8K elements -- within 1.5 %; a finish that issues all its slot loads
// up front -- no change: its time is a chain of latencies.  Earlier, against
// 256 threads at the 32-register cap with four loads issued together: eight
// cp.async copies per thread into shared-memory slots were 3 and 12 %
// slower; 32-byte loads read no faster than 16-byte ones in this order.)
// Plain reads in the same order reach 7.44 TB/s on GB300.
constexpr int kNormThreads = 128;
constexpr int kDepth = 8;            // 16-byte loads in flight per thread

// Two float-float accumulators (lane x, lane y): value = hi + lo per lane.
struct FF2 {
  f2_t hi, lo;
};

// TwoSum of hi and x per lane; the exact rounding error goes into lo.
__device__ __forceinline__ void ff2_add(FF2& a, f2_t x) {
  const f2_t s = add2(a.hi, x);
  const f2_t bb = sub2(s, a.hi);
  const f2_t aa = sub2(s, bb);
  const f2_t e = add2(sub2(a.hi, aa), sub2(x, bb));
  a.lo = add2(a.lo, e);
  a.hi = s;
}

// BF16 pair in one 32-bit word -> exact squares of both, added.
__device__ __forceinline__ void acc_bf16x2(FF2& a, uint32_t w) {
  const f2_t x = pk(u2f(w << 16), u2f(w & 0xFFFF0000u));
  ff2_add(a, mul2(x, x));
}

// FP32 pair: x*x = p + pe exactly (FMA split), both parts added.
__device__ __forceinline__ void acc_f32x2(FF2& a, float x0, float x1) {
  const f2_t x = pk(x0, x1);
  const f2_t p = mul2(x, x);
  const f2_t pe = fma2(x, x, p ^ 0x8000000080000000ull);   // x*x - p, exact
  ff2_add(a, p);
  a.lo = add2(a.lo, pe);
}

// Scalar float-float accumulator (H, L) += (h, l).
__device__ __forceinline__ void ff_merge(float& H, float& L, float h, float l) {
  const float s = __fadd_rn(H, h);
  const float bb = __fsub_rn(s, H);
  const float aa = __fsub_rn(s, bb);
  float e = __fadd_rn(__fsub_rn(H, aa), __fsub_rn(h, bb));
  e = __fadd_rn(e, __fadd_rn(L, l));
  H = __fadd_rn(s, e);
  L = __fsub_rn(e, __fsub_rn(H, s));
}

template <int GT>
struct GradTraits;
template <>
struct GradTraits<OPT_BF16> {
  static constexpr int kVec = 8;                 // elements per 16-byte vector
  static constexpr uint32_t kHi = 0x5380u;       // |g| <= 2^40 (BF16 bits)
  static constexpr uint32_t kLo = 0x2B80u;       // |g| >= 2^-40
  __device__ static float elem(const void* g, int64_t i) {
    return u2f((uint32_t)(static_cast<const uint16_t*>(g)[i]) << 16);
  }
};
template <>
struct GradTraits<OPT_F32> {
  static constexpr int kVec = 4;
  static constexpr uint32_t kHi = 0x53800000u;   // 2^40
  static constexpr uint32_t kLo = 0x2B800000u;   // 2^-40
  __device__ static float elem(const void* g, int64_t i) {
    return static_cast<const float*>(g)[i];
  }
};

// Accumulate one 16-byte vector; returns the max of |x| bits over it.
template <int GT>
__device__ __forceinline__ uint32_t acc_vec(FF2& a, uint4 w);

template <>
__device__ __forceinline__ uint32_t acc_vec<OPT_BF16>(FF2& a, uint4 w) {
  acc_bf16x2(a, w.x);
  acc_bf16x2(a, w.y);
  acc_bf16x2(a, w.z);
  acc_bf16x2(a, w.w);
  const uint32_t m = __vmaxu2(__vmaxu2(w.x & 0x7FFF7FFFu, w.y & 0x7FFF7FFFu),
                              __vmaxu2(w.z & 0x7FFF7FFFu, w.w & 0x7FFF7FFFu));
  return max(m & 0xFFFFu, m >> 16);
}

template <>
__device__ __forceinline__ uint32_t acc_vec<OPT_F32>(FF2& a, uint4 w) {
  acc_f32x2(a, u2f(w.x), u2f(w.y));
  acc_f32x2(a, u2f(w.z), u2f(w.w));
  return max(max(w.x & 0x7FFFFFFFu, w.y & 0x7FFFFFFFu), max(w.z & 0x7FFFFFFFu, w.w & 0x7FFFFFFFu));
}

// Exact slow path over one thread's own elements of a chunk (rare: only
// when they hold a NaN, an Inf or an extreme magnitude).  Its accumulators
// live in shared memory, one per thread, so that they hold no registers on
// the fast path.
struct SlowAcc {
  double sum;
  unsigned long long nans, infs;
  uint32_t mxbits;
  uint32_t pad;
};

template <int GT>
__device__ __noinline__ void slow_chunk(const char* g, int nvec, int rem, int tid, bool owns_tail,
                                        SlowAcc& a) {
  using T = GradTraits<GT>;
  constexpr int V = T::kVec;
  auto visit = [&](float x) {
    if (x != x) { ++a.nans; return; }
    if (fabsf(x) == __int_as_float(0x7F800000)) { ++a.infs; return; }
    a.sum += (double)x * (double)x;
    a.mxbits = max(a.mxbits, f2u(fabsf(x)));
  };
  for (int vv = tid; vv < nvec; vv += kNormThreads)
    for (int j = 0; j < V; ++j) visit(T::elem(g, (int64_t)vv * V + j));
  if (owns_tail)
    for (int j = 0; j < rem; ++j) visit(T::elem(g, (int64_t)nvec * V + j));
}

// What the finish needs, passed to every pass-1 launch of one norm.
struct NormFinish {
  const NormSlot* all;     // the slots it reduces, in this order
  int n_all;
  unsigned int n_ctas;     // CTAs of all pass-1 launches of this norm
  unsigned int* done;      // completion counter; 0 between norms
  double max_norm;
  opt_norm_result* out;
};

// One CTA reduces n slots in a fixed order (a strided sum per thread, then
// fixed shuffle and shared-memory trees) and writes the result.  The slots
// are read through L2, where the other CTAs' stores landed.
__device__ __forceinline__ void finish_slots(const NormSlot* __restrict__ slots, int n, double max_norm,
                                             opt_norm_result* __restrict__ out) {
  constexpr int kWarps = kNormThreads / 32;
  __shared__ double s_sum[kWarps];
  __shared__ unsigned long long s_nan[kWarps], s_inf[kWarps];
  __shared__ float s_max[kWarps];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  double sum = 0.0;
  unsigned long long nans = 0, infs = 0;
  float mx = 0.0f;
#pragma unroll 4
  for (int i = tid; i < n; i += kNormThreads) {
    const uint4* q = reinterpret_cast<const uint4*>(slots + i);
    const uint4 a = __ldcg(q), b = __ldcg(q + 1);
    sum += __hiloint2double((int)a.y, (int)a.x);
    nans += ((unsigned long long)a.w << 32) | a.z;
    infs += ((unsigned long long)b.y << 32) | b.x;
    mx = fmaxf(mx, __uint_as_float(b.z));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    sum += __shfl_xor_sync(0xFFFFFFFFu, sum, o);
    nans += __shfl_xor_sync(0xFFFFFFFFu, nans, o);
    infs += __shfl_xor_sync(0xFFFFFFFFu, infs, o);
    mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o));
  }
  if (lane == 0) {
    s_sum[warp] = sum;
    s_nan[warp] = nans;
    s_inf[warp] = infs;
    s_max[warp] = mx;
  }
  __syncthreads();
  if (tid != 0) return;
  sum = 0.0;
  nans = infs = 0;
  mx = 0.0f;
  for (int w = 0; w < kWarps; ++w) {
    sum += s_sum[w];
    nans += s_nan[w];
    infs += s_inf[w];
    mx = fmaxf(mx, s_max[w]);
  }
  opt_norm_result r;
  r.nan_count = nans;
  r.inf_count = infs;
  if (nans > 0) {
    r.sumsq = r.norm2 = r.norm_inf = __longlong_as_double(0x7FF8000000000000ll);
    r.clip_coef = 1.0f;
    r.status = OPT_ENONFINITE;
  } else if (infs > 0) {
    r.sumsq = r.norm2 = r.norm_inf = __longlong_as_double(0x7FF0000000000000ll);
    r.clip_coef = 1.0f;
    r.status = OPT_ENONFINITE;
  } else {
    r.sumsq = sum;
    r.norm2 = sqrt(sum);
    r.norm_inf = (double)mx;
    double coef = 1.0;
    if (max_norm > 0.0) {
      coef = max_norm / (r.norm2 + 1e-6);
      if (coef > 1.0) coef = 1.0;
    }
    r.clip_coef = (float)coef;
    r.status = OPT_OK;
  }
  *out = r;
}

template <int GT>
__global__ void __launch_bounds__(kNormThreads, 6)
norm_partials_kernel(const NormChunk* __restrict__ chunks, int64_t cbegin, int64_t cend,
                     NormSlot* __restrict__ slots, NormFinish fin) {
  using T = GradTraits<GT>;
  constexpr int V = T::kVec;
  const int tid = threadIdx.x;
  const int slot = blockIdx.x;

  __shared__ SlowAcc s_slow[kNormThreads];
  s_slow[tid] = SlowAcc{0.0, 0ull, 0ull, 0u, 0u};
  float AH = 0.0f, AL = 0.0f;      // fast-path float-float accumulator
  uint32_t mxbits = 0;             // fast-path max |g|, fp32 bits

  // The slot's chunks are c = cbegin + slot + k * OPT_NORM_SLOTS.  A table
  // entry holds the chunk's resolved address, so a chunk starts after one
  // 16-byte load.
  for (int64_t c = cbegin + slot; c < cend; c += OPT_NORM_SLOTS) {
    const NormChunk cur = chunks[c];
    const char* g = static_cast<const char*>(cur.ptr);
    const int nvec = (int)(cur.len / V);
    const int rem = (int)(cur.len % V);

    FF2 acc = {0ull, 0ull};
    uint32_t cmax = 0;
    // this thread's vectors tid, tid + T, ...: kDepth 16-byte loads in
    // flight, rotating -- each register is refilled with the vector kDepth
    // ahead as soon as it has been used -- and two summation chains
    int left = nvec > tid ? (nvec - tid + kNormThreads - 1) / kNormThreads : 0;
    const char* q = g + tid * 16;
    constexpr int kStep = kNormThreads * 16;
    if (left >= kDepth) {
      uint4 w[kDepth];
      FF2 acc2 = {0ull, 0ull};     // a second chain: odd vectors of a round
#pragma unroll
      for (int d = 0; d < kDepth; ++d) w[d] = ld_nc_u4(q + d * kStep);
      q += kDepth * kStep;
      for (left -= kDepth; left >= kDepth; left -= kDepth, q += kDepth * kStep) {
#pragma unroll
        for (int d = 0; d < kDepth; ++d) {
          cmax = max(cmax, acc_vec<GT>((d & 1) ? acc2 : acc, w[d]));
          w[d] = ld_nc_u4(q + d * kStep);
        }
      }
#pragma unroll
      for (int d = 0; d < kDepth; ++d) cmax = max(cmax, acc_vec<GT>((d & 1) ? acc2 : acc, w[d]));
      // fold the second chain in: float-float sum of the two, lane-wise
      const f2_t s = add2(acc.hi, acc2.hi);
      const f2_t bb = sub2(s, acc.hi);
      const f2_t aa = sub2(s, bb);
      const f2_t e = add2(sub2(acc.hi, aa), sub2(acc2.hi, bb));
      acc.lo = add2(add2(acc.lo, acc2.lo), e);
      acc.hi = s;
    }
    for (; left > 0; --left, q += kStep) cmax = max(cmax, acc_vec<GT>(acc, ld_nc_u4(q)));
    // ragged tail: the thread that would own vector nvec loads it element-wise
    const bool owns_tail = rem > 0 && (nvec % kNormThreads) == tid;
    if (owns_tail) {
      uint32_t wv[4] = {0u, 0u, 0u, 0u};
      for (int j = 0; j < rem; ++j) {
        const uint32_t bits = f2u(T::elem(g, (int64_t)nvec * V + j));
        if (GT == OPT_BF16) wv[j >> 1] |= (bits >> 16) << (16 * (j & 1));
        else                wv[j] = bits;
      }
      cmax = max(cmax, acc_vec<GT>(acc, make_uint4(wv[0], wv[1], wv[2], wv[3])));
    }

    const bool fast = cmax <= T::kHi && (cmax >= T::kLo || cmax == 0u);
    if (fast) {
      float hx, hy, lx, ly;
      unpk(acc.hi, hx, hy);
      unpk(acc.lo, lx, ly);
      ff_merge(AH, AL, hx, lx);
      ff_merge(AH, AL, hy, ly);
      mxbits = max(mxbits, GT == OPT_BF16 ? (cmax << 16) : cmax);
    } else {
      slow_chunk<GT>(g, nvec, rem, tid, owns_tail, s_slow[tid]);
    }
  }

  // fixed-order CTA reduction in double
  __shared__ double s_sum[kNormThreads];
  __shared__ unsigned long long s_nan[kNormThreads], s_inf[kNormThreads];
  __shared__ uint32_t s_max[kNormThreads];
  const SlowAcc slow = s_slow[tid];
  s_sum[tid] = ((double)AH + (double)AL) + slow.sum;
  s_nan[tid] = slow.nans;
  s_inf[tid] = slow.infs;
  s_max[tid] = max(mxbits, slow.mxbits);
  __syncthreads();
  for (int w = kNormThreads / 2; w > 0; w >>= 1) {
    if (tid < w) {
      s_sum[tid] += s_sum[tid + w];
      s_nan[tid] += s_nan[tid + w];
      s_inf[tid] += s_inf[tid + w];
      s_max[tid] = max(s_max[tid], s_max[tid + w]);
    }
    __syncthreads();
  }
  __shared__ unsigned int s_ticket;
  if (tid == 0) {
    NormSlot r;
    r.sum = s_sum[0];
    r.nan_count = s_nan[0];
    r.inf_count = s_inf[0];
    r.maxabs = u2f(s_max[0]);
    r.pad = 0;
    slots[slot] = r;
    __threadfence();                         // the slot is visible before the ticket
    s_ticket = atomicAdd(fin.done, 1u);
  }
  __syncthreads();
  if (s_ticket != fin.n_ctas - 1) return;
  __threadfence();                           // every other CTA's slot is visible now
  finish_slots(fin.all, fin.n_all, fin.max_norm, fin.out);
  if (tid == 0) *fin.done = 0u;
}

// The finish alone, for a norm over no elements (no pass-1 launch).
__global__ void __launch_bounds__(kNormThreads)
norm_finalize_kernel(const NormSlot* __restrict__ slots, int n, double max_norm,
                     opt_norm_result* __restrict__ out) {
  finish_slots(slots, n, max_norm, out);
}

}  // namespace

cudaError_t launch_norm(const NormChunk* chunks, const int64_t bucket_begin[3], NormSlot* slots,
                        unsigned int* done, double max_norm, opt_norm_result* out, cudaStream_t s) {
  int used[2], nb = 0;
  for (int b = 0; b < 2; ++b)
    if (bucket_begin[b + 1] > bucket_begin[b]) used[nb++] = b;
  if (nb == 0) {
    norm_finalize_kernel<<<1, kNormThreads, 0, s>>>(slots, 0, max_norm, out);
    return cudaGetLastError();
  }
  NormFinish fin;
  fin.all = slots + used[0] * OPT_NORM_SLOTS;
  fin.n_all = (used[nb - 1] - used[0] + 1) * OPT_NORM_SLOTS;
  fin.n_ctas = (unsigned int)(nb * OPT_NORM_SLOTS);
  fin.done = done;
  fin.max_norm = max_norm;
  fin.out = out;
  for (int k = 0; k < nb; ++k) {
    const int b = used[k];
    NormSlot* sl = slots + b * OPT_NORM_SLOTS;
    if (b == 0)
      norm_partials_kernel<OPT_F32><<<OPT_NORM_SLOTS, kNormThreads, 0, s>>>(chunks, bucket_begin[0],
                                                                          bucket_begin[1], sl, fin);
    else
      norm_partials_kernel<OPT_BF16><<<OPT_NORM_SLOTS, kNormThreads, 0, s>>>(chunks, bucket_begin[1],
                                                                           bucket_begin[2], sl, fin);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
      // a launch that did not start leaves the counter short of its target:
      // clear it behind the launches that did
      if (k > 0) cudaMemsetAsync(done, 0, sizeof(unsigned int), s);
      return e;
    }
  }
  return cudaSuccess;
}

}  // namespace psopt
