// norm.cu -- deterministic global gradient norm in one launch per gradient
// dtype.
//
// "perf(training): fused multi-tensor gradient-norm reduction" (NeMo
// Automodel PR #3685), 'Correctness properties': values are widened in
// registers (never squared in BF16), the decomposition into chunks comes from
// sizes only and no floating-point value is accumulated in arrival order, so
// the norm is bit-identical run to run; NaNs are counted because a max that
// ignores NaN would hide them.  (The only atomics are on integers -- which
// warp takes a chunk, the max of |g| as bits, the NaN and Inf counts, the
// completion ticket -- none of which changes a bit of the result.)
//
// GB300 design.  Blackwell Ultra's FP64 rate is a small fraction of its FP32
// rate, so one fp64 operation per element would make this streaming pass
// compute-bound.  Instead each lane accumulates squares in error-free
// float-float form (Knuth's TwoSum, exact; BF16 squares are exact in fp32 and
// FP32 squares are split exactly with an FMA), two values at a time with the
// packed f32x2 instructions.  A chunk is read by one warp; its lanes'
// float-float sums are merged in a fixed shuffle tree and converted to
// double once per chunk.  A chunk in which any lane's elements hold a NaN,
// an Inf, or a magnitude outside [2^-40, 2^40] (where fp32 squares could
// overflow or lose bits) is read again by the whole warp and summed in
// double -- a rare, exact slow path.
//
// Pass 1 runs OPT_NORM_SLOTS CTAs per dtype bucket, one per SM of a GB300,
// each of 24 warps.  Slot s owns chunks s, s + OPT_NORM_SLOTS, ... of the
// bucket (chunks of 4K-32K elements, the size from the bucket's size, each
// chunk's first element resolved to an address in the table); the slot's
// warps take its chunks one at a time from a counter in shared memory, and
// each chunk's sum, reduced by the warp that read it in a fixed shuffle
// tree, goes to the chunk's own place in shared memory.  The slot's total is
// those sums in chunk order.  Which warp read a chunk varies from run to run,
// but no value depends on it, so the norm is bit-identical run to run.
// (Against 912 CTAs of 128 threads, each summing a fixed set of chunks,
// 6 per SM: the CTAs of one SM ended a median 16 us apart on the 740-tensor
// list and 265 us apart on the Llama-3-8B list, because co-resident CTAs get
// unequal shares of the SM's bandwidth, however equal their work; with the
// warps of a whole SM sharing its chunks they end within about 20 us, and
// the Llama-3-8B norm fell from 2.377 to 2.215 ms.)  Pass 2, the finish,
// reduces all slots in a fixed order and derives norm2, the inf-norm, the
// NaN/Inf status and the clip coefficient.  It runs in whichever CTA of the
// last pass-1 launch completes last: every CTA publishes its slot, then
// takes a ticket from a completion counter; the CTA holding the last ticket
// finishes and resets the counter.  Fusing the finish into pass 1 saves a
// launch and the gap before it.
#include "common.cuh"
#include "internal.h"

namespace psopt {
namespace {

// 24 warps per CTA, one CTA per SM: each thread may hold 85 registers --
// eight 16-byte loads in flight that rotate (each register refilled as soon
// as its vector is summed) and two float-float chains (alternate vectors),
// so that the additions of one vector need not wait for the previous
// vector's.  The SM's 768 threads keep 96 KB in flight, as the 6 CTAs of
// 128 threads before them did.  (Measured in the same probe loop, with the
// AdamW step between norms: 16 warps of eight loads or 32 of six were
// 2-4 % slower.)
constexpr int kNormWarps = 24;
constexpr int kNormThreads = 32 * kNormWarps;
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

// What the finish needs, passed to every pass-1 launch of one norm.
struct NormFinish {
  const NormSlot* all;     // the slots it reduces, in this order
  int n_all;
  unsigned int n_ctas;     // CTAs of all pass-1 launches of this norm
  unsigned int* done;      // completion counter; 0 between norms
  double max_norm;
  opt_norm_result* out;
};

// One warp reduces n slots in a fixed order (lane l: slots l, l + 32, ... in
// order; then a butterfly, after which every lane holds the same values) and
// lane 0 writes the result.  The slots are read through L2, where the other
// CTAs' stores landed.
__device__ __forceinline__ void finish_slots(const NormSlot* __restrict__ slots, int n, double max_norm,
                                             opt_norm_result* __restrict__ out) {
  const int lane = threadIdx.x & 31;
  double sum = 0.0;
  unsigned long long nans = 0, infs = 0;
  float mx = 0.0f;
  for (int i = lane; i < n; i += 32) {
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
  if (lane != 0) return;
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

// One chunk, read and summed by one warp: lane l takes vectors l, l + 32,
// ... (kDepth loads in flight, rotating, into two float-float chains), the
// lane owning vector nvec loads the ragged tail element-wise.  Returns the
// chunk's sum of squares (the lanes' float-float sums merged in a fixed
// shuffle tree, lane 0's value), and adds its max |g| (fp32 bits) and NaN /
// Inf counts to the CTA's.  A chunk holding a NaN, an Inf or a magnitude
// outside [2^-40, 2^40] in any lane (fp32 squares could overflow or lose
// bits) is read again by all lanes and summed exactly in double: rare.
template <int GT>
__device__ __forceinline__ double chunk_sum(const char* __restrict__ g, uint32_t len, int lane,
                                            unsigned int* s_max, unsigned long long* s_nan,
                                            unsigned long long* s_inf) {
  using T = GradTraits<GT>;
  constexpr int V = T::kVec;
  const int nvec = (int)(len / V);
  const int rem = (int)(len % V);
  FF2 acc = {0ull, 0ull};
  uint32_t cmax = 0;
  int left = nvec > lane ? (nvec - lane + 31) / 32 : 0;
  const char* q = g + lane * 16;
  constexpr int kStep = 32 * 16;
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
  const bool owns_tail = rem > 0 && (nvec % 32) == lane;
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
  if (__all_sync(0xFFFFFFFFu, fast)) {
    float H = 0.0f, L = 0.0f, hx, hy, lx, ly;
    unpk(acc.hi, hx, hy);
    unpk(acc.lo, lx, ly);
    ff_merge(H, L, hx, lx);
    ff_merge(H, L, hy, ly);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float H2 = __shfl_xor_sync(0xFFFFFFFFu, H, o), L2 = __shfl_xor_sync(0xFFFFFFFFu, L, o);
      ff_merge(H, L, H2, L2);
    }
    const uint32_t wmax = __reduce_max_sync(0xFFFFFFFFu, cmax);
    if (lane == 0 && wmax) atomicMax(s_max, GT == OPT_BF16 ? (wmax << 16) : wmax);
    return (double)H + (double)L;      // lane 0's is the one kept
  }
  // the exact slow path, out of the fast path's registers
  double ds = 0.0;
  unsigned long long nn = 0, ni = 0;
  uint32_t mb = 0;
  auto visit = [&](float x) {
    if (x != x) { ++nn; return; }
    if (fabsf(x) == __int_as_float(0x7F800000)) { ++ni; return; }
    ds += (double)x * (double)x;
    mb = max(mb, f2u(fabsf(x)));
  };
  for (int vv = lane; vv < nvec; vv += 32)
    for (int j = 0; j < V; ++j) visit(T::elem(g, (int64_t)vv * V + j));
  if (owns_tail)
    for (int j = 0; j < rem; ++j) visit(T::elem(g, (int64_t)nvec * V + j));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    ds += __shfl_xor_sync(0xFFFFFFFFu, ds, o);
    nn += __shfl_xor_sync(0xFFFFFFFFu, nn, o);
    ni += __shfl_xor_sync(0xFFFFFFFFu, ni, o);
    mb = max(mb, __shfl_xor_sync(0xFFFFFFFFu, mb, o));
  }
  if (lane == 0) {
    if (nn) atomicAdd(s_nan, nn);
    if (ni) atomicAdd(s_inf, ni);
    if (mb) atomicMax(s_max, mb);
  }
  return ds;
}

template <int GT>
__global__ void __launch_bounds__(kNormThreads, 1)
norm_partials_kernel(const NormChunk* __restrict__ chunks, int64_t cbegin, int64_t cend,
                     NormSlot* __restrict__ slots, NormFinish fin) {
  __shared__ double s_part[OPT_NORM_MAX_PART];   // each chunk's sum, in chunk order
  __shared__ int s_next;                         // the next chunk to take
  __shared__ unsigned int s_max;                 // max |g|, fp32 bits (integer max: any order)
  __shared__ unsigned long long s_nan, s_inf;    // counts (integer sums: any order)
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int slot = blockIdx.x;
  // the slot's chunks: cbegin + slot + j * OPT_NORM_SLOTS, j < nj (at most
  // OPT_NORM_MAX_PART by the table's chunk size; a slot with more would be
  // a broken table: it reads nothing and reports a NaN, so that a step given
  // this norm is skipped)
  const int64_t first = cbegin + slot;
  const int64_t nj64 = first < cend ? (cend - 1 - first) / OPT_NORM_SLOTS + 1 : 0;
  const bool broken = nj64 > OPT_NORM_MAX_PART;
  const int nj = broken ? 0 : (int)nj64;
  if (tid == 0) {
    s_next = 0;
    s_max = 0u;
    s_nan = broken ? 1ull : 0ull;
    s_inf = 0ull;
  }
  __syncthreads();

  // Each warp takes a chunk, and takes the next one (and requests its table
  // entry) before it reads the current one, so that the entry's latency
  // hides behind the chunk.
  int j = 0;
  if (lane == 0) j = atomicAdd(&s_next, 1);
  j = __shfl_sync(0xFFFFFFFFu, j, 0);
  NormChunk cur = {nullptr, 0u, 0u};
  if (j < nj) cur = chunks[first + (int64_t)j * OPT_NORM_SLOTS];
  while (j < nj) {
    int jn = 0;
    if (lane == 0) jn = atomicAdd(&s_next, 1);
    jn = __shfl_sync(0xFFFFFFFFu, jn, 0);
    NormChunk nxt = {nullptr, 0u, 0u};
    if (jn < nj) nxt = chunks[first + (int64_t)jn * OPT_NORM_SLOTS];
    const double part = chunk_sum<GT>(static_cast<const char*>(cur.ptr), cur.len, lane, &s_max, &s_nan, &s_inf);
    if (lane == 0) s_part[j] = part;
    j = jn;
    cur = nxt;
  }
  __syncthreads();
  if (warp != 0) return;

  // warp 0: the slot's total, its chunks' sums in chunk order (lane l:
  // chunks l, l + 32, ...; then a butterfly), published with a ticket
  double sum = 0.0;
  for (int k = lane; k < nj; k += 32) sum += s_part[k];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xFFFFFFFFu, sum, o);
  unsigned int ticket = 0;
  if (lane == 0) {
    NormSlot r;
    r.sum = sum;
    r.nan_count = s_nan;
    r.inf_count = s_inf;
    r.maxabs = u2f(s_max);
    r.pad = 0;
    slots[slot] = r;
    __threadfence();                         // the slot is visible before the ticket
    ticket = atomicAdd(fin.done, 1u);
  }
  ticket = __shfl_sync(0xFFFFFFFFu, ticket, 0);
  if (ticket != fin.n_ctas - 1) return;
  __threadfence();                           // every other CTA's slot is visible now
  finish_slots(fin.all, fin.n_all, fin.max_norm, fin.out);
  if (lane == 0) *fin.done = 0u;
}

// The finish alone, for a norm over no elements (no pass-1 launch).
__global__ void __launch_bounds__(32)
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
    norm_finalize_kernel<<<1, 32, 0, s>>>(slots, 0, max_norm, out);
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
