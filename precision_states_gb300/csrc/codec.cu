// codec.cu -- standalone conversion of fp32 arrays to a state format and
// back, with the same codecs the fused step uses ("When Small Updates
// Disappear", sec. 6-8: the stand-alone fp32 -> BF16 cast with nearest or
// stochastic rounding, one read and one write per element).
//
// The cast needs one 16-bit draw per element, so it spends every bit of a
// Philox call: the call for counter (g, tensor, step) serves the eight
// elements 8g .. 8g+7, element 8g+j taking word j/2, low half for even j and
// high half for odd j.  At one call per eight elements the generator stays
// under the memory time.
//
// Work unit: a group of eight elements (32 input bytes; 16, 8 or 4 output
// bytes), one per thread.  A ragged tail (n mod 8 elements) is finished by
// the thread after the last full group, out of line, with guarded scalar
// accesses; every register array is indexed by compile-time constants only.
#include "common.cuh"
#include "internal.h"

namespace psopt {
namespace {

constexpr int kCodecThreads = 256;
// Occupancy hint: six CTAs per SM, 1536 threads.  (Eight, which caps registers
// at 32, crashes the aarch64 build of ptxas 13.0 on these kernels.)
constexpr int kCodecBlocksPerSM = 6;

// Output bytes of one eight-element group, packed in the order memory
// holds them: BF16 in w.x..w.w, E4M3 in w.x..w.y, E2M2 in w.x.  Two
// elements per converter instruction; with stochastic rounding, draw word k
// (low half for element 2k, high half for 2k+1) is exactly the random-bits
// operand of pair k.
template <int DT>
__device__ __forceinline__ uint4 encode_group(const float (&x)[8], uint4 d, bool sr) {
  const uint32_t words[4] = {d.x, d.y, d.z, d.w};
  uint32_t pr[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float lo = x[2 * k], hi = x[2 * k + 1];
    if (DT == OPT_BF16) pr[k] = sr ? bf16x2_sr(lo, hi, words[k]) : bf16x2_rn(lo, hi);
    else if (DT == OPT_E4M3) pr[k] = sr ? e4m3x2_sr(lo, hi, words[k]) : e4m3x2_rn(lo, hi);
    else {
      const float lo4 = __fmul_rn(lo, 0.25f), hi4 = __fmul_rn(hi, 0.25f);   // exact
      pr[k] = sr ? e2m2x2_sr_q(lo4, hi4, words[k]) : e2m2x2_rn_q(lo4, hi4);
    }
  }
  uint4 w = make_uint4(0u, 0u, 0u, 0u);
  if (DT == OPT_BF16) {
    w = make_uint4(pr[0], pr[1], pr[2], pr[3]);
  } else if (DT == OPT_E4M3) {
    w.x = pr[0] | (pr[1] << 16);
    w.y = pr[2] | (pr[3] << 16);
  } else {
    // pair k holds the two codes in bytes 0 and 1; byte k of the output
    // holds them as nibbles (even element low)
#pragma unroll
    for (int k = 0; k < 4; ++k) w.x |= ((pr[k] | (pr[k] >> 4)) & 0xFFu) << (8 * k);
  }
  return w;
}

template <int DT>
__device__ __forceinline__ void store_group(void* out, int64_t g, uint4 w) {
  if (DT == OPT_BF16) st_cs_u4(static_cast<char*>(out) + 16 * g, w);
  else if (DT == OPT_E4M3) st_cs_u2(static_cast<char*>(out) + 8 * g, make_uint2(w.x, w.y));
  else st_cs_u1(static_cast<char*>(out) + 4 * g, w.x);
}

// The ragged tail (elements 8*full .. n-1, rem of them), by one thread; out
// of line so that its scalar accesses add nothing to the main path's
// registers.
template <int DT, bool SR>
__device__ __noinline__ void encode_tail(const float* __restrict__ in, void* __restrict__ out, int64_t full,
                                         int rem, uint32_t seed_lo, uint32_t seed_hi, uint32_t tensor,
                                         uint32_t step32) {
  const int64_t e0 = full * 8;
  float xt[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) xt[j] = j < rem ? in[e0 + j] : 0.0f;
  const uint4 d = SR ? draw_words((uint64_t)full, tensor, step32, seed_lo, seed_hi) : make_uint4(0u, 0u, 0u, 0u);
  const uint4 w = encode_group<DT>(xt, d, SR);
  const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
  // bytes that belong to the tail's elements (a half-filled E2M2 byte holds
  // 0, the code of the zero padding, in its high nibble)
  const int nbytes = DT == OPT_BF16 ? 2 * rem : (DT == OPT_E4M3 ? rem : (rem + 1) / 2);
  uint8_t* dst = static_cast<uint8_t*>(out) + (DT == OPT_BF16 ? 2 * e0 : (DT == OPT_E4M3 ? e0 : e0 / 2));
#pragma unroll
  for (int b = 0; b < 16; ++b)
    if (b < nbytes) dst[b] = (uint8_t)(ws[b >> 2] >> (8 * (b & 3)));
}

// Thread g0 + (global thread index) encodes group g; the thread at g == full
// finishes a ragged tail.
template <int DT, bool SR>
__global__ void __launch_bounds__(kCodecThreads, kCodecBlocksPerSM)
encode_kernel(const float* __restrict__ in, void* __restrict__ out, int64_t n, int64_t g0, uint32_t seed_lo,
              uint32_t seed_hi, uint32_t tensor, uint32_t step32) {
  const int64_t full = n >> 3;                       // complete groups
  const int64_t g = g0 + (int64_t)blockIdx.x * kCodecThreads + threadIdx.x;
  if (g < full) {
    const char* src = reinterpret_cast<const char*>(in) + 32 * g;
    const uint4 a0 = ld_nc_u4(src), a1 = ld_nc_u4(src + 16);
    const uint4 d = SR ? draw_words((uint64_t)g, tensor, step32, seed_lo, seed_hi) : make_uint4(0u, 0u, 0u, 0u);
    const float x[8] = {u2f(a0.x), u2f(a0.y), u2f(a0.z), u2f(a0.w),
                        u2f(a1.x), u2f(a1.y), u2f(a1.z), u2f(a1.w)};
    store_group<DT>(out, g, encode_group<DT>(x, d, SR));
  } else if (g == full && (n & 7) != 0) {
    encode_tail<DT, SR>(in, out, full, (int)(n & 7), seed_lo, seed_hi, tensor, step32);
  }
}

// Decode, eight elements per group: codes in, two 16-byte stores of fp32 out.
template <int DT>
__device__ __forceinline__ void decode_group(const void* in, int64_t g, float (&x)[8]) {
  if (DT == OPT_BF16) {
    const uint4 w = ld_nc_u4(static_cast<const char*>(in) + 16 * g);
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      x[2 * k] = u2f(ws[k] << 16);
      x[2 * k + 1] = u2f(ws[k] & 0xFFFF0000u);
    }
  } else if (DT == OPT_E4M3) {
    const uint2 w = ld_cs_u2(static_cast<const char*>(in) + 8 * g);
    const uint32_t ws[2] = {w.x, w.y};
#pragma unroll
    for (int k = 0; k < 4; ++k) e4m3x2_dec((ws[k >> 1] >> (16 * (k & 1))) & 0xFFFFu, x[2 * k], x[2 * k + 1]);
  } else {
    const uint32_t w = ld_cs_u1(static_cast<const char*>(in) + 4 * g);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint32_t byte = (w >> (8 * k)) & 0xFFu;
      e2m2x2_dec((byte & 0xFu) | ((byte >> 4) << 8), x[2 * k], x[2 * k + 1]);
    }
  }
}

template <int DT>
__device__ __noinline__ void decode_tail(const void* __restrict__ in, float* __restrict__ out, int64_t full,
                                         int rem) {
  const int64_t e0 = full * 8;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    if (j < rem) {
      float x;
      if (DT == OPT_BF16) x = bf16_dec(static_cast<const uint16_t*>(in)[e0 + j]);
      else if (DT == OPT_E4M3) x = e4m3_dec(static_cast<const uint8_t*>(in)[e0 + j]);
      else x = e2m2_dec((static_cast<const uint8_t*>(in)[(e0 + j) >> 1] >> (4 * (j & 1))) & 0xFu);
      out[e0 + j] = x;
    }
  }
}

template <int DT>
__global__ void __launch_bounds__(kCodecThreads, kCodecBlocksPerSM)
decode_kernel(const void* __restrict__ in, float* __restrict__ out, int64_t n, int64_t g0) {
  const int64_t full = n >> 3;
  const int64_t g = g0 + (int64_t)blockIdx.x * kCodecThreads + threadIdx.x;
  if (g < full) {
    float x[8];
    decode_group<DT>(in, g, x);
    st_cs_u4(out + 8 * g, make_uint4(f2u(x[0]), f2u(x[1]), f2u(x[2]), f2u(x[3])));
    st_cs_u4(out + 8 * g + 4, make_uint4(f2u(x[4]), f2u(x[5]), f2u(x[6]), f2u(x[7])));
  } else if (g == full && (n & 7) != 0) {
    decode_tail<DT>(in, out, full, (int)(n & 7));
  }
}

// Grid: one thread per group (plus one for a ragged tail), not a persistent
// grid -- for this pure stream, fresh CTAs that start with their loads kept
// HBM busier than resident CTAs looping grid-stride (about 10 % more
// bandwidth measured on GB300).  Launches of at most kMaxGrid CTAs, each
// from a group offset, cover any n.
constexpr int64_t kMaxGrid = (int64_t)1 << 30;

template <int DT, bool SR>
cudaError_t launch_enc(const float* in, void* out, int64_t n, uint32_t seed_lo, uint32_t seed_hi,
                       uint32_t tensor, uint32_t step32, cudaStream_t s) {
  const int64_t threads = (n >> 3) + ((n & 7) ? 1 : 0);
  for (int64_t g0 = 0; g0 < threads; g0 += kMaxGrid * kCodecThreads) {
    const int64_t left = (threads - g0 + kCodecThreads - 1) / kCodecThreads;
    const int grid = (int)(left < kMaxGrid ? left : kMaxGrid);
    encode_kernel<DT, SR><<<grid, kCodecThreads, 0, s>>>(in, out, n, g0, seed_lo, seed_hi, tensor, step32);
  }
  return cudaGetLastError();
}

template <int DT>
cudaError_t launch_dec(const void* in, float* out, int64_t n, cudaStream_t s) {
  const int64_t threads = (n >> 3) + ((n & 7) ? 1 : 0);
  for (int64_t g0 = 0; g0 < threads; g0 += kMaxGrid * kCodecThreads) {
    const int64_t left = (threads - g0 + kCodecThreads - 1) / kCodecThreads;
    const int grid = (int)(left < kMaxGrid ? left : kMaxGrid);
    decode_kernel<DT><<<grid, kCodecThreads, 0, s>>>(in, out, n, g0);
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_encode(const float* in, void* out, int64_t n, int dtype, int stochastic,
                          uint32_t seed_lo, uint32_t seed_hi, uint32_t tensor, uint32_t step32,
                          int sm_count, cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  (void)sm_count;
#define PS_ENC(DT, SRV) launch_enc<DT, SRV>(in, out, n, seed_lo, seed_hi, tensor, step32, s)
  if (dtype == OPT_BF16) return stochastic ? PS_ENC(OPT_BF16, true) : PS_ENC(OPT_BF16, false);
  if (dtype == OPT_E4M3) return stochastic ? PS_ENC(OPT_E4M3, true) : PS_ENC(OPT_E4M3, false);
  return stochastic ? PS_ENC(OPT_E2M2, true) : PS_ENC(OPT_E2M2, false);
#undef PS_ENC
}

cudaError_t launch_decode(const void* in, float* out, int64_t n, int dtype, int sm_count,
                          cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  (void)sm_count;
  if (dtype == OPT_BF16) return launch_dec<OPT_BF16>(in, out, n, s);
  if (dtype == OPT_E4M3) return launch_dec<OPT_E4M3>(in, out, n, s);
  return launch_dec<OPT_E2M2>(in, out, n, s);
}

}  // namespace psopt
