// codec.cu -- standalone conversion of fp32 arrays to a state format and
// back, with the same codecs and draws the fused step uses ("When Small
// Updates Disappear", sec. 6-8: the stand-alone fp32 -> BF16 cast with
// nearest or stochastic rounding, one read and one write per element).
// Element i takes the v draw of element i of the given tensor and step.
#include "common.cuh"
#include "internal.h"

namespace psopt {
namespace {

constexpr int kCodecThreads = 256;

// stochastic encoders (nearest goes through the paired hardware converters)
template <int DT>
__device__ __forceinline__ uint32_t enc_sr(float x, uint32_t r16) {
  if (DT == OPT_BF16) return bf16_enc_sr(x, r16);
  if (DT == OPT_E2M2) return e2m2_enc_sr(x, r16);
  return e4m3_enc_sr(x, r16);
}

template <int DT, bool SR>
__global__ void __launch_bounds__(kCodecThreads)
encode_kernel(const float* __restrict__ in, void* __restrict__ out, int64_t n, uint32_t seed_lo,
              uint32_t seed_hi, uint32_t tensor, uint32_t step32) {
  const int64_t groups = (n + 7) / 8;
  for (int64_t gi = blockIdx.x * (int64_t)kCodecThreads + threadIdx.x; gi < groups;
       gi += (int64_t)gridDim.x * kCodecThreads) {
    const int64_t e0 = gi * 8;
    const int cnt = (int)min((int64_t)8, n - e0);
    float x[8];
    if (cnt == 8) {
      const uint4 a = ld_nc_u4(in + e0), b = ld_nc_u4(in + e0 + 4);
      x[0] = u2f(a.x); x[1] = u2f(a.y); x[2] = u2f(a.z); x[3] = u2f(a.w);
      x[4] = u2f(b.x); x[5] = u2f(b.y); x[6] = u2f(b.z); x[7] = u2f(b.w);
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j) x[j] = j < cnt ? in[e0 + j] : 0.0f;
    }
    uint32_t r[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    if (SR) {
      const uint4 d0 = draw_words((uint64_t)e0 >> 2, tensor, step32, seed_lo, seed_hi);
      const uint4 d1 = draw_words(((uint64_t)e0 >> 2) + 1, tensor, step32, seed_lo, seed_hi);
      r[0] = d0.x >> 16; r[1] = d0.y >> 16; r[2] = d0.z >> 16; r[3] = d0.w >> 16;
      r[4] = d1.x >> 16; r[5] = d1.y >> 16; r[6] = d1.z >> 16; r[7] = d1.w >> 16;
    }
    uint32_t c[8];
    if (SR) {
#pragma unroll
      for (int j = 0; j < 8; ++j) c[j] = enc_sr<DT>(x[j], r[j]);
    } else if (DT == OPT_BF16) {
#pragma unroll
      for (int j = 0; j < 8; ++j) c[j] = bf16_enc_rn(x[j]);
    } else {
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint32_t pair = DT == OPT_E4M3 ? e4m3x2_rn(x[2 * k], x[2 * k + 1])
                                             : e2m2x2_rn(x[2 * k], x[2 * k + 1]);
        c[2 * k] = pair & 0xFFu;
        c[2 * k + 1] = pair >> 8;
      }
    }
    if (cnt == 8) {
      if (DT == OPT_BF16)
        st_cs_u4(static_cast<uint16_t*>(out) + e0,
                 make_uint4(c[0] | (c[1] << 16), c[2] | (c[3] << 16), c[4] | (c[5] << 16),
                            c[6] | (c[7] << 16)));
      else if (DT == OPT_E4M3)
        st_cs_u2(static_cast<uint8_t*>(out) + e0,
                 make_uint2(c[0] | (c[1] << 8) | (c[2] << 16) | (c[3] << 24),
                            c[4] | (c[5] << 8) | (c[6] << 16) | (c[7] << 24)));
      else {
        uint32_t w = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) w |= c[j] << (4 * j);
        st_cs_u1(static_cast<uint8_t*>(out) + (e0 >> 1), w);
      }
    } else {
      for (int j = 0; j < cnt; ++j) {
        if (DT == OPT_BF16) static_cast<uint16_t*>(out)[e0 + j] = (uint16_t)c[j];
        else if (DT == OPT_E4M3) static_cast<uint8_t*>(out)[e0 + j] = (uint8_t)c[j];
      }
      if (DT == OPT_E2M2)
        for (int k = 0; 2 * k < cnt; ++k)
          static_cast<uint8_t*>(out)[(e0 >> 1) + k] =
              (uint8_t)(c[2 * k] | ((2 * k + 1 < cnt ? c[2 * k + 1] : 0u) << 4));
    }
  }
}

template <int DT>
__global__ void __launch_bounds__(kCodecThreads)
decode_kernel(const void* __restrict__ in, float* __restrict__ out, int64_t n) {
  for (int64_t i = blockIdx.x * (int64_t)kCodecThreads + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * kCodecThreads) {
    float x;
    if (DT == OPT_BF16) x = bf16_dec(static_cast<const uint16_t*>(in)[i]);
    else if (DT == OPT_E4M3) x = e4m3_dec(static_cast<const uint8_t*>(in)[i]);
    else x = e2m2_dec((static_cast<const uint8_t*>(in)[i >> 1] >> (4 * (i & 1))) & 0xFu);
    out[i] = x;
  }
}

int grid_for(int64_t items, int sm_count) {
  const int64_t want = (items + kCodecThreads - 1) / kCodecThreads;
  const int64_t cap = (int64_t)sm_count * 8;
  return (int)(want < 1 ? 1 : (want < cap ? want : cap));
}

}  // namespace

cudaError_t launch_encode(const float* in, void* out, int64_t n, int dtype, int stochastic,
                          uint32_t seed_lo, uint32_t seed_hi, uint32_t tensor, uint32_t step32,
                          int sm_count, cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  const int grid = grid_for((n + 7) / 8, sm_count);
#define PS_ENC(DT, SRV) encode_kernel<DT, SRV><<<grid, kCodecThreads, 0, s>>>(in, out, n, seed_lo, seed_hi, tensor, step32)
  if (dtype == OPT_BF16) { if (stochastic) PS_ENC(OPT_BF16, true); else PS_ENC(OPT_BF16, false); }
  else if (dtype == OPT_E4M3) { if (stochastic) PS_ENC(OPT_E4M3, true); else PS_ENC(OPT_E4M3, false); }
  else { if (stochastic) PS_ENC(OPT_E2M2, true); else PS_ENC(OPT_E2M2, false); }
#undef PS_ENC
  return cudaGetLastError();
}

cudaError_t launch_decode(const void* in, float* out, int64_t n, int dtype, int sm_count,
                          cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  const int grid = grid_for(n, sm_count);
  if (dtype == OPT_BF16) decode_kernel<OPT_BF16><<<grid, kCodecThreads, 0, s>>>(in, out, n);
  else if (dtype == OPT_E4M3) decode_kernel<OPT_E4M3><<<grid, kCodecThreads, 0, s>>>(in, out, n);
  else decode_kernel<OPT_E2M2><<<grid, kCodecThreads, 0, s>>>(in, out, n);
  return cudaGetLastError();
}

}  // namespace psopt
