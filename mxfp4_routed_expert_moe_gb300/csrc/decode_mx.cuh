// decode_mx.cuh — shape rules and the preparation step of the persistent
// block-scaled decode kernel (decode_mx.cu), shared with the router kernel,
// which runs the preparation while it computes the scores.
#pragma once

#include "common.cuh"

namespace moe {

struct DmxDims {
  int ns_gu;  // gate/up slices (H / 128)
  int spp;    // slices per chunk of gate/up scale words
  int rt;     // gate/up row tiles = down slices (I / 128)
  int rh;     // down row tiles (H / 128)
  int umax;   // active experts at most: min(E, T k)
};
__host__ __device__ inline DmxDims dmx_dims(int T, int H, int E, int I, int k) {
  DmxDims d;
  d.ns_gu = H / 128;
  d.spp = dmx_spp(d.ns_gu);
  d.rt = I / 128;
  d.rh = H / 128;
  d.umax = E < T * k ? E : T * k;
  return d;
}
// Counter words: the tensor maps built and the CTAs done (the first
// kDmxCntHead words), then the h-tile readiness [umax][rt].
__host__ __device__ inline size_t dmx_counter_words(const DmxDims& d, int) {
  return kDmxCntHead + (size_t)d.umax * d.rt;
}

// One E4M3 code of v (round to nearest even, saturating) and its value.
__device__ __forceinline__ uint32_t dmx_e4m3(float v) {
  unsigned short q;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(q) : "f"(0.f), "f"(v));
  return q & 0xFFu;
}
__device__ __forceinline__ float dmx_e4m3_value(uint32_t q) {
  uint32_t f2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(f2) : "h"((unsigned short)q));
  return __half2float(__ushort_as_half((unsigned short)(f2 & 0xFFFFu)));
}

// Token t (bf16, H values) as two E4M3 terms x1 + x2 / 16 of x 2^tau, tau =
// 7 - floor(log2 max|x|) (the largest magnitude in [128, 256)): x1 =
// e4m3(x 2^tau), x2 = e4m3(16 (x 2^tau - x1)), exact for every element that
// stays an E4M3 normal number (within 2^-13 of the maximum); rows 2t and
// 2t + 1 of xq (H bytes each); x8scale[t] = 2^-tau.  All threads of the CTA
// call it.
__device__ __forceinline__ void dmx_x_terms(const uint16_t* xrow, int H, uint8_t* x1, uint8_t* x2, float* scale) {
  __shared__ float smax[32];
  float m = 0.f;
  for (int h = threadIdx.x * 8; h < H; h += blockDim.x * 8) {
    const uint4 v = *reinterpret_cast<const uint4*>(xrow + h);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j)
      m = fmaxf(m, fmaxf(fabsf(__uint_as_float(w[j] << 16)), fabsf(__uint_as_float(w[j] & 0xFFFF0000u))));
  }
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
  if ((threadIdx.x & 31) == 0) smax[threadIdx.x >> 5] = m;
  __syncthreads();
  m = 0.f;
  for (int w = 0; w < (int)(blockDim.x >> 5); ++w) m = fmaxf(m, smax[w]);
  int tau = 0;
  if (m > 0.f && m < INFINITY) tau = 7 - ((int)((__float_as_uint(m) >> 23) & 0xFF) - 127);
  tau = tau > 126 ? 126 : (tau < -126 ? -126 : tau);
  const float up = __int_as_float((tau + 127) << 23);
  if (threadIdx.x == 0) *scale = __int_as_float((127 - tau) << 23);
  for (int h = threadIdx.x * 4; h < H; h += blockDim.x * 4) {
    const uint2 v = *reinterpret_cast<const uint2*>(xrow + h);
    const float a[4] = {__uint_as_float(v.x << 16), __uint_as_float(v.x & 0xFFFF0000u), __uint_as_float(v.y << 16),
                        __uint_as_float(v.y & 0xFFFF0000u)};
    uint32_t o1 = 0u, o2 = 0u;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float s = a[j] * up;
      const uint32_t q1 = dmx_e4m3(s);
      const uint32_t q2 = dmx_e4m3((s - dmx_e4m3_value(q1)) * 16.f);
      o1 |= q1 << (8 * j);
      o2 |= q2 << (8 * j);
    }
    *reinterpret_cast<uint32_t*>(x1 + h) = o1;
    *reinterpret_cast<uint32_t*>(x2 + h) = o2;
  }
  __syncthreads();  // smax is reused by the next call
}

// The preparation of a step: the tokens' E4M3 terms and scales, and the
// kernel's counters cleared.  CTA b of n takes tokens b, b + n, .. and a
// share of the counters.  x is bf16.
__device__ __forceinline__ void dmx_prepare(const void* x, int T, int H, int E, int I, int k, const Ws& ws, int b,
                                            int n) {
  const DmxDims d = dmx_dims(T, H, E, I, k);
  const size_t nw = dmx_counter_words(d, T);
  for (size_t i = (size_t)b * blockDim.x + threadIdx.x; i < nw; i += (size_t)n * blockDim.x) ws.dmx_cnt[i] = 0u;
  for (int t = b; t < T; t += n)
    dmx_x_terms(reinterpret_cast<const uint16_t*>(x) + (size_t)t * H, H, ws.dmx_xq + (size_t)(2 * t) * H,
                ws.dmx_xq + (size_t)(2 * t + 1) * H, &ws.x8scale[t]);
}

}  // namespace moe
