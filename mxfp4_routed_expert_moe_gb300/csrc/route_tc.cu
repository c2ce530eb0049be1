// route_tc.cu — router scores s = x Wr^T (+ b) of bf16 batches above 64
// tokens: an approximate product on tcgen05 tensor cores screens the experts,
// and the exact scores are computed only for the experts that can still be in
// a token's top k [Deltafin's custom compiled runtime, "Complete target
// sequence tape" (top-16 routing per position); the router is an fp32 linear
// map of the hidden state].
//
//   1. k_router_prep: Wr (fp32) as two bf16 terms, hi = bf16(W) and
//      mid = bf16(W - hi), so |W - hi - mid| <= 2^-16 |W|; the Euclidean norm
//      of each row, rounded up; clears the per-expert token masks.
//   2. k_router_tc: s~ = x (hi + mid)^T + b on tensor cores (kind::f16, bf16
//      operands), 128-token x 128-expert tiles fed by tensor-map copies; the
//      MMAs accumulate chunks of kChunk slices in Tensor Memory (alternating
//      two buffers), and the epilogue adds the chunks in fp32 registers.
//   3. k_router_exact, one CTA per token: a bound B(e) on |s~ - s|, the k-th
//      largest lower bound L = kth_e(s~ - B), and the candidates {e :
//      s~ + B >= L}, which include every expert of the true top k; their
//      scores are computed exactly as the CUDA-core GEMM does (fp32 products
//      summed in chunks of 16, chunk sums carried in double-float, the bias
//      added in double-float), and the kernel selects the top k among them,
//      writes their renormalised weights and sets the token's mask bits (the
//      other experts' scores are never needed).
//
// The bound.  With S = sum_h |x_h| |W_eh| <= ||x|| ||W_e|| (Cauchy-Schwarz):
//   * the split: |sum x (W - hi - mid)| <= 2^-16 S;
//   * the accumulation: each MMA adds 16 exact bf16 x bf16 products to the
//     accumulator; taking its error as at most 18 units of 2^-23 of the sum
//     of the magnitudes of its 17 addends (alignment and truncation of every
//     addend plus a final rounding, a worst-case model of the tensor core's
//     fp32 sum), a chunk of M MMAs errs by at most 18 2^-23 (M + 1) S_chunk,
//     so all chunks together by 18 2^-23 (M + 1) (1 + 2^-7) S, with
//     M = 8 min(kChunk, H / 64) (8 MMAs per 64-element slice); adding the C
//     chunks in fp32 registers errs by at most C 2^-24 (1 + 2^-7) S;
//   * the fp32 addition of the bias: at most 2^-24 (|s~| + |b|).
// B(e) adds these with the norms rounded up by 2^-9 and a further 2^-22 of
// (|s~| + B) for the rounding of s~ -+ B themselves.
#include <cuda.h>
#include <cuda_bf16.h>
#include <string.h>

#include "async.cuh"
#include "kernels.h"
#include "route_small.cuh"
#include "tcgen05.cuh"

namespace moe {

namespace rtc {
constexpr int kTile = 128;                  // tokens (M) and experts (N) per tile
constexpr int kSliceK = 64;                 // contraction elements per stage (128 bytes of bf16)
constexpr int kStages = 4;
constexpr int kTileBytes = kTile * 128;     // one 128-row x 64-element bf16 tile
constexpr int kStageBytes = 3 * kTileBytes; // x tile, W hi tile, W mid tile
constexpr int kThreads = 192;               // warp 0 MMA issuer (owns TMEM), warp 1 producer, warps 2-5 epilogue
constexpr uint32_t kTmemCols = 256;         // two accumulator buffers of 128 columns
constexpr int kExactThreads = 256;
constexpr int kMaxE = 4096;
constexpr int kChunk = 14;                  // slices per accumulation chunk (896 elements)
constexpr uint32_t kPollMma = 0, kPollTma = 32, kPollEp = 128;
}  // namespace rtc

// Coefficient of S in the bound (see the file comment).
__device__ __forceinline__ float rtc_alpha(int H) {
  const int ns = H / rtc::kSliceK;
  const int per_chunk = (ns < rtc::kChunk ? ns : rtc::kChunk) * 2 * (rtc::kSliceK / 16);  // MMAs
  const int chunks = (ns + rtc::kChunk - 1) / rtc::kChunk;
  return 0x1p-16f + (18.f * 0x1p-23f * (float)(per_chunk + 1) + 0x1p-24f * (float)chunks) * (1.f + 1.f / 128.f);
}

// ------------------------------------------------------------------ prep --
// One warp per expert row.
__global__ void __launch_bounds__(256) k_router_prep(RouteParams p) {
  const int e = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (e >= p.E) return;
  const int H = p.H;
  const float* w = p.wr + (size_t)e * H;
  uint16_t* hi = p.ws.wr16 + (size_t)e * H;
  uint16_t* mid = hi + (size_t)p.E * H;
  float ss = 0.f;
  for (int h = lane * 4; h < H; h += 128) {
    const float4 v = *reinterpret_cast<const float4*>(w + h);
    const float a[4] = {v.x, v.y, v.z, v.w};
    uint32_t oh[2], om[2];
#pragma unroll
    for (int j = 0; j < 4; j += 2) {
      const __nv_bfloat16 h0 = __float2bfloat16_rn(a[j]), h1 = __float2bfloat16_rn(a[j + 1]);
      const __nv_bfloat16 m0 = __float2bfloat16_rn(a[j] - __bfloat162float(h0));
      const __nv_bfloat16 m1 = __float2bfloat16_rn(a[j + 1] - __bfloat162float(h1));
      oh[j / 2] = (uint32_t)__bfloat16_as_ushort(h0) | ((uint32_t)__bfloat16_as_ushort(h1) << 16);
      om[j / 2] = (uint32_t)__bfloat16_as_ushort(m0) | ((uint32_t)__bfloat16_as_ushort(m1) << 16);
      ss = fmaf(a[j], a[j], ss);
      ss = fmaf(a[j + 1], a[j + 1], ss);
    }
    *reinterpret_cast<uint2*>(hi + h) = make_uint2(oh[0], oh[1]);
    *reinterpret_cast<uint2*>(mid + h) = make_uint2(om[0], om[1]);
  }
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) ss += __shfl_xor_sync(0xFFFFFFFFu, ss, o);
  // The fp32 sum of H squares is within H 2^-24 of exact, so its square root
  // within half that: 2^-9 covers every H <= 16384.
  if (lane == 0) p.ws.wrnorm[e] = sqrtf(ss) * (1.f + 1.f / 512.f);
  const int W = (p.T + 31) / 32;
  for (int i = lane; i < W; i += 32) p.ws.mask[(size_t)e * W + i] = 0u;
}

// ------------------------------------------------------------- screen GEMM --
struct RtcShared {
  uint64_t full[rtc::kStages];   // stage filled: producer, with the copies' bytes
  uint64_t empty[rtc::kStages];  // stage consumed: tcgen05.commit
  uint64_t accf[2];              // accumulator buffer ready: tcgen05.commit
  uint64_t acce[2];              // accumulator buffer drained: 4 epilogue warps
  uint32_t tmem_base;
  int abort_flag;
};

__device__ __forceinline__ bool rtc_wait(RtcShared& sh, uint64_t* bar, uint32_t parity, WsHeader* hdr,
                                         uint32_t backoff_ns, long long limit) {
  const bool diag = limit < kWaitCycles;
  if (diag ? mbar_test_wait(bar, parity) : mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  for (;;) {
    if (backoff_ns) __nanosleep(backoff_ns);
    if (diag ? mbar_test_wait(bar, parity) : mbar_try_wait(bar, parity)) return true;
    if (*(volatile int*)&sh.abort_flag) return false;
    if (clock64() - t0 > limit) {
      set_status(hdr, MOE_ERR_TIMEOUT);
      *(volatile int*)&sh.abort_flag = 1;
      return false;
    }
  }
}

// Persistent, one CTA per SM; items are (128-token tile, 128-expert tile),
// expert tiles inner.  Per 64-element slice the producer loads the token tile
// (x, bf16) and both W terms with two tensor-map copies; the MMA thread issues
// 4 K-steps x 2 terms (M = N = 128, K = 16) into the item's accumulator
// buffer; the epilogue warps add the bias and store s~ in fp32.
__global__ void __launch_bounds__(rtc::kThreads, 1)
    k_router_tc(RouteParams p, const __grid_constant__ CUtensorMap xmap, const __grid_constant__ CUtensorMap wmap) {
  extern __shared__ uint8_t rtc_dyn[];
  __shared__ RtcShared sh;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (warp == 0) {
    tmem_alloc(&sh.tmem_base, rtc::kTmemCols);
    tmem_relinquish();
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < rtc::kStages; ++s) {
      mbar_init(&sh.full[s], 1);
      mbar_init(&sh.empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sh.accf[b], 1);
      mbar_init(&sh.acce[b], 4);
    }
    sh.abort_flag = 0;
    mbar_init_fence();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sh.tmem_base;
  uint8_t* ring = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(rtc_dyn) + 1023) & ~(uintptr_t)1023);
  const int etiles = (p.E + rtc::kTile - 1) / rtc::kTile;
  const int n_items = ((p.T + rtc::kTile - 1) / rtc::kTile) * etiles;
  const int ns = p.H / rtc::kSliceK;
  WsHeader* hdr = p.ws.hdr;
  const long long lim = p.wait_limit;
  if (warp == 1) {
    // Producer.
    int issued[rtc::kStages];
#pragma unroll
    for (int i = 0; i < rtc::kStages; ++i) issued[i] = -1;
    int gs = 0;
    bool ok = true;
    for (int item = blockIdx.x; item < n_items && ok; item += gridDim.x) {
      const int t0 = (item / etiles) * rtc::kTile, e0 = (item % etiles) * rtc::kTile;
      for (int s = 0; s < ns; ++s, ++gs) {
        const int st = gs % rtc::kStages, use = gs / rtc::kStages;
        bool got = true;
        if (lane == 0 && use > 0) got = rtc_wait(sh, &sh.empty[st], (use - 1) & 1, hdr, rtc::kPollTma, lim);
        if (!__shfl_sync(0xFFFFFFFFu, got, 0)) {
          ok = false;
          break;
        }
        if (lane == 0) {
          uint8_t* sb = ring + (size_t)st * rtc::kStageBytes;
          mbar_arrive_expect_tx(&sh.full[st], (uint32_t)rtc::kStageBytes);
          tma_load_2d(sb, &xmap, s * rtc::kSliceK, t0, &sh.full[st]);
          tma_load_3d(sb + rtc::kTileBytes, &wmap, s * rtc::kSliceK, e0, 0, &sh.full[st]);
#pragma unroll
          for (int i = 0; i < rtc::kStages; ++i)
            if (i == st) issued[i] = use;
        }
        __syncwarp();
      }
    }
    if (lane == 0)
#pragma unroll
      for (int i = 0; i < rtc::kStages; ++i)
        if (issued[i] >= 0 && !mbar_wait(&sh.full[i], issued[i] & 1)) set_status(hdr, MOE_ERR_TIMEOUT);
  } else if (warp == 0) {
    if (lane == 0) {
      // MMA issuer: chunk cc (global over the CTA's items) goes to buffer
      // cc & 1, which the epilogue has drained since its use two chunks ago.
      const uint32_t idesc = idesc_bf16_f32(rtc::kTile, rtc::kTile);
      int cc = 0, gs = 0;
      bool ok = true;
      for (int item = blockIdx.x; item < n_items && ok; item += gridDim.x) {
        int b = 0;
        for (int s = 0; s < ns; ++s, ++gs) {
          if (s % rtc::kChunk == 0) {
            b = cc & 1;
            const int use = cc >> 1;
            if (use >= 1 && !rtc_wait(sh, &sh.acce[b], (use - 1) & 1, hdr, rtc::kPollMma, lim)) {
              ok = false;
              break;
            }
            tc_fence_after();
          }
          const int st = gs % rtc::kStages;
          if (!rtc_wait(sh, &sh.full[st], (gs / rtc::kStages) & 1, hdr, rtc::kPollMma, lim)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sbase = smem_u32(ring + (size_t)st * rtc::kStageBytes);
#pragma unroll
          for (int kb = 0; kb < rtc::kSliceK / 16; ++kb) {
            const uint64_t ad = sdesc_sw128(sbase + 32 * kb);
#pragma unroll
            for (int term = 0; term < 2; ++term)
              umma_f16(tmem + (uint32_t)(b * rtc::kTile), ad,
                       sdesc_sw128(sbase + (uint32_t)((1 + term) * rtc::kTileBytes) + 32 * kb), idesc,
                       (s % rtc::kChunk > 0 || kb > 0 || term > 0) ? 1u : 0u);
          }
          umma_commit(&sh.empty[st]);
          if (s % rtc::kChunk == rtc::kChunk - 1 || s == ns - 1) {
            umma_commit(&sh.accf[b]);
            ++cc;
          }
        }
        if (!ok && ns > 0 && gs % rtc::kChunk != 0) {
          // A chunk broken off: commit it so that the drain below waits for it.
          umma_commit(&sh.accf[b]);
          ++cc;
        }
      }
      if (cc > 0 && !mbar_wait(&sh.accf[(cc - 1) & 1], ((cc - 1) >> 1) & 1)) set_status(hdr, MOE_ERR_TIMEOUT);
    }
  } else {
    // Epilogue warps 2-5: TMEM lane quarter q = warp % 4, token t0 + 32 q +
    // lane; the item's chunks are added in fp32 registers in chunk order.
    const int q = warp & 3;
    const int nchunks = (ns + rtc::kChunk - 1) / rtc::kChunk;
    int cc = 0;
    bool ok = true;
    for (int item = blockIdx.x; item < n_items && ok; item += gridDim.x) {
      const int t0 = (item / etiles) * rtc::kTile, e0 = (item % etiles) * rtc::kTile;
      float acc[rtc::kTile];
#pragma unroll
      for (int j = 0; j < rtc::kTile; ++j) acc[j] = 0.f;
      for (int ch = 0; ch < nchunks; ++ch, ++cc) {
        const int b = cc & 1;
        bool got = rtc_wait(sh, &sh.accf[b], (cc >> 1) & 1, hdr, rtc::kPollEp, lim);
        if (!__all_sync(0xFFFFFFFFu, got)) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int c0 = 0; c0 < rtc::kTile; c0 += 32) {
          uint32_t v[32];
          tmem_ld32(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(b * rtc::kTile + c0), v);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 32; ++j) acc[c0 + j] += __uint_as_float(v[j]);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sh.acce[b]);
      }
      if (!ok) break;
      const int t = t0 + q * 32 + lane;
      if (t < p.T) {
        float* dst = p.ws.sapprox + (size_t)t * p.E;
#pragma unroll
        for (int j = 0; j < rtc::kTile; ++j) {
          const int e = e0 + j;
          if (e < p.E) dst[e] = acc[j] + (p.br ? __ldg(&p.br[e]) : 0.f);
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, rtc::kTmemCols);
  }
}

// ------------------------------------------------------ screen + exact scores --
// One CTA per token.  Shared memory: x (fp32) [H], lower bounds [E] (float2,
// for warp_topk), candidate list [E].
__device__ __forceinline__ float rtc_bound(float sa, float b, float xw, float alpha) {
  const float B = alpha * xw + 0x1p-24f * (fabsf(sa) + fabsf(b));
  return B + 0x1p-22f * (fabsf(sa) + B) + 0x1p-126f;
}

__global__ void __launch_bounds__(rtc::kExactThreads) k_router_exact(RouteParams p) {
  extern __shared__ float4 rx_dyn[];
  const int H = p.H, E = p.E, k = p.k;
  float* xs = reinterpret_cast<float*>(rx_dyn);
  float2* row = reinterpret_cast<float2*>(xs + H);
  int* cand = reinterpret_cast<int*>(row + E);
  __shared__ float red[rtc::kExactThreads / 32];
  __shared__ float xnorm, kth;
  __shared__ int ncand;
  const int t = blockIdx.x, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint16_t* xb = reinterpret_cast<const uint16_t*>(p.x) + (size_t)t * H;
  float ss = 0.f;
  for (int h = tid * 4; h < H; h += rtc::kExactThreads * 4) {
    const uint2 v = *reinterpret_cast<const uint2*>(xb + h);
    const float a0 = __uint_as_float(v.x << 16), a1 = __uint_as_float(v.x & 0xFFFF0000u);
    const float a2 = __uint_as_float(v.y << 16), a3 = __uint_as_float(v.y & 0xFFFF0000u);
    *reinterpret_cast<float4*>(xs + h) = make_float4(a0, a1, a2, a3);
    ss = fmaf(a0, a0, ss);
    ss = fmaf(a1, a1, ss);
    ss = fmaf(a2, a2, ss);
    ss = fmaf(a3, a3, ss);
  }
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) ss += __shfl_xor_sync(0xFFFFFFFFu, ss, o);
  if (lane == 0) red[warp] = ss;
  if (tid == 0) ncand = 0;
  __syncthreads();
  if (tid == 0) {
    float tot = 0.f;
    for (int w = 0; w < rtc::kExactThreads / 32; ++w) tot += red[w];
    xnorm = sqrtf(tot) * (1.f + 1.f / 512.f);
  }
  __syncthreads();
  const float alpha = rtc_alpha(H);
  const float xn = xnorm;
  const float* sa_row = p.ws.sapprox + (size_t)t * E;
  for (int e = tid; e < E; e += rtc::kExactThreads) {
    const float sa = sa_row[e];
    const float bias = p.br ? __ldg(&p.br[e]) : 0.f;
    const float B = rtc_bound(sa, bias, xn * __ldg(&p.ws.wrnorm[e]), alpha);
    row[e] = make_float2(sa - B, 0.f);
  }
  __syncthreads();
  if (warp == 0) {
    int my_e;
    float2 my_s;
    warp_topk(row, E, k, my_e, my_s);
    if (lane == k - 1) kth = my_s.x;
  }
  __syncthreads();
  const float L = kth;
  for (int e = tid; e < E; e += rtc::kExactThreads) {
    const float sa = sa_row[e];
    const float bias = p.br ? __ldg(&p.br[e]) : 0.f;
    const float B = rtc_bound(sa, bias, xn * __ldg(&p.ws.wrnorm[e]), alpha);
    if (sa + B >= L) cand[atomicAdd(&ncand, 1)] = e;
  }
  __syncthreads();
  if (ncand < k) {
    // Only non-finite scores leave fewer than k candidates: every expert is one.
    __syncthreads();
    if (tid == 0) ncand = 0;
    __syncthreads();
    for (int e = tid; e < E; e += rtc::kExactThreads) cand[atomicAdd(&ncand, 1)] = e;
    __syncthreads();
  }
  const int nc = ncand;
  float2* csc = row;  // the candidates' exact scores, in candidate order (the bounds are done)
  for (int c = warp; c < nc; c += rtc::kExactThreads / 32) {
    const int e = cand[c];
    const float* w = p.wr + (size_t)e * H;
    float hi = 0.f, lo = 0.f;
    // Chunks of 16 products per lane (four float4 steps of the warp), summed
    // in fp32, then carried in double-float.
    for (int base = 0; base < H; base += 512) {
      float acc = 0.f;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int h = base + 128 * j + lane * 4;
        if (h < H) {
          const float4 wv = __ldg(reinterpret_cast<const float4*>(w + h));
          const float4 xv = *reinterpret_cast<const float4*>(xs + h);
          acc = fmaf(xv.x, wv.x, acc);
          acc = fmaf(xv.y, wv.y, acc);
          acc = fmaf(xv.z, wv.z, acc);
          acc = fmaf(xv.w, wv.w, acc);
        }
      }
      df_add_f(hi, lo, acc);
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
      const float rh = __shfl_xor_sync(0xFFFFFFFFu, hi, o);
      const float rl = __shfl_xor_sync(0xFFFFFFFFu, lo, o);
      df_add(hi, lo, rh, rl, hi, lo);
    }
    if (lane == 0) {
      float sh, sl;
      df_add(hi, lo, p.br ? __ldg(&p.br[e]) : 0.f, 0.f, sh, sl);
      csc[c] = make_float2(sh, sl);
    }
  }
  __syncthreads();
  // The top k among the candidates (they include the true top k), their
  // renormalised weights, and the token's bit in each selected expert's mask.
  if (warp == 0) {
    int my_e;
    float2 my_s;
    warp_topk_list(csc, cand, nc, k, my_e, my_s);
    const float wt = warp_route_weight(my_s, k);
    if (lane < k) {
      p.ids[(size_t)t * k + lane] = my_e;
      p.w[(size_t)t * k + lane] = wt;
      const int W = (p.T + 31) / 32;
      atomicOr(&p.ws.mask[(size_t)my_e * W + (t >> 5)], 1u << (t & 31));
    }
  }
}

// ---------------------------------------------------------------- launcher --
namespace {
// Tensor map of a bf16 matrix [rows][K] (row stride K * 2 bytes): boxes of 64
// elements x 128 rows, 128-byte swizzle, rows past the end read as zero.
cudaError_t encode_bf16_rows(CUtensorMap* m, const void* base, int K, int rows) {
  const EncodeTiledFn enc = encode_tiled_fn();
  if (!enc) return cudaErrorNotSupported;
  const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)K * 2};
  const cuuint32_t box[2] = {(cuuint32_t)rtc::kSliceK, (cuuint32_t)rtc::kTile};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}
// The two W terms as a [2][E][H] bf16 tensor: boxes of 64 elements x 128 rows
// x both terms (hi tile, then mid tile in shared memory).
cudaError_t encode_w_terms(CUtensorMap* m, const void* base, int H, int E) {
  const EncodeTiledFn enc = encode_tiled_fn();
  if (!enc) return cudaErrorNotSupported;
  const cuuint64_t dims[3] = {(cuuint64_t)H, (cuuint64_t)E, 2};
  const cuuint64_t strides[2] = {(cuuint64_t)H * 2, (cuuint64_t)E * H * 2};
  const cuuint32_t box[3] = {(cuuint32_t)rtc::kSliceK, (cuuint32_t)rtc::kTile, 2};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}
}  // namespace

cudaError_t launch_router_tc(const RouteParams& p, cudaStream_t s) {
  if (!p.x_bf16 || p.T <= kDecodeMaxT || p.H % rtc::kSliceK != 0 || p.E > rtc::kMaxE || !p.ws.wr16 ||
      ((uintptr_t)p.x & 15u) != 0)
    return cudaErrorNotSupported;
  CUtensorMap xmap, wmap;
  memset(&xmap, 0, sizeof xmap);
  memset(&wmap, 0, sizeof wmap);
  cudaError_t err;
  if ((err = encode_bf16_rows(&xmap, p.x, p.H, p.T)) != cudaSuccess) return err;
  if ((err = encode_w_terms(&wmap, p.ws.wr16, p.H, p.E)) != cudaSuccess) return err;
  k_router_prep<<<(p.E + 7) / 8, 256, 0, s>>>(p);
  if ((err = cudaGetLastError()) != cudaSuccess) return err;
  constexpr size_t gemm_smem = (size_t)rtc::kStages * rtc::kStageBytes + 1024;
  if ((err = ensure_smem_attr((const void*)k_router_tc, gemm_smem)) != cudaSuccess) return err;
  const int items = ((p.T + rtc::kTile - 1) / rtc::kTile) * ((p.E + rtc::kTile - 1) / rtc::kTile);
  const int nsm = device_sm_count();
  k_router_tc<<<items < nsm ? items : nsm, rtc::kThreads, gemm_smem, s>>>(p, xmap, wmap);
  if ((err = cudaGetLastError()) != cudaSuccess) return err;
  const size_t exact_smem = (size_t)p.H * 4 + (size_t)p.E * 12;
  if ((err = ensure_smem_attr((const void*)k_router_exact, exact_smem)) != cudaSuccess) return err;
  k_router_exact<<<p.T, rtc::kExactThreads, exact_smem, s>>>(p);
  return cudaGetLastError();
}

}  // namespace moe
