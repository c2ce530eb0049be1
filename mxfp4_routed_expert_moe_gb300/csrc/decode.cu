// decode.cu — weight-streaming MXFP4 expert GEMV for small batches (T <= 64).
//
// The fused MXFP4 dequant+GEMV of [deltafin, "The techniques that bought the
// 82x"] (16-entry table lookup, E8M0 scale as a power of two on the fp32
// exponent) is re-designed for the GPU:
//   * each thread owns one 32-element block column of the weight matrix and
//     keeps the matching activations of up to NT tokens in registers, so the
//     weights stream from HBM exactly once per routed expert (tokens sharing
//     an expert reuse the same load);
//   * one 128-bit load is one MX block (32 nibbles); two E2M1 codes convert to
//     an exact f16x2 with one cvt, then to fp32 for the FMAs; the block's
//     partial sum is scaled once by 2^(e-127), which is exact;
//   * partial sums are reduced across the warp by a transpose-reduce and
//     across warps in a fixed order, so each token's result does not depend
//     on the batch;
//   * the k expert outputs of a token are combined in slot order ([Deltafin's
//     custom compiled runtime, "The native build"]: ordered reduction).
#include <utility>

#include "kernels.h"

namespace moe {

// Dot product of one MX block (16 bytes q, scale s) with NT activation blocks
// of 32 fp32 values each, accumulated into acc[nt] (scaled by 2^(s-127)).
template <int NT>
__device__ __forceinline__ void mx_block_dot(const uint4 q, uint32_t s, const float (&xr)[NT][32], float (&acc)[NT]) {
  float pe[NT], po[NT];
#pragma unroll
  for (int n = 0; n < NT; ++n) { pe[n] = 0.f; po[n] = 0.f; }
  const uint32_t words[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
  for (int wd = 0; wd < 4; ++wd) {
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const float2 f = f16x2_f32x2(e2m1x2_f16x2(words[wd], b));
      const int c = wd * 8 + b * 2;
#pragma unroll
      for (int n = 0; n < NT; ++n) {
        pe[n] = fmaf(f.x, xr[n][c], pe[n]);
        po[n] = fmaf(f.y, xr[n][c + 1], po[n]);
      }
    }
  }
  const float sc = e8m0_f32(s);
#pragma unroll
  for (int n = 0; n < NT; ++n) acc[n] = fmaf(pe[n] + po[n], sc, acc[n]);
}

template <bool XBF16>
__device__ __forceinline__ void load_act_block(const void* x, int64_t base, float (&dst)[32]) {
  if (XBF16) {
    const uint4* src = reinterpret_cast<const uint4*>(reinterpret_cast<const uint16_t*>(x) + base);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint4 v = src[i];
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        dst[i * 8 + j * 2] = __uint_as_float(w[j] << 16);
        dst[i * 8 + j * 2 + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
      }
    }
  } else {
    const float4* src = reinterpret_cast<const float4*>(reinterpret_cast<const float*>(x) + base);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float4 v = src[i];
      dst[i * 4] = v.x; dst[i * 4 + 1] = v.y; dst[i * 4 + 2] = v.z; dst[i * 4 + 3] = v.w;
    }
  }
}

// --------------------------------------------------------------- gate / up --
// Work item = (active expert u, tile of R = 8/NT rows of gate and of up).
// Thread tau < H/32 owns block column tau.  For each group of NT routed pairs
// of the expert: h[p][r] = silu(g) * u with g = Wg[r] . x_t, u = Wu[r] . x_t.
constexpr int kGuVals = 16;  // values reduced per warp: 2 matrices x R rows x NT

template <int NT, bool XBF16>
__global__ void __launch_bounds__(256) k_dec_gateup(ExpertParams p) {
  constexpr int R = 8 / NT;
  __shared__ float red[16][kGuVals];
  __shared__ int s_item;
  const int H = p.H, I = p.I, k = p.k;
  const int nbH = H / 32;
  const int tau = threadIdx.x;
  const bool col = tau < nbH;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nwarps = blockDim.x >> 5;
  pdl_wait();
  pdl_trigger();
  const int U = (int)p.ws.hdr->n_active;
  const int tiles = (I + R - 1) / R;
  const int n_items = U * tiles;
  float* hout = reinterpret_cast<float*>(p.ws.h);
  for (;;) {
    if (threadIdx.x == 0) s_item = (int)atomicAdd(&p.ws.hdr->queue[kQGateUp], 1u);
    __syncthreads();
    const int item = s_item;
    __syncthreads();
    if (item >= n_items) break;
    const int u = item / tiles, rt = item % tiles;
    const int e = p.ws.act_e[u];
    const int b0 = p.offsets[e], n = p.offsets[e + 1] - b0;
    const moe_expert ex = p.experts[e];
    const int r0 = rt * R;
    for (int pass = 0; pass < n; pass += NT) {
      int pe[NT];
      float xr[NT][32];
#pragma unroll
      for (int i = 0; i < NT; ++i) {
        pe[i] = pass + i < n ? p.sorted[b0 + pass + i] : -1;
        if (pe[i] >= p.T * k) {
          set_status(p.ws.hdr, MOE_ERR_DEVICE_CHECK);
          pe[i] = -1;
        }
        const int t = pe[i] >= 0 ? pe[i] / k : 0;
        if (col && pe[i] >= 0)
          load_act_block<XBF16>(p.x, (int64_t)t * H + (int64_t)tau * 32, xr[i]);
        else
#pragma unroll
          for (int c = 0; c < 32; ++c) xr[i][c] = 0.f;
      }
      float acc[kGuVals];
#pragma unroll
      for (int v = 0; v < kGuVals; ++v) acc[v] = 0.f;
      if (col) {
#pragma unroll
        for (int r = 0; r < R; ++r) {
          const int row = r0 + r < I ? r0 + r : I - 1;
          const size_t qo = (size_t)row * (H / 2) + (size_t)tau * 16;
          const size_t so = (size_t)row * nbH + tau;
          const uint4 gq = ldg_stream(ex.gate.q + qo);
          const uint4 uq = ldg_stream(ex.up.q + qo);
          const uint32_t gs = ldg_u8(ex.gate.s + so);
          const uint32_t us = ldg_u8(ex.up.s + so);
          float ag[NT], au[NT];
#pragma unroll
          for (int i = 0; i < NT; ++i) { ag[i] = 0.f; au[i] = 0.f; }
          mx_block_dot<NT>(gq, gs, xr, ag);
          mx_block_dot<NT>(uq, us, xr, au);
#pragma unroll
          for (int i = 0; i < NT; ++i) {
            acc[r * NT + i] = ag[i];
            acc[R * NT + r * NT + i] = au[i];
          }
        }
      }
      const float tot = warp_transpose_reduce<kGuVals>(acc);
      if (lane < kGuVals) red[warp][lane] = tot;
      __syncthreads();
      if (warp == 0) {
        float s = 0.f;
        if (lane < kGuVals)
          for (int w = 0; w < nwarps; ++w) s += red[w][lane];
        const float uval = __shfl_down_sync(0xFFFFFFFFu, s, R * NT);
        if (lane < R * NT) {
          const int r = lane / NT, i = lane % NT;
          const int row = r0 + r;
          if (row < I && pe[i] >= 0) hout[(size_t)pe[i] * I + row] = silu_f32(s) * uval;
        }
      }
      __syncthreads();
    }
  }
}

// -------------------------------------------------------------------- down --
// Work item = (active expert u, tile of G*4 rows of Wd).  Thread
// tau = g * (I/32) + b owns block column b of rows r0 + i*G + g, and keeps
// the h blocks of NT routed pairs in registers.  y[p][row] = Wd[row] . h[p].
constexpr int kDnMaxThreads = 384;
constexpr int kDnRowsPerGroup = 4;

// Row groups per CTA for a given I: as many as fit in kDnMaxThreads, at most 8.
inline int down_groups(int I) {
  const int nbI = I / 32;
  int g = kDnMaxThreads / nbI;
  return g > 8 ? 8 : (g < 1 ? 1 : g);
}

template <int NT>
__global__ void __launch_bounds__(kDnMaxThreads) k_dec_down(ExpertParams p, int G) {
  extern __shared__ float4 dyn_smem4[];
  float* part = reinterpret_cast<float*>(dyn_smem4);  // [nthreads][kDnRowsPerGroup * NT]
  __shared__ int s_item;
  const int H = p.H, I = p.I;
  const int nbI = I / 32;
  const int rows_per_item = G * kDnRowsPerGroup;
  const int nthr = G * nbI;
  const int tau = threadIdx.x;
  const int g = tau / nbI, b = tau % nbI;
  const bool act = tau < nthr;
  pdl_wait();
  pdl_trigger();
  const int U = (int)p.ws.hdr->n_active;
  const int tiles = (H + rows_per_item - 1) / rows_per_item;
  const int n_items = U * tiles;
  const float* hin = reinterpret_cast<const float*>(p.ws.h);
  for (;;) {
    if (threadIdx.x == 0) s_item = (int)atomicAdd(&p.ws.hdr->queue[kQDown], 1u);
    __syncthreads();
    const int item = s_item;
    __syncthreads();
    if (item >= n_items) break;
    const int u = item / tiles, rt = item % tiles;
    const int e = p.ws.act_e[u];
    const int b0 = p.offsets[e], n = p.offsets[e + 1] - b0;
    const moe_expert ex = p.experts[e];
    const int r0 = rt * rows_per_item;
    for (int pass = 0; pass < n; pass += NT) {
      int pe[NT];
      float hr[NT][32];
#pragma unroll
      for (int i = 0; i < NT; ++i) {
        pe[i] = pass + i < n ? p.sorted[b0 + pass + i] : -1;
        if (pe[i] >= p.T * p.k) {
          set_status(p.ws.hdr, MOE_ERR_DEVICE_CHECK);
          pe[i] = -1;
        }
        if (act && pe[i] >= 0)
          load_act_block<false>(hin, (int64_t)pe[i] * I + (int64_t)b * 32, hr[i]);
        else
#pragma unroll
          for (int c = 0; c < 32; ++c) hr[i][c] = 0.f;
      }
      float acc[kDnRowsPerGroup][NT];
#pragma unroll
      for (int r = 0; r < kDnRowsPerGroup; ++r)
#pragma unroll
        for (int i = 0; i < NT; ++i) acc[r][i] = 0.f;
      if (act) {
#pragma unroll
        for (int r = 0; r < kDnRowsPerGroup; ++r) {
          const int row0 = r0 + r * G + g;
          const int row = row0 < H ? row0 : H - 1;
          const uint4 q = ldg_stream(ex.down.q + (size_t)row * (I / 2) + (size_t)b * 16);
          const uint32_t s = ldg_u8(ex.down.s + (size_t)row * nbI + b);
          mx_block_dot<NT>(q, s, hr, acc[r]);
        }
#pragma unroll
        for (int r = 0; r < kDnRowsPerGroup; ++r)
#pragma unroll
          for (int i = 0; i < NT; ++i) part[(size_t)tau * (kDnRowsPerGroup * NT) + r * NT + i] = acc[r][i];
      }
      __syncthreads();
      // Sum over the block columns b = 0..nbI-1 in order.
      for (int o = threadIdx.x; o < rows_per_item * NT; o += blockDim.x) {
        const int i = o % NT, rr = o / NT;        // rr in [0, rows_per_item)
        const int gg = rr % G, r = rr / G;
        const int row = r0 + r * G + gg;
        float s = 0.f;
        for (int bb = 0; bb < nbI; ++bb) s += part[(size_t)(gg * nbI + bb) * (kDnRowsPerGroup * NT) + r * NT + i];
        if (row < H && pe[i] >= 0) p.ws.y[(size_t)pe[i] * H + row] = s;
      }
      __syncthreads();
    }
  }
}

// ----------------------------------------------------------------- combine --
// out[t][h] = (accumulate ? out[t][h] : 0) + sum_{j=0}^{k-1} w[t][j] * y[t*k+j][h]
// in slot order.
__global__ void k_dec_combine(ExpertParams p) {
  pdl_wait();
  const int H = p.H, k = p.k;
  const int H4 = H / 4;
  const int64_t n4 = (int64_t)p.T * H4;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += (int64_t)gridDim.x * blockDim.x) {
    const int t = (int)(i / H4), c4 = (int)(i % H4);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int j = 0; j < k; ++j) {
      const float wj = p.w[t * k + j];
      const float4 y = reinterpret_cast<const float4*>(p.ws.y + (size_t)(t * k + j) * H)[c4];
      acc.x = fmaf(wj, y.x, acc.x);
      acc.y = fmaf(wj, y.y, acc.y);
      acc.z = fmaf(wj, y.z, acc.z);
      acc.w = fmaf(wj, y.w, acc.w);
    }
    float4* o = reinterpret_cast<float4*>(p.out + (size_t)t * H) + c4;
    if (p.accumulate) {
      const float4 r = *o;
      acc.x += r.x; acc.y += r.y; acc.z += r.z; acc.w += r.w;
    }
    *o = acc;
  }
}

template <int NT>
static cudaError_t launch_decode_nt(const ExpertParams& p, cudaStream_t s) {
  const int nsm = device_sm_count();
  const int nbH = p.H / 32;
  const int gu_threads = ((nbH + 31) / 32) * 32;
  auto gu = p.x_bf16 ? k_dec_gateup<NT, true> : k_dec_gateup<NT, false>;
  int occ = 0;
  cudaError_t err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, gu, gu_threads, 0);
  if (err != cudaSuccess) return err;
  if (occ < 1) occ = 1;
  err = launch_pdl(gu, dim3(nsm * occ), dim3(gu_threads), 0, s, p);
  if (err != cudaSuccess) return err;

  const int nbI = p.I / 32;
  const int groups = down_groups(p.I);
  if (nbI > kDnMaxThreads) return cudaErrorNotSupported;
  const int dn_threads = ((groups * nbI + 31) / 32) * 32;
  const size_t dn_smem = (size_t)dn_threads * kDnRowsPerGroup * NT * 4;
  auto dn = k_dec_down<NT>;
  err = cudaFuncSetAttribute(dn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dn_smem);
  if (err != cudaSuccess) return err;
  err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, dn, dn_threads, dn_smem);
  if (err != cudaSuccess) return err;
  if (occ < 1) occ = 1;
  err = launch_pdl(dn, dim3(nsm * occ), dim3(dn_threads), dn_smem, s, p, groups);
  if (err != cudaSuccess) return err;

  const int64_t n4 = (int64_t)p.T * (p.H / 4);
  int cgrid = (int)((n4 + 255) / 256);
  if (cgrid > nsm * 8) cgrid = nsm * 8;
  return launch_pdl(k_dec_combine, dim3(cgrid), dim3(256), 0, s, p);
}

// NT = routed pairs of one expert processed per weight pass.  The choice
// changes only how many times a shared expert's weights are read, never the
// arithmetic of a pair.
cudaError_t launch_decode_experts(const ExpertParams& p, cudaStream_t s) {
  if (p.T == 1) return launch_decode_nt<1>(p, s);
  return launch_decode_nt<2>(p, s);
}

}  // namespace moe
