// route.cu — router scores, top-k with renormalised weights, and the bucket
// layout (counting sort by expert).
//
// Routing follows [Deltafin's custom compiled runtime, "Complete target
// sequence tape"]: an authoritative top-16 route of ids and fp32 weights in a
// fixed route order; here the order is descending score with ties to the
// lower expert index, and the weights are the softmax of the selected scores.
// The bucket layout groups the routed (token, slot) pairs by expert, which is
// the order of the route union [Deltafin's custom compiled runtime, "Exact
// next-layer expert prefetch"].
#include <utility>

#include "async.cuh"
#include "kernels.h"
#include "decode_mx.cuh"
#include "route_small.cuh"

namespace moe {

// Exclusive scan of per-expert counts (held in ws.offsets[0..E) on entry) into
// ws.offsets (and the caller's copy), plus the active-expert list and the
// prefill tile prefixes.  Called by every thread of one CTA.
__device__ void plan_scan(const BucketParams& p) {
  __shared__ int warp_tot[4][32];
  __shared__ int carry[4];
  const int E = p.E, tid = threadIdx.x, nthreads = blockDim.x;
  const int lane = tid & 31, warp = tid >> 5, nw = nthreads >> 5;
  if (tid < 4) carry[tid] = 0;
  __syncthreads();
  for (int base = 0; base < E; base += nthreads) {
    const int e = base + tid;
    const int c = e < E ? __ldcg(&p.ws.offsets[e]) : 0;
    int v[4] = {c, c > 0 ? 1 : 0, c > 0 ? (c + p.n_tile - 1) / p.n_tile : 0,
                c > 0 ? (c + p.n_tile_gu - 1) / p.n_tile_gu : 0};
    int incl[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      incl[q] = v[q];
#pragma unroll
      for (int m = 1; m < 32; m <<= 1) {
        const int o = __shfl_up_sync(0xFFFFFFFFu, incl[q], m);
        if (lane >= m) incl[q] += o;
      }
      if (lane == 31) warp_tot[q][warp] = incl[q];
    }
    __syncthreads();
    int excl[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      int pre = carry[q];
      for (int w = 0; w < warp; ++w) pre += warp_tot[q][w];
      excl[q] = pre + incl[q] - v[q];
    }
    __syncthreads();
    if (e < E) {
      p.ws.offsets[e] = excl[0];
      if (p.offsets_out) p.offsets_out[e] = excl[0];
      if (c > 0) {
        p.ws.act_e[excl[1]] = e;
        p.ws.act_pref_gu[excl[1]] = excl[3] * p.m_tiles_gu;
        p.ws.act_pref_dn[excl[1]] = excl[2] * p.m_tiles_dn;
      }
    }
    if (tid == 0) {
#pragma unroll
      for (int q = 0; q < 4; ++q)
        for (int w = 0; w < nw; ++w) carry[q] += warp_tot[q][w];
    }
    __syncthreads();
  }
  if (tid == 0) {
    p.ws.offsets[E] = carry[0];
    if (p.offsets_out) p.offsets_out[E] = carry[0];
    p.ws.hdr->n_active = (uint32_t)carry[1];
    p.ws.act_pref_gu[carry[1]] = carry[3] * p.m_tiles_gu;
    p.ws.act_pref_dn[carry[1]] = carry[2] * p.m_tiles_dn;
  }
}

// ------------------------------------------------------ decode router GEMV --
// s[t][e] = sum_h x[t][h] * Wr[e][h] (+ b[e]) for T <= 64, H <= 8192.  Each CTA
// bulk-copies 2 contiguous rows of Wr (57 KB at H = 7168) into shared memory
// while its threads load the activations, then walks the tokens in pairs;
// thread tau handles columns 4*tau + 1024*i.  Four values (2 rows x 2 tokens)
// are reduced per warp in double-float, so every score is summed by the same
// tree whatever T is: a token's route does not depend on the rest of the batch.
constexpr int kRgRows = 2;
constexpr int kRgThreads = 256;
constexpr int kRgChunks = 8;  // float4 chunks per thread per row: H <= 8192

template <bool XBF16>
__device__ __forceinline__ float4 load_x4(const void* x, int64_t idx) {
  if (XBF16) {
    const uint2 v = *reinterpret_cast<const uint2*>(reinterpret_cast<const uint16_t*>(x) + idx);
    return make_float4(__uint_as_float(v.x << 16), __uint_as_float(v.x & 0xFFFF0000u),
                       __uint_as_float(v.y << 16), __uint_as_float(v.y & 0xFFFF0000u));
  } else {
    return *reinterpret_cast<const float4*>(reinterpret_cast<const float*>(x) + idx);
  }
}

template <bool XBF16>
__global__ void __launch_bounds__(kRgThreads) k_router_gemv(RouteParams p) {
  extern __shared__ __align__(128) uint8_t rsm[];  // [kRgRows][H] fp32
  __shared__ uint64_t bar;
  __shared__ float2 red[kRgThreads / 32][kRgRows * 2];
  const int H = p.H, E = p.E, T = p.T;
  const int ncols4 = H / 4;
  const int e0 = blockIdx.x * kRgRows;
  const int nrows = E - e0 < kRgRows ? E - e0 : kRgRows;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const float* wrs = reinterpret_cast<const float*>(rsm);
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    mbar_init_fence();
    mbar_arrive_expect_tx(&bar, (uint32_t)(nrows * H * 4));
    bulk_g2s(rsm, p.wr + (size_t)e0 * H, (uint32_t)(nrows * H * 4), &bar);
  }
  pdl_trigger();
  // The decode expert kernels read the activations as f16 with a per-token
  // shift, or (the persistent block-scaled kernel) as E4M3 terms with its
  // counters cleared: CTA b converts tokens b, b + gridDim.x, .. (bf16 input)
  // while its copy lands.
  if (XBF16 && p.dmx_I > 0) {
    dmx_prepare(p.x, T, H, E, p.dmx_I, p.k, p.ws, blockIdx.x, gridDim.x);
  } else if (XBF16) {
    for (int t = blockIdx.x; t < T; t += gridDim.x) {
      x_row_to_f16(reinterpret_cast<const uint16_t*>(p.x) + (size_t)t * H, H, p.ws.xh + (size_t)t * H,
                   &p.ws.xscale[t]);
      __syncthreads();  // x_row_to_f16 reuses its shared maxima
    }
  }
  __syncthreads();
  bool rows_ready = false;
  for (int tp = 0; tp < T; tp += 2) {
    float4 xr[2][kRgChunks];
#pragma unroll
    for (int i = 0; i < kRgChunks; ++i) {
      const int c4 = threadIdx.x + i * kRgThreads;
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const int t = tp + q;
        xr[q][i] = (c4 < ncols4 && t < T) ? load_x4<XBF16>(p.x, (int64_t)t * H + (int64_t)c4 * 4)
                                         : make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
    if (!rows_ready) {
      if (!mbar_wait_for(&bar, 0, p.wait_limit)) {
        set_status(p.ws.hdr, MOE_ERR_TIMEOUT);
        mbar_wait(&bar, 0);  // bounded drain of the copy in flight
        return;
      }
      rows_ready = true;
    }
    // Each float4 chunk (4 products) is summed in fp32, then added into a
    // double-float accumulator; the reductions below stay double-float.
    float ah[4], al[4];
#pragma unroll
    for (int v = 0; v < 4; ++v) { ah[v] = 0.f; al[v] = 0.f; }
#pragma unroll
    for (int i = 0; i < kRgChunks; ++i) {
      const int c4 = threadIdx.x + i * kRgThreads;
      if (c4 < ncols4) {
#pragma unroll
        for (int r = 0; r < kRgRows; ++r) {
          const float4 wv = reinterpret_cast<const float4*>(wrs + (size_t)(r < nrows ? r : 0) * H)[c4];
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            float a = wv.x * xr[q][i].x;
            a = fmaf(wv.y, xr[q][i].y, a);
            a = fmaf(wv.z, xr[q][i].z, a);
            a = fmaf(wv.w, xr[q][i].w, a);
            df_add_f(ah[r * 2 + q], al[r * 2 + q], a);
          }
        }
      }
    }
    float th, tl;
    warp_transpose_reduce_df<4>(ah, al, th, tl);
    if (lane < 4) red[warp][lane] = make_float2(th, tl);
    __syncthreads();
    if (threadIdx.x < 4) {
      float sh = 0.f, sl = 0.f;
      for (int w = 0; w < kRgThreads / 32; ++w) df_add(sh, sl, red[w][threadIdx.x].x, red[w][threadIdx.x].y, sh, sl);
      const int r = threadIdx.x >> 1, q = threadIdx.x & 1;
      const int e = e0 + r, t = tp + q;
      if (r < nrows && t < T) {
        if (p.br) df_add(sh, sl, p.br[e], 0.f, sh, sl);
        p.ws.logits[(size_t)t * E + e] = make_float2(sh, sl);
      }
    }
    __syncthreads();
  }
  if (!rows_ready) mbar_wait(&bar, 0);  // T == 0 cannot happen; keep the copy drained
}

// Standalone small-batch routing (moe_route): top-k, weights and buckets of
// T <= 64 tokens from the scores, by one CTA.
__global__ void __launch_bounds__(256) k_route_small(RouteParams p) {
  extern __shared__ __align__(16) uint8_t dsm[];
  pdl_wait();
  const int npairs = p.T * p.k;
  const int umax = p.E < npairs ? p.E : npairs;
  SmallPlan plan;
  plan.ue = reinterpret_cast<int*>(dsm);
  plan.ub0 = plan.ue + umax;
  plan.un = plan.ub0 + umax;
  plan.pairs = plan.un + umax;
  char* scratch = reinterpret_cast<char*>(
      (reinterpret_cast<uintptr_t>(plan.pairs + npairs) + 15) & ~(uintptr_t)15);
  route_small(p, scratch, plan, true);
}

size_t small_plan_bytes(int E, int npairs) {
  const int umax = E < npairs ? E : npairs;
  return (size_t)(3 * umax + npairs) * 4;
}

bool route_decode_supported(int T, int H, int E, int k) {
  return T <= kDecodeMaxT && H <= kRgChunks * 4 * kRgThreads && E <= 4096 && k <= kMaxK;
}

cudaError_t launch_router_gemv(const RouteParams& p, cudaStream_t s) {
  const size_t smem = (size_t)kRgRows * p.H * 4;
  const dim3 grid((p.E + kRgRows - 1) / kRgRows);
  auto kern = p.x_bf16 ? k_router_gemv<true> : k_router_gemv<false>;
  cudaError_t err = ensure_smem_attr((const void*)kern, smem);
  if (err != cudaSuccess) return err;
  prof_before(MOE_STAGE_ROUTE, s);
  kern<<<grid, kRgThreads, smem, s>>>(p);
  prof_after(MOE_STAGE_ROUTE, s);
  return cudaGetLastError();
}

cudaError_t launch_route_decode(const RouteParams& p, cudaStream_t s) {
  cudaError_t err = launch_router_gemv(p, s);
  if (err != cudaSuccess) return err;
  const size_t smem = small_plan_bytes(p.E, p.T * p.k) + 16 + route_small_scratch_bytes(p.E, 8, p.T);
  if ((err = ensure_smem_attr((const void*)k_route_small, smem)) != cudaSuccess) return err;
  return launch_pdl(k_route_small, dim3(1), dim3(256), smem, s, p);
}

// df_add_f on two accumulators at once: (h0, l0) += p.x and (h1, l1) += p.y,
// each lane the same two-sum (a - b written as fma(b, -1, a), exact like the
// subtraction).
__device__ __forceinline__ void df_add_f2(float& h0, float& h1, float& l0, float& l1, float2 p) {
  const float2 m1 = make_float2(-1.f, -1.f);
  const float2 a = make_float2(h0, h1);
  const float2 s = __fadd2_rn(a, p);
  const float2 bp = __ffma2_rn(a, m1, s);           // s - a
  const float2 t = __ffma2_rn(bp, m1, s);           // s - bp
  const float2 e1 = __ffma2_rn(t, m1, a);           // a - (s - bp)
  const float2 e2 = __ffma2_rn(bp, m1, p);          // p - bp
  const float2 lo = __fadd2_rn(make_float2(l0, l1), __fadd2_rn(e1, e2));
  h0 = s.x;
  h1 = s.y;
  l0 = lo.x;
  l1 = lo.y;
}

// ------------------------------------------------------- prefill router GEMM --
// s = x Wr^T (+ b) in fp32 on CUDA cores.  A CTA computes 64 experts x 64
// tokens; thread (tx, ty) of 16 x 16 holds 4 experts x 4 tokens.  Each
// 16-wide K step is staged through double-buffered shared memory (vector
// loads for the next step are in flight while this one is computed), summed
// in fp32 and added into a double-float accumulator (hi, lo).  Also clears
// the per-expert token masks.  Small batches have few tiles: the contraction
// is then split over blockIdx.z (router_splits), each split writes its
// (hi, lo) partial sums, and k_router_reduce adds them in split order.
constexpr int kGmTT = 64, kGmTE = 64, kGmK = 16;

template <bool XBF16>
__global__ void __launch_bounds__(256) k_router_gemm(RouteParams p) {
  constexpr int TT = kGmTT, TE = kGmTE, KS = kGmK, NE = TE / 16, NW = TE * 4 / 256;
  __shared__ __align__(16) float xs[2][KS][TT + 4];
  __shared__ __align__(16) float ws_[2][KS][TE + 4];
  const int T = p.T, H = p.H, E = p.E;
  const int t0 = blockIdx.y * TT, e0 = blockIdx.x * TE;
  const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
  // This CTA's part of the contraction: K steps [kbeg, kend).
  const int nsplit = gridDim.z, steps = (H / KS + nsplit - 1) / nsplit;
  const int kbeg = min(H, (int)blockIdx.z * steps * KS), kend = min(H, kbeg + steps * KS);
  {
    const size_t nmask = (size_t)E * ((T + 31) / 32);
    const size_t gtid =
        (((size_t)blockIdx.z * gridDim.y + blockIdx.y) * gridDim.x + blockIdx.x) * blockDim.x + threadIdx.x;
    const size_t gsz = (size_t)gridDim.x * gridDim.y * gridDim.z * blockDim.x;
    for (size_t i = gtid; i < nmask; i += gsz) p.ws.mask[i] = 0u;
  }
  float4 wreg[NW];
  uint4 xreg = make_uint4(0, 0, 0, 0);
  // Global loads of K step kk: W rows (float4 = 4 consecutive k of one
  // expert) and token rows (8 bf16 or 4 fp32 consecutive k of one token).
  auto gload = [&](int kk) {
#pragma unroll
    for (int i = 0; i < NW; ++i) {
      const int idx = tid + i * 256, row = idx >> 2, q = idx & 3, e = e0 + row;
      wreg[i] = e < E ? *reinterpret_cast<const float4*>(p.wr + (size_t)e * H + kk + q * 4)
                      : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    if (XBF16) {
      if (tid < 2 * TT) {
        const int row = tid >> 1, hf = tid & 1, t = t0 + row;
        xreg = t < T ? *reinterpret_cast<const uint4*>(reinterpret_cast<const uint16_t*>(p.x) + (size_t)t * H + kk + hf * 8)
                     : make_uint4(0, 0, 0, 0);
      }
    } else {
      const int row = tid >> 2, q = tid & 3, t = t0 + row;
      xreg = t < T ? *reinterpret_cast<const uint4*>(reinterpret_cast<const float*>(p.x) + (size_t)t * H + kk + q * 4)
                   : make_uint4(0, 0, 0, 0);
    }
  };
  // Store the loaded step k-major into buffer `buf`.
  auto sstore = [&](int buf) {
#pragma unroll
    for (int i = 0; i < NW; ++i) {
      const int idx = tid + i * 256, row = idx >> 2, q = idx & 3;
      ws_[buf][q * 4 + 0][row] = wreg[i].x;
      ws_[buf][q * 4 + 1][row] = wreg[i].y;
      ws_[buf][q * 4 + 2][row] = wreg[i].z;
      ws_[buf][q * 4 + 3][row] = wreg[i].w;
    }
    const uint32_t w[4] = {xreg.x, xreg.y, xreg.z, xreg.w};
    if (XBF16) {
      if (tid < 2 * TT) {
        const int row = tid >> 1, hf = tid & 1;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          xs[buf][hf * 8 + 2 * j][row] = __uint_as_float(w[j] << 16);
          xs[buf][hf * 8 + 2 * j + 1][row] = __uint_as_float(w[j] & 0xFFFF0000u);
        }
      }
    } else {
      const int row = tid >> 2, q = tid & 3;
#pragma unroll
      for (int j = 0; j < 4; ++j) xs[buf][q * 4 + j][row] = __uint_as_float(w[j]);
    }
  };
  float ah[4][NE], al[4][NE];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < NE; ++j) { ah[i][j] = 0.f; al[i][j] = 0.f; }
  if (kbeg < kend) {
    gload(kbeg);
    sstore(0);
  }
  __syncthreads();
  int buf = 0;
  for (int kk = kbeg; kk < kend; kk += KS, buf ^= 1) {
    const bool more = kk + KS < kend;
    if (more) gload(kk + KS);
    // The chunk's fp32 sums, two experts per packed FMA (each lane one fmaf).
    float2 acc[4][NE / 2];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < NE / 2; ++j) acc[i][j] = make_float2(0.f, 0.f);
#pragma unroll
    for (int k = 0; k < KS; ++k) {
      const float4 a4 = *reinterpret_cast<const float4*>(&xs[buf][k][ty * 4]);
      const float a[4] = {a4.x, a4.y, a4.z, a4.w};
      float2 b[NE / 2];
#pragma unroll
      for (int j = 0; j < NE; j += 4) {
        const float4 b4 = *reinterpret_cast<const float4*>(&ws_[buf][k][tx * NE + j]);
        b[j / 2] = make_float2(b4.x, b4.y);
        b[j / 2 + 1] = make_float2(b4.z, b4.w);
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < NE / 2; ++j) acc[i][j] = __ffma2_rn(make_float2(a[i], a[i]), b[j], acc[i][j]);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < NE / 2; ++j) df_add_f2(ah[i][2 * j], ah[i][2 * j + 1], al[i][2 * j], al[i][2 * j + 1], acc[i][j]);
    if (more) sstore(buf ^ 1);
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int t = t0 + ty * 4 + i;
    if (t >= T) continue;
#pragma unroll
    for (int j = 0; j < NE; ++j) {
      const int e = e0 + tx * NE + j;
      if (e < E) {
        if (nsplit > 1) {
          p.ws.rpart[((size_t)blockIdx.z * T + t) * E + e] = make_float2(ah[i][j], al[i][j]);
        } else {
          float sh, sl;
          df_add(ah[i][j], al[i][j], p.br ? p.br[e] : 0.f, 0.f, sh, sl);
          p.ws.logits[(size_t)t * E + e] = make_float2(sh, sl);
        }
      }
    }
  }
}

// logits = the S partial sums added in split order, then the bias.
__global__ void __launch_bounds__(256) k_router_reduce(RouteParams p, int nsplit) {
  const size_t n = (size_t)p.T * p.E;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
    float sh = 0.f, sl = 0.f;
    for (int z = 0; z < nsplit; ++z) {
      const float2 v = p.ws.rpart[(size_t)z * n + i];
      df_add(sh, sl, v.x, v.y, sh, sl);
    }
    const int e = (int)(i % p.E);
    df_add(sh, sl, p.br ? p.br[e] : 0.f, 0.f, sh, sl);
    p.ws.logits[i] = make_float2(sh, sl);
  }
}

// One warp per token: top-k, softmax weights, and the token's bit in the mask
// of each selected expert.
__global__ void __launch_bounds__(256) k_topk(RouteParams p) {
  extern __shared__ float4 dyn_smem4[];
  float2* rows = reinterpret_cast<float2*>(dyn_smem4);
  const int E = p.E, k = p.k, T = p.T;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * (blockDim.x >> 5) + warp;
  if (t >= T) return;
  float2* row = rows + (size_t)warp * E;
  for (int e0 = lane; e0 < E; e0 += 256) {
    float2 v[8];
#pragma unroll
    for (int q = 0; q < 8; ++q)
      if (e0 + 32 * q < E) v[q] = p.ws.logits[(size_t)t * E + e0 + 32 * q];
#pragma unroll
    for (int q = 0; q < 8; ++q)
      if (e0 + 32 * q < E) row[e0 + 32 * q] = v[q];
  }
  __syncwarp();
  int my_e;
  float2 my_s;
  warp_topk(row, E, k, my_e, my_s);
  const float wt = warp_route_weight(my_s, k);
  if (lane < k) {
    p.ids[(size_t)t * k + lane] = my_e;
    p.w[(size_t)t * k + lane] = wt;
    const int W = (T + 31) / 32;
    atomicOr(&p.ws.mask[(size_t)my_e * W + (t >> 5)], 1u << (t & 31));
  }
}

// Mask bits from caller-given ids (experts-only calls without a bucket layout).
__global__ void k_mask_from_ids(BucketParams p) {
  const int T = p.T, k = p.k, E = p.E;
  const int W = (T + 31) / 32;
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= T * k) return;
  const int e = p.ids[i];
  if (e < 0 || e >= E) {
    set_status(p.ws.hdr, MOE_ERR_DEVICE_CHECK);
    return;
  }
  const int t = i / k;
  atomicOr(&p.ws.mask[(size_t)e * W + (t >> 5)], 1u << (t & 31));
}

// One warp per expert: popcounts of its token-mask words, their exclusive
// prefix (wprefix) and its count.  The last CTA to finish scans the counts
// into offsets and builds the plan.
__global__ void __launch_bounds__(256) k_bucket_count(BucketParams p) {
  __shared__ int is_last;
  const int E = p.E, T = p.T;
  const int W = (T + 31) / 32;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int e = blockIdx.x * (blockDim.x >> 5) + warp;
  if (e < E) {
    int run = 0;
    for (int base = 0; base < W; base += 32) {
      const int wi = base + lane;
      const int c = wi < W ? __popc(p.ws.mask[(size_t)e * W + wi]) : 0;
      int incl = c;
#pragma unroll
      for (int m = 1; m < 32; m <<= 1) {
        const int o = __shfl_up_sync(0xFFFFFFFFu, incl, m);
        if (lane >= m) incl += o;
      }
      if (wi < W) p.ws.wprefix[(size_t)e * W + wi] = run + incl - c;
      run += __shfl_sync(0xFFFFFFFFu, incl, 31);
    }
    if (lane == 0) p.ws.offsets[e] = run;  // the count; scanned by the last CTA
  }
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) is_last = atomicAdd(&p.ws.hdr->ticket, 1u) == gridDim.x - 1;
  __syncthreads();
  if (!is_last) return;
  __threadfence();
  plan_scan(p);
  if (threadIdx.x == 0) p.ws.hdr->ticket = 0u;
}

// One thread per routed pair: its position in the expert's bucket.
__global__ void k_bucket_scatter(BucketParams p) {
  const int T = p.T, k = p.k;
  const int W = (T + 31) / 32;
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= T * k) return;
  const int t = i / k;
  const int e = p.ids[i];
  if (e < 0 || e >= p.E) return;
  const uint32_t word = p.ws.mask[(size_t)e * W + (t >> 5)];
  const int pos = p.ws.offsets[e] + p.ws.wprefix[(size_t)e * W + (t >> 5)] + __popc(word & ((1u << (t & 31)) - 1u));
  p.ws.sorted[pos] = i;
  if (p.sorted_out) p.sorted_out[pos] = i;
}

// A checked copy of a caller-given pair list (see launch_copy_pairs).
__global__ void k_copy_pairs(const int32_t* in, int32_t* out, int npairs, WsHeader* hdr) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= npairs) return;
  int v = in[i];
  if (v < 0 || v >= npairs) {
    set_status(hdr, MOE_ERR_DEVICE_CHECK);
    v = -1;
  }
  out[i] = v;
}

// Plan from a caller-given offsets array: counts, then the same scan.
// A layout that is not a partition of [0, T*k) (decreasing offsets, or
// offsets outside that range) is flagged and no expert work is planned.
__global__ void __launch_bounds__(1024) k_plan_from_offsets(BucketParams p, const int32_t* offsets_in) {
  __shared__ int bad;
  if (threadIdx.x == 0) bad = (offsets_in[0] != 0 || offsets_in[p.E] > p.T * p.k) ? 1 : 0;
  __syncthreads();
  for (int e = threadIdx.x; e < p.E; e += blockDim.x) {
    const int c = offsets_in[e + 1] - offsets_in[e];
    if (c < 0) bad = 1;
    p.ws.offsets[e] = c < 0 ? 0 : c;
  }
  __syncthreads();
  if (bad) {
    if (threadIdx.x == 0) {
      set_status(p.ws.hdr, MOE_ERR_DEVICE_CHECK);
      p.ws.hdr->n_active = 0u;
    }
    return;
  }
  __threadfence_block();
  __syncthreads();
  BucketParams q = p;
  q.offsets_out = nullptr;
  plan_scan(q);
}

cudaError_t launch_route_prefill(const RouteParams& p, const BucketParams& b, cudaStream_t s) {
  // 64-expert x 64-token tiles: 80 registers, three CTAs per SM (a 128-expert
  // tile needs 137 registers and one CTA per SM, and was slower).
  const int nsplit = router_splits(p.T, p.E, p.H);
  const dim3 g1((p.E + kGmTE - 1) / kGmTE, (p.T + kGmTT - 1) / kGmTT, nsplit);
  prof_before(MOE_STAGE_ROUTE, s);
  // bf16 batches: the tensor-core screen with exact scores for the candidates
  // (route_tc.cu); otherwise the CUDA-core GEMM for every score.
  cudaError_t err = launch_router_tc(p, s);
  const bool screened = err == cudaSuccess;
  if (err == cudaErrorNotSupported) {
    if (p.x_bf16)
      k_router_gemm<true><<<g1, 256, 0, s>>>(p);
    else
      k_router_gemm<false><<<g1, 256, 0, s>>>(p);
    err = cudaGetLastError();
  }
  if (err == cudaSuccess && !screened && nsplit > 1) {
    const size_t n = (size_t)p.T * p.E;
    const size_t cap = (size_t)device_sm_count() * 8;
    const int grid = (int)((n + 255) / 256 < cap ? (n + 255) / 256 : cap);
    k_router_reduce<<<grid, 256, 0, s>>>(p, nsplit);
    err = cudaGetLastError();
  }
  prof_after(MOE_STAGE_ROUTE, s);
  if (err != cudaSuccess) return err;
  if (!screened) {  // the screen selects the top k itself
    const size_t smem = (size_t)8 * p.E * 8;
    err = ensure_smem_attr((const void*)k_topk, smem);
    if (err != cudaSuccess) return err;
    k_topk<<<(p.T + 7) / 8, 256, smem, s>>>(p);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
  }
  k_bucket_count<<<(p.E + 7) / 8, 256, 0, s>>>(b);
  if ((err = cudaGetLastError()) != cudaSuccess) return err;
  k_bucket_scatter<<<(p.T * p.k + 255) / 256, 256, 0, s>>>(b);
  return cudaGetLastError();
}

cudaError_t launch_copy_pairs(const int32_t* in, int32_t* out, int npairs, WsHeader* hdr, cudaStream_t s) {
  k_copy_pairs<<<(npairs + 255) / 256, 256, 0, s>>>(in, out, npairs, hdr);
  return cudaGetLastError();
}

cudaError_t launch_bucket_from_ids(const BucketParams& b, cudaStream_t s) {
  const size_t W = ((size_t)b.T + 31) / 32;
  cudaError_t err = cudaMemsetAsync(b.ws.mask, 0, (size_t)b.E * W * 4, s);
  if (err != cudaSuccess) return err;
  k_mask_from_ids<<<(b.T * b.k + 255) / 256, 256, 0, s>>>(b);
  if ((err = cudaGetLastError()) != cudaSuccess) return err;
  k_bucket_count<<<(b.E + 7) / 8, 256, 0, s>>>(b);
  if ((err = cudaGetLastError()) != cudaSuccess) return err;
  k_bucket_scatter<<<(b.T * b.k + 255) / 256, 256, 0, s>>>(b);
  return cudaGetLastError();
}

cudaError_t launch_plan_from_offsets(const BucketParams& b, const int32_t* offsets, cudaStream_t s) {
  k_plan_from_offsets<<<1, 1024, 0, s>>>(b, offsets);
  return cudaGetLastError();
}

namespace {
struct KeyVal { const void* k; int a; size_t b; int v; };
KeyVal g_smem_attr[64];
KeyVal g_occ[64];
int g_n_smem = 0, g_n_occ = 0;
}  // namespace

cudaError_t ensure_smem_attr(const void* kernel, size_t bytes) {
  for (int i = 0; i < g_n_smem; ++i)
    if (g_smem_attr[i].k == kernel && g_smem_attr[i].b >= bytes) return cudaSuccess;
  cudaError_t err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (err != cudaSuccess) return err;
  for (int i = 0; i < g_n_smem; ++i)
    if (g_smem_attr[i].k == kernel) { g_smem_attr[i].b = bytes; return cudaSuccess; }
  if (g_n_smem < 64) g_smem_attr[g_n_smem++] = {kernel, 0, bytes, 0};
  return cudaSuccess;
}

cudaError_t cached_occupancy(const void* kernel, int threads, size_t smem, int* out) {
  for (int i = 0; i < g_n_occ; ++i)
    if (g_occ[i].k == kernel && g_occ[i].a == threads && g_occ[i].b == smem) { *out = g_occ[i].v; return cudaSuccess; }
  int occ = 0;
  cudaError_t err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kernel, threads, smem);
  if (err != cudaSuccess) return err;
  if (occ < 1) occ = 1;
  if (g_n_occ < 64) g_occ[g_n_occ++] = {kernel, threads, smem, occ};
  *out = occ;
  return cudaSuccess;
}

int device_sm_count() {
  static int cached = 0;
  if (cached == 0) {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) == cudaSuccess && cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess)
      cached = n;
    else
      cached = kNumSMs;
  }
  return cached;
}

}  // namespace moe
