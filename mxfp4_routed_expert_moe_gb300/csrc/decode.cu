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

#include "async.cuh"
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
__global__ void __launch_bounds__(256) k_dec_gateup_ldg(ExpertParams p) {
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
    if (!expert_ptrs_ok(ex)) {
      if (threadIdx.x == 0) set_status(p.ws.hdr, MOE_ERR_DEVICE_CHECK);
      continue;
    }
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
__global__ void __launch_bounds__(kDnMaxThreads) k_dec_down_ldg(ExpertParams p, int G) {
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
    if (!expert_ptrs_ok(ex)) {
      if (threadIdx.x == 0) set_status(p.ws.hdr, MOE_ERR_DEVICE_CHECK);
      continue;
    }
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
static cudaError_t launch_decode_ldg(const ExpertParams& p, cudaStream_t s) {
  const int nsm = device_sm_count();
  const int nbH = p.H / 32;
  const int gu_threads = ((nbH + 31) / 32) * 32;
  auto gu = p.x_bf16 ? k_dec_gateup_ldg<NT, true> : k_dec_gateup_ldg<NT, false>;
  cudaError_t err;
  int occ = 0;
  if ((err = cached_occupancy((const void*)gu, gu_threads, 0, &occ)) != cudaSuccess) return err;
  prof_before(MOE_STAGE_GATEUP, s);
  err = launch_pdl(gu, dim3(nsm * occ), dim3(gu_threads), 0, s, p);
  prof_after(MOE_STAGE_GATEUP, s);
  if (err != cudaSuccess) return err;

  const int nbI = p.I / 32;
  const int groups = down_groups(p.I);
  if (nbI > kDnMaxThreads) return cudaErrorNotSupported;
  const int dn_threads = ((groups * nbI + 31) / 32) * 32;
  const size_t dn_smem = (size_t)dn_threads * kDnRowsPerGroup * NT * 4;
  auto dn = k_dec_down_ldg<NT>;
  if ((err = ensure_smem_attr((const void*)dn, dn_smem)) != cudaSuccess) return err;
  if ((err = cached_occupancy((const void*)dn, dn_threads, dn_smem, &occ)) != cudaSuccess) return err;
  prof_before(MOE_STAGE_DOWN, s);
  err = launch_pdl(dn, dim3(nsm * occ), dim3(dn_threads), dn_smem, s, p, groups);
  prof_after(MOE_STAGE_DOWN, s);
  if (err != cudaSuccess) return err;

  const int64_t n4 = (int64_t)p.T * (p.H / 4);
  int cgrid = (int)((n4 + 255) / 256);
  if (cgrid > nsm * 8) cgrid = nsm * 8;
  prof_before(MOE_STAGE_COMBINE, s);
  err = launch_pdl(k_dec_combine, dim3(cgrid), dim3(256), 0, s, p);
  prof_after(MOE_STAGE_COMBINE, s);
  return err;
}

// ===================================================== bulk-copy staged path --
// A producer warp streams each work item's weight rows (contiguous ranges of
// nibbles and scales) into a ring of shared-memory stages with the bulk-copy
// engine; consumer warps dequantize from shared memory.  The ring keeps
// ~100 KB per SM in flight independently of the consumers' registers.
constexpr int kGuGroups = 2;       // consumer row groups (one block column per thread each)
constexpr int kGuGroupVals = 8;    // values reduced per warp: 2 matrices x (R/2) rows x NT
constexpr int kMaxStages = 8;

struct RingSmem {
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  int item[kMaxStages];
  int abort_flag;
};

// Producer side of the ring, run by one thread.  `issue(item, stage_ptr, bar)`
// starts the copies of one item; returns false if the ring was aborted.
template <typename NextItem, typename Issue>
__device__ void ring_produce(RingSmem& rs, uint8_t* data, int stages, uint32_t stage_bytes, WsHeader* hdr,
                            NextItem next_item, Issue issue) {
  int issued_use[kMaxStages];
  for (int i = 0; i < kMaxStages; ++i) issued_use[i] = -1;
  bool ok = true;
  for (int it = 0;; ++it) {
    const int s = it % stages, use = it / stages;
    if (use > 0 && !mbar_wait(&rs.empty[s], (use - 1) & 1)) {
      ok = false;
      break;
    }
    if (*(volatile int*)&rs.abort_flag) { ok = false; break; }
    const int item = next_item();
    rs.item[s] = item;
    if (item < 0) {
      mbar_arrive(&rs.full[s]);
      break;
    }
    issue(item, data + (size_t)s * stage_bytes, &rs.full[s]);
    issued_use[s] = use;
  }
  if (!ok) {
    set_status(hdr, MOE_ERR_TIMEOUT);
    rs.abort_flag = 1;
    // Drain: the CTA must not exit while copies into its shared memory are in
    // flight.  Each wait is bounded.
    for (int s = 0; s < stages; ++s)
      if (issued_use[s] >= 0) mbar_wait(&rs.full[s], issued_use[s] & 1);
  }
}

// Gate/up + SwiGLU.  Item = (active expert u, tile of R = 8/NT rows); consumer
// group c (threads [c*ncw*32, (c+1)*ncw*32)) handles local rows c, c+2, ...
template <int NT, bool XBF16>
__global__ void __launch_bounds__(544, 1) k_dec_gateup_tma(ExpertParams p, int stages, uint32_t stage_bytes) {
  constexpr int R = 8 / NT;
  constexpr int RG = R / kGuGroups;  // rows per group
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ RingSmem rs;
  __shared__ float red[16][kGuGroupVals];
  const int H = p.H, I = p.I, k = p.k;
  const int nbH = H / 32;
  const int ncw = (nbH + 31) / 32;           // consumer warps per group
  const int ncons = kGuGroups * ncw * 32;    // consumer threads
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const size_t qrow = (size_t)H / 2;
  const uint32_t qbytes = (uint32_t)(R * qrow), sbytes = (uint32_t)(R * nbH);
  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(&rs.full[s], 1);
      mbar_init(&rs.empty[s], kGuGroups * ncw);
    }
    rs.abort_flag = 0;
    mbar_init_fence();
  }
  __syncthreads();
  pdl_wait();
  pdl_trigger();
  const int U = (int)p.ws.hdr->n_active;
  const int tiles = I / R;
  const int n_items = U * tiles;
  if (warp == kGuGroups * ncw) {
    if (lane == 0) {
      ring_produce(rs, smem, stages, stage_bytes, p.ws.hdr,
                   [&]() {
                     const int item = (int)atomicAdd(&p.ws.hdr->queue[kQGateUp], 1u);
                     return item < n_items ? item : -1;
                   },
                   [&](int item, uint8_t* st, uint64_t* bar) {
                     const int u = item / tiles, rt = item % tiles;
                     const moe_expert ex = p.experts[p.ws.act_e[u]];
                     const size_t r0 = (size_t)rt * R;
                     if (!expert_ptrs_ok(ex)) {
                       set_status(p.ws.hdr, MOE_ERR_DEVICE_CHECK);
                       mbar_arrive(bar);
                       return;
                     }
                     mbar_arrive_expect_tx(bar, 2 * qbytes + 2 * sbytes);
                     bulk_g2s(st, ex.gate.q + r0 * qrow, qbytes, bar);
                     bulk_g2s(st + qbytes, ex.up.q + r0 * qrow, qbytes, bar);
                     bulk_g2s(st + 2 * qbytes, ex.gate.s + r0 * nbH, sbytes, bar);
                     bulk_g2s(st + 2 * qbytes + sbytes, ex.up.s + r0 * nbH, sbytes, bar);
                   });
    }
    return;
  }
  const int grp = warp / ncw;
  const int tau = threadIdx.x - grp * ncw * 32;  // block column
  const bool col = tau < nbH;
  const int gw = warp - grp * ncw;                // warp index inside the group
  float* hout = reinterpret_cast<float*>(p.ws.h);
  float xr[NT][32];
  int xt[NT];
#pragma unroll
  for (int i = 0; i < NT; ++i) xt[i] = -2;
  for (int it = 0;; ++it) {
    const int s = it % stages, use = it / stages;
    if (!mbar_wait(&rs.full[s], use & 1)) {
      set_status(p.ws.hdr, MOE_ERR_TIMEOUT);
      rs.abort_flag = 1;
      break;
    }
    const int item = rs.item[s];
    if (item < 0) break;
    const int u = item / tiles, rt = item % tiles;
    const int e = p.ws.act_e[u];
    const int b0 = p.offsets[e], n = p.offsets[e + 1] - b0;
    const int r0 = rt * R;
    const uint8_t* st = smem + (size_t)s * stage_bytes;
    for (int pass = 0; pass < n; pass += NT) {
      int pe[NT];
#pragma unroll
      for (int i = 0; i < NT; ++i) {
        pe[i] = pass + i < n ? p.sorted[b0 + pass + i] : -1;
        if (pe[i] >= p.T * k) {
          set_status(p.ws.hdr, MOE_ERR_DEVICE_CHECK);
          pe[i] = -1;
        }
        const int t = pe[i] >= 0 ? pe[i] / k : -1;
        if (t != xt[i]) {
          if (col && t >= 0)
            load_act_block<XBF16>(p.x, (int64_t)t * H + (int64_t)tau * 32, xr[i]);
          else
#pragma unroll
            for (int c = 0; c < 32; ++c) xr[i][c] = 0.f;
          xt[i] = t;
        }
      }
      float acc[kGuGroupVals];
#pragma unroll
      for (int v = 0; v < kGuGroupVals; ++v) acc[v] = 0.f;
      if (col) {
#pragma unroll
        for (int r = 0; r < RG; ++r) {
          const int rl = grp + kGuGroups * r;  // local row in the tile
          const uint4 gq = lds128(st + (size_t)rl * qrow + (size_t)tau * 16);
          const uint4 uq = lds128(st + qbytes + (size_t)rl * qrow + (size_t)tau * 16);
          const uint32_t gs = st[2 * qbytes + rl * nbH + tau];
          const uint32_t us = st[2 * qbytes + sbytes + rl * nbH + tau];
          float ag[NT], au[NT];
#pragma unroll
          for (int i = 0; i < NT; ++i) { ag[i] = 0.f; au[i] = 0.f; }
          mx_block_dot<NT>(gq, gs, xr, ag);
          mx_block_dot<NT>(uq, us, xr, au);
#pragma unroll
          for (int i = 0; i < NT; ++i) {
            acc[r * NT + i] = ag[i];
            acc[RG * NT + r * NT + i] = au[i];
          }
        }
      }
      const float tot = warp_transpose_reduce<kGuGroupVals>(acc);
      if (lane < kGuGroupVals) red[warp][lane] = tot;
      named_sync(1, ncons);
      if (gw == 0) {
        float v = 0.f;
        if (lane < kGuGroupVals)
          for (int w = 0; w < ncw; ++w) v += red[grp * ncw + w][lane];
        const float uval = __shfl_down_sync(0xFFFFFFFFu, v, RG * NT);
        if (lane < RG * NT) {
          const int r = lane / NT, i = lane % NT;
          const int row = r0 + grp + kGuGroups * r;
          if (pe[i] >= 0) hout[(size_t)pe[i] * I + row] = silu_f32(v) * uval;
        }
      }
      named_sync(1, ncons);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&rs.empty[s]);
  }
}

// Down.  Item = (active expert u, tile of 4G rows of Wd); thread
// tau = g * (I/32) + b owns block column b of local rows r*G + g.
template <int NT>
__global__ void __launch_bounds__(416, 1) k_dec_down_tma(ExpertParams p, int G, int stages, uint32_t stage_bytes) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ RingSmem rs;
  __shared__ float part[384 * kDnRowsPerGroup * NT];
  const int H = p.H, I = p.I;
  const int nbI = I / 32;
  const int nthr = G * nbI;
  const int ncons = ((nthr + 31) / 32) * 32;
  const int rows_per_item = G * kDnRowsPerGroup;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const size_t qrow = (size_t)I / 2;
  const uint32_t qbytes = (uint32_t)(rows_per_item * qrow), sbytes = (uint32_t)(rows_per_item * nbI);
  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(&rs.full[s], 1);
      mbar_init(&rs.empty[s], ncons / 32);
    }
    rs.abort_flag = 0;
    mbar_init_fence();
  }
  __syncthreads();
  pdl_wait();
  pdl_trigger();
  const int U = (int)p.ws.hdr->n_active;
  const int tiles = H / rows_per_item;
  const int n_items = U * tiles;
  if (warp == ncons / 32) {
    if (lane == 0) {
      ring_produce(rs, smem, stages, stage_bytes, p.ws.hdr,
                   [&]() {
                     const int item = (int)atomicAdd(&p.ws.hdr->queue[kQDown], 1u);
                     return item < n_items ? item : -1;
                   },
                   [&](int item, uint8_t* st, uint64_t* bar) {
                     const int u = item / tiles, rt = item % tiles;
                     const moe_expert ex = p.experts[p.ws.act_e[u]];
                     const size_t r0 = (size_t)rt * rows_per_item;
                     if (!expert_ptrs_ok(ex)) {
                       set_status(p.ws.hdr, MOE_ERR_DEVICE_CHECK);
                       mbar_arrive(bar);
                       return;
                     }
                     mbar_arrive_expect_tx(bar, qbytes + sbytes);
                     bulk_g2s(st, ex.down.q + r0 * qrow, qbytes, bar);
                     bulk_g2s(st + qbytes, ex.down.s + r0 * nbI, sbytes, bar);
                   });
    }
    return;
  }
  const int tau = threadIdx.x;
  const int g = tau / nbI, b = tau % nbI;
  const bool act = tau < nthr;
  const float* hin = reinterpret_cast<const float*>(p.ws.h);
  for (int it = 0;; ++it) {
    const int s = it % stages, use = it / stages;
    if (!mbar_wait(&rs.full[s], use & 1)) {
      set_status(p.ws.hdr, MOE_ERR_TIMEOUT);
      rs.abort_flag = 1;
      break;
    }
    const int item = rs.item[s];
    if (item < 0) break;
    const int u = item / tiles, rt = item % tiles;
    const int e = p.ws.act_e[u];
    const int b0 = p.offsets[e], n = p.offsets[e + 1] - b0;
    const int r0 = rt * rows_per_item;
    const uint8_t* st = smem + (size_t)s * stage_bytes;
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
      if (act) {
        float acc[kDnRowsPerGroup][NT];
#pragma unroll
        for (int r = 0; r < kDnRowsPerGroup; ++r)
#pragma unroll
          for (int i = 0; i < NT; ++i) acc[r][i] = 0.f;
#pragma unroll
        for (int r = 0; r < kDnRowsPerGroup; ++r) {
          const int rl = r * G + g;
          const uint4 q = lds128(st + (size_t)rl * qrow + (size_t)b * 16);
          const uint32_t sc = st[qbytes + rl * nbI + b];
          mx_block_dot<NT>(q, sc, hr, acc[r]);
        }
#pragma unroll
        for (int r = 0; r < kDnRowsPerGroup; ++r)
#pragma unroll
          for (int i = 0; i < NT; ++i) part[(size_t)tau * (kDnRowsPerGroup * NT) + r * NT + i] = acc[r][i];
      }
      named_sync(1, ncons);
      for (int o = threadIdx.x; o < rows_per_item * NT; o += ncons) {
        const int i = o % NT, rr = o / NT;
        const int gg = rr % G, r = rr / G;
        float sum = 0.f;
        for (int bb = 0; bb < nbI; ++bb) sum += part[(size_t)(gg * nbI + bb) * (kDnRowsPerGroup * NT) + r * NT + i];
        if (pe[i] >= 0) p.ws.y[(size_t)pe[i] * H + r0 + r * G + gg] = sum;
      }
      named_sync(1, ncons);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&rs.empty[s]);
  }
}

// Stages that fit the dynamic shared memory budget (>= 2).
static int ring_stages(uint32_t stage_bytes, size_t budget) {
  int n = (int)(budget / stage_bytes);
  return n > kMaxStages ? kMaxStages : n;
}

template <int NT>
static bool tma_path_ok(const ExpertParams& p, int G) {
  const int R = 8 / NT;
  const int nbH = p.H / 32, nbI = p.I / 32;
  const int rd = G * kDnRowsPerGroup;
  return (R * nbH) % 16 == 0 && (rd * nbI) % 16 == 0 && p.H % rd == 0 && (G & (G - 1)) == 0 &&
         G * nbI <= 384 && nbH <= 256;
}

template <int NT>
static cudaError_t launch_decode_tma(const ExpertParams& p, cudaStream_t s) {
  constexpr int R = 8 / NT;
  const int nsm = device_sm_count();
  const size_t budget = 200 * 1024;
  cudaError_t err;
  // gate/up
  const int nbH = p.H / 32;
  const int ncw = (nbH + 31) / 32;
  const uint32_t gu_stage = (uint32_t)(2 * R * (p.H / 2) + 2 * R * nbH);
  const int gu_stages = ring_stages(gu_stage, budget);
  auto gu = p.x_bf16 ? k_dec_gateup_tma<NT, true> : k_dec_gateup_tma<NT, false>;
  const size_t gu_smem = (size_t)gu_stages * gu_stage;
  if ((err = ensure_smem_attr((const void*)gu, gu_smem)) != cudaSuccess) return err;
  prof_before(MOE_STAGE_GATEUP, s);
  err = launch_pdl(gu, dim3(nsm), dim3(kGuGroups * ncw * 32 + 32), gu_smem, s, p, gu_stages, gu_stage);
  prof_after(MOE_STAGE_GATEUP, s);
  if (err != cudaSuccess) return err;
  // down
  int G = down_groups(p.I);
  while (G & (G - 1)) --G;
  const int nbI = p.I / 32;
  const int rd = G * kDnRowsPerGroup;
  const uint32_t dn_stage = (uint32_t)(rd * (p.I / 2) + rd * nbI);
  const int dn_stages = ring_stages(dn_stage, budget);
  const size_t dn_smem = (size_t)dn_stages * dn_stage;
  auto dn = k_dec_down_tma<NT>;
  if ((err = ensure_smem_attr((const void*)dn, dn_smem)) != cudaSuccess) return err;
  const int ncons = ((G * nbI + 31) / 32) * 32;
  prof_before(MOE_STAGE_DOWN, s);
  err = launch_pdl(dn, dim3(nsm), dim3(ncons + 32), dn_smem, s, p, G, dn_stages, dn_stage);
  prof_after(MOE_STAGE_DOWN, s);
  if (err != cudaSuccess) return err;
  const int64_t n4 = (int64_t)p.T * (p.H / 4);
  int cgrid = (int)((n4 + 255) / 256);
  if (cgrid > nsm * 8) cgrid = nsm * 8;
  prof_before(MOE_STAGE_COMBINE, s);
  err = launch_pdl(k_dec_combine, dim3(cgrid), dim3(256), 0, s, p);
  prof_after(MOE_STAGE_COMBINE, s);
  return err;
}

template <int NT>
static cudaError_t launch_decode_nt(const ExpertParams& p, cudaStream_t s) {
  int G = down_groups(p.I);
  while (G & (G - 1)) --G;
  if (tma_path_ok<NT>(p, G)) return launch_decode_tma<NT>(p, s);
  return launch_decode_ldg<NT>(p, s);
}

// NT = routed pairs of one expert processed per weight pass.  The choice
// changes only how many times a shared expert's weights are read, never the
// arithmetic of a pair.
cudaError_t launch_decode_experts(const ExpertParams& p, cudaStream_t s) {
  if (p.T == 1) return launch_decode_nt<1>(p, s);
  return launch_decode_nt<2>(p, s);
}

}  // namespace moe
