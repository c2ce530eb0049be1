// decode.cu — weight-streaming MXFP4 expert kernels: decode steps of up to 64
// tokens, and bf16 batches of up to 1024 tokens whose experts each have few
// routed pairs.
//
// The fused MXFP4 dequant+GEMV of [deltafin, "The techniques that bought the
// 82x"] (16-entry table lookup, E8M0 scale as a power of two on the fp32
// exponent) is re-designed for the GPU:
//   * the weights of each routed expert stream from HBM once (bulk copies into
//     a shared-memory ring fed by a producer warp); tokens sharing an expert
//     reuse the same pass;
//   * two E2M1 codes convert to an exact f16x2 with one cvt; each 32-element
//     block's partial sum is scaled once by 2^(e-127), which is exact;
//   * gate/up with bf16 activations (k_dec_gateup_mma) multiplies on warp
//     tensor cores: m16n8k16 MMAs over 8 gate + 8 up rows against 8 routed
//     pairs, the activations carried as f16 with a per-token power-of-two
//     shift so that every product is exact;
//   * down runs on CUDA cores up to 64 tokens (k_dec_down_tma: exact
//     products, one MX block column per thread) and on warp tensor cores for
//     larger batches (k_dec_down_mma: 8 routed pairs per pass); the
//     fp32-activation gate/up and the register-streaming kernels also sum
//     exact products on CUDA cores;
//   * partial sums are added across lanes and warps in a fixed order, so a
//     token's result does not depend on the batch, among batches of up to 64
//     tokens and among larger ones;
//   * the k expert outputs of a token are combined in slot order ([Deltafin's
//     custom compiled runtime, "The native build"]: ordered reduction).
#include <string.h>

#include <utility>

#include "async.cuh"
#include "kernels.h"
#include "route_small.cuh"

namespace moe {

// Dot product of one MX block (16 bytes q, scale s) with NT activation blocks
// of 32 fp32 values each, accumulated into acc[nt] (scaled by 2^(s-127)).
// Even and odd elements accumulate separately (.x and .y), each lane of the
// packed FMA one fmaf.
template <int NT>
__device__ __forceinline__ void mx_block_dot(const uint4 q, uint32_t s, const float (&xr)[NT][32], float (&acc)[NT]) {
  float2 pp[NT];
#pragma unroll
  for (int n = 0; n < NT; ++n) pp[n] = make_float2(0.f, 0.f);
  const uint32_t words[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
  for (int wd = 0; wd < 4; ++wd) {
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const float2 f = f16x2_f32x2(e2m1x2_f16x2(words[wd], b));
      const int c = wd * 8 + b * 2;
#pragma unroll
      for (int n = 0; n < NT; ++n) pp[n] = __ffma2_rn(f, make_float2(xr[n][c], xr[n][c + 1]), pp[n]);
    }
  }
  const float sc = e8m0_f32(s);
#pragma unroll
  for (int n = 0; n < NT; ++n) acc[n] = fmaf(pp[n].x + pp[n].y, sc, acc[n]);
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
    float wj[kMaxK];
    float4 y[kMaxK];
#pragma unroll
    for (int j = 0; j < kMaxK; ++j)
      if (j < k) {
        wj[j] = p.w[t * k + j];
        y[j] = reinterpret_cast<const float4*>(p.ws.y + (size_t)(t * k + j) * H)[c4];
      }
#pragma unroll
    for (int j = 0; j < kMaxK; ++j)
      if (j < k) {
        acc.x = fmaf(wj[j], y[j].x, acc.x);
        acc.y = fmaf(wj[j], y[j].y, acc.y);
        acc.z = fmaf(wj[j], y[j].z, acc.z);
        acc.w = fmaf(wj[j], y[j].w, acc.w);
      }
    float4* o = reinterpret_cast<float4*>(p.out + (size_t)t * H) + c4;
    if (p.accumulate) {
      const float4 r = *o;
      acc.x += r.x; acc.y += r.y; acc.z += r.z; acc.w += r.w;
    }
    *o = acc;
  }
}

static cudaError_t launch_decode_combine(const ExpertParams& p, cudaStream_t s) {
  const int64_t n4 = (int64_t)p.T * (p.H / 4);
  const int64_t cap = (int64_t)device_sm_count() * 8;
  const int cgrid = (int)((n4 + 255) / 256 < cap ? (n4 + 255) / 256 : cap);
  prof_before(MOE_STAGE_COMBINE, s);
  const cudaError_t err = launch_pdl(k_dec_combine, dim3(cgrid), dim3(256), 0, s, p);
  prof_after(MOE_STAGE_COMBINE, s);
  return err;
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

  return launch_decode_combine(p, s);
}

// ===================================================== bulk-copy staged path --
// Per CTA (one per SM), three roles:
//   * a producer thread streams each work item's weight rows (contiguous
//     ranges of nibbles and scales) into a ring of shared-memory stages with
//     the bulk-copy engine, keeping ~100 KB per SM in flight;
//   * consumer warps dequantize from shared memory and reduce each row's
//     partial sums inside the warp (transpose-reduce, fixed tree);
//   * a reducer warp adds the warps' partials in a fixed order and writes the
//     results, fed through two mbarrier-guarded slots, so the consumers never
//     wait on a CTA-wide barrier.
// Bucket metadata (active experts, their bucket offsets and the routed pairs)
// is read once per CTA into shared memory; above kPlanSmemPairs routed pairs
// (batches of more than 64 tokens) the pair list stays in the workspace,
// where it only ever holds checked entries (see load_plan).
constexpr int kMaxStages = 8;
// Sleep between polls of the producer and reducer waits (ns): those warps
// share sub-partitions with the consumer warps, whose issue rate bounds the
// kernels.
constexpr uint32_t kDecPollProducer = 64, kDecPollReducer = 32;
constexpr int kPlanSmemPairs = kDecodeMaxT * kMaxK;
constexpr int kMaxPairs = kDecodeBatchMaxT * kMaxK;  // routed pairs of a decode batch

struct Ring {
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  uint64_t red_full[2];
  uint64_t red_empty[2];
  int item[kMaxStages];
  int abort_flag;
};

// Bucket metadata: per active expert its id, bucket offset, size and the NP
// tensor pointers the kernel streams (read and checked once per CTA, in
// shared memory); and every routed pair (sorted by expert): in shared memory
// (pairs_s) for up to kPlanSmemPairs pairs, else the workspace list.
struct Plan {
  int U;
  int* ue;
  int* ub0;
  int* un;
  int* pairs_s;      // shared-memory copy, or null
  const int* pairs;  // the list the kernel reads: pairs_s or the workspace's
  const uint8_t** ptrs;  // [umax][NP], null for an expert with a bad descriptor
};

__host__ __device__ inline bool plan_pairs_in_smem(int npairs) { return npairs <= kPlanSmemPairs; }

__host__ __device__ inline size_t plan_smem_bytes(int E, int npairs, int np) {
  const int umax = E < npairs ? E : npairs;
  const int sp = plan_pairs_in_smem(npairs) ? npairs : 0;
  return (size_t)(3 * umax + sp) * 4 + 16 + (size_t)umax * np * 8;
}

__device__ Plan plan_carve(const ExpertParams& p, uint8_t* buf, int np) {
  Plan pl;
  const int npairs = p.T * p.k;
  const int umax = p.E < npairs ? p.E : npairs;
  const int sp = plan_pairs_in_smem(npairs) ? npairs : 0;
  pl.U = 0;
  pl.ue = reinterpret_cast<int*>(buf);
  pl.ub0 = pl.ue + umax;
  pl.un = pl.ub0 + umax;
  pl.pairs_s = sp ? pl.un + umax : nullptr;
  pl.pairs = sp ? pl.pairs_s : p.sorted;
  pl.ptrs = reinterpret_cast<const uint8_t**>((reinterpret_cast<uintptr_t>(pl.un + umax + sp) + 15) & ~(uintptr_t)15);
  return pl;
}

// Plan from the published route (workspace / caller layout).  The pairs are
// checked on their way into shared memory; a list too long for that is read
// in place, and the library only passes such a list from its own workspace:
// built by its bucketing kernels, or a checked copy of the caller's (the
// experts-only call copies it with k_copy_pairs first).
__device__ void load_plan(const ExpertParams& p, Plan& pl) {
  pl.U = (int)p.ws.hdr->n_active;
  const int npairs = p.T * p.k;
  for (int u = threadIdx.x; u < pl.U; u += blockDim.x) {
    const int e = p.ws.act_e[u];
    const int b0 = p.offsets[e];
    pl.ue[u] = e;
    pl.ub0[u] = b0;
    pl.un[u] = p.offsets[e + 1] - b0;
  }
  if (!pl.pairs_s) return;
  for (int i = threadIdx.x; i < npairs; i += blockDim.x) {
    int v = p.sorted[i];
    if (v < 0 || v >= npairs) {
      set_status(p.ws.hdr, MOE_ERR_DEVICE_CHECK);
      v = -1;
    }
    pl.pairs_s[i] = v;
  }
}

// Cache the tensor pointers of the active experts (after ue is known).
// which: 0 = gate/up (gate.q, up.q, gate.s, up.s), 1 = down (down.q, down.s).
__device__ void plan_cache_ptrs(const ExpertParams& p, Plan& pl, int which) {
  for (int u = threadIdx.x; u < pl.U; u += blockDim.x) {
    const moe_expert ex = p.experts[pl.ue[u]];
    const bool ok = expert_ptrs_ok(ex);
    if (!ok) set_status(p.ws.hdr, MOE_ERR_DEVICE_CHECK);
    if (which == 0) {
      pl.ptrs[u * 4 + 0] = ok ? ex.gate.q : nullptr;
      pl.ptrs[u * 4 + 1] = ok ? ex.up.q : nullptr;
      pl.ptrs[u * 4 + 2] = ok ? ex.gate.s : nullptr;
      pl.ptrs[u * 4 + 3] = ok ? ex.up.s : nullptr;
    } else {
      pl.ptrs[u * 2 + 0] = ok ? ex.down.q : nullptr;
      pl.ptrs[u * 2 + 1] = ok ? ex.down.s : nullptr;
    }
  }
}

// Producer loop (one thread).  issue(item, stage, bar) starts one item's
// copies.  On a timed-out wait it records MOE_ERR_TIMEOUT, tells the
// consumers and drains its copies in flight before returning.
template <typename NextItem, typename Issue>
__device__ void ring_produce(Ring& rs, uint8_t* data, int stages, uint32_t stage_bytes, WsHeader* hdr,
                             long long wait_limit, NextItem next_item, Issue issue) {
  int issued_use[kMaxStages];
  for (int i = 0; i < kMaxStages; ++i) issued_use[i] = -1;
  bool ok = true;
  for (int it = 0;; ++it) {
    const int s = it % stages, use = it / stages;
    if (use > 0 && !mbar_wait_backoff(&rs.empty[s], (use - 1) & 1, kDecPollProducer, wait_limit)) {
      ok = false;
      break;
    }
    if (*(volatile int*)&rs.abort_flag) {
      ok = false;
      break;
    }
    const int item = next_item();
    rs.item[s] = item;
    if (item < 0) {
      mbar_arrive(&rs.full[s]);
      issued_use[s] = use;
      break;
    }
    issue(item, data + (size_t)s * stage_bytes, &rs.full[s]);
    issued_use[s] = use;
  }
  if (!ok) {
    set_status(hdr, MOE_ERR_TIMEOUT);
    rs.abort_flag = 1;
  }
  // Before the CTA may exit, every copy issued has landed: wait for the last
  // phase this producer started on each stage (complete at once in a normal
  // run; bounded by the default limit).
  for (int s = 0; s < stages; ++s)
    if (issued_use[s] >= 0) mbar_wait(&rs.full[s], issued_use[s] & 1);
}

// h between the staged gate/up and down kernels is stored block-interleaved:
// within each group of 4 blocks (128 values) the 16-byte chunk c of block
// b sits at (c * 4 + b % 4) * 16 bytes, so the four blocks a warp of the down
// kernel needs are read as 64 contiguous bytes per chunk (no bank conflict).
// Requires I % 128 == 0.
__device__ __forceinline__ size_t h_swz(int row) {
  const int b = row >> 5, j = row & 31;
  return (size_t)(b >> 2) * 128 + (size_t)(j >> 2) * 16 + (size_t)(b & 3) * 4 + (size_t)(j & 3);
}

// ---------------------------------------------------------- gate/up + SwiGLU --
// Item = (active expert u, tile of R = 8/NT rows of gate and of up).  Consumer
// group c (ncw warps, one block column per thread) handles local rows c, c+2..
// With bf16 activations each token is carried in f16 scaled by 2^sigma_t
// (largest magnitude in [2^12, 2^13)): an E2M1 weight times such a value has
// at most 10 significant bits, so the f16 product is exact and the sums run in
// fp32 (mixed f16 + f32 adds); 2^-sigma_t is applied to the final sums.
constexpr int kGuGroups = 2;
constexpr int kGuTmaVals = 8;  // per warp and pass: 2 matrices x (R/2) rows x NT
constexpr int kGuRowsNT = 8;   // rows per item x NT (R = 8 / NT)

struct GuRedMeta {
  int r0;
  int ent[2];
  float inv[2];
};

// One MX block dotted with NT tokens held as scaled f16 pairs: acc[n] += sum.
template <int NT>
__device__ __forceinline__ void mx_block_dot_f16(const uint4 q, uint32_t s, const uint32_t (&xh)[NT][16],
                                                 float (&acc)[NT]) {
  // Four accumulator chains per token (even/odd element x even/odd word).
  float pa[NT][4];
#pragma unroll
  for (int n = 0; n < NT; ++n)
#pragma unroll
    for (int c = 0; c < 4; ++c) pa[n][c] = 0.f;
  const uint32_t words[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
  for (int wd = 0; wd < 4; ++wd) {
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const uint32_t w2 = e2m1x2_f16x2(words[wd], b);
      const int c0 = (wd & 1) * 2;
#pragma unroll
      for (int n = 0; n < NT; ++n) {
        uint32_t pr;
        asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(pr) : "r"(w2), "r"(xh[n][wd * 4 + b]));
        asm("{\n .reg .f16 pl, ph;\n mov.b32 {pl, ph}, %2;\n add.rn.f32.f16 %0, pl, %0;\n add.rn.f32.f16 %1, ph, %1;\n}"
            : "+f"(pa[n][c0]), "+f"(pa[n][c0 + 1])
            : "r"(pr));
      }
    }
  }
  const float sc = e8m0_f32(s);
#pragma unroll
  for (int n = 0; n < NT; ++n) acc[n] = fmaf((pa[n][0] + pa[n][1]) + (pa[n][2] + pa[n][3]), sc, acc[n]);
}

template <int NT, bool XBF16>
__global__ void __launch_bounds__(576, 1) k_dec_gateup_tma(ExpertParams p, int stages, uint32_t stage_bytes) {
  constexpr int R = kGuRowsNT / NT;
  constexpr int RG = R / kGuGroups;
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ Ring rs;
  __shared__ float red[2][16][kGuTmaVals];
  __shared__ GuRedMeta rmeta[2];
  __shared__ float gmax[kGuGroups][8];
  const int H = p.H, I = p.I, k = p.k;
  const int nbH = H / 32;
  const int ncw = (nbH + 31) / 32;
  const int ncons_w = kGuGroups * ncw;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const size_t qrow = (size_t)H / 2;
  const uint32_t qbytes = (uint32_t)(R * qrow), sbytes = (uint32_t)(R * nbH);
  uint8_t* ring_data = smem;
  const size_t ring_bytes = (size_t)stages * stage_bytes;
  const size_t scratch_bytes = p.fused_route ? route_small_scratch_bytes(p.E, blockDim.x / 32, p.T) : 0;
  Plan pl = plan_carve(p, smem + (ring_bytes > scratch_bytes ? ring_bytes : scratch_bytes), 4);
  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(&rs.full[s], 1);
      mbar_init(&rs.empty[s], ncons_w);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&rs.red_full[s], ncons_w);
      mbar_init(&rs.red_empty[s], 1);
    }
    rs.abort_flag = 0;
    mbar_init_fence();
  }
  pdl_wait();
  pdl_trigger();
  // Zero the down kernel's per-row-tile completion counters (stream order
  // puts this kernel's completion before the down kernel reads them).
  if (blockIdx.x == 0)
    for (int i = threadIdx.x; i < (H + 31) / 32; i += blockDim.x) p.ws.rowdone[i] = 0u;
  if (p.fused_route) {
    // Route the batch from the router scores in scratch that aliases the
    // (still idle) ring; CTA 0 publishes the route for the down kernel and
    // the caller.
    SmallPlan sp;
    sp.ue = pl.ue;
    sp.ub0 = pl.ub0;
    sp.un = pl.un;
    sp.pairs = pl.pairs_s;
    route_small(p.rp, reinterpret_cast<char*>(ring_data), sp, blockIdx.x == 0);
    pl.U = sp.U;
    // Generic-proxy writes to the ring must be ordered before the bulk
    // copies (async proxy) that will overwrite it.
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  } else {
    load_plan(p, pl);
  }
  __syncthreads();
  plan_cache_ptrs(p, pl, 0);
  __syncthreads();
  const int tiles = I / R;
  const int n_items = pl.U * tiles;

  if (warp == ncons_w + 1) {  // producer
    if (lane == 0)
      ring_produce(rs, ring_data, stages, stage_bytes, p.ws.hdr, p.wait_limit,
                   [&]() {
                     const int item = (int)atomicAdd(&p.ws.hdr->queue[kQGateUp], 1u);
                     return item < n_items ? item : -1;
                   },
                   [&](int item, uint8_t* st, uint64_t* bar) {
                     const int u = item / tiles, rt = item % tiles;
                     const uint8_t* const* pp = pl.ptrs + u * 4;
                     const size_t r0 = (size_t)rt * R;
                     if (!pp[0]) {  // bad descriptor: flagged in the plan, not read
                       mbar_arrive(bar);
                       return;
                     }
                     mbar_arrive_expect_tx(bar, 2 * qbytes + 2 * sbytes);
                     bulk_g2s(st, pp[0] + r0 * qrow, qbytes, bar);
                     bulk_g2s(st + qbytes, pp[1] + r0 * qrow, qbytes, bar);
                     bulk_g2s(st + 2 * qbytes, pp[2] + r0 * nbH, sbytes, bar);
                     bulk_g2s(st + 2 * qbytes + sbytes, pp[3] + r0 * nbH, sbytes, bar);
                   });
    return;
  }

  float* hout = reinterpret_cast<float*>(p.ws.h);
  if (warp == ncons_w) {  // reducer
    for (int pc = 0;; ++pc) {
      const int slot = pc & 1;
      if (!mbar_wait_for(&rs.red_full[slot], (pc >> 1) & 1, p.wait_limit)) {
        set_status(p.ws.hdr, MOE_ERR_TIMEOUT);
        rs.abort_flag = 1;
        break;
      }
      const GuRedMeta m = rmeta[slot];
      if (m.r0 < 0) break;
      const int grp = lane / kGuTmaVals, v = lane % kGuTmaVals;
      float sum = 0.f;
      if (lane < kGuGroups * kGuTmaVals)
        for (int w = 0; w < ncw; ++w) sum += red[slot][grp * ncw + w][v];
      const float other = __shfl_down_sync(0xFFFFFFFFu, sum, RG * NT);
      if (lane < kGuGroups * kGuTmaVals && v < RG * NT) {
        const int r = v / NT, i = v % NT;
        const int row = m.r0 + grp + kGuGroups * r;
        if (m.ent[i] >= 0) {
          const float g = sum * m.inv[i], u = other * m.inv[i];
          hout[(size_t)m.ent[i] * I + h_swz(row)] = silu_f32(g) * u;
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&rs.red_empty[slot]);
    }
    return;
  }

  // consumers
  const int grp = warp / ncw;
  const int gw = warp - grp * ncw;
  const int tau = threadIdx.x - grp * ncw * 32;  // block column
  const bool col = tau < nbH;
  float xr[NT][32];       // fp32 activations (fp32 input)
  uint32_t xh[NT][16];    // scaled f16 pairs (bf16 input)
  float inv[NT];
  int xt[NT];
#pragma unroll
  for (int i = 0; i < NT; ++i) { xt[i] = -2; inv[i] = 1.f; }
  int pc = 0;
  for (int it = 0;; ++it) {
    const int s = it % stages, use = it / stages;
    if (!mbar_wait_for(&rs.full[s], use & 1, p.wait_limit)) {
      set_status(p.ws.hdr, MOE_ERR_TIMEOUT);
      rs.abort_flag = 1;
      break;
    }
    const int item = rs.item[s];
    if (item < 0) break;
    const int u = item / tiles, rt = item % tiles;
    const int b0 = pl.ub0[u], n = pl.un[u];
    const int r0 = rt * R;
    const uint8_t* st = ring_data + (size_t)s * stage_bytes;
    bool dead = false;
    for (int pass = 0; pass < n; pass += NT) {
      int pe[NT];
      bool reload = false;
#pragma unroll
      for (int i = 0; i < NT; ++i) {
        pe[i] = pass + i < n ? pl.pairs[b0 + pass + i] : -1;
        const int t = pe[i] >= 0 ? pe[i] / k : -1;
        reload |= t != xt[i];
      }
      if (reload) {
#pragma unroll
        for (int i = 0; i < NT; ++i) {
          const int t = pe[i] >= 0 ? pe[i] / k : -1;
          float v[32];
          if (col && t >= 0)
            load_act_block<XBF16>(p.x, (int64_t)t * H + (int64_t)tau * 32, v);
          else
#pragma unroll
            for (int c = 0; c < 32; ++c) v[c] = 0.f;
          xt[i] = t;
          if (XBF16) {
            float m = 0.f;
#pragma unroll
            for (int c = 0; c < 32; ++c) m = fmaxf(m, fabsf(v[c]));
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
            if (lane == 0) gmax[grp][gw] = m;
            named_sync(2 + grp, ncw * 32);
            m = 0.f;
            for (int w = 0; w < ncw; ++w) m = fmaxf(m, gmax[grp][w]);
            named_sync(2 + grp, ncw * 32);
            // sigma: largest magnitude scaled into [2^12, 2^13).
            int sig = 0;
            if (m > 0.f) sig = 12 - ((int)((__float_as_uint(m) >> 23) & 0xFF) - 127);
            sig = sig > 100 ? 100 : (sig < -100 ? -100 : sig);
            const float up = __int_as_float((sig + 127) << 23);
            inv[i] = __int_as_float((127 - sig) << 23);
#pragma unroll
            for (int c = 0; c < 16; ++c) {
              const __half2 h2 = __floats2half2_rn(v[2 * c] * up, v[2 * c + 1] * up);
              xh[i][c] = *reinterpret_cast<const uint32_t*>(&h2);
            }
          } else {
#pragma unroll
            for (int c = 0; c < 32; ++c) xr[i][c] = v[c];
            inv[i] = 1.f;
          }
        }
      }
      float acc[kGuTmaVals];
#pragma unroll
      for (int v = 0; v < kGuTmaVals; ++v) acc[v] = 0.f;
      if (col) {
#pragma unroll
        for (int r = 0; r < RG; ++r) {
          const int rl = grp + kGuGroups * r;
          const uint4 gq = lds128(st + (size_t)rl * qrow + (size_t)tau * 16);
          const uint4 uq = lds128(st + qbytes + (size_t)rl * qrow + (size_t)tau * 16);
          const uint32_t gs = st[2 * qbytes + rl * nbH + tau];
          const uint32_t us = st[2 * qbytes + sbytes + rl * nbH + tau];
          float ag[NT], au[NT];
#pragma unroll
          for (int i = 0; i < NT; ++i) { ag[i] = 0.f; au[i] = 0.f; }
          if (XBF16) {
            mx_block_dot_f16<NT>(gq, gs, xh, ag);
            mx_block_dot_f16<NT>(uq, us, xh, au);
          } else {
            mx_block_dot<NT>(gq, gs, xr, ag);
            mx_block_dot<NT>(uq, us, xr, au);
          }
#pragma unroll
          for (int i = 0; i < NT; ++i) {
            acc[r * NT + i] = ag[i];
            acc[RG * NT + r * NT + i] = au[i];
          }
        }
      }
      const float tot = warp_transpose_reduce<kGuTmaVals>(acc);
      const int slot = pc & 1;
      if (pc >= 2 && !mbar_wait_for(&rs.red_empty[slot], ((pc >> 1) - 1) & 1, p.wait_limit)) {
        set_status(p.ws.hdr, MOE_ERR_TIMEOUT);
        rs.abort_flag = 1;
        dead = true;
        break;
      }
      if (lane < kGuTmaVals) red[slot][warp][lane] = tot;
      if (warp == 0 && lane == 0) {
        GuRedMeta m;
        m.r0 = r0;
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          m.ent[i] = i < NT ? pe[i < NT ? i : 0] : -1;
          m.inv[i] = i < NT ? inv[i < NT ? i : 0] : 1.f;
        }
        rmeta[slot] = m;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&rs.red_full[slot]);
      ++pc;
    }
    if (dead) break;
    __syncwarp();
    if (lane == 0) mbar_arrive(&rs.empty[s]);
  }
  // Tell the reducer there is no more work.
  {
    const int slot = pc & 1;
    // After an abort the reducer leaves on its own (its wait gives up).
    if (*(volatile int*)&rs.abort_flag) return;
    if (pc >= 2) mbar_wait(&rs.red_empty[slot], ((pc >> 1) - 1) & 1);
    if (warp == 0 && lane == 0) rmeta[slot].r0 = -1;
    __syncwarp();
    if (lane == 0) mbar_arrive(&rs.red_full[slot]);
  }
}

// ------------------------------------ gate/up + SwiGLU on warp tensor cores --
// bf16 activations, H % 128 == 0.  Item = (active expert u, 8 rows of gate and
// the same 8 rows of up), stacked as the 16 rows of one m16n8k16 A tile; the
// MMA's 8 columns are 8 routed pairs of the expert (one pass).  Consumer warp
// w owns the K-blocks [w*QB, (w+1)*QB), QB = 4*QW, for every item, and keeps
// the activations of its pass columns for those blocks in registers.
//   * Thread (g = lane/4, t = lane%4) reads bytes [4t, 4t+4) of each block
//     (elements 8t..8t+7) of rows g and g+8; one E2M1 byte converts to an
//     exact f16 pair.  The MMA's logical k is permuted so that its slots
//     2t, 2t+1, 2t+8, 2t+9 take elements 8t..8t+3 (first MMA) and 8t+4..8t+7
//     (second); the activation fragment is the same 16 bytes of the pass
//     column's row, so both operands use one permutation and the dot
//     product is unchanged.
//   * Products of an E2M1 value and an f16 activation are exact in the MMA's
//     fp32 accumulation; the block's sum is multiplied once by 2^(s-127).
//   * Rows sit at a stride of H/2 + 16 bytes in shared memory (one bulk copy
//     per row), so the 32 lanes' 4-byte reads fall in 32 distinct banks.
// Warps' partial sums are added by the reducer warp in warp order, and each
// column's arithmetic is independent of the other columns: a pair's result
// does not depend on the rest of the batch.
constexpr int kGmRows = 16;    // rows per item (8 gate over 8 up)
constexpr int kGmCols = 8;     // routed pairs per pass
constexpr int kGmMaxWarps = 14;   // consumer warps
constexpr int kGmProducers = 1;   // producer warps (alternate stages)

struct GmRedMeta {
  int r0;
  int b0;
  int n;
  int pass;
  int release;  // stage to hand back to the producers after this pass, or -1
};

__device__ __forceinline__ void mma_f16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                              uint32_t b0, uint32_t b1, const float (&c)[4]) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%10, %11, %12, %13};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(c[0]), "f"(c[1]), "f"(c[2]), "f"(c[3]));
}

__device__ __forceinline__ uint32_t lds32(const uint8_t* p) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(smem_u32(p)));
  return v;
}

// Bit 7 of a byte of the result is set when that byte of w is 0 or 255 (the
// E8M0 codes that are not a plain exponent field: 2^-127 is subnormal, 255 is
// NaN); other bits are don't-care.
__device__ __forceinline__ uint32_t e8m0_special4(uint32_t w) {
  return ((w - 0x01010101u) & ~w) | ((0xFEFEFEFEu - w) & w);
}


// One K-block of the 16-row tile: acc += (A_blk . B_blk) * 2^(s-127) per row.
template <bool PLAIN, int J>
__device__ __forceinline__ void gm_block(const uint8_t* ag, const uint8_t* au, const uint4 xb, uint32_t sg,
                                         uint32_t su, float (&acc)[4]) {
  const uint32_t wg = lds32(ag), wu = lds32(au);
  const float zero[4] = {0.f, 0.f, 0.f, 0.f};
  float d[4];
  mma_f16_16816(d, e2m1x2_f16x2(wg, 0), e2m1x2_f16x2(wu, 0), e2m1x2_f16x2(wg, 1), e2m1x2_f16x2(wu, 1), xb.x, xb.y,
                zero);
  mma_f16_16816(d, e2m1x2_f16x2(wg, 2), e2m1x2_f16x2(wu, 2), e2m1x2_f16x2(wg, 3), e2m1x2_f16x2(wu, 3), xb.z, xb.w,
                d);
  float fg, fu;
  if (PLAIN) {
    fg = __uint_as_float(((sg >> (8 * J)) & 0xFFu) << 23);
    fu = __uint_as_float(((su >> (8 * J)) & 0xFFu) << 23);
  } else {
    fg = e8m0_f32((sg >> (8 * J)) & 0xFFu);
    fu = e8m0_f32((su >> (8 * J)) & 0xFFu);
  }
  // acc += d * scale, two rows' fmaf per packed FMA.
  const float2 a01 = __ffma2_rn(make_float2(d[0], d[1]), make_float2(fg, fg), make_float2(acc[0], acc[1]));
  const float2 a23 = __ffma2_rn(make_float2(d[2], d[3]), make_float2(fu, fu), make_float2(acc[2], acc[3]));
  acc[0] = a01.x;
  acc[1] = a01.y;
  acc[2] = a23.x;
  acc[3] = a23.y;
}

// One pass over the warp's QW quads of K-blocks with the scales taken as plain
// exponent fields; the scales of rows g and g+8 are read as one word per 4
// blocks from sgp / sup.  Returns nonzero when one of them was 0 or 255 (the
// pass must then be redone by gm_pass_exact).
template <int QW>
__device__ __forceinline__ uint32_t gm_pass(const uint8_t* ag, const uint8_t* au, const uint4 (&xb)[4 * QW],
                                            const uint8_t* sgp, const uint8_t* sup, float (&acc)[4]) {
  uint32_t spec = 0u;
#pragma unroll
  for (int q = 0; q < QW; ++q) {
    const uint32_t sg = lds32(sgp + 4 * q), su = lds32(sup + 4 * q);
    spec |= e8m0_special4(sg) | e8m0_special4(su);
    gm_block<true, 0>(ag + 64 * q, au + 64 * q, xb[4 * q], sg, su, acc);
    gm_block<true, 1>(ag + 64 * q + 16, au + 64 * q + 16, xb[4 * q + 1], sg, su, acc);
    gm_block<true, 2>(ag + 64 * q + 32, au + 64 * q + 32, xb[4 * q + 2], sg, su, acc);
    gm_block<true, 3>(ag + 64 * q + 48, au + 64 * q + 48, xb[4 * q + 3], sg, su, acc);
  }
  return spec & 0x80808080u;
}

// The same pass with every scale converted exactly, block by block (kept
// compact: it runs only for weights holding the codes 0 or 255); the
// activation fragments are read again from xr (null: zeros).
__device__ __noinline__ void gm_pass_exact(const uint8_t* ag, const uint8_t* au, const uint16_t* xr,
                                           const uint8_t* sgp, const uint8_t* sup, int nblk, float (&acc)[4]) {
#pragma unroll 1
  for (int j = 0; j < nblk; ++j) {
    const uint4 x = xr ? *reinterpret_cast<const uint4*>(xr + j * 32) : make_uint4(0u, 0u, 0u, 0u);
    const uint32_t sg = sgp[j], su = sup[j];
    gm_block<false, 0>(ag + 16 * j, au + 16 * j, x, sg, su, acc);
  }
}

__host__ __device__ inline uint32_t gm_row_stride(int H) { return (uint32_t)(H / 2 + 16); }
__host__ __device__ inline uint32_t gm_stage_bytes(int H) {
  const uint32_t b = (uint32_t)kGmRows * gm_row_stride(H) + (uint32_t)kGmRows * (uint32_t)(H / 32);
  return (b + 127u) & ~127u;
}

template <int QW>
__global__ void __launch_bounds__((kGmMaxWarps + kGmProducers + 1) * 32, 1)
    k_dec_gateup_mma(ExpertParams p, int stages, uint32_t stage_bytes) {
  constexpr int QB = 4 * QW;  // K-blocks per consumer warp
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ Ring rs;
  __shared__ float2 red[2][kGmMaxWarps][kGmRows][kGmCols / 2];
  __shared__ GmRedMeta rmeta[2];
  __shared__ float xs_s[kDecodeMaxT];  // 2^-sigma of the first 64 tokens (the others: ws.xscale)
  // Per stage, written by the producer with the item: first row, bucket
  // offset and size, and the tokens of the first pass's 8 columns.
  __shared__ int4 imeta[kMaxStages];
  __shared__ int itok[kMaxStages][kGmCols];
  const int H = p.H, I = p.I, k = p.k;
  const int nbH = H / 32;
  const int W = nbH / QB;  // consumer warps
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t qrow = (uint32_t)(H / 2), qs = gm_row_stride(H);
  const uint32_t sc_off = (uint32_t)kGmRows * qs;
  uint8_t* ring_data = smem;
  const size_t ring_bytes = (size_t)stages * stage_bytes;
  const size_t scratch_bytes = p.fused_route ? route_small_scratch_bytes(p.E, blockDim.x / 32, p.T) : 0;
  Plan pl = plan_carve(p, smem + (ring_bytes > scratch_bytes ? ring_bytes : scratch_bytes), 4);
  if (threadIdx.x == 0) {
    // The reducer hands a stage back once it has read the partial sums of
    // the item's last pass (every consumer warp has finished reading the
    // stage by then).
    for (int s = 0; s < stages; ++s) {
      mbar_init(&rs.full[s], 1);
      mbar_init(&rs.empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&rs.red_full[s], W);
      mbar_init(&rs.red_empty[s], 1);
    }
    rs.abort_flag = 0;
    mbar_init_fence();
  }
  pdl_wait();
  pdl_trigger();
  if (blockIdx.x == 0)
    for (int i = threadIdx.x; i < (H + 31) / 32; i += blockDim.x) p.ws.rowdone[i] = 0u;
  for (int t = threadIdx.x; t < p.T && t < kDecodeMaxT; t += blockDim.x) xs_s[t] = p.ws.xscale[t];
  if (p.fused_route) {
    SmallPlan sp;
    sp.ue = pl.ue;
    sp.ub0 = pl.ub0;
    sp.un = pl.un;
    sp.pairs = pl.pairs_s;
    route_small(p.rp, reinterpret_cast<char*>(ring_data), sp, blockIdx.x == 0);
    pl.U = sp.U;
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  } else {
    load_plan(p, pl);
  }
  __syncthreads();
  plan_cache_ptrs(p, pl, 0);
  __syncthreads();
  const int tiles = I / 8;
  const int n_items = pl.U * tiles;
  // Every item costs the same weight bytes: each CTA takes a contiguous range
  // (consecutive items share an expert, so the consumers' activation
  // registers stay valid), and two producer warps fill alternate stages.
  const int beg = (int)((long long)n_items * blockIdx.x / gridDim.x);
  const int n_mine = (int)((long long)n_items * (blockIdx.x + 1) / gridDim.x) - beg;

  if (warp >= W && warp < W + kGmProducers) {  // producers: 18 lanes issue one item's copies
    int issued_use[kMaxStages];
    for (int i = 0; i < kMaxStages; ++i) issued_use[i] = -1;
    bool ok = true;
    for (int it = warp - W;; it += kGmProducers) {
      const int s = it % stages, use = it / stages;
      const int item = it < n_mine ? beg + it : -1;
      if (lane == 0) {
        if (use > 0 && !mbar_wait_backoff(&rs.empty[s], (use - 1) & 1, kDecPollProducer, p.wait_limit)) ok = false;
        if (ok && *(volatile int*)&rs.abort_flag) ok = false;
        if (ok) rs.item[s] = item;
      }
      ok = __shfl_sync(0xFFFFFFFFu, ok ? 1 : 0, 0) != 0;
      if (!ok) break;
      uint64_t* bar = &rs.full[s];
      if (item < 0) {
        if (lane == 0) {
          mbar_arrive(bar);
          issued_use[s] = use;
        }
        break;
      }
      const int u = item / tiles, rt = item % tiles;
      const uint8_t* const* pp = pl.ptrs + u * 4;
      {
        const int b0 = pl.ub0[u], n = pl.un[u];
        if (lane == 0) imeta[s] = make_int4(rt * 8, b0, n, 0);
        if (lane < kGmCols) {
          const int pe = lane < n ? pl.pairs[b0 + lane] : -1;
          itok[s][lane] = pe >= 0 ? pe / k : -1;
        }
        __syncwarp();
      }
      if (!pp[0]) {  // bad descriptor: flagged in the plan, not read
        if (lane == 0) {
          mbar_arrive(bar);
          issued_use[s] = use;
        }
        continue;
      }
      const size_t r0 = (size_t)rt * 8;
      if (lane == 0) {
        mbar_arrive_expect_tx(bar, (uint32_t)kGmRows * qrow + (uint32_t)kGmRows * (uint32_t)nbH);
        issued_use[s] = use;
      }
      __syncwarp();
      uint8_t* st = ring_data + (size_t)s * stage_bytes;
      if (lane < kGmRows)
        bulk_g2s(st + (size_t)lane * qs, pp[lane >> 3] + (r0 + (lane & 7)) * qrow, qrow, bar);
      else if (lane < kGmRows + 2)
        bulk_g2s(st + sc_off + (size_t)(lane - kGmRows) * 8 * nbH, pp[2 + lane - kGmRows] + r0 * nbH,
                 (uint32_t)(8 * nbH), bar);
    }
    if (lane == 0) {
      if (!ok) {
        set_status(p.ws.hdr, MOE_ERR_TIMEOUT);
        rs.abort_flag = 1;
      }
      // Every copy issued has landed before the CTA may exit (the last phase
      // started on each stage; complete at once in a normal run).
      for (int s = 0; s < stages; ++s)
        if (issued_use[s] >= 0) mbar_wait(&rs.full[s], issued_use[s] & 1);
    }
    return;
  }

  float* hout = reinterpret_cast<float*>(p.ws.h);
  if (warp == W + kGmProducers) {  // reducer: lane = (row r = lane/4, columns 2(lane%4), +1)
    const int r = lane >> 2, c = 2 * (lane & 3);
    for (int pc = 0;; ++pc) {
      const int slot = pc & 1;
      if (!mbar_wait_backoff(&rs.red_full[slot], (pc >> 1) & 1, kDecPollReducer, p.wait_limit)) {
        set_status(p.ws.hdr, MOE_ERR_TIMEOUT);
        rs.abort_flag = 1;
        break;
      }
      const GmRedMeta m = rmeta[slot];
      if (m.r0 < 0) break;
      if (lane == 0 && m.release >= 0) mbar_arrive(&rs.empty[m.release]);  // all warps are past the stage
      float2 gs = make_float2(0.f, 0.f), us = make_float2(0.f, 0.f);
#pragma unroll
      for (int w = 0; w < kGmMaxWarps; ++w)
        if (w < W) {  // warp order; all loads issued together
          const float2 a = red[slot][w][r][c >> 1], b = red[slot][w][r + 8][c >> 1];
          gs.x += a.x;
          gs.y += a.y;
          us.x += b.x;
          us.y += b.y;
        }
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int col = m.pass + c + i;
        if (col < m.n) {
          const int ent = pl.pairs[m.b0 + col];
          if (ent >= 0) {
            const int tk = ent / k;
            const float xs = tk < kDecodeMaxT ? xs_s[tk] : __ldg(&p.ws.xscale[tk]);
            const float g = (i ? gs.y : gs.x) * xs, uu = (i ? us.y : us.x) * xs;
            hout[(size_t)ent * I + h_swz(m.r0 + r)] = silu_f32(g) * uu;
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&rs.red_empty[slot]);
    }
    return;
  }

  // consumers
  const int g = lane >> 2, t = lane & 3;
  const int kb0 = warp * QB;  // first K-block of this warp
  uint4 xb[QB];
#pragma unroll
  for (int j = 0; j < QB; ++j) xb[j] = make_uint4(0u, 0u, 0u, 0u);
  int xt = -1;  // token whose activations are in xb (-1: zeros)
  // The first item's activations are read now, ahead of the burst of weight
  // copies that all CTAs start at once.
  if (n_mine > 0) {
    const int u = beg / tiles, n = pl.un[u];
    const int pe = g < n ? pl.pairs[pl.ub0[u] + g] : -1;
    if (pe >= 0) {
      xt = pe / k;
      const uint16_t* xr = p.ws.xh + (size_t)xt * H + (size_t)kb0 * 32 + 8 * t;
#pragma unroll
      for (int j = 0; j < QB; ++j) xb[j] = *reinterpret_cast<const uint4*>(xr + j * 32);
    }
  }
  int pc = 0;
  bool dead = false;
  int s = 0;
  uint32_t phase = 0u;
  for (;; s = s + 1 == stages ? 0 : s + 1, phase ^= s == 0 ? 1u : 0u) {
    if (!mbar_wait_for(&rs.full[s], phase, p.wait_limit)) {
      set_status(p.ws.hdr, MOE_ERR_TIMEOUT);
      rs.abort_flag = 1;
      break;
    }
    if (rs.item[s] < 0) break;
    const int4 im = imeta[s];
    const int r0 = im.x, b0 = im.y, n = im.z;
    const uint8_t* st = ring_data + (size_t)s * stage_bytes;
    const uint8_t* ag = st + (size_t)g * qs + (size_t)kb0 * 16 + 4 * t;
    const uint8_t* au = ag + (size_t)8 * qs;
    const uint8_t* sgp = st + sc_off + (size_t)g * nbH + kb0;
    const uint8_t* sup = sgp + (size_t)8 * nbH;
    const int npass = n > 0 ? (n + kGmCols - 1) / kGmCols : 1;  // a pass also hands the stage back
    for (int pi = 0; pi < npass; ++pi) {
      const int pass = pi * kGmCols;
      int tok = itok[s][g];
      if (pi > 0) {
        const int pe = pass + g < n ? pl.pairs[b0 + pass + g] : -1;
        tok = pe >= 0 ? pe / k : -1;
      }
      if (tok != xt) {
        if (tok >= 0) {
          const uint16_t* xr = p.ws.xh + (size_t)tok * H + (size_t)kb0 * 32 + 8 * t;
#pragma unroll
          for (int j = 0; j < QB; ++j) xb[j] = *reinterpret_cast<const uint4*>(xr + j * 32);
        } else {
#pragma unroll
          for (int j = 0; j < QB; ++j) xb[j] = make_uint4(0u, 0u, 0u, 0u);
        }
        xt = tok;
      }
      __syncwarp();
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
      // Scale codes 0 and 255 need the exact conversion: the pass is redone
      // (warp-uniform: the MMAs need all lanes).
      if (__any_sync(0xFFFFFFFFu, gm_pass<QW>(ag, au, xb, sgp, sup, acc) != 0u)) {
        acc[0] = acc[1] = acc[2] = acc[3] = 0.f;
        gm_pass_exact(ag, au, tok >= 0 ? p.ws.xh + (size_t)tok * H + (size_t)kb0 * 32 + 8 * t : nullptr, sgp, sup,
                      QB, acc);
      }
      const int slot = pc & 1;
      if (pc >= 2 && !mbar_wait_for(&rs.red_empty[slot], ((pc >> 1) - 1) & 1, p.wait_limit)) {
        set_status(p.ws.hdr, MOE_ERR_TIMEOUT);
        rs.abort_flag = 1;
        dead = true;
        break;
      }
      red[slot][warp][g][t] = make_float2(acc[0], acc[1]);
      red[slot][warp][g + 8][t] = make_float2(acc[2], acc[3]);
      if (warp == 0 && lane == 0) {
        GmRedMeta m;
        m.r0 = r0;
        m.b0 = b0;
        m.n = n;
        m.pass = pass;
        m.release = pi == npass - 1 ? s : -1;
        rmeta[slot] = m;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&rs.red_full[slot]);
      ++pc;
    }
    if (dead) break;
  }
  // Tell the reducer there is no more work.
  {
    const int slot = pc & 1;
    // After an abort the reducer leaves on its own (its wait gives up).
    if (*(volatile int*)&rs.abort_flag) return;
    if (pc >= 2) mbar_wait(&rs.red_empty[slot], ((pc >> 1) - 1) & 1);
    if (warp == 0 && lane == 0) rmeta[slot].r0 = -1;
    __syncwarp();
    if (lane == 0) mbar_arrive(&rs.red_full[slot]);
  }
}

// -------------------------------------------------------- down + combine --
// Item = (active expert u, tile of 64 rows of Wd), one contiguous bulk copy.
// Warp w owns block columns 4w..4w+3 of all 64 rows; lane l owns block column
// 4w + (l & 3) of local rows r*8 + g, g = 2*(l >> 3) + ((l >> 2) & 1), so a
// quarter-warp reads one even and one odd 704-byte row x 4 consecutive 16-byte
// chunks: 8 distinct bank groups, no conflict.  The warp's sum over its 4
// block columns is two xor-shuffle steps; the reducer adds the warps in
// order.  h of the item's first NT pairs is staged by the producer.  For up
// to 64 tokens, when all active experts have written a row tile, the reducer
// that finished last combines it into out in slot order; larger batches are
// combined by k_dec_combine after the kernel (the same arithmetic, spread
// over the whole grid instead of one warp per row tile).
constexpr int kDnG = 8;                 // row groups
constexpr int kDnRPG = 8;               // rows per group
constexpr int kDnRows = kDnG * kDnRPG;  // rows per item

struct DnRedMeta {
  int r0;
  int rt;
  int last;  // 1 on the item's last pass
  int ent[2];
};

template <int NT>
__global__ void __launch_bounds__(448, 1) k_dec_down_tma(ExpertParams p, int stages, uint32_t stage_bytes) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ Ring rs;
  __shared__ float red[2][12][kDnRows * NT];
  __shared__ DnRedMeta rmeta[2];
  const int H = p.H, I = p.I, k = p.k, T = p.T;
  const int nbI = I / 32;
  const int ncons = nbI * kDnG;                // multiple of 32 when nbI % 4 == 0
  const int ncons_w = ncons / 32;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const size_t qrow = (size_t)I / 2;
  const uint32_t qbytes = (uint32_t)(kDnRows * qrow), sbytes = (uint32_t)(kDnRows * nbI);
  const uint32_t hbytes = (uint32_t)(I * 4);
  uint8_t* ring_data = smem;
  Plan pl = plan_carve(p, smem + (size_t)stages * stage_bytes, 2);
  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(&rs.full[s], 1);
      mbar_init(&rs.empty[s], ncons_w);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&rs.red_full[s], ncons_w);
      mbar_init(&rs.red_empty[s], 1);
    }
    rs.abort_flag = 0;
    mbar_init_fence();
  }
  pdl_wait();
  pdl_trigger();
  load_plan(p, pl);
  __syncthreads();
  plan_cache_ptrs(p, pl, 1);
  __syncthreads();
  const int tiles = H / kDnRows;
  const int n_items = pl.U * tiles;
  const float* hin = reinterpret_cast<const float*>(p.ws.h);

  if (warp == ncons_w + 1) {  // producer
    if (lane == 0)
      ring_produce(rs, ring_data, stages, stage_bytes, p.ws.hdr, p.wait_limit,
                   [&]() {
                     const int item = (int)atomicAdd(&p.ws.hdr->queue[kQDown], 1u);
                     return item < n_items ? item : -1;
                   },
                   [&](int item, uint8_t* st, uint64_t* bar) {
                     const int u = item / tiles, rt = item % tiles;
                     const uint8_t* const* pp = pl.ptrs + u * 2;
                     const size_t r0 = (size_t)rt * kDnRows;
                     if (!pp[0]) {  // bad descriptor: flagged in the plan, not read
                       mbar_arrive(bar);
                       return;
                     }
                     const int b0 = pl.ub0[u], n = pl.un[u];
                     int nh = 0;
                     for (int i = 0; i < NT && i < n; ++i) nh += pl.pairs[b0 + i] >= 0 ? 1 : 0;
                     mbar_arrive_expect_tx(bar, qbytes + sbytes + nh * hbytes);
                     bulk_g2s(st, pp[0] + r0 * qrow, qbytes, bar);
                     bulk_g2s(st + qbytes, pp[1] + r0 * nbI, sbytes, bar);
                     for (int i = 0; i < NT && i < n; ++i) {
                       const int pe = pl.pairs[b0 + i];
                       if (pe >= 0) bulk_g2s(st + qbytes + sbytes + i * hbytes, hin + (size_t)pe * I, hbytes, bar);
                     }
                   });
    return;
  }

  if (warp == ncons_w) {  // reducer (+ combine)
    for (int pc = 0;; ++pc) {
      const int slot = pc & 1;
      if (!mbar_wait_backoff(&rs.red_full[slot], (pc >> 1) & 1, kDecPollReducer, p.wait_limit)) {
        set_status(p.ws.hdr, MOE_ERR_TIMEOUT);
        rs.abort_flag = 1;
        break;
      }
      const DnRedMeta m = rmeta[slot];
      if (m.r0 < 0) break;
      // lane owns output rows lane and lane + 32; NT pairs each.
#pragma unroll
      for (int h2 = 0; h2 < kDnRows / 32; ++h2)
#pragma unroll
        for (int i = 0; i < NT; ++i) {
          const int rl = lane + 32 * h2;
          float sum = 0.f;
          for (int w = 0; w < ncons_w; ++w) sum += red[slot][w][rl * NT + i];
          if (m.ent[i] >= 0) p.ws.y[(size_t)m.ent[i] * H + m.r0 + rl] = sum;
        }
      __syncwarp();
      if (lane == 0) mbar_arrive(&rs.red_empty[slot]);
      if (m.last && T <= kDecodeMaxT) {
        __threadfence();
        __syncwarp();
        unsigned prev = 0;
        if (lane == 0) prev = atomicAdd(&p.ws.rowdone[m.rt], 1u);
        prev = __shfl_sync(0xFFFFFFFFu, prev, 0);
        if (prev == (unsigned)pl.U - 1) {
          __threadfence();
          // Last expert of this row tile: out[t][row] in slot order.
          for (int h2 = 0; h2 < kDnRows / 32; ++h2)
          for (int t = 0; t < T; ++t) {
            const int row = m.r0 + lane + 32 * h2;
            float yv[kMaxK], wv[kMaxK];
#pragma unroll
            for (int j = 0; j < kMaxK; ++j) {
              if (j < k) {
                yv[j] = __ldcg(&p.ws.y[(size_t)(t * k + j) * H + row]);
                wv[j] = __ldg(&p.w[t * k + j]);
              }
            }
            float acc = 0.f;
#pragma unroll
            for (int j = 0; j < kMaxK; ++j)
              if (j < k) acc = fmaf(wv[j], yv[j], acc);
            float* o = p.out + (size_t)t * H + row;
            if (p.accumulate) acc += *o;
            *o = acc;
          }
        }
      }
    }
    return;
  }

  // consumers
  const int b = 4 * warp + (lane & 3);
  const int g = 2 * (lane >> 3) + ((lane >> 2) & 1);
  float hr[NT][32];
  int hcur[NT];
#pragma unroll
  for (int i = 0; i < NT; ++i) hcur[i] = -2;
  int pc = 0;
  for (int it = 0;; ++it) {
    const int s = it % stages, use = it / stages;
    if (!mbar_wait_for(&rs.full[s], use & 1, p.wait_limit)) {
      set_status(p.ws.hdr, MOE_ERR_TIMEOUT);
      rs.abort_flag = 1;
      break;
    }
    const int item = rs.item[s];
    if (item < 0) break;
    const int u = item / tiles, rt = item % tiles;
    const int b0 = pl.ub0[u], n = pl.un[u];
    const int r0 = rt * kDnRows;
    const uint8_t* st = ring_data + (size_t)s * stage_bytes;
    bool dead = false;
    for (int pass = 0; pass < n; pass += NT) {
      int pe[NT];
#pragma unroll
      for (int i = 0; i < NT; ++i) {
        pe[i] = pass + i < n ? pl.pairs[b0 + pass + i] : -1;
        if (pe[i] != hcur[i]) {
          if (pe[i] < 0) {
#pragma unroll
            for (int c = 0; c < 32; ++c) hr[i][c] = 0.f;
          } else {
            // Block b of the interleaved h: chunk c at float4 (b/4)*32 + c*4 + b%4.
            const float4* src = pass == 0 ? reinterpret_cast<const float4*>(st + qbytes + sbytes + i * hbytes)
                                          : reinterpret_cast<const float4*>(hin + (size_t)pe[i] * I);
            src += (b >> 2) * 32 + (b & 3);
#pragma unroll
            for (int c = 0; c < 8; ++c) {
              const float4 v = src[c * 4];
              hr[i][4 * c] = v.x; hr[i][4 * c + 1] = v.y; hr[i][4 * c + 2] = v.z; hr[i][4 * c + 3] = v.w;
            }
          }
          hcur[i] = pe[i];
        }
      }
      float acc[kDnRPG][NT];
#pragma unroll
      for (int r = 0; r < kDnRPG; ++r)
#pragma unroll
        for (int i = 0; i < NT; ++i) acc[r][i] = 0.f;
#pragma unroll
      for (int r = 0; r < kDnRPG; ++r) {
        const int rl = r * kDnG + g;
        const uint4 q = lds128(st + (size_t)rl * qrow + (size_t)b * 16);
        const uint32_t sc = st[qbytes + rl * nbI + b];
        mx_block_dot<NT>(q, sc, hr, acc[r]);
      }
      // Sum the warp's 4 block columns (lanes with equal g): xor 1, xor 2.
#pragma unroll
      for (int r = 0; r < kDnRPG; ++r)
#pragma unroll
        for (int i = 0; i < NT; ++i) {
          float v = acc[r][i];
          v += __shfl_xor_sync(0xFFFFFFFFu, v, 1);
          v += __shfl_xor_sync(0xFFFFFFFFu, v, 2);
          acc[r][i] = v;
        }
      const int slot = pc & 1;
      if (pc >= 2 && !mbar_wait_for(&rs.red_empty[slot], ((pc >> 1) - 1) & 1, p.wait_limit)) {
        set_status(p.ws.hdr, MOE_ERR_TIMEOUT);
        rs.abort_flag = 1;
        dead = true;
        break;
      }
      if ((lane & 3) == 0) {
#pragma unroll
        for (int r = 0; r < kDnRPG; ++r)
#pragma unroll
          for (int i = 0; i < NT; ++i) red[slot][warp][(r * kDnG + g) * NT + i] = acc[r][i];
      }
      if (warp == 0 && lane == 0) {
        DnRedMeta m;
        m.r0 = r0;
        m.rt = rt;
        m.last = pass + NT >= n ? 1 : 0;
#pragma unroll
        for (int i = 0; i < 2; ++i) m.ent[i] = i < NT ? pe[i < NT ? i : 0] : -1;
        rmeta[slot] = m;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&rs.red_full[slot]);
      ++pc;
    }
    if (dead) break;
    __syncwarp();
    if (lane == 0) mbar_arrive(&rs.empty[s]);
  }
  {
    const int slot = pc & 1;
    // After an abort the reducer leaves on its own (its wait gives up).
    if (*(volatile int*)&rs.abort_flag) return;
    if (pc >= 2) mbar_wait(&rs.red_empty[slot], ((pc >> 1) - 1) & 1);
    if (warp == 0 && lane == 0) rmeta[slot].r0 = -1;
    __syncwarp();
    if (lane == 0) mbar_arrive(&rs.red_full[slot]);
  }
}

// ------------------------------------- down + combine on warp tensor cores --
// Decode batches above 64 tokens (after k_dec_gateup_mma), I % 128 == 0.
// (Up to 64 tokens k_dec_down_tma runs: it is faster at one token, and one
// kernel serves that whole range so that a token's result does not depend
// on the batch.)  Item =
// (active expert u, 64 rows of Wd) = four m16n8k16 A tiles; the MMA's 8
// columns are 8 routed pairs (one pass).  Consumer warp w owns the K-blocks
// [4w, 4w+4) of I for every item and keeps the pass columns' h for them in
// registers as two f16 terms, hi + lo, of h * 2^sigma (about 22 significant
// bits; sigma per pair and warp puts the largest magnitude of that range in
// [2^14, 2^15)); the sum is multiplied by 2^-sigma after the warp's blocks.
// Rows are copied in pairs (or one by one when I/2 is a multiple of 128
// bytes) with 16 bytes of padding per copy, which puts the 8 rows a fragment
// read touches at 8 distinct 16-byte bank groups.  Two reducer warps (one per
// hand-off slot) add the warps' partial sums in order and write y; the
// slot-ordered combine into out is the next launch (k_dec_combine, spread
// over the whole GPU).
constexpr int kDmRows = 64;                // rows of Wd per item
constexpr int kDmTiles = kDmRows / 16;     // MMA row tiles per item
constexpr int kDmMaxWarps = 12;            // consumer warps (I <= 1536)

struct DmRedMeta {
  int r0;    // first row of the item
  int b0;    // bucket offset of the expert
  int n;     // routed pairs of the expert
  int pass;  // first pair of this pass
};

constexpr int kDmRpcOverride = 0;
__host__ __device__ inline int dm_rows_per_copy(int I) {
  return kDmRpcOverride ? kDmRpcOverride : ((I / 2) % 128 == 64 ? 2 : 1);
}
__host__ __device__ inline uint32_t dm_group_stride(int I) {
  return (uint32_t)(dm_rows_per_copy(I) * (I / 2) + 16);
}
__host__ __device__ inline uint32_t dm_row_off(int r, int I) {
  const int rpc = dm_rows_per_copy(I);
  return (uint32_t)(r / rpc) * dm_group_stride(I) + (uint32_t)(r % rpc) * (uint32_t)(I / 2);
}
__host__ __device__ inline uint32_t dm_scale_off(int I) {
  return (uint32_t)(kDmRows / dm_rows_per_copy(I)) * dm_group_stride(I);
}
__host__ __device__ inline uint32_t dm_stage_bytes(int I) {
  return (dm_scale_off(I) + (uint32_t)kDmRows * (uint32_t)(I / 32) + 127u) & ~127u;
}

// One K-block of one 16-row tile against the hi and lo activation terms.
template <bool PLAIN, int J>
__device__ __forceinline__ void dm_block(const uint32_t wg, const uint32_t wu, const uint4 hb, const uint4 lb,
                                         uint32_t sg, uint32_t su, float (&acc)[4]) {
  const float zero[4] = {0.f, 0.f, 0.f, 0.f};
  const uint32_t a0 = e2m1x2_f16x2(wg, 0), a1 = e2m1x2_f16x2(wu, 0), a2 = e2m1x2_f16x2(wg, 1),
                 a3 = e2m1x2_f16x2(wu, 1);
  const uint32_t a4 = e2m1x2_f16x2(wg, 2), a5 = e2m1x2_f16x2(wu, 2), a6 = e2m1x2_f16x2(wg, 3),
                 a7 = e2m1x2_f16x2(wu, 3);
  float d[4];
  mma_f16_16816(d, a0, a1, a2, a3, hb.x, hb.y, zero);
  mma_f16_16816(d, a4, a5, a6, a7, hb.z, hb.w, d);
  mma_f16_16816(d, a0, a1, a2, a3, lb.x, lb.y, d);
  mma_f16_16816(d, a4, a5, a6, a7, lb.z, lb.w, d);
  float fg, fu;
  if (PLAIN) {
    fg = __uint_as_float(((sg >> (8 * J)) & 0xFFu) << 23);
    fu = __uint_as_float(((su >> (8 * J)) & 0xFFu) << 23);
  } else {
    fg = e8m0_f32((sg >> (8 * J)) & 0xFFu);
    fu = e8m0_f32((su >> (8 * J)) & 0xFFu);
  }
  acc[0] = fmaf(d[0], fg, acc[0]);
  acc[1] = fmaf(d[1], fg, acc[1]);
  acc[2] = fmaf(d[2], fu, acc[2]);
  acc[3] = fmaf(d[3], fu, acc[3]);
}

// The four blocks of one tile: rows at ag (row g) and au (row g + 8), scale
// words sg / su.
template <bool PLAIN>
__device__ __forceinline__ void dm_tile(const uint8_t* ag, const uint8_t* au, const uint4 (&hb)[4],
                                        const uint4 (&lb)[4], uint32_t sg, uint32_t su, float (&acc)[4]) {
  dm_block<PLAIN, 0>(lds32(ag), lds32(au), hb[0], lb[0], sg, su, acc);
  dm_block<PLAIN, 1>(lds32(ag + 16), lds32(au + 16), hb[1], lb[1], sg, su, acc);
  dm_block<PLAIN, 2>(lds32(ag + 32), lds32(au + 32), hb[2], lb[2], sg, su, acc);
  dm_block<PLAIN, 3>(lds32(ag + 48), lds32(au + 48), hb[3], lb[3], sg, su, acc);
}

__global__ void __launch_bounds__((kDmMaxWarps + 3) * 32, 1)
    k_dec_down_mma(ExpertParams p, int stages, uint32_t stage_bytes) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ Ring rs;
  __shared__ float2 red[2][kDmMaxWarps][kDmTiles][16][kGmCols / 2];
  __shared__ DmRedMeta rmeta[2];
  const int H = p.H, I = p.I;
  const int nbI = I / 32;
  const int W = nbI / 4;  // consumer warps
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t qrow = (uint32_t)(I / 2);
  const int rpc = dm_rows_per_copy(I);
  const uint32_t gstride = dm_group_stride(I), sc_off = dm_scale_off(I);
  uint8_t* ring_data = smem;
  Plan pl = plan_carve(p, smem + (size_t)stages * stage_bytes, 2);
  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(&rs.full[s], 1);
      mbar_init(&rs.empty[s], W);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&rs.red_full[s], W);
      mbar_init(&rs.red_empty[s], 1);
    }
    rs.abort_flag = 0;
    mbar_init_fence();
  }
  pdl_wait();
  pdl_trigger();
  load_plan(p, pl);
  __syncthreads();
  plan_cache_ptrs(p, pl, 1);
  __syncthreads();
  const int tiles = H / kDmRows;
  const int n_items = pl.U * tiles;
  const int beg = (int)((long long)n_items * blockIdx.x / gridDim.x);
  const int n_mine = (int)((long long)n_items * (blockIdx.x + 1) / gridDim.x) - beg;
  const float* hin = reinterpret_cast<const float*>(p.ws.h);

  if (warp == W) {  // producer: the lanes issue one item's copies
    int issued_use[kMaxStages];
    for (int i = 0; i < kMaxStages; ++i) issued_use[i] = -1;
    bool ok = true;
    const int ncopy = kDmRows / rpc;
    for (int it = 0;; ++it) {
      const int s = it % stages, use = it / stages;
      const int item = it < n_mine ? beg + it : -1;
      if (lane == 0) {
        if (use > 0 && !mbar_wait_for(&rs.empty[s], (use - 1) & 1, p.wait_limit)) ok = false;
        if (ok && *(volatile int*)&rs.abort_flag) ok = false;
        if (ok) rs.item[s] = item;
      }
      ok = __shfl_sync(0xFFFFFFFFu, ok ? 1 : 0, 0) != 0;
      if (!ok) break;
      uint64_t* bar = &rs.full[s];
      if (item < 0) {
        if (lane == 0) {
          mbar_arrive(bar);
          issued_use[s] = use;
        }
        break;
      }
      const int u = item / tiles, rt = item % tiles;
      const uint8_t* const* pp = pl.ptrs + u * 2;
      if (!pp[0]) {  // bad descriptor: flagged in the plan, not read
        if (lane == 0) {
          mbar_arrive(bar);
          issued_use[s] = use;
        }
        continue;
      }
      const size_t r0 = (size_t)rt * kDmRows;
      if (lane == 0) {
        mbar_arrive_expect_tx(bar, (uint32_t)kDmRows * qrow + (uint32_t)kDmRows * (uint32_t)nbI);
        issued_use[s] = use;
      }
      __syncwarp();
      uint8_t* st = ring_data + (size_t)s * stage_bytes;
      for (int c = lane; c < ncopy; c += 32)
        bulk_g2s(st + (size_t)c * gstride, pp[0] + (r0 + (size_t)c * rpc) * qrow, (uint32_t)rpc * qrow, bar);
      if (lane == 31) bulk_g2s(st + sc_off, pp[1] + r0 * nbI, (uint32_t)(kDmRows * nbI), bar);
    }
    if (lane == 0) {
      if (!ok) {
        set_status(p.ws.hdr, MOE_ERR_TIMEOUT);
        rs.abort_flag = 1;
      }
      // Every copy issued has landed before the CTA may exit (the last phase
      // started on each stage; complete at once in a normal run).
      for (int s = 0; s < stages; ++s)
        if (issued_use[s] >= 0) mbar_wait(&rs.full[s], issued_use[s] & 1);
    }
    return;
  }

  if (warp == W + 1 || warp == W + 2) {  // reducers: reducer r takes the passes that use slot r
    const int slot = warp - (W + 1);
    for (int j = 0;; ++j) {
      if (!mbar_wait_for(&rs.red_full[slot], j & 1, p.wait_limit)) {
        set_status(p.ws.hdr, MOE_ERR_TIMEOUT);
        rs.abort_flag = 1;
        break;
      }
      const DmRedMeta m = rmeta[slot];
      if (m.r0 < 0) break;
      // Lane: outputs o = lane + 32 q = (tile, row, column pair cp), columns
      // 2cp and 2cp+1 of the pass; the warps' partial sums are added in warp
      // order (all loads issued together).
      constexpr int kOut = kDmTiles * 16 * (kGmCols / 2) / 32;
      float2 sums[kOut];
#pragma unroll
      for (int q = 0; q < kOut; ++q) {
        const int o = lane + 32 * q;
        const int tile = o / (16 * (kGmCols / 2)), rem = o % (16 * (kGmCols / 2));
        const int r = rem / (kGmCols / 2), cp = rem % (kGmCols / 2);
        float2 sum = make_float2(0.f, 0.f);
#pragma unroll
        for (int w = 0; w < kDmMaxWarps; ++w)
          if (w < W) {
            const float2 v = red[slot][w][tile][r][cp];
            sum.x += v.x;
            sum.y += v.y;
          }
        sums[q] = sum;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&rs.red_empty[slot]);
#pragma unroll
      for (int q = 0; q < kOut; ++q) {
        const int o = lane + 32 * q;
        const int tile = o / (16 * (kGmCols / 2)), rem = o % (16 * (kGmCols / 2));
        const int r = rem / (kGmCols / 2), cp = rem % (kGmCols / 2);
        const float2 sum = sums[q];
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const int col = m.pass + 2 * cp + i;
          if (col < m.n) {
            const int ent = pl.pairs[m.b0 + col];
            if (ent >= 0) p.ws.y[(size_t)ent * H + m.r0 + 16 * tile + r] = i ? sum.y : sum.x;
          }
        }
      }
    }
    return;
  }

  // consumers
  const int g = lane >> 2, t = lane & 3;
  const int kb0 = warp * 4;  // first K-block of this warp
  uint4 hb[4], lb[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) hb[j] = lb[j] = make_uint4(0u, 0u, 0u, 0u);
  float cs[2] = {1.f, 1.f};  // 2^-sigma of columns 2t and 2t+1
  int hcur = -2;             // pair whose h is in hb / lb (-1: zeros)
  int pc = 0;
  bool dead = false;
  for (int it = 0; !dead; ++it) {
    const int s = it % stages;
    if (!mbar_wait_for(&rs.full[s], (it / stages) & 1, p.wait_limit)) {
      set_status(p.ws.hdr, MOE_ERR_TIMEOUT);
      rs.abort_flag = 1;
      break;
    }
    const int item = rs.item[s];
    if (item < 0) break;
    const int u = item / tiles, rt = item % tiles;
    const int b0 = pl.ub0[u], n = pl.un[u];
    const uint8_t* st = ring_data + (size_t)s * stage_bytes;
    const uint8_t* scp = st + sc_off + (size_t)kb0;  // + row * nbI
    const int npass = n > 0 ? (n + kGmCols - 1) / kGmCols : 1;
    for (int pi = 0; pi < npass; ++pi) {
      const int pass = pi * kGmCols;
      const int pe = pass + g < n ? pl.pairs[b0 + pass + g] : -1;
      if (__any_sync(0xFFFFFFFFu, pe != hcur)) {
        // h of pair pe (column g), elements 8t..8t+7 of the warp's 4 blocks;
        // h is stored block-interleaved (h_swz): the 4 floats of chunk c of
        // block b sit at float (b/4)*128 + c*16 + (b%4)*4.
        float v[4][8];
        float m = 0.f;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int b = kb0 + j;
          if (pe >= 0) {
            const float* src = hin + (size_t)pe * I + (size_t)(b >> 2) * 128 + (b & 3) * 4;
            const float4 x0 = *reinterpret_cast<const float4*>(src + (2 * t) * 16);
            const float4 x1 = *reinterpret_cast<const float4*>(src + (2 * t + 1) * 16);
            v[j][0] = x0.x; v[j][1] = x0.y; v[j][2] = x0.z; v[j][3] = x0.w;
            v[j][4] = x1.x; v[j][5] = x1.y; v[j][6] = x1.z; v[j][7] = x1.w;
          } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) v[j][e] = 0.f;
          }
#pragma unroll
          for (int e = 0; e < 8; ++e) m = fmaxf(m, fabsf(v[j][e]));
        }
        m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));
        m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, 2));
        int sig = 0;
        if (m > 0.f) sig = 14 - ((int)((__float_as_uint(m) >> 23) & 0xFF) - 127);
        sig = sig > 100 ? 100 : (sig < -100 ? -100 : sig);
        const float up = __int_as_float((sig + 127) << 23);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          uint32_t hi[4], lo[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float a = v[j][2 * e] * up, b = v[j][2 * e + 1] * up;
            const __half2 h2 = __floats2half2_rn(a, b);
            const float2 hf = __half22float2(h2);
            const __half2 l2 = __floats2half2_rn(a - hf.x, b - hf.y);
            hi[e] = *reinterpret_cast<const uint32_t*>(&h2);
            lo[e] = *reinterpret_cast<const uint32_t*>(&l2);
          }
          hb[j] = make_uint4(hi[0], hi[1], hi[2], hi[3]);
          lb[j] = make_uint4(lo[0], lo[1], lo[2], lo[3]);
        }
        const float inv = __int_as_float((127 - sig) << 23);
        cs[0] = __shfl_sync(0xFFFFFFFFu, inv, 4 * (2 * t));
        cs[1] = __shfl_sync(0xFFFFFFFFu, inv, 4 * (2 * t + 1));
        hcur = pe;
      }
      float acc[kDmTiles][4];
#pragma unroll
      for (int tl = 0; tl < kDmTiles; ++tl) acc[tl][0] = acc[tl][1] = acc[tl][2] = acc[tl][3] = 0.f;
      uint32_t spec = 0u;
#pragma unroll
      for (int tl = 0; tl < kDmTiles; ++tl) {
        const int rg = 16 * tl + g;
        const uint32_t sg = lds32(scp + (size_t)rg * nbI), su = lds32(scp + (size_t)(rg + 8) * nbI);
        spec |= e8m0_special4(sg) | e8m0_special4(su);
        dm_tile<true>(st + dm_row_off(rg, I) + kb0 * 16 + 4 * t, st + dm_row_off(rg + 8, I) + kb0 * 16 + 4 * t, hb,
                      lb, sg, su, acc[tl]);
      }
      // Scale codes 0 and 255 need the exact conversion: the pass is redone
      // (warp-uniform: the MMAs need all lanes).
      if (__any_sync(0xFFFFFFFFu, (spec & 0x80808080u) != 0u)) {
#pragma unroll 1
        for (int tl = 0; tl < kDmTiles; ++tl) {
          const int rg = 16 * tl + g;
          float a[4] = {0.f, 0.f, 0.f, 0.f};
          dm_tile<false>(st + dm_row_off(rg, I) + kb0 * 16 + 4 * t, st + dm_row_off(rg + 8, I) + kb0 * 16 + 4 * t,
                         hb, lb, lds32(scp + (size_t)rg * nbI), lds32(scp + (size_t)(rg + 8) * nbI), a);
#pragma unroll
          for (int i = 0; i < 4; ++i) acc[tl][i] = a[i];
        }
      }
      const int slot = pc & 1;
      if (pc >= 2 && !mbar_wait_for(&rs.red_empty[slot], ((pc >> 1) - 1) & 1, p.wait_limit)) {
        set_status(p.ws.hdr, MOE_ERR_TIMEOUT);
        rs.abort_flag = 1;
        dead = true;
        break;
      }
#pragma unroll
      for (int tl = 0; tl < kDmTiles; ++tl) {
        red[slot][warp][tl][g][t] = make_float2(acc[tl][0] * cs[0], acc[tl][1] * cs[1]);
        red[slot][warp][tl][g + 8][t] = make_float2(acc[tl][2] * cs[0], acc[tl][3] * cs[1]);
      }
      if (warp == 0 && lane == 0) {
        DmRedMeta m;
        m.r0 = rt * kDmRows;
        m.b0 = b0;
        m.n = n;
        m.pass = pass;
        rmeta[slot] = m;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&rs.red_full[slot]);
      ++pc;
    }
    if (dead) break;
    __syncwarp();
    if (lane == 0) mbar_arrive(&rs.empty[s]);
  }
  // Tell both reducers there is no more work.
  for (int e = 0; e < 2; ++e, ++pc) {
    const int slot = pc & 1;
    // After an abort the reducer leaves on its own (its wait gives up).
    if (*(volatile int*)&rs.abort_flag) return;
    if (pc >= 2) mbar_wait(&rs.red_empty[slot], ((pc >> 1) - 1) & 1);
    if (warp == 0 && lane == 0) rmeta[slot].r0 = -1;
    __syncwarp();
    if (lane == 0) mbar_arrive(&rs.red_full[slot]);
  }
}

template <int NT>
static bool tma_path_ok(const ExpertParams& p) {
  const int R = kGuRowsNT / NT;
  const int nbH = p.H / 32, nbI = p.I / 32;
  return p.T * p.k <= kMaxPairs && plan_smem_bytes(p.E, p.T * p.k, 4) <= 48 * 1024 && (R * nbH) % 16 == 0 &&
         nbI % 4 == 0 && nbI <= 48 && nbH <= 256 && p.H % kDnRows == 0 && (kDnRows * nbI) % 16 == 0 &&
         p.k <= kMaxK && p.E <= 4096;
}

template <int NT>
static cudaError_t launch_decode_down(const ExpertParams& p, cudaStream_t s, size_t smem_max);

// K-blocks per consumer warp of the tensor-core gate/up kernel, in quads of
// 4 blocks (0: the kernel does not apply to this shape / dtype).
static int gm_quads_per_warp(const ExpertParams& p) {
  if (!p.x_bf16 || p.H % 128 != 0 || p.I % 8 != 0) return 0;
  const int quads = p.H / 128;
  for (int qw = 1; qw <= 4; qw *= 2)
    if (quads % qw == 0 && quads / qw <= kGmMaxWarps) return qw;
  return 0;
}

template <int QW>
static cudaError_t launch_gateup_mma(const ExpertParams& p, cudaStream_t s, size_t smem_max) {
  const int W = p.H / 128 / QW;
  const int threads = (W + kGmProducers + 1) * 32;
  auto kern = k_dec_gateup_mma<QW>;
  // The dynamic ring and plan share the SM's 227 KB with the static arrays.
  cudaFuncAttributes fa;
  cudaError_t err = cudaFuncGetAttributes(&fa, (const void*)kern);
  if (err != cudaSuccess) return err;
  const size_t cap = (size_t)227 * 1024 - fa.sharedSizeBytes;
  smem_max = smem_max < cap ? smem_max : cap;
  const size_t plan = plan_smem_bytes(p.E, p.T * p.k, 4);
  const uint32_t stage = gm_stage_bytes(p.H);
  int stages = (int)((smem_max - plan) / stage);
  stages = stages > kMaxStages ? kMaxStages : stages;
  if (stages < 2) return cudaErrorNotSupported;
  size_t front = (size_t)stages * stage;
  if (p.fused_route) {
    const size_t scratch = route_small_scratch_bytes(p.E, threads / 32, p.T);
    if (scratch > front) front = scratch;
  }
  const size_t smem = front + plan;
  if (smem > smem_max) return cudaErrorNotSupported;
  if (!p.fused_route && (err = launch_x_to_f16(p, s)) != cudaSuccess) return err;
  if ((err = ensure_smem_attr((const void*)kern, smem)) != cudaSuccess) return err;
  prof_before(MOE_STAGE_GATEUP, s);
  err = launch_pdl(kern, dim3(device_sm_count()), dim3(threads), smem, s, p, stages, stage);
  prof_after(MOE_STAGE_GATEUP, s);
  return err;
}

// Tensor-core down (after the tensor-core gate/up, batches above 64 tokens):
// I % 128 == 0, at most kDmMaxWarps consumer warps, H % 64 == 0.
static bool dm_ok(const ExpertParams& p) {
  const int nbI = p.I / 32;
  return p.I % 128 == 0 && nbI / 4 >= 1 && nbI / 4 <= kDmMaxWarps && p.H % kDmRows == 0;
}

static cudaError_t launch_down_mma(const ExpertParams& p, cudaStream_t s, size_t smem_max) {
  const int W = p.I / 128;
  const int threads = (W + 3) * 32;
  auto kern = k_dec_down_mma;
  cudaFuncAttributes fa;
  cudaError_t err = cudaFuncGetAttributes(&fa, (const void*)kern);
  if (err != cudaSuccess) return err;
  const size_t cap = (size_t)227 * 1024 - fa.sharedSizeBytes;
  smem_max = smem_max < cap ? smem_max : cap;
  const size_t plan = plan_smem_bytes(p.E, p.T * p.k, 2);
  const uint32_t stage = dm_stage_bytes(p.I);
  int stages = (int)((smem_max - plan) / stage);
  stages = stages > kMaxStages ? kMaxStages : stages;
  if (stages < 2) return cudaErrorNotSupported;
  const size_t smem = (size_t)stages * stage + plan;
  if ((err = ensure_smem_attr((const void*)kern, smem)) != cudaSuccess) return err;
  prof_before(MOE_STAGE_DOWN, s);
  err = launch_pdl(kern, dim3(device_sm_count()), dim3(threads), smem, s, p, stages, stage);
  prof_after(MOE_STAGE_DOWN, s);
  if (err != cudaSuccess) return err;
  return launch_decode_combine(p, s);
}

template <int NT>
static cudaError_t launch_decode_tma(const ExpertParams& p, cudaStream_t s) {
  constexpr int R = kGuRowsNT / NT;
  const int nsm = device_sm_count();
  cudaError_t err;
  const size_t smem_max = 200 * 1024;
  // gate/up (+ routing prologue)
  const int qw = gm_quads_per_warp(p);
  if (qw) {
    err = qw == 1 ? launch_gateup_mma<1>(p, s, smem_max)
                  : (qw == 2 ? launch_gateup_mma<2>(p, s, smem_max) : launch_gateup_mma<4>(p, s, smem_max));
    if (err != cudaSuccess) return err;
    if (p.T > kDecodeMaxT && dm_ok(p)) return launch_down_mma(p, s, (size_t)227 * 1024);
    return launch_decode_down<NT>(p, s, smem_max);
  }
  const int nbH = p.H / 32;
  const int ncw = (nbH + 31) / 32;
  const int gu_threads = kGuGroups * ncw * 32 + 64;
  const size_t gu_plan = plan_smem_bytes(p.E, p.T * p.k, 4);
  const uint32_t gu_stage = (uint32_t)(2 * R * (p.H / 2) + 2 * R * nbH);
  int gu_stages = (int)((smem_max - gu_plan) / gu_stage);
  gu_stages = gu_stages > kMaxStages ? kMaxStages : gu_stages;
  if (gu_stages < 2) return cudaErrorNotSupported;
  size_t gu_front = (size_t)gu_stages * gu_stage;
  if (p.fused_route) {
    const size_t scratch = route_small_scratch_bytes(p.E, gu_threads / 32, p.T);
    if (scratch > gu_front) gu_front = scratch;
  }
  const size_t gu_smem = gu_front + gu_plan;
  if (gu_smem > smem_max) return cudaErrorNotSupported;
  auto gu = p.x_bf16 ? k_dec_gateup_tma<NT, true> : k_dec_gateup_tma<NT, false>;
  if ((err = ensure_smem_attr((const void*)gu, gu_smem)) != cudaSuccess) return err;
  prof_before(MOE_STAGE_GATEUP, s);
  err = launch_pdl(gu, dim3(nsm), dim3(gu_threads), gu_smem, s, p, gu_stages, gu_stage);
  prof_after(MOE_STAGE_GATEUP, s);
  if (err != cudaSuccess) return err;
  return launch_decode_down<NT>(p, s, smem_max);
}

// down (+ combine)
template <int NT>
static cudaError_t launch_decode_down(const ExpertParams& p, cudaStream_t s, size_t smem_max) {
  cudaError_t err;
  const int nsm = device_sm_count();
  const int nbI = p.I / 32;
  const size_t dn_plan = plan_smem_bytes(p.E, p.T * p.k, 2);
  const uint32_t dn_stage = (uint32_t)(kDnRows * (p.I / 2) + kDnRows * nbI + NT * p.I * 4);
  // Two stages: the producer claims an item from the queue per free stage,
  // so a deeper ring leaves claimed items waiting in some CTAs at the end
  // while others run out of work (measured: three stages were 1-3 % slower).
  constexpr int kDnStages = 2;
  if ((size_t)kDnStages * dn_stage + dn_plan > smem_max) return cudaErrorNotSupported;
  const int dn_stages = kDnStages;
  const size_t dn_smem = (size_t)dn_stages * dn_stage + dn_plan;
  auto dn = k_dec_down_tma<NT>;
  if ((err = ensure_smem_attr((const void*)dn, dn_smem)) != cudaSuccess) return err;
  prof_before(MOE_STAGE_DOWN, s);
  err = launch_pdl(dn, dim3(nsm), dim3(nbI * kDnG + 64), dn_smem, s, p, dn_stages, dn_stage);
  prof_after(MOE_STAGE_DOWN, s);
  if (err != cudaSuccess || p.T <= kDecodeMaxT) return err;
  return launch_decode_combine(p, s);
}

template <int NT>
static cudaError_t launch_decode_nt(const ExpertParams& p, cudaStream_t s) {
  if (tma_path_ok<NT>(p)) return launch_decode_tma<NT>(p, s);
  return launch_decode_ldg<NT>(p, s);
}

// The whole decode layer: router scores, then (when the staged kernels apply)
// gate/up with the routing fused into its prologue and down + combine;
// otherwise the standalone routing kernels and the register-streaming path.
// With mx: the router scores, then the persistent block-scaled kernel.
cudaError_t launch_decode_forward(const RouteParams& rp, const BucketParams& bp, ExpertParams p, cudaStream_t s,
                                  bool mx) {
  const bool small_route = route_decode_supported(rp.T, rp.H, rp.E, rp.k);
  const bool staged = p.T == 1 ? tma_path_ok<1>(p) : tma_path_ok<2>(p);
  if (mx) {
    if (!small_route || !dmx_supported(p)) return cudaErrorNotSupported;
    // Router scores (and the E4M3 activation terms), then the persistent
    // block-scaled kernel routes and runs every routed expert.
    RouteParams r2 = rp;
    r2.dmx_I = p.I;
    cudaError_t err = launch_router_gemv(r2, s);
    if (err != cudaSuccess) return err;
    p.fused_route = 1;
    p.rp = r2;
    return launch_dec_mx(p, s);
  }
  if (small_route && staged) {
    cudaError_t err = launch_router_gemv(rp, s);
    if (err != cudaSuccess) return err;
    p.fused_route = 1;
    p.rp = rp;
    return p.T == 1 ? launch_decode_tma<1>(p, s) : launch_decode_tma<2>(p, s);
  }
  cudaError_t err = small_route ? launch_route_decode(rp, s) : launch_route_prefill(rp, bp, s);
  if (err != cudaSuccess) return err;
  p.fused_route = 0;
  return launch_decode_experts(p, s);
}

bool decode_batch_supported(int T, int H, int E, int I, int k) {
  ExpertParams p;
  memset(&p, 0, sizeof p);
  p.T = T; p.H = H; p.E = E; p.I = I; p.k = k;
  p.x_bf16 = 1;
  return T >= 1 && T <= kDecodeBatchMaxT && H <= 8192 && tma_path_ok<2>(p) && gm_quads_per_warp(p) != 0;
}

// NT = routed pairs of one expert processed per weight pass.  The choice
// changes only how many times a shared expert's weights are read, never the
// arithmetic of a pair.
cudaError_t launch_decode_experts(const ExpertParams& p, cudaStream_t s) {
  if (p.T == 1) return launch_decode_nt<1>(p, s);
  return launch_decode_nt<2>(p, s);
}

}  // namespace moe
