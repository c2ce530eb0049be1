// route_small.cuh — top-k with renormalised weights and the bucket plan for a
// small batch (T <= 64 tokens, E <= 4096), computed by one CTA from the router
// scores in the workspace.  Used as the prologue of the decode gate/up kernel
// (every CTA computes the route for itself; CTA 0 publishes it) and by the
// standalone routing kernel.
#pragma once

#include "common.cuh"

namespace moe {

constexpr uint32_t kTaken = 0xFFFFFFFFu;  // hi bits of an already selected expert (prefill top-k)

__device__ __forceinline__ uint32_t ord32(float f) {
  const uint32_t b = __float_as_uint(f + 0.0f);  // -0 -> +0
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);  // monotone in f
}

// Orderable key of a double-float score (hi, lo): value order; a taken entry
// (hi bits kTaken) sorts below every real score.  (Prefill top-k.)
__device__ __forceinline__ unsigned long long score_key(float2 v) {
  if (__float_as_uint(v.x) == kTaken) return 0ull;
  return ((unsigned long long)ord32(v.x) << 32) | ord32(v.y);
}

__device__ __forceinline__ void lane_best(const float2* row, int E, int lane, unsigned long long& best, int& best_e) {
  best = 0ull;
  best_e = 0x7FFFFFFF;
  for (int e = lane; e < E; e += 32) {
    const unsigned long long kk = score_key(row[e]);
    if (kk > best) { best = kk; best_e = e; }
  }
}

// Top-k of one token by one warp over its double-float scores in shared
// memory `row` (destroyed): larger score first, lower expert index on equal
// scores.  Lane j < k returns slot j's expert and score.  Each lane keeps the
// best of its own entries; a round is one warp argmax over the lanes' bests,
// after which only the winning lane rescans its entries.  (Prefill top-k.)
__device__ __forceinline__ void warp_topk(float2* row, int E, int k, int& my_e, float2& my_s) {
  const int lane = threadIdx.x & 31;
  my_e = -1;
  my_s = make_float2(0.f, 0.f);
  unsigned long long lb;
  int le;
  lane_best(row, E, lane, lb, le);
  for (int j = 0; j < k; ++j) {
    unsigned long long best = lb;
    int best_e = le;
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) {
      const unsigned long long ok = __shfl_xor_sync(0xFFFFFFFFu, best, m);
      const int oe = __shfl_xor_sync(0xFFFFFFFFu, best_e, m);
      if (ok > best || (ok == best && oe < best_e)) { best = ok; best_e = oe; }
    }
    if (lane == j) {
      my_e = best_e;
      my_s = row[best_e];
    }
    __syncwarp();
    if ((best_e & 31) == lane) {  // the winner's lane takes it out and rescans
      row[best_e].x = __uint_as_float(kTaken);
      lane_best(row, E, lane, lb, le);
    }
    __syncwarp();
  }
}

// Top-k of one token by one warp over a list of n scored experts (sc[c] the
// double-float score of expert id[c]; sc is destroyed): larger score first,
// lower expert index on equal scores; lane j < k returns slot j's expert and
// score.  Entry c belongs to lane c % 32.
__device__ __forceinline__ void warp_topk_list(float2* sc, const int* id, int n, int k, int& my_e, float2& my_s) {
  const int lane = threadIdx.x & 31;
  my_e = -1;
  my_s = make_float2(0.f, 0.f);
  auto scan = [&](unsigned long long& best, int& best_e, int& best_c) {
    best = 0ull;
    best_e = 0x7FFFFFFF;
    best_c = -1;
    for (int c = lane; c < n; c += 32) {
      const unsigned long long kk = score_key(sc[c]);
      const int e = id[c];
      if (kk > best || (kk == best && kk != 0ull && e < best_e)) {
        best = kk;
        best_e = e;
        best_c = c;
      }
    }
  };
  unsigned long long lb;
  int le, lc;
  scan(lb, le, lc);
  for (int j = 0; j < k; ++j) {
    unsigned long long best = lb;
    int best_e = le, best_c = lc;
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) {
      const unsigned long long ok = __shfl_xor_sync(0xFFFFFFFFu, best, m);
      const int oe = __shfl_xor_sync(0xFFFFFFFFu, best_e, m);
      const int oc = __shfl_xor_sync(0xFFFFFFFFu, best_c, m);
      if (ok > best || (ok == best && oe < best_e)) {
        best = ok;
        best_e = oe;
        best_c = oc;
      }
    }
    if (lane == j && best_c >= 0) {
      my_e = best_e;
      my_s = sc[best_c];
    }
    __syncwarp();
    if (best_c >= 0 && (best_c & 31) == lane) {  // the winner's lane takes it out and rescans
      sc[best_c].x = __uint_as_float(kTaken);
      scan(lb, le, lc);
    }
    __syncwarp();
  }
}

// ---- small-batch top-k on packed keys (E <= 4096) ----
// key = ord(hi) << 32 | (ord(lo) with its low 12 bits replaced by 4095 - e):
// value order first (hi, then the top 20 bits of lo, far below any score
// resolution that matters), then the lower expert index; 0 = taken.
__device__ __forceinline__ unsigned long long packed_key(float2 v, int e) {
  return ((unsigned long long)ord32(v.x) << 32) | (ord32(v.y) & 0xFFFFF000u) | (uint32_t)(4095 - e);
}

__device__ __forceinline__ unsigned long long lane_best_key(const unsigned long long* keys, int E, int lane) {
  unsigned long long best = 0ull;
  for (int e0 = lane; e0 < E; e0 += 32 * 8) {
    unsigned long long v[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) v[q] = e0 + 32 * q < E ? keys[e0 + 32 * q] : 0ull;
#pragma unroll
    for (int q = 0; q < 8; ++q) best = v[q] > best ? v[q] : best;
  }
  return best;
}

// Warp maximum of a 64-bit key: hardware reductions over the high word, then
// over the low word of the lanes holding that high word.
__device__ __forceinline__ unsigned long long warp_max_key(unsigned long long v) {
  const uint32_t hi = (uint32_t)(v >> 32);
  const uint32_t mhi = __reduce_max_sync(0xFFFFFFFFu, hi);
  const uint32_t mlo = __reduce_max_sync(0xFFFFFFFFu, hi == mhi ? (uint32_t)v : 0u);
  return ((unsigned long long)mhi << 32) | mlo;
}

// Top-k by one warp over packed keys in shared memory (destroyed): lane j < k
// returns slot j's expert.  k rounds of warp argmax; after each round only
// the winning lane rescans its entries.
__device__ __forceinline__ int warp_topk_keys_rounds(unsigned long long* keys, int E, int k) {
  const int lane = threadIdx.x & 31;
  int my_e = -1;
  unsigned long long lb = lane_best_key(keys, E, lane);
  for (int j = 0; j < k; ++j) {
    const unsigned long long best = warp_max_key(lb);
    const int e = 4095 - (int)(best & 0xFFFull);
    if (lane == j) my_e = e;
    if ((e & 31) == lane) {  // the winner's lane takes it out and rescans
      keys[e] = 0ull;
      lb = lane_best_key(keys, E, lane);
    }
    __syncwarp();
  }
  return my_e;
}

// Ascending bitonic sort of 64 keys held as element lane (x0) and element
// lane + 32 (x1).  Element i pairs with i ^ j; it keeps the smaller key when
// it is the lower of the two and its block of size k sorts upward.
__device__ __forceinline__ void warp_sort64(unsigned long long& x0, unsigned long long& x1) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int k = 2; k <= 64; k <<= 1) {
#pragma unroll
    for (int j = k >> 1; j >= 1; j >>= 1) {
      if (j == 32) {
        const unsigned long long lo = x0 < x1 ? x0 : x1, hi = x0 < x1 ? x1 : x0;
        x0 = lo;
        x1 = hi;
      } else {
        const unsigned long long p0 = __shfl_xor_sync(0xFFFFFFFFu, x0, j);
        const unsigned long long p1 = __shfl_xor_sync(0xFFFFFFFFu, x1, j);
        const bool lower = (lane & j) == 0;
        const bool min0 = lower == ((lane & k) == 0);
        const bool min1 = lower == (((lane + 32) & k) == 0);
        x0 = min0 ? (p0 < x0 ? p0 : x0) : (p0 < x0 ? x0 : p0);
        x1 = min1 ? (p1 < x1 ? p1 : x1) : (p1 < x1 ? x1 : p1);
      }
    }
  }
}

// Top-k (k <= 32) by one warp over packed keys in shared memory; lane j < k
// returns slot j's expert.  Each lane keeps its three largest keys; the two
// largest of every lane (64 keys) are sorted, giving a candidate k-th key K.
// A key left out is at most its lane's third largest, so when no lane's third
// largest exceeds K the sorted candidates hold the whole top k (the usual
// case).  Otherwise the k-round selection runs (it overwrites `keys`).  Keys
// are unique (the expert index is part of the key): the result is the same
// either way.
__device__ __forceinline__ int warp_topk_keys(unsigned long long* keys, int E, int k) {
  const int lane = threadIdx.x & 31;
  unsigned long long b1 = 0ull, b2 = 0ull, b3 = 0ull;
  for (int e0 = lane; e0 < E; e0 += 32 * 8) {
    unsigned long long v[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) v[q] = e0 + 32 * q < E ? keys[e0 + 32 * q] : 0ull;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const unsigned long long x = v[q];
      const bool g1 = x > b1, g2 = x > b2, g3 = x > b3;
      b3 = g2 ? b2 : (g3 ? x : b3);
      b2 = g1 ? b1 : (g2 ? x : b2);
      b1 = g1 ? x : b1;
    }
  }
  unsigned long long x0 = b1, x1 = b2;
  warp_sort64(x0, x1);
  // Slot j is the (j+1)-th largest: element 63 - j, i.e. x1 of lane 31 - j.
  const unsigned long long best = __shfl_sync(0xFFFFFFFFu, x1, 31 - lane);
  const unsigned long long kth = __shfl_sync(0xFFFFFFFFu, x1, 32 - k);
  if (__any_sync(0xFFFFFFFFu, b3 > kth)) return warp_topk_keys_rounds(keys, E, k);
  return lane < k ? 4095 - (int)(best & 0xFFFull) : -1;
}

// Softmax of the selected scores held by lanes 0..k-1 (slot order): lane j
// gets exp(s_j - s_0) / sum_i exp(s_i - s_0), the differences taken from the
// double-float scores.
__device__ __forceinline__ float warp_route_weight(float2 my_s, int k) {
  const int lane = threadIdx.x & 31;
  const float h0 = __shfl_sync(0xFFFFFFFFu, my_s.x, 0);
  const float l0 = __shfl_sync(0xFFFFFFFFu, my_s.y, 0);
  const float d = (my_s.x - h0) + (my_s.y - l0);
  const float ex = lane < k ? expf(d) : 0.0f;
  float z = ex;
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) z += __shfl_xor_sync(0xFFFFFFFFu, z, m);
  return ex / z;
}

// Bucket plan of a small batch in shared memory.
struct SmallPlan {
  int U;        // active experts
  int* ue;      // [umax] expert id of active expert u (ascending)
  int* ub0;     // [umax] bucket offset
  int* un;      // [umax] bucket size
  int* pairs;   // [T*k]  routed pairs t*k+j grouped by expert, ascending inside
  float* wts = nullptr;  // [T*k] the pairs' weights (optional; filled by every CTA)
};

constexpr int kRouteWarps = 8;  // warps that route tokens (one token per warp at a time)

// Scratch bytes of route_small for T tokens: token masks, counts, offsets,
// the selected ids, and one packed-key row per routing warp.
__host__ __device__ inline size_t route_small_scratch_bytes(int E, int nwarps, int T) {
  int rw = nwarps < T ? nwarps : T;
  rw = rw < kRouteWarps ? rw : kRouteWarps;
  return (size_t)E * 8 + (size_t)E * 4 + (size_t)(E + 1) * 4 + (size_t)kDecodeMaxT * kMaxK * 4 + 32 +
         (size_t)rw * E * 8;
}

// Route T <= 64 tokens (E <= 4096).  `scratch` (route_small_scratch_bytes,
// 16-byte aligned) may alias memory the caller reuses afterwards; `plan`
// arrays must not alias it.  With `publish`, ids/w/offsets/sorted/act_e/
// n_active are also written to global memory (workspace and the caller's
// copies).  All threads of the CTA call it; it ends with __syncthreads().
static __device__ void route_small(const RouteParams& p, char* scratch, SmallPlan& plan, bool publish) {
  const int T = p.T, E = p.E, k = p.k;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nwarps = blockDim.x >> 5;
  const int rwarps = nwarps < kRouteWarps ? nwarps : kRouteWarps;
  unsigned long long* tmask = reinterpret_cast<unsigned long long*>(scratch);  // [E] token bits
  int* cnt = reinterpret_cast<int*>(tmask + E);                                // [E]
  int* off = cnt + E;                                                           // [E+1]
  int* s_ids = off + E + 1;                                                     // [T*k]
  s_ids = reinterpret_cast<int*>((reinterpret_cast<uintptr_t>(s_ids) + 15) & ~(uintptr_t)15);
  // One key row per token routed at once (at most min(rwarps, T), as
  // route_small_scratch_bytes counts them).
  unsigned long long* keyrows = reinterpret_cast<unsigned long long*>(s_ids + kDecodeMaxT * kMaxK);
  __shared__ int s_wtot[32][2];
  __shared__ int s_nact;
  for (int e = threadIdx.x; e < E; e += blockDim.x) tmask[e] = 0ull;
  __syncthreads();
  for (int t0 = 0; t0 < T; t0 += rwarps) {
    const int nt = T - t0 < rwarps ? T - t0 : rwarps;
    // Scores -> packed keys for tokens t0 .. t0+nt-1, by all threads; eight
    // loads in flight per thread before their stores.
    const int n = nt * E;
    const float2* lg = p.ws.logits + (size_t)t0 * E;
    for (int i0 = threadIdx.x; i0 < n; i0 += 8 * blockDim.x) {
      float2 v[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const int i = i0 + q * (int)blockDim.x;
        v[q] = i < n ? __ldcg(&lg[i]) : make_float2(0.f, 0.f);
      }
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const int i = i0 + q * (int)blockDim.x;
        if (i < n) keyrows[i] = packed_key(v[q], i % E);
      }
    }
    __syncthreads();
    if (warp < nt) {
      const int t = t0 + warp;
      const int my_e = warp_topk_keys(keyrows + (size_t)warp * E, E, k);
      float2 my_s = make_float2(0.f, 0.f);
      if (lane < k) my_s = __ldcg(&p.ws.logits[(size_t)t * E + my_e]);
      const float wt = warp_route_weight(my_s, k);
      if (lane < k) {
        if (publish) {
          p.ids[t * k + lane] = my_e;
          p.w[t * k + lane] = wt;
        }
        s_ids[t * k + lane] = my_e;
        if (plan.wts) plan.wts[t * k + lane] = wt;
        atomicOr(&tmask[my_e], 1ull << t);
      }
    }
    __syncthreads();
  }
  // Counts, then a CTA-wide exclusive scan of (count, active flag) over the
  // experts; each thread owns a run of consecutive experts.
  const int per = (E + blockDim.x - 1) / blockDim.x;
  const int e_lo = threadIdx.x * per, e_hi = e_lo + per < E ? e_lo + per : E;
  int csum = 0, asum = 0;
  for (int e = e_lo; e < e_hi; ++e) {
    const int c = __popcll(tmask[e]);
    cnt[e] = c;
    csum += c;
    asum += c > 0 ? 1 : 0;
  }
  int ci = csum, ai = asum;
#pragma unroll
  for (int m = 1; m < 32; m <<= 1) {
    const int oc = __shfl_up_sync(0xFFFFFFFFu, ci, m);
    const int oa = __shfl_up_sync(0xFFFFFFFFu, ai, m);
    if (lane >= m) { ci += oc; ai += oa; }
  }
  if (lane == 31) { s_wtot[warp][0] = ci; s_wtot[warp][1] = ai; }
  __syncthreads();
  int cpre = 0, apre = 0;
  for (int w = 0; w < warp; ++w) { cpre += s_wtot[w][0]; apre += s_wtot[w][1]; }
  int crun = cpre + ci - csum, arun = apre + ai - asum;
  for (int e = e_lo; e < e_hi; ++e) {
    const int c = cnt[e];
    off[e] = crun;
    if (c > 0) {
      plan.ue[arun] = e;
      plan.ub0[arun] = crun;
      plan.un[arun] = c;
      ++arun;
    }
    crun += c;
  }
  if (threadIdx.x == blockDim.x - 1) {
    off[E] = crun;
    s_nact = arun;
  }
  __syncthreads();
  plan.U = s_nact;
  // Stable scatter: the rank of token t in expert e's bucket is the number of
  // tokens below t routed to e (a token selects an expert at most once).
  for (int i = threadIdx.x; i < T * k; i += blockDim.x) {
    const int t = i / k;
    const int e = s_ids[i];
    const unsigned long long below = t == 0 ? 0ull : (tmask[e] & ((1ull << t) - 1ull));
    const int pos = off[e] + __popcll(below);
    plan.pairs[pos] = i;
    if (publish) {
      p.ws.sorted[pos] = i;
      if (p.sorted) p.sorted[pos] = i;
    }
  }
  if (publish) {
    for (int e = threadIdx.x; e <= E; e += blockDim.x) {
      p.ws.offsets[e] = off[e];
      if (p.offsets) p.offsets[e] = off[e];
    }
    for (int u = threadIdx.x; u < plan.U; u += blockDim.x) p.ws.act_e[u] = plan.ue[u];
    if (threadIdx.x == 0) p.ws.hdr->n_active = (uint32_t)plan.U;
  }
  __syncthreads();
}

}  // namespace moe
