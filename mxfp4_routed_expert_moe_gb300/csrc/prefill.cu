// prefill.cu — grouped MXFP4 expert GEMMs on tcgen05 tensor cores (bf16
// activations, any T; the automatic path uses it for T > 64).
//
// The expert step is a grouped GEMM over the bucket layout: for an active
// expert e with n_e routed tokens, G = Wg_e X_e^T, U = Wu_e X_e^T and
// Y = Wd_e H_e^T.  Weights form the M side of 128-row tiles, the tokens of
// the bucket the N side (up to 128 per tile); the contraction runs in
// 64-element slices through a shared-memory ring.
//   * Weights are dequantized from MXFP4 to f16 by CUDA-core warps: one exact
//     conversion of two E2M1 codes and one f16x2 multiply by
//     2^(e - 127 + sigma_r) per pair, where the row shift sigma_r puts the
//     row's largest block scale at 6 * 2^13, so every dequantized value is an
//     exact f16.
//   * Activations are f16 with a per-token shift (largest magnitude in
//     [2^14, 2^15)), exact for bf16 inputs.
//   * Products are exact and accumulate in fp32 in Tensor Memory; the
//     epilogue removes both shifts.
// gate/up: the epilogue applies SwiGLU and stores h in fp32, bucket order,
// raising the largest |h| of each h row; a pass then writes each row in f16
// scaled by a power of two that puts its largest magnitude in [2^14, 2^15)
// (no overflow for any finite h; 11 significant bits for every element within
// 2^28 of the row's maximum).
// down: the epilogue removes that shift and adds w[t][j] * y into out with
// fp32 atomics.
// The optional bf16 shared expert runs as extra work items of the same
// kernels (identity token map, weight 1); its rows get the same kind of
// power-of-two shift, computed by a pre-pass.
//
// Prior art on the pages is a CPU / Metal fused dequant+GEMV [deltafin, "The
// techniques that bought the 82x"]; a batch of positions sharing experts
// [Deltafin's custom compiled runtime, "Complete target sequence tape"] is
// what makes the contraction dense enough for tensor cores here.
#include <utility>

#include "async.cuh"
#include "kernels.h"
#include "tcgen05.cuh"

namespace moe {

constexpr int kPfSliceK = 64;            // contraction elements per stage (one 128-byte swizzle row)
constexpr int kPfTileBytes = 128 * 128;  // one 128-row x 64-element f16 tile
// Weight dequant: two groups of 8 warps; group k converts the slices of parity
// k (2 threads per weight row in each group), so each warp's per-slice chain
// of waits, conversion and signalling overlaps the other group's.
constexpr int kPfDqGroups = 2;
constexpr int kPfDqGroupWarps = 8;
constexpr int kPfDqGroupThreads = kPfDqGroupWarps * 32;
constexpr int kPfDqWarps = kPfDqGroups * kPfDqGroupWarps;  // warps 0-15
constexpr int kPfLdWarps = 4;            // warps 16-19: token rows (cp.async)
constexpr int kPfEpWarps = 4;            // warps 20-23: epilogue (warp % 4 = TMEM lane quarter)
// MMA issue: one thread issues a tcgen05.mma only every ~100 cycles whatever
// its size, so the gate/up kernel issues from two warps, one accumulator each
// (gate, up).  The down kernel has one accumulator and one issuer.
constexpr int kPfMmaWarp = kPfDqWarps + kPfLdWarps + kPfEpWarps;  // warps 24-25: MMA issuers; 24 owns TMEM
constexpr int kPfMmaWarps = 2;
constexpr int kPfThreads = (kPfMmaWarp + kPfMmaWarps) * 32;
constexpr int kPfMaxStages = 8;
// Rings (per kernel): f16 weight tiles from the dequant warps (A), f16 token
// rows from the loader warps (B), raw MXFP4 bytes of the dequant threads.
constexpr int kPfAStagesGateUp = 3, kPfBStagesGateUp = 5;
constexpr int kPfAStagesDown = 3, kPfBStagesDown = 6;
constexpr int kPfL2Window = 256;         // bytes of each weight row prefetched into L2 at a time
constexpr uint32_t kPfTmemCols = 512;    // 2 accumulator buffers x (gate 128 + up 128) columns
constexpr int kPfSigRing = 4;            // items whose row shifts are published ahead
// Raw MXFP4 ring of each dequant group: per slice and thread 16 bytes of
// codes and the 4-byte scale word per matrix, cp.async'd this many of the
// group's slices ahead (about 48 KB in flight per SM for either kernel).
constexpr int kPfRawGateUp = 2;
constexpr int kPfRawDown = 6;
template <int NA>
struct PfRaw {
  static constexpr int kQ = NA * kPfDqGroupThreads * 16;              // codes
  static constexpr int kStage = kQ + NA * kPfDqGroupThreads * 4;      // + scale words
};
static_assert(kPfEpWarps == 4 && (kPfDqWarps + kPfLdWarps) % 4 == 0, "epilogue warps must cover lane quarters 0-3");

// ------------------------------------------------------------ pre-passes --
// xh[t][h] = f16(x[t][h] * 2^sigma_t), xscale[t] = 2^-sigma_t (one CTA per token).
// Also clears the h-row maxima of token t's routed pairs and of its
// shared-expert row, which the gate/up epilogue raises with atomicMax.
__global__ void __launch_bounds__(256) k_x_to_f16(ExpertParams p) {
  const int t = blockIdx.x;
  x_row_to_f16(reinterpret_cast<const uint16_t*>(p.x) + (size_t)t * p.H, p.H, p.ws.xh + (size_t)t * p.H,
               &p.ws.xscale[t]);
  if ((int)threadIdx.x < p.k) p.ws.hmax[(size_t)t * p.k + threadIdx.x] = 0u;
  if (threadIdx.x == 0) p.ws.hmax[(size_t)p.T * p.k + t] = 0u;
}

// f16 copy of the fp32 h rows [row0, row1) for the down GEMM: row r is scaled
// by 2^tau_r, tau_r = 14 - floor(log2 max|h_r|), which puts the row's largest
// magnitude in [2^14, 2^15): no overflow, and every element within 2^28 of the
// maximum keeps the full 11-bit f16 significand.  hscale[r] = 2^-tau_r is
// removed in the down epilogue.  A row whose maximum is zero, infinite or NaN
// keeps tau = 0 (NaN and infinity propagate).  One warp per row; I % 32 == 0.
__global__ void __launch_bounds__(256) k_h_to_f16(ExpertParams p, int row0, int row1) {
  const int row = row0 + blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= row1) return;
  const uint32_t m = p.ws.hmax[row];
  const int e = (int)((m >> 23) & 0xFFu);
  int tau = (m == 0u || e == 0xFF) ? 0 : 14 - (e - 127);
  tau = tau > 100 ? 100 : (tau < -100 ? -100 : tau);
  const float up = __int_as_float((tau + 127) << 23);
  if (lane == 0) p.ws.hscale[row] = __int_as_float((127 - tau) << 23);
  const float* src = reinterpret_cast<const float*>(p.ws.h) + (size_t)row * p.I;
  uint16_t* dst = p.ws.h16 + (size_t)row * p.I;
  for (int c = lane * 4; c < p.I; c += 128) {
    const float4 v = *reinterpret_cast<const float4*>(src + c);
    const __half2 a = __floats2half2_rn(v.x * up, v.y * up);
    const __half2 b = __floats2half2_rn(v.z * up, v.w * up);
    *reinterpret_cast<uint2*>(dst + c) =
        make_uint2(*reinterpret_cast<const uint32_t*>(&a), *reinterpret_cast<const uint32_t*>(&b));
  }
}

cudaError_t launch_x_to_f16(const ExpertParams& p, cudaStream_t s) {
  k_x_to_f16<<<p.T, 256, 0, s>>>(p);
  return cudaGetLastError();
}

// Row shifts of the bf16 shared expert: shsig[r] = 14 - floor(log2 max|row|)
// for the I gate rows, I up rows and H down rows (0 for an all-zero row).
// One warp per row.
__global__ void __launch_bounds__(256) k_shared_sigma(ExpertParams p) {
  const int row = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  const int I = p.I, H = p.H;
  if (row >= 2 * I + H) return;
  const uint16_t* src;
  int len;
  if (row < I) { src = p.sh_gate + (size_t)row * H; len = H; }
  else if (row < 2 * I) { src = p.sh_up + (size_t)(row - I) * H; len = H; }
  else { src = p.sh_down + (size_t)(row - 2 * I) * I; len = I; }
  uint32_t emax = 0;  // largest exponent field of the row's bf16 values
  for (int c = lane * 8; c < len; c += 256) {
    const uint4 v = *reinterpret_cast<const uint4*>(src + c);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      emax = max(emax, (w[j] >> 7) & 0xFFu);
      emax = max(emax, (w[j] >> 23) & 0xFFu);
    }
  }
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) emax = max(emax, __shfl_xor_sync(0xFFFFFFFFu, emax, o));
  if (lane == 0) {
    int sig = emax == 0 ? 0 : 14 - ((int)emax - 127);
    if (emax == 255) sig = 0;  // inf / NaN in the row: leave it unscaled, it propagates
    p.ws.shsig[row] = sig > 100 ? 100 : (sig < -100 ? -100 : sig);
  }
}

// ------------------------------------------------------------ work items --
// Items are (expert, 128-row weight tile, 128-token tile).  Routed items come
// first, active experts in ascending order, row tiles outer; then the shared
// expert's items when there is one.
struct PfItem {
  int shared;  // 1: the bf16 shared expert
  int e;       // routed expert
  int m0;      // first weight row
  int p0;      // routed: first bucket position; shared: first token
  int cnt;     // tokens in the tile (1..128)
  int hpos0;   // row of the tile's first token in h ([T*k + T][I])
};

__device__ __forceinline__ PfItem pf_item(int item, const ExpertParams& p, const int32_t* pref, int U,
                                          int n_routed) {
  PfItem it;
  if (item >= n_routed) {
    const int local = item - n_routed;
    const int nts = (p.T + kPfNTile - 1) / kPfNTile;
    const int m = local / nts, nt = local - m * nts;
    it.shared = 1;
    it.e = 0;
    it.m0 = m * kPfMTile;
    it.p0 = nt * kPfNTile;
    it.cnt = min(kPfNTile, p.T - it.p0);
    it.hpos0 = p.T * p.k + it.p0;
    return it;
  }
  int lo = 0, hi = U - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(&pref[mid]) <= item) lo = mid; else hi = mid - 1;
  }
  const int local = item - __ldg(&pref[lo]);
  const int e = __ldg(&p.ws.act_e[lo]);
  const int b0 = __ldg(&p.offsets[e]);
  const int n = __ldg(&p.offsets[e + 1]) - b0;
  const int ntiles = (n + kPfNTile - 1) / kPfNTile;
  const int m = local / ntiles, nt = local - m * ntiles;
  it.shared = 0;
  it.e = e;
  it.m0 = m * kPfMTile;
  it.p0 = b0 + nt * kPfNTile;
  it.cnt = min(kPfNTile, n - nt * kPfNTile);
  it.hpos0 = it.p0;
  return it;
}

// ----------------------------------------------------------- dequant --
// f16 bits of 2^d (0 below the subnormal range; d <= 15 by construction).
__device__ __forceinline__ uint32_t f16_pow2(int d) {
  if (d >= -14) return (uint32_t)((d > 15 ? 30 : d + 15) << 10);
  if (d >= -24) return 1u << (d + 24);
  return 0u;
}

// Shift of an MXFP4 weight row from its E8M0 scales: sigma = 140 - max scale
// (NaN scales ignored), so the largest block reaches 6 * 2^13 < 65504.  The
// row's `nwords` 4-byte words of scales are split over `parts` cooperating
// threads (`part` = this thread's index); the caller combines the parts with
// a max.
__device__ __forceinline__ int row_smax_part(const uint8_t* srow, int nwords, int part, int parts) {
  int smax = -1;
  for (int i = part; i < nwords; i += parts) {
    const uint32_t w = __ldg(reinterpret_cast<const uint32_t*>(srow) + i);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int s = (int)((w >> (8 * j)) & 0xFF);
      if (s != 255 && s > smax) smax = s;
    }
  }
  return smax;
}
__device__ __forceinline__ int sigma_from_smax(int smax) { return smax < 0 ? 0 : 140 - smax; }

// One MX block (32 elements: 16 bytes of codes, one scale byte) of weight row
// r -> four 16-byte f16 chunks c0..c0+3 of the row in a SW128 tile, scaled by
// 2^sigma.
__device__ __forceinline__ void dq_mx_block(uint8_t* tile, uint32_t r, uint32_t c0, uint4 q, uint32_t s, int sigma) {
  const uint32_t mul16 = s == 255u ? 0x7E00u : f16_pow2((int)s - 127 + sigma);
  const uint32_t mul2 = mul16 | (mul16 << 16);
  const uint32_t words[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
  for (int wd = 0; wd < 4; ++wd) {
    uint32_t o[4];
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const uint32_t w2 = e2m1x2_f16x2(words[wd], b);
      asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(o[b]) : "r"(w2), "r"(mul2));
    }
    *reinterpret_cast<uint4*>(tile + sw128_offset(r, c0 + wd)) = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

// 32 bf16 weights (four 16-byte loads) -> four f16 chunks, scaled by `scale`
// (a power of two).
__device__ __forceinline__ void dq_bf16_block(uint8_t* tile, uint32_t r, uint32_t c0, const uint4 (&v)[4],
                                              float scale) {
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t w[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const __half2 h2 =
          __floats2half2_rn(__uint_as_float(w[i] << 16) * scale, __uint_as_float(w[i] & 0xFFFF0000u) * scale);
      o[i] = *reinterpret_cast<const uint32_t*>(&h2);
    }
    *reinterpret_cast<uint4*>(tile + sw128_offset(r, c0 + j)) = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

// -------------------------------------------------------- CTA control --
struct PfShared {
  uint64_t a_full[kPfMaxStages];   // weight tile stage filled: the 8 warps of one dequant group
  uint64_t a_empty[kPfMaxStages];  // ... consumed: tcgen05.commit
  uint64_t b_full[kPfMaxStages];   // token tile stage filled: 128 loader threads (cp.async arrivals)
  uint64_t b_empty[kPfMaxStages];  // ... consumed: tcgen05.commit
  uint64_t accf[2];              // accumulator buffer ready: tcgen05.commit of each issuer
  uint64_t acce[2];              // accumulator buffer drained: 4 epilogue warps
  uint64_t sig_full[kPfSigRing];  // row shifts of an item published: 4 epilogue warps
  uint64_t sig_empty[kPfSigRing]; // ... and read: 16 dequant + 4 epilogue warps
  uint32_t tmem_base;
  int abort_flag;
  int sig[kPfSigRing][2][kPfMTile];       // row shifts (gate/down, up) of upcoming items
  float col_scale[kPfEpWarps][kPfNTile];  // per epilogue warp: token shift (gate/up) or route weight (down)
  int col_tok[kPfEpWarps][kPfNTile];      // per epilogue warp: token of each column (down)
};

// Bounded wait that also gives up as soon as another role has aborted.  The
// waiting thread sleeps in try_wait (at most kPfSleepNs per call) instead of
// spinning: each SM sub-partition hosts waiting warps of several roles.
constexpr uint32_t kPfSleepNs = 20000;
__device__ __forceinline__ bool pf_wait(PfShared& sh, uint64_t* bar, uint32_t parity, WsHeader* hdr) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  for (;;) {
    if (mbar_try_wait_sleep(bar, parity, kPfSleepNs)) return true;
    if (*(volatile int*)&sh.abort_flag) return false;
    if (clock64() - t0 > kWaitCycles) {
      set_status(hdr, MOE_ERR_TIMEOUT);
      *(volatile int*)&sh.abort_flag = 1;
      return false;
    }
  }
}

// Shared pipeline state of the four roles of one CTA.
struct PfCtx {
  PfShared* sh;
  uint8_t* smem_a;   // weight tile ring (NA tiles per stage), 1024-byte aligned
  uint8_t* smem_b;   // token tile ring, 1024-byte aligned
  uint8_t* raw;      // raw MXFP4 ring of the dequant threads
  int a_stages, b_stages;
  int a_bytes;       // bytes of one weight tile stage
  int n_items;       // routed + shared items
  int n_routed;
  int U;
  const int32_t* pref;
  int K, M, nslices;
  WsHeader* hdr;
};

// All lanes of a warp wait; the warp proceeds only if every lane succeeded.
__device__ __forceinline__ bool pf_warp_wait(const PfCtx& c, uint64_t* bar, uint32_t parity) {
  const bool ok = pf_wait(*c.sh, bar, parity, c.hdr);
  return __all_sync(0xFFFFFFFFu, ok);
}

// Claim the ring stage of global slice gs for writing (wait until its
// previous use was consumed by the tensor core).
__device__ __forceinline__ bool pf_claim(const PfCtx& c, uint64_t* empty, int nstages, int gs) {
  const int st = gs % nstages, use = gs / nstages;
  if (use == 0) return true;
  return pf_warp_wait(c, &empty[st], (use - 1) & 1);
}

__device__ __forceinline__ void cp_async4(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}

// Prefetch cursor of a dequant thread: walks the CTA's items slice by slice
// ahead of the consumer and issues one cp.async group per slice into the raw
// ring (an empty group for slices of the shared expert or past the end, so
// group counts stay aligned with slices).  It also keeps the rows streaming
// from DRAM in long runs: each weight row is prefetched into L2 in
// kPfL2Window-byte windows eight slices ahead of the cursor, and the first
// 512 bytes of the next item's rows near the end of the current item (the
// per-slice copies alone read 32 bytes per row, which DRAM serves poorly).
template <int NA>
struct PfCursor {
  int item, s;
  bool mx;                 // this slice's item is a routed MXFP4 item with a valid row
  const uint8_t* row[NA];  // codes of the row
  const uint8_t* sw[NA];   // scale row (one 4-byte word covers two slices)
};

// Codes of weight row m0 + r of matrix a of `item`; null unless it is a
// routed item with a valid row.
__device__ __forceinline__ const uint8_t* item_row_codes(const ExpertParams& p, const PfCtx& c, bool gateup, int item,
                                                         uint32_t r, int a, const uint8_t** scales) {
  if (item >= c.n_items) return nullptr;
  const PfItem it = pf_item(item, p, c.pref, c.U, c.n_routed);
  if (it.shared) return nullptr;
  const moe_expert ex = p.experts[it.e];
  const int row = it.m0 + (int)r;
  if (row >= c.M || !expert_ptrs_ok(ex)) return nullptr;
  const moe_mx_mat m = a == 0 ? (gateup ? ex.gate : ex.down) : ex.up;
  if (scales) *scales = m.s + (size_t)row * (c.K / 32);
  return m.q + (size_t)row * (c.K / 2);
}

// The matrix whose L2 prefetches this thread issues (-1: none).
template <int NA>
__device__ __forceinline__ int prefetch_matrix(int half) {
  return NA == 2 ? half : (half == 0 ? 0 : -1);
}

template <int NA>
__device__ __forceinline__ void cursor_enter(PfCursor<NA>& cur, const ExpertParams& p, const PfCtx& c, bool gateup,
                                             uint32_t r) {
  cur.mx = true;
#pragma unroll
  for (int a = 0; a < NA; ++a) {
    cur.row[a] = item_row_codes(p, c, gateup, cur.item, r, a, &cur.sw[a]);
    cur.mx = cur.mx && cur.row[a] != nullptr;
  }
}

// Issue the cursor's slice into slot j % R of the group's raw ring, then move
// the cursor kPfDqGroups slices on (the group's next slice).
template <int NA, int R>
__device__ __forceinline__ void cursor_issue(PfCursor<NA>& cur, const ExpertParams& p, const PfCtx& c, bool gateup,
                                             uint32_t r, int half, uint8_t* raw, int j) {
  const int tid = threadIdx.x % kPfDqGroupThreads;
  uint8_t* slot = raw + (size_t)(j % R) * PfRaw<NA>::kStage;
  if (cur.item < c.n_items) {
    const int ns = c.nslices;
    const int rowbytes = c.K / 2;
    const int pa = prefetch_matrix<NA>(half);
    if (cur.mx) {
      if (pa >= 0 && (cur.s & 7) == 0) {
        const int off = (cur.s + 8) * 32;
        if (off < rowbytes) prefetch_l2(cur.row[pa] + off, (uint32_t)min(kPfL2Window, rowbytes - off));
      }
#pragma unroll
      for (int a = 0; a < NA; ++a) {
        cp_async16(slot + a * (kPfDqGroupThreads * 16) + tid * 16, cur.row[a] + (size_t)cur.s * 32 + half * 16);
        cp_async4(slot + PfRaw<NA>::kQ + a * (kPfDqGroupThreads * 4) + tid * 4, cur.sw[a] + (cur.s >> 1) * 4);
      }
    }
    if (pa >= 0 && cur.s == (ns > 16 ? ns - 16 : 0)) {
      const uint8_t* nq = item_row_codes(p, c, gateup, cur.item + gridDim.x, r, pa, nullptr);
      if (nq) prefetch_l2(nq, (uint32_t)min(512, rowbytes));
    }
    cur.s += kPfDqGroups;
    if (cur.s >= ns) {
      cur.s -= ns;
      cur.item += gridDim.x;
      cursor_enter(cur, p, c, gateup, r);
    }
  }
  cp_async_commit();
}

// Dequant warps: group k (warps 8k .. 8k+7) converts the slices s of every
// item with s % 2 == k; in a group, thread (row r, half) produces MX block
// 2s + half of weight row m0 + r, for gate and up (GATEUP) or down.  Routed
// MXFP4 rows come through the group's raw ring; the bf16 shared expert's rows
// are loaded directly.  (The slice count per item, K / 64, is even.)
template <bool GATEUP>
__device__ void pf_dequant_role(const ExpertParams& p, const PfCtx& c) {
  constexpr int NA = GATEUP ? 2 : 1;
  constexpr int R = GATEUP ? kPfRawGateUp : kPfRawDown;
  const int grp = threadIdx.x / kPfDqGroupThreads;
  const int tid = threadIdx.x % kPfDqGroupThreads;
  const int lane = threadIdx.x & 31;
  const uint32_t r = (uint32_t)tid >> 1;
  const int half = tid & 1;
  const uint32_t c0 = (uint32_t)half * 4;
  const int ns = c.nslices;
  PfShared& sh = *c.sh;
  uint8_t* raw = c.raw + (size_t)grp * R * PfRaw<NA>::kStage;
  PfCursor<NA> cur;
  cur.item = blockIdx.x;
  cur.s = grp;
  cursor_enter(cur, p, c, GATEUP, r);
  if (grp == 0 && cur.mx && prefetch_matrix<NA>(half) >= 0)
    prefetch_l2(cur.row[prefetch_matrix<NA>(half)], (uint32_t)min(512, c.K / 2));
  for (int j = 0; j < R; ++j) cursor_issue<NA, R>(cur, p, c, GATEUP, r, half, raw, j);
  int j = 0, ci = 0;  // j: the group's slices consumed so far
  bool ok = true;
  for (int item = blockIdx.x; item < c.n_items && ok; item += gridDim.x, ++ci) {
    const PfItem it = pf_item(item, p, c.pref, c.U, c.n_routed);
    // Row shifts of this item, published by the epilogue warps.
    const int slot = ci % kPfSigRing;
    if (!pf_warp_wait(c, &sh.sig_full[slot], (ci / kPfSigRing) & 1)) break;
    int sig[NA];
#pragma unroll
    for (int a = 0; a < NA; ++a) sig[a] = sh.sig[slot][a][r];
    __syncwarp();
    if (lane == 0) mbar_arrive(&sh.sig_empty[slot]);
    const uint16_t* wp[NA];
    float scale[NA];
    if (it.shared) {
      const int row = it.m0 + (int)r;
      const int rowc = row < c.M ? row : c.M - 1;
#pragma unroll
      for (int a = 0; a < NA; ++a) {
        const uint16_t* base = GATEUP ? (a == 0 ? p.sh_gate : p.sh_up) : p.sh_down;
        wp[a] = base + (size_t)rowc * c.K + half * 32;
        scale[a] = __int_as_float((sig[a] + 127) << 23);
      }
    }
    for (int s = grp; s < ns; s += kPfDqGroups, ++j) {
      const int g = ci * ns + s;
      cp_async_wait<R - 1>();  // this slice's group (empty for the shared expert)
      uint8_t* base = c.smem_a + (size_t)(g % c.a_stages) * c.a_bytes;
      if (!it.shared) {
        const uint8_t* rs = raw + (size_t)(j % R) * PfRaw<NA>::kStage;
        uint4 q[NA];
        uint32_t sc[NA];
        const int byte = ((s & 1) << 1) | half;
#pragma unroll
        for (int a = 0; a < NA; ++a) {
          q[a] = lds128(rs + a * (kPfDqGroupThreads * 16) + tid * 16);
          sc[a] = (*reinterpret_cast<const uint32_t*>(rs + PfRaw<NA>::kQ + a * (kPfDqGroupThreads * 4) + tid * 4) >>
                   (8 * byte)) & 0xFFu;
        }
        if (!pf_claim(c, sh.a_empty, c.a_stages, g)) {
          ok = false;
          break;
        }
#pragma unroll
        for (int a = 0; a < NA; ++a) dq_mx_block(base + a * kPfTileBytes, r, c0, q[a], sc[a], sig[a]);
      } else {
        // bf16 shared expert: 32 weights (64 bytes) per thread and slice.
        uint4 w[NA][4];
#pragma unroll
        for (int a = 0; a < NA; ++a)
#pragma unroll
          for (int jj = 0; jj < 4; ++jj) w[a][jj] = ldg_stream(wp[a] + (size_t)s * kPfSliceK + jj * 8);
        if (!pf_claim(c, sh.a_empty, c.a_stages, g)) {
          ok = false;
          break;
        }
#pragma unroll
        for (int a = 0; a < NA; ++a) dq_bf16_block(base + a * kPfTileBytes, r, c0, w[a], scale[a]);
      }
      fence_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh.a_full[g % c.a_stages]);
      cursor_issue<NA, R>(cur, p, c, GATEUP, r, half, raw, j + R);
    }
    if (*(volatile int*)&sh.abort_flag) ok = false;
  }
  cp_async_wait<0>();
}

// Loader warps: the item's token rows of the B operand (f16 activations for
// gate/up, f16 h for down), 16-byte cp.async chunks into the SW128 layout;
// rows between the token count and the next multiple of 16 are zero-filled
// by cp.async as well.  Each thread then arrives on the stage's barrier
// through cp.async.mbarrier.arrive, which fires when its copies have landed,
// so the loader never waits for its own copies: it runs ahead as far as the
// ring allows and each stage is ready as soon as its data is.
template <bool GATEUP>
__device__ void pf_loader_role(const ExpertParams& p, const PfCtx& c) {
  const int l = threadIdx.x - kPfDqWarps * 32;  // 0..127
  const int ns = c.nslices;
  const int npairs = p.T * p.k;
  bool ok = true;
  int gbase = 0;
  for (int item = blockIdx.x; item < c.n_items && ok; item += gridDim.x, gbase += ns) {
    const PfItem it = pf_item(item, p, c.pref, c.U, c.n_routed);
    const int nmma = (it.cnt + 15) & ~15;
    const uint16_t* src[8];
    uint32_t dst[8];
    bool use_chunk[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int idx = l + j * 128;
      const int n = idx >> 3, ch = idx & 7;
      use_chunk[j] = n < nmma;
      dst[j] = sw128_offset((uint32_t)n, (uint32_t)ch);
      src[j] = nullptr;
      if (n < it.cnt) {
        if (!GATEUP) {
          src[j] = p.ws.h16 + (size_t)(it.hpos0 + n) * p.I + ch * 8;
        } else if (it.shared) {
          src[j] = p.ws.xh + (size_t)(it.p0 + n) * p.H + ch * 8;
        } else {
          int pr = __ldg(&p.sorted[it.p0 + n]);
          if (pr < 0 || pr >= npairs) {
            set_status(c.hdr, MOE_ERR_DEVICE_CHECK);
            pr = 0;
          }
          src[j] = p.ws.xh + (size_t)(pr / p.k) * p.H + ch * 8;
        }
      }
    }
    for (int s = 0; s < ns; ++s) {
      const int gs = gbase + s;
      if (!pf_claim(c, c.sh->b_empty, c.b_stages, gs)) {
        ok = false;
        break;
      }
      uint8_t* btile = c.smem_b + (size_t)(gs % c.b_stages) * kPfTileBytes;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        if (!use_chunk[j]) continue;
        if (src[j])
          cp_async16(btile + dst[j], src[j] + (size_t)s * kPfSliceK);
        else
          cp_async16_zfill(btile + dst[j], p.ws.xh, 0u);
      }
      cp_async_mbar_arrive(&c.sh->b_full[gs % c.b_stages]);
    }
    if (*(volatile int*)&c.sh->abort_flag) ok = false;
  }
  cp_async_wait_all();
}

// Row shifts of local item j (the CTA's j-th item) into the shift ring, by
// the epilogue warps (thread = one weight row).  Routed rows: from the E8M0
// scales (sigma = 140 - max scale); shared-expert rows: from the pre-pass.
template <bool GATEUP>
__device__ __forceinline__ bool pf_publish_sig(const ExpertParams& p, const PfCtx& c, int j) {
  PfShared& sh = *c.sh;
  const int slot = j % kPfSigRing, use = j / kPfSigRing;
  if (use > 0 && !pf_warp_wait(c, &sh.sig_empty[slot], (use - 1) & 1)) return false;
  const int item = blockIdx.x + j * gridDim.x;
  const PfItem it = pf_item(item, p, c.pref, c.U, c.n_routed);
  const int rl = ((threadIdx.x >> 5) & 3) * 32 + (threadIdx.x & 31);
  const int row = it.m0 + rl;
  int s0 = 0, s1 = 0;
  if (row < c.M) {
    if (!it.shared) {
      const moe_expert ex = p.experts[it.e];
      if (expert_ptrs_ok(ex)) {
        s0 = sigma_from_smax(row_smax_part((GATEUP ? ex.gate.s : ex.down.s) + (size_t)row * (c.K / 32), c.K / 128, 0, 1));
        if (GATEUP) s1 = sigma_from_smax(row_smax_part(ex.up.s + (size_t)row * (c.K / 32), c.K / 128, 0, 1));
      }
    } else {
      s0 = __ldg(&p.ws.shsig[GATEUP ? row : 2 * p.I + row]);
      if (GATEUP) s1 = __ldg(&p.ws.shsig[p.I + row]);
    }
  }
  sh.sig[slot][0][rl] = s0;
  sh.sig[slot][1][rl] = s1;
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(&sh.sig_full[slot]);
  return true;
}

// Epilogue warps: warp q (= warp % 4) reads TMEM lanes 32q..32q+31, i.e.
// weight rows m0 + 32q + lane, one fp32 column per token.
//   gate/up: h[hpos0 + n][row] = f16(silu(g) * u), shifts removed;
//   down:    out[token(n)][row] += weight(n) * y.
// Before each item they publish the row shifts of the item kPfSigRing - 1
// places ahead, so the dequant warps never wait on the scale reads.
template <bool GATEUP>
__device__ void pf_epilogue_role(const ExpertParams& p, const PfCtx& c, uint32_t tmem) {
  const int q = (threadIdx.x >> 5) & 3;
  const int lane = threadIdx.x & 31;
  const int npairs = p.T * p.k;
  PfShared& sh = *c.sh;
  const int n_local = blockIdx.x < c.n_items ? (c.n_items - blockIdx.x + gridDim.x - 1) / gridDim.x : 0;
  int published = 0;
  int ci = 0;
  for (int item = blockIdx.x; item < c.n_items; item += gridDim.x, ++ci) {
    bool ok = true;
    while (ok && published < n_local && published < ci + kPfSigRing) ok = pf_publish_sig<GATEUP>(p, c, published++);
    if (!ok) break;
    const PfItem it = pf_item(item, p, c.pref, c.U, c.n_routed);
    const int b = ci & 1;
    const int rl = q * 32 + lane;
    const int row = it.m0 + rl;
    bool valid = row < c.M;
    if (!it.shared) valid = valid && expert_ptrs_ok(p.experts[it.e]);
    const int slot = ci % kPfSigRing;
    if (!pf_warp_wait(c, &sh.sig_full[slot], (ci / kPfSigRing) & 1)) break;
    const float rs0 = ldexpf(1.f, -sh.sig[slot][0][rl]);  // 2^-sigma of the row: gate (or down), up
    const float rs1 = ldexpf(1.f, -sh.sig[slot][1][rl]);
    __syncwarp();
    if (lane == 0) mbar_arrive(&sh.sig_empty[slot]);
    // Per-column token and factor.  Each warp builds its own copy: a barrier
    // across the epilogue warps could not be left by a warp that aborts.
    float* col_scale = sh.col_scale[q];
    int* col_tok = sh.col_tok[q];
    __syncwarp();
    for (int n = lane; n < it.cnt; n += 32) {
      int t;
      float wgt = 1.f;
      if (it.shared) {
        t = it.p0 + n;
      } else {
        int pr = __ldg(&p.sorted[it.p0 + n]);
        if (pr < 0 || pr >= npairs) pr = 0;  // flagged by the loader
        t = pr / p.k;
        wgt = __ldg(&p.w[pr]);
      }
      col_tok[n] = t;
      col_scale[n] = GATEUP ? __ldg(&p.ws.xscale[t]) : wgt * __ldg(&p.ws.hscale[it.hpos0 + n]);
    }
    __syncwarp();
    if (!pf_warp_wait(c, &sh.accf[b], (ci >> 1) & 1)) break;
    tc_fence_after();
    const uint32_t tbase = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(b * 256);
    for (int c0 = 0; c0 < it.cnt; c0 += 16) {
      uint32_t g[16];
      tmem_ld16(tbase + (uint32_t)c0, g);
      if (GATEUP) {
        uint32_t u[16];
        tmem_ld16(tbase + 128u + (uint32_t)c0, u);
        tmem_ld_wait();
        // h in fp32, and the largest |h| of each column (h row) over this
        // warp's 32 weight rows raised into hmax (non-negative floats order
        // as their bits; NaN orders above infinity).
        float* hout = reinterpret_cast<float*>(p.ws.h);
        uint32_t habs = 0u;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int n = c0 + i;
          uint32_t a = 0u;
          if (valid && n < it.cnt) {
            const float xs = col_scale[n];
            const float gv = __uint_as_float(g[i]) * rs0 * xs;
            const float uv = __uint_as_float(u[i]) * rs1 * xs;
            const float hv = silu_f32(gv) * uv;
            hout[(size_t)(it.hpos0 + n) * p.I + row] = hv;
            a = __float_as_uint(hv) & 0x7FFFFFFFu;
          }
          const uint32_t mx = __reduce_max_sync(0xFFFFFFFFu, a);
          if (lane == i) habs = mx;
        }
        if (lane < 16 && c0 + lane < it.cnt && habs != 0u) atomicMax(&p.ws.hmax[it.hpos0 + c0 + lane], habs);
      } else {
        tmem_ld_wait();
        if (valid) {
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int n = c0 + i;
            if (n < it.cnt) {
              const float v = (__uint_as_float(g[i]) * rs0) * col_scale[n];
              atomicAdd(&p.out[(size_t)col_tok[n] * p.H + row], v);
            }
          }
        }
      }
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(&sh.acce[b]);
  }
}

// MMA issuers (lane 0 of warp 24, and of warp 25 in the gate/up kernel): per
// item, wait for a free accumulator buffer, then per stage for the weight and
// token tiles, issue 4 K = 16 MMAs M = 128 x N = round16(tokens) into
// accumulator `which` (gate/up: matrix `which`; down: the one accumulator),
// and release the stages with tcgen05.commit; each issuer's last commit of the
// item counts towards the accumulator buffer being ready.  (Splitting the down
// contraction into even and odd stages over two issuers gave wrong tiles and
// a stalled wait in testing; it is not used.)
template <bool GATEUP>
__device__ void pf_mma_role(const ExpertParams& p, const PfCtx& c, uint32_t tmem, int which) {
  if (!GATEUP && which != 0) return;
  PfShared& sh = *c.sh;
  const int ns = c.nslices;
  int ci = 0;
  for (int item = blockIdx.x; item < c.n_items; item += gridDim.x, ++ci) {
    const PfItem it = pf_item(item, p, c.pref, c.U, c.n_routed);
    const int b = ci & 1;
    if (ci >= 2 && !pf_wait(sh, &sh.acce[b], ((ci >> 1) - 1) & 1, c.hdr)) break;
    tc_fence_after();
    const int nmma = (it.cnt + 15) & ~15;
    const uint32_t idesc = idesc_f16_f32(kPfMTile, nmma);
    const uint32_t dcol = tmem + (uint32_t)(b * 256 + which * 128);
    bool ok = true;
    bool first = true;
    for (int s = 0; s < ns; ++s) {
      const int gs = ci * ns + s;
      const int sa = gs % c.a_stages, sb = gs % c.b_stages;
      if (!pf_wait(sh, &sh.a_full[sa], (gs / c.a_stages) & 1, c.hdr) ||
          !pf_wait(sh, &sh.b_full[sb], (gs / c.b_stages) & 1, c.hdr)) {
        ok = false;
        break;
      }
      fence_async_smem();  // the token tile was written by cp.async (generic proxy)
      tc_fence_after();
      const uint32_t abase = smem_u32(c.smem_a + (size_t)sa * c.a_bytes + (GATEUP ? which * kPfTileBytes : 0));
      const uint32_t bbase = smem_u32(c.smem_b + (size_t)sb * kPfTileBytes);
#pragma unroll
      for (int kk = 0; kk < kPfSliceK / 16; ++kk) {
        umma_f16(dcol, sdesc_sw128(abase + kk * 32), sdesc_sw128(bbase + kk * 32), idesc, first ? 0u : 1u);
        first = false;
      }
      umma_commit(&sh.a_empty[sa]);
      umma_commit(&sh.b_empty[sb]);
    }
    umma_commit(&sh.accf[b]);
    if (!ok) {
      ++ci;
      break;
    }
  }
  // Every MMA issued must have finished before TMEM is released.
  if (ci > 0) {
    const int last = ci - 1;
    if (!mbar_wait(&sh.accf[last & 1], (last >> 1) & 1)) set_status(c.hdr, MOE_ERR_TIMEOUT);
  }
}

// Persistent grouped GEMM, one CTA per SM.  GATEUP: A = gate and up rows (M =
// I), K = H, B = f16 activations; else A = down rows (M = H), K = I, B = h.
template <bool GATEUP>
__global__ void __launch_bounds__(kPfThreads, 1) k_pf_gemm(ExpertParams p) {
  constexpr int NA = GATEUP ? 2 : 1;
  constexpr int AS = GATEUP ? kPfAStagesGateUp : kPfAStagesDown;
  constexpr int BS = GATEUP ? kPfBStagesGateUp : kPfBStagesDown;
  extern __shared__ uint8_t pf_dyn[];
  __shared__ PfShared sh;
  const int warp = threadIdx.x >> 5;
  if (warp == kPfMmaWarp) {
    tmem_alloc(&sh.tmem_base, kPfTmemCols);
    tmem_relinquish();
  }
  if (threadIdx.x == 0) {
    // gate/up: both issuers read every stage; down: one issuer per stage.
    for (int s = 0; s < AS; ++s) {
      mbar_init(&sh.a_full[s], kPfDqGroupWarps);
      mbar_init(&sh.a_empty[s], GATEUP ? kPfMmaWarps : 1);
    }
    for (int s = 0; s < BS; ++s) {
      mbar_init(&sh.b_full[s], kPfLdWarps * 32);
      mbar_init(&sh.b_empty[s], GATEUP ? kPfMmaWarps : 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sh.accf[b], GATEUP ? kPfMmaWarps : 1);
      mbar_init(&sh.acce[b], kPfEpWarps);
    }
    for (int i = 0; i < kPfSigRing; ++i) {
      mbar_init(&sh.sig_full[i], kPfEpWarps);
      mbar_init(&sh.sig_empty[i], kPfDqWarps + kPfEpWarps);
    }
    sh.abort_flag = 0;
    mbar_init_fence();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sh.tmem_base;

  PfCtx c;
  c.sh = &sh;
  c.smem_a = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(pf_dyn) + 1023) & ~(uintptr_t)1023);
  c.a_stages = AS;
  c.b_stages = BS;
  c.a_bytes = NA * kPfTileBytes;
  c.smem_b = c.smem_a + (size_t)AS * c.a_bytes;
  c.raw = c.smem_b + (size_t)BS * kPfTileBytes;
  c.K = GATEUP ? p.H : p.I;
  c.M = GATEUP ? p.I : p.H;
  c.nslices = c.K / kPfSliceK;
  c.hdr = p.ws.hdr;
  c.U = (int)p.ws.hdr->n_active;
  c.pref = GATEUP ? p.ws.act_pref_gu : p.ws.act_pref_dn;
  c.n_routed = c.U > 0 ? __ldg(&c.pref[c.U]) : 0;
  const int m_tiles = (c.M + kPfMTile - 1) / kPfMTile;
  c.n_items = c.n_routed + (p.sh_gate ? m_tiles * ((p.T + kPfNTile - 1) / kPfNTile) : 0);

  if (warp < kPfDqWarps)
    pf_dequant_role<GATEUP>(p, c);
  else if (warp < kPfDqWarps + kPfLdWarps)
    pf_loader_role<GATEUP>(p, c);
  else if (warp < kPfMmaWarp)
    pf_epilogue_role<GATEUP>(p, c, tmem);
  else if ((threadIdx.x & 31) == 0)
    pf_mma_role<GATEUP>(p, c, tmem, warp - kPfMmaWarp);

  tc_fence_before();
  __syncthreads();
  if (warp == kPfMmaWarp) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kPfTmemCols);
  }
}

bool prefill_supported(int H, int I) { return H % 128 == 0 && I % 128 == 0; }

cudaError_t launch_prefill_experts(const ExpertParams& p, cudaStream_t s) {
  if (!p.x_bf16 || !prefill_supported(p.H, p.I)) return cudaErrorNotSupported;
  const int nsm = device_sm_count();
  cudaError_t err;
  // Bucket layout, active experts and tile prefixes come from the routing or
  // bucketing kernels already on the stream.
  k_x_to_f16<<<p.T, 256, 0, s>>>(p);
  if ((err = cudaGetLastError()) != cudaSuccess) return err;
  if (p.sh_gate) {
    k_shared_sigma<<<(2 * p.I + p.H + 7) / 8, 256, 0, s>>>(p);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
  }
  if (!p.accumulate) {
    if ((err = cudaMemsetAsync(p.out, 0, (size_t)p.T * p.H * sizeof(float), s)) != cudaSuccess) return err;
  }
  // Weight tile ring + token tile ring + raw MXFP4 ring + alignment slack.
  const size_t gu_smem = (size_t)(kPfAStagesGateUp * 2 + kPfBStagesGateUp) * kPfTileBytes +
                         (size_t)kPfDqGroups * kPfRawGateUp * PfRaw<2>::kStage + 1024;
  const size_t dn_smem = (size_t)(kPfAStagesDown + kPfBStagesDown) * kPfTileBytes +
                         (size_t)kPfDqGroups * kPfRawDown * PfRaw<1>::kStage + 1024;
  if ((err = ensure_smem_attr((const void*)k_pf_gemm<true>, gu_smem)) != cudaSuccess) return err;
  if ((err = ensure_smem_attr((const void*)k_pf_gemm<false>, dn_smem)) != cudaSuccess) return err;
  prof_before(MOE_STAGE_PF_GATEUP, s);
  k_pf_gemm<true><<<nsm, kPfThreads, gu_smem, s>>>(p);
  prof_after(MOE_STAGE_PF_GATEUP, s);
  if ((err = cudaGetLastError()) != cudaSuccess) return err;
  // f16 h rows for the down GEMM: the routed pairs' rows (none when the
  // shared expert runs alone) and the shared expert's.
  const int hrow0 = p.shared_only ? p.T * p.k : 0;
  const int hrow1 = p.T * p.k + (p.sh_gate ? p.T : 0);
  if (hrow1 > hrow0) {
    k_h_to_f16<<<(hrow1 - hrow0 + 7) / 8, 256, 0, s>>>(p, hrow0, hrow1);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
  }
  prof_before(MOE_STAGE_PF_DOWN, s);
  k_pf_gemm<false><<<nsm, kPfThreads, dn_smem, s>>>(p);
  prof_after(MOE_STAGE_PF_DOWN, s);
  return cudaGetLastError();
}

}  // namespace moe
