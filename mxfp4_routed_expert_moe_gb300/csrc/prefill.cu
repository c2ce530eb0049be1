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
// gate/up: the epilogue applies SwiGLU and stores h in f16, bucket order.
// down: the epilogue adds w[t][j] * y into out with fp32 atomics.
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
constexpr int kPfDqWarps = 8;            // warps 0-7: weight dequant (2 threads per weight row)
constexpr int kPfLdWarps = 4;            // warps 8-11: token rows (cp.async)
constexpr int kPfEpWarps = 4;            // warps 12-15: epilogue (warp % 4 = TMEM lane quarter)
constexpr int kPfMmaWarp = kPfDqWarps + kPfLdWarps + kPfEpWarps;  // warp 16: TMEM owner, MMA issuer
constexpr int kPfThreads = (kPfMmaWarp + 1) * 32;
constexpr int kPfBDepth = 3;             // cp.async groups in flight per loader thread
constexpr int kPfMaxStages = 8;
constexpr uint32_t kPfTmemCols = 512;    // 2 accumulator buffers x (gate 128 + up 128) columns
static_assert(kPfEpWarps == 4 && (kPfDqWarps + kPfLdWarps) % 4 == 0, "epilogue warps must cover lane quarters 0-3");

// ------------------------------------------------------------ pre-passes --
// xh[t][h] = f16(x[t][h] * 2^sigma_t), xscale[t] = 2^-sigma_t, with sigma_t
// putting the token's largest magnitude in [2^14, 2^15).
__global__ void __launch_bounds__(256) k_x_to_f16(ExpertParams p) {
  __shared__ float wmax[8];
  const int t = blockIdx.x;
  const int H = p.H;
  const uint16_t* xb = reinterpret_cast<const uint16_t*>(p.x) + (size_t)t * H;
  float m = 0.f;
  for (int h = threadIdx.x * 8; h < H; h += blockDim.x * 8) {
    const uint4 v = *reinterpret_cast<const uint4*>(xb + h);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j)
      m = fmaxf(m, fmaxf(fabsf(__uint_as_float(w[j] << 16)), fabsf(__uint_as_float(w[j] & 0xFFFF0000u))));
  }
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
  if ((threadIdx.x & 31) == 0) wmax[threadIdx.x >> 5] = m;
  __syncthreads();
  m = 0.f;
  for (int w = 0; w < (int)(blockDim.x >> 5); ++w) m = fmaxf(m, wmax[w]);
  int sig = 0;
  if (m > 0.f) sig = 14 - ((int)((__float_as_uint(m) >> 23) & 0xFF) - 127);
  sig = sig > 100 ? 100 : (sig < -100 ? -100 : sig);
  const float up = __int_as_float((sig + 127) << 23);
  if (threadIdx.x == 0) p.ws.xscale[t] = __int_as_float((127 - sig) << 23);
  uint16_t* xo = p.ws.xh + (size_t)t * H;
  for (int h = threadIdx.x * 8; h < H; h += blockDim.x * 8) {
    const uint4 v = *reinterpret_cast<const uint4*>(xb + h);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const __half2 h2 = __floats2half2_rn(__uint_as_float(w[j] << 16) * up, __uint_as_float(w[j] & 0xFFFF0000u) * up);
      o[j] = *reinterpret_cast<const uint32_t*>(&h2);
    }
    *reinterpret_cast<uint4*>(xo + h) = make_uint4(o[0], o[1], o[2], o[3]);
  }
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
  uint64_t full[kPfMaxStages];   // stage filled: 8 dequant + 4 loader warp arrivals
  uint64_t empty[kPfMaxStages];  // stage consumed: tcgen05.commit
  uint64_t accf[2];              // accumulator buffer ready: tcgen05.commit
  uint64_t acce[2];              // accumulator buffer drained: 4 epilogue warps
  uint32_t tmem_base;
  int abort_flag;
  float col_scale[kPfEpWarps][kPfNTile];  // per epilogue warp: token shift (gate/up) or route weight (down)
  int col_tok[kPfEpWarps][kPfNTile];      // per epilogue warp: token of each column (down)
};

// Bounded wait that also gives up as soon as another role has aborted.
__device__ __forceinline__ bool pf_wait(PfShared& sh, uint64_t* bar, uint32_t parity, WsHeader* hdr) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  for (;;) {
    if (mbar_try_wait(bar, parity)) return true;
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
  uint8_t* smem;     // stage ring, 1024-byte aligned
  int stages;
  int stage_bytes;
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

// Claim stage of global slice gs for writing (wait until its previous use was
// consumed by the tensor core).
__device__ __forceinline__ bool pf_claim(const PfCtx& c, int gs) {
  const int st = gs % c.stages, use = gs / c.stages;
  if (use == 0) return true;
  return pf_warp_wait(c, &c.sh->empty[st], (use - 1) & 1);
}

template <int NA>
struct MxBuf {
  uint4 q[NA];
  uint32_t s[NA];
};

template <int NA>
__device__ __forceinline__ void mx_load(MxBuf<NA>& b, const uint8_t* const (&qp)[NA], const uint8_t* const (&sp)[NA],
                                        int s) {
#pragma unroll
  for (int a = 0; a < NA; ++a) {
    b.q[a] = ldg_stream(qp[a] + (size_t)s * 32);
    b.s[a] = ldg_u8(sp[a] + (size_t)s * 2);
  }
}

// Dequantize one slice from registers into its stage and signal it.
template <int NA>
__device__ __forceinline__ bool mx_slice(const PfCtx& c, int gs, uint32_t r, uint32_t c0, const MxBuf<NA>& b,
                                         const int (&sig)[NA]) {
  if (!pf_claim(c, gs)) return false;
  const int st = gs % c.stages;
  uint8_t* base = c.smem + (size_t)st * c.stage_bytes;
#pragma unroll
  for (int a = 0; a < NA; ++a) dq_mx_block(base + a * kPfTileBytes, r, c0, b.q[a], b.s[a], sig[a]);
  fence_async_smem();
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(&c.sh->full[st]);
  return true;
}

// Dequant warps: thread (row r, half) produces MX block 2s + half of weight
// row m0 + r for every slice s, for gate and up (GATEUP) or down.
template <bool GATEUP>
__device__ void pf_dequant_role(const ExpertParams& p, const PfCtx& c) {
  constexpr int NA = GATEUP ? 2 : 1;
  const uint32_t r = threadIdx.x >> 1;
  const int half = threadIdx.x & 1;
  const uint32_t c0 = (uint32_t)half * 4;
  const int ns = c.nslices;
  int gbase = 0;
  for (int item = blockIdx.x; item < c.n_items; item += gridDim.x, gbase += ns) {
    const PfItem it = pf_item(item, p, c.pref, c.U, c.n_routed);
    const int row = it.m0 + (int)r;
    bool ok = true;
    if (!it.shared) {
      const moe_expert ex = p.experts[it.e];
      const bool valid = row < c.M && expert_ptrs_ok(ex);
      if (!expert_ptrs_ok(ex) && threadIdx.x == 0) set_status(c.hdr, MOE_ERR_DEVICE_CHECK);
      const moe_mx_mat mats[2] = {GATEUP ? ex.gate : ex.down, ex.up};
      const uint8_t* qp[NA];
      const uint8_t* sp[NA];
      int sig[NA];
#pragma unroll
      for (int a = 0; a < NA; ++a) {
        qp[a] = valid ? mats[a].q + (size_t)row * (c.K / 2) + half * 16 : nullptr;
        sp[a] = valid ? mats[a].s + (size_t)row * (c.K / 32) + half : nullptr;
        int smax = valid ? row_smax_part(mats[a].s + (size_t)row * (c.K / 32), c.K / 128, half, 2) : -1;
        smax = max(smax, __shfl_xor_sync(0xFFFFFFFFu, smax, 1));
        sig[a] = sigma_from_smax(smax);
      }
      MxBuf<NA> b0, b1, b2;
#pragma unroll
      for (int a = 0; a < NA; ++a) {
        b0.q[a] = b1.q[a] = b2.q[a] = make_uint4(0, 0, 0, 0);
        b0.s[a] = b1.s[a] = b2.s[a] = 0;
      }
      if (valid) {
        mx_load(b0, qp, sp, 0);
        if (ns > 1) mx_load(b1, qp, sp, 1);
      }
      for (int s = 0; s < ns && ok; s += 3) {
        if (valid && s + 2 < ns) mx_load(b2, qp, sp, s + 2);
        ok = mx_slice(c, gbase + s, r, c0, b0, sig);
        if (!ok || s + 1 >= ns) break;
        if (valid && s + 3 < ns) mx_load(b0, qp, sp, s + 3);
        ok = mx_slice(c, gbase + s + 1, r, c0, b1, sig);
        if (!ok || s + 2 >= ns) break;
        if (valid && s + 4 < ns) mx_load(b1, qp, sp, s + 4);
        ok = mx_slice(c, gbase + s + 2, r, c0, b2, sig);
      }
    } else {
      // bf16 shared expert: 32 weights (64 bytes) per thread and slice.
      const uint16_t* wp[NA];
      float scale[NA];
      const int rowc = row < c.M ? row : c.M - 1;
#pragma unroll
      for (int a = 0; a < NA; ++a) {
        const uint16_t* base = GATEUP ? (a == 0 ? p.sh_gate : p.sh_up) : p.sh_down;
        const int sidx = GATEUP ? a * p.I + rowc : 2 * p.I + rowc;
        wp[a] = base + (size_t)rowc * c.K + half * 32;
        scale[a] = __int_as_float((__ldg(&p.ws.shsig[sidx]) + 127) << 23);
      }
      uint4 cur[NA][4];
#pragma unroll
      for (int a = 0; a < NA; ++a)
#pragma unroll
        for (int j = 0; j < 4; ++j) cur[a][j] = ldg_stream(wp[a] + j * 8);
      for (int s = 0; s < ns; ++s) {
        uint4 nxt[NA][4];
        const int sn = s + 1 < ns ? s + 1 : s;
#pragma unroll
        for (int a = 0; a < NA; ++a)
#pragma unroll
          for (int j = 0; j < 4; ++j) nxt[a][j] = ldg_stream(wp[a] + (size_t)sn * kPfSliceK + j * 8);
        ok = pf_claim(c, gbase + s);
        if (!ok) break;
        const int st = (gbase + s) % c.stages;
        uint8_t* base = c.smem + (size_t)st * c.stage_bytes;
#pragma unroll
        for (int a = 0; a < NA; ++a) dq_bf16_block(base + a * kPfTileBytes, r, c0, cur[a], scale[a]);
        fence_async_smem();
        __syncwarp();
        if ((threadIdx.x & 31) == 0) mbar_arrive(&c.sh->full[st]);
#pragma unroll
        for (int a = 0; a < NA; ++a)
#pragma unroll
          for (int j = 0; j < 4; ++j) cur[a][j] = nxt[a][j];
      }
    }
    if (!ok || *(volatile int*)&c.sh->abort_flag) break;
  }
}

// Loader warps: the item's token rows of the B operand (f16 activations for
// gate/up, f16 h for down), 16-byte cp.async chunks into the SW128 layout;
// rows between the token count and the next multiple of 16 are zero.  Each
// slice is one cp.async group; a group's stage is signalled kPfBDepth - 1
// groups later, so several slices are in flight per thread.
template <bool GATEUP>
__device__ void pf_loader_role(const ExpertParams& p, const PfCtx& c) {
  constexpr int NA = GATEUP ? 2 : 1;
  const int l = threadIdx.x - kPfDqWarps * 32;  // 0..127
  const int lane = threadIdx.x & 31;
  const int ns = c.nslices;
  const int npairs = p.T * p.k;
  int pending = 0;  // groups committed so far == global slices issued
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
          src[j] = reinterpret_cast<const uint16_t*>(p.ws.h) + (size_t)(it.hpos0 + n) * p.I + ch * 8;
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
      if (!pf_claim(c, gs)) {
        ok = false;
        break;
      }
      uint8_t* btile = c.smem + (size_t)(gs % c.stages) * c.stage_bytes + NA * kPfTileBytes;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        if (!use_chunk[j]) continue;
        if (src[j])
          cp_async16(btile + dst[j], src[j] + (size_t)s * kPfSliceK);
        else
          *reinterpret_cast<uint4*>(btile + dst[j]) = make_uint4(0, 0, 0, 0);
      }
      cp_async_commit();
      ++pending;
      if (pending >= kPfBDepth) {
        cp_async_wait<kPfBDepth - 1>();
        fence_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&c.sh->full[(pending - kPfBDepth) % c.stages]);
      }
    }
    if (*(volatile int*)&c.sh->abort_flag) ok = false;
  }
  // Complete and signal the groups still in flight.
  cp_async_wait<0>();
  fence_async_smem();
  __syncwarp();
  if (ok && lane == 0)
    for (int g = pending - (kPfBDepth - 1) > 0 ? pending - (kPfBDepth - 1) : 0; g < pending; ++g)
      mbar_arrive(&c.sh->full[g % c.stages]);
}

// Epilogue warps: warp q (= warp % 4) reads TMEM lanes 32q..32q+31, i.e.
// weight rows m0 + 32q + lane, one fp32 column per token.
//   gate/up: h[hpos0 + n][row] = f16(silu(g) * u), shifts removed;
//   down:    out[token(n)][row] += weight(n) * y.
template <bool GATEUP>
__device__ void pf_epilogue_role(const ExpertParams& p, const PfCtx& c, uint32_t tmem) {
  const int q = (threadIdx.x >> 5) & 3;
  const int lane = threadIdx.x & 31;
  const int npairs = p.T * p.k;
  PfShared& sh = *c.sh;
  int ci = 0;
  for (int item = blockIdx.x; item < c.n_items; item += gridDim.x, ++ci) {
    const PfItem it = pf_item(item, p, c.pref, c.U, c.n_routed);
    const int b = ci & 1;
    const int row = it.m0 + q * 32 + lane;
    bool valid = row < c.M;
    float rs0 = 1.f, rs1 = 1.f;  // 2^-sigma of the row: gate (or down), up
    if (!it.shared) {
      const moe_expert ex = p.experts[it.e];
      valid = valid && expert_ptrs_ok(ex);
      if (valid) {
        const uint8_t* s0 = (GATEUP ? ex.gate.s : ex.down.s) + (size_t)row * (c.K / 32);
        rs0 = ldexpf(1.f, -sigma_from_smax(row_smax_part(s0, c.K / 128, 0, 1)));
        if (GATEUP)
          rs1 = ldexpf(1.f, -sigma_from_smax(row_smax_part(ex.up.s + (size_t)row * (c.K / 32), c.K / 128, 0, 1)));
      }
    } else if (valid) {
      rs0 = ldexpf(1.f, -__ldg(&p.ws.shsig[GATEUP ? row : 2 * p.I + row]));
      if (GATEUP) rs1 = ldexpf(1.f, -__ldg(&p.ws.shsig[p.I + row]));
    }
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
      col_scale[n] = GATEUP ? __ldg(&p.ws.xscale[t]) : wgt;
    }
    __syncwarp();
    if (!pf_warp_wait(c, &sh.accf[b], (ci >> 1) & 1)) break;
    tc_fence_after();
    const uint32_t tbase = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(b * 256);
    for (int c0 = 0; c0 < it.cnt; c0 += 32) {
      uint32_t g[32];
      tmem_ld32(tbase + (uint32_t)c0, g);
      if (GATEUP) {
        uint32_t u[32];
        tmem_ld32(tbase + 128u + (uint32_t)c0, u);
        tmem_ld_wait();
        if (valid) {
          __half* hout = reinterpret_cast<__half*>(p.ws.h) + (size_t)(it.hpos0 + c0) * p.I + row;
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            if (c0 + i < it.cnt) {
              const float xs = col_scale[c0 + i];
              const float gv = (__uint_as_float(g[i]) * rs0) * xs;
              const float uv = (__uint_as_float(u[i]) * rs1) * xs;
              const float hv = silu_f32(gv) * uv;
              if (fabsf(hv) > 65504.f) set_status(c.hdr, MOE_ERR_RANGE);
              hout[(size_t)i * p.I] = __float2half_rn(hv);
            }
          }
        }
      } else {
        tmem_ld_wait();
        if (valid) {
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            if (c0 + i < it.cnt) {
              const float v = (__uint_as_float(g[i]) * rs0) * col_scale[c0 + i];
              atomicAdd(&p.out[(size_t)col_tok[c0 + i] * p.H + row], v);
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

// MMA warp, lane 0: per item, waits for a free accumulator buffer, then per
// slice for a full stage, issues 4 (x2 for gate and up) K = 16 MMAs
// M = 128 x N = round16(tokens), and releases the stage with tcgen05.commit;
// the item's last commit marks the accumulator ready.
template <bool GATEUP>
__device__ void pf_mma_role(const ExpertParams& p, const PfCtx& c, uint32_t tmem) {
  constexpr int NA = GATEUP ? 2 : 1;
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
    const uint32_t dcol = tmem + (uint32_t)(b * 256);
    bool ok = true;
    for (int s = 0; s < ns; ++s) {
      const int gs = ci * ns + s;
      const int st = gs % c.stages, use = gs / c.stages;
      if (!pf_wait(sh, &sh.full[st], use & 1, c.hdr)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t abase = smem_u32(c.smem + (size_t)st * c.stage_bytes);
      const uint32_t bbase = abase + NA * kPfTileBytes;
#pragma unroll
      for (int kk = 0; kk < kPfSliceK / 16; ++kk) {
        const uint64_t bdesc = sdesc_sw128(bbase + kk * 32);
#pragma unroll
        for (int a = 0; a < NA; ++a)
          umma_f16(dcol + (uint32_t)(a * 128), sdesc_sw128(abase + a * kPfTileBytes + kk * 32), bdesc, idesc,
                   (s | kk) != 0 ? 1u : 0u);
      }
      umma_commit(&sh.empty[st]);
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
__global__ void __launch_bounds__(kPfThreads, 1) k_pf_gemm(ExpertParams p, int stages) {
  constexpr int NA = GATEUP ? 2 : 1;
  extern __shared__ uint8_t pf_dyn[];
  __shared__ PfShared sh;
  const int warp = threadIdx.x >> 5;
  if (warp == kPfMmaWarp) {
    tmem_alloc(&sh.tmem_base, kPfTmemCols);
    tmem_relinquish();
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(&sh.full[s], kPfDqWarps + kPfLdWarps);
      mbar_init(&sh.empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sh.accf[b], 1);
      mbar_init(&sh.acce[b], kPfEpWarps);
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
  c.smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(pf_dyn) + 1023) & ~(uintptr_t)1023);
  c.stages = stages;
  c.stage_bytes = (NA + 1) * kPfTileBytes;
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
    pf_mma_role<GATEUP>(p, c, tmem);

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
  const int gu_stages = 4, dn_stages = 6;
  const size_t gu_smem = (size_t)gu_stages * 3 * kPfTileBytes + 1024;
  const size_t dn_smem = (size_t)dn_stages * 2 * kPfTileBytes + 1024;
  if ((err = ensure_smem_attr((const void*)k_pf_gemm<true>, gu_smem)) != cudaSuccess) return err;
  if ((err = ensure_smem_attr((const void*)k_pf_gemm<false>, dn_smem)) != cudaSuccess) return err;
  prof_before(MOE_STAGE_PF_GATEUP, s);
  k_pf_gemm<true><<<nsm, kPfThreads, gu_smem, s>>>(p, gu_stages);
  prof_after(MOE_STAGE_PF_GATEUP, s);
  if ((err = cudaGetLastError()) != cudaSuccess) return err;
  prof_before(MOE_STAGE_PF_DOWN, s);
  k_pf_gemm<false><<<nsm, kPfThreads, dn_smem, s>>>(p, dn_stages);
  prof_after(MOE_STAGE_PF_DOWN, s);
  return cudaGetLastError();
}

}  // namespace moe
