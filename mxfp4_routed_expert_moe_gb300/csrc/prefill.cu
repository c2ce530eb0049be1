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
#include <cuda.h>
#include <string.h>

#include <mutex>
#include <utility>

#include "async.cuh"
#include "kernels.h"
#include "tcgen05.cuh"

namespace moe {

constexpr int kPfSliceK = 64;            // contraction elements per stage (one 128-byte swizzle row)
constexpr int kPfTileBytes = 128 * 128;  // one 128-row x 64-element f16 token tile
// Roles: 16 dequant warps (one weight row per thread and matrix; they write
// the f16 A operand straight into Tensor Memory), 4 loader warps (token rows,
// cp.async), 4 epilogue warps (warp % 4 = TMEM lane quarter), 2 MMA issuers.
// MMA issue: one thread issues a tcgen05.mma only every ~100 cycles whatever
// its size, so the gate/up kernel issues from two warps, one accumulator each
// (gate, up).  The down kernel has one accumulator per buffer and one issuer.
constexpr int kPfDqWarps = 16;           // warps 0-15
constexpr int kPfLdWarps = 4;            // warps 16-19
constexpr int kPfEpWarps = 4;            // warps 20-23
constexpr int kPfMmaWarp = kPfDqWarps + kPfLdWarps + kPfEpWarps;  // warps 24-25; 24 owns TMEM
constexpr int kPfMmaWarps = 2;
constexpr int kPfGuIssuers = 2;          // gate/up: one thread per matrix issues its MMAs (1: one thread both)
constexpr int kPfThreads = (kPfMmaWarp + kPfMmaWarps) * 32;
constexpr int kPfMaxStages = 8;
constexpr int kPfL2Window = 256;         // bytes of each weight row prefetched into L2 at a time
constexpr uint32_t kPfTmemCols = 512;
constexpr uint32_t kPfAccCols = 256;     // TMEM columns [0, 256): accumulators; [256, 512): A stages
constexpr int kPfSigRing = 4;            // items whose row shifts are published ahead
// Per kernel:
//   NA    matrices per item (gate/up: 2, down: 1)
//   GW    warps of one dequant group (4 per matrix: one TMEM lane quarter
//         each); a group fills one A stage, and the NG groups take turns
//         over the CTA's slices
//   ACCB  accumulator buffers: gate/up one (gate columns 0-127, up 128-255),
//         down two of 128 columns (the epilogue of one item overlaps the
//         next item's MMAs)
//   AS    A stages in TMEM, ACOLS columns each (64 f16 of a row = 32 columns
//         per matrix)
//   BS    token ring stages (shared memory)
//   R     raw MXFP4 slots per dequant group (its slices copied ahead)
template <bool GATEUP>
struct PfCfg {
  static constexpr int NA = GATEUP ? 2 : 1;
  static constexpr int GW = 4 * NA;
  static constexpr int NG = kPfDqWarps / GW;
  static constexpr int NI = GATEUP ? kPfGuIssuers : 1;  // MMA-issuing threads
  static constexpr int ACCB = GATEUP ? 1 : 2;
  static constexpr int ACCW = GATEUP ? 256 : 128;  // columns per accumulator buffer
  static constexpr int ACOLS = 32 * NA;
  static constexpr int AS = (int)(kPfTmemCols - kPfAccCols) / ACOLS;  // 4 or 8
  static constexpr int BS = 8;                      // (a power of two, as AS)
  static constexpr int R = GATEUP ? 3 : 4;
  // Raw slot: the 32 bytes of codes of each group thread (first 16 bytes of
  // every thread, then the second 16), then its 4-byte scale word.
  static constexpr int kThreads = GW * 32;
  static constexpr int kQ = kThreads * 32;
  static constexpr int kStage = kQ + kThreads * 4;
};
static_assert(kPfEpWarps == 4 && (kPfDqWarps + kPfLdWarps) % 4 == 0, "epilogue warps must cover lane quarters 0-3");
static_assert(PfCfg<true>::AS <= kPfMaxStages && PfCfg<false>::AS <= kPfMaxStages, "A stages");
static_assert((PfCfg<true>::AS & (PfCfg<true>::AS - 1)) == 0 && (PfCfg<false>::AS & (PfCfg<false>::AS - 1)) == 0 &&
                  (PfCfg<true>::BS & (PfCfg<true>::BS - 1)) == 0 && PfCfg<true>::BS <= kPfMaxStages,
              "ring depths are powers of two (stage and phase by mask and shift)");

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

// x[t] (bf16) as two E4M3 terms for the block-scaled gate/up GEMM: with
// tau_t = 7 - floor(log2 max_h |x[t][h]|), v = x * 2^tau_t has its largest
// magnitude in [128, 256); x1 = e4m3(v) (round to nearest even) keeps the top
// 4 significant bits of v and x2 = e4m3(16 (v - x1)) the remaining 4 of a bf16
// value, so v = x1 + x2 / 16 exactly for every element that is an E4M3 normal
// number after scaling (|v| >= 2^-6, i.e. within 2^-13 of the maximum); below
// that, the absolute error is at most 2^-14 (2^-21 of the maximum).
// The terms are written once per routed pair of the token, at its bucket
// position r = pinv[t k + j]: xp[0][r] = x1, xp[1][r] = x2 (one byte per
// element, in h order), so that each GEMM item's token rows are contiguous;
// x8scale[t] = 2^-tau_t.  One CTA per token; also clears the token's h-row
// maxima.
__global__ void __launch_bounds__(256) k_x_to_e4m3(ExpertParams p) {
  __shared__ float wmax[8];
  __shared__ int pos[32];
  const int t = blockIdx.x, H = p.H, k = p.k;
  if ((int)threadIdx.x < k) pos[threadIdx.x] = p.ws.pinv[(size_t)t * k + threadIdx.x];
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
#pragma unroll
  for (int w = 0; w < 8; ++w) m = fmaxf(m, wmax[w]);
  int tau = 0;
  if (m > 0.f && m < INFINITY) tau = 7 - ((int)((__float_as_uint(m) >> 23) & 0xFF) - 127);
  tau = tau > 126 ? 126 : (tau < -126 ? -126 : tau);
  const float up = __int_as_float((tau + 127) << 23);
  if (threadIdx.x == 0) p.ws.x8scale[t] = __int_as_float((127 - tau) << 23);
  const size_t plane = (size_t)p.T * k * H;
  for (int h = threadIdx.x * 8; h < H; h += blockDim.x * 8) {
    const uint4 v = *reinterpret_cast<const uint4*>(xb + h);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t o1[2], o2[2];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      // Elements h + 2j (low bf16 half) and h + 2j + 1: the first goes to the
      // low byte (cvt puts its first source operand in the high byte).
      const float a = __uint_as_float(w[j] << 16) * up, b = __uint_as_float(w[j] & 0xFFFF0000u) * up;
      unsigned short q1, q2;
      uint32_t f2;
      asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(q1) : "f"(b), "f"(a));
      asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(f2) : "h"(q1));
      const float2 x1f = __half22float2(*reinterpret_cast<const __half2*>(&f2));
      asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(q2) : "f"((b - x1f.y) * 16.f), "f"((a - x1f.x) * 16.f));
      const int wd = j >> 1, sh = 16 * (j & 1);
      if ((j & 1) == 0) {
        o1[wd] = q1;
        o2[wd] = q2;
      } else {
        o1[wd] |= (uint32_t)q1 << sh;
        o2[wd] |= (uint32_t)q2 << sh;
      }
    }
    for (int j = 0; j < k; ++j) {
      const int r = pos[j];
      if (r < 0) continue;
      uint8_t* x1 = p.ws.xp + (size_t)r * H + h;
      *reinterpret_cast<uint2*>(x1) = make_uint2(o1[0], o1[1]);
      *reinterpret_cast<uint2*>(x1 + plane) = make_uint2(o2[0], o2[1]);
    }
  }
  if ((int)threadIdx.x < p.k) p.ws.hmax[(size_t)t * p.k + threadIdx.x] = 0u;
  if (threadIdx.x == 0) p.ws.hmax[(size_t)p.T * p.k + t] = 0u;
}

// pinv[sorted[r]] = r for every bucket position r (entries outside [0, T k)
// were flagged when the list was checked and are skipped here).
__global__ void k_pf_pinv(ExpertParams p) {
  const int n = p.T * p.k;
  for (int r = blockIdx.x * blockDim.x + threadIdx.x; r < n; r += gridDim.x * blockDim.x) {
    const int pr = __ldg(&p.sorted[r]);
    if (pr >= 0 && pr < n) p.ws.pinv[pr] = r;
  }
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

// Routed h rows [0, T k) (fp32, bucket order) as three E4M3 terms for the
// block-scaled down GEMM: with tau_r = 7 - floor(log2 max|h_r|), v = h * 2^tau_r
// has its largest magnitude in [128, 256); h1 = e4m3(v), h2 = e4m3(16 (v - h1)),
// h3 = e4m3(16 (16 (v - h1) - h2)), so v = h1 + h2 / 16 + h3 / 256 up to the
// rounding of h3: 12 significant bits (one more than f16) for every element
// that stays an E4M3 normal number through the terms, and an absolute error
// below 2^-18 (2^-25 of the row's maximum) for the others.  hscale[r] =
// 2^-tau_r.  A row holding an infinity or NaN (its maximum's bits at or above
// infinity) becomes NaN in every term (E4M3 has no infinity).  One warp per
// row; I % 128 == 0.
__device__ __forceinline__ uint32_t e4m3x2_bits(float lo, float hi) {
  unsigned short q;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(q) : "f"(hi), "f"(lo));
  return q;
}
__device__ __forceinline__ float2 e4m3x2_value(uint32_t q) {
  uint32_t f2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(f2) : "h"((unsigned short)q));
  return __half22float2(*reinterpret_cast<const __half2*>(&f2));
}
__global__ void __launch_bounds__(256) k_h_to_e4m3(ExpertParams p) {
  const int row = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  const int n = p.T * p.k, I = p.I;
  if (row >= n) return;
  const uint32_t m = p.ws.hmax[row];
  const int e = (int)((m >> 23) & 0xFFu);
  const bool bad = e == 0xFF;
  int tau = (m == 0u || bad) ? 0 : 7 - (e - 127);
  tau = tau > 126 ? 126 : (tau < -126 ? -126 : tau);
  const float up = __int_as_float((tau + 127) << 23);
  if (lane == 0) p.ws.hscale[row] = __int_as_float((127 - tau) << 23);
  const float* src = reinterpret_cast<const float*>(p.ws.h) + (size_t)row * I;
  uint8_t* d1 = p.ws.h8 + (size_t)row * I;
  uint8_t* d2 = d1 + (size_t)n * I;
  uint8_t* d3 = d2 + (size_t)n * I;
  for (int c = lane * 4; c < I; c += 128) {
    uint32_t o1 = 0x7F7F7F7Fu, o2 = 0x7F7F7F7Fu, o3 = 0x7F7F7F7Fu;
    if (!bad) {
      const float4 v4 = *reinterpret_cast<const float4*>(src + c);
      const float v[4] = {v4.x * up, v4.y * up, v4.z * up, v4.w * up};
      o1 = o2 = o3 = 0u;
#pragma unroll
      for (int pr = 0; pr < 2; ++pr) {
        const float a = v[2 * pr], b = v[2 * pr + 1];
        const uint32_t q1 = e4m3x2_bits(a, b);
        const float2 f1 = e4m3x2_value(q1);
        const float ra = (a - f1.x) * 16.f, rb = (b - f1.y) * 16.f;
        const uint32_t q2 = e4m3x2_bits(ra, rb);
        const float2 f2 = e4m3x2_value(q2);
        const uint32_t q3 = e4m3x2_bits((ra - f2.x) * 16.f, (rb - f2.y) * 16.f);
        o1 |= q1 << (16 * pr);
        o2 |= q2 << (16 * pr);
        o3 |= q3 << (16 * pr);
      }
    }
    *reinterpret_cast<uint32_t*>(d1 + c) = o1;
    *reinterpret_cast<uint32_t*>(d2 + c) = o2;
    *reinterpret_cast<uint32_t*>(d3 + c) = o3;
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
// Items are (expert, 128-row weight tile, token tile).  Routed items come
// first, active experts in ascending order, row tiles outer; then the shared
// expert's items when there is one.  The shared expert's token tiles hold up
// to 128 tokens, the routed items (block-scaled GEMMs) up to kPfNTileGu
// (gate/up) or kPfNTileDn (down).
struct PfItem {
  int shared;  // 1: the bf16 shared expert
  int e;       // routed expert
  int m0;      // first weight row
  int p0;      // routed: first bucket position; shared: first token
  int cnt;     // tokens in the tile (1..128)
  int hpos0;   // row of the tile's first token in h ([T*k + T][I])
};

// Item tables of both GEMMs, written once per call from the bucket layout
// (so each role reads an item with one load): for every active expert u its
// items [pref[u], pref[u+1]) in row-tile-major order, then the shared
// expert's items.  One warp per active expert.
__device__ __forceinline__ void pf_fill_items(const ExpertParams& p, const int32_t* pref, int4* items, int M, int u,
                                              int U, int ntile) {
  const int lane = threadIdx.x & 31;
  const int m_tiles = (M + kPfMTile - 1) / kPfMTile;
  if (u < U) {
    const int e = p.ws.act_e[u];
    const int b0 = p.offsets[e];
    const int n = p.offsets[e + 1] - b0;
    const int ntiles = (n + ntile - 1) / ntile;
    const int base = pref[u];
    const int count = ntiles * m_tiles;
    for (int local = lane; local < count; local += 32) {
      const int m = local / ntiles, nt = local - m * ntiles;
      items[base + local] = make_int4(e, m * kPfMTile, b0 + nt * ntile, min(ntile, n - nt * ntile));
    }
  } else if (p.sh_gate) {
    const int base = U > 0 ? pref[U] : 0;
    const int nts = (p.T + kPfNTile - 1) / kPfNTile;
    for (int local = lane; local < m_tiles * nts; local += 32) {
      const int m = local / nts, nt = local - m * nts;
      items[base + local] = make_int4(-1, m * kPfMTile, nt * kPfNTile, min(kPfNTile, p.T - nt * kPfNTile));
    }
  }
}

__global__ void __launch_bounds__(256) k_pf_items(ExpertParams p) {
  const int U = (int)p.ws.hdr->n_active;
  const int nwarps = (int)(gridDim.x * blockDim.x) >> 5;
  for (int w = (int)((blockIdx.x * blockDim.x + threadIdx.x) >> 5); w <= 2 * U + 1; w += nwarps) {
    if (w <= U)
      pf_fill_items(p, p.ws.act_pref_gu, p.ws.items_gu, p.I, w, U, kPfNTileGu);
    else
      pf_fill_items(p, p.ws.act_pref_dn, p.ws.items_dn, p.H, w - U - 1, U, kPfNTileDn);
  }
}

__device__ __forceinline__ PfItem pf_item(int item, const ExpertParams& p, const int4* items) {
  const int4 v = __ldg(&items[item]);
  PfItem it;
  it.shared = v.x < 0 ? 1 : 0;
  it.e = v.x < 0 ? 0 : v.x;
  it.m0 = v.y;
  it.p0 = v.z;
  it.cnt = v.w;
  it.hpos0 = v.x < 0 ? p.T * p.k + v.z : v.z;
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

// 64 E2M1 codes of one weight row (q0: elements 0-31 = MX block 2s, q1:
// elements 32-63 = block 2s + 1, scale bytes s0, s1) -> 32 f16x2 words in K
// order (word c holds elements 2c, 2c + 1), scaled by 2^(e - 127 + sigma):
// one exact conversion of two codes and one exact f16x2 multiply per word
// (the row shift keeps every product in the f16 normal range).
__device__ __forceinline__ void dq_row_mx(uint4 q0, uint4 q1, uint32_t s0, uint32_t s1, int sigma,
                                          uint32_t (&o)[32]) {
  uint32_t m0 = s0 == 255u ? 0x7E00u : f16_pow2((int)s0 - 127 + sigma);
  uint32_t m1 = s1 == 255u ? 0x7E00u : f16_pow2((int)s1 - 127 + sigma);
  m0 |= m0 << 16;
  m1 |= m1 << 16;
  const uint32_t w[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
#pragma unroll
  for (int wd = 0; wd < 8; ++wd)
#pragma unroll
    for (int bt = 0; bt < 4; ++bt) {
      const uint32_t c2 = e2m1x2_f16x2(w[wd], bt);
      asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(o[4 * wd + bt]) : "r"(c2), "r"(wd < 4 ? m0 : m1));
    }
}

// 64 bf16 weights of one row (eight 16-byte loads) -> 32 f16x2 words, scaled
// by `scale` (a power of two).
__device__ __forceinline__ void dq_row_bf16(const uint16_t* src, float scale, uint32_t (&o)[32]) {
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const uint4 v = ldg_stream(src + j * 8);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const __half2 h2 =
          __floats2half2_rn(__uint_as_float(w[i] << 16) * scale, __uint_as_float(w[i] & 0xFFFF0000u) * scale);
      o[4 * j + i] = *reinterpret_cast<const uint32_t*>(&h2);
    }
  }
}

// -------------------------------------------------------- CTA control --
struct PfShared {
  uint64_t a_full[kPfMaxStages];   // A stage written to TMEM: the GW warps of one dequant group
  uint64_t a_empty[kPfMaxStages];  // ... consumed: tcgen05.commit of each issuer
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

// Bounded wait that also gives up as soon as another role has aborted.
// Between polls the waiting warp sleeps for `backoff_ns` (nanosleep: it
// issues nothing meanwhile), so that waiting warps leave the issue slots to
// the warps doing work; the roles on the tensor core's critical path poll
// without sleeping, the others with longer sleeps the longer their waits
// usually are.
constexpr uint32_t kPfPollMma = 0, kPfPollDq = 32, kPfPollSig = 64, kPfPollLd = 128, kPfPollEp = 256;
__device__ __forceinline__ bool pf_wait(PfShared& sh, uint64_t* bar, uint32_t parity, WsHeader* hdr,
                                        uint32_t backoff_ns, long long limit) {
  const bool diag = limit < kWaitCycles;  // diagnostic limit: non-blocking probes (see mbar_wait_diag)
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

// Shared pipeline state of the four roles of one CTA.
struct PfCtx {
  PfShared* sh;
  uint8_t* smem_b;   // token tile ring, 1024-byte aligned
  uint8_t* raw;      // raw MXFP4 slots of the dequant groups
  int a_stages, b_stages;
  int n_items;       // routed + shared items
  int n_routed;
  int U;
  const int32_t* pref;
  const int4* items;  // this GEMM's item table
  int K, M, nslices;
  WsHeader* hdr;
  long long wait_limit;  // cycles before a wait on another role gives up
};

// All lanes of a warp wait; the warp proceeds only if every lane succeeded.
__device__ __forceinline__ bool pf_warp_wait(const PfCtx& c, uint64_t* bar, uint32_t parity, uint32_t backoff_ns) {
  const bool ok = pf_wait(*c.sh, bar, parity, c.hdr, backoff_ns, c.wait_limit);
  return __all_sync(0xFFFFFFFFu, ok);
}

// Claim the ring stage of global slice gs for writing (wait until its
// previous use was consumed by the tensor core).
__device__ __forceinline__ bool pf_claim(const PfCtx& c, uint64_t* empty, int nstages, int gs, uint32_t backoff_ns) {
  const int st = (int)((unsigned)gs % (unsigned)nstages), use = (int)((unsigned)gs / (unsigned)nstages);
  if (use == 0) return true;
  return pf_warp_wait(c, &empty[st], (use - 1) & 1, backoff_ns);
}

__device__ __forceinline__ void cp_async4(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}

// Row shift sigma of weight row `row` of matrix `a` (gate/down 0, up 1) of an
// item: routed MXFP4 rows from their E8M0 scales (sigma = 140 - max scale),
// shared-expert rows from the pre-pass; 0 for a row outside the matrix or an
// expert with a bad descriptor (flagged elsewhere, not read).
template <bool GATEUP>
__device__ __forceinline__ int pf_row_sigma(const ExpertParams& p, const PfCtx& c, const PfItem& it, int a,
                                            int row) {
  if (row >= c.M) return 0;
  if (it.shared) return __ldg(&p.ws.shsig[GATEUP ? (a == 0 ? row : p.I + row) : 2 * p.I + row]);
  const moe_expert ex = p.experts[it.e];
  if (!expert_ptrs_ok(ex)) return 0;
  const uint8_t* sc = GATEUP ? (a == 0 ? ex.gate.s : ex.up.s) : ex.down.s;
  return sigma_from_smax(row_smax_part(sc + (size_t)row * (c.K / 32), c.K / 128, 0, 1));
}

// Codes and scales of weight row m0 + r of matrix a of `item`; null unless it
// is a routed item with a valid row.
__device__ __forceinline__ const uint8_t* item_row_codes(const ExpertParams& p, const PfCtx& c, bool gateup, int item,
                                                         int r, int a, const uint8_t** scales) {
  if (item >= c.n_items) return nullptr;
  const PfItem it = pf_item(item, p, c.items);
  if (it.shared) return nullptr;
  const moe_expert ex = p.experts[it.e];
  const int row = it.m0 + r;
  if (row >= c.M || !expert_ptrs_ok(ex)) return nullptr;
  const moe_mx_mat m = a == 0 ? (gateup ? ex.gate : ex.down) : ex.up;
  if (scales) *scales = m.s + (size_t)row * (c.K / 32);
  return m.q + (size_t)row * (c.K / 2);
}

// Raw-copy cursor of a dequant thread (matrix a, row r): walks the CTA's
// global slice sequence g = ci * nslices + s (ci: the CTA's ci-th item) over
// the slices of its group (g = grp, grp + NG, ...) ahead of the conversion
// and issues one cp.async group per slice into the group's raw slots (an
// empty group for the shared expert or past the end, so group counts stay
// aligned with slices).  It also keeps the row streaming from DRAM in long
// runs: the row is prefetched into L2 in kPfL2Window-byte windows eight
// slices ahead, and the first 512 bytes of the next item's row near the end
// of the current item (the per-slice copies alone read 32 bytes per row,
// which DRAM serves poorly).
struct PfCursor {
  int g, ci;
  const uint8_t* q;   // codes of the row (null: no MXFP4 copy)
  const uint8_t* sw;  // scale row
};

__device__ __forceinline__ void cursor_enter(PfCursor& cur, const ExpertParams& p, const PfCtx& c, bool gateup,
                                             int r, int a) {
  cur.q = item_row_codes(p, c, gateup, blockIdx.x + cur.ci * (int)gridDim.x, r, a, &cur.sw);
}

template <bool GATEUP>
__device__ __forceinline__ void cursor_issue(PfCursor& cur, const ExpertParams& p, const PfCtx& c, int r, int a,
                                             int tid, uint8_t* raw, int j) {
  using C = PfCfg<GATEUP>;
  uint8_t* slot = raw + (size_t)(j % C::R) * C::kStage;
  const int ns = c.nslices;
  if (blockIdx.x + cur.ci * (int)gridDim.x < c.n_items) {
    const int s = cur.g - cur.ci * ns;
    const int rowbytes = c.K / 2;
    if (cur.q) {
      if ((s & 7) == 0) {
        const int off = (s + 8) * 32;
        if (off < rowbytes) prefetch_l2(cur.q + off, (uint32_t)min(kPfL2Window, rowbytes - off));
      }
      cp_async16(slot + tid * 16, cur.q + (size_t)s * 32);
      cp_async16(slot + C::kThreads * 16 + tid * 16, cur.q + (size_t)s * 32 + 16);
      cp_async4(slot + C::kQ + tid * 4, cur.sw + (s >> 1) * 4);
    }
    if (s >= ns - 16 && s < ns - 16 + C::NG) {
      const uint8_t* nq = item_row_codes(p, c, GATEUP, blockIdx.x + (cur.ci + 1) * (int)gridDim.x, r, a, nullptr);
      if (nq) prefetch_l2(nq, (uint32_t)min(512, rowbytes));
    }
    cur.g += C::NG;
    if (cur.g >= (cur.ci + 1) * ns) {
      cur.ci = cur.g / ns;
      cursor_enter(cur, p, c, GATEUP, r, a);
    }
  }
  cp_async_commit();
}

// Dequant warps.  Warp w is in group w / GW; inside its group it converts
// matrix a = (w % GW) / 4 (gate/down 0, up 1), TMEM lane quarter w % 4: thread
// (lane l) owns weight row m0 + 32 * (w % 4) + l of every item.  For each of
// its group's slices it converts the row's 64 elements of the slice into 32
// f16x2 columns and stores them into the slice's A stage in Tensor Memory
// (tcgen05.st, 32 lanes x 32 columns per warp), then signals the stage.
// Routed MXFP4 rows arrive through the group's raw slots (cp.async); the bf16
// shared expert's rows are loaded directly.
template <bool GATEUP>
__device__ void pf_dequant_role(const ExpertParams& p, const PfCtx& c, uint32_t tmem) {
  using C = PfCfg<GATEUP>;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int grp = warp / C::GW;
  const int a = (warp % C::GW) >> 2;
  const int quarter = warp & 3;
  const int r = quarter * 32 + lane;
  const int tid = threadIdx.x % C::kThreads;
  const int ns = c.nslices;
  PfShared& sh = *c.sh;
  uint8_t* raw = c.raw + (size_t)grp * C::R * C::kStage;
  const uint32_t tbase = tmem + ((uint32_t)(quarter * 32) << 16) + kPfAccCols + (uint32_t)(a * 32);
  PfCursor cur;
  cur.g = grp;
  cur.ci = grp / ns;
  cursor_enter(cur, p, c, GATEUP, r, a);
  for (int j = 0; j < C::R; ++j) cursor_issue<GATEUP>(cur, p, c, r, a, tid, raw, j);
  int ci_cur = -1;
  int sig_next = 0;  // next local item whose row-shift slot this warp consumes
  bool ok = true;
  PfItem it{};
  int sigma = 0;
  float bscale = 1.f;
  const uint16_t* wrow = nullptr;
  int ci = grp / ns, s = grp - (grp / ns) * ns;  // item (CTA-local) and slice of global slice g
  for (int g = grp, j = 0;; g += C::NG, ++j) {
    if (j > 0) {
      s += C::NG;
      while (s >= ns) {
        s -= ns;
        ++ci;
      }
    }
    const int item = blockIdx.x + ci * (int)gridDim.x;
    if (item >= c.n_items) break;
    if (ci != ci_cur) {
      ci_cur = ci;
      it = pf_item(item, p, c.items);
      // Row shifts of this item from the ring (and release of the slots of
      // items this group has no slice of).
      for (; sig_next <= ci && ok; ++sig_next) {
        const int slot = sig_next % kPfSigRing;
        if (!pf_warp_wait(c, &sh.sig_full[slot], (sig_next / kPfSigRing) & 1, kPfPollSig)) {
          ok = false;
          break;
        }
        if (sig_next == ci) sigma = sh.sig[slot][a][r];
        __syncwarp();
        if (lane == 0) mbar_arrive(&sh.sig_empty[slot]);
      }
      if (!ok) break;
      if (it.shared) {
        const int row = min(it.m0 + r, c.M - 1);
        const uint16_t* base = GATEUP ? (a == 0 ? p.sh_gate : p.sh_up) : p.sh_down;
        wrow = base + (size_t)row * c.K;
        bscale = __int_as_float((sigma + 127) << 23);
      }
    }
    cp_async_wait<C::R - 1>();  // this slice's group (empty for the shared expert)
    uint32_t o[32];
    if (!it.shared) {
      const uint8_t* rs = raw + (size_t)(j % C::R) * C::kStage;
      const uint4 q0 = lds128(rs + tid * 16);
      const uint4 q1 = lds128(rs + C::kThreads * 16 + tid * 16);
      const uint32_t sw = *reinterpret_cast<const uint32_t*>(rs + C::kQ + tid * 4) >> (16 * (s & 1));
      // A row not copied (bad descriptor: flagged) converts stale slot bytes;
      // the epilogue discards that row's outputs.
      dq_row_mx(q0, q1, sw & 0xFFu, (sw >> 8) & 0xFFu, sigma, o);
    } else {
      dq_row_bf16(wrow + (size_t)s * kPfSliceK, bscale, o);
    }
    if (!pf_claim(c, sh.a_empty, C::AS, g, kPfPollDq)) break;
    tc_fence_after();
    tmem_st32(tbase + (uint32_t)(((unsigned)g % C::AS) * C::ACOLS), o);
    tmem_st_wait();
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(&sh.a_full[(unsigned)g % C::AS]);
    cursor_issue<GATEUP>(cur, p, c, r, a, tid, raw, j + C::R);
    if (*(volatile int*)&sh.abort_flag) {
      ok = false;
      break;
    }
  }
  // Release the row-shift slots of the CTA's remaining items.
  const int n_local = blockIdx.x < c.n_items ? (c.n_items - blockIdx.x + gridDim.x - 1) / gridDim.x : 0;
  for (; ok && sig_next < n_local; ++sig_next) {
    const int slot = sig_next % kPfSigRing;
    if (!pf_warp_wait(c, &sh.sig_full[slot], (sig_next / kPfSigRing) & 1, kPfPollSig)) break;
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(&sh.sig_empty[slot]);
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
__device__ void pf_loader_role(const ExpertParams& p, const PfCtx& c, const CUtensorMap* tmap_h) {
  const int l = threadIdx.x - kPfDqWarps * 32;  // 0..127
  const int ns = c.nslices;
  if (!GATEUP) {
    // down: the token tile of slice s is the box (x = 64 s, y = hpos0) of the
    // f16 h rows, one tensor-map copy by the first loader thread; rows past
    // the end of h read as zero.
    if (l >= 32) return;
    constexpr int BS = PfCfg<GATEUP>::BS;
    int issued[BS];  // last use of each stage with a copy issued (-1: none)
#pragma unroll
    for (int i = 0; i < BS; ++i) issued[i] = -1;
    int gs = 0;
    bool ok = true;
    for (int item = blockIdx.x; item < c.n_items && ok; item += gridDim.x) {
      const PfItem it = pf_item(item, p, c.items);
      for (int s = 0; s < ns; ++s, ++gs) {
        if (!pf_claim(c, c.sh->b_empty, BS, gs, kPfPollLd)) {
          ok = false;
          break;
        }
        if (l == 0) {
          const int st = (int)((unsigned)gs % BS);
          uint64_t* bar = &c.sh->b_full[st];
          mbar_arrive_expect_tx(bar, (uint32_t)kPfTileBytes);
          tma_load_2d(c.smem_b + (size_t)st * kPfTileBytes, tmap_h, s * kPfSliceK, it.hpos0, bar);
#pragma unroll
          for (int i = 0; i < BS; ++i)
            if (i == st) issued[i] = (int)((unsigned)gs / BS);
        }
        __syncwarp();
      }
      if (*(volatile int*)&c.sh->abort_flag) ok = false;
    }
    // Every copy issued has landed before the CTA may exit (immediate after a
    // normal run: the MMA issuer waited for each of them).
    if (l == 0)
#pragma unroll
      for (int i = 0; i < BS; ++i)
        if (issued[i] >= 0 && !mbar_wait(&c.sh->b_full[i], issued[i] & 1)) set_status(c.hdr, MOE_ERR_TIMEOUT);
    return;
  }
  const int npairs = p.T * p.k;
  bool ok = true;
  int gbase = 0;
  for (int item = blockIdx.x; item < c.n_items && ok; item += gridDim.x, gbase += ns) {
    const PfItem it = pf_item(item, p, c.items);
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
      if (!pf_claim(c, c.sh->b_empty, PfCfg<GATEUP>::BS, gs, kPfPollLd)) {
        ok = false;
        break;
      }
      uint8_t* btile = c.smem_b + (size_t)((unsigned)gs % PfCfg<GATEUP>::BS) * kPfTileBytes;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        if (!use_chunk[j]) continue;
        if (src[j])
          cp_async16(btile + dst[j], src[j] + (size_t)s * kPfSliceK);
        else
          cp_async16_zfill(btile + dst[j], p.ws.xh, 0u);
      }
      cp_async_mbar_arrive(&c.sh->b_full[(unsigned)gs % PfCfg<GATEUP>::BS]);
    }
    if (*(volatile int*)&c.sh->abort_flag) ok = false;
  }
  cp_async_wait_all();
}

// Row shifts of local item j (the CTA's j-th item) into the shift ring, by
// the epilogue warps (thread = one weight row).
template <bool GATEUP>
__device__ __forceinline__ bool pf_publish_sig(const ExpertParams& p, const PfCtx& c, int j) {
  PfShared& sh = *c.sh;
  const int slot = j % kPfSigRing, use = j / kPfSigRing;
  if (use > 0 && !pf_warp_wait(c, &sh.sig_empty[slot], (use - 1) & 1, kPfPollSig)) return false;
  const int item = blockIdx.x + j * gridDim.x;
  const PfItem it = pf_item(item, p, c.items);
  const int rl = ((threadIdx.x >> 5) & 3) * 32 + (threadIdx.x & 31);
  const int row = it.m0 + rl;
  sh.sig[slot][0][rl] = pf_row_sigma<GATEUP>(p, c, it, 0, row);
  sh.sig[slot][1][rl] = GATEUP ? pf_row_sigma<GATEUP>(p, c, it, 1, row) : 0;
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(&sh.sig_full[slot]);
  return true;
}

// Epilogue warps: warp q (= warp % 4) reads TMEM lanes 32q..32q+31, i.e.
// weight rows m0 + 32q + lane, one fp32 column per token.
//   gate/up: h[hpos0 + n][row] = silu(g) * u in fp32, shifts removed, and the
//            largest |h| of each h row raised into hmax;
//   down:    out[token(n)][row] += weight(n) * 2^-tau(n) * y.
// Before each item they publish the row shifts of the item kPfSigRing - 1
// places ahead, so the dequant warps never wait on the scale reads.
template <bool GATEUP>
__device__ void pf_epilogue_role(const ExpertParams& p, const PfCtx& c, uint32_t tmem) {
  using C = PfCfg<GATEUP>;
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
    const PfItem it = pf_item(item, p, c.items);
    const int b = ci % C::ACCB, use = ci / C::ACCB;
    const int rl = q * 32 + lane;
    const int row = it.m0 + rl;
    bool valid = row < c.M;
    if (!it.shared) valid = valid && expert_ptrs_ok(p.experts[it.e]);
    const int slot = ci % kPfSigRing;
    if (!pf_warp_wait(c, &sh.sig_full[slot], (ci / kPfSigRing) & 1, kPfPollSig)) break;
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
    if (!pf_warp_wait(c, &sh.accf[b], use & 1, kPfPollEp)) break;
    tc_fence_after();
    const uint32_t tbase = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(b * C::ACCW);
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
          uint32_t av = 0u;
          if (valid && n < it.cnt) {
            const float xs = col_scale[n];
            const float gv = __uint_as_float(g[i]) * rs0 * xs;
            const float uv = __uint_as_float(u[i]) * rs1 * xs;
            const float hv = silu_f32(gv) * uv;
            hout[(size_t)(it.hpos0 + n) * p.I + row] = hv;
            av = __float_as_uint(hv) & 0x7FFFFFFFu;
          }
          const uint32_t mx = __reduce_max_sync(0xFFFFFFFFu, av);
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
// item, wait for a free accumulator buffer, then per slice for the A stage
// (Tensor Memory) and the token tile (shared memory), issue 4 K = 16 MMAs
// M = 128 x N = round16(tokens) with A read from Tensor Memory into
// accumulator `which` (gate/up: matrix `which`; down: the item's buffer), and
// release both stages with tcgen05.commit; each issuer's last commit of the
// item counts towards the accumulator being ready.
template <bool GATEUP>
__device__ void pf_mma_role(const ExpertParams& p, const PfCtx& c, uint32_t tmem, int which) {
  using C = PfCfg<GATEUP>;
  if (which >= C::NI) return;
  constexpr int MPT = C::NA / C::NI;  // matrices this issuer covers
  PfShared& sh = *c.sh;
  const int ns = c.nslices;
  int ci = 0;
  for (int item = blockIdx.x; item < c.n_items; item += gridDim.x, ++ci) {
    const PfItem it = pf_item(item, p, c.items);
    const int b = ci % C::ACCB, use = ci / C::ACCB;
    if (use >= 1 && !pf_wait(sh, &sh.acce[b], (use - 1) & 1, c.hdr, kPfPollMma, c.wait_limit)) break;
    tc_fence_after();
    const int nmma = (it.cnt + 15) & ~15;
    const uint32_t idesc = idesc_f16_f32(kPfMTile, nmma);
    const uint32_t dcol = tmem + (uint32_t)(b * C::ACCW + which * MPT * 128);
    bool ok = true;
    bool first = true;
    for (int s = 0; s < ns; ++s) {
      const int gs = ci * ns + s;
      const unsigned ug = (unsigned)gs;
      const int sa = (int)(ug % C::AS), sb = (int)(ug % C::BS);
      if (!pf_wait(sh, &sh.a_full[sa], (ug / C::AS) & 1, c.hdr, kPfPollMma, c.wait_limit) ||
          !pf_wait(sh, &sh.b_full[sb], (ug / C::BS) & 1, c.hdr, kPfPollMma, c.wait_limit)) {
        ok = false;
        break;
      }
      if (GATEUP) fence_async_smem();  // the token tile was written by cp.async (generic proxy)
      tc_fence_after();
      const uint32_t acol = tmem + kPfAccCols + (uint32_t)(sa * C::ACOLS + which * MPT * 32);
      const uint32_t bbase = smem_u32(c.smem_b + (size_t)sb * kPfTileBytes);
#pragma unroll
      for (int kk = 0; kk < kPfSliceK / 16; ++kk)
#pragma unroll
        for (int m = 0; m < MPT; ++m)
          umma_f16_ts(dcol + (uint32_t)(m * 128), acol + (uint32_t)(m * 32 + kk * 8), sdesc_sw128(bbase + kk * 32),
                      idesc, (first && kk == 0) ? 0u : 1u);
      first = false;
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
    if (!mbar_wait(&sh.accf[last % C::ACCB], (last / C::ACCB) & 1)) set_status(c.hdr, MOE_ERR_TIMEOUT);
  }
}

// Persistent grouped GEMM, one CTA per SM.  GATEUP: A = gate and up rows (M =
// I), K = H, B = f16 activations; else A = down rows (M = H), K = I, B = h.
template <bool GATEUP>
__global__ void __launch_bounds__(kPfThreads, 1) k_pf_gemm(ExpertParams p, const __grid_constant__ CUtensorMap tmap_h) {
  using C = PfCfg<GATEUP>;
  extern __shared__ uint8_t pf_dyn[];
  __shared__ PfShared sh;
  const int warp = threadIdx.x >> 5;
  if (warp == kPfMmaWarp) {
    tmem_alloc(&sh.tmem_base, kPfTmemCols);
    tmem_relinquish();
  }
  if (threadIdx.x == 0) {
    // gate/up: both issuers read every stage; down: one issuer.
    for (int s = 0; s < C::AS; ++s) {
      mbar_init(&sh.a_full[s], C::GW);
      mbar_init(&sh.a_empty[s], C::NI);
    }
    for (int s = 0; s < C::BS; ++s) {
      mbar_init(&sh.b_full[s], GATEUP ? kPfLdWarps * 32 : 1);
      mbar_init(&sh.b_empty[s], C::NI);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sh.accf[b], C::NI);
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
  c.smem_b = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(pf_dyn) + 1023) & ~(uintptr_t)1023);
  c.a_stages = C::AS;
  c.b_stages = C::BS;
  c.raw = c.smem_b + (size_t)C::BS * kPfTileBytes;
  c.K = GATEUP ? p.H : p.I;
  c.M = GATEUP ? p.I : p.H;
  c.nslices = c.K / kPfSliceK;
  c.hdr = p.ws.hdr;
  c.wait_limit = p.wait_limit;
  c.U = (int)p.ws.hdr->n_active;
  c.pref = GATEUP ? p.ws.act_pref_gu : p.ws.act_pref_dn;
  c.items = GATEUP ? p.ws.items_gu : p.ws.items_dn;
  c.n_routed = c.U > 0 ? __ldg(&c.pref[c.U]) : 0;
  const int m_tiles = (c.M + kPfMTile - 1) / kPfMTile;
  c.n_items = c.n_routed + (p.sh_gate ? m_tiles * ((p.T + kPfNTile - 1) / kPfNTile) : 0);
  if (p.shared_only) {
    // The shared expert's items alone (its routed items run elsewhere, or
    // there are none).
    c.items += c.n_routed;
    c.n_items -= c.n_routed;
    c.n_routed = 0;
  }

  if (warp < kPfDqWarps)
    pf_dequant_role<GATEUP>(p, c, tmem);
  else if (warp < kPfDqWarps + kPfLdWarps)
    pf_loader_role<GATEUP>(p, c, &tmap_h);
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

// ------------------------------------------------ block-scaled expert GEMMs --
// The tensor core takes the MXFP4 weights as they are stored: tcgen05.mma
// kind::mxf8f6f4 with A = E2M1 codes and their E8M0 block scales, and B = the
// activations as E4M3 terms in bucket order: for gate/up the token rows as two
// terms (k_x_to_e4m3, x * 2^tau = x1 + x2 / 16, exact for bf16), for down the
// h rows as three (k_h_to_e4m3, h * 2^tau ~ h1 + h2 / 16 + h3 / 256, 12
// significant bits).  The terms enter with constant block scales 2^0, 2^-4,
// 2^-8.  Products are exact and accumulate in fp32 in Tensor Memory; nothing
// is converted on CUDA cores and no operand passes through registers.  Work
// items are those of k_pf_gemm (routed experts only).  Per 128-element slice
// of the contraction (four MX blocks):
//   * one producer thread loads the 128 weight rows of each matrix with one
//     tensor-map copy (4-bit elements in the 16-codes-then-8-byte-gap layout
//     the MMA reads, 128-byte swizzle; per-expert maps written by
//     k_pf_mx_maps) and the item's activation rows of all terms, contiguous
//     in bucket order, as one box of rows x terms (the box height is the token
//     count rounded up to 32: one of four maps);
//   * 4 scale warps (one per TMEM lane quarter) write the rows' scale words
//     (4 bytes = the slice's four blocks) into the stage's scale columns;
//   * two threads issue the MMAs (K-steps x terms, M = 128, N =
//     round16(tokens), K = 32; the terms share one read of A through the A
//     collector), each into its own accumulator (gate/up: one matrix each;
//     down: two of the four K-steps each), and release the stage with
//     tcgen05.commit: a block-scaled MMA costs its issuing thread about 60
//     cycles whatever N is (4096-token workload: gate/up 3.58 -> 2.74 ms,
//     down 2.93 -> 2.65 ms with the second issuer);
//   * 4 epilogue warps read one of two accumulator buffers while the MMAs fill
//     the other: gate/up apply SwiGLU with the token's 2^-tau and store h in
//     fp32 (with each h row's largest |h|); down adds w * 2^-tau * y into out
//     with fp32 atomics.
// Code matrices must be 32-byte aligned for their tensor maps (checked: an
// expert whose codes are not is flagged and skipped).
namespace mxk {
constexpr int kSliceK = 128;
constexpr int kMaxStages = 4;
constexpr int kTile = 128 * 128;                // one 128-row operand tile (bytes)
constexpr int kCodeTx = 128 * 64;                // bytes a code tile's copy delivers (4-bit codes)
constexpr int kXBox = 32;                        // granule of the activation box heights
constexpr int kXMaps = 4;                        // box heights 32, 64, 96, 128
constexpr int kTmaWarp = 1;                      // warp 0: MMA issuer, owns TMEM
constexpr int kSfWarp0 = 2, kSfWarps = 4;        // warps 2-5
constexpr int kEpWarp0 = kSfWarp0 + kSfWarps, kEpWarps = 4;  // warps 6-9
constexpr int kMma2Warp = kEpWarp0 + kEpWarps;                 // warp 10: gate/up's second issuer (up)
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kPollMma = 0, kPollTma = 32, kPollSf = 64, kPollEp = 256;
}  // namespace mxk

// Per GEMM: a stage holds the NA weight tiles and an activation box of up to
// N rows (rounded up to 32) of each of the NT terms (gate/up: N = 112, three
// 64 KB stages; down: N = 96, four 52 KB stages; a fourth gate/up stage with
// 96-token tiles was slower, more items outweighing the deeper ring).  Two
// threads issue the MMAs, each into an accumulator of its own: gate/up one
// matrix each, down two of a slice's four K-steps each (the epilogue adds the
// two).  TMEM columns: two buffers of AccW columns (accumulator i at i * N of
// the buffer); the terms' constant scales (4 columns each) at ColSfb; the
// weight scales of stage st, matrix a at ColSfa + 4 (NA st + a).
template <bool GU>
struct MxCfg {
  static constexpr int NA = GU ? 2 : 1;                   // weight matrices per item
  static constexpr int NT = GU ? 2 : 3;                   // activation terms
  static constexpr int N = GU ? kPfNTileGu : kPfNTileDn;  // tokens per tile (at most)
  static constexpr int XROWS = (N + mxk::kXBox - 1) / mxk::kXBox * mxk::kXBox;
  static constexpr int STAGE = NA * mxk::kTile + NT * XROWS * 128;
  static constexpr int STAGES = GU ? 3 : 4;
  // MMA-issuing threads, one accumulator each (four gate/up issuers, which
  // leave room for a single accumulator buffer only, were slower: 2.79 ->
  // 3.29 ms on the 4096-token workload).
  static constexpr int NI = 2;
  static constexpr int ACCB = NI * N * 2 + 4 * NT + 4 * NA * STAGES <= 512 ? 2 : 1;  // accumulator buffers
  static constexpr int KB = 4 * NA / NI;                  // K-steps of a slice per issuer
  static constexpr int THREADS = (mxk::kMma2Warp + NI - 1) * 32;
  static constexpr uint32_t AccW = NI * N;
  static constexpr uint32_t ColSfb = ACCB * AccW;
  static constexpr uint32_t ColSfa = ColSfb + 4 * NT;
  static_assert(ColSfa + 4 * NA * STAGES <= mxk::kTmemCols, "TMEM columns");
  static_assert(STAGES <= mxk::kMaxStages && STAGE % 1024 == 0, "stages");
};

template <bool GU>
struct MxShared {
  uint64_t full[mxk::kMaxStages];   // stage filled: producer (with the copies' bytes) + 4 scale warps
  uint64_t empty[mxk::kMaxStages];  // stage consumed: tcgen05.commit
  uint64_t accf[2];                 // accumulator buffer ready: tcgen05.commit
  uint64_t acce[2];                 // accumulator buffer drained: 4 epilogue warps
  uint32_t tmem_base;
  int abort_flag;
  float col_scale[mxk::kEpWarps][MxCfg<GU>::N];       // per epilogue warp: factor of each column
  int col_tok[mxk::kEpWarps][GU ? 1 : MxCfg<GU>::N];  // per epilogue warp: token of each column (down)
};

// Maps of the bucket-order activation rows of all terms, one per box height.
struct MxXMaps {
  CUtensorMap m[mxk::kXMaps];
};

template <bool GU>
struct MxCtx {
  MxShared<GU>* sh;
  uint8_t* ring;  // STAGES x STAGE bytes, 1024-byte aligned
  int n_items;
  const int4* items;
  int ns;         // slices per item
  int srow;       // scale bytes per weight row (K / 32)
  WsHeader* hdr;
  long long wait_limit;
};

template <bool GU>
__device__ __forceinline__ bool mx_wait(const MxCtx<GU>& c, uint64_t* bar, uint32_t parity, uint32_t backoff_ns) {
  MxShared<GU>& sh = *c.sh;
  const bool diag = c.wait_limit < kWaitCycles;
  if (diag ? mbar_test_wait(bar, parity) : mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  for (;;) {
    if (backoff_ns) __nanosleep(backoff_ns);
    if (diag ? mbar_test_wait(bar, parity) : mbar_try_wait(bar, parity)) return true;
    if (*(volatile int*)&sh.abort_flag) return false;
    if (clock64() - t0 > c.wait_limit) {
      set_status(c.hdr, MOE_ERR_TIMEOUT);
      *(volatile int*)&sh.abort_flag = 1;
      return false;
    }
  }
}
template <bool GU>
__device__ __forceinline__ bool mx_warp_wait(const MxCtx<GU>& c, uint64_t* bar, uint32_t parity, uint32_t backoff_ns) {
  const bool ok = mx_wait(c, bar, parity, backoff_ns);
  return __all_sync(0xFFFFFFFFu, ok);
}
// Wait until ring stage gs % STAGES is free for global slice gs.
template <bool GU>
__device__ __forceinline__ bool mx_claim(const MxCtx<GU>& c, int gs, uint32_t backoff_ns) {
  constexpr int S = MxCfg<GU>::STAGES;
  const int st = gs % S, use = gs / S;
  if (use == 0) return true;
  return mx_warp_wait(c, &c.sh->empty[st], (use - 1) & 1, backoff_ns);
}

// Code matrices of one GEMM usable by the tensor-map copies.
template <bool GU>
__device__ __forceinline__ bool mx_codes_ok(const moe_expert& ex) {
  const uintptr_t q = GU ? ((uintptr_t)ex.gate.q | (uintptr_t)ex.up.q) : (uintptr_t)ex.down.q;
  return expert_ptrs_ok(ex) && (q & 31u) == 0;
}
// Scale matrix a of an expert in one GEMM.
template <bool GU>
__device__ __forceinline__ const uint8_t* mx_scales(const moe_expert& ex, int a) {
  return GU ? (a == 0 ? ex.gate.s : ex.up.s) : ex.down.s;
}

// Tensor maps of the active experts' codes, [E][3] (gate, up, down): the
// templates (gate/up: dims H x I, row stride H / 2 bytes; down: I x H, I / 2;
// boxes of 128 elements x 128 rows, 4-bit elements with 8-byte gaps, 128-byte
// swizzle) with the expert's address.  Experts whose codes cannot be mapped
// are flagged (MOE_ERR_DEVICE_CHECK) and get no map; the GEMMs skip their
// copies.  One thread per (active expert, matrix).
__global__ void k_pf_mx_maps(ExpertParams p, const __grid_constant__ CUtensorMap tmpl_gu,
                             const __grid_constant__ CUtensorMap tmpl_dn) {
  const int U = (int)p.ws.hdr->n_active;
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < 3 * U; i += gridDim.x * blockDim.x) {
    const int e = __ldg(&p.ws.act_e[i / 3]), a = i % 3;
    const moe_expert ex = p.experts[e];
    const uint8_t* q = a == 0 ? ex.gate.q : (a == 1 ? ex.up.q : ex.down.q);
    if (!expert_ptrs_ok(ex) || ((uintptr_t)q & 31u) != 0) {
      set_status(p.ws.hdr, MOE_ERR_DEVICE_CHECK);
      continue;
    }
    uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<uint8_t*>(p.ws.tmaps) + (size_t)(3 * e + a) * 128);
    const uint4* src = reinterpret_cast<const uint4*>(a < 2 ? &tmpl_gu : &tmpl_dn);
#pragma unroll
    for (int j = 0; j < 8; ++j) dst[j] = src[j];
    asm volatile("tensormap.replace.tile.global_address.global.b1024.b64 [%0], %1;" ::"l"(dst), "l"(q) : "memory");
    asm volatile("fence.proxy.tensormap::generic.release.gpu;" ::: "memory");
  }
}

constexpr int kMxAhead = 4;
// Producer warp.  Per slice: claim the stage; lane 0 arms the stage's barrier
// with the bytes of all copies and issues the code-tile copies and the
// activation box (rows past the item's tokens belong to the next bucket or
// read as zero: they only feed accumulator columns that the epilogue
// ignores).  Its lane issues nothing else: the copy unit's queue is what the
// tensor core waits on.
template <bool GU>
__device__ void mx_producer_role(const ExpertParams& p, const MxCtx<GU>& c, const MxXMaps* xmaps) {
  using C = MxCfg<GU>;
  const int lane = threadIdx.x & 31;
  MxShared<GU>& sh = *c.sh;
  int gs = 0;
  bool ok = true;
  constexpr int S = C::STAGES;
  int issued[S];  // last use of each stage with copies issued (-1: none)
#pragma unroll
  for (int i = 0; i < S; ++i) issued[i] = -1;
  for (int item = blockIdx.x; item < c.n_items && ok; item += gridDim.x) {
    const PfItem it = pf_item(item, p, c.items);
    const moe_expert ex = p.experts[it.e];
    const bool wok = mx_codes_ok<GU>(ex);
    const int nbox = (it.cnt + mxk::kXBox - 1) / mxk::kXBox;  // box height / 32
    const CUtensorMap* xmap = &xmaps->m[nbox - 1];
    const uint8_t* maps = reinterpret_cast<const uint8_t*>(p.ws.tmaps) + (size_t)(3 * it.e + (GU ? 0 : 2)) * 128;
    if (wok && lane == 0)
#pragma unroll
      for (int a = 0; a < C::NA; ++a) tmap_acquire(maps + a * 128);
    const uint32_t tx =
        (wok ? (uint32_t)C::NA * mxk::kCodeTx : 0u) + (uint32_t)(C::NT * nbox * mxk::kXBox) * mxk::kSliceK;
    for (int s = 0; s < c.ns; ++s, ++gs) {
      if (!mx_claim(c, gs, mxk::kPollTma)) {
        ok = false;
        break;
      }
      if (lane == 0) {
        const int st = gs % S;
        uint8_t* sb = c.ring + (size_t)st * C::STAGE;
        uint64_t* bar = &sh.full[st];
        mbar_arrive_expect_tx(bar, tx);
        if (wok)
#pragma unroll
          for (int a = 0; a < C::NA; ++a)
            tma_load_2d(sb + a * mxk::kTile, maps + a * 128, s * mxk::kSliceK, it.m0, bar);
        tma_load_3d(sb + C::NA * mxk::kTile, xmap, s * mxk::kSliceK, it.hpos0, 0, bar);
        // The code boxes kMxAhead slices on into L2 (they come from DRAM).
        if (wok && s + kMxAhead < c.ns)
#pragma unroll
          for (int a = 0; a < C::NA; ++a) tma_prefetch_2d(maps + a * 128, (s + kMxAhead) * mxk::kSliceK, it.m0);
#pragma unroll
        for (int i = 0; i < S; ++i)
          if (i == st) issued[i] = gs / S;
      }
      __syncwarp();
    }
    if (*(volatile int*)&sh.abort_flag) ok = false;
  }
  // Every copy issued has landed before the CTA may exit (immediate after a
  // normal run: the MMA issuer waited for each of them).
  if (lane == 0)
#pragma unroll
    for (int i = 0; i < S; ++i)
      if (issued[i] >= 0 && !mbar_wait(&sh.full[i], issued[i] & 1)) set_status(c.hdr, MOE_ERR_TIMEOUT);
}

// Scale warps: warp quarter q writes, in lanes 32q..32q+31, the terms'
// constant scales once, then per slice the scale words of rows lane + 32 j
// (j = 0..3) of each matrix into the stage's columns (the same words in every
// quarter).  An expert that is skipped gets scale 1 (its rows are discarded by
// the epilogue).  A slice reads 4 bytes of each scale row, so the words are
// loaded kSfAhead slices ahead into a register ring, and the rows are
// prefetched into L2 when an item starts (and the next item's halfway
// through).
constexpr int kSfAhead = 4;
template <bool GU>
__device__ __forceinline__ void mx_prefetch_scale_rows(const ExpertParams& p, const MxCtx<GU>& c, int item, int r) {
  using C = MxCfg<GU>;
  if (item >= c.n_items) return;
  const PfItem it = pf_item(item, p, c.items);
  const moe_expert ex = p.experts[it.e];
  if (!mx_codes_ok<GU>(ex)) return;
#pragma unroll
  for (int a = 0; a < C::NA; ++a) {
    const uint8_t* row = mx_scales<GU>(ex, a) + (size_t)(it.m0 + r) * c.srow;
    for (int o = 0; o < c.srow; o += 128) prefetch_l2_line(row + o);
    prefetch_l2_line(row + c.srow - 1);
  }
}

template <bool GU>
__device__ void mx_scale_role(const ExpertParams& p, const MxCtx<GU>& c, uint32_t tmem) {
  using C = MxCfg<GU>;
  constexpr int NW = 4 * C::NA;  // scale words a lane writes per slice
  const int q = (threadIdx.x >> 5) & 3, lane = threadIdx.x & 31;
  const uint32_t lbase = tmem + ((uint32_t)(q * 32) << 16);
#pragma unroll
  for (int j = 0; j < C::NT; ++j) {
    const uint32_t v = (uint32_t)(127 - 4 * j) * 0x01010101u;  // 2^(-4 j)
    tmem_st4(lbase + C::ColSfb + 4 * j, v, v, v, v);
  }
  const size_t jstride = 32 * (size_t)c.srow / 4;  // words between rows lane and lane + 32
  int gs = 0;
  bool ok = true;
  mx_prefetch_scale_rows<GU>(p, c, blockIdx.x, q * 32 + lane);
  for (int item = blockIdx.x; item < c.n_items && ok; item += gridDim.x) {
    const PfItem it = pf_item(item, p, c.items);
    const moe_expert ex = p.experts[it.e];
    const bool wok = mx_codes_ok<GU>(ex);
    const uint32_t* sp[C::NA];
#pragma unroll
    for (int a = 0; a < C::NA; ++a)
      sp[a] = wok ? reinterpret_cast<const uint32_t*>(mx_scales<GU>(ex, a) + (size_t)(it.m0 + lane) * c.srow)
                  : nullptr;
    // Words of slice sl: w[4 a + j] = row lane + 32 j of matrix a.
    auto load = [&](uint32_t (&w)[NW], int sl) {
#pragma unroll
      for (int a = 0; a < C::NA; ++a)
#pragma unroll
        for (int j = 0; j < 4; ++j) w[4 * a + j] = (wok && sl < c.ns) ? __ldg(sp[a] + j * jstride + sl) : 0x7F7F7F7Fu;
    };
    uint32_t ring[kSfAhead][NW];
#pragma unroll
    for (int i = 0; i < kSfAhead; ++i) load(ring[i], i);
    for (int s0 = 0; s0 < c.ns && ok; s0 += kSfAhead) {
#pragma unroll
      for (int i = 0; i < kSfAhead; ++i) {
        const int s = s0 + i;
        if (s >= c.ns) break;
        if (s == c.ns / 2) mx_prefetch_scale_rows<GU>(p, c, item + gridDim.x, q * 32 + lane);
        if (!mx_claim(c, gs, mxk::kPollSf)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const int st = gs % C::STAGES;
#pragma unroll
        for (int a = 0; a < C::NA; ++a)
          tmem_st4(lbase + C::ColSfa + 4 * (C::NA * st + a), ring[i][4 * a], ring[i][4 * a + 1], ring[i][4 * a + 2],
                   ring[i][4 * a + 3]);
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&c.sh->full[st]);
        ++gs;
        load(ring[i], s + kSfAhead);
      }
    }
    if (*(volatile int*)&c.sh->abort_flag) ok = false;
  }
  tmem_st_wait();
}

// MMA issuer (lane 0 of warp 0): per item, wait for its accumulator buffer
// (item parity) to be drained, then per slice for the stage, issue the MMAs
// and commit the stage; after the last slice commit the buffer.  The operands
// were written by tensor-map copies (async proxy), so no proxy fence is
// needed.
template <bool GU>
__device__ void mx_mma_role(const ExpertParams& p, const MxCtx<GU>& c, uint32_t tmem, int which) {
  using C = MxCfg<GU>;
  // Issuer `which` takes matrix which / (NI / NA) and KB consecutive K-steps
  // of each slice, into accumulator `which`.
  constexpr int KB = C::KB;
  const int a = which / (C::NI / C::NA);
  const int kb0 = (which % (C::NI / C::NA)) * KB;
  MxShared<GU>& sh = *c.sh;
  int ci = 0, gs = 0;
  for (int item = blockIdx.x; item < c.n_items; item += gridDim.x, ++ci) {
    const PfItem it = pf_item(item, p, c.items);
    const int b = ci % C::ACCB, use = ci / C::ACCB;
    if (use >= 1 && !mx_wait(c, &sh.acce[b], (use - 1) & 1, mxk::kPollMma)) break;
    tc_fence_after();
    const int nmma = (it.cnt + 15) & ~15;
    const uint32_t ibase = idesc_mx_f32(kPfMTile, nmma, kMxE2M1, kMxE4M3, 0, 0);
    // Term j's rows start j box heights x 128 bytes into the activation box.
    const uint32_t xstep = (uint32_t)((it.cnt + mxk::kXBox - 1) / mxk::kXBox) * mxk::kXBox * 128;
    bool ok = true;
    for (int s = 0; s < c.ns; ++s, ++gs) {
      const int st = gs % C::STAGES;
      if (!mx_wait(c, &sh.full[st], (gs / C::STAGES) & 1, mxk::kPollMma)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t sbase = smem_u32(c.ring + (size_t)st * C::STAGE);
      const uint32_t xbase = sbase + C::NA * mxk::kTile;
      const uint32_t d = tmem + (uint32_t)b * C::AccW + (uint32_t)(which * C::N);
      const uint32_t sfa = tmem + C::ColSfa + (uint32_t)(4 * (C::NA * st + a));
#pragma unroll
      for (int i = 0; i < KB; ++i) {
        const int kb = kb0 + i;
        const uint32_t idesc = ibase | ((uint32_t)kb << 29) | ((uint32_t)kb << 4);
        const uint64_t ad = sdesc_sw128(sbase + a * mxk::kTile + 32 * kb);
#pragma unroll
        for (int j = 0; j < C::NT; ++j) {
          const uint64_t bd = sdesc_sw128(xbase + j * xstep + 32 * kb);
          const uint32_t sfb = tmem + C::ColSfb + 4u * j;
          if (j == 0)
            umma_mx_fill(d, ad, bd, idesc, sfa, sfb, (s > 0 || i > 0) ? 1u : 0u);
          else if (j < C::NT - 1)
            umma_mx_use(d, ad, bd, idesc, sfa, sfb, 1u);
          else
            umma_mx_lastuse(d, ad, bd, idesc, sfa, sfb, 1u);
        }
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
  if (ci > 0 && !mbar_wait(&sh.accf[(ci - 1) % C::ACCB], ((ci - 1) / C::ACCB) & 1))
    set_status(c.hdr, MOE_ERR_TIMEOUT);
}

// Epilogue warps: warp q reads TMEM lanes 32q..32q+31 (weight rows m0 + 32q +
// lane).
//   gate/up: h[hpos0 + n][row] = silu(g) * u with both scaled by the token's
//            2^-tau, in fp32, raising each h row's largest |h| into hmax;
//   down:    out[token(n)][row] += w(n) * 2^-tau(n) * y.
// A row with a NaN block scale (E8M0 code 255) gives NaN, as the definition
// of the format has it (checked here, while the item's MMAs run).
template <bool GU>
__device__ void mx_epilogue_role(const ExpertParams& p, const MxCtx<GU>& c, uint32_t tmem) {
  using C = MxCfg<GU>;
  MxShared<GU>& sh = *c.sh;
  const int q = (threadIdx.x >> 5) & 3, lane = threadIdx.x & 31;
  const int npairs = p.T * p.k;
  const int nsw = c.srow / 4;  // scale words per row
  float* hout = reinterpret_cast<float*>(p.ws.h);
  int ci = 0;
  for (int item = blockIdx.x; item < c.n_items; item += gridDim.x, ++ci) {
    const PfItem it = pf_item(item, p, c.items);
    const int row = it.m0 + q * 32 + lane;
    const moe_expert ex = p.experts[it.e];
    const bool valid = mx_codes_ok<GU>(ex);
    bool nan_row = false;
    if (valid) {
      uint32_t any = 0u;
#pragma unroll
      for (int a = 0; a < C::NA; ++a) {
        const uint32_t* sr = reinterpret_cast<const uint32_t*>(mx_scales<GU>(ex, a) + (size_t)row * c.srow);
#pragma unroll 8
        for (int i = 0; i < nsw; ++i) {
          const uint32_t w = __ldg(sr + i);
          // A byte equal to 0xFF: all of its bits set (per-byte test without carries).
          any |= (w & (w >> 1) & (w >> 2) & (w >> 3) & (w >> 4) & (w >> 5) & (w >> 6) & (w >> 7)) & 0x01010101u;
        }
      }
      nan_row = any != 0u;
    }
    float* col_scale = sh.col_scale[q];
    int* col_tok = sh.col_tok[q];
    __syncwarp();
    for (int n = lane; n < it.cnt; n += 32) {
      int pr = __ldg(&p.sorted[it.p0 + n]);
      if (pr < 0 || pr >= npairs) pr = 0;  // flagged when the list was checked
      const int t = pr / p.k;
      if (GU) {
        col_scale[n] = __ldg(&p.ws.x8scale[t]);
      } else {
        col_tok[n] = t;
        col_scale[n] = __ldg(&p.w[pr]) * __ldg(&p.ws.hscale[it.hpos0 + n]);
      }
    }
    __syncwarp();
    const int b = ci % C::ACCB;
    if (!mx_warp_wait(c, &sh.accf[b], (ci / C::ACCB) & 1, mxk::kPollEp)) break;
    tc_fence_after();
    const uint32_t tbase = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)b * C::AccW;
    constexpr int PER = C::NI / C::NA;  // accumulators per matrix (added here)
    for (int c0 = 0; c0 < it.cnt; c0 += 16) {
      uint32_t g[16];
      tmem_ld16(tbase + (uint32_t)c0, g);
      if (GU) {
        uint32_t u[16];
        tmem_ld16(tbase + (uint32_t)(PER * C::N) + (uint32_t)c0, u);
        if (PER == 2) {
          uint32_t g2[16], u2[16];
          tmem_ld16(tbase + (uint32_t)C::N + (uint32_t)c0, g2);
          tmem_ld16(tbase + (uint32_t)(3 * C::N) + (uint32_t)c0, u2);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            g[i] = __float_as_uint(__uint_as_float(g[i]) + __uint_as_float(g2[i]));
            u[i] = __float_as_uint(__uint_as_float(u[i]) + __uint_as_float(u2[i]));
          }
        }
        tmem_ld_wait();
        uint32_t habs = 0u;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int n = c0 + i;
          uint32_t av = 0u;
          if (valid && n < it.cnt) {
            const float xs = col_scale[n];
            float hv = silu_f32(__uint_as_float(g[i]) * xs) * (__uint_as_float(u[i]) * xs);
            if (nan_row) hv = __int_as_float(0x7FC00000);
            hout[(size_t)(it.hpos0 + n) * p.I + row] = hv;
            av = __float_as_uint(hv) & 0x7FFFFFFFu;
          }
          const uint32_t mx = __reduce_max_sync(0xFFFFFFFFu, av);
          if (lane == i) habs = mx;
        }
        if (lane < 16 && c0 + lane < it.cnt && habs != 0u) atomicMax(&p.ws.hmax[it.hpos0 + c0 + lane], habs);
      } else {
        uint32_t g2[16];  // the second issuer's accumulator (K-steps 2 and 3)
        tmem_ld16(tbase + (uint32_t)C::N + (uint32_t)c0, g2);
        tmem_ld_wait();
        if (valid) {
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int n = c0 + i;
            if (n < it.cnt) {
              float v = (__uint_as_float(g[i]) + __uint_as_float(g2[i])) * col_scale[n];
              if (nan_row) v = __int_as_float(0x7FC00000);
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

template <bool GU>
__global__ void __launch_bounds__(MxCfg<GU>::THREADS, 1) k_pf_mx(ExpertParams p, const __grid_constant__ MxXMaps xmaps) {
  using C = MxCfg<GU>;
  extern __shared__ uint8_t mx_dyn[];
  __shared__ MxShared<GU> sh;
  const int warp = threadIdx.x >> 5;
  if (warp == 0) {
    tmem_alloc(&sh.tmem_base, mxk::kTmemCols);
    tmem_relinquish();
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&sh.full[s], 1 + mxk::kSfWarps);
      mbar_init(&sh.empty[s], C::NI);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sh.accf[b], C::NI);
      mbar_init(&sh.acce[b], mxk::kEpWarps);
    }
    sh.abort_flag = 0;
    mbar_init_fence();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sh.tmem_base;
  MxCtx<GU> c;
  c.sh = &sh;
  c.ring = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(mx_dyn) + 1023) & ~(uintptr_t)1023);
  const int U = (int)p.ws.hdr->n_active;
  c.n_items = U > 0 ? __ldg(&(GU ? p.ws.act_pref_gu : p.ws.act_pref_dn)[U]) : 0;
  c.items = GU ? p.ws.items_gu : p.ws.items_dn;
  const int K = GU ? p.H : p.I;
  c.ns = K / mxk::kSliceK;
  c.srow = K / 32;
  c.hdr = p.ws.hdr;
  c.wait_limit = p.wait_limit;
  if (warp == 0 || warp >= mxk::kMma2Warp) {
    // Issuer 0 is warp 0 (it owns TMEM); issuers 1.. are warps kMma2Warp...
    if ((threadIdx.x & 31) == 0) mx_mma_role<GU>(p, c, tmem, warp == 0 ? 0 : warp - mxk::kMma2Warp + 1);
  } else if (warp == mxk::kTmaWarp) {
    mx_producer_role<GU>(p, c, &xmaps);
  } else if (warp < mxk::kEpWarp0) {
    mx_scale_role<GU>(p, c, tmem);
  } else {
    mx_epilogue_role<GU>(p, c, tmem);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, mxk::kTmemCols);
  }
}

bool prefill_supported(int H, int I) { return H % 128 == 0 && I % 128 == 0; }

// cuTensorMapEncodeTiled from the driver, looked up once through the runtime
// (no link-time dependency on the driver library); null if unavailable.
EncodeTiledFn encode_tiled_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
  });
  return fn;
}

namespace {

// Tensor map of the f16 h rows [rows][I] for the down GEMM's token tiles:
// boxes of 64 elements (128 bytes) x 128 rows, 128-byte swizzle (the MMA's
// K-major operand layout), out-of-range rows read as zero.
cudaError_t encode_h16_map(CUtensorMap* m, void* base, int rows, int I) {
  const EncodeTiledFn enc = encode_tiled_fn();
  if (!enc) return cudaErrorNotSupported;
  const cuuint64_t dims[2] = {(cuuint64_t)I, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)I * 2};
  const cuuint32_t box[2] = {(cuuint32_t)kPfSliceK, (cuuint32_t)kPfNTile};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, base, dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// Map of bucket-order E4M3 activation rows as a [terms][T k][K] byte tensor
// (term, row, byte): boxes of 128 bytes x `rows` rows x all terms, 128-byte
// swizzle, the terms' rows one after the other in shared memory; rows past
// the end read as zero.
cudaError_t encode_terms_map(CUtensorMap* m, void* base, int npairs, int K, int terms, int rows) {
  const EncodeTiledFn enc = encode_tiled_fn();
  if (!enc) return cudaErrorNotSupported;
  const cuuint64_t dims[3] = {(cuuint64_t)K, (cuuint64_t)npairs, (cuuint64_t)terms};
  const cuuint64_t strides[2] = {(cuuint64_t)K, (cuuint64_t)npairs * K};
  const cuuint32_t box[3] = {(cuuint32_t)mxk::kSliceK, (cuuint32_t)rows, (cuuint32_t)terms};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, base, dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}
}  // namespace

// Template of the per-expert code maps of the block-scaled GEMMs: an [M][K]
// matrix of 4-bit codes (row stride K / 2 bytes), boxes of 128 elements x 128
// rows, each 16 codes stored as 8 bytes followed by an 8-byte gap, 128-byte
// swizzle.  `base` only has to be a valid 32-byte-aligned address:
// the kernels replace it per expert.
cudaError_t encode_code_map_template(CUtensorMap* m, void* base, int K, int M) {
  const EncodeTiledFn enc = encode_tiled_fn();
  if (!enc) return cudaErrorNotSupported;
  const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)M};
  const cuuint64_t strides[1] = {(cuuint64_t)K / 2};
  const cuuint32_t box[2] = {(cuuint32_t)mxk::kSliceK, (cuuint32_t)kPfMTile};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 2, base, dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <bool GATEUP>
constexpr size_t pf_smem_bytes() {
  using C = PfCfg<GATEUP>;
  // Token tile ring + raw MXFP4 slots + alignment slack.
  return (size_t)C::BS * kPfTileBytes + (size_t)C::NG * C::R * C::kStage + 1024;
}

cudaError_t launch_prefill_experts(const ExpertParams& p, cudaStream_t s) {
  if (!p.x_bf16 || !prefill_supported(p.H, p.I)) return cudaErrorNotSupported;
  const int nsm = device_sm_count();
  const int npairs = p.T * p.k;
  cudaError_t err;
  // Bucket layout, active experts and tile prefixes come from the routing or
  // bucketing kernels already on the stream.  Routed experts run on the
  // block-scaled GEMMs (E4M3 activation terms); the bf16 shared expert on
  // k_pf_gemm (f16 operands).
  const bool routed = !p.shared_only;
  if (routed) {
    // Bucket position of every routed pair, then the pairs' E4M3 rows.
    if ((err = cudaMemsetAsync(p.ws.pinv, 0xFF, (size_t)npairs * 4, s)) != cudaSuccess) return err;
    k_pf_pinv<<<(npairs + 255) / 256, 256, 0, s>>>(p);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
    k_x_to_e4m3<<<p.T, 256, 0, s>>>(p);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
  }
  if (p.sh_gate) {
    k_x_to_f16<<<p.T, 256, 0, s>>>(p);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
    k_shared_sigma<<<(2 * p.I + p.H + 7) / 8, 256, 0, s>>>(p);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
  }
  if (!p.accumulate) {
    if ((err = cudaMemsetAsync(p.out, 0, (size_t)p.T * p.H * sizeof(float), s)) != cudaSuccess) return err;
  }
  k_pf_items<<<nsm, 256, 0, s>>>(p);
  if ((err = cudaGetLastError()) != cudaSuccess) return err;
  constexpr size_t mxgu_smem = (size_t)MxCfg<true>::STAGES * MxCfg<true>::STAGE + 1024;
  constexpr size_t mxdn_smem = (size_t)MxCfg<false>::STAGES * MxCfg<false>::STAGE + 1024;
  constexpr size_t gu_smem = pf_smem_bytes<true>();
  constexpr size_t dn_smem = pf_smem_bytes<false>();
  static_assert(gu_smem + sizeof(PfShared) <= 227 * 1024 && dn_smem + sizeof(PfShared) <= 227 * 1024, "smem");
  static_assert(mxgu_smem + sizeof(MxShared<true>) <= 227 * 1024, "smem");
  static_assert(mxdn_smem + sizeof(MxShared<false>) <= 227 * 1024, "smem");
  if ((err = ensure_smem_attr((const void*)k_pf_mx<true>, mxgu_smem)) != cudaSuccess) return err;
  if ((err = ensure_smem_attr((const void*)k_pf_mx<false>, mxdn_smem)) != cudaSuccess) return err;
  if ((err = ensure_smem_attr((const void*)k_pf_gemm<true>, gu_smem)) != cudaSuccess) return err;
  if ((err = ensure_smem_attr((const void*)k_pf_gemm<false>, dn_smem)) != cudaSuccess) return err;
  CUtensorMap tmap_h, tmpl_gu, tmpl_dn;
  MxXMaps xmaps, hmaps;
  memset(&tmap_h, 0, sizeof tmap_h);
  memset(&tmpl_gu, 0, sizeof tmpl_gu);
  memset(&tmpl_dn, 0, sizeof tmpl_dn);
  memset(&xmaps, 0, sizeof xmaps);
  memset(&hmaps, 0, sizeof hmaps);
  if ((err = encode_h16_map(&tmap_h, p.ws.h16, npairs + p.T, p.I)) != cudaSuccess) return err;
  if (routed) {
    if ((err = encode_code_map_template(&tmpl_gu, p.ws.tmaps, p.H, p.I)) != cudaSuccess) return err;
    if ((err = encode_code_map_template(&tmpl_dn, p.ws.tmaps, p.I, p.H)) != cudaSuccess) return err;
    for (int i = 0; i < mxk::kXMaps; ++i) {
      const int rows = (i + 1) * mxk::kXBox;
      if ((err = encode_terms_map(&xmaps.m[i], p.ws.xp, npairs, p.H, MxCfg<true>::NT, rows)) != cudaSuccess ||
          (err = encode_terms_map(&hmaps.m[i], p.ws.h8, npairs, p.I, MxCfg<false>::NT, rows)) != cudaSuccess)
        return err;
    }
    k_pf_mx_maps<<<(3 * p.E + 255) / 256, 256, 0, s>>>(p, tmpl_gu, tmpl_dn);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
  }
  ExpertParams ps = p;  // the shared expert's items alone
  ps.shared_only = 1;
  prof_before(MOE_STAGE_PF_GATEUP, s);
  if (routed) k_pf_mx<true><<<nsm, MxCfg<true>::THREADS, mxgu_smem, s>>>(p, xmaps);
  if ((err = cudaGetLastError()) == cudaSuccess && p.sh_gate) {
    k_pf_gemm<true><<<nsm, kPfThreads, gu_smem, s>>>(ps, tmap_h);
    err = cudaGetLastError();
  }
  prof_after(MOE_STAGE_PF_GATEUP, s);
  if (err != cudaSuccess) return err;
  // Down operands: the routed pairs' h rows as E4M3 terms, the shared
  // expert's as f16.
  if (routed) {
    k_h_to_e4m3<<<(npairs + 7) / 8, 256, 0, s>>>(p);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
  }
  if (p.sh_gate) {
    k_h_to_f16<<<(p.T + 7) / 8, 256, 0, s>>>(p, npairs, npairs + p.T);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
  }
  prof_before(MOE_STAGE_PF_DOWN, s);
  if (routed) k_pf_mx<false><<<nsm, MxCfg<false>::THREADS, mxdn_smem, s>>>(p, hmaps);
  if ((err = cudaGetLastError()) == cudaSuccess && p.sh_gate) {
    k_pf_gemm<false><<<nsm, kPfThreads, dn_smem, s>>>(ps, tmap_h);
    err = cudaGetLastError();
  }
  prof_after(MOE_STAGE_PF_DOWN, s);
  return err;
}

}  // namespace moe
