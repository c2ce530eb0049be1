// common.cuh — shared device helpers, workspace layout and kernel parameter
// blocks of the routed MXFP4 MoE library (sm_103a).
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "moe_mxfp4.h"

namespace moe {

constexpr int kDecodeMaxT = MOE_DECODE_MAX_T;
constexpr int kDecodeBatchMaxT = MOE_DECODE_BATCH_MAX_T;
constexpr int kMaxK = 32;
constexpr int kNumSMs = 152;  // GB300; launch code queries the device instead

// ---------------------------------------------------------------- workspace --
// Header at the start of the workspace (zeroed at the start of every call).
struct WsHeader {
  uint32_t status;      // first nonzero moe_status a kernel recorded
  uint32_t ticket;      // last-block-done counter of the bucket count kernel
  uint32_t n_active;    // number of experts with at least one routed pair
  uint32_t route_ticket;
  uint32_t queue[16];   // work counters of persistent kernels
  uint32_t pad[44];
};
static_assert(sizeof(WsHeader) == 256, "header is 256 bytes");

enum Queue { kQGateUp = 0, kQDown = 1, kQPfGateUp = 2, kQPfDown = 3, kQShared = 4, kQSharedDown = 5 };

// Device pointers into one workspace.
struct Ws {
  WsHeader* hdr;
  float2* logits;       // [T][E] router scores as (hi, lo) double-floats
  int32_t* ids;         // [T][k]  (used when the caller gives none)
  float* w;             // [T][k]
  uint32_t* mask;       // [E][W]  W = ceil(T/32): token bitmask per expert
  int32_t* wprefix;     // [E][W]  exclusive popcount prefix of mask words
  int32_t* offsets;     // [E+1]
  int32_t* sorted;      // [T*k]
  int32_t* act_e;       // [E]     active experts, ascending
  int32_t* act_pref_gu; // [E+1]   prefix of prefill gate/up tiles per active expert
  int32_t* act_pref_dn; // [E+1]   prefix of prefill down tiles per active expert
  int4* items_gu;       // prefill gate/up work items {e (-1: shared expert), m0, p0, cnt}
  int4* items_dn;       // prefill down work items, the same fields
  uint16_t* xh;         // [T][H]  fp16 activations (prefill)
  float* xscale;        // [T]     2^-sigma_t of the fp16 activations
  uint8_t* xp;          // [2][T*k][H] prefill: each routed pair's activations as two E4M3
                        // terms, rows in bucket order (aliases y)
  int32_t* pinv;        // [T*k] prefill: bucket position of each routed pair (-1: none)
  void* tmaps;          // [E][3] prefill: tensor maps (128 bytes each) of the gate, up, down codes
  uint8_t* h8;          // [3][T*k][I] prefill: routed h rows as three E4M3 terms (in y's region,
                        // after the f16 h rows)
  float* x8scale;       // [T]     2^-tau_t of token t's E4M3 terms
  void* h;              // fp32 h: [T*k][I] (decode) or [T*k + T][I] (prefill; rows
                        // T*k.. hold the shared expert's h)
  uint16_t* h16;        // [T*k + T][I] prefill: f16 h scaled by 2^tau_row (aliases y)
  uint32_t* hmax;       // [T*k + T]  prefill: bits of max |h| over each h row
  float* hscale;        // [T*k + T]  prefill: 2^-tau_row of each f16 h row
  int32_t* shsig;       // [2I + H] row shifts of the bf16 shared expert (gate, up, down)
  float* y;             // [T*k][H] fp32 (decode, T <= 1024)
  float2* rpart;        // [S][T][E] router partial sums of the S K-splits (S > 1 only)
  uint16_t* wr16;       // [2][E][H] router weights as two bf16 terms (T > 64 only)
  float* wrnorm;        // [E] Euclidean norm of each router row, rounded up (T > 64 only)
  float* sapprox;       // [T][E] tensor-core approximation of the router scores (T > 64 only)
  uint32_t* rowdone;    // [ceil(H/32)] per-row-tile completion counters
  // Persistent block-scaled decode kernel (T <= 8; empty otherwise):
  uint8_t* dmx_xq;      // [16][H] the tokens' E4M3 terms (rows 2t, 2t + 1)
  uint8_t* dmx_hq;      // [3 T k][I] h of each routed pair (bucket order) as three E4M3 terms
  uint8_t* dmx_hs;      // [3 T k][I / 32] E8M0 scale of each 32-element block of those rows
  uint32_t* dmx_cnt;    // counters (see dmx_counter_words)
  size_t total;
};

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Tokens per tile of the prefill path's block-scaled GEMMs (two accumulator
// buffers of two accumulators each fit Tensor Memory next to the scales).
constexpr int kPfNTileGu = 112;
constexpr int kPfNTileDn = 96;

// Splits of the contraction of the router GEMM (64 experts x 64 tokens per
// CTA) for batches above 64 tokens (smaller ones keep their workspace size;
// their decode route is the GEMV): enough CTAs for about three per SM on 152
// SMs, each split at least 256 long, at most 16.  A function of the shape
// only, so that the workspace size needs no device query and a shape always
// sums in the same order.
__host__ __device__ inline int router_splits(int T, int E, int H) {
  if (T <= kDecodeMaxT) return 1;
  const int tiles = ((E + 63) / 64) * ((T + 63) / 64);
  int s = (456 + tiles - 1) / tiles;
  const int smax = H / 256;
  s = s < smax ? s : smax;
  s = s < 16 ? s : 16;
  return s < 1 ? 1 : s;
}

// Persistent block-scaled decode kernel (decode_mx.cu): batch and tile limits.
constexpr int kDmxMaxT = 8;        // tokens of a step the kernel takes
constexpr int kDmxNGu = 16;        // gate/up B rows: two E4M3 terms of each of up to 8 tokens
constexpr int kDmxNDn = 32;        // down B rows: three E4M3 terms of each of up to 8 pairs (+ padding)
constexpr int kDmxCntHead = 32;     // counter words before the per-tile counters

// Shapes whose workspace holds the kernel's buffers.
__host__ __device__ inline bool dmx_shape_ok(int T, int H, int I) {
  return T >= 1 && T <= kDmxMaxT && H >= 128 && H % 128 == 0 && I >= 256 && I % 128 == 0;
}
// Gate/up slices (128 elements) whose scale words the persistent decode
// kernel stages at a time: the smallest divisor of the slice count that is
// at least 12 (or all of them; at most 16).
__host__ __device__ inline int dmx_spp(int ns) {
  for (int d = 12; d < ns; ++d)
    if (ns % d == 0) return d;
  return ns;
}

// Layout of the workspace for a shape; pointers are offsets from `base`.
inline Ws ws_layout(const moe_shape& s, void* base) {
  const size_t T = (size_t)s.T, H = (size_t)s.H, E = (size_t)s.E, I = (size_t)s.I, k = (size_t)s.k;
  const size_t W = (T + 31) / 32;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    size_t o = off;
    off = align_up(off + bytes, 256);
    return (char*)base + o;
  };
  Ws ws;
  ws.hdr = (WsHeader*)take(sizeof(WsHeader));
  ws.logits = (float2*)take(T * E * 8);
  ws.ids = (int32_t*)take(T * k * 4);
  ws.w = (float*)take(T * k * 4);
  ws.mask = (uint32_t*)take(E * W * 4);
  ws.wprefix = (int32_t*)take(E * W * 4);
  ws.offsets = (int32_t*)take((E + 1) * 4);
  ws.sorted = (int32_t*)take(T * k * 4);
  ws.act_e = (int32_t*)take(E * 4);
  ws.act_pref_gu = (int32_t*)take((E + 1) * 4);
  ws.act_pref_dn = (int32_t*)take((E + 1) * 4);
  {
    // Work items of the prefill GEMMs: (active expert, 128-row tile, token
    // tile of up to 128), then the shared expert's tiles.  The token tiles of
    // all active experts number at most ceil(T*k/128) + min(E, T*k).
    const size_t pairs = T * k;
    const size_t ntiles = (pairs + kPfNTileDn - 1) / kPfNTileDn + (E < pairs ? E : pairs);
    const size_t ntiles_gu = (pairs + kPfNTileGu - 1) / kPfNTileGu + (E < pairs ? E : pairs);
    const size_t shtiles = (T + 127) / 128;
    const size_t mgu = (I + 127) / 128, mdn = (H + 127) / 128;
    ws.items_gu = (int4*)take((ntiles_gu + shtiles) * mgu * 16);
    ws.items_dn = (int4*)take((ntiles + shtiles) * mdn * 16);
  }
  ws.xh = (uint16_t*)take(T * H * 2);
  ws.xscale = (float*)take(T * 4);
  ws.x8scale = (float*)take(T * 4);
  ws.pinv = (int32_t*)take(T * k * 4);
  ws.tmaps = (void*)take(E * 3 * 128);
  // Tokens the decode path may take for this shape (0: it cannot).
  const size_t Td = T <= (size_t)kDecodeBatchMaxT ? T : 0;
  // h in fp32: Td*k rows for the decode path, T*k + T rows for the prefill
  // path (routed pairs, then the shared expert's tokens).
  const size_t hrows = T * k + T;
  const size_t h_dec = Td * k * I * 4, h_pf = hrows * I * 4;
  ws.h = (void*)take(h_dec > h_pf ? h_dec : h_pf);
  ws.hmax = (uint32_t*)take(hrows * 4);
  ws.hscale = (float*)take(hrows * 4);
  ws.shsig = (int32_t*)take((2 * I + H) * 4);
  // y (decode), the prefill path's E4M3 activation rows and its f16 h share
  // one region: the prefill kernels run on the decode path only for the
  // shared expert, after the routed experts' combine has consumed y (and then
  // without the E4M3 rows); on the prefill path the f16 h is written after
  // the gate/up GEMM, the last reader of the E4M3 rows.
  // The E4M3 h terms follow the f16 h rows (both are read by the down GEMMs).
  const size_t h8_off = align_up(hrows * I * 2, 256);
  const size_t y_dec = Td * k * H * 4, hy_pf = h8_off + 3 * T * k * I, xp_pf = 2 * T * k * H;
  size_t yreg = y_dec > hy_pf ? y_dec : hy_pf;
  yreg = yreg > xp_pf ? yreg : xp_pf;
  ws.y = (float*)take(yreg);
  ws.h16 = (uint16_t*)ws.y;
  ws.xp = (uint8_t*)ws.y;
  ws.h8 = (uint8_t*)ws.y + h8_off;
  ws.rowdone = (uint32_t*)take(((H + 31) / 32) * 4);
  {
    // The persistent block-scaled decode kernel's buffers.
    const bool dmx = dmx_shape_ok(s.T, s.H, s.I);
    const size_t rt = I / 128;
    const size_t umax = E < T * k ? E : T * k;
    ws.dmx_xq = (uint8_t*)take(dmx ? (size_t)kDmxNGu * H : 0);
    ws.dmx_hq = (uint8_t*)take(dmx ? 3 * T * k * I : 0);
    ws.dmx_hs = (uint8_t*)take(dmx ? 3 * T * k * (I / 32) : 0);
    ws.dmx_cnt = (uint32_t*)take(dmx ? (kDmxCntHead + umax * rt) * 4 : 0);
  }
  const size_t S = (size_t)router_splits(s.T, s.E, s.H);
  ws.rpart = (float2*)take(S > 1 ? S * T * E * 8 : 0);
  const bool rtc = T > (size_t)kDecodeMaxT;  // batches routed by the tensor-core screen
  ws.wr16 = (uint16_t*)take(rtc ? 2 * E * H * 2 : 0);
  ws.wrnorm = (float*)take(rtc ? E * 4 : 0);
  ws.sapprox = (float*)take(rtc ? T * E * 4 : 0);
  ws.total = off;
  return ws;
}

// ------------------------------------------------------------- device utils --
__device__ __forceinline__ void set_status(WsHeader* hdr, uint32_t st) {
  atomicCAS(&hdr->status, 0u, st);
}

// Every tensor pointer of an expert descriptor non-null and 16-byte aligned
// (bulk copies and 128-bit loads require it).
__device__ __forceinline__ bool expert_ptrs_ok(const moe_expert& ex) {
  const uintptr_t a = (uintptr_t)ex.gate.q | (uintptr_t)ex.gate.s | (uintptr_t)ex.up.q | (uintptr_t)ex.up.s |
                      (uintptr_t)ex.down.q | (uintptr_t)ex.down.s;
  return (a & 15u) == 0 && ex.gate.q && ex.gate.s && ex.up.q && ex.up.s && ex.down.q && ex.down.s;
}

// E8M0 scale byte -> fp32 2^(s-127); s = 0 gives the subnormal 2^-127, s = 255 NaN.
__device__ __forceinline__ float e8m0_f32(uint32_t s) {
  uint32_t bits = s == 0u ? 0x00400000u : (s << 23);
  bits = s == 255u ? 0x7FC00000u : bits;
  return __uint_as_float(bits);
}

// Two E2M1 codes (low byte of v: element 0 in bits 3..0, element 1 in 7..4)
// -> f16x2 (element 0 in the low half).  Exact: every E2M1 value is an fp16.
__device__ __forceinline__ uint32_t e2m1x2_f16x2(uint32_t v, int byte) {
  uint32_t r;
  switch (byte) {
    case 0: asm("{\n .reg .b8 b0, b1, b2, b3;\n mov.b32 {b0, b1, b2, b3}, %1;\n cvt.rn.f16x2.e2m1x2 %0, b0;\n}" : "=r"(r) : "r"(v)); break;
    case 1: asm("{\n .reg .b8 b0, b1, b2, b3;\n mov.b32 {b0, b1, b2, b3}, %1;\n cvt.rn.f16x2.e2m1x2 %0, b1;\n}" : "=r"(r) : "r"(v)); break;
    case 2: asm("{\n .reg .b8 b0, b1, b2, b3;\n mov.b32 {b0, b1, b2, b3}, %1;\n cvt.rn.f16x2.e2m1x2 %0, b2;\n}" : "=r"(r) : "r"(v)); break;
    default: asm("{\n .reg .b8 b0, b1, b2, b3;\n mov.b32 {b0, b1, b2, b3}, %1;\n cvt.rn.f16x2.e2m1x2 %0, b3;\n}" : "=r"(r) : "r"(v)); break;
  }
  return r;
}

__device__ __forceinline__ float2 f16x2_f32x2(uint32_t h2) {
  return __half22float2(*reinterpret_cast<const __half2*>(&h2));
}

__device__ __forceinline__ float bf16_f32(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }

// Streaming 16-byte load that does not allocate in L1.
__device__ __forceinline__ uint4 ldg_stream(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ uint32_t ldg_u8(const uint8_t* p) {
  uint16_t v;
  asm volatile("ld.global.nc.L1::no_allocate.u8 %0, [%1];" : "=h"(v) : "l"(p));
  return (uint32_t)v;
}

// Programmatic dependent launch: wait for the preceding kernel's memory.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Sum over the 32 lanes of v[lane % V] for V values per lane (V a power of two
// <= 32): returns, on each lane, the warp total of value index (lane & (V-1)).
// The addition tree is the same for every value index and every V-sized
// packing, so a value's total does not depend on what else is packed with it.
template <int V>
__device__ __forceinline__ float warp_transpose_reduce(float (&v)[V]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int m = V / 2; m >= 1; m /= 2) {
    const bool upper = (lane & m) != 0;
#pragma unroll
    for (int i = 0; i < m; ++i) {
      const float send = upper ? v[i] : v[i + m];
      const float keep = upper ? v[i + m] : v[i];
      v[i] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, m);
    }
  }
#pragma unroll
  for (int m = V; m < 32; m *= 2) v[0] += __shfl_xor_sync(0xFFFFFFFFu, v[0], m);
  return v[0];
}

__device__ __forceinline__ float silu_f32(float z) { return z / (1.0f + expf(-z)); }

// One token row of bf16 activations -> f16 scaled by 2^sigma_t, with sigma_t
// putting the row's largest magnitude in [2^14, 2^15) (exact: bf16 has 8
// significant bits); xscale_t = 2^-sigma_t.  Called by all threads of a CTA
// (any multiple of 32 up to 1024); H % 8 == 0.
__device__ __forceinline__ void x_row_to_f16(const uint16_t* xb, int H, uint16_t* xo, float* xscale) {
  __shared__ float xr_wmax[32];
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
  if ((threadIdx.x & 31) == 0) xr_wmax[threadIdx.x >> 5] = m;
  __syncthreads();
  m = 0.f;
  for (int w = 0; w < (int)(blockDim.x >> 5); ++w) m = fmaxf(m, xr_wmax[w]);
  int sig = 0;
  if (m > 0.f) sig = 14 - ((int)((__float_as_uint(m) >> 23) & 0xFF) - 127);
  sig = sig > 100 ? 100 : (sig < -100 ? -100 : sig);
  const float up = __int_as_float((sig + 127) << 23);
  if (threadIdx.x == 0) *xscale = __int_as_float((127 - sig) << 23);
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

// ------------------------------------------------ double-float arithmetic --
// A value is carried as an unevaluated sum hi + lo of two floats (Knuth's
// TwoSum / Dekker's Fast2Sum error-free transformations), which keeps router
// scores accurate to ~2^-44 relative: the fp32 weights derived from them do
// not inherit fp32 rounding of large scores.
__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
  s = a + b;
  const float bp = s - a;
  e = (a - (s - bp)) + (b - bp);
}

// (hi, lo) += p, lo collecting the rounding errors (not renormalised).
__device__ __forceinline__ void df_add_f(float& hi, float& lo, float p) {
  float s, e;
  two_sum(hi, p, s, e);
  hi = s;
  lo += e;
}

// (hi, lo) = (ahi, alo) + (bhi, blo), renormalised.
__device__ __forceinline__ void df_add(float ahi, float alo, float bhi, float blo, float& hi, float& lo) {
  float s, e;
  two_sum(ahi, bhi, s, e);
  e += alo + blo;
  hi = s + e;
  lo = e - (hi - s);
}

// Double-float version of warp_transpose_reduce (same addition tree).
template <int V>
__device__ __forceinline__ void warp_transpose_reduce_df(float (&vh)[V], float (&vl)[V], float& oh, float& ol) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int m = V / 2; m >= 1; m /= 2) {
    const bool upper = (lane & m) != 0;
#pragma unroll
    for (int i = 0; i < m; ++i) {
      const float sh = upper ? vh[i] : vh[i + m];
      const float sl = upper ? vl[i] : vl[i + m];
      const float kh = upper ? vh[i + m] : vh[i];
      const float kl = upper ? vl[i + m] : vl[i];
      const float rh = __shfl_xor_sync(0xFFFFFFFFu, sh, m);
      const float rl = __shfl_xor_sync(0xFFFFFFFFu, sl, m);
      df_add(kh, kl, rh, rl, vh[i], vl[i]);
    }
  }
#pragma unroll
  for (int m = V; m < 32; m *= 2) {
    const float rh = __shfl_xor_sync(0xFFFFFFFFu, vh[0], m);
    const float rl = __shfl_xor_sync(0xFFFFFFFFu, vl[0], m);
    df_add(vh[0], vl[0], rh, rl, vh[0], vl[0]);
  }
  oh = vh[0];
  ol = vl[0];
}

// ----------------------------------------------------------- kernel params --
struct RouteParams {
  int T, H, E, k;
  const void* x;
  int x_bf16;
  const float* wr;
  const float* br;
  int32_t* ids;
  float* w;
  int32_t* offsets;     // bucket outputs (may alias workspace)
  int32_t* sorted;
  int want_buckets;
  int dmx_I;             // > 0: the router kernel also prepares the persistent decode kernel (intermediate size)
  long long wait_limit;  // cycles before a bounded wait gives up (kWaitCycles unless diagnosing)
  Ws ws;
};

// Bucketing / planning: counting sort of routed pairs by expert, the active
// expert list and the prefill tile prefixes.
struct BucketParams {
  int T, E, k;
  const int32_t* ids;      // [T][k]
  int32_t* offsets_out;    // [E+1] caller copy or NULL
  int32_t* sorted_out;     // [T*k] caller copy or NULL
  int n_tile;              // prefill token tile (columns of one MMA tile) of the routed down GEMM
  int n_tile_gu;           // prefill token tile of the routed gate/up GEMM
  int m_tiles_gu;          // prefill row tiles of gate/up (ceil(I/128))
  int m_tiles_dn;          // prefill row tiles of down (ceil(H/128))
  Ws ws;
};

struct ExpertParams {
  int T, H, E, I, k;
  const void* x;
  int x_bf16;
  const moe_expert* experts;  // device [E]
  const int32_t* ids;
  const float* w;
  const int32_t* offsets;
  const int32_t* sorted;
  float* out;
  int accumulate;
  const moe_dense_bf16* shared_dev;  // unused on device; shared pointers below
  const uint16_t *sh_gate, *sh_up, *sh_down;
  int shared_only;       // prefill kernels: the shared expert alone (decode path), no routed h rows
  int fused_route;       // decode: the gate/up kernel routes (from ws.logits) first
  RouteParams rp;        // the route to compute when fused_route
  long long wait_limit;  // cycles before a bounded wait gives up (kWaitCycles unless diagnosing)
  Ws ws;
};

}  // namespace moe
