// decode_mx.cu — the routed experts of a decode step of up to 8 tokens (bf16
// activations) as one persistent kernel on block-scaled tcgen05 MMAs.
//
// The fused MXFP4 dequant+GEMV of [deltafin, "The techniques that bought the
// 82x"] streams each routed expert's weights once; here the tensor core reads
// the E2M1 codes and their E8M0 block scales as stored (tcgen05.mma
// kind::mxf8f6f4.block_scale, M = 128 weight rows), so no CUDA-core
// instruction is spent per weight, and one launch streams every routed
// expert's gate, up and down weights:
//   * prologue: every CTA routes the batch from the router scores (top-k,
//     weights, buckets; CTA 0 publishes them), and the CTAs build the tensor
//     maps of the active experts' codes together;
//   * gate/up items (expert, 128 rows of I, all of H): A = the gate and up
//     code tiles, B = the tokens' activations as two exact E4M3 terms (one B
//     row per term: 16 rows for 8 tokens, the terms' weights 2^0 and 2^-4 in
//     the B scales); the epilogue applies SwiGLU and stores h as three E4M3
//     terms with one E8M0 scale per 32-row block (the B operand of down), then
//     marks the h tile ready;
//   * down items (expert, 128 rows of H, all of I): A = the down code tiles,
//     B = the expert's h terms (three rows per routed pair), after its h
//     tiles are ready; each pair's weighted row goes to the workspace;
//   * once every CTA is done, each adds a share of the tokens' k rows in slot
//     order into out ([Deltafin's custom compiled runtime, "The native
//     build"]: ordered reduction).
// A token's arithmetic does not depend on the batch: every sum is taken over
// the whole contraction in one accumulator and in a fixed order.
//
// Roles of a CTA (one per SM): warps 0 and 10 (lane 0) issue the MMAs
// (accumulator 0: gate rows / even down slices; accumulator 1: up rows / odd
// down slices; warp 0 owns Tensor Memory); warps 1, 11, 14 and 15 copy the
// code boxes (box 0 or 1 of the even or the odd stages), warps 12 and 13 the
// B tiles (even and odd stages): the copy unit serves the copies of one
// issuing thread one after another, so one thread cannot keep the stream
// busy; warps 2-5 stage the block scales and write
// them into Tensor Memory; warps 6-9 drain the accumulators.  Gate/up tiles
// are dealt to the CTAs in waves, so each expert's h is finished early;
// down items go mostly to the CTAs with one gate/up tile fewer, so the weight
// bytes per CTA even out.  Every wait is bounded (MOE_ERR_TIMEOUT).
#include <cuda.h>
#include <string.h>

#include "async.cuh"
#include "decode_mx.cuh"
#include "kernels.h"
#include "route_small.cuh"
#include "tcgen05.cuh"

namespace moe {

namespace dmx {
constexpr int kSliceK = 128;                   // contraction elements per slice
constexpr int kStages = 4;
constexpr int kBox = 128 * 128;                // shared-memory bytes of a 128 x 128 code box
constexpr int kCodeTx = 128 * 64;              // bytes a code box's copy delivers (4-bit codes)
constexpr int kBGu = kDmxNGu * 128;            // gate/up B tile of one slice
constexpr int kBDn = kDmxNDn * 128;            // down B tile of one slice
constexpr int kStage = 2 * kBox + 2 * kBDn;    // two code boxes, two B tiles
constexpr int kTmaWarp = 1, kSfWarp0 = 2, kSfWarps = 4, kEpWarp0 = 6, kEpWarps = 4, kMma2Warp = 10;
// Producers (role, stage parity): warp 1 (box 0, even), 11 (box 1, even),
// 12 (B, even), 13 (B, odd), 14 (box 0, odd), 15 (box 1, odd).
constexpr int kTma2Warp = 11, kTmaBWarp = 12, kTmaOddWarp = 14;
constexpr int kProducers = 3;                  // producers arming each stage: two code boxes, one B
static_assert(kSfWarp0 == kTmaWarp + 1 && kSfWarp0 + kSfWarps == kEpWarp0 && kEpWarp0 + kEpWarps == kMma2Warp &&
                  kTma2Warp == kMma2Warp + 1 && kTmaBWarp == kTma2Warp + 1,
              "warp roles");
static_assert(kTmaOddWarp == kTmaBWarp + 2, "warp roles");
constexpr int kThreads = (kTmaOddWarp + 2) * 32;
constexpr uint32_t kTmemCols = 256;
constexpr uint32_t kAccN = 32;                         // columns per accumulator
constexpr uint32_t kColSfbGu = 4 * kAccN;              // two buffers of two accumulators, then
constexpr uint32_t kColSfa = kColSfbGu + 4;            //   gate/up B scales; A scales of stage st,
constexpr uint32_t kColSfbDn = kColSfa + 8 * kStages;  //   box w at +8 st + 4 w; down B scales likewise
static_assert(kColSfbDn + 8 * kStages <= kTmemCols, "TMEM columns");
static_assert(kStage % 1024 == 0 && kBox % 1024 == 0 && kBDn % 1024 == 0, "1024-byte aligned tiles");
static_assert(kStages % 2 == 0, "the two B producers take even and odd stages");
constexpr int kNanRing = 8;  // items whose NaN-row flags are kept (scale warps run at most 6 items ahead)
constexpr uint32_t kPollMma = 0, kPollTma = 32, kPollSf = 64, kPollEp = 128, kPollDep = 256;
}  // namespace dmx

// Tensor maps of one launch: the code templates (the device puts each
// expert's address in), the tokens' E4M3 terms and the h terms.
struct DmxMaps {
  CUtensorMap gu;  // [I][H] 4-bit codes, 128 x 128 boxes
  CUtensorMap dn;  // [H][I] 4-bit codes, 128 x 128 boxes
  CUtensorMap xq;  // [2T][H] bytes, 128 x 16 boxes (rows past 2T read as zero)
  CUtensorMap hq;  // [3Tk][I] bytes, 128 x 32 boxes (rows past the end read as zero)
};

struct DmxShared {
  uint64_t full[dmx::kStages];   // stage filled: 3 producers (with their copies' bytes) + 4 scale warps
  uint64_t empty[dmx::kStages];  // stage consumed: both issuers' tcgen05.commit
  uint64_t accf[2];              // accumulator buffer ready: both issuers
  uint64_t acce[2];              // accumulator buffer drained: 4 epilogue warps
  uint64_t sbar[2];              // scale chunk buffer loaded: 128 scale threads (cp.async arrivals)
  uint64_t sfree[2];             // scale chunk buffer read to the end: 4 scale warps
  uint32_t tmem_base;
  int abort_flag;
  int U;
  int n_gu, n_dn;                // this CTA's gate/up tiles and down items
  int x_h, nl;                   // down dealing: items of a heavy CTA; CTAs sharing the later rounds
  uint32_t tok_mask[kDmxMaxT];   // slots of each token present in the plan
  int tok_cnt[kDmxMaxT];
  uint8_t ok_u[256];             // per active expert: descriptor usable by the tensor-map copies
  uint8_t nanf[dmx::kNanRing][128];  // per item (ring): rows with an E8M0 scale of 255
  uint32_t sfbw[4][16 * 32];     // per scale warp: the current down item's B scale words [slice][row]
  uint32_t sbuf[2][2][16][128];  // A scale words of a chunk of slices [box matrix][word][row]
};

struct DmxCtx {
  DmxShared* sh;
  uint8_t* ring;
  const int* ue;
  const int* ub0;
  const int* un;
  const int* pairs;
  const float* wts;
  DmxDims d;
  const uint8_t* maps;  // tensor maps [E][3] (gate, up, down codes) in the workspace
  WsHeader* hdr;
  long long wait_limit;
};

struct DmxItem {
  bool gu;
  int u, r;  // expert slot, row tile (gate/up: of I; down: of H)
  int e, b0, cnt;
  int map;   // index of the first tensor map (gate/up: gate, up at map + 1; down)
};

__device__ __forceinline__ int dmx_nitems(const DmxShared& sh) { return sh.n_gu + sh.n_dn; }

// Item li of this CTA.  Gate/up tile g (expert-major) goes to CTA g % G;
// down items (expert-major) are dealt in rounds in descending CTA order,
// first to all CTAs (x_h rounds), then only to the nl CTAs with one gate/up
// tile fewer.
__device__ __forceinline__ DmxItem dmx_item(const DmxCtx& c, int li) {
  const DmxShared& sh = *c.sh;
  const int G = gridDim.x, cb = blockIdx.x;
  DmxItem it;
  it.gu = li < sh.n_gu;
  if (it.gu) {
    const int g = cb + li * G;
    it.u = g / c.d.rt;
    it.r = g - it.u * c.d.rt;
  } else {
    const int j = li - sh.n_gu;
    const int dd = (j < sh.x_h ? j : sh.x_h) * G + (j > sh.x_h ? j - sh.x_h : 0) * sh.nl + (G - 1 - cb);
    it.u = dd / c.d.rh;
    it.r = dd - it.u * c.d.rh;
  }
  it.e = c.ue[it.u];
  it.b0 = c.ub0[it.u];
  it.cnt = c.un[it.u];
  it.map = 3 * it.e + (it.gu ? 0 : 2);
  return it;
}

// Ring stages an item takes: a gate/up slice each, or two down slices.
__device__ __forceinline__ int dmx_item_stages(const DmxCtx& c, const DmxItem& it) {
  return it.gu ? c.d.ns_gu : (c.d.rt + 1) / 2;
}

__device__ __forceinline__ bool dmx_wait(const DmxCtx& c, uint64_t* bar, uint32_t parity, uint32_t backoff_ns) {
  DmxShared& sh = *c.sh;
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
__device__ __forceinline__ bool dmx_warp_wait(const DmxCtx& c, uint64_t* bar, uint32_t parity, uint32_t backoff_ns) {
  const bool ok = dmx_wait(c, bar, parity, backoff_ns);
  return __all_sync(0xFFFFFFFFu, ok);
}
// Wait until ring stage gs % kStages is free for global stage gs.
__device__ __forceinline__ bool dmx_claim(const DmxCtx& c, int gs, uint32_t backoff_ns) {
  const int st = gs % dmx::kStages, use = gs / dmx::kStages;
  if (use == 0) return true;
  return dmx_wait(c, &c.sh->empty[st], (use - 1) & 1, backoff_ns);
}

__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
// Wait (bounded) until another CTA's counter reaches `target`.
__device__ __forceinline__ bool dmx_wait_count(const DmxCtx& c, const uint32_t* cnt, uint32_t target) {
  if (ld_acquire_u32(cnt) >= target) return true;
  const long long t0 = clock64();
  for (;;) {
    __nanosleep(dmx::kPollDep);
    if (ld_acquire_u32(cnt) >= target) return true;
    if (*(volatile int*)&c.sh->abort_flag) return false;
    if (clock64() - t0 > c.wait_limit) {
      set_status(c.hdr, MOE_ERR_TIMEOUT);
      *(volatile int*)&c.sh->abort_flag = 1;
      return false;
    }
  }
}
// Wait (bounded) until all rt h tiles of an expert are ready; one thread
// reads the rt counters together (one round trip per poll).  rt <= 16.
__device__ bool dmx_wait_h_ready(const DmxCtx& c, const uint32_t* ra) {
  const int rt = c.d.rt;
  auto ready = [&]() {
    uint32_t v[16];
#pragma unroll
    for (int r = 0; r < 16; ++r) v[r] = r < rt ? ld_acquire_u32(ra + r) : 4u;
    bool ok = true;
#pragma unroll
    for (int r = 0; r < 16; ++r) ok = ok && v[r] >= 4u;
    return ok;
  };
  if (ready()) return true;
  const long long t0 = clock64();
  for (;;) {
    __nanosleep(dmx::kPollDep);
    if (ready()) return true;
    if (*(volatile int*)&c.sh->abort_flag) return false;
    if (clock64() - t0 > c.wait_limit) {
      set_status(c.hdr, MOE_ERR_TIMEOUT);
      *(volatile int*)&c.sh->abort_flag = 1;
      return false;
    }
  }
}
// Order this thread's generic-proxy global writes (or reads acquired from
// other CTAs) with its async-proxy accesses (tensor-map copies).
__device__ __forceinline__ void fence_async_global() { asm volatile("fence.proxy.async.global;" ::: "memory"); }

// Counters (see dmx_counter_words): maps built, CTAs done, h-tile readiness.
__device__ __forceinline__ uint32_t* dmx_mapcnt(const Ws& ws) { return ws.dmx_cnt; }
__device__ __forceinline__ uint32_t* dmx_donecnt(const Ws& ws) { return ws.dmx_cnt + 1; }
__device__ __forceinline__ uint32_t* dmx_hready(const Ws& ws) { return ws.dmx_cnt + kDmxCntHead; }

// ------------------------------------------------------------ stage cursor --
// A position in this CTA's sequence of ring stages: item li, its stage j.
struct DmxCursor {
  int li, j, nst;
  DmxItem it;
  bool wok;
};
__device__ __forceinline__ void cur_enter(const DmxCtx& c, DmxCursor& cu, int li) {
  cu.li = li;
  cu.j = 0;
  cu.nst = 0;
  cu.wok = false;
  if (li < dmx_nitems(*c.sh)) {
    cu.it = dmx_item(c, li);
    cu.nst = dmx_item_stages(c, cu.it);
    cu.wok = c.sh->ok_u[cu.it.u] != 0;
  }
}
__device__ __forceinline__ void cur_next(const DmxCtx& c, DmxCursor& cu) {
  if (++cu.j >= cu.nst) cur_enter(c, cu, cu.li + 1);
}
__device__ __forceinline__ bool cur_valid(const DmxCtx& c, const DmxCursor& cu) { return cu.li < dmx_nitems(*c.sh); }

// ---------------------------------------------------------------- producers --
// Six warps, lane 0 each, one (role, stage parity) pair per warp: role 0
// and role 1 copy their own of the stage's two code boxes (gate and up, or
// the down slices 2j and 2j + 1), role 2 the B tiles (the tokens' terms, or
// the h terms once the expert's h tiles are ready), each for the even or the
// odd stages.  Each claims its stages and arms their barrier with its own
// bytes (an arrival without bytes where it has none); code boxes of an
// expert whose codes cannot be mapped (flagged in the prologue) are not
// copied.
__device__ void dmx_producer(const ExpertParams& p, const DmxCtx& c, const DmxMaps* mp, int role, int odd) {
  DmxShared& sh = *c.sh;
  constexpr int S = dmx::kStages;
  int issued[S];
#pragma unroll
  for (int i = 0; i < S; ++i) issued[i] = -1;
  const uint32_t* hready = dmx_hready(p.ws);
  // The maps of all active experts are built by the CTAs together (three
  // per expert, a share each): the code roles wait until all are published.
  if (role < 2 && !dmx_wait_count(c, dmx_mapcnt(p.ws), 3u * (uint32_t)sh.U)) return;
  DmxCursor cu;
  cur_enter(c, cu, 0);
  int gs = 0;
  if (odd && cur_valid(c, cu)) {
    cur_next(c, cu);
    gs = 1;
  }
  int seen_li = -1;  // item entered (maps acquired, or h tiles known ready)
  bool ok = true;
  while (ok && cur_valid(c, cu)) {
    const DmxItem& it = cu.it;
    // Code box of this role: gate/up: matrix `role`; down: slice 2j + role.
    const uint8_t* ma = c.maps + (size_t)(it.map + (it.gu ? role : 0)) * 128;
    if (role < 2 && cu.li != seen_li) {
      if (cu.wok) tmap_acquire(ma);
      seen_li = cu.li;
    }
    if (role == 2 && !it.gu && cu.li != seen_li) {
      if (!dmx_wait_h_ready(c, hready + (size_t)it.u * c.d.rt)) {
        ok = false;  // the abort flag is set: the other roles stop too
        break;
      }
      fence_async_global();
      seen_li = cu.li;
    }
    if (!dmx_claim(c, gs, dmx::kPollTma)) {
      ok = false;
      break;
    }
    const int st = gs % S;
    uint8_t* sb = c.ring + (size_t)st * dmx::kStage;
    uint64_t* bar = &sh.full[st];
    if (role < 2) {
      const int s = it.gu ? cu.j : 2 * cu.j + role;
      if (cu.wok && (it.gu || s < c.d.rt)) {
        mbar_arrive_expect_tx(bar, (uint32_t)dmx::kCodeTx);
        tma_load_2d(sb + role * dmx::kBox, ma, s * dmx::kSliceK, it.r * 128, bar);
      } else {
        mbar_arrive(bar);
      }
    } else if (it.gu) {
      mbar_arrive_expect_tx(bar, (uint32_t)dmx::kBGu);
      tma_load_2d(sb + 2 * dmx::kBox, &mp->xq, cu.j * dmx::kSliceK, 0, bar);
    } else {
      const int sa = 2 * cu.j, sbn = 2 * cu.j + 1;
      const bool two = sbn < c.d.rt;
      mbar_arrive_expect_tx(bar, (two ? 2u : 1u) * (uint32_t)dmx::kBDn);
      tma_load_2d(sb + 2 * dmx::kBox, &mp->hq, sa * dmx::kSliceK, 3 * it.b0, bar);
      if (two) tma_load_2d(sb + 2 * dmx::kBox + dmx::kBDn, &mp->hq, sbn * dmx::kSliceK, 3 * it.b0, bar);
    }
#pragma unroll
    for (int i = 0; i < S; ++i)
      if (i == st) issued[i] = gs / S;
    cur_next(c, cu);
    ++gs;
    if (cur_valid(c, cu)) {  // every other stage
      cur_next(c, cu);
      ++gs;
    }
    if (*(volatile int*)&sh.abort_flag) ok = false;
  }
  // Every copy issued has landed before the CTA may exit.
#pragma unroll
  for (int i = 0; i < S; ++i)
    if (issued[i] >= 0 && !mbar_wait(&sh.full[i], issued[i] & 1)) set_status(c.hdr, MOE_ERR_TIMEOUT);
}

// ------------------------------------------------------------- scale warps --
// Warp quarter q writes lanes 32q..32q+31: first the gate/up B scales (B row
// 2t: 2^0, row 2t + 1: 2^-4, the same word in every quarter); then per stage
// the A scale words of rows lane + 32 i (i = 0..3) of both boxes (gate and
// up, or the two down slices); a down stage also gets the B scale words of B
// row `lane` (h row 3 b0 + lane) of its slices, read for the whole item once
// its expert's h tiles are ready.  The A scale words come in chunks (a
// gate/up tile's slices `spp` at a time; a down item's I / 128 words): the
// 128 scale threads copy row tid's words of the next chunk into shared
// memory with 4-byte cp.async while the current chunk runs (two buffers),
// and row tid's flag of an E8M0 code 255 (NaN) is kept per item for the
// epilogue.
__device__ __forceinline__ void dmx_cp4(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
// Chunk (li, k): slices [k spp, min(ns, (k + 1) spp)) of gate/up item li, or
// all of down item li (k = 0).
__device__ __forceinline__ void dmx_chunk_next(const DmxCtx& c, int& li, int& k) {
  const int n = dmx_nitems(*c.sh);
  if (li >= n) return;
  if (li < c.sh->n_gu && (k + 1) * c.d.spp < c.d.ns_gu) {
    ++k;
  } else {
    ++li;
    k = 0;
  }
}
__device__ void dmx_load_chunk(const ExpertParams& p, const DmxCtx& c, int li, int k, int b, int tid) {
  DmxShared& sh = *c.sh;
  if (li < dmx_nitems(sh)) {
    const DmxItem it = dmx_item(c, li);
    if (sh.ok_u[it.u]) {
      const moe_expert& ex = p.experts[it.e];
      const int row = it.r * 128 + tid;
      if (it.gu) {
        const int srow = p.H / 32, w0 = k * c.d.spp;
        const int nw = (c.d.ns_gu - w0) < c.d.spp ? c.d.ns_gu - w0 : c.d.spp;
        const uint32_t* g = reinterpret_cast<const uint32_t*>(ex.gate.s + (size_t)row * srow) + w0;
        const uint32_t* u = reinterpret_cast<const uint32_t*>(ex.up.s + (size_t)row * srow) + w0;
        for (int w = 0; w < nw; ++w) {
          dmx_cp4(&sh.sbuf[b][0][w][tid], g + w);
          dmx_cp4(&sh.sbuf[b][1][w][tid], u + w);
        }
      } else {
        const uint32_t* dsc = reinterpret_cast<const uint32_t*>(ex.down.s + (size_t)row * (p.I / 32));
        for (int w = 0; w < c.d.rt; ++w) dmx_cp4(&sh.sbuf[b][0][w][tid], dsc + w);
      }
    }
  }
  cp_async_mbar_arrive(&sh.sbar[b]);
}
__device__ __forceinline__ uint32_t dmx_nan_bytes(uint32_t v) {
  // A byte equal to 0xFF: all of its bits set (per-byte test without carries).
  return (v & (v >> 1) & (v >> 2) & (v >> 3) & (v >> 4) & (v >> 5) & (v >> 6) & (v >> 7)) & 0x01010101u;
}

__device__ void dmx_scales(const ExpertParams& p, const DmxCtx& c, uint32_t tmem) {
  const int q = (threadIdx.x >> 5) & 3, lane = threadIdx.x & 31;
  const int wq = (threadIdx.x >> 5) - dmx::kSfWarp0;
  const int tid = wq * 32 + lane;  // 0..127: the row this thread copies and checks
  const uint32_t lbase = tmem + ((uint32_t)(q * 32) << 16);
  {
    const uint32_t v = (lane & 1) ? 0x7B7B7B7Bu : 0x7F7F7F7Fu;
    tmem_st4(lbase + dmx::kColSfbGu, v, v, v, v);
  }
  DmxShared& sh = *c.sh;
  const uint32_t* hready = dmx_hready(p.ws);
  const int nhrows = 3 * p.T * p.k, rt = c.d.rt;
  uint32_t* sfbw = sh.sfbw[wq];  // [16 slices][32 lanes]
  const int n = dmx_nitems(sh);
  dmx_load_chunk(p, c, 0, 0, 0, tid);
  int nli = 0, nk = 0;  // the chunk after the current one
  dmx_chunk_next(c, nli, nk);
  int gs = 0, ch = 0;
  uint32_t nan_acc = 0u;
  bool ok = true;
  for (int li = 0; li < n && ok; ++li) {
    const DmxItem it = dmx_item(c, li);
    const bool wok = sh.ok_u[it.u] != 0;
    if (!it.gu) {
      // The expert's h tiles: lane r polls tile r.
      bool got = true;
      if (lane < rt) got = dmx_wait_count(c, hready + (size_t)it.u * rt + lane, 4u);
      if (!__all_sync(0xFFFFFFFFu, got)) {
        ok = false;
        break;
      }
      const int hr = 3 * it.b0 + lane;
      const uint32_t* hs = reinterpret_cast<const uint32_t*>(p.ws.dmx_hs) + (size_t)hr * (p.I / 128);
      uint32_t v[16];
#pragma unroll
      for (int sl = 0; sl < 16; ++sl) v[sl] = (sl < rt && hr < nhrows) ? __ldcg(hs + sl) : 0x7F7F7F7Fu;
#pragma unroll
      for (int sl = 0; sl < 16; ++sl) sfbw[sl * 32 + lane] = v[sl];
      __syncwarp();
    }
    const int nchunks = it.gu ? (c.d.ns_gu + c.d.spp - 1) / c.d.spp : 1;
    for (int k = 0; k < nchunks && ok; ++k, ++ch) {
      const int b = ch & 1;
      // The next chunk's words into the other buffer, once every warp has
      // read chunk ch - 1 from it.
      if (ch >= 1 && !dmx_warp_wait(c, &sh.sfree[(ch - 1) & 1], ((ch - 1) >> 1) & 1, dmx::kPollSf)) {
        ok = false;
        break;
      }
      dmx_load_chunk(p, c, nli, nk, b ^ 1, tid);
      dmx_chunk_next(c, nli, nk);
      if (!dmx_warp_wait(c, &sh.sbar[b], (ch >> 1) & 1, dmx::kPollSf)) {
        ok = false;
        break;
      }
      const int s0 = it.gu ? k * c.d.spp : 0;
      const int nw = it.gu ? ((c.d.ns_gu - s0) < c.d.spp ? c.d.ns_gu - s0 : c.d.spp) : rt;
      if (wok) {
        for (int w = 0; w < nw; ++w) {
          nan_acc |= dmx_nan_bytes(sh.sbuf[b][0][w][tid]);
          if (it.gu) nan_acc |= dmx_nan_bytes(sh.sbuf[b][1][w][tid]);
        }
      }
      if (k == nchunks - 1) {
        sh.nanf[li % dmx::kNanRing][tid] = nan_acc != 0u ? 1 : 0;
        nan_acc = 0u;
      }
      const int nst = it.gu ? nw : (rt + 1) / 2;
      for (int j = 0; j < nst; ++j, ++gs) {
        // Words of this stage: box 0 (gate / slice 2j), box 1 (up / slice 2j + 1).
        int m1, w0, w1;
        if (it.gu) {
          m1 = 1;
          w0 = w1 = j;
        } else {
          m1 = 0;
          w0 = 2 * j;
          w1 = 2 * j + 1 < rt ? 2 * j + 1 : 2 * j;
        }
        uint32_t a[4], u[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          a[i] = wok ? sh.sbuf[b][0][w0][lane + 32 * i] : 0x7F7F7F7Fu;
          u[i] = wok ? sh.sbuf[b][m1][w1][lane + 32 * i] : 0x7F7F7F7Fu;
        }
        const bool claimed = dmx_claim(c, gs, dmx::kPollSf);
        if (!__all_sync(0xFFFFFFFFu, claimed)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const int st = gs % dmx::kStages;
        tmem_st4(lbase + dmx::kColSfa + 8 * st, a[0], a[1], a[2], a[3]);
        tmem_st4(lbase + dmx::kColSfa + 8 * st + 4, u[0], u[1], u[2], u[3]);
        if (!it.gu) {
          const uint32_t b0w = sfbw[(2 * j) * 32 + lane];
          const uint32_t b1w = 2 * j + 1 < rt ? sfbw[(2 * j + 1) * 32 + lane] : 0x7F7F7F7Fu;
          tmem_st4(lbase + dmx::kColSfbDn + 8 * st, b0w, b0w, b0w, b0w);
          tmem_st4(lbase + dmx::kColSfbDn + 8 * st + 4, b1w, b1w, b1w, b1w);
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sh.full[st]);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh.sfree[b]);
    }
    if (*(volatile int*)&sh.abort_flag) ok = false;
  }
  // No cp.async of this thread may still be landing when the CTA exits.
  cp_async_wait_all();
  tmem_st_wait();
}

// ------------------------------------------------------------------- MMAs --
// Issuer w (0: warp 0, 1: warp 10), lane 0.  Per item: wait until its
// accumulator buffer (item parity) is drained; per stage: gate/up issue the
// four K = 32 steps of box w (gate or up) against the tokens' terms, down
// those of slice 2 j + w against the h terms; commit the stage; after the
// item commit the buffer.
__device__ void dmx_mma(const ExpertParams& p, const DmxCtx& c, uint32_t tmem, int w) {
  DmxShared& sh = *c.sh;
  const int n = dmx_nitems(sh);
  int ci = 0, gs = 0;
  bool ok = true;
  for (int li = 0; li < n && ok; ++li, ++ci) {
    const DmxItem it = dmx_item(c, li);
    const int b = ci & 1, use = ci >> 1;
    if (use >= 1 && !dmx_wait(c, &sh.acce[b], (use - 1) & 1, dmx::kPollMma)) {
      ok = false;
      break;
    }
    tc_fence_after();
    const uint32_t d = tmem + (uint32_t)b * 2 * dmx::kAccN + (uint32_t)w * dmx::kAccN;
    const uint32_t ibase = idesc_mx_f32(128, it.gu ? kDmxNGu : kDmxNDn, kMxE2M1, kMxE4M3, 0, 0);
    const int nst = dmx_item_stages(c, it);
    for (int j = 0; j < nst; ++j, ++gs) {
      const int st = gs % dmx::kStages;
      if (!dmx_wait(c, &sh.full[st], (gs / dmx::kStages) & 1, dmx::kPollMma)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t sbase = smem_u32(c.ring + (size_t)st * dmx::kStage);
      const uint32_t sfa = tmem + dmx::kColSfa + 8u * st + 4u * w;
      const bool run = it.gu || 2 * j + w < c.d.rt;
      if (run) {
        const uint32_t abase = sbase + (uint32_t)w * dmx::kBox;
        const uint32_t bbase = sbase + 2 * dmx::kBox + (it.gu ? 0u : (uint32_t)w * dmx::kBDn);
        const uint32_t sfb = it.gu ? tmem + dmx::kColSfbGu : tmem + dmx::kColSfbDn + 8u * st + 4u * w;
#pragma unroll
        for (int kb = 0; kb < 4; ++kb) {
          const uint32_t idesc = ibase | ((uint32_t)kb << 29) | ((uint32_t)kb << 4);
          umma_mx(d, sdesc_sw128(abase + 32 * kb), sdesc_sw128(bbase + 32 * kb), idesc, sfa, sfb,
                  (j > 0 || kb > 0) ? 1u : 0u);
        }
      }
      umma_commit(&sh.empty[st]);
    }
    umma_commit(&sh.accf[b]);
  }
  // Every MMA issued must have finished before Tensor Memory is released.
  if (ci > 0 && !mbar_wait(&sh.accf[(ci - 1) & 1], ((ci - 1) >> 1) & 1)) set_status(c.hdr, MOE_ERR_TIMEOUT);
}

// --------------------------------------------------------------- epilogue --
// The pair's h (fp32, one value per lane = one row of a 32-row block) as
// three E4M3 terms with the block's scale: tau = 7 - floor(log2 max|h|) over
// the block (clamped so that every term's E8M0 scale 127 - tau - 4 q is a
// code); a block holding an infinity or NaN becomes NaN.
__device__ __forceinline__ void dmx_h_terms(float h, int lane, uint8_t* row0, size_t rstride, uint8_t* s0,
                                            size_t sstride) {
  const uint32_t a = __float_as_uint(h) & 0x7FFFFFFFu;
  const uint32_t m = __reduce_max_sync(0xFFFFFFFFu, a);
  const bool bad = m >= 0x7F800000u;
  int tau = (m == 0u || bad) ? 0 : 7 - ((int)(m >> 23) - 127);
  tau = tau > 119 ? 119 : (tau < -126 ? -126 : tau);
  uint32_t q1 = 0x7Fu, q2 = 0x7Fu, q3 = 0x7Fu;
  if (!bad) {
    const float v = h * __int_as_float((tau + 127) << 23);
    q1 = dmx_e4m3(v);
    const float r1 = (v - dmx_e4m3_value(q1)) * 16.f;
    q2 = dmx_e4m3(r1);
    q3 = dmx_e4m3((r1 - dmx_e4m3_value(q2)) * 16.f);
  }
  row0[lane] = (uint8_t)q1;
  row0[rstride + lane] = (uint8_t)q2;
  row0[2 * rstride + lane] = (uint8_t)q3;
  if (lane < 3) s0[lane * sstride] = (uint8_t)(bad ? 127 : 127 - tau - 4 * lane);
}

// Warp quarter q drains TMEM lanes 32q..32q+31 (rows 32q + lane of the
// item's 128-row tile).
//   gate/up: h = silu(g 2^-tau_t) (u 2^-tau_t) of each routed pair, as E4M3
//            terms with block scales (dmx_h_terms), then the tile's
//            readiness count is raised;
//   down:    y[pair][row] = w(pair) * (sum of the pair's three term columns).
// A row with a NaN block scale (E8M0 code 255) gives NaN, as the definition
// of the format has it (flagged by the scale warps).
__device__ void dmx_epilogue(const ExpertParams& p, const DmxCtx& c, uint32_t tmem) {
  DmxShared& sh = *c.sh;
  const int q = (threadIdx.x >> 5) & 3, lane = threadIdx.x & 31;
  const int n = dmx_nitems(sh);
  const int k = p.k, H = p.H, I = p.I, rt = c.d.rt;
  uint32_t* hready = dmx_hready(p.ws);
  int ci = 0;
  for (int li = 0; li < n; ++li, ++ci) {
    const DmxItem it = dmx_item(c, li);
    const bool wok = sh.ok_u[it.u] != 0;
    const int tr = q * 32 + lane;  // row within the tile
    const int row = it.r * 128 + tr;
    const int b = ci & 1;
    if (!dmx_warp_wait(c, &sh.accf[b], (ci >> 1) & 1, dmx::kPollEp)) break;
    tc_fence_after();
    const bool nan_row = wok && sh.nanf[li % dmx::kNanRing][tr] != 0;
    const uint32_t tb = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)b * 2 * dmx::kAccN;
    if (it.gu) {
      uint32_t g[kDmxNGu], u[kDmxNGu];
      tmem_ld16(tb, g);
      tmem_ld16(tb + dmx::kAccN, u);
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh.acce[b]);
      // B columns 2t (x1) and 2t + 1 (x2 / 16) of token t.
      for (int j = 0; j < it.cnt; ++j) {
        const int pr = c.pairs[it.b0 + j];
        if (pr < 0) continue;
        const int t = pr / k;
        float gs = 0.f, us = 0.f;
#pragma unroll
        for (int tt = 0; tt < kDmxMaxT; ++tt)
          if (tt == t) {
            gs = __uint_as_float(g[2 * tt]) + __uint_as_float(g[2 * tt + 1]);
            us = __uint_as_float(u[2 * tt]) + __uint_as_float(u[2 * tt + 1]);
          }
        const float xs = __ldg(&p.ws.x8scale[t]);
        float h = wok ? silu_f32(gs * xs) * (us * xs) : 0.f;
        if (nan_row) h = __int_as_float(0x7FC00000);
        const size_t hr = (size_t)3 * (it.b0 + j);
        dmx_h_terms(h, lane, p.ws.dmx_hq + hr * I + it.r * 128 + q * 32, (size_t)I,
                    p.ws.dmx_hs + hr * (I / 32) + it.r * 4 + q, (size_t)(I / 32));
      }
      fence_async_global();
      __threadfence();
      __syncwarp();
      if (lane == 0) atomicAdd(&hready[(size_t)it.u * rt + it.r], 1u);
    } else {
      uint32_t a0[kDmxNDn], a1[kDmxNDn];
      tmem_ld32(tb, a0);
      tmem_ld32(tb + dmx::kAccN, a1);
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh.acce[b]);
      for (int j = 0; j < it.cnt; ++j) {
        const int pr = c.pairs[it.b0 + j];
        if (pr < 0) continue;
        // B columns 3 j + m hold term m of pair j (scales applied); smaller
        // terms first.
        float y = 0.f;
#pragma unroll
        for (int jj = 0; jj < kDmxMaxT; ++jj)
          if (jj == j) {
            const float t3 = __uint_as_float(a0[3 * jj + 2]) + __uint_as_float(a1[3 * jj + 2]);
            const float t2 = __uint_as_float(a0[3 * jj + 1]) + __uint_as_float(a1[3 * jj + 1]);
            const float t1 = __uint_as_float(a0[3 * jj]) + __uint_as_float(a1[3 * jj]);
            y = (t3 + t2) + t1;
          }
        if (!wok) y = 0.f;
        if (nan_row) y = __int_as_float(0x7FC00000);
        p.ws.y[(size_t)pr * H + row] = c.wts[pr] * y;
      }
    }
  }
  __threadfence();  // the rows written here before this CTA reports done
}

// ------------------------------------------------------------------ kernel --
// Dynamic shared memory: the stage ring (the routing scratch aliases it),
// then the plan: ue, ub0, un [umax], pairs [T k], weights [T k].
__global__ void __launch_bounds__(dmx::kThreads, 1) k_dec_mx(ExpertParams p, const __grid_constant__ DmxMaps maps) {
  extern __shared__ uint8_t dmx_dyn[];
  __shared__ DmxShared sh;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int T = p.T, k = p.k, npairs = T * k;
  const DmxDims d = dmx_dims(T, p.H, p.E, p.I, k);
  uint8_t* ring = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dmx_dyn) + 1023) & ~(uintptr_t)1023);
  int* ue = reinterpret_cast<int*>(ring + (size_t)dmx::kStages * dmx::kStage);
  int* ub0 = ue + d.umax;
  int* un = ub0 + d.umax;
  int* pairs = un + d.umax;
  float* wts = reinterpret_cast<float*>(pairs + npairs);
  if (warp == 0) {
    tmem_alloc(&sh.tmem_base, dmx::kTmemCols);
    tmem_relinquish();
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < dmx::kStages; ++s) {
      mbar_init(&sh.full[s], dmx::kProducers + dmx::kSfWarps);
      mbar_init(&sh.empty[s], 2);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sh.accf[b], 2);
      mbar_init(&sh.acce[b], dmx::kEpWarps);
      mbar_init(&sh.sbar[b], 32 * dmx::kSfWarps);
      mbar_init(&sh.sfree[b], dmx::kSfWarps);
    }
    sh.abort_flag = 0;
    mbar_init_fence();
  }
  if (threadIdx.x < kDmxMaxT) {
    sh.tok_mask[threadIdx.x] = 0u;
    sh.tok_cnt[threadIdx.x] = 0;
  }
  pdl_wait();
  pdl_trigger();
  // ---- the plan: routed here, or the published one
  if (p.fused_route) {
    SmallPlan sp;
    sp.ue = ue;
    sp.ub0 = ub0;
    sp.un = un;
    sp.pairs = pairs;
    sp.wts = wts;
    route_small(p.rp, reinterpret_cast<char*>(ring), sp, blockIdx.x == 0);
    if (threadIdx.x == 0) sh.U = sp.U;
    // The scratch's generic writes before the copies (async proxy) into the ring.
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  } else {
    const int U = (int)p.ws.hdr->n_active;
    for (int u = threadIdx.x; u < U; u += blockDim.x) {
      const int e = p.ws.act_e[u];
      const int b0 = p.offsets[e];
      ue[u] = e;
      ub0[u] = b0;
      un[u] = p.offsets[e + 1] - b0;
    }
    for (int i = threadIdx.x; i < npairs; i += blockDim.x) {
      int v = p.sorted[i];
      if (v < 0 || v >= npairs) {
        set_status(p.ws.hdr, MOE_ERR_DEVICE_CHECK);
        v = -1;
      }
      pairs[i] = v;
      wts[i] = p.w[i];
    }
    if (threadIdx.x == 0) sh.U = U;
  }
  __syncthreads();
  for (int i = threadIdx.x; i < npairs; i += blockDim.x) {
    const int v = pairs[i];
    if (v >= 0) {
      atomicOr(&sh.tok_mask[v / k], 1u << (v % k));
      atomicAdd(&sh.tok_cnt[v / k], 1);
    }
  }
  // ---- this CTA's items (see dmx_item) and the experts' usable descriptors
  {
    const int U = sh.U, G = gridDim.x, cb = blockIdx.x;
    for (int u = threadIdx.x; u < U; u += blockDim.x) {
      const moe_expert ex = p.experts[ue[u]];
      const uintptr_t q = (uintptr_t)ex.gate.q | (uintptr_t)ex.up.q | (uintptr_t)ex.down.q;
      sh.ok_u[u] = (expert_ptrs_ok(ex) && (q & 31u) == 0) ? 1 : 0;
    }
    if (threadIdx.x == 0) {
      // Gate/up tiles in waves: h CTAs carry one tile more (heavy).  Down
      // items: x_h rounds to every CTA, then rounds to the nl light CTAs, so
      // that a heavy CTA's extra tile (2 H / I down items' worth of weight
      // bytes) is offset.
      const int n_tiles = U * d.rt, n_dn = U * d.rh;
      const int h = n_tiles % G, bt = n_tiles / G;
      int x_h = 0, nl = G;
      if (h != 0) {
        const int bg = 2 * d.ns_gu, bd = d.rt;
        const int delta = (bg + bd / 2) / bd;
        nl = G - h;
        x_h = (n_dn - nl * delta) / G;
        x_h = x_h < 0 ? 0 : x_h;
      }
      const int rem = n_dn - h * x_h, base_l = rem / nl, extra_l = rem % nl;
      sh.n_gu = bt + (cb < h ? 1 : 0);
      sh.n_dn = cb < h ? x_h : base_l + (cb >= G - extra_l ? 1 : 0);
      sh.x_h = x_h;
      sh.nl = nl;
    }
  }
  __syncthreads();
  // ---- the tensor maps of the active experts' codes, [E][3] in the
  // workspace: map i (expert u = i / 3, matrix i % 3) is built by CTA
  // i % G; each CTA then adds its count to the published total.
  {
    const int U = sh.U, G = gridDim.x;
    int mine = 0;
    for (int i = blockIdx.x; i < 3 * U; i += G) ++mine;
    const int i = blockIdx.x + (int)threadIdx.x * G;
    if ((int)threadIdx.x < mine) {
      const int u = i / 3, a = i - 3 * (i / 3);
      const int e = ue[u];
      if (!sh.ok_u[u]) {
        set_status(p.ws.hdr, MOE_ERR_DEVICE_CHECK);
      } else {
        const moe_expert ex = p.experts[e];
        const uint8_t* q = a == 0 ? ex.gate.q : (a == 1 ? ex.up.q : ex.down.q);
        uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<uint8_t*>(p.ws.tmaps) + (size_t)(3 * e + a) * 128);
        const uint4* src = reinterpret_cast<const uint4*>(a < 2 ? &maps.gu : &maps.dn);
#pragma unroll
        for (int j = 0; j < 8; ++j) dst[j] = src[j];
        asm volatile("tensormap.replace.tile.global_address.global.b1024.b64 [%0], %1;" ::"l"(dst), "l"(q) : "memory");
        asm volatile("fence.proxy.tensormap::generic.release.gpu;" ::: "memory");
      }
      __threadfence();
    }
    __syncthreads();
    if (threadIdx.x == 0 && mine > 0) atomicAdd(dmx_mapcnt(p.ws), (uint32_t)mine);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  DmxCtx c;
  c.sh = &sh;
  c.ring = ring;
  c.ue = ue;
  c.ub0 = ub0;
  c.un = un;
  c.pairs = pairs;
  c.wts = wts;
  c.d = d;
  c.maps = reinterpret_cast<const uint8_t*>(p.ws.tmaps);
  c.hdr = p.ws.hdr;
  c.wait_limit = p.wait_limit;
  const uint32_t tmem = sh.tmem_base;
  if (warp == 0 || warp == dmx::kMma2Warp) {
    if (lane == 0) dmx_mma(p, c, tmem, warp == 0 ? 0 : 1);
  } else if (warp == dmx::kTmaWarp || warp >= dmx::kTma2Warp) {
    int role, odd;
    if (warp == dmx::kTmaWarp) {
      role = 0;
      odd = 0;
    } else if (warp == dmx::kTma2Warp) {
      role = 1;
      odd = 0;
    } else if (warp < dmx::kTmaOddWarp) {
      role = 2;
      odd = warp - dmx::kTmaBWarp;
    } else {
      role = warp - dmx::kTmaOddWarp;
      odd = 1;
    }
    if (lane == 0) dmx_producer(p, c, &maps, role, odd);
  } else if (warp < dmx::kEpWarp0) {
    dmx_scales(p, c, tmem);
  } else {
    dmx_epilogue(p, c, tmem);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, dmx::kTmemCols);
  }
  // ---- the combine: once every CTA is done, CTA b adds rows [b T H / G,
  // (b + 1) T H / G) of the tokens' k weighted rows, in slot order, into out.
  __shared__ int all_done;
  if (threadIdx.x == 0) {
    __threadfence();
    atomicAdd(dmx_donecnt(p.ws), 1u);
    all_done = dmx_wait_count(c, dmx_donecnt(p.ws), gridDim.x) ? 1 : 0;
  }
  __syncthreads();
  if (!all_done) return;
  __threadfence();
  const long long tot = (long long)T * p.H;
  const long long i0 = tot * blockIdx.x / gridDim.x, i1 = tot * (blockIdx.x + 1) / gridDim.x;
  for (long long i = i0 + threadIdx.x; i < i1; i += blockDim.x) {
    const int t = (int)(i / p.H), row = (int)(i - (long long)t * p.H);
    const uint32_t m = sh.tok_mask[t];
    const float* ys = p.ws.y + (size_t)t * k * p.H + row;
    float v[kMaxK];
#pragma unroll
    for (int sl = 0; sl < kMaxK; ++sl) v[sl] = (sl < k && ((m >> sl) & 1u)) ? __ldcg(ys + (size_t)sl * p.H) : 0.f;
    float s = 0.f;
#pragma unroll
    for (int sl = 0; sl < kMaxK; ++sl)
      if (sl < k && ((m >> sl) & 1u)) s += v[sl];
    p.out[i] = p.accumulate ? p.out[i] + s : s;
  }
}

// The preparation for a call whose route is given (no router kernel ran):
// the tokens' E4M3 terms and the counters.
__global__ void __launch_bounds__(256) k_dec_mx_prepare(ExpertParams p) {
  dmx_prepare(p.x, p.T, p.H, p.E, p.I, p.k, p.ws, blockIdx.x, gridDim.x);
}

// ------------------------------------------------------------------- host --
namespace {
cudaError_t encode_bytes_map(CUtensorMap* m, void* base, int K, int rows, int box_rows) {
  const EncodeTiledFn enc = encode_tiled_fn();
  if (!enc) return cudaErrorNotSupported;
  const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)K};
  const cuuint32_t box[2] = {(cuuint32_t)dmx::kSliceK, (cuuint32_t)box_rows};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, base, dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

size_t dmx_smem_bytes(const ExpertParams& p) {
  const DmxDims d = dmx_dims(p.T, p.H, p.E, p.I, p.k);
  const size_t npairs = (size_t)p.T * p.k;
  return 1024 + (size_t)dmx::kStages * dmx::kStage + (size_t)(3 * d.umax + 2 * npairs) * 4;
}
}  // namespace

bool dmx_shape_supported(int T, int H, int E, int I, int k) {
  return dmx_shape_ok(T, H, I) && k >= 1 && k <= kMaxK && E <= 4096 && T * k <= 256 && I / 128 <= 16 &&
         dmx_spp(H / 128) <= 16 && route_decode_supported(T, H, E, k);
}

bool dmx_supported(const ExpertParams& p) {
  if (!p.x_bf16 || !dmx_shape_supported(p.T, p.H, p.E, p.I, p.k)) return false;
  const int G = device_sm_count();
  if (G < 1 || 3 * 256 > G * 352) return false;  // every map-building CTA builds at most blockDim maps
  if (dmx_smem_bytes(p) + sizeof(DmxShared) > 227 * 1024) return false;
  if (route_small_scratch_bytes(p.E, dmx::kThreads / 32, p.T) > (size_t)dmx::kStages * dmx::kStage) return false;
  return encode_tiled_fn() != nullptr;
}

cudaError_t launch_dec_mx(const ExpertParams& p, cudaStream_t s) {
  DmxMaps maps;
  memset(&maps, 0, sizeof maps);
  cudaError_t err;
  if ((err = encode_code_map_template(&maps.gu, p.ws.tmaps, p.H, p.I)) != cudaSuccess) return err;
  if ((err = encode_code_map_template(&maps.dn, p.ws.tmaps, p.I, p.H)) != cudaSuccess) return err;
  if ((err = encode_bytes_map(&maps.xq, p.ws.dmx_xq, p.H, 2 * p.T, kDmxNGu)) != cudaSuccess) return err;
  if ((err = encode_bytes_map(&maps.hq, p.ws.dmx_hq, p.I, 3 * p.T * p.k, kDmxNDn)) != cudaSuccess) return err;
  if (!p.fused_route) {
    k_dec_mx_prepare<<<p.T, 256, 0, s>>>(p);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
  }
  const size_t smem = dmx_smem_bytes(p);
  if ((err = ensure_smem_attr((const void*)k_dec_mx, smem)) != cudaSuccess) return err;
  prof_before(MOE_STAGE_GATEUP, s);
  err = launch_pdl(k_dec_mx, dim3(device_sm_count()), dim3(dmx::kThreads), smem, s, p, maps);
  prof_after(MOE_STAGE_GATEUP, s);
  prof_before(MOE_STAGE_DOWN, s);
  prof_after(MOE_STAGE_DOWN, s);
  return err;
}

}  // namespace moe
