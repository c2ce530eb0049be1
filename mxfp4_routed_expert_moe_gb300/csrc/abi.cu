// abi.cu — the exported C entry points: argument validation, workspace
// layout, and the launch sequence of each call.  Nothing here allocates or
// synchronises except moe_device_status().
#include <string.h>


#include "async.cuh"
#include "kernels.h"

using namespace moe;

namespace moe {
ProfHook g_prof = {};
}

namespace {
// Cycles before a bounded device wait gives up (moe_set_wait_limit; the
// default only ends waits that can never complete).
long long g_wait_limit = kWaitCycles;
}  // namespace

namespace {

bool aligned(const void* p, size_t a) { return ((uintptr_t)p % a) == 0; }

int validate_shape(const moe_shape* s) {
  if (!s) return MOE_ERR_INVALID_ARG;
  if (s->T < 1 || s->H < 32 || s->I < 32 || s->E < 1 || s->k < 1) return MOE_ERR_INVALID_ARG;
  if (s->H % 32 != 0 || s->I % 32 != 0 || s->k > s->E) return MOE_ERR_INVALID_ARG;
  if (s->k > kMaxK || s->T > 65536 || s->H > 16384 || s->I > 8192 || s->E > 65536) return MOE_ERR_UNSUPPORTED;
  if (s->k * (s->I / 32) > 1024) return MOE_ERR_UNSUPPORTED;
  if ((int64_t)s->T * s->k > (1 << 24)) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

int check_ws(const moe_shape* s, void* ws, size_t ws_bytes) {
  if (!ws || !aligned(ws, 256)) return MOE_ERR_INVALID_ARG;
  if (ws_bytes < ws_layout(*s, nullptr).total) return MOE_ERR_WORKSPACE;
  return MOE_OK;
}

int cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

bool decode_experts_supported(const moe_shape* s, int x_dtype) {
  // Up to 64 tokens: every decode kernel family (decode gate/up keeps one
  // block column per thread, H <= 8192).  Larger bf16 batches: the staged
  // kernels only.
  if (s->T <= kDecodeMaxT) return s->H <= 8192;
  return x_dtype == MOE_DT_BF16 && decode_batch_supported(s->T, s->H, s->E, s->I, s->k);
}

// Resolve MOE_PATH_AUTO (the rule is stated with moe_path in the header) and
// check the chosen path's limits.
int resolve_path(const moe_shape* s, int x_dtype, bool has_shared, int path, int* out) {
  if (path == MOE_PATH_AUTO) {
    if (s->T <= kDecodeMaxT || x_dtype == MOE_DT_F32)
      path = MOE_PATH_DECODE;
    else if ((int64_t)s->T * s->k <= (int64_t)MOE_DECODE_AUTO_PAIRS_PER_EXPERT * s->E &&
             decode_experts_supported(s, x_dtype))
      path = MOE_PATH_DECODE;
    else
      path = MOE_PATH_PREFILL;
    // A shape the decode kernels do not take (e.g. H > 8192) runs on the
    // prefill path when that path takes it.
    if (path == MOE_PATH_DECODE && !decode_experts_supported(s, x_dtype) && x_dtype == MOE_DT_BF16 &&
        prefill_supported(s->H, s->I))
      path = MOE_PATH_PREFILL;
  }
  if (path == MOE_PATH_DECODE) {
    if (!decode_experts_supported(s, x_dtype)) return MOE_ERR_UNSUPPORTED;
    // The decode path runs a shared expert on the prefill kernels.
    if (has_shared && (x_dtype != MOE_DT_BF16 || !prefill_supported(s->H, s->I))) return MOE_ERR_UNSUPPORTED;
  } else if (path == MOE_PATH_PREFILL) {
    if (x_dtype != MOE_DT_BF16 || !prefill_supported(s->H, s->I)) return MOE_ERR_UNSUPPORTED;
  } else if (path == MOE_PATH_DECODE_MX) {
    if (x_dtype != MOE_DT_BF16 || !dmx_shape_supported(s->T, s->H, s->E, s->I, s->k)) return MOE_ERR_UNSUPPORTED;
    if (has_shared && !prefill_supported(s->H, s->I)) return MOE_ERR_UNSUPPORTED;
  } else {
    return MOE_ERR_INVALID_ARG;
  }
  *out = path;
  return MOE_OK;
}

BucketParams bucket_params(const moe_shape* s, const int32_t* ids, int32_t* offsets_out, int32_t* sorted_out,
                           const Ws& ws) {
  BucketParams b;
  b.T = s->T; b.E = s->E; b.k = s->k;
  b.ids = ids;
  b.offsets_out = offsets_out;
  b.sorted_out = sorted_out;
  b.n_tile = kPfNTileDn;
  b.n_tile_gu = kPfNTileGu;
  b.m_tiles_gu = (s->I + kPfMTile - 1) / kPfMTile;
  b.m_tiles_dn = (s->H + kPfMTile - 1) / kPfMTile;
  b.ws = ws;
  return b;
}

RouteParams route_params(const moe_shape* s, const void* x, int x_dtype, const float* wr, const float* br,
                         int32_t* ids, float* w, int32_t* offsets, int32_t* sorted, const Ws& ws) {
  RouteParams p;
  p.T = s->T; p.H = s->H; p.E = s->E; p.k = s->k;
  p.x = x;
  p.x_bf16 = x_dtype == MOE_DT_BF16;
  p.wr = wr;
  p.br = br;
  p.ids = ids;
  p.w = w;
  p.offsets = offsets;
  p.sorted = sorted;
  p.want_buckets = 1;
  p.dmx_I = 0;
  p.wait_limit = g_wait_limit;
  p.ws = ws;
  return p;
}

int do_route(const moe_shape* s, const void* x, int x_dtype, const float* wr, const float* br, int32_t* ids, float* w,
             int32_t* offsets, int32_t* sorted, const Ws& ws, bool want_decode_route, cudaStream_t st) {
  RouteParams p;
  p.T = s->T; p.H = s->H; p.E = s->E; p.k = s->k;
  p.x = x;
  p.x_bf16 = x_dtype == MOE_DT_BF16;
  p.wr = wr;
  p.br = br;
  p.ids = ids;
  p.w = w;
  p.offsets = offsets;
  p.sorted = sorted;
  p.want_buckets = 1;
  p.dmx_I = 0;
  p.wait_limit = g_wait_limit;
  p.ws = ws;
  if (want_decode_route && route_decode_supported(s->T, s->H, s->E, s->k)) return cuda_status(launch_route_decode(p, st));
  return cuda_status(launch_route_prefill(p, bucket_params(s, ids, offsets, sorted, ws), st));
}

ExpertParams expert_params(const moe_shape* s, const void* x, int x_dtype, const moe_expert* experts,
                           const int32_t* ids, const float* w, const int32_t* offsets, const int32_t* sorted,
                           float* out, int accumulate, const moe_dense_bf16* shared, const Ws& ws) {
  ExpertParams p;
  memset(&p, 0, sizeof p);
  p.T = s->T; p.H = s->H; p.E = s->E; p.I = s->I; p.k = s->k;
  p.x = x;
  p.x_bf16 = x_dtype == MOE_DT_BF16;
  p.experts = experts;
  p.ids = ids;
  p.w = w;
  p.offsets = offsets;
  p.sorted = sorted;
  p.out = out;
  p.accumulate = accumulate ? 1 : 0;
  p.wait_limit = g_wait_limit;
  if (shared) {
    p.sh_gate = shared->gate;
    p.sh_up = shared->up;
    p.sh_down = shared->down;
  }
  p.ws = ws;
  return p;
}

int run_experts(const ExpertParams& p, int path, cudaStream_t st) {
  if (path == MOE_PATH_DECODE_MX) {
    if (p.sh_gate) return MOE_ERR_UNSUPPORTED;
    if (!dmx_supported(p)) return MOE_ERR_UNSUPPORTED;
    return cuda_status(launch_dec_mx(p, st));
  }
  if (path == MOE_PATH_DECODE) {
    if (p.sh_gate) return MOE_ERR_UNSUPPORTED;
    return cuda_status(launch_decode_experts(p, st));
  }
  return cuda_status(launch_prefill_experts(p, st));
}

// Workspace of moe_forward_static_scratch: a fixed region in the library's own
// device memory (one instance per device), so that call allocates nothing.
static __device__ __align__(256) unsigned char g_static_scratch[MOE_STATIC_SCRATCH_BYTES];

// Device address of g_static_scratch in the current context, looked up on
// every call: a cached address would go stale after cudaDeviceReset or under
// another context on the same device.
int static_scratch_ptr(void** out) {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || !p) return MOE_ERR_CUDA;
  *out = p;
  return MOE_OK;
}

// Diagnostic of the bounded-wait mechanism: one thread waits, with the
// library's wait helper and a limit of max_cycles, on a barrier phase that
// never completes (two arrivals expected, one made), and records the outcome.
__global__ void k_wait_selftest(long long max_cycles, int* status) {
  __shared__ uint64_t bar;
  if (threadIdx.x != 0) return;
  mbar_init(&bar, 2);
  mbar_init_fence();
  mbar_arrive(&bar);
  *status = mbar_wait_for(&bar, 0, max_cycles) ? MOE_OK : MOE_ERR_TIMEOUT;
}

}  // namespace

extern "C" {

uint32_t moe_abi_version(void) { return MOE_ABI_VERSION; }

int moe_select_path(const moe_shape* shape, int x_dtype, int has_shared, int path, int* path_out) {
  int st = validate_shape(shape);
  if (st != MOE_OK) return st;
  if (!path_out || (x_dtype != MOE_DT_F32 && x_dtype != MOE_DT_BF16)) return MOE_ERR_INVALID_ARG;
  int rpath;
  if ((st = resolve_path(shape, x_dtype, has_shared != 0, path, &rpath)) != MOE_OK) return st;
  *path_out = rpath;
  return MOE_OK;
}

const char* moe_status_string(int status) {
  switch (status) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument (null or misaligned pointer, bad shape or enum)";
    case MOE_ERR_UNSUPPORTED: return "request outside the supported limits of this build";
    case MOE_ERR_WORKSPACE: return "workspace smaller than moe_workspace_bytes(shape)";
    case MOE_ERR_CUDA: return "a CUDA launch or query failed";
    case MOE_ERR_TIMEOUT: return "a bounded device wait gave up";
    case MOE_ERR_DEVICE_CHECK: return "device check failed: expert id or bucket entry out of range";
    case MOE_ERR_RANGE: return "reserved status (not raised by this version)";
    default: return "unknown status";
  }
}

size_t moe_workspace_bytes(const moe_shape* shape) {
  if (validate_shape(shape) != MOE_OK) return 0;
  return ws_layout(*shape, nullptr).total;
}

int moe_route(const moe_shape* shape, const void* x, int x_dtype, const float* w_router, const float* b_router,
              int32_t* ids, float* w, int32_t* offsets, int32_t* sorted_idx, void* ws, size_t ws_bytes, void* stream) {
  int st = validate_shape(shape);
  if (st != MOE_OK) return st;
  if ((st = check_ws(shape, ws, ws_bytes)) != MOE_OK) return st;
  if (x_dtype != MOE_DT_F32 && x_dtype != MOE_DT_BF16) return MOE_ERR_INVALID_ARG;
  if (!x || !w_router || !ids || !w) return MOE_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(w_router, 16) || !aligned(ids, 4) || !aligned(w, 4)) return MOE_ERR_INVALID_ARG;
  if ((b_router && !aligned(b_router, 4)) || (offsets && !aligned(offsets, 4)) || (sorted_idx && !aligned(sorted_idx, 4)))
    return MOE_ERR_INVALID_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  const Ws L = ws_layout(*shape, ws);
  if ((st = cuda_status(cudaMemsetAsync(L.hdr, 0, sizeof(WsHeader), s))) != MOE_OK) return st;
  return do_route(shape, x, x_dtype, w_router, b_router, ids, w, offsets, sorted_idx, L, shape->T <= kDecodeMaxT, s);
}

int moe_mxfp4_experts(const moe_shape* shape, const void* x, int x_dtype, const moe_expert* experts,
                      const int32_t* ids, const float* w, const int32_t* offsets, const int32_t* sorted_idx,
                      float* out, int accumulate, int path, void* ws, size_t ws_bytes, void* stream) {
  int st = validate_shape(shape);
  if (st != MOE_OK) return st;
  if ((st = check_ws(shape, ws, ws_bytes)) != MOE_OK) return st;
  if (x_dtype != MOE_DT_F32 && x_dtype != MOE_DT_BF16) return MOE_ERR_INVALID_ARG;
  if (!x || !experts || !ids || !w || !out) return MOE_ERR_INVALID_ARG;
  if ((offsets == nullptr) != (sorted_idx == nullptr)) return MOE_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(out, 16) || !aligned(experts, 8) || !aligned(ids, 4) || !aligned(w, 4))
    return MOE_ERR_INVALID_ARG;
  int rpath;
  if ((st = resolve_path(shape, x_dtype, false, path, &rpath)) != MOE_OK) return st;
  cudaStream_t s = (cudaStream_t)stream;
  const Ws L = ws_layout(*shape, ws);
  if ((st = cuda_status(cudaMemsetAsync(L.hdr, 0, sizeof(WsHeader), s))) != MOE_OK) return st;
  BucketParams b = bucket_params(shape, ids, nullptr, nullptr, L);
  if (offsets) {
    if ((st = cuda_status(launch_plan_from_offsets(b, offsets, s))) != MOE_OK) return st;
    // The kernels read a checked copy of the caller's pair list.
    if ((st = cuda_status(launch_copy_pairs(sorted_idx, L.sorted, shape->T * shape->k, L.hdr, s))) != MOE_OK)
      return st;
    sorted_idx = L.sorted;
  } else {
    if ((st = cuda_status(launch_bucket_from_ids(b, s))) != MOE_OK) return st;
    offsets = L.offsets;
    sorted_idx = L.sorted;
  }
  const ExpertParams p = expert_params(shape, x, x_dtype, experts, ids, w, offsets, sorted_idx, out, accumulate, nullptr, L);
  return run_experts(p, rpath, s);
}

int moe_forward(const moe_shape* shape, const void* x, int x_dtype, const float* w_router, const float* b_router,
                const moe_expert* experts, const moe_dense_bf16* shared, float* out, int accumulate, int32_t* ids_out,
                float* w_out, int path, void* ws, size_t ws_bytes, void* stream) {
  int st = validate_shape(shape);
  if (st != MOE_OK) return st;
  if ((st = check_ws(shape, ws, ws_bytes)) != MOE_OK) return st;
  if (x_dtype != MOE_DT_F32 && x_dtype != MOE_DT_BF16) return MOE_ERR_INVALID_ARG;
  if (!x || !w_router || !experts || !out) return MOE_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(w_router, 16) || !aligned(out, 16) || !aligned(experts, 8)) return MOE_ERR_INVALID_ARG;
  if ((b_router && !aligned(b_router, 4)) || (ids_out && !aligned(ids_out, 4)) || (w_out && !aligned(w_out, 4)))
    return MOE_ERR_INVALID_ARG;
  if (shared && (!shared->gate || !shared->up || !shared->down || !aligned(shared->gate, 16) ||
                 !aligned(shared->up, 16) || !aligned(shared->down, 16)))
    return MOE_ERR_INVALID_ARG;
  int rpath;
  if ((st = resolve_path(shape, x_dtype, shared != nullptr, path, &rpath)) != MOE_OK) return st;
  cudaStream_t s = (cudaStream_t)stream;
  const Ws L = ws_layout(*shape, ws);
  int32_t* ids = ids_out ? ids_out : L.ids;
  float* w = w_out ? w_out : L.w;
  if ((st = cuda_status(cudaMemsetAsync(L.hdr, 0, sizeof(WsHeader), s))) != MOE_OK) return st;
  const ExpertParams p = expert_params(shape, x, x_dtype, experts, ids, w, L.offsets, L.sorted, out, accumulate, shared, L);
  if (rpath == MOE_PATH_DECODE || rpath == MOE_PATH_DECODE_MX) {
    const RouteParams rp = route_params(shape, x, x_dtype, w_router, b_router, ids, w, nullptr, nullptr, L);
    if (rpath == MOE_PATH_DECODE_MX && !dmx_supported(p)) return MOE_ERR_UNSUPPORTED;
    st = cuda_status(launch_decode_forward(rp, bucket_params(shape, ids, nullptr, nullptr, L), p, s,
                                           rpath == MOE_PATH_DECODE_MX));
    if (st != MOE_OK || !shared) return st;
    // The shared expert: the prefill GEMM kernels with no routed items (the
    // active-expert count cleared), adding its output into out.
    if ((st = cuda_status(cudaMemsetAsync(&L.hdr->n_active, 0, sizeof(uint32_t), s))) != MOE_OK) return st;
    ExpertParams ps = p;
    ps.accumulate = 1;
    ps.shared_only = 1;
    return cuda_status(launch_prefill_experts(ps, s));
  }
  if ((st = do_route(shape, x, x_dtype, w_router, b_router, ids, w, nullptr, nullptr, L, false, s)) != MOE_OK) return st;
  return run_experts(p, rpath, s);
}

int moe_forward_static_scratch(const moe_shape* shape, const void* x, int x_dtype, const float* w_router,
                               const float* b_router, const moe_expert* experts, const moe_dense_bf16* shared,
                               float* out, int accumulate, int32_t* ids_out, float* w_out, int path,
                               int32_t* status_dev, void* stream) {
  int st = validate_shape(shape);
  if (st != MOE_OK) return st;
  if (ws_layout(*shape, nullptr).total > MOE_STATIC_SCRATCH_BYTES) return MOE_ERR_WORKSPACE;
  if (status_dev && !aligned(status_dev, 4)) return MOE_ERR_INVALID_ARG;
  void* scratch = nullptr;
  if ((st = static_scratch_ptr(&scratch)) != MOE_OK) return st;
  st = moe_forward(shape, x, x_dtype, w_router, b_router, experts, shared, out, accumulate, ids_out, w_out, path,
                   scratch, MOE_STATIC_SCRATCH_BYTES, stream);
  if (st != MOE_OK) return st;
  if (status_dev &&
      cudaMemcpyAsync(status_dev, scratch, sizeof(int32_t), cudaMemcpyDeviceToDevice, (cudaStream_t)stream) !=
          cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}

int moe_wait_selftest(long long max_cycles, void* stream, int* status_out) {
  if (!status_out || max_cycles < 1 || max_cycles > kWaitCycles) return MOE_ERR_INVALID_ARG;
  // The device status is written into the caller-visible result below; a
  // 4-byte device word is borrowed from the static scratch region.
  void* scratch = nullptr;
  int st = static_scratch_ptr(&scratch);
  if (st != MOE_OK) return st;
  cudaStream_t s = (cudaStream_t)stream;
  int* dev_status = reinterpret_cast<int*>(scratch);
  k_wait_selftest<<<1, 32, 0, s>>>(max_cycles, dev_status);
  if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;
  int v = -1;
  if (cudaMemcpyAsync(&v, dev_status, sizeof v, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess)
    return MOE_ERR_CUDA;
  *status_out = v;
  return MOE_OK;
}

int moe_set_wait_limit(long long cycles) {
  if (cycles < 0 || cycles > kWaitCycles) return MOE_ERR_INVALID_ARG;
  g_wait_limit = cycles == 0 ? kWaitCycles : cycles;
  return MOE_OK;
}

int moe_profile_events(int stage, void* before, void* after) {
  if (stage < 1 || stage >= MOE_STAGE_COUNT) return MOE_ERR_INVALID_ARG;
  g_prof.before[stage] = (cudaEvent_t)before;
  g_prof.after[stage] = (cudaEvent_t)after;
  return MOE_OK;
}

int moe_device_status(const void* ws, void* stream, int* status_out) {
  if (!ws || !status_out) return MOE_ERR_INVALID_ARG;
  if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return MOE_ERR_CUDA;
  uint32_t v = 0;
  if (cudaMemcpy(&v, ws, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess) return MOE_ERR_CUDA;
  *status_out = (int)v;
  return MOE_OK;
}

}  // extern "C"
