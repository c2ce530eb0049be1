// kernels.h — host-side launchers of the library's kernels (one per stage).
#pragma once

#include <cuda.h>

#include "common.cuh"

namespace moe {

// Launch with programmatic dependent launch enabled: the kernel may start
// while the previous kernel on the stream finishes; it must call pdl_wait()
// before touching that kernel's outputs.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

int device_sm_count();

// Raise a kernel's dynamic shared memory limit to at least `bytes` (once per
// kernel and size; later calls are a table lookup).
cudaError_t ensure_smem_attr(const void* kernel, size_t bytes);
// Resident CTAs per SM of a kernel for a block size and dynamic smem (>= 1),
// memoised.
cudaError_t cached_occupancy(const void* kernel, int threads, size_t smem, int* out);

// Profiling hook state (see moe_profile_events in the header).
struct ProfHook {
  cudaEvent_t before[MOE_STAGE_COUNT];
  cudaEvent_t after[MOE_STAGE_COUNT];
};
extern ProfHook g_prof;
inline void prof_before(int stage, cudaStream_t s) {
  if (g_prof.before[stage]) cudaEventRecord(g_prof.before[stage], s);
}
inline void prof_after(int stage, cudaStream_t s) {
  if (g_prof.after[stage]) cudaEventRecord(g_prof.after[stage], s);
}

// cuTensorMapEncodeTiled from the driver (looked up once through the
// runtime); null if unavailable.
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn encode_tiled_fn();
// Template of the per-expert code maps of the block-scaled GEMMs: an [M][K]
// matrix of 4-bit codes, boxes of 128 elements x 128 rows (prefill.cu).
cudaError_t encode_code_map_template(CUtensorMap* m, void* base, int K, int M);

// decode_mx.cu
// Whether the persistent block-scaled decode kernel takes this call (bf16,
// T <= 8, 128 | H, 128 | I, I >= 256, the device's SM count and shared memory).
bool dmx_supported(const ExpertParams& p);
// The shape part of dmx_supported (host, no device query).
bool dmx_shape_supported(int T, int H, int E, int I, int k);
// The routed experts of a decode step in one launch (routing first when
// p.fused_route; otherwise from the published buckets, after a preparation
// kernel).
cudaError_t launch_dec_mx(const ExpertParams& p, cudaStream_t s);

// route_tc.cu
// Router scores of a bf16 batch above 64 tokens on tensor cores (a screen)
// plus exact double-float scores of the experts that can reach the top k,
// into ws.logits (the others get -inf); cudaErrorNotSupported for a shape it
// does not take (the caller then runs the CUDA-core GEMM).
cudaError_t launch_router_tc(const RouteParams& p, cudaStream_t s);

// route.cu
bool route_decode_supported(int T, int H, int E, int k);
size_t small_plan_bytes(int E, int npairs);
cudaError_t launch_router_gemv(const RouteParams& p, cudaStream_t s);
cudaError_t launch_route_decode(const RouteParams& p, cudaStream_t s);
cudaError_t launch_route_prefill(const RouteParams& p, const BucketParams& b, cudaStream_t s);
cudaError_t launch_bucket_from_ids(const BucketParams& b, cudaStream_t s);
cudaError_t launch_plan_from_offsets(const BucketParams& b, const int32_t* offsets, cudaStream_t s);
// out[i] = in[i] for i < npairs, or -1 (and MOE_ERR_DEVICE_CHECK in hdr) where
// in[i] is not in [0, npairs).
cudaError_t launch_copy_pairs(const int32_t* in, int32_t* out, int npairs, WsHeader* hdr, cudaStream_t s);

// decode.cu
// Whether the staged decode kernels take a bf16 batch of this shape (the
// decode path of batches above 64 tokens runs only on them).
bool decode_batch_supported(int T, int H, int E, int I, int k);
cudaError_t launch_decode_experts(const ExpertParams& p, cudaStream_t s);
cudaError_t launch_decode_forward(const RouteParams& rp, const BucketParams& bp, ExpertParams p, cudaStream_t s,
                                  bool mx = false);

// prefill.cu
constexpr int kPfNTile = 128;   // tokens per MMA tile (N)
constexpr int kPfMTile = 128;   // weight rows per MMA tile (M)
// The prefill path needs H % 128 == 0 and I % 128 == 0 (64-element contraction
// slices; 4-byte scale rows) and bf16 activations.
bool prefill_supported(int H, int I);
cudaError_t launch_prefill_experts(const ExpertParams& p, cudaStream_t s);
// bf16 activations -> ws.xh (f16, per-token power-of-two shift) and ws.xscale.
cudaError_t launch_x_to_f16(const ExpertParams& p, cudaStream_t s);

}  // namespace moe
