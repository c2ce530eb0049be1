/*
 * moe_mxfp4.h — C ABI of the routed MXFP4 mixture-of-experts layer on GB300
 * (sm_103a), exported by libmoe_mxfp4.so.
 *
 * The layer (per token t, hidden size H, E experts, top-k routing, expert
 * intermediate size I):
 *
 *   s[t][e]  = sum_h x[t][h] * Wr[e][h] + b[e]                 router scores
 *   ids[t]   = the k largest s[t][.], descending, ties to the lower index
 *   w[t][j]  = exp(s_j - s_0) / sum_i exp(s_i - s_0)           over the k
 *   y[t][j]  = Wd_e (silu(Wg_e x_t) * (Wu_e x_t)),  e = ids[t][j]
 *   out[t]   = (accumulate ? out[t] : 0) + sum_{j=0}^{k-1} w[t][j] y[t][j]
 *              (+ an optional always-on bf16 shared expert, weight 1)
 *
 * Where the definition comes from:
 *   - one layer routes each token to 16 of 896 experts whose weights are MXFP4
 *     [deltafin, "How it splits the model"];
 *   - the provider hands back an authoritative top-16 "route mailbox" of ids
 *     and fp32 weights whose route order and weight bits are checked at every
 *     ABI transition [Deltafin's custom compiled runtime, "Complete target
 *     sequence tape"]; a trace of it records the 16 ids and fp32 weight bits
 *     [How the native runtime works, "Router tracing and offline expert
 *     warming"];
 *   - the MXFP4 experts are used unchanged, activations stay fp32, all 16
 *     selected experts run [Deltafin's custom compiled runtime, "Weight
 *     fidelity"];
 *   - each expert is six tensors (gate, up, down; nibbles and E8M0 scales)
 *     [deltafin, "The techniques that bought the 82x"]; experts may sit in
 *     scattered spans that the provider accepts without a copy [Deltafin's
 *     custom compiled runtime, "Exact next-layer expert prefetch"], hence the
 *     per-expert descriptor table below;
 *   - a small versioned C ABI, descriptor-driven binding, failures fail closed
 *     [Deltafin's custom compiled runtime, "Production ownership", "Coarse
 *     provider binding", "Configuration and device selection"].
 * The router nonlinearity, the SwiGLU activation, the nibble order and the
 * block axis are not on those pages; this library takes: softmax over the
 * selected scores; silu(z) = z / (1 + e^-z); element 2i of a block is the low
 * nibble of byte i; blocks of 32 run along the contraction axis.
 *
 * MXFP4 matrix (moe_mx_mat) with R rows and C columns (C % 32 == 0):
 *   q: uint8 [R][C/2]   E2M1 codes, element 2i low nibble, 2i+1 high nibble
 *   s: uint8 [R][C/32]  E8M0 scales, value 2^(s-127), 255 = NaN
 *   element (r, c) = e2m1(code) * 2^(s[r][c/32] - 127),
 *   e2m1 codes: {0, .5, 1, 1.5, 2, 3, 4, 6}, bit 3 = sign (OCP MX v1.0).
 * Expert e: gate and up are [I][H] (rows = intermediate features), down is
 * [H][I] (rows = hidden features).
 *
 * Conventions for every call:
 *   - Memory: every data pointer is a DEVICE pointer owned by the caller; the
 *     library allocates nothing and keeps no pointer after the call returns
 *     (work is enqueued on `stream`, so buffers must stay valid until it has
 *     run).  `shape` and `shared` point to HOST structs; `experts` points to a
 *     DEVICE array of E moe_expert descriptors.
 *   - Alignment: x, out, shared-expert tensors: 16 bytes; ws: 256 bytes;
 *     every expert tensor (q and s): 16 bytes, and on the prefill path the
 *     gate and up codes (q) 32 bytes (they are read by tensor-map copies of
 *     4-bit elements); everything else: its element size.  Host-visible
 *     misalignment is MOE_ERR_INVALID_ARG; an expert descriptor (device
 *     memory) with a null or misaligned tensor is detected on the device
 *     (MOE_ERR_DEVICE_CHECK) and that expert is not read.
 *   - Asynchrony: calls enqueue kernels on `stream` (a cudaStream_t; NULL is
 *     the legacy default stream) and return; there is no host synchronisation
 *     except in moe_device_status().  The calls make no CUDA allocation.
 *   - Errors: argument problems are reported before anything is launched
 *     (MOE_ERR_INVALID_ARG / MOE_ERR_UNSUPPORTED / MOE_ERR_WORKSPACE); a launch
 *     failure returns MOE_ERR_CUDA.  Problems the kernels detect (an expert id
 *     or bucket entry out of range, a bounded wait that gave up) set a status
 *     word inside `ws` that moe_device_status() reads; outputs of such a call
 *     are unspecified.
 *   - Workspace: `ws` must hold moe_workspace_bytes(shape) bytes; its contents
 *     need not be initialised and are overwritten.  One workspace must not be
 *     used by two calls that may run concurrently.
 *   - Limits: 1 <= T <= 65536, 32 <= H <= 16384, 32 <= I <= 8192, H % 32 ==
 *     I % 32 == 0, 1 <= k <= min(E, 32), k * (I/32) <= 1024, E <= 65536.
 *     The decode path takes fp32 or bf16 activations for T <= 64 and bf16
 *     activations up to T = MOE_DECODE_BATCH_MAX_T; the prefill path takes
 *     bf16 activations.
 */
#ifndef MOE_MXFP4_H
#define MOE_MXFP4_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MOE_ABI_VERSION 1u

/* Status codes returned by every call (and stored in the device status word). */
typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,  /* null / misaligned pointer, bad shape, bad enum */
  MOE_ERR_UNSUPPORTED = 2,  /* valid request outside this build's limits */
  MOE_ERR_WORKSPACE = 3,    /* ws_bytes < moe_workspace_bytes(shape) */
  MOE_ERR_CUDA = 4,         /* a CUDA launch or query failed */
  MOE_ERR_TIMEOUT = 5,      /* device: a bounded wait gave up */
  MOE_ERR_DEVICE_CHECK = 6, /* device: an expert id out of [0, E) */
  MOE_ERR_RANGE = 7         /* reserved: no call of this version raises it */
} moe_status;

/* Activation element types. */
typedef enum { MOE_DT_F32 = 0, MOE_DT_BF16 = 1 } moe_dtype;

/* Expert execution path.
 *   decode:  the experts' weights stream once through shared memory; gate/up
 *            on warp tensor cores (bf16 x) or CUDA cores (fp32 x); down on
 *            CUDA cores up to 64 tokens and on warp tensor cores above; the
 *            k outputs of a token combined in slot order.
 *            T <= MOE_DECODE_MAX_T (the router and top-k then run as one
 *            GEMV plus a prologue of the gate/up kernel), or bf16 x and
 *            T <= MOE_DECODE_BATCH_MAX_T (routed with the tiled router GEMM).
 *            A shared expert (bf16 x) runs after the routed experts on the
 *            prefill path's GEMM kernels, alone, adding into out.
 *   prefill: grouped MXFP4 GEMM on tcgen05 tensor cores, bf16 x, with the
 *            shared expert's tiles after the routed ones.
 *   auto:    decode for T <= MOE_DECODE_MAX_T or fp32 x; else decode while
 *            the batch has at most MOE_DECODE_AUTO_PAIRS_PER_EXPERT routed
 *            pairs per expert (T * k <= that * E) and T <=
 *            MOE_DECODE_BATCH_MAX_T; else prefill.  A bf16 shape that the
 *            decode kernels do not take (H > 8192) goes to prefill when that
 *            path takes it.  The bound is the measured crossover of the two
 *            paths on GB300 (T near 265 at H = 7168, E = 896, k = 16,
 *            I = 1408): below it the decode path's single pass over the
 *            active experts' weights is faster than the tensor-core GEMMs,
 *            whose per-tile cost needs many tokens per expert. */
typedef enum {
  MOE_PATH_AUTO = 0,
  MOE_PATH_DECODE = 1,
  MOE_PATH_PREFILL = 2,
  /* The decode step as one persistent kernel on block-scaled tensor-core
   * MMAs (the E2M1 codes and E8M0 scales read by the MMA as stored): routing,
   * gate/up + SwiGLU, down and the slot-ordered combine in one launch after
   * the router scores.  bf16 x, T <= 8, H and I multiples of 128, I >= 256,
   * I <= 2048.  Never chosen automatically: measured on GB300 at the
   * pages' layer shape it is slower than MOE_PATH_DECODE (0.140 against
   * 0.091 ms at 1 token, 0.43 against 0.41 ms at 8 tokens). */
  MOE_PATH_DECODE_MX = 3
} moe_path;

#define MOE_DECODE_MAX_T 64
#define MOE_DECODE_BATCH_MAX_T 1024
#define MOE_DECODE_AUTO_PAIRS_PER_EXPERT 5

typedef struct { const uint8_t* q; const uint8_t* s; } moe_mx_mat;   /* see above */
typedef struct { moe_mx_mat gate, up, down; } moe_expert;            /* six tensors */
typedef struct { const uint16_t *gate, *up, *down; } moe_dense_bf16; /* bf16 bits */
typedef struct { int32_t T, H, E, I, k; } moe_shape;

/* MOE_ABI_VERSION of the loaded library. */
uint32_t moe_abi_version(void);

/* The path a call with this shape, activation type, shared expert (0 / 1)
 * and `path` argument runs, without running it: *path_out receives
 * MOE_PATH_DECODE, MOE_PATH_PREFILL or (when requested) MOE_PATH_DECODE_MX.  Returns the status the call would
 * return for these arguments before launching (MOE_ERR_INVALID_ARG for a bad
 * shape, enum or null path_out; MOE_ERR_UNSUPPORTED when the requested path
 * cannot take them).  Host only; no CUDA call. */
int moe_select_path(const moe_shape* shape, int x_dtype, int has_shared, int path, int* path_out);

/* Static English text for a status code (never NULL). */
const char* moe_status_string(int status);

/* Bytes of device workspace every call on this shape needs (0 if the shape is
 * invalid).  The same workspace serves moe_route, moe_mxfp4_experts and
 * moe_forward. */
size_t moe_workspace_bytes(const moe_shape* shape);

/* Routing only: router scores, top-k with renormalised fp32 weights, and the
 * bucket layout of a counting sort by expert.
 *   x         [T][H] activations of type x_dtype (MOE_DT_F32 / MOE_DT_BF16)
 *   w_router  [E][H] fp32;  b_router [E] fp32 or NULL (added to the scores)
 *   ids       [T][k] int32 out, descending score, ties to the lower index
 *   w         [T][k] fp32  out, softmax of the selected scores
 *   offsets   [E+1] int32 out or NULL: offsets[e] = number of (t, j) pairs
 *             routed to experts below e; offsets[E] = T*k
 *   sorted_idx[T*k] int32 out or NULL: flat pairs t*k+j grouped by expert,
 *             ascending (t, j) inside each expert (stable)
 * [Deltafin's custom compiled runtime, "Complete target sequence tape";
 *  "Exact next-layer expert prefetch": the final expert array is ordered by
 *  the real route union.] */
int moe_route(const moe_shape* shape, const void* x, int x_dtype, const float* w_router,
              const float* b_router, int32_t* ids, float* w, int32_t* offsets, int32_t* sorted_idx,
              void* ws, size_t ws_bytes, void* stream);

/* Experts only, given routes (as moe_route produces them):
 *   out[t] = (accumulate ? out[t] : 0) + sum_j w[t][j] * y_{ids[t][j]}(x_t)
 *   experts   device array [E] of descriptors (gate/up [I][H], down [H][I])
 *   offsets, sorted_idx: the bucket layout of ids, or both NULL (then it is
 *             rebuilt in ws from ids)
 *   out       [T][H] fp32
 *   path      moe_path
 * The decode path sums the k expert outputs of a token in slot order, and a
 * token's result is bitwise independent of the other tokens in the batch
 * among batches of 1 to 64 tokens, and among batches of 65 to
 * MOE_DECODE_BATCH_MAX_T tokens (the two ranges run different down kernels);
 * the prefill path adds them with fp32 atomics (order not fixed).
 * [deltafin, "The techniques that bought the 82x": fused MXFP4 dequant+GEMV;
 *  Deltafin's custom compiled runtime, "The native build": ordered reduction.] */
int moe_mxfp4_experts(const moe_shape* shape, const void* x, int x_dtype, const moe_expert* experts,
                      const int32_t* ids, const float* w, const int32_t* offsets, const int32_t* sorted_idx,
                      float* out, int accumulate, int path, void* ws, size_t ws_bytes, void* stream);

/* The whole layer: moe_route then moe_mxfp4_experts, plus the optional shared
 * expert (shared == NULL for none; host struct of device bf16 pointers, gate/up
 * [I][H], down [H][I], added with weight 1).  ids_out [T][k] / w_out [T][k]
 * receive the route when non-NULL. */
int moe_forward(const moe_shape* shape, const void* x, int x_dtype, const float* w_router,
                const float* b_router, const moe_expert* experts, const moe_dense_bf16* shared, float* out,
                int accumulate, int32_t* ids_out, float* w_out, int path, void* ws, size_t ws_bytes,
                void* stream);

/* Size of the library's own static device scratch (see below). */
#define MOE_STATIC_SCRATCH_BYTES (8u << 20)

/* moe_forward for callers that cannot provide a workspace: the same launch
 * sequence and results as moe_forward, but the workspace is a fixed
 * MOE_STATIC_SCRATCH_BYTES region of device memory that the library itself
 * declares (one per device), so the call allocates nothing and needs no
 * `ws` argument.  This entry point has no counterpart on the pages; it exists
 * for host programs that hold only the layer's own buffers and have no
 * device allocator to hand the library (or must not allocate while serving).
 *   - Limit: shapes with moe_workspace_bytes(shape) > MOE_STATIC_SCRATCH_BYTES
 *     are rejected with MOE_ERR_WORKSPACE before anything is launched (the
 *     pages' layer shape H = 7168, E = 896, k = 16, I = 1408 fits up to T = 13).
 *   - Set-up: the first call on a device (that device current) looks up the
 *     scratch address once; a CUDA failure there returns MOE_ERR_CUDA.  If the
 *     caller records its work into a CUDA graph, make one call before
 *     recording so that this set-up is not part of the recorded work.  The
 *     address is kept for the life of the process: after cudaDeviceReset()
 *     on a device (or in another driver context on it) the kept address is
 *     stale, and this entry point must not be called there again.
 *   - Contents: the scratch needs no initialisation; every call resets what it
 *     relies on (the status word and the counters) at its start.
 *   - Concurrency: all calls on one device share the one scratch region.  Two
 *     calls that may overlap in time (different streams, or host threads
 *     without ordering between them) race on it and give undefined results;
 *     order them (one stream, or events).
 *   - status_dev: a DEVICE int32 that receives the call's device status word
 *     (what moe_device_status reports for an explicit workspace), copied on
 *     `stream` after the layer; NULL to skip.
 * Other arguments as for moe_forward. */
int moe_forward_static_scratch(const moe_shape* shape, const void* x, int x_dtype, const float* w_router,
                               const float* b_router, const moe_expert* experts, const moe_dense_bf16* shared,
                               float* out, int accumulate, int32_t* ids_out, float* w_out, int path,
                               int32_t* status_dev, void* stream);

/* Diagnostic of the device-side failure detection: launches one thread that
 * waits, with the same bounded-wait code the kernels use but a limit of
 * max_cycles SM clock cycles (1 <= max_cycles <= 4e9), on a barrier that
 * never completes, then synchronises `stream` and stores the outcome in
 * *status_out: MOE_ERR_TIMEOUT when the wait gave up as designed.  The GPU
 * context stays usable.  It borrows 4 bytes of the static scratch region of
 * moe_forward_static_scratch (do not overlap the two).  No counterpart on the
 * pages; their runtime gives each test child a deadline [Deltafin's custom
 * compiled runtime, "One native build and test graph"]. */
int moe_wait_selftest(long long max_cycles, void* stream, int* status_out);

/* Diagnostic of the device-side failure handling: every bounded wait of the
 * layer's kernels on another part of the same CTA (copies landing, a ring
 * stage freed, partial sums handed over) gives up after `cycles` SM clock
 * cycles instead of the default (about 4e9 cycles, ~2 s), records
 * MOE_ERR_TIMEOUT in the workspace status word and takes the kernel's abort
 * path: the other roles of the CTA stop, copies already issued are drained
 * and Tensor Memory is released before the CTA exits (those draining waits
 * keep the default limit).  cycles = 0 restores the default; otherwise
 * 1 <= cycles <= 4e9, else MOE_ERR_INVALID_ARG.  Process-wide, read when a
 * call launches its kernels (not thread-safe, like the profiling hook).  The
 * outputs of a call that timed out are unspecified.  No counterpart on the
 * pages: a small limit lets tests make real waits of the product kernels run
 * out, without faulting or hanging the GPU. */
int moe_set_wait_limit(long long cycles);

/* Synchronises `stream`, then reads the device status word of `ws` into
 * *status_out (MOE_OK if no kernel flagged a problem since the last call that
 * began with this workspace).  Returns MOE_ERR_CUDA if the synchronisation or
 * the copy fails. */
int moe_device_status(const void* ws, void* stream, int* status_out);

/* Kernel stages, for the profiling hook below. */
typedef enum {
  MOE_STAGE_ROUTE = 1,        /* router scores (+ fused top-k/bucketing on the decode path) */
  MOE_STAGE_GATEUP = 2,       /* decode gate/up MXFP4 GEMV + SwiGLU */
  MOE_STAGE_DOWN = 3,         /* decode down MXFP4 GEMV */
  MOE_STAGE_COMBINE = 4,      /* decode slot-ordered combine */
  MOE_STAGE_PF_GATEUP = 5,    /* prefill grouped gate/up GEMM + SwiGLU */
  MOE_STAGE_PF_DOWN = 6,      /* prefill grouped down GEMM + combine */
  MOE_STAGE_COUNT = 7
} moe_stage;

/* Profiling hook, for benchmarks (process-wide, not thread-safe): while set,
 * every call records the CUDA event `before` (a cudaEvent_t) on its stream
 * right before it launches the kernel of `stage`, and `after` right after.
 * Recording events between kernels removes the programmatic-dependent-launch
 * overlap at that point, so a hooked call is slightly slower than an unhooked
 * one.  Pass NULL events to clear.  Returns MOE_ERR_INVALID_ARG for an unknown
 * stage.  [Deltafin's custom compiled runtime, "Verification boundaries":
 * benchmark events that refuse oracle-mismatched runs.] */
int moe_profile_events(int stage, void* before, void* after);

#ifdef __cplusplus
}
#endif

#endif /* MOE_MXFP4_H */
