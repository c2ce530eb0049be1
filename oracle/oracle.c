/*
 * oracle.c — fp64 CPU oracle of the routed MXFP4 mixture-of-experts layer.
 *
 * TEST INFRASTRUCTURE.  Only the tests, the package's smoke check and the
 * benchmark's CPU-baseline / reference arm may load this library.  The CUDA
 * library never includes, links or calls it, and it includes nothing of the
 * CUDA library: the two share no code.
 *
 * It computes the plain definition of the layer, one output element at a
 * time, with fp64 accumulation and straightforward loops:
 *
 *   1. router scores   s[t][e] = sum_h x[t][h] * Wr[e][h] + b[e]
 *   2. top-k           the k largest scores, ties to the lower expert index,
 *                      in descending order; weights are the softmax of the
 *                      selected scores (renormalised over the k)
 *   3. bucketing       a counting sort of the (token, slot) pairs by expert
 *   4. expert MLP      g = Wg x, u = Wu x, h = silu(g) * u, y = Wd h, with the
 *                      MXFP4 weights decoded element by element
 *   5. combine         out[t] = residual[t] + sum_j w[t][j] * y[t][j]
 *                      (+ an always-on shared expert with weight 1)
 *
 * Sources:
 *   - [deltafin, "How it splits the model"]: 896 routed experts per layer,
 *     16 selected per layer, MXFP4 expert weights.
 *   - [Deltafin's custom compiled runtime, "Complete target sequence tape"]:
 *     the provider returns the authoritative top-16 route mailbox (ids and
 *     fp32 weights, route order checked bit for bit).
 *   - [Deltafin's custom compiled runtime, "Weight fidelity"]: the released
 *     MXFP4 experts are used unchanged, activations stay fp32, and all 16
 *     selected experts run.
 *   - [deltafin, "The techniques that bought the 82x"]: the fused MXFP4
 *     dequant+GEMV decodes each element through a 16-entry table and applies
 *     the E8M0 block scale as a power of two on the fp32 exponent; all six
 *     tensors of an expert (gate, up, down: nibbles and scales) sit together.
 *   - [Deltafin's custom compiled runtime, "The native build"]: the batched
 *     CPU path ends in an ordered reduction (here: slot order j = 0..k-1).
 *   - OCP Microscaling Formats (MX) v1.0: E2M1 element values
 *     {0, 0.5, 1, 1.5, 2, 3, 4, 6} with a sign bit, E8M0 scale 2^(e-127),
 *     e = 255 is NaN, 32 elements per block.
 *
 * Readings where the pages are silent (each is listed with its reason in the
 * design notes): the router is a softmax over the selected scores; a router
 * bias adds to the scores before selection; the activation is SwiGLU with
 * silu(z) = z / (1 + e^-z); element 2i of a block is the low nibble of byte i;
 * blocks run along the contraction axis (the rows of an [out][in] matrix).
 *
 * Parity is pinned for every function here by the oracle tests (format
 * tables, hand-worked blocks, closed forms, brute force).  Agreement with the
 * numerics of real trained weights is not pinned: no trained weights or
 * reference outputs exist on the pages.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

#define ORC_OK 0
#define ORC_EINVAL 1
#define ORC_ENOMEM 2

/* ---------------------------------------------------------------- formats -- */

/* E2M1 element value of a 4-bit code: bit 3 is the sign, bits 2..0 index the
 * magnitude table {0, 0.5, 1, 1.5, 2, 3, 4, 6} (OCP MX v1.0, FP4 E2M1). */
double orc_e2m1(int code) {
  static const double mag[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};
  double m = mag[code & 7];
  return (code & 8) ? -m : m;
}

/* E8M0 scale: 2^(e-127); e = 255 encodes NaN (OCP MX v1.0, E8M0). */
double orc_e8m0(int e) {
  if (e == 255) return NAN;
  return ldexp(1.0, e - 127);
}

/* Element (r, c) of an MX matrix with `cols` columns: q is [rows][cols/2]
 * (element 2i low nibble, 2i+1 high nibble of byte i), s is [rows][cols/32]. */
double orc_mx_at(const uint8_t* q, const uint8_t* s, int64_t cols, int64_t r, int64_t c) {
  uint8_t byte = q[r * (cols / 2) + c / 2];
  int code = (c % 2 == 0) ? (byte & 0xF) : (byte >> 4);
  int e = s[r * (cols / 32) + c / 32];
  return orc_e2m1(code) * orc_e8m0(e);
}

/* Decode a whole MX matrix to fp64 (rows x cols). */
int orc_dequant(const uint8_t* q, const uint8_t* s, int64_t rows, int64_t cols, double* out) {
  if (cols % 32 != 0 || rows < 0) return ORC_EINVAL;
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t c = 0; c < cols; ++c) out[r * cols + c] = orc_mx_at(q, s, cols, r, c);
  return ORC_OK;
}

/* Activation element as fp64: dtype 0 = fp32, 1 = bf16 (upper half of fp32). */
static double orc_act(const void* x, int dtype, int64_t i) {
  if (dtype == 0) return (double)((const float*)x)[i];
  uint32_t bits = (uint32_t)((const uint16_t*)x)[i] << 16;
  float f;
  memcpy(&f, &bits, sizeof f);
  return (double)f;
}

static double orc_bf16(uint16_t v) {
  uint32_t bits = (uint32_t)v << 16;
  float f;
  memcpy(&f, &bits, sizeof f);
  return (double)f;
}

static double orc_silu(double z) { return z / (1.0 + exp(-z)); }

/* ------------------------------------------------------------- threading -- */

typedef struct orc_pool_job {
  void (*fn)(void* ctx, int64_t item);
  void* ctx;
  int64_t n;
  int64_t next;
  pthread_mutex_t mu;
} orc_pool_job;

static void* orc_pool_worker(void* arg) {
  orc_pool_job* job = (orc_pool_job*)arg;
  for (;;) {
    pthread_mutex_lock(&job->mu);
    int64_t item = job->next++;
    pthread_mutex_unlock(&job->mu);
    if (item >= job->n) break;
    job->fn(job->ctx, item);
  }
  return NULL;
}

/* Run fn(ctx, i) for i in [0, n) on up to nthreads threads.  Each item writes
 * its own outputs, so the result does not depend on the thread count. */
static void orc_parallel(int nthreads, int64_t n, void (*fn)(void*, int64_t), void* ctx) {
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 512) nthreads = 512;
  orc_pool_job job;
  job.fn = fn; job.ctx = ctx; job.n = n; job.next = 0;
  pthread_mutex_init(&job.mu, NULL);
  pthread_t th[512];
  int ok[512];
  for (int t = 0; t < nthreads; ++t) ok[t] = pthread_create(&th[t], NULL, orc_pool_worker, &job) == 0;
  orc_pool_worker(&job); /* the calling thread works too */
  for (int t = 0; t < nthreads; ++t)
    if (ok[t]) pthread_join(th[t], NULL);
  pthread_mutex_destroy(&job.mu);
}

int orc_default_threads(void) {
  long n = sysconf(_SC_NPROCESSORS_ONLN);
  return n > 0 ? (int)n : 1;
}

/* ----------------------------------------------------------------- router -- */

typedef struct {
  int T, H, E;
  const void* x;
  int dtype;
  const float* wr;
  const float* br;
  double* s;
} orc_logit_ctx;

static void orc_logit_item(void* vctx, int64_t t) {
  orc_logit_ctx* c = (orc_logit_ctx*)vctx;
  for (int e = 0; e < c->E; ++e) {
    double acc = 0.0;
    for (int h = 0; h < c->H; ++h)
      acc += orc_act(c->x, c->dtype, t * (int64_t)c->H + h) * (double)c->wr[(int64_t)e * c->H + h];
    if (c->br) acc += (double)c->br[e];
    c->s[t * (int64_t)c->E + e] = acc;
  }
}

/* Router scores s[t][e] = sum_h x[t][h] * Wr[e][h] (+ b[e]) in fp64.
 * x is [T][H] (fp32 or bf16), Wr is [E][H] fp32, b is [E] fp32 or NULL. */
int orc_router_logits(int T, int H, int E, const void* x, int dtype, const float* wr, const float* br,
                      int nthreads, double* s) {
  if (T < 0 || H < 1 || E < 1 || (dtype != 0 && dtype != 1)) return ORC_EINVAL;
  orc_logit_ctx c = {T, H, E, x, dtype, wr, br, s};
  orc_parallel(nthreads, T, orc_logit_item, &c);
  return ORC_OK;
}

/* Ordering of (score, expert) pairs: larger score first, lower index on ties. */
typedef struct { double s; int e; } orc_pair;
static int orc_pair_cmp(const void* a, const void* b) {
  const orc_pair* p = (const orc_pair*)a;
  const orc_pair* q = (const orc_pair*)b;
  if (p->s > q->s) return -1;
  if (p->s < q->s) return 1;
  return (p->e > q->e) - (p->e < q->e);
}

/* Top-k with renormalised weights, from given scores s [T][E]:
 * ids[t][j] is the j-th largest score's expert (ties to the lower index) and
 * w[t][j] = exp(s_j - s_0) / sum_i exp(s_i - s_0) over the k selected.
 * If margin != NULL it receives, per token, the smallest gap between
 * consecutive scores among the first min(k+1, E) sorted entries. */
int orc_topk(int T, int E, int k, const double* s, int32_t* ids, double* w, double* margin) {
  if (T < 0 || E < 1 || k < 1 || k > E) return ORC_EINVAL;
  orc_pair* p = (orc_pair*)malloc(sizeof(orc_pair) * (size_t)E);
  if (!p) return ORC_ENOMEM;
  for (int t = 0; t < T; ++t) {
    for (int e = 0; e < E; ++e) { p[e].s = s[(int64_t)t * E + e]; p[e].e = e; }
    qsort(p, (size_t)E, sizeof(orc_pair), orc_pair_cmp);
    double z = 0.0;
    for (int j = 0; j < k; ++j) z += exp(p[j].s - p[0].s);
    for (int j = 0; j < k; ++j) {
      ids[(int64_t)t * k + j] = p[j].e;
      w[(int64_t)t * k + j] = exp(p[j].s - p[0].s) / z;
    }
    if (margin) {
      int last = k < E ? k : E - 1;
      double m = INFINITY;
      for (int j = 0; j < last; ++j) {
        double g = p[j].s - p[j + 1].s;
        if (g < m) m = g;
      }
      margin[t] = m;
    }
  }
  free(p);
  return ORC_OK;
}

/* ------------------------------------------------------------- bucketing -- */

/* Counting sort of the flat pairs i = t*k + j by expert ids[t][j]:
 * offsets[e] = number of pairs with a smaller expert id (offsets[E] = T*k);
 * sorted_idx lists, expert by expert, the pairs of that expert in ascending
 * (t, j).  Plain loop over e, then t, then j. */
int orc_bucket(int T, int E, int k, const int32_t* ids, int32_t* offsets, int32_t* sorted_idx) {
  if (T < 0 || E < 1 || k < 1) return ORC_EINVAL;
  int64_t pos = 0;
  for (int e = 0; e < E; ++e) {
    offsets[e] = (int32_t)pos;
    for (int t = 0; t < T; ++t)
      for (int j = 0; j < k; ++j)
        if (ids[(int64_t)t * k + j] == e) sorted_idx[pos++] = t * k + j;
  }
  offsets[E] = (int32_t)pos;
  for (int64_t i = 0; i < (int64_t)T * k; ++i)
    if (ids[i] < 0 || ids[i] >= E) return ORC_EINVAL;
  return ORC_OK;
}

/* ------------------------------------------------------------ expert MLP -- */

/* Host pointers of one expert's six tensors (gate/up: [I][H], down: [H][I]). */
typedef struct {
  const uint8_t *gate_q, *gate_s, *up_q, *up_s, *down_q, *down_s;
} orc_expert;

/* One expert on one activation vector: y = Wd (silu(Wg x) * (Wu x)), fp64. */
int orc_expert_mlp(int H, int I, const double* x, const orc_expert* ex, double* y) {
  if (H % 32 != 0 || I % 32 != 0 || !ex || !ex->gate_q || !ex->gate_s || !ex->up_q || !ex->up_s ||
      !ex->down_q || !ex->down_s)
    return ORC_EINVAL;
  double* h = (double*)malloc(sizeof(double) * (size_t)I);
  if (!h) return ORC_ENOMEM;
  for (int r = 0; r < I; ++r) {
    double g = 0.0, u = 0.0;
    for (int c = 0; c < H; ++c) {
      g += orc_mx_at(ex->gate_q, ex->gate_s, H, r, c) * x[c];
      u += orc_mx_at(ex->up_q, ex->up_s, H, r, c) * x[c];
    }
    h[r] = orc_silu(g) * u;
  }
  for (int o = 0; o < H; ++o) {
    double acc = 0.0;
    for (int c = 0; c < I; ++c) acc += orc_mx_at(ex->down_q, ex->down_s, I, o, c) * h[c];
    y[o] = acc;
  }
  free(h);
  return ORC_OK;
}

/* Dense bf16 SwiGLU expert (the always-on shared expert): gate/up [I][H],
 * down [H][I], bf16 row-major. */
int orc_dense_mlp_bf16(int H, int I, const double* x, const uint16_t* wg, const uint16_t* wu,
                       const uint16_t* wd, double* y) {
  if (H < 1 || I < 1 || !wg || !wu || !wd) return ORC_EINVAL;
  double* h = (double*)malloc(sizeof(double) * (size_t)I);
  if (!h) return ORC_ENOMEM;
  for (int r = 0; r < I; ++r) {
    double g = 0.0, u = 0.0;
    for (int c = 0; c < H; ++c) {
      g += orc_bf16(wg[(int64_t)r * H + c]) * x[c];
      u += orc_bf16(wu[(int64_t)r * H + c]) * x[c];
    }
    h[r] = orc_silu(g) * u;
  }
  for (int o = 0; o < H; ++o) {
    double acc = 0.0;
    for (int c = 0; c < I; ++c) acc += orc_bf16(wd[(int64_t)o * I + c]) * h[c];
    y[o] = acc;
  }
  free(h);
  return ORC_OK;
}

/* ----------------------------------------------------------- whole layer -- */

typedef struct {
  int H, I, k, nsel;
  const void* x;
  int dtype;
  const int32_t* tokens;
  const int32_t* ids;       /* [nsel][k] */
  const orc_expert* experts;
  const uint16_t *sg, *su, *sd;
  double* y;                /* [nsel][k+1][H] */
  int status;
} orc_layer_ctx;

static void orc_layer_item(void* vctx, int64_t item) {
  orc_layer_ctx* c = (orc_layer_ctx*)vctx;
  int64_t n = item / (c->k + 1);
  int j = (int)(item % (c->k + 1));
  double* x = (double*)malloc(sizeof(double) * (size_t)c->H);
  if (!x) { c->status = ORC_ENOMEM; return; }
  int64_t t = c->tokens[n];
  for (int h = 0; h < c->H; ++h) x[h] = orc_act(c->x, c->dtype, t * c->H + h);
  double* y = c->y + (n * (c->k + 1) + j) * (int64_t)c->H;
  int rc = ORC_OK;
  if (j < c->k) {
    rc = orc_expert_mlp(c->H, c->I, x, &c->experts[c->ids[n * c->k + j]], y);
  } else if (c->sg) {
    rc = orc_dense_mlp_bf16(c->H, c->I, x, c->sg, c->su, c->sd, y);
  } else {
    for (int h = 0; h < c->H; ++h) y[h] = 0.0;
  }
  if (rc != ORC_OK) c->status = rc;
  free(x);
}

/* The layer for the tokens listed in tokens[0..nsel): routes them (scores in
 * fp64, top-k, renormalised weights), runs the k selected experts and the
 * optional shared expert (sg/su/sd, bf16, weight 1), and combines
 *   out[n][h] = residual[t][h] + sum_{j=0}^{k-1} w[n][j] * y_j[h] + shared[h]
 * with the sum taken in slot order.  residual may be NULL (treated as 0).
 * experts is a host array of E descriptors; only selected experts are read. */
int orc_moe_tokens(int T, int H, int E, int I, int k, const void* x, int dtype, const float* wr,
                   const float* br, const orc_expert* experts, const uint16_t* sg, const uint16_t* su,
                   const uint16_t* sd, const float* residual, int nsel, const int32_t* tokens,
                   int nthreads, double* out, int32_t* ids, double* w) {
  if (T < 1 || H % 32 != 0 || I % 32 != 0 || E < 1 || k < 1 || k > E || nsel < 0) return ORC_EINVAL;
  for (int n = 0; n < nsel; ++n)
    if (tokens[n] < 0 || tokens[n] >= T) return ORC_EINVAL;
  if ((sg || su || sd) && !(sg && su && sd)) return ORC_EINVAL;
  /* 1-2: route the selected tokens. */
  double* s = (double*)malloc(sizeof(double) * (size_t)E * (size_t)(nsel > 0 ? nsel : 1));
  void* xs = malloc((size_t)(dtype == 0 ? 4 : 2) * (size_t)H * (size_t)(nsel > 0 ? nsel : 1));
  if (!s || !xs) { free(s); free(xs); return ORC_ENOMEM; }
  for (int n = 0; n < nsel; ++n)
    memcpy((char*)xs + (size_t)n * H * (dtype == 0 ? 4 : 2),
           (const char*)x + (size_t)tokens[n] * H * (dtype == 0 ? 4 : 2), (size_t)H * (dtype == 0 ? 4 : 2));
  int rc = orc_router_logits(nsel, H, E, xs, dtype, wr, br, nthreads, s);
  if (rc == ORC_OK) rc = orc_topk(nsel, E, k, s, ids, w, NULL);
  free(s);
  free(xs);
  if (rc != ORC_OK) return rc;
  /* 4: every (token, slot) expert evaluation, plus the shared expert. */
  double* y = (double*)malloc(sizeof(double) * (size_t)H * (size_t)(k + 1) * (size_t)(nsel > 0 ? nsel : 1));
  if (!y) return ORC_ENOMEM;
  orc_layer_ctx c = {H, I, k, nsel, x, dtype, tokens, ids, experts, sg, su, sd, y, ORC_OK};
  orc_parallel(nthreads, (int64_t)nsel * (k + 1), orc_layer_item, &c);
  if (c.status != ORC_OK) { free(y); return c.status; }
  /* 5: ordered combine. */
  for (int n = 0; n < nsel; ++n) {
    for (int h = 0; h < H; ++h) {
      double acc = 0.0;
      for (int j = 0; j < k; ++j) acc += w[(int64_t)n * k + j] * y[((int64_t)n * (k + 1) + j) * H + h];
      acc += y[((int64_t)n * (k + 1) + k) * H + h];
      if (residual) acc += (double)residual[(int64_t)tokens[n] * H + h];
      out[(int64_t)n * H + h] = acc;
    }
  }
  free(y);
  return ORC_OK;
}
