/*
 * synth_host.c — host-side fill routines over synth.h (input bytes only).
 *
 * Exported with C linkage for the Python wrapper.  Threads split index ranges;
 * every element is a pure function of its index, so the result does not
 * depend on the thread count.
 */
#include "synth.h"

#include <pthread.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
  int kind;          /* 0 normal->f32, 1 normal->bf16, 2 mx matrix, 3 weight->bf16 */
  uint64_t key;
  int64_t lo, hi;    /* element (or row) range */
  double scale;
  float* f32;
  uint16_t* bf16;
  int64_t cols;
  uint8_t* q;
  uint8_t* s;
} syn_job;

static void* syn_worker(void* arg) {
  syn_job* j = (syn_job*)arg;
  if (j->kind == 0) {
    for (int64_t i = j->lo; i < j->hi; ++i)
      j->f32[i] = (float)(syn_normal(j->key, (uint64_t)i) * j->scale);
  } else if (j->kind == 1) {
    for (int64_t i = j->lo; i < j->hi; ++i)
      j->bf16[i] = syn_bf16_rne((float)(syn_normal(j->key, (uint64_t)i) * j->scale));
  } else if (j->kind == 2) {
    int64_t nb = j->cols / 32;
    for (int64_t r = j->lo; r < j->hi; ++r)
      for (int64_t b = 0; b < nb; ++b)
        syn_mx_block(j->key, j->cols, r, b, j->q + r * (j->cols / 2) + b * 16, j->s + r * nb + b);
  }
  return NULL;
}

static int syn_run(syn_job base, int64_t n, int nthreads) {
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  if ((int64_t)nthreads > n) nthreads = n > 0 ? (int)n : 1;
  pthread_t th[256];
  int joined[256];
  syn_job jobs[256];
  int64_t per = (n + nthreads - 1) / nthreads;
  for (int t = 0; t < nthreads; ++t) {
    joined[t] = 0;
    jobs[t] = base;
    jobs[t].lo = (int64_t)t * per;
    jobs[t].hi = jobs[t].lo + per < n ? jobs[t].lo + per : n;
    if (jobs[t].lo >= jobs[t].hi) continue;
    if (pthread_create(&th[t], NULL, syn_worker, &jobs[t]) == 0)
      joined[t] = 1;
    else
      syn_worker(&jobs[t]); /* no thread available: do this range inline */
  }
  for (int t = 0; t < nthreads; ++t)
    if (joined[t]) pthread_join(th[t], NULL);
  return 0;
}

uint64_t syn_key_c(uint64_t seed, uint64_t tag) { return syn_key(seed, tag); }
uint64_t syn_u64_c(uint64_t key, uint64_t i) { return syn_u64(key, i); }
double syn_normal_c(uint64_t key, uint64_t i) { return syn_normal(key, i); }
uint16_t syn_bf16_c(float f) { return syn_bf16_rne(f); }

/* out[i] = (float)(scale * z_i), i in [0, n). */
int syn_fill_f32(uint64_t key, int64_t n, double scale, float* out, int nthreads) {
  syn_job j;
  memset(&j, 0, sizeof j);
  j.kind = 0; j.key = key; j.scale = scale; j.f32 = out;
  return syn_run(j, n, nthreads);
}

/* out[i] = bf16_rne((float)(scale * z_i)), i in [0, n). */
int syn_fill_bf16(uint64_t key, int64_t n, double scale, uint16_t* out, int nthreads) {
  syn_job j;
  memset(&j, 0, sizeof j);
  j.kind = 1; j.key = key; j.scale = scale; j.bf16 = out;
  return syn_run(j, n, nthreads);
}

/* MX-quantised rows x cols matrix (cols % 32 == 0): q [rows][cols/2], s [rows][cols/32]. */
int syn_fill_mx(uint64_t key, int64_t rows, int64_t cols, uint8_t* q, uint8_t* s, int nthreads) {
  if (cols % 32 != 0 || rows < 0) return 1;
  syn_job j;
  memset(&j, 0, sizeof j);
  j.kind = 2; j.key = key; j.cols = cols; j.q = q; j.s = s;
  return syn_run(j, rows, nthreads);
}

/* Quantise caller-given reals (for hand-made tests of the quantiser). */
int syn_quant_row(const double* v, int64_t cols, uint8_t* q, uint8_t* s) {
  if (cols % 32 != 0) return 1;
  for (int64_t b = 0; b < cols / 32; ++b) syn_quant_block(v + b * 32, q + b * 16, s + b);
  return 0;
}
