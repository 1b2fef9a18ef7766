/* svgen.c -- host bulk fill of the seeded synthetic inputs (see svgen.h).
 * Elements are independent, so the fill is split over threads without any
 * effect on the values. */
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>

#include "svgen.h"

typedef struct {
  void* out;
  uint64_t begin, end;
  uint64_t stream;
  double stdv;
  int kind; /* 0 weight, 1 gain, 2 constant one, 3 token */
  uint32_t vocab;
} svg_job;

static void* svg_worker(void* arg) {
  svg_job* j = (svg_job*)arg;
  if (j->kind == 3) {
    int32_t* o = (int32_t*)j->out;
    for (uint64_t i = j->begin; i < j->end; ++i) o[i] = svg_token(j->stream, i, j->vocab);
    return NULL;
  }
  uint16_t* o = (uint16_t*)j->out;
  for (uint64_t i = j->begin; i < j->end; ++i) {
    if (j->kind == 0)
      o[i] = svg_weight_bf16(j->stream, i, j->stdv);
    else if (j->kind == 1)
      o[i] = svg_gain_bf16(j->stream, i, j->stdv);
    else
      o[i] = 0x3F80u; /* bf16 1.0 */
  }
  return NULL;
}

static int svg_run(void* out, uint64_t n, uint64_t stream, double stdv, int kind, uint32_t vocab,
                   int nthreads) {
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  if ((uint64_t)nthreads > n / 65536u + 1u) nthreads = (int)(n / 65536u + 1u);
  pthread_t th[256];
  int joined[256];
  svg_job jobs[256];
  uint64_t chunk = (n + (uint64_t)nthreads - 1u) / (uint64_t)nthreads;
  for (int t = 0; t < nthreads; ++t) {
    uint64_t b = chunk * (uint64_t)t, e = b + chunk;
    if (b > n) b = n;
    if (e > n) e = n;
    jobs[t] = (svg_job){out, b, e, stream, stdv, kind, vocab};
    joined[t] = 0;
    if (t == 0) continue;
    if (pthread_create(&th[t], NULL, svg_worker, &jobs[t]) == 0)
      joined[t] = 1;
    else
      svg_worker(&jobs[t]); /* run inline if a thread cannot be made */
  }
  svg_worker(&jobs[0]);
  for (int t = 1; t < nthreads; ++t)
    if (joined[t]) pthread_join(th[t], NULL);
  return 0;
}

/* Fill out[0..n) with bf16 weights ~ z * stdv of tensor `tensor_id`. */
int svg_fill_weights(uint16_t* out, uint64_t n, uint64_t seed, uint64_t tensor_id, double stdv,
                     int nthreads) {
  return svg_run(out, n, svg_stream(seed, tensor_id), stdv, 0, 0, nthreads);
}

/* Fill out[0..n) with bf16 gains 1 + z * stdv (stdv == 0 gives exact ones). */
int svg_fill_gains(uint16_t* out, uint64_t n, uint64_t seed, uint64_t tensor_id, double stdv,
                   int nthreads) {
  return svg_run(out, n, svg_stream(seed, tensor_id), stdv, stdv == 0.0 ? 2 : 1, 0, nthreads);
}

/* Fill out[0..n) with token ids uniform in [0, vocab). */
int svg_fill_tokens(int32_t* out, uint64_t n, uint64_t seed, uint64_t tensor_id, uint32_t vocab) {
  return svg_run(out, n, svg_stream(seed, tensor_id), 0.0, 3, vocab, 1);
}

/* Single elements, for spot checks against the device generator. */
uint16_t svg_weight_at(uint64_t seed, uint64_t tensor_id, uint64_t i, double stdv) {
  return svg_weight_bf16(svg_stream(seed, tensor_id), i, stdv);
}
uint16_t svg_gain_at(uint64_t seed, uint64_t tensor_id, uint64_t i, double stdv) {
  if (stdv == 0.0) return 0x3F80u;
  return svg_gain_bf16(svg_stream(seed, tensor_id), i, stdv);
}
uint64_t svg_draw_at(uint64_t seed, uint64_t tensor_id, uint64_t i) {
  return svg_draw(svg_stream(seed, tensor_id), i);
}
