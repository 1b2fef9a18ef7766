/* oracle.c -- plain CPU reference of greedy block verification.
 *
 * TEST INFRASTRUCTURE ONLY (tests, smoke check, benchmark CPU baseline).
 * Deliberately simple: one token at a time, every reduction sequential in
 * index order in fp32, bf16 (round to nearest even) at these boundaries:
 *   RMSNorm output before and after the gain multiply; every linear output
 *   (q|k|v, attention projection, gate|up, down, logits); q and k after the
 *   per-head norm and after RoPE (the cached K); V as projected; the attention
 *   output; each residual sum; act(gate) and its product with up.
 * Block verify follows "Phase 23: Speculative Verify Parity" section 2 (write
 * the window's K/V into the committed cache, row r attends to pos+r+1
 * positions, truncate to the accepted prefix on rejection) and the acceptance
 * rule of "Shape and cache history in Gemma block verification" (section
 * "Mechanism and failure"): a draft is kept only while it equals the target's
 * greedy token after the same preceding ids.  Ties in argmax go to the lowest
 * id, as the exact 22.75/22.75 tie resolving to the lower id 12630 in that
 * page's position-60 table shows.
 *
 * Compile with -ffp-contract=off: a fused multiply-add would change the
 * rounding the definitions above state.
 */
#include "oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------ bf16 values */
uint16_t orc_bf16(float x) {
  uint32_t u;
  memcpy(&u, &x, 4);
  if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x7FFFFFu)) return (uint16_t)((u >> 16) | 0x40u);
  u += 0x7FFFu + ((u >> 16) & 1u); /* round to nearest, ties to even */
  return (uint16_t)(u >> 16);
}

float orc_f32(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float x;
  memcpy(&x, &u, 4);
  return x;
}

static float rb(float x) { return orc_f32(orc_bf16(x)); } /* round through bf16 */

int32_t orc_argmax(const float* v, int n) {
  int32_t best = 0;
  for (int i = 1; i < n; ++i)
    if (v[i] > v[best]) best = i; /* strictly greater: the lowest id wins a tie */
  return best;
}

/* ------------------------------------------------------------- operations */
void orc_rmsnorm(const uint16_t* x, const uint16_t* g, int n, float eps, uint16_t* y) {
  float ss = 0.0f;
  for (int i = 0; i < n; ++i) {
    float v = orc_f32(x[i]);
    ss += v * v;
  }
  float rstd = 1.0f / sqrtf(ss / (float)n + eps);
  for (int i = 0; i < n; ++i) y[i] = orc_bf16(rb(orc_f32(x[i]) * rstd) * orc_f32(g[i]));
}

void orc_linear(const uint16_t* W, const uint16_t* x, int rows, int cols, uint16_t* y) {
  float* xf = (float*)malloc(sizeof(float) * (size_t)cols);
  for (int k = 0; k < cols; ++k) xf[k] = orc_f32(x[k]);
#pragma omp parallel for schedule(static) if ((long)rows * cols >= (1L << 18))
  for (int r = 0; r < rows; ++r) {
    const uint16_t* w = W + (size_t)r * cols;
    float acc = 0.0f;
    for (int k = 0; k < cols; ++k) acc += orc_f32(w[k]) * xf[k];
    y[r] = orc_bf16(acc);
  }
  free(xf);
}

/* Rotate-half RoPE: pair (i, i + d/2) turns by pos * theta^(-2i/d).  The angle
 * and its cosine and sine are taken in double, then cos/sin rounded to fp32. */
void orc_rope(uint16_t* x, int d, int pos, float theta) {
  int half = d / 2;
  for (int i = 0; i < half; ++i) {
    double inv_freq = pow((double)theta, -2.0 * (double)i / (double)d);
    double ang = (double)pos * inv_freq;
    float c = (float)cos(ang), s = (float)sin(ang);
    float a = orc_f32(x[i]), b = orc_f32(x[i + half]);
    float lo = a * c - b * s;
    float hi = b * c + a * s;
    x[i] = orc_bf16(lo);
    x[i + half] = orc_bf16(hi);
  }
}

void orc_attend(const uint16_t* q, const uint16_t* K, const uint16_t* V, int ctx, int d,
                int stride, uint16_t* out) {
  float scale = (float)(1.0 / sqrt((double)d));
  float* s = (float*)malloc(sizeof(float) * (size_t)(ctx > 0 ? ctx : 1));
  float* acc = (float*)calloc((size_t)d, sizeof(float));
  float mx = -INFINITY;
  for (int j = 0; j < ctx; ++j) {
    float dot = 0.0f;
    for (int i = 0; i < d; ++i) dot += orc_f32(q[i]) * orc_f32(K[(size_t)j * stride + i]);
    s[j] = dot * scale;
    if (s[j] > mx) mx = s[j];
  }
  float l = 0.0f;
  for (int j = 0; j < ctx; ++j) {
    float e = expf(s[j] - mx);
    l += e;
    for (int i = 0; i < d; ++i) acc[i] += e * orc_f32(V[(size_t)j * stride + i]);
  }
  for (int i = 0; i < d; ++i) out[i] = orc_bf16(acc[i] / l);
  free(s);
  free(acc);
}

float orc_silu(float x) { return x / (1.0f + expf(-x)); }

float orc_gelu_tanh(float x) {
  const float k0 = 0.7978845608028654f; /* sqrt(2/pi) */
  const float k1 = 0.044715f;
  return 0.5f * x * (1.0f + tanhf(k0 * (x + k1 * x * x * x)));
}

void orc_glu(const uint16_t* gate, const uint16_t* up, int n, int act, uint16_t* a) {
  for (int i = 0; i < n; ++i) {
    float g = orc_f32(gate[i]), u = orc_f32(up[i]);
    float y = act == 0 ? orc_silu(g) : orc_gelu_tanh(g);
    a[i] = orc_bf16(rb(y) * u);
  }
}

/* ------------------------------------------------------------ model state */
struct orc_model {
  orc_config c;
  orc_weights w;
  const uint16_t** arrays; /* private copies of the per-layer pointer arrays */
  int max_len, len;
  uint16_t *kc, *vc; /* [layer][position][n_kv_heads * head_dim] */
};

static int cfg_ok(const orc_config* c) {
  return c && c->n_layers >= 0 && c->hidden > 0 && c->n_q_heads > 0 && c->n_kv_heads > 0 &&
         c->n_q_heads % c->n_kv_heads == 0 && c->head_dim > 0 && c->head_dim % 2 == 0 &&
         c->ffn > 0 && c->vocab > 0 && (c->act == 0 || c->act == 1);
}

static size_t kv_row(const orc_config* c) { return (size_t)c->n_kv_heads * c->head_dim; }

orc_model* orc_create(const orc_config* cfg, const orc_weights* w, int max_len) {
  if (!cfg_ok(cfg) || !w || max_len <= 0) return NULL;
  orc_model* m = (orc_model*)calloc(1, sizeof(orc_model));
  m->c = *cfg;
  m->w = *w;
  int L = cfg->n_layers;
  m->arrays = (const uint16_t**)calloc((size_t)(9 * (L > 0 ? L : 1)), sizeof(void*));
  const uint16_t* const* src[8] = {w->attn_norm, w->wqkv, w->q_norm, w->k_norm,
                                   w->wo, w->ffn_norm, w->w_gate_up, w->w_down};
  const uint16_t* const** dst[8] = {&m->w.attn_norm, &m->w.wqkv, &m->w.q_norm, &m->w.k_norm,
                                    &m->w.wo, &m->w.ffn_norm, &m->w.w_gate_up, &m->w.w_down};
  for (int t = 0; t < 8; ++t) {
    const uint16_t** a = m->arrays + (size_t)t * L;
    for (int l = 0; l < L; ++l) a[l] = src[t] ? src[t][l] : NULL;
    *dst[t] = a;
  }
  m->max_len = max_len;
  size_t n = (size_t)L * max_len * kv_row(cfg);
  m->kc = (uint16_t*)calloc(n ? n : 1, 2);
  m->vc = (uint16_t*)calloc(n ? n : 1, 2);
  return m;
}

void orc_destroy(orc_model* m) {
  if (!m) return;
  free(m->kc);
  free(m->vc);
  free(m->arrays);
  free(m);
}

int orc_len(const orc_model* m) { return m ? m->len : -1; }

int orc_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* Work buffers of one token's pass through the layers. */
typedef struct {
  uint16_t *x, *y, *qkv, *o, *att, *gu, *a, *dn;
} orc_tmp;

static void tmp_init(orc_tmp* t, const orc_config* c) {
  t->x = (uint16_t*)malloc(2 * (size_t)c->hidden);
  t->y = (uint16_t*)malloc(2 * (size_t)c->hidden);
  t->qkv = (uint16_t*)malloc(2 * (size_t)(c->n_q_heads + 2 * c->n_kv_heads) * c->head_dim);
  t->o = (uint16_t*)malloc(2 * (size_t)c->n_q_heads * c->head_dim);
  t->att = (uint16_t*)malloc(2 * (size_t)c->hidden);
  t->gu = (uint16_t*)malloc(2 * 2 * (size_t)c->ffn);
  t->a = (uint16_t*)malloc(2 * (size_t)c->ffn);
  t->dn = (uint16_t*)malloc(2 * (size_t)c->hidden);
}

static void tmp_free(orc_tmp* t) {
  free(t->x); free(t->y); free(t->qkv); free(t->o);
  free(t->att); free(t->gu); free(t->a); free(t->dn);
}

/* Attention half of layer l for a token at position pos: norm, q|k|v, per-head
 * norm, RoPE; stores k,v (bf16) into kdst/vdst.  q is left in t->qkv. */
static void layer_qkv(const orc_config* c, const orc_weights* w, int l, int pos, orc_tmp* t,
                      uint16_t* kdst, uint16_t* vdst) {
  int d = c->head_dim, Hq = c->n_q_heads, Hkv = c->n_kv_heads, H = c->hidden;
  orc_rmsnorm(t->x, w->attn_norm[l], H, c->rms_eps, t->y);
  orc_linear(w->wqkv[l], t->y, (Hq + 2 * Hkv) * d, H, t->qkv);
  uint16_t* q = t->qkv;
  uint16_t* k = t->qkv + (size_t)Hq * d;
  uint16_t* v = k + (size_t)Hkv * d;
  uint16_t* tmp = (uint16_t*)malloc(2 * (size_t)d);
  for (int h = 0; h < Hq; ++h) {
    if (c->qk_norm) {
      orc_rmsnorm(q + (size_t)h * d, w->q_norm[l], d, c->rms_eps, tmp);
      memcpy(q + (size_t)h * d, tmp, 2 * (size_t)d);
    }
    orc_rope(q + (size_t)h * d, d, pos, c->rope_theta);
  }
  for (int h = 0; h < Hkv; ++h) {
    if (c->qk_norm) {
      orc_rmsnorm(k + (size_t)h * d, w->k_norm[l], d, c->rms_eps, tmp);
      memcpy(k + (size_t)h * d, tmp, 2 * (size_t)d);
    }
    orc_rope(k + (size_t)h * d, d, pos, c->rope_theta);
  }
  free(tmp);
  memcpy(kdst, k, 2 * (size_t)Hkv * d);
  memcpy(vdst, v, 2 * (size_t)Hkv * d);
}

/* Rest of layer l once the keys/values of positions 0..pos are in kbase/vbase
 * (rows of n_kv_heads*head_dim): attention, projection + residual, FFN. */
static void layer_rest(const orc_config* c, const orc_weights* w, int l, int pos, orc_tmp* t,
                       const uint16_t* kbase, const uint16_t* vbase) {
  int d = c->head_dim, Hq = c->n_q_heads, Hkv = c->n_kv_heads, H = c->hidden, F = c->ffn;
  int group = Hq / Hkv; /* query head h reads kv head h / group */
  int stride = Hkv * d;
  for (int h = 0; h < Hq; ++h) {
    int kvh = h / group;
    orc_attend(t->qkv + (size_t)h * d, kbase + (size_t)kvh * d, vbase + (size_t)kvh * d, pos + 1,
               d, stride, t->o + (size_t)h * d);
  }
  orc_linear(w->wo[l], t->o, H, Hq * d, t->att);
  for (int i = 0; i < H; ++i) t->x[i] = orc_bf16(orc_f32(t->x[i]) + orc_f32(t->att[i]));
  orc_rmsnorm(t->x, w->ffn_norm[l], H, c->rms_eps, t->y);
  orc_linear(w->w_gate_up[l], t->y, 2 * F, H, t->gu);
  orc_glu(t->gu, t->gu + F, F, c->act, t->a);
  orc_linear(w->w_down[l], t->a, H, F, t->dn);
  for (int i = 0; i < H; ++i) t->x[i] = orc_bf16(orc_f32(t->x[i]) + orc_f32(t->dn[i]));
}

static void final_logits(const orc_config* c, const orc_weights* w, orc_tmp* t, float* logits) {
  orc_rmsnorm(t->x, w->final_norm, c->hidden, c->rms_eps, t->y);
  uint16_t* lg = (uint16_t*)malloc(2 * (size_t)c->vocab);
  orc_linear(w->lm_head, t->y, c->vocab, c->hidden, lg);
  for (int i = 0; i < c->vocab; ++i) logits[i] = orc_f32(lg[i]);
  free(lg);
}

int orc_forward(orc_model* m, int32_t token, float* logits) {
  const orc_config* c = &m->c;
  if (token < 0 || token >= c->vocab || m->len >= m->max_len) return -1;
  int pos = m->len;
  size_t row = kv_row(c);
  orc_tmp t;
  tmp_init(&t, c);
  memcpy(t.x, m->w.embed + (size_t)token * c->hidden, 2 * (size_t)c->hidden);
  for (int l = 0; l < c->n_layers; ++l) {
    uint16_t* kl = m->kc + (size_t)l * m->max_len * row;
    uint16_t* vl = m->vc + (size_t)l * m->max_len * row;
    layer_qkv(c, &m->w, l, pos, &t, kl + (size_t)pos * row, vl + (size_t)pos * row);
    layer_rest(c, &m->w, l, pos, &t, kl, vl);
  }
  if (logits) final_logits(c, &m->w, &t, logits);
  tmp_free(&t);
  m->len = pos + 1;
  return 0;
}

int orc_prefill(orc_model* m, const int32_t* tokens, int n, float* last_logits,
                int32_t* next_token) {
  if (!m || n <= 0 || m->len + n > m->max_len) return -1;
  float* lg = (float*)malloc(sizeof(float) * (size_t)m->c.vocab);
  for (int i = 0; i < n; ++i) {
    if (orc_forward(m, tokens[i], i == n - 1 ? lg : NULL)) {
      free(lg);
      return -1;
    }
  }
  if (last_logits) memcpy(last_logits, lg, sizeof(float) * (size_t)m->c.vocab);
  if (next_token) *next_token = orc_argmax(lg, m->c.vocab);
  free(lg);
  return 0;
}

int orc_decode(orc_model* m, int32_t token, float* logits, int32_t* next_token) {
  return orc_prefill(m, &token, 1, logits, next_token);
}

int orc_verify(orc_model* m, const int32_t* tokens, int K, float* logits, int32_t* argmax,
               int32_t* n_accepted, int32_t* correction) {
  if (!m || K <= 0 || m->len + K > m->max_len) return -1;
  int V = m->c.vocab, len0 = m->len;
  float* lg = (float*)malloc(sizeof(float) * (size_t)V);
  int32_t* am = (int32_t*)malloc(sizeof(int32_t) * (size_t)K);
  for (int r = 0; r < K; ++r) { /* row r: same pass as a decode at len0 + r */
    if (orc_forward(m, tokens[r], lg)) {
      m->len = len0;
      free(lg);
      free(am);
      return -1;
    }
    am[r] = orc_argmax(lg, V);
    if (logits) memcpy(logits + (size_t)r * V, lg, sizeof(float) * (size_t)V);
  }
  int n = 0;
  while (n < K - 1 && tokens[n + 1] == am[n]) ++n; /* longest matching prefix */
  m->len = len0 + 1 + n;                            /* keep pending + accepted rows */
  if (argmax) memcpy(argmax, am, sizeof(int32_t) * (size_t)K);
  if (n_accepted) *n_accepted = n;
  if (correction) *correction = am[n];
  free(lg);
  free(am);
  return 0;
}

int orc_truncate(orc_model* m, int new_len) {
  if (!m || new_len < 0 || new_len > m->len) return -1;
  m->len = new_len;
  return 0;
}

int orc_kv(const orc_model* m, int layer, int pos, uint16_t* k_out, uint16_t* v_out) {
  if (!m || layer < 0 || layer >= m->c.n_layers || pos < 0 || pos >= m->len) return -1;
  size_t row = kv_row(&m->c);
  size_t off = ((size_t)layer * m->max_len + pos) * row;
  if (k_out) memcpy(k_out, m->kc + off, 2 * row);
  if (v_out) memcpy(v_out, m->vc + off, 2 * row);
  return 0;
}

/* The per-token pass of orc_forward cut at one layer: the rows run one after
 * another in position order, each writing its own K/V before it attends, so
 * row r sees the given cache and rows 0 .. r. */
int orc_layer(const orc_config* c, const orc_weights* w, int layer, int pos, int K,
              const uint16_t* k_cache, const uint16_t* v_cache, const uint16_t* x_in,
              uint16_t* x_out, uint16_t* k_out, uint16_t* v_out) {
  if (!cfg_ok(c) || !w || layer < 0 || layer >= c->n_layers || pos < 0 || K <= 0 || !x_in || !x_out)
    return -1;
  if (pos > 0 && (!k_cache || !v_cache)) return -1;
  size_t row = kv_row(c), H = (size_t)c->hidden;
  uint16_t* kb = (uint16_t*)malloc(2 * (size_t)(pos + K) * row);
  uint16_t* vb = (uint16_t*)malloc(2 * (size_t)(pos + K) * row);
  if (pos > 0) {
    memcpy(kb, k_cache, 2 * (size_t)pos * row);
    memcpy(vb, v_cache, 2 * (size_t)pos * row);
  }
  orc_tmp t;
  tmp_init(&t, c);
  for (int r = 0; r < K; ++r) {
    memcpy(t.x, x_in + (size_t)r * H, 2 * H);
    layer_qkv(c, w, layer, pos + r, &t, kb + (size_t)(pos + r) * row, vb + (size_t)(pos + r) * row);
    layer_rest(c, w, layer, pos + r, &t, kb, vb);
    memcpy(x_out + (size_t)r * H, t.x, 2 * H);
  }
  if (k_out) memcpy(k_out, kb + (size_t)pos * row, 2 * (size_t)K * row);
  if (v_out) memcpy(v_out, vb + (size_t)pos * row, 2 * (size_t)K * row);
  tmp_free(&t);
  free(kb);
  free(vb);
  return 0;
}

int orc_head(const orc_config* c, const orc_weights* w, const uint16_t* x, float* logits) {
  if (!cfg_ok(c) || !w || !x || !logits) return -1;
  orc_tmp t;
  tmp_init(&t, c);
  memcpy(t.x, x, 2 * (size_t)c->hidden);
  final_logits(c, w, &t, logits);
  tmp_free(&t);
  return 0;
}

/* Layer-major recompute with no cache carried between calls: every layer is
 * applied to all n positions before the next layer starts. */
int orc_bruteforce(const orc_config* c, const orc_weights* w, const int32_t* tokens, int n,
                   float* logits) {
  if (!cfg_ok(c) || !w || n <= 0) return -1;
  for (int i = 0; i < n; ++i)
    if (tokens[i] < 0 || tokens[i] >= c->vocab) return -1;
  int H = c->hidden;
  size_t row = kv_row(c);
  size_t qrow = (size_t)(c->n_q_heads + 2 * c->n_kv_heads) * c->head_dim;
  uint16_t* X = (uint16_t*)malloc(2 * (size_t)n * H);
  uint16_t* Q = (uint16_t*)malloc(2 * (size_t)n * qrow);
  uint16_t* Kall = (uint16_t*)malloc(2 * (size_t)n * row);
  uint16_t* Vall = (uint16_t*)malloc(2 * (size_t)n * row);
  for (int t = 0; t < n; ++t)
    memcpy(X + (size_t)t * H, w->embed + (size_t)tokens[t] * H, 2 * (size_t)H);
  orc_tmp tp;
  tmp_init(&tp, c);
  for (int l = 0; l < c->n_layers; ++l) {
    for (int t = 0; t < n; ++t) { /* projections of every position first */
      memcpy(tp.x, X + (size_t)t * H, 2 * (size_t)H);
      layer_qkv(c, w, l, t, &tp, Kall + (size_t)t * row, Vall + (size_t)t * row);
      memcpy(Q + (size_t)t * qrow, tp.qkv, 2 * qrow);
    }
    for (int t = 0; t < n; ++t) { /* then causal attention and the FFN */
      memcpy(tp.x, X + (size_t)t * H, 2 * (size_t)H);
      memcpy(tp.qkv, Q + (size_t)t * qrow, 2 * qrow);
      layer_rest(c, w, l, t, &tp, Kall, Vall);
      memcpy(X + (size_t)t * H, tp.x, 2 * (size_t)H);
    }
  }
  for (int t = 0; t < n; ++t) {
    memcpy(tp.x, X + (size_t)t * H, 2 * (size_t)H);
    final_logits(c, w, &tp, logits + (size_t)t * c->vocab);
  }
  tmp_free(&tp);
  free(X); free(Q); free(Kall); free(Vall);
  return 0;
}
