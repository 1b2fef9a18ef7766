/* oracle.h -- plain, slow CPU reference of greedy block verification.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may include, link or
 * call this code; only the tests, the smoke check and the benchmark's CPU
 * baseline use it.  It shares no code, header or table with the CUDA library.
 *
 * What it computes (a decoder-only transformer, one token at a time):
 *   - Greedy speculative acceptance: a draft token is kept only if it equals the
 *     target's greedy next token after the same preceding ids; a causal block
 *     forward decides all of them at once ("Shape and cache history in Gemma
 *     block verification", section "Mechanism and failure").
 *   - Block verify writes the window's K/V into the committed cache, gives each
 *     row its own context length pos+r+1, and on a rejection truncates the
 *     cache to the accepted prefix ("Phase 23: Speculative Verify Parity",
 *     section 2, steps 1, 2 and 5).
 *   - Rows are computed exactly like single-token decode (same section, step 3).
 * Precision: weights and activations are bf16 values; every reduction runs in
 * fp32 in index order; results are rounded to bf16 (nearest even) at the layer
 * boundaries listed in oracle.c.  Logits are returned as fp32 holding bf16
 * values; argmax ties go to the lowest token id.
 */
#ifndef SV_ORACLE_H
#define SV_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct {
  int n_layers, hidden, n_q_heads, n_kv_heads, head_dim, ffn, vocab;
  float rms_eps, rope_theta;
  int qk_norm; /* 1: per-head RMSNorm of q and k before RoPE */
  int act;     /* 0: SwiGLU silu(gate)*up; 1: GeGLU with tanh-approximated GELU */
} orc_config;

/* bf16 bit patterns, row-major. Per-layer arrays hold n_layers pointers.
 *   wqkv      [(Hq + 2 Hkv) d, hidden]  rows: q heads, then k heads, then v heads
 *   wo        [hidden, Hq d]
 *   w_gate_up [2 ffn, hidden]           rows: gate, then up
 *   w_down    [hidden, ffn]
 *   embed / lm_head [vocab, hidden]; norms: [hidden] or [head_dim]        */
typedef struct {
  const uint16_t *embed, *lm_head, *final_norm;
  const uint16_t *const *attn_norm, *const *wqkv, *const *q_norm, *const *k_norm;
  const uint16_t *const *wo, *const *ffn_norm, *const *w_gate_up, *const *w_down;
} orc_weights;

typedef struct orc_model orc_model;

/* -------- whole-model calls (return 0, or -1 on a bad argument) -------- */
orc_model* orc_create(const orc_config* cfg, const orc_weights* w, int max_len);
void orc_destroy(orc_model* m);
int orc_len(const orc_model* m);
int orc_threads(void);
/* One token at position len; appends its K/V. logits: [vocab] or NULL. */
int orc_forward(orc_model* m, int32_t token, float* logits);
int orc_prefill(orc_model* m, const int32_t* tokens, int n, float* last_logits,
                int32_t* next_token);
int orc_decode(orc_model* m, int32_t token, float* logits, int32_t* next_token);
/* Block verify of rows [pending, d_1 .. d_{K-1}]: logits [K, vocab] (or NULL),
 * argmax [K] (or NULL); accepts the longest matching prefix and truncates. */
int orc_verify(orc_model* m, const int32_t* tokens, int K, float* logits, int32_t* argmax,
               int32_t* n_accepted, int32_t* correction);
int orc_truncate(orc_model* m, int new_len);
/* K and V (bf16 bits, [n_kv_heads * head_dim] each) cached at (layer, pos). */
int orc_kv(const orc_model* m, int layer, int pos, uint16_t* k_out, uint16_t* v_out);
/* No-cache recompute: logits [n, vocab] of every prefix tokens[0..t]. */
int orc_bruteforce(const orc_config* cfg, const orc_weights* w, const int32_t* tokens, int n,
                   float* logits);

/* -------- one layer / the head on given inputs (teacher forcing) -------- */
/* Layer `layer` applied to K consecutive rows at positions pos .. pos+K-1,
 * given that layer's cached K and V of positions 0 .. pos-1 (k_cache, v_cache:
 * [pos][n_kv_heads * head_dim] bf16 bits, may be NULL when pos = 0).  Row r
 * attends to the given cache plus the keys of rows 0 .. r, exactly as a decode
 * at position pos+r would.  x_in, x_out: [K][hidden] (the residual stream
 * before and after the layer); k_out, v_out: [K][n_kv_heads * head_dim] (the
 * rows' own cached K and V) or NULL. */
int orc_layer(const orc_config* cfg, const orc_weights* w, int layer, int pos, int K,
              const uint16_t* k_cache, const uint16_t* v_cache, const uint16_t* x_in,
              uint16_t* x_out, uint16_t* k_out, uint16_t* v_out);
/* Final RMSNorm + LM head of one residual-stream row x [hidden]: logits [vocab]
 * (fp32 holding bf16 values). */
int orc_head(const orc_config* cfg, const orc_weights* w, const uint16_t* x, float* logits);

/* -------- single operations, exposed so tests can pin them -------- */
uint16_t orc_bf16(float x);
float orc_f32(uint16_t b);
int32_t orc_argmax(const float* v, int n);
void orc_rmsnorm(const uint16_t* x, const uint16_t* g, int n, float eps, uint16_t* y);
void orc_linear(const uint16_t* W, const uint16_t* x, int rows, int cols, uint16_t* y);
void orc_rope(uint16_t* x, int d, int pos, float theta);
/* One query row over ctx cached positions of one kv head (all bf16 bits):
 * q [d]; K, V: ctx rows of stride `stride` elements; out [d]. */
void orc_attend(const uint16_t* q, const uint16_t* K, const uint16_t* V, int ctx, int d,
                int stride, uint16_t* out);
float orc_silu(float x);
float orc_gelu_tanh(float x);
/* Gated unit of one row: a[i] = bf16(bf16(act(gate[i])) * up[i]), act 0 = silu,
 * 1 = tanh-approximated GELU. */
void orc_glu(const uint16_t* gate, const uint16_t* up, int n, int act, uint16_t* a);

#ifdef __cplusplus
}
#endif
#endif
