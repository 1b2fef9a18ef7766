/* sv.h -- batch-invariant block verify for greedy speculative decoding (sm_103a).
 *
 * One context holds one sequence of a decoder-only transformer whose weights
 * live in device memory.  Its committed prefix is kept in a paged K/V cache
 * (page size 16, block table, pages from a fixed pool).  Every call runs the
 * same hand-written CUDA kernels on the context's stream:
 *   embed -> per layer [RMSNorm+QKV linear with QK-norm, RoPE and paged K/V
 *   write fused in its epilogue; split-KV paged attention (row r of a call sees
 *   pos+r+1 positions); attention projection + residual; RMSNorm+gate|up
 *   linear with SwiGLU/GeGLU; down projection + residual] -> final RMSNorm +
 *   LM head with per-tile argmax -> argmax/accept/truncate.
 *
 * Verify semantics follow "Phase 23: Speculative Verify Parity" section 2:
 * write the window's K/V into the committed cache in one shot (step 1), give
 * each row its own context length (step 2), compute rows with the same
 * rounding path as single-token decode (step 3), keep the K/V on acceptance
 * (step 4), truncate to the accepted prefix on rejection (step 5).  The
 * acceptance rule is the greedy one of "Shape and cache history in Gemma block
 * verification", section "Mechanism and failure": a draft is kept only while it
 * equals the target's greedy token after the same preceding ids; the
 * correction token is the target's greedy token at the first mismatch.
 *
 * Batch invariance: row r of any call is bit-identical to a single-token
 * decode at the same prefix, and results do not depend on how the cache was
 * built (one-token commits, block commits, one prefill) or on which physical
 * pages hold it.  Logits are returned as fp32 holding bf16 values; argmax ties
 * go to the lowest token id.
 *
 * The pending token: after every commit the library knows the target's
 * greedy token after the committed sequence (sv_prefill's next_token,
 * sv_decode's next_token, sv_verify's correction_token).  A verify window
 * starts with it ("Phase 23" section 2: the window is the known-correct next
 * token plus the drafts), so sv_verify and sv_decode reject any other
 * tokens[0] with SV_E_STATE and change nothing.  Committing tokens the model
 * did not choose (a prompt, forced ids) is sv_prefill's job.  After
 * sv_truncate to a shorter length the pending token is not known, and the
 * next window may start with any id.
 *
 * Conventions for every call:
 *   - Return 0 (SV_OK) or a negative SV_E_* code; sv_last_error() then gives a
 *     message.  On SV_E_INVAL / SV_E_NOMEM / SV_E_STATE the sequence state is
 *     unchanged.
 *     SV_E_CUDA means a CUDA call or a kernel's own bounds/timeout check
 *     failed; the context should then be destroyed.
 *   - Host pointers are read or written before the call returns; device
 *     pointers must stay valid until the work on the context's stream is done.
 *   - Calls on one context must not overlap (one host thread at a time).
 */
#ifndef SV_H
#define SV_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define SV_OK 0
#define SV_E_INVAL (-1)       /* bad argument or unsupported shape */
#define SV_E_NOMEM (-2)       /* page pool or device memory exhausted */
#define SV_E_CUDA (-3)        /* CUDA error or a kernel reported a failed check */
#define SV_E_STATE (-4)       /* call not valid in the current state (asynchronous work
                                 pending, or tokens[0] not the pending greedy token) */

#define SV_PAGE_SIZE 16       /* positions per KV page */
#define SV_MAX_K 32           /* most rows in one verify step */
#define SV_MAX_PREFILL_ROWS 128 /* most rows in one prefill block (tcgen05 linears) */

typedef struct sv_ctx sv_ctx;

/* Model shape and context limits.
 *   hidden % 128 == 0; ffn % 64 == 0; (n_q_heads + 2 n_kv_heads) head_dim % 128
 *   == 0; head_dim in {64, 128, 256}; qk_norm requires head_dim <= 128;
 *   n_q_heads % n_kv_heads == 0 and 16 % (n_q_heads / n_kv_heads) == 0.
 *   act: 0 = SwiGLU silu(gate)*up, 1 = GeGLU with tanh-approximated GELU.
 *   page_size must be 16.  max_k in [1, 32].  max_seq: longest sequence
 *   (committed + window), in [max_k, 1048576]; max_pages: KV pool size in
 *   pages (>= max_seq/16 for one full sequence). */
typedef struct {
  int32_t n_layers, hidden, n_q_heads, n_kv_heads, head_dim, ffn, vocab;
  float rms_eps, rope_theta;
  int32_t qk_norm, act, tie_embeddings;
  int32_t page_size, max_pages, max_k, max_seq;
  /* kv_delayed: when to write a verify window's K/V into the cache.
   *   0 = write-then-truncate: the step writes every window row into the
   *       cache pages and, after acceptance, zeroes the rejected rows.
   *   1 = delayed write-through ("Phase B decision — post-v4", section
   *       "Phase C gating item (new)", candidate C0 "Delayed KV write-through":
   *       verify produces its logits without committing K/V; K/V are committed
   *       once acceptance is decided): the window is written into three
   *       scratch pages per layer (seeded with the committed rows of its pages)
   *       and only the accepted rows are copied into the cache.  Rejected
   *       drafts never reach the cache pages.
   *   Both give bit-identical logits, argmax, acceptance and cache contents;
   *   1 costs 3 more pages per layer and one copy kernel per verify step.
   *   Prefill and decode steps commit every row and take path 0 either way. */
  int32_t kv_delayed;
} sv_config;

/* Device pointers to bf16 weights, row-major, borrowed for the context's
 * lifetime (the caller keeps them allocated and unchanged).  Each must be
 * 16-byte aligned.  Per-layer fields are HOST arrays of n_layers device
 * pointers (read during sv_create only).  sv_create also copies every linear
 * weight (wqkv, wo, w_gate_up, w_down, the LM head) into a tiled layout the
 * context owns and streams from: each 64-column k-block of a 128-row tile one
 * contiguous 16 KB run (the same memory again, 15.1 GB for the 8B shape);
 * SV_NO_TILED=1 streams the borrowed row-major weights instead.
 *   embed, lm_head [vocab, hidden] (lm_head may equal embed); final_norm [hidden]
 *   attn_norm, ffn_norm [hidden]; q_norm, k_norm [head_dim] (ignored if !qk_norm)
 *   wqkv [(n_q_heads + 2 n_kv_heads) head_dim, hidden]: q heads, k heads, v heads
 *   wo [hidden, n_q_heads head_dim]
 *   w_gate_up [2 ffn, hidden]: gate rows then up rows
 *   w_down [hidden, ffn]                                                        */
typedef struct {
  const void *embed, *lm_head, *final_norm;
  const void *const *attn_norm, *const *wqkv, *const *q_norm, *const *k_norm;
  const void *const *wo, *const *ffn_norm, *const *w_gate_up, *const *w_down;
} sv_weights;

/* Create a context on the current CUDA device.  cuda_stream: the caller's
 * stream (cudaStream_t), or NULL for the legacy stream.  A stream of the
 * caller's (not NULL, cudaStreamLegacy or cudaStreamPerThread) is the one
 * every call of the context runs on; it must outlive the context.  For the
 * default streams, which take no stream capture or programmatic dependent
 * launch, the library runs on a stream of its own, ordered after the
 * caller's stream at the start of each call and the caller's stream after
 * the library's work at the end.  Allocates the KV pool, block
 * table, activations, workspaces and the tiled weight copies (all owned by
 * the context); it synchronises the device first, since it reads the
 * weights.
 *
 * Environment switches, read here (results are bit-identical whichever are
 * set, the last one excepted; they change only how the work is launched):
 *   SV_NO_TC=1        steps of 9..32 rows use the mma.sync linear instead of
 *                     the tcgen05 one;
 *   SV_NO_GRAPHS=1    launch every step's kernels directly instead of through
 *                     a CUDA graph per (rows, mode, logits buffer);
 *   SV_NO_PDL=1       no programmatic dependent launch between a step's kernels;
 *   SV_NO_TILED=1     no tiled weight copies: the linears read the borrowed
 *                     row-major weights (less memory, slower streaming);
 *   SV_L2_PREFETCH=n  1: each linear prefetches the next one's first k-blocks
 *                     into L2; 2: only the QKV linear does, for the attention
 *                     projection (off by default: it measured slower);
 *   SV_TEST_WITHHOLD_PARTIAL=c  failure-detection test only: in the first
 *                     linear of every step (steps of at most 8 rows), CTA c
 *                     never hands its split-tile partial to the CTA that
 *                     finishes the tile, whose bounded wait (2 s) then gives
 *                     up: the call returns SV_E_CUDA (status bit 1, timeout)
 *                     and the context must be destroyed.  Results are then
 *                     wrong; never set it otherwise. */
int sv_create(const sv_config* cfg, const sv_weights* w, void* cuda_stream, sv_ctx** out);
void sv_destroy(sv_ctx* ctx);

/* Commit n tokens (host array) at positions len .. len+n-1, processed in the
 * row blocks sv_prefill_blocks gives (whatever max_k is; each block streams
 * every weight once).  last_logits_dev: device fp32 [vocab] for the logits
 * after the last token, or NULL.  next_token: the greedy token after the
 * last one (the new pending token).  Any ids may be committed.  The K/V of
 * every position are bit-identical to those of one-token commits, whatever
 * the block sizes ("Shape and cache history in Gemma block verification",
 * section "Same-prefix controls": one fresh prefill of the committed prefix
 * is one of the three cache histories that must agree).  Synchronous. */
int sv_prefill(sv_ctx* ctx, const int32_t* tokens_host, int n, float* last_logits_dev,
               int32_t* next_token);

/* Commit the pending token and return the greedy next token; logits_dev
 * [vocab] or NULL.  Identical to sv_verify with K = 1 (the single-token
 * decode every verify row must equal: "Phase 23" section 2 step 3), including
 * the SV_E_STATE check of `token`.  Synchronous. */
int sv_decode(sv_ctx* ctx, int32_t token, float* logits_dev, int32_t* next_token);

/* Block verify of K rows (host array) [pending, d_1 .. d_{K-1}] at positions
 * pos .. pos+K-1 (pos = current length): the window's K/V go into the cache
 * in one shot and row r attends to pos+r+1 positions ("Phase 23" section 2
 * steps 1-2).  Row 0 is always committed; drafts are accepted while d_{j+1}
 * equals the argmax of row j (the greedy rule of the Gemma page, section
 * "Mechanism and failure").  On return n_accepted in [0, K-1],
 * correction_token = argmax of row n_accepted (the new pending token), the
 * length is pos + 1 + n_accepted, and the K/V of rejected rows are zeroed
 * ("Phase 23" section 2 steps 4-5).  tokens[0] must be the pending token
 * when one is known (else SV_E_STATE, nothing changed).  logits_dev: device
 * fp32 [K, vocab] or NULL.  Synchronous. */
int sv_verify(sv_ctx* ctx, const int32_t* tokens_host, int K, float* logits_dev,
              int32_t* n_accepted, int32_t* correction_token);

/* Asynchronous verify with device-resident input and output, for callers that
 * keep drafts on the GPU (the same step as sv_verify).  tokens_dev: int32 [K];
 * result_dev: int32 [4] = {n_accepted, correction_token, new_length, status
 * (0 = ok)}; both memory of the context's device (else SV_E_INVAL, nothing
 * queued), 4-byte aligned, read and written by the step's kernels themselves
 * (so they must stay valid until the step is done).  The sequence length and
 * pending token are tracked on the device; pages must already cover every
 * position the call writes (see sv_reserve), otherwise the kernels skip the
 * writes and report a nonzero status.  A step whose tokens[0] is not the pending token commits nothing:
 * its result is {-1, pending, old length, status | 8}, and the next sv_sync
 * returns SV_E_STATE.  Call sv_sync before any synchronous call. */
int sv_verify_async(sv_ctx* ctx, const int32_t* tokens_dev, int K, float* logits_dev,
                    int32_t* result_dev);

/* Make pages cover positions [0, len) (page-table bookkeeping of the paged
 * cache that "Phase 23" section 2 step 1 writes into).  Synchronous. */
int sv_reserve(sv_ctx* ctx, int len);

/* Wait for asynchronous calls, read the device length and pending token back
 * and report any kernel status error (SV_E_CUDA) or a rejected window
 * (SV_E_STATE, see sv_verify_async).  Pages beyond the length are released
 * by the next synchronous call that changes the length. */
int sv_sync(sv_ctx* ctx);

/* Roll the sequence back to new_len <= length: zero the K/V of the removed
 * positions and release their pages ("Phase 23" section 2 step 5: truncate
 * the target cache to the accepted prefix).  A shorter length forgets the
 * pending token.  Synchronous. */
int sv_truncate(sv_ctx* ctx, int new_len);

/* Greedy speculative generation: `draft` proposes, `target` verifies.
 * (Phase 23: Speculative Verify Parity, section 2: drafts are checked by one
 * batched target forward, the longest matching prefix is accepted and the
 * rejected tail rolled back.)  Both contexts hold the same committed tokens
 * (e.g. one prompt prefilled into each) and share the vocabulary; `pending`
 * is the target's greedy token after them (sv_prefill's next_token).  Each
 * round the drafter decodes K-1 tokens after the pending one, the target
 * verifies the K-row block [pending, drafts], and the drafter is rolled back
 * (or advanced) to the target's length.  Rounds run until at least n_new
 * tokens are committed.  The tokens are the target's own greedy continuation,
 * whatever the drafter proposes.
 *   K in [1, target max_k]; K = 1 is plain decoding.  Both contexts need
 *   max_seq >= length + n_new + K.
 *   out_tokens: host int32 [n_new + K - 1]; *n_out (n_new .. n_new + K - 1)
 *   of them are written: every token committed, in order, starting with
 *   `pending`.  *next_pending: the target's greedy token after them.
 *   stats (or NULL): int32 [3] = {verify steps, drafts accepted, drafts
 *   proposed}.
 * Errors: SV_E_INVAL (arguments), SV_E_STATE (lengths differ or asynchronous
 * work pending), or those of the calls it makes (a drafter's error is
 * reported through the target's sv_last_error).  Synchronous. */
int sv_spec_generate(sv_ctx* target, sv_ctx* draft, int32_t pending, int K, int n_new,
                     int32_t* out_tokens, int32_t* n_out, int32_t* next_pending, int32_t* stats);

/* Current committed length (as of the last synchronous call or sv_sync). */
int sv_seq_len(const sv_ctx* ctx);

/* Test read of the paged cache ("Phase 23" section 2 step 1 is what writes
 * it).  Copies the cached K and V of positions [first, first+count) of one
 * layer into two device buffers k_dst_dev, v_dst_dev, each bf16 [count,
 * n_kv_heads, head_dim].  Positions may run to the end of the last page the
 * sequence holds, past its length: every slot there is zero (rejected rows
 * and truncated positions are zeroed), which tests check.  Synchronous. */
int sv_kv_read(sv_ctx* ctx, int layer, int first, int count, void* k_dst_dev, void* v_dst_dev);

/* Shuffle the order in which free pages are handed out (seeded).  Results
 * must not depend on it; tests use it to build the same prefix on different
 * physical pages (a cache-history change in the sense of the Gemma page,
 * section "Same-prefix controls"). */
int sv_shuffle_pages(sv_ctx* ctx, uint64_t seed);

/* Test hook for per-layer comparisons.  While hidden_dev is not NULL, every
 * step of at most max_rows rows (1..32) also copies its residual stream into
 * hidden_dev, bf16 [n_layers + 1][rows][hidden]: entry 0 holds the embedded
 * rows, entry l + 1 the output of layer l (the last one is the input of the
 * final RMSNorm).  Such steps run without CUDA graphs or programmatic
 * dependent launch; results are bit-identical either way.  NULL turns it off.
 * The buffer must stay valid while it is set. */
int sv_trace_hidden(sv_ctx* ctx, void* hidden_dev, int max_rows);

/* Number of kernel launches in one step of K rows: with_head = 1 counts a
 * verify step (LM head and acceptance, and for kv_delayed with K > 1 the
 * window copy), 0 a prefill block without the LM head (a block of more than
 * 32 rows is embedded 32 rows a launch).  Steps of more than 8 rows on the
 * tcgen05 form add one row normalisation before each QKV, gate|up and LM
 * head linear. */
int sv_step_kernel_count(const sv_ctx* ctx, int K, int with_head);

/* The row blocks sv_prefill cuts n tokens into, in order, written to
 * sizes[0 .. count-1]; returns count, or SV_E_INVAL if n < 1 or more than
 * max_blocks blocks would be needed (sizes may be NULL to ask for the count
 * only, with max_blocks 0).  The last block holds the 1..SV_MAX_K rows left
 * over; the others hold SV_MAX_K rows, or with use_tc (the tcgen05 linears,
 * the default unless SV_NO_TC=1 was set when the context was created) up to
 * SV_MAX_PREFILL_ROWS rows, always a multiple of SV_MAX_K.  Host only: needs
 * no context and no GPU. */
int sv_prefill_blocks(int n, int use_tc, int32_t* sizes, int max_blocks);

/* Measurement hook for the dominant kernel class.  Launches one linear of the
 * model for K rows, once per layer (distinct weights, so every launch streams
 * from HBM), `reps` times after one untimed pass, chained as inside a step on
 * the context's stream, and timed with CUDA events on that stream.
 *   which: SV_LIN_O, SV_LIN_GATE_UP, SV_LIN_DOWN or SV_LIN_LM_HEAD
 *   avg_us: mean device time per launch
 *   bytes_per_launch (or NULL): algorithmic bytes of one launch = weight bytes
 *     + input rows + output rows (bf16)
 * Overwrites the step's scratch activations; the sequence and its cache are
 * untouched.  Synchronous. */
#define SV_LIN_O 1
#define SV_LIN_GATE_UP 2
#define SV_LIN_DOWN 3
#define SV_LIN_LM_HEAD 4
int sv_time_linear(sv_ctx* ctx, int which, int K, int reps, float* avg_us, double* bytes_per_launch);

/* LM-head step that allocates no device memory.  There is no counterpart to
 * this call on the pages the library follows; it exists for callers that may
 * not call cudaMalloc: code running in a process whose GPU memory is already
 * reserved by another allocator (a serving runtime's pool, or a plugin inside
 * one), and latency-critical code that cannot accept the device-wide
 * synchronisation an allocation may cause.
 *
 * Computes, for M rows x (bf16 [M, hidden], device):
 *   logits = bf16(RMSNorm(x; gain, eps) . W^T)   as fp32 [M, vocab] (device)
 *   argmax[m] = greedy token of row m (largest logit, lowest id on ties)
 * with the same K split and rounding as the context's LM head.  It runs the
 * mma.sync form of the batch-invariant linear for every M; the context runs
 * that form up to 8 rows and the tcgen05 form for 9-32 rows, and the two are
 * bit-identical, so for a model with no layers this call's logits and argmax
 * equal sv_verify's bit for bit at every M.
 *   gain: bf16 [hidden]; W: bf16 [vocab, hidden]; all inputs 16-byte aligned.
 *   argmax_dev: int32 [M] or NULL; status_dev: int32 [1] or NULL, set to 0, or
 *     to the kernels' failure bits (1 timeout).  When the call returns non-zero,
 *     logits_dev, argmax_dev and status_dev are undefined (work already queued
 *     may or may not have written them).
 *   cuda_stream: the stream to run on (NULL = legacy stream).  Asynchronous.
 * Scratch: the split-K partials (one slot per CTA), the argmax partials and
 * the row statistics live in one fixed 8 MiB device array inside the library
 * (held on every GPU that loads it until the process exits).  Shapes whose
 * scratch would not fit return SV_E_NOMEM; the scratch is about
 *   8 * M * ceil(vocab/128) + 4 * G * 128 * (8, 16 or 32 for M <= 8, 16, 32)
 *   bytes, G <= the SM count (one CTA per SM, equal shares of W): with 152
 *   SMs a vocabulary of up to about 2.9 million ids fits at any M.
 * Other limits: 1 <= M <= 32, hidden % 128 == 0 (else SV_E_INVAL).
 * The first call on a device looks up the array's address and sets kernel
 * attributes for that device; make that first call before any stream capture.
 * Every call uses the same array: calls that overlap on the GPU (other
 * streams, other threads) race and must be serialised by the caller. */
int sv_lm_head_noalloc(const void* x_dev, const void* gain_dev, const void* w_dev, int M, int hidden,
                       int vocab, float eps, float* logits_dev, int32_t* argmax_dev,
                       int32_t* status_dev, void* cuda_stream);

const char* sv_last_error(const sv_ctx* ctx);

#ifdef __cplusplus
}
#endif
#endif
