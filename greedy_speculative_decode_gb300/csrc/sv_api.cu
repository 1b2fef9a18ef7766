// sv_api.cu -- the C-ABI: context, page pool and block table, step
// orchestration (one CUDA graph per step shape, kernels chained with
// programmatic dependent launch), and the synchronous / asynchronous calls.
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <string>
#include <vector>

#include "sv_internal.h"
#include "linear_tc.h"

using namespace sv;

struct GraphEntry {
  int M, mode;
  float* logits;
  cudaGraph_t graph;  // kept: its nodes name the ones of `exec` to update
  cudaGraphExec_t exec;
  cudaGraphNode_t io_nodes[2];  // the embedding and accept nodes (both or none)
  int n_io;
  StepIo io;  // what those nodes take now
};

struct sv_ctx {
  sv_config cfg;
  int device = 0, num_sms = 0;
  cudaStream_t user_stream = nullptr, stream = nullptr;
  cudaEvent_t ev = nullptr;
  bool use_graphs = true;
  bool use_pdl = true;  // chain a step's kernels with programmatic dependent launch
  bool use_tc = true;   // 9-32 row linears on tcgen05 (bit-identical to the mma.sync form)
  bool use_tiled = true;  // stream the linear weights from the context's tiled copy
  int prefetch_mode = 0;  // 0 none, 1 every linear prefetches the next one into L2, 2 only QKV -> O
  int withhold_cta1 = 0;  // test hook: see LinParams::withhold_cta1 (first linear of a step only)
  // weights
  const bf16 *embed = nullptr, *lm_head = nullptr, *final_norm = nullptr;
  std::vector<const bf16*> attn_norm, q_norm, k_norm, ffn_norm;
  std::vector<LinearDesc> lin_qkv, lin_o, lin_gu, lin_down;
  LinearDesc lin_head;
  CUtensorMap kmap, vmap;
  // input rows of the tcgen05 linears: boxes of 64 columns x 32 rows, and x 128 rows
  CUtensorMap xmap_x, xmap_o, xmap_a, xmap_xn, xmap128_x, xmap128_o, xmap128_a, xmap128_xn;
  // device memory owned by the context
  std::vector<void*> allocs;
  bf16 *kpool = nullptr, *vpool = nullptr;
  size_t layer_stride = 0;  // elements per layer in each pool
  int pool_pages = 0;       // pages per layer: max_pages, plus kWinPages scratch pages when delayed
  int* block_table = nullptr;
  int* bt_shadow = nullptr;  // delayed write-through: block table with the window on scratch pages
  SvState* st = nullptr;
  bf16 *x = nullptr, *q = nullptr, *o = nullptr, *a = nullptr;
  bf16* xn = nullptr;  // normalised input rows of a prefill block of more than kMaxK rows
  float* x_ss = nullptr;
  float2* rope = nullptr;
  float2* part_ml = nullptr;
  float* part_o = nullptr;
  int max_splits = 0;
  uint32_t* ws = nullptr;     // split-tile partial slots, one per CTA (every byte 0xff when idle)
  uint32_t* ws_tc = nullptr;         // the same for the tcgen05 form (every byte 0xff when idle)
  float* am_val = nullptr;
  int* am_idx = nullptr;
  // pinned host staging
  int32_t* pin_in = nullptr;   // [cap_len, tokens...] per row block of one call
  size_t pin_in_len = 0;       // ints: max_seq + one cap_len slot per block of a full prefill
  SvState* pin_out = nullptr;  // read-back of the device state
  // the same two as the kernels address them (pinned host memory is mapped
  // under unified addressing); null: the synchronous verify copies instead
  int32_t* pin_in_dev = nullptr;
  SvState* pin_out_dev = nullptr;
  int dev_cap = -1;  // st->cap_len as last set by the host (-1: not known)
  int* pin_bt = nullptr;       // block table mirror
  // test hook: the residual stream of each step's rows after every layer
  bf16* trace = nullptr;  // [n_layers + 1][rows][hidden]
  int trace_rows = 0;
  // host-side sequence state
  int seq_len = 0;
  int pending = -1;  // greedy token after the committed sequence (-1: not known)
  int n_alloc = 0;  // logical pages with a physical page
  int bt_len = 0;   // entries of the block table
  std::vector<int> free_pages;
  bool async_pending = false;
  std::vector<GraphEntry> graphs;
  std::string err;
};

namespace sv {

bool make_bf16_map(CUtensorMap* m, const void* ptr, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  // the driver's encoder, looked up once per process (thread-safe initialisation)
  static const PFN_cuTensorMapEncodeTiled_v12000 enc = []() -> PFN_cuTensorMapEncodeTiled_v12000 {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }();
  if (!enc) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box,
                   estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace sv

namespace {

int fail(sv_ctx* c, int code, const char* fmt, ...) {
  if (c) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    c->err = buf;
  }
  return code;
}

#define CK(call)                                                                           \
  do {                                                                                     \
    cudaError_t e_ = (call);                                                               \
    if (e_ != cudaSuccess)                                                                 \
      return fail(ctx, SV_E_CUDA, "%s failed: %s", #call, cudaGetErrorString(e_));        \
  } while (0)

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int make_linear(sv_ctx* ctx, LinearDesc* d, const void* w, int rows, int Kd, int n_tiles, int map) {
  if (!w || !aligned16(w)) return fail(ctx, SV_E_INVAL, "weight pointer null or not 16-byte aligned");
  d->N = rows;
  d->Kd = Kd;
  d->n_tiles = n_tiles;
  linear_partition(n_tiles, Kd, ctx->num_sms, &d->grid, &d->max_seg);
  if (d->max_seg > kLinMaxSeg)
    return fail(ctx, SV_E_INVAL, "weight of %d x %d is split over %d CTAs per tile (max %d)", rows, Kd,
                d->max_seg, kLinMaxSeg);
  d->map_kind = map;
  if (!make_bf16_map(&d->map, w, (uint64_t)rows, (uint64_t)Kd, 64))
    return fail(ctx, SV_E_CUDA, "cuTensorMapEncodeTiled failed for a weight of %d x %d", rows, Kd);
  d->tiled = nullptr;
  if (ctx->use_tiled) {
    // the context's own copy in the tiled layout: every k-block one
    // contiguous 16 KB run, streamed with one bulk copy (every byte is
    // written by the repack, so no clearing)
    void* t = nullptr;
    const size_t bytes = tiled_bytes(n_tiles, Kd);
    cudaError_t e = cudaMalloc(&t, bytes);
    if (e != cudaSuccess)
      return fail(ctx, SV_E_NOMEM, "cudaMalloc(%zu) for a tiled weight failed: %s", bytes, cudaGetErrorString(e));
    ctx->allocs.push_back(t);
    d->tiled = static_cast<uint8_t*>(t);
    e = launch_tile_weight(static_cast<const bf16*>(w), rows, Kd, n_tiles, map, map == MAP_GATE_UP ? rows / 2 : 0,
                           d->tiled, ctx->stream);
    if (e != cudaSuccess) return fail(ctx, SV_E_CUDA, "weight repack failed: %s", cudaGetErrorString(e));
  }
  return SV_OK;
}

template <typename T>
int dalloc(sv_ctx* ctx, T** p, size_t count) {
  void* q = nullptr;
  size_t bytes = count * sizeof(T);
  if (bytes == 0) bytes = 16;
  cudaError_t e = cudaMalloc(&q, bytes);
  if (e != cudaSuccess) return fail(ctx, SV_E_NOMEM, "cudaMalloc(%zu) failed: %s", bytes, cudaGetErrorString(e));
  ctx->allocs.push_back(q);
  *p = static_cast<T*>(q);
  e = cudaMemset(q, 0, bytes);
  if (e != cudaSuccess) return fail(ctx, SV_E_CUDA, "cudaMemset failed: %s", cudaGetErrorString(e));
  return SV_OK;
}

int mp_of(int M) { return M <= 8 ? 8 : (M <= 16 ? 16 : 32); }

// Rows of the next prefill block when `rest` prompt tokens are left: the
// last block takes the 1..kMaxK rows left over, the others kMaxK rows, or
// with the tcgen05 linear up to kTcMaxRows (a multiple of kMaxK).
int prefill_block(int rest, bool use_tc) {
  const int tail = (rest - 1) % kMaxK + 1;
  if (rest == tail) return rest;
  return use_tc ? std::min(kTcMaxRows, rest - tail) : kMaxK;
}

// One linear of a step: blocks of more than 8 rows go to the tcgen05 form.
cudaError_t run_linear(sv_ctx* ctx, const LinearDesc& d, const LinParams& p, int epi, bool norm,
                       cudaStream_t s, bool pdl, const LinearDesc* next) {
  if (ctx->use_tc && p.M > 8) {
    const bool big = p.M > kMaxK;
    const CUtensorMap* xm = p.X == ctx->xn ? (big ? &ctx->xmap128_xn : &ctx->xmap_xn)
                            : p.X == ctx->x ? (big ? &ctx->xmap128_x : &ctx->xmap_x)
                                            : (p.X == ctx->o ? (big ? &ctx->xmap128_o : &ctx->xmap_o)
                                                             : (big ? &ctx->xmap128_a : &ctx->xmap_a));
    return launch_linear_tc(d, *xm, ctx->ws_tc, p, epi, norm, s, pdl, next);
  }
  return launch_linear(d, p, epi, norm, s, pdl, next);
}

// ------------------------------------------------------------------ the step
enum LinWhich { LIN_QKV = 0, LIN_O = 1, LIN_GU = 2, LIN_DOWN = 3, LIN_HEAD = 4 };

// Delayed write-through applies to verify steps of more than one row (a
// single row is committed whenever the step is).
bool step_delayed(const sv_ctx* ctx, int M, int mode) {
  return ctx->bt_shadow != nullptr && mode == MODE_VERIFY && M > 1;
}

// The block table through which a step's kernels write and read K/V.
const int* step_table(const sv_ctx* ctx, int M, int mode) {
  return step_delayed(ctx, M, mode) ? ctx->bt_shadow : ctx->block_table;
}

KvDelay kv_delay(const sv_ctx* ctx, int M, int mode) {
  KvDelay dl = {};
  dl.bt_shadow = step_delayed(ctx, M, mode) ? ctx->bt_shadow : nullptr;
  dl.win0 = ctx->cfg.max_pages;
  dl.bt_len = ctx->bt_len;
  return dl;
}

// Parameters of one linear of one step of M rows.
LinParams lin_params(sv_ctx* ctx, int which, int l, int M, int mode, float* logits, int* epi,
                     bool* norm, const LinearDesc** desc) {
  const sv_config& c = ctx->cfg;
  const int H = c.hidden, d = c.head_dim, Hq = c.n_q_heads;
  LinParams p = {};
  p.ss_tiles = H / 128;
  p.eps = c.rms_eps;
  p.M = M;
  p.ffn = c.ffn;
  p.head_dim = d;
  p.ws = ctx->ws;
  p.block_table = step_table(ctx, M, mode);
  p.rope = ctx->rope;
  p.n_q_heads = Hq;
  p.n_kv_heads = c.n_kv_heads;
  p.act = c.act;
  p.vocab = c.vocab;
  p.st = ctx->st;
  const LinearDesc* ld = nullptr;
  if (which == LIN_QKV) {
    ld = &ctx->lin_qkv[l];
    *epi = EPI_QKV;
    *norm = true;
    p.X = ctx->x;
    p.x_ss = ctx->x_ss;
    p.gain = ctx->attn_norm[l];
    p.out = ctx->q;
    p.out_stride = Hq * d;
    p.kcache = ctx->kpool + (size_t)l * ctx->layer_stride;
    p.vcache = ctx->vpool + (size_t)l * ctx->layer_stride;
    p.q_gain = c.qk_norm ? ctx->q_norm[l] : nullptr;
    p.k_gain = c.qk_norm ? ctx->k_norm[l] : nullptr;
  } else if (which == LIN_O) {
    ld = &ctx->lin_o[l];
    *epi = EPI_RESID;
    *norm = false;
    p.X = ctx->o;
    p.out = ctx->x;
    p.out_stride = H;
    p.out_ss = ctx->x_ss;
  } else if (which == LIN_GU) {
    ld = &ctx->lin_gu[l];
    *epi = EPI_GLU;
    *norm = true;
    p.X = ctx->x;
    p.x_ss = ctx->x_ss;
    p.gain = ctx->ffn_norm[l];
    p.out = ctx->a;
    p.out_stride = c.ffn;
  } else if (which == LIN_DOWN) {
    ld = &ctx->lin_down[l];
    *epi = EPI_RESID;
    *norm = false;
    p.X = ctx->a;
    p.out = ctx->x;
    p.out_stride = H;
    p.out_ss = ctx->x_ss;
  } else {
    ld = &ctx->lin_head;
    *epi = EPI_LOGITS;
    *norm = true;
    p.X = ctx->x;
    p.x_ss = ctx->x_ss;
    p.gain = ctx->final_norm;
    p.logits = logits;
    p.logits_row0 = (mode == MODE_PREFILL) ? M - 1 : 0;
    p.am_val = ctx->am_val;
    p.am_idx = ctx->am_idx;
  }
  p.Kd = ld->Kd;
  p.n_tiles = ld->n_tiles;
  p.max_seg = ld->max_seg;
  p.map = ld->map_kind;
  p.grid = ld->grid;
  p.wt = ld->tiled;
  *desc = ld;
  return p;
}

AttnParams attn_params(sv_ctx* ctx, int l, int M, int mode) {
  const sv_config& c = ctx->cfg;
  AttnParams ap = {};
  ap.q = ctx->q;
  ap.block_table = step_table(ctx, M, mode);
  ap.st = ctx->st;
  ap.part_ml = ctx->part_ml;
  ap.part_o = ctx->part_o;
  ap.out = ctx->o;
  ap.M = M;
  ap.n_q_heads = c.n_q_heads;
  ap.n_kv_heads = c.n_kv_heads;
  ap.max_splits = ctx->max_splits;
  ap.max_pages = ctx->pool_pages;
  ap.layer = l;
  ap.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)c.head_dim));
  return ap;
}

// Enqueue every kernel of one step of M rows on ctx->stream.
int enqueue_step(sv_ctx* ctx, int M, int mode, float* logits, const StepIo& io) {
  const sv_config& c = ctx->cfg;
  const int H = c.hidden, d = c.head_dim, Hkv = c.n_kv_heads;
  cudaStream_t s = ctx->stream;
  // the trace hook copies the residual stream between kernels: no programmatic
  // dependent launch while it is on
  const bool tracing = ctx->trace != nullptr && M <= ctx->trace_rows;
  const bool pdl = ctx->use_pdl && !tracing;
  const KvDelay dl = kv_delay(ctx, M, mode);
  if (dl.bt_shadow != nullptr)
    CK(launch_kv_window_in(ctx->kpool, ctx->vpool, ctx->layer_stride, ctx->block_table, dl, ctx->st, c.n_layers,
                           Hkv, d, M, s));
  // (blocks of more than kMaxK rows are embedded before the step, kMaxK rows
  // at a time: see sv_prefill)
  if (M <= kMaxK)
    CK(launch_embed(ctx->embed, H, c.vocab, M, ctx->x, ctx->x_ss, ctx->st, mode == MODE_VERIFY, s,
                    pdl && dl.bt_shadow != nullptr, io));
  auto trace_copy = [&](int entry) -> cudaError_t {
    if (!tracing) return cudaSuccess;
    return cudaMemcpyAsync(ctx->trace + (size_t)entry * M * H, ctx->x, (size_t)M * H * sizeof(bf16),
                           cudaMemcpyDeviceToDevice, s);
  };
  CK(trace_copy(0));
  const int G = c.n_q_heads / Hkv;
  const int n_rb = (M + kAttnQ / G - 1) / (kAttnQ / G);
  const int attn_items_max = ctx->max_splits * Hkv * n_rb;  // attention work items at max_seq
  const int attn_grid = std::max(1, std::min(attn_items_max, ctx->num_sms));
  const bool attn_multi = attn_items_max > attn_grid;
  int epi;
  bool norm;
  const LinearDesc* ld;
  // the weight each linear prefetches into L2: the next one of the step (the
  // last one's next is the first of the following step)
  const bool head = mode != MODE_BODY;
  auto next_of = [&](int which, int l) -> const LinearDesc* {
    if (ctx->prefetch_mode == 0) return nullptr;
    if (ctx->prefetch_mode == 2) return which == LIN_QKV ? &ctx->lin_o[l] : nullptr;
    switch (which) {
      case LIN_QKV: return &ctx->lin_o[l];
      case LIN_O: return &ctx->lin_gu[l];
      case LIN_GU: return &ctx->lin_down[l];
      case LIN_DOWN:
        if (l + 1 < c.n_layers) return &ctx->lin_qkv[l + 1];
        return head ? &ctx->lin_head : &ctx->lin_qkv[0];
      default: return c.n_layers > 0 ? &ctx->lin_qkv[0] : nullptr;
    }
  };
  // Steps of more than 8 rows (the tcgen05 form) normalise the input rows of
  // QKV, gate|up and the LM head once, in a kernel of their own, instead of
  // in every CTA's prologue (and at every restage of the input window, or for
  // 128-row blocks every ring stage): the same values (k_norm_rows).  On the
  // 8B shape K=16 3408 -> 3374 us, K=32 4258 -> 3960.
  auto prenorm = [&](LinParams& p, bool& nm) -> cudaError_t {
    if (M <= 8 || !nm || !ctx->use_tc) return cudaSuccess;
    cudaError_t e = launch_norm_rows(p.X, p.x_ss, p.gain, ctx->xn, M, H, c.rms_eps, s, pdl);
    p.X = ctx->xn;
    nm = false;
    return e;
  };
  for (int l = 0; l < c.n_layers; ++l) {
    LinParams p = lin_params(ctx, LIN_QKV, l, M, mode, logits, &epi, &norm, &ld);
    if (l == 0) p.withhold_cta1 = ctx->withhold_cta1;
    CK(prenorm(p, norm));
    CK(run_linear(ctx, *ld, p, epi, norm, s, pdl, next_of(LIN_QKV, l)));
    AttnParams ap = attn_params(ctx, l, M, mode);
    CK(launch_attention(ctx->kmap, ctx->vmap, ap, d, attn_grid, attn_multi, s, pdl));
    CK(launch_attn_combine(ap, d, s, pdl));
    for (int w : {LIN_O, LIN_GU, LIN_DOWN}) {
      p = lin_params(ctx, w, l, M, mode, logits, &epi, &norm, &ld);
      CK(prenorm(p, norm));
      CK(run_linear(ctx, *ld, p, epi, norm, s, pdl, next_of(w, l)));
    }
    CK(trace_copy(l + 1));
  }
  if (head) {  // final RMSNorm + LM head + per-tile argmax
    LinParams p = lin_params(ctx, LIN_HEAD, 0, M, mode, logits, &epi, &norm, &ld);
    CK(prenorm(p, norm));
    CK(run_linear(ctx, *ld, p, epi, norm, s, pdl, next_of(LIN_HEAD, 0)));
  }
  CK(launch_accept(ctx->st, ctx->am_val, ctx->am_idx, ctx->lin_head.n_tiles, M, mode, ctx->kpool,
                   ctx->vpool, ctx->layer_stride, ctx->block_table, c.n_layers, Hkv, d, dl, s, pdl, io));
  return SV_OK;
}

void destroy_graphs(sv_ctx* ctx) {
  for (auto& g : ctx->graphs) {
    cudaGraphExecDestroy(g.exec);
    cudaGraphDestroy(g.graph);
  }
  ctx->graphs.clear();
}

// The graph of this step shape, captured on first use (with the state
// block's tokens and result: StepIo{}).  Returns its index in ctx->graphs.
int step_graph(sv_ctx* ctx, int M, int mode, float* logits, size_t* index) {
  for (size_t i = 0; i < ctx->graphs.size(); ++i) {
    const GraphEntry& g = ctx->graphs[i];
    if (g.M == M && g.mode == mode && g.logits == logits) {
      *index = i;
      return SV_OK;
    }
  }
  if (ctx->graphs.size() >= 64) {  // (launches of the cached graphs may still be queued)
    CK(cudaStreamSynchronize(ctx->stream));
    destroy_graphs(ctx);
  }
  CK(cudaStreamBeginCapture(ctx->stream, cudaStreamCaptureModeThreadLocal));
  int rc = enqueue_step(ctx, M, mode, logits, StepIo{});
  cudaGraph_t graph = nullptr;
  cudaError_t e = cudaStreamEndCapture(ctx->stream, &graph);
  if (rc != SV_OK) {
    if (graph) cudaGraphDestroy(graph);
    return rc;
  }
  if (e != cudaSuccess) return fail(ctx, SV_E_CUDA, "stream capture failed: %s", cudaGetErrorString(e));
  GraphEntry g = {M, mode, logits, graph, nullptr, {nullptr, nullptr}, 0, StepIo{}};
  size_t n = 0;
  std::vector<cudaGraphNode_t> nodes;
  if (cudaGraphGetNodes(graph, nullptr, &n) == cudaSuccess) {
    nodes.resize(n);
    if (cudaGraphGetNodes(graph, nodes.data(), &n) != cudaSuccess) nodes.clear();
  }
  cudaGetLastError();
  for (cudaGraphNode_t node : nodes)
    if (step_io_node(node) && g.n_io < 2) g.io_nodes[g.n_io++] = node;
  if (g.n_io != 2) g.n_io = 0;  // (a block of more than kMaxK rows has no embedding node)
  e = cudaGraphInstantiate(&g.exec, graph, 0);
  if (e != cudaSuccess) {
    cudaGraphDestroy(graph);
    return fail(ctx, SV_E_CUDA, "graph instantiate failed: %s", cudaGetErrorString(e));
  }
  // the nodes take a new StepIo only if the runtime hands their captured
  // arguments back; otherwise the calls fall back to copies (step_takes_io)
  for (int k = 0; k < g.n_io; ++k)
    if (set_step_io(g.exec, g.io_nodes[k], StepIo{}) != cudaSuccess) {
      cudaGetLastError();
      g.n_io = 0;
    }
  ctx->graphs.push_back(g);
  *index = ctx->graphs.size() - 1;
  return SV_OK;
}

// Whether a step of this shape can take its tokens and result from and to
// the caller's buffers (StepIo) instead of the state block.
bool step_takes_io(sv_ctx* ctx, int M, int mode, float* logits) {
  if (!ctx->use_graphs || ctx->trace) return true;
  size_t i = 0;
  if (step_graph(ctx, M, mode, logits, &i) != SV_OK) return false;  // run_step reports it
  return ctx->graphs[i].n_io == 2;
}

// Run one step: replay (capturing on first use) the graph of this shape,
// its embedding and accept nodes pointed at `io` first where they differ.
int run_step(sv_ctx* ctx, int M, int mode, float* logits, const StepIo& io = StepIo{}) {
  if (!ctx->use_graphs || ctx->trace) return enqueue_step(ctx, M, mode, logits, io);
  size_t i = 0;
  int rc = step_graph(ctx, M, mode, logits, &i);
  if (rc) return rc;
  GraphEntry& g = ctx->graphs[i];
  if (g.io.tokens != io.tokens || g.io.result != io.result) {
    if (g.n_io != 2) return fail(ctx, SV_E_INVAL, "this step's graph takes no caller buffers");
    for (int k = 0; k < 2; ++k) CK(set_step_io(g.exec, g.io_nodes[k], io));
    g.io = io;
  }
  CK(cudaGraphLaunch(g.exec, ctx->stream));
  return SV_OK;
}

// ------------------------------------------------------------------ pages
int pages_for(int len) { return (len + kPage - 1) / kPage; }

// Give logical pages [n_alloc, pages_for(len)) physical pages and upload them.
int ensure_pages(sv_ctx* ctx, int len) {
  const int need = pages_for(len);
  if (need > ctx->bt_len) return fail(ctx, SV_E_INVAL, "length %d exceeds max_seq %d", len, ctx->cfg.max_seq);
  if (need <= ctx->n_alloc) return SV_OK;
  if ((int)ctx->free_pages.size() < need - ctx->n_alloc)
    return fail(ctx, SV_E_NOMEM, "KV page pool exhausted (%d free, %d needed)",
                (int)ctx->free_pages.size(), need - ctx->n_alloc);
  const int first = ctx->n_alloc;
  for (int lp = first; lp < need; ++lp) {
    ctx->pin_bt[lp] = ctx->free_pages.back();
    ctx->free_pages.pop_back();
  }
  ctx->n_alloc = need;
  CK(cudaMemcpyAsync(ctx->block_table + first, ctx->pin_bt + first, (need - first) * sizeof(int),
                     cudaMemcpyHostToDevice, ctx->stream));
  if (ctx->bt_shadow)
    CK(cudaMemcpyAsync(ctx->bt_shadow + first, ctx->pin_bt + first, (need - first) * sizeof(int),
                       cudaMemcpyHostToDevice, ctx->stream));
  return SV_OK;
}

// Return pages wholly beyond `len` to the pool (their table entries stay
// stale on the device; cap_len keeps kernels away from them).
void release_pages(sv_ctx* ctx, int len) {
  const int keep = pages_for(len);
  for (int lp = ctx->n_alloc - 1; lp >= keep; --lp) {
    ctx->free_pages.push_back(ctx->pin_bt[lp]);
    ctx->pin_bt[lp] = -1;
  }
  if (keep < ctx->n_alloc) ctx->n_alloc = keep;
}

// The library's stream after the caller's work so far, and the caller's
// stream after the library's work (nothing to do when they are one stream).
int join_user_stream(sv_ctx* ctx) {
  if (ctx->stream == ctx->user_stream) return SV_OK;
  CK(cudaEventRecord(ctx->ev, ctx->user_stream));
  CK(cudaStreamWaitEvent(ctx->stream, ctx->ev, 0));
  return SV_OK;
}
int join_library_stream(sv_ctx* ctx) {
  if (ctx->stream == ctx->user_stream) return SV_OK;
  CK(cudaEventRecord(ctx->ev, ctx->stream));
  CK(cudaStreamWaitEvent(ctx->user_stream, ctx->ev, 0));
  return SV_OK;
}

int begin_call(sv_ctx* ctx) {
  if (ctx->async_pending) return fail(ctx, SV_E_STATE, "asynchronous calls pending: call sv_sync first");
  return join_user_stream(ctx);
}

int end_call(sv_ctx* ctx) { return join_library_stream(ctx); }

// Stage [cap_len, tokens[0..n)] at slot `at` of the pinned input buffer and
// copy it into the device state.
int upload_tokens(sv_ctx* ctx, const int32_t* tokens, int n, int at) {
  if (at < 0 || (size_t)at + n + 1 > ctx->pin_in_len)
    return fail(ctx, SV_E_INVAL, "token staging of %d at %d exceeds %zu", n, at, ctx->pin_in_len);
  int32_t* src = ctx->pin_in + at;
  src[0] = ctx->n_alloc * kPage;
  memcpy(src + 1, tokens, n * sizeof(int32_t));
  CK(cudaMemcpyAsync(&ctx->st->cap_len, src, (n + 1) * sizeof(int32_t), cudaMemcpyHostToDevice,
                     ctx->stream));
  ctx->dev_cap = src[0];
  return SV_OK;
}

// A synchronous verify step's input without a copy of the tokens: they go
// into the pinned staging that the embedding kernel reads (StepIo); cap_len
// is copied only when it changed.  The previous call has finished with the
// staging (every synchronous call ends with a stream synchronisation).
int stage_tokens_mapped(sv_ctx* ctx, const int32_t* tokens, int n) {
  int32_t* src = ctx->pin_in;
  memcpy(src + 1, tokens, n * sizeof(int32_t));
  const int cap = ctx->n_alloc * kPage;
  if (cap != ctx->dev_cap) {
    src[0] = cap;
    CK(cudaMemcpyAsync(&ctx->st->cap_len, src, sizeof(int32_t), cudaMemcpyHostToDevice, ctx->stream));
    ctx->dev_cap = cap;
  }
  return SV_OK;
}

int check_tokens(sv_ctx* ctx, const int32_t* t, int n) {
  if (!t) return fail(ctx, SV_E_INVAL, "token array is null");
  for (int i = 0; i < n; ++i)
    if (t[i] < 0 || t[i] >= ctx->cfg.vocab)
      return fail(ctx, SV_E_INVAL, "token %d out of range [0, %d)", t[i], ctx->cfg.vocab);
  return SV_OK;
}

// mapped: the accept kernel wrote the result into the pinned read-back itself.
int finish_sync_step(sv_ctx* ctx, int32_t* result, bool mapped = false) {
  if (!mapped)
    CK(cudaMemcpyAsync(ctx->pin_out->result, ctx->st->result, 4 * sizeof(int32_t), cudaMemcpyDeviceToHost,
                       ctx->stream));
  CK(cudaStreamSynchronize(ctx->stream));
  memcpy(result, ctx->pin_out->result, 4 * sizeof(int32_t));
  if (result[3] & ~ST_BAD_STATE)
    return fail(ctx, SV_E_CUDA, "a kernel reported status 0x%x (1 timeout, 2 bad page, 4 bad token)",
                result[3]);
  ctx->seq_len = result[2];
  release_pages(ctx, ctx->seq_len);
  if (result[3] & ST_BAD_STATE) {  // the host check below makes this unreachable; kept as a backstop
    CK(cudaMemsetAsync(&ctx->st->state_err, 0, sizeof(int32_t), ctx->stream));
    CK(cudaStreamSynchronize(ctx->stream));
    return fail(ctx, SV_E_STATE, "tokens[0] is not the pending greedy token; nothing was committed");
  }
  ctx->pending = result[1];
  return SV_OK;
}

int validate(const sv_config* c) {
  if (!c) return 0;
  if (c->n_layers < 0 || c->hidden <= 0 || c->hidden % 128) return 0;
  if (c->head_dim != 64 && c->head_dim != 128 && c->head_dim != 256) return 0;
  if (c->n_q_heads <= 0 || c->n_kv_heads <= 0 || c->n_q_heads % c->n_kv_heads) return 0;
  if (16 % (c->n_q_heads / c->n_kv_heads)) return 0;
  if (((c->n_q_heads + 2 * c->n_kv_heads) * c->head_dim) % 128) return 0;
  if ((c->n_q_heads * c->head_dim) % 64) return 0;
  if (c->ffn <= 0 || c->ffn % 64) return 0;
  if (c->vocab <= 0) return 0;
  if (c->qk_norm && c->head_dim > 128) return 0;
  if (c->act != 0 && c->act != 1) return 0;
  if (c->page_size != kPage || c->max_k < 1 || c->max_k > kMaxK) return 0;
  if (c->max_seq < c->max_k || c->max_seq > kMaxSeq || c->max_pages < 1) return 0;
  if (c->kv_delayed != 0 && c->kv_delayed != 1) return 0;
  return 1;
}

}  // namespace

// ====================================================================== API
extern "C" {

int sv_create(const sv_config* cfg, const sv_weights* w, void* cuda_stream, sv_ctx** out) {
  if (!out) return SV_E_INVAL;
  *out = nullptr;
  if (!validate(cfg) || !w) return SV_E_INVAL;
  sv_ctx* ctx = new sv_ctx();
  ctx->cfg = *cfg;
  const sv_config& c = ctx->cfg;
  int rc = SV_OK;
  auto bail = [&](int code) {
    sv_destroy(ctx);
    return code;
  };
  if (cudaGetDevice(&ctx->device) != cudaSuccess) return bail(SV_E_CUDA);
  cudaDeviceGetAttribute(&ctx->num_sms, cudaDevAttrMultiProcessorCount, ctx->device);
  if (ctx->num_sms <= 0) ctx->num_sms = 1;
  ctx->user_stream = static_cast<cudaStream_t>(cuda_stream);
  // A stream of the caller's is the library's too: no event join at every
  // call (about 6 us a step on the 8B shape).  The default streams (legacy,
  // per-thread) take no capture or programmatic dependent launch, so their
  // callers get a stream of the library's, joined to theirs at each call.
  const bool user_default = ctx->user_stream == nullptr || ctx->user_stream == cudaStreamLegacy ||
                            ctx->user_stream == cudaStreamPerThread;
  if (!user_default)
    ctx->stream = ctx->user_stream;
  else if (cudaStreamCreateWithFlags(&ctx->stream, cudaStreamNonBlocking) != cudaSuccess)
    return bail(SV_E_CUDA);
  if (cudaEventCreateWithFlags(&ctx->ev, cudaEventDisableTiming) != cudaSuccess) return bail(SV_E_CUDA);
  const char* ng = getenv("SV_NO_GRAPHS");
  ctx->use_graphs = !(ng && ng[0] == '1');
  const char* np = getenv("SV_NO_PDL");
  ctx->use_pdl = !(np && np[0] == '1');
  // Off by default: on the 8B-shaped verify step it measured 2 % slower (the
  // prefetches compete with the slowest CTAs of the current launch).
  const char* pf = getenv("SV_L2_PREFETCH");
  ctx->prefetch_mode = pf ? atoi(pf) : 0;
  const char* nt = getenv("SV_NO_TC");
  ctx->use_tc = !(nt && nt[0] == '1');
  const char* nl = getenv("SV_NO_TILED");
  ctx->use_tiled = !(nl && nl[0] == '1');
  const char* wh = getenv("SV_TEST_WITHHOLD_PARTIAL");
  ctx->withhold_cta1 = wh ? atoi(wh) + 1 : 0;
  if (prepare_linear_kernels() != cudaSuccess || prepare_linear_tc_kernels() != cudaSuccess ||
      prepare_attention_kernels() != cudaSuccess)
    return bail(SV_E_CUDA);
  // the weights are read below (the tiled copies) on the library's stream:
  // let every stream's earlier work, which may still be writing them, finish
  if (cudaDeviceSynchronize() != cudaSuccess) return bail(SV_E_CUDA);

  const int L = c.n_layers, H = c.hidden, d = c.head_dim, Hq = c.n_q_heads, Hkv = c.n_kv_heads;
  ctx->embed = static_cast<const bf16*>(w->embed);
  ctx->lm_head = static_cast<const bf16*>(w->lm_head ? w->lm_head : w->embed);
  ctx->final_norm = static_cast<const bf16*>(w->final_norm);
  if (!ctx->embed || !ctx->final_norm || !aligned16(ctx->final_norm)) return bail(SV_E_INVAL);
  if (L > 0 && (!w->attn_norm || !w->wqkv || !w->wo || !w->ffn_norm || !w->w_gate_up || !w->w_down ||
                (c.qk_norm && (!w->q_norm || !w->k_norm))))
    return bail(SV_E_INVAL);
  ctx->lin_qkv.resize(L);
  ctx->lin_o.resize(L);
  ctx->lin_gu.resize(L);
  ctx->lin_down.resize(L);
  const int qkv_rows = (Hq + 2 * Hkv) * d;
  for (int l = 0; l < L; ++l) {
    ctx->attn_norm.push_back(static_cast<const bf16*>(w->attn_norm[l]));
    ctx->ffn_norm.push_back(static_cast<const bf16*>(w->ffn_norm[l]));
    ctx->q_norm.push_back(c.qk_norm ? static_cast<const bf16*>(w->q_norm[l]) : nullptr);
    ctx->k_norm.push_back(c.qk_norm ? static_cast<const bf16*>(w->k_norm[l]) : nullptr);
    if (!aligned16(w->attn_norm[l]) || !aligned16(w->ffn_norm[l]) || !w->attn_norm[l] || !w->ffn_norm[l])
      return bail(SV_E_INVAL);
    if ((rc = make_linear(ctx, &ctx->lin_qkv[l], w->wqkv[l], qkv_rows, H, qkv_rows / 128,
                          d == 256 ? MAP_HEAD256 : MAP_PLAIN)))
      return bail(rc);
    if ((rc = make_linear(ctx, &ctx->lin_o[l], w->wo[l], H, Hq * d, H / 128, MAP_PLAIN))) return bail(rc);
    if ((rc = make_linear(ctx, &ctx->lin_gu[l], w->w_gate_up[l], 2 * c.ffn, H, c.ffn / 64, MAP_GATE_UP)))
      return bail(rc);
    if ((rc = make_linear(ctx, &ctx->lin_down[l], w->w_down[l], H, c.ffn, H / 128, MAP_PLAIN)))
      return bail(rc);
  }
  if ((rc = make_linear(ctx, &ctx->lin_head, ctx->lm_head, c.vocab, H, (c.vocab + 127) / 128, MAP_PLAIN)))
    return bail(rc);

  // ---- device memory
  const int MP = mp_of(kMaxK);  // prefill blocks take kMaxK rows whatever max_k is
  ctx->bt_len = pages_for(c.max_seq);
  ctx->pool_pages = c.max_pages + (c.kv_delayed ? kWinPages : 0);
  ctx->layer_stride = (size_t)ctx->pool_pages * Hkv * kPage * d;
  // kernels address the pools' rows of head_dim elements with 32-bit indices
  if ((size_t)ctx->pool_pages * Hkv * kPage * (L > 0 ? L : 1) >= (size_t)INT32_MAX)
    return bail(SV_E_INVAL);
  const size_t pool = ctx->layer_stride * (L > 0 ? L : 1);
  ctx->max_splits = attn_n_splits(c.max_seq, d);
  size_t ws_words = 0;
  auto acc_ws = [&](const LinearDesc& ld) {
    if (ld.max_seg > 1) ws_words = std::max(ws_words, (size_t)ld.grid * kLinRows * MP);
  };
  for (int l = 0; l < L; ++l) {
    acc_ws(ctx->lin_qkv[l]);
    acc_ws(ctx->lin_o[l]);
    acc_ws(ctx->lin_gu[l]);
    acc_ws(ctx->lin_down[l]);
  }
  acc_ws(ctx->lin_head);
  // the tcgen05 form's slots hold kTcMaxRows token rows; activations hold a
  // prefill block of kTcMaxRows rows (a step takes at most kMaxK)
  const size_t ws_tc_words = ws_words / MP * kTcMaxRows;
  const int kRows = std::max(kMaxK, kTcMaxRows);
  if ((rc = dalloc(ctx, &ctx->kpool, pool)) || (rc = dalloc(ctx, &ctx->vpool, pool)) ||
      (rc = dalloc(ctx, &ctx->block_table, (size_t)ctx->bt_len)) || (rc = dalloc(ctx, &ctx->st, 1)) ||
      (rc = dalloc(ctx, &ctx->x, (size_t)kRows * H)) || (rc = dalloc(ctx, &ctx->xn, (size_t)kRows * H)) ||
      (rc = dalloc(ctx, &ctx->q, (size_t)kRows * Hq * d)) ||
      (rc = dalloc(ctx, &ctx->o, (size_t)kRows * Hq * d)) ||
      (rc = dalloc(ctx, &ctx->a, (size_t)kRows * c.ffn)) ||
      (rc = dalloc(ctx, &ctx->x_ss, (size_t)kRows * (H / 128))) ||
      (rc = dalloc(ctx, &ctx->rope, (size_t)c.max_seq * (d / 2))) ||
      (rc = dalloc(ctx, &ctx->part_ml, (size_t)kRows * Hq * ctx->max_splits)) ||
      (rc = dalloc(ctx, &ctx->part_o, (size_t)kRows * Hq * ctx->max_splits * d)) ||
      (rc = dalloc(ctx, &ctx->ws, ws_words)) || (rc = dalloc(ctx, &ctx->ws_tc, ws_tc_words)) ||
      (rc = dalloc(ctx, &ctx->am_val, (size_t)kMaxK * ctx->lin_head.n_tiles)) ||
      (rc = dalloc(ctx, &ctx->am_idx, (size_t)kMaxK * ctx->lin_head.n_tiles)))
    return bail(rc);
  if (c.kv_delayed && (rc = dalloc(ctx, &ctx->bt_shadow, (size_t)ctx->bt_len))) return bail(rc);
  if (cudaMemset(ctx->ws, 0xff, ws_words * sizeof(uint32_t)) != cudaSuccess ||
      cudaMemset(ctx->ws_tc, 0xff, ws_tc_words * sizeof(uint32_t)) != cudaSuccess)
    return bail(SV_E_CUDA);
  if (!make_bf16_map(&ctx->kmap, ctx->kpool, pool / d, d, kPage) ||
      !make_bf16_map(&ctx->vmap, ctx->vpool, pool / d, d, kPage) ||
      !make_bf16_map(&ctx->xmap_x, ctx->x, kRows, H, kMaxK) || !make_bf16_map(&ctx->xmap_o, ctx->o, kRows, Hq * d, kMaxK) ||
      !make_bf16_map(&ctx->xmap_a, ctx->a, kRows, c.ffn, kMaxK) ||
      !make_bf16_map(&ctx->xmap128_x, ctx->x, kRows, H, kTcMaxRows) ||
      !make_bf16_map(&ctx->xmap128_xn, ctx->xn, kRows, H, kTcMaxRows) ||
      !make_bf16_map(&ctx->xmap_xn, ctx->xn, kRows, H, kMaxK) ||
      !make_bf16_map(&ctx->xmap128_o, ctx->o, kRows, Hq * d, kTcMaxRows) ||
      !make_bf16_map(&ctx->xmap128_a, ctx->a, kRows, c.ffn, kTcMaxRows))
    return bail(SV_E_CUDA);
  // a prefill of max_seq tokens stages every block [cap_len, tokens] side by side
  ctx->pin_in_len = (size_t)c.max_seq + (c.max_seq + kMaxK - 1) / kMaxK + kMaxK + 8;
  if (cudaMallocHost(&ctx->pin_in, sizeof(int32_t) * ctx->pin_in_len) != cudaSuccess ||
      cudaMallocHost(&ctx->pin_out, sizeof(SvState)) != cudaSuccess ||
      cudaMallocHost(&ctx->pin_bt, sizeof(int) * (size_t)ctx->bt_len) != cudaSuccess)
    return bail(SV_E_NOMEM);
  // the device's addresses of the staging (unified addressing maps pinned
  // host memory); without them the synchronous verify copies instead
  {
    void *din = nullptr, *dout = nullptr;
    if (cudaHostGetDevicePointer(&din, ctx->pin_in, 0) == cudaSuccess &&
        cudaHostGetDevicePointer(&dout, ctx->pin_out, 0) == cudaSuccess) {
      ctx->pin_in_dev = static_cast<int32_t*>(din);
      ctx->pin_out_dev = static_cast<SvState*>(dout);
    }
    cudaGetLastError();
  }
  for (int i = 0; i < ctx->bt_len; ++i) ctx->pin_bt[i] = -1;
  if (cudaMemcpy(ctx->block_table, ctx->pin_bt, sizeof(int) * ctx->bt_len, cudaMemcpyHostToDevice) !=
          cudaSuccess ||
      (ctx->bt_shadow &&
       cudaMemcpy(ctx->bt_shadow, ctx->pin_bt, sizeof(int) * ctx->bt_len, cudaMemcpyHostToDevice) != cudaSuccess))
    return bail(SV_E_CUDA);
  for (int pg = c.max_pages - 1; pg >= 0; --pg) ctx->free_pages.push_back(pg);
  if (launch_rope_table(ctx->rope, c.max_seq, d, c.rope_theta, ctx->stream) != cudaSuccess ||
      launch_set_len(ctx->st, 0, 0, -1, ctx->stream) != cudaSuccess ||
      cudaStreamSynchronize(ctx->stream) != cudaSuccess)
    return bail(SV_E_CUDA);
  ctx->dev_cap = 0;
  *out = ctx;
  return SV_OK;
}

void sv_destroy(sv_ctx* ctx) {
  if (!ctx) return;
  if (ctx->stream) cudaStreamSynchronize(ctx->stream);
  destroy_graphs(ctx);
  for (void* p : ctx->allocs) cudaFree(p);
  if (ctx->pin_in) cudaFreeHost(ctx->pin_in);
  if (ctx->pin_out) cudaFreeHost(ctx->pin_out);
  if (ctx->pin_bt) cudaFreeHost(ctx->pin_bt);
  if (ctx->ev) cudaEventDestroy(ctx->ev);
  if (ctx->stream && ctx->stream != ctx->user_stream) cudaStreamDestroy(ctx->stream);
  delete ctx;
}

int sv_verify(sv_ctx* ctx, const int32_t* tokens_host, int K, float* logits_dev, int32_t* n_accepted,
              int32_t* correction_token) {
  if (!ctx) return SV_E_INVAL;
  if (K < 1 || K > ctx->cfg.max_k) return fail(ctx, SV_E_INVAL, "K=%d outside [1, %d]", K, ctx->cfg.max_k);
  int rc;
  if ((rc = check_tokens(ctx, tokens_host, K))) return rc;
  if (ctx->seq_len + K > ctx->cfg.max_seq)
    return fail(ctx, SV_E_INVAL, "length %d + %d exceeds max_seq", ctx->seq_len, K);
  if ((rc = begin_call(ctx))) return rc;
  if (ctx->pending >= 0 && tokens_host[0] != ctx->pending)
    return fail(ctx, SV_E_STATE, "tokens[0] = %d is not the pending greedy token %d", tokens_host[0],
                ctx->pending);
  if ((rc = ensure_pages(ctx, ctx->seq_len + K))) return rc;
  // the step reads its tokens from, and writes its result into, the pinned
  // staging itself where that is mapped and the step's graph takes buffers
  // (StepIo): no copy on either side of the step
  const bool mapped = ctx->pin_in_dev && step_takes_io(ctx, K, MODE_VERIFY, logits_dev);
  if (mapped) {
    if ((rc = stage_tokens_mapped(ctx, tokens_host, K))) return rc;
    rc = run_step(ctx, K, MODE_VERIFY, logits_dev, StepIo{ctx->pin_in_dev + 1, ctx->pin_out_dev->result});
  } else {
    if ((rc = upload_tokens(ctx, tokens_host, K, 0))) return rc;
    rc = run_step(ctx, K, MODE_VERIFY, logits_dev);
  }
  if (rc) return rc;
  int32_t res[4];
  if ((rc = finish_sync_step(ctx, res, mapped))) return rc;
  if (n_accepted) *n_accepted = res[0];
  if (correction_token) *correction_token = res[1];
  return end_call(ctx);
}

int sv_decode(sv_ctx* ctx, int32_t token, float* logits_dev, int32_t* next_token) {
  int32_t n = 0;
  return sv_verify(ctx, &token, 1, logits_dev, &n, next_token);
}

int sv_prefill_blocks(int n, int use_tc, int32_t* sizes, int max_blocks) {
  if (n < 1) return SV_E_INVAL;
  int count = 0;
  for (int done = 0; done < n; ++count) {
    const int M = prefill_block(n - done, use_tc != 0);
    if (sizes) {
      if (count >= max_blocks) return SV_E_INVAL;
      sizes[count] = M;
    }
    done += M;
  }
  return count;
}

int sv_prefill(sv_ctx* ctx, const int32_t* tokens_host, int n, float* last_logits_dev,
               int32_t* next_token) {
  if (!ctx) return SV_E_INVAL;
  if (n < 1) return fail(ctx, SV_E_INVAL, "prefill of %d tokens", n);
  int rc;
  if ((rc = check_tokens(ctx, tokens_host, n))) return rc;
  if (ctx->seq_len + n > ctx->cfg.max_seq)
    return fail(ctx, SV_E_INVAL, "length %d + %d exceeds max_seq", ctx->seq_len, n);
  if ((rc = begin_call(ctx))) return rc;
  if ((rc = ensure_pages(ctx, ctx->seq_len + n))) return rc;
  // Each block streams every weight once, and no row's arithmetic depends on
  // the block's size, so the blocks are as large as the kernels allow: the
  // last one (whose final row gives the next token) has the 1..kMaxK rows
  // left over, the others kMaxK rows each, or up to kTcMaxRows with the
  // tcgen05 linear.  Blocks of more than kMaxK rows are embedded here, kMaxK
  // rows at a time, before their step.
  const int H = ctx->cfg.hidden;
  int at = 0;
  for (int done = 0; done < n;) {
    const int M = prefill_block(n - done, ctx->use_tc);
    const bool last = done + M == n;
    if (M > kMaxK) {
      for (int r = 0; r < M; r += kMaxK) {
        const int mr = std::min(kMaxK, M - r);
        if ((rc = upload_tokens(ctx, tokens_host + done + r, mr, at))) return rc;
        at += mr + 1;
        CK(launch_embed(ctx->embed, H, ctx->cfg.vocab, mr, ctx->x + (size_t)r * H,
                        ctx->x_ss + (size_t)r * (H / 128), ctx->st, false, ctx->stream, false, StepIo{}));
      }
    } else {
      if ((rc = upload_tokens(ctx, tokens_host + done, M, at))) return rc;
      at += M + 1;
    }
    if ((rc = run_step(ctx, M, last ? MODE_PREFILL : MODE_BODY, last ? last_logits_dev : nullptr)))
      return rc;
    done += M;
  }
  int32_t res[4];
  if ((rc = finish_sync_step(ctx, res))) return rc;
  if (next_token) *next_token = res[1];
  return end_call(ctx);
}

int sv_verify_async(sv_ctx* ctx, const int32_t* tokens_dev, int K, float* logits_dev, int32_t* result_dev) {
  if (!ctx) return SV_E_INVAL;
  if (K < 1 || K > ctx->cfg.max_k) return fail(ctx, SV_E_INVAL, "K=%d outside [1, %d]", K, ctx->cfg.max_k);
  if (!tokens_dev || !result_dev) return fail(ctx, SV_E_INVAL, "null device pointer");
  for (const void* ptr : {static_cast<const void*>(tokens_dev), static_cast<const void*>(result_dev)}) {
    cudaPointerAttributes pa;
    if (cudaPointerGetAttributes(&pa, ptr) != cudaSuccess ||
        (pa.type != cudaMemoryTypeDevice && pa.type != cudaMemoryTypeManaged) || pa.device != ctx->device) {
      cudaGetLastError();
      return fail(ctx, SV_E_INVAL, "tokens_dev and result_dev must be memory of the context's device");
    }
  }
  int rc = join_user_stream(ctx);
  if (rc) return rc;
  ctx->async_pending = true;
  // The step's graph reads the tokens and writes the result in the caller's
  // buffers itself (its embedding and accept nodes re-pointed), saving a copy
  // on each side of it; otherwise the state block takes them by copies.
  if (step_takes_io(ctx, K, MODE_VERIFY, logits_dev)) {
    if ((rc = run_step(ctx, K, MODE_VERIFY, logits_dev, StepIo{tokens_dev, result_dev}))) return rc;
    return join_library_stream(ctx);
  }
  CK(cudaMemcpyAsync(ctx->st->tokens, tokens_dev, K * sizeof(int32_t), cudaMemcpyDeviceToDevice, ctx->stream));
  rc = run_step(ctx, K, MODE_VERIFY, logits_dev);
  if (rc) return rc;
  CK(cudaMemcpyAsync(result_dev, ctx->st->result, 4 * sizeof(int32_t), cudaMemcpyDeviceToDevice, ctx->stream));
  return join_library_stream(ctx);
}

int sv_reserve(sv_ctx* ctx, int len) {
  if (!ctx) return SV_E_INVAL;
  if (len < 0 || len > ctx->cfg.max_seq) return fail(ctx, SV_E_INVAL, "reserve %d outside [0, max_seq]", len);
  int rc;
  if ((rc = begin_call(ctx))) return rc;
  if ((rc = ensure_pages(ctx, len))) return rc;
  CK(launch_set_len(ctx->st, ctx->seq_len, ctx->n_alloc * kPage, kKeepPending, ctx->stream));
  ctx->dev_cap = ctx->n_alloc * kPage;
  CK(cudaStreamSynchronize(ctx->stream));
  return end_call(ctx);
}

int sv_sync(sv_ctx* ctx) {
  if (!ctx) return SV_E_INVAL;
  CK(cudaStreamSynchronize(ctx->stream));
  CK(cudaMemcpy(ctx->pin_out, ctx->st, sizeof(SvState), cudaMemcpyDeviceToHost));
  ctx->async_pending = false;
  ctx->seq_len = ctx->pin_out->seq_len;
  ctx->pending = ctx->pin_out->pending;
  if (ctx->pin_out->status != 0)
    return fail(ctx, SV_E_CUDA, "a kernel reported status 0x%x (1 timeout, 2 bad page, 4 bad token)",
                ctx->pin_out->status);
  if (ctx->pin_out->state_err != 0) {
    CK(cudaMemsetAsync(&ctx->st->state_err, 0, sizeof(int32_t), ctx->stream));
    CK(cudaStreamSynchronize(ctx->stream));
    return fail(ctx, SV_E_STATE,
                "an asynchronous verify step had tokens[0] != the pending greedy token; that step "
                "committed nothing");
  }
  return SV_OK;
}

int sv_truncate(sv_ctx* ctx, int new_len) {
  if (!ctx) return SV_E_INVAL;
  if (new_len < 0 || new_len > ctx->seq_len)
    return fail(ctx, SV_E_INVAL, "truncate to %d outside [0, %d]", new_len, ctx->seq_len);
  int rc;
  if ((rc = begin_call(ctx))) return rc;
  const sv_config& c = ctx->cfg;
  CK(launch_kv_zero(ctx->kpool, ctx->vpool, ctx->layer_stride, ctx->block_table, c.n_layers,
                    c.n_kv_heads, c.head_dim, new_len, ctx->seq_len, ctx->stream));
  // a shorter sequence has no known greedy token until the next commit
  const int pending = new_len == ctx->seq_len ? kKeepPending : -1;
  if (pending == -1) ctx->pending = -1;
  ctx->seq_len = new_len;
  release_pages(ctx, new_len);
  CK(launch_set_len(ctx->st, new_len, ctx->n_alloc * kPage, pending, ctx->stream));
  ctx->dev_cap = ctx->n_alloc * kPage;
  CK(cudaStreamSynchronize(ctx->stream));
  return end_call(ctx);
}

int sv_seq_len(const sv_ctx* ctx) { return ctx ? ctx->seq_len : SV_E_INVAL; }

int sv_kv_read(sv_ctx* ctx, int layer, int first, int count, void* k_dst_dev, void* v_dst_dev) {
  if (!ctx) return SV_E_INVAL;
  const sv_config& c = ctx->cfg;
  int rc;
  if ((rc = begin_call(ctx))) return rc;
  if (layer < 0 || layer >= c.n_layers || first < 0 || count < 0 ||
      first + count > ctx->n_alloc * kPage || !k_dst_dev || !v_dst_dev)
    return fail(ctx, SV_E_INVAL, "kv_read(layer %d, %d, %d) outside the allocated pages (%d positions)",
                layer, first, count, ctx->n_alloc * kPage);
  CK(launch_kv_gather(ctx->kpool, ctx->vpool, ctx->layer_stride, ctx->block_table, layer, c.n_kv_heads,
                      c.head_dim, first, count, static_cast<bf16*>(k_dst_dev), static_cast<bf16*>(v_dst_dev),
                      ctx->stream));
  CK(cudaStreamSynchronize(ctx->stream));
  return end_call(ctx);
}

int sv_trace_hidden(sv_ctx* ctx, void* hidden_dev, int max_rows) {
  if (!ctx) return SV_E_INVAL;
  if (hidden_dev && (max_rows < 1 || max_rows > kMaxK))
    return fail(ctx, SV_E_INVAL, "trace of %d rows outside [1, %d]", max_rows, kMaxK);
  ctx->trace = static_cast<bf16*>(hidden_dev);
  ctx->trace_rows = hidden_dev ? max_rows : 0;
  return SV_OK;
}

int sv_shuffle_pages(sv_ctx* ctx, uint64_t seed) {
  if (!ctx) return SV_E_INVAL;
  uint64_t z = seed;
  auto next = [&z]() {  // splitmix64 step
    z += 0x9E3779B97F4A7C15ull;
    uint64_t r = z;
    r = (r ^ (r >> 30)) * 0xBF58476D1CE4E5B9ull;
    r = (r ^ (r >> 27)) * 0x94D049BB133111EBull;
    return r ^ (r >> 31);
  };
  auto& f = ctx->free_pages;
  for (size_t i = f.size(); i > 1; --i) std::swap(f[i - 1], f[next() % i]);
  return SV_OK;
}

int sv_spec_generate(sv_ctx* target, sv_ctx* draft, int32_t pending, int K, int n_new,
                     int32_t* out_tokens, int32_t* n_out, int32_t* next_pending, int32_t* stats) {
  if (!target || !draft || target == draft) return SV_E_INVAL;
  const sv_config& tc = target->cfg;
  if (n_new < 1 || !out_tokens || !n_out || !next_pending || K < 1 || K > tc.max_k)
    return fail(target, SV_E_INVAL, "sv_spec_generate(K=%d, n_new=%d)", K, n_new);
  if (pending < 0 || pending >= tc.vocab)
    return fail(target, SV_E_INVAL, "pending token %d out of range [0, %d)", pending, tc.vocab);
  if (draft->cfg.vocab != tc.vocab)
    return fail(target, SV_E_INVAL, "drafter vocabulary %d differs from the target's %d", draft->cfg.vocab,
                tc.vocab);
  if (target->async_pending || draft->async_pending || target->seq_len != draft->seq_len)
    return fail(target, SV_E_STATE, "sv_spec_generate needs two synchronised contexts of equal length");
  const long long need = (long long)target->seq_len + n_new + K;
  if (need > tc.max_seq || need > draft->cfg.max_seq)
    return fail(target, SV_E_INVAL, "length + n_new + K = %lld exceeds max_seq", need);
  // a drafter call that fails reports through the target's error message
  auto drafter = [&](int code) { return fail(target, code, "drafter: %s", draft->err.c_str()); };
  int rc;
  int32_t ignored = 0;
  std::vector<int32_t> block(K);
  int produced = 0, steps = 0, accepted = 0, proposed = 0;
  while (produced < n_new) {
    const int base = target->seq_len;  // == draft->seq_len
    block[0] = pending;
    // the drafter commits block[j - 1] and proposes block[j]: block[0] is the
    // target's token, not the drafter's own greedy one, so it goes in as a
    // one-token prefill; the later ones are the drafter's pending tokens
    for (int j = 1; j < K; ++j) {
      rc = j == 1 ? sv_prefill(draft, &block[0], 1, nullptr, &block[1])
                  : sv_decode(draft, block[j - 1], nullptr, &block[j]);
      if (rc != SV_OK) return drafter(rc);
    }
    int32_t n = 0, corr = 0;
    if ((rc = sv_verify(target, block.data(), K, nullptr, &n, &corr)) != SV_OK) return rc;
    ++steps;
    accepted += n;
    proposed += K - 1;
    for (int j = 0; j <= n; ++j) out_tokens[produced++] = block[j];
    // the drafter holds block[0 .. K-2]; the target committed block[0 .. n]
    if (n + 1 < K - 1) {
      if ((rc = sv_truncate(draft, base + n + 1)) != SV_OK) return drafter(rc);
    } else if (n + 1 == K) {
      if ((rc = sv_prefill(draft, &block[K - 1], 1, nullptr, &ignored)) != SV_OK) return drafter(rc);
    }
    pending = corr;
  }
  *n_out = produced;
  *next_pending = pending;
  if (stats) {
    stats[0] = steps;
    stats[1] = accepted;
    stats[2] = proposed;
  }
  return SV_OK;
}

int sv_step_kernel_count(const sv_ctx* ctx, int K, int with_head) {
  if (!ctx || K < 1) return SV_E_INVAL;
  // steps of more than 8 rows normalise the input rows once per linear
  // (enqueue_step's prenorm): before QKV and gate|up, and before the LM head
  const bool prenorm = K > 8 && ctx->use_tc;
  const int embeds = (K + kMaxK - 1) / kMaxK;  // larger blocks are embedded kMaxK rows a launch
  const int per_layer = 6 + (prenorm ? 2 : 0);
  const int tail = with_head ? 2 + (prenorm ? 1 : 0) : 1;  // [norm,] LM head, accept; or accept
  const int window = with_head && step_delayed(ctx, K, MODE_VERIFY) ? 1 : 0;
  return embeds + per_layer * ctx->cfg.n_layers + tail + window;
}

int sv_time_linear(sv_ctx* ctx, int which, int K, int reps, float* avg_us, double* bytes_per_launch) {
  if (!ctx) return SV_E_INVAL;
  const sv_config& c = ctx->cfg;
  if (which < SV_LIN_O || which > SV_LIN_LM_HEAD || K < 1 || K > c.max_k || reps < 1 || !avg_us)
    return fail(ctx, SV_E_INVAL, "sv_time_linear(which=%d, K=%d, reps=%d)", which, K, reps);
  if (which != SV_LIN_LM_HEAD && c.n_layers < 1) return fail(ctx, SV_E_INVAL, "model has no layers");
  int rc;
  if ((rc = begin_call(ctx))) return rc;
  const int H = c.hidden;
  LinParams base = {};
  base.ss_tiles = H / 128;
  base.eps = c.rms_eps;
  base.M = K;
  base.ffn = c.ffn;
  base.head_dim = c.head_dim;
  base.ws = ctx->ws;
  base.n_q_heads = c.n_q_heads;
  base.n_kv_heads = c.n_kv_heads;
  base.act = c.act;
  base.vocab = c.vocab;
  base.st = ctx->st;
  base.x_ss = ctx->x_ss;
  base.am_val = ctx->am_val;
  base.am_idx = ctx->am_idx;
  // one launch per layer (distinct weights, so nothing is served from L2),
  // chained with programmatic dependent launch as inside a step
  const int per = (which == SV_LIN_LM_HEAD) ? 1 : c.n_layers;
  cudaEvent_t e0, e1;
  CK(cudaEventCreate(&e0));
  CK(cudaEventCreate(&e1));
  double bytes = 0.0;
  for (int r = -1; r < reps; ++r) {  // r = -1: untimed warm-up pass
    if (r == 0) CK(cudaEventRecord(e0, ctx->stream));
    for (int l = 0; l < per; ++l) {
      LinParams p = base;
      const LinearDesc* ld;
      int epi;
      bool norm;
      if (which == SV_LIN_O) {
        ld = &ctx->lin_o[l]; epi = EPI_RESID; norm = false; p.X = ctx->o; p.out = ctx->x; p.out_stride = H;
        p.out_ss = ctx->x_ss;
      } else if (which == SV_LIN_GATE_UP) {
        ld = &ctx->lin_gu[l]; epi = EPI_GLU; norm = true; p.X = ctx->x; p.gain = ctx->ffn_norm[l];
        p.out = ctx->a; p.out_stride = c.ffn;
      } else if (which == SV_LIN_DOWN) {
        ld = &ctx->lin_down[l]; epi = EPI_RESID; norm = false; p.X = ctx->a; p.out = ctx->x; p.out_stride = H;
        p.out_ss = ctx->x_ss;
      } else {
        ld = &ctx->lin_head; epi = EPI_LOGITS; norm = true; p.X = ctx->x; p.gain = ctx->final_norm;
      }
      p.Kd = ld->Kd; p.n_tiles = ld->n_tiles; p.max_seg = ld->max_seg; p.map = ld->map_kind;
      p.grid = ld->grid; p.wt = ld->tiled;
      // the same class of the next layer is prefetched, as much as inside a step
      const LinearDesc* next = nullptr;
      if (ctx->prefetch_mode == 1 && which != SV_LIN_LM_HEAD) {
        const int ln = (l + 1) % c.n_layers;
        next = which == SV_LIN_O ? &ctx->lin_o[ln]
                                 : (which == SV_LIN_GATE_UP ? &ctx->lin_gu[ln] : &ctx->lin_down[ln]);
      }
      CK(run_linear(ctx, *ld, p, epi, norm, ctx->stream, !(r == 0 && l == 0), next));
      if (r == 0) {
        const double n_out = which == SV_LIN_GATE_UP ? (double)c.ffn : (double)ld->N;
        bytes += 2.0 * ld->N * ld->Kd + 2.0 * K * ld->Kd + 2.0 * K * n_out;
      }
    }
  }
  CK(cudaEventRecord(e1, ctx->stream));
  CK(cudaEventSynchronize(e1));
  float ms = 0.0f;
  CK(cudaEventElapsedTime(&ms, e0, e1));
  cudaEventDestroy(e0);
  cudaEventDestroy(e1);
  *avg_us = 1000.0f * ms / (float)(reps * per);
  if (bytes_per_launch) *bytes_per_launch = bytes / per;
  return end_call(ctx);
}

const char* sv_last_error(const sv_ctx* ctx) { return ctx ? ctx->err.c_str() : "null context"; }

}  // extern "C"
