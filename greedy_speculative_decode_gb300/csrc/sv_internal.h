// sv_internal.h -- shared declarations of the sv library's kernels and host code.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/sv.h"

namespace sv {

typedef __nv_bfloat16 bf16;

constexpr int kPage = SV_PAGE_SIZE;
constexpr int kMaxK = SV_MAX_K;

// Linear kernel geometry: a tile is 128 output rows (two 64-row chunks that
// TMA loads as separate 64x64 boxes), streamed in 64-column k blocks.
constexpr int kLinRows = 128;
constexpr int kLinBK = 64;
constexpr int kLinChunkBytes = 64 * 128;           // one 64 x 64 bf16 box, 128B-swizzled
constexpr int kLinStageBytes = 2 * kLinChunkBytes;  // both chunks of one k block
constexpr int kLinStages = 8;
// Input columns a CTA stages at once, for 8 padded token rows (half as many
// for 16): 64 KB of shared memory.
constexpr int kLinXCols = 4096;
// Ring stages and staged input columns of the kernel for MT tiles of 8 token
// rows.  32 rows (MT = 4) give up half the ring for a 2048-column window:
// half as many restages of 4096-wide inputs, on steps the ring does not bound.
template <int MT>
struct LinGeom {
  static constexpr int kStages = MT == 4 ? kLinStages / 2 : kLinStages;
  static constexpr int kXCols = MT == 4 ? kLinXCols / 2 : kLinXCols / MT;
};
// Fewest k-blocks (16 KB of weight each) a CTA streams: small matrices use
// fewer CTAs rather than split tiles into many tiny partial sums.
constexpr int kLinMinShare = 4;
// Most CTAs one 128-row tile may be divided over (checked when a weight is set up).
constexpr int kLinMaxSeg = 16;
// k-blocks of the next linear each CTA prefetches into L2: 256 KB per CTA,
// about 39 MB over a full grid of a GB300, some 6 us of HBM time -- about the
// gap a launch boundary leaves.
constexpr int kLinPrefetchBlocks = 16;
constexpr int kLinConsumerWarps = 8;
constexpr int kLinThreads = (kLinConsumerWarps + 1) * 32;  // consumers, then the TMA producer

// Attention geometry.  Splits are fixed ranges of absolute positions: 128
// positions each below position 2048 (one page per warp for head_dim <= 128,
// whose CTAs have 8 warps; two for 256, 4 warps), then four pages per warp
// (512 positions, or 256 for head_dim 256).  Short contexts get many short
// dependent chains; long ones fewer work items, each merging more positions.
constexpr int kAttnSplitA = 128;                           // split size below kAttnRegionA
constexpr int kAttnRegionA = 2048;
constexpr int kAttnSplitsA = kAttnRegionA / kAttnSplitA;   // 16
constexpr int kAttnPagesB = 4;                             // pages per warp beyond kAttnRegionA
__host__ __device__ constexpr int attn_warps(int head_dim) { return head_dim <= 128 ? 8 : 4; }
__host__ __device__ constexpr int attn_split_b(int head_dim) { return kAttnPagesB * 16 * attn_warps(head_dim); }
// Splits that cover positions [0, ctx).
__host__ __device__ inline int attn_n_splits(int ctx, int head_dim) {
  if (ctx <= kAttnRegionA) return (ctx + kAttnSplitA - 1) / kAttnSplitA;
  const int sb = attn_split_b(head_dim);
  return kAttnSplitsA + (ctx - kAttnRegionA + sb - 1) / sb;
}
// First position of split s, and pages per warp in it.
__host__ __device__ inline int attn_split_start(int s, int head_dim) {
  return s < kAttnSplitsA ? s * kAttnSplitA : kAttnRegionA + (s - kAttnSplitsA) * attn_split_b(head_dim);
}
__host__ __device__ inline int attn_split_pages(int s, int head_dim) {
  return s < kAttnSplitsA ? kAttnSplitA / 16 / attn_warps(head_dim) : kAttnPagesB;
}
// Splits whose partials the light merge requests in one round: every row
// whose context lies in the short-split region.  Longer rows take the staged
// merge.
constexpr int kCombineChunk = kAttnSplitsA;
// Longest sequence a context may hold (the staged merge keeps the (m, l)
// pairs of every split in shared memory: at most 33 KB).
constexpr int kMaxSeq = 1 << 20;
constexpr int kAttnQ = 16;  // query rows (token rows x heads of one group) per work item

// Kinds of linear epilogue.
enum LinEpi : int { EPI_QKV = 0, EPI_RESID = 1, EPI_GLU = 2, EPI_LOGITS = 3 };
// How a tile index maps to its two 64-row chunks of the weight matrix.
enum LinMap : int { MAP_PLAIN = 0, MAP_GATE_UP = 1, MAP_HEAD256 = 2 };
// Step kinds.
enum StepMode : int { MODE_VERIFY = 0, MODE_PREFILL = 1, MODE_BODY = 2 };
// Status bits a kernel can raise.  The first three are sticky (st->status):
// the context is unusable after them.  ST_BAD_STATE is reported only in the
// result of the step it concerns: tokens[0] of a verify step was not the
// pending greedy token, so the step committed nothing.
enum Status : int { ST_TIMEOUT = 1, ST_BAD_PAGE = 2, ST_BAD_TOKEN = 4, ST_BAD_STATE = 8 };

// Device-resident state of the sequence and of the current step.
// cap_len and tokens are adjacent so the host sets both with one copy.
struct SvState {
  int32_t seq_len;   // committed length
  int32_t step_pos;  // length when the current step started
  int32_t status;    // Status bits raised so far (sticky)
  int32_t cap_len;   // positions < cap_len have pages
  int32_t tokens[kMaxK];
  int32_t result[4];  // n_accepted, correction, new_len, status
  int32_t argmax[kMaxK];
  int32_t pending;      // greedy token after the committed sequence (-1: not known)
  int32_t step_reject;  // this verify step's tokens[0] != pending (set by the embedding kernel)
  int32_t state_err;    // a step was rejected since the host last looked (cleared by sv_sync)
};

// Delayed K/V write-through (sv_config.kv_delayed): during a verify step the
// window's logical pages pos/16 .. pos/16 + kWinPages - 1 are mapped, in a
// shadow block table, to kWinPages scratch pages at the end of each layer's
// pool, which first receive a copy of the real pages; the step writes and
// reads the window there, and only the rows it accepts are copied into the
// real pages afterwards.  A window of up to 32 rows spans at most 3 pages.
constexpr int kWinPages = 3;
struct KvDelay {
  int* bt_shadow;  // null: write-then-truncate
  int win0;        // first scratch page of each layer
  int bt_len;      // entries of the block tables
};

struct LinParams {
  // the weight in the tiled layout (see LinearDesc::tiled), or null: the
  // producer then reads the row-major weight through the kernel's tensor map
  const uint8_t* wt;
  const uint8_t* pf_wt;  // the same for the weight of the L2 prefetch
  // input activations [M, Kd] bf16 and, for an RMSNorm prologue, the
  // per-128-column partial sums of squares of each row and the gain
  const bf16* X;
  const float* x_ss;  // [kMaxK, ss_tiles]
  const bf16* gain;   // [Kd]
  int ss_tiles;
  float eps;
  int M, Kd, n_tiles, max_seg, map, ffn, head_dim;
  int grid;      // CTAs the weight is divided over (one per SM, at most one per k-block)
  // split-tile partials, one slot per CTA: [grid][128][MP] fp32 words, all
  // 0xffffffff when idle; a CTA whose range starts inside a tile leaves its
  // partial of that tile in its slot, the tile's first CTA adds it and puts
  // the marker back
  uint32_t* ws;
  // epilogue operands
  bf16* out;           // EPI_QKV: q [M, Hq d]; EPI_RESID: x [M, N] (in place); EPI_GLU: a [M, ffn]
  int out_stride;
  float* out_ss;       // EPI_RESID: [kMaxK, n_tiles] partial sums of squares of the new rows
  bf16* kcache;        // EPI_QKV: this layer's K pages [pages, Hkv, 16, d]
  bf16* vcache;
  const int* block_table;
  const float2* rope;  // [max_seq, d/2] (cos, sin)
  const bf16* q_gain;  // [d] or null
  const bf16* k_gain;
  int n_q_heads, n_kv_heads, act;
  float* logits;       // EPI_LOGITS: rows m >= logits_row0 go to logits[m - logits_row0, :]
  int logits_row0;
  float* am_val;       // [kMaxK, n_tiles]
  int* am_idx;
  int vocab;
  SvState* st;
  // L2 prefetch: once the producer has issued its own stream, it prefetches
  // the first pf_blocks k-blocks that the CTA of the same index streams in the
  // next linear of the step (that weight's tensor map is the kernel's second
  // parameter), so the next launch starts from L2 instead of a cold HBM ramp.
  int pf_blocks, pf_n_tiles, pf_Kd, pf_grid, pf_map, pf_ffn;
  // Failure-detection test hook: CTA (withhold_cta1 - 1) never hands over its
  // split-tile partial, so the tile's reducer polls a tag that nothing sets
  // until its bounded wait gives up (0: off, the zero-initialised default).
  int withhold_cta1;
};

struct AttnParams {
  const bf16* q;  // [M, Hq d]
  const int* block_table;
  SvState* st;
  float2* part_ml;  // [kMaxK, Hq, max_splits] (running max in log2 units, sum)
  float* part_o;    // [kMaxK, Hq, max_splits, d]
  bf16* out;        // [M, Hq d]
  int M, n_q_heads, n_kv_heads, max_splits;
  int layer, max_pages;  // row coordinate of a page in the pool's tensor maps
  float scale_log2;      // log2(e) / sqrt(d)
};

// ------------------------------------------------------------------ launches
// A weight matrix as the linear kernel streams it: grid = one CTA per SM (at
// most one per k-block), max_seg = most CTAs any 128-row tile is split over.
// map: the row-major weight, 64 x 64 boxes.  tiled (or null): the same weight
// as n_tiles x (Kd/64) blocks of kLinStageBytes, tile-major, each block the
// exact shared-memory image of one k-block of one tile -- its two 64-row
// chunks, each 64 rows x 128 bytes with the 16-byte units of row r at
// positions u ^ (r mod 8) (the 128B swizzle the tensor map would apply) --
// so one contiguous bulk copy replaces two strided box loads.
struct LinearDesc {
  CUtensorMap map;
  int N, Kd, n_tiles, grid, max_seg, map_kind;
  uint8_t* tiled = nullptr;
};
// Bytes of the tiled layout of a weight.
inline size_t tiled_bytes(int n_tiles, int Kd) { return (size_t)n_tiles * (Kd / kLinBK) * kLinStageBytes; }
// Write the tiled layout of a row-major bf16 weight [N, Kd] (rows past N are zero).
cudaError_t launch_tile_weight(const bf16* w, int N, int Kd, int n_tiles, int map_kind, int ffn, uint8_t* out,
                               cudaStream_t s);
void linear_partition(int n_tiles, int Kd, int num_sms, int* grid, int* max_seg);

cudaError_t prepare_linear_kernels();
cudaError_t prepare_attention_kernels();
cudaError_t launch_linear(const LinearDesc& d, const LinParams& p, int epi, bool norm,
                          cudaStream_t s, bool pdl, const LinearDesc* next = nullptr);
size_t linear_smem_bytes(int mt);
// multi: some CTA of the grid runs more than one work item (long contexts)
cudaError_t launch_attention(const CUtensorMap& kmap, const CUtensorMap& vmap, const AttnParams& p,
                             int head_dim, int grid, bool multi, cudaStream_t s, bool pdl);
cudaError_t launch_attn_combine(const AttnParams& p, int head_dim, cudaStream_t s, bool pdl);
// Where a step takes its tokens and leaves its result besides the state
// block: the asynchronous verify call's device buffers of the caller, read by
// the embedding kernel (which copies them into st->tokens for the accept
// kernel) and written by the accept kernel.  Null: st->tokens, st->result only.
struct StepIo {
  const int32_t* tokens;  // [M]
  int32_t* result;        // [4]
};
// check: a verify step, whose tokens[0] must equal st->pending when that is known.
// pdl: launched as a programmatic dependent of the delayed write-through
// window copy (the kernel then ends only after the copy has).
cudaError_t launch_embed(const bf16* E, int hidden, int vocab, int M, bf16* x, float* x_ss,
                         SvState* st, bool check, cudaStream_t s, bool pdl, const StepIo& io);
cudaError_t launch_accept(SvState* st, const float* am_val, const int* am_idx, int n_tiles, int M,
                          int mode, bf16* kpool, bf16* vpool, size_t layer_stride,
                          const int* block_table, int n_layers, int n_kv_heads, int head_dim,
                          const KvDelay& dl, cudaStream_t s, bool pdl, const StepIo& io);
// A captured step graph's embedding and accept nodes: step_io_node tells
// whether `node` runs one of the two; set_step_io gives such a node, in the
// instantiated `exec`, the StepIo `io` (its other arguments as captured).
bool step_io_node(cudaGraphNode_t node);
cudaError_t set_step_io(cudaGraphExec_t exec, cudaGraphNode_t node, const StepIo& io);
// Delayed write-through, before a verify step of M rows: map the window's
// pages to the scratch pages in the shadow table and copy the real pages'
// contents there (zeros for pages not yet held).
cudaError_t launch_kv_window_in(bf16* kpool, bf16* vpool, size_t layer_stride, const int* block_table,
                                const KvDelay& dl, const SvState* st, int n_layers, int n_kv_heads,
                                int head_dim, int M, cudaStream_t s);
cudaError_t launch_rope_table(float2* tab, int max_seq, int head_dim, float theta, cudaStream_t s);
cudaError_t launch_kv_zero(bf16* kpool, bf16* vpool, size_t layer_stride, const int* block_table,
                           int n_layers, int n_kv_heads, int head_dim, int first, int last,
                           cudaStream_t s);
cudaError_t launch_kv_gather(const bf16* kpool, const bf16* vpool, size_t layer_stride,
                             const int* block_table, int layer, int n_kv_heads, int head_dim,
                             int first, int count, bf16* kdst, bf16* vdst, cudaStream_t s);
// pending: the new pending token, -1 for "not known", kKeepPending to leave it
constexpr int kKeepPending = -2;
cudaError_t launch_set_len(SvState* st, int len, int cap_len, int pending, cudaStream_t s);
// 2D bf16 tensor map [rows, cols] row-major, boxes of box_rows x 64 columns,
// 128B swizzle (the driver's encoder is looked up once per process).
bool make_bf16_map(CUtensorMap* m, const void* ptr, uint64_t rows, uint64_t cols, uint32_t box_rows);

}  // namespace sv
