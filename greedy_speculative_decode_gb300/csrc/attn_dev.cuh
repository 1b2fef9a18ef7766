// attn_dev.cuh -- multi-row paged decode attention with per-row context lengths.
//
// Row r of a step attends to positions [0, pos + r + 1) ("Phase 23:
// Speculative Verify Parity" section 2 step 2: one metadata row per draft
// token with context length pos+1 upward).  Work is split over absolute
// positions (attn_split_start: 128-position splits up to position 2048, then
// 4 pages per warp) and warp w of the CTA takes a fixed run of the split's
// 16-position pages.  Because these boundaries are
// absolute, the partial result a row gets from a split does not depend on how
// many other rows share the step, on the cache's history, or on its physical
// pages; positions a row may not see are masked to exact zeros.  Partials are
// merged in fixed order: pages within a warp (online softmax), warps within
// the CTA, then splits in a second kernel.  That is what keeps a verify row
// bit-identical to single-token decode here; the page notes that attention
// implementations which reorder scaling or softmax arithmetic by shape change
// rounded scores ("Shape and cache history in Gemma block verification",
// section "Source evidence and competing explanations").
//
// One work item is (split, kv head, block of 16/G token rows) so that the
// G query heads of a group times the rows make one 16-row mma tile.  K and V
// pages arrive by TMA (128B-swizzled 16 x 64 boxes) into a per-warp ring;
// Q K^T and P V run on bf16 mma.sync with fp32 accumulation.
#pragma once
#include "sv_internal.h"
#include "sv_ptx.cuh"

namespace sv {
namespace {

template <int D>
struct AttnCfg {
  // warps per CTA, each over up to kMaxPages consecutive 16-position pages of a split
  static constexpr int kWarps = attn_warps(D);
  static constexpr int kMaxPages = kAttnPagesB;
  static constexpr int kThreads = kWarps * 32;
  static constexpr int kBoxes = D / 64;                // 64-column boxes per page row
  static constexpr int kPageBytes = kPage * D * 2;     // one K (or V) page of one head
  static constexpr int kBufBytes = 2 * kPageBytes;     // K + V
  static constexpr int kBufs = 2;  // pages in flight per warp
  static constexpr int kQStride = D + 8;               // bf16 elements
  static constexpr int kRingBytes = kWarps * kBufs * kBufBytes;
  static constexpr int kQTileBytes = 16 * kQStride * 2;
  // warp-merge scratch: o rows of stride kOS floats (kOS = 8 mod 32 banks, so a
  // warp's float2 stores and float4 loads take the minimum two wavefronts),
  // then the (m, l) pairs, the per-(query, warp) scales and the query maxima
  static constexpr int kOS = D + 8;
  static constexpr int kScratchBytes = kWarps * 16 * kOS * 4 + kWarps * 16 * 8 + 16 * kWarps * 4 + 16 * 4;
};

// Shared memory of the attention work: per-warp page buffers, the warp-merge
// scratch, the Q tile(s) and the page barriers.  With kMulti (CTAs that run
// several work items) the scratch has its own region and there are two Q
// tiles, so that the next item's pages and Q can land while this item's warps
// merge; otherwise the scratch aliases the page buffers.
template <int D, bool kMulti>
struct AttnSmem {
  uint8_t* ring;
  bf16* Qs;
  uint64_t* bars;
  float* scratch;
  using C = AttnCfg<D>;
  static constexpr int kRegion =
      kMulti ? C::kRingBytes + C::kScratchBytes
             : (C::kRingBytes > C::kScratchBytes ? C::kRingBytes : C::kScratchBytes);
  static constexpr int kQ = (kMulti ? 2 : 1) * C::kQTileBytes;
  __device__ __forceinline__ void carve(uint8_t* base) {
    ring = base;
    scratch = reinterpret_cast<float*>(base + (kMulti ? C::kRingBytes : 0));
    Qs = reinterpret_cast<bf16*>(base + kRegion);
    bars = reinterpret_cast<uint64_t*>(base + kRegion + kQ);
  }
  // dynamic shared memory of a launch (with slack to align the base to 1 KB)
  static constexpr int kSmem = 1024 + kRegion + kQ + C::kWarps * C::kBufs * 8 + 64;
};

// Initialise the page barriers (one thread).
template <int D, bool kMulti>
__device__ __forceinline__ void attn_init_bars(const AttnSmem<D, kMulti>& sm) {
  for (int i = 0; i < AttnCfg<D>::kWarps * AttnCfg<D>::kBufs; ++i) mbar_init(&sm.bars[i], 1);
  fence_barrier_init();
}

// The item's warps' partials merged in warp order into the split partial
// (m, l, o) of each of its nrows * G queries, written to global memory.  Each
// (query, warp) scale exp2(m_w - m) is computed once, then every 8-column
// group of a query takes the same ordered sums.  Named barrier 2; the caller
// has synchronised the warps' use of `scratch` before.
template <int D>
__device__ __forceinline__ void attn_merge_warps(const AttnParams& p, float* scratch, int nrows, int G, int r0,
                                                 int h, int split, const float (&m_run)[2], const float (&l_run)[2],
                                                 const float (&o)[D / 8][4]) {
  using C = AttnCfg<D>;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, q4 = lane & 3;
  // scratch: o [warp][16][kOS], (m, l) [warp][16], scale [16][warp], max [16]
  float* so = scratch;
  float2* sml = reinterpret_cast<float2*>(scratch + C::kWarps * 16 * C::kOS);
  float* s_sc = reinterpret_cast<float*>(sml + C::kWarps * 16);
  float* s_mx = s_sc + 16 * C::kWarps;
  if (q4 == 0) {
    sml[warp * 16 + g] = make_float2(m_run[0], l_run[0]);
    sml[warp * 16 + g + 8] = make_float2(m_run[1], l_run[1]);
  }
  {
    float* r0p = so + (warp * 16 + g) * C::kOS + 2 * q4;
    float* r1p = r0p + 8 * C::kOS;
#pragma unroll
    for (int n = 0; n < D / 8; ++n) {
      *reinterpret_cast<float2*>(r0p + n * 8) = make_float2(o[n][0], o[n][1]);
      *reinterpret_cast<float2*>(r1p + n * 8) = make_float2(o[n][2], o[n][3]);
    }
  }
  named_sync(2, C::kThreads);
  const int nq = nrows * G;
  // the query's maximum over the warps, and each warp's scale against it
  // (-1: the warp saw none of the query's positions and is skipped)
  for (int e = tid; e < nq * C::kWarps; e += C::kThreads) {
    const int qi = e / C::kWarps, ww = e % C::kWarps;
    float mx = -INFINITY;
#pragma unroll
    for (int w2 = 0; w2 < C::kWarps; ++w2) mx = fmaxf(mx, sml[w2 * 16 + qi].x);
    const float mw = sml[ww * 16 + qi].x;
    s_sc[qi * C::kWarps + ww] = (mx == -INFINITY || mw == -INFINITY) ? -1.0f : exp2f(__fsub_rn(mw, mx));
    if (ww == 0) s_mx[qi] = mx;
  }
  named_sync(2, C::kThreads);
  // ordered sums over the warps, 8 columns per thread
  for (int e = tid; e < nq * (D / 8); e += C::kThreads) {
    const int qi = e / (D / 8), c0 = (e % (D / 8)) * 8;
    float L = 0.0f, acc[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) acc[c] = 0.0f;
#pragma unroll
    for (int ww = 0; ww < C::kWarps; ++ww) {
      const float sc = s_sc[qi * C::kWarps + ww];
      if (sc < 0.0f) continue;
      const float* src = so + (ww * 16 + qi) * C::kOS + c0;
      const float4 v0 = *reinterpret_cast<const float4*>(src);
      const float4 v1 = *reinterpret_cast<const float4*>(src + 4);
      const float vv[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
      if (c0 == 0) L = __fadd_rn(L, __fmul_rn(sml[ww * 16 + qi].y, sc));
#pragma unroll
      for (int c = 0; c < 8; ++c) acc[c] = __fadd_rn(acc[c], __fmul_rn(vv[c], sc));
    }
    const int r = r0 + qi / G, hq = h * G + qi % G;
    const size_t slot = ((size_t)r * p.n_q_heads + hq) * p.max_splits + split;
    if (c0 == 0) p.part_ml[slot] = make_float2(s_mx[qi], L);
    float* dst = p.part_o + slot * D + c0;
    *reinterpret_cast<float4*>(dst) = make_float4(acc[0], acc[1], acc[2], acc[3]);
    *reinterpret_cast<float4*>(dst + 4) = make_float4(acc[4], acc[5], acc[6], acc[7]);
  }
}

// Work items w = cta, cta + G_ctas, ... of this step's attention, run by
// the CTA's AttnCfg<D>::kWarps warps (named barrier 2), in the layout whose
// merge scratch aliases the page buffers (grids with a CTA for every item).  `phase` holds each buffer's
// parity.  `pos` is the committed length, final for the whole step: the
// pages of the first item that hold only positions < pos (written by earlier
// steps) are requested before the wait on the previous kernel; Q and the page
// with the step's own rows after it.  Each item writes its split partial (m,
// l, o), merged by the combine kernel.  Returns false if a page never arrived.
template <int D>
__device__ bool attn_items_single(const AttnParams& p, const CUtensorMap* kmap_p,
                                  const CUtensorMap* vmap_p, int cta, int G_ctas,
                                  const AttnSmem<D, false>& sm, uint32_t& phase, int pos) {
  using C = AttnCfg<D>;
  const CUtensorMap& kmap = *kmap_p;
  const CUtensorMap& vmap = *vmap_p;
  const int layer = p.layer, max_pages = p.max_pages;
  uint8_t* ring = sm.ring;
  bf16* Qs = sm.Qs;
  uint64_t* bars = sm.bars;
  float* scratch = sm.scratch;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, q4 = lane & 3;
  const int G = p.n_q_heads / p.n_kv_heads;
  const int RB = kAttnQ / G;  // token rows per work item
  const int M = p.M;
  const int n_rb = (M + RB - 1) / RB;
  const int n_splits = attn_n_splits(pos + M, D);
  const int work = n_splits * p.n_kv_heads * n_rb;
  uint64_t* my_bars = bars + warp * C::kBufs;
  uint8_t* my_ring = ring + warp * C::kBufs * C::kBufBytes;
  const uint64_t pol = policy_evict_first();
  bool all_ok = true;
  bool waited = false;
  if (cta >= work) {  // nothing to do: wait only so that the grid completes in order
    pdl_wait();
    return true;
  }

  for (int w = cta; w < work; w += G_ctas) {
    const int rb = w % n_rb;
    const int h = (w / n_rb) % p.n_kv_heads;
    const int split = w / (n_rb * p.n_kv_heads);
    const int r0 = rb * RB;
    const int nrows = min(RB, M - r0);
    const int ctx_max = pos + r0 + nrows;  // largest context of the block's rows

    // ---- this warp's pages of the split
    const int ppw = attn_split_pages(split, D);
    const int wpos0 = attn_split_start(split, D) + warp * (ppw * kPage);
    int npages = 0;
    while (npages < ppw && wpos0 + npages * kPage < ctx_max) ++npages;
    int page_id[C::kMaxPages];
    for (int j = 0; j < C::kMaxPages; ++j) {
      int pg = -1;
      if (j < npages) {
        const int lp = (wpos0 + j * kPage) / kPage;
        pg = p.block_table[lp];
        if (pg < 0 || pg >= max_pages) pg = -1;
      }
      page_id[j] = pg;
    }
    auto issue = [&](int j) {
      const int b = j % C::kBufs;
      uint8_t* kb = my_ring + b * C::kBufBytes;
      uint8_t* vb = kb + C::kPageBytes;
      mbar_arrive_expect_tx(&my_bars[b], C::kBufBytes);
      const int row0 = ((layer * max_pages + page_id[j]) * p.n_kv_heads + h) * kPage;
      for (int cb = 0; cb < C::kBoxes; ++cb) {
        tma_load_2d(kb + cb * 2048, &kmap, cb * 64, row0, &my_bars[b], pol);
        tma_load_2d(vb + cb * 2048, &vmap, cb * 64, row0, &my_bars[b], pol);
      }
    };
    bool bad = false;
    for (int j = 0; j < npages; ++j) bad |= page_id[j] < 0;
    if (bad) {
      if (lane == 0) atomicOr(&p.st->status, ST_BAD_PAGE);
      npages = 0;
    }
    // pages of positions < pos only: written by earlier steps, requested now
    int n_old = 0;
    while (n_old < npages && n_old < C::kBufs && wpos0 + (n_old + 1) * kPage <= pos) ++n_old;
    if (lane == 0)
      for (int j = 0; j < n_old; ++j) issue(j);
    if (!waited) {
      pdl_wait();  // Q and the K/V of the step's own rows come from the QKV kernel
      waited = true;
    }
    if (lane == 0) {
      asm volatile("fence.proxy.async.global;" ::: "memory");  // K/V written with plain stores
      for (int j = n_old; j < npages && j < C::kBufs; ++j) issue(j);
    }
    // ---- Q tile: query qi = (token row r0 + qi / G, head h G + qi % G)
    for (int v = tid; v < 16 * (D / 8); v += C::kThreads) {
      const int qi = v / (D / 8), c8 = v % (D / 8);
      uint4 val = make_uint4(0u, 0u, 0u, 0u);
      if (qi < nrows * G) {
        const int r = r0 + qi / G, hq = h * G + qi % G;
        val = __ldcg(reinterpret_cast<const uint4*>(p.q + (size_t)r * p.n_q_heads * D + hq * D + c8 * 8));
      }
      *reinterpret_cast<uint4*>(Qs + qi * C::kQStride + c8 * 8) = val;
    }
    named_sync(2, C::kThreads);

    // query rows held by this lane: g and g + 8
    const int ctx_lo = pos + r0 + g / G + 1;
    const int ctx_hi = pos + r0 + (g + 8) / G + 1;
    float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.0f, 0.0f};
    float o[D / 8][4];
#pragma unroll
    for (int n = 0; n < D / 8; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.0f;

    const uint32_t q_base = smem_u32(Qs) + (uint32_t)((((lane & 7) + ((lane >> 3) & 1) * 8) * C::kQStride +
                                                       (lane >> 4) * 8) * 2);
    bool ok = true;
    for (int j = 0; j < npages; ++j) {
      const int b = j % C::kBufs;
      if (!mbar_wait(&my_bars[b], (phase >> b) & 1u)) {
        ok = false;
        break;
      }
      phase ^= 1u << b;
      const uint32_t kb = smem_u32(my_ring + b * C::kBufBytes);
      const uint32_t vb = kb + C::kPageBytes;
      // S = Q K^T for 16 queries x 16 positions
      float s[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        uint32_t a[4];
        ldsm_x4(q_base + kk * 32, a[0], a[1], a[2], a[3]);
        const int pr = (lane & 7) + ((lane >> 4) & 1) * 8;
        const int ch = (kk & 3) * 2 + ((lane >> 3) & 1);
        uint32_t b0, b1, b2, b3;
        ldsm_x4(kb + (kk >> 2) * 2048 + pr * 128 + ((ch ^ (pr & 7)) << 4), b0, b1, b2, b3);
        mma_bf16(s[0], a, b0, b1);
        mma_bf16(s[1], a, b2, b3);
      }
      // mask (exact -inf beyond each row's context), scale to log2 units
      const int pbase = wpos0 + j * kPage;
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int pabs = pbase + nt * 8 + 2 * q4 + (e & 1);
          const int ctx = e < 2 ? ctx_lo : ctx_hi;
          s[nt][e] = pabs < ctx ? __fmul_rn(s[nt][e], p.scale_log2) : -INFINITY;
        }
      // online softmax on rows g (e = 0, 1) and g + 8 (e = 2, 3).  The weights
      // p stay fp32: the denominator sums them unrounded, and P V is taken as
      // P_hi V + P_lo V with P_hi = bf16(p) and P_lo = bf16(p - P_hi) (the
      // tensor cores take bf16), which carries p to about 2^-16 -- a bf16-only
      // P would shift every attention output by up to half a bf16 step.
      float alpha[2];
      uint32_t pa[4], pl[4];
#pragma unroll
      for (int rr = 0; rr < 2; ++rr) {
        float mx = fmaxf(fmaxf(s[0][2 * rr], s[0][2 * rr + 1]), fmaxf(s[1][2 * rr], s[1][2 * rr + 1]));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
        const float m_new = fmaxf(m_run[rr], mx);
        float pv[4];
        if (m_new == -INFINITY) {
          alpha[rr] = 1.0f;
          pv[0] = pv[1] = pv[2] = pv[3] = 0.0f;
        } else {
          alpha[rr] = exp2f(__fsub_rn(m_run[rr], m_new));
          pv[0] = exp2f(__fsub_rn(s[0][2 * rr], m_new));
          pv[1] = exp2f(__fsub_rn(s[0][2 * rr + 1], m_new));
          pv[2] = exp2f(__fsub_rn(s[1][2 * rr], m_new));
          pv[3] = exp2f(__fsub_rn(s[1][2 * rr + 1], m_new));
        }
        float sum = __fadd_rn(__fadd_rn(pv[0], pv[1]), __fadd_rn(pv[2], pv[3]));
        sum = __fadd_rn(sum, __shfl_xor_sync(0xffffffffu, sum, 1));
        sum = __fadd_rn(sum, __shfl_xor_sync(0xffffffffu, sum, 2));
        l_run[rr] = __fadd_rn(__fmul_rn(l_run[rr], alpha[rr]), sum);
        m_run[rr] = m_new;
        pa[rr] = pack_bf16x2(pv[0], pv[1]);      // positions 2q, 2q+1
        pa[2 + rr] = pack_bf16x2(pv[2], pv[3]);  // positions 8+2q, 9+2q
        pl[rr] = pack_bf16x2(__fsub_rn(pv[0], bf16r(pv[0])), __fsub_rn(pv[1], bf16r(pv[1])));
        pl[2 + rr] = pack_bf16x2(__fsub_rn(pv[2], bf16r(pv[2])), __fsub_rn(pv[3], bf16r(pv[3])));
      }
#pragma unroll
      for (int n = 0; n < D / 8; ++n) {
        o[n][0] = __fmul_rn(o[n][0], alpha[0]);
        o[n][1] = __fmul_rn(o[n][1], alpha[0]);
        o[n][2] = __fmul_rn(o[n][2], alpha[1]);
        o[n][3] = __fmul_rn(o[n][3], alpha[1]);
      }
      // O += P_hi V + P_lo V
      const uint32_t afr[4] = {pa[0], pa[1], pa[2], pa[3]};
      const uint32_t afl[4] = {pl[0], pl[1], pl[2], pl[3]};
#pragma unroll
      for (int dn = 0; dn < D / 16; ++dn) {
        const int pr = (lane & 7) + ((lane >> 3) & 1) * 8;
        const int ch = ((dn * 16) & 63) / 8 + (lane >> 4);
        uint32_t b0, b1, b2, b3;
        ldsm_x4_trans(vb + ((dn * 16) >> 6) * 2048 + pr * 128 + ((ch ^ (pr & 7)) << 4), b0, b1, b2, b3);
        mma_bf16(o[2 * dn], afr, b0, b1);
        mma_bf16(o[2 * dn + 1], afr, b2, b3);
        mma_bf16(o[2 * dn], afl, b0, b1);
        mma_bf16(o[2 * dn + 1], afl, b2, b3);
      }
      fence_proxy_async_smem();  // reads of buffer b precede its next TMA write
      __syncwarp();
      if (lane == 0 && j + C::kBufs < npages) issue(j + C::kBufs);
    }
    if (!ok) all_ok = false;
    named_sync(2, C::kThreads);  // every warp is done with its ring: reuse it as scratch

    attn_merge_warps<D>(p, scratch, nrows, G, r0, h, split, m_run, l_run, o);
    fence_proxy_async_smem();  // scratch (in the ring) is overwritten by TMA next item
    named_sync(2, C::kThreads);            // scratch (= ring) and Qs are rewritten by the next item
  }
  return all_ok;
}

// The same work for grids whose CTAs run several items (long contexts), in
// the layout with a separate merge scratch and two Q tiles: each warp hands a
// page buffer to the CTA's next item as soon as this item is done with it,
// and the next item's page ids and Q tile are fetched while this one runs, so
// the next item's loads overlap this item's merge.  Same arithmetic, in the
// same order, as attn_items_single.
template <int D>
__device__ bool attn_items_multi(const AttnParams& p, const CUtensorMap* kmap_p,
                                 const CUtensorMap* vmap_p, int cta, int G_ctas,
                                 const AttnSmem<D, true>& sm, uint32_t& phase, int pos) {
  using C = AttnCfg<D>;
  const CUtensorMap& kmap = *kmap_p;
  const CUtensorMap& vmap = *vmap_p;
  const int layer = p.layer, max_pages = p.max_pages;
  uint8_t* ring = sm.ring;
  uint64_t* bars = sm.bars;
  float* scratch = sm.scratch;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, q4 = lane & 3;
  const int G = p.n_q_heads / p.n_kv_heads;
  const int RB = kAttnQ / G;  // token rows per work item
  const int M = p.M;
  const int n_rb = (M + RB - 1) / RB;
  const int n_splits = attn_n_splits(pos + M, D);
  const int work = n_splits * p.n_kv_heads * n_rb;
  uint64_t* my_bars = bars + warp * C::kBufs;
  uint8_t* my_ring = ring + warp * C::kBufs * C::kBufBytes;
  const uint64_t pol = policy_evict_first();
  bool all_ok = true;
  if (cta >= work) {  // nothing to do: wait only so that the grid completes in order
    pdl_wait();
    return true;
  }

  // This warp's pages of work item w: positions wpos0 + 16 j, j < npages, of
  // kv head h; page_id[j] their physical pages (npages = 0 and ST_BAD_PAGE
  // on an invalid block-table entry).
  struct Pages {
    int h, wpos0, npages;
    int page_id[C::kMaxPages];
  };
  auto pages_of = [&](int w) {
    Pages pg;
    const int rb = w % n_rb;
    pg.h = (w / n_rb) % p.n_kv_heads;
    const int split = w / (n_rb * p.n_kv_heads);
    const int ctx_max = pos + min(rb * RB + RB, M);  // largest context of the block's rows
    const int ppw = attn_split_pages(split, D);
    pg.wpos0 = attn_split_start(split, D) + warp * (ppw * kPage);
    pg.npages = 0;
    while (pg.npages < ppw && pg.wpos0 + pg.npages * kPage < ctx_max) ++pg.npages;
    bool bad = false;
#pragma unroll
    for (int j = 0; j < C::kMaxPages; ++j) {
      int id = -1;
      if (j < pg.npages) {
        id = p.block_table[(pg.wpos0 + j * kPage) / kPage];
        if (id < 0 || id >= max_pages) {
          id = -1;
          bad = true;
        }
      }
      pg.page_id[j] = id;
    }
    if (bad) {
      if (lane == 0) atomicOr(&p.st->status, ST_BAD_PAGE);
      pg.npages = 0;
    }
    return pg;
  };
  // TMA of page j of `pg` into buffer j % kBufs (lane 0)
  auto issue = [&](const Pages& pg, int j) {
    const int b = j % C::kBufs;
    uint8_t* kb = my_ring + b * C::kBufBytes;
    uint8_t* vb = kb + C::kPageBytes;
    mbar_arrive_expect_tx(&my_bars[b], C::kBufBytes);
    int id = pg.page_id[0];  // select with constant indices: the ids stay in registers
#pragma unroll
    for (int t = 1; t < C::kMaxPages; ++t)
      if (j == t) id = pg.page_id[t];
    const int row0 = ((layer * max_pages + id) * p.n_kv_heads + pg.h) * kPage;
    for (int cb = 0; cb < C::kBoxes; ++cb) {
      tma_load_2d(kb + cb * 2048, &kmap, cb * 64, row0, &my_bars[b], pol);
      tma_load_2d(vb + cb * 2048, &vmap, cb * 64, row0, &my_bars[b], pol);
    }
  };
  // the 16 x D Q tile of work item w (query qi = token row r0 + qi / G, head
  // h G + qi % G): element vector v of this thread, zero past the block's rows
  auto q_vec = [&](int w, int v) {
    const int rb = w % n_rb, h = (w / n_rb) % p.n_kv_heads;
    const int qi = v / (D / 8), c8 = v % (D / 8);
    uint4 val = make_uint4(0u, 0u, 0u, 0u);
    if (qi < min(RB, M - rb * RB) * G) {
      const int r = rb * RB + qi / G, hq = h * G + qi % G;
      val = __ldcg(reinterpret_cast<const uint4*>(p.q + (size_t)r * p.n_q_heads * D + hq * D + c8 * 8));
    }
    return val;
  };
  constexpr int kQV = (16 * (D / 8) + C::kThreads - 1) / C::kThreads;  // Q vectors per thread

  // ---- the first item: pages of earlier steps requested before the wait
  Pages cur = pages_of(cta);
  {
    int n_old = 0;  // pages of positions < pos only: written by earlier steps
    while (n_old < cur.npages && n_old < C::kBufs && cur.wpos0 + (n_old + 1) * kPage <= pos) ++n_old;
    if (lane == 0)
      for (int j = 0; j < n_old; ++j) issue(cur, j);
    pdl_wait();  // Q and the K/V of the step's own rows come from the QKV kernel
    if (lane == 0) {
      asm volatile("fence.proxy.async.global;" ::: "memory");  // K/V written with plain stores
      for (int j = n_old; j < cur.npages && j < C::kBufs; ++j) issue(cur, j);
    }
    for (int k = 0; k < kQV; ++k) {
      const int v = tid + k * C::kThreads;
      if (v < 16 * (D / 8))
        *reinterpret_cast<uint4*>(sm.Qs + (v / (D / 8)) * C::kQStride + (v % (D / 8)) * 8) = q_vec(cta, v);
    }
  }
  int qb = 0;        // Q buffer of the current item
  bool ready = true;  // the current item's first pages are requested and its Q tile staged

  for (int w = cta; w < work; w += G_ctas) {
    const int rb = w % n_rb;
    const int h = cur.h;
    const int split = w / (n_rb * p.n_kv_heads);
    const int r0 = rb * RB;
    const int nrows = min(RB, M - r0);
    const int wpos0 = cur.wpos0, npages = cur.npages;
    bf16* Qs = sm.Qs + qb * 16 * C::kQStride;
    if (!ready) {  // not requested by the previous item: request it now
      if (lane == 0)
        for (int j = 0; j < npages && j < C::kBufs; ++j) issue(cur, j);
      for (int k = 0; k < kQV; ++k) {
        const int v = tid + k * C::kThreads;
        if (v < 16 * (D / 8))
          *reinterpret_cast<uint4*>(Qs + (v / (D / 8)) * C::kQStride + (v % (D / 8)) * 8) = q_vec(w, v);
      }
    }
    // the next item of this CTA: its page ids and Q, fetched while this one runs
    const int wn = w + G_ctas;
    const bool has_next = wn < work;
    Pages nxt;
    nxt.npages = 0;
    uint4 qn[kQV];
    if (has_next) {
      nxt = pages_of(wn);
      for (int k = 0; k < kQV; ++k) {
        const int v = tid + k * C::kThreads;
        qn[k] = v < 16 * (D / 8) ? q_vec(wn, v) : make_uint4(0u, 0u, 0u, 0u);
      }
      // buffers this item leaves unused go to the next item right away
      if (lane == 0)
        for (int b = npages; b < C::kBufs && b < nxt.npages; ++b) issue(nxt, b);
    }
    named_sync(2, C::kThreads);  // the Q tile is in place

    // query rows held by this lane: g and g + 8
    const int ctx_lo = pos + r0 + g / G + 1;
    const int ctx_hi = pos + r0 + (g + 8) / G + 1;
    float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.0f, 0.0f};
    float o[D / 8][4];
#pragma unroll
    for (int n = 0; n < D / 8; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.0f;

    const uint32_t q_base = smem_u32(Qs) + (uint32_t)((((lane & 7) + ((lane >> 3) & 1) * 8) * C::kQStride +
                                                       (lane >> 4) * 8) * 2);
    bool ok = true;
    for (int j = 0; j < npages; ++j) {
      const int b = j % C::kBufs;
      if (!mbar_wait(&my_bars[b], (phase >> b) & 1u)) {
        ok = false;
        break;
      }
      phase ^= 1u << b;
      const uint32_t kb = smem_u32(my_ring + b * C::kBufBytes);
      const uint32_t vb = kb + C::kPageBytes;
      // S = Q K^T for 16 queries x 16 positions
      float s[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        uint32_t a[4];
        ldsm_x4(q_base + kk * 32, a[0], a[1], a[2], a[3]);
        const int pr = (lane & 7) + ((lane >> 4) & 1) * 8;
        const int ch = (kk & 3) * 2 + ((lane >> 3) & 1);
        uint32_t b0, b1, b2, b3;
        ldsm_x4(kb + (kk >> 2) * 2048 + pr * 128 + ((ch ^ (pr & 7)) << 4), b0, b1, b2, b3);
        mma_bf16(s[0], a, b0, b1);
        mma_bf16(s[1], a, b2, b3);
      }
      // mask (exact -inf beyond each row's context), scale to log2 units
      const int pbase = wpos0 + j * kPage;
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int pabs = pbase + nt * 8 + 2 * q4 + (e & 1);
          const int ctx = e < 2 ? ctx_lo : ctx_hi;
          s[nt][e] = pabs < ctx ? __fmul_rn(s[nt][e], p.scale_log2) : -INFINITY;
        }
      // online softmax on rows g (e = 0, 1) and g + 8 (e = 2, 3).  The weights
      // p stay fp32: the denominator sums them unrounded, and P V is taken as
      // P_hi V + P_lo V with P_hi = bf16(p) and P_lo = bf16(p - P_hi) (the
      // tensor cores take bf16), which carries p to about 2^-16 -- a bf16-only
      // P would shift every attention output by up to half a bf16 step.
      float alpha[2];
      uint32_t pa[4], pl[4];
#pragma unroll
      for (int rr = 0; rr < 2; ++rr) {
        float mx = fmaxf(fmaxf(s[0][2 * rr], s[0][2 * rr + 1]), fmaxf(s[1][2 * rr], s[1][2 * rr + 1]));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
        const float m_new = fmaxf(m_run[rr], mx);
        float pv[4];
        if (m_new == -INFINITY) {
          alpha[rr] = 1.0f;
          pv[0] = pv[1] = pv[2] = pv[3] = 0.0f;
        } else {
          alpha[rr] = exp2f(__fsub_rn(m_run[rr], m_new));
          pv[0] = exp2f(__fsub_rn(s[0][2 * rr], m_new));
          pv[1] = exp2f(__fsub_rn(s[0][2 * rr + 1], m_new));
          pv[2] = exp2f(__fsub_rn(s[1][2 * rr], m_new));
          pv[3] = exp2f(__fsub_rn(s[1][2 * rr + 1], m_new));
        }
        float sum = __fadd_rn(__fadd_rn(pv[0], pv[1]), __fadd_rn(pv[2], pv[3]));
        sum = __fadd_rn(sum, __shfl_xor_sync(0xffffffffu, sum, 1));
        sum = __fadd_rn(sum, __shfl_xor_sync(0xffffffffu, sum, 2));
        l_run[rr] = __fadd_rn(__fmul_rn(l_run[rr], alpha[rr]), sum);
        m_run[rr] = m_new;
        pa[rr] = pack_bf16x2(pv[0], pv[1]);      // positions 2q, 2q+1
        pa[2 + rr] = pack_bf16x2(pv[2], pv[3]);  // positions 8+2q, 9+2q
        pl[rr] = pack_bf16x2(__fsub_rn(pv[0], bf16r(pv[0])), __fsub_rn(pv[1], bf16r(pv[1])));
        pl[2 + rr] = pack_bf16x2(__fsub_rn(pv[2], bf16r(pv[2])), __fsub_rn(pv[3], bf16r(pv[3])));
      }
#pragma unroll
      for (int n = 0; n < D / 8; ++n) {
        o[n][0] = __fmul_rn(o[n][0], alpha[0]);
        o[n][1] = __fmul_rn(o[n][1], alpha[0]);
        o[n][2] = __fmul_rn(o[n][2], alpha[1]);
        o[n][3] = __fmul_rn(o[n][3], alpha[1]);
      }
      // O += P_hi V + P_lo V
      const uint32_t afr[4] = {pa[0], pa[1], pa[2], pa[3]};
      const uint32_t afl[4] = {pl[0], pl[1], pl[2], pl[3]};
#pragma unroll
      for (int dn = 0; dn < D / 16; ++dn) {
        const int pr = (lane & 7) + ((lane >> 3) & 1) * 8;
        const int ch = ((dn * 16) & 63) / 8 + (lane >> 4);
        uint32_t b0, b1, b2, b3;
        ldsm_x4_trans(vb + ((dn * 16) >> 6) * 2048 + pr * 128 + ((ch ^ (pr & 7)) << 4), b0, b1, b2, b3);
        mma_bf16(o[2 * dn], afr, b0, b1);
        mma_bf16(o[2 * dn + 1], afr, b2, b3);
        mma_bf16(o[2 * dn], afl, b0, b1);
        mma_bf16(o[2 * dn + 1], afl, b2, b3);
      }
      fence_proxy_async_smem();  // reads of buffer b precede its next TMA write
      __syncwarp();
      if (lane == 0) {
        if (j + C::kBufs < npages)
          issue(cur, j + C::kBufs);
        else if (has_next && b < nxt.npages)
          issue(nxt, b);  // buffer b's last page of this item: the next item's page b
      }
    }
    if (!ok) all_ok = false;

    attn_merge_warps<D>(p, scratch, nrows, G, r0, h, split, m_run, l_run, o);
    if (has_next) {  // the next item's Q tile, into the other buffer
      bf16* Qn = sm.Qs + (qb ^ 1) * 16 * C::kQStride;
      for (int k = 0; k < kQV; ++k) {
        const int v = tid + k * C::kThreads;
        if (v < 16 * (D / 8)) *reinterpret_cast<uint4*>(Qn + (v / (D / 8)) * C::kQStride + (v % (D / 8)) * 8) = qn[k];
      }
    }
    named_sync(2, C::kThreads);  // the scratch is rewritten by the next item
    if (has_next) {
      qb ^= 1;
      cur = nxt;
    } else if (wn < work) {
      cur = pages_of(wn);
    }
    ready = has_next;
  }
  return all_ok;
}

// One element of the split merge: out[r, hq, i] from the partials of the
// splits that cover [0, pos + r + 1), merged in order.  The partials of up to
// kCombineChunk splits (contexts up to 2048) are requested together; longer
// contexts take the maximum in a first pass and accumulate in a second,
// kCombineChunk at a time.
template <int D>
__device__ __forceinline__ void combine_element(const AttnParams& p, int r, int hq, int i, int pos) {
  constexpr int kChunk = kCombineChunk;
  const int ctx = pos + r + 1;
  const int ns = attn_n_splits(ctx, D);
  const size_t base = ((size_t)r * p.n_q_heads + hq) * p.max_splits;
  float2 ml[kChunk];
  float ov[kChunk];
  float mx = -INFINITY;
  if (ns > kChunk)
    for (int s = 0; s < ns; ++s) mx = fmaxf(mx, __ldcg(&p.part_ml[base + s].x));
  float L = 0.0f, acc = 0.0f;
  for (int s0 = 0; s0 < ns; s0 += kChunk) {
#pragma unroll
    for (int j = 0; j < kChunk; ++j) {
      if (s0 + j < ns) {
        ml[j] = __ldcg(&p.part_ml[base + s0 + j]);
        ov[j] = __ldcg(&p.part_o[(base + s0 + j) * D + i]);
      }
    }
    if (ns <= kChunk) {
#pragma unroll
      for (int j = 0; j < kChunk; ++j)
        if (j < ns) mx = fmaxf(mx, ml[j].x);
    }
#pragma unroll
    for (int j = 0; j < kChunk; ++j) {
      if (s0 + j >= ns || ml[j].x == -INFINITY) continue;
      const float sc = exp2f(__fsub_rn(ml[j].x, mx));
      L = __fadd_rn(L, __fmul_rn(ml[j].y, sc));
      acc = __fadd_rn(acc, __fmul_rn(ov[j], sc));
    }
  }
  p.out[(size_t)r * p.n_q_heads * D + hq * D + i] = __float2bfloat16_rn(__fdiv_rn(acc, L));
  asm volatile("fence.proxy.async.global;" ::: "memory");  // read next by bulk copies
}

// The merge for contexts of more than eight splits, all D elements of (row r,
// head hq) by the block's D threads (thread i: element i).  The (m, l) pairs
// of every split are staged in shared memory (s_ml, ns entries) with their
// maximum taken block-wide; then each thread adds its element's splits in
// order, the loads of the next 16 splits in flight while the previous 16 are
// added.  Same maximum, same ordered sums and so the same bits as the chunked
// loop of combine_element, without one L2 round trip per eight splits.
template <int D>
__device__ __forceinline__ void combine_long(const AttnParams& p, int r, int hq, int ns, float2* s_ml,
                                             float* s_red) {
  constexpr int C = 16;
  const int i = threadIdx.x, lane = i & 31, warp = i >> 5;
  const size_t base = ((size_t)r * p.n_q_heads + hq) * p.max_splits;
  float m = -INFINITY;
  for (int s = i; s < ns; s += D) {
    const float2 v = __ldcg(&p.part_ml[base + s]);
    s_ml[s] = v;
    m = fmaxf(m, v.x);
  }
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if (lane == 0) s_red[warp] = m;
  __syncthreads();
  float mx = -INFINITY;
#pragma unroll
  for (int w = 0; w < D / 32; ++w) mx = fmaxf(mx, s_red[w]);
  float ov[2][C];
  float L = 0.0f, acc = 0.0f;
  auto load = [&](float (&dst)[C], int s0) {
#pragma unroll
    for (int j = 0; j < C; ++j)
      if (s0 + j < ns) dst[j] = __ldcg(&p.part_o[(base + s0 + j) * D + i]);
  };
  auto add = [&](const float (&src)[C], int s0) {
#pragma unroll
    for (int j = 0; j < C; ++j) {
      if (s0 + j >= ns) break;
      const float2 v = s_ml[s0 + j];
      if (v.x == -INFINITY) continue;
      const float sc = exp2f(__fsub_rn(v.x, mx));
      L = __fadd_rn(L, __fmul_rn(v.y, sc));
      acc = __fadd_rn(acc, __fmul_rn(src[j], sc));
    }
  };
  load(ov[0], 0);
  for (int s0 = 0; s0 < ns; s0 += 2 * C) {
    load(ov[1], s0 + C);
    add(ov[0], s0);
    load(ov[0], s0 + 2 * C);
    add(ov[1], s0 + C);
  }
  p.out[(size_t)r * p.n_q_heads * D + hq * D + i] = __float2bfloat16_rn(__fdiv_rn(acc, L));
  asm volatile("fence.proxy.async.global;" ::: "memory");  // read next by bulk copies
}

}  // namespace
}  // namespace sv
