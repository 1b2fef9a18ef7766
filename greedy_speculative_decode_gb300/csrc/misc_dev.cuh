// misc_dev.cuh -- the small pieces of a step as device functions: the embedding gather
// (with the row statistics the first RMSNorm needs) and the argmax +
// acceptance + truncation of the window.
#pragma once
#include "sv_internal.h"
#include "sv_ptx.cuh"

namespace sv {
namespace {

// x[m, 128t + i] = E[token_m, 128t + i] for i < 128 threads of one group
// (named barrier `bar`), and x_ss[m, t] = the tile's sum of squares.
__device__ __forceinline__ void embed_tile(const bf16* __restrict__ E, int hidden, int vocab,
                                           bf16* __restrict__ x, float* __restrict__ x_ss,
                                           int ss_tiles, SvState* st, int m, int t, int i,
                                           float* part, int bar, const int32_t* tok_src) {
  int tok = tok_src ? tok_src[m] : st->tokens[m];
  if (tok_src && t == 0 && i == 0) st->tokens[m] = tok;  // for the accept kernel
  if (tok < 0 || tok >= vocab) {
    if (i == 0) atomicOr(&st->status, ST_BAD_TOKEN);
    tok = 0;
  }
  const int col = t * 128 + i;
  const bf16 v = E[(size_t)tok * hidden + col];
  x[(size_t)m * hidden + col] = v;
  asm volatile("fence.proxy.async.global;" ::: "memory");  // x is read next by bulk copies
  float f = __bfloat162float(v);
  float ss = __fmul_rn(f, f);
  for (int o = 16; o > 0; o >>= 1) ss = __fadd_rn(ss, __shfl_xor_sync(0xffffffffu, ss, o));
  if ((i & 31) == 0) part[i >> 5] = ss;
  named_sync(bar, 128);
  if (i == 0)
    x_ss[m * ss_tiles + t] = __fadd_rn(__fadd_rn(part[0], part[1]), __fadd_rn(part[2], part[3]));
  named_sync(bar, 128);  // part is reused by the group's next tile
}

// Greedy argmax of each row from the LM head's per-tile partials (largest
// value, lowest id on ties), then acceptance: n = number of leading drafts
// tokens[j+1] equal to argmax[j]; the row count committed is n + 1.  CTA 0
// writes the results; the K/V of rejected rows are zeroed in layers
// cta, cta + G_ctas, ...  A verify step whose tokens[0] was not the pending
// greedy token (step_reject) commits no row: every row of it is zeroed and
// the length and pending token stay as they were.  With delayed write-through
// (dl.bt_shadow) a verify step's rows are in the scratch pages instead: the
// accepted ones are copied into the real pages, nothing needs zeroing, and
// the shadow table gets the real pages back.  Runs on 256 threads (named
// barrier 1).
__device__ void accept_work(SvState* st, const float* am_val, const int* am_idx, int n_tiles, int M,
                            int mode, bf16* kpool, bf16* vpool, size_t layer_stride,
                            const int* block_table, int n_layers, int n_kv_heads, int head_dim,
                            const KvDelay& dl, int cta, int G_ctas, int* s_am, int* s_n,
                            int32_t* res_dst) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int pos = __ldcg(&st->step_pos);
  // the step's result, into the state block and, if given, the caller's buffer
  auto put_result = [&](int a, int b, int c, int d) {
    st->result[0] = a;
    st->result[1] = b;
    st->result[2] = c;
    st->result[3] = d;
    if (res_dst) {  // 4-byte aligned only
      res_dst[0] = a;
      res_dst[1] = b;
      res_dst[2] = c;
      res_dst[3] = d;
    }
  };
  if (mode == MODE_BODY) {
    if (cta == 0 && tid == 0) {
      st->seq_len = pos + M;
      put_result(M - 1, -1, pos + M, st->status);
    }
    return;
  }
  // Lane l takes tiles l, l + 32, ... in that order (so the result is the
  // same however the loads are batched), eight loads in flight at a time.
  for (int r = warp; r < M; r += 8) {
    float best = -INFINITY;
    int bidx = 0x7fffffff;
    for (int t0 = lane; t0 < n_tiles; t0 += 32 * 8) {
      float v[8];
      int id[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int t = t0 + 32 * u;
        v[u] = t < n_tiles ? __ldcg(&am_val[r * n_tiles + t]) : -INFINITY;
        id[u] = t < n_tiles ? __ldcg(&am_idx[r * n_tiles + t]) : 0x7fffffff;
      }
#pragma unroll
      for (int u = 0; u < 8; ++u)
        if (id[u] != 0x7fffffff && (bidx == 0x7fffffff || v[u] > best || (v[u] == best && id[u] < bidx))) {
          best = v[u];
          bidx = id[u];
        }
    }
    for (int o = 1; o < 32; o <<= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, best, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bidx, o);
      if (oi != 0x7fffffff && (bidx == 0x7fffffff || ov > best || (ov == best && oi < bidx))) {
        best = ov;
        bidx = oi;
      }
    }
    if (lane == 0) s_am[r] = bidx;
  }
  named_sync(1, 256);
  const bool reject = mode == MODE_VERIFY && __ldcg(&st->step_reject) != 0;
  if (tid == 0) {
    int n = M - 1;
    if (mode == MODE_VERIFY) {
      n = 0;
      while (n < M - 1 && st->tokens[n + 1] == s_am[n]) ++n;
    }
    *s_n = reject ? -1 : n;
  }
  named_sync(1, 256);
  const int n = *s_n;
  const int new_len = pos + 1 + n;  // pos when the step is rejected
  if (cta == 0 && tid == 0) {
    for (int r = 0; r < M; ++r) st->argmax[r] = s_am[r];
    st->seq_len = new_len;
    if (reject) {
      put_result(-1, st->pending, new_len, st->status | ST_BAD_STATE);
      st->state_err = 1;
    } else {
      st->pending = s_am[n];
      put_result(n, s_am[n], new_len, st->status);
    }
  }
  // K/V rows move in 16-byte vectors: a row of one kv head is head_dim
  // contiguous elements of its page.  Only positions below cap_len have pages.
  const int cap = __ldcg(&st->cap_len);
  const int vh = head_dim / 8;                   // vectors per (row, kv head)
  const int vrow = n_kv_heads * vh;              // vectors per row
  const size_t pv = (size_t)n_kv_heads * kPage * vh;  // vectors per page
  auto vec_off = [&](int page, int ps, int u) {  // vector u of row ps in `page`
    return (size_t)page * pv + ((size_t)(u / vh) * kPage + ps % kPage) * vh + u % vh;
  };
  if (dl.bt_shadow != nullptr && mode == MODE_VERIFY) {
    const int lp0 = pos / kPage;
    for (int l = cta; l < n_layers; l += G_ctas) {
      uint4* kl = reinterpret_cast<uint4*>(kpool + (size_t)l * layer_stride);
      uint4* vl = reinterpret_cast<uint4*>(vpool + (size_t)l * layer_stride);
      for (int e = tid; e < (new_len - pos) * vrow; e += 256) {  // the accepted rows
        const int ps = pos + e / vrow, u = e % vrow;
        const int page = ps < cap ? block_table[ps / kPage] : -1;
        if (page < 0) continue;
        const size_t src = vec_off(dl.win0 + ps / kPage - lp0, ps, u), dst = vec_off(page, ps, u);
        kl[dst] = kl[src];
        vl[dst] = vl[src];
      }
    }
    if (cta == 0 && tid < kWinPages) {
      const int lp = lp0 + tid;
      if (lp < dl.bt_len) dl.bt_shadow[lp] = block_table[lp];
    }
    return;
  }
  const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
  for (int l = cta; l < n_layers; l += G_ctas) {
    uint4* kl = reinterpret_cast<uint4*>(kpool + (size_t)l * layer_stride);
    uint4* vl = reinterpret_cast<uint4*>(vpool + (size_t)l * layer_stride);
    for (int e = tid; e < (pos + M - new_len) * vrow; e += 256) {  // the rejected rows
      const int ps = new_len + e / vrow, u = e % vrow;
      const int page = ps < cap ? block_table[ps / kPage] : -1;
      if (page < 0) continue;
      const size_t idx = vec_off(page, ps, u);
      kl[idx] = zero;
      vl[idx] = zero;
    }
  }
}

}  // namespace
}  // namespace sv
