// lin_dev.cuh -- the batch-invariant linear: Y[m, n] = sum_k X[m, k] W[n, k]
// for the few rows m of a decode / verify step, with fused prologue and
// epilogues.
//
// Weights are the only large operand, so the kernel is built to stream them
// once from HBM at full bandwidth: one producer warp issues TMA loads of
// 128-row x 64-column weight boxes (128B-swizzled) into an 8-stage mbarrier
// ring; eight consumer warps feed them to bf16 tensor-core mma.sync with the
// weight rows as the 16-row A operand and the token rows as the 8-column B
// operand ("swap AB").  Every output element is the same sequence of mma
// instructions over the same k order whatever M is (token rows are
// independent mma columns, padded with zeros to 8, 16 or 32), the split of K
// over CTAs depends only on the weight shape, and split partials are summed
// in split order by whichever CTA arrives last.  So row r of an M-row call is
// bit-identical to the same row computed alone: the requirement of
// "Phase 23: Speculative Verify Parity" section 2 step 3 (verify rows must
// round exactly like single-token decode), met here without the page's
// per-row GEMV, which re-reads every weight once per row.
//
// Prologue (norm): X rows are RMS-normalised on the fly from per-128-column
// partial sums of squares written by the producer of X.
// Epilogues: QKV (per-head RMSNorm of q and k, rotate-half RoPE, paged K/V
// write of rows pos..pos+M-1), RESID (residual add in place + new partial
// sums of squares), GLU (act(gate) * up), LOGITS (bf16 logits + per-tile
// argmax with ties to the lowest id).
#pragma once
#include "sv_internal.h"
#include "sv_ptx.cuh"

namespace sv {
namespace {

struct TileRows {
  int a0, b0;  // first weight row of chunk A (local rows 0..63) and chunk B (64..127)
};

__device__ __forceinline__ TileRows tile_rows_of(int map, int ffn, int tile) {
  TileRows t;
  if (map == MAP_GATE_UP) {
    t.a0 = tile * 64;
    t.b0 = ffn + tile * 64;
  } else if (map == MAP_HEAD256) {
    int h = tile >> 1, j = tile & 1;
    t.a0 = h * 256 + j * 64;
    t.b0 = t.a0 + 128;
  } else {
    t.a0 = tile * kLinRows;
    t.b0 = t.a0 + 64;
  }
  return t;
}

__device__ __forceinline__ TileRows tile_rows(const LinParams& p, int tile) {
  return tile_rows_of(p.map, p.ffn, tile);
}

__device__ __forceinline__ int local_to_row(const TileRows& t, int lr) {
  return lr < 64 ? t.a0 + lr : t.b0 + (lr - 64);
}

__device__ __forceinline__ float act_fn(float g, int act) {
  if (act == 0) return g / (1.0f + expf(-g));
  const float k0 = 0.7978845608028654f, k1 = 0.044715f;
  return 0.5f * g * (1.0f + tanhf(k0 * (g + k1 * g * g * g)));
}

// Epilogue operands that live in global memory, loaded for a tile as soon as
// the CTA has finished its share of it -- before it learns whether it is the
// CTA that completes the tile -- so their latency overlaps the exchange of
// partial sums.  Each is held by the thread whose epilogue uses it: in the
// one-warp-per-token-row epilogues, warp w takes rows m = w + 8 k and lane l
// the tile rows l + 32 j; in the general QKV epilogue, element j of thread tid
// is e = tid + j * 256 (tile row e mod 128, token row e / 128).
template <int MP>
struct EpiPre {
  static constexpr int N = (kLinRows * MP + kLinConsumerWarps * 32 - 1) / (kLinConsumerWarps * 32);
  // EPI_RESID: the residual x[m, n0 + lr]; QKV, head_dim 128: the QK-norm gain
  // of elements lane + 32 j (j < 4).  Raw bf16 bits, widened where they are
  // used: nothing here consumes a preloaded value, so the thread goes on to
  // request the split partials without waiting for these loads.
  uint32_t resb[N];
  float2 cs[N];   // EPI_QKV: (cos, sin) of the element's RoPE angle
  int page[N];    // EPI_QKV: physical page of position pos + m (-1: none)
};

template <int MP, int EPI>
__device__ __forceinline__ void epi_preload(const LinParams& p, int tile, int pos, int cap,
                                            EpiPre<MP>& pre) {
  const int tid = threadIdx.x, nthr = kLinConsumerWarps * 32;
  if (EPI == EPI_RESID) {  // warp w: rows m = w + 8 k, elements lane + 32 j (see epilogue_resid)
    const int warp = tid >> 5, lane = tid & 31;
#pragma unroll
    for (int k = 0; k < MP / 8; ++k) {
      const int m = warp + 8 * k;
      if (m < p.M) {
        const bf16* row = p.out + (size_t)m * p.out_stride + tile * kLinRows + lane;
#pragma unroll
        for (int j = 0; j < 4; ++j)  // written by other CTAs: bypass L1
          pre.resb[4 * k + j] = __ldcg(reinterpret_cast<const unsigned short*>(row + 32 * j));
      }
    }
  } else if (EPI == EPI_QKV && p.head_dim == kLinRows) {
    // one head per tile, one warp per token row (see epilogue_qkv): row
    // m = warp + 8 k, lane's RoPE angles for elements lane and lane + 32
    const int warp = tid >> 5, lane = tid & 31, half = kLinRows / 2;
    const bool kv = tile * kLinRows >= p.n_q_heads * kLinRows;
    if (p.q_gain != nullptr && tile < p.n_q_heads + p.n_kv_heads) {  // q or k: its norm gain
      const bf16* g = kv ? p.k_gain : p.q_gain;
#pragma unroll
      for (int j = 0; j < 4; ++j) pre.resb[j] = __ldg(reinterpret_cast<const unsigned short*>(g + lane + 32 * j));
    }
#pragma unroll
    for (int k = 0; k < MP / 8; ++k) {
      const int m = warp + 8 * k;
      pre.cs[2 * k] = pre.cs[2 * k + 1] = make_float2(1.0f, 0.0f);
      pre.page[k] = -1;
      if (m < p.M) {
        const float2* rp = p.rope + (size_t)(pos + m) * half;
        pre.cs[2 * k] = rp[lane];
        pre.cs[2 * k + 1] = rp[lane + 32];
        if (kv && pos + m < cap) pre.page[k] = p.block_table[(pos + m) / kPage];
      }
    }
  } else if (EPI == EPI_QKV) {
    const TileRows tr = tile_rows(p, tile);
    const int d = p.head_dim, half = d / 2;
    const int qrows = p.n_q_heads * d, krows = p.n_kv_heads * d;
#pragma unroll
    for (int j = 0; j < EpiPre<MP>::N; ++j) {
      const int e = tid + j * nthr;
      pre.cs[j] = make_float2(1.0f, 0.0f);
      pre.page[j] = -1;
      if (e < kLinRows * p.M) {
        const int lr = e % kLinRows, m = e / kLinRows;
        const int f = local_to_row(tr, lr), i = f % d;
        if (f < qrows + krows) pre.cs[j] = p.rope[(size_t)(pos + m) * half + (i < half ? i : i - half)];
        const int ps = pos + m;
        if (f >= qrows && ps < cap) pre.page[j] = p.block_table[ps / kPage];
      }
    }
  }
}

// QKV epilogue: per-head norm + RoPE + stores.  T: [128][TS] fp32 tile,
// already summed over splits, columns m < M valid.
template <int MP>
__device__ void epilogue_qkv(const LinParams& p, int tile, float* T, int TS, float* s_rstd, int pos,
                             const EpiPre<MP>& pre) {
  const int tid = threadIdx.x, M = p.M, d = p.head_dim;
  const int nthr = kLinConsumerWarps * 32;
  const int qrows = p.n_q_heads * d, krows = p.n_kv_heads * d;
  if (d == kLinRows) {
    // The tile is exactly one head (q, k or v).  One warp per token row; lane
    // holds elements i = lane + 32 j, j = 0..3, so the head's norm is a warp
    // reduction and the RoPE partners (i, i + 64) sit in the same lane: no
    // CTA barrier.  Same arithmetic, in the same order, as the general path.
    const int warp = tid >> 5, lane = tid & 31;
    const int f0 = tile * kLinRows, head = tile;
    const bool is_q = f0 < qrows, is_k = !is_q && f0 < qrows + krows;
#pragma unroll
    for (int k = 0; k < MP / 8; ++k) {
      const int m = warp + 8 * k;
      if (m >= M) break;
      float v[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) v[j] = bf16r(T[(lane + 32 * j) * TS + m]);
      if (p.q_gain != nullptr && (is_q || is_k)) {
        float ss = 0.0f;
#pragma unroll
        for (int j = 0; j < 4; ++j) ss = __fadd_rn(ss, __fmul_rn(v[j], v[j]));
        for (int o = 16; o > 0; o >>= 1) ss = __fadd_rn(ss, __shfl_xor_sync(0xffffffffu, ss, o));
        const float r = 1.0f / sqrtf(ss / (float)d + p.eps);
#pragma unroll
        for (int j = 0; j < 4; ++j) v[j] = bf16r(__fmul_rn(bf16r(__fmul_rn(v[j], r)), __uint_as_float(pre.resb[j] << 16)));
      }
      float outv[4] = {v[0], v[1], v[2], v[3]};
      if (is_q || is_k) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {  // pairs (j, j + 2): elements i and i + 64
          const float2 cs = pre.cs[2 * k + h];
          outv[h] = __fsub_rn(__fmul_rn(v[h], cs.x), __fmul_rn(v[h + 2], cs.y));
          outv[h + 2] = __fadd_rn(__fmul_rn(v[h + 2], cs.x), __fmul_rn(v[h], cs.y));
        }
      }
      if (is_q) {
        bf16* dst = p.out + (size_t)m * p.out_stride + f0;
#pragma unroll
        for (int j = 0; j < 4; ++j) dst[lane + 32 * j] = __float2bfloat16_rn(outv[j]);
      } else {
        const int page = pre.page[k], ps = pos + m;
        if (page < 0) {
          if (lane == 0) atomicOr(&p.st->status, ST_BAD_PAGE);
          continue;
        }
        const int kvh = is_k ? head - p.n_q_heads : head - p.n_q_heads - p.n_kv_heads;
        bf16* dst = (is_k ? p.kcache : p.vcache) +
                    (((size_t)page * p.n_kv_heads + kvh) * kPage + (ps % kPage)) * d;
#pragma unroll
        for (int j = 0; j < 4; ++j) dst[lane + 32 * j] = __float2bfloat16_rn(outv[j]);
      }
    }
    // the cached K/V are read next through TMA (the async proxy)
    asm volatile("fence.proxy.async.global;" ::: "memory");
    return;
  }
  const TileRows tr = tile_rows(p, tile);
  // 1. round the projection to bf16
  for (int e = tid; e < kLinRows * M; e += nthr) {
    int lr = e % kLinRows, m = e / kLinRows;
    T[lr * TS + m] = bf16r(T[lr * TS + m]);
  }
  named_sync(1, nthr);
  // 2. per-head RMSNorm of q and k (head_dim <= 128: whole heads in the tile)
  const int heads_in_tile = d <= 128 ? kLinRows / d : 0;
  const bool tile_qk = local_to_row(tr, 0) < qrows + krows;
  if (p.q_gain != nullptr && heads_in_tile > 0 && tile_qk) {
    const int warp = tid >> 5, lane = tid & 31;
    for (int seg = warp; seg < M * heads_in_tile; seg += kLinConsumerWarps) {
      int m = seg / heads_in_tile, hh = seg % heads_in_tile;
      float ss = 0.0f;
      for (int i = lane; i < d; i += 32) {
        float v = T[(hh * d + i) * TS + m];
        ss = __fadd_rn(ss, __fmul_rn(v, v));
      }
      for (int o = 16; o > 0; o >>= 1) ss = __fadd_rn(ss, __shfl_xor_sync(0xffffffffu, ss, o));
      if (lane == 0) s_rstd[seg] = 1.0f / sqrtf(ss / (float)d + p.eps);
    }
    named_sync(1, nthr);
    for (int e = tid; e < kLinRows * M; e += nthr) {
      int lr = e % kLinRows, m = e / kLinRows;
      int f = local_to_row(tr, lr);
      if (f >= qrows + krows) continue;
      const bf16* g = f < qrows ? p.q_gain : p.k_gain;
      float r = s_rstd[m * heads_in_tile + lr / d];
      T[lr * TS + m] = bf16r(bf16r(T[lr * TS + m] * r) * __bfloat162float(g[lr % d]));
    }
    named_sync(1, nthr);
  }
  // 3. RoPE on q and k pairs (i, i + d/2), then the stores
  const int half = d / 2;
#pragma unroll
  for (int j = 0; j < EpiPre<MP>::N; ++j) {
    const int e = tid + j * nthr;
    if (e >= kLinRows * M) break;
    int lr = e % kLinRows, m = e / kLinRows;
    int f = local_to_row(tr, lr);
    int i = f % d;
    int head = f / d;
    float v = T[lr * TS + m];
    float outv = v;
    if (f < qrows + krows) {
      int lp = (i < half) ? lr + (d <= 128 ? half : 64) : lr - (d <= 128 ? half : 64);
      float other = T[lp * TS + m];
      const float2 cs = pre.cs[j];
      outv = (i < half) ? __fsub_rn(__fmul_rn(v, cs.x), __fmul_rn(other, cs.y))
                        : __fadd_rn(__fmul_rn(v, cs.x), __fmul_rn(other, cs.y));
    }
    bf16 ob = __float2bfloat16_rn(outv);
    if (f < qrows) {
      p.out[(size_t)m * p.out_stride + f] = ob;
    } else {
      int kvh = (f < qrows + krows) ? head - p.n_q_heads : head - p.n_q_heads - p.n_kv_heads;
      const int ps = pos + m;
      const int page = pre.page[j];
      if (page < 0) {
        atomicOr(&p.st->status, ST_BAD_PAGE);
        continue;
      }
      size_t idx = (((size_t)page * p.n_kv_heads + kvh) * kPage + (ps % kPage)) * d + i;
      if (f < qrows + krows)
        p.kcache[idx] = ob;
      else
        p.vcache[idx] = ob;
    }
  }
  // the cached K/V are read next through TMA (the async proxy)
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// Residual epilogue: x[m, n0 + lr] += bf16(T[lr, m]) (rounded to bf16), and
// the tile's sum of squares of each new row for the next RMSNorm.  One warp
// per token row, lane l holding tile rows l + 32 j: no CTA barrier.
template <int MP>
__device__ void epilogue_resid(const LinParams& p, int tile, float* T, int TS, const EpiPre<MP>& pre) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n0 = tile * kLinRows;
#pragma unroll
  for (int k = 0; k < MP / 8; ++k) {
    const int m = warp + 8 * k;
    if (m >= p.M) break;
    bf16* row = p.out + (size_t)m * p.out_stride + n0 + lane;
    float ss = 0.0f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float v = bf16r(__fadd_rn(__uint_as_float(pre.resb[4 * k + j] << 16), bf16r(T[(lane + 32 * j) * TS + m])));
      row[32 * j] = __float2bfloat16_rn(v);
      ss = __fadd_rn(ss, __fmul_rn(v, v));
    }
    for (int o = 16; o > 0; o >>= 1) ss = __fadd_rn(ss, __shfl_xor_sync(0xffffffffu, ss, o));
    if (lane == 0) p.out_ss[m * p.n_tiles + tile] = ss;
  }
  // the next linear reads these rows with bulk copies (the async proxy)
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

__device__ void epilogue_glu(const LinParams& p, int tile, const float* T, int TS) {
  const int tid = threadIdx.x, M = p.M, nthr = kLinConsumerWarps * 32;
  for (int e = tid; e < 64 * M; e += nthr) {
    int lr = e % 64, m = e / 64;
    float g = bf16r(T[lr * TS + m]);
    float u = bf16r(T[(lr + 64) * TS + m]);
    float a = bf16r(act_fn(g, p.act));
    p.out[(size_t)m * p.out_stride + tile * 64 + lr] = __float2bfloat16_rn(__fmul_rn(a, u));
  }
  asm volatile("fence.proxy.async.global;" ::: "memory");  // read next by bulk copies
}

// LM-head epilogue: bf16 logits (stored for rows m >= logits_row0 when a
// buffer is given) and the tile's argmax of each row: largest value, lowest id
// among equal values.  One warp per token row; lane l scans tile rows 4 l ..
// 4 l + 3 in order, then a fixed xor tree combines the lanes.
template <int MP>
__device__ void epilogue_logits(const LinParams& p, int tile, float* T, int TS) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n0 = tile * kLinRows;
#pragma unroll
  for (int k = 0; k < MP / 8; ++k) {
    const int m = warp + 8 * k;
    if (m >= p.M) break;
    const bool store = p.logits != nullptr && m >= p.logits_row0;
    float* lrow = store ? p.logits + (size_t)(m - p.logits_row0) * p.vocab + n0 : nullptr;
    float best = -INFINITY;
    int bidx = 0x7fffffff;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int lr = lane * 4 + j;
      if (n0 + lr >= p.vocab) continue;
      const float v = bf16r(T[lr * TS + m]);
      if (store) lrow[lr] = v;
      if (bidx == 0x7fffffff || v > best) {
        best = v;
        bidx = n0 + lr;
      }
    }
    for (int o = 1; o < 32; o <<= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, best, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bidx, o);
      if (ov > best || (ov == best && oi < bidx)) {
        best = ov;
        bidx = oi;
      }
    }
    if (lane == 0) {
      p.am_val[m * p.n_tiles + tile] = best;
      p.am_idx[m * p.n_tiles + tile] = bidx;
    }
  }
}

// Split-tile partial slots of this form: fp32 words [CTA][128 tile rows][MP
// token rows].  A word not yet written holds kLinEmpty, a NaN with the sign
// bit set: arithmetic only produces the canonical NaN 0x7fffffff, so no
// partial sum equals it.  Each 32-bit element of a .v2 access is single-copy
// atomic, so a word is either the value or still empty: the stores are the
// message (no fence, no flag).  The reducer writes kLinEmpty back into every
// word it consumed; the slots are all kLinEmpty between launches.
constexpr uint32_t kLinEmpty = 0xffffffffu;

__device__ __forceinline__ void st_relaxed_v2_u32(uint32_t* p, uint32_t a, uint32_t b) {
  asm volatile("st.relaxed.gpu.global.v2.u32 [%0], {%1, %2};" ::"l"(p), "r"(a), "r"(b) : "memory");
}

__device__ __forceinline__ void ld_relaxed_v2_u32(const uint32_t* p, uint32_t& a, uint32_t& b) {
  asm volatile("ld.relaxed.gpu.global.v2.u32 {%0, %1}, [%2];" : "=r"(a), "=r"(b) : "l"(p) : "memory");
}

// Split-tile segments the reducer requests at once: three for 16 padded rows,
// one for 32; for 8, the smallest of two, four or six (4, 8 or 12 word pairs
// a thread) that takes a tile's other max_seg - 1 segments in the fewest
// rounds: the smaller batch is the cheaper code (measured 1-5% faster steps on
// the 0.6B- and Gemma-shaped models, 0.5% on the 8B-shaped one).  The sums and
// their order do not depend on it.
__host__ __device__ constexpr int lin_seg_batch(int mt, int max_seg) {
  return mt == 2 ? 3
         : mt == 4 ? 1
         : max_seg <= 3 ? 2
         : ((max_seg + 2) / 4 <= (max_seg + 4) / 6 ? 4 : 6);
}

// Reducer side of a split tile: acc holds segment 0 (this CTA's); add the
// partials that CTAs cta + 1 ... cta + nseg - 1 left in their slots, segment
// by segment, each thread for the elements its accumulators hold, and empty
// the words it consumed.  The words of B segments are requested together and
// the missing ones re-requested in rounds, so a batch costs one L2 round trip
// once its partials have landed.  Returns false if a partial never arrived
// (bounded by kWaitLimitNs).
template <int MT, int B>
__device__ __forceinline__ bool gather_partials(uint32_t* ws, int cta, int nseg, int lr0, int q,
                                                float (&acc)[MT][4]) {
  constexpr int MP = MT * 8;
  constexpr int NP = B * MT * 2;            // word pairs per thread and batch (registers: 4 B MT)
  static_assert(NP <= 32, "one bit per pair");
  bool ok = true;
  for (int j0 = 1; j0 < nseg; j0 += B) {
    // pair i = (segment j0 + i / (2 MT), accumulator t = (i / 2) % MT, row half i % 2)
    auto addr = [&](int i) {
      const int jj = i / (2 * MT), t = (i / 2) % MT, half = i % 2;
      return ws + (size_t)(cta + j0 + jj) * kLinRows * MP + (lr0 + 8 * half) * MP + t * 8 + 2 * q;
    };
    uint32_t x[NP], y[NP];
    uint32_t live = 0;
#pragma unroll
    for (int i = 0; i < NP; ++i) {
      x[i] = y[i] = 0u;
      if (j0 + i / (2 * MT) < nseg) {
        live |= 1u << i;
        ld_relaxed_v2_u32(addr(i), x[i], y[i]);
      }
    }
    auto missing = [&]() {
      uint32_t m = 0;
#pragma unroll
      for (int i = 0; i < NP; ++i)
        if (((live >> i) & 1u) && (x[i] == kLinEmpty || y[i] == kLinEmpty)) m |= 1u << i;
      return m;
    };
    uint32_t m = missing();
    if (m != 0) {
      const unsigned long long t0 = globaltimer_ns();
      for (;;) {
#pragma unroll
        for (int i = 0; i < NP; ++i)
          if ((m >> i) & 1u) ld_relaxed_v2_u32(addr(i), x[i], y[i]);
        m = missing();
        if (m == 0) break;
        if (globaltimer_ns() - t0 > kWaitLimitNs) {
          ok = false;
          break;
        }
      }
    }
#pragma unroll
    for (int i = 0; i < NP; ++i) {
      if ((live >> i) & 1u) {
        const int t = (i / 2) % MT, half = i % 2;
        acc[t][2 * half] = __fadd_rn(acc[t][2 * half], __uint_as_float(x[i]));
        acc[t][2 * half + 1] = __fadd_rn(acc[t][2 * half + 1], __uint_as_float(y[i]));
        st_relaxed_v2_u32(addr(i), kLinEmpty, kLinEmpty);
      }
    }
  }
  return ok;
}

// Owner of flattened k-block kb under the even split of T k-blocks over G CTAs
// (CTA c owns [c T / G, (c + 1) T / G)).
__device__ __forceinline__ int owner_cta(long long kb, long long T, int G) {
  return (int)(((kb + 1) * G - 1) / T);
}

// Input staging.  The CTA's input window is columns c0 + t (mod Kd), t in
// [0, ncols), of the M rows; it is staged XC columns at a time (usually all at
// once).  One thread bulk-copies each row's run of the chunk into xs (row
// stride XS) -- two copies where the window wraps past Kd -- so the whole
// chunk is one L2 round trip; with NORM the rows are then RMS-normalised in
// place.  Rows M..MP-1 are zero (set before the kernel waits on its
// predecessor).  c0, t0, XC and Kd are multiples of 64.

// Thread 0: issue the bulk copies of chunk [t0, t0 + nc) of the M rows.
__device__ __forceinline__ void stage_issue(const LinParams& p, bf16* xs, int XS, int c0, int t0,
                                            int nc, uint64_t* xbar) {
  mbar_arrive_expect_tx(xbar, (uint32_t)(p.M * nc * (int)sizeof(bf16)));
  int k0 = c0 + t0;
  if (k0 >= p.Kd) k0 -= p.Kd;
  const int first = min(nc, p.Kd - k0);  // columns before the wrap
  for (int m = 0; m < p.M; ++m) {
    const bf16* row = p.X + (size_t)m * p.Kd;
    bf16* dst = xs + (size_t)m * XS;
    bulk_load(dst, row + k0, (uint32_t)(first * sizeof(bf16)), xbar);
    if (first < nc) bulk_load(dst + first, row, (uint32_t)((nc - first) * sizeof(bf16)), xbar);
  }
}

// y = bf16(bf16(x * rstd) * gain) of two packed bf16 values (low half first).
__device__ __forceinline__ uint32_t norm2(uint32_t x2, float r, uint32_t g2) {
  const float x0 = __uint_as_float(x2 << 16), x1 = __uint_as_float(x2 & 0xffff0000u);
  const uint32_t t2 = pack_bf16x2(__fmul_rn(x0, r), __fmul_rn(x1, r));
  const float t0 = __uint_as_float(t2 << 16), t1 = __uint_as_float(t2 & 0xffff0000u);
  const float g0 = __uint_as_float(g2 << 16), g1 = __uint_as_float(g2 & 0xffff0000u);
  return pack_bf16x2(__fmul_rn(t0, g0), __fmul_rn(t1, g1));
}

// The same for eight values.
__device__ __forceinline__ uint4 norm8(uint4 x, float r, uint4 g) {
  return make_uint4(norm2(x.x, r, g.x), norm2(x.y, r, g.y), norm2(x.z, r, g.z), norm2(x.w, r, g.w));
}

// Shared-memory carve-up of a linear CTA (see linear_smem_bytes).
struct LinSmem {
  uint8_t* ring;
  uint64_t* full;
  uint64_t* empty;
  uint64_t* xbar;  // completion of the input rows' bulk copies
  uint64_t* gbar;  // completion of the gain window's bulk copy
  bf16* xs;
  float* T;
  bf16* gs;        // gain of the input window (NORM)
  float* s_rstd;   // [kMaxK] row rstd of the input
  float* s_hrstd;  // [64] per-head rstd (QKV epilogue)
  int* s_flag;
};

template <int MT>
__device__ __forceinline__ LinSmem lin_smem(uint8_t* smem) {
  constexpr int MP = MT * 8, TS = MP + 1, XC = LinGeom<MT>::kXCols, XS = XC + 8;
  LinSmem sm;
  sm.ring = smem;
  sm.xs = reinterpret_cast<bf16*>(smem + LinGeom<MT>::kStages * kLinStageBytes);
  sm.T = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(sm.xs) + MP * XS * sizeof(bf16));
  sm.gs = reinterpret_cast<bf16*>(reinterpret_cast<uint8_t*>(sm.T) +
                                  ((kLinRows * TS * sizeof(float) + 15) & ~size_t(15)));
  sm.full = reinterpret_cast<uint64_t*>(sm.gs + kLinXCols);  // the gain of windows up to 4096 columns
  sm.empty = sm.full + kLinStages;
  sm.xbar = sm.empty + kLinStages;
  sm.gbar = sm.xbar + 1;
  sm.s_rstd = reinterpret_cast<float*>(sm.gbar + 1);
  sm.s_hrstd = sm.s_rstd + kMaxK;
  sm.s_flag = reinterpret_cast<int*>(sm.s_hrstd + 64);
  return sm;
}

// k-block range [kb_begin, kb_end) of CTA `cta` of G over the flattened
// n_tiles x (Kd/64) blocks.
__device__ __forceinline__ void lin_range(const LinParams& p, int cta, int G, long long& kb_begin,
                                          long long& kb_end) {
  const long long Tk = (long long)p.n_tiles * (p.Kd / kLinBK);
  kb_begin = (long long)cta * Tk / G;
  kb_end = (long long)(cta + 1) * Tk / G;
}

// One k-block (both 64-row chunks of `tile` at k-block kk) into `dst`,
// completing on `bar`: one bulk copy from the tiled layout, else two box
// loads from the row-major weight.  Either way the shared-memory bytes are
// the same.
__device__ __forceinline__ void load_weight_block(const LinParams& p, const CUtensorMap* wmap, uint8_t* dst,
                                                  int tile, int kk, uint64_t* bar, uint64_t pol) {
  if (p.wt != nullptr) {
    const size_t blk = (size_t)tile * (p.Kd / kLinBK) + kk;
    bulk_load_hint(dst, p.wt + blk * kLinStageBytes, kLinStageBytes, bar, pol);
  } else {
    const TileRows tr = tile_rows(p, tile);
    tma_load_2d(dst, wmap, kk * kLinBK, tr.a0, bar, pol);
    tma_load_2d(dst + kLinChunkBytes, wmap, kk * kLinBK, tr.b0, bar, pol);
  }
}

// Producer (one thread): TMA the CTA's weight boxes into the ring.  `it`
// counts ring uses (stage = it mod stages, parity = its quotient's low bit),
// kept in step with the consumers'.  Returns false on a timeout.
template <int S>  // ring stages
__device__ bool lin_produce(const LinParams& p, const CUtensorMap* wmap, int cta, int G,
                            const LinSmem& sm, int& it, uint64_t pol) {
  const int KB = p.Kd / kLinBK;
  long long kb_begin, kb_end;
  lin_range(p, cta, G, kb_begin, kb_end);
  int tile = (int)(kb_begin / KB), kk = (int)(kb_begin % KB);  // walked without division
  for (long long kb = kb_begin; kb < kb_end; ++kb, ++it) {
    const int s = it % S;
    if (it >= S && !mbar_wait(&sm.empty[s], ((it / S) & 1) ^ 1)) return false;
    mbar_arrive_expect_tx(&sm.full[s], kLinStageBytes);
    load_weight_block(p, wmap, sm.ring + s * kLinStageBytes, tile, kk, &sm.full[s], pol);
    if (++kk == KB) {
      kk = 0;
      ++tile;
    }
  }
  return true;
}

// Producer, after its own stream: prefetch into L2 the first pf_blocks
// k-blocks that CTA `cta` streams in the next linear of the step.
__device__ void lin_prefetch_next(const LinParams& p, const CUtensorMap* pfmap, int cta) {
  if (p.pf_blocks <= 0 || cta >= p.pf_grid) return;
  const int KB = p.pf_Kd / kLinBK;
  const long long Tk = (long long)p.pf_n_tiles * KB;
  const long long b0 = (long long)cta * Tk / p.pf_grid;
  long long b1 = (long long)(cta + 1) * Tk / p.pf_grid;
  if (b1 > b0 + p.pf_blocks) b1 = b0 + p.pf_blocks;
  int tile = (int)(b0 / KB), kk = (int)(b0 % KB);
  if (p.pf_wt != nullptr) {  // the tiled blocks are contiguous in this order
    bulk_prefetch_l2(p.pf_wt + (size_t)b0 * kLinStageBytes, (uint32_t)((b1 - b0) * kLinStageBytes));
    return;
  }
  for (long long kb = b0; kb < b1; ++kb) {
    const TileRows tr = tile_rows_of(p.pf_map, p.pf_ffn, tile);
    tma_prefetch_l2(pfmap, kk * kLinBK, tr.a0);
    tma_prefetch_l2(pfmap, kk * kLinBK, tr.b0);
    if (++kk == KB) {
      kk = 0;
      ++tile;
    }
  }
}

// The input window of CTA `cta`: columns c0 + t (mod Kd), t < ncols.
__device__ __forceinline__ void lin_window(const LinParams& p, long long kb_begin, long long kb_end,
                                           int& c0, int& ncols) {
  const int KB = p.Kd / kLinBK;
  c0 = (int)(kb_begin % KB) * kLinBK;
  const long long n = (kb_end - kb_begin) * kLinBK;
  ncols = (int)(n < p.Kd ? n : p.Kd);
}

// Normalise in place the 16-byte vectors v = first + tid, first + tid + 256,
// ... < last of the staged window (vector v: row v / per_row, column vector
// c8_0 + v % per_row), one or two per thread.
template <int XS>
__device__ __forceinline__ void norm_vectors(const LinSmem& sm, int c8_0, int per_row, int nv, int tid,
                                             int nthr) {
  const uint4* gs = reinterpret_cast<const uint4*>(sm.gs);
  for (int v = tid; v < nv; v += nthr) {
    const int m = v / per_row, c8 = c8_0 + v % per_row;
    uint4* ptr = reinterpret_cast<uint4*>(sm.xs + (size_t)m * XS + c8 * 8);
    *ptr = norm8(*ptr, sm.s_rstd[m], gs[c8]);
  }
}

// Consumers (the kLinConsumerWarps warps, named barrier 1): multiply the
// CTA's share of the weight with the staged input rows and finish every tile
// that ends in this CTA.  Returns false if a stage never arrived.
template <int MT, int EPI, bool NORM, int SB = lin_seg_batch(MT, kLinMaxSeg)>
__device__ bool lin_consume(const LinParams& p, int cta, int G, const LinSmem& sm, int& it) {
  constexpr int MP = MT * 8;          // padded token rows
  constexpr int TS = MP + 1;          // epilogue tile row stride
  constexpr int XC = LinGeom<MT>::kXCols;  // input columns staged at once
  constexpr int S = LinGeom<MT>::kStages;  // ring stages
  constexpr int XS = XC + 8;          // staged row stride in elements (16B pad: no bank conflicts)
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nthr = kLinConsumerWarps * 32;
  const int KB = p.Kd / kLinBK;
  const long long Tk = (long long)p.n_tiles * KB;
  long long kb_begin, kb_end;
  lin_range(p, cta, G, kb_begin, kb_end);
  if (kb_begin >= kb_end) return true;
  float* T = sm.T;
  int c0, ncols;
  lin_window(p, kb_begin, kb_end, c0, ncols);
  // A window that fits xs is staged once, right after the wait below; with
  // NORM it is normalised 256 columns (a group) at a time: group 0 before the
  // main loop, group g + 1 by all consumers while they stream group g, so
  // only the first group's normalisation is on the critical path.
  const bool one_chunk = ncols <= XC;
  constexpr int kGroup = 4 * kLinBK;  // columns per normalisation group
  const int ngroups = (ncols + kGroup - 1) / kGroup;

  // ---- before the wait on the previous kernel: nothing here depends on it
  // the gain window, staged whole for windows of up to kLinXCols columns
  // (a window of several chunks then normalises each chunk from it)
  const bool gain_staged = NORM && ncols <= kLinXCols;
  if (gain_staged && tid == 0) {
    const int first = min(ncols, p.Kd - c0);
    mbar_arrive_expect_tx(sm.gbar, (uint32_t)(ncols * sizeof(bf16)));
    bulk_load(sm.gs, p.gain + c0, (uint32_t)(first * sizeof(bf16)), sm.gbar);
    if (first < ncols) bulk_load(sm.gs + first, p.gain, (uint32_t)((ncols - first) * sizeof(bf16)), sm.gbar);
  }
  for (int v = tid; v < (MP - p.M) * (XS / 8); v += nthr)  // the padding rows are zero
    reinterpret_cast<uint4*>(sm.xs + (size_t)p.M * XS)[v] = make_uint4(0u, 0u, 0u, 0u);
  pdl_wait();  // X, its sums of squares and the step state come from earlier kernels
  if (one_chunk && tid == 0) stage_issue(p, sm.xs, XS, c0, 0, ncols, sm.xbar);
  int pos = 0, cap = 0;
  if (EPI == EPI_QKV) {
    pos = __ldcg(&p.st->step_pos);
    cap = __ldcg(&p.st->cap_len);
  }
  bool ok = true;
  if (one_chunk) {
    if (NORM) {  // row rstd (one warp per row) while the copies fly, then group 0
      for (int m = warp; m < p.M; m += kLinConsumerWarps) {
        float ss = 0.0f;
        for (int t = lane; t < p.ss_tiles; t += 32) ss = __fadd_rn(ss, __ldcg(p.x_ss + m * p.ss_tiles + t));
        for (int o = 16; o > 0; o >>= 1) ss = __fadd_rn(ss, __shfl_xor_sync(0xffffffffu, ss, o));
        if (lane == 0) sm.s_rstd[m] = 1.0f / sqrtf(ss / (float)p.Kd + p.eps);
      }
      named_sync(1, nthr);
      if (!mbar_wait(sm.xbar, 0) || !mbar_wait(sm.gbar, 0)) ok = false;
      const int w0 = min(kGroup, ncols) / 8;
      norm_vectors<XS>(sm, 0, w0, p.M * w0, tid, nthr);
    } else {
      if (!mbar_wait(sm.xbar, 0)) ok = false;
    }
  }
  named_sync(1, nthr);  // every warp reads every row (padding, group 0)

  const int chunk = warp >> 2, rg = warp & 3;
  const int g = lane >> 2, q = lane & 3;
  const int lr0 = chunk * 64 + rg * 16 + g;
  const int a_row = rg * 16 + ((lane >> 3) & 1) * 8 + (lane & 7);  // row within the 64-row chunk
  const int a_khalf = lane >> 4;
  const uint32_t xs_base =
      smem_u32(sm.xs) + (uint32_t)(((lane & 7) * XS + ((lane >> 3) & 1) * 8) * sizeof(bf16));
  // x4 form: lanes 16-31 address token rows 8-15 (the next token tile)
  const uint32_t xs_base4 = xs_base + (uint32_t)(((lane >> 4) & 1) * 8 * XS * sizeof(bf16));
  float acc[MT][4];
#pragma unroll
  for (int t = 0; t < MT; ++t) acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.0f;
  EpiPre<MP> pre;

  static_assert((S & (S - 1)) == 0, "the ring index is taken with a mask");
  const int Kd = p.Kd;
  int staged = one_chunk ? 0 : -1;  // chunk in xs
  uint32_t xphase = 0;
  // one-chunk NORM windows: at the first block of group g (window column
  // g * kGroup, g < ngroups) the consumers sync -- group g is then complete
  // everywhere -- and normalise group g + 1; norm_at is the next such column
  int norm_next = 1;
  int norm_at = (NORM && one_chunk && ngroups > 1) ? 0 : -1;
  int tile = (int)(kb_begin / KB), kk0 = (int)(kb_begin % KB);
  long long left = kb_end - kb_begin;
  int jw = 0;  // window column of the next k-block
  while (left > 0) {
    const int nblk = (int)(left < KB - kk0 ? left : KB - kk0);  // k-blocks of `tile` in this CTA
    for (int j = 0; j < nblk; ++j, ++it) {
      if (NORM && jw == norm_at) {
        named_sync(1, nthr);
        if (norm_next < ngroups) {
          const int w = min(kGroup, ncols - norm_next * kGroup) / 8;
          norm_vectors<XS>(sm, norm_next * (kGroup / 8), w, p.M * w, tid, nthr);
        }
        ++norm_next;
        norm_at = norm_next <= ngroups ? (norm_next - 1) * kGroup : -1;
      }
      int xcol = jw;
      if (!one_chunk) {  // a window of several chunks, staged here chunk by chunk
        const int xchunk = jw / XC;
        xcol = jw - xchunk * XC;
        if (xchunk != staged) {
          const int t0 = xchunk * XC, nc = min(XC, ncols - t0);
          fence_proxy_async_smem();  // earlier reads and writes of xs precede the bulk copies
          named_sync(1, nthr);
          if (tid == 0) stage_issue(p, sm.xs, XS, c0, t0, nc, sm.xbar);
          if (NORM && staged < 0) {  // row rstd, one warp per row, while the copies fly
            for (int m = warp; m < p.M; m += kLinConsumerWarps) {
              float ss = 0.0f;
              for (int t = lane; t < p.ss_tiles; t += 32) ss = __fadd_rn(ss, __ldcg(p.x_ss + m * p.ss_tiles + t));
              for (int o = 16; o > 0; o >>= 1) ss = __fadd_rn(ss, __shfl_xor_sync(0xffffffffu, ss, o));
              if (lane == 0) sm.s_rstd[m] = 1.0f / sqrtf(ss / (float)p.Kd + p.eps);
            }
            named_sync(1, nthr);
          }
          if (!mbar_wait(sm.xbar, xphase)) ok = false;
          xphase ^= 1u;
          if (NORM) {
            if (gain_staged && staged < 0 && !mbar_wait(sm.gbar, 0)) ok = false;
            for (int c8 = tid; c8 * 8 < nc; c8 += nthr) {
              int k = c0 + t0 + c8 * 8;
              if (k >= Kd) k -= Kd;
              const uint4 gv = gain_staged ? reinterpret_cast<const uint4*>(sm.gs)[t0 / 8 + c8]
                                           : __ldg(reinterpret_cast<const uint4*>(p.gain + k));
              for (int m = 0; m < p.M; ++m) {
                uint4* ptr = reinterpret_cast<uint4*>(sm.xs + (size_t)m * XS + c8 * 8);
                *ptr = norm8(*ptr, sm.s_rstd[m], gv);
              }
            }
          }
          named_sync(1, nthr);
          staged = xchunk;
        }
      }
      const int s = it & (S - 1);
      if (ok && !mbar_wait(&sm.full[s], (uint32_t)(it / S) & 1u)) ok = false;
      if (ok) {
        // every fragment of the block first, then the mma: the loads are
        // issued back to back instead of each waiting behind the previous mma
        // (each accumulator still takes its k16 steps in order)
        const uint32_t tile_base = smem_u32(sm.ring + s * kLinStageBytes + chunk * kLinChunkBytes);
        constexpr int K16 = kLinBK / 16;
        uint32_t a[K16][4], b[K16][MT][2];
#pragma unroll
        for (int k16 = 0; k16 < K16; ++k16) {
          const int kc = k16 * 2 + a_khalf;
          ldsm_x4(tile_base + a_row * 128 + ((kc ^ (a_row & 7)) << 4), a[k16][0], a[k16][1], a[k16][2],
                  a[k16][3]);
          if (MT == 1) {
            ldsm_x2(xs_base + (uint32_t)((xcol + k16 * 16) * sizeof(bf16)), b[k16][0][0], b[k16][0][1]);
          } else {
#pragma unroll
            for (int t = 0; t < MT; t += 2)  // the fragments of token tiles t and t + 1 at once
              ldsm_x4(xs_base4 + (uint32_t)(((t * 8) * XS + xcol + k16 * 16) * sizeof(bf16)), b[k16][t][0],
                      b[k16][t][1], b[k16][t + 1 < MT ? t + 1 : t][0], b[k16][t + 1 < MT ? t + 1 : t][1]);
          }
        }
#pragma unroll
        for (int k16 = 0; k16 < K16; ++k16)
#pragma unroll
          for (int t = 0; t < MT; ++t) mma_bf16(acc[t], a[k16], b[k16][t][0], b[k16][t][1]);
      }
      fence_proxy_async_smem();  // our ldmatrix reads of stage s precede its next TMA write
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.empty[s]);
      jw += kLinBK;
      if (jw == Kd) jw = 0;
    }
    // ------------ this CTA's part of the tile is complete (k-blocks kk_first..kk)
    const int kk = kk0 + nblk - 1, kk_first = kk0, tile_done = tile;
    left -= nblk;
    ++tile;
    kk0 = 0;
    if (kk_first != 0) {
      // A later segment of a split tile.  It is the first piece of this
      // CTA's range (every later tile starts at a tile boundary), so a CTA
      // leaves at most one partial: in its own slot (words kLinEmpty until
      // written).  The stores are the message: no fence, no ticket, and
      // nothing waits here.
      uint32_t* slot = p.ws + (size_t)cta * kLinRows * MP;
      const bool withheld = cta == p.withhold_cta1 - 1;  // test hook (see LinParams)
#pragma unroll
      for (int t = 0; t < MT; ++t) {
        const int m0 = t * 8 + 2 * q;
        if (!withheld) {
          st_relaxed_v2_u32(slot + lr0 * MP + m0, __float_as_uint(acc[t][0]), __float_as_uint(acc[t][1]));
          st_relaxed_v2_u32(slot + (lr0 + 8) * MP + m0, __float_as_uint(acc[t][2]), __float_as_uint(acc[t][3]));
        }
        acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.0f;
      }
      continue;
    }
    epi_preload<MP, EPI>(p, tile_done, pos, cap, pre);
    if (kk != KB - 1) {
      // The first segment of a split tile: the last piece of this CTA's
      // range, so waiting here holds up no stream.  The other segments belong
      // to CTAs cta + 1 ... c_last, in k order; add their partials in that
      // order (the same sums, in the same order, whichever CTAs ran them).
      const int nseg = owner_cta((long long)tile_done * KB + KB - 1, Tk, G) - cta + 1;
      if (!gather_partials<MT, SB>(p.ws, cta, nseg, lr0, q, acc)) ok = false;
    }
    named_sync(1, nthr);  // the previous tile's epilogue is done with T
#pragma unroll
    for (int t = 0; t < MT; ++t) {
      const int m0 = t * 8 + 2 * q;
      T[lr0 * TS + m0] = acc[t][0];
      T[lr0 * TS + m0 + 1] = acc[t][1];
      T[(lr0 + 8) * TS + m0] = acc[t][2];
      T[(lr0 + 8) * TS + m0 + 1] = acc[t][3];
      acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.0f;
    }
    named_sync(1, nthr);
    if (EPI == EPI_QKV)
      epilogue_qkv<MP>(p, tile_done, T, TS, sm.s_hrstd, pos, pre);
    else if (EPI == EPI_RESID)
      epilogue_resid<MP>(p, tile_done, T, TS, pre);
    else if (EPI == EPI_GLU)
      epilogue_glu(p, tile_done, T, TS);
    else
      epilogue_logits<MP>(p, tile_done, T, TS);
  }
  return ok;
}

}  // namespace
}  // namespace sv
