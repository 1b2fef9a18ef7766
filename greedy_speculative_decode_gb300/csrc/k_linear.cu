// k_linear.cu -- the batch-invariant linear: Y[m, n] = sum_k X[m, k] W[n, k]
// for the few rows m of a decode / verify step, with fused prologue and
// epilogues.
//
// Weights are the only large operand, so the kernel is built to stream them
// once from HBM at full bandwidth: one producer warp issues TMA loads of
// 128-row x 64-column weight boxes (128B-swizzled) into a 4-stage mbarrier
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
#include "sv_internal.h"
#include "sv_ptx.cuh"

namespace sv {

namespace {

struct TileRows {
  int a0, b0;  // first weight row of chunk A (local rows 0..63) and chunk B (64..127)
};

__device__ __forceinline__ TileRows tile_rows(const LinParams& p, int tile) {
  TileRows t;
  if (p.map == MAP_GATE_UP) {
    t.a0 = tile * 64;
    t.b0 = p.ffn + tile * 64;
  } else if (p.map == MAP_HEAD256) {
    int h = tile >> 1, j = tile & 1;
    t.a0 = h * 256 + j * 64;
    t.b0 = t.a0 + 128;
  } else {
    t.a0 = tile * kLinRows;
    t.b0 = t.a0 + 64;
  }
  return t;
}

__device__ __forceinline__ int local_to_row(const TileRows& t, int lr) {
  return lr < 64 ? t.a0 + lr : t.b0 + (lr - 64);
}

__device__ __forceinline__ float act_fn(float g, int act) {
  if (act == 0) return g / (1.0f + expf(-g));
  const float k0 = 0.7978845608028654f, k1 = 0.044715f;
  return 0.5f * g * (1.0f + tanhf(k0 * (g + k1 * g * g * g)));
}

// QKV epilogue: per-head norm + RoPE + stores.  T: [128][TS] fp32 tile,
// already summed over splits, columns m < M valid.
__device__ void epilogue_qkv(const LinParams& p, int tile, float* T, int TS, float* s_rstd) {
  const int tid = threadIdx.x, M = p.M, d = p.head_dim;
  const int nthr = kLinConsumerWarps * 32;
  const TileRows tr = tile_rows(p, tile);
  const int pos = p.st->step_pos;
  const int qrows = p.n_q_heads * d, krows = p.n_kv_heads * d;
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
  for (int e = tid; e < kLinRows * M; e += nthr) {
    int lr = e % kLinRows, m = e / kLinRows;
    int f = local_to_row(tr, lr);
    int i = f % d;
    int head = f / d;
    float v = T[lr * TS + m];
    float outv = v;
    if (f < qrows + krows) {
      int lp = (i < half) ? lr + (d <= 128 ? half : 64) : lr - (d <= 128 ? half : 64);
      float other = T[lp * TS + m];
      int ii = i < half ? i : i - half;
      float2 cs = p.rope[(size_t)(pos + m) * half + ii];
      outv = (i < half) ? __fsub_rn(__fmul_rn(v, cs.x), __fmul_rn(other, cs.y))
                        : __fadd_rn(__fmul_rn(v, cs.x), __fmul_rn(other, cs.y));
    }
    bf16 ob = __float2bfloat16_rn(outv);
    if (f < qrows) {
      p.out[(size_t)m * p.out_stride + f] = ob;
    } else {
      int kvh = (f < qrows + krows) ? head - p.n_q_heads : head - p.n_q_heads - p.n_kv_heads;
      int ps = pos + m;
      int page = (ps < p.st->cap_len) ? p.block_table[ps / kPage] : -1;
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
}

__device__ void epilogue_resid(const LinParams& p, int tile, float* T, int TS) {
  const int tid = threadIdx.x, M = p.M, nthr = kLinConsumerWarps * 32;
  const int n0 = tile * kLinRows;
  for (int e = tid; e < kLinRows * M; e += nthr) {
    int lr = e % kLinRows, m = e / kLinRows;
    size_t o = (size_t)m * p.out_stride + n0 + lr;
    float r = __bfloat162float(p.out[o]);
    float v = bf16r(__fadd_rn(r, bf16r(T[lr * TS + m])));
    p.out[o] = __float2bfloat16_rn(v);
    T[lr * TS + m] = v;
  }
  named_sync(1, nthr);
  const int warp = tid >> 5, lane = tid & 31;
  for (int m = warp; m < M; m += kLinConsumerWarps) {
    float ss = 0.0f;
    for (int j = 0; j < kLinRows / 32; ++j) {
      float v = T[(lane + 32 * j) * TS + m];
      ss = __fadd_rn(ss, __fmul_rn(v, v));
    }
    for (int o = 16; o > 0; o >>= 1) ss = __fadd_rn(ss, __shfl_xor_sync(0xffffffffu, ss, o));
    if (lane == 0) p.out_ss[m * p.n_tiles + tile] = ss;
  }
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
}

__device__ void epilogue_logits(const LinParams& p, int tile, float* T, int TS) {
  const int tid = threadIdx.x, M = p.M, nthr = kLinConsumerWarps * 32;
  const int n0 = tile * kLinRows;
  for (int e = tid; e < kLinRows * M; e += nthr) {
    int lr = e % kLinRows, m = e / kLinRows;
    float v = bf16r(T[lr * TS + m]);
    T[lr * TS + m] = v;
    if (p.logits != nullptr && m >= p.logits_row0 && n0 + lr < p.vocab)
      p.logits[(size_t)(m - p.logits_row0) * p.vocab + n0 + lr] = v;
  }
  named_sync(1, nthr);
  const int warp = tid >> 5, lane = tid & 31;
  for (int m = warp; m < M; m += kLinConsumerWarps) {
    // each lane scans 4 consecutive rows in order, then a fixed tree picks the
    // largest value, the lowest id among equal values
    float best = -INFINITY;
    int bidx = 0x7fffffff;
    for (int j = 0; j < 4; ++j) {
      int lr = lane * 4 + j;
      if (n0 + lr >= p.vocab) continue;
      float v = T[lr * TS + m];
      if (bidx == 0x7fffffff || v > best) {
        best = v;
        bidx = n0 + lr;
      }
    }
    for (int o = 1; o < 32; o <<= 1) {
      float ov = __shfl_xor_sync(0xffffffffu, best, o);
      int oi = __shfl_xor_sync(0xffffffffu, bidx, o);
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

// Owner of flattened k-block kb under the even split of T k-blocks over G CTAs
// (CTA c owns [c T / G, (c + 1) T / G)).
__device__ __forceinline__ int owner_cta(long long kb, long long T, int G) {
  return (int)(((kb + 1) * G - 1) / T);
}

// Stage input columns c0 + t (mod Kd), t in [t0, t0 + ncols), of the M rows
// into xs (row stride XS), RMS-normalising them when NORM; rows M..MP-1 and
// columns past ncols are zero.  c0, t0 and Kd are multiples of 64.
template <int MP, int XS, bool NORM>
__device__ __forceinline__ void stage_x(const LinParams& p, bf16* xs, int c0, int t0, int ncols,
                                        const float* s_rstd, int tid, int nthr) {
  constexpr int VPR = (XS - 8) / 8;  // 16-byte vectors per staged row
  for (int v = tid; v < MP * VPR; v += nthr) {
    const int m = v / VPR, c8 = v % VPR;
    uint4 val = make_uint4(0u, 0u, 0u, 0u);
    if (m < p.M && c8 * 8 < ncols) {
      int k = c0 + t0 + c8 * 8;
      if (k >= p.Kd) k -= p.Kd;
      val = *reinterpret_cast<const uint4*>(p.X + (size_t)m * p.Kd + k);
      if (NORM) {
        const float r = s_rstd[m];
        const uint4 gv = *reinterpret_cast<const uint4*>(p.gain + k);
        const bf16* xb = reinterpret_cast<const bf16*>(&val);
        const bf16* gb = reinterpret_cast<const bf16*>(&gv);
        uint32_t w[4];
        for (int j = 0; j < 4; ++j) {
          float y0 = bf16r(__fmul_rn(bf16r(__fmul_rn(__bfloat162float(xb[2 * j]), r)),
                                     __bfloat162float(gb[2 * j])));
          float y1 = bf16r(__fmul_rn(bf16r(__fmul_rn(__bfloat162float(xb[2 * j + 1]), r)),
                                     __bfloat162float(gb[2 * j + 1])));
          w[j] = pack_bf16x2(y0, y1);
        }
        val = make_uint4(w[0], w[1], w[2], w[3]);
      }
    }
    *reinterpret_cast<uint4*>(xs + (size_t)m * XS + c8 * 8) = val;
  }
}

// Persistent stream-K linear.  The n_tiles x (Kd/64) k-blocks of the weight,
// tile-major, are cut into gridDim.x equal contiguous ranges, one per CTA.
// A tile whose k-blocks all fall in one CTA is finished there; a tile cut by
// range boundaries is finished by the last of its CTAs to arrive, which sums
// the per-CTA partials in k order.  The partition depends only on the weight
// shape and the grid (one CTA per SM), never on M.
template <int MT, int EPI, bool NORM>
__global__ void __launch_bounds__(kLinThreads, 1)
    k_linear(const __grid_constant__ CUtensorMap wmap, const LinParams p) {
  constexpr int MP = MT * 8;                                  // padded token rows
  constexpr int TS = MP + 1;                                  // epilogue tile row stride
  constexpr int XC = kLinXCols / MT;  // input columns staged at once
  constexpr int XS = XC + 8;          // staged row stride in elements (16B pad: no bank conflicts)
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* ring = smem;
  bf16* xs = reinterpret_cast<bf16*>(smem + kLinStages * kLinStageBytes);
  float* T = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(xs) + MP * XS * sizeof(bf16));
  uint64_t* full = reinterpret_cast<uint64_t*>(reinterpret_cast<uint8_t*>(T) +
                                               ((kLinRows * TS * sizeof(float) + 15) & ~size_t(15)));
  uint64_t* empty = full + kLinStages;
  float* s_rstd = reinterpret_cast<float*>(empty + kLinStages);  // [32] row rstd of the input
  float* s_hrstd = s_rstd + kMaxK;                               // [64] per-head rstd (QKV)
  int* s_flag = reinterpret_cast<int*>(s_hrstd + 64);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int KB = p.Kd / kLinBK;
  const long long Tk = (long long)p.n_tiles * KB;
  const int G = gridDim.x;
  const long long kb_begin = (long long)blockIdx.x * Tk / G;
  const long long kb_end = (long long)(blockIdx.x + 1) * Tk / G;

  if (tid == 0) {
    for (int s = 0; s < kLinStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kLinConsumerWarps);
    }
    fence_barrier_init();
  }
  __syncthreads();
  // Let the next kernel in the stream start its own weight prefetch.
  pdl_trigger();

  if (warp == kLinConsumerWarps) {
    // ---------------- producer: weights do not depend on earlier kernels
    if (lane == 0) {
      prefetch_tensormap(&wmap);
      const uint64_t pol = policy_evict_first();
      bool ok = true;
      int it = 0;
      int tile = (int)(kb_begin / KB), kk = (int)(kb_begin % KB);  // walked without division
      for (long long kb = kb_begin; kb < kb_end; ++kb, ++it) {
        const int s = it % kLinStages;
        if (it >= kLinStages) ok = mbar_wait(&empty[s], ((it / kLinStages) & 1) ^ 1);
        if (!ok) break;
        const TileRows tr = tile_rows(p, tile);
        mbar_arrive_expect_tx(&full[s], kLinStageBytes);
        uint8_t* dst = ring + s * kLinStageBytes;
        tma_load_2d(dst, &wmap, kk * kLinBK, tr.a0, &full[s], pol);
        tma_load_2d(dst + kLinChunkBytes, &wmap, kk * kLinBK, tr.b0, &full[s], pol);
        if (++kk == KB) {
          kk = 0;
          ++tile;
        }
      }
      if (!ok) atomicOr(&p.st->status, ST_TIMEOUT);
    }
    return;
  }

  // ---------------- consumers
  pdl_wait();  // X, its sums of squares and the step state come from earlier kernels
  const int nthr = kLinConsumerWarps * 32;
  if (NORM) {
    if (tid < p.M) {
      float ss = 0.0f;
      for (int t = 0; t < p.ss_tiles; ++t) ss = __fadd_rn(ss, p.x_ss[tid * p.ss_tiles + t]);
      s_rstd[tid] = 1.0f / sqrtf(ss / (float)p.Kd + p.eps);
    }
  }

  const int chunk = warp >> 2, rg = warp & 3;
  const int g = lane >> 2, q = lane & 3;
  const int lr0 = chunk * 64 + rg * 16 + g;
  const int a_row = rg * 16 + ((lane >> 3) & 1) * 8 + (lane & 7);  // row within the 64-row chunk
  const int a_khalf = lane >> 4;
  const uint32_t xs_base =
      smem_u32(xs) + (uint32_t)(((lane & 7) * XS + ((lane >> 3) & 1) * 8) * sizeof(bf16));
  float acc[MT][4];
#pragma unroll
  for (int t = 0; t < MT; ++t) acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.0f;

  // The input columns this CTA reads form one circular window of Kd starting
  // at its first k-block; it is staged XC columns at a time, usually once.
  const int c0 = (int)(kb_begin % KB) * kLinBK;
  const int ncols = (int)((kb_end - kb_begin) * kLinBK < p.Kd ? (kb_end - kb_begin) * kLinBK : p.Kd);
  bool ok = true;
  int staged = -1;
  long long seg_begin = kb_begin;
  int it = 0;
  int tile_c = (int)(kb_begin / KB), kk_c = (int)(kb_begin % KB);  // walked without division
  for (long long kb = kb_begin; kb < kb_end; ++kb, ++it) {
    const int tile = tile_c, kk = kk_c;
    if (++kk_c == KB) {
      kk_c = 0;
      ++tile_c;
    }
    int jw = kk * kLinBK - c0;  // column offset within the window
    if (jw < 0) jw += p.Kd;
    const int xchunk = jw / XC;
    if (xchunk != staged) {
      named_sync(1, nthr);  // all warps are done with the previous chunk (and s_rstd is set)
      stage_x<MP, XS, NORM>(p, xs, c0, xchunk * XC, min(XC, ncols - xchunk * XC), s_rstd, tid, nthr);
      named_sync(1, nthr);
      staged = xchunk;
    }
    const int s = it % kLinStages;
    if (ok && !mbar_wait(&full[s], (it / kLinStages) & 1)) ok = false;
    if (ok) {
      const uint32_t tile_base = smem_u32(ring + s * kLinStageBytes + chunk * kLinChunkBytes);
      const uint32_t xcol = (uint32_t)(jw - xchunk * XC);
#pragma unroll
      for (int k16 = 0; k16 < kLinBK / 16; ++k16) {
        uint32_t a[4];
        const int kc = k16 * 2 + a_khalf;
        ldsm_x4(tile_base + a_row * 128 + ((kc ^ (a_row & 7)) << 4), a[0], a[1], a[2], a[3]);
#pragma unroll
        for (int t = 0; t < MT; ++t) {
          uint32_t b0, b1;
          ldsm_x2(xs_base + (uint32_t)(((t * 8) * XS + xcol + k16 * 16) * sizeof(bf16)), b0, b1);
          mma_bf16(acc[t], a, b0, b1);
        }
      }
    }
    fence_proxy_async_smem();  // our ldmatrix reads of stage s precede its next TMA write
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);

    if (kk != KB - 1 && kb != kb_end - 1) continue;
    // ------------ this CTA's part of `tile` is complete
    const int kk_first = kb - seg_begin >= kk ? 0 : kk - (int)(kb - seg_begin);
    seg_begin = kb + 1;
    named_sync(1, nthr);  // the previous tile's epilogue is done with T
    if (kk_first == 0 && kk == KB - 1) {
#pragma unroll
      for (int t = 0; t < MT; ++t) {
        const int m0 = t * 8 + 2 * q;
        T[lr0 * TS + m0] = acc[t][0];
        T[lr0 * TS + m0 + 1] = acc[t][1];
        T[(lr0 + 8) * TS + m0] = acc[t][2];
        T[(lr0 + 8) * TS + m0 + 1] = acc[t][3];
      }
    } else {
      const int c_first = owner_cta((long long)tile * KB, Tk, G);
      const int c_last = owner_cta((long long)tile * KB + KB - 1, Tk, G);
      const int nseg = c_last - c_first + 1, seg = blockIdx.x - c_first;
      float* wsb = p.ws + ((size_t)(tile * p.max_seg + seg) * kLinRows) * MP;
#pragma unroll
      for (int t = 0; t < MT; ++t) {
        const int m0 = t * 8 + 2 * q;
        *reinterpret_cast<float2*>(wsb + lr0 * MP + m0) = make_float2(acc[t][0], acc[t][1]);
        *reinterpret_cast<float2*>(wsb + (lr0 + 8) * MP + m0) = make_float2(acc[t][2], acc[t][3]);
      }
      __threadfence();
      named_sync(1, nthr);
      if (tid == 0) {
        const int prev = atomicAdd(&p.counters[tile], 1);
        *s_flag = (prev == nseg - 1);
      }
      named_sync(1, nthr);
      const bool last = *s_flag != 0;
      if (last) {
        __threadfence();
        // last CTA of this tile: sum the partials of its CTAs in k order
        const float* wst = p.ws + ((size_t)tile * p.max_seg * kLinRows) * MP;
        for (int e = tid; e < kLinRows * p.M; e += nthr) {
          const int lr = e / p.M, m = e % p.M;
          float v = __ldcg(wst + lr * MP + m);
          for (int j = 1; j < nseg; ++j)
            v = __fadd_rn(v, __ldcg(wst + ((size_t)j * kLinRows + lr) * MP + m));
          T[lr * TS + m] = v;
        }
        if (tid == 0) p.counters[tile] = 0;  // ready for the next launch
      }
#pragma unroll
      for (int t = 0; t < MT; ++t) acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.0f;
      if (!last) continue;
    }
#pragma unroll
    for (int t = 0; t < MT; ++t) acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.0f;
    named_sync(1, nthr);
    if (EPI == EPI_QKV)
      epilogue_qkv(p, tile, T, TS, s_hrstd);
    else if (EPI == EPI_RESID)
      epilogue_resid(p, tile, T, TS);
    else if (EPI == EPI_GLU)
      epilogue_glu(p, tile, T, TS);
    else
      epilogue_logits(p, tile, T, TS);
  }
  if (!ok && lane == 0) atomicOr(&p.st->status, ST_TIMEOUT);
}

template <int MT, int EPI, bool NORM>
cudaError_t launch_t(const LinearDesc& d, const LinParams& p, cudaStream_t s, bool pdl) {
  const size_t smem = linear_smem_bytes(MT);
  auto kern = k_linear<MT, EPI, NORM>;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(d.grid);
  cfg.blockDim = dim3(kLinThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, d.map, p);
}

template <int MT, int EPI, bool NORM>
cudaError_t prepare_t() {
  return cudaFuncSetAttribute(k_linear<MT, EPI, NORM>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)linear_smem_bytes(MT));
}

template <int MT>
cudaError_t prepare_mt() {
  cudaError_t e;
  if ((e = prepare_t<MT, EPI_QKV, true>()) != cudaSuccess) return e;
  if ((e = prepare_t<MT, EPI_RESID, false>()) != cudaSuccess) return e;
  if ((e = prepare_t<MT, EPI_GLU, true>()) != cudaSuccess) return e;
  return prepare_t<MT, EPI_LOGITS, true>();
}

template <int MT>
cudaError_t launch_mt(const LinearDesc& d, const LinParams& p, int epi, bool norm, cudaStream_t s,
                      bool pdl) {
  switch (epi) {
    case EPI_QKV:
      return norm ? launch_t<MT, EPI_QKV, true>(d, p, s, pdl) : cudaErrorInvalidValue;
    case EPI_RESID:
      return norm ? cudaErrorInvalidValue : launch_t<MT, EPI_RESID, false>(d, p, s, pdl);
    case EPI_GLU:
      return norm ? launch_t<MT, EPI_GLU, true>(d, p, s, pdl) : cudaErrorInvalidValue;
    case EPI_LOGITS:
      return norm ? launch_t<MT, EPI_LOGITS, true>(d, p, s, pdl) : cudaErrorInvalidValue;
  }
  return cudaErrorInvalidValue;
}

}  // namespace

size_t linear_smem_bytes(int mt) {
  const int mp = mt * 8;
  const int xc = kLinXCols / mt;
  size_t b = 1024;  // alignment slack
  b += (size_t)kLinStages * kLinStageBytes;
  b += (size_t)mp * (xc + 8) * sizeof(bf16);
  b += ((size_t)kLinRows * (mp + 1) * sizeof(float) + 15) & ~size_t(15);
  b += 2 * kLinStages * sizeof(uint64_t) + (kMaxK + 64) * sizeof(float) + 16;
  return b;
}

void linear_partition(int n_tiles, int Kd, int num_sms, int* grid, int* max_seg) {
  const long long KB = Kd / kLinBK, T = (long long)n_tiles * KB;
  const int G = (int)(T < num_sms ? T : num_sms);
  int ms = 1;
  for (int t = 0; t < n_tiles; ++t) {
    const int c0 = (int)(((t * KB + 1) * G - 1) / T);
    const int c1 = (int)(((t * KB + KB) * G - 1) / T);
    if (c1 - c0 + 1 > ms) ms = c1 - c0 + 1;
  }
  *grid = G;
  *max_seg = ms;
}

cudaError_t prepare_linear_kernels() {
  cudaError_t e;
  if ((e = prepare_mt<1>()) != cudaSuccess) return e;
  if ((e = prepare_mt<2>()) != cudaSuccess) return e;
  return prepare_mt<4>();
}

cudaError_t launch_linear(const LinearDesc& d, const LinParams& p, int epi, bool norm,
                          cudaStream_t s, bool pdl) {
  if (p.M <= 8) return launch_mt<1>(d, p, epi, norm, s, pdl);
  if (p.M <= 16) return launch_mt<2>(d, p, epi, norm, s, pdl);
  if (p.M <= 32) return launch_mt<4>(d, p, epi, norm, s, pdl);
  return cudaErrorInvalidValue;
}

}  // namespace sv
