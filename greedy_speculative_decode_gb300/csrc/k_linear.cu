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

template <int MT, int EPI, bool NORM>
__global__ void __launch_bounds__(kLinThreads, 2)
    k_linear(const __grid_constant__ CUtensorMap wmap, const LinParams p) {
  constexpr int MP = MT * 8;  // padded token rows
  constexpr int TS = MP + 1;  // epilogue tile row stride (floats)
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* ring = smem;
  const int xs_stride = p.Kc + 8;  // bf16 elements per staged row (16B pad vs bank conflicts)
  bf16* xs = reinterpret_cast<bf16*>(smem + kLinStages * kLinStageBytes);
  uint64_t* full = reinterpret_cast<uint64_t*>(reinterpret_cast<uint8_t*>(xs) +
                                               (size_t)MP * xs_stride * sizeof(bf16));
  uint64_t* empty = full + kLinStages;
  float* s_rstd = reinterpret_cast<float*>(empty + kLinStages);  // [64]
  int* s_flag = reinterpret_cast<int*>(s_rstd + 64);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int tile = blockIdx.x / p.splits, split = blockIdx.x % p.splits;
  const int k0 = split * p.Kc;
  const int n_iter = p.Kc / kLinBK;
  const TileRows tr = tile_rows(p, tile);

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
      for (int it = 0; it < n_iter && ok; ++it) {
        const int s = it % kLinStages;
        if (it >= kLinStages) ok = mbar_wait(&empty[s], ((it / kLinStages) & 1) ^ 1);
        if (!ok) break;
        mbar_arrive_expect_tx(&full[s], kLinStageBytes);
        uint8_t* dst = ring + s * kLinStageBytes;
        const int kc = k0 + it * kLinBK;
        tma_load_2d(dst, &wmap, kc, tr.a0, &full[s], pol);
        tma_load_2d(dst + kLinChunkBytes, &wmap, kc, tr.b0, &full[s], pol);
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
    named_sync(1, nthr);
  }
  {
    const int vec_per_row = p.Kc / 8;
    for (int v = tid; v < MP * vec_per_row; v += nthr) {
      const int m = v / vec_per_row, c8 = v % vec_per_row;
      uint4 val = make_uint4(0u, 0u, 0u, 0u);
      if (m < p.M) {
        const int k = k0 + c8 * 8;
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
      *reinterpret_cast<uint4*>(xs + (size_t)m * xs_stride + c8 * 8) = val;
    }
  }
  named_sync(1, nthr);

  const int chunk = warp >> 2, rg = warp & 3;
  float acc[MT][4];
#pragma unroll
  for (int t = 0; t < MT; ++t) acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.0f;

  // per-lane ldmatrix geometry
  const int a_row = rg * 16 + ((lane >> 3) & 1) * 8 + (lane & 7);  // row within the 64-row chunk
  const int a_khalf = lane >> 4;
  const uint32_t xs_base = smem_u32(xs) +
                           (uint32_t)(((lane & 7) * xs_stride + ((lane >> 3) & 1) * 8) * sizeof(bf16));
  bool ok = true;
  for (int it = 0; it < n_iter; ++it) {
    const int s = it % kLinStages;
    if (!mbar_wait(&full[s], (it / kLinStages) & 1)) {
      ok = false;
      break;
    }
    const uint32_t tile_base = smem_u32(ring + s * kLinStageBytes + chunk * kLinChunkBytes);
#pragma unroll
    for (int kk = 0; kk < kLinBK / 16; ++kk) {
      uint32_t a[4];
      const int kchunk = kk * 2 + a_khalf;
      ldsm_x4(tile_base + a_row * 128 + ((kchunk ^ (a_row & 7)) << 4), a[0], a[1], a[2], a[3]);
#pragma unroll
      for (int t = 0; t < MT; ++t) {
        uint32_t b0, b1;
        ldsm_x2(xs_base + (uint32_t)(((t * 8) * xs_stride + it * kLinBK + kk * 16) * sizeof(bf16)),
                b0, b1);
        mma_bf16(acc[t], a, b0, b1);
      }
    }
    fence_proxy_async_smem();  // our ldmatrix reads of stage s precede its next TMA write
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
  }
  if (!ok && lane == 0) atomicOr(&p.st->status, ST_TIMEOUT);

  // All stages consumed (or abandoned): reuse the ring for the fp32 tile.
  named_sync(1, nthr);
  float* T = reinterpret_cast<float*>(ring);
  const int g = lane >> 2, q = lane & 3;
  const int lr0 = chunk * 64 + rg * 16 + g;
  if (p.splits == 1) {
#pragma unroll
    for (int t = 0; t < MT; ++t) {
      const int m0 = t * 8 + 2 * q;
      T[lr0 * TS + m0] = acc[t][0];
      T[lr0 * TS + m0 + 1] = acc[t][1];
      T[(lr0 + 8) * TS + m0] = acc[t][2];
      T[(lr0 + 8) * TS + m0 + 1] = acc[t][3];
    }
  } else {
    float* wsb = p.ws + ((size_t)(tile * p.splits + split) * kLinRows) * MP;
#pragma unroll
    for (int t = 0; t < MT; ++t) {
      const int m0 = t * 8 + 2 * q;
      *reinterpret_cast<float2*>(wsb + lr0 * MP + m0) = make_float2(acc[t][0], acc[t][1]);
      *reinterpret_cast<float2*>(wsb + (lr0 + 8) * MP + m0) = make_float2(acc[t][2], acc[t][3]);
    }
    __threadfence();
    named_sync(1, nthr);
    if (tid == 0) {
      int prev = atomicAdd(&p.counters[tile], 1);
      *s_flag = (prev == p.splits - 1);
    }
    named_sync(1, nthr);
    if (!*s_flag) return;
    __threadfence();
    // Last CTA of this tile: sum the split partials in split order.
    const float* wst = p.ws + ((size_t)tile * p.splits * kLinRows) * MP;
    for (int e = tid; e < kLinRows * p.M; e += nthr) {
      const int lr = e / p.M, m = e % p.M;
      float v = __ldcg(wst + lr * MP + m);
      for (int sp = 1; sp < p.splits; ++sp)
        v = __fadd_rn(v, __ldcg(wst + ((size_t)sp * kLinRows + lr) * MP + m));
      T[lr * TS + m] = v;
    }
    if (tid == 0) p.counters[tile] = 0;  // ready for the next launch
  }
  named_sync(1, nthr);

  if (EPI == EPI_QKV)
    epilogue_qkv(p, tile, T, TS, s_rstd);
  else if (EPI == EPI_RESID)
    epilogue_resid(p, tile, T, TS);
  else if (EPI == EPI_GLU)
    epilogue_glu(p, tile, T, TS);
  else
    epilogue_logits(p, tile, T, TS);
}

template <int MT, int EPI, bool NORM>
cudaError_t launch_t(const LinearDesc& d, const LinParams& p, cudaStream_t s, bool pdl) {
  const size_t smem = linear_smem_bytes(MT, d.Kc);
  auto kern = k_linear<MT, EPI, NORM>;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(d.n_tiles * d.splits);
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
                              (int)linear_smem_bytes(MT, kLinKcMax));
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

size_t linear_smem_bytes(int mt, int Kc) {
  size_t b = 1024;  // alignment slack
  b += (size_t)kLinStages * kLinStageBytes;
  b += (size_t)mt * 8 * (Kc + 8) * sizeof(bf16);
  b += 2 * kLinStages * sizeof(uint64_t) + 64 * sizeof(float) + 16;
  size_t tile_bytes = (size_t)kLinRows * (mt * 8 + 1) * sizeof(float);
  if (tile_bytes > (size_t)kLinStages * kLinStageBytes) b += tile_bytes;  // never for mt <= 4
  return b;
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
