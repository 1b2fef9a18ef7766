// k_misc.cu -- the small kernels of a step: embedding gather, the
// argmax + accept + truncate kernel, and cache housekeeping.
#include "sv_internal.h"
#include "sv_ptx.cuh"

namespace sv {

namespace {

// x[m, :] = E[token_m, :]; x_ss[m, t] = sum of squares of x[m, 128t .. 128t+127].
// Also opens the step: step_pos = seq_len.
__global__ void __launch_bounds__(128) k_embed(const bf16* __restrict__ E, int hidden, int vocab,
                                               bf16* __restrict__ x, float* __restrict__ x_ss,
                                               int ss_tiles, SvState* st) {
  pdl_trigger();
  const int t = blockIdx.x, m = blockIdx.y, i = threadIdx.x;
  if (t == 0 && m == 0 && i == 0) st->step_pos = st->seq_len;
  int tok = st->tokens[m];
  if (tok < 0 || tok >= vocab) {
    if (i == 0) atomicOr(&st->status, ST_BAD_TOKEN);
    tok = 0;
  }
  const int col = t * 128 + i;
  const bf16 v = E[(size_t)tok * hidden + col];
  x[(size_t)m * hidden + col] = v;
  float f = __bfloat162float(v);
  float ss = __fmul_rn(f, f);
  for (int o = 16; o > 0; o >>= 1) ss = __fadd_rn(ss, __shfl_xor_sync(0xffffffffu, ss, o));
  __shared__ float part[4];
  if ((i & 31) == 0) part[i >> 5] = ss;
  __syncthreads();
  if (i == 0)
    x_ss[m * ss_tiles + t] = __fadd_rn(__fadd_rn(part[0], part[1]), __fadd_rn(part[2], part[3]));
}

// Greedy argmax of each row from the LM head's per-tile partials (largest
// value, lowest id on ties), then acceptance: n = number of leading drafts
// tokens[j+1] equal to argmax[j]; the row count committed is n + 1; rejected
// window slots are zeroed in every layer (CTA l zeroes layer l).
__global__ void __launch_bounds__(256) k_accept(SvState* st, const float* __restrict__ am_val,
                                                const int* __restrict__ am_idx, int n_tiles, int M,
                                                int mode, bf16* kpool, bf16* vpool,
                                                size_t layer_stride, const int* block_table,
                                                int n_layers, int n_kv_heads, int head_dim) {
  pdl_trigger();
  pdl_wait();
  __shared__ int s_am[kMaxK];
  __shared__ int s_n;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int pos = st->step_pos;
  if (mode == MODE_BODY) {
    if (blockIdx.x == 0 && tid == 0) {
      st->seq_len = pos + M;
      st->result[0] = M - 1;
      st->result[1] = -1;
      st->result[2] = pos + M;
      st->result[3] = st->status;
    }
    return;
  }
  for (int r = warp; r < M; r += 8) {
    float best = -INFINITY;
    int bidx = 0x7fffffff;
    for (int t = lane; t < n_tiles; t += 32) {
      const float v = am_val[r * n_tiles + t];
      const int id = am_idx[r * n_tiles + t];
      if (bidx == 0x7fffffff || v > best || (v == best && id < bidx)) {
        best = v;
        bidx = id;
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
  __syncthreads();
  if (tid == 0) {
    int n = M - 1;
    if (mode == MODE_VERIFY) {
      n = 0;
      while (n < M - 1 && st->tokens[n + 1] == s_am[n]) ++n;
    }
    s_n = n;
  }
  __syncthreads();
  const int n = s_n;
  const int new_len = pos + 1 + n;
  if (blockIdx.x == 0 && tid == 0) {
    for (int r = 0; r < M; ++r) st->argmax[r] = s_am[r];
    st->seq_len = new_len;
    st->result[0] = n;
    st->result[1] = s_am[n];
    st->result[2] = new_len;
    st->result[3] = st->status;
  }
  // zero the K/V of rejected rows (positions new_len .. pos + M - 1) of layer blockIdx.x
  const int l = blockIdx.x;
  if (l >= n_layers) return;
  const int row = n_kv_heads * head_dim;
  for (int e = tid; e < (pos + M - new_len) * row; e += blockDim.x) {
    const int ps = new_len + e / row, hi = e % row;
    const int page = block_table[ps / kPage];
    if (page < 0) continue;
    const int h = hi / head_dim, i = hi % head_dim;
    const size_t idx = (size_t)l * layer_stride +
                       (((size_t)page * n_kv_heads + h) * kPage + ps % kPage) * head_dim + i;
    kpool[idx] = __float2bfloat16_rn(0.0f);
    vpool[idx] = __float2bfloat16_rn(0.0f);
  }
}

// cos/sin of pos * theta^(-2i/d), taken in double and rounded to fp32.
__global__ void k_rope_table(float2* tab, int max_seq, int head_dim, float theta) {
  const int half = head_dim / 2;
  const size_t n = (size_t)max_seq * half;
  for (size_t e = (size_t)blockIdx.x * blockDim.x + threadIdx.x; e < n;
       e += (size_t)gridDim.x * blockDim.x) {
    const int ps = (int)(e / half), i = (int)(e % half);
    const double inv = pow((double)theta, -2.0 * (double)i / (double)head_dim);
    const double ang = (double)ps * inv;
    double s, c;
    sincos(ang, &s, &c);
    tab[e] = make_float2((float)c, (float)s);
  }
}

__global__ void k_kv_zero(bf16* kpool, bf16* vpool, size_t layer_stride, const int* block_table,
                          int n_layers, int n_kv_heads, int head_dim, int first, int last) {
  const size_t row = (size_t)n_kv_heads * head_dim;
  const size_t n = (size_t)n_layers * (last - first) * row;
  for (size_t e = (size_t)blockIdx.x * blockDim.x + threadIdx.x; e < n;
       e += (size_t)gridDim.x * blockDim.x) {
    const size_t per_layer = (size_t)(last - first) * row;
    const int l = (int)(e / per_layer);
    const size_t r = e % per_layer;
    const int ps = first + (int)(r / row);
    const int hi = (int)(r % row);
    const int page = block_table[ps / kPage];
    if (page < 0) continue;
    const int h = hi / head_dim, i = hi % head_dim;
    const size_t idx = (size_t)l * layer_stride +
                       (((size_t)page * n_kv_heads + h) * kPage + ps % kPage) * head_dim + i;
    kpool[idx] = __float2bfloat16_rn(0.0f);
    vpool[idx] = __float2bfloat16_rn(0.0f);
  }
}

__global__ void k_kv_gather(const bf16* kpool, const bf16* vpool, size_t layer_stride,
                            const int* block_table, int layer, int n_kv_heads, int head_dim,
                            int first, int count, bf16* kdst, bf16* vdst) {
  const size_t row = (size_t)n_kv_heads * head_dim;
  const size_t n = (size_t)count * row;
  for (size_t e = (size_t)blockIdx.x * blockDim.x + threadIdx.x; e < n;
       e += (size_t)gridDim.x * blockDim.x) {
    const int ps = first + (int)(e / row);
    const int hi = (int)(e % row);
    const int page = block_table[ps / kPage];
    const int h = hi / head_dim, i = hi % head_dim;
    bf16 kv = __float2bfloat16_rn(0.0f), vv = kv;
    if (page >= 0) {
      const size_t idx = (size_t)layer * layer_stride +
                         (((size_t)page * n_kv_heads + h) * kPage + ps % kPage) * head_dim + i;
      kv = kpool[idx];
      vv = vpool[idx];
    }
    kdst[e] = kv;
    vdst[e] = vv;
  }
}

__global__ void k_set_len(SvState* st, int len, int cap_len) {
  st->seq_len = len;
  st->step_pos = len;
  if (cap_len >= 0) st->cap_len = cap_len;
}

cudaLaunchConfig_t make_cfg(dim3 grid, dim3 block, cudaStream_t s, cudaLaunchAttribute* attr,
                            bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.stream = s;
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cfg;
}

}  // namespace

cudaError_t launch_embed(const bf16* E, int hidden, int vocab, int M, bf16* x, float* x_ss,
                         SvState* st, cudaStream_t s) {
  k_embed<<<dim3(hidden / 128, M), 128, 0, s>>>(E, hidden, vocab, x, x_ss, hidden / 128, st);
  return cudaGetLastError();
}

cudaError_t launch_accept(SvState* st, const float* am_val, const int* am_idx, int n_tiles, int M,
                          int mode, bf16* kpool, bf16* vpool, size_t layer_stride,
                          const int* block_table, int n_layers, int n_kv_heads, int head_dim,
                          cudaStream_t s, bool pdl) {
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = make_cfg(dim3(n_layers > 0 ? n_layers : 1), dim3(256), s, attr, pdl);
  return cudaLaunchKernelEx(&cfg, k_accept, st, am_val, am_idx, n_tiles, M, mode, kpool, vpool,
                            layer_stride, block_table, n_layers, n_kv_heads, head_dim);
}

cudaError_t launch_rope_table(float2* tab, int max_seq, int head_dim, float theta, cudaStream_t s) {
  k_rope_table<<<1024, 256, 0, s>>>(tab, max_seq, head_dim, theta);
  return cudaGetLastError();
}

cudaError_t launch_kv_zero(bf16* kpool, bf16* vpool, size_t layer_stride, const int* block_table,
                           int n_layers, int n_kv_heads, int head_dim, int first, int last,
                           cudaStream_t s) {
  if (last <= first || n_layers <= 0) return cudaSuccess;
  k_kv_zero<<<1024, 256, 0, s>>>(kpool, vpool, layer_stride, block_table, n_layers, n_kv_heads,
                                 head_dim, first, last);
  return cudaGetLastError();
}

cudaError_t launch_kv_gather(const bf16* kpool, const bf16* vpool, size_t layer_stride,
                             const int* block_table, int layer, int n_kv_heads, int head_dim,
                             int first, int count, bf16* kdst, bf16* vdst, cudaStream_t s) {
  if (count <= 0) return cudaSuccess;
  k_kv_gather<<<256, 256, 0, s>>>(kpool, vpool, layer_stride, block_table, layer, n_kv_heads,
                                  head_dim, first, count, kdst, vdst);
  return cudaGetLastError();
}

cudaError_t launch_set_len(SvState* st, int len, int cap_len, cudaStream_t s) {
  k_set_len<<<1, 1, 0, s>>>(st, len, cap_len);
  return cudaGetLastError();
}

}  // namespace sv
