// k_misc.cu -- the small kernels of a step: embedding gather, the
// argmax + accept + truncate kernel, and cache housekeeping.
#include "misc_dev.cuh"

namespace sv {

namespace {

// x[m, :] = E[token_m, :]; x_ss[m, t] = sum of squares of x[m, 128t .. 128t+127].
// Also opens the step: step_pos = seq_len, and for a verify step (check) notes
// whether tokens[0] differs from the pending greedy token, in which case the
// accept kernel commits nothing.
__global__ void __launch_bounds__(128) k_embed(const bf16* __restrict__ E, int hidden, int vocab,
                                               bf16* __restrict__ x, float* __restrict__ x_ss,
                                               int ss_tiles, SvState* st, int check, StepIo io) {
  pdl_trigger();
  __shared__ float part[4];
  const int t = blockIdx.x, m = blockIdx.y, i = threadIdx.x;
  if (t == 0 && m == 0 && i == 0) {
    st->step_pos = st->seq_len;
    const int pending = st->pending;
    const int tok0 = io.tokens ? io.tokens[0] : st->tokens[0];
    st->step_reject = (check && pending >= 0 && tok0 != pending) ? 1 : 0;
  }
  embed_tile(E, hidden, vocab, x, x_ss, ss_tiles, st, m, t, i, part, 3, io.tokens);
  // Launched as a dependent of the delayed write-through window copy, which
  // touches none of the above, this kernel ends only after the copy has: the
  // step's later kernels wait for this one.  (No-op otherwise.)
  pdl_wait();
}

// Acceptance for the whole step; CTA l zeroes the rejected rows of layer l.
__global__ void __launch_bounds__(256) k_accept(SvState* st, const float* __restrict__ am_val,
                                                const int* __restrict__ am_idx, int n_tiles, int M,
                                                int mode, bf16* kpool, bf16* vpool,
                                                size_t layer_stride, const int* block_table,
                                                int n_layers, int n_kv_heads, int head_dim, KvDelay dl,
                                                StepIo io) {
  pdl_trigger();
  pdl_wait();
  __shared__ int s_am[kMaxK];
  __shared__ int s_n;
  accept_work(st, am_val, am_idx, n_tiles, M, mode, kpool, vpool, layer_stride, block_table,
              n_layers, n_kv_heads, head_dim, dl, blockIdx.x, gridDim.x, s_am, &s_n, io.result);
}

// Delayed write-through: before a verify step of M rows at pos = seq_len,
// map its window's logical pages (those that hold a physical page: below
// cap_len) to the scratch pages in the shadow table and copy the real pages
// there (positions past the length are zero in the real pages), 16 bytes per
// thread-iteration.
__global__ void k_kv_window_in(bf16* kpool, bf16* vpool, size_t layer_stride, const int* block_table,
                               KvDelay dl, const SvState* st, int n_layers, int n_kv_heads, int head_dim,
                               int M) {
  pdl_trigger();  // the embedding gather runs beside the copy
  const int pos = st->seq_len, cap = st->cap_len;
  const int lp0 = pos / kPage;
  const int lp_last = min(min(dl.bt_len, (cap + kPage - 1) / kPage) - 1, (pos + M - 1) / kPage);
  const int npg = lp_last - lp0 + 1;  // at most kWinPages; none when the window has no page
  if (npg <= 0) return;
  if (blockIdx.x == 0 && (int)threadIdx.x < npg) dl.bt_shadow[lp0 + threadIdx.x] = dl.win0 + threadIdx.x;
  const size_t pv = (size_t)n_kv_heads * kPage * head_dim / 8;  // 16-byte vectors per page
  const size_t n = (size_t)n_layers * npg * pv;
  for (size_t e = (size_t)blockIdx.x * blockDim.x + threadIdx.x; e < n; e += (size_t)gridDim.x * blockDim.x) {
    const int l = (int)(e / (npg * pv));
    const size_t r = e % (npg * pv);
    const int t = (int)(r / pv);
    const size_t w = r % pv;
    const int real = block_table[lp0 + t];
    uint4* kd = reinterpret_cast<uint4*>(kpool + (size_t)l * layer_stride) + (size_t)(dl.win0 + t) * pv + w;
    uint4* vd = reinterpret_cast<uint4*>(vpool + (size_t)l * layer_stride) + (size_t)(dl.win0 + t) * pv + w;
    uint4 kv = make_uint4(0u, 0u, 0u, 0u), vv = kv;
    if (real >= 0 && real < dl.win0) {
      kv = reinterpret_cast<const uint4*>(kpool + (size_t)l * layer_stride)[(size_t)real * pv + w];
      vv = reinterpret_cast<const uint4*>(vpool + (size_t)l * layer_stride)[(size_t)real * pv + w];
    }
    *kd = kv;
    *vd = vv;
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

__global__ void k_set_len(SvState* st, int len, int cap_len, int pending) {
  st->seq_len = len;
  st->step_pos = len;
  if (cap_len >= 0) st->cap_len = cap_len;
  if (pending != kKeepPending) st->pending = pending;
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
                         SvState* st, bool check, cudaStream_t s, bool pdl, const StepIo& io) {
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = make_cfg(dim3(hidden / 128, M), dim3(128), s, attr, pdl);
  return cudaLaunchKernelEx(&cfg, k_embed, E, hidden, vocab, x, x_ss, hidden / 128, st, check ? 1 : 0, io);
}

cudaError_t launch_accept(SvState* st, const float* am_val, const int* am_idx, int n_tiles, int M,
                          int mode, bf16* kpool, bf16* vpool, size_t layer_stride,
                          const int* block_table, int n_layers, int n_kv_heads, int head_dim,
                          const KvDelay& dl, cudaStream_t s, bool pdl, const StepIo& io) {
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = make_cfg(dim3(n_layers > 0 ? n_layers : 1), dim3(256), s, attr, pdl);
  return cudaLaunchKernelEx(&cfg, k_accept, st, am_val, am_idx, n_tiles, M, mode, kpool, vpool,
                            layer_stride, block_table, n_layers, n_kv_heads, head_dim, dl, io);
}

namespace {
template <typename... A>
constexpr int n_params(void (*)(A...)) {
  return (int)sizeof...(A);
}
}  // namespace

bool step_io_node(cudaGraphNode_t node) {
  cudaGraphNodeType type;
  cudaKernelNodeParams kp;
  if (cudaGraphNodeGetType(node, &type) != cudaSuccess || type != cudaGraphNodeTypeKernel ||
      cudaGraphKernelNodeGetParams(node, &kp) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return kp.func == reinterpret_cast<void*>(k_embed) || kp.func == reinterpret_cast<void*>(k_accept);
}

// The captured argument list with its last entry (the StepIo of both
// kernels) replaced.
cudaError_t set_step_io(cudaGraphExec_t exec, cudaGraphNode_t node, const StepIo& io) {
  cudaKernelNodeParams kp;
  cudaError_t e = cudaGraphKernelNodeGetParams(node, &kp);
  if (e != cudaSuccess) return e;
  constexpr int kEmbed = n_params(k_embed), kAccept = n_params(k_accept);
  constexpr int kMax = kEmbed > kAccept ? kEmbed : kAccept;
  int n;
  if (kp.func == reinterpret_cast<void*>(k_embed))
    n = kEmbed;
  else if (kp.func == reinterpret_cast<void*>(k_accept))
    n = kAccept;
  else
    return cudaErrorInvalidValue;
  if (kp.kernelParams == nullptr || kp.extra != nullptr) return cudaErrorNotSupported;
  // the node as captured: the state block's tokens and result
  const StepIo* captured = static_cast<const StepIo*>(kp.kernelParams[n - 1]);
  if (captured == nullptr || captured->tokens != nullptr || captured->result != nullptr)
    return cudaErrorInvalidValue;
  void* args[kMax];
  for (int i = 0; i < n - 1; ++i) args[i] = kp.kernelParams[i];
  StepIo v = io;
  args[n - 1] = &v;
  kp.kernelParams = args;
  return cudaGraphExecKernelNodeSetParams(exec, node, &kp);
}

cudaError_t launch_kv_window_in(bf16* kpool, bf16* vpool, size_t layer_stride, const int* block_table,
                                const KvDelay& dl, const SvState* st, int n_layers, int n_kv_heads,
                                int head_dim, int M, cudaStream_t s) {
  if (n_layers <= 0) return cudaSuccess;
  k_kv_window_in<<<608, 256, 0, s>>>(kpool, vpool, layer_stride, block_table, dl, st, n_layers, n_kv_heads,
                                      head_dim, M);
  return cudaGetLastError();
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

cudaError_t launch_set_len(SvState* st, int len, int cap_len, int pending, cudaStream_t s) {
  k_set_len<<<1, 1, 0, s>>>(st, len, cap_len, pending);
  return cudaGetLastError();
}

}  // namespace sv
