// k_attn.cu -- multi-row paged decode attention with per-row context lengths.
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
#include "attn_dev.cuh"

namespace sv {

namespace {

// kMulti: the form for grids whose CTAs run several work items (long
// contexts), which requests each CTA's next item while it merges this one.
template <int D, bool kMulti>
__global__ void __launch_bounds__(AttnCfg<D>::kThreads, 1)
    k_attention(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                const AttnParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  AttnSmem<D, kMulti> sm;
  sm.carve(smem);
  if (threadIdx.x == 0) attn_init_bars<D, kMulti>(sm);
  __syncthreads();
  pdl_trigger();
  // The committed length is final for the whole step (only the step's last
  // kernel, or the host between steps, changes it), so it may be read before
  // the wait on the previous kernel; attn_items waits once it has requested
  // the cache pages that earlier steps wrote.
  const int pos = __ldcg(&p.st->seq_len);
  uint32_t phase = 0;
  bool ok;
  if constexpr (kMulti)
    ok = attn_items_multi<D>(p, &kmap, &vmap, blockIdx.x, gridDim.x, sm, phase, pos);
  else
    ok = attn_items_single<D>(p, &kmap, &vmap, blockIdx.x, gridDim.x, sm, phase, pos);
  if (!ok && (threadIdx.x & 31) == 0)
    atomicOr(&p.st->status, ST_TIMEOUT);
}

// One block per (row, query head), one thread per element.  Contexts of at
// most kCombineChunk splits use this light form (few registers, so its blocks fit
// beside the attention kernel's and are resident before it ends).
template <int D>
__global__ void __launch_bounds__(D) k_attn_combine(const AttnParams p) {
  pdl_trigger();
  // The committed length is final for the whole step (only the step's last
  // kernel, or the host between steps, changes it) and equals the step's
  // start: read it before the wait, as the attention kernel does, so that
  // the partials' loads are the only round trip after it.
  const int pos = __ldcg(&p.st->seq_len);
  pdl_wait();
  combine_element<D>(p, blockIdx.x / p.n_q_heads, blockIdx.x % p.n_q_heads, threadIdx.x, pos);
}

// Longer contexts: rows of more than kCombineChunk splits take combine_long.
// Dynamic shared memory: the (m, l) pairs of up to max_splits splits.
// (Its register cap lets its blocks fit beside an attention block.)
template <int D>
__global__ void __launch_bounds__(D, 768 / D) k_attn_combine_long(const AttnParams p) {
  extern __shared__ float2 s_ml[];
  __shared__ float s_red[D / 32];
  pdl_trigger();
  const int pos = __ldcg(&p.st->seq_len);  // final for the whole step (see k_attn_combine)
  pdl_wait();
  const int r = blockIdx.x / p.n_q_heads, hq = blockIdx.x % p.n_q_heads;
  const int ns = attn_n_splits(pos + r + 1, D);  // splits row r sees
  if (ns <= kCombineChunk)
    combine_element<D>(p, r, hq, threadIdx.x, pos);
  else
    combine_long<D>(p, r, hq, ns, s_ml, s_red);
}

template <int D, bool kMulti>
cudaError_t launch_attn_t(const CUtensorMap& kmap, const CUtensorMap& vmap, const AttnParams& p,
                          int grid, cudaStream_t s, bool pdl) {
  const int smem = AttnSmem<D, kMulti>::kSmem;
  auto kern = k_attention<D, kMulti>;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(AttnCfg<D>::kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, kmap, vmap, p);
}

template <int D>
cudaError_t launch_comb_t(const AttnParams& p, cudaStream_t s, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.M * p.n_q_heads);
  cfg.blockDim = dim3(D);
  const bool long_ctx = p.max_splits > kCombineChunk;
  cfg.dynamicSmemBytes = long_ctx ? (size_t)p.max_splits * sizeof(float2) : 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return long_ctx ? cudaLaunchKernelEx(&cfg, k_attn_combine_long<D>, p)
                  : cudaLaunchKernelEx(&cfg, k_attn_combine<D>, p);
}


template <int D, bool kMulti>
cudaError_t prepare_attn_t() {
  cudaError_t e = cudaFuncSetAttribute(k_attention<D, kMulti>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       AttnSmem<D, kMulti>::kSmem);
  if (e != cudaSuccess || kMulti) return e;
  // the staged merge's (m, l) pairs: up to the splits of kMaxSeq positions
  return cudaFuncSetAttribute(k_attn_combine_long<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)(attn_n_splits(kMaxSeq, D) * sizeof(float2)));
}

}  // namespace

cudaError_t prepare_attention_kernels() {
  cudaError_t e;
  if ((e = prepare_attn_t<64, false>()) != cudaSuccess || (e = prepare_attn_t<64, true>()) != cudaSuccess ||
      (e = prepare_attn_t<128, false>()) != cudaSuccess || (e = prepare_attn_t<128, true>()) != cudaSuccess ||
      (e = prepare_attn_t<256, false>()) != cudaSuccess)
    return e;
  return prepare_attn_t<256, true>();
}

cudaError_t launch_attention(const CUtensorMap& kmap, const CUtensorMap& vmap, const AttnParams& p,
                             int head_dim, int grid, bool multi, cudaStream_t s, bool pdl) {
  switch (head_dim) {
    case 64:
      return multi ? launch_attn_t<64, true>(kmap, vmap, p, grid, s, pdl)
                   : launch_attn_t<64, false>(kmap, vmap, p, grid, s, pdl);
    case 128:
      return multi ? launch_attn_t<128, true>(kmap, vmap, p, grid, s, pdl)
                   : launch_attn_t<128, false>(kmap, vmap, p, grid, s, pdl);
    case 256:
      return multi ? launch_attn_t<256, true>(kmap, vmap, p, grid, s, pdl)
                   : launch_attn_t<256, false>(kmap, vmap, p, grid, s, pdl);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_attn_combine(const AttnParams& p, int head_dim, cudaStream_t s, bool pdl) {
  switch (head_dim) {
    case 64: return launch_comb_t<64>(p, s, pdl);
    case 128: return launch_comb_t<128>(p, s, pdl);
    case 256: return launch_comb_t<256>(p, s, pdl);
  }
  return cudaErrorInvalidValue;
}

}  // namespace sv
