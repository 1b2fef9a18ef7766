// k_linear.cu -- the batch-invariant linear: Y[m, n] = sum_k X[m, k] W[n, k]
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
#include "lin_dev.cuh"

namespace sv {
namespace {

// Persistent stream-K linear.  The n_tiles x (Kd/64) k-blocks of the weight,
// tile-major, are cut into gridDim.x equal contiguous ranges, one per CTA.
// A tile whose k-blocks all fall in one CTA is finished there; a tile cut by
// range boundaries is finished by the last of its CTAs to arrive, which sums
// the per-CTA partials in k order.  The partition depends only on the weight
// shape and the grid (one CTA per SM), never on M.
template <int MT, int EPI, bool NORM, int SB>
__global__ void __launch_bounds__(kLinThreads, 1)
    k_linear(const __grid_constant__ CUtensorMap wmap, const __grid_constant__ CUtensorMap pfmap,
             const LinParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const LinSmem sm = lin_smem<MT>(smem);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int s = 0; s < kLinStages; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], kLinConsumerWarps);
    }
    mbar_init(sm.xbar, 1);
    mbar_init(sm.gbar, 1);
    fence_barrier_init();
  }
  __syncthreads();
  // Let the next kernel in the stream start its own weight prefetch.
  pdl_trigger();
  int it = 0;
  if (warp == kLinConsumerWarps) {  // producer: weights do not depend on earlier kernels
    if (lane == 0) {
      prefetch_tensormap(&wmap);
      if (!lin_produce<LinGeom<MT>::kStages>(p, &wmap, blockIdx.x, gridDim.x, sm, it, policy_evict_first()))
        atomicOr(&p.st->status, ST_TIMEOUT);
      else
        lin_prefetch_next(p, &pfmap, blockIdx.x);
    }
    return;
  }
  // (the consumers wait for the previous kernel inside, after the work that does not need it)
  if (!lin_consume<MT, EPI, NORM, SB>(p, blockIdx.x, gridDim.x, sm, it) && lane == 0)
    atomicOr(&p.st->status, ST_TIMEOUT);
}

template <int MT, int EPI, bool NORM, int SB>
cudaError_t launch_t(const LinearDesc& d, const LinParams& p, cudaStream_t s, bool pdl,
                     const CUtensorMap& pfmap) {
  const size_t smem = linear_smem_bytes(MT);
  auto kern = k_linear<MT, EPI, NORM, SB>;
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
  return cudaLaunchKernelEx(&cfg, kern, d.map, pfmap, p);
}

template <int MT, int EPI, bool NORM, int SB>
cudaError_t prepare_t() {
  return cudaFuncSetAttribute(k_linear<MT, EPI, NORM, SB>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)linear_smem_bytes(MT));
}

template <int MT, int SB>
cudaError_t prepare_sb() {
  cudaError_t e;
  if ((e = prepare_t<MT, EPI_QKV, true, SB>()) != cudaSuccess) return e;
  if ((e = prepare_t<MT, EPI_RESID, false, SB>()) != cudaSuccess) return e;
  if ((e = prepare_t<MT, EPI_GLU, true, SB>()) != cudaSuccess) return e;
  return prepare_t<MT, EPI_LOGITS, true, SB>();
}

template <int MT, int SB>
cudaError_t launch_sb(const LinearDesc& d, const LinParams& p, int epi, bool norm, cudaStream_t s,
                      bool pdl, const CUtensorMap& pf) {
  switch (epi) {
    case EPI_QKV:
      return norm ? launch_t<MT, EPI_QKV, true, SB>(d, p, s, pdl, pf) : cudaErrorInvalidValue;
    case EPI_RESID:
      return norm ? cudaErrorInvalidValue : launch_t<MT, EPI_RESID, false, SB>(d, p, s, pdl, pf);
    case EPI_GLU:
      return norm ? launch_t<MT, EPI_GLU, true, SB>(d, p, s, pdl, pf) : cudaErrorInvalidValue;
    case EPI_LOGITS:
      return norm ? launch_t<MT, EPI_LOGITS, true, SB>(d, p, s, pdl, pf) : cudaErrorInvalidValue;
  }
  return cudaErrorInvalidValue;
}

template <int MT>
cudaError_t prepare_mt() {
  return prepare_sb<MT, lin_seg_batch(MT, kLinMaxSeg)>();
}

template <int MT>
cudaError_t launch_mt(const LinearDesc& d, const LinParams& p, int epi, bool norm, cudaStream_t s,
                      bool pdl, const CUtensorMap& pf) {
  return launch_sb<MT, lin_seg_batch(MT, kLinMaxSeg)>(d, p, epi, norm, s, pdl, pf);
}

}  // namespace

size_t linear_smem_bytes(int mt) {
  const int mp = mt * 8;
  const int xc = mt == 2 ? LinGeom<2>::kXCols : (mt == 4 ? LinGeom<4>::kXCols : LinGeom<1>::kXCols);
  const int stages = mt == 2 ? LinGeom<2>::kStages : (mt == 4 ? LinGeom<4>::kStages : LinGeom<1>::kStages);
  size_t b = 1024;  // alignment slack
  b += (size_t)stages * kLinStageBytes;
  b += (size_t)mp * (xc + 8) * sizeof(bf16);
  b += ((size_t)kLinRows * (mp + 1) * sizeof(float) + 15) & ~size_t(15);
  b += (size_t)kLinXCols * sizeof(bf16);  // gain window
  b += (2 * kLinStages + 2) * sizeof(uint64_t) + (kMaxK + 64) * sizeof(float) + 16;
  return b;
}

namespace {

// One 16-byte unit per thread-iteration: unit u of row r of chunk ch of block
// blk (= tile * KB + kk) goes to granule u ^ (r mod 8) of that row.
__global__ void k_tile_weight(const bf16* __restrict__ w, int N, int Kd, int n_tiles, int map_kind, int ffn,
                              uint8_t* __restrict__ out) {
  const int KB = Kd / kLinBK;
  const size_t units = (size_t)n_tiles * KB * 1024;
  for (size_t e = (size_t)blockIdx.x * blockDim.x + threadIdx.x; e < units; e += (size_t)gridDim.x * blockDim.x) {
    const int u = (int)(e & 7), r = (int)((e >> 3) & 63), ch = (int)((e >> 9) & 1);
    const size_t blk = e >> 10;
    const int tile = (int)(blk / KB), kk = (int)(blk % KB);
    const TileRows tr = tile_rows_of(map_kind, ffn, tile);
    const int row = (ch == 0 ? tr.a0 : tr.b0) + r;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (row < N) v = __ldg(reinterpret_cast<const uint4*>(w + (size_t)row * Kd + kk * kLinBK + u * 8));
    *reinterpret_cast<uint4*>(out + blk * kLinStageBytes + ch * kLinChunkBytes + r * 128 + ((u ^ (r & 7)) << 4)) = v;
  }
}

}  // namespace

cudaError_t launch_tile_weight(const bf16* w, int N, int Kd, int n_tiles, int map_kind, int ffn, uint8_t* out,
                               cudaStream_t s) {
  k_tile_weight<<<1024, 256, 0, s>>>(w, N, Kd, n_tiles, map_kind, ffn, out);
  return cudaGetLastError();
}

void linear_partition(int n_tiles, int Kd, int num_sms, int* grid, int* max_seg) {
  const long long KB = Kd / kLinBK, T = (long long)n_tiles * KB;
  const long long by_share = T / kLinMinShare > 0 ? T / kLinMinShare : 1;
  const int G = (int)(by_share < num_sms ? by_share : num_sms);
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
  if ((e = prepare_sb<1, 4>()) != cudaSuccess || (e = prepare_sb<1, 2>()) != cudaSuccess) return e;  // (prepare_mt<1>: the batch of 6)
  if ((e = prepare_mt<2>()) != cudaSuccess) return e;
  return prepare_mt<4>();
}

cudaError_t launch_linear(const LinearDesc& d, const LinParams& p_in, int epi, bool norm,
                          cudaStream_t s, bool pdl, const LinearDesc* next) {
  LinParams p = p_in;
  if (next) {
    p.pf_blocks = kLinPrefetchBlocks;
    p.pf_n_tiles = next->n_tiles;
    p.pf_Kd = next->Kd;
    p.pf_grid = next->grid;
    p.pf_map = next->map_kind;
    p.pf_ffn = next->N / 2;  // gate|up: the up rows start at ffn
    p.pf_wt = next->tiled;
  } else {
    p.pf_blocks = 0;
    p.pf_wt = nullptr;
  }
  const CUtensorMap& pf = next ? next->map : d.map;
  if (p.M <= 8)  // the gather batch of the weight's partition (the same for every M)
    return lin_seg_batch(1, d.max_seg) == 2 ? launch_sb<1, 2>(d, p, epi, norm, s, pdl, pf)
           : lin_seg_batch(1, d.max_seg) == 4 ? launch_sb<1, 4>(d, p, epi, norm, s, pdl, pf)
                                            : launch_sb<1, 6>(d, p, epi, norm, s, pdl, pf);
  if (p.M <= 16) return launch_mt<2>(d, p, epi, norm, s, pdl, pf);
  if (p.M <= 32) return launch_mt<4>(d, p, epi, norm, s, pdl, pf);
  return cudaErrorInvalidValue;
}

}  // namespace sv
