// sv_noalloc.cu -- the LM-head step (final RMSNorm, logits, greedy argmax)
// for callers that may not allocate device memory.
//
// Who needs it: code that runs inside a process whose device memory is owned
// by someone else -- a serving runtime that reserves the GPU's memory up front
// for its own pool, or a plugin invoked by such a runtime -- where a
// cudaMalloc either fails or carves memory out from under the owner, and
// latency-critical callers that cannot afford the implicit device
// synchronisation a cudaMalloc/cudaFree may cause.  The context API needs
// buffers from sv_create; this one call needs none beyond its own inputs and
// outputs.
//
// The split-tile partial slots (one per CTA, each value a tagged 64-bit word),
// the per-tile argmax partials, the row sums of squares and the kernels'
// status word live in one file-scope device array of kNoAllocScratchBytes.
// Every GPU that loads the library keeps that array until the process exits.
#include <mutex>

#include "sv_internal.h"
#include "sv_ptx.cuh"

namespace sv {
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(8) << 20;  // 8 MiB
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Per-device set-up: the array's device address (host code only sees a
// host-side stand-in for the symbol) and the kernels' shared-memory limits.
struct DeviceSetup {
  void* base = nullptr;
  bool ready = false;
};
std::mutex g_setup_mu;
DeviceSetup g_setup[kMaxDevices];

// Sum of squares of each 128-column tile of each row, reduced in the same
// order as the embedding kernel does for the context path.
__global__ void __launch_bounds__(128) k_rows_ss(const bf16* __restrict__ x, int hidden,
                                                 float* __restrict__ x_ss, int ss_tiles) {
  const int t = blockIdx.x, m = blockIdx.y, i = threadIdx.x;
  const float f = __bfloat162float(x[(size_t)m * hidden + t * 128 + i]);
  float ss = __fmul_rn(f, f);
  for (int o = 16; o > 0; o >>= 1) ss = __fadd_rn(ss, __shfl_xor_sync(0xffffffffu, ss, o));
  __shared__ float part[4];
  if ((i & 31) == 0) part[i >> 5] = ss;
  __syncthreads();
  if (i == 0)
    x_ss[m * ss_tiles + t] = __fadd_rn(__fadd_rn(part[0], part[1]), __fadd_rn(part[2], part[3]));
}

// Row argmax over the per-tile partials (largest value, lowest id on ties),
// and the status word of the call.
__global__ void __launch_bounds__(256) k_rows_argmax(const float* __restrict__ am_val,
                                                     const int* __restrict__ am_idx, int n_tiles,
                                                     int M, int32_t* out, const SvState* st,
                                                     int32_t* status_out) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
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
    if (lane == 0 && out) out[r] = bidx;
  }
  if (threadIdx.x == 0 && status_out) *status_out = st->status;
}

size_t round256(size_t b) { return (b + 255) & ~size_t(255); }

}  // namespace
}  // namespace sv

using namespace sv;

extern "C" int sv_lm_head_noalloc(const void* x_dev, const void* gain_dev, const void* w_dev, int M,
                                  int hidden, int vocab, float eps, float* logits_dev,
                                  int32_t* argmax_dev, int32_t* status_dev, void* cuda_stream) {
  if (!x_dev || !gain_dev || !w_dev || M < 1 || M > kMaxK || hidden <= 0 || hidden % 128 ||
      vocab < 1)
    return SV_E_INVAL;
  const uintptr_t misaligned = (reinterpret_cast<uintptr_t>(x_dev) | reinterpret_cast<uintptr_t>(gain_dev) |
                                reinterpret_cast<uintptr_t>(w_dev)) & 15u;
  if (misaligned) return SV_E_INVAL;

  // Where each piece of scratch goes, and whether it fits.
  const int n_tiles = (vocab + kLinRows - 1) / kLinRows;
  int dev = 0, num_sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SV_E_CUDA;
  if (cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return SV_E_CUDA;
  // the same partition of the K dimension as the context's LM head
  int grid = 1, max_seg = 1;
  linear_partition(n_tiles, hidden, num_sms, &grid, &max_seg);
  if (max_seg > kLinMaxSeg) return SV_E_INVAL;
  const int mp = M <= 8 ? 8 : (M <= 16 ? 16 : 32);
  const size_t off_state = 0;
  const size_t off_ss = round256(off_state + sizeof(SvState));
  const size_t off_amv = round256(off_ss + sizeof(float) * (size_t)M * (hidden / 128));
  const size_t off_ami = round256(off_amv + sizeof(float) * (size_t)M * n_tiles);
  const size_t off_ws = round256(off_ami + sizeof(int) * (size_t)M * n_tiles);
  const size_t ws_bytes = max_seg > 1 ? sizeof(uint32_t) * (size_t)grid * kLinRows * mp : 0;
  const size_t end = off_ws + ws_bytes;
  if (end > kNoAllocScratchBytes) return SV_E_NOMEM;  // larger than the fixed array

  {
    std::lock_guard<std::mutex> lock(g_setup_mu);
    DeviceSetup& ds = g_setup[dev];
    if (!ds.ready) {
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return SV_E_CUDA;
      if (prepare_linear_kernels() != cudaSuccess) return SV_E_CUDA;
      ds.base = p;
      ds.ready = true;
    }
  }
  unsigned char* base = static_cast<unsigned char*>(g_setup[dev].base);
  SvState* st = reinterpret_cast<SvState*>(base + off_state);
  float* x_ss = reinterpret_cast<float*>(base + off_ss);
  float* am_val = reinterpret_cast<float*>(base + off_amv);
  int* am_idx = reinterpret_cast<int*>(base + off_ami);
  uint32_t* ws = reinterpret_cast<uint32_t*>(base + off_ws);

  // Tensor map of the weight: a host-side encoding (the driver's encoder is
  // looked up once per process), no device memory.
  LinearDesc d;
  d.N = vocab;
  d.Kd = hidden;
  d.n_tiles = n_tiles;
  d.grid = grid;
  d.max_seg = max_seg;
  d.map_kind = MAP_PLAIN;
  if (!make_bf16_map(&d.map, w_dev, (uint64_t)vocab, (uint64_t)hidden, 64)) return SV_E_CUDA;

  cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
  // The status word starts at zero and every split-tile partial slot empty
  // (0xff bytes; a call that stopped early could have left words written).
  if (cudaMemsetAsync(st, 0, sizeof(SvState), s) != cudaSuccess ||
      (ws_bytes > 0 && cudaMemsetAsync(ws, 0xff, ws_bytes, s) != cudaSuccess))
    return SV_E_CUDA;
  k_rows_ss<<<dim3(hidden / 128, M), 128, 0, s>>>(static_cast<const bf16*>(x_dev), hidden, x_ss,
                                                  hidden / 128);
  if (cudaGetLastError() != cudaSuccess) return SV_E_CUDA;

  LinParams p = {};
  p.X = static_cast<const bf16*>(x_dev);
  p.x_ss = x_ss;
  p.gain = static_cast<const bf16*>(gain_dev);
  p.ss_tiles = hidden / 128;
  p.eps = eps;
  p.M = M;
  p.Kd = hidden;
  p.n_tiles = n_tiles;
  p.max_seg = max_seg;
  p.grid = grid;
  p.map = MAP_PLAIN;
  p.ws = ws;
  p.logits = logits_dev;
  p.logits_row0 = 0;
  p.am_val = am_val;
  p.am_idx = am_idx;
  p.vocab = vocab;
  p.st = st;
  if (launch_linear(d, p, EPI_LOGITS, true, s, false) != cudaSuccess) return SV_E_CUDA;
  k_rows_argmax<<<1, 256, 0, s>>>(am_val, am_idx, n_tiles, M, argmax_dev, st, status_dev);
  if (cudaGetLastError() != cudaSuccess) return SV_E_CUDA;
  return SV_OK;
}
