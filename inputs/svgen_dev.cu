// svgen_dev.cu -- device bulk fill of the seeded synthetic inputs.
// Same definition as the host fill in svgen.c (both include svgen.h), used
// to materialise multi-GB weight sets directly in device memory.
#include <cuda_runtime.h>
#include <stdint.h>

#include "svgen.h"

__global__ void svg_fill_kernel(uint16_t* __restrict__ out, uint64_t n, uint64_t stream, double stdv,
                                int kind) {
  uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
  for (uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
    uint16_t v;
    if (kind == 0)
      v = svg_weight_bf16(stream, i, stdv);
    else if (kind == 1)
      v = svg_gain_bf16(stream, i, stdv);
    else
      v = 0x3F80u;
    out[i] = v;
  }
}

// kind: 0 weight (z * stdv), 1 gain (1 + z * stdv; stdv == 0 gives ones).
// Returns 0 or the CUDA error code of the launch.
extern "C" int svg_dev_fill(void* out_dev, uint64_t n, uint64_t seed, uint64_t tensor_id, double stdv,
                            int kind, void* stream) {
  if (n == 0) return 0;
  if (kind == 1 && stdv == 0.0) kind = 2;
  int blocks = 152 * 8;
  svg_fill_kernel<<<blocks, 256, 0, (cudaStream_t)stream>>>((uint16_t*)out_dev, n,
                                                            svg_stream(seed, tensor_id), stdv, kind);
  return (int)cudaGetLastError();
}
