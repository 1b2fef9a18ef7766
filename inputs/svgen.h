/* svgen.h -- seeded synthetic inputs shared by the CPU oracle and the GPU path.
 *
 * This module holds no arithmetic of the decoding method.  It only turns
 * (seed, tensor id, element index) into a bf16 bit pattern or a token id, so
 * that both sides of a parity test see exactly the same weights and prompts.
 *
 * Generator (counter-based, stateless):
 *   mix64(x)        = splitmix64 finaliser of x + 0x9E3779B97F4A7C15
 *   stream(s, t)    = mix64(mix64(s) ^ (t * 0xD1B54A32D192ED03))
 *   draw(st, c)     = mix64(st + c)
 *
 * Approximately normal values use the classic "sum of twelve uniforms"
 * method (Irwin-Hall, n = 12): element i takes draws 3i, 3i+1, 3i+2 of its
 * stream, splits each 64-bit draw into four 16-bit uniforms u_q, and forms
 *   z = (sum_q u_q + 6 - 6 * 65536) / 65536        (exact in double)
 * which has mean 0 and variance 1 (each (u + 1/2)/65536 is uniform on (0,1)).
 * A weight is bf16(float(z * std)); a norm gain is bf16(float(1 + z * std)).
 * Every step is integer arithmetic or a single correctly-rounded IEEE
 * operation, so a C host and a CUDA device implementation of this definition
 * produce identical bits by construction.
 *
 * Token ids: token i of stream st is draw(st, i) mod vocab.
 */
#ifndef SVGEN_H
#define SVGEN_H
#include <stdint.h>

#if defined(__CUDACC__)
#define SVG_FN static __host__ __device__ __forceinline__
#else
#define SVG_FN static inline
#endif

SVG_FN uint64_t svg_mix64(uint64_t x) {
  uint64_t z = x + 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

SVG_FN uint64_t svg_stream(uint64_t seed, uint64_t tensor_id) {
  return svg_mix64(svg_mix64(seed) ^ (tensor_id * 0xD1B54A32D192ED03ull));
}

SVG_FN uint64_t svg_draw(uint64_t stream, uint64_t counter) {
  return svg_mix64(stream + counter);
}

/* Sum of the twelve 16-bit uniforms of element i, in [0, 12 * 65535]. */
SVG_FN uint32_t svg_irwin_hall12(uint64_t stream, uint64_t i) {
  uint32_t acc = 0;
  for (int j = 0; j < 3; ++j) {
    uint64_t u = svg_draw(stream, 3u * i + (uint64_t)j);
    acc += (uint32_t)(u & 0xFFFFu) + (uint32_t)((u >> 16) & 0xFFFFu) +
           (uint32_t)((u >> 32) & 0xFFFFu) + (uint32_t)((u >> 48) & 0xFFFFu);
  }
  return acc;
}

/* float -> bf16 bits, round to nearest even; NaN maps to a quiet NaN. */
SVG_FN uint16_t svg_f32_to_bf16(float f) {
  union { float f; uint32_t u; } v;
  v.f = f;
  if ((v.u & 0x7F800000u) == 0x7F800000u && (v.u & 0x007FFFFFu) != 0u)
    return (uint16_t)((v.u >> 16) | 0x0040u);
  uint32_t r = v.u + 0x7FFFu + ((v.u >> 16) & 1u);
  return (uint16_t)(r >> 16);
}

/* z of element i as an exact double in [-6, 6). */
SVG_FN double svg_z(uint64_t stream, uint64_t i) {
  return ((double)svg_irwin_hall12(stream, i) + 6.0 - 393216.0) / 65536.0;
}

#if defined(__CUDA_ARCH__)
#define SVG_DMUL(a, b) __dmul_rn((a), (b))
#define SVG_DADD(a, b) __dadd_rn((a), (b))
#define SVG_D2F(a) __double2float_rn(a)
#else
#define SVG_DMUL(a, b) ((a) * (b))
#define SVG_DADD(a, b) ((a) + (b))
#define SVG_D2F(a) ((float)(a))
#endif

SVG_FN uint16_t svg_weight_bf16(uint64_t stream, uint64_t i, double stdv) {
  double w = SVG_DMUL(svg_z(stream, i), stdv);
  return svg_f32_to_bf16(SVG_D2F(w));
}

SVG_FN uint16_t svg_gain_bf16(uint64_t stream, uint64_t i, double stdv) {
  double w = SVG_DADD(1.0, SVG_DMUL(svg_z(stream, i), stdv));
  return svg_f32_to_bf16(SVG_D2F(w));
}

SVG_FN int32_t svg_token(uint64_t stream, uint64_t i, uint32_t vocab) {
  return (int32_t)(svg_draw(stream, i) % (uint64_t)vocab);
}

/* Tensor ids of a decoder's weights (one id space per model seed). */
enum {
  SVG_T_EMBED = 1,
  SVG_T_LM_HEAD = 2,
  SVG_T_FINAL_NORM = 3,
  SVG_T_LAYER_BASE = 100, /* + 16 * layer + one of the offsets below */
  SVG_T_ATTN_NORM = 0,
  SVG_T_WQKV = 1,
  SVG_T_Q_NORM = 2,
  SVG_T_K_NORM = 3,
  SVG_T_WO = 4,
  SVG_T_FFN_NORM = 5,
  SVG_T_W_GATE_UP = 6,
  SVG_T_W_DOWN = 7
};

SVG_FN uint64_t svg_layer_tensor(int layer, int which) {
  return (uint64_t)SVG_T_LAYER_BASE + 16u * (uint64_t)layer + (uint64_t)which;
}

#endif /* SVGEN_H */
