// linear_tc.h -- host side of the tcgen05 form of the batch-invariant linear,
// used for blocks of 9 to 32 rows.
#pragma once
#include "sv_internal.h"

namespace sv {

// Most rows of one call of the tcgen05 form (prefill blocks); verify steps
// take at most kMaxK.
constexpr int kTcMaxRows = 128;

// Dynamic shared memory of one CTA for calls of up to mp rows.
size_t linear_tc_smem_bytes(int mp);
// Raise the shared-memory limit of every variant (once per process is enough).
cudaError_t prepare_linear_tc_kernels();
// Same contract as launch_linear for 1 <= p.M <= kTcMaxRows (rows padded to
// 16, 32 or 128; the LM-head epilogue takes at most 32), same grid and split,
// bit-identical results.  xmap: tensor map of p.X ([kTcMaxRows rows, p.Kd]
// bf16, row-major, 128B swizzle) with boxes of 64 columns x 32 rows for
// p.M <= 32, x 128 rows above.  slots: the split-tile exchange of this form
// (p.ws is not used), d.grid x 128 x kTcMaxRows 32-bit words, every byte 0xff
// before the first launch; each launch leaves them so.
// xn[m, :] = the RMS-normalised row m of x (m < M), exactly as the norm
// prologue computes it; for steps of more than 8 rows, whose QKV, gate|up
// and LM head linears then take xn without a norm prologue.
cudaError_t launch_norm_rows(const bf16* x, const float* x_ss, const bf16* gain, bf16* xn, int M, int H,
                             float eps, cudaStream_t s, bool pdl);
cudaError_t launch_linear_tc(const LinearDesc& d, const CUtensorMap& xmap, uint32_t* slots, const LinParams& p,
                             int epi, bool norm, cudaStream_t s, bool pdl, const LinearDesc* next = nullptr);

}  // namespace sv
