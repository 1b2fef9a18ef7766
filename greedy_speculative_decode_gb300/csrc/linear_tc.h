// linear_tc.h -- host side of the tcgen05 form of the batch-invariant linear,
// used for blocks of 9 to 32 rows.
#pragma once
#include "sv_internal.h"

namespace sv {

// Dynamic shared memory of one CTA.
size_t linear_tc_smem_bytes();
// Raise the shared-memory limit of every variant (once per process is enough).
cudaError_t prepare_linear_tc_kernels();
// Same contract as launch_linear for 1 <= p.M <= 32 (rows padded to 16 or 32),
// same grid and split,
// bit-identical results.  xmap: tensor map of p.X ([32 rows, p.Kd] bf16,
// row-major, box 32 rows x 64 columns, 128B swizzle).  slots: the split-tile
// exchange of this form (p.ws is not used), d.grid x 128 x 32 32-bit words,
// every byte 0xff before the first launch; each launch leaves them so.
cudaError_t launch_linear_tc(const LinearDesc& d, const CUtensorMap& xmap, uint32_t* slots, const LinParams& p,
                             int epi, bool norm, cudaStream_t s, bool pdl, const LinearDesc* next = nullptr);

}  // namespace sv
