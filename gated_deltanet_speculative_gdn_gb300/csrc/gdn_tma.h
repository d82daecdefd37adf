// gdn_tma.h - host helpers shared by the translation units that launch TMA
// kernels.  Not part of the public ABI.
#pragma once

#include <cuda.h>

#include <cstdint>

namespace gdn {

// xc viewed as [N rows][C floats] with boxes of [rows][cols] floats, in the
// 128-byte swizzle when `swizzle` (the tensor cores' K-major operand layout
// for 32-float rows); GDN_OK or GDN_ERR_TMA.
int encode_xc_tiles(CUtensorMap *map, const float *xc, int64_t N, int64_t C, uint32_t rows, uint32_t cols,
                    bool swizzle);

// Multiprocessors of the current device (0 on error).
int sm_count_current();

}  // namespace gdn
