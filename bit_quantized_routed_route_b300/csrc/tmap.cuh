// tmap.cuh -- tensor maps (TMA descriptors) shared by the tensor-core kernels.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>

#include "ds4g_common.cuh"

namespace ds4g {

// cuTensorMapEncodeTiled from the CUDA driver API, looked up once.
cudaError_t get_encode(PFN_cuTensorMapEncodeTiled_v12000 *out);

// 3-D map over [experts][rows / phases][phases * row_bytes / 4 words] of
// one quantized weight tensor: `phases` (1, 2 or 4) consecutive rows form a
// super-row whose size is a multiple of 16 bytes.  Box = box_words (28:
// 112 bytes for the 84- and 70-byte blocks, 36: 144 bytes for a 136-byte
// MXFP4 unit) x (128 / phases) super-rows x 1 expert, no swizzle, zero fill
// outside the tensor; one box at word x = floor16(p * row_bytes + B * kb) / 4
// holds the B-byte unit kb of row phase p of 128 / phases super-rows.
cudaError_t weight_map(CUtensorMap *m, const void *base, int64_t row_bytes, int64_t rows,
                       int64_t expert_stride, int64_t experts, int phases, int box_words = 28);

}  // namespace ds4g
