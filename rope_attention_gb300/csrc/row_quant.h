// Internal interface of the row FP8 quantiser (row_quant.cu) for the C-ABI layer.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace ra {

// x [T, H] bf16 -> codes [T, H] E4M3 + scale [T] fp32 (packed == false), or the
// row-packed [T, H + 4] layout in `codes` (packed == true; `scale` unused).
cudaError_t launch_row_quantize(const uint16_t* x, int64_t T, int64_t H, uint8_t* codes, float* scale,
                                bool packed, cudaStream_t stream);

}  // namespace ra
