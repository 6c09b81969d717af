// vmx_intpsnr.h -- integer_psnr launch arguments, shared by the C-ABI
// (vmx_abi.cpp) and its kernel (vmx_intpsnr.cu).
#pragma once

#include <stdint.h>

#include <cuda_runtime.h>

namespace vmx {

struct IntPsnrArgs {
    const unsigned char *ref, *dis;  // plane pairs, frame f at base + f * height * stride
    int width, height, frames;
    int64_t stride;                  // bytes between rows
    int bytes;                       // bytes per sample: 1 (8 bpc) or 2
    uint64_t *sse;                   // device [frames]: exact sums of squared differences
    double *mse;                     // device [frames]: sse / (width * height)
    uint64_t *rows;                  // device [frames][height] row sums, or NULL
    uint32_t check_shrink;           // tests of a checked build: rows' extent taken as one less
};

// Enqueue the plane's sums (clearing sse first) and the MSE on `stream`.
cudaError_t launch_integer_psnr(const IntPsnrArgs &a, cudaStream_t stream);

// A checked build: the current device's flags of failed index checks in
// integer_psnr launches (read after `stream`, then cleared); 0 otherwise.
cudaError_t integer_psnr_check_flags(uint32_t *flags, cudaStream_t stream);

}  // namespace vmx
