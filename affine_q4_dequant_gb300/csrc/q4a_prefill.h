// q4a_prefill.h -- launchers of the prefill helpers (q4a_elementwise.cu), called by the C ABI.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "q4a.h"

namespace q4a {

// 4-bit min/max quantiser: w fp32 [rows][in_dim] -> packed codes, bf16 scales and biases.
q4a_status launch_quantize(uint8_t* w_packed, uint16_t* s, uint16_t* b, const float* w, int64_t rows,
                           int64_t in_dim, cudaStream_t stream);

// y fp32 [nb][out_dim] = W x for fp32 activations x [nb][in_dim], accumulated in fp32.
q4a_status launch_gemv_f32x(float* y, const uint8_t* w, const uint16_t* s, const uint16_t* b, const float* x,
                            int64_t nb, int64_t out_dim, int64_t in_dim, cudaStream_t stream);

}  // namespace q4a
