// Launch interface of the block-scaled variant (k_blockq.cu) for the C ABI.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace bi {

cudaError_t launch_quantize_q6(const float *w, int64_t ldw, int N, int K, uint8_t *ql, uint8_t *qh, int8_t *sc,
                               float *d, cudaStream_t stream);
cudaError_t launch_quantize_act_blocks(const uint16_t *x, int64_t ldx, int M, int K, int8_t *q, float *d_a,
                                       cudaStream_t stream);
cudaError_t launch_linear_q6(const int8_t *qa, const float *d_a, int M, int K, const uint8_t *ql, const uint8_t *qh,
                             const int8_t *sc, const float *d, int N, float *y, bool pdl, cudaStream_t stream);

}  // namespace bi
