// Launch interface of the split-KV verify attention (k_attn.cu) for the C ABI.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace bi {

struct AttnArgs {
    const uint16_t *q;   // [M, Hq, D] bf16
    const uint16_t *k;   // [S, Hkv, D] bf16 (k, v, o: 16-byte aligned)
    const uint16_t *v;   // [S, Hkv, D] bf16
    uint16_t *o;         // [M, Hq, D] bf16
    float *ws;           // [M, Hq, Cmax, D + 4] fp32 chunk results: mx, l, 2 unused, a[D]
    float scale;
    int M, Hq, Hkv, D, T0, Cmax;
    int sms;             // the device's SM count (chooses between chunk kernels)
};

// Chunks of 256 positions the last query (which sees T0 + M positions) covers.
int attn_chunks(int T0, int M);
// D is 64 or 128.
cudaError_t launch_attention(const AttnArgs &a, cudaStream_t stream);

}  // namespace bi
