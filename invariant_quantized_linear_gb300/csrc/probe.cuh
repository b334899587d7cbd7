// Launch interface of the bandwidth probes (k_probe.cu) for the C ABI.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace bi {

// Streams n16 16-byte words once; out[0] = xor of all 64-bit words.
cudaError_t launch_probe_read(const uint4 *buf, size_t n16, unsigned long long *out, cudaStream_t stream);
// dst = src, n16 16-byte words.
cudaError_t launch_probe_copy(const uint4 *src, uint4 *dst, size_t n16, cudaStream_t stream);

}  // namespace bi
