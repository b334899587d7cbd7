// Bandwidth probes: the device's own read-only and copy ceilings, measured with
// the access pattern the weight streams use (16-byte loads, many in flight per
// thread, a grid sized to the SM count), to set beside a library copy's figure.
#include "probe.cuh"

namespace bi {

namespace {

constexpr int kProbeThreads = 512;
constexpr int kProbeUnroll = 8;        // independent 16-byte loads in flight per thread

__global__ void __launch_bounds__(kProbeThreads) probe_read_kernel(const uint4 *__restrict__ buf, size_t n16,
                                                                   unsigned long long *out)
{
    const size_t stride = static_cast<size_t>(gridDim.x) * kProbeThreads;
    size_t i = static_cast<size_t>(blockIdx.x) * kProbeThreads + threadIdx.x;
    unsigned long long acc = 0;
    for (; i + (kProbeUnroll - 1) * stride < n16; i += kProbeUnroll * stride) {
        uint4 v[kProbeUnroll];
#pragma unroll
        for (int k = 0; k < kProbeUnroll; ++k) v[k] = __ldcs(buf + i + k * stride);
#pragma unroll
        for (int k = 0; k < kProbeUnroll; ++k)
            acc ^= (static_cast<unsigned long long>(v[k].y) << 32 | v[k].x) ^
                   (static_cast<unsigned long long>(v[k].w) << 32 | v[k].z);
    }
    for (; i < n16; i += stride) {
        const uint4 v = __ldcs(buf + i);
        acc ^= (static_cast<unsigned long long>(v.y) << 32 | v.x) ^ (static_cast<unsigned long long>(v.w) << 32 | v.z);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc ^= __shfl_xor_sync(0xffffffffu, acc, o);
    if ((threadIdx.x & 31) == 0 && acc != 0) atomicXor(out, acc);
}

__global__ void __launch_bounds__(kProbeThreads) probe_copy_kernel(const uint4 *__restrict__ src, uint4 *__restrict__ dst,
                                                                   size_t n16)
{
    const size_t stride = static_cast<size_t>(gridDim.x) * kProbeThreads;
    size_t i = static_cast<size_t>(blockIdx.x) * kProbeThreads + threadIdx.x;
    for (; i + (kProbeUnroll - 1) * stride < n16; i += kProbeUnroll * stride) {
        uint4 v[kProbeUnroll];
#pragma unroll
        for (int k = 0; k < kProbeUnroll; ++k) v[k] = __ldcs(src + i + k * stride);
#pragma unroll
        for (int k = 0; k < kProbeUnroll; ++k) __stcs(dst + i + k * stride, v[k]);
    }
    for (; i < n16; i += stride) __stcs(dst + i, __ldcs(src + i));
}

unsigned grid_for(size_t n16)
{
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) !=
                                                 cudaSuccess || sms <= 0)
        sms = 1;
    const size_t want = (n16 + kProbeThreads - 1) / kProbeThreads;
    const size_t g = static_cast<size_t>(sms) * 4;     // four CTAs of 512 threads per SM
    return static_cast<unsigned>(want < g ? (want > 0 ? want : 1) : g);
}

}  // namespace

cudaError_t launch_probe_read(const uint4 *buf, size_t n16, unsigned long long *out, cudaStream_t stream)
{
    cudaError_t e = cudaMemsetAsync(out, 0, sizeof(unsigned long long), stream);
    if (e != cudaSuccess) return e;
    probe_read_kernel<<<grid_for(n16), kProbeThreads, 0, stream>>>(buf, n16, out);
    return cudaGetLastError();
}

cudaError_t launch_probe_copy(const uint4 *src, uint4 *dst, size_t n16, cudaStream_t stream)
{
    probe_copy_kernel<<<grid_for(n16), kProbeThreads, 0, stream>>>(src, dst, n16);
    return cudaGetLastError();
}

}  // namespace bi
