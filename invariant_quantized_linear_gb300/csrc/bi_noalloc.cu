// bi_linear_w8a8_noalloc: the weight-streaming linear layer with its scratch
// memory held by the library itself, for callers that cannot allocate device
// memory.
//
// Some callers have no way to obtain a workspace: code that runs where the
// allocator is off limits (inside a custom allocator or a memory-pool
// callback, in a plugin that is handed only input and output pointers by its
// host framework, or in a process that must not grow its device footprint
// after start-up).  For them the scratch the kernel needs (split-K partial
// sums, their counters, a status word) lives in one file-scope __device__
// array below, loaded with the library on every GPU that uses it and kept
// until the process exits.
#include "bi.h"
#include "kernels.cuh"
#include "ptx.cuh"

#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

namespace {

// The scratch: exactly the workspace layout of the weight-streaming kernel
// (kWsBytes, about 1.03 MiB), shared by every call on a device.
static_assert(bi::kWsBytes == BI_NOALLOC_SCRATCH_BYTES, "documented scratch size");
static_assert(bi::kMaxTok >= BI_NOALLOC_MAX_M, "scratch holds BI_NOALLOC_MAX_M token columns");
static __device__ __align__(256) unsigned char g_noalloc_scratch[bi::kWsBytes];

constexpr int kMaxDevices = 64;
void *g_scratch_addr[kMaxDevices] = {};
std::mutex g_scratch_mutex;

// Device address of the scratch array on the current device.  In host code
// the array's name is only a host-side stand-in, so the address is looked up
// once per device with that device current.
bi_status scratch_address(void **out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return BI_ERR_UNSUPPORTED;
    if (dev < 0 || dev >= kMaxDevices) return BI_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (!g_scratch_addr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return BI_ERR_CUDA;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return BI_OK;
}

// Same 2-D int8 TMA descriptor as the allocating entry point builds.
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn()
{
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

bi_status encode(CUtensorMap *map, const void *base, long long rows, long long cols, int box_rows, bool once)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn) return BI_ERR_UNSUPPORTED;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols)};
    cuuint32_t box[2] = {128u, static_cast<cuuint32_t>(box_rows)};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    once ? CU_TENSOR_MAP_L2_PROMOTION_L2_256B : CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? BI_OK : BI_ERR_CUDA;
}

}  // namespace

extern "C" BI_API bi_status bi_linear_w8a8_noalloc(const int8_t *q, const float *s_a, int M, int K,
                                                   const int8_t *w_q, const float *s_w, int N, uint16_t *y,
                                                   unsigned flags, bi_stream_t stream)
{
    if (!q || !s_a || !w_q || !s_w || !y) return BI_ERR_INVALID_ARG;
    if (N < 1 || M < 1) return BI_ERR_INVALID_ARG;
    if (M > BI_NOALLOC_MAX_M) return BI_ERR_UNSUPPORTED;  // beyond what the fixed scratch holds
    if (K < 16 || (K % 16) != 0) return BI_ERR_INVALID_ARG;
    if (static_cast<long long>(K) > 133144) return BI_ERR_INT32_BOUND;
    if ((reinterpret_cast<uintptr_t>(q) & 15u) || (reinterpret_cast<uintptr_t>(w_q) & 15u) ||
        (reinterpret_cast<uintptr_t>(s_a) & 3u) || (reinterpret_cast<uintptr_t>(s_w) & 3u))
        return BI_ERR_ALIGNMENT;

    int dev = 0, major = 0, minor = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return BI_ERR_UNSUPPORTED;
    if (major != 10 || minor != 3) return BI_ERR_UNSUPPORTED;

    void *scratch = nullptr;
    bi_status st = scratch_address(&scratch);
    if (st != BI_OK) return st;

    bi::SkinnyArgs a;
    st = encode(&a.map_w, w_q, N, K, bi::kBM, true);
    if (st != BI_OK) return st;
    st = encode(&a.map_q, q, M, K, M > 8 ? 16 : 8, false);
    if (st != BI_OK) return st;

    // The kernel needs its status word, counters and partial sums at zero.
    // A completed call leaves them so, but the array is shared by every call
    // and keeps whatever the last one left (for instance after a timeout), so
    // they are cleared here, on the same stream, before the launch.
    char *base = static_cast<char *>(scratch);
    if (cudaMemsetAsync(base, 0, bi::kWsBestOff, stream) != cudaSuccess) return BI_ERR_CUDA;
    if (cudaMemsetAsync(base + bi::kWsPartialOff, 0, bi::kWsBytes - bi::kWsPartialOff, stream) != cudaSuccess)
        return BI_ERR_CUDA;

    a.s_a = s_a;
    a.s_w = s_w;
    a.y = y;
    a.argmax = nullptr;
    a.M = M;
    a.N = N;
    a.K = K;
    a.ws = bi::workspace_view(scratch);
    a.pdl = (flags & BI_FLAG_PDL) != 0;
    a.grid = sms < bi::kMaxGrid ? sms : bi::kMaxGrid;
    return bi::launch_skinny(a, stream) == cudaSuccess ? BI_OK : BI_ERR_CUDA;
}
