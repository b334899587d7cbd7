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
#include "host_common.h"
#include "kernels.cuh"
#include "ptx.cuh"

#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

namespace {

// The scratch: exactly the workspace layout of the weight-streaming kernel
// (kWsBytes, about 2.1 MiB), shared by every call on a device.  Static device
// memory starts zeroed, and the kernel leaves its counters and partial sums at
// zero when it completes, so a call needs no clearing before it.
static_assert(bi::kWsBytes == BI_NOALLOC_SCRATCH_BYTES, "documented scratch size");
static_assert(bi::kMaxTok >= BI_NOALLOC_MAX_M, "scratch holds BI_NOALLOC_MAX_M token columns");
static __device__ __align__(256) unsigned char g_noalloc_scratch[bi::kWsBytes];

constexpr int kMaxDevices = 64;
struct ScratchAddr {
    CUcontext ctx;
    void *addr;
};
ScratchAddr g_scratch[kMaxDevices] = {};
std::mutex g_scratch_mutex;

typedef CUresult (*CtxGetCurrentFn)(CUcontext *);

// Device address of the scratch array on the current device.  In host code
// the array's name is only a host-side stand-in, so the address is looked up
// with that device current: once per device, and again if the device's
// context was replaced since (a reset reloads the library's module).
bi_status scratch_address(void **out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return BI_ERR_UNSUPPORTED;
    if (dev < 0 || dev >= kMaxDevices) return BI_ERR_UNSUPPORTED;
    static CtxGetCurrentFn ctx_fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] { ctx_fn = reinterpret_cast<CtxGetCurrentFn>(bi::host::driver_entry("cuCtxGetCurrent")); });
    if (!ctx_fn) return BI_ERR_UNSUPPORTED;
    CUcontext ctx = nullptr;   // null before the runtime has made a context current
    if (ctx_fn(&ctx) != CUDA_SUCCESS) return BI_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    ScratchAddr &s = g_scratch[dev];
    if (!s.addr || !ctx || s.ctx != ctx) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return BI_ERR_CUDA;
        if (ctx_fn(&ctx) != CUDA_SUCCESS || !ctx) return BI_ERR_CUDA;   // the lookup made it current
        s.ctx = ctx;
        s.addr = p;
    }
    *out = s.addr;
    return BI_OK;
}

}  // namespace

namespace bi {
namespace host {

bi_status noalloc_status_word(int **out)
{
    void *scratch = nullptr;
    const bi_status st = scratch_address(&scratch);
    if (st != BI_OK) return st;
    *out = static_cast<int *>(scratch);   // the status word leads the workspace layout
    return BI_OK;
}

}  // namespace host
}  // namespace bi

extern "C" BI_API bi_status bi_linear_w8a8_noalloc(const int8_t *q, const float *s_a, int M, int K,
                                                   const int8_t *w_q, const float *s_w, int N, uint16_t *y,
                                                   unsigned flags, bi_stream_t stream)
{
    bi_status st = bi::host::check_linear_operands(q, s_a, M, K, w_q, s_w, N);
    if (st != BI_OK) return st;
    if (!y) return BI_ERR_INVALID_ARG;
    if (M > BI_NOALLOC_MAX_M) return BI_ERR_UNSUPPORTED;  // beyond what the fixed scratch holds
    int sms = 0;
    st = bi::host::device_info(&sms);
    if (st != BI_OK) return st;

    void *scratch = nullptr;
    st = scratch_address(&scratch);
    if (st != BI_OK) return st;

    bi::SkinnyArgs a;
    st = bi::host::encode_int8_2d(&a.map_w, w_q, N, K, 128, bi::kBM, true);
    if (st != BI_OK) return st;
    st = bi::host::encode_int8_2d(&a.map_q, q, M, K, 128, M > 8 ? 16 : 8, false);
    if (st != BI_OK) return st;
    a.s_a = s_a;
    a.s_w = s_w;
    a.y = y;
    a.argmax = nullptr;
    a.M = M;
    a.N = N;
    a.K = K;
    a.ws = bi::workspace_view(scratch);
    a.pdl = (flags & BI_FLAG_PDL) != 0;
    a.grid = bi::host::skinny_grid(sms, N, K, bi::kMaxGrid);
    return bi::launch_skinny(a, stream) == cudaSuccess ? BI_OK : BI_ERR_CUDA;
}

extern "C" BI_API bi_status bi_linear_w8a8_noalloc_status(bi_stream_t stream)
{
    bi_status st = bi::host::device_info(nullptr);
    if (st != BI_OK) return st;
    void *scratch = nullptr;
    st = scratch_address(&scratch);
    if (st != BI_OK) return st;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return BI_ERR_CUDA;
    int word = 0;
    if (cudaMemcpy(&word, scratch, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return BI_ERR_CUDA;
    if (word == bi::DEV_OK) return BI_OK;
    // A wait gave up: the call's counters and partial sums may be left
    // non-zero.  Restore the whole scratch, status word included.
    if (cudaMemsetAsync(scratch, 0, bi::kWsBytes, stream) != cudaSuccess || cudaStreamSynchronize(stream) != cudaSuccess)
        return BI_ERR_CUDA;
    return BI_ERR_TIMEOUT;
}
