// Host-side checks and TMA descriptor encoding shared by the entry points
// (bi_api.cu, bi_noalloc.cu), so that every entry point validates the same
// operands the same way.
#pragma once

#include "bi.h"

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

namespace bi {
namespace host {

constexpr long long kMaxK = 133144;  // largest K with K * 127^2 < 2^31

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline bool aligned4(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

// K range shared by every entry point.
inline bi_status check_k(int K)
{
    if (K < 16 || (K % 16) != 0) return BI_ERR_INVALID_ARG;
    if (static_cast<long long>(K) > kMaxK) return BI_ERR_INT32_BOUND;
    return BI_OK;
}

// The library is built for sm_103a only.
inline bi_status device_info(int *sm_count)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return BI_ERR_UNSUPPORTED;
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
        return BI_ERR_UNSUPPORTED;
    if (major != 10 || minor != 3) return BI_ERR_UNSUPPORTED;
    if (sm_count) {
        if (cudaDeviceGetAttribute(sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return BI_ERR_UNSUPPORTED;
    }
    return BI_OK;
}

// The operands of a linear layer (codes, scales, weights), without the
// workspace: null pointers, shapes, the K range and alignment.
inline bi_status check_linear_operands(const int8_t *q, const float *s_a, int M, int K, const int8_t *w_q,
                                       const float *s_w, int N)
{
    if (!q || !s_a || !w_q || !s_w) return BI_ERR_INVALID_ARG;
    if (M < 1 || M > 65535 || N < 1) return BI_ERR_INVALID_ARG;
    const bi_status s = check_k(K);
    if (s != BI_OK) return s;
    if (!aligned16(q) || !aligned16(w_q) || !aligned4(s_a) || !aligned4(s_w)) return BI_ERR_ALIGNMENT;
    return BI_OK;
}

// A driver entry point fetched through the runtime, so that the library does
// not link libcuda directly (null if the driver lacks it).
inline void *driver_entry(const char *name)
{
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion(name, &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
        return nullptr;
    return p;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

inline EncodeTiledFn encode_fn()
{
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] { fn = reinterpret_cast<EncodeTiledFn>(driver_entry("cuTensorMapEncodeTiled")); });
    return fn;
}

// 2-D int8 tensor [rows, cols] (row stride cols bytes), box box_cols x box_rows,
// 128-byte swizzle, zero fill outside the tensor.
inline bi_status encode_int8_2d(CUtensorMap *map, const void *base, long long rows, long long cols, int box_cols,
                                int box_rows, bool stream_once)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn) return BI_ERR_UNSUPPORTED;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols)};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows)};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    stream_once ? CU_TENSOR_MAP_L2_PROMOTION_L2_256B : CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? BI_OK : BI_ERR_CUDA;
}

// 2-D f16 tensor [rows, cols] (row stride 2 * cols bytes), box box_cols x
// box_rows, 128-byte swizzle, zero fill outside the tensor.
inline bi_status encode_f16_2d(CUtensorMap *map, const void *base, long long rows, long long cols, int box_cols,
                               int box_rows)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn) return BI_ERR_UNSUPPORTED;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(2 * cols)};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows)};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? BI_OK : BI_ERR_CUDA;
}

// CTAs of the weight-streaming kernel: two per SM for a large weight matrix
// (measured faster from about 50 MB up: more bytes in flight per SM), one per
// SM for smaller ones (faster below about 25 MB: less fixed cost per CTA).
inline int skinny_grid(int sms, int N, int K, int max_grid)
{
    const bool large = static_cast<long long>(N) * K >= (32LL << 20);
    const int g = large ? 2 * sms : sms;
    return g < max_grid ? g : max_grid;
}

// The status word of the no-alloc entry point's fixed scratch on the current
// device (defined with that scratch, in bi_noalloc.cu).
bi_status noalloc_status_word(int **out);

}  // namespace host
}  // namespace bi
