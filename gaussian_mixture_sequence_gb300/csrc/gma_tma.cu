// Tensor maps for TMA (bulk tensor) loads, encoded on the host.
#include "gma_internal.cuh"

#include <string.h>

#include <atomic>
#include <mutex>

namespace gma {
namespace {

using EncodeTiled = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                 const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                 CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiled encoder()
{
    static EncodeTiled fn = []() -> EncodeTiled {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return nullptr;
        return reinterpret_cast<EncodeTiled>(p);
    }();
    return fn;
}

} // namespace

bool make_tma_2d(CUtensorMap *m, const void *base, bool bf16, unsigned long long rows, unsigned long long cols,
                 unsigned box_rows)
{
    EncodeTiled enc = encoder();
    if (!enc) return false;
    const unsigned e = bf16 ? 2 : 4;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols * e};
    cuuint32_t box[2] = {128 / e, box_rows};
    cuuint32_t es[2] = {1, 1};
    return enc(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2,
               const_cast<void *>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_tma_3d(CUtensorMap *m, const void *base, bool bf16, unsigned long long d0, unsigned long long d1,
                 unsigned long long d2, unsigned box1)
{
    EncodeTiled enc = encoder();
    if (!enc) return false;
    const unsigned e = bf16 ? 2 : 4;
    cuuint64_t dims[3] = {d0, d1, d2};
    cuuint64_t strides[2] = {d0 * e, d0 * d1 * e};
    cuuint32_t box[3] = {128 / e, box1, 1};
    cuuint32_t es[3] = {1, 1, 1};
    return enc(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3,
               const_cast<void *>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// SM count per device ordinal, looked up once per device (0 = not yet known).
int sm_count()
{
    constexpr int kMaxDev = 64;
    static std::atomic<int> cache[kMaxDev];
    int dev = 0, v = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 152;
    if (dev < 0 || dev >= kMaxDev) {
        return cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && v > 0 ? v : 152;
    }
    const int c = cache[dev].load(std::memory_order_relaxed);
    if (c > 0) return c;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0) return 152;
    cache[dev].store(v, std::memory_order_relaxed);
    return v;
}

namespace {
constexpr int kFlagDevices = 64;
std::mutex g_flag_mu;
std::atomic<unsigned int *> g_flags{nullptr};   // host pointer, kFlagDevices words

int current_device()
{
    int dev = -1;
    return cudaGetDevice(&dev) == cudaSuccess && dev >= 0 && dev < kFlagDevices ? dev : -1;
}
} // namespace

unsigned int *timeout_flag_dev()
{
    const int dev = current_device();
    if (dev < 0) return nullptr;
    unsigned int *h = g_flags.load(std::memory_order_acquire);
    if (!h) {
        std::lock_guard<std::mutex> lk(g_flag_mu);
        h = g_flags.load(std::memory_order_relaxed);
        if (!h) {
            void *p = nullptr;
            if (cudaHostAlloc(&p, kFlagDevices * sizeof(unsigned int), cudaHostAllocMapped | cudaHostAllocPortable) !=
                cudaSuccess)
                return nullptr;
            memset(p, 0, kFlagDevices * sizeof(unsigned int));
            h = static_cast<unsigned int *>(p);
            g_flags.store(h, std::memory_order_release);
        }
    }
    void *d = nullptr;
    if (cudaHostGetDevicePointer(&d, h + dev, 0) != cudaSuccess) return nullptr;
    return static_cast<unsigned int *>(d);
}

volatile unsigned int *timeout_flag_host()
{
    const int dev = current_device();
    unsigned int *h = g_flags.load(std::memory_order_acquire);
    return dev >= 0 && h ? h + dev : nullptr;
}

} // namespace gma
