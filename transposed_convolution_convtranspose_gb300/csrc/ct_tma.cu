// ct_tma.cu -- host helpers: tensor-map encoding through the driver entry
// point, SM count (cached per device) and per-kernel launch attributes.
#include <atomic>
#include <mutex>
#include <unordered_map>

#include "ct_tma.h"

namespace ct {

namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode()
{
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

std::mutex g_mu;

}  // namespace

bool encode_tiled(CUtensorMap *map, CUtensorMapDataType dt, int rank, const void *base,
                  const uint64_t *dims, const uint64_t *strides_bytes, const uint32_t *box,
                  CUtensorMapSwizzle swizzle)
{
    EncodeTiledFn fn = get_encode();
    if (!fn) return false;
    cuuint64_t d[5], s[4];
    cuuint32_t b[5], e[5];
    for (int i = 0; i < rank; ++i) {
        d[i] = dims[i];
        b[i] = box[i];
        e[i] = 1;
        if (i + 1 < rank) s[i] = strides_bytes[i];
    }
    const CUresult r = fn(map, dt, (cuuint32_t)rank, const_cast<void *>(base), d, s, b, e,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

int sm_count()
{
    static std::atomic<int> cache[64];      // zero-initialised (static storage)
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    int n = cache[dev].load(std::memory_order_relaxed);
    if (!n) {
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        cache[dev].store(n, std::memory_order_relaxed);
    }
    return n;
}

cudaError_t prepare_kernel(const void *fn, int threads, size_t smem, int *blocks_per_sm)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    struct Key {
        const void *fn;
        int dev, threads;
        size_t smem;
        bool operator==(const Key &o) const
        {
            return fn == o.fn && dev == o.dev && threads == o.threads && smem == o.smem;
        }
    };
    struct Hash {
        size_t operator()(const Key &k) const
        {
            return std::hash<const void *>()(k.fn) ^ (k.smem * 131) ^ ((size_t)k.dev << 40) ^ k.threads;
        }
    };
    // blocks per SM depend on the device, the function and the launch shape only
    static std::unordered_map<Key, int, Hash> cache;
    const Key key{fn, dev, threads, smem};
    std::lock_guard<std::mutex> lk(g_mu);
    // The dynamic shared-memory limit is an attribute of the function in the
    // current context, which a cudaDeviceReset (or a context of the caller's
    // own) starts again from the default: it is read back on every call and
    // raised when below the request -- never lowered, so that a smaller request
    // does not undercut a larger launch of the same function.
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, fn);
    if (e != cudaSuccess) return e;
    if ((size_t)fa.maxDynamicSharedSizeBytes < smem) {
        e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    auto it = cache.find(key);
    if (it != cache.end()) {
        *blocks_per_sm = it->second;
        return cudaSuccess;
    }
    int per = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, fn, threads, smem);
    if (e != cudaSuccess) return e;
    cache[key] = per;
    *blocks_per_sm = per;
    return cudaSuccess;
}

}  // namespace ct
