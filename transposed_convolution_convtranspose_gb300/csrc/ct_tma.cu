// ct_tma.cu -- host helpers: tensor-map encoding through the driver entry
// point, SM count and per-kernel launch attributes (cached).
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
    static int cache[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    if (!cache[dev]) {
        int n = 0;
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        cache[dev] = n;
    }
    return cache[dev];
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
    static std::unordered_map<Key, int, Hash> cache;
    // The shared-memory limit is an attribute of the function on a device, not
    // of a launch: keep it at the largest size requested so far, so that a
    // smaller request never lowers it under a larger one that was cached.
    static std::unordered_map<Key, size_t, Hash> limit;
    const Key key{fn, dev, threads, smem};
    const Key fkey{fn, dev, 0, 0};
    {
        std::lock_guard<std::mutex> lk(g_mu);
        auto it = cache.find(key);
        if (it != cache.end()) {
            *blocks_per_sm = it->second;
            return cudaSuccess;
        }
    }
    std::lock_guard<std::mutex> lk(g_mu);
    auto lt = limit.find(fkey);
    if (lt == limit.end() || lt->second < smem) {
        e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        limit[fkey] = smem;
    }
    int per = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, fn, threads, smem);
    if (e != cudaSuccess) return e;
    cache[key] = per;
    *blocks_per_sm = per;
    return cudaSuccess;
}

}  // namespace ct
