// qmv_launch.cuh - host-side launch helpers: cudaLaunchKernelEx with optional
// programmatic dependent launch, dynamic shared-memory opt-in, and cached
// device properties for sizing persistent grids.
#pragma once

#include <cuda_runtime.h>

#include <mutex>
#include <utility>

namespace qmv {

// Number of SMs of the current device (cached per device, up to 64 devices).
inline int sm_count() {
    static int cache[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 1;
    if (cache[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1)
            n = 1;
        cache[dev] = n;
    }
    return cache[dev];
}

// Per-device memo of (kernel, value) pairs, so attribute setting and
// occupancy queries run once per kernel and device (and not inside a stream
// capture after the first call).
struct KernelMemo {
    std::mutex mu;
    const void *key[256];
    int dev[256];
    long long val[256];
    int n = 0;
    bool find(const void *k, int d, long long &v) {
        std::lock_guard<std::mutex> g(mu);
        for (int i = 0; i < n; ++i)
            if (key[i] == k && dev[i] == d) { v = val[i]; return true; }
        return false;
    }
    void put(const void *k, int d, long long v) {
        std::lock_guard<std::mutex> g(mu);
        if (n < 256) { key[n] = k; dev[n] = d; val[n] = v; ++n; }
    }
};

inline KernelMemo &smem_memo() { static KernelMemo m; return m; }
inline KernelMemo &occ_memo() { static KernelMemo m; return m; }

// Opts a kernel into `bytes` of dynamic shared memory (once per device).
template <class K>
inline cudaError_t set_smem(K *kernel, size_t bytes) {
    if (bytes <= 48 * 1024) return cudaSuccess;
    int dev = 0;
    cudaGetDevice(&dev);
    long long have = 0;
    if (smem_memo().find((const void *)kernel, dev, have) && have >= (long long)bytes)
        return cudaSuccess;
    cudaError_t e =
        cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (e == cudaSuccess) smem_memo().put((const void *)kernel, dev, (long long)bytes);
    return e;
}

template <class K>
inline int max_ctas_per_sm(K *kernel, int threads, size_t smem) {
    int dev = 0;
    cudaGetDevice(&dev);
    long long v = 0;
    if (occ_memo().find((const void *)kernel, dev, v)) return (int)v;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, threads, smem) != cudaSuccess ||
        n < 1)
        n = 1;
    occ_memo().put((const void *)kernel, dev, n);
    return n;
}

// Launches `kernel`; with pdl == true the kernel may start before the previous
// kernel on the stream finishes and must call griddepcontrol.wait before it
// reads that kernel's results.
template <class... KArgs, class... Args>
inline cudaError_t launch(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                          cudaStream_t st, bool pdl, Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = pdl ? attr : nullptr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

}  // namespace qmv
