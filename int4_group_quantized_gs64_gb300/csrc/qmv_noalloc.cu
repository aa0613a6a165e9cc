// qmv_noalloc.cu - a dense int4-gs64 GEMV entry point that needs no caller
// workspace and allocates nothing.
//
// Some callers cannot call cudaMalloc: code that must never make the device
// synchronise (cudaMalloc and cudaFree can), hosts that forbid device
// allocation after start-up, and C callers with nowhere to keep a workspace
// between calls. For them, the activation split that qmv_int4_gs writes into
// a caller workspace goes into one file-scope device array instead. The array
// is part of the library image: every GPU that loads the library holds it
// until the process exits.
#include "../../include/qmv.h"
#include "qmv_internal.h"

namespace {

constexpr size_t kNoAllocMaxValues = 65536;  // S * K at most
constexpr size_t kNoAllocBytes = kNoAllocMaxValues * 4 + (kNoAllocMaxValues / 64) * 4;

// fp16 hi/lo fragments of the activations (4 bytes per value) followed by one
// factor per 64 values: 266,240 bytes.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocBytes];

// Device address of the array in the current device's context. Host code
// must not pass the symbol itself to a kernel: on the host it is only a
// stand-in for the device array. The lookup runs on every call rather than
// being cached, so a device reset or another context on the same device never
// leaves a stale address behind; once the library's module is loaded on the
// device it is a host-side lookup that allocates nothing.
void *noalloc_scratch() {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) return nullptr;
    return p;
}

}  // namespace

extern "C" int qmv_int4_gs_noalloc(const uint8_t *wq, const float *scales, int N, int K, int gs,
                                   const float *x, float *y, int S, qmv_stream_t stream) {
    if (!wq || !scales || !x || !y || N < 1 || S < 1 || gs != 64) return QMV_EINVAL;
    if (K < 64 || K % 64 || K > 65536) return QMV_ESHAPE;
    if ((size_t)S * (size_t)K > kNoAllocMaxValues) return QMV_EWORKSPACE;
    if (((uintptr_t)wq % 16) || ((uintptr_t)scales % 4) || ((uintptr_t)x % 4) || ((uintptr_t)y % 4))
        return QMV_EALIGN;
    void *scratch = noalloc_scratch();
    if (!scratch) return QMV_ECUDA;
    const cudaError_t e = qmv::launch_dense_int4(wq, scales, N, K, x, y, S, scratch,
                                                 reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? QMV_OK : QMV_ECUDA;
}
