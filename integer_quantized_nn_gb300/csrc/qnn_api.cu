// qnn_api.cu -- status reporting and the device status word.
#include <cuda_runtime.h>
#include <atomic>
#include <cstdint>
#include "qnn_internal.h"
#include "qnn_ptx.cuh"

namespace qnn {

// Set by kernels (atomicOr of kStatus* bits) when a bounded wait gives up.
__device__ uint32_t g_status_word;

namespace {
constexpr int kMaxDevices = 64;
std::atomic<uintptr_t> g_status_addr[kMaxDevices];
std::atomic<int> g_sm_count[kMaxDevices];

int current_device()
{
    int d = -1;
    if (cudaGetDevice(&d) != cudaSuccess) return -1;
    return (d >= 0 && d < kMaxDevices) ? d : -1;
}
}  // namespace

uint32_t *status_word()
{
    const int d = current_device();
    if (d < 0) return nullptr;
    uintptr_t a = g_status_addr[d].load(std::memory_order_acquire);
    if (a == 0) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) {
            (void)cudaGetLastError();
            return nullptr;
        }
        a = reinterpret_cast<uintptr_t>(p);
        g_status_addr[d].store(a, std::memory_order_release);
    }
    return reinterpret_cast<uint32_t *>(a);
}

int sm_count()
{
    const int d = current_device();
    if (d < 0) return 1;
    int n = g_sm_count[d].load(std::memory_order_relaxed);
    if (n <= 0) {
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, d) != cudaSuccess || n <= 0) {
            (void)cudaGetLastError();
            n = 1;
        }
        g_sm_count[d].store(n, std::memory_order_relaxed);
    }
    return n;
}

namespace {
// One block: thread 0 waits on a barrier that nothing ever arrives at.
__global__ void wait_timeout_kernel(uint32_t *status, uint64_t limit_ns)
{
    __shared__ __align__(8) uint64_t bar;
    const uint32_t b = smem_u32(&bar);
    if (threadIdx.x == 0) {
        mbar_init(b, 1);
        fence_mbar_init();
        (void)mbar_wait_slow(b, 0, status, limit_ns);
    }
}
}  // namespace

}  // namespace qnn

extern "C" const char *qnn_status_string(qnn_status s)
{
    switch (s) {
    case QNN_OK: return "ok";
    case QNN_ERR_INVALID_ARG: return "invalid argument";
    case QNN_ERR_UNSUPPORTED: return "unsupported";
    case QNN_ERR_ALIGNMENT: return "misaligned pointer or row pitch";
    case QNN_ERR_OVERFLOW_RISK: return "int32 accumulator overflow risk";
    case QNN_ERR_CUDA: return "CUDA error";
    case QNN_ERR_TIMEOUT: return "device wait timed out";
    default: return "unknown status";
    }
}

extern "C" qnn_status qnn_check_device_error(qnn_stream_t stream)
{
    if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return QNN_ERR_CUDA;
    uint32_t *w = qnn::status_word();
    if (!w) return QNN_ERR_CUDA;
    uint32_t v = 0;
    if (cudaMemcpy(&v, w, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return QNN_ERR_CUDA;
    if (v != 0) {
        const uint32_t zero = 0;
        if (cudaMemcpy(w, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess)
            return QNN_ERR_CUDA;
        if (v & qnn::kStatusTimeout) return QNN_ERR_TIMEOUT;
        if (v & qnn::kStatusBadArg) return QNN_ERR_INVALID_ARG;
    }
    return QNN_OK;
}

extern "C" qnn_status qnn_selftest_wait_timeout(uint64_t limit_ns, qnn_stream_t stream)
{
    if (limit_ns > 1000000000ull) return QNN_ERR_INVALID_ARG;
    uint32_t *w = qnn::status_word();
    if (!w) return QNN_ERR_CUDA;
    qnn::wait_timeout_kernel<<<1, 32, 0, (cudaStream_t)stream>>>(w, limit_ns);
    return qnn::launch_status();
}
