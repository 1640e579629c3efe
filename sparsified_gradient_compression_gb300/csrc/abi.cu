// abi.cu -- small entry points of libdgc: status helpers, the launch counter, the SM count
// cache, and the self-test of the bounded look-back wait.
#include <atomic>

#include "dgc_device.cuh"

namespace {
std::atomic<uint64_t> g_launches{0};
int g_sms[128] = {0};

// Two look-back words that no tile ever publishes: tile 1 waits on tile 0 forever, which the
// spin limit must end.
__device__ uint64_t g_never_set[2];

__global__ void k_selftest_wait(int32_t* status, uint32_t spin_limit) {
    if (threadIdx.x < 32) dgc::lookback_exclusive(g_never_set, 1u, 1u, spin_limit, status, nullptr);
}
}  // namespace

void dgc_internal_count_launches(uint64_t k) { g_launches.fetch_add(k, std::memory_order_relaxed); }

int dgc_internal_sm_count() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return -1;
    if (dev < 128 && g_sms[dev] > 0) return g_sms[dev];
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
    if (dev < 128) g_sms[dev] = sms;
    return sms;
}

extern "C" uint64_t dgc_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

extern "C" int dgc_set_l2_fetch_granularity(int32_t bytes) {
    if (bytes < 0 || bytes > 128) return DGC_EINVAL;
    if (cudaDeviceSetLimit(cudaLimitMaxL2FetchGranularity, (size_t)bytes) != cudaSuccess) {
        cudaGetLastError();
        return DGC_ECUDA;
    }
    return DGC_OK;
}

extern "C" const char* dgc_status_string(int code) {
    switch (code) {
        case DGC_OK: return "ok";
        case DGC_EINVAL: return "invalid argument";
        case DGC_ECAPACITY: return "output buffer too small";
        case DGC_ECUDA: return "CUDA error";
        case DGC_ETIMEOUT: return "device-side wait timed out";
        case DGC_ECORRUPT: return "malformed message";
        case DGC_EUNSUPPORTED: return "unsupported size";
        default: return "unknown status";
    }
}

extern "C" int dgc_read_status(const int32_t* status_dev, dgc_stream_t stream) {
    if (!status_dev) return DGC_EINVAL;
    int32_t h = 0;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (cudaMemcpyAsync(&h, status_dev, sizeof h, cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return DGC_ECUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return DGC_ECUDA;
    return h;
}

extern "C" int dgc_selftest_wait_timeout(int32_t* status, uint32_t spin_limit, dgc_stream_t stream) {
    if (!status) return DGC_EINVAL;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    k_selftest_wait<<<1, 32, 0, s>>>(status, spin_limit);
    dgc_internal_count_launches(1);
    if (cudaPeekAtLastError() != cudaSuccess) {
        cudaGetLastError();
        return DGC_ECUDA;
    }
    return DGC_OK;
}
