// noalloc.cu -- dgc_compress_noalloc: the compressor for callers that cannot allocate device
// memory.
//
// dgc_compress needs a scratch workspace that the caller allocates. Some callers cannot do that
// at the point where they compress: a framework whose caching allocator owns all device memory
// and gives none out for a library's private use, code that runs while a CUDA graph is being
// captured or inside a latency-critical loop where cudaMalloc (which may synchronize the device)
// is not allowed, or a plug-in that must not change the process's device-memory footprint once it
// is running. For them this entry point uses a scratch array that the library itself holds: a
// file-scope __device__ array of kNoAllocScratchBytes, created on every GPU that loads the library
// and kept until the process exits. The caller still provides the inputs and outputs.
//
// In host code the array's name is only a stand-in, not a device address, so the address is
// looked up with cudaGetSymbolAddress once per device (on the first call with that device
// current) and cached. Each call then runs the ordinary dgc_compress pipeline on that scratch;
// the pipeline's first kernel clears every counter, histogram and look-back word it later reads,
// so the previous call's leftovers do not matter. All calls on a device share the one array:
// calls whose GPU work can overlap (different streams without ordering, several host threads)
// race on it and must be serialized by the caller.
#include <mutex>

#include "dgc_device.cuh"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;  // 16 MiB on each GPU
constexpr int kMaxDevices = 128;

__device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_scratch_mutex;
void* g_scratch_addr[kMaxDevices] = {nullptr};

// Device address of the scratch array on the current device (looked up once per device).
int scratch_address(void** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return DGC_ECUDA;
    if (dev < 0 || dev >= kMaxDevices) return DGC_EUNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (!g_scratch_addr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
            cudaGetLastError();
            return DGC_ECUDA;
        }
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return DGC_OK;
}

}  // namespace

extern "C" int dgc_compress_noalloc(const float* g, float* u, float* v, int64_t n,
                                    const int64_t* seg_off, int32_t nseg, const dgc_params* params,
                                    uint32_t* out_idx, float* out_val, int64_t out_cap,
                                    int64_t* out_count, dgc_seg_stats* stats, int32_t* status,
                                    dgc_stream_t stream) {
    size_t need = 0;
    int rc = dgc_compress_workspace(n, nseg, params, &need);
    if (rc != DGC_OK) return rc;
    if (need > kNoAllocScratchBytes) return DGC_EUNSUPPORTED;  // the problem does not fit
    void* scratch = nullptr;
    rc = scratch_address(&scratch);
    if (rc != DGC_OK) return rc;
    return dgc_compress(g, u, v, n, seg_off, nseg, params, out_idx, out_val, out_cap, out_count,
                        stats, status, scratch, kNoAllocScratchBytes, stream);
}
