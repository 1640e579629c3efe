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
// current) and cached together with the identity of the CUDA context it belongs to. A device
// reset, or a primary context torn down and created again, loads the device code anew and may
// place the array elsewhere; the next call sees a different context and looks the address up
// again. Each call then runs the ordinary dgc_compress pipeline on that scratch;
// the pipeline's first kernel clears every counter, histogram and look-back word it later reads,
// so the previous call's leftovers do not matter. All calls on a device share the one array:
// calls whose GPU work can overlap (different streams without ordering, several host threads)
// race on it and must be serialized by the caller.
#include <cuda.h>

#include <mutex>

#include "dgc_device.cuh"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;  // 16 MiB on each GPU
constexpr int kMaxDevices = 128;

__device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// The driver calls that name the current context, fetched through the runtime so that the
// library does not link the driver library itself.
typedef CUresult (*ctx_get_current_fn)(CUcontext*);
typedef CUresult (*ctx_get_id_fn)(CUcontext, unsigned long long*);

struct ScratchSlot {
    void* addr = nullptr;
    unsigned long long ctx_id = 0;  // the context the address was looked up in
    bool have_id = false;
};

std::mutex g_scratch_mutex;
ScratchSlot g_scratch[kMaxDevices];
bool g_driver_looked_up = false;
ctx_get_current_fn g_ctx_get_current = nullptr;
ctx_get_id_fn g_ctx_get_id = nullptr;

// The unique id of the current context (unique for the process's lifetime, unlike the handle,
// which a new context may reuse); false when it cannot be had.
bool current_context_id(unsigned long long* id) {
    if (!g_driver_looked_up) {
        g_driver_looked_up = true;
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess && q == cudaDriverEntryPointSuccess)
            g_ctx_get_current = reinterpret_cast<ctx_get_current_fn>(f);
        f = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            g_ctx_get_id = reinterpret_cast<ctx_get_id_fn>(f);
        cudaGetLastError();
    }
    if (!g_ctx_get_current || !g_ctx_get_id) return false;
    CUcontext ctx = nullptr;
    if (g_ctx_get_current(&ctx) != CUDA_SUCCESS || !ctx) return false;
    return g_ctx_get_id(ctx, id) == CUDA_SUCCESS;
}

// Device address of the scratch array in the current context: looked up once per device and
// context. Without a context id (no current context yet, or a driver without the call) the
// address is looked up on every call instead, which is correct, only slower.
int scratch_address(void** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return DGC_ECUDA;
    if (dev < 0 || dev >= kMaxDevices) return DGC_EUNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    ScratchSlot& slot = g_scratch[dev];
    unsigned long long id = 0;
    const bool have_id = current_context_id(&id);
    if (slot.addr && have_id && slot.have_id && slot.ctx_id == id) {
        *out = slot.addr;
        return DGC_OK;
    }
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
        cudaGetLastError();
        slot = ScratchSlot();
        return DGC_ECUDA;
    }
    // the lookup made the primary context current if none was: name it now
    slot.addr = p;
    slot.have_id = have_id || current_context_id(&id);
    slot.ctx_id = id;
    *out = p;
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
