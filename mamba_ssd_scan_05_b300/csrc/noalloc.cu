// noalloc.cu -- ssd_scan_fwd_noalloc: the scan for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc (or any allocator) at the moment they need the scan:
// code running inside a framework that owns all device memory through its own pool, plugins
// loaded into a host process that forbids device allocations after start-up, or paths that
// must not allocate while a CUDA graph is being captured.  ssd_scan_fwd needs a caller-owned
// workspace; this entry point instead uses a fixed scratch buffer that lives in the library's
// own device image, so the caller passes only its inputs and outputs.
//
// The buffer is a file-scope __device__ array.  Host code cannot use its name as a device
// address (in host code the name is only a host-side shadow), so the first call on each device
// looks the address up with cudaGetSymbolAddress while that device is current and caches it.
#include <mutex>

#include "common.cuh"

namespace {

constexpr size_t kScratchBytes = SSD_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

// Scratch of the no-allocation entry point (every device that loads this module holds it).
static __device__ __align__(256) uint8_t g_noalloc_scratch[kScratchBytes];

std::mutex g_mutex;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch buffer on the current device (looked up once per device).
int scratch_address(void** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SSD_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!g_scratch_addr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return SSD_ERR_CUDA;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return SSD_OK;
}

}  // namespace

extern "C" int ssd_scan_fwd_noalloc(const ssd_dims* dims, const void* x, const void* dt,
                                    const float* A, const void* B, const void* C, const float* D,
                                    const float* initial_state, int chunk_size, void* y,
                                    float* final_state, void* stream) {
    // size check first, so an oversized problem is rejected before anything touches the GPU
    const size_t need = ssd_scan_workspace_bytes(dims, chunk_size, SSD_PATH_CHUNKED);
    if (need == 0) {
        const int r = ssd_scan_resolve_path(dims, chunk_size, SSD_PATH_CHUNKED);
        return r < 0 ? -r : SSD_ERR_INVALID;
    }
    if (need > kScratchBytes) return SSD_ERR_WORKSPACE;
    // the scratch address is the current device's: the stream must belong to that device
    if (stream) {
        int dev = -1, sdev = -1;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaStreamGetDevice(static_cast<cudaStream_t>(stream), &sdev) != cudaSuccess)
            return SSD_ERR_CUDA;
        if (dev != sdev) return SSD_ERR_INVALID;
    }
    void* scratch = nullptr;
    const int rc = scratch_address(&scratch);
    if (rc != SSD_OK) return rc;
    // ssd_scan_fwd_path zeroes the status word on `stream` before its kernels run and
    // overwrites every other byte of the scratch it uses.
    return ssd_scan_fwd_path(dims, x, dt, A, B, C, D, initial_state, chunk_size, y, final_state,
                             scratch, kScratchBytes, stream, SSD_PATH_CHUNKED);
}
