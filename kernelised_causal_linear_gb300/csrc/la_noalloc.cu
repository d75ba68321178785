// la_noalloc.cu -- la_forward for callers that cannot allocate device memory.
//
// Some callers of this library cannot hand it a workspace: a plugin living
// inside a host application whose own pool owns every byte of device memory
// and forbids allocations behind its back, or latency-critical serving code
// that must never call cudaMalloc / cudaFree because those calls can
// synchronise the whole device and stall every other stream.  For them,
// la_forward_noalloc runs the same forward with its scratch taken from a
// fixed array that lives in the library's own device image.
//
// The array below is a file-scope __device__ variable: every GPU on which the
// library is loaded holds LA_NOALLOC_SCRATCH_BYTES of it until the process
// exits.  Host code must never pass the symbol itself to a kernel -- on the
// host it is only a stand-in, not a device address -- so the device address
// is looked up with cudaGetSymbolAddress once per device, with that device
// current, on the first call made on that device.
#include <mutex>

#include "la_internal.cuh"

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[LA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_addr[kMaxDevices];

// Device address of the scratch array on the current device, or NULL.
void* scratch_address()
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return nullptr;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_addr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p)
            return nullptr;
        g_addr[dev] = p;
    }
    return g_addr[dev];
}

}  // namespace

extern "C" la_status la_forward_noalloc(const void* q, const void* k, const void* v, float* out,
                                        int64_t B, int64_t H, int64_t N, int d, int dv,
                                        int causal, int feature_map, const float* gamma,
                                        int dtype, la_stream_t stream)
{
    const size_t need = la_forward_workspace_size(B, H, N, d, dv, causal, dtype);
    if (need > (size_t)LA_NOALLOC_SCRATCH_BYTES)
        return LA_ERR_TOO_LARGE;
    void* scratch = nullptr;
    if (need > 0) {
        scratch = scratch_address();
        if (!scratch)
            return LA_ERR_CUDA;
    }
    // la_forward checks every argument, clears whatever part of the scratch
    // must start at zero, and only enqueues work on `stream`.
    return la_forward(q, k, v, out, B, H, N, d, dv, causal, feature_map, gamma, dtype, scratch,
                      (size_t)LA_NOALLOC_SCRATCH_BYTES, stream);
}
