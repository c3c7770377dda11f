// noalloc.cu -- gqa_decode_attn for callers that cannot allocate device memory.
//
// Some callers of this library never get to call cudaMalloc. A plugin or
// custom operator inside a host inference framework receives only its input
// and output pointers, because the framework owns all device memory and
// forbids allocation while it runs. Code on a latency-critical decode loop may
// not allocate either, because cudaMalloc and cudaFree can synchronise the
// device and stall the stream. gqa_decode_attn needs a scratch workspace for
// its split-context partials, which such callers cannot provide. This entry
// point instead uses a fixed scratch array that lives in the library's own
// device memory.
//
// The scratch is one file-scope __device__ array of kStaticScratchBytes. Every
// GPU that loads the library holds it until the process exits. Host code must
// not use the array's name as a device address. On the host that name is
// only a stand-in symbol. Its device address is looked up with
// cudaGetSymbolAddress once per device, with that device current, the first
// time this entry point runs on it, and kept for the life of the process: the
// library must not be used on a device after cudaDeviceReset (which unloads
// the module and frees the array).
#include <mutex>

#include "internal.h"

namespace gqaq {
namespace {

constexpr size_t kStaticScratchBytes = size_t(1) << 20;  // 1 MiB per device
constexpr int kMaxScratchDevices = 64;

static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

void *g_scratch_addr[kMaxScratchDevices] = {};
std::mutex g_scratch_mutex;

// Device address of the scratch array on the current device (set up once).
int static_scratch(void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return GQAQ_ERR_CUDA;
    if (dev < 0 || dev >= kMaxScratchDevices) return GQAQ_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (g_scratch_addr[dev] == nullptr) {
        void *ptr = nullptr;
        const cudaError_t err = cudaGetSymbolAddress(&ptr, g_static_scratch);
        if (err != cudaSuccess || ptr == nullptr) return GQAQ_ERR_CUDA;
        g_scratch_addr[dev] = ptr;
    }
    *out = g_scratch_addr[dev];
    return GQAQ_OK;
}

}  // namespace
}  // namespace gqaq

// Same computation, arguments and results as gqa_decode_attn, without the
// workspace arguments. The workspace's arrival counters must start at zero:
// a __device__ array is zero-filled when the module loads, and every call
// leaves the counters at zero again. Calls that overlap on the GPU (on
// different streams, or from different host threads without ordering) share
// the one array and race.
extern "C" GQAQ_API int gqa_decode_attn_noalloc(const gqaq_dims *dims, const gqaq_half *q,
                                                const gqaq_half *k_cache, const gqaq_half *v_cache,
                                                const int32_t *valid_len, float scale, gqaq_half *out,
                                                void *stream) {
    void *scratch = nullptr;
    const int rc = gqaq::static_scratch(&scratch);
    if (rc != GQAQ_OK) return rc;
    // gqa_decode_attn computes this shape's exact scratch need (its grid after
    // the per-shape cap) and returns GQAQ_ERR_WORKSPACE, launching nothing,
    // when the 1 MiB array is too small.
    return gqa_decode_attn(dims, q, k_cache, v_cache, valid_len, scale, out, scratch,
                           gqaq::kStaticScratchBytes, stream);
}
