// bitlin_forward_noalloc: the decode GEMV with its scratch memory taken from a
// fixed array compiled into the library instead of memory the handle
// allocates.
//
// Who needs it: callers that may not allocate device memory on their call
// path - code inside a runtime that owns every device allocation (a memory
// pool or arena that forbids outside cudaMalloc), and latency-critical loops
// that must never enter the allocator (cudaMalloc and cudaFree can
// synchronize the whole device).  bitlin_forward grows the handle's split-K
// scratch the first time it sees a larger token count; this entry point never
// does.
//
// The scratch is the file-scope array below.  Every GPU that loads this
// library holds it (kNoallocScratchBytes) until the process exits.  Host code
// cannot use the array's name as a device address, so the first call on each
// device, with that device current, looks the address up with
// cudaGetSymbolAddress and caches it; make that first call before any stream
// capture.  All calls share the array and it keeps the previous call's
// contents; nothing in it needs clearing: each call writes all the partial
// sums it reads.  Two calls whose kernels overlap on the GPU (different
// streams, or concurrent host threads) race on it.
#include <cuda_runtime.h>

#include <mutex>

#include "bitlin_internal.cuh"

using namespace bitlin_impl;

namespace {

constexpr size_t kNoallocScratchBytes = (size_t)16 << 20;  // 16 MiB

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

std::mutex g_setup_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on `dev` (looked up once per device).
cudaError_t scratch_address(int dev, void** out)
{
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (!g_scratch_ptr[dev]) {
        void* ptr = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_ptr[dev] = ptr;
    }
    *out = g_scratch_ptr[dev];
    return cudaSuccess;
}

}  // namespace

extern "C" size_t bitlin_noalloc_scratch_bytes(void) { return kNoallocScratchBytes; }

extern "C" bitlin_status bitlin_forward_noalloc(bitlin_t h, const float* x, int M, float* y,
                                                bitlin_stream_t stream)
{
    if (!h || !x || !y || M < 1) return BITLIN_EINVAL;
    if (h->sticky != BITLIN_OK) return h->sticky;

    // Scratch layout: the split-K partials [S][M][T*32] f32.
    const size_t partial_bytes = (size_t)h->S * (size_t)M * h->T * kTileRows * sizeof(float);
    if (partial_bytes > kNoallocScratchBytes) return BITLIN_ESCRATCH;

    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        h->last_cuda_error = (int)e;
        return BITLIN_ECUDA;
    }
    if (dev != h->device) return BITLIN_EINVAL;
    void* base = nullptr;
    e = scratch_address(dev, &base);
    if (e == cudaSuccess) {
        cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
        {
            DecodeParams p;
            p.bits = h->dbits;
            p.scales = h->dscales;
            p.signs = h->signs;
            p.x = x;
            p.y = y;
            p.partials = static_cast<float*>(base);
            p.M = M;
            p.N = h->N;
            p.K = h->K;
            p.S = h->S;
            p.T = h->T;
            p.perm = h->perm;
            p.ctas_per_slice = 0;
            p.cluster = 0;
            p.allow_cluster = 0;  // this entry point's split-K goes through the static scratch
            p.swiglu = 0;
            p.ids = nullptr;
            p.amax_cand = nullptr;
            p.amax_tickets = nullptr;
            e = bitlin_launch_decode(p, h->num_sms, s);
        }
    }
    if (e != cudaSuccess) {
        h->last_cuda_error = (int)e;
        return BITLIN_ECUDA;
    }
    return BITLIN_OK;
}
