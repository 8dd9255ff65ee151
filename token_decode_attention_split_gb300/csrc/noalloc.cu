// decode_attn_dense_noalloc: the dense call with its workspace in a fixed, library-owned
// device array instead of caller-provided memory.
//
// Some callers cannot allocate device memory at the point where they run decode attention: a
// plugin or custom operator inside a host framework that owns every device allocation and hands
// the operator only its inputs and outputs; latency-critical decode loops, where cudaMalloc may
// synchronise the device; processes that reserve nearly all HBM up front.  For them this entry
// point uses a file-scope __device__ array as the workspace.
//
// Costs and limits: the array (DECODE_ATTN_NOALLOC_SCRATCH_BYTES) exists on every GPU that loads
// the library, until the process exits.  Every call shares it, so calls that can overlap on the
// GPU (different streams, or different host threads on one device) race on it; serialise them.
// Each call clears the array's merge counters before its kernel starts, because they must start
// at zero and the array keeps whatever the previous call left there.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "decode_attn.h"
#include "host_api.h"

namespace {

constexpr int kMaxDevices = 64;

__device__ __align__(256) unsigned char g_noalloc_scratch[DECODE_ATTN_NOALLOC_SCRATCH_BYTES];

std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevices];
unsigned long long g_scratch_ctx[kMaxDevices];   // context the cached address belongs to

// Device address of this device's copy of the array.  The first call on each device asks the
// runtime for it (with that device current) and caches it; in host code the array's name is only
// a host-side stand-in, never a usable device address.  The cache is tied to the CUDA context: a
// device reset replaces the context (and may move the array), and the next call asks again.
void* scratch_address(int dev) {
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    const unsigned long long ctx = da::current_context_id();
    if (g_scratch_addr[dev] == nullptr || ctx == 0 || ctx != g_scratch_ctx[dev]) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr)
            return nullptr;
        g_scratch_addr[dev] = ptr;
        g_scratch_ctx[dev] = da::current_context_id();
    }
    return g_scratch_addr[dev];
}

}  // namespace

extern "C" da_status decode_attn_dense_noalloc(const void* q, const void* k, const void* v,
                                               void* out, int B, int Hq, int Hkv, int D,
                                               int64_t capacity, int64_t k_len,
                                               float softmax_scale, void* stream) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return DA_ERR_CUDA;
    const size_t need = decode_attn_workspace_size(DA_VARIANT_DENSE, B, Hq, Hkv, D, 0);
    if (need > DECODE_ATTN_NOALLOC_SCRATCH_BYTES) return DA_ERR_WORKSPACE_TOO_SMALL;
    void* scratch = scratch_address(dev);
    if (scratch == nullptr) return DA_ERR_CUDA;
    // every argument check of decode_attn_dense runs before the counters are cleared, so a
    // rejected call enqueues nothing
    return da::dense_clearing_workspace(q, k, v, out, B, Hq, Hkv, D, capacity, k_len,
                                        softmax_scale, scratch, DECODE_ATTN_NOALLOC_SCRATCH_BYTES,
                                        stream);
}
