// decode_attn_dense_noalloc: the dense call with its workspace in a fixed, library-owned
// device array instead of caller-provided memory.
//
// Some callers cannot allocate device memory at the point where they run decode attention: a
// plugin or custom operator inside a host framework that owns every device allocation and hands
// the operator only its inputs and outputs; code issuing work while a stream is being captured
// into a CUDA graph, where cudaMalloc is not allowed; latency-critical decode loops, where
// cudaMalloc may synchronise the device; processes that reserve nearly all HBM up front.  For
// them this entry point uses a file-scope __device__ array as the workspace.
//
// Costs and limits: the array (DECODE_ATTN_NOALLOC_SCRATCH_BYTES) exists on every GPU that loads
// the library, until the process exits.  Every call shares it, so calls that can overlap on the
// GPU (different streams, or different host threads on one device) race on it; serialise them.
// Each call clears the part of the array it uses before launching, because the merge counters
// must start at zero and the array keeps whatever the previous call left.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "decode_attn.h"

namespace {

constexpr int kMaxDevices = 64;

__device__ __align__(256) unsigned char g_noalloc_scratch[DECODE_ATTN_NOALLOC_SCRATCH_BYTES];

std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevices];

// Device address of this device's copy of the array.  The first call on each device asks the
// runtime for it (with that device current) and caches it; in host code the array's name is only
// a host-side stand-in, never a usable device address.
void* scratch_address(int dev) {
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (g_scratch_addr[dev] == nullptr) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr)
            return nullptr;
        g_scratch_addr[dev] = ptr;
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
    void* scratch = scratch_address(dev);
    if (scratch == nullptr) return DA_ERR_CUDA;
    const size_t need = decode_attn_workspace_size(DA_VARIANT_DENSE, B, Hq, Hkv, D, 0);
    if (need > DECODE_ATTN_NOALLOC_SCRATCH_BYTES) return DA_ERR_WORKSPACE_TOO_SMALL;
    // Clear the scratch only for a call that can run; anything else goes straight to
    // decode_attn_dense, which reports why it rejects the arguments (need == 0: bad shape).
    auto a16 = [](const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; };
    const bool runnable = need > 0 && B > 0 && q && k && v && out && a16(q) && a16(k) && a16(v) &&
                          a16(out) && capacity >= 1 && k_len >= 0 && k_len <= capacity &&
                          std::isfinite(softmax_scale);
    if (runnable &&
        cudaMemsetAsync(scratch, 0, need, static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return DA_ERR_CUDA;
    return decode_attn_dense(q, k, v, out, B, Hq, Hkv, D, capacity, k_len, softmax_scale, scratch,
                             DECODE_ATTN_NOALLOC_SCRATCH_BYTES, stream);
}
