// Internal host-side interface between the C ABI (api.cu) and the no-allocation entry point
// (noalloc.cu).  Not part of the public ABI.
#pragma once

#include <cstddef>
#include <cstdint>

#include "decode_attn.h"

namespace da {

// Unique id of the CUDA context current on the calling thread, 0 when none is current yet (or
// the driver cannot tell).  A device reset replaces the primary context and with it the id, so
// device addresses of the library's __device__ variables cached under the old id are looked up
// again.
unsigned long long current_context_id();

// decode_attn_dense with one difference: once every argument check has passed, right before the
// kernel launch, the workspace's merge counters (the part that must start at zero) are cleared on
// `stream`.  A rejected call enqueues nothing, like every other entry point.
da_status dense_clearing_workspace(const void* q, const void* k, const void* v, void* out, int B,
                                   int Hq, int Hkv, int D, int64_t capacity, int64_t k_len,
                                   float softmax_scale, void* workspace, size_t workspace_bytes,
                                   void* stream);

}  // namespace da
