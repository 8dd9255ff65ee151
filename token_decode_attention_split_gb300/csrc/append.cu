// KV append: the step before decode attention that writes this step's new K/V rows into the
// cache the attention kernels read.
//   decode_attn_append_paged  "DflashScratch" (dflash_head), field slot_mapping_dev: row t goes to
//                             the paged-cache slot slot_mapping[t] (i64) of every KV head.
//   decode_attn_append_ring   "AttnV41" (attn_v41), method decode_body: the window ring write at
//                             pos % window, the position read on the device.
// Both are plain HBM-bound copies: one warp moves one new row (K and V of every KV head) with
// 16-byte loads issued in batches before their stores; the first batch of a row's data is
// requested together with its slot word (the loads do not depend on it), so a warp waits on
// memory about once per row.  The slot or position is read on the device and never validated by
// a sync.
#include <cuda_runtime.h>

#include <cstdint>

#include "decode_attn.h"
#include "ptx.cuh"

namespace {

constexpr int kAppendThreads = 256;   // 8 warps, one new row each per step
constexpr int kAppendBatch = 8;       // 16-byte loads in flight per lane

struct AppendArgs {
    const uint4* k_new;   // [rows, Hkv, D] as 16-byte chunks
    const uint4* v_new;
    uint4* k_pool;
    uint4* v_pool;
    const int64_t* where;  // slot per row (paged) or position per sequence (ring)
    int64_t rows;          // T (paged) or B (ring)
    int Hkv;
    int chunks;            // 16-byte chunks per row: D / 8
    int64_t page_size;     // paged
    int64_t num_slots;     // paged: num_pages * page_size
    int64_t pool_rows;     // ring
    int64_t window;        // ring
    int ring;
};

// First destination row (in rows of D elements) of new row `row` and the stride between its KV
// heads' destination rows, or false when the slot or position says to skip the row.
__device__ __forceinline__ bool dest_rows(const AppendArgs& a, int64_t row, int64_t& base,
                                          int64_t& head_stride) {
    const int64_t w = a.where[row];
    if (a.ring) {
        if (w < 0) return false;
        base = row * a.Hkv * a.pool_rows + w % a.window;
        head_stride = a.pool_rows;
        return true;
    }
    if (w < 0 || w >= a.num_slots) return false;
    const int64_t page = w / a.page_size, off = w - page * a.page_size;
    base = page * a.Hkv * a.page_size + off;
    head_stride = a.page_size;
    return true;
}

__global__ void __launch_bounds__(kAppendThreads) append_kernel(const AppendArgs a) {
    da::grid_dependency_wait();
    da::allow_dependent_launch();
    const int lane = threadIdx.x & 31;
    const int64_t warps = static_cast<int64_t>(gridDim.x) * (kAppendThreads / 32);
    const int half = a.Hkv * a.chunks;    // 16-byte chunks of one new row's K (or V), all heads
    for (int64_t row = blockIdx.x * (kAppendThreads / 32) + (threadIdx.x >> 5); row < a.rows;
         row += warps) {
        const int64_t src0 = row * half;
        int64_t base = 0, head_stride = 0;
        for (int c0 = 0; c0 < 2 * half; c0 += 32 * kAppendBatch) {
            uint4 x[kAppendBatch];
#pragma unroll
            for (int i = 0; i < kAppendBatch; ++i) {
                const int c = c0 + i * 32 + lane;
                if (c < 2 * half) {
                    const bool isv = c >= half;
                    x[i] = __ldg((isv ? a.v_new : a.k_new) + src0 + (isv ? c - half : c));
                }
            }
            // the slot word, requested after the first batch: a skipped row stores nothing
            if (c0 == 0 && !dest_rows(a, row, base, head_stride)) break;
#pragma unroll
            for (int i = 0; i < kAppendBatch; ++i) {
                const int c = c0 + i * 32 + lane;
                if (c < 2 * half) {
                    const bool isv = c >= half;
                    const int r = isv ? c - half : c;          // chunk within K (or V) of all heads
                    const int g = r / a.chunks, cc = r - g * a.chunks;
                    (isv ? a.v_pool : a.k_pool)[(base + g * head_stride) * a.chunks + cc] = x[i];
                }
            }
        }
    }
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

da_status launch(const AppendArgs& a, void* stream) {
    const int64_t work = a.rows;
    if (work == 0) return DA_OK;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return DA_ERR_CUDA;
    const int64_t want = (work + kAppendThreads / 32 - 1) / (kAppendThreads / 32);
    // at most six CTAs per SM (6 x 8 warps x 4 KB of loads in flight): every row in flight at
    // once (8 per SM) queues more than the memory system overlaps (append_paged 12.66 -> 12.46
    // us; four per SM 12.49, two or three 14.5)
    const int grid = static_cast<int>(want < 6LL * sms ? want : 6LL * sms);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kAppendThreads);
    cfg.stream = static_cast<cudaStream_t>(stream);
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, append_kernel, a) == cudaSuccess ? DA_OK : DA_ERR_CUDA;
}

da_status check_rows(const void* k_new, const void* v_new, void* k_pool, void* v_pool,
                     const int64_t* where, int64_t rows, int Hkv, int D) {
    if (!k_new || !v_new || !k_pool || !v_pool || !where) return DA_ERR_INVALID_ARGUMENT;
    if (!aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(k_pool, 16) || !aligned(v_pool, 16) ||
        !aligned(where, 8))
        return DA_ERR_INVALID_ARGUMENT;
    if (rows < 0 || Hkv <= 0 || D <= 0) return DA_ERR_INVALID_ARGUMENT;
    if (D % 8 != 0 || D > 1024) return DA_ERR_UNSUPPORTED;
    return DA_OK;
}

}  // namespace

extern "C" da_status decode_attn_append_paged(const void* k_new, const void* v_new, void* k_pool,
                                              void* v_pool, const int64_t* slot_mapping, int64_t T,
                                              int Hkv, int D, int page_size, int64_t num_pages,
                                              void* stream) {
    const da_status st = check_rows(k_new, v_new, k_pool, v_pool, slot_mapping, T, Hkv, D);
    if (st != DA_OK) return st;
    if (page_size <= 0 || num_pages < 0) return DA_ERR_INVALID_ARGUMENT;
    AppendArgs a{};
    a.k_new = static_cast<const uint4*>(k_new);
    a.v_new = static_cast<const uint4*>(v_new);
    a.k_pool = static_cast<uint4*>(k_pool);
    a.v_pool = static_cast<uint4*>(v_pool);
    a.where = slot_mapping;
    a.rows = T;
    a.Hkv = Hkv;
    a.chunks = D / 8;
    a.page_size = page_size;
    a.num_slots = num_pages * page_size;
    a.ring = 0;
    return launch(a, stream);
}

extern "C" da_status decode_attn_append_ring(const void* k_new, const void* v_new, void* k_pool,
                                             void* v_pool, const int64_t* positions, int B,
                                             int Hkv, int D, int64_t pool_rows, int window,
                                             void* stream) {
    const da_status st = check_rows(k_new, v_new, k_pool, v_pool, positions, B, Hkv, D);
    if (st != DA_OK) return st;
    if (window <= 0 || pool_rows < window) return DA_ERR_INVALID_ARGUMENT;
    AppendArgs a{};
    a.k_new = static_cast<const uint4*>(k_new);
    a.v_new = static_cast<const uint4*>(v_new);
    a.k_pool = static_cast<uint4*>(k_pool);
    a.v_pool = static_cast<uint4*>(v_pool);
    a.where = positions;
    a.rows = B;
    a.Hkv = Hkv;
    a.chunks = D / 8;
    a.pool_rows = pool_rows;
    a.window = window;
    a.ring = 1;
    return launch(a, stream);
}
