// C ABI of the decode-attention library: argument checks, tensor-map descriptors, workspace
// layout, grid sizing and the kernel launch.  Every path either launches work on the caller's
// stream or returns an error before anything is enqueued.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <mutex>
#include <set>
#include <utility>

#include "decode_attn.h"
#include "launch.h"

namespace da {

// Device error word: kernels whose bounded waits time out record a code here.
__device__ unsigned int g_device_error_word;

namespace {

constexpr int kMaxDevices = 64;
std::atomic<int> g_grid_limit{0};
std::mutex g_mu;
// (kernel, context id) pairs whose shared-memory opt-in is done: the attribute belongs to the
// module loaded in that context, so a device reset (a new primary context) needs it again
std::set<std::pair<const void*, unsigned long long>> g_configured;
int g_sm_count[kMaxDevices];                          // 0 = not queried yet
unsigned* g_err_ptr[kMaxDevices];
unsigned long long g_err_ctx[kMaxDevices];            // context the cached address belongs to

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                             &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return static_cast<EncodeTiledFn>(nullptr);
        return reinterpret_cast<EncodeTiledFn>(f);
    }();
    return fn;
}

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

template <typename Fn>
Fn driver_fn(const char* name) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion(name, &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
        return nullptr;
    return reinterpret_cast<Fn>(f);
}

int current_device() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return -1;
    return dev;
}

int sm_count(int dev) {
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_sm_count[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
            return 0;
        g_sm_count[dev] = n;
    }
    return g_sm_count[dev];
}

unsigned* device_error_ptr(int dev) {
    std::lock_guard<std::mutex> lk(g_mu);
    const unsigned long long ctx = current_context_id();
    if (g_err_ptr[dev] == nullptr || ctx == 0 || ctx != g_err_ctx[dev]) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_device_error_word) != cudaSuccess) return nullptr;
        g_err_ptr[dev] = static_cast<unsigned*>(ptr);
        g_err_ctx[dev] = current_context_id();
    }
    return g_err_ptr[dev];
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int padded_group(int G) {
    if (G <= 8) return 8;
    if (G <= 16) return 16;
    if (G <= 32) return 32;
    if (G <= 64) return 64;
    return 0;
}

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

struct WsLayout {
    size_t counters, lse, o, total;
};

// counters: one u32 per merge unit; lse: [segments][G]; o: [segments][G][D] (G = heads per segment)
WsLayout ws_layout(long long units, long long segments, int G, int D) {
    WsLayout w;
    w.counters = 0;
    w.lse = round_up(static_cast<size_t>(units) * 4, 256);
    w.o = w.lse + round_up(static_cast<size_t>(segments) * G * 4, 256);
    w.total = w.o + static_cast<size_t>(segments) * G * D * 4;
    if (w.total == 0) w.total = 256;
    return w;
}

// Checks shared by every variant; returns DA_OK when the heads, dims and scale are usable.
da_status check_common(const void* q, const void* out, int B, int Hq, int Hkv, int D, float scale,
                       const void* ws) {
    if (!q || !out || !ws) return DA_ERR_INVALID_ARGUMENT;
    if (!aligned(q, 16) || !aligned(out, 16) || !aligned(ws, 16)) return DA_ERR_INVALID_ARGUMENT;
    if (B < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0) return DA_ERR_INVALID_ARGUMENT;
    if (!std::isfinite(scale)) return DA_ERR_INVALID_ARGUMENT;
    if (D != 64 && D != 128) return DA_ERR_UNSUPPORTED;
    if (padded_group(Hq / Hkv) == 0) return DA_ERR_UNSUPPORTED;
    if (static_cast<long long>(B) * Hq * D >= (1ll << 40)) return DA_ERR_UNSUPPORTED;
    return DA_OK;
}

Params base_params(const void* q, void* out, int B, int Hq, int Hkv, float scale, unsigned* err) {
    Params p{};
    p.q = static_cast<const __nv_bfloat16*>(q);
    p.out = static_cast<__nv_bfloat16*>(out);
    p.B = B;
    p.Hq = Hq;
    p.Hkv = Hkv;
    p.G = Hq / Hkv;
    p.seg_heads = p.G;
    p.kh = 1;
    p.tile_keys = kTileKeys;
    p.sq = 1;
    p.causal = 0;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.err = err;
    return p;
}

void bind_workspace(Params& p, void* ws, const WsLayout& w) {
    unsigned char* base = static_cast<unsigned char*>(ws);
    p.counters = reinterpret_cast<unsigned*>(base + w.counters);
    p.part_lse = reinterpret_cast<float*>(base + w.lse);
    p.part_o = reinterpret_cast<float*>(base + w.o);
}

da_status zero_output(void* out, int B, int Hq, int D, cudaStream_t st) {
    const size_t bytes = static_cast<size_t>(B) * Hq * D * 2;
    return cudaMemsetAsync(out, 0, bytes, st) == cudaSuccess ? DA_OK : DA_ERR_CUDA;
}

bool encode_3d(CUtensorMap* map, const void* base, cuuint64_t d0, cuuint64_t d1, cuuint64_t d2,
               cuuint64_t stride1_bytes, cuuint64_t stride2_bytes, cuuint32_t box1) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[3] = {d0, d1, d2};
    const cuuint64_t strides[2] = {stride1_bytes, stride2_bytes};
    const cuuint32_t box[3] = {64, box1, 1};
    const cuuint32_t estride[3] = {1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
              estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// KV heads per paged unit: the smallest power of two that makes a page of those heads (kh adjacent
// heads are kh * page_size contiguous rows) at least one 64-row tile, so a paged tile moves as one
// 64-row TMA box per 64-column half, exactly like a dense tile; limited so kh divides Hkv and the
// unit's kh * G query heads fit one CTA.
int paged_kv_heads(int Hkv, int G, int page_size) {
    int kh = 1;
    while (kh * page_size < kTileKeys && Hkv % (2 * kh) == 0 && 2 * kh * G <= 64) kh *= 2;
    return kh;
}

// Dense units of at most this many 64-row tiles are not split across CTAs.
constexpr long long kShortUnitTiles = 8;

// CTAs for a persistent dense/paged launch on `dev`.
int persistent_ctas(int dev) {
    const int sms = sm_count(dev);
    const int lim = g_grid_limit.load();
    return (lim > 0 && lim < sms) ? lim : sms;
}

// Sparse work split: items of (sequence and KV head, chunk of 512 selection entries) with all
// of the unit's G <= 64 query heads.  33..64 heads run on the tensor-core kernel, up to 32 on the
// mma.sync kernel (which holds at most 32 query columns).  The chunk depends on nothing, not on
// the width, B or the device, so trailing pads never move a chunk boundary.
bool sparse_uses_tc(int G, int D) {
    return (D == 64 || D == 128) && G > kSparseMaxHeads && G <= 64;
}
int sparse_padded_group(int G) { return G <= 8 ? 8 : G <= 16 ? 16 : 32; }
long long sparse_chunks(long long width) {
    return (width + kSparseChunkUnit - 1) / kSparseChunkUnit;
}

}  // namespace

unsigned long long current_context_id() {
    static const CtxGetCurrentFn get_current = driver_fn<CtxGetCurrentFn>("cuCtxGetCurrent");
    static const CtxGetIdFn get_id = driver_fn<CtxGetIdFn>("cuCtxGetId");
    if (!get_current || !get_id) return 0;
    CUcontext ctx = nullptr;
    if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return 0;
    unsigned long long id = 0;
    return get_id(ctx, &id) == CUDA_SUCCESS ? id : 0;
}

cudaError_t launch_kernel(const void* kernel, int smem, const Launch& L) {
    const int dev = current_device();
    if (dev < 0) return cudaErrorInvalidDevice;
    const unsigned long long ctx = current_context_id();
    bool need = true;
    if (ctx != 0) {
        std::lock_guard<std::mutex> lk(g_mu);
        need = g_configured.find({kernel, ctx}) == g_configured.end();
    }
    if (need) {
        cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        if (ctx != 0) {
            std::lock_guard<std::mutex> lk(g_mu);
            g_configured.insert({kernel, ctx});
        }
    }
    void* args[] = {const_cast<CUtensorMap*>(&L.tm_k), const_cast<CUtensorMap*>(&L.tm_v),
                    const_cast<Params*>(&L.p)};
    // Programmatic stream serialization: the kernel may be scheduled while the previous kernel
    // in the stream drains; it waits for that kernel's completion before touching memory.
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(L.grid);
    cfg.blockDim = dim3(L.threads);
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cfg.stream = L.stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelExC(&cfg, kernel, args);
}

}  // namespace da

using namespace da;

extern "C" {

int decode_attn_abi_version(void) { return DECODE_ATTN_ABI_VERSION; }

const char* decode_attn_status_string(int status) {
    switch (status) {
        case DA_OK: return "ok";
        case DA_ERR_INVALID_ARGUMENT: return "invalid argument";
        case DA_ERR_UNSUPPORTED: return "unsupported shape or option";
        case DA_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
        case DA_ERR_CUDA: return "CUDA error";
        default: return "unknown status";
    }
}

size_t decode_attn_workspace_size(int variant, int B, int Hq, int Hkv, int D, int64_t max_kv) {
    if (B < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || (D != 64 && D != 128)) return 0;
    const int G = Hq / Hkv;
    if (padded_group(G) == 0) return 0;
    const long long units = static_cast<long long>(B) * Hkv;
    long long segments = 0;
    if (variant == DA_VARIANT_DENSE || variant == DA_VARIANT_PAGED) {
        const int dev = current_device();
        if (dev < 0) return 0;
        const int sms = sm_count(dev);
        if (sms <= 0) return 0;
        if (variant == DA_VARIANT_PAGED) {
            // the page size is not an argument here: size for every unit width a call may use
            size_t most = 0;
            for (int kh = 1; kh <= 8; kh *= 2) {
                if (Hkv % kh != 0 || kh * G > 64) break;
                const long long u = units / kh;
                most = std::max(most, ws_layout(u, u + sms, kh * G, D).total);
            }
            return most;
        }
        segments = units + sms;
    } else if (variant == DA_VARIANT_SPARSE) {
        if (max_kv < 0) return 0;
        return ws_layout(units, units * sparse_chunks(max_kv), G, D).total;
    } else {
        return 0;
    }
    return ws_layout(units, segments, G, D).total;
}

da_status decode_attn_workspace_init(void* workspace, size_t bytes, void* stream) {
    if (!workspace && bytes) return DA_ERR_INVALID_ARGUMENT;
    if (bytes == 0) return DA_OK;
    return cudaMemsetAsync(workspace, 0, bytes, static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? DA_OK
               : DA_ERR_CUDA;
}

da_status decode_attn_spec_check(const decode_attn_spec* spec) {
    if (!spec || !std::isfinite(spec->softmax_scale)) return DA_ERR_INVALID_ARGUMENT;
    if (spec->has_alibi || spec->has_window_left || spec->has_window_right || spec->has_softcap)
        return DA_ERR_UNSUPPORTED;
    return DA_OK;   // causal: a single query row attends the whole live prefix anyway
}

da_status decode_attn_dense_spec(const decode_attn_spec* spec, const void* q, const void* k,
                                 const void* v, void* out, int B, int Hq, int Hkv, int D,
                                 int64_t capacity, int64_t k_len, void* workspace,
                                 size_t workspace_bytes, void* stream) {
    const da_status st = decode_attn_spec_check(spec);
    if (st != DA_OK) return st;
    return decode_attn_dense(q, k, v, out, B, Hq, Hkv, D, capacity, k_len, spec->softmax_scale,
                             workspace, workspace_bytes, stream);
}

da_status decode_attn_set_grid_limit(int max_ctas) {
    if (max_ctas < 0) return DA_ERR_INVALID_ARGUMENT;
    g_grid_limit.store(max_ctas);
    return DA_OK;
}

da_status decode_attn_read_device_error(uint32_t* code) {
    if (!code) return DA_ERR_INVALID_ARGUMENT;
    const int dev = current_device();
    if (dev < 0) return DA_ERR_CUDA;
    unsigned* ptr = device_error_ptr(dev);
    if (!ptr) return DA_ERR_CUDA;
    unsigned v = 0;
    if (cudaDeviceSynchronize() != cudaSuccess) return DA_ERR_CUDA;
    if (cudaMemcpy(&v, ptr, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess) return DA_ERR_CUDA;
    if (cudaMemset(ptr, 0, sizeof v) != cudaSuccess) return DA_ERR_CUDA;
    *code = v;
    return DA_OK;
}

da_status decode_attn_check_wait_timeout(uint32_t limit_us, void* stream) {
    if (limit_us < 1 || limit_us > 1000000) return DA_ERR_INVALID_ARGUMENT;
    const int dev = current_device();
    if (dev < 0) return DA_ERR_CUDA;
    unsigned* ptr = device_error_ptr(dev);
    if (!ptr) return DA_ERR_CUDA;
    return launch_wait_check(ptr, static_cast<uint64_t>(limit_us) * 1000ull,
                             static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? DA_OK
               : DA_ERR_CUDA;
}

}  // extern "C"

namespace {

// Dense call with the length either known on the host (k_len_dev == nullptr) or read by the
// kernel from device memory (then k_len is ignored and capacity bounds everything).
da_status run_dense(const void* q, const void* k, const void* v, void* out, int B, int Hq, int Hkv,
                    int D, int64_t capacity, int64_t k_len, const uint32_t* k_len_dev,
                    float softmax_scale, void* workspace, size_t workspace_bytes, void* stream,
                    int sq = 1, int causal = 0, bool clear_workspace = false) {
    da_status st = check_common(q, out, B, Hq, Hkv, D, softmax_scale, workspace);
    if (st != DA_OK) return st;
    if (sq < 1) return DA_ERR_INVALID_ARGUMENT;
    if (padded_group((Hq / Hkv) * sq) == 0) return DA_ERR_UNSUPPORTED;
    if (!k || !v || !aligned(k, 16) || !aligned(v, 16)) return DA_ERR_INVALID_ARGUMENT;
    if (capacity < 1) return DA_ERR_INVALID_ARGUMENT;
    if (!k_len_dev && (k_len < 0 || k_len > capacity)) return DA_ERR_INVALID_ARGUMENT;
    if (k_len_dev && !aligned(k_len_dev, 4)) return DA_ERR_INVALID_ARGUMENT;
    if (capacity >= (1ll << 31)) return DA_ERR_UNSUPPORTED;
    const long long units = static_cast<long long>(B) * Hkv;
    const long long rows = k_len_dev ? capacity : k_len;      // most rows a call can attend
    const long long tiles = (rows + kTileKeys - 1) / kTileKeys;
    if (units * ((capacity + kTileKeys - 1) / kTileKeys) >= (1ll << 31)) return DA_ERR_UNSUPPORTED;
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    if (B == 0) return DA_OK;
    const int dev = current_device();
    if (dev < 0) return DA_ERR_CUDA;
    const int sms = sm_count(dev);
    if (sms <= 0) return DA_ERR_CUDA;
    const int G = Hq / Hkv, GP = padded_group(G * sq);
    const WsLayout w = ws_layout(units, units + sms, G * sq, D);
    if (workspace_bytes < w.total) return DA_ERR_WORKSPACE_TOO_SMALL;
    if (!k_len_dev && k_len == 0) return zero_output(out, B, Hq * sq, D, cs);

    Launch L{};
    const cuuint64_t row_bytes = static_cast<cuuint64_t>(D) * 2;
    // rows past the live length lie outside the descriptor when the host knows it, so they are
    // never read; with a device-resident length the descriptor spans the capacity and the last
    // tile's rows past the length are fetched but masked
    if (!encode_3d(&L.tm_k, k, D, rows, units, row_bytes, row_bytes * capacity, kTileKeys) ||
        !encode_3d(&L.tm_v, v, D, rows, units, row_bytes, row_bytes * capacity, kTileKeys))
        return DA_ERR_CUDA;
    L.p = base_params(q, out, B, Hq, Hkv, softmax_scale, device_error_ptr(dev));
    bind_workspace(L.p, workspace, w);
    L.p.k_len = static_cast<int>(rows);
    L.p.dense_tiles = static_cast<int>(tiles);
    L.p.k_len_dev = reinterpret_cast<const unsigned*>(k_len_dev);
    L.p.capacity = static_cast<int>(capacity);
    L.p.sq = sq;
    L.p.causal = causal ? 1 : 0;
    L.p.seg_heads = G * sq;
    // Whole units, one per CTA, when they are about as many as the SMs (the units of a dense
    // call have equal lengths, so they then stream without any split, on at least 80% of the
    // SMs, whatever the length), or when the host knows they are short (splitting would trade a
    // few tiles of streaming for a cross-CTA merge that costs more); otherwise every tile is
    // spread over all SMs.
    const bool near_sms = 5 * units >= 4LL * sms && units <= sms;
    const bool whole_units = near_sms || (!k_len_dev && tiles <= kShortUnitTiles);
    const long long spread = whole_units ? units : units * tiles;
    L.grid = static_cast<int>(std::min<long long>(persistent_ctas(dev), spread));
    L.stream = cs;
    L.threads = Roles<kDense>::kThreads;
    // the merge counters are all that must start at zero (partial rows are written before any
    // CTA reads them)
    if (clear_workspace && cudaMemsetAsync(workspace, 0, w.lse - w.counters, cs) != cudaSuccess)
        return DA_ERR_CUDA;
    return launch_dense(D, GP, L) == cudaSuccess ? DA_OK : DA_ERR_CUDA;
}

}  // namespace

namespace da {

da_status dense_clearing_workspace(const void* q, const void* k, const void* v, void* out, int B,
                                   int Hq, int Hkv, int D, int64_t capacity, int64_t k_len,
                                   float softmax_scale, void* workspace, size_t workspace_bytes,
                                   void* stream) {
    return run_dense(q, k, v, out, B, Hq, Hkv, D, capacity, k_len, nullptr, softmax_scale,
                     workspace, workspace_bytes, stream, 1, 0, true);
}

}  // namespace da

extern "C" {

da_status decode_attn_dense(const void* q, const void* k, const void* v, void* out, int B, int Hq,
                            int Hkv, int D, int64_t capacity, int64_t k_len, float softmax_scale,
                            void* workspace, size_t workspace_bytes, void* stream) {
    return run_dense(q, k, v, out, B, Hq, Hkv, D, capacity, k_len, nullptr, softmax_scale,
                     workspace, workspace_bytes, stream);
}

da_status decode_attn_dense_device_len(const void* q, const void* k, const void* v, void* out,
                                       int B, int Hq, int Hkv, int D, int64_t capacity,
                                       const uint32_t* k_len, float softmax_scale, void* workspace,
                                       size_t workspace_bytes, void* stream) {
    if (!k_len) return DA_ERR_INVALID_ARGUMENT;
    return run_dense(q, k, v, out, B, Hq, Hkv, D, capacity, 0, k_len, softmax_scale, workspace,
                     workspace_bytes, stream);
}

}  // extern "C"

namespace {

da_status run_paged(const void* q, const void* k_pool, const void* v_pool, void* out,
                    const int32_t* block_table, int max_pages_per_seq, int page_size,
                    int64_t num_pages, const uint32_t* kv_lens, int kv_len_stride, int B, int Hq,
                    int Hkv, int D, float softmax_scale, void* workspace, size_t workspace_bytes,
                    void* stream, int sq, int causal) {
    da_status st = check_common(q, out, B, Hq, Hkv, D, softmax_scale, workspace);
    if (st != DA_OK) return st;
    if (sq < 1) return DA_ERR_INVALID_ARGUMENT;
    if (padded_group((Hq / Hkv) * sq) == 0) return DA_ERR_UNSUPPORTED;
    if (!k_pool || !v_pool || !aligned(k_pool, 16) || !aligned(v_pool, 16)) return DA_ERR_INVALID_ARGUMENT;
    if (!block_table || !kv_lens || !aligned(block_table, 4) || !aligned(kv_lens, 4))
        return DA_ERR_INVALID_ARGUMENT;
    if (max_pages_per_seq < 1 || page_size < 1 || num_pages < 1) return DA_ERR_INVALID_ARGUMENT;
    if (kv_len_stride != 1 && kv_len_stride != 3) return DA_ERR_INVALID_ARGUMENT;
    if (page_size < 8 || page_size > 256 || (page_size & (page_size - 1)) != 0) return DA_ERR_UNSUPPORTED;
    if (num_pages >= (1ll << 31)) return DA_ERR_UNSUPPORTED;
    if (B > kMaxPagedBatch) return DA_ERR_UNSUPPORTED;
    const long long cap = static_cast<long long>(max_pages_per_seq) * page_size;
    if (cap >= (1ll << 31)) return DA_ERR_UNSUPPORTED;
    const long long units = static_cast<long long>(B) * Hkv;
    if (units * ((cap + kTileKeys - 1) / kTileKeys) >= (1ll << 31)) return DA_ERR_UNSUPPORTED;
    if (static_cast<long long>(Hkv) * page_size >= (1ll << 31)) return DA_ERR_UNSUPPORTED;
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    if (B == 0) return DA_OK;
    const int dev = current_device();
    if (dev < 0) return DA_ERR_CUDA;
    const int sms = sm_count(dev);
    if (sms <= 0) return DA_ERR_CUDA;
    const int G = Hq / Hkv;
    Launch L{};
    const cuuint64_t row_bytes = static_cast<cuuint64_t>(D) * 2;
    const cuuint64_t page_bytes = row_bytes * page_size * Hkv;
    // Pools viewed as [num_pages][Hkv * page_size rows][D]; a box is min(kh * page_size, 64)
    // rows of one page (kh adjacent heads) by one 64-column half.
    const int kh = paged_kv_heads(Hkv, G * sq, page_size);
    const cuuint32_t rows = static_cast<cuuint32_t>(std::min(kh * page_size, kTileKeys));
    if (!encode_3d(&L.tm_k, k_pool, D, static_cast<cuuint64_t>(Hkv) * page_size, num_pages,
                   row_bytes, page_bytes, rows) ||
        !encode_3d(&L.tm_v, v_pool, D, static_cast<cuuint64_t>(Hkv) * page_size, num_pages,
                   row_bytes, page_bytes, rows))
        return DA_ERR_CUDA;
    const int GP = padded_group(kh * G * sq);
    const long long punits = units / kh;
    const WsLayout w = ws_layout(punits, punits + sms, kh * G * sq, D);
    if (workspace_bytes < w.total) return DA_ERR_WORKSPACE_TOO_SMALL;
    L.p = base_params(q, out, B, Hq, Hkv, softmax_scale, device_error_ptr(dev));
    bind_workspace(L.p, workspace, w);
    L.p.block_table = block_table;
    L.p.max_pages = max_pages_per_seq;
    L.p.page_size = page_size;
    L.p.num_pages = static_cast<int>(num_pages);
    L.p.kv_lens = kv_lens;
    L.p.kv_stride = kv_len_stride;
    L.p.kh = kh;
    L.p.tile_keys = kTileKeys / kh;
    L.p.seg_heads = kh * G * sq;
    L.p.sq = sq;
    L.p.causal = causal ? 1 : 0;
    L.grid = persistent_ctas(dev);
    L.stream = cs;
    L.threads = Roles<kPaged>::kThreads;
    // Each consumer warp's 16 rows lie in one KV head when pages hold >= 16 rows; with <= 8
    // query columns per KV head the warp then needs only that head's columns.
    const bool warp_head = kh > 1 && page_size >= 16 && G * sq <= 8 && GP == 16;
    const cudaError_t e = kh == 1 ? launch_paged_single(D, GP, L)
                                  : launch_paged_multi(D, GP, warp_head, L);
    return e == cudaSuccess ? DA_OK : DA_ERR_CUDA;
}

}  // namespace

extern "C" {

da_status decode_attn_paged(const void* q, const void* k_pool, const void* v_pool, void* out,
                            const int32_t* block_table, int max_pages_per_seq, int page_size,
                            int64_t num_pages, const uint32_t* kv_lens, int kv_len_stride, int B,
                            int Hq, int Hkv, int D, float softmax_scale, void* workspace,
                            size_t workspace_bytes, void* stream) {
    return run_paged(q, k_pool, v_pool, out, block_table, max_pages_per_seq, page_size, num_pages,
                     kv_lens, kv_len_stride, B, Hq, Hkv, D, softmax_scale, workspace,
                     workspace_bytes, stream, 1, 0);
}

da_status decode_attn_paged_mq(const void* q, const void* k_pool, const void* v_pool, void* out,
                               const int32_t* block_table, int max_pages_per_seq, int page_size,
                               int64_t num_pages, const uint32_t* kv_lens, int kv_len_stride,
                               int B, int Hq, int Hkv, int D, int Sq, int causal,
                               float softmax_scale, void* workspace, size_t workspace_bytes,
                               void* stream) {
    return run_paged(q, k_pool, v_pool, out, block_table, max_pages_per_seq, page_size, num_pages,
                     kv_lens, kv_len_stride, B, Hq, Hkv, D, softmax_scale, workspace,
                     workspace_bytes, stream, Sq, causal);
}

da_status decode_attn_dense_mq(const void* q, const void* k, const void* v, void* out, int B,
                               int Hq, int Hkv, int D, int Sq, int causal, int64_t capacity,
                               int64_t k_len, float softmax_scale, void* workspace,
                               size_t workspace_bytes, void* stream) {
    return run_dense(q, k, v, out, B, Hq, Hkv, D, capacity, k_len, nullptr, softmax_scale,
                     workspace, workspace_bytes, stream, Sq, causal);
}

da_status decode_attn_sparse(const void* q, const void* k_pool, const void* v_pool, void* out,
                             int64_t pool_rows, const int32_t* sel, int width, int B, int Hq,
                             int Hkv, int D, float softmax_scale, void* workspace,
                             size_t workspace_bytes, void* stream) {
    da_status st = check_common(q, out, B, Hq, Hkv, D, softmax_scale, workspace);
    if (st != DA_OK) return st;
    if (!k_pool || !v_pool || !aligned(k_pool, 16) || !aligned(v_pool, 16)) return DA_ERR_INVALID_ARGUMENT;
    if (width < 0 || pool_rows < 1) return DA_ERR_INVALID_ARGUMENT;
    if (width > 0 && (!sel || !aligned(sel, 4))) return DA_ERR_INVALID_ARGUMENT;
    if (pool_rows >= (1ll << 31)) return DA_ERR_UNSUPPORTED;
    const long long units = static_cast<long long>(B) * Hkv;
    const int G = Hq / Hkv;
    const long long chunks = sparse_chunks(width);
    if (units * chunks >= (1ll << 31)) return DA_ERR_UNSUPPORTED;
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    if (B == 0) return DA_OK;
    const int dev = current_device();
    if (dev < 0) return DA_ERR_CUDA;
    const int GP = sparse_padded_group(G);
    const WsLayout w = ws_layout(units, units * chunks, G, D);
    if (workspace_bytes < w.total) return DA_ERR_WORKSPACE_TOO_SMALL;
    if (width == 0) return zero_output(out, B, Hq, D, cs);

    Launch L{};
    L.p = base_params(q, out, B, Hq, Hkv, softmax_scale, device_error_ptr(dev));
    bind_workspace(L.p, workspace, w);
    L.p.sel = sel;
    L.p.width = width;
    L.p.pool_rows = static_cast<int>(pool_rows);
    L.p.nchunks = static_cast<int>(chunks);
    L.p.seg_heads = G;
    L.p.k_pool = static_cast<const __nv_bfloat16*>(k_pool);
    L.p.v_pool = static_cast<const __nv_bfloat16*>(v_pool);
    L.stream = cs;
    if (sparse_uses_tc(G, D)) {
        // one CTA per (unit, chunk)
        L.grid = static_cast<int>(units * chunks);
        L.threads = sparse_tc_threads();
        return launch_sparse_tc(D, L) == cudaSuccess ? DA_OK : DA_ERR_CUDA;
    }
    // persistent: each CTA takes a contiguous range of whole (unit, chunk) items
    L.grid = static_cast<int>(std::min<long long>(persistent_ctas(dev), units * chunks));
    L.threads = Roles<kSparse>::kThreads;
    return launch_sparse(D, GP, L) == cudaSuccess ? DA_OK : DA_ERR_CUDA;
}

}  // extern "C"
