// Sparse decode attention on the fifth-generation tensor cores (tcgen05), for units of 33..64
// query heads per KV head at head dim 64 or 128.
//
// Why a second sparse kernel.  The mma.sync kernel holds at most 32 query columns, so a larger
// group would be split into groups of 32 with every selected row gathered once per group, and
// its warp-level MMAs bound the per-tile time.  Here one CTA holds all of the unit's heads: the
// group is a real dense tile (S = Q K^T is 128 x 64 x D with the heads zero-padded to 128
// rows), so both products run as tcgen05.mma with the accumulators in tensor memory.
//
// Work split.  CTA = (unit u = (b, g), chunk of 512 selection entries); the chunk depends on
// nothing but the kernel, so trailing -1 pads cannot move a chunk boundary.  Chunk pieces are
// merged across CTAs by log-sum-exp exactly as in the mma.sync kernel (partial rows, a per-unit
// counter, the last CTA merges in segment order).
//
// Inside a CTA (12 warps; warp w issues on the SM's scheduler w % 4, and the two softmax warps
// that hold heads run on schedulers 0 and 1, so the producers are warps 6, 7, 10 and 11, on
// schedulers 2 and 3 — 2.3% faster per call than sharing the softmax warps' schedulers — and
// warps 5, 8 and 9 exit after the set-up):
//   warps 6, 7, 10, 11  producers: gather the chunk's selected K and V rows with 16-byte
//              cp.async into a 128 KB ring of stages (64 rows of K and of V each: 4 stages at
//              D = 128, 8 at D = 64; 128-byte swizzle; rows outside [0, pool_rows)
//              zero-filled); a stage's full barrier completes when every producer thread's
//              copies for it have landed (cp.async.mbarrier.arrive), so the producers run ahead
//              as far as the ring allows;
//   warp 4     allocates 256 TMEM columns; one lane issues S(t) = Q K(t)^T into one of two
//              64-column S buffers and O += P(t) V(t) into the D-column O accumulator (after
//              acquiring a stage it fences the generic proxy, in which cp.async wrote the rows,
//              against the async proxy the MMAs read them through);
//   warps 0-3  softmax: thread h owns query head h (TMEM lane h).  It reads its row of S(t),
//              masks invalid rows, updates the running maximum and sum, writes its bf16 weights
//              P(t) into a shared-memory P buffer (the A operand of the second MMA) and, at the
//              end, normalises its O row; the rows go through shared memory so the stores of
//              the output (one chunk) or of the partial rows and log-sum-exps are coalesced.
//              The last CTA of a unit merges: up to four chunks from shared memory, filled by
//              bulk copies (tc_merge), more with merge_unit, in the same arithmetic.
// The running maximum used for the weights only moves when a tile's maximum exceeds it by more
// than 8 (log2 units); the O row is rescaled in TMEM then.  Weights are therefore at most 2^8
// before bf16 rounding, and the result is the same softmax with a different reference point.
//
// Safety.  Every wait is bounded (about one second) and raises the CTA's abort flag on timeout;
// the MMA warp waits for all of its MMAs and for the softmax warps' last TMEM access before it
// frees the tensor memory, on every path.
#include "launch.h"

namespace da {
namespace {

constexpr int kTcM = 128;                        // MMA rows: the unit's query heads, zero-padded
constexpr int kTcChunk = kSparseChunkUnit;       // selection entries per CTA (512)
constexpr int kTcPBytes = kTcM * kTileKeys * 2;  // [128 rows][128 B]: one tile's bf16 weights
constexpr int kTcSoftmaxWarps = 4;
constexpr int kTcMmaWarp = 4;
constexpr int kTcProducerWarps = 4;
constexpr int kTcThreads = 32 * 12;               // producers on warps 6, 7, 10, 11 (see above)
static_assert(kTcProducerWarps == 4, "the producers are warps 6, 7, 10 and 11");
constexpr uint32_t kTcCols = 256;                // TMEM: S buffers at columns 0 and 64, O at 128
constexpr uint32_t kTcColO = 128;
constexpr float kTcRescaleLog2 = 8.f;
constexpr int kTcRingBytes = 128 * 1024;         // the stage ring
constexpr int kTcMaxStages = 8;
constexpr int kTcMergeSegments = 4;              // tc_merge stages up to this many segments

// Head-dim dependent sizes and the shared-memory layout (from a 1024-byte aligned base).
template <int D>
struct TcGeom {
    static_assert(D == 64 || D == 128, "head dim");
    static constexpr int kHalves = D / 64;                     // 64-column (128-byte) halves
    static constexpr int kTileBytes = kTileKeys * D * 2;       // one K (or V) tile
    static constexpr int kStageBytes = 2 * kTileBytes;
    static constexpr int kStages = kTcRingBytes / kStageBytes; // 4 at D 128, 8 at D 64
    static constexpr int kQBytes = kTcM * D * 2;               // [halves][128 rows][128 B]
    static constexpr int kD4 = D / 4;                          // float4 columns of a row
    static constexpr int kHeadsPerInstr = 32 / kD4;            // rows one warp access covers
    static constexpr int kRowStride = D + 4;                   // floats between staged O rows
    static constexpr int kOffQ = kTcRingBytes;
    static constexpr int kOffP = kOffQ + kQBytes;
    static constexpr int kOffBar = kOffP + 2 * kTcPBytes;
    static constexpr int kOffIdx = kOffBar + 1024;
    static constexpr int kSmemBytes = 1024 + kOffIdx + kTcChunk * 4;
    static_assert(kStages <= kTcMaxStages, "stage ring");
    static_assert(kSmemBytes <= kSmemBudget, "shared memory");
    static_assert(64 * kRowStride * 4 <= kTcRingBytes, "staged O rows");
    static_assert(kTcMergeSegments * 64 * D * 4 <= kTcRingBytes, "merge rows");
    static_assert((kTcMergeSegments + 3) * 64 * 4 <= kQBytes, "merge weights");
};
static_assert(kTcSoftmaxWarps * 32 == kConsumerThreads, "the merge runs on the softmax warps");

struct TcBars {
    uint64_t full[kTcMaxStages];   // stage's K and V rows landed (count: producer threads + 1)
    uint64_t empty[kTcMaxStages];  // stage's P.V completed (tcgen05.commit)
    uint64_t s_ready[2];           // S buffer written (tcgen05.commit)
    uint64_t s_free[2];            // S buffer read by the softmax warps (count: active warps)
    uint64_t p_ready[2];           // P buffer written, O rescaled (count: active warps)
    uint64_t pv_done[2];           // P.V of the tile with this parity completed (tcgen05.commit)
    uint64_t q_ready;              // Q in shared memory (count: softmax threads)
    uint64_t tmem_done;            // softmax warps finished with TMEM (count: softmax warps)
    uint64_t drain;                // every MMA issued so far completed (tcgen05.commit)
    uint64_t group;                // softmax-warp group barrier of the merge
    uint64_t mrows;                // merge: the partial rows landed (bulk copies)
    uint64_t stage_mask[kTcMaxStages];
    uint32_t tmem_base;
    int abort;
    int last_flag;
};
static_assert(sizeof(TcBars) <= 1024, "barrier block");

// Merges the nseg <= kTcMergeSegments partial rows of a unit of G <= 64 heads (workspace
// segments first_seg, ...; one segment's rows are G * D * 4 contiguous bytes) by log-sum-exp in
// segment order and stores its bf16 output rows; runs on the 128 softmax threads.  The arithmetic
// is merge_unit's: the maximum over every segment's LSE, weights exp2(lse - max) of the live
// segments summed in segment order from the first live one, rows accumulated in the same order by
// fma from zero, the output acc * (1 / sum), and a head with a single live segment copies that
// segment's row.  All rows land in `rows_sm` (the idle stage ring) by bulk copies that thread 0
// issues while the per-head weights are formed in `w_sm`; a warp access then covers
// kHeadsPerInstr heads (lane = one float4 column of one of them), and a thread takes its heads
// four at a time with every load of a pass in flight.  The caller has acquired every segment's
// rows (the unit's counter) before the call.
// pick ? a : b, component by component, as a select instruction (kept a select, so that a chain
// of them over a register array never becomes an indexed access to local memory)
__device__ __forceinline__ float4 select4(bool pick, const float4& a, const float4& b) {
    float4 r;
    asm("{\n\t.reg .pred q;\n\tsetp.ne.u32 q, %8, 0;\n\t"
        "selp.f32 %0, %4, %9, q;\n\tselp.f32 %1, %5, %10, q;\n\t"
        "selp.f32 %2, %6, %11, q;\n\tselp.f32 %3, %7, %12, q;\n\t}"
        : "=f"(r.x), "=f"(r.y), "=f"(r.z), "=f"(r.w)
        : "f"(a.x), "f"(a.y), "f"(a.z), "f"(a.w), "r"(static_cast<unsigned>(pick)), "f"(b.x),
          "f"(b.y), "f"(b.z), "f"(b.w));
    return r;
}

template <int D>
__device__ __forceinline__ bool tc_merge(const Params& p, const SmemPtrs& sm, float* w_sm,
                                         unsigned char* rows_sm, uint64_t* mrows, int hq0, int G,
                                         int first_seg, int nseg, uint32_t& gphase) {
    using Tg = TcGeom<D>;
    constexpr int D4 = Tg::kD4;
    constexpr int R = Tg::kHeadsPerInstr;                    // heads per warp access
    constexpr int kHeadsPerThread = 64 / (kTcSoftmaxWarps * R);
    constexpr int kPass = 4;                                 // heads per pass and thread
    const int tid = threadIdx.x, wv = tid >> 5;
    const int c = (tid & 31) % D4, sub = (tid & 31) / D4;
    auto head_of = [&](int j) { return (wv + kTcSoftmaxWarps * j) * R + sub; };
    const size_t SH = static_cast<size_t>(p.seg_heads);
    const uint32_t seg_bytes = static_cast<uint32_t>(G) * D * 4;
    const float* lse = p.part_lse + static_cast<size_t>(first_seg) * SH;
    const float4* src =
        reinterpret_cast<const float4*>(p.part_o) + static_cast<size_t>(first_seg) * SH * D4;
    const float4* rs = reinterpret_cast<const float4*>(rows_sm);
    // per head h: its segments' weights in w4[h] and {1 / sum, live count, last live segment}
    // in h_meta[h], one 16-byte load each
    static_assert(kTcMergeSegments == 4, "one float4 of weights per head");
    float4* w4 = reinterpret_cast<float4*>(w_sm);            // [64]
    float4* h_meta = w4 + 64;                                // [64]
    if (tid == 0) {
        fence_proxy_async_global();
        mbar_arrive_expect_tx(mrows, nseg * seg_bytes);
        for (int k = 0; k < nseg; ++k)
            bulk_load(rows_sm + k * seg_bytes, src + static_cast<size_t>(k) * SH * D4, seg_bytes,
                      mrows);
    }
    if (tid < G) {
        float l[kTcMergeSegments];
        float M = -CUDART_INF_F;
#pragma unroll
        for (int k = 0; k < kTcMergeSegments; ++k) {
            l[k] = k < nseg ? __ldcg(lse + static_cast<size_t>(k) * SH + tid) : -CUDART_INF_F;
            M = fmaxf(M, l[k]);
        }
        float L = 0.f;
        int live = 0, only = 0;
        float w[kTcMergeSegments];
#pragma unroll
        for (int k = 0; k < kTcMergeSegments; ++k) {
            w[k] = 0.f;
            if (l[k] != -CUDART_INF_F) {
                w[k] = fast_exp2(l[k] - M);
                L = live ? L + w[k] : w[k];
                ++live;
                only = k;
            }
        }
        w4[tid] = make_float4(w[0], w[1], w[2], w[3]);
        h_meta[tid] = make_float4(live ? 1.0f / L : 0.f, __int_as_float(live),
                                  __int_as_float(only), 0.f);
    }
    if (!mbar_wait_warp(mrows, 0, sm.abort)) {
        *sm.abort = 1;
        record_error(p.err, kErrWaitFull);
        // the copies in flight land before the CTA can exit
        if (tid == 0 && !mbar_wait(mrows, 0, nullptr, kWaitLimitNs)) record_error(p.err, kErrDrain);
        return false;
    }
    if (!group_sync(sm, gphase, p.err)) return false;   // weights visible
    // Every load of a pass (the heads' statistics and all their segments' weights and rows) is
    // independent of the others and predicated rather than branched around, so they are all in
    // flight together.
#pragma unroll 1
    for (int j0 = 0; j0 < kHeadsPerThread; j0 += kPass) {
        int live[kPass], only[kPass];
        float inv[kPass];
        float w[kTcMergeSegments][kPass];
#pragma unroll
        for (int j = 0; j < kPass; ++j) {
            const int hj = head_of(j0 + j);
            const int h = min(hj, G - 1);
            const float4 m = h_meta[h];
            const float4 wj = w4[h];
            inv[j] = m.x;
            live[j] = __float_as_int(m.y);
            only[j] = __float_as_int(m.z);
            // a head past G contributes nothing (its store is skipped too)
            w[0][j] = hj < G ? wj.x : 0.f;
            w[1][j] = hj < G ? wj.y : 0.f;
            w[2][j] = hj < G ? wj.z : 0.f;
            w[3][j] = hj < G ? wj.w : 0.f;
        }
        float4 o[kTcMergeSegments][kPass];
#pragma unroll
        for (int k = 0; k < kTcMergeSegments; ++k)
#pragma unroll
            for (int j = 0; j < kPass; ++j) {
                const int h = min(head_of(j0 + j), G - 1);
                o[k][j] = rs[(min(k, nseg - 1) * G + h) * D4 + c];
            }
#pragma unroll
        for (int j = 0; j < kPass; ++j) {
            // segment order; a dead segment (w == 0) leaves the accumulator as it is
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int k = 0; k < kTcMergeSegments; ++k) {
                const float4 f = fma4(w[k][j], o[k][j], acc);
                acc = w[k][j] != 0.f ? f : acc;
            }
            const int h = head_of(j0 + j);
            float4 single = o[0][j];
#pragma unroll
            for (int k = 1; k < kTcMergeSegments; ++k)
                single = select4(k == only[j], o[k][j], single);
            const float4 scaled =
                make_float4(acc.x * inv[j], acc.y * inv[j], acc.z * inv[j], acc.w * inv[j]);
            const float4 v =
                live[j] == 1 ? single : (live[j] > 1 ? scaled : make_float4(0.f, 0.f, 0.f, 0.f));
            if (h < G)
                *reinterpret_cast<uint2*>(p.out + static_cast<size_t>(hq0 + h) * D + 4 * c) =
                    make_uint2(pack_bf16x2(v.x, v.y), pack_bf16x2(v.z, v.w));
        }
    }
    return true;
}

template <int D>
__global__ void __launch_bounds__(kTcThreads, 1)
sparse_tc_kernel(const __grid_constant__ CUtensorMap, const __grid_constant__ CUtensorMap,
                 const Params p) {
    using Tg = TcGeom<D>;
    constexpr int S = Tg::kStages;
    extern __shared__ unsigned char smem_raw[];
    // 1024-byte aligned by an offset into the shared array, so accesses through `base` stay
    // shared-memory accesses for the compiler
    unsigned char* base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    TcBars& bar = *reinterpret_cast<TcBars*>(base + Tg::kOffBar);
    int* sidx = reinterpret_cast<int*>(base + Tg::kOffIdx);
    volatile int* abort = &bar.abort;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = p.G;
    const int nact = (G + 31) >> 5;              // softmax warps that hold real heads

    const int u = blockIdx.x / p.nchunks;
    const int chunk = blockIdx.x - u * p.nchunks;
    const int key0 = chunk * kTcChunk;
    const int nkeys = min(kTcChunk, p.width - key0);
    const int ntiles = (nkeys + kTileKeys - 1) / kTileKeys;
    const int b = u / p.Hkv, g = u - b * p.Hkv;
    const int hq0 = b * p.Hq + g * G;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&bar.full[s], 32 * kTcProducerWarps + 1);
            mbar_init(&bar.empty[s], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bar.s_ready[i], 1);
            mbar_init(&bar.s_free[i], nact);
            mbar_init(&bar.p_ready[i], nact);
            mbar_init(&bar.pv_done[i], 1);
        }
        mbar_init(&bar.q_ready, 32 * kTcSoftmaxWarps);
        mbar_init(&bar.tmem_done, kTcSoftmaxWarps);
        mbar_init(&bar.drain, 1);
        mbar_init(&bar.group, kConsumerThreads);
        mbar_init(&bar.mrows, 1);
        bar.abort = 0;
        bar.last_flag = 0;
        fence_mbarrier_init();
    }
    if (warp == kTcMmaWarp) {
        tmem_alloc(&bar.tmem_base, kTcCols);
        tmem_relinquish_alloc_permit();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = bar.tmem_base;
    // nothing above touched global memory
    grid_dependency_wait();
    allow_dependent_launch();

    if (warp > kTcMmaWarp) {
        // ============================================================ producer warps
        if ((warp & 3) < 2) return;                          // warps 5, 8, 9: no role
        const int pw = (warp & 1) + ((warp >> 3) << 1);      // warps 6, 7, 10, 11 -> 0..3
        const int ptid = pw * 32 + lane;
        const int* selrow = p.sel + static_cast<size_t>(b) * p.width + key0;
        for (int i = ptid; i < nkeys; i += 32 * kTcProducerWarps) {
            const int idx = __ldg(selrow + i);
            sidx[i] = (idx >= 0 && idx < p.pool_rows) ? idx : -1;
        }
        asm volatile("bar.sync 1, %0;" ::"r"(32 * kTcProducerWarps) : "memory");   // producers only
        // a warp instruction copies kRowsPerInstr rows: in each group of 2 * CH lanes the first CH
        // copy the 16-byte chunks of a K row, the other CH those of the V row
        constexpr int CH = D / 8;
        constexpr int kRowsPerInstr = 32 / (2 * CH);
        const int sub = lane / (2 * CH), w = lane % (2 * CH);
        const bool isv = w >= CH;
        const int c = isv ? w - CH : w;
        const __nv_bfloat16* pool = (isv ? p.v_pool : p.k_pool) +
                                    static_cast<size_t>(u) * p.pool_rows * D + c * 8;
        constexpr int kRowsPerWarp = kTileKeys / kTcProducerWarps;
        bool ok = true;
        int t = 0;
        for (; t < ntiles; ++t) {
            const int s = t % S;
            if (!mbar_wait_warp(&bar.empty[s], ((t / S) & 1) ^ 1u, abort)) {
                ok = false;
                break;
            }
            const int l0 = t * kTileKeys;
            if (pw == 0) {
                const int i0 = l0 + lane, i1 = l0 + 32 + lane;
                const bool v0 = i0 < nkeys && sidx[i0] >= 0;
                const bool v1 = i1 < nkeys && sidx[i1] >= 0;
                const uint64_t mask = static_cast<uint64_t>(__ballot_sync(0xffffffffu, v0)) |
                                      (static_cast<uint64_t>(__ballot_sync(0xffffffffu, v1)) << 32);
                if (lane == 0) bar.stage_mask[s] = mask;
            }
            unsigned char* tile = base + s * Tg::kStageBytes + (isv ? Tg::kTileBytes : 0);
#pragma unroll 8
            for (int rb = pw * kRowsPerWarp; rb < (pw + 1) * kRowsPerWarp; rb += kRowsPerInstr) {
                const int r = rb + sub;
                const int li = l0 + r;
                const int idx = li < nkeys ? sidx[li] : -1;
                const bool valid = idx >= 0;
                cp_async_16(tile + tile_offset<Tg::kHalves>(r, c, 6),
                            pool + static_cast<size_t>(valid ? idx : 0) * D, valid ? 16u : 0u);
            }
            cp_async_arrive_noinc(&bar.full[s]);
            if (ptid == 0) mbar_arrive(&bar.full[s]);   // publishes the stage mask
        }
        if (!ok) {
            // let every copy this thread issued land before the CTA can exit
            cp_async_wait_all();
            *abort = 1;
            record_error(p.err, kErrWaitEmpty);
        }
        return;
    }

    if (warp == kTcMmaWarp) {
        // ============================================================ MMA warp
        if (lane == 0) {
            constexpr uint32_t kIdS = umma_idesc_bf16(kTcM, kTileKeys, false);
            constexpr uint32_t kIdO = umma_idesc_bf16(kTcM, D, true);
            const uint32_t q_s = smem_u32(base + Tg::kOffQ);
            // S(t) = Q K(t)^T into S buffer t % 2: A = Q (K-major), B = the K tile (K-major)
            auto issue_s = [&](int t) -> bool {
                const int s = t % S, sb = t & 1;
                if (!mbar_wait(&bar.full[s], (t / S) & 1, abort, kWaitLimitNs)) return false;
                if (t >= 2 && !mbar_wait(&bar.s_free[sb], ((t - 2) >> 1) & 1, abort, kWaitLimitNs))
                    return false;
                fence_proxy_async_smem();
                tc_fence_after_sync();
                const uint32_t k_s = smem_u32(base + s * Tg::kStageBytes);
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    const uint32_t off = (ks & 3) * 32u;   // 16 dims = 32 B into the swizzled row
                    const uint64_t a =
                        umma_desc_sw128(q_s + (ks >> 2) * (kTcM * 128) + off, 16, 1024);
                    const uint64_t bd =
                        umma_desc_sw128(k_s + (ks >> 2) * (kTileKeys * 128) + off, 16, 1024);
                    umma_bf16(tmem + sb * kTileKeys, a, bd, kIdS, ks > 0 ? 1u : 0u);
                }
                umma_commit(&bar.s_ready[sb]);
                return true;
            };
            bool ok = mbar_wait(&bar.q_ready, 0, abort, kWaitLimitNs);
            if (ok) {
                tc_fence_after_sync();
                ok = issue_s(0);
            }
            for (int t = 0; ok && t < ntiles; ++t) {
                if (t + 1 < ntiles && !issue_s(t + 1)) {
                    ok = false;
                    break;
                }
                const int s = t % S, pb = t & 1;
                if (!mbar_wait(&bar.p_ready[pb], (t >> 1) & 1, abort, kWaitLimitNs)) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                // O += P(t) V(t): A = P (K-major), B = the V tile (MN-major: dims contiguous)
                const uint32_t p_s = smem_u32(base + Tg::kOffP + pb * kTcPBytes);
                const uint32_t v_s = smem_u32(base + s * Tg::kStageBytes + Tg::kTileBytes);
#pragma unroll
                for (int ks = 0; ks < kTileKeys / 16; ++ks) {
                    const uint64_t a = umma_desc_sw128(p_s + ks * 32, 16, 1024);
                    const uint64_t bd = umma_desc_sw128(v_s + ks * 16 * 128, kTileKeys * 128, 1024);
                    umma_bf16(tmem + kTcColO, a, bd, kIdO, (t > 0 || ks > 0) ? 1u : 0u);
                }
                umma_commit(&bar.pv_done[pb]);
                umma_commit(&bar.empty[s]);
            }
            if (!ok) {
                *abort = 1;
                record_error(p.err, kErrWaitFull);
            }
            // every MMA issued above completes, and the softmax warps are done with TMEM,
            // before the columns are freed
            umma_commit(&bar.drain);
            if (!mbar_wait(&bar.drain, 0, nullptr, kWaitLimitNs)) record_error(p.err, kErrDrain);
            if (!mbar_wait(&bar.tmem_done, 0, nullptr, kWaitLimitNs))
                record_error(p.err, kErrDrain);
        }
        __syncwarp();
        tc_fence_after_sync();
        tmem_dealloc(tmem, kTcCols);
        return;
    }

    // ================================================================ softmax warps
    const int h = threadIdx.x;                   // query head of this thread = its TMEM lane
    const bool warp_active = warp < nact;
    const bool live = h < G;
    const uint32_t t_lane = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    {
        // Q rows of the unit (zero past G) in the A-operand layout; zero P rows past G
        unsigned char* qs = base + Tg::kOffQ;
        constexpr int CQ = D / 8;                                     // 16-byte chunks per row
        constexpr int kPer = kTcM * CQ / kConsumerThreads;            // 16-byte chunks per thread
        uint4 v[kPer];
#pragma unroll
        for (int k = 0; k < kPer; ++k) {
            const int i = threadIdx.x + k * kConsumerThreads, r = i / CQ, c = i % CQ;
            v[k] = r < G ? __ldg(reinterpret_cast<const uint4*>(p.q +
                                 static_cast<size_t>(hq0 + r) * D) + c)
                         : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int k = 0; k < kPer; ++k) {
            const int i = threadIdx.x + k * kConsumerThreads, r = i / CQ, c = i % CQ;
            *reinterpret_cast<uint4*>(qs + (c >> 3) * (kTcM * 128) + r * 128 +
                                      (((c ^ r) & 7) << 4)) = v[k];
        }
        // (each thread starts at its own swizzled 16-byte slot, so the eight rows a quarter warp
        // writes at once fall in different banks)
        if (!live)
            for (int i = 0; i < 2 * (kTileKeys / 8); ++i)
                *reinterpret_cast<uint4*>(base + Tg::kOffP + (i >> 3) * kTcPBytes + h * 128 +
                                          (((i ^ h) & 7) << 4)) = make_uint4(0u, 0u, 0u, 0u);
        fence_proxy_async_smem();
        mbar_arrive(&bar.q_ready);
    }

    float m_run = -CUDART_INF_F;   // reference maximum of the weights (log2 domain)
    float l_run = 0.f;             // sum of the bf16-rounded weights
    bool ok = true;
    if (warp_active) {
        for (int t = 0; t < ntiles; ++t) {
            const int s = t % S, sb = t & 1;
            if (!mbar_wait_warp(&bar.full[s], (t / S) & 1, abort) ||
                !mbar_wait_warp(&bar.s_ready[sb], (t >> 1) & 1, abort)) {
                ok = false;
                break;
            }
            tc_fence_after_sync();
            uint32_t sr[2][32];
            tmem_ld32(t_lane + sb * kTileKeys, sr[0]);
            tmem_ld32(t_lane + sb * kTileKeys + 32, sr[1]);
            tmem_wait_ld();
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar.s_free[sb]);

            // scores in the log2 domain, invalid rows at -inf
            const uint64_t mask = bar.stage_mask[s];
            float x[kTileKeys];
            float mt = -CUDART_INF_F;
#pragma unroll
            for (int j = 0; j < kTileKeys; ++j) {
                const float v = __uint_as_float(sr[j >> 5][j & 31]) * p.scale_log2;
                x[j] = ((mask >> j) & 1ull) ? v : -CUDART_INF_F;
                mt = fmaxf(mt, x[j]);
            }
            // move the reference maximum only on a large increase; O holds earlier weights
            // (and needs the same rescale) only once some row has been seen
            float alpha = 1.f;
            if (mt > m_run + kTcRescaleLog2) {
                alpha = fast_exp2(m_run - mt);   // 0 while m_run is -inf
                m_run = mt;
            }
            const bool rescale = alpha != 1.f && l_run > 0.f;
            if (__any_sync(0xffffffffu, rescale)) {
                // the accumulator holds P.V up to tile t - 1 once that MMA has completed
                if (!mbar_wait_warp(&bar.pv_done[(t - 1) & 1], ((t - 1) >> 1) & 1, abort)) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                const float a = rescale ? alpha : 1.f;
#pragma unroll
                for (int cb = 0; cb < D / 32; ++cb) {
                    uint32_t o[32];
                    tmem_ld32(t_lane + kTcColO + cb * 32, o);
                    tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * a);
                    tmem_st32(t_lane + kTcColO + cb * 32, o);
                }
                tmem_wait_st();
            }
            l_run *= alpha;

            // bf16 weights; the sum takes the rounded values
            const float m_use = m_run == -CUDART_INF_F ? 0.f : m_run;
            uint32_t pk[kTileKeys / 2];
            float lsum = 0.f;
#pragma unroll
            for (int j = 0; j < kTileKeys / 2; ++j) {
                const uint32_t w = live ? pack_bf16x2(fast_exp2(x[2 * j] - m_use),
                                                      fast_exp2(x[2 * j + 1] - m_use))
                                        : 0u;
                lsum += bf16_lo_to_f32(w) + bf16_hi_to_f32(w);
                pk[j] = w;
            }
            l_run += lsum;
            // this P buffer was last read by the P.V of tile t - 2
            if (t >= 2 && !mbar_wait_warp(&bar.pv_done[sb], ((t - 2) >> 1) & 1, abort)) {
                ok = false;
                break;
            }
            unsigned char* prow = base + Tg::kOffP + sb * kTcPBytes + h * 128;
#pragma unroll
            for (int c = 0; c < 8; ++c)
                *reinterpret_cast<uint4*>(prow + (((c ^ h) & 7) << 4)) =
                    make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
            fence_proxy_async_smem();
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar.p_ready[sb]);
        }
        if (ok && !mbar_wait_warp(&bar.pv_done[(ntiles - 1) & 1], ((ntiles - 1) >> 1) & 1, abort))
            ok = false;
    }

    // The normalised O rows go through shared memory (row h of the idle stage ring,
    // Tg::kRowStride floats apart) so that the global stores are coalesced: the output rows (one
    // chunk) or this chunk's partial rows and LSEs.
    const bool whole = p.nchunks == 1;
    const size_t SH = static_cast<size_t>(p.seg_heads);
    float* orow_sm = reinterpret_cast<float*>(base);
    if (warp_active && ok) {
        tc_fence_after_sync();
        const bool empty = !(l_run > 0.f);
        const float inv = empty ? 0.f : 1.0f / l_run;
#pragma unroll
        for (int cb = 0; cb < D / 32; cb += 2) {
            // two 32-column loads in flight per wait
            uint32_t o[2][32];
            tmem_ld32(t_lane + kTcColO + cb * 32, o[0]);
            tmem_ld32(t_lane + kTcColO + (cb + 1) * 32, o[1]);
            tmem_wait_ld();
            if (!live) continue;
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                float4* dst =
                    reinterpret_cast<float4*>(orow_sm + h * Tg::kRowStride + (cb + half) * 32);
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    dst[j] = make_float4(__uint_as_float(o[half][4 * j]) * inv,
                                         __uint_as_float(o[half][4 * j + 1]) * inv,
                                         __uint_as_float(o[half][4 * j + 2]) * inv,
                                         __uint_as_float(o[half][4 * j + 3]) * inv);
            }
        }
        if (!whole && live)
            p.part_lse[static_cast<size_t>(blockIdx.x) * SH + h] =
                empty ? -CUDART_INF_F : m_run + fast_log2(l_run);
    }
    tc_fence_before_sync();
    __syncwarp();
    if (lane == 0) mbar_arrive(&bar.tmem_done);
    if (!ok) {
        *abort = 1;
        record_error(p.err, kErrWaitFull);
        return;
    }
    SmemPtrs sm{};
    sm.merge_o = reinterpret_cast<float*>(base);
    sm.group = &bar.group;
    sm.abort = abort;
    sm.last_flag = &bar.last_flag;
    uint32_t gphase = 0;
    if (!group_sync(sm, gphase, p.err)) return;   // rows staged
    {
        // a warp access covers kHeadsPerInstr heads, lane = one float4 column of one of them; a
        // fixed trip count, so all of a thread's shared-memory loads are in flight before the
        // stores
        constexpr int D4 = Tg::kD4, R = Tg::kHeadsPerInstr;
        constexpr int kPer = 64 / (kTcSoftmaxWarps * R);
        const int c = lane % D4, sub = lane / D4;
        float4 v[kPer];
#pragma unroll
        for (int j = 0; j < kPer; ++j)
            v[j] = *reinterpret_cast<const float4*>(
                orow_sm + min((warp + kTcSoftmaxWarps * j) * R + sub, G - 1) * Tg::kRowStride +
                4 * c);
#pragma unroll
        for (int j = 0; j < kPer; ++j) {
            const int hh = (warp + kTcSoftmaxWarps * j) * R + sub;
            if (hh >= G) continue;
            if (whole)
                *reinterpret_cast<uint2*>(p.out + static_cast<size_t>(hq0 + hh) * D + 4 * c) =
                    make_uint2(pack_bf16x2(v[j].x, v[j].y), pack_bf16x2(v[j].z, v[j].w));
            else
                *reinterpret_cast<float4*>(p.part_o +
                    (static_cast<size_t>(blockIdx.x) * SH + hh) * D + 4 * c) = v[j];
        }
    }
    if (whole) return;

    // cross-CTA merge of the unit's chunks (the stage ring is free now and serves as scratch)
    Unit U{};
    U.b = b;
    U.g = g;
    U.u = u;
    U.hq0 = hq0;
    U.nh = G;
    U.cu = u;
    // the group barrier orders every thread's partial-row stores before thread 0's release on
    // the unit's counter; the CTA that completes the count acquires all chunks' rows there
    if (!group_sync(sm, gphase, p.err)) return;
    if (threadIdx.x == 0) {
        const unsigned prev = atomic_add_acq_rel_gpu(p.counters + u);
        *sm.last_flag = (prev == static_cast<unsigned>(p.nchunks - 1)) ? 1 : 0;
    }
    if (!group_sync(sm, gphase, p.err)) return;
    if (*sm.last_flag) {
        // the Q area holds the merge's per-segment weights and the stage ring its rows; more
        // chunks take the general merge (same arithmetic; the stage ring is its scratch)
        const bool ok_m = p.nchunks <= kTcMergeSegments
                              ? tc_merge<D>(p, sm, reinterpret_cast<float*>(base + Tg::kOffQ), base,
                                            &bar.mrows, hq0, G, u * p.nchunks, p.nchunks, gphase)
                              : merge_unit<D, 64, true>(p, sm, U, u * p.nchunks, p.nchunks, gphase);
        if (!ok_m) return;
        if (threadIdx.x == 0) p.counters[u] = 0u;
    }
    group_sync(sm, gphase, p.err);
}

}  // namespace

int sparse_tc_threads() { return kTcThreads; }

cudaError_t launch_sparse_tc(int D, const Launch& L) {
    if (D == 128)
        return launch_kernel(reinterpret_cast<const void*>(&sparse_tc_kernel<128>),
                             TcGeom<128>::kSmemBytes, L);
    if (D == 64)
        return launch_kernel(reinterpret_cast<const void*>(&sparse_tc_kernel<64>),
                             TcGeom<64>::kSmemBytes, L);
    return cudaErrorInvalidValue;
}

}  // namespace da
