// Single-query decode attention on sm_103a: one kernel per call.
//
// Work decomposition.  A "unit" is one (sequence b, KV head g); its G = Hq/Hkv query heads (times
// the query tokens, for several tokens per sequence) are processed together so every K/V row is
// read from HBM exactly once.  Paged units may take kh adjacent KV heads (kh * G query columns):
// a page of kh adjacent heads is kh * page_size contiguous rows, so with kh * page_size = 64 a
// paged tile is one 64-row TMA box per half, the same transfer as a dense tile; each query
// column then only sees its own KV head's rows.  A unit's live rows are cut into 64-row tiles.
// Dense and paged calls run a persistent grid (one CTA per SM): the tiles of all units are laid
// end to end and CTA c takes the contiguous range [c*N/C, (c+1)*N/C), so the load is balanced to
// one tile whatever the lengths.  Sparse calls (up to 32 query heads per KV head; larger groups
// run on the tensor-core kernel) cut each unit's selection into chunks of 512 entries — fixed, so
// trailing -1 pads cannot move a chunk boundary — and also run a persistent grid: the (unit,
// chunk) items are numbered end to end and CTA c takes a contiguous range of whole items, each
// finished as its own segment while the producers already gather the next item's rows.  Each
// CTA's piece of a unit is a "segment".
//
// Inside a CTA.  The producer warps (one for dense, two taking alternate tiles for paged, four
// sharing every tile for sparse) stream K and V tiles into a ring of shared-memory stages (TMA
// tile loads with 128-byte swizzle for dense and paged; cp.async 16-byte gathers with the same
// swizzle for sparse) and post a per-stage validity mask.  Warps 0-3 consume: the GQA group
// sits on the N side of mma.m16n8k16 (S^T = K * Q^T, then O^T += V^T * P^T), so each K/V
// element read from shared memory feeds all G heads; the online softmax (running max, sum and
// accumulator) stays in fp32 registers.  For units of one KV head every column mask is a
// compile-time constant, so a stage's MMAs are straight-line code.
//
// Merge.  A segment covering a whole unit writes the bf16 output directly.  Otherwise it writes
// its normalised partial row and log2-sum-exp to the workspace and bumps the unit's counter
// (acquire-release); the CTA that completes the unit merges all its partials by log-sum-exp in
// segment order (so the result does not depend on which CTA finishes last) and resets the
// counter to zero.
//
// Launch.  Kernels are launched with programmatic stream serialization: a CTA sets up its shared
// memory while the previous kernel in the stream drains, then waits for that kernel's completion
// (griddepcontrol.wait) before its first global-memory access.
//
// Safety.  Every wait is bounded (about one second); on timeout the CTA records an error code in
// the device error word, waits for its own copies in flight and returns.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math_constants.h>
#include <stdint.h>

#include "ptx.cuh"

namespace da {

constexpr int kTileKeys = 64;                 // K/V rows per pipeline stage
constexpr int kConsumerWarps = 4;
constexpr int kConsumerThreads = kConsumerWarps * 32;
// Producer warps per CTA: one TMA-issuing warp for dense; two for paged, which take alternate
// tiles (the block-table lookup makes a paged tile's issue path longer than a dense one); the
// sparse gather issues 16-byte cp.async copies, and one warp cannot keep enough of them in
// flight, so it gets four that share every tile.
template <int VAR>
struct Roles {
    static constexpr int kProducerWarps = VAR == 2 ? 4 : VAR == 1 ? 2 : 1;
    static constexpr int kThreads = kConsumerThreads + 32 * kProducerWarps;
};
constexpr uint64_t kWaitLimitNs = 1000000000ull;

// A bounded wait executed by every lane of a warp whose outcome is the same on every lane: each
// lane's limit runs on its own clock, and what follows a wait (a ballot, a shuffle, a warp-wide
// MMA or load) needs all 32 lanes, so on a timeout the whole warp gives up together.
__device__ __forceinline__ bool mbar_wait_warp(uint64_t* bar, uint32_t parity, volatile int* abort) {
    return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort, kWaitLimitNs));
}
constexpr int kSparseMaxHeads = 32;          // query heads per KV head of this kernel's sparse units
constexpr int kSparseChunkUnit = 512;         // sparse chunk: selection entries per CTA
constexpr int kMaxPagedBatch = 1024;
constexpr int kSmemBudget = 232448;           // opt-in dynamic shared memory per block

enum : int { kDense = 0, kPaged = 1, kSparse = 2 };
enum : uint32_t { kErrWaitFull = 1, kErrWaitEmpty = 2, kErrWaitGroup = 3, kErrDrain = 4,
                  kErrWaitCheck = 5 };

template <int D, int GP>
struct Geometry {
    static_assert(D == 64 || D == 128, "head dim");
    static_assert(GP == 8 || GP == 16 || GP == 32 || GP == 64, "padded group");
    static constexpr int kHalves = D / 64;                      // 128-byte swizzle spans
    static constexpr int kTileBytes = kHalves * kTileKeys * 128;  // one K (or V) tile
    static constexpr int kStageBytes = 2 * kTileBytes;
    static constexpr int HS = GP <= 16 ? 1 : GP / 16;           // warps splitting the heads
    static constexpr int NT = GP / 8 / HS;                      // 8-head n-tiles per warp
    static constexpr int KS = kConsumerWarps / HS;              // warps splitting a tile's rows
    static constexpr int MT = kTileKeys / 16 / KS;              // 16-row m-tiles per warp
    static constexpr int KSTEPS = D / 16;                       // k-steps of S^T = K Q^T
    static constexpr int DT = D / 16;                           // 16-row d tiles of O^T
    // merge slot rows are D + 4 floats apart, so the stash's stores (lanes 2 heads apart) fall
    // in distinct banks
    static constexpr int kMergeStride = D + 4;
    static constexpr int kMergeFloats = KS * GP * kMergeStride + 2 * KS * GP + 4 * GP;   // + per-head stats
    static constexpr int kMiscBytes = 1024;                     // barriers, masks, flags
    static constexpr int kSchedBytes = (2 * kMaxPagedBatch + 2) * 4;
    static constexpr int kFixedBytes = kMergeFloats * 4 + kMiscBytes + kSchedBytes;
    static constexpr int kStagesFit = (kSmemBudget - 1024 - kFixedBytes) / kStageBytes;
    static constexpr int kStages = kStagesFit > 8 ? 8 : kStagesFit;
    static constexpr int kSmemBytes = 1024 + kStages * kStageBytes + kFixedBytes;
    static_assert(kStages >= 2, "pipeline depth");
    static_assert(kSmemBytes <= kSmemBudget, "shared memory");
};

struct Params {
    const __nv_bfloat16* q;   // [B, Hq, D]
    __nv_bfloat16* out;       // [B, Hq, D]
    int B, Hq, Hkv, G;
    float scale_log2;         // softmax_scale * log2(e)
    unsigned* counters;       // one per merge unit, zero between calls
    float* part_o;            // [segments, seg_heads, D]
    float* part_lse;          // [segments, seg_heads] (log2 domain)
    int seg_heads;            // partial rows per segment: the unit's query columns (kh * G * sq)
    unsigned* err;            // device error word
    // dense
    int k_len;
    int dense_tiles;          // ceil(k_len / 64)
    const unsigned* k_len_dev;  // if set, k_len is read here on the device (clamped to capacity)
    int capacity;
    // paged
    const int* block_table;
    int max_pages, page_size, num_pages;
    int kh;                   // KV heads per unit (paged; 1 otherwise), a power of two
    int tile_keys;            // keys per stage and KV head: 64 / kh
    int sq;                   // query tokens per sequence (q, out [B, Hq, sq, D]); 1 = decode
    int causal;               // sq > 1: token i attends rows [0, len - sq + i]
    const unsigned* kv_lens;
    int kv_stride;
    // sparse
    const int* sel;
    int width, pool_rows, nchunks;
    const __nv_bfloat16* k_pool;
    const __nv_bfloat16* v_pool;
};

struct Unit {
    int b, g, u;
    int len;    // live rows
    int nt;     // tiles
    int base;   // global index of the unit's first tile
    int hq0;    // q / out row of the first query head this CTA handles
    int nh;     // query heads this CTA handles
    int cu;     // merge counter of this unit
};

struct SmemPtrs {
    unsigned char* stages;
    float* merge_o;
    float* merge_m;
    float* merge_l;
    float* head_inv;   // [GP] 1 / (sum of weights), 0 for an empty head
    float* head_lse;   // [GP] log2-domain log-sum-exp of the head's slots
    int* head_live;    // [GP] bit k: merge slot k holds a live piece
    uint64_t* full;
    uint64_t* empty;
    uint64_t* group;
    uint64_t* stage_mask;
    volatile int* abort;
    int* last_flag;
    int* seq_prefix;   // [B + 1] exclusive prefix of per-sequence tiles (paged)
    int* seq_len;      // [B] live rows per sequence (paged)
};

template <int D, int GP>
__device__ __forceinline__ SmemPtrs carve_smem(unsigned char* raw) {
    using Gm = Geometry<D, GP>;
    SmemPtrs s;
    // 1024-byte aligned by an offset into the shared array, so accesses through these pointers
    // stay shared-memory accesses for the compiler
    unsigned char* base = raw + ((1024u - (smem_u32(raw) & 1023u)) & 1023u);
    s.stages = base;
    unsigned char* p = base + Gm::kStages * Gm::kStageBytes;
    s.merge_o = reinterpret_cast<float*>(p);
    s.merge_m = s.merge_o + Gm::KS * GP * Gm::kMergeStride;
    s.merge_l = s.merge_m + Gm::KS * GP;
    s.head_inv = s.merge_l + Gm::KS * GP;
    s.head_lse = s.head_inv + GP;
    s.head_live = reinterpret_cast<int*>(s.head_lse + GP);
    p += Gm::kMergeFloats * 4;
    p += (16u - (smem_u32(p) & 15u)) & 15u;
    s.full = reinterpret_cast<uint64_t*>(p);
    s.empty = s.full + 8;
    s.group = s.empty + 8;
    s.stage_mask = s.group + 1;
    s.abort = reinterpret_cast<volatile int*>(s.stage_mask + 8);
    s.last_flag = const_cast<int*>(reinterpret_cast<volatile int*>(s.abort)) + 1;
    s.seq_prefix = reinterpret_cast<int*>(base + Gm::kStages * Gm::kStageBytes +
                                          Gm::kMergeFloats * 4 + Gm::kMiscBytes);
    s.seq_len = s.seq_prefix + kMaxPagedBatch + 2;
    return s;
}

__device__ __forceinline__ void record_error(unsigned* err, unsigned code) {
    if (err) atomicCAS(err, 0u, code);
}

// Byte offset, inside one K or V tile, of 16-byte chunk c (of D/8) of row r.  The tile is cut
// into blocks of 2^rb_shift rows (64 for dense and sparse, one page for paged); a block holds its
// 64-column halves one after the other, each [rows][128 B] with the 16-byte chunk index XOR
// (row & 7).  That is the layout a TMA tile load with 128-byte swizzle writes for one block, and
// the one the sparse gather writes by hand.
template <int HALVES>
__device__ __forceinline__ uint32_t tile_offset(int r, int c, int rb_shift) {
    const int blk = r >> rb_shift;
    const int rr = r & ((1 << rb_shift) - 1);
    return static_cast<uint32_t>(((blk * HALVES + (c >> 3)) << (rb_shift + 7)) + rr * 128 +
                                 (((c & 7) ^ (r & 7)) << 4));
}

// ------------------------------------------------------------------ schedule
__device__ __forceinline__ int tile_owner(int t, int N, int C) {
    // the CTA whose range [c*N/C, (c+1)*N/C) holds tile t
    return static_cast<int>((static_cast<long long>(t + 1) * C + N - 1) / N) - 1;
}

__device__ __forceinline__ Unit locate_dense(const Params& p, int t, int k_len, int tiles) {
    Unit U;
    U.nt = tiles;
    U.u = t / U.nt;
    U.b = U.u / p.Hkv;
    U.g = U.u - U.b * p.Hkv;
    U.len = k_len;
    U.base = U.u * U.nt;
    U.hq0 = (U.b * p.Hq + U.g * p.G) * p.sq;
    U.nh = p.G * p.sq;
    U.cu = U.u;
    return U;
}

// Paged units: (b, KV-head group gk of kh heads), gk fastest; U.g is gk.
__device__ __forceinline__ Unit locate_paged(const Params& p, const SmemPtrs& sm, int t) {
    const int upb = p.Hkv / p.kh;   // units per sequence
    // largest b with seq_prefix[b] * upb <= t
    int lo = 0, hi = p.B - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (sm.seq_prefix[mid] * upb <= t) lo = mid; else hi = mid - 1;
    }
    Unit U;
    U.b = lo;
    U.nt = sm.seq_prefix[lo + 1] - sm.seq_prefix[lo];
    const int r = t - sm.seq_prefix[lo] * upb;
    U.g = r / U.nt;
    U.u = U.b * upb + U.g;
    U.len = sm.seq_len[lo];
    U.base = sm.seq_prefix[lo] * upb + U.g * U.nt;
    U.hq0 = (U.b * p.Hq + U.g * p.kh * p.G) * p.sq;
    U.nh = p.kh * p.G * p.sq;
    U.cu = U.u;
    return U;
}

// ------------------------------------------------------------------ consumer warp state
// GW: query columns a warp holds in registers.  GW == GP: every warp holds all of the unit's
// columns.  GW == 8 < GP (paged units of kh > 1 KV heads with pages of >= 16 rows): the 16 rows
// of each warp belong to one KV head, so the warp holds only that head's <= 8 columns, starting
// at unit column col0; the merge slots stay GP columns wide and the warp marks the others empty.
// MULTI: a unit spans several KV heads (paged, kh > 1), so the column and n-tile masks depend on
// the lane and are computed at run time; otherwise every mask is a compile-time constant, which
// leaves the MMAs of consume() unguarded straight-line code.
template <int D, int GP, int GW = GP, bool MULTI = false>
struct ConsumerState {
    using Gm = Geometry<D, GW>;
    static_assert(GW == GP || (GW == 8 && MULTI && Gm::KS == kConsumerWarps &&
                               Geometry<D, GP>::KS == kConsumerWarps),
                  "warp-per-head columns need one 16-row m-tile per warp");
    static constexpr uint32_t kAllNeed = (Gm::MT * Gm::NT >= 32) ? 0xffffffffu
                                                                 : ((1u << (Gm::MT * Gm::NT)) - 1u);
    static constexpr uint32_t kAllNt = (1u << Gm::NT) - 1u;
    static constexpr uint32_t kAllCols = (Gm::MT * Gm::NT * 4 >= 32)
                                             ? 0xffffffffu
                                             : ((1u << (Gm::MT * Gm::NT * 4)) - 1u);
    int lane, hg, kg, gq, qd;
    int col0;                             // first unit column held by this warp
    uint32_t qf[Gm::KSTEPS][Gm::NT][2];   // Q^T as mma B fragments
    float o[Gm::DT][Gm::NT][4];           // O^T accumulator fragments
    float m_run[Gm::NT][2];               // running max (log2 domain) of heads 2qd, 2qd+1
    float l_run[Gm::NT][2];               // this thread's share of the running sum
    // Per-kernel constants of this lane, set once by init():
    uint32_t k_row_off[Gm::MT];           // byte offset of this lane's K ldmatrix row, chunk 0
    uint32_t v_row_off[Gm::MT];           // same for the transposed V ldmatrix
    uint32_t half_stride;                 // bytes between the two 64-column halves of a block
    uint32_t col_ok;                      // bit (mt*NT + nt)*4 + e: score element may be kept
    uint32_t need;                        // bit mt*NT + nt: the n-tile can see the m-tile's rows
    uint32_t nt_any;                      // bit nt: some m-tile of this warp needs n-tile nt
    int col_tok[Gm::NT][2];               // query token (0..sq-1) of each of this thread's columns
    int rbs, hsh;                         // rb_shift and head_shift (row -> key offset)

    // rb_shift: log2 of the rows per block of the tile layout; kh > 1 (paged units of kh KV
    // heads): row r of the tile belongs to the unit's KV head (r >> head_shift) & (kh - 1), and a
    // query column c to KV head c / G (G: query columns per KV head, heads * tokens) and to
    // token c % sq.
    __device__ __forceinline__ void init(int warp, int lane_, int G, int kh, int rb_shift,
                                         int head_shift, int sq) {
        lane = lane_;
        rbs = rb_shift;
        hsh = head_shift;
        hg = warp % Gm::HS;
        kg = warp / Gm::HS;
        gq = lane >> 2;
        qd = lane & 3;
        col0 = GW == GP ? 0 : (((kg * 16) >> head_shift) & (kh - 1)) * G;
#pragma unroll
        for (int nt = 0; nt < Gm::NT; ++nt)
#pragma unroll
            for (int hc = 0; hc < 2; ++hc) col_tok[nt][hc] = head_of(nt, hc) % sq;
        const int row0 = kg * Gm::MT * 16;
        half_stride = 1u << (rb_shift + 7);
        auto block_row = [&](int r) -> uint32_t {
            return static_cast<uint32_t>((((r >> rb_shift) * Gm::kHalves) << (rb_shift + 7)) +
                                         (r & ((1 << rb_shift) - 1)) * 128);
        };
        col_ok = 0;
        need = 0;
        nt_any = 0;
#pragma unroll
        for (int mt = 0; mt < Gm::MT; ++mt) {
            k_row_off[mt] = block_row(row0 + mt * 16 + (lane & 7) + ((lane >> 3) & 1) * 8);
            v_row_off[mt] = block_row(row0 + mt * 16 + (lane & 7) + ((lane >> 4) << 3));
#pragma unroll
            for (int nt = 0; nt < Gm::NT; ++nt) {
                const int first = row0 + mt * 16;
                const int ha = (first >> head_shift) & (kh - 1);
                const int hb = ((first + 15) >> head_shift) & (kh - 1);
                const int c0 = col0 + hg * Gm::NT * 8 + nt * 8;
                const bool nd = kh == 1 || (c0 / G <= max(ha, hb) && (c0 + 7) / G >= min(ha, hb));
                if (nd) {
                    need |= 1u << (mt * Gm::NT + nt);
                    nt_any |= 1u << nt;
                }
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int row = first + gq + (e >= 2 ? 8 : 0);
                    const int col = head_of(nt, e & 1);
                    if (kh == 1 || ((row >> head_shift) & (kh - 1)) == col / G)
                        col_ok |= 1u << ((mt * Gm::NT + nt) * 4 + e);
                }
            }
        }
        if (!MULTI || GW != GP) {   // every n-tile of the warp sees its rows
            need = kAllNeed;
            nt_any = kAllNt;
        }
        if (!MULTI) col_ok = kAllCols;
    }

    __device__ __forceinline__ int head_of(int nt, int hc) const {
        return col0 + hg * Gm::NT * 8 + nt * 8 + 2 * qd + hc;
    }

    // Q rows hq0 .. hq0 + nh - 1 as B fragments (heads past nh are zero)
    __device__ __forceinline__ void load_q(const Params& p, int hq0, int nh) {
#pragma unroll
        for (int nt = 0; nt < Gm::NT; ++nt) {
            const int head = col0 + hg * Gm::NT * 8 + nt * 8 + gq;
            const bool ok = head < nh;
            const __nv_bfloat16* row = p.q + (static_cast<size_t>(hq0) + (ok ? head : 0)) * D;
            const uint32_t* row32 = reinterpret_cast<const uint32_t*>(row);
#pragma unroll
            for (int ks = 0; ks < Gm::KSTEPS; ++ks) {
                qf[ks][nt][0] = ok ? __ldg(row32 + (16 * ks + 2 * qd) / 2) : 0u;
                qf[ks][nt][1] = ok ? __ldg(row32 + (16 * ks + 8 + 2 * qd) / 2) : 0u;
            }
        }
    }

    __device__ __forceinline__ void reset() {
#pragma unroll
        for (int dt = 0; dt < Gm::DT; ++dt)
#pragma unroll
            for (int nt = 0; nt < Gm::NT; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) o[dt][nt][e] = 0.f;
#pragma unroll
        for (int nt = 0; nt < Gm::NT; ++nt) {
            m_run[nt][0] = m_run[nt][1] = -CUDART_INF_F;
            l_run[nt][0] = l_run[nt][1] = 0.f;
        }
    }

    // ldmatrix address of 16-byte chunk c (of D/8) in the row whose block offset is `row_off`
    __device__ __forceinline__ uint32_t chunk_addr(uint32_t tile, uint32_t row_off, int c) const {
        return tile + row_off + static_cast<uint32_t>(c >> 3) * half_stride +
               ((static_cast<uint32_t>(c & 7) ^ static_cast<uint32_t>(lane & 7)) << 4);
    }

    // One stage: this warp's MT*16 rows of the tile.  `mask` bit r = row r of the tile is valid.
    // Scores outside col_ok (another KV head's rows) are dropped; n-tiles outside `need` skip
    // their MMAs and, when no m-tile of the stage needs them, their whole softmax update (their
    // state is unchanged, exactly as if every score were masked).
    // Causal (several query tokens): the tile's row r holds key key0 + off(r) of the unit; a
    // score is dropped where that key lies past causal_base + token.  Only tiles reaching a key
    // >= causal_from (the first key some token cannot see) pay for the test.
    __device__ __forceinline__ void consume(uint32_t k_tile, uint32_t v_tile, uint64_t mask,
                                            float scale_log2, int key0, int causal_base,
                                            int causal_from) {
        constexpr int kRows = Gm::MT * 16;
        const uint64_t rows_mask = kRows == 64 ? ~0ull : ((1ull << kRows) - 1ull);
        const uint64_t wmask = (mask >> (kg * kRows)) & rows_mask;
        if (wmask == 0) return;               // no valid row: the state is unchanged
        const bool all_valid = wmask == rows_mask;
        const bool all_cols = col_ok == kAllCols;

        // S^T[row, head] = sum_d K[row, d] * Q[head, d]
        float s[Gm::MT][Gm::NT][4];
#pragma unroll
        for (int mt = 0; mt < Gm::MT; ++mt)
#pragma unroll
            for (int nt = 0; nt < Gm::NT; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) s[mt][nt][e] = 0.f;
#pragma unroll
        for (int mt = 0; mt < Gm::MT; ++mt) {
#pragma unroll
            for (int ks = 0; ks < Gm::KSTEPS; ++ks) {
                uint32_t a[4];
                ldmatrix_x4(a, chunk_addr(k_tile, k_row_off[mt], 2 * ks + (lane >> 4)));
#pragma unroll
                for (int nt = 0; nt < Gm::NT; ++nt)
                    if (need & (1u << (mt * Gm::NT + nt)))
                        mma_bf16_16816(s[mt][nt], a, qf[ks][nt][0], qf[ks][nt][1]);
            }
        }

        // scale into the log2 domain; invalid rows and other KV heads' rows -> -inf
#pragma unroll
        for (int mt = 0; mt < Gm::MT; ++mt)
#pragma unroll
            for (int nt = 0; nt < Gm::NT; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    float x = s[mt][nt][e] * scale_log2;
                    const int rr = mt * 16 + gq + (e >= 2 ? 8 : 0);
                    if (!all_valid && !((wmask >> rr) & 1ull)) x = -CUDART_INF_F;
                    if (key0 + kTileKeys > causal_from) {
                        const int r = kg * kRows + rr;
                        const int key = key0 + ((r >> rbs) << hsh) + (r & ((1 << hsh) - 1));
                        if (key > causal_base + col_tok[nt][e & 1]) x = -CUDART_INF_F;
                    }
                    if (!all_cols && !((col_ok >> ((mt * Gm::NT + nt) * 4 + e)) & 1u)) x = -CUDART_INF_F;
                    s[mt][nt][e] = x;
                }

        // online softmax update per head column
#pragma unroll
        for (int nt = 0; nt < Gm::NT; ++nt) {
            if (!((nt_any >> nt) & 1u)) continue;   // no row of this warp reaches these heads
#pragma unroll
            for (int hc = 0; hc < 2; ++hc) {
                float mx = -CUDART_INF_F;
#pragma unroll
                for (int mt = 0; mt < Gm::MT; ++mt) mx = fmaxf(mx, fmaxf(s[mt][nt][hc], s[mt][nt][hc + 2]));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
                const float m_new = fmaxf(m_run[nt][hc], mx);
                const float m_use = m_new == -CUDART_INF_F ? 0.f : m_new;
                const float alpha = fast_exp2(m_run[nt][hc] - m_use);
                m_run[nt][hc] = m_new;
                l_run[nt][hc] *= alpha;
#pragma unroll
                for (int dt = 0; dt < Gm::DT; ++dt) {
                    o[dt][nt][hc] *= alpha;
                    o[dt][nt][hc + 2] *= alpha;
                }
#pragma unroll
                for (int mt = 0; mt < Gm::MT; ++mt) {
                    s[mt][nt][hc] = fast_exp2(s[mt][nt][hc] - m_use);
                    s[mt][nt][hc + 2] = fast_exp2(s[mt][nt][hc + 2] - m_use);
                }
            }
        }

        // P (rounded to bf16; the sum uses the rounded weights) -> P^T B fragments
        uint32_t pb[Gm::MT][Gm::NT][2];
#pragma unroll
        for (int mt = 0; mt < Gm::MT; ++mt)
#pragma unroll
            for (int nt = 0; nt < Gm::NT; ++nt) {
                if (!(need & (1u << (mt * Gm::NT + nt)))) {
                    pb[mt][nt][0] = pb[mt][nt][1] = 0u;
                    continue;
                }
                const uint32_t r0 = pack_bf16x2(s[mt][nt][0], s[mt][nt][1]);  // row gq
                const uint32_t r1 = pack_bf16x2(s[mt][nt][2], s[mt][nt][3]);  // row gq + 8
                l_run[nt][0] += bf16_lo_to_f32(r0) + bf16_lo_to_f32(r1);
                l_run[nt][1] += bf16_hi_to_f32(r0) + bf16_hi_to_f32(r1);
                pb[mt][nt][0] = movmatrix_trans(r0);
                pb[mt][nt][1] = movmatrix_trans(r1);
            }

        // O^T[d, head] += sum_row V[row, d] * P[row, head]
#pragma unroll
        for (int mt = 0; mt < Gm::MT; ++mt) {
            uint32_t keep_lo = 0xffffffffu, keep_hi = 0xffffffffu;
            if (!all_valid) {
                const int k0 = mt * 16 + 2 * qd;
                keep_lo = (((wmask >> k0) & 1ull) ? 0x0000ffffu : 0u) |
                          (((wmask >> (k0 + 1)) & 1ull) ? 0xffff0000u : 0u);
                keep_hi = (((wmask >> (k0 + 8)) & 1ull) ? 0x0000ffffu : 0u) |
                          (((wmask >> (k0 + 9)) & 1ull) ? 0xffff0000u : 0u);
            }
#pragma unroll
            for (int dt = 0; dt < Gm::DT; ++dt) {
                uint32_t a[4];
                ldmatrix_x4_trans(a, chunk_addr(v_tile, v_row_off[mt], 2 * dt + ((lane >> 3) & 1)));
                if (!all_valid) {   // rows never loaded or past the length may hold NaN
                    a[0] &= keep_lo;
                    a[1] &= keep_lo;
                    a[2] &= keep_hi;
                    a[3] &= keep_hi;
                }
#pragma unroll
                for (int nt = 0; nt < Gm::NT; ++nt)
                    if (need & (1u << (mt * Gm::NT + nt)))
                        mma_bf16_16816(o[dt][nt], a, pb[mt][nt][0], pb[mt][nt][1]);
            }
        }
    }

    // Writes this warp's (m, l, O) for its heads into merge slot kg (with GW < GP the slot's
    // other columns are marked empty first).
    __device__ __forceinline__ void stash(const SmemPtrs& sm) {
        if (GW != GP) {
            for (int c = lane; c < GP; c += 32) sm.merge_m[kg * GP + c] = -CUDART_INF_F;
            __syncwarp();
        }
#pragma unroll
        for (int nt = 0; nt < Gm::NT; ++nt)
#pragma unroll
            for (int hc = 0; hc < 2; ++hc) {
                float l = l_run[nt][hc];
                l += __shfl_xor_sync(0xffffffffu, l, 4);
                l += __shfl_xor_sync(0xffffffffu, l, 8);
                l += __shfl_xor_sync(0xffffffffu, l, 16);
                const int head = head_of(nt, hc);
                if (GW != GP && head >= GP) continue;   // past the unit's last column
                const int slot = kg * GP + head;
                if (gq == 0) {
                    sm.merge_m[slot] = m_run[nt][hc];
                    sm.merge_l[slot] = l;
                }
#pragma unroll
                for (int dt = 0; dt < Gm::DT; ++dt) {
                    sm.merge_o[slot * Gm::kMergeStride + dt * 16 + gq] = o[dt][nt][hc];
                    sm.merge_o[slot * Gm::kMergeStride + dt * 16 + gq + 8] = o[dt][nt][hc + 2];
                }
            }
    }
};

// Consumer-group barrier (128 threads) on an mbarrier, bounded; every lane of a warp returns the
// same outcome.
__device__ __forceinline__ bool group_sync(const SmemPtrs& sm, uint32_t& phase, unsigned* err) {
    mbar_arrive(sm.group);
    const bool ok = mbar_wait_warp(sm.group, phase, sm.abort);
    phase ^= 1u;
    if (!ok) {
        *sm.abort = 1;
        record_error(err, kErrWaitGroup);
    }
    return ok;
}

// acc + w * o, one rounding per component (the merges' accumulation step)
__device__ __forceinline__ float4 fma4(float w, const float4& o, const float4& acc) {
    return make_float4(__fmaf_rn(w, o.x, acc.x), __fmaf_rn(w, o.y, acc.y), __fmaf_rn(w, o.z, acc.z),
                       __fmaf_rn(w, o.w, acc.w));
}

// Merges the nseg partial rows of unit U (workspace segments first_seg, first_seg + 1, ...) by
// log-sum-exp, in segment order, and stores the bf16 output row of each of the G heads.  Runs on
// the 128 consumer threads of the CTA that completed the unit and uses the merge area of shared
// memory as scratch: the partial LSEs are read once, coalesced, into shared memory; each thread
// then owns float4 slices of the output and keeps several partial rows in flight.
// kNoPrefetch: never issue the row loads ahead (fewer registers, for callers whose register
// budget is tight; same arithmetic).
template <int D, int GP, bool kNoPrefetch = false>
__device__ __forceinline__ bool merge_unit(const Params& p, const SmemPtrs& sm, const Unit& U,
                                           int first_seg, int nseg, uint32_t& gphase) {
    using Gm = Geometry<D, GP>;
    constexpr int D4 = D / 4;                        // float4 columns per row
    constexpr int HQ = kConsumerThreads / D4;        // heads covered per pass (4 or 8)
    constexpr int NH = (GP + HQ - 1) / HQ;           // heads per thread
    constexpr int SU = NH >= 16 ? 1 : 16 / NH;       // segments whose rows are loaded together
    constexpr int SB = Gm::KS * D - 4;               // segments per shared-memory batch
    const int tid = threadIdx.x;
    const int G = U.nh;                              // heads of this unit
    const int SH = p.seg_heads;                      // partial-row stride per segment
    float* h_max = sm.merge_o;                       // [GP]
    float* h_inv = h_max + GP;                       // [GP]
    int* h_live = reinterpret_cast<int*>(h_inv + GP);  // [GP]
    int* h_only = h_live + GP;                       // [GP]
    float* w_sm = reinterpret_cast<float*>(h_only + GP);  // [SB][GP]
    const float* lse = p.part_lse + static_cast<size_t>(first_seg) * SH;
    const float4* orow = reinterpret_cast<const float4*>(p.part_o + static_cast<size_t>(first_seg) * SH * D);
    const bool one_batch = nseg <= SB;

    if (!one_batch && tid < G) {
        // many segments: per-head statistics straight from global memory
        float M = -CUDART_INF_F;
#pragma unroll 8
        for (int k = 0; k < nseg; ++k) M = fmaxf(M, __ldcg(lse + static_cast<size_t>(k) * SH + tid));
        float L = 0.f;
        int live = 0, only = 0;
#pragma unroll 8
        for (int k = 0; k < nseg; ++k) {
            const float l = __ldcg(lse + static_cast<size_t>(k) * SH + tid);
            if (l != -CUDART_INF_F) {
                const float w = fast_exp2(l - M);
                L = live ? L + w : w;
                ++live;
                only = k;
            }
        }
        h_max[tid] = M;
        h_inv[tid] = live ? 1.0f / L : 0.f;
        h_live[tid] = live;
        h_only[tid] = only;
    }

    const int d4 = tid % D4, hq = tid / D4;
    float4 acc[NH];
#pragma unroll
    for (int j = 0; j < NH; ++j) acc[j] = make_float4(0.f, 0.f, 0.f, 0.f);

    // Few segments (the usual case): issue the partial-row loads now, together with the LSE
    // loads below, so the merge costs one L2 round trip instead of two.
    // (Not for 64-head groups, whose 16 rows per thread would not fit the register budget.)
    constexpr bool kPrefetch = NH <= 8 && !kNoPrefetch;
    constexpr int PU = kPrefetch ? SU : 1, PH = kPrefetch ? NH : 1;
    const bool prefetched = kPrefetch && one_batch && nseg <= SU;
    float4 pre[PU][PH];
#pragma unroll
    for (int u = 0; u < PU; ++u)
#pragma unroll
        for (int j = 0; j < PH; ++j) {
            const int h = hq + j * HQ;
            pre[u][j] = (prefetched && u < nseg && h < G)
                            ? __ldcg(orow + (static_cast<size_t>(u) * SH + h) * D4 + d4)
                            : make_float4(0.f, 0.f, 0.f, 0.f);
        }

    for (int s0 = 0; s0 < nseg; s0 += SB) {
        const int nb = min(SB, nseg - s0);
        for (int i = tid; i < nb * G; i += kConsumerThreads) {
            const int sgi = i / G, h = i - sgi * G;
            w_sm[sgi * GP + h] = __ldcg(lse + static_cast<size_t>(s0 + sgi) * SH + h);
        }
        if (!group_sync(sm, gphase, p.err)) return false;
        if (one_batch) {
            if (tid < G) {
                float M = -CUDART_INF_F;
                for (int k = 0; k < nb; ++k) M = fmaxf(M, w_sm[k * GP + tid]);
                float L = 0.f;
                int live = 0, only = 0;
                for (int k = 0; k < nb; ++k) {
                    const float l = w_sm[k * GP + tid];
                    float w = 0.f;
                    if (l != -CUDART_INF_F) {
                        w = fast_exp2(l - M);
                        L = live ? L + w : w;
                        ++live;
                        only = k;
                    }
                    w_sm[k * GP + tid] = w;
                }
                h_max[tid] = M;
                h_inv[tid] = live ? 1.0f / L : 0.f;
                h_live[tid] = live;
                h_only[tid] = only;
            }
        } else {
            for (int i = tid; i < nb * G; i += kConsumerThreads) {
                const int sgi = i / G, h = i - sgi * G;
                const float l = w_sm[sgi * GP + h];
                w_sm[sgi * GP + h] = l == -CUDART_INF_F ? 0.f : fast_exp2(l - h_max[h]);
            }
        }
        if (!group_sync(sm, gphase, p.err)) return false;
        for (int sgi = 0; sgi < nb; sgi += SU) {
            float w[SU][NH];
            float4 o4[SU][NH];
#pragma unroll
            for (int u = 0; u < SU; ++u)
#pragma unroll
                for (int j = 0; j < NH; ++j) {
                    const int h = hq + j * HQ;
                    w[u][j] = (sgi + u < nb && h < G) ? w_sm[(sgi + u) * GP + h] : 0.f;
                    if (prefetched)
                        o4[u][j] = pre[kPrefetch ? u : 0][kPrefetch ? j : 0];
                    else
                        o4[u][j] = w[u][j] != 0.f
                                       ? __ldcg(orow + (static_cast<size_t>(s0 + sgi + u) * SH + h) * D4 + d4)
                                       : make_float4(0.f, 0.f, 0.f, 0.f);
                }
#pragma unroll
            for (int u = 0; u < SU; ++u)
#pragma unroll
                for (int j = 0; j < NH; ++j)
                    if (w[u][j] != 0.f) acc[j] = fma4(w[u][j], o4[u][j], acc[j]);
        }
        if (!group_sync(sm, gphase, p.err)) return false;
    }

    const size_t out_row0 = static_cast<size_t>(U.hq0);
#pragma unroll
    for (int j = 0; j < NH; ++j) {
        const int h = hq + j * HQ;
        if (h >= G) continue;
        const int live = h_live[h];
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (live == 1) {
            v = __ldcg(orow + (static_cast<size_t>(h_only[h]) * SH + h) * D4 + d4);
        } else if (live > 1) {
            const float inv = h_inv[h];
            v = make_float4(acc[j].x * inv, acc[j].y * inv, acc[j].z * inv, acc[j].w * inv);
        }
        uint2 packed;
        packed.x = pack_bf16x2(v.x, v.y);
        packed.y = pack_bf16x2(v.z, v.w);
        *reinterpret_cast<uint2*>(p.out + (out_row0 + h) * D + 4 * d4) = packed;
    }
    return true;
}

// Finishes one segment of unit U: merges the key-split warps, then either stores the output or
// publishes a partial and, in the CTA that completes the unit, merges all partials.  With
// `defer`, a partial is only stored: the caller counts it on the unit's counter later
// (publish_and_merge).
template <int D, int GP, class CS>
__device__ __forceinline__ bool finish_segment(const Params& p, const SmemPtrs& sm,
                                               CS& cs, const Unit& U,
                                               bool whole, int seg, int first_seg, int nseg,
                                               uint32_t& gphase, bool defer = false) {
    using Gm = Geometry<D, GP>;
    const int tid = threadIdx.x;   // 0..127 (consumers)
    cs.stash(sm);
    if (!group_sync(sm, gphase, p.err)) return false;

    const size_t out_row0 = static_cast<size_t>(U.hq0);
    const size_t SH = static_cast<size_t>(p.seg_heads);
    // Per head, once: the slots' weights relative to the largest slot maximum (stored over the
    // maxima), which slots are live, 1 / (sum of weights) and the log-sum-exp.  A dead slot
    // (maximum -inf) is skipped, and sums start from the first live term.
    if (tid < U.nh) {
        const int h = tid;
        float M = -CUDART_INF_F;
#pragma unroll
        for (int k = 0; k < Gm::KS; ++k) M = fmaxf(M, sm.merge_m[k * GP + h]);
        float L = 0.f;
        int live = 0;
        if (M != -CUDART_INF_F) {
#pragma unroll
            for (int k = 0; k < Gm::KS; ++k) {
                const float mk = sm.merge_m[k * GP + h];
                if (mk == -CUDART_INF_F) continue;
                const float w = fast_exp2(mk - M);
                const float lk = w * sm.merge_l[k * GP + h];
                L = live ? L + lk : lk;
                live |= 1 << k;
                sm.merge_m[k * GP + h] = w;
            }
        }
        const bool empty = !(L > 0.f);
        sm.head_inv[h] = empty ? 0.f : 1.0f / L;
        sm.head_lse[h] = empty ? -CUDART_INF_F : M + fast_log2(L);
        sm.head_live[h] = empty ? 0 : live;
    }
    if (!group_sync(sm, gphase, p.err)) return false;
    constexpr int D4 = D / 4;
    for (int i = tid; i < U.nh * D4; i += kConsumerThreads) {
        const int h = i / D4, d = (i - h * D4) * 4;
        const int live = sm.head_live[h];
        float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
        bool first = true;
#pragma unroll
        for (int k = 0; k < Gm::KS; ++k) {
            if (!((live >> k) & 1)) continue;
            const float w = sm.merge_m[k * GP + h];
            const float4 o = *reinterpret_cast<const float4*>(sm.merge_o + (k * GP + h) * Gm::kMergeStride + d);
            if (first) {
                O = make_float4(w * o.x, w * o.y, w * o.z, w * o.w);
                first = false;
            } else {
                O.x += w * o.x; O.y += w * o.y; O.z += w * o.z; O.w += w * o.w;
            }
        }
        const float inv = sm.head_inv[h];
        const float4 v = make_float4(O.x * inv, O.y * inv, O.z * inv, O.w * inv);
        if (whole) {
            __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y), hi = __floats2bfloat162_rn(v.z, v.w);
            uint2 packed;
            packed.x = *reinterpret_cast<uint32_t*>(&lo);
            packed.y = *reinterpret_cast<uint32_t*>(&hi);
            *reinterpret_cast<uint2*>(p.out + (out_row0 + h) * D + d) = packed;
        } else {
            *reinterpret_cast<float4*>(p.part_o + (static_cast<size_t>(seg) * SH + h) * D + d) = v;
        }
    }
    if (!whole && tid < U.nh) p.part_lse[static_cast<size_t>(seg) * SH + tid] = sm.head_lse[tid];
    if (!whole && !defer) {
        // The group barrier orders every consumer's partial-row stores before thread 0's
        // release on the unit's counter; the CTA that takes the counter to nseg acquires all
        // segments' rows there, and the next group barrier hands that on to its other threads.
        if (!group_sync(sm, gphase, p.err)) return false;
        if (tid == 0) {
            const unsigned prev = atomic_add_acq_rel_gpu(p.counters + U.cu);
            *sm.last_flag = (prev == static_cast<unsigned>(nseg - 1)) ? 1 : 0;
        }
        if (!group_sync(sm, gphase, p.err)) return false;
        if (*sm.last_flag) {
            if (!merge_unit<D, GP>(p, sm, U, first_seg, nseg, gphase)) return false;
            if (tid == 0) p.counters[U.cu] = 0u;
        }
    }
    return group_sync(sm, gphase, p.err);
}

// Counts the segments a CTA stored with finish_segment(..., defer) on their units' counters --
// the items [it_begin, it_end) of nchunks segments per unit, all published by one acquire-release
// add per unit, the units taken by the CTA's threads side by side -- and merges every unit this
// CTA completes, in unit order, with merge_unit (segment order within a unit, so the result does
// not depend on which CTA completes it).  A unit whose every segment this CTA stored is merged
// without touching its counter; a GPU-scope fence then makes those partial rows visible to the
// merge's L2 loads.  The caller's last group barrier orders every partial store before these
// releases and fences.  `flags` is scratch for kConsumerThreads ints.
template <int D, int GP>
__device__ __forceinline__ bool publish_and_merge(const Params& p, const SmemPtrs& sm, int* flags,
                                                  int it_begin, int it_end, uint32_t& gphase) {
    const int tid = threadIdx.x;
    const int nck = p.nchunks;
    const int u_first = it_begin / nck, u_last = (it_end - 1) / nck;
    for (int u0 = u_first; u0 <= u_last; u0 += kConsumerThreads) {
        const int u = u0 + tid;
        int last = 0;
        if (u <= u_last) {
            const int lo = max(it_begin, u * nck), hi = min(it_end, (u + 1) * nck);
            const unsigned n = static_cast<unsigned>(hi - lo);
            if (n == static_cast<unsigned>(nck)) {
                asm volatile("fence.acq_rel.gpu;" ::: "memory");
                last = 1;
            } else {
                unsigned prev;
                asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;"
                             : "=r"(prev) : "l"(p.counters + u), "r"(n) : "memory");
                last = prev + n == static_cast<unsigned>(nck) ? 1 : 0;
            }
        }
        flags[tid] = last;
        if (!group_sync(sm, gphase, p.err)) return false;
        const int nu = min(kConsumerThreads, u_last - u0 + 1);
        for (int i = 0; i < nu; ++i) {
            if (!flags[i]) continue;
            Unit U;
            U.u = u0 + i;
            U.b = U.u / p.Hkv;
            U.g = U.u - U.b * p.Hkv;
            U.len = p.width;
            U.nt = 0;
            U.base = 0;
            U.hq0 = U.b * p.Hq + U.g * p.G;
            U.nh = p.G;
            U.cu = U.u;
            if (!merge_unit<D, GP>(p, sm, U, U.u * nck, nck, gphase)) return false;
            // (a unit merged without its counter left it at zero)
            if (tid == 0) p.counters[U.cu] = 0u;
        }
        if (!group_sync(sm, gphase, p.err)) return false;   // flags reused
    }
    return true;
}

// ------------------------------------------------------------------ the kernel
template <int VAR, int D, int GP, int GW = GP, bool MULTI = false>
__global__ void __launch_bounds__(Roles<VAR>::kThreads, 1)
decode_attn_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                   const Params p) {
    using Gm = Geometry<D, GP>;
    extern __shared__ unsigned char smem_raw[];
    const SmemPtrs sm = carve_smem<D, GP>(smem_raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // Stages of the ring in use: more rows in flight than a stream needs only lengthen the memory
    // queues.  Dense units of up to 8 query columns stream fastest with 128 KB in flight per SM
    // (four 32 KB stages at D = 128: dense_long 317.5 -> 296.1 us against the six that fit,
    // dense_batched 42.6 -> 41.3 us; three are slower again), the paged gather with 160 KB
    // (paged_ragged_p64 603.0 -> 588.6 us with five stages instead of six; four: 595.7);
    // heavier dense consumers (more columns) and the sparse gathers keep every stage that fits.
    constexpr int kRingCap = (VAR == kDense && GP <= 8) ? 128 * 1024 / Gm::kStageBytes
                             : VAR == kPaged            ? 160 * 1024 / Gm::kStageBytes
                                                        : Gm::kStages;
    constexpr int S = kRingCap < Gm::kStages ? kRingCap : Gm::kStages;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(sm.full + s, VAR == kSparse ? 32u * Roles<VAR>::kProducerWarps + 1u : 1u);
            mbar_init(sm.empty + s, kConsumerWarps);
        }
        mbar_init(sm.group, kConsumerThreads);
        *sm.abort = 0;
        *sm.last_flag = 0;
        fence_mbarrier_init();
    }
    if (VAR != kSparse && threadIdx.x == kConsumerThreads) {
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
    }
    // Everything above touches only shared memory and the kernel parameters, so it overlaps the
    // tail of the previous kernel in the stream; no global memory is read or written before the
    // previous kernels have completed.
    grid_dependency_wait();
    allow_dependent_launch();

    // ---- schedule
    int N = 0, C = 1, t0 = 0, t1 = 0;
    if (VAR == kPaged) {
        const int cap = p.max_pages * p.page_size;
        for (int b = threadIdx.x; b < p.B; b += Roles<VAR>::kThreads) {
            const unsigned raw = __ldg(p.kv_lens + static_cast<size_t>(b) * p.kv_stride);
            const int len = raw > static_cast<unsigned>(cap) ? cap : static_cast<int>(raw);
            sm.seq_len[b] = len;
            sm.seq_prefix[b + 1] = (len + p.tile_keys - 1) / p.tile_keys;
        }
        __syncthreads();
        if (warp == 0) {
            int carry = 0;
            for (int base = 0; base < p.B; base += 32) {
                const int b = base + lane;
                int v = b < p.B ? sm.seq_prefix[b + 1] : 0;
#pragma unroll
                for (int off = 1; off < 32; off <<= 1) {
                    const int y = __shfl_up_sync(0xffffffffu, v, off);
                    if (lane >= off) v += y;
                }
                if (b < p.B) sm.seq_prefix[b + 1] = v + carry;
                carry += __shfl_sync(0xffffffffu, v, 31);
            }
            if (lane == 0) sm.seq_prefix[0] = 0;
        }
    }
    __syncthreads();

    // dense: the live length, given on the host or read here from device memory
    int dlen = p.k_len, dtiles = p.dense_tiles;
    if (VAR == kDense && p.k_len_dev != nullptr) {
        const unsigned raw = *p.k_len_dev;
        dlen = raw > static_cast<unsigned>(p.capacity) ? p.capacity : static_cast<int>(raw);
        dtiles = (dlen + kTileKeys - 1) / kTileKeys;
    }
    if (VAR == kDense) {
        N = p.B * p.Hkv * dtiles;
        C = min(static_cast<int>(gridDim.x), N);
    } else if (VAR == kPaged) {
        N = sm.seq_prefix[p.B] * (p.Hkv / p.kh);
        C = min(static_cast<int>(gridDim.x), N);
    }
    if (VAR != kSparse && static_cast<int>(blockIdx.x) < C && N > 0) {
        t0 = static_cast<int>(static_cast<long long>(blockIdx.x) * N / C);
        t1 = static_cast<int>(static_cast<long long>(blockIdx.x + 1) * N / C);
    }
    // sparse: the items (unit u, chunk) are numbered u * nchunks + chunk; CTA c takes a
    // contiguous range of them, each a whole chunk (so a chunk boundary never moves) finished as
    // its own segment.  With I = q * C + r, the first r CTAs take q + 1 items and the rest q, the
    // longer ranges first: when q + 1 is the chunk count, each longer range is one whole unit,
    // which that CTA merges by itself, and the merges of units split across CTAs fall to the
    // CTAs that finish a whole item earlier.
    int it_begin = 0, it_end = 0;
    if (VAR == kSparse) {
        const int I = p.B * p.Hkv * p.nchunks;
        C = min(static_cast<int>(gridDim.x), I);
        const int c = static_cast<int>(blockIdx.x);
        if (c < C) {
            const int q = I / C, r = I - q * C;
            it_begin = c < r ? c * (q + 1) : r * (q + 1) + (c - r) * q;
            it_end = it_begin + (c < r ? q + 1 : q);
        }
    }
    // one item's unit, first key and key count, and its tiles [t0, t1) of 64 selection entries
    auto sparse_item = [&](int item, int& u, int& key0, int& nkeys, int& ta, int& tb) {
        u = item / p.nchunks;
        key0 = (item - u * p.nchunks) * kSparseChunkUnit;
        nkeys = min(kSparseChunkUnit, p.width - key0);
        ta = key0 / kTileKeys;
        tb = (key0 + nkeys + kTileKeys - 1) / kTileKeys;
    };

    if (warp >= kConsumerWarps) {
        // ================================================================ producer warps
        int it = 0;
        bool ok = true;
        if (VAR == kSparse) {
            constexpr int NPW = Roles<VAR>::kProducerWarps;
            constexpr int kRowsPerWarp = kTileKeys / NPW;  // rows of a tile each producer warp copies
            const int ptid = threadIdx.x - kConsumerThreads;
            const int pw = ptid >> 5;
            constexpr int CH = D / 8;                     // 16-byte chunks per row
            constexpr int kRowsPerInstr = 32 / (2 * CH);  // K and V of 1 (D=128) or 2 (D=64) rows
            const int sub = lane / (2 * CH);
            const int w = lane % (2 * CH);
            const bool isv = w >= CH;
            const int c = isv ? w - CH : w;
            const __nv_bfloat16* pool = isv ? p.v_pool : p.k_pool;
            // an item's entries, read once (coalesced, all in flight) with every entry outside
            // [0, pool_rows) folded to -1, go to one of two index buffers: the next item's are
            // fetched into registers while this item's copies are issued, so no item waits for
            // its indices
            constexpr int kIdxPer = kSparseChunkUnit / (32 * NPW);   // entries per producer thread
            static_assert(kIdxPer * 32 * NPW == kSparseChunkUnit, "chunk split over producers");
            static_assert(2 * kSparseChunkUnit <= kMaxPagedBatch + 2, "two index buffers fit");
            int nidx[kIdxPer];
            auto fetch_idx = [&](int item) {
                int u, key0, nkeys, ta, tb;
                sparse_item(item, u, key0, nkeys, ta, tb);
                const int* selrow = p.sel + static_cast<size_t>(u / p.Hkv) * p.width + key0;
#pragma unroll
                for (int k = 0; k < kIdxPer; ++k) {
                    const int i = ptid + k * 32 * NPW;
                    const int idx = i < nkeys ? __ldg(selrow + i) : -1;
                    nidx[k] = (idx >= 0 && idx < p.pool_rows) ? idx : -1;
                }
            };
            auto store_idx = [&](int* buf) {
#pragma unroll
                for (int k = 0; k < kIdxPer; ++k) buf[ptid + k * 32 * NPW] = nidx[k];
            };
            if (it_begin < it_end) {
                fetch_idx(it_begin);
                store_idx(sm.seq_prefix);
            }
            // every producer warp passes every item's barrier, also after one of its waits gave
            // up (it then issues nothing), so no warp is left waiting at a barrier
            for (int item = it_begin; item < it_end; ++item) {
                int sp_u, sp_key0, sp_nkeys, ta, tb;
                sparse_item(item, sp_u, sp_key0, sp_nkeys, ta, tb);
                int* sidx = sm.seq_prefix + ((item - it_begin) & 1) * kSparseChunkUnit;
                // this item's entries are stored, and every producer has issued the previous
                // item's copies (which read the other buffer)
                asm volatile("bar.sync 1, %0;" ::"r"(32 * NPW) : "memory");   // producer warps only
                if (!ok) continue;
                if (item + 1 < it_end) fetch_idx(item + 1);
                const __nv_bfloat16* base =
                    pool + static_cast<size_t>(sp_u) * p.pool_rows * D + c * 8;
                for (int t = ta; t < tb; ++t, ++it) {
                    const int s = it % S;
                    const uint32_t ph = (it / S) & 1;
                    if (!mbar_wait_warp(sm.empty + s, ph ^ 1u, sm.abort)) { ok = false; break; }
                    const int l0 = t * kTileKeys - sp_key0;
                    const int i0 = l0 + lane, i1 = l0 + 32 + lane;
                    const int idx0 = i0 < sp_nkeys ? sidx[i0] : -1;
                    const int idx1 = i1 < sp_nkeys ? sidx[i1] : -1;
                    const bool v0 = idx0 >= 0;
                    const bool v1 = idx1 >= 0;
                    const uint64_t mask =
                        static_cast<uint64_t>(__ballot_sync(0xffffffffu, v0)) |
                        (static_cast<uint64_t>(__ballot_sync(0xffffffffu, v1)) << 32);
                    unsigned char* tile =
                        sm.stages + s * Gm::kStageBytes + (isv ? Gm::kTileBytes : 0);
                    const int row_begin = pw * kRowsPerWarp;
                    // independent iterations: each lane reads its row's entry from shared memory,
                    // so the unrolled loop keeps several index reads and copies in flight
#pragma unroll 8
                    for (int rb = row_begin; rb < row_begin + kRowsPerWarp; rb += kRowsPerInstr) {
                        const int r = rb + sub;
                        const int li = l0 + r;
                        const int idx = li < sp_nkeys ? sidx[li] : -1;
                        const bool valid = idx >= 0;
                        const __nv_bfloat16* src = base + static_cast<size_t>(valid ? idx : 0) * D;
                        cp_async_16(tile + tile_offset<Gm::kHalves>(r, c, 6), src,
                                    valid ? 16u : 0u);
                    }
                    if (ptid == 0) sm.stage_mask[s] = mask;
                    cp_async_arrive_noinc(sm.full + s);
                    if (ptid == 0) mbar_arrive(sm.full + s);
                }
                if (item + 1 < it_end)
                    store_idx(sm.seq_prefix + ((item + 1 - it_begin) & 1) * kSparseChunkUnit);
            }
            if (!ok) {
                cp_async_wait_all();
                *sm.abort = 1;
                record_error(p.err, kErrWaitEmpty);
            }
        } else {
            // dense / paged: lane 0 issues TMA; paged uses all lanes to fetch block-table entries
            const int P = p.page_size;
            // paged: a page group is the kh adjacent heads of one page, kh * P contiguous rows;
            // box_rows = min(kh * P, 64) rows of it per box and half
            const int TK = VAR == kPaged ? p.tile_keys : kTileKeys;   // keys per stage and KV head
            const int page_shift = VAR == kPaged ? 31 - __clz(P) : 0;
            const int box_rows = VAR == kPaged ? min(P * p.kh, kTileKeys) : kTileKeys;
            const int head_rows = VAR == kPaged ? min(P, TK) : kTileKeys;   // rows per head and page
            const int pages_per_tile = VAR == kPaged ? (P >= TK ? 1 : TK / P) : 1;
            const uint32_t box_bytes = static_cast<uint32_t>(box_rows) * 128u;
            int bt_b = -1, bt_base = -1;   // current batch: slots [bt_base, bt_base + 32) of sequence bt_b
            int bt_cur = -1, bt_nxt = -1;
            // producer warp pw takes the tiles t0 + pw, t0 + pw + NPW, ...; `it` stays the tile's
            // index in this CTA's range, which fixes its stage and phase
            constexpr int NPW = Roles<VAR>::kProducerWarps;
            const int pw = warp - kConsumerWarps;
            it = pw;
            for (int t = t0 + pw; t < t1 && ok;) {
                const Unit U = VAR == kDense ? locate_dense(p, t, dlen, dtiles) : locate_paged(p, sm, t);
                const int tend = min(t1, U.base + U.nt);
                const int npages_seq = VAR == kPaged ? (U.len + P - 1) / P : 0;
                for (; t < tend; t += NPW, it += NPW) {
                    const int s = it % S;
                    const uint32_t ph = (it / S) & 1;
                    if (!mbar_wait_warp(sm.empty + s, ph ^ 1u, sm.abort)) { ok = false; break; }
                    const int j = t - U.base;
                    const int key0 = j * TK;
                    const int nvalid = min(TK, U.len - key0);
                    uint64_t mask = nvalid >= 64 ? ~0ull : ((1ull << nvalid) - 1ull);
                    unsigned char* ktile = sm.stages + s * Gm::kStageBytes;
                    unsigned char* vtile = ktile + Gm::kTileBytes;
                    if (VAR == kDense) {
                        if (lane == 0) {
                            sm.stage_mask[s] = mask;
                            mbar_arrive_expect_tx(sm.full + s, 2u * Gm::kTileBytes);
#pragma unroll
                            for (int h = 0; h < Gm::kHalves; ++h) {
                                tma_load_3d(ktile + h * kTileKeys * 128, &tm_k, 64 * h, key0, U.u, sm.full + s);
                                tma_load_3d(vtile + h * kTileKeys * 128, &tm_v, 64 * h, key0, U.u, sm.full + s);
                            }
                        }
                    } else {
                        const int slot0 = key0 >> page_shift;   // page size: a power of two
                        const int want = slot0 & ~31;
                        if (U.b != bt_b || want != bt_base) {
                            const int* row = p.block_table + static_cast<size_t>(U.b) * p.max_pages;
                            if (U.b == bt_b && want == bt_base + 32) {
                                bt_cur = bt_nxt;
                            } else {
                                const int sl = want + lane;
                                bt_cur = sl < npages_seq ? __ldg(row + sl) : -1;
                            }
                            bt_b = U.b;
                            bt_base = want;
                            const int sn = want + 32 + lane;
                            bt_nxt = sn < npages_seq ? __ldg(row + sn) : -1;
                        }
                        const int row_in_page = P > TK ? (key0 & (P - 1)) : 0;
                        uint32_t page_ok = 0;
                        int pages[8];
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            if (i < pages_per_tile) {   // warp-uniform
                                pages[i] = __shfl_sync(0xffffffffu, bt_cur, (slot0 - bt_base + i) & 31);
                                if (slot0 + i < npages_seq && pages[i] >= 0 && pages[i] < p.num_pages)
                                    page_ok |= 1u << i;
                            }
                        }
                        const uint32_t all_pages = (1u << pages_per_tile) - 1u;
                        if (lane == 0) {
                            // rows of the tile: page i (a block of box_rows rows), then KV head hh
                            // of the unit (head_rows rows each), then slot.  A tile inside the
                            // length whose pages are all in range has every row valid.
                            const bool full = page_ok == all_pages && key0 + TK <= U.len;
                            uint32_t nloaded = full ? static_cast<uint32_t>(pages_per_tile) : 0u;
                            uint64_t rows = full ? ~0ull : 0ull;
                            for (int i = 0; i < (full ? 0 : pages_per_tile); ++i) {
                                if (!(page_ok & (1u << i))) continue;   // page_ok only: no pages[i]
                                ++nloaded;
                                const int nv = min(head_rows, U.len - (key0 + i * head_rows));
                                if (nv <= 0) continue;
                                const uint64_t bits = nv >= 64 ? ~0ull : ((1ull << nv) - 1ull);
                                for (int hh = 0; hh < p.kh; ++hh)
                                    rows |= bits << (i * box_rows + hh * head_rows);
                            }
                            mask = rows;
                            sm.stage_mask[s] = mask;
                            mbar_arrive_expect_tx(sm.full + s, nloaded * 2u * Gm::kHalves * box_bytes);
                            const int row_coord = U.g * p.kh * P + row_in_page;
                            // constant trip count: pages[] stays in registers
#pragma unroll
                            for (int i = 0; i < 8; ++i) {
                                if (!(page_ok & (1u << i))) continue;   // also every i >= pages_per_tile
                                const int dst = i * Gm::kHalves * box_rows * 128;   // block i
#pragma unroll
                                for (int h = 0; h < Gm::kHalves; ++h) {
                                    const int dh = dst + h * box_rows * 128;
                                    tma_load_3d(ktile + dh, &tm_k, 64 * h, row_coord, pages[i], sm.full + s);
                                    tma_load_3d(vtile + dh, &tm_v, 64 * h, row_coord, pages[i], sm.full + s);
                                }
                            }
                        }
                    }
                    __syncwarp();
                }
            }
            if (!ok) {
                *sm.abort = 1;
                record_error(p.err, kErrWaitEmpty);
                if (lane == 0) {
                    // let every load this warp issued land before the CTA can exit
                    for (int k = it - NPW; k >= 0 && k >= it - S; k -= NPW) {
                        if (!mbar_wait(sm.full + (k % S), (k / S) & 1, nullptr, kWaitLimitNs)) {
                            record_error(p.err, kErrDrain);
                            break;
                        }
                    }
                }
            }
        }
        return;
    }

    // ==================================================================== consumer warps
    const int rb_shift = VAR == kPaged ? 31 - __clz(min(p.page_size * p.kh, kTileKeys)) : 6;
    const int kh = VAR == kPaged ? p.kh : 1;
    const int head_shift = VAR == kPaged ? 31 - __clz(p.page_size) : 6;
    ConsumerState<D, GP, GW, MULTI> cs;
    cs.init(warp, lane, p.G * p.sq, kh, rb_shift, head_shift, p.sq);
    uint32_t gphase = 0;

    if (VAR == kDense && dlen == 0) {
        // a device-resident length of 0: every row is a zero row (null-row convention)
        for (size_t idx = static_cast<size_t>(blockIdx.x) * kConsumerThreads + threadIdx.x;
             idx < static_cast<size_t>(p.B) * p.Hq * p.sq * D;
             idx += static_cast<size_t>(gridDim.x) * kConsumerThreads)
            p.out[idx] = __float2bfloat16_rn(0.f);
    }
    if (VAR == kPaged) {
        // sequences with no rows get zero rows (null-row convention)
        for (int b = blockIdx.x; b < p.B; b += gridDim.x) {
            if (sm.seq_len[b] != 0) continue;
            for (int idx = threadIdx.x; idx < p.Hq * p.sq * D; idx += kConsumerThreads)
                p.out[static_cast<size_t>(b) * p.Hq * p.sq * D + idx] = __float2bfloat16_rn(0.f);
        }
    }

    int it = 0;
    if (VAR == kSparse) {
        for (int item = it_begin; item < it_end; ++item) {
            int sp_u, sp_key0, sp_nkeys, ta, tb;
            sparse_item(item, sp_u, sp_key0, sp_nkeys, ta, tb);
            Unit U;
            U.u = sp_u;
            U.b = sp_u / p.Hkv;
            U.g = sp_u - U.b * p.Hkv;
            U.len = p.width;
            U.nt = 0;
            U.base = 0;
            U.hq0 = U.b * p.Hq + U.g * p.G;
            U.nh = p.G;
            U.cu = sp_u;
            cs.load_q(p, U.hq0, U.nh);
            cs.reset();
            for (int t = ta; t < tb; ++t, ++it) {
                const int s = it % S;
                const uint32_t ph = (it / S) & 1;
                if (!mbar_wait_warp(sm.full + s, ph, sm.abort)) {
                    *sm.abort = 1;
                    record_error(p.err, kErrWaitFull);
                    return;
                }
                const uint32_t ktile = smem_u32(sm.stages + s * Gm::kStageBytes);
                cs.consume(ktile, ktile + Gm::kTileBytes, sm.stage_mask[s], p.scale_log2, 0, 0,
                           0x7fffffff);
                __syncwarp();
                if (lane == 0) mbar_arrive(sm.empty + s);
            }
            // a partial is only stored here; its unit's counter is bumped after the last item
            if (!finish_segment<D, GP>(p, sm, cs, U, p.nchunks == 1, item, sp_u * p.nchunks,
                                       p.nchunks, gphase, true))
                return;
        }
        if (p.nchunks > 1 && it_begin < it_end)
            publish_and_merge<D, GP>(p, sm, sm.seq_len, it_begin, it_end, gphase);
        return;
    }

    Unit U;
    if (t0 < t1) {
        U = VAR == kDense ? locate_dense(p, t0, dlen, dtiles) : locate_paged(p, sm, t0);
        cs.load_q(p, U.hq0, U.nh);
    }
    for (int t = t0; t < t1;) {
        const int tend = min(t1, U.base + U.nt);
        const bool whole = (t == U.base) && (tend == U.base + U.nt);
        const int c_first = tile_owner(U.base, N, C);
        const int c_last = tile_owner(U.base + U.nt - 1, N, C);
        const int tk = VAR == kPaged ? p.tile_keys : kTileKeys;
        const int causal_base = U.len - p.sq;
        const int causal_from = p.causal ? causal_base + 1 : 0x7fffffff;
        cs.reset();
        for (; t < tend; ++t, ++it) {
            const int s = it % S;
            const uint32_t ph = (it / S) & 1;
            if (!mbar_wait_warp(sm.full + s, ph, sm.abort)) {
                *sm.abort = 1;
                record_error(p.err, kErrWaitFull);
                return;
            }
            const uint32_t ktile = smem_u32(sm.stages + s * Gm::kStageBytes);
            cs.consume(ktile, ktile + Gm::kTileBytes, sm.stage_mask[s], p.scale_log2,
                       (t - U.base) * tk, causal_base, causal_from);
            __syncwarp();
            if (lane == 0) mbar_arrive(sm.empty + s);
        }
        // the next segment's Q rows are fetched now so their latency hides behind the finish
        Unit next = U;
        if (t < t1) {
            next = VAR == kDense ? locate_dense(p, t, dlen, dtiles) : locate_paged(p, sm, t);
            cs.load_q(p, next.hq0, next.nh);
        }
        if (!finish_segment<D, GP>(p, sm, cs, U, whole, static_cast<int>(blockIdx.x) + U.u,
                                   c_first + U.u, c_last - c_first + 1, gphase))
            return;
        U = next;
    }
}

}  // namespace da
