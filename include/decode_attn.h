/*
 * decode_attn.h -- C ABI of the GB300 (sm_103a) single-query decode-attention library.
 *
 * One query row per (sequence b, query head h) attends a KV cache with softmax_scale and GQA
 * grouping (query head h reads KV head h / (Hq / Hkv)).  There is no ALiBi, no sliding window
 * and no logit softcap, and causal masking is not a parameter: with one query row it changes
 * nothing ("DecodeFlashSpec", fuel_dispatch::decode_flash, fields alibi / causal /
 * window_size_left / window_size_right / softcap).  Three forms:
 *   decode_attn_dense   rows [0, k_len) of a capacity buffer      (DecodeFlashSpec, k / v / k_len)
 *   decode_attn_paged   per-sequence kv_len read on the device from an args buffer, rows gathered
 *                       through a block table       ("DflashScratch", option_b_indirect_args_dev)
 *   decode_attn_sparse  a fixed-width int32 selection whose -1 pads add exactly nothing
 *                       ("AttnV41", decode_fixed_topk / decode_prep)
 *
 * Conventions shared by every entry point
 *   - Element type: every q / k / v / out buffer holds bfloat16 values (2 bytes each); the
 *     arithmetic is fp32 (scores, online softmax, accumulation), the output is rounded to bf16
 *     round-to-nearest-even.
 *   - Pointers: q, k, v, pools, out, block_table, kv_lens, sel and the workspace are DEVICE
 *     pointers of the current CUDA device, owned by the caller; q, k, v, pools, out and the
 *     workspace must be 16-byte aligned, block_table / kv_lens / sel 4-byte aligned.
 *   - Layouts are dense row-major with D contiguous:
 *       q, out          [B, Hq, 1, D]
 *       dense k, v      [B, Hkv, capacity, D]
 *       paged pools     [num_pages, Hkv, page_size, D]   (one page of one KV head is contiguous)
 *       block_table     int32 [B, max_pages_per_seq]
 *       kv_lens         u32 words; sequence b's kv_len is kv_lens[b * kv_len_stride]
 *       sparse pools    [B, Hkv, pool_rows, D]
 *       sel             int32 [B, width], shared by every KV head of a sequence
 *   - Supported: D in {64, 128}; 1 <= Hq / Hkv <= 64.  Other shapes return DA_ERR_UNSUPPORTED
 *     (fail closed, nothing launched).
 *   - Streams: a call only enqueues work on `stream` (a cudaStream_t; NULL is the legacy
 *     default stream).  It allocates nothing, frees nothing and never synchronises.  The calls
 *     that take a caller-owned workspace, and the append calls, can therefore be captured in a
 *     CUDA graph; the tensor-map descriptors and launch arguments they build are baked into the
 *     launch.
 *   - Values that live on the device (kv_lens, block_table, sel) are never checked by a
 *     device-to-host copy.  They are handled on the device: kv_len is clamped to
 *     max_pages_per_seq * page_size; a row whose block-table entry lies outside [0, num_pages),
 *     and a selection entry outside [0, pool_rows) (-1 or any other), is skipped; an empty row
 *     set (k_len = 0, kv_len = 0, an all-pad selection) yields a zero output row.
 *   - Errors: the return value is checked on the host before anything is enqueued; on any
 *     status other than DA_OK nothing was launched and `out` is untouched.
 *   - Workspace: caller-owned device scratch of at least decode_attn_workspace_size() bytes.
 *     It must be zero-filled once before its first use (decode_attn_workspace_init or
 *     cudaMemset); every completed call leaves its counters at zero again, so later calls need
 *     no clearing.  One workspace must not be shared by calls that can run concurrently.  A call
 *     that stopped on a timed-out wait (decode_attn_read_device_error returns nonzero) may leave
 *     counters set: zero-fill the workspace again before reusing it.
 */
#ifndef DECODE_ATTN_H
#define DECODE_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define DECODE_ATTN_ABI_VERSION 1

typedef enum {
    DA_OK = 0,
    DA_ERR_INVALID_ARGUMENT = 1,   /* null/misaligned pointer, bad shape or length, bad scale */
    DA_ERR_UNSUPPORTED = 2,        /* valid request outside the kernels' shape support */
    DA_ERR_WORKSPACE_TOO_SMALL = 3,
    DA_ERR_CUDA = 4                /* a CUDA runtime call or kernel launch failed */
} da_status;

typedef enum { DA_VARIANT_DENSE = 0, DA_VARIANT_PAGED = 1, DA_VARIANT_SPARSE = 2 } da_variant;

/* DECODE_ATTN_ABI_VERSION of the built library. */
int decode_attn_abi_version(void);

/* Static, human-readable text for a da_status value (never NULL). */
const char *decode_attn_status_string(int status);

/* Workspace bytes a call of `variant` needs on the current device for these shapes.
 * max_kv is the selection width for DA_VARIANT_SPARSE and is ignored otherwise.
 * Returns 0 for arguments the calls would reject. */
size_t decode_attn_workspace_size(int variant, int B, int Hq, int Hkv, int D, int64_t max_kv);

/* Zero-fills `bytes` of a workspace on `stream` (cudaMemsetAsync). */
da_status decode_attn_workspace_init(void *workspace, size_t bytes, void *stream);

/*
 * Dense decode attention over the live prefix of a capacity buffer.
 * Follows "DecodeFlashSpec" (docs.rs fuel_dispatch::decode_flash): q [B,Hq,1,D] attends rows
 * [0, k_len) of k, v [B,Hkv,capacity,D]; k_len is the live length cached_len + seq
 * (field k_len, resolved to a concrete value per call); rows at or past k_len are never read.
 *   0 <= k_len <= capacity, capacity >= 1; k_len = 0 writes zeros.
 *   softmax_scale: finite; typically 1/sqrt(D) (field softmax_scale).
 */
da_status decode_attn_dense(const void *q, const void *k, const void *v, void *out, int B, int Hq,
                            int Hkv, int D, int64_t capacity, int64_t k_len, float softmax_scale,
                            void *workspace, size_t workspace_bytes, void *stream);

/*
 * decode_attn_dense with the live length read on the device.
 * Follows "DecodeFlashSpec", field k_len: for a persistent (plan-once) decode graph k_len is a
 * symbol bound to the live length each token; here it is one u32 in device memory (*k_len), read
 * by the kernel at entry and clamped to capacity, so a captured graph replays for every token
 * while the caller rewrites that word in place (k_len = 0 writes zeros).  The last tile of each
 * (b, kv head) may fetch up to 63 rows past the length (inside the capacity buffer); they never
 * contribute.  Other arguments as for decode_attn_dense; k_len must be 4-byte aligned.
 */
da_status decode_attn_dense_device_len(const void *q, const void *k, const void *v, void *out,
                                       int B, int Hq, int Hkv, int D, int64_t capacity,
                                       const uint32_t *k_len, float softmax_scale,
                                       void *workspace, size_t workspace_bytes, void *stream);

/*
 * Paged decode attention with per-sequence lengths read on the device.
 * Follows "DflashScratch" (docs.metrale.ai dflash_head), field option_b_indirect_args_dev: the
 * kernel reads kv_len of sequence b at entry from kv_lens[b * kv_len_stride]; stride 3 reads
 * the first word of the 12-byte record {u32 kv_len, u32 q_offset, u32 q_rope_pos}, stride 1 a
 * plain u32 array.  Row j of sequence b is slot j % page_size of page block_table[b][j /
 * page_size].  The pointer stays fixed while the host rewrites the values between launches.
 *   page_size: a power of two in [8, 256]; max_pages_per_seq >= 1; 1 <= num_pages < 2^31;
 *   kv_len_stride in {1, 3}; B <= 1024.
 */
da_status decode_attn_paged(const void *q, const void *k_pool, const void *v_pool, void *out,
                            const int32_t *block_table, int max_pages_per_seq, int page_size,
                            int64_t num_pages, const uint32_t *kv_lens, int kv_len_stride, int B,
                            int Hq, int Hkv, int D, float softmax_scale, void *workspace,
                            size_t workspace_bytes, void *stream);

/*
 * Several query tokens per sequence (a multi-token verify step): q, out [B, Hq, Sq, D].
 * Follows "DecodeFlashSpec" (q is [B, Hq, Sq, D]; field causal) and "AttnV41" method forward
 * (attention for m tokens at start_pos): the Sq new tokens are the last Sq rows of each
 * sequence's live prefix, so with causal != 0 token i attends rows [0, len - Sq + i] (a token with
 * no row gets a zero output row); with causal == 0 every token attends [0, len).  len is k_len
 * (dense) or the device-resident kv_len (paged).  Sq = 1 is decode_attn_dense /
 * decode_attn_paged.  Requires (Hq / Hkv) * Sq <= 64.  Workspace: decode_attn_workspace_size()
 * with Hq * Sq in place of Hq.  Other arguments as for the single-token calls.
 */
da_status decode_attn_dense_mq(const void *q, const void *k, const void *v, void *out, int B,
                               int Hq, int Hkv, int D, int Sq, int causal, int64_t capacity,
                               int64_t k_len, float softmax_scale, void *workspace,
                               size_t workspace_bytes, void *stream);

da_status decode_attn_paged_mq(const void *q, const void *k_pool, const void *v_pool, void *out,
                               const int32_t *block_table, int max_pages_per_seq, int page_size,
                               int64_t num_pages, const uint32_t *kv_lens, int kv_len_stride,
                               int B, int Hq, int Hkv, int D, int Sq, int causal,
                               float softmax_scale, void *workspace, size_t workspace_bytes,
                               void *stream);

/*
 * Sparse decode attention over a fixed-width selection.
 * Follows "AttnV41" (docs.metrale.ai attn_v41), methods decode_fixed_topk and decode_prep: each
 * sequence's selection lists pool rows (window slots, then the shared index selection, then -1
 * pads up to the fixed width); each valid entry adds its row once (duplicates count once per
 * entry); a -1 entry adds an exact zero to the denominator and nothing to the output.
 * Appending -1 pads to a selection leaves every output bit unchanged: the work is split into
 * chunks of 512 entries, a size that depends on nothing (not the width, B, G or the device), and
 * each chunk is computed and merged the same way whichever CTA takes it.  33 <= G <= 64 runs on
 * the fifth-generation tensor cores (tcgen05, accumulators in tensor memory), one CTA per
 * (sequence and KV head, chunk) holding all G heads; G <= 32 runs on warp-level MMAs, one CTA
 * per SM taking a contiguous range of whole chunks.
 *   1 <= pool_rows < 2^31; width >= 0 (width = 0 writes zeros).
 */
da_status decode_attn_sparse(const void *q, const void *k_pool, const void *v_pool, void *out,
                             int64_t pool_rows, const int32_t *sel, int width, int B, int Hq,
                             int Hkv, int D, float softmax_scale, void *workspace,
                             size_t workspace_bytes, void *stream);

/*
 * KV append into the paged cache (reshape_and_cache): the step before decode_attn_paged.
 * Follows "DflashScratch" (docs.metrale.ai dflash_head), field slot_mapping_dev: row t of k_new /
 * v_new ([T, Hkv, D], bf16) is written to every KV head of slot s = slot_mapping[t] (i64, device
 * memory) of the pools [num_pages, Hkv, page_size, D]: page s / page_size, position
 * s % page_size.  A slot outside [0, num_pages * page_size) (-1 padding or any other) writes
 * nothing; the slots are read on the device and never validated by a sync.  Two rows naming the
 * same slot race (one of them wins).  D a multiple of 8, at most 1024; k_new, v_new and the pools
 * 16-byte aligned, slot_mapping 8-byte aligned.  Enqueues one kernel on `stream`.
 */
da_status decode_attn_append_paged(const void *k_new, const void *v_new, void *k_pool,
                                   void *v_pool, const int64_t *slot_mapping, int64_t T, int Hkv,
                                   int D, int page_size, int64_t num_pages, void *stream);

/*
 * KV append into a ring window: the step before decode_attn_sparse.
 * Follows "AttnV41" (docs.metrale.ai attn_v41), method decode_body: the window ring write at
 * pos % window, the slot read on the device.  Row b of k_new / v_new ([B, Hkv, D]) is written to
 * row positions[b] % window (i64, device memory) of sequence b's pools [B, Hkv, pool_rows, D]
 * (the window occupies rows [0, window)); a negative position writes nothing.
 * 1 <= window <= pool_rows; alignment as for decode_attn_append_paged.
 */
da_status decode_attn_append_ring(const void *k_new, const void *v_new, void *k_pool,
                                  void *v_pool, const int64_t *positions, int B, int Hkv, int D,
                                  int64_t pool_rows, int window, void *stream);

/*
 * The options of a decode-attention region, as "DecodeFlashSpec" (docs.rs
 * fuel_dispatch::decode_flash) carries them next to q / k / v / k_len: nonzero has_* fields mean
 * the option is present.
 */
typedef struct {
    int has_alibi;          /* ALiBi slopes [Hq] present */
    int causal;             /* causal masking requested */
    int has_window_left;    /* left sliding-window bound present */
    int has_window_right;   /* right sliding-window bound present */
    int has_softcap;        /* logit softcap present */
    float softmax_scale;
} decode_attn_spec;

/*
 * Whether these kernels can compute the region (DecodeFlashSpec's gate): ALiBi, either
 * sliding-window bound or a softcap disqualify it (DA_ERR_UNSUPPORTED: the kernels have no such
 * parameter, so the caller keeps its decomposed path); causal is accepted and ignored, since one
 * query row attends the whole live prefix; a null spec or a non-finite scale is
 * DA_ERR_INVALID_ARGUMENT.  Host only; touches no device.
 */
da_status decode_attn_spec_check(const decode_attn_spec *spec);

/* decode_attn_spec_check, then decode_attn_dense with spec->softmax_scale. */
da_status decode_attn_dense_spec(const decode_attn_spec *spec, const void *q, const void *k,
                                 const void *v, void *out, int B, int Hq, int Hkv, int D,
                                 int64_t capacity, int64_t k_len, void *workspace,
                                 size_t workspace_bytes, void *stream);

/* Caps the number of CTAs the dense and paged calls spread their work over (0 = one per SM,
 * the default).  Process-wide; a smaller grid gives every KV head more split segments, which
 * exercises the cross-CTA log-sum-exp merge.  Returns DA_ERR_INVALID_ARGUMENT for a negative
 * value. */
da_status decode_attn_set_grid_limit(int max_ctas);

/* Reads and clears the device error word of the current device (synchronises the device).
 * A kernel whose bounded wait on a pipeline barrier timed out (about one second) stops its
 * work, records a nonzero code here and returns instead of hanging; 0 means no such event.
 * Codes: 1 a consumer's wait for a filled stage, 2 a producer's wait for a free stage, 3 the
 * consumer-group barrier, 4 the producer's drain of its own copies after an abort, 5 the check
 * below.  The first code recorded stays until it is read. */
da_status decode_attn_read_device_error(uint32_t *code);

/* A check of the failure path (packed_fused_kda_decode's fail-closed convention carried to the
 * device): enqueues one small kernel whose thread waits, with the bounded wait the decode
 * pipelines use, on a barrier that nothing completes; after limit_us microseconds the wait gives
 * up, code 5 is recorded in the device error word and the kernel returns.  The context stays
 * usable.  1 <= limit_us <= 1000000, else DA_ERR_INVALID_ARGUMENT.  The pages have no such
 * call; it exists so that a caller (and the tests) can see a timed-out wait surface as an error. */
da_status decode_attn_check_wait_timeout(uint32_t limit_us, void *stream);

/* Bytes of the library-owned device scratch that decode_attn_dense_noalloc uses: 4 MiB, present
 * on every GPU that loads the library until the process exits. */
#define DECODE_ATTN_NOALLOC_SCRATCH_BYTES (4u * 1024u * 1024u)

/*
 * decode_attn_dense without a workspace argument, for callers that cannot allocate device memory
 * where they call it: a plugin or custom operator inside a host framework that owns every device
 * allocation and passes the operator only its inputs and outputs; latency-critical decode loops,
 * where cudaMalloc may synchronise the device; processes that reserve nearly all HBM up front.
 * No counterpart in the pages: this entry point is an addition of this library.
 *
 * Same arguments, layouts and results as decode_attn_dense, minus the workspace: the scratch is a
 * file-scope device array of DECODE_ATTN_NOALLOC_SCRATCH_BYTES bytes inside the library.
 *   - Shapes whose workspace (decode_attn_workspace_size(DA_VARIANT_DENSE, ...)) exceeds that
 *     size return DA_ERR_WORKSPACE_TOO_SMALL before anything is enqueued.
 *   - Every call shares the array: calls that can overlap on the GPU (different streams, or
 *     several host threads on one device) race on it and must be serialised by the caller.
 *   - The array keeps the previous call's contents, so each call clears its merge counters (the
 *     part that must start at zero) on `stream` right before its kernel; that clearing and the
 *     kernel are all it enqueues, and a call rejected by an argument check enqueues nothing.
 *   - The first call on each device looks up the array's device address (with that device
 *     current) and caches it; make that first call before any stream capture on the device.  The
 *     cache belongs to the CUDA context: after a device reset the next call looks it up again
 *     (that call, too, should come before any stream capture).
 *   - It allocates nothing: no cudaMalloc, cudaFree or allocating library routine.
 */
da_status decode_attn_dense_noalloc(const void *q, const void *k, const void *v, void *out, int B,
                                    int Hq, int Hkv, int D, int64_t capacity, int64_t k_len,
                                    float softmax_scale, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* DECODE_ATTN_H */
