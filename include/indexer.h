/*
 * indexer.h -- C ABI of the GB300 (sm_103a) dense prefill indexer.
 *
 * The indexer scores every query row t of a prefill chunk against every
 * compressed prefix key j of the row's request,
 *
 *     logit[t,j] = sum_h w[t,h] * ReLU( s_q[t,h] * s_k[j] * <q[t,h,:], k[j,:]> ),
 *
 * for j < compress_len(t) (the row's causal length), and keeps each row's
 * top-k keys.  Sources, by page and section:
 *   - "chunked-prefill-memory.md", section 1: the low-ratio indexer scores the
 *     chunk's T rows against the whole compressed prefix L and writes
 *     [T, max_seqlen_k] fp32 logits; section 2.3: key blocks with a per-block
 *     top-k and an exact top-k of the union; 8-key block pooling with the
 *     top-2048 blocks as candidates; consumers mask non-candidates.
 *   - SGLang PR #39187 "Bound the dense prefill indexer transient",
 *     Motivation/Modifications: DeepGEMM fp8_fp4_mqa_logits scoring, ragged
 *     requests, a caller-owned `selected` output, masks built straight into
 *     one preallocated buffer, a bounded transient; a block-level mask as the
 *     follow-up format.
 *   - SGLang fork commit log, the ragged-plan commit: per-batch metadata is
 *     built once and reused by every layer; host lengths avoid device syncs.
 * The score formula is the DeepSeek-V4 / NSA indexer's own (ReLU of the
 * scaled per-head dot products, weighted by w over the heads); the pages name
 * its kernels (fp8 / fp8_fp4 MQA logits) but never print it.
 *
 * Conventions shared by every entry point:
 *   - Layout.  Rows of all requests are packed: request r owns global rows
 *     [cu_seqlens_q[r], cu_seqlens_q[r+1]) and packed keys
 *     [cu_seqlens_k[r], cu_seqlens_k[r+1]).  Key indices in outputs are
 *     request-local (0 = first key of the row's request).
 *   - Eligibility.  Key j is eligible for row t iff j < compress_len[t]
 *     (compress_len is clamped to the request's key count) and, when a
 *     candidate mask is given, its block byte is non-zero.
 *   - Ties.  Equal scores are ordered by the lower key index.
 *   - Output order.  Kept indices are listed in ascending key order, then -1
 *     padding; `out_val` (optional) holds each kept key's score, -inf for
 *     padding.  Results are bitwise reproducible run to run and do not
 *     depend on the workspace size or the key-block size.
 *   - Ownership.  The caller owns every buffer (inputs, outputs, workspace).
 *     The plan owns only host metadata; the library allocates no device
 *     memory.  Device pointers are CUDA device addresses on the current
 *     device; `stream` is a cudaStream_t (NULL = legacy default stream).
 *   - Errors.  Return codes only (no exceptions, no exit, no printing).
 *     Argument errors are caught on the host before any launch.  Calls are
 *     asynchronous and never synchronize; a device-side failure (a wait that
 *     timed out) sets a status word in the workspace that indexer_status()
 *     reads.
 *   - Preconditions the library does not check on the device: q/k codes are
 *     finite (no e4m3 NaN codes 0x7F/0xFF, no ue8m0 255), scales s_q, s_k are
 *     positive and finite (so ReLU(s*x) = s*ReLU(x)), w is finite.
 */
#ifndef GB300_PREFILL_INDEXER_H
#define GB300_PREFILL_INDEXER_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes. */
#define IDX_OK 0
#define IDX_ERR_INVALID_ARG (-1)   /* bad size, pointer, alignment or layout */
#define IDX_ERR_UNSUPPORTED (-2)   /* shape/format the library has no kernel for, or not sm_103 */
#define IDX_ERR_WORKSPACE (-3)     /* workspace too small, or budget impossible at plan time */
#define IDX_ERR_CUDA (-4)          /* a CUDA runtime/driver call failed */
#define IDX_ERR_TIMEOUT (-5)       /* a device-side wait ran out (reported by indexer_status) */
#define IDX_ERR_DEVICE_CHECK (-6)  /* a device-side check failed (reported by indexer_status) */

/* Key formats. */
#define IDX_K_FP8_E4M3 0           /* k: e4m3 [keys, D]; k_scale: float s_k[keys] */
#define IDX_K_FP4_E2M1_UE8M0 1     /* k: e2m1 [keys, D/2], element 2i in the low nibble;
                                      k_scale: uint8 ue8m0 [keys, D/32]; s_k is 1.  With 32
                                      heads of 128 the block-scaled MMA applies the block
                                      scales (any block-scale span; k_scale 4-byte
                                      aligned); other head counts score the keys through
                                      their exact e4m3 form (see indexer_convert_fp4) */

/* Query formats. */
#define IDX_Q_FP8_E4M3 0           /* q: e4m3 [T, H, D]; s_q: float [T, H] */
#define IDX_Q_FP4_E2M1_UE8M0 1     /* q: e2m1 [T, H, D/2], element 2i in the low nibble;
                                      the s_q argument carries its block scales instead of
                                      float scales: uint8 ue8m0 [T, H, D/32] (4-byte
                                      aligned, passed as (const float*)); value =
                                      e2m1(code) * 2^(e - 127).  Needs kdtype
                                      IDX_K_FP4_E2M1_UE8M0 and 32 heads of 128: both operands
                                      then stay e2m1 in the block-scaled fp4 MMA
                                      (tcgen05 kind::mxf4, ue8m0 per 32 elements), any
                                      block-scale span on either side */

/* Row selection strategies of indexer_fused_topk (both exact). */
#define IDX_SELECT_AUTO 0          /* sampled row thresholds where rows are long enough,
                                      the running-threshold stream for undecided rows */
#define IDX_SELECT_STREAM 1        /* the running-threshold stream for every row */

/*
 * Problem description, read only by indexer_plan (host memory, copied).
 *   num_requests  R >= 1 (at most 256)
 *   total_rows    T = cu_seqlens_q[R];  total_keys = cu_seqlens_k[R]
 *   H, D          heads and head dim of q; k has D too.  Built shapes:
 *                 (H, D) in {(32,128), (16,128), (64,128), (8,64), (4,64)}; 4 heads run
 *                 as 8 (zero-padded into the workspace, which adds exactly 0)
 *   topk          keys kept per row, 1 <= topk <= 2048
 *   cu_seqlens_q  [R+1] non-decreasing row offsets, starts at 0
 *   cu_seqlens_k  [R+1] non-decreasing key offsets, starts at 0
 *   compress_len  [T] causal length of every row, 0 <= compress_len[t] <= the
 *                 keys of its request (e.g. floor((pos+1)/ratio))
 *   kdtype        IDX_K_FP8_E4M3 or IDX_K_FP4_E2M1_UE8M0
 *   qdtype        IDX_Q_FP8_E4M3 (0) or IDX_Q_FP4_E2M1_UE8M0; other values
 *                 IDX_ERR_INVALID_ARG, an unsupported pairing IDX_ERR_UNSUPPORTED
 *   cand_block    keys per candidate block: 1, 2, 4 or 8 (0 means 8)
 *   cand_topk     candidate blocks kept per row by indexer_candidate_blocks,
 *                 1..4096 (e.g. 2048); 0 = the plan makes no candidate-block
 *                 calls and reserves no workspace for them
 *   key_block     keys per key block of the streamed top-k (0 = planner's
 *                 choice; else a multiple of 128)
 *   transient_budget_bytes  cap on the workspace of the top-k and candidate
 *                 calls (0 means 2 GiB); the planner shrinks key blocks and
 *                 row chunks to fit and fails with IDX_ERR_WORKSPACE if it
 *                 cannot.
 *   select_mode   IDX_SELECT_AUTO or IDX_SELECT_STREAM.  AUTO scores every
 *                 32nd-or-so key tile first and takes, per row, a threshold a
 *                 little below the expected k-th score; the lists then hold every
 *                 key at or above it, and a row whose lists hold fewer than k
 *                 keys (or overflow) is selected again by the stream.  Results
 *                 are identical; only the work differs.
 */
typedef struct indexer_problem {
    int32_t num_requests;
    int32_t total_rows;
    int32_t total_keys;
    int32_t H;
    int32_t D;
    int32_t topk;
    const int32_t* cu_seqlens_q;
    const int32_t* cu_seqlens_k;
    const int32_t* compress_len;
    int32_t kdtype;
    int32_t cand_block;
    int32_t cand_topk;
    int32_t key_block;
    uint64_t transient_budget_bytes;
    int32_t select_mode;
    int32_t qdtype;
} indexer_problem;

typedef struct indexer_plan_s* indexer_plan_t;

/*
 * Validate a problem and build its plan (host metadata only: ragged tables,
 * key-block and row-chunk sizes, workspace layout).  Built once per batch and
 * reused by every layer of that batch (SGLang fork commit log, ragged-plan
 * commit).  *workspace_bytes receives the workspace every call on this plan
 * needs.  Needs no GPU.  Returns IDX_OK, IDX_ERR_INVALID_ARG,
 * IDX_ERR_UNSUPPORTED or IDX_ERR_WORKSPACE (budget impossible).
 */
int indexer_plan(const indexer_problem* problem, indexer_plan_t* out_plan,
                 size_t* workspace_bytes);
void indexer_plan_destroy(indexer_plan_t plan);

/* Key-block size, row-chunk size, key splits per row and key-tile sampling
 * stride (0 = no sampled thresholds) the plan chose (for reporting); any
 * pointer may be NULL. */
int indexer_plan_info(indexer_plan_t plan, int32_t* key_block, int32_t* row_chunk,
                      int32_t* max_splits, int32_t* sample_stride);

/*
 * Dense logits ("chunked-prefill-memory.md" section 1: [T, max_seqlen_k] fp32).
 *   q        e4m3 [T, H, D] (16-byte aligned)
 *   s_q, w   float [T, H]
 *   k        see kdtype (16-byte aligned); k_scale see kdtype
 *   compress_len  int32 [T] on the device, same values as the plan's
 *   logits   float [T, ld], ld >= the largest key count of the batch;
 *            logits[t, j] for j < compress_len[t], -inf for the rest of the row
 * ws/ws_bytes: the plan's workspace (256-byte aligned).
 * Range: every head's score (its fp32 dot product, block scales included) is applied
 * exactly for 2^-62 <= |S| < 2^64 (smaller ones keep an absolute error below 2^-150
 * times the head weight), with |w * s_q| < 2^64.
 */
int indexer_logits(indexer_plan_t plan, const void* q, const float* s_q, const float* w,
                   const void* k, const void* k_scale, const int32_t* compress_len,
                   float* logits, int64_t ld, void* ws, size_t ws_bytes, void* stream);

/*
 * Ragged per-row top-k over given logits [T, ld] (the ragged top-k of
 * "chunked-prefill-memory.md" section 2.3).  Entries j >= compress_len[t] and
 * -inf entries are not eligible.  out_idx int32 [T, topk]; out_val float
 * [T, topk] or NULL.  A row's kept keys are written in ascending key order,
 * then -1 (value -inf) padding.
 * With at least the plan's workspace, rows are sampled for a threshold and read
 * once (for 16-byte aligned rows of at most 65,536 keys the candidates and the
 * exact selection stay in shared memory); rows the sample cannot decide, and
 * every row when ws holds only the status area (256 bytes), get a direct exact
 * selection.  All of these give identical outputs.
 */
int indexer_topk(indexer_plan_t plan, const float* logits, int64_t ld,
                 const int32_t* compress_len, int32_t* out_idx, float* out_val, void* ws,
                 size_t ws_bytes, void* stream);

/*
 * Fused logits + top-k with a bounded transient: keys are scored block by
 * block and only per-block top-k candidates are kept, then merged exactly
 * ("chunked-prefill-memory.md" section 2.3); the [T, L] logits are never
 * materialised.  cand_mask (nullable) uint8 [T, ld_mask]: one byte per
 * cand_block-key block, non-zero = candidate (the consumer layer's mask);
 * ld_mask >= ceil(L/cand_block) for every request.
 */
int indexer_fused_topk(indexer_plan_t plan, const void* q, const float* s_q, const float* w,
                       const void* k, const void* k_scale, const int32_t* compress_len,
                       const uint8_t* cand_mask, int64_t ld_mask, int32_t* out_idx,
                       float* out_val, void* ws, size_t ws_bytes, void* stream);

/*
 * Candidate-source layer: pool each row's logits over cand_block-key blocks
 * (maximum over eligible keys, blocks aligned at key 0), keep the cand_topk
 * blocks with the largest pooled score (ties to the lower block) and write a
 * block-level mask: cand_mask uint8 [T, ld_mask], 1 = kept, 0 otherwise
 * (every byte of every row is written).  ld_mask >= ceil(L/cand_block).
 */
int indexer_candidate_blocks(indexer_plan_t plan, const void* q, const float* s_q,
                             const float* w, const void* k, const void* k_scale,
                             const int32_t* compress_len, uint8_t* cand_mask, int64_t ld_mask,
                             void* ws, size_t ws_bytes, void* stream);

/*
 * Expand a block-level mask to the key-level bool layout the pages' consumer
 * format uses: key_mask uint8 [T, ld], key_mask[t,j] = cand_mask[t, j/cand_block]
 * for j < compress_len[t], 0 otherwise.
 */
int indexer_expand_mask(indexer_plan_t plan, const uint8_t* cand_mask, int64_t ld_mask,
                        const int32_t* compress_len, uint8_t* key_mask, int64_t ld,
                        void* stream);

/*
 * Synchronizes `stream`, then reads the device status word in `ws`: IDX_OK,
 * IDX_ERR_TIMEOUT or IDX_ERR_DEVICE_CHECK.  Every compute call clears the
 * word when it starts.
 */
int indexer_status(indexer_plan_t plan, const void* ws, void* stream);

/*
 * Self-test of the bounded waits: launches one tiny kernel that waits on a
 * barrier nothing arrives on, with a budget of `cycles` SM cycles; it must
 * give up and set the timeout bit in the status word of `ws` (then
 * indexer_status returns IDX_ERR_TIMEOUT).  Never hangs.
 */
int indexer_selftest_timeout(void* ws, long long cycles, void* stream);

/* Budget, in SM clock cycles, of every device-side wait of later calls
   (default about two seconds). */
int indexer_set_wait_budget(indexer_plan_t plan, long long cycles);

/*
 * Fused top-k without a caller-provided workspace (no counterpart on the
 * pages: this entry point exists for callers that cannot allocate device
 * memory).  Some callers have no way to obtain device memory for a workspace:
 * a plugin whose host application owns all device memory through its own pool
 * and exposes no allocator, or a serving loop in which a cudaMalloc would
 * stall every stream on the device.  This variant computes exactly what
 * indexer_fused_topk computes, with the same arguments minus ws/ws_bytes; its
 * workspace is a file-scope device array of IDX_NOALLOC_SCRATCH_BYTES (64 MiB)
 * that every GPU loading this library holds until the process exits.
 *   - Limit: the plan's workspace must fit the array; build the plan with
 *     transient_budget_bytes <= 64 MiB.  A larger plan is rejected with
 *     IDX_ERR_WORKSPACE before anything is launched.
 *   - Allocation: none.  No cudaMalloc, cudaFree or allocating library call.
 *   - Set-up: the first call on a device resolves the array's device address
 *     (cudaGetSymbolAddress) with that device current and caches it; make
 *     that first call before any stream capture.
 *   - Sharing: every call uses the same array and it keeps the previous call's
 *     contents (the call clears what it needs cleared).  Calls whose work
 *     overlaps on the GPU (different streams, or several threads) race on the
 *     array: serialize them.
 *   - Status: device-side failures of a call (a wait that ran out, an e2m1 key
 *     the e4m3 conversion cannot represent, a candidate-mask row out of range) are recorded
 *     in the array's status word, which the call clears when it starts.
 *     indexer_noalloc_status reads it, as indexer_status reads a workspace.
 */
#define IDX_NOALLOC_SCRATCH_BYTES (64ull << 20)
int indexer_fused_topk_noalloc(indexer_plan_t plan, const void* q, const float* s_q,
                               const float* w, const void* k, const void* k_scale,
                               const int32_t* compress_len, const uint8_t* cand_mask,
                               int64_t ld_mask, int32_t* out_idx, float* out_val, void* stream);

/* Status of the last indexer_fused_topk_noalloc call on the current device
 * (no counterpart in the pages either: it is the allocation-free variant's
 * indexer_status).  Synchronizes `stream`, then reads the status word of the
 * library's scratch array: IDX_OK, IDX_ERR_TIMEOUT or IDX_ERR_DEVICE_CHECK
 * exactly as indexer_status; IDX_ERR_CUDA if a CUDA call fails,
 * IDX_ERR_UNSUPPORTED on a device other than sm_103.  Allocates nothing. */
int indexer_noalloc_status(void* stream);

/* Diagnostic: synchronizes `stream` and returns how many rows the last
   indexer_fused_topk / indexer_candidate_blocks / indexer_topk call on this
   workspace sent to the exact path (rows its sampled threshold could not
   decide), or a negative status.  The result is right only while the
   workspace has not been used by another call since. */
long long indexer_fallback_rows(indexer_plan_t plan, const void* ws, void* stream);

/* Number of kernels this library has launched in this process (a
   diagnostic counter for benchmarks; never reset). */
long long indexer_launch_count(void);

/* Benchmark diagnostic: while set, every indexer_fused_topk /
   indexer_candidate_blocks call records start_event (a cudaEvent_t) on its
   stream just before the first list-filling logits launch of its first pass
   and stop_event just after it, so the caller can time the dominant kernel
   inside a step.  NULL, NULL turns it off.  Process-wide, not thread-safe;
   the events are owned by the caller. */
void indexer_profile_main_kernel(void* start_event, void* stop_event);

/* ------------------------------------------- tail-only candidates, row maps
 * Under a decoder sliding-window bounded replay only each request's tail rows
 * are consumed by the later layers ("[SGLang PR 39187]", the third change:
 * publish only each request's tail rows, since the consumer slices every mask
 * down to them anyway).
 *
 * indexer_candidate_blocks_tail: indexer_candidate_blocks for request r's last
 *   publish_rows[r] rows only (host array [num_requests], 0 <= publish_rows[r]
 *   <= rows of r), packed: cand_mask is [sum_r publish_rows[r], ld_mask], request
 *   order, each request's rows in order.  Only those rows are scored.  A row's
 *   mask is byte-identical to the one indexer_candidate_blocks gives it.
 *   IDX_ERR_INVALID_ARG for a count out of range or a NULL array.
 *
 * indexer_fused_topk_mapped: indexer_fused_topk with a candidate mask whose rows
 *   are addressed through a row map: row t of the batch uses mask row
 *   mask_rows[t] (device int32 [total_rows]) of cand_mask [mask_row_count,
 *   ld_mask].  A map entry outside [0, mask_row_count) is reported by
 *   indexer_status as IDX_ERR_DEVICE_CHECK (that row then reads mask row 0).
 *   cand_mask and mask_rows are required (IDX_ERR_INVALID_ARG otherwise).
 */
int indexer_candidate_blocks_tail(indexer_plan_t plan, const void* q, const float* s_q,
                                  const float* w, const void* k, const void* k_scale,
                                  const int32_t* compress_len, const int32_t* publish_rows,
                                  uint8_t* cand_mask, int64_t ld_mask, void* ws,
                                  size_t ws_bytes, void* stream);
int indexer_fused_topk_mapped(indexer_plan_t plan, const void* q, const float* s_q,
                              const float* w, const void* k, const void* k_scale,
                              const int32_t* compress_len, const uint8_t* cand_mask,
                              int64_t ld_mask, const int32_t* mask_rows, int64_t mask_row_count,
                              int32_t* out_idx, float* out_val, void* ws, size_t ws_bytes,
                              void* stream);

/* ------------------------------------------------------------ fp4 operands
 * Exact conversion of e2m1 codes with one ue8m0 exponent per 32 elements
 * (OCP MX fp4: value = e2m1(code) * 2^(e - 127)) into e4m3 codes and one fp32
 * scale per row, value = e4m3(out) * out_scale[row] exactly, out_scale =
 * 2^(largest block exponent of the row - 127).  This is how the library runs
 * e2m1 keys for head counts without a block-scaled kernel (inside the calls, kdtype
 * IDX_K_FP4_E2M1_UE8M0; 32 heads of 128 use the block-scaled MMA instead), and how a
 * caller runs e2m1 queries with those head counts: convert q as T*H rows of D and pass
 * the e4m3 codes as q and the row scales as s_q (qdtype IDX_Q_FP8_E4M3).  With 32 heads
 * of 128, qdtype IDX_Q_FP4_E2M1_UE8M0 scores e2m1 queries natively instead.
 *   codes: device [rows, D/2] bytes, element 2i in the low nibble;
 *   block_scales: device [rows, D/32]; D a multiple of 32 (64 or 128 here);
 *   out_e4m3: device [rows, D]; out_scale: device fp32 [rows];
 *   ws: at least 256 bytes of device memory, 256-byte aligned: its status word is
 *   cleared, and a row whose smaller blocks fall below e4m3's range sets a bit
 *   that indexer_status(NULL, ws) reports as IDX_ERR_DEVICE_CHECK (read it before
 *   the workspace is used by another call, which clears it).
 * Async on `stream`, no allocation.
 */
int indexer_convert_fp4(const uint8_t* codes, const uint8_t* block_scales, int64_t rows,
                        int32_t D, uint8_t* out_e4m3, float* out_scale, void* ws,
                        size_t ws_bytes, void* stream);

/* ------------------------------------------------------ page-index transform
 * The indexer's selected keys as KV-cache slots ("[SGLang PR 39187]",
 * Accuracy / equivalence: the indexer's outputs are page_indices and
 * raw_indices; the pages name the top-k-then-transform step without printing
 * it, so this is the usual paged addressing):
 *     page_idx[t, i] = page_table[r, j / page_size] * page_size + j % page_size
 * for j = raw_idx[t, i] with 0 <= j < L_r, r the request of row t (the plan's
 * cu_seqlens_q) and L_r its key count (cu_seqlens_k); -1 where j is -1 or out
 * of [0, L_r), where the table entry is negative (an unmapped page), or where
 * the slot does not fit an int32.
 *   raw_idx, page_idx: device int32 [total_rows, topk] (the plan's topk), row-major;
 *     page_idx may equal raw_idx (in place).
 *   page_table: device int32 [num_requests, ld_page_table], row r holds request
 *     r's physical page of each logical page; ld_page_table must be at least
 *     ceil(max L_r / page_size), else IDX_ERR_INVALID_ARG.
 *   page_size >= 1 (a power of two takes a shift path).
 * Async on `stream`, no allocation, no workspace, no device-side errors.
 */
int indexer_page_indices(indexer_plan_t plan, const int32_t* raw_idx, const int32_t* page_table,
                         int64_t ld_page_table, int32_t page_size, int32_t* page_idx,
                         void* stream);

/* ------------------------------------------------------------ chunk planner
 * Adaptive prefill chunk ("chunked-prefill-memory.md", section 2.1, for callers
 * that still materialise [T, L] fp32 logits and must keep T x L under a budget):
 * for a prefix of prefix_len compressed keys
 *     chunk(L) = clamp( round_down( budget_token2 / L ), chunk_min, chunk_max )
 * where round_down goes to a multiple of `page` (pow2 == 0: the section's
 * formula) or to a power of two (pow2 != 0: this reproduces the schedule the
 * section prints -- 2048 up to ~98k keys, 1024 to ~195k, 512 to ~390k, 256
 * beyond).  The section's values: budget_token2 = 2.0e8, chunk_min = 256,
 * chunk_max = 2048, page = 256.  prefix_len <= 0 gives chunk_max.
 * Returns the chunk (>= chunk_min > 0), or IDX_ERR_INVALID_ARG when
 * budget_token2 <= 0 (or not finite), chunk_min < 1, chunk_max < chunk_min or
 * page < 1.  Host only: no device, no allocation, thread-safe.
 */
int indexer_chunk_rows(int64_t prefix_len, double budget_token2, int32_t chunk_min,
                       int32_t chunk_max, int32_t page, int32_t pow2);

const char* indexer_error_string(int status);
int indexer_version(void);

#ifdef __cplusplus
}
#endif
#endif
