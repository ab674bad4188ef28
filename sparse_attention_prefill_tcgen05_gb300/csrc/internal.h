// Internal interfaces between the host library and the kernels.  Nothing in
// here crosses the C ABI.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace idx {

// Launch with programmatic stream serialization: the kernel may begin before the
// previous kernel in the stream has finished; it calls pdl_wait_then_release() before
// any global memory access.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t st, Args&&... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<Args&&>(args)...);
}

constexpr int kTileKeys = 128;   // MMA M: keys per tile (one TMEM lane each)
constexpr int kTileN = 256;      // MMA N: (row, head) columns per tile
constexpr int kMaxSegments = 48;
constexpr int kMaxRequests = 256;

// Device status word bits (OR-ed by kernels, read by indexer_status).
constexpr uint32_t kStatusTimeout = 1u << 0;
constexpr uint32_t kStatusBadArg = 1u << 1;
constexpr uint32_t kStatusListOverflow = 1u << 2;   // a streamed list lost entries
constexpr uint32_t kStatusFp4Range = 1u << 3;       // an e2m1 key has no exact e4m3 form

// Key formats.

// What the logits kernel does with each (row, key) score.
constexpr int kSinkLogits = 0;   // write fp32 to a [rows, ld] buffer
constexpr int kSinkStream = 1;   // append threshold-passing (score, key) to per-row lists
constexpr int kSinkPool = 2;     // same over cand_block-key block maxima (candidate blocks)
constexpr int kSinkFilter = 3;   // append entries at or above a fixed per-row threshold
constexpr int kSinkPoolFilter = 4;  // the same over cand_block-key block maxima

constexpr int kListsPerSplit = 4;     // one candidate sub-list per epilogue warp quadrant
constexpr int kMaxStreamSlots = 256;  // sub-lists per row (key splits x kListsPerSplit)
constexpr int kMaxMergePieces = 64;   // row pieces per merge launch

// A contiguous piece of work: some rows of one request against a key range
// of that request.  Units (row group x key chunk) are numbered per launch.
struct Segment {
    int32_t row_begin;   // first global row
    int32_t nrows;
    int32_t key_base;    // packed key row of request-local key 0
    int32_t key_count;   // keys of the request; compress_len is clamped to it
    int32_t j_begin;     // request-local first key scored here
    int32_t j_end;       // request-local end (exclusive) of keys written here
    int32_t unit_begin;  // first unit number of this segment in the launch
    int32_t n_row_groups;
    int32_t n_chunks;
    int32_t unit_tiles;  // key tiles per unit
    int32_t tile_stride; // 1: every key tile; s: tiles 0, s, 2s, ... (sampled keys, whose
                         // logits go to consecutive output columns)
    int32_t cap;         // list sinks: entries per sub-list
    int64_t out_offset;  // logits: element offset of (row_begin, j_begin) in the output;
                         // streams: entry offset of row_begin's list for this split
    int64_t out_ld;      // logits: elements between rows; streams: entries between rows
    int64_t cnt_offset;  // streams: counts index of row_begin for this split
    int64_t cnt_ld;      // streams: counts between rows
};

struct LogitsParams {
    CUtensorMap tmap_q;  // [rows*H, D] bytes, box [256 rows, D]; e2m1 queries: [rows*H, D/2]
                         // packed, 64-byte swizzled
    CUtensorMap tmap_k;  // [keys, D] bytes, box [128 rows, D]; e2m1 keys: [keys, D/2]
                         // packed, unpacked by the map into 16-byte groups of 16 codes
    const float* s_q;    // [rows, H]; nullptr for e2m1 queries
    const float* w;      // [rows, H]
    const float* s_k;    // fp8 keys: [keys]
    const int32_t* compress_len;  // [rows]
    const uint8_t* cand_mask;     // nullable [rows, ld_mask] 0/1 per key block
    int64_t ld_mask;
    const int32_t* mask_rows;     // nullable [rows]: row t reads mask row mask_rows[t]
    int64_t mask_row_count;       // rows of cand_mask when mask_rows is set
    int32_t mask_block;
    int32_t num_segments;
    int32_t total_units;
    int32_t pad0_;
    long long timeout_cycles;
    float* out;
    uint32_t* status;
    // streamed top-k
    uint2* lists;         // (score bits, key or block index) entries
    uint32_t* counts;     // entries appended per (row, split), clamped to cap
    uint32_t* gtau;       // [rows] shared lower bound (ord of a score) per row
    int32_t keep;         // k (keys) or cand_topk (blocks)
    int32_t pool;         // keys per block for kSinkPool
    int32_t update_tiles; // tiles between threshold refreshes
    const uint32_t* tau_row;   // kSinkFilter: [rows] fixed threshold (ord of a score)
    const uint32_t* row_fail;  // nullable [rows]: only row groups with a set row run
    const uint32_t* fail_any;  // nullable: the whole launch has no work while it reads 0
    Segment seg[kMaxSegments];
    const uint32_t* k_sf; // e2m1 keys scored natively: [keys] four ue8m0 block scales
                          // (byte b: elements 32b..32b+31); nullptr for e4m3 keys
    const uint32_t* q_sf; // e2m1 queries (with e2m1 keys): [rows * H] four ue8m0 block
                          // scales per query vector; nullptr for e4m3 queries
};

// Host-side launchers (defined in the .cu files).
cudaError_t launch_logits(const LogitsParams& p, int H, int D, int sink, int grid,
                          cudaStream_t stream);
int logits_rows_per_group(int H, bool fp4_keys);   // query rows per MMA tile
bool logits_fp4_native(int H, int D);   // e2m1 keys scored by the block-scaled MMA

// Exact selection over the lists appended by the streaming sinks.  A piece is
// a row range of one request whose lists were filled by the same launch; one
// CTA per row.
struct MergePiece {
    int32_t row_begin;      // first global row
    int32_t nrows;
    int32_t cta_begin;      // first CTA of the piece in the launch
    int32_t slots;          // key splits (lists) per row
    int32_t cap;            // entries per list
    int32_t key_count;      // keys (or blocks) of the piece's request: indices are below it
    int64_t mask_delta;     // mask output: row t of the piece writes mask row t + mask_delta
    int64_t list_offset;    // entry offset of row_begin's first list
    int64_t count_offset;   // counts index of row_begin's first list
};
struct StreamMergeParams {
    const uint2* lists;
    const uint32_t* counts;
    const uint32_t* gtau;   // per-row lower bound on the k-th key: entries below it are skipped
    uint32_t* row_fail;     // [rows] verify: set for rows the lists cannot decide;
                            // only_failed: rows with a clear entry are skipped
    const uint32_t* tau_row;  // verify: the threshold the lists were filled with
    const uint32_t* smax_row; // nullable, verify: the largest sample of each row (ord)
    uint32_t* fail_any;       // verify: set when any row is flagged; only_failed: 0 = no work
    int32_t verify;
    int32_t only_failed;
    int32_t k;
    int32_t num_pieces;
    int32_t total_ctas;
    int32_t bitmap;            // 1: index-order output by bitmap where a row's keys allow
    int32_t* out_idx;
    float* out_val;
    uint8_t* mask;             // blocks: [rows, ld_mask]
    int64_t ld_mask;
    MergePiece piece[kMaxMergePieces];
};
cudaError_t launch_stream_merge(const StreamMergeParams& p, cudaStream_t stream);

// Standalone top-k over user logits [rows, ld].
struct TopkParams {
    const float* logits;
    int64_t ld;
    const int32_t* compress_len;
    int32_t k;
    int32_t total_rows;
    int32_t num_requests;
    int32_t pad_;
    int32_t* out_idx;
    float* out_val;
    const uint32_t* row_fail;    // nullable: only rows with a set flag (none while fail_any is 0)
    const uint32_t* fail_any;
    int32_t req_row_begin[kMaxRequests + 1];
    int32_t req_key_count[kMaxRequests];
};
cudaError_t launch_topk_dense(const TopkParams& p, cudaStream_t stream);

// Sampled path of the top-k over caller logits, one pass of rows [row0, row0 + rows):
// gather every tile_stride-th 128-key tile of each row into samples [rows, sample_cols]
// (keys past the row's length read as -inf), then (after the threshold kernel) append
// every entry at or above the row's threshold to its list.
struct DensePiece {
    int32_t row_begin;      // first global row
    int32_t nrows;
    int32_t request;
    int32_t slots;          // lists per row: key chunk c of the row appends to list c
    int32_t chunk;          // keys per chunk
    int32_t cap;            // entries per list
    int64_t list_offset;    // entry offset of row_begin's first list
    int64_t count_offset;   // counts index of row_begin's first list
};
struct DenseFilterParams {
    const float* logits;
    int64_t ld;
    const int32_t* compress_len;
    float* samples;              // gather: [rows of the pass, sample_cols]
    int32_t sample_cols;
    int32_t num_pieces;
    const uint32_t* tau_row;     // filter: [total rows]
    uint2* lists;
    uint32_t* counts;
    int32_t num_requests;
    int32_t pad_;
    int32_t req_stride[kMaxRequests];   // sampled tile stride (0: not sampled)
    int32_t req_key_count[kMaxRequests];
    DensePiece piece[kMaxMergePieces];
};
cudaError_t launch_dense_gather(const DenseFilterParams& p, int rows, cudaStream_t stream);
cudaError_t launch_dense_filter(const DenseFilterParams& p, int rows, int max_slots,
                                cudaStream_t stream);

// Per-row thresholds from sampled logits [rows, ld] (row t at t - row0): about
// the largest sample of rank mu + 5 sqrt(mu) + 4, mu = k * the row's sampled
// fraction, or 0 (everything passes) for rows of unsampled requests (stride 0),
// rows with at most k valid keys and rows with fewer samples.  With pool > 1 the
// ranked samples are the maxima of aligned pool-key blocks of the sampled keys
// and k counts blocks.
struct SampleParams {
    const float* samples;
    int64_t ld;
    int32_t row0;
    int32_t rows;
    int32_t k;
    int32_t num_requests;
    int32_t pool;                // keys per ranked entry (1: keys; 2, 4, 8: block maxima)
    int32_t pad_;
    const int32_t* compress_len;
    const float* logits;         // nullable: read the samples from caller logits [rows, ld]
                                 // (row t at t, sample e at key (e / 128) stride 128 + e % 128)
                                 // instead of `samples`
    int64_t ld_logits;
    uint32_t* tau_row;           // [total rows], written at row0 .. row0 + rows - 1
    uint32_t* smax_row;          // [total rows]: ord of the row's largest ranked sample where
                                 // tau is nonzero, else 0
    int32_t req_row_begin[kMaxRequests + 1];
    int32_t req_rank[kMaxRequests];    // sampling stride of the request, 0: not sampled
    int32_t req_key_count[kMaxRequests];
    int32_t req_cols[kMaxRequests];    // sample columns a row of the request fills (<= ld)
};
cudaError_t launch_sample_threshold(const SampleParams& p, cudaStream_t stream);

// Top-k over caller logits in one read per row (rows of at most 65,536 keys, k <= 2048):
// every entry at or above the row's sampled threshold is kept in shared memory and the
// exact selection runs there.  Rows it cannot decide (fewer than k entries at or above
// the threshold, more candidates than it holds) are flagged for the direct kernel.
struct RowTopkParams {
    const float* logits;         // [rows, ld], 16-byte aligned rows
    int64_t ld;
    const int32_t* compress_len;
    const uint32_t* tau_row;     // [rows] ord threshold, 0: every finite entry
    const uint32_t* smax_row;    // [rows] ord of the largest sample (bucket range)
    uint32_t* row_fail;
    uint32_t* fail_any;
    uint32_t* row_counter;       // zero at launch: rows are taken in order by the CTAs
    uint32_t* status;
    long long timeout_cycles;
    int32_t* out_idx;
    float* out_val;              // nullable
    int32_t k;
    int32_t total_rows;
    int32_t num_requests;
    int32_t pad_;
    int32_t req_row_begin[kMaxRequests + 1];
    int32_t req_key_count[kMaxRequests];
};
cudaError_t launch_row_topk(const RowTopkParams& p, cudaStream_t st);
int row_topk_max_keys();   // longest row (keys) the kernel takes

// Mask rows of rows with at most cand_topk candidate blocks: row t (of row0 .. row0 +
// rows - 1) writes mask row t + delta, 1 for its blocks below ceil(min(clen[t], keys) /
// block), 0 for the rest of the ld bytes.
cudaError_t launch_fill_mask_rows(uint8_t* mask, int64_t ld, const int32_t* clen, int row0,
                                  int rows, int keys, int block, int64_t delta, cudaStream_t st);
cudaError_t launch_expand_mask(const uint8_t* cand_mask, int64_t ld_mask, const int32_t* clen,
                               uint8_t* key_mask, int64_t ld, int block, int rows,
                               cudaStream_t st);
cudaError_t launch_selftest_timeout(uint32_t* status, long long cycles, cudaStream_t st);

// Page (KV slot) indices of selected raw key indices: out[t, i] =
// table[r, j / page] * page + j % page for 0 <= j < L_r (r the request of row t),
// else -1; -1 also where the table entry is negative or the slot does not fit int32.
struct PageIndexParams {
    const int32_t* raw;          // [rows, k]
    int32_t* out;                // [rows, k] (may be raw itself)
    const int32_t* table;        // [num_requests, ld_table]
    int64_t ld_table;
    int32_t page;
    int32_t k;
    int32_t rows;
    int32_t num_requests;
    int32_t req_row_begin[kMaxRequests + 1];
    int32_t req_key_count[kMaxRequests];
};
cudaError_t launch_page_indices(const PageIndexParams& p, cudaStream_t st);
// e2m1 keys [keys, D/2] (element 2i in the low nibble) with ue8m0 scales
// [keys, D/32] -> e4m3 keys [keys, D] and fp32 s_k [keys] = 2^(largest block
// exponent - 127), exactly; a key whose smaller blocks would need more than
// e4m3's range sets kStatusFp4Range in *status.
cudaError_t launch_fp4_to_fp8(const uint8_t* k4, const uint8_t* sf, int keys, int D, uint8_t* k8,
                              float* s_k, uint32_t* status, cudaStream_t st);
cudaError_t launch_pad_heads(const void* q, const float* s_q, const float* w, void* q_out,
                             float* s_q_out, float* w_out, int rows, int h_in, int h_out, int D,
                             cudaStream_t st);

}  // namespace idx
