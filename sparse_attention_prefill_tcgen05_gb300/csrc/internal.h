// Internal interfaces between the host library and the kernels.  Nothing in
// here crosses the C ABI.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace idx {

constexpr int kTileKeys = 128;   // MMA M: keys per tile (one TMEM lane each)
constexpr int kTileN = 256;      // MMA N: (row, head) columns per tile
constexpr int kMaxSegments = 48;
constexpr int kMaxRequests = 256;
constexpr int kEpiWarps = 8;
constexpr int kThreads = 384;    // warp 0 TMA, warp 1 MMA/TMEM, 2-3 spare, 4-11 epilogue

// Device status word bits (OR-ed by kernels, read by indexer_status).
constexpr uint32_t kStatusTimeout = 1u << 0;
constexpr uint32_t kStatusBadArg = 1u << 1;

// Key formats.
constexpr int kKeyFp8 = 0;
constexpr int kKeyFp4 = 1;

// What the logits kernel does with each (row, key) score.
constexpr int kSinkLogits = 0;   // write fp32 to a [rows, ld] buffer

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
    int32_t pad_;
    int64_t out_offset;  // element offset of (row_begin, j_begin) in the output
    int64_t out_ld;      // elements between consecutive rows of the output
};

struct LogitsParams {
    CUtensorMap tmap_q;  // [rows*H, D] bytes, box [256 rows, D]
    CUtensorMap tmap_k;  // [keys, D or D/2] bytes, box [128 rows, ...]
    const float* s_q;    // [rows, H]
    const float* w;      // [rows, H]
    const float* s_k;    // fp8 keys: [keys]
    const uint8_t* k_sf; // fp4 keys: ue8m0 [keys, D/32]
    const int32_t* compress_len;  // [rows]
    const uint8_t* cand_mask;     // nullable [rows, ld_mask] 0/1 per key block
    int64_t ld_mask;
    int32_t mask_block;
    int32_t num_segments;
    int32_t total_units;
    int32_t chunk_tiles;  // key tiles per unit
    long long timeout_cycles;
    float* out;
    uint32_t* status;
    Segment seg[kMaxSegments];
};

// One (row range, key split) piece of the selection kernels.
struct SelSegment {
    int32_t row_begin;    // first global row
    int32_t nrows;
    int32_t j_begin;      // request-local key (or block) index of entry 0
    int32_t n_entries;    // entries in this piece (keys, or blocks when pooling)
    int32_t key_count;    // keys of the request (clamps compress_len)
    int32_t cand_slot;    // split index within the row's candidate slots
    int32_t n_slots;      // candidate slots per row of this request
    int32_t pad_;
    int64_t src_offset;   // element offset of (row_begin, entry 0) in the dense source
    int64_t src_ld;
    int64_t cand_offset;  // entry offset of the request's first row in the candidate area
    int32_t row_block;    // first CTA (= row) of this piece in the launch
    int32_t pad2_;
};

struct SelParams {
    const float* src;            // dense scores
    const int32_t* compress_len;
    int32_t k;                   // entries kept per row
    int32_t pool;                // 0: entries are keys; >0: entries are blocks of `pool` keys
    int32_t num_segments;
    int32_t total_rows_launch;
    float* cand_val;             // [.., k] per slot
    int32_t* cand_idx;
    SelSegment seg[kMaxSegments];
};

// Host-side launchers (defined in the .cu files).
cudaError_t launch_logits(const LogitsParams& p, int H, int D, int kfmt, int grid,
                          cudaStream_t stream);
size_t logits_smem_bytes(int H, int D, int kfmt);
int logits_rows_per_group(int H, int kfmt);   // query rows per MMA tile

// Per-row top-k of dense rows into candidate slots (rows = total of segs).
cudaError_t launch_select_dense(const SelParams& p, cudaStream_t stream);

// Final merge: per row, exact top-k of its n_slots*k candidates into out_idx/out_val,
// or (blocks) into a 0/1 mask.
struct MergeParams {
    const float* cand_val;
    const int32_t* cand_idx;
    int32_t k;                 // kept per row
    int32_t num_requests;
    int32_t total_rows;
    int32_t pad_;
    int32_t* out_idx;          // [rows, k] or null
    float* out_val;            // [rows, k] or null
    uint8_t* mask;             // [rows, ld_mask] or null (block selection)
    int64_t ld_mask;
    int32_t req_row_begin[kMaxRequests + 1];
    int32_t req_slots[kMaxRequests];
    int64_t req_cand_offset[kMaxRequests];
};
cudaError_t launch_merge(const MergeParams& p, cudaStream_t stream);

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
    int32_t req_row_begin[kMaxRequests + 1];
    int32_t req_key_count[kMaxRequests];
};
cudaError_t launch_topk_dense(const TopkParams& p, cudaStream_t stream);

cudaError_t launch_expand_mask(const uint8_t* cand_mask, int64_t ld_mask, const int32_t* clen,
                               uint8_t* key_mask, int64_t ld, int block, int rows,
                               cudaStream_t st);
cudaError_t launch_selftest_timeout(uint32_t* status, long long cycles, cudaStream_t st);

}  // namespace idx
