// Host side of the C ABI: problem validation, the per-batch plan, workspace
// layout, TMA descriptors and kernel launches.  No device memory is ever
// allocated here; every call is asynchronous on the caller's stream.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstring>
#include <mutex>
#include <new>
#include <vector>

#include "indexer.h"
#include "internal.h"
#include "ptx.cuh"

using namespace idx;

namespace {

// Rows [a, b) of request r whose lists live at list_off (entries) during one pass.
struct PassPiece {
    int r, a, b;
    int64_t list_off;
};

// One pass of the streamed top-k: a logits launch that fills the pieces' lists
// and the merge launch that selects from them.  Passes reuse the list area.
struct Pass {
    std::vector<PassPiece> pieces;
};

constexpr int kUpdateTiles = 4;          // tiles between threshold refreshes
constexpr int kSampleTiles = 16;         // sampled key tiles per row (at least, once sampled)
constexpr int kSampleTilesMax = 128;     // ... and at most (16,384 sampled keys per row)
constexpr double kMinSampledMu = 8.0;    // expected samples among a row's top keep, at least

// Sampling stride of a request of `tiles` key tiles whose rows keep `keep` entries: every
// st-th tile, at least kSampleTiles of them, and enough that a row's top `keep` keys hold
// kMinSampledMu samples on average (a small expected count makes the rank of the sampled
// threshold small and the number of keys above it spread widely); 0 = not sampled (short
// requests keep every entry).
int sample_stride_for(int tiles, int keep)
{
    if (tiles < 2 * kSampleTiles)
        return 0;
    const int want = (int)std::ceil(kMinSampledMu * tiles / std::max(keep, 1));
    const int n = std::min(kSampleTilesMax, std::max(kSampleTiles, want));
    return (int)((tiles + n - 1) / n);
}

// Upper-tail factor of the number of keys above a row's sampled threshold, relative to its
// mean keep * rank / mu: that number is about the mean times Gamma(rank) / rank, and
// 1 + 5 / sqrt(rank) + 10 / rank is above its 1 - 1e-7 quantile for the ranks used here
// (3.05 at rank 14, 1.57 at rank 108).
double rank_tail_factor(double rank) { return 1.0 + 5.0 / std::sqrt(rank) + 10.0 / rank; }
constexpr int kSampleUnitTiles = 4;      // sampled tiles per work unit of the sampled pass
constexpr int64_t kPlanSms = 152;        // SMs the planner balances for (GB300)
constexpr int64_t kUnitsPerSm = 6;       // work units per SM wanted for load balance

}  // namespace

struct indexer_plan_s {
    int R = 0, T = 0, Lk = 0, H = 0, D = 0, topk = 0, kdtype = 0;
    int kH = 0;                       // heads the kernels run with (H, or H padded with zero heads)
    size_t off_pad = 0;               // padded q / s_q / w when kH != H
    bool fp4_native = false;          // e2m1 keys scored by the block-scaled MMA
    bool fp4_queries = false;         // e2m1 queries as well (the fp4 MMA kind)
    size_t off_k8 = 0;                // e4m3 keys [Lk, D] + s_k [Lk] converted from e2m1
                                      // (shapes without a block-scaled kernel)
    size_t pad_end = 0;               // end of the per-call input preparation area
    int cand_block = 8, cand_topk = 0;
    int G = 8;                        // query rows per MMA tile
    std::vector<int32_t> row_begin;   // [R+1]
    std::vector<int32_t> key_begin;   // [R+1]
    std::vector<int32_t> L;           // [R]
    std::vector<int32_t> clen;        // [T]
    int max_L = 0;
    uint64_t budget = 0;
    // streamed selection
    int split_keys = 0;               // largest key split of any request (for reporting)
    std::vector<int32_t> split_r;     // keys per split of each request (multiple of 128)
    std::vector<int32_t> n_splits;    // per request
    std::vector<int32_t> cap_k;       // sub-list capacity per (row, split, quadrant), keys
    std::vector<int32_t> cap_b;       // sub-list capacity per (row, split, quadrant), blocks
    std::vector<int64_t> cnt_base;    // counts index of the request's first row
    std::vector<Pass> passes_k, passes_b;
    int max_piece_rows = 0;
    // workspace layout (bytes)
    // sampled thresholds (top-k): per request every stride_r-th key tile, the
    // threshold at the rank_r-th largest sample (rank 0: the request is not
    // sampled and its rows keep everything); sample_cols columns per row;
    // sample_stride = the largest stride, 0 = no request is sampled
    int sample_stride = 0, sample_cols = 0;
    // the candidate-block path samples too (its pass list areas hold the samples)
    bool sample_blocks = false;
    std::vector<int32_t> sample_stride_r, sample_rank_r;
    size_t off_gtau = 0, off_fail = 0, off_tau = 0, off_counts = 0, off_lists = 0, ws_bytes = 0;
    long long wait_budget = 4000000000LL;
};

namespace {

std::atomic<long long> g_launches{0};  // kernels launched by this library (diagnostic)
// events recorded around the main logits launch of the next top-k calls (diagnostic)
std::atomic<void*> g_prof_start{nullptr}, g_prof_stop{nullptr};

constexpr size_t kStatusBytes = 256;
constexpr uint64_t kDefaultBudget = 2ull << 30;

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

bool supported_shape(int H, int D, int kdtype)
{
    // e2m1 keys are converted to e4m3 exactly (misc.cu) and scored like fp8 keys
    (void)kdtype;
    return (H == 32 && D == 128) || (H == 16 && D == 128) || (H == 64 && D == 128) ||
           (H == 8 && D == 64) || (H == 4 && D == 64);
}

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Group the rows of every request into passes whose lists fit `entries`.
// Returns false if even one row of some request does not fit.
bool build_passes(const indexer_plan_s& p, const std::vector<int32_t>& cap, int64_t entries,
                  std::vector<Pass>& passes, int& max_rows)
{
    passes.clear();
    Pass cur;
    int64_t used = 0;
    int segs = 0;
    for (int r = 0; r < p.R; ++r) {
        const int rb = p.row_begin[r], re = p.row_begin[r + 1];
        if (re == rb)
            continue;
        const int64_t per_row = (int64_t)p.n_splits[r] * kListsPerSplit * cap[r];
        int64_t fit = entries / per_row;
        if (fit < 1)
            return false;
        if (fit >= p.G)
            fit = fit / p.G * p.G;
        for (int a = rb; a < re;) {
            const int b = (int)std::min<int64_t>(re, a + fit);
            const int64_t need = (int64_t)(b - a) * per_row;
            if (!cur.pieces.empty() &&
                (used + need > entries || segs + p.n_splits[r] > kMaxSegments ||
                 (int)cur.pieces.size() == kMaxMergePieces)) {
                passes.push_back(cur);
                cur.pieces.clear();
                used = 0;
                segs = 0;
            }
            cur.pieces.push_back(PassPiece{r, a, b, used});
            used += need;
            segs += p.n_splits[r];
            max_rows = std::max(max_rows, b - a);
            a = b;
        }
    }
    if (!cur.pieces.empty())
        passes.push_back(cur);
    return true;
}

int64_t pass_entries(const indexer_plan_s& p, const std::vector<Pass>& passes,
                     const std::vector<int32_t>& cap)
{
    int64_t m = 0;
    for (const Pass& ps : passes) {
        int64_t u = 0;
        for (const PassPiece& pc : ps.pieces)
            u += (int64_t)(pc.b - pc.a) * p.n_splits[pc.r] * kListsPerSplit * cap[pc.r];
        m = std::max(m, u);
    }
    return m;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn()
{
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(f);
    });
    return fn;
}

// 2-D map over a row-major byte matrix [rows, row_bytes] with a box of
// [box_rows, row_bytes], swizzled to the row width for the MMA.
bool make_map(CUtensorMap* m, const void* base, uint64_t rows, uint32_t row_bytes,
              uint32_t box_rows)
{
    EncodeTiledFn enc = encode_fn();
    if (!enc)
        return false;
    const cuuint64_t dims[2] = {row_bytes, rows};
    const cuuint64_t strides[1] = {row_bytes};
    const cuuint32_t box[2] = {row_bytes, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    const CUtensorMapSwizzle sw = row_bytes == 128  ? CU_TENSOR_MAP_SWIZZLE_128B
                                  : row_bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                                    : CU_TENSOR_MAP_SWIZZLE_32B;
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D map over packed e2m1 keys [rows, D/2 bytes] that unpacks each group of 16 codes
// into a 16-byte shared-memory slot (8 data bytes, 8 bytes of padding): the 8-bit
// container layout the f8f6f4 MMA kinds read 4-bit operands in.  A box of D = 128 codes
// x box_rows lands as box_rows rows of 128 bytes, 128-byte swizzled like the e4m3 tiles.
bool make_map_fp4(CUtensorMap* m, const void* base, uint64_t rows, uint32_t D,
                  uint32_t box_rows)
{
    EncodeTiledFn enc = encode_fn();
    if (!enc)
        return false;
    const cuuint64_t dims[2] = {D, rows};
    const cuuint64_t strides[1] = {D / 2};
    const cuuint32_t box[2] = {D, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 2, const_cast<void*>(base), dims, strides,
               box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
}

struct DeviceInfo {
    int sms = 0;
    bool ok = false;
};

DeviceInfo device_info()
{
    DeviceInfo d;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return d;
    int maj = 0, min = 0;
    cudaDeviceGetAttribute(&maj, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&min, cudaDevAttrComputeCapabilityMinor, dev);
    cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
    d.ok = (maj == 10 && min == 3);
    return d;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int check_common(const indexer_plan_s* p, void* ws, size_t ws_bytes)
{
    if (!p)
        return IDX_ERR_INVALID_ARG;
    if (!ws || !aligned(ws, 256))
        return IDX_ERR_INVALID_ARG;
    if (ws_bytes < p->ws_bytes)
        return IDX_ERR_WORKSPACE;
    return IDX_OK;
}

int check_inputs(const indexer_plan_s* p, const void* q, const float* s_q, const float* w,
                 const void* k, const void* k_scale, const int32_t* clen)
{
    if (!q || !s_q || !w || !k || !k_scale || !clen)
        return IDX_ERR_INVALID_ARG;
    // e2m1 keys scored natively read their block scales as one 32-bit word per key, and
    // e2m1 queries theirs (passed as s_q) as one word per query vector
    if (!aligned(q, 16) || !aligned(k, p->kdtype == IDX_K_FP8_E4M3 ? 16 : 32) ||
        !aligned(s_q, 4) || !aligned(w, 4) || !aligned(clen, 4) ||
        ((p->kdtype == IDX_K_FP8_E4M3 || p->fp4_native) && !aligned(k_scale, 4)))
        return IDX_ERR_INVALID_ARG;
    return IDX_OK;
}

struct Ctx {
    const indexer_plan_s* p;
    LogitsParams lp;
    int sms;
    cudaStream_t st;
    // candidate blocks for each request's last tail[r] rows only (nullptr: every row),
    // written to mask row t + mask_delta[r] (empty: row t)
    const int32_t* tail = nullptr;
    std::vector<int64_t> mask_delta;
};

int fill_maps(Ctx& c, const void* q, const void* k)
{
    const indexer_plan_s* p = c.p;
    std::memset(&c.lp, 0, sizeof(c.lp));
    if (!make_map(&c.lp.tmap_q, q, (uint64_t)p->T * p->kH, p->fp4_queries ? p->D / 2 : p->D,
                  p->G * p->kH))
        return IDX_ERR_CUDA;
    const uint64_t krows = (uint64_t)std::max(p->Lk, 1);
    // e2m1 keys: unpacked to the 8-bit container layout for the mxf8f6f4 kind, kept packed
    // (64-byte rows) for the fp4 kind that e2m1 queries take
    const bool unpack = p->fp4_native && !p->fp4_queries;
    if (!(unpack ? make_map_fp4(&c.lp.tmap_k, k, krows, p->D, kTileKeys)
                 : make_map(&c.lp.tmap_k, k, krows, p->fp4_queries ? p->D / 2 : p->D,
                            kTileKeys)))
        return IDX_ERR_CUDA;
    return IDX_OK;
}

// Launch the logits kernel over a list of segments (<= kMaxSegments) whose
// n_row_groups / n_chunks / unit_tiles are set; unit numbering is filled here.
int run_logits(Ctx& c, std::vector<Segment>& segs, int sink)
{
    const indexer_plan_s* p = c.p;
    LogitsParams& lp = c.lp;
    lp.num_segments = (int)segs.size();
    int units = 0;
    for (size_t i = 0; i < segs.size(); ++i) {
        segs[i].unit_begin = units;
        units += segs[i].n_row_groups * segs[i].n_chunks;
        lp.seg[i] = segs[i];
    }
    lp.total_units = units;
    lp.timeout_cycles = p->wait_budget;
    if (units == 0)
        return IDX_OK;
    const int grid = std::min(units, c.sms);
    g_launches.fetch_add(1, std::memory_order_relaxed);
    return launch_logits(lp, p->kH, p->D, sink, grid, c.st) == cudaSuccess
               ? IDX_OK
               : IDX_ERR_CUDA;
}

// Segments and merge pieces of one pass for a list-filling sink: every piece
// against every key split of its request.
int pass_launches(Ctx& c, const Pass& ps, const std::vector<int32_t>& cap, int sink,
                  StreamMergeParams& mp)
{
    const indexer_plan_s* p = c.p;
    LogitsParams& lp = c.lp;
    std::memset(&mp, 0, sizeof(mp));
    std::vector<Segment> segs;
    int ctas = 0;
    auto flush = [&]() -> int {
        if (segs.empty())
            return IDX_OK;
        int rc = run_logits(c, segs, sink);
        segs.clear();
        return rc;
    };
    for (const PassPiece& pc : ps.pieces) {
        const int r = pc.r;
        const int ns = p->n_splits[r];
        if ((int)segs.size() + ns > kMaxSegments) {
            int rc = flush();
            if (rc != IDX_OK)
                return rc;
        }
        for (int s = 0; s < ns; ++s) {
            Segment sg;
            std::memset(&sg, 0, sizeof(sg));
            sg.row_begin = pc.a;
            sg.nrows = pc.b - pc.a;
            sg.key_base = p->key_begin[r];
            sg.key_count = p->L[r];
            sg.j_begin = s * p->split_r[r];
            sg.j_end = std::min(p->L[r], (s + 1) * p->split_r[r]);
            sg.unit_tiles = (int)ceil_div(std::max(0, sg.j_end - sg.j_begin), kTileKeys);
            sg.tile_stride = 1;
            sg.cap = cap[r];
            sg.n_row_groups = (int)ceil_div(sg.nrows, p->G);
            sg.n_chunks = 1;
            // row-major [row][split][quadrant][cap]
            sg.out_offset = pc.list_off + (int64_t)s * kListsPerSplit * cap[r];
            sg.out_ld = (int64_t)ns * kListsPerSplit * cap[r];
            sg.cnt_offset = p->cnt_base[r] +
                            (int64_t)(pc.a - p->row_begin[r]) * ns * kListsPerSplit +
                            (int64_t)s * kListsPerSplit;
            sg.cnt_ld = ns * kListsPerSplit;
            segs.push_back(sg);
        }
        MergePiece& mpc = mp.piece[mp.num_pieces++];
        mpc.row_begin = pc.a;
        mpc.nrows = pc.b - pc.a;
        mpc.cta_begin = ctas;
        mpc.slots = ns * kListsPerSplit;
        mpc.cap = cap[r];
        mpc.key_count = p->L[r];
        mpc.mask_delta = c.mask_delta.empty() ? 0 : c.mask_delta[r];
        mpc.list_offset = pc.list_off;
        mpc.count_offset = p->cnt_base[r] + (int64_t)(pc.a - p->row_begin[r]) * ns * kListsPerSplit;
        ctas += pc.b - pc.a;
    }
    mp.total_ctas = ctas;
    mp.lists = lp.lists;
    mp.counts = lp.counts;
    return flush();
}

void record_prof(Ctx& c, std::atomic<void*>& ev)
{
    void* e = ev.load(std::memory_order_relaxed);
    if (e)
        cudaEventRecord(static_cast<cudaEvent_t>(e), c.st);
}

int launch_merge(Ctx& c, StreamMergeParams& mp)
{
    g_launches.fetch_add(1, std::memory_order_relaxed);
    return launch_stream_merge(mp, c.st) == cudaSuccess ? IDX_OK : IDX_ERR_CUDA;
}

// Each row's threshold for its top `keep` keys (pool = 1) or pool-key blocks, from
// the pass's samples [rows, sample_cols] (row t at t - the pass's first row).
int row_thresholds(Ctx& c, const Pass& ps, float* samples, uint32_t* tau_row, int pool,
                   int keep)
{
    const indexer_plan_s* p = c.p;
    const int first = ps.pieces.front().a;
    SampleParams sp;
    std::memset(&sp, 0, sizeof(sp));
    sp.samples = samples;
    sp.ld = p->sample_cols;
    sp.k = keep;
    sp.pool = pool > 1 ? pool : 1;
    sp.compress_len = c.lp.compress_len;
    sp.tau_row = tau_row;
    sp.smax_row = tau_row + p->T;
    sp.num_requests = p->R;
    for (int r = 0; r < p->R; ++r) {
        sp.req_row_begin[r] = p->row_begin[r];
        sp.req_rank[r] = p->sample_rank_r[r] > 0 ? p->sample_stride_r[r] : 0;
        sp.req_key_count[r] = p->L[r];
        // the sampled pass writes ceil(tiles / stride) tiles of 128 columns per row
        sp.req_cols[r] = p->sample_rank_r[r] > 0
                             ? (int)ceil_div(ceil_div(std::max(1, p->L[r]), kTileKeys),
                                             p->sample_stride_r[r]) * kTileKeys
                             : 0;
    }
    sp.req_row_begin[p->R] = p->row_begin[p->R];
    // one launch per run of adjacent pieces (a pass restricted to some rows of its
    // requests has gaps, whose sample rows are never written)
    for (size_t i = 0; i < ps.pieces.size();) {
        size_t e = i + 1;
        while (e < ps.pieces.size() && ps.pieces[e].a == ps.pieces[e - 1].b)
            ++e;
        sp.row0 = ps.pieces[i].a;
        sp.rows = ps.pieces[e - 1].b - ps.pieces[i].a;
        sp.samples = samples + (int64_t)(ps.pieces[i].a - first) * p->sample_cols;
        g_launches.fetch_add(1, std::memory_order_relaxed);
        if (launch_sample_threshold(sp, c.st) != cudaSuccess)
            return IDX_ERR_CUDA;
        i = e;
    }
    return IDX_OK;
}

// Sampled logits of the pass's rows (every sample_stride-th key tile of each
// request) into `samples` [rows, sample_cols], then each row's threshold for its
// top `keep` keys (pool = 1) or its top `keep` pool-key blocks.
int pass_thresholds(Ctx& c, const Pass& ps, float* samples, uint32_t* tau_row, int pool,
                    int keep)
{
    const indexer_plan_s* p = c.p;
    LogitsParams& lp = c.lp;
    const int first = ps.pieces.front().a;
    std::vector<Segment> segs;
    for (const PassPiece& pc : ps.pieces) {
        const int r = pc.r;
        Segment sg;
        std::memset(&sg, 0, sizeof(sg));
        sg.row_begin = pc.a;
        sg.nrows = pc.b - pc.a;
        sg.key_base = p->key_begin[r];
        sg.key_count = p->L[r];
        sg.j_begin = 0;
        sg.j_end = p->L[r];
        if (p->sample_rank_r[r] == 0)
            continue;                          // its rows keep every entry (threshold 0)
        sg.tile_stride = p->sample_stride_r[r];
        // the sampled tiles of a row group in units of a few tiles, so that the pass's
        // few units per SM spread evenly over the SMs
        const int sampled =
            (int)ceil_div(ceil_div(std::max(1, p->L[r]), kTileKeys), p->sample_stride_r[r]);
        sg.unit_tiles = std::min(sampled, kSampleUnitTiles);
        sg.n_row_groups = (int)ceil_div(sg.nrows, p->G);
        sg.n_chunks = (int)ceil_div(sampled, sg.unit_tiles);
        sg.out_offset = (int64_t)(pc.a - first) * p->sample_cols;
        sg.out_ld = p->sample_cols;
        segs.push_back(sg);
        if ((int)segs.size() == kMaxSegments) {
            lp.out = samples;
            int rc = run_logits(c, segs, kSinkLogits);
            if (rc != IDX_OK)
                return rc;
            segs.clear();
        }
    }
    if (!segs.empty()) {
        lp.out = samples;
        int rc = run_logits(c, segs, kSinkLogits);
        if (rc != IDX_OK)
            return rc;
    }
    return row_thresholds(c, ps, samples, tau_row, pool, keep);
}

// Streamed top-k (pool = 0) or candidate blocks (pool > 0), pass by pass.
//   exact:   the logits kernel appends entries that pass each row's running
//            threshold (histograms, compaction, shared bound), then the merge
//            selects exactly from the lists;
//   sampled: (top-k, when the plan samples) a threshold per row from sampled
//            logits, lists of every entry at or above it, a merge that
//            decides the rows whose lists hold at least k entries and did not
//            overflow, and the exact path for the rows it could not decide.
int run_streamed(Ctx& c, uint8_t* ws, int pool, int32_t* out_idx, float* out_val,
                 uint8_t* mask, int64_t ld_mask)
{
    const indexer_plan_s* p = c.p;
    const std::vector<int32_t>& cap = pool ? p->cap_b : p->cap_k;
    // the plan's passes, or their pieces cut down to each request's last tail[r] rows
    // (a piece keeps its list area: its first kept row's lists start per_row entries
    // further per skipped row)
    // candidate blocks: a request whose rows have at most cand_topk blocks keeps every
    // valid block of every row, whatever its logits; its mask rows are written directly
    // and its rows are left out of the passes
    std::vector<char> whole(p->R, 0);
    bool any_whole = false;
    if (pool) {
        for (int r = 0; r < p->R; ++r) {
            whole[r] = ceil_div(std::max(p->L[r], 0), p->cand_block) <= p->cand_topk;
            any_whole = any_whole || whole[r];
            if (!whole[r])
                continue;
            const int b = p->row_begin[r + 1];
            const int a = c.tail ? b - c.tail[r] : p->row_begin[r];
            g_launches.fetch_add(1, std::memory_order_relaxed);
            if (launch_fill_mask_rows(mask, ld_mask, c.lp.compress_len, a, b - a, p->L[r],
                                      p->cand_block, c.mask_delta.empty() ? 0 : c.mask_delta[r],
                                      c.st) != cudaSuccess)
                return IDX_ERR_CUDA;
        }
    }
    std::vector<Pass> cut;
    if (c.tail || any_whole) {
        for (const Pass& ps : pool ? p->passes_b : p->passes_k) {
            Pass f;
            for (const PassPiece& pc : ps.pieces) {
                if (whole[pc.r])
                    continue;
                const int lo = c.tail ? std::max(pc.a, p->row_begin[pc.r + 1] - c.tail[pc.r])
                                      : pc.a;
                if (lo >= pc.b)
                    continue;
                const int64_t per_row = (int64_t)p->n_splits[pc.r] * kListsPerSplit * cap[pc.r];
                f.pieces.push_back(PassPiece{pc.r, lo, pc.b, pc.list_off + (lo - pc.a) * per_row});
            }
            if (!f.pieces.empty())
                cut.push_back(f);
        }
    }
    const std::vector<Pass>& passes =
        c.tail || any_whole ? cut : (pool ? p->passes_b : p->passes_k);
    const int keep = pool ? p->cand_topk : p->topk;
    const bool sampled = pool == 0 ? p->sample_stride > 0 : p->sample_blocks;
    LogitsParams& lp = c.lp;
    lp.lists = reinterpret_cast<uint2*>(ws + p->off_lists);
    lp.counts = reinterpret_cast<uint32_t*>(ws + p->off_counts);
    lp.gtau = reinterpret_cast<uint32_t*>(ws + p->off_gtau);
    uint32_t* row_fail = reinterpret_cast<uint32_t*>(ws + p->off_fail);
    uint32_t* tau_row = reinterpret_cast<uint32_t*>(ws + p->off_tau);
    // second word of the per-call status area (zeroed at the start of every call)
    uint32_t* fail_any = reinterpret_cast<uint32_t*>(ws) + 1;
    lp.keep = keep;
    lp.pool = pool ? pool : 1;
    lp.update_tiles = kUpdateTiles;
    auto finish = [&](StreamMergeParams& mp) {
        mp.k = keep;
        mp.out_idx = out_idx;
        mp.out_val = out_val;
        mp.mask = mask;
        mp.ld_mask = ld_mask;
        mp.bitmap = pool ? 0 : 1;
    };
    for (const Pass& ps : passes) {
        StreamMergeParams mp;
        int rc;
        if (sampled) {
            if ((rc = pass_thresholds(c, ps, reinterpret_cast<float*>(lp.lists), tau_row, pool,
                                      keep)) != IDX_OK)
                return rc;
            lp.tau_row = tau_row;
            lp.row_fail = nullptr;
            const bool prof = &ps == &passes.front();
            if (prof) record_prof(c, g_prof_start);
            if ((rc = pass_launches(c, ps, cap, pool ? kSinkPoolFilter : kSinkFilter, mp)) !=
                IDX_OK)
                return rc;
            if (prof) record_prof(c, g_prof_stop);
            finish(mp);
            mp.gtau = nullptr;
            mp.verify = 1;
            mp.tau_row = tau_row;
            mp.smax_row = tau_row + p->T;
            mp.row_fail = row_fail;
            mp.fail_any = fail_any;
            if ((rc = launch_merge(c, mp)) != IDX_OK)
                return rc;
            // the exact path, for the undecided rows only (no work at all when the
            // merge flagged none)
            lp.row_fail = row_fail;
            lp.fail_any = fail_any;
        } else {
            lp.row_fail = nullptr;
            lp.fail_any = nullptr;
        }
        const bool prof = !sampled && &ps == &passes.front();
        if (prof) record_prof(c, g_prof_start);
        if ((rc = pass_launches(c, ps, cap, pool ? kSinkPool : kSinkStream, mp)) != IDX_OK)
            return rc;
        if (prof) record_prof(c, g_prof_stop);
        finish(mp);
        mp.gtau = lp.gtau;
        mp.verify = 0;
        mp.only_failed = sampled ? 1 : 0;
        mp.row_fail = row_fail;
        mp.fail_any = fail_any;
        if ((rc = launch_merge(c, mp)) != IDX_OK)
            return rc;
    }
    lp.row_fail = nullptr;
    lp.fail_any = nullptr;
    return IDX_OK;
}

int begin_call(Ctx& c, const indexer_plan_s* p, void* ws, void* stream)
{
    DeviceInfo d = device_info();
    if (!d.ok)
        return IDX_ERR_UNSUPPORTED;
    c.p = p;
    c.sms = d.sms;
    c.st = reinterpret_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(ws, 0, kStatusBytes, c.st) != cudaSuccess)
        return IDX_ERR_CUDA;
    return IDX_OK;
}

void set_inputs(Ctx& c, const float* s_q, const float* w, const void* k_scale,
                const int32_t* clen, void* ws)
{
    // e2m1 queries: s_q carries their ue8m0 block scales, four bytes per query vector
    c.lp.s_q = c.p->fp4_queries ? nullptr : s_q;
    c.lp.q_sf = c.p->fp4_queries ? reinterpret_cast<const uint32_t*>(s_q) : nullptr;
    c.lp.w = w;
    // e2m1 keys scored natively keep their block scales (the MMA applies them); others
    // arrive here as e4m3 keys with s_k (converted from e2m1 where they were e2m1)
    if (c.p->fp4_native) {
        c.lp.k_sf = static_cast<const uint32_t*>(k_scale);
        c.lp.s_k = nullptr;
    } else {
        c.lp.k_sf = nullptr;
        c.lp.s_k = static_cast<const float*>(k_scale);
    }
    c.lp.compress_len = clen;
    c.lp.status = static_cast<uint32_t*>(ws);
    c.lp.mask_block = c.p->cand_block;
}

// Tensor maps and input pointers of a call; pads the heads first when the
// kernels run with more heads than the problem has.
int prepare(Ctx& c, const void* q, const float* s_q, const float* w, const void* k,
            const void* k_scale, const int32_t* clen, void* ws)
{
    const indexer_plan_s* p = c.p;
    if (p->kH != p->H) {
        uint8_t* base = static_cast<uint8_t*>(ws) + p->off_pad;
        void* q_pad = base;
        float* s_q_pad = reinterpret_cast<float*>(base + (size_t)p->T * p->kH * p->D);
        float* w_pad = s_q_pad + (size_t)p->T * p->kH;
        g_launches.fetch_add(1, std::memory_order_relaxed);
        if (launch_pad_heads(q, s_q, w, q_pad, s_q_pad, w_pad, p->T, p->H, p->kH, p->D, c.st) !=
            cudaSuccess)
            return IDX_ERR_CUDA;
        q = q_pad;
        s_q = s_q_pad;
        w = w_pad;
    }
    if (p->kdtype == IDX_K_FP4_E2M1_UE8M0 && !p->fp4_native) {
        uint8_t* k8 = static_cast<uint8_t*>(ws) + p->off_k8;
        float* s_k = reinterpret_cast<float*>(k8 + (size_t)std::max(p->Lk, 1) * p->D);
        g_launches.fetch_add(1, std::memory_order_relaxed);
        if (launch_fp4_to_fp8(static_cast<const uint8_t*>(k), static_cast<const uint8_t*>(k_scale),
                              p->Lk, p->D, k8, s_k, static_cast<uint32_t*>(ws), c.st) !=
            cudaSuccess)
            return IDX_ERR_CUDA;
        k = k8;
        k_scale = s_k;
    }
    int rc = fill_maps(c, q, k);
    if (rc != IDX_OK)
        return rc;
    set_inputs(c, s_q, w, k_scale, clen, ws);
    return IDX_OK;
}

}  // namespace

extern "C" {

int indexer_version(void) { return 2; }

int indexer_chunk_rows(int64_t prefix_len, double budget_token2, int32_t chunk_min,
                       int32_t chunk_max, int32_t page, int32_t pow2)
{
    if (!(budget_token2 > 0.0) || !std::isfinite(budget_token2) || chunk_min < 1 ||
        chunk_max < chunk_min || page < 1)
        return IDX_ERR_INVALID_ARG;
    if (prefix_len <= 0)
        return chunk_max;
    // budget / L, floored; anything at or above 2^40 rounds the same as 2^40
    const double x = std::floor(budget_token2 / static_cast<double>(prefix_len));
    const int64_t xi = x >= 1099511627776.0 ? (int64_t)1099511627776 : static_cast<int64_t>(x);
    int64_t c = 0;
    if (pow2) {
        if (xi >= 1)
            for (c = 1; c * 2 <= xi; c *= 2) {
            }
    } else {
        c = xi / page * page;
    }
    return static_cast<int>(std::min<int64_t>(chunk_max, std::max<int64_t>(chunk_min, c)));
}

long long indexer_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

void indexer_profile_main_kernel(void* start_event, void* stop_event)
{
    g_prof_start.store(start_event, std::memory_order_relaxed);
    g_prof_stop.store(stop_event, std::memory_order_relaxed);
}

const char* indexer_error_string(int s)
{
    switch (s) {
    case IDX_OK: return "ok";
    case IDX_ERR_INVALID_ARG: return "invalid argument";
    case IDX_ERR_UNSUPPORTED: return "unsupported shape, format or device";
    case IDX_ERR_WORKSPACE: return "workspace too small or budget impossible";
    case IDX_ERR_CUDA: return "CUDA call failed";
    case IDX_ERR_TIMEOUT: return "device wait timed out";
    case IDX_ERR_DEVICE_CHECK: return "device-side check failed";
    default: return "unknown status";
    }
}

int indexer_plan(const indexer_problem* pr, indexer_plan_t* out, size_t* ws_bytes)
{
    if (!pr || !out)
        return IDX_ERR_INVALID_ARG;
    *out = nullptr;
    const int R = pr->num_requests;
    if (R < 1 || R > kMaxRequests || pr->total_rows < 0 || pr->total_keys < 0 ||
        !pr->cu_seqlens_q || !pr->cu_seqlens_k || (pr->total_rows > 0 && !pr->compress_len))
        return IDX_ERR_INVALID_ARG;
    if (pr->topk < 1 || pr->topk > 2048 || pr->H < 1 || pr->D < 1)
        return IDX_ERR_INVALID_ARG;
    if (pr->kdtype != IDX_K_FP8_E4M3 && pr->kdtype != IDX_K_FP4_E2M1_UE8M0)
        return IDX_ERR_INVALID_ARG;
    if (pr->qdtype != IDX_Q_FP8_E4M3 && pr->qdtype != IDX_Q_FP4_E2M1_UE8M0)
        return IDX_ERR_INVALID_ARG;
    const int cb = pr->cand_block ? pr->cand_block : 8;
    const int ct = pr->cand_topk;
    if (cb < 1 || cb > 8 || (cb & (cb - 1)) != 0 || ct < 0 || ct > 4096)
        return IDX_ERR_INVALID_ARG;
    if (pr->key_block < 0 || (pr->key_block % kTileKeys) != 0)
        return IDX_ERR_INVALID_ARG;
    if (pr->cu_seqlens_q[0] != 0 || pr->cu_seqlens_k[0] != 0 ||
        pr->cu_seqlens_q[R] != pr->total_rows || pr->cu_seqlens_k[R] != pr->total_keys)
        return IDX_ERR_INVALID_ARG;
    if ((int64_t)pr->total_rows * pr->H > INT32_MAX)
        return IDX_ERR_INVALID_ARG;
    indexer_plan_s* p = new (std::nothrow) indexer_plan_s();
    if (!p)
        return IDX_ERR_INVALID_ARG;
    p->R = R;
    p->T = pr->total_rows;
    p->Lk = pr->total_keys;
    p->H = pr->H;
    p->D = pr->D;
    p->topk = pr->topk;
    p->kdtype = pr->kdtype;
    p->cand_block = cb;
    p->cand_topk = ct;
    p->budget = pr->transient_budget_bytes ? pr->transient_budget_bytes : kDefaultBudget;
    p->row_begin.assign(pr->cu_seqlens_q, pr->cu_seqlens_q + R + 1);
    p->key_begin.assign(pr->cu_seqlens_k, pr->cu_seqlens_k + R + 1);
    p->L.resize(R);
    for (int r = 0; r < R; ++r) {
        if (p->row_begin[r + 1] < p->row_begin[r] || p->key_begin[r + 1] < p->key_begin[r]) {
            delete p;
            return IDX_ERR_INVALID_ARG;
        }
        p->L[r] = p->key_begin[r + 1] - p->key_begin[r];
        p->max_L = std::max(p->max_L, p->L[r]);
    }
    p->clen.assign(pr->compress_len, pr->compress_len + p->T);
    for (int r = 0; r < R; ++r)
        for (int t = p->row_begin[r]; t < p->row_begin[r + 1]; ++t)
            if (p->clen[t] < 0 || p->clen[t] > p->L[r]) {
                delete p;
                return IDX_ERR_INVALID_ARG;
            }
    if (!supported_shape(p->H, p->D, p->kdtype)) {
        delete p;
        return IDX_ERR_UNSUPPORTED;
    }
    // 4 heads run as 8 (zero heads 4..7 add exactly 0 to every logit)
    p->kH = p->H == 4 ? 8 : p->H;
    p->fp4_native = p->kdtype == IDX_K_FP4_E2M1_UE8M0 && logits_fp4_native(p->kH, p->D);
    // e2m1 queries run with e2m1 keys on the block-scaled fp4 MMA (32 heads of 128)
    p->fp4_queries = pr->qdtype == IDX_Q_FP4_E2M1_UE8M0;
    if (p->fp4_queries && !p->fp4_native) {
        delete p;
        return IDX_ERR_UNSUPPORTED;
    }
    p->G = logits_rows_per_group(p->kH, p->fp4_native);
    const int G = p->G;

    // Key splits: the caller's size, else per request the fewest splits that keep
    // every (row group x split) unit within 1/(kUnitsPerSm x kPlanSms) of the whole
    // batch's work (row groups x key tiles), and splits of at least 8K keys, so that
    // one long request among short ones does not leave most SMs idle at the end.
    const int round_L = (int)std::max<int64_t>(kTileKeys, ceil_div(p->max_L, kTileKeys) * kTileKeys);
    int64_t total_tiles = 0;
    for (int r = 0; r < R; ++r)
        total_tiles += ceil_div(p->row_begin[r + 1] - p->row_begin[r], G) *
                       std::max<int64_t>(1, ceil_div(p->L[r], kTileKeys));
    const int64_t unit_tiles_max =
        std::max<int64_t>(8192 / kTileKeys, ceil_div(total_tiles, kUnitsPerSm * kPlanSms));
    p->split_r.resize(R);
    int S = 0;
    for (int r = 0; r < R; ++r) {
        int Sr;
        if (pr->key_block) {
            Sr = std::min(pr->key_block, round_L);
        } else {
            const int64_t tiles = std::max<int64_t>(1, ceil_div(p->L[r], kTileKeys));
            const int64_t ns = ceil_div(tiles, unit_tiles_max);
            Sr = (int)(ceil_div(ceil_div(tiles, ns), 1) * kTileKeys);
        }
        p->split_r[r] = std::max(Sr, (int)kTileKeys);
        S = std::max(S, p->split_r[r]);
    }
    p->split_keys = S;
    p->n_splits.resize(R);
    p->cap_k.resize(R);
    p->cap_b.resize(R);
    p->cnt_base.resize(R);
    // Each of a split's four sub-lists receives 32 of every 128 keys (its warp's
    // TMEM lanes), or 32 / cand_block blocks.  A sub-list holds a whole split when
    // that is small, and for requests too short to be sampled (their rows keep every
    // entry).  Otherwise it needs room for two things:
    //   * the exact stream: a compaction leaves a quarter of the kept set in each of
    //     the four sub-lists, plus two refresh intervals of appends;
    //   * the fixed-threshold pass: the upper tail (rank_tail_factor) of the entries a
    //     sub-list receives when the row's sampled threshold sits at the sample of rank
    //     mu + 5 sqrt(mu) + 4 (on average keep * rank / mu entries per row, spread over
    //     the row's splits x 4 sub-lists), plus 64.  A plan with a candidate path may serve
    //     masked consumers, whose passing entries come in candidate blocks of up to
    //     cand_block keys that all land in one sub-list, so they spread unevenly over
    //     the splits: those plans size for all of a row's entries in one split.  A
    //     sub-list that still overflows sends its row to the exact stream, so this only
    //     sizes the common case.
    const int slack = 2 * kUpdateTiles * 32;
    auto sub_cap = [&](int keep, int split_units, int ns, int st) {
        if (st == 0)
            return split_units;   // not sampled: every entry is kept
        int need = (keep + 3) / 4 + slack;
        {
            const double mu = (double)keep / st;
            const double rank = std::ceil(mu + 5.0 * std::sqrt(mu) + 4.0);
            const int spread = ct > 0 ? 1 : ns;
            need = std::max(need, (int)std::ceil(rank_tail_factor(rank) * keep * (rank / mu) /
                                                 (kListsPerSplit * spread)) + 64);
        }
        return std::min(split_units, need);
    };
    int64_t counts = 0;
    for (int r = 0; r < R; ++r) {
        const int ns = (int)std::max<int64_t>(1, ceil_div(p->L[r], p->split_r[r]));
        if ((int64_t)ns * kListsPerSplit > kMaxStreamSlots) {
            delete p;
            return IDX_ERR_UNSUPPORTED;
        }
        p->n_splits[r] = ns;
        const int split_tiles =
            (int)ceil_div(std::max(1, std::min(p->split_r[r], p->L[r])), kTileKeys);
        // the sampling stride this request gets below (0: not sampled)
        const int tiles_r = (int)ceil_div(std::max(1, p->L[r]), kTileKeys);
        const int st = pr->select_mode == IDX_SELECT_AUTO ? sample_stride_for(tiles_r, p->topk)
                                                           : 0;
        p->cap_k[r] = sub_cap(p->topk, split_tiles * 32, ns, st);
        p->cap_b[r] = ct ? sub_cap(ct, split_tiles * (32 / cb), ns, st) : 1;
        p->cnt_base[r] = counts;
        counts += (int64_t)(p->row_begin[r + 1] - p->row_begin[r]) * ns * kListsPerSplit;
    }
    // Sampled thresholds, per request with at least 2 x kSampleTiles key tiles:
    // tiles 0, s, 2s, ... (sample_stride_for: at least kSampleTiles per row, more where a
    // row's top k would hold fewer than kMinSampledMu samples).  With mu = k / s samples
    // expected among a row's top k (keys in random order), the threshold is the
    // sample of rank mu + 5 sqrt(mu) + 4, so that a row whose lists end up with
    // fewer than k entries (decided again by the exact path) is rare.  Shorter
    // requests are not sampled: their lists hold every entry.
    p->sample_stride_r.assign(R, 0);
    p->sample_rank_r.assign(R, 0);
    if (pr->select_mode == IDX_SELECT_AUTO) {
        for (int r = 0; r < R; ++r) {
            const int tiles = (int)ceil_div(std::max(1, p->L[r]), kTileKeys);
            const int st = sample_stride_for(tiles, p->topk);
            if (st == 0)
                continue;
            const double mu = (double)p->topk / st;
            const int cols = (int)ceil_div(tiles, st) * kTileKeys;
            p->sample_stride_r[r] = st;
            p->sample_rank_r[r] = (int)std::ceil(mu + 5.0 * std::sqrt(mu) + 4.0);   // (nonzero:
            // sampled; the kernel ranks each row by its own sample fraction)
            p->sample_stride = std::max(p->sample_stride, st);
            p->sample_cols = std::max(p->sample_cols, cols);
        }
        // every row of a sampled pass has a sample row, sampled or not
        p->sample_blocks = ct > 0 && p->sample_stride > 0;
    }
    size_t off = kStatusBytes;
    p->off_pad = off;
    if (p->kH != p->H)
        off = align_up(off + (size_t)p->T * p->kH * (p->D + 8), 256);
    p->off_k8 = off;
    if (p->kdtype == IDX_K_FP4_E2M1_UE8M0 && !p->fp4_native)
        off = align_up(off + (size_t)std::max(p->Lk, 1) * (p->D + 4), 256);
    p->pad_end = off;
    p->off_gtau = off;                       // [T] shared bound, then [T] row flags
    p->off_fail = off + (size_t)std::max(p->T, 1) * 4;
    off = align_up(p->off_fail + (size_t)std::max(p->T, 1) * 4, 256);
    p->off_tau = off;                        // [T] sampled thresholds, then [T] sample maxima
    off = align_up(off + (size_t)std::max(p->T, 1) * 8, 256);
    p->off_counts = off;
    off = align_up(off + (size_t)std::max<int64_t>(counts, 1) * 4, 256);
    p->off_lists = off;
    if (off >= p->budget) {
        delete p;
        return IDX_ERR_WORKSPACE;
    }
    const int64_t entries = (int64_t)((p->budget - off) / 8);
    if (!build_passes(*p, p->cap_k, entries, p->passes_k, p->max_piece_rows) ||
        (ct && !build_passes(*p, p->cap_b, entries, p->passes_b, p->max_piece_rows))) {
        delete p;
        return IDX_ERR_WORKSPACE;
    }
    int64_t need = pass_entries(*p, p->passes_k, p->cap_k);
    if (ct)
        need = std::max(need, pass_entries(*p, p->passes_b, p->cap_b));
    // a pass's sampled logits [rows, sample_cols] go to the list area first; a path
    // whose samples do not fit the budget is not sampled
    auto sample_entries = [&](const std::vector<Pass>& passes) {
        int64_t m = 0;
        for (const Pass& ps : passes)
            m = std::max<int64_t>(m, (int64_t)(ps.pieces.back().b - ps.pieces.front().a) *
                                         p->sample_cols / 2);
        return m;
    };
    if (p->sample_stride > 0) {
        const int64_t sk = sample_entries(p->passes_k);
        if (sk <= entries) {
            need = std::max(need, sk);
        } else {
            p->sample_stride = 0;
            p->sample_rank_r.assign(R, 0);
            p->sample_blocks = false;
        }
    }
    if (p->sample_blocks) {
        const int64_t sb = sample_entries(p->passes_b);
        if (sb <= entries)
            need = std::max(need, sb);
        else
            p->sample_blocks = false;
    }
    p->ws_bytes = align_up(off + (size_t)std::max<int64_t>(need, 1) * 8, 256);
    *out = p;
    if (ws_bytes)
        *ws_bytes = p->ws_bytes;
    return IDX_OK;
}

void indexer_plan_destroy(indexer_plan_t p) { delete p; }

int indexer_plan_info(indexer_plan_t p, int32_t* key_block, int32_t* row_chunk,
                      int32_t* max_splits, int32_t* sample_stride)
{
    if (!p)
        return IDX_ERR_INVALID_ARG;
    if (sample_stride)
        *sample_stride = p->sample_stride;
    if (key_block)
        *key_block = p->split_keys;
    if (row_chunk)
        *row_chunk = p->max_piece_rows;
    if (max_splits)
        *max_splits = *std::max_element(p->n_splits.begin(), p->n_splits.end());
    return IDX_OK;
}

int indexer_set_wait_budget(indexer_plan_t p, long long cycles)
{
    if (!p || cycles <= 0)
        return IDX_ERR_INVALID_ARG;
    p->wait_budget = cycles;
    return IDX_OK;
}

int indexer_logits(indexer_plan_t p, const void* q, const float* s_q, const float* w,
                   const void* k, const void* k_scale, const int32_t* clen, float* logits,
                   int64_t ld, void* ws, size_t ws_bytes, void* stream)
{
    if (!p || !ws || !aligned(ws, 256))
        return IDX_ERR_INVALID_ARG;
    if (ws_bytes < p->pad_end)
        return IDX_ERR_WORKSPACE;
    int rc = check_inputs(p, q, s_q, w, k, k_scale, clen);
    if (rc != IDX_OK)
        return rc;
    if (!logits || !aligned(logits, 4) || ld < std::max(p->max_L, 1) || ld > INT32_MAX)
        return IDX_ERR_INVALID_ARG;
    Ctx c;
    if ((rc = begin_call(c, p, ws, stream)) != IDX_OK)
        return rc;
    if (p->T == 0)
        return IDX_OK;
    if ((rc = prepare(c, q, s_q, w, k, k_scale, clen, ws)) != IDX_OK)
        return rc;
    c.lp.out = logits;
    // key tiles per unit: enough units for every SM to get several
    int64_t work = 0;
    for (int r = 0; r < p->R; ++r)
        work += ceil_div(p->row_begin[r + 1] - p->row_begin[r], p->G) * ceil_div(ld, kTileKeys);
    const int chunk = (int)std::min<int64_t>(64, std::max<int64_t>(4, work / (8LL * c.sms)));
    std::vector<Segment> segs;
    for (int r = 0; r < p->R; ++r) {
        const int rb = p->row_begin[r], re = p->row_begin[r + 1];
        if (re == rb)
            continue;
        Segment s;
        std::memset(&s, 0, sizeof(s));
        s.row_begin = rb;
        s.nrows = re - rb;
        s.key_base = p->key_begin[r];
        s.key_count = p->L[r];
        s.j_begin = 0;
        s.j_end = (int)ld;
        s.unit_tiles = chunk;
        s.n_row_groups = (int)ceil_div(s.nrows, p->G);
        s.n_chunks = (int)ceil_div(ceil_div(ld, kTileKeys), chunk);
        s.out_offset = (int64_t)rb * ld;
        s.out_ld = ld;
        segs.push_back(s);
        if ((int)segs.size() == kMaxSegments) {
            if ((rc = run_logits(c, segs, kSinkLogits)) != IDX_OK)
                return rc;
            segs.clear();
        }
    }
    return segs.empty() ? IDX_OK : run_logits(c, segs, kSinkLogits);
}

// Top-k over caller logits by the sampled path, pass by pass: samples gathered from
// the logits, row thresholds, one read of every row appending the entries at or
// above its threshold to its list, the verify merge; rows it cannot decide go to the
// direct kernel afterwards.
static int dense_sampled(Ctx& c, uint8_t* ws, const float* logits, int64_t ld,
                         const int32_t* clen, TopkParams& tp)
{
    const indexer_plan_s* p = c.p;
    uint32_t* tau_row = reinterpret_cast<uint32_t*>(ws + p->off_tau);
    uint32_t* row_fail = reinterpret_cast<uint32_t*>(ws + p->off_fail);
    uint32_t* fail_any = reinterpret_cast<uint32_t*>(ws) + 1;
    uint2* lists = reinterpret_cast<uint2*>(ws + p->off_lists);
    uint32_t* counts = reinterpret_cast<uint32_t*>(ws + p->off_counts);
    if (cudaMemsetAsync(ws + p->off_gtau, 0, (size_t)p->T * 8, c.st) != cudaSuccess ||
        cudaMemsetAsync(counts, 0, p->off_lists - p->off_counts, c.st) != cudaSuccess)
        return IDX_ERR_CUDA;
    c.lp.compress_len = clen;
    for (const Pass& ps : p->passes_k) {
        DenseFilterParams dp;
        std::memset(&dp, 0, sizeof(dp));
        dp.logits = logits;
        dp.ld = ld;
        dp.compress_len = clen;
        dp.samples = reinterpret_cast<float*>(lists);
        dp.sample_cols = p->sample_cols;
        dp.tau_row = tau_row;
        dp.lists = lists;
        dp.counts = counts;
        dp.num_requests = p->R;
        for (int r = 0; r < p->R; ++r) {
            dp.req_stride[r] = p->sample_rank_r[r] > 0 ? p->sample_stride_r[r] : 0;
            dp.req_key_count[r] = p->L[r];
        }
        StreamMergeParams mp;
        std::memset(&mp, 0, sizeof(mp));
        int ctas = 0, max_slots = 0;
        for (const PassPiece& pc : ps.pieces) {
            // the fused path's list layout: slots = splits x 4 lists of cap_k per row,
            // here one per key chunk of the row (a list that overflows sends its row to
            // the direct kernel)
            const int r = pc.r;
            const int slots = p->n_splits[r] * kListsPerSplit;
            const int chunk = (int)std::max<int64_t>(256, ceil_div(ceil_div(std::max(p->L[r], 1),
                                                                            slots), 256) * 256);
            const int64_t cnt = p->cnt_base[r] + (int64_t)(pc.a - p->row_begin[r]) * slots;
            dp.piece[dp.num_pieces++] =
                DensePiece{pc.a, pc.b - pc.a, r, slots, chunk, p->cap_k[r], pc.list_off, cnt};
            MergePiece& m = mp.piece[mp.num_pieces++];
            m.row_begin = pc.a;
            m.nrows = pc.b - pc.a;
            m.cta_begin = ctas;
            m.slots = slots;
            m.cap = p->cap_k[r];
            m.key_count = p->L[r];
            m.list_offset = pc.list_off;
            m.count_offset = cnt;
            ctas += pc.b - pc.a;
            max_slots = std::max(max_slots, slots);
        }
        const int first = ps.pieces.front().a;
        const int rows = ps.pieces.back().b - first;
        g_launches.fetch_add(3, std::memory_order_relaxed);
        if (launch_dense_gather(dp, rows, c.st) != cudaSuccess)
            return IDX_ERR_CUDA;
        int rc = row_thresholds(c, ps, dp.samples, tau_row, 1, p->topk);
        if (rc != IDX_OK)
            return rc;
        if (launch_dense_filter(dp, rows, max_slots, c.st) != cudaSuccess)
            return IDX_ERR_CUDA;
        mp.total_ctas = ctas;
        mp.lists = lists;
        mp.counts = counts;
        mp.verify = 1;
        mp.tau_row = tau_row;
        mp.smax_row = tau_row + p->T;
        mp.row_fail = row_fail;
        mp.fail_any = fail_any;
        mp.k = p->topk;
        mp.bitmap = 1;
        mp.out_idx = tp.out_idx;
        mp.out_val = tp.out_val;
        if (launch_stream_merge(mp, c.st) != cudaSuccess)
            return IDX_ERR_CUDA;
    }
    tp.row_fail = row_fail;
    tp.fail_any = fail_any;
    return IDX_OK;
}

// Top-k over caller logits in one read of every row: each row's sampled threshold
// straight from the logits, then the single-read kernel (candidates and the exact
// selection in shared memory); rows it cannot decide go to the direct kernel afterwards.
// For plans whose requests have at most 65,536 keys and 16-byte aligned logits rows.
static int dense_single_read(Ctx& c, uint8_t* ws, const float* logits, int64_t ld,
                             const int32_t* clen, TopkParams& tp)
{
    const indexer_plan_s* p = c.p;
    uint32_t* tau_row = reinterpret_cast<uint32_t*>(ws + p->off_tau);
    uint32_t* row_fail = reinterpret_cast<uint32_t*>(ws + p->off_fail);
    uint32_t* fail_any = reinterpret_cast<uint32_t*>(ws) + 1;
    uint32_t* row_counter = reinterpret_cast<uint32_t*>(ws) + 2;   // zeroed with the status
    if (cudaMemsetAsync(ws + p->off_gtau, 0, (size_t)p->T * 8, c.st) != cudaSuccess)
        return IDX_ERR_CUDA;
    SampleParams sp;
    std::memset(&sp, 0, sizeof(sp));
    sp.samples = nullptr;
    sp.logits = logits;
    sp.ld_logits = ld;
    sp.ld = p->sample_cols;
    sp.row0 = 0;
    sp.rows = p->T;
    sp.k = p->topk;
    sp.pool = 1;
    sp.compress_len = clen;
    sp.tau_row = tau_row;
    sp.smax_row = tau_row + p->T;
    sp.num_requests = p->R;
    for (int r = 0; r < p->R; ++r) {
        sp.req_row_begin[r] = p->row_begin[r];
        sp.req_rank[r] = p->sample_rank_r[r] > 0 ? p->sample_stride_r[r] : 0;
        sp.req_key_count[r] = p->L[r];
        sp.req_cols[r] = p->sample_rank_r[r] > 0
                             ? (int)ceil_div(ceil_div(std::max(1, p->L[r]), kTileKeys),
                                             p->sample_stride_r[r]) * kTileKeys
                             : 0;
    }
    sp.req_row_begin[p->R] = p->row_begin[p->R];
    RowTopkParams rp;
    std::memset(&rp, 0, sizeof(rp));
    rp.logits = logits;
    rp.ld = ld;
    rp.compress_len = clen;
    rp.tau_row = tau_row;
    rp.smax_row = tau_row + p->T;
    rp.row_fail = row_fail;
    rp.fail_any = fail_any;
    rp.row_counter = row_counter;
    rp.status = reinterpret_cast<uint32_t*>(ws);
    rp.timeout_cycles = p->wait_budget;
    rp.out_idx = tp.out_idx;
    rp.out_val = tp.out_val;
    rp.k = p->topk;
    rp.total_rows = p->T;
    rp.num_requests = p->R;
    for (int r = 0; r < p->R; ++r) {
        rp.req_row_begin[r] = p->row_begin[r];
        rp.req_key_count[r] = p->L[r];
    }
    rp.req_row_begin[p->R] = p->row_begin[p->R];
    g_launches.fetch_add(2, std::memory_order_relaxed);
    if (launch_sample_threshold(sp, c.st) != cudaSuccess ||
        launch_row_topk(rp, c.st) != cudaSuccess)
        return IDX_ERR_CUDA;
    tp.row_fail = row_fail;
    tp.fail_any = fail_any;
    return IDX_OK;
}

int indexer_topk(indexer_plan_t p, const float* logits, int64_t ld, const int32_t* clen,
                 int32_t* out_idx, float* out_val, void* ws, size_t ws_bytes, void* stream)
{
    if (!p || !ws || !aligned(ws, 256))
        return IDX_ERR_INVALID_ARG;
    if (ws_bytes < kStatusBytes)
        return IDX_ERR_WORKSPACE;
    if (!logits || !clen || !out_idx || ld < std::max(p->max_L, 1) || !aligned(logits, 4) ||
        !aligned(out_idx, 4) || (out_val && !aligned(out_val, 4)))
        return IDX_ERR_INVALID_ARG;
    Ctx c;
    int rc;
    if ((rc = begin_call(c, p, ws, stream)) != IDX_OK)
        return rc;
    TopkParams tp;
    std::memset(&tp, 0, sizeof(tp));
    tp.logits = logits;
    tp.ld = ld;
    tp.compress_len = clen;
    tp.k = p->topk;
    tp.total_rows = p->T;
    tp.num_requests = p->R;
    tp.out_idx = out_idx;
    tp.out_val = out_val;
    for (int r = 0; r < p->R; ++r) {
        tp.req_row_begin[r] = p->row_begin[r];
        tp.req_key_count[r] = p->L[r];
    }
    tp.req_row_begin[p->R] = p->row_begin[p->R];
    // with the plan's whole workspace, the sampled path decides most rows; the direct
    // kernel then handles only the rows it could not (or every row, without it)
    if (ws_bytes >= p->ws_bytes && p->sample_stride > 0 && p->T > 0) {
        const bool single = p->max_L <= row_topk_max_keys() && ld % 4 == 0 &&
                            aligned(logits, 16);
        if ((rc = single ? dense_single_read(c, static_cast<uint8_t*>(ws), logits, ld, clen, tp)
                         : dense_sampled(c, static_cast<uint8_t*>(ws), logits, ld, clen, tp)) !=
            IDX_OK)
            return rc;
    }
    g_launches.fetch_add(1, std::memory_order_relaxed);
    return launch_topk_dense(tp, c.st) == cudaSuccess ? IDX_OK : IDX_ERR_CUDA;
}

static int fused_topk_impl(indexer_plan_t p, const void* q, const float* s_q, const float* w,
                       const void* k, const void* k_scale, const int32_t* clen,
                       const uint8_t* cand_mask, int64_t ld_mask, const int32_t* mask_rows,
                       int64_t mask_row_count, int32_t* out_idx, float* out_val, void* ws,
                       size_t ws_bytes, void* stream)
{
    int rc = check_common(p, ws, ws_bytes);
    if (rc != IDX_OK)
        return rc;
    if ((rc = check_inputs(p, q, s_q, w, k, k_scale, clen)) != IDX_OK)
        return rc;
    if (!out_idx || !aligned(out_idx, 4) || (out_val && !aligned(out_val, 4)))
        return IDX_ERR_INVALID_ARG;
    if (cand_mask && ld_mask < (p->max_L + p->cand_block - 1) / p->cand_block)
        return IDX_ERR_INVALID_ARG;
    Ctx c;
    if ((rc = begin_call(c, p, ws, stream)) != IDX_OK)
        return rc;
    if (p->T == 0)
        return IDX_OK;
    if ((rc = prepare(c, q, s_q, w, k, k_scale, clen, ws)) != IDX_OK)
        return rc;
    c.lp.cand_mask = cand_mask;
    c.lp.ld_mask = ld_mask;
    c.lp.mask_rows = mask_rows;
    c.lp.mask_row_count = mask_row_count;
    uint8_t* wsb = static_cast<uint8_t*>(ws);
    // shared bounds and row flags
    if (cudaMemsetAsync(wsb + p->off_gtau, 0, (size_t)p->T * 8, c.st) != cudaSuccess)
        return IDX_ERR_CUDA;
    return run_streamed(c, wsb, 0, out_idx, out_val, nullptr, 0);
}

int indexer_fused_topk(indexer_plan_t p, const void* q, const float* s_q, const float* w,
                       const void* k, const void* k_scale, const int32_t* clen,
                       const uint8_t* cand_mask, int64_t ld_mask, int32_t* out_idx,
                       float* out_val, void* ws, size_t ws_bytes, void* stream)
{
    return fused_topk_impl(p, q, s_q, w, k, k_scale, clen, cand_mask, ld_mask, nullptr, 0,
                           out_idx, out_val, ws, ws_bytes, stream);
}

int indexer_fused_topk_mapped(indexer_plan_t p, const void* q, const float* s_q, const float* w,
                              const void* k, const void* k_scale, const int32_t* clen,
                              const uint8_t* cand_mask, int64_t ld_mask, const int32_t* mask_rows,
                              int64_t mask_row_count, int32_t* out_idx, float* out_val, void* ws,
                              size_t ws_bytes, void* stream)
{
    if (!cand_mask || !mask_rows || !aligned(mask_rows, 4) || mask_row_count < 1)
        return IDX_ERR_INVALID_ARG;
    return fused_topk_impl(p, q, s_q, w, k, k_scale, clen, cand_mask, ld_mask, mask_rows,
                           mask_row_count, out_idx, out_val, ws, ws_bytes, stream);
}

static int candidates_impl(indexer_plan_t p, const void* q, const float* s_q, const float* w,
                             const void* k, const void* k_scale, const int32_t* clen,
                             const int32_t* tail, uint8_t* cand_mask, int64_t ld_mask, void* ws,
                             size_t ws_bytes, void* stream)
{
    int rc = check_common(p, ws, ws_bytes);
    if (rc != IDX_OK)
        return rc;
    if ((rc = check_inputs(p, q, s_q, w, k, k_scale, clen)) != IDX_OK)
        return rc;
    if (!cand_mask || ld_mask < (p->max_L + p->cand_block - 1) / p->cand_block ||
        p->cand_topk == 0)
        return IDX_ERR_INVALID_ARG;
    Ctx c;
    if (tail) {
        // request r's last tail[r] rows, packed: mask row of row t = t + delta_r
        int64_t packed = 0;
        c.mask_delta.resize(p->R);
        for (int r = 0; r < p->R; ++r) {
            const int rows = p->row_begin[r + 1] - p->row_begin[r];
            if (tail[r] < 0 || tail[r] > rows)
                return IDX_ERR_INVALID_ARG;
            c.mask_delta[r] = packed - (p->row_begin[r + 1] - tail[r]);
            packed += tail[r];
        }
        c.tail = tail;
    }
    if ((rc = begin_call(c, p, ws, stream)) != IDX_OK)
        return rc;
    if (p->T == 0)
        return IDX_OK;
    if ((rc = prepare(c, q, s_q, w, k, k_scale, clen, ws)) != IDX_OK)
        return rc;
    uint8_t* wsb = static_cast<uint8_t*>(ws);
    // shared bounds and row flags (contiguous)
    if (cudaMemsetAsync(wsb + p->off_gtau, 0, (size_t)p->T * 8, c.st) != cudaSuccess)
        return IDX_ERR_CUDA;
    return run_streamed(c, wsb, p->cand_block, nullptr, nullptr, cand_mask, ld_mask);
}

int indexer_candidate_blocks(indexer_plan_t p, const void* q, const float* s_q, const float* w,
                             const void* k, const void* k_scale, const int32_t* clen,
                             uint8_t* cand_mask, int64_t ld_mask, void* ws, size_t ws_bytes,
                             void* stream)
{
    return candidates_impl(p, q, s_q, w, k, k_scale, clen, nullptr, cand_mask, ld_mask, ws,
                           ws_bytes, stream);
}

int indexer_candidate_blocks_tail(indexer_plan_t p, const void* q, const float* s_q,
                                  const float* w, const void* k, const void* k_scale,
                                  const int32_t* clen, const int32_t* publish_rows,
                                  uint8_t* cand_mask, int64_t ld_mask, void* ws, size_t ws_bytes,
                                  void* stream)
{
    if (!publish_rows)
        return IDX_ERR_INVALID_ARG;
    return candidates_impl(p, q, s_q, w, k, k_scale, clen, publish_rows, cand_mask, ld_mask, ws,
                           ws_bytes, stream);
}

int indexer_expand_mask(indexer_plan_t p, const uint8_t* cand_mask, int64_t ld_mask,
                        const int32_t* clen, uint8_t* key_mask, int64_t ld, void* stream)
{
    if (!p || !cand_mask || !clen || !key_mask || ld < std::max(p->max_L, 1) ||
        ld_mask < (p->max_L + p->cand_block - 1) / p->cand_block)
        return IDX_ERR_INVALID_ARG;
    if (!device_info().ok)
        return IDX_ERR_UNSUPPORTED;
    g_launches.fetch_add(1, std::memory_order_relaxed);
    return launch_expand_mask(cand_mask, ld_mask, clen, key_mask, ld, p->cand_block, p->T,
                              reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
               ? IDX_OK
               : IDX_ERR_CUDA;
}

int indexer_convert_fp4(const uint8_t* codes, const uint8_t* block_scales, int64_t rows,
                        int32_t D, uint8_t* out_e4m3, float* out_scale, void* ws,
                        size_t ws_bytes, void* stream)
{
    if (!codes || !block_scales || !out_e4m3 || !out_scale || !ws || ws_bytes < kStatusBytes ||
        !aligned(ws, 256) || rows < 0 || rows > 0x7FFFFFFF || D < 32 || D % 32 != 0 ||
        !aligned(codes, 4) || !aligned(out_e4m3, 8))
        return IDX_ERR_INVALID_ARG;
    if (!device_info().ok)
        return IDX_ERR_UNSUPPORTED;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(ws, 0, kStatusBytes, st) != cudaSuccess)
        return IDX_ERR_CUDA;
    if (rows == 0)
        return IDX_OK;
    g_launches.fetch_add(1, std::memory_order_relaxed);
    return launch_fp4_to_fp8(codes, block_scales, static_cast<int>(rows), D, out_e4m3, out_scale,
                             static_cast<uint32_t*>(ws), st) == cudaSuccess
               ? IDX_OK
               : IDX_ERR_CUDA;
}

int indexer_page_indices(indexer_plan_t p, const int32_t* raw_idx, const int32_t* page_table,
                         int64_t ld_page_table, int32_t page_size, int32_t* page_idx,
                         void* stream)
{
    if (!p || !raw_idx || !page_table || !page_idx || page_size < 1 ||
        ld_page_table < (p->max_L + page_size - 1) / page_size || p->R > kMaxRequests)
        return IDX_ERR_INVALID_ARG;
    if (!device_info().ok)
        return IDX_ERR_UNSUPPORTED;
    if (p->T == 0 || p->topk == 0)
        return IDX_OK;
    PageIndexParams pp;
    std::memset(&pp, 0, sizeof(pp));
    pp.raw = raw_idx;
    pp.out = page_idx;
    pp.table = page_table;
    pp.ld_table = ld_page_table;
    pp.page = page_size;
    pp.k = p->topk;
    pp.rows = p->T;
    pp.num_requests = p->R;
    for (int r = 0; r < p->R; ++r) {
        pp.req_row_begin[r] = p->row_begin[r];
        pp.req_key_count[r] = p->L[r];
    }
    pp.req_row_begin[p->R] = p->row_begin[p->R];
    g_launches.fetch_add(1, std::memory_order_relaxed);
    return launch_page_indices(pp, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
               ? IDX_OK
               : IDX_ERR_CUDA;
}

int indexer_selftest_timeout(void* ws, long long cycles, void* stream)
{
    if (!ws || !aligned(ws, 256) || cycles <= 0)
        return IDX_ERR_INVALID_ARG;
    if (!device_info().ok)
        return IDX_ERR_UNSUPPORTED;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(ws, 0, kStatusBytes, st) != cudaSuccess)
        return IDX_ERR_CUDA;
    g_launches.fetch_add(1, std::memory_order_relaxed);
    return launch_selftest_timeout(static_cast<uint32_t*>(ws), cycles, st) == cudaSuccess
               ? IDX_OK
               : IDX_ERR_CUDA;
}

// ---------------------------------------------------------------------------
// Allocation-free fused top-k.  Some callers cannot obtain device memory for a
// workspace: plugins whose host application owns every byte of device memory
// through its own pool and exposes no allocator, or serving loops where a
// cudaMalloc would stall every stream on the device.  For them the workspace
// lives in this fixed, file-scope device array instead.  Every GPU that loads
// the library reserves it until the process exits.
// ---------------------------------------------------------------------------
namespace {

constexpr size_t kNoAllocScratchBytes = IDX_NOALLOC_SCRATCH_BYTES;  // 64 MiB
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_noalloc_mu;
void* g_noalloc_addr[256] = {};  // device address of the array, per device ordinal

// Device address of the array on the current device.  The first call on a device
// resolves it with cudaGetSymbolAddress (the host-side name of the array is a
// stand-in, not a device address); later calls reuse the cached pointer.
int noalloc_scratch(void** out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 256)
        return IDX_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (!g_noalloc_addr[dev]) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr)
            return IDX_ERR_CUDA;
        g_noalloc_addr[dev] = ptr;
    }
    *out = g_noalloc_addr[dev];
    return IDX_OK;
}

}  // namespace

int indexer_fused_topk_noalloc(indexer_plan_t p, const void* q, const float* s_q, const float* w,
                               const void* k, const void* k_scale, const int32_t* clen,
                               const uint8_t* cand_mask, int64_t ld_mask, int32_t* out_idx,
                               float* out_val, void* stream)
{
    if (!p)
        return IDX_ERR_INVALID_ARG;
    if (p->ws_bytes > kNoAllocScratchBytes)
        return IDX_ERR_WORKSPACE;
    if (!device_info().ok)
        return IDX_ERR_UNSUPPORTED;
    void* scratch = nullptr;
    int rc = noalloc_scratch(&scratch);
    if (rc != IDX_OK)
        return rc;
    return indexer_fused_topk(p, q, s_q, w, k, k_scale, clen, cand_mask, ld_mask, out_idx,
                              out_val, scratch, kNoAllocScratchBytes, stream);
}

int indexer_noalloc_status(void* stream)
{
    if (!device_info().ok)
        return IDX_ERR_UNSUPPORTED;
    void* scratch = nullptr;
    const int rc = noalloc_scratch(&scratch);
    if (rc != IDX_OK)
        return rc;
    return indexer_status(nullptr, scratch, stream);
}

long long indexer_fallback_rows(indexer_plan_t p, const void* ws, void* stream)
{
    if (!p || !ws)
        return IDX_ERR_INVALID_ARG;
    if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
        return IDX_ERR_CUDA;
    std::vector<uint32_t> flags(std::max(p->T, 1));
    if (p->T > 0 && cudaMemcpy(flags.data(), static_cast<const uint8_t*>(ws) + p->off_fail,
                               (size_t)p->T * 4, cudaMemcpyDeviceToHost) != cudaSuccess)
        return IDX_ERR_CUDA;
    long long n = 0;
    for (int t = 0; t < p->T; ++t)
        n += flags[t] != 0;
    return n;
}

int indexer_status(indexer_plan_t p, const void* ws, void* stream)
{
    (void)p;
    if (!ws)
        return IDX_ERR_INVALID_ARG;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(st) != cudaSuccess)
        return IDX_ERR_CUDA;
    uint32_t word = 0;
    if (cudaMemcpy(&word, ws, 4, cudaMemcpyDeviceToHost) != cudaSuccess)
        return IDX_ERR_CUDA;
    if (word & kStatusTimeout)
        return IDX_ERR_TIMEOUT;
    if (word)
        return IDX_ERR_DEVICE_CHECK;
    return IDX_OK;
}

}  // extern "C"
