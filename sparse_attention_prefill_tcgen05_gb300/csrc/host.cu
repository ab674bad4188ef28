// Host side of the C ABI: problem validation, the per-batch plan, workspace
// layout, TMA descriptors and kernel launches.  No device memory is ever
// allocated here; every call is asynchronous on the caller's stream.
#include <algorithm>
#include <atomic>
#include <cstring>
#include <mutex>
#include <new>
#include <vector>

#include "../../include/indexer.h"
#include "internal.h"
#include "ptx.cuh"

using namespace idx;

struct indexer_plan_s {
    int R = 0, T = 0, Lk = 0, H = 0, D = 0, topk = 0, kdtype = 0;
    int cand_block = 8, cand_topk = 0;
    std::vector<int32_t> row_begin;   // [R+1]
    std::vector<int32_t> key_begin;   // [R+1]
    std::vector<int32_t> L;           // [R]
    std::vector<int32_t> clen;        // [T]
    int max_L = 0;
    uint64_t budget = 0;
    // blocked top-k
    int key_block = 0;                // B_k (multiple of 128)
    int row_chunk = 0;                // rows of scratch logits per pass
    std::vector<int32_t> n_splits;    // per request
    std::vector<int64_t> cand_off;    // per request, entries (topk per slot)
    std::vector<int64_t> cblk_off;    // per request, entries (cand_topk per slot)
    int64_t cand_entries = 0, cblk_entries = 0;
    // workspace layout (bytes)
    size_t off_cand_val = 0, off_cand_idx = 0, off_cblk_val = 0, off_cblk_idx = 0;
    size_t off_scratch = 0, scratch_bytes = 0, ws_bytes = 0;
    long long wait_budget = 4000000000LL;
};

namespace {

std::atomic<long long> g_launches{0};  // kernels launched by this library (diagnostic)

constexpr size_t kStatusBytes = 256;
constexpr uint64_t kDefaultBudget = 2ull << 30;

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

bool supported_shape(int H, int D, int kdtype)
{
    // e2m1 keys: the block-scaled MMA kernel raised an illegal instruction on its
    // first GB300 run and is not launched until that is understood.
    if (kdtype == IDX_K_FP4_E2M1_UE8M0)
        return false;
    return (H == 32 && D == 128) || (H == 16 && D == 128) || (H == 64 && D == 128) ||
           (H == 4 && D == 64);
}

// Lay out the workspace for a key block and row chunk; returns total bytes.
size_t layout(indexer_plan_s& p, int key_block, int row_chunk)
{
    p.key_block = key_block;
    p.row_chunk = row_chunk;
    p.n_splits.assign(p.R, 1);
    p.cand_off.assign(p.R, 0);
    p.cblk_off.assign(p.R, 0);
    int64_t ce = 0, be = 0;
    for (int r = 0; r < p.R; ++r) {
        const int ns = std::max(1, (p.L[r] + key_block - 1) / key_block);
        p.n_splits[r] = ns;
        p.cand_off[r] = ce;
        p.cblk_off[r] = be;
        const int64_t rows = p.row_begin[r + 1] - p.row_begin[r];
        ce += rows * ns * p.topk;
        be += rows * ns * p.cand_topk;
    }
    if (p.cand_topk == 0)
        be = 0;
    p.cand_entries = ce;
    p.cblk_entries = be;
    // top-k candidates and candidate-block candidates are never live in the
    // same call, so they share one area
    const size_t area = (size_t)std::max(ce, be) * 4;
    size_t off = kStatusBytes;
    p.off_cand_val = p.off_cblk_val = off;
    off = align_up(off + area, 256);
    p.off_cand_idx = p.off_cblk_idx = off;
    off = align_up(off + area, 256);
    p.off_scratch = off;
    p.scratch_bytes = (size_t)row_chunk * key_block * 4;
    off = align_up(off + p.scratch_bytes, 256);
    p.ws_bytes = off;
    return off;
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

// Map over packed e2m1 keys [rows, D/2 bytes] that unpacks each 16-element
// group into a 16-byte shared-memory slot (8 data bytes, 8 bytes gap): the
// 8-bit-container layout the f8f6f4 MMA kinds read 4-bit operands from.  A
// box of 128 elements x box_rows lands as box_rows rows of 128 bytes,
// 128-byte swizzled like the e4m3 tiles.
bool make_map_fp4(CUtensorMap* m, const void* base, uint64_t rows, uint32_t D,
                  uint32_t box_rows)
{
    EncodeTiledFn enc = encode_fn();
    if (!enc)
        return false;
    const cuuint64_t dims[2] = {D, rows};
    const cuuint64_t strides[1] = {D / 2};
    const cuuint32_t box[2] = {128, box_rows};
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
    if (!aligned(q, 16) || !aligned(k, p->kdtype == IDX_K_FP8_E4M3 ? 16 : 32) ||
        !aligned(s_q, 4) || !aligned(w, 4) ||
        !aligned(clen, 4) || (p->kdtype == IDX_K_FP8_E4M3 && !aligned(k_scale, 4)))
        return IDX_ERR_INVALID_ARG;
    return IDX_OK;
}

// One piece of blocked work: rows [a, b) of request r against key split s.
struct Piece {
    int r, a, b, s;
    int width;  // keys of the split, rounded up to a tile (scratch row length)
};

struct Ctx {
    const indexer_plan_s* p;
    LogitsParams lp;
    int sms;
    cudaStream_t st;
};

int fill_maps(Ctx& c, const void* q, const void* k)
{
    const indexer_plan_s* p = c.p;
    std::memset(&c.lp, 0, sizeof(c.lp));
    const int G = logits_rows_per_group(p->H, p->kdtype);
    if (!make_map(&c.lp.tmap_q, q, (uint64_t)p->T * p->H, p->D, G * p->H))
        return IDX_ERR_CUDA;
    const uint64_t krows = (uint64_t)std::max(p->Lk, 1);
    const bool ok = p->kdtype == IDX_K_FP8_E4M3
                        ? make_map(&c.lp.tmap_k, k, krows, p->D, kTileKeys)
                        : make_map_fp4(&c.lp.tmap_k, k, krows, p->D, kTileKeys);
    return ok ? IDX_OK : IDX_ERR_CUDA;
}

// Launch the logits kernel over a list of segments (<= kMaxSegments).
int run_logits(Ctx& c, const std::vector<Segment>& segs_in, float* out)
{
    const indexer_plan_s* p = c.p;
    const int G = logits_rows_per_group(p->H, p->kdtype);
    // choose key tiles per unit so that there are several units per SM
    int64_t work = 0;
    for (const Segment& s : segs_in)
        work += (int64_t)((s.nrows + G - 1) / G) * ((s.j_end - s.j_begin + kTileKeys - 1) / kTileKeys);
    int chunk = (int)std::min<int64_t>(64, std::max<int64_t>(4, work / (8LL * c.sms)));
    LogitsParams& lp = c.lp;
    lp.chunk_tiles = chunk;
    lp.num_segments = (int)segs_in.size();
    int units = 0;
    for (size_t i = 0; i < segs_in.size(); ++i) {
        Segment s = segs_in[i];
        s.n_row_groups = (s.nrows + G - 1) / G;
        const int tiles = (s.j_end - s.j_begin + kTileKeys - 1) / kTileKeys;
        s.n_chunks = (tiles + chunk - 1) / chunk;
        s.unit_begin = units;
        units += s.n_row_groups * s.n_chunks;
        lp.seg[i] = s;
    }
    lp.total_units = units;
    lp.out = out;
    lp.timeout_cycles = p->wait_budget;
    if (units == 0)
        return IDX_OK;
    const int grid = std::min(units, c.sms);
    g_launches.fetch_add(1, std::memory_order_relaxed);
    return launch_logits(lp, p->H, p->D, p->kdtype, grid, c.st) == cudaSuccess ? IDX_OK
                                                                              : IDX_ERR_CUDA;
}

// Blocked pass shared by fused top-k (pool = 0) and candidate blocks (pool = block):
// score rows against key splits into scratch, keep per-split top-k candidates.
int run_blocked(Ctx& c, uint8_t* ws, int pool)
{
    const indexer_plan_s* p = c.p;
    float* scratch = reinterpret_cast<float*>(ws + p->off_scratch);
    const int kk = pool ? p->cand_topk : p->topk;
    float* cval = reinterpret_cast<float*>(ws + (pool ? p->off_cblk_val : p->off_cand_val));
    int32_t* cidx = reinterpret_cast<int32_t*>(ws + (pool ? p->off_cblk_idx : p->off_cand_idx));
    const int64_t cap = (int64_t)p->row_chunk * p->key_block;  // scratch floats

    std::vector<Piece> batch;
    int64_t used = 0;
    auto flush = [&]() -> int {
        if (batch.empty())
            return IDX_OK;
        std::vector<Segment> segs;
        SelParams sp;
        std::memset(&sp, 0, sizeof(sp));
        int64_t off = 0;
        int rows = 0;
        for (size_t i = 0; i < batch.size(); ++i) {
            const Piece& pc = batch[i];
            const int r = pc.r;
            const int j0 = pc.s * p->key_block;
            const int j1 = std::min(p->L[r], j0 + p->key_block);
            Segment s;
            std::memset(&s, 0, sizeof(s));
            s.row_begin = pc.a;
            s.nrows = pc.b - pc.a;
            s.key_base = p->key_begin[r];
            s.key_count = p->L[r];
            s.j_begin = j0;
            s.j_end = j1;
            s.out_offset = off;
            s.out_ld = pc.width;
            segs.push_back(s);
            SelSegment& q = sp.seg[i];
            q.row_begin = pc.a;
            q.nrows = pc.b - pc.a;
            q.j_begin = pool ? j0 / pool : j0;
            q.n_entries = pool ? (j1 - j0 + pool - 1) / pool : (j1 - j0);
            q.key_count = p->L[r];
            q.cand_slot = pc.s;
            q.n_slots = p->n_splits[r];
            q.src_offset = off;
            q.src_ld = pc.width;
            q.cand_offset = (pool ? p->cblk_off[r] : p->cand_off[r]) +
                            (int64_t)(pc.a - p->row_begin[r]) * p->n_splits[r] * kk;
            q.row_block = rows;
            rows += pc.b - pc.a;
            off += (int64_t)(pc.b - pc.a) * pc.width;
        }
        int rc = run_logits(c, segs, scratch);
        if (rc != IDX_OK)
            return rc;
        sp.src = scratch;
        sp.compress_len = c.lp.compress_len;
        sp.k = kk;
        sp.pool = pool;
        sp.num_segments = (int)batch.size();
        sp.total_rows_launch = rows;
        sp.cand_val = cval;
        sp.cand_idx = cidx;
        g_launches.fetch_add(1, std::memory_order_relaxed);
        if (launch_select_dense(sp, c.st) != cudaSuccess)
            return IDX_ERR_CUDA;
        batch.clear();
        used = 0;
        return IDX_OK;
    };

    for (int r = 0; r < p->R; ++r) {
        const int rb = p->row_begin[r], re = p->row_begin[r + 1];
        if (re == rb)
            continue;
        for (int s = 0; s < p->n_splits[r]; ++s) {
            const int j0 = s * p->key_block;
            const int j1 = std::min(p->L[r], j0 + p->key_block);
            const int width = std::max(kTileKeys, (j1 - j0 + kTileKeys - 1) / kTileKeys * kTileKeys);
            const int rows_fit = (int)std::max<int64_t>(1, cap / width);
            for (int a = rb; a < re; a += rows_fit) {
                const int b = std::min(re, a + rows_fit);
                const int64_t need = (int64_t)(b - a) * width;
                if (used + need > cap || (int)batch.size() == kMaxSegments) {
                    int rc = flush();
                    if (rc != IDX_OK)
                        return rc;
                }
                batch.push_back(Piece{r, a, b, s, width});
                used += need;
            }
        }
    }
    return flush();
}

int run_merge(Ctx& c, uint8_t* ws, int pool, int32_t* out_idx, float* out_val, uint8_t* mask,
              int64_t ld_mask)
{
    const indexer_plan_s* p = c.p;
    MergeParams mp;
    std::memset(&mp, 0, sizeof(mp));
    mp.cand_val = reinterpret_cast<const float*>(ws + (pool ? p->off_cblk_val : p->off_cand_val));
    mp.cand_idx = reinterpret_cast<const int32_t*>(ws + (pool ? p->off_cblk_idx : p->off_cand_idx));
    mp.k = pool ? p->cand_topk : p->topk;
    mp.num_requests = p->R;
    mp.total_rows = p->T;
    mp.out_idx = out_idx;
    mp.out_val = out_val;
    mp.mask = mask;
    mp.ld_mask = ld_mask;
    for (int r = 0; r < p->R; ++r) {
        mp.req_row_begin[r] = p->row_begin[r];
        mp.req_slots[r] = p->n_splits[r];
        mp.req_cand_offset[r] = pool ? p->cblk_off[r] : p->cand_off[r];
    }
    mp.req_row_begin[p->R] = p->row_begin[p->R];
    g_launches.fetch_add(1, std::memory_order_relaxed);
    return launch_merge(mp, c.st) == cudaSuccess ? IDX_OK : IDX_ERR_CUDA;
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
    c.lp.s_q = s_q;
    c.lp.w = w;
    c.lp.s_k = c.p->kdtype == IDX_K_FP8_E4M3 ? static_cast<const float*>(k_scale) : nullptr;
    c.lp.k_sf = c.p->kdtype == IDX_K_FP8_E4M3 ? nullptr : static_cast<const uint8_t*>(k_scale);
    c.lp.compress_len = clen;
    c.lp.status = static_cast<uint32_t*>(ws);
    c.lp.mask_block = c.p->cand_block;
}

}  // namespace

extern "C" {

int indexer_version(void) { return 1; }

long long indexer_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

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
    const int cb = pr->cand_block ? pr->cand_block : 8;
    const int ct = pr->cand_topk;
    if (cb < 1 || ct < 0 || ct > 4096 || (kTileKeys % cb) != 0)
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
    // Key block: the caller's, else the candidate (whole prefix, 64K, 32K, ... 1K keys)
    // needing the fewest logits passes within the budget.
    const int round_L = std::max(kTileKeys, (p->max_L + kTileKeys - 1) / kTileKeys * kTileKeys);
    const int G = logits_rows_per_group(p->H, p->kdtype);
    std::vector<int> cands;
    if (pr->key_block)
        cands.push_back(std::min(pr->key_block, round_L));
    else {
        cands.push_back(round_L);
        for (int kb = 65536; kb >= 1024; kb /= 2)
            if (kb < round_L)
                cands.push_back(kb);
    }
    int best_kb = 0, best_rc = 0;
    int64_t best_passes = INT64_MAX;
    for (int kb : cands) {
        const size_t fixed = layout(*p, kb, 0);
        if (fixed >= p->budget)
            continue;
        const int64_t rows = (int64_t)((p->budget - fixed) / ((size_t)kb * 4));
        const int64_t rc = rows >= p->T ? std::max(p->T, 1) : rows / G * G;
        if (rc < 1)
            continue;
        int64_t passes = 0;
        for (int r = 0; r < R; ++r)
            passes += (p->row_begin[r + 1] - p->row_begin[r] + rc - 1) / rc * p->n_splits[r];
        if (passes < best_passes || (passes == best_passes && kb <= 65536 && kb > best_kb)) {
            best_passes = passes;
            best_kb = kb;
            best_rc = (int)rc;
        }
    }
    if (best_kb == 0) {
        delete p;
        return IDX_ERR_WORKSPACE;
    }
    layout(*p, best_kb, best_rc);
    *out = p;
    if (ws_bytes)
        *ws_bytes = p->ws_bytes;
    return IDX_OK;
}

void indexer_plan_destroy(indexer_plan_t p) { delete p; }

int indexer_plan_info(indexer_plan_t p, int32_t* key_block, int32_t* row_chunk,
                      int32_t* max_splits)
{
    if (!p)
        return IDX_ERR_INVALID_ARG;
    if (key_block)
        *key_block = p->key_block;
    if (row_chunk)
        *row_chunk = p->row_chunk;
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
    int rc = check_common(p, ws, ws_bytes);
    if (rc != IDX_OK)
        return rc;
    if ((rc = check_inputs(p, q, s_q, w, k, k_scale, clen)) != IDX_OK)
        return rc;
    if (!logits || !aligned(logits, 4) || ld < std::max(p->max_L, 1) || ld > INT32_MAX)
        return IDX_ERR_INVALID_ARG;
    Ctx c;
    if ((rc = begin_call(c, p, ws, stream)) != IDX_OK)
        return rc;
    if (p->T == 0)
        return IDX_OK;
    if ((rc = fill_maps(c, q, k)) != IDX_OK)
        return rc;
    set_inputs(c, s_q, w, k_scale, clen, ws);
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
        s.out_offset = (int64_t)rb * ld;
        s.out_ld = ld;
        segs.push_back(s);
        if ((int)segs.size() == kMaxSegments) {
            if ((rc = run_logits(c, segs, logits)) != IDX_OK)
                return rc;
            segs.clear();
        }
    }
    return segs.empty() ? IDX_OK : run_logits(c, segs, logits);
}

int indexer_topk(indexer_plan_t p, const float* logits, int64_t ld, const int32_t* clen,
                 int32_t* out_idx, float* out_val, void* ws, size_t ws_bytes, void* stream)
{
    int rc = check_common(p, ws, ws_bytes);
    if (rc != IDX_OK)
        return rc;
    if (!logits || !clen || !out_idx || ld < std::max(p->max_L, 1) || !aligned(logits, 4) ||
        !aligned(out_idx, 4) || (out_val && !aligned(out_val, 4)))
        return IDX_ERR_INVALID_ARG;
    Ctx c;
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
    g_launches.fetch_add(1, std::memory_order_relaxed);
    return launch_topk_dense(tp, c.st) == cudaSuccess ? IDX_OK : IDX_ERR_CUDA;
}

int indexer_fused_topk(indexer_plan_t p, const void* q, const float* s_q, const float* w,
                       const void* k, const void* k_scale, const int32_t* clen,
                       const uint8_t* cand_mask, int64_t ld_mask, int32_t* out_idx,
                       float* out_val, void* ws, size_t ws_bytes, void* stream)
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
    if ((rc = fill_maps(c, q, k)) != IDX_OK)
        return rc;
    set_inputs(c, s_q, w, k_scale, clen, ws);
    c.lp.cand_mask = cand_mask;
    c.lp.ld_mask = ld_mask;
    uint8_t* wsb = static_cast<uint8_t*>(ws);
    if ((rc = run_blocked(c, wsb, 0)) != IDX_OK)
        return rc;
    return run_merge(c, wsb, 0, out_idx, out_val, nullptr, 0);
}

int indexer_candidate_blocks(indexer_plan_t p, const void* q, const float* s_q, const float* w,
                             const void* k, const void* k_scale, const int32_t* clen,
                             uint8_t* cand_mask, int64_t ld_mask, void* ws, size_t ws_bytes,
                             void* stream)
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
    if ((rc = begin_call(c, p, ws, stream)) != IDX_OK)
        return rc;
    if (p->T == 0)
        return IDX_OK;
    if ((rc = fill_maps(c, q, k)) != IDX_OK)
        return rc;
    set_inputs(c, s_q, w, k_scale, clen, ws);
    uint8_t* wsb = static_cast<uint8_t*>(ws);
    if ((rc = run_blocked(c, wsb, p->cand_block)) != IDX_OK)
        return rc;
    return run_merge(c, wsb, p->cand_block, nullptr, nullptr, cand_mask, ld_mask);
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
