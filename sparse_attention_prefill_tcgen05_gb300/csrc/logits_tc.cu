// Indexer logits on the 5th-generation tensor cores (sm_103a), with the
// selection fused into the epilogue.
//
//   logit[t, j] = s_k[j] * sum_h c[t,h] * max(S[t,h,j], 0),   c = w * s_q,
//   S[t,h,j]    = <q[t,h,:], k[j,:]>  (fp8 e4m3 x fp8 e4m3, fp32 accumulate)
//
// which equals sum_h w * ReLU(s_q * s_k * S) because the scales are
// positive ("[DeepSeek-V4.1] Bound the dense prefill indexer transient",
// Motivation: the DeepGEMM fp8 MQA logits the indexer scores with;
// "chunked-prefill-memory.md" section 1: T query rows against the whole
// compressed prefix, -inf past the row's causal length).
//
// Mapping.  One MMA tile is M = 128 keys (TMEM lanes) x N = (rows x H heads)
// columns x K = D.  The head reduction of one (row, key) is a run of H
// accumulator columns on one TMEM lane.
//
// Roles (one CTA per SM, persistent over work units; 640 threads for the list
// sinks, 384 for plain logits):
//   warp 0       TMA producer: the unit's Q tile (double-buffered) and a ring
//                of K tiles, 128-byte-swizzled for the MMA.
//   warp 1       allocates 512 TMEM columns (two accumulators), issues
//                tcgen05.mma (D/32 per tile) and tcgen05.commit.
//   warps 4..    epilogue: four (list sinks) or two (logits) column parts x
//                four TMEM lane quadrants.  A warp reads its 32 keys x its
//                part's columns with tcgen05.ld 16x256b,
//                which gives thread (g, q) columns 2q and 2q+1 of every 8-column
//                group for two keys, so its head weights stay in registers; the
//                head sums are finished by a shuffle reduce-scatter over the four
//                q lanes of a key.  Then key scale, causal and candidate masks,
//                and one of four sinks:
//   * kSinkLogits: fp32 store of the [rows, ld] logits (also used, with a key
//     tile stride, for the sampled keys of the fused top-k);
//   * kSinkFilter: append every entry at or above the row's fixed threshold to
//     the warp's sub-list of its (row, key split), its position from a
//     shared-memory counter; the merge checks that the lists decide the row;
//   * kSinkStream: streamed exact top-k ("chunked-prefill-memory.md" section
//     2.3 scores key blocks and keeps per-block top-k; here the block top-k is
//     kept on the fly).  A key is appended to its row's list only if it is at
//     or above the row's threshold tau.  tau is always a valid lower bound of
//     the row's k-th best (composite) score: it comes from a two-level
//     histogram of the appended scores (256 bins of the top byte of the
//     order-preserving image, then 256 bins of the next byte inside the
//     boundary bin), from an exact compaction of the list when it fills, and
//     from the other key splits of the same row through a per-row atomic max
//     in global memory.  Nothing that can be in the row's top-k is ever
//     skipped, so the exact selection over the lists (select.cu) equals the
//     top-k over all keys.
//   * kSinkPool: the same over the maximum of each cand_block-key block
//     (candidate blocks, same section: 8-key block pooling, top-2048 blocks);
//   * kSinkPoolFilter: kSinkFilter over those block maxima.
// The accumulator is double-buffered so the epilogue of tile i overlaps the
// MMAs of tile i+1, and it is handed back as soon as its last column is in
// registers.
#include "groupsel.cuh"
#include "internal.h"

namespace idx {
namespace {

constexpr int kHalfThreads = 128;

// Operand kinds of the contraction.
constexpr int kOpsE4M3 = 0;   // e4m3 keys x e4m3 queries, kind::f8f6f4
constexpr int kOpsE2M1K = 1;  // e2m1 keys x e4m3 queries, kind::mxf8f6f4 (ue8m0 key scales)
constexpr int kOpsE2M1 = 2;   // e2m1 keys x e2m1 queries, kind::mxf4 (ue8m0 scales on both)

// e2m1 keys (one ue8m0 scale per 32 elements) are scored by the block-scaled MMA.  Their
// tiles are 192 columns (6 rows of 32 heads): two accumulators of 192 columns and the
// scale factors fit the 512 TMEM columns (24 columns of key scales, one 4-column group
// per K stage, then the query scales: 8 columns of 2^0 for e4m3 queries, two buffers of 8
// for e2m1 queries, one per Q tile buffer).  e2m1 queries take the fp4 kind: both
// operands stay packed in shared memory (64-byte rows for D = 128), K = 64 per MMA.
template <int H, int D, int SINK, int OPS = kOpsE4M3>
struct Cfg {
    static constexpr bool FP4K = OPS != kOpsE4M3;   // e2m1 keys
    static constexpr bool FP4Q = OPS == kOpsE2M1;   // e2m1 queries too
    // tiles are 256 columns (16 rows for small H; 192 for e2m1 keys)
    static constexpr int NMAX = FP4K ? 192 : (H >= 16 ? kTileN : 16 * H);
    static constexpr int G = NMAX / H;                 // query rows per tile
    static constexpr int N = G * H;                    // MMA N
    static constexpr int QROW = FP4Q ? D / 2 : D;      // bytes of a Q row in shared memory
    // bytes of a K row in shared memory: e2m1 keys of the f8f6f4 kinds are unpacked into
    // 16-byte groups of 16 codes on the way in; the fp4 kind reads them packed
    static constexpr int KROW = FP4Q ? D / 2 : D;
    static constexpr int QBYTES = N * QROW;            // Q tile: N rows
    static constexpr int KBYTES = kTileKeys * KROW;    // K tile in shared memory
    // bytes a K tile's TMA load counts on its barrier: the packed bytes it reads
    static constexpr int KTX = (FP4K && !FP4Q) ? KBYTES / 2 : KBYTES;
    static constexpr int STAGES = (D >= 128) ? 6 : 8;
    static constexpr int KSTEPS = D / (FP4Q ? 64 : 32);   // MMA K = 32 elements (64 for fp4)
    // epilogue warps: 16 for the list sinks (their per-tile selection work needs the
    // latency hiding), 8 for plain logits (fewer instructions per tile, 168 registers)
    static constexpr int EPI = FP4K ? 12 : (SINK == kSinkLogits ? 8 : 16);
    static constexpr int THREADS = 128 + 32 * EPI;
    static constexpr int NPART = EPI / 4;              // column parts (4 warps each)
    static constexpr int RPH = G / NPART;              // rows of one column part
    static constexpr int HALF_COLS = N / NPART;        // columns of one column part
    static constexpr int NCH = HALF_COLS / 32;         // 32-column chunks per part
    static constexpr int ACC_COLS = N;                 // TMEM columns per accumulator
    static constexpr bool STREAM = SINK != kSinkLogits;
    static_assert(D == 32 || D == 64 || D == 128, "D must be 32, 64 or 128");
    static_assert(G >= 2 && N % 16 == 0, "H must leave at least two rows per tile");
    static_assert(G % NPART == 0 && HALF_COLS % 32 == 0,
                  "a column part must be whole rows and whole 32-column loads");
    static_assert(H >= 8 && (RPH == 1 || RPH == 2 || RPH == 4 || RPH == 8),
                  "the epilogue's head split needs 8..64 heads");
    static_assert(!STREAM || G <= 16, "streamed selection keeps at most 16 rows per CTA");
    static_assert(!FP4K || (H == 32 && D == 128), "e2m1 keys: 32 heads of 128");
    // TMEM columns of the scale factors (after the two accumulators)
    static constexpr int SFA_COL = 2 * ACC_COLS;            // + 4 per K stage
    static constexpr int SFB_COL = SFA_COL + 4 * STAGES;    // 8 columns
    static constexpr int SFB_COLS = FP4Q ? 16 : 8;
    static_assert(!FP4K || SFB_COL + SFB_COLS <= 512, "scale factors must fit the allocation");
    // shared memory carve-up (offsets from a 1024-byte aligned base)
    static constexpr int OFF_Q = 0;
    static constexpr int OFF_K = OFF_Q + ((2 * QBYTES + 1023) / 1024) * 1024;
    // e2m1 keys: per K stage the tile's key scale words, 16 bytes per key (the layout
    // tcgen05.cp 128x128b reads)
    static constexpr int OFF_SF = OFF_K + STAGES * KBYTES;
    static constexpr int SF_BYTES = FP4K ? kTileKeys * 16 : 0;
    // e2m1 queries: per Q buffer the tile's query scale words as two 128-row x 16-byte
    // sources of tcgen05.cp 128x128b (row 32 quadrant + m, word i of copy j: query column
    // 32 (4 j + i) + m, the same in every quadrant)
    static constexpr int OFF_QSF = OFF_SF + STAGES * SF_BYTES;
    static constexpr int QSF_ONE = 2 * kTileKeys * 16;
    static constexpr int QSF_BYTES = FP4Q ? 2 * QSF_ONE : 0;
    static constexpr int OFF_C = OFF_QSF + QSF_BYTES;               // float c[2][kTileN]
    static constexpr int OFF_HIST = OFF_C + 2 * kTileN * 4;          // u32 [G][2][256]
    static constexpr int HIST_BYTES = STREAM ? G * 2 * 256 * 4 : 0;
    static constexpr int OFF_ROWS = OFF_HIST + HIST_BYTES;           // row state [G]
    static constexpr int ROWS_BYTES = STREAM ? G * 32 : 0;
    static constexpr int OFF_SEL = OFF_ROWS + ROWS_BYTES;            // compaction scratch x2
    static constexpr int SEL_ONE = (int)((sizeof(SelScratch<kHalfThreads>) + 15) / 16 * 16);
    static constexpr int SEL_BYTES = STREAM ? NPART * SEL_ONE : 0;
    static constexpr int OFF_BAR = OFF_SEL + SEL_BYTES;
    static constexpr int NBARS = 2 + 2 + 2 * STAGES + 2 + 2 + 1;
    static constexpr int OFF_MISC = OFF_BAR + NBARS * 8;
    static constexpr int SMEM = OFF_MISC + 16 + 1024;              // + alignment slack
};

// Per-row state of the streamed selection (shared memory, one per row of the group).
struct RowState {
    uint32_t wcnt[4];  // entries each epilogue warp of the row's column part appended (the
                       // fixed-threshold sinks count here directly; the streams publish
                       // their register counts here at each refresh)
    uint32_t tau_hi;   // candidate iff (ord(score), ~index) >= (tau_hi, tau_lo)
    uint32_t tau_lo;
    uint32_t b1;       // boundary bin of the top-byte histogram (256 = none yet)
    uint32_t compact;  // set by the threshold refresh: the lists must be compacted
};

struct UnitInfo {
    int seg;
    int t0;        // first global row of the row group
    int nr;        // valid rows in the group
    int j0;        // request-local first key of the unit
    int col0;      // output column of the unit's first key (sampled segments)
    int step;      // keys between consecutive tiles (tile_stride * 128)
    int jend;      // request-local end of keys covered by the unit
    int ntiles;    // tiles covering [j0, jend)
    int ntiles_mma;
    bool skip;     // second pass: no row of the group needs it
};

// Decode a unit number.  Units run chunk-major inside a segment so that the
// CTAs running at the same time share key tiles through L2.
template <int G>
__device__ __forceinline__ UnitInfo decode_unit(const LogitsParams& p, int u, int lane)
{
    UnitInfo ui;
    int s = 0;
    while (s + 1 < p.num_segments && p.seg[s + 1].unit_begin <= u)
        ++s;
    const Segment& sg = p.seg[s];
    const int local = u - sg.unit_begin;
    const int chunk = local / sg.n_row_groups;
    const int g = local - chunk * sg.n_row_groups;
    const int step = (sg.tile_stride > 0 ? sg.tile_stride : 1) * kTileKeys;   // tile to tile
    ui.skip = false;
    ui.seg = s;
    ui.t0 = sg.row_begin + g * G;
    ui.nr = min(G, sg.row_begin + sg.nrows - ui.t0);
    ui.j0 = sg.j_begin + chunk * sg.unit_tiles * step;
    ui.col0 = chunk * sg.unit_tiles * kTileKeys;
    ui.step = step;
    ui.jend = min(sg.j_end, ui.j0 + sg.unit_tiles * step);
    ui.ntiles = (ui.jend - ui.j0 + step - 1) / step;
    // longest causal length in the group (warp-cooperative), clamped to the request
    int m = 0;
    for (int r = lane; r < ui.nr; r += 32)
        m = max(m, min(p.compress_len[ui.t0 + r], sg.key_count));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
    const int mma_end = min(ui.jend, m);
    ui.ntiles_mma = mma_end > ui.j0 ? (mma_end - ui.j0 + step - 1) / step : 0;
    if (p.row_fail != nullptr) {
        // second pass over the rows the first one could not decide: other row
        // groups have no work
        bool any = false;
        for (int r = lane; r < ui.nr; r += 32)
            any |= p.row_fail[ui.t0 + r] != 0;
        if (!__any_sync(0xffffffffu, any)) {
            ui.ntiles = 0;
            ui.ntiles_mma = 0;
            ui.skip = true;
        }
    }
    return ui;
}

__device__ __forceinline__ void report(const LogitsParams& p, volatile int* abort_flag,
                                       uint32_t bits)
{
    *abort_flag = 1;
    atomicOr(p.status, bits);
}

__device__ __forceinline__ void red_add_shared(uint32_t* addr, uint32_t v)
{
    asm volatile("red.shared.add.u32 [%0], %1;" ::"r"(smem_u32(addr)), "r"(v) : "memory");
}

// Append this warp's threshold-passing entries of one row to the warp's own
// sub-list and count them in the row's histograms.  The lanes set in
// `rowmask` hold entries of this row (other lanes hold other rows); the
// append position comes from the warp-uniform count `wcnt` and a ballot
// prefix, so no atomics touch the list.  Histogram counts are fire-and-forget
// shared reductions: h2 counts the second byte of entries whose top byte is
// the boundary bin b1, h1 counts the top byte of all other entries.  Returns
// the new count.
__device__ __forceinline__ uint32_t stream_push(uint32_t* h1, uint32_t* h2, uint2* sub,
                                                uint32_t cap, uint32_t wcnt, uint32_t tau_hi,
                                                uint32_t tau_lo, uint32_t b1, float v,
                                                uint32_t idx, bool active, uint32_t rowmask,
                                                int lane)
{
    const uint32_t o = f2ord(v);
    const bool cand =
        active && o > kOrdNegInf && (o > tau_hi || (o == tau_hi && ~idx >= tau_lo));
    const uint32_t m = __ballot_sync(0xffffffffu, cand) & rowmask;
    if (cand) {
        const uint32_t pos = wcnt + __popc(m & ((1u << lane) - 1u));
        if (pos < cap)
            sub[pos] = make_uint2(__float_as_uint(v), idx);
        const uint32_t t8 = o >> 24;
        if (t8 == b1)
            red_add_shared(&h2[(o >> 16) & 255u], 1u);
        else
            red_add_shared(&h1[t8], 1u);
    }
    return wcnt + __popc(m);
}

// Suffix-count search over 256 bins held 8 per lane (lane L: bins 8L..8L+7),
// with add_val added to bin add_bin: the highest bin b with sum(bins >= b) >=
// need.  Returns 256 if the total is below need; *above gets sum(bins > b).
// Warp-wide.
__device__ __forceinline__ uint32_t boundary_bin(const uint32_t* hist, uint32_t need, int lane,
                                                 uint32_t* above, uint32_t add_bin = 256u,
                                                 uint32_t add_val = 0u)
{
    const uint4 a = reinterpret_cast<const uint4*>(hist)[lane * 2];
    const uint4 b = reinterpret_cast<const uint4*>(hist)[lane * 2 + 1];
    uint32_t c[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
    for (int i = 0; i < 8; ++i)
        if (static_cast<uint32_t>(lane * 8 + i) == add_bin)
            c[i] += add_val;
    uint32_t lsum = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i)
        lsum += c[i];
    uint32_t incl = lsum;  // sum over lanes >= this lane
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const uint32_t y = __shfl_down_sync(0xffffffffu, incl, off);
        if (lane + off < 32)
            incl += y;
    }
    const uint32_t hit = __ballot_sync(0xffffffffu, incl >= need);
    if (hit == 0) {
        *above = 0;
        return 256u;
    }
    const int bl = 31 - __clz(hit);
    uint32_t bin = 0, abv = 0;
    if (lane == bl) {
        uint32_t cum = incl - lsum;
        for (int i = 7; i >= 0; --i) {
            if (cum + c[i] >= need) {
                bin = static_cast<uint32_t>(bl * 8 + i);
                abv = cum;
                break;
            }
            cum += c[i];
        }
    }
    *above = __shfl_sync(0xffffffffu, abv, bl);
    return __shfl_sync(0xffffffffu, bin, bl);
}

__device__ __forceinline__ uint32_t warp_sum_bins(const uint32_t* hist, int lane)
{
    const uint4 a = reinterpret_cast<const uint4*>(hist)[lane * 2];
    const uint4 b = reinterpret_cast<const uint4*>(hist)[lane * 2 + 1];
    uint32_t s = a.x + a.y + a.z + a.w + b.x + b.y + b.z + b.w;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        s += __shfl_xor_sync(0xffffffffu, s, o);
    return s;
}

// MASK: the launch applies a candidate-block mask (a separate instantiation, so that
// the unmasked kernels carry none of its registers).
template <int H, int D, int SINK, bool MASK, int OPS>
__global__ void __launch_bounds__(Cfg<H, D, SINK, OPS>::THREADS, 1)
    logits_tc_kernel(const __grid_constant__ LogitsParams p)
{
    pdl_wait_then_release();
    using C = Cfg<H, D, SINK, OPS>;
    constexpr bool FP4K = C::FP4K;
    constexpr bool FP4Q = C::FP4Q;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* q_s = smem + C::OFF_Q;
    uint8_t* k_s = smem + C::OFF_K;
    uint8_t* sf_s = smem + C::OFF_SF;
    uint8_t* qsf_s = smem + C::OFF_QSF;
    float* c_s = reinterpret_cast<float*>(smem + C::OFF_C);
    uint32_t* hist_s = reinterpret_cast<uint32_t*>(smem + C::OFF_HIST);
    RowState* rows_s = reinterpret_cast<RowState*>(smem + C::OFF_ROWS);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
    uint64_t* q_full = bars;
    uint64_t* q_empty = bars + 2;
    uint64_t* k_full = bars + 4;
    uint64_t* k_empty = k_full + C::STAGES;
    uint64_t* a_full = k_empty + C::STAGES;
    uint64_t* a_empty = a_full + 2;
    uint64_t* drain = a_empty + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // a second pass with no flagged row anywhere has nothing to do (the flag was
    // written by an earlier launch, so every thread reads the same value)
    if (p.fail_any != nullptr && *p.fail_any == 0u)
        return;

    if (threadIdx.x == 0) {
        for (int i = 0; i < 2; ++i) {
            // e2m1 queries: one arrival with the TMA bytes, one when the scales are staged
            mbar_init(&q_full[i], FP4Q ? 2 : 1);
            mbar_init(&q_empty[i], 1);
            mbar_init(&a_full[i], 1);
            mbar_init(&a_empty[i], C::EPI);
        }
        for (int i = 0; i < C::STAGES; ++i) {
            // e2m1 keys: one arrival with the TMA bytes, one when the scales are staged
            mbar_init(&k_full[i], FP4K ? 2 : 1);
            mbar_init(&k_empty[i], 1);
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&p.tmap_q);
        tma_prefetch_desc(&p.tmap_k);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const long long budget = p.timeout_cycles;
    if constexpr (FP4K && !FP4Q) {
        // e4m3 queries carry no block scale: every query scale cell holds 2^0 (ue8m0 127)
        // in all four bytes, in every lane quadrant (each quadrant reads its own copy)
        if (warp >= 4 && warp < 8) {
            tmem_st_32x32b_x8_fill(tmem_base + (static_cast<uint32_t>((warp & 3) * 32) << 16) +
                                       C::SFB_COL,
                                   0x7F7F7F7Fu);
            tmem_wait_st();
        }
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
    }
    if (warp == 0) {
        // ------------------------------------------------------ TMA producer
        int issued[C::STAGES];
        int q_issued[2] = {0, 0};
        for (int i = 0; i < C::STAGES; ++i)
            issued[i] = 0;
        int ks = 0, kph = 0, qb = 0, qph = 0;
        bool ok = true;
        for (int u = blockIdx.x; u < p.total_units && ok; u += gridDim.x) {
            const UnitInfo ui = decode_unit<C::G>(p, u, lane);
            if (ui.ntiles_mma == 0)
                continue;
            const Segment sg = p.seg[ui.seg];   // by value: loop-invariant registers
            if (lane == 0) {
                if (!mbar_wait(&q_empty[qb], qph ^ 1, budget, abort_flag)) {
                    report(p, abort_flag, kStatusTimeout);
                    ok = false;
                } else {
                    mbar_arrive_expect_tx(&q_full[qb], C::QBYTES);
                    tma_load_2d(q_s + qb * C::QBYTES, &p.tmap_q, &q_full[qb], 0, ui.t0 * H);
                    ++q_issued[qb];
                }
            }
            ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
            if constexpr (FP4Q) {
                if (ok) {
                    // the tile's query scale words (four ue8m0 bytes of query column n = row
                    // x H + head) into the buffer's two copy sources; columns of rows past
                    // the group and past N read as 2^0.  The previous unit on this buffer
                    // finished its MMAs (q_empty), and with them the copies that read it.
                    uint32_t wv[8];
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        const int n = 32 * c + lane;
                        wv[c] = (n < C::N && n / H < ui.nr)
                                    ? __ldg(p.q_sf + (size_t)ui.t0 * H + n)
                                    : 0x7F7F7F7Fu;
                    }
                    uint8_t* dst = qsf_s + qb * C::QSF_ONE;
#pragma unroll
                    for (int j = 0; j < 2; ++j)
#pragma unroll
                        for (int quad4 = 0; quad4 < 4; ++quad4)
                            *reinterpret_cast<uint4*>(dst + j * (C::QSF_ONE / 2) +
                                                      16 * (32 * quad4 + lane)) =
                                make_uint4(wv[4 * j], wv[4 * j + 1], wv[4 * j + 2], wv[4 * j + 3]);
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0)
                        mbar_arrive(&q_full[qb]);
                }
            }
            for (int i = 0; i < ui.ntiles_mma && ok; ++i) {
                const int key0 = sg.key_base + ui.j0 + i * ui.step;
                if (lane == 0) {
                    if (!mbar_wait(&k_empty[ks], kph ^ 1, budget, abort_flag)) {
                        report(p, abort_flag, kStatusTimeout);
                        ok = false;
                    } else {
                        mbar_arrive_expect_tx(&k_full[ks], C::KTX);
                        tma_load_2d(k_s + ks * C::KBYTES, &p.tmap_k, &k_full[ks], 0, key0);
                        ++issued[ks];
                    }
                }
                ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
                if (!ok)
                    break;
                if constexpr (FP4K) {
                    // the tile's key scale words (four ue8m0 bytes, one per 32-element
                    // block) into the stage's scale area: key r at byte 16 r + 4 (r / 32),
                    // so that the 128x128b copy puts it in TMEM lane r, column r / 32 of
                    // the stage's four columns, the cell the block-scaled MMA reads for
                    // row r; keys past the request read as 2^0 (they are masked anyway).
                    // The previous MMAs of this stage finished (k_empty), and with them
                    // the copy that read the area.
                    uint8_t* sf = sf_s + ks * C::SF_BYTES;
#pragma unroll
                    for (int r0 = 0; r0 < kTileKeys; r0 += 32) {
                        const int r = r0 + lane;
                        const int local = ui.j0 + i * ui.step + r;
                        const uint32_t word =
                            local < sg.key_count ? __ldg(p.k_sf + key0 + r) : 0x7F7F7F7Fu;
                        *reinterpret_cast<uint32_t*>(sf + 16 * r + 4 * (r0 / 32)) = word;
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0)
                        mbar_arrive(&k_full[ks]);
                }
                if (++ks == C::STAGES) {
                    ks = 0;
                    kph ^= 1;
                }
            }
            if (++qb == 2) {
                qb = 0;
                qph ^= 1;
            }
        }
        // make sure no copy is still landing in shared memory when the CTA exits
        if (lane == 0) {
            volatile int no_abort = 0;
            for (int i = 0; i < C::STAGES; ++i)
                if (issued[i] > 0)
                    mbar_wait(&k_full[i], (issued[i] - 1) & 1, budget, &no_abort);
            for (int i = 0; i < 2; ++i)
                if (q_issued[i] > 0)
                    mbar_wait(&q_full[i], (q_issued[i] - 1) & 1, budget, &no_abort);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------- MMA issuer
        constexpr uint32_t idesc = idesc_f8f6f4(kTileKeys, C::N, 0, 0);
        int ks = 0, kph = 0, qb = 0, qph = 0, ab = 0, aph = 0;
        bool ok = true;
        bool any = false;
        for (int u = blockIdx.x; u < p.total_units && ok; u += gridDim.x) {
            const UnitInfo ui = decode_unit<C::G>(p, u, lane);
            if (ui.ntiles_mma == 0)
                continue;
            if (lane == 0) {
                if (!mbar_wait(&q_full[qb], qph, budget, abort_flag)) {
                    report(p, abort_flag, kStatusTimeout);
                    ok = false;
                }
                [[maybe_unused]] const uint32_t sfb = tmem_base + C::SFB_COL + (FP4Q ? 8 * qb : 0);
                if constexpr (FP4Q) {
                    // the unit's query scales into this Q buffer's 8 scale columns
                    if (ok) {
                        tc_fence_after();
                        const uint32_t src = smem_u32(qsf_s + qb * C::QSF_ONE);
                        tmem_cp_128x128b(sfb, smem_desc_noswizzle(src, 128));
                        tmem_cp_128x128b(sfb + 4, smem_desc_noswizzle(src + C::QSF_ONE / 2, 128));
                    }
                }
                const uint32_t q_addr = smem_u32(q_s + qb * C::QBYTES);
                for (int i = 0; i < ui.ntiles_mma && ok; ++i) {
                    if (!mbar_wait(&a_empty[ab], aph ^ 1, budget, abort_flag) ||
                        !mbar_wait(&k_full[ks], kph, budget, abort_flag)) {
                        report(p, abort_flag, kStatusTimeout);
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t k_addr = smem_u32(k_s + ks * C::KBYTES);
                    const uint32_t d_tmem = tmem_base + ab * C::ACC_COLS;
                    if constexpr (FP4Q) {
                        // the stage's key scales into TMEM, then one fp4 MMA per two
                        // 32-element blocks (64 packed codes, 32 bytes of each row): scale
                        // bytes 2 kk and 2 kk + 1 of each cell
                        const uint32_t sfa = tmem_base + C::SFA_COL + 4 * ks;
                        tmem_cp_128x128b(sfa, smem_desc_noswizzle(smem_u32(sf_s + ks * C::SF_BYTES), 128));
#pragma unroll
                        for (int kk = 0; kk < C::KSTEPS; ++kk) {
                            const uint64_t adesc = smem_desc_kmajor(k_addr + kk * 32, C::KROW);
                            const uint64_t bdesc = smem_desc_kmajor(q_addr + kk * 32, C::QROW);
                            mma_mxf4(d_tmem, adesc, bdesc,
                                     idesc_mxf4(kTileKeys, C::N, 2 * kk, 2 * kk), sfa, sfb,
                                     kk > 0 ? 1u : 0u);
                        }
                    } else if constexpr (FP4K) {
                        // the stage's key scales into TMEM, then one block-scaled MMA per
                        // 32-element block (A = e2m1 keys, B = e4m3 queries); the scale
                        // byte of block kk is byte kk of each cell
                        const uint32_t sfa = tmem_base + C::SFA_COL + 4 * ks;
                        tmem_cp_128x128b(sfa, smem_desc_noswizzle(smem_u32(sf_s + ks * C::SF_BYTES), 128));
#pragma unroll
                        for (int kk = 0; kk < C::KSTEPS; ++kk) {
                            const uint64_t adesc = smem_desc_kmajor(k_addr + kk * 32, D);
                            const uint64_t bdesc = smem_desc_kmajor(q_addr + kk * 32, D);
                            mma_mxf8f6f4(d_tmem, adesc, bdesc,
                                         idesc_mxf8f6f4(kTileKeys, C::N, 5, 0, kk, kk), sfa,
                                         sfb, kk > 0 ? 1u : 0u);
                        }
                    } else {
#pragma unroll
                        for (int kk = 0; kk < C::KSTEPS; ++kk) {
                            const uint64_t adesc = smem_desc_kmajor(k_addr + kk * 32, D);
                            const uint64_t bdesc = smem_desc_kmajor(q_addr + kk * 32, D);
                            mma_f8f6f4(d_tmem, adesc, bdesc, idesc, kk > 0 ? 1u : 0u);
                        }
                    }
                    mma_commit(&k_empty[ks]);
                    mma_commit(&a_full[ab]);
                    any = true;
                    if (++ks == C::STAGES) {
                        ks = 0;
                        kph ^= 1;
                    }
                    if (++ab == 2) {
                        ab = 0;
                        aph ^= 1;
                    }
                }
                if (ok)
                    mma_commit(&q_empty[qb]);
            }
            ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
            if (++qb == 2) {
                qb = 0;
                qph ^= 1;
            }
        }
        // every MMA this thread issued has finished before TMEM is released
        if (lane == 0 && any) {
            volatile int no_abort = 0;
            mma_commit(drain);
            mbar_wait(drain, 0, budget, &no_abort);
        }
    } else if (warp >= 4) {
        // ---------------------------------------------------------- epilogue
        // Warp (half, quad) reduces TMEM lanes [32 quad, +32) (keys) x columns
        // [half * HALF_COLS, +HALF_COLS) (RPH rows x H heads).  It reads them with
        // the 16x256b shape: thread (g = lane / 4, q = lane % 4) gets, for each
        // 8-column group, columns 2q and 2q + 1 of the lanes g and g + 8 of a
        // 16-lane block.  Each thread therefore needs only 2 head weights per
        // group (one 8-byte shared load that four lanes share, instead of a
        // broadcast of every weight to all 32 lanes), and the head sums are
        // finished by a reduce-scatter over the four q lanes.
        const int ew = warp - 4;                 // 0..7
        const int quad = warp & 3;               // TMEM lane quadrant of this warp
        const int half = ew >> 2;                // column part: rows [half*RPH, +RPH)
        const int etid = ew * 32 + lane;         // 0..255
        const int htid = quad * 32 + lane;       // 0..127 within the column part
        const int g = lane >> 2;
        const int q = lane & 3;
        constexpr int RPH = C::RPH;
        constexpr int F = 4 * RPH;               // partial sums per thread per tile
        constexpr int RO = RPH >= 4 ? RPH / 4 : 1;   // rows a thread finishes
        constexpr int NK = RPH >= 4 ? 4 : RPH;       // key slots a thread finishes
        constexpr int NLD = 2 * C::NCH;          // 16-lane x 32-column loads per tile
        // finished value m: f = q * RPH + m = rr * 4 + slot-in-row, rr = f / 4
        auto own_rr = [&](int ro) { return RPH >= 4 ? q * (RPH / 4) + ro : (q * RPH) >> 2; };
        auto slot_bl = [&](int s) { return RPH >= 4 ? s : ((q * RPH + s) & 3); };
        // lanes that finish the same rows as this one
        const uint32_t rowmask = RPH >= 4   ? (0x11111111u << q)
                                 : RPH == 2 ? (0x33333333u << (q & 2))
                                            : 0xFFFFFFFFu;
        const bool row_leader = g == 0 && (RPH >= 4 || (q & (4 / RPH - 1)) == 0);
        [[maybe_unused]] const uint32_t lanes_below = (1u << lane) - 1u;
        const NamedSync half_sync{2 + half, kHalfThreads};
        const NamedSync epi_sync{1, C::EPI * 32};
        SelScratch<kHalfThreads>* sel_s =
            reinterpret_cast<SelScratch<kHalfThreads>*>(smem + C::OFF_SEL + half * C::SEL_ONE);
        int ab = 0, aph = 0, it = 0;
        bool alive = true;
        // Every epilogue warp walks every unit and every tile, also after a
        // timeout ("not alive": waits are skipped), so the named barriers always
        // see all of their threads.
        for (int u = blockIdx.x; u < p.total_units; u += gridDim.x, ++it) {
            const UnitInfo ui = decode_unit<C::G>(p, u, lane);
            const Segment sg = p.seg[ui.seg];   // by value: loop-invariant registers
            // head weights c[n] = w * s_q of column n = row * H + head; odd columns
            // carry 2^64 (their relu is a saturating multiply by 2^-64).  Double
            // buffered by unit: the other half may still read the previous one.
            float* cbuf = c_s + (it & 1) * kTileN;
            if (etid < C::N) {
                const int rl = etid / H;
                const size_t o = (size_t)(ui.t0 + rl) * H + (etid % H);
                // (e2m1 queries: their scales are inside the MMA)
                const float cv = rl < ui.nr ? (FP4Q ? p.w[o] : p.w[o] * p.s_q[o]) : 0.0f;
                cbuf[etid] = (etid & 1) ? cv * 18446744073709551616.0f : cv;
            }
            if constexpr (C::STREAM) {
                for (int i = etid; i < C::G * 512; i += C::EPI * 32)
                    hist_s[i] = 0;
                if (etid < C::G) {
                    RowState& rs = rows_s[etid];
                    for (int w4 = 0; w4 < 4; ++w4)
                        rs.wcnt[w4] = 0;
                    rs.tau_hi = etid < ui.nr ? p.gtau[ui.t0 + etid] : 0u;
                    rs.tau_lo = 0;
                    rs.b1 = 256;
                    rs.compact = 0;
                }
            }
            epi_sync();
            // this thread's head weights: columns 2q, 2q + 1 of every 8-column group
            float2 cw[C::NCH * 4];
#pragma unroll
            for (int gi = 0; gi < C::NCH * 4; ++gi)
                cw[gi] = reinterpret_cast<const float2*>(cbuf + half * C::HALF_COLS)[gi * 4 + q];
            // the rows this thread finishes
            int clen[RO];
            uint32_t tau_hi[RO], tau_lo[RO], b1[RO], wcnt[RO];
#pragma unroll
            for (int ro = 0; ro < RO; ++ro) {
                const int rl = half * RPH + own_rr(ro);
                clen[ro] = rl < ui.nr ? min(p.compress_len[ui.t0 + rl], sg.key_count) : 0;
                tau_hi[ro] = 0;
                tau_lo[ro] = 0;
                b1[ro] = 256;
                wcnt[ro] = 0;
                if constexpr (SINK == kSinkFilter || SINK == kSinkPoolFilter) {
                    // as a float: v >= it <=> ord(v) >= tau for every v but -0.0 against
                    // tau = ord(+0.0), which only lets -0.0 entries through as well (still
                    // every entry at or above a threshold); tau = 0 passes every finite v
                    // (a row past the group's end gets +inf: nothing of it is appended)
                    const uint32_t tr = rl < ui.nr ? p.tau_row[ui.t0 + rl] : 0u;
                    tau_hi[ro] = rl >= ui.nr         ? 0x7F800000u   // +inf
                                 : tr > kOrdNegInf ? __float_as_uint(ord2f(tr))
                                                   : 0xFF7FFFFFu;   // -FLT_MAX
                } else if constexpr (C::STREAM) {
                    tau_hi[ro] = rows_s[rl].tau_hi;
                    tau_lo[ro] = rows_s[rl].tau_lo;
                }
            }
            // this warp's sub-list of each row the thread finishes
            uint2* sub_own[RO];
#pragma unroll
            for (int ro = 0; ro < RO; ++ro) {
                const int rl = half * RPH + own_rr(ro);
                sub_own[ro] = p.lists + sg.out_offset +
                              (int64_t)(ui.t0 + rl - sg.row_begin) * sg.out_ld +
                              (int64_t)quad * sg.cap;
            }
            // smallest causal length among the half's rows (rows past nr are never
            // stored or selected)
            int clen_min = INT_MAX;
            for (int r = 0; r < RPH; ++r)
                if (half * RPH + r < ui.nr)
                    clen_min = min(clen_min, min(p.compress_len[ui.t0 + half * RPH + r],
                                                 sg.key_count));
            // the shared thresholds of the rows this warp refreshes, read one
            // refresh interval ahead of use
            constexpr int kOwned = (RPH + 3) / 4;
            uint32_t gpre[kOwned];
#pragma unroll
            for (int oi = 0; oi < kOwned; ++oi) {
                const int rl = half * RPH + quad + 4 * oi;
                gpre[oi] = 0;
                if (C::STREAM && quad + 4 * oi < RPH && rl < ui.nr)
                    gpre[oi] = ld_relaxed_gpu(p.gtau + ui.t0 + rl);
            }
            // key scale of key (quadrant base + lane), one tile ahead; the owners
            // of each key fetch it by a shuffle.  The index is clamped instead of
            // tested, so no instruction waits on the load before its use: keys at
            // or past key_count are masked to -inf whatever scale they get.
            const float* sk_row = p.s_k + sg.key_base;
            const int sk_last = max(sg.key_count - 1, 0);
            float sk_next = 1.0f;   // e2m1 keys: the scales are inside the MMA
            if (!FP4K && ui.ntiles_mma > 0)
                sk_next = __ldg(sk_row + min(ui.j0 + quad * 32 + lane, sk_last));
            // candidate-mask bytes of this thread's keys, one tile ahead like the key
            // scales (row and key indices clamped: a byte read for a key that the
            // causal test drops does not matter)
            constexpr bool has_mask = MASK;
            const int mshift = has_mask ? __ffs(p.mask_block) - 1 : 0;
            const uint8_t* mrow[RO];
#pragma unroll
            for (int ro = 0; ro < RO; ++ro) {
                mrow[ro] = nullptr;
                if constexpr (has_mask) {
                    // the row's mask row: itself, or its entry of the caller's row map
                    // (an entry outside the mask is reported and read as row 0)
                    const int t = ui.t0 + min(half * RPH + own_rr(ro), ui.nr - 1);
                    int64_t mr = t;
                    if (p.mask_rows != nullptr) {
                        mr = __ldg(p.mask_rows + t);
                        if (mr < 0 || mr >= p.mask_row_count) {
                            atomicOr(p.status, kStatusBadArg);
                            mr = 0;
                        }
                    }
                    mrow[ro] = p.cand_mask + mr * p.ld_mask;
                }
            }
            auto mask_at = [&](int m, int jt0) -> uint32_t {
                const int ro = RPH >= 4 ? (m >> 2) : 0;
                const int j = min(jt0 + 8 * slot_bl(RPH >= 4 ? (m & 3) : m) + g, sk_last);
                return __ldg(mrow[ro] + (j >> mshift));
            };
            uint32_t mk_next[RPH];
#pragma unroll
            for (int m = 0; m < RPH; ++m)
                mk_next[m] = (has_mask && ui.ntiles_mma > 0) ? mask_at(m, ui.j0 + quad * 32) : 1u;
            // a warp's sub-list sees 32 of every 128 keys (or its lanes' blocks)
            const int unit_entries_warp =
                (SINK == kSinkPool || SINK == kSinkPoolFilter)
                    ? ui.ntiles * (32 / (p.pool > 0 ? p.pool : 1))
                    : ui.ntiles * 32;
            const bool no_overflow = unit_entries_warp <= sg.cap;
            for (int i = 0; i < ui.ntiles; ++i) {
                const int jt = ui.j0 + i * ui.step + quad * 32;   // first key of the quadrant
                float val[RPH];
                uint32_t mk_cur[RPH];
#pragma unroll
                for (int m = 0; m < RPH; ++m) {
                    val[m] = -INFINITY;
                    mk_cur[m] = 1u;
                }
                if (i < ui.ntiles_mma) {
                    const float sk_lane = sk_next;
                    if (!FP4K && i + 1 < ui.ntiles_mma)
                        sk_next = __ldg(sk_row + min(jt + ui.step + lane, sk_last));
                    if constexpr (has_mask) {
#pragma unroll
                        for (int m = 0; m < RPH; ++m)
                            mk_cur[m] = mk_next[m];
                        if (i + 1 < ui.ntiles_mma) {
#pragma unroll
                            for (int m = 0; m < RPH; ++m)
                                mk_next[m] = mask_at(m, jt + ui.step);
                        }
                    }
                    bool got = alive && mbar_wait(&a_full[ab], aph, budget, abort_flag);
                    got = __all_sync(0xffffffffu, got);
                    if (!got && alive) {
                        if (lane == 0)
                            report(p, abort_flag, kStatusTimeout);
                        alive = false;
                    }
                    if (got) {
                        tc_fence_after();
                        // partial sums [row][block][lane g or g+8], two heads per packed
                        // FMA: relu by max (ALU pipe) for column 2q, by a saturating
                        // multiply with 2^-64 (FMA pipe) for column 2q + 1, whose weight
                        // carries 2^64; every product and sum is bit-identical to
                        // fmaf(c, max(S, 0), part).
                        // (the list sinks start every accumulator with the first product of
                        // its chunk, equal to fmaf(c, max(S, 0), 0) up to the sign of a zero;
                        // the dense-logits sink, with registers to spare, starts from zero)
                        constexpr bool kMulFirst = SINK != kSinkLogits;
                        float2 acc2[RPH][2][2];
                        if constexpr (!kMulFirst) {
#pragma unroll
                            for (int r = 0; r < RPH; ++r)
#pragma unroll
                                for (int b2 = 0; b2 < 2; ++b2) {
                                    acc2[r][b2][0] = make_float2(0.0f, 0.0f);
                                    acc2[r][b2][1] = make_float2(0.0f, 0.0f);
                                }
                        }
                        const uint32_t tbase = tmem_base +
                                               (static_cast<uint32_t>(quad * 32) << 16) +
                                               ab * C::ACC_COLS + half * C::HALF_COLS;
                        // load ld = (chunk, block): 16 lanes x 32 columns; the next one
                        // is in flight while the current one is reduced
                        float va[16], vb[16];
                        tmem_ld_16x256b_x4(tbase, va);
                        tmem_wait_ld();
#pragma unroll
                        for (int ld = 0; ld < NLD; ++ld) {
                            float(&cur)[16] = (ld & 1) ? vb : va;
                            float(&nxt)[16] = (ld & 1) ? va : vb;
                            if (ld + 1 < NLD) {
                                const int ch1 = (ld + 1) >> 1, b1n = (ld + 1) & 1;
                                tmem_ld_16x256b_x4(
                                    tbase + (static_cast<uint32_t>(16 * b1n) << 16) + ch1 * 32, nxt);
                            }
                            const int ch = ld >> 1, blk = ld & 1;
#pragma unroll
                            for (int k = 0; k < 4; ++k) {
                                const int r = (ch * 32 + 8 * k) / H;
                                const float2 c2 = cw[ch * 4 + k];
                                const float2 lo = make_float2(fmaxf(cur[4 * k + 0], 0.0f),
                                                              relu_scaled(cur[4 * k + 1]));
                                const float2 hi = make_float2(fmaxf(cur[4 * k + 2], 0.0f),
                                                              relu_scaled(cur[4 * k + 3]));
                                if (kMulFirst && (ch * 32 + 8 * k) % H == 0) {   // a row's first group
                                    acc2[r][blk][0] = __fmul2_rn(c2, lo);
                                    acc2[r][blk][1] = __fmul2_rn(c2, hi);
                                } else {
                                    acc2[r][blk][0] = __ffma2_rn(c2, lo, acc2[r][blk][0]);
                                    acc2[r][blk][1] = __ffma2_rn(c2, hi, acc2[r][blk][1]);
                                }
                            }
                            if (ld + 1 < NLD)
                                tmem_wait_ld();
                            if (ld + 2 == NLD) {
                                // every column of the accumulator is in registers: hand
                                // it back to the MMA before the last chunk's arithmetic
                                tc_fence_before();
                                __syncwarp();
                                if (lane == 0)
                                    mbar_arrive(&a_empty[ab]);
                            }
                        }
                        // reduce-scatter over the four q lanes: thread q keeps the
                        // sums f = q * RPH + m, f = row * 4 + block * 2 + (g or g+8)
                        float pf[F];
#pragma unroll
                        for (int r = 0; r < RPH; ++r)
#pragma unroll
                            for (int b2 = 0; b2 < 2; ++b2)
#pragma unroll
                                for (int l2 = 0; l2 < 2; ++l2)
                                    pf[r * 4 + b2 * 2 + l2] =
                                        acc2[r][b2][l2].x + acc2[r][b2][l2].y;
                        float rs1[F / 2];
#pragma unroll
                        for (int x = 0; x < F / 2; ++x) {
                            const float keep = (q & 2) ? pf[F / 2 + x] : pf[x];
                            const float send = (q & 2) ? pf[x] : pf[F / 2 + x];
                            rs1[x] = keep + __shfl_xor_sync(0xffffffffu, send, 2);
                        }
#pragma unroll
                        for (int x = 0; x < F / 4; ++x) {
                            const float keep = (q & 1) ? rs1[F / 4 + x] : rs1[x];
                            const float send = (q & 1) ? rs1[x] : rs1[F / 4 + x];
                            val[x] = keep + __shfl_xor_sync(0xffffffffu, send, 1);
                        }
#pragma unroll
                        for (int s2 = 0; s2 < NK; ++s2) {
                            const float skv =
                                __shfl_sync(0xffffffffu, sk_lane, 8 * slot_bl(s2) + g);
#pragma unroll
                            for (int x = s2; x < F / 4; x += NK)
                                val[x] *= skv;
                        }
                    }
                    if (++ab == 2) {
                        ab = 0;
                        aph ^= 1;
                    }
                }
                // causal and candidate masks (most tiles lie below every row's causal
                // length: one warp-uniform test skips the per-value work there); the
                // fixed-threshold sink tests a key's eligibility only for the few values
                // at or above the threshold, in its append branch below
                if (SINK != kSinkFilter &&
                    (has_mask || ui.j0 + i * ui.step + kTileKeys > clen_min)) {
#pragma unroll
                    for (int m = 0; m < RPH; ++m) {
                        const int ro = RPH >= 4 ? (m >> 2) : 0;
                        const int rl = half * RPH + own_rr(ro);
                        const int j = jt + 8 * slot_bl(RPH >= 4 ? (m & 3) : m) + g;
                        if (!(rl < ui.nr && j < clen[ro] && mk_cur[m] != 0u))
                            val[m] = -INFINITY;
                    }
                }
                if constexpr (SINK == kSinkLogits) {
                    // column of key j: (j - j_begin) for every tile, or the sample
                    // number for a sampled segment
                    float* out_base = p.out + sg.out_offset + ui.col0 + i * kTileKeys + quad * 32;
#pragma unroll
                    for (int m = 0; m < RPH; ++m) {
                        const int ro = RPH >= 4 ? (m >> 2) : 0;
                        const int rl = half * RPH + own_rr(ro);
                        const int kk = 8 * slot_bl(RPH >= 4 ? (m & 3) : m) + g;
                        if (rl < ui.nr && jt + kk < ui.jend)
                            out_base[(size_t)(ui.t0 + rl - sg.row_begin) * sg.out_ld + kk] =
                                val[m];
                    }
                } else if constexpr (SINK == kSinkFilter) {
                    // fixed threshold: append, no histograms, no refresh (a sub-list
                    // that overflows is detected by the merge from its count).  A
                    // candidate (about one value in twenty) takes its position from a
                    // shared-memory counter of the (row, warp) sub-list: no warp-wide
                    // ballot and prefix count for the other nineteen.
#pragma unroll
                    for (int m = 0; m < RPH; ++m) {
                        const int ro = RPH >= 4 ? (m >> 2) : 0;
                        const int rl = half * RPH + own_rr(ro);
                        const int j = jt + 8 * slot_bl(RPH >= 4 ? (m & 3) : m) + g;
                        if (val[m] >= __uint_as_float(tau_hi[ro]) && j < clen[ro] &&
                            (!has_mask || mk_cur[m] != 0u)) {
                            const uint32_t pos = atomicAdd(&rows_s[rl].wcnt[quad], 1u);
                            if (pos < static_cast<uint32_t>(sg.cap))
                                sub_own[ro][pos] =
                                    make_uint2(__float_as_uint(val[m]), static_cast<uint32_t>(j));
                        }
                    }
                } else if constexpr (SINK == kSinkPoolFilter) {
                    // the same over the maxima of cand_block-key blocks: the keys of a
                    // block are lanes g of one q (xor over the g bits), its first lane
                    // appends (block maximum, block index)
#pragma unroll
                    for (int m = 0; m < RPH; ++m) {
                        const int ro = RPH >= 4 ? (m >> 2) : 0;
                        const int rl = half * RPH + own_rr(ro);
                        const int j = jt + 8 * slot_bl(RPH >= 4 ? (m & 3) : m) + g;
                        float bm = val[m];
                        for (int o = 1; o < p.pool; o <<= 1)
                            bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 4 * o));
                        if ((g % p.pool) == 0 && bm >= __uint_as_float(tau_hi[ro])) {
                            const uint32_t pos = atomicAdd(&rows_s[rl].wcnt[quad], 1u);
                            if (pos < static_cast<uint32_t>(sg.cap))
                                sub_own[ro][pos] = make_uint2(__float_as_uint(bm),
                                                              static_cast<uint32_t>(j / p.pool));
                        }
                    }
                } else {
                    const uint32_t cap = static_cast<uint32_t>(sg.cap);
#pragma unroll
                    for (int m = 0; m < RPH; ++m) {
                        const int ro = RPH >= 4 ? (m >> 2) : 0;
                        const int rl = half * RPH + own_rr(ro);
                        const int j = jt + 8 * slot_bl(RPH >= 4 ? (m & 3) : m) + g;
                        uint32_t* h1 = hist_s + rl * 512;
                        uint2* sub = p.lists + sg.out_offset +
                                     (int64_t)(ui.t0 + rl - sg.row_begin) * sg.out_ld +
                                     (int64_t)quad * sg.cap;
                        if constexpr (SINK == kSinkStream) {
                            wcnt[ro] = stream_push(h1, h1 + 256, sub, cap, wcnt[ro], tau_hi[ro],
                                                   tau_lo[ro], b1[ro], val[m],
                                                   static_cast<uint32_t>(j), rl < ui.nr,
                                                   rowmask, lane);
                        } else {
                            // block maximum over `pool` consecutive keys: lanes g..
                            float bm = val[m];
                            for (int o = 1; o < p.pool; o <<= 1)
                                bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 4 * o));
                            const bool lead = (g % p.pool) == 0;
                            wcnt[ro] = stream_push(h1, h1 + 256, sub, cap, wcnt[ro], tau_hi[ro],
                                                   tau_lo[ro], b1[ro], bm,
                                                   static_cast<uint32_t>(j / p.pool),
                                                   lead && rl < ui.nr, rowmask, lane);
                        }
                    }
                    const bool refresh = ((i + 1) % p.update_tiles) == 0 || i + 1 == ui.ntiles;
                    if (refresh) {
                        // publish this warp's counts, then the row owners refresh tau
                        if (row_leader) {
#pragma unroll
                            for (int ro = 0; ro < RO; ++ro)
                                rows_s[half * RPH + own_rr(ro)].wcnt[quad] = wcnt[ro];
                        }
                        half_sync();
                        // rows of this half: warp `quad` refreshes rows quad, quad+4, ...
#pragma unroll
                        for (int oi = 0; oi < kOwned; ++oi) {
                            const int rr = quad + 4 * oi;
                            const int rl = half * RPH + rr;
                            if (rr >= RPH)
                                continue;
                            if (rl >= ui.nr)
                                continue;
                            RowState& rs = rows_s[rl];
                            uint32_t* h1 = hist_s + rl * 512;
                            uint32_t* h2 = h1 + 256;
                            const uint32_t keep = static_cast<uint32_t>(p.keep);
                            const uint32_t cur_b1 = rs.b1;
                            const uint32_t sum2 = cur_b1 < 256 ? warp_sum_bins(h2, lane) : 0u;
                            uint32_t above1 = 0, tau_new = 0;
                            const uint32_t bin1 =
                                boundary_bin(h1, keep, lane, &above1, cur_b1, sum2);
                            if (bin1 < 256) {
                                __syncwarp();
                                if (cur_b1 == 256 || bin1 > cur_b1) {
                                    for (int i2 = lane; i2 < 256; i2 += 32)
                                        h2[i2] = 0;
                                    __syncwarp();
                                    tau_new = bin1 << 24;
                                    if (lane == 0)
                                        rs.b1 = bin1;
                                } else {
                                    uint32_t above2 = 0;
                                    const uint32_t bin2 =
                                        boundary_bin(h2, keep - above1, lane, &above2);
                                    tau_new = (bin1 << 24) | (bin2 < 256 ? bin2 << 16 : 0u);
                                }
                            }
                            if (lane == 0) {
                                const int t = ui.t0 + rl;
                                const uint32_t gv = gpre[oi];
                                if (tau_new > gv)
                                    atomicMax(p.gtau + t, tau_new);
                                const uint32_t best = max(tau_new, gv);
                                if (best > rs.tau_hi) {
                                    rs.tau_hi = best;
                                    rs.tau_lo = 0;
                                }
                                // a sub-list must have room for the next refresh interval
                                const uint32_t slack =
                                    static_cast<uint32_t>(p.update_tiles) * 32u;
                                bool full = false, lost = false;
                                for (int w4 = 0; w4 < 4; ++w4) {
                                    full |= rs.wcnt[w4] + slack > cap;
                                    lost |= rs.wcnt[w4] > cap;
                                }
                                rs.compact = (full && !no_overflow) ? 1u : 0u;
                                if (lost)
                                    atomicOr(p.status, kStatusListOverflow);
                            }
                        }
                        half_sync();
                        // exact compaction of any row whose sub-lists are about to fill
                        // (all 128 threads): keep the top `keep` entries of the four
                        // sub-lists, written to the front of sub-list 0
                        for (int rr = 0; rr < RPH; ++rr) {
                            const int rl = half * RPH + rr;
                            if (rl >= ui.nr || rows_s[rl].compact == 0)
                                continue;
                            RowState& rs = rows_s[rl];
                            uint2* list = p.lists + sg.out_offset +
                                          (int64_t)(ui.t0 + rl - sg.row_begin) * sg.out_ld;
                            const int n0 = static_cast<int>(min(rs.wcnt[0], cap));
                            const int n1 = static_cast<int>(min(rs.wcnt[1], cap));
                            const int n2 = static_cast<int>(min(rs.wcnt[2], cap));
                            const int n3 = static_cast<int>(min(rs.wcnt[3], cap));
                            const int o1 = n0, o2 = n0 + n1, o3 = n0 + n1 + n2;
                            const int n = o3 + n3;
                            auto at = [&](int e) -> uint2* {
                                const int w4 = (e >= o1) + (e >= o2) + (e >= o3);
                                const int base =
                                    w4 == 0 ? 0 : (w4 == 1 ? o1 : (w4 == 2 ? o2 : o3));
                                return list + (int64_t)w4 * sg.cap + (e - base);
                            };
                            auto load = [&](int e, uint32_t& hi, uint32_t& lo) {
                                const uint2 ent = *at(e);
                                hi = f2ord(__uint_as_float(ent.x));
                                lo = ~ent.y;
                            };
                            const CompositeThr thr = group_threshold<kHalfThreads>(
                                *sel_s, htid, n, static_cast<uint32_t>(p.keep), load, half_sync);
                            // kept entry number pos goes to list[pos] (the four sub-lists
                            // are contiguous), at or before the entry's own place: pos <= e
                            // and entry e lies at or after list[e]
                            auto emit = [&](int pos, int e, uint32_t hi, uint32_t lo) {
                                (void)e;
                                list[pos] = make_uint2(__float_as_uint(ord2f(hi)), ~lo);
                            };
                            const int kept = group_emit<kHalfThreads>(*sel_s, htid, n, thr, load,
                                                                      emit, half_sync);
                            half_sync();
                            // spread the kept entries so that sub-list w holds
                            // c_w = (kept + 3 - w) / 4 (at most cap - slack): the entries
                            // past c_w of a sub-list the linear fill left above c_w move, in
                            // order, to the free slots [n_d, c_d) of the sub-lists below; the
                            // two sets of slots are disjoint, so the copies need no order
                            int fill[4], goal[4], surplus[4], room[4], moves = 0;
#pragma unroll
                            for (int w4 = 0; w4 < 4; ++w4) {
                                fill[w4] = min(max(kept - w4 * static_cast<int>(cap), 0),
                                               static_cast<int>(cap));
                                goal[w4] = (kept + 3 - w4) / 4;
                                surplus[w4] = max(fill[w4] - goal[w4], 0);
                                room[w4] = max(goal[w4] - fill[w4], 0);
                                moves += surplus[w4];
                            }
                            for (int x = htid; x < moves; x += kHalfThreads) {
                                int ws = 0, rs_ = x;
                                while (rs_ >= surplus[ws]) {
                                    rs_ -= surplus[ws];
                                    ++ws;
                                }
                                int wd = 0, rd = x;
                                while (rd >= room[wd]) {
                                    rd -= room[wd];
                                    ++wd;
                                }
                                list[(int64_t)wd * sg.cap + fill[wd] + rd] =
                                    list[(int64_t)ws * sg.cap + goal[ws] + rs_];
                            }
                            half_sync();
                            if (htid == 0) {
#pragma unroll
                                for (int w4 = 0; w4 < 4; ++w4)
                                    rs.wcnt[w4] = static_cast<uint32_t>(goal[w4]);
                                rs.compact = 0;
                                // later entries must reach the kept set's threshold
                                if (thr.phi > rs.tau_hi ||
                                    (thr.phi == rs.tau_hi && thr.plo > rs.tau_lo)) {
                                    rs.tau_hi = thr.phi;
                                    rs.tau_lo = thr.plo;
                                }
                                const int t = ui.t0 + rl;
                                const uint32_t gv =
                                    *reinterpret_cast<volatile uint32_t*>(p.gtau + t);
                                if (thr.phi > gv)
                                    atomicMax(p.gtau + t, thr.phi);
                            }
                            half_sync();
                        }
#pragma unroll
                        for (int oi = 0; oi < kOwned; ++oi) {
                            const int rl = half * RPH + quad + 4 * oi;
                            if (quad + 4 * oi < RPH && rl < ui.nr)
                                gpre[oi] = ld_relaxed_gpu(p.gtau + ui.t0 + rl);
                        }
#pragma unroll
                        for (int ro = 0; ro < RO; ++ro) {
                            const int rl = half * RPH + own_rr(ro);
                            tau_hi[ro] = rows_s[rl].tau_hi;
                            tau_lo[ro] = rows_s[rl].tau_lo;
                            b1[ro] = rows_s[rl].b1;
                            wcnt[ro] = rows_s[rl].wcnt[quad];
                        }
                    }
                }
            }
            if constexpr (C::STREAM) {
                // unit end: every warp publishes its own sub-list lengths (also for
                // units with no tiles; not for units a second pass skips, whose rows
                // keep the first pass's lists)
                if constexpr (SINK == kSinkFilter || SINK == kSinkPoolFilter) {
                    // the fixed-threshold sinks count in shared memory (this warp's own
                    // counters: its lanes' atomics are done once the warp converges)
                    __syncwarp();
#pragma unroll
                    for (int ro = 0; ro < RO; ++ro)
                        wcnt[ro] = rows_s[half * RPH + own_rr(ro)].wcnt[quad];
                }
                if (row_leader && !ui.skip) {
#pragma unroll
                    for (int ro = 0; ro < RO; ++ro) {
                        const int rl = half * RPH + own_rr(ro);
                        if (rl < ui.nr)
                            p.counts[sg.cnt_offset +
                                     (int64_t)(ui.t0 + rl - sg.row_begin) * sg.cnt_ld + quad] =
                                (SINK == kSinkFilter || SINK == kSinkPoolFilter)
                                    ? wcnt[ro]
                                    : min(wcnt[ro], static_cast<uint32_t>(sg.cap));
                    }
                }
                // both halves are done with the row state before the next unit resets it
                epi_sync();
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1)
        tmem_dealloc(tmem_base, 512);
}

template <int H, int D, int SINK, bool MASK, int OPS>
cudaError_t launch_one(const LogitsParams& p, int grid, cudaStream_t stream)
{
    using C = Cfg<H, D, SINK, OPS>;
    auto kern = logits_tc_kernel<H, D, SINK, MASK, OPS>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::SMEM);
    if (e != cudaSuccess)
        return e;
    return launch_pdl(kern, dim3(grid), dim3(C::THREADS), C::SMEM, stream, p);
}

template <int H, int D, int OPS = kOpsE4M3>
cudaError_t launch_sink(const LogitsParams& p, int sink, int grid, cudaStream_t stream)
{
    // masked launches: the consumer's key paths (samples, fixed threshold, stream);
    // the candidate producer itself is never masked
    const bool m = p.cand_mask != nullptr;
    if (sink == kSinkLogits)
        return m ? launch_one<H, D, kSinkLogits, true, OPS>(p, grid, stream)
                 : launch_one<H, D, kSinkLogits, false, OPS>(p, grid, stream);
    if (sink == kSinkStream)
        return m ? launch_one<H, D, kSinkStream, true, OPS>(p, grid, stream)
                 : launch_one<H, D, kSinkStream, false, OPS>(p, grid, stream);
    if (sink == kSinkFilter)
        return m ? launch_one<H, D, kSinkFilter, true, OPS>(p, grid, stream)
                 : launch_one<H, D, kSinkFilter, false, OPS>(p, grid, stream);
    if (m)
        return cudaErrorInvalidValue;
    if (sink == kSinkPool)
        return launch_one<H, D, kSinkPool, false, OPS>(p, grid, stream);
    if (sink == kSinkPoolFilter)
        return launch_one<H, D, kSinkPoolFilter, false, OPS>(p, grid, stream);
    return cudaErrorInvalidValue;
}

}  // namespace

bool logits_fp4_native(int H, int D) { return H == 32 && D == 128; }

int logits_rows_per_group(int H, bool fp4_keys)
{
    if (fp4_keys && logits_fp4_native(H, 128))
        return Cfg<32, 128, kSinkFilter, kOpsE2M1K>::G;
    return H >= 16 ? kTileN / H : 16;
}

cudaError_t launch_logits(const LogitsParams& p, int H, int D, int sink, int grid,
                          cudaStream_t stream)
{
    if (p.k_sf != nullptr && p.q_sf != nullptr)
        return (H == 32 && D == 128) ? launch_sink<32, 128, kOpsE2M1>(p, sink, grid, stream)
                                     : cudaErrorInvalidValue;
    if (p.k_sf != nullptr)
        return (H == 32 && D == 128) ? launch_sink<32, 128, kOpsE2M1K>(p, sink, grid, stream)
                                     : cudaErrorInvalidValue;
    if (p.q_sf != nullptr)
        return cudaErrorInvalidValue;
    if (H == 32 && D == 128)
        return launch_sink<32, 128>(p, sink, grid, stream);
    if (H == 16 && D == 128)
        return launch_sink<16, 128>(p, sink, grid, stream);
    if (H == 64 && D == 128)
        return launch_sink<64, 128>(p, sink, grid, stream);
    if (H == 8 && D == 64)
        return launch_sink<8, 64>(p, sink, grid, stream);
    return cudaErrorInvalidValue;
}

}  // namespace idx
