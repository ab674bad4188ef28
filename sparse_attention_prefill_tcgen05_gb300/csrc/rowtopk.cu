// Top-k over caller logits [rows, ld] in one read of every row ("chunked-prefill-
// memory.md" section 2.3: the ragged top-k after the logits), for rows of at most
// 65,536 keys and k <= 2048.
//
// The row's sampled threshold tau (from the sampled tiles, computed beforehand) keeps
// about 1.7 k of its entries; those fit in shared memory, so the exact selection of a
// row needs no global lists and no second kernel.  One persistent CTA per SM, three
// roles:
//   warp 0        producer: takes rows in order from a global counter (the next row's
//                 number, length and thresholds read while the current row streams) and
//                 streams each row through a ring of three 32 KB stages with bulk copies;
//   warps 1..8    filter: each warp takes its 1/8 of every stage; a lane tests its 32
//                 values against tau, and the warp appends the passing ones (positions
//                 from a warp prefix sum of the lanes' counts, values read again from
//                 the stage) to its own region of the row's candidate buffer (two
//                 buffers, rows alternate); the warps never wait for one another;
//   warps 9..16   select: the exact top-k of a full buffer (2048 equal-width value
//                 buckets from tau to the row's largest sample, larger values in the top
//                 one; the bucket holding the k-th entry, its entries ranked directly, a
//                 bitmap of the kept keys, their positions by a prefix sum) written in
//                 ascending key order, each kept entry straight to its place, while the
//                 filter warps fill the other buffer.
// A row whose candidates cannot decide it (fewer than k at or above tau, or more than the
// warps' regions and the shared spill area hold) is flagged for the direct kernel.  Every wait is bounded: a
// timeout sets the status word and every role leaves its loop.
#include "groupsel.cuh"
#include "internal.h"

#include <algorithm>

namespace idx {
namespace {

// (more filter or select warps measured slower: the selection is bound by the latency
// of its shared-memory passes, and extra warps only take issue slots from it)
constexpr int kFiltWarps = 8;
constexpr int kSelWarps = 8;
constexpr int kFiltThreads = 32 * kFiltWarps;              // 256
constexpr int kSelThr = 32 * kSelWarps;                    // 256
constexpr int kRtThreads = 32 + kFiltThreads + kSelThr;    // 544
constexpr int kChunk = 8192;                               // floats per ring stage (32 KB)
constexpr int kStages = 3;                                 // (a larger stage count does not fit)
constexpr int kF4 = kChunk / (4 * kFiltThreads);           // float4 per filter lane per stage
constexpr int kRegion = 512;                               // candidates per filter warp
constexpr int kSpill = 1024;                               // shared by the warps, after their own
constexpr int kCand = kFiltWarps * kRegion + kSpill;       // per buffer
constexpr int kRtBuckets = 2048;
constexpr int kRtMaxK = 2048;
constexpr int kRtWords = 2048;                             // bitmap words: keys < 65536
constexpr int kRtBucketCands = 256;
constexpr int kBarSel = 2;                                 // named barrier of the select warps
static_assert(kChunk == 4 * kF4 * kFiltThreads && kF4 <= 8, "a filter thread takes kF4 float4 of a stage");
static_assert(kFiltWarps % kSelWarps == 0, "a select warp takes whole filter regions");

// What the producer publishes with each stage.
struct StageMeta {
    int32_t t;       // global row, -1: no more rows
    int32_t chunk;   // chunk number within the row
    int32_t nfl;     // valid floats in the stage
    int32_t last;    // the row's last chunk
    int32_t keys;    // keys of the row's request
    uint32_t tau;    // the row's sampled threshold (ord of a score)
    uint32_t smax;   // the row's largest sample (ord of a score)
    int32_t pad_;
};

// What the producer knows of a row before streaming it.
struct RowInfo {
    int t;           // global row (>= total_rows: no more rows)
    int keys;        // keys of its request
    int n;           // keys streamed (its causal length, clamped)
    uint32_t tau, smax;
};

// A full candidate buffer, as the select warps find it (written by filter warp 0).
struct RowSlot {
    int32_t t;
    int32_t keys;
    uint32_t tau;
    uint32_t smax;
};

// shared memory carve-up (bytes from a 128-byte aligned base)
constexpr size_t kOffRing = 0;
constexpr size_t kOffCand = kOffRing + (size_t)kStages * kChunk * 4;      // 96 KB
constexpr size_t kOffHist = kOffCand + 2 * (size_t)kCand * 8;             // + 80 KB
constexpr size_t kOffBits = kOffHist + (size_t)kRtBuckets * 4;            // + 8 KB
constexpr size_t kOffWpre = kOffBits + (size_t)kRtWords * 4;              // + 8 KB
constexpr size_t kOffMeta = kOffWpre + (size_t)kRtWords * 4;              // + 8 KB
constexpr size_t kOffSlot = kOffMeta + kStages * sizeof(StageMeta);
constexpr size_t kOffRcnt = kOffSlot + 2 * sizeof(RowSlot);               // [2][kFiltWarps]
constexpr size_t kOffSpill = kOffRcnt + 2 * kFiltWarps * 4;               // [2] spill counts
constexpr size_t kOffBar = (kOffSpill + 2 * 4 + 7) / 8 * 8;
constexpr int kNumBars = 2 * kStages + 4;
constexpr size_t kOffMisc = kOffBar + kNumBars * 8;
constexpr size_t kRtSmem = kOffMisc + 64 + 128;                          // + alignment slack
static_assert(kRtSmem <= 227 * 1024, "shared memory of the row top-k kernel");

__device__ __forceinline__ int rt_request(const RowTopkParams& p, int t)
{
    int lo = 0, hi = p.num_requests - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (p.req_row_begin[mid] <= t)
            lo = mid;
        else
            hi = mid - 1;
    }
    return lo;
}

// Exclusive prefix sum over the select warps (named barrier kBarSel); `wsum` holds one
// word per select warp.
__device__ __forceinline__ uint32_t sel_exclusive_sum(uint32_t v, int st, uint32_t* wsum)
{
    const int lane = st & 31, w = st >> 5;
    uint32_t incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o)
            incl += y;
    }
    if (lane == 31)
        wsum[w] = incl;
    bar_all(true, kBarSel, kSelThr);
    uint32_t before = 0;
#pragma unroll
    for (int x = 0; x < kSelWarps; ++x)
        before += x < w ? wsum[x] : 0u;
    bar_all(true, kBarSel, kSelThr);
    return before + incl - v;
}

__global__ void __launch_bounds__(kRtThreads, 1) row_topk_kernel(const __grid_constant__ RowTopkParams p)
{
    pdl_wait_then_release();
    extern __shared__ __align__(128) uint8_t rt_smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(rt_smem_raw) + 127) & ~static_cast<uintptr_t>(127));
    float* ring = reinterpret_cast<float*>(smem + kOffRing);
    uint2* cand = reinterpret_cast<uint2*>(smem + kOffCand);
    uint32_t* hist = reinterpret_cast<uint32_t*>(smem + kOffHist);
    uint32_t* bits = reinterpret_cast<uint32_t*>(smem + kOffBits);
    uint32_t* wpre = reinterpret_cast<uint32_t*>(smem + kOffWpre);
    StageMeta* meta = reinterpret_cast<StageMeta*>(smem + kOffMeta);
    RowSlot* slot = reinterpret_cast<RowSlot*>(smem + kOffSlot);
    uint32_t* rcnt = reinterpret_cast<uint32_t*>(smem + kOffRcnt);   // [2][kFiltWarps]
    uint32_t* spill_n = reinterpret_cast<uint32_t*>(smem + kOffSpill);   // [2]
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
    uint64_t* full = bars;                 // ring stage filled (producer, bytes)
    uint64_t* empty = bars + kStages;      // ring stage read (one arrival per filter warp)
    uint64_t* cfull = bars + 2 * kStages;  // candidate buffer ready (one per filter warp)
    uint64_t* cempty = cfull + 2;          // candidate buffer free (select warps)
    uint32_t* wsum = reinterpret_cast<uint32_t*>(smem + kOffMisc);        // [kSelWarps]
    uint32_t* bcast = wsum + kSelWarps;                                   // [4]
    volatile int* abort_flag = reinterpret_cast<volatile int*>(bcast + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kFiltWarps);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&cfull[b], kFiltWarps);
            mbar_init(&cempty[b], 1);
        }
        *abort_flag = 0;
        spill_n[0] = 0;
        spill_n[1] = 0;
        fence_mbar_init();
    }
    __syncthreads();
    const long long budget = p.timeout_cycles;
    auto report_timeout = [&]() {
        *abort_flag = 1;
        atomicOr(p.status, kStatusTimeout);
    };

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane != 0)
            return;
        int uses[kStages];   // phases of each stage this thread started
        for (int s = 0; s < kStages; ++s)
            uses[s] = 0;
        int s = 0, ph = 0;
        bool ok = true;
        auto next_stage = [&]() -> bool {
            if (!mbar_wait_backoff(&empty[s], ph ^ 1, budget, abort_flag)) {
                report_timeout();
                return false;
            }
            return true;
        };
        auto advance = [&]() {
            if (++s == kStages) {
                s = 0;
                ph ^= 1;
            }
        };
        // A row's number, length and threshold come from a chain of dependent global
        // reads; the next row's chain runs while the current row's first stages stream,
        // so the ring does not drain at row boundaries.
        auto row_info = [&](int t) {
            RowInfo ri;
            ri.t = t;
            ri.keys = 0;
            ri.n = 0;
            ri.tau = 0;
            ri.smax = 0;
            if (t < p.total_rows) {
                const int r = rt_request(p, t);
                ri.keys = p.req_key_count[r];
                ri.n = max(0, min(p.compress_len[t], ri.keys));
                ri.tau = p.tau_row[t];
                ri.smax = p.smax_row[t];
            }
            return ri;
        };
        RowInfo cur = row_info(static_cast<int>(atomicAdd(p.row_counter, 1u)));
        while (ok && cur.t < p.total_rows) {
            const int t = cur.t;
            const int keys = cur.keys;
            const int n = cur.n;
            // the next row's number, taken now; its reads are issued after this row's
            // first stage
            const int t_next = static_cast<int>(atomicAdd(p.row_counter, 1u));
            RowInfo nxt = {p.total_rows, 0, 0, 0u, 0u};
            const float* row = p.logits + (int64_t)t * p.ld;
            const int nchunks = max(1, (n + kChunk - 1) / kChunk);
            for (int c = 0; c < nchunks && ok; ++c) {
                if (!(ok = next_stage()))
                    break;
                const int nfl = min(kChunk, n - c * kChunk);
                StageMeta& m = meta[s];
                m.t = t;
                m.chunk = c;
                m.nfl = max(nfl, 0);
                m.last = c == nchunks - 1;
                m.keys = keys;
                m.tau = cur.tau;
                m.smax = cur.smax;
                if (nfl > 0) {
                    // whole 16-byte groups: ld is a multiple of 4, so the group holding
                    // the row's last key is inside the row
                    const uint32_t bytes = static_cast<uint32_t>((nfl + 3) / 4) * 16u;
                    mbar_arrive_expect_tx(&full[s], bytes);
                    bulk_load(ring + (size_t)s * kChunk, row + (size_t)c * kChunk, bytes, &full[s]);
                } else {
                    mbar_arrive(&full[s]);
                }
                ++uses[s];
                advance();
                if (c == 0)
                    nxt = row_info(t_next);
            }
            if (!ok)
                break;
            cur = nxt;
        }
        if (ok && next_stage()) {
            meta[s].t = -1;   // no more rows
            mbar_arrive(&full[s]);
            ++uses[s];
        }
        // no copy may still be landing in shared memory when the CTA exits: wait for the
        // last phase of every stage (a stage's phases complete in order)
        volatile int no_abort = 0;
        for (int x = 0; x < kStages; ++x)
            if (uses[x] > 0)
                mbar_wait(&full[x], (uses[x] - 1) & 1, budget, &no_abort);
        return;
    }

    if (warp <= kFiltWarps) {
        // -------------------------------------------------------------- filter
        // thread ft takes float4 ft + 256 u (u < kF4) of every stage, so warp fw covers
        // floats [128 fw, 128 fw + 128) of every 1024; decisions are per warp
        const int fw = warp - 1;
        const int ft = threadIdx.x - 32;
        int s = 0, ph = 0, b = 0, bph = 0;
        float tauf = 0.0f;
        uint32_t count = 0;   // entries this warp found in the row
        while (true) {
            bool got = mbar_wait_backoff(&full[s], ph, budget, abort_flag);
            if (!__all_sync(0xffffffffu, got)) {
                if (lane == 0)
                    report_timeout();
                break;
            }
            const StageMeta m = meta[s];
            if (m.t < 0 || m.chunk == 0) {
                // a new row (or the end) takes the next candidate buffer, once the select
                // warps are done with its previous row
                got = mbar_wait_backoff(&cempty[b], bph ^ 1, budget, abort_flag);
                if (!__all_sync(0xffffffffu, got)) {
                    if (lane == 0)
                        report_timeout();
                    break;
                }
                if (m.t < 0) {
                    if (lane == 0) {
                        if (fw == 0)
                            slot[b].t = -1;
                        mbar_arrive(&cfull[b]);
                    }
                    break;
                }
                const uint32_t tau = m.tau;
                // at or above tau as a float: every v whose ord is at least tau (and
                // -0.0 against +0.0, harmless); tau = 0 keeps every finite entry
                tauf = tau > kOrdNegInf ? ord2f(tau) : -3.402823466e38f;
                count = 0;
                if (fw == 0 && lane == 0) {
                    slot[b].t = m.t;
                    slot[b].keys = m.keys;
                    slot[b].tau = tau;
                    slot[b].smax = m.smax;
                }
            }
            const float* stage = ring + (size_t)s * kChunk;
            const float4* src = reinterpret_cast<const float4*>(stage);
            uint32_t pm = 0;   // which of the lane's values pass
#pragma unroll
            for (int u = 0; u < kF4; ++u) {
                const float4 x = src[ft + kFiltThreads * u];
                pm |= (x.x >= tauf ? 1u : 0u) << (4 * u);
                pm |= (x.y >= tauf ? 1u : 0u) << (4 * u + 1);
                pm |= (x.z >= tauf ? 1u : 0u) << (4 * u + 2);
                pm |= (x.w >= tauf ? 1u : 0u) << (4 * u + 3);
            }
            if (m.nfl < kChunk) {
                // the row's last, partial stage: only its first nfl floats are keys
#pragma unroll
                for (int e = 0; e < 4 * kF4; ++e)
                    if (4 * (ft + kFiltThreads * (e >> 2)) + (e & 3) >= m.nfl)
                        pm &= ~(1u << e);
            }
            // positions: the warp's count so far plus the lanes before this one
            const uint32_t c = __popc(pm);
            uint32_t incl = c;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o)
                    incl += y;
            }
            const uint32_t wtot = __shfl_sync(0xffffffffu, incl, 31);
            uint32_t pos = count + incl - c;
            uint2* region = cand + (size_t)b * kCand + (size_t)fw * kRegion;
            uint2* spill = cand + (size_t)b * kCand + (size_t)kFiltWarps * kRegion;
            const uint32_t jbase = static_cast<uint32_t>(m.chunk * kChunk);
            while (pm != 0) {
                const int e = __ffs(pm) - 1;
                pm &= pm - 1;
                const int jl = 4 * (ft + kFiltThreads * (e >> 2)) + (e & 3);
                const uint2 ent = make_uint2(__float_as_uint(stage[jl]),
                                             jbase + static_cast<uint32_t>(jl));
                if (pos < static_cast<uint32_t>(kRegion)) {
                    region[pos] = ent;
                } else {
                    // the warp's region is full: the shared spill area (its count past
                    // kSpill marks the row as overflowed)
                    const uint32_t sp = atomicAdd(&spill_n[b], 1u);
                    if (sp < static_cast<uint32_t>(kSpill))
                        spill[sp] = ent;
                }
                ++pos;
            }
            count += wtot;
            // the stage has been read (the passing values were read again above)
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&empty[s]);
            if (m.last) {
                // the warp's part of the row is done: its count (past its region: the
                // rest went to the spill area), then its arrival on the buffer
                if (lane == 0) {
                    rcnt[b * kFiltWarps + fw] = count;
                    mbar_arrive(&cfull[b]);
                }
                if (++b == 2) {
                    b = 0;
                    bph ^= 1;
                }
            }
            if (++s == kStages) {
                s = 0;
                ph ^= 1;
            }
        }
        return;
    }

    // ------------------------------------------------------------------ select
    const int st = threadIdx.x - 32 - kFiltThreads;   // 0..255
    const uint32_t k = static_cast<uint32_t>(p.k);
    SelScratch<kSelThr>& gsh = *reinterpret_cast<SelScratch<kSelThr>*>(bits);   // radix scratch
    int b = 0, bph = 0;
    while (true) {
        const bool got = mbar_wait_backoff(&cfull[b], bph, budget, abort_flag);
        if (!bar_all(got, kBarSel, kSelThr)) {
            if (st == 0)
                report_timeout();
            break;
        }
        const RowSlot sl = slot[b];
        if (sl.t < 0)
            break;
        const int t = sl.t;
        uint2* cb = cand + (size_t)b * kCand;
        const uint32_t* rc = rcnt + b * kFiltWarps;
        // the warps' regions, then the spill area (overflowed when its count passed it)
        const uint32_t nspill = spill_n[b];
        const bool overflow = nspill > static_cast<uint32_t>(kSpill);
        const int spilled = static_cast<int>(min(nspill, static_cast<uint32_t>(kSpill)));
        uint32_t total_c = static_cast<uint32_t>(spilled);
#pragma unroll
        for (int w = 0; w < kFiltWarps; ++w)
            total_c += min(rc[w], static_cast<uint32_t>(kRegion));
        // candidate e (of the kCand places) holds an entry iff it is below its warp
        // region's count, or below the spill count in the spill area
        auto valid = [&](int e) {
            if (e >= kFiltWarps * kRegion)
                return e - kFiltWarps * kRegion < spilled;
            const int w = e / kRegion;
            return static_cast<uint32_t>(e - w * kRegion) < rc[w];
        };
        // f(e) for every candidate: select warp sw walks the regions sw, sw + 8, ... with
        // all of its lanes, then all select threads share the spill area
        // f(e, entry e) for every candidate: select warp sw walks the regions sw, sw + 8,
        // ... with all of its lanes, then all select threads share the spill area; each
        // thread loads four entries before it works on any of them
        auto each_cand = [&](auto&& f) {
            auto walk = [&](const int base, const int n, int i0, const int step) {
                for (; i0 < n; i0 += 4 * step) {
                    uint2 en[4];
#pragma unroll
                    for (int u = 0; u < 4; ++u)
                        en[u] = cb[base + min(i0 + u * step, n - 1)];
#pragma unroll
                    for (int u = 0; u < 4; ++u)
                        if (i0 + u * step < n)
                            f(base + i0 + u * step, en[u]);
                }
            };
            const int sw = st >> 5, sln = st & 31;
#pragma unroll 1
            for (int w = sw; w < kFiltWarps; w += kSelWarps)
                walk(w * kRegion, static_cast<int>(min(rc[w], static_cast<uint32_t>(kRegion))),
                     sln, 32);
            walk(kFiltWarps * kRegion, spilled, st, kSelThr);
        };
        if (overflow || (sl.tau > kOrdNegInf && total_c < k)) {
            // the candidates cannot decide the row: the direct kernel will
            if (st == 0) {
                p.row_fail[t] = 1u;
                atomicOr(p.fail_any, 1u);
            }
        } else {
            // composite key (ord(score), ~index) of a candidate
            auto comp = [](const uint2 en) {
                return (static_cast<uint64_t>(f2ord(__uint_as_float(en.x))) << 32) |
                       static_cast<uint32_t>(~(en.y & 0xFFFFu));
            };
            // which candidates are kept: all of them (at most k); those above the
            // boundary bucket, with the whole boundary bucket or the best of it; or (no
            // bucket range, or a boundary bucket too large to rank directly) the radix
            // threshold over the candidates
            int mode = 0;   // 0 all, 1 buckets down to the boundary one, 2 radix,
                            // 3 buckets above the boundary one plus its best `need`
            uint32_t bnd = 0, need = 0, bsize = 0;
            CompositeThr thr{0u, 0u, 0u, 0u};
            float bvmin = 0.0f, bscale = 0.0f;
            // a candidate's value bucket (the same arithmetic in every pass)
            auto bucket_of = [&](const uint32_t vbits) {
                return static_cast<uint32_t>(min(kRtBuckets - 1, static_cast<int>(
                    __fmul_rn(__fsub_rn(__uint_as_float(vbits), bvmin), bscale))));
            };
            if (total_c > k) {
                mode = 2;
                const uint32_t smax = sl.smax;
                bool bucketed = false;
                if (sl.tau > kOrdNegInf && smax > sl.tau) {
                    bvmin = ord2f(sl.tau);
                    const float range = __fsub_rn(ord2f(smax), bvmin);
                    bscale = range > 0.0f ? __fdiv_rn(static_cast<float>(kRtBuckets), range)
                                          : 0.0f;
                    bucketed = bscale > 0.0f && bscale < INFINITY;
                }
                if (bucketed) {
                    // value buckets, counted
                    for (int i = st; i < kRtBuckets / 4; i += kSelThr)
                        reinterpret_cast<uint4*>(hist)[i] = make_uint4(0u, 0u, 0u, 0u);
                    bar_all(true, kBarSel, kSelThr);
                    each_cand([&](const int, const uint2 en) {
                        atomicAdd(&hist[bucket_of(en.x)], 1u);
                    });
                    bar_all(true, kBarSel, kSelThr);
                    // the bucket holding the k-th largest, from the top: thread i owns
                    // buckets [2048 - 8 (i + 1), 2048 - 8 i)
                    constexpr int kPer = kRtBuckets / kSelThr;
                    const int top = kRtBuckets - kPer * st;
                    uint32_t c8[kPer], local = 0;
#pragma unroll
                    for (int x = 0; x < kPer; ++x) {
                        c8[x] = hist[top - 1 - x];
                        local += c8[x];
                    }
                    const uint32_t above = sel_exclusive_sum(local, st, wsum);
                    if (above < k && above + local >= k) {
                        uint32_t cum = above;
#pragma unroll
                        for (int x = 0; x < kPer; ++x) {
                            if (cum + c8[x] >= k) {
                                bcast[0] = static_cast<uint32_t>(top - 1 - x);
                                bcast[1] = k - cum;
                                bcast[2] = c8[x];
                                break;
                            }
                            cum += c8[x];
                        }
                    }
                    bar_all(true, kBarSel, kSelThr);
                    bnd = bcast[0];
                    need = bcast[1];
                    bsize = bcast[2];
                    if (bsize == need)
                        mode = 1;   // the whole boundary bucket is kept
                    else if (bsize <= static_cast<uint32_t>(kRtBucketCands))
                        mode = 3;   // its entries are collected with the bitmap and ranked
                }
                if (mode == 2) {
                    auto load = [&](int e, uint32_t& hi, uint32_t& lo) {
                        const uint2 en = cb[e];
                        hi = valid(e) ? f2ord(__uint_as_float(en.x)) : 0u;   // 0: not eligible
                        lo = ~(en.y & 0xFFFFu);
                    };
                    thr = group_threshold<kSelThr>(gsh, st, kCand, k, load,
                                                   NamedSync{kBarSel, kSelThr});
                    bar_all(true, kBarSel, kSelThr);   // (the radix scratch becomes the bitmap)
                }
            }
            // the kept keys as a bitmap (mode 3: the boundary bucket's entries are
            // collected on the way, its best `need` added after), then their output
            // positions in key order
            uint64_t* bc = reinterpret_cast<uint64_t*>(wpre);   // free until the prefix sums
            const int nw = max((sl.keys + 31) / 32, 1);
            for (int w = st; w < nw; w += kSelThr)
                bits[w] = 0;
            if (st == 0)
                bcast[3] = 0;
            bar_all(true, kBarSel, kSelThr);
            each_cand([&](const int, const uint2 en) {
                bool keep = true;
                if (mode == 2) {
                    keep = thr.kept(f2ord(__uint_as_float(en.x)), ~(en.y & 0xFFFFu));
                } else if (mode != 0) {
                    const uint32_t bk = bucket_of(en.x);
                    keep = bk > bnd || (mode == 1 && bk == bnd);
                    if (mode == 3 && bk == bnd) {
                        const uint32_t x = atomicAdd(&bcast[3], 1u);
                        if (x < static_cast<uint32_t>(kRtBucketCands))
                            bc[x] = comp(en);
                    }
                }
                if (keep) {
                    const uint32_t j = en.y & 0xFFFFu;
                    atomicOr(&bits[j >> 5], 1u << (j & 31));
                }
            });
            bar_all(true, kBarSel, kSelThr);
            if (mode == 3) {
                // the boundary bucket's best `need`: the entries with fewer than `need`
                // above them (composite keys are distinct)
                for (int i = st; i < static_cast<int>(bsize); i += kSelThr) {
                    const uint64_t mine = bc[i];
                    uint32_t rank = 0;
                    for (int x = 0; x < static_cast<int>(bsize); ++x)
                        rank += bc[x] > mine;
                    if (rank < need) {
                        const uint32_t j = ~static_cast<uint32_t>(mine) & 0xFFFFu;
                        atomicOr(&bits[j >> 5], 1u << (j & 31));
                    }
                }
                bar_all(true, kBarSel, kSelThr);
            }
            constexpr int kPerW = kRtWords / kSelThr;   // consecutive words per thread
            const int w0 = st * kPerW;
            uint32_t local = 0;
#pragma unroll
            for (int w = 0; w < kPerW; ++w)
                local += w0 + w < nw ? __popc(bits[w0 + w]) : 0u;
            uint32_t run = sel_exclusive_sum(local, st, wsum);
#pragma unroll
            for (int w = 0; w < kPerW; ++w) {
                if (w0 + w < nw) {
                    wpre[w0 + w] = run;
                    run += __popc(bits[w0 + w]);
                }
            }
            if (st == kSelThr - 1)
                bcast[0] = run;   // kept entries
            bar_all(true, kBarSel, kSelThr);
            const int total = static_cast<int>(bcast[0]);
            // each kept entry straight to its place in the output row (a shared-memory
            // copy of the row and a coalesced pass measured no faster), then the padding
            int32_t* oi = p.out_idx + (int64_t)t * p.k;
            float* ov = p.out_val ? p.out_val + (int64_t)t * p.k : nullptr;
            each_cand([&](const int, const uint2 en) {
                const uint32_t j = en.y & 0xFFFFu;
                const uint32_t word = bits[j >> 5];
                if ((word >> (j & 31)) & 1u) {
                    const int pos =
                        static_cast<int>(wpre[j >> 5] + __popc(word & ((1u << (j & 31)) - 1u)));
                    oi[pos] = static_cast<int32_t>(j);
                    if (ov)
                        ov[pos] = __uint_as_float(en.x);
                }
            });
            for (int i = total + st; i < p.k; i += kSelThr) {
                oi[i] = -1;
                if (ov)
                    ov[i] = -INFINITY;
            }
        }
        // everything of the buffer has been read: release it, its
        // spill count zeroed for its next row
        bar_all(true, kBarSel, kSelThr);
        if (st == 0) {
            spill_n[b] = 0;
            mbar_arrive(&cempty[b]);
        }
        if (++b == 2) {
            b = 0;
            bph ^= 1;
        }
    }
}

}  // namespace

int row_topk_max_keys() { return 65536; }

cudaError_t launch_row_topk(const RowTopkParams& p, cudaStream_t st)
{
    if (p.total_rows <= 0)
        return cudaSuccess;
    if (p.k < 1 || p.k > kRtMaxK || p.ld % 4 != 0 ||
        (reinterpret_cast<uintptr_t>(p.logits) & 15) != 0)
        return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(row_topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kRtSmem));
    if (e != cudaSuccess)
        return e;
    int dev = 0, sms = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
        return e;
    const int grid = std::min(p.total_rows, std::max(sms, 1));
    return launch_pdl(row_topk_kernel, dim3(grid), dim3(kRtThreads), kRtSmem, st, p);
}

}  // namespace idx
