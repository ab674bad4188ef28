// Exact per-row top-k selection kernels.
//
// Selection rule: among the eligible entries of a row (finite score, inside
// the row's causal length, a candidate block for masked consumers) keep the
// k with the largest score; on equal scores the lower key index wins.  Used
// for
//   * the ragged top-k over dense logits (indexer_topk, the ragged top-k that
//     "chunked-prefill-memory.md" section 2.3 runs after the logits);
//   * the exact merge of the candidate lists that the streaming logits kernel
//     appends per key split: the top-k of the union of the splits' candidates
//     is the top-k of the row (same section, "holds exactly");
//   * candidate blocks: the same over 8-key block maxima, written as a mask.
// The threshold search and ordered emission are in groupsel.cuh.
#include "groupsel.cuh"
#include "internal.h"

namespace idx {
namespace {

constexpr int kSelThreads = 512;
using Scratch = SelScratch<kSelThreads>;

__device__ __forceinline__ int find_request(const int32_t* row_begin, int nreq, int t)
{
    int lo = 0, hi = nreq - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (row_begin[mid] <= t)
            lo = mid;
        else
            hi = mid - 1;
    }
    return lo;
}

// Top-k of entries 0..n-1; load(e) -> (score, index).  Emits in ascending e.
template <class LoadVJ, class Emit>
__device__ int cta_topk(Scratch& sh, int n, int k, const LoadVJ& load_vj, const Emit& emit)
{
    auto load = [&](int e, uint32_t& hi, uint32_t& lo) {
        float v;
        int32_t j;
        load_vj(e, v, j);
        hi = f2ord(v);
        lo = ~static_cast<uint32_t>(j);
    };
    const CompositeThr thr =
        group_threshold<kSelThreads>(sh, threadIdx.x, n, static_cast<uint32_t>(k), load, CtaSync{});
    auto emit_e = [&](int pos, int e, uint32_t hi, uint32_t lo) {
        if (pos < k)
            emit(pos, e, ord2f(hi), static_cast<int32_t>(~lo));
    };
    const int count = group_emit<kSelThreads>(sh, threadIdx.x, n, thr, load, emit_e, CtaSync{});
    return min(count, k);
}

// --------------------------------------------------- streamed-list merge

// Bitonic sort of n2 (a power of two) (key, value) pairs in shared memory,
// ascending by key.
__device__ void bitonic_sort(int32_t* key, float* val, int n2)
{
    for (int size = 2; size <= n2; size <<= 1) {
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            __syncthreads();
            for (int i = threadIdx.x; i < n2 / 2; i += kSelThreads) {
                const int lo = 2 * i - (i & (stride - 1));
                const int hi = lo + stride;
                const bool up = (lo & size) == 0;
                const int32_t a = key[lo], b = key[hi];
                if ((a > b) == up) {
                    key[lo] = b;
                    key[hi] = a;
                    const float fa = val[lo];
                    val[lo] = val[hi];
                    val[hi] = fa;
                }
            }
        }
    }
    __syncthreads();
}

constexpr int kMaxSortK = 4096;
constexpr int kBitmapWords = 2048;    // index-order output by bitmap for keys < 65536

// Exclusive prefix sum of one value per thread over the CTA.
__device__ uint32_t block_exclusive_sum(uint32_t v, Scratch& sh)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint32_t incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o)
            incl += y;
    }
    if (lane == 31)
        sh.warp_sum[warp] = incl;
    __syncthreads();
    uint32_t wbefore = 0;
    for (int w = 0; w < warp; ++w)
        wbefore += sh.warp_sum[w];
    __syncthreads();
    return wbefore + incl - v;
}
// wpre[w] = set bits in bits[0, w); returns the total.  All threads call.
__device__ int bitmap_prefix(const uint32_t* bits, uint32_t* wpre, int nw, Scratch& sh,
                             int& s_total)
{
    constexpr int kPer = kBitmapWords / kSelThreads;   // consecutive words per thread
    const int w0 = threadIdx.x * kPer;
    uint32_t local = 0;
#pragma unroll
    for (int w = 0; w < kPer; ++w)
        local += w0 + w < nw ? __popc(bits[w0 + w]) : 0u;
    const uint32_t before = block_exclusive_sum(local, sh);
    uint32_t run = before;
#pragma unroll
    for (int w = 0; w < kPer; ++w) {
        if (w0 + w < nw) {
            wpre[w0 + w] = run;
            run += __popc(bits[w0 + w]);
        }
    }
    if (threadIdx.x == kSelThreads - 1)
        s_total = static_cast<int>(run);
    __syncthreads();
    return s_total;
}

// Threshold by value buckets (one counting pass instead of up to eight radix
// passes): 2048 equal-width buckets between the smallest and largest staged
// score, the boundary bucket by a suffix scan, and the composite keys of that
// bucket's entries ranked directly when it holds few of them.  kept(v, j) is
// then "bucket(v) above the boundary, or in it with a composite key at least
// the cut".  bucket() is one exact subtraction and one multiplication, the
// same instructions wherever it is evaluated, and monotone in v.
constexpr int kBuckets = 2048;
constexpr int kBucketCands = 256;

struct BucketThr {
    float vmin, scale;
    int boundary;          // -1: every entry is kept
    uint64_t cut;          // composite key cut inside the boundary bucket
    __device__ __forceinline__ int bucket(float v) const
    {
        const float x = __fmul_rn(__fsub_rn(v, vmin), scale);
        return min(kBuckets - 1, static_cast<int>(x));
    }
    __device__ __forceinline__ bool kept(float v, uint32_t j) const
    {
        if (boundary < 0)
            return true;
        const int b = bucket(v);
        if (b != boundary)
            return b > boundary;
        return ((static_cast<uint64_t>(f2ord(v)) << 32) | ~j) >= cut;
    }
};

constexpr int kStageEntries = 4608;   // candidates staged in shared memory per row (36 KB)
static_assert(kStageEntries * 8 >= kBitmapWords * 8, "the bitmap reuses the staging area");

// (three CTAs per SM: the staging area allows no more)
__global__ void __launch_bounds__(kSelThreads, 3)
    stream_merge_kernel(const __grid_constant__ StreamMergeParams p)
{
    __shared__ Scratch sh;
    __shared__ int32_t s_off[kMaxStreamSlots + 1];
    extern __shared__ __align__(16) uint8_t dyn[];
    // [stage: kStageEntries x 8 B][keys: n2 x 4 B][values: n2 x 4 B], n2 = k rounded up
    // to a power of two
    int n2 = 1;
    while (n2 < p.k)
        n2 <<= 1;
    uint2* stage = reinterpret_cast<uint2*>(dyn);
    int32_t* skey = reinterpret_cast<int32_t*>(dyn + sizeof(uint2) * kStageEntries);
    float* sval = reinterpret_cast<float*>(dyn + sizeof(uint2) * kStageEntries + sizeof(int32_t) * n2);

    __shared__ int32_t s_staged;
    __shared__ int32_t s_nall;
    __shared__ int32_t s_overflow;
    __shared__ int s_total;
    __shared__ int s_bnd, s_need, s_bsize, s_bcount;
    __shared__ uint64_t s_cut;
    __shared__ uint32_t s_omin, s_omax;   // range of the staged entries' order keys
    if (threadIdx.x == 0) {
        s_overflow = 0;
        s_staged = 0;
        s_nall = 0;
        s_omin = 0xFFFFFFFFu;
        s_omax = 0u;
    }
    __syncthreads();
    const int cta = blockIdx.x;
    int pi = 0;
    while (pi + 1 < p.num_pieces && p.piece[pi + 1].cta_begin <= cta)
        ++pi;
    const MergePiece& pc = p.piece[pi];
    const int tr = cta - pc.cta_begin;
    const int t = pc.row_begin + tr;
    const int nslots = pc.slots;
    const int64_t lbase = pc.list_offset + (int64_t)tr * nslots * pc.cap;
    const int64_t cbase = pc.count_offset + (int64_t)tr * nslots;
    if (p.only_failed && (*p.fail_any == 0u || p.row_fail[t] == 0))
        return;   // decided by the first pass
    // entries below the row's final threshold bound cannot be among its top k
    const uint32_t floor_ord = p.gtau ? p.gtau[t] : 0u;
    // copy the entries that pass the floor into shared memory (order is irrelevant:
    // the selection is by unique composite keys); every pass below reads them there.
    // One warp per sub-list, which reads its own length, so the sub-lists' loads
    // are in flight together.
    {
        const int lane = threadIdx.x & 31;
        uint32_t omin = 0xFFFFFFFFu, omax = 0u;
        for (int s = threadIdx.x >> 5; s < nslots; s += kSelThreads / 32) {
            const uint32_t raw = p.counts[cbase + s];
            const int c = static_cast<int>(min(raw, static_cast<uint32_t>(pc.cap)));
            if (lane == 0) {
                if (raw > static_cast<uint32_t>(pc.cap))
                    s_overflow = 1;   // benign race: every writer stores 1
                atomicAdd(&s_nall, c);
            }
            const uint2* src = p.lists + lbase + (int64_t)s * pc.cap;
            for (int i0 = 0; i0 < c; i0 += 32 * 8) {
                // eight loads in flight per lane before any of them is used
                // (clamped indices: no load result is selected on, so all eight
                // are in flight at once; entries past c are dropped below)
                uint2 ent[8];
#pragma unroll
                for (int u = 0; u < 8; ++u)
                    ent[u] = src[min(i0 + u * 32 + lane, c - 1)];
                // the round's passing entries: one shared atomic reserves the warp's room
                uint32_t passm = 0;
                int round = 0, mine = 0;
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int i = i0 + u * 32 + lane;
                    const uint32_t o = f2ord(__uint_as_float(ent[u].x));
                    const bool pass = i < c && o >= floor_ord;
                    const uint32_t m = __ballot_sync(0xffffffffu, pass);
                    if (pass) {
                        passm |= 1u << u;
                        omin = min(omin, o);
                        omax = max(omax, o);
                    }
                    round += __popc(m);
                    mine += __popc(m & ((1u << lane) - 1u));
                }
                if (round == 0)
                    continue;
                int base = 0;
                if (lane == 0)
                    base = atomicAdd(&s_staged, round);
                base = __shfl_sync(0xffffffffu, base, 0);
                // lane's entries go after the lower lanes' entries of the round
                int pos = base + mine;
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    if (passm & (1u << u)) {
                        if (pos < kStageEntries)
                            stage[pos] = ent[u];
                        ++pos;
                    }
                }
            }
        }
        omin = __reduce_min_sync(0xffffffffu, omin);
        omax = __reduce_max_sync(0xffffffffu, omax);
        if (lane == 0 && omin <= omax) {
            atomicMin(&s_omin, omin);
            atomicMax(&s_omax, omax);
        }
    }
    __syncthreads();
    const int n_all = s_nall;
    if (p.verify) {
        // the lists hold every entry at or above the row's threshold unless a
        // sub-list overflowed; they decide the row iff that holds and they have
        // at least k entries (or the threshold let everything through)
        const bool decided = s_overflow == 0 && (p.tau_row[t] == 0u || n_all >= p.k);
        if (!decided) {
            if (threadIdx.x == 0) {
                p.row_fail[t] = 1u;
                atomicOr(p.fail_any, 1u);
            }
            return;
        }
    }
    const bool staged = s_staged <= kStageEntries;
    const int n = staged ? s_staged : n_all;
    if (!staged) {
        // the entries stay in the lists: exclusive prefix of the sub-list lengths
        if (threadIdx.x < 32) {
            int carry = 0;
            for (int s0 = 0; s0 < nslots; s0 += 32) {
                const int s = s0 + static_cast<int>(threadIdx.x);
                const int c = s < nslots ? static_cast<int>(min(p.counts[cbase + s],
                                                                static_cast<uint32_t>(pc.cap)))
                                         : 0;
                int incl = c;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const int y = __shfl_up_sync(0xffffffffu, incl, o);
                    if ((threadIdx.x & 31) >= static_cast<unsigned>(o))
                        incl += y;
                }
                if (s < nslots)
                    s_off[s] = carry + incl - c;
                carry += __shfl_sync(0xffffffffu, incl, 31);
            }
            if (threadIdx.x == 0)
                s_off[nslots] = carry;
        }
        __syncthreads();
    }
    const int k = p.k;
    // bitmap words for this row's key indices (0: too many keys, sort instead)
    const int row_words = (pc.key_count + 31) / 32;
    const int nw_row = p.bitmap && row_words <= kBitmapWords ? max(row_words, 1) : 0;
    if (staged && !p.mask && nw_row > 0) {
        // threshold over the staged entries, then the kept keys in ascending order
        // straight from a bitmap: no ordered emission, no sort
        auto load = [&](int e, uint32_t& hi, uint32_t& lo) {
            const uint2 ent = stage[e];
            hi = f2ord(__uint_as_float(ent.x));
            lo = ~ent.y;
        };
        // --- value buckets (the scratch below is the bitmap's, free until then)
        uint32_t* bhist = reinterpret_cast<uint32_t*>(skey);
        uint64_t* bcand = reinterpret_cast<uint64_t*>(bhist + kBuckets);
        const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
        for (int i = threadIdx.x; i < kBuckets; i += kSelThreads)
            bhist[i] = 0;
        if (threadIdx.x == 0)
            s_bcount = 0;
        __syncthreads();
        BucketThr bt;
        {
            // the staged entries' range, gathered while staging
            const uint32_t a = s_omin, b = s_omax;
            bt.vmin = ord2f(a);
            const float range = __fsub_rn(ord2f(b), bt.vmin);
            bt.scale = range > 0.0f ? __fdiv_rn(static_cast<float>(kBuckets), range) : 0.0f;
        }
        const bool use_buckets = n > k && bt.scale > 0.0f && bt.scale < INFINITY;
        bool resolved = false;
        if (n <= k) {
            bt.boundary = -1;                 // every staged entry is kept
            resolved = true;
        }
        if (use_buckets) {
            for (int e = threadIdx.x; e < n; e += kSelThreads)
                atomicAdd(&bhist[bt.bucket(__uint_as_float(stage[e].x))], 1u);
            __syncthreads();
            // suffix counts: thread t owns buckets [2048 - 4(t+1), 2048 - 4t)
            constexpr int kPer = kBuckets / kSelThreads;
            const int top = kBuckets - kPer * threadIdx.x;
            uint32_t c[kPer], local = 0;
#pragma unroll
            for (int x = 0; x < kPer; ++x) {
                c[x] = bhist[top - 1 - x];
                local += c[x];
            }
            const uint32_t above_me = block_exclusive_sum(local, sh);
            if (above_me < static_cast<uint32_t>(k) && above_me + local >= static_cast<uint32_t>(k)) {
                uint32_t cum = above_me;
#pragma unroll
                for (int x = 0; x < kPer; ++x) {
                    if (cum + c[x] >= static_cast<uint32_t>(k)) {
                        s_bnd = top - 1 - x;
                        s_need = static_cast<int>(k - cum);
                        s_bsize = static_cast<int>(c[x]);
                        break;
                    }
                    cum += c[x];
                }
            }
            __syncthreads();
            bt.boundary = s_bnd;
            const int need = s_need, bsize = s_bsize;
            if (bsize == need) {
                bt.cut = 0;                   // the whole boundary bucket is kept
                resolved = true;
            } else if (bsize <= kBucketCands) {
                for (int e = threadIdx.x; e < n; e += kSelThreads) {
                    const uint2 ent = stage[e];
                    const float v = __uint_as_float(ent.x);
                    if (bt.bucket(v) == bt.boundary)
                        bcand[atomicAdd(&s_bcount, 1)] =
                            (static_cast<uint64_t>(f2ord(v)) << 32) | ~ent.y;
                }
                __syncthreads();
                // the need-th largest candidate: the one with exactly need-1 above it
                for (int i = threadIdx.x; i < bsize; i += kSelThreads) {
                    const uint64_t mine = bcand[i];
                    int rank = 0;
                    for (int x = 0; x < bsize; ++x)
                        rank += bcand[x] > mine;
                    if (rank == need - 1)
                        s_cut = mine;
                }
                __syncthreads();
                bt.cut = s_cut;
                resolved = true;
            }
        }
        CompositeThr thr{0u, 0u, 0u, 0u};
        if (!resolved) {
            bt.boundary = -1;                 // not used: the radix threshold decides
            thr = group_threshold<kSelThreads>(sh, threadIdx.x, n, static_cast<uint32_t>(k),
                                               load, CtaSync{});
        }
        auto keep_entry = [&](uint32_t hi, uint32_t lo) {
            return resolved ? bt.kept(ord2f(hi), ~lo) : thr.kept(hi, lo);
        };
        __syncthreads();                      // the bucket scratch becomes the bitmap
        uint32_t* bits = reinterpret_cast<uint32_t*>(skey);
        uint32_t* wpre = bits + kBitmapWords;
        const int nw = nw_row;
        for (int w = threadIdx.x; w < nw; w += kSelThreads)
            bits[w] = 0;
        __syncthreads();
        for (int e = threadIdx.x; e < n; e += kSelThreads) {
            uint32_t hi, lo;
            load(e, hi, lo);
            if (hi > kOrdNegInf && keep_entry(hi, lo))
                atomicOr(&bits[(~lo) >> 5], 1u << ((~lo) & 31));
        }
        __syncthreads();
        const int total = bitmap_prefix(bits, wpre, nw, sh, s_total);
        int32_t* oi = p.out_idx + (int64_t)t * k;
        float* ov = p.out_val ? p.out_val + (int64_t)t * k : nullptr;
        // a row's list entries have distinct keys, so an entry is kept iff its key's
        // bit is set
        for (int e = threadIdx.x; e < n; e += kSelThreads) {
            const uint2 ent = stage[e];
            const uint32_t j = ent.y;
            const uint32_t word = bits[j >> 5];
            if ((word >> (j & 31)) & 1u) {
                const int pos = static_cast<int>(wpre[j >> 5] +
                                                 __popc(word & ((1u << (j & 31)) - 1u)));
                oi[pos] = static_cast<int32_t>(j);
                if (ov)
                    ov[pos] = __uint_as_float(ent.x);
            }
        }
        for (int i = total + threadIdx.x; i < k; i += kSelThreads) {
            oi[i] = -1;
            if (ov)
                ov[i] = -INFINITY;
        }
        return;
    }
    for (int i = threadIdx.x; i < n2; i += kSelThreads) {
        skey[i] = INT32_MAX;
        sval[i] = -INFINITY;
    }
    __syncthreads();
    auto emit = [&](int pos, int e, float v, int32_t j) {
        (void)e;
        skey[pos] = j;
        sval[pos] = v;
    };
    int count;
    if (staged) {
        auto load = [&](int e, float& v, int32_t& j) {
            const uint2 ent = stage[e];
            v = __uint_as_float(ent.x);
            j = static_cast<int32_t>(ent.y);
        };
        count = cta_topk(sh, n, k, load, emit);
    } else {
        auto load = [&](int e, float& v, int32_t& j) {
            int lo = 0, hi = nslots - 1;   // the slot s with s_off[s] <= e < s_off[s + 1]
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if (s_off[mid] <= e)
                    lo = mid;
                else
                    hi = mid - 1;
            }
            const uint2 ent = p.lists[lbase + (int64_t)lo * pc.cap + (e - s_off[lo])];
            v = __uint_as_float(ent.x);
            if (f2ord(v) < floor_ord)
                v = -INFINITY;
            j = static_cast<int32_t>(ent.y);
        };
        count = cta_topk(sh, n, k, load, emit);
    }
    __syncthreads();
    if (p.mask) {
        uint8_t* m = p.mask + (t + pc.mask_delta) * p.ld_mask;
        const int64_t n = p.ld_mask;
        if (n > static_cast<int64_t>(kStageEntries) * 64 - 64) {
            // (a mask row longer than the staging area holds as a bitmap)
            for (int64_t b = threadIdx.x; b < n; b += kSelThreads)
                m[b] = 0;
            __syncthreads();
            for (int i = threadIdx.x; i < count; i += kSelThreads)
                if (skey[i] >= 0 && skey[i] < n)
                    m[skey[i]] = 1;
            return;
        }
        // the kept blocks as a bitmap in the staging area (free now), then the row in
        // one pass: bytes up to a 16-byte boundary, 16 bytes per store, the tail
        uint32_t* bits = reinterpret_cast<uint32_t*>(stage);
        const int nwords = static_cast<int>((n + 31) / 32) + 1;
        for (int w = threadIdx.x; w < nwords; w += kSelThreads)
            bits[w] = 0;
        __syncthreads();
        for (int i = threadIdx.x; i < count; i += kSelThreads)
            if (skey[i] >= 0 && skey[i] < n)
                atomicOr(&bits[skey[i] >> 5], 1u << (skey[i] & 31));
        __syncthreads();
        auto bit = [&](int64_t b) -> uint32_t { return (bits[b >> 5] >> (b & 31)) & 1u; };
        const int64_t head = min(n, static_cast<int64_t>((16 - (reinterpret_cast<uintptr_t>(m) & 15)) & 15));
        for (int64_t b = threadIdx.x; b < head; b += kSelThreads)
            m[b] = static_cast<uint8_t>(bit(b));
        const int64_t nvec = (n - head) / 16;
        uint4* mv = reinterpret_cast<uint4*>(m + head);
        for (int64_t v = threadIdx.x; v < nvec; v += kSelThreads) {
            const int64_t b0 = head + v * 16;
            const int sh = static_cast<int>(b0 & 31);
            const uint64_t two = static_cast<uint64_t>(bits[b0 >> 5]) |
                                 (static_cast<uint64_t>(bits[(b0 >> 5) + 1]) << 32);
            const uint32_t x = static_cast<uint32_t>(two >> sh) & 0xFFFFu;   // 16 block flags
            // four flags -> four bytes of 0 / 1
            auto spread = [](uint32_t nib) { return (nib * 0x00204081u) & 0x01010101u; };
            mv[v] = make_uint4(spread(x & 15u), spread((x >> 4) & 15u), spread((x >> 8) & 15u),
                               spread(x >> 12));
        }
        for (int64_t b = head + nvec * 16 + threadIdx.x; b < n; b += kSelThreads)
            m[b] = static_cast<uint8_t>(bit(b));
        return;
    }
    int32_t* oi = p.out_idx + (int64_t)t * k;
    float* ov = p.out_val ? p.out_val + (int64_t)t * k : nullptr;
    if (nw_row > 0) {
        // ascending key order without a sort: a bitmap of the kept keys (in the
        // staging area, free now) and an exclusive scan of its word popcounts give
        // every kept key its output position directly
        uint32_t* bits = reinterpret_cast<uint32_t*>(stage);
        uint32_t* wpre = bits + kBitmapWords;
        const int nw = nw_row;
        for (int w = threadIdx.x; w < nw; w += kSelThreads)
            bits[w] = 0;
        __syncthreads();
        for (int i = threadIdx.x; i < count; i += kSelThreads)
            atomicOr(&bits[skey[i] >> 5], 1u << (skey[i] & 31));
        __syncthreads();
        bitmap_prefix(bits, wpre, nw, sh, s_total);
        for (int i = threadIdx.x; i < count; i += kSelThreads) {
            const int j = skey[i];
            const int pos = static_cast<int>(wpre[j >> 5] +
                                             __popc(bits[j >> 5] & ((1u << (j & 31)) - 1u)));
            oi[pos] = j;
            if (ov)
                ov[pos] = sval[i];
        }
        for (int i = count + threadIdx.x; i < k; i += kSelThreads) {
            oi[i] = -1;
            if (ov)
                ov[i] = -INFINITY;
        }
        return;
    }
    bitonic_sort(skey, sval, n2);
    for (int i = threadIdx.x; i < k; i += kSelThreads) {
        const bool have = i < count;
        oi[i] = have ? skey[i] : -1;
        if (ov)
            ov[i] = have ? sval[i] : -INFINITY;
    }
}

// ------------------------------------------------- sampled row thresholds

// tau[t] = the smallest ord among the samples of row t that lie in or above
// the value bucket holding its rank-th largest finite sample (2048 equal-width
// buckets between the row's smallest and largest finite sample), or 0 when the
// row has fewer than rank finite samples.  At least rank samples are at or
// above it.  Any threshold keeps the selection exact (rows the lists cannot
// decide are selected again); this one is close to the rank-th sample.
// POOLED: the ranked entries are block maxima (p.pool > 1); the key version keeps
// its registers low enough for four CTAs per SM.
template <bool POOLED>
__global__ void __launch_bounds__(kSelThreads, 2048 / kSelThreads)
    sample_threshold_kernel(const __grid_constant__ SampleParams p)
{
    __shared__ Scratch sh;
    __shared__ uint32_t bhist[kBuckets];
    __shared__ int s_bnd;
    extern __shared__ __align__(16) float srow[];
    const int t = p.row0 + blockIdx.x;
    const int req = find_request(p.req_row_begin, p.num_requests, t);
    const int stride = p.req_rank[req];     // sampling stride (0: not sampled)
    const int clen = min(p.compress_len[t], p.req_key_count[req]);
    const int pool = POOLED ? p.pool : 1;
    const int units = (clen + pool - 1) / pool;   // keys, or blocks, the row ranks
    uint32_t* tau_out = p.tau_row + t;
    // rows that keep every entry: unsampled requests and rows with at most k keys
    // (blocks)
    if (stride == 0 || units <= p.k) {
        if (threadIdx.x == 0)
            *tau_out = 0u;
        return;
    }
    const int64_t ld = p.ld;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const float* row = p.samples + (int64_t)blockIdx.x * ld;
    // the row once into shared memory (ld is a multiple of 128: float4 loads), with
    // the range and the count of its finite samples (keys)
    uint32_t omin = 0xFFFFFFFFu, omax = 0u, cnt = 0;
    auto count = [&](float v) {
        const uint32_t o = f2ord(v);
        if (o > kOrdNegInf) {
            omin = min(omin, o);
            omax = max(omax, o);
            ++cnt;
        }
    };
    // only the columns the request's sampled tiles fill (a row of a request with fewer
    // sampled tiles than the widest one leaves the rest of its sample row unwritten)
    const int cols = p.req_cols[req] > 0 ? min(p.req_cols[req], static_cast<int>(ld))
                                         : static_cast<int>(ld);
    for (int e = threadIdx.x; e < cols / 4; e += kSelThreads) {
        const float4 v4 = reinterpret_cast<const float4*>(row)[e];
        reinterpret_cast<float4*>(srow)[e] = v4;
        if constexpr (!POOLED) {
            count(v4.x);
            count(v4.y);
            count(v4.z);
            count(v4.w);
        }
    }
    // blocks: the maximum of each aligned pool-key group (sampled tiles are whole
    // 128-key tiles, so every group is a whole block of the row), then their range
    // and count
    const int n = cols / pool;
    float* vals = srow;
    if constexpr (POOLED) {
        __syncthreads();
        vals = srow + ld;
        for (int b = threadIdx.x; b < n; b += kSelThreads) {
            float m = -INFINITY;
            for (int x = 0; x < pool; ++x)
                m = fmaxf(m, srow[b * pool + x]);
            vals[b] = m;
            count(m);
        }
    }
    for (int i = threadIdx.x; i < kBuckets; i += kSelThreads)
        bhist[i] = 0;
    omin = __reduce_min_sync(0xffffffffu, omin);
    omax = __reduce_max_sync(0xffffffffu, omax);
    cnt = __reduce_add_sync(0xffffffffu, cnt);
    if (lane == 0) {
        sh.hist[0][warp] = omin;
        sh.hist[1][warp] = omax;
        sh.warp_sum[warp] = cnt;
    }
    __syncthreads();
    uint32_t a = 0xFFFFFFFFu, b = 0u, m = 0;
    for (int w = 0; w < kSelThreads / 32; ++w) {
        a = min(a, sh.hist[0][w]);
        b = max(b, sh.hist[1][w]);
        m += sh.warp_sum[w];
    }
    // mu = samples expected among the row's top k: k times the sampled fraction,
    // which is m / units for a short row (its first tile is always sampled) and
    // 1 / stride when a candidate mask leaves fewer eligible keys than clen; the
    // threshold is the sample of rank mu + 5 sqrt(mu) + 4
    const float frac = fmaxf(static_cast<float>(m) / static_cast<float>(units),
                             1.0f / static_cast<float>(stride));
    const float mu = static_cast<float>(p.k) * frac;
    const int rank = static_cast<int>(ceilf(mu + 5.0f * sqrtf(mu) + 4.0f));
    if (m < static_cast<uint32_t>(rank)) {
        if (threadIdx.x == 0)
            *tau_out = 0u;
        return;
    }
    BucketThr bt;
    bt.vmin = ord2f(a);
    const float range = __fsub_rn(ord2f(b), bt.vmin);
    bt.scale = range > 0.0f ? __fdiv_rn(static_cast<float>(kBuckets), range) : 0.0f;
    if (!(bt.scale < INFINITY))
        bt.scale = 0.0f;                      // degenerate range: one bucket
    __syncthreads();                          // (sh is reused by the scan below)
    for (int e = threadIdx.x; e < n; e += kSelThreads) {
        const float v = vals[e];
        if (f2ord(v) > kOrdNegInf)
            atomicAdd(&bhist[bt.bucket(v)], 1u);
    }
    __syncthreads();
    constexpr int kPer = kBuckets / kSelThreads;
    const int top = kBuckets - kPer * threadIdx.x;
    uint32_t c[kPer], local = 0;
#pragma unroll
    for (int x = 0; x < kPer; ++x) {
        c[x] = bhist[top - 1 - x];
        local += c[x];
    }
    const uint32_t above_me = block_exclusive_sum(local, sh);
    const uint32_t r = static_cast<uint32_t>(rank);
    if (above_me < r && above_me + local >= r) {
        uint32_t cum = above_me;
#pragma unroll
        for (int x = 0; x < kPer; ++x) {
            if (cum + c[x] >= r) {
                s_bnd = top - 1 - x;
                break;
            }
            cum += c[x];
        }
    }
    __syncthreads();
    const int bnd = s_bnd;
    uint32_t tmin = 0xFFFFFFFFu;
    for (int e = threadIdx.x; e < n; e += kSelThreads) {
        const float v = vals[e];
        const uint32_t o = f2ord(v);
        if (o > kOrdNegInf && bt.bucket(v) >= bnd)
            tmin = min(tmin, o);
    }
    tmin = __reduce_min_sync(0xffffffffu, tmin);
    if (lane == 0)
        sh.hist[0][warp] = tmin;
    __syncthreads();
    if (threadIdx.x == 0) {
        uint32_t x = 0xFFFFFFFFu;
        for (int w = 0; w < kSelThreads / 32; ++w)
            x = min(x, sh.hist[0][w]);
        *tau_out = x;
    }
}

// ------------------------------------------------------- standalone top-k

__global__ void __launch_bounds__(kSelThreads) topk_dense_kernel(const __grid_constant__ TopkParams p)
{
    __shared__ Scratch sh;
    const int t = blockIdx.x;
    if (p.row_fail != nullptr && (*p.fail_any == 0u || p.row_fail[t] == 0u))
        return;   // decided by the sampled pass
    const int r = find_request(p.req_row_begin, p.num_requests, t);
    const int n = max(0, min(p.compress_len[t], p.req_key_count[r]));
    const float* row = p.logits + (int64_t)t * p.ld;
    int32_t* oi = p.out_idx + (int64_t)t * p.k;
    float* ov = p.out_val ? p.out_val + (int64_t)t * p.k : nullptr;
    auto load = [&](int e, float& v, int32_t& j) {
        v = row[e];
        j = e;
    };
    auto emit = [&](int pos, int e, float v, int32_t j) {
        (void)e;
        oi[pos] = j;
        if (ov)
            ov[pos] = v;
    };
    const int count = cta_topk(sh, n, p.k, load, emit);
    for (int i = count + threadIdx.x; i < p.k; i += kSelThreads) {
        oi[i] = -1;
        if (ov)
            ov[i] = -INFINITY;
    }
}

// ------------------------------------------- sampled top-k over caller logits

__device__ __forceinline__ int dense_piece(const DenseFilterParams& p, int t)
{
    int i = 0;
    while (i + 1 < p.num_pieces && p.piece[i + 1].row_begin <= t)
        ++i;
    return i;
}

// One CTA per row of the pass: sample column e reads key (e / 128) * stride * 128 +
// e % 128 of the row, -inf at or past the row's length; rows of unsampled requests
// are left alone (threshold 0).  VEC: 16-byte aligned rows, four columns per load (a
// group of four never straddles a 128-key tile).
template <bool VEC>
__global__ void __launch_bounds__(256) dense_gather_kernel(const __grid_constant__ DenseFilterParams p)
{
    const int t = p.piece[0].row_begin + static_cast<int>(blockIdx.x);
    const DensePiece& pc = p.piece[dense_piece(p, t)];
    if (t >= pc.row_begin + pc.nrows)
        return;                          // a gap between pieces
    const int stride = p.req_stride[pc.request];
    if (stride == 0)
        return;
    const int clen = min(p.compress_len[t], p.req_key_count[pc.request]);
    const float* row = p.logits + (int64_t)t * p.ld;
    float* out = p.samples + (int64_t)blockIdx.x * p.sample_cols;
    if constexpr (VEC) {
        for (int e = 4 * static_cast<int>(threadIdx.x); e < p.sample_cols; e += 4 * blockDim.x) {
            const int j = (e / kTileKeys) * stride * kTileKeys + (e % kTileKeys);
            float4 x = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
            if (j + 3 < clen) {
                x = *reinterpret_cast<const float4*>(row + j);
            } else {
                if (j < clen) x.x = row[j];
                if (j + 1 < clen) x.y = row[j + 1];
                if (j + 2 < clen) x.z = row[j + 2];
            }
            *reinterpret_cast<float4*>(out + e) = x;
        }
    } else {
        for (int e = threadIdx.x; e < p.sample_cols; e += blockDim.x) {
            const int j = (e / kTileKeys) * stride * kTileKeys + (e % kTileKeys);
            out[e] = j < clen ? row[j] : -INFINITY;
        }
    }
}

// grid (key chunks, rows of the pass): every entry of the chunk at or above the row's
// threshold (ord; 0 passes every finite entry) goes to the chunk's own list of the
// row, which no other CTA writes.  The chunk's keys are read before the row's causal
// length arrives (bounded by the request's key count, a launch parameter), so the
// loads do not wait on it.  VEC: rows are 16-byte aligned (aligned base, ld a multiple
// of 4), a thread reads four entries per load with U loads (128 bytes) in flight;
// otherwise one entry per load.  Positions come from a block-wide scan of the
// threads' pass counts, and the list length is written once at the end.
constexpr int kFilterThreads = 128;

template <bool VEC>
__global__ void __launch_bounds__(kFilterThreads) dense_filter_kernel(const __grid_constant__ DenseFilterParams p)
{
    constexpr int U = 8;                      // loads in flight per thread
    constexpr int W = VEC ? 4 : 1;            // entries per load
    constexpr int PER = U * W;                // entries per thread per round
    constexpr int NW = kFilterThreads / 32;
    __shared__ uint32_t s_warp[NW];
    const int t = p.piece[0].row_begin + static_cast<int>(blockIdx.y);
    const DensePiece& pc = p.piece[dense_piece(p, t)];
    if (t >= pc.row_begin + pc.nrows || static_cast<int>(blockIdx.x) >= pc.slots)
        return;
    const int L = p.req_key_count[pc.request];
    const int j0 = static_cast<int>(blockIdx.x) * pc.chunk;
    const int jmax = min(L, j0 + pc.chunk);
    if (j0 >= jmax)
        return;
    const float* row = p.logits + (int64_t)t * p.ld;
    const int clen_raw = p.compress_len[t];
    const uint32_t tau = p.tau_row[t];
    const int64_t list0 = pc.list_offset + ((int64_t)(t - pc.row_begin) * pc.slots + blockIdx.x) * pc.cap;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint32_t cap = static_cast<uint32_t>(pc.cap);
    uint32_t total = 0;   // entries of the chunk appended so far (same in every thread)
    for (int jb = j0; jb < jmax; jb += kFilterThreads * PER) {
        float v[PER];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int j = jb + (u * kFilterThreads + static_cast<int>(threadIdx.x)) * W;
            if constexpr (VEC) {
                // j is a multiple of 4 and j < jmax <= ld keeps the whole load inside
                // the row; a load at or past jmax is replaced by -inf
                float4 x = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
                if (j < jmax)
                    x = __ldcs(reinterpret_cast<const float4*>(row + j));
                v[4 * u] = x.x;
                v[4 * u + 1] = x.y;
                v[4 * u + 2] = x.z;
                v[4 * u + 3] = x.w;
            } else {
                v[u] = j < jmax ? __ldcs(row + j) : -INFINITY;
            }
        }
        const int j1 = min(jmax, clen_raw);
        uint32_t pass = 0;
#pragma unroll
        for (int e = 0; e < PER; ++e) {
            const int j = jb + ((e / W) * kFilterThreads + static_cast<int>(threadIdx.x)) * W + e % W;
            const uint32_t o = f2ord(v[e]);
            if (j < j1 && o > kOrdNegInf && o >= tau)
                pass |= 1u << e;
        }
        const uint32_t c = __popc(pass);
        uint32_t incl = c;   // inclusive scan of the counts over the warp, then the CTA
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o)
                incl += y;
        }
        if (lane == 31)
            s_warp[warp] = incl;
        __syncthreads();
        uint32_t before = 0, round = 0;
#pragma unroll
        for (int w = 0; w < NW; ++w) {
            const uint32_t x = s_warp[w];
            before += w < warp ? x : 0u;
            round += x;
        }
        __syncthreads();
        uint32_t pos = total + before + incl - c;
#pragma unroll
        for (int e = 0; e < PER; ++e) {
            if (pass & (1u << e)) {
                const int j = jb + ((e / W) * kFilterThreads + static_cast<int>(threadIdx.x)) * W + e % W;
                if (pos < cap)
                    p.lists[list0 + pos] = make_uint2(__float_as_uint(v[e]), static_cast<uint32_t>(j));
                ++pos;
            }
        }
        total += round;
    }
    if (threadIdx.x == 0)
        p.counts[pc.count_offset + (int64_t)(t - pc.row_begin) * pc.slots + blockIdx.x] = total;
}

}  // namespace

cudaError_t launch_dense_gather(const DenseFilterParams& p, int rows, cudaStream_t stream)
{
    if (rows <= 0)
        return cudaSuccess;
    // samples rows are sample_cols (a multiple of 128) floats apart in the workspace
    const bool vec = (reinterpret_cast<uintptr_t>(p.logits) % 16) == 0 && p.ld % 4 == 0 &&
                     (reinterpret_cast<uintptr_t>(p.samples) % 16) == 0;
    if (vec)
        dense_gather_kernel<true><<<rows, 256, 0, stream>>>(p);
    else
        dense_gather_kernel<false><<<rows, 256, 0, stream>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_dense_filter(const DenseFilterParams& p, int rows, int max_slots,
                                cudaStream_t stream)
{
    if (rows <= 0 || max_slots <= 0)
        return cudaSuccess;
    const dim3 grid(max_slots, rows);
    const bool vec = (reinterpret_cast<uintptr_t>(p.logits) % 16) == 0 && p.ld % 4 == 0;
    if (vec)
        dense_filter_kernel<true><<<grid, kFilterThreads, 0, stream>>>(p);
    else
        dense_filter_kernel<false><<<grid, kFilterThreads, 0, stream>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_stream_merge(const StreamMergeParams& p, cudaStream_t stream)
{
    if (p.total_ctas <= 0)
        return cudaSuccess;
    if (p.k > kMaxSortK)
        return cudaErrorInvalidValue;
    int n2 = 1;
    while (n2 < p.k)
        n2 <<= 1;
    const size_t dyn = sizeof(uint2) * kStageEntries +
                       std::max<size_t>((sizeof(int32_t) + sizeof(float)) * n2, 8 * kBitmapWords);
    cudaError_t e = cudaFuncSetAttribute(stream_merge_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dyn);
    if (e != cudaSuccess)
        return e;
    stream_merge_kernel<<<p.total_ctas, kSelThreads, dyn, stream>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_sample_threshold(const SampleParams& p, cudaStream_t stream)
{
    if (p.rows <= 0)
        return cudaSuccess;
    if (p.ld % 4 != 0 || p.ld > 16384)
        return cudaErrorInvalidValue;
    const bool pooled = p.pool > 1;
    const size_t dyn = (p.ld + (pooled ? p.ld / p.pool : 0)) * sizeof(float);
    auto kern = pooled ? sample_threshold_kernel<true> : sample_threshold_kernel<false>;
    if (dyn > 48 * 1024) {
        cudaError_t e =
            cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dyn);
        if (e != cudaSuccess)
            return e;
    }
    kern<<<p.rows, kSelThreads, dyn, stream>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_topk_dense(const TopkParams& p, cudaStream_t stream)
{
    if (p.total_rows <= 0)
        return cudaSuccess;
    topk_dense_kernel<<<p.total_rows, kSelThreads, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace idx
