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
#include <algorithm>

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
// dynamic shared memory of the merge: [stage: kStageEntries x 8 B][scratch: keys and
// values n2 x 4 B each, or the bitmap and its prefix] (output rows go straight to global
// memory)
__host__ __device__ constexpr size_t merge_smem_bytes(int n2)
{
    return 8 * (size_t)kStageEntries + (8 * (size_t)n2 > 8 * (size_t)kBitmapWords
                                            ? 8 * (size_t)n2
                                            : 8 * (size_t)kBitmapWords);
}

// The verify merge of a row whose lists were filled at a sampled threshold tau (every
// listed entry is at or above it) and whose keys fit the bitmap (at most 65,536): the
// entries go to shared memory at the prefix of the sub-list lengths, bucketed on the way
// (2048 equal-width buckets from tau to the row's largest sample; larger values share
// the top bucket) with the bucket kept in the upper 16 bits of the entry's key field;
// then the boundary bucket, the bitmap of kept keys and the ordered output as in the
// general path.  Returns false, having written nothing to global memory, when the row
// needs the general path (no sampled range, more entries than the staging area holds,
// a boundary bucket too large to rank directly); true when the row is done (flagged or
// written).  Every thread calls it; the result is the same in all of them.
__device__ __forceinline__ bool merge_row_verified(const StreamMergeParams& p, const MergePiece& pc,
                                                   const int t, const int64_t lbase,
                                                   const int64_t cbase, const int n2,
                                                   uint8_t* dyn, Scratch& sh)
{
    __shared__ uint32_t v_cnt[kMaxStreamSlots];
    __shared__ int v_bcount, v_total;
    __shared__ uint64_t v_cut;
    const uint32_t tau = p.tau_row[t];
    const uint32_t smax = p.smax_row[t];
    const int nslots = pc.slots, cap = pc.cap;
    // (a candidate-mask merge ranks blocks: its bitmap spans the mask row)
    const int row_words = p.mask ? static_cast<int>((p.ld_mask + 31) / 32) : (pc.key_count + 31) / 32;
    if (tau <= kOrdNegInf || smax <= tau || !(p.bitmap || p.mask) || cap <= 0)
        return false;
    // rows of at most 65,536 keys keep the bucket in the upper 16 bits of the key field and
    // write the kept keys in order from a bitmap; longer rows recompute the bucket and sort
    // the kept keys.  A mask row is written from the bitmap (one word past the row's last
    // is read, so it must fit too)
    const bool packed = row_words <= kBitmapWords;
    if (p.mask && row_words + 1 > kBitmapWords)
        return false;
    BucketThr bt;
    bt.vmin = ord2f(tau);
    {
        const float range = __fsub_rn(ord2f(smax), bt.vmin);
        bt.scale = range > 0.0f ? __fdiv_rn(static_cast<float>(kBuckets), range) : 0.0f;
        if (!(bt.scale > 0.0f && bt.scale < INFINITY))
            return false;
    }
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    constexpr int kWarps = kSelThreads / 32;
    uint2* stage = reinterpret_cast<uint2*>(dyn);
    uint32_t* bhist = reinterpret_cast<uint32_t*>(dyn + 8 * (size_t)kStageEntries);
    uint64_t* bcand = reinterpret_cast<uint64_t*>(bhist + kBuckets);
    for (int i = tid; i < kBuckets; i += kSelThreads)
        bhist[i] = 0;
    if (tid == 0)
        v_bcount = 0;
    // the first 256 entries of the warp's first sub-list load together with the counts
    // (indices clamped to the capacity: the loads do not wait for the count)
    uint2 ent[8];
    if (warp < nslots) {
        const uint2* src = p.lists + lbase + (int64_t)warp * cap;
#pragma unroll
        for (int u = 0; u < 8; ++u)
            ent[u] = src[min(u * 32 + lane, cap - 1)];
    }
    int over = 0;
    for (int s = tid; s < nslots; s += kSelThreads) {
        const uint32_t raw = p.counts[cbase + s];
        v_cnt[s] = min(raw, static_cast<uint32_t>(cap));
        over |= raw > static_cast<uint32_t>(cap);
    }
    const int overflow = __syncthreads_or(over);
    uint32_t tot = 0;
    for (int s = lane; s < nslots; s += 32)
        tot += v_cnt[s];
    const int n = static_cast<int>(__reduce_add_sync(0xffffffffu, tot));
    if (overflow || n < p.k) {
        // the lists hold every entry at or above tau unless a sub-list overflowed; with
        // fewer than k of them they cannot decide the row
        if (tid == 0) {
            p.row_fail[t] = 1u;
            atomicOr(p.fail_any, 1u);
        }
        return true;
    }
    if (n > kStageEntries)
        return false;
    for (int s = warp; s < nslots; s += kWarps) {
        uint32_t o = 0;
        for (int x = lane; x < s; x += 32)
            o += v_cnt[x];
        const int off = static_cast<int>(__reduce_add_sync(0xffffffffu, o));
        const int c = static_cast<int>(v_cnt[s]);
        const uint2* src = p.lists + lbase + (int64_t)s * cap;
        for (int i0 = 0; i0 < c; i0 += 256) {
            if (s != warp || i0 > 0) {
#pragma unroll
                for (int u = 0; u < 8; ++u)
                    ent[u] = src[min(i0 + u * 32 + lane, c - 1)];
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int i = i0 + u * 32 + lane;
                if (i < c) {
                    const uint32_t b = static_cast<uint32_t>(bt.bucket(__uint_as_float(ent[u].x)));
                    atomicAdd(&bhist[b], 1u);
                    stage[off + i] =
                        packed ? make_uint2(ent[u].x, (ent[u].y & 0xFFFFu) | (b << 16)) : ent[u];
                }
            }
        }
    }
    __syncthreads();
    // the bucket holding the k-th largest entry, from the top: thread i owns buckets
    // [2048 - 4 (i + 1), 2048 - 4 i)
    const uint32_t k = static_cast<uint32_t>(p.k);
    {
        constexpr int kPer = kBuckets / kSelThreads;
        const int top = kBuckets - kPer * tid;
        uint32_t c4[kPer], local = 0;
#pragma unroll
        for (int x = 0; x < kPer; ++x) {
            c4[x] = bhist[top - 1 - x];
            local += c4[x];
        }
        const uint32_t above_me = block_exclusive_sum(local, sh);
        if (above_me < k && above_me + local >= k) {
            uint32_t cum = above_me;
#pragma unroll
            for (int x = 0; x < kPer; ++x) {
                if (cum + c4[x] >= k) {
                    sh.bcast[0] = static_cast<uint32_t>(top - 1 - x);
                    sh.bcast[1] = k - cum;
                    sh.bcast[2] = c4[x];
                    break;
                }
                cum += c4[x];
            }
        }
        __syncthreads();
    }
    const uint32_t bnd = sh.bcast[0], need = sh.bcast[1], bsize = sh.bcast[2];
    // a staged entry's key, bucket and composite key (ord(score), ~index)
    auto key_of = [&](const uint2 en) { return packed ? (en.y & 0xFFFFu) : en.y; };
    auto bucket_of = [&](const uint2 en) {
        return packed ? (en.y >> 16)
                      : static_cast<uint32_t>(bt.bucket(__uint_as_float(en.x)));
    };
    auto comp = [&](const uint2 en) {
        return (static_cast<uint64_t>(f2ord(__uint_as_float(en.x))) << 32) |
               static_cast<uint32_t>(~key_of(en));
    };
    uint64_t cut = 0;   // the whole boundary bucket is kept when it gives all of its entries
    // rows of the bitmap path collect the boundary bucket's entries during the bitmap pass
    const bool collect = packed && bsize != need;
    if (bsize != need) {
        if (bsize > static_cast<uint32_t>(kBucketCands))
            return false;
    }
    if (bsize != need && !packed) {
        for (int e = tid; e < n; e += kSelThreads) {
            const uint2 en = stage[e];
            if (bucket_of(en) == bnd)
                bcand[atomicAdd(&v_bcount, 1)] = comp(en);
        }
        __syncthreads();
        // the need-th largest candidate: the one with exactly need - 1 above it
        for (int i = tid; i < static_cast<int>(bsize); i += kSelThreads) {
            const uint64_t mine = bcand[i];
            uint32_t rank = 0;
            for (int x = 0; x < static_cast<int>(bsize); ++x)
                rank += bcand[x] > mine;
            if (rank == need - 1)
                v_cut = mine;
        }
        __syncthreads();
        cut = v_cut;
    }
    __syncthreads();   // the bucket scratch becomes the bitmap (or the sort area)
    int32_t* oi = p.out_idx + (int64_t)t * p.k;
    float* ov = p.out_val ? p.out_val + (int64_t)t * p.k : nullptr;
    if (!packed) {
        // the k kept entries (any order), then sorted by key
        int32_t* skey = reinterpret_cast<int32_t*>(bhist);
        float* sval = reinterpret_cast<float*>(skey + n2);
        if (tid == 0)
            v_total = 0;
        for (int i = tid; i < n2; i += kSelThreads) {
            skey[i] = INT32_MAX;
            sval[i] = -INFINITY;
        }
        __syncthreads();
        for (int e = tid; e < n; e += kSelThreads) {
            const uint2 en = stage[e];
            const uint32_t b = bucket_of(en);
            if (b > bnd || (b == bnd && comp(en) >= cut)) {
                const int pos = atomicAdd(&v_total, 1);
                if (pos < n2) {
                    skey[pos] = static_cast<int32_t>(en.y);
                    sval[pos] = __uint_as_float(en.x);
                }
            }
        }
        bitonic_sort(skey, sval, n2);
        __syncthreads();
        const int total = min(v_total, static_cast<int>(k));
        for (int i = tid; i < p.k; i += kSelThreads) {
            const bool have = i < total;
            oi[i] = have ? skey[i] : -1;
            if (ov)
                ov[i] = have ? sval[i] : -INFINITY;
        }
        return true;
    }
    uint32_t* bits = bhist;
    uint32_t* wpre = bits + kBitmapWords;
    const int nw = max(row_words, 1);
    for (int w = tid; w < nw + (p.mask ? 1 : 0); w += kSelThreads)
        bits[w] = 0;
    __syncthreads();
    // f(staged entry) for every staged entry, four loaded before any is used
    auto each_staged = [&](auto&& f) {
        for (int e0 = tid; e0 < n; e0 += 4 * kSelThreads) {
            uint2 en[4];
#pragma unroll
            for (int u = 0; u < 4; ++u)
                en[u] = stage[min(e0 + u * kSelThreads, n - 1)];
#pragma unroll
            for (int u = 0; u < 4; ++u)
                if (e0 + u * kSelThreads < n)
                    f(en[u]);
        }
    };
    // the kept keys: buckets above the boundary one, the whole boundary bucket when it
    // gives all of its entries, else its entries collected (bcand lies past the bitmap,
    // in the prefix area, which is written only after the ranking) and their best `need`
    each_staged([&](const uint2 en) {
        const uint32_t b = en.y >> 16, j = en.y & 0xFFFFu;
        if (b > bnd || (b == bnd && !collect))
            atomicOr(&bits[j >> 5], 1u << (j & 31));
        else if (b == bnd) {
            const int x = atomicAdd(&v_bcount, 1);
            if (x < kBucketCands)
                bcand[x] = comp(en);
        }
    });
    __syncthreads();
    if (collect) {
        // the entries with fewer than `need` above them (composite keys are distinct)
        for (int i = tid; i < static_cast<int>(bsize); i += kSelThreads) {
            const uint64_t mine = bcand[i];
            uint32_t rank = 0;
            for (int x = 0; x < static_cast<int>(bsize); ++x)
                rank += bcand[x] > mine;
            if (rank < need) {
                const uint32_t j = ~static_cast<uint32_t>(mine) & 0xFFFFu;
                atomicOr(&bits[j >> 5], 1u << (j & 31));
            }
        }
        __syncthreads();
    }
    if (p.mask) {
        // the candidate-mask row from the bitmap of kept blocks: bytes up to a 16-byte
        // boundary, 16 bytes per store, the tail; every byte of the row is written
        uint8_t* m = p.mask + (t + pc.mask_delta) * p.ld_mask;
        const int64_t nb = p.ld_mask;
        auto bit = [&](int64_t b) -> uint32_t { return (bits[b >> 5] >> (b & 31)) & 1u; };
        const int64_t head =
            min(nb, static_cast<int64_t>((16 - (reinterpret_cast<uintptr_t>(m) & 15)) & 15));
        for (int64_t b = tid; b < head; b += kSelThreads)
            m[b] = static_cast<uint8_t>(bit(b));
        const int64_t nvec = (nb - head) / 16;
        uint4* mv = reinterpret_cast<uint4*>(m + head);
        for (int64_t v = tid; v < nvec; v += kSelThreads) {
            const int64_t b0 = head + v * 16;
            const int shf = static_cast<int>(b0 & 31);
            const uint64_t two = static_cast<uint64_t>(bits[b0 >> 5]) |
                                 (static_cast<uint64_t>(bits[(b0 >> 5) + 1]) << 32);
            const uint32_t x = static_cast<uint32_t>(two >> shf) & 0xFFFFu;   // 16 block flags
            // four flags -> four bytes of 0 / 1
            auto spread = [](uint32_t nib) { return (nib * 0x00204081u) & 0x01010101u; };
            mv[v] = make_uint4(spread(x & 15u), spread((x >> 4) & 15u), spread((x >> 8) & 15u),
                               spread(x >> 12));
        }
        for (int64_t b = head + nvec * 16 + tid; b < nb; b += kSelThreads)
            m[b] = static_cast<uint8_t>(bit(b));
        return true;
    }
    const int total = bitmap_prefix(bits, wpre, nw, sh, v_total);
    // each kept entry straight to its place in the output row, then the padding
    each_staged([&](const uint2 en) {
        const uint32_t j = en.y & 0xFFFFu;
        const uint32_t word = bits[j >> 5];
        if ((word >> (j & 31)) & 1u) {
            const int pos = static_cast<int>(wpre[j >> 5] + __popc(word & ((1u << (j & 31)) - 1u)));
            oi[pos] = static_cast<int32_t>(j);
            if (ov)
                ov[pos] = __uint_as_float(en.x);
        }
    });
    for (int i = total + tid; i < p.k; i += kSelThreads) {
        oi[i] = -1;
        if (ov)
            ov[i] = -INFINITY;
    }
    return true;
}

// Row `cta` of a merge launch (its rows are numbered across the pieces).  Every thread
// of the CTA calls it; every return is taken by the whole CTA.  FAST: verify merges try
// merge_row_verified first.
template <bool FAST>
__device__ __forceinline__ void merge_row(const StreamMergeParams& p, const int cta)
{
    __shared__ Scratch sh;
    __shared__ int32_t s_off[kMaxStreamSlots + 1];
    extern __shared__ __align__(16) uint8_t dyn[];
    // [stage: kStageEntries x 8 B][keys: n2 x 4 B][values: n2 x 4 B], n2 = k rounded up
    // to a power of two (merge_smem_bytes)
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
    if constexpr (FAST) {
        if (p.verify && p.smax_row != nullptr &&
            merge_row_verified(p, pc, t, lbase, cbase, n2, dyn, sh))
            return;
    }
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
            const uint2* src = p.lists + lbase + (int64_t)s * pc.cap;
            // the first round's entries are loaded together with the count (indices
            // clamped to the sub-list's capacity, not to its count: the loads do not
            // wait for it; entries past the count are dropped below)
            uint2 ent[8];
#pragma unroll
            for (int u = 0; u < 8; ++u)
                ent[u] = pc.cap > 0 ? src[min(u * 32 + lane, pc.cap - 1)] : make_uint2(0u, 0u);
            const uint32_t raw = p.counts[cbase + s];
            const int c = static_cast<int>(min(raw, static_cast<uint32_t>(pc.cap)));
            if (lane == 0) {
                if (raw > static_cast<uint32_t>(pc.cap))
                    s_overflow = 1;   // benign race: every writer stores 1
                atomicAdd(&s_nall, c);
            }
            for (int i0 = 0; i0 < c; i0 += 32 * 8) {
                // eight loads in flight per lane before any of them is used
                // (clamped indices: no load result is selected on, so all eight
                // are in flight at once; entries past c are dropped below)
                if (i0 > 0) {
#pragma unroll
                    for (int u = 0; u < 8; ++u)
                        ent[u] = src[min(i0 + u * 32 + lane, c - 1)];
                }
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
        // bit is set; it goes straight to its position in the output row, then the
        // padding
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

// WALK = false: one row per CTA.  WALK = true (the merge of undecided rows, usually
// none): a grid of one wave walking the rows.  Three CTAs per SM: the staging area
// allows no more.
template <bool WALK>
__global__ void __launch_bounds__(kSelThreads, 3)
    stream_merge_kernel(const __grid_constant__ StreamMergeParams p)
{
    pdl_wait_then_release();
    // a merge of undecided rows with none flagged anywhere has nothing to do (the flag
    // was written by an earlier launch, so every thread reads the same value)
    if (p.only_failed && *p.fail_any == 0u)
        return;
    if constexpr (!WALK) {
        merge_row<true>(p, blockIdx.x);
    } else {
        for (int r = blockIdx.x; r < p.total_ctas; r += gridDim.x) {
            merge_row<false>(p, r);
            __syncthreads();   // the next row resets the shared state
        }
    }
}

// ------------------------------------------------- sampled row thresholds

// tau[t] = the smallest ord among the samples of row t that lie in or above
// the value bucket holding its rank-th largest finite sample (2048 equal-width
// buckets between the row's smallest and largest finite sample), or 0 when the
// row has fewer than rank finite samples.  At least rank samples are at or
// above it.  Any threshold keeps the selection exact (rows the lists cannot
// decide are selected again); this one is close to the rank-th sample.
// One CTA of 128 threads per row, its bucket counts in shared memory; the row is read
// three times (range, counts, threshold): from L2, where the sampled pass just wrote it,
// then from L1.  POOL > 1: the ranked entries are the maxima of aligned POOL-sample
// blocks.
constexpr int kThrThreads = 128;

template <int POOL>
__global__ void __launch_bounds__(kThrThreads, 16)
    sample_threshold_kernel(const __grid_constant__ SampleParams p)
{
    pdl_wait_then_release();
    __shared__ __align__(16) uint32_t hist[kBuckets];
    __shared__ uint32_t s_red[3][kThrThreads / 32];
    __shared__ uint32_t s_bcast[2];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    constexpr int kWarps = kThrThreads / 32;
    const int tl = blockIdx.x;   // row of the launch
    const int t = p.row0 + tl;
    const int req = find_request(p.req_row_begin, p.num_requests, t);
    const int stride = p.req_rank[req];     // sampling stride (0: not sampled)
    const int clen = min(p.compress_len[t], p.req_key_count[req]);
    const int units = (clen + POOL - 1) / POOL;   // keys, or blocks, the row ranks
    uint32_t* tau_out = p.tau_row + t;
    // rows that keep every entry: unsampled requests and rows with at most k keys
    // (blocks)
    if (stride == 0 || units <= p.k) {
        if (tid == 0) {
            *tau_out = 0u;
            p.smax_row[t] = 0u;
        }
        return;
    }
    const float* row = p.samples + (int64_t)tl * p.ld;
    // only the columns the request's sampled tiles fill (a row of a request with fewer
    // sampled tiles than the widest one leaves the rest of its sample row unwritten);
    // a multiple of 128, so every thread's group of 8 samples is whole
    const int cols = p.req_cols[req] > 0 ? min(p.req_cols[req], static_cast<int>(p.ld))
                                         : static_cast<int>(p.ld);
    // samples read from the caller's logits: group b of 8 is keys key0 .. key0 + 7 of
    // the row, key0 = (b / 128) stride 128 + b % 128 (one 128-key tile), keys at or past
    // the row's length read as -inf (a float4 is loaded only when its first key is below
    // it, which keeps it inside the row: ld and key0 are multiples of 4)
    const float* lrow = p.logits ? p.logits + (int64_t)t * p.ld_logits : nullptr;
    // f(v) for every ranked value of the row: thread i takes samples [8 i, 8 i + 8) of
    // every 1024, two such groups in flight per round
    auto visit = [&](auto&& f) {
        constexpr int kGroups = 2;
        for (int b0 = 0; b0 < cols; b0 += kGroups * 8 * kThrThreads) {
            float x[kGroups][8];
#pragma unroll
            for (int u = 0; u < kGroups; ++u) {
                const int b = b0 + (u * kThrThreads + tid) * 8;
                float4 lo = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY), hi = lo;
                if (b < cols) {
                    if (lrow == nullptr) {
                        lo = __ldg(reinterpret_cast<const float4*>(row + b));
                        hi = __ldg(reinterpret_cast<const float4*>(row + b + 4));
                    } else {
                        const int key0 = (b / kTileKeys) * stride * kTileKeys + b % kTileKeys;
                        if (key0 < clen)
                            lo = __ldg(reinterpret_cast<const float4*>(lrow + key0));
                        if (key0 + 4 < clen)
                            hi = __ldg(reinterpret_cast<const float4*>(lrow + key0 + 4));
                        if (key0 + 1 >= clen) lo.y = -INFINITY;
                        if (key0 + 2 >= clen) lo.z = -INFINITY;
                        if (key0 + 3 >= clen) lo.w = -INFINITY;
                        if (key0 + 5 >= clen) hi.y = -INFINITY;
                        if (key0 + 6 >= clen) hi.z = -INFINITY;
                        if (key0 + 7 >= clen) hi.w = -INFINITY;
                    }
                }
                x[u][0] = lo.x; x[u][1] = lo.y; x[u][2] = lo.z; x[u][3] = lo.w;
                x[u][4] = hi.x; x[u][5] = hi.y; x[u][6] = hi.z; x[u][7] = hi.w;
            }
#pragma unroll
            for (int u = 0; u < kGroups; ++u)
#pragma unroll
                for (int g = 0; g < 8 / POOL; ++g) {
                    float m = x[u][g * POOL];
#pragma unroll
                    for (int i = 1; i < POOL; ++i)
                        m = fmaxf(m, x[u][g * POOL + i]);
                    f(m);
                }
        }
    };
    for (int i = tid; i < kBuckets / 4; i += kThrThreads)
        reinterpret_cast<uint4*>(hist)[i] = make_uint4(0u, 0u, 0u, 0u);
    // range and count of the finite ranked values
    uint32_t omin = 0xFFFFFFFFu, omax = 0u, cnt = 0;
    visit([&](float v) {
        const uint32_t o = f2ord(v);
        if (o > kOrdNegInf) {
            omin = min(omin, o);
            omax = max(omax, o);
            ++cnt;
        }
    });
    omin = __reduce_min_sync(0xffffffffu, omin);
    omax = __reduce_max_sync(0xffffffffu, omax);
    cnt = __reduce_add_sync(0xffffffffu, cnt);
    if (lane == 0) {
        s_red[0][warp] = omin;
        s_red[1][warp] = omax;
        s_red[2][warp] = cnt;
    }
    __syncthreads();
    uint32_t m = 0;
    omin = 0xFFFFFFFFu;
    omax = 0u;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
        omin = min(omin, s_red[0][w]);
        omax = max(omax, s_red[1][w]);
        m += s_red[2][w];
    }
    // mu = samples expected among the row's top k: k times the sampled fraction,
    // which is m / units for a short row (its first tile is always sampled) and
    // 1 / stride when a candidate mask leaves fewer eligible keys than clen; the
    // threshold is the sample of rank mu + 5 sqrt(mu) + 4
    const float frac = fmaxf(static_cast<float>(m) / static_cast<float>(units),
                             1.0f / static_cast<float>(stride));
    const float mu = static_cast<float>(p.k) * frac;
    const uint32_t r = static_cast<uint32_t>(ceilf(mu + 5.0f * sqrtf(mu) + 4.0f));
    if (m < r) {
        if (tid == 0) {
            *tau_out = 0u;
            p.smax_row[t] = 0u;
        }
        return;
    }
    BucketThr bt;
    bt.vmin = ord2f(omin);
    const float range = __fsub_rn(ord2f(omax), bt.vmin);
    bt.scale = range > 0.0f ? __fdiv_rn(static_cast<float>(kBuckets), range) : 0.0f;
    if (!(bt.scale < INFINITY))
        bt.scale = 0.0f;                      // degenerate range: one bucket
    visit([&](float v) {
        if (f2ord(v) > kOrdNegInf)
            atomicAdd(&hist[bt.bucket(v)], 1u);
    });
    __syncthreads();
    // the bucket holding the r-th largest value, from the top: thread i owns buckets
    // [2048 - 16 (i + 1), 2048 - 16 i)
    constexpr int kPer = kBuckets / kThrThreads;
    const int top = kBuckets - kPer * tid;
    uint32_t local = 0;
    {
        const uint4* h4 = reinterpret_cast<const uint4*>(hist + top - kPer);
#pragma unroll
        for (int x = 0; x < kPer / 4; ++x) {
            const uint4 c = h4[x];
            local += c.x + c.y + c.z + c.w;
        }
    }
    uint32_t incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o)
            incl += y;
    }
    if (lane == 31)
        s_red[0][warp] = incl;
    __syncthreads();
    uint32_t above = incl - local;
#pragma unroll
    for (int w = 0; w < kWarps; ++w)
        above += w < warp ? s_red[0][w] : 0u;
    if (above < r && above + local >= r) {
        uint32_t cum = above;
        for (int x = 0; x < kPer; ++x) {
            const uint32_t c = hist[top - 1 - x];
            if (cum + c >= r) {
                s_bcast[0] = static_cast<uint32_t>(top - 1 - x);
                break;
            }
            cum += c;
        }
    }
    __syncthreads();
    const int bnd = static_cast<int>(s_bcast[0]);
    uint32_t tmin = 0xFFFFFFFFu;
    visit([&](float v) {
        const uint32_t o = f2ord(v);
        if (o > kOrdNegInf && bt.bucket(v) >= bnd)
            tmin = min(tmin, o);
    });
    tmin = __reduce_min_sync(0xffffffffu, tmin);
    if (lane == 0)
        s_red[1][warp] = tmin;
    __syncthreads();
    if (tid == 0) {
        uint32_t x = 0xFFFFFFFFu;
#pragma unroll
        for (int w = 0; w < kWarps; ++w)
            x = min(x, s_red[1][w]);
        *tau_out = x;
        p.smax_row[t] = omax;
    }
}

// ------------------------------------------------------- standalone top-k

// Exact top-k of one row of caller logits (all threads of the CTA call it).
__device__ __forceinline__ void topk_dense_row(const TopkParams& p, Scratch& sh, const int t)
{
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

// One row per CTA, or (rows the sampled pass left undecided, usually none) a small grid
// walking the flagged rows.
__global__ void __launch_bounds__(kSelThreads) topk_dense_kernel(const __grid_constant__ TopkParams p)
{
    pdl_wait_then_release();
    __shared__ Scratch sh;
    if (p.row_fail != nullptr && *p.fail_any == 0u)
        return;   // every row decided by the sampled pass
    for (int t = blockIdx.x; t < p.total_rows; t += gridDim.x) {
        if (p.row_fail == nullptr || p.row_fail[t] != 0u) {
            topk_dense_row(p, sh, t);
            __syncthreads();   // the next row reuses the scratch
        }
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
    pdl_wait_then_release();
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
    pdl_wait_then_release();
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
    return launch_pdl(vec ? dense_gather_kernel<true> : dense_gather_kernel<false>, dim3(rows),
                      dim3(256), 0, stream, p);
}

cudaError_t launch_dense_filter(const DenseFilterParams& p, int rows, int max_slots,
                                cudaStream_t stream)
{
    if (rows <= 0 || max_slots <= 0)
        return cudaSuccess;
    const dim3 grid(max_slots, rows);
    const bool vec = (reinterpret_cast<uintptr_t>(p.logits) % 16) == 0 && p.ld % 4 == 0;
    return launch_pdl(vec ? dense_filter_kernel<true> : dense_filter_kernel<false>, dim3(grid),
                      dim3(kFilterThreads), 0, stream, p);
}

// SMs of the current device (read once per device)
int sm_count()
{
    static int cached[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return 152;
    if (cached[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            n <= 0)
            n = 152;
        cached[dev] = n;
    }
    return cached[dev];
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
    const size_t dyn = merge_smem_bytes(n2);
    cudaError_t e = cudaFuncSetAttribute(p.only_failed ? stream_merge_kernel<true>
                                                       : stream_merge_kernel<false>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dyn);
    if (e != cudaSuccess)
        return e;
    // the merge of undecided rows: a grid of one wave (it walks the flagged rows, and
    // exits at once when there are none)
    if (p.only_failed)
        return launch_pdl(stream_merge_kernel<true>, dim3(std::min(p.total_ctas, 3 * sm_count())),
                          dim3(kSelThreads), dyn, stream, p);
    return launch_pdl(stream_merge_kernel<false>, dim3(p.total_ctas), dim3(kSelThreads), dyn,
                      stream, p);
}

cudaError_t launch_sample_threshold(const SampleParams& p, cudaStream_t stream)
{
    if (p.rows <= 0)
        return cudaSuccess;
    if (p.ld % 8 != 0 || p.ld > 16384)
        return cudaErrorInvalidValue;
    for (int r = 0; r < p.num_requests; ++r)
        if (p.req_cols[r] % 8 != 0)
            return cudaErrorInvalidValue;
    const int grid = p.rows;
    void (*kern)(SampleParams) = nullptr;
    switch (p.pool) {
    case 1: kern = sample_threshold_kernel<1>; break;
    case 2: kern = sample_threshold_kernel<2>; break;
    case 4: kern = sample_threshold_kernel<4>; break;
    case 8: kern = sample_threshold_kernel<8>; break;
    default: return cudaErrorInvalidValue;
    }
    return launch_pdl(kern, dim3(grid), dim3(kThrThreads), 0, stream, p);
}

cudaError_t launch_topk_dense(const TopkParams& p, cudaStream_t stream)
{
    if (p.total_rows <= 0)
        return cudaSuccess;
    const int grid = p.row_fail != nullptr ? std::min(p.total_rows, 4 * sm_count()) : p.total_rows;
    return launch_pdl(topk_dense_kernel, dim3(grid), dim3(kSelThreads), 0, stream, p);
}

}  // namespace idx
