// Exact per-row top-k selection kernels.
//
// Selection rule: among the eligible entries of a row (finite score, inside
// the row's causal length), keep the k with the largest score; on equal
// scores the lower key index wins.  Used three ways:
//   * per key split: the top-k of one block of keys ("chunked-prefill-
//     memory.md" section 2.3: score against key blocks, keep the per-block
//     top-k values and indices);
//   * merge: the top-k of the union of the per-block candidates, which is
//     exactly the top-k of the whole row (same section: "topk(union) ==
//     topk(union of per-block topk) holds exactly");
//   * candidate blocks: the same, over the maximum score of each 8-key block
//     (same section: block pooling over 8-key blocks, top-2048 blocks).
//
// Algorithm: radix select on the order-preserving 32-bit image of the fp32
// score, 8 bits per pass from the top, stopping as soon as the boundary bin
// is taken whole; exact ties at the k-th score are resolved by position
// (= key order) in a final ordered pass.  The output lists the kept entries
// in ascending key order, so results are bitwise reproducible.
#include "internal.h"
#include "ptx.cuh"

namespace idx {
namespace {

constexpr int kSelThreads = 512;
constexpr int kSelWarps = kSelThreads / 32;

struct SelShared {
    uint32_t hist[256];
    uint32_t warp_a[kSelWarps];
    uint32_t warp_b[kSelWarps];
    uint32_t bcast[4];
};

// Warp-aggregated histogram increment: lanes with the same digit add once.
__device__ __forceinline__ void hist_add(uint32_t* hist, uint32_t digit, bool active)
{
    const uint32_t d = active ? digit : 256u;
    const uint32_t peers = __match_any_sync(0xffffffffu, d);
    const int leader = __ffs(peers) - 1;
    if (active && (threadIdx.x & 31) == leader)
        atomicAdd(&hist[d], static_cast<uint32_t>(__popc(peers)));
}

// Block-wide exclusive scan of two counters (one entry per thread).
__device__ __forceinline__ void block_scan2(SelShared& sh, uint32_t a, uint32_t b, uint32_t& pa,
                                            uint32_t& pb, uint32_t& ta, uint32_t& tb)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint32_t ia = a, ib = b;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t xa = __shfl_up_sync(0xffffffffu, ia, o);
        const uint32_t xb = __shfl_up_sync(0xffffffffu, ib, o);
        if (lane >= o) {
            ia += xa;
            ib += xb;
        }
    }
    if (lane == 31) {
        sh.warp_a[warp] = ia;
        sh.warp_b[warp] = ib;
    }
    __syncthreads();
    uint32_t wa = 0, wb = 0;
    ta = 0;
    tb = 0;
    for (int w = 0; w < kSelWarps; ++w) {
        const uint32_t x = sh.warp_a[w], y = sh.warp_b[w];
        if (w < warp) {
            wa += x;
            wb += y;
        }
        ta += x;
        tb += y;
    }
    pa = wa + ia - a;
    pb = wb + ib - b;
    __syncthreads();
}

// Top-k of entries 0..n-1 of one row.  load(e) -> fp32 score (-inf = not
// eligible).  emit(pos, e, v) writes output slot pos (0 <= pos < k) in
// ascending e.  Returns the number of entries emitted (<= k).
template <class Load, class Emit>
__device__ int block_topk(SelShared& sh, int n, int k, const Load& load, const Emit& emit)
{
    const int tid = threadIdx.x;
    uint32_t prefix = 0, pmask = 0;
    uint32_t remaining = static_cast<uint32_t>(k);
    bool take_all = false;     // every eligible entry is kept
    bool resolved = false;     // boundary bin taken whole: keep (ord & pmask) >= prefix
    uint32_t tie_quota = 0;    // after 32 bits: how many entries equal to prefix to keep

    for (int pass = 0; pass < 4; ++pass) {
        const int shift = 24 - 8 * pass;
        for (int i = tid; i < 256; i += kSelThreads)
            sh.hist[i] = 0;
        __syncthreads();
        for (int base = 0; base < n; base += kSelThreads) {
            const int e = base + tid;
            bool act = false;
            uint32_t dig = 0;
            if (e < n) {
                const uint32_t o = f2ord(load(e));
                act = o > kOrdNegInf && (o & pmask) == prefix;
                dig = (o >> shift) & 255u;
            }
            hist_add(sh.hist, dig, act);
        }
        __syncthreads();
        if (tid == 0) {
            uint32_t total = 0;
            for (int b = 0; b < 256; ++b)
                total += sh.hist[b];
            uint32_t flag = 0, bin = 0, above = 0;
            if (pass == 0 && total <= remaining) {
                flag = 1;  // fewer eligible entries than k
            } else {
                uint32_t cum = 0;
                for (int b = 255; b >= 0; --b) {
                    const uint32_t c = sh.hist[b];
                    if (cum + c >= remaining) {
                        bin = static_cast<uint32_t>(b);
                        above = cum;
                        flag = (cum + c == remaining) ? 2 : 0;
                        break;
                    }
                    cum += c;
                }
            }
            sh.bcast[0] = flag;
            sh.bcast[1] = bin;
            sh.bcast[2] = above;
        }
        __syncthreads();
        const uint32_t flag = sh.bcast[0];
        if (flag == 1) {
            take_all = true;
            break;
        }
        prefix |= sh.bcast[1] << shift;
        pmask |= 255u << shift;
        remaining -= sh.bcast[2];
        __syncthreads();
        if (flag == 2) {
            resolved = true;
            break;
        }
    }
    if (!take_all && !resolved)
        tie_quota = remaining;   // keep > prefix, plus the first tie_quota entries == prefix

    // ordered output pass
    uint32_t sel_before = 0, ties_before = 0;
    for (int base = 0; base < n; base += kSelThreads) {
        const int e = base + tid;
        uint32_t sel = 0, tie = 0;
        float v = -INFINITY;
        if (e < n) {
            v = load(e);
            const uint32_t o = f2ord(v);
            if (o > kOrdNegInf) {
                if (take_all)
                    sel = 1;
                else if (resolved)
                    sel = (o & pmask) >= prefix ? 1u : 0u;
                else if (o > prefix)
                    sel = 1;
                else if (o == prefix)
                    tie = 1;
            }
        }
        uint32_t ps, pt, ts, tt;
        block_scan2(sh, sel, tie, ps, pt, ts, tt);
        if (tie && ties_before + pt < tie_quota)
            sel = 1;
        // positions: entries are emitted in ascending e, so count kept entries before e
        const uint32_t kept_tie_before =
            min(tie_quota, ties_before + pt) - min(tie_quota, ties_before);
        const uint32_t pos = sel_before + ps + kept_tie_before;
        if (sel && pos < static_cast<uint32_t>(k))
            emit(static_cast<int>(pos), e, v);
        const uint32_t kept_ties_chunk = min(tie_quota, ties_before + tt) - min(tie_quota, ties_before);
        sel_before += ts + kept_ties_chunk;
        ties_before += tt;
    }
    return static_cast<int>(min(sel_before, static_cast<uint32_t>(k)));
}

// ------------------------------------------------------------ per-split

__global__ void __launch_bounds__(kSelThreads) select_dense_kernel(const __grid_constant__ SelParams p)
{
    __shared__ SelShared sh;
    const int cta = blockIdx.x;
    int s = 0;
    while (s + 1 < p.num_segments && p.seg[s + 1].row_block <= cta)
        ++s;
    const SelSegment& sg = p.seg[s];
    const int tr = cta - sg.row_block;       // row within the segment
    const int t = sg.row_begin + tr;
    const int clen = min(p.compress_len[t], sg.key_count);
    const float* src = p.src + sg.src_offset + (int64_t)tr * sg.src_ld;
    const int64_t out_base = sg.cand_offset + ((int64_t)tr * sg.n_slots + sg.cand_slot) * p.k;
    float* cv = p.cand_val + out_base;
    int32_t* ci = p.cand_idx + out_base;
    int count;
    if (p.pool == 0) {
        const int n = max(0, min(clen - sg.j_begin, sg.n_entries));
        auto load = [&](int e) { return src[e]; };
        auto emit = [&](int pos, int e, float v) {
            cv[pos] = v;
            ci[pos] = sg.j_begin + e;
        };
        count = block_topk(sh, n, p.k, load, emit);
    } else {
        const int pool = p.pool;
        const int nkeys = max(0, min(clen - sg.j_begin * pool, sg.n_entries * pool));
        const int n = (nkeys + pool - 1) / pool;
        auto load = [&](int e) {
            float m = -INFINITY;
            const int k0 = e * pool;
            const int k1 = min(k0 + pool, nkeys);
            for (int kk = k0; kk < k1; ++kk)
                m = fmaxf(m, src[kk]);
            return m;
        };
        auto emit = [&](int pos, int e, float v) {
            cv[pos] = v;
            ci[pos] = sg.j_begin + e;
        };
        count = block_topk(sh, n, p.k, load, emit);
    }
    for (int i = count + threadIdx.x; i < p.k; i += kSelThreads) {
        cv[i] = -INFINITY;
        ci[i] = -1;
    }
}

// ---------------------------------------------------------------- merge

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

__global__ void __launch_bounds__(kSelThreads) merge_kernel(const __grid_constant__ MergeParams p)
{
    __shared__ SelShared sh;
    const int t = blockIdx.x;
    const int r = find_request(p.req_row_begin, p.num_requests, t);
    const int tr = t - p.req_row_begin[r];
    const int nslots = p.req_slots[r];
    const int64_t base = p.req_cand_offset[r] + (int64_t)tr * nslots * p.k;
    const float* cv = p.cand_val + base;
    const int32_t* ci = p.cand_idx + base;
    const int n = nslots * p.k;
    auto load = [&](int e) { return cv[e]; };
    if (p.mask) {
        uint8_t* m = p.mask + (int64_t)t * p.ld_mask;
        for (int64_t b = threadIdx.x; b < p.ld_mask; b += kSelThreads)
            m[b] = 0;
        __syncthreads();
        auto emit = [&](int pos, int e, float v) {
            (void)pos;
            (void)v;
            const int b = ci[e];
            if (b >= 0 && b < p.ld_mask)
                m[b] = 1;
        };
        block_topk(sh, n, p.k, load, emit);
    } else {
        int32_t* oi = p.out_idx + (int64_t)t * p.k;
        float* ov = p.out_val ? p.out_val + (int64_t)t * p.k : nullptr;
        auto emit = [&](int pos, int e, float v) {
            oi[pos] = ci[e];
            if (ov)
                ov[pos] = v;
        };
        const int count = block_topk(sh, n, p.k, load, emit);
        for (int i = count + threadIdx.x; i < p.k; i += kSelThreads) {
            oi[i] = -1;
            if (ov)
                ov[i] = -INFINITY;
        }
    }
}

// ------------------------------------------------------- standalone top-k

__global__ void __launch_bounds__(kSelThreads) topk_dense_kernel(const __grid_constant__ TopkParams p)
{
    __shared__ SelShared sh;
    const int t = blockIdx.x;
    const int r = find_request(p.req_row_begin, p.num_requests, t);
    const int n = max(0, min(p.compress_len[t], p.req_key_count[r]));
    const float* row = p.logits + (int64_t)t * p.ld;
    int32_t* oi = p.out_idx + (int64_t)t * p.k;
    float* ov = p.out_val ? p.out_val + (int64_t)t * p.k : nullptr;
    auto load = [&](int e) { return row[e]; };
    auto emit = [&](int pos, int e, float v) {
        oi[pos] = e;
        if (ov)
            ov[pos] = v;
    };
    const int count = block_topk(sh, n, p.k, load, emit);
    for (int i = count + threadIdx.x; i < p.k; i += kSelThreads) {
        oi[i] = -1;
        if (ov)
            ov[i] = -INFINITY;
    }
}

}  // namespace

cudaError_t launch_select_dense(const SelParams& p, cudaStream_t stream)
{
    if (p.total_rows_launch <= 0)
        return cudaSuccess;
    select_dense_kernel<<<p.total_rows_launch, kSelThreads, 0, stream>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_merge(const MergeParams& p, cudaStream_t stream)
{
    if (p.total_rows <= 0)
        return cudaSuccess;
    merge_kernel<<<p.total_rows, kSelThreads, 0, stream>>>(p);
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
