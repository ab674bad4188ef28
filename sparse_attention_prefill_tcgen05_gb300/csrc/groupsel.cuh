// Exact top-k selection by a group of threads (a whole CTA or one named-
// barrier group), shared by the selection kernels and the in-kernel list
// compaction of the streaming top-k.
//
// Entries are ranked by the composite 64-bit key (ord(score), ~index): a
// larger score first, then the lower key index ("ties to the lower index").
// Keys are unique, so the k-th largest key splits the entries into exactly
// min(k, eligible) kept entries.  The threshold is found by radix select,
// 8 bits per pass from the top, stopping as soon as the boundary bin is
// taken whole; entries with a score of -inf are never eligible.
#pragma once
#include "ptx.cuh"

namespace idx {

struct CtaSync {
    __device__ __forceinline__ void operator()() const { __syncthreads(); }
};

// Named barrier over `count` threads (whole warps).
struct NamedSync {
    int id;
    int count;
    __device__ __forceinline__ void operator()() const
    {
        asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
    }
};

template <int NT>
struct SelScratch {
    alignas(16) uint32_t hist[2][256];   // alternate passes: one is counted, the other zeroed
    uint32_t warp_sum[NT / 32];
    uint32_t bcast[4];
};

// A threshold on the composite key: entry kept iff kept(hi, lo).
struct CompositeThr {
    uint32_t phi, plo, mhi, mlo;  // prefix and mask of the resolved bits
    __device__ __forceinline__ bool kept(uint32_t hi, uint32_t lo) const
    {
        if ((hi & mhi) != phi)
            return (hi & mhi) > phi;
        return (lo & mlo) >= plo;
    }
};

__device__ __forceinline__ void hist_add_aggregated(uint32_t* hist, uint32_t digit, bool active)
{
    const uint32_t d = active ? digit : 256u;
    const uint32_t peers = __match_any_sync(0xffffffffu, d);
    const int leader = __ffs(peers) - 1;
    if (active && (threadIdx.x & 31) == leader)
        atomicAdd(&hist[d], static_cast<uint32_t>(__popc(peers)));
}

// Find the threshold keeping the k largest composite keys among entries
// [0, n).  load(e, hi, lo) must set hi = ord(score) and lo = ~index; entries
// with hi <= ord(-inf) are not eligible.  All NT threads of the group call
// this (tid in [0, NT)).
template <int NT, class Sync, class Load>
__device__ CompositeThr group_threshold(SelScratch<NT>& sh, int tid, int n, uint32_t k,
                                        const Load& load, const Sync& sync, int max_passes = 8,
                                        uint32_t* eligible = nullptr)
{
    CompositeThr thr{0u, 0u, 0u, 0u};
    uint32_t remaining = k;
    for (int i = tid; i < 256; i += NT)
        sh.hist[0][i] = 0;
    sync();
    // two barriers per pass: after counting (this pass's histogram complete, the
    // other one zeroed for the next pass) and after the boundary search
    for (int pass = 0; pass < max_passes; ++pass) {
        const bool in_hi = pass < 4;
        const int shift = 24 - 8 * (pass & 3);
        uint32_t* hist = sh.hist[pass & 1];
        for (int i = tid; i < 256; i += NT)
            sh.hist[(pass + 1) & 1][i] = 0;
        for (int base = 0; base < n; base += NT) {
            const int e = base + tid;
            bool act = false;
            uint32_t dig = 0;
            if (e < n) {
                uint32_t hi, lo;
                load(e, hi, lo);
                act = hi > kOrdNegInf && (hi & thr.mhi) == thr.phi && (lo & thr.mlo) == thr.plo;
                dig = ((in_hi ? hi : lo) >> shift) & 255u;
            }
            hist_add_aggregated(hist, dig, act);
        }
        sync();
        if (tid < 32) {
            // boundary bin by one warp: 8 bins per lane, suffix sums across lanes
            const int lane = tid;
            const uint4 a = reinterpret_cast<const uint4*>(hist)[lane * 2];
            const uint4 b = reinterpret_cast<const uint4*>(hist)[lane * 2 + 1];
            const uint32_t c[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
            const uint32_t lsum = c[0] + c[1] + c[2] + c[3] + c[4] + c[5] + c[6] + c[7];
            uint32_t suf = lsum;  // sum over lanes >= this one
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const uint32_t y = __shfl_down_sync(0xffffffffu, suf, o);
                if (lane + o < 32)
                    suf += y;
            }
            const uint32_t total = __shfl_sync(0xffffffffu, suf, 0);
            if (pass == 0 && lane == 0)
                sh.bcast[3] = total;
            const uint32_t holders = __ballot_sync(0xffffffffu, suf >= remaining);
            if (total <= remaining) {
                if (lane == 0) {
                    sh.bcast[0] = 1;  // everything still undecided is kept
                    sh.bcast[1] = 0;
                    sh.bcast[2] = 0;
                }
            } else if (lane == 31 - __clz(holders)) {
                uint32_t cum = suf - lsum;
                uint32_t bin = 0, above = 0, flag = 0;
#pragma unroll
                for (int i = 7; i >= 0; --i) {
                    if (cum + c[i] >= remaining) {
                        bin = static_cast<uint32_t>(lane * 8 + i);
                        above = cum;
                        flag = (cum + c[i] == remaining) ? 2u : 0u;
                        break;
                    }
                    cum += c[i];
                }
                sh.bcast[0] = flag;
                sh.bcast[1] = bin;
                sh.bcast[2] = above;
            }
        }
        sync();
        // (bcast is rewritten only after the next pass's counting barrier)
        const uint32_t flag = sh.bcast[0];
        const uint32_t bin = sh.bcast[1];
        const uint32_t above = sh.bcast[2];
        if (pass == 0 && eligible)
            *eligible = sh.bcast[3];
        if (flag == 1)
            break;  // the current prefix already keeps exactly what must be kept
        if (in_hi) {
            thr.phi |= bin << shift;
            thr.mhi |= 255u << shift;
        } else {
            thr.plo |= bin << shift;
            thr.mlo |= 255u << shift;
        }
        remaining -= above;
        if (flag == 2)
            break;
    }
    return thr;
}

// Ordered emission: calls emit(pos, e, hi, lo) for every kept entry, pos
// counting kept entries in ascending e, (hi, lo) the entry's composite key as
// loaded.  Loads happen before the group barrier inside the scan and emits
// after it, so emit may overwrite entries at positions <= e (in-place
// compaction) as long as it uses the (hi, lo) it is given.  Returns the
// number of kept entries.
template <int NT, class Sync, class Load, class Emit>
__device__ int group_emit(SelScratch<NT>& sh, int tid, int n, const CompositeThr& thr,
                          const Load& load, const Emit& emit, const Sync& sync)
{
    const int lane = tid & 31, warp = tid >> 5;
    uint32_t before = 0;
    for (int base = 0; base < n; base += NT) {
        const int e = base + tid;
        bool sel = false;
        uint32_t hi = 0, lo = 0;
        if (e < n) {
            load(e, hi, lo);
            sel = hi > kOrdNegInf && thr.kept(hi, lo);
        }
        const uint32_t m = __ballot_sync(0xffffffffu, sel);
        if (lane == 0)
            sh.warp_sum[warp] = __popc(m);
        sync();
        uint32_t wbefore = 0, total = 0;
#pragma unroll
        for (int w = 0; w < NT / 32; ++w) {
            const uint32_t x = sh.warp_sum[w];
            wbefore += w < warp ? x : 0u;
            total += x;
        }
        sync();
        if (sel)
            emit(static_cast<int>(before + wbefore + __popc(m & ((1u << lane) - 1u))), e, hi, lo);
        before += total;
    }
    return static_cast<int>(before);
}

}  // namespace idx
