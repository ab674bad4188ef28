// Indexer logits on the 5th-generation tensor cores (sm_103a).
//
//   logit[t, j] = s_k[j] * sum_h c[t,h] * max(S[t,h,j], 0),   c = w * s_q,
//   S[t,h,j]    = <q[t,h,:], k[j,:]>  (fp8 e4m3 x fp8 e4m3, fp32 accumulate)
//
// which equals sum_h w * ReLU(s_q * s_k * S) because the scales are
// positive ("[DeepSeek-V4.1] Bound the dense prefill indexer transient",
// Motivation: the DeepGEMM fp8 MQA logits the indexer scores with;
// "chunked-prefill-memory.md" section 1: T query rows against the whole
// compressed prefix, [T, max_seqlen_k] fp32 output, -inf past the row's
// causal length).
//
// Mapping.  One MMA tile is M = 128 keys (TMEM lanes) x N = 256 (row, head)
// columns (256/H query rows x H heads) x K = D.  With keys on the lanes, the
// head reduction of one (row, key) is a run of H consecutive accumulator
// columns held by ONE thread: no shuffles, no shared-memory reduction.
//
// Roles (384 threads, one CTA per SM, persistent over work units):
//   warp 0      TMA producer: the unit's Q tile (double-buffered) and a ring
//               of K tiles, 128-byte-swizzled for the MMA.
//   warp 1      allocates 512 TMEM columns (two 256-column accumulators),
//               issues tcgen05.mma (D/32 per tile) and tcgen05.commit.
//   warps 4-11  epilogue: tcgen05.ld 32x32b, ReLU, head-weighted sum, key
//               scale, causal mask (and candidate mask), coalesced store.
// The accumulator is double-buffered so the epilogue of tile i overlaps the
// MMAs of tile i+1.
#include "internal.h"
#include "ptx.cuh"

namespace idx {
namespace {

template <int H, int D, int KFMT>
struct Cfg {
    // fp4 keys need TMEM columns for the block scales, so their tiles are
    // 192 columns wide (two accumulators of 192 + scale columns <= 512).
    static constexpr int NMAX = KFMT == kKeyFp8 ? kTileN : 192;
    static constexpr int G = NMAX / H;                 // query rows per tile
    static constexpr int N = G * H;                    // MMA N
    static constexpr int QBYTES = N * D;               // Q tile: N rows of D bytes
    static constexpr int KBYTES = kTileKeys * D;       // K tile in smem (fp4 unpacked to bytes)
    static constexpr int STAGES = (D >= 128) ? 6 : 8;
    static constexpr int KSTEPS = D / 32;              // MMA K = 32 elements
    static constexpr int ROWS_PER_HALF = G / 2;        // rows one epilogue thread reduces
    static constexpr int HALF_COLS = N / 2;
    static constexpr int ACC_COLS = N;                 // TMEM columns per accumulator
    static constexpr int SF_BYTES = KFMT == kKeyFp4 ? kTileKeys * 16 : 0;  // per stage
    static constexpr int TMEM_SFA = 2 * ACC_COLS;      // 4 columns per stage
    static constexpr int TMEM_SFB = TMEM_SFA + 4 * STAGES;
    static_assert(D == 32 || D == 64 || D == 128, "D must be 32, 64 or 128");
    static_assert(G >= 2 && G % 2 == 0 && N % 16 == 0, "H must leave an even row count");
    static_assert(HALF_COLS % 32 == 0, "half tile must be whole 32-column loads");
    static_assert(KFMT == kKeyFp8 || (D == 128 && TMEM_SFB + 4 <= 512), "fp4 needs D=128");
    // shared memory carve-up (offsets from a 1024-byte aligned base)
    static constexpr int OFF_Q = 0;
    static constexpr int OFF_K = OFF_Q + ((2 * QBYTES + 1023) / 1024) * 1024;
    static constexpr int OFF_SF = OFF_K + STAGES * KBYTES;
    static constexpr int OFF_C = OFF_SF + STAGES * SF_BYTES;        // float c[2][N]
    static constexpr int OFF_BAR = OFF_C + 2 * kTileN * 4;
    static constexpr int NBARS = 2 + 2 + 2 * STAGES + 2 + 2 + 1;
    static constexpr int OFF_MISC = OFF_BAR + NBARS * 8;
    static constexpr int SMEM = OFF_MISC + 16 + 1024;              // + alignment slack
};

struct UnitInfo {
    int seg;
    int t0;        // first global row of the row group
    int nr;        // valid rows in the group
    int j0;        // request-local first key of the unit
    int jend;      // request-local end of keys written by the unit
    int ntiles;    // tiles covering [j0, jend)
    int ntiles_mma;
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
    ui.seg = s;
    ui.t0 = sg.row_begin + g * G;
    ui.nr = min(G, sg.row_begin + sg.nrows - ui.t0);
    ui.j0 = sg.j_begin + chunk * p.chunk_tiles * kTileKeys;
    ui.jend = min(sg.j_end, ui.j0 + p.chunk_tiles * kTileKeys);
    ui.ntiles = (ui.jend - ui.j0 + kTileKeys - 1) / kTileKeys;
    // longest causal length in the group (warp-cooperative), clamped to the request
    int m = 0;
    for (int r = lane; r < ui.nr; r += 32)
        m = max(m, min(p.compress_len[ui.t0 + r], sg.key_count));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
    const int mma_end = min(ui.jend, m);
    ui.ntiles_mma = mma_end > ui.j0 ? (mma_end - ui.j0 + kTileKeys - 1) / kTileKeys : 0;
    return ui;
}

__device__ __forceinline__ void report(const LogitsParams& p, volatile int* abort_flag,
                                       uint32_t bits)
{
    *abort_flag = 1;
    atomicOr(p.status, bits);
}

template <int H, int D, int KFMT>
__global__ void __launch_bounds__(kThreads, 1)
    logits_tc_kernel(const __grid_constant__ LogitsParams p)
{
    using C = Cfg<H, D, KFMT>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* q_s = smem + C::OFF_Q;
    uint8_t* k_s = smem + C::OFF_K;
    uint8_t* sf_s = smem + C::OFF_SF;
    float* c_s = reinterpret_cast<float*>(smem + C::OFF_C);
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

    if (threadIdx.x == 0) {
        for (int i = 0; i < 2; ++i) {
            mbar_init(&q_full[i], 1);
            mbar_init(&q_empty[i], 1);
            mbar_init(&a_full[i], 1);
            mbar_init(&a_empty[i], kEpiWarps);
        }
        for (int i = 0; i < C::STAGES; ++i) {
            // fp4: one arrival with the TMA bytes plus one after the scales are staged
            mbar_init(&k_full[i], KFMT == kKeyFp4 ? 2 : 1);
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
        tmem_alloc(tmem_slot, 2 * C::ACC_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const long long budget = p.timeout_cycles;
    if (KFMT == kKeyFp4) {
        // q carries no block scale: every B scale is 2^0 (ue8m0 127) in all bytes
        if (warp >= 4 && warp < 8) {
            const uint32_t one = 0x7F7F7F7Fu;
            tmem_st_32x32b_x4(tmem_base + (static_cast<uint32_t>((warp & 3) * 32) << 16) +
                                  C::TMEM_SFB,
                              one, one, one, one);
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
            const Segment& sg = p.seg[ui.seg];
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
            for (int i = 0; i < ui.ntiles_mma && ok; ++i) {
                const int key0 = sg.key_base + ui.j0 + i * kTileKeys;
                if (lane == 0) {
                    if (!mbar_wait(&k_empty[ks], kph ^ 1, budget, abort_flag)) {
                        report(p, abort_flag, kStatusTimeout);
                        ok = false;
                    } else {
                        mbar_arrive_expect_tx(&k_full[ks], C::KBYTES);
                        tma_load_2d(k_s + ks * C::KBYTES, &p.tmap_k, &k_full[ks], 0, key0);
                        ++issued[ks];
                    }
                }
                ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
                if (!ok)
                    break;
                if (KFMT == kKeyFp4) {
                    // stage the tile's ue8m0 scales, one 32-bit word (4 blocks of 32
                    // elements) per key, at a 16-byte row pitch for tcgen05.cp
                    uint8_t* sf = sf_s + ks * C::SF_BYTES;
                    const uint32_t* src = reinterpret_cast<const uint32_t*>(p.k_sf);
#pragma unroll
                    for (int r = 0; r < kTileKeys / 32; ++r) {
                        const int m = r * 32 + lane;
                        const int key = key0 + m;
                        const int local = ui.j0 + i * kTileKeys + m;
                        const uint32_t word = local < sg.key_count ? __ldg(src + key) : 0x7F7F7F7Fu;
                        *reinterpret_cast<uint32_t*>(sf + m * 16) = word;
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
                    if (KFMT == kKeyFp8) {
#pragma unroll
                        for (int kk = 0; kk < C::KSTEPS; ++kk) {
                            const uint64_t adesc = smem_desc_kmajor(k_addr + kk * 32, D);
                            const uint64_t bdesc = smem_desc_kmajor(q_addr + kk * 32, D);
                            mma_f8f6f4(d_tmem, adesc, bdesc, idesc, kk > 0 ? 1u : 0u);
                        }
                    } else {
                        // key scales of this stage into TMEM, then one block-scaled MMA per
                        // 32-element block (A = e2m1 keys, B = e4m3 queries)
                        const uint32_t sfa = tmem_base + C::TMEM_SFA + 4 * ks;
                        tmem_cp_128x128b(sfa, smem_desc_noswizzle(smem_u32(sf_s + ks * C::SF_BYTES), 128));
#pragma unroll
                        for (int kk = 0; kk < C::KSTEPS; ++kk) {
                            const uint64_t adesc = smem_desc_kmajor(k_addr + kk * 32, D);
                            const uint64_t bdesc = smem_desc_kmajor(q_addr + kk * 32, D);
                            mma_mxf8f6f4(d_tmem, adesc, bdesc,
                                         idesc_mxf8f6f4(kTileKeys, C::N, 5, 0, kk, kk), sfa,
                                         tmem_base + C::TMEM_SFB, kk > 0 ? 1u : 0u);
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
        const int ew = warp - 4;                 // 0..7
        const int quad = warp & 3;               // TMEM lane quadrant of this warp
        const int half = ew >> 2;                // column half: rows [half*G/2, +G/2)
        const int kq = quad * 32 + lane;         // key within the tile
        const int etid = ew * 32 + lane;         // 0..255
        int ab = 0, aph = 0, it = 0;
        bool ok = true;
        // Every epilogue warp walks every unit (also after an abort) so that the
        // named barrier below always sees all 256 threads.
        for (int u = blockIdx.x; u < p.total_units; u += gridDim.x, ++it) {
            const UnitInfo ui = decode_unit<C::G>(p, u, lane);
            const Segment& sg = p.seg[ui.seg];
            float* cbuf = c_s + (it & 1) * kTileN;
            if (etid < C::N) {   // c[n] = w * s_q for column n = row * H + head
                const int rl = etid / H;
                const int t = ui.t0 + rl;
                cbuf[etid] = rl < ui.nr ? p.w[(size_t)t * H + (etid % H)] *
                                              p.s_q[(size_t)t * H + (etid % H)]
                                        : 0.0f;
            }
            asm volatile("bar.sync 1, 256;" ::: "memory");
            if (!ok)
                continue;
            int clen[C::ROWS_PER_HALF];
#pragma unroll
            for (int r = 0; r < C::ROWS_PER_HALF; ++r) {
                const int rl = half * C::ROWS_PER_HALF + r;
                clen[r] = rl < ui.nr ? min(p.compress_len[ui.t0 + rl], sg.key_count) : 0;
            }
            float* out_base = p.out + sg.out_offset - sg.j_begin;
            for (int i = 0; i < ui.ntiles; ++i) {
                const int j = ui.j0 + i * kTileKeys + kq;
                float acc[C::ROWS_PER_HALF];
                bool have = false;
                if (i < ui.ntiles_mma) {
                    float sk = 1.0f;
                    if (KFMT == kKeyFp8)
                        sk = j < sg.key_count ? __ldg(p.s_k + sg.key_base + j) : 0.0f;
                    const bool got = mbar_wait(&a_full[ab], aph, budget, abort_flag);
                    if (!__all_sync(0xffffffffu, got)) {
                        if (lane == 0)
                            report(p, abort_flag, kStatusTimeout);
                        ok = false;
                        break;
                    }
                    tc_fence_after();
#pragma unroll
                    for (int r = 0; r < C::ROWS_PER_HALF; ++r)
                        acc[r] = 0.0f;
                    const uint32_t tbase = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) +
                                           ab * C::ACC_COLS + half * C::HALF_COLS;
                    const float4* cc4 =
                        reinterpret_cast<const float4*>(cbuf + half * C::HALF_COLS);
#pragma unroll
                    for (int ch = 0; ch < C::HALF_COLS / 32; ++ch) {
                        float v[32];
                        tmem_ld_32x32b_x32(tbase + ch * 32, v);
                        tmem_wait_ld();
#pragma unroll
                        for (int e4 = 0; e4 < 8; ++e4) {
                            const float4 c4 = cc4[ch * 8 + e4];
                            const float cv[4] = {c4.x, c4.y, c4.z, c4.w};
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const int col = ch * 32 + e4 * 4 + e;
                                acc[col / H] = fmaf(cv[e], fmaxf(v[e4 * 4 + e], 0.0f), acc[col / H]);
                            }
                        }
                    }
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0)
                        mbar_arrive(&a_empty[ab]);
                    if (++ab == 2) {
                        ab = 0;
                        aph ^= 1;
                    }
#pragma unroll
                    for (int r = 0; r < C::ROWS_PER_HALF; ++r)
                        acc[r] *= sk;
                    have = true;
                }
                if (j < ui.jend) {
#pragma unroll
                    for (int r = 0; r < C::ROWS_PER_HALF; ++r) {
                        const int rl = half * C::ROWS_PER_HALF + r;
                        if (rl < ui.nr) {
                            const int t = ui.t0 + rl;
                            bool valid = have && j < clen[r];
                            if (valid && p.cand_mask)
                                valid = p.cand_mask[(size_t)t * p.ld_mask + j / p.mask_block] != 0;
                            out_base[(size_t)(t - sg.row_begin) * sg.out_ld + j] =
                                valid ? acc[r] : -INFINITY;
                        }
                    }
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1)
        tmem_dealloc(tmem_base, 2 * C::ACC_COLS);
}

template <int H, int D, int KFMT>
cudaError_t launch_one(const LogitsParams& p, int grid, cudaStream_t stream)
{
    using C = Cfg<H, D, KFMT>;
    auto kern = logits_tc_kernel<H, D, KFMT>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::SMEM);
    if (e != cudaSuccess)
        return e;
    kern<<<grid, kThreads, C::SMEM, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace

size_t logits_smem_bytes(int H, int D, int kfmt)
{
    if (kfmt == kKeyFp4)
        return (H == 32 && D == 128) ? Cfg<32, 128, kKeyFp4>::SMEM : 0;
    if (H == 32 && D == 128)
        return Cfg<32, 128, kKeyFp8>::SMEM;
    if (H == 4 && D == 64)
        return Cfg<4, 64, kKeyFp8>::SMEM;
    if (H == 64 && D == 128)
        return Cfg<64, 128, kKeyFp8>::SMEM;
    if (H == 16 && D == 128)
        return Cfg<16, 128, kKeyFp8>::SMEM;
    return 0;
}

int logits_rows_per_group(int H, int kfmt) { return (kfmt == kKeyFp4 ? 192 : kTileN) / H; }

cudaError_t launch_logits(const LogitsParams& p, int H, int D, int kfmt, int grid,
                          cudaStream_t stream)
{
    if (kfmt == kKeyFp8) {
        if (H == 32 && D == 128)
            return launch_one<32, 128, kKeyFp8>(p, grid, stream);
        if (H == 4 && D == 64)
            return launch_one<4, 64, kKeyFp8>(p, grid, stream);
        if (H == 64 && D == 128)
            return launch_one<64, 128, kKeyFp8>(p, grid, stream);
        if (H == 16 && D == 128)
            return launch_one<16, 128, kKeyFp8>(p, grid, stream);
    } else if (kfmt == kKeyFp4) {
        if (H == 32 && D == 128)
            return launch_one<32, 128, kKeyFp4>(p, grid, stream);
    }
    return cudaErrorInvalidValue;
}

}  // namespace idx
