// Inline-PTX helpers for sm_103a: mbarriers with bounded waits, TMA tile
// loads, tcgen05 (TMEM allocation, MMA, commit, loads) and the shared-memory
// matrix descriptors the MMA reads its operands through.
//
// Every wait here gives up after a cycle budget and reports failure, so a
// kernel that never receives an arrival ends with an error status instead
// of spinning forever.
#pragma once
#include <cstdint>
#include <cuda.h>

namespace idx {

__device__ __forceinline__ uint32_t smem_u32(const void* p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ------------------------------------------------------------- mbarriers

// Relaxed device-scope load of a value other CTAs update with atomics.
__device__ __forceinline__ uint32_t ld_relaxed_gpu(const uint32_t* p)
{
    uint32_t v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void fence_mbar_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// try_wait that lets the hardware suspend the thread until the phase completes
// or `hint_ns` nanoseconds pass, instead of returning at once (a waiting warp
// then takes no issue slots from the warps doing work).
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t* bar, uint32_t parity,
                                                    uint32_t hint_ns)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns)
        : "memory");
    return ok != 0;
}

// Wait until the phase with the given parity has completed.  Returns false
// when `budget` SM cycles pass first or when *abort becomes non-zero.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, long long budget,
                                          volatile int* abort)
{
    if (mbar_try_wait(bar, parity))
        return true;
    const long long t0 = clock64();
    while (true) {
        if (mbar_try_wait_sleep(bar, parity, 20000u))
            return true;
        if (*abort)
            return false;
        if (clock64() - t0 > budget)
            return false;
    }
}

// The same wait for roles that spend most of their time waiting: between polls the
// thread sleeps (32 ns, doubling up to max_ns), so waiting warps take almost no issue
// slots from the warps doing work.
__device__ __forceinline__ bool mbar_wait_backoff(uint64_t* bar, uint32_t parity,
                                                  long long budget, volatile int* abort,
                                                  uint32_t max_ns = 512u)
{
    if (mbar_try_wait(bar, parity))
        return true;
    const long long t0 = clock64();
    uint32_t ns = 32;
    while (true) {
        __nanosleep(ns);
        if (mbar_try_wait(bar, parity))
            return true;
        if (*abort)
            return false;
        if (clock64() - t0 > budget)
            return false;
        ns = ns < max_ns ? 2u * ns : max_ns;
    }
}

// ------------------------------------------------------------------ TMA

__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map)
{
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 2-D tiled load of a box into shared memory; completion is counted in bytes
// on `bar`.  x is the innermost coordinate (bytes for the 8-bit tensors used
// here, always 0, so it is 16-byte aligned), y the row.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int32_t x, int32_t y)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y)
        : "memory");
}

// Bulk copy of `bytes` (a multiple of 16; both addresses 16-byte aligned) from global
// to shared memory, counted in bytes on `bar`.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes,
                                          uint64_t* bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes),
        "r"(smem_u32(bar))
        : "memory");
}

// Named barrier `id` over `count` threads that also returns whether `v` holds in all
// of them.
__device__ __forceinline__ bool bar_all(bool v, int id, int count)
{
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.and.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(v ? 1u : 0u), "r"(id), "r"(count)
        : "memory");
    return r != 0;
}

// ---------------------------------------------------------------- tcgen05

// TMEM allocation: executed by one full warp; the allocated base address is
// written to shared memory.
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish()
{
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr),
                 "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before()
{
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after()
{
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, kind::f8f6f4 (8-bit or narrower operands,
// fp32 accumulate), one CTA.
__device__ __forceinline__ void mma_f8f6f4(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                           uint32_t idesc, uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Block-scaled variant, kind::mxf8f6f4: D (+)= (A x 2^sfa) * (B x 2^sfb)^T with one
// ue8m0 scale per row and 32-element K block for A (keys) and for B (query columns).
// The scales live in TMEM: sfa_tmem / sfb_tmem address 32-bit cells holding four scale
// bytes, the instruction descriptor's scale IDs select the byte of this K block.
__device__ __forceinline__ void mma_mxf8f6f4(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                             uint32_t idesc, uint32_t sfa_tmem,
                                             uint32_t sfb_tmem, uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, "
        "[%4], [%5], p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
        : "memory");
}

// Block-scaled fp4 x fp4, kind::mxf4: both operands packed e2m1 (two codes a byte,
// K = 64 per MMA), one ue8m0 scale per row and 32-element K block, two blocks per MMA
// (scale_vec::2X): the scale IDs select bytes {0,1} or {2,3} of each 32-bit cell.
__device__ __forceinline__ void mma_mxf4(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                         uint32_t idesc, uint32_t sfa_tmem, uint32_t sfb_tmem,
                                         uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf4.block_scale.scale_vec::2X [%0], %1, %2, %3, "
        "[%4], [%5], p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
        : "memory");
}

// Copy 128 rows x 128 bits from shared memory (no-swizzle canonical layout, row r at
// byte 16 r) into TMEM: row r lands in lane r, four 32-bit columns.  Asynchronous,
// ordered with the tcgen05.mma this thread issues after it.
__device__ __forceinline__ void tmem_cp_128x128b(uint32_t taddr, uint64_t sdesc)
{
    asm volatile("tcgen05.cp.cta_group::1.128x128b [%0], %1;" ::"r"(taddr), "l"(sdesc)
                 : "memory");
}

// 32 lanes x 8 columns of 32-bit from registers into TMEM (the warp's lane quadrant),
// the same value in every cell.
__device__ __forceinline__ void tmem_st_32x32b_x8_fill(uint32_t taddr, uint32_t v)
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %1, %1, %1, %1, %1, %1, %1};" ::"r"(
            taddr),
        "r"(v)
        : "memory");
}

__device__ __forceinline__ void tmem_wait_st()
{
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Make this thread's shared-memory writes visible to the async proxy (tcgen05.cp, TMA).
__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Arrive once on `bar` when every tcgen05 operation this thread issued so
// far has completed.
__device__ __forceinline__ void mma_commit(uint64_t* bar)
{
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void tmem_wait_ld()
{
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// 16 lanes x 256 bits, repeated 4 times along the columns (32 columns): thread
// t = 4g + q gets, for repetition k, columns 8k + 2q and 8k + 2q + 1 of lane g
// (v[4k], v[4k+1]) and of lane g + 8 (v[4k+2], v[4k+3]), lanes counted from
// the address's lane field.
__device__ __forceinline__ void tmem_ld_16x256b_x4(uint32_t taddr, float (&v)[16])
{
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.16x256b.x4.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
#pragma unroll
    for (int i = 0; i < 16; ++i)
        v[i] = __uint_as_float(r[i]);
}

// Shared-memory matrix descriptor for a K-major operand tile stored in the
// canonical swizzled layout that a TMA load with the matching swizzle mode
// writes: rows of `row_bytes` (32, 64 or 128 = the swizzle width), groups
// of 8 rows `8*row_bytes` apart.  Fields: start address >> 4 (bits 0-13),
// leading byte offset >> 4 (16-29, unused for this layout), stride byte
// offset >> 4 (32-45), the fixed descriptor version 1 (46-47), base offset 0
// (49-51, tiles are aligned to the swizzle repeat), layout (61-63).
__device__ __forceinline__ uint64_t smem_desc_kmajor(uint32_t saddr, int row_bytes)
{
    const uint64_t layout = row_bytes == 128 ? 2ull : (row_bytes == 64 ? 4ull : 6ull);
    const uint64_t sbo = static_cast<uint64_t>(8 * row_bytes) >> 4;
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
    d |= 1ull << 16;
    d |= sbo << 32;
    d |= 1ull << 46;
    d |= layout << 61;
    return d;
}

// Instruction descriptor, kind::f8f6f4, fp32 accumulator, both operands
// K-major, no negation/sparsity.  a_fmt/b_fmt: 0 = e4m3, 5 = e2m1.
// Fields: D format (bits 4-5, 1 = f32), A format (7-9), B format (10-12),
// N >> 3 (17-22), M >> 4 (24-28).
__host__ __device__ constexpr uint32_t idesc_f8f6f4(int M, int N, int a_fmt, int b_fmt)
{
    return (1u << 4) | (static_cast<uint32_t>(a_fmt) << 7) |
           (static_cast<uint32_t>(b_fmt) << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
           (static_cast<uint32_t>(M >> 4) << 24);
}


// Shared-memory descriptor of a no-swizzle K-major matrix of 16-byte rows whose 8-row
// core matrices are `sbo` bytes apart (the layout tcgen05.cp 128x128b reads).
__device__ __forceinline__ uint64_t smem_desc_noswizzle(uint32_t saddr, uint32_t sbo)
{
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
    d |= 1ull << 16;
    d |= static_cast<uint64_t>(sbo >> 4) << 32;
    d |= 1ull << 46;
    return d;
}

// Instruction descriptor, kind::mxf8f6f4 with ue8m0 scales (fp32 accumulator, both
// operands K-major): B scale byte ID (bits 4-5), A format (7-9), B format (10-12),
// N >> 3 (17-22), scale type ue8m0 (bit 23), M >> 4 (24-28), A scale byte ID (29-30).
// Formats: 0 = e4m3, 5 = e2m1.
__host__ __device__ constexpr uint32_t idesc_mxf8f6f4(int M, int N, int a_fmt, int b_fmt,
                                                      int a_sf_id, int b_sf_id)
{
    return (static_cast<uint32_t>(b_sf_id & 3) << 4) | (static_cast<uint32_t>(a_fmt) << 7) |
           (static_cast<uint32_t>(b_fmt) << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
           (1u << 23) | (static_cast<uint32_t>(M >> 4) << 24) |
           (static_cast<uint32_t>(a_sf_id & 3) << 29);
}

// Instruction descriptor, kind::mxf4 with ue8m0 scales: the same fields, e2m1 coded 1
// for both operands (the only format of this kind), dense K = 64 (bit 31 clear).  The
// scale IDs of scale_vec::2X are 0 or 2.
__host__ __device__ constexpr uint32_t idesc_mxf4(int M, int N, int a_sf_id, int b_sf_id)
{
    return idesc_mxf8f6f4(M, N, 1, 1, a_sf_id, b_sf_id);
}

// ReLU on the FMA pipe, scaled by 2^-64: sat(x * 2^-64) clamps to [0, 1], which equals
// max(x, 0) * 2^-64 exactly whenever 2^-62 <= |x| < 2^64 (scaling by a power of two is
// exact there; below, the scaled value is subnormal and keeps an absolute error under
// 2^-150).  e4m3 x e4m3 scores lie in [2^-18, D * 448^2] when not zero; block-scaled e2m1
// scores carry their block scales and can be far larger, hence the wide margin.  FMNMX
// runs on the ALU pipe at half the FMA rate, so the epilogue spreads its ReLUs over both.
__device__ __forceinline__ float relu_scaled(float x)
{
    float r;
    asm("mul.rn.sat.f32 %0, %1, %2;" : "=f"(r) : "f"(x), "f"(5.42101086242752217e-20f));
    return r;
}

// Order-preserving map of an fp32 value to uint32 (larger float -> larger key).
__device__ __forceinline__ uint32_t f2ord(float f)
{
    uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float ord2f(uint32_t u)
{
    return __uint_as_float((u & 0x80000000u) ? (u & 0x7FFFFFFFu) : ~u);
}

// ord(-inf): anything at or below it is "not eligible" for selection.
constexpr uint32_t kOrdNegInf = 0x007FFFFFu;

// Programmatic dependent launch.  Every kernel of the library is launched so that it
// may start while the previous kernel of its stream is still running: it first waits
// for that kernel to complete (its writes visible), then lets the next kernel's blocks
// be placed as resources free up (they in turn wait before touching anything).  Both
// are no-ops for a kernel launched the ordinary way.
__device__ __forceinline__ void pdl_wait_then_release()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

}  // namespace idx
