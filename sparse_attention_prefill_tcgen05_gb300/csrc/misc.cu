// Small kernels: block-mask expansion, the page-index transform and the bounded-wait self-test.
#include "internal.h"
#include "ptx.cuh"
#include <algorithm>

namespace idx {
namespace {

// key_mask[t, j] = (j < compress_len[t]) && cand_mask[t, j / block]
__global__ void expand_mask_kernel(const uint8_t* __restrict__ cand_mask, int64_t ld_mask,
                                   const int32_t* __restrict__ clen, uint8_t* __restrict__ key_mask,
                                   int64_t ld, int block, int rows)
{
    pdl_wait_then_release();
    const int t = blockIdx.y;
    if (t >= rows)
        return;
    const int c = clen[t];
    for (int64_t j = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; j < ld;
         j += (int64_t)gridDim.x * blockDim.x) {
        uint8_t v = 0;
        if (j < c)
            v = cand_mask[(int64_t)t * ld_mask + j / block] ? 1 : 0;
        key_mask[(int64_t)t * ld + j] = v;
    }
}

// Head padding: q [rows, h_in, D] bytes -> q_out [rows, h_out, D] with zero
// heads past h_in, and s_q / w [rows, h_in] -> [rows, h_out] with zeros.  A
// zero head contributes exactly 0 to every logit (its weight is 0 and its
// dot product is 0), so the padded problem scores every key identically.
__global__ void pad_heads_kernel(const uint4* __restrict__ q, const float* __restrict__ s_q,
                                 const float* __restrict__ w, uint4* __restrict__ q_out,
                                 float* __restrict__ s_q_out, float* __restrict__ w_out, int rows,
                                 int h_in, int h_out, int d16)
{
    pdl_wait_then_release();
    const int64_t nq = (int64_t)rows * h_out * d16;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < nq;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t row_head = i / d16;
        const int h = static_cast<int>(row_head % h_out);
        const int64_t t = row_head / h_out;
        q_out[i] = h < h_in ? q[(t * h_in + h) * d16 + i % d16] : make_uint4(0u, 0u, 0u, 0u);
    }
    const int64_t ns = (int64_t)rows * h_out;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < ns;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int h = static_cast<int>(i % h_out);
        const int64_t t = i / h_out;
        s_q_out[i] = h < h_in ? s_q[t * h_in + h] : 0.0f;
        w_out[i] = h < h_in ? w[t * h_in + h] : 0.0f;
    }
}

// e2m1 (OCP MX): sign, 2 exponent bits (bias 1), 1 mantissa bit; codes 0..7 are
// 0, 0.5, 1, 1.5, 2, 3, 4, 6.  A nonzero magnitude is m * 2^E with m in {1, 1.5}.
// Scaled by 2^-n (n >= 0: its block exponent below the key's largest) it is an
// e4m3 value iff E - n >= -6 (normal: exponent field E - n + 7, mantissa 0 or
// 0b100) or it is a subnormal multiple of 2^-9 (m = 1: E - n >= -9; m = 1.5:
// E - n >= -8).  One thread per (key, 8 elements).
__global__ void fp4_to_fp8_kernel(const uint8_t* __restrict__ k4, const uint8_t* __restrict__ sf,
                                  int keys, int D, uint8_t* __restrict__ k8,
                                  float* __restrict__ s_k, uint32_t* status)
{
    pdl_wait_then_release();
    const int per_key = D / 8;
    const int64_t n = (int64_t)keys * per_key;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t j = i / per_key;
        const int part = static_cast<int>(i % per_key);      // elements 8*part .. 8*part+7
        const uint8_t* sfj = sf + j * (D / 32);
        int emax = 0;
        for (int b = 0; b < D / 32; ++b)
            emax = max(emax, static_cast<int>(sfj[b]));
        if (part == 0)
            s_k[j] = ldexpf(1.0f, emax - 127);
        const int shift = emax - static_cast<int>(sfj[(part * 8) / 32]);   // n
        const uint32_t packed = *reinterpret_cast<const uint32_t*>(k4 + j * (D / 2) + part * 4);
        uint32_t lo = 0, hi = 0;
        bool ok = true;
        for (int e = 0; e < 8; ++e) {
            const uint32_t code = (packed >> (4 * e)) & 15u;
            const uint32_t sign = code >> 3, mag = code & 7u;
            uint32_t out = sign << 7;
            if (mag != 0) {
                // mag 1: 0.5 = 1*2^-1; 2: 1; 3: 1.5; 4: 2; 5: 3 = 1.5*2; 6: 4; 7: 6 = 1.5*4
                const int E = mag == 1 ? -1 : static_cast<int>((mag - 2) >> 1);
                const bool half = mag >= 2 && (mag & 1u);    // m = 1.5
                const int Es = E - shift;
                if (Es >= -6) {
                    out |= static_cast<uint32_t>(Es + 7) << 3 | (half ? 4u : 0u);
                } else if (!half && Es >= -9) {
                    out |= 1u << (Es + 9);
                } else if (half && Es >= -8) {
                    out |= 3u << (Es + 8);
                } else {
                    ok = false;
                }
            }
            if (e < 4)
                lo |= out << (8 * e);
            else
                hi |= out << (8 * (e - 4));
        }
        *reinterpret_cast<uint2*>(k8 + j * D + part * 8) = make_uint2(lo, hi);
        if (!ok)
            atomicOr(status, kStatusFp4Range);
    }
}

// Waits on a barrier that nothing arrives on; must give up after `cycles`.
__global__ void selftest_timeout_kernel(uint32_t* status, long long cycles)
{
    __shared__ uint64_t bar;
    __shared__ int no_abort;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        no_abort = 0;
        fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        if (!mbar_wait(&bar, 0, cycles, &no_abort))
            atomicOr(status, kStatusTimeout);
    }
}

// Candidate mask rows of rows with at most cand_topk blocks (every one of their valid
// blocks is a candidate, whatever the logits): row t of rows [row0, row0 + rows) writes
// mask row t + delta, 1 for the blocks below ceil(min(clen[t], keys) / block), 0 for the
// rest of its ld bytes.  One CTA per row; 16-byte stores between the row's unaligned head
// and tail.
__global__ void fill_mask_rows_kernel(uint8_t* __restrict__ mask, int64_t ld,
                                      const int32_t* __restrict__ clen, int row0, int keys,
                                      int block, int64_t delta)
{
    pdl_wait_then_release();
    const int t = row0 + static_cast<int>(blockIdx.x);
    const int n = max(0, min(clen[t], keys));
    const int64_t nb = (n + block - 1) / block;   // candidate blocks of the row
    uint8_t* m = mask + (t + delta) * ld;
    const int64_t head = min(ld, static_cast<int64_t>((16 - (reinterpret_cast<uintptr_t>(m) & 15)) & 15));
    for (int64_t b = threadIdx.x; b < head; b += blockDim.x)
        m[b] = b < nb ? 1 : 0;
    const int64_t nvec = (ld - head) / 16;
    uint4* mv = reinterpret_cast<uint4*>(m + head);
    for (int64_t v = threadIdx.x; v < nvec; v += blockDim.x) {
        const int64_t b0 = head + 16 * v;
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            uint32_t x = 0;
#pragma unroll
            for (int j = 0; j < 4; ++j)
                x |= (b0 + 4 * i + j < nb ? 1u : 0u) << (8 * j);
            w[i] = x;
        }
        mv[v] = make_uint4(w[0], w[1], w[2], w[3]);
    }
    for (int64_t b = head + 16 * nvec + threadIdx.x; b < ld; b += blockDim.x)
        m[b] = b < nb ? 1 : 0;
}

}  // namespace

// Page-index transform: one thread per four consecutive entries of a row (k a
// multiple of 4) or per entry; the request of a row by binary search over the
// batch's row offsets; a power-of-two page divides by shifts.
__device__ __forceinline__ int32_t page_slot(const PageIndexParams& p, int r, int32_t j,
                                             int shift)
{
    if (j < 0 || j >= p.req_key_count[r])
        return -1;
    const int32_t pi = shift >= 0 ? (j >> shift) : j / p.page;
    const int32_t off = shift >= 0 ? (j & (p.page - 1)) : j - pi * p.page;
    const int64_t pg = p.table[(int64_t)r * p.ld_table + pi];
    if (pg < 0)
        return -1;
    const int64_t slot = pg * p.page + off;
    return slot <= 0x7FFFFFFF ? static_cast<int32_t>(slot) : -1;
}

__device__ __forceinline__ int row_request(const PageIndexParams& p, int t)
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

__global__ void page_indices_kernel(const __grid_constant__ PageIndexParams p, int shift, int vec)
{
    pdl_wait_then_release();
    const int64_t total = (int64_t)p.rows * p.k;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    if (vec) {
        for (int64_t v = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; v < total / 4;
             v += stride) {
            const int t = static_cast<int>((v * 4) / p.k);
            const int r = row_request(p, t);
            const int4 j = reinterpret_cast<const int4*>(p.raw)[v];
            reinterpret_cast<int4*>(p.out)[v] =
                make_int4(page_slot(p, r, j.x, shift), page_slot(p, r, j.y, shift),
                          page_slot(p, r, j.z, shift), page_slot(p, r, j.w, shift));
        }
    } else {
        for (int64_t e = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; e < total; e += stride) {
            const int t = static_cast<int>(e / p.k);
            p.out[e] = page_slot(p, row_request(p, t), p.raw[e], shift);
        }
    }
}

cudaError_t launch_page_indices(const PageIndexParams& p, cudaStream_t st)
{
    const int64_t total = (int64_t)p.rows * p.k;
    if (total <= 0)
        return cudaSuccess;
    int shift = -1;
    if ((p.page & (p.page - 1)) == 0)
        for (shift = 0; (1 << shift) < p.page; ++shift) {
        }
    const int vec = (p.k % 4 == 0 && (reinterpret_cast<uintptr_t>(p.raw) & 15) == 0 &&
                     (reinterpret_cast<uintptr_t>(p.out) & 15) == 0)
                        ? 1
                        : 0;
    const int64_t items = vec ? total / 4 : total;
    // a grid of whole waves: 152 SMs x 8 blocks of 256 threads at most
    const int blocks = static_cast<int>(std::min<int64_t>((items + 255) / 256, 152 * 8));
    return launch_pdl(page_indices_kernel, dim3(blocks), dim3(256), 0, st, p, shift, vec);
}

cudaError_t launch_fill_mask_rows(uint8_t* mask, int64_t ld, const int32_t* clen, int row0,
                                  int rows, int keys, int block, int64_t delta, cudaStream_t st)
{
    if (rows <= 0)
        return cudaSuccess;
    return launch_pdl(fill_mask_rows_kernel, dim3(rows), dim3(256), 0, st, mask, ld, clen, row0,
                      keys, block, delta);
}

cudaError_t launch_expand_mask(const uint8_t* cand_mask, int64_t ld_mask, const int32_t* clen,
                               uint8_t* key_mask, int64_t ld, int block, int rows,
                               cudaStream_t st)
{
    if (rows <= 0)
        return cudaSuccess;
    const int64_t per_row = (ld + 255) / 256;
    dim3 grid((unsigned)std::min<int64_t>(per_row, 64), (unsigned)rows);
    return launch_pdl(expand_mask_kernel, grid, dim3(256), 0, st, cand_mask, ld_mask, clen,
                      key_mask, ld, block, rows);
}

cudaError_t launch_fp4_to_fp8(const uint8_t* k4, const uint8_t* sf, int keys, int D, uint8_t* k8,
                              float* s_k, uint32_t* status, cudaStream_t st)
{
    if (keys <= 0)
        return cudaSuccess;
    const int64_t n = (int64_t)keys * (D / 8);
    const int blocks = (int)std::min<int64_t>((n + 255) / 256, 8192);
    return launch_pdl(fp4_to_fp8_kernel, dim3(blocks), dim3(256), 0, st, k4, sf, keys, D, k8, s_k,
                      status);
}

cudaError_t launch_pad_heads(const void* q, const float* s_q, const float* w, void* q_out,
                             float* s_q_out, float* w_out, int rows, int h_in, int h_out, int D,
                             cudaStream_t st)
{
    if (rows <= 0)
        return cudaSuccess;
    const int64_t nq = (int64_t)rows * h_out * (D / 16);
    const int blocks = (int)std::min<int64_t>((nq + 255) / 256, 4096);
    return launch_pdl(pad_heads_kernel, dim3(blocks), dim3(256), 0, st,
                      static_cast<const uint4*>(q), s_q, w, static_cast<uint4*>(q_out), s_q_out,
                      w_out, rows, h_in, h_out, D / 16);
}

cudaError_t launch_selftest_timeout(uint32_t* status, long long cycles, cudaStream_t st)
{
    selftest_timeout_kernel<<<1, 32, 0, st>>>(status, cycles);
    return cudaGetLastError();
}

}  // namespace idx
