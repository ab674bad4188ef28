// Small kernels: block-mask expansion and the bounded-wait self-test.
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

}  // namespace

cudaError_t launch_expand_mask(const uint8_t* cand_mask, int64_t ld_mask, const int32_t* clen,
                               uint8_t* key_mask, int64_t ld, int block, int rows,
                               cudaStream_t st)
{
    if (rows <= 0)
        return cudaSuccess;
    const int64_t per_row = (ld + 255) / 256;
    dim3 grid((unsigned)std::min<int64_t>(per_row, 64), (unsigned)rows);
    expand_mask_kernel<<<grid, 256, 0, st>>>(cand_mask, ld_mask, clen, key_mask, ld, block, rows);
    return cudaGetLastError();
}

cudaError_t launch_selftest_timeout(uint32_t* status, long long cycles, cudaStream_t st)
{
    selftest_timeout_kernel<<<1, 32, 0, st>>>(status, cycles);
    return cudaGetLastError();
}

}  // namespace idx
