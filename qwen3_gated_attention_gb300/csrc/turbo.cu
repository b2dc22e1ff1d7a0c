// turbo.cu -- the standalone Turbo4 quantizer (gattn_turbo4_quantize_device):
// one warp per row, the same device routine the q|k|v projection's epilogue
// runs on the step's new V rows.
#include "common.cuh"
#include "kernels.cuh"

namespace gattn {

__global__ void __launch_bounds__(256) turbo4_quantize_kernel(const uint16_t *v, long long rows,
                                                              int d, uint8_t *codes,
                                                              uint8_t *scales, const TurboTables t)
{
    const int lane = threadIdx.x & 31;
    const long long row = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
    if (row >= rows)
        return;                 // the whole warp leaves together
    const int per = d >> 5;
    float x[8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
        x[i] = i < per ? __uint_as_float((uint32_t)v[row * d + lane + 32 * i] << 16) : 0.f;
    turbo4_quantize_warp(x, per, lane, t, codes + row * (d / 2), scales + row * (d / 16));
}

cudaError_t launch_turbo4_quantize(const uint16_t *v, long long rows, int d, uint8_t *codes,
                                   uint8_t *scales, const TurboTables &t, cudaStream_t s)
{
    if (rows <= 0)
        return cudaSuccess;
    const unsigned grid = (unsigned)((rows + 7) / 8);
    return launch_plain(turbo4_quantize_kernel, dim3(grid), dim3(256), 0, s, v, rows, d, codes,
                        scales, t);
}

}  // namespace gattn
