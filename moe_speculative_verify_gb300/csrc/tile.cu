// tile.cu -- row-major e4m3 weight matrices into the tiled layout: every
// 128x128 block (the unit of the per-block weight scales) stored as 16 KB of
// its own, blocks in row-block-major order, so that the expert GEMMs, which
// stream the blocks of a row-block along K, read their weights sequentially.
#include "common.cuh"
#include "kernels.h"

namespace moe {

constexpr int kTileThreads = 256;

// One 16 KB block per loop trip: 1024 16-byte words, four per thread; the
// reads take eight words (one 128-byte row segment) per eight threads, the
// writes are contiguous.
__global__ void __launch_bounds__(kTileThreads) tile_weights_kernel(const uint4* __restrict__ src,
                                                                   uint4* __restrict__ dst,
                                                                   int64_t n_blocks, int kb_per_row,
                                                                   int64_t row_words) {
    for (int64_t t = blockIdx.x; t < n_blocks; t += gridDim.x) {
        const int64_t rb = t / kb_per_row;   // row-block over all matrices
        const int kb = static_cast<int>(t - rb * kb_per_row);
        const uint4* s = src + rb * 128 * row_words + kb * 8;
        uint4* d = dst + t * 1024;
#pragma unroll
        for (int i = 0; i < 1024 / kTileThreads; ++i) {
            const int q = threadIdx.x + i * kTileThreads;
            d[q] = __ldg(s + (q >> 3) * row_words + (q & 7));
        }
    }
}

cudaError_t launch_tile_weights(const uint8_t* src, uint8_t* dst, int64_t n, int rows, int cols,
                                cudaStream_t stream) {
    const int64_t n_blocks = n * (rows / 128) * (cols / 128);
    if (n_blocks == 0) return cudaSuccess;
    const int grid = static_cast<int>(n_blocks < 8192 ? n_blocks : 8192);
    tile_weights_kernel<<<grid, kTileThreads, 0, stream>>>(
        reinterpret_cast<const uint4*>(src), reinterpret_cast<uint4*>(dst), n_blocks, cols / 128,
        cols / 16);
    return cudaGetLastError();
}

}  // namespace moe
