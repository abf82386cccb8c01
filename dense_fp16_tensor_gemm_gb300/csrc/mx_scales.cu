// mx_scales.cu -- block scales from the plain layout (one E8M0 byte per row
// and per 32 consecutive K elements, rows of ceil(K/32) bytes) into the atom
// layout the block-scaled tcgen05 kernel copies to Tensor Memory: for every
// 128 rows and every 128 elements of K a 512-byte atom whose byte 16*r + 4*q
// + s holds the scale of row 32*q + r, K block s (atoms of one matrix stored
// row block-major, matrices of a batch one after another).  Rows and K blocks
// past the matrix get 127, a scale of one.
#include <algorithm>

#include "internal.h"

namespace gnt {

namespace {

__global__ void mx_pack_kernel(const uint8_t* __restrict__ plain, int64_t ld, int64_t stride,
                               uint8_t* __restrict__ packed, int64_t rows, int64_t kblocks, int64_t kgroups,
                               int64_t per_matrix, int64_t total)
{
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t b = i / per_matrix, rem = i - b * per_matrix;
        const int64_t atom = rem >> 9, within = rem & 511;
        const int64_t rb = atom / kgroups, kg = atom - rb * kgroups;
        const int64_t r = within >> 4, q = (within >> 2) & 3, s = within & 3;
        const int64_t row = rb * 128 + 32 * q + r, col = kg * 4 + s;
        packed[i] = (row < rows && col < kblocks) ? plain[b * stride + row * ld + col] : static_cast<uint8_t>(127);
    }
}

}  // namespace

cudaError_t mx_pack_launch(const uint8_t* plain, int64_t ld, int64_t stride, uint8_t* packed, int64_t rows,
                           int64_t K, int64_t batch, cudaStream_t stream)
{
    const int64_t kgroups = (K + 127) / 128, per_matrix = ((rows + 127) / 128) * kgroups * 512;
    const int64_t total = per_matrix * batch;
    const int64_t blocks = std::min<int64_t>((total + 255) / 256, 152 * 8);
    mx_pack_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(plain, ld, batch > 1 ? stride : 0, packed, rows,
                                                                      (K + 31) / 32, kgroups, per_matrix, total);
    return cudaGetLastError();
}

}  // namespace gnt
