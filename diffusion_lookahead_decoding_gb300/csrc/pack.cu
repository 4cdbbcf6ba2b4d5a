// Weight repacking for the projection GEMMs.
//
// The GEMMs read a weight matrix [rows][K] (bf16, row-major) as tiles of tile_rows x 64
// elements.  Row-major, one tile touches tile_rows separate 128-byte pieces, each in a
// different DRAM page.  Packed tile-major, [rows/tile_rows][K/64][tile_rows][64], every
// tile is one contiguous 16 KB (or 32 KB) run.  The packing runs once, at context set-up;
// rows past the end of the matrix are zero-filled up to a whole tile.
#include "common.cuh"
#include "internal.h"

namespace lopa {

namespace {

// One CTA per (tile, k-block); 16-byte chunks, 8 per 64-element row.
__global__ void pack_tiles_kernel(const bf16* __restrict__ src, bf16* __restrict__ dst, int rows,
                                  int K, int tile_rows) {
  const int kb_total = K / 64;
  const int tile = blockIdx.x / kb_total, kb = blockIdx.x - tile * kb_total;
  bf16* out = dst + (size_t)blockIdx.x * tile_rows * 64;
  for (int c = threadIdx.x; c < tile_rows * 8; c += blockDim.x) {
    const int r = c >> 3, col = (c & 7) * 8;
    const int row = tile * tile_rows + r;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (row < rows) v = *reinterpret_cast<const uint4*>(src + (size_t)row * K + kb * 64 + col);
    *reinterpret_cast<uint4*>(out + r * 64 + col) = v;
  }
}

}  // namespace

size_t packed_elems(int rows, int K, int tile_rows) {
  return (size_t)((rows + tile_rows - 1) / tile_rows) * tile_rows * K;
}

cudaError_t launch_pack_tiles(const bf16* src, bf16* dst, int rows, int K, int tile_rows,
                              cudaStream_t s) {
  if (K % 64 || tile_rows % 8) return cudaErrorInvalidValue;
  const int tiles = (rows + tile_rows - 1) / tile_rows;
  pack_tiles_kernel<<<tiles * (K / 64), 256, 0, s>>>(src, dst, rows, K, tile_rows);
  return cudaGetLastError();
}

}  // namespace lopa
