// Weight repacking for the projection GEMMs.
//
// The GEMMs read a weight matrix [rows][K] (bf16, row-major) as tiles of tile_rows x 64
// elements.  Row-major, one tile touches tile_rows separate 128-byte pieces, each in a
// different DRAM page.  Packed tile-major, [rows/tile_rows][K/64][tile_rows][64], every
// tile is one contiguous 16 KB (or 32 KB) run.  The packing runs once, at context set-up;
// it also stacks the matrices that one GEMM streams together (q, k and v; gate and up)
// into one packed matrix.  Rows past the end are zero-filled up to a whole tile.
#include "common.cuh"
#include "internal.h"

namespace lopa {

namespace {

// One CTA per (tile, k-block); 16-byte chunks, 8 per 64-element row.  Row r of the stacked
// matrix is row r of src[0], then of src[1], then of src[2].
__global__ void pack_tiles_kernel(PackSources src, bf16* __restrict__ dst, int K, int tile_rows) {
  const int kb_total = K / 64;
  const int tile = blockIdx.x / kb_total, kb = blockIdx.x - tile * kb_total;
  bf16* out = dst + (size_t)blockIdx.x * tile_rows * 64;
  for (int c = threadIdx.x; c < tile_rows * 8; c += blockDim.x) {
    const int r = c >> 3, col = (c & 7) * 8;
    int row = tile * tile_rows + r;
    uint4 v = make_uint4(0, 0, 0, 0);
    for (int i = 0; i < PackSources::kMax; ++i) {
      if (row < src.rows[i]) {
        v = *reinterpret_cast<const uint4*>(src.ptr[i] + (size_t)row * K + kb * 64 + col);
        break;
      }
      row -= src.rows[i];
    }
    *reinterpret_cast<uint4*>(out + r * 64 + col) = v;
  }
}

}  // namespace

size_t packed_elems(int rows, int K, int tile_rows) {
  return (size_t)((rows + tile_rows - 1) / tile_rows) * tile_rows * K;
}

cudaError_t launch_pack_tiles(const PackSources& src, bf16* dst, int K, int tile_rows,
                              cudaStream_t s) {
  if (K % 64 || tile_rows % 8) return cudaErrorInvalidValue;
  int rows = 0;
  for (int i = 0; i < PackSources::kMax; ++i) rows += src.rows[i];
  const int tiles = (rows + tile_rows - 1) / tile_rows;
  pack_tiles_kernel<<<tiles * (K / 64), 256, 0, s>>>(src, dst, K, tile_rows);
  return cudaGetLastError();
}

}  // namespace lopa
