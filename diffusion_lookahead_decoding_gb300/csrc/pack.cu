// Weight repacking for the projection GEMMs.
//
// The GEMMs read a weight matrix [rows][K] (bf16, row-major) as tiles of tile_rows x 64
// elements.  Row-major, one tile touches tile_rows separate 128-byte pieces, each in a
// different DRAM page.  Packed tile-major, [rows/tile_rows][K/64][tile_rows][64], every
// tile is one contiguous 16 KB (or 32 KB) run.  The packing runs once, at context set-up;
// it also stacks the matrices that one GEMM streams together (q, k and v; gate and up)
// into one packed matrix.  Rows past the end are zero-filled up to a whole tile.
//
// The E4M3 weight stream packs the same tiles as 8-bit codes (64 bytes per row per
// k-block) with one float32 scale per row: s = max|w| / 448, code = E4M3(w / s) rounded to
// nearest even with finite saturation, both quotients formed in float32 (an all-zero row
// gets s = 1).  448 is the largest finite E4M3 magnitude (1 sign, 4 exponent bits with
// bias 7, 3 fraction bits; S.1111.111 is NaN).
#include <cuda_fp8.h>

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

// Row r of the stacked sources (zero past the end).
__device__ __forceinline__ const bf16* stacked_row(const PackSources& src, int row, int K) {
  for (int i = 0; i < PackSources::kMax; ++i) {
    if (row < src.rows[i]) return src.ptr[i] + (size_t)row * K;
    row -= src.rows[i];
  }
  return nullptr;
}

// One warp per row: scale[row] = max|w| / 448 (1 for an all-zero row or a row past the end).
__global__ void row_scale_kernel(PackSources src, int K, float* __restrict__ scale, int rows_out) {
  const int row = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows_out) return;
  const bf16* p = stacked_row(src, row, K);
  float m = 0.f;
  if (p)
    for (int c = lane * 8; c < K; c += 256) {
      const uint4 v = *reinterpret_cast<const uint4*>(p + c);
      const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float2 f = __bfloat1622float2(h[j]);
        m = fmaxf(m, fmaxf(fabsf(f.x), fabsf(f.y)));
      }
    }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if (lane == 0) scale[row] = m > 0.f ? __fdiv_rn(m, 448.0f) : 1.0f;
}

// Codes of 16 consecutive elements of row `row`, columns [col, col + 16).
__device__ __forceinline__ uint4 e4m3_codes16(const bf16* p, int col, float s) {
  uint4 out = make_uint4(0, 0, 0, 0);
  if (!p) return out;
  const uint4 v0 = *reinterpret_cast<const uint4*>(p + col);
  const uint4 v1 = *reinterpret_cast<const uint4*>(p + col + 8);
  const __nv_bfloat162* h0 = reinterpret_cast<const __nv_bfloat162*>(&v0);
  const __nv_bfloat162* h1 = reinterpret_cast<const __nv_bfloat162*>(&v1);
  uint16_t c[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const float2 f = __bfloat1622float2(j < 4 ? h0[j] : h1[j - 4]);
    // x -> low byte, y -> high byte: element order is kept in memory.
    c[j] = __nv_cvt_float2_to_fp8x2(make_float2(__fdiv_rn(f.x, s), __fdiv_rn(f.y, s)),
                                    __NV_SATFINITE, __NV_E4M3);
  }
  out.x = (uint32_t)c[0] | ((uint32_t)c[1] << 16);
  out.y = (uint32_t)c[2] | ((uint32_t)c[3] << 16);
  out.z = (uint32_t)c[4] | ((uint32_t)c[5] << 16);
  out.w = (uint32_t)c[6] | ((uint32_t)c[7] << 16);
  return out;
}

// One CTA per (tile, k-block) as pack_tiles_kernel; 16 codes (16 bytes) per thread item.
// Tile-major: [tiles][K/64][tile_rows][64] bytes; row-major (row_major = 1, one "tile" per
// CTA row range): [rows][K] bytes.
__global__ void pack_e4m3_kernel(PackSources src, const float* __restrict__ scale,
                                 uint8_t* __restrict__ dst, int K, int tile_rows, int row_major,
                                 int rows_out) {
  const int kb_total = K / 64;
  const int tile = blockIdx.x / kb_total, kb = blockIdx.x - tile * kb_total;
  for (int c = threadIdx.x; c < tile_rows * 4; c += blockDim.x) {
    const int r = c >> 2, col = (c & 3) * 16;
    const int row = tile * tile_rows + r;
    if (row >= rows_out) continue;
    const uint4 v = e4m3_codes16(stacked_row(src, row, K), kb * 64 + col, scale[row]);
    uint8_t* o = row_major ? dst + (size_t)row * K + kb * 64 + col
                           : dst + ((size_t)blockIdx.x * tile_rows + r) * 64 + col;
    *reinterpret_cast<uint4*>(o) = v;
  }
}

}  // namespace

cudaError_t launch_row_scales(const PackSources& src, int K, float* scale, int rows_out,
                              cudaStream_t s) {
  if (K % 64 || rows_out <= 0) return cudaErrorInvalidValue;
  row_scale_kernel<<<(rows_out + 7) / 8, 256, 0, s>>>(src, K, scale, rows_out);
  return cudaGetLastError();
}

cudaError_t launch_pack_e4m3(const PackSources& src, const float* scale, uint8_t* dst, int K,
                             int tile_rows, bool row_major, int rows_out, cudaStream_t s) {
  if (K % 64 || tile_rows % 8 || rows_out <= 0) return cudaErrorInvalidValue;
  const int tiles = (rows_out + tile_rows - 1) / tile_rows;
  pack_e4m3_kernel<<<tiles * (K / 64), 256, 0, s>>>(src, scale, dst, K, tile_rows,
                                                    row_major ? 1 : 0, rows_out);
  return cudaGetLastError();
}

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
