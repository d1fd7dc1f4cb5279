// Create-time repack of canonical Q2_K / Q8_0 rows into the units that the decode GEMV and the
// prefill GEMM read (layout described in common.cuh). One thread writes one 32-bit word.
#include "common.cuh"

namespace ds4 {
namespace {

__device__ __forceinline__ uint32_t q2k_q(const uint8_t* blk, int k) {  // canonical 2-bit quant
  return (blk[16 + (k >> 2)] >> (2 * (k & 3))) & 3u;
}

__global__ void repack_q2k_kernel(const uint8_t* __restrict__ src, uint8_t* __restrict__ dst, int total_rows,
                                  int k) {
  const int n_kb = k / 256;
  const size_t row_bytes = (size_t)n_kb * 84;
  const size_t words_per_unit = kQ2kUnitBytes / 4;
  const size_t n_units = (size_t)(total_rows / 16) * n_kb;
  const size_t total = n_units * words_per_unit;
  for (size_t gid = blockIdx.x * (size_t)blockDim.x + threadIdx.x; gid < total; gid += (size_t)gridDim.x * blockDim.x) {
    const size_t u = gid / words_per_unit;
    const int w = (int)(gid % words_per_unit);
    const int rg = (int)(u / n_kb), kb = (int)(u % n_kb);
    const uint8_t* rowblk = src + (size_t)(rg * 16) * row_bytes + (size_t)kb * 84;  // row 0 of the group
    uint32_t word = 0;
    if (w < 256) {  // quants: region (g, t) at position lane_region(g, t), words (row half, k-pair half)
      const int c = w / 128, pos = (w % 128) / 4, r = w % 4;
      const int g = pos >> 2, t = (pos & 3) ^ ((g >> 1) & 3);
      const int row = g + 8 * (r >> 1);
      const int koff = 2 * t + 8 * (r & 1);
      const uint8_t* blk = rowblk + (size_t)row * row_bytes;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int kk = 16 * (8 * c + i) + koff;
        word |= q2k_q(blk, kk) << (2 * i);
        word |= q2k_q(blk, kk + 1) << (16 + 2 * i);
      }
    } else if (w < 320) {  // scale bytes
      const int c = (w - 256) / 32, lane = (w - 256) % 32;
      const int g = lane >> 2, t = lane & 3;
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const int row = g + 8 * (b >> 1);
        const int sub = 8 * c + 2 * t + (b & 1);
        word |= (uint32_t)rowblk[(size_t)row * row_bytes + sub] << (8 * b);
      }
    } else {  // d, dmin of row w - 320
      const uint8_t* blk = rowblk + (size_t)(w - 320) * row_bytes;
      word = (uint32_t)blk[80] | ((uint32_t)blk[81] << 8) | ((uint32_t)blk[82] << 16) | ((uint32_t)blk[83] << 24);
    }
    reinterpret_cast<uint32_t*>(dst + unit_offset(rg, kb, n_kb, kQ2kUnitBytes))[w] = word;
  }
}

__global__ void repack_q80_kernel(const uint8_t* __restrict__ src, uint8_t* __restrict__ dst, int total_rows,
                                  int k) {
  const int n_kb = k / 128;
  const size_t row_bytes = (size_t)(k / 32) * 34;
  const size_t words_per_unit = kQ80UnitBytes / 4;
  const size_t n_units = (size_t)(total_rows / 16) * n_kb;
  const size_t total = n_units * words_per_unit;
  for (size_t gid = blockIdx.x * (size_t)blockDim.x + threadIdx.x; gid < total; gid += (size_t)gridDim.x * blockDim.x) {
    const size_t u = gid / words_per_unit;
    const int w = (int)(gid % words_per_unit);
    const int rg = (int)(u / n_kb), kb = (int)(u % n_kb);
    const uint8_t* row0 = src + (size_t)(rg * 16) * row_bytes;
    uint32_t word = 0;
    if (w < 512) {  // region (g, t) at position lane_region(g, t): words (row half, sub-block)
      const int j = w / 128, pos = (w % 128) / 4, ww = w % 4;
      const int g = pos >> 2, t = (pos & 3) ^ ((g >> 1) & 3);
      const int row = g + 8 * (ww >> 1), i = 2 * j + (ww & 1);
#pragma unroll
      for (int e = 0; e < 4; ++e) {  // bytes: k = 2t, 2t + 1, 2t + 8, 2t + 9 of sub-block i
        const int kk = kb * 128 + 16 * i + 2 * t + 8 * (e >> 1) + (e & 1);
        const uint8_t qb = row0[(size_t)row * row_bytes + (size_t)(kk / 32) * 34 + 2 + (kk % 32)];
        word |= (uint32_t)(uint8_t)(qb ^ 0x80u) << (8 * e);  // u = q + 128
      }
    } else {
      const int lane = w - 512, g = lane >> 2, t = lane & 3;
      const int blk = kb * 4 + t;
      const uint8_t* a = row0 + (size_t)g * row_bytes + (size_t)blk * 34;
      const uint8_t* b = row0 + (size_t)(g + 8) * row_bytes + (size_t)blk * 34;
      word = (uint32_t)a[0] | ((uint32_t)a[1] << 8) | ((uint32_t)b[0] << 16) | ((uint32_t)b[1] << 24);
    }
    reinterpret_cast<uint32_t*>(dst + unit_offset(rg, kb, n_kb, kQ80UnitBytes))[w] = word;
  }
}

// Largest |d| of all super-blocks of a repacked Q2_K stack (as float bits, for atomicMax).
__global__ void q2k_dmax_kernel(const uint8_t* __restrict__ packed, size_t n_units, unsigned* __restrict__ out) {
  unsigned m = 0;
  for (size_t u = blockIdx.x * (size_t)blockDim.x + threadIdx.x; u < n_units * 16; u += (size_t)gridDim.x * blockDim.x) {
    const __half dh = *reinterpret_cast<const __half*>(packed + (u / 16) * kQ2kUnitBytes + kQ2kDdOff + 4 * (u % 16));
    m = max(m, __float_as_uint(fabsf(__half2float(dh))));
  }
  atomicMax(out, m);
}

}  // namespace

void launch_q2k_dmax(const uint8_t* packed, size_t bytes, unsigned* out, cudaStream_t s) {
  q2k_dmax_kernel<<<152 * 4, 256, 0, s>>>(packed, bytes / kQ2kUnitBytes, out);
}

void launch_repack(int fmt, const uint8_t* src, uint8_t* dst, int total_rows, int k, cudaStream_t s) {
  const int threads = 256, blocks = 152 * 8;
  if (fmt == FMT_Q2_K)
    repack_q2k_kernel<<<blocks, threads, 0, s>>>(src, dst, total_rows, k);
  else
    repack_q80_kernel<<<blocks, threads, 0, s>>>(src, dst, total_rows, k);
}

}  // namespace ds4
