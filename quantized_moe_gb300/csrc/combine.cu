// Deterministic combine: out[t] = sum over the token's routed slots, in ascending expert id,
// of w_j * Y[position of slot j], then + the shared expert's row, all fp32, no atomics. Slots
// without a bucketed position (experts the handle does not hold) contribute nothing.
#include <algorithm>

#include "common.cuh"

namespace ds4 {
namespace {

constexpr int kMaxK = 16;

__global__ void __launch_bounds__(256) combine_kernel(const int* __restrict__ idx, const float* __restrict__ wts,
                                                      const int* __restrict__ rowof, const float* __restrict__ y,
                                                      const float* __restrict__ ys, int top_k, int d,
                                                      float* __restrict__ out) {
  __shared__ int s_pos[kMaxK];
  __shared__ float s_w[kMaxK];
  __shared__ int s_n;
  const int t = blockIdx.y;
  if (threadIdx.x == 0) {
    int e[kMaxK], p[kMaxK];
    float w[kMaxK];
    for (int j = 0; j < top_k; ++j) {  // insertion sort by expert id (ids are distinct)
      const int ej = idx[t * top_k + j];
      const float wj = wts[t * top_k + j];
      const int pj = rowof[t * top_k + j];
      int i = j;
      while (i > 0 && e[i - 1] > ej) { e[i] = e[i - 1]; w[i] = w[i - 1]; p[i] = p[i - 1]; --i; }
      e[i] = ej; w[i] = wj; p[i] = pj;
    }
    int n = 0;
    for (int j = 0; j < top_k; ++j)
      if (p[j] >= 0) {
        s_pos[n] = p[j];
        s_w[n++] = w[j];
      }
    s_n = n;
  }
  __syncthreads();
  // the slot loop is unrolled with predicated loads so that all of a column's loads are in flight
  // together (the fixed order of the sum is kept); small batches spread a row over several CTAs
  const int n = s_n;
  for (int i4 = (blockIdx.x * blockDim.x + threadIdx.x) * 4; i4 < d; i4 += gridDim.x * blockDim.x * 4) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int j = 0; j < kMaxK; ++j) {
      if (j < n) {
        const float4 v = __ldcs(reinterpret_cast<const float4*>(y + (size_t)s_pos[j] * d + i4));  // read once
        const float w = s_w[j];
        acc.x = fmaf(w, v.x, acc.x);
        acc.y = fmaf(w, v.y, acc.y);
        acc.z = fmaf(w, v.z, acc.z);
        acc.w = fmaf(w, v.w, acc.w);
      }
    }
    if (ys) {
      const float4 v = __ldcs(reinterpret_cast<const float4*>(ys + (size_t)t * d + i4));
      acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
    }
    __stcs(reinterpret_cast<float4*>(out + (size_t)t * d + i4), acc);
  }
}

// dst[i] = src[i] for `bytes` bytes (16-byte aligned), with 16-byte loads and stores: a copy run by
// the SMs, for buffers in page-locked host memory that kernels address directly.
__global__ void __launch_bounds__(256) copy16_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst,
                                                     size_t n16) {
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n16; i += (size_t)gridDim.x * blockDim.x)
    dst[i] = __ldcs(src + i);
}

}  // namespace

void launch_copy16(const void* src, void* dst, size_t bytes, cudaStream_t s) {
  const size_t n16 = bytes / 16;
  const int blocks = (int)std::min<size_t>((n16 + 255) / 256, 152 * 8);
  copy16_kernel<<<std::max(blocks, 1), 256, 0, s>>>(static_cast<const uint4*>(src), static_cast<uint4*>(dst), n16);
}

void launch_combine(const int* idx, const float* wts, const int* rowof, const float* y, const float* ys, int n_tok,
                    int top_k, int d, float* out, cudaStream_t s) {
  // up to 256 tokens a row is split over CTAs of 1024 columns (more CTAs than tokens); beyond, one CTA
  // per token row (measured at 4096 tokens: 123 us vs 128 us with the split)
  const int split = n_tok <= 256 ? (d + 1023) / 1024 : 1;
  combine_kernel<<<dim3(split, n_tok), 256, 0, s>>>(idx, wts, rowof, y, ys, top_k, d, out);
}

}  // namespace ds4
