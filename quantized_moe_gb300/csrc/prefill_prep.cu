// Prefill preparation: activations to scaled fp16 (token order and bucketed order) and the
// list of (expert, first position, rows) GEMM tiles.
#include "common.cuh"

namespace ds4 {
namespace {

// One CTA per token: s = power-of-two scale from max|x|, xs16 = fp16(x * s), inv_s = 1 / s.
__global__ void __launch_bounds__(256) xprep_kernel(const __nv_bfloat16* __restrict__ x, int d, __half* __restrict__ xs16,
                                                    float* __restrict__ inv_s) {
  __shared__ float part[8];
  const int t = blockIdx.x;
  const __nv_bfloat16* xr = x + (size_t)t * d;
  float m = 0.f;
  for (int i = threadIdx.x * 8; i < d; i += 256 * 8) {
    const uint4 v = *reinterpret_cast<const uint4*>(xr + i);
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 f = __bfloat1622float2(h[e]);
      m = fmaxf(m, fmaxf(fabsf(f.x), fabsf(f.y)));
    }
  }
  m = warp_max(m);
  if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = m;
  __syncthreads();
  float mx = 0.f;
#pragma unroll
  for (int w = 0; w < 8; ++w) mx = fmaxf(mx, part[w]);
  const float sc = fp16_row_scale(mx);
  for (int i = threadIdx.x * 8; i < d; i += 256 * 8) {
    const uint4 v = *reinterpret_cast<const uint4*>(xr + i);
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
    uint4 o;
    uint32_t* ov = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 f = __bfloat1622float2(h[e]);
      const __half2 r = __floats2half2_rn(f.x * sc, f.y * sc);
      ov[e] = *reinterpret_cast<const uint32_t*>(&r);
    }
    *reinterpret_cast<uint4*>(xs16 + (size_t)t * d + i) = o;
  }
  if (threadIdx.x == 0) inv_s[t] = 1.f / sc;
}

// One warp per bucketed position: copy the token's fp16 row; each lane issues eight 16-byte loads
// before its stores, so a warp keeps 4 KB in flight. The bucketed positions end at *n_pos (every
// slot, or the slots of the experts the handle holds).
__global__ void __launch_bounds__(256) gather_kernel(const __half* __restrict__ xs16, const float* __restrict__ inv_s,
                                                     const int* __restrict__ perm, const int* __restrict__ n_pos,
                                                     int n_slots, int top_k, int d, __half* __restrict__ xp16,
                                                     float* __restrict__ inv_p) {
  const int pos = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (pos >= n_slots || pos >= *n_pos) return;
  const int tok = perm[pos] / top_k;
  const uint4* src = reinterpret_cast<const uint4*>(xs16 + (size_t)tok * d);
  uint4* dst = reinterpret_cast<uint4*>(xp16 + (size_t)pos * d);
  const int n16 = d / 8;
  for (int i0 = 0; i0 < n16; i0 += 32 * 8) {
    uint4 v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int i = i0 + u * 32 + lane;
      if (i < n16) v[u] = src[i];
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int i = i0 + u * 32 + lane;
      if (i < n16) __stcs(dst + i, v[u]);
    }
  }
  if (lane == 0) inv_p[pos] = inv_s[tok];
}

// One thread per expert: ceil(count / tile_n) tiles, placed by an exclusive scan over experts.
// The tile's first field is the expert's weight slot (local_of[e], or e when every expert is held).
__global__ void __launch_bounds__(256) tiles_kernel(const int* __restrict__ counts, const int* __restrict__ offsets,
                                                    int n_exp, const int* __restrict__ local_of, int tile_n,
                                                    int4* __restrict__ tiles, int* __restrict__ n_tiles) {
  __shared__ int wsum[8];
  const int e = threadIdx.x, lane = e & 31, warp = e >> 5;
  const int cnt = e < n_exp ? counts[e] : 0;
  const int nt = (cnt + tile_n - 1) / tile_n;
  int inc = nt;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += v;
  }
  if (lane == 31) wsum[warp] = inc;
  __syncthreads();
  int base = 0, total = 0;
  for (int w = 0; w < 8; ++w) {
    if (w < warp) base += wsum[w];
    total += wsum[w];
  }
  const int first = base + inc - nt;
  const int off = e < n_exp ? offsets[e] : 0;
  const int slot = (e < n_exp && local_of) ? local_of[e] : e;
  for (int j = 0; j < nt; ++j) tiles[first + j] = make_int4(slot, off + j * tile_n, min(tile_n, cnt - j * tile_n), 0);
  if (e == 0) *n_tiles = total;
}

}  // namespace

void launch_xprep(const __nv_bfloat16* x, int n_tok, int d, __half* xs16, float* inv_s, cudaStream_t s) {
  xprep_kernel<<<n_tok, 256, 0, s>>>(x, d, xs16, inv_s);
}

void launch_gather(const __half* xs16, const float* inv_s, const int* perm, const int* n_pos, int n_slots, int top_k,
                   int d, __half* xp16, float* inv_p, cudaStream_t s) {
  gather_kernel<<<(n_slots + 7) / 8, 256, 0, s>>>(xs16, inv_s, perm, n_pos, n_slots, top_k, d, xp16, inv_p);
}

void launch_tiles(const int* counts, const int* offsets, int n_exp, const int* local_of, int tile_n, int4* tiles,
                  int* n_tiles, cudaStream_t s) {
  tiles_kernel<<<1, 256, 0, s>>>(counts, offsets, n_exp, local_of, tile_n, tiles, n_tiles);
}

}  // namespace ds4
