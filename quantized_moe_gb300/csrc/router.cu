// Router (fp32 logits, sigmoid top-k, table routing) and bucketing of (token, slot) pairs by
// expert. Every reduction runs in a fixed order, so routes are identical run to run.
#include "common.cuh"

namespace ds4 {
namespace {

constexpr int kRouterTok = 8;    // tokens per CTA
constexpr int kRouterWarps = 8;  // one expert per warp

// logits[t][e] = sum_k x[t][k] * W_r[e][k] + b[e], fp32 products and sums.
__global__ void __launch_bounds__(256) router_logits_kernel(const __nv_bfloat16* __restrict__ x, int n_tok, int d,
                                                            const float* __restrict__ w, const float* __restrict__ b,
                                                            int n_exp, float* __restrict__ logits) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  __nv_bfloat16* xs = reinterpret_cast<__nv_bfloat16*>(smem_raw);  // [kRouterTok][d]
  const int t0 = blockIdx.x * kRouterTok;
  const int nt = min(kRouterTok, n_tok - t0);
  for (int i = threadIdx.x * 8; i < kRouterTok * d; i += blockDim.x * 8) {
    const int tt = i / d;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (tt < nt) v = *reinterpret_cast<const uint4*>(x + (size_t)(t0 + tt) * d + (i % d));
    *reinterpret_cast<uint4*>(xs + i) = v;
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int e = blockIdx.y * kRouterWarps + warp;
  if (e >= n_exp) return;
  float acc[kRouterTok];
#pragma unroll
  for (int tt = 0; tt < kRouterTok; ++tt) acc[tt] = 0.f;
  const float* wr = w + (size_t)e * d;
  for (int k0 = lane * 4; k0 < d; k0 += 128) {
    const float4 wv = *reinterpret_cast<const float4*>(wr + k0);
#pragma unroll
    for (int tt = 0; tt < kRouterTok; ++tt) {
      const uint2 xv = *reinterpret_cast<const uint2*>(xs + tt * d + k0);
      const float2 x01 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&xv.x));
      const float2 x23 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&xv.y));
      acc[tt] = fmaf(wv.x, x01.x, acc[tt]);
      acc[tt] = fmaf(wv.y, x01.y, acc[tt]);
      acc[tt] = fmaf(wv.z, x23.x, acc[tt]);
      acc[tt] = fmaf(wv.w, x23.y, acc[tt]);
    }
  }
  const float bias = b ? b[e] : 0.f;
#pragma unroll
  for (int tt = 0; tt < kRouterTok; ++tt) {
    const float s = warp_sum(acc[tt]);
    if (lane == 0 && tt < nt) logits[(size_t)(t0 + tt) * n_exp + e] = s + bias;
  }
}

// One warp per token. Learned tokens: sigmoid scores, k rounds of warp argmax with ties to the
// lower expert index, weights renormalised to sum 1. Table tokens: experts = table[id], 1/k.
__global__ void topk_kernel(const float* __restrict__ logits, int n_learned, int n_exp, int top_k,
                            const int* __restrict__ token_ids, int n_hash, const int* __restrict__ table, int vocab,
                            int* __restrict__ idx, float* __restrict__ wts, int* __restrict__ err) {
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  const int n_tok = n_hash + n_learned;
  if (warp >= n_tok) return;
  const int t = warp;
  if (t < n_hash) {
    const int id = token_ids[t];
    const bool ok = id >= 0 && id < vocab;
    if (!ok && lane == 0) atomicOr(err, 1);
    if (lane < top_k) {
      idx[t * top_k + lane] = ok ? table[(size_t)id * top_k + lane] : 0;
      wts[t * top_k + lane] = ok ? 1.f / (float)top_k : 0.f;
    }
    return;
  }
  const float* z = logits + (size_t)(t - n_hash) * n_exp;
  constexpr int kPer = 8;  // n_exp <= 256
  float s[kPer];
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const int e = lane + 32 * i;
    s[i] = e < n_exp ? 1.f / (1.f + expf(-z[e])) : -1.f;
  }
  float sel_sum = 0.f;
  float my_w = 0.f;
  int my_e = 0;
  for (int j = 0; j < top_k; ++j) {
    // lane-local best (first max wins: lower index within the lane)
    float bv = s[0];
    int bi = lane;
#pragma unroll
    for (int i = 1; i < kPer; ++i)
      if (s[i] > bv) { bv = s[i]; bi = lane + 32 * i; }
    // warp argmax by (value desc, index asc)
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      if (ov > bv || (ov == bv && oi < bi)) { bv = ov; bi = oi; }
    }
    if ((bi & 31) == lane) s[bi >> 5] = -2.f;  // remove the winner
    sel_sum += bv;
    if (lane == j) { my_w = bv; my_e = bi; }
  }
  if (lane < top_k) {
    idx[t * top_k + lane] = my_e;
    wts[t * top_k + lane] = my_w / sel_sum;
  }
}

// CTA e counts the slots routed to expert e.
__global__ void bucket_count_kernel(const int* __restrict__ idx, int n_slots, int* __restrict__ counts) {
  __shared__ int part[32];
  const int e = blockIdx.x;
  int c = 0;
  for (int i = threadIdx.x; i < n_slots; i += blockDim.x) c += idx[i] == e;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
  if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = c;
  __syncthreads();
  if (threadIdx.x == 0) {
    int tot = 0;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) tot += part[w];
    counts[e] = tot;
  }
}

// CTA e: offset of expert e, its index among the active experts, and an order-preserving
// compaction of its slots (so positions are sorted by (expert, token, slot)).
__global__ void bucket_scatter_kernel(const int* __restrict__ idx, int n_slots, int n_exp,
                                      const int* __restrict__ counts, int* __restrict__ offsets,
                                      int* __restrict__ active, int* __restrict__ n_active, int* __restrict__ perm,
                                      int* __restrict__ rowof) {
  __shared__ int s_off, s_act, s_nact;
  __shared__ int warp_tot[32];
  const int e = blockIdx.x;
  if (threadIdx.x == 0) { s_off = 0; s_act = 0; s_nact = 0; }
  __syncthreads();
  int off = 0, act = 0, nact = 0;
  for (int i = threadIdx.x; i < n_exp; i += blockDim.x) {
    const int c = counts[i];
    if (i < e) { off += c; act += c > 0; }
    nact += c > 0;
  }
  atomicAdd(&s_off, off);  // integer sums: order does not change the result
  atomicAdd(&s_act, act);
  atomicAdd(&s_nact, nact);
  __syncthreads();
  const int base = s_off;
  if (threadIdx.x == 0) {
    offsets[e] = base;
    if (e == n_exp - 1) offsets[n_exp] = base + counts[e];
    if (counts[e] > 0) active[s_act] = e;
    if (e == 0) *n_active = s_nact;
  }
  if (counts[e] == 0) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  int running = base;
  for (int i0 = 0; i0 < n_slots; i0 += blockDim.x) {
    const int i = i0 + threadIdx.x;
    const bool hit = i < n_slots && idx[i] == e;
    const unsigned m = __ballot_sync(0xffffffffu, hit);
    __syncthreads();
    if (lane == 0) warp_tot[warp] = __popc(m);
    __syncthreads();
    int before = 0, tot = 0;
    for (int w = 0; w < nw; ++w) {
      const int c = warp_tot[w];
      if (w < warp) before += c;
      tot += c;
    }
    if (hit) {
      const int pos = running + before + __popc(m & ((1u << lane) - 1u));
      perm[pos] = i;
      rowof[i] = pos;
    }
    running += tot;
  }
}

}  // namespace

void launch_router_logits(const __nv_bfloat16* x, int n_tok, int d, const float* w, const float* b, int n_exp,
                          float* logits, cudaStream_t s) {
  const size_t smem = (size_t)kRouterTok * d * sizeof(__nv_bfloat16);
  static bool attr_set = false;  // per-process; the attribute is per function, not per device
  if (!attr_set) {
    cudaFuncSetAttribute(router_logits_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
    attr_set = true;
  }
  dim3 grid((n_tok + kRouterTok - 1) / kRouterTok, (n_exp + kRouterWarps - 1) / kRouterWarps);
  router_logits_kernel<<<grid, 256, smem, s>>>(x, n_tok, d, w, b, n_exp, logits);
}

void launch_topk(const float* logits, int n_learned, int n_exp, int top_k, const int* token_ids, int n_hash,
                 const int* table, int vocab, int* idx, float* wts, int* err, cudaStream_t s) {
  const int n_tok = n_learned + n_hash;
  const int warps_per_block = 8;
  topk_kernel<<<(n_tok + warps_per_block - 1) / warps_per_block, 32 * warps_per_block, 0, s>>>(
      logits, n_learned, n_exp, top_k, token_ids, n_hash, table, vocab, idx, wts, err);
}

void launch_bucket_count(const int* idx, int n_slots, int n_exp, int* counts, cudaStream_t s) {
  bucket_count_kernel<<<n_exp, 256, 0, s>>>(idx, n_slots, counts);
}

void launch_bucket_scatter(const int* idx, int n_slots, int n_exp, const int* counts, int* offsets, int* active,
                           int* n_active, int* perm, int* rowof, cudaStream_t s) {
  bucket_scatter_kernel<<<n_exp, 256, 0, s>>>(idx, n_slots, n_exp, counts, offsets, active, n_active, perm, rowof);
}

}  // namespace ds4
