// Router (fp32 logits, sigmoid top-k, table routing) and bucketing of (token, slot) pairs by
// expert. Every reduction runs in a fixed order, so routes are identical run to run.
#include "common.cuh"

namespace ds4 {
namespace {

constexpr int kRouterTok = 8;    // tokens per CTA
constexpr int kRouterWarps = 8;  // one expert per warp (measured: four per CTA was slower)

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
  // four weight loads per lane and step (d is a multiple of 128), the next step's issued before
  // this step's FMAs; the products are summed in the same order as one k step after another
  float4 nx[4];
#pragma unroll
  for (int u = 0; u < 4; ++u)
    nx[u] = lane * 4 + 128 * u < d ? *reinterpret_cast<const float4*>(wr + lane * 4 + 128 * u) : make_float4(0.f, 0.f, 0.f, 0.f);
  for (int k0 = lane * 4; k0 < d; k0 += 512) {
    float4 wv[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) wv[u] = nx[u];
#pragma unroll
    for (int u = 0; u < 4; ++u)
      nx[u] = k0 + 512 + 128 * u < d ? *reinterpret_cast<const float4*>(wr + k0 + 512 + 128 * u)
                                     : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      if (k0 + 128 * u >= d) break;
#pragma unroll
      for (int tt = 0; tt < kRouterTok; ++tt) {
        const uint2 xv = *reinterpret_cast<const uint2*>(xs + tt * d + k0 + 128 * u);
        const float2 x01 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&xv.x));
        const float2 x23 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&xv.y));
        acc[tt] = fmaf(wv[u].x, x01.x, acc[tt]);
        acc[tt] = fmaf(wv[u].y, x01.y, acc[tt]);
        acc[tt] = fmaf(wv[u].z, x23.x, acc[tt]);
        acc[tt] = fmaf(wv[u].w, x23.y, acc[tt]);
      }
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
      idx[t * top_k + lane] = ok ? table[(size_t)id * top_k + lane] : lane;  // bad id: distinct experts, weight 0
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
// Bucketing in two passes over chunks of kChunk slots (one CTA each, 256 threads, E <= 256).
constexpr int kChunk = 1024;

// Pass 1: per-chunk histogram of the experts (integer counts, order-free).
__global__ void __launch_bounds__(256) bucket_hist_kernel(const int* __restrict__ idx, int n_slots, int n_exp,
                                                          const int* __restrict__ local_of, int* __restrict__ ghist) {
  __shared__ int hist[256];
  if (threadIdx.x < n_exp) hist[threadIdx.x] = 0;
  __syncthreads();
  const int s0 = blockIdx.x * kChunk;
  for (int i = threadIdx.x; i < kChunk && s0 + i < n_slots; i += 256) {
    const int e = idx[s0 + i];
    if (!local_of || local_of[e] >= 0) atomicAdd(&hist[e], 1);  // only the experts this handle holds
  }
  __syncthreads();
  if (threadIdx.x < n_exp) ghist[(size_t)blockIdx.x * n_exp + threadIdx.x] = hist[threadIdx.x];
}

// Pass 2: chunk b places its slots at offsets[e] + (slots of e in earlier chunks) + (earlier slots
// of e in this chunk), so positions are sorted by (expert, slot) = (expert, token, slot). Ranks
// inside a round of 256 slots come from warp match masks and per-warp counts. Chunk 0 also
// publishes counts, offsets, the active experts and their number. Slots of experts the handle does
// not hold get no position (rowof = -1).
__global__ void __launch_bounds__(256) bucket_place_kernel(const int* __restrict__ idx, int n_slots, int n_exp,
                                                           const int* __restrict__ ghist, int n_chunks,
                                                           const int* __restrict__ local_of,
                                                           int* __restrict__ counts, int* __restrict__ offsets,
                                                           int* __restrict__ active, int* __restrict__ n_active,
                                                           int* __restrict__ perm, int* __restrict__ rowof) {
  __shared__ int run[256];        // next position of each expert for this chunk
  __shared__ int wcnt[8][256];    // slots of each expert per warp in the current round
  __shared__ int scan_w[8], scan_a[8];
  const int e = threadIdx.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int tot = 0, pre = 0;
  if (e < n_exp)
    for (int b = 0; b < n_chunks; ++b) {
      const int c = ghist[(size_t)b * n_exp + e];
      tot += c;
      if (b < (int)blockIdx.x) pre += c;
    }
  // exclusive scans over the experts of the totals and of the active flags (block-wide)
  int inc = tot, inca = tot > 0;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, inc, o), va = __shfl_up_sync(0xffffffffu, inca, o);
    if (lane >= o) { inc += v; inca += va; }
  }
  if (lane == 31) { scan_w[warp] = inc; scan_a[warp] = inca; }
  __syncthreads();
  int wbase = 0, abase = 0, all = 0, all_a = 0;
  for (int w = 0; w < 8; ++w) {
    if (w < warp) { wbase += scan_w[w]; abase += scan_a[w]; }
    all += scan_w[w];
    all_a += scan_a[w];
  }
  const int off = wbase + inc - tot;  // exclusive
  if (e < n_exp) {
    run[e] = off + pre;
    if (blockIdx.x == 0) {
      counts[e] = tot;
      offsets[e] = off;
      if (tot > 0) active[abase + inca - 1] = e;
    }
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    offsets[n_exp] = all;
    *n_active = all_a;
  }
  const unsigned lt = (1u << lane) - 1u;
  const int s0 = blockIdx.x * kChunk;
  for (int r0 = 0; r0 < kChunk; r0 += 256) {
    for (int k = threadIdx.x; k < 8 * 256; k += 256) (&wcnt[0][0])[k] = 0;
    __syncthreads();
    const int sl = s0 + r0 + threadIdx.x;
    int ex = sl < n_slots ? idx[sl] : -1;
    if (ex >= 0 && local_of && local_of[ex] < 0) {
      rowof[sl] = -1;
      ex = -1;
    }
    const unsigned m = __match_any_sync(0xffffffffu, ex);
    const int rank = __popc(m & lt);
    if (ex >= 0 && rank == 0) wcnt[warp][ex] = __popc(m);
    __syncthreads();
    if (ex >= 0) {
      int pos = run[ex] + rank;
      for (int w = 0; w < warp; ++w) pos += wcnt[w][ex];
      perm[pos] = sl;
      rowof[sl] = pos;
    }
    __syncthreads();
    if (e < n_exp) {
      int add = 0;
      for (int w = 0; w < 8; ++w) add += wcnt[w][e];
      run[e] += add;
    }
    __syncthreads();
  }
}

}  // namespace

void launch_router_logits(const __nv_bfloat16* x, int n_tok, int d, const float* w, const float* b, int n_exp,
                          float* logits, cudaStream_t s) {
  const size_t smem = (size_t)kRouterTok * d * sizeof(__nv_bfloat16);
  dim3 grid((n_tok + kRouterTok - 1) / kRouterTok, (n_exp + kRouterWarps - 1) / kRouterWarps);
  router_logits_kernel<<<grid, 32 * kRouterWarps, smem, s>>>(x, n_tok, d, w, b, n_exp, logits);
}

// The kernel stages up to 8 x 12288 bf16 activations (192 KB) in shared memory. Function
// attributes belong to the current device's context: call once per device before launching there.
cudaError_t router_logits_prepare() {
  return cudaFuncSetAttribute(router_logits_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              kRouterTok * 12288 * (int)sizeof(__nv_bfloat16));
}

void launch_topk(const float* logits, int n_learned, int n_exp, int top_k, const int* token_ids, int n_hash,
                 const int* table, int vocab, int* idx, float* wts, int* err, cudaStream_t s) {
  const int n_tok = n_learned + n_hash;
  const int warps_per_block = 8;
  topk_kernel<<<(n_tok + warps_per_block - 1) / warps_per_block, 32 * warps_per_block, 0, s>>>(
      logits, n_learned, n_exp, top_k, token_ids, n_hash, table, vocab, idx, wts, err);
}

int bucket_chunks(int n_slots) { return (n_slots + kChunk - 1) / kChunk; }

void launch_bucket_count(const int* idx, int n_slots, int n_exp, const int* local_of, int* ghist, cudaStream_t s) {
  bucket_hist_kernel<<<bucket_chunks(n_slots), 256, 0, s>>>(idx, n_slots, n_exp, local_of, ghist);
}

void launch_bucket_scatter(const int* idx, int n_slots, int n_exp, const int* ghist, const int* local_of, int* counts,
                           int* offsets, int* active, int* n_active, int* perm, int* rowof, cudaStream_t s) {
  const int nc = bucket_chunks(n_slots);
  bucket_place_kernel<<<nc, 256, 0, s>>>(idx, n_slots, n_exp, ghist, nc, local_of, counts, offsets, active, n_active,
                                         perm, rowof);
}

}  // namespace ds4
