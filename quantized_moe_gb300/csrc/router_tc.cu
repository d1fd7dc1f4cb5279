// Batched router logits on the tensor cores with fp32 accuracy.
//
// The fp32 router weights are split once, at create time, into three bf16 parts
// w = w_hi + w_mid + w_lo (8 + 8 + 8 significand bits cover all 24 of fp32). The activations are
// bf16 already, so every product x * w_part is exact in fp32; the three MMAs of each 16-wide K
// step go into a fresh fp32 accumulator, which is added to the running sum with ordinary fp32
// adds: the accuracy of fp32 FMAs on the CUDA cores, at tensor-core throughput.
//
// CTA = TT tokens x TE experts (TE = 64, or 32 for batches up to 1024 tokens), one warp per 16
// tokens x 16 experts (TT = 96, TE = 64 gives 24 warps: enough per SM to hide the MMA -> add
// chains); K staged through shared memory 32 at a time in a four-deep cp.async pipeline (three steps
// of loads in flight). TT is chosen per call from the token count so that the grid fills the SMs in
// as few rounds as possible; every logit is the same sequence of operations whatever the tile, so
// the result does not depend on TT or TE.
#include "common.cuh"

namespace ds4 {
namespace {

constexpr int KS = 32;
constexpr int PAD = 8;  // bf16 elements of padding per shared row (keeps ldmatrix conflict-free)
constexpr int LDS = KS + PAD;
constexpr int NSTAGE = 4;
template <int TT, int TE>
struct Stage {
  __nv_bfloat16 x[TT][LDS];
  __nv_bfloat16 w[3][TE][LDS];
};
template <int TT, int TE>
constexpr int smem_bytes() { return NSTAGE * (int)sizeof(Stage<TT, TE>); }
template <int TT, int TE>
constexpr int threads_of() { return TT / 16 * (TE / 16) * 32; }  // warps: token groups x expert groups

__device__ __forceinline__ void cp_async16(void* dst, const void* src, bool pred) {
  const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(dst));
  const int sz = pred ? 16 : 0;  // zero-fill rows past the end
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(d), "l"(src), "r"(sz) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory"); }

__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldmatrix_x2(uint32_t addr, uint32_t& r0, uint32_t& r1) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];\n" : "=r"(r0), "=r"(r1) : "r"(addr));
}
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// w3: [3][E][d] bf16 parts of the router weights
template <int TT, int TE>
__global__ void __launch_bounds__(threads_of<TT, TE>()) router_tc_kernel(const __nv_bfloat16* __restrict__ x, int n_tok,
                                                                     int d, const __nv_bfloat16* __restrict__ w3,
                                                                     const float* __restrict__ b, int n_exp,
                                                                     float* __restrict__ logits) {
  constexpr int kThreads = threads_of<TT, TE>(), NTG = TT / 16, CPR = KS / 8;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  Stage<TT, TE>* st = reinterpret_cast<Stage<TT, TE>*>(smem_raw);
  const int t0 = blockIdx.x * TT, e0 = blockIdx.y * TE;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const size_t plane = (size_t)n_exp * d;
  auto stage = [&](int buf, int k0) {
    // TT rows of x and 3 x 64 rows of weight parts, 32 k = 4 chunks of 16 bytes each
    for (int c = threadIdx.x; c < (TT + 3 * TE) * CPR; c += kThreads) {
      const int row = c / CPR, kc = c % CPR;
      if (row < TT) {
        const int t = t0 + row;
        cp_async16(&st[buf].x[row][kc * 8], x + (size_t)min(t, n_tok - 1) * d + k0 + kc * 8, t < n_tok);
      } else {
        const int which = (row - TT) / TE, r = (row - TT) % TE, e = e0 + r;
        cp_async16(&st[buf].w[which][r][kc * 8], w3 + which * plane + (size_t)min(e, n_exp - 1) * d + k0 + kc * 8,
                   e < n_exp);
      }
    }
    cp_async_commit();
  };
  const int tw = warp % NTG, ew = warp / NTG;  // token group (16 tokens), expert group (16 experts)
  float acc[2][4];
#pragma unroll
  for (int j = 0; j < 2; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;
  const int n_k = d / KS;
  for (int s0 = 0; s0 < NSTAGE - 1; ++s0) {
    if (s0 < n_k)
      stage(s0, s0 * KS);
    else
      cp_async_commit();  // empty group: the group count stays in step
  }
  for (int ks = 0; ks < n_k; ++ks) {
    const int buf = ks % NSTAGE;
    cp_async_wait<NSTAGE - 2>();  // step ks has landed (for this thread)
    __syncthreads();              // ... for every thread, and step ks - 1's buffer is free again
    const int nxt = ks + NSTAGE - 1;
    if (nxt < n_k)
      stage(nxt % NSTAGE, nxt * KS);
    else
      cp_async_commit();
#pragma unroll
    for (int kk = 0; kk < KS; kk += 16) {
      uint32_t a[4];
      {  // A: 16 tokens x 16 k of this warp (row-major)
        const int r = tw * 16 + (lane & 15), c = kk + (lane >> 4) * 8;
        ldmatrix_x4(static_cast<uint32_t>(__cvta_generic_to_shared(&st[buf].x[r][c])), a[0], a[1], a[2], a[3]);
      }
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        // The tensor core's accumulation truncates; a long chain of MMAs into one accumulator
        // would bias the sum. Each 16-wide K step therefore starts from zero and is added to
        // the running fp32 sum with round-to-nearest adds.
        float tmp[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int part = 0; part < 3; ++part) {  // B: 8 experts x 16 k (expert rows, k contiguous)
          const int r = ew * 16 + j * 8 + (lane & 7), c = kk + ((lane >> 3) & 1) * 8;
          uint32_t b0, b1;
          ldmatrix_x2(static_cast<uint32_t>(__cvta_generic_to_shared(&st[buf].w[part][r][c])), b0, b1);
          mma_bf16_16816(tmp, a, b0, b1);
        }
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[j][c] += tmp[c];
      }
    }
  }
  cp_async_wait<0>();
  // C fragment: rows g, g+8 (tokens), columns 2t, 2t+1 (experts)
  const int g = lane >> 2, t = lane & 3;
#pragma unroll
  for (int j = 0; j < 2; ++j)
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int tok = t0 + tw * 16 + g + 8 * (c >> 1), e = e0 + ew * 16 + j * 8 + 2 * t + (c & 1);
      if (tok < n_tok && e < n_exp) logits[(size_t)tok * n_exp + e] = acc[j][c] + (b ? b[e] : 0.f);
    }
}

// w -> (hi, mid, lo) bf16 parts with w = hi + mid + lo (round to nearest at each step).
__global__ void split3_kernel(const float* __restrict__ w, size_t n, __nv_bfloat16* __restrict__ out) {
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
    const float v = w[i];
    const __nv_bfloat16 hi = __float2bfloat16_rn(v);
    const float r1 = v - __bfloat162float(hi);
    const __nv_bfloat16 mid = __float2bfloat16_rn(r1);
    const __nv_bfloat16 lo = __float2bfloat16_rn(r1 - __bfloat162float(mid));
    out[i] = hi;
    out[n + i] = mid;
    out[2 * n + i] = lo;
  }
}

}  // namespace

void launch_router_split(const float* w, size_t n, __nv_bfloat16* w3, cudaStream_t s) {
  split3_kernel<<<152 * 4, 256, 0, s>>>(w, n, w3);
}

namespace {
template <int TT, int TE>
void launch_tt(const __nv_bfloat16* x, int n_tok, int d, const __nv_bfloat16* w3, const float* b, int n_exp,
               float* logits, cudaStream_t s) {
  const dim3 grid((n_tok + TT - 1) / TT, (n_exp + TE - 1) / TE);
  router_tc_kernel<TT, TE><<<grid, threads_of<TT, TE>(), smem_bytes<TT, TE>(), s>>>(x, n_tok, d, w3, b, n_exp, logits);
}
template <int TT, int TE>
cudaError_t prepare_tt() {
  return cudaFuncSetAttribute(router_tc_kernel<TT, TE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              smem_bytes<TT, TE>());
}
template <int TE>
cudaError_t prepare_te() {
  cudaError_t e = prepare_tt<96, TE>();
  if (e == cudaSuccess) e = prepare_tt<64, TE>();
  if (e == cudaSuccess) e = prepare_tt<32, TE>();
  if (e == cudaSuccess) e = prepare_tt<16, TE>();
  return e;
}
template <int TE>
void launch_te(int tt, const __nv_bfloat16* x, int n_tok, int d, const __nv_bfloat16* w3, const float* b, int n_exp,
               float* logits, cudaStream_t s) {
  switch (tt) {
    case 96: launch_tt<96, TE>(x, n_tok, d, w3, b, n_exp, logits, s); break;
    case 32: launch_tt<32, TE>(x, n_tok, d, w3, b, n_exp, logits, s); break;
    case 16: launch_tt<16, TE>(x, n_tok, d, w3, b, n_exp, logits, s); break;
    default: launch_tt<64, TE>(x, n_tok, d, w3, b, n_exp, logits, s); break;
  }
}
// Expert tile: 32 experts per CTA up to 1024 tokens (twice the CTAs, more of them resident: 95 ->
// 78 us at 512 tokens), 64 above (fewer re-reads of each token tile: 158 vs 163 us at 3072).
int router_tile_experts(int n_tok) { return n_tok <= 1024 ? 32 : 64; }
}  // namespace

// Function attributes belong to the current device's context: called once per device (by the
// handle's create, with the handle's device current) before any launch there.
cudaError_t router_tc_prepare() {
  cudaError_t e = prepare_te<64>();
  if (e == cudaSuccess) e = prepare_te<32>();
  return e;
}

// Token tile: the one with the fewest rounds of CTAs over the SMs, weighting a CTA's time by
// TT + 32 (its weight tile costs about as much as 32 tokens), larger tiles winning ties.
int router_tile_tokens(int n_tok, int n_exp, int n_sm, int te) {
  static const int cand[4] = {96, 64, 32, 16};
  int best = 64;
  long best_cost = -1;
  for (int tt : cand) {
    const long ctas = (long)((n_tok + tt - 1) / tt) * ((n_exp + te - 1) / te);
    const long cost = (ctas + n_sm - 1) / n_sm * (tt + 32);
    if (best_cost < 0 || cost < best_cost) {
      best_cost = cost;
      best = tt;
    }
  }
  return best;
}

void launch_router_tc(const __nv_bfloat16* x, int n_tok, int d, const __nv_bfloat16* w3, const float* b, int n_exp,
                      float* logits, cudaStream_t s) {
  static int n_sm[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !n_sm[dev]) cudaDeviceGetAttribute(&n_sm[dev], cudaDevAttrMultiProcessorCount, dev);
  const int sms = (dev >= 0 && dev < 64 && n_sm[dev] > 0) ? n_sm[dev] : 152;
  const int te = router_tile_experts(n_tok), tt = router_tile_tokens(n_tok, n_exp, sms, te);
  if (te == 32)
    launch_te<32>(tt, x, n_tok, d, w3, b, n_exp, logits, s);
  else
    launch_te<64>(tt, x, n_tok, d, w3, b, n_exp, logits, s);
}

}  // namespace ds4
