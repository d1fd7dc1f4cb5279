// Fused dequant expert GEMV/GEMM on the warp-level tensor-core path (mma.m16n8k16, fp16 in,
// fp32 accumulate), for the gate/up (+SwiGLU) and down projections of routed and shared
// experts.
//
// Dequantization is folded into the MMA instead of being done per weight:
//  * A fragments are built from the packed quants with one AND (Q2_K) or one PRMT (Q8_0) per
//    register: the quant lands in the low mantissa bits of an fp16 with a zero exponent,
//    i.e. the exact subnormal value q * 2^(p-24). No conversion instruction, no rounding.
//  * The B operand is the activation row, scaled by a power of two into fp16 range (exact).
//    For MMA i of a 128-wide K chunk, only lanes of group g == i pass their activations, so
//    column n of the accumulator holds the dot product of sub-block n alone: after eight MMAs
//    each lane owns two rows x two sub-blocks and applies their scales itself, and all four
//    lanes of a row group do useful work even for a single token.
//  * Per sub-block scales and mins are applied in fp32 FMAs on the accumulator:
//      Q2_K: sum_j d s_j (q . x)_j - dmin m_j X_j      Q8_0: sum_b scale_b ((u . x)_b - 128 X_b)
//    with X the sub-block sums of the (scaled) activations and u = q + 128.
// Each CTA owns 16 output rows of one expert and splits K over its 8 warps; partial sums are
// combined in a fixed order, so results are bitwise repeatable.
#include "common.cuh"

namespace ds4 {
namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kTmax = 4;  // token rows per pass

struct Stage {
  __half* xs;     // [kTmax][k] scaled fp16 rows
  float* xsum;    // [kTmax][k/16] sub-block sums of the scaled rows
  float* red;     // [kWarps][2][kTmax][16] per-warp row partials
  float* inv;     // [kTmax] 1 / row scale
};

__device__ __forceinline__ Stage carve(unsigned char* smem, int k) {
  Stage s;
  s.xs = reinterpret_cast<__half*>(smem);
  s.xsum = reinterpret_cast<float*>(smem + (size_t)kTmax * k * 2);
  s.red = s.xsum + kTmax * (k / 16);
  s.inv = s.red + kWarps * 2 * kTmax * 16;
  return s;
}

__device__ __forceinline__ float block_max(float v, float* scratch) {
  v = warp_max(v);
  __syncthreads();
  if ((threadIdx.x & 31) == 0) scratch[threadIdx.x >> 5] = v;
  __syncthreads();
  float m = 0.f;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) m = fmaxf(m, scratch[w]);
  return m;
}

// Stage one input row (bf16 or fp32) as scaled fp16 plus 16-wide sub-block sums. Each lane
// converts 8 elements (half a sub-block); k is a multiple of 128, so the pair of lanes that
// shares a sub-block is always both in or both out of range.
template <typename T>
__device__ void stage_row(const T* __restrict__ src, int k, __half* dst, float* sums, float* inv_out,
                          float* scratch) {
  float mx = 0.f;
  for (int i = threadIdx.x; i < k; i += kThreads) mx = fmaxf(mx, fabsf((float)src[i]));
  mx = block_max(mx, scratch);
  const float sc = fp16_row_scale(mx);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int base = warp * 256; base < k; base += kThreads * 8) {  // warp-uniform bound
    const int i0 = base + lane * 8;
    const bool ok = i0 < k;
    float part = 0.f;
    uint32_t packed[4] = {0u, 0u, 0u, 0u};
    if (ok) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const __half2 h2 = __floats2half2_rn((float)src[i0 + 2 * e] * sc, (float)src[i0 + 2 * e + 1] * sc);
        const float2 back = __half22float2(h2);
        part += back.x + back.y;
        packed[e] = *reinterpret_cast<const uint32_t*>(&h2);
      }
      *reinterpret_cast<uint4*>(dst + i0) = make_uint4(packed[0], packed[1], packed[2], packed[3]);
    }
    part += __shfl_xor_sync(0xffffffffu, part, 1);  // the neighbour holds the other half
    if (ok && (lane & 1) == 0) sums[i0 >> 4] = part;
  }
  if (threadIdx.x == 0) *inv_out = 1.f / sc;
}

// Exact small-integer extraction through an fp32 with exponent 2^23: (bits | 0x4B000000)
// equals 2^23 + field * 2^pos; fmaf(v, c, -2^23 c) then yields field * 2^pos * c exactly.
__device__ __forceinline__ float magic_scaled(uint32_t masked_bits, float c) {
  return fmaf(__uint_as_float(masked_bits | 0x4B000000u), c, -8388608.f * c);
}

// Q2_K: per-lane constants 2^(24 - p) for the lane's two columns (MMA slot shift p).
__device__ __forceinline__ float q2k_col_scale(int n) {  // n = sub-block in chunk 0..7
  const int p = n < 5 ? 2 * n : 2 * (n - 5);
  return ldexpf(1.f, 24 - p);
}

// Process one Q2_K unit (16 rows x 256 k) of one matrix for nt token rows.
// acc[tt][rho]: lane partial of row g + 8 rho for token tt.
__device__ __forceinline__ void q2k_unit(const uint8_t* __restrict__ ub, const Stage& st, int k, int kbase, int nt,
                                         float (&acc)[kTmax][2], float c0, float c1) {
  const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
  const uint4 qv[2] = {ldg_nc_v4(ub + 16 * lane), ldg_nc_v4(ub + 512 + 16 * lane)};
  const uint32_t scw[2] = {ldg_nc_u32(ub + kQ2kScOff + 4 * lane), ldg_nc_u32(ub + kQ2kScOff + 128 + 4 * lane)};
  const uint32_t dd0 = ldg_nc_u32(ub + kQ2kDdOff + 4 * g);
  const uint32_t dd1 = ldg_nc_u32(ub + kQ2kDdOff + 4 * (g + 8));
  float as_[kTmax][2], am_[kTmax][2];
#pragma unroll
  for (int tt = 0; tt < kTmax; ++tt) as_[tt][0] = as_[tt][1] = am_[tt][0] = am_[tt][1] = 0.f;
#pragma unroll
  for (int c = 0; c < 2; ++c) {
    const uint32_t w[4] = {qv[c].x, qv[c].y, qv[c].z, qv[c].w};
    const uint32_t wh[4] = {w[0] >> 10, w[1] >> 10, w[2] >> 10, w[3] >> 10};
    const uint32_t sc = scw[c], sh = scw[c] >> 16;
    // scales s (times the column constant) and mins m of (row rho, column n)
    const float s00 = magic_scaled(sc & 0xFu, c0), s01 = magic_scaled(sc & 0xF00u, c1 * (1.f / 256.f));
    const float s10 = magic_scaled(sh & 0xFu, c0), s11 = magic_scaled(sh & 0xF00u, c1 * (1.f / 256.f));
    const float m00 = magic_scaled(sc & 0xF0u, 1.f / 16.f), m01 = magic_scaled(sc & 0xF000u, 1.f / 4096.f);
    const float m10 = magic_scaled(sh & 0xF0u, 1.f / 16.f), m11 = magic_scaled(sh & 0xF000u, 1.f / 4096.f);
    const int kc = kbase + 128 * c;
#pragma unroll
    for (int tt = 0; tt < kTmax; ++tt) {
      if (tt >= nt) break;
      const __half* xr = st.xs + tt * k + kc;
      const uint32_t xb0 = *reinterpret_cast<const uint32_t*>(xr + 16 * g + 2 * t);
      const uint32_t xb1 = *reinterpret_cast<const uint32_t*>(xr + 16 * g + 2 * t + 8);
      const float2 xsum = *reinterpret_cast<const float2*>(st.xsum + tt * (k / 16) + kc / 16 + 2 * t);
      float dacc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const uint32_t mask = 0x00030003u << (2 * (i < 5 ? i : i - 5));
        uint32_t a[4];
#pragma unroll
        for (int r = 0; r < 4; ++r) a[r] = (i < 5 ? w[r] : wh[r]) & mask;
        const bool mine = g == i;
        mma_f16_16816(dacc, a, mine ? xb0 : 0u, mine ? xb1 : 0u);
      }
      as_[tt][0] = fmaf(s00, dacc[0], fmaf(s01, dacc[1], as_[tt][0]));
      as_[tt][1] = fmaf(s10, dacc[2], fmaf(s11, dacc[3], as_[tt][1]));
      am_[tt][0] = fmaf(m00, xsum.x, fmaf(m01, xsum.y, am_[tt][0]));
      am_[tt][1] = fmaf(m10, xsum.x, fmaf(m11, xsum.y, am_[tt][1]));
    }
  }
  const float2 d0 = __half22float2(*reinterpret_cast<const __half2*>(&dd0));  // (d, dmin) of row g
  const float2 d1 = __half22float2(*reinterpret_cast<const __half2*>(&dd1));  // row g + 8
#pragma unroll
  for (int tt = 0; tt < kTmax; ++tt) {
    if (tt >= nt) break;
    acc[tt][0] = fmaf(d0.x, as_[tt][0], fmaf(-d0.y, am_[tt][0], acc[tt][0]));
    acc[tt][1] = fmaf(d1.x, as_[tt][1], fmaf(-d1.y, am_[tt][1], acc[tt][1]));
  }
}

// Process one Q8_0 unit (16 rows x 128 k) of one matrix.
__device__ __forceinline__ void q80_unit(const uint8_t* __restrict__ ub, const Stage& st, int k, int kbase, int nt,
                                         float (&acc)[kTmax][2]) {
  const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
  uint4 v[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) v[j] = ldg_nc_v4(ub + 512 * j + 16 * lane);
  const uint32_t scw = ldg_nc_u32(ub + kQ80ScOff + 4 * lane);
  const float2 sc = __half22float2(*reinterpret_cast<const __half2*>(&scw));  // rows g, g+8 of block t
#pragma unroll
  for (int tt = 0; tt < kTmax; ++tt) {
    if (tt >= nt) break;
    const __half* xr = st.xs + tt * k + kbase;
    const uint32_t xb0 = *reinterpret_cast<const uint32_t*>(xr + 16 * g + 2 * t);
    const uint32_t xb1 = *reinterpret_cast<const uint32_t*>(xr + 16 * g + 2 * t + 8);
    const float2 xsum = *reinterpret_cast<const float2*>(st.xsum + tt * (k / 16) + kbase / 16 + 2 * t);
    float dacc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int j = i >> 1, m = i & 1;
      const uint32_t wa = m ? v[j].z : v[j].x;  // registers 0, 1
      const uint32_t wb = m ? v[j].w : v[j].y;  // registers 2, 3
      const uint32_t a[4] = {prmt(wa, 0u, 0x4140u), prmt(wa, 0u, 0x4342u), prmt(wb, 0u, 0x4140u),
                             prmt(wb, 0u, 0x4342u)};
      const bool mine = g == i;
      mma_f16_16816(dacc, a, mine ? xb0 : 0u, mine ? xb1 : 0u);
    }
    const float xs2 = 128.f * (xsum.x + xsum.y);
    acc[tt][0] = fmaf(sc.x, fmaf(16777216.f, dacc[0] + dacc[1], -xs2), acc[tt][0]);
    acc[tt][1] = fmaf(sc.y, fmaf(16777216.f, dacc[2] + dacc[3], -xs2), acc[tt][1]);
  }
}

template <int FMT, bool GATEUP>
__global__ void __launch_bounds__(kThreads) expert_gemv_kernel(GemvArgs a) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  __shared__ float scratch[kWarps];
  const int k = a.k;
  const Stage st = carve(smem_raw, k);
  const int rg = blockIdx.x;
  int e = 0, pos0 = 0, cnt = a.n_tokens;
  const bool routed = a.active != nullptr;
  if (routed) {
    if ((int)blockIdx.y >= *a.n_active) return;
    e = a.active[blockIdx.y];
    pos0 = a.offsets[e];
    cnt = a.offsets[e + 1] - pos0;
  }
  constexpr int NM = GATEUP ? 2 : 1;
  const uint8_t* wm[2] = {a.w0 + (size_t)e * a.mat_bytes, GATEUP ? a.w1 + (size_t)e * a.mat_bytes : nullptr};
  const int n_kb = k / unit_k(FMT);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
  const float c0 = q2k_col_scale(2 * t), c1 = q2k_col_scale(2 * t + 1);

  for (int p0 = 0; p0 < cnt; p0 += kTmax) {
    const int nt = min(kTmax, cnt - p0);
    __syncthreads();  // the previous pass is done with shared memory
    for (int tt = 0; tt < nt; ++tt) {
      const int pos = pos0 + p0 + tt;
      if (GATEUP) {
        const int tok = routed ? a.perm[pos] / a.top_k : pos;
        stage_row(a.x + (size_t)tok * k, k, st.xs + tt * k, st.xsum + tt * (k / 16), st.inv + tt, scratch);
      } else {
        stage_row(a.hin + (size_t)pos * k, k, st.xs + tt * k, st.xsum + tt * (k / 16), st.inv + tt, scratch);
      }
    }
    __syncthreads();
    float acc[NM][kTmax][2];
#pragma unroll
    for (int m = 0; m < NM; ++m)
#pragma unroll
      for (int tt = 0; tt < kTmax; ++tt) acc[m][tt][0] = acc[m][tt][1] = 0.f;
    for (int kb = warp; kb < n_kb; kb += kWarps) {
#pragma unroll
      for (int m = 0; m < NM; ++m) {
        const uint8_t* ub = wm[m] + unit_offset(rg, kb, n_kb, unit_bytes(FMT));
        if (FMT == FMT_Q2_K)
          q2k_unit(ub, st, k, kb * kQ2kUnitK, nt, acc[m], c0, c1);
        else
          q80_unit(ub, st, k, kb * kQ80UnitK, nt, acc[m]);
      }
    }
    // reduce the four lanes of each row group, then the warps in a fixed order
#pragma unroll
    for (int m = 0; m < NM; ++m)
#pragma unroll
      for (int tt = 0; tt < kTmax; ++tt)
#pragma unroll
        for (int rho = 0; rho < 2; ++rho) {
          float v = acc[m][tt][rho];
          v += __shfl_xor_sync(0xffffffffu, v, 1);
          v += __shfl_xor_sync(0xffffffffu, v, 2);
          if (t == 0) st.red[((warp * 2 + m) * kTmax + tt) * 16 + g + 8 * rho] = v;
        }
    __syncthreads();
    if (threadIdx.x < 16 * nt) {
      const int tt = threadIdx.x >> 4, r = threadIdx.x & 15;
      float s0 = 0.f, s1 = 0.f;
      for (int w = 0; w < kWarps; ++w) {
        s0 += st.red[((w * 2 + 0) * kTmax + tt) * 16 + r];
        if (GATEUP) s1 += st.red[((w * 2 + 1) * kTmax + tt) * 16 + r];
      }
      const float inv = st.inv[tt];
      const float val = GATEUP ? silu_mul(s0 * inv, s1 * inv) : s0 * inv;
      a.out[(size_t)(pos0 + p0 + tt) * a.rows + rg * 16 + r] = val;
    }
  }
}

size_t gemv_smem(int k) { return (size_t)kTmax * k * 2 + (size_t)kTmax * (k / 16) * 4 + kWarps * 2 * kTmax * 16 * 4 + 64; }

template <int FMT, bool GATEUP>
void launch_gemv(const GemvArgs& a, int max_active, cudaStream_t s) {
  static bool attr_set = false;
  if (!attr_set) {
    cudaFuncSetAttribute(expert_gemv_kernel<FMT, GATEUP>, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
    attr_set = true;
  }
  dim3 grid(a.rows / 16, a.active ? max_active : 1);
  expert_gemv_kernel<FMT, GATEUP><<<grid, kThreads, gemv_smem(a.k), s>>>(a);
}

}  // namespace

void launch_gateup(int fmt, const GemvArgs& a, int max_active, cudaStream_t s) {
  if (fmt == FMT_Q2_K)
    launch_gemv<FMT_Q2_K, true>(a, max_active, s);
  else
    launch_gemv<FMT_Q8_0, true>(a, max_active, s);
}

void launch_down(int fmt, const GemvArgs& a, int max_active, cudaStream_t s) {
  if (fmt == FMT_Q2_K)
    launch_gemv<FMT_Q2_K, false>(a, max_active, s);
  else
    launch_gemv<FMT_Q8_0, false>(a, max_active, s);
}

}  // namespace ds4
