// Warp-level building blocks of the fused dequant GEMV on mma.m16n8k16 (fp16 in, fp32 acc),
// shared by the decode kernels. Layouts of the repacked units are described in common.cuh.
//
// One K chunk is 128 wide: 8 sub-blocks of 16. For MMA i of a chunk, only lanes of group
// g == i pass their activations as B, so accumulator column n holds sub-block n alone. Each lane
// then owns rows (g, g+8) x sub-blocks (2t, 2t+1) of the chunk and applies their scales.
#pragma once

#include "common.cuh"

namespace ds4 {

// B fragment of one token for one chunk, plus the sums of the lane's two accumulator columns.
struct XFrag {
  uint32_t b0, b1;  // fp16x2: k = 16g + 2t (+1) and 16g + 2t + 8 (+9) of the chunk, scaled
  float s0, s1;     // sums over sub-blocks 2t and 2t+1 of the scaled fp16 values
};

__device__ __forceinline__ uint32_t h2_bits(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }

// Sub-block sums through the quad of lanes that hold one sub-block, then moved to the lanes
// whose accumulator columns they belong to.
__device__ __forceinline__ void xfrag_sums(XFrag& f, float p) {
  const int lane = threadIdx.x & 31, t = lane & 3;
  p += __shfl_xor_sync(0xffffffffu, p, 1);
  p += __shfl_xor_sync(0xffffffffu, p, 2);  // every lane of group g holds the sum of sub-block g
  f.s0 = __shfl_sync(0xffffffffu, p, 8 * t);
  f.s1 = __shfl_sync(0xffffffffu, p, 8 * t + 4);
}

// Raw (unconverted) activation words of one lane for one chunk: bf16 pairs at k = 16g + 2t
// and 16g + 2t + 8. Loading them early and converting later keeps the load off the critical path.
__device__ __forceinline__ uint2 xraw_bf16(const __nv_bfloat16* __restrict__ chunk) {
  const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
  return make_uint2(*reinterpret_cast<const uint32_t*>(chunk + 16 * g + 2 * t),
                    *reinterpret_cast<const uint32_t*>(chunk + 16 * g + 2 * t + 8));
}

__device__ __forceinline__ XFrag xfrag_from_bf16(uint2 raw, float sc) {
  const float2 v0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.x));
  const float2 v1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.y));
  const __half2 h0 = __floats2half2_rn(v0.x * sc, v0.y * sc);
  const __half2 h1 = __floats2half2_rn(v1.x * sc, v1.y * sc);
  XFrag f;
  f.b0 = *reinterpret_cast<const uint32_t*>(&h0);
  f.b1 = *reinterpret_cast<const uint32_t*>(&h1);
  const float2 a = __half22float2(h0), b = __half22float2(h1);
  float p = (a.x + a.y) + (b.x + b.y);
  const int t = threadIdx.x & 3;
  p += __shfl_xor_sync(0xffffffffu, p, 1);
  p += __shfl_xor_sync(0xffffffffu, p, 2);
  f.s0 = __shfl_sync(0xffffffffu, p, 8 * t);
  f.s1 = __shfl_sync(0xffffffffu, p, 8 * t + 4);
  return f;
}

// From a bf16 row (chunk base pointer), scaled by sc.
__device__ __forceinline__ XFrag xfrag_bf16(const __nv_bfloat16* __restrict__ chunk, float sc) {
  const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
  const uint32_t r0 = *reinterpret_cast<const uint32_t*>(chunk + 16 * g + 2 * t);
  const uint32_t r1 = *reinterpret_cast<const uint32_t*>(chunk + 16 * g + 2 * t + 8);
  const float2 v0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&r0));
  const float2 v1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&r1));
  const __half2 h0 = __floats2half2_rn(v0.x * sc, v0.y * sc);
  const __half2 h1 = __floats2half2_rn(v1.x * sc, v1.y * sc);
  XFrag f;
  f.b0 = h2_bits(h0);
  f.b1 = h2_bits(h1);
  const float2 a = __half22float2(h0), b = __half22float2(h1);
  xfrag_sums(f, (a.x + a.y) + (b.x + b.y));
  return f;
}

// From an fp32 row (chunk base pointer), scaled by sc.
__device__ __forceinline__ XFrag xfrag_f32(const float* __restrict__ chunk, float sc) {
  const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
  const float2 v0 = *reinterpret_cast<const float2*>(chunk + 16 * g + 2 * t);
  const float2 v1 = *reinterpret_cast<const float2*>(chunk + 16 * g + 2 * t + 8);
  const __half2 h0 = __floats2half2_rn(v0.x * sc, v0.y * sc);
  const __half2 h1 = __floats2half2_rn(v1.x * sc, v1.y * sc);
  XFrag f;
  f.b0 = h2_bits(h0);
  f.b1 = h2_bits(h1);
  const float2 a = __half22float2(h0), b = __half22float2(h1);
  xfrag_sums(f, (a.x + a.y) + (b.x + b.y));
  return f;
}

// Lane selectors for the B operand, as fp16x2 multipliers: 1.0 in MMA i for the lanes of group
// g == i, 0 otherwise. The selection is an fp16 multiply (FMA pipe) rather than an AND: the integer
// pipe already carries the quant field extraction. (x * 1.0 is x exactly; x * 0 is a signed zero.)
#ifndef DS4_BSEL_AND
#define DS4_BSEL_AND 0
#endif
struct BMask {
  uint32_t m[8];
  __device__ __forceinline__ BMask() {
    const int g = (threadIdx.x & 31) >> 2;
#pragma unroll
    for (int i = 0; i < 8; ++i) m[i] = (g == i) ? (DS4_BSEL_AND ? 0xffffffffu : 0x3C003C00u) : 0u;
  }
};

__device__ __forceinline__ uint32_t bsel(uint32_t b, uint32_t sel) {
#if DS4_BSEL_AND
  return b & sel;
#else
  uint32_t r;
  asm("mul.rn.f16x2 %0, %1, %2;\n" : "=r"(r) : "r"(b), "r"(sel));
  return r;
#endif
}

// Exact small-integer extraction through an fp32 with exponent 2^23: (bits | 0x4B000000) is
// 2^23 + field * 2^pos, and fmaf(v, c, -2^23 c) gives field * 2^pos * c exactly.
__device__ __forceinline__ float magic_field(uint32_t masked_bits, float c, float neg_magic_c) {
  return fmaf(__uint_as_float(masked_bits | 0x4B000000u), c, neg_magic_c);
}

// Q2_K: 2^(24 - p) where p is the bit position of sub-block n's quant in the A registers.
__device__ __forceinline__ float q2k_col_scale(int n) {
  const int p = n < 5 ? 2 * n : 2 * (n - 5);
  return ldexpf(1.f, 24 - p);
}

// Per-lane constants of a Q2_K chunk: scale of columns 2t, 2t+1 (with the 2^(24-p) factor
// folded in) for rows g, g+8, and the mins.
struct Q2kLaneConst {
  float c0, c1, nc0, nc1;  // c0 = col scale of column 2t, c1 = of 2t+1 divided by 256; nc = -2^23 c
  __device__ __forceinline__ Q2kLaneConst() {
    const int t = threadIdx.x & 3;
    c0 = q2k_col_scale(2 * t);
    c1 = q2k_col_scale(2 * t + 1) * (1.f / 256.f);
    nc0 = -8388608.f * c0;
    nc1 = -8388608.f * c1;
  }
};

struct Q2kChunkScales {
  float s00, s01, s10, s11;  // [row rho][column n]
  float m00, m01, m10, m11;
};

__device__ __forceinline__ Q2kChunkScales q2k_chunk_scales(uint32_t sc, const Q2kLaneConst& k) {
  const uint32_t sh = sc >> 16;
  Q2kChunkScales r;
  r.s00 = magic_field(sc & 0xFu, k.c0, k.nc0);
  r.s01 = magic_field(sc & 0xF00u, k.c1, k.nc1);
  r.s10 = magic_field(sh & 0xFu, k.c0, k.nc0);
  r.s11 = magic_field(sh & 0xF00u, k.c1, k.nc1);
  r.m00 = magic_field(sc & 0xF0u, 1.f / 16.f, -8388608.f / 16.f);
  r.m01 = magic_field(sc & 0xF000u, 1.f / 4096.f, -8388608.f / 4096.f);
  r.m10 = magic_field(sh & 0xF0u, 1.f / 16.f, -8388608.f / 16.f);
  r.m11 = magic_field(sh & 0xF000u, 1.f / 4096.f, -8388608.f / 4096.f);
  return r;
}

// A registers of MMA i (sub-block i of the chunk) from the lane's four quant words.
template <int I>
__device__ __forceinline__ void q2k_a(const uint32_t (&w)[4], const uint32_t (&wh)[4], uint32_t (&a)[4]) {
  constexpr uint32_t mask = 0x00030003u << (2 * (I < 5 ? I : I - 5));
#pragma unroll
  for (int r = 0; r < 4; ++r) a[r] = (I < 5 ? w[r] : wh[r]) & mask;
}

// Eight MMAs of one Q2_K chunk for one token: returns the 4 accumulator values (rows g, g+8 x
// columns 2t, 2t+1), each the dot product of a sub-block times 2^(p-24).
__device__ __forceinline__ void q2k_chunk_mma(const uint32_t (&w)[4], const uint32_t (&wh)[4], const BMask& bm,
                                              const XFrag& x, float (&d)[4]) {
  float e[4] = {0.f, 0.f, 0.f, 0.f};  // second accumulator: two shorter dependency chains
  d[0] = d[1] = d[2] = d[3] = 0.f;
  uint32_t a[4];
  q2k_a<0>(w, wh, a); mma_f16_16816(d, a, bsel(x.b0, bm.m[0]), bsel(x.b1, bm.m[0]));
  q2k_a<1>(w, wh, a); mma_f16_16816(e, a, bsel(x.b0, bm.m[1]), bsel(x.b1, bm.m[1]));
  q2k_a<2>(w, wh, a); mma_f16_16816(d, a, bsel(x.b0, bm.m[2]), bsel(x.b1, bm.m[2]));
  q2k_a<3>(w, wh, a); mma_f16_16816(e, a, bsel(x.b0, bm.m[3]), bsel(x.b1, bm.m[3]));
  q2k_a<4>(w, wh, a); mma_f16_16816(d, a, bsel(x.b0, bm.m[4]), bsel(x.b1, bm.m[4]));
  q2k_a<5>(w, wh, a); mma_f16_16816(e, a, bsel(x.b0, bm.m[5]), bsel(x.b1, bm.m[5]));
  q2k_a<6>(w, wh, a); mma_f16_16816(d, a, bsel(x.b0, bm.m[6]), bsel(x.b1, bm.m[6]));
  q2k_a<7>(w, wh, a); mma_f16_16816(e, a, bsel(x.b0, bm.m[7]), bsel(x.b1, bm.m[7]));
  // columns are disjoint between the two accumulators' contributions except for zeros
  d[0] += e[0]; d[1] += e[1]; d[2] += e[2]; d[3] += e[3];
}

// Q8_0: eight MMAs of one chunk (16 rows x 128 k) for one token.
__device__ __forceinline__ void q80_chunk_mma(const uint4 (&v)[4], const BMask& bm, const XFrag& x, float (&d)[4]) {
  float e[4] = {0.f, 0.f, 0.f, 0.f};
  d[0] = d[1] = d[2] = d[3] = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int j = i >> 1;
    const uint32_t wg = (i & 1) ? v[j].y : v[j].x;   // row g of sub-block i: k 2t, 2t+1, 2t+8, 2t+9
    const uint32_t wg8 = (i & 1) ? v[j].w : v[j].z;  // row g + 8
    const uint32_t a[4] = {prmt(wg, 0u, 0x4140u), prmt(wg8, 0u, 0x4140u), prmt(wg, 0u, 0x4342u),
                           prmt(wg8, 0u, 0x4342u)};
    if (i & 1)
      mma_f16_16816(e, a, bsel(x.b0, bm.m[i]), bsel(x.b1, bm.m[i]));
    else
      mma_f16_16816(d, a, bsel(x.b0, bm.m[i]), bsel(x.b1, bm.m[i]));
  }
  d[0] += e[0]; d[1] += e[1]; d[2] += e[2]; d[3] += e[3];
}

// Loaded bytes of one Q2_K unit (16 rows x 256 k) for the calling lane.
struct Q2kUnitRegs {
  uint4 q[2];
  uint32_t sc[2];
  uint32_t dd0, dd1;
};

__device__ __forceinline__ Q2kUnitRegs q2k_load(const uint8_t* __restrict__ ub) {
  const int lane = threadIdx.x & 31, g = lane >> 2;
  const int off = 16 * lane_region(g, lane & 3);
  const uint4 q0 = ldg_nc_v4(ub + off), q1 = ldg_nc_v4(ub + 512 + off);
  Q2kUnitRegs r;
  r.q[0] = make_uint4(q0.x, q0.z, q0.y, q0.w);  // the region's words in A register order
  r.q[1] = make_uint4(q1.x, q1.z, q1.y, q1.w);
  r.sc[0] = ldg_nc_u32(ub + kQ2kScOff + 4 * lane);
  r.sc[1] = ldg_nc_u32(ub + kQ2kScOff + 128 + 4 * lane);
  r.dd0 = ldg_nc_u32(ub + kQ2kDdOff + 4 * g);
  r.dd1 = ldg_nc_u32(ub + kQ2kDdOff + 4 * (g + 8));
  return r;
}

struct Q80UnitRegs {
  uint4 v[4];
  uint32_t sc;
};

__device__ __forceinline__ Q80UnitRegs q80_load(const uint8_t* __restrict__ ub) {
  const int lane = threadIdx.x & 31;
  const int off = 16 * lane_region(lane >> 2, lane & 3);
  Q80UnitRegs r;
#pragma unroll
  for (int j = 0; j < 4; ++j) r.v[j] = ldg_nc_v4(ub + 512 * j + off);
  r.sc = ldg_nc_u32(ub + kQ80ScOff + 4 * lane);
  return r;
}

// Warp-wide L2 prefetch of a byte range (one request per 128-byte line).
__device__ __forceinline__ void prefetch_l2(const uint8_t* p, int bytes) {
  const int lane = threadIdx.x & 31;
  for (int off = lane * 128; off < bytes; off += 32 * 128)
    asm volatile("prefetch.global.L2 [%0];\n" ::"l"(p + off));
}

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;\n" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory"); }

}  // namespace ds4
