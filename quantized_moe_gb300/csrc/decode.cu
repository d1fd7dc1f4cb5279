// Decode path (1..16 tokens): three kernels chained with programmatic dependent launch.
//
//  route_decode_kernel    one CTA per routed expert computes its fp32 logits for every token;
//                         the last CTA to finish (atomic arrival counter, no waiting) runs the
//                         sigmoid top-k (or table routing), the bucketing and the bookkeeping.
//                         CTA 0 also records max|x| per token for the fp16 activation scale.
//  gateup_decode_kernel   CTA = 16 rows of f of one active expert (or of the shared expert),
//                         K split over 8 warps; h = silu(g) * u written in fp32, and max|h| per
//                         row of H reduced with an integer atomicMax (order-free).
//  down_decode_kernel     CTA = 16 rows of d for ALL touched experts and the shared expert; the
//                         per-slot results stay in shared memory and the CTA writes the final
//                         out rows: routed terms in ascending expert id, then the shared expert.
//
// Before waiting on its predecessor, each dependent kernel streams the weights that do not
// depend on the routing (and, for the down kernel, the routed weights, whose routing is final
// by then) into L2, so weight reads overlap the previous kernel.
#include "mma_units.cuh"

namespace ds4 {
namespace {

constexpr int kWarps = 8;
constexpr int kThreads = 256;
constexpr int kMaxTok = 16;  // decode path limit

// ----------------------------------------------------------------------------- route

__global__ void __launch_bounds__(kThreads) route_decode_kernel(DecodeArgs a) {
  __shared__ float part[kWarps][kMaxTok];
  __shared__ float xmx[kWarps][kMaxTok];
  __shared__ int s_last;
  __shared__ int s_idx[kMaxTok * 16];
  __shared__ int s_cnt[256], s_off[257], s_act[256], s_nact;
  const int e = blockIdx.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int d = a.d, nt = a.n_tok;
  // ---- logits of expert e for the learned tokens (and max|x| of every token in CTA 0)
  const int per_warp = d / kWarps;
  const float* wr = a.wr + (size_t)e * d;
  float acc[kMaxTok], mx[kMaxTok];
#pragma unroll
  for (int t = 0; t < kMaxTok; ++t) acc[t] = mx[t] = 0.f;
  for (int k0 = warp * per_warp + lane * 4; k0 < (warp + 1) * per_warp; k0 += 128) {
    const float4 wv = *reinterpret_cast<const float4*>(wr + k0);
#pragma unroll
    for (int t = 0; t < kMaxTok; ++t) {
      if (t >= nt) break;
      const uint2 xv = *reinterpret_cast<const uint2*>(a.x + (size_t)t * d + k0);
      const float2 x01 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&xv.x));
      const float2 x23 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&xv.y));
      acc[t] = fmaf(wv.x, x01.x, acc[t]);
      acc[t] = fmaf(wv.y, x01.y, acc[t]);
      acc[t] = fmaf(wv.z, x23.x, acc[t]);
      acc[t] = fmaf(wv.w, x23.y, acc[t]);
      mx[t] = fmaxf(mx[t], fmaxf(fmaxf(fabsf(x01.x), fabsf(x01.y)), fmaxf(fabsf(x23.x), fabsf(x23.y))));
    }
  }
#pragma unroll
  for (int t = 0; t < kMaxTok; ++t) {
    if (t >= nt) break;
    const float s = warp_sum(acc[t]);
    const float m = warp_max(mx[t]);
    if (lane == 0) { part[warp][t] = s; xmx[warp][t] = m; }
  }
  __syncthreads();
  if (threadIdx.x < nt) {
    const int t = threadIdx.x;
    if (t >= a.n_hash) {
      float s = 0.f;
      for (int w = 0; w < kWarps; ++w) s += part[w][t];
      a.logits[(size_t)(t - a.n_hash) * a.n_exp + e] = s + (a.br ? a.br[e] : 0.f);
    }
    if (e == 0) {
      float m = 0.f;
      for (int w = 0; w < kWarps; ++w) m = fmaxf(m, xmx[w][t]);
      a.xmax[t] = m;
    }
  }
  // ---- arrival: the last CTA continues with the top-k and the bucketing
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) s_last = atomicAdd(a.counter, 1u) == gridDim.x - 1;
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  const int K = a.top_k, E = a.n_exp, n_slots = nt * K;
  for (int t = warp; t < nt; t += kWarps) {
    if (t < a.n_hash) {
      const int id = a.token_ids[t];
      const bool ok = id >= 0 && id < a.vocab;
      if (!ok && lane == 0) atomicOr(a.err, 1);
      if (lane < K) {
        const int ex = ok ? a.table[(size_t)id * K + lane] : 0;
        a.idx[t * K + lane] = ex;
        a.wts[t * K + lane] = ok ? 1.f / (float)K : 0.f;
        s_idx[t * K + lane] = ex;
      }
      continue;
    }
    const float* z = a.logits + (size_t)(t - a.n_hash) * E;
    float s[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int ex = lane + 32 * i;
      s[i] = ex < E ? 1.f / (1.f + expf(-__ldcg(z + ex))) : -1.f;
    }
    float sel_sum = 0.f, my_w = 0.f;
    int my_e = 0;
    for (int j = 0; j < K; ++j) {
      float bv = s[0];
      int bi = lane;
#pragma unroll
      for (int i = 1; i < 8; ++i)
        if (s[i] > bv) { bv = s[i]; bi = lane + 32 * i; }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
        if (ov > bv || (ov == bv && oi < bi)) { bv = ov; bi = oi; }
      }
      if ((bi & 31) == lane) s[bi >> 5] = -2.f;
      sel_sum += bv;
      if (lane == j) { my_w = bv; my_e = bi; }
    }
    if (lane < K) {
      a.idx[t * K + lane] = my_e;
      a.wts[t * K + lane] = my_w / sel_sum;
      s_idx[t * K + lane] = my_e;
    }
  }
  for (int i = threadIdx.x; i < E; i += kThreads) s_cnt[i] = 0;
  __syncthreads();
  for (int sl = threadIdx.x; sl < n_slots; sl += kThreads) atomicAdd(&s_cnt[s_idx[sl]], 1);  // integer counts
  __syncthreads();
  if (warp == 0) {  // exclusive scans of the counts and of the active flags (E <= 256: 8 per lane)
    int c[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) c[i] = (lane * 8 + i < E) ? s_cnt[lane * 8 + i] : 0;
    int tot = 0, tota = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) { tot += c[i]; tota += c[i] > 0; }
    int inc = tot, inca = tota;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, inc, o), va = __shfl_up_sync(0xffffffffu, inca, o);
      if (lane >= o) { inc += v; inca += va; }
    }
    int run = inc - tot, runa = inca - tota;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int ex = lane * 8 + i;
      if (ex < E) {
        s_off[ex] = run;
        if (c[i] > 0) s_act[runa++] = ex;
        run += c[i];
      }
    }
    if (lane == 31) { s_off[E] = inc; s_nact = inca; }
  }
  __syncthreads();
  for (int i = threadIdx.x; i < E; i += kThreads) {
    a.counts[i] = s_cnt[i];
    a.offsets[i] = s_off[i];
    if (i < s_nact) a.active[i] = s_act[i];
  }
  if (threadIdx.x == 0) {
    a.offsets[E] = s_off[E];
    *a.n_active = s_nact;
  }
  for (int sl = threadIdx.x; sl < n_slots; sl += kThreads) {  // stable rank among equal experts
    const int ex = s_idx[sl];
    int r = 0;
    for (int j = 0; j < sl; ++j) r += s_idx[j] == ex;
    const int pos = s_off[ex] + r;
    a.perm[pos] = sl;
    a.rowof[sl] = pos;
  }
  for (int i = threadIdx.x; i < n_slots + nt; i += kThreads) a.hmax[i] = 0.f;
  if (threadIdx.x == 0) *a.counter = 0u;  // every CTA has arrived: ready for the next forward
}

// ----------------------------------------------------------------------------- gate/up

// kPass: token rows per pass through the weights (1 for a single token, else 4)
template <int FMT_R, int FMT_S, int kPass>
__global__ void __launch_bounds__(kThreads) gateup_decode_kernel(DecodeArgs a, int max_active) {
  __shared__ float red[kWarps][2][kPass][16];
  const int rg = blockIdx.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
  const bool shared = (int)blockIdx.y == max_active;
  const int d = a.d;
  const int rows = shared ? a.fs : a.f;
  if (rg * 16 >= rows) {
    pdl_wait();
    return;
  }
  const int fmt = shared ? FMT_S : FMT_R;
  const int n_kb = d / unit_k(fmt);
  const int ub = unit_bytes(fmt);
  const uint8_t* w0 = shared ? a.sgate : a.gate;
  const uint8_t* w1 = shared ? a.sup : a.up;
  const size_t mb = shared ? a.mb_sgu : a.mb_gu;
  if (shared) {  // routing-independent weights: start their reads before the router finishes
    for (int kb = warp; kb < n_kb; kb += kWarps) {
      prefetch_l2(w0 + unit_offset(rg, kb, n_kb, ub), ub);
      prefetch_l2(w1 + unit_offset(rg, kb, n_kb, ub), ub);
    }
  }
  pdl_wait();
  pdl_trigger();
  int pos0 = 0, cnt = a.n_tok;
  if (!shared) {
    if ((int)blockIdx.y >= *a.n_active) return;
    const int e = a.active[blockIdx.y];
    pos0 = a.offsets[e];
    cnt = a.offsets[e + 1] - pos0;
    w0 += (size_t)e * mb;
    w1 += (size_t)e * mb;
  }
  const BMask bm;
  const Q2kLaneConst qc;
  for (int p0 = 0; p0 < cnt; p0 += kPass) {
    const int np = min(kPass, cnt - p0);
    const __nv_bfloat16* xrow[kPass];
    float sc[kPass];
#pragma unroll
    for (int tt = 0; tt < kPass; ++tt) {
      const int pos = pos0 + p0 + min(tt, np - 1);
      const int tok = shared ? pos : a.perm[pos] / a.top_k;
      xrow[tt] = a.x + (size_t)tok * d;
      sc[tt] = fp16_row_scale(a.xmax[tok]);
    }
    float acc[2][kPass][2];
#pragma unroll
    for (int m = 0; m < 2; ++m)
#pragma unroll
      for (int tt = 0; tt < kPass; ++tt) acc[m][tt][0] = acc[m][tt][1] = 0.f;
    for (int kb = warp; kb < n_kb; kb += kWarps) {
      if (fmt == FMT_Q2_K) {
        const Q2kUnitRegs u0 = q2k_load(w0 + unit_offset(rg, kb, n_kb, kQ2kUnitBytes));
        const Q2kUnitRegs u1 = q2k_load(w1 + unit_offset(rg, kb, n_kb, kQ2kUnitBytes));
        float as[2][kPass][2], am[2][kPass][2];
#pragma unroll
        for (int m = 0; m < 2; ++m)
#pragma unroll
          for (int tt = 0; tt < kPass; ++tt) as[m][tt][0] = as[m][tt][1] = am[m][tt][0] = am[m][tt][1] = 0.f;
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const int kc = kb * 256 + 128 * c;
          XFrag xf[kPass];
#pragma unroll
          for (int tt = 0; tt < kPass; ++tt)
            if (tt < np) xf[tt] = xfrag_bf16(xrow[tt] + kc, sc[tt]);
#pragma unroll
          for (int m = 0; m < 2; ++m) {
            const Q2kUnitRegs& u = m ? u1 : u0;
            const uint32_t w[4] = {u.q[c].x, u.q[c].y, u.q[c].z, u.q[c].w};
            const uint32_t wh[4] = {w[0] >> 10, w[1] >> 10, w[2] >> 10, w[3] >> 10};
            const Q2kChunkScales s = q2k_chunk_scales(u.sc[c], qc);
#pragma unroll
            for (int tt = 0; tt < kPass; ++tt) {
              if (tt >= np) break;
              float dd[4];
              q2k_chunk_mma(w, wh, bm, xf[tt], dd);
              as[m][tt][0] = fmaf(s.s00, dd[0], fmaf(s.s01, dd[1], as[m][tt][0]));
              as[m][tt][1] = fmaf(s.s10, dd[2], fmaf(s.s11, dd[3], as[m][tt][1]));
              am[m][tt][0] = fmaf(s.m00, xf[tt].s0, fmaf(s.m01, xf[tt].s1, am[m][tt][0]));
              am[m][tt][1] = fmaf(s.m10, xf[tt].s0, fmaf(s.m11, xf[tt].s1, am[m][tt][1]));
            }
          }
        }
#pragma unroll
        for (int m = 0; m < 2; ++m) {
          const Q2kUnitRegs& u = m ? u1 : u0;
          const float2 d0 = __half22float2(*reinterpret_cast<const __half2*>(&u.dd0));
          const float2 d1 = __half22float2(*reinterpret_cast<const __half2*>(&u.dd1));
#pragma unroll
          for (int tt = 0; tt < kPass; ++tt) {
            if (tt >= np) break;
            acc[m][tt][0] = fmaf(d0.x, as[m][tt][0], fmaf(-d0.y, am[m][tt][0], acc[m][tt][0]));
            acc[m][tt][1] = fmaf(d1.x, as[m][tt][1], fmaf(-d1.y, am[m][tt][1], acc[m][tt][1]));
          }
        }
      } else {
        const Q80UnitRegs u0 = q80_load(w0 + unit_offset(rg, kb, n_kb, kQ80UnitBytes));
        const Q80UnitRegs u1 = q80_load(w1 + unit_offset(rg, kb, n_kb, kQ80UnitBytes));
        const int kc = kb * 128;
        XFrag xf[kPass];
#pragma unroll
        for (int tt = 0; tt < kPass; ++tt)
          if (tt < np) xf[tt] = xfrag_bf16(xrow[tt] + kc, sc[tt]);
#pragma unroll
        for (int m = 0; m < 2; ++m) {
          const Q80UnitRegs& u = m ? u1 : u0;
          const float2 s = __half22float2(*reinterpret_cast<const __half2*>(&u.sc));
#pragma unroll
          for (int tt = 0; tt < kPass; ++tt) {
            if (tt >= np) break;
            float dd[4];
            q80_chunk_mma(u.v, bm, xf[tt], dd);
            const float off = 128.f * (xf[tt].s0 + xf[tt].s1);
            acc[m][tt][0] = fmaf(s.x, fmaf(16777216.f, dd[0] + dd[1], -off), acc[m][tt][0]);
            acc[m][tt][1] = fmaf(s.y, fmaf(16777216.f, dd[2] + dd[3], -off), acc[m][tt][1]);
          }
        }
      }
    }
    // reduce the quad, then the warps in a fixed order
#pragma unroll
    for (int m = 0; m < 2; ++m)
#pragma unroll
      for (int tt = 0; tt < kPass; ++tt)
#pragma unroll
        for (int rho = 0; rho < 2; ++rho) {
          float v = acc[m][tt][rho];
          v += __shfl_xor_sync(0xffffffffu, v, 1);
          v += __shfl_xor_sync(0xffffffffu, v, 2);
          if (t == 0) red[warp][m][tt][g + 8 * rho] = v;
        }
    __syncthreads();
    // whole warps take part (the 16-lane shuffles below name all 32 lanes): warp 0 for one
    // token per pass, warps 0 and 1 for four
    if (threadIdx.x < (kPass == 1 ? 32 : 16 * kPass)) {
      const int tt = min(threadIdx.x >> 4, kPass - 1), r = threadIdx.x & 15;
      const bool valid = (int)(threadIdx.x >> 4) < np;
      float s0 = 0.f, s1 = 0.f;
      for (int w = 0; w < kWarps; ++w) {
        s0 += red[w][0][tt][r];
        s1 += red[w][1][tt][r];
      }
      const float inv = 1.f / sc[tt];
      const float h = valid ? silu_mul(s0 * inv, s1 * inv) : 0.f;
      const int pos = pos0 + p0 + tt;
      if (valid) {
        float* hrow = shared ? a.Hs + (size_t)pos * a.fs : a.H + (size_t)pos * a.f;
        hrow[rg * 16 + r] = h;
      }
      float m = fabsf(h);  // max over the 16 rows of this CTA (16 consecutive lanes)
#pragma unroll
      for (int o = 8; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o, 16));
      if (valid && r == 0) {
        unsigned* hm = reinterpret_cast<unsigned*>(a.hmax + (shared ? a.n_tok * a.top_k + pos : pos));
        atomicMax(hm, __float_as_uint(m));  // non-negative floats order like their bit patterns
      }
    }
    __syncthreads();
  }
}

// ----------------------------------------------------------------------------- down + combine

template <int FMT_R, int FMT_S, int kPass>
__global__ void __launch_bounds__(kThreads) down_decode_kernel(DecodeArgs a, int max_active) {
  __shared__ float ys[kMaxTok * 16][16];     // per bucketed slot position
  __shared__ float ysh[kWarps][kMaxTok][16];  // shared expert partials per warp
  const int rg = blockIdx.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
  const int nt = a.n_tok, K = a.top_k;
  const int n_kb_r = a.f / unit_k(FMT_R), ub_r = unit_bytes(FMT_R);
  const int n_kb_s = a.n_shared ? a.fs / unit_k(FMT_S) : 0, ub_s = unit_bytes(FMT_S);
  // routing is final (its kernel completed before the gate/up kernel passed its wait): stream
  // this CTA's rows of every touched expert, and of the shared expert, into L2 now
  {
    const int n_act = *a.n_active;
    for (int item = warp; item < n_act * n_kb_r; item += kWarps) {
      const int e = a.active[item / n_kb_r], kb = item % n_kb_r;
      prefetch_l2(a.down + (size_t)e * a.mb_d + unit_offset(rg, kb, n_kb_r, ub_r), ub_r);
    }
    for (int kb = warp; kb < n_kb_s; kb += kWarps) prefetch_l2(a.sdown + unit_offset(rg, kb, n_kb_s, ub_s), ub_s);
  }
  pdl_wait();
  const int n_act = *a.n_active;
  const BMask bm;
  const Q2kLaneConst qc;
  // routed: warp w takes the touched experts w, w+8, ... over the full K
  for (int ai = warp; ai < n_act; ai += kWarps) {
    const int e = a.active[ai];
    const int pos0 = a.offsets[e], cnt = a.offsets[e + 1] - pos0;
    const uint8_t* wd = a.down + (size_t)e * a.mb_d;
    for (int p0 = 0; p0 < cnt; p0 += kPass) {
      const int np = min(kPass, cnt - p0);
      const float* hrow[kPass];
      float sc[kPass];
#pragma unroll
      for (int tt = 0; tt < kPass; ++tt) {
        const int pos = pos0 + p0 + min(tt, np - 1);
        hrow[tt] = a.H + (size_t)pos * a.f;
        sc[tt] = fp16_row_scale(__ldcg(a.hmax + pos));
      }
      float acc[kPass][2];
#pragma unroll
      for (int tt = 0; tt < kPass; ++tt) acc[tt][0] = acc[tt][1] = 0.f;
      for (int kb = 0; kb < n_kb_r; ++kb) {
        if (FMT_R == FMT_Q2_K) {
          const Q2kUnitRegs u = q2k_load(wd + unit_offset(rg, kb, n_kb_r, kQ2kUnitBytes));
          float as[kPass][2], am[kPass][2];
#pragma unroll
          for (int tt = 0; tt < kPass; ++tt) as[tt][0] = as[tt][1] = am[tt][0] = am[tt][1] = 0.f;
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            const int kc = kb * 256 + 128 * c;
            const uint32_t w[4] = {u.q[c].x, u.q[c].y, u.q[c].z, u.q[c].w};
            const uint32_t wh[4] = {w[0] >> 10, w[1] >> 10, w[2] >> 10, w[3] >> 10};
            const Q2kChunkScales s = q2k_chunk_scales(u.sc[c], qc);
#pragma unroll
            for (int tt = 0; tt < kPass; ++tt) {
              if (tt >= np) break;
              const XFrag xf = xfrag_f32(hrow[tt] + kc, sc[tt]);
              float dd[4];
              q2k_chunk_mma(w, wh, bm, xf, dd);
              as[tt][0] = fmaf(s.s00, dd[0], fmaf(s.s01, dd[1], as[tt][0]));
              as[tt][1] = fmaf(s.s10, dd[2], fmaf(s.s11, dd[3], as[tt][1]));
              am[tt][0] = fmaf(s.m00, xf.s0, fmaf(s.m01, xf.s1, am[tt][0]));
              am[tt][1] = fmaf(s.m10, xf.s0, fmaf(s.m11, xf.s1, am[tt][1]));
            }
          }
          const float2 d0 = __half22float2(*reinterpret_cast<const __half2*>(&u.dd0));
          const float2 d1 = __half22float2(*reinterpret_cast<const __half2*>(&u.dd1));
#pragma unroll
          for (int tt = 0; tt < kPass; ++tt) {
            if (tt >= np) break;
            acc[tt][0] = fmaf(d0.x, as[tt][0], fmaf(-d0.y, am[tt][0], acc[tt][0]));
            acc[tt][1] = fmaf(d1.x, as[tt][1], fmaf(-d1.y, am[tt][1], acc[tt][1]));
          }
        } else {
          const Q80UnitRegs u = q80_load(wd + unit_offset(rg, kb, n_kb_r, kQ80UnitBytes));
          const float2 s = __half22float2(*reinterpret_cast<const __half2*>(&u.sc));
#pragma unroll
          for (int tt = 0; tt < kPass; ++tt) {
            if (tt >= np) break;
            const XFrag xf = xfrag_f32(hrow[tt] + kb * 128, sc[tt]);
            float dd[4];
            q80_chunk_mma(u.v, bm, xf, dd);
            const float off = 128.f * (xf.s0 + xf.s1);
            acc[tt][0] = fmaf(s.x, fmaf(16777216.f, dd[0] + dd[1], -off), acc[tt][0]);
            acc[tt][1] = fmaf(s.y, fmaf(16777216.f, dd[2] + dd[3], -off), acc[tt][1]);
          }
        }
      }
#pragma unroll
      for (int tt = 0; tt < kPass; ++tt) {
        if (tt >= np) break;
#pragma unroll
        for (int rho = 0; rho < 2; ++rho) {
          float v = acc[tt][rho];
          v += __shfl_xor_sync(0xffffffffu, v, 1);
          v += __shfl_xor_sync(0xffffffffu, v, 2);
          if (t == 0) ys[pos0 + p0 + tt][g + 8 * rho] = v / sc[tt];
        }
      }
    }
  }
  // shared expert: every warp takes a slice of K for all tokens
  if (a.n_shared) {
    for (int p0 = 0; p0 < nt; p0 += kPass) {
      const int np = min(kPass, nt - p0);
      const float* hrow[kPass];
      float sc[kPass];
#pragma unroll
      for (int tt = 0; tt < kPass; ++tt) {
        const int tok = p0 + min(tt, np - 1);
        hrow[tt] = a.Hs + (size_t)tok * a.fs;
        sc[tt] = fp16_row_scale(__ldcg(a.hmax + nt * K + tok));
      }
      float acc[kPass][2];
#pragma unroll
      for (int tt = 0; tt < kPass; ++tt) acc[tt][0] = acc[tt][1] = 0.f;
      for (int kb = warp; kb < n_kb_s; kb += kWarps) {
        if (FMT_S == FMT_Q2_K) {
          const Q2kUnitRegs u = q2k_load(a.sdown + unit_offset(rg, kb, n_kb_s, kQ2kUnitBytes));
          float as[kPass][2], am[kPass][2];
#pragma unroll
          for (int tt = 0; tt < kPass; ++tt) as[tt][0] = as[tt][1] = am[tt][0] = am[tt][1] = 0.f;
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            const int kc = kb * 256 + 128 * c;
            const uint32_t w[4] = {u.q[c].x, u.q[c].y, u.q[c].z, u.q[c].w};
            const uint32_t wh[4] = {w[0] >> 10, w[1] >> 10, w[2] >> 10, w[3] >> 10};
            const Q2kChunkScales s = q2k_chunk_scales(u.sc[c], qc);
#pragma unroll
            for (int tt = 0; tt < kPass; ++tt) {
              if (tt >= np) break;
              const XFrag xf = xfrag_f32(hrow[tt] + kc, sc[tt]);
              float dd[4];
              q2k_chunk_mma(w, wh, bm, xf, dd);
              as[tt][0] = fmaf(s.s00, dd[0], fmaf(s.s01, dd[1], as[tt][0]));
              as[tt][1] = fmaf(s.s10, dd[2], fmaf(s.s11, dd[3], as[tt][1]));
              am[tt][0] = fmaf(s.m00, xf.s0, fmaf(s.m01, xf.s1, am[tt][0]));
              am[tt][1] = fmaf(s.m10, xf.s0, fmaf(s.m11, xf.s1, am[tt][1]));
            }
          }
          const float2 d0 = __half22float2(*reinterpret_cast<const __half2*>(&u.dd0));
          const float2 d1 = __half22float2(*reinterpret_cast<const __half2*>(&u.dd1));
#pragma unroll
          for (int tt = 0; tt < kPass; ++tt) {
            if (tt >= np) break;
            acc[tt][0] = fmaf(d0.x, as[tt][0], fmaf(-d0.y, am[tt][0], acc[tt][0]));
            acc[tt][1] = fmaf(d1.x, as[tt][1], fmaf(-d1.y, am[tt][1], acc[tt][1]));
          }
        } else {
          const Q80UnitRegs u = q80_load(a.sdown + unit_offset(rg, kb, n_kb_s, kQ80UnitBytes));
          const float2 s = __half22float2(*reinterpret_cast<const __half2*>(&u.sc));
#pragma unroll
          for (int tt = 0; tt < kPass; ++tt) {
            if (tt >= np) break;
            const XFrag xf = xfrag_f32(hrow[tt] + kb * 128, sc[tt]);
            float dd[4];
            q80_chunk_mma(u.v, bm, xf, dd);
            const float off = 128.f * (xf.s0 + xf.s1);
            acc[tt][0] = fmaf(s.x, fmaf(16777216.f, dd[0] + dd[1], -off), acc[tt][0]);
            acc[tt][1] = fmaf(s.y, fmaf(16777216.f, dd[2] + dd[3], -off), acc[tt][1]);
          }
        }
      }
#pragma unroll
      for (int tt = 0; tt < kPass; ++tt) {
        if (tt >= np) break;
#pragma unroll
        for (int rho = 0; rho < 2; ++rho) {
          float v = acc[tt][rho];
          v += __shfl_xor_sync(0xffffffffu, v, 1);
          v += __shfl_xor_sync(0xffffffffu, v, 2);
          if (t == 0) ysh[warp][p0 + tt][g + 8 * rho] = v / sc[tt];
        }
      }
    }
  }
  __syncthreads();
  // combine: out[t][r] = sum over the token's slots in ascending expert id, then the shared expert
  if (threadIdx.x < nt * 16) {
    const int tok = threadIdx.x >> 4, r = threadIdx.x & 15;
    int ex[16], ps[16];
    float wv[16];
    for (int j = 0; j < K; ++j) {
      const int ej = a.idx[tok * K + j];
      const float wj = a.wts[tok * K + j];
      const int pj = a.rowof[tok * K + j];
      int i = j;
      while (i > 0 && ex[i - 1] > ej) { ex[i] = ex[i - 1]; wv[i] = wv[i - 1]; ps[i] = ps[i - 1]; --i; }
      ex[i] = ej; wv[i] = wj; ps[i] = pj;
    }
    float o = 0.f;
    for (int j = 0; j < K; ++j) o = fmaf(wv[j], ys[ps[j]][r], o);
    if (a.n_shared) {
      float s = 0.f;
      for (int w = 0; w < kWarps; ++w)
        if (w < n_kb_s) s += ysh[w][tok][r];
      o += s;
    }
    a.out[(size_t)tok * a.d + rg * 16 + r] = o;
  }
}

template <typename Kern>
cudaError_t launch_pdl(Kern kernel, dim3 grid, cudaStream_t s, bool pdl, const DecodeArgs& a, int max_active) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, a, max_active);
}

}  // namespace

int decode_max_tokens() { return kMaxTok; }

cudaError_t launch_decode(const DecodeArgs& a, int fmt_r_gu, int fmt_r_d, int fmt_s, bool pdl, cudaStream_t s,
                          int* launches, const DecodeHooks* hooks) {
  const int max_active = min(a.n_exp, a.n_tok * a.top_k);
  route_decode_kernel<<<a.n_exp, kThreads, 0, s>>>(a);
  if (hooks) hooks->mark(hooks->ctx, "route");
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const dim3 g_gu((max(a.f, a.n_shared ? a.fs : 0)) / 16, max_active + (a.n_shared ? 1 : 0));
  const int fsg = a.n_shared ? fmt_s : fmt_r_gu;
  const bool one = a.n_tok == 1;
#define DS4_GU(R, S)                                                                          \
  e = one ? launch_pdl(gateup_decode_kernel<R, S, 1>, g_gu, s, pdl, a, max_active)            \
          : launch_pdl(gateup_decode_kernel<R, S, 4>, g_gu, s, pdl, a, max_active)
  if (fmt_r_gu == FMT_Q2_K && fsg == FMT_Q2_K) DS4_GU(FMT_Q2_K, FMT_Q2_K);
  else if (fmt_r_gu == FMT_Q2_K) DS4_GU(FMT_Q2_K, FMT_Q8_0);
  else if (fsg == FMT_Q2_K) DS4_GU(FMT_Q8_0, FMT_Q2_K);
  else DS4_GU(FMT_Q8_0, FMT_Q8_0);
#undef DS4_GU
  if (e != cudaSuccess) return e;
  if (hooks) hooks->mark(hooks->ctx, "gateup");
  const int fsd = a.n_shared ? fmt_s : fmt_r_d;
  const dim3 g_dn(a.d / 16);
#define DS4_DN(R, S)                                                                          \
  e = one ? launch_pdl(down_decode_kernel<R, S, 1>, g_dn, s, pdl, a, max_active)              \
          : launch_pdl(down_decode_kernel<R, S, 4>, g_dn, s, pdl, a, max_active)
  if (fmt_r_d == FMT_Q2_K && fsd == FMT_Q2_K) DS4_DN(FMT_Q2_K, FMT_Q2_K);
  else if (fmt_r_d == FMT_Q2_K) DS4_DN(FMT_Q2_K, FMT_Q8_0);
  else if (fsd == FMT_Q2_K) DS4_DN(FMT_Q8_0, FMT_Q2_K);
  else DS4_DN(FMT_Q8_0, FMT_Q8_0);
#undef DS4_DN
  if (e != cudaSuccess) return e;
  if (hooks) hooks->mark(hooks->ctx, "down_combine");
  if (launches) *launches = 3;
  return cudaSuccess;
}

}  // namespace ds4
