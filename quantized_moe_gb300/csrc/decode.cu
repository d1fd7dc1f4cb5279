// Decode path (1..16 tokens, at most 128 routed slots): three kernels chained with
// programmatic dependent launch.
//
//  route_decode_kernel    one CTA per routed expert computes its fp32 logits for every token;
//                         the last CTA to finish (atomic arrival counter, no waiting) runs the
//                         sigmoid top-k (or table routing), the bucketing, and publishes a work
//                         list (expert, first position, count) per active expert, the token of
//                         every bucketed position and the fp16 scale of every token. It lets the
//                         gate/up kernel launch at once.
//  gateup_decode_kernel   CTA = 16 rows of f of one active expert, K split over 8 warps, each warp
//                         streaming its units through a two-deep register pipeline; h = silu(g) * u
//                         in fp32 plus max|h| per row of H (integer atomicMax: order-free). Its first
//                         grid row computes the shared expert's gate/up (one CTA per 16 rows of
//                         f_shared): it needs no routing, so those CTAs do not wait for the route
//                         kernel and overlap it; the routed CTAs wait for it.
//  down_decode_kernel     CTA = 16 rows of d for every touched expert and the shared expert;
//                         (expert, K unit) items are dealt round-robin to the warps, each warp
//                         accumulates its partials in shared memory in a fixed order, and the
//                         CTA writes the final rows: routed terms in ascending expert id, then
//                         the shared expert.
//
// Tokens are processed one per pass (an expert with several tokens streams its weight units once
// per token, the later passes from L2). Weights that do not depend on the previous kernel's output
// are loaded before waiting on it: every down unit (the routing being final by then).
#include "mma_units.cuh"

namespace ds4 {
namespace {

constexpr int kWarps = 8;
constexpr int kThreads = 256;
// the one-token top-k of the route kernel ranks one expert per thread (n_experts <= 256)
static_assert(kThreads >= 256, "route kernel: one thread per expert");
constexpr int kMaxTok = 16;
constexpr int kMaxSlots = 128;
constexpr int kMaxJ = 12;  // d <= 12288: float4 loads per lane of one router row slice
// Tokens per pass of the GEMV kernels. One: every pass streams the item's weight units again (the
// later passes from L2), and the kernels fit in 128 registers, so two CTAs (16 warps) run per SM.
// Passes of two tokens needed up to 254 registers (one CTA per SM) and measured slower on batched
// decode (16 tokens: 753 against 608 us per forward).
constexpr int kPass = 1;

// ----------------------------------------------------------------------------- route

template <int FMT_S>
__device__ void shared_gateup_cta(const DecodeArgs& a, int rg);

__global__ void __launch_bounds__(kThreads, 2) route_decode_kernel(DecodeArgs a) {
  // The gate/up kernel may launch now: its shared-expert CTAs need no routing and overlap this
  // kernel (its routed CTAs wait for this grid to complete).
  pdl_trigger();
  __shared__ float part[kWarps][kMaxTok];
  __shared__ float xmx[kWarps][kMaxTok];
  __shared__ int s_last;
  __shared__ int s_idx[kMaxSlots];
  __shared__ int s_cnt[256], s_off[257], s_act[256], s_nact;
  const int e = blockIdx.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int d = a.d, nt = a.n_tok;
  // ---- logits of expert e for the learned tokens (and max|x| of every token in CTA 0);
  // each lane first issues all its loads of the router row slice
  // lane covers k = warp * per_warp + 4 lane + 128 j (per_warp is a multiple of 16)
  const int per_warp = d / kWarps, nj = per_warp > 4 * lane ? (per_warp - 4 * lane + 127) / 128 : 0;
  const float* wr = a.wr + (size_t)e * d + warp * per_warp + lane * 4;
  float4 wv[kMaxJ];
#pragma unroll
  for (int j = 0; j < kMaxJ; ++j)
    if (j < nj) wv[j] = *reinterpret_cast<const float4*>(wr + 128 * j);
  for (int t = 0; t < nt; ++t) {
    const __nv_bfloat16* xr = a.x + (size_t)t * d + warp * per_warp + lane * 4;
    uint2 xv[kMaxJ];
#pragma unroll
    for (int j = 0; j < kMaxJ; ++j)
      if (j < nj) xv[j] = *reinterpret_cast<const uint2*>(xr + 128 * j);
    float acc = 0.f, mx = 0.f;
#pragma unroll
    for (int j = 0; j < kMaxJ; ++j) {
      if (j >= nj) break;
      const float2 x01 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&xv[j].x));
      const float2 x23 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&xv[j].y));
      acc = fmaf(wv[j].x, x01.x, acc);
      acc = fmaf(wv[j].y, x01.y, acc);
      acc = fmaf(wv[j].z, x23.x, acc);
      acc = fmaf(wv[j].w, x23.y, acc);
      mx = fmaxf(mx, fmaxf(fmaxf(fabsf(x01.x), fabsf(x01.y)), fmaxf(fabsf(x23.x), fabsf(x23.y))));
    }
    acc = warp_sum(acc);
    mx = warp_max(mx);
    if (lane == 0) { part[warp][t] = acc; xmx[warp][t] = mx; }
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
      a.xscale[t] = fp16_row_scale(m);  // final once this grid completes
    }
  }
  // ---- arrival: the last CTA continues with the top-k and the bucketing. The barrier orders the
  // CTA's writes before thread 0's release-acquire arrival, whose gpu-scope ordering covers them.
  __syncthreads();
  if (threadIdx.x == 0) {
    unsigned prev;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;\n" : "=r"(prev) : "l"(a.counter) : "memory");
    s_last = prev == (unsigned)a.n_exp - 1;  // the router CTAs only
  }
  __syncthreads();
  if (!s_last) return;
  const int K = a.top_k, E = a.n_exp, n_slots = nt * K;
  if (threadIdx.x == 0) *a.err = 0;  // only this CTA writes the error word
  if (nt == 1 && a.n_hash == 0) {
    // One learned token: thread e ranks expert e among all (higher score first, ties to the
    // lower index: the order of the warp selection below), and the k winners are bucketed in
    // closed form (one position each, in ascending expert id).
    __shared__ float s_sc[256], s_selw[16];
    __shared__ int s_sel[16], s_loc[16];
    const int ex = threadIdx.x;
    const float sc = ex < E ? 1.f / (1.f + expf(-__ldcg(a.logits + ex))) : -1.f;
    s_sc[ex] = sc;
    __syncthreads();
    int rank = 0;
    if (ex < E) {
#pragma unroll 8
      for (int j = 0; j < E; ++j) {
        const float v = s_sc[j];
        rank += (v > sc) || (v == sc && j < ex);
      }
      if (rank < K) {
        s_sel[rank] = ex;
        s_selw[rank] = sc;
        s_loc[rank] = a.local_of ? a.local_of[ex] : ex;  // < 0: an expert this handle does not hold
      }
    }
    __syncthreads();
    // the selected experts this handle holds take one bucketed position each, in ascending id
    int n_own = 0;
    for (int q = 0; q < K; ++q) n_own += s_loc[q] >= 0;
    if (threadIdx.x < K) {
      const int r = threadIdx.x, er = s_sel[r];
      float sum = 0.f;
      for (int q = 0; q < K; ++q) sum += s_selw[q];  // selection order, as the warp version
      int pos = 0;
      for (int q = 0; q < K; ++q) pos += s_sel[q] < er && s_loc[q] >= 0;
      a.idx[r] = er;
      a.wts[r] = s_selw[r] / sum;
      if (s_loc[r] >= 0) {
        a.perm[pos] = r;
        a.rowof[r] = pos;
        a.tokof[pos] = 0;
        a.active[pos] = er;
        a.work[pos] = make_int4(s_loc[r], pos, 1, 1);
      } else {
        a.rowof[r] = -1;
      }
      if (r >= n_own) a.work[r] = make_int4(0, 0, 0, 0);  // the work list ends at n_own
    }
    if (ex < E) {
      int off = 0;
      bool own = false;
      for (int q = 0; q < K; ++q) {
        off += s_sel[q] < ex && s_loc[q] >= 0;
        own |= s_sel[q] == ex && s_loc[q] >= 0;
      }
      a.counts[ex] = own ? 1 : 0;
      a.offsets[ex] = off;
    }
    if (threadIdx.x == 0) {
      a.offsets[E] = n_own;
      *a.n_active = n_own;
    }
    for (int i = threadIdx.x; i < n_slots; i += kThreads) a.hmax[i] = 0.f;
    if (threadIdx.x == 0) *a.counter = 0u;
    return;
  }
  for (int t = warp; t < nt; t += kWarps) {
    if (t < a.n_hash) {
      const int id = a.token_ids[t];
      const bool ok = id >= 0 && id < a.vocab;
      if (!ok && lane == 0) atomicOr(a.err, 1);
      if (lane < K) {
        const int ex = ok ? a.table[(size_t)id * K + lane] : lane;  // bad id: distinct experts, weight 0
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
  for (int sl = threadIdx.x; sl < n_slots; sl += kThreads)  // integer counts of the experts held
    if (!a.local_of || a.local_of[s_idx[sl]] >= 0) atomicAdd(&s_cnt[s_idx[sl]], 1);
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
  }
  const int max_active = min(E, n_slots);
  for (int i = threadIdx.x; i < max_active; i += kThreads) {  // the work list, empty past n_active
    int4 w = make_int4(0, 0, 0, 0);
    if (i < s_nact) {
      const int ex = s_act[i];
      w = make_int4(a.local_of ? a.local_of[ex] : ex, s_off[ex], s_cnt[ex], 0);
      a.active[i] = ex;
    }
    a.work[i] = w;
  }
  if (threadIdx.x == 0) {
    a.offsets[E] = s_off[E];
    *a.n_active = s_nact;
  }
  for (int sl = threadIdx.x; sl < n_slots; sl += kThreads) {  // stable rank among equal experts
    const int ex = s_idx[sl];
    if (a.local_of && a.local_of[ex] < 0) {  // not held: no bucketed position, no term
      a.rowof[sl] = -1;
      continue;
    }
    int r = 0;
    for (int j = 0; j < sl; ++j) r += s_idx[j] == ex;
    const int pos = s_off[ex] + r;
    a.perm[pos] = sl;
    a.rowof[sl] = pos;
    a.tokof[pos] = sl / K;
  }
  for (int i = threadIdx.x; i < n_slots; i += kThreads) a.hmax[i] = 0.f;
  if (threadIdx.x == 0) *a.counter = 0u;  // every CTA has arrived: ready for the next forward
}

// ----------------------------------------------------------------------------- unit pipelines

template <int FMT>
struct Unit;
template <>
struct Unit<FMT_Q2_K> {
  Q2kUnitRegs r;
  __device__ __forceinline__ void load(const uint8_t* p) { r = q2k_load(p); }
  static constexpr int kChunks = 2;
};
template <>
struct Unit<FMT_Q8_0> {
  Q80UnitRegs r;
  __device__ __forceinline__ void load(const uint8_t* p) { r = q80_load(p); }
  static constexpr int kChunks = 1;
};

// Accumulates one unit of one matrix for np token fragments; acc[tt][rho] is the lane partial of
// row g + 8 rho (scaled by the token's fp16 scale).
template <int P>
__device__ __forceinline__ void unit_mma(const Unit<FMT_Q2_K>& u, const XFrag (&xf)[P][2], int np, const BMask& bm,
                                         const Q2kLaneConst& qc, float (&acc)[P][2]) {
  float as[P][2], am[P][2];
#pragma unroll
  for (int tt = 0; tt < P; ++tt) as[tt][0] = as[tt][1] = am[tt][0] = am[tt][1] = 0.f;
#pragma unroll
  for (int c = 0; c < 2; ++c) {
    const uint32_t w[4] = {u.r.q[c].x, u.r.q[c].y, u.r.q[c].z, u.r.q[c].w};
    const uint32_t wh[4] = {w[0] >> 10, w[1] >> 10, w[2] >> 10, w[3] >> 10};
    const Q2kChunkScales s = q2k_chunk_scales(u.r.sc[c], qc);
#pragma unroll
    for (int tt = 0; tt < P; ++tt) {
      if (tt >= np) break;
      float dd[4];
      q2k_chunk_mma(w, wh, bm, xf[tt][c], dd);
      as[tt][0] = fmaf(s.s00, dd[0], fmaf(s.s01, dd[1], as[tt][0]));
      as[tt][1] = fmaf(s.s10, dd[2], fmaf(s.s11, dd[3], as[tt][1]));
      am[tt][0] = fmaf(s.m00, xf[tt][c].s0, fmaf(s.m01, xf[tt][c].s1, am[tt][0]));
      am[tt][1] = fmaf(s.m10, xf[tt][c].s0, fmaf(s.m11, xf[tt][c].s1, am[tt][1]));
    }
  }
  const float2 d0 = __half22float2(*reinterpret_cast<const __half2*>(&u.r.dd0));
  const float2 d1 = __half22float2(*reinterpret_cast<const __half2*>(&u.r.dd1));
#pragma unroll
  for (int tt = 0; tt < P; ++tt) {
    if (tt >= np) break;
    acc[tt][0] = fmaf(d0.x, as[tt][0], fmaf(-d0.y, am[tt][0], acc[tt][0]));
    acc[tt][1] = fmaf(d1.x, as[tt][1], fmaf(-d1.y, am[tt][1], acc[tt][1]));
  }
}

template <int P>
__device__ __forceinline__ void unit_mma(const Unit<FMT_Q8_0>& u, const XFrag (&xf)[P][2], int np, const BMask& bm,
                                         const Q2kLaneConst&, float (&acc)[P][2]) {
  const float2 s = __half22float2(*reinterpret_cast<const __half2*>(&u.r.sc));
#pragma unroll
  for (int tt = 0; tt < P; ++tt) {
    if (tt >= np) break;
    float dd[4];
    q80_chunk_mma(u.r.v, bm, xf[tt][0], dd);
    const float off = 128.f * (xf[tt][0].s0 + xf[tt][0].s1);
    acc[tt][0] = fmaf(s.x, fmaf(16777216.f, dd[0] + dd[1], -off), acc[tt][0]);
    acc[tt][1] = fmaf(s.y, fmaf(16777216.f, dd[2] + dd[3], -off), acc[tt][1]);
  }
}

// ----------------------------------------------------------------------------- gate/up

// One pipeline stage of the gate/up kernel: the gate and up units of one K unit plus the raw
// activation words of the pass's tokens for its chunks.
template <int FMT, int P>
struct GuStage {
  Unit<FMT> g, u;
  uint2 xr[P][2];
};

template <int FMT, int P>
__device__ __forceinline__ void gu_load_w(GuStage<FMT, P>& st, const uint8_t* w0, const uint8_t* w1, int rg, int kb,
                                          int n_kb) {
  st.g.load(w0 + unit_offset(rg, kb, n_kb, unit_bytes(FMT)));
  st.u.load(w1 + unit_offset(rg, kb, n_kb, unit_bytes(FMT)));
}

template <int FMT, int P>
__device__ __forceinline__ void gu_load_x(GuStage<FMT, P>& st, const __nv_bfloat16* const (&xrow)[P], int np, int kb) {
#pragma unroll
  for (int tt = 0; tt < P; ++tt) {
    if (tt >= np) break;
#pragma unroll
    for (int c = 0; c < Unit<FMT>::kChunks; ++c) st.xr[tt][c] = xraw_bf16(xrow[tt] + kb * unit_k(FMT) + 128 * c);
  }
}

template <int FMT, int P>
__device__ __forceinline__ void gu_compute(const GuStage<FMT, P>& st, const float (&sc)[P], int np, const BMask& bm,
                                           const Q2kLaneConst& qc, float (&accg)[P][2], float (&accu)[P][2]) {
  XFrag xf[P][2];
#pragma unroll
  for (int tt = 0; tt < P; ++tt) {
    if (tt >= np) break;
#pragma unroll
    for (int c = 0; c < Unit<FMT>::kChunks; ++c) xf[tt][c] = xfrag_from_bf16(st.xr[tt][c], sc[tt]);
  }
  unit_mma<P>(st.g, xf, np, bm, qc, accg);
  unit_mma<P>(st.u, xf, np, bm, qc, accu);
}

// The K units kb = warp + 8 i of one CTA row group, through a two-deep register pipeline.
// The first two stages may already hold their weights (loaded before the dependency wait).
template <int FMT, int P>
__device__ __forceinline__ void gu_stream(GuStage<FMT, P>& s0, GuStage<FMT, P>& s1, bool preloaded,
                                          const uint8_t* w0, const uint8_t* w1, int rg, int n_kb,
                                          const __nv_bfloat16* const (&xrow)[P], const float (&sc)[P], int np,
                                          const BMask& bm, const Q2kLaneConst& qc, float (&accg)[P][2],
                                          float (&accu)[P][2]) {
  const int warp = threadIdx.x >> 5;
  const int nk = n_kb > warp ? (n_kb - warp + kWarps - 1) / kWarps : 0;
  if (!preloaded) {
    if (nk > 0) gu_load_w(s0, w0, w1, rg, warp, n_kb);
    if (nk > 1) gu_load_w(s1, w0, w1, rg, warp + kWarps, n_kb);
  }
  if (nk > 0) gu_load_x(s0, xrow, np, warp);
  if (nk > 1) gu_load_x(s1, xrow, np, warp + kWarps);
  for (int i = 0; i < nk; i += 2) {
    gu_compute(s0, sc, np, bm, qc, accg, accu);
    if (i + 2 < nk) {
      gu_load_w(s0, w0, w1, rg, warp + kWarps * (i + 2), n_kb);
      gu_load_x(s0, xrow, np, warp + kWarps * (i + 2));
    }
    if (i + 1 < nk) {
      gu_compute(s1, sc, np, bm, qc, accg, accu);
      if (i + 3 < nk) {
        gu_load_w(s1, w0, w1, rg, warp + kWarps * (i + 3), n_kb);
        gu_load_x(s1, xrow, np, warp + kWarps * (i + 3));
      }
    }
  }
}

// Quad and warp reductions of one pass, SwiGLU, store of h and of max|h| over the 16 rows: into
// hmax[row0 + tt] with an integer atomicMax (order-free), or, with GROUP_MAX, as a plain store into
// hmax[(row0 + tt) * n_groups + rg] (one entry per row group, reduced by the reader).
template <int P, bool GROUP_MAX = false>
__device__ __forceinline__ void gu_epilogue(float (&red)[kWarps][2][P][16], const float (&accg)[P][2],
                                            const float (&accu)[P][2], const float (&sc)[P], int np, float* hbase,
                                            int ldh, int row0, int rg, float* hmax, int n_groups = 0) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
#pragma unroll
  for (int tt = 0; tt < P; ++tt)
#pragma unroll
    for (int rho = 0; rho < 2; ++rho) {
      float vg = accg[tt][rho], vu = accu[tt][rho];
      vg += __shfl_xor_sync(0xffffffffu, vg, 1);
      vg += __shfl_xor_sync(0xffffffffu, vg, 2);
      vu += __shfl_xor_sync(0xffffffffu, vu, 1);
      vu += __shfl_xor_sync(0xffffffffu, vu, 2);
      if (t == 0) { red[warp][0][tt][g + 8 * rho] = vg; red[warp][1][tt][g + 8 * rho] = vu; }
    }
  __syncthreads();
  if (threadIdx.x < (P == 1 ? 32 : 16 * P)) {  // whole warps: the 16-lane shuffles below name all 32
    const int tt = min((int)threadIdx.x >> 4, P - 1), r = threadIdx.x & 15;
    const bool valid = (int)(threadIdx.x >> 4) < np;
    float sg = 0.f, su = 0.f;
    for (int w = 0; w < kWarps; ++w) { sg += red[w][0][tt][r]; su += red[w][1][tt][r]; }
    const float inv = 1.f / sc[tt];
    const float h = valid ? silu_mul(sg * inv, su * inv) : 0.f;
    if (valid) hbase[(size_t)(row0 + tt) * ldh + rg * 16 + r] = h;
    float m = fabsf(h);
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o, 16));
    if (valid && r == 0) {
      if (GROUP_MAX)
        hmax[(size_t)(row0 + tt) * n_groups + rg] = m;
      else
        atomicMax(reinterpret_cast<unsigned*>(hmax + row0 + tt), __float_as_uint(m));
    }
  }
  __syncthreads();
}

template <int FMT_R, int FMT_S, int P>
__global__ void __launch_bounds__(kThreads, 2) gateup_decode_kernel(DecodeArgs a, int max_active) {
  __shared__ float red[kWarps][2][P][16];
  const int rg = blockIdx.x, warp = threadIdx.x >> 5;
  if (a.n_shared && blockIdx.y == 0) {  // the shared expert (row group rg): no routing, no wait
    pdl_trigger();
    shared_gateup_cta<FMT_S>(a, rg);
    return;
  }
  const BMask bm;
  const Q2kLaneConst qc;
  if (rg * 16 >= a.f) return;
  pdl_wait();
  pdl_trigger();
  const int4 wk = a.work[blockIdx.y - (a.n_shared ? 1 : 0)];  // expert, first position, count (0 past the active ones)
  const int e = wk.x, pos0 = wk.y, cnt = wk.z;
  if (cnt == 0) return;
  const uint8_t* w0 = a.gate + (size_t)e * a.mb_gu;
  const uint8_t* w1 = a.up + (size_t)e * a.mb_gu;
  const int n_kb = a.d / unit_k(FMT_R);
  GuStage<FMT_R, P> s0, s1;
  for (int p0 = 0; p0 < cnt; p0 += P) {
    const int np = min(P, cnt - p0);
    const __nv_bfloat16* xrow[P];
    float sc[P];
#pragma unroll
    for (int tt = 0; tt < P; ++tt) {
      const int tok = a.tokof[pos0 + p0 + min(tt, np - 1)];
      xrow[tt] = a.x + (size_t)tok * a.d;
      sc[tt] = a.xscale[tok];
    }
    float accg[P][2], accu[P][2];
#pragma unroll
    for (int tt = 0; tt < P; ++tt) accg[tt][0] = accg[tt][1] = accu[tt][0] = accu[tt][1] = 0.f;
    gu_stream<FMT_R, P>(s0, s1, false, w0, w1, rg, n_kb, xrow, sc, np, bm, qc, accg, accu);
    gu_epilogue<P>(red, accg, accu, sc, np, a.H, a.f, pos0 + p0, rg, a.hmax);
  }
}

// The shared expert's gate/up for 16 rows (row group rg of f_shared) and every token, run by the
// gate/up kernel's first grid row without waiting for the route kernel. The token scales are
// computed here (the router's CTA 0 publishes them only after the routing); max|h| of the 16 rows
// goes to hsg[token][rg] (the down kernel reduces over the row groups).
template <int FMT_S>
__device__ void shared_gateup_cta(const DecodeArgs& a, int rg) {
  constexpr int P = kPass;
  __shared__ float red[kWarps][2][P][16];
  __shared__ float s_xsc[kMaxTok];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (rg * 16 >= a.fs) return;
  const BMask bm;
  const Q2kLaneConst qc;
  const int n_kb = a.d / unit_k(FMT_S);
  GuStage<FMT_S, P> s0, s1;
  const int nk = n_kb > warp ? (n_kb - warp + kWarps - 1) / kWarps : 0;
  // the first units are in flight while the token scales are computed
  if (nk > 0) gu_load_w(s0, a.sgate, a.sup, rg, warp, n_kb);
  if (nk > 1) gu_load_w(s1, a.sgate, a.sup, rg, warp + kWarps, n_kb);
  for (int t = warp; t < a.n_tok; t += kWarps) {
    const __nv_bfloat16* xr = a.x + (size_t)t * a.d;
    float m = 0.f;
    for (int k = lane * 8; k < a.d; k += 256) {
      const uint4 v = *reinterpret_cast<const uint4*>(xr + k);
      const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 f = __bfloat1622float2(h[i]);
        m = fmaxf(m, fmaxf(fabsf(f.x), fabsf(f.y)));
      }
    }
    m = warp_max(m);
    if (lane == 0) s_xsc[t] = fp16_row_scale(m);
  }
  __syncthreads();
  const int n_groups = a.fs / 16;
  for (int p0 = 0; p0 < a.n_tok; p0 += P) {
    const int np = min(P, a.n_tok - p0);
    const __nv_bfloat16* xrow[P];
    float sc[P];
#pragma unroll
    for (int tt = 0; tt < P; ++tt) {
      const int tok = p0 + min(tt, np - 1);
      xrow[tt] = a.x + (size_t)tok * a.d;
      sc[tt] = s_xsc[tok];
    }
    float accg[P][2], accu[P][2];
#pragma unroll
    for (int tt = 0; tt < P; ++tt) accg[tt][0] = accg[tt][1] = accu[tt][0] = accu[tt][1] = 0.f;
    gu_stream<FMT_S, P>(s0, s1, p0 == 0, a.sgate, a.sup, rg, n_kb, xrow, sc, np, bm, qc, accg, accu);
    gu_epilogue<P, true>(red, accg, accu, sc, np, a.Hs, a.fs, p0, rg, a.hsg, n_groups);
  }
}

// ----------------------------------------------------------------------------- down + combine

// Item i of a CTA: routed items first (work entry i / n_kb_r, K unit i % n_kb_r), then the
// shared expert's K units.
struct DownItem {
  int shared, kb, pos0, cnt;
  const uint8_t* w;
};

__device__ __forceinline__ DownItem down_item(const DecodeArgs& a, int i, int n_routed, int n_kb_r) {
  DownItem it;
  it.shared = i >= n_routed;
  if (!it.shared) {
    const int4 wk = a.work[i / n_kb_r];
    it.kb = i % n_kb_r;
    it.pos0 = wk.y;
    it.cnt = wk.z;
    it.w = a.down + (size_t)wk.x * a.mb_d;
  } else {
    it.kb = i - n_routed;
    it.pos0 = 0;
    it.cnt = a.n_tok;
    it.w = a.sdown;
  }
  return it;
}

// The lane's h values (two float2 per chunk) and max|h| of the first pass of an item's rows,
// loaded together with its weight unit so that the first pass waits on no L2 round trip.
template <int P>
struct HPre {
  float2 v[P][2][2];
  float hm[P];
};

// max|h| of row `row` of the item's h: routed slots from the gate/up kernel's atomic maxima, the
// shared expert's tokens from the CTA's shared-memory copy (s_hms).
__device__ __forceinline__ float item_hmax(const DecodeArgs& a, const DownItem& it, int row, const float* s_hms) {
  return it.shared ? s_hms[row] : __ldcg(a.hmax + row);
}

template <int FMT, int P>
__device__ __forceinline__ void h_prefetch(const DecodeArgs& a, const DownItem& it, HPre<P>& hp, const float* s_hms) {
  const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
  const float* hbase = it.shared ? a.Hs : a.H;
  const int kdim = it.shared ? a.fs : a.f;
#pragma unroll
  for (int tt = 0; tt < P; ++tt) {
    if (tt >= it.cnt) break;
    const int row = it.pos0 + tt;
    hp.hm[tt] = item_hmax(a, it, row, s_hms);
#pragma unroll
    for (int c = 0; c < Unit<FMT>::kChunks; ++c) {
      const float* base = hbase + (size_t)row * kdim + it.kb * unit_k(FMT) + 128 * c;
      hp.v[tt][c][0] = __ldcg(reinterpret_cast<const float2*>(base + 16 * g + 2 * t));
      hp.v[tt][c][1] = __ldcg(reinterpret_cast<const float2*>(base + 16 * g + 2 * t + 8));
    }
  }
}

// B fragment from h values already in registers (what xfrag_f32 computes after its loads).
__device__ __forceinline__ XFrag xfrag_vals(float2 v0, float2 v1, float sc) {
  const __half2 h0 = __floats2half2_rn(v0.x * sc, v0.y * sc);
  const __half2 h1 = __floats2half2_rn(v1.x * sc, v1.y * sc);
  XFrag f;
  f.b0 = h2_bits(h0);
  f.b1 = h2_bits(h1);
  const float2 a = __half22float2(h0), b = __half22float2(h1);
  xfrag_sums(f, (a.x + a.y) + (b.x + b.y));
  return f;
}

// One item: the unit times the item's h rows (in passes of P), added to the warp's partial rows.
// The first pass uses the prefetched values.
template <int FMT, int P>
__device__ __forceinline__ void down_item_compute(const DecodeArgs& a, const DownItem& it, const Unit<FMT>& u,
                                                  const HPre<P>& hp, float* part_rows, const BMask& bm,
                                                  const Q2kLaneConst& qc, int kdim, const float* s_hms) {
  const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
  const float* hbase = it.shared ? a.Hs : a.H;
  for (int p0 = 0; p0 < it.cnt; p0 += P) {
    const int np = min(P, it.cnt - p0);
    float sc[P];
    XFrag xf[P][2];
#pragma unroll
    for (int tt = 0; tt < P; ++tt) {
      if (tt >= np) break;
      const int row = it.pos0 + p0 + tt;
      if (p0 == 0) {
        sc[tt] = fp16_row_scale(hp.hm[tt]);
#pragma unroll
        for (int c = 0; c < Unit<FMT>::kChunks; ++c) xf[tt][c] = xfrag_vals(hp.v[tt][c][0], hp.v[tt][c][1], sc[tt]);
      } else {
        sc[tt] = fp16_row_scale(item_hmax(a, it, row, s_hms));
#pragma unroll
        for (int c = 0; c < Unit<FMT>::kChunks; ++c)
          xf[tt][c] = xfrag_f32(hbase + (size_t)row * kdim + it.kb * unit_k(FMT) + 128 * c, sc[tt]);
      }
    }
    float acc[P][2];
#pragma unroll
    for (int tt = 0; tt < P; ++tt) acc[tt][0] = acc[tt][1] = 0.f;
    unit_mma<P>(u, xf, np, bm, qc, acc);
#pragma unroll
    for (int tt = 0; tt < P; ++tt) {
      if (tt >= np) break;
#pragma unroll
      for (int rho = 0; rho < 2; ++rho) {
        float v = acc[tt][rho];
        v += __shfl_xor_sync(0xffffffffu, v, 1);
        v += __shfl_xor_sync(0xffffffffu, v, 2);
        if (t == 0) part_rows[(size_t)(it.pos0 + p0 + tt) * 16 + g + 8 * rho] += v / sc[tt];
      }
    }
  }
}

// Registers of one loaded unit of either format (a Q8_0 unit fills v[0..3] and w[0]; a Q2_K
// unit fills v[0..1] and w[0..3]), so that both item kinds share one pipeline buffer.
struct RawUnit {
  uint4 v[4];
  uint32_t w[4];
};

template <int FMT>
__device__ __forceinline__ void raw_load(RawUnit& b, const uint8_t* __restrict__ ub) {
  const int lane = threadIdx.x & 31, g = lane >> 2;
  const int off = 16 * lane_region(g, lane & 3);
  if (FMT == FMT_Q2_K) {
    const uint4 q0 = ldg_nc_v4(ub + off), q1 = ldg_nc_v4(ub + 512 + off);
    b.v[0] = make_uint4(q0.x, q0.z, q0.y, q0.w);  // the region's words in A register order
    b.v[1] = make_uint4(q1.x, q1.z, q1.y, q1.w);
    b.w[0] = ldg_nc_u32(ub + kQ2kScOff + 4 * lane);
    b.w[1] = ldg_nc_u32(ub + kQ2kScOff + 128 + 4 * lane);
    b.w[2] = ldg_nc_u32(ub + kQ2kDdOff + 4 * g);
    b.w[3] = ldg_nc_u32(ub + kQ2kDdOff + 4 * (g + 8));
  } else {
#pragma unroll
    for (int j = 0; j < 4; ++j) b.v[j] = ldg_nc_v4(ub + 512 * j + off);
    b.w[0] = ldg_nc_u32(ub + kQ80ScOff + 4 * lane);
  }
}

__device__ __forceinline__ Unit<FMT_Q2_K> as_q2k(const RawUnit& b) {
  Unit<FMT_Q2_K> u;
  u.r.q[0] = b.v[0];
  u.r.q[1] = b.v[1];
  u.r.sc[0] = b.w[0];
  u.r.sc[1] = b.w[1];
  u.r.dd0 = b.w[2];
  u.r.dd1 = b.w[3];
  return u;
}

__device__ __forceinline__ Unit<FMT_Q8_0> as_q80(const RawUnit& b) {
  Unit<FMT_Q8_0> u;
#pragma unroll
  for (int j = 0; j < 4; ++j) u.r.v[j] = b.v[j];
  u.r.sc = b.w[0];
  return u;
}

template <int FMT>
__device__ __forceinline__ Unit<FMT> as_unit(const RawUnit& b);
template <>
__device__ __forceinline__ Unit<FMT_Q2_K> as_unit<FMT_Q2_K>(const RawUnit& b) { return as_q2k(b); }
template <>
__device__ __forceinline__ Unit<FMT_Q8_0> as_unit<FMT_Q8_0>(const RawUnit& b) { return as_q80(b); }

template <int FMT_R, int FMT_S>
__device__ __forceinline__ void down_load(const DownItem& it, RawUnit& b, int rg, int n_kb_r, int n_kb_s) {
  if (it.shared)
    raw_load<FMT_S>(b, it.w + unit_offset(rg, it.kb, n_kb_s, unit_bytes(FMT_S)));
  else
    raw_load<FMT_R>(b, it.w + unit_offset(rg, it.kb, n_kb_r, unit_bytes(FMT_R)));
}

template <int FMT_R, int FMT_S, int P>
__device__ __forceinline__ void down_item_run(const DecodeArgs& a, const DownItem& it, const RawUnit& b,
                                              const HPre<P>& hp, float* part, float* parts, const BMask& bm,
                                              const Q2kLaneConst& qc, const float* s_hms) {
  if (it.shared)
    down_item_compute<FMT_S, P>(a, it, as_unit<FMT_S>(b), hp, parts, bm, qc, a.fs, s_hms);
  else
    down_item_compute<FMT_R, P>(a, it, as_unit<FMT_R>(b), hp, part, bm, qc, a.f, s_hms);
}

template <int FMT_R, int FMT_S, int P>
__device__ __forceinline__ void down_h_prefetch(const DecodeArgs& a, const DownItem& it, HPre<P>& hp,
                                                const float* s_hms) {
  if (it.shared)
    h_prefetch<FMT_S, P>(a, it, hp, s_hms);
  else
    h_prefetch<FMT_R, P>(a, it, hp, s_hms);
}

template <int FMT_R, int FMT_S, int P>
__global__ void __launch_bounds__(kThreads, 2) down_decode_kernel(DecodeArgs a, int max_active) {
  extern __shared__ __align__(16) float dsm[];
  const int rg = blockIdx.x, warp = threadIdx.x >> 5;
  const int nt = a.n_tok, K = a.top_k, n_slots = nt * K;
  float* part = dsm + (size_t)warp * n_slots * 16;                               // [warp][position][16]
  float* parts = dsm + (size_t)kWarps * n_slots * 16 + (size_t)warp * nt * 16;  // [warp][token][16]
  const int n_kb_r = a.f / unit_k(FMT_R);
  const int n_kb_s = a.n_shared ? a.fs / unit_k(FMT_S) : 0;
  const BMask bm;
  const Q2kLaneConst qc;
  for (int i = threadIdx.x & 31; i < n_slots * 16; i += 32) part[i] = 0.f;
  for (int i = threadIdx.x & 31; i < nt * 16; i += 32) parts[i] = 0.f;
  // The routing is final once this kernel runs (its kernel completed before the gate/up kernel
  // passed its wait): the work list is valid, and the first down units can be loaded right away.
  const int n_act = *a.n_active;
  const int n_routed = n_act * n_kb_r, n_items = n_routed + n_kb_s;
  RawUnit b0, b1;
  DownItem it0{}, it1{};
  if (warp < n_items) {
    it0 = down_item(a, warp, n_routed, n_kb_r);
    down_load<FMT_R, FMT_S>(it0, b0, rg, n_kb_r, n_kb_s);
  }
  if (warp + kWarps < n_items) {
    it1 = down_item(a, warp + kWarps, n_routed, n_kb_r);
    down_load<FMT_R, FMT_S>(it1, b1, rg, n_kb_r, n_kb_s);
  }
  pdl_wait();
  // max|h| of each token of the shared expert, over the per-row-group maxima of its gate/up CTAs
  __shared__ float s_hms[kMaxTok];
  if (a.n_shared) {
    const int n_groups = a.fs / 16, lane = threadIdx.x & 31;
    for (int t = warp; t < nt; t += kWarps) {
      float m = 0.f;
      for (int j = lane; j < n_groups; j += 32) m = fmaxf(m, __ldcg(a.hsg + (size_t)t * n_groups + j));
      m = warp_max(m);
      if (lane == 0) s_hms[t] = m;
    }
  }
  __syncthreads();
  // h of the two preloaded items (H is complete now); later items fetch theirs with their units
  HPre<P> h0, h1;
  if (warp < n_items) down_h_prefetch<FMT_R, FMT_S, P>(a, it0, h0, s_hms);
  if (warp + kWarps < n_items) down_h_prefetch<FMT_R, FMT_S, P>(a, it1, h1, s_hms);
  for (int i = warp; i < n_items; i += 2 * kWarps) {
    down_item_run<FMT_R, FMT_S, P>(a, it0, b0, h0, part, parts, bm, qc, s_hms);
    if (i + 2 * kWarps < n_items) {
      it0 = down_item(a, i + 2 * kWarps, n_routed, n_kb_r);
      down_load<FMT_R, FMT_S>(it0, b0, rg, n_kb_r, n_kb_s);
      down_h_prefetch<FMT_R, FMT_S, P>(a, it0, h0, s_hms);
    }
    if (i + kWarps < n_items) {
      down_item_run<FMT_R, FMT_S, P>(a, it1, b1, h1, part, parts, bm, qc, s_hms);
      if (i + 3 * kWarps < n_items) {
        it1 = down_item(a, i + 3 * kWarps, n_routed, n_kb_r);
        down_load<FMT_R, FMT_S>(it1, b1, rg, n_kb_r, n_kb_s);
        down_h_prefetch<FMT_R, FMT_S, P>(a, it1, h1, s_hms);
      }
    }
  }
  __syncthreads();
  // combine: out[t][r] = routed terms in ascending expert id (each the fixed-order sum of the
  // warps' partials), then the shared expert
  const float* part0 = dsm;
  const float* parts0 = dsm + (size_t)kWarps * n_slots * 16;
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
    for (int j = 0; j < K; ++j) {
      if (ps[j] < 0) continue;  // an expert this handle does not hold
      float y = 0.f;
      for (int w = 0; w < kWarps; ++w) y += part0[((size_t)w * n_slots + ps[j]) * 16 + r];
      o = fmaf(wv[j], y, o);
    }
    if (a.n_shared) {
      float s = 0.f;
      for (int w = 0; w < kWarps; ++w) s += parts0[((size_t)w * nt + tok) * 16 + r];
      o += s;
    }
    a.out[(size_t)tok * a.d + rg * 16 + r] = o;
  }
}

template <typename Kern>
cudaError_t launch_ex(Kern kernel, dim3 grid, size_t smem, cudaStream_t s, bool pdl, const DecodeArgs& a,
                      int max_active) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, a, max_active);
}

template <int R, int S>
cudaError_t launch_gu(dim3 grid, cudaStream_t s, bool pdl, const DecodeArgs& a, int max_active) {
  return launch_ex(gateup_decode_kernel<R, S, kPass>, grid, 0, s, pdl, a, max_active);
}

template <int R, int S, int P>
cudaError_t launch_dn_p(dim3 grid, size_t smem, cudaStream_t s, bool pdl, const DecodeArgs& a, int max_active) {
  return launch_ex(down_decode_kernel<R, S, P>, grid, smem, s, pdl, a, max_active);
}

template <int R, int S>
cudaError_t prepare_dn() {
  return cudaFuncSetAttribute(down_decode_kernel<R, S, kPass>, cudaFuncAttributeMaxDynamicSharedMemorySize, 96 * 1024);
}

template <int R, int S>
cudaError_t launch_dn(dim3 grid, size_t smem, cudaStream_t s, bool pdl, const DecodeArgs& a, int max_active) {
  return launch_dn_p<R, S, kPass>(grid, smem, s, pdl, a, max_active);
}

}  // namespace

cudaError_t decode_prepare() {
  cudaError_t e = prepare_dn<FMT_Q2_K, FMT_Q2_K>();
  if (e == cudaSuccess) e = prepare_dn<FMT_Q2_K, FMT_Q8_0>();
  if (e == cudaSuccess) e = prepare_dn<FMT_Q8_0, FMT_Q2_K>();
  if (e == cudaSuccess) e = prepare_dn<FMT_Q8_0, FMT_Q8_0>();
  return e;
}

int decode_max_tokens() { return kMaxTok; }
int decode_max_slots() { return kMaxSlots; }

cudaError_t launch_decode(const DecodeArgs& a, int fmt_r_gu, int fmt_r_d, int fmt_s, bool pdl, cudaStream_t s,
                          int* launches, const DecodeHooks* hooks) {
  const int max_active = min(a.n_exp, a.n_tok * a.top_k);
  route_decode_kernel<<<a.n_exp, kThreads, 0, s>>>(a);  // one CTA per routed expert
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (hooks) hooks->mark(hooks->ctx, "route");
  // row y = 0: the shared expert's row groups (when it exists); rows 1..: the active experts
  const int fsg = a.n_shared ? fmt_s : fmt_r_gu;
  const dim3 g_gu(max(a.f, a.n_shared ? a.fs : 0) / 16, max_active + (a.n_shared ? 1 : 0));
  if (fmt_r_gu == FMT_Q2_K)
    e = fsg == FMT_Q2_K ? launch_gu<FMT_Q2_K, FMT_Q2_K>(g_gu, s, pdl, a, max_active)
                        : launch_gu<FMT_Q2_K, FMT_Q8_0>(g_gu, s, pdl, a, max_active);
  else
    e = fsg == FMT_Q2_K ? launch_gu<FMT_Q8_0, FMT_Q2_K>(g_gu, s, pdl, a, max_active)
                        : launch_gu<FMT_Q8_0, FMT_Q8_0>(g_gu, s, pdl, a, max_active);
  if (e != cudaSuccess) return e;
  if (hooks) hooks->mark(hooks->ctx, "gateup");
  const int fsd = a.n_shared ? fmt_s : fmt_r_d;
  const dim3 g_dn(a.d / 16);
  const size_t smem = (size_t)kWarps * (a.n_tok * a.top_k + a.n_tok) * 16 * sizeof(float);
  if (fmt_r_d == FMT_Q2_K && fsd == FMT_Q2_K) e = launch_dn<FMT_Q2_K, FMT_Q2_K>(g_dn, smem, s, pdl, a, max_active);
  else if (fmt_r_d == FMT_Q2_K) e = launch_dn<FMT_Q2_K, FMT_Q8_0>(g_dn, smem, s, pdl, a, max_active);
  else if (fsd == FMT_Q2_K) e = launch_dn<FMT_Q8_0, FMT_Q2_K>(g_dn, smem, s, pdl, a, max_active);
  else e = launch_dn<FMT_Q8_0, FMT_Q8_0>(g_dn, smem, s, pdl, a, max_active);
  if (e != cudaSuccess) return e;
  if (hooks) hooks->mark(hooks->ctx, "down_combine");
  if (launches) *launches = 3;
  return cudaSuccess;
}

}  // namespace ds4
