// Prefill expert GEMMs on the 5th-generation tensor cores (tcgen05, TMEM accumulators).
//
// Persistent: one CTA per SM loops over work items, each a 128-row x N-token tile of one expert
// (N <= 192 tokens; the MMA's N is the token count rounded up to 16):
//   gate/up: the 128 rows interleave 64 gate rows and the 64 up rows of the same features, so
//            the epilogue forms h = silu(g) * u for 64 features and writes it as fp16;
//   down:    128 rows of d, written as fp32 per bucketed slot for the fixed-order combine.
// The weight, activation and dequantized-tile pipelines run on across items, and the fp32
// accumulator is double-buffered in TMEM (2 x 256 columns), so the epilogue of one item overlaps
// the main loop of the next. Each K stage (64 wide) has one full barrier, completed by the
// dequant group that wrote its A tile and by the activation TMA, and one empty barrier, completed
// by the MMA commit; four stages are in flight.
// Warp roles (23 warps):
//   warp 0     weight producer: bulk-copies the packed weight units of each K unit (256 k for
//              Q2_K, 128 k for Q8_0) of the tile's rows;
//   warp 1     allocates TMEM; the converged warp runs the MMA loop and one elected lane issues
//              the tcgen05.mma and commits of every stage;
//   warp 2     activation producer: TMA-loads the fp16 activation tile (128-byte swizzle) of each
//              K stage, in 128-row boxes and at most one 64-row box;
//   warps 3-18 dequantize, in one group per K stage of a raw unit (four groups of four warps for
//              Q2_K, two of eight for Q8_0) taking the stages round-robin: each warp turns its
//              16-row groups' 64-wide K stage into fp16 weights in registers (exact small-integer
//              quants, one fp16 FMA with the sub-block scale and min) and writes them with
//              stmatrix straight into the swizzled A tile;
//   warps 19-22 epilogue: read the accumulator from TMEM (tcgen05.ld), one warp per lane
//              quadrant, and release its buffer to the MMA.
// Every mbarrier wait is bounded (tc::mbar_wait): on a timeout the CTA raises error bit 2 and
// unwinds instead of hanging.
#include <cudaTypedefs.h>

#include <algorithm>

#include "tc_ptx.cuh"

namespace ds4 {
namespace {

using namespace tc;

constexpr int BM = 128, BK = 64;
constexpr int A_BYTES = BM * BK * 2;            // 16 KB
constexpr int BOX_ROWS = 64;                    // rows per activation TMA box (8 KB)
constexpr int kDeqWarps = 16;
constexpr int kFirstDeq = 3;  // warps 0-2: weight producer, MMA, activation producer
constexpr int kEpiWarps = 4;  // warps 19-22: epilogue, one per TMEM lane quadrant
constexpr int kThreads = (kFirstDeq + kDeqWarps + kEpiWarps) * 32;  // 736
constexpr int ACC_COLS = 256;            // TMEM columns per accumulator (128 x N fp32, N <= 256)
constexpr int TMEM_COLS = 2 * ACC_COLS;  // double-buffered: the epilogue of one item overlaps the next

// Packed weight stages: eight 16-row units (one K unit of the 128-row tile) each; four stages of
// Q2_K (256 k each) or three of Q8_0 (128 k each) keep the next units' HBM reads in flight.
// Four K stages of 64 (A and B tiles) with token tiles of 192.
#ifndef GEMM_STAGES
#define GEMM_STAGES 4
#endif
#ifndef GEMM_BN
#define GEMM_BN 192
#endif
template <int FMT>
struct Cfg {
  static constexpr int RAW_BYTES = 8 * unit_bytes(FMT);
  static constexpr int RAWS = FMT == FMT_Q2_K ? 4 : 3;
  // Token tile (MMA N at most): 192 tokens, so that four K stages fit in shared memory beside the
  // raw weight stages.
  static constexpr int BN = GEMM_BN;
  static constexpr int B_BYTES = BN * BK * 2;
  // K stages in flight: each holds a dequantized weight tile (A) and an activation tile (B)
  static constexpr int STAGES = GEMM_STAGES;
  static constexpr int OFF_A = 0;
  static constexpr int OFF_B = OFF_A + STAGES * A_BYTES;
  static constexpr int OFF_RAW = OFF_B + STAGES * B_BYTES;
  static_assert(BN % BOX_ROWS == 0 && BN <= ACC_COLS, "token tile");
  static constexpr int OFF_BAR = OFF_RAW + RAWS * RAW_BYTES;
  static constexpr int N_BARS = 2 * STAGES + 2 * RAWS + 4;
  static constexpr int OFF_MISC = OFF_BAR + N_BARS * 8;
  static constexpr int OFF_GBUF = (OFF_MISC + 16 + 15) / 16 * 16;
  // gate/up epilogue: two parities x (8 columns of g + 8 columns of u) x 64 features fp32, then the
  // 1 / scale of each token of the tile
  static constexpr int GBUF_BYTES = 2 * 2 * 8 * 64 * 4 + 256 * 4;
  static constexpr int SMEM_BYTES = OFF_GBUF + GBUF_BYTES + 1024;  // + alignment slack
  static_assert(SMEM_BYTES <= 232448, "shared memory budget");
};

// One full/empty pair per K stage for both operands: the MMA thread makes one wait and one commit
// per stage, and the dequant warps and the activation producer wait on the same release.
struct Bars {
  uint64_t* full;       // [STAGES] dequant group (A) + activation TMA (B, with its bytes) -> MMA
  uint64_t* empty;      // [STAGES] MMA commit -> dequant group and activation producer
  uint64_t* raw_full;   // [RAWS] weight bulk copy -> dequant
  uint64_t* raw_empty;  // [RAWS] dequant -> producer
  uint64_t* acc_full;   // [2] MMA -> epilogue
  uint64_t* acc_empty;  // [2] epilogue -> MMA
};

// silu(g) * u with the hardware exponential and division (a few ulp, far inside the tolerance):
// the epilogue shares issue slots with the dequant warps.
__device__ __forceinline__ float silu_mul_fast(float g, float u) { return __fdividef(g, 1.f + __expf(-g)) * u; }

__device__ __forceinline__ uint32_t h2u(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }
__device__ __forceinline__ __half2 u2h(uint32_t u) { return *reinterpret_cast<__half2*>(&u); }

// stmatrix row address of this lane for the 16x16 block (row group rg16 of the tile, 16-k
// sub-block sb of the 64-k stage) in the 128-byte swizzled A tile.
__device__ __forceinline__ uint32_t a_row_addr(uint32_t a_base, int rg16, int sb) {
  const int lane = threadIdx.x & 31, j = lane >> 3, q = lane & 7;
  const int row = 16 * rg16 + q + 8 * (j & 1);
  const int kc = 2 * sb + (j >> 1);  // 16-byte chunk of the 128-byte row
  return a_base + (row >> 3) * 1024 + (row & 7) * 128 + ((kc ^ (row & 7)) << 4);
}

// Per-row constants of a Q2_K unit for this lane's rows (g, g+8): 2^16 d (exact: only the exponent
// changes; create refuses super-blocks whose 2^16 d * 15 would leave the fp16 range), -dmin and
// 1024 dmin (m is read as the fp16 1024 + m, so one FMA gives -dmin * m rounded once).
struct Q2kRowConst {
  __half2 d2, ndm2, dm1024;
};

__device__ __forceinline__ Q2kRowConst q2k_row_const(uint32_t unit) {
  const int g = (threadIdx.x & 31) >> 2;
  const uint32_t dd0 = lds32(unit + kQ2kDdOff + 4 * g), dd1 = lds32(unit + kQ2kDdOff + 4 * (g + 8));
  const __half2 k256 = __float2half2_rn(256.f);
  const __half2 dm2 = u2h(prmt(dd0, dd1, 0x7632u));  // (dmin of row g, dmin of row g+8)
  Q2kRowConst r;
  r.d2 = __hmul2(__hmul2(u2h(prmt(dd0, dd1, 0x5410u)), k256), k256);
  r.ndm2 = __hneg2(dm2);
  r.dm1024 = __hmul2(dm2, __float2half2_rn(1024.f));
  return r;
}

// All four 16-k sub-blocks I0..I0+3 of a Q2_K stage for this lane's rows in each of the warp's NR
// 16-row groups: the arithmetic of every (group, sub-block) pair is independent and interleaves,
// then the stores follow.
template <int I0, int NR>
__device__ __forceinline__ void deq_q2k_quad(const uint32_t (&w)[NR][4], const uint32_t (&sc01)[NR],
                                             const uint32_t (&sc23)[NR], const Q2kRowConst (&rc)[NR],
                                             uint32_t a_base, const uint32_t (&aoff)[NR][4]) {
  const __half2 k1024 = __float2half2_rn(1024.f);
  uint32_t a[NR][4][4];
#pragma unroll
  for (int n = 0; n < NR; ++n) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int sh = 8 - 2 * (I0 + j);  // left shift of sub-block I0 + j's field (negative: right)
      const uint32_t sc = (j < 2 ? sc01[n] : sc23[n]) >> (8 * (j & 1));
      const __half2 ds = __hmul2(__hsub2(u2h((sc & 0x000F000Fu) | 0x64006400u), k1024), rc[n].d2);
      const __half2 ndm = __hfma2(u2h(((sc >> 4) & 0x000F000Fu) | 0x64006400u), rc[n].ndm2, rc[n].dm1024);
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const uint32_t qb = (sh >= 0 ? (w[n][r] << sh) : (w[n][r] >> -sh)) & 0x03000300u;
        a[n][j][r] = h2u((r & 1) ? __hfma2(u2h(qb), __high2half2(ds), __high2half2(ndm))
                                 : __hfma2(u2h(qb), __low2half2(ds), __low2half2(ndm)));
      }
    }
  }
#pragma unroll
  for (int n = 0; n < NR; ++n)
#pragma unroll
    for (int j = 0; j < 4; ++j) stmatrix_x4(a_base + aoff[n][j], a[n][j][0], a[n][j][1], a[n][j][2], a[n][j][3]);
}

// The 16 rows x 64 k of K stage su (0..3) of NR Q2_K units (one per 16-row group of the warp).
template <int NR>
__device__ __forceinline__ void deq_q2k_stage(const uint32_t (&unit)[NR], int su, uint32_t a_base,
                                              const uint32_t (&aoff)[NR][4], const Q2kRowConst (&rc)[NR]) {
  const int lane = threadIdx.x & 31, g = lane >> 2;
  const int c = su >> 1, i0 = (su & 1) * 4;
  uint32_t w[NR][4], sc01[NR], sc23[NR];
#pragma unroll
  for (int n = 0; n < NR; ++n) {
    const uint4 qw = lds128(unit[n] + c * 512 + 16 * lane);
    w[n][0] = qw.x;
    w[n][1] = qw.y;
    w[n][2] = qw.z;
    w[n][3] = qw.w;
    sc01[n] = lds32(unit[n] + kQ2kScOff + c * 128 + 4 * (4 * g + i0 / 2));
    sc23[n] = lds32(unit[n] + kQ2kScOff + c * 128 + 4 * (4 * g + i0 / 2 + 1));
  }
  if (i0 == 0)
    deq_q2k_quad<0, NR>(w, sc01, sc23, rc, a_base, aoff);
  else
    deq_q2k_quad<4, NR>(w, sc01, sc23, rc, a_base, aoff);
}

// Waits (bounded, without raising errors) for a phase: used only to let copies land, or issued MMAs
// finish, before the CTA exits.
__device__ __forceinline__ void bounded_try(uint64_t* bar, uint32_t parity, long long limit) {
  const long long t0 = clock64();
  while (!mbar_try(bar, parity) && clock64() - t0 < limit) {
  }
}

// mbar_wait by lane 0 of a converged warp, its result given to every lane.
__device__ __forceinline__ bool lane0_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag, int* err, int site,
                                           long long limit) {
  bool ok = true;
  if ((threadIdx.x & 31) == 0) ok = mbar_wait(bar, parity, abort_flag, err, site, limit);
  return __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
}

// The tile of work item `it` (token tile, 128-row slice of the weights): `nbox` activation boxes
// of 64 rows are loaded, and the MMA's N (the accumulator columns the epilogue reads) is the row
// count rounded up to the instruction's granularity of 16, not to the box.
struct Item {
  int expert, row0, rows, nbox, n, mt;
};

template <int BN>
__device__ __forceinline__ Item item_of(const GemmArgs& p, int it) {
  Item t;
  const int tile = it / p.m_tiles;
  t.mt = it - tile * p.m_tiles;
  if (p.tiles) {
    const int4 v = __ldg(p.tiles + tile);
    t.expert = v.x;
    t.row0 = v.y;
    t.rows = v.z;
  } else {
    t.expert = -1;
    t.row0 = tile * BN;
    t.rows = min(BN, p.n_rows - t.row0);
  }
  t.nbox = (max(t.rows, 1) + BOX_ROWS - 1) / BOX_ROWS;
  t.n = (max(t.rows, 1) + 15) / 16 * 16;
  return t;
}

// Work items of the launch: (token tiles) x (128-row slices of the weights), slices fastest so that
// the CTAs running at the same time share their activation tiles through L2.
template <int BN>
__device__ __forceinline__ int item_count(const GemmArgs& p) {
  const int tiles = p.tiles ? *p.n_tiles : (p.n_rows + BN - 1) / BN;
  return tiles * p.m_tiles;
}

// The 16 rows x 64 k of one Q8_0 unit (128 k) that fall in K stage su (0..1): loads first, then
// the four sub-blocks, then the stores.
__device__ __forceinline__ void deq_q80_stage(uint32_t unit, int su, uint32_t a_base, const uint32_t (&aoff)[4]) {
  const int lane = threadIdx.x & 31, g = lane >> 2;
  const __half2 k1152 = __float2half2_rn(1152.f);
  uint4 v[2];
  uint32_t scw[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {  // 32-weight block 2 su + h: sub-blocks 2h, 2h + 1 of the stage
    v[h] = lds128(unit + 512 * (2 * su + h) + 16 * lane);
    scw[h] = lds32(unit + kQ80ScOff + 4 * (4 * g + 2 * su + h));
  }
  uint32_t a[4][4];
#pragma unroll
  for (int ii = 0; ii < 4; ++ii) {
    const uint4 vv = v[ii >> 1];
    const uint32_t wa = (ii & 1) ? vv.z : vv.x, wb = (ii & 1) ? vv.w : vv.y;
    const __half2 sc = u2h(scw[ii >> 1]);  // (row g, row g+8)
    const uint32_t raw[4] = {prmt(wa, 0x64u, 0x4140u), prmt(wa, 0x64u, 0x4342u), prmt(wb, 0x64u, 0x4140u),
                             prmt(wb, 0x64u, 0x4342u)};  // fp16 1024 + u, u = q + 128
#pragma unroll
    for (int r = 0; r < 4; ++r)
      a[ii][r] = h2u(__hmul2(__hsub2(u2h(raw[r]), k1152), (r & 1) ? __high2half2(sc) : __low2half2(sc)));
  }
#pragma unroll
  for (int ii = 0; ii < 4; ++ii) stmatrix_x4(a_base + aoff[ii], a[ii][0], a[ii][1], a[ii][2], a[ii][3]);
}

template <int FMT, bool GATEUP>
__global__ void __launch_bounds__(kThreads, 1) expert_gemm_tc_kernel(const __grid_constant__ CUtensorMap tmap64,
                                                                      const __grid_constant__ CUtensorMap tmap128,
                                                                      GemmArgs p) {
  using C = Cfg<FMT>;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr int UK = unit_k(FMT), UB = unit_bytes(FMT), RAWS = C::RAWS;
  constexpr int STAGES = C::STAGES;
  // dequant groups (one per K stage of a raw unit), warps per group, 16-row groups per warp
  constexpr int NG = UK / BK, WPG = kDeqWarps / NG, RPW = 8 / WPG;
  static_assert(NG <= STAGES && WPG * RPW == 8, "dequant groups");
  const int n_kb = p.k / UK, n_stages = p.k / BK, kpu = UK / BK;
  const int n_items = item_count<C::BN>(p);
  // gate/up: 64 gate rows then the 64 up rows of features 64 mt .. 64 mt + 63; down: 128 rows of d
  const uint32_t raw_copy = GATEUP ? 4 * UB : 8 * UB;
  const long long limit = p.timeout_cycles > 0 ? p.timeout_cycles : kTimeoutCycles;

  Bars b;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  b.full = bars;
  b.empty = bars + STAGES;
  b.raw_full = bars + 2 * STAGES;
  b.raw_empty = b.raw_full + RAWS;
  b.acc_full = b.raw_empty + RAWS;   // [2]
  b.acc_empty = b.acc_full + 2;      // [2]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
  float* gbuf = reinterpret_cast<float*>(smem + C::OFF_GBUF);
  float* ibuf = gbuf + 2048;

  if (threadIdx.x == 0) {
    for (int i = 0; i < STAGES; ++i) {
      mbar_init(&b.full[i], WPG + 1);  // one group of dequant warps + the activation producer
      mbar_init(&b.empty[i], 1);
    }
    for (int r = 0; r < RAWS; ++r) {
      mbar_init(&b.raw_full[r], 1);
      mbar_init(&b.raw_empty[r], kDeqWarps);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&b.acc_full[i], 1);
      mbar_init(&b.acc_empty[i], kEpiWarps);
    }
    *abort_flag = 0;
    mbar_init_fence();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------------ weight producer
    if (lane == 0) {
      uint32_t gu = 0;  // K units issued by this CTA over all its items
      for (int it = blockIdx.x; it < n_items && !*abort_flag; it += gridDim.x) {
        const Item t = item_of<C::BN>(p, it);
        const size_t eoff = t.expert >= 0 ? (size_t)t.expert * p.mat_bytes : 0;
        const uint8_t* src0 = p.w0 + eoff;
        const uint8_t* src1 = GATEUP ? p.w1 + eoff : nullptr;
        const int rg0 = GATEUP ? 4 * t.mt : 8 * t.mt;  // first 16-row group of the slice
        for (int uN = 0; uN < n_kb; ++uN, ++gu) {
          const int rs = gu % RAWS;
          if (!mbar_wait(&b.raw_empty[rs], ((gu / RAWS) & 1) ^ 1, abort_flag, p.err, 1, limit)) break;
          unsigned char* dst = smem + C::OFF_RAW + rs * C::RAW_BYTES;
          mbar_expect_tx(&b.raw_full[rs], GATEUP ? 2 * raw_copy : raw_copy);
          bulk_load(dst, src0 + unit_offset(rg0, uN, n_kb, UB), raw_copy, &b.raw_full[rs]);
          if (GATEUP) bulk_load(dst + raw_copy, src1 + unit_offset(rg0, uN, n_kb, UB), raw_copy, &b.raw_full[rs]);
        }
      }
      // the last copies land before the CTA may exit (after an abort they may still be in flight)
      for (uint32_t k = gu > (uint32_t)RAWS ? gu - RAWS : 0; k < gu; ++k)
        bounded_try(&b.raw_full[k % RAWS], (k / RAWS) & 1, limit);
    }
  } else if (warp == 2) {
    // ------------------------------------------------------------------ activation producer
    if (lane == 0) {
      uint32_t gs = 0;  // stages issued over all items
      for (int it = blockIdx.x; it < n_items && !*abort_flag; it += gridDim.x) {
        const Item t = item_of<C::BN>(p, it);
        for (int sB = 0; sB < n_stages; ++sB, ++gs) {
          const int sb = gs % STAGES;
          if (!mbar_wait(&b.empty[sb], ((gs / STAGES) & 1) ^ 1, abort_flag, p.err, 2, limit)) break;
          unsigned char* bdst = smem + C::OFF_B + sb * C::B_BYTES;
          const int rows = t.nbox * BOX_ROWS;  // rows fetched: 128-row boxes, then a 64-row one
          mbar_expect_tx(&b.full[sb], rows * BK * 2);
          int r = 0;
          for (; rows - r >= 2 * BOX_ROWS; r += 2 * BOX_ROWS)
            tma_load_2d(bdst + r * BK * 2, &tmap128, sB * BK, t.row0 + r, &b.full[sb]);
          if (r < rows) tma_load_2d(bdst + r * BK * 2, &tmap64, sB * BK, t.row0 + r, &b.full[sb]);
        }
      }
      for (uint32_t k = gs > (uint32_t)STAGES ? gs - STAGES : 0; k < gs; ++k)
        bounded_try(&b.full[k % STAGES], (k / STAGES) & 1, limit);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    // The whole warp runs the loop; lane 0 polls the barriers and one elected lane issues.
    uint32_t gs = 0;
    int local = 0;  // items of this CTA so far: accumulator buffer local & 1
    for (int it = blockIdx.x; it < n_items && !*abort_flag; it += gridDim.x, ++local) {
      const Item t = item_of<C::BN>(p, it);
      const int buf = local & 1;
      // the epilogue has drained this buffer (item local - 2)
      if (!lane0_wait(&b.acc_empty[buf], ((local >> 1) & 1) ^ 1, abort_flag, p.err, 6, limit)) break;
      tc_fence_after();
      const uint32_t idesc = idesc_f16_f32(BM, t.n);
      const uint32_t acc = tmem + (uint32_t)(buf * ACC_COLS);
      bool ok = true;
      for (int s = 0; s < n_stages; ++s, ++gs) {
        const int st = gs % STAGES;
        if (!lane0_wait(&b.full[st], (gs / STAGES) & 1, abort_flag, p.err, 7, limit)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint64_t ad = sw128_desc(su32(smem + C::OFF_A + st * A_BYTES));
        const uint64_t bd = sw128_desc(su32(smem + C::OFF_B + st * C::B_BYTES));
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk)  // advance 16 fp16 = 32 bytes along K per MMA
          tc_mma_f16_elect(acc, ad + 2 * kk, bd + 2 * kk, idesc, (s | kk) != 0);
        tc_commit_elect(&b.empty[st]);
      }
      if (!ok) break;
      tc_commit_elect(&b.acc_full[buf]);
    }
    // After an abort, the MMAs already issued must finish before TMEM is freed: the commit of the
    // last issued stage (stage gs - 1) arrives only once all of them have completed.
    if (*abort_flag && gs > 0 && lane == 0) bounded_try(&b.empty[(gs - 1) % STAGES], ((gs - 1) / STAGES) & 1, limit);
    __syncwarp();
  } else if (warp < kFirstDeq + kDeqWarps) {
    // ------------------------------------------------------------------ dequant
    // NG groups of warps take K stages round-robin, NG = the stages per raw unit (Q2_K four, Q8_0
    // two), so each group dequantizes one stage of every unit and NG stages are in progress at
    // once. In a stage, each warp of a group turns all four 16-k sub-blocks of its RPW 16-row
    // groups into fp16: 4 * RPW independent pieces of work per lane.
    const int dw = warp - kFirstDeq;
    const int grp = dw / WPG, wi = dw % WPG;
    // this lane's stmatrix row offsets for the sub-blocks of a stage (fixed per warp)
    uint32_t aoff[RPW][4];
#pragma unroll
    for (int n = 0; n < RPW; ++n)
#pragma unroll
      for (int j = 0; j < 4; ++j) aoff[n][j] = a_row_addr(0, wi + WPG * n, j);
    uint32_t gs0 = 0;  // stages of the CTA's earlier items
    for (int it = blockIdx.x; it < n_items && !*abort_flag; it += gridDim.x) {
      bool ok = true;
      // An item's stage count is a multiple of NG, so stage gs0 + s is this group's for s = grp,
      // grp + NG, ...: the group steps over its own stages only.
      for (int s = grp; s < n_stages; s += NG) {
        const uint32_t gs = gs0 + s;
        // the raw units follow the stages: unit gs / kpu of the CTA's sequence (kpu == NG)
        const uint32_t gu = gs / kpu;
        const int rs = gu % RAWS, sa = gs % STAGES, su = gs % kpu;
        if (!mbar_wait(&b.raw_full[rs], (gu / RAWS) & 1, abort_flag, p.err, 3, limit)) { ok = false; break; }
        if (!mbar_wait(&b.empty[sa], ((gs / STAGES) & 1) ^ 1, abort_flag, p.err, 4, limit)) { ok = false; break; }
        const uint32_t raw = su32(smem + C::OFF_RAW + rs * C::RAW_BYTES);
        const uint32_t a_base = su32(smem + C::OFF_A + sa * A_BYTES);
        if constexpr (FMT == FMT_Q2_K) {
          uint32_t unit[RPW];
          Q2kRowConst rc[RPW];
#pragma unroll
          for (int n = 0; n < RPW; ++n) {
            unit[n] = raw + (wi + WPG * n) * UB;
            rc[n] = q2k_row_const(unit[n]);
          }
          deq_q2k_stage<RPW>(unit, su, a_base, aoff, rc);
        } else {
#pragma unroll
          for (int n = 0; n < RPW; ++n) deq_q80_stage(raw + (wi + WPG * n) * UB, su, a_base, aoff[n]);
        }
        fence_proxy_async();  // the generic-proxy stores must be visible to the tensor core
        __syncwarp();
        if (lane == 0) {
          // (a test of the timeout path withholds one arrival: that stage never becomes full)
          if (!(p.test_stall && blockIdx.x == 0 && gs + 1 == (uint32_t)p.test_stall)) mbar_arrive(&b.full[sa]);
          mbar_arrive(&b.raw_empty[rs]);  // the group's only stage of this unit is done
        }
      }
      if (!ok) break;
      gs0 += n_stages;
    }
  } else {
    // ------------------------------------------------------------------ epilogue
    const int quad = warp & 3;            // TMEM lane quadrant this warp may access
    const int row = 32 * quad + lane;     // slice row = TMEM lane
    int local = 0;
    for (int it = blockIdx.x; it < n_items; it += gridDim.x, ++local) {
      const Item t = item_of<C::BN>(p, it);
      const int buf = local & 1;
      // all four warps enter the item's epilogue (it has named barriers) only together
      if (!named_bar_all(1, 32 * kEpiWarps, mbar_wait(&b.acc_full[buf], (local >> 1) & 1, abort_flag, p.err, 5, limit)))
        break;
      tc_fence_after();
      if (GATEUP) {  // the tile's activation scales, once per item
        for (int i = threadIdx.x - 32 * (kFirstDeq + kDeqWarps); i < t.n; i += 32 * kEpiWarps)
          ibuf[i] = i < t.rows ? __ldg(p.inv_scale + t.row0 + i) : 0.f;
        named_bar(1, 32 * kEpiWarps);
      }
      const uint32_t taddr = tmem + (uint32_t)(buf * ACC_COLS) + ((uint32_t)(32 * quad) << 16);
      for (int c0 = 0; c0 < t.n; c0 += 16) {
        uint32_t r[16];
        tmem_ld16(taddr + c0, r);
        tmem_ld_wait();
        if (GATEUP) {
          // The gate warps (TMEM lanes 0-63) form h for the chunk's first 8 columns, the up warps
          // (lanes 64-127) for the last 8: each hands the other half of its accumulator rows over.
          const int pb = (c0 >> 4) & 1, feat = row & 63;
          float* xg = gbuf + pb * 1024;  // [8][64] g of columns c0+8 .. c0+15
          float* xu = xg + 512;          // [8][64] u of columns c0 .. c0+7
          const bool gate = quad < 2;
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            if (gate) xg[j * 64 + feat] = __uint_as_float(r[8 + j]);
            else xu[j * 64 + feat] = __uint_as_float(r[j]);
          }
          named_bar(1, 32 * kEpiWarps);
          const int cb = c0 + (gate ? 0 : 8);
          unsigned bad = 0;
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const int col = cb + j;
            if (col < t.rows) {
              const float g = gate ? __uint_as_float(r[j]) : xg[j * 64 + feat];
              const float u = gate ? xu[j * 64 + feat] : __uint_as_float(r[8 + j]);
              const float iv = ibuf[col];
              const float h = silu_mul_fast(g * iv, u * iv);
              bad |= !(fabsf(h) <= 65504.f);
              p.h_out[(size_t)(t.row0 + col) * p.ld_out + 64 * t.mt + feat] = __float2half_rn(h);
            }
          }
          if (__any_sync(0xffffffffu, bad) && lane == 0) atomicOr(p.err, 8);
        } else {
          const int drow = 128 * t.mt + row;
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int col = c0 + j;
            if (col < t.rows) p.y_out[(size_t)(t.row0 + col) * p.ld_out + drow] = __uint_as_float(r[j]);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&b.acc_empty[buf]);  // the MMA may overwrite this buffer
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, TMEM_COLS);
}

template <int FMT, bool GATEUP>
cudaError_t launch_one(const ActMaps& tm, const GemmArgs& p, dim3 grid, cudaStream_t s) {
  expert_gemm_tc_kernel<FMT, GATEUP><<<grid, kThreads, Cfg<FMT>::SMEM_BYTES, s>>>(tm.r64, tm.r128, p);
  return cudaGetLastError();
}

template <int FMT, bool GATEUP>
cudaError_t prepare_one() {
  return cudaFuncSetAttribute(expert_gemm_tc_kernel<FMT, GATEUP>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              Cfg<FMT>::SMEM_BYTES);
}

}  // namespace

int gemm_tile_n(int fmt) { return fmt == FMT_Q2_K ? Cfg<FMT_Q2_K>::BN : Cfg<FMT_Q8_0>::BN; }

cudaError_t gemm_prepare() {
  cudaError_t e = prepare_one<FMT_Q2_K, true>();
  if (e == cudaSuccess) e = prepare_one<FMT_Q2_K, false>();
  if (e == cudaSuccess) e = prepare_one<FMT_Q8_0, true>();
  if (e == cudaSuccess) e = prepare_one<FMT_Q8_0, false>();
  return e;
}

// Persistent launch: one CTA per SM (at most), each looping over the (token tile, weight slice)
// items; n_tiles bounds the token tiles (the routed count itself is read on the device).
cudaError_t launch_gemm(int fmt, bool gateup, const ActMaps& tm, const GemmArgs& args, int m_tiles, int n_tiles,
                        cudaStream_t s) {
  static int n_sm[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !n_sm[dev]) cudaDeviceGetAttribute(&n_sm[dev], cudaDevAttrMultiProcessorCount, dev);
  const int sms = (dev >= 0 && dev < 64 && n_sm[dev] > 0) ? n_sm[dev] : 152;
  GemmArgs p = args;
  p.m_tiles = m_tiles;
  const dim3 grid(std::max(1, std::min(sms, m_tiles * n_tiles)));
  if (fmt == FMT_Q2_K) return gateup ? launch_one<FMT_Q2_K, true>(tm, p, grid, s) : launch_one<FMT_Q2_K, false>(tm, p, grid, s);
  return gateup ? launch_one<FMT_Q8_0, true>(tm, p, grid, s) : launch_one<FMT_Q8_0, false>(tm, p, grid, s);
}

// fp16 2D tensor map over a row-major [rows x cols] buffer, boxes of 64 columns x box_rows rows
// with the 128-byte swizzle (the K-major canonical layout of the MMA's B operand).
int make_tmap_f16(CUtensorMap* tm, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
  if (!encode) {
    cudaDriverEntryPointQueryResult q;
    void* fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn)
      return -1;
    encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * 2};
  const cuuint32_t box[2] = {BK, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = encode(tm, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? 0 : -2;
}

int make_act_maps(ActMaps* tm, const void* base, uint64_t rows, uint64_t cols) {
  const int r = make_tmap_f16(&tm->r64, base, rows, cols, BOX_ROWS);
  return r ? r : make_tmap_f16(&tm->r128, base, rows, cols, 2 * BOX_ROWS);
}

}  // namespace ds4
