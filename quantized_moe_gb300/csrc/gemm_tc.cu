// Prefill expert GEMMs on the 5th-generation tensor cores (tcgen05, TMEM accumulators).
//
// Persistent: one CTA per SM loops over work items, each a 128-row x N-token tile of one expert
// (N <= 192 tokens; the MMA's N is the token count rounded up to 16):
//   gate/up: the 128 rows interleave 64 gate rows and the 64 up rows of the same features, so
//            the epilogue forms h = silu(g) * u for 64 features and writes it as fp16;
//   down:    128 rows of d, written as fp32 per bucketed slot for the fixed-order combine.
// The dequantized weight tile (the MMA's A operand) never touches shared memory: the dequant
// warps write it into tensor memory (tcgen05.st) and the MMA reads A from there and only the
// activation tile (B) from shared memory. Tensor memory holds two fp32 accumulators of 192
// columns (the epilogue of one item overlaps the main loop of the next) and two pipeline stages of
// A (128 k = 64 columns each); shared memory holds three activation stages and the packed weight
// units. A pipeline stage is two 64-k sub-tiles (one 128-byte swizzle span each) and carries eight
// MMAs per barrier wait and commit: the MMA thread's loop of barrier operations, more than the
// tensor pipe, bounds the stage rate. The A stages have their own full barrier (the two dequant
// groups that wrote the sub-tiles) and empty barrier (MMA commit), and so have the activation
// stages (TMA bytes; MMA commit), so that the activation ring can run a stage further ahead.
// With an even number of weight slices the CTAs run in clusters of two on adjacent slices of the
// same token tile and each loads half of every activation stage, multicast to both.
// Warp roles (23 warps):
//   warp 0     weight producer: bulk-copies the packed weight units of each K unit (256 k for
//              Q2_K, 128 k for Q8_0) of the tile's rows;
//   warp 1     allocates TMEM; the converged warp runs the MMA loop and one elected lane issues
//              the tcgen05.mma and commits of every stage;
//   warp 2     activation producer: TMA-loads the fp16 activation sub-tiles (128-byte swizzle)
//              of each stage, exactly the MMA's N rows, in boxes of 128, 64, 32 and 16 rows
//              issued by parallel lanes (one thread issuing them in turn was the critical path);
//   warps 3-18 dequantize, in four groups of four warps taking the 64-k sub-tiles round-robin.
//              A warp may only access its TMEM lane quadrant (warp % 4), so the four warps of a
//              group cover the tile's 128 rows, one row per thread: the thread reads its row's
//              quants and scales of the sub-tile from shared memory, forms the 64 fp16 weights
//              (exact small-integer quants, one fp16 FMA with the sub-block scale and min) and
//              stores them as 32 columns of its TMEM lane;
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

constexpr int BM = 128, BK = 64;  // BK: K of one 128-byte swizzled sub-tile (64 fp16)
constexpr int kDeqWarps = 16;
constexpr int kDeqGroups = 4;  // groups of four warps (one per TMEM lane quadrant)
constexpr int kFirstDeq = 3;   // warps 0-2: weight producer, MMA, activation producer
constexpr int kEpiWarps = 4;   // warps 19-22: epilogue, one per TMEM lane quadrant
constexpr int kThreads = (kFirstDeq + kDeqWarps + kEpiWarps) * 32;  // 736
constexpr int TMEM_COLS = 512;

// Two tile geometries, chosen per forward (gemm_geometry): token tile BN (the MMA's N at most),
// sub-tiles per pipeline stage SUB, activation stages and raw weight units in flight.
//   0 (wide):  BN = 192, SUB = 2: for batches whose experts average 64 tokens or more;
//   1 (small): BN = 128, SUB = 4: 16 MMAs per barrier wait and commit. With few tokens per expert
//              the MMA warp's per-stage loop, not the tensor pipe or HBM, bounds a stage, and a
//              256-k stage halves the number of stages (measured: decode-16 gate/up 0.197 ->
//              0.172 ms, prefill-512 0.452 -> 0.427 ms; prefill-4096 would lose 28 %: experts
//              above 128 tokens would be dequantized twice).
template <int GEOM>
struct Geo;
template <>
struct Geo<0> {
  static constexpr int BN = 192, SUB = 2, BS_Q2K = 3, BS_Q80 = 3;
};
template <>
struct Geo<1> {
  static constexpr int BN = 128, SUB = 4, BS_Q2K = 2, BS_Q80 = 2;
};

template <int FMT, int GEOM>
struct Cfg {
  static constexpr int BN = Geo<GEOM>::BN;      // token tile
  static constexpr int SUB = Geo<GEOM>::SUB;    // 64-k sub-tiles per pipeline stage
  static constexpr int SK = SUB * BK;           // K of one pipeline stage
  // Tensor memory: two accumulators of BN fp32 columns, then the A stages (SK of fp16 = SK / 2
  // columns) in the columns left over.
  static constexpr int ACC_COLS = BN;
  static constexpr int A_COLS = SK / 2;
  static constexpr int A_COL0 = 2 * ACC_COLS;
  static constexpr int A_STAGES = (TMEM_COLS - A_COL0) / A_COLS < 8 ? (TMEM_COLS - A_COL0) / A_COLS : 8;
  static_assert(A_STAGES >= 2 && A_COL0 + A_STAGES * A_COLS <= TMEM_COLS, "tensor memory budget");
  static constexpr int RAW_BYTES = 8 * unit_bytes(FMT);  // one K unit of the 128-row tile
  static constexpr int RAWS = 4;                         // K units in flight
  static constexpr int SUB_BYTES = BN * BK * 2;          // one 64-k activation sub-tile
  static constexpr int B_BYTES = SUB * SUB_BYTES;
  // activation stages: more than the A stages where shared memory allows, so that the TMA of a
  // stage is issued well before the MMA needs it (an L2 read under load takes ~a thousand cycles)
  static constexpr int B_STAGES = FMT == FMT_Q2_K ? Geo<GEOM>::BS_Q2K : Geo<GEOM>::BS_Q80;
  static constexpr int OFF_B = 0;
  static constexpr int OFF_RAW = OFF_B + B_STAGES * B_BYTES;
  static_assert(BN <= 256 && BN % 16 == 0, "token tile");
  static constexpr int OFF_BAR = OFF_RAW + RAWS * RAW_BYTES;
  static constexpr int N_BARS = 2 * A_STAGES + 2 * B_STAGES + 2 * RAWS + 4;
  static constexpr int OFF_MISC = OFF_BAR + N_BARS * 8;
  static constexpr int OFF_GBUF = (OFF_MISC + 16 + 15) / 16 * 16;
  // gate/up epilogue: two parities x (8 columns of g + 8 columns of u) x 64 features fp32, then the
  // 1 / scale of each token of the tile
  static constexpr int GBUF_BYTES = 2 * 2 * 8 * 64 * 4 + 256 * 4;
  static constexpr int SMEM_BYTES = OFF_GBUF + GBUF_BYTES + 1024;  // + alignment slack
  static_assert(SMEM_BYTES <= 232448, "shared memory budget");
};

struct Bars {
  uint64_t* a_full;     // [A_STAGES] the dequant groups' warps -> MMA
  uint64_t* a_empty;    // [A_STAGES] MMA commit -> dequant groups
  uint64_t* b_full;     // [B_STAGES] activation TMA (with its bytes) -> MMA
  uint64_t* b_empty;    // [B_STAGES] MMA commits of every CTA of the cluster -> activation producer
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

// One row of one K stage of a Q2_K unit: 64 fp16 weights as 32 columns, column 8i + kp holding
// k = 16i + 2kp and k + 1 of the stage (sub-block i = 0..3, k-pair kp = 0..7). The stage is half
// H of chunk c; its sub-blocks are fields 4H .. 4H + 3 of the row's eight k-pair words.
// Each field is shifted to bits 8-9 of its half: as an fp16 subnormal that is q * 2^-16, and the
// sub-block scale carries 2^16 d * s (exact: only the exponent changes; create refuses
// super-blocks whose 2^16 d * 15 would leave the fp16 range), so one FMA with the min gives
// d s q - dmin m rounded once.
template <int H>
__device__ __forceinline__ void deq_q2k_row(uint32_t unit, int c, int g, int ah, uint32_t (&v)[32]) {
  const int sw = (g >> 1) & 3;
  uint32_t w[8];  // k-pair kp of this row: the chunk's eight sub-blocks, 2 bits each per half
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    const uint2 x = lds64(unit + c * 512 + 16 * (4 * g + (t ^ sw)) + 8 * ah);
    w[t] = x.x;
    w[t + 4] = x.y;
  }
  // scale words 2H and 2H + 1 of the chunk hold sub-blocks 4H .. 4H + 3 in bytes 2ah, 2ah + 1
  const uint4 scw = lds128(unit + kQ2kScOff + c * 128 + 16 * g);
  const uint32_t dd = lds32(unit + kQ2kDdOff + 4 * (g + 8 * ah));  // fp16 d, dmin of the row
  const __half2 k256 = __float2half2_rn(256.f), k1024 = __float2half2_rn(1024.f);
  const __half2 d16 = __hmul2(__hmul2(__low2half2(u2h(dd)), k256), k256);
  const __half2 dm = __high2half2(u2h(dd));
  const __half2 ndm = __hneg2(dm), dm1024 = __hmul2(dm, k1024);
  const uint32_t sel = ah ? 0x4342u : 0x4140u;
  __half2 ds[4], nm[4];
#pragma unroll
  for (int p = 0; p < 2; ++p) {
    const uint32_t sc = prmt(p == 0 ? (H ? scw.z : scw.x) : (H ? scw.w : scw.y), 0u, sel);  // (sub 2p, sub 2p+1)
    const __half2 s2 = __hmul2(__hsub2(u2h((sc & 0x000F000Fu) | 0x64006400u), k1024), d16);
    const __half2 m2 = __hfma2(u2h(((sc >> 4) & 0x000F000Fu) | 0x64006400u), ndm, dm1024);
    ds[2 * p] = __low2half2(s2);
    ds[2 * p + 1] = __high2half2(s2);
    nm[2 * p] = __low2half2(m2);
    nm[2 * p + 1] = __high2half2(m2);
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int f = 4 * H + i;        // field of sub-block i in the k-pair words
    const int sh = 8 - 2 * f;       // left shift to bits 8-9 (negative: right)
#pragma unroll
    for (int kp = 0; kp < 8; ++kp) {
      const uint32_t qb = (sh >= 0 ? (w[kp] << sh) : (w[kp] >> -sh)) & 0x03000300u;
      v[8 * i + kp] = h2u(__hfma2(u2h(qb), ds[i], nm[i]));
    }
  }
}

// One row of one K stage (half H of the unit: 32-k blocks 2H, 2H + 1) of a Q8_0 unit, in the
// column order of deq_q2k_row: fp16 (1024 + u) by byte permutation, minus 1152 gives q exactly,
// times the block scale.
template <int H>
__device__ __forceinline__ void deq_q80_row(uint32_t unit, int g, int ah, uint32_t (&v)[32]) {
  const int sw = (g >> 1) & 3;
  const uint2 scw = lds64(unit + kQ80ScOff + 16 * g + 8 * H);  // blocks 2H, 2H+1: (row g, row g+8)
  const __half2 k1152 = __float2half2_rn(1152.f);
#pragma unroll
  for (int jl = 0; jl < 2; ++jl) {
    const uint32_t sw32 = jl == 0 ? scw.x : scw.y;
    const __half2 s = ah ? __high2half2(u2h(sw32)) : __low2half2(u2h(sw32));
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const uint2 x = lds64(unit + 512 * (2 * H + jl) + 16 * (4 * g + (t ^ sw)) + 8 * ah);
      // x.x: sub-block 2j, x.y: sub-block 2j + 1; bytes k = 2t, 2t+1, 2t+8, 2t+9
      const uint32_t raw[4] = {prmt(x.x, 0x64u, 0x4140u), prmt(x.x, 0x64u, 0x4342u), prmt(x.y, 0x64u, 0x4140u),
                               prmt(x.y, 0x64u, 0x4342u)};
      const int col[4] = {16 * jl + t, 16 * jl + t + 4, 16 * jl + 8 + t, 16 * jl + 12 + t};
#pragma unroll
      for (int e = 0; e < 4; ++e) v[col[e]] = h2u(__hmul2(__hsub2(u2h(raw[e]), k1152), s));
    }
  }
}

// Waits (bounded, without raising errors) for a phase: used only to let copies land, or issued MMAs
// finish, before the CTA exits.
__device__ __forceinline__ void bounded_try(uint64_t* bar, uint32_t parity, long long limit) {
  const long long t0 = clock64();
  while (!mbar_try(bar, parity) && clock64() - t0 < limit) {
  }
}

// mbar_wait by every lane of a converged warp: no divergent branch and no shuffle to hand the
// result over (a lane-0 wait plus shuffle cost the MMA loop about 100 cycles per stage).
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag, int* err, int site,
                                          long long limit) {
  return mbar_wait(bar, parity, abort_flag, err, site, limit);
}

// The tile of work item `it` (token tile, 128-row slice of the weights): the MMA's N (the
// activation rows loaded and the accumulator columns the epilogue reads) is the row count rounded
// up to the instruction's granularity of 16.
struct Item {
  int expert, row0, rows, n, mt;
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

// CS = 1, or the size (2 or 4) of a cluster of CTAs that take adjacent weight slices of the same
// token tile (items CS c + r + k G, r < CS, the weight slices fastest and their count a multiple
// of CS): each loads its share of the rows of every activation stage and multicasts it to all,
// and each MMA commit releases the stage in all of them, so the activation tile crosses L2 once
// per cluster.
template <int FMT, bool GATEUP, int CS, int GEOM>
__global__ void __launch_bounds__(kThreads, 1) expert_gemm_tc_kernel(const __grid_constant__ CUtensorMap tmap16,
                                                                      const __grid_constant__ CUtensorMap tmap32,
                                                                      const __grid_constant__ CUtensorMap tmap64,
                                                                      const __grid_constant__ CUtensorMap tmap128,
                                                                      GemmArgs p) {
  using C = Cfg<FMT, GEOM>;
  constexpr int SUB = C::SUB, SK = C::SK, A_STAGES = C::A_STAGES, A_COLS = C::A_COLS, A_COL0 = C::A_COL0;
  constexpr int ACC_COLS = C::ACC_COLS;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr int UK = unit_k(FMT), UB = unit_bytes(FMT), RAWS = C::RAWS, BS = C::B_STAGES;
  constexpr int kpu = UK / BK;  // 64-k sub-tiles per raw unit: Q2_K four, Q8_0 two
  const int n_kb = p.k / UK, n_stages = p.k / SK, n_subs = p.k / BK;
  const int n_items = item_count<C::BN>(p);
  // gate/up: 64 gate rows then the 64 up rows of features 64 mt .. 64 mt + 63; down: 128 rows of d
  const uint32_t raw_copy = GATEUP ? 4 * UB : 8 * UB;
  const long long limit = p.timeout_cycles > 0 ? p.timeout_cycles : kTimeoutCycles;

  Bars b;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  b.a_full = bars;
  b.a_empty = b.a_full + A_STAGES;
  b.b_full = b.a_empty + A_STAGES;
  b.b_empty = b.b_full + BS;
  b.raw_full = b.b_empty + BS;
  b.raw_empty = b.raw_full + RAWS;
  b.acc_full = b.raw_empty + RAWS;  // [2]
  b.acc_empty = b.acc_full + 2;     // [2]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
  float* gbuf = reinterpret_cast<float*>(smem + C::OFF_GBUF);
  float* ibuf = gbuf + 2048;

  if (threadIdx.x == 0) {
    for (int i = 0; i < A_STAGES; ++i) {
      mbar_init(&b.a_full[i], SUB * (kDeqWarps / kDeqGroups));  // four warps per sub-tile
      mbar_init(&b.a_empty[i], 1);
    }
    for (int i = 0; i < BS; ++i) {
      mbar_init(&b.b_full[i], 1);
      mbar_init(&b.b_empty[i], CS);  // the MMA commit of every CTA of the cluster
    }
    for (int r = 0; r < RAWS; ++r) {
      mbar_init(&b.raw_full[r], 1);
      mbar_init(&b.raw_empty[r], (kDeqWarps / kDeqGroups) * kpu);  // every warp of the unit's kpu stages
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
  if (CS > 1)
    cluster_sync();  // the peer's barriers are initialized before any multicast reaches them
  else
    __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int rank = CS > 1 ? (int)cluster_ctarank() : 0;
  if (warp == 2 && lane == 0) {  // the activation producer's descriptors, ahead of its first loads
    tmap_prefetch(&tmap16);
    tmap_prefetch(&tmap32);
    tmap_prefetch(&tmap64);
    tmap_prefetch(&tmap128);
  }
  constexpr uint16_t kMask = (uint16_t)((1u << CS) - 1u);

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
    // The warp waits for a free stage together; lane 0 announces the stage's bytes and lane 8j + q
    // issues box q of sub-tile j: the CTA's rows [lo, hi) of the MMA's N rows as boxes of 128,
    // 128, 64, 32 and 16 rows (those the length needs), so that all of a stage's loads go out in
    // one instruction instead of one after another from a single thread.
    uint32_t gs = 0;  // stages issued over all items
    const int j = lane >> 3, q = lane & 7;
    for (int it = blockIdx.x; it < n_items && !*abort_flag; it += gridDim.x) {
      const Item t = item_of<C::BN>(p, it);
      const int rows = t.n;  // all of them land in this CTA
      const int lo = 16 * ((rows / 16) * rank / CS), hi = 16 * ((rows / 16) * (rank + 1) / CS);
      const int len = hi - lo, n128 = len / 128, rem = len - 128 * n128;
      int r = -1;
      const CUtensorMap* map = &tmap16;
      if (q < 2) {
        if (q < n128) r = lo + 128 * q, map = &tmap128;
      } else if (q == 2) {
        if (rem & 64) r = lo + 128 * n128, map = &tmap64;
      } else if (q == 3) {
        if (rem & 32) r = lo + 128 * n128 + (rem & 64), map = &tmap32;
      } else if (q == 4) {
        if (rem & 16) r = lo + 128 * n128 + (rem & 96), map = &tmap16;
      }
      const bool issue = j < SUB && r >= 0;
      for (int sB = 0; sB < n_stages; ++sB, ++gs) {
        const int sb = gs % BS;
        if (!warp_wait(&b.b_empty[sb], ((gs / BS) & 1) ^ 1, abort_flag, p.err, 2, limit)) break;
        if (lane == 0) mbar_expect_tx(&b.b_full[sb], SUB * rows * BK * 2);
        if (issue) {
          unsigned char* dst = smem + C::OFF_B + sb * C::B_BYTES + j * C::SUB_BYTES + r * BK * 2;
          const int x = (sB * SUB + j) * BK;
          if (CS > 1)
            tma_load_2d_mc(dst, map, x, t.row0 + r, &b.b_full[sb], kMask);
          else
            tma_load_2d(dst, map, x, t.row0 + r, &b.b_full[sb]);
        }
      }
    }
    if (lane == 0)
      for (uint32_t k = gs > (uint32_t)BS ? gs - BS : 0; k < gs; ++k)
        bounded_try(&b.b_full[k % BS], (k / BS) & 1, limit);
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    // The whole warp runs the loop and polls the barriers; one elected lane issues.
    uint32_t gs = 0;
    int local = 0;  // items of this CTA so far: accumulator buffer local & 1
    for (int it = blockIdx.x; it < n_items && !*abort_flag; it += gridDim.x, ++local) {
      const Item t = item_of<C::BN>(p, it);
      const int buf = local & 1;
      // the epilogue has drained this buffer (item local - 2)
      if (!warp_wait(&b.acc_empty[buf], ((local >> 1) & 1) ^ 1, abort_flag, p.err, 6, limit)) break;
      tc_fence_after();
      const uint32_t idesc = idesc_f16_f32(BM, t.n);
      const uint32_t acc = tmem + (uint32_t)(buf * ACC_COLS);
      bool ok = true;
      for (int s = 0; s < n_stages; ++s, ++gs) {
        const int st = gs % A_STAGES;
        const int sb = gs % BS;
        if (!warp_wait(&b.b_full[sb], (gs / BS) & 1, abort_flag, p.err, 7, limit) ||
            !warp_wait(&b.a_full[st], (gs / A_STAGES) & 1, abort_flag, p.err, 7, limit)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t ta = tmem + (uint32_t)(A_COL0 + st * A_COLS);
        const uint32_t bsm = su32(smem + C::OFF_B + sb * C::B_BYTES);
        // 16 fp16 of K per MMA: 8 TMEM columns of A, 32 bytes of a B sub-tile; blocks of eight
        static_assert(SUB % 2 == 0, "the stage's MMAs are issued in blocks of eight (two sub-tiles)");
#pragma unroll
        for (int h = 0; h < SUB / 2; ++h)
          tc_mma8_ts_elect(acc, ta + 64 * h, sw128_desc(bsm + 2 * h * C::SUB_BYTES),
                           sw128_desc(bsm + (2 * h + 1) * C::SUB_BYTES), idesc, (s | h) != 0);
        tc_commit2_elect(&b.b_empty[sb], CS > 1 ? kMask : 0, &b.a_empty[st]);
      }
      if (!ok) break;
      tc_commit_elect(&b.acc_full[buf]);
    }
    // The MMAs already issued must finish before TMEM is freed (after an abort), and in a cluster
    // every commit of both CTAs must have reached its barriers before either CTA exits: the
    // last stage's empty phase completes only then.
    if ((*abort_flag || CS > 1) && gs > 0 && lane == 0)
      bounded_try(&b.b_empty[(gs - 1) % BS], ((gs - 1) / BS) & 1, limit);
    __syncwarp();
  } else if (warp < kFirstDeq + kDeqWarps) {
    // ------------------------------------------------------------------ dequant
    // Four groups of four warps take the CTA's 64-k sub-tiles round-robin: group g dequantizes the
    // sub-tiles gs = g (mod 4), sub-tile gs % SUB of pipeline stage gs / SUB. Warp w accesses TMEM
    // lanes 32 (w % 4) .. + 31, and a group's four consecutive warps cover all four quadrants; a
    // thread owns tile row = its lane.
    const int dw = warp - kFirstDeq;
    const int grp = dw / (kDeqWarps / kDeqGroups);
    const int quad = warp & 3;
    const int row = 32 * quad + lane;                      // tile row = TMEM lane
    const int rho = row & 15, g = rho & 7, ah = rho >> 3;  // row inside its 16-row unit
    const uint32_t t_q = tmem + ((uint32_t)(32 * quad) << 16) + (uint32_t)A_COL0;
    uint32_t gs0 = 0;  // sub-tiles of the CTA's earlier items
    for (int it = blockIdx.x; it < n_items && !*abort_flag; it += gridDim.x) {
      bool ok = true;
      for (int s = (grp - (int)(gs0 % kDeqGroups) + kDeqGroups) % kDeqGroups; s < n_subs; s += kDeqGroups) {
        const uint32_t gs = gs0 + s;
        const uint32_t gu = gs / kpu;  // the raw units follow the sub-tiles
        const int rs = gu % RAWS, su = gs % kpu;
        if (!mbar_wait(&b.raw_full[rs], (gu / RAWS) & 1, abort_flag, p.err, 3, limit)) { ok = false; break; }
        const uint32_t ps = gs / SUB;  // pipeline stage
        const int sa = ps % A_STAGES;
        if (!mbar_wait(&b.a_empty[sa], ((ps / A_STAGES) & 1) ^ 1, abort_flag, p.err, 4, limit)) { ok = false; break; }
        tc_fence_after();
        const uint32_t unit = su32(smem + C::OFF_RAW + rs * C::RAW_BYTES) + (row >> 4) * UB;
        uint32_t v[32];
        if constexpr (FMT == FMT_Q2_K) {
          if (su & 1)
            deq_q2k_row<1>(unit, su >> 1, g, ah, v);
          else
            deq_q2k_row<0>(unit, su >> 1, g, ah, v);
        } else {
          if (su & 1)
            deq_q80_row<1>(unit, g, ah, v);
          else
            deq_q80_row<0>(unit, g, ah, v);
        }
        tmem_st32(t_q + (uint32_t)(sa * A_COLS + (gs % SUB) * (BK / 2)), v);
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          // (a test of the timeout path withholds one arrival: that stage never becomes full)
          if (!(p.test_stall && blockIdx.x == 0 && gs + 1 == (uint32_t)p.test_stall)) mbar_arrive(&b.a_full[sa]);
          mbar_arrive(&b.raw_empty[rs]);
        }
      }
      if (!ok) break;
      gs0 += n_subs;
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
  if (CS > 1)
    cluster_sync();  // no copy or commit of either CTA still targets the other's shared memory
  else
    __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, TMEM_COLS);
}

template <int FMT, bool GATEUP, int CS, int GEOM>
cudaError_t launch_one(const ActMaps& tm, const GemmArgs& p, int grid, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = Cfg<FMT, GEOM>::SMEM_BYTES;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CS;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = CS > 1 ? 1 : 0;  // a plain launch without clusters
  return cudaLaunchKernelEx(&cfg, expert_gemm_tc_kernel<FMT, GATEUP, CS, GEOM>, tm.r16, tm.r32, tm.r64, tm.r128, p);
}

// Clusters of CS CTAs that can be resident at once (0 if none).
template <int FMT, bool GATEUP, int CS, int GEOM>
int max_clusters() {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * CS);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = Cfg<FMT, GEOM>::SMEM_BYTES;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CS;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, expert_gemm_tc_kernel<FMT, GATEUP, CS, GEOM>, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

template <int FMT, bool GATEUP, int CS, int GEOM>
cudaError_t prepare_one() {
  return cudaFuncSetAttribute(expert_gemm_tc_kernel<FMT, GATEUP, CS, GEOM>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<FMT, GEOM>::SMEM_BYTES);
}

// Per device, geometry and (format, gate/up or down) kernel: resident clusters of two and four.
int g_pairs[64][2][4], g_quads[64][2][4];

template <int FMT, bool GATEUP, int GEOM>
cudaError_t prepare_fmt(int dev, int k) {
  cudaError_t e = prepare_one<FMT, GATEUP, 1, GEOM>();
  if (e == cudaSuccess) e = prepare_one<FMT, GATEUP, 2, GEOM>();
  if (e == cudaSuccess) e = prepare_one<FMT, GATEUP, 4, GEOM>();
  if (e == cudaSuccess && dev >= 0 && dev < 64) {
    g_pairs[dev][GEOM][k] = max_clusters<FMT, GATEUP, 2, GEOM>();
    g_quads[dev][GEOM][k] = max_clusters<FMT, GATEUP, 4, GEOM>();
  }
  return e;
}

template <int GEOM>
cudaError_t prepare_geom(int dev) {
  cudaError_t e = prepare_fmt<FMT_Q2_K, true, GEOM>(dev, 0);
  if (e == cudaSuccess) e = prepare_fmt<FMT_Q2_K, false, GEOM>(dev, 1);
  if (e == cudaSuccess) e = prepare_fmt<FMT_Q8_0, true, GEOM>(dev, 2);
  if (e == cudaSuccess) e = prepare_fmt<FMT_Q8_0, false, GEOM>(dev, 3);
  return e;
}

template <int CS, int GEOM>
cudaError_t launch_cs(int fmt, bool gateup, const ActMaps& tm, const GemmArgs& p, int grid, cudaStream_t s) {
  if (fmt == FMT_Q2_K)
    return gateup ? launch_one<FMT_Q2_K, true, CS, GEOM>(tm, p, grid, s)
                  : launch_one<FMT_Q2_K, false, CS, GEOM>(tm, p, grid, s);
  return gateup ? launch_one<FMT_Q8_0, true, CS, GEOM>(tm, p, grid, s) : launch_one<FMT_Q8_0, false, CS, GEOM>(tm, p, grid, s);
}

template <int GEOM>
cudaError_t launch_geom(int fmt, bool gateup, const ActMaps& tm, const GemmArgs& p, int items, int m_tiles, int sms,
                        int dev, cudaStream_t s) {
  const bool known = dev >= 0 && dev < 64;
  const int k = (fmt == FMT_Q2_K ? 0 : 2) + (gateup ? 0 : 1);
  const int quads = known ? g_quads[dev][GEOM][k] : 0, pairs = known ? g_pairs[dev][GEOM][k] : 0;
  if (!p.tiles && m_tiles % 4 == 0 && quads > 0)
    return launch_cs<4, GEOM>(fmt, gateup, tm, p, 4 * std::max(1, std::min(quads, items / 4)), s);
  if (m_tiles % 2 == 0 && pairs > 0)
    return launch_cs<2, GEOM>(fmt, gateup, tm, p, 2 * std::max(1, std::min(pairs, items / 2)), s);
  return launch_cs<1, GEOM>(fmt, gateup, tm, p, std::max(1, std::min(sms, items)), s);
}

}  // namespace

int gemm_tile_n(int geom) { return geom ? Geo<1>::BN : Geo<0>::BN; }

int gemm_geometry(int n_tokens, int top_k, int n_experts, int k_gcd) {
  // fewer than 64 tokens per expert on average, and every K a multiple of the 256-k stage
  return (int64_t)n_tokens * top_k < 64ll * n_experts && k_gcd % (Geo<1>::SUB * BK) == 0 ? 1 : 0;
}

cudaError_t gemm_prepare() {
  int dev = 0;
  cudaGetDevice(&dev);
  cudaError_t e = prepare_geom<0>(dev);
  if (e == cudaSuccess) e = prepare_geom<1>(dev);
  return e;
}

// Persistent launch: one CTA per SM (at most), each looping over the (token tile, weight slice)
// items; n_tiles bounds the token tiles (the routed count itself is read on the device). When the
// weight slices divide evenly, the CTAs run in clusters that share the activation loads: of four
// for the dense (shared expert) GEMMs, of two for the routed ones (measured: clusters of four leave
// more SMs idle than the routed GEMMs gain from the smaller activation traffic).
cudaError_t launch_gemm(int fmt, bool gateup, const ActMaps& tm, const GemmArgs& args, int m_tiles, int n_tiles,
                        int geom, cudaStream_t s) {
  static int n_sm[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  const bool known = dev >= 0 && dev < 64;
  if (known && !n_sm[dev]) cudaDeviceGetAttribute(&n_sm[dev], cudaDevAttrMultiProcessorCount, dev);
  const int sms = (known && n_sm[dev] > 0) ? n_sm[dev] : 152;
  GemmArgs p = args;
  p.m_tiles = m_tiles;
  const int items = m_tiles * n_tiles;
  return geom ? launch_geom<1>(fmt, gateup, tm, p, items, m_tiles, sms, dev, s)
              : launch_geom<0>(fmt, gateup, tm, p, items, m_tiles, sms, dev, s);
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
  int r = make_tmap_f16(&tm->r16, base, rows, cols, 16);
  if (!r) r = make_tmap_f16(&tm->r32, base, rows, cols, 32);
  if (!r) r = make_tmap_f16(&tm->r64, base, rows, cols, 64);
  return r ? r : make_tmap_f16(&tm->r128, base, rows, cols, 128);
}

}  // namespace ds4
