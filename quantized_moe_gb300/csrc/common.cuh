// Shared definitions of the ds4moe CUDA library: repacked weight layouts, launch helpers
// and the warp-level MMA wrapper. Device code targets sm_103a only.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <cuda_bf16.h>
#include <stdint.h>

namespace ds4 {

// ----------------------------------------------------------------------------- layouts
//
// Quantized matrices are repacked at create time into "units" of 16 rows (a row-group)
// by one K-chunk, ordered tile-major: [row-tile of 128 rows][K-unit][row-group in tile][unit].
// The layout serves two readers: a warp of the decode GEMV, where lane L = 4g + t loads the bits
// of its m16n8k16 A fragments as one coalesced 16-byte piece ("region") per chunk, and a thread of
// the prefill GEMM, which dequantizes one whole row and reads that row's half of a region (8
// bytes) from shared memory. Region 4g + t of a chunk lies at position lane_region(g, t), which
// permutes the four regions of each g so that the 8-byte row reads of a half-warp hit 32 distinct
// banks; a warp's 16-byte loads still cover the chunk's 512 bytes exactly.
//
// Fragment map of mma.m16n8k16 (lane = 4*g + t): A register r holds row g + 8*(r&1) at
// k = 2t + 8*(r>>1) (low half) and k+1 (high half); B register r holds k = 2t + 8*r (+1)
// of column g; C element c holds row g + 8*(c>>1), column 2t + (c&1).
//
// Q2_K unit = 16 rows x 256 k (one super-block per row), 1344 bytes:
//   [0, 1024)    quants of k-chunk 0 then k-chunk 1 (128 k each). Region (g, t) of a chunk holds
//                4 words (row g, k-pair t), (row g, k-pair t+4), (row g+8, k-pair t),
//                (row g+8, k-pair t+4): A registers 0, 2, 1, 3. A word holds, for sub-block
//                i = 0..7 of the chunk, the 2-bit q at k = 16i + 2 * (k-pair) in bits [2i, 2i+2)
//                (low half) and of k+1 in bits [16+2i, 18+2i) (high half).
//   [1024, 1280) scale bytes of chunk 0 then chunk 1, lane L owns bytes [4L, 4L+4):
//                (row g, sub 2t), (row g, sub 2t+1), (row g+8, sub 2t), (row g+8, sub 2t+1),
//                sub counted inside the chunk; each byte keeps s in the low nibble, m high.
//   [1280, 1344) row r (0..15): fp16 d, fp16 dmin.
// Q8_0 unit = 16 rows x 128 k (four blocks per row), 2176 bytes:
//   [0, 2048)    u = q + 128 as bytes, one 512-byte piece per 32-k block j (sub-blocks 2j,
//                2j+1). Region (g, t) of block j holds 4 words: (row g, sub 2j), (row g,
//                sub 2j+1), (row g+8, sub 2j), (row g+8, sub 2j+1), each with the bytes of
//                k = 2t, 2t+1, 2t+8, 2t+9 of its sub-block.
//   [2048, 2176) lane L owns bytes [4L, 4L+4): fp16 scale of (row g, block t), (row g+8, block t).
constexpr int kRowGroup = 16;
constexpr int kTileRows = 128;
constexpr int kQ2kUnitK = 256;
constexpr int kQ2kUnitBytes = 1344;
constexpr int kQ2kScOff = 1024;
constexpr int kQ2kDdOff = 1280;
constexpr int kQ80UnitK = 128;
constexpr int kQ80UnitBytes = 2176;
constexpr int kQ80ScOff = 2048;

enum Fmt : int { FMT_Q8_0 = 0, FMT_Q2_K = 1 };

__host__ __device__ constexpr int unit_k(int fmt) { return fmt == FMT_Q2_K ? kQ2kUnitK : kQ80UnitK; }
__host__ __device__ constexpr int unit_bytes(int fmt) { return fmt == FMT_Q2_K ? kQ2kUnitBytes : kQ80UnitBytes; }
__host__ __device__ constexpr int canon_block(int fmt) { return fmt == FMT_Q2_K ? 256 : 32; }
__host__ __device__ constexpr int canon_block_bytes(int fmt) { return fmt == FMT_Q2_K ? 84 : 34; }

// Position (in 16-byte regions) of region (g, t) inside a 512-byte chunk of quants.
__host__ __device__ constexpr int lane_region(int g, int t) { return 4 * g + (t ^ ((g >> 1) & 3)); }

// Byte offset of unit (row-group rg, K-unit kb) in a repacked matrix with n_kb K-units.
__host__ __device__ inline size_t unit_offset(int rg, int kb, int n_kb, int ubytes) {
  const int tile = rg >> 3, rgi = rg & 7;
  return ((size_t)(tile * n_kb + kb) * 8 + rgi) * (size_t)ubytes;
}

// Bytes of one repacked (or canonical: the sizes agree) [rows x k] matrix.
__host__ __device__ inline size_t matrix_bytes(int fmt, int rows, int k) {
  return (size_t)rows * (size_t)(k / canon_block(fmt)) * canon_block_bytes(fmt);
}

// ----------------------------------------------------------------------------- device helpers

__device__ __forceinline__ void mma_f16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint4 ldg_nc_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ uint32_t ldg_nc_u32(const void* p) {
  uint32_t v;
  asm volatile("ld.global.nc.L1::no_allocate.u32 %0, [%1];\n" : "=r"(v) : "l"(p));
  return v;
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;\n" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
  return r;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Power-of-two scale that maps a row maximum into [2^14, 2^15) so the row converts to fp16
// without overflow; exact (only the exponent changes). Returns 1 for an all-zero row.
__device__ __forceinline__ float fp16_row_scale(float amax) {
  if (!(amax > 0.f) || !isfinite(amax)) return 1.f;
  int e;
  frexpf(amax, &e);  // amax = m * 2^e, m in [0.5, 1)
  return ldexpf(1.f, 15 - e);
}

__device__ __forceinline__ float silu_mul(float g, float u) { return g / (1.f + expf(-g)) * u; }

}  // namespace ds4

// ----------------------------------------------------------------------------- host launchers
// (defined in the kernel translation units, called by the C-ABI shim)

namespace ds4 {

// Everything the three decode kernels read and write (device pointers).
struct DecodeArgs {
  const __nv_bfloat16* x;
  int n_tok, d;
  const float* wr;
  const float* br;
  int n_exp, top_k;
  const int* token_ids;
  int n_hash;
  const int* table;
  int vocab;
  float* logits;      // [n_learned x E]
  float* xmax;        // [n_tok] max |x| per token
  int* idx;           // [n_tok x top_k]
  float* wts;
  int* counts;        // [E]
  int* offsets;       // [E+1]
  int* active;        // [E]
  int* n_active;
  int* perm;          // [n_tok x top_k]
  int* rowof;
  int4* work;         // [E] per active expert: expert's weight slot, first bucketed position, count (0 past n_active)
  const int* local_of;  // [E] weight slot of each expert, -1 if the handle does not hold it; null: slot = id
  int* tokof;         // [n_tok x top_k] token of each bucketed position
  float* xscale;      // [n_tok] power-of-two fp16 scale of each token
  int* err;
  unsigned int* counter;  // arrival counter of the route kernel, zero between forwards
  float* hmax;        // [n_tok x top_k] max |h| per routed slot position
  float* hsg;         // [n_tok][fs / 16] max |h| of the shared expert per token and 16-row group
  const uint8_t* gate;
  const uint8_t* up;
  const uint8_t* down;
  size_t mb_gu, mb_d;
  int f;
  const uint8_t* sgate;
  const uint8_t* sup;
  const uint8_t* sdown;
  size_t mb_sgu, mb_sd;
  int fs, n_shared;
  float* H;           // [n_tok x top_k x f] by bucketed position
  float* Hs;          // [n_tok x fs]
  float* out;         // [n_tok x d]
};

// Optional callback after each launch (per-launch timing).
struct DecodeHooks {
  void (*mark)(void* ctx, const char* name);
  void* ctx;
};

int decode_max_tokens();
cudaError_t decode_prepare();  // sets kernel attributes once per device (not inside a capture)
int decode_max_slots();
cudaError_t launch_decode(const DecodeArgs& a, int fmt_r_gu, int fmt_r_d, int fmt_s, bool pdl, cudaStream_t s,
                          int* launches, const DecodeHooks* hooks);

// Prefill tensor-core GEMM of one expert group (see gemm_tc.cu).
struct GemmArgs {
  const uint8_t* w0;       // gate (gate/up) or down stack, repacked
  const uint8_t* w1;       // up stack (gate/up only)
  size_t mat_bytes;        // bytes of one expert's matrix (0 for the shared expert)
  int k;                   // reduction length
  const int4* tiles;       // routed: device tile list (expert, first row, rows); nullptr: dense
  const int* n_tiles;      // routed: number of tiles
  int n_rows;              // dense: rows of the activation operand (tokens)
  int m_tiles;             // 128-row slices of the weight matrix (set by launch_gemm)
  const float* inv_scale;  // gate/up: 1 / fp16 scale of each activation row
  __half* h_out;           // gate/up output [row][ld_out] fp16
  float* y_out;            // down output [row][ld_out] fp32
  int ld_out;
  int* err;                // error bits: 4 = a pipeline wait timed out, 8 = |h| beyond fp16 range
  long long timeout_cycles;  // limit of every pipeline wait in SM cycles; 0: the default (~1 s)
  int test_stall;          // 0; or s + 1: the first CTA withholds one dequant arrival of its K stage s (tests
                           // of the timeout path: the MMA's wait for that stage runs out)
};

// Tile geometry of the expert GEMMs for a forward (0: 192-token tiles; 1: 128-token tiles with
// 256-k pipeline stages, for batches whose experts average fewer than 64 tokens when every GEMM's
// K, whose greatest common divisor is k_gcd, is a multiple of 256), and its token tile (the routed
// tiling of a forward must use the same geometry as its GEMM launches).
int gemm_geometry(int n_tokens, int top_k, int n_experts, int k_gcd);
int gemm_tile_n(int geom);
cudaError_t gemm_prepare();
// TMA maps of one row-major fp16 activation buffer: boxes of 64 columns x 16, 32, 64 and 128 rows
// (a tile's rows are fetched exactly, with as few boxes as these sizes allow).
struct ActMaps {
  CUtensorMap r16, r32, r64, r128;  // boxes of 64 columns x 16 / 32 / 64 / 128 rows
};
cudaError_t launch_gemm(int fmt, bool gateup, const ActMaps& tm, const GemmArgs& p, int m_tiles, int n_tiles,
                        int geom, cudaStream_t s);
int make_act_maps(ActMaps* tm, const void* base, uint64_t rows, uint64_t cols);

// Prefill preparation (see prefill_prep.cu).
void launch_xprep(const __nv_bfloat16* x, int n_tok, int d, __half* xs16, float* inv_s, cudaStream_t s);
void launch_gather(const __half* xs16, const float* inv_s, const int* perm, const int* n_pos, int n_slots, int top_k,
                   int d, __half* xp16, float* inv_p, cudaStream_t s);
void launch_tiles(const int* counts, const int* offsets, int n_exp, const int* local_of, int tile_n, int4* tiles,
                  int* n_tiles, cudaStream_t s);

void launch_repack(int fmt, const uint8_t* src, uint8_t* dst, int total_rows, int k, cudaStream_t s);
void launch_q2k_dmax(const uint8_t* packed, size_t bytes, unsigned* out, cudaStream_t s);
void launch_router_split(const float* w, size_t n, __nv_bfloat16* w3, cudaStream_t s);
cudaError_t router_tc_prepare();      // kernel attributes, once per device (not inside a capture)
cudaError_t router_logits_prepare();  // the same for the scalar router
void launch_router_tc(const __nv_bfloat16* x, int n_tok, int d, const __nv_bfloat16* w3, const float* b, int n_exp,
                      float* logits, cudaStream_t s);
void launch_router_logits(const __nv_bfloat16* x, int n_tok, int d, const float* w, const float* b, int n_exp,
                          float* logits, cudaStream_t s);
void launch_topk(const float* logits, int n_learned, int n_exp, int top_k, const int* token_ids, int n_hash,
                 const int* table, int vocab, int* idx, float* wts, int* err, cudaStream_t s);
int bucket_chunks(int n_slots);  // ints of the bucketing scratch: bucket_chunks(n_slots) * n_exp
// local_of: [n_exp] weight slot of each expert, -1 for experts the handle does not hold (their slots
// are left out of the bucketing); null when the handle holds every expert.
void launch_bucket_count(const int* idx, int n_slots, int n_exp, const int* local_of, int* ghist, cudaStream_t s);
void launch_bucket_scatter(const int* idx, int n_slots, int n_exp, const int* ghist, const int* local_of, int* counts,
                           int* offsets, int* active, int* n_active, int* perm, int* rowof, cudaStream_t s);
void launch_combine(const int* idx, const float* wts, const int* rowof, const float* y, const float* ys, int n_tok,
                    int top_k, int d, float* out, cudaStream_t s);

}  // namespace ds4
