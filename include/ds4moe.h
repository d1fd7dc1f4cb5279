/*
 * ds4moe -- forward pass of a DeepSeek-V4-style quantized Mixture-of-Experts layer on one
 * NVIDIA GB300 (sm_103a). C ABI: plain pointers and sizes, no C++ or framework types.
 *
 * What one forward computes, for each token x (a row of d bf16 values):
 *
 *   learned routing   z = W_r x + b (fp32), s = sigmoid(z); the top_k experts by
 *                     (s descending, expert index ascending); w_j = s_j / sum of the
 *                     selected s. The bias b (optional) is added before the sigmoid.
 *   table routing     for the first n_hash tokens of a call: experts = table[token id],
 *                     w_j = 1 / top_k (arc PR #89 "expert parallelism stage 0 + stage 1
 *                     (EP=2) for V4's MoE", section "Stage 0": early layers route by a
 *                     fixed token-id table).
 *   routed experts    E_e(x) = W_d (silu(W_g x) * (W_u x)), weights dequantized from
 *                     Q2_K or Q8_0 blocks inside the kernels.
 *   combine           out = sum_j w_j E_{e_j}(x) + S(x): routed terms in ascending expert
 *                     id, then the shared expert S (same SwiGLU form, unscaled), all fp32,
 *                     fixed order, no floating-point atomics, so repeated calls are
 *                     bitwise identical. The plain-sum combine is the one the expert
 *                     parallel page describes (arc PR #89, section "Stage 1 -- EP=2"); its
 *                     bitwise repeatability answers the scheduling-dependent float
 *                     atomicAdd down projection recorded in TrevorS/ds4 PR #13 ("Tested").
 *
 * Tensor mix (ds4 PR #754 "CUDA: add DGX Spark network expert/tensor parallelism", section
 * "Supported paths and safety"): 2-bit Q2_K routed experts, Q8_0 shared expert. Each of
 * routed gate/up, routed down and shared may be either format.
 *
 * Canonical weight bytes accepted by ds4moe_create (little endian). A quantized [R x K]
 * matrix is R rows, each row its K/block blocks back to back; a routed stack is n_experts
 * such matrices back to back.
 *   DS4MOE_FMT_Q8_0: block of 32 weights, 34 bytes = fp16 scale, 32 x int8 q; w = scale*q.
 *   DS4MOE_FMT_Q2_K: super-block of 256 weights, 84 bytes = 16 scale bytes (byte j: low
 *     nibble s_j, high nibble m_j, sub-block j = weights 16j..16j+15), 64 quant bytes
 *     (weight i at byte i>>2, bits 2*(i&3)), fp16 d, fp16 dmin; w_i = d*s_j*q_i - dmin*m_j.
 *
 * Shapes: routed gate/up are [f_routed x d], routed down [d x f_routed], shared gate/up
 * [f_shared x d], shared down [d x f_shared]. Every K dimension must be a multiple of 256
 * for Q2_K and of 128 for Q8_0; d, f_routed and f_shared must be multiples of 128, with
 * d <= 12288 and f_routed, f_shared <= 16384.
 *
 * Error convention: every int-returning call returns DS4MOE_OK (0) or a negative code and
 * records a message readable with ds4moe_last_error() on the calling thread. Device-side
 * faults (none are expected) surface at the caller's next synchronisation.
 */
#ifndef DS4MOE_H
#define DS4MOE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define DS4MOE_OK 0
#define DS4MOE_ERR_INVALID_ARG -1        /* null pointer, bad size or shape */
#define DS4MOE_ERR_UNSUPPORTED_FORMAT -2 /* format enum not Q8_0 / Q2_K, or shape not tileable; also
                                            a Q2_K super-block with |d| >= 0.0666 (more precisely,
                                            15 * 2^16 * |d| >= 65504) on a handle whose max_tokens
                                            needs the batched path (max_tokens > 16 or
                                            max_tokens * top_k > 128): that path dequantizes Q2_K
                                            weights in fp16 as q * 2^-16 times 2^16 * d * s. Handles
                                            with max_tokens <= 16 (and max_tokens * top_k <= 128)
                                            accept any fp16 d: with such scales they serve every
                                            forward on the decode path */
#define DS4MOE_ERR_DEVICE_MISMATCH -3    /* a device pointer lives on another GPU than the handle */
#define DS4MOE_ERR_CAPACITY -4           /* n_tokens > max_tokens given at create */
#define DS4MOE_ERR_OOM -5                /* device allocation failed or exceeded workspace_limit */
#define DS4MOE_ERR_CUDA -6               /* a CUDA runtime call failed */

typedef enum ds4moe_format { DS4MOE_FMT_Q8_0 = 0, DS4MOE_FMT_Q2_K = 1 } ds4moe_format;

typedef struct ds4moe_shapes {
    int32_t d;             /* hidden size */
    int32_t f_routed;      /* routed expert intermediate size */
    int32_t f_shared;      /* shared expert intermediate size (ignored when n_shared == 0) */
    int32_t n_experts;     /* routed experts E, 1..256 */
    int32_t top_k;         /* experts per token, 1..min(E, 16) */
    int32_t n_shared;      /* 0 or 1 always-on shared expert */
    int32_t fmt_gate_up;   /* ds4moe_format of the routed gate and up projections */
    int32_t fmt_down;      /* ds4moe_format of the routed down projection */
    int32_t fmt_shared;    /* ds4moe_format of the shared expert's three projections */
    int32_t has_bias;      /* 1: router_b is read */
    int32_t hash_vocab;    /* rows of the token-id routing table; 0 = no table routing */
    int32_t max_tokens;    /* largest n_tokens of any later forward; sizes the workspace */
    int32_t device;        /* CUDA device ordinal the handle lives on */
    int32_t reserved;
    int64_t workspace_limit; /* bytes; 0 = unlimited. Exceeding it returns DS4MOE_ERR_OOM */
} ds4moe_shapes;

/* Each pointer may be host memory (pageable or pinned) or device memory on shapes.device.
 * ds4moe_create copies and repacks everything; the caller keeps ownership and may free or
 * reuse its buffers as soon as the call returns. */
typedef struct ds4moe_weights {
    const float* router_w;      /* fp32 [E x d] row-major */
    const float* router_b;      /* fp32 [E], read when has_bias, else may be NULL */
    const void* gate;           /* routed gate stack, E x [f_routed x d] canonical blocks */
    const void* up;             /* routed up stack, same shape */
    const void* down;           /* routed down stack, E x [d x f_routed] */
    const void* shared_gate;    /* [f_shared x d], NULL when n_shared == 0 */
    const void* shared_up;      /* [f_shared x d] */
    const void* shared_down;    /* [d x f_shared] */
    const int32_t* hash_table;  /* int32 [hash_vocab x top_k], distinct ids in [0, E) per row (checked
                                   at create: DS4MOE_ERR_INVALID_ARG otherwise); NULL if none */
} ds4moe_weights;

typedef struct ds4moe_stats {
    int32_t n_tokens;          /* tokens of the last forward */
    int32_t distinct_experts;  /* routed experts with at least one token in the last forward */
    int32_t error_flags;       /* device-side conditions of the last forward (0 = none). The
                                  forward itself has already returned DS4MOE_OK when they arise:
                                  read them here after a forward whose result matters.
                                  bit 0: a token id was outside [0, hash_vocab); that token's
                                         routed part was skipped (weights 0), the rest is valid.
                                  bit 2: a pipeline wait of the batched expert GEMM gave up after
                                         its time limit (about one second); the GEMM stopped and
                                         the output rows of that launch are incomplete. One of
                                         bits 17..23 names the wait: 17 weight producer (raw slot
                                         free), 18 activation producer (stage free), 19 dequant
                                         (raw weights landed), 20 dequant (stage free), 21
                                         epilogue (accumulator full), 22 MMA (accumulator free),
                                         23 MMA (stage full).
                                  bit 3: in the batched path, an intermediate |h| = |silu(g) u|
                                         exceeded the fp16 range (65504); it was stored as an
                                         infinity and the affected output rows are not finite.
                                  Other bits are reserved. */
    int32_t reserved;
    int32_t counts[256];       /* tokens per routed expert in the last forward */
} ds4moe_stats;

typedef struct ds4moe_handle ds4moe_handle;

/* Validates shapes, allocates the device weights and a workspace for max_tokens, copies and
 * repacks the weights. Synchronous. On failure *out is set to NULL and nothing leaks.
 * Forwards take one of two paths (same results up to fp32 rounding; both deterministic): the
 * decode path (three kernels, each touched expert read once per token; up to 16 tokens and
 * 128 slots) and the batched path (tensor-core expert GEMMs, each touched expert read once for
 * all its tokens). Forwards of fewer than 8 tokens take the decode path, larger ones the batched
 * path when the handle has it (max_tokens >= 8 and weights within the batched path's Q2_K scale
 * range, see DS4MOE_ERR_UNSUPPORTED_FORMAT). The environment variable DS4MOE_BATCHED_FROM, read
 * here, replaces the 8 (17 keeps every forward the decode kernels can take on the decode path). */
int ds4moe_create(const ds4moe_weights* w, const ds4moe_shapes* s, ds4moe_handle** out);

/* Expert-parallel partial on one GPU (arc PR #89 "expert parallelism stage 0 + stage 1 (EP=2)",
 * section "Stage 1 -- EP=2": a rank holds a subset of the routed experts and computes the sum over
 * its owned slots of w_j E_j(x); the layer output is the plain sum of the ranks' partials).
 * As ds4moe_create, but the handle holds (copies and repacks) only the routed experts
 * owned[0..n_owned): distinct ids in [0, n_experts), in any order, read from host memory during
 * the call; w still describes the full expert stacks. Its forwards route every token over all
 * n_experts exactly as ds4moe_forward does (the router weights and the hash table are whole), and
 * write out = the sum over the token's slots whose expert is held of w_j E_j(x), held terms in
 * ascending expert id, plus S(x) when include_shared is nonzero. With include_shared == 0 the
 * shared expert is neither copied nor run. The partials of handles whose owned sets partition the
 * experts, exactly one of them with include_shared, add up to ds4moe_forward's output up to the
 * fp32 rounding of that sum. ds4moe_get_route returns the whole routing; ds4moe_get_stats counts
 * only the held experts (counts of the others are 0, distinct_experts counts held experts touched).
 * Every block format is sliceable by expert (an expert's matrices are whole), so none is refused
 * here. Errors: DS4MOE_ERR_INVALID_ARG for a NULL owned, n_owned outside 1..n_experts, or an id
 * out of range or named twice; otherwise as ds4moe_create. */
int ds4moe_create_subset(const ds4moe_weights* w, const ds4moe_shapes* s, const int32_t* owned, int32_t n_owned,
                         int32_t include_shared, ds4moe_handle** out);

/* Learned routing for every token. x: device bf16 [n_tokens x d]; out: device fp32
 * [n_tokens x d]; both caller-owned, on the handle's device. stream: a cudaStream_t (NULL =
 * legacy default stream). Asynchronous and stream-ordered: no host synchronisation. A handle
 * serves one stream at a time (its workspace is shared by all calls on it). n_tokens == 0 is
 * a no-op. */
int ds4moe_forward(ds4moe_handle* h, const void* x, int32_t n_tokens, float* out, void* stream);

/* As ds4moe_forward, but tokens 0..n_hash-1 take table routing by token_ids (device int32
 * [n_hash]). n_hash must be 0 when the handle has no table. */
int ds4moe_forward_ex(ds4moe_handle* h, const void* x, int32_t n_tokens, const int32_t* token_ids,
                      int32_t n_hash, float* out, void* stream);

/* As ds4moe_forward_ex with host buffers: copies x (and token_ids) to the device, runs the
 * forward and copies out back, then synchronises the stream before returning. With page-locked
 * host buffers the copies and the kernels replay as one cached CUDA graph (keyed by the token
 * counts and buffer addresses; device forwards cache their kernels' graph the same way), and x and
 * out (when 16-byte aligned) are copied by a kernel that addresses them directly rather than by
 * the copy engines (DS4MOE_SM_COPIES=0 at create turns that off); pageable buffers take separate
 * copies. */
int ds4moe_forward_host(ds4moe_handle* h, const void* x_host, int32_t n_tokens,
                        const int32_t* token_ids_host, int32_t n_hash, float* out_host, void* stream);

/* Copies the last forward's routing to host arrays idx [n_tokens x top_k] and w
 * [n_tokens x top_k] in top-k order (score descending). Synchronises the handle's last
 * stream; meant for tests and measurement, not for a timed path. */
int ds4moe_get_route(ds4moe_handle* h, int32_t* idx_host, float* w_host, int32_t n_tokens);

/* Per-expert token counts, distinct experts touched and error flags of the last forward.
 * Synchronises like ds4moe_get_route. */
int ds4moe_get_stats(ds4moe_handle* h, ds4moe_stats* st);

/* Bytes of device memory the handle holds (weights + workspace). */
int64_t ds4moe_device_bytes(const ds4moe_handle* h);

/* Number of kernel launches one forward of n_tokens learned-routed tokens issues. */
int32_t ds4moe_launches_per_forward(const ds4moe_handle* h, int32_t n_tokens);

/* Per-launch timing for measurement: when enabled, every later forward records a CUDA event
 * after each kernel launch on its stream (this adds event records between launches).
 * ds4moe_get_phase_times waits for the last profiled forward and returns, for each launch in
 * order, its stream time in milliseconds (ms, may be NULL) and a static name (names, may be
 * NULL); *n_phases receives the number of launches (0 when profiling is off). */
int ds4moe_set_profiling(ds4moe_handle* h, int32_t enable);
int ds4moe_get_phase_times(ds4moe_handle* h, float* ms, const char** names, int32_t max_phases,
                           int32_t* n_phases);

/* Routing step alone, allocating nothing (the paper has no counterpart: this is a library
 * convenience). Some callers cannot call cudaMalloc -- an engine that carves its device memory
 * up front and forbids later allocations, a plugin whose host owns the memory budget, a
 * latency-critical path where cudaMalloc may synchronise the device. This call needs no handle:
 * it computes fp32 logits of router_w (device fp32 [n_experts x d]) and router_b (device fp32
 * [n_experts] or NULL) for x (device bf16 [n_tokens x d]), then the sigmoid top-k with ties to
 * the lower index and weights renormalised to sum 1, into idx (device int32
 * [n_tokens x top_k]) and w (device fp32 [n_tokens x top_k]), in top-k order. It computes the
 * same routing as ds4moe_forward with its own kernel (fp32 FMA logits): the fp32 summation order
 * differs from the forward's routers, so logits may differ in the last bits, and the chosen
 * experts agree with the forward's except where the k-th and (k+1)-th scores are within about
 * 1e-6 of each other. Runs on the calling thread's current device, asynchronously on stream.
 * The logits live in a static device array of DS4MOE_NOALLOC_MAX_LOGITS floats that the library
 * image carries (held by every GPU that loads the library until exit): n_tokens * n_experts
 * above that returns DS4MOE_ERR_CAPACITY. The first call on a device looks the array's address
 * up (cudaGetSymbolAddress) and sets the router kernel's attributes in that device's context;
 * make it before any stream capture. All calls on a device share the array, so calls that may
 * overlap on the GPU (unordered streams) race. */
#define DS4MOE_NOALLOC_MAX_LOGITS 262144
int ds4moe_route_noalloc(const float* router_w, const float* router_b, const void* x, int32_t n_tokens,
                         int32_t d, int32_t n_experts, int32_t top_k, int32_t* idx, float* w, void* stream);

/* Test hook of the failure path (no counterpart in the paper: it exists so that the bounded waits
 * of the batched expert GEMM can be shown to end with an error status instead of a hang). The next
 * batched forward of h (more than 16 tokens, or more than 128 routed slots) runs its routed
 * gate/up GEMM with every pipeline wait limited to about 1 ms instead of about 1 s, and the first
 * CTA of that launch withholds one dequant arrival of its K stage `stage` (counted over the CTA's
 * work items). That stage never becomes full, so the MMA's wait for it runs out: the CTA stops,
 * lets its issued copies and MMAs finish, frees its tensor memory and records error bit 2 plus a
 * bit naming the wait (see ds4moe_stats.error_flags); that forward's output is incomplete. The
 * hook applies to one forward and then clears itself. stage >= 0; DS4MOE_ERR_INVALID_ARG
 * otherwise. */
int ds4moe_set_test_stall(ds4moe_handle* h, int32_t stage);

/* Frees everything the handle owns. NULL is allowed. Synchronises the device first. */
void ds4moe_destroy(ds4moe_handle* h);

/* Message of the last failed call on this thread ("" if none). */
const char* ds4moe_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* DS4MOE_H */
