// C-ABI shim of the ds4moe library: argument validation, device memory, create-time repack
// and the launch sequence of one forward. Host code only; kernels live in the other units.
#include <algorithm>
#include <numeric>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <string>
#include <vector>

#include "../../include/ds4moe.h"
#include "common.cuh"

namespace {

thread_local std::string g_last_error;

int fail(int code, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
int fail(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return code;
}

#define DS4_CUDA(call)                                                                          \
  do {                                                                                          \
    cudaError_t e_ = (call);                                                                    \
    if (e_ != cudaSuccess) return fail(DS4MOE_ERR_CUDA, "%s failed: %s", #call, cudaGetErrorString(e_)); \
  } while (0)

// Restores the caller's current device on scope exit.
struct DeviceGuard {
  int prev = -1;
  bool ok = false;
  explicit DeviceGuard(int dev) {
    if (cudaGetDevice(&prev) == cudaSuccess && cudaSetDevice(dev) == cudaSuccess) ok = true;
  }
  ~DeviceGuard() {
    if (prev >= 0) cudaSetDevice(prev);
  }
};

enum PtrKind { PTR_HOST, PTR_DEVICE, PTR_OTHER_DEVICE };

PtrKind classify(const void* p, int device) {
  cudaPointerAttributes attr;
  if (cudaPointerGetAttributes(&attr, p) != cudaSuccess) {
    cudaGetLastError();  // clear: an unknown pointer is plain host memory
    return PTR_HOST;
  }
  if (attr.type == cudaMemoryTypeDevice || attr.type == cudaMemoryTypeManaged)
    return attr.device == device ? PTR_DEVICE : PTR_OTHER_DEVICE;
  return PTR_HOST;
}

}  // namespace

namespace ds4 {
// Lets the other translation units report errors through ds4moe_last_error.
int set_error(int code, const char* msg) { return fail(code, "%s", msg); }
// A 16-byte-vector copy run by the SMs (combine.cu; bytes a multiple of 16, both pointers 16-byte
// aligned and addressable by kernels: device memory or page-locked host memory under unified
// addressing).
void launch_copy16(const void* src, void* dst, size_t bytes, cudaStream_t s);
}  // namespace ds4

struct ds4moe_handle {
  ds4moe_shapes s{};
  int64_t bytes = 0;
  std::vector<void*> allocs;
  // weights
  float* router_w = nullptr;
  float* router_b = nullptr;
  __nv_bfloat16* router_w3 = nullptr;  // batched path: the router weights as three bf16 parts
  uint8_t* gate = nullptr;
  uint8_t* up = nullptr;
  uint8_t* down = nullptr;
  uint8_t* sgate = nullptr;
  uint8_t* sup = nullptr;
  uint8_t* sdown = nullptr;
  int* table = nullptr;
  size_t mb_gu = 0, mb_d = 0, mb_sgu = 0, mb_sd = 0;
  // expert subset (ds4moe_create_subset): weight slot of each expert, -1 where not held; null when
  // the handle holds every expert
  int* local_of = nullptr;
  int n_local = 0;  // experts held (weight slots)
  // workspace
  float* logits = nullptr;
  int* idx = nullptr;
  float* wts = nullptr;
  int* counts = nullptr;
  int* offsets = nullptr;
  int* active = nullptr;
  int* n_active = nullptr;
  int* perm = nullptr;
  int* rowof = nullptr;
  int* ghist = nullptr;  // batched bucketing: per-chunk expert histograms
  float* H = nullptr;   // decode: h per routed slot, fp32
  float* Hs = nullptr;  // decode: h of the shared expert, fp32
  float* hsg = nullptr;  // decode: max |h| of the shared expert per token and 16-row group
  float* Y = nullptr;   // prefill: down output per bucketed slot, fp32
  float* Ys = nullptr;  // prefill: shared expert output per token, fp32
  // prefill tensor-core path
  __half* Xs16 = nullptr;
  __half* Xp16 = nullptr;
  __half* H16 = nullptr;
  __half* Hs16 = nullptr;
  float* inv_s = nullptr;
  float* inv_p = nullptr;
  int4* tiles = nullptr;
  int* n_tiles = nullptr;
  bool has_prefill = false;
  ds4::ActMaps tm_xp, tm_xs, tm_h, tm_hs;
  int* err = nullptr;
  float* xmax = nullptr;
  float* hmax = nullptr;
  int4* work = nullptr;
  int* tokof = nullptr;
  float* xscale = nullptr;
  unsigned int* counter = nullptr;
  // host-call staging
  __nv_bfloat16* x_stage = nullptr;
  int* tid_stage = nullptr;
  float* out_stage = nullptr;
  // device pointers already verified by a forward (a small ring)
  static constexpr int kChecked = 32;
  const void* checked[kChecked] = {};
  int checked_next = 0;
  // last forward
  cudaStream_t last_stream = nullptr;
  int last_n = 0;
  // optional per-launch timing (events recorded between launches on the forward's stream)
  bool profile = false;
  static constexpr int kMaxPhases = 16;
  cudaEvent_t ev[kMaxPhases + 1] = {};
  const char* phase_name[kMaxPhases] = {};
  int n_phases = 0;
  // test of the GEMM timeout path (ds4moe_set_test_stall): stage + 1 for the next batched forward
  int test_stall = 0;
  // Forwards of up to decode_upto tokens (and top_k slots within the decode kernels' limit) take the
  // decode path, larger ones the batched path. The batched path reads each touched expert once for
  // all its tokens; the decode kernels re-read it per token but launch three kernels instead of
  // twelve. A handle without the batched path's buffers decodes up to the decode kernels' limit.
  int decode_upto = 16;

  // Decode forwards replay a captured CUDA graph of their three launches (launching each kernel
  // from the host costs far more than a graph node). Graphs are keyed by the call's token
  // counts and buffer pointers; at most kGraphs are kept, the least recently used is replaced.
  bool use_graphs = true;
  cudaStream_t cap_stream = nullptr;
  struct GraphEntry {
    int kind = 0;  // 0: decode path, 1: batched path
    int n = -1, n_hash = 0;
    const void* x = nullptr;
    const int* tid = nullptr;
    float* out = nullptr;
    // host entry point: pinned host buffers copied inside the graph (null for device forwards)
    const void* hx = nullptr;
    const int* htid = nullptr;
    float* hout = nullptr;
    cudaGraphExec_t exec = nullptr;
    uint64_t used = 0;
  };
  struct HostIo {
    const void* x = nullptr;
    const int* tid = nullptr;
    float* out = nullptr;
    // the same x and out as kernels address them (page-locked memory under unified addressing),
    // or null: copied by the SMs instead of the copy engines when present
    const void* x_k = nullptr;
    float* out_k = nullptr;
  };
  bool sm_copies = true;
  static constexpr int kGraphs = 16;
  GraphEntry graphs[kGraphs];
  uint64_t tick = 0;

  // The graph of one forward's launches (launch(stream) returns a DS4MOE status), captured on first
  // use for this (path, token counts, buffers) and replayed afterwards.
  template <typename Launch>
  int cached_graph(int kind, int n, int n_hash, const void* x, const int* tid, float* out, const HostIo* io,
                   Launch&& launch, cudaGraphExec_t* exec_out);
  void release_graphs() {
    for (GraphEntry& g : graphs)
      if (g.exec) {
        cudaGraphExecDestroy(g.exec);
        g = GraphEntry();
      }
    if (cap_stream) {
      cudaStreamDestroy(cap_stream);
      cap_stream = nullptr;
    }
  }

  int alloc(void** p, size_t n) {
    if (n == 0) n = 16;
    if (s.workspace_limit > 0 && bytes + (int64_t)n > s.workspace_limit)
      return fail(DS4MOE_ERR_OOM, "device allocation of %zu bytes exceeds workspace_limit %lld (held %lld)", n,
                  (long long)s.workspace_limit, (long long)bytes);
    cudaError_t e = cudaMalloc(p, n);
    if (e != cudaSuccess) {
      cudaGetLastError();
      *p = nullptr;
      return fail(DS4MOE_ERR_OOM, "cudaMalloc(%zu) failed: %s", n, cudaGetErrorString(e));
    }
    allocs.push_back(*p);
    bytes += (int64_t)n;
    return DS4MOE_OK;
  }
  template <typename T>
  int alloc_t(T** p, size_t n) {
    return alloc(reinterpret_cast<void**>(p), n);
  }
  void release() {
    release_graphs();
    for (cudaEvent_t& e : ev)
      if (e) {
        cudaEventDestroy(e);
        e = nullptr;
      }
    for (void* p : allocs) cudaFree(p);
    allocs.clear();
    bytes = 0;
  }
};

template <typename Launch>
int ds4moe_handle::cached_graph(int kind, int n, int nh, const void* x, const int* tid, float* o, const HostIo* io,
                                Launch&& launch, cudaGraphExec_t* exec_out) {
  const HostIo hio = io ? *io : HostIo();
  GraphEntry* hit = nullptr;
  GraphEntry* victim = &graphs[0];
  for (GraphEntry& g : graphs) {
    if (g.exec && g.kind == kind && g.n == n && g.n_hash == nh && g.x == x && g.tid == tid && g.out == o &&
        g.hx == hio.x && g.htid == hio.tid && g.hout == hio.out)
      hit = &g;
    if (!g.exec || g.used < victim->used) victim = &g;
  }
  if (!hit) {
    if (!cap_stream) DS4_CUDA(cudaStreamCreateWithFlags(&cap_stream, cudaStreamNonBlocking));
    if (victim->exec) {
      cudaGraphExecDestroy(victim->exec);
      *victim = GraphEntry();
    }
    cudaGraph_t graph = nullptr;
    DS4_CUDA(cudaStreamBeginCapture(cap_stream, cudaStreamCaptureModeThreadLocal));
    const size_t d = (size_t)s.d;
    cudaError_t e = cudaSuccess;
    int rc = DS4MOE_OK;
    if (hio.x && hio.x_k) {
      ds4::launch_copy16(hio.x_k, const_cast<void*>(x), (size_t)n * d * 2, cap_stream);
      e = cudaGetLastError();
    } else if (hio.x) {
      e = cudaMemcpyAsync(const_cast<void*>(x), hio.x, (size_t)n * d * 2, cudaMemcpyHostToDevice, cap_stream);
    }
    if (e == cudaSuccess && hio.tid && nh > 0)
      e = cudaMemcpyAsync(const_cast<int*>(tid), hio.tid, (size_t)nh * 4, cudaMemcpyHostToDevice, cap_stream);
    if (e == cudaSuccess) rc = launch(cap_stream);
    if (e == cudaSuccess && rc == DS4MOE_OK && hio.out && hio.out_k) {
      ds4::launch_copy16(o, hio.out_k, (size_t)n * d * 4, cap_stream);
      e = cudaGetLastError();
    } else if (e == cudaSuccess && rc == DS4MOE_OK && hio.out) {
      e = cudaMemcpyAsync(hio.out, o, (size_t)n * d * 4, cudaMemcpyDeviceToHost, cap_stream);
    }
    cudaError_t e2 = cudaStreamEndCapture(cap_stream, &graph);
    if (e != cudaSuccess || e2 != cudaSuccess || rc != DS4MOE_OK) {
      if (graph) cudaGraphDestroy(graph);
      cudaGetLastError();
      if (rc != DS4MOE_OK) return rc;
      return fail(DS4MOE_ERR_CUDA, "forward graph capture: %s", cudaGetErrorString(e != cudaSuccess ? e : e2));
    }
    cudaGraphExec_t exec = nullptr;
    e = cudaGraphInstantiate(&exec, graph, 0);
    cudaGraphDestroy(graph);
    if (e != cudaSuccess) return fail(DS4MOE_ERR_CUDA, "forward graph instantiate: %s", cudaGetErrorString(e));
    victim->kind = kind;
    victim->n = n;
    victim->n_hash = nh;
    victim->x = x;
    victim->tid = tid;
    victim->out = o;
    victim->hx = hio.x;
    victim->htid = hio.tid;
    victim->hout = hio.out;
    victim->exec = exec;
    hit = victim;
  }
  hit->used = ++tick;
  *exec_out = hit->exec;
  return DS4MOE_OK;
}

namespace {

bool fmt_ok(int f) { return f == DS4MOE_FMT_Q8_0 || f == DS4MOE_FMT_Q2_K; }

// Token tile of the routed expert GEMMs of a forward (the gate/up and the down GEMM share one
// tiling), and the largest number of routed tiles a forward of n tokens can have with it.
int routed_tile_n(int geom) { return ds4::gemm_tile_n(geom); }
size_t max_routed_tiles(size_t slots, int n_experts, int tn) { return (slots + tn - 1) / tn + std::min<size_t>(n_experts, slots); }

int check_shapes(const ds4moe_shapes* s) {
  // the router stages 8 token rows of d bf16 values in shared memory: d <= 12288 keeps that under 200 KB
  if (s->d <= 0 || s->d % 128 || s->d > 12288) return fail(DS4MOE_ERR_INVALID_ARG, "d=%d must be a positive multiple of 128 up to 12288", s->d);
  if (s->f_routed <= 0 || s->f_routed % 128 || s->f_routed > 16384)
    return fail(DS4MOE_ERR_INVALID_ARG, "f_routed=%d must be a positive multiple of 128 up to 16384", s->f_routed);
  if (s->n_shared != 0 && s->n_shared != 1) return fail(DS4MOE_ERR_INVALID_ARG, "n_shared=%d must be 0 or 1", s->n_shared);
  if (s->n_shared && (s->f_shared <= 0 || s->f_shared % 128 || s->f_shared > 16384))
    return fail(DS4MOE_ERR_INVALID_ARG, "f_shared=%d must be a positive multiple of 128 up to 16384", s->f_shared);
  if (s->n_experts < 1 || s->n_experts > 256) return fail(DS4MOE_ERR_INVALID_ARG, "n_experts=%d must be in 1..256", s->n_experts);
  if (s->top_k < 1 || s->top_k > 16 || s->top_k > s->n_experts)
    return fail(DS4MOE_ERR_INVALID_ARG, "top_k=%d must be in 1..min(n_experts, 16)", s->top_k);
  if (s->max_tokens < 1 || s->max_tokens > 65535) return fail(DS4MOE_ERR_INVALID_ARG, "max_tokens=%d must be in 1..65535", s->max_tokens);
  if (s->hash_vocab < 0) return fail(DS4MOE_ERR_INVALID_ARG, "hash_vocab=%d is negative", s->hash_vocab);
  const int fm[3] = {s->fmt_gate_up, s->fmt_down, s->fmt_shared};
  const char* nm[3] = {"fmt_gate_up", "fmt_down", "fmt_shared"};
  for (int i = 0; i < 3; ++i)
    if (!fmt_ok(fm[i]) && !(i == 2 && !s->n_shared))
      return fail(DS4MOE_ERR_UNSUPPORTED_FORMAT, "%s=%d is not a supported block format (Q8_0=0, Q2_K=1)", nm[i], fm[i]);
  auto kq = [](int fmt, int k) { return k % ds4::unit_k(fmt) == 0; };
  if (!kq(s->fmt_gate_up, s->d)) return fail(DS4MOE_ERR_UNSUPPORTED_FORMAT, "d=%d is not a multiple of %d required by fmt_gate_up", s->d, ds4::unit_k(s->fmt_gate_up));
  if (!kq(s->fmt_down, s->f_routed)) return fail(DS4MOE_ERR_UNSUPPORTED_FORMAT, "f_routed=%d is not a multiple of %d required by fmt_down", s->f_routed, ds4::unit_k(s->fmt_down));
  if (s->n_shared && (!kq(s->fmt_shared, s->d) || !kq(s->fmt_shared, s->f_shared)))
    return fail(DS4MOE_ERR_UNSUPPORTED_FORMAT, "shared expert K dims (d=%d, f_shared=%d) are not multiples of %d", s->d, s->f_shared, ds4::unit_k(s->fmt_shared));
  return DS4MOE_OK;
}

int check_device(int device) {
  int ndev = 0;
  if (cudaGetDeviceCount(&ndev) != cudaSuccess || ndev == 0) {
    cudaGetLastError();
    return fail(DS4MOE_ERR_CUDA, "no CUDA device available");
  }
  if (device < 0 || device >= ndev) return fail(DS4MOE_ERR_INVALID_ARG, "device=%d out of range (%d devices)", device, ndev);
  return DS4MOE_OK;
}

// Copies `bytes` from a host or device source into dst (device).
int copy_in(void* dst, const void* src, size_t bytes, int device, const char* what) {
  const PtrKind k = classify(src, device);
  if (k == PTR_OTHER_DEVICE) return fail(DS4MOE_ERR_DEVICE_MISMATCH, "%s lives on another device than %d", what, device);
  DS4_CUDA(cudaMemcpy(dst, src, bytes, k == PTR_DEVICE ? cudaMemcpyDeviceToDevice : cudaMemcpyHostToDevice));
  return DS4MOE_OK;
}

// Repacks n_mat canonical [rows x k] matrices into dst (back to back): matrices mats[0..n_mat) of
// the source stack, or its first n_mat when mats is null.
int repack_stack(ds4moe_handle* h, int fmt, const void* src, uint8_t* dst, int n_mat, int rows, int k,
                 const char* what, const int* mats = nullptr) {
  const size_t mb = ds4::matrix_bytes(fmt, rows, k);
  const PtrKind kind = classify(src, h->s.device);
  if (kind == PTR_OTHER_DEVICE) return fail(DS4MOE_ERR_DEVICE_MISMATCH, "%s lives on another device than %d", what, h->s.device);
  const uint8_t* src8 = static_cast<const uint8_t*>(src);
  if (kind == PTR_DEVICE) {
    if (!mats) {
      ds4::launch_repack(fmt, src8, dst, n_mat * rows, k, 0);
    } else {
      for (int m = 0; m < n_mat; ++m) ds4::launch_repack(fmt, src8 + mb * mats[m], dst + mb * m, rows, k, 0);
    }
    DS4_CUDA(cudaGetLastError());
    DS4_CUDA(cudaDeviceSynchronize());
    return DS4MOE_OK;
  }
  // host source: stage a batch of matrices at a time (at most ~256 MB of staging)
  int per = (int)std::max<size_t>(1, (size_t)(256u << 20) / mb);
  per = std::min(per, n_mat);
  uint8_t* stage = nullptr;
  cudaError_t e = cudaMalloc(&stage, mb * per);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return fail(DS4MOE_ERR_OOM, "staging buffer of %zu bytes: %s", mb * per, cudaGetErrorString(e));
  }
  int rc = DS4MOE_OK;
  for (int m0 = 0; m0 < n_mat && rc == DS4MOE_OK; m0 += per) {
    const int n = std::min(per, n_mat - m0);
    if (!mats) {
      e = cudaMemcpy(stage, src8 + mb * m0, mb * n, cudaMemcpyHostToDevice);
    } else {
      e = cudaSuccess;
      for (int m = 0; m < n && e == cudaSuccess; ++m)
        e = cudaMemcpy(stage + mb * m, src8 + mb * mats[m0 + m], mb, cudaMemcpyHostToDevice);
    }
    if (e == cudaSuccess) {
      ds4::launch_repack(fmt, stage, dst + mb * m0, n * rows, k, 0);
      e = cudaGetLastError();
    }
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e != cudaSuccess) rc = fail(DS4MOE_ERR_CUDA, "repack of %s: %s", what, cudaGetErrorString(e));
  }
  cudaFree(stage);
  return rc;
}

// Every table entry must name a routed expert: the bucketing indexes per-expert arrays by it.
int check_table(const int* dev_table, size_t rows, int k, int n_exp) {
  std::vector<int> host(rows * k);
  DS4_CUDA(cudaMemcpy(host.data(), dev_table, host.size() * 4, cudaMemcpyDeviceToHost));
  for (size_t i = 0; i < host.size(); ++i)
    if (host[i] < 0 || host[i] >= n_exp)
      return fail(DS4MOE_ERR_INVALID_ARG, "hash_table entry %zu is %d, outside [0, n_experts=%d)", i, host[i], n_exp);
  for (size_t r = 0; r < rows; ++r)  // a token is routed to k distinct experts
    for (int a = 0; a < k; ++a)
      for (int b = a + 1; b < k; ++b)
        if (host[r * k + a] == host[r * k + b])
          return fail(DS4MOE_ERR_INVALID_ARG, "hash_table row %zu names expert %d twice", r, host[r * k + a]);
  return DS4MOE_OK;
}

// The batched path dequantizes Q2_K weights in fp16 as q * 2^-16 times 2^16 d s: every super-
// block needs 15 * 2^16 * |d| inside the fp16 range, i.e. |d| < 0.0666 (typical d are ~1e-3).
int check_q2k_scales(ds4moe_handle* h) {
  const ds4moe_shapes& s = h->s;
  const uint8_t* stacks[4] = {nullptr, nullptr, nullptr, nullptr};
  size_t bytes[4] = {0, 0, 0, 0};
  if (s.fmt_gate_up == DS4MOE_FMT_Q2_K) {
    stacks[0] = h->gate; bytes[0] = h->mb_gu * h->n_local;
    stacks[1] = h->up; bytes[1] = h->mb_gu * h->n_local;
  }
  if (s.fmt_down == DS4MOE_FMT_Q2_K) { stacks[2] = h->down; bytes[2] = h->mb_d * h->n_local; }
  unsigned* dmax = nullptr;
  DS4_CUDA(cudaMalloc(&dmax, 4));
  cudaError_t e = cudaMemset(dmax, 0, 4);
  for (int i = 0; i < 3 && e == cudaSuccess; ++i)
    if (stacks[i]) {
      ds4::launch_q2k_dmax(stacks[i], bytes[i], dmax, 0);
      e = cudaGetLastError();
    }
  if (s.n_shared && s.fmt_shared == DS4MOE_FMT_Q2_K && e == cudaSuccess) {
    ds4::launch_q2k_dmax(h->sgate, h->mb_sgu, dmax, 0);
    ds4::launch_q2k_dmax(h->sup, h->mb_sgu, dmax, 0);
    ds4::launch_q2k_dmax(h->sdown, h->mb_sd, dmax, 0);
    e = cudaGetLastError();
  }
  unsigned bits = 0;
  if (e == cudaSuccess) e = cudaMemcpy(&bits, dmax, 4, cudaMemcpyDeviceToHost);
  cudaFree(dmax);
  if (e != cudaSuccess) return fail(DS4MOE_ERR_CUDA, "Q2_K scale check: %s", cudaGetErrorString(e));
  float d;
  memcpy(&d, &bits, 4);
  if (!(d * 15.f * 65536.f < 65504.f))
    return fail(DS4MOE_ERR_UNSUPPORTED_FORMAT, "Q2_K super-block scale |d| = %g: the batched path needs |d| < 0.0666", d);
  return DS4MOE_OK;
}

#define DS4_TRY(call)          \
  do {                         \
    int rc_ = (call);          \
    if (rc_ != DS4MOE_OK) {    \
      h->release();            \
      delete h;                \
      return rc_;              \
    }                          \
  } while (0)

}  // namespace

// owned: host list of the experts the handle holds (null: all); include_shared: keep the shared expert.
static int create_impl(const ds4moe_weights* w, const ds4moe_shapes* s_in, const int32_t* owned, int n_owned,
                int include_shared, ds4moe_handle** out) {
  if (!out) return fail(DS4MOE_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  if (!w || !s_in) return fail(DS4MOE_ERR_INVALID_ARG, "weights or shapes is NULL");
  int rc = check_shapes(s_in);
  if (rc != DS4MOE_OK) return rc;
  ds4moe_shapes shp = *s_in;
  const ds4moe_shapes* s = &shp;
  std::vector<int> held;  // the experts held, ascending; local slot = position in this list
  std::vector<int> local_of;
  if (owned) {
    if (n_owned < 1 || n_owned > s->n_experts)
      return fail(DS4MOE_ERR_INVALID_ARG, "n_owned=%d must be in 1..n_experts=%d", n_owned, s->n_experts);
    local_of.assign(s->n_experts, -1);
    for (int i = 0; i < n_owned; ++i) {
      const int e = owned[i];
      if (e < 0 || e >= s->n_experts) return fail(DS4MOE_ERR_INVALID_ARG, "owned[%d]=%d is outside [0, n_experts=%d)", i, e, s->n_experts);
      if (local_of[e] != -1) return fail(DS4MOE_ERR_INVALID_ARG, "owned names expert %d twice", e);
      local_of[e] = 0;
    }
    for (int e = 0; e < s->n_experts; ++e)
      if (local_of[e] == 0) {
        local_of[e] = (int)held.size();
        held.push_back(e);
      }
    if (!include_shared) shp.n_shared = 0;  // this handle's partial leaves the shared expert out
  }
  if (!w->router_w || !w->gate || !w->up || !w->down) return fail(DS4MOE_ERR_INVALID_ARG, "router_w, gate, up and down are required");
  if (s->has_bias && !w->router_b) return fail(DS4MOE_ERR_INVALID_ARG, "has_bias set but router_b is NULL");
  if (s->n_shared && (!w->shared_gate || !w->shared_up || !w->shared_down))
    return fail(DS4MOE_ERR_INVALID_ARG, "n_shared=1 but a shared expert tensor is NULL");
  if (s->hash_vocab > 0 && !w->hash_table) return fail(DS4MOE_ERR_INVALID_ARG, "hash_vocab>0 but hash_table is NULL");
  rc = check_device(s->device);
  if (rc != DS4MOE_OK) return rc;
  DeviceGuard guard(s->device);
  if (!guard.ok) return fail(DS4MOE_ERR_CUDA, "cannot select device %d", s->device);

  ds4moe_handle* h = new ds4moe_handle();
  h->s = *s;
  if (const char* ev = getenv("DS4MOE_NO_GRAPHS")) h->use_graphs = ev[0] == '0';
  if (const char* ev = getenv("DS4MOE_SM_COPIES")) h->sm_copies = ev[0] != '0';
  // fewest tokens that take the batched path (measured on GB300 at d = 4096, 256 experts top-8,
  // f = 2048: the decode path is faster up to 6 tokens, the batched path from 8: 298 vs 319 us at
  // 8 tokens, 392 vs 599 us at 16); DS4MOE_BATCHED_FROM overrides it (17: decode path up to the
  // decode kernels' limit of 16 tokens)
  int small_batch_from = 8;
  if (const char* ev = getenv("DS4MOE_BATCHED_FROM")) small_batch_from = std::max(1, atoi(ev));
  const int E = s->n_experts, d = s->d, f = s->f_routed, fs = s->f_shared, K = s->top_k;
  h->mb_gu = ds4::matrix_bytes(s->fmt_gate_up, f, d);
  h->mb_d = ds4::matrix_bytes(s->fmt_down, d, f);
  h->n_local = owned ? (int)held.size() : E;
  const int L = h->n_local;
  const int* mats = owned ? held.data() : nullptr;
  // weights
  DS4_TRY(h->alloc_t(&h->router_w, (size_t)E * d * 4));
  DS4_TRY(copy_in(h->router_w, w->router_w, (size_t)E * d * 4, s->device, "router_w"));
  if (s->has_bias) {
    DS4_TRY(h->alloc_t(&h->router_b, (size_t)E * 4));
    DS4_TRY(copy_in(h->router_b, w->router_b, (size_t)E * 4, s->device, "router_b"));
  }
  DS4_TRY(h->alloc_t(&h->gate, h->mb_gu * L));
  DS4_TRY(h->alloc_t(&h->up, h->mb_gu * L));
  DS4_TRY(h->alloc_t(&h->down, h->mb_d * L));
  DS4_TRY(repack_stack(h, s->fmt_gate_up, w->gate, h->gate, L, f, d, "gate", mats));
  DS4_TRY(repack_stack(h, s->fmt_gate_up, w->up, h->up, L, f, d, "up", mats));
  DS4_TRY(repack_stack(h, s->fmt_down, w->down, h->down, L, d, f, "down", mats));
  if (owned) {
    DS4_TRY(h->alloc_t(&h->local_of, (size_t)E * 4));
    DS4_TRY(copy_in(h->local_of, local_of.data(), (size_t)E * 4, s->device, "expert map"));
  }
  if (s->n_shared) {
    h->mb_sgu = ds4::matrix_bytes(s->fmt_shared, fs, d);
    h->mb_sd = ds4::matrix_bytes(s->fmt_shared, d, fs);
    DS4_TRY(h->alloc_t(&h->sgate, h->mb_sgu));
    DS4_TRY(h->alloc_t(&h->sup, h->mb_sgu));
    DS4_TRY(h->alloc_t(&h->sdown, h->mb_sd));
    DS4_TRY(repack_stack(h, s->fmt_shared, w->shared_gate, h->sgate, 1, fs, d, "shared_gate"));
    DS4_TRY(repack_stack(h, s->fmt_shared, w->shared_up, h->sup, 1, fs, d, "shared_up"));
    DS4_TRY(repack_stack(h, s->fmt_shared, w->shared_down, h->sdown, 1, d, fs, "shared_down"));
  }
  if (s->hash_vocab > 0) {
    DS4_TRY(h->alloc_t(&h->table, (size_t)s->hash_vocab * K * 4));
    DS4_TRY(copy_in(h->table, w->hash_table, (size_t)s->hash_vocab * K * 4, s->device, "hash_table"));
    DS4_TRY(check_table(h->table, (size_t)s->hash_vocab, K, E));
  }
  // workspace for max_tokens
  const size_t M = (size_t)s->max_tokens, slots = M * K;
  DS4_TRY(h->alloc_t(&h->logits, M * E * 4));
  DS4_TRY(h->alloc_t(&h->idx, slots * 4));
  DS4_TRY(h->alloc_t(&h->wts, slots * 4));
  DS4_TRY(h->alloc_t(&h->counts, (size_t)E * 4));
  DS4_TRY(h->alloc_t(&h->offsets, (size_t)(E + 1) * 4));
  DS4_TRY(h->alloc_t(&h->active, (size_t)E * 4));
  DS4_TRY(h->alloc_t(&h->n_active, 4));
  DS4_TRY(h->alloc_t(&h->perm, slots * 4));
  DS4_TRY(h->alloc_t(&h->rowof, slots * 4));
  DS4_TRY(h->alloc_t(&h->ghist, (size_t)ds4::bucket_chunks((int)slots) * E * 4));
  const size_t Md = std::min<size_t>(M, (size_t)ds4::decode_max_tokens());  // decode buffers
  DS4_TRY(h->alloc_t(&h->H, Md * K * f * 4));
  if (s->n_shared) {
    DS4_TRY(h->alloc_t(&h->Hs, Md * fs * 4));
    DS4_TRY(h->alloc_t(&h->hsg, Md * (size_t)(fs / 16) * 4));
  }
  // The batched path is needed beyond the decode kernels' limits, and serves smaller forwards from
  // small_batch_from tokens on when the weights allow its fp16 dequantization (a handle that only
  // needs it for small forwards falls back to the decode path rather than refusing the weights).
  const bool need_batched = M > (size_t)ds4::decode_max_tokens() || slots > (size_t)ds4::decode_max_slots();
  h->has_prefill = need_batched;
  bool scales_checked = false;
  if (!need_batched && M >= (size_t)small_batch_from) {
    const int sc = check_q2k_scales(h);
    if (sc == DS4MOE_OK)
      h->has_prefill = scales_checked = true;
    else if (sc != DS4MOE_ERR_UNSUPPORTED_FORMAT)
      DS4_TRY(sc);
  }
  if (h->has_prefill) h->decode_upto = small_batch_from - 1;
  if (h->has_prefill) {
    DS4_TRY(h->alloc_t(&h->Y, slots * d * 4));
    DS4_TRY(h->alloc_t(&h->Xs16, M * d * 2));
    DS4_TRY(h->alloc_t(&h->Xp16, slots * d * 2));
    DS4_TRY(h->alloc_t(&h->H16, slots * f * 2));
    DS4_TRY(h->alloc_t(&h->inv_s, M * 4));
    DS4_TRY(h->alloc_t(&h->inv_p, slots * 4));
    const size_t max_tiles = std::max(max_routed_tiles(slots, E, routed_tile_n(0)), max_routed_tiles(slots, E, routed_tile_n(1)));
    DS4_TRY(h->alloc_t(&h->tiles, max_tiles * sizeof(int4)));
    DS4_TRY(h->alloc_t(&h->n_tiles, 4));
    if (s->n_shared) {
      DS4_TRY(h->alloc_t(&h->Ys, M * d * 4));
      DS4_TRY(h->alloc_t(&h->Hs16, M * fs * 2));
    }
    int tr = ds4::make_act_maps(&h->tm_xp, h->Xp16, slots, d);
    if (!tr) tr = ds4::make_act_maps(&h->tm_xs, h->Xs16, M, d);
    if (!tr) tr = ds4::make_act_maps(&h->tm_h, h->H16, slots, f);
    if (!tr && s->n_shared) tr = ds4::make_act_maps(&h->tm_hs, h->Hs16, M, fs);
    if (tr) DS4_TRY(fail(DS4MOE_ERR_CUDA, "tensor map encoding failed (%d)", tr));
    if (!scales_checked) DS4_TRY(check_q2k_scales(h));
    DS4_TRY(h->alloc_t(&h->router_w3, (size_t)3 * E * d * 2));
    ds4::launch_router_split(h->router_w, (size_t)E * d, h->router_w3, 0);
  }
  DS4_TRY(h->alloc_t(&h->err, 4));
  DS4_TRY(h->alloc_t(&h->xmax, M * 4));
  DS4_TRY(h->alloc_t(&h->hmax, (slots + M) * 4));
  DS4_TRY(h->alloc_t(&h->counter, 4));
  DS4_TRY(h->alloc_t(&h->work, (size_t)E * sizeof(int4)));
  DS4_TRY(h->alloc_t(&h->tokof, slots * 4));
  DS4_TRY(h->alloc_t(&h->xscale, M * 4));
  DS4_TRY(h->alloc_t(&h->x_stage, M * d * 2));
  DS4_TRY(h->alloc_t(&h->tid_stage, M * 4));
  DS4_TRY(h->alloc_t(&h->out_stage, M * d * 4));
  cudaError_t e = ds4::decode_prepare();
  if (e == cudaSuccess) e = ds4::gemm_prepare();
  if (e == cudaSuccess) e = ds4::router_tc_prepare();
  if (e == cudaSuccess) e = ds4::router_logits_prepare();
  if (e == cudaSuccess) e = cudaMemset(h->err, 0, 4);
  if (e == cudaSuccess) e = cudaMemset(h->counts, 0, (size_t)E * 4);
  if (e == cudaSuccess) e = cudaMemset(h->n_active, 0, 4);
  if (e == cudaSuccess) e = cudaMemset(h->counter, 0, 4);
  if (e == cudaSuccess) e = cudaMemset(h->hmax, 0, (slots + M) * 4);
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e != cudaSuccess) {
    rc = fail(DS4MOE_ERR_CUDA, "workspace init: %s", cudaGetErrorString(e));
    h->release();
    delete h;
    return rc;
  }
  *out = h;
  return DS4MOE_OK;
}

extern "C" int ds4moe_create(const ds4moe_weights* w, const ds4moe_shapes* s, ds4moe_handle** out) {
  return create_impl(w, s, nullptr, 0, 1, out);
}

extern "C" int ds4moe_create_subset(const ds4moe_weights* w, const ds4moe_shapes* s, const int32_t* owned,
                                    int32_t n_owned, int32_t include_shared, ds4moe_handle** out) {
  if (!owned) {
    if (out) *out = nullptr;
    return fail(DS4MOE_ERR_INVALID_ARG, "owned is NULL");
  }
  return create_impl(w, s, owned, n_owned, include_shared, out);
}

// Arguments of the decode kernels for one forward over the handle's workspace.
static ds4::DecodeArgs decode_args(ds4moe_handle* h, const __nv_bfloat16* xb, int n, const int32_t* token_ids, int n_hash,
                            float* out) {
  const ds4moe_shapes& s = h->s;
  ds4::DecodeArgs da{};
  da.x = xb; da.n_tok = n; da.d = s.d; da.wr = h->router_w; da.br = h->router_b; da.n_exp = s.n_experts;
  da.top_k = s.top_k; da.token_ids = token_ids; da.n_hash = n_hash; da.table = h->table; da.vocab = s.hash_vocab;
  da.logits = h->logits; da.xmax = h->xmax; da.idx = h->idx; da.wts = h->wts; da.counts = h->counts;
  da.offsets = h->offsets; da.active = h->active; da.n_active = h->n_active; da.perm = h->perm;
  da.rowof = h->rowof; da.err = h->err; da.counter = h->counter; da.hmax = h->hmax;
  da.work = h->work; da.tokof = h->tokof; da.xscale = h->xscale;
  da.gate = h->gate; da.up = h->up; da.down = h->down; da.mb_gu = h->mb_gu; da.mb_d = h->mb_d; da.f = s.f_routed;
  da.sgate = h->sgate; da.sup = h->sup; da.sdown = h->sdown; da.mb_sgu = h->mb_sgu; da.mb_sd = h->mb_sd;
  da.fs = s.f_shared; da.n_shared = s.n_shared; da.H = h->H; da.Hs = h->Hs; da.hsg = h->hsg; da.out = out;
  da.local_of = h->local_of;
  return da;
}

static bool is_decode(const ds4moe_handle* h, int n) {
  return n <= h->decode_upto && n <= ds4::decode_max_tokens() && n * h->s.top_k <= ds4::decode_max_slots();
}

// Host memory that is page-locked (a graph may copy from and to it). Asked of the driver on every
// call: a buffer freed and reallocated at the same address may have changed kind.
static bool host_pinned(const void* p) {
  cudaPointerAttributes at{};
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return at.type == cudaMemoryTypeHost;
}

// The address by which kernels reach page-locked host memory (null if they cannot, or if it is not
// 16-byte aligned).
static void* kernel_view(const void* p) {
  cudaPointerAttributes at{};
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  if (at.type != cudaMemoryTypeHost || !at.devicePointer || ((uintptr_t)at.devicePointer & 15)) return nullptr;
  return at.devicePointer;
}

// Tokens up to which the batched path routes with the fp32 FMA router kernel.
constexpr int kSmallRouterTokens = 32;

// The batched path's launches on stream st (router, top-k, bucketing, activation prep and gather,
// tile list, the expert GEMMs, combine); mark(name) follows each launch.
template <typename Mark>
static int batched_launches(ds4moe_handle* h, const __nv_bfloat16* xb, int n, const int32_t* token_ids, int n_hash,
                            float* out, cudaStream_t st, Mark&& mark) {
  const ds4moe_shapes& s = h->s;
  const int E = s.n_experts, K = s.top_k, d = s.d, f = s.f_routed, fs = s.f_shared;
  const int n_learned = n - n_hash;
  if (n_learned > 0) {
    // a few tokens: the fp32 FMA router (one warp per expert); more: the tensor-core router, whose
    // tiles cover 64 experts each and would leave most SMs idle
    if (n_learned <= kSmallRouterTokens)
      ds4::launch_router_logits(xb + (size_t)n_hash * d, n_learned, d, h->router_w, h->router_b, E, h->logits, st);
    else
      ds4::launch_router_tc(xb + (size_t)n_hash * d, n_learned, d, h->router_w3, h->router_b, E, h->logits, st);
    mark("router_logits");
  }
  DS4_CUDA(cudaMemsetAsync(h->err, 0, 4, st));
  ds4::launch_topk(h->logits, n_learned, E, K, token_ids, n_hash, h->table, s.hash_vocab, h->idx, h->wts, h->err, st);
  mark("topk");
  ds4::launch_bucket_count(h->idx, n * K, E, h->local_of, h->ghist, st);
  mark("bucket_count");
  ds4::launch_bucket_scatter(h->idx, n * K, E, h->ghist, h->local_of, h->counts, h->offsets, h->active, h->n_active,
                             h->perm, h->rowof, st);
  mark("bucket_scatter");
  ds4::launch_xprep(xb, n, d, h->Xs16, h->inv_s, st);
  mark("xprep");
  ds4::launch_gather(h->Xs16, h->inv_s, h->perm, h->offsets + E, n * K, K, d, h->Xp16, h->inv_p, st);
  mark("gather");
  const int k_gcd = std::gcd(std::gcd(d, f), s.n_shared ? fs : d);  // the K of every GEMM of the forward
  const int geom = ds4::gemm_geometry(n, K, E, k_gcd);
  const int TN = routed_tile_n(geom);  // one tiling serves the gate/up and the down GEMM
  ds4::launch_tiles(h->counts, h->offsets, E, h->local_of, TN, h->tiles, h->n_tiles, st);
  mark("tiles");
  const int routed_tiles = (int)max_routed_tiles((size_t)n * K, E, TN), dense_tiles = (n + TN - 1) / TN;
  ds4::GemmArgs g{};
  g.w0 = h->gate; g.w1 = h->up; g.mat_bytes = h->mb_gu; g.k = d; g.tiles = h->tiles; g.n_tiles = h->n_tiles;
  g.inv_scale = h->inv_p; g.h_out = h->H16; g.ld_out = f; g.err = h->err;
  if (h->test_stall) {  // one-shot: withhold one arrival, waits give up after ~1 ms (2e6 cycles)
    g.test_stall = h->test_stall;
    g.timeout_cycles = 2000000;
    h->test_stall = 0;
  }
  cudaError_t ge = ds4::launch_gemm(s.fmt_gate_up, true, h->tm_xp, g, f / 64, routed_tiles, geom, st);
  if (ge != cudaSuccess) return fail(DS4MOE_ERR_CUDA, "gate/up GEMM launch: %s", cudaGetErrorString(ge));
  mark("routed_gateup");
  if (s.n_shared) {
    ds4::GemmArgs gs{};
    gs.w0 = h->sgate; gs.w1 = h->sup; gs.k = d; gs.n_rows = n; gs.inv_scale = h->inv_s; gs.h_out = h->Hs16;
    gs.ld_out = fs; gs.err = h->err;
    ge = ds4::launch_gemm(s.fmt_shared, true, h->tm_xs, gs, fs / 64, dense_tiles, geom, st);
    if (ge != cudaSuccess) return fail(DS4MOE_ERR_CUDA, "shared gate/up GEMM launch: %s", cudaGetErrorString(ge));
    mark("shared_gateup");
  }
  ds4::GemmArgs gd{};
  gd.w0 = h->down; gd.mat_bytes = h->mb_d; gd.k = f; gd.tiles = h->tiles; gd.n_tiles = h->n_tiles;
  gd.y_out = h->Y; gd.ld_out = d; gd.err = h->err;
  ge = ds4::launch_gemm(s.fmt_down, false, h->tm_h, gd, d / 128, routed_tiles, geom, st);
  if (ge != cudaSuccess) return fail(DS4MOE_ERR_CUDA, "down GEMM launch: %s", cudaGetErrorString(ge));
  mark("routed_down");
  if (s.n_shared) {
    ds4::GemmArgs gsd{};
    gsd.w0 = h->sdown; gsd.k = fs; gsd.n_rows = n; gsd.y_out = h->Ys; gsd.ld_out = d; gsd.err = h->err;
    ge = ds4::launch_gemm(s.fmt_shared, false, h->tm_hs, gsd, d / 128, dense_tiles, geom, st);
    if (ge != cudaSuccess) return fail(DS4MOE_ERR_CUDA, "shared down GEMM launch: %s", cudaGetErrorString(ge));
    mark("shared_down");
  }
  ds4::launch_combine(h->idx, h->wts, h->rowof, h->Y, s.n_shared ? h->Ys : nullptr, n, K, d, out, st);
  mark("combine");
  DS4_CUDA(cudaGetLastError());
  return DS4MOE_OK;
}

extern "C" int ds4moe_forward_ex(ds4moe_handle* h, const void* x, int32_t n, const int32_t* token_ids,
                                 int32_t n_hash, float* out, void* stream) {
  if (!h) return fail(DS4MOE_ERR_INVALID_ARG, "handle is NULL");
  const ds4moe_shapes& s = h->s;
  if (n < 0) return fail(DS4MOE_ERR_INVALID_ARG, "n_tokens=%d is negative", n);
  if (n > s.max_tokens) return fail(DS4MOE_ERR_CAPACITY, "n_tokens=%d exceeds max_tokens=%d", n, s.max_tokens);
  if (n_hash < 0 || n_hash > n) return fail(DS4MOE_ERR_INVALID_ARG, "n_hash=%d must be in 0..n_tokens", n_hash);
  if (n_hash > 0 && (s.hash_vocab == 0 || !token_ids))
    return fail(DS4MOE_ERR_INVALID_ARG, "n_hash=%d needs a handle with a hash table and token_ids", n_hash);
  if (n == 0) return DS4MOE_OK;
  if (!x || !out) return fail(DS4MOE_ERR_INVALID_ARG, "x or out is NULL");
  if (((uintptr_t)x & 15) || ((uintptr_t)out & 15)) return fail(DS4MOE_ERR_INVALID_ARG, "x and out must be 16-byte aligned");
  const void* ptrs[3] = {x, out, n_hash ? token_ids : nullptr};
  const char* names[3] = {"x", "out", "token_ids"};
  for (int i = 0; i < 3; ++i) {
    if (!ptrs[i]) continue;
    bool seen = false;  // pointers already verified on this handle skip the driver query
    for (const void* p : h->checked)
      if (p == ptrs[i]) seen = true;
    if (seen) continue;
    const PtrKind k = classify(ptrs[i], s.device);
    if (k == PTR_OTHER_DEVICE) return fail(DS4MOE_ERR_DEVICE_MISMATCH, "%s lives on another device than the handle's (%d)", names[i], s.device);
    if (k != PTR_DEVICE) return fail(DS4MOE_ERR_INVALID_ARG, "%s is not device memory (use ds4moe_forward_host for host buffers)", names[i]);
    h->checked[h->checked_next++ % ds4moe_handle::kChecked] = ptrs[i];
  }
  DeviceGuard guard(s.device);
  if (!guard.ok) return fail(DS4MOE_ERR_CUDA, "cannot select device %d", s.device);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const auto* xb = static_cast<const __nv_bfloat16*>(x);
  int phase = 0;
  if (h->profile) DS4_CUDA(cudaEventRecord(h->ev[0], st));
  auto mark = [&](const char* name) {
    if (h->profile && phase < ds4moe_handle::kMaxPhases) {
      h->phase_name[phase] = name;
      cudaEventRecord(h->ev[++phase], st);
    }
  };
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  DS4_CUDA(cudaStreamIsCapturing(st, &cap));
  // direct launches when profiling, when graphs are off, and when the caller is capturing its own graph
  const bool direct = h->profile || cap != cudaStreamCaptureStatusNone || !h->use_graphs;
  cudaGraphExec_t exec = nullptr;
  if (is_decode(h, n)) {
    // decode path: three kernels, chained with programmatic dependent launch unless profiling
    const ds4::DecodeArgs da = decode_args(h, xb, n, token_ids, n_hash, out);
    if (direct) {
      struct Ctx {
        decltype(mark)* m;
      } ctx{&mark};
      ds4::DecodeHooks hooks{[](void* c, const char* name) { (*static_cast<Ctx*>(c)->m)(name); }, &ctx};
      cudaError_t e = ds4::launch_decode(da, s.fmt_gate_up, s.fmt_down, s.fmt_shared, !h->profile, st, nullptr,
                                         h->profile ? &hooks : nullptr);
      if (e != cudaSuccess) return fail(DS4MOE_ERR_CUDA, "decode launch: %s", cudaGetErrorString(e));
    } else {
      int rc = h->cached_graph(0, n, n_hash, x, token_ids, out, nullptr, [&](cudaStream_t cs) {
        const cudaError_t e = ds4::launch_decode(da, s.fmt_gate_up, s.fmt_down, s.fmt_shared, true, cs, nullptr, nullptr);
        return e == cudaSuccess ? (int)DS4MOE_OK : fail(DS4MOE_ERR_CUDA, "decode launch: %s", cudaGetErrorString(e));
      }, &exec);
      if (rc != DS4MOE_OK) return rc;
      DS4_CUDA(cudaGraphLaunch(exec, st));
    }
  } else {
    if (!h->has_prefill) return fail(DS4MOE_ERR_CAPACITY, "n_tokens=%d needs the batched path, not sized at create", n);
    if (direct || h->test_stall) {  // (the timeout test's one-shot setting is not captured)
      int rc = batched_launches(h, xb, n, token_ids, n_hash, out, st, mark);
      if (rc != DS4MOE_OK) return rc;
    } else {
      int rc = h->cached_graph(1, n, n_hash, x, token_ids, out, nullptr, [&](cudaStream_t cs) {
        return batched_launches(h, xb, n, token_ids, n_hash, out, cs, [](const char*) {});
      }, &exec);
      if (rc != DS4MOE_OK) return rc;
      DS4_CUDA(cudaGraphLaunch(exec, st));
    }
  }
  h->n_phases = phase;
  h->last_stream = st;
  h->last_n = n;
  return DS4MOE_OK;
}

extern "C" int ds4moe_forward(ds4moe_handle* h, const void* x, int32_t n, float* out, void* stream) {
  return ds4moe_forward_ex(h, x, n, nullptr, 0, out, stream);
}

extern "C" int ds4moe_forward_host(ds4moe_handle* h, const void* x_host, int32_t n, const int32_t* tid_host,
                                   int32_t n_hash, float* out_host, void* stream) {
  if (!h) return fail(DS4MOE_ERR_INVALID_ARG, "handle is NULL");
  if (n < 0 || n > h->s.max_tokens)
    return fail(n < 0 ? DS4MOE_ERR_INVALID_ARG : DS4MOE_ERR_CAPACITY, "n_tokens=%d outside 0..max_tokens=%d", n, h->s.max_tokens);
  if (n == 0) return DS4MOE_OK;
  if (!x_host || !out_host || (n_hash > 0 && !tid_host)) return fail(DS4MOE_ERR_INVALID_ARG, "x, out or token_ids is NULL");
  if (n_hash < 0 || n_hash > n) return fail(DS4MOE_ERR_INVALID_ARG, "n_hash=%d must be in 0..n_tokens", n_hash);
  if (n_hash > 0 && h->s.hash_vocab == 0)
    return fail(DS4MOE_ERR_INVALID_ARG, "n_hash=%d needs a handle with a hash table and token_ids", n_hash);
  DeviceGuard guard(h->s.device);
  if (!guard.ok) return fail(DS4MOE_ERR_CUDA, "cannot select device %d", h->s.device);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t d = (size_t)h->s.d;
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  DS4_CUDA(cudaStreamIsCapturing(st, &cap));
  if (h->use_graphs && !h->profile && !h->test_stall && cap == cudaStreamCaptureStatusNone &&
      (is_decode(h, n) || h->has_prefill) && host_pinned(x_host) && host_pinned(out_host) &&
      (n_hash == 0 || host_pinned(tid_host))) {
    // one graph: host -> device copies, the forward's kernels, device -> host copy
    const auto* xs = reinterpret_cast<const __nv_bfloat16*>(h->x_stage);
    const int* ts = n_hash > 0 ? h->tid_stage : nullptr;
    ds4moe_handle::HostIo io;
    io.x = x_host;
    io.tid = n_hash > 0 ? tid_host : nullptr;
    io.out = out_host;
    if (h->sm_copies) {
      io.x_k = kernel_view(x_host);
      io.out_k = static_cast<float*>(kernel_view(out_host));
    }
    cudaGraphExec_t exec = nullptr;
    int rc;
    if (is_decode(h, n)) {
      const ds4::DecodeArgs da = decode_args(h, xs, n, ts, n_hash, h->out_stage);
      rc = h->cached_graph(0, n, n_hash, h->x_stage, ts, h->out_stage, &io, [&](cudaStream_t cs) {
        const cudaError_t e = ds4::launch_decode(da, h->s.fmt_gate_up, h->s.fmt_down, h->s.fmt_shared, true, cs, nullptr,
                                                 nullptr);
        return e == cudaSuccess ? (int)DS4MOE_OK : fail(DS4MOE_ERR_CUDA, "decode launch: %s", cudaGetErrorString(e));
      }, &exec);
    } else {
      rc = h->cached_graph(1, n, n_hash, h->x_stage, ts, h->out_stage, &io, [&](cudaStream_t cs) {
        return batched_launches(h, xs, n, ts, n_hash, h->out_stage, cs, [](const char*) {});
      }, &exec);
    }
    if (rc != DS4MOE_OK) return rc;
    DS4_CUDA(cudaGraphLaunch(exec, st));
    DS4_CUDA(cudaStreamSynchronize(st));
    h->n_phases = 0;
    h->last_stream = st;
    h->last_n = n;
    return DS4MOE_OK;
  }
  DS4_CUDA(cudaMemcpyAsync(h->x_stage, x_host, (size_t)n * d * 2, cudaMemcpyHostToDevice, st));
  if (n_hash > 0) DS4_CUDA(cudaMemcpyAsync(h->tid_stage, tid_host, (size_t)n_hash * 4, cudaMemcpyHostToDevice, st));
  int rc = ds4moe_forward_ex(h, h->x_stage, n, n_hash > 0 ? h->tid_stage : nullptr, n_hash, h->out_stage, stream);
  if (rc != DS4MOE_OK) return rc;
  DS4_CUDA(cudaMemcpyAsync(out_host, h->out_stage, (size_t)n * d * 4, cudaMemcpyDeviceToHost, st));
  DS4_CUDA(cudaStreamSynchronize(st));
  return DS4MOE_OK;
}

extern "C" int ds4moe_get_route(ds4moe_handle* h, int32_t* idx_host, float* w_host, int32_t n) {
  if (!h || !idx_host || !w_host) return fail(DS4MOE_ERR_INVALID_ARG, "NULL argument");
  if (n < 0 || n > h->last_n) return fail(DS4MOE_ERR_INVALID_ARG, "n_tokens=%d exceeds the last forward's %d", n, h->last_n);
  DeviceGuard guard(h->s.device);
  DS4_CUDA(cudaStreamSynchronize(h->last_stream));
  const size_t sl = (size_t)n * h->s.top_k;
  DS4_CUDA(cudaMemcpy(idx_host, h->idx, sl * 4, cudaMemcpyDeviceToHost));
  DS4_CUDA(cudaMemcpy(w_host, h->wts, sl * 4, cudaMemcpyDeviceToHost));
  return DS4MOE_OK;
}

extern "C" int ds4moe_get_stats(ds4moe_handle* h, ds4moe_stats* st) {
  if (!h || !st) return fail(DS4MOE_ERR_INVALID_ARG, "NULL argument");
  DeviceGuard guard(h->s.device);
  DS4_CUDA(cudaStreamSynchronize(h->last_stream));
  memset(st, 0, sizeof *st);
  st->n_tokens = h->last_n;
  if (h->last_n > 0) {
    DS4_CUDA(cudaMemcpy(st->counts, h->counts, (size_t)h->s.n_experts * 4, cudaMemcpyDeviceToHost));
    DS4_CUDA(cudaMemcpy(&st->distinct_experts, h->n_active, 4, cudaMemcpyDeviceToHost));
    DS4_CUDA(cudaMemcpy(&st->error_flags, h->err, 4, cudaMemcpyDeviceToHost));
  }
  return DS4MOE_OK;
}

extern "C" int64_t ds4moe_device_bytes(const ds4moe_handle* h) { return h ? h->bytes : 0; }

extern "C" int32_t ds4moe_launches_per_forward(const ds4moe_handle* h, int32_t n_tokens) {
  if (!h || n_tokens <= 0) return 0;
  if (is_decode(h, n_tokens)) return 3;  // route, gate/up, down + combine
  // router, top-k, 2 bucketing, activation prep + gather, tile list, routed gate/up and down GEMMs,
  // the same for the shared expert, combine
  return 1 + 1 + 2 + 2 + 1 + 2 + (h->s.n_shared ? 2 : 0) + 1;
}

extern "C" int ds4moe_set_test_stall(ds4moe_handle* h, int32_t stage) {
  if (!h) return fail(DS4MOE_ERR_INVALID_ARG, "handle is NULL");
  if (stage < 0) return fail(DS4MOE_ERR_INVALID_ARG, "stage=%d is negative", stage);
  h->test_stall = stage + 1;
  return DS4MOE_OK;
}

extern "C" int ds4moe_set_profiling(ds4moe_handle* h, int32_t enable) {
  if (!h) return fail(DS4MOE_ERR_INVALID_ARG, "handle is NULL");
  DeviceGuard guard(h->s.device);
  if (enable && !h->ev[0])
    for (cudaEvent_t& e : h->ev) DS4_CUDA(cudaEventCreate(&e));
  h->profile = enable != 0;
  h->n_phases = 0;
  return DS4MOE_OK;
}

extern "C" int ds4moe_get_phase_times(ds4moe_handle* h, float* ms, const char** names, int32_t max_phases,
                                      int32_t* n_phases) {
  if (!h || !n_phases) return fail(DS4MOE_ERR_INVALID_ARG, "NULL argument");
  DeviceGuard guard(h->s.device);
  *n_phases = h->profile ? h->n_phases : 0;
  if (*n_phases == 0) return DS4MOE_OK;
  DS4_CUDA(cudaEventSynchronize(h->ev[h->n_phases]));
  for (int i = 0; i < h->n_phases && i < max_phases; ++i) {
    if (ms) DS4_CUDA(cudaEventElapsedTime(&ms[i], h->ev[i], h->ev[i + 1]));
    if (names) names[i] = h->phase_name[i];
  }
  return DS4MOE_OK;
}

extern "C" void ds4moe_destroy(ds4moe_handle* h) {
  if (!h) return;
  DeviceGuard guard(h->s.device);
  cudaDeviceSynchronize();
  h->release();
  delete h;
}

extern "C" const char* ds4moe_last_error(void) { return g_last_error.c_str(); }
