// api.cu -- the extern "C" entry points of liblora_sgmv.so: argument
// validation, problem descriptors, kernel dispatch and the device status word.
// The routing builder (lora_build_routing) lives in routing.cpp.
#include <cmath>
#include <cstdint>
#include <mutex>

#include "internal.h"

namespace lora {

// Device status word: an OR of LORA_DEV_* flags raised by the kernels.
__device__ unsigned g_status_word;

// Where lora_get_device_status's exchange leaves the old value of the word.
__device__ unsigned g_status_snapshot;

// Kernel families and launch count of the current entry-point call on this
// host thread (lora_last_call_path).
thread_local unsigned t_path_bits = 0;
thread_local unsigned t_launches = 0;

void note_launch(unsigned path_bits) {
  t_path_bits |= path_bits;
  ++t_launches;
}

int device_sm_count() {
  static std::mutex mu;
  static int sms[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  std::lock_guard<std::mutex> lk(mu);
  if (!sms[dev]) {
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0) return 0;
    sms[dev] = v;
  }
  return sms[dev];
}

namespace {

void begin_call() {
  t_path_bits = 0;
  t_launches = 0;
}

std::mutex g_sym_mu;
unsigned* g_status_ptr[64] = {nullptr};
unsigned* g_snapshot_ptr[64] = {nullptr};

// Device addresses of the status word and its snapshot on the current
// device, looked up once per device (with that device current).
bool status_ptrs(unsigned** word, unsigned** snap) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
  std::lock_guard<std::mutex> lk(g_sym_mu);
  if (!g_status_ptr[dev] || !g_snapshot_ptr[dev]) {
    void* p = nullptr;
    void* q = nullptr;
    if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess || !p) return false;
    if (cudaGetSymbolAddress(&q, g_status_snapshot) != cudaSuccess || !q) return false;
    g_status_ptr[dev] = static_cast<unsigned*>(p);
    g_snapshot_ptr[dev] = static_cast<unsigned*>(q);
  }
  *word = g_status_ptr[dev];
  if (snap) *snap = g_snapshot_ptr[dev];
  return true;
}

unsigned* status_ptr() {
  unsigned* w = nullptr;
  return status_ptrs(&w, nullptr) ? w : nullptr;
}

// One thread: read and clear the status word in one atomic exchange.
__global__ void status_exchange_kernel(unsigned* word, unsigned* snap) { *snap = atomicExch(word, 0u); }

lora_status_t validate_problem(const lora_problem_t* p) {
  if (!p) return LORA_ERR_NULL;
  if (p->dtype != LORA_DTYPE_F32 && p->dtype != LORA_DTYPE_BF16) return LORA_ERR_DTYPE;
  if (p->num_tokens < 0 || p->in_dim < 1 || p->max_num_loras < 1 || p->max_lora_rank < 1 ||
      p->max_lora_rank > 1024)
    return LORA_ERR_SHAPE;
  if (p->num_slices < 1 || p->num_slices > LORA_MAX_SLICES) return LORA_ERR_SHAPE;
  if (!p->x) return LORA_ERR_NULL;
  if (p->x_row_stride < p->in_dim) return LORA_ERR_SHAPE;
  const long long R = p->max_lora_rank;
  for (int j = 0; j < p->num_slices; ++j) {
    const lora_slice_t& s = p->slices[j];
    if (!s.A || !s.B || !s.y) return LORA_ERR_NULL;
    if (s.out_dim < 1) return LORA_ERR_SHAPE;
    if (s.A_slot_stride < R * p->in_dim) return LORA_ERR_SHAPE;
    if (s.B_slot_stride < R * s.out_dim) return LORA_ERR_SHAPE;
    if (s.y_row_stride < s.out_dim) return LORA_ERR_SHAPE;
    if (s.bias && s.bias_slot_stride < s.out_dim) return LORA_ERR_SHAPE;
  }
  return LORA_OK;
}

lora_status_t validate_routing(const lora_problem_t* p, const lora_routing_t* r) {
  if (!r) return LORA_ERR_NULL;
  if (r->num_groups > p->max_num_loras) return LORA_ERR_TOO_MANY_GROUPS;
  if (r->num_groups < 0) return LORA_ERR_ROUTING;
  if (r->end < 0 || r->end > p->num_tokens) return LORA_ERR_ROUTING;
  if (r->num_groups == 0 && r->end != 0) return LORA_ERR_ROUTING;
  if (r->num_groups > 0 && (!r->lora_ids || !r->grouped_offsets)) return LORA_ERR_NULL;
  if (r->host_lora_ids && !r->host_grouped_offsets) return LORA_ERR_NULL;
  if (const int32_t* o = r->host_grouped_offsets) {
    if (r->num_groups > 0 && o[0] != 0) return LORA_ERR_ROUTING;
    for (int g = 0; g < r->num_groups; ++g)
      if (o[g + 1] < o[g]) return LORA_ERR_ROUTING;
    if (r->num_groups > 0 && o[r->num_groups] != r->end) return LORA_ERR_ROUTING;
  }
  if (const int32_t* ids = r->host_lora_ids)
    for (int g = 0; g < r->num_groups; ++g)
      if (ids[g] < 0 || ids[g] >= p->max_num_loras) return LORA_ERR_SLOT_RANGE;
  return LORA_OK;
}

// The launch-parameter summary of a validated routing's host triple (G = 0:
// no host copy of both arrays).
HostRouting host_routing(const lora_routing_t* r) {
  HostRouting h{};
  if (!r->host_grouped_offsets || !r->host_lora_ids) return h;
  h.G = r->num_groups;
  for (int g = 0; g < r->num_groups; ++g)
    h.digest += routing_digest_term(g, r->host_grouped_offsets[g], r->host_lora_ids[g]);
  return h;
}

ProblemDesc make_desc(const lora_problem_t* p, const lora_routing_t* r) {
  ProblemDesc d{};
  d.dtype = p->dtype;
  d.num_tokens = p->num_tokens;
  d.in_dim = p->in_dim;
  d.S = p->max_num_loras;
  d.R = p->max_lora_rank;
  d.n_slices = p->num_slices;
  d.x = p->x;
  d.x_row_stride = p->x_row_stride;
  for (int j = 0; j < p->num_slices; ++j) {
    const lora_slice_t& s = p->slices[j];
    d.sl[j] = SliceDesc{s.A, (long long)s.A_slot_stride, s.B, (long long)s.B_slot_stride,
                        s.out_dim, s.y, (long long)s.y_row_stride, s.bias, (long long)s.bias_slot_stride};
  }
  d.slot_ranks = p->slot_ranks;
  if (r) {
    d.lora_ids = r->lora_ids;
    d.offs = r->grouped_offsets;
    d.G = r->num_groups;
    d.end = r->end;
    d.token_rows = r->token_rows;
  }
  d.status = status_ptr();
  d.seg_lo = 0;
  d.seg_hi = 0x7FFFFFFF;
  return d;
}

lora_status_t cuda_status(cudaError_t e) { return e == cudaSuccess ? LORA_OK : LORA_ERR_CUDA; }

bool is_noop(const lora_routing_t* r) { return r->num_groups == 0 || r->end == 0; }

// One fp32 plane of the intermediate u [end, n*R].
size_t plane_bytes(const lora_problem_t* p, int32_t end) {
  const size_t raw = (size_t)(end > 0 ? end : 0) * (size_t)p->num_slices * (size_t)p->max_lora_rank * 4;
  return (raw + 255) & ~(size_t)255;
}

// lora_sgmv_apply's workspace holds the intermediate.  Its shrink may split the input dimension into up to 16 partial planes
// (apply_splits), summed by the expand; on the tensor-core path for ranks 64
// and 128 it holds u packed per 128-row tile (at most max_num_loras + end /
// 128 tiles), and when the kernels are picked per group both are live at
// once: the packed region first, the planes after it.
size_t planes_bound(const lora_problem_t* p, int32_t end) {
  int splits = apply_splits(end, p->in_dim, p->num_slices * p->max_lora_rank);
  const int tc = tc_shrink_splits(end, p->in_dim, kMaxSmsForWorkspace);
  if (tc > splits) splits = tc;
  const size_t raw = (size_t)splits * (size_t)(end > 0 ? end : 0) * (size_t)p->num_slices *
                     (size_t)p->max_lora_rank * 4;
  return (raw + 255) & ~(size_t)255;
}

size_t packed_region(const lora_problem_t* p, int32_t end) {
  const size_t packed = tc_packed_bytes(p->max_num_loras, end, p->num_slices, p->max_lora_rank);
  return (packed + 255) & ~(size_t)255;
}

size_t ws_bytes(const lora_problem_t* p, int32_t end) { return packed_region(p, end) + planes_bound(p, end); }

// Long groups (tcgen05 tiles) and short groups of a routing whose host copy
// of the offsets is given.
void count_classes(const lora_routing_t* r, int* n_long, int* n_short) {
  *n_long = *n_short = 0;
  const int32_t* o = r->host_grouped_offsets;
  for (int g = 0; g < r->num_groups; ++g) {
    const int len = o[g + 1] - o[g];
    if (len >= LORA_TC_MIN_ROWS) ++*n_long;
    else if (len > 0) ++*n_short;
  }
}

}  // namespace
}  // namespace lora

using namespace lora;

extern "C" lora_status_t lora_set_slot(const lora_problem_t* problem, int32_t slice, int32_t slot,
                                       int32_t r, double lora_alpha, int32_t use_rslora,
                                       const void* A_raw, const void* B_raw,
                                       lora_dtype_t raw_dtype, lora_stream_t stream) {
  begin_call();
  lora_status_t st = validate_problem(problem);
  if (st != LORA_OK) return st;
  if (slice < 0 || slice >= problem->num_slices) return LORA_ERR_SHAPE;
  if (slot < 0 || slot >= problem->max_num_loras) return LORA_ERR_SLOT_RANGE;
  if (r < 0 || r > problem->max_lora_rank) return LORA_ERR_RANK;
  if (raw_dtype != LORA_DTYPE_F32 && raw_dtype != LORA_DTYPE_BF16) return LORA_ERR_DTYPE;
  if (r > 0 && (!A_raw || !B_raw)) return LORA_ERR_NULL;
  float scale = 0.f;
  if (r > 0) {
    const double denom = use_rslora ? std::sqrt((double)r) : (double)r;
    scale = (float)(lora_alpha / denom);
  }
  ProblemDesc d = make_desc(problem, nullptr);
  return cuda_status(launch_set_slot(d, slice, slot, r, scale, A_raw, B_raw, raw_dtype,
                                     reinterpret_cast<cudaStream_t>(stream)));
}

extern "C" lora_status_t lora_set_slot_bias(const lora_problem_t* problem, int32_t slice, int32_t slot,
                                            const void* bias_raw, lora_dtype_t raw_dtype, lora_stream_t stream) {
  begin_call();
  lora_status_t st = validate_problem(problem);
  if (st != LORA_OK) return st;
  if (slice < 0 || slice >= problem->num_slices) return LORA_ERR_SHAPE;
  if (!problem->slices[slice].bias) return LORA_ERR_NULL;
  if (slot < 0 || slot >= problem->max_num_loras) return LORA_ERR_SLOT_RANGE;
  if (raw_dtype != LORA_DTYPE_F32 && raw_dtype != LORA_DTYPE_BF16) return LORA_ERR_DTYPE;
  ProblemDesc d = make_desc(problem, nullptr);
  return cuda_status(launch_set_bias(d, slice, slot, bias_raw, raw_dtype, reinterpret_cast<cudaStream_t>(stream)));
}

extern "C" lora_status_t lora_shrink(const lora_problem_t* problem, const lora_routing_t* routing,
                                     float* u, lora_stream_t stream) {
  begin_call();
  lora_status_t st = validate_problem(problem);
  if (st != LORA_OK) return st;
  if ((st = validate_routing(problem, routing)) != LORA_OK) return st;
  if (is_noop(routing)) return LORA_OK;
  if (!u) return LORA_ERR_NULL;
  ProblemDesc d = make_desc(problem, routing);
  if (!d.status) return LORA_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (fast_path_ok(d, u)) {
    if (tc_shrink_ok(d)) {
      const cudaError_t e = launch_tc_shrink(d, u, s, 1);
      if (e != cudaErrorNotSupported) return cuda_status(e);
    }
    return cuda_status(launch_shrink_bf16(d, u, s));
  }
  return cuda_status(launch_shrink_simple(d, u, s));
}

extern "C" lora_status_t lora_expand(const lora_problem_t* problem, const lora_routing_t* routing,
                                     const float* u, lora_stream_t stream) {
  begin_call();
  lora_status_t st = validate_problem(problem);
  if (st != LORA_OK) return st;
  if ((st = validate_routing(problem, routing)) != LORA_OK) return st;
  if (is_noop(routing)) return LORA_OK;
  if (!u) return LORA_ERR_NULL;
  ProblemDesc d = make_desc(problem, routing);
  if (!d.status) return LORA_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (fast_path_ok(d, u)) {
    if (tc_expand_ok(d)) {
      const cudaError_t e = launch_tc_expand(d, u, s, false, 1);
      if (e != cudaErrorNotSupported) return cuda_status(e);
    }
    return cuda_status(launch_expand_bf16(d, u, s, false, 1));
  }
  return cuda_status(launch_expand_simple(d, u, s, false));
}

extern "C" size_t lora_workspace_bytes(const lora_problem_t* problem, int32_t end) {
  if (!problem || problem->num_slices < 1 || problem->max_lora_rank < 1) return 0;
  return ws_bytes(problem, end);
}

extern "C" lora_status_t lora_sgmv_apply(const lora_problem_t* problem, const lora_routing_t* routing,
                                         void* workspace, size_t workspace_bytes,
                                         lora_stream_t stream) {
  begin_call();
  lora_status_t st = validate_problem(problem);
  if (st != LORA_OK) return st;
  if ((st = validate_routing(problem, routing)) != LORA_OK) return st;
  if (is_noop(routing)) return LORA_OK;
  if (!workspace || workspace_bytes < ws_bytes(problem, routing->end)) return LORA_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 15u) != 0) return LORA_ERR_ALIGN;
  ProblemDesc d = make_desc(problem, routing);
  if (!d.status) return LORA_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  void* inter = workspace;
  float* u = static_cast<float*>(inter);
  if (fast_path_ok(d, u) && routing->host_grouped_offsets && tc_expand_shapes_ok(d)) {
    // Kernels per group: the long groups on tcgen05 (packed u in the first
    // region), the short ones on mma.sync (planes in the second region).
    int n_long = 0, n_short = 0;
    count_classes(routing, &n_long, &n_short);
    if (n_long > 0 && n_short > 0) {
      ProblemDesc dl = d, ds = d;
      dl.seg_lo = LORA_TC_MIN_ROWS;
      ds.seg_hi = LORA_TC_MIN_ROWS;
      float* up = reinterpret_cast<float*>(static_cast<uint8_t*>(inter) + packed_region(problem, routing->end));
      cudaError_t e = launch_tc_apply_packed(dl, inter, s);
      if (e != cudaErrorNotSupported) {
        if ((st = cuda_status(e)) != LORA_OK) return st;
        int splits = 1;
        const HostRouting hr = host_routing(routing);
        if ((st = cuda_status(launch_shrink_partial_bf16(ds, up, s, routing, &splits))) != LORA_OK) return st;
        return cuda_status(launch_expand_bf16(ds, up, s, true, splits, &hr));
      }
    }
  }
  if (fast_path_ok(d, u)) {
    if (tc_expand_ok(d)) {
      const cudaError_t e = launch_tc_apply_packed(d, inter, s);
      if (e != cudaErrorNotSupported) return cuda_status(e);
    }
    if (tc_shrink_ok(d)) {
      const int tcs = tc_shrink_splits(d.end, d.in_dim, device_sm_count());
      const cudaError_t e = launch_tc_shrink(d, u, s, tcs);
      if (e != cudaErrorNotSupported) {
        if (e != cudaSuccess) return LORA_ERR_CUDA;
        return cuda_status(launch_expand_bf16(d, u, s, true, tcs));
      }
    }
    int splits = 1;
    const HostRouting hr = host_routing(routing);
    if ((st = cuda_status(launch_shrink_partial_bf16(d, u, s, routing, &splits))) != LORA_OK) return st;
    return cuda_status(launch_expand_bf16(d, u, s, true, splits, &hr));
  }
  if ((st = cuda_status(launch_shrink_simple(d, u, s))) != LORA_OK) return st;
  return cuda_status(launch_expand_simple(d, u, s, true));
}

extern "C" lora_status_t lora_get_device_status(lora_stream_t stream, uint32_t* flags) {
  begin_call();
  if (!flags) return LORA_ERR_NULL;
  unsigned *word = nullptr, *snap = nullptr;
  if (!status_ptrs(&word, &snap)) return LORA_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // The snapshot word is shared by the device's callers: one at a time.
  static std::mutex mu;
  std::lock_guard<std::mutex> lk(mu);
  status_exchange_kernel<<<1, 1, 0, s>>>(word, snap);
  if (cudaGetLastError() != cudaSuccess) return LORA_ERR_CUDA;
  unsigned v = 0;
  if (cudaMemcpyAsync(&v, snap, sizeof(v), cudaMemcpyDeviceToHost, s) != cudaSuccess) return LORA_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return LORA_ERR_CUDA;
  *flags = v;
  return LORA_OK;
}

extern "C" uint32_t lora_last_call_path(uint32_t* num_launches) {
  if (num_launches) *num_launches = t_launches;
  return t_path_bits;
}

extern "C" lora_status_t lora_base_gemm_apply(const lora_problem_t* problem, const lora_routing_t* routing,
                                              const lora_base_weight_t* base, void* workspace,
                                              size_t workspace_bytes, lora_stream_t stream) {
  begin_call();
  lora_status_t st = validate_problem(problem);
  if (st != LORA_OK) return st;
  if ((st = validate_routing(problem, routing)) != LORA_OK) return st;
  if (routing->token_rows) return LORA_ERR_SHAPE;  // rows must be in sorted order
  if (!base) return LORA_ERR_NULL;
  BaseWeights wts{};
  for (int j = 0; j < problem->num_slices; ++j) {
    if (!base[j].W0) return LORA_ERR_NULL;
    if (base[j].row_stride < problem->in_dim) return LORA_ERR_SHAPE;
    wts.W0[j] = base[j].W0;
    wts.row_stride[j] = (long long)base[j].row_stride;
  }
  if (problem->num_tokens == 0) return LORA_OK;
  const bool noop = is_noop(routing);
  if (!noop && (!workspace || workspace_bytes < ws_bytes(problem, routing->end))) return LORA_ERR_WORKSPACE;
  if (workspace && (reinterpret_cast<uintptr_t>(workspace) & 15u) != 0) return LORA_ERR_ALIGN;
  ProblemDesc d = make_desc(problem, routing);
  if (!d.status) return LORA_ERR_CUDA;
  if (noop) {  // base rows only: no groups to add
    d.G = 0;
    d.end = 0;
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  float* u = static_cast<float*>(workspace);
  if (base_tc_ok(d, wts) && (noop || fast_path_ok(d, u)) && base_maps_ok(d, wts)) {
    int nsplit = 0;
    if (!noop) {
      cudaError_t e = cudaErrorNotSupported;
      if (tc_shrink_ok(d)) {
        nsplit = tc_shrink_splits(d.end, d.in_dim, device_sm_count());
        e = launch_tc_shrink(d, u, s, nsplit);
      }
      if (e == cudaErrorNotSupported) {
        nsplit = apply_splits_for(d);
        e = launch_shrink_partial_bf16(d, u, s);
      }
      if ((st = cuda_status(e)) != LORA_OK) return st;
    }
    return cuda_status(launch_base_gemm(d, wts, u, nsplit, !noop, s));
  }
  if (!noop && (st = cuda_status(launch_shrink_simple(d, u, s))) != LORA_OK) return st;
  return cuda_status(launch_base_gemm_simple(d, wts, u, !noop, s));
}

extern "C" lora_status_t lora_selftest_wait_timeout(uint32_t polls, lora_stream_t stream) {
  begin_call();
  unsigned* p = status_ptr();
  if (!p) return LORA_ERR_CUDA;
  return cuda_status(launch_selftest_timeout(p, polls, reinterpret_cast<cudaStream_t>(stream)));
}

extern "C" const char* lora_status_string(lora_status_t status) {
  switch (status) {
    case LORA_OK: return "LORA_OK";
    case LORA_ERR_NULL: return "LORA_ERR_NULL: a required pointer is NULL";
    case LORA_ERR_SHAPE: return "LORA_ERR_SHAPE: a count, size or stride is out of range";
    case LORA_ERR_RANK: return "LORA_ERR_RANK: adapter rank exceeds max_lora_rank";
    case LORA_ERR_SLOT_RANGE: return "LORA_ERR_SLOT_RANGE: slot id out of range";
    case LORA_ERR_ROUTING: return "LORA_ERR_ROUTING: routing triple inconsistent";
    case LORA_ERR_DTYPE: return "LORA_ERR_DTYPE: unknown storage type";
    case LORA_ERR_ALIGN: return "LORA_ERR_ALIGN: pointer or stride misaligned";
    case LORA_ERR_WORKSPACE: return "LORA_ERR_WORKSPACE: workspace missing or too small";
    case LORA_ERR_CUDA: return "LORA_ERR_CUDA: a CUDA call failed";
    case LORA_ERR_TOO_MANY_GROUPS: return "LORA_ERR_TOO_MANY_GROUPS: more groups than adapter slots";
  }
  return "unknown lora_status_t";
}

// ---------------------------------------------------------------------------
// lora_sgmv_apply_noalloc: the same shrink + expand as lora_sgmv_apply, with
// the fp32 intermediate held in a fixed array compiled into the library
// instead of a caller-provided workspace.  For callers that cannot allocate
// device memory at all (see the header).
//
// The array is a file-scope __device__ variable: every GPU that loads this
// library holds it until the process exits.  Its name in host code is only a
// host-side stand-in, so the device address is looked up once per device
// with cudaGetSymbolAddress (with that device current) and cached.
// ---------------------------------------------------------------------------
namespace lora {
namespace {

constexpr size_t kStaticWorkspaceFloats = LORA_NOALLOC_MAX_WORKSPACE_BYTES / sizeof(float);
static_assert(kStaticWorkspaceFloats * sizeof(float) == LORA_NOALLOC_MAX_WORKSPACE_BYTES,
              "the limit must be a whole number of floats");

static __device__ __align__(256) float g_static_workspace[kStaticWorkspaceFloats];

std::mutex g_static_mu;
float* g_static_ptr[64] = {nullptr};

// Device address of the static workspace on the current device (nullptr on
// failure).  First call per device does the lookup.
float* static_workspace_ptr() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lk(g_static_mu);
  if (!g_static_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_workspace) != cudaSuccess || !p) return nullptr;
    g_static_ptr[dev] = static_cast<float*>(p);
  }
  return g_static_ptr[dev];
}

}  // namespace
}  // namespace lora

extern "C" lora_status_t lora_sgmv_apply_noalloc(const lora_problem_t* problem,
                                                 const lora_routing_t* routing,
                                                 lora_stream_t stream) {
  begin_call();
  lora_status_t st = validate_problem(problem);
  if (st != LORA_OK) return st;
  if ((st = validate_routing(problem, routing)) != LORA_OK) return st;
  if (is_noop(routing)) return LORA_OK;
  // Every byte of the intermediate that the expand reads is written by the
  // shrink of the same call, so nothing in the array has to start at zero.
  if (plane_bytes(problem, routing->end) > lora::kStaticWorkspaceFloats * sizeof(float))
    return LORA_ERR_WORKSPACE;
  float* u = static_workspace_ptr();
  if (!u) return LORA_ERR_CUDA;
  ProblemDesc d = make_desc(problem, routing);
  if (!d.status) return LORA_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (fast_path_ok(d, u)) {
    if ((st = cuda_status(launch_shrink_bf16(d, u, s))) != LORA_OK) return st;
    return cuda_status(launch_expand_bf16(d, u, s, true, 1));
  }
  if ((st = cuda_status(launch_shrink_simple(d, u, s))) != LORA_OK) return st;
  return cuda_status(launch_expand_simple(d, u, s, true));
}
