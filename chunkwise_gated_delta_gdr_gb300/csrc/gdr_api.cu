// gdr_api.cu -- the C ABI: argument checks, workspace layout, path choice.
//
// Every entry point validates its arguments before enqueuing anything and
// reports failures as gdr_status codes; nothing here allocates device memory.
#include <math.h>
#include <string.h>

#include "gdr_internal.cuh"

namespace gdr {
namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

gdr_status check_dims(const gdr_dims* d, int chunk_size, int gate_mode) {
  if (!d) return GDR_ERR_INVALID_ARG;
  if (d->B < 0 || d->T < 0 || d->H <= 0 || d->HV <= 0 || d->K <= 0 || d->V <= 0)
    return GDR_ERR_INVALID_ARG;
  if (d->HV % d->H != 0) return GDR_ERR_INVALID_ARG;
  if (gate_mode != GDR_GATE_SCALAR && gate_mode != GDR_GATE_PER_KEY && gate_mode != GDR_GATE_NONE)
    return GDR_ERR_INVALID_ARG;
  if ((d->in_dtype != GDR_F32 && d->in_dtype != GDR_BF16) ||
      (d->out_dtype != GDR_F32 && d->out_dtype != GDR_BF16))
    return GDR_ERR_INVALID_ARG;
  if (chunk_size != 16 && chunk_size != 32 && chunk_size != 64 && chunk_size != 128)
    return GDR_ERR_UNSUPPORTED;
  // The general path streams K and V in tiles; its state kernel keeps a K x 32
  // state tile in shared memory.
  if (d->K > 256 || d->V > 256) return GDR_ERR_UNSUPPORTED;
  if (d->HV > 65535 || d->B > 65535) return GDR_ERR_UNSUPPORTED;
  // Element counts must fit the kernels' 64-bit indexing and the grid limits.
  if ((long long)d->T * d->HV * (d->V > d->K ? d->V : d->K) > (1LL << 46)) return GDR_ERR_UNSUPPORTED;
  return GDR_OK;
}

Problem make_problem(const void* q, const void* k, const void* v, const float* g,
                     const float* beta, const float* s0, int chunk_size, float scale,
                     int use_l2, int gate_mode, void* out, float* sT, const gdr_dims* d) {
  Problem p;
  p.q = q; p.k = k; p.v = v; p.g = g; p.beta = beta; p.s0 = s0; p.out = out; p.sT = sT;
  p.B = d->B; p.T = d->T; p.H = d->H; p.HV = d->HV; p.K = d->K; p.V = d->V;
  p.C = chunk_size;
  p.N = (d->T + chunk_size - 1) / chunk_size;
  p.in_bf16 = d->in_dtype == GDR_BF16;
  p.out_bf16 = d->out_dtype == GDR_BF16;
  // Ungated: the scalar-gate path with g identically zero (g is never read).
  p.gate_mode = gate_mode == GDR_GATE_NONE ? GDR_GATE_SCALAR : gate_mode;
  if (gate_mode == GDR_GATE_NONE) p.g = nullptr;
  p.use_l2 = use_l2 != 0;
  p.scale = scale;
  return p;
}

size_t body_bytes(const Problem& p) {
  if (tc_supported(p)) return tc_workspace_bytes(p);
  return general_workspace_bytes(p);
}

size_t elem_in(const gdr_dims* d) { return d->in_dtype == GDR_BF16 ? 2 : 4; }
// Bytes of g for a gate mode (none for the ungated mode).
size_t gate_bytes(const gdr_dims* d, int gate_mode) {
  if (gate_mode == GDR_GATE_NONE) return 0;
  return (size_t)d->B * d->T * d->HV * (gate_mode == GDR_GATE_PER_KEY ? d->K : 1) * sizeof(float);
}
size_t elem_out(const gdr_dims* d) { return d->out_dtype == GDR_BF16 ? 2 : 4; }

struct HostLayout {
  size_t q, k, v, g, beta, s0, out, sT, ws, total;
};

HostLayout host_layout(const gdr_dims* d, int chunk_size, int gate_mode, int with_s0, int with_sT) {
  HostLayout L;
  const size_t BT = (size_t)d->B * d->T;
  const size_t qk = BT * d->H * d->K * elem_in(d);
  const size_t vv = BT * d->HV * d->V * elem_in(d);
  const size_t gg = gate_bytes(d, gate_mode);
  const size_t bb = BT * d->HV * sizeof(float);
  const size_t st = (size_t)d->B * d->HV * d->K * d->V * sizeof(float);
  const size_t oo = BT * d->HV * d->V * elem_out(d);
  size_t off = 0;
  L.q = off; off += align_up(qk);
  L.k = off; off += align_up(qk);
  L.v = off; off += align_up(vv);
  L.g = off; off += align_up(gg);
  L.beta = off; off += align_up(bb);
  L.s0 = off; off += with_s0 ? align_up(st) : 0;
  L.out = off; off += align_up(oo);
  L.sT = off; off += with_sT ? align_up(st) : 0;
  L.ws = off; off += gdr_chunk_fwd_workspace_size(d, chunk_size, gate_mode);
  L.total = off;
  return L;
}

}  // namespace
}  // namespace gdr

using namespace gdr;

extern "C" {

int gdr_version(void) { return (0 << 16) | (1 << 8) | 0; }

const char* gdr_status_string(gdr_status s) {
  switch (s) {
    case GDR_OK: return "GDR_OK";
    case GDR_ERR_INVALID_ARG: return "GDR_ERR_INVALID_ARG: invalid argument";
    case GDR_ERR_UNSUPPORTED: return "GDR_ERR_UNSUPPORTED: shape, chunk size or dtype not supported";
    case GDR_ERR_ALIGNMENT: return "GDR_ERR_ALIGNMENT: tensor base not 16-byte aligned";
    case GDR_ERR_WORKSPACE: return "GDR_ERR_WORKSPACE: workspace missing or too small";
    case GDR_ERR_CUDA: return "GDR_ERR_CUDA: CUDA runtime or launch error";
    case GDR_ERR_TIMEOUT: return "GDR_ERR_TIMEOUT: a device-side bounded wait gave up";
  }
  return "unknown gdr_status";
}

size_t gdr_chunk_fwd_workspace_size(const gdr_dims* dims, int chunk_size, int gate_mode) {
  if (check_dims(dims, chunk_size, gate_mode) != GDR_OK) return 0;
  Problem p = make_problem(nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, chunk_size,
                           1.f, 0, gate_mode, nullptr, nullptr, dims);
  return sizeof(WorkspaceHeader) + align_up(body_bytes(p));
}

size_t gdr_ssd_chunk_fwd_workspace_size(const gdr_dims* dims, int chunk_size, int gate_mode) {
  if (check_dims(dims, chunk_size, gate_mode) != GDR_OK) return 0;
  Problem p = make_problem(nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, chunk_size,
                           1.f, 0, gate_mode, nullptr, nullptr, dims);
  p.ssd = 1;
  return sizeof(WorkspaceHeader) + align_up(body_bytes(p));
}

int gdr_chunk_fwd_path(const gdr_dims* dims, int chunk_size, int gate_mode, gdr_status* status) {
  gdr_status st = check_dims(dims, chunk_size, gate_mode);
  if (status) *status = st;
  if (st != GDR_OK) return -1;
  Problem p = make_problem(nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, chunk_size,
                           1.f, 0, gate_mode, nullptr, nullptr, dims);
  if (!tc_supported(p)) return 0;
  return tc_one_launch(p) ? 2 : 1;
}

}  // extern "C"

namespace {

// Shared body of gdr_chunk_fwd (stage 3), gdr_chunk_prepare (1) and
// gdr_chunk_recur (2).
gdr_status run(int stage, const void* q, const void* k, const void* v, const float* g,
               const float* beta, const float* initial_state, int chunk_size, float scale,
               int use_qk_l2norm, int gate_mode, void* out, float* final_state,
               const gdr_dims* dims, void* workspace, size_t workspace_bytes,
               gdr_stream_t stream, int ssd = 0, int zero_u = 0, int recur_mode = 0) {
  gdr_status st = check_dims(dims, chunk_size, gate_mode);
  if (st != GDR_OK) return st;
  if (!(isfinite(scale) && scale > 0.f)) return GDR_ERR_INVALID_ARG;
  const bool work = dims->B > 0 && dims->T > 0;
  if (work && (!q || !k)) return GDR_ERR_INVALID_ARG;
  if (work && (stage & 1) && (!v || (!g && gate_mode != GDR_GATE_NONE) || (!beta && !ssd)))
    return GDR_ERR_INVALID_ARG;
  if (work && (stage & 2) && !out) return GDR_ERR_INVALID_ARG;
  const void* ptrs[] = {q, k, v, g, beta, initial_state, out, final_state};
  for (const void* ptr : ptrs)
    if (ptr && !aligned16(ptr)) return GDR_ERR_ALIGNMENT;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const size_t state_bytes = (size_t)dims->B * dims->HV * dims->K * dims->V * sizeof(float);
  if (dims->B == 0) return GDR_OK;
  if (dims->T == 0) {
    if (!(stage & 2) || !final_state) return GDR_OK;
    cudaError_t e = initial_state
                        ? (final_state == initial_state
                               ? cudaSuccess
                               : cudaMemcpyAsync(final_state, initial_state, state_bytes,
                                                 cudaMemcpyDeviceToDevice, s))
                        : cudaMemsetAsync(final_state, 0, state_bytes, s);
    return e == cudaSuccess ? GDR_OK : GDR_ERR_CUDA;
  }
  const size_t need = ssd ? gdr_ssd_chunk_fwd_workspace_size(dims, chunk_size, gate_mode)
                          : gdr_chunk_fwd_workspace_size(dims, chunk_size, gate_mode);
  if (!workspace || workspace_bytes < need) return GDR_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & (kAlign - 1)) != 0) return GDR_ERR_ALIGNMENT;

  Problem p = make_problem(q, k, v, g, beta, initial_state, chunk_size, scale, use_qk_l2norm,
                           gate_mode, out, final_state, dims);
  p.ssd = ssd;
  p.zero_u = zero_u;
  p.recur_mode = recur_mode;
  auto* hdr = static_cast<WorkspaceHeader*>(workspace);
  if ((stage & 1) &&
      cudaMemsetAsync(&hdr->error_word, 0, sizeof(unsigned int), s) != cudaSuccess)
    return GDR_ERR_CUDA;
  void* body = static_cast<char*>(workspace) + sizeof(WorkspaceHeader);
  if (tc_supported(p)) return launch_tc(p, body, &hdr->error_word, s, stage);
  if (recur_mode == 2) return GDR_OK;   // the general path writes outputs with the states
  return launch_general(p, body, s, stage);
}

}  // namespace

extern "C" {

gdr_status gdr_chunk_fwd(const void* q, const void* k, const void* v, const float* g,
                         const float* beta, const float* initial_state, int chunk_size,
                         float scale, int use_qk_l2norm, int gate_mode, void* out,
                         float* final_state, const gdr_dims* dims, void* workspace,
                         size_t workspace_bytes, gdr_stream_t stream) {
  return run(3, q, k, v, g, beta, initial_state, chunk_size, scale, use_qk_l2norm, gate_mode,
             out, final_state, dims, workspace, workspace_bytes, stream);
}

gdr_status gdr_chunk_prepare(const void* q, const void* k, const void* v, const float* g,
                             const float* beta, int chunk_size, float scale, int use_qk_l2norm,
                             int gate_mode, const gdr_dims* dims, void* workspace,
                             size_t workspace_bytes, gdr_stream_t stream) {
  return run(1, q, k, v, g, beta, nullptr, chunk_size, scale, use_qk_l2norm, gate_mode, nullptr,
             nullptr, dims, workspace, workspace_bytes, stream);
}

gdr_status gdr_ssd_chunk_fwd(const void* q, const void* k, const void* v, const float* g,
                             const float* initial_state, int chunk_size, float scale,
                             int use_qk_l2norm, int gate_mode, void* out, float* final_state,
                             const gdr_dims* dims, void* workspace, size_t workspace_bytes,
                             gdr_stream_t stream) {
  return run(3, q, k, v, g, nullptr, initial_state, chunk_size, scale, use_qk_l2norm, gate_mode,
             out, final_state, dims, workspace, workspace_bytes, stream, 1);
}

gdr_status gdr_chunk_recur(const void* q, const void* k, const float* initial_state,
                           int chunk_size, float scale, int use_qk_l2norm, int gate_mode,
                           void* out, float* final_state, const gdr_dims* dims, void* workspace,
                           size_t workspace_bytes, gdr_stream_t stream) {
  return run(2, q, k, nullptr, nullptr, nullptr, initial_state, chunk_size, scale, use_qk_l2norm,
             gate_mode, out, final_state, dims, workspace, workspace_bytes, stream);
}

size_t gdr_chunk_fwd_host_buffer_size(const gdr_dims* dims, int chunk_size, int gate_mode,
                                      int with_initial_state, int with_final_state) {
  if (check_dims(dims, chunk_size, gate_mode) != GDR_OK) return 0;
  return host_layout(dims, chunk_size, gate_mode, with_initial_state, with_final_state).total;
}

gdr_status gdr_chunk_fwd_host(const void* q, const void* k, const void* v, const float* g,
                              const float* beta, const float* initial_state, int chunk_size,
                              float scale, int use_qk_l2norm, int gate_mode, void* out,
                              float* final_state, const gdr_dims* dims, void* device_buffer,
                              size_t device_buffer_bytes, gdr_stream_t stream) {
  gdr_status st = check_dims(dims, chunk_size, gate_mode);
  if (st != GDR_OK) return st;
  if (!(isfinite(scale) && scale > 0.f)) return GDR_ERR_INVALID_ARG;
  const bool work = dims->B > 0 && dims->T > 0;
  if (work && (!q || !k || !v || (!g && gate_mode != GDR_GATE_NONE) || !beta || !out))
    return GDR_ERR_INVALID_ARG;
  const void* ptrs[] = {q, k, v, g, beta, initial_state, out, final_state};
  for (const void* ptr : ptrs)
    if (ptr && !aligned16(ptr)) return GDR_ERR_ALIGNMENT;
  HostLayout L = host_layout(dims, chunk_size, gate_mode, initial_state != nullptr,
                             final_state != nullptr);
  if (!device_buffer || device_buffer_bytes < L.total) return GDR_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(device_buffer) & (kAlign - 1)) != 0) return GDR_ERR_ALIGNMENT;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  char* dev = static_cast<char*>(device_buffer);
  const size_t BT = (size_t)dims->B * dims->T;
  const size_t qk = BT * dims->H * dims->K * elem_in(dims);
  const size_t vv = BT * dims->HV * dims->V * elem_in(dims);
  const size_t gg = gate_bytes(dims, gate_mode);
  const size_t bb = BT * dims->HV * sizeof(float);
  const size_t stb = (size_t)dims->B * dims->HV * dims->K * dims->V * sizeof(float);
  const size_t oo = BT * dims->HV * dims->V * elem_out(dims);
  struct Copy { void* dst; const void* src; size_t n; };
  const Copy in[] = {{dev + L.q, q, qk}, {dev + L.k, k, qk}, {dev + L.v, v, vv},
                     {dev + L.g, g, gg}, {dev + L.beta, beta, bb},
                     {dev + L.s0, initial_state, initial_state ? stb : 0}};
  for (const Copy& c : in) {
    if (c.n == 0 || !c.src) continue;
    if (cudaMemcpyAsync(c.dst, c.src, c.n, cudaMemcpyHostToDevice, s) != cudaSuccess)
      return GDR_ERR_CUDA;
  }
  st = gdr_chunk_fwd(dev + L.q, dev + L.k, dev + L.v, reinterpret_cast<const float*>(dev + L.g),
                     reinterpret_cast<const float*>(dev + L.beta),
                     initial_state ? reinterpret_cast<const float*>(dev + L.s0) : nullptr,
                     chunk_size, scale, use_qk_l2norm, gate_mode, dev + L.out,
                     final_state ? reinterpret_cast<float*>(dev + L.sT) : nullptr, dims,
                     dev + L.ws, device_buffer_bytes - L.ws, stream);
  if (st != GDR_OK) return st;
  if (oo && cudaMemcpyAsync(out, dev + L.out, oo, cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return GDR_ERR_CUDA;
  if (final_state &&
      cudaMemcpyAsync(final_state, dev + L.sT, stb, cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return GDR_ERR_CUDA;
  return GDR_OK;
}

int64_t gdr_set_flag_wait_limit(int64_t polls) { return set_wait_limit(polls); }

gdr_status gdr_stream_status(gdr_stream_t stream, void* workspace) {
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return GDR_ERR_CUDA;
  if (cudaGetLastError() != cudaSuccess) return GDR_ERR_CUDA;
  if (!workspace) return GDR_OK;
  unsigned int word = 0;
  auto* hdr = static_cast<WorkspaceHeader*>(workspace);
  if (cudaMemcpy(&word, &hdr->error_word, sizeof word, cudaMemcpyDeviceToHost) != cudaSuccess)
    return GDR_ERR_CUDA;
  return word ? GDR_ERR_TIMEOUT : GDR_OK;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Segmented scan (gdr_segment.cu has the plan).
namespace {

struct SegLayout {
  size_t inner, bst, ast, sin, oscr, total;
};

// The sequences viewed as B P sequences of T / P tokens.
gdr_dims segment_dims(const gdr_dims* d, int P) {
  gdr_dims d2 = *d;
  d2.B = d->B * P;
  d2.T = d->T / P;
  return d2;
}

SegLayout seg_layout(const gdr_dims* d2, int chunk_size, int gate_mode) {
  SegLayout L;
  const size_t st = (size_t)d2->B * d2->HV * d2->K * d2->V * sizeof(float);
  const size_t oo = (size_t)d2->B * d2->T * d2->HV * d2->V * elem_out(d2);
  size_t off = 0;
  L.inner = gdr_chunk_fwd_workspace_size(d2, chunk_size, gate_mode);
  off = align_up(L.inner);
  L.bst = off; off += align_up(st);
  L.ast = off; off += align_up(st);
  L.sin = off; off += align_up(st);
  L.oscr = off; off += align_up(oo);
  L.total = off;
  return L;
}

gdr_status segment_check(const gdr_dims* d, int chunk_size, int gate_mode, int segments) {
  const gdr_status st = check_dims(d, chunk_size, gate_mode);
  if (st != GDR_OK) return st;
  if (segments < 1) return GDR_ERR_INVALID_ARG;
  if (segments == 1) return GDR_OK;
  if (d->K != d->V) return GDR_ERR_UNSUPPORTED;               // A_p is a K x K state
  if (d->T % (segments * chunk_size) != 0) return GDR_ERR_UNSUPPORTED;
  const gdr_dims d2 = segment_dims(d, segments);
  return check_dims(&d2, chunk_size, gate_mode);
}

}  // namespace

extern "C" {

size_t gdr_chunk_fwd_segmented_workspace_size(const gdr_dims* dims, int chunk_size, int gate_mode,
                                              int segments) {
  if (segment_check(dims, chunk_size, gate_mode, segments) != GDR_OK) return 0;
  if (segments == 1) return gdr_chunk_fwd_workspace_size(dims, chunk_size, gate_mode);
  const gdr_dims d2 = segment_dims(dims, segments);
  return seg_layout(&d2, chunk_size, gate_mode).total;
}

gdr_status gdr_chunk_fwd_segmented(const void* q, const void* k, const void* v, const float* g,
                                   const float* beta, const float* initial_state,
                                   int chunk_size, float scale, int use_qk_l2norm, int gate_mode,
                                   int segments, void* out, float* final_state,
                                   const gdr_dims* dims, void* workspace,
                                   size_t workspace_bytes, gdr_stream_t stream) {
  gdr_status st = segment_check(dims, chunk_size, gate_mode, segments);
  if (st != GDR_OK) return st;
  if (segments == 1 || dims->B == 0 || dims->T == 0)
    return gdr_chunk_fwd(q, k, v, g, beta, initial_state, chunk_size, scale, use_qk_l2norm,
                         gate_mode, out, final_state, dims, workspace, workspace_bytes, stream);
  if (!(isfinite(scale) && scale > 0.f)) return GDR_ERR_INVALID_ARG;
  if (!q || !k || !v || !out || (!g && gate_mode != GDR_GATE_NONE) || !beta)
    return GDR_ERR_INVALID_ARG;
  const gdr_dims d2 = segment_dims(dims, segments);
  const SegLayout L = seg_layout(&d2, chunk_size, gate_mode);
  if (!workspace || workspace_bytes < L.total) return GDR_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & (kAlign - 1)) != 0) return GDR_ERR_ALIGNMENT;
  if ((initial_state && !aligned16(initial_state)) || (final_state && !aligned16(final_state)))
    return GDR_ERR_ALIGNMENT;
  char* base = static_cast<char*>(workspace);
  float* Bst = reinterpret_cast<float*>(base + L.bst);
  float* Ast = reinterpret_cast<float*>(base + L.ast);
  float* Sin = reinterpret_cast<float*>(base + L.sin);
  void* oscr = base + L.oscr;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // 1. chunk-local kernel on the B P segments
  st = run(1, q, k, v, g, beta, nullptr, chunk_size, scale, use_qk_l2norm, gate_mode, nullptr,
           nullptr, &d2, workspace, L.inner, stream);
  if (st != GDR_OK) return st;
  // 2. B_p: each segment from a zero state (states only where outputs are separate)
  st = run(2, q, k, nullptr, nullptr, nullptr, nullptr, chunk_size, scale, use_qk_l2norm,
           gate_mode, oscr, Bst, &d2, workspace, L.inner, stream, 0, 0, 1);
  if (st != GDR_OK) return st;
  // 3. A_p: each segment from the identity, U read as zero (final state in place)
  st = launch_segment_identity(Ast, (long)d2.B * d2.HV, d2.K, s);
  if (st != GDR_OK) return st;
  st = run(2, q, k, nullptr, nullptr, nullptr, Ast, chunk_size, scale, use_qk_l2norm, gate_mode,
           oscr, Ast, &d2, workspace, L.inner, stream, 0, 1, 1);
  if (st != GDR_OK) return st;
  // 4. segment initial states and the final state
  st = launch_segment_combine(Ast, Bst, initial_state, Sin, final_state, dims->B, segments,
                              dims->HV, dims->K, s);
  if (st != GDR_OK) return st;
  // 5. each segment from its true initial state, states and outputs (for the
  // scalar gate on tensor cores: the chains with their output items beside
  // them in one launch when they fit on the SMs at once)
  return run(2, q, k, nullptr, nullptr, nullptr, Sin, chunk_size, scale, use_qk_l2norm, gate_mode,
             out, nullptr, &d2, workspace, L.inner, stream, 0, 0, 0);
}

}  // extern "C"
