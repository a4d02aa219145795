// gdr_tc.cu -- dispatch of the fast path (bf16 inputs, K = V = 128, C = 64).
#include "gdr_fast.cuh"

namespace gdr {

bool tc_supported(const Problem& p) {
  // SSD with the per-key gate stays on the general path.
  return !(p.ssd && p.gate_mode) && p.in_bf16 && p.K == fast::K && p.V == fast::V && p.C == fast::C;
}

namespace {

// Workspace body of the fast path: the chunk slabs, then (scalar gate) the
// exchange blocks of the state chain and its per-chain progress flags.
struct TcLayout {
  size_t xchg = 0, flags = 0, total = 0;
};

TcLayout tc_layout(const Problem& p) {
  const size_t nch = (size_t)p.B * p.HV * p.N;
  TcLayout L;
  size_t off = nch * fast::Slab::bytes(p.gate_mode);
  if (p.gate_mode == 0) {
    off = align_up(off, 1024);
    L.xchg = off;
    off += nch * fast::Xchg::BYTES;
    off = align_up(off, 256);
    L.flags = off;
    off += (size_t)p.B * p.HV * (fast::V / fast::VT) * sizeof(unsigned int);
  }
  L.total = off;
  return L;
}

}  // namespace

size_t tc_workspace_bytes(const Problem& p) { return tc_layout(p).total; }

gdr_status launch_tc(const Problem& p, void* ws_body, unsigned int* error_word,
                     cudaStream_t stream, int stage) {
  fast::Params f;
  f.q = static_cast<const __nv_bfloat16*>(p.q);
  f.k = static_cast<const __nv_bfloat16*>(p.k);
  f.v = static_cast<const __nv_bfloat16*>(p.v);
  f.g = p.g;
  f.beta = p.beta;
  f.s0 = p.s0;
  f.out = p.out;
  f.sT = p.sT;
  f.slabs = static_cast<uint8_t*>(ws_body);
  const TcLayout L = tc_layout(p);
  f.xchg = p.gate_mode == 0 ? f.slabs + L.xchg : nullptr;
  f.flags = p.gate_mode == 0 ? reinterpret_cast<unsigned int*>(f.slabs + L.flags) : nullptr;
  f.error_word = error_word;
  f.B = p.B;
  f.T = p.T;
  f.H = p.H;
  f.HV = p.HV;
  f.N = p.N;
  f.out_bf16 = p.out_bf16;
  f.gate_mode = p.gate_mode;
  f.use_l2 = p.use_l2;
  f.ssd = p.ssd;
  f.zero_u = p.zero_u;
  f.recur_mode = p.recur_mode;
  f.zero_flags = (stage == 3 && f.flags) ? 1 : 0;
  f.scale = p.scale;
  f.slab_bytes = fast::Slab::bytes(p.gate_mode);
  if (stage & 1) {
    gdr_status st = fast::launch_chunk_tc(f, stream);
    if (st != GDR_OK) return st;
  }
  if (stage & 2) return fast::launch_state(f, stream);
  return GDR_OK;
}

}  // namespace gdr
