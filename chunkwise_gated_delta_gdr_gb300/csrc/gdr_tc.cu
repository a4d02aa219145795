// gdr_tc.cu -- dispatch of the fast path (bf16 inputs, K = V = 128, C = 64).
#include <atomic>

#include "gdr_fast.cuh"

namespace gdr {

bool tc_supported(const Problem& p) {
  // SSD with the per-key gate stays on the general path.
  // (the scalar gate's output pass puts the chunk index in gridDim.y)
  return !(p.ssd && p.gate_mode) && p.in_bf16 && p.K == fast::K && p.V == fast::V &&
         p.C == fast::C && (p.gate_mode != 0 || p.N <= 65535);
}

namespace {

// Polls of a chain's wait on a chunk flag (one-launch forward), about 64 ns
// apart: 2^24 is about a second.
constexpr long long kDefaultWaitLimit = 1LL << 24;
std::atomic<long long> g_wait_limit{kDefaultWaitLimit};

// Workspace body of the fast path: the chunk slabs, then (scalar gate) the
// exchange blocks the recurrence writes for the output pass and, for the
// one-launch forward, one ready flag per chunk, one export mark per (sequence,
// 32 value columns) and an output item counter.
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
    off += (nch + (size_t)p.B * p.HV * (fast::V / 32) + 1) * sizeof(unsigned int);
  }
  L.total = off;
  return L;
}

}  // namespace

long long set_wait_limit(long long polls) {
  return polls < 0 ? g_wait_limit.load() : g_wait_limit.exchange(polls);
}

size_t tc_workspace_bytes(const Problem& p) { return tc_layout(p).total; }

bool tc_one_launch(const Problem& p) {
  return tc_supported(p) && p.gate_mode == 0 && fast::fused_fits(p.B, p.HV);
}

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
  f.xmark = f.flags ? f.flags + (size_t)p.B * p.HV * p.N : nullptr;
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
  f.scale = p.scale;
  f.slab_bytes = fast::Slab::bytes(p.gate_mode);
  f.wait_limit = (long)g_wait_limit.load();
  // Both stages in one call, scalar gate: one cooperative launch when the
  // chains leave enough SMs to the producers.
  if (stage == 3 && p.gate_mode == 0 && p.recur_mode == 0) {
    const gdr_status st = fast::launch_fused(f, stream);
    if (st != GDR_ERR_UNSUPPORTED) return st;
  }
  if (stage & 1) {
    gdr_status st = fast::launch_chunk_tc(f, stream);
    if (st != GDR_OK) return st;
  }
  if (stage & 2) {
    // The per-key recurrence writes the outputs with the states (no separate
    // output pass, recur_mode 2 is nothing); the scalar-gate chain leaves them
    // to the output pass (recur_mode 1: the states alone).
    if (p.gate_mode) return p.recur_mode == 2 ? GDR_OK : fast::launch_state_kda_tc(f, stream);
    if (p.recur_mode == 0) {
      const gdr_status st = fast::launch_chain_outputs(f, stream);
      if (st != GDR_ERR_UNSUPPORTED) return st;
    }
    if (p.recur_mode != 2) {
      const gdr_status st = fast::launch_chain(f, stream);
      if (st != GDR_OK || p.recur_mode == 1) return st;
    }
    return fast::launch_outputs(f, stream);
  }
  return GDR_OK;
}

}  // namespace gdr
