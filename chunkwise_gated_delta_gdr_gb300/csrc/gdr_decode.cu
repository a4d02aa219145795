// gdr_decode.cu -- the token-by-token (recurrent) form of the gated delta rule,
// the step a decoder takes for each generated token.
//
// For each (batch b, value head hv) and token t, in order, the recurrence the
// "分块并行计算（Chunkwise）" notes start from (section "为什么需要分块？"):
//     S   <- diag(exp(g_t)) S                    (decay; scalar or per key channel)
//     S   <- S + beta_t k_t (v_t - S^T k_t)^T     (delta write)
//     o_t  = S^T (scale q_t)
// with q_t, k_t optionally L2-normalised. The state S [K][V] fp32 is read from
// `state` once, kept in registers across the T tokens of the call and written
// back once, in place: the per-token HBM traffic is the token's q, k, v, gate
// and o, and a call's total is one read and one write of every state.
//
// One CTA per (V tile of 32 columns, hv, b), 16 warps: warp w holds state rows
// [8 w, 8 w + 8) of the tile's columns (lane = column), so every state access
// is a coalesced 128-byte row segment; 64 registers per thread keep two CTAs
// (32 warps) per SM in flight, which the HBM stream needs. Per token the column sums
// (S^T k and S^T q over all rows) are combined across the warps through
// shared memory; everything else is per element.
#include <math.h>

#include "gdr_internal.cuh"

namespace gdr {
namespace {

constexpr int kWarps = 16, kRows = 128 / kWarps, kThreads = kWarps * 32, kCols = 32;
static_assert(kWarps * kRows == 128, "rows per CTA must cover K <= 128");

struct DecodeArgs {
  const void* q;
  const void* k;
  const void* v;
  const float* g;       // [B,T,HV] or [B,T,HV,K]; null: ungated
  const float* beta;    // [B,T,HV]
  float* state;         // [B,HV,K,V], updated in place
  void* out;            // [B,T,HV,V]
  int B, T, H, HV, K, V;
  int in_bf16, out_bf16, per_key, use_l2;
  float scale;
};

__device__ __forceinline__ float ld_x(const void* p, size_t i, int bf16) {
  if (bf16) return __bfloat162float(static_cast<const __nv_bfloat16*>(p)[i]);
  return static_cast<const float*>(p)[i];
}

__global__ void __launch_bounds__(kThreads, 2) recurrent_kernel(DecodeArgs a) {
  __shared__ float kr[128], qr[128], dec[128];
  __shared__ float red_u[kWarps][kCols], red_o[kWarps][kCols];
  __shared__ float tok[4];   // |k|^-1, scale |q|^-1, beta, q~ . k^
  const int vt = blockIdx.x, hv = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int h = hv / (a.HV / a.H);
  const int K = a.K, V = a.V;
  const int col = vt * kCols + lane;
  const bool cok = col < V;
  const int r0 = warp * kRows;
  const size_t sbase = ((size_t)b * a.HV + hv) * K * V;

  float S[kRows];
#pragma unroll
  for (int i = 0; i < kRows; ++i) {
    const int c = r0 + i;
    S[i] = (c < K && cok) ? a.state[sbase + (size_t)c * V + col] : 0.f;
  }

  for (int t = 0; t < a.T; ++t) {
    const size_t bt = (size_t)b * a.T + t;
    // Every load of the token is issued up front, beside the state loads.
    const float vv = cok ? ld_x(a.v, (bt * a.HV + hv) * V + col, a.in_bf16) : 0.f;
    const float bet = tid == 0 ? a.beta[bt * a.HV + hv] : 0.f;
    if (tid < K) {
      const size_t qk = (bt * a.H + h) * K + tid;
      kr[tid] = ld_x(a.k, qk, a.in_bf16);
      qr[tid] = ld_x(a.q, qk, a.in_bf16);
      float g = 0.f;
      if (a.g) g = a.per_key ? a.g[(bt * a.HV + hv) * K + tid] : a.g[bt * a.HV + hv];
      dec[tid] = expf(g);
    }
    __syncthreads();
    if (warp == 0) {
      float sk = 0.f, sq = 0.f, sqk = 0.f;
      for (int c = lane; c < K; c += 32) {
        sk = fmaf(kr[c], kr[c], sk);
        sq = fmaf(qr[c], qr[c], sq);
        sqk = fmaf(qr[c], kr[c], sqk);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        sk += __shfl_xor_sync(0xffffffffu, sk, o);
        sq += __shfl_xor_sync(0xffffffffu, sq, o);
        sqk += __shfl_xor_sync(0xffffffffu, sqk, o);
      }
      if (lane == 0) {
        const float nk = a.use_l2 ? 1.f / sqrtf(sk + 1e-6f) : 1.f;
        const float nq = a.scale * (a.use_l2 ? 1.f / sqrtf(sq + 1e-6f) : 1.f);
        tok[0] = nk;
        tok[1] = nq;
        tok[2] = bet;
        tok[3] = nq * nk * sqk;
      }
    }
    __syncthreads();
    const float nk = tok[0], nq = tok[1], beta = tok[2], qk = tok[3];
    // Decay, then this warp's share of (D S)^T k^ and (D S)^T q~.
    float pu = 0.f, po = 0.f;
#pragma unroll
    for (int i = 0; i < kRows; ++i) {
      const int c = r0 + i;
      if (c < K) {
        S[i] *= dec[c];
        pu = fmaf(kr[c] * nk, S[i], pu);
        po = fmaf(qr[c] * nq, S[i], po);
      }
    }
    red_u[warp][lane] = pu;
    red_o[warp][lane] = po;
    __syncthreads();
    float u = 0.f, oq = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      u += red_u[w][lane];
      oq += red_o[w][lane];
    }
    const float wv = beta * (vv - u);                 // delta-rule write of this column
#pragma unroll
    for (int i = 0; i < kRows; ++i) {
      const int c = r0 + i;
      if (c < K) S[i] = fmaf(kr[c] * nk, wv, S[i]);
    }
    if (warp == 0 && cok) {
      const float o = fmaf(qk, wv, oq);               // S'^T q~ = (D S)^T q~ + (q~ . k^) w
      const size_t off = (bt * a.HV + hv) * V + col;
      if (a.out_bf16)
        static_cast<__nv_bfloat16*>(a.out)[off] = __float2bfloat16_rn(o);
      else
        static_cast<float*>(a.out)[off] = o;
    }
    __syncthreads();   // kr / qr / dec / red are rewritten by the next token
  }

#pragma unroll
  for (int i = 0; i < kRows; ++i) {
    const int c = r0 + i;
    if (c < K && cok) a.state[sbase + (size_t)c * V + col] = S[i];
  }
}

}  // namespace
}  // namespace gdr

using namespace gdr;

extern "C" gdr_status gdr_recurrent_fwd(const void* q, const void* k, const void* v, const float* g,
                                        const float* beta, float* state, float scale,
                                        int use_qk_l2norm, int gate_mode, void* out,
                                        const gdr_dims* d, gdr_stream_t stream) {
  if (!d) return GDR_ERR_INVALID_ARG;
  if (d->B < 0 || d->T < 0 || d->H <= 0 || d->HV <= 0 || d->K <= 0 || d->V <= 0 ||
      d->HV % d->H != 0)
    return GDR_ERR_INVALID_ARG;
  if (gate_mode != GDR_GATE_SCALAR && gate_mode != GDR_GATE_PER_KEY && gate_mode != GDR_GATE_NONE)
    return GDR_ERR_INVALID_ARG;
  if ((d->in_dtype != GDR_F32 && d->in_dtype != GDR_BF16) ||
      (d->out_dtype != GDR_F32 && d->out_dtype != GDR_BF16))
    return GDR_ERR_INVALID_ARG;
  if (!(isfinite(scale) && scale > 0.f)) return GDR_ERR_INVALID_ARG;
  if (d->K > 128) return GDR_ERR_UNSUPPORTED;
  if (d->HV > 65535 || d->B > 65535) return GDR_ERR_UNSUPPORTED;
  if (d->B == 0 || d->T == 0) return GDR_OK;
  if (!q || !k || !v || !beta || !state || !out || (!g && gate_mode != GDR_GATE_NONE))
    return GDR_ERR_INVALID_ARG;
  DecodeArgs a;
  a.q = q;
  a.k = k;
  a.v = v;
  a.g = gate_mode == GDR_GATE_NONE ? nullptr : g;
  a.beta = beta;
  a.state = state;
  a.out = out;
  a.B = d->B;
  a.T = d->T;
  a.H = d->H;
  a.HV = d->HV;
  a.K = d->K;
  a.V = d->V;
  a.in_bf16 = d->in_dtype == GDR_BF16;
  a.out_bf16 = d->out_dtype == GDR_BF16;
  a.per_key = gate_mode == GDR_GATE_PER_KEY;
  a.use_l2 = use_qk_l2norm != 0;
  a.scale = scale;
  dim3 grid((d->V + kCols - 1) / kCols, d->HV, d->B);
  recurrent_kernel<<<grid, kThreads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(a);
  return cudaGetLastError() == cudaSuccess ? GDR_OK : GDR_ERR_CUDA;
}
