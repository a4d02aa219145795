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
// Main kernel (V <= 128 and a multiple of 4, state 16-byte aligned): one
// persistent CTA per SM walks the heads. Each head's whole state (K x V fp32,
// one TMA box of up to 512-byte rows) streams through a three-stage
// shared-memory ring, so about 190 KB per SM are in flight. Two groups of 8
// warps take alternate heads; a warp takes 16 rows x 4 consecutive columns per
// lane into registers, the group releases the stage at once (its first warp
// refills it with the head three places on while they apply the tokens) and
// writes the finished state back from registers, one 512-byte row per warp
// store. A group's barriers and column sums overlap the other group's work.
// (Boxes of 128-byte rows were served several times slower.)
//
// Fallback kernel (any V, K <= 256): one CTA per (V tile of 32 columns, hv, b),
// 16 warps: warp w holds state rows [R w, R w + R) of the tile's columns
// (lane = column; R = 8 for K <= 128, 16 for K <= 256), so every state access
// is a coalesced 128-byte row segment; with R = 8, 64 registers per thread keep
// two CTAs (32 warps) per SM in flight, which the HBM stream needs. Per token the column sums
// (S^T k and S^T q over all rows) are combined across the warps through
// shared memory; everything else is per element.
#include <math.h>
#include <string.h>

#include <cuda.h>

#include "gdr_internal.cuh"
#include "gdr_ptx.cuh"
#include "gdr_tmap.cuh"

namespace gdr {
namespace {

constexpr int kWarps = 16, kThreads = kWarps * 32, kCols = 32;

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
  unsigned int* error_word;   // null: waits that give up are not reported
};

__device__ __forceinline__ float ld_x(const void* p, size_t i, int bf16) {
  if (bf16) return __bfloat162float(static_cast<const __nv_bfloat16*>(p)[i]);
  return static_cast<const float*>(p)[i];
}

// kRows state rows per warp: the CTA covers K <= 16 kRows.
template <int kRows>
__global__ void __launch_bounds__(kThreads, 128 / (8 * kRows)) recurrent_kernel(DecodeArgs a) {
  __shared__ float kr[kWarps * kRows], qr[kWarps * kRows], dec[kWarps * kRows];
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

// ------------------------------------------------------------ pipelined kernel
// Whole-head tiles: the K x V state of one (b, hv) is one TMA box of V-element
// (up to 512-byte) rows, streamed through a three-stage ring. The 16 warps
// form two groups of 8 that take alternate heads of the CTA's list, each with
// its own named barriers and token staging, so one group's barriers and
// column sums overlap the other group's loads, arithmetic and stores. There is
// no producer warp (a 17th warp would cap every thread at 96 registers): once a
// group holds head i in registers, its first warp refills that stage with head
// i + STAGES.
namespace pipe {
constexpr int GROUPS = 2, GW = 8, CW = GROUPS * GW;   // warp groups, warps per group, compute warps
constexpr int ROWS = 16, CPL = 4;                    // rows per warp, consecutive columns per lane
constexpr int GT = GW * 32;                          // threads per group
constexpr int STAGES = 3, TILE = 128 * 128 * 4;      // 64 KB stage
constexpr int THREADS = CW * 32;
constexpr int OFF_BAR = STAGES * TILE, SMEM = OFF_BAR + 2 * STAGES * 8 + 1024;
constexpr long kWaitLimit = 1L << 24;
static_assert(GW * ROWS == 128 && CPL * 32 == 128, "a group's tile covers K, V <= 128");
static_assert(GT >= 128, "one group thread per channel and per column");
__device__ __forceinline__ void nb_sync(int id, int n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}
}  // namespace pipe

__global__ void __launch_bounds__(pipe::THREADS, 1)
    recurrent_pipe_kernel(const __grid_constant__ CUtensorMap smap, DecodeArgs a, int nplanes) {
  using namespace pipe;
  using namespace ptx;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  // Per warp group: the staged tokens (two buffers, alternating per token;
  // zero past K) and their beta, the warps' (k^T D S, q^T D S) partials per
  // column, the delta-rule write per column.
  __shared__ __align__(16) float kr[GROUPS][2][128], qr[GROUPS][2][128], dec[GROUPS][2][128];
  __shared__ __align__(16) float2 red[GROUPS][GW][128];
  __shared__ __align__(16) float wcol[GROUPS][128];
  __shared__ float tok[GROUPS][2];
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + OFF_BAR);
  uint64_t* done = full + STAGES;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int K = a.K, V = a.V;
  // Plane i of this CTA: blockIdx.x + i * gridDim.x (= b * HV + hv).
  const int my = nplanes > (int)blockIdx.x ? (nplanes - 1 - blockIdx.x) / gridDim.x + 1 : 0;
  const uint32_t tbytes = (uint32_t)K * V * 4;
  if (tid == 0) {
    for (int i = 0; i < STAGES; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&done[i], GW);
    }
    mbar_fence_init();
    // The first STAGES planes; stage s takes plane i + STAGES once the group
    // holding plane i has it in registers (below).
    for (int i = 0; i < STAGES && i < my; ++i) {
      mbar_expect_tx(&full[i], tbytes);
      tma_load3(smem_u32(sm + i * TILE), &smap, 0, 0, blockIdx.x + i * gridDim.x, &full[i]);
    }
  }
  __syncthreads();
  bool ok = true;
  {
    // ------------------------------------------------------------ compute warps
    // Group g (warps 8 g .. 8 g + 7) takes planes g, g + 2, ... of the CTA.
    // Warp gw holds rows [16 gw, 16 gw + 16) of columns [4 lane, 4 lane + 4).
    // Per token two barriers of the group: C (column partials written) and D
    // (the delta-rule write per column written, and the next token's inputs
    // staged). Every warp forms the token's norms itself from the staged k and
    // q. Group threads 0-127 load a token's inputs (channel / column gt) into
    // registers two tokens ahead (across planes too), so that a load has a
    // whole token's work to arrive in, and stage the next token between C and
    // D into the other buffer, whose previous token every warp of the group
    // finished before C.
    const int g = warp / GW, gw = warp % GW, gt = tid - g * GT, bar = 1 + g;
    float* wg = wcol[g];
    int tb = 0;                                         // buffer of the current token
    const int r0 = gw * ROWS, c0 = CPL * lane;
    struct Tok {
      float k, q, g, v, beta;
    };
    auto load_tok = [&](int plane, int tk, Tok& x) {
      x.k = x.q = x.g = x.v = x.beta = 0.f;
      if (gt >= 128) return;
      const int b = plane / a.HV, hv = plane % a.HV, h = hv / (a.HV / a.H);
      const size_t bt = (size_t)b * a.T + tk;
      if (gt < K) {
        const size_t qk = (bt * a.H + h) * K + gt;
        x.k = ld_x(a.k, qk, a.in_bf16);
        x.q = ld_x(a.q, qk, a.in_bf16);
        if (a.g) x.g = a.per_key ? a.g[(bt * a.HV + hv) * K + gt] : a.g[bt * a.HV + hv];
      }
      if (gt < V) x.v = ld_x(a.v, (bt * a.HV + hv) * V + gt, a.in_bf16);
      if (gt == 0) x.beta = a.beta[bt * a.HV + hv];
    };
    auto stage_tok = [&](const Tok& x, int buf) {
      if (gt < 128) {
        kr[g][buf][gt] = x.k;
        qr[g][buf][gt] = x.q;
        dec[g][buf][gt] = gt < K ? expf(x.g) : 0.f;
        if (gt == 0) tok[g][buf] = x.beta;
      }
    };
    // Token j of the group: plane g + GROUPS (j / T) of the CTA, token j % T.
    auto load_nth = [&](int j, Tok& x) {
      const int ij = g + GROUPS * (j / a.T);
      if (ij < my) load_tok(blockIdx.x + ij * gridDim.x, j % a.T, x);
    };
    Tok nx, nn;                                         // the next token, the one after it
    float cv = 0.f;                                     // this token's v (the rest is staged)
    if (g < my) {
      load_nth(0, nx);
      stage_tok(nx, 0);
      cv = nx.v;
      load_nth(1, nx);
    }
    nb_sync(bar, GT);                                   // the first token is staged
    int jt = 0;                                         // the group's token index
    for (int i = g; i < my; i += GROUPS) {
      const int s = i % STAGES;
      const int plane = blockIdx.x + i * gridDim.x;
      const int b = plane / a.HV, hv = plane % a.HV;
      const float* tile = reinterpret_cast<const float*>(sm + s * TILE);   // [K][V] fp32
      ok = ok && mbar_wait(&full[s], (i / STAGES) & 1, kWaitLimit);
      const bool cok = c0 < V;                          // V % 4 == 0: all four columns or none
      float S[ROWS][CPL];
#pragma unroll
      for (int r = 0; r < ROWS; ++r) {
        float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
        if (r0 + r < K && cok) x = *reinterpret_cast<const float4*>(tile + (r0 + r) * V + c0);
        S[r][0] = x.x; S[r][1] = x.y; S[r][2] = x.z; S[r][3] = x.w;
      }
      // The head is in registers: stage s may be refilled, with plane
      // i + STAGES, once all 8 warps of the group are done with it.
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&done[s]);
        if (gw == 0 && i + STAGES < my) {
          ok = ok && mbar_wait(&done[s], (i / STAGES) & 1, kWaitLimit);
          if (ok) {
            mbar_expect_tx(&full[s], tbytes);
            tma_load3(smem_u32(sm + s * TILE), &smap, 0, 0, blockIdx.x + (i + STAGES) * gridDim.x,
                      &full[s]);
          }
        }
      }
      __syncwarp();
      for (int tk = 0; tk < a.T; ++tk) {
        const size_t bt = (size_t)b * a.T + tk;
        const float xv = cv;
        const float* kg = kr[g][tb];
        const float* qg = qr[g][tb];
        const float* dg = dec[g][tb];
        const bool more = tk + 1 < a.T || i + GROUPS < my;
        load_nth(jt + 2, nn);
        // Norms of the staged k and q (zero past K), every warp for itself.
        float sk = 0.f, sq = 0.f, sqk = 0.f;
#pragma unroll
        for (int c = lane; c < 128; c += 32) {
          const float kc = kg[c], qc = qg[c];
          sk = fmaf(kc, kc, sk);
          sq = fmaf(qc, qc, sq);
          sqk = fmaf(qc, kc, sqk);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          sk += __shfl_xor_sync(0xffffffffu, sk, o);
          sq += __shfl_xor_sync(0xffffffffu, sq, o);
          sqk += __shfl_xor_sync(0xffffffffu, sqk, o);
        }
        const float nk = a.use_l2 ? 1.f / sqrtf(sk + 1e-6f) : 1.f;
        const float nq = a.scale * (a.use_l2 ? 1.f / sqrtf(sq + 1e-6f) : 1.f);
        const float qk = nq * nk * sqk, beta = tok[g][tb];
        // Decay, then this warp's share of k^T (D S) and q^T (D S) per column
        // (the row factors are shared-memory broadcasts).
        float pu[CPL] = {0.f, 0.f, 0.f, 0.f}, po[CPL] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int r = 0; r < ROWS; r += 4) {
          // (four rows' factors at a time: the compiler would otherwise hold
          // all 48 at once beside the 64 state values)
          asm volatile("" ::: "memory");
          const float4 d4 = *reinterpret_cast<const float4*>(dg + r0 + r);
          const float4 k4 = *reinterpret_cast<const float4*>(kg + r0 + r);
          const float4 q4 = *reinterpret_cast<const float4*>(qg + r0 + r);
          const float dd[4] = {d4.x, d4.y, d4.z, d4.w}, kk[4] = {k4.x, k4.y, k4.z, k4.w},
                      qq[4] = {q4.x, q4.y, q4.z, q4.w};
#pragma unroll
          for (int e = 0; e < 4; ++e)
#pragma unroll
            for (int m = 0; m < CPL; ++m) {
              S[r + e][m] *= dd[e];
              pu[m] = fmaf(kk[e], S[r + e][m], pu[m]);
              po[m] = fmaf(qq[e], S[r + e][m], po[m]);
            }
        }
        float4* rp = reinterpret_cast<float4*>(&red[g][gw][c0]);
        rp[0] = make_float4(pu[0], po[0], pu[1], po[1]);
        rp[1] = make_float4(pu[2], po[2], pu[3], po[3]);
        nb_sync(bar, GT);                               // C: partials written
        if (gt < 128) {
          // Column gt: sum the group's partials, form the write and the output.
          float u = 0.f, oq = 0.f;
#pragma unroll
          for (int w = 0; w < GW; ++w) {
            const float2 pr = red[g][w][gt];
            u += pr.x;
            oq += pr.y;
          }
          const float wv = beta * (xv - nk * u);
          wg[gt] = nk * wv;                             // times k^ = nk k
          if (gt < V) {
            const float o = fmaf(qk, wv, nq * oq);      // S'^T q~ = (D S)^T q~ + (q~ . k^) w
            const size_t off = (bt * a.HV + hv) * V + gt;
            if (a.out_bf16)
              static_cast<__nv_bfloat16*>(a.out)[off] = __float2bfloat16_rn(o);
            else
              static_cast<float*>(a.out)[off] = o;
          }
          if (more) stage_tok(nx, tb ^ 1);              // the next token's inputs
        }
        nb_sync(bar, GT);                               // D: writes and next inputs visible
        cv = nx.v;
        nx = nn;
        ++jt;
        const float4 wk4 = *reinterpret_cast<const float4*>(wg + c0);
        const float wk[CPL] = {wk4.x, wk4.y, wk4.z, wk4.w};
#pragma unroll
        for (int r = 0; r < ROWS; r += 4) {
          asm volatile("" ::: "memory");
          const float4 k4 = *reinterpret_cast<const float4*>(kg + r0 + r);
          const float kk[4] = {k4.x, k4.y, k4.z, k4.w};
#pragma unroll
          for (int e = 0; e < 4; ++e)
#pragma unroll
            for (int m = 0; m < CPL; ++m) S[r + e][m] = fmaf(kk[e], wk[m], S[r + e][m]);
        }
        tb ^= 1;
      }
      // Row r0 + r of the head: each warp store is one contiguous 512-byte row.
      float* dst = a.state + (size_t)plane * K * V;
#pragma unroll
      for (int r = 0; r < ROWS; ++r)
        if (r0 + r < K && cok)
          *reinterpret_cast<float4*>(dst + (size_t)(r0 + r) * V + c0) =
              make_float4(S[r][0], S[r][1], S[r][2], S[r][3]);
    }
  }
  if (!ok && a.error_word) atomicOr(a.error_word, 16u);
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
  if (d->K > 256) return GDR_ERR_UNSUPPORTED;
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
  a.error_word = nullptr;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (d->K <= 128 && d->V % 4 == 0 && d->V <= 128 &&
      (reinterpret_cast<uintptr_t>(state) & 15) == 0) {
    // State viewed as [B HV][K][V] fp32; box = one whole head (K rows x V columns).
    CUtensorMap m;
    memset(&m, 0, sizeof m);
    const cuuint64_t dims[3] = {(cuuint64_t)d->V, (cuuint64_t)d->K, (cuuint64_t)d->B * d->HV};
    const cuuint64_t strides[2] = {(cuuint64_t)d->V * 4, (cuuint64_t)d->K * d->V * 4};
    const cuuint32_t box[3] = {(cuuint32_t)d->V, (cuuint32_t)d->K, 1};
    if (fast::tmap_encode(&m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, state, dims, strides, box,
                          CU_TENSOR_MAP_SWIZZLE_NONE)) {
      static int sms = 0;
      if (sms == 0) {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (sms <= 0) sms = 1;
      }
      if (cudaFuncSetAttribute(recurrent_pipe_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               pipe::SMEM) != cudaSuccess)
        return GDR_ERR_CUDA;
      const long long planes = (long long)d->B * d->HV;
      if (planes <= (1LL << 30)) {
        const int grid = (int)(planes < sms ? planes : sms);
        recurrent_pipe_kernel<<<grid, pipe::THREADS, pipe::SMEM, st>>>(m, a, (int)planes);
        return cudaGetLastError() == cudaSuccess ? GDR_OK : GDR_ERR_CUDA;
      }
    }
  }
  dim3 grid((d->V + kCols - 1) / kCols, d->HV, d->B);
  if (d->K <= 128)
    recurrent_kernel<8><<<grid, kThreads, 0, st>>>(a);
  else
    recurrent_kernel<16><<<grid, kThreads, 0, st>>>(a);
  return cudaGetLastError() == cudaSuccess ? GDR_OK : GDR_ERR_CUDA;
}
