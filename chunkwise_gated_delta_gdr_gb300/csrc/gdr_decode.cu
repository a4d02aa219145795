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
// Main kernel (state V a multiple of 4, 16-byte aligned): persistent CTAs walk
// the (b, hv, 32-column V tile) tiles. A producer warp streams the state tiles
// (K x 32 fp32, 16 KB) through a four-stage shared-memory ring by TMA and
// stores each finished tile back by TMA, so several tiles per SM are in
// flight; 8 compute warps each hold 16 rows of the tile (lane = column) in
// registers while they apply the tokens.
//
// Fallback kernel (any V): one CTA per (V tile of 32 columns, hv, b), 16 warps: warp w holds state rows
// [8 w, 8 w + 8) of the tile's columns (lane = column), so every state access
// is a coalesced 128-byte row segment; 64 registers per thread keep two CTAs
// (32 warps) per SM in flight, which the HBM stream needs. Per token the column sums
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
  unsigned int* error_word;   // null: waits that give up are not reported
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

// ------------------------------------------------------------ pipelined kernel
namespace pipe {
constexpr int CW = 8, ROWS = 16, STAGES = 4, TILE = 128 * kCols * 4;   // 16 KB stage
constexpr int THREADS = (CW + 1) * 32;
constexpr int OFF_BAR = STAGES * TILE, SMEM = OFF_BAR + 2 * STAGES * 8 + 1024;
constexpr long kWaitLimit = 1L << 24;
__device__ __forceinline__ void nb_sync(int id, int n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}
}  // namespace pipe

__global__ void __launch_bounds__(pipe::THREADS, 2)
    recurrent_pipe_kernel(const __grid_constant__ CUtensorMap smap, DecodeArgs a, int ntiles) {
  using namespace pipe;
  using namespace ptx;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  __shared__ __align__(16) float kr[128], qr[128], dec[128];   // zero past K
  __shared__ float2 red[CW][kCols];                            // (k^T D S, q^T D S) partials
  __shared__ float tok[4];
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + OFF_BAR);
  uint64_t* done = full + STAGES;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int vtiles = (a.V + kCols - 1) / kCols;
  const int K = a.K, V = a.V;
  if (tid == 0) {
    for (int i = 0; i < STAGES; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&done[i], CW);
    }
    mbar_fence_init();
  }
  __syncthreads();
  bool ok = true;
  // Tile i of this CTA: global tile blockIdx.x + i * gridDim.x -> (plane = b HV + hv, vt).
  const int my = ntiles > (int)blockIdx.x ? (ntiles - 1 - blockIdx.x) / gridDim.x + 1 : 0;

  if (warp == CW) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      const uint32_t tbytes = (uint32_t)K * kCols * 4;
      auto coords = [&](int i, int& plane, int& vt) {
        const int t = blockIdx.x + i * gridDim.x;
        plane = t / vtiles;
        vt = t % vtiles;
      };
      for (int i = 0; i < my + STAGES && ok; ++i) {
        const int s = i % STAGES;
        if (i >= STAGES) {
          // Tile i - STAGES is finished in stage s: store it, then reuse the stage.
          ok = mbar_wait(&done[s], ((i / STAGES) - 1) & 1, kWaitLimit);
          if (!ok) break;
          int plane, vt;
          coords(i - STAGES, plane, vt);
          tma_store3(&smap, smem_u32(sm + s * TILE), vt * kCols, 0, plane);
          bulk_commit();
          bulk_wait_read<0>();
        }
        if (i < my) {
          int plane, vt;
          coords(i, plane, vt);
          mbar_expect_tx(&full[s], tbytes);
          tma_load3(smem_u32(sm + s * TILE), &smap, vt * kCols, 0, plane, &full[s]);
        }
      }
      bulk_wait<0>();
    }
  } else {
    // ------------------------------------------------------------ compute warps
    // The inputs of a tile's first token are loaded into registers while the
    // previous tile is still being processed (and before the TMA wait).
    const int r0 = warp * ROWS;
    struct Tok {
      float v, beta, k, q, g;
    };
    auto load_tok = [&](int i, int tk, Tok& x) {
      const int t = blockIdx.x + i * gridDim.x;
      const int plane = t / vtiles, vt = t % vtiles;
      const int b = plane / a.HV, hv = plane % a.HV, h = hv / (a.HV / a.H);
      const int col = vt * kCols + lane;
      const size_t bt = (size_t)b * a.T + tk;
      x.v = col < V ? ld_x(a.v, (bt * a.HV + hv) * V + col, a.in_bf16) : 0.f;
      x.beta = tid == 0 ? a.beta[bt * a.HV + hv] : 0.f;
      x.k = x.q = x.g = 0.f;
      if (tid < K) {
        const size_t qk = (bt * a.H + h) * K + tid;
        x.k = ld_x(a.k, qk, a.in_bf16);
        x.q = ld_x(a.q, qk, a.in_bf16);
        if (a.g) x.g = a.per_key ? a.g[(bt * a.HV + hv) * K + tid] : a.g[bt * a.HV + hv];
      }
    };
    Tok nx;
    if (my > 0) load_tok(0, 0, nx);
    for (int i = 0; i < my; ++i) {
      const int s = i % STAGES;
      const int t = blockIdx.x + i * gridDim.x;
      const int plane = t / vtiles, vt = t % vtiles;
      const int b = plane / a.HV, hv = plane % a.HV;
      const int col = vt * kCols + lane;
      const bool cok = col < V;
      float* tile = reinterpret_cast<float*>(sm + s * TILE);   // [K][32] fp32, row = key channel
      ok = ok && mbar_wait(&full[s], (i / STAGES) & 1, kWaitLimit);
      float S[ROWS];
#pragma unroll
      for (int r = 0; r < ROWS; ++r) S[r] = (r0 + r < K) ? tile[(r0 + r) * kCols + lane] : 0.f;
      for (int tk = 0; tk < a.T; ++tk) {
        const size_t bt = (size_t)b * a.T + tk;
        Tok x = nx;
        if (tk > 0) load_tok(i, tk, x);
        const float vv = x.v, bet = x.beta;
        if (tid < 128) {
          kr[tid] = tid < K ? x.k : 0.f;
          qr[tid] = tid < K ? x.q : 0.f;
          dec[tid] = tid < K ? expf(x.g) : 0.f;
        }
        nb_sync(1, CW * 32);
        if (warp == 0) {
          float sk = 0.f, sq = 0.f, sqk = 0.f;
#pragma unroll
          for (int c = lane; c < 128; c += 32) {
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
        nb_sync(1, CW * 32);
        const float nk = tok[0], nq = tok[1], beta = tok[2], qk = tok[3];
        // Decay, then this warp's share of k^T (D S) and q^T (D S) (raw k, q: the
        // norms are applied to the sums). Rows past K hold zeros throughout.
        const float4* k4 = reinterpret_cast<const float4*>(kr + r0);
        const float4* q4 = reinterpret_cast<const float4*>(qr + r0);
        const float4* d4 = reinterpret_cast<const float4*>(dec + r0);
        float pu = 0.f, po = 0.f;
#pragma unroll
        for (int r = 0; r < ROWS / 4; ++r) {
          const float4 kk = k4[r], qq = q4[r], dd = d4[r];
          S[4 * r + 0] *= dd.x;
          S[4 * r + 1] *= dd.y;
          S[4 * r + 2] *= dd.z;
          S[4 * r + 3] *= dd.w;
          pu = fmaf(kk.x, S[4 * r + 0], pu);
          po = fmaf(qq.x, S[4 * r + 0], po);
          pu = fmaf(kk.y, S[4 * r + 1], pu);
          po = fmaf(qq.y, S[4 * r + 1], po);
          pu = fmaf(kk.z, S[4 * r + 2], pu);
          po = fmaf(qq.z, S[4 * r + 2], po);
          pu = fmaf(kk.w, S[4 * r + 3], pu);
          po = fmaf(qq.w, S[4 * r + 3], po);
        }
        red[warp][lane] = make_float2(pu, po);
        nb_sync(1, CW * 32);
        float u = 0.f, oq = 0.f;
#pragma unroll
        for (int w = 0; w < CW; ++w) {
          const float2 pr = red[w][lane];
          u += pr.x;
          oq += pr.y;
        }
        const float wv = beta * (vv - nk * u);           // delta-rule write of this column
        const float wk = nk * wv;                        // times k^ = nk k
#pragma unroll
        for (int r = 0; r < ROWS / 4; ++r) {
          const float4 kk = k4[r];
          S[4 * r + 0] = fmaf(kk.x, wk, S[4 * r + 0]);
          S[4 * r + 1] = fmaf(kk.y, wk, S[4 * r + 1]);
          S[4 * r + 2] = fmaf(kk.z, wk, S[4 * r + 2]);
          S[4 * r + 3] = fmaf(kk.w, wk, S[4 * r + 3]);
        }
        if (warp == 0 && cok) {
          const float o = fmaf(qk, wv, nq * oq);        // S'^T q~ = (D S)^T q~ + (q~ . k^) w
          const size_t off = (bt * a.HV + hv) * V + col;
          if (a.out_bf16)
            static_cast<__nv_bfloat16*>(a.out)[off] = __float2bfloat16_rn(o);
          else
            static_cast<float*>(a.out)[off] = o;
        }
        nb_sync(1, CW * 32);   // kr / qr / dec / red are rewritten by the next token
      }
#pragma unroll
      for (int r = 0; r < ROWS; ++r)
        if (r0 + r < K) tile[(r0 + r) * kCols + lane] = S[r];
      fence_async_shared();                            // the TMA store reads the tile
      __syncwarp();
      if (lane == 0) mbar_arrive(&done[s]);
      if (i + 1 < my) load_tok(i + 1, 0, nx);
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
  a.error_word = nullptr;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (d->V % 4 == 0 && (reinterpret_cast<uintptr_t>(state) & 15) == 0) {
    // State viewed as [B HV][K][V] fp32; box = all K rows x 32 columns.
    CUtensorMap m;
    memset(&m, 0, sizeof m);
    const cuuint64_t dims[3] = {(cuuint64_t)d->V, (cuuint64_t)d->K, (cuuint64_t)d->B * d->HV};
    const cuuint64_t strides[2] = {(cuuint64_t)d->V * 4, (cuuint64_t)d->K * d->V * 4};
    const cuuint32_t box[3] = {(cuuint32_t)kCols, (cuuint32_t)d->K, 1};
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
      const long long tiles = (long long)d->B * d->HV * ((d->V + kCols - 1) / kCols);
      if (tiles <= (1LL << 30)) {
        const int grid = (int)(tiles < 2LL * sms ? tiles : 2LL * sms);
        recurrent_pipe_kernel<<<grid, pipe::THREADS, pipe::SMEM, st>>>(m, a, (int)tiles);
        return cudaGetLastError() == cudaSuccess ? GDR_OK : GDR_ERR_CUDA;
      }
    }
  }
  dim3 grid((d->V + kCols - 1) / kCols, d->HV, d->B);
  recurrent_kernel<<<grid, kThreads, 0, st>>>(a);
  return cudaGetLastError() == cudaSuccess ? GDR_OK : GDR_ERR_CUDA;
}
