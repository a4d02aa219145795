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
// persistent CTA per SM walks the heads. A producer warp streams each head's
// whole state (K x V fp32, one TMA box of up to 512-byte rows) through a
// three-stage shared-memory ring, so about 190 KB per SM are in flight; 16
// compute warps each take 8 rows x 4 columns into registers, release the stage
// at once (the producer refills it while they apply the tokens) and write the
// finished state back with coalesced 128-byte stores from registers. (Boxes of
// 128-byte rows were served several times slower.)
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
// (up to 512-byte) rows, streamed through a three-stage ring.
namespace pipe {
constexpr int CW = 16, ROWS = 8, CPL = 4;          // compute warps, rows per warp, columns per lane
constexpr int STAGES = 3, TILE = 128 * 128 * 4;    // 64 KB stage
constexpr int THREADS = (CW + 1) * 32;
constexpr int OFF_BAR = STAGES * TILE, SMEM = OFF_BAR + 2 * STAGES * 8 + 1024;
constexpr long kWaitLimit = 1L << 24;
static_assert(CW * ROWS == 128 && CPL * 32 == 128, "tile covers K, V <= 128");
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
  __shared__ __align__(16) float kr[128], qr[128], dec[128];   // zero past K
  __shared__ float2 red[CW][128];                              // (k^T D S, q^T D S) partials
  __shared__ float wcol[128];                                  // delta-rule write per column
  __shared__ float tok[4];
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + OFF_BAR);
  uint64_t* done = full + STAGES;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
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
  // Plane i of this CTA: blockIdx.x + i * gridDim.x (= b * HV + hv).
  const int my = nplanes > (int)blockIdx.x ? (nplanes - 1 - blockIdx.x) / gridDim.x + 1 : 0;

  if (warp == CW) {
    // ---------------------------------------------------------------- producer
    // Stage s takes plane i once the compute warps hold plane i - STAGES in
    // registers (completion i / STAGES - 1 of done[s]).
    if (lane == 0) {
      const uint32_t tbytes = (uint32_t)K * V * 4;
      for (int i = 0; i < my && ok; ++i) {
        const int s = i % STAGES;
        if (i >= STAGES) ok = mbar_wait(&done[s], ((i / STAGES) - 1) & 1, kWaitLimit);
        if (!ok) break;
        mbar_expect_tx(&full[s], tbytes);
        tma_load3(smem_u32(sm + s * TILE), &smap, 0, 0, blockIdx.x + i * gridDim.x, &full[s]);
      }
    }
  } else {
    // ------------------------------------------------------------ compute warps
    // Warp w holds rows [8 w, 8 w + 8) of columns lane + 32 m (m < 4).
    // Per token two CTA barriers: C (column partials written) and D (the
    // delta-rule write per column written, and the next token's inputs staged).
    // Every warp forms the token's norms itself from the staged k and q.
    // Threads 0-127 load a token's inputs (channel / column tid) into registers
    // one token ahead (across heads too) and stage them between C and D: every
    // read of the staged inputs of a token happens before its barrier C.
    const int r0 = warp * ROWS;
    struct Tok {
      float k, q, g, v, beta;
    };
    auto load_tok = [&](int plane, int tk, Tok& x) {
      x.k = x.q = x.g = x.v = x.beta = 0.f;
      if (tid >= 128) return;
      const int b = plane / a.HV, hv = plane % a.HV, h = hv / (a.HV / a.H);
      const size_t bt = (size_t)b * a.T + tk;
      if (tid < K) {
        const size_t qk = (bt * a.H + h) * K + tid;
        x.k = ld_x(a.k, qk, a.in_bf16);
        x.q = ld_x(a.q, qk, a.in_bf16);
        if (a.g) x.g = a.per_key ? a.g[(bt * a.HV + hv) * K + tid] : a.g[bt * a.HV + hv];
      }
      if (tid < V) x.v = ld_x(a.v, (bt * a.HV + hv) * V + tid, a.in_bf16);
      if (tid == 0) x.beta = a.beta[bt * a.HV + hv];
    };
    auto stage_tok = [&](const Tok& x) {
      if (tid < 128) {
        kr[tid] = x.k;
        qr[tid] = x.q;
        dec[tid] = tid < K ? expf(x.g) : 0.f;
        if (tid == 0) tok[0] = x.beta;
      }
    };
    Tok nx;
    if (my > 0) {
      load_tok(blockIdx.x, 0, nx);
      stage_tok(nx);
    }
    nb_sync(1, CW * 32);                               // the first token is staged
    for (int i = 0; i < my; ++i) {
      const int s = i % STAGES;
      const int plane = blockIdx.x + i * gridDim.x;
      const int b = plane / a.HV, hv = plane % a.HV;
      const float* tile = reinterpret_cast<const float*>(sm + s * TILE);   // [K][V] fp32
      ok = ok && mbar_wait(&full[s], (i / STAGES) & 1, kWaitLimit);
      float S[ROWS][CPL];
#pragma unroll
      for (int r = 0; r < ROWS; ++r)
#pragma unroll
        for (int m = 0; m < CPL; ++m) {
          const int c = lane + 32 * m;
          S[r][m] = (r0 + r < K && c < V) ? tile[(r0 + r) * V + c] : 0.f;
        }
      // The head is in registers: stage s may be refilled.
      __syncwarp();
      if (lane == 0) mbar_arrive(&done[s]);
      for (int tk = 0; tk < a.T; ++tk) {
        const size_t bt = (size_t)b * a.T + tk;
        const Tok x = nx;                              // this token (staged)
        const bool more = tk + 1 < a.T || i + 1 < my;
        if (tk + 1 < a.T)
          load_tok(plane, tk + 1, nx);
        else if (i + 1 < my)
          load_tok(plane + gridDim.x, 0, nx);
        // Norms of the staged k and q (zero past K), every warp for itself.
        float sk = 0.f, sq = 0.f, sqk = 0.f;
#pragma unroll
        for (int c = lane; c < 128; c += 32) {
          const float kc = kr[c], qc = qr[c];
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
        const float qk = nq * nk * sqk, beta = tok[0];
        // Decay, then this warp's share of k^T (D S) and q^T (D S) per column.
        const float4 kk0 = *reinterpret_cast<const float4*>(kr + r0);
        const float4 kk1 = *reinterpret_cast<const float4*>(kr + r0 + 4);
        const float4 qq0 = *reinterpret_cast<const float4*>(qr + r0);
        const float4 qq1 = *reinterpret_cast<const float4*>(qr + r0 + 4);
        const float4 dd0 = *reinterpret_cast<const float4*>(dec + r0);
        const float4 dd1 = *reinterpret_cast<const float4*>(dec + r0 + 4);
        const float kv[ROWS] = {kk0.x, kk0.y, kk0.z, kk0.w, kk1.x, kk1.y, kk1.z, kk1.w};
        const float qv[ROWS] = {qq0.x, qq0.y, qq0.z, qq0.w, qq1.x, qq1.y, qq1.z, qq1.w};
        const float dv[ROWS] = {dd0.x, dd0.y, dd0.z, dd0.w, dd1.x, dd1.y, dd1.z, dd1.w};
#pragma unroll
        for (int m = 0; m < CPL; ++m) {
          float pu = 0.f, po = 0.f;
#pragma unroll
          for (int r = 0; r < ROWS; ++r) {
            S[r][m] *= dv[r];
            pu = fmaf(kv[r], S[r][m], pu);
            po = fmaf(qv[r], S[r][m], po);
          }
          red[warp][lane + 32 * m] = make_float2(pu, po);
        }
        nb_sync(1, CW * 32);                           // C: partials written
        if (tid < 128) {
          // Column tid: sum the warps' partials, form the write and the output.
          float u = 0.f, oq = 0.f;
#pragma unroll
          for (int w = 0; w < CW; ++w) {
            const float2 pr = red[w][tid];
            u += pr.x;
            oq += pr.y;
          }
          const float wv = beta * (x.v - nk * u);
          wcol[tid] = nk * wv;                              // times k^ = nk k
          if (tid < V) {
            const float o = fmaf(qk, wv, nq * oq);         // S'^T q~ = (D S)^T q~ + (q~ . k^) w
            const size_t off = (bt * a.HV + hv) * V + tid;
            if (a.out_bf16)
              static_cast<__nv_bfloat16*>(a.out)[off] = __float2bfloat16_rn(o);
            else
              static_cast<float*>(a.out)[off] = o;
          }
          if (more) stage_tok(nx);                     // the next token's inputs
        }
        nb_sync(1, CW * 32);                           // D: writes and next inputs visible
#pragma unroll
        for (int m = 0; m < CPL; ++m) {
          const float wk = wcol[lane + 32 * m];
#pragma unroll
          for (int r = 0; r < ROWS; ++r) S[r][m] = fmaf(kv[r], wk, S[r][m]);
        }
      }
      // Row r0 + r of the head: each warp store is one 128-byte segment.
      float* dst = a.state + (size_t)plane * K * V;
#pragma unroll
      for (int r = 0; r < ROWS; ++r)
#pragma unroll
        for (int m = 0; m < CPL; ++m) {
          const int c = lane + 32 * m;
          if (r0 + r < K && c < V) dst[(size_t)(r0 + r) * V + c] = S[r][m];
        }
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
