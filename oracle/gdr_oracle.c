/*
 * gdr_oracle.c -- float64 CPU oracle for the gated delta rule forward pass.
 *
 * TEST INFRASTRUCTURE. This file is the correctness reference that the CUDA
 * library is compared against. Only the test suite, the smoke check and the
 * CPU-baseline leg of the benchmark load it; the product library never links,
 * loads or calls it, and it shares no code, header, table or constant with the
 * CUDA sources. It is deliberately slow and plain: loops in the order the
 * sources state the method, float64 throughout, no blocking or fusion.
 *
 * Sources (cited by page title and section):
 *   [notes]  "分块并行计算（Chunkwise）" lecture notes (sec-03): sections
 *            "为什么需要分块？", "chunk 内的 cumsum 与下三角解", the listings
 *            "naive_chunk_kda" (代码对照) and the inter-chunk loop (chunk 间递推),
 *            the shape table (形状流水线) and "_decayed_dot" (Decayed dot 函数).
 *   [blog]   "Chunkwise 并行算法 —— 线性注意力": §1.1-1.2 (Mamba2 SSD), §2.1 (Householder form),
 *            §2.3 (UT transform, Neumann series, row recursion), §2.4.
 *   [optim]  "DeltaNet chunk kernel optimization" (deltanet_chunk_optimize.py):
 *            _l2norm, the padding and trimming steps, the row-beta weighted
 *            projections, the default scale.
 *
 * Functions:
 *   gdr_oracle_recurrent        token-by-token recurrence (the definition).
 *   gdr_oracle_chunkwise        chunk form with beta on the columns of A_kk
 *                               and on r at the write ([notes]).
 *   gdr_oracle_chunkwise_rowbeta chunk form with beta on the rows and in the
 *                               right-hand sides ([blog] §2.3, [optim]).
 *   gdr_oracle_bruteforce       explicit products of the one-step maps
 *                               (I - beta k k^T) D_t ([blog] §2.1), for tiny T, K.
 *   gdr_oracle_ssd_recurrent    the Mamba2 SSD recurrence S_t = diag(alpha_t) S_{t-1}
 *                               + k_t v_t^T, o_t = S_t^T q_t (no delta erase, no
 *                               beta; [blog] §1.1), token by token.
 *   gdr_oracle_unit_lower_inverse  (I + L)^{-1} three ways ([notes] solve,
 *                               [blog] §2.3 Neumann series and row recursion).
 *
 * Tensor conventions (all row-major, contiguous), identical to the library's:
 *   q, k  [B, T, H,  K]      v     [B, T, HV, V]
 *   g     [B, T, HV]  (gate_mode 0: one scalar log-decay per token and head)
 *         [B, T, HV, K] (gate_mode 1: one log-decay per key channel, KDA)
 *   beta  [B, T, HV]         s0    [B, HV, K, V] or NULL (zero state)
 * Outputs are written per selected sequence s (a flat index b*HV + hv):
 *   o_out [nsel, T, V]       s_out [nsel, K, V] (may be NULL)
 * With sel == NULL every sequence is computed, in the order b*HV + hv.
 * The state S of one sequence is K x V (rows = key channels) and o_t = S^T q.
 *
 * Value head hv reads query/key head hv / (HV/H) (repeat_interleave over the
 * head axis, [notes] listing naive_chunk_kda).
 *
 * Input element types: qkv_dtype and gate_dtype are one of
 *   ORACLE_F64 = 0, ORACLE_F32 = 1, ORACLE_BF16 = 2 (uint16 bit patterns).
 * Every such value is exactly representable in float64.
 *
 * Return value: 0 on success, a negative number for invalid arguments.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORACLE_F64 = 0, ORACLE_F32 = 1, ORACLE_BF16 = 2 };

/* Read element i of a tensor of the given element type, as float64 (exact). */
static double rd(const void* p, int dtype, long i) {
  if (dtype == ORACLE_F64) return ((const double*)p)[i];
  if (dtype == ORACLE_F32) return (double)((const float*)p)[i];
  uint32_t bits = ((uint32_t)((const uint16_t*)p)[i]) << 16;
  float f;
  memcpy(&f, &bits, sizeof f);
  return (double)f;
}

typedef struct {
  const void *q, *k, *v, *g, *beta, *s0;
  int qkv_dtype, gate_dtype;
  int B, T, H, HV, K, V, gate_mode, use_qk_l2norm;
  double scale;
} problem;

static int check_problem(const problem* p) {
  if (p->B < 0 || p->T < 0) return -1;
  if (p->H <= 0 || p->HV <= 0 || p->K <= 0 || p->V <= 0) return -2;
  if (p->HV % p->H != 0) return -3;
  if (p->gate_mode != 0 && p->gate_mode != 1) return -4;
  if (p->qkv_dtype < 0 || p->qkv_dtype > 2) return -5;
  if (p->gate_dtype < 0 || p->gate_dtype > 2) return -5;
  if ((p->B > 0 && p->T > 0) && (!p->q || !p->k || !p->v || !p->g || !p->beta)) return -6;
  return 0;
}

/* Load q_t (or k_t) of head h as float64 and L2-normalise it when asked:
 * x * 1/sqrt(sum x^2 + 1e-6), the eps inside the root ([optim] _l2norm). */
static void load_qk(const problem* p, const void* x, int b, int t, int h, double* out) {
  long base = (((long)b * p->T + t) * p->H + h) * p->K;
  for (int c = 0; c < p->K; ++c) out[c] = rd(x, p->qkv_dtype, base + c);
  if (p->use_qk_l2norm) {
    double ss = 0.0;
    for (int c = 0; c < p->K; ++c) ss += out[c] * out[c];
    double inv = 1.0 / sqrt(ss + 1e-6);
    for (int c = 0; c < p->K; ++c) out[c] *= inv;
  }
}

static double load_v(const problem* p, int b, int t, int hv, int j) {
  return rd(p->v, p->qkv_dtype, (((long)b * p->T + t) * p->HV + hv) * p->V + j);
}

/* Log-decay of token t, value head hv, key channel c (channel ignored for a
 * scalar gate). */
static double load_g(const problem* p, int b, int t, int hv, int c) {
  if (p->gate_mode == 0) return rd(p->g, p->gate_dtype, ((long)b * p->T + t) * p->HV + hv);
  return rd(p->g, p->gate_dtype, (((long)b * p->T + t) * p->HV + hv) * p->K + c);
}

static double load_beta(const problem* p, int b, int t, int hv) {
  return rd(p->beta, p->gate_dtype, ((long)b * p->T + t) * p->HV + hv);
}

static void load_s0(const problem* p, int b, int hv, double* S) {
  long n = (long)p->K * p->V;
  if (!p->s0) {
    memset(S, 0, sizeof(double) * n);
    return;
  }
  long base = ((long)b * p->HV + hv) * n;
  for (long i = 0; i < n; ++i) S[i] = rd(p->s0, p->gate_dtype, base + i);
}

static int resolve_threads(int nthreads) {
#ifdef _OPENMP
  return nthreads > 0 ? nthreads : omp_get_max_threads();
#else
  (void)nthreads;
  return 1;
#endif
}

/* ---------------------------------------------------------------------------
 * The recurrence (the method's definition).
 *
 * Per token, for one (b, hv) sequence with state S (K x V):
 *   S <- exp(g_t) S                     (decay first; per row c for a per-key gate)
 *   S <- S + beta_t k_t (v_t - S^T k_t)^T   (delta write with the decayed state)
 *   o_t = S^T (scale q_t)               (output from the state after the write)
 * [notes] "为什么需要分块？" (the naive recurrent form the chunk form must equal),
 * [blog] §2.1 (the same rule, transposed and ungated), [optim] _l2norm and the
 * default scale 1/sqrt(K).
 *
 * `mutation` is a test hook that plants one known mistake (0 = faithful):
 *   1 drop the decay; 2 write before decaying; 3 output from the pre-write
 *   state; 4 read the state transposed in the erase term (needs K == V);
 *   5 flip the sign of the erase term; 6 map value heads to q/k heads modulo H;
 *   7 drop beta from the write; 8 drop the scale; 9 use the previous token's
 *   gate. The oracle's own pins must reject every one of them.
 * ------------------------------------------------------------------------- */
int gdr_oracle_recurrent(const void* q, const void* k, const void* v, const void* g,
                         const void* beta, const void* s0, int qkv_dtype, int gate_dtype,
                         int B, int T, int H, int HV, int K, int V, int gate_mode,
                         double scale, int use_qk_l2norm, const int* sel, int nsel,
                         double* o_out, double* s_out, int nthreads, int mutation) {
  problem p = {q, k, v, g, beta, s0, qkv_dtype, gate_dtype, B, T, H, HV, K, V,
               gate_mode, use_qk_l2norm, scale};
  int rc = check_problem(&p);
  if (rc) return rc;
  if (mutation == 4 && K != V) return -7;
  long nseq = sel ? nsel : (long)B * HV;
  int group = HV / H;

#pragma omp parallel for num_threads(resolve_threads(nthreads)) schedule(dynamic, 1)
  for (long s = 0; s < nseq; ++s) {
    long bh = sel ? sel[s] : s;
    int b = (int)(bh / HV), hv = (int)(bh % HV);
    int h = (mutation == 6) ? hv % H : hv / group;
    double* S = malloc(sizeof(double) * K * V);
    double* qt = malloc(sizeof(double) * K);
    double* kt = malloc(sizeof(double) * K);
    double* u = malloc(sizeof(double) * V);
    double* pre = malloc(sizeof(double) * K * V);
    load_s0(&p, b, hv, S);
    for (int t = 0; t < T; ++t) {
      load_qk(&p, q, b, t, h, qt);
      load_qk(&p, k, b, t, h, kt);
      double bt = load_beta(&p, b, t, hv);
      int tg = (mutation == 9) ? (t > 0 ? t - 1 : 0) : t;
      if (mutation == 2) { /* write first, then decay */
        for (int j = 0; j < V; ++j) {
          double sk = 0.0;
          for (int c = 0; c < K; ++c) sk += S[(long)c * V + j] * kt[c];
          u[j] = load_v(&p, b, t, hv, j) - sk;
        }
        for (int c = 0; c < K; ++c)
          for (int j = 0; j < V; ++j) S[(long)c * V + j] += bt * kt[c] * u[j];
      }
      if (mutation != 1) {
        for (int c = 0; c < K; ++c) {
          double d = exp(load_g(&p, b, tg, hv, c));
          for (int j = 0; j < V; ++j) S[(long)c * V + j] *= d;
        }
      }
      if (mutation == 3) memcpy(pre, S, sizeof(double) * K * V);
      if (mutation != 2) {
        for (int j = 0; j < V; ++j) {
          double sk = 0.0;
          for (int c = 0; c < K; ++c)
            sk += (mutation == 4 ? S[(long)j * V + c] : S[(long)c * V + j]) * kt[c];
          u[j] = load_v(&p, b, t, hv, j) + (mutation == 5 ? sk : -sk);
        }
        double w = (mutation == 7) ? 1.0 : bt;
        for (int c = 0; c < K; ++c)
          for (int j = 0; j < V; ++j) S[(long)c * V + j] += w * kt[c] * u[j];
      }
      const double* So = (mutation == 3) ? pre : S;
      double sc = (mutation == 8) ? 1.0 : scale;
      for (int j = 0; j < V; ++j) {
        double acc = 0.0;
        for (int c = 0; c < K; ++c) acc += So[(long)c * V + j] * sc * qt[c];
        o_out[((long)s * T + t) * V + j] = acc;
      }
    }
    if (s_out) memcpy(s_out + s * (long)K * V, S, sizeof(double) * K * V);
    free(S); free(qt); free(kt); free(u); free(pre);
  }
  return 0;
}

/* ---------------------------------------------------------------------------
 * Mamba2 SSD ([blog] §1.1): per (b, hv), S <- diag(exp(g_t)) S + k_t v_t^T,
 * o_t = S^T (scale q_t), token by token; q_t, k_t L2-normalised when asked.
 * Same tensor conventions as gdr_oracle_recurrent; there is no beta.
 * ------------------------------------------------------------------------- */
int gdr_oracle_ssd_recurrent(const void* q, const void* k, const void* v, const void* g,
                             const void* s0, int qkv_dtype, int gate_dtype, int B, int T, int H,
                             int HV, int K, int V, int gate_mode, double scale, int use_qk_l2norm,
                             const int* sel, int nsel, double* o_out, double* s_out,
                             int nthreads) {
  /* beta is never read: g stands in for it so that the shared checks apply. */
  problem p = {q, k, v, g, g, s0, qkv_dtype, gate_dtype, B, T, H, HV, K, V,
               gate_mode, use_qk_l2norm, scale};
  int rc = check_problem(&p);
  if (rc) return rc;
  long nseq = sel ? nsel : (long)B * HV;
  int group = HV / H;

#pragma omp parallel for num_threads(resolve_threads(nthreads)) schedule(dynamic, 1)
  for (long s = 0; s < nseq; ++s) {
    long bh = sel ? sel[s] : s;
    int b = (int)(bh / HV), hv = (int)(bh % HV);
    int h = hv / group;
    double* S = malloc(sizeof(double) * K * V);
    double* qt = malloc(sizeof(double) * K);
    double* kt = malloc(sizeof(double) * K);
    load_s0(&p, b, hv, S);
    for (int t = 0; t < T; ++t) {
      load_qk(&p, q, b, t, h, qt);
      load_qk(&p, k, b, t, h, kt);
      for (int c = 0; c < K; ++c) {
        double d = exp(load_g(&p, b, t, hv, c));
        for (int j = 0; j < V; ++j)
          S[(long)c * V + j] = d * S[(long)c * V + j] + kt[c] * load_v(&p, b, t, hv, j);
      }
      for (int j = 0; j < V; ++j) {
        double acc = 0.0;
        for (int c = 0; c < K; ++c) acc += S[(long)c * V + j] * scale * qt[c];
        o_out[((long)s * T + t) * V + j] = acc;
      }
    }
    if (s_out) memcpy(s_out + s * (long)K * V, S, sizeof(double) * K * V);
    free(S); free(qt); free(kt);
  }
  return 0;
}

/* ---------------------------------------------------------------------------
 * (I + L)^{-1} for a strictly lower-triangular C x C matrix L (row-major).
 * method 0: forward substitution, column by column of the identity
 *           (the triangular solve of [notes] "chunk 内的 cumsum 与下三角解").
 * method 1: the Neumann series sum_{n<C} (-L)^n, exact because L^C = 0
 *           ([blog] §2.3, with N = -L).
 * method 2: the row recursion of [blog] §2.3 / [optim] docstring: start from
 *           Y = -L, then for i = 1..C-1 replace row i by
 *           Y[i,:i] + sum_k Y[i,k] Y[k,:i] (rows above already final);
 *           the inverse is I + Y.
 * ------------------------------------------------------------------------- */
int gdr_oracle_unit_lower_inverse(const double* L, int C, int method, double* X) {
  if (C <= 0 || !L || !X) return -1;
  if (method == 0) {
    for (int col = 0; col < C; ++col) {
      for (int i = 0; i < C; ++i) {
        double acc = (i == col) ? 1.0 : 0.0;
        for (int j = 0; j < i; ++j) acc -= L[i * C + j] * X[j * C + col];
        X[i * C + col] = acc;
      }
    }
    return 0;
  }
  if (method == 1) {
    double* P = malloc(sizeof(double) * C * C);   /* current power (-L)^n */
    double* Q = malloc(sizeof(double) * C * C);
    for (int i = 0; i < C * C; ++i) X[i] = 0.0, P[i] = 0.0;
    for (int i = 0; i < C; ++i) X[i * C + i] = 1.0, P[i * C + i] = 1.0;
    for (int n = 1; n < C; ++n) {
      for (int i = 0; i < C; ++i)
        for (int j = 0; j < C; ++j) {
          double acc = 0.0;
          for (int m = 0; m < C; ++m) acc += P[i * C + m] * (-L[m * C + j]);
          Q[i * C + j] = acc;
        }
      memcpy(P, Q, sizeof(double) * C * C);
      for (int i = 0; i < C * C; ++i) X[i] += P[i];
    }
    free(P); free(Q);
    return 0;
  }
  if (method == 2) {
    double* Y = malloc(sizeof(double) * C * C);
    double* row = malloc(sizeof(double) * C);
    for (int i = 0; i < C; ++i)
      for (int j = 0; j < C; ++j) Y[i * C + j] = (j < i) ? -L[i * C + j] : 0.0;
    for (int i = 1; i < C; ++i) {
      for (int j = 0; j < i; ++j) row[j] = Y[i * C + j];
      for (int j = 0; j < i; ++j) {
        double acc = row[j];
        for (int m = 0; m < i; ++m) acc += row[m] * Y[m * C + j];
        Y[i * C + j] = acc;
      }
    }
    for (int i = 0; i < C; ++i)
      for (int j = 0; j < C; ++j) X[i * C + j] = Y[i * C + j] + (i == j ? 1.0 : 0.0);
    free(Y); free(row);
    return 0;
  }
  return -2;
}

/* Dense product Z = X (n x m) times Y (m x p), row-major. */
static void matmul(const double* X, const double* Y, double* Z, int n, int m, int p) {
  for (int i = 0; i < n; ++i)
    for (int j = 0; j < p; ++j) {
      double acc = 0.0;
      for (int l = 0; l < m; ++l) acc += X[(long)i * m + l] * Y[(long)l * p + j];
      Z[(long)i * p + j] = acc;
    }
}

/* Per-sequence padded copy of the inputs. Rows t >= T are zero for q, k, v, g
 * and beta ([optim] "Pad to chunk boundary"); q is normalised and scaled, k
 * normalised, g broadcast over the K channels for a scalar gate. */
typedef struct {
  int Tp;
  double *qs, *kn, *vv, *gg, *bb;
} padded_seq;

static void pad_sequence(const problem* p, int b, int hv, int C, padded_seq* ps) {
  int group = p->HV / p->H, h = hv / group;
  int K = p->K, V = p->V;
  int Tp = ((p->T + C - 1) / C) * C;
  ps->Tp = Tp;
  ps->qs = calloc((size_t)Tp * K, sizeof(double));
  ps->kn = calloc((size_t)Tp * K, sizeof(double));
  ps->vv = calloc((size_t)Tp * V, sizeof(double));
  ps->gg = calloc((size_t)Tp * K, sizeof(double));
  ps->bb = calloc((size_t)Tp, sizeof(double));
  for (int t = 0; t < p->T; ++t) {
    load_qk(p, p->q, b, t, h, ps->qs + (long)t * K);
    for (int c = 0; c < K; ++c) ps->qs[(long)t * K + c] *= p->scale;
    load_qk(p, p->k, b, t, h, ps->kn + (long)t * K);
    for (int j = 0; j < V; ++j) ps->vv[(long)t * V + j] = load_v(p, b, t, hv, j);
    for (int c = 0; c < K; ++c) ps->gg[(long)t * K + c] = load_g(p, b, t, hv, c);
    ps->bb[t] = load_beta(p, b, t, hv);
  }
}

static void free_padded(padded_seq* ps) {
  free(ps->qs); free(ps->kn); free(ps->vv); free(ps->gg); free(ps->bb);
}

/* <x_i, exp(G_i - G_j) * k_j> over the K channels: the decayed dot of
 * [notes] "Decayed dot 函数". */
static double decayed_dot(const double* xi, const double* kj, const double* Gi,
                          const double* Gj, int K) {
  double acc = 0.0;
  for (int c = 0; c < K; ++c) acc += xi[c] * exp(Gi[c] - Gj[c]) * kj[c];
  return acc;
}

/* Solve (I + L) X = R for X (C x n), L strictly lower (C x C), by forming
 * the inverse with the given method and multiplying (method 0 solves by
 * forward substitution directly). */
static void unit_lower_solve(const double* L, const double* R, double* X, int C, int n,
                             int method) {
  if (method == 0) {
    for (int i = 0; i < C; ++i)
      for (int j = 0; j < n; ++j) {
        double acc = R[(long)i * n + j];
        for (int m = 0; m < i; ++m) acc -= L[i * C + m] * X[(long)m * n + j];
        X[(long)i * n + j] = acc;
      }
    return;
  }
  double* Minv = malloc(sizeof(double) * C * C);
  gdr_oracle_unit_lower_inverse(L, C, method, Minv);
  matmul(Minv, R, X, C, C, n);
  free(Minv);
}

/* ---------------------------------------------------------------------------
 * Chunk form, beta on the columns ([notes] "chunk 内的 cumsum 与下三角解",
 * listings naive_chunk_kda and the inter-chunk loop). For each chunk n of C
 * tokens:
 *   G_i  = sum_{j<=i} g_j (per channel)                       (cumsum)
 *   A_kk[i,j] = <k_i, exp(G_i - G_j) k_j>,  A_qk likewise with q  (decayed dots)
 *   M    = I + tril(A_kk * beta[None, :], -1)                 (beta on column j)
 *   W    = M^{-1} (exp(G) * k),   U = M^{-1} v                (triangular solve)
 *   A_qk = (A_qk * beta[None, :]) with the diagonal kept, upper part zero
 *   r    = U - W S
 *   o_n  = (q * exp(G)) S + A_qk r
 *   S    = exp(G_last) S + (exp(G_last - G) * k)^T (r * beta)
 * The sequence is zero-padded to a multiple of C and the outputs trimmed.
 * solve_method selects how M^{-1} is applied (see unit_lower_solve).
 * ------------------------------------------------------------------------- */
static void chunk_sequence(const problem* p, int b, int hv, int C, int solve_method,
                           int row_beta, double* o_seq, double* S) {
  int K = p->K, V = p->V;
  padded_seq ps;
  pad_sequence(p, b, hv, C, &ps);
  double* G = malloc(sizeof(double) * C * K);
  double* Akk = malloc(sizeof(double) * C * C);
  double* Aqk = malloc(sizeof(double) * C * C);
  double* L = malloc(sizeof(double) * C * C);
  double* Rw = malloc(sizeof(double) * C * K);
  double* Rv = malloc(sizeof(double) * C * V);
  double* W = malloc(sizeof(double) * C * K);
  double* U = malloc(sizeof(double) * C * V);
  double* WS = malloc(sizeof(double) * C * V);
  double* r = malloc(sizeof(double) * C * V);
  double* QS = malloc(sizeof(double) * C * V);
  double* Qe = malloc(sizeof(double) * C * K);
  double* dS = malloc(sizeof(double) * K * V);
  int nchunks = ps.Tp / C;
  for (int n = 0; n < nchunks; ++n) {
    const double* qn = ps.qs + (long)n * C * K;
    const double* kn = ps.kn + (long)n * C * K;
    const double* vn = ps.vv + (long)n * C * V;
    const double* gn = ps.gg + (long)n * C * K;
    const double* bn = ps.bb + (long)n * C;
    for (int c = 0; c < K; ++c) {
      double acc = 0.0;
      for (int i = 0; i < C; ++i) {
        acc += gn[i * K + c];
        G[i * K + c] = acc;
      }
    }
    for (int i = 0; i < C; ++i)
      for (int j = 0; j < C; ++j) {
        Akk[i * C + j] = (j < i) ? decayed_dot(kn + i * K, kn + j * K, G + i * K, G + j * K, K) : 0.0;
        Aqk[i * C + j] = (j <= i) ? decayed_dot(qn + i * K, kn + j * K, G + i * K, G + j * K, K) : 0.0;
      }
    if (!row_beta) {
      for (int i = 0; i < C; ++i)
        for (int j = 0; j < C; ++j) L[i * C + j] = (j < i) ? Akk[i * C + j] * bn[j] : 0.0;
      for (int j = 0; j < C; ++j) {
        for (int c = 0; c < K; ++c) Rw[j * K + c] = exp(G[j * K + c]) * kn[j * K + c];
        for (int c = 0; c < V; ++c) Rv[j * V + c] = vn[j * V + c];
      }
      for (int i = 0; i < C; ++i)
        for (int j = 0; j < C; ++j) Aqk[i * C + j] *= bn[j];
    } else {
      /* [blog] §2.3: T = [I + strictLower(diag(beta) A_kk)]^{-1} diag(beta),
       * W = T (exp(G) k), U = T v; A_qk keeps no beta ([optim] "Weighted
       * projections": k_beta, v_beta as right-hand sides, system I + A). */
      for (int i = 0; i < C; ++i)
        for (int j = 0; j < C; ++j) L[i * C + j] = (j < i) ? bn[i] * Akk[i * C + j] : 0.0;
      for (int j = 0; j < C; ++j) {
        for (int c = 0; c < K; ++c) Rw[j * K + c] = bn[j] * exp(G[j * K + c]) * kn[j * K + c];
        for (int c = 0; c < V; ++c) Rv[j * V + c] = bn[j] * vn[j * V + c];
      }
    }
    unit_lower_solve(L, Rw, W, C, K, solve_method);
    unit_lower_solve(L, Rv, U, C, V, solve_method);
    matmul(W, S, WS, C, K, V);
    for (int i = 0; i < C * V; ++i) r[i] = U[i] - WS[i];
    for (int i = 0; i < C; ++i)
      for (int c = 0; c < K; ++c) Qe[i * K + c] = qn[i * K + c] * exp(G[i * K + c]);
    matmul(Qe, S, QS, C, K, V);
    for (int i = 0; i < C; ++i) {
      int t = n * C + i;
      for (int j = 0; j < V; ++j) {
        double acc = QS[i * V + j];
        for (int m = 0; m <= i; ++m) acc += Aqk[i * C + m] * r[m * V + j];
        if (t < p->T) o_seq[(long)t * V + j] = acc;
      }
    }
    const double* Gl = G + (C - 1) * K;
    for (int c = 0; c < K; ++c)
      for (int j = 0; j < V; ++j) {
        double acc = 0.0;
        for (int m = 0; m < C; ++m) {
          double w = exp(Gl[c] - G[m * K + c]) * kn[m * K + c];
          acc += w * (row_beta ? r[m * V + j] : r[m * V + j] * bn[m]);
        }
        dS[c * V + j] = acc;
      }
    for (int c = 0; c < K; ++c)
      for (int j = 0; j < V; ++j) S[c * V + j] = exp(Gl[c]) * S[c * V + j] + dS[c * V + j];
  }
  free(G); free(Akk); free(Aqk); free(L); free(Rw); free(Rv); free(W); free(U);
  free(WS); free(r); free(QS); free(Qe); free(dS);
  free_padded(&ps);
}

static int chunk_driver(const problem* p, int C, int solve_method, int row_beta,
                        const int* sel, int nsel, double* o_out, double* s_out,
                        int nthreads) {
  int rc = check_problem(p);
  if (rc) return rc;
  if (C <= 0) return -8;
  if (solve_method < 0 || solve_method > 2) return -9;
  long nseq = sel ? nsel : (long)p->B * p->HV;
  int K = p->K, V = p->V, T = p->T, HV = p->HV;
#pragma omp parallel for num_threads(resolve_threads(nthreads)) schedule(dynamic, 1)
  for (long s = 0; s < nseq; ++s) {
    long bh = sel ? sel[s] : s;
    int b = (int)(bh / HV), hv = (int)(bh % HV);
    double* S = malloc(sizeof(double) * K * V);
    load_s0(p, b, hv, S);
    chunk_sequence(p, b, hv, C, solve_method, row_beta, o_out + s * (long)T * V, S);
    if (s_out) memcpy(s_out + s * (long)K * V, S, sizeof(double) * K * V);
    free(S);
  }
  return 0;
}

int gdr_oracle_chunkwise(const void* q, const void* k, const void* v, const void* g,
                         const void* beta, const void* s0, int qkv_dtype, int gate_dtype,
                         int B, int T, int H, int HV, int K, int V, int gate_mode,
                         double scale, int use_qk_l2norm, int chunk_size, int solve_method,
                         const int* sel, int nsel, double* o_out, double* s_out,
                         int nthreads) {
  problem p = {q, k, v, g, beta, s0, qkv_dtype, gate_dtype, B, T, H, HV, K, V,
               gate_mode, use_qk_l2norm, scale};
  return chunk_driver(&p, chunk_size, solve_method, 0, sel, nsel, o_out, s_out, nthreads);
}

int gdr_oracle_chunkwise_rowbeta(const void* q, const void* k, const void* v, const void* g,
                                 const void* beta, const void* s0, int qkv_dtype,
                                 int gate_dtype, int B, int T, int H, int HV, int K, int V,
                                 int gate_mode, double scale, int use_qk_l2norm,
                                 int chunk_size, int solve_method, const int* sel, int nsel,
                                 double* o_out, double* s_out, int nthreads) {
  problem p = {q, k, v, g, beta, s0, qkv_dtype, gate_dtype, B, T, H, HV, K, V,
               gate_mode, use_qk_l2norm, scale};
  return chunk_driver(&p, chunk_size, solve_method, 1, sel, nsel, o_out, s_out, nthreads);
}

/* ---------------------------------------------------------------------------
 * Brute force from the Householder form ([blog] §2.1, gated): each token is
 * the affine map S_t = P_t S_{t-1} + beta_t k_t v_t^T with the explicit K x K
 * matrix P_t = (I - beta_t k_t k_t^T) D_t, D_t = diag(exp(g_t)). The state
 * after token t is formed as a sum of explicit matrix products,
 *   S_t = [P_t ... P_1] S_0 + sum_{u<=t} [P_t ... P_{u+1}] beta_u k_u v_u^T,
 * each bracket multiplied out from scratch, and o_t = S_t^T (scale q_t).
 * Cost O(T^3 K^3): meant for T <= 8 and small K.
 * ------------------------------------------------------------------------- */
int gdr_oracle_bruteforce(const void* q, const void* k, const void* v, const void* g,
                          const void* beta, const void* s0, int qkv_dtype, int gate_dtype,
                          int B, int T, int H, int HV, int K, int V, int gate_mode,
                          double scale, int use_qk_l2norm, double* o_out, double* s_out) {
  problem p = {q, k, v, g, beta, s0, qkv_dtype, gate_dtype, B, T, H, HV, K, V,
               gate_mode, use_qk_l2norm, scale};
  int rc = check_problem(&p);
  if (rc) return rc;
  int group = HV / H;
  double* P = malloc(sizeof(double) * (T > 0 ? T : 1) * K * K);
  double* Ks = malloc(sizeof(double) * (T > 0 ? T : 1) * K);
  double* Qs = malloc(sizeof(double) * (T > 0 ? T : 1) * K);
  double* prod = malloc(sizeof(double) * K * K);
  double* tmp = malloc(sizeof(double) * K * K);
  double* S0 = malloc(sizeof(double) * K * V);
  double* St = malloc(sizeof(double) * K * V);
  double* term = malloc(sizeof(double) * K * V);
  double* X = malloc(sizeof(double) * K * V);
  for (long s = 0; s < (long)B * HV; ++s) {
    int b = (int)(s / HV), hv = (int)(s % HV), h = hv / group;
    load_s0(&p, b, hv, S0);
    for (int t = 0; t < T; ++t) {
      double* kt = Ks + (long)t * K;
      load_qk(&p, q, b, t, h, Qs + (long)t * K);
      load_qk(&p, k, b, t, h, kt);
      double bt = load_beta(&p, b, t, hv);
      double* Pt = P + (long)t * K * K;
      for (int i = 0; i < K; ++i)
        for (int j = 0; j < K; ++j)
          Pt[i * K + j] = ((i == j) ? 1.0 : 0.0) - bt * kt[i] * kt[j];
      for (int i = 0; i < K; ++i)
        for (int j = 0; j < K; ++j) Pt[i * K + j] *= exp(load_g(&p, b, t, hv, j));
    }
    for (int t = 0; t < T; ++t) {
      /* [P_t ... P_1] S_0 */
      for (int i = 0; i < K * K; ++i) prod[i] = (i / K == i % K) ? 1.0 : 0.0;
      for (int u = 0; u <= t; ++u) {
        matmul(P + (long)u * K * K, prod, tmp, K, K, K);
        memcpy(prod, tmp, sizeof(double) * K * K);
      }
      matmul(prod, S0, St, K, K, V);
      for (int u = 0; u <= t; ++u) {
        /* [P_t ... P_{u+1}] beta_u k_u v_u^T */
        for (int i = 0; i < K * K; ++i) prod[i] = (i / K == i % K) ? 1.0 : 0.0;
        for (int w = u + 1; w <= t; ++w) {
          matmul(P + (long)w * K * K, prod, tmp, K, K, K);
          memcpy(prod, tmp, sizeof(double) * K * K);
        }
        double bu = load_beta(&p, b, u, hv);
        for (int i = 0; i < K; ++i)
          for (int j = 0; j < V; ++j) X[i * V + j] = bu * Ks[(long)u * K + i] * load_v(&p, b, u, hv, j);
        matmul(prod, X, term, K, K, V);
        for (int i = 0; i < K * V; ++i) St[i] += term[i];
      }
      for (int j = 0; j < V; ++j) {
        double acc = 0.0;
        for (int c = 0; c < K; ++c) acc += St[c * V + j] * scale * Qs[(long)t * K + c];
        o_out[((long)s * T + t) * V + j] = acc;
      }
    }
    if (s_out) memcpy(s_out + s * (long)K * V, T > 0 ? St : S0, sizeof(double) * K * V);
  }
  free(P); free(Ks); free(Qs); free(prod); free(tmp); free(S0); free(St); free(term); free(X);
  return 0;
}
