/*
 * gdr.h -- C ABI of the GB300 chunkwise gated delta rule forward library.
 *
 * The operation. For each batch row b and value head hv, with the state S a
 * K x V matrix (rows = key channels) that starts at initial_state[b, hv] (or 0),
 * every token t applies
 *     S <- exp(g_t) * S                        (decay: one scalar per token and head,
 *                                               or one factor per key channel)
 *     S <- S + beta_t k_t (v_t - S^T k_t)^T    (delta-rule write)
 *     o_t = S^T (scale * q_t)
 * where q_t, k_t are L2-normalised first when use_qk_l2norm is set
 * (x / sqrt(sum x^2 + 1e-6)). Value head hv reads query/key head hv / (HV / H).
 * This is the recurrence of the "分块并行计算（Chunkwise）" lecture notes
 * (section "为什么需要分块？") with the gate of Gated DeltaNet / KDA, the L2 norm
 * and default scale of "DeltaNet chunk kernel optimization" (_l2norm,
 * 1/sqrt(K)), and the tensor shapes of the notes' shape table (形状流水线).
 *
 * The library computes it in the chunk form of the same notes (section
 * "chunk 内的 cumsum 与下三角解" and the inter-chunk loop): per chunk of C tokens
 * a gate cumsum, the decayed dots A_kk and A_qk, the unit lower-triangular
 * system M = I + tril(A_kk * beta, -1) solved for W = M^-1 (exp(G) k) and
 * U = M^-1 v, then the state recurrence across chunks. A sequence whose length
 * is not a multiple of C is handled as if zero-padded (q = k = v = g = beta = 0
 * on the padding, "Pad to chunk boundary" of the optimisation script); padded
 * rows are never written.
 *
 * Conventions for every entry point:
 *  - All tensors are dense, row-major, contiguous, in the layouts given below.
 *  - Pointers marked (device) are device pointers on the current CUDA device;
 *    pointers marked (host) are host pointers (pinned memory gives asynchronous
 *    copies; pageable memory works but the copies then block the host).
 *  - Every device or host tensor base must be 16-byte aligned
 *    (GDR_ERR_ALIGNMENT otherwise).
 *  - The caller owns every buffer. The library allocates no device memory
 *    and frees nothing; it keeps no state between calls except the
 *    per-device cache of kernel attributes.
 *  - Work is enqueued asynchronously on `stream` (NULL = the legacy default
 *    stream). Argument errors are reported synchronously and enqueue nothing.
 *  - Launch failures return GDR_ERR_CUDA. A device-side bounded wait that
 *    gives up records an error word in the workspace; gdr_stream_status then
 *    returns GDR_ERR_TIMEOUT.
 */
#ifndef GDR_H_
#define GDR_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t / CUstream, declared here so that this header
 * needs no CUDA include. */
typedef struct CUstream_st* gdr_stream_t;

typedef enum {
  GDR_OK = 0,
  GDR_ERR_INVALID_ARG = 1,  /* null pointer, negative or inconsistent size, HV % H != 0, bad scale */
  GDR_ERR_UNSUPPORTED = 2,  /* valid but not implemented: head dim, chunk size, dtype combination */
  GDR_ERR_ALIGNMENT = 3,    /* a tensor base is not 16-byte aligned */
  GDR_ERR_WORKSPACE = 4,    /* workspace missing or smaller than gdr_chunk_fwd_workspace_size */
  GDR_ERR_CUDA = 5,         /* a CUDA runtime call or kernel launch failed */
  GDR_ERR_TIMEOUT = 6       /* a device-side bounded wait gave up (see gdr_stream_status) */
} gdr_status;

typedef enum { GDR_F32 = 0, GDR_BF16 = 1 } gdr_dtype;

typedef enum {
  GDR_GATE_SCALAR = 0,   /* g [B, T, HV]: one log-decay per token and value head (Gated DeltaNet) */
  GDR_GATE_PER_KEY = 1,  /* g [B, T, HV, K]: one log-decay per key channel (KDA) */
  GDR_GATE_NONE = 2      /* ungated delta rule (DeltaNet): g is not read and may be NULL;
                            every decay factor is 1, i.e. g identically 0 */
} gdr_gate_mode;

/* Problem sizes. q, k have H heads of K channels; v, o have HV value heads of
 * V channels (HV a multiple of H); B batch rows of T tokens. */
typedef struct {
  int B, T, H, HV, K, V;
  int in_dtype;   /* gdr_dtype of q, k, v */
  int out_dtype;  /* gdr_dtype of o */
} gdr_dims;

/*
 * gdr_chunk_fwd -- chunkwise gated delta rule forward pass on the GPU.
 *
 *   q, k           (device) [B, T, H, K]   in_dtype
 *   v              (device) [B, T, HV, V]  in_dtype
 *   g              (device) fp32, [B, T, HV] (GDR_GATE_SCALAR) or [B, T, HV, K] (GDR_GATE_PER_KEY);
 *                  natural-log decay per token (any sign; |in-chunk cumsum span| must stay
 *                  below ~80 so that exp() of it is finite in fp32); not read, and may be
 *                  NULL, with GDR_GATE_NONE
 *   beta           (device) fp32 [B, T, HV]
 *   initial_state  (device) fp32 [B, HV, K, V], or NULL for a zero state
 *   chunk_size     C: 16, 32, 64 (64 is the tensor-core path) or 128 (general path)
 *   scale          multiplies q after the optional L2 norm; finite and > 0
 *                  (the usual choice is 1/sqrt(K))
 *   use_qk_l2norm  nonzero: L2-normalise q and k per token and head first
 *   gate_mode      gdr_gate_mode
 *   out            (device) [B, T, HV, V] out_dtype
 *   final_state    (device) fp32 [B, HV, K, V], or NULL to skip it; may alias
 *                  initial_state (each state is read before it is written)
 *   workspace      (device) scratch of at least gdr_chunk_fwd_workspace_size()
 *                  bytes, 256-byte aligned; contents on entry do not matter
 *
 * Supported: K, V in 1..256 (independently) on the general fp32 path, which
 * streams the head dims through shared memory; bf16 inputs with K = V = 128 and
 * C = 64 take the tcgen05 tensor-core path. Larger head dims return
 * GDR_ERR_UNSUPPORTED.
 * T == 0 writes final_state = initial_state (or zeros) and nothing else.
 * Concurrent calls must use distinct workspaces.
 */
gdr_status gdr_chunk_fwd(const void* q, const void* k, const void* v, const float* g,
                         const float* beta, const float* initial_state, int chunk_size,
                         float scale, int use_qk_l2norm, int gate_mode, void* out,
                         float* final_state, const gdr_dims* dims, void* workspace,
                         size_t workspace_bytes, gdr_stream_t stream);

/*
 * gdr_chunk_prepare / gdr_chunk_recur -- gdr_chunk_fwd in its two stages.
 *
 * gdr_chunk_prepare runs the chunk-local kernel: per chunk, the gate cumsum,
 * the decayed dots A_kk / A_qk, the triangular solve for W and U, written into
 * `workspace` (the "chunk 内的 cumsum 与下三角解" section of the notes).
 * gdr_chunk_recur then runs the state recurrence across chunks (the notes'
 * inter-chunk loop) and writes out / final_state. gdr_chunk_fwd computes what
 * prepare followed by recur on the same stream computes (in one cooperative
 * launch where it can, see gdr_set_flag_wait_limit).
 *
 * The prepared workspace does not depend on the initial state: after one
 * prepare, recur may run any number of times with different initial states
 * (each run overwrites out / final_state). Every recur must use the q, k,
 * chunk_size, scale, use_qk_l2norm, gate_mode and dims of the prepare that
 * filled the workspace, and q / k must still hold the same values. Argument
 * meaning, layouts, alignment and errors are those of gdr_chunk_fwd; prepare
 * ignores out / final_state, recur ignores v / g / beta.
 */
gdr_status gdr_chunk_prepare(const void* q, const void* k, const void* v, const float* g,
                             const float* beta, int chunk_size, float scale, int use_qk_l2norm,
                             int gate_mode, const gdr_dims* dims, void* workspace,
                             size_t workspace_bytes, gdr_stream_t stream);

gdr_status gdr_chunk_recur(const void* q, const void* k, const float* initial_state,
                           int chunk_size, float scale, int use_qk_l2norm, int gate_mode,
                           void* out, float* final_state, const gdr_dims* dims, void* workspace,
                           size_t workspace_bytes, gdr_stream_t stream);

/* Bytes of device workspace gdr_chunk_fwd needs for these sizes (0 if the
 * arguments are invalid or unsupported). */
size_t gdr_chunk_fwd_workspace_size(const gdr_dims* dims, int chunk_size, int gate_mode);

/*
 * gdr_chunk_fwd_host -- the same forward pass on HOST tensors.
 *
 * Copies q, k, v, g, beta and initial_state (host, same layouts and dtypes as
 * above) into `device_buffer`, runs gdr_chunk_fwd there, and copies o and
 * final_state back to `out` and `final_state` (host), all enqueued on `stream`.
 * The call returns once the work is enqueued; synchronise `stream` (or call
 * gdr_stream_status) before reading the outputs. device_buffer (device) must
 * hold gdr_chunk_fwd_host_buffer_size() bytes and be 256-byte aligned.
 */
gdr_status gdr_chunk_fwd_host(const void* q, const void* k, const void* v, const float* g,
                              const float* beta, const float* initial_state, int chunk_size,
                              float scale, int use_qk_l2norm, int gate_mode, void* out,
                              float* final_state, const gdr_dims* dims, void* device_buffer,
                              size_t device_buffer_bytes, gdr_stream_t stream);

size_t gdr_chunk_fwd_host_buffer_size(const gdr_dims* dims, int chunk_size, int gate_mode,
                                      int with_initial_state, int with_final_state);

/*
 * gdr_stream_status -- synchronise `stream`, then report errors.
 * Returns GDR_ERR_CUDA if the stream reports an error, GDR_ERR_TIMEOUT if a
 * kernel that ran with this workspace recorded a bounded-wait timeout (the
 * word is cleared by the next gdr_chunk_fwd on that workspace), else GDR_OK.
 * `workspace` may be NULL to check only the stream.
 */
gdr_status gdr_stream_status(gdr_stream_t stream, void* workspace);

/*
 * gdr_set_flag_wait_limit -- bound of the device waits of the one-launch forward.
 *
 * With the scalar gate on the tensor-core path, gdr_chunk_fwd runs both stages
 * in one cooperative launch when the problem has few enough chains (B HV
 * value heads x 4 chains at most half the SMs): CTAs produce each chunk's
 * operands and raise a flag for it, chain CTAs of the same launch wait for
 * the flag before they read the chunk, and the outputs of each chunk are
 * formed once its chains have marked it exported. A chain polls a flag, and an
 * output item a mark, at most `polls` times, about 64 ns apart. If it is still
 * down, the CTA records GDR_ERR_TIMEOUT in the workspace error word
 * (gdr_stream_status reports it) and runs to its end on whatever the
 * workspace holds: the call then finishes with wrong outputs instead of
 * hanging. The default, 2^24 polls (about a second), is far beyond any real
 * wait.
 *
 *   polls   >= 0: the new bound, for calls enqueued from now on (all devices,
 *           all threads); < 0: leave the bound as it is.
 * Returns the bound in force before the call.
 */
int64_t gdr_set_flag_wait_limit(int64_t polls);

/*
 * gdr_chunk_fwd_noalloc -- gdr_chunk_fwd without a caller workspace.
 *
 * There is no counterpart of this entry point in the method's sources; it
 * exists for callers that cannot hand the library a device buffer. Examples:
 * code that runs under an allocator other than CUDA's (or none), plug-ins that
 * must not touch the device heap, and callers in a region where cudaMalloc is
 * not allowed (it synchronises the device and is illegal while a stream is
 * being captured). Such callers still pass their inputs and outputs; the
 * scratch space comes from a fixed array in device global memory owned by the
 * library: GDR_NOALLOC_SCRATCH_BYTES per device that loads the library, held
 * until the process exits. Neither this call nor anything it calls allocates
 * or frees memory.
 *
 * Arguments, layouts and errors are those of gdr_chunk_fwd, minus the
 * workspace. Sizes whose gdr_chunk_fwd_workspace_size() exceeds
 * GDR_NOALLOC_SCRATCH_BYTES are rejected with GDR_ERR_WORKSPACE before
 * anything is enqueued. 64 MiB fits, for example, B=1, T=4096, 4 value heads,
 * K=V=128, C=64, scalar gate, bf16 inputs (a workspace of about 54.8 MB); the
 * same call with 5 value heads (about 68.5 MB) does not. (The scalar-gate fast
 * path needs about 214 KB per chunk of 64 tokens and value head.)
 *
 * The first call on a device looks up the array's device address (with that
 * device current) and caches it; make that first call before any stream
 * capture. Later calls outside capture look the address up again, so a
 * cudaDeviceReset leaves no stale address behind; calls on a stream being
 * captured use the cached one. All calls on a device share the one array,
 * which keeps whatever the last call left in it (each call rewrites everything
 * it reads, and clears the error word itself). Calls that can overlap on the
 * GPU (different streams without ordering) race on the array and must not be
 * issued. A device-side timeout of such a call is reported by
 * gdr_noalloc_stream_status, not by gdr_stream_status.
 */
#define GDR_NOALLOC_SCRATCH_BYTES (64u * 1024u * 1024u)

gdr_status gdr_chunk_fwd_noalloc(const void* q, const void* k, const void* v, const float* g,
                                 const float* beta, const float* initial_state, int chunk_size,
                                 float scale, int use_qk_l2norm, int gate_mode, void* out,
                                 float* final_state, const gdr_dims* dims, gdr_stream_t stream);

/*
 * gdr_noalloc_stream_status -- gdr_stream_status for gdr_chunk_fwd_noalloc.
 * The library-owned array holds the error word of the last no-alloc call on
 * the current device; this synchronises `stream` and reports it:
 * GDR_ERR_CUDA if the stream reports an error, GDR_ERR_TIMEOUT if a device
 * wait of that call gave up, else GDR_OK. No counterpart in the method's
 * sources; it completes gdr_chunk_fwd_noalloc, whose callers hold no
 * workspace to pass to gdr_stream_status.
 */
gdr_status gdr_noalloc_stream_status(gdr_stream_t stream);

/*
 * gdr_recurrent_fwd -- the token-by-token (recurrent) form, for decoding.
 *
 * Applies, for each (b, hv) and token t = 0 .. T-1 in order, the recurrence
 * of the "分块并行计算（Chunkwise）" notes (section "为什么需要分块？"):
 *   S <- diag(exp(g_t)) S;  S <- S + beta_t k_t (v_t - S^T k_t)^T;  o_t = S^T (scale q_t)
 * with q_t, k_t L2-normalised when use_qk_l2norm is nonzero. T = 1 is the
 * single-token decode step; T > 1 runs the tokens one after another with the
 * state held on chip (one read and one write of each state per call). The
 * result equals gdr_chunk_fwd on the same tokens up to rounding.
 *
 *   q, k     (device) [B, T, H, K]   in_dtype
 *   v        (device) [B, T, HV, V]  in_dtype
 *   g, beta  as for gdr_chunk_fwd (g may be NULL with GDR_GATE_NONE)
 *   state    (device) fp32 [B, HV, K, V]: read as the state before token 0 and
 *            overwritten with the state after token T-1 (caller-owned)
 *   out      (device) [B, T, HV, V] out_dtype; must not overlap the inputs
 *   dims     as for gdr_chunk_fwd; K <= 256, any V (K <= 128 with V a multiple
 *            of 4 up to 128 and a 16-byte aligned state take the pipelined kernel)
 *
 * Errors: invalid arguments return synchronously and enqueue nothing;
 * B == 0 or T == 0 is a no-op. No workspace and no device waits.
 */
gdr_status gdr_recurrent_fwd(const void* q, const void* k, const void* v, const float* g,
                             const float* beta, float* state, float scale, int use_qk_l2norm,
                             int gate_mode, void* out, const gdr_dims* dims, gdr_stream_t stream);

/*
 * gdr_ssd_chunk_fwd -- chunkwise forward of the Mamba2 SSD recurrence, the
 * second workload of the "Chunkwise 并行算法 —— 线性注意力" page (§1.1-1.2):
 *   S <- diag(exp(g_t)) S + k_t v_t^T,   o_t = S^T (scale q_t)
 * i.e. the gated recurrence without the delta erase and without beta. It
 * runs on the same chunk machinery with the triangular solve dropped
 * (M = I, W = 0, U = v): for bf16 inputs with K = V = 128, C = 64 and the
 * scalar gate on the tensor-core path, where each chunk's state increment
 * k^T diag(exp(G_last - G) |k|^-1) v is formed with the chunk-local work and
 * the chain across chunks is a plain fp32 scan (the same launches as
 * gdr_chunk_fwd: one cooperative launch when the chains fit beside the
 * producers), otherwise on the general fp32 path. Arguments as for
 * gdr_chunk_fwd, minus beta; the workspace must hold
 * gdr_ssd_chunk_fwd_workspace_size() bytes.
 */
gdr_status gdr_ssd_chunk_fwd(const void* q, const void* k, const void* v, const float* g,
                             const float* initial_state, int chunk_size, float scale,
                             int use_qk_l2norm, int gate_mode, void* out, float* final_state,
                             const gdr_dims* dims, void* workspace, size_t workspace_bytes,
                             gdr_stream_t stream);
size_t gdr_ssd_chunk_fwd_workspace_size(const gdr_dims* dims, int chunk_size, int gate_mode);

/*
 * Segmented (parallel) scan of the same forward pass. Over a chunk the state
 * map of the chunk form is affine in S ("DeltaNet chunk kernel optimization",
 * cross-chunk state passing as a keyed scan of affine maps), so each sequence
 * is split into `segments` equal parts that run their recurrences at the same
 * time: each part's map S -> A_p S + B_p is computed (A_p from the identity
 * with the values' contribution dropped, B_p from a zero state), the maps are
 * chained serially to give every part its initial state, and the parts are
 * run once more from those states to write the outputs. The serial chain is
 * T / segments chunks long instead of T, at about three times the recurrence
 * work: it pays for few, long sequences (few chains for many SMs).
 *
 * Arguments as for gdr_chunk_fwd, plus
 *   segments   P >= 1 (1: exactly gdr_chunk_fwd). P > 1 needs K == V and T a
 *              multiple of P * chunk_size (else GDR_ERR_UNSUPPORTED), and the
 *              B P sequences of T / P tokens must be a supported problem.
 *   workspace  gdr_chunk_fwd_segmented_workspace_size() bytes (0: unsupported).
 *   final_state may alias initial_state, as for gdr_chunk_fwd.
 * Results equal gdr_chunk_fwd's up to rounding; errors as for gdr_chunk_fwd
 * (gdr_stream_status reads this workspace).
 */
gdr_status gdr_chunk_fwd_segmented(const void* q, const void* k, const void* v, const float* g,
                                   const float* beta, const float* initial_state,
                                   int chunk_size, float scale, int use_qk_l2norm, int gate_mode,
                                   int segments, void* out, float* final_state,
                                   const gdr_dims* dims, void* workspace,
                                   size_t workspace_bytes, gdr_stream_t stream);
size_t gdr_chunk_fwd_segmented_workspace_size(const gdr_dims* dims, int chunk_size,
                                              int gate_mode, int segments);

/* Static, human-readable name of a status code. */
const char* gdr_status_string(gdr_status s);

/* Which kernel path gdr_chunk_fwd takes for these arguments on the current
 * device: 0 = general fp32 CUDA-core path, 1 = tcgen05 tensor-core path in two
 * launches (chunk-local kernel, then the recurrence), 2 = tensor-core path in
 * one cooperative launch (scalar gate, few enough sequences for the device's
 * SMs: chains and chunk producers side by side), -1 = arguments rejected (the
 * status is written to *status if non-NULL). */
int gdr_chunk_fwd_path(const gdr_dims* dims, int chunk_size, int gate_mode, gdr_status* status);

/* Library version, (major << 16) | (minor << 8) | patch. */
int gdr_version(void);

#ifdef __cplusplus
}
#endif

#endif /* GDR_H_ */
