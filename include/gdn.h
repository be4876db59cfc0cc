/*
 * gdn.h -- C ABI of the GB300 (sm_103a) chunked Gated DeltaNet library.
 *
 * The operation is the gated delta-rule recurrence
 *
 *     S_t = alpha_t S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T,
 *     o_t = S_t q_t,                      alpha_t = exp(g_t),
 *
 * with a d_v x d_k state per (sequence, head), evaluated in chunks of 64 tokens
 * with the WY representation (onedev.kr summary of the FlashQLA AICon 2026
 * talk, paragraph on the WY representation: intra-chunk K K^T and its inverse,
 * W and U, the chunk-to-chunk state pass, the output).  Background for the
 * recurrence itself: same page, paragraphs on the linear-attention background
 * (d x d state, O(N d^2)) and on the effective sliding window (alpha in (0,1),
 * L2-normalised keys).
 *
 * Conventions for every entry point
 *  - All tensor pointers are DEVICE pointers, contiguous, 16-byte aligned.
 *  - q, k [B, T, H, d_k]; v, o, dO [B, T, H, d_v] (token-major, then head,
 *    then feature).  With cu_seqlens != NULL the batch is packed: B == 1 and
 *    sequence n occupies tokens cu_seqlens[n] .. cu_seqlens[n+1]-1.
 *  - g, beta, dg, dbeta: fp32 [B, T, H].
 *  - States S0, S_T, dS_T, dS0: fp32 [N, H, d_v, d_k] row-major, N = number of
 *    sequences (B, or num_seqs when packed).  Row index = value feature.
 *  - The caller owns all memory.  The library never allocates: scratch memory
 *    is the caller's `workspace`, sized by the *_workspace_size queries.
 *  - Calls are asynchronous on `stream` and never synchronise the host.
 *  - Argument errors are detected on the host before any launch and return
 *    GDN_ERR_INVALID_ARG / GDN_ERR_UNSUPPORTED / GDN_ERR_WORKSPACE; a failed
 *    launch returns GDN_ERR_CUDA.  gdn_last_error_string() (thread-local)
 *    gives a one-line reason.
 *  - Results are deterministic (no floating-point atomics).
 *  - Log-gates: g = log(alpha) with alpha in (0, 1) per (token, head), any
 *    depth of decay (onedev.kr talk summary, paragraph on the effective sliding
 *    window, puts no lower bound on alpha).  Values below -128 act as -128: the
 *    decay across such a token is zero in fp32 either way.  A chunk whose
 *    in-chunk decay span is too wide for the factored form of the decay
 *    ratios takes them pairwise (see the forward below); results are the same
 *    up to rounding.
 */
#ifndef GDN_H_
#define GDN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *gdn_stream_t; /* same type as cudaStream_t; NULL = default stream */

typedef enum { GDN_BF16 = 0, GDN_FP32 = 1 } gdn_dtype;

enum {
  GDN_OK = 0,
  GDN_ERR_INVALID_ARG = 1, /* bad pointer, shape, stride or alignment                 */
  GDN_ERR_UNSUPPORTED = 2, /* valid but not implemented (e.g. d not in {64, 128})      */
  GDN_ERR_WORKSPACE = 3,   /* workspace NULL or smaller than the size query          */
  GDN_ERR_CUDA = 4,        /* a CUDA call or kernel launch failed                     */
  GDN_ERR_TIMEOUT = 5,     /* device side: a bounded wait expired (status bits 2, 3)  */
  GDN_ERR_NUMERIC = 6      /* device side: an fp16 operand overflowed (status bit 0)  */
};

enum {
  GDN_L2NORM_QK = 1u,  /* normalise q and k per token in-kernel: x / sqrt(|x|^2 + 1e-6)   */
  GDN_SP_OFF = 2u,     /* no intra-card sequence parallelism: one segment per sequence    */
  GDN_WINDOW_OFF = 4u, /* never skip the segment-start correction (always exact path)     */
  /* bf16, d = 128: run pass A, the start-state fix-up and pass B of each direction as one
   * launch (CTAs take work items in start order and wait, bounded, for the items they need)
   * instead of three.  Results are identical; measured on GB300 it is not faster (the
   * segments that need the fix-up keep the serial pass A -> fix-up -> pass B path, and the
   * launches it removes overlap their neighbours), so it is off by default. */
  GDN_SP_SINGLE_LAUNCH = 8u,
  /* Test hook for the bounded device waits (bf16, d = 128 chunk kernels): each tensor-core
   * kernel of the call first waits on a barrier that nothing arrives at, with a short bound;
   * the wait expires, sets status value 4 (see gdn_get_device_status) and the kernel returns
   * before any copy or product.  Outputs of such a call are not written. */
  GDN_DEBUG_WAIT_TIMEOUT = 0x80000000u,
  /* Test hook for the bounded waits between CTAs of the single-launch sequence parallelism
   * (GDN_SP_SINGLE_LAUNCH, with segments that take the exact fix-up): every segment whose start (end, reversed) is
   * fixed up waits for one more fix-up block than exists, with a short bound; the wait expires, sets
   * status value 16 and that segment's CTA returns without writing its outputs. */
  GDN_DEBUG_PEER_TIMEOUT = 0x40000000u
};

/* Problem description shared by the forward, the backward and the size queries. */
typedef struct {
  int B, T, H;                /* with cu_seqlens: B == 1 and T = total packed tokens     */
  int Dk, Dv;                 /* d_k == d_v, 64 or 128                                   */
  const int32_t *cu_seqlens;  /* device [num_seqs + 1], or NULL                          */
  int num_seqs;               /* number of sequences when cu_seqlens != NULL             */
  gdn_dtype dtype;            /* dtype of q, k, v, o, dO, dq, dk, dv                     */
  float scale;                /* o_t = S_t (scale * q_t), applied after normalisation    */
  unsigned flags;             /* GDN_L2NORM_QK | GDN_SP_OFF | GDN_WINDOW_OFF | GDN_SP_SINGLE_LAUNCH */
  int seg_chunks;             /* chunks per segment for sequence parallelism; 0 = auto   */
  int seg_first;              /* chunks of each sequence's first segment (needs          */
                              /* seg_chunks > 0); 0 = seg_chunks, or auto with it        */
  int reserved[2];            /* must be 0                                               */
} gdn_shape;

/* Workspace bytes needed by gdn_chunk_fwd / gdn_chunk_bwd for this shape on the
 * current device (the segment plan depends on its SM count).  0 on error. */
size_t gdn_fwd_workspace_size(const gdn_shape *shape);
size_t gdn_bwd_workspace_size(const gdn_shape *shape);

/*
 * Forward.  Computes o (and S_T if non-NULL) from q, k, v, g, beta and the
 * initial state S0 (NULL = zero state).
 *
 * Steps (all in sm_103a kernels on `stream`): segment plan from cu_seqlens;
 * gate scan (per-chunk log-decay sums, which mark segment starts inside an
 * effective sliding window -- onedev.kr talk summary, paragraph on the
 * effective sliding window; with bf16 and d = 128 the chunk-local half of the
 * forward forms these sums and decisions itself, no separate launch); pass A
 * over segments whose start must be corrected (state from zero plus the
 * composed d_k x d_k transition -- paragraph on parallelism); the sequential
 * start-state fix-up; pass B, the WY + state pass + output over every
 * segment (bf16, d = 128: the chunk-local half of every chunk, then the
 * recurrent half; equal-length batches may give each sequence a shorter
 * first segment, see seg_first, so that the recurrent passes fill the SMs in
 * one wave).  With bf16, d = 128 and
 * GDN_SP_SINGLE_LAUNCH, pass A, the fix-up and pass B are one launch: its CTAs
 * take work items in start order from lists the gate scan builds, and an item
 * that needs others' results (a fix-up, a fixed-up segment) waits for them
 * with a bound; the segments that need no fix-up run alongside pass A.
 * Decay ratios gamma_r / gamma_i inside a chunk are factored as
 * exp(G_r - G_mid) exp(G_mid - G_i) (G = in-chunk prefix of g, G_mid its
 * value at the chunk middle), one exponential per token (same page, paragraph
 * on SFU load); a chunk with |G_r - G_mid| > 80 for some r, where a factor
 * would leave fp32, takes exp(G_r - G_i) pairwise instead.
 */
int gdn_chunk_fwd(const gdn_shape *shape,
                  const void *q, const void *k, const void *v,
                  const float *g, const float *beta,
                  const float *S0, /* nullable */
                  void *o, float *S_T, /* S_T nullable */
                  void *workspace, size_t workspace_bytes, gdn_stream_t stream);

/*
 * Forward without any memory allocation by the caller or the library: the same
 * computation as gdn_chunk_fwd, with its scratch taken from a fixed device
 * array of GDN_STATIC_SCRATCH_BYTES that the library declares (the paper has no
 * counterpart; this serves callers that cannot call cudaMalloc, such as code
 * running inside another runtime's allocator-free region, a plugin host that
 * forbids device allocations, or a process whose memory pool is fully
 * reserved).  The caller still passes every input and output.
 *  - Every GPU that loads the library holds the array until the process exits.
 *  - The first call on a device looks the array's device address up (once per
 *    device, with that device current); make that first call before any stream
 *    capture.
 *  - If the shape's scratch with sequence parallelism does not fit, the call
 *    runs one segment per sequence (as with GDN_SP_OFF); if it still does not
 *    fit, it returns GDN_ERR_WORKSPACE and launches nothing.
 *  - All calls share the one array: calls that overlap on the GPU (other
 *    streams, other threads) race and must be serialised by the caller.
 *  - No cudaMalloc, cudaFree or allocating library routine is called.
 *  - A first call on a device made while `stream` is being captured returns
 *    GDN_ERR_INVALID_ARG and launches nothing.
 *  - The looked-up address is kept for the life of the process: after
 *    cudaDeviceReset (or any loss of the device's primary context) it is stale,
 *    and the library must not be called on that device again.
 *  - The device status word of the last call is read with
 *    gdn_get_device_status(shape, NULL, stream).
 */
#define GDN_STATIC_SCRATCH_BYTES (16u << 20)
int gdn_chunk_fwd_static(const gdn_shape *shape,
                         const void *q, const void *k, const void *v,
                         const float *g, const float *beta,
                         const float *S0, /* nullable */
                         void *o, float *S_T, /* S_T nullable */
                         gdn_stream_t stream);

/*
 * Backward (stateless: recomputes everything from the inputs).  Given dO and
 * dS_T (NULL = zero), writes dq, dk, dv (input dtype), dg, dbeta (fp32) and,
 * when S0 != NULL, dS0 (fp32; required then).  Gradients of q and k are with
 * respect to the raw inputs (through the optional normalisation and scale).
 * The WY backward forms dA and dA^T into one symmetric matrix multiplied with
 * K once (onedev.kr talk summary, paragraph on SFU load, last sentence).
 */
int gdn_chunk_bwd(const gdn_shape *shape,
                  const void *q, const void *k, const void *v,
                  const float *g, const float *beta,
                  const float *S0,   /* nullable */
                  const void *dO,
                  const float *dS_T, /* nullable */
                  void *dq, void *dk, void *dv, float *dg, float *dbeta,
                  float *dS0,        /* required iff S0 != NULL */
                  void *workspace, size_t workspace_bytes, gdn_stream_t stream);

/*
 * Saved-context training pair: the forward also leaves, in a caller-owned
 * buffer `saved`, what the backward would otherwise recompute -- the state at
 * every chunk start (fp16 for bf16 inputs, fp32 for fp32 inputs; [chunks, H,
 * d_v, d_k]) and, for bf16 with d = 128, the chunk context after it, in this
 * order: fp16 64 x 64 tiles [chunks, H, 5, 64, 64] X1 = Ahat diag(beta),
 * X2 = lower(diag(gamma) Ahat diag(beta / gamma)), Ahat = (I + diag(beta) N)^{-1},
 * P = diag(gamma) tril(Q K^T) diag(1 / gamma) and N (the strict lower
 * triangle of K K^T, normalised keys), with gamma_r = exp(in-chunk prefix sum
 * of g); fp16 128 x 64 tiles [chunks, H, 2, 128, 64] W^T (columns scaled by
 * gamma) and Ut^T = U^T - S0 W^T; the fp16 operand tiles [chunks, H, 3, 64,
 * 128] of K, Q (normalised, Q scaled) and V; fp32 [chunks, H, 2, 64]
 * reciprocal norms 1/|k|, 1/|q| (onedev.kr FlashQLA talk summary, paragraph
 * on the WY representation, which names these intra-chunk quantities).  Last,
 * for every dtype and d, the fp32 sum of g over each chunk [chunks, H] (the
 * gate scan's result, from which the backward decides its segment warm-ups
 * without reading g again).  The backward then starts at the reverse chain.  This trades memory for time
 * (d = 128, bf16: 152.5 KB per chunk and head, 640 MB for 32 heads x 8192
 * tokens); the chunked algorithm as published recomputes these in the
 * backward instead, and gdn_chunk_bwd keeps that form.
 *  - gdn_saved_size: bytes of `saved` for this shape (0 on error).
 *  - gdn_bwd_saved_workspace_size: workspace bytes of gdn_chunk_bwd_saved
 *    (smaller than gdn_bwd_workspace_size by the recomputed regions).
 *  - gdn_chunk_fwd_save: exactly gdn_chunk_fwd (same o and S_T) plus the
 *    writes to `saved` (non-NULL, 16-byte aligned, >= gdn_saved_size bytes,
 *    else GDN_ERR_INVALID_ARG / GDN_ERR_WORKSPACE before any launch).
 *  - gdn_chunk_bwd_saved: exactly gdn_chunk_bwd, reading `saved` instead of
 *    recomputing.  The shape (including cu_seqlens contents, flags and
 *    scale), q, k, v, g, beta and S0 must be those of the forward that wrote
 *    `saved`, and `saved` must not have been modified since; the library
 *    cannot check this, and other inputs give gradients of another problem.
 *    The segment plan (seg_chunks, GDN_SP_OFF) may differ between the two
 *    calls: `saved` is indexed by chunk, not by segment.
 */
size_t gdn_saved_size(const gdn_shape *shape);
size_t gdn_bwd_saved_workspace_size(const gdn_shape *shape);
int gdn_chunk_fwd_save(const gdn_shape *shape,
                       const void *q, const void *k, const void *v,
                       const float *g, const float *beta,
                       const float *S0, /* nullable */
                       void *o, float *S_T, /* S_T nullable */
                       void *saved, size_t saved_bytes,
                       void *workspace, size_t workspace_bytes, gdn_stream_t stream);
int gdn_chunk_bwd_saved(const gdn_shape *shape,
                        const void *q, const void *k, const void *v,
                        const float *g, const float *beta,
                        const float *S0,   /* nullable */
                        const void *dO,
                        const float *dS_T, /* nullable */
                        void *dq, void *dk, void *dv, float *dg, float *dbeta,
                        float *dS0,        /* required iff S0 != NULL */
                        const void *saved, size_t saved_bytes,
                        void *workspace, size_t workspace_bytes, gdn_stream_t stream);

/* Token-by-token (recurrent) forward for decoding a few tokens per sequence,
 * e.g. after a chunked prefill: for every sequence n < B, head h and token
 * t = 0 .. T-1 in order,
 *     S <- exp(g_t) S;   S <- S + beta_t (v_t - S k_t) k_t^T;   o_t = S (scale q_t)
 * with q_t, k_t L2-normalised first when GDN_L2NORM_QK is set.  This is the
 * recurrence stated in the header above, evaluated without chunking (the
 * tilnote.io note on FlashQLA, section on the workloads it wins, names
 * agentic inference as a target use; the onedev.kr summary's background
 * paragraph states the d x d state update).
 *   q, k, v, o: [B, T, H, d] (dtype of the shape); g, beta: fp32 [B, T, H];
 *   S_in: fp32 [B, H, d_v, d_k] or NULL (zero state); S_out: fp32 [B, H, d_v, d_k],
 *   which may be the same buffer as S_in (updated in place).
 * The shape must have cu_seqlens == NULL (GDN_ERR_UNSUPPORTED otherwise),
 * d 64 or 128, bf16 or fp32 (fp32 also at d = 128); seg_chunks and the SP flags
 * are ignored.  T == 0 copies S_in (or zeros) to S_out.  No workspace; state
 * precision fp32 throughout; asynchronous on `stream`. */
int gdn_recurrent_fwd(const gdn_shape *shape, const void *q, const void *k, const void *v, const float *g,
                      const float *beta, const float *S_in, void *o, float *S_out, gdn_stream_t stream);

/* Reads the device status word that the kernels of the last call on `stream`
 * set (synchronises the stream).  Every bit means the outputs of that call are
 * not reliable:
 *   bit 0 (1): numeric guard -- a value that becomes an fp16 tensor-core
 *              operand (q, k, v or dO widened from bf16, a chunk-start state,
 *              dS, Ut or dUt) was not finite or beyond +-65504;
 *   bit 1 (2): cu_seqlens is not non-decreasing, or describes more chunks or
 *              segments than the workspace was sized for;
 *   bit 2 (4): a tensor-core completion wait ran past its iteration limit (the
 *              kernel stopped that work item and returned);
 *   bit 3 (8): a TMA tile-load wait ran past its iteration limit (likewise);
 *   bit 4 (16): a wait for another CTA's work item of the single-launch
 *              sequence parallelism ran past its limit (the waiting item
 *              returned without output).
 * Returns the word (0 = clean), or -1 on a CUDA error.  `workspace` is the one
 * passed to that call, or NULL for a call of gdn_chunk_fwd_static (then the
 * word is read from the static scratch on the current device).  The status
 * lives in the caller's workspace because the library allocates nothing, which
 * is why this takes the workspace and not the stream alone. */
int gdn_get_device_status(const gdn_shape *shape, const void *workspace, gdn_stream_t stream);

/* Maps a status word of gdn_get_device_status to one status code: GDN_OK (0),
 * GDN_ERR_INVALID_ARG (bit 1), GDN_ERR_TIMEOUT (bits 2, 3, 4), GDN_ERR_NUMERIC
 * (bit 0), in that order of precedence; GDN_ERR_CUDA for -1. */
int gdn_device_status_code(int word);

/* The segment plan for this shape on the current device: chunks per segment,
 * an upper bound on the number of segments, on the number of chunks, and the
 * chunks of each sequence's first segment.  Any output pointer may be NULL. */
int gdn_plan_query(const gdn_shape *shape, int *seg_chunks, int *max_segments, int *max_chunks, int *seg_first);

/* The library's cost model of that plan: the modelled time in microseconds of the forward's state
 * pass and of the backward's reverse chain on the current device (the passes whose length the
 * segment plan sets; the chunk-parallel kernels do not depend on it).  The automatic plan is the
 * segment length that minimises their sum.  The model's constants are GB300 measurements; the
 * paragraph on parallelism of the onedev.kr talk summary calls the pages' own split model coarse. */
int gdn_plan_estimate(const gdn_shape *shape, double *fwd_us, double *bwd_us);

/* Diagnostics for benchmarks: when enabled, every kernel launch of the library
 * is bracketed by CUDA events (from a pool created on the first enable) on its
 * stream.  gdn_profile_report() waits for the recorded events and writes one
 * line "<kernel> <launches> <total_ms>" per kernel into buf (truncated to len),
 * returning the full report length; reset != 0 clears the totals. */
int gdn_profile_enable(int on);
int gdn_profile_report(char *buf, size_t len, int reset);
/* Restrict the bracketing to launches of one kernel name as it appears in the
 * report (NULL or "" = every launch), so that a timed loop carries the events of
 * the kernel it measures and no others. */
int gdn_profile_only(const char *name);

const char *gdn_status_string(int status);
const char *gdn_last_error_string(void); /* thread-local, "" if none */

#ifdef __cplusplus
}
#endif
#endif /* GDN_H_ */
