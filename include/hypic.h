/*
 * hypic.h -- C ABI of libhypic, the GB300 (sm_103a) linear-attention segment
 * transition cache.
 *
 * The method (HYPIC reading notes: "HYPIC: Accelerating Hybrid-Attention LLM
 * Serving with Position-Independent Caching"):
 *   every linear-attention head runs S_i = T_i S_{i-1} + u_i, o_i = q_i^T S_i
 *   (paper Eq. (2)).  A segment C = (1..m) is cached as the affine map
 *   F_C(S) = T_C S + S_{C|0} with T_C = T_m...T_1 and
 *   S_{C|0} = sum_t T_m...T_{t+1} u_t (Method 2).  Reuse composes the cached
 *   pairs in prompt order, S <- T_C S + S_{C|0} (paper Eq. (6)), after the
 *   running state has been advanced through the first w "seam" tokens of each
 *   inner segment (Method 5, seam windows).
 *
 * Conventions shared by every call
 * --------------------------------
 * Pointers: every tensor pointer is DEVICE memory owned by the caller,
 *   contiguous, 16-byte aligned, in the layout stated.  The library never
 *   allocates, frees or keeps a pointer after the call returns.
 * Execution: every call only enqueues work on `stream` (NULL = the legacy
 *   default stream) and returns; results are ready when the stream is.  A call
 *   may fork part of its work to a library-owned stream and join it back to
 *   `stream` with events before returning (the build with per-token outputs
 *   does); the ordering seen from `stream`, including under stream capture, is
 *   unchanged.
 * Shapes: d_k == d_v in {16, 32, 64, 128}; H >= 0; counts >= 0.  An empty
 *   batch (H, B or n_seg == 0) is a no-op that returns HYPIC_OK.
 * Errors: arguments are checked on the host before anything is enqueued and
 *   give HYPIC_EINVAL (bad pointer, size or layout) or HYPIC_EUNSUPPORTED
 *   (valid but not implemented shape); a failed launch gives HYPIC_ECUDA.
 *   Checks that need device data (pool indices, segment bounds) and bounded
 *   waits inside kernels record the first error in a per-device status word
 *   instead of faulting; hypic_stream_status() returns and clears it.
 * Families (paper Table 1), with the storage form of T_C (paper Table 3):
 *   SCALAR_CONST  T_i = gamma_h I,                u_i = k v^T   T_C: 1 float
 *   SCALAR        T_i = a_i I,                    u_i = k v^T   T_C: 1 float
 *   DIAG          T_i = diag(alpha_i),            u_i = k v^T   T_C: d_k floats
 *   DELTA         T_i = I - b_i k k^T,            u_i = b k v^T T_C: d_k x d_k
 *   GATED_DELTA   T_i = a_i (I - b_i k k^T),      u_i = b k v^T T_C: d_k x d_k
 *   KDA           T_i = (I - b_i k k^T) diag(g_i), u_i = b k v^T T_C: d_k x d_k
 * Token layouts: k, q, v [tokens, H, d] in the shape's in_dtype (fp32 or
 *   bf16); alpha fp32 [tokens, H] (SCALAR, GATED_DELTA), [tokens, H, d_k]
 *   (DIAG, and g of KDA), [H] (SCALAR_CONST), ignored for DELTA; beta fp32
 *   [tokens, H] (DELTA, GATED_DELTA, KDA only).  States and pairs are fp32, row index = key
 *   channel: S [.., H, d_k, d_v], T [.., H, t_size].
 */
#ifndef HYPIC_H
#define HYPIC_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* The same type as cudaStream_t (so this header needs no CUDA header). */
typedef struct CUstream_st *hypic_stream_t;

typedef enum {
    HYPIC_OK = 0,
    HYPIC_EINVAL = -1,      /* bad argument (null, misaligned, negative size, bad enum) */
    HYPIC_EUNSUPPORTED = -2,/* valid request the library does not implement */
    HYPIC_ECUDA = -3,       /* a CUDA runtime call or launch failed */
    HYPIC_ETIMEOUT = -4,    /* a bounded wait inside a kernel ran out */
    HYPIC_ENOSPACE = -5,    /* workspace too small for the request */
    HYPIC_EDEVICE = -6      /* a device-side check failed (index or bound out of range) */
} hypic_status;

typedef enum {
    HYPIC_FAM_SCALAR_CONST = 0,
    HYPIC_FAM_SCALAR = 1,
    HYPIC_FAM_DIAG = 2,
    HYPIC_FAM_DELTA = 3,
    HYPIC_FAM_GATED_DELTA = 4,
    HYPIC_FAM_KDA = 5       /* builds on the token-by-token path at every size */
} hypic_family;

typedef enum { HYPIC_F32 = 0, HYPIC_BF16 = 1 } hypic_dtype;

typedef struct {
    int32_t H;        /* heads (layers may be folded in: layer-major)       */
    int32_t d_k;      /* key width; must equal d_v                           */
    int32_t d_v;      /* value width                                         */
    int32_t family;   /* hypic_family                                        */
    int32_t in_dtype; /* hypic_dtype of k, q, v                              */
} hypic_shape;

/* Number of floats of one head's T_C: 1, d_k or d_k*d_k by family; 0 if invalid. */
int64_t hypic_t_size(const hypic_shape *shape);

/*
 * Segment build: (T_C, S_{C|0}) of one segment body for every head.
 * Defines: Method 2 (T_C = T_m...T_1, S_{C|0} from a zero state) and the
 * two-pass build of paper Sec. 5 (S_0 = 0 with writes -> S_{C|0}; S_0 = I with
 * u = 0 -> T_C), which this library evaluates in one pass over the
 * augmented state [T | S].
 *   k, v, q   [len, H, d]   q may be NULL; it is read only when o_out != NULL
 *   alpha, beta             gate layouts above, over the same len tokens
 *   T_out     [H, t_size]   S_out [H, d_k, d_v]
 *   o_out     [len, H, d_v] nullable: o_t = q_t^T S_t of the segment run from
 *                           a zero state (the independent-prefill outputs)
 *   ws, ws_bytes            workspace, see hypic_build_workspace_bytes()
 * len == 0 gives T_C = I and S_{C|0} = 0.
 */
hypic_status hypic_segment_build(const hypic_shape *shape, const void *k, const void *v,
                                 const void *q, const float *alpha, const float *beta, int64_t len,
                                 float *T_out, float *S_out, float *o_out, void *ws, size_t ws_bytes,
                                 hypic_stream_t stream);

/*
 * Batched segment build over n_seg bodies that sit anywhere on one token axis.
 *   seg_bounds DEVICE int64 [n_seg][2]: [begin, end) token range of body i;
 *              0 <= begin <= end <= n_tokens and end - begin <= max_len, else
 *              the body is skipped and HYPIC_EDEVICE is recorded.
 *   n_tokens   extent of the token axis of k, v, q, alpha, beta
 *   T_out [n_seg, H, t_size], S_out [n_seg, H, d_k, d_v]
 *   o_out [n_tokens, H, d_v] nullable, written at the bodies' token rows.
 */
hypic_status hypic_segment_build_batched(const hypic_shape *shape, int32_t n_seg,
                                         const int64_t *seg_bounds, int64_t max_len, int64_t n_tokens,
                                         const void *k, const void *v, const void *q, const float *alpha,
                                         const float *beta, float *T_out, float *S_out, float *o_out,
                                         void *ws, size_t ws_bytes, hypic_stream_t stream);

/*
 * (Both batched builds read whole 64-token chunks: the rows after a body's end up to its last
 * chunk boundary, or the end of the token axis, are read and enter with zero gates, so they must
 * hold finite values.)
 *
 * The batched build from inputs in host memory, with the host-to-device copies overlapped with
 * the build (the segment bodies of one request arrive over the host link while the earlier ones
 * are being built; the pair construction itself is that of hypic_segment_build_batched, HYPIC
 * reading notes Method 2 and paper Sec. 5).  The segments are taken in groups of consecutive
 * segments holding about an eighth of the body tokens each (at most 16 groups); each group's
 * token rows (its first body's begin through the end of its last body's last 64-token chunk) are
 * copied on copy_stream while the previous group builds on stream.
 *   seg_bounds_host         host array [n_seg][2], checked on the host (HYPIC_EINVAL if a body
 *                           leaves [0, n_tokens) or is longer than max_len) and copied to
 *                           bounds_dev (device, [n_seg][2])
 *   k_host, v_host          host [n_tokens, H, d] in in_dtype; alpha_host [n_tokens, H] (or
 *                           [n_tokens, H, d] for DIAG and KDA), unused for DELTA; beta_host
 *                           [n_tokens, H], delta families only.  Pinned memory lets the copies
 *                           run asynchronously; pageable memory works but the copies then block.
 *   k_dev, v_dev, alpha_dev, beta_dev
 *                           device buffers of the same shapes, 16-byte aligned; only the rows of
 *                           the bodies are written.  Caller-owned; the call makes the copies wait
 *                           for the work already on stream before overwriting them.
 *   T_out, S_out, ws        as in hypic_segment_build_batched (workspace sized by
 *                           hypic_build_workspace_bytes for the whole request).
 *   stream                  the build's stream; everything enqueued on it later sees the pairs.
 *   copy_stream             the copies' stream (null or equal to stream: no overlap).
 *   ready_event             a cudaEvent_t after which nothing reads the device input buffers any
 *                           more, or null: the copies then wait for all work already on stream.
 *                           A caller that alternates two sets of device buffers passes the event
 *                           it recorded after the earlier build of the same set, so that one
 *                           request's copies run while the previous request still computes.
 * Asynchronous; events the library creates once per device order the two streams.  Calls on one
 * device are serialised on the host while they enqueue.
 */
hypic_status hypic_segment_build_batched_host(const hypic_shape *shape, int32_t n_seg,
                                              const int64_t *seg_bounds_host, int64_t max_len, int64_t n_tokens,
                                              const void *k_host, const void *v_host, const float *alpha_host,
                                              const float *beta_host, void *k_dev, void *v_dev, float *alpha_dev,
                                              float *beta_dev, int64_t *bounds_dev, float *T_out, float *S_out,
                                              void *ws, size_t ws_bytes, hypic_stream_t stream,
                                              hypic_stream_t copy_stream, void *ready_event);

/*
 * Workspace bytes the build prefers for n_seg bodies of at most max_len tokens
 * (0 when the shape runs without one).  The d = 128 bf16 delta-family build
 * keeps one 49,664-byte operand record per (64-token chunk, head) in it; it
 * processes the heads in blocks that fit the workspace it is given, so any size
 * that holds one head's records (n_seg * ceil(max_len / 64) * 49,664 bytes)
 * works, and less gives HYPIC_ENOSPACE.  The preferred size covers all heads up
 * to about 4 GiB of records, plus N * 131,072 + 3,072 bytes for the split chain
 * schedule, N = min(256, max(U, U * ceil(max_len / 64) / 8)) with U = n_seg * heads:
 * the chain then runs at most one CTA per SM over equal shares of all chunks (a
 * cooperative launch), segments cut between CTAs (once when U exceeds the SMs,
 * into pieces of at least 8 chunks when there are fewer units) are rejoined by
 * composing their pieces' pairs in the kernel.  Without that room each unit gets
 * its own CTA; results agree to rounding either way.  The KDA family at d = 128
 * with bf16 inputs (pairs only) keeps an 82,432-byte record per (64-token chunk,
 * head) -- W_k^T, -A diag(b) and the per-channel decayed keys in hi and lo
 * pieces plus the chunk's channel decays -- so any size holding one head's
 * records (n_seg * ceil(max_len / 64) * 82,432 bytes) works; its preferred size
 * covers all heads up to about 4 GiB and has no split-schedule area.  The
 * workspace is caller-owned device memory, 16-byte aligned, and must not be used
 * by anything else until the stream reaches the end of the call.
 */
size_t hypic_build_workspace_bytes(const hypic_shape *shape, int32_t n_seg, int64_t max_len);

/*
 * The same for builds that also emit per-token outputs (q and o_out given): the tensor-core
 * build then keeps a 66,560-byte record per (64-token chunk, head) -- the 49,664 bytes above
 * plus gamma_t and the intra-chunk matrix M_ts = exp(G_t - G_s) q_t.k_s -- so any size holding
 * one head's records (n_seg * ceil(max_len / 64) * 66,560 bytes) works, and less gives
 * HYPIC_ENOSPACE.  0 when the shape builds without a workspace.
 */
size_t hypic_build_workspace_bytes_outputs(const hypic_shape *shape, int32_t n_seg, int64_t max_len);

/*
 * Allocation-free batched build.  No counterpart in the paper: it exists for
 * callers that cannot allocate device memory themselves -- code embedded in a
 * host framework that owns every device allocation through its own pool and
 * hands out no allocator, or a serving process that must not allocate after
 * start-up -- and so cannot pass the workspace hypic_segment_build_batched
 * wants.  Arguments, layouts and results are those of
 * hypic_segment_build_batched; the caller still passes inputs and outputs.
 * It allocates nothing: where the build needs a workspace it uses a fixed
 * scratch array of HYPIC_NOALLOC_SCRATCH_BYTES that lives in the library, so
 * every GPU that loads the library holds that memory until the process exits.
 * Limit: one head's operand records must fit the scratch.  Without outputs
 * (o_out NULL) a record is 49,664 bytes per (64-token chunk, head):
 * n_seg * ceil(max_len / 64) <= 1351.  With per-token outputs (q and o_out
 * given) it is 66,560 bytes: n_seg * ceil(max_len / 64) <= 1008.  The KDA
 * family's records are 82,432 bytes: n_seg * ceil(max_len / 64) <= 814.  Larger
 * requests return HYPIC_ENOSPACE before anything is enqueued.  More heads are
 * processed in blocks that fit.  The first call on a device looks up the
 * scratch array's device address (with that device current; a lookup that
 * fails is tried again on the next call); make that first call before any
 * stream capture.  All calls on a device share the one scratch array:
 * calls that overlap on the GPU (other streams, other host threads) race and
 * corrupt each other's results, so serialise them.  Nothing in the scratch has
 * to start at zero; every call writes each record before reading it.
 */
#define HYPIC_NOALLOC_SCRATCH_BYTES ((size_t)64 << 20)
hypic_status hypic_segment_build_batched_noalloc(const hypic_shape *shape, int32_t n_seg,
                                                 const int64_t *seg_bounds, int64_t max_len, int64_t n_tokens,
                                                 const void *k, const void *v, const void *q,
                                                 const float *alpha, const float *beta, float *T_out,
                                                 float *S_out, float *o_out, hypic_stream_t stream);

/*
 * Compose: S = T[i_{n-1}](...(T[i_0] S_init + S0[i_0])...) + S0[i_{n-1}] for
 * each of B requests and every head -- paper Eq. (6) evaluated as n
 * sequential S <- T_C S + S_{C|0} (Method 2).  The pairs live in a pool and
 * each request lists its own order:
 *   idx     DEVICE int32 [B, n], entries in [0, pool_size) (else HYPIC_EDEVICE)
 *   pool_T  [pool_size, H, t_size]   pool_S [pool_size, H, d_k, d_v]
 *   S_init  [B, H, d_k, d_v] or NULL (zero state)
 *   S_out   [B, H, d_k, d_v]; may be the same pointer as S_init.
 */
hypic_status hypic_compose(const hypic_shape *shape, int32_t B, int32_t n, const int32_t *idx,
                           int64_t pool_size, const float *pool_T, const float *pool_S,
                           const float *S_init, float *S_out, hypic_stream_t stream);

/*
 * Inclusive scan over affine maps (Method 2 composition rule
 * (T2,S2) o (T1,S1) = (T2 T1, T2 S1 + S2), associative, not commutative):
 *   (Tp_0, Sp_0) = (T_0, S_0),  (Tp_i, Sp_i) = (T_i, S_i) o (Tp_{i-1}, Sp_{i-1}).
 *   T, T_prefix [n, H, t_size];  S, S_prefix [n, H, d_k, d_v].
 *   Outputs must not overlap inputs.  ws is optional (NULL: one sequential
 *   chain per head).  Given at least hypic_scan_workspace_bytes() bytes
 *   (16-byte aligned), the delta families at d_k = d_v = 128 with fewer heads
 *   than fill the device run a two-level scan instead, using the composition
 *   rule's associativity: chunk totals, a scan of the totals, then every chunk
 *   again from its carry; about twice the work in far fewer sequential steps.
 *   hypic_scan_workspace_bytes() returns 0 when no workspace would be used.
 */
hypic_status hypic_affine_scan(const hypic_shape *shape, int32_t n, const float *T, const float *S,
                               float *T_prefix, float *S_prefix, void *ws, size_t ws_bytes,
                               hypic_stream_t stream);
size_t hypic_scan_workspace_bytes(const hypic_shape *shape, int32_t n);

/*
 * Seam advance (Method 5, seam windows): run the recurrence from the current
 * running state through w seam tokens of each of B requests, emitting
 * o_i = q_i^T S_i (post-update state, paper Eq. (2)).
 *   S_inout [B, H, d_k, d_v]           updated in place
 *   q, k, v [B, w, H, d]               alpha, beta: gate layouts over B*w tokens
 *   o_out   [B, w, H, d_v] or NULL
 */
hypic_status hypic_seam_advance(const hypic_shape *shape, int32_t B, float *S_inout, const void *q,
                                const void *k, const void *v, const float *alpha, const float *beta,
                                int32_t w, float *o_out, hypic_stream_t stream);

/*
 * Request assembly, fused: for each request b and head, starting from S_init
 * (or zero), for j = 0..n-1: if j >= 1 and w > 0, advance through the w seam
 * tokens of segment j and emit their outputs; then S <- T[idx[b,j]] S +
 * S0[idx[b,j]].  Segment 0 (the system prompt) has no seam (Method 5).
 *   seam_q, seam_k, seam_v [B, n-1, w, H, d]; seam_alpha, seam_beta: gate
 *   layouts over B*(n-1)*w tokens; o_out [B, n-1, w, H, d_v] or NULL.
 *   Other arguments as hypic_compose.  w == 0 is hypic_compose.
 */
hypic_status hypic_assemble(const hypic_shape *shape, int32_t B, int32_t n, int32_t w,
                            const int32_t *idx, int64_t pool_size, const float *pool_T,
                            const float *pool_S, const void *seam_q, const void *seam_k,
                            const void *seam_v, const float *seam_alpha, const float *seam_beta,
                            const float *S_init, float *S_out, float *o_out, hypic_stream_t stream);

/*
 * 16-bit storage of cached pairs (HYPIC notes, Method 3, Table 3: the cache sizes there
 * assume 16-bit T_C and S).  Rounds n_pairs fp32 pairs to bf16, round to nearest even:
 *   T [n_pairs, H, t_size] fp32 -> T_lp, same layout, bf16
 *   S [n_pairs, H, d_k, d_v] fp32 -> S_lp, same layout, bf16
 * Device pointers, 16-byte aligned; the outputs must not overlap the inputs.  bf16 keeps
 * fp32's exponent range, so a T_C that has decayed far stays representable; each stored
 * value carries a relative rounding error of at most 2^-9.
 * Errors: HYPIC_EINVAL (null or misaligned pointer, n_pairs < 0), HYPIC_EUNSUPPORTED (shape),
 * HYPIC_ECUDA.
 */
hypic_status hypic_pairs_to_bf16(const hypic_shape *shape, int64_t n_pairs, const float *T, const float *S,
                                 void *T_lp, void *S_lp, hypic_stream_t stream);

/*
 * hypic_compose and hypic_assemble over a pool stored in bf16 (as written by
 * hypic_pairs_to_bf16; same layouts, half the bytes).  The running state, S_init, S_out and
 * o_out stay fp32; each step computes S <- T S + S0 with the stored bf16 values taken
 * exactly (no further rounding of T or S0), so the result matches a float64 composition of
 * the same stored values to fp32 accuracy.  Supported for every family at d_k = d_v = 128 and
 * for the scalar and diagonal families at every size; the delta families at d < 128 return
 * HYPIC_EUNSUPPORTED before anything is enqueued.  Other arguments and errors as in
 * hypic_compose / hypic_assemble.
 */
hypic_status hypic_compose_bf16(const hypic_shape *shape, int32_t B, int32_t n, const int32_t *idx,
                                int64_t pool_size, const void *pool_T, const void *pool_S,
                                const float *S_init, float *S_out, hypic_stream_t stream);
hypic_status hypic_assemble_bf16(const hypic_shape *shape, int32_t B, int32_t n, int32_t w,
                                 const int32_t *idx, int64_t pool_size, const void *pool_T,
                                 const void *pool_S, const void *seam_q, const void *seam_k,
                                 const void *seam_v, const float *seam_alpha, const float *seam_beta,
                                 const float *S_init, float *S_out, float *o_out, hypic_stream_t stream);

/* ---- Boundary patches (HYPIC notes, Method 6: causal convolution and RoPE at segment
 * boundaries; paper Sec. 4.2-4.3, Eqs. (7), (8)).  None allocates; all are asynchronous on
 * `stream`; pointers are caller-owned device memory, 16-byte aligned. */

typedef enum { HYPIC_ACT_IDENTITY = 0, HYPIC_ACT_SILU = 1 } hypic_activation;

/*
 * RoPE key shift, Eq. (8): K_b = R(b - a) K_a, for keys cached at one start position and reused
 * at another (delta = b - a, any sign).  K_in, K_out [n_rows, d] (n_rows = tokens x heads),
 * dtype HYPIC_F32 or HYPIC_BF16, K_out may equal K_in.  Rotate-half convention: dims i and
 * i + rot_dim/2 (i < rot_dim/2) form a pair turned by delta * base^(-2i/rot_dim); dims >=
 * rot_dim pass through.  2 <= rot_dim <= d <= 512, rot_dim even, base > 1.  The angle is
 * reduced modulo 2 pi in double precision, the rotation applied in fp32 (bf16 outputs are
 * rounded to nearest even).  Errors: HYPIC_EINVAL (pointers, sizes), HYPIC_ECUDA; a staged copy
 * that never lands (bounded wait) is recorded as HYPIC_ETIMEOUT for hypic_stream_status.
 */
hypic_status hypic_rope_shift(int64_t n_rows, int32_t d, int32_t rot_dim, double base, int64_t delta,
                              hypic_dtype dtype, const void *K_in, void *K_out, hypic_stream_t stream);

/*
 * Linear-layer state re-rotation, Eq. (7): S_{C|b} = R(b - a) S_{C|a} applied to the key (row)
 * index of S [n, H, d_k, d_v] fp32, in place; T_C is unchanged.  Exact only when the transition
 * commutes with the rotation, so only the scalar families are accepted (HYPIC_FAM_SCALAR_CONST,
 * HYPIC_FAM_SCALAR); others return HYPIC_EUNSUPPORTED.  Rotation as in hypic_rope_shift, with
 * rot_dim <= d_k; errors as there.
 */
hypic_status hypic_state_rerotate(const hypic_shape *shape, int64_t n, float *S_inout, int32_t rot_dim,
                                  double base, int64_t delta, hypic_stream_t stream);

/*
 * Causal-convolution tail of each segment body (what the cache keeps so that the next
 * segment's first k - 1 conv outputs can be recomputed): tail_out [n_seg, k-1, C] = rows
 * end-(k-1) .. end-1 of x [n_tokens, C] for body [begin, end) = seg_bounds[s] (device, int64
 * [n_seg][2]), zero where a row falls before begin.  dtype of x and tail_out: HYPIC_F32 or
 * HYPIC_BF16.  1 <= k <= 64.  Bad bounds are recorded as HYPIC_EDEVICE (hypic_stream_status)
 * and give zero rows.
 */
hypic_status hypic_conv_tail(int32_t C, int32_t k, int32_t n_seg, const int64_t *seg_bounds, int64_t n_tokens,
                             hypic_dtype dtype, const void *x, void *tail_out, hypic_stream_t stream);

/*
 * Depthwise causal convolution over the first w tokens of B segments, continuing from each
 * previous segment's tail:
 *   y[b, t, c] = act(bias[c] + sum_{j<k} weight[c, j] * x_{t-k+1+j}[c]),
 * where x_s = x_seam[b, s] for s >= 0 and tail[b, k-1+s] for s < 0.  x_seam [B, w, C] and tail
 * [B, k-1, C] in dtype (HYPIC_F32 or HYPIC_BF16; tail may be NULL when k == 1), weight [C, k]
 * and bias [C] (or NULL) fp32, y_out [B, w, C] fp32.  act: hypic_activation.  1 <= k <= 64.
 */
hypic_status hypic_conv_seam(int32_t B, int32_t w, int32_t C, int32_t k, hypic_dtype dtype, const void *x_seam,
                             const void *tail, const float *weight, const float *bias, int32_t act, float *y_out,
                             hypic_stream_t stream);

/*
 * Waits for `stream`, then returns and clears the status word of the current
 * device: HYPIC_OK, HYPIC_EDEVICE or HYPIC_ETIMEOUT (first error recorded by
 * any kernel since the last call), or HYPIC_ECUDA if the stream itself failed.
 */
hypic_status hypic_stream_status(hypic_stream_t stream);

/*
 * Self-test of failure detection (no counterpart in the paper).  Every wait inside
 * the library's kernels is bounded: when it runs out, the kernel records
 * HYPIC_ETIMEOUT in the status word and returns instead of hanging.  This call
 * enqueues a one-thread kernel whose wait can never be satisfied, bounded by
 * limit_cycles SM clock cycles (0 .. 4e9; a million cycles is about half a
 * millisecond), so a caller or a test can check that the timeout is reported by
 * hypic_stream_status() and that the device stays usable afterwards.
 */
hypic_status hypic_selftest_bounded_wait(int64_t limit_cycles, hypic_stream_t stream);

/* Static, never NULL. */
const char *hypic_strerror(hypic_status status);

/* Incremented on any incompatible change of this header. */
int32_t hypic_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* HYPIC_H */
