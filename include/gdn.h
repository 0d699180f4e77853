/*
 * gdn.h -- C ABI of the GB300 (sm_103a) chunkwise Gated DeltaNet forward with per-segment
 * affine state summaries.
 *
 * The operation (per batch b and head h; K x V fp32 state H):
 *   residual_t = beta_t * (v_t - k_t @ H_{t-1})
 *   H_t        = exp(g_t) * H_{t-1} + outer(k_t, residual_t)
 *   o_t        = q_t @ H_t
 * -- "RFC: HyperParallel Linear Attention Context Parallel", section 2.1. The state reads
 * the un-decayed H_{t-1}; g is a natural-log decay (g <= 0: the kernels rely on the state
 * only decaying); there is no query scale.
 * Computed in chunks of 64 tokens (gate cumsum, chunk K K^T, lower-triangular solve, WY
 * form, inter-chunk state scan, output) -- "Context Parallelism in ART", section 08,
 * "First parallelize within a GPU".
 * A contiguous segment of tokens acts on its incoming state as H_out = M @ H_in + S, with
 * M [K,K] and S [K,V]; two segments in order compose as M = M1 @ M0, S = M1 @ S0 + S1
 * (associative, not commutative) -- RFC section 2.2; ART section 08, "Then parallelize
 * across GPUs". Segments play the role of the pages' context-parallel ranks, here all on
 * one GPU.
 *
 * ---------------------------------------------------------------------------------------
 * Conventions shared by every call
 * ---------------------------------------------------------------------------------------
 * Layouts (row-major, contiguous, no strides):
 *   q, k     [B, T, H, K]        in_dtype
 *   v        [B, T, H, V]        in_dtype
 *   g, beta  [B, T, H]           in_dtype   (g: [B, T, H, K] when gate_k is set)
 *   o        [B, T, H, V]        out_dtype
 *   h0, h_final                  [B, H, K, V]           fp32
 *   M                            [nseg, B, H, K, K]     fp32   ((M@X)[i,v] = sum_j M[i,j] X[j,v])
 *   S, H_in                      [nseg, B, H, K, V]     fp32
 * Segment s covers tokens [s*T/nseg, (s+1)*T/nseg) of every sequence.
 *
 * Supported set (anything else returns an error and launches nothing):
 *   chunk == 64; K == V and K in {64, 128}; B, H >= 1; T >= 0; T % (64*nseg) == 0;
 *   1 <= nseg (and nseg <= T/64 when T > 0); B*T*H*max(K,V) < 2^40.
 *   in_dtype  in {GDN_DTYPE_F32, GDN_DTYPE_BF16}; out_dtype in {GDN_DTYPE_F32, GDN_DTYPE_BF16}.
 *   bf16 inputs with K == V == 128 run the tcgen05 tensor-core kernels (fp32 accumulation);
 *   fp32 inputs, and bf16 inputs with K == V == 64, run the fp32 CUDA-core kernels.
 *   Every device pointer must be 16-byte aligned (GDN_ERR_MISALIGNED otherwise).
 *
 * Ownership: the caller allocates every buffer (device memory) and keeps it alive until the
 * stream work completes. The library allocates nothing, keeps no state between calls and
 * never synchronises the stream, except gdn_check_device_error. One exception:
 * gdn_segmented_fwd_noalloc takes its scratch from an array the library itself owns (held
 * on every GPU that loads it), caches that array's address per device, and leaves the last
 * call's contents in it; calls to it that overlap on the GPU must be serialised (see its
 * description).
 *
 * Workspace: a caller-provided device buffer of at least gdn_workspace_bytes() bytes, whose
 * first 256 bytes must be zero before the first call that uses it (it holds the device
 * error word, see gdn_check_device_error). Calls that share a workspace must not overlap.
 *
 * Streams: `stream` is a cudaStream_t (NULL = the legacy default stream). Every call is
 * asynchronous on that stream. The returned status covers argument validation and launch
 * errors only; faults the kernels detect on the device (a bounded wait that ran out) are
 * recorded in the workspace's error word and reported by gdn_check_device_error.
 *
 * There is no CPU fallback: a call either launches its CUDA kernels or returns an error.
 */
#ifndef GDN_H_
#define GDN_H_

#include <stddef.h>

#if defined(__GNUC__)
#define GDN_API __attribute__((visibility("default")))
#else
#define GDN_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    GDN_OK = 0,
    GDN_ERR_INVALID_ARG = 1,       /* NULL required pointer, bad count, bad nseg */
    GDN_ERR_UNSUPPORTED_SHAPE = 2, /* K/V/chunk/T outside the supported set */
    GDN_ERR_UNSUPPORTED_DTYPE = 3, /* dtype code outside the supported set */
    GDN_ERR_MISALIGNED = 4,        /* a device pointer is not 16-byte aligned */
    GDN_ERR_WORKSPACE = 5,         /* workspace NULL or smaller than gdn_workspace_bytes() */
    GDN_ERR_CUDA = 6,              /* a CUDA runtime call or launch failed */
    GDN_ERR_TIMEOUT = 7,           /* a kernel's bounded wait ran out (device error word) */
    GDN_ERR_DEVICE = 8             /* the current device is not an sm_103 GPU */
} gdn_status;

typedef enum { GDN_DTYPE_F32 = 0, GDN_DTYPE_BF16 = 1 } gdn_dtype;

typedef struct {
    int B, T, H, K, V;
    int chunk;           /* tokens per chunk; must be 64 */
    gdn_dtype in_dtype;  /* storage type of q, k, v, g, beta */
    gdn_dtype out_dtype; /* storage type of o */
    /* 0: the read sees the state before this token's decay, r_t = beta_t (v_t - k_t@H_{t-1})
     *    (RFC section 2.1; transition exp(g_t) I - beta_t k_t k_t^T).
     * 1: the read sees the decayed state, r_t = beta_t (v_t - k_t@(exp(g_t) H_{t-1})) (ART
     *    section 08 "What a GDN token does to the state"; KDA design section 1.2; transition
     *    exp(g_t) (I - beta_t k_t k_t^T)). Every call below follows the flag. */
    int decay_first;
    /* 0: one gate per token and head, g is [B, T, H] (Gated DeltaNet).
     * 1: one gate per key channel, g is [B, T, H, K], and the state decays row by row,
     *    diag(exp(g_t)) H ("KDA Chunk Backward -- TPU/Pallas Kernel Design", section 1.2;
     *    with either reading above). Runs the fp32 CUDA-core kernels for every dtype. */
    int gate_k;
} gdn_problem;

/* Bytes of workspace the calls below need for this problem split into nseg segments
 * (nseg = 1 for gdn_chunk_fwd and gdn_segment_summary). Returns 0 for an invalid problem.
 * It holds the error word; for the tensor-core shapes (bf16 in, K == V == 128) the
 * per-chunk WY factors A diag(beta) and A diag(beta exp-decay), A = (I + L)^-1, as two bf16
 * 64 x 64 tiles per chunk without their zero blocks above the diagonal (10 KiB per chunk and
 * head, formed by one launch before the chains); and, with P = gdn_segmented_pieces(p, nseg)
 * pieces per sequence, fp32 [P,B,H,K,K]
 * and [P,B,H,K,V] arrays for the piece summaries (P >= 3) and one [P,B,H,K,V] for the state
 * entering each piece (P >= 2). P depends on the current device's SM count: size and run on
 * the same device. */
GDN_API size_t gdn_workspace_bytes(const gdn_problem* p, int nseg);

/* Pieces per sequence that gdn_segmented_fwd (and gdn_chunk_fwd, nseg = 1) cuts the tokens
 * into on the current device. The forward of piece 0 runs from h0 beside the affine summaries
 * of pieces 1..P-2 (RFC section 2.2), an in-order scan gives the state entering every piece,
 * and pieces 1..P-1 then run their chunked forward from those states: each phase has
 * B*H*(P-1) independent chains, so the GPU stays busy when B*H alone would not fill it. The
 * plan balances wave fill, chain length and scan steps: either P equal pieces with P a
 * multiple of nseg (segment starts are piece starts), or -- on the tensor-core path, when
 * each phase fits in one wave -- a piece 0 sized so that its forward ends with the summaries
 * and P-1 equal pieces after it, whose starts need not be segment starts (nseg equal pieces
 * when no device is current). Returns 0 for an invalid problem. */
GDN_API int gdn_segmented_pieces(const gdn_problem* p, int nseg);

/* The piece plan behind gdn_segmented_pieces: returns P (0 for an invalid problem) and, when
 * the pointers are non-NULL, the chunks of piece 0 (*first_chunks) and of each later piece
 * (*rest_chunks); first == rest for an equal-piece plan. For accounting of the work a call
 * does (which summaries run); same device dependence as gdn_segmented_pieces. */
GDN_API int gdn_segmented_plan(const gdn_problem* p, int nseg, int* first_chunks,
                               int* rest_chunks);

/* Chunked forward over all T tokens from the initial state h0.
 *   RFC section 2.1 (recurrence); ART section 08 "First parallelize within a GPU" (chunks).
 *   Runs as gdn_segmented_fwd with one segment (cut into gdn_segmented_pieces(p, 1) pieces);
 *   workspace: gdn_workspace_bytes(p, 1).
 *   h0       [B,H,K,V] fp32, or NULL for a zero initial state.
 *   o        [B,T,H,V] out_dtype, written.
 *   h_final  [B,H,K,V] fp32, the state after token T-1; NULL skips it.
 * T == 0 writes only h_final (= h0, or zeros). */
GDN_API gdn_status gdn_chunk_fwd(const gdn_problem* p, const void* q, const void* k, const void* v,
                         const void* g, const void* beta, const float* h0, void* o,
                         float* h_final, void* workspace, size_t workspace_bytes,
                         void* stream);

/* Affine summary of each of the nseg contiguous segments: H_out = M @ H_in + S.
 *   RFC section 2.2: S is the state the segment reaches from H_in = 0 and M is its
 *   linear action on any incoming state. Built chunk by chunk in WY form, so M is the
 *   ordered product of the per-token factors exp(g_t) I - beta_t k_t k_t^T.
 *   M [nseg,B,H,K,K] fp32 and S [nseg,B,H,K,V] fp32, written. */
GDN_API gdn_status gdn_segment_summary(const gdn_problem* p, int nseg, const void* k, const void* v,
                               const void* g, const void* beta, float* M, float* S,
                               void* workspace, size_t workspace_bytes, void* stream);

/* Exclusive in-order prefix scan of segment summaries (RFC section 2.2 compose; ART
 * section 08 prefix scan, made exclusive):
 *   H_in[0] = h0 (zeros if h0 == NULL),  H_in[s] = M[s-1] @ H_in[s-1] + S[s-1].
 *   M [nseg,B,H,K,K], S [nseg,B,H,K,V] fp32 in (M[nseg-1], S[nseg-1] are not read);
 *   H_in [nseg,B,H,K,V] fp32 out. Computed in fp32 on CUDA cores. Only p->B, p->H, p->K,
 *   p->V are read from the problem. */
GDN_API gdn_status gdn_summary_scan(const gdn_problem* p, int nseg, const float* M, const float* S,
                            const float* h0, float* H_in, void* stream);

/* The chunked forward of every segment from the state given for its start -- the last two
 * stages of the RFC's forward flow, "forward_apply_state" (per-chunk states) and
 * "forward_output" (token output), section 6.4.2, run by every emulated rank at once once it
 * has its H_in. Composed with gdn_segment_summary and gdn_summary_scan it is the pages'
 * literal flow: every rank's summary, the in-order summary apply, then each rank's local
 * forward (RFC sections 6.4.1 and 6.5).
 *   H_in     [nseg,B,H,K,V] fp32: the state entering each segment (NULL: zero for every
 *            segment); read only.
 *   o        [B,T,H,V] out_dtype, written.
 *   h_final  [B,H,K,V] fp32: the state after the last segment's last token; NULL skips it.
 *   Workspace: gdn_workspace_bytes(p, 1). Segment s covers tokens [s*T/nseg, (s+1)*T/nseg)
 *   and runs as one chain per (b, h, segment). T == 0 writes only h_final (= H_in[nseg-1],
 *   or zeros). */
GDN_API gdn_status gdn_segment_fwd(const gdn_problem* p, int nseg, const void* q, const void* k,
                                   const void* v, const void* g, const void* beta,
                                   const float* H_in, void* o, float* h_final, void* workspace,
                                   size_t workspace_bytes, void* stream);

/* The segmented forward (RFC section 6.4.1/6.4.2 forward flow on one GPU): with P =
 * gdn_segmented_pieces(p, nseg) pieces per sequence, piece 0's forward from h0 beside the
 * summaries of pieces 1..P-2, the in-order scan of those summaries from the state piece 0
 * ends in, then the chunked forward of pieces 1..P-1 from their scanned states. The state
 * entering segment s is written by the scan when it is a piece start, else by the forward of
 * the piece that contains it. o and h_final equal gdn_chunk_fwd's up to rounding.
 *   H_in_out [nseg,B,H,K,V] fp32: if non-NULL receives the scanned states; if NULL they
 *   live in the workspace. Workspace: gdn_workspace_bytes(p, nseg). */
GDN_API gdn_status gdn_segmented_fwd(const gdn_problem* p, int nseg, const void* q, const void* k,
                             const void* v, const void* g, const void* beta, const float* h0,
                             void* o, float* h_final, float* H_in_out, void* workspace,
                             size_t workspace_bytes, void* stream);

/* gdn_segmented_fwd with stage markers, for timing each kernel from the caller. If
 * stage_events is non-NULL it points to five cudaEvent_t that are recorded on `stream`
 * before the WY-factor launch, before the first phase (piece 0's forward and the piece
 * summaries), before the scan, before the second phase (the forward of pieces 1..P-1) and
 * after it (the WY launch is skipped on the CUDA-core path; with one piece the scan and the
 * second phase are empty). Same results as gdn_segmented_fwd. */
GDN_API gdn_status gdn_segmented_fwd_timed(const gdn_problem* p, int nseg, const void* q,
                                           const void* k, const void* v, const void* g,
                                           const void* beta, const float* h0, void* o,
                                           float* h_final, float* H_in_out, void* workspace,
                                           size_t workspace_bytes, void* stream,
                                           void* const* stage_events);

/* Size of the fixed scratch array behind gdn_segmented_fwd_noalloc (64 MiB). */
#define GDN_NOALLOC_SCRATCH_BYTES (64u * 1024u * 1024u)

/* gdn_segmented_fwd without a workspace, for callers that cannot allocate device memory:
 * a host framework that owns all device memory through its own pool, a request path that
 * must not pay an allocation's implicit synchronisation, or a program that only holds
 * buffers imported from another process. (The pages have no counterpart: this is an
 * interface choice of this library.)
 *   Arguments and results are those of gdn_segmented_fwd, minus H_in_out and the
 *   workspace. The scratch (WY tiles, summaries, scanned states, the error word) lives in one
 *   array of GDN_NOALLOC_SCRATCH_BYTES in the library's own device memory; every GPU that
 *   loads the library holds it until the process exits. The call allocates nothing.
 *   Limit: problems with gdn_workspace_bytes(p, nseg) > GDN_NOALLOC_SCRATCH_BYTES are
 *   rejected with GDN_ERR_WORKSPACE (at bf16, K = V = 128 and P >= 3 pieces that is
 *   B*H*(T/64*10 KiB + P*192 KiB) + 256 bytes at most 64 MiB, e.g. B*H = 32 heads of
 *   T = 2048 in 4 segments (4 pieces) take 34 MiB).
 *   device_error: optional (NULL to skip) 8-byte-aligned device pointer to two unsigned
 *   words that receive this call's device error word {code, detail} (see
 *   gdn_check_device_error for the codes) when the call's stream work completes.
 *   First call on a device: it looks up that device's copy of the array
 *   (cudaGetSymbolAddress) with the device current and caches the address per device; make
 *   it before any stream capture. The cache assumes the runtime's primary context of each
 *   device: calls made with another driver context current, or after cudaDeviceReset, are
 *   not supported (the cached address would belong to a context that is gone).
 *   All calls share the one array, which keeps the last call's contents (the call clears
 *   the error word itself): calls that overlap on the GPU -- on different streams, or from
 *   different host threads -- race on it and must be serialised by the caller. */
GDN_API gdn_status gdn_segmented_fwd_noalloc(const gdn_problem* p, int nseg, const void* q,
                                             const void* k, const void* v, const void* g,
                                             const void* beta, const float* h0, void* o,
                                             float* h_final, unsigned* device_error,
                                             void* stream);

/* ---------------------------------------------------------------------------------------
 * Backward: the state-gradient path (RFC section 6.4.3, reverse flow)
 * ---------------------------------------------------------------------------------------
 * The loss is L = sum_t dO_t . o_t + <dht, h_final>. The gradient on the state runs
 * backwards through the transposed token transitions (exp(g_t) I - beta_t k_t k_t^T, or
 * exp(g_t)(I - beta_t k_t k_t^T) with decay_first; both symmetric), so it needs q, k, g,
 * beta and dO but neither v nor any forward state. The RFC's flow computes it per segment
 * (dS_local), then applies the segment summaries backwards: dH_in = M^T dH_out + dS_local.
 * Per-channel gates (gate_k) are not supported here (GDN_ERR_UNSUPPORTED_SHAPE). */

/* Per-segment state-gradient summary (RFC 6.4.3 "backward_state_gradient_summary").
 *   dS[s] = dL_s/dH_in[s]: the gradient on the state entering segment s of
 *   L_s = sum over the segment's tokens of dO_t . o_t + <dH_end[s], state leaving s>,
 *   computed chunk by chunk backwards (dR = Kd D + C^T dO; D <- exp(G_c) D + Qd^T dO - W^T dR).
 *   Shapes and layouts as the forward: q, k [B,T,H,K] and g, beta [B,T,H] in in_dtype;
 *   dO [B,T,H,V] in out_dtype (the output's dtype); dH_end [nseg,B,H,K,V] fp32 or NULL
 *   (zero: the RFC's dS_local); dS [nseg,B,H,K,V] fp32, written. With nseg == 1 and
 *   dH_end = dht, dS[0] is dh0, the initial-state gradient. T % (64*nseg) == 0, K = V in
 *   {64, 128}; every pointer 16-byte aligned; B*H*nseg*(V/32) < 2^31 (one CTA per 32-column
 *   tile of every segment's state gradient). dS must not overlap any input (dH_end included).
 *   fp32 arithmetic on CUDA cores; no workspace. Asynchronous on `stream`. */
GDN_API gdn_status gdn_state_grad_summary(const gdn_problem* p, int nseg, const void* q,
                                          const void* k, const void* g, const void* beta,
                                          const void* dO, const float* dH_end, float* dS,
                                          void* stream);

/* Reverse scan of the state gradients (RFC 6.4.3 "backward_summary_apply"):
 *   dH_in[nseg] = dht (zeros if NULL),  dH_in[s] = M[s]^T dH_in[s+1] + dS[s]  (s = nseg-1..0).
 *   M [nseg,B,H,K,K] from gdn_segment_summary, dS [nseg,B,H,K,V] from
 *   gdn_state_grad_summary, dht [B,H,K,V], dH_in [nseg,B,H,K,V] out, all fp32. dH_in[s] is
 *   the gradient of L on the state entering segment s; dH_in[0] is dh0, and dH_in[s+1] (dht
 *   for the last segment) is what segment s's own backward starts from. Only p->B, p->H,
 *   p->K, p->V are read from the problem. */
GDN_API gdn_status gdn_state_grad_scan(const gdn_problem* p, int nseg, const float* M,
                                       const float* dS, const float* dht, float* dH_in,
                                       void* stream);

/* The whole backward (RFC 6.4.3, the reverse flow through "backward_state" and
 * "backward_finish"): the gradients of L = sum_t dO_t . o_t + <dht, h_final> with respect to
 * every input, for the problem gdn_segmented_fwd computes.
 *   Steps: the forward once more with one segment per chunk, which yields the state entering
 *   every chunk; then the gradient on the state leaving every chunk, by state-gradient chains
 *   that run backwards over P pieces of each sequence. The library picks P for the GPU: when the
 *   chains of whole sequences (B*H times the column tiles) fit in one wave, P = 1 and one pass
 *   from dht gives every chunk's gradient and dh0; otherwise the pieces' summaries M, their
 *   state gradients dS_local and the reverse scan dH_in = M^T dH_out + dS_local (the pieces
 *   stand in for ranks), then each piece's chunks again from the gradient leaving it. Last,
 *   every chunk's gradients at once, independently, from its inputs, the state entering it
 *   and the gradient leaving it. nseg is validated as for gdn_segmented_fwd; the results do
 *   not depend on it.
 *   Inputs as gdn_segmented_fwd (q, k, v, g, beta in in_dtype, h0 fp32 or NULL); dO
 *   [B,T,H,V] in out_dtype; dht [B,H,K,V] fp32 or NULL (zero).
 *   Outputs, fp32, written: dq, dk [B,T,H,K]; dv [B,T,H,V]; dg, dbeta [B,T,H]; dh0 [B,H,K,V]
 *   (NULL skips it).
 *   With bf16 inputs the products of the state-gradient chains and of the per-chunk gradients
 *   run on the tensor cores with tf32 operands (fp32 accumulation); with fp32 inputs they are
 *   fp32 CUDA-core arithmetic. The forward's recomputation follows gdn_segmented_fwd's paths.
 *   Per-channel gates (gate_k) are not supported (GDN_ERR_UNSUPPORTED_SHAPE). Workspace:
 *   gdn_chunk_bwd_workspace_bytes(p, nseg) (the same for every nseg), whose first 256 bytes
 *   must be zero before the first call (the device error word). */
GDN_API size_t gdn_chunk_bwd_workspace_bytes(const gdn_problem* p, int nseg);
GDN_API gdn_status gdn_chunk_bwd(const gdn_problem* p, int nseg, const void* q, const void* k,
                                 const void* v, const void* g, const void* beta, const float* h0,
                                 const void* dO, const float* dht, float* dq, float* dk,
                                 float* dv, float* dg, float* dbeta, float* dh0, void* workspace,
                                 size_t workspace_bytes, void* stream);

/* gdn_chunk_bwd with stage markers, for timing each step from the caller. If stage_events is
 * non-NULL it points to six cudaEvent_t recorded on `stream` before the forward's
 * recomputation, before the pieces' summaries M, before the first pass of the state-gradient
 * chains (then the reverse scan), before their second pass, before the per-chunk gradients and
 * after them. With one piece the summaries and the second pass are empty stages and the first
 * pass is the only one. None is recorded when T == 0. Same results as gdn_chunk_bwd. */
GDN_API gdn_status gdn_chunk_bwd_timed(const gdn_problem* p, int nseg, const void* q,
                                       const void* k, const void* v, const void* g,
                                       const void* beta, const float* h0, const void* dO,
                                       const float* dht, float* dq, float* dk, float* dv,
                                       float* dg, float* dbeta, float* dh0, void* workspace,
                                       size_t workspace_bytes, void* stream,
                                       void* const* stage_events);

/* ---------------------------------------------------------------------------------------
 * Packed variable-length sequences
 * ---------------------------------------------------------------------------------------
 * nseq sequences of different lengths share one token axis: sequence s holds tokens
 * cu_seqlens[s] .. cu_seqlens[s+1]-1 of q, k, v, g, beta and o, which are laid out as for
 * B = 1 ([1, T, H, *], T = cu_seqlens[nseq] the total). Each sequence runs the recurrence
 * from its own initial state and is cut into chunks of 64 tokens counted from its own first
 * token (its last chunk may be shorter), so no state crosses from one sequence into the
 * next -- "KDA Chunk Backward -- TPU/Pallas Kernel Design", section 3.8 "Fixed Shapes
 * Supporting varlen" (cu_seqlens; every sequence aligned to the chunk size). The tokens stay
 * packed in memory: the alignment is in the chunk numbering, not a padded copy.
 * Supported set: p->B == 1, T >= 0 (any length), nseq >= 1, the K/V/dtype set above;
 * bf16 inputs with K == V == 128 and T >= 64 run the tcgen05 kernels, the rest the CUDA-core
 * kernels. On the tcgen05 path, when every sequence's chains fit the SMs at once, a plan made
 * on the device may cut long sequences into pieces as gdn_segmented_fwd cuts its sequences
 * (RFC section 2.2): piece 0's forward beside the summaries of the middle pieces, their scan,
 * then the forwards of the other pieces, so that a long sequence no longer sets the time
 * alone. The results are those of the uncut recurrence within the bf16 tolerance. */

/* Workspace bytes for gdn_varlen_fwd: the error word, the WY tiles of at most T/64 + nseq
 * chunks per head (tensor-core shapes), two int arrays of nseq + 1 and (tensor-core shapes)
 * the piece plan: its tables and, for at most 256 / H pieces past the first ones, their fp32
 * states and summaries (about 48 MiB at K = V = 128). Depends on T, H, K, V, the dtypes and
 * nseq only, not on the lengths. Returns 0 for an invalid problem. */
GDN_API size_t gdn_varlen_workspace_bytes(const gdn_problem* p, int nseq);

/* Chunked forward of every packed sequence (RFC section 2.1 per sequence).
 *   cu_seqlens  [nseq + 1] int32 DEVICE array: 0 first, T last, non-decreasing (empty
 *               sequences allowed). It is checked on the device: a bad array is recorded in
 *               the workspace's error word as GDN_ERR_INVALID_ARG (gdn_check_device_error)
 *               and the call then treats every sequence as empty (o is not written and
 *               h_final = h0).
 *   h0       [nseq, H, K, V] fp32, or NULL for zero initial states.
 *   o        [1, T, H, V] out_dtype, written.
 *   h_final  [nseq, H, K, V] fp32, the state after each sequence's last token; NULL skips it.
 *   Workspace: gdn_varlen_workspace_bytes(p, nseq). Nothing is read back to the host: the
 *   call can be captured in a CUDA graph. */
GDN_API gdn_status gdn_varlen_fwd(const gdn_problem* p, int nseq, const int* cu_seqlens,
                                  const void* q, const void* k, const void* v, const void* g,
                                  const void* beta, const float* h0, void* o, float* h_final,
                                  void* workspace, size_t workspace_bytes, void* stream);

/* gdn_varlen_fwd with stage markers: if stage_events is non-NULL it points to five
 * cudaEvent_t recorded on `stream` before the length check (which also makes the plan, when a
 * cut is possible) and the WY-factor launch; before the first phase (the whole forward when
 * no sequence is cut); before the scan; before the second phase; and after it. Same results
 * as gdn_varlen_fwd. */
GDN_API gdn_status gdn_varlen_fwd_timed(const gdn_problem* p, int nseq, const int* cu_seqlens,
                                        const void* q, const void* k, const void* v,
                                        const void* g, const void* beta, const float* h0,
                                        void* o, float* h_final, void* workspace,
                                        size_t workspace_bytes, void* stream,
                                        void* const* stage_events);

/* Self-test of the failure path every kernel wait takes: one CTA waits on a barrier that
 * nothing arrives at, with a limit of limit_cycles SM clock cycles (1 .. 2^32), then records
 * GDN_ERR_TIMEOUT (detail word 0x5E) in the workspace's device error word and returns, as a
 * chain kernel does when a wait runs out; the context stays usable. Asynchronous on `stream`:
 * read the result with gdn_check_device_error. workspace: any workspace of the calls above
 * (only its first 8 bytes are touched). Returns GDN_ERR_INVALID_ARG for a limit out of range. */
GDN_API gdn_status gdn_selftest_wait_timeout(void* workspace, long long limit_cycles, void* stream);

/* Static, NUL-terminated description of a status code. */
GDN_API const char* gdn_status_string(gdn_status s);

/* Synchronises `stream`, reads the workspace's device error word, clears it, and returns
 * GDN_OK, GDN_ERR_TIMEOUT (a bounded wait ran out; the results of the affected calls are
 * invalid), GDN_ERR_INVALID_ARG (gdn_varlen_fwd got a bad cu_seqlens) or GDN_ERR_CUDA. If `detail` is non-NULL it receives the recorded detail word
 * (which wait gave up), or 0. */
GDN_API gdn_status gdn_check_device_error(void* workspace, void* stream, unsigned* detail);

#ifdef __cplusplus
}
#endif

#endif /* GDN_H_ */
