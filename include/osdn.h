/*
 * osdn.h -- C ABI of the GB300 (sm_103a) Online Scaled DeltaNet forward pass
 * and its gradients.
 *
 * The method: "OSDN: Improving Delta Rule with Provable Online
 * Preconditioning in Linear Attention" (arXiv 2605.13473), as summarised on
 * the gist.science pages.  Section 2.2 states the forward pass as two phases,
 * and the library has one call per phase:
 *
 *   Phase 1  osdn_precond_scan  -- the O(K) scan over the key stream that
 *            produces the preconditioned keys ktilde_t = d_t (.) k_t and
 *            updates the diagonal preconditioner d (sections 2.1-2.3);
 *   Phase 2  osdn_chunk_fwd     -- the chunkwise delta-rule pass with ktilde
 *            in place of k in the chunk Gram matrix and the intra-chunk scores
 *            (section 2.1), producing o_t = S_t q_t and the final state.
 *
 * Around them: osdn_precond_scan_residual (Phase 1 plus the per-sequence
 * log of the residual ratios, section 3 and section 4.2), osdn_decode_step
 * (both phases at T = 1, in place, for inference), osdn_backward (the
 * gradients of both phases, for training), and osdn_chunk_fwd_kda /
 * osdn_backward_kda (Phase 2 and the gradients with a decay per key channel,
 * the Kimi-Delta-Attention-style backbone of section 4).
 *
 * Conventions shared by every call
 * --------------------------------
 *  - All tensor pointers are DEVICE pointers owned by the caller; the
 *    library allocates no device or host memory and keeps no pointer after a
 *    call returns.  Every tensor is dense, row-major, with the layouts named
 *    below, and must start on a 16-byte boundary.
 *  - Shapes: B, H, T >= 0 (a call with B*H*T == 0 is valid; see each call);
 *    K = d_k and V = d_v must each be 64 or 128.
 *  - Layouts: q, k, ktilde  [B][H][T][K]      v, o        [B][H][T][V]
 *             beta, r, alpha [B][H][T] fp32   d0, dT      [B][H][K] fp32
 *             S0, ST [B][H][V][K] fp32, S[i][j] with i the value row and j
 *             the key column, so that S k is a V-vector.
 *  - io selects the element type of q, k, ktilde, v and o: OSDN_F32 (fp32)
 *    or OSDN_BF16 (bfloat16).  Gates and states are always fp32.
 *  - stream is a cudaStream_t passed as void*; NULL is the legacy default
 *    stream.  Calls are asynchronous: they validate on the host, enqueue
 *    their kernels and return.
 *  - The compute calls may be captured into a CUDA graph on `stream`
 *    (stream capture), after one call of the same kind and shape outside
 *    the capture has set the kernels' attributes and created the library's
 *    streams; the bf16 Phase 2's library streams then join the capture.  The
 *    workspace and every buffer must outlive the graph, and the status word
 *    is read (osdn_check_status) only outside the capture.
 *  - Return value: OSDN_OK, or a negative osdn_status.  Every argument check
 *    happens before anything is enqueued, so a non-zero return means nothing
 *    ran.  OSDN_ERR_CUDA means a launch was rejected by the CUDA runtime.
 *  - Device-side faults never trap: a kernel that detects a problem (a wait
 *    that ran out, an impossible index) writes its code into the status word
 *    at the start of the workspace and exits.  osdn_check_status reads it.
 *  - No C++ exception crosses this boundary and the library never exits or
 *    aborts the process.
 *
 * Workspace
 * ---------
 *  Each call takes a caller-allocated device workspace of at least the size
 *  its *_workspace_bytes function returns.  Its first 256 bytes hold the
 *  device status word and are shared by all calls; the rest is scratch for
 *  the call in flight (calls that use one workspace concurrently on
 *  different streams race on it).  Zero the first 256 bytes once before the
 *  first call (osdn_workspace_init does that on a stream); the status word is
 *  sticky until the caller zeroes it again.  The header's second word is a
 *  test word: while it is nonzero, the bf16 osdn_chunk_fwd's state recurrence
 *  loads nothing and shortens its bounded waits, so that they run out and the
 *  status word reads OSDN_ERR_TIMEOUT -- the way the timeout path is
 *  exercised without a fault.  Keep it zero otherwise.
 */
#ifndef OSDN_H
#define OSDN_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { OSDN_F32 = 0, OSDN_BF16 = 1 } osdn_dtype;

typedef enum {
    OSDN_OK = 0,
    OSDN_ERR_NULL = -1,      /* a required pointer is NULL                     */
    OSDN_ERR_DIMS = -2,      /* negative size, B*H > 2^24, or K / V not in {64, 128} */
    OSDN_ERR_DTYPE = -3,     /* io is not OSDN_F32 / OSDN_BF16                 */
    OSDN_ERR_ALIGN = -4,     /* a pointer is not 16-byte aligned               */
    OSDN_ERR_WORKSPACE = -5, /* workspace NULL or smaller than required        */
    OSDN_ERR_CUDA = -6,      /* the CUDA runtime rejected a launch or query    */
    OSDN_ERR_TIMEOUT = -7,   /* device: a bounded wait ran out (status word)   */
    OSDN_ERR_DEVICE = -8,    /* device: an input checked on the device is invalid
                                (osdn_chunk_fwd, bf16: a decay alpha that is not
                                positive and finite, or a beta that is not finite) */
    OSDN_ERR_ALIAS = -9,     /* an output overlaps an input it must not alias  */
    OSDN_ERR_ARCH = -10,     /* the current device is not sm_103 (GB300)       */
    OSDN_ERR_SCRATCH = -11   /* osdn_precond_scan_noalloc: shape needs more
                                scratch than its static buffer holds         */
} osdn_status;

/* Bytes of workspace osdn_precond_scan needs for this shape (>= 256). */
size_t osdn_precond_scan_workspace_bytes(int B, int H, int T, int K);

/*
 * Phase 1: the preconditioner scan (sections 2.2 and 2.3).
 *
 * For each sequence (b,h), starting from d_0 (d0, or all ones if d0 is NULL),
 * for t = 0 .. T-1:
 *     ktilde_t = d_t (.) k_t
 *     d_{t+1}  = r_t d_t + eta beta_t (1 - beta_t <d_t, k_t^2>) k_t^2 / ||k_t||^2
 * which is d_{t+1} = r_t d_t - eta grad_d h_t(d_t) for the closed-form
 * surrogate h_t(d) = ((1 - beta_t <d, k_t^2>)^2 - 1) / (2 ||k_t||^2)
 * (section 2.2), taken as a DESCENT step (section 2.3 prints "+eta grad h";
 * section 2.2 calls the update online gradient descent on h).  A zero key
 * contributes no gradient.  r is the adaptive-preconditioner-forgetting
 * retention gate (section 2.3); r == NULL means r = 1 (plain OSDN).
 *
 *   k      in   [B][H][T][K] io
 *   beta   in   [B][H][T] fp32
 *   r      in   [B][H][T] fp32, or NULL
 *   eta    in   scalar step size of the preconditioner update
 *   d0     in   [B][H][K] fp32, or NULL (all ones)
 *   ktilde out  [B][H][T][K] io; must not overlap k
 *   dT     out  [B][H][K] fp32, or NULL (not written)
 * With T == 0 the call writes dT = d0 and nothing else.
 */
int osdn_precond_scan(int io, int B, int H, int T, int K, const void *k, const float *beta,
                      const float *r, float eta, const float *d0, void *ktilde, float *dT,
                      void *workspace, size_t workspace_bytes, void *stream);

/*
 * Phase 1 with the residual diagnostic.  Computes exactly what
 * osdn_precond_scan computes and, per sequence,
 *
 *     log_ratio[b][h] = sum_t log((1 - beta_t <d_t, k_t^2>)^2)
 *
 * the log of the product of the token-local residual ratios
 * f_t(S_t) / f_t(S_{t-1}) with f_t(S) = 1/2 ||S k_t - v_t||^2 (gist.science
 * summary of arXiv 2605.13473, section 3, theorem 5.2): writing
 * ktilde_t = d_t (.) k_t into the state scales the token's residual by
 * 1 - beta_t <ktilde_t, k_t>.  exp(log_ratio / T) is the geometric-mean
 * residual ratio q_geo of section 4.2.  With a decay alpha in Phase 2 the
 * ratio is taken against the decayed state alpha_t S_{t-1}.  A token whose
 * factor is exactly zero makes the sum -inf; T == 0 gives 0.
 *
 *   log_ratio out [B][H] fp32, 16-byte aligned, must not overlap the other
 *             arguments; the rest as for osdn_precond_scan (same workspace
 *             size).  NULL log_ratio: OSDN_ERR_NULL.
 */
int osdn_precond_scan_residual(int io, int B, int H, int T, int K, const void *k,
                               const float *beta, const float *r, float eta, const float *d0,
                               void *ktilde, float *dT, float *log_ratio, void *workspace,
                               size_t workspace_bytes, void *stream);

/*
 * Phase 1 without a workspace, for callers that cannot allocate device
 * memory: code running where cudaMalloc is off limits (inside a region being
 * captured under a memory pool that forbids new allocations, a plugin whose
 * host owns every allocation, or a caller that must never fail with
 * out-of-memory after start-up).  The paper has no counterpart to this call;
 * it computes exactly what osdn_precond_scan computes, with the same
 * arguments minus the workspace.
 *
 * Scratch: a file-scope device array of 2 MiB, present on every GPU that
 * loads the library until the process exits.  The first call on a device
 * resolves the array's device address there (cudaGetSymbolAddress), so that
 * first call should be made before any stream capture.  The call allocates
 * nothing: no cudaMalloc, no cudaFree, no allocating library routine.
 * Shapes whose speculative segments need more than 2 MiB of scratch (about
 * B*H*ceil(T/L)*8*K bytes, L the segment length of 256 to 1024 tokens, and
 * none without a retention gate) return OSDN_ERR_SCRATCH before anything is
 * enqueued.  All calls share the array and it keeps the last call's
 * contents: calls whose kernels may overlap on the GPU (unordered streams)
 * race on it and must be serialised by the caller.  Kernels of this call
 * report no device status word.
 */
int osdn_precond_scan_noalloc(int io, int B, int H, int T, int K, const void *k,
                              const float *beta, const float *r, float eta, const float *d0,
                              void *ktilde, float *dT, void *stream);

/*
 * Bytes of workspace osdn_chunk_fwd needs for this shape (>= 256).  With
 * io == OSDN_BF16 the call prepares every chunk's operands before it runs the
 * state recurrence and keeps them in the workspace: about
 * B*H*ceil(T/64) * (2K^2 + 256K + 8196) bytes (72 KB a chunk at K = 128),
 * plus 8*B*H*V*K bytes for the state carried between slabs of chunks.
 */
size_t osdn_chunk_fwd_workspace_bytes(int io, int B, int H, int T, int K, int V);

/*
 * Phase 2: the chunkwise delta-rule pass with preconditioned keys
 * (section 2.1; section 2.2, item 2).
 *
 * For each sequence (b,h), starting from S_0 (S0, or zeros if S0 is NULL),
 * for t = 0 .. T-1:
 *     S_t = alpha_t S_{t-1} + beta_t (v_t - alpha_t S_{t-1} k_t) ktilde_t^T
 *     o_t = S_t q_t
 * alpha == NULL means alpha = 1, the update S_t = S_{t-1} + beta_t (v_t -
 * S_{t-1} k_t) ktilde_t^T of section 2.1.  A non-NULL alpha is a per-token
 * state decay in the style of the Gated DeltaNet backbone named in section 4
 * (the pages print no formula for it; this is the plainest reading).  The
 * output is read from the state after token t and q is not scaled.
 *
 * The kernels evaluate this chunk by chunk: with the keys of a chunk in the
 * rows of K, Ktilde, Q and the scaled residuals in U,
 *     (I + tril(diag(beta) (Gamma . K Ktilde^T), -1)) U
 *                                  = diag(beta) (V - diag(gamma) K S_0^T),
 *     O = diag(gamma) Q S_0^T + tril(Gamma . Q Ktilde^T) U,
 *     S = gamma_C S_0 + U^T diag(gamma_C / gamma) Ktilde,
 * gamma the within-chunk cumulative product of alpha and Gamma_ij =
 * gamma_i / gamma_j -- the stored keys replaced by Ktilde in the Gram matrix
 * and the intra-chunk scores exactly as section 2.1 says.
 *
 *   q, k, ktilde in [B][H][T][K] io
 *   v            in [B][H][T][V] io
 *   beta         in [B][H][T] fp32
 *   alpha        in [B][H][T] fp32, or NULL
 *   S0           in [B][H][V][K] fp32, or NULL (zeros)
 *   o            out [B][H][T][V] io; must not overlap any input
 *   ST           out [B][H][V][K] fp32, or NULL (not written)
 * io == OSDN_BF16 runs on the tensor cores (bf16 operands, fp32
 * accumulation, state carried in fp32); io == OSDN_F32 runs in fp32 FFMA.
 * For sequences longer than 64 chunks of 64 tokens (or of 32 to 64 chunks
 * when the state recurrence leaves at least half the SMs free) the bf16
 * path overlaps the preparation of later chunks with the state recurrence of
 * earlier ones on two library-owned streams per device (created on first
 * use, forked from and joined back to `stream` with events); the library
 * serialises the enqueue of such calls.  With a decay alpha and few
 * sequences the recurrence instead runs in speculative time segments: each
 * segment starts from a zero state four chunks early, and a segment whose
 * start differs from its predecessor's end by more than 2^-16 of that end's
 * largest entry (per block of 64 value rows) is recomputed from that end, so
 * the speculation changes the result by no more than that bound.
 * With T == 0 the call writes ST = S0 and nothing else.  With io ==
 * OSDN_BF16, T may be at most 1,073,741,760 (the chunk rows of the prepared
 * operands are addressed with 32-bit TMA coordinates); a longer sequence
 * returns OSDN_ERR_DIMS (split it and chain the state through S0 / ST).
 * Test hook: while the workspace header's test word is nonzero, the bf16
 * path's state-recurrence kernel loads nothing, so its bounded waits run out
 * (after limits shortened to milliseconds) and the call leaves
 * OSDN_ERR_TIMEOUT in the status word with o and ST unwritten; the device
 * stays usable.  It exists to test the timeout path.
 */
int osdn_chunk_fwd(int io, int B, int H, int T, int K, int V, const void *q, const void *k,
                   const void *ktilde, const void *v, const float *beta, const float *alpha,
                   const float *S0, void *o, float *ST, void *workspace, size_t workspace_bytes,
                   void *stream);

/*
 * Bytes of workspace osdn_forward needs for this shape (>= 256).  bf16: the
 * preconditioner scan's segment scratch, the scan's checkpoints (4 B*H*T for
 * e_t and 4 B*H*ceil(T/64)*K for d at every 64th token) and the tensor-core
 * Phase 2 workspace of osdn_chunk_fwd, each rounded up to 256 bytes.  fp32:
 * the scan's scratch and ktilde (4 B*H*T*K).
 */
size_t osdn_forward_workspace_bytes(int io, int B, int H, int T, int K, int V);

/*
 * Both phases in one call, with the preconditioned keys kept off global
 * memory (section 2.2: the two phases; the preconditioner scan's cost is the
 * throughput overhead section 4.3 reports).  The results are those of
 * osdn_precond_scan followed by osdn_chunk_fwd on the same inputs, except
 * that ktilde is not returned:
 *   q, k    in [B][H][T][K] io          v   in [B][H][T][V] io
 *   beta    in [B][H][T] fp32;  r, alpha in [B][H][T] fp32 or NULL (1)
 *   eta     the step size;  d0 in [B][H][K] fp32 or NULL (ones)
 *   S0      in [B][H][V][K] fp32 or NULL (zeros)
 *   o       out [B][H][T][V] io;  dT out [B][H][K] fp32 or NULL;
 *   ST      out [B][H][V][K] fp32 or NULL
 * io == OSDN_BF16: the scan writes, instead of ktilde, its coefficient e_t
 * (d_{t+1} = r_t d_t + e_t k_t^2) for every token and d at every 64-token
 * boundary -- 12 bytes a token-head at K = 128 where ktilde takes 256 -- and
 * Phase 2's chunk preparation rebuilds each chunk's ktilde in shared memory
 * from them (rho d_c + P W, one small tensor-core product).  The rebuilt
 * preconditioner differs from the scan's own by about 2^-16 relative, well
 * inside the rounding of bf16 ktilde, so o and S_T agree with the two-call
 * path to within the bf16 tolerance, not bit for bit.
 * io == OSDN_F32: the two phases run as osdn_precond_scan + osdn_chunk_fwd,
 * with ktilde held in the workspace.
 * Outputs must not overlap inputs, each other or the workspace
 * (OSDN_ERR_ALIAS).  The limits, the status word and the errors are those
 * of the two calls.
 */
int osdn_forward(int io, int B, int H, int T, int K, int V, const void *q, const void *k,
                 const void *v, const float *beta, const float *r, float eta, const float *d0,
                 const float *alpha, const float *S0, void *o, float *dT, float *ST,
                 void *workspace, size_t workspace_bytes, void *stream);

/*
 * One recurrent step (T = 1) of both phases, in place: the inference form of
 * the method (section 1: constant-memory recurrent inference; section 2.2
 * for the preconditioner step, section 2.1 for the state update).  For every
 * sequence (b,h), with w = k (.) k and n = ||k||^2:
 *     ktilde = d (.) k                               (d before the step)
 *     d     <- r d + eta beta (1 - beta <d, w>) w / n   (r = 1 if r == NULL;
 *                                                       the step is 0 if n = 0)
 *     S     <- alpha S + beta (v - alpha S k) ktilde^T  (alpha = 1 if NULL)
 *     o      = S q                                   (the updated state)
 * The same arithmetic as osdn_precond_scan + osdn_chunk_fwd with T = 1.
 *
 *   q, k    in [B][H][K] io          v   in [B][H][V] io
 *   beta    in [B][H] fp32;  r, alpha in [B][H] fp32 or NULL
 *   d       in/out [B][H][K] fp32    S   in/out [B][H][V][K] fp32
 *   o       out [B][H][V] io;  ktilde out [B][H][K] io, or NULL
 * The workspace only carries the status word (>= 256 bytes).  Outputs must
 * not overlap inputs or each other (OSDN_ERR_ALIAS).
 */
int osdn_decode_step(int io, int B, int H, int K, int V, const void *q, const void *k,
                     const void *v, const float *beta, const float *r, float eta,
                     const float *alpha, float *d, float *S, void *o, void *ktilde,
                     void *workspace, size_t workspace_bytes, void *stream);

/*
 * Bytes of workspace osdn_backward needs for this shape (>= 256): the state
 * of each value row every 16 tokens (4 B*H*ceil(T/16)*V*K), one partial of
 * the row-summed gradients per block of 8 value rows for one window of up to
 * 1024 tokens (4 B*H*(V/8)*min(T,1024)*(3K+2); the reverse sweep runs window
 * by window), the state gradient carried between windows (4 B*H*V*K),
 * 4 B*H*(T*(2K+1) + ceil(T/16)*K) for Phase 1's inputs and checkpoints, the
 * forward scan's segment scratch (as for osdn_precond_scan), and per time
 * segment of the Phase 1 adjoint 8K + 8 bytes, each rounded up to 256 bytes.
 */
size_t osdn_backward_workspace_bytes(int B, int H, int T, int K, int V);

/*
 * Gradients of the forward pass through both phases (the derivative of the
 * recurrences of osdn_precond_scan and osdn_chunk_fwd: sections 2.1, 2.2 and
 * 2.3), for training.  Given the forward's inputs, the ktilde it produced and
 * the cotangents of its outputs, the call returns the gradient of
 *     L = <o, d_o> + <S_T, d_ST> + <d_T, d_dT> + <ktilde, d_ktilde>
 * with respect to every input.  Cotangents given as NULL count as zero.
 *
 * Inputs (the forward's, with its defaults for NULL):
 *   q, k, ktilde in [B][H][T][K] io  (ktilde as osdn_precond_scan wrote it)
 *   v            in [B][H][T][V] io
 *   beta         in [B][H][T] fp32;  r, alpha in [B][H][T] fp32 or NULL (1)
 *   eta          the step size;  d0 in [B][H][K] fp32 or NULL (ones)
 *   S0           in [B][H][V][K] fp32 or NULL (zeros)
 *   d_o          in [B][H][T][V] io or NULL;   d_ST in [B][H][V][K] fp32 or NULL
 *   d_dT         in [B][H][K] fp32 or NULL;    d_ktilde in [B][H][T][K] io or NULL
 * Outputs:
 *   dq, dk       out [B][H][T][K] io;   dv out [B][H][T][V] io
 *   dbeta        out [B][H][T] fp32
 *   dr, dalpha   out [B][H][T] fp32, or NULL (not written)
 *   dd0          out [B][H][K] fp32, or NULL;  dS0 out [B][H][V][K] fp32, or NULL
 *   deta         out [B][H] fp32, or NULL: each sequence's share of dL/deta
 *                (the gradient of the shared scalar eta is their sum)
 * The arithmetic is fp32 for both I/O types (bf16 inputs are widened, bf16
 * outputs rounded once at the end).  The pass runs token by token in
 * reverse time: Phase 2's state gradient one value row per warp, with the
 * forward states recomputed 16 tokens at a time from checkpoints; then the
 * Phase 1 adjoint one sequence per warp.  The results are deterministic
 * (row sums in a fixed order, no atomics).  Outputs must not overlap inputs
 * or each other (OSDN_ERR_ALIAS).  With T == 0 the call writes dS0 = d_ST,
 * dd0 = d_dT (zeros for NULL) and deta = 0.
 */
int osdn_backward(int io, int B, int H, int T, int K, int V, const void *q, const void *k,
                  const void *ktilde, const void *v, const float *beta, const float *r,
                  float eta, const float *d0, const float *alpha, const float *S0,
                  const void *d_o, const float *d_ST, const float *d_dT, const void *d_ktilde,
                  void *dq, void *dk, void *dv, float *dbeta, float *dr, float *dalpha,
                  float *dd0, float *dS0, float *deta, void *workspace, size_t workspace_bytes,
                  void *stream);

/*
 * Phase 2 with a decay per key channel: the Kimi Delta Attention backbone
 * named in section 4 (no formula printed there), read as GDN's scalar gate
 * made a K-vector that scales the key columns of the state:
 *     S_t = S_{t-1} Diag(alpha_t) + beta_t (v_t - S_{t-1} Diag(alpha_t) k_t) ktilde_t^T
 *     o_t = S_t q_t
 * Phase 1 (osdn_precond_scan) is unchanged and produces ktilde.
 *
 *   q, k, ktilde in [B][H][T][K] io;  v in [B][H][T][V] io
 *   beta         in [B][H][T] fp32
 *   alpha_k      in [B][H][T][K] fp32, or NULL (no decay)
 *   S0           in [B][H][V][K] fp32, or NULL (zeros)
 *   o            out [B][H][T][V] io;  ST out [B][H][V][K] fp32, or NULL
 * io == OSDN_BF16 runs on the tensor cores, like osdn_chunk_fwd: with
 * Gam the within-chunk product of alpha per channel, the chunk Gram and
 * scores take (Gam . k) . (ktilde / Gam), evaluated against a reference
 * point per 16-token block so that no factor leaves the fp32 range; the
 * state rows decay by their own channel's product.  There every entry of
 * alpha_k must lie in [2^-6, 2^6]; one outside it (or not finite) is
 * recorded as OSDN_ERR_DEVICE in the status word and the outputs are then
 * undefined.  The workspace holds the prepared operands of every chunk and
 * each chunk's per-channel decay product (osdn_chunk_fwd_kda_workspace_bytes);
 * T is limited as for osdn_chunk_fwd.  io == OSDN_F32 runs the token
 * recurrence in fp32 FFMA, one CTA per 32 value rows, with any decay, and
 * needs only the 256-byte status header.  With T == 0 the call writes
 * ST = S0.  Outputs must not overlap inputs (OSDN_ERR_ALIAS).
 */
size_t osdn_chunk_fwd_kda_workspace_bytes(int io, int B, int H, int T, int K, int V);
int osdn_chunk_fwd_kda(int io, int B, int H, int T, int K, int V, const void *q, const void *k,
                       const void *ktilde, const void *v, const float *beta,
                       const float *alpha_k, const float *S0, void *o, float *ST,
                       void *workspace, size_t workspace_bytes, void *stream);

/*
 * osdn_backward for the per-channel decay of osdn_chunk_fwd_kda: the same
 * arguments and outputs, with alpha_k [B][H][T][K] fp32 (or NULL) in place
 * of alpha and dalpha_k [B][H][T][K] fp32 (or NULL) in place of dalpha.
 * Its workspace holds K + 1 rather than 2 values of dalpha and dbeta per
 * token in each row-block partial: 4 B*H*(V/8)*min(T,1024)*(4K+1) bytes
 * instead of 4 B*H*(V/8)*min(T,1024)*(3K+2), the rest as
 * osdn_backward_workspace_bytes.
 */
size_t osdn_backward_kda_workspace_bytes(int B, int H, int T, int K, int V);
int osdn_backward_kda(int io, int B, int H, int T, int K, int V, const void *q, const void *k,
                      const void *ktilde, const void *v, const float *beta, const float *r,
                      float eta, const float *d0, const float *alpha_k, const float *S0,
                      const void *d_o, const float *d_ST, const float *d_dT,
                      const void *d_ktilde, void *dq, void *dk, void *dv, float *dbeta,
                      float *dr, float *dalpha_k, float *dd0, float *dS0, float *deta,
                      void *workspace, size_t workspace_bytes, void *stream);

/*
 * osdn_decode_step with a decay per key channel (the recurrent step of
 * osdn_chunk_fwd_kda): alpha_k in [B][H][K] fp32, or NULL, in place of
 * alpha; the state row is decayed column by column,
 *     S <- S Diag(alpha) + beta (v - S Diag(alpha) k) ktilde^T,   o = S q.
 * Everything else as osdn_decode_step.
 */
int osdn_decode_step_kda(int io, int B, int H, int K, int V, const void *q, const void *k,
                         const void *v, const float *beta, const float *r, float eta,
                         const float *alpha_k, float *d, float *S, void *o, void *ktilde,
                         void *workspace, size_t workspace_bytes, void *stream);

/* Zero the 256-byte status area at the start of a workspace (async). */
int osdn_workspace_init(void *workspace, size_t workspace_bytes, void *stream);

/*
 * Synchronise `stream`, read the device status word of `workspace` and
 * return it (OSDN_OK if no kernel reported a problem).  Returns
 * OSDN_ERR_CUDA if the stream itself reports an error.
 */
int osdn_check_status(const void *workspace, void *stream);

/* A static, human-readable name for a status code. */
const char *osdn_status_string(int code);

/* Library version as MAJOR*10000 + MINOR*100 + PATCH. */
int osdn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* OSDN_H */
