/*
 * mdn.h — C ABI of the Momentum DeltaNet (MDN) memory-update library for
 * NVIDIA GB300 (sm_103a).
 *
 * The method: "MDN: Parallelizing Stepwise Momentum for Delta Linear
 * Attention" (arXiv 2605.05838).  Per head, two states S, M in R^{dk x dv}
 * (memory and momentum) and four scalar gates per token (alpha retention,
 * mu momentum retention, beta step, eta gradient scale) evolve as
 *
 *     vres_t = v_t - alpha_t S_{t-1}^T k_t
 *     M_t    = mu_t M_{t-1} - eta_t k_t vres_t^T
 *     S_t    = alpha_t S_{t-1} - beta_t M_t
 *     o_t    = S_t^T q_t
 *
 * (paper-reading slides, frame "MDN adds a momentum matrix to the delta
 * update", Eqs. (3)-(5); reading notes section 2.2).
 *
 * General conventions
 *  - Every pointer argument except cu_seqlens' host use is a DEVICE pointer
 *    to memory the caller owns; the library keeps no pointer after a call
 *    returns and allocates no device memory.
 *  - All device work is enqueued on `stream` (a cudaStream_t; NULL means the
 *    legacy default stream) and runs asynchronously; a call returns as soon as
 *    its kernels are enqueued.
 *  - The enqueueing calls (mdn_chunk_fwd and its variants, mdn_decode_step,
 *    mdn_prepare_inputs) may be captured into a CUDA graph once one call has
 *    run on the device (the first call looks up the device's status word with
 *    cudaGetSymbolAddress); a replay reads the pointers given at capture.
 *    mdn_get_device_status synchronises and must not be captured.
 *  - Gates and states are fp32.  q, k, v, o share one element type `dtype`.
 *    Accumulation is fp32.  Inputs are never modified (except the in-place
 *    states of mdn_decode_step).
 *  - Tensors are dense, row-major, innermost dimension last; no strides.
 *  - Preconditions documented, not checked on the device: alpha in (0, 1],
 *    mu in [0, 1], beta >= 0, eta >= 0, all finite.  mu = 0 is supported.
 *  - Errors: a call validates its arguments before enqueuing anything and
 *    returns MDN_ERR_INVALID_ARG (null required pointer, non-positive or
 *    inconsistent size, pointer not 16-byte aligned, workspace too small),
 *    MDN_ERR_UNSUPPORTED (dk != dv, dk not in {64, 128}, chunk != 64, device
 *    is not compute capability 10.3) or MDN_ERR_CUDA (a CUDA call or launch
 *    failed; cudaGetLastError() is cleared).  On any error nothing was
 *    enqueued except for MDN_ERR_CUDA, where earlier launches of the same call
 *    may have been.  Device-side bounded waits that expire set
 *    MDN_ERR_DEVICE_TIMEOUT in a device status word read by
 *    mdn_get_device_status; the kernel then returns without hanging.
 */
#ifndef MDN_H_
#define MDN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MDN_ABI_VERSION 2

typedef enum mdn_status {
    MDN_OK = 0,
    MDN_ERR_INVALID_ARG = 1,
    MDN_ERR_UNSUPPORTED = 2,
    MDN_ERR_CUDA = 3,
    MDN_ERR_DEVICE_TIMEOUT = 4
} mdn_status;

typedef enum mdn_dtype {
    MDN_F32 = 0,   /* IEEE binary32 */
    MDN_BF16 = 1   /* bfloat16 */
} mdn_dtype;

/* Returns MDN_ABI_VERSION of the built library. */
int mdn_abi_version(void);

/* Static, NUL-terminated description of a status code (never NULL). */
const char *mdn_status_string(mdn_status status);

/*
 * Bytes of device workspace mdn_chunk_fwd needs for these sizes (a multiple
 * of 256; 0 for invalid sizes).  The bound covers every split of T_total into
 * n_seq sequences, so it does not need cu_seqlens.
 */
size_t mdn_chunk_fwd_workspace_size(int n_seq, int T_total, int H, int dk,
                                    int dv, mdn_dtype dtype);

/*
 * mdn_chunk_fwd — prefill: run the recurrence above over whole sequences in
 * the exact chunkwise-parallel form.
 *
 * Defined by: slides, frames "Reorder the triangular sum to isolate scalar
 * coefficients" (Eqs. (7)-(9), Appendix C Eqs. (30)-(31)), "Solve the unknown
 * residuals with a lower triangular system" (Eqs. (15)-(18)), "Chunk outputs
 * combine incoming states and local writes" (Appendix C Eqs. (40)-(42)) and
 * the backup frames on the row shift and on the log-domain coefficients
 * (Algorithm 1); reading notes sections 2.3-2.6.  In exact arithmetic the
 * result equals the token recurrence; chunks hold 64 tokens and each sequence
 * is chunked from its own start (a shorter last chunk uses its own length).
 *
 * Layout.  Without cu_seqlens: B sequences of T tokens each, n_seq == B,
 *   q, k [B, T, H, dk];  v, o [B, T, H, dv];  alpha, mu, eta, beta [B, T, H].
 * With cu_seqlens (device int32 [n_seq + 1], cu_seqlens[0] = 0, non-
 *   decreasing, cu_seqlens[n_seq] == T): B must be 1 and the n_seq sequences
 *   are packed along T; sequence s owns tokens [cu_seqlens[s],
 *   cu_seqlens[s+1]).  Empty sequences are allowed (their final states equal
 *   their initial states).  cu_seqlens lives on the device, so it is checked
 *   there: an array that breaks one of the three conditions makes the call
 *   write MDN_ERR_INVALID_ARG into the device status word (see
 *   mdn_get_device_status) and treat every sequence as empty (o is then not
 *   written; S_T, M_T receive the initial states).  With T == 0 every
 *   sequence is empty and cu_seqlens is not read.
 * States S0, M0, S_T, M_T: [n_seq, H, dk, dv] fp32.
 *
 * Arguments
 *   q, k, v        inputs (dtype)
 *   alpha, mu, eta gates (fp32), required when B * T > 0
 *   beta           step gate (fp32) or NULL for beta = 1
 *   S0, M0         initial states or NULL for zero (each independently)
 *   o              output (dtype), written for every token
 *   S_T, M_T       final states, or NULL to skip writing that state.  S_T may
 *                  alias S0 and M_T may alias M0 (same pointer, not partial
 *                  overlap); no other output may overlap an input.  Long
 *                  equal-length bf16 sequences with both given run in time
 *                  segments that hand their states on through S_T, M_T
 *                  (the next segment's preparation overlapping the current
 *                  segment's state pass); the results are the same bits.
 *   workspace      device scratch of at least workspace_bytes >=
 *                  mdn_chunk_fwd_workspace_size(...), 256-byte aligned; its
 *                  contents on entry do not matter and are undefined on exit.
 *                  Two calls in flight at once need separate workspaces.
 *   chunk          must be 64
 *   stream         cudaStream_t (as void*) the work is enqueued on
 */
mdn_status mdn_chunk_fwd(const void *q, const void *k, const void *v,
                         const float *alpha, const float *mu, const float *eta,
                         const float *beta, const float *S0, const float *M0,
                         void *o, float *S_T, float *M_T,
                         const int32_t *cu_seqlens, int n_seq, int B, int T,
                         int H, int dk, int dv, mdn_dtype dtype, int chunk,
                         void *workspace, size_t workspace_bytes, void *stream);

/*
 * mdn_chunk_fwd_vres — mdn_chunk_fwd that also writes every token's residual
 *   vres_t = v_t - S_{t-1}^T (alpha_t k_t)
 * (the corrected values of Eq. (3)), which the slides' frame "Backward
 * computation" (Sec. 3.1, Algorithm 1) has the forward save so that a
 * gradient pass can rebuild the states without storing every (S, M) pair;
 * reading notes section 2.6 ends with the same trade.
 *
 * Arguments as mdn_chunk_fwd, plus
 *   vres   output laid out like v ([B, T, H, dv], or packed), in dtype,
 *          16-byte aligned; required when B * T > 0; must not be q, k, v or o.
 * Errors: as mdn_chunk_fwd; MDN_ERR_INVALID_ARG for a missing or aliasing
 * vres.  o, S_T and M_T are the same values mdn_chunk_fwd writes.
 */
mdn_status mdn_chunk_fwd_vres(const void *q, const void *k, const void *v,
                              const float *alpha, const float *mu, const float *eta,
                              const float *beta, const float *S0, const float *M0,
                              void *o, float *S_T, float *M_T, void *vres,
                              const int32_t *cu_seqlens, int n_seq, int B, int T,
                              int H, int dk, int dv, mdn_dtype dtype, int chunk,
                              void *workspace, size_t workspace_bytes, void *stream);

/*
 * mdn_chunk_state_slots — how many chunk slots the entry-state outputs of
 * mdn_chunk_fwd_states must hold: B * ceil(T / 64) for equal-length batches
 * (packed == 0, n_seq == B), floor(T_total / 64) + n_seq for packed
 * sequences (packed != 0, T_total = B * T; an upper bound of
 * sum_s ceil(L_s / 64)).  Returns 0 for negative sizes.
 */
size_t mdn_chunk_state_slots(int n_seq, int B, int T, int packed);

/*
 * mdn_chunk_fwd_states — mdn_chunk_fwd that also writes the entry states of
 * every chunk: for chunk c of sequence s (its tokens 64 c .. 64 c + 63, the
 * last chunk possibly shorter), the states after the sequence's first 64 c
 * tokens, S_{64c} and M_{64c} (for c = 0 the initial states).  These are
 * the chunk-boundary states the chunk carry of the slides' frame "Chunk
 * outputs combine incoming states and local writes" (Eqs. (17)-(18)) passes
 * on; a gradient pass can start every chunk from them instead of replaying
 * the sequence.
 *
 * Arguments as mdn_chunk_fwd, plus
 *   S_chunks, M_chunks  outputs [slots, H, dk, dv] (row-major) in the
 *          input precision: bf16 for bf16 inputs (the gradient pass uses
 *          them as bf16 tensor-core operands, so nothing it reads is
 *          lost), fp32 for fp32 inputs.  slots at least
 *          mdn_chunk_state_slots(...), both required when B * T > 0,
 *          16-byte aligned, overlapping no other argument.  Chunk c of
 *          sequence s sits at slot s * ceil(T / 64) + c (equal lengths) or
 *          off_s + c with off_s = sum_{s' < s} ceil(L_{s'} / 64) (packed);
 *          other slots are not written.
 * Memory: 2 * dk * dv * (2 or 4) bytes per (chunk, head): 64 KiB at d = 128
 * for bf16 inputs, i.e. 1 KiB per (token, head) against 768 B for that
 * token's q, k and v.
 * Errors: as mdn_chunk_fwd; MDN_ERR_INVALID_ARG for a missing, misaligned
 * or aliasing state output.  o, S_T and M_T are the values mdn_chunk_fwd
 * writes.
 */
mdn_status mdn_chunk_fwd_states(const void *q, const void *k, const void *v,
                                const float *alpha, const float *mu, const float *eta,
                                const float *beta, const float *S0, const float *M0,
                                void *o, float *S_T, float *M_T, void *S_chunks,
                                void *M_chunks, const int32_t *cu_seqlens, int n_seq,
                                int B, int T, int H, int dk, int dv, mdn_dtype dtype,
                                int chunk, void *workspace, size_t workspace_bytes,
                                void *stream);

/*
 * Bytes of device workspace mdn_chunk_bwd needs (a multiple of 256; 0 for
 * invalid sizes): per (chunk slot, head) the chunk's matrices and vectors
 * (84 KB), the state adjoints at the chunk's end (2 dk dv fp32) and the
 * residual adjoints (64 dv fp32); the slot bound is mdn_chunk_state_slots'.
 */
size_t mdn_chunk_bwd_workspace_size(int n_seq, int T_total, int H, int dk,
                                    int dv, mdn_dtype dtype);

/*
 * mdn_chunk_bwd — gradient of the chunk forward: given the adjoints of its
 * outputs (dout for o, dS_T and dM_T for the final states), the gradients
 * with respect to every input, q, k, v, the four gates and the initial
 * states.
 *
 * Defined by: the pages give the training storage policy, not gradient
 * formulas: the forward keeps what the backward needs so that states need
 * not be stored per token (slides, frame "The implementation trades saved
 * residuals for throughput" and its "Backward computation" block; reading
 * notes, end of section 2.6).  Here the saved data are the entry states of
 * every chunk (mdn_chunk_fwd_states), and the result is the exact
 * vector-Jacobian product of the chunk equations (frames "Solve the unknown
 * residuals with a lower triangular system", Eqs. (15)-(18), and "Chunk
 * outputs combine incoming states and local writes", Appendix C Eqs.
 * (40)-(42)): a reverse pass over the chunks carries the state adjoints,
 * then every chunk forms its input gradients in parallel.  The gates'
 * gradients go through the chunk coefficients without dividing by a gate,
 * so mu = 0 is exact.  bf16 inputs: the reverse pass and the per-chunk
 * products on the tensor cores (bf16 operands, fp32 accumulation; T and
 * A_O T from the forward's own prep), the gate gradients in fp32 on the
 * CUDA cores; relative errors a few 1e-3.  fp32 inputs: every step in fp32
 * on the CUDA cores (relative errors near 1e-6).
 *
 * Layout and sizes as mdn_chunk_fwd (equal lengths, or packed with
 * cu_seqlens; the same device checks of cu_seqlens apply).
 * Arguments
 *   q, k, v, alpha, mu, eta, beta   the forward's inputs (beta NULL: 1)
 *   S_chunks, M_chunks   the forward's chunk entry states, exactly as
 *                  mdn_chunk_fwd_states wrote them for these inputs and
 *                  initial states ([slots, H, dk, dv], bf16 or fp32 as
 *                  the inputs)
 *   fwd_workspace  NULL, or (bf16 inputs) the workspace that
 *                  mdn_chunk_fwd_states used for these inputs, unchanged
 *                  since that call: the gradient then takes the matrices T
 *                  and A_O T from the chunk blocks the forward left there
 *                  instead of recomputing them (its prep kernel is skipped;
 *                  the results are the same bits).  Read only; 256-byte
 *                  aligned.  Ignored for fp32 inputs.
 *   dout           adjoint of o (dtype, laid out like o); required
 *   dS_T, dM_T     adjoints of the final states (fp32 [n_seq, H, dk, dv]) or
 *                  NULL for zero
 *   dq, dk, dv     gradients (dtype, laid out like q, k, v); required
 *   dalpha, dmu, deta   gradients of the gates (fp32 [B, T, H]); required
 *   dbeta          gradient of beta (fp32) or NULL to skip it; with beta
 *                  NULL it is the gradient at beta = 1
 *   dS0, dM0       gradients of the initial states (fp32) or NULL to skip
 *   workspace      at least mdn_chunk_bwd_workspace_size(...) bytes,
 *                  256-byte aligned; contents undefined on exit
 * Every output must be distinct from every input and from the other
 * outputs.  Errors: as mdn_chunk_fwd, and MDN_ERR_INVALID_ARG for a missing
 * required pointer, a misaligned one, an output that aliases, or a workspace
 * that is too small.
 */
mdn_status mdn_chunk_bwd(const void *q, const void *k, const void *v,
                         const float *alpha, const float *mu, const float *eta,
                         const float *beta, const void *S_chunks,
                         const void *M_chunks, const void *fwd_workspace,
                         const void *dout,
                         const float *dS_T, const float *dM_T, void *dq,
                         void *dk_out, void *dv_out, float *dalpha, float *dmu,
                         float *deta, float *dbeta, float *dS0, float *dM0,
                         const int32_t *cu_seqlens, int n_seq, int B, int T,
                         int H, int dk, int dv, mdn_dtype dtype, int chunk,
                         void *workspace, size_t workspace_bytes, void *stream);

/*
 * Bytes of device workspace mdn_block_fwd needs (a multiple of 256; 0 for
 * invalid sizes).
 */
size_t mdn_block_fwd_workspace_size(int n_seq, int T_total, int H, int d,
                                    int d_model, mdn_dtype dtype);

/*
 * mdn_block_fwd — the MDN token-mixer block around the memory core.
 *
 * Defined by: slides, frame "The memory sits inside a familiar
 * language-model block" (Sec. 3.3, Fig. 3 of the paper) and reading notes
 * section 2.9: project, short-convolve and activate q, k, v; correct the
 * query (q - d k, Comba) and L2-normalise q and k; generate the four gates
 * (mdn_prepare_inputs' parameterisation); update memory and momentum
 * (mdn_chunk_fwd); then y_t = W_o [sigmoid(W_g x_t) * RMSNorm(o_t)].
 * Readings where the pages are silent: the short convolution is causal,
 * depthwise along the tokens, of width 4 without bias, and restarts at
 * every sequence start; SiLU follows it on q, k and v; RMSNorm runs over
 * each head's d outputs with one weight vector of d entries shared by the
 * heads and epsilon rms_eps.
 *
 * Layout (row-major, innermost last): x, y [B * T, d_model] (dtype);
 *   W_in [d_model, 4 H d + 4 H] (dtype), columns q | k | v | g (H d each,
 *   head-major) | z_alpha | z_beta | z_mu | z_eta (H each);
 *   conv_w [3 H d, 4] fp32 (tap j multiplies the input 3 - j tokens back),
 *   rows in W_in's q | k | v column order; rms_w [d] fp32;
 *   W_o [H d, d_model] (dtype); states as mdn_chunk_fwd ([n_seq, H, d, d]
 *   fp32, S0/M0 NULL for zero, S_T/M_T NULL to skip); cu_seqlens as
 *   mdn_chunk_fwd (packed sequences; the convolution restarts at each).
 *   Gate parameters a, b, s, tau, log_mu_min, comba_d as mdn_prepare_inputs.
 * The two projections run as cuBLAS GEMMs (fp32 accumulation; bf16 inputs
 * give fp32 projections, then bf16 q, k, v, o and y); the first call on a
 * device creates that device's cuBLAS handle (cuBLAS allocates a little
 * device memory of its own then); GEMM scratch comes from the workspace.
 * Calls on one device are serialised by the library.
 * Errors: MDN_ERR_INVALID_ARG for missing or misaligned pointers (16 bytes,
 * 4 for cu_seqlens), inconsistent sizes or a short workspace;
 * MDN_ERR_UNSUPPORTED for d not in {64, 128} or d_model not a multiple of 8;
 * the errors of mdn_prepare_inputs and mdn_chunk_fwd; MDN_ERR_CUDA for a
 * failed launch or GEMM.
 */
mdn_status mdn_block_fwd(const void *x, const void *W_in, const float *conv_w,
                         const float *rms_w, const void *W_o, float a, float b,
                         float s, float tau, float log_mu_min, float comba_d,
                         float rms_eps, const float *S0, const float *M0,
                         void *y, float *S_T, float *M_T,
                         const int32_t *cu_seqlens, int n_seq, int B, int T,
                         int H, int d, int d_model, mdn_dtype dtype,
                         void *workspace, size_t workspace_bytes, void *stream);

/* Implementation paths of mdn_chunk_fwd (reported by the profiled variant). */
typedef enum mdn_path {
    MDN_PATH_CUDA_CORE = 0,   /* no tensor-core work: a call without tokens
                                 (the initial states pass through) */
    MDN_PATH_TENSOR_CORE = 1  /* tcgen05 state pass: every call with tokens;
                                 bf16 inputs directly (tcgen05 prep), fp32
                                 inputs as hi / lo bf16 parts with three
                                 products per contraction (fp32 prep) */
} mdn_path;

/*
 * mdn_chunk_fwd_profiled — exactly mdn_chunk_fwd (same arguments, same
 * results, same errors) plus two instrumentation outputs:
 *   stage_events    NULL, or an array of n_stage_events cudaEvent_t handles
 *                   (as void*) created by the caller.  Event i is recorded on
 *                   `stream` before stage i; the last one after the last
 *                   stage.  Stages: 0 = per-chunk preparation (offsets,
 *                   coefficients, Gram matrices, triangular inverse),
 *                   1 = sequential state pass (residuals, outputs, carry).
 *                   n_stage_events must be 0 or 3.  With stage events the
 *                   call runs whole sequences (no time segments), so that
 *                   the two stages follow one another.
 *   path_out        NULL, or receives the mdn_path that ran.
 */
mdn_status mdn_chunk_fwd_profiled(
    const void *q, const void *k, const void *v, const float *alpha,
    const float *mu, const float *eta, const float *beta, const float *S0,
    const float *M0, void *o, float *S_T, float *M_T,
    const int32_t *cu_seqlens, int n_seq, int B, int T, int H, int dk, int dv,
    mdn_dtype dtype, int chunk, void *workspace, size_t workspace_bytes,
    void *stream, void *const *stage_events, int n_stage_events,
    int *path_out);

/*
 * mdn_chunk_fwd_kernel_count — how many kernels one mdn_chunk_fwd call with
 * these sizes enqueues on the current device (a diagnostic, e.g. for launch
 * counts in a benchmark; it does not launch anything).  `packed` is nonzero
 * when cu_seqlens is given (then B is 1 and T the packed total),
 * `final_states` nonzero when both S_T and M_T are given.  The count covers
 * the chunk-offset kernel (packed sequences), the split of fp32 inputs, the
 * preparation and the state pass, or, for long equal-length bf16 sequences
 * on narrow state slices, two kernels per time segment.  0 for sizes the
 * call would reject.  No citation: a property of this implementation.
 */
int mdn_chunk_fwd_kernel_count(int n_seq, int B, int T, int H, int dk, int dv, mdn_dtype dtype,
                               int packed, int final_states);

/* Size of the library-owned scratch array of mdn_chunk_fwd_static_ws. */
#define MDN_STATIC_WORKSPACE_BYTES (32u << 20)

/*
 * mdn_chunk_fwd_static_ws — mdn_chunk_fwd without a caller-provided
 * workspace, for callers that cannot allocate device memory where they run
 * the prefill (for example a server that reserves all device memory at start
 * and forbids allocation afterwards, since cudaMalloc may synchronise the
 * device and take unbounded time, or plugin code with no handle to its host's
 * allocator).  The paper has no counterpart: this is a deployment interface.
 *
 * Arguments, layouts, results and errors are those of mdn_chunk_fwd (minus
 * workspace and workspace_bytes).  The scratch is a file-scope device array of
 * MDN_STATIC_WORKSPACE_BYTES (32 MiB) inside the library; a device holds it
 * from the first use until the process exits.  The call allocates and frees
 * nothing.
 *  - Size limit: if mdn_chunk_fwd_workspace_size(n_seq, B*T, H, dk, dv, dtype)
 *    exceeds MDN_STATIC_WORKSPACE_BYTES the call returns MDN_ERR_UNSUPPORTED
 *    and enqueues nothing.
 *  - Set-up: the first call on a device looks up the array's device address
 *    (cudaGetSymbolAddress, with that device current).  With lazy module
 *    loading (the CUDA default) that lookup is also when the array receives
 *    its device memory, so it can fail with MDN_ERR_CUDA if the device is out
 *    of memory then: make the first call on each device before reserving the
 *    device's memory, and before any stream capture.
 *  - Sharing: every call on a device uses the same array.  Nothing in it must
 *    start at zero (each call writes all it reads), but calls whose work
 *    overlaps on the GPU (other streams, other host threads) race on it:
 *    serialise them, e.g. on one stream.
 */
mdn_status mdn_chunk_fwd_static_ws(const void *q, const void *k, const void *v,
                                   const float *alpha, const float *mu,
                                   const float *eta, const float *beta,
                                   const float *S0, const float *M0, void *o,
                                   float *S_T, float *M_T,
                                   const int32_t *cu_seqlens, int n_seq, int B,
                                   int T, int H, int dk, int dv,
                                   mdn_dtype dtype, int chunk, void *stream);

/*
 * mdn_prepare_inputs — the inputs of one MDN layer in one pass: the four gates
 * from their per-head scalar projections z = W x_t, and the L2-normalised
 * queries and keys with the Comba output correction.
 *
 * Defined by: slides, frame "Coupled gates restrict the spectral region"
 * (Sec. 3.3) and reading notes section 2.8 for the gates,
 *   eta   = 1 + tanh(z_eta / tau)                           in (0, 2)
 *   alpha = alpha_max exp(f(z_alpha)),   alpha_max = cos^2(arctan(s eta))
 *   beta  = sigmoid(z_beta) beta_max,    beta_max  = sin^2(arctan(s eta))
 *   mu    = exp(max(f(z_mu), log_mu_min)),   f(z) = -a softplus(z + b)
 * (so alpha + beta <= 1; the reported experiments use log_mu_min = -2), and
 * reading notes section 2.9 for q_hat = (q - comba_d k) / |q - comba_d k|,
 * k_hat = k / |k| per (token, head); a row of norm zero is written as zeros.
 *
 * Layout: q_in, k_in, q_out, k_out [n_tokens, H, d] in dtype (d = 64 or 128),
 *   16-byte aligned; z_* and the gate outputs [n_tokens, H] fp32, the layout
 *   mdn_chunk_fwd and mdn_decode_step take.
 * Ownership: all buffers are the caller's device memory.  q_out may be q_in
 *   and k_out may be k_in (in place); no other overlap.
 * Errors: MDN_ERR_INVALID_ARG for a missing or misaligned pointer, a negative
 *   size, a <= 0 or tau <= 0; MDN_ERR_UNSUPPORTED for d not in {64, 128};
 *   MDN_ERR_CUDA for a launch failure.  Asynchronous on `stream`.
 */
mdn_status mdn_prepare_inputs(const void *q_in, const void *k_in, const float *z_alpha,
                              const float *z_beta, const float *z_mu, const float *z_eta,
                              void *q_out, void *k_out, float *alpha, float *beta,
                              float *mu, float *eta, int n_tokens, int H, int d,
                              mdn_dtype dtype, float a, float b, float s, float tau,
                              float log_mu_min, float comba_d, void *stream);

/*
 * mdn_decode_step — one recurrent step for N sequences (one token each),
 * updating both states in place.
 *
 * Defined by: the token recurrence above (slides Eqs. (3)-(5); reading notes
 * section 2.2); the slides note decoding uses this recurrence with the two
 * fixed-size states ("Chunk outputs combine incoming states ..." frame).
 *
 * Layout: q, k [N, H, dk]; v, o [N, H, dv] (dtype); alpha, mu, eta, beta
 * [N, H] fp32 (beta NULL = 1); S, M [N, H, dk, dv] fp32, read and replaced by
 * S_t, M_t.  o receives S_t^T q.  o must not overlap any input.
 */
mdn_status mdn_decode_step(const void *q, const void *k, const void *v,
                           const float *alpha, const float *mu,
                           const float *eta, const float *beta, float *S,
                           float *M, void *o, int N, int H, int dk, int dv,
                           mdn_dtype dtype, void *stream);

/*
 * Synchronises `stream`, then reads and clears the device status word of the
 * current device.  Returns MDN_OK if no kernel reported a problem since the
 * last read, MDN_ERR_DEVICE_TIMEOUT if a bounded device-side wait expired
 * (that launch's outputs are then undefined), MDN_ERR_INVALID_ARG if a chunk
 * forward found its cu_seqlens malformed (see mdn_chunk_fwd), MDN_ERR_CUDA
 * if the synchronisation or the read failed.
 */
mdn_status mdn_get_device_status(void *stream);

/*
 * mdn_wait_selftest — checks the device-side failure path on the current
 * device without faulting it.  Every wait inside the library's kernels is
 * bounded: when it expires the kernel records MDN_ERR_DEVICE_TIMEOUT in the
 * device status word, stops its other warps, frees its tensor memory and
 * returns, so the context stays usable.  This call enqueues one small
 * kernel (one CTA of two warps holding 32 tensor-memory columns) that waits
 * with that same helper on a barrier nothing ever arrives at, with a limit
 * of limit_us microseconds instead of the kernels' 1 s, so the limit always
 * expires.  A later mdn_get_device_status(stream) then returns
 * MDN_ERR_DEVICE_TIMEOUT (and clears it).  Not part of the method (the
 * paper has no counterpart); it exists so that tests can exercise the
 * timeout path.
 *
 * Arguments: limit_us in [1, 1000000]; stream as elsewhere.
 * Errors: MDN_ERR_INVALID_ARG for limit_us out of range; MDN_ERR_UNSUPPORTED
 * for a device other than compute capability 10.3; MDN_ERR_CUDA for a failed
 * launch.
 */
mdn_status mdn_wait_selftest(int limit_us, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* MDN_H_ */
