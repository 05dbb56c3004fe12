/*
 * ida.h -- C ABI of the GB300 (sm_103a) Interdomain Attention token mixer.
 *
 * The operation is the token mixer of "Interdomain Attention: Beyond
 * Token-Level Key-Value Memory" (arXiv 2605.24330) in its scalable form, as
 * the German technical summary of that paper states it in the section
 * "Skalierbare Implementierung" (the Dutch summary, "Schaalbare
 * Implementatie", says the same).  Per batch row b and head h, with
 * x_t in R^R the raw query or key row and v_t in R^d the value row:
 *
 *   feature map     xi(x) = SiLU(SC(x)) / ||SiLU(SC(x))||^2, SC a causal
 *                   depthwise conv of width W (own taps for q and for k);
 *   normalisation   kt = RMSNorm(xi(k)) * w_k + b_k,  vt = RMSNorm(v) * w_v + b_v
 *                   (per-head weights and biases on the key and value halves);
 *   recurrent core  one complex diagonal S4D recurrence over z_t = [kt_t ; vt_t]:
 *                   X_t = lambda o X_{t-1} + B o z_t, X_{-1} = 0, with
 *                   U_t = X_t[:, :R] (M x R) and Gamma_t = X_t[:, R:] (M x d),
 *                   the state shapes of the paper's Fig. 1 caption;
 *   readout         o_t = Re( xi(q_t)^T U_t^T Gamma_t )  (denominator-free), or
 *                   with IDA_READOUT_ETA the ratio form of the summary's
 *                   "Theoretische Herleitung": o_t /= Re( xi(q_t)^T U_t^T eta_t ),
 *                   eta_t = lambda o eta_{t-1} + B.
 *
 * Readings where the pages are silent: ||.||^2 is the squared Euclidean norm
 * plus IDA_EPS_FEAT; RMSNorm uses mean square + IDA_EPS_RMS; conv taps in
 * cross-correlation order (tap W-1 on the current token), zero left padding,
 * no conv bias, v not convolved, q not RMS-normed; lambda and B are the
 * discretised complex parameters (no conjugation, real part taken last, no
 * factor 2); the eta division has no epsilon.
 *
 * Conventions for every call:
 *   - All data pointers are device pointers owned by the caller, 16-byte
 *     aligned (ida_forward_host excepted: its sequence buffers are host
 *     memory).  The library allocates no device memory per call.
 *   - Calls are asynchronous on `stream` and never synchronise.  The return
 *     value reports argument errors (nothing is launched) and launch errors.
 *   - Kernels never trap.  A device-side fault detected by a kernel (e.g. a
 *     bounded wait that ran out) is recorded in a device error word and
 *     returned as IDA_ERR_DEVICE by the next call (or by ida_device_error).
 *   - Outputs must not alias inputs.
 *   - Supported: 8 <= R,d <= 256 with R % 8 == 0 and d % 8 == 0,
 *     1 <= M <= 128, 1 <= W <= 4.  Other shapes return IDA_ERR_UNSUPPORTED.
 */
#ifndef IDA_H
#define IDA_H

#include <stddef.h>

#if defined(__GNUC__)
#define IDA_API __attribute__((visibility("default")))
#else
#define IDA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Same underlying type as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st *ida_stream_t;

typedef enum {
    IDA_OK = 0,
    IDA_ERR_ARG = 1,          /* null/misaligned pointer, negative size, bad enum */
    IDA_ERR_UNSUPPORTED = 2,  /* valid but outside the supported shape set       */
    IDA_ERR_CUDA = 3,         /* a CUDA runtime call or launch failed             */
    IDA_ERR_DEVICE = 4        /* a kernel recorded a device-side error            */
} ida_status;

enum { IDA_F32 = 0, IDA_BF16 = 1 };            /* dtype of q, k, v and out */

enum {
    IDA_READOUT_ETA = 1,        /* eta-normalised readout instead of denominator-free */
    IDA_FEAT_L2 = 2,            /* feature map SiLU(s) / (||SiLU(s)||_2 + IDA_EPS_FEAT), the "SiLU/l_2"
                                   wording of the Chinese summary's introduction, instead of the
                                   squared norm of the German and Dutch summaries' feature map */
    IDA_PATH_SEQUENTIAL = 256   /* force the token-sequential CUDA-core prefill kernel */
};

#define IDA_EPS_FEAT 1e-6f
#define IDA_EPS_RMS 1e-6f

/*
 * Number of floats of one (b,h) recurrent state, the format shared by
 * ida_forward's final_state and ida_decode_step's state_inout:
 *   [2M][R+d]  planar complex state: rows 0..M-1 hold Re, rows M..2M-1 hold Im;
 *              columns 0..R-1 are U, columns R..R+d-1 are Gamma;
 *   [2M]       eta (Re then Im), maintained whichever readout is used;
 *   [W-1][R]   raw q rows of the last W-1 positions (conv tail), oldest first;
 *   [W-1][R]   raw k rows, same;
 *   0..3       padding floats so that every unit starts on a 16-byte boundary.
 * Positions before the first token are zero.  Returns 0 for invalid sizes.
 */
IDA_API size_t ida_state_floats(int d, int R, int M, int W);

/*
 * Prefill: run the mixer over N positions of B x H independent (b,h) units,
 * starting from the zero state.
 *   q, k    [B, N, H, R]  dtype (IDA_F32: float, IDA_BF16: bfloat16)
 *   v       [B, N, H, d]  dtype
 *   conv_w  [2, H, R, W]  float; [0] = query taps, [1] = key taps
 *   norm_w  [H, R + d]    float; RMSNorm weights, key half first
 *   bias    [H, R + d]    float; RMSNorm biases, key half first
 *   lambda  [H, M, 2]     float; complex modes (re, im)
 *   Bvec    [H, M, 2]     float; complex input gains (re, im)
 *   out     [B, N, H, d]  dtype; written
 *   final_state  NULL, or [B, H] x ida_state_floats(d, R, M, W) floats:
 *           receives the state after the last position.
 *   flags   IDA_READOUT_ETA, IDA_FEAT_L2 and/or IDA_PATH_SEQUENTIAL.
 * N == 0 writes nothing but the zero final_state (if given).
 */
IDA_API ida_status ida_forward(const void *q, const void *k, const void *v,
                       const float *conv_w, const float *norm_w,
                       const float *bias, const float *lambda,
                       const float *Bvec, void *out, float *final_state,
                       int B, int H, int N, int d, int R, int M, int dtype,
                       int W, int flags, ida_stream_t stream);

/*
 * Prefill with a caller-provided device workspace.  Same arguments and
 * results as ida_forward, plus:
 *   workspace        NULL, or a 16-byte aligned device buffer owned by the
 *                    caller, not shared with a concurrent call;
 *   workspace_bytes  its size.
 * With a workspace of at least ida_forward_workspace_bytes(...) bytes the
 * tensor-core path splits each (b,h) sequence into segments that run on
 * separate SMs (their local end states, then their start states, are kept
 * in the workspace); with a smaller or NULL workspace it runs as
 * ida_forward.  The workspace's contents on entry are ignored.
 */
IDA_API ida_status ida_forward_ws(const void *q, const void *k, const void *v,
                          const float *conv_w, const float *norm_w,
                          const float *bias, const float *lambda,
                          const float *Bvec, void *out, float *final_state,
                          int B, int H, int N, int d, int R, int M, int dtype,
                          int W, int flags, void *workspace,
                          size_t workspace_bytes, ida_stream_t stream);

/*
 * Prefill that continues from a given state: the recurrence starts from
 * state_in instead of zero, and the causal conv of the first positions reads
 * the raw q, k rows carried in its conv tails (the positions before 0).
 * Chunked prefill and serving can resume a sequence this way.  The pages
 * state the recurrence and the fixed-size state it carries ("Interdomain
 * Attention: Beyond Token-Level Key-Value Memory", German technical summary,
 * "Rekurrenter Kern"); resuming from a stored state is this library's use of
 * it.  Same arguments and results as ida_forward_ws, plus:
 *   state_in  NULL (the zero state: then this is ida_forward_ws), or a
 *             16-byte aligned device buffer of [B, H] x ida_state_floats(...)
 *             floats in the layout above (a final_state of an earlier
 *             prefill, or a decode state).  Read only.  It must not overlap
 *             final_state (IDA_ERR_ARG).  For bf16 inputs the tails are
 *             rounded to bf16 where the tensor-core path stages them.
 * N == 0 copies state_in to final_state (if given).  The eta readout and
 * other shapes that run token by token take a slower fp32 kernel from a
 * non-zero state.
 */
IDA_API ida_status ida_forward_from(const void *q, const void *k, const void *v,
                            const float *conv_w, const float *norm_w,
                            const float *bias, const float *lambda,
                            const float *Bvec, const float *state_in,
                            void *out, float *final_state,
                            int B, int H, int N, int d, int R, int M, int dtype,
                            int W, int flags, void *workspace,
                            size_t workspace_bytes, ida_stream_t stream);

/*
 * Workspace bytes that let ida_forward_ws split sequences across the SMs of
 * the current device for this shape; 0 when no split applies (the call then
 * needs no workspace).  Queries the device (no other CUDA work).
 */
IDA_API size_t ida_forward_workspace_bytes(int B, int H, int N, int d, int R,
                                           int M, int dtype, int W, int flags);

/*
 * Prefill for callers that cannot allocate device memory.  (The paper has no
 * counterpart: this is a property of the library, not of the method.)
 *
 * Same arguments and results as ida_forward; it runs what ida_forward_ws
 * runs with a workspace, but takes that workspace from one array of static
 * device memory built into this library instead of from the caller.  Use it
 * where the calling code may not allocate: a plug-in that a host framework
 * hands only its input and output buffers, a serving loop that must not
 * touch the allocator after start-up, code with no allocator in reach.
 *   - It calls no cudaMalloc, cudaFree or other device-memory allocator.
 *     One thing is set up once per process by whichever entry point runs
 *     first (this one included): a pinned, mapped host word (cudaHostAlloc,
 *     4 bytes) where kernels report device-side errors.  A caller that may
 *     not do even that makes any other prefill or decode call first.
 *   - Limit: the array holds 32 MiB on every GPU that loads the library,
 *     kept until the process exits.  Every supported shape runs: sequences
 *     are split across SMs only as finely as 32 MiB of segment states allow
 *     (ida_forward_ws with a larger workspace may split more finely; with a
 *     workspace of ida_forward_workspace_bytes(...) <= 32 MiB both run the
 *     same plan and give the same bytes).
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current and keeps it for the
 *     process; make that first call before any stream capture.  A
 *     cudaDeviceReset (or anything else that tears down the device's primary
 *     context) invalidates the kept address: do not call this entry point on
 *     that device afterwards.
 *   - Every call on a device shares the one array and leaves its contents
 *     behind; nothing in it needs to start at zero, but calls that overlap
 *     on the GPU (e.g. on two streams) race on it.
 */
IDA_API ida_status ida_forward_noalloc(const void *q, const void *k, const void *v,
                               const float *conv_w, const float *norm_w,
                               const float *bias, const float *lambda,
                               const float *Bvec, void *out, float *final_state,
                               int B, int H, int N, int d, int R, int M,
                               int dtype, int W, int flags, ida_stream_t stream);

/*
 * Prefill from host memory.  (The paper has no counterpart: this is a property
 * of the library.)  The same computation as ida_forward_from, with the
 * sequence data in host memory:
 *   q, k, v, out             host buffers, shapes and dtype as in ida_forward;
 *   state_in, final_state    NULL or host buffers of [B, H] x
 *                            ida_state_floats(d, R, M, W) floats (as in
 *                            ida_forward_from); they must not overlap;
 *   conv_w ... Bvec          device pointers, as in ida_forward;
 *   staging                  16-byte aligned device buffer owned by the
 *                            caller, not shared with a concurrent call;
 *   staging_bytes            at least ida_forward_host_staging_bytes(...).
 * Host buffers need no alignment.  Pinned (page-locked) host memory lets the
 * copies run at full speed and overlap the kernels; pageable memory works
 * but the copies then serialise.
 *
 * On the tensor-core path (see ida_forward_ws) the positions are cut into
 * slices of at least 512 (a multiple of 64, the last one shorter).  The copy
 * of slice i to the device, the prefill of slice i-1 (resumed from the state
 * after slice i-2, as ida_forward_from does) and the copy of slice i-2's
 * outputs to the host run at the same time, on three streams the library
 * creates once per device; the staging buffer holds two slices of q, k, v and
 * out, two states and a prefill workspace.  Other shapes run as one slice.
 * The split changes only the rounding of the carried state, within the
 * path's tolerance of an unsplit call.
 *
 * Asynchronous like every call: the copies and kernels are ordered after the
 * work queued on `stream` before the call, and work queued on `stream` after
 * it runs after the last copy to the host.  The host buffers must stay valid
 * and unchanged until then.  Calls on one device are enqueued one at a time
 * (a mutex per device); their copies and kernels may still overlap on the
 * GPU, so concurrent calls need separate staging buffers.  A device error
 * reported while the slices are enqueued stops the enqueueing: the call
 * returns IDA_ERR_DEVICE and `stream` still waits for what was enqueued.
 */
IDA_API ida_status ida_forward_host(const void *q, const void *k, const void *v,
                            const float *conv_w, const float *norm_w,
                            const float *bias, const float *lambda,
                            const float *Bvec, const float *state_in,
                            void *out, float *final_state,
                            int B, int H, int N, int d, int R, int M, int dtype,
                            int W, int flags, void *staging,
                            size_t staging_bytes, ida_stream_t stream);

/*
 * Staging bytes ida_forward_host needs for this shape (with or without
 * state_in / final_state); 0 when B*H == 0 or the arguments are invalid.
 * Queries the device (no other CUDA work).
 */
IDA_API size_t ida_forward_host_staging_bytes(int B, int H, int N, int d, int R,
                                              int M, int dtype, int W, int flags);

/*
 * One recurrent decode step (one new position per (b,h) unit): the fixed-size
 * state is updated in O(1) work per position, independent of the number of
 * positions before it ("Interdomain Attention: Beyond Token-Level Key-Value
 * Memory", translated paper text, section 1, on constant-cost recurrent
 * inference; German technical summary, "Problemstellung").
 *   q, k [B, H, R], v [B, H, d] in dtype; parameters as for ida_forward;
 *   state_inout [B, H] x ida_state_floats(...) floats, read and updated in
 *   place (state, eta and the conv tails); out [B, H, d] in dtype.
 *   flags: IDA_READOUT_ETA and/or IDA_FEAT_L2 (IDA_PATH_SEQUENTIAL is
 *   accepted and has no effect: a step is always one position).
 * A prefill's final_state is a valid state_inout; use the same IDA_FEAT_L2
 * setting for the prefill and the steps that continue it.
 */
IDA_API ida_status ida_decode_step(const void *q, const void *k, const void *v,
                           const float *conv_w, const float *norm_w,
                           const float *bias, const float *lambda,
                           const float *Bvec, float *state_inout, void *out,
                           int B, int H, int d, int R, int M, int dtype,
                           int W, int flags, ida_stream_t stream);

/*
 * Backward pass of ida_forward (from the zero state): the gradients of a loss
 * L with respect to the inputs and every parameter, given dL/d out.  The
 * pages train the layer in models of 125M to 1.3B parameters ("Interdomain
 * Attention: Beyond Token-Level Key-Value Memory", German technical summary,
 * "Hauptbeiträge"), which takes these gradients; the forward it differentiates
 * is the one ida_forward computes, readings included.
 *   q, k, v, conv_w, norm_w, bias, lambda, Bvec  as for ida_forward;
 *   dout    [B, N, H, d] dtype: dL/d out;
 *   dq, dk  [B, N, H, R] dtype, dv [B, N, H, d] dtype: written;
 *   dconv_w [2, H, R, W], dnorm_w / dbias [H, R + d], dlambda / dBvec [H, M, 2]:
 *           float, written (not accumulated), summed over the batch rows;
 *           complex parameters get (dL/d Re, dL/d Im);
 *   flags   IDA_READOUT_ETA and/or IDA_FEAT_L2, as given to the forward;
 *   workspace  a 16-byte aligned device buffer of at least
 *           ida_backward_workspace_bytes(...) bytes (required when N > 0;
 *           contents on entry ignored): feature rows, their gradients, the
 *           state every 64 positions and the states of one 64-position chunk
 *           per unit.
 * The arithmetic is fp64 for fp32 inputs and fp32 for bf16 inputs; sums run
 * in a fixed order, so the results are deterministic.  N == 0 writes zero
 * parameter gradients (q, k, v, dout, dq, dk, dv may then be NULL).  Same
 * shape support as ida_forward.
 */
IDA_API ida_status ida_backward(const void *q, const void *k, const void *v,
                        const float *conv_w, const float *norm_w,
                        const float *bias, const float *lambda,
                        const float *Bvec, const void *dout,
                        void *dq, void *dk, void *dv,
                        float *dconv_w, float *dnorm_w, float *dbias,
                        float *dlambda, float *dBvec,
                        int B, int H, int N, int d, int R, int M, int dtype,
                        int W, int flags, void *workspace,
                        size_t workspace_bytes, ida_stream_t stream);

/* Workspace bytes ida_backward needs for this shape (0 for invalid sizes or
 * N == 0).  Host-only arithmetic: queries nothing. */
IDA_API size_t ida_backward_workspace_bytes(int B, int H, int N, int d, int R,
                                            int M, int dtype, int W, int flags);

/*
 * The ideal interdomain layer on random Fourier features: the layer the paper
 * derives before its scalable form ("Interdomain Attention: Beyond
 * Token-Level Key-Value Memory", translated paper text, section 3.1: the
 * finite-feature ratio of Eq. 4 with the Fourier features of Eqs. 5-6, read
 * out through the recurrent state of Fig. 1b).  Per (b,h) unit:
 *   xi(x)  = D^-1/2 [cos(Omega_h x); sin(Omega_h x)]  (feature width 2D),
 *   X_t    = lambda o X_{t-1} + B o [xi(k_t); v_t],  eta_t = lambda o eta_{t-1} + B,
 *   o_t    = Re(xi(q_t)^T U_t^T Gamma_t) / Re(xi(q_t)^T U_t^T eta_t),
 * from the zero state, with no conv and no normalisation (the derivation has
 * neither).
 *   q, k   [B, N, H, R_in] dtype;  v, out [B, N, H, d] dtype;
 *   omega  [H, D, R_in] float: the random frequencies (drawn by the caller);
 *   lambda, Bvec [H, M, 2] float, as for ida_forward.
 * Supported: R_in <= 256, D <= 128, d <= 256, M <= 128.  fp64 arithmetic for
 * fp32 inputs, fp32 for bf16; deterministic.  Allocates nothing.
 */
IDA_API ida_status ida_forward_ideal(const void *q, const void *k, const void *v,
                             const float *omega, const float *lambda,
                             const float *Bvec, void *out,
                             int B, int H, int N, int d, int R_in, int D,
                             int M, int dtype, ida_stream_t stream);

/*
 * Rotary position embeddings on the mixer's queries and keys, in place.  The
 * pages embed the token mixer in a Llama-style decoder with rotary position
 * embeddings ("Interdomain Attention: Beyond Token-Level Key-Value Memory",
 * German technical summary, "Skalierbare Implementierung", "Architektur");
 * the library reads that as the decoder's usual RoPE on q and k before the
 * mixer (the pages give no formula).  Channel pairs (2i, 2i+1) of the row at
 * position p = pos0 + t rotate by the angle p * base^(-2i/R):
 *   x'_{2i}   = x_{2i} cos(a) - x_{2i+1} sin(a),
 *   x'_{2i+1} = x_{2i} sin(a) + x_{2i+1} cos(a).
 *   q, k   [B, N, H, R] dtype, contiguous, 16-byte aligned, rotated in place
 *          (k may be NULL: only q is rotated; k must not alias q);
 *   pos0   the position of row t = 0 (>= 0), e.g. the length already decoded;
 *   base   the frequency base (> 1; 10000 in the Llama decoder).
 * Supported: 8 <= R <= 256 with R % 8 == 0, H*R <= 2^24.  Each frequency is
 * formed in fp64 and the angle reduced modulo 2 pi exactly (a 64-bit
 * fixed-point phase); sin / cos and the rotation run in fp32 (bf16 inputs
 * are rounded back to bf16).  N == 0, B == 0 or H == 0 does nothing.
 * Asynchronous on `stream`; allocates nothing.
 */
IDA_API ida_status ida_rope(void *q, void *k, int B, int N, int H, int R,
                            int pos0, float base, int dtype,
                            ida_stream_t stream);

/*
 * Self-test of the failure reporting (no counterpart in the paper: a property
 * of the library).  Launches one warp on `stream` that waits, through the
 * bounded-wait helper every prefill kernel uses, on an mbarrier nothing
 * arrives on; after about limit_cycles SM clock cycles (1 .. 4e9) the wait
 * gives up and the kernel records the wait-timeout code (1) in the device
 * error word and returns.  The GPU and the context stay usable: the next
 * call returns IDA_ERR_DEVICE, or ida_device_error() reports and clears the
 * word, once the stream has reached the kernel.  Allocates nothing beyond the
 * once-per-process error word.
 */
IDA_API ida_status ida_selftest_bounded_wait(long long limit_cycles, ida_stream_t stream);

/* Reads and clears the device error word without synchronising; returns
 * IDA_OK or IDA_ERR_DEVICE.  *code (nullable) receives the raw word. */
IDA_API ida_status ida_device_error(unsigned *code);

/* Static text for a status code. */
IDA_API const char *ida_status_str(ida_status s);

/* Human-readable reason of the last non-OK status on the calling thread. */
IDA_API const char *ida_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* IDA_H */
