/*
 * prism.h -- C ABI of the GB300 (sm_103a) PRISM memory-recurrence forward.
 *
 * The operation ("PRISM: Parallel Residual Iterative Sequence Model",
 * arXiv 2602.10796; reading notes at liuzhao09.github.io/papers/prism.html,
 * sections 2.2 "Write-Forget Decoupling" and 2.3 "Input-Anchored
 * Simulation"; Tencent article at youzy.cn, part 03 "PRISM", items two to
 * four).  Per (batch b, head h), for t = 0..T-1, with R = L - 1:
 *
 *   h_t     = sum_{j=0..3} w_j (.) v_{t-j}              (v_{<0} = 0)
 *   g_t     = GELU'(h_t),   e_t = v_t - GELU(h_t)        (exact erf GELU)
 *   r_{t,1} = e_t,  r_{t,l+1} = r_{t,l} (.) (1 - eta_{t,l} g_t)
 *   S_t     = alpha_t S_{t-1} (I - beta_t k_t k_t^T)
 *             + beta_t v_t k_t^T + sum_{l=1..R} gamma_{t,l} (g_t (.) r_{t,l}) u_{t,l}^T
 *   o_t     = S_t q_t,     S_0 = 0,   S_t in R^{dv x dk}
 *
 * With L = 1 this is the gated delta rule (GDN).  The sequence is evaluated in
 * 64-token chunks (a WY/UT form of the products of the rank-1 transitions);
 * the state is passed between chunks either segment-parallel (tensor-core
 * path, dk = dv = 64, L <= 4) or as per-chunk affine maps S -> S A_c + B_c
 * applied in order (tensor-core path, dk = dv = 128, L <= 16); the result
 * equals the sequential definition up to floating-point rounding.
 *
 * Tensor layouts (all row-major and contiguous, caller-owned device memory):
 *   q, k    [B,H,T,dk]   io dtype        v, out [B,H,T,dv]   io dtype
 *   u       [B,H,T,R,dk] io dtype        conv_w [H,4,dv]     io dtype
 *           (slot l-1 holds level l; tap j of conv_w multiplies v_{t-j})
 *   beta, alpha [B,H,T]  float32         gamma, eta [B,H,T,R] float32
 *           (eta[..., R-1] is never read: it would only shape a residual
 *            that no level uses)
 * The io dtype is fixed by the plan (float32 or bfloat16); `out` has the io
 * dtype unless PRISM_OPT_OUT_DTYPE selects float32.  Every io tensor and `out`
 * must start on a 16-byte boundary, every float32 gate tensor on 4 bytes.
 *
 * Errors.  Every call returns a prism_status.  Argument errors are reported
 * before anything is launched.  A failed launch returns PRISM_ERR_CUDA.
 * Conditions detected on the device (an internal bound check, a bounded
 * wait that expired) are written to a status word in the plan's workspace;
 * read it with prism_plan_last_device_status() after synchronising the
 * stream.  prism_last_error_message() gives a one-line description of the
 * last error reported on the calling thread.
 *
 * Only NVIDIA sm_103 devices (GB300) are supported; there is no CPU path.
 */
#ifndef PRISM_GB300_H
#define PRISM_GB300_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st; /* the CUDA runtime's cudaStream_t is a pointer to this */

#if defined(__GNUC__)
#define PRISM_API __attribute__((visibility("default")))
#else
#define PRISM_API
#endif

typedef enum prism_status {
    PRISM_OK = 0,
    PRISM_ERR_INVALID_ARG = 1, /* null pointer, bad size, L differs from the plan's */
    PRISM_ERR_UNSUPPORTED = 2, /* a size outside dk,dv in {64,128}, 1 <= L <= 16 */
    PRISM_ERR_MISALIGNED = 3,  /* a tensor not aligned as stated above */
    PRISM_ERR_ARCH = 4,        /* current device is not sm_103 */
    PRISM_ERR_CUDA = 5,        /* a CUDA runtime call or launch failed */
    PRISM_ERR_TIMEOUT = 6,     /* a bounded device-side wait expired */
    PRISM_ERR_DEVICE = 7       /* a device-side bound check failed */
} prism_status;

typedef enum prism_dtype {
    PRISM_F32 = 0,  /* q, k, v, u, conv_w, out in float32 (fp32 arithmetic throughout) */
    PRISM_BF16 = 1  /* ... in bfloat16; tensor-core operands bf16, accumulation fp32 */
} prism_dtype;

typedef enum prism_option {
    PRISM_OPT_SEGMENTS = 0,  /* segments per sequence for the segment-parallel state passing
                                (dk = dv = 64 tensor-core kernels); 0 = automatic */
    PRISM_OPT_PATH = 1,      /* 0 = automatic, 1 = portable fp32 kernels, 2 = tensor-core path (bf16 io
                                with dk = dv = 64 and L <= 4, or dk = dv = 128 and L <= 16; other
                                shapes return PRISM_ERR_UNSUPPORTED); automatic takes the tensor-core
                                path wherever it applies */
    PRISM_OPT_WAIT_NS = 2,   /* bound of any device-side wait in ns; 0 = default (100 ms) */
    PRISM_OPT_TIMING = 3,    /* 1 = record CUDA events around each kernel (see prism_plan_kernel_times) */
    PRISM_OPT_OUT_DTYPE = 4  /* prism_dtype of `out`; default = the plan's io dtype.  float32 output
                                keeps the fp32-accumulated result unrounded (bf16 io only changes
                                the inputs and the tensor-core operands) */
} prism_option;

/* Duration of one kernel launch of the last forward (see prism_plan_kernel_times). */
typedef struct prism_kernel_time {
    const char *name; /* static string naming the kernel */
    float ms;         /* event-measured duration on the launch stream; -1 if timing was off */
} prism_kernel_time;

typedef struct prism_plan_s *prism_plan_t;

/*
 * prism_plan -- validate the problem sizes, bind the plan to the current CUDA
 * device and allocate its workspace (device memory owned by the plan until
 * prism_plan_destroy).  B, H >= 1, T >= 1; dk, dv in {64, 128}; 1 <= L <= 16.
 * On success *out_plan receives the handle; on error it is set to NULL.
 * A plan may be used by one stream at a time.
 */
PRISM_API prism_status prism_plan(int B, int H, int T, int dk, int dv, int L, prism_dtype io,
                        prism_plan_t *out_plan);

/* Set a plan option (see prism_option).  Takes effect at the next forward. */
PRISM_API prism_status prism_plan_set_option(prism_plan_t plan, prism_option opt, long long value);

/*
 * prism_forward -- enqueue the forward on `stream` (NULL = the legacy default
 * stream) and return without synchronising.  All pointers are device pointers
 * in the layouts above; they are only read (out is only written) and are not
 * retained after the call.  L must equal the plan's L.  With L = 1, u, gamma
 * and eta are not read and may be NULL.
 */
PRISM_API prism_status prism_forward(prism_plan_t plan, const void *q, const void *k, const void *v,
                           const float *beta, const float *alpha, const void *u,
                           const float *gamma, const float *eta, const void *conv_w, int L,
                           void *out, struct CUstream_st *stream);

/*
 * prism_forward_host -- the same forward for callers whose tensors live in
 * host memory (pinned memory makes the copies asynchronous and faster).  The
 * inputs are copied into device buffers owned by the plan (allocated on the
 * first call), the forward runs on `stream`, the output is copied back to
 * `out`, and the call returns after the stream has drained.
 */
PRISM_API prism_status prism_forward_host(prism_plan_t plan, const void *q, const void *k, const void *v,
                                const float *beta, const float *alpha, const void *u,
                                const float *gamma, const float *eta, const void *conv_w, int L,
                                void *out, struct CUstream_st *stream);

/*
 * prism_forward_state -- prism_forward for one part of a sequence that is evaluated over
 * consecutive calls (a prefill in pieces, streaming input, a prefill followed by
 * prism_decode_step).  The recurrence above starts from S_0 = S_init, and the anchor's window
 * reaches back into the previous call: for t - j < 0, v_{t-j} comes from v_hist.  A sequence
 * split into calls this way gives the outputs and final state of one call over the whole
 * sequence, up to floating-point rounding.  (The state is the recurrent state of the layer's
 * RNN form, notes on PRISM, section 2.2; the window is the causal four-tap anchor of
 * section 2.3.)
 *
 * Arguments after conv_w (device pointers, each may be NULL, each 16-byte aligned):
 *   v_hist      [B,H,3,dv]  io dtype  v_{-3}, v_{-2}, v_{-1}, oldest first; NULL = zeros
 *   S_init      [B,H,dv,dk] float32   the state before the first token; NULL = zero state
 *   S_final     [B,H,dv,dk] float32   receives the state after the last token; may be S_init
 *   v_hist_out  [B,H,3,dv]  io dtype  receives the last three tokens of [v_hist; v], the next
 *                                      call's v_hist; may be v_hist
 * Apart from those two pairs, no buffer may overlap another.  The state is carried in fp32;
 * on the tensor-core path the part of the outputs that S_init contributes goes through fp16
 * operands, like the state at every segment boundary.  Otherwise as prism_forward.
 */
PRISM_API prism_status prism_forward_state(prism_plan_t plan, const void *q, const void *k, const void *v,
                                 const float *beta, const float *alpha, const void *u,
                                 const float *gamma, const float *eta, const void *conv_w, int L,
                                 const void *v_hist, const float *S_init, void *out, float *S_final,
                                 void *v_hist_out, struct CUstream_st *stream);

/*
 * prism_decode_step -- one token for each of the plan's B x H sequences: the recurrent form
 * of the layer (notes on PRISM, section 2.2), for serving after a prefill.  It reads and
 * updates the state and the convolution history in place and writes o = S q after the update.
 *   q, k        [B,H,dk]     io dtype        v [B,H,dv]  io dtype     u [B,H,R,dk] io dtype
 *   beta, alpha [B,H]        float32         gamma, eta [B,H,R] float32
 *   conv_w      [H,4,dv]     io dtype
 *   v_hist      [B,H,3,dv]   io dtype: v_{-3}, v_{-2}, v_{-1}; on return shifted by one
 *                            token, with v as the newest
 *   S           [B,H,dv,dk]  float32: the state; on return the state after the token
 *   out         [B,H,dv]     the plan's output dtype
 * The step equals prism_forward_state with T = 1, S_final = S_init = S and v_hist_out =
 * v_hist.  The plan's T is not used, so the plan of a prefill can be reused.  Pointers are
 * device pointers, 16-byte aligned (gates: 4 bytes), not overlapping.  L must equal the
 * plan's L; with L = 1, u, gamma and eta are not read.  Returns once the step is enqueued
 * on `stream`.
 */
PRISM_API prism_status prism_decode_step(prism_plan_t plan, const void *q, const void *k, const void *v,
                               const float *beta, const float *alpha, const void *u,
                               const float *gamma, const float *eta, const void *conv_w, int L,
                               void *v_hist, float *S, void *out, struct CUstream_st *stream);

/*
 * prism_forward_nonlinear -- the non-linear residual variant of the write path (notes on
 * PRISM, section 2.3, "greedy residual subtraction"): a gain vector p_{t,l}, predicted from
 * the anchor outside this library like the directions u_{t,l}, replaces GELU'(h_t), and each
 * level takes a non-linear step off the residual:
 *   r_{t,1} = e_t = v_t - GELU(h_t)
 *   delta_{t,l} = GELU(p_{t,l} (.) r_{t,l}),   r_{t,l+1} = r_{t,l} - delta_{t,l}
 *   S_t = alpha_t S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T
 *         + sum_{l=1..R} gamma_{t,l} delta_{t,l} u_{t,l}^T,      o_t = S_t q_t
 * Only the token-local injection factors differ from prism_forward.  Arguments as
 * prism_forward_state, with p_gain [B,H,T,R,dv] in the io dtype (16-byte aligned; slot l-1
 * holds level l) in place of eta, which this variant does not have.  With L = 1 it equals
 * prism_forward_state.  It runs on the same path as prism_forward for the plan's shape (the
 * tensor-core kernels for bf16 io with dk = dv = 64 and L <= 4 or dk = dv = 128 and L <= 16,
 * else the portable fp32 kernels): only their prep, which steps the chain level by level, differs.
 */
PRISM_API prism_status prism_forward_nonlinear(prism_plan_t plan, const void *q, const void *k, const void *v,
                                     const float *beta, const float *alpha, const void *u,
                                     const float *gamma, const void *p_gain, const void *conv_w, int L,
                                     const void *v_hist, const float *S_init, void *out, float *S_final,
                                     void *v_hist_out, struct CUstream_st *stream);

/*
 * prism_project -- the block's input projections that produce the recurrence's directions,
 * gains and step gates from the layer input (notes on PRISM, section 2.3, "Input-Anchored
 * Simulation": a short causal convolution over the input gives the anchor; per refinement
 * level, projections of the anchor give the basis k^(l), the gain p^(l) and the gate
 * beta^(l)).  Per batch b and token t:
 *   a_t = sum_{j=0..3} conv_x[j] (.) X_{t-j}     (depthwise, zero before t = 0)
 *   y   = W a_t                                  W [N,D], N = H R dk + H R dv + H R
 *   u_{t,l}     (head h) = the dk entries of basis row block (h, l) of y, divided by their norm
 *                          (0 if the norm is 0)
 *   p_{t,l}     (head h) = the dv entries of gain row block (h, l) of y
 *   gamma_{t,l} (head h) = sigmoid(gate row (h, l) of y)
 * The rows of W are ordered: the basis rows (h, l, c) for c < dk, then the gain rows (h, l, c)
 * for c < dv, then the H R gate rows (h, l).  The outputs are the u, p (prism_forward_nonlinear's
 * gains) and gamma inputs of the recurrence.
 *   X [B,T,D] bf16, conv_x [4,D] bf16, W [N,D] bf16 (inputs)
 *   u [B,H,T,R,dk] bf16, p [B,H,T,R,dv] bf16, gamma [B,H,T,R] float32 (outputs)
 * Sizes B, H, T, dk, dv and R = L - 1 (at least 1) come from the plan, which must have bf16
 * io; D is a multiple of 64.  All pointers are device pointers, 16-byte aligned (gamma: 4).
 * The anchor enters the tensor cores rounded to bf16; products accumulate in fp32.  It is
 * formed once into a scratch buffer owned by the plan (B T D 2 bytes, allocated by the first
 * call that needs it, so make that call before capturing a stream).  Returns once the work is
 * enqueued on `stream`; an expired device-side wait is reported by
 * prism_plan_last_device_status.
 */
PRISM_API prism_status prism_project(prism_plan_t plan, int D, const void *X, const void *conv_x, const void *W,
                                     void *u, void *p, float *gamma, struct CUstream_st *stream);

/*
 * prism_backward -- the cotangents of every input of prism_forward_state (the linear residual
 * chain), given dout = dLoss/d out and optionally dS_final = dLoss/d S_final: reverse-mode
 * differentiation of the definition at the top of this file, token by token backwards.
 * With P = S_{t-1}, y = P k_t and dS_t the cotangent of S_t (dout_t q_t^T included), z = dS_t k_t:
 *   dS_{t-1} = alpha_t (dS_t - beta_t z k_t^T)
 *   dq_t = S_t^T dout_t      dk_t = dS_t^T (beta_t v_t - alpha_t beta_t y) - alpha_t beta_t P^T z
 *   dalpha_t = <dS_t, P> - beta_t y.z      dbeta_t = v_t.z - alpha_t y.z
 *   du_{t,l} = dS_t^T x_{t,l}              dx_{t,l} = dS_t u_{t,l}   (x = the injection factors)
 * and through the residual chain, the gain (GELU''), the residual and the convolution to dv,
 * dgamma, deta and dconv_w.
 * Inputs: q .. L, v_hist and S_init exactly as prism_forward_state (v_hist, S_init may be NULL);
 *   dout      [B,H,T,dv]  float32
 *   dS_final  [B,H,dv,dk] float32 or NULL (zero)
 * Outputs (float32, each with its input's layout, overwritten):
 *   dq, dk [B,H,T,dk]  dv [B,H,T,dv]  dbeta, dalpha [B,H,T]  du [B,H,T,R,dk]  dgamma, deta [B,H,T,R]
 *   (deta[..., R-1] = 0: that gain is never read)  dconv_w [H,4,dv] (summed over the batch)
 *   dv_hist   [B,H,3,dv]  or NULL: the cotangent of the three history slots (also when v_hist is
 *                         NULL, i.e. with respect to the zeros that stand in for them)
 *   dS_init   [B,H,dv,dk] or NULL: the cotangent of the initial state
 * With L = 1, u, gamma, eta, du, dgamma and deta are not touched (dconv_w and dv_hist are 0).
 * dout, dS_final, dq, dk, dv, du, dv_hist and dS_init start on 16-byte boundaries; dbeta,
 * dalpha, dgamma, deta and dconv_w on 4.  No output overlaps another buffer.
 * Two forms compute this.
 *   Chunked (bf16 io, dk = dv = 64, L <= 4; taken unless PRISM_OPT_PATH = 1): the state entering
 *     every 64-token chunk and the cotangent flowing into every chunk's last state come from
 *     chunk-level recurrences S_{c+1} = S_c A_c + B_c and G_{c-1} = G_c A_c^T + Bbar_c whose maps
 *     depend on the chunk's inputs only (notes on PRISM, section 2.1; the transition of section
 *     2.2 is symmetric, so the cotangent runs through A_c^T); every per-token cotangent of a chunk
 *     is then a set of chunk-sized products (tcgen05 tensor cores, fp16 operands, fp32
 *     accumulation), the WY factors of the forward reused.  Workspace: per-chunk maps, states and
 *     factors, O(B H ceil(T/64) dv dk) -- about 0.5 GB for B H T = 131072 tokens of heads of 64.
 *     dalpha_t comes from alpha_t dalpha_t = <G, S'> + a suffix sum over the chunk of per-token
 *     terms of order one, which cancels down to order alpha_t: its rounding error grows like
 *     1 / alpha_t (within 1e-2 of rms for alpha_t >= 0.5; use PRISM_OPT_PATH = 1, the
 *     token-serial form, where gates far below that matter).
 *   Token-serial (every other shape, and PRISM_OPT_PATH = 1): fp32 from the io values, keeping
 *     S_{t-1} and dS_t of every token (2 B H T dv dk floats plus per-token buffers).
 * The workspace is owned by the plan (prism_workspace_bytes reports it) and allocated by the first
 * call of a form, so make that call before capturing a stream.  Returns once the work is enqueued
 * on `stream`; a bounded device wait that runs out is reported by prism_plan_last_device_status.
 */
PRISM_API prism_status prism_backward(prism_plan_t plan, const void *q, const void *k, const void *v,
                                      const float *beta, const float *alpha, const void *u, const float *gamma,
                                      const float *eta, const void *conv_w, int L, const void *v_hist,
                                      const float *S_init, const float *dout, const float *dS_final, float *dq,
                                      float *dk, float *dv, float *dbeta, float *dalpha, float *du, float *dgamma,
                                      float *deta, float *dconv_w, float *dv_hist, float *dS_init,
                                      struct CUstream_st *stream);

/*
 * prism_backward_nonlinear -- the cotangents of every input of prism_forward_nonlinear (the
 * non-linear residual chain of section 2.3 of the notes on PRISM): arguments, layouts, forms and
 * workspace as prism_backward, with the gains p_gain [B,H,T,R,dv] (io dtype, 16-byte aligned) in
 * place of eta and their cotangent dp_gain [B,H,T,R,dv] (float32, 16-byte aligned, overwritten)
 * in place of deta.  Only the token-local chain differs from the linear one; with z = p_{t,l} (.)
 * r_{t,l} and the cotangent of r_{t,R+1} zero, for l = R .. 1:
 *   ddelta = gamma_{t,l} dx_{t,l} - dr_{t,l+1}      dgamma_{t,l} = sum_c GELU(z) dx_{t,l}
 *   dz = ddelta (.) GELU'(z)    dp_{t,l} = dz (.) r_{t,l}    dr_{t,l} = dr_{t,l+1} + dz (.) p_{t,l}
 * then dv_t gains dr_{t,1} and the anchor's cotangent is -GELU'(h_t) (.) dr_{t,1}.  With L = 1,
 * p_gain and dp_gain are not touched (and may be NULL); the call equals prism_backward's.
 */
PRISM_API prism_status prism_backward_nonlinear(prism_plan_t plan, const void *q, const void *k, const void *v,
                                                const float *beta, const float *alpha, const void *u,
                                                const float *gamma, const void *p_gain, const void *conv_w, int L,
                                                const void *v_hist, const float *S_init, const float *dout,
                                                const float *dS_final, float *dq, float *dk, float *dv, float *dbeta,
                                                float *dalpha, float *du, float *dgamma, float *dp_gain,
                                                float *dconv_w, float *dv_hist, float *dS_init,
                                                struct CUstream_st *stream);

/* Free the plan and its workspace.  NULL is accepted. */
PRISM_API prism_status prism_plan_destroy(prism_plan_t plan);

/* Bytes of device workspace the plan holds (informational). */
PRISM_API size_t prism_workspace_bytes(prism_plan_t plan);

/*
 * Read and clear the plan's device status word.  Call after the stream used
 * by the last forward has been synchronised.  Returns PRISM_OK, or
 * PRISM_ERR_TIMEOUT / PRISM_ERR_DEVICE as recorded by the kernels.
 */
PRISM_API prism_status prism_plan_last_device_status(prism_plan_t plan);

/*
 * prism_plan_kernel_times -- per-kernel durations of the last forward.  With
 * PRISM_OPT_TIMING = 1 each forward records a CUDA event pair around every
 * kernel it launches, on the launch stream.  After that stream has been
 * synchronised, this fills up to `max` entries of `out` (which may be NULL
 * when max = 0) and returns the number of kernels the last forward launched,
 * or -1 on error.
 */
PRISM_API int prism_plan_kernel_times(prism_plan_t plan, prism_kernel_time *out, int max);

/* Static description of a status code. */
PRISM_API const char *prism_status_string(prism_status s);

/* One-line description of the last error returned on the calling thread. */
PRISM_API const char *prism_last_error_message(void);

/*
 * prism_forward_noalloc -- the forward for callers that cannot allocate device memory
 * while they run.  The method's pages have no counterpart to this entry point; it is an
 * engineering variant of prism_forward (tensor-core path) that needs no plan.
 *
 * Who needs it: code that runs inside a device-memory allocator or pool hook (a nested
 * cudaMalloc would recurse or deadlock), real-time loops whose memory is reserved up front
 * and must not grow, and hosts that forbid allocation after start-up.  prism_plan
 * allocates workspace; this call allocates nothing.  Its scratch (segment maps, segment
 * start states, a per-chunk stash, a status word) is one fixed array of
 * PRISM_NOALLOC_SCRATCH_BYTES compiled into the library: every GPU that loads the library
 * holds that array until the process exits.
 *
 * Sizes and tensors are those of prism_forward (layouts at the top of this file), with
 * bf16 io and out, dk = dv = 64 and 1 <= L <= 4.  The call uses prism_forward's automatic
 * segment count when its scratch fits (24 KiB per 64-token chunk of all sequences plus
 * 40 KiB per sequence and segment: up to about 170K token-heads); otherwise one segment per
 * sequence, which needs no per-chunk stash (40 KiB per sequence, any length, slower); and it
 * returns PRISM_ERR_UNSUPPORTED (with a message) when even that does not fit -- more than
 * about 1600 sequences (B * H).
 *
 * The first call on each device resolves the array's device address and sets a kernel
 * attribute; make that first call before any stream capture.  All calls share the one
 * array, which keeps the last call's contents: calls that can overlap on the GPU
 * (different streams or host threads) race on it and must be serialised by the caller.
 * With device_status = NULL the call returns once the work is enqueued on `stream`;
 * otherwise it waits for `stream`, stores the device status word (0 = no condition) in
 * *device_status and returns PRISM_ERR_TIMEOUT or PRISM_ERR_DEVICE if one was recorded.
 */
#define PRISM_NOALLOC_SCRATCH_BYTES (64u << 20)
PRISM_API prism_status prism_forward_noalloc(int B, int H, int T, int dk, int dv, int L, const void *q,
                                             const void *k, const void *v, const float *beta,
                                             const float *alpha, const void *u, const float *gamma,
                                             const float *eta, const void *conv_w, void *out,
                                             struct CUstream_st *stream, int *device_status);

/* Version of this library, "major.minor.patch". */
PRISM_API const char *prism_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PRISM_GB300_H */
