/*
 * gdn.h — C ABI of the B300 (sm_103a) frame-wise Gated DeltaNet forward library
 * (libgdn_b300.so).
 *
 * The operation (summary page "SANA-WM: Efficient Minute-Scale World Modeling
 * with Hybrid Linear Diffusion Transformer", section 方法步骤详情, module 2
 * "Memory-Efficient Long-Context"; section 前置知识 "Gated DeltaNet"):
 * for every chain (b, h) the D x D state is carried across latent frames
 * f = 0..F-1,
 *     k^_n   = k_n / ||k_n||_2 * c_k          (c_k = key_scale, default 1/sqrt(D*N))
 *     q^_n   = q_n / ||q_n||_2
 *     A_f    = sum_n beta_n k^_n k^_n^T,  U_f = sum_n beta_n v_n k^_n^T
 *     S_f    = S_{f-1} (gamma_f I - A_f) + U_f      (= S_{f-1} M_f + U_f)
 *     o_{f,n} = S_f q^_n                             (every token of frame f)
 * with ||x||_2 = sqrt(sum x^2 + 1e-12).  S[i][j]: i = value index (row),
 * j = key index (column).
 *
 * Layouts (all row-major, innermost dimension contiguous):
 *   q, k, v, o : [B][F*N][H][D]   token-major, heads interleaved (bf16 or fp32)
 *   beta       : [B][F*N][H]      fp32
 *   gamma      : [B][F][H]        fp32
 *   S_in/S_out : [B][H][D][D]     fp32
 *
 * Conventions shared by every entry point:
 *   - Memory: the caller owns every buffer.  The library never allocates;
 *     scratch comes from the caller as `workspace` of at least the size the
 *     matching *_workspace_size() returns.  All pointers are device pointers.
 *   - Asynchrony: work is enqueued on `stream` (a cudaStream_t; NULL = legacy
 *     default stream) and the call returns without synchronising.  Argument
 *     errors are detected on the host and returned before anything is
 *     enqueued.  A device-side failure (a bounded wait that expired) is
 *     recorded in a per-device status word, read by gdn_device_status().
 *   - Alignment: q, k, v, o, S_in, S_out and workspace must be 16-byte
 *     aligned; beta and gamma 4-byte aligned.
 *   - Aliasing: S_out may alias S_in; no other buffers may overlap.
 *   - S_in == NULL means a zero initial state; S_out == NULL skips writing the
 *     final state.
 *   - Degenerate sizes: B*H == 0 is a no-op; F == 0 copies S_in (or zeros) to
 *     S_out; N == 0 applies pure decay S_f = gamma_f S_{f-1} and writes no o.
 */
#ifndef GDN_B300_GDN_H
#define GDN_B300_GDN_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    GDN_OK = 0,
    GDN_ERR_INVALID_ARG = 1,  /* null/misaligned pointer, negative size, bad workspace size */
    GDN_ERR_UNSUPPORTED = 2,  /* valid request this build does not implement (e.g. D != 112 on bf16) */
    GDN_ERR_CUDA = 3,         /* a CUDA runtime call failed (no device, launch failure, ...) */
    GDN_ERR_TIMEOUT = 4,      /* a bounded device-side wait expired (see gdn_device_status) */
    GDN_ERR_WORKSPACE = 5     /* workspace pointer missing or smaller than required */
} gdn_status_t;

/* A cudaStream_t, passed through untouched. */
typedef void *gdn_stream_t;

/* Library version, MAJOR*10000 + MINOR*100 + PATCH. */
int gdn_version(void);

/* Static text for a status code (never NULL). */
const char *gdn_status_string(gdn_status_t status);

/*
 * Bytes of device workspace gdn_frame_fwd needs for these sizes (bf16 path).
 * Returns 0 for sizes that need none (degenerate sizes) and (size_t)-1 for
 * invalid sizes.  The layout is private to the library.
 */
size_t gdn_frame_fwd_workspace_size(int B, int H, int F, int N, int D);

/*
 * Frame-wise GDN forward over F frames, bf16 q/k/v/o, fp32 beta/gamma/state.
 * Computes the recurrence above for every (b, h) chain; writes o for every
 * token and the final state S_{F-1} to S_out.
 *   q, k, v   : bf16 [B][F*N][H][D], read only
 *   o         : bf16 [B][F*N][H][D], written
 *   beta      : fp32 [B][F*N][H];  gamma: fp32 [B][F][H]
 *   S_in      : fp32 [B][H][D][D] or NULL;  S_out: fp32 [B][H][D][D] or NULL
 *   key_scale : c_k; <= 0 selects the default 1/sqrt(D*N)
 *   workspace : >= gdn_frame_fwd_workspace_size(B,H,F,N,D) bytes, 16-byte aligned
 * This build implements D == 112 (the model's head size); other D return
 * GDN_ERR_UNSUPPORTED.  Results match the fp64 definition within a relative
 * Frobenius error of 5e-3 on o and S_out for inputs drawn as in the tests.
 */
gdn_status_t gdn_frame_fwd(const void *q, const void *k, const void *v,
                           const float *beta, const float *gamma,
                           const float *S_in, float *S_out, void *o,
                           int B, int H, int F, int N, int D, float key_scale,
                           void *workspace, size_t workspace_bytes,
                           gdn_stream_t stream);

/*
 * Token-ordered ("product") reading of the same layer.  The summary page
 * (section 方法步骤详情, module 2) prints the frame transition as
 * M_f = gamma_f I - K^ beta K^^T and says the layer generalises token-wise
 * Gated DeltaNet (section 技术新颖性).  gdn_frame_fwd reads beta as the
 * diagonal of the frame's token weights (the first-order sum); this entry
 * reads it as the UT-transform matrix, so the frame's tokens act in order:
 *   M_f = gamma_f I - Abar_f,  I - Abar_f = prod_n (I - beta_n k^_n k^_n^T)
 *   U_f = sum_n beta_n v_n k^_n^T (I - beta_{n+1} k^_{n+1} k^_{n+1}^T) ... (I - beta_N k^_N k^_N^T)
 *   S_f = S_{f-1} M_f + U_f,   o = S_f q^ (as gdn_frame_fwd)
 * i.e. within a frame the state follows the delta rule token by token from
 * the frame's start state, and the decay gamma_f is applied once per frame.
 * The two readings differ at order (c_k^2 ||k^||^2)^2 per token pair: at the
 * default key_scale they agree to about 1e-8; with unit keys (key_scale = 1)
 * they differ at first order.  Arguments, layouts, ownership and status codes
 * are those of gdn_frame_fwd; the workspace size has its own query (larger than
 * gdn_frame_fwd's: it also holds the UT transform's T of every 64-token
 * sub-chunk, 8 KB each, formed by a pre-pass over all sub-chunks).  Results
 * match the fp64 definition within 5e-3 relative Frobenius error on o and
 * S_out for inputs drawn as in the tests, key_scale up to 1.
 */
size_t gdn_frame_fwd_product_workspace_size(int B, int H, int F, int N, int D);
gdn_status_t gdn_frame_fwd_product(const void *q, const void *k, const void *v,
                                   const float *beta, const float *gamma,
                                   const float *S_in, float *S_out, void *o,
                                   int B, int H, int F, int N, int D, float key_scale,
                                   void *workspace, size_t workspace_bytes,
                                   gdn_stream_t stream);

/*
 * Forward with options.  `flags` is a bitwise OR of:
 *   GDN_FWD_PRODUCT - the token-ordered reading (as gdn_frame_fwd_product);
 *   GDN_FWD_REVERSE - reverse-direction scan for the bidirectional stage-1
 *     model (summary page, section 局限与改进, compares the stage-1
 *     bidirectional model with the chunk-causal one; the CSDN article's §六
 *     stage 4 derives the streaming variant from the bidirectional model).
 *     The frames are visited from the last to the
 *     first: S_F' = S_in, S_f' = S_{f+1}' M_f + U_f for f = F-1 .. 0 (U_f,
 *     M_f of the chosen reading), o of frame f = S_f' q^, and S_out = S_0'.
 *     This equals gdn_frame_fwd on the frame-reversed sequence with its
 *     outputs put back in frame order.  How the two directions' outputs are
 *     combined is not stated on the pages and is left to the caller.
 *   GDN_FWD_FUSED - the sum reading as one fused chained-scan launch
 *     (statistics, chunk-boundary states and scan/output in one cooperative
 *     grid, one CTA per (frame chunk, chain); each chunk's CTA forms the next
 *     chunk's start state from its own composites, S_start(c+1) =
 *     S_start(c) C_c + H_c, the C_p / H_p prefix of the summary page, section
 *     技术新颖性, and passes it on through a flag in the workspace).  Same
 *     results as the three-launch path up to fp32 rounding of the start states
 *     (bf16 hi + lo products instead of fp32 FMAs).  When the chunks x chains
 *     cannot all be resident at once it runs the three-launch path instead.
 *     With GDN_FWD_PRODUCT: GDN_ERR_UNSUPPORTED ((size_t)-1 from the size
 *     query).
 * flags == 0 is gdn_frame_fwd.  Unknown bits return GDN_ERR_INVALID_ARG (and
 * (size_t)-1 from the size query).  Arguments, layouts, ownership and the
 * other status codes are those of gdn_frame_fwd; the workspace must hold
 * gdn_frame_fwd_ex_workspace_size(B, H, F, N, D, flags) bytes.
 */
#define GDN_FWD_PRODUCT 1u
#define GDN_FWD_REVERSE 2u
#define GDN_FWD_FUSED 4u
size_t gdn_frame_fwd_ex_workspace_size(int B, int H, int F, int N, int D, unsigned flags);
gdn_status_t gdn_frame_fwd_ex(const void *q, const void *k, const void *v,
                              const float *beta, const float *gamma,
                              const float *S_in, float *S_out, void *o,
                              int B, int H, int F, int N, int D, float key_scale,
                              unsigned flags, void *workspace, size_t workspace_bytes,
                              gdn_stream_t stream);

/*
 * Backward pass of gdn_frame_fwd (the sum reading), for training (the CSDN
 * article's §六: the layer is trained end to end).  Given dO = dL/do (bf16,
 * layout of o) and dS_out = dL/dS_out (fp32 [B][H][D][D], NULL: zero), writes
 *   dq, dk, dv : fp32 [B][F*N][H][D]      dbeta  : fp32 [B][F*N][H]
 *   dgamma     : fp32 [B][F][H]           dS_in  : fp32 [B][H][D][D] (may be NULL)
 * for the same q, k, v, beta, gamma, S_in (NULL: zero) and key_scale as the
 * forward.  It recomputes the forward states; nothing from a forward call is
 * kept.  Workspace: gdn_frame_bwd_workspace_size(B,H,F,N,D) bytes, 256-byte
 * aligned (about 1.0 GB for B=1, H=20, F=121, N=880: two statistics
 * workspaces, the per-frame states, the gradient states and their
 * symmetrised products).  F must stay below 65,535 (a grid dimension of the
 * per-frame kernels): larger F returns GDN_ERR_UNSUPPORTED before anything is
 * enqueued, and the size query returns (size_t)-1.  F = 0 copies
 * dS_out to dS_in; N = 0 with F > 0 returns GDN_ERR_UNSUPPORTED; D != 112
 * returns GDN_ERR_UNSUPPORTED.  Gradients match the fp64 chain rule (itself
 * checked against finite differences) within a relative Frobenius error of
 * 5e-3 per tensor for inputs drawn as in the tests.
 */
size_t gdn_frame_bwd_workspace_size(int B, int H, int F, int N, int D);
gdn_status_t gdn_frame_bwd(const void *q, const void *k, const void *v,
                           const float *beta, const float *gamma, const float *S_in,
                           const void *dO, const float *dS_out,
                           float *dq, float *dk, float *dv, float *dbeta, float *dgamma,
                           float *dS_in, int B, int H, int F, int N, int D, float key_scale,
                           void *workspace, size_t workspace_bytes, gdn_stream_t stream);

/*
 * Streaming step: one latent frame (F = 1) per call, state carried by the
 * caller (chunk-causal / autoregressive generation, the chunk-wise variant of
 * the CSDN article's §六 stage 4; resume by passing the previous call's S_out
 * as S_in).  Same layouts with F = 1:
 *   q, k, v, o : bf16 [B][N][H][D];  beta: fp32 [B][N][H];  gamma: fp32 [B][H]
 * One launch: a thread-block cluster per (b, h) chain splits the frame's
 * tokens across its CTAs and sums their partial statistics on chip, so the
 * step needs no scratch: gdn_frame_step_workspace_size() returns 0 for every
 * size this build supports (D == 112) and `workspace` may be NULL.  S_out may
 * alias S_in.  Output equals gdn_frame_fwd run frame by frame on the same
 * S_in, within the tolerance stated there.
 */
size_t gdn_frame_step_workspace_size(int B, int H, int N, int D);
gdn_status_t gdn_frame_step(const void *q, const void *k, const void *v,
                            const float *beta, const float *gamma,
                            const float *S_in, float *S_out, void *o,
                            int B, int H, int N, int D, float key_scale,
                            void *workspace, size_t workspace_bytes,
                            gdn_stream_t stream);

/*
 * Context-parallel building blocks (summary page, section 技术新颖性: a run of
 * frames acts on the state as the affine map S -> S C + H, with the
 * transition composite C = M_{f0} M_{f0+1} ... M_{f1-1} and the input
 * composite H = the state the run reaches from S = 0; composing the runs'
 * maps in frame order reproduces the single-device result exactly).  A rank
 * that owns frames [f0, f1) computes its (C, H), all ranks exchange them, each
 * composes the maps of the ranks before it onto S_in with gdn_state_compose to
 * get its start state, and runs gdn_frame_fwd on its frames from there.
 *
 * gdn_frame_composite: per chain (b, h), (C, H) of the F frames given, same
 * layouts and key_scale as gdn_frame_fwd (frames [0, F) of the arrays passed);
 * C_out, H_out: fp32 [B][H][D][D] (either may be NULL).  Workspace:
 * gdn_frame_composite_workspace_size() bytes (0 for F == 0 or N == 0, where
 * C = (prod gamma) I and H = 0; otherwise the size gdn_frame_fwd needs for the
 * same frames).  Same errors as gdn_frame_fwd.  The call runs the forward's
 * frame-statistics pass over all the frames (every SM busy) and composes the
 * per-chunk composites in frame order; the per-frame statistics stay in the
 * workspace, so that gdn_frame_fwd_resume can finish the forward of the same
 * frames without reading k, v or beta again.
 *
 * gdn_frame_fwd_resume: the rest of gdn_frame_fwd for the frames of the last
 * gdn_frame_composite call on `workspace` (same k, v, beta, gamma, B, H, F, N,
 * D, key_scale; the workspace untouched in between): from S_in (NULL: zero)
 * it writes o for every token and S_out, reading only q and gamma.  In the
 * context-parallel form each rank therefore reads its k and v once.  With any
 * other workspace contents the results are undefined.  Statuses as
 * gdn_frame_fwd (workspace size: gdn_frame_composite_workspace_size()).
 */
size_t gdn_frame_composite_workspace_size(int B, int H, int F, int N, int D);
gdn_status_t gdn_frame_composite(const void *k, const void *v, const float *beta,
                                 const float *gamma, float *C_out, float *H_out,
                                 int B, int H, int F, int N, int D, float key_scale,
                                 void *workspace, size_t workspace_bytes,
                                 gdn_stream_t stream);

gdn_status_t gdn_frame_fwd_resume(const void *q, const float *gamma, const float *S_in, float *S_out,
                                  void *o, int B, int H, int F, int N, int D,
                                  void *workspace, size_t workspace_bytes, gdn_stream_t stream);

/*
 * gdn_state_compose: S_out = S C + Hc for each of BH chains (fp32
 * [BH][D][D], row = value index; S == NULL means S = 0).  S_out may alias S;
 * it must not alias C or Hc.  D == 112 only.  No workspace.
 */
gdn_status_t gdn_state_compose(const float *S, const float *C, const float *Hc, float *S_out,
                               int BH, int D, gdn_stream_t stream);

/*
 * fp32 validation entry: the same operation with fp32 q/k/v/o, computed with
 * fp32 CUDA-core arithmetic (one CTA per chain).  Any 1 <= D <= 128.  Needs no
 * workspace.  Intended for numerical validation (relative error ~1e-6), not
 * for speed.
 */
gdn_status_t gdn_frame_fwd_f32(const float *q, const float *k, const float *v,
                               const float *beta, const float *gamma,
                               const float *S_in, float *S_out, float *o,
                               int B, int H, int F, int N, int D, float key_scale,
                               gdn_stream_t stream);

/*
 * gdn_frame_fwd that also records CUDA events around its internal launches,
 * for per-stage timing.  `events` points to 4 cudaEvent_t created by the
 * caller; they are recorded on `stream` before the frame-statistics kernel,
 * after it, after the chunk-boundary scan and after the output kernel, so that
 * cudaEventElapsedTime(e[i], e[i+1]) is the duration of stage i.  Same
 * arguments, errors and results as gdn_frame_fwd otherwise; `events` may be
 * NULL.  For degenerate sizes no event is recorded.
 */
gdn_status_t gdn_frame_fwd_profiled(const void *q, const void *k, const void *v,
                                    const float *beta, const float *gamma,
                                    const float *S_in, float *S_out, void *o,
                                    int B, int H, int F, int N, int D, float key_scale,
                                    void *workspace, size_t workspace_bytes,
                                    gdn_stream_t stream, void **events);

/*
 * Host-buffer form of gdn_frame_fwd: q/k/v/beta/gamma/S_in are host pointers
 * (pinned memory gives asynchronous copies), o and S_out are host pointers
 * written on completion.  `device_buffer` (caller-owned device memory of
 * gdn_frame_fwd_host_buffer_size() bytes, 256-byte aligned) holds the device
 * copies and the workspace.  S_in may be NULL (zero state); S_out may be NULL.
 * The call enqueues everything and returns; the results are valid after
 * `stream` is synchronised.  Runs of 32 frames or more are pipelined: the
 * frames are cut into up to 8 pieces of at least 16 frames, and piece p's
 * host-to-device copies, piece p-1's forward (on `stream`, continuing from the
 * state the piece before it left) and piece p-2's device-to-host copies run at
 * the same time, the copies on two copy streams the library creates once per
 * device.  The copies start after the work already on `stream`, and `stream`
 * waits for the last copy out.  The pieces re-associate the state sums like
 * split gdn_frame_fwd calls (results agree within the stated tolerance, not
 * bit for bit, with one gdn_frame_fwd call); shorter runs are one piece.  Calls
 * from several host threads are serialised inside the library while they
 * enqueue.
 */
size_t gdn_frame_fwd_host_buffer_size(int B, int H, int F, int N, int D);
gdn_status_t gdn_frame_fwd_host(const void *q, const void *k, const void *v,
                                const float *beta, const float *gamma,
                                const float *S_in, float *S_out, void *o,
                                int B, int H, int F, int N, int D, float key_scale,
                                void *device_buffer, size_t device_buffer_bytes,
                                gdn_stream_t stream);

/*
 * GDN block with its projections (summary page, section 方法步骤详情 module 1:
 * the DiT's GDN blocks have d_model = H * D = 2240, 20 heads of 112).  The
 * pages print no projection shapes; these entries take the plainest block of
 * that width, with nn.Linear-style weights W[out][in] (bf16, row-major):
 *   [q | k | v | a | g] = x W_in^T            W_in : [3*H*D + 2*H][H*D]
 *   beta_{n,h}  = sigmoid(a_{n,h})             (per token and head)
 *   gamma_{f,h} = exp(-softplus(mean_{n in frame f} g_{n,h}))   (per frame and head)
 *   (o, S_out)  = gdn_frame_fwd(q, k, v, beta, gamma, S_in)
 *   y           = o W_out^T                    W_out: [H*D][H*D]
 * x and y are bf16 [B][F*N][H*D] (the token-major layout whose [H][D] view is
 * the layer's q/k/v/o layout).  q, k, v are rounded to bf16 as the layer's
 * inputs; the gates stay fp32.  The input projection is one tcgen05 GEMM whose
 * epilogue writes q, k, v, beta and the per-frame decay-logit sums directly
 * (no activation or re-layout pass over memory); a small kernel turns the sums
 * into gamma.  The output projection is the same GEMM with a plain bf16
 * epilogue.  D == 112 only (GDN_ERR_UNSUPPORTED otherwise); N == 0 with F > 0
 * returns GDN_ERR_UNSUPPORTED (the frame mean needs tokens).  All pointers are
 * device pointers, 16-byte aligned (beta, gamma: 4).  Results match the fp64
 * definition (x W^T in fp64, q/k/v rounded to bf16 as the layer's inputs)
 * within a relative Frobenius error of 5e-3 on y and S_out for inputs drawn
 * as in the tests.
 *
 * gdn_block_in_proj : x -> q, k, v (bf16 [B][F*N][H][D]), beta (fp32
 *                     [B][F*N][H]), gamma (fp32 [B][F][H]); no workspace.
 * gdn_block_out_proj: o (bf16 [B][F*N][H*D]) -> y; no workspace.
 * gdn_block_fwd     : the whole block; workspace of
 *                     gdn_block_fwd_workspace_size() bytes, 256-byte aligned
 *                     (holds q, k, v, o, beta, gamma and the forward's
 *                     workspace).  S_in may be NULL (zero state), S_out NULL.
 */
gdn_status_t gdn_block_in_proj(const void *x, const void *W_in, void *q, void *k, void *v,
                               float *beta, float *gamma,
                               int B, int H, int F, int N, int D, gdn_stream_t stream);
gdn_status_t gdn_block_out_proj(const void *o, const void *W_out, void *y,
                                int B, int H, int F, int N, int D, gdn_stream_t stream);
size_t gdn_block_fwd_workspace_size(int B, int H, int F, int N, int D);
gdn_status_t gdn_block_fwd(const void *x, const void *W_in, const void *W_out,
                           const float *S_in, float *S_out, void *y,
                           int B, int H, int F, int N, int D, float key_scale,
                           void *workspace, size_t workspace_bytes, gdn_stream_t stream);

/*
 * Streaming step without caller-supplied scratch.  The paper has no
 * counterpart: this is a library convenience.  Same arguments, layouts and
 * results as gdn_frame_step, minus the workspace.
 *
 * It is for callers that cannot allocate device memory where they run a
 * frame.  Examples: a host that owns the whole device memory budget and hands
 * plug-ins only input and output pointers; a per-frame real-time loop that
 * must not take the allocator's locks or latency; code inside a stream capture
 * in which allocation calls are prohibited.  It runs the frame through the
 * multi-frame kernels of gdn_frame_fwd with F = 1, whose per-frame statistics
 * and chunk composites need scratch; that scratch is a fixed 16 MiB device
 * array inside the library (gdn_frame_step_noalloc_limit_bytes()).  Every GPU
 * that loads the library holds it until the process exits.
 *   - Limit: gdn_frame_fwd_workspace_size(B, H, 1, N, D) must not exceed the
 *     array (about 226 KiB per chain at D = 112, so B*H <= 72).  Larger
 *     requests return GDN_ERR_WORKSPACE before anything is enqueued.
 *   - Status codes: for every argument list the call returns what
 *     gdn_frame_fwd (F = 1) returns when given a workspace of the array's
 *     size, checked in the same order (negative sizes, then D, then
 *     pointers, then the size plan, then the scratch limit).
 *   - It calls no cudaMalloc, cudaFree or other allocating routine.
 *   - Set-up: the first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current.  Make that first call
 *     before any stream capture.
 *   - Sharing: all calls on a device share the one array, which keeps the last
 *     call's contents.  No part of it needs to start at zero, because every
 *     byte a call reads is written earlier in the same call.  Calls that
 *     overlap on the GPU (other streams, other host threads) race on it and
 *     corrupt each other's results: serialise them.
 */
size_t gdn_frame_step_noalloc_limit_bytes(void);
gdn_status_t gdn_frame_step_noalloc(const void *q, const void *k, const void *v,
                                    const float *beta, const float *gamma,
                                    const float *S_in, float *S_out, void *o,
                                    int B, int H, int N, int D, float key_scale,
                                    gdn_stream_t stream);

/*
 * Failure-detection test entry: gdn_frame_fwd (sum reading, same arguments,
 * checks and status codes) with the frame-statistics kernel told to issue no
 * loads.  Its consumers' bounded waits on the first pipeline stage then run
 * out (after about 2 s of GPU time: the wait limit is ~4e9 SM cycles), the
 * kernel sets its abort flag, lets every role leave its loop, frees its tensor
 * memory and exits; no fault, trap or unbounded wait is involved.  The
 * following kernels of the call still run (on undefined statistics), so o and
 * S_out are undefined, and gdn_device_status() afterwards returns
 * GDN_ERR_TIMEOUT.  The context stays usable: later calls behave normally.
 * There is no counterpart on the pages; it exists so that tests can exercise
 * the timeout path end to end.
 */
gdn_status_t gdn_test_frame_fwd_expired_wait(const void *q, const void *k, const void *v,
                                             const float *beta, const float *gamma,
                                             const float *S_in, float *S_out, void *o,
                                             int B, int H, int F, int N, int D, float key_scale,
                                             void *workspace, size_t workspace_bytes,
                                             gdn_stream_t stream);

/*
 * Synchronises `stream`, then returns and clears the current device's status
 * word: GDN_OK, or GDN_ERR_TIMEOUT if a kernel's bounded wait expired since the
 * last call (that launch's outputs are then undefined).
 */
gdn_status_t gdn_device_status(gdn_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* GDN_B300_GDN_H */
