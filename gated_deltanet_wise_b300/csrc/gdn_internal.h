// gdn_internal.h — declarations shared by the library's translation units
// (never installed, never seen by callers of include/gdn.h).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace gdn {

// fp32 validation path (gdn_f32.cu)
size_t f32_smem_bytes(int D);
cudaError_t launch_frame_fwd_f32(const float *q, const float *k, const float *v, const float *beta,
                                 const float *gamma, const float *S_in, float *S_out, float *o, int B, int H, int F,
                                 int N, int D, float c, cudaStream_t stream);
cudaError_t launch_decay_only(const float *gamma, const float *S_in, float *S_out, int B, int H, int F, int D,
                              cudaStream_t stream);

// Address of the current device's status word (device memory), or nullptr.
unsigned *device_status_word();

// 4-D TMA view (D, H, N, B*F) of a bf16 [B][F*N][H][D] token tensor, 128-byte
// swizzle, boxes of 64 head-dim elements x `rows` tokens (gdn_tc.cu).
bool make_token_map(CUtensorMap *m, const void *base, int B, int H, int F, int N, int rows);
// 2-D view of a bf16 row-major [rows][cols] matrix, 128-byte swizzle, boxes of
// 64 columns x `box_rows` rows (gdn_tc.cu).
bool make_matrix_map(CUtensorMap *m, const void *base, int rows, int cols, int box_rows);
// Same 4-D view of an fp32 token tensor for TMA stores, 64-byte swizzle, boxes
// of 16 head-dim elements x `rows` tokens (gdn_tc.cu).
bool make_f32_row_map(CUtensorMap *m, void *base, int B, int H, int F, int N, int rows);

// Block projections (gdn_proj.cu), tcgen05 GEMMs C = A W^T with bf16 A [M][K]
// and W [N][K]: the plain form (C bf16 [M][N]) and the input projection of the
// GDN block, whose epilogue writes q, k, v (bf16 [M][H*112] each), beta =
// sigmoid(logit) (fp32 [M][H]) and gamma = exp(-softplus(frame mean of the
// decay logit)) (fp32 [B][F][H]).
cudaError_t launch_linear_tc(const void *A, const void *W, void *C, int M, int N, int K, unsigned *status,
                             cudaStream_t stream);
cudaError_t launch_in_proj_tc(const void *x, const void *W_in, void *q, void *k, void *v, float *beta,
                              float *gamma, int B, int H, int F, int N, unsigned *status, cudaStream_t stream);

// tensor-core path (gdn_tc.cu); D == 112.
struct TcPlan {
    int B, H, F, N;
    int chunk;       // frames of the longest chunk (K1 / K2 work unit; chunk_frames gives each range)
    int n_chunks;    // chunks per chain
    size_t ws_bytes; // total workspace
    size_t off_frames, off_comp, off_start;  // workspace sections
    size_t off_flags;                         // chunk-hop flags of the fused chained scan
    // Failure-detection test only: the frame-statistics kernel issues no loads,
    // so its first bounded wait expires and the status word records a timeout.
    int withhold_loads = 0;
};
// force_chunks > 0 fixes the number of frame chunks (1: one chunk per chain,
// whose composite is then the whole range's); 0 lets the plan choose.
bool tc_plan(int B, int H, int F, int N, int force_chunks, TcPlan *plan);
// Per-chain composites (C, H) of all F frames: K1 over the plan's chunks, then the
// chunk composites composed in frame order (the statistics stay in the workspace).
cudaError_t launch_frame_composite_tc(const void *k, const void *v, const float *beta, const float *gamma,
                                      float *C_out, float *H_out, const TcPlan &plan, float c, void *workspace,
                                      unsigned *status, cudaStream_t stream);
// K1b + K2 from statistics a launch_frame_composite_tc call left in the workspace.
cudaError_t launch_fwd_resume_tc(const void *q, const float *gamma, const float *S_in, float *S_out, void *o,
                                 const TcPlan &plan, void *workspace, unsigned *status, cudaStream_t stream);
// S_out = S C + H per chain (S may be null: zero), fp32.
cudaError_t launch_state_compose_tc(const float *S, const float *C, const float *H, float *S_out, int BH,
                                    unsigned *status, cudaStream_t stream);
// The fused chained scan: the forward in one cooperative launch (statistics,
// chunk-boundary hops and scan); cudaErrorCooperativeLaunchTooLarge (nothing
// launched) when the plan's CTAs cannot all be resident.
cudaError_t launch_frame_fwd_fused_tc(const void *q, const void *k, const void *v, const float *beta,
                                      const float *gamma, const float *S_in, float *S_out, void *o, const TcPlan &plan,
                                      float c, int reverse, void *workspace, unsigned *status, cudaStream_t stream);
// reverse = 1 visits the frames from the last to the first (reverse-direction scan).
cudaError_t launch_frame_fwd_tc(const void *q, const void *k, const void *v, const float *beta, const float *gamma,
                                const float *S_in, float *S_out, void *o, const TcPlan &plan, float c, int reverse,
                                void *workspace, unsigned *status, cudaStream_t stream,
                                cudaEvent_t *events = nullptr);

// token-ordered ("product") reading, D == 112: per-frame transitions by the
// UT-transform kernel into the plan's frame workspace and their chunk
// composites (gdn_product.cu), and the whole forward (gdn_tc.cu).
// Workspace of the product reading: the plan's, then the pre-pass's T_off images.
size_t product_ws_T_offset(const TcPlan &plan);
size_t product_ws_bytes(const TcPlan &plan);
cudaError_t launch_frame_product_tc(const void *k, const void *v, const float *beta, const TcPlan &plan, float c,
                                    int reverse, void *workspace, unsigned *status, cudaStream_t stream);
cudaError_t launch_chunk_composite_tc(const float *gamma, const TcPlan &plan, int reverse, void *workspace,
                                      unsigned *status, cudaStream_t stream);
cudaError_t launch_frame_fwd_product_tc(const void *q, const void *k, const void *v, const float *beta,
                                        const float *gamma, const float *S_in, float *S_out, void *o,
                                        const TcPlan &plan, float c, int reverse, void *workspace, unsigned *status,
                                        cudaStream_t stream);

// K1 alone (per-frame statistics into the plan's workspace).
cudaError_t launch_frame_stats_tc(const void *k, const void *v, const float *beta, const float *gamma,
                                  const TcPlan &plan, float c, int reverse, void *workspace, unsigned *status,
                                  cudaStream_t stream, uint8_t *ws_rev = nullptr, int e_mode = 0);
// The state chain alone (K1b + K2 without outputs) over a plan whose workspace
// holds statistics and chunk composites; every state to states (gdn_tc.cu).
cudaError_t launch_states_tc(const void *q, const float *gamma, const float *S_in, float *S_out, float *states,
                             const TcPlan &plan, uint8_t *ws, unsigned *status, cudaStream_t stream);
// backward pass of the sum reading (gdn_bwd.cu); D == 112.
size_t bwd_workspace_bytes(int B, int H, int F, int N);
cudaError_t launch_frame_bwd_tc(const void *q, const void *k, const void *v, const float *beta, const float *gamma,
                                const float *S_in, const void *dO, const float *dS_out, float *dq, float *dk,
                                float *dv, float *dbeta, float *dgamma, float *dS_in, int B, int H, int F, int N,
                                float c, void *workspace, unsigned *status, cudaStream_t stream);

// fused single-frame step (gdn_step.cu); D == 112.
cudaError_t launch_frame_step_tc(const void *q, const void *k, const void *v, const float *beta,
                                 const float *gamma, const float *S_in, float *S_out, void *o, int B, int H, int N,
                                 float c, unsigned *status, cudaStream_t stream);

}  // namespace gdn
