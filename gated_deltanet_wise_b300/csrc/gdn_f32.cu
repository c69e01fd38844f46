// gdn_f32.cu — fp32 validation path: the frame-wise GDN forward with fp32
// inputs and fp32 CUDA-core arithmetic, one CTA per (batch, head) chain.
//
// Per frame f (summary page "SANA-WM: Efficient Minute-Scale World Modeling
// with Hybrid Linear Diffusion Transformer", section 方法步骤详情, module 2):
//   A_f = sum_n beta_n k^_n k^_n^T,  U_f = sum_n beta_n v_n k^_n^T,
//   S_f = gamma_f S_{f-1} - S_{f-1} A_f + U_f,   o_{f,n} = S_f q^_n,
// with k^ = k / ||k|| * c and q^ = q / ||q||.  The state, A_f and U_f live in
// shared memory (3 D^2 floats); tokens stream through in blocks of 16.  Any
// 1 <= D <= 128.  This path exists to validate the tensor-core path and the
// method at fp32 accuracy; it is not tuned.
#include <cuda_runtime.h>

#include "gdn_internal.h"

namespace gdn {

constexpr int kF32Threads = 256;
constexpr int kF32TokBlock = 16;
constexpr float kNormEps = 1e-12f;

size_t f32_smem_bytes(int D)
{
    return sizeof(float) * (3 * (size_t)D * D + 2 * (size_t)kF32TokBlock * D + 2 * kF32TokBlock);
}

__global__ void __launch_bounds__(kF32Threads)
    frame_fwd_f32_kernel(const float *__restrict__ q, const float *__restrict__ k, const float *__restrict__ v,
                         const float *__restrict__ beta, const float *__restrict__ gamma, const float *S_in,
                         float *S_out, float *__restrict__ o, int H, int F, int N, int D, float c)
{
    extern __shared__ float sm[];
    const int DD = D * D;
    float *S = sm;
    float *A = S + DD;
    float *U = A + DD;
    float *tb = U + DD;                      // [kF32TokBlock][D] keys (or queries)
    float *vb = tb + kF32TokBlock * D;       // [kF32TokBlock][D] values
    float *w1 = vb + kF32TokBlock * D;       // per-token weight on A (or 1/||q||)
    float *w2 = w1 + kF32TokBlock;           // per-token weight on U
    const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
    const int bh = blockIdx.x, b = bh / H, h = bh % H;
    const size_t FN = (size_t)F * N;

    for (int e = tid; e < DD; e += kF32Threads) S[e] = S_in ? S_in[(size_t)bh * DD + e] : 0.f;
    __syncthreads();

    for (int f = 0; f < F; ++f) {
        for (int e = tid; e < DD; e += kF32Threads) { A[e] = 0.f; U[e] = 0.f; }
        __syncthreads();
        for (int n0 = 0; n0 < N; n0 += kF32TokBlock) {
            const int nt = min(kF32TokBlock, N - n0);
            for (int idx = tid; idx < nt * D; idx += kF32Threads) {
                const int n = idx / D, d = idx % D;
                const size_t g = (((size_t)b * FN + (size_t)f * N + n0 + n) * H + h) * D + d;
                tb[idx] = k[g];
                vb[idx] = v[g];
            }
            __syncthreads();
            for (int n = warp; n < nt; n += kF32Threads / 32) {
                float ss = 0.f;
                for (int d = lane; d < D; d += 32) ss += tb[n * D + d] * tb[n * D + d];
                for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
                if (lane == 0) {
                    const float inv = c / sqrtf(ss + kNormEps);
                    const float bt = beta[((size_t)b * FN + (size_t)f * N + n0 + n) * H + h];
                    w1[n] = bt * inv * inv;
                    w2[n] = bt * inv;
                }
            }
            __syncthreads();
            for (int e = tid; e < DD; e += kF32Threads) {
                const int i = e / D, j = e % D;
                float a = A[e], u = U[e];
                for (int n = 0; n < nt; ++n) {
                    const float kj = tb[n * D + j];
                    a += w1[n] * tb[n * D + i] * kj;
                    u += w2[n] * vb[n * D + i] * kj;
                }
                A[e] = a;
                U[e] = u;
            }
            __syncthreads();
        }
        // S_f = gamma_f S_{f-1} - S_{f-1} A_f + U_f, written over U, then swap.
        const float gf = gamma[((size_t)b * F + f) * H + h];
        for (int e = tid; e < DD; e += kF32Threads) {
            const int i = e / D, j = e % D;
            float s = 0.f;
            for (int l = 0; l < D; ++l) s += S[i * D + l] * A[l * D + j];
            U[e] = gf * S[e] - s + U[e];
        }
        __syncthreads();
        float *t = S;
        S = U;
        U = t;
        // o_{f,n} = S_f q^_n
        for (int n0 = 0; n0 < N; n0 += kF32TokBlock) {
            const int nt = min(kF32TokBlock, N - n0);
            for (int idx = tid; idx < nt * D; idx += kF32Threads) {
                const int n = idx / D, d = idx % D;
                tb[idx] = q[(((size_t)b * FN + (size_t)f * N + n0 + n) * H + h) * D + d];
            }
            __syncthreads();
            for (int n = warp; n < nt; n += kF32Threads / 32) {
                float ss = 0.f;
                for (int d = lane; d < D; d += 32) ss += tb[n * D + d] * tb[n * D + d];
                for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
                if (lane == 0) w1[n] = 1.f / sqrtf(ss + kNormEps);
            }
            __syncthreads();
            for (int idx = tid; idx < nt * D; idx += kF32Threads) {
                const int n = idx / D, i = idx % D;
                float s = 0.f;
                for (int j = 0; j < D; ++j) s += S[i * D + j] * tb[n * D + j];
                o[(((size_t)b * FN + (size_t)f * N + n0 + n) * H + h) * D + i] = s * w1[n];
            }
            __syncthreads();
        }
    }
    if (S_out)
        for (int e = tid; e < DD; e += kF32Threads) S_out[(size_t)bh * DD + e] = S[e];
}

cudaError_t launch_frame_fwd_f32(const float *q, const float *k, const float *v, const float *beta,
                                 const float *gamma, const float *S_in, float *S_out, float *o, int B, int H, int F,
                                 int N, int D, float c, cudaStream_t stream)
{
    const size_t smem = f32_smem_bytes(D);
    cudaError_t e = cudaFuncSetAttribute(frame_fwd_f32_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    frame_fwd_f32_kernel<<<B * H, kF32Threads, smem, stream>>>(q, k, v, beta, gamma, S_in, S_out, o, H, F, N, D, c);
    return cudaGetLastError();
}

// S_out = (prod_f gamma_f) S_in: the whole forward when a frame has no tokens.
__global__ void decay_only_kernel(const float *__restrict__ gamma, const float *S_in, float *S_out, int H, int F,
                                  int D)
{
    const int bh = blockIdx.x, b = bh / H, h = bh % H;
    float g = 1.f;
    for (int f = 0; f < F; ++f) g *= gamma[((size_t)b * F + f) * H + h];
    const size_t DD = (size_t)D * D;
    for (size_t e = threadIdx.x; e < DD; e += blockDim.x) S_out[bh * DD + e] = S_in ? g * S_in[bh * DD + e] : 0.f;
}

cudaError_t launch_decay_only(const float *gamma, const float *S_in, float *S_out, int B, int H, int F, int D,
                              cudaStream_t stream)
{
    decay_only_kernel<<<B * H, 256, 0, stream>>>(gamma, S_in, S_out, H, F, D);
    return cudaGetLastError();
}

}  // namespace gdn
