// gdn_proj.cu — the GDN block's input and output projections around the layer,
// with the gate activations and the q/k/v layout fused into the projection
// GEMM's epilogue.
//
// Summary page "SANA-WM: Efficient Minute-Scale World Modeling with Hybrid
// Linear Diffusion Transformer", section 方法步骤详情 module 1: the GDN blocks of
// the DiT have d_model = 2240 = 20 heads x 112.  The pages give no projection
// shapes; the block here is the plainest one with that width:
//     [q | k | v | a | g] = x W_in^T      (W_in: [3 H D + 2 H] x [H D])
//     beta_{n,h} = sigmoid(a_{n,h}),  gamma_{f,h} = exp(-softplus(mean_{n in f} g_{n,h}))
//     (o, S_out) = frame-wise GDN(q, k, v, beta, gamma, S_in)
//     y = o W_out^T                      (W_out: [H D] x [H D])
// One tcgen05 GEMM kernel serves both projections: C = A B^T with A [M][K]
// and B [N][K] bf16 (K-major, the nn.Linear weight layout), fp32 accumulation
// in tensor memory.  Its epilogue either stores C as bf16 (output projection)
// or splits the columns of the input projection into the q, k, v tensors in
// the layer's token-major layout, the write strengths beta (fp32), and
// per-(frame, head) sums of the decay logits; a small kernel then turns the
// sums into gamma.  No activation or re-layout pass touches memory in between.
//
// Kernel: persistent, one CTA per SM, 128 x 256 output tiles, K in blocks of
// 64 (one 128-byte swizzled row of A and B per token / output feature), four
// stages of TMA loads; warp 0 issues the loads, warp 1 the MMAs (M = 128,
// N = 256, K = 16 each), warps 2..9 drain the accumulator (two TMEM
// accumulators of 256 columns, so the epilogue of one tile overlaps the main
// loop of the next).
#include <cuda.h>
#include <cuda_runtime.h>
#include <math.h>

#include "gdn_internal.h"
#include "gdn_tile.cuh"

namespace gdn {

constexpr int kGBM = 128, kGBN = 256, kGBK = 64;
constexpr int kGStages = 4;
constexpr uint32_t kGABytes = kGBM * kRowB;              // 16384: A block (128 rows x 64 K)
constexpr uint32_t kGBBytes = kGBN * kRowB;              // 32768: B block (256 rows x 64 K)
constexpr uint32_t kGStageBytes = kGABytes + kGBBytes;   // 49152
constexpr uint32_t kGOffBar = kGStages * kGStageBytes;   // 196608
constexpr uint32_t kGSmem = kGOffBar + 256 + 1024;
constexpr int kGThreads = 320;                           // producer, MMA, 8 epilogue warps
constexpr uint32_t kGIdesc = idesc_bf16(kGBM, kGBN, false, false);
static_assert(kGSmem <= kMaxSmem, "projection GEMM shared memory");

struct GemmParams {
    int M, N, K;
    int mode;           // 0: C bf16 [M][N];  1: input projection epilogue
    void *C;            // mode 0
    void *q, *k, *v;    // mode 1: bf16 [M][HD] each
    float *beta;        // mode 1: fp32 [M][H]
    float *gsum;        // mode 1: fp32 [B][F][H], decay-logit sums per frame (zeroed by the caller)
    int H, HD, FN, Nf;  // mode 1: heads, H*D, tokens per batch item (F*N), tokens per frame
    unsigned *status;
};

__device__ __forceinline__ float sigmoid_f(float x) { return 1.f / (1.f + __expf(-x)); }

// Named barrier over the eight epilogue warps (id 0 is __syncthreads).
__device__ __forceinline__ void epi_sync() { asm volatile("bar.sync 3, 256;" ::: "memory"); }

__global__ void __launch_bounds__(kGThreads, 1)
    gdn_proj_gemm_kernel(const __grid_constant__ CUtensorMap mapA, const __grid_constant__ CUtensorMap mapB,
                         const GemmParams p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + kGOffBar);
    uint64_t *full = bars, *empty = bars + kGStages, *acc_full = bars + 2 * kGStages, *acc_empty = acc_full + 2;
    uint64_t *drain = acc_full + 4;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(acc_full + 5);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(acc_full + 6);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_m = (p.M + kGBM - 1) / kGBM, n_n = (p.N + kGBN - 1) / kGBN;
    const int n_tiles = n_m * n_n, n_kb = (p.K + kGBK - 1) / kGBK;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kGStages; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&acc_full[i], 1);
            mbar_init(&acc_empty[i], 8);
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t sbase = smem_u32(sm);
    griddep_launch_dependents();
    griddep_wait();

    if (warp == 0) {
        // ------------------------------------------------------ TMA producer
        if (lane == 0) {
            int it = 0;
            bool ok = true;
            for (int tile = blockIdx.x; tile < n_tiles && ok; tile += gridDim.x) {
                const int tm = tile / n_n, tn = tile % n_n;
                for (int kb = 0; kb < n_kb; ++kb, ++it) {
                    const int s = it % kGStages, use = it / kGStages;
                    if (use >= 1 && !(ok = mbar_wait(&empty[s], (use - 1) & 1, abort_flag))) break;
                    uint8_t *st = sm + s * kGStageBytes;
                    mbar_arrive_expect_tx(&full[s], kGStageBytes);
                    tma_load_2d(st, &mapA, &full[s], kb * kGBK, tm * kGBM);
                    tma_load_2d(st + kGABytes, &mapB, &full[s], kb * kGBK, tn * kGBN);
                }
            }
            if (*abort_flag)  // let loads in flight land before the CTA exits
                for (int s = 0; s < kGStages && s < it; ++s)
                    mbar_wait_drain(&full[s], ((it - 1 - s) / kGStages) & 1);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------- MMA issuer
        if (lane == 0) {
            int it = 0, tc = 0;
            bool ok = true;
            for (int tile = blockIdx.x; tile < n_tiles && ok; tile += gridDim.x, ++tc) {
                const int acc = tc & 1, use = tc >> 1;
                if (use >= 1 && !(ok = mbar_wait(&acc_empty[acc], (use - 1) & 1, abort_flag))) break;
                tc_fence_after();
                const uint32_t d = tmem + acc * kGBN;
                for (int kb = 0; kb < n_kb; ++kb, ++it) {
                    const int s = it % kGStages;
                    if (!(ok = mbar_wait(&full[s], (it / kGStages) & 1, abort_flag))) break;
                    tc_fence_after();
                    const uint32_t a = sbase + s * kGStageBytes, b = a + kGABytes;
#pragma unroll
                    for (int ks = 0; ks < kGBK / 16; ++ks)
                        mma_bf16(d, sdesc_sw128(a + ks * 32, 16, 1024), sdesc_sw128(b + ks * 32, 16, 1024), kGIdesc,
                                 (kb > 0 || ks > 0) ? 1u : 0u);
                    mma_commit(&empty[s]);
                }
                if (ok) mma_commit(&acc_full[acc]);
            }
            mma_commit(drain);
            mbar_wait_drain(drain, 0);
        }
    } else {
        // ------------------------------------------------- epilogue warps
        // Warp quadrant = TMEM lanes (output rows), two warps per quadrant take
        // the two 128-column halves of the tile; thread = one output row.
        const int quad = warp & 3, half = (warp - 2) >> 2;
        const int row = quad * 32 + lane;
        const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
        int tc = 0;
        bool ok = true;
        for (int tile = blockIdx.x; tile < n_tiles; tile += gridDim.x, ++tc) {
            const int acc = tc & 1, use = tc >> 1;
            const int tm = tile / n_n, tn = tile % n_n;
            if (ok) ok = mbar_wait_warp(&acc_full[acc], use & 1, abort_flag);
            tc_fence_after();
            const int m = tm * kGBM + row;
            if (ok) {
#pragma unroll 1
                for (int cc = 0; cc < 8; ++cc) {
                    const int col = half * 128 + cc * 16;  // column inside the tile
                    const int n0 = tn * kGBN + col;          // output column of this 16-column chunk
                    uint32_t r[16];
                    tmem_ld16(tmem + lane_off + acc * kGBN + col, r);
                    tmem_ld_wait();
                    if (m >= p.M || n0 >= p.N) continue;
                    float x[16];
#pragma unroll
                    for (int j = 0; j < 16; ++j) x[j] = __uint_as_float(r[j]);
                    if (p.mode == 0) {
                        uint4 *dst = reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(p.C) + (size_t)m * p.N + n0);
                        if (n0 + 16 <= p.N) {
                            dst[0] = f32x8_to_bf16(x);
                            dst[1] = f32x8_to_bf16(x + 8);
                        } else {
                            __nv_bfloat16 *e = static_cast<__nv_bfloat16 *>(p.C) + (size_t)m * p.N;
                            for (int j = 0; j < 16 && n0 + j < p.N; ++j) e[n0 + j] = __float2bfloat16_rn(x[j]);
                        }
                    } else if (n0 < 3 * p.HD) {
                        // q | k | v: HD is a multiple of 16, so a chunk lies inside one of them
                        const int which = n0 / p.HD, c = n0 - which * p.HD;
                        void *base = which == 0 ? p.q : which == 1 ? p.k : p.v;
                        uint4 *dst = reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(base) + (size_t)m * p.HD + c);
                        dst[0] = f32x8_to_bf16(x);
                        dst[1] = f32x8_to_bf16(x + 8);
                    } else {
                        // gate logits: columns 3HD .. 3HD + H are a (write strength), the next H are g (decay)
                        const int b = m / p.FN, f = (m - b * p.FN) / p.Nf;
                        const int F = p.FN / p.Nf;
                        for (int j = 0; j < 16; ++j) {
                            const int c = n0 + j - 3 * p.HD;
                            if (c >= 2 * p.H) break;
                            if (c < p.H) p.beta[(size_t)m * p.H + c] = sigmoid_f(x[j]);
                            else atomicAdd(p.gsum + ((size_t)b * F + f) * p.H + (c - p.H), x[j]);
                        }
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acc_empty[acc]);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (*abort_flag && threadIdx.x == 0) raise_status(p.status);
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// gamma_{b,f,h} = exp(-softplus(gsum / N)) = 1 / (1 + exp(mean logit)), in place.
__global__ void gdn_gamma_from_logits_kernel(float *g, int count, float inv_n)
{
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < count) g[i] = 1.f / (1.f + expf(g[i] * inv_n));
}

namespace {
constexpr int kMaxDevProj = 64;
bool g_proj_attr[kMaxDevProj];

cudaError_t prepare_proj()
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevProj) return cudaErrorInvalidDevice;
    if (g_proj_attr[dev]) return cudaSuccess;
    e = cudaFuncSetAttribute(gdn_proj_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kGSmem);
    if (e == cudaSuccess) g_proj_attr[dev] = true;
    return e;
}

cudaError_t launch_gemm(const void *A, const void *Bw, const GemmParams &p, cudaStream_t stream)
{
    CUtensorMap ma, mb;
    if (!make_matrix_map(&ma, A, p.M, p.K, kGBM) || !make_matrix_map(&mb, Bw, p.N, p.K, kGBN))
        return cudaErrorInvalidValue;
    cudaError_t e = prepare_proj();
    if (e != cudaSuccess) return e;
    const int tiles = ((p.M + kGBM - 1) / kGBM) * ((p.N + kGBN - 1) / kGBN);
    const int grid = tiles < kSms ? tiles : kSms;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kGThreads);
    cfg.dynamicSmemBytes = kGSmem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, gdn_proj_gemm_kernel, ma, mb, p);
}
}  // namespace

cudaError_t launch_linear_tc(const void *A, const void *W, void *C, int M, int N, int K, unsigned *status,
                             cudaStream_t stream)
{
    GemmParams p = {};
    p.M = M;
    p.N = N;
    p.K = K;
    p.mode = 0;
    p.C = C;
    p.status = status;
    return launch_gemm(A, W, p, stream);
}

cudaError_t launch_in_proj_tc(const void *x, const void *W_in, void *q, void *k, void *v, float *beta,
                              float *gamma, int B, int H, int F, int N, unsigned *status, cudaStream_t stream)
{
    const int HD = H * kD;
    GemmParams p = {};
    p.M = B * F * N;
    p.N = 3 * HD + 2 * H;
    p.K = HD;
    p.mode = 1;
    p.q = q;
    p.k = k;
    p.v = v;
    p.beta = beta;
    p.gsum = gamma;
    p.H = H;
    p.HD = HD;
    p.FN = F * N;
    p.Nf = N;
    p.status = status;
    const size_t ng = (size_t)B * F * H;
    cudaError_t e = cudaMemsetAsync(gamma, 0, ng * sizeof(float), stream);
    if (e != cudaSuccess) return e;
    if ((e = launch_gemm(x, W_in, p, stream)) != cudaSuccess) return e;
    gdn_gamma_from_logits_kernel<<<(unsigned)((ng + 255) / 256), 256, 0, stream>>>(gamma, (int)ng, 1.f / (float)N);
    return cudaGetLastError();
}

}  // namespace gdn
