// gdn_bwd.cu — backward pass of the frame-wise GDN (sum reading), D = 112.
//
// Forward (summary page "SANA-WM: Efficient Minute-Scale World Modeling with
// Hybrid Linear Diffusion Transformer", 方法步骤详情 module 2):
//   k^ = c k / r, q^ = q / rho,  A_f = sum beta k^ k^^T,  U_f = sum beta v k^^T,
//   S_f = S_{f-1} (gamma_f I - A_f) + U_f,  o = S_f q^.
// Given dO = dL/do and dS_out = dL/dS_out the chain rule gives, per chain:
//   G_f = dL/dS_f:  G_{F-1} = dS_out + E_{F-1},  G_{f-1} = G_f M_f + E_{f-1}
//                   (M_f is symmetric),  E_f = sum_{n in f} do_n q^_n^T,  dS_in = G_0 M_0
//   dM_f = S_{f-1}^T G_f,  dgamma_f = trace(dM_f),  dA_f = -dM_f
//   dq^_n = S_f^T do_n,  dk^_n = beta ((dA + dA^T) k^ + G^T v),  dv_n = beta G k^,
//   dbeta_n = k^^T dA k^ + v^T G k^,  then through the two normalisations.
//
// The path reuses the forward kernels and adds three:
//   1. K1 on (k, v): A_f images, U_f and chunk composites in a workspace; the
//      chunk-boundary kernel and the scan kernel without outputs, from S_in,
//      store every S_f.
//   2. K1 on (k := q, v := dO, beta := 1, c := 1): its U_f slots are E_f.
//   3. kb_build_reverse_ws lays out the reverse scan: slot p holds A of frame
//      F - p (none for p = 0) and E_{F-1-p} (none for p = F), gamma likewise;
//      its chunk composites (K1c), the chunk-boundary kernel and the scan
//      kernel without outputs, from dS_out, visit G_{F-1}, ..., G_0 and end at
//      dS_in.
//   4. kb_frame_grad: dM_f = S_{f-1}^T G_f (fp32 CUDA cores), dgamma_f, and
//      Dsym_f = dA_f + dA_f^T.
//   5. kg_token_grad_kernel (tcgen05), twice: dO S_f, with q's normalisation
//      Jacobian in the epilogue, gives dq; k Dsym_f, v G_f and k G_f^T (one G
//      image read K-major and MN-major), with k's, give dk, dv and dbeta.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "gdn_internal.h"
#include "gdn_tile.cuh"

namespace gdn {

namespace {
size_t up256(size_t x) { return (x + 255) / 256 * 256; }
}  // namespace

// ------------------------------------------------------------------ helpers
__global__ void kb_fill(float *p, size_t n, float value)
{
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x)
        p[i] = value;
}

// Reverse-scan workspace, one block per (chain, slot p = 0..F).
__global__ void kb_build_reverse_ws(const uint8_t *ws_fwd, const uint8_t *ws_E, uint8_t *ws_G, const float *gamma,
                                    float *gamma_G, int B, int H, int F)
{
    const int bh = blockIdx.x, p = blockIdx.y;
    const int b = bh / H, h = bh % H;
    uint4 *dst = reinterpret_cast<uint4 *>(ws_G + ((size_t)bh * (F + 1) + p) * kFrameWs);
    const uint4 *srcA = p >= 1 ? reinterpret_cast<const uint4 *>(ws_fwd + ((size_t)bh * F + (F - p)) * kFrameWs)
                               : nullptr;
    const uint4 *srcU =
        p <= F - 1 ? reinterpret_cast<const uint4 *>(ws_E + ((size_t)bh * F + (F - 1 - p)) * kFrameWs + kAimgBytes)
                   : nullptr;
    constexpr int nA = kAimgBytes / 16, nU = kUBytes / 16;
    for (int i = threadIdx.x; i < nA; i += blockDim.x) dst[i] = srcA ? srcA[i] : make_uint4(0, 0, 0, 0);
    for (int i = threadIdx.x; i < nU; i += blockDim.x) dst[nA + i] = srcU ? srcU[i] : make_uint4(0, 0, 0, 0);
    if (threadIdx.x == 0)
        gamma_G[((size_t)b * (F + 1) + p) * H + h] = p >= 1 ? gamma[((size_t)b * F + (F - p)) * H + h] : 1.f;
}

// dM = S_{f-1}^T G_f, dgamma_f = trace(dM), Dsym_f = -(dM + dM^T).  One block of
// 256 threads per (chain, frame); thread (ty, tx) owns the 7 x 7 block of rows
// 7 ty.., columns 7 tx...
constexpr uint32_t kFgSmem = 2 * (uint32_t)kStateBytes + 16;
__global__ void __launch_bounds__(256) kb_frame_grad(const float *S_in, const float *Sst, const float *Gst,
                                                     float *dgamma, float *Dsym, int B, int H, int F)
{
    extern __shared__ __align__(16) float fg_smem[];
    float *Sp = fg_smem, *Gf = fg_smem + kStateFloats;
    float *tr = fg_smem + 2 * kStateFloats;
    const int bh = blockIdx.x, f = blockIdx.y;
    const int b = bh / H, h = bh % H;
    const float *sp = f == 0 ? (S_in ? S_in + (size_t)bh * kStateFloats : nullptr)
                             : Sst + ((size_t)bh * F + f - 1) * kStateFloats;
    const float *gf = Gst + ((size_t)bh * (F + 1) + (F - 1 - f)) * kStateFloats;
    for (int e = threadIdx.x; e < (int)kStateFloats / 4; e += 256) {
        reinterpret_cast<float4 *>(Sp)[e] = sp ? reinterpret_cast<const float4 *>(sp)[e] : make_float4(0, 0, 0, 0);
        reinterpret_cast<float4 *>(Gf)[e] = reinterpret_cast<const float4 *>(gf)[e];
    }
    if (threadIdx.x == 0) *tr = 0.f;
    __syncthreads();
    const int ty = threadIdx.x >> 4, tx = threadIdx.x & 15;
    const int i0 = ty * 7, j0 = tx * 7;
    float acc[7][7];
#pragma unroll
    for (int a = 0; a < 7; ++a)
#pragma unroll
        for (int c = 0; c < 7; ++c) acc[a][c] = 0.f;
    for (int l = 0; l < kD; ++l) {
        float sv[7], gv[7];
#pragma unroll
        for (int a = 0; a < 7; ++a) {
            sv[a] = Sp[l * kD + i0 + a];
            gv[a] = Gf[l * kD + j0 + a];
        }
#pragma unroll
        for (int a = 0; a < 7; ++a)
#pragma unroll
            for (int c = 0; c < 7; ++c) acc[a][c] = fmaf(sv[a], gv[c], acc[a][c]);
    }
    __syncthreads();  // Sp is reused for dM
#pragma unroll
    for (int a = 0; a < 7; ++a)
#pragma unroll
        for (int c = 0; c < 7; ++c) Sp[(i0 + a) * kD + j0 + c] = acc[a][c];
    if (ty == tx) {
        float d = 0.f;
#pragma unroll
        for (int a = 0; a < 7; ++a) d += acc[a][a];
        atomicAdd(tr, d);
    }
    __syncthreads();
    float *ds = Dsym + ((size_t)bh * F + f) * kStateFloats;
#pragma unroll
    for (int a = 0; a < 7; ++a)
#pragma unroll
        for (int c = 0; c < 7; ++c) {
            const int i = i0 + a, j = j0 + c;
            ds[i * kD + j] = -(Sp[i * kD + j] + Sp[j * kD + i]);
        }
    if (threadIdx.x == 0) dgamma[((size_t)b * F + f) * H + h] = *tr;
}

// ------------------------------------------------ token-row gradient kernels
// One CTA per (frame, chain), 128-token tiles of the frame's rows through TMA
// into tcgen05 GEMMs against per-frame fp32 matrices given as hi + lo bf16
// images (image row j = column j of the matrix, K-major); the epilogue (thread
// = token row) applies the chain rule through the normalisations and writes
// the final fp32 gradients.
//   kMode 0: acc = dO W (W = S_f)  ->  dq^ = S_f^T do;  dq = (dq^ - q (q.dq^)/rho^2) / rho
//            two stages of (dO, q) tiles, two accumulator slots.
//   kMode 1: acc0 = k Dsym, acc1 = v G, acc2 = k G^T (the G image read MN-major:
//            row j, column i holds G[i][j], which is B[n = i][k = j] = G[i][j]);
//            with k^ = (c/r) k: dk^ = beta ((c/r) acc0 + acc1),
//            dk = (c/r)(dk^ - k (k.dk^)/r^2),  dv = beta (c/r) acc2,
//            dbeta = 1/2 (c/r)^2 k.acc0 + (c/r) k.acc1;  one stage of (k, v).
constexpr int kGThreads = 320;                    // producer, MMA, 4 image warps, 4 output warps
constexpr uint32_t kGOffImg = 0;  // W0 hi, W0 lo (, W1 hi, W1 lo), 32 KB each; then the (x0, x1) tile stages
// mode 0: 2 images + 2 stages x 2 tiles; mode 1: 4 images + 1 stage x 2 tiles: both 196,608 B
constexpr uint32_t kGOffBar = 6 * kImgBytes;
constexpr uint32_t kGSmem = kGOffBar + 256 + 1024;
static_assert(kGSmem <= kMaxSmem, "token-gradient kernel shared memory");
constexpr uint32_t kIdescKMN = idesc_bf16(128, kD, false, true);

struct TokGradParams {
    const float *W0, *W1;   // mode 0: S states [BH][F]; mode 1: Dsym [BH][F], G states [BH][F+1] (G_f at F-1-f)
    const float *beta;
    float *g0, *g1, *g_beta;  // mode 0: dq; mode 1: dk, dv, dbeta
    unsigned *status;
    int B, H, F, N;
    float c;
};

template <int kMode>
__global__ void __launch_bounds__(kGThreads, 1)
    kg_token_grad_kernel(const __grid_constant__ CUtensorMap mapX0, const __grid_constant__ CUtensorMap mapX1,
                         const TokGradParams p)
{
    constexpr int kStages = kMode == 0 ? 2 : 1;
    constexpr int kAcc = kMode == 0 ? 1 : 3;       // accumulators per tile
    constexpr uint32_t kOffBar = kGOffBar;
    constexpr uint32_t kOffX = kMode == 0 ? 2 * kImgBytes : 4 * kImgBytes;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + kOffBar);
    uint64_t *x_full = bars + 0, *x_empty = bars + 2, *acc_full = bars + 4, *acc_free = bars + 6;
    uint64_t *img_ready = bars + 8, *drain = bars + 9;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 10);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(bars + 11);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int BH = p.B * p.H;
    const int f = blockIdx.x / BH, bh = blockIdx.x % BH;
    const int b = bh / p.H, h = bh % p.H;
    const int bf = b * p.F + f;
    const int n_tiles = (p.N + 127) / 128;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&x_full[i], 1);
            mbar_init(&x_empty[i], 5);  // the tile's MMAs + the four output warps (epilogue reads x1 / x0)
            mbar_init(&acc_full[i], 1);
            mbar_init(&acc_free[i], 4);
        }
        mbar_init(img_ready, 4);
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
    auto xtile = [&](int s, int which) { return kOffX + (uint32_t)(2 * s + which) * kImgBytes; };

    if (warp == 0) {
        if (lane == 0) {
            const uint64_t pol = policy_evict_first();
            int issued = 0;
            for (int t = 0; t < n_tiles; ++t) {
                const int s = t % kStages, u = t / kStages;
                if (u >= 1 && !mbar_wait(&x_empty[s], (u - 1) & 1, abort_flag)) break;
                mbar_arrive_expect_tx(&x_full[s], 2 * kImgBytes);
                for (int w = 0; w < 2; ++w) {
                    uint8_t *dst = sm + xtile(s, w);
                    const CUtensorMap *m = w ? &mapX1 : &mapX0;
                    tma_load_4d(dst, m, &x_full[s], 0, h, t * 128, bf, pol);
                    tma_load_4d(dst + kImgPanel, m, &x_full[s], 64, h, t * 128, bf, pol);
                }
                ++issued;
            }
            if (*abort_flag)
                for (int s = 0; s < kStages && s < issued; ++s) {
                    const int last = ((issued - 1 - s) / kStages) * kStages + s;
                    mbar_wait_drain(&x_full[s], (last / kStages) & 1);
                }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            bool ok = mbar_wait(img_ready, 0, abort_flag);
            tc_fence_after();
            for (int t = 0; t < n_tiles && ok; ++t) {
                const int s = t % kStages, u = t / kStages;
                if (!(ok = mbar_wait(&x_full[s], u & 1, abort_flag))) break;
                if (u >= 1 && !(ok = mbar_wait(&acc_free[s], (u - 1) & 1, abort_flag))) break;
                tc_fence_after();
                const uint32_t x0 = sbase + xtile(s, 0), x1 = sbase + xtile(s, 1);
                const uint32_t acc = tmem + 128 * kAcc * s;
#pragma unroll
                for (int ks = 0; ks < 7; ++ks) {
                    const uint32_t koff = (ks >> 2) * kImgPanel + (ks & 3) * 32;
                    const uint32_t w0 = sbase + kGOffImg + koff, w1 = sbase + kGOffImg + 2 * kImgBytes + koff;
                    const uint64_t a0 = sdesc_sw128(x0 + koff, 16, 1024);
                    mma_bf16(acc, a0, sdesc_sw128(w0, 16, 1024), kIdescK, ks > 0);
                    mma_bf16(acc, a0, sdesc_sw128(w0 + kImgBytes, 16, 1024), kIdescK, 1u);
                    if (kMode == 1) {
                        const uint64_t a1 = sdesc_sw128(x1 + koff, 16, 1024);
                        mma_bf16(acc + 128, a1, sdesc_sw128(w1, 16, 1024), kIdescK, ks > 0);
                        mma_bf16(acc + 128, a1, sdesc_sw128(w1 + kImgBytes, 16, 1024), kIdescK, 1u);
                        // k G^T: the G image as an MN-major B operand, 16 image rows (K) per step
                        const uint32_t wm = sbase + kGOffImg + 2 * kImgBytes + ks * 2048;
                        mma_bf16(acc + 256, a0, sdesc_sw128(wm, kImgPanel, 1024), kIdescKMN, ks > 0);
                        mma_bf16(acc + 256, a0, sdesc_sw128(wm + kImgBytes, kImgPanel, 1024), kIdescKMN, 1u);
                    }
                }
                mma_commit(&acc_full[s]);
                mma_commit(&x_empty[s]);
            }
            mma_commit(drain);
            mbar_wait_drain(drain, 0);
        }
    } else if (warp < 6) {
        // images: row j = column j of W (W0 then W1), hi + lo bf16; rows and
        // columns 112..127 zero
        const int j = (warp & 3) * 32 + lane;
        for (int w = 0; w < (kMode == 1 ? 2 : 1); ++w) {
            const float *W = w == 0 ? p.W0 + ((size_t)bh * p.F + f) * kStateFloats
                                    : p.W1 + ((size_t)bh * (p.F + 1) + (p.F - 1 - f)) * kStateFloats;
            uint8_t *img = sm + kGOffImg + w * 2 * kImgBytes;
#pragma unroll 1
            for (int c8 = 0; c8 < 16; ++c8) {
                float x[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const int i = c8 * 8 + e;
                    x[e] = (j < kD && i < kD) ? W[i * kD + j] : 0.f;
                }
                uint4 hi, lo;
                split_bf16x8(x, hi, lo);
                const uint32_t off = (c8 >> 3) * kImgPanel + sw128_off(j, c8 & 7);
                *reinterpret_cast<uint4 *>(img + off) = hi;
                *reinterpret_cast<uint4 *>(img + kImgBytes + off) = lo;
            }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(img_ready);
    } else {
        // output warps: thread = token row r of the tile
        const int quad = warp & 3, r = quad * 32 + lane;
        const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
        bool ok = true;
        for (int t = 0; t < n_tiles; ++t) {
            const int s = t % kStages, u = t / kStages;
            // the row the normalisation applies to: q (x1) in mode 0, k (x0) in mode 1
            const uint8_t *xr = sm + xtile(s, kMode == 0 ? 1 : 0);
            if (ok) ok = mbar_wait_warp(&acc_full[s], u & 1, abort_flag);
            tc_fence_after();
            const int tok = t * 128 + r;
            const bool live = ok && tok < p.N;
            const size_t rowi = ((size_t)bf * p.N + tok) * p.H + h;
            const uint32_t acc = tmem + 128 * kAcc * s + lane_off;
            auto xrow = [&](int cc, float *o16) {  // 16 bf16 values of this thread's row, columns 16 cc..
                bf16x8_to_f32(*reinterpret_cast<const uint4 *>(xr + ((2 * cc) >> 3) * kImgPanel +
                                                               sw128_off(r, (2 * cc) & 7)), o16);
                bf16x8_to_f32(*reinterpret_cast<const uint4 *>(xr + ((2 * cc + 1) >> 3) * kImgPanel +
                                                               sw128_off(r, (2 * cc + 1) & 7)), o16 + 8);
            };
            if (kMode == 0) {
                float sqq = 0.f, sqd = 0.f;
#pragma unroll 1
                for (int cc = 0; cc < 7; ++cc) {
                    uint32_t ra[16];
                    tmem_ld16(acc + cc * 16, ra);
                    tmem_ld_wait();
                    float xq[16];
                    xrow(cc, xq);
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        sqq = fmaf(xq[e], xq[e], sqq);
                        sqd = fmaf(xq[e], __uint_as_float(ra[e]), sqd);
                    }
                }
                const float p2 = sqq + kEps, pinv = rsqrtf(p2), corr = sqd / p2;
                float *dq = p.g0 + rowi * kD;
#pragma unroll 1
                for (int cc = 0; cc < 7; ++cc) {
                    uint32_t ra[16];
                    tmem_ld16(acc + cc * 16, ra);
                    tmem_ld_wait();
                    float xq[16];
                    xrow(cc, xq);
                    if (live) {
                        float4 *d4 = reinterpret_cast<float4 *>(dq + cc * 16);
#pragma unroll
                        for (int q4 = 0; q4 < 4; ++q4) {
                            float o[4];
#pragma unroll
                            for (int e = 0; e < 4; ++e)
                                o[e] = pinv * (__uint_as_float(ra[4 * q4 + e]) - xq[4 * q4 + e] * corr);
                            d4[q4] = make_float4(o[0], o[1], o[2], o[3]);
                        }
                    }
                }
            } else {
                float skk = 0.f, s2 = 0.f, s3 = 0.f;
#pragma unroll 1
                for (int cc = 0; cc < 7; ++cc) {
                    uint32_t r0[16], r1[16];
                    tmem_ld16(acc + cc * 16, r0);
                    tmem_ld16(acc + 128 + cc * 16, r1);
                    tmem_ld_wait();
                    float xk[16];
                    xrow(cc, xk);
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        skk = fmaf(xk[e], xk[e], skk);
                        s2 = fmaf(xk[e], __uint_as_float(r0[e]), s2);
                        s3 = fmaf(xk[e], __uint_as_float(r1[e]), s3);
                    }
                }
                const float r2 = skk + kEps, kh = p.c * rsqrtf(r2);   // c / r
                const float bt = live ? __ldg(p.beta + rowi) : 0.f;
                const float kdk = bt * (kh * s2 + s3);                 // k . dk^
                if (live) p.g_beta[rowi] = 0.5f * kh * kh * s2 + kh * s3;
                float *dk = p.g0 + rowi * kD, *dv = p.g1 + rowi * kD;
#pragma unroll 1
                for (int cc = 0; cc < 7; ++cc) {
                    uint32_t r0[16], r1[16], r2v[16];
                    tmem_ld16(acc + cc * 16, r0);
                    tmem_ld16(acc + 128 + cc * 16, r1);
                    tmem_ld16(acc + 256 + cc * 16, r2v);
                    tmem_ld_wait();
                    float xk[16];
                    xrow(cc, xk);
                    if (live) {
                        float4 *k4 = reinterpret_cast<float4 *>(dk + cc * 16);
                        float4 *v4 = reinterpret_cast<float4 *>(dv + cc * 16);
#pragma unroll
                        for (int q4 = 0; q4 < 4; ++q4) {
                            float ok4[4], ov4[4];
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const int i = 4 * q4 + e;
                                const float dkh = bt * (kh * __uint_as_float(r0[i]) + __uint_as_float(r1[i]));
                                ok4[e] = kh * (dkh - xk[i] * kdk / r2);
                                ov4[e] = bt * kh * __uint_as_float(r2v[i]);
                            }
                            k4[q4] = make_float4(ok4[0], ok4[1], ok4[2], ok4[3]);
                            v4[q4] = make_float4(ov4[0], ov4[1], ov4[2], ov4[3]);
                        }
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (ok && lane == 0) {
                mbar_arrive(&acc_free[s]);
                mbar_arrive(&x_empty[s]);
            }
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

// ------------------------------------------------------------ orchestration
namespace {
struct BwdLayout {
    TcPlan plan, plan_G;  // F frames; the reverse scan's F + 1 slots
    size_t ws_fwd, ws_E, ones, ws_G, gamma_G, Sst, Gst, Dsym, total;
};

bool bwd_layout(int B, int H, int F, int N, BwdLayout *L)
{
    if (!tc_plan(B, H, F, N, 0, &L->plan) || !tc_plan(B, H, F + 1, N, 0, &L->plan_G)) return false;
    const size_t BH = (size_t)B * H;
    size_t o = 0;
    L->ws_fwd = o; o = up256(o + L->plan.ws_bytes);
    L->ws_E = o; o = up256(o + L->plan.ws_bytes);
    L->ones = o; o = up256(o + (size_t)B * F * N * H * 4);
    L->ws_G = o; o = up256(o + L->plan_G.ws_bytes);
    L->gamma_G = o; o = up256(o + (size_t)B * (F + 1) * H * 4);
    L->Sst = o; o = up256(o + BH * F * kStateBytes);
    L->Gst = o; o = up256(o + BH * (F + 1) * kStateBytes);
    L->Dsym = o; o = up256(o + BH * F * kStateBytes);
    L->total = o;
    return true;
}

constexpr int kMaxDevB = 64;
bool g_b_attr[kMaxDevB];

cudaError_t prepare_bwd_kernels()
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevB) return cudaErrorInvalidDevice;
    if (g_b_attr[dev]) return cudaSuccess;
    if ((e = cudaFuncSetAttribute(kg_token_grad_kernel<0>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)kGSmem)) != cudaSuccess)
        return e;
    if ((e = cudaFuncSetAttribute(kg_token_grad_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)kGSmem)) != cudaSuccess)
        return e;
    if ((e = cudaFuncSetAttribute(kb_frame_grad, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kFgSmem)) !=
        cudaSuccess)
        return e;
    g_b_attr[dev] = true;
    return cudaSuccess;
}

cudaError_t token_grads(const void *dO, const void *q, const void *k, const void *v, const float *beta,
                        const float *Sst, const float *Dsym, const float *Gst, float *dq, float *dk, float *dv,
                        float *dbeta, int B, int H, int F, int N, float c, unsigned *status, cudaStream_t stream)
{
    CUtensorMap mdo, mq, mk, mv;
    if (!make_token_map(&mdo, dO, B, H, F, N, 128) || !make_token_map(&mq, q, B, H, F, N, 128) ||
        !make_token_map(&mk, k, B, H, F, N, 128) || !make_token_map(&mv, v, B, H, F, N, 128))
        return cudaErrorInvalidValue;
    TokGradParams p;
    p.beta = beta;
    p.status = status;
    p.B = B;
    p.H = H;
    p.F = F;
    p.N = N;
    p.c = c;
    p.W0 = Sst;
    p.W1 = nullptr;
    p.g0 = dq;
    p.g1 = nullptr;
    p.g_beta = nullptr;
    kg_token_grad_kernel<0><<<B * H * F, kGThreads, kGSmem, stream>>>(mdo, mq, p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    p.W0 = Dsym;
    p.W1 = Gst;
    p.g0 = dk;
    p.g1 = dv;
    p.g_beta = dbeta;
    kg_token_grad_kernel<1><<<B * H * F, kGThreads, kGSmem, stream>>>(mk, mv, p);
    return cudaGetLastError();
}
}  // namespace

size_t bwd_workspace_bytes(int B, int H, int F, int N)
{
    BwdLayout L;
    return bwd_layout(B, H, F, N, &L) ? L.total : (size_t)-1;
}

cudaError_t launch_frame_bwd_tc(const void *q, const void *k, const void *v, const float *beta, const float *gamma,
                                const float *S_in, const void *dO, const float *dS_out, float *dq, float *dk,
                                float *dv, float *dbeta, float *dgamma, float *dS_in, int B, int H, int F, int N,
                                float c, void *workspace, unsigned *status, cudaStream_t stream)
{
    BwdLayout L;
    if (!bwd_layout(B, H, F, N, &L)) return cudaErrorInvalidValue;
    cudaError_t e = prepare_bwd_kernels();
    if (e != cudaSuccess) return e;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    const int BH = B * H;
    const size_t rows = (size_t)B * F * N * H;  // token rows (beta entries)
    float *ones = reinterpret_cast<float *>(ws + L.ones);
    float *gamma_G = reinterpret_cast<float *>(ws + L.gamma_G);
    float *Sst = reinterpret_cast<float *>(ws + L.Sst), *Gst = reinterpret_cast<float *>(ws + L.Gst);
    float *Dsym = reinterpret_cast<float *>(ws + L.Dsym);
    // 1. forward statistics and every state S_f
    if ((e = launch_frame_stats_tc(k, v, beta, gamma, L.plan, c, 0, ws + L.ws_fwd, status, stream)) != cudaSuccess)
        return e;
    if ((e = launch_states_tc(q, gamma, S_in, nullptr, Sst, L.plan, ws + L.ws_fwd, status, stream)) != cudaSuccess)
        return e;
    // 2. E_f = dO^T q^ through the statistics kernel (k := q, v := dO, beta := 1, c := 1)
    kb_fill<<<296, 256, 0, stream>>>(ones, rows, 1.f);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if ((e = launch_frame_stats_tc(q, dO, ones, gamma, L.plan, 1.f, 0, ws + L.ws_E, status, stream)) != cudaSuccess)
        return e;
    // 3. reverse scan G_{F-1} .. G_0, ending at dS_in
    kb_build_reverse_ws<<<dim3(BH, F + 1), 256, 0, stream>>>(ws + L.ws_fwd + L.plan.off_frames,
                                                              ws + L.ws_E + L.plan.off_frames,
                                                              ws + L.ws_G + L.plan_G.off_frames, gamma, gamma_G, B, H,
                                                              F);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if ((e = launch_chunk_composite_tc(gamma_G, L.plan_G, 0, ws + L.ws_G, status, stream)) != cudaSuccess) return e;
    if ((e = launch_states_tc(q, gamma_G, dS_out, dS_in, Gst, L.plan_G, ws + L.ws_G, status, stream)) != cudaSuccess)
        return e;
    // 4. per-frame dgamma and Dsym = dA + dA^T
    kb_frame_grad<<<dim3(BH, F), 256, kFgSmem, stream>>>(S_in, Sst, Gst, dgamma, Dsym, B, H, F);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    // 5. token gradients: dq from dO S_f; dk, dv, dbeta from k Dsym_f, v G_f, k G_f^T
    if ((e = token_grads(dO, q, k, v, beta, Sst, Dsym, Gst, dq, dk, dv, dbeta, B, H, F, N, c, status, stream)) !=
        cudaSuccess)
        return e;
    return cudaSuccess;  // dS_in: written by the reverse scan as its final state
}

}  // namespace gdn
