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
//   1. K1 on (k, v): A_f images and U_f in a workspace; the state chain kernel
//      from S_in stores every S_f.
//   2. K1 on (k := q, v := dO, beta := 1, c := 1): its U_f slots are E_f.
//   3. kb_build_reverse_ws lays out the reverse scan: slot p holds A of frame
//      F - p (none for p = 0) and E_{F-1-p} (none for p = F), gamma likewise, so
//      that the state chain kernel from dS_out visits G_{F-1}, ..., G_0 and
//      ends at dS_in.
//   4. kb_frame_grad: dM_f = S_{f-1}^T G_f (fp32 CUDA cores), dgamma_f, and
//      Dsym_f = dA_f + dA_f^T.
//   5. kt_token_matrix_kernel (tcgen05): for every token row x_t of a frame,
//      x_t^T W_f with W_f one of S_f, Dsym_f, G_f, G_f^T (hi + lo bf16 images),
//      rows scaled by c / ||k_t|| where the row is k: dq^, k^^T Dsym, v^T G,
//      k^^T G^T, fp32.
//   6. kb_finalize: dk^, dv, dbeta, then dk and dq through the normalisations.
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

// ------------------------------------------------------- token x matrix GEMM
// out[t][j] = scale_t sum_i x[t][i] W[i][j] for every token t of frame f and
// chain bh, W = W_base[bh][slot(f)] (fp32 D x D), slot(f) = w_rev ? F - 1 - f : f
// over w_slots slots per chain; w_rows: use W^T instead (the image rows are W's
// rows).  norm_c > 0: scale_t = norm_c / ||x_t||, else 1.  One CTA per (frame,
// chain): four warps build W's hi/lo bf16 images once, then 128-token x tiles
// stream through TMA (two stages) into tcgen05 GEMMs (two TMEM slots), and four
// warps write the fp32 rows.
constexpr int kTThreads = 320;
constexpr uint32_t kTOffX = 0;                            // two x stages, 32 KB each
constexpr uint32_t kTOffWhi = 2 * kImgBytes;              // 65536
constexpr uint32_t kTOffWlo = kTOffWhi + kImgBytes;       // 98304
constexpr uint32_t kTOffBar = kTOffWlo + kImgBytes;       // 131072
constexpr uint32_t kTSmem = kTOffBar + 256 + 1024;

struct TokMatParams {
    const float *W;
    float *out;  // [B][F*N][H][D] fp32
    unsigned *status;
    int B, H, F, N;
    int w_slots, w_rev, w_rows;
    float norm_c;
};

__global__ void __launch_bounds__(kTThreads, 1)
    kt_token_matrix_kernel(const __grid_constant__ CUtensorMap mapX, const TokMatParams p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + kTOffBar);
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
        for (int i = 0; i < 2; ++i) {
            mbar_init(&x_full[i], 1);
            mbar_init(&x_empty[i], 5);  // the tile's MMAs + the four output warps (norms read)
            mbar_init(&acc_full[i], 1);
            mbar_init(&acc_free[i], 4);
        }
        mbar_init(img_ready, 4);
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, 256);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t sbase = smem_u32(sm);

    if (warp == 0) {
        if (lane == 0) {
            const uint64_t pol = policy_evict_first();
            int issued = 0;
            for (int t = 0; t < n_tiles; ++t) {
                const int s = t & 1;
                if (t >= 2 && !mbar_wait(&x_empty[s], ((t >> 1) - 1) & 1, abort_flag)) break;
                mbar_arrive_expect_tx(&x_full[s], kImgBytes);
                uint8_t *dst = sm + kTOffX + s * kImgBytes;
                tma_load_4d(dst, &mapX, &x_full[s], 0, h, t * 128, bf, pol);
                tma_load_4d(dst + kImgPanel, &mapX, &x_full[s], 64, h, t * 128, bf, pol);
                ++issued;
            }
            if (*abort_flag)
                for (int s = 0; s < 2 && s < issued; ++s) {
                    const int last = ((issued - 1 - s) / 2) * 2 + s;
                    mbar_wait_drain(&x_full[s], (last >> 1) & 1);
                }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            bool ok = mbar_wait(img_ready, 0, abort_flag);
            tc_fence_after();
            for (int t = 0; t < n_tiles && ok; ++t) {
                const int s = t & 1;
                if (!(ok = mbar_wait(&x_full[s], (t >> 1) & 1, abort_flag))) break;
                if (t >= 2 && !(ok = mbar_wait(&acc_free[s], ((t >> 1) - 1) & 1, abort_flag))) break;
                tc_fence_after();
                const uint32_t xb = sbase + kTOffX + s * kImgBytes;
#pragma unroll
                for (int ks = 0; ks < 7; ++ks) {
                    const uint32_t koff = (ks >> 2) * kImgPanel + (ks & 3) * 32;
                    const uint64_t ad = sdesc_sw128(xb + koff, 16, 1024);
                    mma_bf16(tmem + 128 * s, ad, sdesc_sw128(sbase + kTOffWhi + koff, 16, 1024), kIdescK, ks > 0);
                    mma_bf16(tmem + 128 * s, ad, sdesc_sw128(sbase + kTOffWlo + koff, 16, 1024), kIdescK, 1u);
                }
                mma_commit(&acc_full[s]);
                mma_commit(&x_empty[s]);
            }
            mma_commit(drain);
            mbar_wait_drain(drain, 0);
        }
    } else if (warp < 6) {
        // W images: image row j holds column j of W (row j of W when w_rows),
        // as hi + lo bf16 in the 128B-swizzled K-major layout; rows 112..127
        // and columns 112..127 are zero.
        const int j = (warp & 3) * 32 + lane;
        const int slot = p.w_rev ? p.F - 1 - f : f;
        const float *W = p.W + ((size_t)bh * p.w_slots + slot) * kStateFloats;
#pragma unroll 1
        for (int c8 = 0; c8 < 16; ++c8) {
            float x[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const int i = c8 * 8 + e;
                x[e] = (j < kD && i < kD) ? (p.w_rows ? W[j * kD + i] : W[i * kD + j]) : 0.f;
            }
            uint4 hi, lo;
            split_bf16x8(x, hi, lo);
            const uint32_t off = (c8 >> 3) * kImgPanel + sw128_off(j, c8 & 7);
            *reinterpret_cast<uint4 *>(sm + kTOffWhi + off) = hi;
            *reinterpret_cast<uint4 *>(sm + kTOffWlo + off) = lo;
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
            const int s = t & 1;
            const uint8_t *xs = sm + kTOffX + s * kImgBytes;
            if (ok) ok = mbar_wait_warp(&x_full[s], (t >> 1) & 1, abort_flag);
            float scale = 1.f;
            if (ok && p.norm_c > 0.f) {
                float ss = 0.f;
#pragma unroll
                for (int c = 0; c < 16; ++c) {
                    const uint4 u = *reinterpret_cast<const uint4 *>(xs + (c >> 3) * kImgPanel + r * kRowB +
                                                                     (((c & 7) ^ (r & 7)) << 4));
                    float f8[8];
                    bf16x8_to_f32(u, f8);
#pragma unroll
                    for (int e = 0; e < 8; ++e) ss = fmaf(f8[e], f8[e], ss);
                }
                scale = p.norm_c * rsqrtf(ss + kEps);
            }
            __syncwarp();
            if (ok && lane == 0) mbar_arrive(&x_empty[s]);
            if (ok) ok = mbar_wait_warp(&acc_full[s], (t >> 1) & 1, abort_flag);
            tc_fence_after();
            if (ok) {
                const int tok = t * 128 + r;
                float *dst = p.out + (((size_t)bf * p.N + tok) * p.H + h) * kD;
#pragma unroll
                for (int cc = 0; cc < 7; ++cc) {
                    uint32_t ra[16];
                    tmem_ld16(tmem + 128 * s + lane_off + cc * 16, ra);
                    tmem_ld_wait();
                    if (tok < p.N) {
                        float4 *d4 = reinterpret_cast<float4 *>(dst + cc * 16);
#pragma unroll
                        for (int q4 = 0; q4 < 4; ++q4)
                            d4[q4] = make_float4(scale * __uint_as_float(ra[4 * q4]), scale * __uint_as_float(ra[4 * q4 + 1]),
                                                 scale * __uint_as_float(ra[4 * q4 + 2]),
                                                 scale * __uint_as_float(ra[4 * q4 + 3]));
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (ok && lane == 0) mbar_arrive(&acc_free[s]);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (*abort_flag && threadIdx.x == 0) raise_status(p.status);
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 256);
    }
}

// ------------------------------------------------------------------ finalize
// One warp per (token, head) row; lane l holds elements 4l .. 4l+3 (l < 28).
__global__ void __launch_bounds__(256) kb_finalize(const __nv_bfloat16 *q, const __nv_bfloat16 *k,
                                                   const float *beta, const float *dqh, const float *x23,
                                                   const float *x4, const float *x5, float *dq, float *dk, float *dv,
                                                   float *dbeta, float c, size_t rows)
{
    const size_t row = (size_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= rows) return;
    const bool act = lane < kD / 4;
    const size_t base = row * kD + 4 * lane;
    float kv[4] = {0, 0, 0, 0}, qv[4] = {0, 0, 0, 0}, a23[4] = {0, 0, 0, 0}, a4[4] = {0, 0, 0, 0};
    float a5[4] = {0, 0, 0, 0}, dh[4] = {0, 0, 0, 0};
    if (act) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            kv[e] = __bfloat162float(k[base + e]);
            qv[e] = __bfloat162float(q[base + e]);
        }
        const float4 t23 = *reinterpret_cast<const float4 *>(x23 + base);
        const float4 t4 = *reinterpret_cast<const float4 *>(x4 + base);
        const float4 t5 = *reinterpret_cast<const float4 *>(x5 + base);
        const float4 td = *reinterpret_cast<const float4 *>(dqh + base);
        a23[0] = t23.x, a23[1] = t23.y, a23[2] = t23.z, a23[3] = t23.w;
        a4[0] = t4.x, a4[1] = t4.y, a4[2] = t4.z, a4[3] = t4.w;
        a5[0] = t5.x, a5[1] = t5.y, a5[2] = t5.z, a5[3] = t5.w;
        dh[0] = td.x, dh[1] = td.y, dh[2] = td.z, dh[3] = td.w;
    }
    // warp sums: |k|^2, |q|^2, k . x23, k . x4, q . dq^
    float s[5] = {0, 0, 0, 0, 0};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        s[0] = fmaf(kv[e], kv[e], s[0]);
        s[1] = fmaf(qv[e], qv[e], s[1]);
        s[2] = fmaf(kv[e], a23[e], s[2]);
        s[3] = fmaf(kv[e], a4[e], s[3]);
        s[4] = fmaf(qv[e], dh[e], s[4]);
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1)
#pragma unroll
        for (int i = 0; i < 5; ++i) s[i] += __shfl_xor_sync(0xffffffffu, s[i], o);
    const float bt = beta[row];
    const float r2 = s[0] + kEps, rinv = rsqrtf(r2), kh = c * rinv;  // k^ = kh * k
    const float p2 = s[1] + kEps, pinv = rsqrtf(p2);
    // dk^ = beta (x23 + x4);  k . dk^ = beta (k . x23 + k . x4)
    const float kdk = bt * (s[2] + s[3]);
    if (act) {
        float4 o_dk, o_dv, o_dq;
        float *pk = &o_dk.x, *pv = &o_dv.x, *pq = &o_dq.x;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float dkh = bt * (a23[e] + a4[e]);
            pk[e] = kh * (dkh - kv[e] * kdk / r2);
            pv[e] = bt * a5[e];
            pq[e] = pinv * (dh[e] - qv[e] * s[4] / p2);
        }
        *reinterpret_cast<float4 *>(dk + base) = o_dk;
        *reinterpret_cast<float4 *>(dv + base) = o_dv;
        *reinterpret_cast<float4 *>(dq + base) = o_dq;
    }
    // dbeta = k^ dA k^ + v G k^ = 1/2 k^ . x23 + x4 . k^
    if (lane == 0) dbeta[row] = kh * (0.5f * s[2] + s[3]);
}

// ------------------------------------------------------------ orchestration
namespace {
struct BwdLayout {
    TcPlan plan;
    size_t ws_fwd, ws_E, ones, ws_G, gamma_G, Sst, Gst, Dsym, dqh, x23, x4, x5, total;
};

bool bwd_layout(int B, int H, int F, int N, BwdLayout *L)
{
    if (!tc_plan(B, H, F, N, 0, &L->plan)) return false;
    const size_t BH = (size_t)B * H, tokf = (size_t)B * F * N * H * kD * 4;
    size_t o = 0;
    L->ws_fwd = o; o = up256(o + L->plan.ws_bytes);
    L->ws_E = o; o = up256(o + L->plan.ws_bytes);
    L->ones = o; o = up256(o + (size_t)B * F * N * H * 4);
    L->ws_G = o; o = up256(o + BH * (F + 1) * kFrameWs);
    L->gamma_G = o; o = up256(o + (size_t)B * (F + 1) * H * 4);
    L->Sst = o; o = up256(o + BH * F * kStateBytes);
    L->Gst = o; o = up256(o + BH * (F + 1) * kStateBytes);
    L->Dsym = o; o = up256(o + BH * F * kStateBytes);
    L->dqh = o; o = up256(o + tokf);
    L->x23 = o; o = up256(o + tokf);
    L->x4 = o; o = up256(o + tokf);
    L->x5 = o; o = up256(o + tokf);
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
    if ((e = cudaFuncSetAttribute(kt_token_matrix_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)kTSmem)) != cudaSuccess)
        return e;
    if ((e = cudaFuncSetAttribute(kb_frame_grad, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kFgSmem)) !=
        cudaSuccess)
        return e;
    g_b_attr[dev] = true;
    return cudaSuccess;
}

cudaError_t token_matrix(const void *x, const float *W, int w_slots, int w_rev, int w_rows, float norm_c, float *out,
                         int B, int H, int F, int N, unsigned *status, cudaStream_t stream)
{
    CUtensorMap mx;
    if (!make_token_map(&mx, x, B, H, F, N, 128)) return cudaErrorInvalidValue;
    TokMatParams p;
    p.W = W;
    p.out = out;
    p.status = status;
    p.B = B;
    p.H = H;
    p.F = F;
    p.N = N;
    p.w_slots = w_slots;
    p.w_rev = w_rev;
    p.w_rows = w_rows;
    p.norm_c = norm_c;
    kt_token_matrix_kernel<<<B * H * F, kTThreads, kTSmem, stream>>>(mx, p);
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
    const size_t rows = (size_t)B * F * N * H;
    float *ones = reinterpret_cast<float *>(ws + L.ones);
    float *gamma_G = reinterpret_cast<float *>(ws + L.gamma_G);
    float *Sst = reinterpret_cast<float *>(ws + L.Sst), *Gst = reinterpret_cast<float *>(ws + L.Gst);
    float *Dsym = reinterpret_cast<float *>(ws + L.Dsym);
    float *dqh = reinterpret_cast<float *>(ws + L.dqh), *x23 = reinterpret_cast<float *>(ws + L.x23);
    float *x4 = reinterpret_cast<float *>(ws + L.x4), *x5 = reinterpret_cast<float *>(ws + L.x5);
    // 1. forward statistics and every state S_f
    if ((e = launch_frame_stats_tc(k, v, beta, gamma, L.plan, c, 0, ws + L.ws_fwd, status, stream)) != cudaSuccess)
        return e;
    if ((e = launch_state_chain_tc(gamma, ws + L.ws_fwd + L.plan.off_frames, S_in, Sst, B, H, F, status, stream)) !=
        cudaSuccess)
        return e;
    // 2. E_f = dO^T q^ through the statistics kernel (k := q, v := dO, beta := 1, c := 1)
    kb_fill<<<296, 256, 0, stream>>>(ones, rows, 1.f);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if ((e = launch_frame_stats_tc(q, dO, ones, gamma, L.plan, 1.f, 0, ws + L.ws_E, status, stream)) != cudaSuccess)
        return e;
    // 3. reverse scan G_{F-1} .. G_0, ending at dS_in
    kb_build_reverse_ws<<<dim3(BH, F + 1), 256, 0, stream>>>(ws + L.ws_fwd + L.plan.off_frames,
                                                              ws + L.ws_E + L.plan.off_frames, ws + L.ws_G, gamma,
                                                              gamma_G, B, H, F);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if ((e = launch_state_chain_tc(gamma_G, ws + L.ws_G, dS_out, Gst, B, H, F + 1, status, stream)) != cudaSuccess)
        return e;
    // 4. per-frame dgamma and Dsym = dA + dA^T
    kb_frame_grad<<<dim3(BH, F), 256, kFgSmem, stream>>>(S_in, Sst, Gst, dgamma, Dsym, B, H, F);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    // 5. token rows times per-frame matrices
    if ((e = token_matrix(dO, Sst, F, 0, 0, 0.f, dqh, B, H, F, N, status, stream)) != cudaSuccess) return e;
    if ((e = token_matrix(k, Dsym, F, 0, 0, c, x23, B, H, F, N, status, stream)) != cudaSuccess) return e;
    if ((e = token_matrix(v, Gst, F + 1, 1, 0, 0.f, x4, B, H, F, N, status, stream)) != cudaSuccess) return e;
    if ((e = token_matrix(k, Gst, F + 1, 1, 1, c, x5, B, H, F, N, status, stream)) != cudaSuccess) return e;
    // 6. dk, dv, dq, dbeta
    kb_finalize<<<(unsigned)((rows + 7) / 8), 256, 0, stream>>>(
        static_cast<const __nv_bfloat16 *>(q), static_cast<const __nv_bfloat16 *>(k), beta, dqh, x23, x4, x5, dq, dk,
        dv, dbeta, c, rows);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    // 7. dS_in = the reverse scan's last state
    if (dS_in)
        e = cudaMemcpy2DAsync(dS_in, kStateBytes, Gst + (size_t)F * kStateFloats, (F + 1) * kStateBytes, kStateBytes,
                              BH, cudaMemcpyDeviceToDevice, stream);
    return e;
}

}  // namespace gdn
