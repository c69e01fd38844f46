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
//   2. K1 on (k := q, v := dO, beta := 1, c := 1) in its E mode forms only the
//      U_f slots, which are E_f.
//   3. The reverse scan: slot p holds A of frame F - p (none for p = 0) and
//      E_{F-1-p} (none for p = F), gamma likewise; the two K1 passes write
//      those slots directly and kb_reverse_edges fills the empty ends; its chunk
//      composites (K1c), the chunk-boundary kernel and the scan kernel without
//      outputs, from dS_out, visit G_{F-1}, ..., G_0 and end at dS_in.
//   4. kb_frame_grad_tc: dM_f = S_{f-1}^T G_f (tcgen05, hi + lo bf16), dgamma_f, and
//      Dsym_f = dA_f + dA_f^T and G_f as bf16 MMA-operand images for step 5.
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
// The reverse scan's workspace: slot p of a chain holds A of frame F - p and E
// of frame F - 1 - p, written there by the two statistics passes; this kernel
// fills the two empty ends (no A in slot 0, no E in slot F) with zeros and lays
// out gamma in slot order (1 for slot 0).  One block per chain.
__global__ void kb_reverse_edges(uint8_t *ws_G, const float *gamma, float *gamma_G, int B, int H, int F)
{
    const int bh = blockIdx.x;
    const int b = bh / H, h = bh % H;
    uint4 *a0 = reinterpret_cast<uint4 *>(ws_G + (size_t)bh * (F + 1) * kFrameWs);
    uint4 *uF = reinterpret_cast<uint4 *>(ws_G + ((size_t)bh * (F + 1) + F) * kFrameWs + kAimgBytes);
    for (int i = threadIdx.x; i < (int)(kAimgBytes / 16); i += blockDim.x) a0[i] = make_uint4(0, 0, 0, 0);
    for (int i = threadIdx.x; i < (int)(kUBytes / 16); i += blockDim.x) uF[i] = make_uint4(0, 0, 0, 0);
    for (int q = threadIdx.x; q <= F; q += blockDim.x)
        gamma_G[((size_t)b * (F + 1) + q) * H + h] = q >= 1 ? gamma[((size_t)b * F + (F - q)) * H + h] : 1.f;
}

// dM_f = S_{f-1}^T G_f, dgamma_f = trace(dM_f), Dsym_f = -(dM_f + dM_f^T), on
// tcgen05.  Persistent: one CTA per SM walks (frame, chain) items.  With
// m = i, n = j, k = l, dM[i][j] = sum_l S[l][i] G[l][j] takes both operands
// MN-major, so the images are plain row-major copies of S_{f-1} and G_f (image
// row l = matrix row l), each as bf16 hi + lo; three MMAs per 16-row k-step
// (S_hi G_hi + S_lo G_hi + S_hi G_lo) keep the product near fp32.  Warps:
// 1 issues the MMAs, 2..5 build the images (the next item's matrices are
// prefetched into L2 first), 6..9 read dM out of TMEM (two accumulator sets,
// so the next item's MMAs run meanwhile) into a padded fp32 tile in shared
// memory, from which the trace and the symmetrised Dsym are written.  The
// token-gradient kernel reads Dsym_f and G_f as bf16 MMA operands, so both
// leave as ready images (row-major, 128 rows x two 128B-swizzled 64-column
// panels, rows and columns 112.. zero): Dsym_f built here with coalesced
// 16-byte stores, G_f bulk-copied from this kernel's own hi image.
constexpr int kFgThreads = 320;
constexpr uint32_t kFgDMStride = kD + 1;  // odd row stride: row writes and column reads are conflict-free
constexpr uint32_t kFgOffDM = 4 * kImgBytes;
constexpr uint32_t kFgOffBar = kFgOffDM + ((kD * kFgDMStride * 4 + 1023) / 1024) * 1024;
constexpr uint32_t kFgSmem = kFgOffBar + 256 + 1024;
static_assert(kFgSmem <= kMaxSmem, "frame-gradient kernel shared memory");

struct FrameGradParams {
    const float *S_in;  // [BH] states or null (zero)
    const float *Sst;   // S_f after every frame, [BH][F]
    const float *Gst;   // G_f, [BH][F+1] (G_f at slot F-1-f)
    float *dgamma;      // [B][F][H]
    uint8_t *img_out;   // [BH][F] x (Dsym_f image, G_f image), kImgBytes each
    unsigned *status;
    int B, H, F;
};

// Epilogue warps 6..9 (id 0 is __syncthreads).
__device__ __forceinline__ void fg_epi_sync() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

__global__ void __launch_bounds__(kFgThreads, 1) kb_frame_grad_tc(const FrameGradParams p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    float *dM = reinterpret_cast<float *>(sm + kFgOffDM);
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + kFgOffBar);
    uint64_t *acc_full = bars + 0, *acc_free = bars + 2, *img_ready = bars + 4, *img_free = bars + 5;
    uint64_t *drain = bars + 6;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 7);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(bars + 8);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int BH = p.B * p.H;
    const int n_items = BH * p.F;  // item = (frame f, chain bh), f major
    // the item's two matrices: S_{f-1} (null: zero) and G_f
    auto mat = [&](int w, int it) -> const float * {
        const int f = it / BH, bh = it % BH;
        if (w == 1) return p.Gst + ((size_t)bh * (p.F + 1) + (p.F - 1 - f)) * kStateFloats;
        if (f == 0) return p.S_in ? p.S_in + (size_t)bh * kStateFloats : nullptr;
        return p.Sst + ((size_t)bh * p.F + f - 1) * kStateFloats;
    };

    if (threadIdx.x == 0) {
        for (int i = 0; i < 2; ++i) {
            mbar_init(&acc_full[i], 1);
            mbar_init(&acc_free[i], 4);
        }
        mbar_init(img_ready, 4);
        mbar_init(img_free, 1);
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

    if (warp == 1) {
        if (lane == 0) {
            bool ok = true;
            int i = 0;
            for (int it = blockIdx.x; it < n_items && ok; it += gridDim.x, ++i) {
                const int a = i & 1, ua = i >> 1;
                if (!(ok = mbar_wait(img_ready, i & 1, abort_flag))) break;
                if (ua >= 1 && !(ok = mbar_wait(&acc_free[a], (ua - 1) & 1, abort_flag))) break;
                tc_fence_after();
                const uint32_t acc = tmem + 128 * a;
#pragma unroll
                for (int ks = 0; ks < 7; ++ks) {
                    const uint32_t o = ks * 2048;  // image rows 16 ks .. 16 ks + 15 (k = l)
                    const uint64_t s_hi = sdesc_sw128(sbase + o, kImgPanel, 1024);
                    const uint64_t s_lo = sdesc_sw128(sbase + kImgBytes + o, kImgPanel, 1024);
                    const uint64_t g_hi = sdesc_sw128(sbase + 2 * kImgBytes + o, kImgPanel, 1024);
                    const uint64_t g_lo = sdesc_sw128(sbase + 3 * kImgBytes + o, kImgPanel, 1024);
                    mma_bf16(acc, s_hi, g_hi, kIdescMN, ks > 0);
                    mma_bf16(acc, s_lo, g_hi, kIdescMN, 1u);
                    mma_bf16(acc, s_hi, g_lo, kIdescMN, 1u);
                }
                mma_commit(&acc_full[a]);
                mma_commit(img_free);  // the images may be rebuilt once these MMAs have read them
            }
            mma_commit(drain);
            mbar_wait_drain(drain, 0);
        }
    } else if (warp >= 2 && warp < 6) {
        // images: thread = matrix row l (0..127; rows 112.. and columns 112.. zero)
        const int l = (warp - 2) * 32 + lane;
        bool ok = true;
        int i = 0;
        for (int it = blockIdx.x; it < n_items && ok; it += gridDim.x, ++i) {
            if (warp == 2 && lane < 2 && it + (int)gridDim.x < n_items) {
                const float *nxt = mat(lane, it + gridDim.x);
                if (nxt) bulk_prefetch_l2(nxt, kStateBytes);
            }
            if (i >= 1 && !(ok = mbar_wait_warp(img_free, (i - 1) & 1, abort_flag))) break;
            if (lane == 0) bulk_wait_read_all();  // the previous item's G image export has read these rows
            __syncwarp();
            const float *W[2] = {mat(0, it), mat(1, it)};
#pragma unroll 1
            for (int half = 0; half < 2; ++half) {  // 8-column groups 7 half .. 7 half + 6, both matrices in flight
                float x[2][7][8];
#pragma unroll
                for (int w = 0; w < 2; ++w)
#pragma unroll
                    for (int g = 0; g < 7; ++g) {
                        const int c8 = 7 * half + g;
                        if (W[w] && l < kD) {
                            const float4 a4 = __ldg(reinterpret_cast<const float4 *>(W[w] + l * kD + 8 * c8));
                            const float4 b4 = __ldg(reinterpret_cast<const float4 *>(W[w] + l * kD + 8 * c8 + 4));
                            x[w][g][0] = a4.x; x[w][g][1] = a4.y; x[w][g][2] = a4.z; x[w][g][3] = a4.w;
                            x[w][g][4] = b4.x; x[w][g][5] = b4.y; x[w][g][6] = b4.z; x[w][g][7] = b4.w;
                        } else {
#pragma unroll
                            for (int e = 0; e < 8; ++e) x[w][g][e] = 0.f;
                        }
                    }
#pragma unroll
                for (int w = 0; w < 2; ++w)
#pragma unroll
                    for (int g = 0; g < 7; ++g) {
                        const int c8 = 7 * half + g;
                        const uint32_t off = (c8 >> 3) * kImgPanel + sw128_off(l, c8 & 7);
                        uint4 hi, lo;
                        split_bf16x8(x[w][g], hi, lo);
                        *reinterpret_cast<uint4 *>(sm + 2 * w * kImgBytes + off) = hi;
                        *reinterpret_cast<uint4 *>(sm + (2 * w + 1) * kImgBytes + off) = lo;
                    }
            }
#pragma unroll
            for (int c8 = 14; c8 < 16; ++c8) {
                const uint32_t off = kImgPanel + sw128_off(l, c8 & 7);
#pragma unroll
                for (int m = 0; m < 4; ++m) *reinterpret_cast<uint4 *>(sm + m * kImgBytes + off) = make_uint4(0, 0, 0, 0);
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(img_ready);
                // this warp's 32 rows of the G_f hi image, both panels, to the token-gradient kernel
                const int f = it / BH, bh = it % BH;
                uint8_t *gi = p.img_out + ((size_t)bh * p.F + f) * 2 * kImgBytes + kImgBytes;
                const uint32_t ro = (uint32_t)(warp - 2) * 32 * kRowB;
                bulk_s2g(gi + ro, sm + 2 * kImgBytes + ro, 32 * kRowB);
                bulk_s2g(gi + kImgPanel + ro, sm + 2 * kImgBytes + kImgPanel + ro, 32 * kRowB);
                bulk_commit();
            }
        }
        if (lane == 0) bulk_wait_all();
    } else if (warp >= 6) {
        // epilogue: thread = row i of dM
        const int quad = warp & 3, row = quad * 32 + lane, t = threadIdx.x - 192;  // t: 0..127
        const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
        // every warp runs every item and both named barriers; after a timeout the
        // work is skipped (the abort flag makes the other warps' waits return)
        bool ok = true;
        int i = 0;
        for (int it = blockIdx.x; it < n_items; it += gridDim.x, ++i) {
            const int a = i & 1, ua = i >> 1;
            const int f = it / BH, bh = it % BH, b = bh / p.H, h = bh % p.H;
            if (ok) ok = mbar_wait_warp(&acc_full[a], ua & 1, abort_flag);
            tc_fence_after();
            if (ok) {
#pragma unroll
                for (int cp = 0; cp < 7; cp += 4) {
                    uint32_t r4[4][16];
#pragma unroll
                    for (int hf = 0; hf < 4 && cp + hf < 7; ++hf)
                        tmem_ld16(tmem + 128 * a + lane_off + (cp + hf) * 16, r4[hf]);
                    tmem_ld_wait();
                    if (row < kD)
#pragma unroll
                        for (int hf = 0; hf < 4 && cp + hf < 7; ++hf)
#pragma unroll
                            for (int j = 0; j < 16; ++j)
                                dM[row * kFgDMStride + (cp + hf) * 16 + j] = __uint_as_float(r4[hf][j]);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (ok && lane == 0) mbar_arrive(&acc_free[a]);
            fg_epi_sync();  // dM complete in shared memory
            if (ok && !*abort_flag) {
                if (warp == 6) {
                    float d = 0.f;
                    for (int r = lane; r < kD; r += 32) d += dM[r * kFgDMStride + r];
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) d += __shfl_xor_sync(0xffffffffu, d, o);
                    if (lane == 0) p.dgamma[((size_t)b * p.F + f) * p.H + h] = d;
                }
                // Dsym_f image: thread = (row r, 8-column group c8), 16-byte stores along each row
                uint8_t *di = p.img_out + ((size_t)bh * p.F + f) * 2 * kImgBytes;
                for (int e = t; e < 128 * 16; e += 128) {
                    const int r = e >> 4, c8 = e & 15;
                    float x[8];
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        const int c = 8 * c8 + k;
                        x[k] = (r < kD && c < kD) ? -(dM[r * kFgDMStride + c] + dM[c * kFgDMStride + r]) : 0.f;
                    }
                    *reinterpret_cast<uint4 *>(di + (c8 >> 3) * kImgPanel + sw128_off(r, c8 & 7)) = f32x8_to_bf16(x);
                }
            }
            fg_epi_sync();  // dM may be overwritten by the next item
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

// ------------------------------------------------ token-row gradient kernels
// One CTA per (frame, chain), 128-token tiles of the frame's rows through TMA
// into tcgen05 GEMMs against per-frame fp32 matrices given as bf16 images
// (image row j = column j of the matrix, K-major), hi only or hi + lo; the
// epilogue (thread = token row) applies the chain rule through the
// normalisations and writes the final fp32 gradients.
//   kMode 0: acc = dO W (W = S_f)  ->  dq^ = S_f^T do;  dq = (dq^ - q (q.dq^)/rho^2) / rho
//   kMode 1: acc0 = k Dsym, acc1 = v G, acc2 = k G^T from the frame-gradient
//            kernel's row-major images (image row l = matrix row l): v G reads
//            the G image MN-major (B[n = j][k = i] = G[i][j]), k G^T K-major
//            (B[n][k] = G[n][k]), Dsym is symmetric;
//            with k^ = (c/r) k: dk^ = beta ((c/r) acc0 + acc1),
//            dk = (c/r)(dk^ - k (k.dk^)/r^2),  dv = beta (c/r) acc2,
//            dbeta = 1/2 (c/r)^2 k.acc0 + (c/r) k.acc1.
// Shared memory is seven 32 KB slots: the images first, then as many stages
// of the two token tiles as fit, the last slot staging the gradient rows for
// TMA stores (per output warp two 32-row x 16-column boxes of each output,
// 64-byte swizzle).  TMEM holds one accumulator set per stage in mode 0 and a
// single set of three in mode 1.
#ifndef GDN_BWD_LO0
#define GDN_BWD_LO0 1  // mode 0 keeps the lo image of S_f
#endif
#ifndef GDN_BWD_TMA_ST
#define GDN_BWD_TMA_ST 1  // gradient rows leave through shared memory and TMA stores
#endif
constexpr int kGThreads = 320;  // producer, MMA, 4 image warps, 4 output warps
constexpr int kGSlots = 7;
constexpr uint32_t kGOffImg = 0;
constexpr uint32_t kGOffBar = kGSlots * kImgBytes;
constexpr uint32_t kGOffStg = (kGSlots - 1) * kImgBytes;  // staging slot: 8 KB per output warp
constexpr uint32_t kGSmem = kGOffBar + 256 + 1024;
static_assert(kGSmem <= kMaxSmem, "token-gradient kernel shared memory");
constexpr uint32_t kIdescKMN = idesc_bf16(128, kD, false, true);

template <int kMode> struct TokGradShape {
    static constexpr int kLo = kMode == 0 ? GDN_BWD_LO0 : 0;       // mode 1: hi images (bulk-loaded)
    static constexpr int kMats = kMode == 0 ? 1 : 2;
    static constexpr int kImgPer = kLo ? 2 : 1;                     // images per matrix
    static constexpr int kImgs = kMats * kImgPer;
    static constexpr int kStages = (kGSlots - GDN_BWD_TMA_ST - kImgs) / 2;   // (x0, x1) tile stages
    static constexpr int kAcc = kMode == 0 ? 1 : 3;                 // accumulators per tile
    static constexpr int kAccSets = kMode == 0 ? (kStages < 4 ? kStages : 4) : 1;
    static_assert(kStages >= 1 && kStages <= 4, "token-gradient stages");
    static_assert(kAcc * kAccSets * 128 <= 512, "token-gradient TMEM");
};

struct TokGradParams {
    const float *W0;        // mode 0: S states [BH][F]
    const uint8_t *img1;    // mode 1: (Dsym_f, G_f) images [BH][F], kImgBytes each
    const float *beta;
    float *g0, *g1, *g_beta;  // mode 0: dq; mode 1: dk, dv, dbeta
    unsigned *status;
    int B, H, F, N;
    float c;
};

template <int kMode>
__global__ void __launch_bounds__(kGThreads, 1)
    kg_token_grad_kernel(const __grid_constant__ CUtensorMap mapX0, const __grid_constant__ CUtensorMap mapX1,
                         const __grid_constant__ CUtensorMap mapG0, const __grid_constant__ CUtensorMap mapG1,
                         const TokGradParams p)
{
    using Sh = TokGradShape<kMode>;
    constexpr int kStages = Sh::kStages, kAccSets = Sh::kAccSets, kAcc = Sh::kAcc;
    constexpr uint32_t kOffX = Sh::kImgs * kImgBytes;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + kGOffBar);
    uint64_t *x_full = bars + 0, *x_empty = bars + 4, *acc_full = bars + 8, *acc_free = bars + 12;
    uint64_t *img_ready = bars + 16, *img_free = bars + 17, *drain = bars + 18;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 19);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(bars + 20);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int BH = p.B * p.H;
    const int n_items = BH * p.F;  // item = (frame f, chain bh), f major
    const int n_tiles = (p.N + 127) / 128;
    // mode 0: the frame's state S_f; mode 1: the item's two images
    auto mat = [&](int, int it) {
        const int f = it / BH, bh = it % BH;
        return p.W0 + ((size_t)bh * p.F + f) * kStateFloats;
    };
    auto imgs = [&](int it) {
        const int f = it / BH, bh = it % BH;
        return p.img1 + ((size_t)bh * p.F + f) * 2 * kImgBytes;
    };

    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&x_full[i], 1);
            mbar_init(&x_empty[i], 5);  // the tile's MMAs + the four output warps (epilogue reads x1 / x0)
        }
        for (int i = 0; i < kAccSets; ++i) {
            mbar_init(&acc_full[i], 1);
            mbar_init(&acc_free[i], 4);
        }
        mbar_init(img_ready, kMode == 0 ? 4 : 1);
        mbar_init(img_free, 1);
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
            const uint64_t pol = policy_stream();
            int g = 0;  // tiles issued by this CTA
            bool ok = true;
            for (int it = blockIdx.x; it < n_items && ok; it += gridDim.x) {
                const int f = it / BH, bh = it % BH;
                const int b = bh / p.H, h = bh % p.H, bf = b * p.F + f;
                for (int t = 0; t < n_tiles; ++t, ++g) {
                    const int s = g % kStages, u = g / kStages;
                    if (u >= 1 && !(ok = mbar_wait(&x_empty[s], (u - 1) & 1, abort_flag))) break;
                    mbar_arrive_expect_tx(&x_full[s], 2 * kImgBytes);
                    for (int w = 0; w < 2; ++w) {
                        uint8_t *dst = sm + xtile(s, w);
                        const CUtensorMap *m = w ? &mapX1 : &mapX0;
                        tma_load_4d(dst, m, &x_full[s], 0, h, t * 128, bf, pol);
                        tma_load_4d(dst + kImgPanel, m, &x_full[s], 64, h, t * 128, bf, pol);
                    }
                }
            }
            if (*abort_flag)
                for (int s = 0; s < kStages && s < g; ++s) {
                    const int last = ((g - 1 - s) / kStages) * kStages + s;
                    mbar_wait_drain(&x_full[s], (last / kStages) & 1);
                }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            bool ok = true;
            int g = 0, i = 0;  // tiles, items of this CTA
            for (int it = blockIdx.x; it < n_items && ok; it += gridDim.x, ++i) {
                if (!(ok = mbar_wait(img_ready, i & 1, abort_flag))) break;
                tc_fence_after();
                for (int t = 0; t < n_tiles; ++t, ++g) {
                    const int s = g % kStages, u = g / kStages;
                    const int a = g % kAccSets, ua = g / kAccSets;
                    if (!(ok = mbar_wait(&x_full[s], u & 1, abort_flag))) break;
                    if (ua >= 1 && !(ok = mbar_wait(&acc_free[a], (ua - 1) & 1, abort_flag))) break;
                    tc_fence_after();
                    const uint32_t x0 = sbase + xtile(s, 0), x1 = sbase + xtile(s, 1);
                    const uint32_t acc = tmem + 128 * kAcc * a;
#pragma unroll
                    for (int ks = 0; ks < 7; ++ks) {
                        const uint32_t koff = (ks >> 2) * kImgPanel + (ks & 3) * 32;
                        const uint32_t w0 = sbase + kGOffImg + koff;
                        const uint32_t w1 = sbase + kGOffImg + Sh::kImgPer * kImgBytes + koff;
                        const uint64_t a0 = sdesc_sw128(x0 + koff, 16, 1024);
                        mma_bf16(acc, a0, sdesc_sw128(w0, 16, 1024), kIdescK, ks > 0);
                        if (Sh::kLo) mma_bf16(acc, a0, sdesc_sw128(w0 + kImgBytes, 16, 1024), kIdescK, 1u);
                        if (kMode == 1) {
                            // v G: the row-major G image as an MN-major B operand, 16 image rows (K) per step
                            const uint64_t a1 = sdesc_sw128(x1 + koff, 16, 1024);
                            const uint32_t wm = sbase + kGOffImg + kImgBytes + ks * 2048;
                            mma_bf16(acc + 128, a1, sdesc_sw128(wm, kImgPanel, 1024), kIdescKMN, ks > 0);
                            // k G^T: the same image K-major
                            mma_bf16(acc + 256, a0, sdesc_sw128(w1, 16, 1024), kIdescK, ks > 0);
                        }
                    }
                    mma_commit(&acc_full[a]);
                    mma_commit(&x_empty[s]);
                }
                mma_commit(img_free);  // the item's MMAs have read the images
            }
            mma_commit(drain);
            mbar_wait_drain(drain, 0);
        }
    } else if (warp < 6 && kMode == 1) {
        // the item's Dsym_f and G_f images, ready-made by the frame-gradient
        // kernel: two bulk copies once the previous item's MMAs have read the
        // slots.  (Prefetching the next item's images into L2 meanwhile was
        // measured 18 us slower per backward on the 20-head layer.)
        if (warp == 2 && lane == 0) {
            bool ok = true;
            int i = 0, issued = 0;
            for (int it = blockIdx.x; it < n_items && ok; it += gridDim.x, ++i) {
                if (i >= 1 && !(ok = mbar_wait(img_free, (i - 1) & 1, abort_flag))) break;
                mbar_arrive_expect_tx(img_ready, 2 * kImgBytes);
                bulk_g2s(sm + kGOffImg, imgs(it), kImgBytes, img_ready);
                bulk_g2s(sm + kGOffImg + kImgBytes, imgs(it) + kImgBytes, kImgBytes, img_ready);
                ++issued;
            }
            if (*abort_flag && issued) mbar_wait_drain(img_ready, (issued - 1) & 1);
        }
    } else if (warp < 6) {
        // images: row j = column j of S_f, bf16 hi (+ lo); rows and columns
        // 112..127 zero.  Four groups of 32 matrix rows, every load of a group
        // issued before the first conversion.  The next item's matrix is
        // prefetched into L2 while this item's tiles run.
        const int j = (warp & 3) * 32 + lane;
        bool ok = true;
        int i = 0;
        for (int it = blockIdx.x; it < n_items && ok; it += gridDim.x, ++i) {
            if (warp == 2 && lane < Sh::kMats && it + (int)gridDim.x < n_items)
                bulk_prefetch_l2(mat(lane, it + gridDim.x), kStateBytes);
            if (i >= 1 && !(ok = mbar_wait_warp(img_free, (i - 1) & 1, abort_flag))) break;
            const float *Wm[Sh::kMats];
#pragma unroll
            for (int w = 0; w < Sh::kMats; ++w) Wm[w] = mat(w, it);
#pragma unroll 1
            for (int g4 = 0; g4 < 4; ++g4) {
                float x[Sh::kMats][32];
#pragma unroll
                for (int w = 0; w < Sh::kMats; ++w)
#pragma unroll
                    for (int e = 0; e < 32; ++e) {
                        const int r = g4 * 32 + e;
                        x[w][e] = (j < kD && r < kD) ? __ldg(Wm[w] + r * kD + j) : 0.f;
                    }
#pragma unroll
                for (int w = 0; w < Sh::kMats; ++w) {
                    uint8_t *img = sm + kGOffImg + w * Sh::kImgPer * kImgBytes;
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        const int c8 = g4 * 4 + c;
                        const uint32_t off = (c8 >> 3) * kImgPanel + sw128_off(j, c8 & 7);
                        if (Sh::kLo) {
                            uint4 hi, lo;
                            split_bf16x8(&x[w][8 * c], hi, lo);
                            *reinterpret_cast<uint4 *>(img + off) = hi;
                            *reinterpret_cast<uint4 *>(img + kImgBytes + off) = lo;
                        } else {
                            *reinterpret_cast<uint4 *>(img + off) = f32x8_to_bf16(&x[w][8 * c]);
                        }
                    }
                }
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(img_ready);
        }
    } else {
        // output warps: thread = token row r of the tile
        const int quad = warp & 3, r = quad * 32 + lane;
        const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
        uint8_t *stg = sm + kGOffStg + quad * 8192;  // two buffers: output 0 at +0, output 1 at +2048
        int nst = 0;                                  // boxes staged by this warp
        // this thread's row of a 32 x 16 fp32 box, 64-byte swizzle
        auto put16 = [&](uint8_t *box, const float *v) {
#pragma unroll
            for (int c = 0; c < 4; ++c)
                *reinterpret_cast<float4 *>(box + lane * 64 + ((c ^ ((lane >> 1) & 3)) << 4)) =
                    make_float4(v[4 * c], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3]);
        };
        auto stage_begin = [&]() -> uint8_t * {  // the buffer used two boxes ago has been read by its store
            if (lane == 0) bulk_wait_read_le1();
            __syncwarp();
            return stg + (nst & 1) * 4096;
        };
        bool ok = true;
        int g = 0;
        for (int it = blockIdx.x; it < n_items && ok; it += gridDim.x) {
            const int f = it / BH, bh = it % BH;
            const int b = bh / p.H, h = bh % p.H, bf = b * p.F + f;
            for (int t = 0; t < n_tiles; ++t, ++g) {
                const int s = g % kStages;
                const int a = g % kAccSets, ua = g / kAccSets;
                // the row the normalisation applies to: q (x1) in mode 0, k (x0) in mode 1
                const uint8_t *xr = sm + xtile(s, kMode == 0 ? 1 : 0);
                if (ok) ok = mbar_wait_warp(&acc_full[a], ua & 1, abort_flag);
                tc_fence_after();
                const int tok = t * 128 + r;
                const bool live = ok && tok < p.N;
                const bool wlive = ok && t * 128 + quad * 32 < p.N;  // any row of this warp in range
                const size_t rowi = ((size_t)bf * p.N + tok) * p.H + h;
                const uint32_t acc = tmem + 128 * kAcc * a + lane_off;
                auto xrow = [&](int cc, float *o16) {  // 16 bf16 values of this thread's row, columns 16 cc..
                    bf16x8_to_f32(*reinterpret_cast<const uint4 *>(xr + ((2 * cc) >> 3) * kImgPanel +
                                                                   sw128_off(r, (2 * cc) & 7)), o16);
                    bf16x8_to_f32(*reinterpret_cast<const uint4 *>(xr + ((2 * cc + 1) >> 3) * kImgPanel +
                                                                   sw128_off(r, (2 * cc + 1) & 7)), o16 + 8);
                };
                auto stage_end = [&](uint8_t *box, int cc) {
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_4d(&mapG0, box, cc * 16, h, t * 128 + quad * 32, bf);
                        if (kMode == 1) tma_store_4d(&mapG1, box + 2048, cc * 16, h, t * 128 + quad * 32, bf);
                        bulk_commit();
                    }
                    ++nst;
                };
                if (kMode == 0) {
                    // the whole accumulator row in registers: TMEM is free before the stores
                    uint32_t ra[7][16];
#pragma unroll
                    for (int cc = 0; cc < 7; ++cc) tmem_ld16(acc + cc * 16, ra[cc]);
                    tmem_ld_wait();
                    tc_fence_before();
                    __syncwarp();
                    if (ok && lane == 0) mbar_arrive(&acc_free[a]);
                    float sqq = 0.f, sqd = 0.f;
#pragma unroll
                    for (int cc = 0; cc < 7; ++cc) {
                        float xq[16];
                        xrow(cc, xq);
#pragma unroll
                        for (int e = 0; e < 16; ++e) {
                            sqq = fmaf(xq[e], xq[e], sqq);
                            sqd = fmaf(xq[e], __uint_as_float(ra[cc][e]), sqd);
                        }
                    }
                    const float p2 = sqq + kEps, pinv = rsqrtf(p2), corr = sqd / p2;
                    float *dq = p.g0 + rowi * kD;
#pragma unroll
                    for (int cc = 0; cc < 7; ++cc) {
                        float xq[16];
                        xrow(cc, xq);
                        float *o = reinterpret_cast<float *>(ra[cc]);  // dq over its accumulator row
#pragma unroll
                        for (int e = 0; e < 16; ++e) o[e] = pinv * (__uint_as_float(ra[cc][e]) - xq[e] * corr);
                        if (GDN_BWD_TMA_ST) {
                            if (wlive) {
                                uint8_t *box = stage_begin();
                                put16(box, o);
                                stage_end(box, cc);
                            }
                        } else if (live) {
                            float4 *d4 = reinterpret_cast<float4 *>(dq + cc * 16);
#pragma unroll
                            for (int q4 = 0; q4 < 4; ++q4)
                                d4[q4] = make_float4(o[4 * q4], o[4 * q4 + 1], o[4 * q4 + 2], o[4 * q4 + 3]);
                        }
                    }
                    __syncwarp();
                    if (ok && lane == 0) mbar_arrive(&x_empty[s]);
                } else {
                    // two 16-column chunks per TMEM wait; chunk 7 (columns 112..127) is loaded and ignored
                    float skk = 0.f, s2 = 0.f, s3 = 0.f;
#pragma unroll 1
                    for (int cc = 0; cc < 7; cc += 2) {
                        uint32_t r0[2][16], r1[2][16];
#pragma unroll
                        for (int q = 0; q < 2; ++q) {
                            tmem_ld16(acc + (cc + q) * 16, r0[q]);
                            tmem_ld16(acc + 128 + (cc + q) * 16, r1[q]);
                        }
                        tmem_ld_wait();
#pragma unroll
                        for (int q = 0; q < 2; ++q) {
                            if (cc + q >= 7) break;
                            float xk[16];
                            xrow(cc + q, xk);
#pragma unroll
                            for (int e = 0; e < 16; ++e) {
                                skk = fmaf(xk[e], xk[e], skk);
                                s2 = fmaf(xk[e], __uint_as_float(r0[q][e]), s2);
                                s3 = fmaf(xk[e], __uint_as_float(r1[q][e]), s3);
                            }
                        }
                    }
                    const float r2 = skk + kEps, kh = p.c * rsqrtf(r2);  // c / r
                    const float bt = live ? __ldg(p.beta + rowi) : 0.f;
                    const float kdk = bt * (kh * s2 + s3);                // k . dk^
                    const float kc = kdk / r2, btkh = bt * kh;
                    if (live) p.g_beta[rowi] = 0.5f * kh * kh * s2 + kh * s3;
                    float *dk = p.g0 + rowi * kD, *dv = p.g1 + rowi * kD;
#pragma unroll 1
                    for (int cc = 0; cc < 7; cc += 2) {
                        uint32_t r0[2][16], r1[2][16], r2v[2][16];
#pragma unroll
                        for (int q = 0; q < 2; ++q) {
                            tmem_ld16(acc + (cc + q) * 16, r0[q]);
                            tmem_ld16(acc + 128 + (cc + q) * 16, r1[q]);
                            tmem_ld16(acc + 256 + (cc + q) * 16, r2v[q]);
                        }
                        tmem_ld_wait();
#pragma unroll
                        for (int q = 0; q < 2; ++q) {
                            if (cc + q >= 7) break;
                            float xk[16], okv[16], ovv[16];
                            xrow(cc + q, xk);
#pragma unroll
                            for (int e = 0; e < 16; ++e) {
                                const float dkh =
                                    bt * fmaf(kh, __uint_as_float(r0[q][e]), __uint_as_float(r1[q][e]));
                                okv[e] = kh * fmaf(-xk[e], kc, dkh);
                                ovv[e] = btkh * __uint_as_float(r2v[q][e]);
                            }
                            if (GDN_BWD_TMA_ST) {
                                if (wlive) {
                                    uint8_t *box = stage_begin();
                                    put16(box, okv);
                                    put16(box + 2048, ovv);
                                    stage_end(box, cc + q);
                                }
                            } else if (live) {
                                float4 *k4 = reinterpret_cast<float4 *>(dk + (cc + q) * 16);
                                float4 *v4 = reinterpret_cast<float4 *>(dv + (cc + q) * 16);
#pragma unroll
                                for (int q4 = 0; q4 < 4; ++q4) {
                                    k4[q4] = make_float4(okv[4 * q4], okv[4 * q4 + 1], okv[4 * q4 + 2],
                                                         okv[4 * q4 + 3]);
                                    v4[q4] = make_float4(ovv[4 * q4], ovv[4 * q4 + 1], ovv[4 * q4 + 2],
                                                         ovv[4 * q4 + 3]);
                                }
                            }
                        }
                    }
                    tc_fence_before();
                    __syncwarp();
                    if (ok && lane == 0) {
                        mbar_arrive(&acc_free[a]);
                        mbar_arrive(&x_empty[s]);
                    }
                }
            }
        }
        if (lane == 0) bulk_wait_all();  // the staged boxes have been read and written
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
    size_t ws_fwd, ws_G, gamma_G, Sst, Gst, Img1, total;
};

bool bwd_layout(int B, int H, int F, int N, BwdLayout *L)
{
    if (!tc_plan(B, H, F, N, 0, &L->plan) || !tc_plan(B, H, F + 1, N, 0, &L->plan_G)) return false;
    const size_t BH = (size_t)B * H;
    size_t o = 0;
    L->ws_fwd = o; o = up256(o + L->plan.ws_bytes);
    L->ws_G = o; o = up256(o + L->plan_G.ws_bytes);
    L->gamma_G = o; o = up256(o + (size_t)B * (F + 1) * H * 4);
    L->Sst = o; o = up256(o + BH * F * kStateBytes);
    L->Gst = o; o = up256(o + BH * (F + 1) * kStateBytes);
    L->Img1 = o; o = up256(o + BH * F * 2 * (size_t)kImgBytes);
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
    if ((e = cudaFuncSetAttribute(kb_frame_grad_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kFgSmem)) !=
        cudaSuccess)
        return e;
    g_b_attr[dev] = true;
    return cudaSuccess;
}

cudaError_t token_grads(const void *dO, const void *q, const void *k, const void *v, const float *beta,
                        const float *Sst, const uint8_t *img1, float *dq, float *dk, float *dv,
                        float *dbeta, int B, int H, int F, int N, float c, unsigned *status, cudaStream_t stream)
{
    CUtensorMap mdo, mq, mk, mv, mdq, mdk, mdv;
    if (!make_token_map(&mdo, dO, B, H, F, N, 128) || !make_token_map(&mq, q, B, H, F, N, 128) ||
        !make_token_map(&mk, k, B, H, F, N, 128) || !make_token_map(&mv, v, B, H, F, N, 128) ||
        !make_f32_row_map(&mdq, dq, B, H, F, N, 32) || !make_f32_row_map(&mdk, dk, B, H, F, N, 32) ||
        !make_f32_row_map(&mdv, dv, B, H, F, N, 32))
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
    p.img1 = img1;
    p.g0 = dq;
    p.g1 = nullptr;
    p.g_beta = nullptr;
    const int grid = B * H * F < kSms ? B * H * F : kSms;  // persistent: items strided over the CTAs
    kg_token_grad_kernel<0><<<grid, kGThreads, kGSmem, stream>>>(mdo, mq, mdq, mdq, p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    p.W0 = nullptr;
    p.g0 = dk;
    p.g1 = dv;
    p.g_beta = dbeta;
    kg_token_grad_kernel<1><<<grid, kGThreads, kGSmem, stream>>>(mk, mv, mdk, mdv, p);
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
    float *gamma_G = reinterpret_cast<float *>(ws + L.gamma_G);
    float *Sst = reinterpret_cast<float *>(ws + L.Sst), *Gst = reinterpret_cast<float *>(ws + L.Gst);
    uint8_t *img1 = ws + L.Img1;
    uint8_t *ws_rev = ws + L.ws_G + L.plan_G.off_frames;
    // 1. forward statistics (A_f images also into the reverse scan's slots) and every state S_f
    if ((e = launch_frame_stats_tc(k, v, beta, gamma, L.plan, c, 0, ws + L.ws_fwd, status, stream, ws_rev, 0)) !=
        cudaSuccess)
        return e;
    if ((e = launch_states_tc(q, gamma, S_in, nullptr, Sst, L.plan, ws + L.ws_fwd, status, stream)) != cudaSuccess)
        return e;
    // 2. E_f = dO^T q^ through the statistics kernel in its E mode (k := q, v := dO, beta := 1,
    //    c := 1), straight into the reverse scan's slots
    if ((e = launch_frame_stats_tc(q, dO, nullptr, gamma, L.plan, 1.f, 0, ws + L.ws_fwd, status, stream, ws_rev,
                                   1)) != cudaSuccess)
        return e;
    // 3. reverse scan G_{F-1} .. G_0, ending at dS_in
    kb_reverse_edges<<<BH, 256, 0, stream>>>(ws_rev, gamma, gamma_G, B, H, F);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if ((e = launch_chunk_composite_tc(gamma_G, L.plan_G, 0, ws + L.ws_G, status, stream)) != cudaSuccess) return e;
    if ((e = launch_states_tc(q, gamma_G, dS_out, dS_in, Gst, L.plan_G, ws + L.ws_G, status, stream)) != cudaSuccess)
        return e;
    // 4. per-frame dgamma, and Dsym = dA + dA^T and G_f as bf16 images for step 5
    {
        FrameGradParams fp;
        fp.S_in = S_in;
        fp.Sst = Sst;
        fp.Gst = Gst;
        fp.dgamma = dgamma;
        fp.img_out = img1;
        fp.status = status;
        fp.B = B;
        fp.H = H;
        fp.F = F;
        const int items = BH * F;
        kb_frame_grad_tc<<<items < kSms ? items : kSms, kFgThreads, kFgSmem, stream>>>(fp);
    }
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    // 5. token gradients: dq from dO S_f; dk, dv, dbeta from k Dsym_f, v G_f, k G_f^T
    if ((e = token_grads(dO, q, k, v, beta, Sst, img1, dq, dk, dv, dbeta, B, H, F, N, c, status, stream)) !=
        cudaSuccess)
        return e;
    return cudaSuccess;  // dS_in: written by the reverse scan as its final state
}

}  // namespace gdn
