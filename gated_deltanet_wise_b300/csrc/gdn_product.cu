// gdn_product.cu — frame transitions of the token-ordered ("product") reading
// of the frame-wise GDN, head size D = 112, bf16 k/v, fp32 beta/state.
//
// Summary page "SANA-WM: Efficient Minute-Scale World Modeling with Hybrid
// Linear Diffusion Transformer": the frame transition is printed as
// gamma_t I - K^_t beta_t K^_t^T (section 方法步骤详情, module 2), and the layer
// generalises token-wise Gated DeltaNet (section 技术新颖性).  Read with beta_t
// as the UT-transform matrix, the frame's tokens act in order:
//     M_f = gamma_f I - Abar_f,   Abar_f = I - prod_n (I - beta_n k^_n k^_n^T),
//     U_f = W_f = the state the frame's tokens reach from zero,
// and the pair (Abar, W) obeys the delta rule with the keys themselves as
// Abar's values.  Over a sub-chunk of 64 tokens (rows K^, K, V):
//     G   = K^ K^^T,  T = (I + StrictLower(diag(beta) G))^-1 diag(beta),
//     R   = [K^ | V] - K^ [Abar ; W]^T                 (residual rows),
//     X   = T R = diag(beta) R + T_off R                (T_off = T - diag(beta)),
//     [Abar ; W] += X^T K^ = (X diag(c/r))^T K         (raw K: an exact operand).
//
// G and T depend only on the sub-chunk's keys and write strengths, never on the
// running pair, so two kernels split the work:
//   K1t, over all sub-chunks of all frames at once: G on tcgen05 from the raw
//     keys, scaled in fp32 by c/r per token, and T by forward substitution on CUDA
//     cores (one column per thread, in registers); T_off goes to the workspace as
//     an 8 KB bf16 MMA image per sub-chunk;
//   K1p, one CTA per (frame, chain), sub-chunks in order: tcgen05 forms R~ (the
//     product K^ [Abar ; W]^T, N = 2 x 128), T_off R (accumulated on top of the
//     fp32 diag(beta) R stored into TMEM, T_off loaded with the keys) and the pair
//     update (fp32 TMEM accumulators, X split hi + lo).
// Abar is accumulated transposed, so the accumulator's lanes are Abar's columns:
// its bf16 image is then directly the B operand the scan kernel multiplies S by,
// and K1p writes (Abar_f^T image, W_f) in the per-frame workspace format of the
// sum reading's frame-statistics kernel.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>

#include "gdn_internal.h"
#include "gdn_tile.cuh"

namespace gdn {

constexpr int kPC = 64;                                // tokens per sub-chunk
constexpr uint32_t kPPanel = kPC * kRowB;              // 8192: a 64-column panel of a 64-row tile
constexpr int kPThreads = 320;                         // producer, MMA, 8 math warps
// shared memory (1024-aligned regions)
constexpr uint32_t kPOffK = 0;                         // raw K tiles, two buffers of 16 KB
constexpr uint32_t kPOffV = 32768;                     // raw V tiles, two buffers of 16 KB
constexpr uint32_t kPOffKh = 65536;                    // K^ = c/r k (bf16), 64 rows x 2 panels
constexpr uint32_t kPOffSA = 81920;                    // Abar^T image: rows = key j, 2 panels of 64 i (B, MN-major)
constexpr uint32_t kPOffSW = 114688;                   // W image: rows = value i, 2 panels of 64 j (B, K-major)
constexpr uint32_t kPSPanel = 128 * kRowB;             // 16384
constexpr uint32_t kPOffT = 147456;                    // T_off image: 64 rows x 1 panel (+ slack: M = 128 reads)
constexpr uint32_t kPOffR = 163840;                    // R_hi image, then X_hi: 64 rows x 4 panels
constexpr uint32_t kPOffXlo = 196608;                  // G (fp32 64 x 64), then X_lo image
constexpr uint32_t kPOffBar = 229376;
constexpr uint32_t kPOffArr = kPOffBar + 256;          // c/r and beta per token (2 x 64 floats)
constexpr uint32_t kPSmem = kPOffArr + 512 + 1024;
static_assert(kPSmem <= kMaxSmem, "product kernel shared memory");

// TMEM: Abar [0,128), W [128,256), G / R~ / X [256,512)
constexpr uint32_t kPTmA = 0, kPTmW = 128, kPTmX = 256;

constexpr uint32_t kIdG = idesc_bf16(128, 64, false, false);    // G = K^ K^^T
constexpr uint32_t kIdRA = idesc_bf16(128, 128, false, true);   // R~_A = K^ Abar^T (B = Abar^T image)
constexpr uint32_t kIdRW = idesc_bf16(128, 128, false, false);  // R~_W = K^ W^T
constexpr uint32_t kIdX = idesc_bf16(128, 256, false, true);    // X += T_off R
constexpr uint32_t kIdU = idesc_bf16(128, kD, true, true);      // pair += X'^T K


// T = (I + StrictLower(diag(beta) G))^-1 diag(beta) for a 64-token sub-chunk, one
// column e per thread, by forward substitution in right-looking order.  The
// caller passes Ls = -diag(beta) G column-major (Ls[r * 64 + a] = -beta_a G[a][r]),
// so that with t initialised to beta_e e_e each step is only
//     t_a += Ls[a][r] t_r   for every a > r
// (t_r is final once the steps before r are done): the loop-carried path is one
// FMA per step, and the column reads of Ls are broadcast float4s that the fully
// unrolled steps can issue early.  The strictly lower part T_off goes to the
// bf16 image `timg` (64 rows of 128 bytes, 128-byte swizzle: row a, column e),
// the diagonal and above as zeros.  R0 > 0: the caller's columns are all >= R0,
// whose entries above row R0 vanish, so the substitution starts there.
template <int R0>
__device__ __noinline__ void solve_T(const float *Ls, const float *bt, uint8_t *timg_bytes, int e)
{
    const float be = bt[e];
    float tc[kPC];
#pragma unroll
    for (int a = 0; a < kPC; ++a) tc[a] = (a == e) ? be : 0.f;
#pragma unroll
    for (int r = R0; r < kPC; ++r) {
#pragma unroll
        for (int a4 = (r + 1) >> 2; a4 < kPC / 4; ++a4) {
            const float4 l4 = reinterpret_cast<const float4 *>(Ls + r * 64)[a4];  // -beta_a G[a][r], a = 4 a4 ..
            const float lv[4] = {l4.x, l4.y, l4.z, l4.w};
#pragma unroll
            for (int j = 0; j < 4; ++j)
                if (4 * a4 + j > r) tc[4 * a4 + j] = fmaf(lv[j], tc[r], tc[4 * a4 + j]);
        }
    }
    __nv_bfloat16 *timg = reinterpret_cast<__nv_bfloat16 *>(timg_bytes);
#pragma unroll
    for (int a = 0; a < kPC; ++a) {
        const uint32_t off = a * kRowB + ((((uint32_t)e >> 3) ^ (a & 7)) << 4) + (e & 7) * 2;
        timg[off >> 1] = __float2bfloat16_rn(a > e ? tc[a] : 0.f);
    }
}

// ===================================================================== K1t
// The UT transform's T of every 64-token sub-chunk, ahead of the pair chain: T
// depends on the sub-chunk's keys and write strengths only, never on the running
// pair (Abar, W), so all of them are formed here in parallel and K1p reads them.
// Persistent CTAs of kTPairs independent warp pairs; a pair takes sub-chunks in
// turn: TMA the raw key tile, norms r_a, G_raw = K K^T on tcgen05 (exact bf16
// products, fp32 accumulation), G = (c/r_a)(c/r_b) G_raw while reading it out of
// TMEM, the solve, and one bulk store of the 8 KB T_off image.  Pairs of warps
// (2p, 2p + 1) sit in TMEM lane quadrants (0, 1) or (2, 3); a pair of the second
// kind points its MMA's A operand 64 rows before the tile, so that the tile's
// rows, and G's, land in lanes 64..127.
constexpr int kTPairs = 4;
constexpr int kTThreads = kTPairs * 64;                     // 256
constexpr uint32_t kTPairBytes = 49152;                     // two key tiles (16 KB each; a consumed one takes
                                                            // its T_off image), G (16 KB fp32)
constexpr uint32_t kTOffBar = kTPairs * kTPairBytes;        // 196608
constexpr uint32_t kTOffArr = kTOffBar + 256;               // per pair: c/r and beta of 64 tokens
constexpr uint32_t kTSmem = kTOffArr + kTPairs * 512 + 1024;
static_assert(kTSmem <= kMaxSmem, "T pre-pass shared memory");

struct TParams {
    const float *beta;
    uint8_t *ws_T;   // [B*H][F][n_sc] x 8 KB T_off images, by processing position
    unsigned *status;
    int B, H, F, N, n_sc;
    float c;
    int reverse;
};

__device__ __forceinline__ void pair_sync(int p) { asm volatile("bar.sync %0, 64;" ::"r"(p + 1) : "memory"); }
// Barrier over one pair that also ANDs a flag across its 64 threads, so both warps
// take the same branch after a bounded wait.
__device__ __forceinline__ bool pair_sync_and(int p, bool v)
{
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred pi, po;\n\tsetp.ne.u32 pi, %1, 0;\n\tbar.red.and.pred po, %2, 64, pi;\n\tselp.u32 %0, 1, 0, po;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)v), "r"(p + 1)
        : "memory");
    return r != 0;
}

__global__ void __launch_bounds__(kTThreads, 1)
    kt_ut_transform_kernel(const __grid_constant__ CUtensorMap mapK, const TParams p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + kTOffBar);
    uint64_t *kfull = bars, *gfull = bars + 2 * kTPairs;  // kfull[pair][buffer], gfull[pair]
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 3 * kTPairs);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(bars + 3 * kTPairs + 1);
    const int warp = threadIdx.x >> 5;
    const int pr = warp >> 1, tn = threadIdx.x & 63;           // pair, thread within the pair
    const int quad = warp & 3, lg = (quad & 2) * 32;           // TMEM lanes of this pair: lg .. lg + 63
    if (threadIdx.x == 0) {
        for (int i = 0; i < kTPairs; ++i) {
            mbar_init(&kfull[2 * i], 1);
            mbar_init(&kfull[2 * i + 1], 1);
            mbar_init(&gfull[i], 1);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0) {
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

    uint8_t *pbase = sm + pr * kTPairBytes;                    // key tiles 0, 1; G
    float *Gs = reinterpret_cast<float *>(pbase + 32768);
    float *cr = reinterpret_cast<float *>(sm + kTOffArr + pr * 512), *bt = cr + 64;
    const uint32_t pbase_addr = sbase + pr * kTPairBytes;
    const uint32_t dcol = tmem + 64u * pr;                     // this pair's 64 accumulator columns
    const long long items = (long long)p.B * p.H * p.F * p.n_sc;
    const long long stride = (long long)gridDim.x * kTPairs;
    const long long first = (long long)blockIdx.x * kTPairs + pr;
    const uint64_t pol = policy_stream();
    // item -> (chain, processing position, sub-chunk) and the key tile's TMA coordinates
    auto decode = [&](long long item, int &bh, int &f, int &sc, int &h, int &bf) {
        sc = (int)(item % p.n_sc);
        const long long bhf = item / p.n_sc;
        f = (int)(bhf % p.F);
        bh = (int)(bhf / p.F);
        const int b = bh / p.H;
        h = bh % p.H;
        bf = b * p.F + frame_at(f, p.F, p.reverse);
    };
    auto issue_tile = [&](long long item, int buf) {  // leader only
        int bh, f, sc, h, bf;
        decode(item, bh, f, sc, h, bf);
        uint8_t *dst = pbase + buf * 16384;
        mbar_arrive_expect_tx(&kfull[2 * pr + buf], 2 * kPPanel);
        tma_load_4d(dst, &mapK, &kfull[2 * pr + buf], 0, h, sc * kPC, bf, pol);
        tma_load_4d(dst + kPPanel, &mapK, &kfull[2 * pr + buf], 64, h, sc * kPC, bf, pol);
    };
    bool ok = true;
    int k_issued = 0, k_waited = 0;  // (leader) key-tile loads issued / consumed, per pair
    bool g_pending = false;          // (leader) a G MMA not yet waited for
    if (tn == 0 && first < items) {
        issue_tile(first, 0);
        ++k_issued;
    }
    int use = 0;
    for (long long item = first; item < items; item += stride, ++use) {
        int bh, f, sc, h, bf;
        decode(item, bh, f, sc, h, bf);
        const int buf = use & 1;
        uint8_t *kbuf = pbase + buf * 16384;
        const uint32_t kaddr = pbase_addr + buf * 16384;
        const int m = min(kPC, p.N - sc * kPC);
        // (1) the next item's key tile into the other buffer, once the store of the
        //     T_off image that the item before this one left there has read it
        if (tn == 0 && item + stride < items) {
            bulk_wait_read_all();
            issue_tile(item + stride, buf ^ 1);
            ++k_issued;
        }
        bt[tn] = tn < m ? __ldg(p.beta + ((size_t)bf * p.N + sc * kPC + tn) * p.H + h) : 0.f;
        ok = mbar_wait_warp(&kfull[2 * pr + buf], (use >> 1) & 1, abort_flag);
        if (tn == 0 && ok) ++k_waited;
        // (2) G_raw on the tensor cores; c / ||k_a|| per token meanwhile
        if (tn == 0 && ok) {
            tc_fence_after();
            const uint32_t abase = kaddr - (uint32_t)lg * kRowB;  // tile rows land in lanes lg..lg + 63
#pragma unroll
            for (int ks = 0; ks < 7; ++ks) {
                const uint32_t koff = (ks >> 2) * kPPanel + (ks & 3) * 32;
                mma_bf16(dcol, sdesc_sw128(abase + koff, 16, 1024), sdesc_sw128(kaddr + koff, 16, 1024), kIdG, ks > 0);
            }
            mma_commit(&gfull[pr]);
            g_pending = true;
        }
        if (ok) {
            float ss = 0.f;
#pragma unroll
            for (int c8 = 0; c8 < 16; ++c8) {  // both panels of token tn's row (columns 112..127 are zero)
                float f8[8];
                bf16x8_to_f32(*reinterpret_cast<const uint4 *>(kbuf + (c8 >> 3) * kPPanel + sw128_off(tn, c8 & 7)), f8);
#pragma unroll
                for (int e = 0; e < 8; ++e) ss = fmaf(f8[e], f8[e], ss);
            }
            cr[tn] = p.c * rsqrtf(ss + kEps);
        }
        if (!(ok = pair_sync_and(pr, ok))) break;
        // (3) Ls = -diag(beta) G with G = (c/r_a)(c/r_b) G_raw, column-major, from this
        //     thread's TMEM lane (row a = tn)
        ok = mbar_wait_warp(&gfull[pr], use & 1, abort_flag);
        if (tn == 0 && ok) g_pending = false;
        if (ok) {
            tc_fence_after();
            const float ia = -bt[tn] * cr[tn];  // row a = tn of Ls = -beta_a (c/r_a)(c/r_b) G_raw[a][b]
            const uint32_t lane_addr = dcol + ((uint32_t)(lg + (warp & 1) * 32) << 16);
            uint32_t rg[4][16];
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) tmem_ld16(lane_addr + q4 * 16, rg[q4]);
            tmem_ld_wait();
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4)
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const int bcol = q4 * 16 + j;
                    Gs[bcol * 64 + tn] = __uint_as_float(rg[q4][j]) * ia * cr[bcol];
                }
        }
        tc_fence_before();
        if (!(ok = pair_sync_and(pr, ok))) break;
        // (4) the solve (the upper 32 columns start at row 32); the T_off image goes over
        //     the consumed key tile
        if (tn < 32) solve_T<0>(Gs, bt, kbuf, tn);
        else solve_T<32>(Gs, bt, kbuf, tn);
        fence_proxy_async_smem();
        pair_sync(pr);
        if (tn == 0) {
            bulk_s2g(p.ws_T + (size_t)item * 8192, kbuf, 8192);
            bulk_commit();
        }
    }
    if (tn == 0) {  // let this pair's copies and MMA in flight land before the CTA exits
        for (int u = k_waited; u < k_issued; ++u) mbar_wait_drain(&kfull[2 * pr + (u & 1)], (u >> 1) & 1);
        if (g_pending) mbar_wait_drain(&gfull[pr], use & 1);
    }
    if (tn == 0) bulk_wait_all();
    tc_fence_before();
    __syncthreads();
    if (*abort_flag && threadIdx.x == 0) raise_status(p.status);
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

struct ProdParams {
    const float *beta;
    const uint8_t *ws_T; // [BH][F][n_sc] x 8 KB T_off images from the pre-pass
    uint8_t *ws_frames;  // [BH][F] x kFrameWs, by processing position
    unsigned *status;
    int B, H, F, N;
    float c;
    int reverse;  // 1: processing position f holds frame F - 1 - f
};

__global__ void __launch_bounds__(kPThreads, 1)
    kp_frame_product_kernel(const __grid_constant__ CUtensorMap mapK, const __grid_constant__ CUtensorMap mapV,
                            const ProdParams p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + kPOffBar);
    uint64_t *kv_full = bars + 0, *kv_empty = bars + 2, *prep_done = bars + 4;
    uint64_t *simg_ready = bars + 7, *rt_full = bars + 8, *r_ready = bars + 9;
    uint64_t *x_full = bars + 10, *x_ready = bars + 11, *upd_done = bars + 12, *drain = bars + 13;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 14);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(bars + 15);
    float *cr = reinterpret_cast<float *>(sm + kPOffArr);   // c / ||k|| per token
    float *bt = cr + 64;                                     // beta per token (0 past the frame)

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int BH = p.B * p.H;
    const int f = blockIdx.x / BH, bh = blockIdx.x % BH;
    const int b = bh / p.H, h = bh % p.H;
    const int bf = b * p.F + frame_at(f, p.F, p.reverse);  // the frame's tokens; workspace slot f
    const int n_sc = (p.N + kPC - 1) / kPC;

    if (threadIdx.x == 0) {
        for (int i = 0; i < 2; ++i) {
            mbar_init(&kv_full[i], 1);
            mbar_init(&kv_empty[i], 1);
        }
        mbar_init(prep_done, 8);
        mbar_init(simg_ready, 8);
        mbar_init(rt_full, 1);
        mbar_init(r_ready, 8);
        mbar_init(x_full, 1);
        mbar_init(x_ready, 4);
        mbar_init(upd_done, 1);
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

    if (warp == 0) {
        // ------------------------------------------------------ TMA producer
        if (lane == 0) {
            const uint64_t pol = policy_stream();
            int issued = 0;
            for (int sc = 0; sc < n_sc; ++sc) {
                const int kb = sc & 1;
                if (sc >= 2 && !mbar_wait(&kv_empty[kb], ((sc >> 1) - 1) & 1, abort_flag)) break;
                uint8_t *kd = sm + kPOffK + kb * 2 * kPPanel, *vd = sm + kPOffV + kb * 2 * kPPanel;
                mbar_arrive_expect_tx(&kv_full[kb], 4 * kPPanel + 8192);
                tma_load_4d(kd, &mapK, &kv_full[kb], 0, h, sc * kPC, bf, pol);
                tma_load_4d(kd + kPPanel, &mapK, &kv_full[kb], 64, h, sc * kPC, bf, pol);
                tma_load_4d(vd, &mapV, &kv_full[kb], 0, h, sc * kPC, bf, pol);
                tma_load_4d(vd + kPPanel, &mapV, &kv_full[kb], 64, h, sc * kPC, bf, pol);
                bulk_g2s(sm + kPOffT + kb * 8192, p.ws_T + ((size_t)(bh * p.F + f) * n_sc + sc) * 8192, 8192,
                         &kv_full[kb]);
                ++issued;
            }
            if (*abort_flag)  // let loads already in flight land before the CTA exits
                for (int kb = 0; kb < 2 && kb < issued; ++kb) {
                    const int last = ((issued - 1 - kb) / 2) * 2 + kb;
                    mbar_wait_drain(&kv_full[kb], (last >> 1) & 1);
                }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------- MMA issuer
        if (lane == 0) {
            bool ok = true;
            for (int sc = 0; sc < n_sc && ok; ++sc) {
                const int kb = sc & 1, ph = sc & 1;
                const uint32_t kraw = sbase + kPOffK + kb * 2 * kPPanel, kh = sbase + kPOffKh;
                if (!(ok = mbar_wait(prep_done, ph, abort_flag))) break;
                // R~ = K^ [Abar ; W]^T once the pair image is current
                if (!(ok = mbar_wait(simg_ready, ph, abort_flag))) break;
                tc_fence_after();
#pragma unroll
                for (int ks = 0; ks < 7; ++ks) {
                    const uint64_t ad = sdesc_sw128(kh + (ks >> 2) * kPPanel + (ks & 3) * 32, 16, 1024);
                    mma_bf16(tmem + kPTmX, ad, sdesc_sw128(sbase + kPOffSA + ks * 2048, kPSPanel, 1024), kIdRA, ks > 0);
                    mma_bf16(tmem + kPTmX + 128, ad,
                             sdesc_sw128(sbase + kPOffSW + (ks >> 2) * kPSPanel + (ks & 3) * 32, 16, 1024), kIdRW, ks > 0);
                }
                mma_commit(rt_full);
                // X = diag(beta) R (already in TMEM) + T_off R_hi
                if (!(ok = mbar_wait(r_ready, ph, abort_flag))) break;
                tc_fence_after();
#pragma unroll
                for (int ks = 0; ks < kPC / 16; ++ks)  // T_off of this sub-chunk from the pre-pass (rows 64.. unused)
                    mma_bf16(tmem + kPTmX, sdesc_sw128(sbase + kPOffT + kb * 8192 + ks * 32, 16, 1024),
                             sdesc_sw128(sbase + kPOffR + ks * 2048, kPPanel, 1024), kIdX, 1u);
                mma_commit(x_full);
                // pair update (X' = X c/r as hi + lo; all operands token-row tiles, MN-major):
                //   Abar^T += K^T X'_A  (lanes = key j),   W += X'_W^T K  (lanes = value i)
                if (!(ok = mbar_wait(x_ready, ph, abort_flag))) break;
                tc_fence_after();
#pragma unroll
                for (int ks = 0; ks < kPC / 16; ++ks) {
                    const uint64_t kd = sdesc_sw128(kraw + ks * 2048, kPPanel, 1024);
                    const uint32_t acc = (sc > 0 || ks > 0) ? 1u : 0u;
                    const uint32_t oa = ks * 2048, ow = 2 * kPPanel + ks * 2048;
                    mma_bf16(tmem + kPTmA, kd, sdesc_sw128(sbase + kPOffR + oa, kPPanel, 1024), kIdU, acc);
                    mma_bf16(tmem + kPTmA, kd, sdesc_sw128(sbase + kPOffXlo + oa, kPPanel, 1024), kIdU, 1u);
                    mma_bf16(tmem + kPTmW, sdesc_sw128(sbase + kPOffR + ow, kPPanel, 1024), kd, kIdU, acc);
                    mma_bf16(tmem + kPTmW, sdesc_sw128(sbase + kPOffXlo + ow, kPPanel, 1024), kd, kIdU, 1u);
                }
                mma_commit(upd_done);
                mma_commit(&kv_empty[kb]);
            }
            mma_commit(drain);  // every MMA issued above has completed once this phase lands
            mbar_wait_drain(drain, 0);
        }
    } else {
        // ------------------------------------------------------- math warps
        const int t = threadIdx.x - 64;                  // 0..255
        const int quad = warp & 3, g = (warp - 2) >> 2;  // TMEM lane quadrant, column half
        const int row = quad * 32 + lane;                // TMEM lane (token or pair row)
        const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
        const bool tok_warp = quad < 2;                  // lanes 0..63 hold the token-indexed results
        bool ok = true;

        // the pair starts at zero: zero image
        for (int e = t; e < (int)(4 * kPSPanel / 16); e += 256)
            reinterpret_cast<uint4 *>(sm + kPOffSA)[e] = make_uint4(0, 0, 0, 0);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(simg_ready);

        for (int sc = 0; sc < n_sc; ++sc) {
            const int kb = sc & 1, ph = sc & 1;
            const int m = min(kPC, p.N - sc * kPC);  // tokens of this sub-chunk
            uint8_t *kraw = sm + kPOffK + kb * 2 * kPPanel, *vraw = sm + kPOffV + kb * 2 * kPPanel;

            // (1) norms; K^ = c/r k as bf16; c/r and beta per token
            {
                const int r = t >> 2, qq = t & 3;
                const uint32_t off = (qq >> 1) * kPPanel + r * kRowB;
                const float bet = r < m ? __ldg(p.beta + ((size_t)bf * p.N + sc * kPC + r) * p.H + h) : 0.f;
                if (ok) ok = mbar_wait_warp(&kv_full[kb], (sc >> 1) & 1, abort_flag);
                if (ok) {
                    float kf[32];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const uint32_t pos = (((i + qq + r) & 3) + 4 * (qq & 1)) << 4;
                        bf16x8_to_f32(*reinterpret_cast<const uint4 *>(kraw + off + pos), kf + 8 * i);
                    }
                    float ss = 0.f;
#pragma unroll
                    for (int i = 0; i < 32; ++i) ss = fmaf(kf[i], kf[i], ss);
                    ss += __shfl_xor_sync(0xffffffffu, ss, 1);
                    ss += __shfl_xor_sync(0xffffffffu, ss, 2);
                    const float inv = p.c * rsqrtf(ss + kEps);
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const uint32_t pos = (((i + qq + r) & 3) + 4 * (qq & 1)) << 4;
                        float kh[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e) kh[e] = inv * kf[8 * i + e];
                        *reinterpret_cast<uint4 *>(sm + kPOffKh + off + pos) = f32x8_to_bf16(kh);
                    }
                    if (qq == 0) {
                        cr[r] = r < m ? inv : 0.f;
                        bt[r] = bet;
                    }
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(prep_done);
            }

            if (!tok_warp) {
                // (3) T_off comes from the pre-pass with the sub-chunk's keys; these warps have
                //     nothing to do in this step
                __syncwarp();
                if (lane == 0) mbar_arrive(r_ready);
            } else if (tok_warp) {
                // (4) R = [K^ | V] - R~ (row = token): R_hi image for the MMA, and the exact
                //     diag(beta) R written over R~ in TMEM as the start of X.  The key part
                //     takes K^ from its bf16 image, the same values R~ was formed from, so
                //     that R's rounding error scales with R rather than with K^.
                if (ok) ok = mbar_wait_warp(rt_full, ph, abort_flag);
                tc_fence_after();
                if (ok) {
                    const float btt = bt[row];
                    // two 16-column chunks per TMEM round trip (a load's latency, not its
                    // bandwidth, sets this loop's pace)
                    for (int cp = 0; cp < 8; cp += 2) {
                    uint32_t rr2[2][16];
                    tmem_ld16(tmem + lane_off + kPTmX + g * 128 + cp * 16, rr2[0]);
                    tmem_ld16(tmem + lane_off + kPTmX + g * 128 + cp * 16 + 16, rr2[1]);
                    tmem_ld_wait();
#pragma unroll
                    for (int half = 0; half < 2; ++half) {
                        const int cc = cp + half;
                        const int n0 = g * 128 + cc * 16;  // column of [Abar | W] (padded to 128 each)
                        const int y0 = cc * 16;            // column inside K or V
                        const uint32_t *rr = rr2[half];
                        float y[16];
                        if (y0 < kD) {
                            const uint8_t *src = g == 0 ? sm + kPOffKh : vraw;
                            const uint32_t pb = (y0 >> 6) * kPPanel;
                            bf16x8_to_f32(*reinterpret_cast<const uint4 *>(src + pb + sw128_off(row, (y0 & 63) >> 3)), y);
                            bf16x8_to_f32(*reinterpret_cast<const uint4 *>(src + pb + sw128_off(row, ((y0 & 63) >> 3) + 1)),
                                          y + 8);
                        } else {
#pragma unroll
                            for (int j = 0; j < 16; ++j) y[j] = 0.f;
                        }
                        float rv[16];
                        uint32_t xd0[8], xd1[8];
#pragma unroll
                        for (int j = 0; j < 16; ++j) rv[j] = y[j] - __uint_as_float(rr[j]);
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            xd0[j] = __float_as_uint(btt * rv[j]);
                            xd1[j] = __float_as_uint(btt * rv[8 + j]);
                        }
                        tmem_st8(tmem + lane_off + kPTmX + n0, xd0);
                        tmem_st8(tmem + lane_off + kPTmX + n0 + 8, xd1);
                        uint8_t *dst = sm + kPOffR + (n0 >> 6) * kPPanel;
                        *reinterpret_cast<uint4 *>(dst + sw128_off(row, (n0 & 63) >> 3)) = f32x8_to_bf16(rv);
                        *reinterpret_cast<uint4 *>(dst + sw128_off(row, ((n0 & 63) >> 3) + 1)) = f32x8_to_bf16(rv + 8);
                    }
                    }
                    tmem_st_wait();
                }
                fence_proxy_async_smem();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(r_ready);
            }

            // (5) X' = X c/r as hi + lo MMA images (token warps)
            if (tok_warp) {
                if (ok) ok = mbar_wait_warp(x_full, ph, abort_flag);
                tc_fence_after();
                if (ok) {
                    const float crt = cr[row];
                    for (int cp = 0; cp < 8; cp += 2) {  // two chunks per TMEM round trip
                    uint32_t rx2[2][16];
                    tmem_ld16(tmem + lane_off + kPTmX + g * 128 + cp * 16, rx2[0]);
                    tmem_ld16(tmem + lane_off + kPTmX + g * 128 + cp * 16 + 16, rx2[1]);
                    tmem_ld_wait();
#pragma unroll
                    for (int half = 0; half < 2; ++half) {
                        const int cc = cp + half;
                        const int n0 = g * 128 + cc * 16;
                        const uint32_t *rx = rx2[half];
                        float xv[16];
#pragma unroll
                        for (int j = 0; j < 16; ++j) xv[j] = __uint_as_float(rx[j]) * crt;
                        uint4 hi0, lo0, hi1, lo1;
                        split_bf16x8(xv, hi0, lo0);
                        split_bf16x8(xv + 8, hi1, lo1);
                        const uint32_t pb = (n0 >> 6) * kPPanel;
                        const uint32_t o0 = pb + sw128_off(row, (n0 & 63) >> 3), o1 = pb + sw128_off(row, ((n0 & 63) >> 3) + 1);
                        *reinterpret_cast<uint4 *>(sm + kPOffR + o0) = hi0;
                        *reinterpret_cast<uint4 *>(sm + kPOffR + o1) = hi1;
                        *reinterpret_cast<uint4 *>(sm + kPOffXlo + o0) = lo0;
                        *reinterpret_cast<uint4 *>(sm + kPOffXlo + o1) = lo1;
                    }
                    }
                }
                fence_proxy_async_smem();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(x_ready);
            }

            // (6) after the update: refresh the pair images (Abar^T row j from lane j, W row i
            //     from lane i), or after the last sub-chunk write the frame's Abar^T image
            //     (bf16) and W_f (fp32) to the workspace
            if (ok) ok = mbar_wait_warp(upd_done, ph, abort_flag);
            tc_fence_after();
            const bool last = sc + 1 == n_sc;
            uint8_t *ws = p.ws_frames + ((size_t)bh * p.F + f) * kFrameWs;
            float *wsU = reinterpret_cast<float *>(ws + kAimgBytes);
            const int cc0 = g ? 4 : 0, cc1 = g ? 7 : 4;  // 16-column chunks: panel g
            if (ok) {
                for (int cc = cc0; cc < cc1; ++cc) {
                    uint32_t ra[16], rw[16];
                    tmem_ld16(tmem + lane_off + kPTmA + cc * 16, ra);
                    tmem_ld16(tmem + lane_off + kPTmW + cc * 16, rw);
                    tmem_ld_wait();
                    if (row < kD) {
                        float a[16], w[16];
#pragma unroll
                        for (int j = 0; j < 16; ++j) {
                            a[j] = __uint_as_float(ra[j]);
                            w[j] = __uint_as_float(rw[j]);
                        }
                        const int c8 = 2 * (cc & 3);
                        if (!last) {
                            uint8_t *da = sm + kPOffSA + (cc >> 2) * kPSPanel, *dw = sm + kPOffSW + (cc >> 2) * kPSPanel;
                            *reinterpret_cast<uint4 *>(da + sw128_off(row, c8)) = f32x8_to_bf16(a);
                            *reinterpret_cast<uint4 *>(da + sw128_off(row, c8 + 1)) = f32x8_to_bf16(a + 8);
                            *reinterpret_cast<uint4 *>(dw + sw128_off(row, c8)) = f32x8_to_bf16(w);
                            *reinterpret_cast<uint4 *>(dw + sw128_off(row, c8 + 1)) = f32x8_to_bf16(w + 8);
                        } else {
                            uint8_t *dst = ws + (cc >> 2) * kAimgPanel;
                            *reinterpret_cast<uint4 *>(dst + sw128_off(row, c8)) = f32x8_to_bf16(a);
                            *reinterpret_cast<uint4 *>(dst + sw128_off(row, c8 + 1)) = f32x8_to_bf16(a + 8);
                            float4 *u4 = reinterpret_cast<float4 *>(wsU) + (cc * 4) * kD + row;
#pragma unroll
                            for (int j = 0; j < 4; ++j)
                                u4[j * kD] = make_float4(w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
                        }
                    }
                }
                if (last && g == 1 && row < kD) {  // key columns 112..127 of the image: zero
                    *reinterpret_cast<uint4 *>(ws + kAimgPanel + sw128_off(row, 6)) = make_uint4(0, 0, 0, 0);
                    *reinterpret_cast<uint4 *>(ws + kAimgPanel + sw128_off(row, 7)) = make_uint4(0, 0, 0, 0);
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (!last && lane == 0) mbar_arrive(simg_ready);
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

// ===================================================================== K1c
// Chunk composites of the product reading, from the per-frame workspace:
// per (chunk, chain) C = M_{f0} ... M_{f1-1} and H = the state the chunk's
// frames reach from zero, i.e. C <- gamma_f C - C Abar_f, H <- gamma_f H -
// H Abar_f + U_f over the chunk's frames (summary page, section 技术新颖性:
// the C_p / H_p composites).  In the sum reading the frame-statistics kernel
// forms them while it builds A_f; here A_f = Abar_f is not small, so C and H
// enter the GEMM as hi + lo bf16 images (fp32-accurate), against the bf16
// Abar_f^T image the scan kernel also uses.  Four warps hold C's rows and four
// H's rows in fp32 registers.
constexpr int kCThreads = 320;                          // producer, MMA, 4 C warps, 4 H warps
constexpr uint32_t kCOffA = 0;                          // Abar_f^T image (K2 layout)
constexpr uint32_t kCOffImg = 32768;                    // C_hi, C_lo, H_hi, H_lo: 128-row images
constexpr uint32_t kCOffBar = kCOffImg + 4 * kImgBytes; // 163840
constexpr uint32_t kCSmem = kCOffBar + 256 + 1024;

struct CompParams {
    const float *gamma;
    const uint8_t *ws_frames;  // [BH][F] x kFrameWs, by processing position
    float *ws_comp;            // [BH][n_chunks] x (C, H) fp32
    unsigned *status;
    int B, H, F, chunk, n_chunks, reverse;
};

__global__ void __launch_bounds__(kCThreads, 1) kc_chunk_composite_kernel(const CompParams p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + kCOffBar);
    uint64_t *a_full = bars + 0, *a_empty = bars + 1, *s_ready = bars + 2, *acc_full = bars + 3, *drain = bars + 4;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 5);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(bars + 6);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int BH = p.B * p.H;
    const int chunk_idx = blockIdx.x / BH, bh = blockIdx.x % BH;
    const int b = bh / p.H, h = bh % p.H;
    int f_begin, nf;
    chunk_frames(chunk_idx, p.F, p.n_chunks, f_begin, nf);

    if (threadIdx.x == 0) {
        mbar_init(a_full, 1);
        mbar_init(a_empty, 1);
        mbar_init(s_ready, 8);
        mbar_init(acc_full, 1);
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, 256);
        tmem_relinquish();
    }
    // zero the images (rows 112..127 and key columns 112..127 stay zero)
    for (int o = threadIdx.x * 16; o < 4 * (int)kImgBytes; o += kCThreads * 16)
        *reinterpret_cast<uint4 *>(sm + kCOffImg + o) = make_uint4(0, 0, 0, 0);
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t sbase = smem_u32(sm);
    const uint8_t *ws_chain = p.ws_frames + ((size_t)bh * p.F + f_begin) * kFrameWs;

    if (warp == 0) {
        if (lane == 0) {
            int issued = 0;
            bulk_prefetch_l2(ws_chain + kAimgBytes, kUBytes);
            for (int it = 0; it < nf; ++it) {
                if (it >= 1 && !mbar_wait(a_empty, (it - 1) & 1, abort_flag)) break;
                mbar_arrive_expect_tx(a_full, kAimgBytes);
                bulk_g2s(sm + kCOffA, ws_chain + (size_t)it * kFrameWs, kAimgBytes, a_full);
                if (it + 1 < nf) bulk_prefetch_l2(ws_chain + (size_t)(it + 1) * kFrameWs + kAimgBytes, kUBytes);
                ++issued;
            }
            if (*abort_flag && issued) mbar_wait_drain(a_full, (issued - 1) & 1);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            bool ok = true;
            for (int it = 0; it < nf && ok; ++it) {
                if (!(ok = mbar_wait(s_ready, it & 1, abort_flag))) break;
                if (!(ok = mbar_wait(a_full, it & 1, abort_flag))) break;
                tc_fence_after();
#pragma unroll
                for (int ks = 0; ks < 7; ++ks) {
                    const uint32_t koff = (ks >> 2) * kImgPanel + (ks & 3) * 32;
                    const uint64_t bd = sdesc_sw128(sbase + kCOffA + (ks >> 2) * kAimgPanel + (ks & 3) * 32, 16, 1024);
#pragma unroll
                    for (int m = 0; m < 2; ++m) {  // m = 0: C, 1: H
                        const uint32_t img = sbase + kCOffImg + m * 2 * kImgBytes + koff;
                        mma_bf16(tmem + 128 * m, sdesc_sw128(img, 16, 1024), bd, kIdescK, ks > 0);
                        mma_bf16(tmem + 128 * m, sdesc_sw128(img + kImgBytes, 16, 1024), bd, kIdescK, 1);
                    }
                }
                mma_commit(acc_full);
                mma_commit(a_empty);
            }
            mma_commit(drain);
            mbar_wait_drain(drain, 0);
        }
    } else {
        const int m = (warp - 2) >> 2;  // 0: C rows, 1: H rows
        const int quad = warp & 3, row = quad * 32 + lane;
        const int urow = row < kD ? row : 0;
        const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
        uint8_t *img_hi = sm + kCOffImg + m * 2 * kImgBytes, *img_lo = img_hi + kImgBytes;
        float S[kD];
#pragma unroll
        for (int j = 0; j < kD; ++j) S[j] = (m == 0 && row == j) ? 1.f : 0.f;
        auto write_images = [&]() {
            if (row < kD) {
#pragma unroll
                for (int c8 = 0; c8 < kD / 8; ++c8) {
                    uint4 hi, lo;
                    split_bf16x8(S + 8 * c8, hi, lo);
                    const uint32_t off = (c8 >> 3) * kImgPanel + sw128_off(row, c8 & 7);
                    *reinterpret_cast<uint4 *>(img_hi + off) = hi;
                    *reinterpret_cast<uint4 *>(img_lo + off) = lo;
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(s_ready);
        };
        write_images();
        const float *gam = p.gamma + (size_t)b * p.F * p.H + h;
        bool ok = true;
        for (int it = 0; it < nf && ok; ++it) {
            const float g = __ldg(gam + (size_t)frame_at(f_begin + it, p.F, p.reverse) * p.H);
            // S <- gamma S (+ U_f for H) while the GEMM runs, then S <- S - S Abar_f
            if (m == 1) {
                const float4 *U4 =
                    reinterpret_cast<const float4 *>(ws_chain + (size_t)it * kFrameWs + kAimgBytes) + urow;
                float4 ub[2][4];  // 16-column chunks, loaded two ahead of their use
#pragma unroll
                for (int c = 0; c < 2; ++c)
#pragma unroll
                    for (int j = 0; j < 4; ++j) ub[c][j] = __ldg(U4 + (c * 4 + j) * kD);
#pragma unroll
                for (int cc = 0; cc < 7; ++cc) {
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const float4 u4 = ub[cc & 1][j];
                        const int c0 = cc * 16 + 4 * j;
                        S[c0] = fmaf(g, S[c0], u4.x);
                        S[c0 + 1] = fmaf(g, S[c0 + 1], u4.y);
                        S[c0 + 2] = fmaf(g, S[c0 + 2], u4.z);
                        S[c0 + 3] = fmaf(g, S[c0 + 3], u4.w);
                    }
                    if (cc + 2 < 7)
#pragma unroll
                        for (int j = 0; j < 4; ++j) ub[cc & 1][j] = __ldg(U4 + ((cc + 2) * 4 + j) * kD);
                }
            } else {
#pragma unroll
                for (int j = 0; j < kD; ++j) S[j] *= g;
            }
            if (!(ok = mbar_wait_warp(acc_full, it & 1, abort_flag))) break;
            tc_fence_after();
#pragma unroll
            for (int cc = 0; cc < 7; ++cc) {
                uint32_t ra[16];
                tmem_ld16(tmem + 128 * m + lane_off + cc * 16, ra);
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 16; ++j) S[cc * 16 + j] -= __uint_as_float(ra[j]);
            }
            tc_fence_before();
            if (it + 1 < nf) write_images();
        }
        if (ok && row < kD) {
            float *dst = p.ws_comp + ((size_t)bh * p.n_chunks + chunk_idx) * 2 * kStateFloats +
                         (size_t)m * kStateFloats + row * kD;
#pragma unroll
            for (int j = 0; j < kD; j += 4)
                *reinterpret_cast<float4 *>(dst + j) = make_float4(S[j], S[j + 1], S[j + 2], S[j + 3]);
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

// The product reading's T_off images (8 KB per 64-token sub-chunk of every frame
// and chain) follow the plan's workspace.
size_t product_ws_T_offset(const TcPlan &pl) { return (pl.ws_bytes + 255) / 256 * 256; }
size_t product_ws_bytes(const TcPlan &pl)
{
    const size_t n_sc = ((size_t)pl.N + kPC - 1) / kPC;
    return product_ws_T_offset(pl) + (size_t)pl.B * pl.H * pl.F * n_sc * 8192;
}

namespace {
constexpr int kMaxDevP = 64;
bool g_p_attr[kMaxDevP];
bool g_t_attr[kMaxDevP];
bool g_c_attr[kMaxDevP];
}  // namespace

cudaError_t launch_frame_product_tc(const void *k, const void *v, const float *beta, const TcPlan &pl, float c,
                                    int reverse, void *workspace, unsigned *status, cudaStream_t stream)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevP) return cudaErrorInvalidDevice;
    if (!g_p_attr[dev]) {
        e = cudaFuncSetAttribute(kp_frame_product_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kPSmem);
        if (e != cudaSuccess) return e;
        g_p_attr[dev] = true;
    }
    CUtensorMap mk, mv;
    if (!make_token_map(&mk, k, pl.B, pl.H, pl.F, pl.N, kPC) || !make_token_map(&mv, v, pl.B, pl.H, pl.F, pl.N, kPC))
        return cudaErrorInvalidValue;
    // the pre-pass: T_off of every sub-chunk
    const int n_sc = (pl.N + kPC - 1) / kPC;
    uint8_t *ws_T = static_cast<uint8_t *>(workspace) + product_ws_T_offset(pl);
    {
        if (!g_t_attr[dev]) {
            e = cudaFuncSetAttribute(kt_ut_transform_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kTSmem);
            if (e != cudaSuccess) return e;
            g_t_attr[dev] = true;
        }
        TParams tp;
        tp.beta = beta;
        tp.ws_T = ws_T;
        tp.status = status;
        tp.B = pl.B;
        tp.H = pl.H;
        tp.F = pl.F;
        tp.N = pl.N;
        tp.n_sc = n_sc;
        tp.c = c;
        tp.reverse = reverse;
        const long long items = (long long)pl.B * pl.H * pl.F * n_sc;
        const long long ctas = (items + kTPairs - 1) / kTPairs;
        const int grid = (int)(ctas < kSms ? ctas : kSms);
        kt_ut_transform_kernel<<<grid, kTThreads, kTSmem, stream>>>(mk, tp);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    ProdParams p;
    p.beta = beta;
    p.ws_T = ws_T;
    p.ws_frames = static_cast<uint8_t *>(workspace) + pl.off_frames;
    p.status = status;
    p.B = pl.B;
    p.H = pl.H;
    p.F = pl.F;
    p.N = pl.N;
    p.c = c;
    p.reverse = reverse;
    const long long grid = (long long)pl.B * pl.H * pl.F;
    if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    kp_frame_product_kernel<<<(unsigned)grid, kPThreads, kPSmem, stream>>>(mk, mv, p);
    return cudaGetLastError();
}


cudaError_t launch_chunk_composite_tc(const float *gamma, const TcPlan &pl, int reverse, void *workspace,
                                      unsigned *status, cudaStream_t stream)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevP) return cudaErrorInvalidDevice;
    if (!g_c_attr[dev]) {
        e = cudaFuncSetAttribute(kc_chunk_composite_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kCSmem);
        if (e != cudaSuccess) return e;
        g_c_attr[dev] = true;
    }
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    CompParams p;
    p.gamma = gamma;
    p.ws_frames = ws + pl.off_frames;
    p.ws_comp = reinterpret_cast<float *>(ws + pl.off_comp);
    p.status = status;
    p.B = pl.B;
    p.H = pl.H;
    p.F = pl.F;
    p.chunk = pl.chunk;
    p.n_chunks = pl.n_chunks;
    p.reverse = reverse;
    kc_chunk_composite_kernel<<<pl.B * pl.H * pl.n_chunks, kCThreads, kCSmem, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace gdn
