// gdn_step.cu — fused single-frame streaming step of the frame-wise GDN
// (head size D = 112, bf16 q/k/v/o, fp32 beta/gamma/state):
//     A = sum_n beta_n k^_n k^_n^T,  U = sum_n beta_n v_n k^_n^T,
//     S_out = S_in (gamma I - A) + U,  o_n = S_out q^_n
// (summary page "SANA-WM: Efficient Minute-Scale World Modeling with Hybrid
// Linear Diffusion Transformer", section 方法步骤详情 module 2; one latent frame
// per call as in the chunk-wise autoregressive variant of the CSDN article's
// §六 stage 4).
//
// One thread-block cluster per (batch, head) chain, one launch per step.  The
// frame's tokens are split across the cluster's CTAs.  Because S_out is linear
// in the frame's statistics, S_out = gamma S_in + sum_r (U_r - S_in A_r) over
// the CTAs' partials (A_r, U_r), so each CTA applies its own partial and only
// one D x D matrix per CTA crosses the cluster:
//   1. each CTA streams its token slice through shared memory (TMA, a ring of
//      three 64-token stages, all issued up front for slices of <= 192
//      tokens), turns keys into the MMA operands k^ and beta c/r k (bf16 hi +
//      lo) and accumulates A_r and U_r with tcgen05 into TMEM; S_in is loaded
//      into registers meanwhile;
//   2. S_in becomes bf16 hi/lo MMA images, A_r a bf16 image, and tcgen05 forms
//      S_in A_r; the delta U_r - S_in A_r goes to a shared-memory staging
//      matrix;
//   3. each row block of the delta is sent with a bulk copy (the TMA engine,
//      shared::cta -> shared::cluster) to the CTA that owns those rows of
//      S_out; the copies complete on the owner's mbarrier.  The receive
//      buffers overlay the stage rings, so the copies start after a cluster
//      barrier that every CTA passes once its own ring is drained;
//   4. each owner sums the deltas of its rows, adds gamma S_in, writes those
//      rows of S_out to global memory and bulk-copies them, as bf16 hi/lo
//      image rows, into every CTA of the cluster;
//   5. every CTA computes O = Q (S_hi + S_lo)^T for its 128-token tiles of Q,
//      scales rows by 1/||q|| and stores bf16 with TMA.
// The kernel needs no global scratch.  Every CTA reads S_in before the first
// cluster barrier and S_out is written after it, so S_out may alias S_in.  A
// last cluster barrier keeps every CTA resident until no copy can still be
// headed into its shared memory.
#include <cuda.h>
#include <cuda_runtime.h>
#include <math.h>

#include <mutex>

#include "gdn_internal.h"
#include "gdn_tile.cuh"

namespace gdn {

constexpr int kSTS = 64;                                   // tokens per stats stage
constexpr uint32_t kSPanel = kSTS * kRowB;                 // 8192: one 64-column panel of a stage
constexpr uint32_t kSStageBytes = 8 * kSPanel;             // K -> K^, V, B_hi, B_lo (2 panels each)
constexpr uint32_t kSOffK = 0, kSOffV = 2 * kSPanel, kSOffBhi = 4 * kSPanel, kSOffBlo = 6 * kSPanel;
constexpr int kSStages = 3;
constexpr int kSThreads = 320;                             // producer, MMA, 8 math warps
constexpr int kTQ = 128;                                   // tokens per Q/O tile
constexpr int kMaxCluster = 8;                             // portable cluster size limit
// Shared memory.  During the stats phase: stages 0 and 1 at [0, 128 KB),
// the Q tile at [128, 160 KB), stage 2 at [160, 224 KB).  Afterwards the
// first 128 KB hold the receive buffer, the A_r image, the delta staging
// matrix (over the image once it is consumed) and the |q|^2 partial sums,
// and [160, 224 KB) holds the S images (S_in, then S_out).
constexpr uint32_t kSOffQ = 131072;                        // Q tile of even tiles, O written over it
constexpr uint32_t kSOffQ2 = 0;                            // Q tile of odd tiles (over the consumed receive buffer)
constexpr uint32_t kSOffShi = 163840, kSOffSlo = 196608;   // 128-row bf16 images of S (hi, lo)
constexpr uint32_t kSOffRecv = 0;                          // fp32 delta rows: one block per source CTA
constexpr uint32_t kRecvBytes = (kD + kMaxCluster - 1) * kD * 4;  // >= cl * ceil(112 / cl) rows
constexpr uint32_t kSOffAimg = 54272;                      // bf16 K-major image of A_r (112 rows)
constexpr uint32_t kSOffDelta = kSOffAimg;                 // fp32 [112][112] delta staging
constexpr uint32_t kSOffQss = kSOffDelta + (uint32_t)kStateBytes;  // [2 buffers][2 groups][128] |q|^2 parts
constexpr uint32_t kSOffBar = 229376;
constexpr uint32_t kSSmem = kSOffBar + 256 + 1024;
static_assert(kSOffRecv + kRecvBytes <= kSOffAimg, "step smem layout");
static_assert(kSOffQss + 2048 <= 2 * kSStageBytes, "step smem layout");
static_assert(kSOffShi == kSOffQ + kImgBytes && kSOffSlo + kImgBytes == kSOffBar, "step smem layout");
static_assert(kSSmem <= kMaxSmem, "step shared memory budget");
static_assert(kSOffAimg % 1024 == 0 && kSOffQ % 1024 == 0 && kSOffShi % 1024 == 0, "swizzle alignment");

__device__ __forceinline__ uint32_t stage_off(int s) { return s < 2 ? (uint32_t)s * kSStageBytes : kSOffShi; }

// Tensor memory (512 columns): A_r, U_r, S_in A_r, O accumulators, 128 columns each.
constexpr uint32_t kTmA = 0, kTmU = 128, kTmS = 256, kTmO = 384;

// ------------------------------------------------------------ cluster helpers
__device__ __forceinline__ uint32_t cluster_rank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t dsmem_addr(uint32_t local, uint32_t rank)
{
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
    return r;
}

// Bulk copy of `bytes` (multiple of 16, 16-byte aligned ends) from this CTA's
// shared memory into a cluster peer's; completes on the peer's mbarrier.
__device__ __forceinline__ void bulk_s2s_cluster(uint32_t dst_cluster, uint32_t src_cta, uint32_t bytes,
                                                 uint32_t mbar_cluster)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            dst_cluster),
        "r"(src_cta), "r"(bytes), "r"(mbar_cluster)
        : "memory");
}

// Cluster-wide barrier, split in two so that a thread may arrive early and
// wait later.  Every thread of every CTA passes each barrier exactly once,
// on every path (including after an aborted wait), so it always completes.
__device__ __forceinline__ void cluster_arrive() { asm volatile("barrier.cluster.arrive.release;" ::: "memory"); }
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire;" ::: "memory"); }

// Named barrier over the 8 math warps (ids 1.., 0 is __syncthreads).
__device__ __forceinline__ void math_sync() { asm volatile("bar.sync 1, 256;" ::: "memory"); }

// fp32 [rows][112] staging matrices in shared memory: float4 c4 of row `row`
// sits at position c4 ^ ((row >> 1) & 3) of the row, so that eight consecutive
// rows (one shared-memory wavefront of float4 accesses) hit eight different
// 16-byte bank groups although a row is 448 bytes long.  Rows stay
// contiguous, so row blocks can be bulk-copied as they are.
__device__ __forceinline__ int f4_pos(int row, int c4) { return (c4 ^ ((row >> 1) & 3)) << 2; }

struct StepParams {
    const float *beta;   // [B][N][H]
    const float *gamma;  // [B][H]
    const float *S_in;   // [B][H][D][D] or null
    float *S_out;        // [B][H][D][D] or null
    unsigned *status;
    int H, N;
    int cl;              // CTAs per chain (cluster size)
    int tok_per_cta;     // stats tokens per CTA
    float c;             // key scale
};

__global__ void __launch_bounds__(kSThreads, 1)
    k4_frame_step_kernel(const __grid_constant__ CUtensorMap mapK, const __grid_constant__ CUtensorMap mapV,
                         const __grid_constant__ CUtensorMap mapQ, const __grid_constant__ CUtensorMap mapO,
                         const StepParams p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + kSOffBar);
    uint64_t *st_full = bars + 0, *st_prep = bars + 3, *st_empty = bars + 6;
    uint64_t *q_full = bars + 9, *q_empty = bars + 11, *stats_done = bars + 13, *simg_ready = bars + 14;
    uint64_t *aimg_ready = bars + 15, *s_done = bars + 16, *o_full = bars + 17, *o_free = bars + 19;
    uint64_t *recv_full = bars + 21, *sout_full = bars + 22, *drain = bars + 23, *recv_free = bars + 24;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 25);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(bars + 26);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_rank();
    const int bh = blockIdx.x / p.cl;
    const int b = bh / p.H, h = bh % p.H;
    const int tok0 = min(p.N, (int)rank * p.tok_per_cta);
    const int tok1 = min(p.N, tok0 + p.tok_per_cta);
    const int n_st = (tok1 - tok0 + kSTS - 1) / kSTS;
    const int n_tiles = (p.N + kTQ - 1) / kTQ;
    const int my_tiles = n_tiles > (int)rank ? (n_tiles - (int)rank + p.cl - 1) / p.cl : 0;
    const int rows_per = (kD + p.cl - 1) / p.cl;  // rows of S_out each CTA owns
    const int r0 = min(kD, (int)rank * rows_per), r1 = min(kD, r0 + rows_per);

    if (threadIdx.x == 0) {
        for (int i = 0; i < kSStages; ++i) {
            mbar_init(&st_full[i], 1);
            mbar_init(&st_prep[i], 8);
            mbar_init(&st_empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&q_full[i], 1);
            mbar_init(&q_empty[i], 1);
            mbar_init(&o_full[i], 1);
            mbar_init(&o_free[i], 8);
        }
        mbar_init(stats_done, 1);
        mbar_init(simg_ready, 8);
        mbar_init(aimg_ready, 8);
        mbar_init(s_done, 1);
        mbar_init(recv_full, 1);
        mbar_init(sout_full, 9);
        mbar_init(drain, 1);
        mbar_init(recv_free, 8);
        *abort_flag = 0;
        fence_mbar_init();
        // bytes this CTA will receive: its rows of every peer's delta, and
        // every other owner's S_out image rows (hi and lo, two panels each)
        mbar_arrive_expect_tx(recv_full, (uint32_t)(p.cl * (r1 - r0) * kD * 4));
        mbar_arrive_expect_tx(sout_full, (uint32_t)((kD - (r1 - r0)) * kRowB * 4));
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
    // Programmatic dependent launch: the next kernel on the stream may be
    // scheduled now, but this grid reads no global memory (q, k, v, beta,
    // gamma, S_in: any of them may come from the previous kernel, e.g. a
    // projection or the previous step) before that kernel has completed and
    // its writes are visible.  Only the prologue above overlaps its tail.
    griddep_launch_dependents();
    griddep_wait();

    if (warp == 0) {
        // ------------------------------------------------------ TMA producer
        bool ok = true;
        int st_issued = 0, q_issued = 0;
        const uint64_t pol = policy_stream();
        if (lane == 0) {
            for (int st = 0; st < n_st; ++st) {
                const int s = st % kSStages, use = st / kSStages;
                if (st == kSStages && my_tiles > 0) {  // the first Q tile, behind the first ring of K/V
                    mbar_arrive_expect_tx(&q_full[0], kImgBytes);
                    tma_load_4d(sm + kSOffQ, &mapQ, &q_full[0], 0, h, (int)rank * kTQ, b, pol);
                    tma_load_4d(sm + kSOffQ + kImgPanel, &mapQ, &q_full[0], 64, h, (int)rank * kTQ, b, pol);
                    ++q_issued;
                }
                if (st >= kSStages && !(ok = mbar_wait(&st_empty[s], (use - 1) & 1, abort_flag))) break;
                uint8_t *stg = sm + stage_off(s);
                const int row = tok0 + st * kSTS;
                mbar_arrive_expect_tx(&st_full[s], 4 * kSPanel);
                tma_load_4d(stg + kSOffK, &mapK, &st_full[s], 0, h, row, b, pol);
                tma_load_4d(stg + kSOffK + kSPanel, &mapK, &st_full[s], 64, h, row, b, pol);
                tma_load_4d(stg + kSOffV, &mapV, &st_full[s], 0, h, row, b, pol);
                tma_load_4d(stg + kSOffV + kSPanel, &mapV, &st_full[s], 64, h, row, b, pol);
                ++st_issued;
            }
            if (ok && !q_issued && my_tiles > 0) {
                mbar_arrive_expect_tx(&q_full[0], kImgBytes);
                tma_load_4d(sm + kSOffQ, &mapQ, &q_full[0], 0, h, (int)rank * kTQ, b, pol);
                tma_load_4d(sm + kSOffQ + kImgPanel, &mapQ, &q_full[0], 64, h, (int)rank * kTQ, b, pol);
                ++q_issued;
            }
        }
        __syncwarp();
        cluster_arrive();  // B0
        cluster_wait();
        if (lane == 0) {
            // odd tiles go to the second Q buffer, over the receive buffer once the
            // deltas in it are summed; later tiles wait for their buffer's epilogue
            for (int i = 1; ok && i < my_tiles; ++i) {
                const int t = (int)rank + i * p.cl, qb = i & 1;
                if (i == 1) ok = mbar_wait(recv_free, 0, abort_flag);
                else ok = mbar_wait(&q_empty[qb], ((i >> 1) - 1) & 1, abort_flag);
                if (!ok) break;
                uint8_t *dst = sm + (qb ? kSOffQ2 : kSOffQ);
                mbar_arrive_expect_tx(&q_full[qb], kImgBytes);
                tma_load_4d(dst, &mapQ, &q_full[qb], 0, h, t * kTQ, b, pol);
                tma_load_4d(dst + kImgPanel, &mapQ, &q_full[qb], 64, h, t * kTQ, b, pol);
                ++q_issued;
            }
            if (*abort_flag) {  // let copies already in flight land before the CTA exits
                for (int s = 0; s < kSStages && s < st_issued; ++s) {
                    const int last = ((st_issued - 1 - s) / kSStages) * kSStages + s;  // last stage index using s
                    mbar_wait_drain(&st_full[s], (last / kSStages) & 1);
                }
                for (int qb = 0; qb < 2 && qb < q_issued; ++qb) {  // last tile index using buffer qb
                    const int last = ((q_issued - 1 - qb) / 2) * 2 + qb;
                    mbar_wait_drain(&q_full[qb], (last >> 1) & 1);
                }
                mbar_wait_drain(recv_full, 0);
                mbar_wait_drain(sout_full, 0);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------- MMA issuer
        bool ok = true;
        if (lane == 0) {
            for (int st = 0; st < n_st; ++st) {
                const int s = st % kSStages, use = st / kSStages;
                if (!(ok = mbar_wait(&st_prep[s], use & 1, abort_flag))) break;
                tc_fence_after();
                const uint32_t stg = sbase + stage_off(s);
#pragma unroll
                for (int ks = 0; ks < kSTS / 16; ++ks) {
                    const uint32_t o = ks * 2048;
                    const uint64_t bhi = sdesc_sw128(stg + kSOffBhi + o, kSPanel, 1024);
                    const uint64_t blo = sdesc_sw128(stg + kSOffBlo + o, kSPanel, 1024);
                    const uint64_t av = sdesc_sw128(stg + kSOffV + o, kSPanel, 1024);
                    const uint32_t acc = (st > 0 || ks > 0) ? 1u : 0u;
                    mma_bf16(tmem + kTmA, sdesc_sw128(stg + kSOffK + o, kSPanel, 1024), bhi, kIdescMN, acc);
                    mma_bf16(tmem + kTmU, av, bhi, kIdescMN, acc);
                    mma_bf16(tmem + kTmU, av, blo, kIdescMN, 1u);
                }
                mma_commit(&st_empty[s]);
            }
            if (ok) mma_commit(stats_done);
            // S_in A_r, with S_in as hi + lo bf16 images (K-major, contraction over the key index)
            if (ok && n_st > 0) ok = mbar_wait(simg_ready, 0, abort_flag);
            if (ok && n_st > 0 && (ok = mbar_wait(aimg_ready, 0, abort_flag))) {
                tc_fence_after();
#pragma unroll
                for (int ks = 0; ks < 7; ++ks) {
                    const uint32_t koff = (ks >> 2) * kImgPanel + (ks & 3) * 32;
                    const uint64_t bd = sdesc_sw128(sbase + kSOffAimg + (ks >> 2) * kAimgPanel + (ks & 3) * 32, 16, 1024);
                    mma_bf16(tmem + kTmS, sdesc_sw128(sbase + kSOffShi + koff, 16, 1024), bd, kIdescK, ks > 0);
                    mma_bf16(tmem + kTmS, sdesc_sw128(sbase + kSOffSlo + koff, 16, 1024), bd, kIdescK, 1u);
                }
                mma_commit(s_done);
            }
        }
        __syncwarp();
        cluster_arrive();  // B0
        cluster_wait();
        if (lane == 0) {
            // every row of the S_out images is in place: this CTA's own (generic
            // stores, fenced by their writers) and the other owners' (bulk copies)
            if (ok) ok = mbar_wait(sout_full, 0, abort_flag);
            tc_fence_after();
            // tiles alternate between two Q buffers and two accumulators (the
            // second over A_r's consumed columns)
            for (int i = 0; ok && i < my_tiles; ++i) {
                const int qb = i & 1, use = i >> 1;
                if (!(ok = mbar_wait(&q_full[qb], use & 1, abort_flag))) break;
                if (i >= 2 && !(ok = mbar_wait(&o_free[qb], (use - 1) & 1, abort_flag))) break;
                tc_fence_after();
                const uint32_t qa = sbase + (qb ? kSOffQ2 : kSOffQ), acc = tmem + (qb ? kTmA : kTmO);
#pragma unroll
                for (int ks = 0; ks < 7; ++ks) {
                    const uint32_t koff = (ks >> 2) * kImgPanel + (ks & 3) * 32;
                    const uint64_t ad = sdesc_sw128(qa + koff, 16, 1024);
                    mma_bf16(acc, ad, sdesc_sw128(sbase + kSOffShi + koff, 16, 1024), kIdescK, ks > 0);
                    mma_bf16(acc, ad, sdesc_sw128(sbase + kSOffSlo + koff, 16, 1024), kIdescK, 1u);
                }
                mma_commit(&o_full[qb]);
            }
            mma_commit(drain);  // every MMA issued above has completed once this phase lands
            mbar_wait_drain(drain, 0);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------- math warps
        const int t = threadIdx.x - 64;                  // 0..255
        const int quad = warp & 3, g = (warp - 2) >> 2;  // TMEM lane quadrant, column group
        const int row = quad * 32 + lane;
        const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
        const int cc0 = g == 0 ? 0 : 4, cc1 = g == 0 ? 4 : 7;  // 16-column groups: panel 0 or panel 1
        const float *sin = p.S_in ? p.S_in + (size_t)bh * kStateFloats : nullptr;
        bool ok = true;

        // 1. prep: four threads per token, each a quarter of the token's 128
        //    swizzled columns (panel qq>>1, chunks rotated to spread banks).
        //    Rows past this CTA's slice get beta = 0 and contribute nothing.
        {
            const int r = t >> 2, qq = t & 3;
            const uint32_t prep_off = (qq >> 1) * kSPanel + r * kRowB;
            for (int st = 0; st < n_st; ++st) {
                const int s = st % kSStages, use = st / kSStages;
                const int n = tok0 + st * kSTS + r;
                const float bt = n < tok1 ? __ldg(p.beta + ((size_t)b * p.N + n) * p.H + h) : 0.f;
                if (!(ok = mbar_wait_warp(&st_full[s], use & 1, abort_flag))) break;
                uint8_t *stg = sm + stage_off(s) + prep_off;
                float kf[32];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const uint32_t pos = (((i + qq + r) & 3) + 4 * (qq & 1)) << 4;
                    bf16x8_to_f32(*reinterpret_cast<const uint4 *>(stg + kSOffK + pos), kf + 8 * i);
                }
                float ss = 0.f;
#pragma unroll
                for (int i = 0; i < 32; ++i) ss = fmaf(kf[i], kf[i], ss);
                ss += __shfl_xor_sync(0xffffffffu, ss, 1);
                ss += __shfl_xor_sync(0xffffffffu, ss, 2);
                const float inv = p.c * rsqrtf(ss + kEps);  // c / ||k||
                const float wb = bt * inv;                  // beta c / ||k||
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const uint32_t pos = (((i + qq + r) & 3) + 4 * (qq & 1)) << 4;
                    float kh[8], y[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        kh[e] = inv * kf[8 * i + e];
                        y[e] = wb * kf[8 * i + e];
                    }
                    uint4 hi, lo;
                    split_bf16x8(y, hi, lo);
                    *reinterpret_cast<uint4 *>(stg + kSOffK + pos) = f32x8_to_bf16(kh);
                    *reinterpret_cast<uint4 *>(stg + kSOffBhi + pos) = hi;
                    *reinterpret_cast<uint4 *>(stg + kSOffBlo + pos) = lo;
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&st_prep[s]);
            }
        }

        // 2b. S_in into registers for its images
        constexpr int kIt = (kD * 14 + 255) / 256;
        float4 x0[kIt], x1[kIt];
#pragma unroll
        for (int it = 0; it < kIt; ++it) {
            const int e = t + it * 256, rr = e / 14, c8 = e % 14;
            x0[it] = x1[it] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (sin && e < kD * 14) {
                x0[it] = __ldg(reinterpret_cast<const float4 *>(sin + rr * kD + c8 * 8));
                x1[it] = __ldg(reinterpret_cast<const float4 *>(sin + rr * kD + c8 * 8 + 4));
            }
        }

        // 3. the ring is drained: S_in images over stage 2, A_r image over stage 0
        if (ok) ok = mbar_wait_warp(stats_done, 0, abort_flag);
        tc_fence_after();
        cluster_arrive();  // B0: peers may copy into this CTA's receive buffer once all arrived
#pragma unroll
        for (int it = 0; it < kIt; ++it) {
            const int e = t + it * 256, rr = e / 14, c8 = e % 14;
            if (e >= kD * 14) break;
            const float x[8] = {x0[it].x, x0[it].y, x0[it].z, x0[it].w, x1[it].x, x1[it].y, x1[it].z, x1[it].w};
            uint4 hi, lo;
            split_bf16x8(x, hi, lo);
            const uint32_t off = (c8 >> 3) * kImgPanel + sw128_off(rr, c8 & 7);
            *reinterpret_cast<uint4 *>(sm + kSOffShi + off) = hi;
            *reinterpret_cast<uint4 *>(sm + kSOffSlo + off) = lo;
        }
        for (int e = t; e < 2 * 2 * 16 * 8; e += 256) {  // rows 112..127 of the S images: zero
            const int img = e >> 8, pan = (e >> 7) & 1, rr = 112 + ((e >> 3) & 15), ch = e & 7;
            *reinterpret_cast<uint4 *>(sm + (img ? kSOffSlo : kSOffShi) + pan * kImgPanel + rr * kRowB + ch * 16) =
                make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(simg_ready);
        if (ok && n_st > 0) {
            for (int cc = cc0; cc < cc1; ++cc) {
                uint32_t ra[16];
                tmem_ld16(tmem + lane_off + kTmA + cc * 16, ra);
                tmem_ld_wait();
                if (row < kD) {
                    float a[16];
#pragma unroll
                    for (int j = 0; j < 16; ++j) a[j] = __uint_as_float(ra[j]);
                    uint8_t *dst = sm + kSOffAimg + (cc >> 2) * kAimgPanel;
                    *reinterpret_cast<uint4 *>(dst + sw128_off(row, 2 * (cc & 3))) = f32x8_to_bf16(a);
                    *reinterpret_cast<uint4 *>(dst + sw128_off(row, 2 * (cc & 3) + 1)) = f32x8_to_bf16(a + 8);
                }
            }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(aimg_ready);

        // 4. delta_r = U_r - S_in A_r into the staging matrix (over the consumed
        //    A_r image), then one bulk copy per owner of its row block
        if (ok && n_st > 0) ok = mbar_wait_warp(s_done, 0, abort_flag);
        tc_fence_after();
        {
            float *dl = reinterpret_cast<float *>(sm + kSOffDelta);
            for (int cc = cc0; cc < cc1; ++cc) {
                uint32_t ru[16], rs[16];
                if (ok && n_st > 0) {  // TMEM loads are warp-collective: all lanes load
                    tmem_ld16(tmem + lane_off + kTmU + cc * 16, ru);
                    tmem_ld16(tmem + lane_off + kTmS + cc * 16, rs);
                    tmem_ld_wait();
                } else {  // no tokens in this CTA (or aborted): a zero delta
#pragma unroll
                    for (int j = 0; j < 16; ++j) ru[j] = rs[j] = 0u;
                }
                if (row < kD) {
#pragma unroll
                    for (int j = 0; j < 16; j += 4)
                        *reinterpret_cast<float4 *>(dl + row * kD + f4_pos(row, cc * 4 + j / 4)) =
                            make_float4(__uint_as_float(ru[j]) - __uint_as_float(rs[j]),
                                        __uint_as_float(ru[j + 1]) - __uint_as_float(rs[j + 1]),
                                        __uint_as_float(ru[j + 2]) - __uint_as_float(rs[j + 2]),
                                        __uint_as_float(ru[j + 3]) - __uint_as_float(rs[j + 3]));
                }
            }
        }
        fence_proxy_async_smem();  // the bulk copies read the staging through the async proxy
        math_sync();
        cluster_wait();  // B0
        if (t == 0) {
            for (int q = 0; q < p.cl; ++q) {
                const int q0 = min(kD, q * rows_per), q1 = min(kD, q0 + rows_per);
                if (q1 <= q0) continue;
                bulk_s2s_cluster(dsmem_addr(sbase + kSOffRecv + (uint32_t)((int)rank * rows_per * kD * 4), q),
                                 sbase + kSOffDelta + (uint32_t)(q0 * kD * 4), (uint32_t)((q1 - q0) * kD * 4),
                                 dsmem_addr(smem_u32(recv_full), q));
            }
        }

        // 5. owned rows: S_out = gamma S_in + the peers' deltas; to global memory,
        //    and as hi/lo image rows into this CTA and, by bulk copies, the others.
        //    The S_in values of this thread's first item and gamma are loaded
        //    while the deltas are still arriving.
        const int n8 = (r1 - r0) * 14;
        float4 pre0 = make_float4(0.f, 0.f, 0.f, 0.f), pre1 = pre0;
        if (sin && t < n8) {
            const int rw = r0 + t / 14, c8 = t % 14;
            pre0 = __ldg(reinterpret_cast<const float4 *>(sin + rw * kD + c8 * 8));
            pre1 = __ldg(reinterpret_cast<const float4 *>(sin + rw * kD + c8 * 8 + 4));
        }
        const float gam = __ldg(p.gamma + (size_t)b * p.H + h);
        if (ok) ok = mbar_wait_warp(recv_full, 0, abort_flag);
        {
            float *sout = p.S_out ? p.S_out + (size_t)bh * kStateFloats : nullptr;
            const float *recv = reinterpret_cast<const float *>(sm + kSOffRecv);
            for (int e = t; e < n8; e += 256) {
                const int lr = e / 14, c8 = e % 14, rw = r0 + lr;
                float4 a0 = pre0, a1 = pre1;
                if (sin && e != t) {
                    a0 = __ldg(reinterpret_cast<const float4 *>(sin + rw * kD + c8 * 8));
                    a1 = __ldg(reinterpret_cast<const float4 *>(sin + rw * kD + c8 * 8 + 4));
                }
                float x[8] = {gam * a0.x, gam * a0.y, gam * a0.z, gam * a0.w,
                              gam * a1.x, gam * a1.y, gam * a1.z, gam * a1.w};
                for (int src = 0; src < p.cl; ++src) {
                    const float *rrow = recv + (src * rows_per + lr) * kD;
                    const float4 d0 = *reinterpret_cast<const float4 *>(rrow + f4_pos(rw, 2 * c8));
                    const float4 d1 = *reinterpret_cast<const float4 *>(rrow + f4_pos(rw, 2 * c8 + 1));
                    x[0] += d0.x;
                    x[1] += d0.y;
                    x[2] += d0.z;
                    x[3] += d0.w;
                    x[4] += d1.x;
                    x[5] += d1.y;
                    x[6] += d1.z;
                    x[7] += d1.w;
                }
                if (sout && ok) {
                    *reinterpret_cast<float4 *>(sout + rw * kD + c8 * 8) = make_float4(x[0], x[1], x[2], x[3]);
                    *reinterpret_cast<float4 *>(sout + rw * kD + c8 * 8 + 4) = make_float4(x[4], x[5], x[6], x[7]);
                }
                uint4 hi, lo;
                split_bf16x8(x, hi, lo);
                const uint32_t off = (c8 >> 3) * kImgPanel + sw128_off(rw, c8 & 7);
                *reinterpret_cast<uint4 *>(sm + kSOffShi + off) = hi;
                *reinterpret_cast<uint4 *>(sm + kSOffSlo + off) = lo;
            }
        }
        fence_proxy_async_smem();
        math_sync();
        __syncwarp();
        if (lane == 0) {
            mbar_arrive(sout_full);  // this CTA's own rows are in place
            mbar_arrive(recv_free);  // the receive buffer may take the second Q tile
        }
        if (t == 0 && r1 > r0) {
            const uint32_t bytes = (uint32_t)(r1 - r0) * kRowB;
            for (int q = 0; q < p.cl; ++q) {
                if (q == (int)rank) continue;
                const uint32_t mb = dsmem_addr(smem_u32(sout_full), q);
#pragma unroll
                for (int part = 0; part < 4; ++part) {
                    const uint32_t off =
                        (part >> 1 ? kSOffSlo : kSOffShi) + (part & 1) * kImgPanel + (uint32_t)r0 * kRowB;
                    bulk_s2s_cluster(dsmem_addr(sbase + off, q), sbase + off, bytes, mb);
                }
            }
        }

        // 6. O = Q S_out^T per 128-token tile, rows scaled by 1/||q||, bf16 over
        //    the Q tile, TMA store.  Every math warp runs every iteration (work
        //    skipped after an abort), so the named barrier inside always sees
        //    all 256 threads.
        float *ssp = reinterpret_cast<float *>(sm + kSOffQss);  // [2 buffers][2 column groups][128 rows]
        for (int i = 0; i < my_tiles; ++i) {
            const int tile = (int)rank + i * p.cl, qb = i & 1, use = i >> 1;
            uint8_t *qs = sm + (qb ? kSOffQ2 : kSOffQ);
            // |q|^2 of this thread's row from the Q tile, while the MMA runs
            if (ok) ok = mbar_wait_warp(&q_full[qb], use & 1, abort_flag);
            float ss = 0.f;
            if (ok) {
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    float f8[8];
                    bf16x8_to_f32(*reinterpret_cast<const uint4 *>(qs + g * kImgPanel + sw128_off(row, c)), f8);
#pragma unroll
                    for (int e = 0; e < 8; ++e) ss = fmaf(f8[e], f8[e], ss);
                }
            }
            ssp[qb * 256 + g * 128 + row] = ss;
            math_sync();
            if (ok) ok = mbar_wait_warp(&o_full[qb], use & 1, abort_flag);
            tc_fence_after();
            const float rq = rsqrtf(ssp[qb * 256 + row] + ssp[qb * 256 + 128 + row] + kEps);
            if (ok) {
                const uint32_t acc = tmem + lane_off + (qb ? kTmA : kTmO);
                for (int cc = cc0; cc < cc1; ++cc) {
                    uint32_t ra[16];
                    tmem_ld16(acc + cc * 16, ra);
                    tmem_ld_wait();
                    float o[16];
#pragma unroll
                    for (int j = 0; j < 16; ++j) o[j] = __uint_as_float(ra[j]) * rq;
                    const int c8 = cc * 2;
                    *reinterpret_cast<uint4 *>(qs + (c8 >> 3) * kImgPanel + sw128_off(row, c8 & 7)) =
                        f32x8_to_bf16(o);
                    *reinterpret_cast<uint4 *>(qs + ((c8 + 1) >> 3) * kImgPanel + sw128_off(row, (c8 + 1) & 7)) =
                        f32x8_to_bf16(o + 8);
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0 && ok) mbar_arrive(&o_free[qb]);
            math_sync();  // the whole tile is in shared memory: one thread stores it as two 128-row boxes
            if (t == 0 && ok) {
                tma_store_4d(&mapO, qs, 0, h, tile * kTQ, b);
                tma_store_4d(&mapO, qs + kImgPanel, 64, h, tile * kTQ, b);
                bulk_commit();
                bulk_wait_read_all();
                mbar_arrive(&q_empty[qb]);
            }
        }
        if (lane == 0) bulk_wait_all();
    }
    // No CTA leaves while a peer may still copy into its shared memory.
    cluster_arrive();
    cluster_wait();
    tc_fence_before();
    __syncthreads();
    if (*abort_flag && threadIdx.x == 0 && p.status) atomicOr(p.status, kStatusTimeout);
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// ================================================================= host side
namespace {

constexpr int kMaxDev = 64;
constexpr int kMaxCl = 8;
std::mutex g_step_mu;
bool g_step_attr[kMaxDev];
int g_max_clusters[kMaxDev][kMaxCl + 1];  // 0 = not queried, -1 = unavailable

cudaError_t prepare_device(int dev)
{
    std::lock_guard<std::mutex> lk(g_step_mu);
    if (g_step_attr[dev]) return cudaSuccess;
    cudaError_t e =
        cudaFuncSetAttribute(k4_frame_step_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSSmem);
    if (e != cudaSuccess) return e;
    for (int cl = 1; cl <= kMaxCl; ++cl) {
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = cl;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.gridDim = dim3(cl * 64);
        cfg.blockDim = dim3(kSThreads);
        cfg.dynamicSmemBytes = kSSmem;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, k4_frame_step_kernel, &cfg) != cudaSuccess || n <= 0) {
            (void)cudaGetLastError();
            n = -1;
        }
        g_max_clusters[dev][cl] = n;
    }
    g_step_attr[dev] = true;
    return cudaSuccess;
}

}  // namespace

// Cluster size per chain: the one that minimises (waves of co-resident
// clusters) x (tokens a CTA streams: its stats slice plus its output tiles),
// with a fixed per-CTA charge for the reduction and the state update.
bool step_plan(int BH, int N, int dev, int *cl_out, int *tok_per_cta_out)
{
    if (dev < 0 || dev >= kMaxDev || BH <= 0 || N <= 0) return false;
    const int n_tiles = (N + kTQ - 1) / kTQ;
    double best = 1e300;
    int best_cl = 0, best_tok = 0;
    for (int cl = 1; cl <= kMaxCl; ++cl) {
        const int active = g_max_clusters[dev][cl];
        if (active <= 0) continue;
        const int per = (N + cl - 1) / cl;
        const int tiles = (n_tiles + cl - 1) / cl;
        const long long waves = ((long long)BH + active - 1) / active;
        const double cost = (double)waves * (per + tiles * kTQ + 256);
        if (cost < best - 1e-9) {
            best = cost;
            best_cl = cl;
            best_tok = per;
        }
    }
    if (!best_cl) return false;
    *cl_out = best_cl;
    *tok_per_cta_out = best_tok;
    return true;
}

cudaError_t launch_frame_step_tc(const void *q, const void *k, const void *v, const float *beta,
                                 const float *gamma, const float *S_in, float *S_out, void *o, int B, int H, int N,
                                 float c, unsigned *status, cudaStream_t stream)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDev) return cudaErrorInvalidDevice;
    if ((e = prepare_device(dev)) != cudaSuccess) return e;
    const int BH = B * H;
    int cl = 0, per = 0;
    if (!step_plan(BH, N, dev, &cl, &per)) return cudaErrorInvalidConfiguration;
    CUtensorMap mk, mv, mq, mo;
    if (!make_token_map(&mk, k, B, H, 1, N, kSTS) || !make_token_map(&mv, v, B, H, 1, N, kSTS) ||
        !make_token_map(&mq, q, B, H, 1, N, kTQ) || !make_token_map(&mo, o, B, H, 1, N, kTQ))
        return cudaErrorInvalidValue;
    StepParams p;
    p.beta = beta;
    p.gamma = gamma;
    p.S_in = S_in;
    p.S_out = S_out;
    p.status = status;
    p.H = H;
    p.N = N;
    p.cl = cl;
    p.tok_per_cta = per;
    p.c = c;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cl;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // prologue overlaps the previous kernel
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3((unsigned)(BH * cl));
    cfg.blockDim = dim3(kSThreads);
    cfg.dynamicSmemBytes = kSSmem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, k4_frame_step_kernel, mk, mv, mq, mo, p);
}

}  // namespace gdn
