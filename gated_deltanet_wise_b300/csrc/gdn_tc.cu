// gdn_tc.cu — tensor-core (tcgen05 + TMA) path of the frame-wise GDN forward,
// head size D = 112, bf16 q/k/v/o, fp32 beta/gamma/state.
//
// The method (summary page "SANA-WM: Efficient Minute-Scale World Modeling with
// Hybrid Linear Diffusion Transformer", section 方法步骤详情, module 2):
//   A_f = sum_n beta_n k^_n k^_n^T,  U_f = sum_n beta_n v_n k^_n^T,
//   S_f = S_{f-1} (gamma_f I - A_f) + U_f,   o_{f,n} = S_f q^_n,
// k^ = k / ||k|| * c, q^ = q / ||q||.  The frame axis is cut into chunks of L
// frames; a chunk's transition composite C = prod M_f and input composite
// H (state reached from zero) let every chunk find its start state with a short
// prefix scan — the C_p / H_p composites of the same page's section 技术新颖性,
// used here across SMs instead of across GPUs.
//
// Three launches:
//   K1 (frame statistics), one CTA per (chunk, chain): streams K and V through
//      shared memory in 32-token stages; CUDA cores turn each key into the MMA
//      operands k^ = c/r k (in place) and B = beta c/r k (as bf16 hi + lo);
//      tcgen05 accumulates A_f = K^^T B_hi and U_f = V^T (B_hi + B_lo) in
//      TMEM, with the raw V tile as an operand.  It writes
//      A_f (bf16, as the MMA-ready image) and U_f (fp32) to the workspace and
//      folds the chunk composite (C, H), held in TMEM, with two more MMAs per
//      frame whose A operands (-bf16 C, -bf16 H) are staged in TMEM as well.
//   K1b (chunk boundaries), row-parallel fp32: S_start(c+1) = S_start(c) C_c + H_c.
//   K2 (state scan + output), one CTA per (chunk, chain): walks the chunk's
//      frames with S in fp32 registers, S_f = gamma S - (S_hi + S_lo) A_f + U_f
//      on tcgen05, and computes O = Q (S_hi + S_lo)^T for 128-token tiles of Q
//      (TMA in, TMA out), scaling each row by 1/||q|| in the epilogue.
//
// Precision: raw bf16 v and q are exact MMA operands; the per-token fp32
// weight beta c/r is folded into the key operand B; U (the part of S that
// matters) uses a hi/lo bf16 split of B, and O uses a hi/lo split of S, so
// the only unavoidable rounding is the bf16 output.  A_f itself is ~1/D in
// norm, so bf16 roundings of its operands, of A_f and of C/H in the composite
// products stay at ~u/D relative.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <math.h>

#include "gdn_internal.h"
#include "gdn_tile.cuh"

namespace gdn {

// ------------------------------------------------------------------ sizes
// K1
#ifndef GDN_K1_TS
#define GDN_K1_TS 64
#endif
#ifndef GDN_K1_STAGES
#define GDN_K1_STAGES 4
#endif
#ifndef GDN_K1_LO
#define GDN_K1_LO 0
#endif
#ifndef GDN_WS_L2HINT
#define GDN_WS_L2HINT 1
#endif
// K1 writes the per-frame workspace with an evict-last L2 policy (its k, v reads
// and K2's q reads are evict-normal), so that part of the 190 MB workspace of the
// 20-head layer is still in the 126 MB L2 when K2 reads it: K2 246 -> 241 us.
constexpr bool kWsKeepL2 = GDN_WS_L2HINT != 0;
constexpr int kTS = GDN_K1_TS;                        // tokens per stage (one TMA box height)
constexpr bool kK1Lo = GDN_K1_LO != 0;                // B as bf16 hi + lo (fp32-accurate U_f)
constexpr uint32_t kTSPanel = kTS * kRowB;            // one 64-column panel of a stage
constexpr uint32_t kStageBytes = (kK1Lo ? 8 : 6) * kTSPanel;  // K->K^, V, B_hi[, B_lo] (2 panels each)
constexpr uint32_t kOffK = 0, kOffV = 2 * kTSPanel, kOffBhi = 4 * kTSPanel, kOffBlo = 6 * kTSPanel;
constexpr int kK1Stages = GDN_K1_STAGES;
static_assert(kTS % 32 == 0 && kTS <= 128, "K1 stage height");
constexpr int kK1Threads = 448;                       // producer, MMA, 2 x 4 prep warps, 4 epilogue warps
constexpr uint32_t kK1OffAimg = kK1Stages * kStageBytes;   // 196608
constexpr uint32_t kK1OffBar = kK1OffAimg + kAimgBytes;    // 225280
constexpr uint32_t kK1Smem = kK1OffBar + 256 + 1024;

// K2
constexpr int kTQ = 128;                              // tokens per Q/O tile
// Three Q tiles in flight and one output staging tile (the most that fits beside
// the A_f image and the S images): with the token rows under an evict-normal L2
// policy the Q stream is bound by its depth, K2 213 -> 193 us against two and two.
#ifndef GDN_K2_QSTAGES
#define GDN_K2_QSTAGES 3
#endif
#ifndef GDN_K2_OSTAGES
#define GDN_K2_OSTAGES 1
#endif
#ifndef GDN_K2_SLO
#define GDN_K2_SLO 1
#endif
#ifndef GDN_K2_SBUF
#define GDN_K2_SBUF 1
#endif
constexpr int kK2QStages = GDN_K2_QSTAGES;            // Q tiles in flight
constexpr int kK2OStages = GDN_K2_OSTAGES;            // output staging tiles (0: rows stored from registers)
constexpr bool kK2Lo = GDN_K2_SLO != 0;               // S as bf16 hi + lo images
constexpr int kK2SBuf = GDN_K2_SBUF;                  // S image sets (2: the next state's images are
                                                      // written while the previous frame's outputs run)
static_assert(kK2QStages >= 2 && kK2QStages <= 4 && kK2OStages >= 0 && kK2OStages <= 2, "K2 rings");
static_assert(kK2SBuf == 1 || kK2SBuf == 2, "K2 S image sets");
#ifndef GDN_K2_SW8
#define GDN_K2_SW8 0
#endif
constexpr int kK2StateWarps = GDN_K2_SW8 ? 8 : 4;     // 8: every state row split over two warps
constexpr int kK2Threads = kK2StateWarps == 8 ? 448 : 320;  // producers, MMA, state warps, 4 output warps
constexpr uint32_t kK2OffO = kK2QStages * kImgBytes;       // output staging tiles
constexpr uint32_t kK2OffA = kK2OffO + kK2OStages * kImgBytes;
constexpr uint32_t kK2SetBytes = (kK2Lo ? 2 : 1) * kImgBytes;  // one S image set: hi [, lo]
constexpr uint32_t kK2OffShi = kK2OffA + kAimgBytes;
constexpr uint32_t kK2OffSlo = kK2OffShi + kImgBytes;      // lo image of set 0 (set i at + i * kK2SetBytes)
constexpr uint32_t kK2OffBar = kK2OffShi + kK2SBuf * kK2SetBytes;
constexpr uint32_t kK2Smem = kK2OffBar + 256 + 1024;
static_assert(kK2OffShi % 1024 == 0 && kK2OffA % 1024 == 0, "K2 smem layout");
static_assert(kK1Smem <= kMaxSmem && kK2Smem <= kMaxSmem, "shared memory budget");

// ===================================================================== K1
struct K1Params {
    const float *beta;
    const float *gamma;
    uint8_t *ws_frames;  // [BH][F] x kFrameWs
    float *ws_comp;      // [BH][n_chunks] x (C, H) fp32
    unsigned *status;
    int B, H, F, N, chunk, n_chunks;
    float c;
    int reverse;  // 1: frames are visited from the last to the first
    int withhold_loads;  // failure-detection test: the producer issues nothing
    // Backward use: the reverse scan's workspace (F + 1 slots per chain), written by the
    // kK1RevA and kK1E instantiations.  beta == null means beta = 1 for every token.
    uint8_t *ws_rev;
};

// K1 instantiations: the forward's; one that also writes each A_f image into slot F - f
// of the reverse scan's workspace; and the E mode, which forms only U_f (the backward's
// E_f = dO^T q^: no A_f MMA, no A_f image, no composites) and writes it to the U area of
// slot F - 1 - f, nothing to the forward workspace.
constexpr int kK1Fwd = 0, kK1RevA = 1, kK1E = 2;

// Tensor memory of K1 (512 columns, fp32 unless noted):
//   [  0,128) acc_A: A_f = X^T K; after read-out it holds the composite MMAs'
//             A operands: -bf16(C) in columns [0,56), -bf16(H) in [56,112)
//             (bf16 pairs per column, one matrix row per lane)
//   [128,256) acc_U: U_f = Y_hi^T K + Y_lo^T K
//   [256,384) T_C: chunk transition composite C = prod M_f
//   [384,512) T_H: chunk input composite H (state reached from zero)
constexpr uint32_t kTmAccA = 0, kTmAccU = 128, kTmC = 256, kTmH = 384, kTmImgC = 0, kTmImgH = 56;

// The kernel body, shared by the standalone launch and the fused chained scan.
// With kKeepTmem the CTA's 512 TMEM columns stay allocated on return (the chunk
// composites C and H still in them) and their address is returned; *aborted
// receives the role abort flag.
template <bool kKeepTmem, int kMode = kK1Fwd>
__device__ __forceinline__ uint32_t k1_body(const CUtensorMap &mapK, const CUtensorMap &mapV, const K1Params &p,
                                            uint8_t *sm, int *aborted)
{
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + kK1OffBar);
    uint64_t *st_full = bars + 0, *st_prep = bars + kK1Stages, *st_empty = bars + 2 * kK1Stages;
    uint64_t *acc_full = bars + 3 * kK1Stages, *comp_ready = acc_full + 1, *comp_done = acc_full + 2;
    uint64_t *drain = acc_full + 3;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(acc_full + 5);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(acc_full + 6);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int BH = p.B * p.H;
    const int chunk_idx = blockIdx.x / BH, bh = blockIdx.x % BH;
    const int b = bh / p.H, h = bh % p.H;
    int f_begin, nf;
    chunk_frames(chunk_idx, p.F, p.n_chunks, f_begin, nf);
    const int n_st = (p.N + kTS - 1) / kTS;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kK1Stages; ++i) {
            mbar_init(&st_full[i], 1);
            mbar_init(&st_prep[i], 4);
            mbar_init(&st_empty[i], 1);
        }
        mbar_init(acc_full, 1);
        mbar_init(comp_ready, 4);
        mbar_init(comp_done, 1);
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
    // Programmatic dependent launch: the next kernel may be scheduled now; no
    // global memory is touched before the previous kernel has completed.
    griddep_launch_dependents();
    griddep_wait();
    const uint32_t sbase = smem_u32(sm);

    if (warp == 0) {
        // ------------------------------------------------------ TMA producer
        if (lane == 0) {
            const uint64_t pol = policy_stream();
            int it = 0;
            bool ok = !p.withhold_loads;  // withheld: no stage ever fills, the consumers' waits expire
            for (int fl = 0; fl < nf && ok; ++fl) {
                const int bf = b * p.F + frame_at(f_begin + fl, p.F, p.reverse);
                for (int st = 0; st < n_st; ++st, ++it) {
                    const int s = it % kK1Stages, use = it / kK1Stages;
                    if (use >= 1 && !(ok = mbar_wait(&st_empty[s], (use - 1) & 1, abort_flag))) break;
                    uint8_t *stg = sm + s * kStageBytes;
                    mbar_arrive_expect_tx(&st_full[s], 4 * kTSPanel);
                    tma_load_4d(stg + kOffK, &mapK, &st_full[s], 0, h, st * kTS, bf, pol);
                    tma_load_4d(stg + kOffK + kTSPanel, &mapK, &st_full[s], 64, h, st * kTS, bf, pol);
                    tma_load_4d(stg + kOffV, &mapV, &st_full[s], 0, h, st * kTS, bf, pol);
                    tma_load_4d(stg + kOffV + kTSPanel, &mapV, &st_full[s], 64, h, st * kTS, bf, pol);
                }
            }
            if (*abort_flag)  // let loads already in flight land before the CTA exits
                for (int s = 0; s < kK1Stages && s < it; ++s)
                    mbar_wait_drain(&st_full[s], ((it - 1 - s) / kK1Stages) & 1);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------- MMA issuer
        if (lane == 0) {
            int it = 0;
            bool ok = true;
            for (int fl = 0; fl < nf && ok; ++fl) {
                // The previous frame's composite MMAs read their A operands from the
                // acc_A columns that this frame's first MMA overwrites: tcgen05.mma
                // operations issued by one thread execute in issue order, so no wait.
                for (int st = 0; st < n_st && ok; ++st, ++it) {
                    const int s = it % kK1Stages, use = it / kK1Stages;
                    if (!(ok = mbar_wait(&st_prep[s], use & 1, abort_flag))) break;
                    tc_fence_after();
                    const uint32_t stg = sbase + s * kStageBytes;
#pragma unroll
                    for (int ks = 0; ks < kTS / 16; ++ks) {
                        const uint32_t o = ks * 2048;
                        const uint64_t bhi = sdesc_sw128(stg + kOffBhi + o, kTSPanel, 1024);
                        const uint64_t blo = sdesc_sw128(stg + kOffBlo + o, kTSPanel, 1024);
                        const uint64_t av = sdesc_sw128(stg + kOffV + o, kTSPanel, 1024);
                        const uint32_t acc = (st > 0 || ks > 0) ? 1u : 0u;
                        if (!(kMode == kK1E))
                            mma_bf16(tmem + kTmAccA, sdesc_sw128(stg + kOffK + o, kTSPanel, 1024), bhi, kIdescMN,
                                     acc);
                        mma_bf16(tmem + kTmAccU, av, bhi, kIdescMN, acc);
                        if (kK1Lo) mma_bf16(tmem + kTmAccU, av, blo, kIdescMN, 1u);
                    }
                    mma_commit(&st_empty[s]);
                }
                if (!ok) break;
                mma_commit(acc_full);
                // composite: T_C += (-C) A_f, T_H += (-H) A_f (T_C, T_H pre-scaled by gamma, T_H += U_f);
                // comp_ready also says the epilogue has read this frame's accumulators
                if (!(ok = mbar_wait(comp_ready, fl & 1, abort_flag))) break;
                tc_fence_after();
                if (kMode != kK1E) {
#pragma unroll
                    for (int ks = 0; ks < 7; ++ks) {
                        const uint64_t bdesc =
                            sdesc_sw128(sbase + kK1OffAimg + (ks >> 2) * kAimgPanel + (ks & 3) * 32, 16, 1024);
                        mma_bf16_tmem_a(tmem + kTmC, tmem + kTmImgC + ks * 8, bdesc, kIdescK, 1u);
                        mma_bf16_tmem_a(tmem + kTmH, tmem + kTmImgH + ks * 8, bdesc, kIdescK, 1u);
                    }
                    mma_commit(comp_done);
                }
            }
            mma_commit(drain);  // every MMA issued above has completed once this phase lands
            mbar_wait_drain(drain, 0);
        }
    } else if (warp < 10) {
        // ------------------------------------------------------ prep warps
        // Two groups of four warps take alternate stages, so two stages are
        // prepared at once.  Thread (token r, quarter qq) handles panel qq>>1,
        // chunks 4*(qq&1).. of its token; the eight threads of a quarter-warp
        // phase touch eight different bank groups.
        constexpr int kTH = kTS / 32;              // 32-token rows of a stage per thread
        const int grpi = (warp - 2) >> 2;          // 0: even stages, 1: odd stages
        const int t = threadIdx.x - 64 - 128 * grpi;  // 0..127
        const int r0 = t >> 2, qq = t & 3;
        const size_t FN = (size_t)p.F * p.N;
        const int total = nf * n_st;
        auto load_beta = [&](int itx, int r) -> float {
            if (itx >= total) return 0.f;
            if (!p.beta) return 1.f;
            const int fl = itx / n_st, n = (itx - fl * n_st) * kTS + r;
            if (n >= p.N) return 0.f;
            return __ldg(p.beta + ((size_t)b * FN + (size_t)frame_at(f_begin + fl, p.F, p.reverse) * p.N + n) * p.H + h);
        };
        float bt_next[kTH];
#pragma unroll
        for (int hh = 0; hh < kTH; ++hh) bt_next[hh] = load_beta(grpi, r0 + 32 * hh);
        for (int it = grpi; it < total; it += 2) {
            const int s = it % kK1Stages, use = it / kK1Stages;
            float bts[kTH];
#pragma unroll
            for (int hh = 0; hh < kTH; ++hh) {
                bts[hh] = bt_next[hh];
                bt_next[hh] = load_beta(it + 2, r0 + 32 * hh);
            }
            if (!mbar_wait_warp(&st_full[s], use & 1, abort_flag)) break;
#pragma unroll
            for (int hh = 0; hh < kTH; ++hh) {
            const int r = r0 + 32 * hh;
            const float bt = bts[hh];
            uint8_t *stg = sm + s * kStageBytes + (qq >> 1) * kTSPanel + r * kRowB;
            float kf[32];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint32_t pos = (((i + qq + r) & 3) + 4 * (qq & 1)) << 4;
                bf16x8_to_f32(*reinterpret_cast<const uint4 *>(stg + kOffK + pos), kf + 8 * i);
            }
            float ss = 0.f;
#pragma unroll
            for (int i = 0; i < 32; ++i) ss = fmaf(kf[i], kf[i], ss);
            ss += __shfl_xor_sync(0xffffffffu, ss, 1);
            ss += __shfl_xor_sync(0xffffffffu, ss, 2);
            const float inv = p.c * rsqrtf(ss + kEps);   // c / ||k||
            const float wb = bt * inv;                   // beta c / ||k||
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint32_t pos = (((i + qq + r) & 3) + 4 * (qq & 1)) << 4;
                float kh[8], y[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    kh[e] = inv * kf[8 * i + e];
                    y[e] = wb * kf[8 * i + e];
                }
                *reinterpret_cast<uint4 *>(stg + kOffK + pos) = f32x8_to_bf16(kh);
                if (kK1Lo) {
                    uint4 hi, lo;
                    split_bf16x8(y, hi, lo);
                    *reinterpret_cast<uint4 *>(stg + kOffBhi + pos) = hi;
                    *reinterpret_cast<uint4 *>(stg + kOffBlo + pos) = lo;
                } else {
                    *reinterpret_cast<uint4 *>(stg + kOffBhi + pos) = f32x8_to_bf16(y);
                }
            }
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&st_prep[s]);
        }
    } else {
        // ------------------------------------------------- epilogue warps
        // One warp per TMEM lane quadrant; thread = matrix row, all 112 columns.
        // Per frame: A_f and U_f out of TMEM into the workspace, the composites
        // scaled by gamma (+U_f into H), and -bf16(C), -bf16(H) staged as the
        // composite MMAs' A operands.
        const int quad = warp & 3;
        const int row = quad * 32 + lane;
        const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
        bool ok = true;
        // composites start at C = I, H = 0 (rows 112..127 stay zero)
#pragma unroll
        for (int c8 = 0; c8 < kD / 8; ++c8) {
            uint32_t wc[8], wz[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                wc[j] = (row == c8 * 8 + j) ? __float_as_uint(1.f) : 0u;
                wz[j] = 0u;
            }
            tmem_st8(tmem + lane_off + kTmC + c8 * 8, wc);
            tmem_st8(tmem + lane_off + kTmH + c8 * 8, wz);
        }
        tmem_st_wait();
        const uint64_t ws_pol = kWsKeepL2 ? policy_evict_last() : 0;  // workspace lines K2 reads next
        // this warp's rows of the A_f image: rows 32*quad.. of each panel
        const int img_rows = quad == 3 ? kD - 96 : 32;
        const uint32_t img_off = quad * 32 * kRowB;
        const float *gam = p.gamma + (size_t)b * p.F * p.H + h;
        float g_next = __ldg(gam + (size_t)frame_at(f_begin, p.F, p.reverse) * p.H);
        for (int fe = 0; fe < nf && ok; ++fe) {
            const int f = f_begin + fe;
            const float g = g_next;
            if (fe + 1 < nf) g_next = __ldg(gam + (size_t)frame_at(f + 1, p.F, p.reverse) * p.H);
            // this warp's previous A_f bulk stores must have finished reading
            if (lane == 0) bulk_wait_read_all();
            __syncwarp();
            if (!(ok = mbar_wait_warp(acc_full, fe & 1, abort_flag))) break;
            tc_fence_after();
            uint8_t *ws = (kMode == kK1E) ? nullptr : p.ws_frames + ((size_t)bh * p.F + f) * kFrameWs;
            float *wsU = reinterpret_cast<float *>(
                (kMode == kK1E) ? p.ws_rev + ((size_t)bh * (p.F + 1) + (p.F - 1 - f)) * kFrameWs + kAimgBytes
                         : ws + kAimgBytes);
            // pass 1: A_f -> bf16 image (shared memory), U_f -> workspace.  TMEM loads
            // go out two 16-column chunks at a time: each wait costs a full load
            // latency, which the frame boundary otherwise pays seven times.
#pragma unroll
            for (int cp = 0; cp < 7; cp += 2) {
            uint32_t ra2[2][16], ru2[2][16];
#pragma unroll
            for (int hf = 0; hf < 2 && cp + hf < 7; ++hf) {
                if (!(kMode == kK1E)) tmem_ld16(tmem + lane_off + kTmAccA + (cp + hf) * 16, ra2[hf]);
                tmem_ld16(tmem + lane_off + kTmAccU + (cp + hf) * 16, ru2[hf]);
            }
            tmem_ld_wait();
#pragma unroll
            for (int hf = 0; hf < 2 && cp + hf < 7; ++hf) {
                const int cc = cp + hf;
                const uint32_t col = cc * 16;
                const uint32_t *ra = ra2[hf], *ru = ru2[hf];
                if (row < kD) {
                    if (!(kMode == kK1E)) {
                        float a[16];
#pragma unroll
                        for (int j = 0; j < 16; ++j) a[j] = __uint_as_float(ra[j]);
                        uint8_t *dst = sm + kK1OffAimg + (cc >> 2) * kAimgPanel;
                        *reinterpret_cast<uint4 *>(dst + sw128_off(row, 2 * (cc & 3))) = f32x8_to_bf16(a);
                        *reinterpret_cast<uint4 *>(dst + sw128_off(row, 2 * (cc & 3) + 1)) = f32x8_to_bf16(a + 8);
                    }
                    float4 *u4 = reinterpret_cast<float4 *>(wsU) + (col / 4) * kD + row;
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const float4 v4 = make_float4(__uint_as_float(ru[4 * j]), __uint_as_float(ru[4 * j + 1]),
                                                      __uint_as_float(ru[4 * j + 2]), __uint_as_float(ru[4 * j + 3]));
                        if (kWsKeepL2) st_global_hint(u4 + j * kD, v4, ws_pol);
                        else u4[j * kD] = v4;
                    }
                }
            }
            }
            if (row < kD && !(kMode == kK1E)) {  // key columns 112..127 of the image: zero
                uint8_t *dst = sm + kK1OffAimg + kAimgPanel;
                *reinterpret_cast<uint4 *>(dst + sw128_off(row, 6)) = make_uint4(0, 0, 0, 0);
                *reinterpret_cast<uint4 *>(dst + sw128_off(row, 7)) = make_uint4(0, 0, 0, 0);
            }
            // pass 2 overwrites acc_A's columns with the composite images: each warp
            // touches only its own TMEM lanes, and has read all of them above
            // pass 2: H <- gamma H + U_f, C <- gamma C; A operands -bf16(H_prev), -bf16(C_prev)
#pragma unroll
            for (int cp = 0; cp < 7 && !(kMode == kK1E); cp += 2) {
            uint32_t ru2[2][16], rh2[2][16], rc2[2][16];
#pragma unroll
            for (int hf = 0; hf < 2 && cp + hf < 7; ++hf) {
                tmem_ld16(tmem + lane_off + kTmAccU + (cp + hf) * 16, ru2[hf]);
                tmem_ld16(tmem + lane_off + kTmH + (cp + hf) * 16, rh2[hf]);
                tmem_ld16(tmem + lane_off + kTmC + (cp + hf) * 16, rc2[hf]);
            }
            tmem_ld_wait();
#pragma unroll
            for (int hf = 0; hf < 2 && cp + hf < 7; ++hf) {
                const uint32_t col = (cp + hf) * 16;
                const uint32_t *ru = ru2[hf], *rh = rh2[hf], *rc = rc2[hf];
                uint32_t hn0[8], hn1[8], cn0[8], cn1[8], ih[8], ic[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    hn0[j] = __float_as_uint(fmaf(g, __uint_as_float(rh[j]), __uint_as_float(ru[j])));
                    hn1[j] = __float_as_uint(fmaf(g, __uint_as_float(rh[8 + j]), __uint_as_float(ru[8 + j])));
                    cn0[j] = __float_as_uint(g * __uint_as_float(rc[j]));
                    cn1[j] = __float_as_uint(g * __uint_as_float(rc[8 + j]));
                    ih[j] = pack_bf16x2(-__uint_as_float(rh[2 * j]), -__uint_as_float(rh[2 * j + 1]));
                    ic[j] = pack_bf16x2(-__uint_as_float(rc[2 * j]), -__uint_as_float(rc[2 * j + 1]));
                }
                tmem_st8(tmem + lane_off + kTmH + col, hn0);
                tmem_st8(tmem + lane_off + kTmH + col + 8, hn1);
                tmem_st8(tmem + lane_off + kTmC + col, cn0);
                tmem_st8(tmem + lane_off + kTmC + col + 8, cn1);
                tmem_st8(tmem + lane_off + kTmImgH + col / 2, ih);
                tmem_st8(tmem + lane_off + kTmImgC + col / 2, ic);
            }
            }
            tmem_st_wait();
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(comp_ready);
                if (!(kMode == kK1E)) {
                    if (kWsKeepL2) {
                        bulk_s2g_hint(ws + img_off, sm + kK1OffAimg + img_off, img_rows * kRowB, ws_pol);
                        bulk_s2g_hint(ws + kAimgPanel + img_off, sm + kK1OffAimg + kAimgPanel + img_off,
                                      img_rows * kRowB, ws_pol);
                    } else {
                        bulk_s2g(ws + img_off, sm + kK1OffAimg + img_off, img_rows * kRowB);
                        bulk_s2g(ws + kAimgPanel + img_off, sm + kK1OffAimg + kAimgPanel + img_off,
                                 img_rows * kRowB);
                    }
                    if (kMode == kK1RevA) {  // the reverse scan's slot F - f holds A_f as well
                        uint8_t *wr = p.ws_rev + ((size_t)bh * (p.F + 1) + (p.F - f)) * kFrameWs;
                        bulk_s2g(wr + img_off, sm + kK1OffAimg + img_off, img_rows * kRowB);
                        bulk_s2g(wr + kAimgPanel + img_off, sm + kK1OffAimg + kAimgPanel + img_off,
                                 img_rows * kRowB);
                    }
                    bulk_commit();
                }
            }
        }
        // chunk composites out: wait for the last frame's composite MMAs
        if (ok && !(kMode == kK1E) && (ok = mbar_wait_warp(comp_done, (nf - 1) & 1, abort_flag))) {
            tc_fence_after();
            float *comp = p.ws_comp + ((size_t)bh * p.n_chunks + chunk_idx) * 2 * kStateFloats;
#pragma unroll
            for (int cc = 0; cc < 7; ++cc) {
                const uint32_t col = cc * 16;
                uint32_t rc[16], rh[16];
                tmem_ld16(tmem + lane_off + kTmC + col, rc);
                tmem_ld16(tmem + lane_off + kTmH + col, rh);
                tmem_ld_wait();
                if (row < kD) {
#pragma unroll
                    for (int j = 0; j < 16; j += 4) {
                        *reinterpret_cast<float4 *>(comp + row * kD + col + j) =
                            make_float4(__uint_as_float(rc[j]), __uint_as_float(rc[j + 1]),
                                        __uint_as_float(rc[j + 2]), __uint_as_float(rc[j + 3]));
                        *reinterpret_cast<float4 *>(comp + kStateFloats + row * kD + col + j) =
                            make_float4(__uint_as_float(rh[j]), __uint_as_float(rh[j + 1]),
                                        __uint_as_float(rh[j + 2]), __uint_as_float(rh[j + 3]));
                    }
                }
            }
        }
        if (lane == 0) bulk_wait_all();
    }
    tc_fence_before();
    __syncthreads();
    *aborted = *abort_flag;
    if (*abort_flag && threadIdx.x == 0) raise_status(p.status);
    if (!kKeepTmem && warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
    return tmem;
}

template <int kMode>
__global__ void __launch_bounds__(kK1Threads, 1)
    k1_frame_stats_kernel(const __grid_constant__ CUtensorMap mapK, const __grid_constant__ CUtensorMap mapV,
                          const K1Params p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    int aborted;
    k1_body<false, kMode>(mapK, mapV, p, sm, &aborted);
}

// ===================================================================== K1b
// S_start(c) for every chunk, row-parallel fp32: rows [16*y, 16*y+16) of chain
// x, seven CTAs per chain (one wave for the 20-head layer).  The chain is
// sequential over chunks, S_start(c+1) = S_start(c) C_c + H_c; the composites
// C_c (50 KB each) are bulk-copied into a ring of three shared-memory buffers,
// up to three steps ahead, so that a step does not wait for its copy.
// The product of a step: four thread groups split the 112-long contraction
// into quarters, and each thread keeps a kTR x kTC block of its quarter's
// partial sums in registers: rows rg, rg + 16/kTR, .. of the CTA's 16 and
// columns kTC*cg.. (rg = i % (16/kTR), cg = i / (16/kTR) for thread i of its
// group).  Per four k steps a thread loads kTR float4 of S and 4*kTC/4 float4
// of C.  A 128-bit shared load is served a quarter-warp at a time whatever its
// addresses, so loads per FMA set the rate (one column and four rows per
// thread: 2.8 us a step; 4 x 4 blocks over the full contraction on 112
// threads: 2.45 us; split four ways: 1.55 us).  Every group leaves its partial
// block in shared memory and all threads add the four up.  The S rows are 116
// floats apart, so the rows a quarter-warp reads at one k fall in different
// bank groups.  With a zero start state (no S_in) the first step is
// S_start(1) = H_0.
#ifndef GDN_K1B_TR
#define GDN_K1B_TR 4
#endif
#ifndef GDN_K1B_TC
#define GDN_K1B_TC 4
#endif
constexpr int kK1bRows = 16;
constexpr int kK1bTR = GDN_K1B_TR;                                   // rows per thread block (4 or 8)
constexpr int kK1bTC = GDN_K1B_TC;                                   // columns per thread block (4 or 8)
constexpr int kK1bRG = kK1bRows / kK1bTR;                           // row sets of a group
constexpr int kK1bGroups = 4;                                       // contraction quarters
constexpr int kK1bTiles = kK1bRG * (kD / kK1bTC);                   // threads per group
constexpr int kK1bThreads = kK1bTiles * kK1bGroups;
constexpr int kK1bLen = kD / kK1bGroups;                            // contraction length per group
constexpr int kK1bPitch = kD + 4;                                   // S and partial row pitch (floats)
constexpr int kK1bBufs = 3;
constexpr uint32_t kK1bRowsBytes = kK1bRows * kK1bPitch * 4;
constexpr uint32_t kK1bOffS = kK1bBufs * (uint32_t)kStateBytes;     // S rows [16][116]
constexpr uint32_t kK1bOffP = kK1bOffS + kK1bRowsBytes;             // partial rows of the four groups
constexpr uint32_t kK1bOffBar = kK1bOffP + kK1bGroups * kK1bRowsBytes;  // mbarriers + abort flag
constexpr uint32_t kK1bSmem = kK1bOffBar + 64;
static_assert((kK1bTR == 4 || kK1bTR == 8) && (kK1bTC == 4 || kK1bTC == 8) && kD % kK1bTC == 0, "K1b blocks");
static_assert(kK1bLen % 4 == 0 && kK1bLen * kK1bGroups == kD && kK1bThreads <= 1024, "K1b contraction split");
static_assert(kK1bPitch % 4 == 0 && (kK1bPitch % 32) % 8 == 4, "K1b row pitch: 16-byte rows, bank groups");
static_assert(kK1bOffS % 16 == 0 && kK1bSmem <= kMaxSmem, "K1b shared memory");
// K1b modes: the start state is the identity (instead of S_in), and/or the input
// composites are zero.  With both the scan composes the transition composites,
// C_0 C_1 ... C_{n-1}; with neither it is the chunk-boundary scan proper.
constexpr int kK1bIdentityIn = 1, kK1bZeroH = 2;

__global__ void __launch_bounds__(kK1bThreads, 1)
    k1b_chunk_boundary_kernel(const float *__restrict__ compC, const float *__restrict__ compH, size_t chain_stride,
                              size_t chunk_stride, float *__restrict__ ws_start, const float *S_in, float *S_out,
                              int n_chunks, unsigned *status, int mode)
{
    constexpr int kC4 = kK1bTC / 4;  // float4 per block row
    extern __shared__ __align__(128) uint8_t k1b_smem[];
    float(*Srows)[kK1bPitch] = reinterpret_cast<float(*)[kK1bPitch]>(k1b_smem + kK1bOffS);
    float(*Part)[kK1bRows][kK1bPitch] = reinterpret_cast<float(*)[kK1bRows][kK1bPitch]>(k1b_smem + kK1bOffP);
    uint64_t *bar = reinterpret_cast<uint64_t *>(k1b_smem + kK1bOffBar);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(bar + kK1bBufs);
    auto cbuf = [&](int i) { return reinterpret_cast<float *>(k1b_smem + (size_t)i * kStateBytes); };
    const int bh = blockIdx.x, r0 = blockIdx.y * kK1bRows;
    const int t = threadIdx.x, grp = t / kK1bTiles, ti = t % kK1bTiles;
    const int rg = ti % kK1bRG, cg = ti / kK1bRG;  // rows rg + kK1bRG*q (q < kTR), columns kTC*cg..
    const int l0 = grp * kK1bLen;                   // this group's contraction quarter
    const float *cC = compC + (size_t)bh * chain_stride, *cH = compH + (size_t)bh * chain_stride;
    const bool zero_start = !(mode & kK1bIdentityIn) && S_in == nullptr;
    if (t == 0) {
        for (int i = 0; i < kK1bBufs; ++i) mbar_init(&bar[i], 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    griddep_launch_dependents();
    griddep_wait();  // composites and S_in come from earlier kernels on the stream
    // composite steps to apply: without S_out the state after the last chunk is not needed
    const int steps = S_out ? n_chunks : n_chunks - 1;
    // group 0's block of H_c (the other groups start their partial sums from zero), loaded one
    // step ahead; the first load goes out before the start rows are filled
    const bool load_h = grp == 0 && (mode & kK1bZeroH) == 0;
    const float *h_ptr = cH + (r0 + rg) * kD + kK1bTC * cg;
    float4 h_next[kK1bTR][kC4];
#pragma unroll
    for (int q = 0; q < kK1bTR; ++q)
#pragma unroll
        for (int u = 0; u < kC4; ++u)
            h_next[q][u] = (load_h && steps > 0)
                               ? *reinterpret_cast<const float4 *>(h_ptr + kK1bRG * q * kD + 4 * u)
                               : make_float4(0.f, 0.f, 0.f, 0.f);
    int issued = 0;
    if (t == 0)
        for (; issued < steps && issued < kK1bBufs; ++issued) {
            mbar_arrive_expect_tx(&bar[issued], (uint32_t)kStateBytes);
            bulk_g2s(cbuf(issued), cC + (size_t)issued * chunk_stride, (uint32_t)kStateBytes, &bar[issued]);
        }
    for (int e = t; e < kK1bRows * kD; e += kK1bThreads) {
        const int rr = e / kD, cc = e % kD;
        Srows[rr][cc] = (mode & kK1bIdentityIn) ? (r0 + rr == cc ? 1.f : 0.f)
                        : S_in ? S_in[(size_t)bh * kStateFloats + (r0 + rr) * kD + cc] : 0.f;
    }
    __syncthreads();
    int c = 0;  // on abort: the step whose copy was not seen to land
    for (; c < n_chunks; ++c) {
        if (ws_start) {
            float *dst = ws_start + ((size_t)bh * n_chunks + c) * kStateFloats + (size_t)r0 * kD;
            for (int e = t; e < kK1bRows * kD / 4; e += kK1bThreads) {
                const int rr = e / (kD / 4), c4 = e % (kD / 4);
                *reinterpret_cast<float4 *>(dst + rr * kD + 4 * c4) =
                    *reinterpret_cast<const float4 *>(&Srows[rr][4 * c4]);
            }
        }
        if (c >= steps) break;
        float4 acc[kK1bTR][kC4];
#pragma unroll
        for (int q = 0; q < kK1bTR; ++q)
#pragma unroll
            for (int u = 0; u < kC4; ++u) acc[q][u] = h_next[q][u];
        h_ptr += chunk_stride;
#pragma unroll
        for (int q = 0; q < kK1bTR; ++q)
#pragma unroll
            for (int u = 0; u < kC4; ++u)
                h_next[q][u] = (load_h && c + 1 < steps)
                                   ? *reinterpret_cast<const float4 *>(h_ptr + kK1bRG * q * kD + 4 * u)
                                   : make_float4(0.f, 0.f, 0.f, 0.f);
        const int buf = c % kK1bBufs;
        if (t == 0 && !mbar_wait(&bar[buf], (c / kK1bBufs) & 1, abort_flag)) *abort_flag = 1;
        __syncthreads();
        if (*abort_flag) break;
        if (!(c == 0 && zero_start)) {  // S_start(0) = 0: S_start(1) = H_0
            const float *C = cbuf(buf) + kK1bTC * cg;
#pragma unroll
            for (int l = l0; l < l0 + kK1bLen; l += 4) {
                float4 cv[4][kC4], sv[kK1bTR];
#pragma unroll
                for (int k = 0; k < 4; ++k)
#pragma unroll
                    for (int u = 0; u < kC4; ++u) cv[k][u] = *reinterpret_cast<const float4 *>(C + (l + k) * kD + 4 * u);
#pragma unroll
                for (int q = 0; q < kK1bTR; ++q) sv[q] = *reinterpret_cast<const float4 *>(&Srows[rg + kK1bRG * q][l]);
#pragma unroll
                for (int q = 0; q < kK1bTR; ++q) {
                    const float sk[4] = {sv[q].x, sv[q].y, sv[q].z, sv[q].w};
#pragma unroll
                    for (int k = 0; k < 4; ++k)
#pragma unroll
                        for (int u = 0; u < kC4; ++u) {
                            acc[q][u].x = fmaf(sk[k], cv[k][u].x, acc[q][u].x);
                            acc[q][u].y = fmaf(sk[k], cv[k][u].y, acc[q][u].y);
                            acc[q][u].z = fmaf(sk[k], cv[k][u].z, acc[q][u].z);
                            acc[q][u].w = fmaf(sk[k], cv[k][u].w, acc[q][u].w);
                        }
                }
            }
        }
#pragma unroll
        for (int q = 0; q < kK1bTR; ++q)
#pragma unroll
            for (int u = 0; u < kC4; ++u)
                *reinterpret_cast<float4 *>(&Part[grp][rg + kK1bRG * q][kK1bTC * cg + 4 * u]) = acc[q][u];
        __syncthreads();  // every thread is done with this buffer and with the old rows
        if (t == 0 && c + kK1bBufs < steps) {
            mbar_arrive_expect_tx(&bar[buf], (uint32_t)kStateBytes);
            bulk_g2s(cbuf(buf), cC + (size_t)(c + kK1bBufs) * chunk_stride, (uint32_t)kStateBytes, &bar[buf]);
            ++issued;
        }
        for (int e = t; e < kK1bRows * kD / 4; e += kK1bThreads) {  // the new rows: sum of the four partials
            const int rr = e / (kD / 4), c4 = e % (kD / 4);
            float4 a = *reinterpret_cast<const float4 *>(&Part[0][rr][4 * c4]);
#pragma unroll
            for (int g = 1; g < kK1bGroups; ++g) {
                const float4 pp = *reinterpret_cast<const float4 *>(&Part[g][rr][4 * c4]);
                a.x += pp.x, a.y += pp.y, a.z += pp.z, a.w += pp.w;
            }
            *reinterpret_cast<float4 *>(&Srows[rr][4 * c4]) = a;
        }
        __syncthreads();
    }
    if (*abort_flag) {
        if (t == 0) {
            // copies 0..c-1 were waited for; each later one is its buffer's pending phase
            for (int i = c; i < issued; ++i) mbar_wait_drain(&bar[i % kK1bBufs], (i / kK1bBufs) & 1);
            if (status) atomicOr(status, kStatusTimeout);
        }
        return;
    }
    if (S_out)
        for (int e = t; e < kK1bRows * kD; e += kK1bThreads)
            S_out[(size_t)bh * kStateFloats + (r0 + e / kD) * kD + e % kD] = Srows[e / kD][e % kD];
}

// ===================================================================== K2
struct K2Params {
    void *o;  // bf16 output (row stores when the kernel is built without output staging)
    const float *gamma;
    const uint8_t *ws_frames;
    const float *ws_start;
    float *S_out;   // non-null: the last chunk's CTAs write the chain's final state here
    float *states;  // non-null: the state after every frame, [B*H][F][D][D] by processing position
    unsigned *status;
    int B, H, F, N, chunk, n_chunks;
    int reverse;      // 1: frames are visited from the last to the first
    int states_only;  // 1: no outputs (the state chain alone)
};

// K2's state role over columns [kC0, kC0 + kCols) of every row: thread = row
// of S (fp32 registers), one warp per TMEM lane quadrant.  The standalone
// kernel runs it on four warps with all 112 columns; the fused chained scan,
// whose 448 threads allow 128 registers each, on eight warps with 56 columns.
// As soon as S_f's images are written, S <- gamma_f S + U_f (U_f read from
// global memory, quad-major: a warp's lanes read 512 contiguous bytes, four
// 8-column chunks ahead of their use), overlapping the S A_f GEMM; when
// that lands, S <- S - S_f A_f.
template <int kCols, int kC0>
__device__ __forceinline__ void k2_state_role(const K2Params &p, uint8_t *sm, uint32_t tmem, uint64_t *s_ready,
                                              uint64_t *accS_full, uint64_t *o_done, volatile int *abort_flag,
                                              int bh, int b, int h, int chunk_idx, int f_begin, int nf,
                                              const uint8_t *ws_chain)
{
    static_assert(kCols % 8 == 0 && kC0 % 8 == 0 && kC0 + kCols <= kD, "state column range");
    constexpr int kCh = kCols / 8;                 // 8-column chunks
    constexpr int kCs = kC0 & ~15, kSkip = kC0 - kCs;
    constexpr int kNld = (kSkip + kCols + 15) / 16;  // 16-column TMEM loads covering the range
    const int lane = threadIdx.x & 31, quad = (threadIdx.x >> 5) & 3, row = quad * 32 + lane;
    const int urow = row < kD ? row : 0;
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    float S[kCols];
    const float *s0 = p.ws_start + ((size_t)bh * p.n_chunks + chunk_idx) * kStateFloats;
#pragma unroll
    for (int j = 0; j < kCols; j += 4) {
        float4 v4 = make_float4(0.f, 0.f, 0.f, 0.f);
        if (row < kD) v4 = __ldcg(reinterpret_cast<const float4 *>(s0 + row * kD + kC0 + j));  // L2: may come from
                                                                                                // another CTA
        S[j] = v4.x;
        S[j + 1] = v4.y;
        S[j + 2] = v4.z;
        S[j + 3] = v4.w;
    }
    auto write_images = [&](int set) {
        if (row < kD) {
            const uint32_t sset = (uint32_t)set * kK2SetBytes;
#pragma unroll
            for (int c8 = 0; c8 < kCh; ++c8) {
                const int g8 = kC0 / 8 + c8;
                const uint32_t off = sset + (g8 >> 3) * kImgPanel + sw128_off(row, g8 & 7);
                if (kK2Lo) {
                    uint4 hi, lo;
                    split_bf16x8(S + 8 * c8, hi, lo);
                    *reinterpret_cast<uint4 *>(sm + kK2OffShi + off) = hi;
                    *reinterpret_cast<uint4 *>(sm + kK2OffSlo + off) = lo;
                } else {
                    *reinterpret_cast<uint4 *>(sm + kK2OffShi + off) = f32x8_to_bf16(S + 8 * c8);
                }
            }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(s_ready);
    };
    write_images(0);
    const float *gam = p.gamma + (size_t)b * p.F * p.H + h;
    float g_next = __ldg(gam + (size_t)frame_at(f_begin, p.F, p.reverse) * p.H);
    for (int it = 0; it < nf; ++it) {
        const float g = g_next;
        if (it + 1 < nf) g_next = __ldg(gam + (size_t)frame_at(f_begin + it + 1, p.F, p.reverse) * p.H);
        const float4 *U4 = reinterpret_cast<const float4 *>(ws_chain + (size_t)it * kFrameWs + kAimgBytes) + urow;
        constexpr int kW = 4;  // 8-column chunks of U_f loaded ahead of their use
        float4 ub[kW][2];
#pragma unroll
        for (int c = 0; c < kW && c < kCh; ++c)
#pragma unroll
            for (int j = 0; j < 2; ++j) ub[c][j] = __ldg(U4 + (kC0 / 4 + 2 * c + j) * kD);
#pragma unroll
        for (int c = 0; c < kCh; ++c) {
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const float4 u4 = ub[c % kW][j];
                const int k0 = c * 8 + 4 * j;
                S[k0] = fmaf(g, S[k0], u4.x);
                S[k0 + 1] = fmaf(g, S[k0 + 1], u4.y);
                S[k0 + 2] = fmaf(g, S[k0 + 2], u4.z);
                S[k0 + 3] = fmaf(g, S[k0 + 3], u4.w);
            }
            if (c + kW < kCh)
#pragma unroll
                for (int j = 0; j < 2; ++j) ub[c % kW][j] = __ldg(U4 + (kC0 / 4 + 2 * (c + kW) + j) * kD);
        }
        if (!mbar_wait_warp(accS_full, it & 1, abort_flag)) break;
        tc_fence_after();
#pragma unroll
        for (int cp = 0; cp < kNld; cp += 2) {  // two 16-column chunks per TMEM round trip
            uint32_t ra2[2][16];
#pragma unroll
            for (int hf = 0; hf < 2 && cp + hf < kNld; ++hf)
                tmem_ld16(tmem + lane_off + kCs + (cp + hf) * 16, ra2[hf]);
            tmem_ld_wait();
#pragma unroll
            for (int hf = 0; hf < 2 && cp + hf < kNld; ++hf)
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const int k = (cp + hf) * 16 + j - kSkip;
                    if (k >= 0 && k < kCols) S[k] -= __uint_as_float(ra2[hf][j]);
                }
        }
        tc_fence_before();
        if (p.states && row < kD) {
            float4 *dst = reinterpret_cast<float4 *>(p.states + ((size_t)bh * p.F + f_begin + it) * kStateFloats +
                                                     row * kD + kC0);
#pragma unroll
            for (int j = 0; j < kCols / 4; ++j) dst[j] = make_float4(S[4 * j], S[4 * j + 1], S[4 * j + 2], S[4 * j + 3]);
        }
        // S_it goes into image set (it + 1) % kK2SBuf, which MMA iteration it + 1 - kK2SBuf
        // read last: with one set, wait for this iteration's outputs (frame it - 1); with
        // two, for the previous iteration's (frame it - 2), whose images are the other set.
        {
            // MMA iteration j commits o_done[j % kK2SBuf], whose phase (j - 1) / kK2SBuf it completes;
            // the next commit there (iteration j + kK2SBuf = it + 1) needs this iteration's images,
            // so the phase waited for is always the latest one of that barrier.
            const int j = it + 1 - kK2SBuf;
            if (j >= 1 && !mbar_wait_warp(&o_done[j % kK2SBuf], ((j - 1) / kK2SBuf) & 1, abort_flag)) break;
        }
        write_images((it + 1) % kK2SBuf);
    }
    if (p.S_out && chunk_idx + 1 == p.n_chunks && row < kD) {
        float *dst = p.S_out + (size_t)bh * kStateFloats + row * kD + kC0;
#pragma unroll
        for (int j = 0; j < kCols; j += 4)
            *reinterpret_cast<float4 *>(dst + j) = make_float4(S[j], S[j + 1], S[j + 2], S[j + 3]);
    }
}

// Named barrier over K2's four output warps (id 0 is __syncthreads).
__device__ __forceinline__ void out_warps_sync() { asm volatile("bar.sync 2, 128;" ::: "memory"); }

// The kernel body, shared by the standalone launch (kStateWarps = 4, TMEM
// allocated here) and the fused chained scan (kStateWarps = 8: warps 10..13 take
// the second half of every state row; tmem_given = the fused kernel's TMEM).
template <int kStateWarps>
__device__ __forceinline__ void k2_body(const CUtensorMap &mapQ, const CUtensorMap &mapO, const K2Params &p,
                                        uint8_t *sm, uint8_t *bar_area, bool own_tmem, uint32_t tmem_given)
{
    static_assert(kStateWarps == 4 || kStateWarps == 8, "K2 state warps");
    uint64_t *bars = reinterpret_cast<uint64_t *>(bar_area);
    uint64_t *q_full = bars + 0, *q_empty = bars + kK2QStages;
    uint64_t *a_full = bars + 2 * kK2QStages, *a_empty = a_full + 1;
    // o_done[m]: the MMAs of iteration j (outputs of frame j - 1) have completed, for j % kK2SBuf == m
    uint64_t *s_ready = a_full + 2, *accS_full = a_full + 3, *o_done = a_full + 4;
    uint64_t *o_full = a_full + 6, *o_free = a_full + 9, *drain = a_full + 12;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(a_full + 13);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(a_full + 14);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int BH = p.B * p.H;
    const int chunk_idx = blockIdx.x / BH, bh = blockIdx.x % BH;
    const int b = bh / p.H, h = bh % p.H;
    int f_begin, nf;
    chunk_frames(chunk_idx, p.F, p.n_chunks, f_begin, nf);
    const int n_tiles = p.states_only ? 0 : (p.N + kTQ - 1) / kTQ;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kK2QStages; ++i) {
            mbar_init(&q_full[i], 1);
            mbar_init(&q_empty[i], 5);  // the tile's MMAs (commit) + the four output warps (norms read)
        }
        mbar_init(drain, 1);
        mbar_init(a_full, 1);
        mbar_init(a_empty, 1);
        mbar_init(s_ready, kStateWarps);
        mbar_init(accS_full, 1);
        for (int i = 0; i < kK2SBuf; ++i) mbar_init(&o_done[i], 1);
        for (int i = 0; i < 3; ++i) {
            mbar_init(&o_full[i], 1);
            mbar_init(&o_free[i], 4);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (own_tmem && warp == 1) {
        tmem_alloc(tmem_slot, 512);
        tmem_relinquish();
    }
    // zero the S images (rows 112..127 and key columns 112..127 stay zero)
    for (int o = threadIdx.x * 16; o < kK2SBuf * (int)kK2SetBytes; o += blockDim.x * 16)
        *reinterpret_cast<uint4 *>(sm + kK2OffShi + o) = make_uint4(0, 0, 0, 0);
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = own_tmem ? *tmem_slot : tmem_given;
    const uint32_t sbase = smem_u32(sm);
    griddep_launch_dependents();
    griddep_wait();
    const uint8_t *ws_chain = p.ws_frames + ((size_t)bh * p.F + f_begin) * kFrameWs;

    if (warp == 0) {
        // ------------------------------------------------------ TMA producers
        // Lane 0 streams the per-frame A_f images, lane 1 the Q tiles, so that
        // neither stream waits behind the other's buffer reuse.  Without
        // outputs lane 0 also prefetches the next frame's U_f into L2 for the
        // state warps; with outputs it does not: a frame ahead, about half of
        // the prefetched lines were evicted by the Q/O stream before their
        // loads (107 MB more DRAM reads per layer, K2 226 -> 239 us).
        if (lane == 0) {
            int a_issued = 0;
            const bool prefetch_u = p.states_only != 0;
            if (prefetch_u) bulk_prefetch_l2(ws_chain + kAimgBytes, kUBytes);
            for (int it = 0; it < nf; ++it) {
                if (it >= 1 && !mbar_wait(a_empty, (it - 1) & 1, abort_flag)) break;
                mbar_arrive_expect_tx(a_full, kAimgBytes);
                bulk_g2s(sm + kK2OffA, ws_chain + (size_t)it * kFrameWs, kAimgBytes, a_full);
                if (prefetch_u && it + 1 < nf)
                    bulk_prefetch_l2(ws_chain + (size_t)(it + 1) * kFrameWs + kAimgBytes, kUBytes);
                ++a_issued;
            }
            if (*abort_flag && a_issued)  // let the copy in flight land before the CTA exits
                mbar_wait_drain(a_full, (a_issued - 1) & 1);
        } else if (lane == 1) {
            const uint64_t pol = policy_stream();
            int qc = 0;
            bool ok = true;
            for (int it = 1; it <= nf && ok; ++it) {
                const int bf = b * p.F + frame_at(f_begin + it - 1, p.F, p.reverse);
                for (int t = 0; t < n_tiles && ok; ++t, ++qc) {
                    const int s = qc % kK2QStages;
                    if (qc >= kK2QStages && !(ok = mbar_wait(&q_empty[s], (qc / kK2QStages - 1) & 1, abort_flag)))
                        break;
                    mbar_arrive_expect_tx(&q_full[s], kImgBytes);
                    uint8_t *dst = sm + s * kImgBytes;
                    tma_load_4d(dst, &mapQ, &q_full[s], 0, h, t * kTQ, bf, pol);
                    tma_load_4d(dst + kImgPanel, &mapQ, &q_full[s], 64, h, t * kTQ, bf, pol);
                }
            }
            if (*abort_flag)
                for (int s = 0; s < kK2QStages && s < qc; ++s) {  // last tile index using stage s
                    const int last = ((qc - 1 - s) / kK2QStages) * kK2QStages + s;
                    mbar_wait_drain(&q_full[s], (last / kK2QStages) & 1);
                }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------- MMA issuer
        if (lane == 0) {
            int qc = 0;
            bool ok = true;
            for (int it = 0; it <= nf && ok; ++it) {
                if (!(ok = mbar_wait(s_ready, it & 1, abort_flag))) break;
                tc_fence_after();
                if (it < nf) {
                    if (!(ok = mbar_wait(a_full, it & 1, abort_flag))) break;
                    tc_fence_after();
                    const uint32_t sset = (uint32_t)(it % kK2SBuf) * kK2SetBytes;
#pragma unroll
                    for (int ks = 0; ks < 7; ++ks) {
                        const uint32_t koff = (ks >> 2) * kImgPanel + (ks & 3) * 32;
                        const uint64_t bd =
                            sdesc_sw128(sbase + kK2OffA + (ks >> 2) * kAimgPanel + (ks & 3) * 32, 16, 1024);
                        mma_bf16(tmem, sdesc_sw128(sbase + kK2OffShi + sset + koff, 16, 1024), bd, kIdescK, ks > 0);
                        if (kK2Lo) mma_bf16(tmem, sdesc_sw128(sbase + kK2OffSlo + sset + koff, 16, 1024), bd, kIdescK, 1);
                    }
                    mma_commit(accS_full);
                    mma_commit(a_empty);
                }
                if (it >= 1) {
                    for (int t = 0; t < n_tiles && ok; ++t, ++qc) {
                        const int s = qc % kK2QStages, slot = qc % 3;
                        if (!(ok = mbar_wait(&q_full[s], (qc / kK2QStages) & 1, abort_flag))) break;
                        if (qc >= 3 && !(ok = mbar_wait(&o_free[slot], ((qc / 3) - 1) & 1, abort_flag))) break;
                        tc_fence_after();
                        const uint32_t acc = tmem + 128 * (slot + 1);
                        const uint32_t qb = sbase + s * kImgBytes;
                        const uint32_t sset = (uint32_t)(it % kK2SBuf) * kK2SetBytes;  // S_{it-1}: image set of iteration it
#pragma unroll
                        for (int ks = 0; ks < 7; ++ks) {
                            const uint32_t koff = (ks >> 2) * kImgPanel + (ks & 3) * 32;
                            const uint64_t ad = sdesc_sw128(qb + koff, 16, 1024);
                            mma_bf16(acc, ad, sdesc_sw128(sbase + kK2OffShi + sset + koff, 16, 1024), kIdescK, ks > 0);
                            if (kK2Lo)
                                mma_bf16(acc, ad, sdesc_sw128(sbase + kK2OffSlo + sset + koff, 16, 1024), kIdescK, 1);
                        }
                        mma_commit(&o_full[slot]);
                        mma_commit(&q_empty[s]);
                    }
                    if (ok) mma_commit(&o_done[it % kK2SBuf]);
                }
            }
            mma_commit(drain);  // every MMA issued above has completed once this phase lands
            mbar_wait_drain(drain, 0);
        }
    } else if (warp < 6) {
        // ------------------------------------------------- state warps (rows)
        if (kStateWarps == 4)
            k2_state_role<kD, 0>(p, sm, tmem, s_ready, accS_full, o_done, abort_flag, bh, b, h, chunk_idx, f_begin, nf,
                                 ws_chain);
        else
            k2_state_role<kD / 2, 0>(p, sm, tmem, s_ready, accS_full, o_done, abort_flag, bh, b, h, chunk_idx,
                                     f_begin, nf, ws_chain);
    } else if (warp >= 10) {
        if (kStateWarps == 8)
            k2_state_role<kD / 2, kD / 2>(p, sm, tmem, s_ready, accS_full, o_done, abort_flag, bh, b, h, chunk_idx,
                                          f_begin, nf, ws_chain);
    } else {
        // ------------------------------------------------ output warps (tokens)
        // Each warp owns 32 token rows of a tile.  It computes their 1/||q||
        // from the Q tile (then releases the Q stage: the tile's MMAs release
        // it too), scales the accumulator rows and writes bf16 into one of two
        // output staging tiles; once all four warps are done, one thread
        // stores the tile as two 128-row boxes (tall boxes stream far better
        // than 32-row ones).  Before a staging tile is rewritten, that thread
        // has seen the store issued from it two tiles earlier finish reading.
        // Every warp runs every iteration (work skipped after an abort), so the
        // named barriers always see all 128 threads.
        const int quad = warp & 3, r = quad * 32 + lane;
        const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
        const bool leader = warp == 6 && lane == 0;
        int qc = 0;
        bool ok = true;
        for (int it = 1; it <= nf; ++it) {
            const int bf = b * p.F + frame_at(f_begin + it - 1, p.F, p.reverse);
            for (int t = 0; t < n_tiles; ++t, ++qc) {
                const int s = qc % kK2QStages, slot = qc % 3;
                const uint8_t *qs = sm + s * kImgBytes;
                uint8_t *os = sm + kK2OffO + (kK2OStages ? qc % kK2OStages : 0) * kImgBytes;
                if (ok) ok = mbar_wait_warp(&q_full[s], (qc / kK2QStages) & 1, abort_flag);
                float rq = 0.f;
                if (ok) {
                    float ss = 0.f;
#pragma unroll
                    for (int c = 0; c < 16; ++c) {
                        const uint4 u = *reinterpret_cast<const uint4 *>(qs + (c >> 3) * kImgPanel + r * kRowB +
                                                                         (((c & 7) ^ (r & 7)) << 4));
                        float f8[8];
                        bf16x8_to_f32(u, f8);
#pragma unroll
                        for (int e = 0; e < 8; ++e) ss = fmaf(f8[e], f8[e], ss);
                    }
                    rq = rsqrtf(ss + kEps);
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&q_empty[s]);
                    ok = mbar_wait_warp(&o_full[slot], (qc / 3) & 1, abort_flag);
                }
                tc_fence_after();
                if (kK2OStages > 0) {
                    if (leader) {  // the store issued from this staging tile kK2OStages tiles ago has read it
                        if (kK2OStages == 2) bulk_wait_read_le1();
                        else bulk_wait_read_all();
                    }
                    out_warps_sync();
                }
                if (ok) {
                    const uint32_t acc = tmem + 128 * (slot + 1) + lane_off;
                    const int n = t * kTQ + r;  // token of this row
                    uint4 *orow = reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(p.o) +
                                                            (((size_t)bf * p.N + n) * p.H + h) * kD);
                    // the row in two TMEM round trips (four chunks, then three)
#pragma unroll
                    for (int cp = 0; cp < 7; cp += 4) {
                    uint32_t ra4[4][16];
#pragma unroll
                    for (int hf = 0; hf < 4 && cp + hf < 7; ++hf) tmem_ld16(acc + (cp + hf) * 16, ra4[hf]);
                    tmem_ld_wait();
#pragma unroll
                    for (int hf = 0; hf < 4 && cp + hf < 7; ++hf) {
                        const int cc = cp + hf;
                        const uint32_t *ra = ra4[hf];
                        float o[16];
#pragma unroll
                        for (int j = 0; j < 16; ++j) o[j] = __uint_as_float(ra[j]) * rq;
                        const int c8 = cc * 2;
                        if (kK2OStages > 0) {
                            *reinterpret_cast<uint4 *>(os + (c8 >> 3) * kImgPanel + sw128_off(r, c8 & 7)) =
                                f32x8_to_bf16(o);
                            *reinterpret_cast<uint4 *>(os + ((c8 + 1) >> 3) * kImgPanel + sw128_off(r, (c8 + 1) & 7)) =
                                f32x8_to_bf16(o + 8);
                        } else if (n < p.N) {  // the row straight to global memory (tail rows past N skipped)
                            orow[c8] = f32x8_to_bf16(o);
                            orow[c8 + 1] = f32x8_to_bf16(o + 8);
                        }
                    }
                    }
                }
                if (kK2OStages > 0) fence_proxy_async_smem();
                tc_fence_before();
                __syncwarp();
                if (lane == 0 && ok) mbar_arrive(&o_free[slot]);
                if (kK2OStages == 0) continue;
                out_warps_sync();
                if (leader && ok) {
                    tma_store_4d(&mapO, os, 0, h, t * kTQ, bf);
                    tma_store_4d(&mapO, os + kImgPanel, 64, h, t * kTQ, bf);
                    bulk_commit();
                }
            }
        }
        if (lane == 0) bulk_wait_all();
    }
    tc_fence_before();
    __syncthreads();
    if (*abort_flag && threadIdx.x == 0) raise_status(p.status);
    if (own_tmem && warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

__global__ void __launch_bounds__(kK2Threads, 1)
    k2_scan_output_kernel(const __grid_constant__ CUtensorMap mapQ, const __grid_constant__ CUtensorMap mapO,
                          const K2Params p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    k2_body<kK2StateWarps>(mapQ, mapO, p, sm, sm + kK2OffBar, true, 0u);
}

// ===================================================================== K5
// Fused chained scan: K1, the chunk-boundary step and K2 in one cooperative
// launch, one CTA per (chunk, chain), all CTAs resident at once.  After its
// frame statistics the CTA still holds its chunk composites C_c and H_c in
// TMEM; it waits for the chunk's start state S_start(c) (published by the
// CTA of chunk c-1; S_in for chunk 0), forms S_start(c+1) = H_c + S_start(c) C_c
// on tcgen05 in place of H_c (S and C as bf16 hi + lo, three MMAs per k-step),
// publishes it with a release flag and runs its own scan and outputs from
// S_start(c).  The chain of start states is the decoupled look-back of the
// chunk aggregates (C_p, H_p composites of the summary page, section
// 技术新颖性), with one hop per chunk instead of a separate launch; every flag
// wait is bounded and sets the timeout status when it runs out.
constexpr uint32_t kK5OffHopS = 0;                     // S_start images: hi, lo (K-major A, row = state row)
constexpr uint32_t kK5OffHopC = 2 * kImgBytes;         // C_c images: hi, lo (MN-major B, row = k index)
constexpr uint32_t kK5OffK2Bar = kK1OffBar + 256;      // K2's barriers (K1's stay at kK1OffBar)
constexpr uint32_t kK5OffHopBar = kK1OffBar + 512;     // hop: MMA barrier + state word
constexpr uint32_t kK5Smem = kK1OffBar + 768 + 1024;
constexpr uint32_t kIdescKMN5 = idesc_bf16(128, kD, false, true);  // A K-major, B MN-major
static_assert(kK5OffHopC + 2 * kImgBytes <= kK2OffBar && kK5Smem <= kMaxSmem, "K5 shared memory");

// Warps 10..13 (the statistics epilogue warps: TMEM lane quadrant = warp & 3).
__device__ __forceinline__ void hop_warps_sync() { asm volatile("bar.sync 5, 128;" ::: "memory"); }

// Returns (to every thread) whether the CTA may run its scan: false after a
// timeout here or in the statistics phase.
__device__ __forceinline__ bool k5_chunk_hop(const K1Params &p1, const K2Params &p2, const float *S_in,
                                             unsigned *flags, uint8_t *sm, uint32_t tmem, int aborted)
{
    uint64_t *bar = reinterpret_cast<uint64_t *>(sm + kK5OffHopBar);
    volatile int *hop_abort = reinterpret_cast<volatile int *>(bar + 1);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int BH = p1.B * p1.H, nch = p1.n_chunks;
    const int chunk_idx = blockIdx.x / BH, bh = blockIdx.x % BH;
    const bool need_next = chunk_idx + 1 < nch;
    float *ws_start = const_cast<float *>(p2.ws_start);
    if (threadIdx.x == 0) {
        mbar_init(bar, 1);
        *hop_abort = aborted ? 1 : 0;
        fence_mbar_init();
    }
    __syncthreads();
    if (warp >= 10 && !*hop_abort) {
        const int quad = warp & 3, row = quad * 32 + lane;
        const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
        // C_c -> bf16 hi/lo images, row = row of C (rows 112.. are zero in TMEM), columns 112..127 zero
        if (need_next) {
#pragma unroll
            for (int cp = 0; cp < 7; cp += 2) {
                uint32_t rc2[2][16];
#pragma unroll
                for (int hf = 0; hf < 2 && cp + hf < 7; ++hf) tmem_ld16(tmem + lane_off + kTmC + (cp + hf) * 16, rc2[hf]);
                tmem_ld_wait();
#pragma unroll
                for (int hf = 0; hf < 2 && cp + hf < 7; ++hf)
#pragma unroll
                    for (int e8 = 0; e8 < 2; ++e8) {
                        const int c8 = 2 * (cp + hf) + e8;
                        float x[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e) x[e] = __uint_as_float(rc2[hf][8 * e8 + e]);
                        uint4 hi, lo;
                        split_bf16x8(x, hi, lo);
                        const uint32_t off = (c8 >> 3) * kImgPanel + sw128_off(row, c8 & 7);
                        *reinterpret_cast<uint4 *>(sm + kK5OffHopC + off) = hi;
                        *reinterpret_cast<uint4 *>(sm + kK5OffHopC + kImgBytes + off) = lo;
                    }
            }
#pragma unroll
            for (int c8 = 14; c8 < 16; ++c8) {
                const uint32_t off = kImgPanel + sw128_off(row, c8 & 7);
                *reinterpret_cast<uint4 *>(sm + kK5OffHopC + off) = make_uint4(0, 0, 0, 0);
                *reinterpret_cast<uint4 *>(sm + kK5OffHopC + kImgBytes + off) = make_uint4(0, 0, 0, 0);
            }
        }
        // the chunk's start state: S_in for chunk 0, else published by chunk c-1
        if (chunk_idx > 0 && warp == 10 && lane == 0) {
            const unsigned *fl = flags + (size_t)bh * nch + chunk_idx;
            const long long t0 = clock64();
            while (ld_acquire_u32(fl) == 0) {
                if (clock64() - t0 > kSpinLimitCycles) {
                    *hop_abort = 1;
                    break;
                }
                __nanosleep(32);
            }
        }
    }
    // every thread loads a part of S_start (one L2 round trip) into the S images;
    // chunk 0 also leaves its copy of S_in where the scan reads its start state
    __syncthreads();
    if (!*hop_abort && (chunk_idx == 0 || need_next)) {
        const float *src = chunk_idx == 0 ? (S_in ? S_in + (size_t)bh * kStateFloats : nullptr)
                                          : ws_start + ((size_t)bh * nch + chunk_idx) * kStateFloats;
        float *own = ws_start + ((size_t)bh * nch + chunk_idx) * kStateFloats;
        constexpr int kItems = 128 * 16;  // (row, 8-column group) of the 128 x 128 images
        constexpr int kPer = (kItems + kK1Threads - 1) / kK1Threads;
        float x[kPer][8];
#pragma unroll
        for (int u = 0; u < kPer; ++u) {
            const int e = threadIdx.x + u * kK1Threads, r = e >> 4, c8 = e & 15;
            if (e < kItems && src && r < kD && c8 < 14) {
                const float4 a4 = __ldcg(reinterpret_cast<const float4 *>(src + r * kD + 8 * c8));
                const float4 b4 = __ldcg(reinterpret_cast<const float4 *>(src + r * kD + 8 * c8 + 4));
                x[u][0] = a4.x; x[u][1] = a4.y; x[u][2] = a4.z; x[u][3] = a4.w;
                x[u][4] = b4.x; x[u][5] = b4.y; x[u][6] = b4.z; x[u][7] = b4.w;
            } else {
#pragma unroll
                for (int i = 0; i < 8; ++i) x[u][i] = 0.f;
            }
        }
#pragma unroll
        for (int u = 0; u < kPer; ++u) {
            const int e = threadIdx.x + u * kK1Threads, r = e >> 4, c8 = e & 15;
            if (e >= kItems) continue;
            if (chunk_idx == 0 && r < kD && c8 < 14) {
                *reinterpret_cast<float4 *>(own + r * kD + 8 * c8) = make_float4(x[u][0], x[u][1], x[u][2], x[u][3]);
                *reinterpret_cast<float4 *>(own + r * kD + 8 * c8 + 4) =
                    make_float4(x[u][4], x[u][5], x[u][6], x[u][7]);
            }
            if (need_next) {
                uint4 hi, lo;
                split_bf16x8(x[u], hi, lo);
                const uint32_t off = (c8 >> 3) * kImgPanel + sw128_off(r, c8 & 7);
                *reinterpret_cast<uint4 *>(sm + kK5OffHopS + off) = hi;
                *reinterpret_cast<uint4 *>(sm + kK5OffHopS + kImgBytes + off) = lo;
            }
        }
        fence_proxy_async_smem();
    }
    tc_fence_before();
    __syncthreads();
    if (warp >= 10) {
        const int quad = warp & 3, row = quad * 32 + lane;
        const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
        if (need_next && !*hop_abort) {
            if (warp == 10 && lane == 0) {
                tc_fence_after();
                const uint32_t sbase = smem_u32(sm);
#pragma unroll
                for (int ks = 0; ks < 7; ++ks) {
                    const uint32_t koff = (ks >> 2) * kImgPanel + (ks & 3) * 32;
                    const uint64_t a_hi = sdesc_sw128(sbase + kK5OffHopS + koff, 16, 1024);
                    const uint64_t a_lo = sdesc_sw128(sbase + kK5OffHopS + kImgBytes + koff, 16, 1024);
                    const uint64_t b_hi = sdesc_sw128(sbase + kK5OffHopC + ks * 2048, kImgPanel, 1024);
                    const uint64_t b_lo = sdesc_sw128(sbase + kK5OffHopC + kImgBytes + ks * 2048, kImgPanel, 1024);
                    mma_bf16(tmem + kTmH, a_hi, b_hi, kIdescKMN5, 1u);
                    mma_bf16(tmem + kTmH, a_lo, b_hi, kIdescKMN5, 1u);
                    mma_bf16(tmem + kTmH, a_hi, b_lo, kIdescKMN5, 1u);
                }
                mma_commit(bar);
            }
            if (mbar_wait_warp(bar, 0, hop_abort)) {
                tc_fence_after();
                float *dst = ws_start + ((size_t)bh * nch + chunk_idx + 1) * kStateFloats;
#pragma unroll
                for (int cp = 0; cp < 7; cp += 4) {
                    uint32_t rh4[4][16];
#pragma unroll
                    for (int hf = 0; hf < 4 && cp + hf < 7; ++hf)
                        tmem_ld16(tmem + lane_off + kTmH + (cp + hf) * 16, rh4[hf]);
                    tmem_ld_wait();
                    if (row < kD)
#pragma unroll
                        for (int hf = 0; hf < 4 && cp + hf < 7; ++hf)
#pragma unroll
                            for (int j = 0; j < 16; j += 4)
                                *reinterpret_cast<float4 *>(dst + row * kD + (cp + hf) * 16 + j) =
                                    make_float4(__uint_as_float(rh4[hf][j]), __uint_as_float(rh4[hf][j + 1]),
                                                __uint_as_float(rh4[hf][j + 2]), __uint_as_float(rh4[hf][j + 3]));
                }
                __threadfence();
                tc_fence_before();
                hop_warps_sync();
                if (warp == 10 && lane == 0) st_release_u32(flags + (size_t)bh * nch + chunk_idx + 1, 1u);
            } else if (warp == 10 && lane == 0) {
                // let the hop's MMAs land before the CTA moves on
                mbar_wait_drain(bar, 0);
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const bool ok = *hop_abort == 0;
    if (!ok && threadIdx.x == 0 && !aborted) raise_status(p1.status);
    return ok;
}

__global__ void __launch_bounds__(kK1Threads, 1)
    k5_fused_scan_kernel(const __grid_constant__ CUtensorMap mapK, const __grid_constant__ CUtensorMap mapV,
                         const __grid_constant__ CUtensorMap mapQ, const __grid_constant__ CUtensorMap mapO,
                         const K1Params p1, const K2Params p2, const float *S_in, unsigned *flags)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    int aborted = 0;
    const uint32_t tmem = k1_body<true>(mapK, mapV, p1, sm, &aborted);
    if (k5_chunk_hop(p1, p2, S_in, flags, sm, tmem, aborted))
        k2_body<8>(mapQ, mapO, p2, sm, sm + kK5OffK2Bar, false, tmem);
    tc_fence_before();
    __syncthreads();
    if ((threadIdx.x >> 5) == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// ================================================================= host side
namespace {

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    }
    return fn;
}

}  // namespace

// 4-D view [B*F][N][H][D] of a bf16 [B][F*N][H][D] tensor, 128B swizzle,
// boxes of 64 head-dim elements x `rows` tokens of one head of one frame.
bool make_token_map(CUtensorMap *m, const void *base, int B, int H, int F, int N, int rows)
{
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[4] = {(cuuint64_t)kD, (cuuint64_t)H, (cuuint64_t)N, (cuuint64_t)B * F};
    cuuint64_t strides[3] = {(cuuint64_t)kD * 2, (cuuint64_t)H * kD * 2, (cuuint64_t)N * H * kD * 2};
    cuuint32_t box[4] = {64, 1, (cuuint32_t)rows, 1};
    cuuint32_t es[4] = {1, 1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(base), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 4-D view [B*F][N][H][D] of an fp32 [B][F*N][H][D] tensor for TMA stores:
// 64-byte swizzle, boxes of 16 head-dim elements x `rows` tokens of one head
// of one frame (the smem box is `rows` rows of 64 bytes, 16-byte chunk c of
// row r at chunk position c ^ ((r >> 1) & 3)).
bool make_f32_row_map(CUtensorMap *m, void *base, int B, int H, int F, int N, int rows)
{
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[4] = {(cuuint64_t)kD, (cuuint64_t)H, (cuuint64_t)N, (cuuint64_t)B * F};
    cuuint64_t strides[3] = {(cuuint64_t)kD * 4, (cuuint64_t)H * kD * 4, (cuuint64_t)N * H * kD * 4};
    cuuint32_t box[4] = {16, 1, (cuuint32_t)rows, 1};
    cuuint32_t es[4] = {1, 1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, base, dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D view of a bf16 row-major [rows][cols] matrix, 128B swizzle, boxes of
// 64 columns (one swizzled 128-byte row) x `box_rows` rows.  cols must be a
// multiple of 8 (16-byte row stride); out-of-range elements load as zero.
bool make_matrix_map(CUtensorMap *m, const void *base, int rows, int cols, int box_rows)
{
    auto fn = encode_fn();
    if (!fn || rows <= 0 || cols <= 0 || cols % 8 != 0 || box_rows <= 0 || box_rows > 256) return false;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
    cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
    cuuint32_t es[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool tc_plan(int B, int H, int F, int N, int force_chunks, TcPlan *plan)
{
    if (B <= 0 || H <= 0 || F <= 0 || N <= 0) return false;
    const long long BH = (long long)B * H;
    if (BH > (1 << 20) || (long long)F * N > (1LL << 30)) return false;
    // Chunk count minimising (waves of one-CTA-per-SM) x (frames per chunk),
    // plus a small charge for each sequential boundary step.
    int best_n = 1;
    double best = 1e300;
    for (int n = 1; n <= F && force_chunks <= 0; ++n) {
        const int L = (F + n - 1) / n;
        const int n_real = (F + L - 1) / L;
        if (n_real != n) continue;
        const long long ctas = BH * n;
        const double waves = (double)((ctas + kSms - 1) / kSms);
        const double cost = waves * L * 1.0 + 0.04 * n;
        if (cost < best - 1e-9) {
            best = cost;
            best_n = n;
        }
    }
    plan->B = B;
    plan->H = H;
    plan->F = F;
    plan->N = N;
    if (force_chunks > F) return false;
    const int n = force_chunks > 0 ? force_chunks : best_n;
    plan->chunk = (F + n - 1) / n;
    plan->n_chunks = (F + plan->chunk - 1) / plan->chunk;
    plan->off_frames = 0;
    plan->off_comp = align_up((size_t)BH * F * kFrameWs, 256);
    plan->off_start = align_up(plan->off_comp + (size_t)BH * plan->n_chunks * 2 * kStateBytes, 256);
    plan->off_flags = align_up(plan->off_start + (size_t)BH * plan->n_chunks * kStateBytes, 256);
    plan->ws_bytes = align_up(plan->off_flags + (size_t)BH * plan->n_chunks * sizeof(unsigned), 256);
    return true;
}

namespace {
// Launch with programmatic stream serialization: the kernel may be scheduled
// while the previous kernel on the stream finishes; it calls griddepcontrol.wait
// before touching global memory.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, int threads, size_t smem, cudaStream_t stream,
                       Args... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

constexpr int kMaxDevTc = 64;
bool g_tc_attrs[kMaxDevTc];

// Opt the kernels into their shared-memory sizes, once per device.
cudaError_t prepare_tc_kernels()
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevTc) return cudaErrorInvalidDevice;
    if (g_tc_attrs[dev]) return cudaSuccess;
    e = cudaFuncSetAttribute(k1_frame_stats_kernel<kK1Fwd>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kK1Smem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(k1_frame_stats_kernel<kK1RevA>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kK1Smem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(k1_frame_stats_kernel<kK1E>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kK1Smem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(k2_scan_output_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kK2Smem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(k1b_chunk_boundary_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kK1bSmem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(k5_fused_scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kK5Smem);
    if (e != cudaSuccess) return e;
    g_tc_attrs[dev] = true;
    return cudaSuccess;
}

K1Params k1_params(const float *beta, const float *gamma, const TcPlan &pl, float c, int reverse, uint8_t *ws,
                   unsigned *status)
{
    K1Params p1;
    p1.beta = beta;
    p1.gamma = gamma;
    p1.ws_frames = ws + pl.off_frames;
    p1.ws_comp = reinterpret_cast<float *>(ws + pl.off_comp);
    p1.status = status;
    p1.B = pl.B;
    p1.H = pl.H;
    p1.F = pl.F;
    p1.N = pl.N;
    p1.chunk = pl.chunk;
    p1.n_chunks = pl.n_chunks;
    p1.c = c;
    p1.reverse = reverse;
    p1.withhold_loads = pl.withhold_loads;
    p1.ws_rev = nullptr;
    return p1;
}
}  // namespace

// Composites of a whole run of frames for context parallelism: K1 over the
// plan's chunks (the same launch as the forward, every SM busy, the per-frame
// statistics left in the workspace), then the chunk composites composed in
// frame order by the chunk-boundary kernel: from the identity with no inputs it
// yields C = C_0 C_1 ... C_{n-1}, from zero with the inputs H = the state the
// run reaches from zero.
cudaError_t launch_frame_composite_tc(const void *k, const void *v, const float *beta, const float *gamma,
                                      float *C_out, float *H_out, const TcPlan &pl, float c, void *workspace,
                                      unsigned *status, cudaStream_t stream)
{
    CUtensorMap mk, mv;
    if (!make_token_map(&mk, k, pl.B, pl.H, pl.F, pl.N, kTS) || !make_token_map(&mv, v, pl.B, pl.H, pl.F, pl.N, kTS))
        return cudaErrorInvalidValue;
    cudaError_t e = prepare_tc_kernels();
    if (e != cudaSuccess) return e;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    const int BH = pl.B * pl.H;
    const K1Params p1 = k1_params(beta, gamma, pl, c, 0, ws, status);
    if ((e = launch_pdl(k1_frame_stats_kernel<kK1Fwd>, dim3(BH * pl.n_chunks), kK1Threads, kK1Smem, stream, mk, mv, p1)) !=
        cudaSuccess)
        return e;
    const float *comp = p1.ws_comp;
    const size_t chain_stride = (size_t)pl.n_chunks * 2 * kStateFloats, chunk_stride = (size_t)2 * kStateFloats;
    if (C_out && (e = launch_pdl(k1b_chunk_boundary_kernel, dim3(BH, kD / kK1bRows), kK1bThreads, kK1bSmem, stream,
                                 comp, comp + kStateFloats, chain_stride, chunk_stride, (float *)nullptr,
                                 (const float *)nullptr, C_out, pl.n_chunks, status,
                                 kK1bIdentityIn | kK1bZeroH)) != cudaSuccess)
        return e;
    if (H_out && (e = launch_pdl(k1b_chunk_boundary_kernel, dim3(BH, kD / kK1bRows), kK1bThreads, kK1bSmem, stream,
                                 comp, comp + kStateFloats, chain_stride, chunk_stride, (float *)nullptr,
                                 (const float *)nullptr, H_out, pl.n_chunks, status, 0)) != cudaSuccess)
        return e;
    return cudaSuccess;
}

cudaError_t launch_state_compose_tc(const float *S, const float *C, const float *H, float *S_out, int BH,
                                    unsigned *status, cudaStream_t stream)
{
    cudaError_t e = prepare_tc_kernels();
    if (e != cudaSuccess) return e;
    return launch_pdl(k1b_chunk_boundary_kernel, dim3(BH, kD / kK1bRows), kK1bThreads, kK1bSmem, stream, C, H,
                      (size_t)kStateFloats, (size_t)0, (float *)nullptr, S, S_out, 1, status, 0);
}

// K1 alone over a plan: per-frame A_f image and U_f (and chunk composites) in the workspace.
cudaError_t launch_frame_stats_tc(const void *k, const void *v, const float *beta, const float *gamma,
                                  const TcPlan &pl, float c, int reverse, void *workspace, unsigned *status,
                                  cudaStream_t stream, uint8_t *ws_rev, int e_mode)
{
    CUtensorMap mk, mv;
    if (!make_token_map(&mk, k, pl.B, pl.H, pl.F, pl.N, kTS) || !make_token_map(&mv, v, pl.B, pl.H, pl.F, pl.N, kTS))
        return cudaErrorInvalidValue;
    cudaError_t e = prepare_tc_kernels();
    if (e != cudaSuccess) return e;
    K1Params p1 = k1_params(beta, gamma, pl, c, reverse, static_cast<uint8_t *>(workspace), status);
    p1.ws_rev = ws_rev;
    if (ws_rev && e_mode)
        return launch_pdl(k1_frame_stats_kernel<kK1E>, dim3(pl.B * pl.H * pl.n_chunks), kK1Threads, kK1Smem, stream,
                          mk, mv, p1);
    if (ws_rev)
        return launch_pdl(k1_frame_stats_kernel<kK1RevA>, dim3(pl.B * pl.H * pl.n_chunks), kK1Threads, kK1Smem,
                          stream, mk, mv, p1);
    return launch_pdl(k1_frame_stats_kernel<kK1Fwd>, dim3(pl.B * pl.H * pl.n_chunks), kK1Threads, kK1Smem, stream, mk, mv,
                      p1);
}

// K1b + K2: chunk-boundary states from the chunk composites in the workspace,
// then the scan/output kernel.  events (optional) get records [2] and [3].
static cudaError_t launch_scan_output_tc(const void *q, const float *gamma, const float *S_in, float *S_out, void *o,
                                         const TcPlan &pl, int reverse, uint8_t *ws, unsigned *status,
                                         cudaStream_t stream, cudaEvent_t *events)
{
    CUtensorMap mq, mo;
    if (!make_token_map(&mq, q, pl.B, pl.H, pl.F, pl.N, kTQ) || !make_token_map(&mo, o, pl.B, pl.H, pl.F, pl.N, kTQ))
        return cudaErrorInvalidValue;
    const int BH = pl.B * pl.H;
    const float *comp = reinterpret_cast<const float *>(ws + pl.off_comp);
    cudaError_t e = launch_pdl(k1b_chunk_boundary_kernel, dim3(BH, kD / kK1bRows), kK1bThreads, kK1bSmem, stream,
                               comp, comp + kStateFloats, (size_t)pl.n_chunks * 2 * kStateFloats,
                               (size_t)2 * kStateFloats, reinterpret_cast<float *>(ws + pl.off_start), S_in,
                               (float *)nullptr, pl.n_chunks, status, 0);
    if (e != cudaSuccess) return e;
    if (events && (e = cudaEventRecord(events[2], stream)) != cudaSuccess) return e;
    K2Params p2;
    p2.o = o;
    p2.gamma = gamma;
    p2.ws_frames = ws + pl.off_frames;
    p2.ws_start = reinterpret_cast<const float *>(ws + pl.off_start);
    p2.S_out = S_out;  // the last chunk's state after its last frame
    p2.states = nullptr;
    p2.states_only = 0;
    p2.status = status;
    p2.B = pl.B;
    p2.H = pl.H;
    p2.F = pl.F;
    p2.N = pl.N;
    p2.chunk = pl.chunk;
    p2.n_chunks = pl.n_chunks;
    p2.reverse = reverse;
    e = launch_pdl(k2_scan_output_kernel, dim3(BH * pl.n_chunks), kK2Threads, kK2Smem, stream, mq, mo, p2);
    if (e != cudaSuccess) return e;
    if (events && (e = cudaEventRecord(events[3], stream)) != cudaSuccess) return e;
    return cudaSuccess;
}

// K1b + K2 over a plan whose workspace already holds K1's statistics and chunk
// composites (left there by launch_frame_composite_tc on the same frames).
cudaError_t launch_fwd_resume_tc(const void *q, const float *gamma, const float *S_in, float *S_out, void *o,
                                 const TcPlan &pl, void *workspace, unsigned *status, cudaStream_t stream)
{
    cudaError_t e = prepare_tc_kernels();
    if (e != cudaSuccess) return e;
    return launch_scan_output_tc(q, gamma, S_in, S_out, o, pl, 0, static_cast<uint8_t *>(workspace), status, stream,
                                 nullptr);
}

// The state chain alone (K1b + K2 without outputs) over a plan whose workspace
// and chunk composites: K1b from S_in (null: zero), then K2 without outputs,
// storing the state after every frame (states, [B*H][F][D][D]) and the final
// state (S_out, may be null).  q only shapes K2's (unused) tensor maps.
cudaError_t launch_states_tc(const void *q, const float *gamma, const float *S_in, float *S_out, float *states,
                             const TcPlan &pl, uint8_t *ws, unsigned *status, cudaStream_t stream)
{
    CUtensorMap mq;
    if (!make_token_map(&mq, q, pl.B, pl.H, pl.F, pl.N, kTQ)) return cudaErrorInvalidValue;
    cudaError_t e = prepare_tc_kernels();
    if (e != cudaSuccess) return e;
    const int BH = pl.B * pl.H;
    const float *comp = reinterpret_cast<const float *>(ws + pl.off_comp);
    e = launch_pdl(k1b_chunk_boundary_kernel, dim3(BH, kD / kK1bRows), kK1bThreads, kK1bSmem, stream, comp,
                   comp + kStateFloats, (size_t)pl.n_chunks * 2 * kStateFloats, (size_t)2 * kStateFloats,
                   reinterpret_cast<float *>(ws + pl.off_start), S_in, (float *)nullptr, pl.n_chunks, status, 0);
    if (e != cudaSuccess) return e;
    K2Params p2;
    p2.o = nullptr;
    p2.gamma = gamma;
    p2.ws_frames = ws + pl.off_frames;
    p2.ws_start = reinterpret_cast<const float *>(ws + pl.off_start);
    p2.S_out = S_out;
    p2.states = states;
    p2.states_only = 1;
    p2.status = status;
    p2.B = pl.B;
    p2.H = pl.H;
    p2.F = pl.F;
    p2.N = pl.N;
    p2.chunk = pl.chunk;
    p2.n_chunks = pl.n_chunks;
    p2.reverse = 0;
    return launch_pdl(k2_scan_output_kernel, dim3(BH * pl.n_chunks), kK2Threads, kK2Smem, stream, mq, mq, p2);
}

cudaError_t launch_frame_fwd_tc(const void *q, const void *k, const void *v, const float *beta, const float *gamma,
                                const float *S_in, float *S_out, void *o, const TcPlan &pl, float c, int reverse,
                                void *workspace, unsigned *status, cudaStream_t stream, cudaEvent_t *events)
{
    CUtensorMap mk, mv;
    if (!make_token_map(&mk, k, pl.B, pl.H, pl.F, pl.N, kTS) || !make_token_map(&mv, v, pl.B, pl.H, pl.F, pl.N, kTS))
        return cudaErrorInvalidValue;
    cudaError_t e = prepare_tc_kernels();
    if (e != cudaSuccess) return e;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    const K1Params p1 = k1_params(beta, gamma, pl, c, reverse, ws, status);
    if (events && (e = cudaEventRecord(events[0], stream)) != cudaSuccess) return e;
    e = launch_pdl(k1_frame_stats_kernel<kK1Fwd>, dim3(pl.B * pl.H * pl.n_chunks), kK1Threads, kK1Smem, stream, mk, mv, p1);
    if (e != cudaSuccess) return e;
    if (events && (e = cudaEventRecord(events[1], stream)) != cudaSuccess) return e;
    return launch_scan_output_tc(q, gamma, S_in, S_out, o, pl, reverse, ws, status, stream, events);
}

// The fused chained scan (K5) in one cooperative launch.  Every CTA must be
// resident at once (the chunk hops wait on one another): when the plan's
// chunk x chain count exceeds the device's SMs, cudaErrorCooperativeLaunchTooLarge
// comes back and nothing is launched.  The hop flags are cleared on the stream
// first.
cudaError_t launch_frame_fwd_fused_tc(const void *q, const void *k, const void *v, const float *beta,
                                      const float *gamma, const float *S_in, float *S_out, void *o, const TcPlan &pl,
                                      float c, int reverse, void *workspace, unsigned *status, cudaStream_t stream)
{
    CUtensorMap mk, mv, mq, mo;
    if (!make_token_map(&mk, k, pl.B, pl.H, pl.F, pl.N, kTS) || !make_token_map(&mv, v, pl.B, pl.H, pl.F, pl.N, kTS) ||
        !make_token_map(&mq, q, pl.B, pl.H, pl.F, pl.N, kTQ) || !make_token_map(&mo, o, pl.B, pl.H, pl.F, pl.N, kTQ))
        return cudaErrorInvalidValue;
    cudaError_t e = prepare_tc_kernels();
    if (e != cudaSuccess) return e;
    int dev = 0, sms = 0, per_sm = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k5_fused_scan_kernel, kK1Threads, kK5Smem)) !=
        cudaSuccess)
        return e;
    const int grid = pl.B * pl.H * pl.n_chunks;
    if ((long long)grid > (long long)sms * per_sm) return cudaErrorCooperativeLaunchTooLarge;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    unsigned *flags = reinterpret_cast<unsigned *>(ws + pl.off_flags);
    if ((e = cudaMemsetAsync(flags, 0, (size_t)pl.B * pl.H * pl.n_chunks * sizeof(unsigned), stream)) != cudaSuccess)
        return e;
    const K1Params p1 = k1_params(beta, gamma, pl, c, reverse, ws, status);
    K2Params p2;
    p2.o = o;
    p2.gamma = gamma;
    p2.ws_frames = ws + pl.off_frames;
    p2.ws_start = reinterpret_cast<const float *>(ws + pl.off_start);
    p2.S_out = S_out;
    p2.states = nullptr;
    p2.states_only = 0;
    p2.status = status;
    p2.B = pl.B;
    p2.H = pl.H;
    p2.F = pl.F;
    p2.N = pl.N;
    p2.chunk = pl.chunk;
    p2.n_chunks = pl.n_chunks;
    p2.reverse = reverse;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kK1Threads);
    cfg.dynamicSmemBytes = kK5Smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k5_fused_scan_kernel, mk, mv, mq, mo, p1, p2, S_in, flags);
}

// Token-ordered reading: per-frame transitions from the UT-transform kernel
// and their chunk composites (gdn_product.cu), in the workspace format the
// sum reading's frame-statistics kernel produces; then K1b and K2 as there.
cudaError_t launch_frame_fwd_product_tc(const void *q, const void *k, const void *v, const float *beta,
                                        const float *gamma, const float *S_in, float *S_out, void *o,
                                        const TcPlan &pl, float c, int reverse, void *workspace, unsigned *status,
                                        cudaStream_t stream)
{
    cudaError_t e = prepare_tc_kernels();
    if (e != cudaSuccess) return e;
    if ((e = launch_frame_product_tc(k, v, beta, pl, c, reverse, workspace, status, stream)) != cudaSuccess) return e;
    if ((e = launch_chunk_composite_tc(gamma, pl, reverse, workspace, status, stream)) != cudaSuccess) return e;
    return launch_scan_output_tc(q, gamma, S_in, S_out, o, pl, reverse, static_cast<uint8_t *>(workspace), status,
                                 stream, nullptr);
}

}  // namespace gdn
