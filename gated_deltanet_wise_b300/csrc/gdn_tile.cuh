// gdn_tile.cuh — layout constants and small device helpers shared by the
// tensor-core kernels of the D = 112 path (multi-frame forward and streaming
// step): swizzled bf16 tile images, fp32 <-> bf16 conversions and the hi/lo
// split used to keep fp32 accuracy through bf16 MMA operands.
#pragma once

#include "gdn_ptx.cuh"

namespace gdn {

constexpr int kD = 112;               // head size this path is built for
constexpr int kSms = 148;             // B300 SM count: the chunk plan targets it
constexpr float kEps = 1e-12f;        // ||x|| = sqrt(sum x^2 + eps)

constexpr uint32_t kRowB = 128;                      // one swizzled row: 64 bf16
constexpr uint32_t kAimgPanel = kD * kRowB;          // 14336: A_f image, 112 rows
constexpr uint32_t kAimgBytes = 2 * kAimgPanel;      // 28672
// U_f in the frame workspace: fp32, stored as float4 column quads, quad-major:
// float4 index (c4 * kD + i) holds U[i][4 c4 .. 4 c4 + 3].  A warp whose lanes
// are consecutive rows reads or writes 512 contiguous bytes per access.
constexpr uint32_t kUBytes = kD * kD * 4;            // 50176
constexpr uint32_t kFrameWs = kAimgBytes + kUBytes;  // 78848 bytes per (chain, frame)
constexpr uint32_t kImgPanel = 128 * kRowB;          // 16384: 128-row bf16 image panel
constexpr uint32_t kImgBytes = 2 * kImgPanel;        // 32768
constexpr uint32_t kStateFloats = kD * kD;           // 12544
constexpr size_t kStateBytes = kStateFloats * 4;     // 50176
constexpr uint32_t kMaxSmem = 232448;                // dynamic shared memory a CTA may opt into

// instruction descriptors (M = 128, N = 112)
constexpr uint32_t kIdescMN = idesc_bf16(128, kD, true, true);    // token-contraction GEMMs
constexpr uint32_t kIdescK = idesc_bf16(128, kD, false, false);   // D-contraction GEMMs

// Frame visited at processing position p: the scan runs over frames in
// increasing order, or, for the reverse-direction scan, from the last frame
// to the first.  Per-frame workspace slots are indexed by processing position.
__host__ __device__ __forceinline__ int frame_at(int p, int F, int reverse) { return reverse ? F - 1 - p : p; }

// Frames [f_begin, f_begin + nf) of chunk c when F frames are cut into n chunks
// as evenly as possible, the longer chunks first (lengths differ by at most one):
// chunks that start their scan later, after more boundary steps, get no more
// frames than earlier ones.
__host__ __device__ __forceinline__ void chunk_frames(int c, int F, int n, int &f_begin, int &nf)
{
    const int base = F / n, rem = F % n;
    nf = base + (c < rem ? 1 : 0);
    f_begin = c * base + (c < rem ? c : rem);
}

__device__ __forceinline__ void raise_status(unsigned *status)
{
    if (status) atomicOr(status, kStatusTimeout);
}

__device__ __forceinline__ void bf16x8_to_f32(const uint4 &u, float *f)
{
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
}

__device__ __forceinline__ uint4 f32x8_to_bf16(const float *f)
{
    uint4 u;
    u.x = pack_bf16x2(f[0], f[1]);
    u.y = pack_bf16x2(f[2], f[3]);
    u.z = pack_bf16x2(f[4], f[5]);
    u.w = pack_bf16x2(f[6], f[7]);
    return u;
}

// hi = bf16(x), lo = bf16(x - hi) for 8 values.
__device__ __forceinline__ void split_bf16x8(const float *x, uint4 &hi, uint4 &lo)
{
    float r[8];
    hi = f32x8_to_bf16(x);
    bf16x8_to_f32(hi, r);
#pragma unroll
    for (int i = 0; i < 8; ++i) r[i] = x[i] - r[i];
    lo = f32x8_to_bf16(r);
}

}  // namespace gdn
