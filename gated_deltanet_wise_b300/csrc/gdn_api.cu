// gdn_api.cu — the C ABI (include/gdn.h): argument validation, workspace
// sizing, the per-device status word, and dispatch to the kernels.
#include <cuda_runtime.h>
#include <math.h>
#include <mutex>

#include "../../include/gdn.h"
#include "gdn_internal.h"

namespace gdn {

// One status word per device.  Kernels OR status bits into it; the host reads
// and clears it in gdn_device_status().
__device__ unsigned g_status_word;

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_mu;
unsigned *g_status_ptr[kMaxDevices];

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

float default_key_scale(float key_scale, int D, int N)
{
    if (key_scale > 0.f) return key_scale;
    return N > 0 ? (float)(1.0 / sqrt((double)D * (double)N)) : 0.f;
}
}  // namespace

unsigned *device_status_word()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_status_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return nullptr;
        g_status_ptr[dev] = static_cast<unsigned *>(p);
    }
    return g_status_ptr[dev];
}

}  // namespace gdn

namespace gdn {
namespace {
// Composite of frames without tokens: C = (prod_f gamma_f) I, H = 0.
__global__ void composite_decay_kernel(const float *gamma, float *C, float *Hc, int H, int F, int D)
{
    const int bh = blockIdx.x, b = bh / H, h = bh % H;
    float g = 1.f;
    for (int f = 0; f < F; ++f) g *= gamma[((size_t)b * F + f) * H + h];
    for (int e = threadIdx.x; e < D * D; e += blockDim.x) {
        if (C) C[(size_t)bh * D * D + e] = (e / D == e % D) ? g : 0.f;
        if (Hc) Hc[(size_t)bh * D * D + e] = 0.f;
    }
}
}  // namespace
}  // namespace gdn

using namespace gdn;

extern "C" {

int gdn_version(void) { return 100; }

const char *gdn_status_string(gdn_status_t s)
{
    switch (s) {
    case GDN_OK: return "ok";
    case GDN_ERR_INVALID_ARG: return "invalid argument";
    case GDN_ERR_UNSUPPORTED: return "unsupported configuration";
    case GDN_ERR_CUDA: return "CUDA runtime error";
    case GDN_ERR_TIMEOUT: return "device-side wait timed out";
    case GDN_ERR_WORKSPACE: return "workspace missing or too small";
    }
    return "unknown status";
}

static size_t fwd_workspace_size(int B, int H, int F, int N, int D, unsigned flags)
{
    if (B < 0 || H < 0 || F < 0 || N < 0 || D <= 0) return (size_t)-1;
    if (flags & ~(unsigned)(GDN_FWD_PRODUCT | GDN_FWD_REVERSE | GDN_FWD_FUSED)) return (size_t)-1;
    if ((flags & GDN_FWD_PRODUCT) && (flags & GDN_FWD_FUSED)) return (size_t)-1;
    if (B == 0 || H == 0 || F == 0 || N == 0) return 0;
    if (D != 112) return (size_t)-1;
    TcPlan plan;
    if (!tc_plan(B, H, F, N, 0, &plan)) return (size_t)-1;
    return (flags & GDN_FWD_PRODUCT) ? product_ws_bytes(plan) : plan.ws_bytes;
}

size_t gdn_frame_fwd_workspace_size(int B, int H, int F, int N, int D) { return fwd_workspace_size(B, H, F, N, D, 0); }

size_t gdn_frame_fwd_product_workspace_size(int B, int H, int F, int N, int D)
{
    return fwd_workspace_size(B, H, F, N, D, GDN_FWD_PRODUCT);
}

size_t gdn_frame_fwd_ex_workspace_size(int B, int H, int F, int N, int D, unsigned flags)
{
    return fwd_workspace_size(B, H, F, N, D, flags);
}

static gdn_status_t frame_fwd_impl(const void *q, const void *k, const void *v, const float *beta,
                                   const float *gamma, const float *S_in, float *S_out, void *o, int B, int H, int F,
                                   int N, int D, float key_scale, unsigned flags, void *workspace,
                                   size_t workspace_bytes, gdn_stream_t stream, void **events,
                                   int withhold_loads = 0)
{
    if (B < 0 || H < 0 || F < 0 || N < 0 || D <= 0) return GDN_ERR_INVALID_ARG;
    if (flags & ~(unsigned)(GDN_FWD_PRODUCT | GDN_FWD_REVERSE | GDN_FWD_FUSED)) return GDN_ERR_INVALID_ARG;
    if (B == 0 || H == 0) return GDN_OK;
    if (D != 112) return GDN_ERR_UNSUPPORTED;
    if ((flags & GDN_FWD_PRODUCT) && (flags & GDN_FWD_FUSED)) return GDN_ERR_UNSUPPORTED;
    if ((S_in && !aligned(S_in, 16)) || (S_out && !aligned(S_out, 16))) return GDN_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (F == 0 || N == 0) {  // no tokens: every reading and direction gives S_out = (prod gamma) S_in
        if (F > 0 && (!gamma || !aligned(gamma, 4))) return GDN_ERR_INVALID_ARG;
        if (!S_out) return GDN_OK;
        return launch_decay_only(gamma, S_in, S_out, B, H, F, D, st) == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
    }
    if (!q || !k || !v || !o || !beta || !gamma) return GDN_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) || !aligned(beta, 4) ||
        !aligned(gamma, 4))
        return GDN_ERR_INVALID_ARG;
    const bool product = (flags & GDN_FWD_PRODUCT) != 0;
    const int reverse = (flags & GDN_FWD_REVERSE) ? 1 : 0;
    TcPlan plan;
    if (!tc_plan(B, H, F, N, 0, &plan)) return GDN_ERR_UNSUPPORTED;
    const size_t need = product ? product_ws_bytes(plan) : plan.ws_bytes;
    if (!workspace || workspace_bytes < need) return GDN_ERR_WORKSPACE;
    if (!aligned(workspace, 16)) return GDN_ERR_INVALID_ARG;
    unsigned *status = device_status_word();
    if (!status) return GDN_ERR_CUDA;
    plan.withhold_loads = withhold_loads;
    const float c = default_key_scale(key_scale, D, N);
    if (flags & GDN_FWD_FUSED) {
        const cudaError_t ef =
            launch_frame_fwd_fused_tc(q, k, v, beta, gamma, S_in, S_out, o, plan, c, reverse, workspace, status, st);
        if (ef != cudaErrorCooperativeLaunchTooLarge) return ef == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
        (void)cudaGetLastError();  // too many CTAs to be resident at once: the three-launch path
    }
    cudaError_t e = product ? launch_frame_fwd_product_tc(q, k, v, beta, gamma, S_in, S_out, o, plan, c, reverse,
                                                          workspace, status, st)
                            : launch_frame_fwd_tc(q, k, v, beta, gamma, S_in, S_out, o, plan, c, reverse, workspace,
                                                  status, st, reinterpret_cast<cudaEvent_t *>(events));
    return e == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

gdn_status_t gdn_frame_fwd(const void *q, const void *k, const void *v, const float *beta, const float *gamma,
                           const float *S_in, float *S_out, void *o, int B, int H, int F, int N, int D,
                           float key_scale, void *workspace, size_t workspace_bytes, gdn_stream_t stream)
{
    return frame_fwd_impl(q, k, v, beta, gamma, S_in, S_out, o, B, H, F, N, D, key_scale, 0, workspace,
                          workspace_bytes, stream, nullptr);
}

gdn_status_t gdn_frame_fwd_product(const void *q, const void *k, const void *v, const float *beta,
                                   const float *gamma, const float *S_in, float *S_out, void *o, int B, int H,
                                   int F, int N, int D, float key_scale, void *workspace, size_t workspace_bytes,
                                   gdn_stream_t stream)
{
    return frame_fwd_impl(q, k, v, beta, gamma, S_in, S_out, o, B, H, F, N, D, key_scale, GDN_FWD_PRODUCT,
                          workspace, workspace_bytes, stream, nullptr);
}

gdn_status_t gdn_frame_fwd_ex(const void *q, const void *k, const void *v, const float *beta, const float *gamma,
                              const float *S_in, float *S_out, void *o, int B, int H, int F, int N, int D,
                              float key_scale, unsigned flags, void *workspace, size_t workspace_bytes,
                              gdn_stream_t stream)
{
    return frame_fwd_impl(q, k, v, beta, gamma, S_in, S_out, o, B, H, F, N, D, key_scale, flags, workspace,
                          workspace_bytes, stream, nullptr);
}

gdn_status_t gdn_frame_fwd_profiled(const void *q, const void *k, const void *v, const float *beta,
                                    const float *gamma, const float *S_in, float *S_out, void *o, int B, int H,
                                    int F, int N, int D, float key_scale, void *workspace, size_t workspace_bytes,
                                    gdn_stream_t stream, void **events)
{
    return frame_fwd_impl(q, k, v, beta, gamma, S_in, S_out, o, B, H, F, N, D, key_scale, 0, workspace,
                          workspace_bytes, stream, events);
}

gdn_status_t gdn_test_frame_fwd_expired_wait(const void *q, const void *k, const void *v, const float *beta,
                                              const float *gamma, const float *S_in, float *S_out, void *o, int B,
                                              int H, int F, int N, int D, float key_scale, void *workspace,
                                              size_t workspace_bytes, gdn_stream_t stream)
{
    return frame_fwd_impl(q, k, v, beta, gamma, S_in, S_out, o, B, H, F, N, D, key_scale, 0, workspace,
                          workspace_bytes, stream, nullptr, 1);
}

// The backward's per-frame kernels put the frame index on a grid dimension
// limited to 65,535, so longer runs are refused before anything is enqueued.
constexpr int kBwdMaxFrames = 65535;

size_t gdn_frame_bwd_workspace_size(int B, int H, int F, int N, int D)
{
    if (B < 0 || H < 0 || F < 0 || N < 0 || D <= 0) return (size_t)-1;
    if (B == 0 || H == 0 || F == 0) return 0;
    if (D != 112 || N == 0 || F >= kBwdMaxFrames) return (size_t)-1;
    return bwd_workspace_bytes(B, H, F, N);
}

gdn_status_t gdn_frame_bwd(const void *q, const void *k, const void *v, const float *beta, const float *gamma,
                           const float *S_in, const void *dO, const float *dS_out, float *dq, float *dk, float *dv,
                           float *dbeta, float *dgamma, float *dS_in, int B, int H, int F, int N, int D,
                           float key_scale, void *workspace, size_t workspace_bytes, gdn_stream_t stream)
{
    if (B < 0 || H < 0 || F < 0 || N < 0 || D <= 0) return GDN_ERR_INVALID_ARG;
    if (B == 0 || H == 0) return GDN_OK;
    if (D != 112) return GDN_ERR_UNSUPPORTED;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const size_t state_bytes = (size_t)B * H * D * D * sizeof(float);
    if ((S_in && !aligned(S_in, 16)) || (dS_out && !aligned(dS_out, 16)) || (dS_in && !aligned(dS_in, 16)))
        return GDN_ERR_INVALID_ARG;
    if (F == 0) {  // no frames: S_out = S_in
        if (!dS_in) return GDN_OK;
        cudaError_t e = dS_out ? cudaMemcpyAsync(dS_in, dS_out, state_bytes, cudaMemcpyDeviceToDevice, st)
                               : cudaMemsetAsync(dS_in, 0, state_bytes, st);
        return e == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
    }
    if (N == 0 || F >= kBwdMaxFrames) return GDN_ERR_UNSUPPORTED;
    if (!q || !k || !v || !beta || !gamma || !dO || !dq || !dk || !dv || !dbeta || !dgamma) return GDN_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(dO, 16) || !aligned(dq, 16) ||
        !aligned(dk, 16) || !aligned(dv, 16) || !aligned(beta, 4) || !aligned(gamma, 4) || !aligned(dbeta, 4) ||
        !aligned(dgamma, 4))
        return GDN_ERR_INVALID_ARG;
    const size_t need = bwd_workspace_bytes(B, H, F, N);
    if (need == (size_t)-1) return GDN_ERR_UNSUPPORTED;
    if (!workspace || workspace_bytes < need) return GDN_ERR_WORKSPACE;
    if (!aligned(workspace, 256)) return GDN_ERR_INVALID_ARG;
    unsigned *status = device_status_word();
    if (!status) return GDN_ERR_CUDA;
    cudaError_t e = launch_frame_bwd_tc(q, k, v, beta, gamma, S_in, dO, dS_out, dq, dk, dv, dbeta, dgamma, dS_in, B,
                                        H, F, N, default_key_scale(key_scale, D, N), workspace, status, st);
    return e == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

// Device staging of the host-buffer form: q, k, v, o (bf16), beta, gamma,
// S_in, S_out (fp32), then the workspace, each 256-byte aligned.  The frames
// are cut into pieces that are copied in, run and copied out as a pipeline, so
// the token tensors are staged piece-major: piece p holds its frames as a
// [B][F_p*N][H][D] (or [B][F_p*N][H], [B][F_p][H]) tensor of its own.
struct HostLayout {
    int pieces;
    size_t tok, beta, gamma, state, ws;
    size_t off_q, off_k, off_v, off_o, off_beta, off_gamma, off_sin, off_sout, off_ws, total;
};

// Frames [piece_f0(p), piece_f0(p + 1)) form piece p; pieces differ by at most one frame.
static int piece_f0(int p, int pieces, int F) { return (int)((long long)F * p / pieces); }

// Pieces of at least 16 frames (so that each piece's forward still fills the
// GPU), at most 8 (beyond that the per-piece launches stop paying off).
static int host_pieces(int F) { return F >= 32 ? (F / 16 < 8 ? F / 16 : 8) : 1; }

static bool host_layout(int B, int H, int F, int N, int D, HostLayout *L)
{
    if (B < 0 || H < 0 || F < 0 || N < 0 || D <= 0) return false;
    const size_t ws = gdn_frame_fwd_workspace_size(B, H, F, N, D);  // covers every piece's plan
    if (ws == (size_t)-1) return false;
    auto up = [](size_t x) { return (x + 255) / 256 * 256; };
    L->pieces = host_pieces(F);
    L->tok = (size_t)B * F * N * H * D * 2;
    L->beta = (size_t)B * F * N * H * 4;
    L->gamma = (size_t)B * F * H * 4;
    L->state = (size_t)B * H * D * D * 4;
    L->ws = ws;
    size_t o = 0;
    L->off_q = o; o = up(o + L->tok);
    L->off_k = o; o = up(o + L->tok);
    L->off_v = o; o = up(o + L->tok);
    L->off_o = o; o = up(o + L->tok);
    L->off_beta = o; o = up(o + L->beta);
    L->off_gamma = o; o = up(o + L->gamma);
    L->off_sin = o; o = up(o + L->state);
    L->off_sout = o; o = up(o + L->state);
    L->off_ws = o; o = up(o + L->ws);
    L->total = o;
    return true;
}

namespace gdn {
namespace {
// Per-device copy streams and events of the host-buffer entry, created on
// first use (never destroyed: they live as long as the process, like the
// library's other per-device state).  Calls are enqueued under a mutex, so
// concurrent callers cannot interleave their event records.
constexpr int kMaxPieces = 8;
struct HostPipe {
    bool ready = false;
    cudaStream_t in = nullptr, out = nullptr;
    cudaEvent_t start = nullptr, in_done[kMaxPieces] = {}, run_done[kMaxPieces] = {}, out_done = nullptr;
};
std::mutex g_pipe_mu;
HostPipe g_pipe[kMaxDevices];

cudaError_t host_pipe(HostPipe **out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    HostPipe &P = g_pipe[dev];
    if (!P.ready) {
        const unsigned ef = cudaEventDisableTiming;
        if ((e = cudaStreamCreateWithFlags(&P.in, cudaStreamNonBlocking)) != cudaSuccess) return e;
        if ((e = cudaStreamCreateWithFlags(&P.out, cudaStreamNonBlocking)) != cudaSuccess) return e;
        if ((e = cudaEventCreateWithFlags(&P.start, ef)) != cudaSuccess) return e;
        if ((e = cudaEventCreateWithFlags(&P.out_done, ef)) != cudaSuccess) return e;
        for (int i = 0; i < kMaxPieces; ++i) {
            if ((e = cudaEventCreateWithFlags(&P.in_done[i], ef)) != cudaSuccess) return e;
            if ((e = cudaEventCreateWithFlags(&P.run_done[i], ef)) != cudaSuccess) return e;
        }
        P.ready = true;
    }
    *out = &P;
    return cudaSuccess;
}
}  // namespace
}  // namespace gdn

size_t gdn_frame_fwd_host_buffer_size(int B, int H, int F, int N, int D)
{
    HostLayout L;
    return host_layout(B, H, F, N, D, &L) ? L.total : (size_t)-1;
}

gdn_status_t gdn_frame_fwd_host(const void *q, const void *k, const void *v, const float *beta, const float *gamma,
                                const float *S_in, float *S_out, void *o, int B, int H, int F, int N, int D,
                                float key_scale, void *device_buffer, size_t device_buffer_bytes,
                                gdn_stream_t stream)
{
    HostLayout L;
    if (!host_layout(B, H, F, N, D, &L)) return D > 0 && D != 112 ? GDN_ERR_UNSUPPORTED : GDN_ERR_INVALID_ARG;
    if (B == 0 || H == 0) return GDN_OK;
    if (!device_buffer || device_buffer_bytes < L.total) return GDN_ERR_WORKSPACE;
    if (!aligned(device_buffer, 256)) return GDN_ERR_INVALID_ARG;
    const bool has_tokens = F > 0 && N > 0;
    if (has_tokens && (!q || !k || !v || !o || !beta)) return GDN_ERR_INVALID_ARG;
    if (F > 0 && !gamma) return GDN_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    uint8_t *d = static_cast<uint8_t *>(device_buffer);
    std::lock_guard<std::mutex> lk(g_pipe_mu);
    HostPipe *P = nullptr;
    if (host_pipe(&P) != cudaSuccess) return GDN_ERR_CUDA;
    // The copy streams start after everything already on `stream`.
    if (cudaEventRecord(P->start, st) != cudaSuccess || cudaStreamWaitEvent(P->in, P->start, 0) != cudaSuccess ||
        cudaStreamWaitEvent(P->out, P->start, 0) != cudaSuccess)
        return GDN_ERR_CUDA;
    auto h2d = [&](size_t off, const void *src, size_t n) {
        return n == 0 || cudaMemcpyAsync(d + off, src, n, cudaMemcpyHostToDevice, P->in) == cudaSuccess;
    };
    auto d2h = [&](void *dst, size_t off, size_t n) {
        return n == 0 || cudaMemcpyAsync(dst, d + off, n, cudaMemcpyDeviceToHost, P->out) == cudaSuccess;
    };
    float *d_sin = S_in ? reinterpret_cast<float *>(d + L.off_sin) : nullptr;
    float *d_sout = reinterpret_cast<float *>(d + L.off_sout);
    if (S_in && !h2d(L.off_sin, S_in, L.state)) return GDN_ERR_CUDA;
    const int pieces = has_tokens ? L.pieces : 1;
    const size_t row = (size_t)N * H;  // token-head rows per frame
    for (int p = 0; p < pieces; ++p) {
        const int f0 = piece_f0(p, pieces, F), fp = piece_f0(p + 1, pieces, F) - f0;
        // piece p's region starts after the pieces before it: B * f0 frames' worth of each tensor
        const size_t tb = (size_t)B * f0 * row * D * 2, bb = (size_t)B * f0 * row * 4, gb = (size_t)B * f0 * H * 4;
        for (int b = 0; b < B; ++b) {
            const size_t hs = ((size_t)b * F + f0) * row, ds = (size_t)b * fp * row;  // first row: host, piece
            if (has_tokens &&
                (!h2d(L.off_q + tb + ds * D * 2, static_cast<const uint8_t *>(q) + hs * D * 2, (size_t)fp * row * D * 2) ||
                 !h2d(L.off_k + tb + ds * D * 2, static_cast<const uint8_t *>(k) + hs * D * 2, (size_t)fp * row * D * 2) ||
                 !h2d(L.off_v + tb + ds * D * 2, static_cast<const uint8_t *>(v) + hs * D * 2, (size_t)fp * row * D * 2) ||
                 !h2d(L.off_beta + bb + ds * 4, beta + hs, (size_t)fp * row * 4)))
                return GDN_ERR_CUDA;
            if (fp > 0 && !h2d(L.off_gamma + gb + (size_t)b * fp * H * 4, gamma + ((size_t)b * F + f0) * H,
                               (size_t)fp * H * 4))
                return GDN_ERR_CUDA;
        }
        if (cudaEventRecord(P->in_done[p], P->in) != cudaSuccess || cudaStreamWaitEvent(st, P->in_done[p], 0) != cudaSuccess)
            return GDN_ERR_CUDA;
        // piece p continues from the state piece p - 1 left in S_out (S_out may alias S_in)
        gdn_status_t s = frame_fwd_impl(d + L.off_q + tb, d + L.off_k + tb, d + L.off_v + tb,
                                        reinterpret_cast<float *>(d + L.off_beta + bb),
                                        reinterpret_cast<float *>(d + L.off_gamma + gb), p == 0 ? d_sin : d_sout,
                                        d_sout, d + L.off_o + tb, B, H, fp, N, D, key_scale, 0,
                                        L.ws ? d + L.off_ws : nullptr, L.ws, stream, nullptr);
        if (s != GDN_OK) return s;
        if (cudaEventRecord(P->run_done[p], st) != cudaSuccess || cudaStreamWaitEvent(P->out, P->run_done[p], 0) != cudaSuccess)
            return GDN_ERR_CUDA;
        for (int b = 0; b < B && has_tokens && o; ++b) {
            const size_t hs = ((size_t)b * F + f0) * row, ds = (size_t)b * fp * row;
            if (!d2h(static_cast<uint8_t *>(o) + hs * D * 2, L.off_o + tb + ds * D * 2, (size_t)fp * row * D * 2))
                return GDN_ERR_CUDA;
        }
    }
    if (S_out && !d2h(S_out, L.off_sout, L.state)) return GDN_ERR_CUDA;
    // `stream` completes only once the last copy out has landed
    if (cudaEventRecord(P->out_done, P->out) != cudaSuccess || cudaStreamWaitEvent(st, P->out_done, 0) != cudaSuccess)
        return GDN_ERR_CUDA;
    return GDN_OK;
}

size_t gdn_frame_step_workspace_size(int B, int H, int N, int D)
{
    if (B < 0 || H < 0 || N < 0 || D <= 0) return (size_t)-1;
    if (B == 0 || H == 0 || N == 0) return 0;
    if (D != 112) return (size_t)-1;
    return 0;  // the fused step keeps its cross-CTA reduction on chip
}

gdn_status_t gdn_frame_step(const void *q, const void *k, const void *v, const float *beta, const float *gamma,
                            const float *S_in, float *S_out, void *o, int B, int H, int N, int D, float key_scale,
                            void * /*workspace*/, size_t /*workspace_bytes*/, gdn_stream_t stream)
{
    if (B < 0 || H < 0 || N < 0 || D <= 0) return GDN_ERR_INVALID_ARG;
    if (B == 0 || H == 0) return GDN_OK;
    if (D != 112) return GDN_ERR_UNSUPPORTED;
    if ((S_in && !aligned(S_in, 16)) || (S_out && !aligned(S_out, 16))) return GDN_ERR_INVALID_ARG;
    if (!gamma || !aligned(gamma, 4)) return GDN_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (N == 0) {
        if (!S_out) return GDN_OK;
        return launch_decay_only(gamma, S_in, S_out, B, H, 1, D, st) == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
    }
    if (!q || !k || !v || !o || !beta) return GDN_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) || !aligned(beta, 4))
        return GDN_ERR_INVALID_ARG;
    if ((long long)B * H > (1 << 20)) return GDN_ERR_UNSUPPORTED;
    unsigned *status = device_status_word();
    if (!status) return GDN_ERR_CUDA;
    cudaError_t e = launch_frame_step_tc(q, k, v, beta, gamma, S_in, S_out, o, B, H, N,
                                         default_key_scale(key_scale, D, N), status, st);
    return e == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

size_t gdn_frame_composite_workspace_size(int B, int H, int F, int N, int D)
{
    if (B < 0 || H < 0 || F < 0 || N < 0 || D <= 0) return (size_t)-1;
    if (B == 0 || H == 0 || F == 0 || N == 0) return 0;
    if (D != 112) return (size_t)-1;
    TcPlan plan;
    if (!tc_plan(B, H, F, N, 0, &plan)) return (size_t)-1;
    return plan.ws_bytes;
}

gdn_status_t gdn_frame_composite(const void *k, const void *v, const float *beta, const float *gamma, float *C_out,
                                 float *H_out, int B, int H, int F, int N, int D, float key_scale, void *workspace,
                                 size_t workspace_bytes, gdn_stream_t stream)
{
    if (B < 0 || H < 0 || F < 0 || N < 0 || D <= 0) return GDN_ERR_INVALID_ARG;
    if (B == 0 || H == 0) return GDN_OK;
    if (D != 112) return GDN_ERR_UNSUPPORTED;
    if ((C_out && !aligned(C_out, 16)) || (H_out && !aligned(H_out, 16))) return GDN_ERR_INVALID_ARG;
    if (F > 0 && (!gamma || !aligned(gamma, 4))) return GDN_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (F == 0 || N == 0) {
        if ((long long)B * H > (1 << 20)) return GDN_ERR_UNSUPPORTED;
        composite_decay_kernel<<<B * H, 256, 0, st>>>(gamma, C_out, H_out, H, F, D);
        return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
    }
    if (!k || !v || !beta) return GDN_ERR_INVALID_ARG;
    if (!aligned(k, 16) || !aligned(v, 16) || !aligned(beta, 4)) return GDN_ERR_INVALID_ARG;
    TcPlan plan;
    if (!tc_plan(B, H, F, N, 0, &plan)) return GDN_ERR_UNSUPPORTED;
    if (!workspace || workspace_bytes < plan.ws_bytes) return GDN_ERR_WORKSPACE;
    if (!aligned(workspace, 16)) return GDN_ERR_INVALID_ARG;
    unsigned *status = device_status_word();
    if (!status) return GDN_ERR_CUDA;
    cudaError_t e = launch_frame_composite_tc(k, v, beta, gamma, C_out, H_out, plan,
                                              default_key_scale(key_scale, D, N), workspace, status, st);
    return e == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

gdn_status_t gdn_frame_fwd_resume(const void *q, const float *gamma, const float *S_in, float *S_out, void *o,
                                  int B, int H, int F, int N, int D, void *workspace, size_t workspace_bytes,
                                  gdn_stream_t stream)
{
    if (B < 0 || H < 0 || F < 0 || N < 0 || D <= 0) return GDN_ERR_INVALID_ARG;
    if (B == 0 || H == 0) return GDN_OK;
    if (D != 112) return GDN_ERR_UNSUPPORTED;
    if ((S_in && !aligned(S_in, 16)) || (S_out && !aligned(S_out, 16))) return GDN_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (F == 0 || N == 0) {  // no statistics to resume from: the forward's degenerate rules
        if (F > 0 && (!gamma || !aligned(gamma, 4))) return GDN_ERR_INVALID_ARG;
        if (!S_out) return GDN_OK;
        return launch_decay_only(gamma, S_in, S_out, B, H, F, D, st) == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
    }
    if (!q || !o || !gamma) return GDN_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(o, 16) || !aligned(gamma, 4)) return GDN_ERR_INVALID_ARG;
    TcPlan plan;
    if (!tc_plan(B, H, F, N, 0, &plan)) return GDN_ERR_UNSUPPORTED;
    if (!workspace || workspace_bytes < plan.ws_bytes) return GDN_ERR_WORKSPACE;
    if (!aligned(workspace, 16)) return GDN_ERR_INVALID_ARG;
    unsigned *status = device_status_word();
    if (!status) return GDN_ERR_CUDA;
    return launch_fwd_resume_tc(q, gamma, S_in, S_out, o, plan, workspace, status, st) == cudaSuccess ? GDN_OK
                                                                                                    : GDN_ERR_CUDA;
}

gdn_status_t gdn_state_compose(const float *S, const float *C, const float *Hc, float *S_out, int BH, int D,
                               gdn_stream_t stream)
{
    if (BH < 0 || D <= 0) return GDN_ERR_INVALID_ARG;
    if (BH == 0) return GDN_OK;
    if (D != 112) return GDN_ERR_UNSUPPORTED;
    if (BH > (1 << 20)) return GDN_ERR_UNSUPPORTED;
    if (!C || !Hc || !S_out) return GDN_ERR_INVALID_ARG;
    if (!aligned(C, 16) || !aligned(Hc, 16) || !aligned(S_out, 16) || (S && !aligned(S, 16)))
        return GDN_ERR_INVALID_ARG;
    unsigned *status = device_status_word();
    if (!status) return GDN_ERR_CUDA;
    cudaError_t e = launch_state_compose_tc(S, C, Hc, S_out, BH, status, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

// ------------------------------------------------------------ block projections
static bool block_sizes_ok(int B, int H, int F, int N, int D)
{
    return B >= 0 && H >= 0 && F >= 0 && N >= 0 && D > 0;
}

gdn_status_t gdn_block_in_proj(const void *x, const void *W_in, void *q, void *k, void *v, float *beta,
                               float *gamma, int B, int H, int F, int N, int D, gdn_stream_t stream)
{
    if (!block_sizes_ok(B, H, F, N, D)) return GDN_ERR_INVALID_ARG;
    if (B == 0 || H == 0 || F == 0) return GDN_OK;
    if (D != 112) return GDN_ERR_UNSUPPORTED;
    if ((long long)B * F * N > (1LL << 30) || H > 512) return GDN_ERR_UNSUPPORTED;
    if (!x || !W_in || !gamma || (N > 0 && (!q || !k || !v || !beta))) return GDN_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(W_in, 16) || !aligned(gamma, 4) ||
        (N > 0 && (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(beta, 4))))
        return GDN_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (N == 0) {  // no tokens: gamma of the frame mean over no tokens is undefined; report it
        return GDN_ERR_UNSUPPORTED;
    }
    unsigned *status = device_status_word();
    if (!status) return GDN_ERR_CUDA;
    return launch_in_proj_tc(x, W_in, q, k, v, beta, gamma, B, H, F, N, status, st) == cudaSuccess ? GDN_OK
                                                                                             : GDN_ERR_CUDA;
}

gdn_status_t gdn_block_out_proj(const void *o, const void *W_out, void *y, int B, int H, int F, int N, int D,
                                gdn_stream_t stream)
{
    if (!block_sizes_ok(B, H, F, N, D)) return GDN_ERR_INVALID_ARG;
    if ((long long)B * F * N == 0 || H == 0) return GDN_OK;
    if (D != 112) return GDN_ERR_UNSUPPORTED;
    if ((long long)B * F * N > (1LL << 30) || H > 512) return GDN_ERR_UNSUPPORTED;
    if (!o || !W_out || !y) return GDN_ERR_INVALID_ARG;
    if (!aligned(o, 16) || !aligned(W_out, 16) || !aligned(y, 16)) return GDN_ERR_INVALID_ARG;
    unsigned *status = device_status_word();
    if (!status) return GDN_ERR_CUDA;
    const int HD = H * D;
    return launch_linear_tc(o, W_out, y, B * F * N, HD, HD, status, static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? GDN_OK
               : GDN_ERR_CUDA;
}

// Block workspace: q, k, v, o (bf16 [B][F*N][H][D]), beta (fp32), gamma (fp32
// [B][F][H]), then the forward's workspace; each 256-byte aligned.
struct BlockLayout {
    size_t tok, beta, gamma, fwd, off_q, off_k, off_v, off_o, off_beta, off_gamma, off_fwd, total;
};

static bool block_layout(int B, int H, int F, int N, int D, BlockLayout *L)
{
    if (!block_sizes_ok(B, H, F, N, D)) return false;
    const size_t fwd = gdn_frame_fwd_workspace_size(B, H, F, N, D);
    if (fwd == (size_t)-1) return false;
    auto up = [](size_t x) { return (x + 255) / 256 * 256; };
    L->tok = (size_t)B * F * N * H * D * 2;
    L->beta = (size_t)B * F * N * H * 4;
    L->gamma = (size_t)B * F * H * 4;
    L->fwd = fwd;
    size_t o = 0;
    L->off_q = o; o = up(o + L->tok);
    L->off_k = o; o = up(o + L->tok);
    L->off_v = o; o = up(o + L->tok);
    L->off_o = o; o = up(o + L->tok);
    L->off_beta = o; o = up(o + L->beta);
    L->off_gamma = o; o = up(o + L->gamma);
    L->off_fwd = o; o = up(o + L->fwd);
    L->total = o;
    return true;
}

size_t gdn_block_fwd_workspace_size(int B, int H, int F, int N, int D)
{
    BlockLayout L;
    if (!block_layout(B, H, F, N, D, &L)) return (size_t)-1;
    if (B == 0 || H == 0 || F == 0 || N == 0) return 0;
    if (D != 112) return (size_t)-1;
    return L.total;
}

gdn_status_t gdn_block_fwd(const void *x, const void *W_in, const void *W_out, const float *S_in, float *S_out,
                           void *y, int B, int H, int F, int N, int D, float key_scale, void *workspace,
                           size_t workspace_bytes, gdn_stream_t stream)
{
    if (!block_sizes_ok(B, H, F, N, D)) return GDN_ERR_INVALID_ARG;
    if (B == 0 || H == 0) return GDN_OK;
    if (D != 112) return GDN_ERR_UNSUPPORTED;
    BlockLayout L;
    if (!block_layout(B, H, F, N, D, &L)) return GDN_ERR_UNSUPPORTED;
    if (F == 0)  // no frames: the state passes through (S_out = S_in, or zero)
        return gdn_frame_fwd(nullptr, nullptr, nullptr, nullptr, nullptr, S_in, S_out, nullptr, B, H, 0, N, D,
                             key_scale, nullptr, 0, stream);
    if (N == 0) return GDN_ERR_UNSUPPORTED;  // the frame-mean decay logit needs tokens
    if (!x || !W_in || !W_out || !y) return GDN_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(W_in, 16) || !aligned(W_out, 16) || !aligned(y, 16) ||
        (S_in && !aligned(S_in, 16)) || (S_out && !aligned(S_out, 16)))
        return GDN_ERR_INVALID_ARG;
    if (!workspace || workspace_bytes < L.total) return GDN_ERR_WORKSPACE;
    if (!aligned(workspace, 256)) return GDN_ERR_INVALID_ARG;
    uint8_t *w = static_cast<uint8_t *>(workspace);
    void *q = w + L.off_q, *k = w + L.off_k, *v = w + L.off_v, *o = w + L.off_o;
    float *beta = reinterpret_cast<float *>(w + L.off_beta), *gamma = reinterpret_cast<float *>(w + L.off_gamma);
    gdn_status_t s = gdn_block_in_proj(x, W_in, q, k, v, beta, gamma, B, H, F, N, D, stream);
    if (s != GDN_OK) return s;
    s = gdn_frame_fwd(q, k, v, beta, gamma, S_in, S_out, o, B, H, F, N, D, key_scale, w + L.off_fwd, L.fwd, stream);
    if (s != GDN_OK) return s;
    return gdn_block_out_proj(o, W_out, y, B, H, F, N, D, stream);
}

gdn_status_t gdn_frame_fwd_f32(const float *q, const float *k, const float *v, const float *beta,
                               const float *gamma, const float *S_in, float *S_out, float *o, int B, int H, int F,
                               int N, int D, float key_scale, gdn_stream_t stream)
{
    if (B < 0 || H < 0 || F < 0 || N < 0 || D <= 0) return GDN_ERR_INVALID_ARG;
    if (B == 0 || H == 0) return GDN_OK;
    if (D > 128) return GDN_ERR_UNSUPPORTED;
    if ((S_in && !aligned(S_in, 16)) || (S_out && !aligned(S_out, 16))) return GDN_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (F == 0 || N == 0) {
        if (F > 0 && (!gamma || !aligned(gamma, 4))) return GDN_ERR_INVALID_ARG;
        if (!S_out) return GDN_OK;
        return launch_decay_only(gamma, S_in, S_out, B, H, F, D, st) == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
    }
    if (!q || !k || !v || !o || !beta || !gamma) return GDN_ERR_INVALID_ARG;
    if (!aligned(q, 4) || !aligned(k, 4) || !aligned(v, 4) || !aligned(o, 4) || !aligned(beta, 4) ||
        !aligned(gamma, 4))
        return GDN_ERR_INVALID_ARG;
    cudaError_t e = launch_frame_fwd_f32(q, k, v, beta, gamma, S_in, S_out, o, B, H, F, N, D,
                                         default_key_scale(key_scale, D, N), st);
    return e == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

gdn_status_t gdn_device_status(gdn_stream_t stream)
{
    unsigned *p = device_status_word();
    if (!p) return GDN_ERR_CUDA;
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return GDN_ERR_CUDA;
    unsigned word = 0;
    if (cudaMemcpyFromSymbol(&word, g_status_word, sizeof(word)) != cudaSuccess) return GDN_ERR_CUDA;
    if (word) {
        const unsigned zero = 0;
        if (cudaMemcpyToSymbol(g_status_word, &zero, sizeof(zero)) != cudaSuccess) return GDN_ERR_CUDA;
        return GDN_ERR_TIMEOUT;
    }
    return GDN_OK;
}

}  // extern "C"
