/*
 * Frame-wise Gated DeltaNet — plain fp64 CPU oracle.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may load, call or link
 * this file: it exists so that tests, the smoke check and the benchmark's CPU
 * baseline can compare the CUDA library against an obviously-correct restatement
 * of the method.  It shares no code, header, constant or helper with the CUDA
 * sources.
 *
 * Source of the method: the paper-summary page "SANA-WM: Efficient Minute-Scale
 * World Modeling with Hybrid Linear Diffusion Transformer", section 方法步骤详情
 * (method details), module 2 "Memory-Efficient Long-Context": the GDN scans the
 * video one latent frame at a time; the state S_t (D x D) follows
 *     S_t = S_{t-1} (gamma_t I - K^_t beta_t K^_t^T) + V_t beta_t K^_t^T,
 * the frame's output is O_t = S_t Q^_t, and the keys carry a 1/sqrt(D S) scale.
 * Same page, section 前置知识 "Gated DeltaNet": the update written as
 * S_t = S_{t-1} M_t + U_t with decay gate gamma_t.  Same page, section
 * 技术新颖性 (novelty): the key scale makes ||M_t||_2 <= gamma_t <= 1, and context
 * parallelism composes a transition composite C_p and an input composite H_p
 * by a prefix scan that reproduces the single-device result exactly.
 *
 * Readings taken where the page is silent or garbled (each is listed in the
 * design notes):
 *   - k^_n = k_n / ||k_n||_2 * c_k with c_k = key_scale, default 1/sqrt(D*N)
 *     ("DS" read as head dim times tokens per frame);
 *   - q^_n = q_n / ||q_n||_2, no further factor;
 *   - ||x||_2 = sqrt(sum x^2 + 1e-12);
 *   - the frame output reads the post-update state S_f;
 *   - M_f is the sum form gamma_f I - sum_n beta_n k^_n k^_n^T exactly as
 *     printed (not the token-ordered product);
 *   - gamma is per (batch, frame, head), beta per (batch, token, head).
 *
 * Layouts (row-major):
 *   q, k, v : [B][F*N][H][D]  (fp32 values; bf16 inputs are passed exactly)
 *   beta    : [B][F*N][H]
 *   gamma   : [B][F][H]
 *   S_in    : [B][H][D][D] or NULL for zeros; S[i][j] with i the value index
 *             (row) and j the key index (column)
 *   o       : [B][F*N][H][D]  (fp64)
 *   S_out   : [B][H][D][D]    (fp64)
 *
 * Parallel execution: the B*H chains are independent problems, run one per
 * OpenMP thread; inside a chain everything is the plain sequential loop.
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_NORM_EPS 1e-12

static double oracle_key_scale(double key_scale, int D, int N)
{
    return key_scale > 0.0 ? key_scale : 1.0 / sqrt((double)D * (double)N);
}

/* Index helpers for the [B][F*N][H][D] token layout. */
static size_t tok_index(int b, int f, int n, int h, int d, int F, int N, int H, int D)
{
    return ((((size_t)b * F * N + (size_t)f * N + n) * H + h) * D) + d;
}
static size_t beta_index(int b, int f, int n, int h, int F, int N, int H)
{
    return ((size_t)b * F * N + (size_t)f * N + n) * H + h;
}

/* x^ = x / ||x||_2 * scale for one token-head vector. */
static void normalise(const float *x, int D, double scale, double *out)
{
    double ss = 0.0;
    for (int d = 0; d < D; ++d) ss += (double)x[d] * (double)x[d];
    double inv = scale / sqrt(ss + ORACLE_NORM_EPS);
    for (int d = 0; d < D; ++d) out[d] = (double)x[d] * inv;
}

/*
 * Per-frame transition of one chain: A_f = sum_n beta_n k^_n k^_n^T and
 * U_f = sum_n beta_n v_n k^_n^T, then M_f = gamma_f I - A_f.
 * (summary page, 方法步骤详情 module 2: M_t = gamma_t I - K^_t beta_t K^_t^T,
 *  U_t = V_t beta_t K^_t^T.)  M and U are D x D, row-major.
 */
static void frame_transition(const float *k, const float *v, const float *beta,
                             const float *gamma, int b, int h, int f,
                             int H, int F, int N, int D, double c,
                             double *M, double *U, double *khat)
{
    memset(M, 0, sizeof(double) * D * D);
    memset(U, 0, sizeof(double) * D * D);
    for (int n = 0; n < N; ++n) {
        normalise(k + tok_index(b, f, n, h, 0, F, N, H, D), D, c, khat);
        const float *vn = v + tok_index(b, f, n, h, 0, F, N, H, D);
        double bn = beta[beta_index(b, f, n, h, F, N, H)];
        for (int i = 0; i < D; ++i)
            for (int j = 0; j < D; ++j) {
                M[i * D + j] -= bn * khat[i] * khat[j];      /* -A_f */
                U[i * D + j] += bn * (double)vn[i] * khat[j];
            }
    }
    double g = gamma[((size_t)b * F + f) * H + h];
    for (int i = 0; i < D; ++i) M[i * D + i] += g;
}

/* C = A * B for D x D row-major matrices. */
static void matmul(const double *A, const double *B, double *C, int D)
{
    for (int i = 0; i < D; ++i)
        for (int j = 0; j < D; ++j) {
            double s = 0.0;
            for (int l = 0; l < D; ++l) s += A[i * D + l] * B[l * D + j];
            C[i * D + j] = s;
        }
}

/* o_{f,n} = S_f q^_n for every token of frame f (module 2: O_t = S_t Q^_t). */
static void frame_output(const float *q, const double *S, int b, int h, int f,
                         int H, int F, int N, int D, double *o, double *qhat)
{
    for (int n = 0; n < N; ++n) {
        size_t base = tok_index(b, f, n, h, 0, F, N, H, D);
        normalise(q + base, D, 1.0, qhat);
        for (int i = 0; i < D; ++i) {
            double s = 0.0;
            for (int j = 0; j < D; ++j) s += S[i * D + j] * qhat[j];
            o[base + i] = s;
        }
    }
}

static void load_state(const float *S_in, int b, int h, int H, int D, double *S)
{
    size_t base = ((size_t)b * H + h) * D * D;
    for (int e = 0; e < D * D; ++e) S[e] = S_in ? (double)S_in[base + e] : 0.0;
}

static void store_state(double *S_out, const double *S, int b, int h, int H, int D)
{
    if (!S_out) return;
    memcpy(S_out + ((size_t)b * H + h) * D * D, S, sizeof(double) * D * D);
}

/*
 * Formulation 1 (the printed recurrence): for each frame build M_f and U_f
 * explicitly, S_f = S_{f-1} M_f + U_f, then o = S_f q^.
 */
void oracle_gdn_frame_fwd(const float *q, const float *k, const float *v,
                          const float *beta, const float *gamma, const float *S_in,
                          int B, int H, int F, int N, int D, double key_scale,
                          double *o, double *S_out)
{
    double c = oracle_key_scale(key_scale, D, N);
#pragma omp parallel for schedule(dynamic, 1)
    for (int bh = 0; bh < B * H; ++bh) {
        int b = bh / H, h = bh % H;
        double *S = malloc(sizeof(double) * D * D);
        double *Sn = malloc(sizeof(double) * D * D);
        double *M = malloc(sizeof(double) * D * D);
        double *U = malloc(sizeof(double) * D * D);
        double *vec = malloc(sizeof(double) * D);
        load_state(S_in, b, h, H, D, S);
        for (int f = 0; f < F; ++f) {
            frame_transition(k, v, beta, gamma, b, h, f, H, F, N, D, c, M, U, vec);
            matmul(S, M, Sn, D);
            for (int e = 0; e < D * D; ++e) S[e] = Sn[e] + U[e];
            if (o) frame_output(q, S, b, h, f, H, F, N, D, o, vec);
        }
        store_state(S_out, S, b, h, H, D);
        free(S); free(Sn); free(M); free(U); free(vec);
    }
}

/*
 * Formulation 2 (token accumulation, an independent loop structure used to
 * check formulation 1): because M_f is a sum over the frame's tokens,
 *   S_f = gamma_f S_{f-1} + sum_n beta_n (v_n - S_{f-1} k^_n) k^_n^T,
 * i.e. every token of the frame writes a delta-rule correction against the
 * frame-start state.
 */
void oracle_gdn_frame_fwd_tokacc(const float *q, const float *k, const float *v,
                                 const float *beta, const float *gamma,
                                 const float *S_in, int B, int H, int F, int N,
                                 int D, double key_scale, double *o, double *S_out)
{
    double c = oracle_key_scale(key_scale, D, N);
#pragma omp parallel for schedule(dynamic, 1)
    for (int bh = 0; bh < B * H; ++bh) {
        int b = bh / H, h = bh % H;
        double *S = malloc(sizeof(double) * D * D);
        double *P = malloc(sizeof(double) * D * D);
        double *kh = malloc(sizeof(double) * D);
        double *err = malloc(sizeof(double) * D);
        load_state(S_in, b, h, H, D, S);
        for (int f = 0; f < F; ++f) {
            memcpy(P, S, sizeof(double) * D * D);           /* frame-start state */
            double g = gamma[((size_t)b * F + f) * H + h];
            for (int e = 0; e < D * D; ++e) S[e] = g * P[e];
            for (int n = 0; n < N; ++n) {
                normalise(k + tok_index(b, f, n, h, 0, F, N, H, D), D, c, kh);
                const float *vn = v + tok_index(b, f, n, h, 0, F, N, H, D);
                double bn = beta[beta_index(b, f, n, h, F, N, H)];
                for (int i = 0; i < D; ++i) {               /* v_n - S_{f-1} k^_n */
                    double s = 0.0;
                    for (int j = 0; j < D; ++j) s += P[i * D + j] * kh[j];
                    err[i] = (double)vn[i] - s;
                }
                for (int i = 0; i < D; ++i)
                    for (int j = 0; j < D; ++j) S[i * D + j] += bn * err[i] * kh[j];
            }
            if (o) frame_output(q, S, b, h, f, H, F, N, D, o, kh);
        }
        store_state(S_out, S, b, h, H, D);
        free(S); free(P); free(kh); free(err);
    }
}

/*
 * The per-frame pair (M_f, U_f) for every (b, f, h), written to
 * M_out, U_out : [B][H][F][D][D].  Used by the tests to check the printed norm
 * bound ||M_t||_2 <= gamma_t and to build composites.
 */
void oracle_gdn_frame_transitions(const float *k, const float *v, const float *beta,
                                  const float *gamma, int B, int H, int F, int N,
                                  int D, double key_scale, double *M_out, double *U_out)
{
    double c = oracle_key_scale(key_scale, D, N);
#pragma omp parallel for schedule(dynamic, 1)
    for (int bhf = 0; bhf < B * H * F; ++bhf) {
        int b = bhf / (H * F), h = (bhf / F) % H, f = bhf % F;
        double *vec = malloc(sizeof(double) * D);
        size_t off = (size_t)bhf * D * D;
        frame_transition(k, v, beta, gamma, b, h, f, H, F, N, D, c,
                         M_out + off, U_out + off, vec);
        free(vec);
    }
}

/*
 * Composite of a run of frames (technical-novelty section: transition composite
 * C_p and input composite H_p).  For frames f0..f1-1 of one chain,
 *   C = M_{f0} M_{f0+1} ... M_{f1-1},   H = state reached from S = 0,
 * so that S_{f1-1} = S_{f0-1} C + H.  M, U are [nF][D][D] for the run.
 */
void oracle_gdn_composite(const double *M, const double *U, int nF, int D,
                          double *C, double *Hc)
{
    double *T = malloc(sizeof(double) * D * D);
    for (int e = 0; e < D * D; ++e) { C[e] = 0.0; Hc[e] = 0.0; }
    for (int i = 0; i < D; ++i) C[i * D + i] = 1.0;
    for (int f = 0; f < nF; ++f) {
        const double *Mf = M + (size_t)f * D * D, *Uf = U + (size_t)f * D * D;
        matmul(C, Mf, T, D);
        memcpy(C, T, sizeof(double) * D * D);
        matmul(Hc, Mf, T, D);
        for (int e = 0; e < D * D; ++e) Hc[e] = T[e] + Uf[e];
    }
    free(T);
}

/*
 * Composition of two adjacent composites (earlier run 1, later run 2):
 *   (C1, H1) then (C2, H2)  ->  (C1 C2, H1 C2 + H2).
 */
void oracle_gdn_compose(const double *C1, const double *H1, const double *C2,
                        const double *H2, int D, double *C, double *Hc)
{
    double *T = malloc(sizeof(double) * D * D);
    matmul(C1, C2, C, D);
    matmul(H1, C2, T, D);
    for (int e = 0; e < D * D; ++e) Hc[e] = T[e] + H2[e];
    free(T);
}

/*
 * Token-ordered ("product") reading of the frame transition.
 *
 * The page writes the frame's transition as gamma_t I - K^_t beta_t K^_t^T with
 * beta_t between K^_t and K^_t^T.  Read with beta_t = diag(beta) this is the sum
 * form above.  The token-wise Gated DeltaNet that the frame-wise one
 * generalises (novelty section) instead applies the frame's tokens one after
 * another, S <- S (I - beta_n k^_n k^_n^T) + beta_n v_n k^_n^T.  This reading
 * keeps the frame's decay where the printed formula puts it:
 *     P_f = (I - beta_1 k^_1 k^_1^T) (I - beta_2 k^_2 k^_2^T) ... (I - beta_N k^_N k^_N^T),
 *     M_f = gamma_f I - (I - P_f),
 *     U_f = the state the frame's tokens reach from zero, in token order.
 * Both are built here by the plain definition, one token at a time: the
 * product P is multiplied on the right by the token's factor, and W (which
 * ends as U_f) takes the token's delta-rule write.
 */
static void frame_transition_product(const float *k, const float *v, const float *beta,
                                     const float *gamma, int b, int h, int f,
                                     int H, int F, int N, int D, double c,
                                     double *M, double *U)
{
    double *P = calloc((size_t)D * D, sizeof(double));         /* running product */
    double *kh = malloc(sizeof(double) * D);
    double *Pk = malloc(sizeof(double) * D);                    /* P k^_n */
    double *Wk = malloc(sizeof(double) * D);                    /* W k^_n */
    for (int i = 0; i < D; ++i) P[i * D + i] = 1.0;
    memset(U, 0, sizeof(double) * D * D);                       /* W starts at zero */
    for (int n = 0; n < N; ++n) {
        normalise(k + tok_index(b, f, n, h, 0, F, N, H, D), D, c, kh);
        const float *vn = v + tok_index(b, f, n, h, 0, F, N, H, D);
        double bn = beta[beta_index(b, f, n, h, F, N, H)];
        for (int i = 0; i < D; ++i) {
            double sp = 0.0, sw = 0.0;
            for (int j = 0; j < D; ++j) {
                sp += P[i * D + j] * kh[j];
                sw += U[i * D + j] * kh[j];
            }
            Pk[i] = sp;
            Wk[i] = sw;
        }
        /* P <- P (I - b k k^T);   W <- W (I - b k k^T) + b v k^T */
        for (int i = 0; i < D; ++i)
            for (int j = 0; j < D; ++j) {
                P[i * D + j] -= bn * Pk[i] * kh[j];
                U[i * D + j] += bn * ((double)vn[i] - Wk[i]) * kh[j];
            }
    }
    /* M = gamma I - (I - P) = P - (1 - gamma) I */
    double g = gamma[((size_t)b * F + f) * H + h];
    for (int e = 0; e < D * D; ++e) M[e] = P[e];
    for (int i = 0; i < D; ++i) M[i * D + i] -= 1.0 - g;
    free(P); free(kh); free(Pk); free(Wk);
}

/* (M_f, U_f) of the product reading for every (b, f, h): [B][H][F][D][D]. */
void oracle_gdn_frame_transitions_product(const float *k, const float *v, const float *beta,
                                          const float *gamma, int B, int H, int F, int N,
                                          int D, double key_scale,
                                          double *M_out, double *U_out)
{
    double c = oracle_key_scale(key_scale, D, N);
#pragma omp parallel for schedule(dynamic, 1)
    for (int bhf = 0; bhf < B * H * F; ++bhf) {
        int b = bhf / (H * F), h = (bhf / F) % H, f = bhf % F;
        size_t off = (size_t)bhf * D * D;
        frame_transition_product(k, v, beta, gamma, b, h, f, H, F, N, D, c,
                                 M_out + off, U_out + off);
    }
}

/*
 * Forward pass of the product reading: S_f = S_{f-1} M_f + U_f with the
 * token-ordered (M_f, U_f) above, o = S_f q^ (output after the update, as in
 * the sum form).
 */
void oracle_gdn_frame_fwd_product(const float *q, const float *k, const float *v,
                                  const float *beta, const float *gamma, const float *S_in,
                                  int B, int H, int F, int N, int D, double key_scale,
                                  double *o, double *S_out)
{
    double c = oracle_key_scale(key_scale, D, N);
#pragma omp parallel for schedule(dynamic, 1)
    for (int bh = 0; bh < B * H; ++bh) {
        int b = bh / H, h = bh % H;
        double *S = malloc(sizeof(double) * D * D);
        double *Sn = malloc(sizeof(double) * D * D);
        double *M = malloc(sizeof(double) * D * D);
        double *U = malloc(sizeof(double) * D * D);
        double *vec = malloc(sizeof(double) * D);
        load_state(S_in, b, h, H, D, S);
        for (int f = 0; f < F; ++f) {
            frame_transition_product(k, v, beta, gamma, b, h, f, H, F, N, D, c, M, U);
            matmul(S, M, Sn, D);
            for (int e = 0; e < D * D; ++e) S[e] = Sn[e] + U[e];
            if (o) frame_output(q, S, b, h, f, H, F, N, D, o, vec);
        }
        store_state(S_out, S, b, h, H, D);
        free(S); free(Sn); free(M); free(U); free(vec);
    }
}

/*
 * Backward pass of the sum reading (training, the CSDN article's §六: the layer
 * is trained end to end; the gradients follow from the forward recurrence by
 * the chain rule).  With upstream gradients dO = dL/do and dS_out = dL/dS_out
 * (either may be NULL: zero), per chain:
 *   G_f = dL/dS_f:  G_{F-1} = dS_out + E_{F-1},  G_{f-1} = G_f M_f^T + E_{f-1},
 *                   E_f = sum_{n in f} do_n q^_n^T;   dS_in = G_0 M_0^T
 *   dL/dM_f = S_{f-1}^T G_f,  dL/dU_f = G_f,  dgamma_f = trace(S_{f-1}^T G_f),
 *   dA_f = -S_{f-1}^T G_f,
 *   dk^_n = beta_n (dA_f + dA_f^T) k^_n + beta_n G_f^T v_n,   dv_n = beta_n G_f k^_n,
 *   dbeta_n = k^_n^T dA_f k^_n + v_n^T G_f k^_n,   dq^_n = S_f^T do_n,
 *   k^ = c k / r:  dk = (c / r) (dk^ - k (k . dk^) / r^2);   q^ = q / rho likewise (c = 1).
 * r and rho include the same epsilon as the forward.  Outputs are fp64, in the
 * input layouts: dq, dk, dv [B][F*N][H][D], dbeta [B][F*N][H], dgamma [B][F][H],
 * dS_in [B][H][D][D].
 */
void oracle_gdn_frame_bwd(const float *q, const float *k, const float *v,
                          const float *beta, const float *gamma, const float *S_in,
                          const float *dO, const float *dS_out,
                          int B, int H, int F, int N, int D, double key_scale,
                          double *dq, double *dk, double *dv, double *dbeta,
                          double *dgamma, double *dS_in)
{
    double c = oracle_key_scale(key_scale, D, N);
#pragma omp parallel for schedule(dynamic, 1)
    for (int bh = 0; bh < B * H; ++bh) {
        int b = bh / H, h = bh % H;
        size_t DD = (size_t)D * D;
        double *S = malloc(sizeof(double) * DD * (F + 1));   /* S_{-1} .. S_{F-1} */
        double *M = malloc(sizeof(double) * DD * (F > 0 ? F : 1));
        double *U = malloc(sizeof(double) * DD);
        double *G = malloc(sizeof(double) * DD);
        double *Gn = malloc(sizeof(double) * DD);
        double *dA = malloc(sizeof(double) * DD);
        double *kh = malloc(sizeof(double) * D);
        double *qh = malloc(sizeof(double) * D);
        double *t1 = malloc(sizeof(double) * D);
        load_state(S_in, b, h, H, D, S);
        for (int f = 0; f < F; ++f) {   /* forward, keeping every state */
            frame_transition(k, v, beta, gamma, b, h, f, H, F, N, D, c, M + f * DD, U, kh);
            matmul(S + f * DD, M + f * DD, S + (f + 1) * DD, D);
            for (size_t e = 0; e < DD; ++e) S[(f + 1) * DD + e] += U[e];
        }
        /* G_{F-1} starts from dS_out */
        for (size_t e = 0; e < DD; ++e)
            G[e] = dS_out ? (double)dS_out[((size_t)b * H + h) * DD + e] : 0.0;
        for (int f = F - 1; f >= 0; --f) {
            const double *Sp = S + f * DD, *Sf = S + (f + 1) * DD;   /* S_{f-1}, S_f */
            /* G_f += E_f (this frame's outputs read S_f) */
            for (int n = 0; n < N; ++n) {
                size_t base = tok_index(b, f, n, h, 0, F, N, H, D);
                normalise(q + base, D, 1.0, qh);
                for (int i = 0; i < D; ++i) {
                    double di = dO ? (double)dO[base + i] : 0.0;
                    for (int j = 0; j < D; ++j) G[i * D + j] += di * qh[j];
                }
            }
            /* dA_f = -S_{f-1}^T G_f;  dgamma_f = trace(S_{f-1}^T G_f) */
            double tr = 0.0;
            for (int i = 0; i < D; ++i)
                for (int j = 0; j < D; ++j) {
                    double sacc = 0.0;
                    for (int l = 0; l < D; ++l) sacc += Sp[l * D + i] * G[l * D + j];
                    dA[i * D + j] = -sacc;
                    if (i == j) tr += sacc;
                }
            dgamma[((size_t)b * F + f) * H + h] = tr;
            /* token gradients of frame f */
            for (int n = 0; n < N; ++n) {
                size_t base = tok_index(b, f, n, h, 0, F, N, H, D);
                size_t bi = beta_index(b, f, n, h, F, N, H);
                const float *kn = k + base, *vn = v + base, *qn = q + base;
                double bn = beta[bi];
                normalise(kn, D, c, kh);
                /* dk^ = beta ((dA + dA^T) k^ + G^T v);  dbeta = k^ dA k^ + v G k^;  dv = beta G k^ */
                double db = 0.0;
                for (int i = 0; i < D; ++i) {
                    double a = 0.0, gv = 0.0, gk = 0.0, ak = 0.0;
                    for (int j = 0; j < D; ++j) {
                        a += (dA[i * D + j] + dA[j * D + i]) * kh[j];
                        gv += G[j * D + i] * (double)vn[j];
                        gk += G[i * D + j] * kh[j];
                        ak += dA[i * D + j] * kh[j];
                    }
                    t1[i] = bn * (a + gv);
                    dv[base + i] = bn * gk;
                    db += kh[i] * ak + (double)vn[i] * gk;
                }
                dbeta[bi] = db;
                /* through k^ = c k / r */
                double ss = 0.0, kd = 0.0;
                for (int i = 0; i < D; ++i) {
                    ss += (double)kn[i] * kn[i];
                    kd += (double)kn[i] * t1[i];
                }
                double r2 = ss + ORACLE_NORM_EPS, r = sqrt(r2);
                for (int i = 0; i < D; ++i) dk[base + i] = c / r * (t1[i] - (double)kn[i] * kd / r2);
                /* dq^ = S_f^T do;  through q^ = q / rho */
                double qs = 0.0, qd = 0.0;
                for (int j = 0; j < D; ++j) {
                    double sacc = 0.0;
                    for (int i = 0; i < D; ++i) sacc += Sf[i * D + j] * (dO ? (double)dO[base + i] : 0.0);
                    t1[j] = sacc;
                    qs += (double)qn[j] * qn[j];
                    qd += (double)qn[j] * sacc;
                }
                double p2 = qs + ORACLE_NORM_EPS, rho = sqrt(p2);
                for (int j = 0; j < D; ++j) dq[base + j] = (t1[j] - (double)qn[j] * qd / p2) / rho;
            }
            /* G_{f-1} = G_f M_f^T */
            const double *Mf = M + f * DD;
            for (int i = 0; i < D; ++i)
                for (int j = 0; j < D; ++j) {
                    double sacc = 0.0;
                    for (int l = 0; l < D; ++l) sacc += G[i * D + l] * Mf[j * D + l];
                    Gn[i * D + j] = sacc;
                }
            memcpy(G, Gn, sizeof(double) * DD);
        }
        if (dS_in) memcpy(dS_in + ((size_t)b * H + h) * DD, G, sizeof(double) * DD);
        free(S); free(M); free(U); free(G); free(Gn); free(dA); free(kh); free(qh); free(t1);
    }
}

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
