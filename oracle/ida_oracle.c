/*
 * ida_oracle.c -- plain fp64 CPU oracle for the Interdomain Attention (IDA)
 * token-mixer forward pass: prefill and one-token recurrent decode.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the CPU
 * baseline leg of the benchmark may load or call this library.  It shares no
 * code, header, table or helper with the CUDA library; the only thing both
 * sides have in common is the seeded input generator and the published state
 * layout (an interface, restated here in code of its own).
 *
 * Sources: "Interdomain Attention: Beyond Token-Level Key-Value Memory"
 * (arXiv 2605.24330), as given on three pages:
 *   [paper]  the translated paper text: Sec. 3.1 (Eqs. 3-4) and the Fig. 1
 *            caption (state U: M x R, Gamma: M x d, eta: M x 1);
 *   [de]     the German technical summary, sections "Theoretische Herleitung"
 *            (query-conditioned readout, matrix form F_q U^T Gamma / F_q U^T eta)
 *            and "Skalierbare Implementierung" (feature map, recurrent core,
 *            normalisation, denominator-free readout);
 *   [nl]     the Dutch technical summary, "Schaalbare Implementatie" (same).
 *
 * What is computed, per (batch b, head h), for t = 0 .. N-1:
 *   a1  s_t[c]  = sum_{j<W} w[c][j] * x_{t-W+1+j}[c], x_{<0} = 0 (or the
 *                 carried tail), for x = q and x = k separately.   [de] feature map
 *   a2  xi(x)_t = SiLU(s_t) / (sum_c SiLU(s_t)[c]^2 + EPS_FEAT).  [de] feature map
 *       With ORC_FEAT_L2 (the "SiLU/l_2" wording of the Chinese summary's
 *       introduction): xi(x)_t = SiLU(s_t) / (||SiLU(s_t)||_2 + EPS_FEAT).
 *   a3  kt_t    = xi(k)_t / sqrt(mean_c xi(k)_t^2 + EPS_RMS) * w_k + b_k,
 *       vt_t    = v_t     / sqrt(mean_c v_t^2     + EPS_RMS) * w_v + b_v.
 *                                                            [de] normalisation
 *   a4  X_t = lambda o X_{t-1} + B o [kt_t ; vt_t],  X_{-1} = 0, complex,
 *       U_t = X_t[:, :R], Gamma_t = X_t[:, R:].               [de] recurrent core
 *   a5  a_t[m] = sum_c xi(q)_t[c] U_t[m][c].
 *   a6  o_t = Re sum_m a_t[m] Gamma_t[m][:]          [de] denominator-free readout
 *   a7  eta variant: eta_t = lambda o eta_{t-1} + B, den_t = Re sum_m a_t[m] eta_t[m],
 *       o_t /= den_t.                   [de] "Theoretische Herleitung", readout ratio
 *
 * Readings where the pages are silent (every one of them is a choice the
 * pages do not fix; the tests pin the arithmetic, not these choices):
 *   - ||.||^2 in the feature map is the squared Euclidean norm;
 *   - EPS_FEAT = 1e-6 is added to that squared norm, EPS_RMS = 1e-6 sits
 *     inside the RMS square root;
 *   - the conv follows the cross-correlation convention (tap W-1 multiplies
 *     the current token), no bias, v is not convolved, q is not RMS-normed;
 *   - lambda and B are the already-discretised complex diagonal S4D
 *     parameters; no conjugation anywhere, the real part is taken last and
 *     there is no factor 2;
 *   - the eta division has no epsilon.
 *
 * State layout (per (b,h), all float64 here, fp32 on the device):
 *   [2M][R+d] planar complex state: rows 0..M-1 are Re, rows M..2M-1 are Im,
 *   columns 0..R-1 are U, columns R..R+d-1 are Gamma;
 *   then eta[2M] (Re then Im);
 *   then the raw q tail [W-1][R] and the raw k tail [W-1][R], oldest first.
 */
#include <complex.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

#define EPS_FEAT 1e-6
#define EPS_RMS 1e-6

enum { ORC_F32 = 0, ORC_BF16 = 1 };
enum { ORC_READOUT_ETA = 1, ORC_FEAT_L2 = 2 };

/* ---- element access -------------------------------------------------- */

static double bf16_bits_to_double(uint16_t bits)
{
    uint32_t u = ((uint32_t)bits) << 16; /* bf16 is the top half of an fp32 */
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static double load_elem(const void *base, int dtype, size_t i)
{
    if (dtype == ORC_BF16)
        return bf16_bits_to_double(((const uint16_t *)base)[i]);
    return (double)((const float *)base)[i];
}

size_t orc_state_doubles(int d, int R, int M, int W)
{
    return (size_t)2 * M * (R + d) + (size_t)2 * M + (size_t)2 * (W - 1) * R;
}

/* ---- a1: causal depthwise conv --------------------------------------- */

/* x: [N][C]; w: [C][W]; tail: [W-1][C] oldest first, or NULL for zeros. */
void orc_causal_conv(const double *x, int N, int C, const double *w, int W,
                     const double *tail, double *s)
{
    for (int t = 0; t < N; ++t)
        for (int c = 0; c < C; ++c) {
            double acc = 0.0;
            for (int j = 0; j < W; ++j) {
                int p = t - (W - 1) + j; /* source position */
                double xv;
                if (p >= 0)
                    xv = x[(size_t)p * C + c];
                else if (tail)
                    xv = tail[(size_t)(W - 1 + p) * C + c];
                else
                    xv = 0.0;
                acc += w[(size_t)c * W + j] * xv;
            }
            s[(size_t)t * C + c] = acc;
        }
}

/* ---- a2: xi = SiLU(s) / (||SiLU(s)||^2 + eps) -------------------------- */

double orc_silu(double x) { return x / (1.0 + exp(-x)); }

void orc_feature_map(const double *s, int N, int C, double *xi)
{
    for (int t = 0; t < N; ++t) {
        const double *row = s + (size_t)t * C;
        double sq = 0.0;
        for (int c = 0; c < C; ++c) {
            double f = orc_silu(row[c]);
            sq += f * f;
        }
        for (int c = 0; c < C; ++c)
            xi[(size_t)t * C + c] = orc_silu(row[c]) / (sq + EPS_FEAT);
    }
}

/* The l_2 reading: SiLU(s) over its Euclidean norm (plus EPS_FEAT). */
void orc_feature_map_l2(const double *s, int N, int C, double *xi)
{
    for (int t = 0; t < N; ++t) {
        const double *row = s + (size_t)t * C;
        double sq = 0.0;
        for (int c = 0; c < C; ++c) {
            double f = orc_silu(row[c]);
            sq += f * f;
        }
        for (int c = 0; c < C; ++c)
            xi[(size_t)t * C + c] = orc_silu(row[c]) / (sqrt(sq) + EPS_FEAT);
    }
}

/* ---- a3: RMSNorm with per-channel weight and bias --------------------- */

void orc_rmsnorm_affine(const double *x, int N, int C, const double *w,
                        const double *b, double *y)
{
    for (int t = 0; t < N; ++t) {
        const double *row = x + (size_t)t * C;
        double ms = 0.0;
        for (int c = 0; c < C; ++c)
            ms += row[c] * row[c];
        ms /= C;
        double r = 1.0 / sqrt(ms + EPS_RMS);
        for (int c = 0; c < C; ++c)
            y[(size_t)t * C + c] = row[c] * r * w[c] + b[c];
    }
}

/*
 * Prologue of one (b,h) unit: q, k, v as float64 rows, conv weights wq/wk
 * [R][W], norm weight/bias [R+d] (key half first).  Outputs xq = xi(q) [N][R],
 * kt [N][R], vt [N][d].  Tails (raw inputs before position 0) may be NULL.
 */
static void unit_features(const double *q, const double *k, const double *v,
                          int N, int R, int d, int W,
                          const double *wq, const double *wk,
                          const double *norm_w, const double *bias,
                          const double *tail_q, const double *tail_k, int feat_l2,
                          double *xq, double *kt, double *vt)
{
    size_t nr = (size_t)N * R;
    double *s = malloc(nr * sizeof(double));
    double *xk = malloc(nr * sizeof(double));
    void (*fmap)(const double *, int, int, double *) = feat_l2 ? orc_feature_map_l2 : orc_feature_map;
    orc_causal_conv(q, N, R, wq, W, tail_q, s);
    fmap(s, N, R, xq);
    orc_causal_conv(k, N, R, wk, W, tail_k, s);
    fmap(s, N, R, xk);
    orc_rmsnorm_affine(xk, N, R, norm_w, bias, kt);
    orc_rmsnorm_affine(v, N, d, norm_w + R, bias + R, vt);
    free(s);
    free(xk);
}

void orc_unit_features(const double *q, const double *k, const double *v,
                       int N, int R, int d, int W,
                       const double *wq, const double *wk,
                       const double *norm_w, const double *bias,
                       const double *tail_q, const double *tail_k,
                       double *xq, double *kt, double *vt)
{
    unit_features(q, k, v, N, R, d, W, wq, wk, norm_w, bias, tail_q, tail_k, 0, xq, kt, vt);
}

/* ---- a4-a7: the S4D recurrence and the query-conditioned readout ------ */

/*
 * Step-by-step recurrence for one unit.  X: complex [M][R+d] (in/out),
 * eta: complex [M] (in/out).  out: [N][d]; den: [N] or NULL (receives
 * den_t whichever readout is used).
 */
static void scan_readout(const double *xq, const double *kt, const double *vt,
                         int N, int R, int d, int M,
                         const double complex *lam, const double complex *Bv,
                         int eta_readout, double complex *X,
                         double complex *eta, double *out, double *den)
{
    int RD = R + d;
    double complex *a = malloc((size_t)M * sizeof(double complex));
    for (int t = 0; t < N; ++t) {
        const double *qr = xq + (size_t)t * R;
        const double *kr = kt + (size_t)t * R;
        const double *vr = vt + (size_t)t * d;
        /* a4: X_t = lambda X_{t-1} + B z_t, z_t = [kt_t ; vt_t] */
        for (int m = 0; m < M; ++m) {
            double complex *row = X + (size_t)m * RD;
            for (int c = 0; c < R; ++c)
                row[c] = lam[m] * row[c] + Bv[m] * kr[c];
            for (int j = 0; j < d; ++j)
                row[R + j] = lam[m] * row[R + j] + Bv[m] * vr[j];
            eta[m] = lam[m] * eta[m] + Bv[m];
        }
        /* a5: a_t[m] = xi(q_t) . U_t[m] */
        for (int m = 0; m < M; ++m) {
            double complex acc = 0.0;
            for (int c = 0; c < R; ++c)
                acc += qr[c] * X[(size_t)m * RD + c];
            a[m] = acc;
        }
        /* a6: o_t = Re sum_m a_t[m] Gamma_t[m] ; a7: den_t */
        double dn = 0.0;
        for (int m = 0; m < M; ++m)
            dn += creal(a[m] * eta[m]);
        for (int j = 0; j < d; ++j) {
            double complex acc = 0.0;
            for (int m = 0; m < M; ++m)
                acc += a[m] * X[(size_t)m * RD + R + j];
            double o = creal(acc);
            out[(size_t)t * d + j] = eta_readout ? o / dn : o;
        }
        if (den)
            den[t] = dn;
    }
    free(a);
}

/* planar [2M][R+d] + eta[2M] <-> complex arrays */
static void state_unpack(const double *st, int M, int RD, double complex *X,
                         double complex *eta)
{
    for (int m = 0; m < M; ++m) {
        for (int c = 0; c < RD; ++c)
            X[(size_t)m * RD + c] = st[(size_t)m * RD + c] +
                                    I * st[(size_t)(M + m) * RD + c];
        eta[m] = st[(size_t)2 * M * RD + m] + I * st[(size_t)2 * M * RD + M + m];
    }
}

static void state_pack(const double complex *X, const double complex *eta,
                       int M, int RD, double *st)
{
    for (int m = 0; m < M; ++m) {
        for (int c = 0; c < RD; ++c) {
            st[(size_t)m * RD + c] = creal(X[(size_t)m * RD + c]);
            st[(size_t)(M + m) * RD + c] = cimag(X[(size_t)m * RD + c]);
        }
        st[(size_t)2 * M * RD + m] = creal(eta[m]);
        st[(size_t)2 * M * RD + M + m] = cimag(eta[m]);
    }
}

/*
 * Full forward on float64 inputs of ONE unit (already gathered rows).
 * Used by the Python tests for the algebraic pins.  state: nullable in/out
 * [2M][R+d] + eta[2M] (+ tails are ignored here; tails are passed apart).
 */
void orc_unit_forward(const double *q, const double *k, const double *v,
                      int N, int R, int d, int M, int W,
                      const double *wq, const double *wk,
                      const double *norm_w, const double *bias,
                      const double *lam_ri, const double *B_ri, int flags,
                      double *state, const double *tail_q,
                      const double *tail_k, double *out, double *den)
{
    int RD = R + d;
    double *xq = malloc((size_t)N * R * sizeof(double) + 1);
    double *kt = malloc((size_t)N * R * sizeof(double) + 1);
    double *vt = malloc((size_t)N * d * sizeof(double) + 1);
    double complex *X = calloc((size_t)M * RD, sizeof(double complex));
    double complex *eta = calloc((size_t)M, sizeof(double complex));
    double complex *lam = malloc((size_t)M * sizeof(double complex));
    double complex *Bv = malloc((size_t)M * sizeof(double complex));
    for (int m = 0; m < M; ++m) {
        lam[m] = lam_ri[2 * m] + I * lam_ri[2 * m + 1];
        Bv[m] = B_ri[2 * m] + I * B_ri[2 * m + 1];
    }
    if (state)
        state_unpack(state, M, RD, X, eta);
    unit_features(q, k, v, N, R, d, W, wq, wk, norm_w, bias, tail_q, tail_k,
                  flags & ORC_FEAT_L2, xq, kt, vt);
    scan_readout(xq, kt, vt, N, R, d, M, lam, Bv, flags & ORC_READOUT_ETA, X,
                 eta, out, den);
    if (state)
        state_pack(X, eta, M, RD, state);
    free(xq); free(kt); free(vt); free(X); free(eta); free(lam); free(Bv);
}

/*
 * Chunked re-association of the same recurrence for one unit, chunk length C
 * (the last chunk may be shorter).  For a chunk starting after state X_p:
 *   X_i  = lambda^{i+1} X_p + B sum_{j<=i} lambda^{i-j} z_j,
 *   a_i  = lambda^{i+1} (xi(q_i).U_p) + B sum_{j<=i} lambda^{i-j} (xi(q_i).kt_j),
 *   o_i  = Re sum_m a_i (lambda^{i+1} Gamma_p + B sum_{j<=i} lambda^{i-j} vt_j),
 *   X_end = lambda^{C} X_p + B sum_j lambda^{C-1-j} z_j.
 * Written term by term (no factoring of the decay) so that it can be checked
 * against the step recurrence: both must agree to fp64 rounding for every C.
 */
void orc_unit_forward_chunked(const double *xq, const double *kt,
                              const double *vt, int N, int R, int d, int M,
                              const double *lam_ri, const double *B_ri,
                              int flags, int C, double *state, double *out,
                              double *den)
{
    int RD = R + d;
    double complex *X = calloc((size_t)M * RD, sizeof(double complex));
    double complex *eta = calloc((size_t)M, sizeof(double complex));
    double complex *lam = malloc((size_t)M * sizeof(double complex));
    double complex *Bv = malloc((size_t)M * sizeof(double complex));
    double complex *pw = malloc((size_t)M * (C + 1) * sizeof(double complex));
    double complex *G = malloc((size_t)M * sizeof(double complex));
    double complex *acc_o = malloc(((size_t)d + 1) * sizeof(double complex));
    for (int m = 0; m < M; ++m) {
        lam[m] = lam_ri[2 * m] + I * lam_ri[2 * m + 1];
        Bv[m] = B_ri[2 * m] + I * B_ri[2 * m + 1];
        pw[(size_t)m * (C + 1)] = 1.0;
        for (int e = 1; e <= C; ++e)
            pw[(size_t)m * (C + 1) + e] = pw[(size_t)m * (C + 1) + e - 1] * lam[m];
    }
    if (state)
        state_unpack(state, M, RD, X, eta);
    for (int t0 = 0; t0 < N; t0 += C) {
        int L = (N - t0 < C) ? (N - t0) : C;
        for (int i = 0; i < L; ++i) {
            int t = t0 + i;
            const double *qr = xq + (size_t)t * R;
            double dn = 0.0;
            for (int j = 0; j < d; ++j)
                acc_o[j] = 0.0;
            for (int m = 0; m < M; ++m) {
                const double complex *pm = pw + (size_t)m * (C + 1);
                /* inter: lambda^{i+1} xi(q).U_p ; intra: B sum lambda^{i-j} G */
                double complex inter = 0.0, intra = 0.0;
                for (int c = 0; c < R; ++c)
                    inter += qr[c] * X[(size_t)m * RD + c];
                for (int j = 0; j <= i; ++j) {
                    const double *kr = kt + (size_t)(t0 + j) * R;
                    double g = 0.0;
                    for (int c = 0; c < R; ++c)
                        g += qr[c] * kr[c];
                    intra += pm[i - j] * g;
                }
                double complex a = pm[i + 1] * inter + Bv[m] * intra;
                /* eta_i = lambda^{i+1} eta_p + B sum_{j<=i} lambda^{i-j} */
                double complex es = 0.0;
                for (int j = 0; j <= i; ++j)
                    es += pm[i - j];
                dn += creal(a * (pm[i + 1] * eta[m] + Bv[m] * es));
                for (int jj = 0; jj < d; ++jj) {
                    double complex g = pm[i + 1] * X[(size_t)m * RD + R + jj];
                    double complex vs = 0.0;
                    for (int j = 0; j <= i; ++j)
                        vs += pm[i - j] * vt[(size_t)(t0 + j) * d + jj];
                    acc_o[jj] += a * (g + Bv[m] * vs);
                }
            }
            for (int jj = 0; jj < d; ++jj) {
                double o = creal(acc_o[jj]);
                out[(size_t)t * d + jj] = (flags & ORC_READOUT_ETA) ? o / dn : o;
            }
            if (den)
                den[t] = dn;
        }
        /* chunk-boundary state: X_end = lambda^L X_p + B sum_j lambda^{L-1-j} z_j */
        for (int m = 0; m < M; ++m) {
            const double complex *pm = pw + (size_t)m * (C + 1);
            for (int c = 0; c < RD; ++c) {
                double complex acc = 0.0;
                for (int j = 0; j < L; ++j) {
                    double z = (c < R) ? kt[(size_t)(t0 + j) * R + c]
                                       : vt[(size_t)(t0 + j) * d + (c - R)];
                    acc += pm[L - 1 - j] * z;
                }
                X[(size_t)m * RD + c] = pm[L] * X[(size_t)m * RD + c] + Bv[m] * acc;
            }
            double complex es = 0.0;
            for (int j = 0; j < L; ++j)
                es += pm[L - 1 - j];
            G[m] = pm[L] * eta[m] + Bv[m] * es;
        }
        for (int m = 0; m < M; ++m)
            eta[m] = G[m];
    }
    if (state)
        state_pack(X, eta, M, RD, state);
    free(X); free(eta); free(lam); free(Bv); free(pw); free(G); free(acc_o);
}

/* ---- batched entry points on raw input bytes ------------------------- */

/*
 * Prefill over [B,N,H,*] inputs (q,k: [B,N,H,R], v: [B,N,H,d]) in fp32 or
 * bf16, parameters in fp32 as the device library takes them:
 * conv_w [2,H,R,W] (0 = q, 1 = k), norm_w/bias [H,R+d], lambda/Bvec [H,M,2].
 * state_in: nullable [B,H][orc_state_doubles], the state before position 0
 * (planar X, eta, and the raw conv tails, which stand for the inputs of
 * positions -(W-1) .. -1); NULL is the zero state.
 * out: [B,N,H,d] float64.  final_state: nullable [B,H][orc_state_doubles].
 * den: nullable [B,N,H].  units: nullable list of unit ids (b*H+h) to
 * compute (others untouched); n_units ignored when units is NULL.
 * nthreads <= 0 uses the OpenMP default.  Returns 0.
 */
int orc_forward_from(const void *q, const void *k, const void *v, int dtype,
                     const float *conv_w, const float *norm_w, const float *bias,
                     const float *lambda, const float *Bvec, const double *state_in,
                     double *out, double *final_state, double *den, int B, int H,
                     int N, int d, int R, int M, int W, int flags,
                     const int *units, int n_units, int nthreads)
{
    int total = units ? n_units : B * H;
    size_t SD = orc_state_doubles(d, R, M, W);
#ifdef _OPENMP
    if (nthreads > 0)
        omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
#endif
    for (int u = 0; u < total; ++u) {
        int id = units ? units[u] : u;
        int b = id / H, h = id % H;
        int RD = R + d;
        double *qr = malloc(((size_t)N * R + 1) * sizeof(double));
        double *kr = malloc(((size_t)N * R + 1) * sizeof(double));
        double *vr = malloc(((size_t)N * d + 1) * sizeof(double));
        double *wq = malloc((size_t)R * W * sizeof(double));
        double *wk = malloc((size_t)R * W * sizeof(double));
        double *nw = malloc((size_t)RD * sizeof(double));
        double *bs = malloc((size_t)RD * sizeof(double));
        double *lr = malloc((size_t)2 * M * sizeof(double));
        double *br = malloc((size_t)2 * M * sizeof(double));
        double *st = calloc(SD, sizeof(double));
        const double *sin = state_in ? state_in + (size_t)id * SD : NULL;
        const double *tin_q = sin ? sin + (size_t)2 * M * (RD + 1) : NULL;
        const double *tin_k = sin ? tin_q + (size_t)(W - 1) * R : NULL;
        if (sin)
            memcpy(st, sin, (size_t)2 * M * (RD + 1) * sizeof(double));
        double *o = malloc(((size_t)N * d + 1) * sizeof(double));
        double *dn = malloc(((size_t)N + 1) * sizeof(double));
        for (int t = 0; t < N; ++t) {
            size_t rowqk = (((size_t)b * N + t) * H + h) * R;
            size_t rowv = (((size_t)b * N + t) * H + h) * d;
            for (int c = 0; c < R; ++c) {
                qr[(size_t)t * R + c] = load_elem(q, dtype, rowqk + c);
                kr[(size_t)t * R + c] = load_elem(k, dtype, rowqk + c);
            }
            for (int j = 0; j < d; ++j)
                vr[(size_t)t * d + j] = load_elem(v, dtype, rowv + j);
        }
        for (int c = 0; c < R; ++c)
            for (int j = 0; j < W; ++j) {
                wq[(size_t)c * W + j] = conv_w[(((size_t)0 * H + h) * R + c) * W + j];
                wk[(size_t)c * W + j] = conv_w[(((size_t)1 * H + h) * R + c) * W + j];
            }
        for (int c = 0; c < RD; ++c) {
            nw[c] = norm_w[(size_t)h * RD + c];
            bs[c] = bias[(size_t)h * RD + c];
        }
        for (int m = 0; m < 2 * M; ++m) {
            lr[m] = lambda[(size_t)h * 2 * M + m];
            br[m] = Bvec[(size_t)h * 2 * M + m];
        }
        orc_unit_forward(qr, kr, vr, N, R, d, M, W, wq, wk, nw, bs, lr, br,
                         flags, st, tin_q, tin_k, o, dn);
        for (int t = 0; t < N; ++t) {
            for (int j = 0; j < d; ++j)
                out[(((size_t)b * N + t) * H + h) * d + j] = o[(size_t)t * d + j];
            if (den)
                den[((size_t)b * N + t) * H + h] = dn[t];
        }
        if (final_state) {
            double *fs = final_state + (size_t)id * SD;
            memcpy(fs, st, (size_t)2 * M * (RD + 1) * sizeof(double));
            /* conv tails: the raw inputs of the last W-1 positions, oldest first
             * (positions before 0 from the starting tails, or zero) */
            double *tq = fs + (size_t)2 * M * (RD + 1);
            double *tk = tq + (size_t)(W - 1) * R;
            for (int r = 0; r < W - 1; ++r) {
                int p = N - (W - 1) + r;
                for (int c = 0; c < R; ++c) {
                    double xq0 = 0.0, xk0 = 0.0;
                    if (p >= 0) {
                        xq0 = qr[(size_t)p * R + c];
                        xk0 = kr[(size_t)p * R + c];
                    } else if (sin) {
                        xq0 = tin_q[(size_t)(p + W - 1) * R + c];
                        xk0 = tin_k[(size_t)(p + W - 1) * R + c];
                    }
                    tq[(size_t)r * R + c] = xq0;
                    tk[(size_t)r * R + c] = xk0;
                }
            }
        }
        free(qr); free(kr); free(vr); free(wq); free(wk); free(nw); free(bs);
        free(lr); free(br); free(st); free(o); free(dn);
    }
    return 0;
}

/* Prefill from the zero state. */
int orc_forward(const void *q, const void *k, const void *v, int dtype,
                const float *conv_w, const float *norm_w, const float *bias,
                const float *lambda, const float *Bvec, double *out,
                double *final_state, double *den, int B, int H, int N, int d,
                int R, int M, int W, int flags, const int *units, int n_units,
                int nthreads)
{
    return orc_forward_from(q, k, v, dtype, conv_w, norm_w, bias, lambda, Bvec,
                            NULL, out, final_state, den, B, H, N, d, R, M, W,
                            flags, units, n_units, nthreads);
}

/*
 * One recurrent decode step over [B,H,*] inputs (one token per unit), state
 * in/out [B,H][orc_state_doubles] float64, out [B,H,d] float64, den nullable
 * [B,H].  The conv uses the carried raw tails, which are then shifted.
 */
int orc_decode_step(const void *q, const void *k, const void *v, int dtype,
                    const float *conv_w, const float *norm_w,
                    const float *bias, const float *lambda, const float *Bvec,
                    double *state, double *out, double *den, int B, int H,
                    int d, int R, int M, int W, int flags, const int *units,
                    int n_units, int nthreads)
{
    int total = units ? n_units : B * H;
    size_t SD = orc_state_doubles(d, R, M, W);
    if (R > 256 || d > 256 || M > 128 || W > 4 || W < 1)
        return -1; /* the fixed-size rows below hold the supported maxima */
#ifdef _OPENMP
    if (nthreads > 0)
        omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 4)
#endif
    for (int u = 0; u < total; ++u) {
        int id = units ? units[u] : u;
        int h = id % H;
        int RD = R + d;
        double *st = state + (size_t)id * SD;
        double qr[256], kr[256], vr[256], o[256];
        double wq[256 * 4], wk[256 * 4], nw[512], bs[512], lr[256], br[256];
        double dn;
        for (int c = 0; c < R; ++c) {
            qr[c] = load_elem(q, dtype, (size_t)id * R + c);
            kr[c] = load_elem(k, dtype, (size_t)id * R + c);
        }
        for (int j = 0; j < d; ++j)
            vr[j] = load_elem(v, dtype, (size_t)id * d + j);
        for (int c = 0; c < R; ++c)
            for (int j = 0; j < W; ++j) {
                wq[c * W + j] = conv_w[(((size_t)0 * H + h) * R + c) * W + j];
                wk[c * W + j] = conv_w[(((size_t)1 * H + h) * R + c) * W + j];
            }
        for (int c = 0; c < RD; ++c) {
            nw[c] = norm_w[(size_t)h * RD + c];
            bs[c] = bias[(size_t)h * RD + c];
        }
        for (int m = 0; m < 2 * M; ++m) {
            lr[m] = lambda[(size_t)h * 2 * M + m];
            br[m] = Bvec[(size_t)h * 2 * M + m];
        }
        double *tq = st + (size_t)2 * M * (RD + 1);
        double *tk = tq + (size_t)(W - 1) * R;
        orc_unit_forward(qr, kr, vr, 1, R, d, M, W, wq, wk, nw, bs, lr, br,
                         flags, st, W > 1 ? tq : NULL, W > 1 ? tk : NULL, o, &dn);
        /* shift the tails: drop the oldest row, append this token */
        for (int r = 0; r + 1 < W - 1; ++r)
            for (int c = 0; c < R; ++c) {
                tq[(size_t)r * R + c] = tq[(size_t)(r + 1) * R + c];
                tk[(size_t)r * R + c] = tk[(size_t)(r + 1) * R + c];
            }
        if (W > 1)
            for (int c = 0; c < R; ++c) {
                tq[(size_t)(W - 2) * R + c] = qr[c];
                tk[(size_t)(W - 2) * R + c] = kr[c];
            }
        for (int j = 0; j < d; ++j)
            out[(size_t)id * d + j] = o[j];
        if (den)
            den[id] = dn;
    }
    return 0;
}

int orc_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
