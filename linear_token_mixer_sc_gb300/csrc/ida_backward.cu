// ida_backward.cu -- gradients of the mixer's prefill (the backward pass).
//
// The forward pass is the token mixer of "Interdomain Attention: Beyond
// Token-Level Key-Value Memory" (German technical summary, "Skalierbare
// Implementierung"; the ratio readout of its "Theoretische Herleitung"): per
// (b,h) unit, from the zero state,
//   xi(q_t), kt_t = RMSNorm(xi(k_t)) w_k + b_k, vt_t = RMSNorm(v_t) w_v + b_v,
//   X_t = lambda X_{t-1} + B z_t  (z_t = [kt_t ; vt_t]),  eta_t = lambda eta_{t-1} + B,
//   a_t[m] = xi(q_t) . U_t[m],  num_t = Re sum_m a_t[m] Gamma_t[m],
//   o_t = num_t  (or num_t / den_t, den_t = Re sum_m a_t[m] eta_t[m], for the eta readout).
// The pages train models built from this layer ("Hauptbeiträge": a scaling study from
// 125M to 1.3B parameters), which needs these gradients.
//
// Complex adjoints: for a real loss and a complex z = x + i y, zbar = dL/dx + i dL/dy.
// Then w = c z gives zbar = conj(c) wbar, and w = z1 z2 gives z1bar = conj(z2) wbar.
// With g_t = dL/do_t, working backwards in time:
//   eta readout:  gn_t = g_t / den_t,  gd_t = -(g_t . o_t) / den_t  (else gn_t = g_t, gd_t = 0)
//   abar_t[m]   = sum_j conj(Gamma_t[m,j]) gn_t[j] + conj(eta_t[m]) gd_t
//   direct adjoint of X_t:  D^U[m,c] = abar_t[m] xi(q_t)[c],  D^Gamma[m,j] = conj(a_t[m]) gn_t[j],
//                           D^eta[m] = conj(a_t[m]) gd_t
//   Y_t = D_t + conj(lambda) Y_{t+1}                         (the adjoint state, reversed in time)
//   dxi(q_t)[c] = sum_m Re(conj(abar_t[m]) U_t[m,c]),  dz_t[c] = sum_m Re(conj(B_m) Y_t[m,c])
//   lambda_bar[m] += sum_c conj(X_{t-1}[m,c]) Y_t[m,c]  (eta included),
//   B_bar[m]      += sum_c z_t[c] Y_t[m,c] + Y^eta_t[m].
// Then the position-local parts: RMSNorm, the feature map and the causal conv.
//
// Kernels (all deterministic: every sum runs in a fixed order):
//   bwd_features   one warp per position: xi(q), kt, vt into the workspace;
//   bwd_scan       one CTA per unit, one thread per state column: the forward recurrence,
//                  storing the state before every chunk of BC positions; then, chunk by
//                  chunk from the end, the chunk's states recomputed from its checkpoint
//                  and the adjoint recurrence walked backwards through them; writes
//                  dxi(q), dkt, dvt per position and per-unit lambda / B gradients;
//   bwd_local      one CTA per (unit, tile of positions): RMSNorm, feature-map and conv
//                  backward, dq, dk, dv, and per-tile partial parameter gradients;
//   bwd_reduce     sums the partials over batch rows and tiles into the parameter gradients.
// Arithmetic type T: double for fp32 inputs, float for bf16 inputs.
#include <cstdint>
#include <string>

#include "ida_common.cuh"

namespace ida {

constexpr int BWD_CHUNK = 64;     // positions between checkpoints
constexpr int BWD_TILE = 32;      // positions per bwd_local CTA
constexpr int BWD_THREADS = 512;  // bwd_scan threads (one per state column; R + d <= 512)
constexpr int BWD_WARPS = BWD_THREADS / 32;

struct BackwardArgs {
    const void *q, *k, *v, *dout;
    const float *conv_w, *norm_w, *bias, *lambda, *Bvec;
    void *dq, *dk, *dv;
    float *dconv_w, *dnorm_w, *dbias, *dlambda, *dBvec;
    int B, H, N, d, R, M, W, dtype, flags;
    unsigned *err;
};

// Workspace layout (elements of T), per unit unless noted.
struct BwdLayout {
    size_t feat;   // [N][2R + d]: xi(q), kt, vt
    size_t gfeat;  // [N][2R + d]: dxi(q), dkt, dvt
    size_t sd;     // state elements: 2M (R + d) planar X, then 2M eta
    size_t ckpt;   // [nck][sd]
    size_t xbuf;   // [BWD_CHUNK + 1][sd]
    size_t adj;    // [3][sd]: Y, lambda-bar terms, B-bar terms (per element, summed over t)
    size_t pscan;  // [4M]: lambda-bar (re, im), B-bar (re, im)
    size_t per_unit;
    size_t plocal_each;  // per (unit, tile): [2][R][W] conv, [R + d] norm weight, [R + d] bias
    int nck, ntile;
    size_t total;  // elements of T
    static BwdLayout of(int B, int H, int N, int d, int R, int M, int W) {
        BwdLayout L;
        const size_t units = (size_t)B * H, F = 2 * (size_t)R + d;
        L.nck = (N + BWD_CHUNK - 1) / BWD_CHUNK;
        L.ntile = (N + BWD_TILE - 1) / BWD_TILE;
        L.sd = 2 * (size_t)M * (R + d) + 2 * (size_t)M;
        L.feat = 0;
        L.gfeat = L.feat + (size_t)N * F;
        L.ckpt = L.gfeat + (size_t)N * F;
        L.xbuf = L.ckpt + (size_t)L.nck * L.sd;
        L.adj = L.xbuf + (size_t)(BWD_CHUNK + 1) * L.sd;
        L.pscan = L.adj + 3 * L.sd;
        L.per_unit = (L.pscan + 4 * (size_t)M + 1) & ~(size_t)1;
        L.plocal_each = 2 * (size_t)R * W + 2 * ((size_t)R + d);
        L.total = units * L.per_unit + units * L.ntile * L.plocal_each;
        return L;
    }
    __host__ __device__ size_t plocal_base(size_t units) const { return units * per_unit; }
};

template <typename T>
__device__ __forceinline__ T sigm(T x) { return T(1) / (T(1) + exp(-x)); }

// d SiLU / ds at s
template <typename T>
__device__ __forceinline__ T silu_grad(T s) {
    const T g = sigm(s);
    return g * (T(1) + s * (T(1) - g));
}

// Causal conv of channel c at position t (taps w[c][0..W-1], tap W-1 on position t).
template <typename T>
__device__ __forceinline__ T conv_at(const void *x, int dtype, size_t base, size_t stride, const float *w, int W,
                                     int t, int c) {
    T s = 0;
    for (int j = 0; j < W; ++j) {
        const int p = t - (W - 1) + j;
        if (p >= 0) s = fma((T)w[(size_t)c * W + j], (T)load_in(x, dtype, base + (size_t)p * stride + c), s);
    }
    return s;
}

template <typename T>
__device__ __forceinline__ T warp_sum_t(T x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

// ---- bwd_features: xi(q), kt, vt per position ------------------------------------------

template <typename T>
__global__ void __launch_bounds__(256) bwd_features_kernel(BackwardArgs a, T *ws, BwdLayout L) {
    const int R = a.R, d = a.d, H = a.H, N = a.N, W = a.W;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int tiles = (N + 7) / 8;
    const int unit = blockIdx.x / tiles, t = (blockIdx.x % tiles) * 8 + warp;
    if (t >= N) return;
    const int b = unit / H, h = unit % H;
    const size_t sqk = (size_t)H * R, sv = (size_t)H * d;
    const size_t base_qk = ((size_t)b * N * H + h) * R, base_v = ((size_t)b * N * H + h) * d;
    const float *nw = a.norm_w + (size_t)h * (R + d), *bs = a.bias + (size_t)h * (R + d);
    T *row = ws + (size_t)unit * L.per_unit + L.feat + (size_t)t * (2 * R + d);
    const bool l2 = (a.flags & IDA_FEAT_L2) != 0;
    for (int which = 0; which < 2; ++which) {
        const void *x = which == 0 ? a.q : a.k;
        const float *cw = a.conv_w + ((size_t)which * H + h) * R * W;
        T ss = 0;
        for (int c = lane; c < R; c += 32) {
            const T f = silu(conv_at<T>(x, a.dtype, base_qk, sqk, cw, W, t, c));
            ss = fma(f, f, ss);
        }
        T n = warp_sum_t(ss);
        if (l2) n = sqrt(n);
        const T inv = T(1) / (n + (T)IDA_EPS_FEAT);
        if (which == 0) {
            for (int c = lane; c < R; c += 32) row[c] = silu(conv_at<T>(x, a.dtype, base_qk, sqk, cw, W, t, c)) * inv;
        } else {
            T ms = 0;
            for (int c = lane; c < R; c += 32) {
                const T xi = silu(conv_at<T>(x, a.dtype, base_qk, sqk, cw, W, t, c)) * inv;
                ms = fma(xi, xi, ms);
            }
            const T r = T(1) / sqrt(warp_sum_t(ms) / R + (T)IDA_EPS_RMS);
            for (int c = lane; c < R; c += 32) {
                const T xi = silu(conv_at<T>(x, a.dtype, base_qk, sqk, cw, W, t, c)) * inv;
                row[R + c] = fma(xi * r, (T)nw[c], (T)bs[c]);
            }
        }
    }
    T ms = 0;
    for (int j = lane; j < d; j += 32) {
        const T x = (T)load_in(a.v, a.dtype, base_v + (size_t)t * sv + j);
        ms = fma(x, x, ms);
    }
    const T r = T(1) / sqrt(warp_sum_t(ms) / d + (T)IDA_EPS_RMS);
    for (int j = lane; j < d; j += 32) {
        const T x = (T)load_in(a.v, a.dtype, base_v + (size_t)t * sv + j);
        row[2 * R + j] = fma(x * r, (T)nw[R + j], (T)bs[R + j]);
    }
}

// ---- bwd_scan: the recurrence and its adjoint ---------------------------------------------
//
// Thread c owns state column c (c < R: U, R <= c < R + d: Gamma) of every mode; threads
// c < M also own mode c's eta entry.  Planar layout of a state (sd elements): Re rows
// [m][R + d], Im rows, then eta Re [M], eta Im [M].

template <typename T>
__global__ void __launch_bounds__(BWD_THREADS, 1) bwd_scan_kernel(BackwardArgs a, T *ws, BwdLayout L) {
    extern __shared__ __align__(16) unsigned char smraw[];
    const int R = a.R, d = a.d, H = a.H, N = a.N, M = a.M, RD = R + d;
    const int unit = blockIdx.x, h = unit % H, b = unit / H;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const bool eta_ro = (a.flags & IDA_READOUT_ETA) != 0;
    T *base = ws + (size_t)unit * L.per_unit;
    const T *feat = base + L.feat;
    T *gfeat = base + L.gfeat;
    T *ckpt = base + L.ckpt, *xbuf = base + L.xbuf, *Y = base + L.adj, *LB = Y + L.sd, *BB = LB + L.sd;
    const size_t plane = (size_t)M * RD, F = 2 * (size_t)R + d;
    // shared: lambda, B [M] complex; a, abar [M] complex; per-warp mode partials
    T *lam_r = reinterpret_cast<T *>(smraw), *lam_i = lam_r + M, *b_r = lam_i + M, *b_i = b_r + M;
    T *a_r = b_i + M, *a_i = a_r + M, *ab_r = a_i + M, *ab_i = ab_r + M;
    T *red = ab_i + M;                 // [BWD_WARPS][2M] partial sums over columns
    T *scal = red + (size_t)BWD_WARPS * 2 * M;  // [BWD_WARPS + 4]
    for (int m = tid; m < M; m += BWD_THREADS) {
        lam_r[m] = (T)a.lambda[((size_t)h * M + m) * 2];
        lam_i[m] = (T)a.lambda[((size_t)h * M + m) * 2 + 1];
        b_r[m] = (T)a.Bvec[((size_t)h * M + m) * 2];
        b_i[m] = (T)a.Bvec[((size_t)h * M + m) * 2 + 1];
    }
    __syncthreads();
    const int c = tid;
    const bool col = c < RD;
    const bool has_eta = tid < M;  // thread m also carries eta[m]
    const size_t zoff = (size_t)R + c;  // z column c in a feature row [xi(q) | kt | vt]
    const size_t eoff = 2 * plane;

    // Phase A: forward recurrence, storing the state before each chunk.
    for (int m = 0; m < M && col; ++m) {
        T xr = 0, xi = 0;
        const T lr = lam_r[m], li = lam_i[m], br = b_r[m], bi = b_i[m];
        for (int t = 0; t < N; ++t) {
            if (t % BWD_CHUNK == 0) {
                T *ck = ckpt + (size_t)(t / BWD_CHUNK) * L.sd;
                ck[(size_t)m * RD + c] = xr;
                ck[plane + (size_t)m * RD + c] = xi;
            }
            const T z = feat[(size_t)t * F + zoff];
            const T nr = fma(lr, xr, fma(-li, xi, br * z)), ni = fma(lr, xi, fma(li, xr, bi * z));
            xr = nr;
            xi = ni;
        }
    }
    if (has_eta) {
        const int m = tid;
        T er = 0, ei = 0;
        const T lr = lam_r[m], li = lam_i[m], br = b_r[m], bi = b_i[m];
        for (int t = 0; t < N; ++t) {
            if (t % BWD_CHUNK == 0) {
                T *ck = ckpt + (size_t)(t / BWD_CHUNK) * L.sd;
                ck[eoff + m] = er;
                ck[eoff + M + m] = ei;
            }
            const T nr = fma(lr, er, fma(-li, ei, br)), ni = fma(lr, ei, fma(li, er, bi));
            er = nr;
            ei = ni;
        }
    }
    // adjoint accumulators start at zero
    for (size_t e = tid; e < L.sd; e += BWD_THREADS) {
        Y[e] = 0;
        LB[e] = 0;
        BB[e] = 0;
    }
    __syncthreads();

    const size_t sdout = (size_t)a.H * d;
    const size_t base_o = ((size_t)b * N * H + h) * d;
    for (int k = L.nck - 1; k >= 0; --k) {
        const int t0 = k * BWD_CHUNK, len = min(BWD_CHUNK, N - t0);
        // Phase B1: the chunk's states, xbuf[i] = X_{t0 - 1 + i}
        const T *ck = ckpt + (size_t)k * L.sd;
        for (int m = 0; m < M && col; ++m) {
            T xr = ck[(size_t)m * RD + c], xi = ck[plane + (size_t)m * RD + c];
            const T lr = lam_r[m], li = lam_i[m], br = b_r[m], bi = b_i[m];
            xbuf[(size_t)m * RD + c] = xr;
            xbuf[plane + (size_t)m * RD + c] = xi;
            for (int i = 0; i < len; ++i) {
                const T z = feat[(size_t)(t0 + i) * F + zoff];
                const T nr = fma(lr, xr, fma(-li, xi, br * z)), ni = fma(lr, xi, fma(li, xr, bi * z));
                xr = nr;
                xi = ni;
                T *xb = xbuf + (size_t)(i + 1) * L.sd;
                xb[(size_t)m * RD + c] = xr;
                xb[plane + (size_t)m * RD + c] = xi;
            }
        }
        if (has_eta) {
            const int m = tid;
            T er = ck[eoff + m], ei = ck[eoff + M + m];
            const T lr = lam_r[m], li = lam_i[m], br = b_r[m], bi = b_i[m];
            xbuf[eoff + m] = er;
            xbuf[eoff + M + m] = ei;
            for (int i = 0; i < len; ++i) {
                const T nr = fma(lr, er, fma(-li, ei, br)), ni = fma(lr, ei, fma(li, er, bi));
                er = nr;
                ei = ni;
                T *xb = xbuf + (size_t)(i + 1) * L.sd;
                xb[eoff + m] = er;
                xb[eoff + M + m] = ei;
            }
        }
        __syncthreads();
        // Phase B2: positions of the chunk, last first
        for (int i = len - 1; i >= 0; --i) {
            const int t = t0 + i;
            const T *X = xbuf + (size_t)(i + 1) * L.sd;   // X_t
            const T *Xp = xbuf + (size_t)i * L.sd;        // X_{t-1}
            const T *frow = feat + (size_t)t * F;
            const T xq = c < R ? frow[c] : T(0);
            // a_t[m] = sum_c xi(q)[c] U_t[m, c]: per-warp partials, then a fixed-order sum
            for (int m = 0; m < M; ++m) {
                T pr = 0, pi = 0;
                if (c < R) {
                    pr = xq * X[(size_t)m * RD + c];
                    pi = xq * X[plane + (size_t)m * RD + c];
                }
                pr = warp_sum_t(pr);
                pi = warp_sum_t(pi);
                if (lane == 0) {
                    red[(size_t)warp * 2 * M + m] = pr;
                    red[(size_t)warp * 2 * M + M + m] = pi;
                }
            }
            __syncthreads();
            for (int m = tid; m < M; m += BWD_THREADS) {
                T sr = 0, si = 0;
                for (int w = 0; w < BWD_WARPS; ++w) {
                    sr += red[(size_t)w * 2 * M + m];
                    si += red[(size_t)w * 2 * M + M + m];
                }
                a_r[m] = sr;
                a_i[m] = si;
            }
            __syncthreads();
            // gn = g (/ den), gd = -(g . o) / den for the eta readout
            T g = 0;
            if (c >= R && col) g = (T)load_in(a.dout, a.dtype, base_o + (size_t)t * sdout + (c - R));
            T gd = 0;
            if (eta_ro) {
                // num[j] (thread j = c - R) and den
                T num = 0;
                if (c >= R && col)
                    for (int m = 0; m < M; ++m)
                        num += a_r[m] * X[(size_t)m * RD + c] - a_i[m] * X[plane + (size_t)m * RD + c];
                T dpart = 0;
                if (has_eta) dpart = a_r[tid] * X[eoff + tid] - a_i[tid] * X[eoff + M + tid];
                // den (sum over modes) and g . num (sum over value columns), fixed order
                T s1 = warp_sum_t(dpart), s2 = warp_sum_t(g * num);
                if (lane == 0) {
                    scal[warp] = s1;
                    scal[BWD_WARPS + warp] = s2;
                }
                __syncthreads();
                T den = 0, gnum = 0;
                for (int w = 0; w < BWD_WARPS; ++w) {
                    den += scal[w];
                    gnum += scal[BWD_WARPS + w];
                }
                g = g / den;
                gd = -gnum / (den * den);
                __syncthreads();  // scal reused below
            }
            // abar[m] = sum_j conj(Gamma[m, j]) gn[j] + conj(eta[m]) gd
            for (int m = 0; m < M; ++m) {
                T pr = 0, pi = 0;
                if (c >= R && col) {
                    pr = X[(size_t)m * RD + c] * g;
                    pi = -X[plane + (size_t)m * RD + c] * g;
                }
                pr = warp_sum_t(pr);
                pi = warp_sum_t(pi);
                if (lane == 0) {
                    red[(size_t)warp * 2 * M + m] = pr;
                    red[(size_t)warp * 2 * M + M + m] = pi;
                }
            }
            __syncthreads();
            for (int m = tid; m < M; m += BWD_THREADS) {
                T sr = 0, si = 0;
                for (int w = 0; w < BWD_WARPS; ++w) {
                    sr += red[(size_t)w * 2 * M + m];
                    si += red[(size_t)w * 2 * M + M + m];
                }
                if (eta_ro) {
                    sr += X[eoff + m] * gd;
                    si -= X[eoff + M + m] * gd;
                }
                ab_r[m] = sr;
                ab_i[m] = si;
            }
            __syncthreads();
            // adjoint update of my column, then the column's gradients
            if (col) {
                T dxq = 0, dz = 0;
                const T zc = frow[zoff];
                for (int m = 0; m < M; ++m) {
                    const size_t er = (size_t)m * RD + c, ei = plane + er;
                    T dr, di;  // direct adjoint of X_t[m, c]
                    if (c < R) {
                        dr = ab_r[m] * xq;
                        di = ab_i[m] * xq;
                    } else {
                        dr = a_r[m] * g;
                        di = -a_i[m] * g;
                    }
                    // Y_t = D_t + conj(lambda) Y_{t+1}
                    const T yr0 = Y[er], yi0 = Y[ei];
                    const T yr = dr + lam_r[m] * yr0 + lam_i[m] * yi0;
                    const T yi = di + lam_r[m] * yi0 - lam_i[m] * yr0;
                    Y[er] = yr;
                    Y[ei] = yi;
                    // dz = sum_m Re(conj(B) Y), lambda_bar += conj(X_{t-1}) Y, B_bar += z Y
                    dz += b_r[m] * yr + b_i[m] * yi;
                    const T pr = Xp[er], pi = Xp[ei];
                    LB[er] += pr * yr + pi * yi;
                    LB[ei] += pr * yi - pi * yr;
                    BB[er] += zc * yr;
                    BB[ei] += zc * yi;
                    if (c < R) dxq += ab_r[m] * X[er] + ab_i[m] * X[ei];  // Re(conj(abar) U)
                }
                T *grow = gfeat + (size_t)t * F;
                if (c < R) grow[c] = dxq;
                grow[R + c] = dz;  // dkt for c < R, dvt for c >= R
            }
            if (has_eta && eta_ro) {
                const int m = tid;
                const size_t er = eoff + m, ei = eoff + M + m;
                const T dr = a_r[m] * gd, di = -a_i[m] * gd;
                const T yr0 = Y[er], yi0 = Y[ei];
                const T yr = dr + lam_r[m] * yr0 + lam_i[m] * yi0;
                const T yi = di + lam_r[m] * yi0 - lam_i[m] * yr0;
                Y[er] = yr;
                Y[ei] = yi;
                const T pr = Xp[er], pi = Xp[ei];
                LB[er] += pr * yr + pi * yi;
                LB[ei] += pr * yi - pi * yr;
                BB[er] += yr;
                BB[ei] += yi;
            }
            __syncthreads();
        }
    }
    // per-mode sums of the lambda / B terms over the columns (and eta), in column order
    T *ps = base + L.pscan;
    for (int m = tid; m < M; m += BWD_THREADS) {
        T lr = 0, li = 0, br = 0, bi = 0;
        for (int cc = 0; cc < RD; ++cc) {
            lr += LB[(size_t)m * RD + cc];
            li += LB[plane + (size_t)m * RD + cc];
            br += BB[(size_t)m * RD + cc];
            bi += BB[plane + (size_t)m * RD + cc];
        }
        if (eta_ro) {
            lr += LB[eoff + m];
            li += LB[eoff + M + m];
            br += BB[eoff + m];
            bi += BB[eoff + M + m];
        }
        ps[m] = lr;
        ps[M + m] = li;
        ps[2 * M + m] = br;
        ps[3 * M + m] = bi;
    }
}

// ---- bwd_local: RMSNorm, feature map and conv backward per position ----------------------
//
// One CTA per (unit, tile of BWD_TILE positions), one warp per position.  ds of the q and k
// convs is needed at positions [t0, t0 + tile + W - 1) for the input gradients of the tile.

template <typename T>
__global__ void __launch_bounds__(256) bwd_local_kernel(BackwardArgs a, T *ws, BwdLayout L) {
    extern __shared__ __align__(16) unsigned char smraw[];
    const int R = a.R, d = a.d, H = a.H, N = a.N, W = a.W;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw8 = blockDim.x >> 5;
    const int unit = blockIdx.x / L.ntile, tile = blockIdx.x % L.ntile;
    const int b = unit / H, h = unit % H;
    const int t0 = tile * BWD_TILE, len = min(BWD_TILE, N - t0), span = min(BWD_TILE + W - 1, N - t0);
    const size_t sqk = (size_t)H * R, sv = (size_t)H * d;
    const size_t base_qk = ((size_t)b * N * H + h) * R, base_v = ((size_t)b * N * H + h) * d;
    const float *nw = a.norm_w + (size_t)h * (R + d);
    const T *gfeat = ws + (size_t)unit * L.per_unit + L.gfeat;
    const size_t F = 2 * (size_t)R + d;
    const bool l2 = (a.flags & IDA_FEAT_L2) != 0;
    // shared: ds [2][BWD_TILE + 3][R]; partials [R + d] norm weight, [R + d] bias (per warp)
    T *ds = reinterpret_cast<T *>(smraw);
    T *pnw = ds + 2 * (size_t)(BWD_TILE + 3) * R;  // [nw8][R + d]
    T *pbs = pnw + (size_t)nw8 * (R + d);          // [nw8][R + d]
    for (size_t e = threadIdx.x; e < (size_t)nw8 * (R + d); e += blockDim.x) {
        pnw[e] = 0;
        pbs[e] = 0;
    }
    __syncthreads();
    for (int p = warp; p < span; p += nw8) {
        const int t = t0 + p;
        const T *grow = gfeat + (size_t)t * F;
        const bool own = p < len;
        for (int which = 0; which < 2; ++which) {
            const void *x = which == 0 ? a.q : a.k;
            const float *cw = a.conv_w + ((size_t)which * H + h) * R * W;
            T ss = 0;
            for (int c = lane; c < R; c += 32) {
                const T f = silu(conv_at<T>(x, a.dtype, base_qk, sqk, cw, W, t, c));
                ss = fma(f, f, ss);
            }
            ss = warp_sum_t(ss);
            const T n = l2 ? sqrt(ss) : ss;
            const T D = n + (T)IDA_EPS_FEAT;
            // dxi: directly (q), or through the key RMSNorm (k)
            T r = 0, sdy = 0;
            if (which == 1) {
                T ms = 0, acc = 0;
                for (int c = lane; c < R; c += 32) {
                    const T xi = silu(conv_at<T>(x, a.dtype, base_qk, sqk, cw, W, t, c)) / D;
                    ms = fma(xi, xi, ms);
                }
                r = sqrt(warp_sum_t(ms) / R + (T)IDA_EPS_RMS);
                for (int c = lane; c < R; c += 32) {
                    const T xi = silu(conv_at<T>(x, a.dtype, base_qk, sqk, cw, W, t, c)) / D;
                    const T dkt = grow[R + c];
                    acc = fma(dkt * (T)nw[c], xi, acc);
                    if (own) {
                        pnw[(size_t)warp * (R + d) + c] += dkt * xi / r;
                        pbs[(size_t)warp * (R + d) + c] += dkt;
                    }
                }
                sdy = warp_sum_t(acc);
            }
            // s = sum_c dxi[c] f[c] / D^2 term of the feature-map backward
            T sdf = 0;
            for (int c = lane; c < R; c += 32) {
                const T f = silu(conv_at<T>(x, a.dtype, base_qk, sqk, cw, W, t, c));
                const T xi = f / D;
                const T dxi = which == 0 ? grow[c] : (grow[R + c] * (T)nw[c]) / r - xi * sdy / ((T)R * r * r * r);
                sdf = fma(dxi, f, sdf);
            }
            sdf = warp_sum_t(sdf);
            for (int c = lane; c < R; c += 32) {
                const T s = conv_at<T>(x, a.dtype, base_qk, sqk, cw, W, t, c);
                const T f = silu(s);
                const T xi = f / D;
                const T dxi = which == 0 ? grow[c] : (grow[R + c] * (T)nw[c]) / r - xi * sdy / ((T)R * r * r * r);
                // dn/df = 2 f (squared norm) or f / n (l_2 norm)
                const T dn = l2 ? (n > T(0) ? f / n : T(0)) : T(2) * f;
                const T df = dxi / D - sdf / (D * D) * dn;
                ds[((size_t)which * (BWD_TILE + 3) + p) * R + c] = df * silu_grad(s);
            }
        }
        if (own) {
            // value RMSNorm backward
            T ms = 0;
            for (int j = lane; j < d; j += 32) {
                const T xv = (T)load_in(a.v, a.dtype, base_v + (size_t)t * sv + j);
                ms = fma(xv, xv, ms);
            }
            const T r = sqrt(warp_sum_t(ms) / d + (T)IDA_EPS_RMS);
            T acc = 0;
            for (int j = lane; j < d; j += 32) {
                const T xv = (T)load_in(a.v, a.dtype, base_v + (size_t)t * sv + j);
                const T dvt = grow[2 * R + j];
                acc = fma(dvt * (T)nw[R + j], xv, acc);
                pnw[(size_t)warp * (R + d) + R + j] += dvt * xv / r;
                pbs[(size_t)warp * (R + d) + R + j] += dvt;
            }
            acc = warp_sum_t(acc);
            for (int j = lane; j < d; j += 32) {
                const T xv = (T)load_in(a.v, a.dtype, base_v + (size_t)t * sv + j);
                const T dvt = grow[2 * R + j];
                const T dv = (dvt * (T)nw[R + j]) / r - xv * acc / ((T)d * r * r * r);
                store_out(a.dv, a.dtype, base_v + (size_t)t * sv + j, (float)dv);
            }
        }
    }
    __syncthreads();
    // input gradients of the tile: dx_p[c] = sum_j w[c][j] ds_{p + W - 1 - j}[c]
    for (int e = threadIdx.x; e < 2 * len * R; e += blockDim.x) {
        const int which = e / (len * R), p = (e / R) % len, c = e % R;
        const float *cw = a.conv_w + ((size_t)which * H + h) * R * W;
        T acc = 0;
        for (int j = 0; j < W; ++j) {
            const int pp = p + W - 1 - j;  // position index within the tile of the ds term
            if (t0 + pp < N) acc = fma((T)cw[(size_t)c * W + j], ds[((size_t)which * (BWD_TILE + 3) + pp) * R + c], acc);
        }
        store_out(which == 0 ? a.dq : a.dk, a.dtype, base_qk + (size_t)(t0 + p) * sqk + c, (float)acc);
    }
    // partials of this tile: conv taps dw[which][c][j] = sum_{own t} x_{t - W + 1 + j}[c] ds_t[c]
    T *pl = ws + L.plocal_base((size_t)a.B * H) + ((size_t)unit * L.ntile + tile) * L.plocal_each;
    for (int e = threadIdx.x; e < 2 * R * W; e += blockDim.x) {
        const int which = e / (R * W), c = (e / W) % R, j = e % W;
        const void *x = which == 0 ? a.q : a.k;
        T acc = 0;
        for (int p = 0; p < len; ++p) {
            const int src = t0 + p - (W - 1) + j;
            if (src >= 0)
                acc = fma((T)load_in(x, a.dtype, base_qk + (size_t)src * sqk + c),
                          ds[((size_t)which * (BWD_TILE + 3) + p) * R + c], acc);
        }
        pl[e] = acc;
    }
    for (int e = threadIdx.x; e < R + d; e += blockDim.x) {
        T sn = 0, sb = 0;
        for (int w = 0; w < nw8; ++w) {
            sn += pnw[(size_t)w * (R + d) + e];
            sb += pbs[(size_t)w * (R + d) + e];
        }
        pl[2 * (size_t)R * W + e] = sn;
        pl[2 * (size_t)R * W + (R + d) + e] = sb;
    }
}

// ---- bwd_reduce: parameter gradients summed over batch rows (and tiles) -------------------

template <typename T>
__global__ void bwd_reduce_kernel(BackwardArgs a, const T *ws, BwdLayout L) {
    const int R = a.R, d = a.d, H = a.H, M = a.M, W = a.W, B = a.B;
    const size_t units = (size_t)B * H;
    const int per_h = 2 * R * W + 2 * (R + d) + 4 * M;
    const int e = blockIdx.x * blockDim.x + threadIdx.x;
    if (e >= H * per_h) return;
    const int h = e / per_h, f = e % per_h;
    T acc = 0;
    if (f < 2 * R * W + 2 * (R + d)) {
        for (int b = 0; b < B; ++b) {
            const size_t unit = (size_t)b * H + h;
            for (int tile = 0; tile < L.ntile; ++tile)
                acc += ws[L.plocal_base(units) + (unit * L.ntile + tile) * L.plocal_each + f];
        }
        if (f < 2 * R * W) {
            const int which = f / (R * W), rest = f % (R * W);
            a.dconv_w[((size_t)which * H + h) * R * W + rest] = (float)acc;
        } else if (f < 2 * R * W + (R + d)) {
            a.dnorm_w[(size_t)h * (R + d) + (f - 2 * R * W)] = (float)acc;
        } else {
            a.dbias[(size_t)h * (R + d) + (f - 2 * R * W - (R + d))] = (float)acc;
        }
    } else {
        const int g = f - (2 * R * W + 2 * (R + d));  // [lambda re, lambda im, B re, B im][M]
        for (int b = 0; b < B; ++b) acc += ws[((size_t)b * H + h) * L.per_unit + L.pscan + g];
        const int kind = g / M, m = g % M;
        float *dst = kind < 2 ? a.dlambda : a.dBvec;
        dst[((size_t)h * M + m) * 2 + (kind & 1)] = (float)acc;
    }
}

template <typename T>
static size_t bwd_scan_smem(int M) {
    return ((size_t)8 * M + (size_t)BWD_WARPS * 2 * M + BWD_WARPS * 2 + 4) * sizeof(T);
}

template <typename T>
static size_t bwd_local_smem(int R, int d) {
    return (2 * (size_t)(BWD_TILE + 3) * R + 2 * 8 * ((size_t)R + d)) * sizeof(T);
}

size_t backward_workspace_bytes(int B, int H, int N, int d, int R, int M, int dtype, int W) {
    if (B <= 0 || H <= 0 || N <= 0) return 0;
    const size_t e = dtype == IDA_F32 ? sizeof(double) : sizeof(float);
    return BwdLayout::of(B, H, N, d, R, M, W).total * e;
}

template <typename T>
static cudaError_t launch_backward_t(const BackwardArgs &a, void *workspace, cudaStream_t st) {
    const BwdLayout L = BwdLayout::of(a.B, a.H, a.N, a.d, a.R, a.M, a.W);
    T *ws = static_cast<T *>(workspace);
    const unsigned units = (unsigned)(a.B * a.H);
    cudaError_t e;
    bwd_features_kernel<T><<<units * (unsigned)((a.N + 7) / 8), 256, 0, st>>>(a, ws, L);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    const size_t s1 = bwd_scan_smem<T>(a.M);
    if ((e = cudaFuncSetAttribute(bwd_scan_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)s1)) !=
        cudaSuccess)
        return e;
    bwd_scan_kernel<T><<<units, BWD_THREADS, s1, st>>>(a, ws, L);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    const size_t s2 = bwd_local_smem<T>(a.R, a.d);
    if ((e = cudaFuncSetAttribute(bwd_local_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)s2)) !=
        cudaSuccess)
        return e;
    bwd_local_kernel<T><<<units * (unsigned)L.ntile, 256, s2, st>>>(a, ws, L);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    const int per_h = 2 * a.R * a.W + 2 * (a.R + a.d) + 4 * a.M;
    const unsigned n = (unsigned)(a.H * per_h);
    bwd_reduce_kernel<T><<<(n + 255) / 256, 256, 0, st>>>(a, ws, L);
    return cudaGetLastError();
}

ida_status launch_backward(const BackwardArgs &a, void *workspace, cudaStream_t st, std::string &why) {
    const cudaError_t e = a.dtype == IDA_F32 ? launch_backward_t<double>(a, workspace, st)
                                             : launch_backward_t<float>(a, workspace, st);
    if (e != cudaSuccess) {
        why = std::string("backward launch: ") + cudaGetErrorString(e);
        return IDA_ERR_CUDA;
    }
    return IDA_OK;
}

ida_status fail_with(ida_status s, const std::string &why);
ida_status device_error_word(unsigned **err, std::string &why);
ida_status check_call(int d, int R, int M, int W, int dtype, int flags, int *num_sms, std::string &why);

}  // namespace ida

extern "C" size_t ida_backward_workspace_bytes(int B, int H, int N, int d, int R, int M, int dtype, int W,
                                               int flags) {
    (void)flags;
    if (B < 0 || H < 0 || N < 0 || d < 1 || R < 1 || M < 1 || W < 1 || W > 4 || R > 256 || d > 256 || M > 128 ||
        (dtype != IDA_F32 && dtype != IDA_BF16))
        return 0;
    return ida::backward_workspace_bytes(B, H, N, d, R, M, dtype, W);
}

extern "C" ida_status ida_backward(const void *q, const void *k, const void *v, const float *conv_w,
                                   const float *norm_w, const float *bias, const float *lambda, const float *Bvec,
                                   const void *dout, void *dq, void *dk, void *dv, float *dconv_w, float *dnorm_w,
                                   float *dbias, float *dlambda, float *dBvec, int B, int H, int N, int d, int R,
                                   int M, int dtype, int W, int flags, void *workspace, size_t workspace_bytes,
                                   ida_stream_t stream) {
    std::string why;
    if (B < 0 || H < 0 || N < 0) return ida::fail_with(IDA_ERR_ARG, "B, H and N must be >= 0");
    if (flags & IDA_PATH_SEQUENTIAL) return ida::fail_with(IDA_ERR_ARG, "IDA_PATH_SEQUENTIAL is a prefill flag");
    int num_sms = 0;
    // shape and flag checks, the device error word (a pending device error is reported here)
    ida_status s = ida::check_call(d, R, M, W, dtype, flags, nullptr, why);
    if (s != IDA_OK) return ida::fail_with(s, why);
    if ((long long)B * H > (1LL << 20)) return ida::fail_with(IDA_ERR_UNSUPPORTED, "B*H above 2^20");
    // the per-position tensors are empty (and may be null) when N == 0
    const void *ptrs[] = {conv_w, norm_w, bias, lambda, Bvec, dconv_w, dnorm_w, dbias, dlambda, dBvec,
                          q, k, v, dout, dq, dk, dv};
    const int nptr = N > 0 ? 17 : 10;
    for (int i = 0; i < nptr; ++i)
        if (!ptrs[i]) return ida::fail_with(IDA_ERR_ARG, "null pointer");
    for (int i = 0; i < nptr; ++i)
        if ((reinterpret_cast<uintptr_t>(ptrs[i]) & 15u) != 0)
            return ida::fail_with(IDA_ERR_ARG, "pointers must be 16-byte aligned");
    if (workspace && (reinterpret_cast<uintptr_t>(workspace) & 15u) != 0)
        return ida::fail_with(IDA_ERR_ARG, "workspace must be 16-byte aligned");
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if ((long long)B * H == 0) return IDA_OK;
    const size_t need = ida::backward_workspace_bytes(B, H, N, d, R, M, dtype, W);
    if (N > 0 && (!workspace || workspace_bytes < need))
        return ida::fail_with(IDA_ERR_ARG, "the backward pass needs a workspace of ida_backward_workspace_bytes(...) = " +
                                               std::to_string(need) + " bytes");
    s = ida::check_call(d, R, M, W, dtype, flags, &num_sms, why);
    if (s != IDA_OK) return ida::fail_with(s, why);
    if (N == 0) {  // no positions: every gradient is zero (dq, dk, dv are empty)
        cudaError_t e = cudaSuccess;
        const size_t H_ = (size_t)H;
        if (e == cudaSuccess) e = cudaMemsetAsync(dconv_w, 0, 2 * H_ * R * W * sizeof(float), st);
        if (e == cudaSuccess) e = cudaMemsetAsync(dnorm_w, 0, H_ * (R + d) * sizeof(float), st);
        if (e == cudaSuccess) e = cudaMemsetAsync(dbias, 0, H_ * (R + d) * sizeof(float), st);
        if (e == cudaSuccess) e = cudaMemsetAsync(dlambda, 0, H_ * M * 2 * sizeof(float), st);
        if (e == cudaSuccess) e = cudaMemsetAsync(dBvec, 0, H_ * M * 2 * sizeof(float), st);
        return e == cudaSuccess ? IDA_OK : ida::fail_with(IDA_ERR_CUDA, cudaGetErrorString(e));
    }
    unsigned *err = nullptr;
    s = ida::device_error_word(&err, why);
    if (s != IDA_OK) return ida::fail_with(s, why);
    ida::BackwardArgs a;
    a.q = q; a.k = k; a.v = v; a.dout = dout;
    a.conv_w = conv_w; a.norm_w = norm_w; a.bias = bias; a.lambda = lambda; a.Bvec = Bvec;
    a.dq = dq; a.dk = dk; a.dv = dv;
    a.dconv_w = dconv_w; a.dnorm_w = dnorm_w; a.dbias = dbias; a.dlambda = dlambda; a.dBvec = dBvec;
    a.B = B; a.H = H; a.N = N; a.d = d; a.R = R; a.M = M; a.W = W; a.dtype = dtype; a.flags = flags;
    a.err = err;
    s = ida::launch_backward(a, workspace, st, why);
    return s == IDA_OK ? IDA_OK : ida::fail_with(s, why);
}
