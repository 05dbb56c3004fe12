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
//   bwd_scan_a     per (unit, slice of modes): the forward recurrence with the state in
//                  registers, storing the state before every chunk of 64 positions (and,
//                  for the eta readout, the slice's parts of numerator and denominator);
//   bwd_scan_nd    eta readout: 1 / den and -(g . o) / den per position;
//   bwd_scan_b     per (unit, slice of modes): chunk by chunk from the end, the chunk's
//                  states recomputed from its checkpoint and the adjoint walked backwards
//                  through them with the adjoint state and its lambda / B sums in
//                  registers; the slice's dxi(q), dkt, dvt per position and the slice's
//                  lambda / B gradients; bwd_sum_slices adds the slices' parts;
//   bwd_local      one CTA per (unit, tile of positions): RMSNorm, feature-map and conv
//                  backward, dq, dk, dv, and per-tile partial parameter gradients;
//   bwd_reduce     sums the partials over batch rows and tiles into the parameter gradients.
// Arithmetic type T: double for fp32 inputs, float for bf16 inputs.
#include <cstdint>
#include <string>

#include "ida_common.cuh"

namespace ida {

constexpr int BWD_TILE = 32;      // positions per bwd_local CTA
constexpr int BWD_LANE_CH = 8;    // channels per lane in the per-position kernels (R, d <= 256)
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

// Mode slicing of the adjoint scan: a CTA of BWD_THREADS threads holds G groups of RDw threads
// (one thread per state column, RDw = R + d rounded up to whole warps); each thread keeps the
// adjoint state of up to BWD_MGT modes of its column in registers, so a CTA covers
// MC = G * BWD_MGT modes and a unit's M modes are split over S = ceil(M / MC) CTAs.
constexpr int BWD_MGT = 8;

struct BwdSlicing {
    int RDw, G, MC, S;
    __host__ __device__ static BwdSlicing of(int R, int d, int M) {
        BwdSlicing q;
        q.RDw = (R + d + 31) / 32 * 32;
        q.G = BWD_THREADS / q.RDw;
        q.MC = q.G * BWD_MGT;
        q.S = (M + q.MC - 1) / q.MC;
        return q;
    }
    // modes of slice s, and the elements of one slice-local state as the scans store it:
    // [Re, Im][thread][BWD_MGT] (a thread's modes contiguous, so it moves them as 16-byte
    // vectors; threads without a column hold zeros), then eta [Re, Im][MC]
    __host__ __device__ int ms(int s, int M) const { return M - s * MC < MC ? M - s * MC : MC; }
    static constexpr size_t plane = (size_t)BWD_THREADS * BWD_MGT;
    __host__ __device__ size_t sds() const { return 2 * plane + 2 * (size_t)MC; }
};

// Positions between checkpoints of the state: the adjoint scan stages one such chunk in
// shared memory, which fits in an SM at 16 fp32 positions or 8 fp64 ones.
template <typename T>
struct BwdChunk {
    static constexpr int C = sizeof(T) == 8 ? 8 : 16;
};

// Workspace layout (elements of T), per unit unless noted.
struct BwdLayout {
    size_t feat;    // [N][2R + d]: xi(q), kt, vt
    size_t gfeat;   // [S][N][2R + d]: per mode slice, its part of dxi(q), dkt, dvt (summed into slice 0)
    size_t nd;      // [S][N][d + 1]: eta readout, per slice: partial numerator and denominator
    size_t gsc;     // [N][2]: eta readout: 1 / den and -(g . o) / den
    size_t ckpt;    // [S][nck][sds]
    size_t xbuf;    // [S][chunk + 1][sds]
    size_t pscan;   // [4M]: lambda-bar (re, im), B-bar (re, im)
    size_t per_unit;
    size_t sds;
    size_t plocal_each;  // per (unit, tile): [2][R][W] conv, [R + d] norm weight, [R + d] bias
    int nck, ntile, S, chunk;
    size_t total;  // elements of T
    // chunk: positions between checkpoints (BwdChunk<T>::C of the arithmetic type)
    static BwdLayout of(int B, int H, int N, int d, int R, int M, int W, bool eta, int chunk) {
        BwdLayout L;
        const BwdSlicing q = BwdSlicing::of(R, d, M);
        const size_t units = (size_t)B * H, F = 2 * (size_t)R + d;
        L.S = q.S;
        L.chunk = chunk;
        L.nck = (N + chunk - 1) / chunk;
        L.ntile = (N + BWD_TILE - 1) / BWD_TILE;
        L.sds = q.sds();
        // every region starts on a multiple of 4 elements (16-byte vectors of the states)
        auto r4 = [](size_t x) { return (x + 3) & ~(size_t)3; };
        L.feat = 0;
        L.gfeat = r4(L.feat + (size_t)N * F);
        L.nd = r4(L.gfeat + (size_t)q.S * N * F);
        L.gsc = r4(L.nd + (eta ? (size_t)q.S * N * (d + 1) : 0));
        L.ckpt = r4(L.gsc + (eta ? 2 * (size_t)N : 0));
        L.xbuf = r4(L.ckpt + (size_t)q.S * L.nck * L.sds);
        L.pscan = r4(L.xbuf + (size_t)q.S * (chunk + 1) * L.sds);
        L.per_unit = r4(L.pscan + 4 * (size_t)M);
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

// a thread's BWD_MGT mode values of one state plane, as 16-byte vectors (p 16-byte aligned)
template <int K>
__device__ __forceinline__ void ldgm(const float *p, float (&o)[K]) {
    static_assert(K % 4 == 0, "whole float4 vectors");
#pragma unroll
    for (int v = 0; v < K / 4; ++v) {
        const float4 x = reinterpret_cast<const float4 *>(p)[v];
        o[4 * v] = x.x;
        o[4 * v + 1] = x.y;
        o[4 * v + 2] = x.z;
        o[4 * v + 3] = x.w;
    }
}
template <int K>
__device__ __forceinline__ void ldgm(const double *p, double (&o)[K]) {
    static_assert(K % 2 == 0, "whole double2 vectors");
#pragma unroll
    for (int v = 0; v < K / 2; ++v) {
        const double2 x = reinterpret_cast<const double2 *>(p)[v];
        o[2 * v] = x.x;
        o[2 * v + 1] = x.y;
    }
}
template <int K>
__device__ __forceinline__ void stgm(float *p, const float (&o)[K]) {
#pragma unroll
    for (int v = 0; v < K / 4; ++v)
        reinterpret_cast<float4 *>(p)[v] = make_float4(o[4 * v], o[4 * v + 1], o[4 * v + 2], o[4 * v + 3]);
}
template <int K>
__device__ __forceinline__ void stgm(double *p, const double (&o)[K]) {
#pragma unroll
    for (int v = 0; v < K / 2; ++v) reinterpret_cast<double2 *>(p)[v] = make_double2(o[2 * v], o[2 * v + 1]);
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
        T fv[BWD_LANE_CH];  // SiLU of the conv of my channels c = lane + 32 i, computed once
        T ss = 0;
#pragma unroll
        for (int i = 0; i < BWD_LANE_CH; ++i) {
            const int c = lane + 32 * i;
            fv[i] = c < R ? silu(conv_at<T>(x, a.dtype, base_qk, sqk, cw, W, t, c)) : T(0);
            ss = fma(fv[i], fv[i], ss);
        }
        T n = warp_sum_t(ss);
        if (l2) n = sqrt(n);
        const T inv = T(1) / (n + (T)IDA_EPS_FEAT);
        if (which == 0) {
#pragma unroll
            for (int i = 0; i < BWD_LANE_CH; ++i)
                if (lane + 32 * i < R) row[lane + 32 * i] = fv[i] * inv;
        } else {
            T ms = 0;
#pragma unroll
            for (int i = 0; i < BWD_LANE_CH; ++i) ms = fma(fv[i] * inv, fv[i] * inv, ms);
            const T r = T(1) / sqrt(warp_sum_t(ms) / R + (T)IDA_EPS_RMS);
#pragma unroll
            for (int i = 0; i < BWD_LANE_CH; ++i) {
                const int c = lane + 32 * i;
                if (c < R) row[R + c] = fma(fv[i] * inv * r, (T)nw[c], (T)bs[c]);
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
// Grid: units x S mode slices.  Thread (group g, column c) owns state column c (c < R: U,
// R <= c < R + d: Gamma) of the slice-local modes g, g + G, g + 2G, ...; thread j < ms also
// owns the eta entry of slice-local mode j.

// Phase A: the forward recurrence of the slice's modes over all positions, storing the state
// before every chunk; for the eta readout also the slice's part of the numerator and of the
// denominator at every position.
template <typename T, bool ETA>
__global__ void __launch_bounds__(BWD_THREADS, 1) bwd_scan_a_kernel(BackwardArgs a, T *ws, BwdLayout L) {
    __shared__ T red[BWD_WARPS][2 * BWD_MGT];
    __shared__ T am[2][BWD_THREADS / 32 * BWD_MGT];  // a_t of the slice's modes (re, im)
    __shared__ T part[BWD_THREADS];
    const int R = a.R, d = a.d, H = a.H, N = a.N, M = a.M, RD = R + d;
    const BwdSlicing q = BwdSlicing::of(R, d, M);
    const int unit = blockIdx.x / q.S, sl = blockIdx.x % q.S, h = unit % H;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = tid / q.RDw, c = tid % q.RDw, ms = q.ms(sl, M);
    const bool col = g < q.G && c < RD;
    constexpr bool eta_ro = ETA;
    T *base = ws + (size_t)unit * L.per_unit;
    const T *feat = base + L.feat;
    T *ckpt = base + L.ckpt + (size_t)sl * L.nck * L.sds;
    T *nd = base + L.nd + (size_t)sl * N * (d + 1);
    const size_t F = 2 * (size_t)R + d, plane = BwdSlicing::plane, eoff = 2 * plane, mine = (size_t)tid * BWD_MGT;
    T lr[BWD_MGT], li[BWD_MGT], br[BWD_MGT], bi[BWD_MGT], xr[BWD_MGT], xi[BWD_MGT];
#pragma unroll
    for (int i = 0; i < BWD_MGT; ++i) {
        const int ml = g + q.G * i, m = sl * q.MC + ml;
        const bool ok = col && ml < ms;
        lr[i] = ok ? (T)a.lambda[((size_t)h * M + m) * 2] : T(0);
        li[i] = ok ? (T)a.lambda[((size_t)h * M + m) * 2 + 1] : T(0);
        br[i] = ok ? (T)a.Bvec[((size_t)h * M + m) * 2] : T(0);
        bi[i] = ok ? (T)a.Bvec[((size_t)h * M + m) * 2 + 1] : T(0);
        xr[i] = 0;
        xi[i] = 0;
    }
    // eta of slice-local mode tid
    const bool eown = tid < ms;
    T elr = 0, eli = 0, ebr = 0, ebi = 0, er = 0, ei = 0;
    if (eown) {
        const int m = sl * q.MC + tid;
        elr = (T)a.lambda[((size_t)h * M + m) * 2];
        eli = (T)a.lambda[((size_t)h * M + m) * 2 + 1];
        ebr = (T)a.Bvec[((size_t)h * M + m) * 2];
        ebi = (T)a.Bvec[((size_t)h * M + m) * 2 + 1];
    }
    const int gwarps = q.RDw / 32;  // warps per group
    if constexpr (!ETA) {
        // chunk by chunk: the checkpoint, then the chunk's z loaded together and the recurrence
        constexpr int C = BwdChunk<T>::C;
        for (int k = 0; k < L.nck; ++k) {
            const int t0 = k * C, len = min(C, N - t0);
            T *ck = ckpt + (size_t)k * L.sds;
            stgm(ck + mine, xr);
            stgm(ck + plane + mine, xi);
            T zv[C];
#pragma unroll
            for (int j = 0; j < C; ++j) zv[j] = col ? feat[(size_t)min(t0 + j, N - 1) * F + R + c] : T(0);
#pragma unroll
            for (int j = 0; j < C; ++j) {
                if (j < len) {
#pragma unroll
                    for (int i = 0; i < BWD_MGT; ++i) {
                        const T nr = fma(lr[i], xr[i], fma(-li[i], xi[i], br[i] * zv[j]));
                        const T ni = fma(lr[i], xi[i], fma(li[i], xr[i], bi[i] * zv[j]));
                        xr[i] = nr;
                        xi[i] = ni;
                    }
                }
            }
        }
        return;
    }
    // eta readout: position by position, with the slice's numerator and denominator parts;
    // z and xi(q) of the next ZP positions in flight (fewer in fp64, for registers)
    constexpr int ZP = sizeof(T) == 8 ? 2 : 8;
    const bool kq = eta_ro && col && c < R;
    T zq[ZP], qq[ZP];
#pragma unroll
    for (int u = 0; u < ZP; ++u) {
        zq[u] = (col && u < N) ? feat[(size_t)u * F + R + c] : T(0);
        qq[u] = (kq && u < N) ? feat[(size_t)u * F + c] : T(0);
    }
    for (int t0 = 0; t0 < N; t0 += ZP)
#pragma unroll
    for (int u = 0; u < ZP; ++u) {
        const int t = t0 + u;
        if (t >= N) break;
        const T z = zq[u], xq = qq[u];
        zq[u] = (col && t + ZP < N) ? feat[(size_t)(t + ZP) * F + R + c] : T(0);
        qq[u] = (kq && t + ZP < N) ? feat[(size_t)(t + ZP) * F + c] : T(0);
        if (t % L.chunk == 0) {
            T *ck = ckpt + (size_t)(t / L.chunk) * L.sds;
            stgm(ck + mine, xr);
            stgm(ck + plane + mine, xi);
            if (eown) {
                ck[eoff + tid] = er;
                ck[eoff + q.MC + tid] = ei;
            }
        }
#pragma unroll
        for (int i = 0; i < BWD_MGT; ++i) {
            const T nr = fma(lr[i], xr[i], fma(-li[i], xi[i], br[i] * z));
            const T ni = fma(lr[i], xi[i], fma(li[i], xr[i], bi[i] * z));
            xr[i] = nr;
            xi[i] = ni;
        }
        if (eown) {
            const T nr = fma(elr, er, fma(-eli, ei, ebr)), ni = fma(elr, ei, fma(eli, er, ebi));
            er = nr;
            ei = ni;
        }
        if (eta_ro) {
            // a_t of the slice's modes: sum over the group's key columns
            T v[2 * BWD_MGT];
#pragma unroll
            for (int i = 0; i < BWD_MGT; ++i) {
                v[2 * i] = xq * xr[i];
                v[2 * i + 1] = xq * xi[i];
            }
            const T s1 = warp_reduce_scatter<2 * BWD_MGT>(v, lane);
            if ((lane & 1) == 0) red[warp][rs_index<2 * BWD_MGT>(lane)] = s1;
            __syncthreads();
            if (tid < q.G * 2 * BWD_MGT) {
                const int gg = tid / (2 * BWD_MGT), k = tid % (2 * BWD_MGT);
                T sum = 0;
                for (int w = 0; w < gwarps; ++w) sum += red[gg * gwarps + w][k];
                am[k & 1][gg * BWD_MGT + (k >> 1)] = sum;  // [re/im][group * MGT + i]
            }
            __syncthreads();
            // numerator part of value column c - R, denominator part of the eta entries
            T pn = 0;
            if (col && c >= R)
#pragma unroll
                for (int i = 0; i < BWD_MGT; ++i) pn += am[0][g * BWD_MGT + i] * xr[i] - am[1][g * BWD_MGT + i] * xi[i];
            part[tid] = pn;
            T pd = 0;
            if (eown) {
                const int gg = tid % q.G, i = tid / q.G;  // slice-local mode tid = gg + G i
                pd = am[0][gg * BWD_MGT + i] * er - am[1][gg * BWD_MGT + i] * ei;
            }
            pd = warp_sum_t(pd);
            __syncthreads();
            if (tid < d) {
                T sum = 0;
                for (int gg = 0; gg < q.G; ++gg) sum += part[gg * q.RDw + R + tid];
                nd[(size_t)t * (d + 1) + tid] = sum;
            }
            if (lane == 0) red[warp][0] = pd;
            __syncthreads();
            if (tid == 0) {
                T sum = 0;
                for (int w = 0; w < BWD_WARPS; ++w) sum += red[w][0];
                nd[(size_t)t * (d + 1) + d] = sum;
            }
            __syncthreads();
        }
    }
}

// eta readout: per position, the numerator and denominator over all slices, then
// 1 / den and gd = -(g . num) / den^2 (one warp per position)
template <typename T>
__global__ void __launch_bounds__(256) bwd_scan_nd_kernel(BackwardArgs a, T *ws, BwdLayout L) {
    const int d = a.d, H = a.H, N = a.N;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int tiles = (N + 7) / 8;
    const int unit = blockIdx.x / tiles, t = (blockIdx.x % tiles) * 8 + warp;
    if (t >= N) return;
    const int b = unit / H, h = unit % H;
    T *base = ws + (size_t)unit * L.per_unit;
    const T *nd = base + L.nd;
    const size_t base_o = ((size_t)b * N * H + h) * d, so = (size_t)H * d;
    T gn = 0, den = 0;
    for (int j = lane; j <= d; j += 32) {
        T sum = 0;
        for (int s = 0; s < L.S; ++s) sum += nd[((size_t)s * N + t) * (d + 1) + j];
        if (j < d)
            gn = fma((T)load_in(a.dout, a.dtype, base_o + (size_t)t * so + j), sum, gn);
        else
            den = sum;
    }
    gn = warp_sum_t(gn);
    den = warp_sum_t(den);
    if (lane == 0) {
        base[L.gsc + 2 * (size_t)t] = T(1) / den;
        base[L.gsc + 2 * (size_t)t + 1] = -gn / (den * den);
    }
}

// four consecutive values from 16-byte aligned shared memory
__device__ __forceinline__ void lds4(const float *p, float (&o)[4]) {
    const float4 x = *reinterpret_cast<const float4 *>(p);
    o[0] = x.x; o[1] = x.y; o[2] = x.z; o[3] = x.w;
}
__device__ __forceinline__ void lds4(const double *p, double (&o)[4]) {
    const double2 x = reinterpret_cast<const double2 *>(p)[0], y = reinterpret_cast<const double2 *>(p)[1];
    o[0] = x.x; o[1] = x.y; o[2] = y.x; o[3] = y.y;
}

// Dynamic shared memory of bwd_scan_b, in elements of T.
template <typename T, bool SPLIT>
struct ScanBSmem {
    static constexpr int C = BwdChunk<T>::C;
    static constexpr int RV = SPLIT ? 2 * BWD_MGT : 4 * BWD_MGT;  // values a warp sums per position
    static constexpr int GM = BWD_THREADS / 32 * BWD_MGT;         // >= G * MGT mode entries
    static constexpr size_t RED = 0;                                   // [C][warp][RV] warp sums
    static constexpr size_t AM = RED + (size_t)C * BWD_WARPS * RV;     // [C][Re, Im][GM] a_t
    static constexpr size_t ABM = AM + (size_t)C * 2 * GM;             // [C][Re, Im][GM] abar_t
    static constexpr size_t PART = ABM + (size_t)C * 2 * GM;           // [C][dz, dxi(q)][thread]
    static constexpr size_t INP = PART + (size_t)C * 2 * BWD_THREADS;  // [C][s, z][thread]
    static constexpr size_t ETAS = INP + (size_t)C * 2 * BWD_THREADS;  // [C + 1][Re, Im][GM] eta at t0 - 1 + j
    static constexpr size_t GD = ETAS + (size_t)(C + 1) * 2 * GM;      // [C] gd
    static constexpr size_t BYTES = (GD + C) * sizeof(T);
    static_assert(BYTES + 4 * GM * sizeof(T) + 4 * BWD_WARPS * sizeof(T) <= 227 * 1024, "shared memory budget");
};

// Phase B: the adjoint, chunk by chunk from the end.  Per chunk of C positions:
//  1. forward from the chunk's checkpoint: the states X_t (kept for step 3 in the replay
//     buffer, in L2), eta_t, the inputs of every position staged in shared memory, and
//     each warp's partial sums of a_t (key columns) and abar_t's Gamma part (value
//     columns) for every position; none of this depends on the adjoint state;
//  2. the sums over each group's warps, for every position at once (plus conj(eta_t) gd
//     for the eta readout);
//  3. the adjoint walked back through the chunk with no barrier: the adjoint state, its
//     lambda / B sums, and each thread's parts of dz and dxi(q) per position;
//  4. the parts summed over the groups into dz and dxi(q) rows.
// Three block barriers per chunk.
template <typename T, bool SPLIT, bool ETA>
__global__ void __launch_bounds__(BWD_THREADS, 1) bwd_scan_b_kernel(BackwardArgs a, T *ws, BwdLayout L) {
    using SM = ScanBSmem<T, SPLIT>;
    constexpr int C = SM::C, RV = SM::RV, GM = SM::GM, NT = BWD_THREADS;
    extern __shared__ __align__(16) unsigned char smraw[];
    T *const sm = reinterpret_cast<T *>(smraw);
    T *const red = sm + SM::RED, *const am = sm + SM::AM, *const abm = sm + SM::ABM;
    T *const part = sm + SM::PART, *const inp = sm + SM::INP, *const etas = sm + SM::ETAS, *const gds = sm + SM::GD;
    __shared__ __align__(16) T lam_s[2][GM];  // lambda, B of the slice's modes, [group * MGT + i],
    __shared__ __align__(16) T bv_s[2][GM];   // zero past them
    __shared__ T fred[BWD_WARPS][4];
    const int R = a.R, d = a.d, H = a.H, N = a.N, M = a.M, RD = R + d;
    const BwdSlicing q = BwdSlicing::of(R, d, M);
    const int unit = blockIdx.x / q.S, sl = blockIdx.x % q.S, h = unit % H, b = unit / H;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = tid / q.RDw, c = tid % q.RDw, ms = q.ms(sl, M);
    const bool col = g < q.G && c < RD, kcol = col && c < R, vcol = col && c >= R;
    const int gwarps = q.RDw / 32, kwarps = R / 32;  // (SPLIT: R % 32 == 0, warps of one kind)
    T *base = ws + (size_t)unit * L.per_unit;
    const T *feat = base + L.feat;
    T *gfeat = base + L.gfeat + (size_t)sl * N * (2 * (size_t)R + d);
    const T *ckpt = base + L.ckpt + (size_t)sl * L.nck * L.sds;
    T *xbuf = base + L.xbuf + (size_t)sl * (C + 1) * L.sds;
    const size_t F = 2 * (size_t)R + d, plane = BwdSlicing::plane, eoff = 2 * plane, mine = (size_t)tid * BWD_MGT;
    const size_t base_o = ((size_t)b * N * H + h) * d, so = (size_t)H * d;
    if (tid < q.G * BWD_MGT) {  // entry gg * MGT + i: slice-local mode gg + G i
        const int ml = tid / BWD_MGT + q.G * (tid % BWD_MGT), m = sl * q.MC + ml;
        const bool ok = ml < ms;
        lam_s[0][tid] = ok ? (T)a.lambda[((size_t)h * M + m) * 2] : T(0);
        lam_s[1][tid] = ok ? (T)a.lambda[((size_t)h * M + m) * 2 + 1] : T(0);
        bv_s[0][tid] = ok ? (T)a.Bvec[((size_t)h * M + m) * 2] : T(0);
        bv_s[1][tid] = ok ? (T)a.Bvec[((size_t)h * M + m) * 2 + 1] : T(0);
    }
    __syncthreads();
    const int gm = (g < q.G ? g : 0) * BWD_MGT;  // my group's mode entries
    T yr[BWD_MGT], yi[BWD_MGT], lbr[BWD_MGT], lbi[BWD_MGT], bbr[BWD_MGT], bbi[BWD_MGT];
#pragma unroll
    for (int i = 0; i < BWD_MGT; ++i) yr[i] = yi[i] = lbr[i] = lbi[i] = bbr[i] = bbi[i] = 0;
    // eta entry of slice-local mode tid (tid < ms): its lambda / B at entry em
    const bool eown = ETA && tid < ms;
    const int em = (tid % q.G) * BWD_MGT + tid / q.G;
    T yer = 0, yei = 0, lber = 0, lbei = 0, bber = 0, bbei = 0;
    const int nsum = q.G * 4 * BWD_MGT;  // group sums per position: a (2 MGT) then abar (2 MGT) per group

    for (int k = L.nck - 1; k >= 0; --k) {
        const int t0 = k * C, len = min(C, N - t0);
        // ---- 1. forward through the chunk
        const T *ck = ckpt + (size_t)k * L.sds;
        T ur[BWD_MGT], ui[BWD_MGT];
        ldgm(ck + mine, ur);
        ldgm(ck + plane + mine, ui);
        if (ETA)
            for (int j = tid; j < len; j += NT) gds[j] = base[L.gsc + 2 * (size_t)(t0 + j) + 1];
        // my inputs of every position of the chunk, all loads issued together: s = xi(q) (key
        // column) or g / den (value column), and z
        if (col) {
            T sv[C], zv[C];
#pragma unroll
            for (int j = 0; j < C; ++j) {
                const int t = min(t0 + j, N - 1);
                const T *frow = feat + (size_t)t * F;
                zv[j] = frow[R + c];
                if (kcol) {
                    sv[j] = frow[c];
                } else {
                    const T gsn = ETA ? base[L.gsc + 2 * (size_t)t] : T(1);
                    sv[j] = (T)load_in(a.dout, a.dtype, base_o + (size_t)t * so + (c - R)) * gsn;
                }
            }
#pragma unroll
            for (int j = 0; j < C; ++j) {
                inp[(size_t)(2 * j) * NT + tid] = sv[j];
                inp[(size_t)(2 * j + 1) * NT + tid] = zv[j];
            }
        } else {
#pragma unroll
            for (int j = 0; j < C; ++j) inp[(size_t)(2 * j) * NT + tid] = inp[(size_t)(2 * j + 1) * NT + tid] = T(0);
        }
        stgm(xbuf + mine, ur);
        stgm(xbuf + plane + mine, ui);
        T er = 0, e_i = 0;
        if (eown) {
            er = ck[eoff + tid];
            e_i = ck[eoff + q.MC + tid];
            etas[tid] = er;
            etas[GM + tid] = e_i;
        }
        for (int j = 0; j < len; ++j) {
            const T s = inp[(size_t)(2 * j) * NT + tid], z = inp[(size_t)(2 * j + 1) * NT + tid];
#pragma unroll
            for (int i0 = 0; i0 < BWD_MGT; i0 += 4) {
                T lr[4], li[4], br[4], bi[4];
                lds4(&lam_s[0][gm + i0], lr);
                lds4(&lam_s[1][gm + i0], li);
                lds4(&bv_s[0][gm + i0], br);
                lds4(&bv_s[1][gm + i0], bi);
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int i = i0 + u;
                    const T nr = fma(lr[u], ur[i], fma(-li[u], ui[i], br[u] * z));
                    const T ni = fma(lr[u], ui[i], fma(li[u], ur[i], bi[u] * z));
                    ur[i] = nr;
                    ui[i] = ni;
                }
            }
            T *xb = xbuf + (size_t)(j + 1) * L.sds;
            stgm(xb + mine, ur);
            stgm(xb + plane + mine, ui);
            if (eown) {
                const T elr = lam_s[0][em], eli = lam_s[1][em], ebr = bv_s[0][em], ebi = bv_s[1][em];
                const T nr = fma(elr, er, fma(-eli, e_i, ebr)), ni = fma(elr, e_i, fma(eli, er, ebi));
                er = nr;
                e_i = ni;
                etas[(size_t)(j + 1) * 2 * GM + tid] = er;
                etas[(size_t)(j + 1) * 2 * GM + GM + tid] = e_i;
            }
            // warp sums: a_t = xi(q) . U_t over key columns, conj(Gamma_t) g over value columns
            T *rw = red + ((size_t)j * BWD_WARPS + warp) * RV;
            if constexpr (SPLIT) {
                const T sg = kcol ? s : -s;
                T v[2 * BWD_MGT];
#pragma unroll
                for (int i = 0; i < BWD_MGT; ++i) {
                    v[2 * i] = s * ur[i];
                    v[2 * i + 1] = sg * ui[i];
                }
                const T s1 = warp_reduce_scatter<2 * BWD_MGT>(v, lane);
                if ((lane & 1) == 0) rw[rs_index<2 * BWD_MGT>(lane)] = s1;
            } else {
                const T sa = kcol ? s : T(0), sb = vcol ? s : T(0);
                T v[4 * BWD_MGT];
#pragma unroll
                for (int i = 0; i < BWD_MGT; ++i) {
                    v[2 * i] = sa * ur[i];
                    v[2 * i + 1] = sa * ui[i];
                    v[2 * BWD_MGT + 2 * i] = sb * ur[i];
                    v[2 * BWD_MGT + 2 * i + 1] = -sb * ui[i];
                }
                rw[rs_index<4 * BWD_MGT>(lane)] = warp_reduce_scatter<4 * BWD_MGT>(v, lane);
            }
        }
        __syncthreads();
        // ---- 2. sums over each group's warps, every position of the chunk
        for (int e = tid; e < len * nsum; e += NT) {
            const int j = e / nsum, r = e % nsum, gg = r / (4 * BWD_MGT), kk = r % (4 * BWD_MGT);
            const int kk2 = kk - 2 * BWD_MGT;
            const T *rr = red + (size_t)j * BWD_WARPS * RV + (size_t)gg * gwarps * RV;
            T sum = 0;
            if constexpr (!SPLIT) {
                for (int w = 0; w < gwarps; ++w) sum += rr[w * RV + kk];
            } else if (kk2 < 0) {
                for (int w = 0; w < kwarps; ++w) sum += rr[w * RV + kk];
            } else {
                for (int w = kwarps; w < gwarps; ++w) sum += rr[w * RV + kk2];
            }
            if (kk2 < 0) {
                am[(size_t)(2 * j + (kk & 1)) * GM + gg * BWD_MGT + (kk >> 1)] = sum;
            } else {
                const int ml = gg + q.G * (kk2 >> 1);
                if (ETA && ml < ms) {  // + conj(eta_t) gd
                    const T ev = etas[(size_t)(j + 1) * 2 * GM + (kk2 & 1) * GM + ml];
                    sum += ((kk2 & 1) ? -ev : ev) * gds[j];
                }
                abm[(size_t)(2 * j + (kk2 & 1)) * GM + gg * BWD_MGT + (kk2 >> 1)] = sum;
            }
        }
        __syncthreads();
        // ---- 3. the adjoint, back through the chunk (ur, ui hold the chunk's last state).
        // xi(q) is zero on value columns and g on key columns, so the direct adjoint is
        // abar xi(q) on key columns and conj(a) g on value columns without a branch; modes
        // past the slice have a = abar = 0 and stay at zero.
        for (int j = len - 1; j >= 0; --j) {
            T pr[BWD_MGT], pi[BWD_MGT];  // X_{t-1}
            const T *xp = xbuf + (size_t)j * L.sds;
            ldgm(xp + mine, pr);
            ldgm(xp + plane + mine, pi);
            const T s = inp[(size_t)(2 * j) * NT + tid], zc = inp[(size_t)(2 * j + 1) * NT + tid];
            const T xq = kcol ? s : T(0), gn = vcol ? s : T(0);
            const T *amj = am + (size_t)(2 * j) * GM + gm, *abj = abm + (size_t)(2 * j) * GM + gm;
            T dz = 0, dxq = 0;
#pragma unroll
            for (int i0 = 0; i0 < BWD_MGT; i0 += 4) {
                T ar[4], aim[4], abr[4], abi[4], lr[4], li[4], br[4], bi[4];
                lds4(amj + i0, ar);
                lds4(amj + GM + i0, aim);
                lds4(abj + i0, abr);
                lds4(abj + GM + i0, abi);
                lds4(&lam_s[0][gm + i0], lr);
                lds4(&lam_s[1][gm + i0], li);
                lds4(&bv_s[0][gm + i0], br);
                lds4(&bv_s[1][gm + i0], bi);
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int i = i0 + u;
                    const T dr = fma(abr[u], xq, ar[u] * gn), di = fma(abi[u], xq, -aim[u] * gn);
                    const T nyr = fma(lr[u], yr[i], fma(li[u], yi[i], dr));
                    const T nyi = fma(lr[u], yi[i], fma(-li[u], yr[i], di));
                    yr[i] = nyr;
                    yi[i] = nyi;
                    bbr[i] = fma(zc, nyr, bbr[i]);
                    bbi[i] = fma(zc, nyi, bbi[i]);
                    dz = fma(br[u], nyr, fma(bi[u], nyi, dz));
                    dxq = fma(abr[u], ur[i], fma(abi[u], ui[i], dxq));
                }
            }
            // lambda-bar last: the only use of X_{t-1}, whose loads were issued first
#pragma unroll
            for (int i = 0; i < BWD_MGT; ++i) {
                lbr[i] = fma(pr[i], yr[i], fma(pi[i], yi[i], lbr[i]));
                lbi[i] = fma(pr[i], yi[i], fma(-pi[i], yr[i], lbi[i]));
            }
            if (eown) {
                const T ar = am[(size_t)(2 * j) * GM + em], aim = am[(size_t)(2 * j + 1) * GM + em];
                const T elr = lam_s[0][em], eli = lam_s[1][em], gd = gds[j];
                const T dr = ar * gd, di = -aim * gd;
                const T nyr = dr + elr * yer + eli * yei;
                const T nyi = di + elr * yei - eli * yer;
                yer = nyr;
                yei = nyi;
                const T per = etas[(size_t)j * 2 * GM + tid], pei = etas[(size_t)j * 2 * GM + GM + tid];
                lber += per * nyr + pei * nyi;
                lbei += per * nyi - pei * nyr;
                bber += nyr;
                bbei += nyi;
            }
            part[(size_t)(2 * j) * NT + tid] = dz;
            part[(size_t)(2 * j + 1) * NT + tid] = kcol ? dxq : T(0);
#pragma unroll
            for (int i = 0; i < BWD_MGT; ++i) {
                ur[i] = pr[i];
                ui[i] = pi[i];
            }
        }
        __syncthreads();
        // ---- 4. dz (all columns) and dxi(q) (key columns) of the chunk's positions
        for (int e = tid; e < len * RD; e += NT) {
            const int j = e / RD, cc = e % RD;
            T sz = 0, sq = 0;
            for (int gg = 0; gg < q.G; ++gg) {
                sz += part[(size_t)(2 * j) * NT + gg * q.RDw + cc];
                sq += part[(size_t)(2 * j + 1) * NT + gg * q.RDw + cc];
            }
            T *grow = gfeat + (size_t)(t0 + j) * F;
            grow[R + cc] = sz;  // dkt for cc < R, dvt for cc >= R
            if (cc < R) grow[cc] = sq;
        }
    }
    __syncthreads();
    // lambda-bar and B-bar of my modes: sum over the group's columns, then the eta terms
    T *ps = base + L.pscan;
    T *pflat = part;  // [4][NT / 4]: lambda-bar re, im, B-bar re, im per mode
#pragma unroll
    for (int i = 0; i < BWD_MGT; ++i) {  // unrolled: the per-mode sums stay in registers
        T v[4] = {lbr[i], lbi[i], bbr[i], bbi[i]};
        const T s1 = warp_reduce_scatter<4>(v, lane);
        __syncthreads();
        if ((lane & 1) == 0) fred[warp][rs_index<4>(lane)] = s1;
        __syncthreads();
        if (tid < q.G * 4) {
            const int gg = tid / 4, kk = tid % 4;
            const int ml = gg + q.G * i;
            T sum = 0;
            for (int w = 0; w < gwarps; ++w) sum += fred[gg * gwarps + w][kk];
            if (ml < ms) pflat[kk * (NT / 4) + ml] = sum;
        }
    }
    __syncthreads();
    if (tid < ms) {
        const int m = sl * q.MC + tid;
        ps[m] = pflat[0 * (NT / 4) + tid] + lber;
        ps[M + m] = pflat[1 * (NT / 4) + tid] + lbei;
        ps[2 * M + m] = pflat[2 * (NT / 4) + tid] + bber;
        ps[3 * M + m] = pflat[3 * (NT / 4) + tid] + bbei;
    }
}

// The dxi(q), dkt, dvt parts of the mode slices summed into slice 0, in slice order.
template <typename T>
__global__ void bwd_sum_slices_kernel(BackwardArgs a, T *ws, BwdLayout L) {
    const size_t F = 2 * (size_t)a.R + a.d, per = (size_t)a.N * F;
    const size_t e = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    const size_t units = (size_t)a.B * a.H;
    if (e >= units * per) return;
    const size_t unit = e / per, i = e % per;
    T *gp = ws + unit * L.per_unit + L.gfeat;
    T sum = gp[i];
    for (int s = 1; s < L.S; ++s) sum += gp[(size_t)s * per + i];
    gp[i] = sum;
}

// ---- bwd_local: RMSNorm, feature map and conv backward per position ----------------------
//
// One CTA per (unit, tile of BWD_TILE positions), one warp per position.  ds of the q and k
// convs is needed at positions [t0, t0 + tile + W - 1) for the input gradients of the tile.

template <typename T>
__global__ void __launch_bounds__(256, 4) bwd_local_kernel(BackwardArgs a, T *ws, BwdLayout L) {
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
            // conv outputs s and SiLU values f of my channels c = lane + 32 i, computed once
            T sv[BWD_LANE_CH], fv[BWD_LANE_CH];
            T ss = 0;
#pragma unroll
            for (int i = 0; i < BWD_LANE_CH; ++i) {
                const int c = lane + 32 * i;
                sv[i] = c < R ? conv_at<T>(x, a.dtype, base_qk, sqk, cw, W, t, c) : T(0);
                fv[i] = c < R ? silu(sv[i]) : T(0);
                ss = fma(fv[i], fv[i], ss);
            }
            ss = warp_sum_t(ss);
            const T n = l2 ? sqrt(ss) : ss;
            const T D = n + (T)IDA_EPS_FEAT;
            // dxi: directly (q), or through the key RMSNorm (k)
            T r = 0, sdy = 0;
            if (which == 1) {
                T ms = 0, acc = 0;
#pragma unroll
                for (int i = 0; i < BWD_LANE_CH; ++i) {
                    const T xi = fv[i] / D;
                    ms = fma(xi, xi, ms);
                }
                r = sqrt(warp_sum_t(ms) / R + (T)IDA_EPS_RMS);
#pragma unroll
                for (int i = 0; i < BWD_LANE_CH; ++i) {
                    const int c = lane + 32 * i;
                    if (c < R) {
                        const T xi = fv[i] / D;
                        const T dkt = grow[R + c];
                        acc = fma(dkt * (T)nw[c], xi, acc);
                        if (own) {
                            pnw[(size_t)warp * (R + d) + c] += dkt * xi / r;
                            pbs[(size_t)warp * (R + d) + c] += dkt;
                        }
                    }
                }
                sdy = warp_sum_t(acc);
            }
            // s = sum_c dxi[c] f[c] / D^2 term of the feature-map backward
            T dxv[BWD_LANE_CH];
            T sdf = 0;
#pragma unroll
            for (int i = 0; i < BWD_LANE_CH; ++i) {
                const int c = lane + 32 * i;
                dxv[i] = 0;
                if (c < R) {
                    const T xi = fv[i] / D;
                    dxv[i] = which == 0 ? grow[c] : (grow[R + c] * (T)nw[c]) / r - xi * sdy / ((T)R * r * r * r);
                    sdf = fma(dxv[i], fv[i], sdf);
                }
            }
            sdf = warp_sum_t(sdf);
#pragma unroll
            for (int i = 0; i < BWD_LANE_CH; ++i) {
                const int c = lane + 32 * i;
                if (c < R) {
                    const T f = fv[i];
                    // dn/df = 2 f (squared norm) or f / n (l_2 norm)
                    const T dn = l2 ? (n > T(0) ? f / n : T(0)) : T(2) * f;
                    const T df = dxv[i] / D - sdf / (D * D) * dn;
                    ds[((size_t)which * (BWD_TILE + 3) + p) * R + c] = df * silu_grad(sv[i]);
                }
            }
        }
        if (own) {
            // value RMSNorm backward (my channels j = lane + 32 i, loaded once)
            T xvv[BWD_LANE_CH];
            T ms = 0;
#pragma unroll
            for (int i = 0; i < BWD_LANE_CH; ++i) {
                const int j = lane + 32 * i;
                xvv[i] = j < d ? (T)load_in(a.v, a.dtype, base_v + (size_t)t * sv + j) : T(0);
                ms = fma(xvv[i], xvv[i], ms);
            }
            const T r = sqrt(warp_sum_t(ms) / d + (T)IDA_EPS_RMS);
            T acc = 0;
#pragma unroll
            for (int i = 0; i < BWD_LANE_CH; ++i) {
                const int j = lane + 32 * i;
                if (j < d) {
                    const T dvt = grow[2 * R + j];
                    acc = fma(dvt * (T)nw[R + j], xvv[i], acc);
                    pnw[(size_t)warp * (R + d) + R + j] += dvt * xvv[i] / r;
                    pbs[(size_t)warp * (R + d) + R + j] += dvt;
                }
            }
            acc = warp_sum_t(acc);
#pragma unroll
            for (int i = 0; i < BWD_LANE_CH; ++i) {
                const int j = lane + 32 * i;
                if (j < d) {
                    const T dvt = grow[2 * R + j];
                    const T dv = (dvt * (T)nw[R + j]) / r - xvv[i] * acc / ((T)d * r * r * r);
                    store_out(a.dv, a.dtype, base_v + (size_t)t * sv + j, (float)dv);
                }
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
static size_t bwd_local_smem(int R, int d) {
    return (2 * (size_t)(BWD_TILE + 3) * R + 2 * 8 * ((size_t)R + d)) * sizeof(T);
}

size_t backward_workspace_bytes(int B, int H, int N, int d, int R, int M, int dtype, int W, int flags) {
    if (B <= 0 || H <= 0 || N <= 0) return 0;
    const size_t e = dtype == IDA_F32 ? sizeof(double) : sizeof(float);
    const int chunk = dtype == IDA_F32 ? BwdChunk<double>::C : BwdChunk<float>::C;
    return BwdLayout::of(B, H, N, d, R, M, W, (flags & IDA_READOUT_ETA) != 0, chunk).total * e;
}

template <typename T>
static cudaError_t launch_backward_t(const BackwardArgs &a, void *workspace, cudaStream_t st) {
    const bool eta = (a.flags & IDA_READOUT_ETA) != 0;
    const BwdLayout L = BwdLayout::of(a.B, a.H, a.N, a.d, a.R, a.M, a.W, eta, BwdChunk<T>::C);
    T *ws = static_cast<T *>(workspace);
    const unsigned units = (unsigned)(a.B * a.H), tiles8 = (unsigned)((a.N + 7) / 8);
    cudaError_t e;
    bwd_features_kernel<T><<<units * tiles8, 256, 0, st>>>(a, ws, L);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if (eta)
        bwd_scan_a_kernel<T, true><<<units * (unsigned)L.S, BWD_THREADS, 0, st>>>(a, ws, L);
    else
        bwd_scan_a_kernel<T, false><<<units * (unsigned)L.S, BWD_THREADS, 0, st>>>(a, ws, L);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if (eta) {
        bwd_scan_nd_kernel<T><<<units * tiles8, 256, 0, st>>>(a, ws, L);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    {
        const bool split = a.R % 32 == 0;
        auto kb = split ? (eta ? bwd_scan_b_kernel<T, true, true> : bwd_scan_b_kernel<T, true, false>)
                        : (eta ? bwd_scan_b_kernel<T, false, true> : bwd_scan_b_kernel<T, false, false>);
        const int sb = (int)(split ? ScanBSmem<T, true>::BYTES : ScanBSmem<T, false>::BYTES);
        if ((e = cudaFuncSetAttribute(kb, cudaFuncAttributeMaxDynamicSharedMemorySize, sb)) != cudaSuccess) return e;
        kb<<<units * (unsigned)L.S, BWD_THREADS, sb, st>>>(a, ws, L);
    }
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if (L.S > 1) {
        const size_t n = (size_t)units * a.N * (2 * (size_t)a.R + a.d);
        bwd_sum_slices_kernel<T><<<(unsigned)((n + 255) / 256), 256, 0, st>>>(a, ws, L);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
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
    if (B < 0 || H < 0 || N < 0 || d < 1 || R < 1 || M < 1 || W < 1 || W > 4 || R > 256 || d > 256 || M > 128 ||
        (dtype != IDA_F32 && dtype != IDA_BF16))
        return 0;
    return ida::backward_workspace_bytes(B, H, N, d, R, M, dtype, W, flags);
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
    const size_t need = ida::backward_workspace_bytes(B, H, N, d, R, M, dtype, W, flags);
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
