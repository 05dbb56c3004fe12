// ida_ideal.cu -- the ideal interdomain layer on random Fourier features.
//
// "Interdomain Attention: Beyond Token-Level Key-Value Memory" derives its layer from
// attention read as kernel regression (translated paper text, section 3.1): a finite
// feature map K(q, k) ~ xi(q)^T xi(k) (Eq. 3) turns attention into the ratio of Eq. 4,
// random Fourier features xi_omega(x) = [cos(omega^T x), sin(omega^T x)] are the
// standard instance for a stationary kernel (Eqs. 5-6), and the interdomain layer
// (Fig. 1b) compresses keys and values with an SSM recurrence into U, Gamma and eta and
// reads out F_q U^T Gamma / (F_q U^T eta).  This kernel computes that layer with D given
// frequencies per head: xi(x) = D^-1/2 [cos(Omega x); sin(Omega x)] (feature width 2D),
// X_t = lambda X_{t-1} + B [xi(k_t); v_t], eta_t = lambda eta_{t-1} + B,
// o_t = Re(xi(q_t)^T U_t^T Gamma_t) / Re(xi(q_t)^T U_t^T eta_t), with no conv and no
// normalisation (the derivation has neither).
//
// Token-sequential on the CUDA cores, the state in shared memory: one cluster of G CTAs
// per (b,h) unit splits the modes (CTA r owns modes [r Mg, (r+1) Mg)); per tile of
// positions, one warp per feature row computes the features, then one warp per mode walks
// the tile (key columns, one batched sum of a_t over the warp, value columns and eta),
// keeping its own partial numerators and denominators in registers; those of all warps
// and CTAs are summed in a fixed order (through distributed shared memory across the
// cluster), so the result is deterministic.  Arithmetic type T: double for fp32 inputs, float
// for bf16 inputs.
#include <cooperative_groups.h>

#include <string>

#include "ida_common.cuh"

namespace cg = cooperative_groups;

namespace ida {

struct IdealArgs {
    const void *q, *k, *v;
    const float *omega, *lambda, *Bvec;
    void *out;
    int B, H, N, d, Rin, D, M, dtype;
    unsigned *err;
};

constexpr int IDL_WARPS = 8;
constexpr int IDL_THREADS = IDL_WARPS * 32;

// Positions per tile: a warp keeps P positions' readout partials of its NC column slots in
// registers, so P shrinks as the columns grow.
template <int NC>
struct IdlTile {
    static constexpr int P = NC <= 2 ? 8 : (NC <= 4 ? 4 : 2);
};

// Omega of the head is staged in shared memory, transposed, when it takes at most this much.
constexpr size_t IDL_OMEGA_STAGE = 48 * 1024;

template <typename T>
static size_t ideal_smem_bytes(int Mg, int F, int d, int P, int Rin, size_t omega_bytes) {
    const size_t e = sizeof(T);
    return ((size_t)Mg * (F + d) * 2 + (size_t)Mg * 2 + (size_t)P * F + (size_t)P * ((size_t)F + d) +
            (size_t)IDL_WARPS * P * d + (size_t)IDL_WARPS * P + (size_t)IDL_WARPS * 2 * P + 2 * (size_t)P * Rin) * e +
           omega_bytes;
}

__device__ __forceinline__ void sincos_t(float x, float *s, float *c) { sincosf(x, s, c); }
__device__ __forceinline__ void sincos_t(double x, double *s, double *c) { sincos(x, s, c); }

// Fourier features of one row x (one warp, x in shared memory): out[i] = cos(omega_i . x) /
// sqrt(D), out[D + i] = sin(omega_i . x) / sqrt(D); omega_i[c] at om[i si + c sc] (si = 1,
// sc = D for the transposed shared-memory copy: lanes then read consecutive words).
template <typename T>
__device__ __forceinline__ void fourier_row(const IdealArgs &a, const T *x, const float *om, int si, int sc, T *out,
                                            int lane) {
    const int Rin = a.Rin, D = a.D;
    const T scale = T(1) / sqrt((T)D);
    for (int i = lane; i < D; i += 32) {
        T th = 0;
        const float *o = om + (size_t)i * si;
#pragma unroll 8
        for (int c = 0; c < Rin; ++c) th = fma((T)o[(size_t)c * sc], x[c], th);
        T sn, cs;
        sincos_t(th, &sn, &cs);
        out[i] = cs * scale;
        out[D + i] = sn * scale;
    }
}

// One cluster of G CTAs per (b,h) unit; CTA r owns modes [r Mg, (r+1) Mg), its warps take
// them in turn.  Per tile of P positions: the features of the tile's rows; then per mode,
// (1) the key-column recurrence and each lane's parts of a_t for the P positions, (2) one
// reduce-scatter of those 2P values over the warp (instead of two full warp sums per
// position), (3) the value-column recurrence, eta, and the readout parts o_t, den_t kept in
// registers over the warp's modes; the parts of all warps and CTAs are summed in a fixed
// order (deterministic).
template <int NC, typename T>
__global__ void __launch_bounds__(IDL_THREADS) ideal_kernel(IdealArgs a, int G, int Mg) {
    constexpr int P = IdlTile<NC>::P, NV = 2 * P;
    extern __shared__ __align__(16) unsigned char smem[];
    const int d = a.d, M = a.M, H = a.H, N = a.N, F = 2 * a.D, FD = F + d;
    const int rank = blockIdx.x % G, unit = blockIdx.x / G;
    const int b = unit / H, h = unit % H;
    const int m0 = rank * Mg, mcount = max(0, min(Mg, M - m0));
    T *Xr = reinterpret_cast<T *>(smem);         // [Mg][F + d]
    T *Xi = Xr + (size_t)Mg * FD;                // [Mg][F + d]
    T *etr = Xi + (size_t)Mg * FD;               // [Mg]
    T *eti = etr + Mg;                           // [Mg]
    T *xq = eti + Mg;                            // [P][F]
    T *z = xq + (size_t)P * F;                   // [P][F + d]
    T *opart = z + (size_t)P * FD;               // [WARPS][P][d]: each warp's partials
    T *dpart = opart + (size_t)IDL_WARPS * P * d;  // [WARPS][P]
    T *abuf = dpart + (size_t)IDL_WARPS * P;     // [WARPS][2P]: a_t of the warp's current mode
    T *xrows = abuf + (size_t)IDL_WARPS * 2 * P;  // [2][P][Rin]: the tile's q and k rows
    float *oms = reinterpret_cast<float *>(xrows + 2 * (size_t)P * a.Rin);  // [Rin][D] omega^T, if staged
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const size_t sqk = (size_t)H * a.Rin, sv = (size_t)H * d;
    const size_t base_qk = ((size_t)b * N * H + h) * a.Rin, base_v = ((size_t)b * N * H + h) * d;
    const float *omg = a.omega + (size_t)h * a.D * a.Rin;
    const bool staged = (size_t)a.D * a.Rin * sizeof(float) <= IDL_OMEGA_STAGE;
    for (int i = threadIdx.x; i < 2 * Mg * FD + 2 * Mg; i += IDL_THREADS) Xr[i] = T(0);
    if (staged)
        for (int e = threadIdx.x; e < a.D * a.Rin; e += IDL_THREADS) {
            const int i = e / a.Rin, c = e % a.Rin;
            oms[(size_t)c * a.D + i] = omg[e];
        }
    const float *om = staged ? oms : omg;
    const int om_si = staged ? 1 : a.Rin, om_sc = staged ? a.D : 1;
    __syncthreads();
    for (int t0 = 0; t0 < N; t0 += P) {
        const int tn = min(P, N - t0);
        // the tile's q and k rows, then the features: rows 0 .. tn-1 are xi(q), rows
        // tn .. 2 tn - 1 are [xi(k); v]
        for (int e = threadIdx.x; e < 2 * tn * a.Rin; e += IDL_THREADS) {
            const int which = e / (tn * a.Rin), p = (e / a.Rin) % tn, c = e % a.Rin;
            xrows[((size_t)which * P + p) * a.Rin + c] =
                (T)load_in(which == 0 ? a.q : a.k, a.dtype, base_qk + (size_t)(t0 + p) * sqk + c);
        }
        __syncthreads();
        for (int r = warp; r < 2 * tn; r += IDL_WARPS) {
            const int p = r < tn ? r : r - tn, t = t0 + p;
            if (r < tn) {
                fourier_row<T>(a, xrows + (size_t)p * a.Rin, om, om_si, om_sc, xq + (size_t)p * F, lane);
            } else {
                fourier_row<T>(a, xrows + ((size_t)P + p) * a.Rin, om, om_si, om_sc, z + (size_t)p * FD, lane);
                for (int j = lane; j < d; j += 32)
                    z[(size_t)p * FD + F + j] = (T)load_in(a.v, a.dtype, base_v + (size_t)t * sv + j);
            }
        }
        __syncthreads();
        T op[P][NC], dn[P];
#pragma unroll
        for (int tt = 0; tt < P; ++tt) {
            dn[tt] = 0;
#pragma unroll
            for (int i = 0; i < NC; ++i) op[tt][i] = 0;
        }
        for (int ml = warp; ml < mcount; ml += IDL_WARPS) {
            const int m = m0 + ml;
            const T lr = a.lambda[((size_t)h * M + m) * 2], li = a.lambda[((size_t)h * M + m) * 2 + 1];
            const T gr = a.Bvec[((size_t)h * M + m) * 2], gi = a.Bvec[((size_t)h * M + m) * 2 + 1];
            // (1) key columns: U_t and my parts of a_t = xi(q_t) . U_t
            T pa[NV];
            {
                T ur[NC], ui[NC];
#pragma unroll
                for (int i = 0; i < NC; ++i) {
                    const int c = lane + 32 * i;
                    ur[i] = c < F ? Xr[(size_t)ml * FD + c] : T(0);
                    ui[i] = c < F ? Xi[(size_t)ml * FD + c] : T(0);
                }
#pragma unroll
                for (int tt = 0; tt < P; ++tt) {
                    T ar = 0, ai = 0;
                    if (tt < tn) {
#pragma unroll
                        for (int i = 0; i < NC; ++i) {
                            const int c = lane + 32 * i;
                            if (c < F) {
                                cstep_t(ur[i], ui[i], lr, li, gr, gi, z[(size_t)tt * FD + c]);
                                const T xv = xq[(size_t)tt * F + c];
                                ar = fma(xv, ur[i], ar);
                                ai = fma(xv, ui[i], ai);
                            }
                        }
                    }
                    pa[2 * tt] = ar;
                    pa[2 * tt + 1] = ai;
                }
#pragma unroll
                for (int i = 0; i < NC; ++i) {
                    const int c = lane + 32 * i;
                    if (c < F) {
                        Xr[(size_t)ml * FD + c] = ur[i];
                        Xi[(size_t)ml * FD + c] = ui[i];
                    }
                }
            }
            // (2) a_t of the tile's positions: one reduce-scatter, then read back by every lane
            {
                const T s1 = warp_reduce_scatter<NV>(pa, lane);
                if ((lane & (32 / NV - 1)) == 0) abuf[(size_t)warp * NV + rs_index<NV>(lane)] = s1;
                __syncwarp();
#pragma unroll
                for (int k = 0; k < NV; ++k) pa[k] = abuf[(size_t)warp * NV + k];
                __syncwarp();
            }
            // (3) value columns and eta: Gamma_t, eta_t, and the readout parts
            {
                T vr[NC], vi[NC];
#pragma unroll
                for (int i = 0; i < NC; ++i) {
                    const int c = lane + 32 * i;
                    vr[i] = c < d ? Xr[(size_t)ml * FD + F + c] : T(0);
                    vi[i] = c < d ? Xi[(size_t)ml * FD + F + c] : T(0);
                }
                T er = etr[ml], ei = eti[ml];
#pragma unroll
                for (int tt = 0; tt < P; ++tt) {
                    if (tt < tn) {
                        const T ar = pa[2 * tt], ai = pa[2 * tt + 1];
#pragma unroll
                        for (int i = 0; i < NC; ++i) {
                            const int c = lane + 32 * i;
                            if (c < d) {
                                cstep_t(vr[i], vi[i], lr, li, gr, gi, z[(size_t)tt * FD + F + c]);
                                op[tt][i] += ar * vr[i] - ai * vi[i];
                            }
                        }
                        cstep_t(er, ei, lr, li, gr, gi, T(1));
                        dn[tt] += ar * er - ai * ei;
                    }
                }
#pragma unroll
                for (int i = 0; i < NC; ++i) {
                    const int c = lane + 32 * i;
                    if (c < d) {
                        Xr[(size_t)ml * FD + F + c] = vr[i];
                        Xi[(size_t)ml * FD + F + c] = vi[i];
                    }
                }
                if (lane == 0) {
                    etr[ml] = er;
                    eti[ml] = ei;
                }
            }
        }
#pragma unroll
        for (int tt = 0; tt < P; ++tt) {
#pragma unroll
            for (int i = 0; i < NC; ++i) {
                const int j = lane + 32 * i;
                if (j < d) opart[((size_t)warp * P + tt) * d + j] = op[tt][i];
            }
            if (lane == 0) dpart[(size_t)warp * P + tt] = dn[tt];
        }
        if (G == 1)
            __syncthreads();
        else
            cg::this_cluster().sync();
        // CTA r writes positions tt = r (mod G): sums over the cluster's CTAs and their warps,
        // in a fixed order
        for (int tt = rank + G * warp; tt < tn; tt += G * IDL_WARPS) {
            T den = 0;
            for (int r = 0; r < G; ++r) {
                const T *pd = G == 1 ? dpart : cg::this_cluster().map_shared_rank(dpart, r);
                for (int w = 0; w < IDL_WARPS; ++w) den += pd[(size_t)w * P + tt];
            }
            for (int j = lane; j < d; j += 32) {
                T o = 0;
                for (int r = 0; r < G; ++r) {
                    const T *po = G == 1 ? opart : cg::this_cluster().map_shared_rank(opart, r);
                    for (int w = 0; w < IDL_WARPS; ++w) o += po[((size_t)w * P + tt) * d + j];
                }
                store_out(a.out, a.dtype, base_v + (size_t)(t0 + tt) * sv + j, (float)(o / den));
            }
        }
        if (G == 1)
            __syncthreads();
        else
            cg::this_cluster().sync();
    }
}

template <int NC, typename T>
static cudaError_t launch_ideal_nc(const IdealArgs &a, int G, int Mg, size_t smem, cudaStream_t st) {
    auto kern = ideal_kernel<NC, T>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)G * (unsigned)(a.B * a.H), 1, 1);
    cfg.blockDim = dim3(IDL_THREADS, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)G;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, a, G, Mg);
}

template <int NC, typename T>
static cudaError_t launch_ideal_p(const IdealArgs &a, int num_sms, std::string &why, cudaStream_t st, bool &fits) {
    // G CTAs per unit (a cluster) split the modes: at least as many as the state's shared
    // memory needs, then the most (up to 8, two modes or more each) whose clusters still fit
    // one wave of two CTAs per SM.  Any G works (the last CTA's mode range may be short): at
    // 96 units on 152 SMs, G = 3 timed 3.98 ms against 4.51 ms for G = 2 and 6.35 ms for G = 4
    constexpr int P = IdlTile<NC>::P;
    const size_t kMaxSmem = 227 * 1024;
    const int F = 2 * a.D;
    const size_t omb = (size_t)a.D * a.Rin * sizeof(float);
    const size_t om_stage = omb <= IDL_OMEGA_STAGE ? omb : 0;
    int G = 1;
    while (G < 8 && ideal_smem_bytes<T>((a.M + G - 1) / G, F, a.d, P, a.Rin, om_stage) > kMaxSmem) G *= 2;
    fits = ideal_smem_bytes<T>((a.M + G - 1) / G, F, a.d, P, a.Rin, om_stage) <= kMaxSmem;
    if (!fits) return cudaSuccess;
    const long units = (long)a.B * a.H;
    for (int g = G + 1; g <= 8 && 2 * g <= a.M; ++g)
        if (units * g <= 2L * num_sms) G = g;
    const int Mg = (a.M + G - 1) / G;
    return launch_ideal_nc<NC, T>(a, G, Mg, ideal_smem_bytes<T>(Mg, F, a.d, P, a.Rin, om_stage), st);
}

template <typename T>
static ida_status launch_ideal_t(const IdealArgs &a, cudaStream_t st, int num_sms, std::string &why) {
    const int F = 2 * a.D;
    const int nc = ((F > a.d ? F : a.d) + 31) / 32;
    bool fits = true;
    cudaError_t e;
    if (nc <= 1)
        e = launch_ideal_p<1, T>(a, num_sms, why, st, fits);
    else if (nc <= 2)
        e = launch_ideal_p<2, T>(a, num_sms, why, st, fits);
    else if (nc <= 4)
        e = launch_ideal_p<4, T>(a, num_sms, why, st, fits);
    else
        e = launch_ideal_p<8, T>(a, num_sms, why, st, fits);
    if (!fits) {
        why = "state of M x (2D + d) does not fit a cluster of 8 CTAs";
        return IDA_ERR_UNSUPPORTED;
    }
    if (e != cudaSuccess) {
        why = std::string("ideal-layer launch: ") + cudaGetErrorString(e);
        return IDA_ERR_CUDA;
    }
    return IDA_OK;
}

ida_status fail_with(ida_status s, const std::string &why);
ida_status device_error_word(unsigned **err, std::string &why);
ida_status check_call(int d, int R, int M, int W, int dtype, int flags, int *num_sms, std::string &why);

}  // namespace ida

extern "C" ida_status ida_forward_ideal(const void *q, const void *k, const void *v, const float *omega,
                                        const float *lambda, const float *Bvec, void *out, int B, int H, int N,
                                        int d, int R_in, int D, int M, int dtype, ida_stream_t stream) {
    std::string why;
    if (B < 0 || H < 0 || N < 0) return ida::fail_with(IDA_ERR_ARG, "B, H and N must be >= 0");
    if (R_in < 1 || D < 1 || d < 1 || M < 1) return ida::fail_with(IDA_ERR_ARG, "R_in, D, d and M must be >= 1");
    if (dtype != IDA_F32 && dtype != IDA_BF16) return ida::fail_with(IDA_ERR_ARG, "dtype must be IDA_F32 or IDA_BF16");
    if (R_in > 256 || D > 128 || d > 256 || M > 128)
        return ida::fail_with(IDA_ERR_UNSUPPORTED, "supported: R_in <= 256, D <= 128, d <= 256, M <= 128");
    if ((long long)B * H > (1LL << 24)) return ida::fail_with(IDA_ERR_UNSUPPORTED, "B*H above 2^24");
    if ((long long)B * H == 0 || N == 0) return IDA_OK;
    const void *ptrs[] = {q, k, v, omega, lambda, Bvec, out};
    for (const void *p : ptrs)
        if (!p) return ida::fail_with(IDA_ERR_ARG, "null pointer");
    for (const void *p : ptrs)
        if ((reinterpret_cast<uintptr_t>(p) & 15u) != 0)
            return ida::fail_with(IDA_ERR_ARG, "pointers must be 16-byte aligned");
    int num_sms = 0;
    ida_status s = ida::check_call(8, 8, 1, 1, dtype, 0, &num_sms, why);  // device set-up, pending errors
    if (s != IDA_OK) return ida::fail_with(s, why);
    unsigned *err = nullptr;
    s = ida::device_error_word(&err, why);
    if (s != IDA_OK) return ida::fail_with(s, why);
    ida::IdealArgs a;
    a.q = q; a.k = k; a.v = v; a.omega = omega; a.lambda = lambda; a.Bvec = Bvec; a.out = out;
    a.B = B; a.H = H; a.N = N; a.d = d; a.Rin = R_in; a.D = D; a.M = M; a.dtype = dtype; a.err = err;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    s = dtype == IDA_F32 ? ida::launch_ideal_t<double>(a, st, num_sms, why) : ida::launch_ideal_t<float>(a, st, num_sms, why);
    return s == IDA_OK ? IDA_OK : ida::fail_with(s, why);
}
