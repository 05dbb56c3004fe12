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
// positions, one warp per position computes the features, then one warp per mode walks
// the tile, keeping its own partial numerators and denominators; those of all warps and
// CTAs are summed in a fixed order (through distributed shared memory across the
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

constexpr int IDL_WARPS = 16;
constexpr int IDL_THREADS = IDL_WARPS * 32;
constexpr int IDL_TILE = 8;  // positions per tile (one warp each in the feature stage)

template <typename T>
static size_t ideal_smem_bytes(int Mg, int F, int d) {
    const size_t e = sizeof(T);
    return ((size_t)Mg * (F + d) * 2 + (size_t)Mg * 2 + IDL_TILE * (size_t)F + IDL_TILE * ((size_t)F + d) +
            (size_t)IDL_WARPS * IDL_TILE * d + (size_t)IDL_WARPS * IDL_TILE) * e;
}

__device__ __forceinline__ void sincos_t(float x, float *s, float *c) { sincosf(x, s, c); }
__device__ __forceinline__ void sincos_t(double x, double *s, double *c) { sincos(x, s, c); }

// Fourier features of one row (one warp): out[i] = cos(omega_i . x) / sqrt(D),
// out[D + i] = sin(omega_i . x) / sqrt(D).
template <typename T>
__device__ __forceinline__ void fourier_row(const IdealArgs &a, const void *x, size_t xbase, const float *om,
                                            T *out, int lane) {
    const int Rin = a.Rin, D = a.D;
    const T scale = T(1) / sqrt((T)D);
    for (int i = lane; i < D; i += 32) {
        T th = 0;
        for (int c = 0; c < Rin; ++c) th = fma((T)om[(size_t)i * Rin + c], (T)load_in(x, a.dtype, xbase + c), th);
        T sn, cs;
        sincos_t(th, &sn, &cs);
        out[i] = cs * scale;
        out[D + i] = sn * scale;
    }
}

template <int NC, typename T>
__global__ void __launch_bounds__(IDL_THREADS, 1) ideal_kernel(IdealArgs a, int G, int Mg) {
    extern __shared__ __align__(16) unsigned char smem[];
    const int d = a.d, M = a.M, H = a.H, N = a.N, F = 2 * a.D, FD = F + d;
    const int rank = blockIdx.x % G, unit = blockIdx.x / G;
    const int b = unit / H, h = unit % H;
    const int m0 = rank * Mg, mcount = max(0, min(Mg, M - m0));
    T *Xr = reinterpret_cast<T *>(smem);         // [Mg][F + d]
    T *Xi = Xr + (size_t)Mg * FD;                // [Mg][F + d]
    T *etr = Xi + (size_t)Mg * FD;               // [Mg]
    T *eti = etr + Mg;                           // [Mg]
    T *xq = eti + Mg;                            // [TILE][F]
    T *z = xq + (size_t)IDL_TILE * F;            // [TILE][F + d]
    T *opart = z + (size_t)IDL_TILE * FD;        // [WARPS][TILE][d]: each mode warp's partials
    T *dpart = opart + (size_t)IDL_WARPS * IDL_TILE * d;  // [WARPS][TILE]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const size_t sqk = (size_t)H * a.Rin, sv = (size_t)H * d;
    const size_t base_qk = ((size_t)b * N * H + h) * a.Rin, base_v = ((size_t)b * N * H + h) * d;
    const float *om = a.omega + (size_t)h * a.D * a.Rin;
    for (int i = threadIdx.x; i < 2 * Mg * FD + 2 * Mg; i += IDL_THREADS) Xr[i] = T(0);
    __syncthreads();
    for (int t0 = 0; t0 < N; t0 += IDL_TILE) {
        const int tn = min(IDL_TILE, N - t0);
        // features, one warp per position; partials cleared
        if (warp < tn) {
            const int t = t0 + warp;
            fourier_row<T>(a, a.q, base_qk + (size_t)t * sqk, om, xq + (size_t)warp * F, lane);
            fourier_row<T>(a, a.k, base_qk + (size_t)t * sqk, om, z + (size_t)warp * FD, lane);
            for (int j = lane; j < d; j += 32) z[(size_t)warp * FD + F + j] = (T)load_in(a.v, a.dtype, base_v + (size_t)t * sv + j);
        }
        for (int i = threadIdx.x; i < IDL_WARPS * IDL_TILE * (d + 1); i += IDL_THREADS) opart[i] = T(0);
        __syncthreads();
        // recurrence and readout, one warp per mode; each warp keeps its own partials
        for (int ml = warp; ml < mcount; ml += IDL_WARPS) {
            const int m = m0 + ml;
            const T lr = a.lambda[((size_t)h * M + m) * 2], li = a.lambda[((size_t)h * M + m) * 2 + 1];
            const T gr = a.Bvec[((size_t)h * M + m) * 2], gi = a.Bvec[((size_t)h * M + m) * 2 + 1];
            T ur[NC], ui[NC], vr[NC], vi[NC];
#pragma unroll
            for (int i = 0; i < NC; ++i) {
                const int c = lane + 32 * i;
                ur[i] = c < F ? Xr[(size_t)ml * FD + c] : T(0);
                ui[i] = c < F ? Xi[(size_t)ml * FD + c] : T(0);
                vr[i] = c < d ? Xr[(size_t)ml * FD + F + c] : T(0);
                vi[i] = c < d ? Xi[(size_t)ml * FD + F + c] : T(0);
            }
            T er = etr[ml], ei = eti[ml];
            for (int tt = 0; tt < tn; ++tt) {
                T ar = 0, ai = 0;
#pragma unroll
                for (int i = 0; i < NC; ++i) {
                    const int c = lane + 32 * i;
                    if (c < F) {
                        cstep_t(ur[i], ui[i], lr, li, gr, gi, z[(size_t)tt * FD + c]);
                        const T xv = xq[(size_t)tt * F + c];
                        ar = fma(xv, ur[i], ar);
                        ai = fma(xv, ui[i], ai);
                    }
                    if (c < d) cstep_t(vr[i], vi[i], lr, li, gr, gi, z[(size_t)tt * FD + F + c]);
                }
                cstep_t(er, ei, lr, li, gr, gi, T(1));
                ar = warp_sum(ar);
                ai = warp_sum(ai);
#pragma unroll
                for (int i = 0; i < NC; ++i) {
                    const int j = lane + 32 * i;
                    if (j < d) opart[((size_t)warp * IDL_TILE + tt) * d + j] += ar * vr[i] - ai * vi[i];
                }
                if (lane == 0) dpart[(size_t)warp * IDL_TILE + tt] += ar * er - ai * ei;
            }
#pragma unroll
            for (int i = 0; i < NC; ++i) {
                const int c = lane + 32 * i;
                if (c < F) {
                    Xr[(size_t)ml * FD + c] = ur[i];
                    Xi[(size_t)ml * FD + c] = ui[i];
                }
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
        if (G == 1)
            __syncthreads();
        else
            cg::this_cluster().sync();
        // CTA r writes positions tt = r (mod G): sums over the cluster's CTAs and their warps,
        // in a fixed order
        for (int tt = rank + G * warp; tt < tn; tt += G * IDL_WARPS) {
            T dn = 0;
            for (int r = 0; r < G; ++r) {
                const T *pd = G == 1 ? dpart : cg::this_cluster().map_shared_rank(dpart, r);
                for (int w = 0; w < IDL_WARPS; ++w) dn += pd[(size_t)w * IDL_TILE + tt];
            }
            for (int j = lane; j < d; j += 32) {
                T o = 0;
                for (int r = 0; r < G; ++r) {
                    const T *po = G == 1 ? opart : cg::this_cluster().map_shared_rank(opart, r);
                    for (int w = 0; w < IDL_WARPS; ++w) o += po[((size_t)w * IDL_TILE + tt) * d + j];
                }
                store_out(a.out, a.dtype, base_v + (size_t)(t0 + tt) * sv + j, (float)(o / dn));
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

template <typename T>
static ida_status launch_ideal_t(const IdealArgs &a, cudaStream_t st, int num_sms, std::string &why) {
    const size_t kMaxSmem = 227 * 1024;
    const int F = 2 * a.D;
    int G = 1;
    while (G < 8 && ideal_smem_bytes<T>((a.M + G - 1) / G, F, a.d) > kMaxSmem) G *= 2;
    if (ideal_smem_bytes<T>((a.M + G - 1) / G, F, a.d) > kMaxSmem) {
        why = "state of M x (2D + d) does not fit a cluster of 8 CTAs";
        return IDA_ERR_UNSUPPORTED;
    }
    const long units = (long)a.B * a.H;
    while (G < 8 && 2 * G <= a.M && units * 2 * G <= num_sms) G *= 2;
    const int Mg = (a.M + G - 1) / G;
    const size_t smem = ideal_smem_bytes<T>(Mg, F, a.d);
    const int nc = ((F > a.d ? F : a.d) + 31) / 32;
    cudaError_t e;
    if (nc <= 1)
        e = launch_ideal_nc<1, T>(a, G, Mg, smem, st);
    else if (nc <= 2)
        e = launch_ideal_nc<2, T>(a, G, Mg, smem, st);
    else if (nc <= 4)
        e = launch_ideal_nc<4, T>(a, G, Mg, smem, st);
    else
        e = launch_ideal_nc<8, T>(a, G, Mg, smem, st);
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
