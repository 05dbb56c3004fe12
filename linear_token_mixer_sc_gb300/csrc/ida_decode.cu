// ida_decode.cu -- one recurrent decode step of the mixer.
//
// "Interdomain Attention: Beyond Token-Level Key-Value Memory" keeps a
// fixed-size state that is updated in O(1) per step (paper text, Sec. 1;
// German technical summary, "Problemstellung" and "Skalierbare
// Implementierung").  One step is: shift the conv tails, compute xi(q),
// kt, vt for the new position, then for every mode m update
// X[m] <- lambda_m X[m] + B_m [kt ; vt], form a[m] = xi(q) . U[m] and
// accumulate o += Re(a[m] Gamma[m]) (and den += Re(a[m] eta[m])).
//
// The step is bound by HBM: the fp32 complex state (2M(R+d) floats per unit,
// 262 KB at M=64, R=d=128) is read and written exactly once, in 128-bit
// coalesced accesses.  One CTA per (b,h) unit; each warp owns a strided set
// of modes, lanes own 4-float column slices, the per-mode dot product is a
// warp-shuffle reduction and the per-warp partial outputs are summed through
// shared memory at the end.  lambda, B and eta of a warp's modes are read once,
// one mode per lane, and broadcast by shuffles, so no mode waits on a load
// issued after the previous mode's stores.  Arithmetic is fp64 for fp32 inputs (see the
// sequential prefill for why) and fp32 for bf16 inputs; the state is stored
// as fp32 either way.
#include <string>

#include "ida_common.cuh"

namespace ida {

constexpr int DEC_WARPS = 4;
constexpr int DEC_THREADS = DEC_WARPS * 32;
constexpr int DEC_UNROLL = 1;  // modes per load group (two groups in flight per warp)

// Features of one new position for one unit, one warp each (q, k, v); a lane handles
// channels lane + 32 i, i < 4 NV (R, d <= 128 NV).  Shifts the raw conv tails of q and k in
// the state.
template <int NV, typename T>
__device__ __forceinline__ void decode_prologue(const DecodeArgs &a, int unit, int h, float *st,
                                                T *xq_s, T *z_s, int warp, int lane) {
    const int R = a.R, d = a.d, W = a.W, H = a.H, M = a.M, RD = R + d;
    const float *nw = a.norm_w + (size_t)h * RD;
    const float *bs = a.bias + (size_t)h * RD;
    if (warp < 2) {
        const int which = warp;  // 0: query, 1: key
        const void *x = which == 0 ? a.q : a.k;
        const float *cw = a.conv_w + ((size_t)which * H + h) * R * W;
        float *tail = st + 2 * (size_t)M * RD + 2 * M + (size_t)which * (W - 1) * R;
        T f[4 * NV];
        T ss = 0;
#pragma unroll
        for (int i = 0; i < 4 * NV; ++i) {
            int c = lane + 32 * i;
            f[i] = 0;
            if (c < R) {
                float xc = load_in(x, a.dtype, (size_t)unit * R + c);
                T s = (T)cw[(size_t)c * W + (W - 1)] * (T)xc;
                for (int j = 0; j < W - 1; ++j) s = fma((T)cw[(size_t)c * W + j], (T)tail[(size_t)j * R + c], s);
                // shift: drop the oldest row, append this position (each lane owns column c)
                for (int j = 0; j + 1 < W - 1; ++j) tail[(size_t)j * R + c] = tail[(size_t)(j + 1) * R + c];
                if (W > 1) tail[(size_t)(W - 2) * R + c] = xc;
                f[i] = silu(s);
                ss = fma(f[i], f[i], ss);
            }
        }
        T nrm = warp_sum(ss);  // squared norm, or its square root for the l_2 reading
        if (a.flags & IDA_FEAT_L2) nrm = sqrt(nrm);
        T inv = T(1) / (nrm + (T)IDA_EPS_FEAT);
        if (which == 0) {
#pragma unroll
            for (int i = 0; i < 4 * NV; ++i) {
                int c = lane + 32 * i;
                if (c < R) xq_s[c] = f[i] * inv;
            }
        } else {
            T ms = 0;
#pragma unroll
            for (int i = 0; i < 4 * NV; ++i) {
                f[i] *= inv;
                ms = fma(f[i], f[i], ms);
            }
            T r = rsqrt_t(warp_sum(ms) / R + (T)IDA_EPS_RMS);
#pragma unroll
            for (int i = 0; i < 4 * NV; ++i) {
                int c = lane + 32 * i;
                if (c < R) z_s[c] = fma(f[i] * r, (T)nw[c], (T)bs[c]);
            }
        }
    } else if (warp == 2) {
        T vv[4 * NV];
        T ms = 0;
#pragma unroll
        for (int i = 0; i < 4 * NV; ++i) {
            int j = lane + 32 * i;
            vv[i] = j < d ? (T)load_in(a.v, a.dtype, (size_t)unit * d + j) : T(0);
            ms = fma(vv[i], vv[i], ms);
        }
        T r = rsqrt_t(warp_sum(ms) / d + (T)IDA_EPS_RMS);
#pragma unroll
        for (int i = 0; i < 4 * NV; ++i) {
            int j = lane + 32 * i;
            if (j < d) z_s[R + j] = fma(vv[i] * r, (T)nw[R + j], (T)bs[R + j]);
        }
    }
}

__device__ __forceinline__ float4 ld_state(const float *p) {
    return __ldcs(reinterpret_cast<const float4 *>(p));
}

template <typename T>
__device__ __forceinline__ void st_state(float *p, const T v[4]) {
    __stcs(reinterpret_cast<float4 *>(p), make_float4((float)v[0], (float)v[1], (float)v[2], (float)v[3]));
}

template <typename T>
__device__ __forceinline__ void unpack4(float4 f, T v[4]) {
    v[0] = f.x;
    v[1] = f.y;
    v[2] = f.z;
    v[3] = f.w;
}

// State slices of DEC_UNROLL modes of one warp: [mode][plane: Re U, Im U, Re G, Im G][slice].
template <int NV>
struct ModeGroup {
    float4 v[DEC_UNROLL][4][NV];
};

template <int NV>
__device__ __forceinline__ void load_group(ModeGroup<NV> &g, const float *st, int mb, int M, int R, int d,
                                           int RD, size_t plane, int lane) {
#pragma unroll
    for (int u = 0; u < DEC_UNROLL; ++u) {
        const int m = mb + u * DEC_WARPS;
#pragma unroll
        for (int iv = 0; iv < NV; ++iv) {
            const int c = 4 * (lane + 32 * iv);
            const float4 zero = make_float4(0.f, 0.f, 0.f, 0.f);
            const bool okm = m < M;
            g.v[u][0][iv] = okm && c < R ? ld_state(st + (size_t)m * RD + c) : zero;
            g.v[u][1][iv] = okm && c < R ? ld_state(st + plane + (size_t)m * RD + c) : zero;
            g.v[u][2][iv] = okm && c < d ? ld_state(st + (size_t)m * RD + R + c) : zero;
            g.v[u][3][iv] = okm && c < d ? ld_state(st + plane + (size_t)m * RD + R + c) : zero;
        }
    }
}

// lambda, B and eta of the warp's modes, one mode per lane: lane i holds mode warp + DEC_WARPS i
// (at most 32 modes per warp since M <= 128)
template <typename T>
struct ModeRegs {
    T lr, li, br, bi, er, ei;
};

// Update the group's modes, store them, accumulate the readout.
template <int NV, typename T>
__device__ __forceinline__ void step_group(const ModeGroup<NV> &g, float *st, int mb, const DecodeArgs &a,
                                           int warp, int RD, size_t plane, int lane, const T (&xq)[NV][4],
                                           const T (&zk)[NV][4], const T (&zv)[NV][4], T (&oacc)[NV][4],
                                           T &dacc, ModeRegs<T> &mr) {
    const int M = a.M, R = a.R, d = a.d;
#pragma unroll
    for (int u = 0; u < DEC_UNROLL; ++u) {
        const int m = mb + u * DEC_WARPS;
        if (m >= M) break;
        const int mi = (m - warp) / DEC_WARPS;  // the lane holding this mode's parameters
        const T lr = __shfl_sync(0xffffffffu, mr.lr, mi), li = __shfl_sync(0xffffffffu, mr.li, mi);
        const T br = __shfl_sync(0xffffffffu, mr.br, mi), bi = __shfl_sync(0xffffffffu, mr.bi, mi);
        T ar = 0, ai = 0;
        T yr[NV][4], yi[NV][4];
#pragma unroll
        for (int iv = 0; iv < NV; ++iv) {
            const int c = 4 * (lane + 32 * iv);
            T xr[4], xi[4];
            unpack4(g.v[u][0][iv], xr);
            unpack4(g.v[u][1][iv], xi);
            unpack4(g.v[u][2][iv], yr[iv]);
            unpack4(g.v[u][3][iv], yi[iv]);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                cstep_t(xr[e], xi[e], lr, li, br, bi, zk[iv][e]);
                ar = fma(xq[iv][e], xr[e], ar);
                ai = fma(xq[iv][e], xi[e], ai);
                cstep_t(yr[iv][e], yi[iv][e], lr, li, br, bi, zv[iv][e]);
            }
            if (c < R) {
                st_state(st + (size_t)m * RD + c, xr);
                st_state(st + plane + (size_t)m * RD + c, xi);
            }
            if (c < d) {
                st_state(st + (size_t)m * RD + R + c, yr[iv]);
                st_state(st + plane + (size_t)m * RD + R + c, yi[iv]);
            }
        }
        ar = warp_sum(ar);
        ai = warp_sum(ai);
#pragma unroll
        for (int iv = 0; iv < NV; ++iv)
#pragma unroll
            for (int e = 0; e < 4; ++e) oacc[iv][e] += ar * yr[iv][e] - ai * yi[iv][e];
        T er = __shfl_sync(0xffffffffu, mr.er, mi), ei = __shfl_sync(0xffffffffu, mr.ei, mi);
        cstep_t(er, ei, lr, li, br, bi, T(1));
        dacc += ar * er - ai * ei;
        if (lane == mi) {
            mr.er = er;
            mr.ei = ei;
        }
    }
}

// NV: float4 slices per lane per row half (ceil(max(R, d) / 128)).
// T: arithmetic type (double for fp32 inputs, float for bf16 inputs); the
// state itself is always stored as fp32.  The state loads of a warp's first
// mode group are issued before the feature prologue, and every later group
// is loaded while the previous one is being updated, so that each warp keeps
// its next loads in flight through the arithmetic.
template <int NV, typename T>
__global__ void __launch_bounds__(DEC_THREADS, 3) decode_kernel(DecodeArgs a) {
    __shared__ __align__(16) T xq_s[256];
    __shared__ __align__(16) T z_s[512];
    __shared__ __align__(16) T ored[DEC_WARPS][256];
    __shared__ T dred[DEC_WARPS];
    const int R = a.R, d = a.d, RD = R + d, M = a.M, H = a.H;
    const int unit = blockIdx.x;
    const int h = unit % H;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    float *st = a.state + (size_t)unit * a.state_floats;
    const size_t plane = (size_t)M * RD;
    constexpr int STRIDE = DEC_WARPS * DEC_UNROLL;  // modes between a warp's consecutive groups

    ModeGroup<NV> ga, gb;
    load_group(ga, st, warp, M, R, d, RD, plane, lane);
    ModeRegs<T> mr = {T(0), T(0), T(0), T(0), T(0), T(0)};
    const int mlane = warp + DEC_WARPS * lane;  // this lane's mode
    if (mlane < M) {
        const float2 lam = *reinterpret_cast<const float2 *>(a.lambda + ((size_t)h * M + mlane) * 2);
        const float2 bb = *reinterpret_cast<const float2 *>(a.Bvec + ((size_t)h * M + mlane) * 2);
        mr = {(T)lam.x, (T)lam.y, (T)bb.x, (T)bb.y, (T)st[2 * plane + mlane], (T)st[2 * plane + M + mlane]};
    }

    decode_prologue<NV, T>(a, unit, h, st, xq_s, z_s, warp, lane);
    __syncthreads();

    // Per-lane slices of xi(q) and z, reused for every mode.
    T xq[NV][4], zk[NV][4], zv[NV][4], oacc[NV][4];
#pragma unroll
    for (int iv = 0; iv < NV; ++iv) {
        const int c = 4 * (lane + 32 * iv);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            xq[iv][e] = c < R ? xq_s[c + e] : T(0);
            zk[iv][e] = c < R ? z_s[c + e] : T(0);
            zv[iv][e] = c < d ? z_s[R + c + e] : T(0);
            oacc[iv][e] = T(0);
        }
    }
    T dacc = 0;

    for (int mb = warp; mb < M; mb += 2 * STRIDE) {
        if (mb + STRIDE < M) load_group(gb, st, mb + STRIDE, M, R, d, RD, plane, lane);
        step_group<NV, T>(ga, st, mb, a, warp, RD, plane, lane, xq, zk, zv, oacc, dacc, mr);
        if (mb + STRIDE >= M) break;
        if (mb + 2 * STRIDE < M) load_group(ga, st, mb + 2 * STRIDE, M, R, d, RD, plane, lane);
        step_group<NV, T>(gb, st, mb + STRIDE, a, warp, RD, plane, lane, xq, zk, zv, oacc, dacc, mr);
    }
#pragma unroll
    for (int iv = 0; iv < NV; ++iv) {
        const int c = 4 * (lane + 32 * iv);
        if (c < d)
#pragma unroll
            for (int e = 0; e < 4; ++e) ored[warp][c + e] = oacc[iv][e];
    }
    if (lane == 0) dred[warp] = dacc;
    if (mlane < M) {
        st[2 * plane + mlane] = (float)mr.er;
        st[2 * plane + M + mlane] = (float)mr.ei;
    }
    __syncthreads();
    const bool eta_ro = (a.flags & IDA_READOUT_ETA) != 0;
    T dn = 0;
    if (eta_ro)
        for (int w = 0; w < DEC_WARPS; ++w) dn += dred[w];
    for (int j = threadIdx.x; j < d; j += DEC_THREADS) {
        T o = 0;
        for (int w = 0; w < DEC_WARPS; ++w) o += ored[w][j];
        if (eta_ro) o = o / dn;
        store_out(a.out, a.dtype, (size_t)unit * d + j, (float)o);
    }
}

ida_status launch_decode(const DecodeArgs &a, cudaStream_t st, std::string &why) {
    const int need = ((a.R > a.d ? a.R : a.d) + 127) / 128;
    const unsigned grid = (unsigned)(a.B * a.H);
    if (a.dtype == IDA_F32) {
        if (need <= 1)
            decode_kernel<1, double><<<grid, DEC_THREADS, 0, st>>>(a);
        else
            decode_kernel<2, double><<<grid, DEC_THREADS, 0, st>>>(a);
    } else {
        if (need <= 1)
            decode_kernel<1, float><<<grid, DEC_THREADS, 0, st>>>(a);
        else
            decode_kernel<2, float><<<grid, DEC_THREADS, 0, st>>>(a);
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        why = std::string("decode launch: ") + cudaGetErrorString(e);
        return IDA_ERR_CUDA;
    }
    return IDA_OK;
}

}  // namespace ida
