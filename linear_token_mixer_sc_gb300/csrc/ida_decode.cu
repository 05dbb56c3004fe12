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
// shared memory at the end.
#include <string>

#include "ida_common.cuh"

namespace ida {

constexpr int DEC_WARPS = 8;
constexpr int DEC_THREADS = DEC_WARPS * 32;
constexpr int DEC_UNROLL = 2;  // modes in flight per warp

// Features of one new position for one unit, one warp each (q, k, v).
// Shifts the raw conv tails of q and k in the state.
__device__ __forceinline__ void decode_prologue(const DecodeArgs &a, int unit, int h, float *st,
                                                float *xq_s, float *z_s, int warp, int lane) {
    const int R = a.R, d = a.d, W = a.W, H = a.H, M = a.M, RD = R + d;
    const float *nw = a.norm_w + (size_t)h * RD;
    const float *bs = a.bias + (size_t)h * RD;
    if (warp < 2) {
        const int which = warp;  // 0: query, 1: key
        const void *x = which == 0 ? a.q : a.k;
        const float *cw = a.conv_w + ((size_t)which * H + h) * R * W;
        float *tail = st + 2 * (size_t)M * RD + 2 * M + (size_t)which * (W - 1) * R;
        float f[8];
        float ss = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            int c = lane + 32 * i;
            f[i] = 0.f;
            if (c < R) {
                float xc = load_in(x, a.dtype, (size_t)unit * R + c);
                float s = cw[(size_t)c * W + (W - 1)] * xc;
                for (int j = 0; j < W - 1; ++j) s = fmaf(cw[(size_t)c * W + j], tail[(size_t)j * R + c], s);
                // shift: drop the oldest row, append this position (each lane owns column c)
                for (int j = 0; j + 1 < W - 1; ++j) tail[(size_t)j * R + c] = tail[(size_t)(j + 1) * R + c];
                if (W > 1) tail[(size_t)(W - 2) * R + c] = xc;
                f[i] = silu(s);
                ss = fmaf(f[i], f[i], ss);
            }
        }
        float inv = 1.f / (warp_sum(ss) + IDA_EPS_FEAT);
        if (which == 0) {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                int c = lane + 32 * i;
                if (c < R) xq_s[c] = f[i] * inv;
            }
        } else {
            float ms = 0.f;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                f[i] *= inv;
                ms = fmaf(f[i], f[i], ms);
            }
            float r = rsqrtf(warp_sum(ms) / R + IDA_EPS_RMS);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                int c = lane + 32 * i;
                if (c < R) z_s[c] = fmaf(f[i] * r, nw[c], bs[c]);
            }
        }
    } else if (warp == 2) {
        float vv[8];
        float ms = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            int j = lane + 32 * i;
            vv[i] = j < d ? load_in(a.v, a.dtype, (size_t)unit * d + j) : 0.f;
            ms = fmaf(vv[i], vv[i], ms);
        }
        float r = rsqrtf(warp_sum(ms) / d + IDA_EPS_RMS);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            int j = lane + 32 * i;
            if (j < d) z_s[R + j] = fmaf(vv[i] * r, nw[R + j], bs[R + j]);
        }
    }
}

// NV: float4 slices per lane per row half (ceil(max(R, d) / 128)).
template <int NV>
__global__ void __launch_bounds__(DEC_THREADS) decode_kernel(DecodeArgs a) {
    __shared__ __align__(16) float xq_s[256];
    __shared__ __align__(16) float z_s[512];
    __shared__ __align__(16) float ored[DEC_WARPS][256];
    __shared__ float dred[DEC_WARPS];
    const int R = a.R, d = a.d, RD = R + d, M = a.M, H = a.H;
    const int unit = blockIdx.x;
    const int h = unit % H;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    float *st = a.state + (size_t)unit * a.state_floats;
    const size_t plane = (size_t)M * RD;

    decode_prologue(a, unit, h, st, xq_s, z_s, warp, lane);
    __syncthreads();

    // Per-lane slices of xi(q) and z, reused for every mode.
    float4 xq4[NV], zk4[NV], zv4[NV];
#pragma unroll
    for (int iv = 0; iv < NV; ++iv) {
        int c = 4 * (lane + 32 * iv);
        xq4[iv] = c < R ? *reinterpret_cast<const float4 *>(xq_s + c) : make_float4(0.f, 0.f, 0.f, 0.f);
        zk4[iv] = c < R ? *reinterpret_cast<const float4 *>(z_s + c) : make_float4(0.f, 0.f, 0.f, 0.f);
        zv4[iv] = c < d ? *reinterpret_cast<const float4 *>(z_s + R + c) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    float4 oacc[NV];
#pragma unroll
    for (int iv = 0; iv < NV; ++iv) oacc[iv] = make_float4(0.f, 0.f, 0.f, 0.f);
    float dacc = 0.f;

    for (int mb = warp; mb < M; mb += DEC_WARPS * DEC_UNROLL) {
        float4 ur[DEC_UNROLL][NV], ui[DEC_UNROLL][NV], gr[DEC_UNROLL][NV], gi[DEC_UNROLL][NV];
        // issue every load of this group of modes before any arithmetic
#pragma unroll
        for (int u = 0; u < DEC_UNROLL; ++u) {
            const int m = mb + u * DEC_WARPS;
#pragma unroll
            for (int iv = 0; iv < NV; ++iv) {
                const int c = 4 * (lane + 32 * iv);
                const float4 zero = make_float4(0.f, 0.f, 0.f, 0.f);
                const bool okm = m < M;
                ur[u][iv] = okm && c < R ? __ldcs(reinterpret_cast<const float4 *>(st + (size_t)m * RD + c)) : zero;
                ui[u][iv] = okm && c < R ? __ldcs(reinterpret_cast<const float4 *>(st + plane + (size_t)m * RD + c)) : zero;
                gr[u][iv] = okm && c < d ? __ldcs(reinterpret_cast<const float4 *>(st + (size_t)m * RD + R + c)) : zero;
                gi[u][iv] = okm && c < d ? __ldcs(reinterpret_cast<const float4 *>(st + plane + (size_t)m * RD + R + c)) : zero;
            }
        }
#pragma unroll
        for (int u = 0; u < DEC_UNROLL; ++u) {
            const int m = mb + u * DEC_WARPS;
            if (m >= M) break;
            const cplx lam = {a.lambda[((size_t)h * M + m) * 2], a.lambda[((size_t)h * M + m) * 2 + 1]};
            const cplx g = {a.Bvec[((size_t)h * M + m) * 2], a.Bvec[((size_t)h * M + m) * 2 + 1]};
            float ar = 0.f, ai = 0.f;
#pragma unroll
            for (int iv = 0; iv < NV; ++iv) {
                float4 &xr = ur[u][iv], &xi = ui[u][iv];
                cstep(xr.x, xi.x, lam, g, zk4[iv].x);
                cstep(xr.y, xi.y, lam, g, zk4[iv].y);
                cstep(xr.z, xi.z, lam, g, zk4[iv].z);
                cstep(xr.w, xi.w, lam, g, zk4[iv].w);
                ar = fmaf(xq4[iv].x, xr.x, fmaf(xq4[iv].y, xr.y, fmaf(xq4[iv].z, xr.z, fmaf(xq4[iv].w, xr.w, ar))));
                ai = fmaf(xq4[iv].x, xi.x, fmaf(xq4[iv].y, xi.y, fmaf(xq4[iv].z, xi.z, fmaf(xq4[iv].w, xi.w, ai))));
                float4 &yr = gr[u][iv], &yi = gi[u][iv];
                cstep(yr.x, yi.x, lam, g, zv4[iv].x);
                cstep(yr.y, yi.y, lam, g, zv4[iv].y);
                cstep(yr.z, yi.z, lam, g, zv4[iv].z);
                cstep(yr.w, yi.w, lam, g, zv4[iv].w);
            }
            ar = warp_sum(ar);
            ai = warp_sum(ai);
#pragma unroll
            for (int iv = 0; iv < NV; ++iv) {
                const float4 yr = gr[u][iv], yi = gi[u][iv];
                oacc[iv].x += ar * yr.x - ai * yi.x;
                oacc[iv].y += ar * yr.y - ai * yi.y;
                oacc[iv].z += ar * yr.z - ai * yi.z;
                oacc[iv].w += ar * yr.w - ai * yi.w;
                const int c = 4 * (lane + 32 * iv);
                if (c < R) {
                    __stcs(reinterpret_cast<float4 *>(st + (size_t)m * RD + c), ur[u][iv]);
                    __stcs(reinterpret_cast<float4 *>(st + plane + (size_t)m * RD + c), ui[u][iv]);
                }
                if (c < d) {
                    __stcs(reinterpret_cast<float4 *>(st + (size_t)m * RD + R + c), yr);
                    __stcs(reinterpret_cast<float4 *>(st + plane + (size_t)m * RD + R + c), yi);
                }
            }
            float er = st[2 * plane + m], ei = st[2 * plane + M + m];
            cstep(er, ei, lam, g, 1.f);
            dacc += ar * er - ai * ei;
            __syncwarp();
            if (lane == 0) {
                st[2 * plane + m] = er;
                st[2 * plane + M + m] = ei;
            }
        }
    }
#pragma unroll
    for (int iv = 0; iv < NV; ++iv) {
        int c = 4 * (lane + 32 * iv);
        if (c < d) *reinterpret_cast<float4 *>(&ored[warp][c]) = oacc[iv];
    }
    if (lane == 0) dred[warp] = dacc;
    __syncthreads();
    const bool eta_ro = (a.flags & IDA_READOUT_ETA) != 0;
    float dn = 0.f;
    if (eta_ro)
        for (int w = 0; w < DEC_WARPS; ++w) dn += dred[w];
    for (int j = threadIdx.x; j < d; j += DEC_THREADS) {
        float o = 0.f;
        for (int w = 0; w < DEC_WARPS; ++w) o += ored[w][j];
        if (eta_ro) o = o / dn;
        store_out(a.out, a.dtype, (size_t)unit * d + j, o);
    }
}

ida_status launch_decode(const DecodeArgs &a, cudaStream_t st, std::string &why) {
    const int need = ((a.R > a.d ? a.R : a.d) + 127) / 128;
    const unsigned grid = (unsigned)(a.B * a.H);
    if (need <= 1)
        decode_kernel<1><<<grid, DEC_THREADS, 0, st>>>(a);
    else
        decode_kernel<2><<<grid, DEC_THREADS, 0, st>>>(a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        why = std::string("decode launch: ") + cudaGetErrorString(e);
        return IDA_ERR_CUDA;
    }
    return IDA_OK;
}

}  // namespace ida
