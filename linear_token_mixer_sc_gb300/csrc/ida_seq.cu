// ida_seq.cu -- token-sequential prefill on CUDA cores.
//
// This is the exact-arithmetic path of the mixer ("Interdomain Attention:
// Beyond Token-Level Key-Value Memory", German technical summary,
// "Skalierbare Implementierung"): it walks the recurrence X_t = lambda X_{t-1}
// + B z_t one position at a time, reads out a_t = xi(q_t) U_t^T and
// o_t = Re(a_t Gamma_t) after every step, and keeps the whole complex state in
// shared memory.  It serves fp32 inputs (where tensor-core rounding would
// break a 1e-5 relative tolerance) and any shape the chunked tensor-core
// kernel does not take.
//
// Work split: one thread-block cluster of G CTAs per (b,h) unit.  The M
// modes are independent in the recurrence, so CTA r of the cluster owns modes
// [r*Mg, (r+1)*Mg) and produces a partial readout over them; the G partials
// of each position are summed through distributed shared memory.  Positions
// are processed in tiles of seq_tile<T>(): the prologue (conv, SiLU feature map,
// RMSNorm) of a tile runs one warp per position, the positions dealt over the
// cluster's CTAs, each storing its rows into every CTA; then every warp walks the
// tile's positions for its modes with the mode's state row in registers.
//
// Arithmetic type T: double for fp32 inputs, float for bf16 inputs.  With
// fp32 inputs the outputs of the synthetic workloads reach |o| ~ 1e4 and the
// eta denominator comes within 1e-2 of zero, so an fp32 recurrence cannot
// hold a 1e-4 absolute error; the fp32 path therefore keeps its state and
// sums in fp64 and rounds once, at the output.
#include <cooperative_groups.h>

#include <string>

#include "ida_common.cuh"

namespace cg = cooperative_groups;

namespace ida {

constexpr int SEQ_WARPS = 16;
constexpr int SEQ_THREADS = SEQ_WARPS * 32;

// positions per tile (at most one per warp in the prologue)
template <typename T>
__host__ __device__ constexpr int seq_tile() { return sizeof(T) == 4 ? 16 : 8; }

template <typename T>
static size_t seq_smem_bytes(int Mg, int R, int d) {
    const size_t RD = (size_t)R + d, e = sizeof(T), TT = seq_tile<T>();
    return (size_t)Mg * RD * 2 * e  // X (complex)
           + (size_t)Mg * 2 * e     // eta
           + TT * R * e             // xi(q)
           + TT * RD * e            // z = [kt ; vt]
           + TT * d * e             // partial outputs
           + TT * e;                // partial denominators
}

// Prologue of one position (one warp): xi(q) -> xq_row, [kt ; vt] -> z_row.  tails: NULL, or
// the raw q rows [W-1][R] then k rows of the positions before 0 (oldest first).
template <int NC, typename T>
__device__ __forceinline__ void seq_prologue(const PrefillArgs &a, int h, size_t base_qk,
                                             size_t base_v, int t, T *xq_row,
                                             T *z_row, int lane, const float *tails) {
    const int R = a.R, d = a.d, W = a.W, H = a.H;
    const size_t sqk = (size_t)H * R, sv = (size_t)H * d;
    const float *nw = a.norm_w + (size_t)h * (R + d);
    const float *bs = a.bias + (size_t)h * (R + d);
#pragma unroll 1
    for (int which = 0; which < 2; ++which) {  // 0: query, 1: key
        const void *x = which == 0 ? a.q : a.k;
        const float *cw = a.conv_w + ((size_t)which * H + h) * R * W;
        T f[NC];
        T ss = 0;
#pragma unroll
        for (int i = 0; i < NC; ++i) {
            int c = lane + 32 * i;
            f[i] = 0;
            if (c < R) {
                T s = 0;
                for (int j = 0; j < W; ++j) {
                    int p = t - (W - 1) + j;
                    if (p >= 0)
                        s = fma((T)cw[(size_t)c * W + j], (T)load_in(x, a.dtype, base_qk + (size_t)p * sqk + c), s);
                    else if (tails)
                        s = fma((T)cw[(size_t)c * W + j],
                                (T)tails[((size_t)which * (W - 1) + (p + W - 1)) * R + c], s);
                }
                f[i] = silu(s);
                ss = fma(f[i], f[i], ss);
            }
        }
        T nrm = warp_sum(ss);  // squared norm, or its square root for the l_2 reading
        if (a.flags & IDA_FEAT_L2) nrm = sqrt(nrm);
        T inv = T(1) / (nrm + (T)IDA_EPS_FEAT);
        if (which == 0) {
#pragma unroll
            for (int i = 0; i < NC; ++i) {
                int c = lane + 32 * i;
                if (c < R) xq_row[c] = f[i] * inv;
            }
        } else {
            T ms = 0;
#pragma unroll
            for (int i = 0; i < NC; ++i) {
                f[i] *= inv;
                ms = fma(f[i], f[i], ms);
            }
            T r = rsqrt_t(warp_sum(ms) / R + (T)IDA_EPS_RMS);
#pragma unroll
            for (int i = 0; i < NC; ++i) {
                int c = lane + 32 * i;
                if (c < R) z_row[c] = fma(f[i] * r, (T)nw[c], (T)bs[c]);
            }
        }
    }
    T vv[NC];
    T ms = 0;
#pragma unroll
    for (int i = 0; i < NC; ++i) {
        int j = lane + 32 * i;
        vv[i] = j < d ? (T)load_in(a.v, a.dtype, base_v + (size_t)t * sv + j) : T(0);
        ms = fma(vv[i], vv[i], ms);
    }
    T r = rsqrt_t(warp_sum(ms) / d + (T)IDA_EPS_RMS);
#pragma unroll
    for (int i = 0; i < NC; ++i) {
        int j = lane + 32 * i;
        if (j < d) z_row[R + j] = fma(vv[i] * r, (T)nw[R + j], (T)bs[R + j]);
    }
}

template <int NC, typename T>
__global__ void __launch_bounds__(SEQ_THREADS, 1) seq_prefill_kernel(PrefillArgs a, int G, int Mg) {
    extern __shared__ __align__(16) unsigned char smem[];
    constexpr int TT = seq_tile<T>();
    const int R = a.R, d = a.d, RD = R + d, M = a.M, W = a.W, H = a.H, N = a.N;
    const int rank = blockIdx.x % G;
    const int unit = blockIdx.x / G;
    const int b = unit / H, h = unit % H;
    const int m0 = rank * Mg;
    const int mcount = max(0, min(Mg, M - m0));
    T *Xr = reinterpret_cast<T *>(smem);       // [Mg][RD] real parts
    T *Xi = Xr + (size_t)Mg * RD;              // [Mg][RD] imaginary parts
    T *etr = Xi + (size_t)Mg * RD;             // [Mg]
    T *eti = etr + Mg;                         // [Mg]
    T *xq = eti + Mg;                          // [TT][R]
    T *z = xq + TT * R;                        // [TT][RD]
    T *opart = z + TT * RD;                    // [TT][d]
    T *dpart = opart + TT * d;                 // [TT]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const size_t sqk = (size_t)H * R, sv = (size_t)H * d;
    const size_t base_qk = ((size_t)b * N * H + h) * R;
    const size_t base_v = ((size_t)b * N * H + h) * d;
    const bool eta_ro = (a.flags & IDA_READOUT_ETA) != 0;

    const float *sin = a.state_in ? a.state_in + (size_t)unit * a.state_floats : nullptr;
    const size_t gplane = (size_t)M * RD;
    for (int i = threadIdx.x; i < 2 * Mg * RD + 2 * Mg; i += SEQ_THREADS) Xr[i] = T(0);
    __syncthreads();
    if (sin) {  // the caller's state before position 0, my modes
        for (int i = threadIdx.x; i < mcount * RD; i += SEQ_THREADS) {
            const int ml = i / RD, c = i % RD;
            Xr[i] = (T)sin[(size_t)(m0 + ml) * RD + c];
            Xi[i] = (T)sin[gplane + (size_t)(m0 + ml) * RD + c];
        }
        for (int ml = threadIdx.x; ml < mcount; ml += SEQ_THREADS) {
            etr[ml] = (T)sin[2 * gplane + m0 + ml];
            eti[ml] = (T)sin[2 * gplane + M + m0 + ml];
        }
    }
    const float *tails = sin ? sin + 2 * gplane + 2 * M : nullptr;

    for (int t0 = 0; t0 < N; t0 += TT) {
        const int tn = min(TT, N - t0);
        // Phase A: prologue, one warp per position, the tile's positions spread over the
        // cluster (CTA r computes positions tt = r (mod G) and stores their rows into every
        // CTA of the cluster); clear the partials.
        for (int tt = rank + G * warp; tt < tn; tt += G * SEQ_WARPS) {
            T *xrow = xq + tt * R, *zrow = z + tt * RD;
            seq_prologue<NC, T>(a, h, base_qk, base_v, t0 + tt, xrow, zrow, lane, tails);
            if (G > 1) {
                __syncwarp();
                for (int r = 0; r < G; ++r) {
                    if (r == rank) continue;
                    T *rx = cg::this_cluster().map_shared_rank(xrow, r);
                    T *rz = cg::this_cluster().map_shared_rank(zrow, r);
                    for (int c = lane; c < R; c += 32) rx[c] = xrow[c];
                    for (int c = lane; c < RD; c += 32) rz[c] = zrow[c];
                }
            }
        }
        for (int i = threadIdx.x; i < tn * d; i += SEQ_THREADS) opart[i] = T(0);
        for (int i = threadIdx.x; i < tn; i += SEQ_THREADS) dpart[i] = T(0);
        if (G == 1)
            __syncthreads();
        else
            cg::this_cluster().sync();
        // Phase B: recurrence + per-mode readout, one warp per mode.
        for (int ml = warp; ml < mcount; ml += SEQ_WARPS) {
            const int m = m0 + ml;
            const T lr = a.lambda[((size_t)h * M + m) * 2], li = a.lambda[((size_t)h * M + m) * 2 + 1];
            const T gr_ = a.Bvec[((size_t)h * M + m) * 2], gi_ = a.Bvec[((size_t)h * M + m) * 2 + 1];
            T ur[NC], ui[NC], vr[NC], vi[NC];
#pragma unroll
            for (int i = 0; i < NC; ++i) {
                int c = lane + 32 * i;
                ur[i] = c < R ? Xr[(size_t)ml * RD + c] : T(0);
                ui[i] = c < R ? Xi[(size_t)ml * RD + c] : T(0);
                vr[i] = c < d ? Xr[(size_t)ml * RD + R + c] : T(0);
                vi[i] = c < d ? Xi[(size_t)ml * RD + R + c] : T(0);
            }
            T er = etr[ml], ei = eti[ml];
            for (int tt = 0; tt < tn; ++tt) {
                T ar = 0, ai = 0;
#pragma unroll
                for (int i = 0; i < NC; ++i) {
                    int c = lane + 32 * i;
                    if (c < R) {
                        cstep_t(ur[i], ui[i], lr, li, gr_, gi_, z[tt * RD + c]);
                        T xv = xq[tt * R + c];
                        ar = fma(xv, ur[i], ar);
                        ai = fma(xv, ui[i], ai);
                    }
                    if (c < d) cstep_t(vr[i], vi[i], lr, li, gr_, gi_, z[tt * RD + R + c]);
                }
                cstep_t(er, ei, lr, li, gr_, gi_, T(1));
                ar = warp_sum(ar);
                ai = warp_sum(ai);
#pragma unroll
                for (int i = 0; i < NC; ++i) {
                    int j = lane + 32 * i;
                    if (j < d) atomicAdd(&opart[tt * d + j], ar * vr[i] - ai * vi[i]);
                }
                if (lane == 0) atomicAdd(&dpart[tt], ar * er - ai * ei);
            }
#pragma unroll
            for (int i = 0; i < NC; ++i) {
                int c = lane + 32 * i;
                if (c < R) {
                    Xr[(size_t)ml * RD + c] = ur[i];
                    Xi[(size_t)ml * RD + c] = ui[i];
                }
                if (c < d) {
                    Xr[(size_t)ml * RD + R + c] = vr[i];
                    Xi[(size_t)ml * RD + R + c] = vi[i];
                }
            }
            if (lane == 0) {
                etr[ml] = er;
                eti[ml] = ei;
            }
        }
        // Phase C: sum the cluster's partials; CTA r writes positions tt = r (mod G).
        if (G == 1) {
            __syncthreads();
        } else {
            cg::this_cluster().sync();
        }
        for (int tt = rank + G * warp; tt < tn; tt += G * SEQ_WARPS) {
            T dn = 0;
            if (eta_ro) {
                for (int r = 0; r < G; ++r) {
                    const T *pd = G == 1 ? dpart : cg::this_cluster().map_shared_rank(dpart, r);
                    dn += pd[tt];
                }
            }
            for (int j = lane; j < d; j += 32) {
                T o = 0;
                for (int r = 0; r < G; ++r) {
                    const T *po = G == 1 ? opart : cg::this_cluster().map_shared_rank(opart, r);
                    o += po[tt * d + j];
                }
                if (eta_ro) o = o / dn;
                store_out(a.out, a.dtype, base_v + (size_t)(t0 + tt) * sv + j, (float)o);
            }
        }
        if (G == 1) {
            __syncthreads();
        } else {
            cg::this_cluster().sync();
        }
    }

    if (a.final_state) {
        float *fs = a.final_state + (size_t)unit * a.state_floats;
        const size_t plane = (size_t)M * RD;
        for (int i = threadIdx.x; i < mcount * RD; i += SEQ_THREADS) {
            int ml = i / RD, c = i % RD;
            fs[(size_t)(m0 + ml) * RD + c] = (float)Xr[i];
            fs[plane + (size_t)(m0 + ml) * RD + c] = (float)Xi[i];
        }
        for (int ml = threadIdx.x; ml < mcount; ml += SEQ_THREADS) {
            fs[2 * plane + m0 + ml] = (float)etr[ml];
            fs[2 * plane + M + m0 + ml] = (float)eti[ml];
        }
        if (rank == 0) {
            float *tq = fs + 2 * plane + 2 * M;
            float *tk = tq + (size_t)(W - 1) * R;
            for (int i = threadIdx.x; i < (W - 1) * R; i += SEQ_THREADS) {
                int r = i / R, c = i % R;
                int p = N - (W - 1) + r;  // before position 0: the initial state's tails
                const size_t tx = (size_t)(p + W - 1) * R + c;
                tq[i] = p >= 0 ? load_in(a.q, a.dtype, base_qk + (size_t)p * sqk + c) : (tails ? tails[tx] : 0.f);
                tk[i] = p >= 0 ? load_in(a.k, a.dtype, base_qk + (size_t)p * sqk + c)
                               : (tails ? tails[(size_t)(W - 1) * R + tx] : 0.f);
            }
            size_t used = 2 * plane + 2 * M + 2 * (size_t)(W - 1) * R;
            for (size_t i = used + threadIdx.x; i < a.state_floats; i += SEQ_THREADS) fs[i] = 0.f;
        }
    }
}

template <int NC, typename T>
static cudaError_t launch_seq_nc(const PrefillArgs &a, int G, int Mg, size_t smem, cudaStream_t st) {
    auto kern = seq_prefill_kernel<NC, T>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)G * (unsigned)(a.B * a.H), 1, 1);
    cfg.blockDim = dim3(SEQ_THREADS, 1, 1);
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
static ida_status launch_seq_t(const PrefillArgs &a, cudaStream_t st, int num_sms, std::string &why) {
    const size_t kMaxSmem = 227 * 1024;
    int G = 1;
    while (G < 8 && seq_smem_bytes<T>((a.M + G - 1) / G, a.R, a.d) > kMaxSmem) G *= 2;
    if (seq_smem_bytes<T>((a.M + G - 1) / G, a.R, a.d) > kMaxSmem) {
        why = "state of M x (R+d) does not fit a cluster of 8 CTAs";
        return IDA_ERR_UNSUPPORTED;
    }
    const long units = (long)a.B * a.H;
    while (G < 8 && 2 * G <= a.M && units * 2 * G <= num_sms) G *= 2;
    const int Mg = (a.M + G - 1) / G;
    const size_t smem = seq_smem_bytes<T>(Mg, a.R, a.d);
    const int nc_need = ((a.R > a.d ? a.R : a.d) + 31) / 32;
    cudaError_t e;
    if (nc_need <= 1)
        e = launch_seq_nc<1, T>(a, G, Mg, smem, st);
    else if (nc_need <= 2)
        e = launch_seq_nc<2, T>(a, G, Mg, smem, st);
    else if (nc_need <= 4)
        e = launch_seq_nc<4, T>(a, G, Mg, smem, st);
    else
        e = launch_seq_nc<8, T>(a, G, Mg, smem, st);
    if (e != cudaSuccess) {
        why = std::string("sequential prefill launch: ") + cudaGetErrorString(e);
        return IDA_ERR_CUDA;
    }
    return IDA_OK;
}

bool launch_seq_modes(const PrefillArgs &a, cudaStream_t st, int num_sms, ida_status &s, std::string &why);

// fp32 inputs: this kernel in fp64.  bf16 inputs: the register-resident kernel of
// ida_seq_modes.cu where it takes the shape, else this kernel in fp32.  The cluster size
// here is the smallest G whose per-CTA state fits in shared memory, then doubled while
// the grid stays within one wave of SMs.
ida_status launch_seq_prefill(const PrefillArgs &a, cudaStream_t st, int num_sms, std::string &why) {
    if (a.dtype == IDA_F32) return launch_seq_t<double>(a, st, num_sms, why);
    ida_status s;
    // the register-resident kernel runs in the scaled state X / B, which a caller's state
    // cannot always be brought into (B = 0 with X != 0): from a given state this kernel runs
    if (!a.state_in && launch_seq_modes(a, st, num_sms, s, why)) return s;
    return launch_seq_t<float>(a, st, num_sms, why);
}

}  // namespace ida
