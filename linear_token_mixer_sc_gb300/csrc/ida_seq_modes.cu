// ida_seq_modes.cu -- token-sequential prefill for bf16 inputs with the state in registers.
//
// The recurrence X_t = lambda X_{t-1} + B z_t and the readouts o_t = Re(a_t Gamma_t) and
// o_t = Re(a_t Gamma_t) / Re(a_t eta_t), a_t = xi(q_t) U_t^T, of "Interdomain Attention:
// Beyond Token-Level Key-Value Memory" (German technical summary, "Skalierbare
// Implementierung" for the recurrent core, "Theoretische Herleitung" for the ratio form),
// walked one position at a time in fp32 on the CUDA cores.  This is the path of the eta
// readout for bf16 inputs (whose denominator can cancel far below the rounding of the
// tensor-core operands) and of bf16 shapes the chunked kernel does not take.
//
// Arithmetic in the scaled state Y = X / B (per mode).  Since B is constant over time,
// Y_t = lambda Y_{t-1} + z_t, so an update costs four fp32 operations per complex element
// instead of six; with alpha_t[m] = xi(q_t) . Y^U_t[m] and beta = B^2 alpha,
//   o_t = Re sum_m beta_t[m] Y^Gamma_t[m],   den_t = Re sum_m beta_t[m] e_t[m],
// where e_t = lambda e_{t-1} + 1 (eta = B e).  The final state is written as X = B Y.
// A mode with B = 0 keeps X = 0 and contributes nothing, as in the unscaled recurrence.
//
// Work split: the modes of a unit are split over a cluster of G CTAs and, inside a CTA,
// over NWC compute warps.  A compute warp owns MPW modes; its lanes form 32/LG groups of
// LG = R/4 lanes, each group owns 4 modes, and a lane owns 4 consecutive key columns and
// 4 consecutive value columns (d = R) of those 4 modes: 64 fp32 state registers per lane.
// a_t needs a sum over the key columns, done per position by a reduce-scatter plus
// all-gather over the LG lanes of the group (17 shuffles at R = 128).
//
// Positions are processed in tiles of TT; CTA r of the cluster owns positions
// [r PT, r PT + PT) of every tile, split between its two helper warps, which run beside
// the compute warps.  A helper warp computes the feature prologue (conv, SiLU feature
// map, RMSNorm) of its positions of the next tile and stores it into the shared memory of
// every CTA of the cluster; then it sums the partial readouts of its positions of the
// previous tile, which every compute warp of the cluster has stored into this CTA's
// shared memory (in a fixed order, so the result does not depend on scheduling), divides
// by the denominator for the eta readout and writes the outputs.  All traffic between
// CTAs is stores; one cluster barrier per tile orders it, and inputs and partials are
// double-buffered.
#include <cooperative_groups.h>

#include <string>

#include "ida_common.cuh"

namespace cg = cooperative_groups;

namespace ida {

namespace {

constexpr int SM_TT = 16;    // positions per tile
constexpr int SM_HELP = 2;   // helper warps per CTA (prologue and output)
constexpr int SM_MAXW = 4 + SM_HELP;
constexpr unsigned FULL = 0xffffffffu;

// Shared memory of one CTA, in floats.  S = G * nwc compute warps of the cluster each
// store their partial readout of a position into the CTA that writes that position's
// output (CTA r writes positions [r PT, r PT + PT) of every tile).
struct ModesLayout {
    size_t xq;     // [2][TT][R]        xi(q) of the tile
    size_t zb;     // [2][TT][2R]       [kt ; vt] of the tile
    size_t op;     // [2][S][PT][R]     partial outputs of this CTA's positions, per warp
    size_t dp;     // [2][S][PT]        partial denominators, per warp
    size_t bytes;
};

__host__ __device__ inline int modes_pt(int G) { return (SM_TT + G - 1) / G; }

__host__ __device__ inline ModesLayout modes_layout(int R, int nwc, int G) {
    const size_t S = (size_t)G * nwc, PT = modes_pt(G);
    ModesLayout L;
    L.xq = 0;
    L.zb = L.xq + (size_t)2 * SM_TT * R;
    L.op = L.zb + (size_t)2 * SM_TT * 2 * R;
    L.dp = L.op + 2 * S * PT * R;
    L.bytes = (L.dp + 2 * S * PT) * sizeof(float);
    return L;
}

// Sum of p[0..8) over the LG lanes of a group, returned to every lane of the group:
// three halving exchanges leave each lane one eighth of the values summed over eight
// lanes, butterflies finish the sum, and eight broadcasts gather the results.
template <int LG>
__device__ __forceinline__ void group_allreduce8(float (&p)[8], int lane) {
    {
        constexpr int o = LG / 2;
        const bool hi = (lane & o) != 0;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float send = hi ? p[i] : p[i + 4];
            const float keep = hi ? p[i + 4] : p[i];
            p[i] = keep + __shfl_xor_sync(FULL, send, o);
        }
    }
    {
        constexpr int o = LG / 4;
        const bool hi = (lane & o) != 0;
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const float send = hi ? p[i] : p[i + 2];
            const float keep = hi ? p[i + 2] : p[i];
            p[i] = keep + __shfl_xor_sync(FULL, send, o);
        }
    }
    {
        constexpr int o = LG / 8;
        const bool hi = (lane & o) != 0;
        const float send = hi ? p[0] : p[1];
        const float keep = hi ? p[1] : p[0];
        p[0] = keep + __shfl_xor_sync(FULL, send, o);
    }
#pragma unroll
    for (int o = LG / 16; o > 0; o >>= 1) p[0] += __shfl_xor_sync(FULL, p[0], o);
    const float s = p[0];
    // value v sits in the lanes whose bits LG/2, LG/4, LG/8 spell v
#pragma unroll
    for (int v = 0; v < 8; ++v)
        p[v] = __shfl_sync(FULL, s, ((v >> 2) & 1) * (LG / 2) + ((v >> 1) & 1) * (LG / 4) + (v & 1) * (LG / 8), LG);
}

// The same for p[0..16) (two positions' values), LG >= 16: four halving exchanges, then
// sixteen broadcasts.
template <int LG>
__device__ __forceinline__ void group_allreduce16(float (&p)[16], int lane) {
    static_assert(LG >= 16, "four halving levels need 16 lanes");
#pragma unroll
    for (int lvl = 0; lvl < 4; ++lvl) {
        const int o = LG >> (lvl + 1), n = 8 >> lvl;  // values kept after this level: n
        const bool hi = (lane & o) != 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            if (i < n) {
                const float send = hi ? p[i] : p[i + n];
                const float keep = hi ? p[i + n] : p[i];
                p[i] = keep + __shfl_xor_sync(FULL, send, o);
            }
        }
    }
#pragma unroll
    for (int o = LG / 32; o > 0; o >>= 1) p[0] += __shfl_xor_sync(FULL, p[0], o);
    const float s = p[0];
    // value v sits in the lanes whose bits LG/2, LG/4, LG/8, LG/16 spell v
#pragma unroll
    for (int v = 0; v < 16; ++v)
        p[v] = __shfl_sync(FULL, s,
                           ((v >> 3) & 1) * (LG / 2) + ((v >> 2) & 1) * (LG / 4) + ((v >> 1) & 1) * (LG / 8) +
                               (v & 1) * (LG / 16),
                           LG);
}

typedef unsigned long long f2_t;  // two fp32 in one 64-bit register

__device__ __forceinline__ f2_t f2_pack(float lo, float hi) {
    f2_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void f2_unpack(f2_t v, float &lo, float &hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ f2_t f2_fma(f2_t a, f2_t b, f2_t c) {
    f2_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ f2_t f2_mul(f2_t a, f2_t b) {
    f2_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

// 32-bit shared-memory addresses: this CTA's, the same offset in CTA r of the cluster,
// and stores through them (a CTA's own shared::cta address is valid in the cluster window)
__device__ __forceinline__ uint32_t smem_u32(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }
__device__ __forceinline__ uint32_t mapa_u32(uint32_t a, uint32_t r) {
    uint32_t d;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(r));
    return d;
}
__device__ __forceinline__ void st_cluster(uint32_t a, float x) {
    asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(a), "f"(x) : "memory");
}
__device__ __forceinline__ void st_cluster(uint32_t a, float x, float y) {
    asm volatile("st.shared::cluster.v2.f32 [%0], {%1, %2};" ::"r"(a), "f"(x), "f"(y) : "memory");
}
__device__ __forceinline__ void st_cluster(uint32_t a, float x, float y, float z, float w) {
    asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(a), "f"(x), "f"(y), "f"(z), "f"(w)
                 : "memory");
}
template <int CPL>
__device__ __forceinline__ void st_cluster_row(uint32_t a, const float (&x)[CPL]) {
    if constexpr (CPL == 4)
        st_cluster(a, x[0], x[1], x[2], x[3]);
    else if constexpr (CPL == 2)
        st_cluster(a, x[0], x[1]);
    else
        st_cluster(a, x[0]);
}

// SiLU with the hardware exponential and divide (a few ulp; the inputs of this kernel are bf16,
// rounded at 2^-8, so the feature map's own rounding is far below theirs)
__device__ __forceinline__ float silu_fast(float x) { return __fdividef(x, 1.f + __expf(-x)); }

template <int CPL>
__device__ __forceinline__ void load_bf16_row(const __nv_bfloat16 *p, float (&x)[CPL]) {
    if constexpr (CPL == 4) {
        const uint2 u = *reinterpret_cast<const uint2 *>(p);
        x[0] = __uint_as_float(u.x << 16);
        x[1] = __uint_as_float(u.x & 0xFFFF0000u);
        x[2] = __uint_as_float(u.y << 16);
        x[3] = __uint_as_float(u.y & 0xFFFF0000u);
    } else if constexpr (CPL == 2) {
        const uint32_t u = *reinterpret_cast<const uint32_t *>(p);
        x[0] = __uint_as_float(u << 16);
        x[1] = __uint_as_float(u & 0xFFFF0000u);
    } else {
        x[0] = __bfloat162float(*p);
    }
}

template <int CPL>
__device__ __forceinline__ void load_f32(const float *p, float (&x)[CPL]) {
    if constexpr (CPL == 4) {
        const float4 u = *reinterpret_cast<const float4 *>(p);
        x[0] = u.x; x[1] = u.y; x[2] = u.z; x[3] = u.w;
    } else if constexpr (CPL == 2) {
        const float2 u = *reinterpret_cast<const float2 *>(p);
        x[0] = u.x; x[1] = u.y;
    } else {
        x[0] = *p;
    }
}

template <int CPL>
__device__ __forceinline__ void store_bf16_row(__nv_bfloat16 *p, const float (&x)[CPL]) {
    if constexpr (CPL == 4) {
        const __nv_bfloat162 a = __floats2bfloat162_rn(x[0], x[1]), b = __floats2bfloat162_rn(x[2], x[3]);
        uint2 u;
        u.x = *reinterpret_cast<const uint32_t *>(&a);
        u.y = *reinterpret_cast<const uint32_t *>(&b);
        *reinterpret_cast<uint2 *>(p) = u;
    } else if constexpr (CPL == 2) {
        *reinterpret_cast<__nv_bfloat162 *>(p) = __floats2bfloat162_rn(x[0], x[1]);
    } else {
        *p = __float2bfloat16_rn(x[0]);
    }
}

}  // namespace

// R = d in {32, 64, 128}, bf16 inputs.  Block: nwc compute warps, then SM_HELP helper warps.
template <int R, bool ETA>
__global__ void __launch_bounds__(SM_MAXW * 32, 2) seq_modes_kernel(PrefillArgs a, int G, int nwc) {
    constexpr int LG = R / 4;      // lanes per mode group
    constexpr int GPW = 32 / LG;   // mode groups per warp
    constexpr int MPW = 4 * GPW;   // modes per compute warp
    constexpr int CPL = R / 32;    // channels per lane in the prologue and output warps
    constexpr int TT = SM_TT;
    extern __shared__ __align__(16) float smf[];
    cg::cluster_group cluster = cg::this_cluster();
    const ModesLayout L = modes_layout(R, nwc, G);
    float *xq = smf + L.xq, *zb = smf + L.zb, *op = smf + L.op, *dp = smf + L.dp;

    const int rank = G > 1 ? (int)cluster.block_rank() : 0;
    const int unit = blockIdx.x / G;
    const int H = a.H, N = a.N, M = a.M, W = a.W;
    const int b = unit / H, h = unit % H;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nt = (N + TT - 1) / TT;
    const int PT = modes_pt(G);  // positions of a tile whose prologue and output this CTA runs
    const int S = G * nwc;       // partial-readout slices per position
    const size_t row_qk = (size_t)H * R;  // elements between consecutive positions (d = R)
    const size_t base = ((size_t)b * N * H + h) * R;
    const __nv_bfloat16 *qg = reinterpret_cast<const __nv_bfloat16 *>(a.q) + base;
    const __nv_bfloat16 *kg = reinterpret_cast<const __nv_bfloat16 *>(a.k) + base;
    const __nv_bfloat16 *vg = reinterpret_cast<const __nv_bfloat16 *>(a.v) + base;

    auto csync = [&]() {
        if (G > 1)
            cluster.sync();
        else
            __syncthreads();
    };

    // ---- helper warps: this warp's positions of a tile are [hlo, hhi) (tile-local)
    const int pw = warp - nwc;
    const bool feat_l2 = (a.flags & IDA_FEAT_L2) != 0;
    const int hper = (PT + SM_HELP - 1) / SM_HELP;
    const int hlo = min(TT, rank * PT + pw * hper);
    const int hhi = min(TT, min(rank * PT + PT, rank * PT + pw * hper + hper));
    float cwq[CPL][4], cwk[CPL][4], nwk[CPL], bsk[CPL], nwv[CPL], bsv[CPL];
    if (pw >= 0) {
        const float *cq = a.conv_w + ((size_t)h * R + CPL * lane) * W;
        const float *ck = a.conv_w + ((size_t)(H + h) * R + CPL * lane) * W;
        const float *nw = a.norm_w + (size_t)h * 2 * R, *bs = a.bias + (size_t)h * 2 * R;
#pragma unroll
        for (int i = 0; i < CPL; ++i) {
#pragma unroll
            for (int j = 0; j < 4; ++j) {  // right-aligned: tap j sits at window row 4 - W + j
                cwq[i][j] = j >= 4 - W ? cq[i * W + j - (4 - W)] : 0.f;
                cwk[i][j] = j >= 4 - W ? ck[i * W + j - (4 - W)] : 0.f;
            }
            nwk[i] = nw[CPL * lane + i];
            bsk[i] = bs[CPL * lane + i];
            nwv[i] = nw[R + CPL * lane + i];
            bsv[i] = bs[R + CPL * lane + i];
        }
    }
    // features of tile kk into every CTA's buffer kk & 1
    auto prologue = [&](int kk) {
        const int lo = kk * TT + hlo, hi = min(N, kk * TT + hhi);
        if (lo >= hi) return;
        // window rows t-3 .. t of raw q and k (zero before position 0); the rows of the next
        // position are loaded one position ahead
        float wq[4][CPL], wk[4][CPL], nq[CPL], nk[CPL], nv[CPL];
#pragma unroll
        for (int r = 1; r < 4; ++r) {
            const int p = lo - 4 + r;
#pragma unroll
            for (int i = 0; i < CPL; ++i) wq[r][i] = wk[r][i] = 0.f;
            if (p >= 0) {
                load_bf16_row<CPL>(qg + (size_t)p * row_qk + CPL * lane, wq[r]);
                load_bf16_row<CPL>(kg + (size_t)p * row_qk + CPL * lane, wk[r]);
            }
        }
        load_bf16_row<CPL>(qg + (size_t)lo * row_qk + CPL * lane, nq);
        load_bf16_row<CPL>(kg + (size_t)lo * row_qk + CPL * lane, nk);
        load_bf16_row<CPL>(vg + (size_t)lo * row_qk + CPL * lane, nv);
        for (int t = lo; t < hi; ++t) {
            float vv[CPL];
#pragma unroll
            for (int i = 0; i < CPL; ++i) {
#pragma unroll
                for (int r = 0; r < 3; ++r) {
                    wq[r][i] = wq[r + 1][i];
                    wk[r][i] = wk[r + 1][i];
                }
                wq[3][i] = nq[i];
                wk[3][i] = nk[i];
                vv[i] = nv[i];
            }
            if (t + 1 < hi) {
                load_bf16_row<CPL>(qg + (size_t)(t + 1) * row_qk + CPL * lane, nq);
                load_bf16_row<CPL>(kg + (size_t)(t + 1) * row_qk + CPL * lane, nk);
                load_bf16_row<CPL>(vg + (size_t)(t + 1) * row_qk + CPL * lane, nv);
            }
            // causal conv over window rows t-3 .. t (the taps before the first are zero)
            float fq[CPL], fk[CPL], ssq = 0.f, ssk = 0.f, ssv = 0.f;
#pragma unroll
            for (int i = 0; i < CPL; ++i) {
                float sq = 0.f, sk = 0.f;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    sq = fmaf(cwq[i][j], wq[j][i], sq);
                    sk = fmaf(cwk[i][j], wk[j][i], sk);
                }
                fq[i] = silu_fast(sq);
                fk[i] = silu_fast(sk);
                ssq = fmaf(fq[i], fq[i], ssq);
                ssk = fmaf(fk[i], fk[i], ssk);
                ssv = fmaf(vv[i], vv[i], ssv);
            }
            float nq = warp_sum(ssq), nk = warp_sum(ssk);  // squared norms, or l_2 norms
            if (feat_l2) {
                nq = sqrtf(nq);
                nk = sqrtf(nk);
            }
            const float iq = 1.f / (nq + (float)IDA_EPS_FEAT);
            const float ik = 1.f / (nk + (float)IDA_EPS_FEAT);
            float msk = 0.f;
#pragma unroll
            for (int i = 0; i < CPL; ++i) {
                fq[i] *= iq;
                fk[i] *= ik;
                msk = fmaf(fk[i], fk[i], msk);
            }
            const float rk = rsqrtf(warp_sum(msk) / R + (float)IDA_EPS_RMS);
            const float rv = rsqrtf(warp_sum(ssv) / R + (float)IDA_EPS_RMS);
#pragma unroll
            for (int i = 0; i < CPL; ++i) {
                fk[i] = fmaf(fk[i] * rk, nwk[i], bsk[i]);
                vv[i] = fmaf(vv[i] * rv, nwv[i], bsv[i]);
            }
            const int tt = t - kk * TT;
            const uint32_t aq = smem_u32(xq + (size_t)(kk & 1) * TT * R + (size_t)tt * R + CPL * lane);
            const uint32_t az = smem_u32(zb + (size_t)(kk & 1) * TT * 2 * R + (size_t)tt * 2 * R + CPL * lane);
            for (int r = 0; r < G; ++r) {
                const uint32_t dq = G > 1 ? mapa_u32(aq, r) : aq, dz = G > 1 ? mapa_u32(az, r) : az;
                st_cluster_row<CPL>(dq, fq);
                st_cluster_row<CPL>(dz, fk);
                st_cluster_row<CPL>(dz + 4 * R, vv);
            }
        }
    };

    // outputs of tile kk: the S partials of each position (all in this CTA's shared
    // memory), summed in a fixed order
    auto output = [&](int kk) {
        const int lo = kk * TT + hlo, hi = min(N, kk * TT + hhi);
        for (int t = lo; t < hi; ++t) {
            const int pl = t - kk * TT - rank * PT;
            const float *src = op + ((size_t)(kk & 1) * S * PT + pl) * R + CPL * lane;
            const float *srd = dp + (size_t)(kk & 1) * S * PT + pl;
            float o[CPL];
#pragma unroll
            for (int i = 0; i < CPL; ++i) o[i] = 0.f;
            float dn = 0.f;
            for (int s0 = 0; s0 < S; s0 += 8) {
                float part[8][CPL], dpart[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
#pragma unroll
                    for (int i = 0; i < CPL; ++i) part[u][i] = 0.f;
                    dpart[u] = 0.f;
                    if (s0 + u < S) {
                        load_f32<CPL>(src + (size_t)(s0 + u) * PT * R, part[u]);
                        if (ETA) dpart[u] = srd[(size_t)(s0 + u) * PT];
                    }
                }
#pragma unroll
                for (int u = 0; u < 8; ++u) {
#pragma unroll
                    for (int i = 0; i < CPL; ++i) o[i] += part[u][i];
                    dn += dpart[u];
                }
            }
            if (ETA) {
#pragma unroll
                for (int i = 0; i < CPL; ++i) o[i] = __fdividef(o[i], dn);
            }
            store_bf16_row<CPL>(reinterpret_cast<__nv_bfloat16 *>(a.out) + base + (size_t)t * row_qk + CPL * lane, o);
        }
    };

    // ---- compute warps: the state of MPW modes in registers
    const int g = lane / LG, gl = lane % LG;
    const int mbase = (rank * nwc + warp) * MPW + 4 * g;
    f2_t ur[4][2], ui[4][2], gr[4][2], gi[4][2];
    f2_t lr2[4], li2[4], nli2[4];
    float b2r[4], b2i[4], er[4], ei[4];
    if (warp < nwc) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int m = mbase + j;
            float2 lam = make_float2(0.f, 0.f), bb = make_float2(0.f, 0.f);
            if (m < M) {
                lam = *reinterpret_cast<const float2 *>(a.lambda + ((size_t)h * M + m) * 2);
                bb = *reinterpret_cast<const float2 *>(a.Bvec + ((size_t)h * M + m) * 2);
            }
            b2r[j] = bb.x * bb.x - bb.y * bb.y;
            b2i[j] = 2.f * bb.x * bb.y;
            er[j] = ei[j] = 0.f;
            lr2[j] = f2_pack(lam.x, lam.x);
            li2[j] = f2_pack(lam.y, lam.y);
            nli2[j] = f2_pack(-lam.y, -lam.y);
#pragma unroll
            for (int i = 0; i < 2; ++i) ur[j][i] = ui[j][i] = gr[j][i] = gi[j][i] = 0ull;
        }
    }
    auto compute = [&](int kk) {
        const int tn = min(TT, N - kk * TT);
        const float *xp = xq + (size_t)(kk & 1) * TT * R + 4 * gl;
        const float *zp = zb + (size_t)(kk & 1) * TT * 2 * R + 4 * gl;
        const uint32_t slice = (uint32_t)((kk & 1) * S + rank * nwc + warp);  // this warp's slice
        const uint32_t ao = smem_u32(op + (size_t)slice * PT * R + 4 * gl), ad = smem_u32(dp + (size_t)slice * PT);
        // uo, ud: where this position's partials go, in the CTA that writes its output
        auto step = [&](uint32_t uo, uint32_t ud) {
            const ulonglong2 x4 = *reinterpret_cast<const ulonglong2 *>(xp);
            const ulonglong2 k4 = *reinterpret_cast<const ulonglong2 *>(zp);
            const ulonglong2 v4 = *reinterpret_cast<const ulonglong2 *>(zp + R);
            const f2_t x[2] = {x4.x, x4.y}, zk[2] = {k4.x, k4.y}, zv[2] = {v4.x, v4.y};
            float p[8];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                f2_t sr = 0ull, si = 0ull;
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    const f2_t t1 = f2_mul(li2[j], ur[j][i]);
                    const f2_t t2 = f2_fma(nli2[j], ui[j][i], zk[i]);
                    ui[j][i] = f2_fma(lr2[j], ui[j][i], t1);
                    ur[j][i] = f2_fma(lr2[j], ur[j][i], t2);
                    sr = i == 0 ? f2_mul(x[i], ur[j][i]) : f2_fma(x[i], ur[j][i], sr);
                    si = i == 0 ? f2_mul(x[i], ui[j][i]) : f2_fma(x[i], ui[j][i], si);
                }
                float a0, a1, b0, b1;
                f2_unpack(sr, a0, a1);
                f2_unpack(si, b0, b1);
                p[2 * j] = a0 + a1;
                p[2 * j + 1] = b0 + b1;
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    const f2_t t1 = f2_mul(li2[j], gr[j][i]);
                    const f2_t t2 = f2_fma(nli2[j], gi[j][i], zv[i]);
                    gi[j][i] = f2_fma(lr2[j], gi[j][i], t1);
                    gr[j][i] = f2_fma(lr2[j], gr[j][i], t2);
                }
                float lrj, lrh, lij, lih;
                f2_unpack(lr2[j], lrj, lrh);
                f2_unpack(li2[j], lij, lih);
                const float t1 = lij * er[j];
                const float t2 = fmaf(-lij, ei[j], 1.f);
                ei[j] = fmaf(lrj, ei[j], t1);
                er[j] = fmaf(lrj, er[j], t2);
            }
            group_allreduce8<LG>(p, lane);
            f2_t o2[2] = {0ull, 0ull};
            float dn = 0.f;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float br = fmaf(b2r[j], p[2 * j], -b2i[j] * p[2 * j + 1]);
                const float nbi = fmaf(-b2r[j], p[2 * j + 1], -b2i[j] * p[2 * j]);  // -Im beta
                const f2_t br2 = f2_pack(br, br), nbi2 = f2_pack(nbi, nbi);
#pragma unroll
                for (int i = 0; i < 2; ++i) o2[i] = f2_fma(br2, gr[j][i], f2_fma(nbi2, gi[j][i], o2[i]));
                if (ETA) dn = fmaf(br, er[j], fmaf(nbi, ei[j], dn));
            }
            float o[4];
            f2_unpack(o2[0], o[0], o[1]);
            f2_unpack(o2[1], o[2], o[3]);
#pragma unroll
            for (int off = LG; off < 32; off <<= 1) {
#pragma unroll
                for (int i = 0; i < 4; ++i) o[i] += __shfl_xor_sync(FULL, o[i], off);
                if (ETA) dn += __shfl_xor_sync(FULL, dn, off);
            }
            if (LG == 32 || lane < LG) st_cluster(uo, o[0], o[1], o[2], o[3]);
            if (ETA && lane == 0) st_cluster(ud, dn);
            xp += R;
            zp += 2 * R;
        };
        // Two positions at once (LG >= 16): the key-column updates and a_t parts of both,
        // one 16-value group all-reduce for both (a_t does not depend on the value columns),
        // then the value-column updates and readouts in order.
        auto step2 = [&](uint32_t uo, uint32_t ud) {
            float p[16];
#pragma unroll
            for (int sp = 0; sp < 2; ++sp) {
                const ulonglong2 x4 = *reinterpret_cast<const ulonglong2 *>(xp + sp * R);
                const ulonglong2 k4 = *reinterpret_cast<const ulonglong2 *>(zp + sp * 2 * R);
                const f2_t x[2] = {x4.x, x4.y}, zk[2] = {k4.x, k4.y};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    f2_t sr = 0ull, si = 0ull;
#pragma unroll
                    for (int i = 0; i < 2; ++i) {
                        const f2_t t1 = f2_mul(li2[j], ur[j][i]);
                        const f2_t t2 = f2_fma(nli2[j], ui[j][i], zk[i]);
                        ui[j][i] = f2_fma(lr2[j], ui[j][i], t1);
                        ur[j][i] = f2_fma(lr2[j], ur[j][i], t2);
                        sr = i == 0 ? f2_mul(x[i], ur[j][i]) : f2_fma(x[i], ur[j][i], sr);
                        si = i == 0 ? f2_mul(x[i], ui[j][i]) : f2_fma(x[i], ui[j][i], si);
                    }
                    float a0, a1, b0, b1;
                    f2_unpack(sr, a0, a1);
                    f2_unpack(si, b0, b1);
                    p[8 * sp + 2 * j] = a0 + a1;
                    p[8 * sp + 2 * j + 1] = b0 + b1;
                }
            }
            if constexpr (LG >= 16) {
                group_allreduce16<LG>(p, lane);
            } else {
                float p0[8], p1[8];
#pragma unroll
                for (int v = 0; v < 8; ++v) {
                    p0[v] = p[v];
                    p1[v] = p[8 + v];
                }
                group_allreduce8<LG>(p0, lane);
                group_allreduce8<LG>(p1, lane);
#pragma unroll
                for (int v = 0; v < 8; ++v) {
                    p[v] = p0[v];
                    p[8 + v] = p1[v];
                }
            }
#pragma unroll
            for (int sp = 0; sp < 2; ++sp) {
                const ulonglong2 v4 = *reinterpret_cast<const ulonglong2 *>(zp + sp * 2 * R + R);
                const f2_t zv[2] = {v4.x, v4.y};
                f2_t o2[2] = {0ull, 0ull};
                float dn = 0.f;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
#pragma unroll
                    for (int i = 0; i < 2; ++i) {
                        const f2_t t1 = f2_mul(li2[j], gr[j][i]);
                        const f2_t t2 = f2_fma(nli2[j], gi[j][i], zv[i]);
                        gi[j][i] = f2_fma(lr2[j], gi[j][i], t1);
                        gr[j][i] = f2_fma(lr2[j], gr[j][i], t2);
                    }
                    float lrj, lrh, lij, lih;
                    f2_unpack(lr2[j], lrj, lrh);
                    f2_unpack(li2[j], lij, lih);
                    const float t1 = lij * er[j];
                    const float t2 = fmaf(-lij, ei[j], 1.f);
                    ei[j] = fmaf(lrj, ei[j], t1);
                    er[j] = fmaf(lrj, er[j], t2);
                    const float br = fmaf(b2r[j], p[8 * sp + 2 * j], -b2i[j] * p[8 * sp + 2 * j + 1]);
                    const float nbi = fmaf(-b2r[j], p[8 * sp + 2 * j + 1], -b2i[j] * p[8 * sp + 2 * j]);  // -Im beta
                    const f2_t br2 = f2_pack(br, br), nbi2 = f2_pack(nbi, nbi);
#pragma unroll
                    for (int i = 0; i < 2; ++i) o2[i] = f2_fma(br2, gr[j][i], f2_fma(nbi2, gi[j][i], o2[i]));
                    if (ETA) dn = fmaf(br, er[j], fmaf(nbi, ei[j], dn));
                }
                float o[4];
                f2_unpack(o2[0], o[0], o[1]);
                f2_unpack(o2[1], o[2], o[3]);
#pragma unroll
                for (int off = LG; off < 32; off <<= 1) {
#pragma unroll
                    for (int i = 0; i < 4; ++i) o[i] += __shfl_xor_sync(FULL, o[i], off);
                    if (ETA) dn += __shfl_xor_sync(FULL, dn, off);
                }
                if (LG == 32 || lane < LG) st_cluster(uo + sp * 4 * R, o[0], o[1], o[2], o[3]);
                if (ETA && lane == 0) st_cluster(ud + sp * 4, dn);
            }
            xp += 2 * R;
            zp += 4 * R;
        };
        // positions [ow PT, ow PT + PT) of the tile are written by CTA ow: their partials are
        // asynchronous stores into its shared memory
        for (int ow = 0; ow * PT < tn; ++ow) {
            uint32_t uo = G > 1 ? mapa_u32(ao, ow) : ao, ud = G > 1 ? mapa_u32(ad, ow) : ad;
            const int te = min(tn, ow * PT + PT);
            int tt = ow * PT;
            for (; tt + 1 < te; tt += 2, uo += 8 * R, ud += 8) step2(uo, ud);
            if (tt < te) step(uo, ud);
        }
    };

    // Each role runs its own loop (so that no role's registers stay live in another's);
    // all of them pass the same nt + 2 barriers.
    if (warp < nwc) {
        csync();
        for (int kk = 0; kk <= nt; ++kk) {
            if (kk < nt) compute(kk);
            csync();
        }
    } else {
        prologue(0);
        csync();
        for (int kk = 0; kk <= nt; ++kk) {
            if (kk + 1 < nt) prologue(kk + 1);
            if (kk >= 1) output(kk - 1);
            csync();
        }
    }

    // ---- final state: X = B Y and eta = B e for this warp's modes; rank 0 adds the conv tails
    if (a.final_state) {
        float *fs = a.final_state + (size_t)unit * a.state_floats;
        const size_t RD = 2 * (size_t)R, plane = (size_t)M * RD;
        if (warp < nwc) {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int m = mbase + j;
                if (m >= M) continue;
                const float2 bb = *reinterpret_cast<const float2 *>(a.Bvec + ((size_t)h * M + m) * 2);
                float xr[4], xi[4], yr[4], yi[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    float a0, a1, b0, b1, c0, c1, d0, d1;
                    f2_unpack(ur[j][i / 2], a0, a1);
                    f2_unpack(ui[j][i / 2], b0, b1);
                    f2_unpack(gr[j][i / 2], c0, c1);
                    f2_unpack(gi[j][i / 2], d0, d1);
                    const float yu_r = i & 1 ? a1 : a0, yu_i = i & 1 ? b1 : b0;
                    const float yg_r = i & 1 ? c1 : c0, yg_i = i & 1 ? d1 : d0;
                    xr[i] = bb.x * yu_r - bb.y * yu_i;
                    xi[i] = bb.x * yu_i + bb.y * yu_r;
                    yr[i] = bb.x * yg_r - bb.y * yg_i;
                    yi[i] = bb.x * yg_i + bb.y * yg_r;
                }
                float *rr = fs + (size_t)m * RD + 4 * gl, *ri = fs + plane + (size_t)m * RD + 4 * gl;
                *reinterpret_cast<float4 *>(rr) = make_float4(xr[0], xr[1], xr[2], xr[3]);
                *reinterpret_cast<float4 *>(ri) = make_float4(xi[0], xi[1], xi[2], xi[3]);
                *reinterpret_cast<float4 *>(rr + R) = make_float4(yr[0], yr[1], yr[2], yr[3]);
                *reinterpret_cast<float4 *>(ri + R) = make_float4(yi[0], yi[1], yi[2], yi[3]);
                if (gl == 0) {
                    fs[2 * plane + m] = bb.x * er[j] - bb.y * ei[j];
                    fs[2 * plane + M + m] = bb.x * ei[j] + bb.y * er[j];
                }
            }
        } else if (pw == 0 && rank == 0) {
            float *tq = fs + 2 * plane + 2 * M;
            float *tk = tq + (size_t)(W - 1) * R;
            for (int i = lane; i < (W - 1) * R; i += 32) {
                const int r = i / R, c = i % R, p = N - (W - 1) + r;
                tq[i] = p >= 0 ? __bfloat162float(qg[(size_t)p * row_qk + c]) : 0.f;
                tk[i] = p >= 0 ? __bfloat162float(kg[(size_t)p * row_qk + c]) : 0.f;
            }
            const size_t used = 2 * plane + 2 * (size_t)M + 2 * (size_t)(W - 1) * R;
            for (size_t i = used + lane; i < a.state_floats; i += 32) fs[i] = 0.f;
        }
    }
}

namespace {

template <int R, bool ETA>
cudaError_t launch_modes_t(const PrefillArgs &a, int G, int nwc, cudaStream_t st) {
    auto kern = seq_modes_kernel<R, ETA>;
    const size_t smem = modes_layout(R, nwc, G).bytes;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)G * (unsigned)(a.B * a.H), 1, 1);
    cfg.blockDim = dim3((unsigned)(nwc + SM_HELP) * 32, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)G;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, a, G, nwc);
}

template <int R>
cudaError_t launch_modes_r(const PrefillArgs &a, int G, int nwc, cudaStream_t st) {
    return (a.flags & IDA_READOUT_ETA) ? launch_modes_t<R, true>(a, G, nwc, st)
                                       : launch_modes_t<R, false>(a, G, nwc, st);
}

}  // namespace

// Takes bf16 inputs with R = d in {32, 64, 128} and M <= 8 * 4 * (modes per warp).  Picks
// the compute warps per CTA (4, else 2 or 1 when the grid would not fill the SMs) and the
// cluster size G (a power of two) covering the modes.  Returns false (nothing launched)
// for other shapes.
bool launch_seq_modes(const PrefillArgs &a, cudaStream_t st, int num_sms, ida_status &s, std::string &why) {
    if (a.dtype != IDA_BF16 || a.R != a.d || (a.R != 32 && a.R != 64 && a.R != 128) || a.W > 4) return false;
    const int mpw = 4 * (32 / (a.R / 4));
    const int wpu = (a.M + mpw - 1) / mpw;  // compute warps per unit
    const long units = (long)a.B * a.H;
    int nwc = 4;
    while (nwc > 1 && units * ((wpu + nwc - 1) / nwc) < num_sms && (wpu + nwc / 2 - 1) / (nwc / 2) <= 8) nwc /= 2;
    int G = 1;  // a power of two; CTAs past the last mode carry only inert modes
    while (G * nwc < wpu) G *= 2;
    if (G > 8) return false;
    if (units * G > 0x7fffffffL) return false;
    cudaError_t e;
    if (a.R == 32)
        e = launch_modes_r<32>(a, G, nwc, st);
    else if (a.R == 64)
        e = launch_modes_r<64>(a, G, nwc, st);
    else
        e = launch_modes_r<128>(a, G, nwc, st);
    if (e != cudaSuccess) {
        s = IDA_ERR_CUDA;
        why = std::string("sequential prefill launch: ") + cudaGetErrorString(e);
    } else {
        s = IDA_OK;
    }
    return true;
}

}  // namespace ida
