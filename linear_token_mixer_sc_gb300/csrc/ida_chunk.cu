// ida_chunk.cu -- chunked prefill on the tcgen05 tensor cores.
//
// The recurrence X_t = lambda X_{t-1} + B z_t and the readout
// o_t = Re(xi(q_t)^T U_t^T Gamma_t) of "Interdomain Attention: Beyond
// Token-Level Key-Value Memory" (German technical summary, "Skalierbare
// Implementierung"; state shapes from the paper's Fig. 1 caption) are
// re-associated over chunks of C = 64 positions.  With X_p the state before
// a chunk and i, j in [0, C) local positions:
//
//   P[i,m]   = xi(q_i) . U_p[m]                           (state read-out)
//   G[i,j]   = xi(q_i) . kt_j,     G'[i,k] = G[i,i-k] for k <= i, else 0
//   L[i,m]   = sum_k G'[i,k] lambda_m^k = sum_{j<=i} lambda_m^{i-j} G[i,j]
//   a[i,m]   = lambda_m^{i+1} P[i,m] + B_m L[i,m]         (= xi(q_i) . U_i[m])
//   A2'[i,k] = Re sum_m a[i,m] B_m lambda_m^k,  A2[i,j] = A2'[i,i-j] (j <= i)
//   o_i      = sum_j A2[i,j] vt_j + Re sum_m a[i,m] lambda_m^{i+1} Gamma_p[m]
//   X_end    = lambda^L X_p + sum_j B lambda^{L-1-j} z_j   (L = chunk length)
//
// Skewing the Gram matrix (G' and A2') makes every intra-chunk decay factor
// a power lambda^k with 0 <= k < C, so no operand grows beyond |lambda| <= 1
// for any stable mode.  Every contraction above is an MMA:
//
//   G     [128 x 64]  = [xiQ ; Kt] . Kt^T          kind::f16  (rows 64..127 unused)
//   P^T   [2M x 64]   = U . xiQ^T                  kind::tf32, U read from TMEM
//   L^T   [2M x 64]   = T_L . G'^T                 kind::f16
//   A2'   [128 x 64]  = Ya . T_A^T                 kind::f16  (rows 64..127 unused)
//   O1    [128 x 64]  = Vt^T . A2^T                kind::f16  (lanes = value channel)
//   O2    [128 x 64]  = Gamma^T . a'^T             kind::tf32, Gamma^T read from TMEM
//   U    += Coef . Kt^T-chunk,  Gamma^T += Vt^T . Coef^T      kind::f16
//
// The complex state never leaves the SM: U (lanes = mode planes 2m / 2m+1 for
// Re / Im, columns = key channels) and Gamma^T (lanes = value channels,
// columns = mode planes) are fp32 MMA accumulators in TMEM; each chunk first
// scales them by lambda^L on the CUDA cores, then accumulates the chunk's
// contribution with two MMAs.  Operands that are unbounded (Ya, A2) are
// stored as fp16 with a power-of-two scale per column / row, undone exactly
// in the matching table or epilogue.
//
// One CTA of 256 threads per (b,h) unit.  Warp w reaches TMEM lanes
// 32*(w%4) .. +31, so warps w and w+4 share a lane quarter and split the
// columns (or positions) of every TMEM-side stage; thread 0 issues the MMAs.
// The raw q, k, v rows of a chunk (with the W-1 = 3 row conv halo) arrive by
// TMA one chunk ahead, into shared memory that is dead between the output
// MMAs and the next a / Ya stage; out-of-range rows (before position 0 or
// past N) are zero-filled by the copy itself.  Every wait (MMA completion or
// TMA arrival) is bounded; on timeout the kernel records kErrWaitTimeout,
// stops issuing, waits (bounded) for its own copy in flight, frees its TMEM
// and returns.
#include <cuda.h>
#include <cuda_fp16.h>

#include <algorithm>
#include <functional>
#include <mutex>
#include <queue>
#include <vector>
#include <string>

#include "ida_common.cuh"
#include "tc_sm103.cuh"

namespace ida {

using namespace tc;

constexpr int CH = 64;       // positions per chunk
constexpr int HALO = 3;      // conv halo rows staged before a chunk (W <= 4)
constexpr int NTH = 256;     // threads per CTA
constexpr int MP = 128;      // mode planes (2M, M = 64)
constexpr int PADLBO = 144;  // core-matrix stride along K for column-wise (transposed) writers

__host__ __device__ constexpr int align1k(int x) { return (x + 1023) / 1024 * 1024; }

template <int R, int D>
struct ChunkSmem {
    // All MMA operands are K-major, no-swizzle core-matrix layouts (8 rows x 16 B).
    static constexpr int XQ16 = 0;                               // [64][R] f16   LBO 128, SBO 16R
    static constexpr int KT16 = XQ16 + CH * R * 2;               // [64][R] f16   (follows XQ16: A rows 64..127)
    static constexpr int XQ32 = KT16 + CH * R * 2;               // [64][R] tf32  LBO 128, SBO 32R; skew scratch
    static constexpr int ZT16 = XQ32 + CH * R * 4;               // [R+D][64] f16 LBO 144, SBO 1168
    static constexpr int ZT_SBO = 8 * PADLBO + 16;               // +16: row blocks start on different banks
    static constexpr int GP16 = ZT16 + (R + D) / 8 * ZT_SBO;     // [64][64] f16  LBO 128, SBO 1024; S5 scratch
    static constexpr int A216 = GP16 + CH * CH * 2;              // [64][64] f16
    static constexpr int TL16 = A216 + CH * CH * 2;              // [128][64] f16 LBO 128, SBO 1024
    static constexpr int CF16 = TL16 + MP * CH * 2;              // [128][64] f16
    static constexpr int TA16 = align1k(CF16 + MP * CH * 2);     // [64][128] f16 LBO 144, SBO 2304
    static constexpr int TY_SBO = 16 * PADLBO;
    static constexpr int YA16 = TA16 + 8 * TY_SBO;               // [64][128] f16 LBO 144, SBO 2304
    static constexpr int AP32 = YA16 + 8 * TY_SBO;               // [64][128] tf32 LBO 144, SBO 4608
    static constexpr int AP_SBO = 32 * PADLBO;
    static constexpr int MISC = AP32 + 8 * AP_SBO;
    // raw bf16 rows of the next chunk, staged over YA16 / AP32 (dead while they land)
    static constexpr int RAWQ_BYTES = align1k((CH + HALO) * R * 2);
    static constexpr int RAWQ = YA16;                            // [67][R] bf16, row r = position t0-3+r
    static constexpr int RAWK = RAWQ + RAWQ_BYTES;               // [67][R] bf16
    static constexpr int RAWV = RAWK + RAWQ_BYTES;               // [64][D] bf16
    static_assert(YA16 % 1024 == 0 && RAWV + CH * D * 2 <= MISC, "raw staging must fit over YA16/AP32");
    static_assert(GP16 % 128 == 0 && A216 == GP16 + CH * CH * 2 && CH * D * 2 <= 2 * CH * CH * 2,
                  "the [64][D] output tile is staged over GP16 / A216");
    static constexpr int BARS = MISC;                            // 8 mbarriers
    static constexpr int TSLOT = BARS + 64;
    static constexpr int OSC = TSLOT + 16;                       // [64] float: row scales of A2
    static constexpr int LAML = OSC + CH * 4;                    // [64] float2: lambda^L per mode
    static constexpr int SUML = LAML + 64 * 8;                   // [64] float2: sum_{k<L} lambda^k per mode
    static constexpr int GBLK = SUML + 64 * 8;                   // [64] float2: lambda^(64 fs), one block's decay
    static constexpr int NWS = GBLK + 64 * 8;                    // [R+D] float RMSNorm weights
    static constexpr int BSS = NWS + (R + D) * 4;                // [R+D] float RMSNorm biases
    static constexpr int TOTAL = BSS + (R + D) * 4;
    static_assert(TOTAL <= 227 * 1024, "shared memory budget");
};

// TMEM column map (512 columns allocated).
template <int R>
struct ChunkTmem {
    static constexpr uint32_t U = 0;     // [2M lanes][R]
    static constexpr uint32_t GT = R;    // [value lanes][2M]
    static constexpr uint32_t G = 256;   // [64 lanes][64], later A2'
    static constexpr uint32_t PT = 320;  // [2M lanes][64], later O1
    static constexpr uint32_t LT = 384;  // [2M lanes][64], later O2
    static constexpr uint32_t TAPS = 448;  // [lane][64]: conv taps (q then k) of channel block lane % (R/8)
};

// byte offset of element (row, k) in a K-major no-swizzle operand
__device__ __forceinline__ int kmaj_off(int row, int k, int esize, int lbo, int sbo) {
    const int T = 16 / esize;
    return (row >> 3) * sbo + (k / T) * lbo + (row & 7) * 16 + (k % T) * esize;
}

__device__ __forceinline__ float pow2i(int e) { return __int_as_float((127 + e) << 23); }

// exponent e >= 0 such that x * 2^-e <= 2^14 (fp16 headroom), for x >= 0
__device__ __forceinline__ int down_exp(float x) {
    if (!(x > 16384.f)) return 0;
    int ex = ((__float_as_int(x) >> 23) & 0xFF) - 127;  // floor(log2 x)
    int e = ex - 13;
    return e > 15 ? 15 : e;
}

// x rounded to the tf32 grid (10 mantissa bits), nearest with ties away from zero, as bits
__device__ __forceinline__ uint32_t tf32_bits(float x) { return (__float_as_uint(x) + 0x1000u) & 0xFFFFE000u; }

// the hardware tanh approximation (relative error about 2^-11, below the fp16 rounding of
// every operand built from it).  SiLU takes one such op: x sigmoid(x) = h + h tanh(h), h = x / 2
__device__ __forceinline__ float tanh_approx(float x) {
    float t;
    asm("tanh.approx.f32 %0, %1;" : "=f"(t) : "f"(x));
    return t;
}

// two fp32 in one 64-bit register for the packed fp32x2 instructions (each lane rounded
// like the scalar instruction)
typedef unsigned long long f2_t;
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

// v[pp] <- v[(pp + rot) % P] for all pp, by log2(P) conditional shifts (P a power of two)
template <int P, int Wd>
__device__ __forceinline__ void rotate_rows(uint32_t (&v)[P][Wd], int rot) {
#pragma unroll
    for (int sh = 1; sh < P; sh <<= 1) {
        const bool on = (rot & sh) != 0;
        uint32_t t[P][Wd];
#pragma unroll
        for (int pp = 0; pp < P; ++pp)
#pragma unroll
            for (int e = 0; e < Wd; ++e) t[pp][e] = on ? v[(pp + sh) % P][e] : v[pp][e];
#pragma unroll
        for (int pp = 0; pp < P; ++pp)
#pragma unroll
            for (int e = 0; e < Wd; ++e) v[pp][e] = t[pp][e];
    }
}

// two floats as one fp16 pair (lo in the low half), one conversion instruction
__device__ __forceinline__ uint32_t pack_h2(float lo, float hi) {
    const __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&h);
}

__device__ __forceinline__ void unpack_bf16x8(uint4 u, float x[8]) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        x[2 * e] = __uint_as_float(w[e] << 16);
        x[2 * e + 1] = __uint_as_float(w[e] & 0xFFFF0000u);
    }
}

__device__ __forceinline__ uint4 pack_f16x8(const float x[8]) {
    return make_uint4(pack_h2(x[0], x[1]), pack_h2(x[2], x[3]), pack_h2(x[4], x[5]), pack_h2(x[6], x[7]));
}

// Work split of a batch of sequences across CTAs.  Each unit's chunks are grouped into nb
// blocks of fs chunks (the last block may be shorter) and its blocks into ppu pieces: the
// first of q0 blocks, the others of q blocks; one CTA runs one piece.  The grid lists the
// later pieces of every unit before the first pieces, so that when there are more pieces
// than SMs the short first pieces fill in behind.  A piece not at the sequence start needs
// the state before its first block: the block state pass computes, from zero, the end
// state of each block before the unit's last piece, and the piece's CTA composes those of
// the blocks before it as it loads its start state.
struct SegPlan {
    int fs;   // chunks per block
    int nb;   // blocks per unit
    int q0;   // blocks in a unit's first piece
    int q;    // blocks in each later piece
    int ppu;  // pieces per unit
};

// Blocks per unit whose end states the state pass computes (all before the last piece).
__host__ __device__ inline int plan_state_blocks(const SegPlan &p) {
    return p.ppu > 1 ? p.q0 + (p.ppu - 2) * p.q : 0;
}

// FACT selects the Gram formulation; a CTA whose head takes the other one returns at once
// (the other instantiation, launched on the same plan, runs that piece).  EXT compiles in the
// options that the default call does not use: a given start state (state_in) and the l_2
// feature map; without it the kernel carries no code for them.
template <int R, int D, bool FACT, bool EXT>
__global__ void __launch_bounds__(NTH, 1)
    chunk_prefill_kernel(PrefillArgs a, const __grid_constant__ CUtensorMap tm_q,
                         const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                         const __grid_constant__ CUtensorMap tm_o, SegPlan plan, const float *seg_start) {
    using S = ChunkSmem<R, D>;
    using T = ChunkTmem<R>;
    extern __shared__ __align__(1024) unsigned char sm[];
    const uint32_t s16 = smem_u32(sm) >> 4;  // shared base for MMA descriptors
    // mbarriers: 0 G, 1 L^T, 2 A2', 3 O2, 4 state update, 5 TMA, 6 P^T, 7 O1
    uint64_t *bar = reinterpret_cast<uint64_t *>(sm + S::BARS);
    uint32_t *tslot = reinterpret_cast<uint32_t *>(sm + S::TSLOT);
    float *osc = reinterpret_cast<float *>(sm + S::OSC);
    float2 *laml = reinterpret_cast<float2 *>(sm + S::LAML);
    float2 *suml = reinterpret_cast<float2 *>(sm + S::SUML);
    float2 *gblk = reinterpret_cast<float2 *>(sm + S::GBLK);
    float *nws = reinterpret_cast<float *>(sm + S::NWS);
    float *bss = reinterpret_cast<float *>(sm + S::BSS);

    // The two instantiations are launched back to back, the second (skewed) as a programmatic
    // dependent of the first: every factorised CTA releases it at once, and every skewed CTA
    // waits for the factorised grid to complete before it does anything.  The skewed grid's
    // launch then overlaps the factorised one, and its completion still implies that of both.
    if constexpr (FACT)
        asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    else
        asm volatile("griddepcontrol.wait;" ::: "memory");
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int q4 = warp & 3, hsel = warp >> 2;        // TMEM lane quarter, column / position half
    const int tl = 32 * q4 + lane;                    // my TMEM lane
    const uint32_t lane_base = (uint32_t)(32 * q4) << 16;
    const int H = a.H, N = a.N, M = 64, W = a.W;
    const int nchunks = (N + CH - 1) / CH;
    const size_t sqk = (size_t)H * R;
    const __nv_bfloat16 *gq = reinterpret_cast<const __nv_bfloat16 *>(a.q);
    const __nv_bfloat16 *gk = reinterpret_cast<const __nv_bfloat16 *>(a.k);
    const uint32_t raw_bytes = 2u * (CH + HALO) * R * 2 + (uint32_t)CH * D * 2;
    // my mode plane in the lane-side stages: plane tl = 2m + (0: Re, 1: Im)
    const int mm = tl >> 1, is_im = tl & 1;

    // TMA destinations need 1 KB-aligned shared memory; refuse rather than fault
    if ((smem_u32(sm) & 1023u) != 0u) {
        if (tid == 0) report_error(a.err, kErrShape);
        return;
    }

    // ---- this CTA's piece: chunks [c_begin, c_end) of unit `unit` ---------------------
    const int nlater = a.B * a.H * (plan.ppu - 1);  // later pieces come first in the grid
    const int unit = (int)blockIdx.x < nlater ? (int)blockIdx.x / (plan.ppu - 1) : (int)blockIdx.x - nlater;
    const int pc = (int)blockIdx.x < nlater ? 1 + (int)blockIdx.x % (plan.ppu - 1) : 0;
    const int j0 = pc == 0 ? 0 : plan.q0 + (pc - 1) * plan.q;
    const int j1 = min(plan.nb, pc == 0 ? plan.q0 : j0 + plan.q);
    const int b = unit / H, h = unit % H;
    const int c_begin = j0 * plan.fs, c_end = min(nchunks, j1 * plan.fs);
    const size_t base_qk = ((size_t)b * N * H + h) * R;
    const float lam_r = a.lambda[((size_t)h * M + mm) * 2], lam_i = a.lambda[((size_t)h * M + mm) * 2 + 1];
    const float b_r = a.Bvec[((size_t)h * M + mm) * 2], b_i = a.Bvec[((size_t)h * M + mm) * 2 + 1];
    // Factorised Gram path: lambda^(i-j) = lambda^i lambda^-j, the table T[j] = B lambda^-j
    // (times 2^-fsc per mode) held in fp16.  Taken when every mode of the head keeps T
    // within fp16 normals with room for the Ya column scaling: |lambda| <= 1,
    // |lambda|^-63 <= 2^8 and 2^-8 <= |B| <= 2^8.  Otherwise the skewed-Gram path (tables
    // lambda^k, bounded by 1 for any stable mode) serves the piece.
    const float m2 = lam_r * lam_r + lam_i * lam_i, bb2 = b_r * b_r + b_i * b_i;
    const float lg63 = -31.5f * log2f(m2);  // log2 |lambda|^-63
    const bool fact = __syncthreads_and(m2 > 0.f && m2 <= 1.001f && lg63 <= 8.f && bb2 >= 1.f / 65536.f &&
                                        bb2 <= 65536.f) != 0;
    if (fact != FACT || c_begin >= c_end) return;  // the other instantiation runs this piece
    // lambda^(32 hsel + 16 is_im + 1): the decay at this lane's first position in the a / Ya stage
    float w0r = lam_r, w0i = lam_i;
    {
        float qr = lam_r, qi = lam_i;
#pragma unroll
        for (int sq = 0; sq < 4; ++sq) {  // lambda^16
            const float nr = qr * qr - qi * qi, ni = 2.f * qr * qi;
            qr = nr;
            qi = ni;
        }
        if (is_im) {
            const float nr = w0r * qr - w0i * qi, ni = w0r * qi + w0i * qr;
            w0r = nr;
            w0i = ni;
        }
        const float q2r = qr * qr - qi * qi, q2i = 2.f * qr * qi;  // lambda^32
        if (hsel) {
            const float nr = w0r * q2r - w0i * q2i, ni = w0r * q2i + w0i * q2r;
            w0r = nr;
            w0i = ni;
        }
    }

    // ---- set-up: barriers, TMEM ---------------------------------------------------
    if (tid == 0) {
        for (int i = 0; i < 8; ++i) mbar_init(&bar[i], 1);
        fence_mbar_init();
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
        tma_prefetch_desc(&tm_o);
    }
    if (warp == 0) {
        tmem_alloc(tslot, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tb = *tslot;

    bool ok = true;
    int it = 0;           // chunks this CTA has run so far: the phase parity of every barrier
    int tma_pending = 0;  // TMA copies issued and not yet waited for
    uint32_t tma_par = 0;  // the bar[5] phase parity that the copy in flight completes
    int ci = 0;
    {
        const int fsc = FACT ? (int)ceilf(0.5f * log2f(bb2) + lg63 + 0.01f) + 1 : 0;  // T max <= 1/2
        const float fS = pow2i(fsc);
        // lambda^(2 ib) with ib = 32 hsel + 16 is_im (this lane's first position in the a / Ya
        // stage) and lambda^2: the running lambda^(2i) of the factorised path
        float v0r = 1.f, v0i = 0.f;
        const float l2r = lam_r * lam_r - lam_i * lam_i, l2i = 2.f * lam_r * lam_i;
        {
            float qr = lam_r, qi = lam_i;
#pragma unroll
            for (int sq = 0; sq < 5; ++sq) {  // lambda^32
                const float nr = qr * qr - qi * qi, ni = 2.f * qr * qi;
                qr = nr;
                qi = ni;
            }
            if (is_im) {
                v0r = qr;
                v0i = qi;
            }
            if (hsel) {
                const float q2r = qr * qr - qi * qi, q2i = 2.f * qr * qi;  // lambda^64
                const float nr = v0r * q2r - v0i * q2i, ni = v0r * q2i + v0i * q2r;
                v0r = nr;
                v0i = ni;
            }
        }
        for (int x = tid; x < R + D; x += NTH) {
            nws[x] = a.norm_w[(size_t)h * (R + D) + x];
            bss[x] = a.bias[(size_t)h * (R + D) + x];
        }
        if (hsel == 0) {
            // T_L row (plane tl): component of lambda_m^k, k = 0..63 (skewed path) or of the
            // factorised table; Coef row: component of B_m lambda_m^(C-1-j); T_A column tl =
            // T_L row (unscaled).
            float pr = 1.f, pi = 0.f, sr = 0.f, si = 0.f;
            __align__(16) __half tl16[CH], cf[CH];
    #pragma unroll
            for (int k = 0; k < CH; ++k) {
                sr += pr;
                si += pi;
                tl16[k] = __float2half_rn(is_im ? pi : pr);
                const float cr = b_r * pr - b_i * pi, ci = b_r * pi + b_i * pr;
                cf[CH - 1 - k] = __float2half_rn(is_im ? ci : cr);
                const float nr = pr * lam_r - pi * lam_i, ni = pr * lam_i + pi * lam_r;
                pr = nr;
                pi = ni;
            }
            // lambda^C by repeated squaring (fewer roundings than the running product)
            float qr = lam_r, qi = lam_i;
    #pragma unroll
            for (int sq = 0; sq < 6; ++sq) {
                const float nr = qr * qr - qi * qi, ni = 2.f * qr * qi;
                qr = nr;
                qi = ni;
            }
            if (!is_im) {
                laml[mm] = make_float2(qr, qi);  // lambda^C
                suml[mm] = make_float2(sr, si);  // sum_{k<C} lambda^k
                // lambda^(C fs) = (lambda^C)^fs, the decay across one block
                float gr = 1.f, gi = 0.f, pr = qr, pi = qi;
                for (unsigned e = (unsigned)plan.fs; e; e >>= 1) {
                    if (e & 1u) {
                        const float nr = gr * pr - gi * pi, ni = gr * pi + gi * pr;
                        gr = nr;
                        gi = ni;
                    }
                    const float nr = pr * pr - pi * pi, ni = 2.f * pr * pi;
                    pr = nr;
                    pi = ni;
                }
                gblk[mm] = make_float2(gr, gi);
            }
            if constexpr (FACT) {
                // factorised table row: component of B lambda^-j 2^-fsc, j = 0..63
                const float ir = lam_r / m2, ii = -lam_i / m2;  // lambda^-1
                float wr = b_r * pow2i(-fsc), wi = b_i * pow2i(-fsc);
#pragma unroll
                for (int j = 0; j < CH; ++j) {
                    tl16[j] = __float2half_rn(is_im ? wi : wr);
                    const float nr = wr * ir - wi * ii, ni = wr * ii + wi * ir;
                    wr = nr;
                    wi = ni;
                }
            }
    #pragma unroll
            for (int k8 = 0; k8 < CH / 8; ++k8) {
                *reinterpret_cast<uint4 *>(sm + S::TL16 + kmaj_off(tl, k8 * 8, 2, 128, 1024)) =
                    *reinterpret_cast<const uint4 *>(&tl16[k8 * 8]);
                *reinterpret_cast<uint4 *>(sm + S::CF16 + kmaj_off(tl, k8 * 8, 2, 128, 1024)) =
                    *reinterpret_cast<const uint4 *>(&cf[k8 * 8]);
            }
    #pragma unroll
            for (int k = 0; k < CH; ++k)
                *reinterpret_cast<__half *>(sm + S::TA16 + kmaj_off(k, tl, 2, PADLBO, S::TY_SBO)) = tl16[k];
        }
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        {
            // start state: X_in (zero, or the caller's state before position 0) at the sequence
            // start, else the state before block j0,
            //   X = g^j0 X_in + sum_{j < j0} g^(j0-1-j) X_local(j),  g = lambda^(C fs) per mode,
            // by Horner over the block end states ([R+128 columns][128 lanes] floats, columns as
            // in TMEM); U columns pair Re / Im across lanes 2m, 2m+1, Gamma^T columns across
            // columns R+2m, R+2m+1.  By column half.
            // The loads of one block state are issued together (the groups' values land in
            // registers, so one memory latency per block); the running sum lives in TMEM.
            constexpr int NG = (R + MP) / 32;  // my 16-column groups: columns 32 g + 16 hsel
            const float *xs = seg_start + (size_t)unit * plan_state_blocks(plan) * (size_t)(R + MP) * 128;
            const float2 gu = gblk[mm];
            const float gus = is_im ? gu.y : -gu.y;  // own(g z) = z_own Re g + z_partner s Im g
            const bool has_in = EXT && a.state_in != nullptr;
            if (has_in) {
                // X_in in the same layout: U[m][c] of plane tl at column c; Gamma^T (value lane
                // tl) at column R + 2m (Re) / R + 2m + 1 (Im)
                const float *xin = a.state_in + (size_t)unit * a.state_floats;
                const size_t RDs = R + D, plane = (size_t)64 * RDs;
                float x[NG][16];
    #pragma unroll
                for (int g = 0; g < NG; ++g) {
                    const int c0 = 32 * g + 16 * hsel;
    #pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const int c = c0 + i;
                        if (c < R) {
                            x[g][i] = xin[(is_im ? plane : 0) + (size_t)mm * RDs + c];
                        } else {
                            const int pl = c - R;
                            x[g][i] = tl < D ? xin[((pl & 1) ? plane : 0) + (size_t)(pl >> 1) * RDs + R + tl] : 0.f;
                        }
                    }
                }
    #pragma unroll
                for (int g = 0; g < NG; ++g) tmem_st16(tb + lane_base + 32 * g + 16 * hsel, x[g]);
                tmem_wait_st();
            }
            for (int j = 0; j < (j0 > 0 ? j0 : (has_in ? 0 : 1)); ++j) {
                float x[NG][16];
    #pragma unroll
                for (int g = 0; g < NG; ++g) {
                    const float *xg = xs + (size_t)j * (R + MP) * 128 + (size_t)(32 * g + 16 * hsel) * 128 + tl;
    #pragma unroll
                    for (int i = 0; i < 16; ++i) x[g][i] = j0 > 0 ? xg[(size_t)i * 128] : 0.f;
                }
                if (j > 0 || has_in) {
    #pragma unroll
                    for (int g = 0; g < NG; ++g) {
                        const int c0 = 32 * g + 16 * hsel;
                        float z[16];
                        tmem_ld16(tb + lane_base + c0, z);
                        tmem_wait_ld();
                        if (c0 < R) {
    #pragma unroll
                            for (int i = 0; i < 16; ++i) {
                                const float zp = __shfl_xor_sync(0xffffffffu, z[i], 1);
                                x[g][i] = fmaf(z[i], gu.x, fmaf(zp, gus, x[g][i]));
                            }
                        } else {
    #pragma unroll
                            for (int i = 0; i < 16; i += 2) {
                                const float2 gg = gblk[(c0 - R + i) >> 1];
                                const float zr = z[i], zi = z[i + 1];
                                x[g][i] = fmaf(gg.x, zr, fmaf(-gg.y, zi, x[g][i]));
                                x[g][i + 1] = fmaf(gg.x, zi, fmaf(gg.y, zr, x[g][i + 1]));
                            }
                        }
                    }
                }
    #pragma unroll
                for (int g = 0; g < NG; ++g) tmem_st16(tb + lane_base + 32 * g + 16 * hsel, x[g]);
                tmem_wait_st();
            }
            if (hsel == 0) {
                // conv taps of channels 8*(tl % (R/8)) .. +7, right-aligned: column 32*which + 4*e + jj
                // multiplies position i - 3 + jj (zero for jj < 4 - W)
                const int cbl = tl % (R / 8);
    #pragma unroll
                for (int which = 0; which < 2; ++which) {
                    const float *cwg = a.conv_w + ((size_t)(which * H + h) * R + 8 * cbl) * W;
                    float t32[32];
    #pragma unroll
                    for (int e = 0; e < 8; ++e)
    #pragma unroll
                        for (int jj = 0; jj < 4; ++jj) t32[4 * e + jj] = jj >= 4 - W ? cwg[e * W + jj - (4 - W)] : 0.f;
                    tmem_st16(tb + lane_base + T::TAPS + 32 * which, t32);
                    tmem_st16(tb + lane_base + T::TAPS + 32 * which + 16, t32 + 16);
                }
            }
            tmem_wait_st();
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        tma_pending = 1;
        if (tid == 0) {
            const int tb0 = c_begin * CH;
            mbar_arrive_expect_tx(&bar[5], raw_bytes);
            tma_load_4d(sm + S::RAWQ, &tm_q, 0, h, tb0 - HALO, b, &bar[5]);
            tma_load_4d(sm + S::RAWK, &tm_k, 0, h, tb0 - HALO, b, &bar[5]);
            tma_load_4d(sm + S::RAWV, &tm_v, 0, h, tb0, b, &bar[5]);
        }


        // eta of my mode at the piece start, lambda^t_begin eta_in + B sum_{k < t_begin} lambda^k
        // (hsel == 0, Re thread)
        float eta_r = 0.f, eta_i = 0.f;
        if (hsel == 0 && !is_im) {
            if (EXT && a.state_in) {
                const float *ein = a.state_in + (size_t)unit * a.state_floats + (size_t)2 * 64 * (R + D);
                eta_r = ein[mm];
                eta_i = ein[64 + mm];
            }
            const float2 ll = laml[mm], sl = suml[mm];
            for (int c = 0; c < c_begin; ++c) {
                const float er = ll.x * eta_r - ll.y * eta_i + b_r * sl.x - b_i * sl.y;
                const float ei = ll.x * eta_i + ll.y * eta_r + b_r * sl.y + b_i * sl.x;
                eta_r = er;
                eta_i = ei;
            }
        }
        int ya_exp = 0;  // scale exponent of my T_A column currently stored
        ci = c_begin;
        for (; ci < c_end; ++ci, ++it) {
            const int t0 = ci * CH;
            const int L = min(CH, N - t0);
            const uint32_t par = it & 1;

            // this chunk's raw rows (the previous chunk's state-update MMAs, which read ZT16 and
            // CF16, are waited for inside the prologue, just before ZT16 is rewritten)
            ok = mbar_wait(&bar[5], par);
            if (ok) tma_pending = 0;
            tc_fence_after();
            if (__syncthreads_or(!ok)) break;
            if (EXT && ci == 0 && a.state_in) {
                // conv halo of the first chunk: the raw rows before position 0 are the initial
                // state's tails (the copy zero-filled them)
                const float *tq = a.state_in + (size_t)unit * a.state_floats + (size_t)2 * 64 * (R + D + 1);
                const float *tk = tq + (size_t)(W - 1) * R;
                __nv_bfloat16 *rq = reinterpret_cast<__nv_bfloat16 *>(sm + S::RAWQ);
                __nv_bfloat16 *rk = reinterpret_cast<__nv_bfloat16 *>(sm + S::RAWK);
                for (int x = tid; x < HALO * R; x += NTH) {
                    const int r = x / R, c = x % R, j = r - HALO + (W - 1);  // tail row of position r - 3
                    if (j >= 0) {
                        rq[x] = __float2bfloat16_rn(tq[(size_t)j * R + c]);
                        rk[x] = __float2bfloat16_rn(tk[(size_t)j * R + c]);
                    }
                }
                __syncthreads();
            }

            // ---- S1: prologue, thread = (8-channel block, block of consecutive positions)
            // query / key: R/8 channel blocks x (64 R/8 / 256) positions per thread
            constexpr int CBQ = R / 8, PPQ = CH * CBQ / NTH;
            uint32_t hk[PPQ][4];  // this thread's key rows (fp16 pairs), kept for the Z^T rows
            {
                const int cb = tid % CBQ, i0 = (tid / CBQ) * PPQ, c0 = 8 * cb;
                // rows are stored rotated: at step pp this thread writes position i0 + (pp + rot) % PPQ,
                // so the channel-block threads of one position hit different banks
                const int rot = cb % PPQ;
                float nwk[8], bsk[8];
                *reinterpret_cast<float4 *>(nwk) = *reinterpret_cast<const float4 *>(nws + c0);
                *reinterpret_cast<float4 *>(nwk + 4) = *reinterpret_cast<const float4 *>(nws + c0 + 4);
                *reinterpret_cast<float4 *>(bsk) = *reinterpret_cast<const float4 *>(bss + c0);
                *reinterpret_cast<float4 *>(bsk + 4) = *reinterpret_cast<const float4 *>(bss + c0 + 4);
                float fk[PPQ][8];
                // taps of my channel block (TMEM lane tl holds block tl % CBQ == cb), q then k, as
                // channel pairs: tp[which][e2][jj] = (tap jj of channel 2 e2, of channel 2 e2 + 1)
                f2_t tp[2][4][4];
                {
                    float w8[2][32];
    #pragma unroll
                    for (int which = 0; which < 2; ++which) {
                        tmem_ld16(tb + lane_base + T::TAPS + 32 * which, w8[which]);
                        tmem_ld16(tb + lane_base + T::TAPS + 32 * which + 16, w8[which] + 16);
                    }
                    tmem_wait_ld();
    #pragma unroll
                    for (int which = 0; which < 2; ++which)
    #pragma unroll
                        for (int e2 = 0; e2 < 4; ++e2)
    #pragma unroll
                            for (int jj = 0; jj < 4; ++jj)
                                tp[which][e2][jj] = f2_pack(w8[which][8 * e2 + jj], w8[which][8 * e2 + 4 + jj]);
                }
    #pragma unroll
                for (int which = 0; which < 2; ++which) {
                    const unsigned char *raw = sm + (which == 0 ? S::RAWQ : S::RAWK);
                    // rows i0 .. i0+PPQ+2 of the staged tile = positions i0-3 .. i0+PPQ-1; the conv
                    // of channel pairs in packed fp32x2 arithmetic
                    f2_t g[PPQ][4];
    #pragma unroll
                    for (int pp = 0; pp < PPQ; ++pp)
    #pragma unroll
                        for (int e2 = 0; e2 < 4; ++e2) g[pp][e2] = 0ull;
    #pragma unroll
                    for (int r = 0; r < PPQ + HALO; ++r) {
                        const uint4 u = *reinterpret_cast<const uint4 *>(raw + ((size_t)(i0 + r) * R + c0) * 2);
                        const uint32_t wv[4] = {u.x, u.y, u.z, u.w};
                        f2_t x2[4];
    #pragma unroll
                        for (int e2 = 0; e2 < 4; ++e2)
                            x2[e2] = f2_pack(__uint_as_float(wv[e2] << 16), __uint_as_float(wv[e2] & 0xFFFF0000u));
                        // tile row r holds position i0 + r - 3: right-aligned tap jj = r - pp of position pp
    #pragma unroll
                        for (int pp = 0; pp < PPQ; ++pp) {
                            const int jj = r - pp;
                            if (jj >= 0 && jj < 4)
    #pragma unroll
                                for (int e2 = 0; e2 < 4; ++e2) g[pp][e2] = f2_fma(tp[which][e2][jj], x2[e2], g[pp][e2]);
                        }
                    }
                    // SiLU (x sigmoid x = h + h tanh h, h = x / 2) and the squared norm, pairwise
                    float acc[PPQ];
                    const f2_t half2 = f2_pack(0.5f, 0.5f);
    #pragma unroll
                    for (int pp = 0; pp < PPQ; ++pp) {
                        f2_t s2 = 0ull;
    #pragma unroll
                        for (int e2 = 0; e2 < 4; ++e2) {
                            const f2_t h2 = f2_mul(g[pp][e2], half2);
                            float hl, hh;
                            f2_unpack(h2, hl, hh);
                            const f2_t t2 = f2_pack(tanh_approx(hl), tanh_approx(hh));
                            g[pp][e2] = f2_fma(h2, t2, h2);
                            s2 = f2_fma(g[pp][e2], g[pp][e2], s2);
                        }
                        float sl, sh;
                        f2_unpack(s2, sl, sh);
                        acc[pp] = sl + sh;
                    }
                    float f[PPQ][8];
    #pragma unroll
                    for (int pp = 0; pp < PPQ; ++pp) {
    #pragma unroll
                        for (int o = 1; o < CBQ; o <<= 1) acc[pp] += __shfl_xor_sync(0xffffffffu, acc[pp], o);
                        // squared norm, or the l_2 norm (acc rsqrt(acc), zero for a zero row)
                        const float nrm = (EXT && (a.flags & IDA_FEAT_L2))
                                              ? (acc[pp] > 0.f ? acc[pp] * rsqrtf(acc[pp]) : 0.f)
                                              : acc[pp];
                        const float inv = (i0 + pp < L) ? __fdividef(1.f, nrm + IDA_EPS_FEAT) : 0.f;
                        const f2_t inv2 = f2_pack(inv, inv);
    #pragma unroll
                        for (int e2 = 0; e2 < 4; ++e2) f2_unpack(f2_mul(g[pp][e2], inv2), f[pp][2 * e2], f[pp][2 * e2 + 1]);
                    }
                    if (which == 0) {
                        // xi(q) rows: fp16 for the Gram MMA, tf32 for the state read-out MMA; row pp
                        // of the rotated set is position i0 + (pp + rot) % PPQ
                        uint32_t w12[PPQ][12];
    #pragma unroll
                        for (int pp = 0; pp < PPQ; ++pp) {
    #pragma unroll
                            for (int e = 0; e < 4; ++e) w12[pp][e] = pack_h2(f[pp][2 * e], f[pp][2 * e + 1]);
    #pragma unroll
                            for (int e = 0; e < 8; ++e) w12[pp][4 + e] = tf32_bits(f[pp][e]);
                        }
                        rotate_rows<PPQ, 12>(w12, rot);
    #pragma unroll
                        for (int pp = 0; pp < PPQ; ++pp) {
                            const int i = i0 + (pp + rot) % PPQ;
                            *reinterpret_cast<uint4 *>(sm + S::XQ16 + kmaj_off(i, c0, 2, 128, 16 * R)) =
                                make_uint4(w12[pp][0], w12[pp][1], w12[pp][2], w12[pp][3]);
                            *reinterpret_cast<uint4 *>(sm + S::XQ32 + kmaj_off(i, c0, 4, 128, 32 * R)) =
                                make_uint4(w12[pp][4], w12[pp][5], w12[pp][6], w12[pp][7]);
                            *reinterpret_cast<uint4 *>(sm + S::XQ32 + kmaj_off(i, c0 + 4, 4, 128, 32 * R)) =
                                make_uint4(w12[pp][8], w12[pp][9], w12[pp][10], w12[pp][11]);
                        }
                    } else {
    #pragma unroll
                        for (int pp = 0; pp < PPQ; ++pp)
    #pragma unroll
                            for (int e = 0; e < 8; ++e) fk[pp][e] = f[pp][e];
                    }
                }
                // key RMSNorm + affine, packed to fp16 once for the Kt rows (rotated) and the
                // transposed key rows of Z^T
    #pragma unroll
                for (int pp = 0; pp < PPQ; ++pp) {
                    float ms = 0.f;
    #pragma unroll
                    for (int e = 0; e < 8; ++e) ms = fmaf(fk[pp][e], fk[pp][e], ms);
    #pragma unroll
                    for (int o = 1; o < CBQ; o <<= 1) ms += __shfl_xor_sync(0xffffffffu, ms, o);
                    const float rk = rsqrtf(ms / R + IDA_EPS_RMS);
                    const bool valid = i0 + pp < L;
    #pragma unroll
                    for (int e = 0; e < 8; ++e) fk[pp][e] = valid ? fmaf(fk[pp][e] * rk, nwk[e], bsk[e]) : 0.f;
    #pragma unroll
                    for (int e = 0; e < 4; ++e) hk[pp][e] = pack_h2(fk[pp][2 * e], fk[pp][2 * e + 1]);
                }
                {
                    uint32_t hr[PPQ][4];
    #pragma unroll
                    for (int pp = 0; pp < PPQ; ++pp)
    #pragma unroll
                        for (int e = 0; e < 4; ++e) hr[pp][e] = hk[pp][e];
                    rotate_rows<PPQ, 4>(hr, rot);
    #pragma unroll
                    for (int pp = 0; pp < PPQ; ++pp) {
                        const int i = i0 + (pp + rot) % PPQ;
                        *reinterpret_cast<uint4 *>(sm + S::KT16 + kmaj_off(i, c0, 2, 128, 16 * R)) =
                            make_uint4(hr[pp][0], hr[pp][1], hr[pp][2], hr[pp][3]);
                    }
                }
            }
            // The previous chunk's state update read U (which P^T reads next) and Z^T, CF16
            // (rewritten below): wait for it before issuing this chunk's MMAs.
            if (it > 0 && !mbar_wait(&bar[4], par ^ 1)) ok = false;
            fence_proxy_async_smem();
            tc_fence_before();
            if (__syncthreads_or(!ok)) break;
            tc_fence_after();

            // ---- S2: G (and P^T on the skewed path; the factorised path issues it in S3) ----------
            if (warp == 0 && elect_one()) {
                const uint32_t idg = idesc(128, 64, 0, 0);
    #pragma unroll
                for (int s = 0; s < R / 16; ++s)
                    mma_f16(tb + T::G, sdesc_at(s16, S::XQ16 + s * 256, 128, 16 * R),
                               sdesc_at(s16, S::KT16 + s * 256, 128, 16 * R), idg, s > 0);
                mma_commit(&bar[0]);
            } else if (!FACT && warp == 1 && elect_one()) {
                // skewed path: P^T from a second issuing thread (an issuing thread stalls while the
                // tensor pipe's queue is full, and one thread issuing both measured slower)
                const uint32_t idp = idesc(128, 64, 2, 2);
    #pragma unroll
                for (int s = 0; s < R / 8; ++s)
                    mma_tf32_t(tb + T::PT, tb + T::U + 8 * s, sdesc_at(s16, S::XQ32 + s * 256, 128, 32 * R), idp, s > 0);
                mma_commit(&bar[6]);
            }
            __syncwarp();

            // ---- S1b, under the G MMA (and P^T on the skewed path): Z^T key rows, the value rows,
            // a ragged Coef
            // (read by the O1 and state-update MMAs, after later proxy fences and barriers)
            {
                const int cb = tid % CBQ, i0 = (tid / CBQ) * PPQ, c0 = 8 * cb;
    #pragma unroll
                for (int e = 0; e < 8; ++e) {
                    // channel c0 + e at positions i0 .. i0 + PPQ - 1: pairs of halves from hk
                    const uint32_t sel = (e & 1) ? 0x7632u : 0x5410u;
                    unsigned char *dst = sm + S::ZT16 + kmaj_off(c0 + e, i0, 2, PADLBO, S::ZT_SBO);
                    const uint32_t w01 = __byte_perm(hk[0][e >> 1], hk[1][e >> 1], sel);
                    if constexpr (PPQ == 4)
                        *reinterpret_cast<uint2 *>(dst) = make_uint2(w01, __byte_perm(hk[2][e >> 1], hk[3][e >> 1], sel));
                    else
                        *reinterpret_cast<uint32_t *>(dst) = w01;
                }
            }
            {
                // value: D/8 channel blocks x (64 D/8 / 256) positions per thread
                constexpr int CBV = D / 8, PPV = CH * CBV / NTH;
                const int cb = tid % CBV, i0 = (tid / CBV) * PPV, j0 = 8 * cb;
                float nwv[8], bsv[8];
                *reinterpret_cast<float4 *>(nwv) = *reinterpret_cast<const float4 *>(nws + R + j0);
                *reinterpret_cast<float4 *>(nwv + 4) = *reinterpret_cast<const float4 *>(nws + R + j0 + 4);
                *reinterpret_cast<float4 *>(bsv) = *reinterpret_cast<const float4 *>(bss + R + j0);
                *reinterpret_cast<float4 *>(bsv + 4) = *reinterpret_cast<const float4 *>(bss + R + j0 + 4);
                float vt[PPV][8];
    #pragma unroll
                for (int pp = 0; pp < PPV; ++pp) {
                    const int i = i0 + pp;
                    float x8[8];
                    unpack_bf16x8(*reinterpret_cast<const uint4 *>(sm + S::RAWV + ((size_t)i * D + j0) * 2), x8);
                    float ms = 0.f;
    #pragma unroll
                    for (int e = 0; e < 8; ++e) ms = fmaf(x8[e], x8[e], ms);
    #pragma unroll
                    for (int o = 1; o < CBV; o <<= 1) ms += __shfl_xor_sync(0xffffffffu, ms, o);
                    const float rv = rsqrtf(ms / D + IDA_EPS_RMS);
                    const bool valid = i < L;
    #pragma unroll
                    for (int e = 0; e < 8; ++e) vt[pp][e] = valid ? fmaf(x8[e] * rv, nwv[e], bsv[e]) : 0.f;
                }
    #pragma unroll
                for (int e = 0; e < 8; ++e) {
                    unsigned char *dst = sm + S::ZT16 + kmaj_off(R + j0 + e, i0, 2, PADLBO, S::ZT_SBO);
                    const uint32_t w01 = pack_h2(vt[0][e], vt[1][e]);
                    if constexpr (PPV == 4)
                        *reinterpret_cast<uint2 *>(dst) = make_uint2(w01, pack_h2(vt[2][e], vt[3][e]));
                    else
                        *reinterpret_cast<uint32_t *>(dst) = w01;
                }
            }
            if (L < CH && hsel == 0) {
                // ragged last chunk: Coef row = component of B lambda^(L-1-j) for j < L, else 0
                float pr = 1.f, pi = 0.f, sr = 0.f, si = 0.f;
                __align__(16) __half cf[CH];
    #pragma unroll
                for (int j = 0; j < CH; ++j) cf[j] = __float2half_rn(0.f);
                for (int k = 0; k < L; ++k) {
                    sr += pr;
                    si += pi;
                    const float cr = b_r * pr - b_i * pi, cim = b_r * pi + b_i * pr;
                    cf[L - 1 - k] = __float2half_rn(is_im ? cim : cr);
                    const float nr = pr * lam_r - pi * lam_i, ni = pr * lam_i + pi * lam_r;
                    pr = nr;
                    pi = ni;
                }
    #pragma unroll
                for (int k8 = 0; k8 < CH / 8; ++k8)
                    *reinterpret_cast<uint4 *>(sm + S::CF16 + kmaj_off(tl, k8 * 8, 2, 128, 1024)) =
                        *reinterpret_cast<const uint4 *>(&cf[k8 * 8]);
                if (!is_im) {
                    laml[mm] = make_float2(pr, pi);  // lambda^L
                    suml[mm] = make_float2(sr, si);  // sum_{k<L} lambda^k
                }
            }
            ok = mbar_wait(&bar[0], par);
            if (tid == 0) bulk_wait_read_all();  // the previous output tile has left GP16 / A216
            tc_fence_after();
            if (__syncthreads_or(!ok)) break;

            // ---- S3: G' = skewed, masked G (skewed path); masked G (factorised path) --------
            if constexpr (FACT) {
                // P^T, first read in S5, issued once G is complete, so that G ran alone on the
                // tensor pipe and P^T runs under the masking, from a warp the masking leaves idle
                // (U is final since the previous state update; XQ32 was fenced before S2)
                if (warp == 2 && elect_one()) {
                    tc_fence_after();
                    const uint32_t idp = idesc(128, 64, 2, 2);
    #pragma unroll
                    for (int s = 0; s < R / 8; ++s)
                        mma_tf32_t(tb + T::PT, tb + T::U + 8 * s, sdesc_at(s16, S::XQ32 + s * 256, 128, 32 * R), idp,
                                   s > 0);
                    mma_commit(&bar[6]);
                }
                __syncwarp();
            }
            // skewed path: scratch [64][64] rotated by row, over YA16: the raw tile there is
            // consumed and YA16 is not rewritten before S5 (XQ32 may still be read by the P^T MMA)
            float *scr = reinterpret_cast<float *>(sm + S::YA16);
            if constexpr (!FACT) {
                if (q4 < 2) {
                    const int i = tl;
        #pragma unroll
                    for (int c0 = 32 * hsel; c0 < 32 * hsel + 32; c0 += 16) {
                        float v[16];
                        tmem_ld16(tb + lane_base + T::G + c0, v);
                        tmem_wait_ld();
        #pragma unroll
                        for (int j = 0; j < 16; ++j) scr[i * 64 + ((c0 + j + i) & 63)] = v[j];
                    }
                }
                __syncthreads();
                {
                    const int i = tid >> 2, p = tid & 3;
        #pragma unroll
                    for (int h8 = 0; h8 < 2; ++h8) {
                        float g8[8];
        #pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            const int k = 16 * p + 8 * h8 + e;
                            g8[e] = k <= i ? scr[i * 64 + ((2 * i - k) & 63)] : 0.f;
                        }
                        *reinterpret_cast<uint4 *>(sm + S::GP16 + kmaj_off(i, 16 * p + 8 * h8, 2, 128, 1024)) = pack_f16x8(g8);
                    }
                }
            } else if (q4 < 2) {
                // row i of G, my half of the columns, masked to j <= i
                const int i = tl;
                float v[32];
                tmem_ld16(tb + lane_base + T::G + 32 * hsel, v);
                tmem_ld16(tb + lane_base + T::G + 32 * hsel + 16, v + 16);
                tmem_wait_ld();
#pragma unroll
                for (int k8 = 0; k8 < 4; ++k8) {
                    float g8[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) g8[e] = 32 * hsel + 8 * k8 + e <= i ? v[8 * k8 + e] : 0.f;
                    *reinterpret_cast<uint4 *>(sm + S::GP16 + kmaj_off(i, 32 * hsel + 8 * k8, 2, 128, 1024)) =
                        pack_f16x8(g8);
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            __syncthreads();
            tc_fence_after();

            // ---- S4: L^T = T_L . G'^T -----------------------------------------------------
            if (warp == 0 && elect_one()) {
                const uint32_t id = idesc(128, 64, 0, 0);
    #pragma unroll
                for (int s = 0; s < CH / 16; ++s)
                    mma_f16(tb + T::LT, sdesc_at(s16, S::TL16 + s * 256, 128, 1024),
                               sdesc_at(s16, S::GP16 + s * 256, 128, 1024), id, s > 0);
                mma_commit(&bar[1]);
            }
            __syncwarp();
            ok = mbar_wait(&bar[1], par) && mbar_wait(&bar[6], par);
            tc_fence_after();
            if (__syncthreads_or(!ok)) break;

            // ---- S5: a, Ya (fp16, column-scaled), a' (tf32) ------------------------------------
            // Lanes 2m, 2m+1 (planes Re / Im of mode m) split the 32 positions of the warp's half:
            // the Re lane takes 32 hsel + p, the Im lane 32 hsel + 16 + p (p < 16), and each computes
            // both planes there, so a mode's two planes are stored as one pair.  Complex values are
            // held as (own, partner) components; with s = +1 on the Im lane and -1 on the Re lane,
            // for z = (zo, zp) and w = (wr, wi): own(z w) = zo wr + zp (s wi), partner(z w) =
            // zp wr - zo (s wi).  The operands hold (Re, -Im) per mode: -s own and +s partner.
            {
                float *ymx = reinterpret_cast<float *>(sm + S::GP16);  // [2][128]; GP16 is consumed
                const float sg = is_im ? 1.f : -1.f;
                const float bs = sg * b_i, ls = sg * lam_i;
                float pv[32], lv[32];
                tmem_ld16(tb + lane_base + T::PT + 32 * hsel, pv);
                tmem_ld16(tb + lane_base + T::PT + 32 * hsel + 16, pv + 16);
                tmem_ld16(tb + lane_base + T::LT + 32 * hsel, lv);
                tmem_ld16(tb + lane_base + T::LT + 32 * hsel + 16, lv + 16);
                float yo[16], yq[16];           // Ya of my plane / of the partner plane, unscaled
                float mo = 0.f, mq = 0.f;
                const int ib = 32 * hsel + 16 * is_im;  // my first position
                tmem_wait_ld();
                if constexpr (!FACT) {
                    float wr = w0r, ws = sg * w0i;  // lambda^(i+1) at my first position, as (Re, s Im)
        #pragma unroll
                    for (int p = 0; p < 16; ++p) {
                        // my plane at my position; the partner needs mine at its position
                        const float pm = is_im ? pv[16 + p] : pv[p], ps = is_im ? pv[p] : pv[16 + p];
                        const float lm = is_im ? lv[16 + p] : lv[p], lsd = is_im ? lv[p] : lv[16 + p];
                        const float po = __shfl_xor_sync(0xffffffffu, ps, 1);
                        const float lo = __shfl_xor_sync(0xffffffffu, lsd, 1);
                        // a = lambda^(i+1) P + B L
                        const float ao = fmaf(pm, wr, fmaf(po, ws, fmaf(lm, b_r, lo * bs)));
                        const float ap = fmaf(po, wr, fmaf(-pm, ws, fmaf(lo, b_r, -lm * bs)));
                        // Ya = a B: -s own(a B) = -s b_r ao - b_i ap ; s partner(a B) = s b_r ap - b_i ao
                        yo[p] = fmaf(ao, -sg * b_r, -b_i * ap);
                        yq[p] = fmaf(ap, sg * b_r, -b_i * ao);
                        mo = fmaxf(mo, fabsf(yo[p]));
                        mq = fmaxf(mq, fabsf(yq[p]));
                        // a' = a lambda^(i+1), both planes, Re plane first
                        const float qo = -sg * fmaf(ao, wr, ap * ws), qq = sg * fmaf(ap, wr, -ao * ws);
                        const uint32_t t_re = tf32_bits(is_im ? qq : qo), t_im = tf32_bits(is_im ? qo : qq);
                        *reinterpret_cast<uint2 *>(sm + S::AP32 + kmaj_off(ib + p, 2 * mm, 4, PADLBO, S::AP_SBO)) =
                            make_uint2(t_re, t_im);
                        const float nr = fmaf(wr, lam_r, -ws * ls), ns = fmaf(wr, ls, ws * lam_r);
                        wr = nr;
                        ws = ns;
                    }
                } else {
                    // factorised: L'' = 2^-fsc B sum_j G[i,j] lambda^-j, u = lambda P + 2^fsc L'',
                    // a = lambda^i u, z = a lambda^i; Ya = 2^fsc z (the table is 2^-fsc B lambda^-j),
                    // a' = a lambda^(i+1) = z lambda
                    const float l2s = sg * l2i;
                    float wr = v0r, ws = sg * v0i;  // lambda^(2i) at my first position, as (Re, s Im)
#pragma unroll
                    for (int p = 0; p < 16; ++p) {
                        const float pm = is_im ? pv[16 + p] : pv[p], ps = is_im ? pv[p] : pv[16 + p];
                        const float lm = is_im ? lv[16 + p] : lv[p], lsd = is_im ? lv[p] : lv[16 + p];
                        const float po = __shfl_xor_sync(0xffffffffu, ps, 1);
                        const float lo = __shfl_xor_sync(0xffffffffu, lsd, 1);
                        const float uo = fmaf(pm, lam_r, fmaf(po, ls, lm * fS));
                        const float up = fmaf(po, lam_r, fmaf(-pm, ls, lo * fS));
                        const float zo = fmaf(uo, wr, up * ws), zp = fmaf(up, wr, -uo * ws);
                        yo[p] = zo * (-sg * fS);
                        yq[p] = zp * (sg * fS);
                        mo = fmaxf(mo, fabsf(yo[p]));
                        mq = fmaxf(mq, fabsf(yq[p]));
                        const float qo = -sg * fmaf(zo, lam_r, zp * ls), qq = sg * fmaf(zp, lam_r, -zo * ls);
                        const uint32_t t_re = tf32_bits(is_im ? qq : qo), t_im = tf32_bits(is_im ? qo : qq);
                        *reinterpret_cast<uint2 *>(sm + S::AP32 + kmaj_off(ib + p, 2 * mm, 4, PADLBO, S::AP_SBO)) =
                            make_uint2(t_re, t_im);
                        const float nr = fmaf(wr, l2r, -ws * l2s), ns = fmaf(wr, l2s, ws * l2r);
                        wr = nr;
                        ws = ns;
                    }
                }
                // column (plane) maxima over the 64 positions: partner lane, then the other half
                mo = fmaxf(mo, __shfl_xor_sync(0xffffffffu, mq, 1));
                ymx[hsel * 128 + tl] = mo;
                __syncthreads();
                const int e = down_exp(fmaxf(ymx[tl], ymx[128 + tl]));
                const int eq = __shfl_xor_sync(0xffffffffu, e, 1);
                const float so = pow2i(-e), sq = pow2i(-eq);
                // the Im lane writes its positions rotated by 4 so that a pair's stores hit other banks
    #pragma unroll
                for (int p = 0; p < 16; ++p) {
                    const int pr = is_im ? ((p + 4) & 15) : p;
                    const float vo = (is_im ? yo[(p + 4) & 15] : yo[p]) * so;
                    const float vq = (is_im ? yq[(p + 4) & 15] : yq[p]) * sq;
                    *reinterpret_cast<uint32_t *>(sm + S::YA16 + kmaj_off(ib + pr, 2 * mm, 2, PADLBO, S::TY_SBO)) =
                        is_im ? pack_h2(vq, vo) : pack_h2(vo, vq);
                }
                if (e != ya_exp) {
                    // T_A column tl = T_L row tl scaled by 2^e (exact in fp16); my half of k
                    const float sup = pow2i(e);
    #pragma unroll
                    for (int k8 = 0; k8 < 4; ++k8) {
                        const int k0 = 32 * hsel + 8 * k8;
                        __align__(16) __half t8[8];
                        *reinterpret_cast<uint4 *>(t8) =
                            *reinterpret_cast<const uint4 *>(sm + S::TL16 + kmaj_off(tl, k0, 2, 128, 1024));
    #pragma unroll
                        for (int u = 0; u < 8; ++u)
                            *reinterpret_cast<__half *>(sm + S::TA16 + kmaj_off(k0 + u, tl, 2, PADLBO, S::TY_SBO)) =
                                __float2half_rn(__half2float(t8[u]) * sup);
                    }
                    ya_exp = e;
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            __syncthreads();
            tc_fence_after();

            // ---- S6: A2' = Ya . T_A^T -----------------------------------------------------
            if (warp == 0 && elect_one()) {
                const uint32_t id = idesc(128, 64, 0, 0);
    #pragma unroll
                for (int s = 0; s < MP / 16; ++s)
                    mma_f16(tb + T::G, sdesc_at(s16, S::YA16 + s * 2 * PADLBO, PADLBO, S::TY_SBO),
                               sdesc_at(s16, S::TA16 + s * 2 * PADLBO, PADLBO, S::TY_SBO), id, s > 0);
                mma_commit(&bar[2]);
            } else if (!FACT && warp == 1 && elect_one()) {
                // skewed path: O2 = Gamma^T . a'^T needs only S5's a' and the state: it runs under S7
                const uint32_t id32 = idesc(128, 64, 2, 2);
    #pragma unroll
                for (int s = 0; s < MP / 8; ++s)
                    mma_tf32_t(tb + T::LT, tb + T::GT + 8 * s, sdesc_at(s16, S::AP32 + s * 2 * PADLBO, PADLBO, S::AP_SBO),
                                id32, s > 0);
                mma_commit(&bar[3]);
            }
            __syncwarp();
            // under the A2' MMA (and O2 on the skewed path): U scaled by lambda^L (its last reader,
            // P^T, is complete; the next one is this chunk's state update)
            {
                // U (lanes = mode planes): the partner lane holds the other component
                const float2 lm = laml[mm];
                constexpr int NB = R / 32;  // 16-column blocks in my half of U
                float v[NB][16];
    #pragma unroll
                for (int bb = 0; bb < NB; ++bb) tmem_ld16(tb + lane_base + T::U + hsel * (R / 2) + 16 * bb, v[bb]);
                tmem_wait_ld();
                // own(lambda^L x) = own(x) Re lambda^L + partner(x) s Im lambda^L, s = +1 on Im planes
                const float lms = is_im ? lm.y : -lm.y;
    #pragma unroll
                for (int bb = 0; bb < NB; ++bb) {
    #pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const float o = __shfl_xor_sync(0xffffffffu, v[bb][j], 1);
                        v[bb][j] = fmaf(v[bb][j], lm.x, o * lms);
                    }
                    tmem_st16(tb + lane_base + T::U + hsel * (R / 2) + 16 * bb, v[bb]);
                }
                tmem_wait_st();
            }
            ok = mbar_wait(&bar[2], par);
            tc_fence_after();
            if (__syncthreads_or(!ok)) break;

            // ---- S7: A2 = unskewed (skewed path), masked A2' (row-scaled fp16) ----------------
            if constexpr (FACT) {
                // O2 = Gamma^T . a'^T, first read in S8, issued once A2' is complete, so that A2'
                // ran alone on the tensor pipe and O2 runs under the masking, from a warp the
                // masking leaves idle (AP32 was fenced before S6; Gamma^T is rescaled only in S8,
                // after O2 completes)
                if (warp == 2 && elect_one()) {
                    tc_fence_after();
                    const uint32_t id32 = idesc(128, 64, 2, 2);
    #pragma unroll
                    for (int s = 0; s < MP / 8; ++s)
                        mma_tf32_t(tb + T::LT, tb + T::GT + 8 * s,
                                   sdesc_at(s16, S::AP32 + s * 2 * PADLBO, PADLBO, S::AP_SBO), id32, s > 0);
                    mma_commit(&bar[3]);
                }
                __syncwarp();
            }
            // skewed path: scratch over XQ32 (P^T, its last reader, is complete)
            if constexpr (!FACT) {
                scr = reinterpret_cast<float *>(sm + S::XQ32);
                if (q4 < 2) {
                    const int i = tl;
        #pragma unroll
                    for (int c0 = 32 * hsel; c0 < 32 * hsel + 32; c0 += 16) {
                        float v[16];
                        tmem_ld16(tb + lane_base + T::G + c0, v);
                        tmem_wait_ld();
        #pragma unroll
                        for (int j = 0; j < 16; ++j) scr[i * 64 + ((c0 + j + i) & 63)] = v[j];
                    }
                }
                __syncthreads();
                {
                    const int i = tid >> 2, p = tid & 3;
                    float v16[16];
                    float amax = 0.f;
        #pragma unroll
                    for (int u = 0; u < 16; ++u) {
                        const int j = 16 * p + u;
                        v16[u] = j <= i ? scr[i * 64 + ((2 * i - j) & 63)] : 0.f;
                        amax = fmaxf(amax, fabsf(v16[u]));
                    }
                    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
                    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
                    const int e = down_exp(amax);
                    const float sdown = pow2i(-e);
                    if (p == 0) osc[i] = pow2i(e);
        #pragma unroll
                    for (int h8 = 0; h8 < 2; ++h8) {
                        float g8[8];
        #pragma unroll
                        for (int u = 0; u < 8; ++u) g8[u] = v16[8 * h8 + u] * sdown;
                        *reinterpret_cast<uint4 *>(sm + S::A216 + kmaj_off(i, 16 * p + 8 * h8, 2, 128, 1024)) = pack_f16x8(g8);
                    }
                }
            } else {
                // row i of A2, my half of the columns, masked to j <= i; the row maximum of both
                // halves via GP16 (consumed)
                float *xch = reinterpret_cast<float *>(sm + S::GP16);
                const int i = tl;
                float v[32];
                if (q4 < 2) {
                    tmem_ld16(tb + lane_base + T::G + 32 * hsel, v);
                    tmem_ld16(tb + lane_base + T::G + 32 * hsel + 16, v + 16);
                    tmem_wait_ld();
                    float amax = 0.f;
#pragma unroll
                    for (int u = 0; u < 32; ++u) {
                        v[u] = 32 * hsel + u <= i ? v[u] : 0.f;
                        amax = fmaxf(amax, fabsf(v[u]));
                    }
                    xch[hsel * 64 + i] = amax;
                }
                __syncthreads();
                if (q4 < 2) {
                    const int e = down_exp(fmaxf(xch[i], xch[64 + i]));
                    const float sdown = pow2i(-e);
                    if (hsel == 0) osc[i] = pow2i(e);
#pragma unroll
                    for (int k8 = 0; k8 < 4; ++k8) {
                        float g8[8];
#pragma unroll
                        for (int u = 0; u < 8; ++u) g8[u] = v[8 * k8 + u] * sdown;
                        *reinterpret_cast<uint4 *>(sm + S::A216 + kmaj_off(i, 32 * hsel + 8 * k8, 2, 128, 1024)) =
                            pack_f16x8(g8);
                    }
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            __syncthreads();
            tc_fence_after();

            // ---- S8: O1 = Vt^T . A2^T (O2 was issued with A2') -----------------------------------
            if (warp == 0 && elect_one()) {
                const uint32_t id16 = idesc(128, 64, 0, 0);
                const int vrow = S::ZT16 + (R / 8) * S::ZT_SBO;  // value rows R .. R+127
    #pragma unroll
                for (int s = 0; s < CH / 16; ++s)
                    mma_f16(tb + T::PT, sdesc_at(s16, vrow + s * 2 * PADLBO, PADLBO, S::ZT_SBO),
                               sdesc_at(s16, S::A216 + s * 256, 128, 1024), id16, s > 0);
                mma_commit(&bar[7]);
            }
            __syncwarp();
            // under the O1 MMA: Gamma^T scaled by lambda^L once O2, its reader, is complete
            ok = mbar_wait(&bar[3], par);
            tc_fence_after();
            if (ok && tid == 0 && ci + 1 < c_end) {
                // A2' (S6) and O2, the last readers of YA16 / AP32, are complete, and the generic
                // writes there were fenced before S6: the next chunk's raw rows land there under
                // the rest of this chunk
                tma_pending = 1;
                tma_par = (uint32_t)((it + 1) & 1);
                const int tn = t0 + CH;
                mbar_arrive_expect_tx(&bar[5], raw_bytes);
                tma_load_4d(sm + S::RAWQ, &tm_q, 0, h, tn - HALO, b, &bar[5]);
                tma_load_4d(sm + S::RAWK, &tm_k, 0, h, tn - HALO, b, &bar[5]);
                tma_load_4d(sm + S::RAWV, &tm_v, 0, h, tn, b, &bar[5]);
            }
            if (ok) {
                // Gamma^T (lanes = value channels, columns = (Re, Im) per mode)
                float v[4][16];
    #pragma unroll
                for (int bb = 0; bb < 4; ++bb) tmem_ld16(tb + lane_base + T::GT + 64 * hsel + 16 * bb, v[bb]);
                tmem_wait_ld();
    #pragma unroll
                for (int bb = 0; bb < 4; ++bb) {
    #pragma unroll
                    for (int j = 0; j < 16; j += 2) {
                        const float2 l2 = laml[(64 * hsel + 16 * bb + j) >> 1];
                        const float xr = v[bb][j], xi = v[bb][j + 1];
                        v[bb][j] = l2.x * xr - l2.y * xi;
                        v[bb][j + 1] = l2.x * xi + l2.y * xr;
                    }
                    tmem_st16(tb + lane_base + T::GT + 64 * hsel + 16 * bb, v[bb]);
                }
                tmem_wait_st();
            }
            ok = ok && mbar_wait(&bar[7], par);
            tc_fence_after();
            if (__syncthreads_or(!ok)) break;

            // ---- S9: outputs; eta (the next chunk's raw rows were issued in S8) --------------------
            if (ci + 1 < c_end) {
                tma_pending = 1;
                tma_par = (uint32_t)((it + 1) & 1);
            }
            {
                // outputs o[i][jv] into the [64][D] bf16 store tile over GP16 / A216 (dead from
                // here to the next chunk's masked Gram; thread 0 waits for the tile's bulk store
                // just before that)
                const int jv = tl;
                __nv_bfloat16 *otile = reinterpret_cast<__nv_bfloat16 *>(sm + S::GP16);
    #pragma unroll
                for (int cc = 0; cc < 2; ++cc) {
                    const int c0 = 32 * hsel + 16 * cc;
                    float o1[16], o2[16], s16[16];
                    tmem_ld16(tb + lane_base + T::PT + c0, o1);
                    tmem_ld16(tb + lane_base + T::LT + c0, o2);
    #pragma unroll
                    for (int j4 = 0; j4 < 4; ++j4)
                        *reinterpret_cast<float4 *>(s16 + 4 * j4) = *reinterpret_cast<const float4 *>(osc + c0 + 4 * j4);
                    tmem_wait_ld();
                    if (jv < D) {
    #pragma unroll
                        for (int j = 0; j < 16; ++j) otile[(c0 + j) * D + jv] = __float2bfloat16_rn(fmaf(o1[j], s16[j], o2[j]));
                    }
                }
                fence_proxy_async_smem();
                if (hsel == 0 && !is_im) {
                    // eta <- lambda^L eta + B sum_{k<L} lambda^k
                    const float2 ll = laml[mm], sl = suml[mm];
                    const float sr = sl.x, si = sl.y;
                    const float er = ll.x * eta_r - ll.y * eta_i + b_r * sr - b_i * si;
                    const float ei = ll.x * eta_i + ll.y * eta_r + b_r * si + b_i * sr;
                    eta_r = er;
                    eta_i = ei;
                }
            }
            tc_fence_before();
            __syncthreads();
            tc_fence_after();

            // ---- S10: U += Coef . Kt ; Gamma^T += Vt^T . Coef^T -----------------------------------
            if (tid == 0) {
                // the chunk's output rows; rows past N are clipped by the copy (thread 0 owns the
                // bulk group it waits on before the next masked Gram)
                tma_store_4d(&tm_o, 0, h, t0, b, sm + S::GP16);
                bulk_commit();
            }
            if (warp == 0 && elect_one()) {
                const uint32_t idu = idesc(128, R, 0, 0);
    #pragma unroll
                for (int s = 0; s < CH / 16; ++s)
                    mma_f16(tb + T::U, sdesc_at(s16, S::CF16 + s * 256, 128, 1024),
                               sdesc_at(s16, S::ZT16 + s * 2 * PADLBO, PADLBO, S::ZT_SBO), idu, 1);
                const uint32_t idg = idesc(128, MP, 0, 0);
                const int vrow = S::ZT16 + (R / 8) * S::ZT_SBO;
    #pragma unroll
                for (int s = 0; s < CH / 16; ++s)
                    mma_f16(tb + T::GT, sdesc_at(s16, vrow + s * 2 * PADLBO, PADLBO, S::ZT_SBO),
                               sdesc_at(s16, S::CF16 + s * 256, 128, 1024), idg, 1);
                mma_commit(&bar[4]);
            }
            __syncwarp();
        }

        // ---- end of the piece: its last state update; the final state ----------------------
        if (tid == 0) bulk_wait_all();  // output stores complete before shared memory is released
        if (ok && c_end > c_begin) {
            ok = mbar_wait(&bar[4], (it - 1) & 1);
            tc_fence_after();
        }
        ok = !__syncthreads_or(!ok);
        if (!ok) {
            // error path: let a copy still in flight land before the CTA exits
            if (tma_pending) mbar_wait(&bar[5], tma_par, 200000000LL);
            if (tid == 0) report_error(a.err, kErrWaitTimeout);
        }
        if (ok && a.final_state && c_end == nchunks) {
            float *fs = a.final_state + (size_t)unit * a.state_floats;
            const int RD = R + D;
            const size_t plane = (size_t)M * RD;
            // U: plane tl -> row (Re: m, Im: M + m), my half of the columns
    #pragma unroll
            for (int c0 = hsel * (R / 2); c0 < (hsel + 1) * (R / 2); c0 += 16) {
                float v[16];
                tmem_ld16(tb + lane_base + T::U + c0, v);
                tmem_wait_ld();
                float *row = fs + (is_im ? plane : 0) + (size_t)mm * RD + c0;
    #pragma unroll
                for (int j = 0; j < 16; ++j) row[j] = v[j];
            }
            // Gamma^T: value lane tl writes column R + tl of every row, my half of the modes
    #pragma unroll
            for (int c0 = 64 * hsel; c0 < 64 * hsel + 64; c0 += 16) {
                float v[16];
                tmem_ld16(tb + lane_base + T::GT + c0, v);
                tmem_wait_ld();
                if (tl < D) {
    #pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const int pl = c0 + j, m = pl >> 1;
                        fs[((pl & 1) ? plane : 0) + (size_t)m * RD + R + tl] = v[j];
                    }
                }
            }
            if (hsel == 0 && !is_im) {
                fs[2 * plane + mm] = eta_r;
                fs[2 * plane + M + mm] = eta_i;
            }
            float *tq = fs + 2 * plane + 2 * M;
            float *tk = tq + (size_t)(W - 1) * R;
            const float *tin = (EXT && a.state_in) ? a.state_in + (size_t)unit * a.state_floats + (tq - fs) : nullptr;
            for (int x = tid; x < (W - 1) * R; x += NTH) {
                const int r = x / R, c = x % R;
                const int p = N - (W - 1) + r;  // before position 0: the initial state's tails
                const size_t tx = (size_t)(p + W - 1) * R + c;
                tq[x] = p >= 0 ? __bfloat162float(gq[base_qk + (size_t)p * sqk + c]) : (tin ? tin[tx] : 0.f);
                tk[x] = p >= 0 ? __bfloat162float(gk[base_qk + (size_t)p * sqk + c])
                               : (tin ? tin[(size_t)(W - 1) * R + tx] : 0.f);
            }
            const size_t used = 2 * plane + 2 * M + 2 * (size_t)(W - 1) * R;
            for (size_t x = used + tid; x < a.state_floats; x += NTH) fs[x] = 0.f;
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tb, 512);
}


// ---- sequence blocks: local end states, then the states before each block ----------------
//
// A unit's sequence is cut into blocks of fs chunks (P = 64 fs positions).  The state
// before block j is
//   X_start(j) = sum_{j' < j} lambda^(P (j - 1 - j')) X_local(j')
// where X_local(j') = sum_{t in j'} B lambda^(P - 1 - t') z_t (t' the position inside the
// block) is the state block j' reaches from zero.  chunk_state_kernel computes X_local of
// every block before the unit's last piece; chunk_prefill_kernel then runs all pieces in
// parallel, each composing its start state from the X_local before it.  States are kept
// as [R + 128 columns][128 lanes] floats, the TMEM image of U and Gamma^T.
//
// X_local is one contraction over the block's positions: per chunk c of the block, the
// state-update MMAs accumulate Coef_c . Kt_c and Vt_c^T . Coef_c^T with
//   Coef_c[j] = lambda^(64 (fs - 1 - c)) B lambda^(63 - j)
// so the accumulator is never rescaled between chunks.  Coefficients of old chunks of
// fast modes underflow in fp16; they are below 2^-24 of the newest ones, beneath the
// accumulator's own precision.

template <int R, int D>
struct StateSmem {
    static constexpr int RAWK = 0;                                    // [67][R] bf16
    static constexpr int RAWV = align1k((CH + HALO) * R * 2);         // [64][D] bf16
    static constexpr int ZT16 = RAWV + align1k(CH * D * 2);           // [R+D][64] f16, as in ChunkSmem
    static constexpr int ZT_SBO = ChunkSmem<R, D>::ZT_SBO;
    static constexpr int CF16 = ZT16 + (R + D) / 8 * ZT_SBO;          // [128][64] f16 (follows ZT16)
    static constexpr int BARS = CF16 + MP * CH * 2;                   // 2 mbarriers: TMA, MMA
    static constexpr int TSLOT = BARS + 16;
    static constexpr int NWS = TSLOT + 16;                            // [R+D] float
    static constexpr int BSS = NWS + (R + D) * 4;                     // [R+D] float
    static constexpr int TOTAL = BSS + (R + D) * 4;
    // two CTAs fit an SM's shared memory and TMEM (256 columns each); the register count
    // (__launch_bounds__(NTH, 1)) keeps the pass at one CTA per SM, which timed faster than two
    // CTAs per SM at 128 registers
    static_assert(RAWV % 1024 == 0 && 2 * TOTAL <= 227 * 1024, "shared memory budget");
};

template <int R, int D, bool EXT>
__global__ void __launch_bounds__(NTH, 1)
    chunk_state_kernel(PrefillArgs a, const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, SegPlan plan, float *seg_state) {
    using S = StateSmem<R, D>;
    extern __shared__ __align__(1024) unsigned char sm[];
    const uint32_t s16 = smem_u32(sm) >> 4;  // shared base for MMA descriptors
    uint64_t *bar = reinterpret_cast<uint64_t *>(sm + S::BARS);  // 0 TMA, 1 MMA
    uint32_t *tslot = reinterpret_cast<uint32_t *>(sm + S::TSLOT);
    float *nws = reinterpret_cast<float *>(sm + S::NWS);
    float *bss = reinterpret_cast<float *>(sm + S::BSS);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int q4 = warp & 3, hsel = warp >> 2, tl = 32 * q4 + lane;
    const uint32_t lane_base = (uint32_t)(32 * q4) << 16;
    const int H = a.H, M = 64, W = a.W;
    // block sgi of unit `unit` (blocks before the unit's last piece are full)
    const int nloc = plan_state_blocks(plan);
    const int unit = blockIdx.x / nloc, sgi = blockIdx.x % nloc, b = unit / H, h = unit % H;
    const int c_begin = sgi * plan.fs, c_end = c_begin + plan.fs;
    const uint32_t raw_bytes = (uint32_t)(CH + HALO) * R * 2 + (uint32_t)CH * D * 2;
    const int mm = tl >> 1, is_im = tl & 1;
    const bool feat_l2 = EXT && (a.flags & IDA_FEAT_L2) != 0;
    const float lam_r = a.lambda[((size_t)h * M + mm) * 2], lam_i = a.lambda[((size_t)h * M + mm) * 2 + 1];
    const float b_r = a.Bvec[((size_t)h * M + mm) * 2], b_i = a.Bvec[((size_t)h * M + mm) * 2 + 1];
    constexpr uint32_t TU = 0, TG = R;  // TMEM columns of U and Gamma^T

    if ((smem_u32(sm) & 1023u) != 0u) {
        if (tid == 0) report_error(a.err, kErrShape);
        return;
    }
    if (tid == 0) {
        mbar_init(&bar[0], 1);
        mbar_init(&bar[1], 1);
        fence_mbar_init();
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
    }
    if (warp == 0) {
        tmem_alloc(tslot, 256);
        tmem_relinquish();
    }
    for (int x = tid; x < R + D; x += NTH) {
        nws[x] = a.norm_w[(size_t)h * (R + D) + x];
        bss[x] = a.bias[(size_t)h * (R + D) + x];
    }
    // Coef row of plane tl, my half of the positions j: B lambda^(63 - j) for j in
    // [32 hsel, 32 hsel + 32), i.e. B lambda^k from k0 = 32 (1 - hsel) down the row;
    // and lambda^64, the decay across one chunk
    float c0r = b_r, c0i = b_i, l64r = lam_r, l64i = lam_i;
    {
        float qr = lam_r, qi = lam_i;
#pragma unroll
        for (int sq = 0; sq < 5; ++sq) {  // lambda^32
            const float nr = qr * qr - qi * qi, ni = 2.f * qr * qi;
            qr = nr;
            qi = ni;
        }
        if (hsel == 0) {
            const float nr = c0r * qr - c0i * qi, ni = c0r * qi + c0i * qr;
            c0r = nr;
            c0i = ni;
        }
        l64r = qr * qr - qi * qi;
        l64i = 2.f * qr * qi;
    }
    // key conv taps of my channel block, right-aligned (as in the readout kernel)
    constexpr int CBQ = R / 8, PPQ = CH * CBQ / NTH;
    const int cb = tid % CBQ, i0 = (tid / CBQ) * PPQ, c0 = 8 * cb;
    // as channel pairs for the packed fp32x2 arithmetic: tp[e2][jj] = (tap jj of channel
    // 2 e2, of channel 2 e2 + 1)
    f2_t tp[4][4];
    {
        const float *cwg = a.conv_w + ((size_t)(1 * H + h) * R + c0) * W;
#pragma unroll
        for (int e2 = 0; e2 < 4; ++e2)
#pragma unroll
            for (int jj = 0; jj < 4; ++jj)
                tp[e2][jj] = jj >= 4 - W ? f2_pack(cwg[(2 * e2) * W + jj - (4 - W)], cwg[(2 * e2 + 1) * W + jj - (4 - W)])
                                         : 0ull;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tb = *tslot;
    if (tid == 0) {
        mbar_arrive_expect_tx(&bar[0], raw_bytes);
        tma_load_4d(sm + S::RAWK, &tm_k, 0, h, c_begin * CH - HALO, b, &bar[0]);
        tma_load_4d(sm + S::RAWV, &tm_v, 0, h, c_begin * CH, b, &bar[0]);
    }
    f2_t nwk[4], bsk[4];  // key RMSNorm weight and bias of my channel pairs
#pragma unroll
    for (int e2 = 0; e2 < 4; ++e2) {
        nwk[e2] = f2_pack(nws[c0 + 2 * e2], nws[c0 + 2 * e2 + 1]);
        bsk[e2] = f2_pack(bss[c0 + 2 * e2], bss[c0 + 2 * e2 + 1]);
    }
    constexpr int CBV = D / 8, PPV = CH * CBV / NTH;
    const int cbv = tid % CBV, iv0 = (tid / CBV) * PPV, j0 = 8 * cbv;
    f2_t nwv[4], bsv[4];  // value RMSNorm weight and bias of my channel pairs
#pragma unroll
    for (int e2 = 0; e2 < 4; ++e2) {
        nwv[e2] = f2_pack(nws[R + j0 + 2 * e2], nws[R + j0 + 2 * e2 + 1]);
        bsv[e2] = f2_pack(bss[R + j0 + 2 * e2], bss[R + j0 + 2 * e2 + 1]);
    }
    bool ok = true;
    int tma_pending = 1;
    int ci = c_begin;
    for (; ci < c_end; ++ci) {
        const int lc = ci - c_begin;
        const uint32_t par = lc & 1;
        ok = mbar_wait(&bar[0], par);
        if (ok) tma_pending = 0;
        if (__syncthreads_or(!ok)) break;
        if (EXT && ci == 0 && a.state_in) {
            // conv halo of the first chunk: the initial state's key tails (the copy zero-filled them)
            const float *tk = a.state_in + (size_t)unit * a.state_floats + (size_t)2 * 64 * (R + D + 1) +
                              (size_t)(W - 1) * R;
            __nv_bfloat16 *rk = reinterpret_cast<__nv_bfloat16 *>(sm + S::RAWK);
            for (int x = tid; x < HALO * R; x += NTH) {
                const int r = x / R, c = x % R, j = r - HALO + (W - 1);
                if (j >= 0) rk[x] = __float2bfloat16_rn(tk[(size_t)j * R + c]);
            }
            __syncthreads();
        }
        // key conv (channel pairs, packed fp32x2) and the raw value rows: the staged tiles
        // are then free for the next chunk
        f2_t g[PPQ][4];
#pragma unroll
        for (int pp = 0; pp < PPQ; ++pp)
#pragma unroll
            for (int e2 = 0; e2 < 4; ++e2) g[pp][e2] = 0ull;
#pragma unroll
        for (int r = 0; r < PPQ + HALO; ++r) {
            const uint4 u = *reinterpret_cast<const uint4 *>(sm + S::RAWK + ((size_t)(i0 + r) * R + c0) * 2);
            const uint32_t wv[4] = {u.x, u.y, u.z, u.w};
            f2_t x2[4];
#pragma unroll
            for (int e2 = 0; e2 < 4; ++e2)
                x2[e2] = f2_pack(__uint_as_float(wv[e2] << 16), __uint_as_float(wv[e2] & 0xFFFF0000u));
#pragma unroll
            for (int pp = 0; pp < PPQ; ++pp) {
                const int jj = r - pp;
                if (jj >= 0 && jj < 4)
#pragma unroll
                    for (int e2 = 0; e2 < 4; ++e2) g[pp][e2] = f2_fma(tp[e2][jj], x2[e2], g[pp][e2]);
            }
        }
        uint4 vraw[PPV];
#pragma unroll
        for (int pp = 0; pp < PPV; ++pp)
            vraw[pp] = *reinterpret_cast<const uint4 *>(sm + S::RAWV + ((size_t)(iv0 + pp) * D + j0) * 2);
        // The TMA below rewrites the tiles just read.  A block barrier orders those generic
        // reads only against other generic accesses: without a proxy fence a shared-memory load
        // still in flight can return the TMA's new row (seen on GB300 as the last key row of a
        // chunk read from the next chunk, in about 3 % of calls at two CTAs per SM).
        fence_proxy_async_smem();
        __syncthreads();
        if (tid == 0 && ci + 1 < c_end) {
            const int tn = (ci + 1) * CH;
            mbar_arrive_expect_tx(&bar[0], raw_bytes);
            tma_load_4d(sm + S::RAWK, &tm_k, 0, h, tn - HALO, b, &bar[0]);
            tma_load_4d(sm + S::RAWV, &tm_v, 0, h, tn, b, &bar[0]);
        }
        if (ci + 1 < c_end) tma_pending = 1;
        // key features, channel pairs in packed fp32x2: SiLU (h + h tanh h, h = x / 2),
        // squared-norm normalisation, RMSNorm + affine
        float fk[PPQ][8];
        {
            const f2_t half2 = f2_pack(0.5f, 0.5f);
#pragma unroll
            for (int pp = 0; pp < PPQ; ++pp) {
                f2_t s2 = 0ull;
#pragma unroll
                for (int e2 = 0; e2 < 4; ++e2) {
                    const f2_t h2 = f2_mul(g[pp][e2], half2);
                    float hl, hh;
                    f2_unpack(h2, hl, hh);
                    g[pp][e2] = f2_fma(h2, f2_pack(tanh_approx(hl), tanh_approx(hh)), h2);
                    s2 = f2_fma(g[pp][e2], g[pp][e2], s2);
                }
                float sl, sh;
                f2_unpack(s2, sl, sh);
                float acc = sl + sh;
#pragma unroll
                for (int o = 1; o < CBQ; o <<= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
                const float inv = __fdividef(1.f, (feat_l2 ? sqrtf(acc) : acc) + IDA_EPS_FEAT);
                const f2_t inv2 = f2_pack(inv, inv);
                f2_t m2 = 0ull;
#pragma unroll
                for (int e2 = 0; e2 < 4; ++e2) {
                    g[pp][e2] = f2_mul(g[pp][e2], inv2);
                    m2 = f2_fma(g[pp][e2], g[pp][e2], m2);
                }
                f2_unpack(m2, sl, sh);
                float ms = sl + sh;
#pragma unroll
                for (int o = 1; o < CBQ; o <<= 1) ms += __shfl_xor_sync(0xffffffffu, ms, o);
                const float rk = rsqrtf(ms / R + IDA_EPS_RMS);
                const f2_t rk2 = f2_pack(rk, rk);
#pragma unroll
                for (int e2 = 0; e2 < 4; ++e2)
                    f2_unpack(f2_fma(f2_mul(g[pp][e2], rk2), nwk[e2], bsk[e2]), fk[pp][2 * e2], fk[pp][2 * e2 + 1]);
            }
        }
        // value RMSNorm + affine, channel pairs in packed fp32x2
        float vt[PPV][8];
#pragma unroll
        for (int pp = 0; pp < PPV; ++pp) {
            const uint32_t wv[4] = {vraw[pp].x, vraw[pp].y, vraw[pp].z, vraw[pp].w};
            f2_t x2[4], m2 = 0ull;
#pragma unroll
            for (int e2 = 0; e2 < 4; ++e2) {
                x2[e2] = f2_pack(__uint_as_float(wv[e2] << 16), __uint_as_float(wv[e2] & 0xFFFF0000u));
                m2 = f2_fma(x2[e2], x2[e2], m2);
            }
            float sl, sh;
            f2_unpack(m2, sl, sh);
            float ms = sl + sh;
#pragma unroll
            for (int o = 1; o < CBV; o <<= 1) ms += __shfl_xor_sync(0xffffffffu, ms, o);
            const float rv = rsqrtf(ms / D + IDA_EPS_RMS);
            const f2_t rv2 = f2_pack(rv, rv);
#pragma unroll
            for (int e2 = 0; e2 < 4; ++e2)
                f2_unpack(f2_fma(f2_mul(x2[e2], rv2), nwv[e2], bsv[e2]), vt[pp][2 * e2], vt[pp][2 * e2 + 1]);
        }
        // Coef_c row: mu = lambda^(64 (fs - 1 - lc)) by squaring, times B lambda^k
        float mr = 1.f, mi = 0.f;
        {
            float pr = l64r, pi = l64i;
            for (unsigned e = (unsigned)(plan.fs - 1 - lc); e; e >>= 1) {
                if (e & 1u) {
                    const float nr = mr * pr - mi * pi, ni = mr * pi + mi * pr;
                    mr = nr;
                    mi = ni;
                }
                const float nr = pr * pr - pi * pi, ni = 2.f * pr * pi;
                pr = nr;
                pi = ni;
            }
        }
        uint32_t cfw[16];  // my plane's Coef entries at j = 32 hsel + 2u, +1
        {
            float wr = mr * c0r - mi * c0i, wi = mr * c0i + mi * c0r;  // at j = 32 hsel + 31
            float cj[32];
#pragma unroll
            for (int k = 0; k < 32; ++k) {
                cj[31 - k] = is_im ? wi : wr;
                const float nr = wr * lam_r - wi * lam_i, ni = wr * lam_i + wi * lam_r;
                wr = nr;
                wi = ni;
            }
#pragma unroll
            for (int u = 0; u < 16; ++u) cfw[u] = pack_h2(cj[2 * u], cj[2 * u + 1]);
        }
        // the previous chunk's MMAs read ZT16 and CF16: wait for them before rewriting
        if (lc > 0 && !mbar_wait(&bar[1], par ^ 1)) ok = false;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            unsigned char *dst = sm + S::ZT16 + kmaj_off(c0 + e, i0, 2, PADLBO, S::ZT_SBO);
            const uint32_t w01 = pack_h2(fk[0][e], fk[1][e]);
            if constexpr (PPQ == 4)
                *reinterpret_cast<uint2 *>(dst) = make_uint2(w01, pack_h2(fk[2][e], fk[3][e]));
            else
                *reinterpret_cast<uint32_t *>(dst) = w01;
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            unsigned char *dst = sm + S::ZT16 + kmaj_off(R + j0 + e, iv0, 2, PADLBO, S::ZT_SBO);
            const uint32_t w01 = pack_h2(vt[0][e], vt[1][e]);
            if constexpr (PPV == 4)
                *reinterpret_cast<uint2 *>(dst) = make_uint2(w01, pack_h2(vt[2][e], vt[3][e]));
            else
                *reinterpret_cast<uint32_t *>(dst) = w01;
        }
#pragma unroll
        for (int k8 = 0; k8 < 4; ++k8)
            *reinterpret_cast<uint4 *>(sm + S::CF16 + kmaj_off(tl, 32 * hsel + 8 * k8, 2, 128, 1024)) =
                make_uint4(cfw[4 * k8], cfw[4 * k8 + 1], cfw[4 * k8 + 2], cfw[4 * k8 + 3]);
        fence_proxy_async_smem();
        tc_fence_before();
        if (__syncthreads_or(!ok)) break;
        tc_fence_after();
        if (warp == 0 && elect_one()) {
            const uint32_t idu = idesc(128, R, 0, 0);
#pragma unroll
            for (int s = 0; s < CH / 16; ++s)
                mma_f16(tb + TU, sdesc_at(s16, S::CF16 + s * 256, 128, 1024),
                        sdesc_at(s16, S::ZT16 + s * 2 * PADLBO, PADLBO, S::ZT_SBO), idu, lc > 0 || s > 0);
            const uint32_t idg = idesc(128, MP, 0, 0);
            const int vrow = S::ZT16 + (R / 8) * S::ZT_SBO;
#pragma unroll
            for (int s = 0; s < CH / 16; ++s)
                mma_f16(tb + TG, sdesc_at(s16, vrow + s * 2 * PADLBO, PADLBO, S::ZT_SBO),
                        sdesc_at(s16, S::CF16 + s * 256, 128, 1024), idg, lc > 0 || s > 0);
            mma_commit(&bar[1]);
        }
        __syncwarp();
    }
    if (ok) {
        ok = mbar_wait(&bar[1], (c_end - 1 - c_begin) & 1);
        tc_fence_after();
    }
    ok = !__syncthreads_or(!ok);
    if (!ok) {
        if (tma_pending) mbar_wait(&bar[0], (uint32_t)((ci - c_begin) & 1), 200000000LL);
        if (tid == 0) report_error(a.err, kErrWaitTimeout);
    } else {
        float *dst = seg_state + ((size_t)unit * nloc + sgi) * (size_t)(R + MP) * 128;
        for (int cc = hsel * 16; cc < R + MP; cc += 32) {
            float v[16];
            tmem_ld16(tb + lane_base + cc, v);
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 16; ++j) dst[(size_t)(cc + j) * 128 + tl] = v[j];
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tb, 256);
}

// ---- host side ---------------------------------------------------------------------------

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn(std::string &why) {
    static std::once_flag once;
    static EncodeTiledFn fn = nullptr;
    static std::string err;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q);
        if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !p)
            err = "cuTensorMapEncodeTiled is not available from the driver";
        else
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    if (!fn) why = err;
    return fn;
}

// [B, N, H, C] bf16 tensor as a 4-D map (C, H, N, B) with a box of `rows`
// positions of one head: box (C, 1, rows, 1).
static bool make_map(EncodeTiledFn fn, CUtensorMap *m, const void *ptr, int B, int N, int H, int C, int rows) {
    cuuint64_t dims[4] = {(cuuint64_t)C, (cuuint64_t)H, (cuuint64_t)N, (cuuint64_t)B};
    cuuint64_t strides[3] = {(cuuint64_t)C * 2, (cuuint64_t)H * C * 2, (cuuint64_t)N * H * C * 2};
    cuuint32_t box[4] = {(cuuint32_t)C, 1, (cuuint32_t)rows, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(ptr), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

template <int R, int D, bool EXT>
static cudaError_t launch_chunk_rd_e(const PrefillArgs &a, cudaStream_t st, const CUtensorMap &mq,
                                     const CUtensorMap &mk, const CUtensorMap &mv, const CUtensorMap &mo,
                                     const SegPlan &plan, float *ws) {
    const unsigned units = (unsigned)(a.B * a.H);
    cudaError_t e;
    if (plan.ppu > 1) {
        using SS = StateSmem<R, D>;
        auto sk = chunk_state_kernel<R, D, EXT>;
        e = cudaFuncSetAttribute(sk, cudaFuncAttributeMaxDynamicSharedMemorySize, SS::TOTAL);
        if (e != cudaSuccess) return e;
        sk<<<units * (unsigned)plan_state_blocks(plan), NTH, SS::TOTAL, st>>>(a, mk, mv, plan, ws);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    using S = ChunkSmem<R, D>;
    const unsigned grid = units * (unsigned)plan.ppu;
    // factorised-Gram heads first, then (usually none) the skewed-Gram ones
    auto kf = chunk_prefill_kernel<R, D, true, EXT>;
    auto ks = chunk_prefill_kernel<R, D, false, EXT>;
    if ((e = cudaFuncSetAttribute(kf, cudaFuncAttributeMaxDynamicSharedMemorySize, S::TOTAL)) != cudaSuccess ||
        (e = cudaFuncSetAttribute(ks, cudaFuncAttributeMaxDynamicSharedMemorySize, S::TOTAL)) != cudaSuccess)
        return e;
    kf<<<grid, NTH, S::TOTAL, st>>>(a, mq, mk, mv, mo, plan, ws);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    // the skewed instantiation as a programmatic dependent of the factorised one (see the kernel)
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(NTH, 1, 1);
    cfg.dynamicSmemBytes = S::TOTAL;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const float *wsc = ws;
    return cudaLaunchKernelEx(&cfg, ks, a, mq, mk, mv, mo, plan, wsc);
}

// The instantiation with the state_in / l_2 code only when the call uses either.
template <int R, int D>
static cudaError_t launch_chunk_rd(const PrefillArgs &a, cudaStream_t st, const CUtensorMap &mq,
                                   const CUtensorMap &mk, const CUtensorMap &mv, const CUtensorMap &mo,
                                   const SegPlan &plan, float *ws) {
    if (a.state_in || (a.flags & IDA_FEAT_L2)) return launch_chunk_rd_e<R, D, true>(a, st, mq, mk, mv, mo, plan, ws);
    return launch_chunk_rd_e<R, D, false>(a, st, mq, mk, mv, mo, plan, ws);
}

static bool chunk_path_takes(const PrefillArgs &a) {
    if (a.dtype != IDA_BF16 || a.M != 64 || (a.flags & IDA_READOUT_ETA) || a.W > 4) return false;
    return (a.R == 64 || a.R == 128) && (a.d == 64 || a.d == 128);
}

// One CTA per unit, whole sequences: the plan without a workspace.
static SegPlan whole_plan(int nchunks) {
    SegPlan p;
    p.fs = nchunks > 0 ? nchunks : 1;
    p.nb = 1;
    p.q0 = 1;
    p.q = 1;
    p.ppu = 1;
    return p;
}

// Blocks of fs chunks, at most ppu equal pieces per unit (fewer if the blocks run out).
static SegPlan block_plan(int nchunks, int fs, int ppu) {
    SegPlan p;
    p.fs = fs;
    p.nb = (nchunks + fs - 1) / fs;
    p.q = (p.nb + ppu - 1) / ppu;
    p.q0 = p.q;
    p.ppu = (p.nb + p.q - 1) / p.q;
    return p;
}

// Two pieces per unit: the first c1 = q0 fs chunks, the second the rest.
static SegPlan two_piece_plan(int nchunks, int fs, int q0) {
    SegPlan p;
    p.fs = fs;
    p.nb = q0 + (nchunks - q0 * fs + fs - 1) / fs;
    p.q0 = q0;
    p.q = p.nb - q0;
    p.ppu = 2;
    return p;
}

static size_t plan_workspace_bytes(const SegPlan &p, long long units, int R) {
    return (size_t)units * (size_t)plan_state_blocks(p) * (size_t)(R + MP) * 128 * sizeof(float);
}

// Modelled time of a plan in microseconds, fitted to GB300 timings of the 125M-, 1.3B- and
// 14K-like workloads under forced plans: the readout's makespan (pieces dealt in grid order
// to the SMs, one CTA each) at kChunkUs per chunk, and, when sequences are split, the block
// state pass (waves of one CTA per SM, each kStateWaveUs plus kStateChunk readout chunks
// per chunk), the start-state loads (kLoadUs per block state a piece composes) and the
// extra launch and set-up (kSplitUs).
constexpr double kStateWaveUs = 4.9, kStateChunk = 0.22, kLoadUs = 0.7, kSplitUs = 13.0;
static double chunk_us(int R) { return R > 64 ? 8.9 : 7.4; }
static double plan_cost(const SegPlan &p, long long units, int nchunks, int num_sms, int R) {
    const double tc = chunk_us(R);
    if (p.ppu == 1) return (double)((units + num_sms - 1) / num_sms) * nchunks * tc;
    // later pieces (the last one may be short) first, then the first pieces
    std::vector<double> free_at((size_t)num_sms, 0.0);
    std::priority_queue<double, std::vector<double>, std::greater<double>> sms(free_at.begin(), free_at.end());
    double makespan = 0.0;
    auto deal = [&](double len) {
        const double t = sms.top() + len;
        sms.pop();
        sms.push(t);
        makespan = std::max(makespan, t);
    };
    for (long long u = 0; u < units; ++u)
        for (int pc = 1; pc < p.ppu; ++pc) {
            const int j0 = p.q0 + (pc - 1) * p.q, j1 = std::min(p.nb, j0 + p.q);
            deal((double)(std::min(nchunks, j1 * p.fs) - j0 * p.fs));
        }
    for (long long u = 0; u < units; ++u) deal((double)std::min(nchunks, p.q0 * p.fs));
    const long long nstate = units * plan_state_blocks(p);
    const long long waves = (nstate + num_sms - 1) / num_sms;
    const double state = (double)waves * (kStateWaveUs + p.fs * kStateChunk * tc);
    const double load = plan_state_blocks(p) * kLoadUs * (R + MP) / 192.0;
    return makespan * tc + state + load + kSplitUs;
}

// The cheapest plan whose workspace fits `budget` bytes, among equal pieces (up to one wave
// of CTAs, any block size) and, with fewer than two SMs per unit, two unequal pieces; ties
// go to the smaller workspace.  Plans are remembered per shape.
static SegPlan choose_plan(const PrefillArgs &a, int num_sms, size_t budget) {
    const int nchunks = (a.N + CH - 1) / CH;
    const long long units = (long long)a.B * a.H;
    SegPlan best = whole_plan(nchunks);
    if (units <= 0 || nchunks < 2 || units >= num_sms) return best;

    struct Key {
        long long units;
        int nchunks, R, num_sms;
        size_t budget;
        bool operator==(const Key &o) const {
            return units == o.units && nchunks == o.nchunks && R == o.R && num_sms == o.num_sms && budget == o.budget;
        }
    };
    static std::mutex mu;
    static std::vector<std::pair<Key, SegPlan>> memo;
    const Key key{units, nchunks, a.R, num_sms, budget};
    {
        std::lock_guard<std::mutex> lock(mu);
        for (const auto &e : memo)
            if (e.first == key) return e.second;
    }

    // a split must model at least 3% faster than whole sequences to be taken
    double best_cost = 0.97 * plan_cost(best, units, nchunks, num_sms, a.R);
    size_t best_ws = 0;
    auto consider = [&](const SegPlan &p) {
        if (p.ppu < 2) return;
        const size_t ws = plan_workspace_bytes(p, units, a.R);
        if (ws > budget) return;
        const double c = plan_cost(p, units, nchunks, num_sms, a.R);
        if (c < best_cost - 1e-9 || (c < best_cost + 1e-9 && ws < best_ws)) {
            best = p;
            best_cost = c;
            best_ws = ws;
        }
    };
    const int max_ppu = (int)(num_sms / units);
    for (int ppu = 2; ppu <= max_ppu && ppu <= nchunks; ++ppu)
        for (int fs = 1; fs <= (nchunks + ppu - 1) / ppu; ++fs) consider(block_plan(nchunks, fs, ppu));
    if (2 * units > num_sms)
        for (int c1 = 1; c1 < nchunks; ++c1)
            for (int fs = 1; fs <= c1; ++fs)
                if (c1 % fs == 0) consider(two_piece_plan(nchunks, fs, c1 / fs));

    std::lock_guard<std::mutex> lock(mu);
    if (memo.size() >= 64) memo.erase(memo.begin());
    memo.emplace_back(key, best);
    return best;
}

// Workspace of the plan chosen within `budget` bytes (0 when no split pays off).
size_t chunk_workspace_bytes(const PrefillArgs &a, int num_sms, size_t budget) {
    if (!chunk_path_takes(a) || a.N <= 0) return 0;
    return plan_workspace_bytes(choose_plan(a, num_sms, budget), (long long)a.B * a.H, a.R);
}

// Whether the tensor-core path takes a prefill of this shape and flags (for callers that
// plan around it; the launch below decides with the same test).
bool chunk_path_shape(int dtype, int M, int R, int d, int W, int flags) {
    PrefillArgs a = {};
    a.dtype = dtype; a.M = M; a.R = R; a.d = d; a.W = W; a.flags = flags;
    return !(flags & IDA_PATH_SEQUENTIAL) && chunk_path_takes(a);
}

// Takes bf16 prefill with M = 64 modes and R, d in {64, 128}, denominator-free
// readout.  The eta readout divides by Re(xi(q)^T U^T eta), which on the
// synthetic workloads comes within 1e-5 of its scale; fp16 / tf32 operand
// rounding then dominates the quotient, so that readout, and every other
// shape, is served by the fp32 sequential kernel.  With a workspace of
// chunk_workspace_bytes() the sequence of each unit is split into segments
// that run on separate SMs; without one, one CTA walks each unit.
ida_status launch_chunk_prefill(const PrefillArgs &a, cudaStream_t st, int num_sms, std::string &why, bool *taken,
                                void *workspace, size_t workspace_bytes) {
    *taken = false;
    if (!chunk_path_takes(a)) return IDA_OK;
    EncodeTiledFn fn = encode_fn(why);
    if (!fn) return IDA_OK;  // no tensor-map support: the sequential kernel serves
    CUtensorMap mq, mk, mv, mo;
    if (!make_map(fn, &mq, a.q, a.B, a.N, a.H, a.R, CH + HALO) ||
        !make_map(fn, &mk, a.k, a.B, a.N, a.H, a.R, CH + HALO) || !make_map(fn, &mv, a.v, a.B, a.N, a.H, a.d, CH) ||
        !make_map(fn, &mo, a.out, a.B, a.N, a.H, a.d, CH)) {
        why = "cuTensorMapEncodeTiled rejected the q/k/v/out layout";
        return IDA_OK;
    }
    const SegPlan plan = choose_plan(a, num_sms, workspace ? workspace_bytes : 0);
    float *ws = plan.ppu > 1 ? static_cast<float *>(workspace) : nullptr;
    *taken = true;
    cudaError_t e;
    if (a.R == 128 && a.d == 128)
        e = launch_chunk_rd<128, 128>(a, st, mq, mk, mv, mo, plan, ws);
    else if (a.R == 64 && a.d == 64)
        e = launch_chunk_rd<64, 64>(a, st, mq, mk, mv, mo, plan, ws);
    else if (a.R == 128 && a.d == 64)
        e = launch_chunk_rd<128, 64>(a, st, mq, mk, mv, mo, plan, ws);
    else
        e = launch_chunk_rd<64, 128>(a, st, mq, mk, mv, mo, plan, ws);
    if (e != cudaSuccess) {
        why = std::string("chunked prefill launch: ") + cudaGetErrorString(e);
        return IDA_ERR_CUDA;
    }
    return IDA_OK;
}

}  // namespace ida
