// ida_rope.cu -- rotary position embeddings on the mixer's q and k, in place.
//
// The pages embed the token mixer in a Llama-style decoder with rotary position
// embeddings ("Interdomain Attention: Beyond Token-Level Key-Value Memory", German
// technical summary, "Skalierbare Implementierung", "Architektur"); as in that decoder
// the rotation is applied to the query and key rows before the mixer.  Channel pairs
// (2i, 2i + 1) of a row at position p rotate by p * base^(-2i / R).
//
// Per (batch row, tile of ROPE_TILE positions), in a persistent grid: the tile's cos / sin table
// [ROPE_TILE][R / 2] is built in shared memory first, its angles reduced modulo 2 pi exactly
// in integer arithmetic (positions reach 1e4 radians and more, where an fp32 angle would
// already be off by 1e-3), then every head of the tile's q rows, and of its k rows with
// the same table, is rotated with 16-byte loads and stores, a thread's loads of all the
// tile's positions issued together.
// HBM-bound: each element is read and written once.
#include <cstdint>
#include <string>

#include "ida_common.cuh"

namespace ida {

constexpr int ROPE_TILE = 4;  // positions per tile: 4 and 8 time the same after an L2 flush and read-back;
                              // with dirty lines left in L2, 4 was the fastest of 1, 2, 4, 8, 16
constexpr int ROPE_THREADS = 256;

template <typename E>
struct RopeVec;  // 16 bytes of elements
template <>
struct RopeVec<float> {
    static constexpr int n = 4;
};
template <>
struct RopeVec<__nv_bfloat16> {
    static constexpr int n = 8;
};

__device__ __forceinline__ void rope_unpack(const uint4 &u, float *x, float) {
    x[0] = __uint_as_float(u.x);
    x[1] = __uint_as_float(u.y);
    x[2] = __uint_as_float(u.z);
    x[3] = __uint_as_float(u.w);
}
__device__ __forceinline__ uint4 rope_pack(const float *x, float) {
    return make_uint4(__float_as_uint(x[0]), __float_as_uint(x[1]), __float_as_uint(x[2]), __float_as_uint(x[3]));
}
__device__ __forceinline__ void rope_unpack(const uint4 &u, float *x, __nv_bfloat16) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        x[2 * e] = __uint_as_float(w[e] << 16);
        x[2 * e + 1] = __uint_as_float(w[e] & 0xFFFF0000u);
    }
}
__device__ __forceinline__ uint4 rope_pack(const float *x, __nv_bfloat16) {
    uint32_t w[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const __nv_bfloat162 h = __floats2bfloat162_rn(x[2 * e], x[2 * e + 1]);
        w[e] = *reinterpret_cast<const uint32_t *>(&h);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

// The cos / sin table of the tile starting at t0 (len positions), as float2 slots laid out
// [position][pair u of a vector][vector cv], pair i = cv (V / 2) + u: for each u the lanes,
// which own consecutive vectors, read consecutive 8-byte words.
template <int V>
__device__ __forceinline__ void rope_table(float2 *tab, const unsigned long long *turn, int pos0, int t0, int len,
                                           int half) {
    constexpr int P2 = V / 2;  // channel pairs per vector
    const int vpr = half / P2;
    for (int e = threadIdx.x; e < len * half; e += ROPE_THREADS) {
        const int tt = e / half, i = e % half;
        const unsigned long long pos = (unsigned long long)pos0 + (unsigned long long)(t0 + tt);
        const unsigned long long ph = pos * turn[i];  // mod 2^64: the fraction of a turn
        const float x = (float)(int)(unsigned)(ph >> 32) * 4.656612873077392578125e-10f;  // * 2^-31
        float sn, cn;
        sincospif(x, &sn, &cn);
        tab[(tt * P2 + i % P2) * vpr + i / P2] = make_float2(cn, sn);
    }
}

// Persistent: a grid of one wave of CTAs, CTA i taking tiles i, i + gridDim.x, ... of the
// B x ceil(N / ROPE_TILE) tiles (no partly filled last wave).  Two tables: the next tile's
// is built while the current tile is rotated, one block barrier per tile.
template <typename E>
__global__ void __launch_bounds__(ROPE_THREADS) rope_kernel(void *q, void *k, int B, int N, int H, int R, int pos0,
                                                            double log2_base) {
    __shared__ unsigned long long turn[128];      // base^(-2i / R) / (2 pi), as a 0.64 fixed-point fraction
    extern __shared__ __align__(16) float2 cs[];  // [2][ROPE_TILE][R / 2]: the two tables (cos, sin)
    constexpr int V = RopeVec<E>::n, P2 = V / 2;
    const int tiles = (N + ROPE_TILE - 1) / ROPE_TILE, half = R / 2;
    const long long ntiles = (long long)B * tiles;
    // thread -> one 16-byte vector cv of channels (c0 = cv V .. c0 + V) in heads h0, h0 + S,
    // ...: its cos / sin entries are read once per position and serve every head it rotates
    const int vpr = R / V, S = ROPE_THREADS / vpr;
    const int cv = threadIdx.x % vpr, c0 = cv * V, h0 = threadIdx.x / vpr;
    // The angle of position p and frequency i is p * base^(-2i/R) radians, i.e. p * turn_i
    // turns.  turn_i is formed once per CTA in fp64 (fp64 is scarce on this part) and kept
    // as a 64-bit binary fraction; p * turn_i mod 1 is then an exact integer product mod
    // 2^64, whose top 32 bits, read as a signed fraction of half a turn, go to sincospif.
    for (int i = threadIdx.x; i < half; i += ROPE_THREADS) {
        const double tr = exp2(-2.0 * i / R * log2_base) * 0.15915494309189533576888376337251;  // / (2 pi)
        turn[i] = __double2ull_rn(ldexp(tr, 64));  // tr < 1 / (2 pi): no overflow
    }
    __syncthreads();
    const size_t rowstride = (size_t)H * R;  // elements between positions
    const bool worker = h0 < S;                // R / V does not divide the block: spare threads
    const int tsize = ROPE_TILE * half;        // float2 slots per table
    long long tile = blockIdx.x;
    if (tile < ntiles) {
        const int t0 = (int)(tile % tiles) * ROPE_TILE;
        rope_table<V>(cs, turn, pos0, t0, min(ROPE_TILE, N - t0), half);
    }
    __syncthreads();
    for (int cur = 0; tile < ntiles; tile += gridDim.x, cur ^= 1) {
        const int b = (int)(tile / tiles), t0 = (int)(tile % tiles) * ROPE_TILE;
        const int len = min(ROPE_TILE, N - t0);
        // the next tile's table, into the buffer last read before the previous barrier
        const long long nxt = tile + gridDim.x;
        if (nxt < ntiles) {
            const int t1 = (int)(nxt % tiles) * ROPE_TILE;
            rope_table<V>(cs + (cur ^ 1) * tsize, turn, pos0, t1, min(ROPE_TILE, N - t1), half);
        }
        const float2 *tab = cs + cur * tsize;
        for (int which = 0; which < 2 && worker; ++which) {
            E *x = static_cast<E *>(which == 0 ? q : k);
            if (!x) break;
            x += ((size_t)b * N + t0) * rowstride + c0;
            for (int h = h0; h < H; h += S) {
                uint4 w[ROPE_TILE];
#pragma unroll
                for (int tt = 0; tt < ROPE_TILE; ++tt)
                    if (tt < len) w[tt] = __ldcs(reinterpret_cast<const uint4 *>(x + tt * rowstride + (size_t)h * R));
#pragma unroll
                for (int tt = 0; tt < ROPE_TILE; ++tt) {
                    if (tt < len) {
                        float v[V];
                        rope_unpack(w[tt], v, E());
#pragma unroll
                        for (int u = 0; u < P2; ++u) {
                            const float2 cn_sn = tab[(tt * P2 + u) * vpr + cv];
                            const float x0 = v[2 * u], x1 = v[2 * u + 1];
                            v[2 * u] = fmaf(x0, cn_sn.x, -x1 * cn_sn.y);
                            v[2 * u + 1] = fmaf(x0, cn_sn.y, x1 * cn_sn.x);
                        }
                        __stcs(reinterpret_cast<uint4 *>(x + tt * rowstride + (size_t)h * R), rope_pack(v, E()));
                    }
                }
            }
        }
        __syncthreads();  // the next table is complete; this one is free after the next build
    }
}

ida_status fail_with(ida_status s, const std::string &why);
ida_status check_call(int d, int R, int M, int W, int dtype, int flags, int *num_sms, std::string &why);

}  // namespace ida

extern "C" ida_status ida_rope(void *q, void *k, int B, int N, int H, int R, int pos0, float base, int dtype,
                               ida_stream_t stream) {
    std::string why;
    if (B < 0 || N < 0 || H < 0) return ida::fail_with(IDA_ERR_ARG, "B, N and H must be >= 0");
    if (pos0 < 0) return ida::fail_with(IDA_ERR_ARG, "pos0 must be >= 0");
    if (!(base > 1.0f) || !(base < 3.0e38f)) return ida::fail_with(IDA_ERR_ARG, "base must be finite and > 1");
    if (dtype != IDA_F32 && dtype != IDA_BF16) return ida::fail_with(IDA_ERR_ARG, "dtype must be IDA_F32 or IDA_BF16");
    if (R < 8 || R > 256 || (R % 8)) return ida::fail_with(IDA_ERR_UNSUPPORTED, "supported: 8 <= R <= 256, R % 8 == 0");
    if ((long long)H * R > (1LL << 24)) return ida::fail_with(IDA_ERR_UNSUPPORTED, "H*R above 2^24");
    if ((long long)B * N * H == 0) return IDA_OK;
    if (!q) return ida::fail_with(IDA_ERR_ARG, "null pointer");
    if ((reinterpret_cast<uintptr_t>(q) & 15u) != 0 || (reinterpret_cast<uintptr_t>(k) & 15u) != 0)
        return ida::fail_with(IDA_ERR_ARG, "q and k must be 16-byte aligned");
    if (k == q) return ida::fail_with(IDA_ERR_ARG, "k must not alias q");
    const long long tiles = (N + ida::ROPE_TILE - 1) / ida::ROPE_TILE;
    if ((long long)B * tiles > 0x7FFFFFFFLL) return ida::fail_with(IDA_ERR_UNSUPPORTED, "too many positions");
    int num_sms = 0;
    ida_status s = ida::check_call(8, R, 1, 1, dtype, 0, &num_sms, why);  // device set-up, pending errors
    if (s != IDA_OK) return ida::fail_with(s, why);
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const size_t smem = 2 * (size_t)ida::ROPE_TILE * (R / 2) * sizeof(float2);
    const double lb = log2((double)base);  // base^(-2i/R) = exp2(-2i/R * lb)
    int per_sm = 0;
    cudaError_t oe = dtype == IDA_F32
                         ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, ida::rope_kernel<float>,
                                                                          ida::ROPE_THREADS, smem)
                         : cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, ida::rope_kernel<__nv_bfloat16>,
                                                                          ida::ROPE_THREADS, smem);
    if (oe != cudaSuccess || per_sm < 1) per_sm = 1;
    const long long wave = (long long)per_sm * num_sms, ntiles = (long long)B * tiles;
    const unsigned grid = (unsigned)(ntiles < wave ? ntiles : wave);
    if (dtype == IDA_F32)
        ida::rope_kernel<float><<<grid, ida::ROPE_THREADS, smem, st>>>(q, k, B, N, H, R, pos0, lb);
    else
        ida::rope_kernel<__nv_bfloat16><<<grid, ida::ROPE_THREADS, smem, st>>>(q, k, B, N, H, R, pos0, lb);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return ida::fail_with(IDA_ERR_CUDA, std::string("rope launch: ") + cudaGetErrorString(e));
    return IDA_OK;
}
