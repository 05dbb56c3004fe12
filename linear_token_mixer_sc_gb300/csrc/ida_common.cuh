// ida_common.cuh -- device helpers shared by the mixer's CUDA kernels.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/ida.h"

namespace ida {

// Plain argument bundle handed to every prefill kernel.
struct PrefillArgs {
    const void *q, *k, *v;
    const float *conv_w, *norm_w, *bias, *lambda, *Bvec;
    void *out;
    float *final_state;
    const float *state_in;  // NULL: the zero state; else [B,H] x state_floats, the state before position 0
    int B, H, N, d, R, M, W, dtype, flags;
    size_t state_floats;
    unsigned *err;  // device-visible error word (host-mapped)
};

struct DecodeArgs {
    const void *q, *k, *v;
    const float *conv_w, *norm_w, *bias, *lambda, *Bvec;
    float *state;
    void *out;
    int B, H, d, R, M, W, dtype, flags;
    size_t state_floats;
    unsigned *err;
};

// Largest workspace the prefill asks for (ida_forward_workspace_bytes): sequences are split
// only as finely as the state slots of that many bytes allow.
constexpr size_t kPreferredWorkspace = size_t(64) << 20;

// Error codes written to the device error word (first writer wins).
enum : unsigned {
    kErrNone = 0,
    kErrWaitTimeout = 1,
    kErrTmemAlloc = 2,
    kErrShape = 3,
};

__device__ __forceinline__ void report_error(unsigned *err, unsigned code) {
    if (err) atomicCAS(err, 0u, code);
}

__device__ __forceinline__ float load_in(const void *base, int dtype, size_t i) {
    if (dtype == IDA_BF16)
        return __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(base)[i]);
    return reinterpret_cast<const float *>(base)[i];
}

__device__ __forceinline__ void store_out(void *base, int dtype, size_t i, float x) {
    if (dtype == IDA_BF16)
        reinterpret_cast<__nv_bfloat16 *>(base)[i] = __float2bfloat16_rn(x);
    else
        reinterpret_cast<float *>(base)[i] = x;
}

__device__ __forceinline__ float silu(float x) { return x / (1.0f + expf(-x)); }
__device__ __forceinline__ double silu(double x) { return x / (1.0 + exp(-x)); }

__device__ __forceinline__ float rsqrt_t(float x) { return rsqrtf(x); }
__device__ __forceinline__ double rsqrt_t(double x) { return 1.0 / sqrt(x); }

template <typename T>
__device__ __forceinline__ T warp_sum(T x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

// Sum of each of NV values over the 32 lanes of a warp by recursive halving: afterwards lane
// l holds the full sum of value index rs_index<NV>(l), and the 32 / NV lanes that differ
// from l only in their low bits hold the same one.  NV is a power of two <= 32; about
// NV shuffles instead of 5 NV.
template <int NV, typename T>
__device__ __forceinline__ T warp_reduce_scatter(T (&v)[NV], int lane) {
    int n = NV;
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
        if (n > 1) {
            const bool hi = (lane & off) != 0;
            const int hn = n >> 1;
#pragma unroll
            for (int k = 0; k < NV / 2; ++k) {
                if (k < hn) {
                    const T send = hi ? v[k] : v[k + hn];
                    const T keep = hi ? v[k + hn] : v[k];
                    v[k] = keep + __shfl_xor_sync(0xffffffffu, send, off);
                }
            }
            n = hn;
        } else {
            v[0] += __shfl_xor_sync(0xffffffffu, v[0], off);
        }
    }
    return v[0];
}
// the value index lane l holds after warp_reduce_scatter<NV>
template <int NV>
__device__ __forceinline__ int rs_index(int lane) {
    int idx = 0, n = NV;
#pragma unroll
    for (int off = 16; off >= 1 && n > 1; off >>= 1) {
        n >>= 1;
        if (lane & off) idx += n;
    }
    return idx;
}

// x <- lam * x + g * z for complex x, lam, g and real z, in arithmetic type T.
template <typename T>
__device__ __forceinline__ void cstep_t(T &xr, T &xi, T lr, T li, T gr, T gi, T z) {
    T nr = fma(lr, xr, fma(-li, xi, gr * z));
    T ni = fma(lr, xi, fma(li, xr, gi * z));
    xr = nr;
    xi = ni;
}

struct cplx {
    float re, im;
};

__device__ __forceinline__ cplx cmul(cplx a, cplx b) {
    return {a.re * b.re - a.im * b.im, a.re * b.im + a.im * b.re};
}

// x <- lam * x + g * z   (z real)
__device__ __forceinline__ void cstep(float &xr, float &xi, cplx lam, cplx g, float z) {
    float nr = fmaf(lam.re, xr, fmaf(-lam.im, xi, g.re * z));
    float ni = fmaf(lam.re, xi, fmaf(lam.im, xr, g.im * z));
    xr = nr;
    xi = ni;
}

}  // namespace ida
