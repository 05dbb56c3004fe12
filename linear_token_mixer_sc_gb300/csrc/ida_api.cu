// ida_api.cu -- the C ABI: argument checks, device error word, dispatch.
//
// Every entry point validates its arguments on the host before touching
// CUDA, so argument errors cost nothing and never leave work in a stream.
#include <cstdint>
#include <mutex>
#include <string>

#include "ida_common.cuh"

namespace ida {
ida_status launch_seq_prefill(const PrefillArgs &a, cudaStream_t st, int num_sms, std::string &why);
ida_status launch_chunk_prefill(const PrefillArgs &a, cudaStream_t st, int num_sms, std::string &why,
                                bool *taken, void *workspace, size_t workspace_bytes);
size_t chunk_workspace_bytes(const PrefillArgs &a, int num_sms, size_t budget);
ida_status launch_decode(const DecodeArgs &a, cudaStream_t st, std::string &why);
}  // namespace ida

namespace {

thread_local std::string g_last_error;

// Device error word: one host-mapped, pinned word per process, allocated on
// first use so that kernels can report without the host synchronising.
std::once_flag g_err_once;
unsigned *g_err_host = nullptr;
unsigned *g_err_dev = nullptr;
cudaError_t g_err_init = cudaSuccess;

ida_status fail(ida_status s, const std::string &why) {
    g_last_error = why;
    return s;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// The host-mapped error word, set up once per process.
ida_status ensure_error_word(std::string &why) {
    std::call_once(g_err_once, [] {
        void *h = nullptr;
        g_err_init = cudaHostAlloc(&h, sizeof(unsigned), cudaHostAllocMapped);
        if (g_err_init != cudaSuccess) return;
        *static_cast<volatile unsigned *>(h) = 0u;
        void *dptr = nullptr;
        g_err_init = cudaHostGetDevicePointer(&dptr, h, 0);
        if (g_err_init != cudaSuccess) return;
        g_err_host = static_cast<unsigned *>(h);
        g_err_dev = static_cast<unsigned *>(dptr);
    });
    if (g_err_init != cudaSuccess) {
        why = std::string("device error word setup: ") + cudaGetErrorString(g_err_init);
        return IDA_ERR_CUDA;
    }
    return IDA_OK;
}

ida_status device_setup(int *num_sms, std::string &why) {
    ida_status s = ensure_error_word(why);
    if (s != IDA_OK) return s;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) {
        why = std::string("device query: ") + cudaGetErrorString(e);
        return IDA_ERR_CUDA;
    }
    unsigned code = *static_cast<volatile unsigned *>(g_err_host);
    if (code != 0u) {
        *static_cast<volatile unsigned *>(g_err_host) = 0u;
        why = "a previous kernel reported device error code " + std::to_string(code);
        return IDA_ERR_DEVICE;
    }
    return IDA_OK;
}

ida_status check_shape(int d, int R, int M, int W, int dtype, int flags, std::string &why) {
    if (d < 1 || R < 1 || M < 1 || W < 1) {
        why = "d, R, M and W must be >= 1";
        return IDA_ERR_ARG;
    }
    if (dtype != IDA_F32 && dtype != IDA_BF16) {
        why = "dtype must be IDA_F32 or IDA_BF16";
        return IDA_ERR_ARG;
    }
    if (flags & ~(IDA_READOUT_ETA | IDA_FEAT_L2 | IDA_PATH_SEQUENTIAL)) {
        why = "unknown flag bits";
        return IDA_ERR_ARG;
    }
    if (R > 256 || d > 256 || R < 8 || d < 8 || (R % 8) || (d % 8) || M > 128 || W > 4) {
        why = "supported: 8 <= R,d <= 256 (multiples of 8), M <= 128, W <= 4";
        return IDA_ERR_UNSUPPORTED;
    }
    return IDA_OK;
}

}  // namespace

namespace ida {
// Library-internal hooks for entry points defined in other files.
ida_status forward_entry(const void *q, const void *k, const void *v, const float *conv_w, const float *norm_w,
                         const float *bias, const float *lambda, const float *Bvec, const float *state_in, void *out,
                         float *final_state, int B, int H, int N, int d, int R, int M, int dtype, int W, int flags,
                         void *workspace, size_t workspace_bytes, ida_stream_t stream);
ida_status fail_with(ida_status s, const std::string &why) { return fail(s, why); }
// Shape and flag checks of a call; with num_sms, also the device set-up (the error word,
// where a pending device error is reported).
ida_status check_call(int d, int R, int M, int W, int dtype, int flags, int *num_sms, std::string &why) {
    ida_status s = check_shape(d, R, M, W, dtype, flags, why);
    if (s != IDA_OK || !num_sms) return s;
    return device_setup(num_sms, why);
}
// The device address of the error word (set up on first use), without reading it.
ida_status device_error_word(unsigned **err, std::string &why) {
    ida_status s = ensure_error_word(why);
    *err = s == IDA_OK ? g_err_dev : nullptr;
    return s;
}
}  // namespace ida

extern "C" {

size_t ida_state_floats(int d, int R, int M, int W) {
    if (d < 1 || R < 1 || M < 1 || W < 1) return 0;
    size_t n = (size_t)2 * M * (R + d) + (size_t)2 * M + (size_t)2 * (W - 1) * R;
    return (n + 3) & ~(size_t)3;
}

const char *ida_status_str(ida_status s) {
    switch (s) {
        case IDA_OK: return "IDA_OK";
        case IDA_ERR_ARG: return "IDA_ERR_ARG: invalid argument";
        case IDA_ERR_UNSUPPORTED: return "IDA_ERR_UNSUPPORTED: shape outside the supported set";
        case IDA_ERR_CUDA: return "IDA_ERR_CUDA: CUDA runtime or launch error";
        case IDA_ERR_DEVICE: return "IDA_ERR_DEVICE: a kernel reported a device-side error";
    }
    return "unknown ida_status";
}

const char *ida_last_error(void) { return g_last_error.c_str(); }

ida_status ida_device_error(unsigned *code) {
    unsigned c = 0;
    if (g_err_host) {
        c = *static_cast<volatile unsigned *>(g_err_host);
        *static_cast<volatile unsigned *>(g_err_host) = 0u;
    }
    if (code) *code = c;
    return c ? IDA_ERR_DEVICE : IDA_OK;
}

}  // extern "C"

ida_status ida::forward_entry(const void *q, const void *k, const void *v, const float *conv_w,
                              const float *norm_w, const float *bias, const float *lambda, const float *Bvec,
                              const float *state_in, void *out, float *final_state, int B, int H, int N, int d,
                              int R, int M, int dtype, int W, int flags, void *workspace, size_t workspace_bytes,
                              ida_stream_t stream) {
    std::string why;
    if (B < 0 || H < 0 || N < 0) return fail(IDA_ERR_ARG, "B, H and N must be >= 0");
    ida_status s = check_shape(d, R, M, W, dtype, flags, why);
    if (s != IDA_OK) return fail(s, why);
    if ((long long)B * H > (1LL << 24)) return fail(IDA_ERR_UNSUPPORTED, "B*H above 2^24");
    if ((long long)B * N * H * (R > d ? R : d) >= (1LL << 62)) return fail(IDA_ERR_ARG, "size overflow");
    const bool work = (long long)B * H > 0 && N > 0;
    if (work) {
        const void *ptrs[] = {q, k, v, conv_w, norm_w, bias, lambda, Bvec, out};
        for (const void *p : ptrs)
            if (!p) return fail(IDA_ERR_ARG, "null input or output pointer");
        for (const void *p : ptrs)
            if (!aligned16(p)) return fail(IDA_ERR_ARG, "pointers must be 16-byte aligned");
    }
    if (final_state && !aligned16(final_state)) return fail(IDA_ERR_ARG, "final_state must be 16-byte aligned");
    if (state_in && !aligned16(state_in)) return fail(IDA_ERR_ARG, "state_in must be 16-byte aligned");
    if (workspace && !aligned16(workspace)) return fail(IDA_ERR_ARG, "workspace must be 16-byte aligned");
    if (state_in && final_state) {
        // the kernels read state_in after some units' final states are written
        const size_t bytes = (size_t)B * H * ida_state_floats(d, R, M, W) * sizeof(float);
        const char *si = reinterpret_cast<const char *>(state_in), *fo = reinterpret_cast<const char *>(final_state);
        if (si < fo + bytes && fo < si + bytes) return fail(IDA_ERR_ARG, "state_in and final_state must not overlap");
    }
    if ((long long)B * H == 0 || (N == 0 && !final_state)) return IDA_OK;
    int num_sms = 0;
    s = device_setup(&num_sms, why);
    if (s != IDA_OK) return fail(s, why);
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const size_t SF = ida_state_floats(d, R, M, W);
    if (N == 0) {  // zero positions: the final state is the start state
        const size_t bytes = (size_t)B * H * SF * sizeof(float);
        cudaError_t e = state_in ? cudaMemcpyAsync(final_state, state_in, bytes, cudaMemcpyDeviceToDevice, st)
                                 : cudaMemsetAsync(final_state, 0, bytes, st);
        if (e != cudaSuccess) return fail(IDA_ERR_CUDA, cudaGetErrorString(e));
        return IDA_OK;
    }
    ida::PrefillArgs a;
    a.q = q; a.k = k; a.v = v;
    a.conv_w = conv_w; a.norm_w = norm_w; a.bias = bias; a.lambda = lambda; a.Bvec = Bvec;
    a.out = out; a.final_state = final_state; a.state_in = state_in;
    a.B = B; a.H = H; a.N = N; a.d = d; a.R = R; a.M = M; a.W = W; a.dtype = dtype; a.flags = flags;
    a.state_floats = SF;
    a.err = g_err_dev;
    if (!(flags & IDA_PATH_SEQUENTIAL)) {
        bool taken = false;
        s = ida::launch_chunk_prefill(a, st, num_sms, why, &taken, workspace, workspace_bytes);
        if (taken) return s == IDA_OK ? IDA_OK : fail(s, why);
    }
    s = ida::launch_seq_prefill(a, st, num_sms, why);
    return s == IDA_OK ? IDA_OK : fail(s, why);
}

extern "C" {

ida_status ida_forward(const void *q, const void *k, const void *v, const float *conv_w,
                       const float *norm_w, const float *bias, const float *lambda,
                       const float *Bvec, void *out, float *final_state, int B, int H, int N,
                       int d, int R, int M, int dtype, int W, int flags, ida_stream_t stream) {
    return ida::forward_entry(q, k, v, conv_w, norm_w, bias, lambda, Bvec, nullptr, out, final_state, B, H, N, d,
                              R, M, dtype, W, flags, nullptr, 0, stream);
}

ida_status ida_forward_ws(const void *q, const void *k, const void *v, const float *conv_w,
                          const float *norm_w, const float *bias, const float *lambda,
                          const float *Bvec, void *out, float *final_state, int B, int H, int N,
                          int d, int R, int M, int dtype, int W, int flags, void *workspace,
                          size_t workspace_bytes, ida_stream_t stream) {
    return ida::forward_entry(q, k, v, conv_w, norm_w, bias, lambda, Bvec, nullptr, out, final_state, B, H, N, d,
                              R, M, dtype, W, flags, workspace, workspace_bytes, stream);
}

ida_status ida_forward_from(const void *q, const void *k, const void *v, const float *conv_w,
                            const float *norm_w, const float *bias, const float *lambda, const float *Bvec,
                            const float *state_in, void *out, float *final_state, int B, int H, int N, int d,
                            int R, int M, int dtype, int W, int flags, void *workspace, size_t workspace_bytes,
                            ida_stream_t stream) {
    return ida::forward_entry(q, k, v, conv_w, norm_w, bias, lambda, Bvec, state_in, out, final_state, B, H, N, d,
                              R, M, dtype, W, flags, workspace, workspace_bytes, stream);
}

}  // extern "C"

namespace ida {
// Workspace bytes of the prefill plan chosen within `budget` bytes on the current device.
size_t forward_workspace_within(int B, int H, int N, int d, int R, int M, int dtype, int W, int flags,
                                size_t budget) {
    std::string why;
    if (B < 0 || H < 0 || N < 0 || check_shape(d, R, M, W, dtype, flags, why) != IDA_OK) return 0;
    if (flags & IDA_PATH_SEQUENTIAL) return 0;
    int dev = 0, num_sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return 0;
    PrefillArgs a = {};
    a.B = B; a.H = H; a.N = N; a.d = d; a.R = R; a.M = M; a.W = W; a.dtype = dtype; a.flags = flags;
    return chunk_workspace_bytes(a, num_sms, budget);
}
}  // namespace ida

extern "C" {

size_t ida_forward_workspace_bytes(int B, int H, int N, int d, int R, int M, int dtype, int W, int flags) {
    return ida::forward_workspace_within(B, H, N, d, R, M, dtype, W, flags, ida::kPreferredWorkspace);
}

ida_status ida_decode_step(const void *q, const void *k, const void *v, const float *conv_w,
                           const float *norm_w, const float *bias, const float *lambda,
                           const float *Bvec, float *state_inout, void *out, int B, int H, int d,
                           int R, int M, int dtype, int W, int flags, ida_stream_t stream) {
    std::string why;
    if (B < 0 || H < 0) return fail(IDA_ERR_ARG, "B and H must be >= 0");
    ida_status s = check_shape(d, R, M, W, dtype, flags & ~IDA_PATH_SEQUENTIAL, why);
    if (s != IDA_OK) return fail(s, why);
    if ((long long)B * H > (1LL << 31) - 1) return fail(IDA_ERR_UNSUPPORTED, "B*H above 2^31-1");
    if ((long long)B * H == 0) return IDA_OK;
    const void *ptrs[] = {q, k, v, conv_w, norm_w, bias, lambda, Bvec, state_inout, out};
    for (const void *p : ptrs)
        if (!p) return fail(IDA_ERR_ARG, "null input, state or output pointer");
    for (const void *p : ptrs)
        if (!aligned16(p)) return fail(IDA_ERR_ARG, "pointers must be 16-byte aligned");
    int num_sms = 0;
    s = device_setup(&num_sms, why);
    if (s != IDA_OK) return fail(s, why);
    ida::DecodeArgs a;
    a.q = q; a.k = k; a.v = v;
    a.conv_w = conv_w; a.norm_w = norm_w; a.bias = bias; a.lambda = lambda; a.Bvec = Bvec;
    a.state = state_inout; a.out = out;
    a.B = B; a.H = H; a.d = d; a.R = R; a.M = M; a.W = W; a.dtype = dtype; a.flags = flags;
    a.state_floats = ida_state_floats(d, R, M, W);
    a.err = g_err_dev;
    s = ida::launch_decode(a, reinterpret_cast<cudaStream_t>(stream), why);
    return s == IDA_OK ? IDA_OK : fail(s, why);
}

}  // extern "C"
