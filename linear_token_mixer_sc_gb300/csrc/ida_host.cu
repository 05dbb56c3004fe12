// ida_host.cu -- prefill from host memory (ida_forward_host).
//
// The positions are cut into slices; the copy of a slice's q, k, v to the device, the
// prefill of the slice before it (resumed from the state the one before that left, as
// ida_forward_from does) and the copy of the outputs before that to the host run on three
// streams at once, so that the host link and the kernels work at the same time.  Device
// staging holds two slices of q, k, v and out (one slice being filled while the other is
// computed on or drained), two states (the carried state alternates between them) and the
// prefill's workspace.  Everything runs on the GPU; the host only enqueues.
#include <climits>
#include <cstdint>
#include <map>
#include <mutex>
#include <string>

#include "ida_common.cuh"

namespace ida {
ida_status forward_entry(const void *q, const void *k, const void *v, const float *conv_w, const float *norm_w,
                         const float *bias, const float *lambda, const float *Bvec, const float *state_in, void *out,
                         float *final_state, int B, int H, int N, int d, int R, int M, int dtype, int W, int flags,
                         void *workspace, size_t workspace_bytes, ida_stream_t stream);
ida_status fail_with(ida_status s, const std::string &why);
ida_status check_call(int d, int R, int M, int W, int dtype, int flags, int *num_sms, std::string &why);
size_t forward_workspace_within(int B, int H, int N, int d, int R, int M, int dtype, int W, int flags,
                                size_t budget);
bool chunk_path_shape(int dtype, int M, int R, int d, int W, int flags);
}  // namespace ida

namespace {

constexpr int kMinSlice = 512;  // positions per slice, at least (8 chunks of 64)
constexpr int kSlices = 8;      // slices aimed for on the tensor-core path

size_t up256(size_t x) { return (x + 255) & ~size_t(255); }

// Byte layout of the staging buffer for one shape.
struct HostPlan {
    int S = 1, L = 0;                 // slices, positions per slice (the last may be shorter)
    size_t off_q[2], off_k[2], off_v[2], off_o[2], off_st[2], off_ws;
    size_t ws = 0, total = 0;
};

HostPlan host_plan(int B, int H, int N, int d, int R, int M, int dtype, int W, int flags) {
    HostPlan p;
    const size_t es = dtype == IDA_BF16 ? 2 : 4;
    p.L = N;
    if (ida::chunk_path_shape(dtype, M, R, d, W, flags) && N >= 2 * kMinSlice) {
        int l = (N + kSlices - 1) / kSlices;
        l = (l + 63) / 64 * 64;
        p.L = l < kMinSlice ? kMinSlice : l;
        p.S = (N + p.L - 1) / p.L;
    }
    const size_t qk = up256((size_t)B * p.L * H * R * es), vo = up256((size_t)B * p.L * H * d * es);
    const size_t st = up256((size_t)B * H * ida_state_floats(d, R, M, W) * sizeof(float));
    size_t off = 0;
    for (int i = 0; i < 2; ++i) {
        if (i == 1 && p.S == 1) {  // one slice: one set of buffers
            p.off_q[1] = p.off_q[0]; p.off_k[1] = p.off_k[0]; p.off_v[1] = p.off_v[0]; p.off_o[1] = p.off_o[0];
            break;
        }
        p.off_q[i] = off; off += qk;
        p.off_k[i] = off; off += qk;
        p.off_v[i] = off; off += vo;
        p.off_o[i] = off; off += vo;
    }
    for (int i = 0; i < 2; ++i) {
        p.off_st[i] = off;
        off += st;
    }
    p.ws = up256(ida::forward_workspace_within(B, H, p.L, d, R, M, dtype, W, flags, ida::kPreferredWorkspace));
    p.off_ws = off;
    p.total = off + p.ws;
    return p;
}

// The library's copy-in, compute and copy-out streams of one device, created on first use
// and kept for the process, with the events that order them.
struct Pipe {
    cudaStream_t in = nullptr, cmp = nullptr, out = nullptr;
    cudaEvent_t ev_in[2] = {}, ev_cmp[2] = {}, ev_out[2] = {}, ev_a = nullptr, ev_b = nullptr;
    std::mutex mu;  // one call's enqueueing at a time
};

std::mutex g_pipes_mu;
std::map<int, Pipe *> g_pipes;

Pipe *get_pipe(int dev, std::string &why) {
    std::lock_guard<std::mutex> lock(g_pipes_mu);
    auto it = g_pipes.find(dev);
    if (it != g_pipes.end()) return it->second;
    Pipe *p = new Pipe;
    cudaError_t e = cudaSuccess;
    for (cudaStream_t *s : {&p->in, &p->cmp, &p->out})
        if (e == cudaSuccess) e = cudaStreamCreateWithFlags(s, cudaStreamNonBlocking);
    for (int i = 0; i < 2 && e == cudaSuccess; ++i)
        for (cudaEvent_t *ev : {&p->ev_in[i], &p->ev_cmp[i], &p->ev_out[i]})
            if (e == cudaSuccess) e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&p->ev_a, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&p->ev_b, cudaEventDisableTiming);
    if (e != cudaSuccess) {
        why = std::string("stream / event creation: ") + cudaGetErrorString(e);
        return nullptr;  // what was created is kept: the call fails, a later one retries
    }
    g_pipes[dev] = p;
    return p;
}

// `rows` rows of `width` bytes between buffers whose rows start `dpitch` / `spitch` apart.
cudaError_t copy_rows(void *dst, size_t dpitch, const void *src, size_t spitch, size_t width, size_t rows,
                      cudaMemcpyKind kind, cudaStream_t s) {
    if (rows == 0 || width == 0) return cudaSuccess;
    if (rows == 1 || (dpitch == width && spitch == width))
        return cudaMemcpyAsync(dst, src, width * rows, kind, s);
    if (dpitch <= (size_t)INT_MAX && spitch <= (size_t)INT_MAX)
        return cudaMemcpy2DAsync(dst, dpitch, src, spitch, width, rows, kind, s);
    for (size_t r = 0; r < rows; ++r) {
        cudaError_t e = cudaMemcpyAsync(static_cast<char *>(dst) + r * dpitch,
                                        static_cast<const char *>(src) + r * spitch, width, kind, s);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace

extern "C" {

size_t ida_forward_host_staging_bytes(int B, int H, int N, int d, int R, int M, int dtype, int W, int flags) {
    std::string why;
    if (B < 0 || H < 0 || N < 0 || (long long)B * H == 0) return 0;
    if (ida::check_call(d, R, M, W, dtype, flags, nullptr, why) != IDA_OK) return 0;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    return host_plan(B, H, N, d, R, M, dtype, W, flags).total;
}

ida_status ida_forward_host(const void *q, const void *k, const void *v, const float *conv_w,
                            const float *norm_w, const float *bias, const float *lambda, const float *Bvec,
                            const float *state_in, void *out, float *final_state, int B, int H, int N, int d,
                            int R, int M, int dtype, int W, int flags, void *staging, size_t staging_bytes,
                            ida_stream_t stream) {
    std::string why;
    if (B < 0 || H < 0 || N < 0) return ida::fail_with(IDA_ERR_ARG, "B, H and N must be >= 0");
    ida_status s = ida::check_call(d, R, M, W, dtype, flags, nullptr, why);
    if (s != IDA_OK) return ida::fail_with(s, why);
    if ((long long)B * H > (1LL << 24)) return ida::fail_with(IDA_ERR_UNSUPPORTED, "B*H above 2^24");
    if ((long long)B * N * H * (R > d ? R : d) >= (1LL << 62)) return ida::fail_with(IDA_ERR_ARG, "size overflow");
    if ((long long)B * H == 0 || (N == 0 && !final_state)) return IDA_OK;
    if (N > 0 && (!q || !k || !v || !out)) return ida::fail_with(IDA_ERR_ARG, "null host q, k, v or out");
    const void *params[] = {conv_w, norm_w, bias, lambda, Bvec};
    for (const void *p : params)
        if (!p || (reinterpret_cast<uintptr_t>(p) & 15u))
            return ida::fail_with(IDA_ERR_ARG, "parameter pointers must be non-null and 16-byte aligned");
    if (!staging || (reinterpret_cast<uintptr_t>(staging) & 15u))
        return ida::fail_with(IDA_ERR_ARG, "staging must be a non-null, 16-byte aligned device buffer");
    const size_t es = dtype == IDA_BF16 ? 2 : 4;
    const size_t SFb = (size_t)B * H * ida_state_floats(d, R, M, W) * sizeof(float);
    if (state_in && final_state) {
        const char *si = reinterpret_cast<const char *>(state_in), *fo = reinterpret_cast<const char *>(final_state);
        if (si < fo + SFb && fo < si + SFb) return ida::fail_with(IDA_ERR_ARG, "state_in and final_state overlap");
    }
    int num_sms = 0;
    s = ida::check_call(d, R, M, W, dtype, flags, &num_sms, why);  // device set-up, pending device errors
    if (s != IDA_OK) return ida::fail_with(s, why);
    const HostPlan P = host_plan(B, H, N, d, R, M, dtype, W, flags);
    if (staging_bytes < P.total)
        return ida::fail_with(IDA_ERR_ARG, "staging smaller than ida_forward_host_staging_bytes(...)");
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return ida::fail_with(IDA_ERR_CUDA, cudaGetErrorString(e));
    Pipe *pp = get_pipe(dev, why);
    if (!pp) return ida::fail_with(IDA_ERR_CUDA, why);
    std::lock_guard<std::mutex> lock(pp->mu);

    cudaStream_t us = reinterpret_cast<cudaStream_t>(stream);
    char *sb = static_cast<char *>(staging);
    float *st[2] = {reinterpret_cast<float *>(sb + P.off_st[0]), reinterpret_cast<float *>(sb + P.off_st[1])};
    // the three streams start after the work already queued on the caller's stream
    e = cudaEventRecord(pp->ev_a, us);
    for (cudaStream_t x : {pp->in, pp->cmp, pp->out})
        if (e == cudaSuccess) e = cudaStreamWaitEvent(x, pp->ev_a, 0);
    if (e != cudaSuccess) return ida::fail_with(IDA_ERR_CUDA, cudaGetErrorString(e));

    ida_status rs = IDA_OK;
    std::string rwhy;
    auto cuda_fail = [&](cudaError_t err) {
        rs = IDA_ERR_CUDA;
        rwhy = cudaGetErrorString(err);
    };
    if (N == 0) {  // no positions: the final state is the start state
        e = state_in ? cudaMemcpyAsync(st[0], state_in, SFb, cudaMemcpyHostToDevice, pp->out)
                     : cudaMemsetAsync(st[0], 0, SFb, pp->out);
        if (e == cudaSuccess) e = cudaMemcpyAsync(final_state, st[0], SFb, cudaMemcpyDeviceToHost, pp->out);
        if (e != cudaSuccess) cuda_fail(e);
    } else {
        if (state_in && (e = cudaMemcpyAsync(st[1], state_in, SFb, cudaMemcpyHostToDevice, pp->in)) != cudaSuccess)
            cuda_fail(e);
        const char *qh = static_cast<const char *>(q), *kh = static_cast<const char *>(k);
        const char *vh = static_cast<const char *>(v);
        char *oh = static_cast<char *>(out);
        const size_t rowq = (size_t)H * R * es, rowv = (size_t)H * d * es;  // bytes of one position
        for (int i = 0; i < P.S && rs == IDA_OK; ++i) {
            const int slot = i & 1, n0 = i * P.L, n = N - n0 < P.L ? N - n0 : P.L;
            void *dq = sb + P.off_q[slot], *dk = sb + P.off_k[slot], *dv = sb + P.off_v[slot];
            void *dout = sb + P.off_o[slot];
            // copy-in of slice i, once the prefill of slice i-2 no longer reads this slot
            if (i >= 2) e = cudaStreamWaitEvent(pp->in, pp->ev_cmp[slot], 0);
            if (e == cudaSuccess)
                e = copy_rows(dq, n * rowq, qh + n0 * rowq, (size_t)N * rowq, n * rowq, B, cudaMemcpyHostToDevice, pp->in);
            if (e == cudaSuccess)
                e = copy_rows(dk, n * rowq, kh + n0 * rowq, (size_t)N * rowq, n * rowq, B, cudaMemcpyHostToDevice, pp->in);
            if (e == cudaSuccess)
                e = copy_rows(dv, n * rowv, vh + n0 * rowv, (size_t)N * rowv, n * rowv, B, cudaMemcpyHostToDevice, pp->in);
            if (e == cudaSuccess) e = cudaEventRecord(pp->ev_in[slot], pp->in);
            // prefill of slice i, once its inputs are in and slice i-2's outputs are out
            if (e == cudaSuccess) e = cudaStreamWaitEvent(pp->cmp, pp->ev_in[slot], 0);
            if (e == cudaSuccess && i >= 2) e = cudaStreamWaitEvent(pp->cmp, pp->ev_out[slot], 0);
            if (e != cudaSuccess) {
                cuda_fail(e);
                break;
            }
            const float *sin = i == 0 ? (state_in ? st[1] : nullptr) : st[(i - 1) & 1];
            float *sout = (i + 1 < P.S || final_state) ? st[i & 1] : nullptr;
            rs = ida::forward_entry(dq, dk, dv, conv_w, norm_w, bias, lambda, Bvec, sin, dout, sout, B, H, n, d,
                                    R, M, dtype, W, flags, sb + P.off_ws, P.ws, reinterpret_cast<ida_stream_t>(pp->cmp));
            if (rs != IDA_OK) {
                rwhy = std::string("slice ") + std::to_string(i) + ": " + ida_last_error();
                break;
            }
            e = cudaEventRecord(pp->ev_cmp[slot], pp->cmp);
            // copy-out of slice i
            if (e == cudaSuccess) e = cudaStreamWaitEvent(pp->out, pp->ev_cmp[slot], 0);
            if (e == cudaSuccess)
                e = copy_rows(oh + n0 * rowv, (size_t)N * rowv, dout, n * rowv, n * rowv, B, cudaMemcpyDeviceToHost, pp->out);
            if (e == cudaSuccess) e = cudaEventRecord(pp->ev_out[slot], pp->out);
            if (e != cudaSuccess) cuda_fail(e);
        }
        if (rs == IDA_OK && final_state &&
            (e = cudaMemcpyAsync(final_state, st[(P.S - 1) & 1], SFb, cudaMemcpyDeviceToHost, pp->out)) != cudaSuccess)
            cuda_fail(e);
    }
    // the caller's stream waits for all three streams, whatever was enqueued
    e = cudaEventRecord(pp->ev_a, pp->in);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(pp->out, pp->ev_a, 0);
    if (e == cudaSuccess) e = cudaEventRecord(pp->ev_b, pp->cmp);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(pp->out, pp->ev_b, 0);
    if (e == cudaSuccess) e = cudaEventRecord(pp->ev_a, pp->out);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(us, pp->ev_a, 0);
    if (e != cudaSuccess && rs == IDA_OK) cuda_fail(e);
    return rs == IDA_OK ? IDA_OK : ida::fail_with(rs, rwhy);
}

}  // extern "C"
