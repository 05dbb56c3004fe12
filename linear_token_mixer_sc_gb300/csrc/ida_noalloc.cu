// ida_noalloc.cu -- prefill for callers that cannot allocate device memory.
//
// ida_forward_ws runs long sequences fastest, but it needs a scratch
// workspace that the caller allocates.  Some callers cannot do that: code
// that runs inside a host framework which owns every device allocation and
// hands a plug-in only its input and output buffers, code that must not
// touch the allocator once it has started (a fixed-memory serving loop,
// a real-time path that may not block on cudaMalloc), or code that runs
// where no allocator is reachable at all.  ida_forward_noalloc gives them the
// same computation with its scratch in one array of static device memory
// that this library carries: every GPU that loads the library holds
// kStaticScratchBytes of it until the process exits, and no call allocates.
#include <mutex>
#include <string>

#include "ida_common.cuh"

namespace ida {
ida_status forward_entry(const void *q, const void *k, const void *v, const float *conv_w, const float *norm_w,
                         const float *bias, const float *lambda, const float *Bvec, const float *state_in, void *out,
                         float *final_state, int B, int H, int N, int d, int R, int M, int dtype, int W, int flags,
                         void *workspace, size_t workspace_bytes, ida_stream_t stream);
ida_status fail_with(ida_status s, const std::string &why);
size_t forward_workspace_within(int B, int H, int N, int d, int R, int M, int dtype, int W, int flags,
                                size_t budget);
}  // namespace ida

// The shared scratch: 32 MiB per device.  The prefill planner never picks a plan
// whose segment states exceed the budget it is given (it falls back to coarser
// splits, or to whole sequences), so every supported shape runs; the size check
// below guards that invariant rather than a case a caller can reach.
static constexpr size_t kStaticScratchBytes = size_t(32) << 20;
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

// Device address of the scratch, looked up once per device.  In host code
// g_static_scratch names a host-side stand-in, not device memory, so the
// kernels are only ever handed the address cudaGetSymbolAddress returns.  The
// address stays valid while the device's primary context lives; a
// cudaDeviceReset invalidates it (the header says so).
static std::mutex g_scratch_mu;
static constexpr int kMaxDevices = 64;
static void *g_scratch_dev[kMaxDevices];

extern "C" ida_status ida_forward_noalloc(const void *q, const void *k, const void *v, const float *conv_w,
                                          const float *norm_w, const float *bias, const float *lambda,
                                          const float *Bvec, void *out, float *final_state, int B, int H, int N,
                                          int d, int R, int M, int dtype, int W, int flags, ida_stream_t stream) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return ida::fail_with(IDA_ERR_CUDA, std::string("cudaGetDevice: ") + cudaGetErrorString(e));
    if (dev < 0 || dev >= kMaxDevices) return ida::fail_with(IDA_ERR_UNSUPPORTED, "device ordinal above 63");
    const size_t need = ida::forward_workspace_within(B, H, N, d, R, M, dtype, W, flags, kStaticScratchBytes);
    if (need > kStaticScratchBytes)  // the planner keeps within its budget: not reached
        return ida::fail_with(IDA_ERR_UNSUPPORTED, "internal: a plan of " + std::to_string(need) +
                                                       " bytes of scratch exceeds the static " +
                                                       std::to_string(kStaticScratchBytes));
    void *scratch = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_scratch_mu);
        if (!g_scratch_dev[dev]) {
            void *p = nullptr;
            e = cudaGetSymbolAddress(&p, g_static_scratch);
            if (e != cudaSuccess || !p)
                return ida::fail_with(IDA_ERR_CUDA, std::string("cudaGetSymbolAddress of the static scratch: ") +
                                                        cudaGetErrorString(e));
            g_scratch_dev[dev] = p;
        }
        scratch = g_scratch_dev[dev];
    }
    // Nothing in the scratch has to start at zero: each call writes every slot
    // it reads (segment end states, then start states) before reading it.
    return ida::forward_entry(q, k, v, conv_w, norm_w, bias, lambda, Bvec, nullptr, out, final_state, B, H, N, d, R,
                              M, dtype, W, flags, scratch, kStaticScratchBytes, stream);
}
