// ida_selftest.cu -- a self-test of the library's failure reporting.
//
// Every wait in the prefill kernels (an mbarrier phase that an MMA commit or a
// TMA copy completes) is bounded: when it runs out, the kernel records an
// error code in the device error word, stops, and returns, and the next call
// on the host reports IDA_ERR_DEVICE.  ida_selftest_bounded_wait exercises that
// path on purpose without faulting anything: one thread waits, through the
// same bounded-wait helper the prefill kernels use, on an mbarrier that nothing
// ever arrives on, gives up after the given number of SM clock cycles and
// records kErrWaitTimeout.
#include <string>

#include "ida_common.cuh"
#include "tc_sm103.cuh"

namespace ida {
ida_status fail_with(ida_status s, const std::string &why);
ida_status device_error_word(unsigned **err, std::string &why);

__global__ void __launch_bounds__(32, 1) bounded_wait_selftest_kernel(unsigned *err, long long limit_cycles) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        tc::mbar_init(&bar, 1);  // expects one arrival, which never comes
        tc::fence_mbar_init();
    }
    __syncwarp();
    if (threadIdx.x == 0 && !tc::mbar_wait(&bar, 0, limit_cycles)) report_error(err, kErrWaitTimeout);
}
}  // namespace ida

extern "C" ida_status ida_selftest_bounded_wait(long long limit_cycles, ida_stream_t stream) {
    if (limit_cycles < 1 || limit_cycles > 4000000000LL)
        return ida::fail_with(IDA_ERR_ARG, "limit_cycles must be in [1, 4e9]");
    unsigned *err = nullptr;
    std::string why;
    ida_status s = ida::device_error_word(&err, why);
    if (s != IDA_OK) return ida::fail_with(s, why);
    ida::bounded_wait_selftest_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(err, limit_cycles);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return ida::fail_with(IDA_ERR_CUDA, std::string("self-test launch: ") + cudaGetErrorString(e));
    return IDA_OK;
}
