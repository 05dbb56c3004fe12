// ida_chunk.cu -- chunked tensor-core prefill (placeholder: not yet taken).
#include <string>

#include "ida_common.cuh"

namespace ida {

ida_status launch_chunk_prefill(const PrefillArgs &, cudaStream_t, int, std::string &, bool *taken) {
    *taken = false;
    return IDA_OK;
}

}  // namespace ida
