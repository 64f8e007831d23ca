// fwd_chunked.cu -- tensor-core (tcgen05) chunked SSE forward.
#include "sse_internal.cuh"

namespace sse {

bool chunked_supported(const sse_config_t &) { return false; }

size_t chunked_extra_workspace(const sse_config_t &, int64_t, int32_t) { return 0; }

cudaError_t launch_forward_chunked(const sse_config_t &, const ForwardArgs &, cudaStream_t, int *) {
    return cudaErrorNotSupported;
}

}  // namespace sse
