// prefill.cu - varlen causal / chunked / sliding-window prefill (tcgen05 + TMEM).
#include "pa_common.cuh"
#include "pa_internal.h"

namespace pa {

cudaError_t launch_prefill(const PrefillArgs &a, cudaStream_t stream) {
    (void)a;
    (void)stream;
    return cudaErrorNotSupported;
}

}  // namespace pa
