// prefill.cu -- placeholder until the tcgen05 prefill kernel lands.
#include "common.cuh"

namespace w4a16 {

bool prefill_config_supported(const w4a16_config &, int, int, int, int) { return false; }

cudaError_t launch_prefill(const GemmArgs &, const w4a16_config &, cudaStream_t) {
    return cudaErrorNotSupported;
}

}  // namespace w4a16
