// prefill.cu -- placeholder until the tcgen05 prefill kernel lands.
#include "rk_device.cuh"

namespace rk {
cudaError_t launch_prefill(const CUtensorMap&, const CUtensorMap&, const CUtensorMap&, const PrefillArgs&,
                           cudaStream_t) {
    return cudaErrorNotSupported;
}
}  // namespace rk
